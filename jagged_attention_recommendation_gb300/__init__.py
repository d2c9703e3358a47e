"""GB300 (sm_103a) jagged attention: forward and backward over offsets-indexed
bf16 Q/K/V with asymmetric lengths, relative-position bias, softmax or GDPA
activation, and 64-token BlockAttention.  The compute path is the C-ABI library
``libjattn.so`` (hand-written CUDA); this package only marshals arguments.
"""
from ._binding import (BF16, ERR_ALIGNMENT, ERR_CUDA, ERR_DEVICE_CHECK, ERR_DEVICE_TIMEOUT, ERR_INVALID_ARG,
                       ERR_NO_DEVICE, ERR_UNSUPPORTED, ERR_WORKSPACE, EXPORTED, FP32, GELU_TANH, LIB_PATH, OK, SILU,
                       SOFTMAX, TILES_KV, TILES_Q, JattnError, Mode, Plan, load, shard, status_str)
from .sharding import local_rows

__all__ = ["Plan", "JattnError", "load", "status_str", "shard", "local_rows", "SOFTMAX", "SILU", "GELU_TANH", "TILES_Q", "TILES_KV"]
