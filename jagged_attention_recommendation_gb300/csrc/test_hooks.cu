// test_hooks.cu -- a test build of the forward kernel whose bounded wait is
// made to run out (fwd_kernel<..., STALL = true>, see fwd_kernel.cuh), so that
// a test can check the error path of a real launch: the status word reports
// JATTN_ERR_DEVICE_TIMEOUT, the kernel returns, and the device stays usable.
#include "fwd_kernel.cuh"

namespace jattn {

template <int D>
static cudaError_t launch_stall_t(const TmapSet &tm, const FwdArgs &a, int n_ctas, cudaStream_t stream) {
    using C = FwdCfg<D, false, kBiasNone>;
    auto kern = fwd_kernel<D, false, kBiasNone, false, false, true>;
    static SmemOnce done;
    cudaError_t e = ensure_smem(kern, C::SMEM_ALLOC, done);
    if (e != cudaSuccess || n_ctas <= 0) return e;
    kern<<<n_ctas, C::THREADS, C::SMEM_ALLOC, stream>>>(tm.q, tm.k, tm.v, a);
    return cudaGetLastError();
}

// softmax, no bias, no window, D in {64, 128}
cudaError_t launch_fwd_stall(int D, const TmapSet &tm, const FwdArgs &a, int n_ctas, cudaStream_t stream) {
    if (a.g.nb > 0 || a.g.window > 0 || a.g.act != kSoftmax || a.g.rope_cos != nullptr) return cudaErrorInvalidValue;
    if (D == 128) return launch_stall_t<128>(tm, a, n_ctas, stream);
    if (D == 64) return launch_stall_t<64>(tm, a, n_ctas, stream);
    return cudaErrorInvalidValue;
}

}  // namespace jattn
