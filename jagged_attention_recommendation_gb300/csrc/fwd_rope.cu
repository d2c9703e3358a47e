// fwd_rope.cu -- launchers of the jagged attention forward with rotary
// position embedding of Q and K ("Training GEM at LLM scale", section
// "BlockAttention"); the kernel is fwd_kernel<..., ROPE = true> of
// fwd_kernel.cuh, compiled here in its own translation unit.
#include "fwd_kernel.cuh"

namespace jattn {

template <int D, bool ACT, int BIAS>
static cudaError_t launch_rope_t(const TmapSet &tm, const FwdArgs &a, int n_ctas, cudaStream_t stream) {
    using C = FwdCfg<D, ACT, BIAS, true>;
    auto kern = fwd_kernel<D, ACT, BIAS, false, true>;
    static SmemOnce done;
    cudaError_t e = ensure_smem(kern, C::SMEM_ALLOC, done);
    if (e != cudaSuccess || n_ctas <= 0) return e;
    kern<<<n_ctas, C::THREADS, C::SMEM_ALLOC, stream>>>(tm.q, tm.k, tm.v, a);
    return cudaGetLastError();
}

template <int D, bool ACT>
static cudaError_t launch_rope_b(const TmapSet &tm, const FwdArgs &a, int n_ctas, cudaStream_t stream) {
    if (a.g.nb <= 0) return launch_rope_t<D, ACT, kBiasNone>(tm, a, n_ctas, stream);
    if (a.g.H * ext_len(a.g.nb) <= kMaxBiasExtFloats) return launch_rope_t<D, ACT, kBiasExt>(tm, a, n_ctas, stream);
    return launch_rope_t<D, ACT, kBiasTable>(tm, a, n_ctas, stream);
}

// softmax only (the host rejects activation mode with the rotation)
cudaError_t launch_fwd_rope(int D, bool act, const TmapSet &tm, const FwdArgs &a, int n_ctas, cudaStream_t stream) {
    if (a.g.rope_cos == nullptr || a.g.rope_sin == nullptr || a.g.window > 0 || act) return cudaErrorInvalidValue;
    if (D == 128) return launch_rope_b<128, false>(tm, a, n_ctas, stream);
    if (D == 64) return launch_rope_b<64, false>(tm, a, n_ctas, stream);
    return cudaErrorInvalidValue;
}

}  // namespace jattn
