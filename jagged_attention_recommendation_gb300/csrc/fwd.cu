// fwd.cu -- launchers of the jagged attention forward (the kernel is in
// fwd_kernel.cuh; the rotary-embedding variants are launched from fwd_rope.cu).
#include "fwd_kernel.cuh"

namespace jattn {

template <int D, bool ACT, int BIAS, bool WIN>
static cudaError_t launch_fwd_w(const TmapSet &tm, const FwdArgs &a, int n_ctas, cudaStream_t stream) {
    using C = FwdCfg<D, ACT, BIAS>;
    auto kern = fwd_kernel<D, ACT, BIAS, WIN>;
    static SmemOnce done;
    cudaError_t e = ensure_smem(kern, C::SMEM_ALLOC, done);
    if (e != cudaSuccess || n_ctas <= 0) return e;
    kern<<<n_ctas, C::THREADS, C::SMEM_ALLOC, stream>>>(tm.q, tm.k, tm.v, a);
    return cudaGetLastError();
}

// MXFP8: softmax, no bias, no window
template <int D>
static cudaError_t launch_fwd_mx(const TmapSet &tm, const FwdArgs &a, int n_ctas, cudaStream_t stream) {
    using C = FwdCfg<D, false, kBiasNone>;
    auto kern = fwd_kernel<D, false, kBiasNone, false, false, false, true>;
    static SmemOnce done;
    cudaError_t e = ensure_smem(kern, C::SMEM_ALLOC, done);
    if (e != cudaSuccess || n_ctas <= 0) return e;
    kern<<<n_ctas, C::THREADS, C::SMEM_ALLOC, stream>>>(tm.q, tm.k, tm.v, a);
    return cudaGetLastError();
}

// tile-parallel (softmax, every query tile meets at most one 128-key block)
template <int D, int BIAS>
static cudaError_t launch_fwd_tp(const TmapSet &tm, const FwdArgs &a, int n_ctas, cudaStream_t stream) {
    using C = FwdCfg<D, false, BIAS>;
    auto kern = fwd_kernel<D, false, BIAS, false, false, false, false, true>;
    static SmemOnce done;
    cudaError_t e = ensure_smem(kern, C::SMEM_ALLOC, done);
    if (e != cudaSuccess || n_ctas <= 0) return e;
    kern<<<n_ctas, C::THREADS, C::SMEM_ALLOC, stream>>>(tm.q, tm.k, tm.v, a);
    return cudaGetLastError();
}

template <int D, bool ACT, int BIAS>
static cudaError_t launch_fwd_t(const TmapSet &tm, const FwdArgs &a, int n_ctas, cudaStream_t stream) {
    if constexpr (!ACT && BIAS == kBiasNone) {
        if (a.g.mxfp8) return a.g.window > 0 ? cudaErrorInvalidValue : launch_fwd_mx<D>(tm, a, n_ctas, stream);
    }
    if (a.g.mxfp8) return cudaErrorInvalidValue;
    if constexpr (!ACT) {
        if (a.g.tile_parallel && a.g.window == 0) return launch_fwd_tp<D, BIAS>(tm, a, n_ctas, stream);
    }
    return a.g.window > 0 ? launch_fwd_w<D, ACT, BIAS, true>(tm, a, n_ctas, stream)
                          : launch_fwd_w<D, ACT, BIAS, false>(tm, a, n_ctas, stream);
}

template <int D, bool ACT>
static cudaError_t launch_fwd_b(const TmapSet &tm, const FwdArgs &a, int n_ctas, cudaStream_t stream) {
    if (a.g.nb <= 0) return launch_fwd_t<D, ACT, kBiasNone>(tm, a, n_ctas, stream);
    if (a.g.H * ext_len(a.g.nb) <= kMaxBiasExtFloats) return launch_fwd_t<D, ACT, kBiasExt>(tm, a, n_ctas, stream);
    return launch_fwd_t<D, ACT, kBiasTable>(tm, a, n_ctas, stream);
}

cudaError_t launch_fwd(int D, bool act, const TmapSet &tm, const FwdArgs &a, int n_ctas, cudaStream_t stream) {
    if (D == 128)
        return act ? launch_fwd_b<128, true>(tm, a, n_ctas, stream) : launch_fwd_b<128, false>(tm, a, n_ctas, stream);
    if (D == 64)
        return act ? launch_fwd_b<64, true>(tm, a, n_ctas, stream) : launch_fwd_b<64, false>(tm, a, n_ctas, stream);
    return cudaErrorInvalidValue;
}

}  // namespace jattn
