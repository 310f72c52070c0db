// decode_fused.cu — the single-layer instantiations of the persistent
// small-batch layer kernel (decode_fused.cuh) and their launcher.
#include "decode_fused.cuh"

namespace moe {

// Whole small-batch layer in one launch (plus the normalising combine when
// the layer asks for per-expert output normalisation).
cudaError_t launch_decode_fused(const LayerDev &L, const Workspace &ws, const uint16_t *x, const uint16_t *res,
                                uint16_t *out, int T, cudaStream_t st) {
    using namespace fused;
    if (L.E > 256 || L.k > 8 || T > 16 || L.d > 32 * kCb) return cudaErrorInvalidValue;
    cudaError_t e;
    const bool fp4 = L.fmt == MOE_W_NVFP4;
#define MOE_FUSED(TMV) e = fp4 ? launch_t<TMV, true, false>(L, ws, x, res, out, T, st) : launch_t<TMV, false, false>(L, ws, x, res, out, T, st)
    if (T <= 1)
        MOE_FUSED(1);
    else if (T <= 2)
        MOE_FUSED(2);
    else if (T <= 4)
        MOE_FUSED(4);
    else if (T <= 8)
        MOE_FUSED(8);
    else
        MOE_FUSED(16);
#undef MOE_FUSED
    if (e != cudaSuccess) return e;
    if (L.expert_norm) e = launch_combine(L, ws, res, out, T, st);
    return e;
}

}  // namespace moe
