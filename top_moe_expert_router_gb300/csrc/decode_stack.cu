// decode_stack.cu — several layers in one launch: the stacked
// instantiations of the persistent small-batch layer kernel (decode_fused.cuh).
// Layer l's input is RMSNorm(x_l); x_{l+1} = x_l + MoE_l(RMSNorm(x_l)). The
// layers run back to back inside the kernel, separated by grid barriers, so
// the launches, the separate RMSNorm kernels and their gaps are gone.
#include "decode_fused.cuh"

namespace moe {

// Stacked layers in one launch; the weights of layer l are ws.stack[l].
cudaError_t launch_decode_stack(const LayerDev &L, const Workspace &ws, int n_layers, float eps, const uint16_t *x,
                                uint16_t *out, uint16_t *layer_out, int T, cudaStream_t st) {
    using namespace fused;
    if (L.E > 256 || L.k > 8 || T < 1 || T > 8 || L.d > 32 * kCb || L.expert_norm || n_layers < 1 ||
        n_layers > kMaxStack)
        return cudaErrorInvalidValue;
    const bool fp4 = L.fmt == MOE_W_NVFP4;
#define MOE_STACK(TMV)                                                                             \
    return fp4 ? launch_t<TMV, true, true>(L, ws, x, nullptr, out, T, st, n_layers, eps, layer_out)     \
               : launch_t<TMV, false, true>(L, ws, x, nullptr, out, T, st, n_layers, eps, layer_out)
    if (T <= 1) MOE_STACK(1);
    if (T <= 2) MOE_STACK(2);
    if (T <= 4) MOE_STACK(4);
    MOE_STACK(8);
#undef MOE_STACK
}

}  // namespace moe
