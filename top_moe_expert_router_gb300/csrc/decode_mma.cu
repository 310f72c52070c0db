// decode_mma.cu — tensor maps, instantiations and launchers of the tensor-core
// small-batch layer kernel (decode_mma.cuh).
#include "decode_mma.cuh"

namespace moe {

using namespace dmma;

size_t mma_maps_bytes() { return sizeof(TMaps); }

// d in 128-row down units, I in 64-row gate/up units, T <= 16 token columns,
// the tokens' rows staged in the ring during the prologue, no per-expert
// output normalisation (that variant keeps the separate normalising combine).
bool mma_supported(const LayerDev &L, int T) {
    if (T < 1 || T > kN || L.d % kDn || L.I % kGu || L.expert_norm || L.E > 256 || L.k > 8 || L.d > 32 * kCb)
        return false;
    if (L.fmt == MOE_W_NVFP4 && (L.d % 256 || L.I % 256)) return false;
    const uint32_t stage = L.fmt == MOE_W_NVFP4 ? Cfg<true>::kStage : Cfg<false>::kStage;
    int ns = (int)((kSmemBudget - kFixed - 1024) / stage);
    if (ns > kMaxSlots) ns = kMaxSlots;
    return (size_t)T * L.d * 2 <= (size_t)ns * stage;
}

bool mma_encode_maps(const LayerDev &L, const LayerW &w, const Workspace &ws, void *maps_host) {
    TMaps *m = static_cast<TMaps *>(maps_host);
    memset(m, 0, sizeof(TMaps));
    const uint64_t gu_rows = (uint64_t)L.E * L.I, dn_rows = (uint64_t)L.E * L.d;
    bool ok = true;
    if (L.fmt == MOE_W_NVFP4) {
        ok = ok && make_tmap_u8(&m->m[0], w.qg, gu_rows, (uint64_t)L.d / 2, 32, kGu);
        ok = ok && make_tmap_u8(&m->m[1], w.qu, gu_rows, (uint64_t)L.d / 2, 32, kGu);
        ok = ok && make_tmap_u8(&m->m[2], w.qd, dn_rows, (uint64_t)L.I / 2, 32, kDn);
        ok = ok && make_tmap_u8(&m->m[3], w.sg, gu_rows, (uint64_t)L.d / 16, 16, kGu);
        ok = ok && make_tmap_u8(&m->m[4], w.su, gu_rows, (uint64_t)L.d / 16, 16, kGu);
        ok = ok && make_tmap_u8(&m->m[5], w.sd, dn_rows, (uint64_t)L.I / 16, 16, kDn);
    } else {
        ok = ok && w.gu_ld >= L.d;   // a row stride below d would alias rows
        ok = ok && make_tmap_bf16_ld(&m->m[0], w.wg, gu_rows, (uint64_t)L.d, (uint64_t)w.gu_ld, kGu);
        ok = ok && make_tmap_bf16_ld(&m->m[1], w.wu, gu_rows, (uint64_t)L.d, (uint64_t)w.gu_ld, kGu);
        ok = ok && make_tmap_bf16(&m->m[2], w.wd, dn_rows, (uint64_t)L.I, kDn);
    }
    ok = ok && make_tmap_bf16(&m->m[6], ws.xb, kN, (uint64_t)L.d, kN);
    ok = ok && make_tmap_bf16(&m->m[7], ws.h, (uint64_t)L.max_T * L.k, (uint64_t)L.I, kN);
    return ok;
}

template <bool FP4, bool STACK>
static cudaError_t launch_t(const LayerDev &L, const Workspace &ws, const TMaps *maps, const uint16_t *x,
                            const uint16_t *res, uint16_t *out, int T, cudaStream_t st, int n_layers, float eps,
                            uint16_t *layer_out) {
    using C = Cfg<FP4>;
    if (!mma_supported(L, T)) return cudaErrorInvalidConfiguration;
    MArgs a{};
    a.x = x;
    a.res = res;
    a.out = out;
    a.lw0 = L.weights();
    a.n_layers = n_layers;
    a.eps = eps;
    a.layer_out = layer_out;
    a.stack_maps = static_cast<const TMaps *>(ws.tmaps);
    a.T = T;
    a.d = L.d;
    a.I = L.I;
    a.E = L.E;
    a.k = L.k;
    a.ws = ws;
    a.xb = ws.xb;
    a.xscale = ws.xscale;
    a.tmem_cols = (int)C::kTmemCols;
    int ns = (int)((kSmemBudget - kFixed - 1024) / C::kStage);
    a.nslots = ns > kMaxSlots ? kMaxSlots : ns;
    const size_t smem = 1024 + kFixed + (size_t)a.nslots * C::kStage;
    static std::atomic<uint64_t> attr_set{0};
    cudaError_t e = set_smem_limit_once((const void *)decode_mma_kernel<FP4, STACK>, (int)smem, attr_set);
    if (e != cudaSuccess) return e;
    TMaps none;
    if (STACK) memset(&none, 0, sizeof(none));
    cudaLaunchConfig_t cfg{};
    cfg.gridDim = dim3(L.num_sms);
    cfg.blockDim = dim3(C::kThreads);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = st;
    cudaLaunchAttribute attrs[1];
    attrs[0].id = cudaLaunchAttributeCooperative;
    attrs[0].val.cooperative = 1;
    cfg.attrs = attrs;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, decode_mma_kernel<FP4, STACK>, a, STACK ? none : *maps);
}

cudaError_t launch_decode_mma(const LayerDev &L, const Workspace &ws, const void *maps_host, const uint16_t *x,
                              const uint16_t *res, uint16_t *out, int T, cudaStream_t st) {
    const TMaps *m = static_cast<const TMaps *>(maps_host);
    return L.fmt == MOE_W_NVFP4 ? launch_t<true, false>(L, ws, m, x, res, out, T, st, 0, 0.f, nullptr)
                                : launch_t<false, false>(L, ws, m, x, res, out, T, st, 0, 0.f, nullptr);
}

cudaError_t launch_decode_mma_stack(const LayerDev &L, const Workspace &ws, int n_layers, float eps,
                                    const uint16_t *x, uint16_t *out, uint16_t *layer_out, int T, cudaStream_t st) {
    if (n_layers < 1 || n_layers > kMaxStack) return cudaErrorInvalidValue;
    return L.fmt == MOE_W_NVFP4 ? launch_t<true, true>(L, ws, nullptr, x, nullptr, out, T, st, n_layers, eps, layer_out)
                                : launch_t<false, true>(L, ws, nullptr, x, nullptr, out, T, st, n_layers, eps, layer_out);
}

}  // namespace moe
