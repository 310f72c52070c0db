// api.cu — the C ABI of libmoe.so (declared in include/moe.h): argument
// validation, workspace layout and the enqueueing of the kernels of one
// Mixture-of-Experts layer forward on the caller's stream.
#include <cuda_runtime.h>
#include <stdint.h>
#include <string.h>

#include <new>
#include <vector>

#include "common.cuh"

struct moe_layer {
    moe::LayerDev L;
    moe::Workspace ws;
    int last_launches;
    int decode_path = MOE_DECODE_AUTO;
    bool mma_maps_ok = false;            // the tensor-core decode kernel's tensor maps are encoded
    std::vector<unsigned char> mma_maps;  // host copy, passed by value at launch
    bool y_bf16 = false;  // the last forward left the expert outputs in bf16 over ws.xperm
    // profiling: events [forward][kernel boundary]
    std::vector<cudaEvent_t> prof_events;
    int prof_max = 0, prof_count = 0, prof_nk = 0;
};

namespace {

using namespace moe;

constexpr int kDecodeMaxT = 16;

bool aligned16(const void *p) { return ((uintptr_t)p & 15u) == 0; }

moe_status check_shape(const moe_layer_desc *d) {
    if (!d) return MOE_ERR_INVALID_ARG;
    if (d->top_k < 1 || d->E < 1 || d->d < 1 || d->I < 1 || d->max_tokens < 1) return MOE_ERR_INVALID_ARG;
    if (d->top_k > 8 || d->E > 256 || d->top_k > d->E) return MOE_ERR_UNSUPPORTED;
    if (d->d % 64 || d->I % 64 || d->d > 8192 || d->I > 4096 || d->max_tokens > 65536) return MOE_ERR_UNSUPPORTED;
    if (d->fmt != MOE_W_BF16 && d->fmt != MOE_W_NVFP4) return MOE_ERR_UNSUPPORTED;
    if (d->fmt == MOE_W_NVFP4 && (d->d % 256 || d->I % 256)) return MOE_ERR_UNSUPPORTED;
    if (d->gate_up_interleaved && d->fmt != MOE_W_BF16) return MOE_ERR_UNSUPPORTED;
    return MOE_OK;
}

moe_status check_desc(const moe_layer_desc *d) {
    moe_status s = check_shape(d);
    if (s != MOE_OK) return s;
    if (!d->w_router || !aligned16(d->w_router)) return MOE_ERR_INVALID_ARG;
    if (d->fmt == MOE_W_BF16) {
        const void *p[] = {d->w_gate, d->gate_up_interleaved ? d->w_gate : d->w_up, d->w_down};
        for (const void *q : p)
            if (!q || !aligned16(q)) return MOE_ERR_INVALID_ARG;
    } else {
        const void *p[] = {d->q_gate, d->q_up, d->q_down, d->s_gate, d->s_up, d->s_down,
                           d->g_gate, d->g_up, d->g_down};
        for (const void *q : p)
            if (!q || !aligned16(q)) return MOE_ERR_INVALID_ARG;
    }
    return MOE_OK;
}

// Largest token count the streaming expert stage takes at hidden size d
// (the tokens' rows are staged in shared memory next to the weight ring).
int decode_max_tokens(int d) {
    int t = kDecodeMaxT;
    while (t > 1 && (size_t)t * d * 2 + 2 * (2 * 2 * (size_t)d * 2) + 4096 > 227 * 1024) t /= 2;
    return t;
}

moe_status cuda_status(cudaError_t e) { return e == cudaSuccess ? MOE_OK : MOE_ERR_CUDA; }

constexpr int kProfSlots = 8;  // event slots per recorded forward

// Records the boundary event `i` of the current forward when profiling.
void prof_mark(moe_layer *ly, int i, cudaStream_t st) {
    if (ly->prof_count < ly->prof_max && i < kProfSlots)
        cudaEventRecord(ly->prof_events[(size_t)ly->prof_count * kProfSlots + i], st);
}

// The tensor-core grouped GEMMs (bf16 or NVFP4 experts) take d a multiple of
// 256 (down-projection N tile) and I a multiple of 128 (gate/up N tile).
bool prefill_supported(const LayerDev &L) { return L.d % 256 == 0 && L.I % 128 == 0; }

// Large-batch forward: tensor-core router, top-k, permutation, row gather,
// grouped gate/up GEMM with SwiGLU, grouped down GEMM, combine.
moe_status forward_prefill(moe_layer *ly, const uint16_t *x, const uint16_t *res, uint16_t *out, int T,
                           cudaStream_t st) {
    const LayerDev &L = ly->L;
    int launches = 0;
    prof_mark(ly, 0, st);
    const bool fp4 = L.fmt == MOE_W_NVFP4;
    cudaError_t e = launch_route_large(L, ly->ws, x, T, st, &launches);
    if (e == cudaSuccess) e = fp4 ? launch_gather_rows_f16(L, ly->ws, x, T, st) : launch_gather_rows(L, ly->ws, x, T, st);
    ++launches;
    prof_mark(ly, 1, st);
    if (e == cudaSuccess)
        e = fp4 ? launch_prefill_experts_fp4(L, ly->ws, T, st, &launches)
                : launch_prefill_experts(L, ly->ws, x, T, st, &launches);
    prof_mark(ly, 2, st);
    const bool y_bf16 = !L.expert_norm;  // the down GEMM's bf16 expert outputs
    if (e == cudaSuccess) e = launch_combine(L, ly->ws, res, out, T, st, y_bf16);
    ++launches;
    ly->y_bf16 = y_bf16;
    prof_mark(ly, 3, st);
    ly->last_launches = launches;
    if (ly->prof_count < ly->prof_max) {
        ly->prof_nk = 3;
        ++ly->prof_count;
    }
    return e == cudaSuccess ? MOE_OK : MOE_ERR_CUDA;
}

// Which small-batch kernel runs T tokens: the tensor-core layer kernel
// (decode_mma) or the CUDA-core one (decode_fused). By default the tensor
// cores take bf16 batches of 8 or more tokens, where the CUDA cores'
// arithmetic, not the weight stream, sets the pace (measured: 16 tokens 0.87
// of the HBM roofline on the tensor cores against 0.75; 4 tokens 0.85 on the
// CUDA cores, whose row-pair stages balance finer than 128-row units).
bool use_mma(const moe_layer *ly, int T) {
    if (ly->decode_path == MOE_DECODE_CUDA_CORES || !ly->mma_maps_ok || !mma_supported(ly->L, T)) return false;
    if (ly->decode_path == MOE_DECODE_TENSOR_CORES) return true;
    return ly->L.fmt == MOE_W_BF16 && T >= 8;
}

// Forward on device buffers; res may be NULL.
moe_status forward_impl(moe_layer *ly, const uint16_t *x, const uint16_t *res, uint16_t *out, int T,
                        cudaStream_t st) {
    const LayerDev &L = ly->L;
    int launches = 0;
    const int tdec = decode_max_tokens(L.d);
    if (T > tdec && prefill_supported(L)) return forward_prefill(ly, x, res, out, T, st);
    ly->y_bf16 = false;
    const bool mma = T <= 16 && use_mma(ly, T);
    if (T <= tdec || mma) {
        // the whole layer in one persistent launch
        prof_mark(ly, 0, st);
        cudaError_t e = mma ? launch_decode_mma(L, ly->ws, ly->mma_maps.data(), x, res, out, T, st)
                            : launch_decode_fused(L, ly->ws, x, res, out, T, st);
        prof_mark(ly, 1, st);
        ly->last_launches = L.expert_norm ? 2 : 1;
        if (ly->prof_count < ly->prof_max) {
            ly->prof_nk = 1;
            ++ly->prof_count;
        }
        return e == cudaSuccess ? MOE_OK : MOE_ERR_CUDA;
    }
    // Token chunks of at most tdec tokens run the streaming expert stage; a
    // chunk is a full layer forward (route, experts, combine) of its tokens.
    for (int t0 = 0; t0 < T; t0 += tdec) {
        const int n = T - t0 < tdec ? T - t0 : tdec;
        const uint16_t *xc = x + (size_t)t0 * L.d;
        cudaError_t e = launch_route_small(L, ly->ws, xc, n, st);
        ++launches;
        if (e == cudaSuccess) e = launch_decode_gateup(L, ly->ws, xc, n, st);
        ++launches;
        if (e == cudaSuccess) e = launch_decode_down(L, ly->ws, xc, n, st);
        ++launches;
        if (e == cudaSuccess)
            e = launch_combine(L, ly->ws, res ? res + (size_t)t0 * L.d : nullptr, out + (size_t)t0 * L.d, n, st);
        ++launches;
        if (e != cudaSuccess) {
            ly->last_launches = launches;
            return MOE_ERR_CUDA;
        }
    }
    ly->last_launches = launches;
    return MOE_OK;
}

// Device-to-device copies of the routing records in the workspace (any
// destination may be NULL).
moe_status copy_records(const moe_layer *ly, int T, int32_t *ids, float *w, int32_t *counts, int32_t *offsets,
                        int32_t *perm, int32_t *pos, cudaStream_t st) {
    const LayerDev &L = ly->L;
    const Workspace &ws = ly->ws;
    const size_t Tk = (size_t)T * L.k;
    struct {
        void *dst;
        const void *src;
        size_t bytes;
    } cp[] = {{ids, ws.ids, Tk * 4}, {w, ws.w, Tk * 4},          {counts, ws.counts, (size_t)L.E * 4},
              {offsets, ws.offsets, (size_t)(L.E + 1) * 4},     {perm, ws.perm, Tk * 4}, {pos, ws.pos, Tk * 4}};
    for (auto &c : cp)
        if (c.dst && cudaMemcpyAsync(c.dst, c.src, c.bytes, cudaMemcpyDeviceToDevice, st) != cudaSuccess)
            return MOE_ERR_CUDA;
    return MOE_OK;
}

}  // namespace

extern "C" {

moe_status moe_workspace_size(const moe_layer_desc *desc, size_t *bytes) {
    moe_status s = check_shape(desc);
    if (s != MOE_OK) return s;
    if (!bytes) return MOE_ERR_INVALID_ARG;
    *bytes = workspace_layout(nullptr, desc->d, desc->E, desc->top_k, desc->I, desc->max_tokens).bytes;
    return MOE_OK;
}

moe_status moe_layer_create(const moe_layer_desc *desc, void *workspace, size_t ws_bytes, moe_layer **out) {
    moe_status s = check_desc(desc);
    if (s != MOE_OK) return s;
    if (!out || !workspace || ((uintptr_t)workspace & 255u)) return MOE_ERR_INVALID_ARG;
    Workspace ws = workspace_layout(workspace, desc->d, desc->E, desc->top_k, desc->I, desc->max_tokens);
    if (ws_bytes < ws.bytes) return MOE_ERR_INVALID_ARG;
    int dev = 0, sms = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return MOE_ERR_CUDA;
    if (cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) return MOE_ERR_CUDA;
    if (cudaMemset(ws.ctrl, 0, control_bytes(ws, desc->E)) != cudaSuccess) return MOE_ERR_CUDA;
    moe_layer *ly = new (std::nothrow) moe_layer();
    if (!ly) return MOE_ERR_INVALID_ARG;
    LayerDev &L = ly->L;
    L.d = desc->d;
    L.E = desc->E;
    L.k = desc->top_k;
    L.I = desc->I;
    L.max_T = desc->max_tokens;
    L.fmt = desc->fmt;
    L.wr = (const uint16_t *)desc->w_router;
    L.bias = desc->router_bias;
    L.wg = (const uint16_t *)desc->w_gate;
    L.wu = desc->gate_up_interleaved ? L.wg + desc->d : (const uint16_t *)desc->w_up;
    L.gu_ld = desc->gate_up_interleaved ? 2 * (int64_t)desc->d : desc->d;
    L.wd = (const uint16_t *)desc->w_down;
    L.qg = desc->q_gate;
    L.qu = desc->q_up;
    L.qd = desc->q_down;
    L.sg = desc->s_gate;
    L.su = desc->s_up;
    L.sd = desc->s_down;
    L.gg = desc->g_gate;
    L.gu = desc->g_up;
    L.gd = desc->g_down;
    L.num_sms = sms;
    L.expert_norm = desc->expert_out_norm ? 1 : 0;
    ly->ws = ws;
    ly->last_launches = 0;
    ly->mma_maps.assign(mma_maps_bytes(), 0);
    const LayerW w = L.weights();
    ly->mma_maps_ok = mma_encode_maps(L, w, ws, ly->mma_maps.data());
    *out = ly;
    return MOE_OK;
}

moe_status moe_set_decode_path(moe_layer *ly, int path) {
    if (!ly || path < MOE_DECODE_AUTO || path > MOE_DECODE_TENSOR_CORES) return MOE_ERR_INVALID_ARG;
    ly->decode_path = path;
    return MOE_OK;
}

moe_status moe_route(moe_layer *ly, const void *x, int T, int32_t *ids, float *w, int32_t *counts,
                     int32_t *offsets, int32_t *perm, int32_t *pos, void *stream) {
    if (!ly || !x || !aligned16(x) || T < 1 || T > ly->L.max_T) return MOE_ERR_INVALID_ARG;
    cudaStream_t st = (cudaStream_t)stream;
    const LayerDev &L = ly->L;
    const Workspace &ws = ly->ws;
    int launches = 0;
    cudaError_t e;
    if (T <= 32) {
        e = launch_route_small(L, ws, (const uint16_t *)x, T, st);
        launches = 1;
    } else {
        e = launch_route_large(L, ws, (const uint16_t *)x, T, st, &launches);
    }
    ly->last_launches = launches;
    if (e != cudaSuccess) return MOE_ERR_CUDA;
    return copy_records(ly, T, ids, w, counts, offsets, perm, pos, st);
}

moe_status moe_debug_route_records(moe_layer *ly, int T, int32_t *ids, float *w, int32_t *counts, int32_t *offsets,
                                   int32_t *perm, int32_t *pos, void *stream) {
    if (!ly || T < 1 || T > ly->L.max_T) return MOE_ERR_INVALID_ARG;
    return copy_records(ly, T, ids, w, counts, offsets, perm, pos, (cudaStream_t)stream);
}

moe_status moe_debug_hold_grid_barrier(moe_layer *ly, int hold, void *stream) {
    if (!ly) return MOE_ERR_INVALID_ARG;
    static const uint32_t kOne = 1u, kZero = 0u;
    return cuda_status(cudaMemcpyAsync(&ly->ws.ctrl->test_hold, hold ? &kOne : &kZero, sizeof(uint32_t),
                                       cudaMemcpyHostToDevice, (cudaStream_t)stream));
}

moe_status moe_forward(moe_layer *ly, const void *x, void *out, int T, void *stream) {
    if (!ly || !x || !out || !aligned16(x) || !aligned16(out) || T < 1 || T > ly->L.max_T || x == out)
        return MOE_ERR_INVALID_ARG;
    return forward_impl(ly, (const uint16_t *)x, nullptr, (uint16_t *)out, T, (cudaStream_t)stream);
}

moe_status moe_forward_residual(moe_layer *ly, const void *x, const void *res, void *out, int T, void *stream) {
    if (!ly || !x || !res || !out || !aligned16(x) || !aligned16(res) || !aligned16(out) || T < 1 ||
        T > ly->L.max_T || x == out)
        return MOE_ERR_INVALID_ARG;
    return forward_impl(ly, (const uint16_t *)x, (const uint16_t *)res, (uint16_t *)out, T, (cudaStream_t)stream);
}

moe_status moe_forward_host(moe_layer *ly, const void *x_host, void *out_host, int T, void *stream) {
    if (!ly || !x_host || !out_host || T < 1 || T > ly->L.max_T) return MOE_ERR_INVALID_ARG;
    cudaStream_t st = (cudaStream_t)stream;
    const size_t bytes = (size_t)T * ly->L.d * 2;
    if (cudaMemcpyAsync(ly->ws.xbuf, x_host, bytes, cudaMemcpyHostToDevice, st) != cudaSuccess) return MOE_ERR_CUDA;
    moe_status s = forward_impl(ly, ly->ws.xbuf, nullptr, ly->ws.obuf, T, st);
    if (s != MOE_OK) return s;
    if (cudaMemcpyAsync(out_host, ly->ws.obuf, bytes, cudaMemcpyDeviceToHost, st) != cudaSuccess) return MOE_ERR_CUDA;
    return cuda_status(cudaStreamSynchronize(st));
}

moe_status moe_debug_expert_outputs(moe_layer *ly, float *Y, int T, void *stream) {
    if (!ly || !Y || T < 1 || T > ly->L.max_T) return MOE_ERR_INVALID_ARG;
    const size_t n = (size_t)T * ly->L.k * ly->L.d;
    if (ly->y_bf16) return cuda_status(launch_bf16_to_f32(ly->ws.xperm, Y, n, (cudaStream_t)stream));
    return cuda_status(cudaMemcpyAsync(Y, ly->ws.Y, n * sizeof(float), cudaMemcpyDeviceToDevice, (cudaStream_t)stream));
}

moe_status moe_rmsnorm(const void *x, void *out, int T, int d, float eps, void *stream) {
    if (!x || !out || !aligned16(x) || !aligned16(out) || T < 1 || d < 8 || d % 8 || !(eps >= 0.f))
        return MOE_ERR_INVALID_ARG;
    return cuda_status(launch_rmsnorm((const uint16_t *)x, (uint16_t *)out, T, d, eps, (cudaStream_t)stream));
}

moe_status moe_quantize_nvfp4(const void *W, int n, int rows, int K, uint8_t *q, uint8_t *s, float *g,
                              void *stream) {
    if (!W || !q || !s || !g || !aligned16(W) || !aligned16(q) || ((uintptr_t)g & 3u) || n < 1 || n > 65535 ||
        rows < 1 || K < 32 || K % 32)
        return MOE_ERR_INVALID_ARG;
    return cuda_status(launch_quantize_nvfp4((const uint16_t *)W, n, rows, K, q, s, g, (cudaStream_t)stream));
}

moe_status moe_get_device_status(moe_layer *ly, void *stream) {
    if (!ly) return MOE_ERR_INVALID_ARG;
    cudaStream_t st = (cudaStream_t)stream;
    if (cudaStreamSynchronize(st) != cudaSuccess) return MOE_ERR_CUDA;
    uint32_t err = 0;
    if (cudaMemcpy(&err, &ly->ws.ctrl->err, sizeof(err), cudaMemcpyDeviceToHost) != cudaSuccess) return MOE_ERR_CUDA;
    if (err && cudaMemset(&ly->ws.ctrl->err, 0, sizeof(err)) != cudaSuccess) return MOE_ERR_CUDA;
    if (err & ERRBIT_TIMEOUT) return MOE_ERR_TIMEOUT;
    if (err) return MOE_ERR_DEVICE;
    return MOE_OK;
}

int moe_last_launch_count(const moe_layer *ly) { return ly ? ly->last_launches : 0; }

moe_status moe_profile_begin(moe_layer *ly, int max_forwards) {
    if (!ly || max_forwards < 1 || max_forwards > (1 << 20)) return MOE_ERR_INVALID_ARG;
    for (cudaEvent_t ev : ly->prof_events) cudaEventDestroy(ev);
    ly->prof_events.assign((size_t)max_forwards * kProfSlots, nullptr);
    for (auto &ev : ly->prof_events)
        if (cudaEventCreate(&ev) != cudaSuccess) return MOE_ERR_CUDA;
    ly->prof_max = max_forwards;
    ly->prof_count = 0;
    ly->prof_nk = 0;
    return MOE_OK;
}

moe_status moe_profile_end(moe_layer *ly, float *ms, int max_kernels, int *n_forwards, int *n_kernels) {
    if (!ly || !n_forwards || !n_kernels || (max_kernels > 0 && !ms)) return MOE_ERR_INVALID_ARG;
    moe_status s = MOE_OK;
    const int nk = ly->prof_nk;
    for (int f = 0; f < ly->prof_count && s == MOE_OK; ++f) {
        cudaEvent_t *ev = &ly->prof_events[(size_t)f * kProfSlots];
        if (cudaEventSynchronize(ev[nk]) != cudaSuccess) s = MOE_ERR_CUDA;
        for (int i = 0; i < nk && i < max_kernels && s == MOE_OK; ++i)
            if (cudaEventElapsedTime(&ms[(size_t)f * max_kernels + i], ev[i], ev[i + 1]) != cudaSuccess)
                s = MOE_ERR_CUDA;
    }
    *n_forwards = ly->prof_count;
    *n_kernels = nk;
    for (cudaEvent_t ev : ly->prof_events) cudaEventDestroy(ev);
    ly->prof_events.clear();
    ly->prof_max = ly->prof_count = 0;
    return s;
}

struct moe_stack {
    moe_layer *first;  // its workspace holds the stack's weight records
    int n_layers;
};

moe_status moe_stack_create(moe_layer *const *layers, int n_layers, moe_stack **out) {
    if (!layers || !out || n_layers < 1 || n_layers > kMaxStack) return MOE_ERR_INVALID_ARG;
    *out = nullptr;
    if (!layers[0]) return MOE_ERR_INVALID_ARG;
    const LayerDev &L0 = layers[0]->L;
    std::vector<LayerW> w((size_t)n_layers);
    for (int l = 0; l < n_layers; ++l) {
        const moe_layer *ly = layers[l];
        if (!ly) return MOE_ERR_INVALID_ARG;
        const LayerDev &L = ly->L;
        if (L.d != L0.d || L.E != L0.E || L.k != L0.k || L.I != L0.I || L.fmt != L0.fmt) return MOE_ERR_INVALID_ARG;
        if (L.expert_norm) return MOE_ERR_UNSUPPORTED;
        w[(size_t)l] = L.weights();
    }
    if (cudaMemcpy(layers[0]->ws.stack, w.data(), sizeof(LayerW) * (size_t)n_layers, cudaMemcpyHostToDevice) !=
        cudaSuccess)
        return MOE_ERR_CUDA;
    // the tensor-core kernel's maps of every layer (weights of layer l; token
    // rows and h in the first layer's workspace, which the stack runs on)
    if (layers[0]->mma_maps_ok) {
        const size_t mb = mma_maps_bytes();
        std::vector<unsigned char> maps(mb * (size_t)n_layers);
        bool ok = true;
        for (int l = 0; l < n_layers && ok; ++l) {
            LayerDev Ll = L0;
            ok = mma_encode_maps(Ll, w[(size_t)l], layers[0]->ws, maps.data() + mb * (size_t)l);
        }
        if (ok && cudaMemcpy(layers[0]->ws.tmaps, maps.data(), maps.size(), cudaMemcpyHostToDevice) != cudaSuccess)
            return MOE_ERR_CUDA;
        if (!ok) layers[0]->mma_maps_ok = false;
    }
    *out = new moe_stack{layers[0], n_layers};
    return MOE_OK;
}

moe_status moe_stack_forward(moe_stack *sk, const void *x, void *out, int T, float eps, void *layer_out,
                             void *stream) {
    if (!sk || !x || !out || !aligned16(x) || !aligned16(out) || (layer_out && !aligned16(layer_out)) || T < 1 ||
        T > 8 || T > sk->first->L.max_T || !(eps >= 0.f))
        return MOE_ERR_INVALID_ARG;
    moe_layer *ly = sk->first;
    const cudaError_t e =
        use_mma(ly, T) ? launch_decode_mma_stack(ly->L, ly->ws, sk->n_layers, eps, (const uint16_t *)x, (uint16_t *)out,
                                                 (uint16_t *)layer_out, T, (cudaStream_t)stream)
                       : launch_decode_stack(ly->L, ly->ws, sk->n_layers, eps, (const uint16_t *)x, (uint16_t *)out,
                                             (uint16_t *)layer_out, T, (cudaStream_t)stream);
    ly->last_launches = 1;
    if (e == cudaErrorInvalidValue || e == cudaErrorInvalidConfiguration) return MOE_ERR_UNSUPPORTED;
    return e == cudaSuccess ? MOE_OK : MOE_ERR_CUDA;
}

moe_status moe_stack_forward_host(moe_stack *sk, const void *x_host, void *out_host, int T, float eps,
                                  void *stream) {
    if (!sk || !x_host || !out_host || T < 1 || T > 8 || T > sk->first->L.max_T || !(eps >= 0.f))
        return MOE_ERR_INVALID_ARG;
    moe_layer *ly = sk->first;
    cudaStream_t st = (cudaStream_t)stream;
    const size_t bytes = (size_t)T * ly->L.d * 2;
    if (cudaMemcpyAsync(ly->ws.xbuf, x_host, bytes, cudaMemcpyHostToDevice, st) != cudaSuccess) return MOE_ERR_CUDA;
    const moe_status s = moe_stack_forward(sk, ly->ws.xbuf, ly->ws.obuf, T, eps, nullptr, stream);
    if (s != MOE_OK) return s;
    if (cudaMemcpyAsync(out_host, ly->ws.obuf, bytes, cudaMemcpyDeviceToHost, st) != cudaSuccess) return MOE_ERR_CUDA;
    return cuda_status(cudaStreamSynchronize(st));
}

moe_status moe_stack_destroy(moe_stack *sk) {
    delete sk;
    return MOE_OK;
}

moe_status moe_layer_destroy(moe_layer *ly) {
    if (ly)
        for (cudaEvent_t ev : ly->prof_events) cudaEventDestroy(ev);
    delete ly;
    return MOE_OK;
}

const char *moe_status_string(moe_status s) {
    switch (s) {
        case MOE_OK: return "ok";
        case MOE_ERR_INVALID_ARG: return "invalid argument";
        case MOE_ERR_UNSUPPORTED: return "unsupported shape or format";
        case MOE_ERR_CUDA: return "CUDA call or launch failed";
        case MOE_ERR_DEVICE: return "kernel flagged an out-of-range index";
        case MOE_ERR_TIMEOUT: return "kernel wait timed out";
    }
    return "unknown status";
}

}  // extern "C"
