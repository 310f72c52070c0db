// common.cuh — shared device helpers of libmoe: inline PTX for mbarriers and
// bulk (TMA) copies, bounded waits, bf16 unpacking, and the workspace layout.
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

#include <atomic>

#include "moe.h"

namespace moe {

// ---------------------------------------------------------------------------
// Error word (first word of the workspace). Kernels OR these bits in; the host
// reads and clears them in moe_get_device_status().
// ---------------------------------------------------------------------------
enum : uint32_t { ERRBIT_TIMEOUT = 1u, ERRBIT_RANGE = 2u };

// A bounded wait gives up after this many nanoseconds of global time.
constexpr unsigned long long kWaitLimitNs = 1500000000ull;  // 1.5 s

// ---------------------------------------------------------------------------
// Workspace layout. All regions 256-byte aligned; sizes depend on the layer
// shape and max_tokens only.
// ---------------------------------------------------------------------------
// One counter alone on a 128-byte line: counters that many CTAs update or poll
// at once do not share a line with each other.
struct CtrLine {
    uint32_t v;
    uint32_t pad[31];
};

struct Control {
    uint32_t err;            // error bits
    uint32_t route_done;     // arrival counter of the router's CTAs (reset by the last)
    int32_t n_uniq;          // number of experts with at least one token
    int32_t n_tiles_gu;      // prefill: gate/up tiles
    int32_t n_tiles_dn;      // prefill: down tiles
    uint32_t test_hold;      // test hook: arrivals the decode kernel's grid barriers wait for beyond the grid (0)
    uint32_t epoch;          // small-batch decode kernel: tag base of the launch's logits (advanced by the last CTA out)
    uint32_t pad0[25];
    CtrLine grid_bar;        // fused decode kernel: grid-barrier arrivals (reset by the last CTA out)
    CtrLine grid_exit;       // fused decode kernel: CTAs that finished
    CtrLine h_ready[2];      // fused decode kernel: h rows written, first / second half of the experts
    CtrLine cb_rows[32];     // fused decode kernel: expert rows done per 256-column block of Y
};

// Tokens per chunk of the large-batch routing (one 32-bit bitmap word per expert).
constexpr int kRouteChunk = 32;

// The large-batch router GEMM splits K (= d) in up to kRouterSplit parts, each
// written to its own slice of the logits region; the large-batch top-k sums
// the parts in order. d is a multiple of 64 (the GEMM's K block).
constexpr int kRouterSplit = 4;
inline int router_ksplit(int d) {
    const int kb = d / 64;
    return kb % kRouterSplit == 0 ? kRouterSplit : (kb % 2 == 0 ? 2 : 1);
}

// One layer's weights, as the kernels see them (bf16 or NVFP4 fields used).
struct LayerW {
    const uint16_t *wr;       // [E, d] router
    const float *bias;        // [E] or null
    const uint16_t *wg, *wu, *wd;
    const uint8_t *qg, *qu, *qd, *sg, *su, *sd;
    const float *gg, *gu, *gd;
    int64_t gu_ld;            // bf16: elements from one gate (or up) row to the next (d, or 2d when interleaved)
};

// Layers one stacked launch can run.
constexpr int kMaxStack = 64;

struct Workspace {
    Control *ctrl;
    LayerW *stack;      // [kMaxStack] weights of the layers of a stacked launch
    float *logits;      // [kRouterSplit][max_T, E] (decode: the first slice)
    uint64_t *tlogits;  // [16, E] small-batch decode: tagged logits (fp32 logit | tag << 32), zeroed at set-up
    int32_t *ids;       // [max_T, k]
    float *w;           // [max_T, k]
    int32_t *counts;    // [E]
    int32_t *offsets;   // [E+1]
    int32_t *uniq;      // [E] experts with tokens, ascending
    int32_t *tile_off;  // [E+1] prefill: exclusive scan of 128-row tiles per expert
    int32_t *perm;      // [max_T*k]
    int32_t *pos;       // [max_T*k]
    uint16_t *xbuf;     // [max_T, d] bf16 staging (host forward, rmsnorm)
    uint16_t *obuf;     // [max_T, d] bf16 staging
    float *h;           // [max_T*k, I] fp32 (decode) / bf16 (prefill)
    float *Y;           // [max_T*k, d] fp32 expert outputs
    uint16_t *xperm;    // [max_T*k, d] bf16 gathered rows (prefill; f16 for NVFP4 experts)
    float *row_scale;   // [max_T*k] NVFP4 prefill: power-of-two scale of each gathered row
    uint16_t *xb;       // [16, d] tensor-core decode: the token rows of the B operand (bf16 / scaled f16)
    float *xscale;      // [16] tensor-core decode, NVFP4: per-token power-of-two scales
    void *tmaps;        // [kMaxStack] tensor-core decode: each stacked layer's tensor maps (1 KB each)
    int32_t *chunk_base;  // [ceil(max_T/kRouteChunk), E] per-chunk counts, then each chunk's first row per expert
    uint32_t *chunk_bm;   // [ceil(max_T/kRouteChunk), E] token bitmaps of each kRouteChunk-token chunk
    size_t bytes;
};

inline size_t align_up(size_t v, size_t a) { return (v + a - 1) / a * a; }

// cudaFuncSetAttribute(MaxDynamicSharedMemorySize) applies to the current
// device only: `done` records, per device ordinal (< 64), where it was set,
// so that one process driving several GPUs sets it on each.
inline cudaError_t set_smem_limit_once(const void *func, int bytes, std::atomic<uint64_t> &done) {
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    const uint64_t bit = dev >= 0 && dev < 64 ? 1ull << dev : 0ull;
    if (bit && (done.load(std::memory_order_acquire) & bit)) return cudaSuccess;
    e = cudaFuncSetAttribute(func, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes);
    if (e == cudaSuccess && bit) done.fetch_or(bit, std::memory_order_acq_rel);
    return e;
}

// Computes the layout; with base == nullptr only the size is meaningful.
inline Workspace workspace_layout(void *base, int d, int E, int k, int I, int max_T) {
    Workspace ws{};
    size_t off = 0;
    auto take = [&](size_t bytes) {
        size_t o = off;
        off = align_up(off + bytes, 256);
        return base ? (void *)((char *)base + o) : nullptr;
    };
    size_t Tk = (size_t)max_T * k;
    ws.ctrl = (Control *)take(sizeof(Control));
    ws.tlogits = (uint64_t *)take(sizeof(uint64_t) * 16 * (size_t)E);   // right after ctrl: one memset clears both
    ws.stack = (LayerW *)take(sizeof(LayerW) * kMaxStack);
    ws.logits = (float *)take(sizeof(float) * (size_t)kRouterSplit * max_T * E);
    ws.ids = (int32_t *)take(sizeof(int32_t) * Tk);
    ws.w = (float *)take(sizeof(float) * Tk);
    ws.counts = (int32_t *)take(sizeof(int32_t) * E);
    ws.offsets = (int32_t *)take(sizeof(int32_t) * (E + 1));
    ws.uniq = (int32_t *)take(sizeof(int32_t) * E);
    ws.tile_off = (int32_t *)take(sizeof(int32_t) * (E + 1));
    ws.perm = (int32_t *)take(sizeof(int32_t) * Tk);
    ws.pos = (int32_t *)take(sizeof(int32_t) * Tk);
    ws.xbuf = (uint16_t *)take(sizeof(uint16_t) * (size_t)max_T * d);
    ws.obuf = (uint16_t *)take(sizeof(uint16_t) * (size_t)max_T * d);
    ws.h = (float *)take(sizeof(float) * Tk * I);
    ws.Y = (float *)take(sizeof(float) * Tk * d);
    ws.xperm = (uint16_t *)take(sizeof(uint16_t) * Tk * d);
    ws.row_scale = (float *)take(sizeof(float) * Tk);
    ws.xb = (uint16_t *)take(sizeof(uint16_t) * 16 * (size_t)d);
    ws.xscale = (float *)take(sizeof(float) * 16);
    ws.tmaps = take((size_t)1024 * kMaxStack);
    const size_t nchunks = ((size_t)max_T + kRouteChunk - 1) / kRouteChunk;
    ws.chunk_base = (int32_t *)take(sizeof(int32_t) * nchunks * E);
    ws.chunk_bm = (uint32_t *)take(sizeof(uint32_t) * nchunks * E);
    ws.bytes = off;
    return ws;
}

// Bytes from ws.ctrl to the end of ws.tlogits (E experts): the control words
// and the tagged logits, cleared together at set-up.
inline size_t control_bytes(const Workspace &ws, int E) {
    return (size_t)((const char *)ws.tlogits - (const char *)ws.ctrl) + sizeof(uint64_t) * 16 * (size_t)E;
}

// ---------------------------------------------------------------------------
// Device helpers
// ---------------------------------------------------------------------------
#ifdef __CUDACC__

__device__ __forceinline__ uint32_t smem_u32(const void *p) {
    return (uint32_t)__cvta_generic_to_shared(p);
}

__device__ __forceinline__ unsigned long long global_ns() {
    unsigned long long t;
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
    return t;
}

// Order-preserving map of a float to an unsigned key (larger float, larger
// key; -0 is taken as +0 so that equal values tie). Key 0 lies below every
// float and marks "no candidate".
__device__ __forceinline__ uint32_t order_key(float f) {
    const uint32_t u = __float_as_uint(f == 0.f ? 0.f : f);
    return (u & 0x80000000u) ? ~u : (u | 0x80000000u);
}

__device__ __forceinline__ float key_value(uint32_t key) {
    return __uint_as_float((key & 0x80000000u) ? (key & 0x7FFFFFFFu) : ~key);
}

// Top-k (k <= 8, E <= 256) of one token's logits by one warp: ids by
// descending logit, ties to the lower id; weights exp(l - l_max) / sum over
// the kept, summed in pick order. Lane l holds experts l, l + 32, ...; each
// pick is a warp-wide max of the lanes' best keys and a warp-wide min of the
// ids that reach it. bypass_l1: read the logits through L2 only (they were
// written by other CTAs of the same launch).
__device__ __forceinline__ void topk_warp(const float *logits_row, int E, int k, int32_t *ids_out, float *w_out,
                                          bool bypass_l1) {
    const int lane = threadIdx.x & 31;
    uint32_t key[8];
#pragma unroll
    for (int i = 0; i < 8; ++i) {
        const int e = lane + 32 * i;
        key[i] = e < E ? order_key(bypass_l1 ? __ldcg(logits_row + e) : logits_row[e]) : 0u;
    }
    uint32_t my_key = 0u;
    int my_id = 0;
    for (int j = 0; j < k; ++j) {
        // this lane's best: largest key, the lowest i (= lowest id) among equals
        uint32_t bk = key[0];
        int bi = 0;
#pragma unroll
        for (int i = 1; i < 8; ++i)
            if (key[i] > bk) {
                bk = key[i];
                bi = i;
            }
        const uint32_t m = __reduce_max_sync(0xFFFFFFFFu, bk);
        const uint32_t win = __reduce_min_sync(0xFFFFFFFFu, bk == m ? (uint32_t)(lane + 32 * bi) : 0xFFFFFFFFu);
        if ((int)(win & 31u) == lane) {
#pragma unroll
            for (int i = 0; i < 8; ++i)
                if (i == (int)(win >> 5)) key[i] = 0u;
        }
        if (lane == j) {
            my_key = m;
            my_id = (int)win;
        }
    }
    const float lmax = __shfl_sync(0xFFFFFFFFu, key_value(my_key), 0);
    const float ex = lane < k ? expf(key_value(my_key) - lmax) : 0.f;
    float sum = 0.f;
    for (int j = 0; j < k; ++j) sum += __shfl_sync(0xFFFFFFFFu, ex, j);
    if (lane < k) {
        ids_out[lane] = my_id;
        w_out[lane] = ex / sum;
    }
}

// Release/acquire fence at GPU scope: with a relaxed atomic it orders this
// thread's earlier stores before the atomic (release side), or the atomic's
// observation before later loads (acquire side). Cheaper than the sequentially
// consistent __threadfence(), whose total order these hand-offs do not need.
__device__ __forceinline__ void fence_acq_rel_gpu() { asm volatile("fence.acq_rel.gpu;" ::: "memory"); }

__device__ __forceinline__ void mbar_init(uint64_t *bar, uint32_t count) {
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(bar)), "r"(count) : "memory");
}

// Ends an mbarrier's life so that its word can be initialised again.
__device__ __forceinline__ void mbar_inval(uint64_t *bar) {
    asm volatile("mbarrier.inval.shared::cta.b64 [%0];" ::"r"(smem_u32(bar)) : "memory");
}

// Makes mbarrier initialisation visible to the async (TMA) proxy.
__device__ __forceinline__ void fence_barrier_init() {
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint64_t *bar, uint32_t bytes) {
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_u32(bar)), "r"(bytes)
                 : "memory");
}

__device__ __forceinline__ void mbar_arrive(uint64_t *bar) {
    asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_u32(bar)) : "memory");
}

__device__ __forceinline__ bool mbar_try_wait(uint64_t *bar, uint32_t parity) {
    uint32_t ok;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(ok)
        : "r"(smem_u32(bar)), "r"(parity)
        : "memory");
    return ok != 0;
}

// Non-blocking test: has the phase of `bar` with the given parity completed?
__device__ __forceinline__ bool mbar_test_wait(uint64_t *bar, uint32_t parity) {
    uint32_t ok;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.test_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(ok)
        : "r"(smem_u32(bar)), "r"(parity)
        : "memory");
    return ok != 0;
}

// Waits until the phase of `bar` with the given parity has completed. Gives up
// after kWaitLimitNs, sets ERRBIT_TIMEOUT in *err and returns false.
__device__ __forceinline__ bool mbar_wait(uint64_t *bar, uint32_t parity, uint32_t *err) {
    if (mbar_try_wait(bar, parity)) return true;
    unsigned long long t0 = global_ns();
    for (uint32_t it = 1;; ++it) {
        if (mbar_try_wait(bar, parity)) return true;
        if ((it & 255u) == 0 && global_ns() - t0 > kWaitLimitNs) {
            atomicOr(err, ERRBIT_TIMEOUT);
            return false;
        }
    }
}

// As mbar_wait, but also gives up (returning false) once *abort is set by
// another warp of the CTA; a timeout sets *abort for the others.
__device__ __forceinline__ bool mbar_wait_or_abort(uint64_t *bar, uint32_t parity, uint32_t *err,
                                                   volatile int *abort) {
    if (mbar_try_wait(bar, parity)) return true;
    unsigned long long t0 = global_ns();
    for (uint32_t it = 1;; ++it) {
        if (mbar_try_wait(bar, parity)) return true;
        if ((it & 255u) == 0) {
            if (*abort) return false;
            if (global_ns() - t0 > kWaitLimitNs) {
                atomicOr(err, ERRBIT_TIMEOUT);
                *abort = 1;
                return false;
            }
        }
    }
}

// Bulk (non-tensor) TMA copy global -> shared, completing on `bar` with a byte count.
// dst and src 16-byte aligned, bytes a multiple of 16.
__device__ __forceinline__ void bulk_g2s(void *dst, const void *src, uint32_t bytes, uint64_t *bar,
                                         uint64_t policy) {
    asm volatile(
        "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes.L2::cache_hint [%0], [%1], %2, [%3], %4;" ::"r"(
            smem_u32(dst)),
        "l"(src), "r"(bytes), "r"(smem_u32(bar)), "l"(policy)
        : "memory");
}

__device__ __forceinline__ uint64_t policy_evict_first() {
    uint64_t p;
    asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(p));
    return p;
}

__device__ __forceinline__ uint64_t policy_evict_last() {
    uint64_t p;
    asm volatile("createpolicy.fractional.L2::evict_last.b64 %0, 1.0;" : "=l"(p));
    return p;
}

// Named barrier over `nthreads` threads (a multiple of 32), id 1..15.
__device__ __forceinline__ void named_bar(uint32_t id, uint32_t nthreads) {
    asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(nthreads) : "memory");
}

__device__ __forceinline__ float bf16lo(uint32_t w) { return __uint_as_float(w << 16); }
__device__ __forceinline__ float bf16hi(uint32_t w) { return __uint_as_float(w & 0xFFFF0000u); }

__device__ __forceinline__ uint16_t f32_to_bf16_rn(float f) {
    uint32_t u = __float_as_uint(f);
    if ((u & 0x7F800000u) == 0x7F800000u && (u & 0x007FFFFFu)) return (uint16_t)((u >> 16) | 0x40u);
    u += 0x7FFFu + ((u >> 16) & 1u);
    return (uint16_t)(u >> 16);
}

__device__ __forceinline__ float warp_sum(float v) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xFFFFFFFFu, v, o);
    return v;
}

__device__ __forceinline__ float silu(float g) { return g / (1.0f + __expf(-g)); }

// Eight E2M1 codes (one 32-bit word, the low nibble of each byte holding the
// lower index) to four f16 pairs, exactly: byte b -> o[b] = {code 2b, code 2b+1}.
// The word is split into its four bytes by the unpacking move, so each pair
// costs one hardware conversion.
__device__ __forceinline__ void e2m1x8_to_f16x2(uint32_t w, uint32_t o[4]) {
    asm("{\n\t.reg .b8 b0, b1, b2, b3;\n\t"
        "mov.b32 {b0, b1, b2, b3}, %4;\n\t"
        "cvt.rn.f16x2.e2m1x2 %0, b0;\n\t"
        "cvt.rn.f16x2.e2m1x2 %1, b1;\n\t"
        "cvt.rn.f16x2.e2m1x2 %2, b2;\n\t"
        "cvt.rn.f16x2.e2m1x2 %3, b3;\n\t}"
        : "=r"(o[0]), "=r"(o[1]), "=r"(o[2]), "=r"(o[3])
        : "r"(w));
}

// Two E4M3 values (low byte first) to an f16 pair, exactly.
__device__ __forceinline__ uint32_t e4m3x2_to_f16x2(uint16_t v) {
    uint32_t o;
    asm("cvt.rn.f16x2.e4m3x2 %0, %1;" : "=r"(o) : "h"(v));
    return o;
}

#endif  // __CUDACC__

// ---------------------------------------------------------------------------
// Launchers (defined in the .cu files), all asynchronous on `st`.
// ---------------------------------------------------------------------------
struct LayerDev {
    int d, E, k, I, max_T;
    moe_wfmt fmt;
    const uint16_t *wr;
    const float *bias;
    const uint16_t *wg, *wu, *wd;
    const uint8_t *qg, *qu, *qd, *sg, *su, *sd;
    const float *gg, *gu, *gd;
    int num_sms;
    int expert_norm;  // RMS-normalise each expert output before the weighted sum
    int64_t gu_ld;    // bf16: elements from one gate (or up) row to the next: d, or 2d when the
                      // rows are interleaved (gate row i, then up row i: wu = wg + d)
    LayerW weights() const { return LayerW{wr, bias, wg, wu, wd, qg, qu, qd, sg, su, sd, gg, gu, gd, gu_ld}; }
};

// route.cu
cudaError_t launch_route_small(const LayerDev &L, const Workspace &ws, const uint16_t *x, int T, cudaStream_t st);
cudaError_t launch_route_large(const LayerDev &L, const Workspace &ws, const uint16_t *x, int T, cudaStream_t st,
                               int *launches);
// decode.cu
cudaError_t launch_decode_gateup(const LayerDev &L, const Workspace &ws, const uint16_t *x, int T, cudaStream_t st);
cudaError_t launch_decode_down(const LayerDev &L, const Workspace &ws, const uint16_t *x, int T, cudaStream_t st);
// decode_fused.cu
cudaError_t launch_decode_fused(const LayerDev &L, const Workspace &ws, const uint16_t *x, const uint16_t *res,
                                uint16_t *out, int T, cudaStream_t st);
// n_layers stacked layers (weights in ws.stack, shapes of L) in one launch:
// x_{l+1} = x_l + MoE_l(RMSNorm(x_l)), x_0 = x, out = x_n; T <= 8.
cudaError_t launch_decode_stack(const LayerDev &L, const Workspace &ws, int n_layers, float eps, const uint16_t *x,
                                uint16_t *out, uint16_t *layer_out, int T, cudaStream_t st);
// misc.cu
cudaError_t launch_combine(const LayerDev &L, const Workspace &ws, const uint16_t *res, uint16_t *out, int T,
                           cudaStream_t st, bool y_bf16 = false);  // y_bf16: expert outputs in bf16 over ws.xperm
cudaError_t launch_bf16_to_f32(const uint16_t *in, float *out, size_t n, cudaStream_t st);
cudaError_t launch_rmsnorm(const uint16_t *x, uint16_t *out, int T, int d, float eps, cudaStream_t st);
cudaError_t launch_quantize_nvfp4(const uint16_t *W, int n, int rows, int K, uint8_t *q, uint8_t *s, float *g,
                                  cudaStream_t st);
cudaError_t launch_gather_rows(const LayerDev &L, const Workspace &ws, const uint16_t *x, int T, cudaStream_t st);
// prefill.cu
cudaError_t launch_router_gemm(const LayerDev &L, const Workspace &ws, const uint16_t *x, int T, cudaStream_t st);
cudaError_t launch_prefill_experts(const LayerDev &L, const Workspace &ws, const uint16_t *x, int T, cudaStream_t st,
                                   int *launches);
// decode_mma.cu: the tensor-core small-batch layer (T <= 16). The tensor maps
// of a layer (weights, token rows, h) are encoded once on the host into a
// 1 KB block; mma_maps_bytes() gives its size.
size_t mma_maps_bytes();
bool mma_encode_maps(const LayerDev &L, const LayerW &w, const Workspace &ws, void *maps_host);
bool mma_supported(const LayerDev &L, int T);
cudaError_t launch_decode_mma(const LayerDev &L, const Workspace &ws, const void *maps_host, const uint16_t *x,
                              const uint16_t *res, uint16_t *out, int T, cudaStream_t st);
// n_layers stacked layers, their maps in ws.tmaps (copied there by the caller)
cudaError_t launch_decode_mma_stack(const LayerDev &L, const Workspace &ws, int n_layers, float eps,
                                    const uint16_t *x, uint16_t *out, uint16_t *layer_out, int T, cudaStream_t st);
// prefill_fp4.cu
cudaError_t launch_gather_rows_f16(const LayerDev &L, const Workspace &ws, const uint16_t *x, int T, cudaStream_t st);
cudaError_t launch_prefill_experts_fp4(const LayerDev &L, const Workspace &ws, int T, cudaStream_t st,
                                       int *launches);

}  // namespace moe
