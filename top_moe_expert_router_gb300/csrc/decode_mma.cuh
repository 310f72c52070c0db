// decode_mma.cuh — the small-batch (T <= 16) MoE layer in one persistent
// launch with the expert FFNs on the 5th-generation tensor cores.
//
// Decode is bound by streaming the active experts' weights from HBM ("How
// SGLang-TorchTPU accelerated an 816B-parameter MoE on TPU v7", sections
// "Introduction" and "Results and interpretation"). With several tokens per
// expert, or with NVFP4 weights, multiplying the stream on CUDA cores costs
// more issue slots than the stream leaves time for; here the weights are the
// M = 128 operand of tcgen05.mma and the (at most 16) tokens the N = 16
// operand, so an expert with one token and one with sixteen cost the same.
//
// Phases (one cooperative launch, one CTA per SM; with STACK, per layer):
//   1. every CTA stages the tokens (RMSNorm of the layer input when stacked)
//      and CTA t < 16 writes token row t of the B operand (bf16, or for NVFP4
//      experts f16 scaled by a power of two per token) to the workspace;
//      every CTA computes the router logits of its experts; grid barrier;
//   2. every CTA routes all tokens in shared memory (decode_common.cuh);
//   3. work units: gate/up = 64 gate rows + 64 up rows of one expert (the A
//      tile's rows 0-63 and 64-127), down = 128 rows of W_down; each CTA takes
//      an even share of, in order, the first half of the active experts'
//      gate/up units, the second half's, the first half's down units, the
//      second half's (so a half's h is complete long before its down units);
//      a unit streams its K in blocks of 64:
//        warp 0 (TMA): the A tile (bf16: 128 rows x 128 B, 128-byte swizzle;
//          NVFP4: 128 rows of E2M1 codes + the E4M3 scales) and the B tile
//          (16 token rows of x or of h) into a ring slot;
//        warps 6-13 (NVFP4 only): widen the codes times their block scale
//          (exact in f16 / bf16) and write the A tile straight into tensor
//          memory (tcgen05.st), so the widened weights never pass through
//          shared memory;
//        warp 1: tcgen05.mma (M=128, N=16, K=16) into one of four TMEM
//          accumulators;
//        warps 2-5 (TMEM lane quarters): gate/up -> the up quarters hand their
//          values to the gate quarters through shared memory, h = silu(g) * u
//          for the expert's tokens, in bf16, and a count of finished h rows per
//          half; down -> the expert outputs Y in fp32;
//   4. combine per 256-column block by the CTA that completes it (as in
//      decode_fused.cuh).
// Every wait is bounded; a timeout sets the error word and unwinds.
#pragma once

#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include "decode_common.cuh"
#include "gemm.cuh"

namespace moe {

namespace dmma {

constexpr int kN = 16;             // MMA N: token columns
constexpr int kGu = 64;            // gate rows (and up rows) per gate/up unit
constexpr int kDn = 128;           // W_down rows per down unit
constexpr int kNAcc = 4;           // units in flight between the MMA and the epilogue
constexpr int kNA = 8;             // NVFP4: widened A tiles in TMEM, 32 columns each
constexpr int kConvGroups = 2;     // NVFP4: converter groups (4 warps each) taking alternate k-blocks
constexpr int kMaxSlots = 32;
constexpr int kSmemBudget = 227 * 1024;
constexpr int kFixed = 16 * 1024;  // barriers, routing scratch, exchange buffer
constexpr int kCb = 256;           // output columns per combine block

template <bool FP4>
struct Cfg {
    static constexpr int kConvWarps = FP4 ? 8 : 0;
    // 0 producer, 1 MMA, 2-5 epilogue, then (NVFP4) 6-13 converters; warps
    // 0-7 also compute the router and the stacked RMSNorm, so bf16 has 8
    static constexpr int kWarps = FP4 ? 14 : 8;
    static constexpr int kThreads = 32 * kWarps;
    static constexpr uint32_t kB = kN * 128;                         // 16 rows x 64 K x 2 B
    static constexpr uint32_t kA = FP4 ? 128 * 32 + 128 * 16 : 128 * 128;
    static constexpr uint32_t kStage = kB + kA;                      // 8 KB or 18 KB
    // A unit's K is split over kKSplit accumulators (k-block kb feeds
    // accumulator kb % kKSplit; the epilogue adds them): consecutive MMAs into
    // one N = 16 accumulator wait for each other, so independent chains keep
    // the tensor pipe busy when a k-block's bytes arrive faster than one chain.
    static constexpr int kKSplit = FP4 ? 4 : 2;
    static constexpr int kAccCols = kNAcc * kN * kKSplit;          // accumulators: 256 or 128 columns
    static constexpr int kAColBase = kAccCols;                     // NVFP4: first column of the A tiles
    static constexpr uint32_t kTmemCols = FP4 ? 512 : 128;         // + (NVFP4) 8 A tiles x 32 columns
    static_assert(!FP4 || kAColBase + kNA * 32 <= 512, "tensor memory holds the accumulators and A tiles");
    static_assert(kStage % 1024 == 0, "ring slots stay 1024-byte aligned");
};

// Tensor maps: 0 gate, 1 up, 2 down (bf16 tiles, or NVFP4 codes), 3-5 the
// NVFP4 scales of gate, up, down, 6 the token rows (B of gate/up), 7 h (B of
// down).
struct TMaps {
    CUtensorMap m[8];
};

struct MArgs {
    const uint16_t *x;         // [T, d] bf16 (stacked: the first layer's input)
    const uint16_t *res;       // [T, d] bf16 or null (single layer)
    uint16_t *out;             // [T, d] bf16
    LayerW lw0;                // the layer's weights (single layer)
    int n_layers;              // 0: one layer; n > 0: stacked, weights in ws.stack, maps in stack_maps
    float eps;
    uint16_t *layer_out;       // stacked: [n_layers, T, d] or null
    const TMaps *stack_maps;   // stacked: [n_layers] in global memory
    int T, d, I, E, k;
    int nslots;
    Workspace ws;
    uint16_t *xb;              // [16, d] token rows of the B operand (workspace)
    float *xscale;             // [16] NVFP4: per-token power-of-two scale
    int tmem_cols;
};

// tcgen05.mma with the A operand in tensor memory.
__device__ __forceinline__ void mma_tmem_a(uint32_t tmem_d, uint32_t tmem_a, uint64_t bdesc, uint32_t idesc,
                                           uint32_t accumulate) {
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "setp.ne.b32 p, %4, 0;\n\t"
        "tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], %2, %3, p;\n\t}" ::"r"(tmem_d),
        "r"(tmem_a), "l"(bdesc), "r"(idesc), "r"(accumulate)
        : "memory");
}

__device__ __forceinline__ void tmem_st16(uint32_t taddr, const uint32_t v[16]) {
    asm volatile(
        "tcgen05.st.sync.aligned.32x32b.x16.b32 [%0], {%1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, "
        "%15, %16};" ::"r"(taddr),
        "r"(v[0]), "r"(v[1]), "r"(v[2]), "r"(v[3]), "r"(v[4]), "r"(v[5]), "r"(v[6]), "r"(v[7]), "r"(v[8]), "r"(v[9]),
        "r"(v[10]), "r"(v[11]), "r"(v[12]), "r"(v[13]), "r"(v[14]), "r"(v[15])
        : "memory");
}

__device__ __forceinline__ void tmem_st_wait() { asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory"); }

__device__ __forceinline__ void fence_proxy_async_global() { asm volatile("fence.proxy.async.global;" ::: "memory"); }

// Instruction descriptors: kind::f16, fp32 accumulator, K-major A and B,
// M = 128, N = 16; A/B type bf16 (1) or f16 (0).
constexpr uint32_t kIdescBf16 = (1u << 4) | (1u << 7) | (1u << 10) | ((uint32_t)(kN >> 3) << 17) | (8u << 24);
constexpr uint32_t kIdescF16 = (1u << 4) | ((uint32_t)(kN >> 3) << 17) | (8u << 24);

// One unit of this CTA's sequence.
struct Unit {
    bool gu;          // gate/up (else down)
    int u, e;         // active-expert index, expert id
    int row;          // gate/up: first gate row i0; down: first W_down row c0
    int kbs;          // k-blocks of 64
};

__device__ __forceinline__ Unit unit_at(const fused::Plan &pl, const fused::Route &R, int n, int n_gu, int d, int I) {
    Unit un;
    if (n < n_gu) {
        const int per = I / kGu;
        const int g = pl.gu_row(n);
        un.gu = true;
        un.u = g / per;
        un.row = (g - un.u * per) * kGu;
        un.kbs = d / 64;
    } else {
        const int per = d / kDn;
        const int g = pl.dn_unit(n - n_gu);
        un.gu = false;
        un.u = g / per;
        un.row = (g - un.u * per) * kDn;
        un.kbs = I / 64;
    }
    un.e = R.uniq[un.u];
    return un;
}

// Widen one half k-block (32 codes) of one A row: NVFP4 codes times their two
// block scales -> 16 words of f16 pairs (F16OUT) or bf16 pairs.
template <bool F16OUT>
__device__ __forceinline__ void widen32(const unsigned char *codes, const unsigned char *scales, uint32_t o[16]) {
    const uint4 cw = *reinterpret_cast<const uint4 *>(codes);
    const uint32_t s2 = e4m3x2_to_f16x2(*reinterpret_cast<const uint16_t *>(scales));
    const __half2 s = *reinterpret_cast<const __half2 *>(&s2);
    const __half2 s_lo = __low2half2(s), s_hi = __high2half2(s);
    const uint32_t words[4] = {cw.x, cw.y, cw.z, cw.w};
#pragma unroll
    for (int j = 0; j < 4; ++j) {
        uint32_t p[4];
        e2m1x8_to_f16x2(words[j], p);
#pragma unroll
        for (int b = 0; b < 4; ++b) {
            const __half2 v = __hmul2(*reinterpret_cast<const __half2 *>(&p[b]), j < 2 ? s_lo : s_hi);
            if (F16OUT) {
                o[4 * j + b] = *reinterpret_cast<const uint32_t *>(&v);
            } else {
                const __nv_bfloat162 bv = __float22bfloat162_rn(__half22float2(v));
                o[4 * j + b] = *reinterpret_cast<const uint32_t *>(&bv);
            }
        }
    }
}

template <bool FP4, bool STACK>
__global__ void __launch_bounds__(Cfg<FP4>::kThreads, 1)
    decode_mma_kernel(const __grid_constant__ MArgs a, const __grid_constant__ TMaps maps0) {
    using C = Cfg<FP4>;
    constexpr int kThreads = C::kThreads, kWarps = C::kWarps;
    extern __shared__ __align__(1024) unsigned char smem_raw[];
    const uint32_t base_u32 = smem_u32(smem_raw);
    unsigned char *smem = smem_raw + (((base_u32 + 1023u) & ~1023u) - base_u32);
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int d = a.d, I = a.I, E = a.E, k = a.k, T = a.T, NS = a.nslots;
    const int G = gridDim.x, b = blockIdx.x;
    uint32_t *err = &a.ws.ctrl->err;
    Control *ctrl = a.ws.ctrl;

    // ---- shared-memory layout ----
    uint64_t *full = reinterpret_cast<uint64_t *>(smem);          // [32]
    uint64_t *empty = full + kMaxSlots;                            // [32]
    uint64_t *afull = empty + kMaxSlots;                           // [4]
    uint64_t *aempty = afull + kNA;                                // [4]
    uint64_t *accfull = aempty + kNA;                              // [4]
    uint64_t *accempty = accfull + kNAcc;                          // [4]
    uint64_t *xfull = accempty + kNAcc;                            // exchange of the up values
    uint64_t *xempty = xfull + 1;
    uint64_t *done = xempty + 1;
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(smem + 768);
    volatile int *abort_flag = reinterpret_cast<volatile int *>(smem + 772);
    uint32_t *hbase = reinterpret_cast<uint32_t *>(smem + 776);    // [2]
    int *cb_rows_s = reinterpret_cast<int *>(smem + 1024);         // [32]
    int *cb_todo = cb_rows_s + 32;                                 // [32]
    int *n_todo = cb_todo + 32;
    float *part = reinterpret_cast<float *>(smem + 2048);          // [8 warps][16] router partials
    unsigned char *rbase = smem + 3072;                            // routing scratch (8 KB)
    fused::Route R;
    R.cnt = reinterpret_cast<int32_t *>(rbase);
    R.off = R.cnt + 260;
    R.uniq = R.off + 260;
    R.scan = R.uniq + 260;
    R.bm = reinterpret_cast<uint32_t *>(R.scan + 260);
    R.ids = reinterpret_cast<int32_t *>(R.bm + 256);
    R.pos = R.ids + 128;
    R.perm = R.pos + 128;
    R.w = reinterpret_cast<float *>(R.perm + 128);
    R.wsum = reinterpret_cast<uint32_t *>(R.w + 128);
    R.n_uniq = reinterpret_cast<int *>(smem + 784);
    float *xch = reinterpret_cast<float *>(smem + 11264);          // [64 rows][16] up values (4 KB)
    unsigned char *ring = smem + kFixed;
    uint16_t *xs = reinterpret_cast<uint16_t *>(ring);             // prologue: the layer's token rows (bf16)

    if (tid == 0) {
        for (int s = 0; s < NS; ++s) {
            mbar_init(&full[s], 1);
            mbar_init(&empty[s], 1 + C::kConvWarps / kConvGroups);   // the MMA's commit + the converting group's warps
        }
        for (int s = 0; s < kNA; ++s) {
            mbar_init(&afull[s], C::kConvWarps > 0 ? C::kConvWarps / kConvGroups : 1);
            mbar_init(&aempty[s], 1);
        }
        for (int s = 0; s < kNAcc; ++s) {
            mbar_init(&accfull[s], 1);
            mbar_init(&accempty[s], 128);
        }
        mbar_init(xfull, 64);
        mbar_init(xempty, 64);
        mbar_init(done, 1);
        *abort_flag = 0;
        hbase[0] = hbase[1] = 0u;
        fence_barrier_init();
    }
    for (int i = tid; i < 32; i += kThreads) cb_rows_s[i] = 0;
    if (warp == 1) tmem_alloc(tmem_slot, (uint32_t)a.tmem_cols);
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem_base = *tmem_slot;

    // running counters of the pipelines (they continue across stacked layers)
    int it_prod = 0, it_conv = 0, it_mma = 0;
    int un_mma = 0, un_epi = 0, gu_epi = 0;

    for (int layer = 0; layer < (STACK ? a.n_layers : 1); ++layer) {
        const LayerW &lw = STACK ? a.ws.stack[layer] : a.lw0;
        const TMaps &mp = STACK ? a.stack_maps[layer] : maps0;
        const uint16_t *xin = STACK ? (layer > 0 ? a.out : a.x) : a.x;

        // ---- 1a. the layer's tokens into shared memory (bf16), and the B rows ----
        if (STACK) {
            // RMSNorm(x_l) with moe_rmsnorm's arithmetic: 256 threads (warps
            // 0-7), 8 elements each per 2048 columns, fp32 squares, warp sums,
            // the 8 warps' sums in order
            if (warp < 8) {
                for (int t = 0; t < T; ++t) {
                    float ss = 0.f;
                    for (int c = tid * 8; c < d; c += 256 * 8) {
                        const uint4 v = __ldcg(reinterpret_cast<const uint4 *>(xin + (size_t)t * d + c));
                        const uint32_t wv[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
                        for (int i = 0; i < 4; ++i) {
                            const float lo = bf16lo(wv[i]), hi = bf16hi(wv[i]);
                            ss = fmaf(lo, lo, ss);
                            ss = fmaf(hi, hi, ss);
                        }
                    }
                    const float ws_ = warp_sum(ss);
                    if (lane == 0) part[warp * 16 + t] = ws_;
                }
            }
            __syncthreads();
            if (warp < 8) {
                for (int t = 0; t < T; ++t) {
                    float tot = 0.f;
#pragma unroll
                    for (int i = 0; i < 8; ++i) tot += part[i * 16 + t];
                    const float rn = 1.0f / sqrtf(tot / (float)d + a.eps);
                    for (int c = tid * 8; c < d; c += 256 * 8) {
                        const uint4 v = __ldcg(reinterpret_cast<const uint4 *>(xin + (size_t)t * d + c));
                        const uint32_t wv[4] = {v.x, v.y, v.z, v.w};
                        uint32_t o[4];
#pragma unroll
                        for (int i = 0; i < 4; ++i)
                            o[i] = (uint32_t)f32_to_bf16_rn(bf16lo(wv[i]) * rn) |
                                   ((uint32_t)f32_to_bf16_rn(bf16hi(wv[i]) * rn) << 16);
                        *reinterpret_cast<uint4 *>(xs + (size_t)t * d + c) = make_uint4(o[0], o[1], o[2], o[3]);
                    }
                }
            }
        } else {
            for (int i = tid; i < T * (d / 8); i += kThreads)
                reinterpret_cast<uint4 *>(xs)[i] = __ldg(reinterpret_cast<const uint4 *>(a.x) + i);
        }
        __syncthreads();
        // CTA t < 16 writes B row t: the token (bf16), or f16 scaled by a power
        // of two 2^-p >= 1/max|x_t| (NVFP4); zeros for t >= T
        if (b < kN) {
            uint16_t *dst = a.xb + (size_t)b * d;
            if (b >= T) {
                for (int i = tid; i < d / 8; i += kThreads) reinterpret_cast<uint4 *>(dst)[i] = make_uint4(0, 0, 0, 0);
            } else if (!FP4) {
                for (int i = tid; i < d / 8; i += kThreads)
                    reinterpret_cast<uint4 *>(dst)[i] = reinterpret_cast<const uint4 *>(xs + (size_t)b * d)[i];
            } else {
                float m = 0.f;
                for (int i = tid; i < d / 2; i += kThreads) {
                    const uint32_t wv = reinterpret_cast<const uint32_t *>(xs + (size_t)b * d)[i];
                    m = fmaxf(m, fmaxf(fabsf(bf16lo(wv)), fabsf(bf16hi(wv))));
                }
                m = fmaxf(m, __shfl_xor_sync(0xFFFFFFFFu, m, 16));
                m = fmaxf(m, __shfl_xor_sync(0xFFFFFFFFu, m, 8));
                m = fmaxf(m, __shfl_xor_sync(0xFFFFFFFFu, m, 4));
                m = fmaxf(m, __shfl_xor_sync(0xFFFFFFFFu, m, 2));
                m = fmaxf(m, __shfl_xor_sync(0xFFFFFFFFu, m, 1));
                if (lane == 0) part[128 + warp] = m;
                __syncthreads();
                m = 0.f;
                for (int i = 0; i < kWarps; ++i) m = fmaxf(m, part[128 + i]);
                int ex = 0;
                if (m > 0.f) frexpf(m, &ex);
                const float inv = ldexpf(1.f, -ex);
                if (tid == 0) a.xscale[b] = ldexpf(1.f, ex);
                for (int i = tid; i < d / 2; i += kThreads) {
                    const uint32_t wv = reinterpret_cast<const uint32_t *>(xs + (size_t)b * d)[i];
                    const __half2 hv = __floats2half2_rn(bf16lo(wv) * inv, bf16hi(wv) * inv);
                    reinterpret_cast<uint32_t *>(dst)[i] = *reinterpret_cast<const uint32_t *>(&hv);
                }
            }
            // the rows are read by TMA (the async proxy) after the grid barrier
            fence_proxy_async_global();
        }

        // ---- 1b. router: logits of experts b, b + G (warps 0-3 / 4-7 take the quarters of one row) ----
        {
            const int nq = d / 32;
            for (int base = b; base < E; base += 2 * G) {
                const int eidx = base + (warp >= 4 ? G : 0);
                const int q = warp & 3;
                float acc[kN];
#pragma unroll
                for (int t = 0; t < kN; ++t) acc[t] = 0.f;
                const bool mine = warp < 8 && eidx < E;
                if (mine) {
                    const uint4 *wrow = reinterpret_cast<const uint4 *>(lw.wr + (size_t)eidx * d) + q * nq;
                    for (int v = lane; v < nq; v += 32) {
                        const uint4 wv = __ldg(wrow + v);
#pragma unroll
                        for (int t = 0; t < kN; ++t) {
                            if (t < T) {
                                const uint4 xv = reinterpret_cast<const uint4 *>(xs + (size_t)t * d)[q * nq + v];
                                float2 s2 = make_float2(0.f, 0.f);
                                s2 = __ffma2_rn(make_float2(bf16lo(wv.x), bf16hi(wv.x)), make_float2(bf16lo(xv.x), bf16hi(xv.x)), s2);
                                s2 = __ffma2_rn(make_float2(bf16lo(wv.y), bf16hi(wv.y)), make_float2(bf16lo(xv.y), bf16hi(xv.y)), s2);
                                s2 = __ffma2_rn(make_float2(bf16lo(wv.z), bf16hi(wv.z)), make_float2(bf16lo(xv.z), bf16hi(xv.z)), s2);
                                s2 = __ffma2_rn(make_float2(bf16lo(wv.w), bf16hi(wv.w)), make_float2(bf16lo(xv.w), bf16hi(xv.w)), s2);
                                acc[t] += s2.x + s2.y;
                            }
                        }
                    }
                }
#pragma unroll
                for (int t = 0; t < kN; ++t) {
                    const float s = warp_sum(acc[t]);
                    if (lane == 0 && warp < 8) part[warp * kN + t] = s;
                }
                __syncthreads();
                if (tid < 2 * kN) {
                    const int half = tid / kN, t = tid % kN;
                    const int e2 = base + half * G;
                    if (e2 < E && t < T) {
                        const float *pp = part + half * 4 * kN;
                        float l = ((pp[0 * kN + t] + pp[1 * kN + t]) + pp[2 * kN + t]) + pp[3 * kN + t];
                        if (lw.bias) l += lw.bias[e2];
                        a.ws.logits[(size_t)t * E + e2] = l;
                    }
                }
                __syncthreads();
            }
        }
        fused::grid_barrier(&ctrl->grid_bar.v, (uint32_t)(2 * layer + 1) * G, err, abort_flag, &ctrl->test_hold);

        // ---- 2. routing, in every CTA ----
        fused::route_tokens(R, a.ws.logits, nullptr, 0u, T, k, E, err, abort_flag);
        const int n_uniq = *R.n_uniq;
        if (b == 0) fused::publish_records(R, a.ws, T, k, E, n_uniq, kThreads);
        const fused::Plan pl = fused::make_plan_rotated(n_uniq, I / kGu, d / kDn, b, G);
        const int n_gu = pl.nA + pl.nB;
        const int n_units = n_gu + pl.nC + pl.nD;
        const int U1 = (n_uniq + 1) / 2;
        // the ring's prologue use (token rows) is over once every warp passed here
        __syncthreads();

        if (warp == 0) {
            // ------------------------------- TMA producer -------------------------------
            if (lane == 0) {
                bool ok = !*abort_flag;
                fence_proxy_async_global();   // the token rows other CTAs wrote, read by TMA below
                for (int n = 0; n < n_units && ok; ++n) {
                    const Unit un = unit_at(pl, R, n, n_gu, d, I);
                    // entering a half's down units (the first of either segment;
                    // a CTA may have none of the first half's): wait for that
                    // half's h rows, written by every CTA's epilogue
                    const int t_dn = n - n_gu;
                    if (!un.gu && (t_dn == 0 || t_dn == pl.nC)) {
                        const int half = t_dn < pl.nC ? 0 : 1;
                        const uint32_t target = hbase[half] + (uint32_t)((half ? n_uniq - U1 : U1) * I);
                        const unsigned long long t0 = global_ns();
                        while (fused::ld_acquire(&ctrl->h_ready[half].v) < target) {
                            if (*abort_flag || global_ns() - t0 > kWaitLimitNs) {
                                atomicOr(err, ERRBIT_TIMEOUT);
                                *abort_flag = 1;
                                ok = false;
                                break;
                            }
                        }
                        if (!ok) break;
                        fence_proxy_async_global();   // h is read by TMA below
                    }
                    const int row0 = R.off[un.e];
                    for (int kb = 0; kb < un.kbs; ++kb, ++it_prod) {
                        const int slot = it_prod % NS;
                        if (!mbar_wait_or_abort(&empty[slot], ((it_prod / NS) & 1) ^ 1, err, abort_flag)) {
                            ok = false;
                            break;
                        }
                        unsigned char *st = ring + (size_t)slot * C::kStage;
                        mbar_arrive_expect_tx(&full[slot], C::kStage);
                        if (un.gu) {
                            const int wrow = un.e * I + un.row;
                            tma_load_2d(st, &mp.m[6], kb * 64, 0, &full[slot]);
                            if (!FP4) {
                                tma_load_2d(st + C::kB, &mp.m[0], kb * 64, wrow, &full[slot]);
                                tma_load_2d(st + C::kB + 64 * 128, &mp.m[1], kb * 64, wrow, &full[slot]);
                            } else {
                                unsigned char *codes = st + C::kB, *scales = codes + 128 * 32;
                                tma_load_2d(codes, &mp.m[0], kb * 32, wrow, &full[slot]);
                                tma_load_2d(codes + 64 * 32, &mp.m[1], kb * 32, wrow, &full[slot]);
                                tma_load_2d(scales, &mp.m[3], (kb >> 2) * 16, wrow, &full[slot]);
                                tma_load_2d(scales + 64 * 16, &mp.m[4], (kb >> 2) * 16, wrow, &full[slot]);
                            }
                        } else {
                            const int wrow = un.e * d + un.row;
                            tma_load_2d(st, &mp.m[7], kb * 64, row0, &full[slot]);
                            if (!FP4) {
                                tma_load_2d(st + C::kB, &mp.m[2], kb * 64, wrow, &full[slot]);
                            } else {
                                unsigned char *codes = st + C::kB, *scales = codes + 128 * 32;
                                tma_load_2d(codes, &mp.m[2], kb * 32, wrow, &full[slot]);
                                tma_load_2d(scales, &mp.m[5], (kb >> 2) * 16, wrow, &full[slot]);
                            }
                        }
                    }
                }
                if (STACK && layer + 1 < a.n_layers) fused::prefetch_next_router(a.ws.stack[layer + 1], b, G, E, d);
            }
        } else if (warp == 1) {
            // -------------------------------- MMA issuer --------------------------------
            if (lane == 0) {
                bool ok = !*abort_flag;
                for (int n = 0; n < n_units && ok; ++n, ++un_mma) {
                    const Unit un = unit_at(pl, R, n, n_gu, d, I);
                    const int ab = un_mma % kNAcc;
                    if (!mbar_wait_or_abort(&accempty[ab], ((un_mma / kNAcc) & 1) ^ 1, err, abort_flag)) break;
                    tc_fence_after();
                    const uint32_t idesc = (FP4 && un.gu) ? kIdescF16 : kIdescBf16;
                    for (int kb = 0; kb < un.kbs; ++kb, ++it_mma) {
                        // partial accumulator kb % kKSplit of unit buffer ab; its first k-block overwrites
                        const uint32_t dtm = tmem_base + (uint32_t)((ab * C::kKSplit + kb % C::kKSplit) * kN);
                        const bool first = kb < C::kKSplit;
                        const int slot = it_mma % NS, as = it_mma % kNA;
                        if (!mbar_wait_or_abort(&full[slot], (it_mma / NS) & 1, err, abort_flag) ||
                            (FP4 && !mbar_wait_or_abort(&afull[as], (it_mma / kNA) & 1, err, abort_flag))) {
                            ok = false;
                            break;
                        }
                        tc_fence_after();
                        const unsigned char *st = ring + (size_t)slot * C::kStage;
                        const uint64_t bd = smem_desc_sw128(smem_u32(st));
                        if (!FP4) {
                            const uint64_t ad = smem_desc_sw128(smem_u32(st + C::kB));
#pragma unroll
                            for (int kk = 0; kk < 4; ++kk)
                                mma_bf16(dtm, ad + (uint64_t)(2 * kk), bd + (uint64_t)(2 * kk), idesc, !first || kk != 0);
                        } else {
                            const uint32_t ta = tmem_base + (uint32_t)(C::kAColBase + as * 32);
#pragma unroll
                            for (int kk = 0; kk < 4; ++kk)
                                mma_tmem_a(dtm, ta + (uint32_t)(8 * kk), bd + (uint64_t)(2 * kk), idesc, !first || kk != 0);
                        }
                        mma_commit(&empty[slot]);             // slot free once these MMAs have read it
                        if (FP4) mma_commit(&aempty[as]);     // and the widened A tile
                    }
                    if (!ok) break;
                    mma_commit(&accfull[ab]);
                }
            }
        } else if (warp < 6) {
            // --------------------------------- epilogue ---------------------------------
            const int q = warp & 3;              // TMEM lane quarter
            const int r128 = q * 32 + lane;      // A row this thread owns
            bool ok = !*abort_flag;
            int done_a = 0, done_b = 0;   // gate warps: h rows written, per half
            for (int n = 0; n < n_units && ok; ++n, ++un_epi) {
                const Unit un = unit_at(pl, R, n, n_gu, d, I);
                const int ab = un_epi % kNAcc;
                if (!mbar_wait_or_abort(&accfull[ab], (un_epi / kNAcc) & 1, err, abort_flag)) break;
                tc_fence_after();
                uint32_t v[16];
                {
                    // the unit's partial accumulators (as many as it had k-blocks, up to kKSplit), added
                    const uint32_t tl = tmem_base + ((uint32_t)(q * 32) << 16) + (uint32_t)(ab * C::kKSplit * kN);
                    tmem_ld16(tl, v);
                    tmem_ld_wait();
                    const int parts = un.kbs < C::kKSplit ? un.kbs : C::kKSplit;
                    for (int pp = 1; pp < parts; ++pp) {
                        uint32_t w[16];
                        tmem_ld16(tl + (uint32_t)(pp * kN), w);
                        tmem_ld_wait();
#pragma unroll
                        for (int t = 0; t < kN; ++t) v[t] = __float_as_uint(__uint_as_float(v[t]) + __uint_as_float(w[t]));
                    }
                }
                tc_fence_before();
                mbar_arrive(&accempty[ab]);
                const int n_e = R.cnt[un.e] < kN ? R.cnt[un.e] : kN;
                const int row0 = R.off[un.e];
                if (un.gu) {
                    // rows 0-63 gate (quarters 0, 1), rows 64-127 up (quarters 2, 3)
                    const int par = gu_epi & 1;
                    ++gu_epi;
                    if (q >= 2) {
                        if (!mbar_wait_or_abort(xempty, par ^ 1, err, abort_flag)) break;
#pragma unroll
                        for (int t = 0; t < kN; ++t) xch[(r128 - 64) * kN + t] = __uint_as_float(v[t]);
                        mbar_arrive(xfull);
                    } else {
                        if (!mbar_wait_or_abort(xfull, par, err, abort_flag)) break;
                        float uv[kN];
#pragma unroll
                        for (int t = 0; t < kN; ++t) uv[t] = xch[r128 * kN + t];
                        mbar_arrive(xempty);
                        const float gsc = FP4 ? lw.gg[un.e] : 1.f, usc = FP4 ? lw.gu[un.e] : 1.f;
                        uint16_t *hb = reinterpret_cast<uint16_t *>(a.ws.h);
                        for (int r = 0; r < n_e; ++r) {
                            const int t = R.perm[row0 + r];
                            float g = 0.f, u = 0.f;
#pragma unroll
                            for (int tt = 0; tt < kN; ++tt)
                                if (tt == t) {
                                    g = __uint_as_float(v[tt]);
                                    u = uv[tt];
                                }
                            if (FP4) {
                                const float xs_ = a.xscale[t];
                                g *= xs_ * gsc;
                                u *= xs_ * usc;
                            }
                            hb[(size_t)(row0 + r) * I + un.row + r128] = f32_to_bf16_rn(silu(g) * u);
                        }
                        if (n < pl.nA)
                            done_a += 32;
                        else
                            done_b += 32;
                        // count this warp's h rows in once its share of a half is written
                        // (other CTAs' TMA loads read them: proxy fence first)
                        if (n + 1 == pl.nA || n + 1 == n_gu) {
                            fence_proxy_async_global();
                            fused::publish_rows(&ctrl->h_ready[n < pl.nA ? 0 : 1].v, n < pl.nA ? done_a : done_b);
                        }
                    }
                } else {
                    const float gsc = FP4 ? lw.gd[un.e] : 1.f;
                    const int c = un.row + r128;
                    for (int r = 0; r < n_e; ++r) {
                        float y = 0.f;
#pragma unroll
                        for (int tt = 0; tt < kN; ++tt)
                            if (tt == r) y = __uint_as_float(v[tt]);
                        a.ws.Y[(size_t)(row0 + r) * d + c] = y * gsc;
                    }
                    __syncwarp();
                    if (lane == 0) atomicAdd(&cb_rows_s[un.row / kCb], 32);
                }
            }
        } else if (FP4) {
            // -------------------------------- converters --------------------------------
            // group g (4 warps, one per TMEM lane quarter) widens the k-blocks
            // it with it % 2 == g: two k-blocks are in conversion at once
            const int q = warp & 3;                    // TMEM lane quarter
            const int grp = (warp - 6) >> 2;
            const int row = q * 32 + lane;             // A row
            bool ok = !*abort_flag;
            for (int n = 0; n < n_units && ok; ++n) {
                const Unit un = unit_at(pl, R, n, n_gu, d, I);
                for (int kb = 0; kb < un.kbs; ++kb, ++it_conv) {
                    if ((it_conv % kConvGroups) != grp) continue;
                    const int slot = it_conv % NS, as = it_conv % kNA;
                    if (!mbar_wait_or_abort(&full[slot], (it_conv / NS) & 1, err, abort_flag) ||
                        !mbar_wait_or_abort(&aempty[as], ((it_conv / kNA) & 1) ^ 1, err, abort_flag)) {
                        ok = false;
                        break;
                    }
                    const unsigned char *st = ring + (size_t)slot * C::kStage;
                    const unsigned char *codes = st + C::kB + row * 32;
                    const unsigned char *scales = st + C::kB + 128 * 32 + row * 16 + (kb & 3) * 4;
                    uint32_t o[32];
                    if (un.gu) {
                        widen32<true>(codes, scales, o);
                        widen32<true>(codes + 16, scales + 2, o + 16);
                    } else {
                        widen32<false>(codes, scales, o);
                        widen32<false>(codes + 16, scales + 2, o + 16);
                    }
                    tc_fence_after();
                    const uint32_t ta = tmem_base + ((uint32_t)(q * 32) << 16) + (uint32_t)(C::kAColBase + as * 32);
                    tmem_st16(ta, o);
                    tmem_st16(ta + 16, o + 16);
                    tmem_st_wait();
                    tc_fence_before();
                    __syncwarp();
                    if (lane == 0) {
                        mbar_arrive(&afull[as]);
                        mbar_arrive(&empty[slot]);
                    }
                }
            }
        }

        // ---- 4. combine, by the CTA that completes each column block ----
        fence_acq_rel_gpu();  // this thread's Y stores before the block's count below
        __syncthreads();
        if (warp == 0) {
            const int ncb = (d + kCb - 1) / kCb;
            bool fin = false;
            fence_acq_rel_gpu();
            if (lane < ncb) {
                const int mine = cb_rows_s[lane];
                if (mine) {
                    const int cols = min(kCb, d - lane * kCb);
                    const uint32_t dn = atomicAdd(&ctrl->cb_rows[lane].v, (uint32_t)mine) + mine;
                    fin = dn == (uint32_t)(n_uniq * cols);
                }
            }
            fence_acq_rel_gpu();
            const uint32_t fin_mask = __ballot_sync(0xFFFFFFFFu, fin);
            if (lane == 0) {
                int nn = 0;
                for (uint32_t m = fin_mask; m; m &= m - 1) cb_todo[nn++] = __ffs(m) - 1;
                *n_todo = nn;
            }
            if (lane < 32) cb_rows_s[lane] = 0;
        }
        __syncthreads();
        for (int ti = 0; ti < *n_todo; ++ti) {
            const int cb = cb_todo[ti];
            const int cols = min(kCb, d - cb * kCb);
            for (int idx = tid; idx < T * (cols / 4); idx += kThreads) {
                const int t = idx / (cols / 4);
                const int c = cb * kCb + (idx % (cols / 4)) * 4;
                float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
                for (int j = 0; j < k; ++j) {
                    const float wj = R.w[t * k + j];
                    const float4 y = __ldcg(reinterpret_cast<const float4 *>(a.ws.Y + (size_t)R.pos[t * k + j] * d + c));
                    acc.x = fmaf(wj, y.x, acc.x);
                    acc.y = fmaf(wj, y.y, acc.y);
                    acc.z = fmaf(wj, y.z, acc.z);
                    acc.w = fmaf(wj, y.w, acc.w);
                }
                const uint16_t *resid = STACK ? xin : a.res;
                if (resid) {
                    const uint2 rv = *reinterpret_cast<const uint2 *>(resid + (size_t)t * d + c);
                    acc.x += bf16lo(rv.x);
                    acc.y += bf16hi(rv.x);
                    acc.z += bf16lo(rv.y);
                    acc.w += bf16hi(rv.y);
                }
                uint2 o;
                o.x = (uint32_t)f32_to_bf16_rn(acc.x) | ((uint32_t)f32_to_bf16_rn(acc.y) << 16);
                o.y = (uint32_t)f32_to_bf16_rn(acc.z) | ((uint32_t)f32_to_bf16_rn(acc.w) << 16);
                *reinterpret_cast<uint2 *>(a.out + (size_t)t * d + c) = o;
                if (STACK && a.layer_out) *reinterpret_cast<uint2 *>(a.layer_out + ((size_t)layer * T + t) * d + c) = o;
            }
            if (tid == 0) ctrl->cb_rows[cb].v = 0u;
        }
        if (STACK && layer + 1 < a.n_layers) {
            if (tid == 0) {
                hbase[0] += (uint32_t)(U1 * I);
                hbase[1] += (uint32_t)((n_uniq - U1) * I);
            }
            fused::grid_barrier(&ctrl->grid_bar.v, (uint32_t)(2 * layer + 2) * G, err, abort_flag, &ctrl->test_hold);
        }
    }  // layers

    // ---- exit: wait for the MMAs and the producer's last copies, free TMEM,
    // the last CTA out resets the counters ----
    if (warp == 1 && lane == 0) {
        mma_commit(done);           // completes once every MMA issued above has
        mbar_wait(done, 0, err);    // (an aborted launch may leave some in flight)
    }
    if (warp == 0 && lane == 0) {
        for (int j = it_prod > NS ? it_prod - NS : 0; j < it_prod; ++j) mbar_wait(&full[j % NS], (j / NS) & 1, err);
    }
    tc_fence_before();
    __syncthreads();
    if (warp == 1) {
        tc_fence_after();
        tmem_dealloc(tmem_base, (uint32_t)a.tmem_cols);
    }
    if (tid == 0) {
        fence_acq_rel_gpu();
        if (atomicAdd(&ctrl->grid_exit.v, 1u) == (uint32_t)G - 1) {
            for (int cb = 0; cb < 32; ++cb) ctrl->cb_rows[cb].v = 0u;
            ctrl->grid_bar.v = 0u;
            ctrl->h_ready[0].v = 0u;
            ctrl->h_ready[1].v = 0u;
            ctrl->grid_exit.v = 0u;
            fence_acq_rel_gpu();
        }
    }
}

}  // namespace dmma

}  // namespace moe
