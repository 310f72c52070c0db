// decode_fused.cuh — one persistent kernel for a whole small-batch (T <= 16)
// MoE layer: router, softmax/top-k/renormalise, permutation, the expert
// weight stream through gate/up and down, and the weighted combine.
//
// Decode is bound by streaming weights from HBM and by the boundaries
// between kernels, which break the overlap of weight streaming and compute
// ("How SGLang-TorchTPU accelerated an 816B-parameter MoE on TPU v7",
// sections "Introduction" and "Key optimisations"). Here the layer is one
// cooperative launch, one CTA per SM:
//   1. router: every CTA computes the logits of its experts (x . Wr[e]) and
//      stores each as one 64-bit word with the layer's tag;
//   2. routing: every CTA reads all logits, waiting for each word's tag (no
//      grid barrier: the tag is the hand-off), and computes top-k and the
//      permutation of all T tokens itself, in shared memory (identical
//      results everywhere; CTA 0 also publishes them);
//   3. producer lanes (polling, never blocking) fill a ring of shared-memory
//      slots with bulk TMA copies: first this CTA's share of the active
//      experts' gate/up rows, then, without a pause, its share of their down
//      rows (shares cut by cost when experts carry several tokens); slot j
//      belongs to consumer warp j % c, which takes the slot's phases in order;
//   4. consumer warps compute h = silu(Wg x) * (Wu x) (fp32, to global) and
//      count the rows in, per half of the active experts; the stream runs
//      first-half gate/up, second-half gate/up, first-half down, second-half
//      down, so a half's h is complete long before its down rows arrive and
//      the weight stream never pauses; then Y = Wd h (fp32, to global);
//   5. combine: per 256-column block of the output, the CTA whose down rows
//      complete the block (a row counter per block) forms
//      out = (res +) sum_j w_j Y_j for those columns, in fp32, j ascending.
// Every wait (mbarrier, tag, h count, grid barrier) is bounded; a timeout
// sets the error word and the kernel unwinds. The tags: the control block's
// epoch, read at entry, gives layer l the tag epoch + 1 + l, and the last CTA
// out advances the epoch by the launch's layer count, so no word left by an
// earlier launch carries a tag a later one waits for (every launch rewrites
// all 16 rows; set-up clears the words and the epoch together). With STACK the kernel loops over layers
// (decode_stack.cu): each layer's input is RMSNorm of the previous output,
// computed in every CTA, and a grid barrier separates the layers.
#pragma once

#include <cuda_fp4.h>
#include <cuda_fp8.h>
#include <cuda_runtime.h>

#include "common.cuh"
#include "decode_common.cuh"

namespace moe {

namespace fused {

// Warps per CTA: 7 consumers and the producer. Registers are handed out per
// group of four warps, so a CTA of 4n warps wastes none; a 9-warp CTA would be
// charged for 12 (capping a thread at 168 registers). (12-warp NVFP4 CTAs
// were measured slower: fewer ring slots per consumer and fewer producer lanes.)
template <int TM, bool FP4>
struct Warps {
    static constexpr int kWarps = 8;
    static constexpr int kThreads = 32 * kWarps;
    static constexpr int kConsumers = kWarps - 1;   // consumer warps at most
    static constexpr int kProducerWarp = kWarps - 1;
};
constexpr int kDnRows = 4;                    // down rows per stage
constexpr int kMaxSlots = 32;
constexpr int kSmemBudget = 227 * 1024;
constexpr int kCb = 256;                      // output columns per combine block
constexpr int kTagRows = 16;                  // token rows of the tagged logits (every row, every layer)

struct Args {
    const uint16_t *x;        // [T, d] bf16 (stacked: the first layer's input)
    const uint16_t *res;      // [T, d] bf16 or null (single layer)
    uint16_t *out;            // [T, d] bf16
    LayerW lw0;               // the layer's weights (single layer)
    int n_layers;             // 0: one layer (lw0); n > 0: n stacked layers, weights in ws.stack,
                              // layer l's input RMSNorm(x_l) (eps), its residual x_l, x_{l+1} in out
    float eps;
    uint16_t *layer_out;      // stacked: [n_layers, T, d] copy of every layer's output, or null
    int T, d, I, E, k;
    int nslots, ncons, nprod;
    uint32_t slot_bytes;
    int x_in_smem;            // tokens' rows staged in shared memory
    int x_router_ring;        // no room for that: the router reads them from the (still idle) ring
    int do_combine;           // 0: leave Y for a separate combine kernel
    Workspace ws;
};

template <bool FP4>
__host__ __device__ constexpr uint32_t rowb(int K) {
    return FP4 ? (uint32_t)K / 2 + (uint32_t)K / 16 : (uint32_t)K * 2;
}

// ---------------------------------------------------------------------------
// small helpers
// ---------------------------------------------------------------------------
__device__ __forceinline__ float2 bf2(uint32_t w) { return make_float2(bf16lo(w), bf16hi(w)); }

__device__ __forceinline__ float2 ffma2(float2 a, float2 b, float2 c) { return __ffma2_rn(a, b, c); }

__device__ __forceinline__ void fp4x16(uint2 q, float2 f[8]) {
    const uint32_t words[2] = {q.x, q.y};
#pragma unroll
    for (int wi = 0; wi < 2; ++wi) {
        uint32_t o[4];
        e2m1x8_to_f16x2(words[wi], o);
#pragma unroll
        for (int b = 0; b < 4; ++b) f[wi * 4 + b] = __half22float2(*reinterpret_cast<const __half2 *>(&o[b]));
    }
}

// Sixteen E2M1 codes (8 bytes) to eight f16 pairs.
__device__ __forceinline__ void fp4x16_h2(uint2 q, __half2 h[8]) {
    uint32_t o[8];
    e2m1x8_to_f16x2(q.x, o);
    e2m1x8_to_f16x2(q.y, o + 4);
#pragma unroll
    for (int b = 0; b < 8; ++b) h[b] = *reinterpret_cast<const __half2 *>(&o[b]);
}

__device__ __forceinline__ float e4m3f(uint8_t s) {
    __half_raw hr = __nv_cvt_fp8_to_halfraw((__nv_fp8_storage_t)s, __NV_E4M3);
    return __half2float(*reinterpret_cast<__half *>(&hr));
}

// Index, within a segment of experts [u_lo, u_hi) holding `per` stages each,
// where CTA bb's share starts when the segment is cut into G parts of equal
// total weight (bb = G gives the segment's end). cw: exclusive prefix over
// experts of one stage's weight. A stage of an expert with n tokens weighs n:
// every stage streams the same bytes, but in a multi-token batch the
// arithmetic, which grows with the tokens, sets the pace (measured at 4 and
// 16 tokens, stage costs 2 + n, 1 + n, 1 + 2n, n and 3n tried: n balances
// best). So cw is the prefix of the experts' token counts, which the routing
// leaves in R.scan.
__device__ __forceinline__ int weighted_start(const int32_t *cw, int u_lo, int u_hi, int per, int bb, int G) {
    if (u_hi <= u_lo) return 0;
    if (bb >= G) return (u_hi - u_lo) * per;
    const long long base = cw[u_lo];
    const long long t = div_u((long long)(cw[u_hi] - base) * per * bb, G);
    int lo = u_lo, hi = u_hi;  // the expert holding weight position t
    while (hi - lo > 1) {
        const int mid = (lo + hi) >> 1;
        if ((long long)(cw[mid] - base) * per <= t)
            lo = mid;
        else
            hi = mid;
    }
    const long long w = cw[lo + 1] - cw[lo];
    const long long j = div_u(t - (long long)(cw[lo] - base) * per + w - 1, (int)w);
    return (lo - u_lo) * per + (int)(j < per ? j : per);
}

// Sums of four rows' per-lane partials (one token), reduced together:
// exchanging halves, lane group q (lanes 8q .. 8q+7) ends with row q, and its
// first lane stores y[q] = sum * scale.
__device__ __forceinline__ void store_four_rows(float r0, float r1, float r2, float r3, float *y, float scale) {
    const int lane = threadIdx.x & 31;
    const bool hi16 = lane & 16, hi8 = lane & 8;
    // lanes < 16 keep rows 0,1; lanes >= 16 keep rows 2,3
    float k0 = hi16 ? r2 : r0, k1 = hi16 ? r3 : r1;
    const float s0 = hi16 ? r0 : r2, s1 = hi16 ? r1 : r3;
    k0 += __shfl_xor_sync(0xFFFFFFFFu, s0, 16);
    k1 += __shfl_xor_sync(0xFFFFFFFFu, s1, 16);
    // within each half, lanes with bit 3 clear keep the first of the two rows
    float k = hi8 ? k1 : k0;
    k += __shfl_xor_sync(0xFFFFFFFFu, hi8 ? k0 : k1, 8);
    k += __shfl_xor_sync(0xFFFFFFFFu, k, 4);
    k += __shfl_xor_sync(0xFFFFFFFFu, k, 2);
    k += __shfl_xor_sync(0xFFFFFFFFu, k, 1);
    if ((lane & 7) == 0) y[lane >> 3] = k * scale;
}

// Per-warp cache of the expert a stage belongs to (read from shared memory).
template <int TM>
struct Seg {
    int u = -1, e = 0, n_e = 0, row0 = 0;
    int tok[TM];
};

template <int TM>
__device__ __forceinline__ void seg_load(Seg<TM> &s, const Route &R, int u) {
    s.u = u;
    if (TM == 1) {
        // one token (the routing leaves R.cnt / R.off to CTA 0): expert
        // uniq[u] holds row u
        s.e = R.uniq[u];
        s.n_e = 1;
        s.row0 = u;
        s.tok[0] = 0;
        return;
    }
    s.e = R.uniq[u];
    s.n_e = R.cnt[s.e] < TM ? R.cnt[s.e] : TM;
    s.row0 = R.off[s.e];
#pragma unroll
    for (int r = 0; r < TM; ++r) s.tok[r] = r < s.n_e ? R.perm[s.row0 + r] : 0;
}

// One gate/up stage (the row pair i of expert seg.e in `st`) for an expert
// with NE tokens at most (seg.n_e <= NE; exactly NE when NE <= 2): h rows of
// its tokens, h = silu(g) * u. Releases the slot once the stage is read.
template <int NE, int TM, bool FP4>
__device__ __forceinline__ void gu_stage(const Args &a, const LayerW &lw, const unsigned char *st,
                                         const unsigned char *xs, const float *xscale, const Seg<TM> &seg,
                                         uint64_t *empty_slot, int i) {
    const int lane = threadIdx.x & 31;
    const int d = a.d, I = a.I;
    const uint32_t rbg = rowb<FP4>(d);
    float2 ag[NE], au[NE];
#pragma unroll
    for (int r = 0; r < NE; ++r) ag[r] = au[r] = make_float2(0.f, 0.f);
    if (!FP4) {
        constexpr int kXV = 8;
        const uint4 *gw = reinterpret_cast<const uint4 *>(st);
        const uint4 *uw = reinterpret_cast<const uint4 *>(st + rbg);
        const int nvec = d / 8;
        if (a.x_in_smem) {
            // vector by vector: each weight vector is unpacked once and
            // used for every token of the expert
#pragma unroll 2
            for (int v = lane; v < nvec; v += 32) {
                const uint4 g4 = gw[v], u4 = uw[v];
                const float2 g0 = bf2(g4.x), g1 = bf2(g4.y), g2 = bf2(g4.z), g3 = bf2(g4.w);
                const float2 u0 = bf2(u4.x), u1 = bf2(u4.y), u2 = bf2(u4.z), u3 = bf2(u4.w);
#pragma unroll
                for (int r = 0; r < NE; ++r) {
                    if (NE <= 2 || r < seg.n_e) {
                        const uint4 xv = reinterpret_cast<const uint4 *>(xs + (size_t)seg.tok[r] * d * 2)[v];
                        const float2 x0 = bf2(xv.x), x1 = bf2(xv.y), x2 = bf2(xv.z), x3 = bf2(xv.w);
                        ag[r] = ffma2(g0, x0, ag[r]);
                        au[r] = ffma2(u0, x0, au[r]);
                        ag[r] = ffma2(g1, x1, ag[r]);
                        au[r] = ffma2(u1, x1, au[r]);
                        ag[r] = ffma2(g2, x2, ag[r]);
                        au[r] = ffma2(u2, x2, au[r]);
                        ag[r] = ffma2(g3, x3, ag[r]);
                        au[r] = ffma2(u3, x3, au[r]);
                    }
                }
            }
        } else {
        // token by token; each lane's vectors in chunks of kXV whose
        // token loads (from global memory) are all issued before the
        // arithmetic: one latency per chunk
#pragma unroll
        for (int r = 0; r < NE; ++r) {
            if (NE <= 2 || r < seg.n_e) {
                const uint4 *xrow = a.x_in_smem
                                        ? reinterpret_cast<const uint4 *>(xs + (size_t)seg.tok[r] * d * 2)
                                        : reinterpret_cast<const uint4 *>(a.x + (size_t)seg.tok[r] * d);
                for (int j0 = 0; j0 * 32 < nvec; j0 += kXV) {
                    uint4 xv[kXV];
#pragma unroll
                    for (int jj = 0; jj < kXV; ++jj) {
                        const int v = lane + 32 * (j0 + jj);
                        xv[jj] = v < nvec ? (a.x_in_smem ? xrow[v] : __ldg(xrow + v)) : make_uint4(0, 0, 0, 0);
                    }
#pragma unroll
                    for (int jj = 0; jj < kXV; ++jj) {
                        const int v = lane + 32 * (j0 + jj);
                        if (v < nvec) {
                            const uint4 g4 = gw[v], u4 = uw[v];
                            const float2 x0 = bf2(xv[jj].x), x1 = bf2(xv[jj].y), x2 = bf2(xv[jj].z),
                                         x3 = bf2(xv[jj].w);
                            ag[r] = ffma2(bf2(g4.x), x0, ag[r]);
                            au[r] = ffma2(bf2(u4.x), x0, au[r]);
                            ag[r] = ffma2(bf2(g4.y), x1, ag[r]);
                            au[r] = ffma2(bf2(u4.y), x1, au[r]);
                            ag[r] = ffma2(bf2(g4.z), x2, ag[r]);
                            au[r] = ffma2(bf2(u4.z), x2, au[r]);
                            ag[r] = ffma2(bf2(g4.w), x3, ag[r]);
                            au[r] = ffma2(bf2(u4.w), x3, au[r]);
                        }
                    }
                }
            }
        }
        }
    } else {
        const unsigned char *gq = st, *gs = st + d / 2, *uq = st + rbg, *us = st + rbg + d / 2;
        if (a.x_in_smem) {
            // tokens in shared memory as fp16(x / max|x|): the 16 products
            // of a block (|e2m1| <= 6, |x'| <= 1) are summed in fp16
            // pairs, scaled by the block scale into fp32 pair sums, and the
            // row's sum by max|x| at the end
            float xsc[NE];  // per-token max|x|
#pragma unroll
            for (int r = 0; r < NE; ++r) xsc[r] = (NE <= 2 || r < seg.n_e) ? xscale[seg.tok[r]] : 0.f;
#pragma unroll 2
            for (int bb = lane; bb < d / 16; bb += 32) {
                const uint2 gqv = *reinterpret_cast<const uint2 *>(gq + bb * 8);
                const uint2 uqv = *reinterpret_cast<const uint2 *>(uq + bb * 8);
                __half2 gh[8], uh[8];
                fp4x16_h2(gqv, gh);
                fp4x16_h2(uqv, uh);
                const float sgb = e4m3f(gs[bb]), sub = e4m3f(us[bb]);
#pragma unroll
                for (int r = 0; r < NE; ++r) {
                    if (NE <= 2 || r < seg.n_e) {
                        const uint4 *xp = reinterpret_cast<const uint4 *>(xs + (size_t)seg.tok[r] * d * 2) + bb * 2;
                        const uint4 xa = xp[0], xb = xp[1];
                        const uint32_t xw[8] = {xa.x, xa.y, xa.z, xa.w, xb.x, xb.y, xb.z, xb.w};
                        // two chains per matrix (even / odd pairs), joined at the end
                        __half2 pg0 = __hmul2(gh[0], *reinterpret_cast<const __half2 *>(&xw[0]));
                        __half2 pu0 = __hmul2(uh[0], *reinterpret_cast<const __half2 *>(&xw[0]));
                        __half2 pg1 = __hmul2(gh[1], *reinterpret_cast<const __half2 *>(&xw[1]));
                        __half2 pu1 = __hmul2(uh[1], *reinterpret_cast<const __half2 *>(&xw[1]));
#pragma unroll
                        for (int q = 2; q < 8; q += 2) {
                            pg0 = __hfma2(gh[q], *reinterpret_cast<const __half2 *>(&xw[q]), pg0);
                            pu0 = __hfma2(uh[q], *reinterpret_cast<const __half2 *>(&xw[q]), pu0);
                            pg1 = __hfma2(gh[q + 1], *reinterpret_cast<const __half2 *>(&xw[q + 1]), pg1);
                            pu1 = __hfma2(uh[q + 1], *reinterpret_cast<const __half2 *>(&xw[q + 1]), pu1);
                        }
                        const float2 fg = __half22float2(__hadd2(pg0, pg1)), fu = __half22float2(__hadd2(pu0, pu1));
                        ag[r] = ffma2(fg, make_float2(sgb, sgb), ag[r]);
                        au[r] = ffma2(fu, make_float2(sub, sub), au[r]);
                    }
                }
            }
#pragma unroll
            for (int r = 0; r < NE; ++r) {
                ag[r] = make_float2((ag[r].x + ag[r].y) * xsc[r], 0.f);
                au[r] = make_float2((au[r].x + au[r].y) * xsc[r], 0.f);
            }
        } else
        for (int bb = lane; bb < d / 16; bb += 32) {
            float2 gf[8], uf[8];
            fp4x16(*reinterpret_cast<const uint2 *>(gq + bb * 8), gf);
            fp4x16(*reinterpret_cast<const uint2 *>(uq + bb * 8), uf);
            const float sgb = e4m3f(gs[bb]), sub = e4m3f(us[bb]);
#pragma unroll
            for (int r = 0; r < NE; ++r) {
                if (NE <= 2 || r < seg.n_e) {
                    const uint4 *xp =
                        a.x_in_smem ? reinterpret_cast<const uint4 *>(xs + (size_t)seg.tok[r] * d * 2) + bb * 2
                                    : reinterpret_cast<const uint4 *>(a.x + (size_t)seg.tok[r] * d) + bb * 2;
                    const uint4 xa = a.x_in_smem ? xp[0] : __ldg(xp), xb = a.x_in_smem ? xp[1] : __ldg(xp + 1);
                    const uint32_t xw[8] = {xa.x, xa.y, xa.z, xa.w, xb.x, xb.y, xb.z, xb.w};
                    float2 pg = make_float2(0.f, 0.f), pu = make_float2(0.f, 0.f);
#pragma unroll
                    for (int q = 0; q < 8; ++q) {
                        const float2 xq = bf2(xw[q]);
                        pg = ffma2(gf[q], xq, pg);
                        pu = ffma2(uf[q], xq, pu);
                    }
                    ag[r].x = fmaf(pg.x + pg.y, sgb, ag[r].x);
                    au[r].x = fmaf(pu.x + pu.y, sub, au[r].x);
                }
            }
        }
    }
    __syncwarp();
    if (lane == 0) mbar_arrive(empty_slot);
    const float gsc = FP4 ? lw.gg[seg.e] : 1.f, usc = FP4 ? lw.gu[seg.e] : 1.f;
    if (seg.n_e == 1) {
        // one token: lanes < 16 reduce the gate sum, lanes >= 16 the up sum
        const bool hi = lane & 16;
        const float gs_ = ag[0].x + ag[0].y, us_ = au[0].x + au[0].y;
        float kk = hi ? us_ : gs_;
        kk += __shfl_xor_sync(0xFFFFFFFFu, hi ? gs_ : us_, 16);
        kk += __shfl_xor_sync(0xFFFFFFFFu, kk, 8);
        kk += __shfl_xor_sync(0xFFFFFFFFu, kk, 4);
        kk += __shfl_xor_sync(0xFFFFFFFFu, kk, 2);
        kk += __shfl_xor_sync(0xFFFFFFFFu, kk, 1);
        const float up_total = __shfl_sync(0xFFFFFFFFu, kk, 16);
        if (lane == 0) a.ws.h[(size_t)seg.row0 * I + i] = silu(kk * gsc) * (up_total * usc);
    } else {
        float hv = 0.f;
#pragma unroll
        for (int r = 0; r < NE; ++r) {
            if (NE <= 2 || r < seg.n_e) {
                const float sg_ = warp_sum(ag[r].x + ag[r].y) * gsc;
                const float su_ = warp_sum(au[r].x + au[r].y) * usc;
                if (lane == r) hv = silu(sg_) * su_;
            }
        }
        if (lane < seg.n_e) a.ws.h[(size_t)(seg.row0 + lane) * I + i] = hv;
    }
}

// Down rows of one stage (kDnRows rows of W_down in `st`) for a group of nr
// tokens of one expert (nr <= NG; exactly NG when NG <= 2), h rows at hg:
// y[t][q] for the group's tokens t, stored at yg[t * d + q] (scaled by gsc).
template <int NG, bool FP4>
__device__ __forceinline__ void dn_group(const Args &a, const unsigned char *st, const float *hg, int nr, float *yg,
                                         float gsc) {
    const int lane = threadIdx.x & 31;
    const int d = a.d, I = a.I;
    const int nvec = I / 8;
    const uint32_t rbd = rowb<FP4>(I);
    float2 acc[kDnRows][NG];
#pragma unroll
    for (int q = 0; q < kDnRows; ++q)
#pragma unroll
        for (int r = 0; r < NG; ++r) acc[q][r] = make_float2(0.f, 0.f);
    if (!FP4) {
        // token by token; h (in L2, written by other CTAs) fetched
        // in chunks of kHV vectors per lane, all loads of a chunk
        // issued before its arithmetic
        constexpr int kHV = 4;
#pragma unroll
        for (int r = 0; r < NG; ++r) {
            if (NG <= 2 || r < nr) {
                const float4 *hr = reinterpret_cast<const float4 *>(hg + (size_t)r * I);
                for (int j0 = 0; j0 * 32 < nvec; j0 += kHV) {
                    float4 h0[kHV], h1[kHV];
#pragma unroll
                    for (int jj = 0; jj < kHV; ++jj) {
                        const int v = lane + 32 * (j0 + jj);
                        if (v < nvec) {
                            h0[jj] = __ldcg(hr + 2 * v);
                            h1[jj] = __ldcg(hr + 2 * v + 1);
                        }
                    }
#pragma unroll
                    for (int jj = 0; jj < kHV; ++jj) {
                        const int v = lane + 32 * (j0 + jj);
                        if (v < nvec) {
                            const float2 ha = make_float2(h0[jj].x, h0[jj].y);
                            const float2 hb = make_float2(h0[jj].z, h0[jj].w);
                            const float2 hc = make_float2(h1[jj].x, h1[jj].y);
                            const float2 hd = make_float2(h1[jj].z, h1[jj].w);
#pragma unroll
                            for (int q = 0; q < kDnRows; ++q) {
                                const uint4 wv = reinterpret_cast<const uint4 *>(st + q * rbd)[v];
                                acc[q][r] = ffma2(bf2(wv.x), ha, acc[q][r]);
                                acc[q][r] = ffma2(bf2(wv.y), hb, acc[q][r]);
                                acc[q][r] = ffma2(bf2(wv.z), hc, acc[q][r]);
                                acc[q][r] = ffma2(bf2(wv.w), hd, acc[q][r]);
                            }
                        }
                    }
                }
            }
        }
    } else {
        const unsigned char *qb = st, *sb = st + kDnRows * (I / 2);
        for (int bb = lane; bb < I / 16; bb += 32) {
            // the block's 16 h values of each token, loaded once for all rows
            float4 hv[NG][4];
#pragma unroll
            for (int r = 0; r < NG; ++r) {
                if (NG <= 2 || r < nr) {
                    const float4 *hp = reinterpret_cast<const float4 *>(hg + (size_t)r * I + bb * 16);
#pragma unroll
                    for (int h4 = 0; h4 < 4; ++h4) hv[r][h4] = __ldcg(hp + h4);
                }
            }
#pragma unroll
            for (int q = 0; q < kDnRows; ++q) {
                float2 wf[8];
                fp4x16(*reinterpret_cast<const uint2 *>(qb + q * (I / 2) + bb * 8), wf);
                const float sc = e4m3f(sb[q * (I / 16) + bb]);
#pragma unroll
                for (int r = 0; r < NG; ++r) {
                    if (NG <= 2 || r < nr) {
                        float2 p = make_float2(0.f, 0.f);
#pragma unroll
                        for (int h4 = 0; h4 < 4; ++h4) {
                            p = ffma2(wf[2 * h4], make_float2(hv[r][h4].x, hv[r][h4].y), p);
                            p = ffma2(wf[2 * h4 + 1], make_float2(hv[r][h4].z, hv[r][h4].w), p);
                        }
                        acc[q][r].x = fmaf(p.x + p.y, sc, acc[q][r].x);
                    }
                }
            }
        }
    }
    if (nr == 1) {
        store_four_rows(acc[0][0].x + acc[0][0].y, acc[1][0].x + acc[1][0].y,
                        acc[2][0].x + acc[2][0].y, acc[3][0].x + acc[3][0].y,
                        yg, gsc);
    } else {
#pragma unroll
        for (int q = 0; q < kDnRows; ++q) {
            float yv = 0.f;
#pragma unroll
            for (int r = 0; r < NG; ++r) {
                if (NG <= 2 || r < nr) {
                    const float sum = warp_sum(acc[q][r].x + acc[q][r].y);
                    if (lane == r) yv = sum * gsc;
                }
            }
            if (lane < nr) yg[(size_t)lane * d + q] = yv;
        }
    }
}

// ---------------------------------------------------------------------------
// the kernel
// ---------------------------------------------------------------------------
template <int TM, bool FP4, bool STACK>
__global__ void __launch_bounds__(Warps<TM, FP4>::kThreads, 1) decode_layer_kernel(const __grid_constant__ Args a) {
    constexpr int kThreads = Warps<TM, FP4>::kThreads;
    constexpr int kConsumers = Warps<TM, FP4>::kConsumers;
    constexpr int kProducerWarp = Warps<TM, FP4>::kProducerWarp;
    extern __shared__ __align__(128) unsigned char smem[];
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int d = a.d, I = a.I, E = a.E, k = a.k, T = a.T, NS = a.nslots, C = a.ncons;
    const int G = gridDim.x, b = blockIdx.x;
    uint32_t *err = &a.ws.ctrl->err;
    Control *ctrl = a.ws.ctrl;
    // the launch's epoch: layer l's logits carry the tag ep0 + 1 + l; the last
    // CTA out advances the epoch past this launch's tags
    const uint32_t ep0 = *reinterpret_cast<const volatile uint32_t *>(&ctrl->epoch);

    // ---- shared-memory layout ----
    uint64_t *full = reinterpret_cast<uint64_t *>(smem);
    uint64_t *empty = full + kMaxSlots;
    uint64_t *xbar = empty + kMaxSlots;             // bytes [512, 520)
    volatile int *abort_flag = reinterpret_cast<volatile int *>(smem + 520);
    int *n_uniq_s = reinterpret_cast<int *>(smem + 524);
    int *cb_rows_s = reinterpret_cast<int *>(smem + 528);   // [32]
    int *cb_todo = cb_rows_s + 32;                  // [32]
    int *n_todo = cb_todo + 32;
    float *xscale = reinterpret_cast<float *>(smem + 800);  // [16] NVFP4: per-token max|x|
    Plan *plan1 = reinterpret_cast<Plan *>(smem + 896);     // one token: the plan, worked out during the routing
    float *part = reinterpret_cast<float *>(smem + 1024);   // [8 warps][TM] router partials
    unsigned char *rbase = smem + 2048;             // routing scratch (8 KB)
    Route R;
    R.cnt = reinterpret_cast<int32_t *>(rbase);     // [257]
    R.off = R.cnt + 260;                            // [257]
    R.uniq = R.off + 260;                           // [256]
    R.scan = R.uniq + 260;                          // [257]
    R.bm = reinterpret_cast<uint32_t *>(R.scan + 260);      // [256]
    R.ids = reinterpret_cast<int32_t *>(R.bm + 256);        // [16 * 8]
    R.pos = R.ids + 128;                            // [16 * 8]
    R.perm = R.pos + 128;                           // [16 * 8]
    R.w = reinterpret_cast<float *>(R.perm + 128);  // [16 * 8]
    R.wsum = reinterpret_cast<uint32_t *>(R.w + 128);       // [8]
    R.n_uniq = n_uniq_s;
    unsigned char *xs = smem + 2048 + 8192;
    const uint32_t x_bytes = a.x_in_smem ? (uint32_t)T * d * 2 : 0u;
    unsigned char *ring = xs + ((x_bytes + 127) / 128) * 128;
    // the router's copy of the tokens: the persistent one, or, before the
    // weight stream starts, the ring
    const uint32_t xr_bytes = (a.x_in_smem || a.x_router_ring) ? (uint32_t)T * d * 2 : 0u;
    const unsigned char *xr = a.x_in_smem ? xs : ring;

    if (tid == 0) {
        for (int s = 0; s < NS; ++s) {
            mbar_init(&full[s], 1);
            mbar_init(&empty[s], 1);
        }
        mbar_init(xbar, 1);
        *abort_flag = 0;
        fence_barrier_init();
    }
    for (int i = tid; i < 32; i += kThreads) cb_rows_s[i] = 0;
    __syncthreads();

    // stacked layers: the h-row counts keep growing from layer to layer; the
    // earlier layers' totals, per half, sit in shared memory (not registers)
    uint32_t *hbase = reinterpret_cast<uint32_t *>(smem + 788);  // [2]
    if (tid == 0) hbase[0] = hbase[1] = 0u;
    for (int layer = 0; layer < (STACK ? a.n_layers : 1); ++layer) {
    constexpr bool stacked = STACK;
    // the weight pointers are read where used (parameter space or the stack
    // record), not held in registers across the layer
    const LayerW &lw = stacked ? a.ws.stack[layer] : a.lw0;
    if (layer > 0) {
        // the previous layer's copies have all landed and been consumed: the
        // ring's barriers start again from phase 0
        if (tid == 0) {
            for (int s = 0; s < NS; ++s) {
                mbar_inval(&full[s]);
                mbar_inval(&empty[s]);
                mbar_init(&full[s], 1);
                mbar_init(&empty[s], 1);
            }
            fence_barrier_init();
        }
        for (int i = tid; i < 32; i += kThreads) cb_rows_s[i] = 0;
        __syncthreads();
    }
    if (stacked) {
        // the layer's input, RMSNorm(x_l) in bf16, into shared memory; the
        // arithmetic (256 threads, 8 elements each per 2048 columns, fp32
        // squares, warp sums, the 8 warps' sums in order) is moe_rmsnorm's
        static_assert(kThreads == 256, "the stacked input norm mirrors a 256-thread RMSNorm");
        float ss[8], rn[8];
        float *pr = part;  // [8 warps][8 tokens]
        const uint16_t *xin = layer > 0 ? a.out : a.x;
#pragma unroll
        for (int t = 0; t < 8; ++t) {
            ss[t] = 0.f;
            if (t < T) {
                for (int c = tid * 8; c < d; c += 256 * 8) {
                    const uint4 v = __ldcg(reinterpret_cast<const uint4 *>(xin + (size_t)t * d + c));
                    const uint32_t wv[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
                    for (int i = 0; i < 4; ++i) {
                        const float lo = bf16lo(wv[i]), hi = bf16hi(wv[i]);
                        ss[t] = fmaf(lo, lo, ss[t]);
                        ss[t] = fmaf(hi, hi, ss[t]);
                    }
                }
                const float wsum = warp_sum(ss[t]);
                if (lane == 0) pr[warp * 8 + t] = wsum;
            }
        }
        __syncthreads();
#pragma unroll
        for (int t = 0; t < 8; ++t) {
            float tot = 0.f;
#pragma unroll
            for (int i = 0; i < 8; ++i) tot += pr[i * 8 + t];
            rn[t] = 1.0f / sqrtf(tot / (float)d + a.eps);
        }
#pragma unroll
        for (int t = 0; t < 8; ++t) {
            if (t < T) {
                for (int c = tid * 8; c < d; c += 256 * 8) {
                    const uint4 v = __ldcg(reinterpret_cast<const uint4 *>(xin + (size_t)t * d + c));
                    const uint32_t wv[4] = {v.x, v.y, v.z, v.w};
                    uint32_t o[4];
#pragma unroll
                    for (int i = 0; i < 4; ++i)
                        o[i] = (uint32_t)f32_to_bf16_rn(bf16lo(wv[i]) * rn[t]) |
                               ((uint32_t)f32_to_bf16_rn(bf16hi(wv[i]) * rn[t]) << 16);
                    *reinterpret_cast<uint4 *>(xs + ((size_t)t * d + c) * 2) = make_uint4(o[0], o[1], o[2], o[3]);
                }
            }
        }
        __syncthreads();
    } else if (tid == 32 * kProducerWarp && xr_bytes) {
        mbar_arrive_expect_tx(xbar, xr_bytes);
        bulk_g2s(const_cast<unsigned char *>(xr), a.x, xr_bytes, xbar, policy_evict_last());
    }

    // ---- 1. router: logits of this CTA's experts ----
    // experts b, b + G, b + 2G, ... two at a time: warps 0-3 / 4-7 take the
    // four quarters of one expert's row
    {
        const int nq = d / 32;  // 16-byte vectors per quarter row (<= 256: at most 8 per lane)
        bool x_ready = xr_bytes == 0 || stacked;
        for (int base = b; base < E; base += 2 * G) {
            const int eidx = base + (warp >= 4 ? G : 0);
            const int q = warp & 3;
            float acc[TM];
#pragma unroll
            for (int t = 0; t < TM; ++t) acc[t] = 0.f;
            // the router rows are requested before waiting for the tokens' copy
            uint4 wpre[8];
            const bool mine = warp < 8 && eidx < E;
            const uint4 *wrow = reinterpret_cast<const uint4 *>(lw.wr + (size_t)eidx * d) + q * nq;
#pragma unroll
            for (int j = 0; j < 8; ++j) {
                const int v = lane + 32 * j;
                wpre[j] = (mine && v < nq) ? __ldg(wrow + v) : make_uint4(0, 0, 0, 0);
            }
            if (!x_ready) {
                mbar_wait_or_abort(xbar, 0, err, abort_flag);  // a timeout: the routing's tag wait gives up at once
                x_ready = true;
            }
            if (mine) {
#pragma unroll
                for (int j = 0; j < 8; ++j) {
                    const int v = lane + 32 * j;
                    if (v >= nq) continue;
                    const uint4 wv = wpre[j];
#pragma unroll
                    for (int t = 0; t < TM; ++t) {
                        if (t < T) {
                            const uint4 xv = xr_bytes
                                                 ? reinterpret_cast<const uint4 *>(xr + (size_t)t * d * 2)[q * nq + v]
                                                 : __ldg(reinterpret_cast<const uint4 *>(a.x + (size_t)t * d) + q * nq + v);
                            float2 s2 = make_float2(0.f, 0.f);
                            s2 = ffma2(bf2(wv.x), bf2(xv.x), s2);
                            s2 = ffma2(bf2(wv.y), bf2(xv.y), s2);
                            s2 = ffma2(bf2(wv.z), bf2(xv.z), s2);
                            s2 = ffma2(bf2(wv.w), bf2(xv.w), s2);
                            acc[t] += s2.x + s2.y;
                        }
                    }
                }
            }
#pragma unroll
            for (int t = 0; t < TM; ++t) {
                const float s = warp_sum(acc[t]);
                if (lane == 0 && warp < 8) part[warp * TM + t] = s;
            }
            __syncthreads();
            if (tid < 2 * kTagRows) {
                // every row of the tagged logits (rows past T hold 0), so each
                // word read later was written by this launch or the previous one
                const int half = tid / kTagRows, t = tid % kTagRows;
                const int e2 = base + half * G;
                if (e2 < E) {
                    float l = 0.f;
                    if (t < T) {
                        const float *pp = part + half * 4 * TM;
                        l = ((pp[0 * TM + t] + pp[1 * TM + t]) + pp[2 * TM + t]) + pp[3 * TM + t];
                        if (lw.bias) l += lw.bias[e2];
                    }
                    st_tagged(a.ws.tlogits + (size_t)t * E + e2, l, ep0 + 1u + (uint32_t)layer);
                }
            }
            __syncthreads();
        }
        if (!x_ready) mbar_wait_or_abort(xbar, 0, err, abort_flag);  // CTAs without router rows
    }

    if (FP4 && x_bytes) {
        // NVFP4 gate/up sums in fp16: keep the staged tokens as fp16(x / max|x|)
        for (int t = warp; t < T; t += kConsumers + 1) {
            const uint32_t *xw = reinterpret_cast<const uint32_t *>(xs + (size_t)t * d * 2);
            float m = 0.f;
            for (int i = lane; i < d / 2; i += 32) {
                const uint32_t wv = xw[i];
                m = fmaxf(m, fmaxf(fabsf(bf16lo(wv)), fabsf(bf16hi(wv))));
            }
#pragma unroll
            for (int o = 16; o > 0; o >>= 1) m = fmaxf(m, __shfl_xor_sync(0xFFFFFFFFu, m, o));
            if (lane == 0) xscale[t] = m > 0.f ? m : 1.f;
        }
        __syncthreads();
        for (int i = tid; i < T * (d / 2); i += kThreads) {
            const float inv = 1.f / xscale[i / (d / 2)];
            uint32_t *xw = reinterpret_cast<uint32_t *>(xs) + i;
            const uint32_t wv = *xw;
            const __half2 hv = __floats2half2_rn(bf16lo(wv) * inv, bf16hi(wv) * inv);
            *xw = *reinterpret_cast<const uint32_t *>(&hv);
        }
        __syncthreads();
    }

    // one token: its k experts are distinct, so the plan (equal shares of k
    // experts' stages) does not wait for the routing; the producer warp,
    // idle while warp 0 waits for the logits, works it out meanwhile
    if (T == 1 && warp == kProducerWarp && lane == 0) *plan1 = make_plan(k, I, d / kDnRows, b, G);
    // ---- 2. routing, computed by every CTA in shared memory ----
    // (the logits come from every CTA's router: each word is waited for by
    // its tag, so no grid barrier stands between the router and the routing;
    // the test hook shifts the awaited tag to one that never comes)
    {
        const uint32_t hold = *reinterpret_cast<const volatile uint32_t *>(&ctrl->test_hold);
        route_tokens(R, nullptr, a.ws.tlogits, ep0 + 1u + (uint32_t)layer + hold, T, k, E, err, abort_flag,
                     b == 0 || T > 1);
    }
    const int n_uniq = *R.n_uniq;
    if (b == 0) publish_records(R, a.ws, T, k, E, n_uniq, kThreads);

    // ---- 3./4. the weight stream ----
    // The active experts are split in two halves, H1 = the first ceil(U/2).
    // Every CTA streams its share of, in order: H1 gate/up rows, H2 gate/up
    // rows, H1 down rows, H2 down rows. Down rows of a half wait for that
    // half's h (a global row count), which the other CTAs finished a whole
    // segment earlier, so the stream does not stop between the two
    // projections. A wait only ever sits at a down stage, and every stage that
    // feeds the counts comes earlier in every CTA's order, so the waits end.
    // One token: every expert costs the same, equal shares. More: experts
    // with more tokens cost more per stage; the shares are cut by weight.
    Plan pl;
    if (T == 1) {
        pl = *plan1;   // n_uniq == k
    } else {
        // the segments cut by weight: the eight cut points, one thread each
        int *cut = reinterpret_cast<int *>(R.wsum);   // free after the routing
        const int U1h = (n_uniq + 1) / 2;
        if (tid < 8) {
            const int sg = tid >> 1;   // A, B, C, D
            const int lo = (sg & 1) ? U1h : 0, hi = (sg & 1) ? n_uniq : U1h;
            cut[tid] = weighted_start(R.scan, lo, hi, sg < 2 ? I : d / kDnRows, b + (tid & 1), G);
        }
        __syncthreads();
        pl.a0 = cut[0];
        pl.nA = cut[1] - cut[0];
        pl.b0 = cut[2];
        pl.nB = cut[3] - cut[2];
        pl.c0 = cut[4];
        pl.nC = cut[5] - cut[4];
        pl.d0 = cut[6];
        pl.nD = cut[7] - cut[6];
        pl.offB = U1h * I;
        pl.offD = U1h * (d / kDnRows);
    }
    const int n_gu = pl.nA + pl.nB;
    const int n_st = n_gu + pl.nC + pl.nD;
    const int U1 = (n_uniq + 1) / 2;
    const uint32_t rbg = rowb<FP4>(d), rbd = rowb<FP4>(I);

    if (warp == kProducerWarp) {
        // a.nprod lanes fill the ring, lane l the slots j with j % nprod == l
        // (nslots is a multiple of nprod), so every slot's fills come from one
        // lane in order. The lanes poll their next slot without blocking and
        // stay converged: a lane that sleeps in a blocking wait holds up the
        // other lanes of its warp, whose slots may long be free.
        const int P = a.nprod;
        const uint64_t pol = policy_evict_first();
        int s = lane;
        unsigned long long t_progress = global_ns();
        for (uint32_t it = 1;; ++it) {
            const bool live = lane < P && s < n_st;
            if (!__any_sync(0xFFFFFFFFu, live)) break;
            const int slot = s % NS;
            const bool ready = live && (s < NS || mbar_test_wait(&empty[slot], ((s / NS) - 1) & 1));
            if (ready) {
                unsigned char *dst = ring + (size_t)slot * a.slot_bytes;
                if (s < n_gu) {
                    const int g = pl.gu_row(s);
                    const int u = g / I, i = g - u * I;
                    const size_t row = (size_t)R.uniq[u] * I + i;
                    mbar_arrive_expect_tx(&full[slot], 2 * rbg);
                    if (!FP4) {
                        const int64_t ld = lw.gu_ld;
                        if (lw.wu == lw.wg + d && ld == 2 * (int64_t)d) {
                            // interleaved rows: gate row i and up row i are one contiguous copy
                            bulk_g2s(dst, lw.wg + (int64_t)row * ld, 2 * rbg, &full[slot], pol);
                        } else {
                            bulk_g2s(dst, lw.wg + (int64_t)row * ld, rbg, &full[slot], pol);
                            bulk_g2s(dst + rbg, lw.wu + (int64_t)row * ld, rbg, &full[slot], pol);
                        }
                    } else {
                        const uint32_t nq = d / 2, nsb = d / 16;
                        bulk_g2s(dst, lw.qg + row * nq, nq, &full[slot], pol);
                        bulk_g2s(dst + nq, lw.sg + row * nsb, nsb, &full[slot], pol);
                        bulk_g2s(dst + rbg, lw.qu + row * nq, nq, &full[slot], pol);
                        bulk_g2s(dst + rbg + nq, lw.su + row * nsb, nsb, &full[slot], pol);
                    }
                } else {
                    const int g = pl.dn_unit(s - n_gu) * kDnRows;
                    const int u = g / d, c0 = g - u * d;
                    const size_t row = (size_t)R.uniq[u] * d + c0;
                    mbar_arrive_expect_tx(&full[slot], kDnRows * rbd);
                    if (!FP4) {
                        bulk_g2s(dst, lw.wd + row * I, kDnRows * rbd, &full[slot], pol);
                    } else {
                        const uint32_t nq = I / 2, nsb = I / 16;
                        bulk_g2s(dst, lw.qd + row * nq, kDnRows * nq, &full[slot], pol);
                        bulk_g2s(dst + kDnRows * nq, lw.sd + row * nsb, kDnRows * nsb, &full[slot], pol);
                    }
                }
                s += P;
            }
            // bounded: give up once no lane has issued for the wait limit
            if (__any_sync(0xFFFFFFFFu, ready)) {
                t_progress = 0;
            } else if ((it & 255u) == 0) {
                const unsigned long long now = global_ns();
                if (t_progress == 0) t_progress = now;
                const bool other_gave_up = *abort_flag != 0;
                const bool timed_out = now - t_progress > kWaitLimitNs;
                if (__any_sync(0xFFFFFFFFu, other_gave_up || timed_out)) {  // the whole warp leaves together
                    if (lane == 0 && !other_gave_up) {
                        atomicOr(err, ERRBIT_TIMEOUT);
                        *abort_flag = 1;
                    }
                    break;
                }
            }
        }
        __syncwarp();
        if (STACK && layer + 1 < a.n_layers && lane == 0) prefetch_next_router(a.ws.stack[layer + 1], b, G, E, d);
        // every copy this lane issued must land before the CTA moves on (in a
        // normal run the consumers have waited for all of them already)
        if (lane < P) {
            // the lane's last fill of each of its slots: stages s - NS .. s - P
            // (s and NS - P are multiples of P apart from lane)
            for (int j = max(lane, s - NS); j < s; j += P) mbar_wait(&full[j % NS], (j / NS) & 1, err);
        }
    } else if (warp < C) {
        // ------------------------------- gate/up -------------------------------
        Seg<TM> seg;
        int s = warp;
        int done_a = 0, done_b = 0;   // this warp's finished h rows of each half
        bool pub_a = false;
        for (; s < n_gu && !*abort_flag; s += C) {
            if (s >= pl.nA && !pub_a) {
                publish_rows(&ctrl->h_ready[0].v, done_a);
                pub_a = true;
            }
            if (s < pl.nA)
                ++done_a;
            else
                ++done_b;
            const int slot = s % NS;
            const int g = pl.gu_row(s);
            const int u = g / I, i = g - u * I;
            if (u != seg.u) seg_load(seg, R, u);
            if (!mbar_wait_or_abort(&full[slot], (s / NS) & 1, err, abort_flag)) break;
            const unsigned char *st = ring + (size_t)slot * a.slot_bytes;
            if (TM == 1 || seg.n_e == 1)
                gu_stage<1, TM, FP4>(a, lw, st, xs, xscale, seg, &empty[slot], i);
            else if (TM == 2 || seg.n_e == 2)
                gu_stage<(TM < 2 ? TM : 2), TM, FP4>(a, lw, st, xs, xscale, seg, &empty[slot], i);
            else if (TM == 4 || seg.n_e <= 4)
                gu_stage<(TM < 4 ? TM : 4), TM, FP4>(a, lw, st, xs, xscale, seg, &empty[slot], i);
            else if (TM == 8 || seg.n_e <= 8)
                gu_stage<(TM < 8 ? TM : 8), TM, FP4>(a, lw, st, xs, xscale, seg, &empty[slot], i);
            else
                gu_stage<TM, TM, FP4>(a, lw, st, xs, xscale, seg, &empty[slot], i);
        }
        // this warp's h rows are written: count them in
        if (!pub_a) publish_rows(&ctrl->h_ready[0].v, done_a);
        publish_rows(&ctrl->h_ready[1].v, done_b);
        bool ready_a = false, ready_b = false;
        // ---------------------------------- down ----------------------------------
        Seg<TM> sd;
        // an expert with one token: its h row stays in registers for all the
        // warp's stages of that expert (I <= 2048)
        constexpr int kHC = 8;
        float4 hc0[kHC], hc1[kHC];
        int hc_u = -1;
        for (; s < n_st && !*abort_flag; s += C) {
            const int t = s - n_gu;
            if (t < pl.nC && !ready_a) {
                if (!wait_rows(&ctrl->h_ready[0].v, hbase[0] + (uint32_t)(U1 * I), err, abort_flag)) break;
                ready_a = true;
            }
            if (t >= pl.nC && !ready_b) {
                if (!wait_rows(&ctrl->h_ready[1].v, hbase[1] + (uint32_t)((n_uniq - U1) * I), err, abort_flag)) break;
                ready_b = true;
            }
            const int slot = s % NS;
            const int g = pl.dn_unit(t) * kDnRows;
            const int u = g / d, c0 = g - u * d;
            if (u != sd.u) seg_load(sd, R, u);
            if (!mbar_wait_or_abort(&full[slot], (s / NS) & 1, err, abort_flag)) break;
            const unsigned char *st = ring + (size_t)slot * a.slot_bytes;
            const float *hrow = a.ws.h + (size_t)sd.row0 * I;
            const float gsc = FP4 ? lw.gd[sd.e] : 1.f;
            const int nvec = I / 8;
            if (!FP4 && sd.n_e == 1 && nvec <= 32 * kHC) {
                // one token, its h row held in registers across the expert's stages
                if (hc_u != sd.u) {
                    const float4 *hr = reinterpret_cast<const float4 *>(hrow);
#pragma unroll
                    for (int jj = 0; jj < kHC; ++jj) {
                        const int v = lane + 32 * jj;
                        if (v < nvec) {
                            hc0[jj] = __ldcg(hr + 2 * v);
                            hc1[jj] = __ldcg(hr + 2 * v + 1);
                        }
                    }
                    hc_u = sd.u;
                }
                float2 acc[kDnRows];
#pragma unroll
                for (int q = 0; q < kDnRows; ++q) acc[q] = make_float2(0.f, 0.f);
#pragma unroll
                for (int jj = 0; jj < kHC; ++jj) {
                    const int v = lane + 32 * jj;
                    if (v < nvec) {
                        const float2 ha = make_float2(hc0[jj].x, hc0[jj].y), hb = make_float2(hc0[jj].z, hc0[jj].w);
                        const float2 hc = make_float2(hc1[jj].x, hc1[jj].y), hd = make_float2(hc1[jj].z, hc1[jj].w);
#pragma unroll
                        for (int q = 0; q < kDnRows; ++q) {
                            const uint4 wv = reinterpret_cast<const uint4 *>(st + q * rbd)[v];
                            acc[q] = ffma2(bf2(wv.x), ha, acc[q]);
                            acc[q] = ffma2(bf2(wv.y), hb, acc[q]);
                            acc[q] = ffma2(bf2(wv.z), hc, acc[q]);
                            acc[q] = ffma2(bf2(wv.w), hd, acc[q]);
                        }
                    }
                }
                __syncwarp();
                if (lane == 0) mbar_arrive(&empty[slot]);
                store_four_rows(acc[0].x + acc[0].y, acc[1].x + acc[1].y, acc[2].x + acc[2].y, acc[3].x + acc[3].y,
                                a.ws.Y + (size_t)sd.row0 * d + c0, gsc);
            } else if (FP4 && sd.n_e == 1 && I / 16 <= 32 * (kHC / 2)) {
                // NVFP4, one token: lane block j (16 elements of h) held across
                // the expert's stages as fp16(h / max|h_block|) in hc0[2j],
                // hc0[2j+1] (eight f16 pairs) with the block's max|h| in
                // hc1[2j].x; the 16 products of a block (|e2m1| <= 6, |h'| <= 1)
                // are summed in fp16, then scaled in fp32
                if (hc_u != sd.u) {
#pragma unroll
                    for (int j = 0; j < kHC / 2; ++j) {
                        const int bb = lane + 32 * j;
                        if (bb < I / 16) {
                            const float4 *hp = reinterpret_cast<const float4 *>(hrow + bb * 16);
                            const float4 v[4] = {__ldcg(hp), __ldcg(hp + 1), __ldcg(hp + 2), __ldcg(hp + 3)};
                            float m = 0.f;
#pragma unroll
                            for (int r = 0; r < 4; ++r)
                                m = fmaxf(m, fmaxf(fmaxf(fabsf(v[r].x), fabsf(v[r].y)), fmaxf(fabsf(v[r].z), fabsf(v[r].w))));
                            const float hs = m > 0.f ? m : 1.f, inv = 1.f / hs;
                            uint32_t hw[8];
#pragma unroll
                            for (int r = 0; r < 4; ++r) {
                                const __half2 lo = __floats2half2_rn(v[r].x * inv, v[r].y * inv);
                                const __half2 hi = __floats2half2_rn(v[r].z * inv, v[r].w * inv);
                                hw[2 * r] = *reinterpret_cast<const uint32_t *>(&lo);
                                hw[2 * r + 1] = *reinterpret_cast<const uint32_t *>(&hi);
                            }
                            hc0[2 * j] = make_float4(__uint_as_float(hw[0]), __uint_as_float(hw[1]),
                                                     __uint_as_float(hw[2]), __uint_as_float(hw[3]));
                            hc0[2 * j + 1] = make_float4(__uint_as_float(hw[4]), __uint_as_float(hw[5]),
                                                         __uint_as_float(hw[6]), __uint_as_float(hw[7]));
                            hc1[2 * j].x = hs;
                        }
                    }
                    hc_u = sd.u;
                }
                const unsigned char *qb = st, *sb = st + kDnRows * (I / 2);
                float acc[kDnRows];
#pragma unroll
                for (int q = 0; q < kDnRows; ++q) acc[q] = 0.f;
#pragma unroll
                for (int j = 0; j < kHC / 2; ++j) {
                    const int bb = lane + 32 * j;
                    if (bb < I / 16) {
                        const float4 A = hc0[2 * j], B = hc0[2 * j + 1];
                        const uint32_t hw[8] = {__float_as_uint(A.x), __float_as_uint(A.y), __float_as_uint(A.z),
                                                __float_as_uint(A.w), __float_as_uint(B.x), __float_as_uint(B.y),
                                                __float_as_uint(B.z), __float_as_uint(B.w)};
                        const __half2 *hh = reinterpret_cast<const __half2 *>(hw);
                        const float hs = hc1[2 * j].x;
#pragma unroll
                        for (int q = 0; q < kDnRows; ++q) {
                            const uint2 cq = *reinterpret_cast<const uint2 *>(qb + q * (I / 2) + bb * 8);
                            __half2 wh[8];
                            fp4x16_h2(cq, wh);
                            __half2 p0 = __hmul2(wh[0], hh[0]), p1 = __hmul2(wh[1], hh[1]);
#pragma unroll
                            for (int m = 2; m < 8; m += 2) {
                                p0 = __hfma2(wh[m], hh[m], p0);
                                p1 = __hfma2(wh[m + 1], hh[m + 1], p1);
                            }
                            const float2 f = __half22float2(__hadd2(p0, p1));
                            acc[q] = fmaf(f.x + f.y, e4m3f(sb[q * (I / 16) + bb]) * hs, acc[q]);
                        }
                    }
                }
                __syncwarp();
                if (lane == 0) mbar_arrive(&empty[slot]);
                store_four_rows(acc[0], acc[1], acc[2], acc[3], a.ws.Y + (size_t)sd.row0 * d + c0, gsc);
            } else {
                // the expert's tokens in groups of up to TG (bounded registers)
                constexpr int TG = TM < 4 ? TM : 4;
                for (int r0 = 0; r0 < sd.n_e; r0 += TG) {
                    const int nr = min(TG, sd.n_e - r0);
                    const float *hg = hrow + (size_t)r0 * I;
                    float *yg = a.ws.Y + (size_t)(sd.row0 + r0) * d + c0;
                    if (nr == 1)
                        dn_group<1, FP4>(a, st, hg, 1, yg, gsc);
                    else if (nr == 2)
                        dn_group<(TG < 2 ? TG : 2), FP4>(a, st, hg, nr, yg, gsc);
                    else if (nr <= 4)
                        dn_group<(TG < 4 ? TG : 4), FP4>(a, st, hg, nr, yg, gsc);
                    else
                        dn_group<TG, FP4>(a, st, hg, nr, yg, gsc);
                }
                __syncwarp();
                if (lane == 0) mbar_arrive(&empty[slot]);
            }
            if (lane == 0) atomicAdd(&cb_rows_s[c0 / kCb], kDnRows);
        }
    }

    // ---- 5. combine, by the CTA that completes each column block ----
    fence_acq_rel_gpu();  // this thread's h and Y stores before the block's count below
    __syncthreads();
    if (a.do_combine) {
        if (warp == 0) {
            // lane cb counts this CTA's rows of column block cb in; the
            // counts go out together rather than one round trip after another
            const int ncb = (d + kCb - 1) / kCb;
            bool fin = false;
            fence_acq_rel_gpu();  // the CTA's stores (ordered by the barrier) before this lane's count
            if (lane < ncb) {
                const int mine = cb_rows_s[lane];
                if (mine) {
                    const int cols = min(kCb, d - lane * kCb);
                    const uint32_t done = atomicAdd(&ctrl->cb_rows[lane].v, (uint32_t)mine) + mine;
                    fin = done == (uint32_t)(n_uniq * cols);
                }
            }
            fence_acq_rel_gpu();
            const uint32_t fin_mask = __ballot_sync(0xFFFFFFFFu, fin);
            if (lane == 0) {
                int n = 0;
                for (uint32_t m = fin_mask; m; m &= m - 1) cb_todo[n++] = __ffs(m) - 1;
                *n_todo = n;
            }
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
                const uint16_t *resid = stacked ? (layer > 0 ? a.out : a.x) : a.res;
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
                if (stacked && a.layer_out)
                    *reinterpret_cast<uint2 *>(a.layer_out + ((size_t)layer * T + t) * d + c) = o;
            }
            if (tid == 0) ctrl->cb_rows[cb].v = 0u;
        }
    }
    // the next layer reads every column of this one's output
    if (stacked && layer + 1 < a.n_layers) {
        if (tid == 0) {  // read by this CTA only, after the barrier below
            hbase[0] += (uint32_t)(U1 * I);
            hbase[1] += (uint32_t)((n_uniq - U1) * I);
        }
        grid_barrier(&ctrl->grid_bar.v, (uint32_t)(layer + 1) * G, err, abort_flag, &ctrl->test_hold);
    }
    }  // layers
    // ---- exit: the last CTA out resets the grid-barrier counters ----
    __syncthreads();
    if (tid == 0) {
        fence_acq_rel_gpu();
        if (atomicAdd(&ctrl->grid_exit.v, 1u) == (uint32_t)G - 1) {
            for (int cb = 0; cb < 32; ++cb) ctrl->cb_rows[cb].v = 0u;  // zero already unless a wait gave up
            ctrl->grid_bar.v = 0u;
            ctrl->h_ready[0].v = 0u;
            ctrl->h_ready[1].v = 0u;
            ctrl->grid_exit.v = 0u;
            ctrl->epoch = ep0 + (uint32_t)(STACK ? a.n_layers : 1);
            fence_acq_rel_gpu();
        }
    }
}

template <int TM, bool FP4>
static int pick(int fit, int &ncons) {
    if (fit > kMaxSlots) fit = kMaxSlots;
    for (int c = Warps<TM, FP4>::kConsumers; c >= 1; --c)
        if (fit / c >= 2) {
            ncons = c;
            return (fit / c) * c;
        }
    ncons = 1;
    return fit;
}

template <int TM, bool FP4, bool STACK>
static cudaError_t launch_t(const LayerDev &L, const Workspace &ws, const uint16_t *x, const uint16_t *res,
                            uint16_t *out, int T, cudaStream_t st, int n_layers = 0, float eps = 0.f,
                            uint16_t *layer_out = nullptr) {
    Args a{};
    a.x = x;
    a.res = res;
    a.out = out;
    a.lw0 = L.weights();
    a.n_layers = n_layers;
    a.eps = eps;
    a.layer_out = layer_out;
    a.T = T;
    a.d = L.d;
    a.I = L.I;
    a.E = L.E;
    a.k = L.k;
    a.ws = ws;
    a.do_combine = L.expert_norm ? 0 : 1;
    const uint32_t slot = (uint32_t)(2 * rowb<FP4>(L.d) > kDnRows * rowb<FP4>(L.I) ? 2 * rowb<FP4>(L.d)
                                                                                     : kDnRows * rowb<FP4>(L.I));
    a.slot_bytes = (slot + 127) / 128 * 128;
    const size_t fixed = 2048 + 8192;
    a.x_in_smem = T <= 8 ? 1 : 0;
    const size_t xb = a.x_in_smem ? align_up((size_t)T * L.d * 2, 128) : 0;
    if (fixed + xb + 2 * (size_t)a.slot_bytes > (size_t)kSmemBudget) {
        a.x_in_smem = 0;
    }
    const size_t xb2 = a.x_in_smem ? xb : 0;
    if (fixed + xb2 + 2 * (size_t)a.slot_bytes > (size_t)kSmemBudget) return cudaErrorInvalidConfiguration;
    if (STACK && (n_layers < 1 || !a.x_in_smem || L.expert_norm)) return cudaErrorInvalidValue;  // tokens in smem
    const int fit = (int)((kSmemBudget - fixed - xb2) / a.slot_bytes);
    a.nslots = pick<TM, FP4>(fit, a.ncons);
    a.x_router_ring = !a.x_in_smem && (size_t)a.nslots * a.slot_bytes >= (size_t)T * L.d * 2 ? 1 : 0;
    a.nprod = a.nslots % 4 == 0 ? 4 : (a.nslots % 2 == 0 ? 2 : 1);
    const size_t smem = fixed + xb2 + (size_t)a.nslots * a.slot_bytes;
    static std::atomic<uint64_t> attr_set{0};
    cudaError_t e = set_smem_limit_once((const void *)decode_layer_kernel<TM, FP4, STACK>, kSmemBudget, attr_set);
    if (e != cudaSuccess) return e;
    cudaLaunchConfig_t cfg{};
    cfg.gridDim = dim3(L.num_sms);
    cfg.blockDim = dim3(Warps<TM, FP4>::kThreads);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = st;
    cudaLaunchAttribute attrs[1];
    attrs[0].id = cudaLaunchAttributeCooperative;
    attrs[0].val.cooperative = 1;
    cfg.attrs = attrs;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, decode_layer_kernel<TM, FP4, STACK>, a);
}

}  // namespace fused

}  // namespace moe
