// decode.cu — expert stage for small batches (decode / speculative verify,
// T <= 16): the active experts' weights are streamed from HBM exactly once
// through a ring of shared-memory stages filled by bulk TMA copies, and the
// FFN arithmetic runs on CUDA cores with fp32 accumulation.
//
// Decode is bound by streaming weights from HBM, not by matmul speed, and
// fetching weights ahead of the compute that needs them hides the wait ("How
// SGLang-TorchTPU accelerated an 816B-parameter MoE on TPU v7", sections
// "Introduction" and "Key optimisations"). With at most 16 tokens, an expert
// sees about one token per step, so each weight element feeds 1-2 FMAs: the
// tensor cores would idle, and the work is a memory stream.
//
// Two persistent kernels, grid = one CTA per SM:
//   gate/up:  h[r, i] = silu(Wg[e,i,:] . x_t) * (Wu[e,i,:] . x_t)   (fp32)
//   down:     Y[r, c] = Wd[e,c,:] . h[r, :]                          (fp32)
// where r runs over the rows of the permuted (token, slot) order of expert e.
// The flattened rows of all active experts are split evenly over the CTAs,
// so every SM streams the same number of bytes whatever the routing.
// Warp roles: warps 0..7 consume stages, warp 8 (one lane) produces them.
//
// Formats: bf16 rows, or NVFP4 rows (packed E2M1 codes + one E4M3 scale per 16
// elements + one fp32 scale per tensor) dequantised in registers as they are
// consumed: the stream then carries 4.5 bits per weight.
#include <cuda_fp4.h>
#include <cuda_fp8.h>
#include <cuda_runtime.h>

#include "common.cuh"

namespace moe {

constexpr int kConsumerWarps = 8;
constexpr int kDecodeThreads = 32 * (kConsumerWarps + 1);
constexpr int kGuRowsPerStage = 2;   // gate/up: rows i per stage (each with gate and up)
constexpr int kDnRowsPerStage = 8;   // down: rows c per stage
constexpr int kMaxStages = 8;
constexpr int kSmemBudget = 227 * 1024;

template <bool FP4>
__host__ __device__ constexpr size_t row_bytes(int K) {
    return FP4 ? (size_t)K / 2 + (size_t)K / 16 : (size_t)K * 2;
}

struct DecodeArgs {
    const uint16_t *x;       // [T, d] bf16
    const uint16_t *wg, *wu, *wd;
    const uint8_t *qg, *qu, *qd, *sg, *su, *sd;
    const float *gg, *gu, *gd;
    int T, d, I, k;
    int nstages;
    Workspace ws;
};

// Segment bookkeeping: a CTA walks a contiguous range of flattened rows
// g = u * R + row over the active experts u (R rows per expert); a stage never
// crosses an expert boundary.
struct StageCursor {
    long long g, end;
    int R, max_rows;
    __device__ int next_len() const {
        long long left_in_expert = R - (g % R);
        long long left = end - g;
        long long n = left < left_in_expert ? left : left_in_expert;
        return (int)(n < max_rows ? n : max_rows);
    }
};

// ---------------------------------------------------------------------------
// dot helpers
// ---------------------------------------------------------------------------
__device__ __forceinline__ void unpack8(uint4 v, float f[8]) {
    f[0] = bf16lo(v.x); f[1] = bf16hi(v.x); f[2] = bf16lo(v.y); f[3] = bf16hi(v.y);
    f[4] = bf16lo(v.z); f[5] = bf16hi(v.z); f[6] = bf16lo(v.w); f[7] = bf16hi(v.w);
}

__device__ __forceinline__ float dot8(const float w[8], uint4 xv) {
    float a = w[0] * bf16lo(xv.x);
    a = fmaf(w[1], bf16hi(xv.x), a);
    a = fmaf(w[2], bf16lo(xv.y), a);
    a = fmaf(w[3], bf16hi(xv.y), a);
    a = fmaf(w[4], bf16lo(xv.z), a);
    a = fmaf(w[5], bf16hi(xv.z), a);
    a = fmaf(w[6], bf16lo(xv.w), a);
    a = fmaf(w[7], bf16hi(xv.w), a);
    return a;
}

// 8 packed bytes -> 16 E2M1 values (exact in fp32)
__device__ __forceinline__ void unpack_fp4x16(uint2 q, float f[16]) {
    uint32_t words[2] = {q.x, q.y};
#pragma unroll
    for (int wi = 0; wi < 2; ++wi) {
#pragma unroll
        for (int b = 0; b < 4; ++b) {
            __nv_fp4x2_storage_t byte = (__nv_fp4x2_storage_t)((words[wi] >> (8 * b)) & 0xFFu);
            __half2_raw hr = __nv_cvt_fp4x2_to_halfraw2(byte, __NV_E2M1);
            float2 p = __half22float2(*reinterpret_cast<__half2 *>(&hr));
            f[wi * 8 + 2 * b] = p.x;      // low nibble: lower index
            f[wi * 8 + 2 * b + 1] = p.y;
        }
    }
}

__device__ __forceinline__ float e4m3_to_f32(uint8_t s) {
    __half_raw hr = __nv_cvt_fp8_to_halfraw((__nv_fp8_storage_t)s, __NV_E4M3);
    return __half2float(*reinterpret_cast<__half *>(&hr));
}

// ---------------------------------------------------------------------------
// gate/up kernel
// ---------------------------------------------------------------------------
template <int TM, bool FP4>
__global__ void __launch_bounds__(kDecodeThreads, 1) decode_gateup_kernel(DecodeArgs a) {
    extern __shared__ __align__(128) unsigned char smem[];
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int d = a.d, I = a.I, NS = a.nstages;
    uint32_t *err = &a.ws.ctrl->err;

    uint64_t *full = reinterpret_cast<uint64_t *>(smem);
    uint64_t *empty = full + kMaxStages;
    uint64_t *xbar = empty + kMaxStages;
    volatile int *abort_flag = reinterpret_cast<volatile int *>(xbar + 1);
    float *red = reinterpret_cast<float *>(smem + 256);  // [2][RP][4][TM][2]
    constexpr int kParts = kConsumerWarps / kGuRowsPerStage;
    const size_t red_bytes = sizeof(float) * 2 * kGuRowsPerStage * kParts * TM * 2;
    unsigned char *xs = smem + 256 + ((red_bytes + 127) / 128) * 128;
    const size_t x_bytes = (size_t)a.T * d * 2;
    unsigned char *ring = xs + ((x_bytes + 127) / 128) * 128;
    const size_t rb = row_bytes<FP4>(d);
    const size_t stage_bytes = 2 * kGuRowsPerStage * rb;

    if (tid == 0) {
        for (int s = 0; s < NS; ++s) {
            mbar_init(&full[s], 1);
            mbar_init(&empty[s], kConsumerWarps);
        }
        mbar_init(xbar, 1);
        *abort_flag = 0;
        fence_barrier_init();
    }
    __syncthreads();

    const long long G = (long long)a.ws.ctrl->n_uniq * I;
    const long long g_begin = (long long)blockIdx.x * G / gridDim.x;
    const long long g_end = (long long)(blockIdx.x + 1) * G / gridDim.x;

    if (warp == kConsumerWarps) {
        // ------------------------------ producer ------------------------------
        if (lane == 0) {
            const uint64_t pol = policy_evict_first();
            mbar_arrive_expect_tx(xbar, (uint32_t)x_bytes);
            bulk_g2s(xs, a.x, (uint32_t)x_bytes, xbar, policy_evict_last());
            StageCursor cur{g_begin, g_end, I, kGuRowsPerStage};
            int s = 0;
            bool ok = true;
            while (cur.g < cur.end && ok) {
                const int slot = s % NS;
                if (s >= NS) ok = mbar_wait_or_abort(&empty[slot], ((s / NS) - 1) & 1, err, abort_flag);
                if (!ok) break;
                const int n = cur.next_len();
                const int u = (int)(cur.g / I), i0 = (int)(cur.g % I);
                const int e = a.ws.uniq[u];
                unsigned char *dst = ring + (size_t)slot * stage_bytes;
                const size_t row0 = (size_t)e * I + i0;
                if (!FP4) {
                    const uint32_t nb = (uint32_t)(n * rb);
                    mbar_arrive_expect_tx(&full[slot], 2 * nb);
                    bulk_g2s(dst, a.wg + row0 * d, nb, &full[slot], pol);
                    bulk_g2s(dst + kGuRowsPerStage * rb, a.wu + row0 * d, nb, &full[slot], pol);
                } else {
                    const uint32_t nq = (uint32_t)(n * (d / 2)), ns_ = (uint32_t)(n * (d / 16));
                    mbar_arrive_expect_tx(&full[slot], 2 * (nq + ns_));
                    unsigned char *gq = dst, *gs = dst + kGuRowsPerStage * (d / 2);
                    unsigned char *uq = dst + kGuRowsPerStage * rb, *us = uq + kGuRowsPerStage * (d / 2);
                    bulk_g2s(gq, a.qg + row0 * (d / 2), nq, &full[slot], pol);
                    bulk_g2s(gs, a.sg + row0 * (d / 16), ns_, &full[slot], pol);
                    bulk_g2s(uq, a.qu + row0 * (d / 2), nq, &full[slot], pol);
                    bulk_g2s(us, a.su + row0 * (d / 16), ns_, &full[slot], pol);
                }
                cur.g += n;
                ++s;
            }
            // drain: every copy issued must land before the CTA exits
            for (int j = (s > NS ? s - NS : 0); j < s; ++j) mbar_wait(&full[j % NS], (j / NS) & 1, err);
            mbar_wait(xbar, 0, err);
        }
        return;
    }

    // -------------------------------- consumers --------------------------------
    const int rr = warp / kParts, part = warp % kParts;
    mbar_wait_or_abort(xbar, 0, err, abort_flag);
    named_bar(1, 32 * kConsumerWarps);
    if (*abort_flag) return;
    StageCursor cur{g_begin, g_end, I, kGuRowsPerStage};
    int s = 0;
    int seg_u = -1, n_e = 0, row_base = 0, e = 0;
    int tok[TM];
#pragma unroll
    for (int r = 0; r < TM; ++r) tok[r] = 0;
    const int kpart = d / kParts;  // columns per part
    while (cur.g < cur.end) {
        const int slot = s % NS;
        const int n = cur.next_len();
        const int u = (int)(cur.g / I), i0 = (int)(cur.g % I);
        if (u != seg_u) {
            seg_u = u;
            e = a.ws.uniq[u];
            n_e = a.ws.counts[e];
            row_base = a.ws.offsets[e];
            if (n_e > TM) {  // cannot happen when T <= TM
                atomicOr(err, ERRBIT_RANGE);
                n_e = TM;
            }
#pragma unroll
            for (int r = 0; r < TM; ++r) tok[r] = (r < n_e) ? a.ws.perm[row_base + r] : 0;
        }
        const bool ok = mbar_wait_or_abort(&full[slot], (s / NS) & 1, err, abort_flag);
        const unsigned char *st = ring + (size_t)slot * stage_bytes;
        float accg[TM], accu[TM];
#pragma unroll
        for (int r = 0; r < TM; ++r) accg[r] = accu[r] = 0.f;
        if (ok && rr < n) {
            if (!FP4) {
                const uint4 *gw = reinterpret_cast<const uint4 *>(st + rr * rb) + part * (kpart / 8);
                const uint4 *uw = reinterpret_cast<const uint4 *>(st + (kGuRowsPerStage + rr) * rb) + part * (kpart / 8);
                for (int v = lane; v < kpart / 8; v += 32) {
                    float gf[8], uf[8];
                    unpack8(gw[v], gf);
                    unpack8(uw[v], uf);
#pragma unroll
                    for (int r = 0; r < TM; ++r) {
                        if (r < n_e) {
                            uint4 xv = reinterpret_cast<const uint4 *>(xs + (size_t)tok[r] * d * 2)[part * (kpart / 8) + v];
                            accg[r] += dot8(gf, xv);
                            accu[r] += dot8(uf, xv);
                        }
                    }
                }
            } else {
                const unsigned char *gq = st, *gs = st + kGuRowsPerStage * (d / 2);
                const unsigned char *uq = st + kGuRowsPerStage * rb, *us = uq + kGuRowsPerStage * (d / 2);
                // one 16-element block per lane iteration
                const int nblk = kpart / 16, blk0 = part * nblk;
                for (int b = lane; b < nblk; b += 32) {
                    const int blk = blk0 + b;
                    float gf[16], uf[16];
                    unpack_fp4x16(*reinterpret_cast<const uint2 *>(gq + (size_t)rr * (d / 2) + blk * 8), gf);
                    unpack_fp4x16(*reinterpret_cast<const uint2 *>(uq + (size_t)rr * (d / 2) + blk * 8), uf);
                    const float sgb = e4m3_to_f32(gs[(size_t)rr * (d / 16) + blk]);
                    const float sub = e4m3_to_f32(us[(size_t)rr * (d / 16) + blk]);
#pragma unroll
                    for (int r = 0; r < TM; ++r) {
                        if (r < n_e) {
                            const uint4 *xp = reinterpret_cast<const uint4 *>(xs + (size_t)tok[r] * d * 2) + blk * 2;
                            uint4 x0 = xp[0], x1 = xp[1];
                            float pg = dot8(gf, x0) + dot8(gf + 8, x1);
                            float pu = dot8(uf, x0) + dot8(uf + 8, x1);
                            accg[r] = fmaf(pg, sgb, accg[r]);
                            accu[r] = fmaf(pu, sub, accu[r]);
                        }
                    }
                }
            }
        }
        float *rd = red + (size_t)(s & 1) * kGuRowsPerStage * kParts * TM * 2;
#pragma unroll
        for (int r = 0; r < TM; ++r) {
            if (r < n_e) {
                float sg_ = warp_sum(accg[r]);
                float su_ = warp_sum(accu[r]);
                if (lane == 0) {
                    rd[((rr * kParts + part) * TM + r) * 2 + 0] = sg_;
                    rd[((rr * kParts + part) * TM + r) * 2 + 1] = su_;
                }
            }
        }
        __syncwarp();
        if (lane == 0 && ok) mbar_arrive(&empty[slot]);
        named_bar(1, 32 * kConsumerWarps);
        if (*abort_flag) return;
        // rows rr < n, tokens r < n_e: h = silu(g) * u
        if (part == 0 && rr < n && lane < n_e) {
            float g = 0.f, uu = 0.f;
#pragma unroll
            for (int p = 0; p < kParts; ++p) {
                g += rd[((rr * kParts + p) * TM + lane) * 2 + 0];
                uu += rd[((rr * kParts + p) * TM + lane) * 2 + 1];
            }
            if (FP4) {
                g *= a.gg[e];
                uu *= a.gu[e];
            }
            a.ws.h[(size_t)(row_base + lane) * I + i0 + rr] = silu(g) * uu;
        }
        cur.g += n;
        ++s;
    }
}

// ---------------------------------------------------------------------------
// down kernel
// ---------------------------------------------------------------------------
template <int TM, bool FP4>
__global__ void __launch_bounds__(kDecodeThreads, 1) decode_down_kernel(DecodeArgs a) {
    extern __shared__ __align__(128) unsigned char smem[];
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int d = a.d, I = a.I, NS = a.nstages;
    uint32_t *err = &a.ws.ctrl->err;

    uint64_t *full = reinterpret_cast<uint64_t *>(smem);
    uint64_t *empty = full + kMaxStages;
    volatile int *abort_flag = reinterpret_cast<volatile int *>(empty + kMaxStages);
    float *hs = reinterpret_cast<float *>(smem + 256);  // [TM][I]
    const size_t h_bytes = sizeof(float) * TM * I;
    unsigned char *ring = smem + 256 + ((h_bytes + 127) / 128) * 128;
    const size_t rb = row_bytes<FP4>(I);
    const size_t stage_bytes = kDnRowsPerStage * rb;

    if (tid == 0) {
        for (int s = 0; s < NS; ++s) {
            mbar_init(&full[s], 1);
            mbar_init(&empty[s], kConsumerWarps);
        }
        *abort_flag = 0;
        fence_barrier_init();
    }
    __syncthreads();

    const long long G = (long long)a.ws.ctrl->n_uniq * d;
    const long long g_begin = (long long)blockIdx.x * G / gridDim.x;
    const long long g_end = (long long)(blockIdx.x + 1) * G / gridDim.x;

    if (warp == kConsumerWarps) {
        if (lane == 0) {
            const uint64_t pol = policy_evict_first();
            StageCursor cur{g_begin, g_end, d, kDnRowsPerStage};
            int s = 0;
            bool ok = true;
            while (cur.g < cur.end && ok) {
                const int slot = s % NS;
                if (s >= NS) ok = mbar_wait_or_abort(&empty[slot], ((s / NS) - 1) & 1, err, abort_flag);
                if (!ok) break;
                const int n = cur.next_len();
                const int u = (int)(cur.g / d), c0 = (int)(cur.g % d);
                const int e = a.ws.uniq[u];
                unsigned char *dst = ring + (size_t)slot * stage_bytes;
                const size_t row0 = (size_t)e * d + c0;
                if (!FP4) {
                    mbar_arrive_expect_tx(&full[slot], (uint32_t)(n * rb));
                    bulk_g2s(dst, a.wd + row0 * I, (uint32_t)(n * rb), &full[slot], pol);
                } else {
                    const uint32_t nq = (uint32_t)(n * (I / 2)), ns_ = (uint32_t)(n * (I / 16));
                    mbar_arrive_expect_tx(&full[slot], nq + ns_);
                    bulk_g2s(dst, a.qd + row0 * (I / 2), nq, &full[slot], pol);
                    bulk_g2s(dst + kDnRowsPerStage * (I / 2), a.sd + row0 * (I / 16), ns_, &full[slot], pol);
                }
                cur.g += n;
                ++s;
            }
            for (int j = (s > NS ? s - NS : 0); j < s; ++j) mbar_wait(&full[j % NS], (j / NS) & 1, err);
        }
        return;
    }

    StageCursor cur{g_begin, g_end, d, kDnRowsPerStage};
    int s = 0;
    int seg_u = -1, n_e = 0, row_base = 0, e = 0;
    float gscale = 1.f;
    while (cur.g < cur.end) {
        const int slot = s % NS;
        const int n = cur.next_len();
        const int u = (int)(cur.g / d), c0 = (int)(cur.g % d);
        if (u != seg_u) {
            // new expert: reload its h rows into shared memory
            named_bar(1, 32 * kConsumerWarps);
            seg_u = u;
            e = a.ws.uniq[u];
            n_e = a.ws.counts[e];
            row_base = a.ws.offsets[e];
            if (n_e > TM) {
                atomicOr(err, ERRBIT_RANGE);
                n_e = TM;
            }
            if (FP4) gscale = a.gd[e];
            const float4 *src = reinterpret_cast<const float4 *>(a.ws.h + (size_t)row_base * I);
            float4 *dst = reinterpret_cast<float4 *>(hs);
            for (int i = tid; i < n_e * I / 4; i += 32 * kConsumerWarps) dst[i] = __ldcg(src + i);
            named_bar(1, 32 * kConsumerWarps);
        }
        const bool ok = mbar_wait_or_abort(&full[slot], (s / NS) & 1, err, abort_flag);
        const unsigned char *st = ring + (size_t)slot * stage_bytes;
        float acc[TM];
#pragma unroll
        for (int r = 0; r < TM; ++r) acc[r] = 0.f;
        if (ok && warp < n) {
            if (!FP4) {
                const uint4 *wrow = reinterpret_cast<const uint4 *>(st + warp * rb);
                for (int v = lane; v < I / 8; v += 32) {
                    float wf[8];
                    unpack8(wrow[v], wf);
#pragma unroll
                    for (int r = 0; r < TM; ++r) {
                        if (r < n_e) {
                            const float4 *hp = reinterpret_cast<const float4 *>(hs + (size_t)r * I + v * 8);
                            float4 h0 = hp[0], h1 = hp[1];
                            float t = wf[0] * h0.x;
                            t = fmaf(wf[1], h0.y, t);
                            t = fmaf(wf[2], h0.z, t);
                            t = fmaf(wf[3], h0.w, t);
                            t = fmaf(wf[4], h1.x, t);
                            t = fmaf(wf[5], h1.y, t);
                            t = fmaf(wf[6], h1.z, t);
                            t = fmaf(wf[7], h1.w, t);
                            acc[r] += t;
                        }
                    }
                }
            } else {
                const unsigned char *q = st + (size_t)warp * (I / 2);
                const unsigned char *sc = st + kDnRowsPerStage * (I / 2) + (size_t)warp * (I / 16);
                for (int b = lane; b < I / 16; b += 32) {
                    float wf[16];
                    unpack_fp4x16(*reinterpret_cast<const uint2 *>(q + b * 8), wf);
                    const float sb = e4m3_to_f32(sc[b]);
#pragma unroll
                    for (int r = 0; r < TM; ++r) {
                        if (r < n_e) {
                            const float4 *hp = reinterpret_cast<const float4 *>(hs + (size_t)r * I + b * 16);
                            float t = 0.f;
#pragma unroll
                            for (int qd = 0; qd < 4; ++qd) {
                                float4 hv = hp[qd];
                                t = fmaf(wf[4 * qd + 0], hv.x, t);
                                t = fmaf(wf[4 * qd + 1], hv.y, t);
                                t = fmaf(wf[4 * qd + 2], hv.z, t);
                                t = fmaf(wf[4 * qd + 3], hv.w, t);
                            }
                            acc[r] = fmaf(t, sb, acc[r]);
                        }
                    }
                }
            }
        }
        __syncwarp();
        if (lane == 0 && ok) mbar_arrive(&empty[slot]);
        named_bar(1, 32 * kConsumerWarps);
        if (*abort_flag) return;
        if (warp < n) {
#pragma unroll
            for (int r = 0; r < TM; ++r) {
                if (r < n_e) {
                    float sum = warp_sum(acc[r]);
                    if (lane == r) a.ws.Y[(size_t)(row_base + r) * d + c0 + warp] = sum * gscale;
                }
            }
        }
        cur.g += n;
        ++s;
    }
}

// ---------------------------------------------------------------------------
// launch
// ---------------------------------------------------------------------------
template <int TM, bool FP4>
static cudaError_t launch_gateup_t(const LayerDev &L, const DecodeArgs &a0, cudaStream_t st) {
    DecodeArgs a = a0;
    constexpr int kParts = kConsumerWarps / kGuRowsPerStage;
    size_t red_bytes = sizeof(float) * 2 * kGuRowsPerStage * kParts * TM * 2;
    size_t fixed = 256 + align_up(red_bytes, 128) + align_up((size_t)a.T * L.d * 2, 128);
    size_t stage = 2 * kGuRowsPerStage * row_bytes<FP4>(L.d);
    if (fixed + 2 * stage > (size_t)kSmemBudget) return cudaErrorInvalidConfiguration;
    int ns = (int)((kSmemBudget - fixed) / stage);
    a.nstages = ns > kMaxStages ? kMaxStages : ns;
    size_t smem = fixed + (size_t)a.nstages * stage;
    static bool attr = false;
    if (!attr) {
        cudaError_t e = cudaFuncSetAttribute(decode_gateup_kernel<TM, FP4>,
                                             cudaFuncAttributeMaxDynamicSharedMemorySize, kSmemBudget);
        if (e != cudaSuccess) return e;
        attr = true;
    }
    decode_gateup_kernel<TM, FP4><<<L.num_sms, kDecodeThreads, smem, st>>>(a);
    return cudaGetLastError();
}

template <int TM, bool FP4>
static cudaError_t launch_down_t(const LayerDev &L, const DecodeArgs &a0, cudaStream_t st) {
    DecodeArgs a = a0;
    size_t fixed = 256 + align_up(sizeof(float) * TM * L.I, 128);
    size_t stage = kDnRowsPerStage * row_bytes<FP4>(L.I);
    if (fixed + 2 * stage > (size_t)kSmemBudget) return cudaErrorInvalidConfiguration;
    int ns = (int)((kSmemBudget - fixed) / stage);
    a.nstages = ns > kMaxStages ? kMaxStages : ns;
    size_t smem = fixed + (size_t)a.nstages * stage;
    static bool attr = false;
    if (!attr) {
        cudaError_t e = cudaFuncSetAttribute(decode_down_kernel<TM, FP4>,
                                             cudaFuncAttributeMaxDynamicSharedMemorySize, kSmemBudget);
        if (e != cudaSuccess) return e;
        attr = true;
    }
    decode_down_kernel<TM, FP4><<<L.num_sms, kDecodeThreads, smem, st>>>(a);
    return cudaGetLastError();
}

template <bool FP4, bool DOWN>
static cudaError_t launch_fmt(const LayerDev &L, const DecodeArgs &a, cudaStream_t st) {
    const int T = a.T;
#define MOE_DEC(TMV) return DOWN ? launch_down_t<TMV, FP4>(L, a, st) : launch_gateup_t<TMV, FP4>(L, a, st)
    if (T <= 1) MOE_DEC(1);
    if (T <= 2) MOE_DEC(2);
    if (T <= 4) MOE_DEC(4);
    if (T <= 8) MOE_DEC(8);
    if (T <= 16) MOE_DEC(16);
#undef MOE_DEC
    return cudaErrorInvalidValue;
}

static DecodeArgs make_args(const LayerDev &L, const Workspace &ws, const uint16_t *x, int T) {
    return DecodeArgs{x, L.wg, L.wu, L.wd, L.qg, L.qu, L.qd, L.sg, L.su, L.sd, L.gg, L.gu, L.gd,
                      T, L.d, L.I, L.k, 0, ws};
}

cudaError_t launch_decode_gateup(const LayerDev &L, const Workspace &ws, const uint16_t *x, int T, cudaStream_t st) {
    DecodeArgs a = make_args(L, ws, x, T);
    return L.fmt == MOE_W_NVFP4 ? launch_fmt<true, false>(L, a, st) : launch_fmt<false, false>(L, a, st);
}

cudaError_t launch_decode_down(const LayerDev &L, const Workspace &ws, const uint16_t *x, int T, cudaStream_t st) {
    DecodeArgs a = make_args(L, ws, x, T);
    return L.fmt == MOE_W_NVFP4 ? launch_fmt<true, true>(L, a, st) : launch_fmt<false, true>(L, a, st);
}

}  // namespace moe
