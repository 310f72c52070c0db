// decode.cu — the split streaming expert stage (two launches per chunk of at
// most 16 tokens), used for NVFP4 batches of more than 16 tokens, which the
// bf16 grouped GEMMs of the prefill path do not take. The single-launch layer
// kernel (decode_fused.cuh) covers every batch of at most 16 tokens.
//
// Decode-sized chunks are bound by streaming weights from HBM, not by matmul
// speed, and fetching weights ahead of the compute that needs them hides the
// wait ("How SGLang-TorchTPU accelerated an 816B-parameter MoE on TPU v7",
// sections "Introduction" and "Key optimisations"). With at most 16 tokens
// per chunk an expert sees about one token, so each weight element feeds 1-2
// FMAs and the work is a memory stream.
//
// Two persistent kernels, grid = one CTA per SM:
//   gate/up:  h[r, i] = silu(Wg[e,i,:] . x_t) * (Wu[e,i,:] . x_t)   (fp32)
//   down:     Y[r, c] = Wd[e,c,:] . h[r, :]                          (fp32)
// where r runs over the rows of the permuted (token, slot) order of expert e.
// The flattened rows of all active experts are split evenly over the CTAs,
// so every SM streams the same number of bytes whatever the routing.
// Warp roles: warp 8 (one lane) fills the ring; stage s is consumed by warp
// s % ncons alone (a whole gate/up row pair, or four down rows; ncons <= 8),
// so the consumer warps drain different stages at once and never wait for
// each other. Both kernels are launched as programmatic dependents of the kernel
// before them: their prologue overlaps its tail, and the down kernel starts
// streaming its weights before the gate/up results it consumes are complete.
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
constexpr int kDnRows = 4;           // down: rows c per stage
constexpr int kMaxStages = 16;
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
    // Consumer warps in use; nstages is a multiple of ncons, so slot j is only
    // ever consumed by warp j % ncons and each warp takes the phases of its own
    // slots in order. A wait by phase parity is then never more than one phase
    // ahead of the slot (bulk copies may complete out of issue order, so a
    // slot shared between warps could show a stale phase of the same parity).
    int ncons;
    Workspace ws;
    int64_t gu_ld;           // elements from one gate (or up) row to the next
};

// ---------------------------------------------------------------------------
// helpers
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

__device__ __forceinline__ float dot8h(const float w[8], float4 h0, float4 h1) {
    float t = w[0] * h0.x;
    t = fmaf(w[1], h0.y, t);
    t = fmaf(w[2], h0.z, t);
    t = fmaf(w[3], h0.w, t);
    t = fmaf(w[4], h1.x, t);
    t = fmaf(w[5], h1.y, t);
    t = fmaf(w[6], h1.z, t);
    t = fmaf(w[7], h1.w, t);
    return t;
}

// 8 packed bytes -> 16 E2M1 values (exact in fp32), low nibble first
__device__ __forceinline__ void unpack_fp4x16(uint2 q, float f[16]) {
    uint32_t words[2] = {q.x, q.y};
#pragma unroll
    for (int wi = 0; wi < 2; ++wi) {
#pragma unroll
        for (int b = 0; b < 4; ++b) {
            __nv_fp4x2_storage_t byte = (__nv_fp4x2_storage_t)((words[wi] >> (8 * b)) & 0xFFu);
            __half2_raw hr = __nv_cvt_fp4x2_to_halfraw2(byte, __NV_E2M1);
            float2 p = __half22float2(*reinterpret_cast<__half2 *>(&hr));
            f[wi * 8 + 2 * b] = p.x;
            f[wi * 8 + 2 * b + 1] = p.y;
        }
    }
}

__device__ __forceinline__ float e4m3_to_f32(uint8_t s) {
    __half_raw hr = __nv_cvt_fp8_to_halfraw((__nv_fp8_storage_t)s, __NV_E4M3);
    return __half2float(*reinterpret_cast<__half *>(&hr));
}

// Programmatic dependent launch: wait for the grid this one depends on (a
// no-op when launched without the attribute); let the next grid launch.
__device__ __forceinline__ void grid_dep_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
__device__ __forceinline__ void grid_dep_launch() { asm volatile("griddepcontrol.launch_dependents;" ::: "memory"); }

// Per-warp cache of the expert a stage belongs to.
template <int TM>
struct ExpertSeg {
    int u = -1, e = 0, n_e = 0, row_base = 0;
    int tok[TM];
    __device__ __forceinline__ void load(const Workspace &ws, int uu, uint32_t *err) {
        u = uu;
        e = ws.uniq[uu];
        n_e = ws.counts[e];
        row_base = ws.offsets[e];
        if (n_e > TM) {  // cannot happen when T <= TM
            atomicOr(err, ERRBIT_RANGE);
            n_e = TM;
        }
#pragma unroll
        for (int r = 0; r < TM; ++r) tok[r] = (r < n_e) ? ws.perm[row_base + r] : 0;
    }
};

// ---------------------------------------------------------------------------
// gate/up kernel: stage s = row pair g_begin + s (gate row i and up row i)
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
    unsigned char *xs = smem + 512;
    const uint32_t x_bytes = (uint32_t)a.T * d * 2;
    unsigned char *ring = xs + ((x_bytes + 127) / 128) * 128;
    const uint32_t rb = (uint32_t)row_bytes<FP4>(d);
    const uint32_t stage_bytes = 2 * rb;

    if (tid == 0) {
        for (int s = 0; s < NS; ++s) {
            mbar_init(&full[s], 1);
            mbar_init(&empty[s], 1);
        }
        mbar_init(xbar, 1);
        *abort_flag = 0;
        fence_barrier_init();
    }
    __syncthreads();
    grid_dep_wait();      // routing results of the previous kernel
    grid_dep_launch();

    const int G = a.ws.ctrl->n_uniq * I;
    const int g_begin = (int)((long long)blockIdx.x * G / gridDim.x);
    const int n_st = (int)((long long)(blockIdx.x + 1) * G / gridDim.x) - g_begin;

    if (warp == kConsumerWarps) {
        // ------------------------------ producer ------------------------------
        if (lane == 0) {
            const uint64_t pol = policy_evict_first();
            mbar_arrive_expect_tx(xbar, x_bytes);
            bulk_g2s(xs, a.x, x_bytes, xbar, policy_evict_last());
            int s = 0;
            for (; s < n_st; ++s) {
                const int slot = s % NS;
                if (s >= NS && !mbar_wait_or_abort(&empty[slot], ((s / NS) - 1) & 1, err, abort_flag)) break;
                const int g = g_begin + s;
                const int u = g / I, i = g - u * I;
                const size_t row = (size_t)a.ws.uniq[u] * I + i;
                unsigned char *dst = ring + (size_t)slot * stage_bytes;
                mbar_arrive_expect_tx(&full[slot], stage_bytes);
                if (!FP4) {
                    bulk_g2s(dst, a.wg + (int64_t)row * a.gu_ld, rb, &full[slot], pol);
                    bulk_g2s(dst + rb, a.wu + (int64_t)row * a.gu_ld, rb, &full[slot], pol);
                } else {
                    const uint32_t nq = d / 2, nsb = d / 16;
                    bulk_g2s(dst, a.qg + row * nq, nq, &full[slot], pol);
                    bulk_g2s(dst + nq, a.sg + row * nsb, nsb, &full[slot], pol);
                    bulk_g2s(dst + rb, a.qu + row * nq, nq, &full[slot], pol);
                    bulk_g2s(dst + rb + nq, a.su + row * nsb, nsb, &full[slot], pol);
                }
            }
            // every copy issued must land before the CTA exits
            for (int j = (s > NS ? s - NS : 0); j < s; ++j) mbar_wait(&full[j % NS], (j / NS) & 1, err);
            mbar_wait(xbar, 0, err);
        }
        return;
    }

    // -------------------------------- consumers --------------------------------
    if (warp >= a.ncons) return;
    if (!mbar_wait_or_abort(xbar, 0, err, abort_flag)) return;
    ExpertSeg<TM> seg;
    for (int s = warp; s < n_st; s += a.ncons) {
        const int slot = s % NS;
        const int g = g_begin + s;
        const int u = g / I, i = g - u * I;
        if (u != seg.u) seg.load(a.ws, u, err);
        if (!mbar_wait_or_abort(&full[slot], (s / NS) & 1, err, abort_flag)) return;
        const unsigned char *st = ring + (size_t)slot * stage_bytes;
        float accg[TM], accu[TM];
#pragma unroll
        for (int r = 0; r < TM; ++r) accg[r] = accu[r] = 0.f;
        if (!FP4) {
            const uint4 *gw = reinterpret_cast<const uint4 *>(st);
            const uint4 *uw = reinterpret_cast<const uint4 *>(st + rb);
            for (int v = lane; v < d / 8; v += 32) {
                float gf[8], uf[8];
                unpack8(gw[v], gf);
                unpack8(uw[v], uf);
#pragma unroll
                for (int r = 0; r < TM; ++r) {
                    if (r < seg.n_e) {
                        const uint4 xv = reinterpret_cast<const uint4 *>(xs + (size_t)seg.tok[r] * d * 2)[v];
                        accg[r] += dot8(gf, xv);
                        accu[r] += dot8(uf, xv);
                    }
                }
            }
        } else {
            const unsigned char *gq = st, *gs = st + d / 2, *uq = st + rb, *us = st + rb + d / 2;
            for (int b = lane; b < d / 16; b += 32) {
                float gf[16], uf[16];
                unpack_fp4x16(*reinterpret_cast<const uint2 *>(gq + b * 8), gf);
                unpack_fp4x16(*reinterpret_cast<const uint2 *>(uq + b * 8), uf);
                const float sgb = e4m3_to_f32(gs[b]), sub = e4m3_to_f32(us[b]);
#pragma unroll
                for (int r = 0; r < TM; ++r) {
                    if (r < seg.n_e) {
                        const uint4 *xp = reinterpret_cast<const uint4 *>(xs + (size_t)seg.tok[r] * d * 2) + b * 2;
                        const uint4 x0 = xp[0], x1 = xp[1];
                        accg[r] = fmaf(dot8(gf, x0) + dot8(gf + 8, x1), sgb, accg[r]);
                        accu[r] = fmaf(dot8(uf, x0) + dot8(uf + 8, x1), sub, accu[r]);
                    }
                }
            }
        }
        __syncwarp();
        if (lane == 0) mbar_arrive(&empty[slot]);   // the stage's shared memory is free again
        const float gsc = FP4 ? a.gg[seg.e] : 1.f, usc = FP4 ? a.gu[seg.e] : 1.f;
        float hv = 0.f;
#pragma unroll
        for (int r = 0; r < TM; ++r) {
            if (r < seg.n_e) {
                const float sg_ = warp_sum(accg[r]) * gsc;
                const float su_ = warp_sum(accu[r]) * usc;
                if (lane == r) hv = silu(sg_) * su_;
            }
        }
        if (lane < seg.n_e) a.ws.h[(size_t)(seg.row_base + lane) * I + i] = hv;
    }
}

// ---------------------------------------------------------------------------
// down kernel: stage s = kDnRows consecutive rows c of one expert
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
    unsigned char *ring = smem + 512;
    const uint32_t rb = (uint32_t)row_bytes<FP4>(I);
    const uint32_t stage_bytes = kDnRows * rb;

    if (tid == 0) {
        for (int s = 0; s < NS; ++s) {
            mbar_init(&full[s], 1);
            mbar_init(&empty[s], 1);
        }
        *abort_flag = 0;
        fence_barrier_init();
    }
    __syncthreads();
    grid_dep_launch();

    // The routing records come from the kernel before the previous one, which
    // completed before the previous kernel started: the weight stream may
    // begin at once. Only h (from the previous kernel) needs the wait below.
    const int units = a.ws.ctrl->n_uniq * (d / kDnRows);
    const int u_begin = (int)((long long)blockIdx.x * units / gridDim.x);
    const int n_st = (int)((long long)(blockIdx.x + 1) * units / gridDim.x) - u_begin;

    if (warp == kConsumerWarps) {
        if (lane == 0) {
            const uint64_t pol = policy_evict_first();
            int s = 0;
            for (; s < n_st; ++s) {
                const int slot = s % NS;
                if (s >= NS && !mbar_wait_or_abort(&empty[slot], ((s / NS) - 1) & 1, err, abort_flag)) break;
                const int g = (u_begin + s) * kDnRows;
                const int u = g / d, c0 = g - u * d;
                const size_t row = (size_t)a.ws.uniq[u] * d + c0;
                unsigned char *dst = ring + (size_t)slot * stage_bytes;
                mbar_arrive_expect_tx(&full[slot], stage_bytes);
                if (!FP4) {
                    bulk_g2s(dst, a.wd + row * I, stage_bytes, &full[slot], pol);
                } else {
                    const uint32_t nq = I / 2, nsb = I / 16;
                    bulk_g2s(dst, a.qd + row * nq, kDnRows * nq, &full[slot], pol);
                    bulk_g2s(dst + kDnRows * nq, a.sd + row * nsb, kDnRows * nsb, &full[slot], pol);
                }
            }
            for (int j = (s > NS ? s - NS : 0); j < s; ++j) mbar_wait(&full[j % NS], (j / NS) & 1, err);
        }
        return;
    }

    if (warp >= a.ncons) return;
    grid_dep_wait();      // h from the gate/up kernel
    ExpertSeg<TM> seg;
    for (int s = warp; s < n_st; s += a.ncons) {
        const int slot = s % NS;
        const int g = (u_begin + s) * kDnRows;
        const int u = g / d, c0 = g - u * d;
        if (u != seg.u) seg.load(a.ws, u, err);
        if (!mbar_wait_or_abort(&full[slot], (s / NS) & 1, err, abort_flag)) return;
        const unsigned char *st = ring + (size_t)slot * stage_bytes;
        const float *hrow = a.ws.h + (size_t)seg.row_base * I;
        float acc[kDnRows][TM];
#pragma unroll
        for (int q = 0; q < kDnRows; ++q)
#pragma unroll
            for (int r = 0; r < TM; ++r) acc[q][r] = 0.f;
        if (!FP4) {
            for (int v = lane; v < I / 8; v += 32) {
                float wf[kDnRows][8];
#pragma unroll
                for (int q = 0; q < kDnRows; ++q) unpack8(reinterpret_cast<const uint4 *>(st + q * rb)[v], wf[q]);
#pragma unroll
                for (int r = 0; r < TM; ++r) {
                    if (r < seg.n_e) {
                        const float4 *hp = reinterpret_cast<const float4 *>(hrow + (size_t)r * I + v * 8);
                        const float4 h0 = __ldcg(hp), h1 = __ldcg(hp + 1);
#pragma unroll
                        for (int q = 0; q < kDnRows; ++q) acc[q][r] += dot8h(wf[q], h0, h1);
                    }
                }
            }
        } else {
            const unsigned char *qb = st, *sb = st + kDnRows * (I / 2);
            for (int b = lane; b < I / 16; b += 32) {
                float wf[kDnRows][16], sc[kDnRows];
#pragma unroll
                for (int q = 0; q < kDnRows; ++q) {
                    unpack_fp4x16(*reinterpret_cast<const uint2 *>(qb + q * (I / 2) + b * 8), wf[q]);
                    sc[q] = e4m3_to_f32(sb[q * (I / 16) + b]);
                }
#pragma unroll
                for (int r = 0; r < TM; ++r) {
                    if (r < seg.n_e) {
                        const float4 *hp = reinterpret_cast<const float4 *>(hrow + (size_t)r * I + b * 16);
                        const float4 h0 = __ldcg(hp), h1 = __ldcg(hp + 1), h2 = __ldcg(hp + 2), h3 = __ldcg(hp + 3);
#pragma unroll
                        for (int q = 0; q < kDnRows; ++q)
                            acc[q][r] = fmaf(dot8h(wf[q], h0, h1) + dot8h(wf[q] + 8, h2, h3), sc[q], acc[q][r]);
                    }
                }
            }
        }
        __syncwarp();
        if (lane == 0) mbar_arrive(&empty[slot]);
        const float gsc = FP4 ? a.gd[seg.e] : 1.f;
#pragma unroll
        for (int q = 0; q < kDnRows; ++q) {
            float yv = 0.f;
#pragma unroll
            for (int r = 0; r < TM; ++r) {
                if (r < seg.n_e) {
                    const float sum = warp_sum(acc[q][r]);
                    if (lane == r) yv = sum * gsc;
                }
            }
            if (lane < seg.n_e) a.ws.Y[(size_t)(seg.row_base + lane) * d + c0 + q] = yv;
        }
    }
}

// ---------------------------------------------------------------------------
// launch (programmatic dependent launches on the caller's stream)
// ---------------------------------------------------------------------------
template <typename K>
static cudaError_t launch_pdl(K kern, int grid, int threads, size_t smem, cudaStream_t st, const DecodeArgs &a) {
    cudaLaunchConfig_t cfg{};
    cfg.gridDim = dim3(grid);
    cfg.blockDim = dim3(threads);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = st;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, kern, a);
}

// Ring shape from the number of stages that fit: the most consumer warps c
// (<= 8) that still own at least two slots each, nstages = c * slots.
static void pick_stages(int fit, DecodeArgs &a) {
    if (fit > kMaxStages) fit = kMaxStages;
    for (int c = kConsumerWarps; c >= 1; --c) {
        if (fit / c >= 2) {
            a.ncons = c;
            a.nstages = (fit / c) * c;
            return;
        }
    }
    a.ncons = 1;
    a.nstages = fit;
}

template <int TM, bool FP4>
static cudaError_t launch_gateup_t(const LayerDev &L, const DecodeArgs &a0, cudaStream_t st) {
    DecodeArgs a = a0;
    const size_t fixed = 512 + align_up((size_t)a.T * L.d * 2, 128);
    const size_t stage = 2 * row_bytes<FP4>(L.d);
    if (fixed + 2 * stage > (size_t)kSmemBudget) return cudaErrorInvalidConfiguration;
    const int ns = (int)((kSmemBudget - fixed) / stage);
    pick_stages(ns, a);
    static std::atomic<uint64_t> attr_set{0};
    const cudaError_t e = set_smem_limit_once((const void *)decode_gateup_kernel<TM, FP4>, kSmemBudget, attr_set);
    if (e != cudaSuccess) return e;
    return launch_pdl(decode_gateup_kernel<TM, FP4>, L.num_sms, kDecodeThreads, fixed + (size_t)a.nstages * stage,
                      st, a);
}

template <int TM, bool FP4>
static cudaError_t launch_down_t(const LayerDev &L, const DecodeArgs &a0, cudaStream_t st) {
    DecodeArgs a = a0;
    const size_t fixed = 512;
    const size_t stage = kDnRows * row_bytes<FP4>(L.I);
    if (fixed + 2 * stage > (size_t)kSmemBudget) return cudaErrorInvalidConfiguration;
    const int ns = (int)((kSmemBudget - fixed) / stage);
    pick_stages(ns, a);
    static std::atomic<uint64_t> attr_set{0};
    const cudaError_t e = set_smem_limit_once((const void *)decode_down_kernel<TM, FP4>, kSmemBudget, attr_set);
    if (e != cudaSuccess) return e;
    return launch_pdl(decode_down_kernel<TM, FP4>, L.num_sms, kDecodeThreads, fixed + (size_t)a.nstages * stage, st,
                      a);
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
                      T, L.d, L.I, L.k, 0, 0, ws, L.gu_ld};
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
