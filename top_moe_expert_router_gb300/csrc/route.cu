// route.cu — router (bf16 x . Wr^T with fp32 accumulation), fp32 softmax,
// top-k with renormalisation, and the token permutation.
//
// Each token picks k of E experts (k = 8, E = 256 in "How SGLang-TorchTPU
// accelerated an 816B-parameter MoE on TPU v7", section "Introduction"). The
// permutation groups the (token, slot) pairs by expert, tokens ascending
// inside each expert, through a per-expert token bitmap: the result depends
// only on ids, never on the order in which threads run.
#include <cuda_runtime.h>
#include <math.h>

#include "common.cuh"
#include "decode_common.cuh"

namespace moe {

// ---------------------------------------------------------------------------
// permutation by one CTA
// ---------------------------------------------------------------------------
// Shared memory needed: (4 * (E + 1) * 4) + E * words * 4 bytes, words = chunk / 32.
struct PermSmem {
    int32_t *cnt, *off, *run, *scratch;
    uint32_t *bm;
    int words;  // bitmap words per expert (chunk of tokens = 32 * words)
};

// Exclusive scan of a[0..n) (n <= 256) by warp 0; returns the total. Only
// lanes of warp 0 call it.
__device__ int warp0_exclusive_scan(const int32_t *a, int32_t *out, int n, int lane) {
    int vals[8];
    int local = 0;
#pragma unroll
    for (int i = 0; i < 8; ++i) {
        int idx = lane * 8 + i;
        vals[i] = idx < n ? a[idx] : 0;
        local += vals[i];
    }
    int incl = local;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        int y = __shfl_up_sync(0xFFFFFFFFu, incl, o);
        if (lane >= o) incl += y;
    }
    int run = incl - local;
#pragma unroll
    for (int i = 0; i < 8; ++i) {
        int idx = lane * 8 + i;
        if (idx < n) out[idx] = run;
        run += vals[i];
    }
    return __shfl_sync(0xFFFFFFFFu, incl, 31);
}

// Permutation for T <= 32 tokens: bm[e] holds one bit per token routed to e,
// so the row of (t, j) is offsets[e] + popcount(bm[e] below bit t).
__device__ void permute_block_small(const int32_t *ids, int T, int k, int E, const Workspace &ws, PermSmem sm) {
    const int tid = threadIdx.x, nth = blockDim.x, lane = tid & 31, warp = tid >> 5;
    const int Tk = T * k;
    for (int e = tid; e < E; e += nth) sm.bm[e] = 0u;
    __syncthreads();
    for (int p = tid; p < Tk; p += nth) {
        const int e = ids[p];
        if ((unsigned)e < (unsigned)E)
            atomicOr(&sm.bm[e], 1u << (p / k));
        else
            atomicOr(&ws.ctrl->err, ERRBIT_RANGE);
    }
    __syncthreads();
    for (int e = tid; e < E; e += nth) {
        const int c = __popc(sm.bm[e]);
        sm.cnt[e] = c;
        sm.scratch[e] = c > 0 ? 1 : 0;
    }
    __syncthreads();
    if (warp == 0) {
        const int total = warp0_exclusive_scan(sm.cnt, sm.off, E, lane);
        const int nu = warp0_exclusive_scan(sm.scratch, sm.run, E, lane);
        __syncwarp();
        for (int e = lane; e < E; e += 32)
            if (sm.cnt[e] > 0) ws.uniq[sm.run[e]] = e;
        if (lane == 0) {
            sm.off[E] = total;
            ws.ctrl->n_uniq = nu;
        }
    }
    __syncthreads();
    for (int e = tid; e < E; e += nth) {
        ws.counts[e] = sm.cnt[e];
        ws.offsets[e] = sm.off[e];
        ws.tile_off[e] = 0;  // the grouped GEMM tiles are unused on the small path
    }
    if (tid == 0) {
        ws.offsets[E] = sm.off[E];
        ws.tile_off[E] = 0;
    }
    for (int p = tid; p < Tk; p += nth) {
        const int e = ids[p];
        if ((unsigned)e >= (unsigned)E) continue;
        const int t = p / k;
        const int row = sm.off[e] + __popc(sm.bm[e] & ((1u << t) - 1u));
        ws.perm[row] = t;
        ws.pos[p] = row;
    }
}

// ---------------------------------------------------------------------------
// Small-T route: router GEMV on all CTAs; the last CTA to finish runs top-k
// and the permutation (one launch for the whole routing step).
// ---------------------------------------------------------------------------
constexpr int kRouteSmallThreads = 256;
constexpr int kRouteExpertsPerCta = 2;

template <int TM>
__global__ void __launch_bounds__(kRouteSmallThreads) route_small_kernel(const uint16_t *__restrict__ x,
                                                                         const uint16_t *__restrict__ wr,
                                                                         const float *__restrict__ bias, int T, int d,
                                                                         int E, int k, Workspace ws) {
    extern __shared__ __align__(16) unsigned char smem_raw[];
    __shared__ float part[kRouteExpertsPerCta][4][TM];
    __shared__ int s_last;
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int eps = warp >> 2, q = warp & 3;
    const int e = blockIdx.x * kRouteExpertsPerCta + eps;
    const int nvec_q = d / 32;  // 16-byte vectors per quarter row
    // the expert stage that follows is launched as a programmatic dependent
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
    float acc[TM];
#pragma unroll
    for (int t = 0; t < TM; ++t) acc[t] = 0.f;
    if (e < E) {
        const uint4 *wrow = reinterpret_cast<const uint4 *>(wr + (size_t)e * d) + q * nvec_q;
#pragma unroll 4
        for (int v = lane; v < nvec_q; v += 32) {
            uint4 wv = __ldg(wrow + v);
            float wf[8] = {bf16lo(wv.x), bf16hi(wv.x), bf16lo(wv.y), bf16hi(wv.y),
                           bf16lo(wv.z), bf16hi(wv.z), bf16lo(wv.w), bf16hi(wv.w)};
#pragma unroll
            for (int t = 0; t < TM; ++t) {
                if (t < T) {
                    uint4 xv = __ldg(reinterpret_cast<const uint4 *>(x + (size_t)t * d) + q * nvec_q + v);
                    acc[t] = fmaf(wf[0], bf16lo(xv.x), acc[t]);
                    acc[t] = fmaf(wf[1], bf16hi(xv.x), acc[t]);
                    acc[t] = fmaf(wf[2], bf16lo(xv.y), acc[t]);
                    acc[t] = fmaf(wf[3], bf16hi(xv.y), acc[t]);
                    acc[t] = fmaf(wf[4], bf16lo(xv.z), acc[t]);
                    acc[t] = fmaf(wf[5], bf16hi(xv.z), acc[t]);
                    acc[t] = fmaf(wf[6], bf16lo(xv.w), acc[t]);
                    acc[t] = fmaf(wf[7], bf16hi(xv.w), acc[t]);
                }
            }
        }
    }
#pragma unroll
    for (int t = 0; t < TM; ++t) {
        float s = warp_sum(acc[t]);
        if (lane == 0) part[eps][q][t] = s;
    }
    __syncthreads();
    if (tid < kRouteExpertsPerCta * TM) {
        int ee = tid / TM, t = tid % TM;
        int eg = blockIdx.x * kRouteExpertsPerCta + ee;
        if (eg < E && t < T) {
            float l = ((part[ee][0][t] + part[ee][1][t]) + part[ee][2][t]) + part[ee][3][t];
            if (bias) l += bias[eg];
            ws.logits[(size_t)t * E + eg] = l;
        }
    }
    // last-CTA hand-off: every CTA publishes its logits, counts itself in;
    // the CTA that completes the count runs the rest of the routing step.
    __threadfence();
    __syncthreads();
    if (tid == 0) s_last = (atomicAdd(&ws.ctrl->route_done, 1u) == gridDim.x - 1);
    __syncthreads();
    if (!s_last) return;
    __threadfence();
    if (tid == 0) ws.ctrl->route_done = 0u;
    for (int t = warp; t < T; t += kRouteSmallThreads / 32)
        topk_warp(ws.logits + (size_t)t * E, E, k, ws.ids + (size_t)t * k, ws.w + (size_t)t * k, true);
    __syncthreads();
    int32_t *si = reinterpret_cast<int32_t *>(smem_raw);
    PermSmem sm{si, si + (E + 1), si + 2 * (E + 1), si + 3 * (E + 1),
                reinterpret_cast<uint32_t *>(si + 4 * (E + 1)), 1};
    permute_block_small(ws.ids, T, k, E, ws, sm);
}

static size_t perm_smem_bytes(int E, int words) { return (size_t)4 * (E + 1) * 4 + (size_t)E * words * 4; }

cudaError_t launch_route_small(const LayerDev &L, const Workspace &ws, const uint16_t *x, int T, cudaStream_t st) {
    int grid = (L.E + kRouteExpertsPerCta - 1) / kRouteExpertsPerCta;
    size_t smem = perm_smem_bytes(L.E, 1);
#define MOE_ROUTE_SMALL(TMV) \
    route_small_kernel<TMV><<<grid, kRouteSmallThreads, smem, st>>>(x, L.wr, L.bias, T, L.d, L.E, L.k, ws)
    if (T <= 1)
        MOE_ROUTE_SMALL(1);
    else if (T <= 2)
        MOE_ROUTE_SMALL(2);
    else if (T <= 4)
        MOE_ROUTE_SMALL(4);
    else if (T <= 8)
        MOE_ROUTE_SMALL(8);
    else if (T <= 16)
        MOE_ROUTE_SMALL(16);
    else if (T <= 32)
        MOE_ROUTE_SMALL(32);
    else
        return cudaErrorInvalidValue;
#undef MOE_ROUTE_SMALL
    return cudaGetLastError();
}

// ---------------------------------------------------------------------------
// Large-T route: router GEMM on the tensor cores (prefill.cu), then
//   route_chunk_kernel: one CTA per 256-token chunk runs top-k (one warp per
//     token), builds the chunk's per-expert token bitmap and counts; the last
//     CTA to finish scans the counts over experts and chunks;
//   route_scatter_kernel: one CTA per chunk places every (token, slot) pair at
//     chunk_base[chunk][e] + (tokens of e earlier in the chunk).
// ---------------------------------------------------------------------------
constexpr int kChunk = kRouteChunk;      // tokens per chunk: one bitmap word per expert
static_assert(kChunk == 32, "one 32-bit bitmap word per expert and chunk");

__global__ void __launch_bounds__(256) route_chunk_kernel(int T, int k, int E, int nsplit, size_t split_stride,
                                                          Workspace ws) {
    __shared__ uint32_t bm[256];
    __shared__ int32_t s_cnt[257], s_off[257], s_flag[257], s_idx[257];
    __shared__ int s_last;
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int c = blockIdx.x, t0 = c * kChunk;
    const int nt = min(kChunk, T - t0);
    for (int i = tid; i < E; i += 256) bm[i] = 0u;
    __syncthreads();
    __shared__ float s_row[8][256];  // one token's summed logits per warp
    for (int tl = warp; tl < nt; tl += 8) {
        const int t = t0 + tl;
        // the logits' parts over K: every load issued first, then added in order
        const float *row = ws.logits + (size_t)t * E;
        float part[kRouterSplit][8];
#pragma unroll
        for (int s = 0; s < kRouterSplit; ++s)
#pragma unroll
            for (int i = 0; i < 8; ++i) {
                const int e = lane + 32 * i;
                part[s][i] = (s < nsplit && e < E) ? row[(size_t)s * split_stride + e] : 0.f;
            }
#pragma unroll
        for (int i = 0; i < 8; ++i) {
            const int e = lane + 32 * i;
            float l = part[0][i];
#pragma unroll
            for (int s = 1; s < kRouterSplit; ++s)
                if (s < nsplit) l += part[s][i];
            if (e < E) s_row[warp][e] = l;
        }
        __syncwarp();
        {
            // lane l takes experts 8l .. 8l+7 (the small-batch kernels' top-k)
            uint32_t key[8];
#pragma unroll
            for (int i = 0; i < 8; ++i) {
                const int e = 8 * lane + i;
                key[i] = e < E ? fused::expert_key(s_row[warp][e]) : 0u;
            }
            fused::topk_sorted(key, k, ws.ids + (size_t)t * k, ws.w + (size_t)t * k);
        }
        __syncwarp();
        if (lane < k) {
            const int e = ws.ids[(size_t)t * k + lane];
            atomicOr(&bm[e], 1u << tl);
        }
    }
    __syncthreads();
    uint32_t *gbm = ws.chunk_bm + (size_t)c * E;
    for (int e = tid; e < E; e += 256) {
        gbm[e] = bm[e];
        ws.chunk_base[(size_t)c * E + e] = __popc(bm[e]);
    }
    // last-CTA hand-off: the CTA that completes the count scans for everyone
    __threadfence();
    __syncthreads();
    if (tid == 0) s_last = (atomicAdd(&ws.ctrl->route_done, 1u) == gridDim.x - 1);
    __syncthreads();
    if (!s_last) return;
    __threadfence();
    const int nch = gridDim.x;
    // per-chunk counts are read 64 at a time, all loads of a batch issued
    // before any use: one L2 round trip per batch, not per chunk
    constexpr int kBatch = 64;
    for (int e = tid; e < E; e += 256) {
        int n = 0;
        for (int c0 = 0; c0 < nch; c0 += kBatch) {
            int v[kBatch];
#pragma unroll
            for (int j = 0; j < kBatch; ++j) v[j] = c0 + j < nch ? __ldcg(ws.chunk_base + (size_t)(c0 + j) * E + e) : 0;
#pragma unroll
            for (int j = 0; j < kBatch; ++j) n += v[j];
        }
        s_cnt[e] = n;
        s_flag[e] = n > 0 ? 1 : 0;
    }
    __syncthreads();
    if (warp == 0) {
        const int total = warp0_exclusive_scan(s_cnt, s_off, E, lane);
        const int nu = warp0_exclusive_scan(s_flag, s_idx, E, lane);
        __syncwarp();
        for (int e = lane; e < E; e += 32) {
            if (s_cnt[e] > 0) ws.uniq[s_idx[e]] = e;
            s_flag[e] = (s_cnt[e] + 127) >> 7;       // 128-row tiles of the grouped GEMMs
        }
        __syncwarp();
        const int ntile = warp0_exclusive_scan(s_flag, ws.tile_off, E, lane);
        if (lane == 0) {
            s_off[E] = total;
            ws.offsets[E] = total;
            ws.tile_off[E] = ntile;
            ws.ctrl->n_uniq = nu;
            ws.ctrl->n_tiles_gu = ntile;
            ws.ctrl->route_done = 0u;
        }
    }
    __syncthreads();
    for (int e = tid; e < E; e += 256) {
        ws.counts[e] = s_cnt[e];
        ws.offsets[e] = s_off[e];
        int run = s_off[e];
        for (int c0 = 0; c0 < nch; c0 += kBatch) {   // chunk counts -> first row of each chunk
            int v[kBatch];
#pragma unroll
            for (int j = 0; j < kBatch; ++j) v[j] = c0 + j < nch ? __ldcg(ws.chunk_base + (size_t)(c0 + j) * E + e) : 0;
#pragma unroll
            for (int j = 0; j < kBatch; ++j) {
                if (c0 + j < nch) {
                    ws.chunk_base[(size_t)(c0 + j) * E + e] = run;
                    run += v[j];
                }
            }
        }
    }
}

__global__ void __launch_bounds__(256) route_scatter_kernel(int T, int k, int E, Workspace ws) {
    const int c = blockIdx.x, t0 = c * kChunk;
    const int nt = min(kChunk, T - t0);
    const uint32_t *gbm = ws.chunk_bm + (size_t)c * E;
    for (int p = threadIdx.x; p < nt * k; p += 256) {
        const int tl = p / k;
        const int t = t0 + tl;
        const int e = ws.ids[(size_t)t0 * k + p];
        if ((unsigned)e >= (unsigned)E) {
            atomicOr(&ws.ctrl->err, ERRBIT_RANGE);
            continue;
        }
        const int rank = __popc(gbm[e] & ((1u << tl) - 1u));
        const int row = ws.chunk_base[(size_t)c * E + e] + rank;
        ws.perm[row] = t;
        ws.pos[(size_t)t0 * k + p] = row;
    }
}

cudaError_t launch_route_large(const LayerDev &L, const Workspace &ws, const uint16_t *x, int T, cudaStream_t st,
                               int *launches) {
    cudaError_t e = launch_router_gemm(L, ws, x, T, st);
    if (e != cudaSuccess) return e;
    const int nch = (T + kChunk - 1) / kChunk;
    route_chunk_kernel<<<nch, 256, 0, st>>>(T, L.k, L.E, router_ksplit(L.d), (size_t)L.max_T * L.E, ws);
    route_scatter_kernel<<<nch, 256, 0, st>>>(T, L.k, L.E, ws);
    *launches += 3;
    return cudaGetLastError();
}

}  // namespace moe
