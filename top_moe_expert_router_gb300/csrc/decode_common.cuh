// decode_common.cuh — pieces shared by the two persistent small-batch layer
// kernels (decode_fused.cuh: experts on CUDA cores; decode_mma.cuh: experts on
// the tensor cores): acquire loads, the bounded grid barrier, even shares,
// the h-row hand-off counters, and the routing of up to 16 tokens computed in
// shared memory by every CTA.
#pragma once

#include "common.cuh"

namespace moe {

namespace fused {

__device__ __forceinline__ uint32_t ld_acquire(const uint32_t *p) {
    uint32_t v;
    asm volatile("ld.acquire.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
    return v;
}

// Grid barrier over all CTAs of the (cooperative) launch: arrival counter
// `target` = (barrier index) x (grid size), plus *hold, a test hook that is 0
// in normal operation (nonzero: an arrival that never comes, so the bounded
// wait runs out). Bounded wait.
__device__ inline bool grid_barrier(uint32_t *ctr, uint32_t target, uint32_t *err, volatile int *abort_flag,
                                    const uint32_t *hold) {
    __syncthreads();
    __shared__ int ok;
    if (threadIdx.x == 0) {
        target += *reinterpret_cast<const volatile uint32_t *>(hold);
        fence_acq_rel_gpu();
        atomicAdd(ctr, 1u);
        ok = 1;
        unsigned long long t0 = global_ns();
        while (ld_acquire(ctr) < target) {
            if (*abort_flag || global_ns() - t0 > kWaitLimitNs) {
                atomicOr(err, ERRBIT_TIMEOUT);
                *abort_flag = 1;
                ok = 0;
                break;
            }
        }
        fence_acq_rel_gpu();
    }
    __syncthreads();
    return ok != 0;
}

__device__ __forceinline__ void share(int total, int b, int G, int &start, int &count) {
    start = (int)((long long)b * total / G);
    count = (int)((long long)(b + 1) * total / G) - start;
}

// This CTA's stages: segment A = first-half gate/up row pairs, B = second-half
// gate/up, C = first-half down units (kDnRows rows), D = second-half down.
struct Plan {
    int nA, nB, nC, nD;        // stages of each segment in this CTA
    int a0, b0, c0, d0;        // first index of this CTA's share within each segment
    int offB, offD;            // global start of the second-half segments
    // flattened gate/up row-pair index (u * I + i) of gate/up stage s
    __device__ __forceinline__ int gu_row(int s) const { return s < nA ? a0 + s : offB + b0 + (s - nA); }
    // flattened down unit index (u * d / kDnRows + c / kDnRows) of down stage t (t = s - nA - nB)
    __device__ __forceinline__ int dn_unit(int t) const { return t < nC ? c0 + t : offD + d0 + (t - nC); }
};

// Even shares with the remainders rotated: in segment s (n_s units) every CTA
// takes n_s / G units and the n_s % G extra ones go to the CTAs from o_s on
// (cyclically), o_s being where the previous segments' extras ended. So a CTA
// that took an extra unit in one segment is the last to take one in the next,
// and the largest share exceeds the mean by at most about one unit overall.
__device__ __forceinline__ void share_rotated(int total, int b, int G, int o, int &start, int &count) {
    const int base = total / G, rem = total % G;
    // extras among CTAs [0, b): those j with (j - o) mod G < rem
    auto extras_before = [&](int bb) {
        int n = 0;
        if (o + rem <= G) {
            n = min(max(bb - o, 0), rem);
        } else {
            n = min(bb, o + rem - G) + min(max(bb - o, 0), G - o);
        }
        return n;
    };
    start = b * base + extras_before(b);
    count = base + (((b - o) % G + G) % G < rem ? 1 : 0);
}

// make_plan with rotated remainders: segments A, B, C, D in that order.
__device__ __forceinline__ Plan make_plan_rotated(int U, int I, int units_per_expert, int b, int G) {
    Plan p;
    const int U1 = (U + 1) / 2, U2 = U - U1;
    const int nA = U1 * I, nB = U2 * I, nC = U1 * units_per_expert, nD = U2 * units_per_expert;
    int o = 0;
    share_rotated(nA, b, G, o, p.a0, p.nA);
    o = (o + nA % G) % G;
    share_rotated(nB, b, G, o, p.b0, p.nB);
    o = (o + nB % G) % G;
    share_rotated(nC, b, G, o, p.c0, p.nC);
    o = (o + nC % G) % G;
    share_rotated(nD, b, G, o, p.d0, p.nD);
    p.offB = nA;
    p.offD = nC;
    return p;
}

__device__ __forceinline__ Plan make_plan(int U, int I, int units_per_expert, int b, int G) {
    Plan p;
    const int U1 = (U + 1) / 2, U2 = U - U1;
    share(U1 * I, b, G, p.a0, p.nA);
    share(U2 * I, b, G, p.b0, p.nB);
    share(U1 * units_per_expert, b, G, p.c0, p.nC);
    share(U2 * units_per_expert, b, G, p.d0, p.nD);
    p.offB = U1 * I;
    p.offD = U1 * units_per_expert;
    return p;
}

// Publish a warp's count of finished h rows (all lanes' h stores first).
__device__ __forceinline__ void publish_rows(uint32_t *ctr, int n) {
    fence_acq_rel_gpu();
    __syncwarp();
    if ((threadIdx.x & 31) == 0 && n) atomicAdd(ctr, (uint32_t)n);
}

// Warp-wide bounded wait until *ctr >= target.
__device__ __forceinline__ bool wait_rows(const uint32_t *ctr, uint32_t target, uint32_t *err,
                                          volatile int *abort_flag) {
    int ok = 1;
    if ((threadIdx.x & 31) == 0) {
        const unsigned long long t0 = global_ns();
        while (ld_acquire(ctr) < target) {
            if (*abort_flag || global_ns() - t0 > kWaitLimitNs) {
                atomicOr(err, ERRBIT_TIMEOUT);
                *abort_flag = 1;
                ok = 0;
                break;
            }
        }
    }
    return __shfl_sync(0xFFFFFFFFu, ok, 0) != 0;
}

// Routing state in shared memory.
struct Route {
    int32_t *ids, *pos, *perm, *cnt, *off, *uniq, *scan;
    float *w;
    uint32_t *bm;
    int *n_uniq;
};

// exclusive scan of a[0..n) (n <= 256) by one warp; returns the total
__device__ inline int warp_scan256(const int32_t *a, int32_t *out, int n) {
    const int lane = threadIdx.x & 31;
    int vals[8], local = 0;
#pragma unroll
    for (int i = 0; i < 8; ++i) {
        const int idx = lane * 8 + i;
        vals[i] = idx < n ? a[idx] : 0;
        local += vals[i];
    }
    int incl = local;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const int y = __shfl_up_sync(0xFFFFFFFFu, incl, o);
        if (lane >= o) incl += y;
    }
    int run = incl - local;
#pragma unroll
    for (int i = 0; i < 8; ++i) {
        const int idx = lane * 8 + i;
        if (idx < n) out[idx] = run;
        run += vals[i];
    }
    return __shfl_sync(0xFFFFFFFFu, incl, 31);
}


// Routing of T <= 16 tokens in shared memory, by every CTA of the launch (the
// logits of all tokens are complete in global memory): warp w takes tokens
// w, w + nwarps, ...: top-k, weights; then one warp builds the permutation:
// experts ascending, tokens ascending within an expert (one token: its k
// distinct experts, ascending, are its k rows). Ends with __syncthreads().
__device__ __forceinline__ void route_tokens(const Route &R, const float *logits, int T, int k, int E, int nwarps) {
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    for (int t = warp; t < T; t += nwarps)
        topk_warp(logits + (size_t)t * E, E, k, R.ids + t * k, R.w + t * k, true);
    if (T > 1) __syncthreads();  // one token: warp 0 picked its experts itself
    if (warp == 0 && T == 1) {
        // one token: its k distinct experts, ascending, are the k rows
        __syncwarp();
        const int my = lane < k ? R.ids[lane] : 0x7FFFFFFF;
        int rank = 0;
        int cnt_i[8], off_i[8];
#pragma unroll
        for (int i = 0; i < 8; ++i) cnt_i[i] = off_i[i] = 0;
        for (int q = 0; q < k; ++q) {
            const int o = __shfl_sync(0xFFFFFFFFu, my, q);
            rank += o < my;
#pragma unroll
            for (int i = 0; i < 8; ++i) {
                const int e = lane + 32 * i;
                cnt_i[i] += o == e;
                off_i[i] += o < e;
            }
        }
#pragma unroll
        for (int i = 0; i < 8; ++i) {
            const int e = lane + 32 * i;
            if (e < E) {
                R.cnt[e] = cnt_i[i];
                R.off[e] = off_i[i];
            }
        }
        if (lane < k) {
            R.uniq[rank] = my;
            R.perm[rank] = 0;
            R.pos[lane] = rank;
        }
        if (lane == 0) {
            R.off[E] = k;
            *R.n_uniq = k;
        }
    } else if (warp == 0) {
        // the permutation (at most 16 x 8 pairs) by one warp: experts ascending,
        // tokens ascending within an expert
        __syncwarp();
        for (int e = lane; e < E; e += 32) R.bm[e] = 0u;
        __syncwarp();
        for (int p = lane; p < T * k; p += 32) {
            const int e = R.ids[p];
            if ((unsigned)e < (unsigned)E) atomicOr(&R.bm[e], 1u << (p / k));
        }
        __syncwarp();
        for (int e = lane; e < E; e += 32) {
            const int c = __popc(R.bm[e]);
            R.cnt[e] = c;
            R.scan[e] = c > 0;
        }
        __syncwarp();
        const int total = warp_scan256(R.cnt, R.off, E);
        __syncwarp();
        const int nu = warp_scan256(R.scan, R.scan, E);
        __syncwarp();
        for (int e = lane; e < E; e += 32)
            if (R.cnt[e] > 0) R.uniq[R.scan[e]] = e;
        if (lane == 0) {
            R.off[E] = total;
            *R.n_uniq = nu;
        }
        __syncwarp();
        for (int p = lane; p < T * k; p += 32) {
            const int e = R.ids[p];
            const int t = p / k;
            const int row = R.off[e] + __popc(R.bm[e] & ((1u << t) - 1u));
            R.perm[row] = t;
            R.pos[p] = row;
        }
    }
    __syncthreads();
}

// CTA 0 publishes the routing records to the workspace (the forward's own
// records, read back by moe_debug_route_records and the separate combine).
__device__ __forceinline__ void publish_records(const Route &R, const Workspace &ws, int T, int k, int E, int n_uniq,
                                       int nthreads) {
    const int tid = threadIdx.x;
    for (int p = tid; p < T * k; p += nthreads) {
        ws.ids[p] = R.ids[p];
        ws.w[p] = R.w[p];
        ws.pos[p] = R.pos[p];
        ws.perm[p] = R.perm[p];
    }
    for (int e = tid; e < E; e += nthreads) {
        ws.counts[e] = R.cnt[e];
        ws.offsets[e] = R.off[e];
        ws.tile_off[e] = 0;
    }
    for (int u = tid; u < n_uniq; u += nthreads) ws.uniq[u] = R.uniq[u];
    if (tid == 0) {
        ws.offsets[E] = R.off[E];
        ws.tile_off[E] = 0;
        ws.ctrl->n_uniq = n_uniq;
    }
}

}  // namespace fused

}  // namespace moe
