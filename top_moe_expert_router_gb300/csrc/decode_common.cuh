// decode_common.cuh — pieces shared by the two persistent small-batch layer
// kernels (decode_fused.cuh: experts on CUDA cores; decode_mma.cuh: experts on
// the tensor cores): acquire loads, the bounded grid barrier, even shares,
// the h-row hand-off counters, the tagged logits, and the routing of up to 16
// tokens computed in shared memory by every CTA.
#pragma once

#include "common.cuh"

namespace moe {

namespace fused {

// Stacked layers: the router rows of the next layer this CTA computes
// (experts b, b + G), fetched into L2 while the current layer's weights
// still stream, so that the next router reads them from L2, not HBM.
__device__ __forceinline__ void prefetch_next_router(const LayerW &next, int b, int G, int E, int d) {
    for (int e = b; e < E && e < b + 2 * G; e += G)
        asm volatile("cp.async.bulk.prefetch.L2.global [%0], %1;" ::"l"(next.wr + (size_t)e * d), "r"((uint32_t)d * 2)
                     : "memory");
}

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

// n / dv for 0 <= n < 2^63, dv > 0, in 32-bit arithmetic whenever n fits
// (every share of these kernels' unit counts does; a 64-bit division is a
// long software sequence on the prologue's critical path).
__device__ __forceinline__ long long div_u(long long n, int dv) {
    return (unsigned long long)n < 0x100000000ull ? (long long)((uint32_t)n / (uint32_t)dv) : n / dv;
}

__device__ __forceinline__ void share(int total, int b, int G, int &start, int &count) {
    start = (int)div_u((long long)b * total, G);
    count = (int)div_u((long long)(b + 1) * total, G) - start;
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
    uint32_t *wsum;    // [8] per-warp totals of the routing scan
    int *n_uniq;
};

// Logits of the small-batch router handed from CTA to CTA without a grid
// barrier: each is one 64-bit word, the fp32 logit in the low half and a tag
// in the high half. The word is stored and loaded whole (single-copy atomic),
// so a reader that sees the tag it expects holds that launch's logit; no
// fence or counter is involved. The tag is the layer's epoch (see
// decode_fused.cuh), different from every tag an earlier launch left behind.
__device__ __forceinline__ void st_tagged(uint64_t *p, float v, uint32_t tag) {
    const uint64_t w = ((uint64_t)tag << 32) | (uint64_t)__float_as_uint(v);
    asm volatile("st.relaxed.gpu.global.b64 [%0], %1;" ::"l"(p), "l"(w) : "memory");
}

__device__ __forceinline__ void ld_tagged2(const uint64_t *p, uint64_t &a, uint64_t &b) {
    asm volatile("ld.relaxed.gpu.global.v2.b64 {%0, %1}, [%2];" : "=l"(a), "=l"(b) : "l"(p) : "memory");
}

// A real expert's order key, never 0 (0 marks an empty place: an expert id
// >= E, or one already picked). Only the one NaN bit pattern whose key would
// be 0 moves up by one.
__device__ __forceinline__ uint32_t expert_key(float f) {
    const uint32_t kk = order_key(f);
    return kk ? kk : 1u;
}

// This lane's eight keys, experts 8 * lane + i, from a plain fp32 logits row
// (written by other CTAs before a grid barrier: read through L2).
__device__ __forceinline__ void lane_keys(const float *row, int E, uint32_t key[8]) {
    const int lane = threadIdx.x & 31;
    const int e0 = 8 * lane;
    if ((E & 7) == 0 && e0 < E) {
        const float4 a = __ldcg(reinterpret_cast<const float4 *>(row + e0));
        const float4 b = __ldcg(reinterpret_cast<const float4 *>(row + e0) + 1);
        const float v[8] = {a.x, a.y, a.z, a.w, b.x, b.y, b.z, b.w};
#pragma unroll
        for (int i = 0; i < 8; ++i) key[i] = expert_key(v[i]);
    } else {
#pragma unroll
        for (int i = 0; i < 8; ++i) key[i] = e0 + i < E ? expert_key(__ldcg(row + e0 + i)) : 0u;
    }
}

// The same from a row of tagged logits, polling until every word of the
// warp's row carries `tag` (bounded: on timeout the error word gets
// ERRBIT_TIMEOUT, the CTA's abort flag is set and whatever was read is used).
__device__ __forceinline__ void lane_keys_tagged(const uint64_t *row, int E, uint32_t tag, uint32_t key[8],
                                                 uint32_t *err, volatile int *abort_flag) {
    const int lane = threadIdx.x & 31;
    const int e0 = 8 * lane;
    uint64_t w[8];
    unsigned long long t0 = 0;
    for (uint32_t it = 0;; ++it) {
        bool ok = true;
        if ((E & 7) == 0) {
            if (e0 < E) {
#pragma unroll
                for (int i = 0; i < 8; i += 2) ld_tagged2(row + e0 + i, w[i], w[i + 1]);
            }
        } else {
#pragma unroll
            for (int i = 0; i < 8; ++i)
                if (e0 + i < E) w[i] = *reinterpret_cast<const volatile uint64_t *>(row + e0 + i);
        }
#pragma unroll
        for (int i = 0; i < 8; ++i) ok = ok && (e0 + i >= E || (uint32_t)(w[i] >> 32) == tag);
        if (__all_sync(0xFFFFFFFFu, ok)) break;
        if ((it & 63u) == 63u) {
            const unsigned long long now = global_ns();
            if (t0 == 0) t0 = now;
            const bool give_up = *abort_flag != 0 || now - t0 > kWaitLimitNs;
            if (__any_sync(0xFFFFFFFFu, give_up)) {
                if (lane == 0) {
                    atomicOr(err, ERRBIT_TIMEOUT);
                    *abort_flag = 1;
                }
                break;
            }
        }
    }
#pragma unroll
    for (int i = 0; i < 8; ++i) key[i] = e0 + i < E ? expert_key(__uint_as_float((uint32_t)w[i])) : 0u;
}

// Top-k (k <= 8) of one token from the warp's keys (lane l: experts 8l .. 8l+7,
// 0 for empty places): ids by descending logit, ties to the lower id; weights
// exp(l - l_max) / sum over the kept, summed in pick order (the same
// arithmetic as topk_warp). Each lane first sorts its eight (key, id) pairs
// (descending key, ascending id among equal keys; a 19-comparator network),
// so a pick is one warp-wide max of the lanes' heads: among the lanes whose
// head reaches it the lowest lane holds the lowest id, since lane l's ids all
// lie below lane l+1's. The winning lane stores the id and drops its head.
__device__ __forceinline__ void topk_sorted(uint32_t key[8], int k, int32_t *ids_out, float *w_out) {
    const int lane = threadIdx.x & 31;
    int id[8];
#pragma unroll
    for (int i = 0; i < 8; ++i) id[i] = 8 * lane + i;
    auto ce = [&](int a, int b) {
        const bool sw = key[b] > key[a] || (key[b] == key[a] && id[b] < id[a]);
        const uint32_t ka = sw ? key[b] : key[a], kb = sw ? key[a] : key[b];
        const int ia = sw ? id[b] : id[a], ib = sw ? id[a] : id[b];
        key[a] = ka;
        key[b] = kb;
        id[a] = ia;
        id[b] = ib;
    };
    ce(0, 2); ce(1, 3); ce(4, 6); ce(5, 7);
    ce(0, 4); ce(1, 5); ce(2, 6); ce(3, 7);
    ce(0, 1); ce(2, 3); ce(4, 5); ce(6, 7);
    ce(2, 4); ce(3, 5);
    ce(1, 4); ce(3, 6);
    ce(1, 2); ce(3, 4); ce(5, 6);
    uint32_t my_key = 0u;
#pragma unroll
    for (int j = 0; j < 8; ++j) {
        if (j < k) {
            const uint32_t m = __reduce_max_sync(0xFFFFFFFFu, key[0]);
            const uint32_t bal = __ballot_sync(0xFFFFFFFFu, key[0] == m);
            if (lane == j) my_key = m;
            if (lane == __ffs(bal) - 1) {
                ids_out[j] = id[0];
#pragma unroll
                for (int i = 0; i < 7; ++i) {
                    key[i] = key[i + 1];
                    id[i] = id[i + 1];
                }
                key[7] = 0u;
            }
        }
    }
    const float lmax = __shfl_sync(0xFFFFFFFFu, key_value(my_key), 0);
    const float ex = lane < k ? expf(key_value(my_key) - lmax) : 0.f;
    float sum = 0.f;
    for (int j = 0; j < k; ++j) sum += __shfl_sync(0xFFFFFFFFu, ex, j);
    if (lane < k) w_out[lane] = ex / sum;
}

// Routing of T <= 16 tokens in shared memory, by every CTA of the launch (all
// blockDim.x >= 256 threads take part; E <= 256, k <= 8):
//  1. warp w takes tokens w, w + nwarps, ...: top-k and weights (from the
//     tagged logits when `tlogits` is set, else from the plain fp32 rows);
//  2. one thread per (token, pick) sets the token's bit in its expert's bitmap;
//  3. one scan over the experts of (count, used) gives each expert's first
//     row (offsets), the used experts ascending (uniq) and, at uniq index u,
//     the rows before expert uniq[u] (R.scan: the prefix of the experts'
//     token counts, n_uniq + 1 entries);
//  4. one thread per (token, pick) places it: experts ascending, tokens
//     ascending within an expert.
// One token skips 2.-4.: warp 0 ranks its k distinct experts (ascending,
// they are its k rows) and fills R.cnt / R.off only with `counts` (otherwise
// expert uniq[u] is known to hold one token, at row u). Ends with
// __syncthreads().
__device__ __forceinline__ void route_tokens(const Route &R, const float *logits, const uint64_t *tlogits,
                                             uint32_t tag, int T, int k, int E, uint32_t *err,
                                             volatile int *abort_flag, bool counts = true) {
    const int tid = threadIdx.x, nthr = blockDim.x, warp = tid >> 5, lane = tid & 31, nwarps = nthr >> 5;
    if (T == 1) {
        // one token: its k distinct experts, ascending, are its k rows (warp
        // 0 alone; the per-expert counts and first rows only with `counts`,
        // after the barrier, for the records CTA 0 publishes)
        if (warp == 0) {
            uint32_t key[8];
            if (tlogits)
                lane_keys_tagged(tlogits, E, tag, key, err, abort_flag);
            else
                lane_keys(logits, E, key);
            topk_sorted(key, k, R.ids, R.w);
            __syncwarp();
            int idq[8];
#pragma unroll
            for (int q = 0; q < 8; ++q) idq[q] = q < k ? R.ids[q] : 0x7FFFFFFF;
            int my = 0x7FFFFFFF;
#pragma unroll
            for (int q = 0; q < 8; ++q)
                if (q == lane) my = idq[q];
            int rank = 0;
#pragma unroll
            for (int q = 0; q < 8; ++q) rank += idq[q] < my;
            if (lane < k) {
                R.uniq[rank] = my;
                R.scan[rank] = rank;
                R.perm[rank] = 0;
                R.pos[lane] = rank;
            }
            if (lane == 0) {
                R.off[E] = k;
                R.scan[k] = k;
                *R.n_uniq = k;
            }
        }
        __syncthreads();
        if (counts) {
            for (int e = tid; e < E; e += nthr) {
                int c = 0, o = 0;
                for (int q = 0; q < k; ++q) {
                    const int id = R.ids[q];
                    c += id == e;
                    o += id < e;
                }
                R.cnt[e] = c;
                R.off[e] = o;
            }
            __syncthreads();
        }
        return;
    }
    for (int e = tid; e < 256; e += nthr) R.bm[e] = 0u;
    for (int t = warp; t < T; t += nwarps) {
        uint32_t key[8];
        if (tlogits)
            lane_keys_tagged(tlogits + (size_t)t * E, E, tag, key, err, abort_flag);
        else
            lane_keys(logits + (size_t)t * E, E, key);
        topk_sorted(key, k, R.ids + t * k, R.w + t * k);
    }
    __syncthreads();
    for (int p = tid; p < T * k; p += nthr) {
        const int e = R.ids[p];
        if ((unsigned)e < (unsigned)E) atomicOr(&R.bm[e], 1u << (p / k));
    }
    __syncthreads();
    // (count, used) packed in one word: counts sum to <= T * k <= 128 and
    // the used experts number <= 256, so neither half carries into the other
    uint32_t v = 0u, inc = 0u;
    int c = 0;
    if (tid < 256) {
        c = tid < E ? __popc(R.bm[tid]) : 0;
        v = (uint32_t)c | ((c > 0 ? 1u : 0u) << 16);
        inc = v;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const uint32_t y = __shfl_up_sync(0xFFFFFFFFu, inc, o);
            if (lane >= o) inc += y;
        }
        if (lane == 31) R.wsum[warp] = inc;
    }
    __syncthreads();
    if (tid < 256) {
        uint32_t pre = 0u;
        for (int i = 0; i < warp; ++i) pre += R.wsum[i];
        const uint32_t ex = pre + inc - v;
        if (tid < E) {
            R.cnt[tid] = c;
            R.off[tid] = (int)(ex & 0xFFFFu);
            if (c > 0) {
                R.uniq[ex >> 16] = tid;
                R.scan[ex >> 16] = (int)(ex & 0xFFFFu);
            }
        }
        if (tid == 255) {
            const uint32_t tot = pre + inc;
            R.off[E] = (int)(tot & 0xFFFFu);
            R.scan[tot >> 16] = (int)(tot & 0xFFFFu);
            *R.n_uniq = (int)(tot >> 16);
        }
    }
    __syncthreads();
    for (int p = tid; p < T * k; p += nthr) {
        const int e = R.ids[p];
        if ((unsigned)e < (unsigned)E) {
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
