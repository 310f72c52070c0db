// prefill_fp4.cu — the large-batch (prefill) expert GEMMs for NVFP4 experts
// on the 5th-generation tensor cores.
//
// The pages run Muse Spark's experts as NVFP4 weights ("How SGLang-TorchTPU
// accelerated an 816B-parameter MoE on TPU v7", section "Results and
// interpretation") and prefill as a fused MoE kernel (same page, "Key
// optimisations"). With NVFP4 weights a 4096-token layer reads 3.55x fewer
// weight bytes than with bf16, so the grouped GEMM turns from weight-bound to
// compute-bound. The activations stay 16-bit (no activation quantisation):
// the weights are widened in shared memory and the MMA is tcgen05 kind::f16.
//
// Per k-block (64 elements of K) of a 128 x 256 output tile:
//   * the TMA producer loads the A tile (128 rows x 64, 128-byte swizzle),
//     the B tile's packed E2M1 codes (256 rows x 32 bytes) and the E4M3 block
//     scales of its rows (16 bytes per row: the scales of 4 k-blocks, of which
//     this k-block uses 4) into one slot of a 5-deep ring;
//   * eight converter warps (one B row per thread) widen the codes: e2m1 pair -> f16 pair (hardware
//     conversion), times the block scale in f16 (exact: the product of an
//     e2m1 and an e4m3 value has at most 6 significant bits and lies in f16's
//     normal range), optionally -> bf16 (exact likewise), and write the
//     256 x 64 B tile in the swizzled K-major layout the MMA descriptor reads,
//     into one of two converted-tile buffers;
//   * one thread issues tcgen05.mma (M=128, N=256, K=16) into a double-
//     buffered TMEM accumulator; four epilogue warps apply the per-row and
//     per-expert scales and the epilogue (SwiGLU -> bf16 h, or the expert
//     output).
// gate/up: A = the gathered token rows in f16, each scaled by a power of two
// 2^-p >= 1/max|x_t| (exact), the accumulator multiplied back by 2^p and the
// tensor scale; down: A = h in bf16, B widened to bf16.
// Warp roles: 0 = TMA producer, 1 = MMA issuer (owns TMEM), 2..5 = epilogue,
// 6..13 = converters.
#include <cuda_fp16.h>
#include <cuda_fp4.h>
#include <cuda_fp8.h>

#include "gemm.cuh"

namespace moe {

namespace fp4gemm {

constexpr int kQStages = 5;                       // TMA ring depth
constexpr int kBStages = 2;                       // converted-tile buffers
constexpr int kConvWarps = 8;                     // two per SM sub-partition: conversion latency hidden
constexpr int kConvThreads = 32 * kConvWarps;
constexpr int kThreads = 192 + kConvThreads;      // producer, MMA, 4 epilogue, 8 converter warps
constexpr uint32_t kABytes = BM * BK * 2;         // 16 KB
constexpr uint32_t kCodeBytes = BN * BK / 2;      // 8 KB: 256 rows x 32 B
constexpr uint32_t kScaleRowBytes = 16;           // the scales of 4 k-blocks
constexpr uint32_t kScaleBytes = BN * kScaleRowBytes;   // 4 KB
constexpr uint32_t kQStageBytes = kABytes + kCodeBytes + kScaleBytes;   // 28 KB (a multiple of 1024)
constexpr uint32_t kBBytes = BN * BK * 2;         // 32 KB
constexpr size_t kSmem = 1024 + (size_t)kBStages * kBBytes + (size_t)kQStages * kQStageBytes + 512;
static_assert(kQStageBytes % 1024 == 0, "A tiles must stay 1024-byte aligned");

// One B row of one k-block, by one converter thread: 64 E2M1 codes (32 bytes,
// stored with the 32-byte swizzle: the halves swapped when bit 2 of the row is
// set) times their four block scales (sc: this k-block's 4 E4M3 bytes), widened
// and written as 8 chunks of 16 bytes at chunk position c ^ (row % 8) of the
// row's 128 bytes. Eight consecutive rows touch eight different 16-byte bank
// groups in every access.
template <bool BF16OUT>
__device__ __forceinline__ void convert_row(const unsigned char *codes_tile, uint32_t sc, unsigned char *btile,
                                            int row) {
    const int sw = (row >> 2) & 1;
    const uint4 c0 = *reinterpret_cast<const uint4 *>(codes_tile + row * 32 + (sw << 4));          // codes 0..31
    const uint4 c1 = *reinterpret_cast<const uint4 *>(codes_tile + row * 32 + ((sw ^ 1) << 4));    // codes 32..63
    const uint32_t s01 = e4m3x2_to_f16x2((uint16_t)(sc & 0xFFFFu)), s23 = e4m3x2_to_f16x2((uint16_t)(sc >> 16));
    const __half2 h01 = *reinterpret_cast<const __half2 *>(&s01), h23 = *reinterpret_cast<const __half2 *>(&s23);
    const __half2 sb[4] = {__low2half2(h01), __high2half2(h01), __low2half2(h23), __high2half2(h23)};
    const uint32_t words[8] = {c0.x, c0.y, c0.z, c0.w, c1.x, c1.y, c1.z, c1.w};
#pragma unroll
    for (int j = 0; j < 8; ++j) {   // word j: codes 8j .. 8j+7, block j / 2
        uint32_t o[4];
        e2m1x8_to_f16x2(words[j], o);
#pragma unroll
        for (int b = 0; b < 4; ++b) {
            const __half2 v = __hmul2(*reinterpret_cast<const __half2 *>(&o[b]), sb[j >> 1]);
            if (BF16OUT) {
                const __nv_bfloat162 bv = __float22bfloat162_rn(__half22float2(v));
                o[b] = *reinterpret_cast<const uint32_t *>(&bv);
            } else {
                o[b] = *reinterpret_cast<const uint32_t *>(&v);
            }
        }
        *reinterpret_cast<uint4 *>(btile + (size_t)row * 128 + ((j ^ (row & 7)) << 4)) = make_uint4(o[0], o[1], o[2], o[3]);
    }
}

__device__ __forceinline__ void fence_proxy_async_smem() {
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

// SPLIT_B: the B tile is 128 rows of tmQ/tmS then 128 rows of tmQ2/tmS2 (gate
// and up); else 256 rows of tmQ/tmS. F16: A and B in f16 (else bf16).
template <int EPI, bool SPLIT_B, bool F16>
__global__ void __launch_bounds__(kThreads, 1)
    grouped_gemm_fp4_kernel(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmQ,
                            const __grid_constant__ CUtensorMap tmQ2, const __grid_constant__ CUtensorMap tmS,
                            const __grid_constant__ CUtensorMap tmS2, GemmParams p) {
    extern __shared__ __align__(1024) unsigned char smem_raw[];
    const uint32_t base_u32 = smem_u32(smem_raw);
    unsigned char *smem = smem_raw + (((base_u32 + 1023u) & ~1023u) - base_u32);
    unsigned char *btiles = smem;                                   // [kBStages][256 x 128 B]
    unsigned char *qring = smem + kBStages * kBBytes;               // [kQStages][A | codes | scales]
    uint64_t *bars = reinterpret_cast<uint64_t *>(qring + kQStages * kQStageBytes);
    uint64_t *qfull = bars, *qempty = bars + kQStages;
    uint64_t *bfull = bars + 2 * kQStages, *bempty = bfull + kBStages;
    uint64_t *tfull = bempty + kBStages, *tempty = tfull + 2, *done = tempty + 2;
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(done + 1);
    volatile int *abort_flag = reinterpret_cast<volatile int *>(tmem_slot + 1);

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    uint32_t *err = p.err;

    if (threadIdx.x == 0) {
        for (int s = 0; s < kQStages; ++s) {
            mbar_init(&qfull[s], 1);
            mbar_init(&qempty[s], 1 + kConvWarps);   // the MMA's commit (A read) + each converter warp (codes read)
        }
        for (int s = 0; s < kBStages; ++s) {
            mbar_init(&bfull[s], kConvWarps);
            mbar_init(&bempty[s], 1);
        }
        for (int b = 0; b < 2; ++b) {
            mbar_init(&tfull[b], 1);
            mbar_init(&tempty[b], 128);
        }
        mbar_init(done, 1);
        *abort_flag = 0;
        fence_barrier_init();
    }
    if (warp == 1) tmem_alloc(tmem_slot, kTmemCols);
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem_base = *tmem_slot;
    const int ntiles = total_tiles(p);
    const int kblocks = p.K / BK;

    if (warp == 0) {
        // ------------------------------- TMA producer -------------------------------
        if (lane == 0) {
            int it = 0;
            bool ok = true;
            for (int tile = blockIdx.x; tile < ntiles && ok; tile += gridDim.x) {
                const TileInfo ti = tile_info(p, tile);
                const int arow = ti.row0 + ti.m * BM;
                const int brow = ti.g * p.b_rows_per_group + ti.n * (SPLIT_B ? BN / 2 : BN);
                for (int kb = 0; kb < kblocks; ++kb, ++it) {
                    const int slot = it % kQStages;
                    if (!mbar_wait_or_abort(&qempty[slot], ((it / kQStages) & 1) ^ 1, err, abort_flag)) {
                        ok = false;
                        break;
                    }
                    unsigned char *st = qring + (size_t)slot * kQStageBytes;
                    unsigned char *codes = st + kABytes, *scales = codes + kCodeBytes;
                    const int xs = (kb >> 2) * (int)kScaleRowBytes;   // 16-byte aligned
                    mbar_arrive_expect_tx(&qfull[slot], kQStageBytes);
                    tma_load_2d(st, &tmA, kb * BK, arow, &qfull[slot]);
                    if (SPLIT_B) {
                        tma_load_2d(codes, &tmQ, kb * (BK / 2), brow, &qfull[slot]);
                        tma_load_2d(codes + kCodeBytes / 2, &tmQ2, kb * (BK / 2), brow, &qfull[slot]);
                        tma_load_2d(scales, &tmS, xs, brow, &qfull[slot]);
                        tma_load_2d(scales + kScaleBytes / 2, &tmS2, xs, brow, &qfull[slot]);
                    } else {
                        tma_load_2d(codes, &tmQ, kb * (BK / 2), brow, &qfull[slot]);
                        tma_load_2d(scales, &tmS, xs, brow, &qfull[slot]);
                    }
                }
            }
            // every load issued must land before the CTA exits
            for (int j = (it > kQStages ? it - kQStages : 0); j < it; ++j)
                mbar_wait(&qfull[j % kQStages], (j / kQStages) & 1, err);
        }
    } else if (warp == 1) {
        // -------------------------------- MMA issuer --------------------------------
        if (lane == 0) {
            int it = 0, lt = 0;
            bool ok = true;
            for (int tile = blockIdx.x; tile < ntiles && ok; tile += gridDim.x, ++lt) {
                const int b = lt & 1, use = lt >> 1;
                if (!mbar_wait_or_abort(&tempty[b], (use & 1) ^ 1, err, abort_flag)) break;
                tc_fence_after();
                const uint32_t dtm = tmem_base + (uint32_t)(b * BN);
                for (int kb = 0; kb < kblocks; ++kb, ++it) {
                    const int qs = it % kQStages, bs = it % kBStages;
                    if (!mbar_wait_or_abort(&qfull[qs], (it / kQStages) & 1, err, abort_flag) ||
                        !mbar_wait_or_abort(&bfull[bs], (it / kBStages) & 1, err, abort_flag)) {
                        ok = false;
                        break;
                    }
                    tc_fence_after();
                    const uint64_t ad = smem_desc_sw128(smem_u32(qring + (size_t)qs * kQStageBytes));
                    const uint64_t bd = smem_desc_sw128(smem_u32(btiles + (size_t)bs * kBBytes));
#pragma unroll
                    for (int kk = 0; kk < BK / 16; ++kk)
                        mma_bf16(dtm, ad + (uint64_t)(2 * kk), bd + (uint64_t)(2 * kk), F16 ? kIdescF16 : kIdesc,
                                 (kb | kk) != 0);
                    mma_commit(&qempty[qs]);   // the A tile is free once these MMAs have read it
                    mma_commit(&bempty[bs]);   // and so is the converted B tile
                }
                if (!ok) break;
                mma_commit(&tfull[b]);  // the accumulator is complete
            }
            mma_commit(done);
            mbar_wait(done, 0, err);
        }
    } else if (warp < 6) {
        // --------------------------------- epilogue ---------------------------------
        const int q = warp & 3;  // TMEM lane quarter this warp may access
        const int row = q * 32 + lane;
        int lt = 0;
        for (int tile = blockIdx.x; tile < ntiles; tile += gridDim.x, ++lt) {
            const TileInfo ti = tile_info(p, tile);
            const int b = lt & 1, use = lt >> 1;
            if (!mbar_wait_or_abort(&tfull[b], use & 1, err, abort_flag)) break;
            tc_fence_after();
            const uint32_t tbase = tmem_base + ((uint32_t)(q * 32) << 16) + (uint32_t)(b * BN);
            epilogue_tile<EPI, true>(p, ti, tbase, row);
            tc_fence_before();
            mbar_arrive(&tempty[b]);
        }
    } else {
        // -------------------------------- converters --------------------------------
        const int row = threadIdx.x - 192;   // the B row this thread widens (0 .. 255)
        int it = 0;
        bool ok = true;
        uint4 sc4 = make_uint4(0, 0, 0, 0);  // the row's scales of 4 k-blocks (read every 4th k-block)
        for (int tile = blockIdx.x; tile < ntiles && ok; tile += gridDim.x) {
            for (int kb = 0; kb < kblocks; ++kb, ++it) {
                const int qs = it % kQStages, bs = it % kBStages;
                if (!mbar_wait_or_abort(&qfull[qs], (it / kQStages) & 1, err, abort_flag) ||
                    !mbar_wait_or_abort(&bempty[bs], ((it / kBStages) & 1) ^ 1, err, abort_flag)) {
                    ok = false;
                    break;
                }
                const unsigned char *codes = qring + (size_t)qs * kQStageBytes + kABytes;
                if ((kb & 3) == 0)
                    sc4 = *reinterpret_cast<const uint4 *>(codes + kCodeBytes + row * kScaleRowBytes);
                const uint32_t sc = (kb & 3) == 0 ? sc4.x : (kb & 3) == 1 ? sc4.y : (kb & 3) == 2 ? sc4.z : sc4.w;
                convert_row<!F16>(codes, sc, btiles + (size_t)bs * kBBytes, row);
                fence_proxy_async_smem();   // these generic-proxy writes, before the MMA (async proxy) reads them
                __syncwarp();
                if (lane == 0) {
                    mbar_arrive(&bfull[bs]);
                    mbar_arrive(&qempty[qs]);
                }
            }
        }
    }
    tc_fence_before();
    __syncthreads();
    if (warp == 1) {
        tc_fence_after();
        tmem_dealloc(tmem_base, kTmemCols);
    }
}

// ---------------------------------------------------------------------------
// gather with per-row scaling: xp[r, :] = f16(x[perm[r], :] * 2^-p_r),
// rscale[r] = 2^p_r >= max_c |x[perm[r], c]| (1 for an all-zero row). The
// scaling is exact; it keeps |xp| <= 1 inside f16's range.
// ---------------------------------------------------------------------------
__global__ void __launch_bounds__(256) gather_rows_f16_kernel(const uint16_t *__restrict__ x,
                                                              const int32_t *__restrict__ perm,
                                                              uint16_t *__restrict__ xp, float *__restrict__ rscale,
                                                              int rows, int d, int T, uint32_t *err) {
    // one warp per gathered row (8 rows per CTA): rows of up to 4096
    // columns are held in registers (16 vectors per lane) between the max
    // and the conversion; longer rows are read twice
    constexpr int kV = 16;
    const int lane = threadIdx.x & 31;
    const int r = blockIdx.x * 8 + (threadIdx.x >> 5);
    if (r >= rows) return;
    const int t = perm[r];
    if ((unsigned)t >= (unsigned)T) {
        if (lane == 0) atomicOr(err, ERRBIT_RANGE);
        return;
    }
    const uint4 *src = reinterpret_cast<const uint4 *>(x + (size_t)t * d);
    uint4 *dst = reinterpret_cast<uint4 *>(xp + (size_t)r * d);
    const int nv = d / 8;
    const bool held = nv <= 32 * kV;
    uint4 v[kV];
    float m = 0.f;
    if (held) {
#pragma unroll
        for (int j = 0; j < kV; ++j) {
            const int i = lane + 32 * j;
            v[j] = i < nv ? __ldg(src + i) : make_uint4(0, 0, 0, 0);
        }
#pragma unroll
        for (int j = 0; j < kV; ++j) {
            const uint32_t w[4] = {v[j].x, v[j].y, v[j].z, v[j].w};
#pragma unroll
            for (int q = 0; q < 4; ++q) m = fmaxf(m, fmaxf(fabsf(bf16lo(w[q])), fabsf(bf16hi(w[q]))));
        }
    } else {
        for (int i = lane; i < nv; i += 32) {
            const uint4 a = __ldg(src + i);
            const uint32_t w[4] = {a.x, a.y, a.z, a.w};
#pragma unroll
            for (int q = 0; q < 4; ++q) m = fmaxf(m, fmaxf(fabsf(bf16lo(w[q])), fabsf(bf16hi(w[q]))));
        }
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) m = fmaxf(m, __shfl_xor_sync(0xFFFFFFFFu, m, o));
    int e = 0;
    if (m > 0.f) frexpf(m, &e);      // m = f * 2^e, f in [0.5, 1): 2^e >= m
    const float inv = ldexpf(1.f, -e);
    if (lane == 0) rscale[r] = ldexpf(1.f, e);
    auto convert = [&](const uint4 &a) {
        const uint32_t w[4] = {a.x, a.y, a.z, a.w};
        uint32_t o[4];
#pragma unroll
        for (int q = 0; q < 4; ++q) {
            const __half2 h = __floats2half2_rn(bf16lo(w[q]) * inv, bf16hi(w[q]) * inv);
            o[q] = *reinterpret_cast<const uint32_t *>(&h);
        }
        return make_uint4(o[0], o[1], o[2], o[3]);
    };
    if (held) {
#pragma unroll
        for (int j = 0; j < kV; ++j) {
            const int i = lane + 32 * j;
            if (i < nv) dst[i] = convert(v[j]);
        }
    } else {
        for (int i = lane; i < nv; i += 32) dst[i] = convert(__ldg(src + i));
    }
}

template <int EPI, bool SPLIT_B, bool F16>
static cudaError_t launch_fp4_gemm(const CUtensorMap &a, const CUtensorMap &q, const CUtensorMap &q2,
                                   const CUtensorMap &s, const CUtensorMap &s2, const GemmParams &p, int grid,
                                   cudaStream_t st) {
    static std::atomic<uint64_t> attr_set{0};
    cudaError_t e =
        set_smem_limit_once((const void *)grouped_gemm_fp4_kernel<EPI, SPLIT_B, F16>, (int)kSmem, attr_set);
    if (e != cudaSuccess) return e;
    grouped_gemm_fp4_kernel<EPI, SPLIT_B, F16><<<grid, kThreads, kSmem, st>>>(a, q, q2, s, s2, p);
    return cudaGetLastError();
}

}  // namespace fp4gemm

cudaError_t launch_gather_rows_f16(const LayerDev &L, const Workspace &ws, const uint16_t *x, int T,
                                   cudaStream_t st) {
    fp4gemm::gather_rows_f16_kernel<<<(T * L.k + 7) / 8, 256, 0, st>>>(x, ws.perm, ws.xperm, ws.row_scale, T * L.k,
                                                                      L.d, T, &ws.ctrl->err);
    return cudaGetLastError();
}

cudaError_t launch_prefill_experts_fp4(const LayerDev &L, const Workspace &ws, int T, cudaStream_t st,
                                       int *launches) {
    using namespace fp4gemm;
    (void)T;
    const uint64_t rows = (uint64_t)L.max_T * L.k;
    const uint64_t gu_rows = (uint64_t)L.E * L.I, dn_rows = (uint64_t)L.E * L.d;
    CUtensorMap ta, qg, qu, sg, su, th, qd, sd;
    if (!make_tmap_bf16(&ta, ws.xperm, rows, (uint64_t)L.d, BM) ||
        !make_tmap_u8(&qg, L.qg, gu_rows, (uint64_t)L.d / 2, BK / 2, BN / 2, true) ||
        !make_tmap_u8(&qu, L.qu, gu_rows, (uint64_t)L.d / 2, BK / 2, BN / 2, true) ||
        !make_tmap_u8(&sg, L.sg, gu_rows, (uint64_t)L.d / 16, kScaleRowBytes, BN / 2) ||
        !make_tmap_u8(&su, L.su, gu_rows, (uint64_t)L.d / 16, kScaleRowBytes, BN / 2) ||
        !make_tmap_bf16(&th, ws.h, rows, (uint64_t)L.I, BM) ||
        !make_tmap_u8(&qd, L.qd, dn_rows, (uint64_t)L.I / 2, BK / 2, BN, true) ||
        !make_tmap_u8(&sd, L.sd, dn_rows, (uint64_t)L.I / 16, kScaleRowBytes, BN))
        return cudaErrorInvalidValue;
    GemmParams p{};
    p.ksplit = 1;
    p.tile_off = ws.tile_off;
    p.row_off = ws.offsets;
    p.groups = L.E;
    p.err = &ws.ctrl->err;
    // gate/up + SwiGLU: f16 tokens (scaled per row), gate rows then up rows
    p.nt = L.I / (BN / 2);
    p.K = L.d;
    p.b_rows_per_group = L.I;
    p.out_bf16 = reinterpret_cast<uint16_t *>(ws.h);
    p.ld = L.I;
    p.row_scale = ws.row_scale;
    p.col_scale = L.gg;
    p.col_scale2 = L.gu;
    cudaError_t e = launch_fp4_gemm<EPI_SWIGLU, true, true>(ta, qg, qu, sg, su, p, L.num_sms, st);
    if (e != cudaSuccess) return e;
    // down: Y = H . Wd^T with bf16 h; stored in bf16 over the gathered rows
    // (fp32 for the per-expert-normalised variant)
    p.nt = L.d / BN;
    p.K = L.I;
    p.b_rows_per_group = L.d;
    p.ld = L.d;
    p.n_valid = L.d;
    p.row_scale = nullptr;
    p.col_scale = L.gd;
    p.col_scale2 = nullptr;
    if (L.expert_norm) {
        p.out_bf16 = nullptr;
        p.out_f32 = ws.Y;
        e = launch_fp4_gemm<EPI_F32, false, false>(th, qd, qd, sd, sd, p, L.num_sms, st);
    } else {
        p.out_bf16 = ws.xperm;
        p.out_f32 = nullptr;
        e = launch_fp4_gemm<EPI_BF16, false, false>(th, qd, qd, sd, sd, p, L.num_sms, st);
    }
    *launches += 2;
    return e;
}

}  // namespace moe
