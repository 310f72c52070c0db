// prefill.cu — grouped GEMMs on the 5th-generation tensor cores for large
// batches (prefill): the router GEMM, the expert gate/up GEMM with the SwiGLU
// epilogue, and the expert down GEMM.
//
// With thousands of tokens every active expert sees a tall block of rows, and
// the expert FFN becomes a dense contraction: the pages' prefill path runs a
// fused MoE kernel ("How SGLang-TorchTPU accelerated an 816B-parameter MoE on
// TPU v7", section "Key optimisations"). Here each expert's rows are a group
// of a persistent grouped GEMM:
//   * operands are K-major bf16 tiles loaded by TMA (cp.async.bulk.tensor,
//     128-byte swizzle) into a 4-stage shared-memory ring;
//   * one thread issues tcgen05.mma (M=128, N=256, K=16, bf16 in, fp32 out)
//     into a double-buffered accumulator in tensor memory (2 x 256 columns);
//   * four epilogue warps read the accumulator with tcgen05.ld and apply the
//     epilogue (router logits + bias; h = silu(gate) * up rounded to bf16;
//     or the fp32 expert output) while the next tile accumulates.
// Warp roles: 0 = TMA producer, 1 = MMA issuer (owns the TMEM allocation),
// 2..5 = epilogue (TMEM lane quarter = warp % 4).
// Tiles run expert by expert, m-tiles fastest, so the CTAs working at the same
// time read the same weight tile and it is fetched from HBM once.
#include <cuda.h>
#include <cudaTypedefs.h>
#include <cuda_runtime.h>

#include "gemm.cuh"

namespace moe {

constexpr int kGemmStages = 4;
constexpr int kGemmThreads = 192;
constexpr uint32_t kABytes = BM * BK * 2;       // 16 KB
constexpr uint32_t kBBytes = BN * BK * 2;       // 32 KB
constexpr uint32_t kStageBytes = kABytes + kBBytes;
constexpr size_t kGemmSmem = 1024 + (size_t)kGemmStages * kStageBytes + 256;

// ---------------------------------------------------------------------------
// the kernel
// ---------------------------------------------------------------------------
template <int EPI, bool SPLIT_B>
__global__ void __launch_bounds__(kGemmThreads, 1)
    grouped_gemm_kernel(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB,
                        const __grid_constant__ CUtensorMap tmB2, GemmParams p) {
    extern __shared__ __align__(1024) unsigned char smem_raw[];
    const uint32_t base_u32 = smem_u32(smem_raw);
    unsigned char *smem = smem_raw + (((base_u32 + 1023u) & ~1023u) - base_u32);
    unsigned char *tiles = smem;                                        // stages, 1024-aligned
    uint64_t *bars = reinterpret_cast<uint64_t *>(smem + kGemmStages * kStageBytes);
    uint64_t *full = bars, *empty = bars + kGemmStages;
    uint64_t *tfull = bars + 2 * kGemmStages, *tempty = tfull + 2, *done = tempty + 2;
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(done + 1);
    volatile int *abort_flag = reinterpret_cast<volatile int *>(tmem_slot + 1);

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    uint32_t *err = p.err;

    if (threadIdx.x == 0) {
        for (int s = 0; s < kGemmStages; ++s) {
            mbar_init(&full[s], 1);
            mbar_init(&empty[s], 1);
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
    const int kblocks = p.K / BK / p.ksplit;  // k-blocks of one tile

    if (warp == 0) {
        // ------------------------------- TMA producer -------------------------------
        if (lane == 0) {
            int it = 0;
            bool ok = true;
            for (int tile = blockIdx.x; tile < ntiles && ok; tile += gridDim.x) {
                const TileInfo ti = tile_info(p, tile);
                const int arow = ti.row0 + ti.m * BM;
                const int brow = ti.g * p.b_rows_per_group + ti.n * (SPLIT_B ? BN / 2 : BN);
                const int kb0 = ti.ks * kblocks;
                for (int kb = kb0; kb < kb0 + kblocks; ++kb, ++it) {
                    const int slot = it % kGemmStages;
                    if (!mbar_wait_or_abort(&empty[slot], ((it / kGemmStages) & 1) ^ 1, err, abort_flag)) {
                        ok = false;
                        break;
                    }
                    unsigned char *st = tiles + (size_t)slot * kStageBytes;
                    mbar_arrive_expect_tx(&full[slot], kStageBytes);
                    tma_load_2d(st, &tmA, kb * BK, arow, &full[slot]);
                    if (SPLIT_B) {
                        tma_load_2d(st + kABytes, &tmB, kb * BK, brow, &full[slot]);
                        tma_load_2d(st + kABytes + kBBytes / 2, &tmB2, kb * BK, brow, &full[slot]);
                    } else {
                        tma_load_2d(st + kABytes, &tmB, kb * BK, brow, &full[slot]);
                    }
                }
            }
            // every load issued must land before the CTA exits
            for (int j = (it > kGemmStages ? it - kGemmStages : 0); j < it; ++j)
                mbar_wait(&full[j % kGemmStages], (j / kGemmStages) & 1, err);
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
                    const int slot = it % kGemmStages;
                    if (!mbar_wait_or_abort(&full[slot], (it / kGemmStages) & 1, err, abort_flag)) {
                        ok = false;
                        break;
                    }
                    tc_fence_after();
                    const uint32_t a_addr = smem_u32(tiles + (size_t)slot * kStageBytes);
                    const uint64_t ad = smem_desc_sw128(a_addr), bd = smem_desc_sw128(a_addr + kABytes);
#pragma unroll
                    for (int kk = 0; kk < BK / 16; ++kk)
                        mma_bf16(dtm, ad + (uint64_t)(2 * kk), bd + (uint64_t)(2 * kk), kIdesc, (kb | kk) != 0);
                    mma_commit(&empty[slot]);  // the stage is free once these MMAs have read it
                }
                if (!ok) break;
                mma_commit(&tfull[b]);  // the accumulator is complete
            }
            mma_commit(done);
            mbar_wait(done, 0, err);
        }
    } else {
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
            epilogue_tile<EPI, false>(p, ti, tbase, row);
            tc_fence_before();
            mbar_arrive(&tempty[b]);
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
// host side: tensor maps and launches
// ---------------------------------------------------------------------------
PFN_cuTensorMapEncodeTiled_v12000 get_encode() {
    static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
    if (!fn) {
        cudaDriverEntryPointQueryResult q;
        void *ptr = nullptr;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &ptr, 12000, cudaEnableDefault, &q) ==
                cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(ptr);
    }
    return fn;
}

bool make_tmap_u8(CUtensorMap *tm, const void *base, uint64_t rows, uint64_t cols, uint32_t box_cols,
                  uint32_t box_rows, bool swz32) {
    auto enc = get_encode();
    if (!enc) return false;
    cuuint64_t dims[2] = {cols, rows};
    cuuint64_t strides[1] = {cols};
    cuuint32_t box[2] = {box_cols, box_rows};
    cuuint32_t estr[2] = {1, 1};
    CUresult r = enc(tm, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, const_cast<void *>(base), dims, strides, box, estr,
                     CU_TENSOR_MAP_INTERLEAVE_NONE, swz32 ? CU_TENSOR_MAP_SWIZZLE_32B : CU_TENSOR_MAP_SWIZZLE_NONE,
                     CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS;
}

// 2-D bf16 tensor [rows, K] row-major; box = 64 K-elements x box_rows rows, 128-byte swizzle.
bool make_tmap_bf16(CUtensorMap *tm, const void *base, uint64_t rows, uint64_t K, uint32_t box_rows) {
    return make_tmap_bf16_ld(tm, base, rows, K, K, box_rows);
}

bool make_tmap_bf16_ld(CUtensorMap *tm, const void *base, uint64_t rows, uint64_t K, uint64_t ld, uint32_t box_rows) {
    auto enc = get_encode();
    if (!enc) return false;
    cuuint64_t dims[2] = {K, rows};
    cuuint64_t strides[1] = {ld * 2};
    cuuint32_t box[2] = {(cuuint32_t)BK, box_rows};
    cuuint32_t estr[2] = {1, 1};
    CUresult r = enc(tm, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void *>(base), dims, strides, box, estr,
                     CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                     CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS;
}

template <int EPI, bool SPLIT_B>
static cudaError_t launch_gemm(const CUtensorMap &a, const CUtensorMap &b, const CUtensorMap &b2,
                               const GemmParams &p, int grid, cudaStream_t st) {
    static std::atomic<uint64_t> attr_set{0};
    cudaError_t e = set_smem_limit_once((const void *)grouped_gemm_kernel<EPI, SPLIT_B>, (int)kGemmSmem, attr_set);
    if (e != cudaSuccess) return e;
    grouped_gemm_kernel<EPI, SPLIT_B><<<grid, kGemmThreads, kGemmSmem, st>>>(a, b, b2, p);
    return cudaGetLastError();
}

cudaError_t launch_router_gemm(const LayerDev &L, const Workspace &ws, const uint16_t *x, int T, cudaStream_t st) {
    CUtensorMap ta, tb;
    if (!make_tmap_bf16(&ta, x, (uint64_t)T, (uint64_t)L.d, BM)) return cudaErrorInvalidValue;
    if (!make_tmap_bf16(&tb, L.wr, (uint64_t)L.E, (uint64_t)L.d, BN)) return cudaErrorInvalidValue;
    GemmParams p{};
    p.tile_off = nullptr;
    p.n_rows = T;
    p.groups = 1;
    p.nt = (L.E + BN - 1) / BN;
    p.K = L.d;
    p.b_rows_per_group = 0;
    p.out_f32 = ws.logits;
    p.ld = L.E;
    p.n_valid = L.E;
    p.bias = L.bias;
    p.err = &ws.ctrl->err;
    // K in kRouterSplit parts (partial logits summed in order by the top-k):
    // T = 4096 has only 32 row tiles, too few for the SMs
    p.ksplit = router_ksplit(L.d);
    p.split_stride = (size_t)L.max_T * L.E;
    int tiles = ((T + BM - 1) / BM) * p.nt * p.ksplit;
    int grid = tiles < L.num_sms ? tiles : L.num_sms;
    return launch_gemm<EPI_LOGITS, false>(ta, tb, tb, p, grid, st);
}

cudaError_t launch_prefill_experts(const LayerDev &L, const Workspace &ws, const uint16_t *x, int T, cudaStream_t st,
                                   int *launches) {
    (void)x;
    const uint64_t rows = (uint64_t)L.max_T * L.k;
    CUtensorMap ta, tg, tu, th, td;
    if (!make_tmap_bf16(&ta, ws.xperm, rows, (uint64_t)L.d, BM) ||
        !make_tmap_bf16_ld(&tg, L.wg, (uint64_t)L.E * L.I, (uint64_t)L.d, (uint64_t)L.gu_ld, BN / 2) ||
        !make_tmap_bf16_ld(&tu, L.wu, (uint64_t)L.E * L.I, (uint64_t)L.d, (uint64_t)L.gu_ld, BN / 2) ||
        !make_tmap_bf16(&th, ws.h, rows, (uint64_t)L.I, BM) ||
        !make_tmap_bf16(&td, L.wd, (uint64_t)L.E * L.d, (uint64_t)L.I, BN))
        return cudaErrorInvalidValue;
    GemmParams p{};
    p.ksplit = 1;
    p.tile_off = ws.tile_off;
    p.row_off = ws.offsets;
    p.groups = L.E;
    p.err = &ws.ctrl->err;
    // gate/up + SwiGLU: N tile = 128 gate columns + the matching 128 up columns
    p.nt = L.I / (BN / 2);
    p.K = L.d;
    p.b_rows_per_group = L.I;
    p.out_bf16 = reinterpret_cast<uint16_t *>(ws.h);
    p.ld = L.I;
    cudaError_t e = launch_gemm<EPI_SWIGLU, true>(ta, tg, tu, p, L.num_sms, st);
    if (e != cudaSuccess) return e;
    // down: Y = H . Wd^T, accumulated in fp32 and stored in bf16 over the
    // gathered token rows, which the gate/up GEMM no longer needs (fp32 Y for
    // the per-expert-normalised variant)
    p.nt = L.d / BN;
    p.K = L.I;
    p.b_rows_per_group = L.d;
    p.ld = L.d;
    p.n_valid = L.d;
    if (L.expert_norm) {  // the normalising combine reads fp32 Y
        p.out_bf16 = nullptr;
        p.out_f32 = ws.Y;
        e = launch_gemm<EPI_F32, false>(th, td, td, p, L.num_sms, st);
    } else {
        p.out_bf16 = ws.xperm;
        p.out_f32 = nullptr;
        e = launch_gemm<EPI_BF16, false>(th, td, td, p, L.num_sms, st);
    }
    *launches += 2;
    return e;
}

}  // namespace moe
