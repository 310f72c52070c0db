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

#include "common.cuh"

namespace moe {

constexpr int BM = 128, BK = 64, BN = 256;
constexpr int kGemmStages = 4;
constexpr int kGemmThreads = 192;
constexpr uint32_t kTmemCols = 512;
constexpr uint32_t kABytes = BM * BK * 2;       // 16 KB
constexpr uint32_t kBBytes = BN * BK * 2;       // 32 KB
constexpr uint32_t kStageBytes = kABytes + kBBytes;
constexpr size_t kGemmSmem = 1024 + (size_t)kGemmStages * kStageBytes + 256;

enum { EPI_LOGITS = 0, EPI_SWIGLU = 1, EPI_F32 = 2, EPI_BF16 = 3 };

struct GemmParams {
    const int32_t *tile_off;  // [G+1] prefix of 128-row tiles per group; nullptr: one group
    const int32_t *row_off;   // [G+1] first row of each group in A and in the output
    int n_rows;               // rows of the single group (tile_off == nullptr)
    int groups;
    int nt;                   // n-tiles per m-tile
    int K;
    int b_rows_per_group;     // rows of B per group (0 for the router)
    float *out_f32;           // logits [rows, ld] / Y [rows, ld]
    uint16_t *out_bf16;       // H [rows, ld] (SwiGLU) / Y [rows, ld] (EPI_BF16)
    int ld;                   // output row stride in elements
    int n_valid;              // columns < n_valid are stored (router: E)
    const float *bias;
    uint32_t *err;
    int ksplit;               // single group only: K split in ksplit parts, part s written at out_f32 + s * split_stride
    size_t split_stride;
};

// ---------------------------------------------------------------------------
// PTX wrappers: TMA tensor loads, tcgen05 (TMEM alloc, MMA, commit, ld)
// ---------------------------------------------------------------------------
__device__ __forceinline__ void tma_load_2d(void *dst, const CUtensorMap *tm, int x, int y, uint64_t *bar) {
    asm volatile(
        "cp.async.bulk.tensor.2d.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1, {%2, %3}], [%4];" ::"r"(
            smem_u32(dst)),
        "l"(reinterpret_cast<uint64_t>(tm)), "r"(x), "r"(y), "r"(smem_u32(bar))
        : "memory");
}

__device__ __forceinline__ void tmem_alloc(uint32_t *dst_smem, uint32_t ncols) {
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(smem_u32(dst_smem)),
                 "r"(ncols)
                 : "memory");
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
}

__device__ __forceinline__ void tmem_dealloc(uint32_t taddr, uint32_t ncols) {
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(ncols) : "memory");
}

__device__ __forceinline__ void tc_fence_before() { asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory"); }
__device__ __forceinline__ void tc_fence_after() { asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory"); }

__device__ __forceinline__ void mma_bf16(uint32_t tmem_d, uint64_t adesc, uint64_t bdesc, uint32_t idesc,
                                         uint32_t accumulate) {
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "setp.ne.b32 p, %4, 0;\n\t"
        "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(tmem_d),
        "l"(adesc), "l"(bdesc), "r"(idesc), "r"(accumulate)
        : "memory");
}

__device__ __forceinline__ void mma_commit(uint64_t *bar) {
    asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(smem_u32(bar))
                 : "memory");
}

__device__ __forceinline__ void tmem_ld16(uint32_t taddr, uint32_t v[16]) {
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x16.b32 {%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, "
        "%15}, [%16];"
        : "=r"(v[0]), "=r"(v[1]), "=r"(v[2]), "=r"(v[3]), "=r"(v[4]), "=r"(v[5]), "=r"(v[6]), "=r"(v[7]),
          "=r"(v[8]), "=r"(v[9]), "=r"(v[10]), "=r"(v[11]), "=r"(v[12]), "=r"(v[13]), "=r"(v[14]), "=r"(v[15])
        : "r"(taddr));
}

__device__ __forceinline__ void tmem_ld_wait() { asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory"); }

// Shared-memory matrix descriptor of a K-major tile written by TMA with the
// 128-byte swizzle: rows of 128 bytes, 8-row groups 1024 bytes apart.
__device__ __forceinline__ uint64_t smem_desc_sw128(uint32_t addr) {
    uint64_t d = 0;
    d |= (uint64_t)((addr & 0x3FFFFu) >> 4);   // start address
    d |= (uint64_t)1 << 16;                    // leading byte offset (unused with this swizzle)
    d |= (uint64_t)(1024 >> 4) << 32;          // stride byte offset: 8 rows x 128 B
    d |= (uint64_t)1 << 46;                    // descriptor version
    d |= (uint64_t)2 << 61;                    // 128-byte swizzle
    return d;
}

// Instruction descriptor: kind::f16 with bf16 A and B, fp32 accumulator,
// both operands K-major, M = 128, N = 256.
constexpr uint32_t kIdesc = (1u << 4) | (1u << 7) | (1u << 10) | ((uint32_t)(BN >> 3) << 17) |
                            ((uint32_t)(BM >> 4) << 24);

// ---------------------------------------------------------------------------
// tile scheduling
// ---------------------------------------------------------------------------
struct TileInfo {
    int g, m, n, row0, rows, ks;
};

__device__ __forceinline__ int total_tiles(const GemmParams &p) {
    if (!p.tile_off) return ((p.n_rows + BM - 1) / BM) * p.nt * p.ksplit;
    return p.tile_off[p.groups] * p.nt;
}

__device__ __forceinline__ TileInfo tile_info(const GemmParams &p, int tile) {
    TileInfo ti;
    if (!p.tile_off) {
        const int mt = (p.n_rows + BM - 1) / BM;
        ti.g = 0;
        ti.m = tile % mt;
        ti.n = (tile / mt) % p.nt;
        ti.ks = tile / (mt * p.nt);
        ti.row0 = 0;
        ti.rows = p.n_rows;
        return ti;
    }
    int lo = 0, hi = p.groups;  // find g: tile_off[g]*nt <= tile < tile_off[g+1]*nt
    while (hi - lo > 1) {
        int mid = (lo + hi) >> 1;
        if (p.tile_off[mid] * p.nt <= tile)
            lo = mid;
        else
            hi = mid;
    }
    while (lo < p.groups - 1 && p.tile_off[lo + 1] * p.nt <= tile) ++lo;  // skip empty groups
    const int mt = p.tile_off[lo + 1] - p.tile_off[lo];
    const int local = tile - p.tile_off[lo] * p.nt;
    ti.g = lo;
    ti.ks = 0;
    ti.m = local % mt;
    ti.n = local / mt;
    ti.row0 = p.row_off[lo];
    ti.rows = p.row_off[lo + 1] - p.row_off[lo];
    return ti;
}

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
            const int grow = ti.m * BM + row;  // row within the group
            const bool valid = grow < ti.rows;
            const size_t orow = (size_t)(ti.row0 + grow);
            if (EPI == EPI_SWIGLU) {
#pragma unroll 1
                for (int j0 = 0; j0 < BN / 2; j0 += 16) {
                    uint32_t g[16], u[16];
                    tmem_ld16(tbase + j0, g);
                    tmem_ld16(tbase + BN / 2 + j0, u);
                    tmem_ld_wait();
                    if (valid) {
                        uint32_t packed[8];
#pragma unroll
                        for (int i = 0; i < 8; ++i) {
                            float h0 = silu(__uint_as_float(g[2 * i])) * __uint_as_float(u[2 * i]);
                            float h1 = silu(__uint_as_float(g[2 * i + 1])) * __uint_as_float(u[2 * i + 1]);
                            packed[i] = (uint32_t)f32_to_bf16_rn(h0) | ((uint32_t)f32_to_bf16_rn(h1) << 16);
                        }
                        uint4 *dst = reinterpret_cast<uint4 *>(p.out_bf16 + orow * p.ld + ti.n * (BN / 2) + j0);
                        dst[0] = make_uint4(packed[0], packed[1], packed[2], packed[3]);
                        dst[1] = make_uint4(packed[4], packed[5], packed[6], packed[7]);
                    }
                }
            } else {
#pragma unroll 1
                for (int j0 = 0; j0 < BN; j0 += 16) {
                    uint32_t v[16];
                    tmem_ld16(tbase + j0, v);
                    tmem_ld_wait();
                    const int col0 = ti.n * BN + j0;
                    if (valid && EPI == EPI_BF16) {
                        uint32_t packed[8];
#pragma unroll
                        for (int i = 0; i < 8; ++i)
                            packed[i] = (uint32_t)f32_to_bf16_rn(__uint_as_float(v[2 * i])) |
                                        ((uint32_t)f32_to_bf16_rn(__uint_as_float(v[2 * i + 1])) << 16);
                        uint4 *dst = reinterpret_cast<uint4 *>(p.out_bf16 + orow * p.ld + col0);
                        dst[0] = make_uint4(packed[0], packed[1], packed[2], packed[3]);
                        dst[1] = make_uint4(packed[4], packed[5], packed[6], packed[7]);
                    } else if (valid) {
                        float *dst = p.out_f32 + (size_t)ti.ks * p.split_stride + orow * p.ld + col0;
                        if (EPI == EPI_LOGITS) {
                            const bool add_bias = p.bias && ti.ks == 0;  // once, with the first part of K
#pragma unroll
                            for (int i = 0; i < 16; ++i)
                                if (col0 + i < p.n_valid)
                                    dst[i] = __uint_as_float(v[i]) + (add_bias ? p.bias[col0 + i] : 0.f);
                        } else {
#pragma unroll
                            for (int i = 0; i < 16; i += 4)
                                *reinterpret_cast<float4 *>(dst + i) =
                                    make_float4(__uint_as_float(v[i]), __uint_as_float(v[i + 1]),
                                                __uint_as_float(v[i + 2]), __uint_as_float(v[i + 3]));
                        }
                    }
                }
            }
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
static PFN_cuTensorMapEncodeTiled_v12000 get_encode() {
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

// 2-D bf16 tensor [rows, K] row-major; box = 64 K-elements x box_rows rows, 128-byte swizzle.
bool make_tmap_bf16(CUtensorMap *tm, const void *base, uint64_t rows, uint64_t K, uint32_t box_rows) {
    auto enc = get_encode();
    if (!enc) return false;
    cuuint64_t dims[2] = {K, rows};
    cuuint64_t strides[1] = {K * 2};
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
        !make_tmap_bf16(&tg, L.wg, (uint64_t)L.E * L.I, (uint64_t)L.d, BN / 2) ||
        !make_tmap_bf16(&tu, L.wu, (uint64_t)L.E * L.I, (uint64_t)L.d, BN / 2) ||
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
