// gemm.cuh — pieces shared by the tensor-core grouped GEMMs (prefill.cu for
// bf16 experts, prefill_fp4.cu for NVFP4 experts): tile scheduling over the
// experts' row groups, inline PTX for TMA tensor loads and tcgen05 (TMEM
// allocation, MMA, commit, loads), shared-memory and instruction descriptors,
// and the epilogue of one accumulator tile.
#pragma once

#include <cuda.h>
#include <cudaTypedefs.h>
#include <cuda_runtime.h>

#include "common.cuh"

namespace moe {

constexpr int BM = 128, BK = 64, BN = 256;
constexpr uint32_t kTmemCols = 512;           // two 128 x 256 fp32 accumulators

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
    const float *row_scale;   // scaled epilogues: per output row, or null
    const float *col_scale;   // scaled epilogues: per group (gate half for SwiGLU), or null
    const float *col_scale2;  // scaled SwiGLU: per group, up half, or null
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
// The same with f16 A and B (the A/B type fields 0 = f16).
constexpr uint32_t kIdescF16 = (1u << 4) | ((uint32_t)(BN >> 3) << 17) | ((uint32_t)(BM >> 4) << 24);

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
// epilogue of one tile, by one of the four epilogue warps (TMEM lane quarter
// = warp % 4, `row` = the tile row this thread owns). SCALED: the
// accumulator is multiplied by the row's scale (p.row_scale, when set) and
// the group's column scale (p.col_scale; for SwiGLU the up half takes
// p.col_scale2) before the epilogue's function.
// ---------------------------------------------------------------------------
template <int EPI, bool SCALED>
__device__ __forceinline__ void epilogue_tile(const GemmParams &p, const TileInfo &ti, uint32_t tbase, int row) {
    const int grow = ti.m * BM + row;  // row within the group
    const bool valid = grow < ti.rows;
    const size_t orow = (size_t)(ti.row0 + grow);
    float sc0 = 1.f, sc1 = 1.f;
    if (SCALED) {
        const float rs = (p.row_scale && valid) ? p.row_scale[orow] : 1.f;
        sc0 = rs * (p.col_scale ? p.col_scale[ti.g] : 1.f);
        sc1 = rs * (p.col_scale2 ? p.col_scale2[ti.g] : 1.f);
    }
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
                    float g0 = __uint_as_float(g[2 * i]), g1 = __uint_as_float(g[2 * i + 1]);
                    float u0 = __uint_as_float(u[2 * i]), u1 = __uint_as_float(u[2 * i + 1]);
                    if (SCALED) {
                        g0 *= sc0;
                        g1 *= sc0;
                        u0 *= sc1;
                        u1 *= sc1;
                    }
                    const float h0 = silu(g0) * u0, h1 = silu(g1) * u1;
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
            if (SCALED) {
#pragma unroll
                for (int i = 0; i < 16; ++i) v[i] = __float_as_uint(__uint_as_float(v[i]) * sc0);
            }
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
                    if (col0 + 16 <= p.n_valid && (p.n_valid & 3) == 0 &&
                        (!add_bias || (reinterpret_cast<uintptr_t>(p.bias) & 15u) == 0)) {
                        // 16-byte stores: a lane's row is its own, so every
                        // scalar store would be a separate L2 transaction
#pragma unroll
                        for (int i = 0; i < 16; i += 4) {
                            float4 o = make_float4(__uint_as_float(v[i]), __uint_as_float(v[i + 1]),
                                                   __uint_as_float(v[i + 2]), __uint_as_float(v[i + 3]));
                            if (add_bias) {
                                const float4 bv = __ldg(reinterpret_cast<const float4 *>(p.bias + col0 + i));
                                o.x += bv.x;
                                o.y += bv.y;
                                o.z += bv.z;
                                o.w += bv.w;
                            }
                            *reinterpret_cast<float4 *>(dst + i) = o;
                        }
                    } else {
#pragma unroll
                        for (int i = 0; i < 16; ++i)
                            if (col0 + i < p.n_valid) dst[i] = __uint_as_float(v[i]) + (add_bias ? p.bias[col0 + i] : 0.f);
                    }
                } else {
#pragma unroll
                    for (int i = 0; i < 16; i += 4)
                        *reinterpret_cast<float4 *>(dst + i) =
                            make_float4(__uint_as_float(v[i]), __uint_as_float(v[i + 1]), __uint_as_float(v[i + 2]),
                                        __uint_as_float(v[i + 3]));
                }
            }
        }
    }
}

// ---------------------------------------------------------------------------
// host side: tensor maps (prefill.cu)
// ---------------------------------------------------------------------------
// 2-D bf16 (or any 2-byte) tensor [rows, K] row-major; box = 64 K-elements x
// box_rows rows, 128-byte swizzle (the K-major layout the MMA descriptors read).
bool make_tmap_bf16(CUtensorMap *tm, const void *base, uint64_t rows, uint64_t K, uint32_t box_rows);
// The same with rows ld elements apart (ld >= K, ld * 2 a multiple of 16).
bool make_tmap_bf16_ld(CUtensorMap *tm, const void *base, uint64_t rows, uint64_t K, uint64_t ld, uint32_t box_rows);
// 2-D byte tensor [rows, cols] row-major; box = box_cols x box_rows, no swizzle
// (swz32: the 32-byte swizzle, box_cols == 32: in shared memory the two 16-byte
// halves of row r are swapped when bit 2 of r is set).
bool make_tmap_u8(CUtensorMap *tm, const void *base, uint64_t rows, uint64_t cols, uint32_t box_cols,
                  uint32_t box_rows, bool swz32 = false);

}  // namespace moe
