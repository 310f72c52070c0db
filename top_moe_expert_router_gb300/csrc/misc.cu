// misc.cu — weighted combine, RMSNorm, NVFP4 quantiser and row gather.
//
// The combine sums the k expert outputs of a token in fp32, slot order fixed
// (j ascending): per-expert outputs are combined after the experts run, and
// bf16 partial sums of expert outputs cost quality ("TensorSharp Muse Spark
// benchmark", sections "Performance" and "Answer quality").
#include <cuda_fp4.h>
#include <cuda_fp8.h>
#include <cuda_runtime.h>

#include "common.cuh"

namespace moe {

// ---------------------------------------------------------------------------
// combine: out[t, c] = bf16( (res[t, c] +) sum_j w[t, j] * Y[pos[t, j], c] )
// ---------------------------------------------------------------------------
// Column q of a 16-byte vector of expert outputs (bf16: 8 columns; fp32: 4).
__device__ __forceinline__ float yelem(const uint4 &v, int q, const uint16_t *) {
    const uint32_t w = q < 2 ? v.x : q < 4 ? v.y : q < 6 ? v.z : v.w;
    return (q & 1) ? bf16hi(w) : bf16lo(w);
}
__device__ __forceinline__ float yelem(const uint4 &v, int q, const float *) {
    return __uint_as_float(q == 0 ? v.x : q == 1 ? v.y : q == 2 ? v.z : v.w);
}

// out[t, c] = bf16( (res[t, c] +) sum_j w[t, j] * Y[pos[t, j], c] ), CPT
// columns per thread (one 16-byte vector per slot); all slot records first,
// then every load (the slots' outputs and the residual, kept packed until
// used, so that four CTAs fit on an SM and hide the two dependent memory
// latencies), then the sum in fp32, j ascending.
template <typename YT, int CPT>
__global__ void __launch_bounds__(256, 4) combine_kernel(const YT *__restrict__ Y, const float *__restrict__ w,
                                                         const int32_t *__restrict__ pos,
                                                         const uint16_t *__restrict__ res, uint16_t *__restrict__ out,
                                                         int T, int d, int k, uint32_t *err, int rows) {
    static_assert(CPT * sizeof(YT) == 16, "one 16-byte vector per slot");
    // launched as a programmatic dependent: Y, w and pos come from the
    // kernels before it
    asm volatile("griddepcontrol.wait;" ::: "memory");
    const int t = blockIdx.y;
    const int c = (blockIdx.x * blockDim.x + threadIdx.x) * CPT;
    if (c >= d) return;
    float wj[8];
    int rj[8];
#pragma unroll
    for (int j = 0; j < 8; ++j) {
        wj[j] = j < k ? __ldcg(w + (size_t)t * k + j) : 0.f;
        rj[j] = j < k ? __ldcg(pos + (size_t)t * k + j) : 0;
        if ((unsigned)rj[j] >= (unsigned)rows) {
            atomicOr(err, ERRBIT_RANGE);
            rj[j] = 0;
            wj[j] = 0.f;
        }
    }
    uint4 yv[8];
#pragma unroll
    for (int j = 0; j < 8; ++j)
        yv[j] = j < k ? __ldcg(reinterpret_cast<const uint4 *>(Y + (size_t)rj[j] * d + c)) : make_uint4(0, 0, 0, 0);
    uint32_t rv[CPT / 2];
#pragma unroll
    for (int q = 0; q < CPT / 2; ++q) rv[q] = 0u;
    if (res) {
        if constexpr (CPT == 8) {
            const uint4 r4 = *reinterpret_cast<const uint4 *>(res + (size_t)t * d + c);
            rv[0] = r4.x;
            rv[1] = r4.y;
            rv[2] = r4.z;
            rv[3] = r4.w;
        } else {
            const uint2 r2 = *reinterpret_cast<const uint2 *>(res + (size_t)t * d + c);
            rv[0] = r2.x;
            rv[1] = r2.y;
        }
    }
    float acc[CPT];
#pragma unroll
    for (int q = 0; q < CPT; ++q) acc[q] = 0.f;
#pragma unroll
    for (int j = 0; j < 8; ++j)
        if (j < k) {
#pragma unroll
            for (int q = 0; q < CPT; ++q) acc[q] = fmaf(wj[j], yelem(yv[j], q, Y), acc[q]);
        }
    if (res) {
#pragma unroll
        for (int q = 0; q < CPT; q += 2) {
            acc[q] += bf16lo(rv[q / 2]);
            acc[q + 1] += bf16hi(rv[q / 2]);
        }
    }
    uint32_t o[CPT / 2];
#pragma unroll
    for (int q = 0; q < CPT / 2; ++q)
        o[q] = (uint32_t)f32_to_bf16_rn(acc[2 * q]) | ((uint32_t)f32_to_bf16_rn(acc[2 * q + 1]) << 16);
    if constexpr (CPT == 8)
        *reinterpret_cast<uint4 *>(out + (size_t)t * d + c) = make_uint4(o[0], o[1], o[2], o[3]);
    else
        *reinterpret_cast<uint2 *>(out + (size_t)t * d + c) = make_uint2(o[0], o[1]);
}

// With per-expert output normalisation: one CTA per token; pass 1 sums the
// squares of each slot's expert output over d, pass 2 forms
// (res +) sum_j w_j * Y_j / sqrt(mean(Y_j^2) + 1e-6) in fp32, j ascending.
__global__ void __launch_bounds__(256) combine_norm_kernel(const float *__restrict__ Y, const float *__restrict__ w,
                                                           const int32_t *__restrict__ pos,
                                                           const uint16_t *__restrict__ res,
                                                           uint16_t *__restrict__ out, int T, int d, int k,
                                                           uint32_t *err, int rows) {
    asm volatile("griddepcontrol.wait;" ::: "memory");
    __shared__ float part[8][8];
    __shared__ float fac[8];
    const int t = blockIdx.x, tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    float wj[8];
    int rj[8];
#pragma unroll
    for (int j = 0; j < 8; ++j) {
        wj[j] = j < k ? __ldcg(w + (size_t)t * k + j) : 0.f;
        rj[j] = j < k ? __ldcg(pos + (size_t)t * k + j) : 0;
        if ((unsigned)rj[j] >= (unsigned)rows) {
            atomicOr(err, ERRBIT_RANGE);
            rj[j] = 0;
            wj[j] = 0.f;
        }
    }
    float ss[8];
#pragma unroll
    for (int j = 0; j < 8; ++j) ss[j] = 0.f;
    for (int c = tid * 4; c < d; c += 1024) {
#pragma unroll
        for (int j = 0; j < 8; ++j) {
            if (j < k) {
                const float4 y = __ldcg(reinterpret_cast<const float4 *>(Y + (size_t)rj[j] * d + c));
                ss[j] = fmaf(y.x, y.x, fmaf(y.y, y.y, fmaf(y.z, y.z, fmaf(y.w, y.w, ss[j]))));
            }
        }
    }
#pragma unroll
    for (int j = 0; j < 8; ++j) {
        const float s = warp_sum(ss[j]);
        if (lane == 0) part[warp][j] = s;
    }
    __syncthreads();
    if (tid < 8) {
        float s = 0.f;
        for (int i = 0; i < 8; ++i) s += part[i][tid];
        fac[tid] = 1.0f / sqrtf(s / (float)d + 1e-6f);
    }
    __syncthreads();
    for (int c = tid * 4; c < d; c += 1024) {
        float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
        for (int j = 0; j < 8; ++j) {
            if (j < k) {
                const float4 y = __ldcg(reinterpret_cast<const float4 *>(Y + (size_t)rj[j] * d + c));
                const float f = fac[j];
                acc.x = fmaf(wj[j], y.x * f, acc.x);
                acc.y = fmaf(wj[j], y.y * f, acc.y);
                acc.z = fmaf(wj[j], y.z * f, acc.z);
                acc.w = fmaf(wj[j], y.w * f, acc.w);
            }
        }
        if (res) {
            const uint2 rv = *reinterpret_cast<const uint2 *>(res + (size_t)t * d + c);
            acc.x += bf16lo(rv.x);
            acc.y += bf16hi(rv.x);
            acc.z += bf16lo(rv.y);
            acc.w += bf16hi(rv.y);
        }
        uint2 o;
        o.x = (uint32_t)f32_to_bf16_rn(acc.x) | ((uint32_t)f32_to_bf16_rn(acc.y) << 16);
        o.y = (uint32_t)f32_to_bf16_rn(acc.z) | ((uint32_t)f32_to_bf16_rn(acc.w) << 16);
        *reinterpret_cast<uint2 *>(out + (size_t)t * d + c) = o;
    }
}

cudaError_t launch_combine(const LayerDev &L, const Workspace &ws, const uint16_t *res, uint16_t *out, int T,
                           cudaStream_t st, bool y_bf16) {
    cudaLaunchConfig_t cfg{};
    if (L.expert_norm) {
        cfg.gridDim = dim3(T);
        cfg.blockDim = dim3(256);
        cfg.stream = st;
        cudaLaunchAttribute attr[1];
        attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
        attr[0].val.programmaticStreamSerializationAllowed = 1;
        cfg.attrs = attr;
        cfg.numAttrs = 1;
        return cudaLaunchKernelEx(&cfg, combine_norm_kernel, (const float *)ws.Y, (const float *)ws.w,
                                  (const int32_t *)ws.pos, res, out, T, L.d, L.k, &ws.ctrl->err, T * L.k);
    }
    const int cpt = y_bf16 ? 8 : 4;   // columns per thread (d is a multiple of 64)
    cfg.gridDim = dim3((L.d / cpt + 255) / 256, T);
    cfg.blockDim = dim3(256);
    cfg.stream = st;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    if (y_bf16)
        return cudaLaunchKernelEx(&cfg, combine_kernel<uint16_t, 8>, (const uint16_t *)ws.xperm, (const float *)ws.w,
                                  (const int32_t *)ws.pos, res, out, T, L.d, L.k, &ws.ctrl->err, T * L.k);
    return cudaLaunchKernelEx(&cfg, combine_kernel<float, 4>, (const float *)ws.Y, (const float *)ws.w,
                              (const int32_t *)ws.pos, res, out, T, L.d, L.k, &ws.ctrl->err, T * L.k);
}

__global__ void __launch_bounds__(256) bf16_to_f32_kernel(const uint16_t *__restrict__ in, float *__restrict__ out,
                                                          size_t n) {
    for (size_t i = blockIdx.x * (size_t)blockDim.x + threadIdx.x; i < n; i += (size_t)gridDim.x * blockDim.x)
        out[i] = __uint_as_float((uint32_t)in[i] << 16);
}

cudaError_t launch_bf16_to_f32(const uint16_t *in, float *out, size_t n, cudaStream_t st) {
    if (n == 0) return cudaSuccess;
    const size_t blocks = (n + 255) / 256;
    bf16_to_f32_kernel<<<(unsigned)(blocks < 4096 ? blocks : 4096), 256, 0, st>>>(in, out, n);
    return cudaGetLastError();
}

// ---------------------------------------------------------------------------
// RMSNorm without learned scale: out = x / sqrt(mean(x^2) + eps)
// ---------------------------------------------------------------------------
__global__ void __launch_bounds__(256) rmsnorm_kernel(const uint16_t *__restrict__ x, uint16_t *__restrict__ out,
                                                      int d, float eps) {
    __shared__ float part[8];
    const int t = blockIdx.x, tid = threadIdx.x;
    const uint16_t *xr = x + (size_t)t * d;
    float ss = 0.f;
    for (int c = tid * 8; c < d; c += 256 * 8) {
        uint4 v = *reinterpret_cast<const uint4 *>(xr + c);
        uint32_t a[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            float lo = bf16lo(a[i]), hi = bf16hi(a[i]);
            ss = fmaf(lo, lo, ss);
            ss = fmaf(hi, hi, ss);
        }
    }
    ss = warp_sum(ss);
    if ((tid & 31) == 0) part[tid >> 5] = ss;
    __syncthreads();
    float tot = 0.f;
#pragma unroll
    for (int i = 0; i < 8; ++i) tot += part[i];
    const float r = 1.0f / sqrtf(tot / (float)d + eps);
    for (int c = tid * 8; c < d; c += 256 * 8) {
        uint4 v = *reinterpret_cast<const uint4 *>(xr + c);
        uint32_t a[4] = {v.x, v.y, v.z, v.w}, o[4];
#pragma unroll
        for (int i = 0; i < 4; ++i)
            o[i] = (uint32_t)f32_to_bf16_rn(bf16lo(a[i]) * r) | ((uint32_t)f32_to_bf16_rn(bf16hi(a[i]) * r) << 16);
        *reinterpret_cast<uint4 *>(out + (size_t)t * d + c) = make_uint4(o[0], o[1], o[2], o[3]);
    }
}

cudaError_t launch_rmsnorm(const uint16_t *x, uint16_t *out, int T, int d, float eps, cudaStream_t st) {
    rmsnorm_kernel<<<T, 256, 0, st>>>(x, out, d, eps);
    return cudaGetLastError();
}

// ---------------------------------------------------------------------------
// NVFP4 quantiser. Tensor scale s_t = amax / (6 * 448); block scale
// E4M3((amax_block / 6) / s_t); codes E2M1(w / (scale * s_t)); fp32 throughout,
// round to nearest even with saturation (the hardware conversions), the sign
// of a code always that of w.
// ---------------------------------------------------------------------------
__global__ void amax_kernel(const uint16_t *__restrict__ W, size_t per_tensor, float *amax_bits) {
    const int n = blockIdx.y;
    const uint16_t *src = W + (size_t)n * per_tensor;
    float m = 0.f;
    for (size_t i = ((size_t)blockIdx.x * blockDim.x + threadIdx.x) * 8; i < per_tensor;
         i += (size_t)gridDim.x * blockDim.x * 8) {
        uint4 v = *reinterpret_cast<const uint4 *>(src + i);
        uint32_t a[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
        for (int j = 0; j < 4; ++j) m = fmaxf(m, fmaxf(fabsf(bf16lo(a[j])), fabsf(bf16hi(a[j]))));
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) m = fmaxf(m, __shfl_xor_sync(0xFFFFFFFFu, m, o));
    // non-negative floats order like their bit patterns
    if ((threadIdx.x & 31) == 0) atomicMax(reinterpret_cast<unsigned int *>(amax_bits + n), __float_as_uint(m));
}

__device__ __forceinline__ float tensor_scale_from_amax(float amax) { return amax > 0.f ? amax / 2688.0f : 1.0f; }

__global__ void quantize_kernel(const uint16_t *__restrict__ W, size_t per_tensor, int K, const float *amax,
                                uint8_t *__restrict__ q, uint8_t *__restrict__ s) {
    const int n = blockIdx.y;
    const size_t nblk = per_tensor / 16;
    const float st = tensor_scale_from_amax(amax[n]);
    for (size_t b = (size_t)blockIdx.x * blockDim.x + threadIdx.x; b < nblk; b += (size_t)gridDim.x * blockDim.x) {
        const uint4 *src = reinterpret_cast<const uint4 *>(W + (size_t)n * per_tensor + b * 16);
        uint4 v0 = src[0], v1 = src[1];
        uint32_t a[8] = {v0.x, v0.y, v0.z, v0.w, v1.x, v1.y, v1.z, v1.w};
        float wv[16];
        float bmax = 0.f;
#pragma unroll
        for (int j = 0; j < 8; ++j) {
            wv[2 * j] = bf16lo(a[j]);
            wv[2 * j + 1] = bf16hi(a[j]);
            bmax = fmaxf(bmax, fmaxf(fabsf(wv[2 * j]), fabsf(wv[2 * j + 1])));
        }
        const float sbf = __fdiv_rn(__fdiv_rn(bmax, 6.0f), st);
        const __nv_fp8_storage_t sc = __nv_cvt_float_to_fp8(sbf, __NV_SATFINITE, __NV_E4M3);
        __half_raw hr = __nv_cvt_fp8_to_halfraw(sc, __NV_E4M3);
        const float scale = __fmul_rn(__half2float(*reinterpret_cast<__half *>(&hr)), st);
        uint32_t packed[2] = {0u, 0u};
#pragma unroll
        for (int j = 0; j < 16; ++j) {
            uint32_t code = 0u;
            if (scale != 0.f) {
                const float r = __fdiv_rn(wv[j], scale);
                code = (uint32_t)__nv_cvt_float_to_fp4(fabsf(r), __NV_E2M1, cudaRoundNearest) & 0x7u;
                code |= (__float_as_uint(wv[j]) >> 31) << 3;
            }
            packed[j >> 3] |= code << (4 * (j & 7));
        }
        *reinterpret_cast<uint2 *>(q + (size_t)n * (per_tensor / 2) + b * 8) = make_uint2(packed[0], packed[1]);
        s[(size_t)n * nblk + b] = (uint8_t)sc;
    }
}

__global__ void finalize_scale_kernel(float *g, int n) {
    int i = blockIdx.x * blockDim.x + threadIdx.x;
    if (i < n) g[i] = tensor_scale_from_amax(g[i]);
}

cudaError_t launch_quantize_nvfp4(const uint16_t *W, int n, int rows, int K, uint8_t *q, uint8_t *s, float *g,
                                  cudaStream_t st) {
    size_t per = (size_t)rows * K;
    cudaError_t e = cudaMemsetAsync(g, 0, sizeof(float) * n, st);
    if (e != cudaSuccess) return e;
    int bx = (int)((per / 8 + 255) / 256);
    if (bx > 1024) bx = 1024;
    amax_kernel<<<dim3(bx, n), 256, 0, st>>>(W, per, g);
    int qx = (int)((per / 16 + 255) / 256);
    if (qx > 2048) qx = 2048;
    quantize_kernel<<<dim3(qx, n), 256, 0, st>>>(W, per, K, g, q, s);
    finalize_scale_kernel<<<(n + 255) / 256, 256, 0, st>>>(g, n);
    return cudaGetLastError();
}

// ---------------------------------------------------------------------------
// gather: xperm[r, :] = x[perm[r], :] (prefill operand rows in expert order)
// ---------------------------------------------------------------------------
// One warp per gathered row (8 rows per CTA): the row's token read once, then
// all of the lane's 16-byte loads issued before its stores.
__global__ void __launch_bounds__(256) gather_rows_kernel(const uint16_t *__restrict__ x,
                                                          const int32_t *__restrict__ perm,
                                                          uint16_t *__restrict__ xp, int rows, int d, int T,
                                                          uint32_t *err) {
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
    constexpr int kV = 8;
    for (int i0 = 0; i0 < nv; i0 += 32 * kV) {
        uint4 v[kV];
#pragma unroll
        for (int j = 0; j < kV; ++j) {
            const int i = i0 + j * 32 + lane;
            if (i < nv) v[j] = __ldg(src + i);
        }
#pragma unroll
        for (int j = 0; j < kV; ++j) {
            const int i = i0 + j * 32 + lane;
            if (i < nv) dst[i] = v[j];
        }
    }
}

cudaError_t launch_gather_rows(const LayerDev &L, const Workspace &ws, const uint16_t *x, int T, cudaStream_t st) {
    const int rows = T * L.k;
    gather_rows_kernel<<<(rows + 7) / 8, 256, 0, st>>>(x, ws.perm, ws.xperm, rows, L.d, T, &ws.ctrl->err);
    return cudaGetLastError();
}

}  // namespace moe
