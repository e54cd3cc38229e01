// Online-FP8 operands of the projections: per-row e4m3 quantisation of bf16
// tensors (weights once at finalize, activations on every encode) and the
// RMSNorm that emits its output already quantised.
//
// Page "vllm-omni vllm_omni/diffusion/models/minimax_h3/encoder.py":
// _validate_encoder_quant_config (online FP8 only) and the _is_quantized_linear
// branches (packed QKV / gate-up as one quantised linear).  Scaling: one fp32
// scale per row, amax / 448; q = e4m3(x * (448 / amax)) with the reciprocal and
// the product each rounded once in fp32, then rounded to nearest even and
// saturating (the e4m3 "fn" variant, largest 448).
#include <cuda_fp8.h>

#include "common.cuh"
#include "kernels.h"

namespace h3 {

namespace {

constexpr int QT = 256;   // threads per row

__device__ __forceinline__ float block_max(float v, float *red) {
    #pragma unroll
    for (int o = 16; o > 0; o >>= 1) v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, o));
    if ((threadIdx.x & 31) == 0) red[threadIdx.x >> 5] = v;
    __syncthreads();
    float m = red[0];
    #pragma unroll
    for (int i = 1; i < QT / 32; ++i) m = fmaxf(m, red[i]);
    return m;
}

// Eight values -> eight e4m3 bytes (x * inv in fp32, then the hardware conversion).
__device__ __forceinline__ uint2 quant8(const float (&f)[8], float inv) {
    uint32_t w[2];
    #pragma unroll
    for (int h = 0; h < 2; ++h) {
        const __nv_fp8x2_storage_t lo =
            __nv_cvt_float2_to_fp8x2(make_float2(__fmul_rn(f[4 * h], inv), __fmul_rn(f[4 * h + 1], inv)),
                                     __NV_SATFINITE, __NV_E4M3);
        const __nv_fp8x2_storage_t hi =
            __nv_cvt_float2_to_fp8x2(make_float2(__fmul_rn(f[4 * h + 2], inv), __fmul_rn(f[4 * h + 3], inv)),
                                     __NV_SATFINITE, __NV_E4M3);
        w[h] = (uint32_t)lo | ((uint32_t)hi << 16);
    }
    return make_uint2(w[0], w[1]);
}

__device__ __forceinline__ void unpack8(const uint4 v, float (&f)[8]) {
    f[0] = bf16_lo(v.x); f[1] = bf16_hi(v.x); f[2] = bf16_lo(v.y); f[3] = bf16_hi(v.y);
    f[4] = bf16_lo(v.z); f[5] = bf16_hi(v.z); f[6] = bf16_lo(v.w); f[7] = bf16_hi(v.w);
}

// One CTA per row: amax pass, then the quantising pass (the row is re-read from L1/L2).
__global__ void __launch_bounds__(QT) quant_rows_kernel(const bf16 *__restrict__ x, int ldx, int cols,
                                                        uint8_t *__restrict__ q, int ldq, float *scale) {
    pdl_trigger();
    pdl_wait();
    __shared__ float red[QT / 32];
    const int row = blockIdx.x;
    const uint4 *xr = reinterpret_cast<const uint4 *>(x + (size_t)row * ldx);
    const int nvec = cols >> 3;
    float amax = 0.f;
    for (int i = threadIdx.x; i < nvec; i += QT) {
        float f[8];
        unpack8(xr[i], f);
        #pragma unroll
        for (int k = 0; k < 8; ++k) amax = fmaxf(amax, fabsf(f[k]));
    }
    amax = block_max(amax, red);
    const float inv = amax > 0.f ? __fdiv_rn(448.0f, amax) : 1.0f;
    if (threadIdx.x == 0) scale[row] = amax > 0.f ? __fdiv_rn(amax, 448.0f) : 1.0f;
    uint2 *qr = reinterpret_cast<uint2 *>(q + (size_t)row * ldq);
    for (int i = threadIdx.x; i < nvec; i += QT) {
        float f[8];
        unpack8(xr[i], f);
        qr[i] = quant8(f, inv);
    }
}

// One CTA per row with the row's amax already known: a single quantising pass; the amax
// slot is cleared for the next producer once every thread has read it.
__global__ void __launch_bounds__(QT) quant_rows_amax_kernel(const bf16 *__restrict__ x, int ldx, int cols,
                                                             uint8_t *__restrict__ q, int ldq, float *scale,
                                                             float *row_amax) {
    pdl_trigger();
    pdl_wait();
    const int row = blockIdx.x;
    const float amax = row_amax[row];
    __syncthreads();
    if (threadIdx.x == 0) {
        row_amax[row] = 0.f;
        scale[row] = amax > 0.f ? __fdiv_rn(amax, 448.0f) : 1.0f;
    }
    const float inv = amax > 0.f ? __fdiv_rn(448.0f, amax) : 1.0f;
    const uint4 *xr = reinterpret_cast<const uint4 *>(x + (size_t)row * ldx);
    uint2 *qr = reinterpret_cast<uint2 *>(q + (size_t)row * ldq);
    const int nvec = cols >> 3;
    // four 16-byte loads in flight per thread before the first conversion
    for (int i0 = threadIdx.x; i0 < nvec; i0 += 4 * QT) {
        uint4 v[4];
        #pragma unroll
        for (int u = 0; u < 4; ++u)
            if (i0 + u * QT < nvec) v[u] = xr[i0 + u * QT];
        #pragma unroll
        for (int u = 0; u < 4; ++u) {
            if (i0 + u * QT < nvec) {
                float f[8];
                unpack8(v[u], f);
                qr[i0 + u * QT] = quant8(f, inv);
            }
        }
    }
}

// RMSNorm of one row kept in registers (cols <= 8192), rounded to bf16, then quantised.
// 128 threads per row, each holding VPT 16-byte vectors of x and of the norm weight (both
// loaded before the first reduction); the bf16 output overwrites x in place (packed, exact),
// so the row costs 8 registers per vector and a 5120-wide row fits one wave of CTAs.
constexpr int NQ_T = 128;
template <int VPT>
__global__ void __launch_bounds__(NQ_T) rmsnorm_q8_kernel(const bf16 *__restrict__ x, const bf16 *__restrict__ w,
                                                          uint8_t *__restrict__ q, float *scale, int cols,
                                                          float eps) {
    pdl_trigger();
    pdl_wait();
    __shared__ float red[2][NQ_T / 32];
    const int row = blockIdx.x;
    const int nvec = cols >> 3;
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const uint4 *xr = reinterpret_cast<const uint4 *>(x + (size_t)row * cols);
    const uint4 *wr = reinterpret_cast<const uint4 *>(w);
    uint4 xv[VPT], gv[VPT];
    #pragma unroll
    for (int i = 0; i < VPT; ++i) {
        const int idx = threadIdx.x + i * NQ_T;
        xv[i] = idx < nvec ? xr[idx] : make_uint4(0u, 0u, 0u, 0u);
        gv[i] = idx < nvec ? wr[idx] : make_uint4(0u, 0u, 0u, 0u);
    }
    float ss = 0.f;
    #pragma unroll
    for (int i = 0; i < VPT; ++i) {
        float f[8];
        unpack8(xv[i], f);
        #pragma unroll
        for (int k = 0; k < 8; ++k) ss = fmaf(f[k], f[k], ss);
    }
    #pragma unroll
    for (int o = 16; o > 0; o >>= 1) ss += __shfl_xor_sync(0xffffffffu, ss, o);
    if (lane == 0) red[0][warp] = ss;
    __syncthreads();
    float tot = 0.f;
    #pragma unroll
    for (int i = 0; i < NQ_T / 32; ++i) tot += red[0][i];
    const float rstd = 1.0f / sqrtf(tot / (float)cols + eps);
    float amax = 0.f;
    #pragma unroll
    for (int i = 0; i < VPT; ++i) {
        float f[8], g[8];
        unpack8(xv[i], f);
        unpack8(gv[i], g);
        uint32_t y[4];
        #pragma unroll
        for (int k = 0; k < 8; k += 2) {
            const float a = round_bf16(f[k] * rstd * g[k]), b = round_bf16(f[k + 1] * rstd * g[k + 1]);
            amax = fmaxf(amax, fmaxf(fabsf(a), fabsf(b)));   // the norm's bf16 output
            y[k >> 1] = pack_bf16x2(a, b);
        }
        xv[i] = make_uint4(y[0], y[1], y[2], y[3]);
    }
    #pragma unroll
    for (int o = 16; o > 0; o >>= 1) amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, o));
    if (lane == 0) red[1][warp] = amax;
    __syncthreads();
    amax = red[1][0];
    #pragma unroll
    for (int i = 1; i < NQ_T / 32; ++i) amax = fmaxf(amax, red[1][i]);
    const float inv = amax > 0.f ? __fdiv_rn(448.0f, amax) : 1.0f;
    if (threadIdx.x == 0) scale[row] = amax > 0.f ? __fdiv_rn(amax, 448.0f) : 1.0f;
    uint2 *qr = reinterpret_cast<uint2 *>(q + (size_t)row * cols);
    #pragma unroll
    for (int i = 0; i < VPT; ++i) {
        const int idx = threadIdx.x + i * NQ_T;
        if (idx < nvec) {
            float f[8];
            unpack8(xv[i], f);
            qr[idx] = quant8(f, inv);
        }
    }
}

}  // namespace

cudaError_t launch_quant_rows(const bf16 *x, int ldx, int rows, int cols, uint8_t *q, int ldq, float *scale,
                              cudaStream_t st) {
    if (rows <= 0) return cudaSuccess;
    if (cols % 8 || ldx % 8 || ldq % 8) return cudaErrorInvalidValue;
    cudaLaunchAttribute at[1];
    cudaLaunchConfig_t cfg = pdl_config(dim3(rows), dim3(QT), 0, st, at);
    return cudaLaunchKernelEx(&cfg, quant_rows_kernel, x, ldx, cols, q, ldq, scale);
}

cudaError_t launch_quant_rows_amax(const bf16 *x, int ldx, int rows, int cols, uint8_t *q, int ldq, float *scale,
                                   float *row_amax, cudaStream_t st) {
    if (rows <= 0) return cudaSuccess;
    if (cols % 8 || ldx % 8 || ldq % 8 || !row_amax) return cudaErrorInvalidValue;
    cudaLaunchAttribute at[1];
    cudaLaunchConfig_t cfg = pdl_config(dim3(rows), dim3(QT), 0, st, at);
    return cudaLaunchKernelEx(&cfg, quant_rows_amax_kernel, x, ldx, cols, q, ldq, scale, row_amax);
}

cudaError_t launch_rmsnorm_q8(const bf16 *x, const bf16 *w, uint8_t *q, float *scale, int rows, int cols, float eps,
                              cudaStream_t st) {
    if (rows <= 0) return cudaSuccess;
    const int vpt = (cols / 8 + NQ_T - 1) / NQ_T;
    if (cols % 8 || vpt < 1 || vpt > 8) return cudaErrorInvalidValue;
    cudaLaunchAttribute at[1];
    cudaLaunchConfig_t cfg = pdl_config(dim3(rows), dim3(NQ_T), 0, st, at);
    switch (vpt) {
        case 1: return cudaLaunchKernelEx(&cfg, rmsnorm_q8_kernel<1>, x, w, q, scale, cols, eps);
        case 2: return cudaLaunchKernelEx(&cfg, rmsnorm_q8_kernel<2>, x, w, q, scale, cols, eps);
        case 3: return cudaLaunchKernelEx(&cfg, rmsnorm_q8_kernel<3>, x, w, q, scale, cols, eps);
        case 4: return cudaLaunchKernelEx(&cfg, rmsnorm_q8_kernel<4>, x, w, q, scale, cols, eps);
        case 5: return cudaLaunchKernelEx(&cfg, rmsnorm_q8_kernel<5>, x, w, q, scale, cols, eps);
        case 6: return cudaLaunchKernelEx(&cfg, rmsnorm_q8_kernel<6>, x, w, q, scale, cols, eps);
        case 7: return cudaLaunchKernelEx(&cfg, rmsnorm_q8_kernel<7>, x, w, q, scale, cols, eps);
        default: return cudaLaunchKernelEx(&cfg, rmsnorm_q8_kernel<8>, x, w, q, scale, cols, eps);
    }
}

}  // namespace h3
