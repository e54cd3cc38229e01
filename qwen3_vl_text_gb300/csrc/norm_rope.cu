// Memory-bound steps of the decoder layer: RMSNorm over the hidden size, the
// pieces of the RMSNorm folded into the projections (row sums of squares of the
// layer input, the norm weight multiplied into the weight columns once at
// finalize) and the M-RoPE cos/sin tables (the per-head q/k RMSNorm + rotary
// embedding runs in the epilogue of the QKV projection, csrc/gemm.cu).
//
// Page "vllm-omni vllm_omni/diffusion/models/minimax_h3/encoder.py":
// MiniMaxH3Qwen3VLRMSNorm (fp32 variance and scaling) and
// MiniMaxH3Qwen3VLTextRotaryEmbedding with _apply_interleaved_mrope.  All
// arithmetic is fp32; RMSNorm rounds its output to bf16 once; the pages' bf16
// cast of cos/sin is not reproduced: the tables stay fp32.
#include <cmath>

#include "common.cuh"
#include "kernels.h"

namespace h3 {

namespace {

constexpr int NORM_THREADS = 128;
constexpr int NORM_VPT = 8;  // 8 x 16-byte vectors per thread -> cols <= 8192

__device__ __forceinline__ float warp_sum(float v) {
    #pragma unroll
    for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
    return v;
}

// One CTA per row.  y = bf16(x * (1/sqrt(mean(x^2) + eps)) * w).
__global__ void __launch_bounds__(NORM_THREADS) rmsnorm_kernel(const bf16 *__restrict__ x,
                                                               const bf16 *__restrict__ w, bf16 *y, int cols,
                                                               float eps) {
    pdl_trigger();
    pdl_wait();
    const int row = blockIdx.x;
    const int nvec = cols >> 3;
    const uint4 *xr = reinterpret_cast<const uint4 *>(x + (size_t)row * cols);
    const uint4 *wr = reinterpret_cast<const uint4 *>(w);
    uint4 v[NORM_VPT];
    float ss = 0.f;
    #pragma unroll
    for (int i = 0; i < NORM_VPT; ++i) {
        const int idx = threadIdx.x + i * NORM_THREADS;
        if (idx < nvec) {
            v[i] = xr[idx];
            const uint32_t u[4] = {v[i].x, v[i].y, v[i].z, v[i].w};
            #pragma unroll
            for (int k = 0; k < 4; ++k) {
                const float a = bf16_lo(u[k]), b = bf16_hi(u[k]);
                ss = fmaf(a, a, ss);
                ss = fmaf(b, b, ss);
            }
        }
    }
    __shared__ float red[NORM_THREADS / 32];
    ss = warp_sum(ss);
    if ((threadIdx.x & 31) == 0) red[threadIdx.x >> 5] = ss;
    __syncthreads();
    float tot = 0.f;
    #pragma unroll
    for (int i = 0; i < NORM_THREADS / 32; ++i) tot += red[i];
    const float rstd = 1.0f / sqrtf(tot / (float)cols + eps);
    uint4 *yr = reinterpret_cast<uint4 *>(y + (size_t)row * cols);
    #pragma unroll
    for (int i = 0; i < NORM_VPT; ++i) {
        const int idx = threadIdx.x + i * NORM_THREADS;
        if (idx < nvec) {
            const uint4 g = wr[idx];
            const uint32_t u[4] = {v[i].x, v[i].y, v[i].z, v[i].w};
            const uint32_t gw[4] = {g.x, g.y, g.z, g.w};
            uint32_t o[4];
            #pragma unroll
            for (int k = 0; k < 4; ++k)
                o[k] = pack_bf16x2(bf16_lo(u[k]) * rstd * bf16_lo(gw[k]), bf16_hi(u[k]) * rstd * bf16_hi(gw[k]));
            yr[idx] = make_uint4(o[0], o[1], o[2], o[3]);
        }
    }
}

// One thread per (row, slot of 128 columns): the slot's sum of squares in column order.  The
// row statistics the projections fold the RMSNorm with (the same sums the residual GEMM
// epilogues emit for their own output).
__global__ void row_sumsq_kernel(const bf16 *__restrict__ x, int rows, int cols, float *ss) {
    pdl_trigger();
    pdl_wait();
    const int slots = cols >> 7;
    const long long i = (long long)blockIdx.x * blockDim.x + threadIdx.x;
    if (i >= (long long)rows * slots) return;
    const int s = (int)(i / rows), r = (int)(i - (long long)s * rows);
    const uint4 *src = reinterpret_cast<const uint4 *>(x + (size_t)r * cols + (size_t)s * 128);
    float acc = 0.f;
    #pragma unroll 4
    for (int k = 0; k < 16; ++k) {
        const uint4 v = src[k];
        const uint32_t u[4] = {v.x, v.y, v.z, v.w};
        #pragma unroll
        for (int t = 0; t < 4; ++t) {
            const float a = bf16_lo(u[t]), b = bf16_hi(u[t]);
            acc = fmaf(a, a, acc);
            acc = fmaf(b, b, acc);
        }
    }
    ss[(size_t)s * rows + r] = acc;
}

// One thread per 8 weights: W[r][k] = bf16(W[r][k] * gamma[k]) on the selected rows.
__global__ void fold_cols_kernel(bf16 *W, int cols, const bf16 *__restrict__ gamma, int r0, int r1, int blk,
                                 int parity) {
    pdl_trigger();
    pdl_wait();
    const int per_row = cols >> 3;
    const long long i = (long long)blockIdx.x * blockDim.x + threadIdx.x;
    if (i >= (long long)(r1 - r0) * per_row) return;
    const int r = r0 + (int)(i / per_row), k8 = (int)(i % per_row);
    if (blk > 0 && ((r / blk) & 1) != parity) return;
    uint4 *w = reinterpret_cast<uint4 *>(W + (size_t)r * cols) + k8;
    const uint4 g = reinterpret_cast<const uint4 *>(gamma)[k8];
    const uint4 v = *w;
    const uint32_t u[4] = {v.x, v.y, v.z, v.w}, gg[4] = {g.x, g.y, g.z, g.w};
    uint32_t o[4];
    #pragma unroll
    for (int t = 0; t < 4; ++t)
        o[t] = pack_bf16x2(bf16_lo(u[t]) * bf16_lo(gg[t]), bf16_hi(u[t]) * bf16_hi(gg[t]));
    *w = make_uint4(o[0], o[1], o[2], o[3]);
}

// One thread per element i of the table, in either layout: row-major [S][d/2] (stride 0), or
// row-interleaved [d/8][stride][4], i = ((j/4) stride + s) 4 + j%4 (padding rows s >= S skipped).
__global__ void rope_table_kernel(const int32_t *__restrict__ pos, int S, const RopeParams rp, float *cos_t,
                                  float *sin_t, int stride) {
    pdl_trigger();
    pdl_wait();
    const int i = blockIdx.x * blockDim.x + threadIdx.x;
    if (i >= (stride ? stride : S) * rp.half_dim) return;
    int s, j;
    if (stride) {
        const int grp = i / (4 * stride), rem = i - grp * 4 * stride;
        s = rem >> 2;
        j = 4 * grp + (rem & 3);
        if (s >= S) return;
    } else {
        s = i / rp.half_dim;
        j = i - s * rp.half_dim;
    }
    const float p = (float)pos[rp.axis[j] * S + s];
    const float ang = __fmul_rn(p, rp.inv_freq[j]);
    float sn, cs;
    sincosf(ang, &sn, &cs);
    cos_t[i] = cs;
    sin_t[i] = sn;
}

}  // namespace

void make_rope_params(RopeParams *p, int head_dim, float theta, const int32_t section[3]) {
    p->half_dim = head_dim / 2;
    for (int j = 0; j < kMaxHalfDim; ++j) {
        p->inv_freq[j] = 0.f;
        p->axis[j] = 0;
    }
    for (int j = 0; j < p->half_dim; ++j) {
        // theta^(-2j/d) evaluated in double, rounded once to fp32
        p->inv_freq[j] = (float)(1.0 / std::pow((double)theta, (2.0 * j) / (double)head_dim));
        int a = 0;
        if (j % 3 == 1 && j < 3 * section[1]) a = 1;
        else if (j % 3 == 2 && j < 3 * section[2]) a = 2;
        p->axis[j] = (int8_t)a;
    }
}

cudaError_t launch_rmsnorm(const bf16 *x, const bf16 *w, bf16 *y, int rows, int cols, float eps, cudaStream_t st) {
    if (rows <= 0) return cudaSuccess;
    cudaLaunchAttribute at[1];
    cudaLaunchConfig_t cfg = pdl_config(dim3(rows), dim3(NORM_THREADS), 0, st, at);
    return cudaLaunchKernelEx(&cfg, rmsnorm_kernel, x, w, y, cols, eps);
}

cudaError_t launch_row_sumsq(const bf16 *x, int rows, int cols, float *ss, cudaStream_t st) {
    if (rows <= 0) return cudaSuccess;
    if (cols <= 0 || cols % 128) return cudaErrorInvalidValue;
    const long long n = (long long)rows * (cols / 128);
    cudaLaunchAttribute at[1];
    cudaLaunchConfig_t cfg = pdl_config(dim3((unsigned)((n + 255) / 256)), dim3(256), 0, st, at);
    return cudaLaunchKernelEx(&cfg, row_sumsq_kernel, x, rows, cols, ss);
}

cudaError_t launch_fold_cols(bf16 *W, int cols, const bf16 *gamma, int r0, int r1, int blk, int parity,
                             cudaStream_t st) {
    if (r1 <= r0) return cudaSuccess;
    if (cols <= 0 || cols % 8 || r0 < 0 || blk < 0) return cudaErrorInvalidValue;
    const long long n = (long long)(r1 - r0) * (cols / 8);
    cudaLaunchAttribute at[1];
    cudaLaunchConfig_t cfg = pdl_config(dim3((unsigned)((n + 255) / 256)), dim3(256), 0, st, at);
    return cudaLaunchKernelEx(&cfg, fold_cols_kernel, W, cols, gamma, r0, r1, blk, parity);
}

cudaError_t launch_rope_table(const int32_t *positions, int S, const RopeParams &rp, float *cos_t, float *sin_t,
                              cudaStream_t st, int stride) {
    if (S <= 0) return cudaSuccess;
    if (stride && (rp.half_dim % 4 || stride < S)) return cudaErrorInvalidValue;
    const int n = (stride ? stride : S) * rp.half_dim;
    cudaLaunchAttribute at[1];
    cudaLaunchConfig_t cfg = pdl_config(dim3((n + 255) / 256), dim3(256), 0, st, at);
    return cudaLaunchKernelEx(&cfg, rope_table_kernel, positions, S, rp, cos_t, sin_t, stride);
}

}  // namespace h3
