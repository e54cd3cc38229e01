// Memory-bound steps of the decoder layer: RMSNorm over the hidden size, the
// M-RoPE cos/sin tables, and the fused per-head q/k RMSNorm + rotary embedding.
//
// Page "vllm-omni vllm_omni/diffusion/models/minimax_h3/encoder.py":
// MiniMaxH3Qwen3VLRMSNorm (fp32 variance and scaling), the q_norm/k_norm calls
// of MiniMaxH3Qwen3VLTextAttention.forward, _rotate_half /
// _apply_rotary_pos_emb, and MiniMaxH3Qwen3VLTextRotaryEmbedding with
// _apply_interleaved_mrope.  All arithmetic is fp32; each kernel rounds its
// output to bf16 once (the pages' bf16 cast of cos/sin is not reproduced:
// the tables stay fp32).
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

// One thread per (token, frequency index j).
__global__ void rope_table_kernel(const int32_t *__restrict__ pos, int S, const RopeParams rp, float *cos_t,
                                  float *sin_t) {
    const int i = blockIdx.x * blockDim.x + threadIdx.x;
    if (i >= S * rp.half_dim) return;
    const int s = i / rp.half_dim;
    const int j = i - s * rp.half_dim;
    const float p = (float)pos[rp.axis[j] * S + s];
    const float ang = __fmul_rn(p, rp.inv_freq[j]);
    float sn, cs;
    sincosf(ang, &sn, &cs);
    cos_t[i] = cs;
    sin_t[i] = sn;
}

// One warp per (token, q-or-k head).  Lane l holds elements [l*E, l*E+E) of
// the head (E = D/32); lanes 0-15 hold the first half, lanes 16-31 the second,
// so the rotate-half partner of a lane's element sits in lane l ^ 16.
template <int D>
__global__ void __launch_bounds__(256) qk_norm_rope_kernel(bf16 *qkv, int S, int nq, int nkv, int ld,
                                                           const bf16 *__restrict__ wq,
                                                           const bf16 *__restrict__ wk, float eps,
                                                           const float *__restrict__ cos_t,
                                                           const float *__restrict__ sin_t) {
    constexpr int E = D / 32;
    constexpr int HALF = D / 2;
    const int lane = threadIdx.x & 31;
    const long long gw = (long long)blockIdx.x * 8 + (threadIdx.x >> 5);
    const int nh = nq + nkv;
    if (gw >= (long long)S * nh) return;
    const int s = (int)(gw / nh);
    const int h = (int)(gw - (long long)s * nh);
    bf16 *p = qkv + (size_t)s * ld + (size_t)h * D + lane * E;
    const bf16 *w = (h < nq ? wq : wk) + lane * E;
    float f[E], g[E];
    if constexpr (E == 4) {
        const uint2 v = *reinterpret_cast<const uint2 *>(p);
        const uint2 u = *reinterpret_cast<const uint2 *>(w);
        f[0] = bf16_lo(v.x); f[1] = bf16_hi(v.x); f[2] = bf16_lo(v.y); f[3] = bf16_hi(v.y);
        g[0] = bf16_lo(u.x); g[1] = bf16_hi(u.x); g[2] = bf16_lo(u.y); g[3] = bf16_hi(u.y);
    } else {
        const uint32_t v = *reinterpret_cast<const uint32_t *>(p);
        const uint32_t u = *reinterpret_cast<const uint32_t *>(w);
        f[0] = bf16_lo(v); f[1] = bf16_hi(v);
        g[0] = bf16_lo(u); g[1] = bf16_hi(u);
    }
    float ss = 0.f;
    #pragma unroll
    for (int e = 0; e < E; ++e) ss = fmaf(f[e], f[e], ss);
    ss = warp_sum(ss);
    const float rstd = 1.0f / sqrtf(ss / (float)D + eps);
    float y[E], o[E];
    #pragma unroll
    for (int e = 0; e < E; ++e) y[e] = f[e] * rstd * g[e];
    const bool first = lane < 16;
    const int j0 = (lane & 15) * E;  // frequency index of element 0 of this lane
    const float *cr = cos_t + (size_t)s * HALF + j0;
    const float *sr = sin_t + (size_t)s * HALF + j0;
    #pragma unroll
    for (int e = 0; e < E; ++e) {
        const float partner = __shfl_xor_sync(0xffffffffu, y[e], 16);
        const float c = cr[e], sn = sr[e];
        o[e] = first ? (y[e] * c - partner * sn) : (y[e] * c + partner * sn);
    }
    if constexpr (E == 4) {
        uint2 r;
        r.x = pack_bf16x2(o[0], o[1]);
        r.y = pack_bf16x2(o[2], o[3]);
        *reinterpret_cast<uint2 *>(p) = r;
    } else {
        *reinterpret_cast<uint32_t *>(p) = pack_bf16x2(o[0], o[1]);
    }
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
    rmsnorm_kernel<<<rows, NORM_THREADS, 0, st>>>(x, w, y, cols, eps);
    return cudaGetLastError();
}

cudaError_t launch_rope_table(const int32_t *positions, int S, const RopeParams &rp, float *cos_t, float *sin_t,
                              cudaStream_t st) {
    if (S <= 0) return cudaSuccess;
    const int n = S * rp.half_dim;
    rope_table_kernel<<<(n + 255) / 256, 256, 0, st>>>(positions, S, rp, cos_t, sin_t);
    return cudaGetLastError();
}

cudaError_t launch_qk_norm_rope(bf16 *qkv, int S, int nq, int nkv, int d, const bf16 *wq, const bf16 *wk,
                                float eps, const float *cos_t, const float *sin_t, cudaStream_t st) {
    if (S <= 0) return cudaSuccess;
    const long long warps = (long long)S * (nq + nkv);
    const unsigned grid = (unsigned)((warps + 7) / 8);
    const int ld = (nq + 2 * nkv) * d;
    if (d == 128)
        qk_norm_rope_kernel<128><<<grid, 256, 0, st>>>(qkv, S, nq, nkv, ld, wq, wk, eps, cos_t, sin_t);
    else if (d == 64)
        qk_norm_rope_kernel<64><<<grid, 256, 0, st>>>(qkv, S, nq, nkv, ld, wq, wk, eps, cos_t, sin_t);
    else
        return cudaErrorInvalidValue;
    return cudaGetLastError();
}

}  // namespace h3
