// Memory-bound steps of the vision tower: LayerNorm, the learned position
// embeddings sampled bilinearly at each patch, and the 2-D rotary tables.
//
// Page "vllm-omni vllm_omni/diffusion/models/minimax_h3/encoder.py", section
// "Qwen3-VL vision tower": nn.LayerNorm of the blocks and mergers,
// MiniMaxH3Qwen3VLVisionModel.fast_pos_embed_interpolate and rot_pos_emb with
// MiniMaxH3Qwen3VLVisionRotaryEmbedding.  Patches are kept in the tower's order:
// frames, then the m x m blocks in row-major block order, then the patches of a
// block row-major.
#include <cmath>

#include "common.cuh"
#include "kernels.h"

namespace h3 {

namespace {

constexpr int LN_VPT = 4;   // 4 x 8 values per thread: cols <= 32 * threads

template <int LN_THREADS>
__device__ __forceinline__ float ln_block_sum(float v, float *red) {
    #pragma unroll
    for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
    __syncthreads();   // red may still be read by the previous reduction
    if ((threadIdx.x & 31) == 0) red[threadIdx.x >> 5] = v;
    __syncthreads();
    float t = 0.f;
    #pragma unroll
    for (int i = 0; i < LN_THREADS / 32; ++i) t += red[i];
    return t;
}

// One CTA per row, the row held in registers: mean, then the mean of the squared deviations,
// then y = bf16((x - mean) / sqrt(var + eps) * w + b).  128 threads up to 4096 columns (more
// rows resident per SM), 256 above.
template <int LN_THREADS>
__global__ void __launch_bounds__(LN_THREADS) layernorm_kernel(const bf16 *__restrict__ x,
                                                               const bf16 *__restrict__ w,
                                                               const bf16 *__restrict__ b, bf16 *y, int cols,
                                                               float eps) {
    pdl_trigger();
    pdl_wait();
    __shared__ float red[LN_THREADS / 32];
    const int row = blockIdx.x;
    const int nvec = cols >> 3;
    const uint4 *xr = reinterpret_cast<const uint4 *>(x + (size_t)row * cols);
    float f[LN_VPT][8];
    float s = 0.f;
    #pragma unroll
    for (int i = 0; i < LN_VPT; ++i) {
        const int idx = threadIdx.x + i * LN_THREADS;
        if (idx < nvec) {
            const uint4 v = xr[idx];
            const uint32_t u[4] = {v.x, v.y, v.z, v.w};
            #pragma unroll
            for (int k = 0; k < 4; ++k) {
                f[i][2 * k] = bf16_lo(u[k]);
                f[i][2 * k + 1] = bf16_hi(u[k]);
            }
            #pragma unroll
            for (int k = 0; k < 8; ++k) s += f[i][k];
        }
    }
    const float mean = ln_block_sum<LN_THREADS>(s, red) / (float)cols;
    float q = 0.f;
    #pragma unroll
    for (int i = 0; i < LN_VPT; ++i) {
        const int idx = threadIdx.x + i * LN_THREADS;
        if (idx < nvec) {
            #pragma unroll
            for (int k = 0; k < 8; ++k) {
                f[i][k] -= mean;
                q = fmaf(f[i][k], f[i][k], q);
            }
        }
    }
    const float rstd = 1.0f / sqrtf(ln_block_sum<LN_THREADS>(q, red) / (float)cols + eps);
    const uint4 *wr = reinterpret_cast<const uint4 *>(w);
    const uint4 *br = reinterpret_cast<const uint4 *>(b);
    uint4 *yr = reinterpret_cast<uint4 *>(y + (size_t)row * cols);
    #pragma unroll
    for (int i = 0; i < LN_VPT; ++i) {
        const int idx = threadIdx.x + i * LN_THREADS;
        if (idx < nvec) {
            const uint4 gw = wr[idx], gb = br[idx];
            const uint32_t wv[4] = {gw.x, gw.y, gw.z, gw.w}, bv[4] = {gb.x, gb.y, gb.z, gb.w};
            uint32_t o[4];
            #pragma unroll
            for (int k = 0; k < 4; ++k)
                o[k] = pack_bf16x2(fmaf(f[i][2 * k] * rstd, bf16_lo(wv[k]), bf16_lo(bv[k])),
                                   fmaf(f[i][2 * k + 1] * rstd, bf16_hi(wv[k]), bf16_hi(bv[k])));
            yr[idx] = make_uint4(o[0], o[1], o[2], o[3]);
        }
    }
}

// One warp per row for rows of up to 2048 columns (the blocks' norms): VPT 16-byte vectors
// of x, w and b per lane, all loaded before the first reduction; mean and variance by warp
// shuffles alone.  Four rows per CTA, so a 3072 x 1024 activation is one wave of CTAs.
constexpr int LNW_ROWS = 4;
template <int VPT>
__global__ void __launch_bounds__(32 * LNW_ROWS) layernorm_warp_kernel(const bf16 *__restrict__ x,
                                                                       const bf16 *__restrict__ w,
                                                                       const bf16 *__restrict__ b, bf16 *y,
                                                                       int rows, int cols, float eps) {
    pdl_trigger();
    pdl_wait();
    const int lane = threadIdx.x & 31;
    const int row = blockIdx.x * LNW_ROWS + (threadIdx.x >> 5);
    if (row >= rows) return;   // whole warps leave; no block-wide barrier follows
    const int nvec = cols >> 3;
    const uint4 *xr = reinterpret_cast<const uint4 *>(x + (size_t)row * cols);
    const uint4 *wr = reinterpret_cast<const uint4 *>(w);
    const uint4 *br = reinterpret_cast<const uint4 *>(b);
    const uint4 zero = make_uint4(0u, 0u, 0u, 0u);
    uint4 xv[VPT], wv[VPT], bv[VPT];
    #pragma unroll
    for (int i = 0; i < VPT; ++i) {
        const int idx = lane + 32 * i;
        const bool ok = idx < nvec;
        xv[i] = ok ? xr[idx] : zero;
        wv[i] = ok ? wr[idx] : zero;
        bv[i] = ok ? br[idx] : zero;
    }
    float s = 0.f;
    #pragma unroll
    for (int i = 0; i < VPT; ++i) {
        const uint32_t u[4] = {xv[i].x, xv[i].y, xv[i].z, xv[i].w};
        #pragma unroll
        for (int k = 0; k < 4; ++k) s += bf16_lo(u[k]) + bf16_hi(u[k]);
    }
    #pragma unroll
    for (int o = 16; o > 0; o >>= 1) s += __shfl_xor_sync(0xffffffffu, s, o);
    const float mean = s / (float)cols;
    float q = 0.f;
    #pragma unroll
    for (int i = 0; i < VPT; ++i) {
        if (lane + 32 * i < nvec) {
            const uint32_t u[4] = {xv[i].x, xv[i].y, xv[i].z, xv[i].w};
            #pragma unroll
            for (int k = 0; k < 4; ++k) {
                const float d0 = bf16_lo(u[k]) - mean, d1 = bf16_hi(u[k]) - mean;
                q = fmaf(d0, d0, q);
                q = fmaf(d1, d1, q);
            }
        }
    }
    #pragma unroll
    for (int o = 16; o > 0; o >>= 1) q += __shfl_xor_sync(0xffffffffu, q, o);
    const float rstd = 1.0f / sqrtf(q / (float)cols + eps);
    uint4 *yr = reinterpret_cast<uint4 *>(y + (size_t)row * cols);
    #pragma unroll
    for (int i = 0; i < VPT; ++i) {
        const int idx = lane + 32 * i;
        if (idx < nvec) {
            const uint32_t u[4] = {xv[i].x, xv[i].y, xv[i].z, xv[i].w};
            const uint32_t wu[4] = {wv[i].x, wv[i].y, wv[i].z, wv[i].w};
            const uint32_t bu[4] = {bv[i].x, bv[i].y, bv[i].z, bv[i].w};
            uint32_t o[4];
            #pragma unroll
            for (int k = 0; k < 4; ++k)
                o[k] = pack_bf16x2(fmaf((bf16_lo(u[k]) - mean) * rstd, bf16_lo(wu[k]), bf16_lo(bu[k])),
                                   fmaf((bf16_hi(u[k]) - mean) * rstd, bf16_hi(wu[k]), bf16_hi(bu[k])));
            yr[idx] = make_uint4(o[0], o[1], o[2], o[3]);
        }
    }
}

// The (row, column) of patch k of the concatenated grids, in the tower's order.
__device__ __forceinline__ void patch_rc(const VisionGrids &gr, int k, int &grid, int &row, int &col) {
    grid = 0;
    while (grid + 1 < gr.n && k >= gr.first[grid + 1]) ++grid;
    const int h = gr.h[grid], w = gr.w[grid], m = gr.merge;
    const int idx = (k - gr.first[grid]) % (h * w);   // inside its frame
    const int blk = idx / (m * m), in = idx % (m * m);
    row = (blk / (w / m)) * m + in / m;
    col = (blk % (w / m)) * m + in % m;
}

// One coordinate of the evenly spaced samples: i * ((G - 1) / (n - 1)) in double, the last one
// exactly G - 1, rounded once to fp32 (the values numpy's linspace gives in float32).
__device__ __forceinline__ float grid_coord(int i, int n, int G) {
    if (n <= 1) return 0.f;
    if (i == n - 1) return (float)(G - 1);
    const double step = (double)(G - 1) / (double)(n - 1);
    return (float)((double)i * step);
}

// One CTA per patch, 8 columns per thread: bilinear sample of the G x G table at the patch's
// coordinates (fp32 weights and products, summed corner by corner in fixed order), bf16.
__global__ void pos_embed_kernel(const bf16 *__restrict__ table, int G, int D, const VisionGrids gr, bf16 *out) {
    pdl_trigger();
    pdl_wait();
    const int k = blockIdx.x;
    int grid, row, col;
    patch_rc(gr, k, grid, row, col);
    const float hs = grid_coord(row, gr.h[grid], G), ws = grid_coord(col, gr.w[grid], G);
    const int h0 = (int)hs, w0 = (int)ws;
    const int h1 = min(h0 + 1, G - 1), w1 = min(w0 + 1, G - 1);
    const float dh = __fsub_rn(hs, (float)h0), dw = __fsub_rn(ws, (float)w0);
    const float c00 = __fmul_rn(__fsub_rn(1.f, dh), __fsub_rn(1.f, dw));
    const float c01 = __fmul_rn(__fsub_rn(1.f, dh), dw);
    const float c10 = __fmul_rn(dh, __fsub_rn(1.f, dw));
    const float c11 = __fmul_rn(dh, dw);
    const uint4 *t00 = reinterpret_cast<const uint4 *>(table + (size_t)(h0 * G + w0) * D);
    const uint4 *t01 = reinterpret_cast<const uint4 *>(table + (size_t)(h0 * G + w1) * D);
    const uint4 *t10 = reinterpret_cast<const uint4 *>(table + (size_t)(h1 * G + w0) * D);
    const uint4 *t11 = reinterpret_cast<const uint4 *>(table + (size_t)(h1 * G + w1) * D);
    uint4 *o = reinterpret_cast<uint4 *>(out + (size_t)k * D);
    for (int v = threadIdx.x; v < (D >> 3); v += blockDim.x) {
        const uint4 a = t00[v], b = t01[v], c = t10[v], d = t11[v];
        const uint32_t ua[4] = {a.x, a.y, a.z, a.w}, ub[4] = {b.x, b.y, b.z, b.w};
        const uint32_t uc[4] = {c.x, c.y, c.z, c.w}, ud[4] = {d.x, d.y, d.z, d.w};
        uint32_t r[4];
        #pragma unroll
        for (int q = 0; q < 4; ++q) {
            float e[2];
            #pragma unroll
            for (int s = 0; s < 2; ++s) {
                const float va = s ? bf16_hi(ua[q]) : bf16_lo(ua[q]), vb = s ? bf16_hi(ub[q]) : bf16_lo(ub[q]);
                const float vc = s ? bf16_hi(uc[q]) : bf16_lo(uc[q]), vd = s ? bf16_hi(ud[q]) : bf16_lo(ud[q]);
                float acc = __fmul_rn(va, c00);
                acc = __fadd_rn(acc, __fmul_rn(vb, c01));
                acc = __fadd_rn(acc, __fmul_rn(vc, c10));
                e[s] = __fadd_rn(acc, __fmul_rn(vd, c11));
            }
            r[q] = pack_bf16x2(e[0], e[1]);
        }
        o[v] = make_uint4(r[0], r[1], r[2], r[3]);
    }
}

// One thread per (patch, angle j < d/2): j < d/4 rotates by row * inv_freq[j], the rest by
// column * inv_freq[j - d/4] (fp32 products); fp32 cos / sin, element i in either layout:
// row-major [n][d/2] (stride 0), or row-interleaved [d/8][stride][4], i = ((j/4) stride + k) 4 + j%4.
__global__ void vision_rope_kernel(const VisionGrids gr, int n, int half_dim, const VisionRope rp, float *cos_t,
                                   float *sin_t, int stride) {
    pdl_trigger();
    pdl_wait();
    const int i = blockIdx.x * blockDim.x + threadIdx.x;
    if (i >= (stride ? stride : n) * half_dim) return;
    int k, j;
    if (stride) {
        const int grp = i / (4 * stride), rem = i - grp * 4 * stride;
        k = rem >> 2;
        j = 4 * grp + (rem & 3);
        if (k >= n) return;
    } else {
        k = i / half_dim;
        j = i - k * half_dim;
    }
    int grid, row, col;
    patch_rc(gr, k, grid, row, col);
    const int quarter = half_dim >> 1;
    const float ang = j < quarter ? __fmul_rn((float)row, rp.inv_freq[j]) : __fmul_rn((float)col, rp.inv_freq[j - quarter]);
    float sn, cs;
    sincosf(ang, &sn, &cs);
    cos_t[i] = cs;
    sin_t[i] = sn;
}

}  // namespace

bool make_vision_grids(VisionGrids *g, const int32_t *thw, int n_grids, int merge, int *n_patches) {
    if (n_grids < 1 || n_grids > kMaxVisionGrids || merge < 1) return false;
    g->n = n_grids;
    g->merge = merge;
    int total = 0;
    for (int i = 0; i < n_grids; ++i) {
        const int t = thw[3 * i], h = thw[3 * i + 1], w = thw[3 * i + 2];
        if (t < 1 || h < 1 || w < 1 || h % merge || w % merge) return false;
        g->first[i] = total;
        g->h[i] = h;
        g->w[i] = w;
        total += t * h * w;
    }
    *n_patches = total;
    return true;
}

void make_vision_rope(VisionRope *r, int head_dim, float theta) {
    const int dim = head_dim / 2;   // the rotary embedding's width
    for (int j = 0; j < kMaxHalfDim; ++j) r->inv_freq[j] = 0.f;
    for (int j = 0; j < dim / 2; ++j)   // theta^(-2j/dim) in double, rounded once to fp32
        r->inv_freq[j] = (float)(1.0 / std::pow((double)theta, (2.0 * j) / (double)dim));
}

cudaError_t launch_layernorm(const bf16 *x, const bf16 *w, const bf16 *b, bf16 *y, int rows, int cols, float eps,
                             cudaStream_t st) {
    if (rows <= 0) return cudaSuccess;
    if (cols % 8 || cols > 256 * LN_VPT * 8) return cudaErrorInvalidValue;
    cudaLaunchAttribute at[1];
    if (cols <= 32 * 8 * 8) {   // a warp per row
        const int vpt = (cols / 8 + 31) / 32;
        cudaLaunchConfig_t cfg = pdl_config(dim3((rows + LNW_ROWS - 1) / LNW_ROWS), dim3(32 * LNW_ROWS), 0, st, at);
        if (vpt <= 1) return cudaLaunchKernelEx(&cfg, layernorm_warp_kernel<1>, x, w, b, y, rows, cols, eps);
        if (vpt <= 2) return cudaLaunchKernelEx(&cfg, layernorm_warp_kernel<2>, x, w, b, y, rows, cols, eps);
        if (vpt <= 4) return cudaLaunchKernelEx(&cfg, layernorm_warp_kernel<4>, x, w, b, y, rows, cols, eps);
        return cudaLaunchKernelEx(&cfg, layernorm_warp_kernel<8>, x, w, b, y, rows, cols, eps);
    }
    if (cols <= 128 * LN_VPT * 8) {
        cudaLaunchConfig_t cfg = pdl_config(dim3(rows), dim3(128), 0, st, at);
        return cudaLaunchKernelEx(&cfg, layernorm_kernel<128>, x, w, b, y, cols, eps);
    }
    cudaLaunchConfig_t cfg = pdl_config(dim3(rows), dim3(256), 0, st, at);
    return cudaLaunchKernelEx(&cfg, layernorm_kernel<256>, x, w, b, y, cols, eps);
}

cudaError_t launch_pos_embed(const bf16 *table, int G, int D, const VisionGrids &gr, int n, bf16 *out,
                             cudaStream_t st) {
    if (n <= 0) return cudaSuccess;
    if (D % 8 || G < 1) return cudaErrorInvalidValue;
    cudaLaunchAttribute at[1];
    const int threads = D / 8 < 128 ? ((D / 8 + 31) / 32) * 32 : 128;
    cudaLaunchConfig_t cfg = pdl_config(dim3(n), dim3(threads), 0, st, at);
    return cudaLaunchKernelEx(&cfg, pos_embed_kernel, table, G, D, gr, out);
}

cudaError_t launch_vision_rope(const VisionGrids &gr, int n, int head_dim, const VisionRope &rp, float *cos_t,
                               float *sin_t, cudaStream_t st, int stride) {
    if (n <= 0) return cudaSuccess;
    if (head_dim % 4 || head_dim / 2 > kMaxHalfDim || (stride && (head_dim % 8 || stride < n)))
        return cudaErrorInvalidValue;
    const int total = (stride ? stride : n) * (head_dim / 2);
    cudaLaunchAttribute at[1];
    cudaLaunchConfig_t cfg = pdl_config(dim3((total + 255) / 256), dim3(256), 0, st, at);
    return cudaLaunchKernelEx(&cfg, vision_rope_kernel, gr, n, head_dim / 2, rp, cos_t, sin_t, stride);
}

}  // namespace h3
