// Causal GQA attention over packed sequences (flash-attention tiling).
//
// Page "vllm-omni vllm_omni/diffusion/models/minimax_h3/encoder.py",
// MiniMaxH3Qwen3VLTextAttention.forward: K/V of kv head h / (nq/nkv) serve q
// head h (repeat_interleave), scaled_dot_product_attention with is_causal=True
// and the default scale 1/sqrt(d).  Packed sequences (cu_seqlens) attend only
// within themselves.  K/V are never expanded: the CTAs of the nq/nkv heads of
// one group run next to each other and share the K/V tiles through L2.
//
// CTA = 128 query rows of one head, 8 warps x 16 rows; keys stream in tiles of
// 64 through a 2-stage cp.async ring; S = Q K^T and O += P V on the warp-level
// bf16 MMA with fp32 accumulation; online softmax in fp32 with exp2.
#include <cmath>

#include "common.cuh"
#include "kernels.h"

namespace h3 {

namespace {

constexpr int QM = 128;
constexpr int KN = 64;
constexpr int ATT_THREADS = 256;

struct AttnArgs {
    const bf16 *qkv;
    bf16 *o;
    int ld_qkv, ld_o;
    int nq, nkv, group;
    int k_col0, v_col0;
    float scale_log2;
    int n_seqs, total_tiles;
    int cu[kMaxSeqs + 1];
    int tile_start[kMaxSeqs + 1];
};

// byte offset of 16-byte chunk c of row r in a [rows][D] bf16 tile (XOR swizzle)
template <int D>
__device__ __forceinline__ uint32_t swz(int r, int c) {
    return (uint32_t)(r * D * 2 + ((c ^ (r & 7)) << 4));
}

template <int D>
__device__ __forceinline__ void load_tile(uint32_t s_base, const bf16 *g_base, int ld, int rows, int valid_rows,
                                          int tid) {
    constexpr int CH = D / 8;
    for (int idx = tid; idx < rows * CH; idx += ATT_THREADS) {
        const int r = idx / CH, c = idx - r * CH;
        const bool ok = r < valid_rows;
        const bf16 *src = g_base + (size_t)(ok ? r : 0) * ld + c * 8;
        cp_async16(s_base + swz<D>(r, c), src, ok ? 16u : 0u);
    }
}

template <int D>
__global__ void __launch_bounds__(ATT_THREADS, 1) attention_kernel(const __grid_constant__ AttnArgs a) {
    extern __shared__ __align__(128) uint8_t smem[];
    const uint32_t sQ = smem_u32(smem);
    const uint32_t sK = sQ + QM * D * 2;
    const uint32_t sV = sK + 2 * KN * D * 2;
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;

    // work item: heads fastest (the heads of one kv group are adjacent), heavy tiles first
    const int head = blockIdx.x % a.nq;
    const int tile_lin = a.total_tiles - 1 - (int)(blockIdx.x / a.nq);
    int seg = 0;
    {
        int lo = 0, hi = a.n_seqs - 1;  // last segment with tile_start <= tile_lin
        while (lo < hi) {
            const int mid = (lo + hi + 1) >> 1;
            if (a.tile_start[mid] <= tile_lin) lo = mid; else hi = mid - 1;
        }
        seg = lo;
    }
    const int seg0 = a.cu[seg];
    const int L = a.cu[seg + 1] - seg0;
    const int q0 = (tile_lin - a.tile_start[seg]) * QM;
    const int kvh = head / a.group;
    const bf16 *gQ = a.qkv + (size_t)(seg0 + q0) * a.ld_qkv + (size_t)head * D;
    const bf16 *gK = a.qkv + (size_t)seg0 * a.ld_qkv + a.k_col0 + (size_t)kvh * D;
    const bf16 *gV = a.qkv + (size_t)seg0 * a.ld_qkv + a.v_col0 + (size_t)kvh * D;

    const int q_valid = min(QM, L - q0);
    const int kend = min(q0 + QM, L);
    const int n_kt = (kend + KN - 1) / KN;

    load_tile<D>(sQ, gQ, a.ld_qkv, QM, q_valid, tid);
    load_tile<D>(sK, gK, a.ld_qkv, KN, min(KN, L), tid);
    load_tile<D>(sV, gV, a.ld_qkv, KN, min(KN, L), tid);
    cp_async_commit();

    constexpr int KS = D / 16;   // k-steps over head_dim
    constexpr int NT = D / 8;    // n-tiles of the output
    uint32_t qa[KS][4];
    float o[NT][4];
    #pragma unroll
    for (int j = 0; j < NT; ++j) o[j][0] = o[j][1] = o[j][2] = o[j][3] = 0.f;
    float m_r[2] = {-INFINITY, -INFINITY};
    float l_r[2] = {0.f, 0.f};
    const int g = lane >> 2, t = lane & 3;
    const int row_a = q0 + warp * 16 + g;   // segment-local rows held by this thread
    const int row_b = row_a + 8;

    for (int kt = 0; kt < n_kt; ++kt) {
        const int buf = kt & 1;
        if (kt + 1 < n_kt) {
            const int nb = buf ^ 1;
            const int k1 = (kt + 1) * KN;
            load_tile<D>(sK + nb * KN * D * 2, gK + (size_t)k1 * a.ld_qkv, a.ld_qkv, KN, min(KN, L - k1), tid);
            load_tile<D>(sV + nb * KN * D * 2, gV + (size_t)k1 * a.ld_qkv, a.ld_qkv, KN, min(KN, L - k1), tid);
            cp_async_commit();
            cp_async_wait<1>();
        } else {
            cp_async_wait<0>();
        }
        __syncthreads();
        if (kt == 0) {
            #pragma unroll
            for (int kk = 0; kk < KS; ++kk) {
                const int mat = lane >> 3;
                const int r = warp * 16 + (mat & 1) * 8 + (lane & 7);
                ldmatrix_x4(sQ + swz<D>(r, 2 * kk + (mat >> 1)), qa[kk][0], qa[kk][1], qa[kk][2], qa[kk][3]);
            }
        }
        const uint32_t kb = sK + buf * KN * D * 2;
        const uint32_t vb = sV + buf * KN * D * 2;

        // S = Q K^T  (16 x 64 per warp)
        float s[8][4];
        #pragma unroll
        for (int j = 0; j < 8; ++j) s[j][0] = s[j][1] = s[j][2] = s[j][3] = 0.f;
        #pragma unroll
        for (int kk = 0; kk < KS; ++kk) {
            #pragma unroll
            for (int np = 0; np < 4; ++np) {
                const int mat = lane >> 3;
                const int key = np * 16 + (mat >> 1) * 8 + (lane & 7);
                uint32_t b0, b1, b2, b3;
                ldmatrix_x4(kb + swz<D>(key, 2 * kk + (mat & 1)), b0, b1, b2, b3);
                mma_bf16_16816(s[2 * np], qa[kk][0], qa[kk][1], qa[kk][2], qa[kk][3], b0, b1);
                mma_bf16_16816(s[2 * np + 1], qa[kk][0], qa[kk][1], qa[kk][2], qa[kk][3], b2, b3);
            }
        }

        // scale, causal mask, online softmax
        const int key0 = kt * KN;
        const bool need_mask = key0 + KN - 1 > q0 + warp * 16;
        float mx[2] = {m_r[0], m_r[1]};
        #pragma unroll
        for (int j = 0; j < 8; ++j) {
            #pragma unroll
            for (int e = 0; e < 4; ++e) {
                float v = s[j][e] * a.scale_log2;
                if (need_mask) {
                    const int key = key0 + j * 8 + 2 * t + (e & 1);
                    const int row = (e < 2) ? row_a : row_b;
                    if (key > row) v = -INFINITY;
                }
                s[j][e] = v;
                mx[e >> 1] = fmaxf(mx[e >> 1], v);
            }
        }
        #pragma unroll
        for (int r = 0; r < 2; ++r) {
            mx[r] = fmaxf(mx[r], __shfl_xor_sync(0xffffffffu, mx[r], 1));
            mx[r] = fmaxf(mx[r], __shfl_xor_sync(0xffffffffu, mx[r], 2));
        }
        float corr[2], rs[2] = {0.f, 0.f};
        #pragma unroll
        for (int r = 0; r < 2; ++r) {
            corr[r] = (m_r[r] == -INFINITY) ? 0.f : exp2f(m_r[r] - mx[r]);
            m_r[r] = mx[r];
        }
        #pragma unroll
        for (int j = 0; j < 8; ++j) {
            #pragma unroll
            for (int e = 0; e < 4; ++e) {
                const float mr = m_r[e >> 1];
                const float p = (mr == -INFINITY) ? 0.f : exp2f(s[j][e] - mr);
                s[j][e] = p;
                rs[e >> 1] += p;
            }
        }
        #pragma unroll
        for (int r = 0; r < 2; ++r) l_r[r] = l_r[r] * corr[r] + rs[r];
        #pragma unroll
        for (int j = 0; j < NT; ++j) {
            o[j][0] *= corr[0]; o[j][1] *= corr[0];
            o[j][2] *= corr[1]; o[j][3] *= corr[1];
        }

        // O += P V
        #pragma unroll
        for (int kk = 0; kk < 4; ++kk) {
            const uint32_t a0 = pack_bf16x2(s[2 * kk][0], s[2 * kk][1]);
            const uint32_t a1 = pack_bf16x2(s[2 * kk][2], s[2 * kk][3]);
            const uint32_t a2 = pack_bf16x2(s[2 * kk + 1][0], s[2 * kk + 1][1]);
            const uint32_t a3 = pack_bf16x2(s[2 * kk + 1][2], s[2 * kk + 1][3]);
            #pragma unroll
            for (int dp = 0; dp < NT / 2; ++dp) {
                const int mat = lane >> 3;
                const int key = kk * 16 + (mat & 1) * 8 + (lane & 7);
                uint32_t b0, b1, b2, b3;
                ldmatrix_x4_trans(vb + swz<D>(key, 2 * dp + (mat >> 1)), b0, b1, b2, b3);
                mma_bf16_16816(o[2 * dp], a0, a1, a2, a3, b0, b1);
                mma_bf16_16816(o[2 * dp + 1], a0, a1, a2, a3, b2, b3);
            }
        }
        __syncthreads();
    }

    // normalise, stage the warp's 16 rows in the Q tile, write 16-byte chunks
    #pragma unroll
    for (int r = 0; r < 2; ++r) {
        l_r[r] += __shfl_xor_sync(0xffffffffu, l_r[r], 1);
        l_r[r] += __shfl_xor_sync(0xffffffffu, l_r[r], 2);
    }
    const float inv0 = l_r[0] > 0.f ? 1.f / l_r[0] : 0.f;
    const float inv1 = l_r[1] > 0.f ? 1.f / l_r[1] : 0.f;
    const int ra = warp * 16 + g, rb = ra + 8;
    #pragma unroll
    for (int j = 0; j < NT; ++j) {
        const uint32_t va = pack_bf16x2(o[j][0] * inv0, o[j][1] * inv0);
        const uint32_t vb2 = pack_bf16x2(o[j][2] * inv1, o[j][3] * inv1);
        asm volatile("st.shared.b32 [%0], %1;" ::"r"(sQ + swz<D>(ra, j) + 4 * t), "r"(va) : "memory");
        asm volatile("st.shared.b32 [%0], %1;" ::"r"(sQ + swz<D>(rb, j) + 4 * t), "r"(vb2) : "memory");
    }
    __syncwarp();
    constexpr int CH = D / 8;
    bf16 *gO = a.o + (size_t)(seg0 + q0) * a.ld_o + (size_t)head * D;
    for (int idx = lane; idx < 16 * CH; idx += 32) {
        const int r = warp * 16 + idx / CH, c = idx % CH;
        if (r < q_valid) {
            uint4 v;
            asm volatile("ld.shared.v4.b32 {%0,%1,%2,%3}, [%4];"
                         : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
                         : "r"(sQ + swz<D>(r, c)));
            *reinterpret_cast<uint4 *>(gO + (size_t)r * a.ld_o + c * 8) = v;
        }
    }
}

template <int D>
cudaError_t launch_d(const AttnArgs &args, int grid, cudaStream_t st) {
    constexpr int smem = (QM + 4 * KN) * D * 2;
    static bool attr = false;
    if (!attr) {
        cudaError_t e = cudaFuncSetAttribute(attention_kernel<D>, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
        if (e != cudaSuccess) return e;
        attr = true;
    }
    attention_kernel<D><<<grid, ATT_THREADS, smem, st>>>(args);
    return cudaGetLastError();
}

}  // namespace

cudaError_t launch_attention(const bf16 *qkv, bf16 *o, int S, int nq, int nkv, int d, const int32_t *cu_host,
                             int n_seqs, cudaStream_t st) {
    if (S <= 0) return cudaSuccess;
    static AttnArgs args;  // large; built on the host for every launch
    args.qkv = qkv;
    args.o = o;
    args.ld_qkv = (nq + 2 * nkv) * d;
    args.ld_o = nq * d;
    args.nq = nq;
    args.nkv = nkv;
    args.group = nq / nkv;
    args.k_col0 = nq * d;
    args.v_col0 = (nq + nkv) * d;
    args.scale_log2 = (float)(1.4426950408889634 / std::sqrt((double)d));
    int n = 0, tiles = 0;
    if (!cu_host) {
        args.cu[0] = 0;
        args.cu[1] = S;
        args.tile_start[0] = 0;
        tiles = (S + QM - 1) / QM;
        n = 1;
    } else {
        // drop empty sequences so every tile has at least one query row
        args.cu[0] = 0;
        for (int i = 0; i < n_seqs; ++i) {
            const int len = cu_host[i + 1] - cu_host[i];
            if (len <= 0) continue;
            args.cu[n] = cu_host[i];
            args.tile_start[n] = tiles;
            tiles += (len + QM - 1) / QM;
            ++n;
            args.cu[n] = cu_host[i + 1];
        }
    }
    if (n == 0) return cudaSuccess;
    args.n_seqs = n;
    args.total_tiles = tiles;
    const int grid = tiles * nq;
    if (d == 128) return launch_d<128>(args, grid, st);
    if (d == 64) return launch_d<64>(args, grid, st);
    return cudaErrorInvalidValue;
}

}  // namespace h3
