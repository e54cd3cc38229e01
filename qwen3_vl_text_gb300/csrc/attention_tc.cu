// Causal GQA attention over packed sequences on the tcgen05 tensor cores.
//
// Page "vllm-omni vllm_omni/diffusion/models/minimax_h3/encoder.py",
// MiniMaxH3Qwen3VLTextAttention.forward: q head h reads kv head h / (nq/nkv)
// (repeat_interleave), scaled_dot_product_attention(is_causal=True) with scale
// 1/sqrt(d), output columns head-major.  Packed sequences (cu_seqlens) attend
// only within themselves.
//
// One CTA = 128 query rows of one head; keys/values stream in tiles of 128.
//   warp 0     TMA: Q once, K and V tiles into a 2-stage ring (128-byte swizzle)
//   warp 1     TMEM allocation; tcgen05.mma from one thread:
//                S_j = Q K_j^T   (M=128, N=128, K=d)   into one of two TMEM S buffers
//                O  += P_j V_j   (M=128, N=d,   K=128) into the TMEM O buffer; V is read
//                                  as an MN-major operand straight from its TMA tile
//   warps 2+   NWG softmax warpgroups (4 for d = 128, 2 for d = 64); thread = one
//              query row (its TMEM lane) x one NWG-th of the key columns: causal
//              mask, online softmax in fp32 with exp2 and a lazily raised running
//              max (row max combined across the warpgroups through shared memory
//              once per tile; O rescaled in TMEM, each warpgroup its own columns,
//              only when the max grows by more than 2^8), P as bf16 into swizzled
//              shared memory; at the end the row sums are combined and O / l ->
//              bf16 -> global
// S_{j+1} is computed while the softmax warps work on S_j.  Every wait is bounded.
#include <cmath>

#include "common.cuh"
#include "kernels.h"

namespace h3 {

namespace {

constexpr int TQ = 128;
constexpr int TK = 128;
template <int D>
constexpr int kNWG = D == 128 ? 4 : 2;          // softmax warpgroups
template <int D>
constexpr int kThreads = 64 + 128 * kNWG<D>;
constexpr float kRescaleThreshold = 8.0f;  // log2 units

struct AttnTcArgs {
    bf16 *o;
    int ld_o;
    int nq, group;
    int k_col0, v_col0;
    float scale_log2;
    int n_seqs, total_tiles;
    int32_t *status;
    int cu[kMaxSeqs + 1];
    int tile_start[kMaxSeqs + 1];
};

template <int D>
struct TcLayout {
    static constexpr int ATOM = TQ * 128;          // one 64-column atom column of a 128-row tile: 16 KB
    static constexpr int Q_BYTES = TQ * D * 2;
    static constexpr int KV_BYTES = TK * D * 2;
    static constexpr int P_BYTES = TQ * TK * 2;
    static constexpr int OFF_Q = 0;
    static constexpr int OFF_K = OFF_Q + Q_BYTES;
    static constexpr int OFF_V = OFF_K + 2 * KV_BYTES;
    static constexpr int OFF_P = OFF_V + 2 * KV_BYTES;
    static constexpr int OFF_RED = OFF_P + P_BYTES;                       // [2][NWG][128] maxima, [NWG][128] sums
    static constexpr int RED_BYTES = 3 * kNWG<D> * TQ * 4;
    static constexpr int OFF_BAR = OFF_RED + RED_BYTES;
    static constexpr int SMEM = 1024 + OFF_BAR + 256;
};

// Barrier over the softmax warps (named barrier 1) returning the AND of v.
template <int NT>
__device__ __forceinline__ bool softmax_bar_and(bool v) {
    uint32_t r;
    asm volatile(
        "{\n\t.reg .pred p, q;\n\t"
        "setp.ne.u32 p, %1, 0;\n\t"
        "bar.red.and.pred q, 1, %2, p;\n\t"
        "selp.u32 %0, 1, 0, q;\n\t}"
        : "=r"(r)
        : "r"((uint32_t)v), "n"(NT)
        : "memory");
    return r != 0;
}

template <int D>
__global__ void __launch_bounds__(kThreads<D>, 1)
    attention_tc_kernel(const __grid_constant__ CUtensorMap tm, const __grid_constant__ AttnTcArgs a) {
    using Lay = TcLayout<D>;
    extern __shared__ uint8_t smem_raw[];
    uint8_t *smem = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    uint8_t *sQ = smem + Lay::OFF_Q;
    uint8_t *sK = smem + Lay::OFF_K;
    uint8_t *sV = smem + Lay::OFF_V;
    uint8_t *sP = smem + Lay::OFF_P;
    uint64_t *bars = reinterpret_cast<uint64_t *>(smem + Lay::OFF_BAR);
    uint64_t *q_full = bars + 0;
    uint64_t *k_full = bars + 1;     // [2]
    uint64_t *v_full = bars + 3;     // [2]
    uint64_t *kv_empty = bars + 5;   // [2]
    uint64_t *s_full = bars + 7;     // [2]
    uint64_t *p_full = bars + 9;
    uint64_t *pv_done = bars + 10;
    uint64_t *drain = bars + 11;
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(bars + 12);
    volatile int *abort_flag = reinterpret_cast<volatile int *>(tmem_slot + 1);

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    pdl_trigger();

    // work item: heads fastest (the heads of one kv group are adjacent), heavy q tiles first
    const int head = blockIdx.x % a.nq;
    const int tile_lin = a.total_tiles - 1 - (int)(blockIdx.x / a.nq);
    int seg = 0;
    {
        int lo = 0, hi = a.n_seqs - 1;
        while (lo < hi) {
            const int mid = (lo + hi + 1) >> 1;
            if (a.tile_start[mid] <= tile_lin) lo = mid; else hi = mid - 1;
        }
        seg = lo;
    }
    const int seg0 = a.cu[seg];
    const int L = a.cu[seg + 1] - seg0;
    const int q0 = (tile_lin - a.tile_start[seg]) * TQ;
    const int kvh = head / a.group;
    const int kend = min(q0 + TQ, L);
    const int n_kt = (kend + TK - 1) / TK;

    if (threadIdx.x == 0) {
        for (int i = 0; i < 12; ++i) mbar_init(bars + i, (bars + i == p_full) ? 4 * kNWG<D> : 1);
        *abort_flag = 0;
        fence_barrier_init();
    }
    if (warp == 0 && lane == 0) prefetch_tmap(&tm);
    if (warp == 1) {
        tmem_alloc(tmem_slot, 512);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    pdl_wait();       // q/k/v are the previous kernel's output; o is read by the previous layer's o_proj
    const uint32_t tmem_base = *tmem_slot;
    const uint32_t tS = tmem_base;          // S buffers at columns 0 and 128
    const uint32_t tO = tmem_base + 256;    // O at columns 256 .. 256+D

    if (warp == 0) {
        if (lane == 0) {
            bool ok = true;
            uint32_t issued[2] = {0, 0};
            mbar_arrive_expect_tx(q_full, Lay::Q_BYTES);
            for (int c = 0; c < D / 64; ++c)
                tma_load_2d(sQ + c * Lay::ATOM, &tm, q_full, head * D + c * 64, seg0 + q0);
            for (int j = 0; j < n_kt && ok; ++j) {
                const int s = j & 1;
                if (j >= 2 && !mbar_wait(&kv_empty[s], ((j >> 1) - 1) & 1, abort_flag)) { ok = false; break; }
                const int y = seg0 + j * TK;
                mbar_arrive_expect_tx(&k_full[s], Lay::KV_BYTES);
                for (int c = 0; c < D / 64; ++c)
                    tma_load_2d(sK + s * Lay::KV_BYTES + c * Lay::ATOM, &tm, &k_full[s], a.k_col0 + kvh * D + c * 64, y);
                mbar_arrive_expect_tx(&v_full[s], Lay::KV_BYTES);
                for (int c = 0; c < D / 64; ++c)
                    tma_load_2d(sV + s * Lay::KV_BYTES + c * Lay::ATOM, &tm, &v_full[s], a.v_col0 + kvh * D + c * 64, y);
                ++issued[s];
            }
            if (!ok) {
                report(a.status, ST_TIMEOUT);
                *abort_flag = 1;
                const int never = 0;
                mbar_wait(q_full, 0, &never);
                for (int s = 0; s < 2; ++s)
                    if (issued[s]) {
                        mbar_wait(&k_full[s], (issued[s] - 1) & 1, &never);
                        mbar_wait(&v_full[s], (issued[s] - 1) & 1, &never);
                    }
            }
        }
    } else if (warp == 1) {
        if (lane == 0) {
            constexpr uint32_t idesc_s = umma_idesc_bf16(TQ, TK);
            constexpr uint32_t idesc_o = umma_idesc_bf16(TQ, D) | (1u << 16);   // B (V) is MN-major
            bool ok = mbar_wait(q_full, 0, abort_flag);
            auto issue_s = [&](int j) {
                const int s = j & 1;
                if (!mbar_wait(&k_full[s], (j >> 1) & 1, abort_flag)) return false;
                tc_fence_after();
                const uint32_t qa = smem_u32(sQ), kb = smem_u32(sK + s * Lay::KV_BYTES);
                #pragma unroll
                for (int kk = 0; kk < D / 16; ++kk) {
                    const uint32_t off = (kk >> 2) * Lay::ATOM + (kk & 3) * 32;
                    umma_bf16(tS + s * TK, sdesc_sw128(qa + off), sdesc_sw128(kb + off), idesc_s, kk > 0);
                }
                umma_commit(&s_full[s]);
                return true;
            };
            if (ok) ok = issue_s(0);
            for (int j = 0; j < n_kt && ok; ++j) {
                if (j + 1 < n_kt && !issue_s(j + 1)) { ok = false; break; }
                if (!mbar_wait(p_full, j & 1, abort_flag)) { ok = false; break; }
                const int s = j & 1;
                if (!mbar_wait(&v_full[s], (j >> 1) & 1, abort_flag)) { ok = false; break; }
                tc_fence_after();
                const uint32_t pa = smem_u32(sP), vb = smem_u32(sV + s * Lay::KV_BYTES);
                #pragma unroll
                for (int kk = 0; kk < TK / 16; ++kk)
                    umma_bf16(tO, sdesc_sw128(pa + (kk >> 2) * Lay::ATOM + (kk & 3) * 32),
                              sdesc_sw128_mn(vb + kk * 2048, Lay::ATOM, 1024), idesc_o, (j > 0 || kk > 0) ? 1u : 0u);
                umma_commit(&kv_empty[s]);
                umma_commit(pv_done);
            }
            if (!ok) {
                report(a.status, ST_TIMEOUT);
                *abort_flag = 1;
            }
            umma_commit(drain);
            const int never = 0;
            mbar_wait(drain, 0, &never);
        }
    } else {
        constexpr int NWG = kNWG<D>;
        constexpr int KC = TK / NWG;                  // key columns of S per warpgroup
        constexpr int OC = D / NWG;                   // columns of O per warpgroup (32)
        const int wg = (warp - 2) >> 2;
        const int quarter = warp & 3;
        const int r = quarter * 32 + lane;            // row of the q tile = TMEM lane
        const int qpos = q0 + r;                      // position inside the sequence
        const uint32_t lane_off = (uint32_t)(quarter * 32) << 16;
        const uint32_t p_row = smem_u32(sP) + r * 128;
        float *red_max = reinterpret_cast<float *>(smem + Lay::OFF_RED);   // [2][NWG][TQ]
        float *red_l = red_max + 2 * NWG * TQ;                             // [NWG][TQ]
        float m_use = -INFINITY, l = 0.f;
        bool good = true;   // every exit is decided at a barrier so all softmax warps leave together
        for (int j = 0; j < n_kt; ++j) {
            good = __all_sync(0xffffffffu, good && mbar_wait(&s_full[j & 1], (j >> 1) & 1, abort_flag));
            const uint32_t sbuf = tS + lane_off + (j & 1) * TK + wg * KC;
            const int key0 = j * TK + wg * KC;
            const bool diag = j * TK + TK - 1 > q0;
            // pass 1: this warpgroup's part of the row max of the scaled, masked scores
            float mt = -INFINITY;
            if (good) {
                tc_fence_after();
                #pragma unroll 1
                for (int c = 0; c < KC / 32; ++c) {
                    uint32_t v[32];
                    tmem_ld32(sbuf + c * 32, v);
                    tmem_ld_wait();
                    #pragma unroll
                    for (int i = 0; i < 32; ++i) {
                        float x = __uint_as_float(v[i]) * a.scale_log2;
                        if (diag && key0 + c * 32 + i > qpos) x = -INFINITY;
                        mt = fmaxf(mt, x);
                    }
                }
            }
            red_max[((j & 1) * NWG + wg) * TQ + r] = mt;
            if (!softmax_bar_and<128 * NWG>(good)) { good = false; break; }
            mt = red_max[((j & 1) * NWG) * TQ + r];
            #pragma unroll
            for (int w2 = 1; w2 < NWG; ++w2) mt = fmaxf(mt, red_max[((j & 1) * NWG + w2) * TQ + r]);
            float alpha = 1.f;
            bool rescale = false;
            if (j == 0) {
                m_use = mt;
            } else if (mt > m_use + kRescaleThreshold) {
                alpha = exp2f(m_use - mt);
                m_use = mt;
                rescale = true;
            }
            // P buffer and O are free once the previous P V product has completed
            if (j > 0) {
                good = __all_sync(0xffffffffu, mbar_wait(pv_done, (j - 1) & 1, abort_flag));
                if (good) tc_fence_after();
            }
            if (good) {
                if (__any_sync(0xffffffffu, rescale)) {
                    uint32_t v[32];
                    tmem_ld32(tO + lane_off + wg * OC, v);
                    tmem_ld_wait();
                    #pragma unroll
                    for (int i = 0; i < 32; ++i) v[i] = __float_as_uint(__uint_as_float(v[i]) * alpha);
                    tmem_st32(tO + lane_off + wg * OC, v);
                    tmem_st_wait();
                }
                l *= alpha;
                // pass 2: P = exp2(x - m_use) as bf16 into the K-major swizzled P tile
                #pragma unroll 1
                for (int c = 0; c < KC / 32; ++c) {
                    uint32_t v[32];
                    tmem_ld32(sbuf + c * 32, v);
                    tmem_ld_wait();
                    uint32_t pk[16];
                    #pragma unroll
                    for (int i = 0; i < 32; i += 2) {
                        float x0 = __uint_as_float(v[i]) * a.scale_log2;
                        float x1 = __uint_as_float(v[i + 1]) * a.scale_log2;
                        if (diag && key0 + c * 32 + i > qpos) x0 = -INFINITY;
                        if (diag && key0 + c * 32 + i + 1 > qpos) x1 = -INFINITY;
                        const float p0 = exp2f(x0 - m_use), p1 = exp2f(x1 - m_use);
                        l += p0 + p1;
                        pk[i >> 1] = pack_bf16x2(p0, p1);
                    }
                    #pragma unroll
                    for (int q = 0; q < 4; ++q) {
                        const int chunk = (wg * KC + c * 32) / 8 + q;      // 16-byte chunk = 8 keys
                        const uint32_t addr = p_row + (chunk >> 3) * Lay::ATOM + (((chunk & 7) ^ (r & 7)) << 4);
                        asm volatile("st.shared.v4.b32 [%0], {%1,%2,%3,%4};" ::"r"(addr), "r"(pk[4 * q]),
                                     "r"(pk[4 * q + 1]), "r"(pk[4 * q + 2]), "r"(pk[4 * q + 3])
                                     : "memory");
                    }
                }
                fence_proxy_async_smem();
                tc_fence_before();
                __syncwarp();
                if (lane == 0) mbar_arrive(p_full);
            }
        }
        // epilogue: row sums combined over the warpgroups, O / l -> bf16 -> global rows of this sequence
        if (good) good = __all_sync(0xffffffffu, mbar_wait(pv_done, (n_kt - 1) & 1, abort_flag));
        red_l[wg * TQ + r] = l;
        if (softmax_bar_and<128 * NWG>(good)) {
            tc_fence_after();
            float lt = 0.f;
            #pragma unroll
            for (int w2 = 0; w2 < NWG; ++w2) lt += red_l[w2 * TQ + r];
            const float inv = lt > 0.f ? 1.f / lt : 0.f;
            const bool live = qpos < L;
            bf16 *dst = a.o + (size_t)(seg0 + qpos) * a.ld_o + (size_t)head * D + wg * OC;
            uint32_t v[32];
            tmem_ld32(tO + lane_off + wg * OC, v);
            tmem_ld_wait();
            if (live) {
                uint4 *d4 = reinterpret_cast<uint4 *>(dst);
                #pragma unroll
                for (int q = 0; q < 4; ++q) {
                    uint4 u;
                    u.x = pack_bf16x2(__uint_as_float(v[8 * q + 0]) * inv, __uint_as_float(v[8 * q + 1]) * inv);
                    u.y = pack_bf16x2(__uint_as_float(v[8 * q + 2]) * inv, __uint_as_float(v[8 * q + 3]) * inv);
                    u.z = pack_bf16x2(__uint_as_float(v[8 * q + 4]) * inv, __uint_as_float(v[8 * q + 5]) * inv);
                    u.w = pack_bf16x2(__uint_as_float(v[8 * q + 6]) * inv, __uint_as_float(v[8 * q + 7]) * inv);
                    d4[q] = u;
                }
            }
        } else {
            good = false;
        }
        if (!good && lane == 0) {
            report(a.status, ST_TIMEOUT);
            *abort_flag = 1;
        }
    }

    __syncthreads();
    if (warp == 1) {
        tc_fence_after();
        tmem_dealloc(tmem_base, 512);
    }
}

template <int D>
cudaError_t launch_tc(const CUtensorMap &tm, const AttnTcArgs &args, int grid, cudaStream_t st) {
    static bool attr = false;
    if (!attr) {
        cudaError_t e = cudaFuncSetAttribute(attention_tc_kernel<D>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                             TcLayout<D>::SMEM);
        if (e != cudaSuccess) return e;
        attr = true;
    }
    cudaLaunchAttribute at[1];
    cudaLaunchConfig_t cfg = pdl_config(dim3(grid), dim3(kThreads<D>), TcLayout<D>::SMEM, st, at);
    return cudaLaunchKernelEx(&cfg, attention_tc_kernel<D>, tm, args);
}

}  // namespace

cudaError_t launch_attention(const bf16 *qkv, bf16 *o, int S, int nq, int nkv, int d, const int32_t *cu_host,
                             int n_seqs, int32_t *status, cudaStream_t st) {
    if (S <= 0) return cudaSuccess;
    if (d != 64 && d != 128) return cudaErrorInvalidValue;
    static AttnTcArgs args;
    const int ld = (nq + 2 * nkv) * d;
    CUtensorMap tm;
    if (!make_tmap_rows(&tm, qkv, (uint64_t)S, (uint64_t)ld, TQ)) return cudaErrorInvalidValue;
    args.o = o;
    args.ld_o = nq * d;
    args.nq = nq;
    args.group = nq / nkv;
    args.k_col0 = nq * d;
    args.v_col0 = (nq + nkv) * d;
    args.scale_log2 = (float)(1.4426950408889634 / std::sqrt((double)d));
    args.status = status;
    int n = 0, tiles = 0;
    if (!cu_host) {
        args.cu[0] = 0;
        args.cu[1] = S;
        args.tile_start[0] = 0;
        tiles = (S + TQ - 1) / TQ;
        n = 1;
    } else {
        args.cu[0] = 0;
        for (int i = 0; i < n_seqs; ++i) {
            const int len = cu_host[i + 1] - cu_host[i];
            if (len <= 0) continue;
            args.cu[n] = cu_host[i];
            args.tile_start[n] = tiles;
            tiles += (len + TQ - 1) / TQ;
            ++n;
            args.cu[n] = cu_host[i + 1];
        }
    }
    if (n == 0) return cudaSuccess;
    args.n_seqs = n;
    args.total_tiles = tiles;
    const int grid = tiles * nq;
    return d == 128 ? launch_tc<128>(tm, args, grid, st) : launch_tc<64>(tm, args, grid, st);
}

}  // namespace h3
