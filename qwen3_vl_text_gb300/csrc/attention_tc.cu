// Causal GQA attention over packed sequences on the tcgen05 tensor cores.
//
// Page "vllm-omni vllm_omni/diffusion/models/minimax_h3/encoder.py",
// MiniMaxH3Qwen3VLTextAttention.forward: q head h reads kv head h / (nq/nkv)
// (repeat_interleave), scaled_dot_product_attention(is_causal=True) with scale
// 1/sqrt(d), output columns head-major.  Packed sequences (cu_seqlens) attend
// only within themselves.  The same kernel runs the vision tower's bidirectional
// attention (MiniMaxH3Qwen3VLVisionAttention.forward: is_causal=False inside each
// frame, one head per kv head) with the causal mask off; there every item costs the same,
// and the pair-items of a thin last round run as single query tiles instead.
//
// Work item = two query tiles of 128 rows that read the same key/value tiles, so each
// K/V tile is staged once for 256 query rows: in causal attention with at least two q
// heads per kv head, the same 128 rows (one tile of the sequence) of two q heads of one
// kv group (A = head 2i, B = head 2i+1; both tiles need the same keys); otherwise two
// consecutive tiles of one head (A = rows q0.., B = rows q0+128..).  Persistent: one CTA per SM takes items heaviest first in
// alternating-direction rounds; TMEM, barriers and the K/V ring carry over from
// item to item, and an item's epilogue overlaps the next item's first products.
//   warp 0     TMA: Q_A and Q_B once, K and V tiles into a 2-stage ring (128-byte swizzle)
//   warp 1     TMEM allocation; tcgen05.mma from one thread, the two tiles interleaved
//              so that the tensor core works on one tile while the other's softmax runs:
//                S_t = Q_t K_j^T  (M=128, N=128, K=d)  into tile t's S columns
//                O_t += P_t V_j   (M=128, N=d, K=128)  P_t read from TMEM (A operand),
//                                  V as an MN-major operand straight from its TMA tile
//              issue order per key tile j: P_A V_j, S_A(j+1), P_B V_j, S_B(j+1)
//   warps 2-5  softmax of tile A, warps 6-9 of tile B: thread = one query row (its
//              TMEM lane) holding the whole 128-key row of S in registers: causal
//              mask, running max raised lazily (O rescaled in TMEM only when the max
//              grows by more than 2^8), P = exp2(s - m) as packed bf16 written over
//              the first 64 columns of its own S row; at the end O / l -> bf16 -> global
// TMEM columns: S_A 0-127, S_B 128-255, O_A 256-(256+d), O_B 384-(384+d).
// No softmax thread waits for another: the row max needs no exchange, and the
// previous P V product is awaited only before a rescale.  Every wait is bounded.
#include <atomic>
#include <cmath>
#include <utility>

#include "common.cuh"
#include "kernels.h"

namespace h3 {

namespace {

constexpr int TQ = 128;
constexpr int TK = 128;
constexpr int kThreads = 64 + 256;
constexpr float kRescaleThreshold = 8.0f;  // log2 units
constexpr int kMaxKeyRanges = 8;           // key ranges a split pair-item is cut into, at most

struct AttnTcArgs {
    bf16 *o;
    int ld_o;
    int nq, group;
    int k_col0, v_col0;
    float scale_log2;
    int n_seqs, total_pairs, n_items;   // "pairs": units of two query tiles (see head_pairs)
    int n_whole;   // items [0, n_whole) are pairs of query tiles; each later pair-item is run as
                   // two single-tile items, or (ks > 0) as ks items over consecutive key ranges
                   // (bidirectional mode, to fill a thin last round)
    int ks;                         // key ranges per split pair-item (0: split into single tiles)
    float *split_ws;                // ks > 0: [unit][tile][D + 2][128] fp32: O, m, l of each range
    int *split_cnt;                 // ks > 0: [split pair-item][tile][quarter] arrivals, 0 between launches
    int32_t *status;
    int cu[kMaxSeqs + 1];
    int pair_start[kMaxSeqs + 1];   // first unit of each sequence (a 128-row tile when head_pairs)
    unsigned long long *trace;      // optional [grid][ATR_COUNT] timeline
    float *row_amax;                // optional [S]: atomic max of |output| per row (bf16 values, >= 0)
    int causal;                     // 1: keys after the query are masked; 0: every key of the segment
    int head_pairs;                 // 1: an item is one 128-row tile of two q heads of one kv group
};

// Timeline of one persistent CTA (h3enc_op_attention_trace_next): %globaltimer at
// the start and the end, clock64 cycles for the phases in between (first item's Q,
// first score tile, last item's last P and last P V product), the SM id and the
// number of key tiles the CTA processed.
enum { ATR_START = 0, ATR_READY, ATR_Q, ATR_S0, ATR_LAST_P, ATR_O, ATR_END, ATR_SMID, ATR_NKT, ATR_COUNT };
__device__ __forceinline__ void astamp_ns(const AttnTcArgs &a, int what) {
    if (a.trace) {
        unsigned long long t;
        asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
        a.trace[(size_t)blockIdx.x * ATR_COUNT + what] = t;
    }
}
__device__ __forceinline__ void astamp_clk(const AttnTcArgs &a, int what) {
    if (a.trace) a.trace[(size_t)blockIdx.x * ATR_COUNT + what] = (unsigned long long)clock64();
}

template <int D>
struct TcLayout {
    static constexpr int ATOM = TQ * 128;          // one 64-column atom column of a 128-row tile: 16 KB
    static constexpr int Q_BYTES = TQ * D * 2;
    static constexpr int KV_BYTES = TK * D * 2;
    static constexpr int OFF_Q = 0;                             // Q_A, Q_B
    static constexpr int OFF_K = OFF_Q + 2 * Q_BYTES;
    static constexpr int OFF_V = OFF_K + 2 * KV_BYTES;
    static constexpr int OFF_BAR = OFF_V + 2 * KV_BYTES;
    static constexpr int SMEM = 1024 + OFF_BAR + 256;   // 15 barriers, TMEM slot, abort flag
};

// Paired fp32 arithmetic (two lanes per instruction) and the three-input maximum.
__device__ __forceinline__ uint64_t f32x2(float lo, float hi) {
    uint64_t r;
    asm("mov.b64 %0, {%1, %2};" : "=l"(r) : "f"(lo), "f"(hi));
    return r;
}
__device__ __forceinline__ void f32x2_split(uint64_t r, float &lo, float &hi) {
    asm("mov.b64 {%0, %1}, %2;" : "=f"(lo), "=f"(hi) : "l"(r));
}
__device__ __forceinline__ uint64_t ffma2(uint64_t a, uint64_t b, uint64_t c) {
    uint64_t r;
    asm("fma.rn.f32x2 %0, %1, %2, %3;" : "=l"(r) : "l"(a), "l"(b), "l"(c));
    return r;
}
__device__ __forceinline__ uint64_t fadd2(uint64_t a, uint64_t b) {
    uint64_t r;
    asm("add.rn.f32x2 %0, %1, %2;" : "=l"(r) : "l"(a), "l"(b));
    return r;
}
__device__ __forceinline__ float fmax3(float a, float b, float c) {
    float r;
    asm("max.f32 %0, %1, %2, %3;" : "=f"(r) : "f"(a), "f"(b), "f"(c));
    return r;
}

__device__ __forceinline__ float ex2(float x) {
    float y;
    asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}

// One work item = (unit, head or head pair); item k in heavy-first order.  Tile A is head
// `head`, rows q0..; tile B is head `head_b`, rows q0_b.. (nkt_b = 0: no tile B).
struct AttnItem {
    int head, head_b, seg0, L, q0, q0_b, nkt_a, nkt_b;
    int kt0;    // first key tile
    int unit;   // >= 0: key-range unit (k - n_whole) of a split pair-item; -1: whole item
};
__device__ __forceinline__ int seq_of_unit(const AttnTcArgs &a, int u) {
    int lo = 0, hi = a.n_seqs - 1;
    while (lo < hi) {
        const int mid = (lo + hi + 1) >> 1;
        if (a.pair_start[mid] <= u) lo = mid; else hi = mid - 1;
    }
    return lo;
}
template <bool CAUSAL>
__device__ __forceinline__ AttnItem attn_item(const AttnTcArgs &a, int k_in) {
    AttnItem it;
    it.kt0 = 0;
    it.unit = -1;
    if (a.head_pairs) {   // causal: heads (2i, 2i+1) share kv head and every key tile
        const int hp = a.nq >> 1;
        it.head = 2 * (k_in % hp);
        it.head_b = it.head + 1;
        const int tile_lin = a.total_pairs - 1 - k_in / hp;   // heavy tiles first
        const int sq = seq_of_unit(a, tile_lin);
        it.seg0 = a.cu[sq];
        it.L = a.cu[sq + 1] - it.seg0;
        it.q0 = it.q0_b = (tile_lin - a.pair_start[sq]) * TQ;
        it.nkt_a = it.nkt_b = (min(it.q0 + TQ, it.L) + TK - 1) / TK;
        return it;
    }
    // past n_whole: item n_whole + 2j + h is tile h of pair-item n_whole + j on its own, or with
    // key ranges (ks > 0) item n_whole + ks j + r is key range r of pair-item n_whole + j
    const int past = CAUSAL ? -1 : k_in - a.n_whole;   // the host splits bidirectional items only
    const int split = past >= 0 && a.ks == 0 ? (past & 1) + 1 : 0;   // 0 whole, 1 tile A, 2 tile B
    const int k = past < 0 ? k_in : a.ks ? a.n_whole + past / a.ks : a.n_whole + (past >> 1);
    it.head = it.head_b = k % a.nq;                       // heads fastest: one kv group's heads adjacent
    const int pair_lin = a.total_pairs - 1 - k / a.nq;    // heavy tile pairs first
    const int lo = seq_of_unit(a, pair_lin);
    it.seg0 = a.cu[lo];
    it.L = a.cu[lo + 1] - it.seg0;
    it.q0 = (pair_lin - a.pair_start[lo]) * (2 * TQ);
    // key tiles of each query tile (tile B is empty when the sequence ends inside tile A): up to
    // the query's own position when causal, the whole segment otherwise
    if (CAUSAL) {
        it.nkt_a = (min(it.q0 + TQ, it.L) + TK - 1) / TK;
        it.nkt_b = it.q0 + TQ < it.L ? (min(it.q0 + 2 * TQ, it.L) + TK - 1) / TK : 0;
    } else {
        const int all = (it.L + TK - 1) / TK;
        it.nkt_a = all;
        it.nkt_b = it.q0 + TQ < it.L ? all : 0;
    }
    if (split) {   // the host splits only pairs whose tile B exists
        if (split == 2) it.q0 += TQ;
        it.nkt_b = 0;
    }
    if (past >= 0 && a.ks) {   // key tiles [kt0, kt1) of the whole segment (bidirectional only)
        const int r = past % a.ks, all = it.nkt_a;
        it.kt0 = r * all / a.ks;
        const int n = (r + 1) * all / a.ks - it.kt0;
        it.nkt_a = n;
        it.nkt_b = it.nkt_b ? n : 0;
        it.unit = past;
    }
    it.q0_b = it.q0 + TQ;
    return it;
}
// The r-th item of CTA b among G persistent CTAs: rounds of G items, alternate rounds
// in reverse so the heavy items of one round pair with the light ones of the next.
__device__ __forceinline__ int attn_item_index(int r, int b, int G) {
    return r * G + ((r & 1) ? G - 1 - b : b);
}

template <int D, bool CAUSAL>
__global__ void __launch_bounds__(kThreads, 1)
    attention_tc_kernel(const __grid_constant__ CUtensorMap tm, const __grid_constant__ AttnTcArgs a) {
    using Lay = TcLayout<D>;
    extern __shared__ uint8_t smem_raw[];
    uint8_t *smem = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    uint8_t *sQ = smem + Lay::OFF_Q;
    uint8_t *sK = smem + Lay::OFF_K;
    uint8_t *sV = smem + Lay::OFF_V;
    uint64_t *bars = reinterpret_cast<uint64_t *>(smem + Lay::OFF_BAR);
    uint64_t *q_full = bars + 0;
    uint64_t *k_full = bars + 1;     // [2] ring stage
    uint64_t *v_full = bars + 3;     // [2]
    uint64_t *kv_empty = bars + 5;   // [2]
    uint64_t *s_full = bars + 7;     // [2] query tile
    uint64_t *p_full = bars + 9;     // [2] query tile (4 softmax warps arrive)
    uint64_t *pv_done = bars + 11;   // [2] query tile
    uint64_t *drain = bars + 13;
    uint64_t *q_empty = bars + 14;   // the item's score MMAs no longer read Q
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(bars + 15);
    volatile int *abort_flag = reinterpret_cast<volatile int *>(tmem_slot + 1);

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int G = gridDim.x, b = blockIdx.x;
    pdl_trigger();
    if (threadIdx.x == 0) {
        astamp_ns(a, ATR_START);
        if (a.trace) {
            uint32_t smid;
            asm volatile("mov.u32 %0, %%smid;" : "=r"(smid));
            a.trace[(size_t)b * ATR_COUNT + ATR_SMID] = smid;
        }
    }

    if (threadIdx.x == 0) {
        for (int i = 0; i < 15; ++i) mbar_init(bars + i, (i == 9 || i == 10) ? 4 : 1);
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
    if (threadIdx.x == 0) astamp_clk(a, ATR_READY);

    if (warp == 0) {
        if (lane == 0) {
            bool ok = true;
            uint32_t g = 0;          // key/value tiles loaded so far (ring position)
            uint32_t issued[2] = {0, 0};
            int steps = 0;
            for (int r = 0, it = 0; ok; ++r, ++it) {
                const int k = attn_item_index(r, b, G);
                if (k >= a.n_items) break;
                const AttnItem w = attn_item<CAUSAL>(a, k);
                const int kvh = w.head / a.group;
                const int n_kt = w.nkt_b > w.nkt_a ? w.nkt_b : w.nkt_a;
                steps += n_kt;
                if (it > 0 && !mbar_wait(q_empty, (it - 1) & 1, abort_flag)) { ok = false; break; }
                const int nq_tiles = w.nkt_b > 0 ? 2 : 1;
                mbar_arrive_expect_tx(q_full, nq_tiles * Lay::Q_BYTES);
                for (int t = 0; t < nq_tiles; ++t)
                    for (int c = 0; c < D / 64; ++c)
                        tma_load_2d(sQ + t * Lay::Q_BYTES + c * Lay::ATOM, &tm, q_full,
                                    (t ? w.head_b : w.head) * D + c * 64, w.seg0 + (t ? w.q0_b : w.q0));
                for (int j = 0; j < n_kt; ++j, ++g) {
                    const int s = g & 1;
                    if (g >= 2 && !mbar_wait(&kv_empty[s], ((g >> 1) - 1) & 1, abort_flag)) { ok = false; break; }
                    const int y = w.seg0 + ((CAUSAL ? 0 : w.kt0) + j) * TK;   // key ranges: bidirectional only
                    mbar_arrive_expect_tx(&k_full[s], Lay::KV_BYTES);
                    for (int c = 0; c < D / 64; ++c)
                        tma_load_2d(sK + s * Lay::KV_BYTES + c * Lay::ATOM, &tm, &k_full[s],
                                    a.k_col0 + kvh * D + c * 64, y);
                    mbar_arrive_expect_tx(&v_full[s], Lay::KV_BYTES);
                    for (int c = 0; c < D / 64; ++c)
                        tma_load_2d(sV + s * Lay::KV_BYTES + c * Lay::ATOM, &tm, &v_full[s],
                                    a.v_col0 + kvh * D + c * 64, y);
                    ++issued[s];
                }
            }
            if (a.trace) a.trace[(size_t)b * ATR_COUNT + ATR_NKT] = (unsigned long long)steps;
            if (!ok) {
                report(a.status, ST_TIMEOUT);
                *abort_flag = 1;
                // the copies still in flight land before the CTA may exit
                const int never = 0;
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
            bool ok = true;
            uint32_t g = 0;               // ring position of the item's first key tile
            uint32_t np[2] = {0, 0};      // P V products issued per query tile (p_full phases)
            // S_t = Q_t K^T for ring position gj into tile t's S columns
            auto issue_s = [&](int t, uint32_t gj) {
                const int s = gj & 1;
                if (!mbar_wait(&k_full[s], (gj >> 1) & 1, abort_flag)) return false;
                tc_fence_after();
                const uint32_t qa = smem_u32(sQ + t * Lay::Q_BYTES), kb = smem_u32(sK + s * Lay::KV_BYTES);
                #pragma unroll
                for (int kk = 0; kk < D / 16; ++kk) {
                    const uint32_t off = (kk >> 2) * Lay::ATOM + (kk & 3) * 32;
                    umma_bf16(tmem_base + t * TQ, sdesc_sw128(qa + off), sdesc_sw128(kb + off), idesc_s, kk > 0);
                }
                umma_commit(&s_full[t]);
                return true;
            };
            // O_t (+)= P_t V with P_t packed in the first 64 columns of tile t's S
            auto issue_pv = [&](int t, uint32_t gj, bool first) {
                const int s = gj & 1;
                if (!mbar_wait(&p_full[t], np[t] & 1, abort_flag)) return false;
                if (!mbar_wait(&v_full[s], (gj >> 1) & 1, abort_flag)) return false;
                ++np[t];
                tc_fence_after();
                const uint32_t vb = smem_u32(sV + s * Lay::KV_BYTES);
                const uint32_t pt = tmem_base + (uint32_t)(t * TQ);
                #pragma unroll
                for (int kk = 0; kk < TK / 16; ++kk)
                    umma_bf16_ts(tmem_base + 256 + t * 128, pt + kk * 8,
                                 sdesc_sw128_mn(vb + kk * 2048, Lay::ATOM, 1024), idesc_o,
                                 (!first || kk > 0) ? 1u : 0u);
                umma_commit(&pv_done[t]);
                return true;
            };
            for (int r = 0, it = 0; ok; ++r, ++it) {
                const int k = attn_item_index(r, b, G);
                if (k >= a.n_items) break;
                const AttnItem w = attn_item<CAUSAL>(a, k);
                const int n_kt = w.nkt_b > w.nkt_a ? w.nkt_b : w.nkt_a;
                if (!mbar_wait(q_full, it & 1, abort_flag)) { ok = false; break; }
                if (it == 0) astamp_clk(a, ATR_Q);
                ok = issue_s(0, g);
                if (ok && w.nkt_b > 0) ok = issue_s(1, g);
                if (ok && n_kt == 1) umma_commit(q_empty);
                for (int j = 0; j < n_kt && ok; ++j) {
                    if (j < w.nkt_a) {
                        if (!issue_pv(0, g + j, j == 0)) { ok = false; break; }
                        if (j + 1 < w.nkt_a && !issue_s(0, g + j + 1)) { ok = false; break; }
                    }
                    if (j < w.nkt_b) {
                        if (!issue_pv(1, g + j, j == 0)) { ok = false; break; }
                        if (j + 1 < w.nkt_b && !issue_s(1, g + j + 1)) { ok = false; break; }
                    }
                    if (j == n_kt - 2) umma_commit(q_empty);   // the item's last score MMAs are issued
                    umma_commit(&kv_empty[(g + j) & 1]);
                }
                g += n_kt;
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
        const int t = (warp - 2) >> 2;                // query tile of this warpgroup
        const int quarter = warp & 3;
        const int r_row = quarter * 32 + lane;        // row of the query tile = TMEM lane
        const uint32_t lane_off = (uint32_t)(quarter * 32) << 16;
        const uint32_t tS = tmem_base + lane_off + (uint32_t)(t * TQ);
        const uint32_t tO = tmem_base + lane_off + (uint32_t)(256 + t * 128);
        uint32_t c = 0;                               // steps of this query tile so far (barrier phases)
        bool good = true;
        for (int r = 0; good; ++r) {
            const int k = attn_item_index(r, b, G);
            if (k >= a.n_items) break;
            const AttnItem w = attn_item<CAUSAL>(a, k);
            const int nkt = t == 0 ? w.nkt_a : w.nkt_b;
            if (nkt == 0) continue;
            const int qtile0 = t ? w.q0_b : w.q0;
            const int qpos = qtile0 + r_row;          // position inside the sequence
            float m_use = -INFINITY, l = 0.f;
            for (int j = 0; j < nkt; ++j, ++c) {
                good = __all_sync(0xffffffffu, mbar_wait(&s_full[t], c & 1, abort_flag));
                if (!good) break;
                if (c == 0 && threadIdx.x == 64) astamp_clk(a, ATR_S0);
                tc_fence_after();
                uint32_t v[TK];
                {
                    uint32_t (&v0)[32] = *reinterpret_cast<uint32_t (*)[32]>(&v[0]);
                    uint32_t (&v1)[32] = *reinterpret_cast<uint32_t (*)[32]>(&v[32]);
                    uint32_t (&v2)[32] = *reinterpret_cast<uint32_t (*)[32]>(&v[64]);
                    uint32_t (&v3)[32] = *reinterpret_cast<uint32_t (*)[32]>(&v[96]);
                    tmem_ld32(tS, v0);
                    tmem_ld32(tS + 32, v1);
                    tmem_ld32(tS + 64, v2);
                    tmem_ld32(tS + 96, v3);
                    tmem_ld_wait();
                }
                // keys after the query masked (causal: the diagonal tile only), else the keys past
                // the segment's end (its last tile only); row max of the raw scores (the scale is
                // positive) as 8 independent chains
                const int key0 = ((CAUSAL ? 0 : w.kt0) + j) * TK;
                if constexpr (CAUSAL) {
                    if (key0 + TK - 1 > qtile0) {
                        #pragma unroll
                        for (int i = 0; i < TK; ++i)
                            if (key0 + i > qpos) v[i] = __float_as_uint(-INFINITY);
                    }
                } else if (key0 + TK > w.L) {
                    #pragma unroll
                    for (int i = 0; i < TK; ++i)
                        if (key0 + i >= w.L) v[i] = __float_as_uint(-INFINITY);
                }
                // (three-input maxima: chain u takes scores u, u + 8, ..., u + 120)
                float mx[8];
                #pragma unroll
                for (int u = 0; u < 8; ++u) {
                    float m = __uint_as_float(v[u]);
                    #pragma unroll
                    for (int k = 1; k < 15; k += 2)
                        m = fmax3(m, __uint_as_float(v[u + 8 * k]), __uint_as_float(v[u + 8 * k + 8]));
                    mx[u] = fmaxf(m, __uint_as_float(v[u + 120]));
                }
                const float mt = fmaxf(fmax3(mx[0], mx[1], mx[2]), fmax3(fmax3(mx[3], mx[4], mx[5]), mx[6], mx[7])) *
                                 a.scale_log2;
                float alpha = 1.f;
                bool rescale = false;
                if (j == 0) {
                    m_use = mt;
                } else if (mt > m_use + kRescaleThreshold) {
                    alpha = ex2(m_use - mt);
                    m_use = mt;
                    rescale = true;
                }
                // P = exp2(s * scale - m) packed as bf16 pairs over the first 64 columns of this
                // row of S; scale-and-subtract and the row sum on fp32 pairs, the sum in 4 chains
                const uint64_t scale2 = f32x2(a.scale_log2, a.scale_log2);
                const uint64_t neg_m2 = f32x2(-m_use, -m_use);
                uint64_t rs2[4] = {0ull, 0ull, 0ull, 0ull};
                #pragma unroll
                for (int h = 0; h < 2; ++h) {
                    uint32_t pk[32];
                    #pragma unroll
                    for (int i = 0; i < 32; ++i) {
                        const uint64_t x2 = ffma2(f32x2(__uint_as_float(v[64 * h + 2 * i]),
                                                        __uint_as_float(v[64 * h + 2 * i + 1])),
                                                  scale2, neg_m2);
                        float x0, x1;
                        f32x2_split(x2, x0, x1);
                        const float p0 = ex2(x0), p1 = ex2(x1);
                        rs2[i & 3] = fadd2(rs2[i & 3], f32x2(p0, p1));
                        pk[i] = pack_bf16x2(p0, p1);
                    }
                    tmem_st32(tS + 32 * h, pk);
                }
                float rs = 0.f;
                #pragma unroll
                for (int q = 0; q < 4; ++q) {
                    float r0, r1;
                    f32x2_split(rs2[q], r0, r1);
                    rs += r0 + r1;
                }
                l = l * alpha + rs;
                // O is rescaled after the previous P V product of this tile has completed
                if (__any_sync(0xffffffffu, rescale)) {
                    good = __all_sync(0xffffffffu, mbar_wait(&pv_done[t], (c - 1) & 1, abort_flag));
                    if (!good) break;
                    tc_fence_after();
                    #pragma unroll 1
                    for (int cc = 0; cc < D / 32; ++cc) {
                        uint32_t o[32];
                        tmem_ld32(tO + cc * 32, o);
                        tmem_ld_wait();
                        #pragma unroll
                        for (int i = 0; i < 32; ++i) o[i] = __float_as_uint(__uint_as_float(o[i]) * alpha);
                        tmem_st32(tO + cc * 32, o);
                    }
                }
                tmem_st_wait();
                tc_fence_before();
                __syncwarp();
                if (lane == 0) mbar_arrive(&p_full[t]);
            }
            if (!good) break;
            if (threadIdx.x == 64) astamp_clk(a, ATR_LAST_P);
            // epilogue: O / l -> bf16 -> global rows of this sequence; the next item's first P V
            // product (which overwrites O) waits for this warp's next P, issued after these reads
            good = __all_sync(0xffffffffu, mbar_wait(&pv_done[t], (c - 1) & 1, abort_flag));
            if (!good) break;
            if (threadIdx.x == 64) astamp_clk(a, ATR_O);
            tc_fence_after();
            const bool live = qpos < w.L;
            bf16 *dst = a.o + (size_t)(w.seg0 + qpos) * a.ld_o + (size_t)(t ? w.head_b : w.head) * D;
            if constexpr (!CAUSAL) {
                if (w.unit >= 0) {
                    // one key range of a split pair-item: its unnormalised O, running max and sum go
                    // to the workspace (consecutive lanes on consecutive floats); the warp whose range
                    // is the last to arrive for these 32 rows merges the ranges in range order
                    const size_t stride = (size_t)(D + 2) * 128;
                    float *mine = a.split_ws + (size_t)(w.unit * 2 + t) * stride;
                    #pragma unroll 1
                    for (int cc = 0; cc < D / 32; ++cc) {
                        uint32_t v[32];
                        tmem_ld32(tO + cc * 32, v);
                        tmem_ld_wait();
                        #pragma unroll
                        for (int i = 0; i < 32; ++i) mine[(size_t)(cc * 32 + i) * 128 + r_row] = __uint_as_float(v[i]);
                    }
                    mine[(size_t)D * 128 + r_row] = m_use;
                    mine[(size_t)(D + 1) * 128 + r_row] = l;
                    __threadfence();
                    __syncwarp();
                    const int r_unit = w.unit % a.ks;
                    int *cnt = a.split_cnt + ((w.unit / a.ks) * 2 + t) * 4 + quarter;
                    int prior = 0;
                    if (lane == 0) prior = atomicAdd(cnt, 1);
                    prior = __shfl_sync(0xffffffffu, prior, 0);
                    if (prior == a.ks - 1) {
                        __threadfence();
                        if (lane == 0) *cnt = 0;   // zero again for the next launch
                        const float *first = a.split_ws + (size_t)((w.unit - r_unit) * 2 + t) * stride;
                        float mx = -INFINITY;
                        for (int i = 0; i < a.ks; ++i)
                            mx = fmaxf(mx, __ldcg(first + (size_t)i * 2 * stride + (size_t)D * 128 + r_row));
                        float f[kMaxKeyRanges], lsum = 0.f;
                        #pragma unroll
                        for (int i = 0; i < kMaxKeyRanges; ++i) {
                            f[i] = 0.f;
                            if (i < a.ks) {
                                const float *u = first + (size_t)i * 2 * stride;
                                f[i] = ex2(__ldcg(u + (size_t)D * 128 + r_row) - mx);
                                lsum += __ldcg(u + (size_t)(D + 1) * 128 + r_row) * f[i];
                            }
                        }
                        const float inv_s = lsum > 0.f ? 1.f / lsum : 0.f;
                        float rmax_s = 0.f;
                        #pragma unroll 1
                        for (int cc = 0; cc < D / 32; ++cc) {
                            float o[32];
                            #pragma unroll
                            for (int k = 0; k < 32; ++k) o[k] = 0.f;
                            #pragma unroll
                            for (int i = 0; i < kMaxKeyRanges; ++i) {
                                if (i < a.ks) {
                                    const float *u = first + (size_t)i * 2 * stride + (size_t)(cc * 32) * 128 + r_row;
                                    #pragma unroll
                                    for (int k = 0; k < 32; ++k) o[k] += __ldcg(u + (size_t)k * 128) * f[i];
                                }
                            }
                            if (live) {
                                uint4 *d4 = reinterpret_cast<uint4 *>(dst + cc * 32);
                                #pragma unroll
                                for (int q = 0; q < 4; ++q) {
                                    uint4 uu;
                                    uu.x = pack_bf16x2(o[8 * q + 0] * inv_s, o[8 * q + 1] * inv_s);
                                    uu.y = pack_bf16x2(o[8 * q + 2] * inv_s, o[8 * q + 3] * inv_s);
                                    uu.z = pack_bf16x2(o[8 * q + 4] * inv_s, o[8 * q + 5] * inv_s);
                                    uu.w = pack_bf16x2(o[8 * q + 6] * inv_s, o[8 * q + 7] * inv_s);
                                    d4[q] = uu;
                                    const uint32_t uw[4] = {uu.x, uu.y, uu.z, uu.w};
                                    #pragma unroll
                                    for (int k = 0; k < 4; ++k)
                                        rmax_s = fmaxf(rmax_s, fmaxf(fabsf(bf16_lo(uw[k])), fabsf(bf16_hi(uw[k]))));
                                }
                            }
                        }
                        if (live && a.row_amax)
                            atomicMax(reinterpret_cast<int *>(a.row_amax + w.seg0 + qpos), __float_as_int(rmax_s));
                    }
                    continue;
                }
            }
            const float inv = l > 0.f ? 1.f / l : 0.f;
            float rmax = 0.f;   // largest |bf16 output| of this row's head
            #pragma unroll 1
            for (int cc = 0; cc < D / 32; ++cc) {
                uint32_t v[32];
                tmem_ld32(tO + cc * 32, v);
                tmem_ld_wait();
                if (live) {
                    uint4 *d4 = reinterpret_cast<uint4 *>(dst + cc * 32);
                    #pragma unroll
                    for (int q = 0; q < 4; ++q) {
                        uint4 u;
                        u.x = pack_bf16x2(__uint_as_float(v[8 * q + 0]) * inv, __uint_as_float(v[8 * q + 1]) * inv);
                        u.y = pack_bf16x2(__uint_as_float(v[8 * q + 2]) * inv, __uint_as_float(v[8 * q + 3]) * inv);
                        u.z = pack_bf16x2(__uint_as_float(v[8 * q + 4]) * inv, __uint_as_float(v[8 * q + 5]) * inv);
                        u.w = pack_bf16x2(__uint_as_float(v[8 * q + 6]) * inv, __uint_as_float(v[8 * q + 7]) * inv);
                        d4[q] = u;
                        const uint32_t uw[4] = {u.x, u.y, u.z, u.w};
                        #pragma unroll
                        for (int k = 0; k < 4; ++k)
                            rmax = fmaxf(rmax, fmaxf(fabsf(bf16_lo(uw[k])), fabsf(bf16_hi(uw[k]))));
                    }
                }
            }
            // non-negative floats order like their bit patterns: an integer max is exact
            if (live && a.row_amax)
                atomicMax(reinterpret_cast<int *>(a.row_amax + w.seg0 + qpos), __float_as_int(rmax));
        }
        if (!good && lane == 0) {
            report(a.status, ST_TIMEOUT);
            *abort_flag = 1;
        }
    }

    __syncwarp();
    tc_fence_before();
    __syncthreads();
    if (threadIdx.x == 0) astamp_ns(a, ATR_END);
    if (warp == 1) {
        tc_fence_after();
        tmem_dealloc(tmem_base, 512);
    }
}

template <int D, bool CAUSAL>
cudaError_t launch_tc(const CUtensorMap &tm, const AttnTcArgs &args, int grid, cudaStream_t st) {
    static std::atomic<bool> attr_of[kMaxDevices];   // per device: the shared-memory opt-in
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return cudaErrorInvalidDevice;
    if (!attr_of[dev].load()) {
        cudaError_t e = cudaFuncSetAttribute(attention_tc_kernel<D, CAUSAL>,
                                             cudaFuncAttributeMaxDynamicSharedMemorySize, TcLayout<D>::SMEM);
        if (e != cudaSuccess) return e;
        attr_of[dev].store(true);
    }
    cudaLaunchAttribute at[1];
    cudaLaunchConfig_t cfg = pdl_config(dim3(grid), dim3(kThreads), TcLayout<D>::SMEM, st, at);
    return cudaLaunchKernelEx(&cfg, attention_tc_kernel<D, CAUSAL>, tm, args);
}

thread_local unsigned long long *t_attn_trace = nullptr;

}  // namespace

void attention_trace_next(unsigned long long *trace) { t_attn_trace = trace; }
int attention_trace_fields() { return ATR_COUNT; }
size_t attention_workspace_bytes(int num_sms, int d) {
    return (size_t)num_sms * 2 * (d + 2) * 128 * sizeof(float) + (size_t)num_sms * 8 * sizeof(int);
}

cudaError_t launch_attention(const bf16 *qkv, bf16 *o, int S, int nq, int nkv, int d, const int32_t *cu_host,
                             int n_seqs, int32_t *status, cudaStream_t st, float *row_amax, bool causal,
                             void *workspace, size_t workspace_bytes) {
    if (S <= 0) return cudaSuccess;
    if (d != 64 && d != 128) return cudaErrorInvalidValue;
    AttnTcArgs args;   // per call: launches from several host threads do not share it
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
    args.trace = t_attn_trace;
    args.row_amax = row_amax;
    args.causal = causal ? 1 : 0;
    args.ks = 0;
    args.split_ws = nullptr;
    args.split_cnt = nullptr;
    // causal with an even number of q heads per kv head: items are one tile of two heads
    args.head_pairs = causal && args.group % 2 == 0 ? 1 : 0;
    const int unit = args.head_pairs ? TQ : 2 * TQ;   // query rows per unit
    t_attn_trace = nullptr;
    int n = 0, pairs = 0;
    if (!cu_host) {
        args.cu[0] = 0;
        args.cu[1] = S;
        args.pair_start[0] = 0;
        pairs = (S + unit - 1) / unit;
        n = 1;
    } else {
        args.cu[0] = 0;
        for (int i = 0; i < n_seqs; ++i) {
            const int len = cu_host[i + 1] - cu_host[i];
            if (len <= 0) continue;
            args.cu[n] = cu_host[i];
            args.pair_start[n] = pairs;
            pairs += (len + unit - 1) / unit;
            ++n;
            args.cu[n] = cu_host[i + 1];
        }
    }
    if (n == 0) return cudaSuccess;
    args.n_seqs = n;
    args.total_pairs = pairs;
    args.n_items = args.head_pairs ? pairs * (nq / 2) : pairs * nq;
    args.n_whole = args.n_items;
    int sms = device_num_sms();
    if (sms <= 0) sms = 1;
    if (!causal && args.n_items > sms) {
        // bidirectional items all cost the same: when the last round would hold few pair-items,
        // cut each into ks ranges of its keys (a workspace holds the ranges' partial results, merged
        // by whichever range finishes last), or without a workspace run them as single query tiles,
        // twice as many and half as long (pairs with a tile B only)
        const int I = args.n_items, rounds = (I + sms - 1) / sms, r = I - (rounds - 1) * sms;
        auto seg_of = [&](int k) {
            const int pair_lin = pairs - 1 - k / nq;
            int seg = 0;
            while (seg + 1 < n && args.pair_start[seg + 1] <= pair_lin) ++seg;
            return std::make_pair(seg, pair_lin);
        };
        if (workspace && workspace_bytes >= attention_workspace_bytes(sms, d) &&
            !(reinterpret_cast<uintptr_t>(workspace) & 15) && r < sms) {
            int ks = sms / r < kMaxKeyRanges ? sms / r : kMaxKeyRanges;
            for (int k = I - r; ks >= 2 && k < I; ++k) {
                const int seg = seg_of(k).first;
                const int all = (args.cu[seg + 1] - args.cu[seg] + TK - 1) / TK;
                if (all < ks) ks = all;
            }
            if (ks >= 2) {
                args.ks = ks;
                args.n_whole = I - r;
                args.n_items = I - r + r * ks;
                args.split_ws = static_cast<float *>(workspace);
                args.split_cnt = reinterpret_cast<int *>(static_cast<char *>(workspace) +
                                                         (size_t)sms * 2 * (d + 2) * 128 * sizeof(float));
            }
        }
        if (!args.ks) {
            bool ok = 2 * r <= sms;
            for (int k = I - r; ok && k < I; ++k) {
                const auto sp = seg_of(k);
                ok = (sp.second - args.pair_start[sp.first]) * 2 * TQ + TQ < args.cu[sp.first + 1] - args.cu[sp.first];
            }
            if (ok) {
                args.n_whole = I - r;
                args.n_items = I + r;
            }
        }
    }
    const int grid = args.n_items < sms ? args.n_items : sms;   // persistent: one CTA per SM
    if (causal) return d == 128 ? launch_tc<128, true>(tm, args, grid, st) : launch_tc<64, true>(tm, args, grid, st);
    return d == 128 ? launch_tc<128, false>(tm, args, grid, st) : launch_tc<64, false>(tm, args, grid, st);
}

}  // namespace h3
