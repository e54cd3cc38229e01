// Projection GEMM C = A * W^T on the 5th-generation tensor cores (tcgen05).
//
// Computes the F.linear calls of the decoder layer (page "vllm-omni
// vllm_omni/diffusion/models/minimax_h3/encoder.py": the QKV projection of
// MiniMaxH3Qwen3VLTextAttention.forward, o_proj, the gate/up pair and down_proj
// of MiniMaxH3Qwen3VLTextMLP.forward) with the element-wise work that follows
// each of them fused into the epilogue: the residual adds of
// MiniMaxH3Qwen3VLTextDecoderLayer.forward, silu(gate) * up, and the DeepStack
// add of MiniMaxH3Qwen3VLTextModel._deepstack_process.
//
// Design: CTA pairs (clusters of 2, one CTA per SM), persistent over 256 x 256
// output tiles.  CTA r of a pair owns output rows [128r, 128r+128) of the tile
// and stages, per k-block of 64, its own 128 x 64 slice of A and its half (128
// rows) of the 256 x 64 weight tile, so the pair reads each operand byte once.
//   warp 0     TMA producer: both slices into a 6-stage ring; the copies of
//              both CTAs complete on the leader CTA's stage barrier
//   warp 1     allocates 512 TMEM columns in both CTAs (two 128-lane x 256-column
//              fp32 accumulators); in the leader CTA one thread issues
//              tcgen05.mma.cta_group::2 (M=256, N=256, K=16) and commits to the
//              barriers of both CTAs
//   warps 2-9  epilogue of each CTA, two warps per 32-lane TMEM quarter, each of
//              the two taking half of the tile's columns: tcgen05.ld, fused
//              element-wise op, bf16 stores; overlaps the next tile's MMAs
// Schedule: the tiles of the full waves run data-parallel (tile = pair + i*pairs,
// M-fastest, so the pairs in flight share each weight tile through L2).  The
// tiles of the last, partial wave would leave SMs idle, so their k-blocks are laid
// end to end and cut into equal contiguous ranges, one per pair (stream-K); a range
// covers parts of at most two tiles.  Every pair runs its range FIRST: each CTA
// writes the fp32 partial of each part to a workspace slot, releases its flag,
// waits for the other contributors of those tiles, and sums the partials of a
// slice of rows in range order (deterministic) with the epilogue applied - all
// while the tensor cores already work on the pair's data-parallel tiles.  The grid
// never exceeds the number of co-resident pairs, so every wait ends.
// Every wait is bounded; on time-out the CTA records ST_TIMEOUT, drains its
// in-flight copies and MMAs, frees TMEM and exits.
#include <cudaTypedefs.h>

#include <atomic>

#include "common.cuh"
#include "kernels.h"

namespace h3 {

namespace {

constexpr int BM = 128;                          // output rows per CTA (a pair covers 256)
constexpr int BN = 256;                          // output columns per tile
constexpr int BK = 64;                           // bf16 elements per k-block (128 bytes per row)
constexpr int BK8 = 128;                         // e4m3 elements per k-block (the same 128 bytes)
constexpr int STAGES = 6;
constexpr int A_BYTES = BM * BK * 2;             // 16 KB
constexpr int B_BYTES = (BN / 2) * BK * 2;       // 16 KB: this CTA's half of the weight tile
constexpr int STAGE_BYTES = A_BYTES + B_BYTES;   // 32 KB per CTA
constexpr int EPI_WARPS = 8;
constexpr int EPI_THREADS = EPI_WARPS * 32;
constexpr int GEMM_THREADS = 64 + EPI_THREADS;
// per epilogue warp two 32 x 32 bf16 staging slots for the TMA tile stores
constexpr int C_SLOT_BYTES = 32 * 32 * 2;
constexpr int C_STAGE_BYTES = EPI_WARPS * 2 * C_SLOT_BYTES;   // 32 KB
constexpr int SMEM_BYTES = 1024 + STAGES * STAGE_BYTES + C_STAGE_BYTES + 256;
static_assert(SMEM_BYTES <= 227 * 1024, "shared memory of one CTA");
constexpr int kMinStreamKBlocks = 4;             // smallest k-range a stream-K pair takes
// cost of the stream-K partial exchange in k-block times (about 0.36 us each): behind
// data-parallel tiles, and alone (measured: ~3 us and ~15 us of the launch)
constexpr long long kSkFixupHidden = 8, kSkFixupExposed = 40;
// A launch of this many full waves or more runs unsplit.  Beside the split's exchange, its
// parts read k-ranges no other pair reads (cold, from DRAM) and its fix-up runs beside the
// mainloop, which then loses about 6-17 us whatever the launch's length (per-CTA timelines at
// seq 1024): more than a split saves at the end of a long launch (gate/up, ten and a half waves:
// 303 us unsplit against 309 us split in bf16, 166 against 176 us in e4m3), less than it saves
// in the one- and two-wave projections.
constexpr long long kSkMaxFullWaves = 8;
static_assert(BM * BN % 4 == 0, "partials are written as float4");

struct GemmArgs {
    int M, N, K;
    int nm, nn, nk;        // nm: 256-row blocks
    __nv_bfloat16 *C;
    int ldc;
    const __nv_bfloat16 *R;
    const __nv_bfloat16 *DS;
    const int32_t *vis_rank;
    int n_vis;
    int32_t *status;
    // stream-K over the last partial wave
    int dp_tiles;      // tiles run data-parallel: [0, dp_tiles)
    int sk_pairs;      // pairs [0, sk_pairs) share the k-blocks of tiles [dp_tiles, nm*nn); 0: none
    long long sk_work; // (nm*nn - dp_tiles) * nk
    float *part;       // [2*grid][BM*BN] fp32 partials: slot 4*pair + 2*part + rank
    uint32_t *flags;   // [grid] release flags: equal to this launch's epoch = "partial written"
    uint32_t *ctrl;    // [2] in device memory: the epoch of the last stream-K launch on this
                       // workspace, and the count of this launch's finished CTAs
    // EPI_QKROPE
    const __nv_bfloat16 *wq, *wk;
    const float *cos_t, *sin_t;
    int cs_rows;       // 0: tables [M][head_dim/2]; > 0: [head_dim/8][cs_rows][4] (see cs_at)
    int head_dim, nq, nkv;
    float eps;
    unsigned long long *trace;   // optional [grid][TR_COUNT] %globaltimer stamps
    // e4m3 operands: C = (A8 * sa[row]) (W8 * sw[col])^T
    const float *sa, *sw;
    float *row_amax;   // EPI_SWIGLU, optional: per-row max |bf16 output| (integer atomic max)
    int w_static;      // W is not written by earlier kernels of the stream: its first stages are
                       // fetched before the dependency wait
    // RMSNorm folded into the projection: ss_in [K/128][M] row sums of squares of A (rows of the
    // accumulator scaled by 1/sqrt(sum/K + norm_eps)); ss_out [N/128][M] the same sums of the
    // bf16 output
    const float *ss_in;
    float *ss_out;
    float norm_eps;
    const __nv_bfloat16 *bias;   // optional [N], added to the accumulator (not with SWIGLU)
};

// Phase stamps of the optional timeline (h3enc_op_gemm_traced).
enum { TR_START = 0, TR_READY, TR_LAST_ACC, TR_FIRST_MMA, TR_LAST_DP_MMA, TR_DP_EPI_DONE, TR_SPLIT_MMA_DONE,
       TR_DUMP_DONE, TR_FLAGS_SEEN, TR_REDUCE_DONE, TR_END, TR_COUNT };
__device__ __forceinline__ void stamp(const GemmArgs &g, int what) {
    if (g.trace) {
        unsigned long long t;
        asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
        g.trace[(size_t)blockIdx.x * TR_COUNT + what] = t;
    }
}

// Epoch of a stream-K launch: one more than the workspace's last one (0 is skipped: it is the
// value of a fresh flag).  Read after the dependency wait; the last CTA to finish stores it, so a
// launch replayed from a CUDA graph gets a new epoch too.
__device__ __forceinline__ uint32_t sk_epoch(const GemmArgs &g) {
    const uint32_t e = __ldcg(g.ctrl) + 1u;
    return e == 0u ? 1u : e;
}

// Stream-K ranges: pair p owns k-iterations [start(p), start(p+1)) of the tail laid
// end to end (tail tile t holds iterations [t*nk, (t+1)*nk)).
__device__ __forceinline__ long long sk_start(const GemmArgs &g, int p) {
    return (long long)p * g.sk_work / g.sk_pairs;
}
// The pair whose range holds iteration x.
__device__ __forceinline__ int sk_pair_of(const GemmArgs &g, long long x) {
    return (int)(((x + 1) * g.sk_pairs - 1) / g.sk_work);
}
// The (at most two) parts of this pair's range, each inside one tile.
struct StreamK {
    int n;
    int tile[2], kb0[2], kb1[2];
};
__device__ __forceinline__ StreamK stream_k(const GemmArgs &g, int pair) {
    StreamK sk{};
    if (pair >= g.sk_pairs) return sk;
    long long x = sk_start(g, pair);
    const long long e = sk_start(g, pair + 1);
    while (x < e && sk.n < 2) {
        const int t = (int)(x / g.nk);
        const long long te = (long long)(t + 1) * g.nk;
        const long long pe = e < te ? e : te;
        sk.tile[sk.n] = t;
        sk.kb0[sk.n] = (int)(x - (long long)t * g.nk);
        sk.kb1[sk.n] = (int)(pe - (long long)t * g.nk);
        ++sk.n;
        x = pe;
    }
    return sk;
}
// Contributors [pa, pb] of tail tile t, and the part index of t within pair q's range.
__device__ __forceinline__ void sk_contributors(const GemmArgs &g, int t, int &pa, int &pb) {
    pa = sk_pair_of(g, (long long)t * g.nk);
    pb = sk_pair_of(g, (long long)(t + 1) * g.nk - 1);
}
__device__ __forceinline__ int sk_part_index(const GemmArgs &g, int q, int t) {
    return sk_start(g, q) < (long long)t * g.nk ? 1 : 0;
}
// Partial slots are written coalesced: float4 (row r, columns col..col+3) of the
// 128 x 256 partial sits at float4 index ((col/32)*8 + (col%32)/4)*128 + r.
__device__ __forceinline__ size_t part_f4(int r, int col) {
    return ((size_t)((col >> 5) * 8 + ((col & 31) >> 2)) << 7) + (size_t)r;
}

// 1/rms of row `row` of A from the slot sums of squares (slots of 128 columns, added in slot
// order: the same value for every tile of the row).
// Element (row, j) of the rotary tables, j a multiple of 4: four consecutive frequencies are
// one aligned float4 in either layout.  Row-interleaved ([d/8][cs_rows][4]) puts the same
// four frequencies of consecutive rows side by side, so an epilogue warp (32 consecutive
// rows, one per lane) reads whole lines instead of touching 32 lines per load.
__device__ __forceinline__ size_t cs_at(const GemmArgs &g, int row, int j) {
    return g.cs_rows ? ((size_t)(j >> 2) * g.cs_rows + row) * 4 + (j & 3)
                     : (size_t)row * (g.head_dim >> 1) + j;
}

__device__ __forceinline__ float norm_rstd(const GemmArgs &g, int row) {
    const int slots = g.K >> 7;
    float s = 0.f;
    for (int i0 = 0; i0 < slots; i0 += 16) {
        float v[16];
        #pragma unroll
        for (int i = 0; i < 16; ++i) v[i] = i0 + i < slots ? __ldcg(g.ss_in + (size_t)(i0 + i) * g.M + row) : 0.f;
        #pragma unroll
        for (int i = 0; i < 16; ++i) s += v[i];
    }
    return 1.0f / sqrtf(s / (float)g.K + g.norm_eps);
}

__device__ __forceinline__ uint32_t ld_acquire(const uint32_t *p) {
    uint32_t v;
    asm volatile("ld.acquire.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
    return v;
}
__device__ __forceinline__ void st_release(uint32_t *p, uint32_t v) {
    asm volatile("st.release.gpu.global.u32 [%0], %1;" ::"l"(p), "r"(v) : "memory");
}
// Barrier over the epilogue warps (named barrier 1) returning the AND of v.
__device__ __forceinline__ bool epi_bar_and(bool v) {
    uint32_t r;
    asm volatile(
        "{\n\t.reg .pred p, q;\n\t"
        "setp.ne.u32 p, %1, 0;\n\t"
        "bar.red.and.pred q, 1, %2, p;\n\t"
        "selp.u32 %0, 1, 0, q;\n\t}"
        : "=r"(r)
        : "r"((uint32_t)v), "n"(EPI_THREADS)
        : "memory");
    return r != 0;
}

// silu(g) * u = g * u / (1 + e^-g), with the fast exponential and division intrinsics (a few
// ulps of fp32, far below the bf16 rounding of the result); a very negative g gives 0.
__device__ __forceinline__ float silu_mul(float g, float u) { return __fdividef(g * u, 1.0f + __expf(-g)); }
// GELU of the vision tower: the tanh form in the blocks' MLP, the exact (erf) form in the mergers.
// tanh from the hardware's approximate instruction (relative error about 2^-11, below the bf16
// rounding of the output)
__device__ __forceinline__ float tanh_hw(float x) {
    float y;
    asm("tanh.approx.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}
__device__ __forceinline__ float gelu_tanh(float x) {
    return 0.5f * x * (1.0f + tanh_hw(0.7978845608028654f * (x + 0.044715f * x * x * x)));   // sqrt(2/pi)
}
__device__ __forceinline__ float gelu_erf(float x) { return 0.5f * x * (1.0f + erff(x * 0.7071067811865476f)); }

__device__ __forceinline__ void load_row32(const __nv_bfloat16 *p, float (&f)[32]) {
    const uint4 *q = reinterpret_cast<const uint4 *>(p);
    #pragma unroll
    for (int i = 0; i < 4; ++i) {
        uint4 v = q[i];
        f[8 * i + 0] = bf16_lo(v.x); f[8 * i + 1] = bf16_hi(v.x);
        f[8 * i + 2] = bf16_lo(v.y); f[8 * i + 3] = bf16_hi(v.y);
        f[8 * i + 4] = bf16_lo(v.z); f[8 * i + 5] = bf16_hi(v.z);
        f[8 * i + 6] = bf16_lo(v.w); f[8 * i + 7] = bf16_hi(v.w);
    }
}

template <int EPI, bool F8>
__global__ void __launch_bounds__(GEMM_THREADS, 1)
    gemm_tcgen05_kernel(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB,
                        const __grid_constant__ CUtensorMap tmC, const GemmArgs g) {
    extern __shared__ uint8_t smem_raw[];
    uint8_t *smem = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    uint8_t *sA = smem;
    uint8_t *sB = smem + STAGES * A_BYTES;
    uint8_t *sC = sB + STAGES * B_BYTES;   // epilogue staging (1024-byte aligned)
    uint64_t *full = reinterpret_cast<uint64_t *>(sC + C_STAGE_BYTES);
    uint64_t *empty = full + STAGES;
    uint64_t *acc_full = empty + STAGES;
    uint64_t *acc_empty = acc_full + 2;
    uint64_t *drain = acc_empty + 2;
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(drain + 1);
    volatile int *abort_flag = reinterpret_cast<volatile int *>(tmem_slot + 1);

    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    const uint32_t rank = cluster_ctarank();       // 0: leader CTA of the pair
    const int pair = blockIdx.x >> 1;
    const int npairs = gridDim.x >> 1;
    pdl_trigger();
    if (threadIdx.x == 0) stamp(g, TR_START);

    if (threadIdx.x == 0) {
        for (int s = 0; s < STAGES; ++s) {
            mbar_init(&full[s], 1);      // leader's arrive.expect_tx; the copies of both CTAs complete on it
            mbar_init(&empty[s], 1);     // leader's MMA commit, multicast to both CTAs
        }
        for (int a = 0; a < 2; ++a) {
            mbar_init(&acc_full[a], 1);  // leader's MMA commit, multicast to both CTAs
            mbar_init(&acc_empty[a], 2 * EPI_WARPS); // the epilogue warps of both CTAs (leader's barrier used)
        }
        mbar_init(drain, 1);
        *abort_flag = 0;
        fence_barrier_init();
    }
    if (warp == 0 && lane == 0) {
        prefetch_tmap(&tmA);
        prefetch_tmap(&tmB);
    }
    if (warp == 1) {
        tmem_alloc_pair(tmem_slot, 512);
        tmem_relinquish_pair();
    }
    tc_fence_before();
    cluster_sync();   // barriers of both CTAs initialised before any cross-CTA signal
    tc_fence_after();
    const uint32_t tmem_base = *tmem_slot;
    // the previous kernel's outputs (A, the residual, the workspace) are touched only after the
    // dependency wait, which each role takes itself
    const StreamK sk = stream_k(g, pair);

    if (warp == 0) {
        if (lane == 0) {
            int stage = 0;
            uint32_t phase = 0;
            uint32_t issued[STAGES];
            #pragma unroll
            for (int s = 0; s < STAGES; ++s) issued[s] = 0;
            bool ok = true;
            auto load_item = [&](int tile, int kb0, int kb1) {
                const int m0 = (tile % g.nm) * (2 * BM) + (int)rank * BM;
                const int n0 = (tile / g.nm) * BN + (int)rank * (BN / 2);
                for (int kb = kb0; kb < kb1; ++kb) {
                    if (!mbar_wait(&empty[stage], phase ^ 1u, abort_flag)) { ok = false; return; }
                    if (rank == 0) mbar_arrive_expect_tx(&full[stage], 2 * STAGE_BYTES);
                    const uint32_t bar = mapa_shared(smem_u32(&full[stage]), 0);
                    constexpr int kbe = F8 ? BK8 : BK;   // elements of one 128-byte k-block row
                    tma_load_2d_pair(sA + stage * A_BYTES, &tmA, bar, kb * kbe, m0);
                    tma_load_2d_pair(sB + stage * B_BYTES, &tmB, bar, kb * kbe, n0);
                    ++issued[stage];
                    if (++stage == STAGES) { stage = 0; phase ^= 1u; }
                }
            };
            // weights that no earlier kernel writes: the first ring stages of the first item get
            // their weight half while the previous kernel is still finishing
            constexpr int kbe0 = F8 ? BK8 : BK;
            int pre = 0;
            {
                const bool has = sk.n > 0 || pair < g.dp_tiles;
                const int ft = sk.n > 0 ? g.dp_tiles + sk.tile[0] : pair;
                const int fk0 = sk.n > 0 ? sk.kb0[0] : 0, fk1 = sk.n > 0 ? sk.kb1[0] : g.nk;
                if (g.w_static && has) {
                    pre = fk1 - fk0 < STAGES ? fk1 - fk0 : STAGES;
                    const int n0 = (ft / g.nm) * BN + (int)rank * (BN / 2);
                    for (int i = 0; i < pre; ++i) {   // a fresh ring: every stage is free
                        if (rank == 0) mbar_arrive_expect_tx(&full[i], 2 * STAGE_BYTES);
                        tma_load_2d_pair(sB + i * B_BYTES, &tmB, mapa_shared(smem_u32(&full[i]), 0),
                                         (fk0 + i) * kbe0, n0);
                    }
                }
                pdl_wait();
                stamp(g, TR_READY);
                if (pre) {
                    const int m0 = (ft % g.nm) * (2 * BM) + (int)rank * BM;
                    for (int i = 0; i < pre; ++i) {
                        tma_load_2d_pair(sA + i * A_BYTES, &tmA, mapa_shared(smem_u32(&full[i]), 0),
                                         (fk0 + i) * kbe0, m0);
                        ++issued[i];
                    }
                    stage = pre % STAGES;
                    if (pre == STAGES) phase ^= 1u;
                }
            }
            int skip = pre;   // k-blocks of the first item already issued
            for (int j = 0; ok && j < sk.n; ++j) {
                load_item(g.dp_tiles + sk.tile[j], sk.kb0[j] + skip, sk.kb1[j]);
                skip = 0;
            }
            for (int tile = pair; ok && tile < g.dp_tiles; tile += npairs) {
                load_item(tile, skip, g.nk);
                skip = 0;
            }
            if (!ok) {
                report(g.status, ST_TIMEOUT);
                *abort_flag = 1;
                // the leader waits (bounded) for the copies still in flight into the pair's rings
                if (rank == 0) {
                    const int never = 0;
                    for (int s = 0; s < STAGES; ++s)
                        if (issued[s]) mbar_wait(&full[s], (issued[s] - 1u) & 1u, &never);
                }
            }
        }
    } else if (warp == 1) {
        pdl_wait();
        if (lane == 0 && rank == 0) {
            constexpr uint32_t idesc = F8 ? umma_idesc_e4m3(2 * BM, BN) : umma_idesc_bf16(2 * BM, BN);
            int stage = 0;
            uint32_t phase = 0;
            int acc = 0;
            uint32_t acc_phase = 0;
            bool ok = true;
            bool first_mma = true;
            auto mma_item = [&](int kb0, int kb1) {
                if (!mbar_wait(&acc_empty[acc], acc_phase ^ 1u, abort_flag)) { ok = false; return; }
                if (first_mma) { stamp(g, TR_FIRST_MMA); first_mma = false; }
                tc_fence_after();
                const uint32_t d_tmem = tmem_base + (uint32_t)(acc * BN);
                for (int kb = kb0; kb < kb1; ++kb) {
                    if (!mbar_wait(&full[stage], phase, abort_flag)) { ok = false; return; }
                    tc_fence_after();
                    const uint32_t a_base = smem_u32(sA + stage * A_BYTES);
                    const uint32_t b_base = smem_u32(sB + stage * B_BYTES);
                    #pragma unroll
                    for (int kk = 0; kk < 4; ++kk)   // 32-byte steps: K = 16 bf16 or K = 32 e4m3 per MMA
                        umma_pair<F8>(d_tmem, sdesc_sw128(a_base + kk * 32), sdesc_sw128(b_base + kk * 32), idesc,
                                       (kb > kb0 || kk > 0) ? 1u : 0u);
                    umma_commit_pair(&empty[stage], 0x3);
                    if (++stage == STAGES) { stage = 0; phase ^= 1u; }
                }
                umma_commit_pair(&acc_full[acc], 0x3);
                acc ^= 1;
                if (acc == 0) acc_phase ^= 1u;
            };
            for (int j = 0; ok && j < sk.n; ++j) mma_item(sk.kb0[j], sk.kb1[j]);
            for (int tile = pair; ok && tile < g.dp_tiles; tile += npairs) mma_item(0, g.nk);
            stamp(g, TR_LAST_DP_MMA);
            if (!ok) {
                report(g.status, ST_TIMEOUT);
                *abort_flag = 1;
            }
            // every MMA issued by this thread has completed once `drain` flips
            umma_commit_pair(drain, 0x1);
            const int never = 0;
            mbar_wait(drain, 0, &never);
        }
    } else {
        pdl_wait();   // the residual, DeepStack rows, scales and the workspace come from earlier kernels
        // epilogue: warp w reads TMEM lanes 32*(w%4) .. +31 = this CTA's tile rows of the same range;
        // warps 2-5 take the first half of the tile's columns, warps 6-9 the second
        const int quarter = warp & 3;
        const int ehalf = (warp - 2) >> 2;
        const int et = threadIdx.x - 64;  // 0..255 over the epilogue warps
        // e4m3 operands: accumulator column n of row m times sa[m] * sw[n] (32 columns from n0; the
        // sw loads are the same address across the warp)
        auto dq32 = [&](uint32_t (&v)[32], int m, bool live_row, int n0) {
            if constexpr (F8) {
                const float sr = live_row ? g.sa[m] : 0.f;
                const float4 *w4 = reinterpret_cast<const float4 *>(g.sw + n0);
                #pragma unroll
                for (int q = 0; q < 8; ++q) {
                    const float4 sw = w4[q];
                    v[4 * q + 0] = __float_as_uint(__uint_as_float(v[4 * q + 0]) * (sr * sw.x));
                    v[4 * q + 1] = __float_as_uint(__uint_as_float(v[4 * q + 1]) * (sr * sw.y));
                    v[4 * q + 2] = __float_as_uint(__uint_as_float(v[4 * q + 2]) * (sr * sw.z));
                    v[4 * q + 3] = __float_as_uint(__uint_as_float(v[4 * q + 3]) * (sr * sw.w));
                }
            }
        };
        auto dq4 = [&](float *f, float sr, int n0) {
            if constexpr (F8) {
                const float4 sw = *reinterpret_cast<const float4 *>(g.sw + n0);
                f[0] *= sr * sw.x; f[1] *= sr * sw.y; f[2] *= sr * sw.z; f[3] *= sr * sw.w;
            }
        };
        // + bias[n0 .. n0 + 32) (the same 64 bytes for the whole warp: broadcast loads)
        auto bias32 = [&](uint32_t (&v)[32], int n0) {
            if (g.bias) {
                const uint4 *b4 = reinterpret_cast<const uint4 *>(g.bias + n0);
                #pragma unroll
                for (int q = 0; q < 4; ++q) {
                    const uint4 bb = __ldg(b4 + q);
                    const uint32_t w4[4] = {bb.x, bb.y, bb.z, bb.w};
                    #pragma unroll
                    for (int t = 0; t < 4; ++t) {
                        v[8 * q + 2 * t] = __float_as_uint(__uint_as_float(v[8 * q + 2 * t]) + bf16_lo(w4[t]));
                        v[8 * q + 2 * t + 1] = __float_as_uint(__uint_as_float(v[8 * q + 2 * t + 1]) + bf16_hi(w4[t]));
                    }
                }
            }
        };
        auto bias4 = [&](float *f, int n0) {
            if (g.bias) {
                const uint2 bb = *reinterpret_cast<const uint2 *>(g.bias + n0);
                f[0] += bf16_lo(bb.x); f[1] += bf16_hi(bb.x); f[2] += bf16_lo(bb.y); f[3] += bf16_hi(bb.y);
            }
        };
        // data-parallel outputs leave through shared memory: the warp's 32 rows x 32 columns are
        // written to one of its two slots (row = lane, 64 bytes each) and stored by one TMA tile
        // store (rows past M are clipped); a slot is refilled once its store has read it
        uint8_t *cslots = sC + (warp - 2) * 2 * C_SLOT_BYTES;
        uint32_t cstores = 0;
        auto store_chunk = [&](const uint32_t (&pk)[16], int col, int row0) {
            uint8_t *slot = cslots + (cstores & 1) * C_SLOT_BYTES;
            if (lane == 0) bulk_wait_read<1>();
            __syncwarp();
            // 64-byte swizzle (as the tensor map): 16-byte unit q of row r at unit q ^ ((r >> 1) & 3),
            // so the warp's four stores are bank-conflict free
            uint4 *dst = reinterpret_cast<uint4 *>(slot + lane * 64);
            const int sw = (lane >> 1) & 3;
            #pragma unroll
            for (int q = 0; q < 4; ++q) dst[q ^ sw] = make_uint4(pk[4 * q], pk[4 * q + 1], pk[4 * q + 2], pk[4 * q + 3]);
            fence_proxy_async_smem();
            __syncwarp();
            if (lane == 0 && row0 < g.M) {   // a box wholly past the last row is not issued
                tma_store_2d(&tmC, slot, col, row0);
                bulk_commit();
            }
            ++cstores;
        };
        auto store_chunk_f = [&](const float (&f)[32], int col, int row0) {
            uint32_t pk[16];
            #pragma unroll
            for (int i = 0; i < 16; ++i) pk[i] = pack_bf16x2(f[2 * i], f[2 * i + 1]);
            store_chunk(pk, col, row0);
        };
        const uint32_t acc_empty_lead[2] = {mapa_shared(smem_u32(&acc_empty[0]), 0),
                                            mapa_shared(smem_u32(&acc_empty[1]), 0)};
        int acc = 0;
        uint32_t acc_phase = 0;
        bool ok = true;
        auto wait_acc = [&]() {
            bool w = mbar_wait(&acc_full[acc], acc_phase, abort_flag);
            w = __all_sync(0xffffffffu, w);
            if (!w) {
                if (lane == 0) {
                    report(g.status, ST_TIMEOUT);
                    *abort_flag = 1;
                }
                ok = false;
                return false;
            }
            tc_fence_after();
            return true;
        };
        auto release_acc = [&]() {
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive_cluster(acc_empty_lead[acc]);
            acc ^= 1;
            if (acc == 0) acc_phase ^= 1u;
        };
        // ---- stream-K parts first: their partials, flags and reduction overlap the MMAs of the
        //      data-parallel tiles ----
        if (sk.n > 0) {
            // 1) the fp32 accumulator of part j (this CTA's 128 rows) goes to slot 4*pair + 2*j + rank;
            //    every epilogue warp reaches each barrier below, failed or not
            bool dumped = true;
            for (int j = 0; j < sk.n; ++j) {
                const bool got = ok && wait_acc();
                if (et == 0 && j == 0) stamp(g, TR_SPLIT_MMA_DONE);
                if (got) {
                    const uint32_t taddr = tmem_base + ((uint32_t)(quarter * 32) << 16) + (uint32_t)(acc * BN);
                    float4 *slot = reinterpret_cast<float4 *>(g.part) + (size_t)(4 * pair + 2 * j + (int)rank) * (BM * BN / 4);
                    const int r = quarter * 32 + lane;
                    #pragma unroll 1
                    for (int c = ehalf * (BN / 64); c < (ehalf + 1) * (BN / 64); ++c) {
                        uint32_t v[32];
                        tmem_ld32(taddr + c * 32, v);
                        tmem_ld_wait();
                        #pragma unroll
                        for (int q = 0; q < 8; ++q)
                            slot[part_f4(r, c * 32 + 4 * q)] =
                                make_float4(__uint_as_float(v[4 * q]), __uint_as_float(v[4 * q + 1]),
                                            __uint_as_float(v[4 * q + 2]), __uint_as_float(v[4 * q + 3]));
                    }
                    release_acc();
                }
                dumped = dumped && got;
            }
            __threadfence();
            if (epi_bar_and(dumped)) {
                if (et == 0) {
                    stamp(g, TR_DUMP_DONE);
                    st_release(g.flags + blockIdx.x, sk_epoch(g));
                }
                for (int j = 0; j < sk.n; ++j) {
                    // 2) wait for the same-rank CTAs of the tile's contributors: thread i polls contributor
                    //    pa + i (all flags in flight at once), then the AND over the epilogue warps
                    const int t = sk.tile[j];
                    int pa, pb;
                    sk_contributors(g, t, pa, pb);
                    const int nc = pb - pa + 1;
                    bool seen = true;
                    if (et < nc) {
                        const long long t0 = clock64();
                        const uint32_t epoch = sk_epoch(g);
                        while (ld_acquire(g.flags + 2 * (pa + et) + rank) != epoch) {
                            if (clock64() - t0 > kSpinLimitCycles) { seen = false; break; }
                        }
                    }
                    const bool all = epi_bar_and(seen);
                    if (et == 0 && j == 0) stamp(g, TR_FLAGS_SEEN);
                    if (!all) {
                        if (et == 0) report(g.status, ST_TIMEOUT);
                        break;
                    }
                    // 3) rows [r0, r1) of this CTA's half: the contributors' partials summed in range order,
                    //    then the epilogue
                    const int ci = pair - pa;
                    const int r0 = ci * BM / nc, r1 = (ci + 1) * BM / nc;
                    const int tile = g.dp_tiles + t;
                    const int m_blk = tile % g.nm, n_blk = tile / g.nm;
                    const int slot_pa = 4 * pa + 2 * sk_part_index(g, pa, t) + (int)rank;
                    auto slot_of = [&](int k) {   // contributor pa + k
                        return reinterpret_cast<const float4 *>(g.part) +
                               (size_t)(k == 0 ? slot_pa : 4 * (pa + k) + (int)rank) * (BM * BN / 4);
                    };
                    // folded input norm: the 1/rms of rows [r0, r1), once per row, in the staging area
                    // (idle until the data-parallel epilogues; barriers on both sides of its use)
                    float *s_rn = reinterpret_cast<float *>(sC);
                    if (g.ss_in) {
                        for (int u = et; u < r1 - r0; u += EPI_THREADS) {
                            const int row = m_blk * (2 * BM) + (int)rank * BM + r0 + u;
                            s_rn[u] = row < g.M ? norm_rstd(g, row) : 1.f;
                        }
                        epi_bar_and(true);
                    }
                    if constexpr (EPI == EPI_QKROPE) {
                        // In chunks of up to 24 rows: (1) the contributors' partials summed in range
                        // order into shared memory, consecutive threads on consecutive rows of one
                        // float4 column group so that each warp load covers whole lines (loads
                        // scattered over many lines cost the MMAs beside them shared-memory
                        // bandwidth); (2) per (row, head) d/8 threads, thread `sub` owning
                        // first-half columns [4 sub, 4 sub + 4) and their RoPE partners d/2 on
                        constexpr int CH = 24, SROW = BN + 4;   // padded rows: no bank conflicts
                        float *s_sum = reinterpret_cast<float *>(sC + 512);   // after s_rn (<= 128 floats)
                        const int d = g.head_dim, half = d >> 1, hpt = BN / d;
                        const int tpu = half >> 2;                      // 16 (d = 128) or 8 (d = 64)
                        const int sub = et & (tpu - 1);
                        const unsigned gmask = (tpu == 16 ? 0xFFFFu : 0xFFu) << (lane & (32 - tpu));
                        #pragma unroll 1
                        for (int c0 = r0; c0 < r1; c0 += CH) {
                            const int nch = min(CH, r1 - c0);
                            #pragma unroll 1
                            for (int u = et; u < nch * (BN / 4); u += EPI_THREADS) {
                                const int rr = u % nch, c4 = (u / nch) * 4;
                                const size_t i4 = part_f4(c0 + rr, c4);
                                float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
                                for (int k0 = 0; k0 < nc; k0 += 8) {
                                    float4 x[8];
                                    #pragma unroll
                                    for (int k = 0; k < 8; ++k)
                                        if (k0 + k < nc) x[k] = __ldcg(slot_of(k0 + k) + i4);
                                    #pragma unroll
                                    for (int k = 0; k < 8; ++k) {
                                        if (k0 + k < nc) {
                                            acc.x += x[k].x; acc.y += x[k].y; acc.z += x[k].z; acc.w += x[k].w;
                                        }
                                    }
                                }
                                if constexpr (F8) {   // the e4m3 scales of row and column
                                    const int row = m_blk * (2 * BM) + (int)rank * BM + c0 + rr;
                                    float f[4] = {acc.x, acc.y, acc.z, acc.w};
                                    dq4(f, row < g.M ? g.sa[row] : 0.f, n_blk * BN + c4);
                                    acc = make_float4(f[0], f[1], f[2], f[3]);
                                }
                                *reinterpret_cast<float4 *>(s_sum + rr * SROW + c4) = acc;
                            }
                            epi_bar_and(true);
                            #pragma unroll 1
                            for (int u = et / tpu; u < nch * hpt; u += EPI_THREADS / tpu) {
                                const int rr = u / hpt, hh = u % hpt;
                                const int r = c0 + rr;
                                const int row = m_blk * (2 * BM) + (int)rank * BM + r;
                                if (row >= g.M) continue;   // same row for the unit's threads
                                const int head = (n_blk * BN) / d + hh;
                                const int jb = 4 * sub;                 // frequency index of a[0]
                                const int ca = hh * d + jb;             // first-half column inside the tile
                                const float4 sa4 = *reinterpret_cast<const float4 *>(s_sum + rr * SROW + ca);
                                const float4 sb4 = *reinterpret_cast<const float4 *>(s_sum + rr * SROW + ca + half);
                                float a[4] = {sa4.x, sa4.y, sa4.z, sa4.w}, b[4] = {sb4.x, sb4.y, sb4.z, sb4.w};
                                if (g.ss_in) {   // the folded input RMSNorm: 1/rms of this row of A
                                    const float rn = s_rn[r - r0];
                                    #pragma unroll
                                    for (int i = 0; i < 4; ++i) {
                                        a[i] *= rn;
                                        b[i] *= rn;
                                    }
                                }
                                bias4(a, n_blk * BN + ca);
                                bias4(b, n_blk * BN + ca + half);
                                __nv_bfloat16 *dst = g.C + (size_t)row * g.ldc + n_blk * BN + ca;
                                const bool is_q = head < g.nq, is_k = !is_q && head < g.nq + g.nkv;
                                if (is_q || is_k) {
                                    const bool qk_norm = g.wq != nullptr;   // the vision tower has none
                                    float rstd = 1.f;
                                    if (qk_norm) {
                                        float ss = 0.f;
                                        #pragma unroll
                                        for (int i = 0; i < 4; ++i) ss = fmaf(a[i], a[i], fmaf(b[i], b[i], ss));
                                        for (int o = 1; o < tpu; o <<= 1) ss += __shfl_xor_sync(gmask, ss, o);
                                        rstd = 1.0f / sqrtf(ss / (float)d + g.eps);
                                    }
                                    const __nv_bfloat16 *w = is_q ? g.wq : g.wk;
                                    const size_t ci = cs_at(g, row, jb);
                                    const float4 co4 = *reinterpret_cast<const float4 *>(g.cos_t + ci);
                                    const float4 si4 = *reinterpret_cast<const float4 *>(g.sin_t + ci);
                                    const float cv[4] = {co4.x, co4.y, co4.z, co4.w};
                                    const float sv[4] = {si4.x, si4.y, si4.z, si4.w};
                                    #pragma unroll
                                    for (int i = 0; i < 4; ++i) {
                                        const float ga = qk_norm ? __bfloat162float(w[jb + i]) : 1.f;
                                        const float gb = qk_norm ? __bfloat162float(w[half + jb + i]) : 1.f;
                                        const float ya = a[i] * rstd * ga;
                                        const float yb = b[i] * rstd * gb;
                                        a[i] = ya * cv[i] - yb * sv[i];
                                        b[i] = yb * cv[i] + ya * sv[i];
                                    }
                                }
                                *reinterpret_cast<uint2 *>(dst) =
                                    make_uint2(pack_bf16x2(a[0], a[1]), pack_bf16x2(a[2], a[3]));
                                *reinterpret_cast<uint2 *>(dst + half) =
                                    make_uint2(pack_bf16x2(b[0], b[1]), pack_bf16x2(b[2], b[3]));
                            }
                            epi_bar_and(true);   // s_sum is rewritten by the next chunk
                        }
                    } else {
                        // consecutive threads take consecutive rows of one float4 column group
                        constexpr int GROUPS = (EPI == EPI_SWIGLU) ? BN / 8 : BN / 4;
                        const int nr = r1 - r0;
                        const int units = nr * GROUPS;
                        for (int u = et; u < units; u += EPI_THREADS) {
                            const int r = r0 + u % nr;
                            const int c4 = (u / nr) * 4;
                            const int row = m_blk * (2 * BM) + (int)rank * BM + r;
                            if (row >= g.M) continue;
                            float4 a = make_float4(0.f, 0.f, 0.f, 0.f), b = a;
                            const size_t ia = part_f4(r, c4), ib = part_f4(r, c4 + BN / 2);
                            // partials in batches of 8 loads in flight, summed in range order
                            for (int k0 = 0; k0 < nc; k0 += 8) {
                                float4 x[8], y[8];
                                #pragma unroll
                                for (int k = 0; k < 8; ++k) {
                                    if (k0 + k < nc) {
                                        const float4 *pk = slot_of(k0 + k);
                                        x[k] = __ldcg(pk + ia);
                                        if constexpr (EPI == EPI_SWIGLU) y[k] = __ldcg(pk + ib);
                                    }
                                }
                                #pragma unroll
                                for (int k = 0; k < 8; ++k) {
                                    if (k0 + k < nc) {
                                        a.x += x[k].x; a.y += x[k].y; a.z += x[k].z; a.w += x[k].w;
                                        if constexpr (EPI == EPI_SWIGLU) {
                                            b.x += y[k].x; b.y += y[k].y; b.z += y[k].z; b.w += y[k].w;
                                        }
                                    }
                                }
                            }
                            float f[4] = {a.x, a.y, a.z, a.w};
                            float up[4] = {b.x, b.y, b.z, b.w};
                            if constexpr (F8) {
                                const float sr = g.sa[row];
                                dq4(f, sr, n_blk * BN + c4);
                                if constexpr (EPI == EPI_SWIGLU) dq4(up, sr, n_blk * BN + BN / 2 + c4);
                            }
                            if (g.ss_in) {   // the folded input RMSNorm: 1/rms of this row of A
                                const float rn = s_rn[r - r0];
                                #pragma unroll
                                for (int i = 0; i < 4; ++i) {
                                    f[i] *= rn;
                                    up[i] *= rn;
                                }
                            }
                            if constexpr (EPI != EPI_SWIGLU) bias4(f, n_blk * BN + c4);
                            if constexpr (EPI == EPI_GELU_TANH || EPI == EPI_GELU_ERF) {
                                #pragma unroll
                                for (int i = 0; i < 4; ++i) f[i] = EPI == EPI_GELU_TANH ? gelu_tanh(f[i]) : gelu_erf(f[i]);
                            }
                            int col;
                            if constexpr (EPI == EPI_SWIGLU) {
                                #pragma unroll
                                for (int i = 0; i < 4; ++i) f[i] = silu_mul(f[i], up[i]);
                                col = n_blk * (BN / 2) + c4;
                            } else {
                                col = n_blk * BN + c4;
                                if constexpr (EPI == EPI_RESIDUAL || EPI == EPI_RESIDUAL_DS) {
                                    const uint2 rv = *reinterpret_cast<const uint2 *>(g.R + (size_t)row * g.ldc + col);
                                    f[0] += bf16_lo(rv.x); f[1] += bf16_hi(rv.x); f[2] += bf16_lo(rv.y); f[3] += bf16_hi(rv.y);
                                }
                                if constexpr (EPI == EPI_RESIDUAL_DS) {
                                    int rank_ds = g.DS != nullptr ? g.vis_rank[row] : -1;
                                    if (rank_ds >= g.n_vis) rank_ds = -1;
                                    if (rank_ds >= 0) {
                                        const uint2 dv = *reinterpret_cast<const uint2 *>(g.DS + (size_t)rank_ds * g.ldc + col);
                                        f[0] = round_bf16(f[0]) + bf16_lo(dv.x); f[1] = round_bf16(f[1]) + bf16_hi(dv.x);
                                        f[2] = round_bf16(f[2]) + bf16_lo(dv.y); f[3] = round_bf16(f[3]) + bf16_hi(dv.y);
                                    }
                                }
                            }
                            uint2 o;
                            o.x = pack_bf16x2(f[0], f[1]);
                            o.y = pack_bf16x2(f[2], f[3]);
                            *reinterpret_cast<uint2 *>(g.C + (size_t)row * g.ldc + col) = o;
                            if constexpr (EPI == EPI_SWIGLU) {
                                if (g.row_amax) {
                                    const float m = fmaxf(fmaxf(fabsf(bf16_lo(o.x)), fabsf(bf16_hi(o.x))),
                                                          fmaxf(fabsf(bf16_lo(o.y)), fabsf(bf16_hi(o.y))));
                                    atomicMax(reinterpret_cast<int *>(g.row_amax + row), __float_as_int(m));
                                }
                            }
                        }
                        if constexpr (EPI != EPI_SWIGLU) {
                            if (g.ss_out) {
                                // row statistics of the rows just stored: each (row, 128-column half)
                                // re-read in column order once every epilogue warp's stores are done
                                epi_bar_and(true);
                                for (int u = et; u < nr * 2; u += EPI_THREADS) {
                                    const int r = r0 + (u >> 1), hf = u & 1;
                                    const int row = m_blk * (2 * BM) + (int)rank * BM + r;
                                    if (row >= g.M) continue;
                                    const uint4 *src = reinterpret_cast<const uint4 *>(
                                        g.C + (size_t)row * g.ldc + n_blk * BN + hf * (BN / 2));
                                    float ssum = 0.f;
                                    #pragma unroll 4
                                    for (int i = 0; i < BN / 16; ++i) {
                                        const uint4 v = __ldcg(src + i);
                                        const uint32_t w4[4] = {v.x, v.y, v.z, v.w};
                                        #pragma unroll
                                        for (int t = 0; t < 4; ++t) {
                                            const float lo = bf16_lo(w4[t]), hi = bf16_hi(w4[t]);
                                            ssum = fmaf(lo, lo, ssum);
                                            ssum = fmaf(hi, hi, ssum);
                                        }
                                    }
                                    g.ss_out[(size_t)(2 * n_blk + hf) * g.M + row] = ssum;
                                }
                            }
                        }
                    }
                    if (g.ss_in) epi_bar_and(true);   // s_rn is read no more (next tile, staging)
                }
            }
            if (et == 0) stamp(g, TR_REDUCE_DONE);
        }
        // the folded input RMSNorm: this thread's row scale, reused while the row block repeats
        int rn_blk = -1;
        float rn = 1.f;
        auto scale32 = [&](uint32_t (&v)[32]) {
            #pragma unroll
            for (int j = 0; j < 32; ++j) v[j] = __float_as_uint(__uint_as_float(v[j]) * rn);
        };
        for (int tile = pair; tile < g.dp_tiles; tile += npairs) {
            const int m_blk = tile % g.nm;
            const int n_blk = tile / g.nm;
            const int row0 = m_blk * (2 * BM) + (int)rank * BM + quarter * 32;   // the warp's first row
            const int row = row0 + lane;
            const bool live = row < g.M;
            if (g.ss_in && m_blk != rn_blk) {   // its loads fly while the MMAs finish
                rn = live ? norm_rstd(g, row) : 1.f;
                rn_blk = m_blk;
            }
            uint4 rpre[BN / 16];   // the warp's 32 rows x BN/2 residual columns, 16 bytes per lane per load
            if constexpr (EPI == EPI_RESIDUAL || EPI == EPI_RESIDUAL_DS) {
                // the residual does not depend on the accumulator: its loads fly while the MMAs finish.
                // Load i covers rows 2i, 2i + 1 of the warp (lanes 0-15, 16-31), 256 bytes each: whole
                // lines (a lane per row would touch 32 lines per load and take L1 data-path time from
                // the MMAs); the chunk loop below turns them into rows through the staging slot
                #pragma unroll
                for (int i = 0; i < BN / 16; ++i) {
                    const int rr = row0 + 2 * i + (lane >> 4);
                    rpre[i] = rr < g.M ? *(reinterpret_cast<const uint4 *>(g.R + (size_t)rr * g.ldc + n_blk * BN +
                                                                           ehalf * (BN / 2)) + (lane & 15))
                                       : make_uint4(0u, 0u, 0u, 0u);
                }
            }
            if constexpr (EPI == EPI_QKROPE) {
                // the warp's cos/sin lines, pulled into L2 while the MMAs finish: by the time the
                // accumulator is ready the streamed operands may have pushed them out
                if ((n_blk * BN) / g.head_dim < g.nq + g.nkv) {
                    const int half = g.head_dim >> 1;
                    const float *tab = ehalf ? g.sin_t : g.cos_t;   // the two warps of a quarter split them
                    if (g.cs_rows) {
                        // group of four frequencies k: the warp's 32 rows are 512 contiguous bytes
                        for (int li = lane; li < half; li += 32) {
                            const int k = li >> 2, part = li & 3;
                            if (row0 + 8 * part < g.M)
                                prefetch_l2(tab + ((size_t)k * g.cs_rows + row0 + 8 * part) * 4);
                        }
                    } else if (live) {
                        for (int off = 0; off < half; off += 32) prefetch_l2(tab + (size_t)row * half + off);
                    }
                }
            }
            if (!wait_acc()) break;
            if (et == 0) stamp(g, TR_LAST_ACC);   // overwritten per tile: the last one stays
            const uint32_t taddr = tmem_base + ((uint32_t)(quarter * 32) << 16) + (uint32_t)(acc * BN);
            if constexpr (EPI == EPI_SWIGLU) {
                float rmax = 0.f;   // largest |bf16 output| of this thread's row in the tile
                #pragma unroll 1
                for (int c = ehalf * (BN / 128); c < (ehalf + 1) * (BN / 128); ++c) {
                    uint32_t vg[32], vu[32];
                    tmem_ld32(taddr + c * 32, vg);
                    tmem_ld32(taddr + BN / 2 + c * 32, vu);
                    tmem_ld_wait();
                    dq32(vg, row, live, n_blk * BN + c * 32);
                    dq32(vu, row, live, n_blk * BN + BN / 2 + c * 32);
                    scale32(vg);
                    scale32(vu);
                    float f[32];
                    #pragma unroll
                    for (int j = 0; j < 32; ++j) {
                        const float gt = __uint_as_float(vg[j]);
                        const float up = __uint_as_float(vu[j]);
                        f[j] = silu_mul(gt, up);
                        rmax = fmaxf(rmax, fabsf(round_bf16(f[j])));
                    }
                    store_chunk_f(f, n_blk * (BN / 2) + c * 32, row0);
                }
                // non-negative floats order like their bit patterns: an integer max is exact
                if (live && g.row_amax) atomicMax(reinterpret_cast<int *>(g.row_amax + row), __float_as_int(rmax));
            } else if constexpr (EPI == EPI_QKROPE) {
                // the tile holds BN/d whole heads: q and k heads get RMSNorm over d and M-RoPE
                // (pairs j, j + d/2 both in this thread's row), v heads are stored as they are
                const int d = g.head_dim, half = d >> 1;
                const int hpt = BN / d;
                #pragma unroll 1
                for (int hh = ehalf * (hpt >> 1); hh < (ehalf + 1) * (hpt >> 1); ++hh) {
                    const int head = (n_blk * BN) / d + hh;
                    const int cb = hh * d;
                    const bool is_q = head < g.nq, is_k = !is_q && head < g.nq + g.nkv;
                    if (!is_q && !is_k) {
                        #pragma unroll 1
                        for (int c = 0; c < d / 32; ++c) {
                            uint32_t v[32];
                            tmem_ld32(taddr + cb + c * 32, v);
                            tmem_ld_wait();
                            dq32(v, row, live, n_blk * BN + cb + c * 32);
                            scale32(v);
                            bias32(v, n_blk * BN + cb + c * 32);
                            float f[32];
                            #pragma unroll
                            for (int j = 0; j < 32; ++j) f[j] = __uint_as_float(v[j]);
                            store_chunk_f(f, n_blk * BN + cb + c * 32, row0);
                        }
                        continue;
                    }
                    const bool qk_norm = g.wq != nullptr;   // the vision tower's q/k have no norm
                    float rstd = 1.f;
                    if (qk_norm) {
                        float ss = 0.f;
                        #pragma unroll 1
                        for (int c = 0; c < d / 32; ++c) {
                            uint32_t v[32];
                            tmem_ld32(taddr + cb + c * 32, v);
                            tmem_ld_wait();
                            dq32(v, row, live, n_blk * BN + cb + c * 32);
                            scale32(v);
                            bias32(v, n_blk * BN + cb + c * 32);
                            #pragma unroll
                            for (int j = 0; j < 32; ++j) ss = fmaf(__uint_as_float(v[j]), __uint_as_float(v[j]), ss);
                        }
                        rstd = 1.0f / sqrtf(ss / (float)d + g.eps);
                    }
                    const __nv_bfloat16 *w = is_q ? g.wq : g.wk;
                    #pragma unroll 1
                    for (int c = 0; c < half / 32; ++c) {
                        uint32_t va[32], vb[32];
                        tmem_ld32(taddr + cb + c * 32, va);
                        tmem_ld32(taddr + cb + half + c * 32, vb);
                        tmem_ld_wait();
                        dq32(va, row, live, n_blk * BN + cb + c * 32);
                        dq32(vb, row, live, n_blk * BN + cb + half + c * 32);
                        scale32(va);
                        scale32(vb);
                        bias32(va, n_blk * BN + cb + c * 32);
                        bias32(vb, n_blk * BN + cb + half + c * 32);
                        uint32_t oa[16], ob[16];
                        #pragma unroll
                        for (int i = 0; i < 16; ++i) oa[i] = ob[i] = 0u;   // rows past M: clipped by the store
                        if (live) {
                            #pragma unroll
                            for (int j = 0; j < 32; j += 4) {
                                // row-interleaved tables: the warp's 32 rows load 512 contiguous bytes
                                const size_t ci = cs_at(g, row, c * 32 + j);
                                const float4 co = *reinterpret_cast<const float4 *>(g.cos_t + ci);
                                const float4 si = *reinterpret_cast<const float4 *>(g.sin_t + ci);
                                const uint2 wa = qk_norm ? *reinterpret_cast<const uint2 *>(w + c * 32 + j)
                                                         : make_uint2(0x3F803F80u, 0x3F803F80u);   // bf16 1.0
                                const uint2 wb = qk_norm ? *reinterpret_cast<const uint2 *>(w + half + c * 32 + j)
                                                         : make_uint2(0x3F803F80u, 0x3F803F80u);
                                const float ga[4] = {bf16_lo(wa.x), bf16_hi(wa.x), bf16_lo(wa.y), bf16_hi(wa.y)};
                                const float gb[4] = {bf16_lo(wb.x), bf16_hi(wb.x), bf16_lo(wb.y), bf16_hi(wb.y)};
                                const float cv[4] = {co.x, co.y, co.z, co.w}, sv[4] = {si.x, si.y, si.z, si.w};
                                float ra[4], rb[4];
                                #pragma unroll
                                for (int t = 0; t < 4; ++t) {
                                    const float ya = __uint_as_float(va[j + t]) * rstd * ga[t];
                                    const float yb = __uint_as_float(vb[j + t]) * rstd * gb[t];
                                    ra[t] = ya * cv[t] - yb * sv[t];
                                    rb[t] = yb * cv[t] + ya * sv[t];
                                }
                                oa[j / 2] = pack_bf16x2(ra[0], ra[1]);
                                oa[j / 2 + 1] = pack_bf16x2(ra[2], ra[3]);
                                ob[j / 2] = pack_bf16x2(rb[0], rb[1]);
                                ob[j / 2 + 1] = pack_bf16x2(rb[2], rb[3]);
                            }
                        }
                        store_chunk(oa, n_blk * BN + cb + c * 32, row0);
                        store_chunk(ob, n_blk * BN + cb + half + c * 32, row0);
                    }
                }
            } else {
                int rank_ds = -1;
                if constexpr (EPI == EPI_RESIDUAL_DS) {
                    if (live && g.DS != nullptr) {
                        rank_ds = g.vis_rank[row];
                        if (rank_ds >= g.n_vis) rank_ds = -1;  // count mismatch is reported by the rank scan
                    }
                }
                float ssum = 0.f;   // sum of squares of this thread's 128 bf16 outputs (ss_out)
                #pragma unroll
                for (int cc = 0; cc < BN / 64; ++cc) {
                    const int c = ehalf * (BN / 64) + cc;
                    const int col = n_blk * BN + c * 32;
                    uint32_t v[32];
                    tmem_ld32(taddr + c * 32, v);
                    tmem_ld_wait();
                    dq32(v, row, live, col);
                    scale32(v);
                    bias32(v, col);
                    float f[32];
                    #pragma unroll
                    for (int j = 0; j < 32; ++j) f[j] = __uint_as_float(v[j]);
                    if constexpr (EPI == EPI_GELU_TANH || EPI == EPI_GELU_ERF) {
                        #pragma unroll
                        for (int j = 0; j < 32; ++j) f[j] = EPI == EPI_GELU_TANH ? gelu_tanh(f[j]) : gelu_erf(f[j]);
                    }
                    uint4 rrow[4];   // this row's residual in the chunk's 32 columns
                    if constexpr (EPI == EPI_RESIDUAL || EPI == EPI_RESIDUAL_DS) {
                        {
                            // the lanes holding the chunk's 16-byte units write them into the staging slot
                            // this chunk's output will use (same swizzle), then each lane reads its row
                            uint8_t *slot = cslots + (cstores & 1) * C_SLOT_BYTES;
                            if (lane == 0) bulk_wait_read<1>();
                            __syncwarp();
                            if (((lane & 15) >> 2) == cc) {
                                const int u = lane & 3;
                                #pragma unroll
                                for (int i = 0; i < BN / 16; ++i) {
                                    const int rr = 2 * i + (lane >> 4);
                                    *reinterpret_cast<uint4 *>(slot + rr * 64 + ((u ^ ((rr >> 1) & 3)) * 16)) = rpre[i];
                                }
                            }
                            __syncwarp();
                            #pragma unroll
                            for (int q = 0; q < 4; ++q)
                                rrow[q] = *reinterpret_cast<const uint4 *>(slot + lane * 64 + ((q ^ ((lane >> 1) & 3)) * 16));
                            __syncwarp();   // read before store_chunk writes this chunk's output over it
                        }
                    }
                    if (live) {
                        if constexpr (EPI == EPI_RESIDUAL || EPI == EPI_RESIDUAL_DS) {
                            #pragma unroll
                            for (int i = 0; i < 4; ++i) {
                                const uint4 rv = rrow[i];
                                f[8 * i + 0] += bf16_lo(rv.x); f[8 * i + 1] += bf16_hi(rv.x);
                                f[8 * i + 2] += bf16_lo(rv.y); f[8 * i + 3] += bf16_hi(rv.y);
                                f[8 * i + 4] += bf16_lo(rv.z); f[8 * i + 5] += bf16_hi(rv.z);
                                f[8 * i + 6] += bf16_lo(rv.w); f[8 * i + 7] += bf16_hi(rv.w);
                            }
                        }
                        if constexpr (EPI == EPI_RESIDUAL_DS) {
                            if (rank_ds >= 0) {
                                float ds[32];
                                load_row32(g.DS + (size_t)rank_ds * g.ldc + col, ds);
                                #pragma unroll
                                for (int j = 0; j < 32; ++j) f[j] = round_bf16(f[j]) + ds[j];
                            }
                        }
                    }
                    uint32_t pk[16];
                    #pragma unroll
                    for (int i = 0; i < 16; ++i) pk[i] = pack_bf16x2(f[2 * i], f[2 * i + 1]);
                    if (g.ss_out) {   // squares of the stored bf16 values, in column order
                        #pragma unroll
                        for (int i = 0; i < 16; ++i) {
                            const float lo = bf16_lo(pk[i]), hi = bf16_hi(pk[i]);
                            ssum = fmaf(lo, lo, ssum);
                            ssum = fmaf(hi, hi, ssum);
                        }
                    }
                    store_chunk(pk, col, row0);
                }
                if (g.ss_out && live) g.ss_out[(size_t)(2 * n_blk + ehalf) * g.M + row] = ssum;
            }
            release_acc();
        }
        if (lane == 0) bulk_wait_all();   // this warp's tile stores have landed
        if (et == 0) stamp(g, TR_DP_EPI_DONE);
    }

    tc_fence_before();
    cluster_sync();   // the peer no longer reads this CTA's shared memory or signals its barriers
    if (threadIdx.x == 0) {
        stamp(g, TR_END);
        if (g.sk_pairs) {
            // the last CTA of the launch records its epoch; every CTA has read it long before
            const uint32_t epoch = sk_epoch(g);
            __threadfence();
            if (atomicAdd(g.ctrl + 1, 1u) == gridDim.x - 1) {
                g.ctrl[1] = 0u;
                __threadfence();
                st_release(g.ctrl, epoch);
            }
        }
    }
    if (warp == 1) {
        tc_fence_after();
        tmem_dealloc_pair(tmem_base, 512);
    }
}

PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
    static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
    if (!fn) {
        void *p = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) ==
                cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
    }
    return fn;
}

// Output map for the epilogue's tile stores: bf16 [rows, ld] row-major, boxes of 32 x 32, no swizzle.
// The epilogue's output map: 32 x 32 boxes staged in 64-byte-swizzled shared memory.
bool make_tmap_c(CUtensorMap *m, void *ptr, uint64_t rows, uint64_t ld) {
    PFN_cuTensorMapEncodeTiled_v12000 fn = encode_fn();
    if (!fn || rows == 0 || ld == 0 || (ld * 2) % 16 != 0 || (reinterpret_cast<uintptr_t>(ptr) & 15)) return false;
    cuuint64_t dims[2] = {ld, rows};
    cuuint64_t strides[1] = {ld * 2};
    cuuint32_t box[2] = {32, 32};
    cuuint32_t estr[2] = {1, 1};
    CUresult r = fn(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, ptr, dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                    CU_TENSOR_MAP_SWIZZLE_64B, CU_TENSOR_MAP_L2_PROMOTION_NONE,
                    CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS;
}

template <int EPI, bool F8>
cudaError_t launch_epi(const GemmPlan &p, cudaStream_t stream) {
    // per device: the shared-memory opt-in and the number of co-resident pairs
    static std::atomic<int> max_pairs_of[kMaxDevices];
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return cudaErrorInvalidDevice;
    int max_pairs = max_pairs_of[dev].load();
    cudaLaunchAttribute attr[2];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = 2;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    if (max_pairs == 0) {
        cudaError_t e = cudaFuncSetAttribute(gemm_tcgen05_kernel<EPI, F8>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                             SMEM_BYTES);
        if (e != cudaSuccess) return e;
        cudaLaunchConfig_t q = {};
        q.gridDim = dim3(2 * (p.num_sms / 2 > 0 ? p.num_sms / 2 : 1));
        q.blockDim = dim3(GEMM_THREADS);
        q.dynamicSmemBytes = SMEM_BYTES;
        q.attrs = attr;
        q.numAttrs = 1;
        int n = 0;
        e = cudaOccupancyMaxActiveClusters(&n, gemm_tcgen05_kernel<EPI, F8>, &q);
        if (e != cudaSuccess) return e;
        if (n <= 0) return cudaErrorInvalidConfiguration;
        max_pairs = n;
        max_pairs_of[dev].store(n);
    }
    GemmArgs g;
    g.M = p.M; g.N = p.N; g.K = p.K;
    g.nm = (p.M + 2 * BM - 1) / (2 * BM);
    g.nn = p.N / BN;
    g.nk = F8 ? (p.K + BK8 - 1) / BK8 : (p.K + BK - 1) / BK;
    g.sa = p.sa; g.sw = p.sw;
    g.row_amax = p.row_amax;
    g.w_static = p.w_static ? 1 : 0;
    g.C = p.C; g.ldc = p.ldc; g.R = p.R; g.DS = p.DS; g.vis_rank = p.vis_rank; g.n_vis = p.n_vis;
    g.status = p.status;
    g.wq = p.wq; g.wk = p.wk; g.cos_t = p.cos_t; g.sin_t = p.sin_t; g.cs_rows = p.cs_rows;
    g.head_dim = p.head_dim; g.nq = p.nq; g.nkv = p.nkv; g.eps = p.eps;
    g.trace = p.trace;
    g.ss_in = p.ss_in;
    g.ss_out = p.ss_out;
    g.norm_eps = p.norm_eps;
    g.bias = p.bias;
    const int tiles = g.nm * g.nn;
    int pairs = p.num_sms / 2 < max_pairs ? p.num_sms / 2 : max_pairs;   // all pairs co-resident
    if (pairs < 1) pairs = 1;
    // full waves data-parallel; the k-blocks of a partial last wave spread over all pairs (stream-K),
    // at least kMinStreamKBlocks per pair; when that leaves one tile per pair it stays data-parallel.
    // The split is kept only where it shortens the launch (in k-block times): the pair's share of
    // the tail plus the partial exchange (hidden behind the data-parallel tiles when there are
    // some, exposed when the tail is all there is) against one more whole tile; long launches
    // (kSkMaxFullWaves) run unsplit.
    const int left = tiles % pairs;
    int sk_pairs = 0;
    if (p.part && p.flags && left) {
        const long long work = (long long)left * g.nk;
        long long ps = work / kMinStreamKBlocks;
        if (ps > pairs) ps = pairs;
        if (ps > EPI_THREADS) ps = EPI_THREADS;   // one polling thread per contributor
        if (ps > left) {
            const long long full = tiles / pairs;
            const long long sk_cost = full * g.nk + (work + ps - 1) / ps + (full ? kSkFixupHidden : kSkFixupExposed);
            if (sk_cost < (full + 1) * g.nk && full < kSkMaxFullWaves) sk_pairs = (int)ps;
        }
    }
    g.sk_pairs = sk_pairs;
    g.sk_work = (long long)left * g.nk;
    g.dp_tiles = sk_pairs ? tiles - left : tiles;
    g.part = p.part;
    g.flags = p.flags;
    g.ctrl = p.flags ? p.flags + p.num_sms : nullptr;
    const int grid_pairs = g.dp_tiles >= pairs ? pairs : (sk_pairs > g.dp_tiles ? sk_pairs : g.dp_tiles);
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(2 * grid_pairs);
    cfg.blockDim = dim3(GEMM_THREADS);
    cfg.dynamicSmemBytes = SMEM_BYTES;
    cfg.stream = stream;
    attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[1].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 2;
    CUtensorMap tmC;
    if (!make_tmap_c(&tmC, p.C, (uint64_t)p.M, (uint64_t)p.ldc)) return cudaErrorInvalidValue;
    return cudaLaunchKernelEx(&cfg, gemm_tcgen05_kernel<EPI, F8>, *p.tmA, *p.tmW, tmC, g);
}

}  // namespace

bool make_tmap_rows(CUtensorMap *m, const void *ptr, uint64_t rows, uint64_t cols, uint32_t box_rows) {
    PFN_cuTensorMapEncodeTiled_v12000 fn = encode_fn();
    if (!fn || rows == 0 || cols == 0 || (cols * 2) % 16 != 0 || (reinterpret_cast<uintptr_t>(ptr) & 15))
        return false;
    cuuint64_t dims[2] = {cols, rows};
    cuuint64_t strides[1] = {cols * 2};
    cuuint32_t box[2] = {(cuuint32_t)BK, box_rows};
    cuuint32_t estr[2] = {1, 1};
    CUresult r = fn(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void *>(ptr), dims, strides, box, estr,
                    CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                    CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS;
}

bool make_tmap_rows_e4m3(CUtensorMap *m, const void *ptr, uint64_t rows, uint64_t cols, uint32_t box_rows) {
    PFN_cuTensorMapEncodeTiled_v12000 fn = encode_fn();
    if (!fn || rows == 0 || cols == 0 || cols % 16 != 0 || (reinterpret_cast<uintptr_t>(ptr) & 15)) return false;
    cuuint64_t dims[2] = {cols, rows};
    cuuint64_t strides[1] = {cols};
    cuuint32_t box[2] = {(cuuint32_t)BK8, box_rows};
    cuuint32_t estr[2] = {1, 1};
    CUresult r = fn(m, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, const_cast<void *>(ptr), dims, strides, box, estr,
                    CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                    CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS;
}

int gemm_box_rows_a() { return BM; }
// Stream-K partials: two 128 x 256 fp32 slots per CTA (a range covers parts of at most two tiles),
// then one release flag per CTA.
size_t gemm_flags_offset(int num_sms) { return (size_t)2 * num_sms * BM * BN * sizeof(float) + 256; }
// then the launch epoch and a finished-CTA counter
size_t gemm_workspace_bytes(int num_sms) { return gemm_flags_offset(num_sms) + (size_t)num_sms * 4 + 8; }
int gemm_box_rows_w() { return BN / 2; }

namespace {
thread_local unsigned long long *t_trace_next = nullptr;
}
void gemm_trace_next(unsigned long long *trace) { t_trace_next = trace; }

cudaError_t launch_gemm(const GemmPlan &p_in, cudaStream_t stream) {
    if (p_in.M <= 0) return cudaSuccess;
    GemmPlan p = p_in;
    if (t_trace_next) {
        p.trace = t_trace_next;
        t_trace_next = nullptr;
    }
    if (p.epi == EPI_QKROPE &&
        ((p.head_dim != 64 && p.head_dim != 128) || (!p.wq != !p.wk) || !p.cos_t || !p.sin_t ||
         (p.cs_rows && p.cs_rows < p.M)))
        return cudaErrorInvalidValue;
    // a bias is read 32 columns at a time from 16-byte-aligned rows
    if (p.bias && (p.epi == EPI_SWIGLU || (reinterpret_cast<uintptr_t>(p.bias) & 15))) return cudaErrorInvalidValue;
    // row statistics come in slots of 128 columns; only the stored (not SwiGLU) outputs emit them
    if ((p.ss_in && p.K % 128) || (p.ss_out && (p.N % 128 || p.epi == EPI_SWIGLU || p.epi == EPI_QKROPE)))
        return cudaErrorInvalidValue;
    if (p.fp8) {
        // the scales are read as float4 groups of 4 columns
        if (!p.sa || !p.sw || (reinterpret_cast<uintptr_t>(p.sw) & 15)) return cudaErrorInvalidValue;
        switch (p.epi) {
            case EPI_STORE: return launch_epi<EPI_STORE, true>(p, stream);
            case EPI_RESIDUAL: return launch_epi<EPI_RESIDUAL, true>(p, stream);
            case EPI_SWIGLU: return launch_epi<EPI_SWIGLU, true>(p, stream);
            case EPI_RESIDUAL_DS: return launch_epi<EPI_RESIDUAL_DS, true>(p, stream);
            case EPI_QKROPE: return launch_epi<EPI_QKROPE, true>(p, stream);
            default: return cudaErrorInvalidValue;
        }
    }
    switch (p.epi) {
        case EPI_STORE: return launch_epi<EPI_STORE, false>(p, stream);
        case EPI_RESIDUAL: return launch_epi<EPI_RESIDUAL, false>(p, stream);
        case EPI_SWIGLU: return launch_epi<EPI_SWIGLU, false>(p, stream);
        case EPI_RESIDUAL_DS: return launch_epi<EPI_RESIDUAL_DS, false>(p, stream);
        case EPI_QKROPE: return launch_epi<EPI_QKROPE, false>(p, stream);
        case EPI_GELU_TANH: return launch_epi<EPI_GELU_TANH, false>(p, stream);
        case EPI_GELU_ERF: return launch_epi<EPI_GELU_ERF, false>(p, stream);
        default: return cudaErrorInvalidValue;
    }
}

}  // namespace h3
