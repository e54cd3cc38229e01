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
// Design (one CTA per SM, persistent over 128 x 256 output tiles):
//   warp 0     TMA producer: A tile 128 x 64 and W tile 256 x 64 (bf16, 128-byte
//              swizzle) per k-block into a 4-stage shared-memory ring
//   warp 1     allocates 512 TMEM columns (two 128 x 256 fp32 accumulators) and
//              issues tcgen05.mma (M=128, N=256, K=16) from one thread
//   warps 2-5  epilogue: tcgen05.ld of their 32 TMEM lanes (= 32 output rows),
//              fused element-wise op, bf16 stores; overlaps the next tile's MMAs
// Every wait is bounded; on time-out the CTA records ST_TIMEOUT, drains its
// in-flight copies and MMAs, frees TMEM and exits.
#include <cudaTypedefs.h>

#include "common.cuh"
#include "kernels.h"

namespace h3 {

namespace {

constexpr int BM = 128, BN = 256, BK = 64, STAGES = 4;
constexpr int A_BYTES = BM * BK * 2;             // 16 KB
constexpr int B_BYTES = BN * BK * 2;             // 32 KB
constexpr int STAGE_BYTES = A_BYTES + B_BYTES;   // 48 KB
constexpr int GEMM_THREADS = 192;
constexpr int SMEM_BYTES = 1024 + STAGES * STAGE_BYTES + 256;

struct GemmArgs {
    int M, N, K;
    int nm, nn, nk;
    __nv_bfloat16 *C;
    int ldc;
    const __nv_bfloat16 *R;
    const __nv_bfloat16 *DS;
    const int32_t *vis_rank;
    int n_vis;
    int32_t *status;
};

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

__device__ __forceinline__ void store_row32(__nv_bfloat16 *p, const float (&f)[32]) {
    uint4 *q = reinterpret_cast<uint4 *>(p);
    #pragma unroll
    for (int i = 0; i < 4; ++i) {
        uint4 v;
        v.x = pack_bf16x2(f[8 * i + 0], f[8 * i + 1]);
        v.y = pack_bf16x2(f[8 * i + 2], f[8 * i + 3]);
        v.z = pack_bf16x2(f[8 * i + 4], f[8 * i + 5]);
        v.w = pack_bf16x2(f[8 * i + 6], f[8 * i + 7]);
        q[i] = v;
    }
}

template <int EPI>
__global__ void __launch_bounds__(GEMM_THREADS, 1)
    gemm_tcgen05_kernel(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB,
                        const GemmArgs g) {
    extern __shared__ uint8_t smem_raw[];
    uint8_t *smem = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    uint8_t *sA = smem;
    uint8_t *sB = smem + STAGES * A_BYTES;
    uint64_t *full = reinterpret_cast<uint64_t *>(sB + STAGES * B_BYTES);
    uint64_t *empty = full + STAGES;
    uint64_t *acc_full = empty + STAGES;
    uint64_t *acc_empty = acc_full + 2;
    uint64_t *drain = acc_empty + 2;
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(drain + 1);
    volatile int *abort_flag = reinterpret_cast<volatile int *>(tmem_slot + 1);

    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;

    if (threadIdx.x == 0) {
        for (int s = 0; s < STAGES; ++s) {
            mbar_init(&full[s], 1);
            mbar_init(&empty[s], 1);
        }
        for (int a = 0; a < 2; ++a) {
            mbar_init(&acc_full[a], 1);
            mbar_init(&acc_empty[a], 4);
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
        tmem_alloc(tmem_slot, 512);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem_base = *tmem_slot;

    const int num_tiles = g.nm * g.nn;

    if (warp == 0) {
        if (lane == 0) {
            int stage = 0;
            uint32_t phase = 0;
            uint32_t issued[STAGES];
            #pragma unroll
            for (int s = 0; s < STAGES; ++s) issued[s] = 0;
            bool ok = true;
            for (int tile = blockIdx.x; ok && tile < num_tiles; tile += gridDim.x) {
                const int m0 = (tile % g.nm) * BM;
                const int n0 = (tile / g.nm) * BN;
                for (int kb = 0; kb < g.nk; ++kb) {
                    if (!mbar_wait(&empty[stage], phase ^ 1u, abort_flag)) { ok = false; break; }
                    mbar_arrive_expect_tx(&full[stage], STAGE_BYTES);
                    tma_load_2d(sA + stage * A_BYTES, &tmA, &full[stage], kb * BK, m0);
                    tma_load_2d(sB + stage * B_BYTES, &tmB, &full[stage], kb * BK, n0);
                    ++issued[stage];
                    if (++stage == STAGES) { stage = 0; phase ^= 1u; }
                }
            }
            if (!ok) {
                report(g.status, ST_TIMEOUT);
                *abort_flag = 1;
                // wait (bounded) for the copies still in flight into the ring
                const int never = 0;
                for (int s = 0; s < STAGES; ++s)
                    if (issued[s]) mbar_wait(&full[s], (issued[s] - 1u) & 1u, &never);
            }
        }
    } else if (warp == 1) {
        if (lane == 0) {
            constexpr uint32_t idesc = umma_idesc_bf16(BM, BN);
            int stage = 0;
            uint32_t phase = 0;
            int acc = 0;
            uint32_t acc_phase = 0;
            bool ok = true;
            for (int tile = blockIdx.x; ok && tile < num_tiles; tile += gridDim.x) {
                if (!mbar_wait(&acc_empty[acc], acc_phase ^ 1u, abort_flag)) { ok = false; break; }
                tc_fence_after();
                const uint32_t d_tmem = tmem_base + (uint32_t)(acc * BN);
                for (int kb = 0; kb < g.nk; ++kb) {
                    if (!mbar_wait(&full[stage], phase, abort_flag)) { ok = false; break; }
                    tc_fence_after();
                    const uint32_t a_base = smem_u32(sA + stage * A_BYTES);
                    const uint32_t b_base = smem_u32(sB + stage * B_BYTES);
                    #pragma unroll
                    for (int kk = 0; kk < BK / 16; ++kk)
                        umma_bf16(d_tmem, sdesc_sw128(a_base + kk * 32), sdesc_sw128(b_base + kk * 32), idesc,
                                  (kb | kk) != 0);
                    umma_commit(&empty[stage]);
                    if (++stage == STAGES) { stage = 0; phase ^= 1u; }
                }
                if (!ok) break;
                umma_commit(&acc_full[acc]);
                acc ^= 1;
                if (acc == 0) acc_phase ^= 1u;
            }
            if (!ok) {
                report(g.status, ST_TIMEOUT);
                *abort_flag = 1;
            }
            // every MMA issued by this thread has completed once `drain` flips
            umma_commit(drain);
            const int never = 0;
            mbar_wait(drain, 0, &never);
        }
    } else {
        // epilogue: warp w reads TMEM lanes 32*(w%4) .. +31 = tile rows of the same range
        const int quarter = warp & 3;
        int acc = 0;
        uint32_t acc_phase = 0;
        for (int tile = blockIdx.x; tile < num_tiles; tile += gridDim.x) {
            const int m_blk = tile % g.nm;
            const int n_blk = tile / g.nm;
            bool ok = mbar_wait(&acc_full[acc], acc_phase, abort_flag);
            ok = __all_sync(0xffffffffu, ok);
            if (!ok) {
                if (lane == 0) {
                    report(g.status, ST_TIMEOUT);
                    *abort_flag = 1;
                }
                break;
            }
            tc_fence_after();
            const int row = m_blk * BM + quarter * 32 + lane;
            const bool live = row < g.M;
            const uint32_t taddr = tmem_base + ((uint32_t)(quarter * 32) << 16) + (uint32_t)(acc * BN);
            if constexpr (EPI == EPI_SWIGLU) {
                #pragma unroll 1
                for (int c = 0; c < BN / 64; ++c) {
                    uint32_t vg[32], vu[32];
                    tmem_ld32(taddr + c * 32, vg);
                    tmem_ld32(taddr + BN / 2 + c * 32, vu);
                    tmem_ld_wait();
                    if (live) {
                        float f[32];
                        #pragma unroll
                        for (int j = 0; j < 32; ++j) {
                            const float gt = __uint_as_float(vg[j]);
                            const float up = __uint_as_float(vu[j]);
                            f[j] = gt / (1.0f + expf(-gt)) * up;
                        }
                        store_row32(g.C + (size_t)row * g.ldc + n_blk * (BN / 2) + c * 32, f);
                    }
                }
            } else {
                int rank = -1;
                if constexpr (EPI == EPI_RESIDUAL_DS) {
                    if (live && g.DS != nullptr) {
                        rank = g.vis_rank[row];
                        if (rank >= g.n_vis) rank = -1;  // count mismatch is reported by the rank scan
                    }
                }
                #pragma unroll 1
                for (int c = 0; c < BN / 32; ++c) {
                    uint32_t v[32];
                    tmem_ld32(taddr + c * 32, v);
                    tmem_ld_wait();
                    if (live) {
                        const int col = n_blk * BN + c * 32;
                        float f[32];
                        #pragma unroll
                        for (int j = 0; j < 32; ++j) f[j] = __uint_as_float(v[j]);
                        if constexpr (EPI == EPI_RESIDUAL || EPI == EPI_RESIDUAL_DS) {
                            float r[32];
                            load_row32(g.R + (size_t)row * g.ldc + col, r);
                            #pragma unroll
                            for (int j = 0; j < 32; ++j) f[j] += r[j];
                        }
                        if constexpr (EPI == EPI_RESIDUAL_DS) {
                            if (rank >= 0) {
                                float ds[32];
                                load_row32(g.DS + (size_t)rank * g.ldc + col, ds);
                                #pragma unroll
                                for (int j = 0; j < 32; ++j) f[j] = round_bf16(f[j]) + ds[j];
                            }
                        }
                        store_row32(g.C + (size_t)row * g.ldc + col, f);
                    }
                }
            }
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(&acc_empty[acc]);
            acc ^= 1;
            if (acc == 0) acc_phase ^= 1u;
        }
    }

    __syncthreads();
    if (warp == 1) {
        tc_fence_after();
        tmem_dealloc(tmem_base, 512);
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

template <int EPI>
cudaError_t launch_epi(const GemmPlan &p, cudaStream_t stream) {
    static bool attr_set = false;
    if (!attr_set) {
        cudaError_t e = cudaFuncSetAttribute(gemm_tcgen05_kernel<EPI>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                             SMEM_BYTES);
        if (e != cudaSuccess) return e;
        attr_set = true;
    }
    GemmArgs g;
    g.M = p.M; g.N = p.N; g.K = p.K;
    g.nm = (p.M + BM - 1) / BM;
    g.nn = p.N / BN;
    g.nk = (p.K + BK - 1) / BK;
    g.C = p.C; g.ldc = p.ldc; g.R = p.R; g.DS = p.DS; g.vis_rank = p.vis_rank; g.n_vis = p.n_vis;
    g.status = p.status;
    const int tiles = g.nm * g.nn;
    const int grid = tiles < p.num_sms ? tiles : p.num_sms;
    gemm_tcgen05_kernel<EPI><<<grid, GEMM_THREADS, SMEM_BYTES, stream>>>(*p.tmA, *p.tmW, g);
    return cudaGetLastError();
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

int gemm_box_rows_a() { return BM; }
int gemm_box_rows_w() { return BN; }

cudaError_t launch_gemm(const GemmPlan &p, cudaStream_t stream) {
    if (p.M <= 0) return cudaSuccess;
    switch (p.epi) {
        case EPI_STORE: return launch_epi<EPI_STORE>(p, stream);
        case EPI_RESIDUAL: return launch_epi<EPI_RESIDUAL>(p, stream);
        case EPI_SWIGLU: return launch_epi<EPI_SWIGLU>(p, stream);
        case EPI_RESIDUAL_DS: return launch_epi<EPI_RESIDUAL_DS>(p, stream);
        default: return cudaErrorInvalidValue;
    }
}

}  // namespace h3
