// Token-embedding gather, visual-row ranks for the DeepStack add, and the
// gate/up weight interleave.
//
// Page "vllm-omni vllm_omni/diffusion/models/minimax_h3/encoder.py":
// embed_tokens (F.embedding) and _deepstack_process, whose boolean-mask
// assignment gives row j of the DeepStack features to the j-th visual row.
#include "common.cuh"
#include "kernels.h"

namespace h3 {

namespace {

// One warp per token: copy the table row with 16-byte accesses (bit-exact).
__global__ void __launch_bounds__(256) embed_kernel(const int32_t *__restrict__ ids,
                                                    const bf16 *__restrict__ table, int vocab, int hidden,
                                                    bf16 *out, int S, int32_t *status) {
    pdl_trigger();
    pdl_wait();
    const int lane = threadIdx.x & 31;
    const int row = blockIdx.x * 8 + (threadIdx.x >> 5);
    if (row >= S) return;
    const int id = ids[row];
    const bool ok = id >= 0 && id < vocab;
    if (!ok && lane == 0) report(status, ST_BOUNDS);
    const int nvec = hidden >> 3;
    const uint4 *src = reinterpret_cast<const uint4 *>(table + (size_t)(ok ? id : 0) * hidden);
    uint4 *dst = reinterpret_cast<uint4 *>(out + (size_t)row * hidden);
    for (int v = lane; v < nvec; v += 32) dst[v] = ok ? src[v] : make_uint4(0, 0, 0, 0);
}

// Single CTA exclusive scan of the visual mask.
constexpr int SCAN_THREADS = 1024;
__global__ void __launch_bounds__(SCAN_THREADS) vis_rank_kernel(const uint8_t *__restrict__ mask, int S,
                                                                int n_vis, int32_t *rank, int32_t *status) {
    __shared__ int warp_tot[SCAN_THREADS / 32];
    __shared__ int carry;
    pdl_trigger();
    pdl_wait();
    const int lane = threadIdx.x & 31;
    const int warp = threadIdx.x >> 5;
    if (threadIdx.x == 0) carry = 0;
    __syncthreads();
    for (int base = 0; base < S; base += SCAN_THREADS) {
        const int i = base + threadIdx.x;
        const int m = (i < S && mask[i]) ? 1 : 0;
        int incl = m;
        #pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const int t = __shfl_up_sync(0xffffffffu, incl, o);
            if (lane >= o) incl += t;
        }
        if (lane == 31) warp_tot[warp] = incl;
        __syncthreads();
        if (warp == 0) {
            int w = warp_tot[lane];
            #pragma unroll
            for (int o = 1; o < 32; o <<= 1) {
                const int t = __shfl_up_sync(0xffffffffu, w, o);
                if (lane >= o) w += t;
            }
            warp_tot[lane] = w;  // inclusive prefix over warps
        }
        __syncthreads();
        const int before = carry + (warp > 0 ? warp_tot[warp - 1] : 0) + incl - m;
        if (i < S) rank[i] = m ? before : -1;
        __syncthreads();
        if (threadIdx.x == 0) carry += warp_tot[SCAN_THREADS / 32 - 1];
        __syncthreads();
    }
    if (threadIdx.x == 0 && carry != n_vis) report(status, ST_SHAPE);
}

}  // namespace

cudaError_t launch_embed(const int32_t *ids, const bf16 *table, int vocab, int hidden, bf16 *out, int S,
                         int32_t *status, cudaStream_t st) {
    if (S <= 0) return cudaSuccess;
    cudaLaunchAttribute at[1];
    cudaLaunchConfig_t cfg = pdl_config(dim3((S + 7) / 8), dim3(256), 0, st, at);
    return cudaLaunchKernelEx(&cfg, embed_kernel, ids, table, vocab, hidden, out, S, status);
}

cudaError_t launch_vis_rank(const uint8_t *mask, int S, int n_vis, int32_t *rank, int32_t *status,
                            cudaStream_t st) {
    if (S <= 0) return cudaSuccess;
    cudaLaunchAttribute at[1];
    cudaLaunchConfig_t cfg = pdl_config(dim3(1), dim3(SCAN_THREADS), 0, st, at);
    return cudaLaunchKernelEx(&cfg, vis_rank_kernel, mask, S, n_vis, rank, status);
}

// which = 0: gate rows -> packed rows [256b, 256b+128); which = 1: up rows -> [256b+128, 256b+256).
cudaError_t pack_gate_up_rows(const bf16 *src, bf16 *W, int I, int K, int which, cudaMemcpyKind kind,
                              cudaStream_t st) {
    const size_t blk = (size_t)128 * K * sizeof(bf16);
    char *dst = reinterpret_cast<char *>(W) + (which ? blk : 0);
    return cudaMemcpy2DAsync(dst, 2 * blk, src, blk, blk, (size_t)I / 128, kind, st);
}

int device_num_sms() {
    int dev = 0, n = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return 0;
    if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) return 0;
    return n;
}

}  // namespace h3
