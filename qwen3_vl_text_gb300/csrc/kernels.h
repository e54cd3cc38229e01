// Host-side launchers of the device kernels (internal to the library).
#pragma once

#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

namespace h3 {

using bf16 = __nv_bfloat16;

enum { EPI_STORE = 0, EPI_RESIDUAL = 1, EPI_SWIGLU = 2, EPI_RESIDUAL_DS = 3, EPI_QKROPE = 4,
       EPI_GELU_TANH = 5, EPI_GELU_ERF = 6 };

constexpr int kMaxSeqs = 1024;
constexpr int kMaxDevices = 64;   // per-device launch caches
constexpr int kMaxHalfDim = 64;

// ---- projection GEMM (gemm.cu)
struct GemmPlan {
    const CUtensorMap *tmA;   // A [rows >= M, K], box 128 x 64
    const CUtensorMap *tmW;   // W [N, K], box 256 x 64
    int M, N, K, epi;
    bf16 *C;
    int ldc;
    const bf16 *R;
    const bf16 *DS;
    const int32_t *vis_rank;
    int n_vis;
    int32_t *status;
    int num_sms;
    float *part;        // stream-K workspace: 2 x num_sms x 128 x 256 fp32 partials (NULL: no split)
    uint32_t *flags;    // num_sms release flags, zero-filled once before first use
    // EPI_QKROPE: per-head RMSNorm of the q and k heads, then M-RoPE with the fp32 tables
    const bf16 *wq = nullptr, *wk = nullptr;
    const float *cos_t = nullptr, *sin_t = nullptr;   // [M, head_dim/2], or row-interleaved:
    int cs_rows = 0;   // > 0: element (row, j) at ((j/4) * cs_rows + row) * 4 + j%4, cs_rows >= M
    int head_dim = 0, nq = 0, nkv = 0;
    float eps = 0.f;
    unsigned long long *trace = nullptr;   // optional per-CTA phase timeline (11 stamps per CTA)
    // e4m3 operands (tensor maps from make_tmap_rows_e4m3): C = (A * sa[row]) (W * sw[col])^T,
    // sa [M] and sw [N] fp32 (sw 16-byte aligned)
    bool fp8 = false;
    const float *sa = nullptr, *sw = nullptr;
    // EPI_SWIGLU (optional): each row's largest |bf16 output| merged with an integer atomic max
    float *row_amax = nullptr;
    // true when no kernel earlier in the stream writes W (model weights): the weight half of the
    // first ring stages is fetched before waiting for the previous kernel
    bool w_static = false;
    // RMSNorm folded into the projection (its weight pre-multiplied into W's columns).
    // ss_in [K/128][M] (optional): per-row sums of squares of A over column slots of 128; every
    // accumulator row is scaled by 1/sqrt(sum / K + norm_eps) before the epilogue.  ss_out
    // [N/128][M] (optional; EPI_STORE, EPI_RESIDUAL, EPI_RESIDUAL_DS): the same sums over this
    // GEMM's bf16 output, for the next projection.
    const float *ss_in = nullptr;
    float *ss_out = nullptr;
    float norm_eps = 0.f;
    // bias [N] (optional; every epilogue but SWIGLU): added to the accumulator before the fused
    // op.  EPI_GELU_TANH / EPI_GELU_ERF store gelu(acc + bias).  EPI_QKROPE with wq = wk = NULL:
    // no per-head norm, M-RoPE only (the vision tower's attention).
    const bf16 *bias = nullptr;
};
// ss[s * rows + r] = sum of x[r][c]^2 over the 128 columns of slot s, accumulated in fp32 in
// column order (x row-major [rows, cols], cols % 128 == 0).
cudaError_t launch_row_sumsq(const bf16 *x, int rows, int cols, float *ss, cudaStream_t st);
// W[r][k] = bf16(W[r][k] * gamma[k]) for rows r in [r0, r1) (with blk > 0: only rows whose
// block r / blk has parity `parity`), W row-major [*, cols], cols % 8 == 0.
cudaError_t launch_fold_cols(bf16 *W, int cols, const bf16 *gamma, int r0, int r1, int blk, int parity,
                             cudaStream_t st);
// Tensor map of a row-major bf16 matrix [rows, cols] read in boxes of
// box_rows x 64 with 128-byte swizzle.  False if the driver refuses it.
bool make_tmap_rows(CUtensorMap *m, const void *ptr, uint64_t rows, uint64_t cols, uint32_t box_rows);
// The same for an e4m3 matrix (one byte per element): boxes of box_rows x 128.
bool make_tmap_rows_e4m3(CUtensorMap *m, const void *ptr, uint64_t rows, uint64_t cols, uint32_t box_rows);
// Per-row e4m3 quantisation: scale[r] = amax(row r) / 448 (1 for a zero row),
// q = e4m3(x / scale) rounded to nearest even, saturating; x and q row-major with
// leading dimensions ldx / ldq (elements).  cols % 8 == 0.
cudaError_t launch_quant_rows(const bf16 *x, int ldx, int rows, int cols, uint8_t *q, int ldq, float *scale,
                              cudaStream_t st);
// The same quantisation with each row's amax given (row_amax, as produced by the attention or
// SwiGLU epilogue): one pass over x; row_amax is reset to zero for its next producer.
cudaError_t launch_quant_rows_amax(const bf16 *x, int ldx, int rows, int cols, uint8_t *q, int ldq, float *scale,
                                   float *row_amax, cudaStream_t st);
// RMSNorm (as launch_rmsnorm, output rounded to bf16) followed by the per-row
// e4m3 quantisation of that bf16 output.
cudaError_t launch_rmsnorm_q8(const bf16 *x, const bf16 *w, uint8_t *q, float *scale, int rows, int cols, float eps,
                              cudaStream_t st);
int gemm_box_rows_a();
int gemm_box_rows_w();
// Bytes of a split workspace (partials then flags) for a grid of num_sms CTAs.
size_t gemm_workspace_bytes(int num_sms);
size_t gemm_flags_offset(int num_sms);   // byte offset of the release flags inside the workspace
cudaError_t launch_gemm(const GemmPlan &p, cudaStream_t stream);
// The next launch_gemm on this thread records its phase timeline into trace ([grid][11] %globaltimer ns).
void gemm_trace_next(unsigned long long *trace);
// The next launch_attention on this thread records a per-CTA timeline into trace
// ([grid][attention_trace_fields()] entries).
void attention_trace_next(unsigned long long *trace);
int attention_trace_fields();

// ---- norms and rotary embedding (norm_rope.cu)
struct RopeParams {
    int half_dim;
    float inv_freq[kMaxHalfDim];
    int8_t axis[kMaxHalfDim];
};
void make_rope_params(RopeParams *p, int head_dim, float theta, const int32_t section[3]);
cudaError_t launch_rmsnorm(const bf16 *x, const bf16 *w, bf16 *y, int rows, int cols, float eps, cudaStream_t st);
// Row stride of the row-interleaved rotary tables for n rows: whole 512-byte runs of 32 rows.
inline int cs_stride(int n) { return (n + 31) & ~31; }
// cos/sin [S, head_dim/2]; stride > 0: row-interleaved [head_dim/8][stride][4] (GemmPlan::cs_rows =
// stride >= S, head_dim % 8 == 0; rows past S are not written).
cudaError_t launch_rope_table(const int32_t *positions, int S, const RopeParams &rp, float *cos_t, float *sin_t,
                              cudaStream_t st, int stride = 0);


// ---- attention on tcgen05 (attention_tc.cu)
// row_amax (optional, [S] floats): each row's largest |bf16 output| is merged in with an
// integer atomic max (the buffer must hold zeros or smaller values beforehand).
// workspace (optional, bidirectional only; attention_workspace_bytes, zero-filled once before
// first use, calls sharing it must not overlap on the GPU): lets a thin last round of items be
// cut along the keys instead of into single query tiles.
cudaError_t launch_attention(const bf16 *qkv, bf16 *o, int S, int nq, int nkv, int d, const int32_t *cu_host,
                             int n_seqs, int32_t *status, cudaStream_t st, float *row_amax = nullptr,
                             bool causal = true, void *workspace = nullptr, size_t workspace_bytes = 0);
size_t attention_workspace_bytes(int num_sms, int d);

// ---- vision tower (vision.cu)
constexpr int kMaxVisionGrids = 64;
// Patch grids of one vision encode, patches concatenated in the tower's order.
struct VisionGrids {
    int n, merge;
    int first[kMaxVisionGrids];   // index of each grid's first patch
    int h[kMaxVisionGrids], w[kMaxVisionGrids];
};
// thw host int32 [n_grids, 3]; false if a grid is empty or not divisible by the merge.
bool make_vision_grids(VisionGrids *g, const int32_t *thw, int n_grids, int merge, int *n_patches);
struct VisionRope {
    float inv_freq[kMaxHalfDim];   // theta^(-2j/(d/2)), j < d/4
};
void make_vision_rope(VisionRope *r, int head_dim, float theta);
// y = bf16((x - mean) / sqrt(var + eps) * w + b) per row; cols % 8 == 0, cols <= 8192.
cudaError_t launch_layernorm(const bf16 *x, const bf16 *w, const bf16 *b, bf16 *y, int rows, int cols, float eps,
                             cudaStream_t st);
// out[k] = bilinear sample of the G x G table [G*G, D] at patch k (bf16), n patches.
cudaError_t launch_pos_embed(const bf16 *table, int G, int D, const VisionGrids &gr, int n, bf16 *out,
                             cudaStream_t st);
// cos/sin [n, head_dim/2] of the 2-D rotary angles (row frequencies, then column frequencies);
// stride > 0: row-interleaved [head_dim/8][stride][4] as launch_rope_table.
cudaError_t launch_vision_rope(const VisionGrids &gr, int n, int head_dim, const VisionRope &rp, float *cos_t,
                               float *sin_t, cudaStream_t st, int stride = 0);

// ---- embedding gather, visual ranks, weight packing (embed.cu)
cudaError_t launch_embed(const int32_t *ids, const bf16 *table, int vocab, int hidden, bf16 *out, int S,
                         int32_t *status, cudaStream_t st);
cudaError_t launch_vis_rank(const uint8_t *mask, int S, int n_vis, int32_t *rank, int32_t *status,
                            cudaStream_t st);
cudaError_t pack_gate_up_rows(const bf16 *src, bf16 *W, int I, int K, int which, cudaMemcpyKind kind,
                              cudaStream_t st);

cudaError_t launch_merge_visual_rows(const int32_t *vis_rank, const bf16 *src, int n_vis, int hidden, bf16 *out,
                                     int S, cudaStream_t st);

int device_num_sms();

// Launch configuration with programmatic stream serialization (see pdl_wait in
// common.cuh); attrs must hold room for the attribute and any extra ones the
// caller appends after it.
inline cudaLaunchConfig_t pdl_config(dim3 grid, dim3 block, size_t smem, cudaStream_t st,
                                     cudaLaunchAttribute *attrs) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = grid;
    cfg.blockDim = block;
    cfg.dynamicSmemBytes = smem;
    cfg.stream = st;
    attrs[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attrs[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attrs;
    cfg.numAttrs = 1;
    return cfg;
}

}  // namespace h3
