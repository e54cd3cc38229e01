/*
 * h3enc op-level entry points: each step of the encode as its own call, for
 * parity tests and kernel benchmarks.  The encode (h3enc.h) launches exactly
 * these kernels.  All pointers are device pointers unless marked HOST; all
 * matrices are row-major bf16 with the stated leading dimension; `stream` is
 * a cudaStream_t (NULL = legacy default).  `status` is an optional device
 * int32 that kernels OR error bits into (1 = bounded wait ran out, 2 = index
 * out of bounds, 4 = visual count mismatch); NULL disables recording.
 * Return: H3ENC_OK, H3ENC_ERR_INVALID_ARG (checked before launch) or
 * H3ENC_ERR_CUDA (launch failed).
 */
#ifndef H3ENC_OPS_H
#define H3ENC_OPS_H

#include <stdint.h>
#include "h3enc.h"

#ifdef __cplusplus
extern "C" {
#endif

/* GEMM epilogues of the projection kernel C = A * W^T (fp32 accumulation). */
enum {
    H3ENC_EPI_STORE = 0,       /* C = bf16(acc)                                   (QKV projection) */
    H3ENC_EPI_RESIDUAL = 1,    /* C = bf16(R + acc); R may equal C                (o_proj + residual) */
    H3ENC_EPI_SWIGLU = 2,      /* W packed by h3enc_op_pack_gate_up (N = 2*I rows):
                                  C[:, i] = bf16(silu(gate_i) * up_i), C has I columns (gate/up + SwiGLU) */
    H3ENC_EPI_RESIDUAL_DS = 3, /* C = bf16(R + acc), then at rows with vis_rank[r] = j in [0, n_vis):
                                  C = bf16(C + DS[j])                             (down_proj + residual + DeepStack) */
    H3ENC_EPI_GELU_TANH = 5,   /* C = bf16(gelu_tanh(acc + bias))                 (vision MLP fc1) */
    H3ENC_EPI_GELU_ERF = 6     /* C = bf16(gelu(acc + bias)), exact erf form      (vision merger fc1) */
};

/* Projection GEMM on the tcgen05 tensor cores (page "vllm-omni ... encoder.py":
 * F.linear of the QKV, o, gate/up and down projections, plus the residual adds
 * of MiniMaxH3Qwen3VLTextDecoderLayer.forward and _deepstack_process).
 *   A [M, K] (lda = K), W [N, K] (ldw = K), C [M, ldc]: ldc = N, or N/2 for SWIGLU.
 *   R [M, ldc] residual (RESIDUAL*), DS [n_vis, ldc] and vis_rank [M] (RESIDUAL_DS).
 *   workspace: NULL, or device memory of at least h3enc_op_gemm_workspace_bytes()
 *   bytes, 256-byte aligned, zero-filled once before its first use and then
 *   reused; with it the k-blocks of the tiles of a partial last wave are spread
 *   evenly over all SMs (stream-K; the result is deterministic for given M, N,
 *   K and SM count).  Calls sharing a workspace must not overlap on the GPU.
 * Requires K % 8 == 0, N % 256 == 0 (of the packed weight for SWIGLU), A and W
 * 16-byte aligned.  M may be any size >= 0. */
H3ENC_API h3enc_status h3enc_op_gemm(const void *A, const void *W, void *C, int32_t M, int32_t N, int32_t K,
                           int32_t epilogue, const void *R, const void *DS, const int32_t *vis_rank,
                           int32_t n_vis, void *workspace, int64_t workspace_bytes, int32_t *status,
                           void *stream);

/* Profiling aid: the next projection GEMM this host thread launches (through
 * h3enc_op_gemm, h3enc_op_gemm_qkv_rope, h3enc_op_gemm_noalloc or inside an
 * encode) records a timeline: CTA c writes 11 %globaltimer stamps (ns) to
 * trace[c * 11 + k]: k = 0 start, 1 prologue done, 2 last data-parallel accumulator
 * ready (epilogue start of the last tile), 3 first
 * MMA, 4 last data-parallel MMA issued, 5 data-parallel epilogues done, 6 first
 * stream-K accumulator ready, 7 stream-K partials written, 8 first tile's
 * contributor flags seen, 9 stream-K reduction done, 10 end.  The stream-K phase
 * runs before the data-parallel tiles; stamps of phases a CTA does not run, and
 * rows of CTAs beyond the grid, keep their contents.  trace: device uint64 of at
 * least 11 * SM-count entries, alive until that GEMM has run. */
H3ENC_API h3enc_status h3enc_op_gemm_trace_next(void *trace, int64_t trace_entries);

/* Profiling aid: the next attention launch on this host thread (through
 * h3enc_op_attention or inside an encode) records a timeline per persistent CTA
 * (one per SM, at most one per work item; work items = heads * sum over
 * sequences of ceil(len / 256)).  CTA c writes 9 entries at trace[c * 9]:
 * 0 start and 6 end as %globaltimer ns; 1 set-up done, 2 first Q tiles landed,
 * 3 first score tile ready, 4 last P written, 5 last P V product done as SM
 * clock64 cycles; then 7 the SM id and 8 the number of key tiles processed.
 * trace: device uint64 of at least 9 * ctas entries (ctas >= the SM count
 * covers every launch), alive until that launch has run. */
H3ENC_API h3enc_status h3enc_op_attention_trace_next(void *trace, int64_t trace_entries, int32_t ctas);

/* Failure-detection self-test (no counterpart on the pages).  Launches one
 * thread on `stream` that waits, through the library's bounded-wait helpers,
 * either until the device word *flag equals `expect` (use_mbarrier = 0) or on a
 * shared-memory mbarrier that nothing arrives on (use_mbarrier = 1).  A wait that
 * is not satisfied within the wait limit (about 2 s of SM clock) ORs ST_TIMEOUT
 * (1) into the device int32 *status and returns; the context stays usable.
 * flag: device memory (ignored when use_mbarrier = 1). */
H3ENC_API h3enc_status h3enc_op_wait_probe(const uint32_t *flag, uint32_t expect, int32_t use_mbarrier,
                                 int32_t *status, void *stream);

/* Workspace bytes h3enc_op_gemm needs on the current device (-1 without a device). */
H3ENC_API int64_t h3enc_op_gemm_workspace_bytes(void);

/* h3enc_op_gemm for callers that cannot allocate device memory (the pages have
 * no counterpart: this is a library convenience).  Some callers have no way to
 * hand over a workspace: code running inside another framework's allocator
 * callback or after a memory pool has reserved the whole device, plugins that
 * receive only their input and output buffers, hosts that forbid cudaMalloc
 * after start-up.  This entry point computes exactly what h3enc_op_gemm
 * computes with a workspace (same kernel, same split of the last wave), but its
 * scratch is a fixed array inside the library's device image:
 * h3enc_op_gemm_noalloc_scratch_bytes() bytes (40 MiB + 904 B, two 128 KiB
 * fp32 slots and one flag per SM for up to 160 SMs), held by every GPU that
 * loads the library until the process exits.  The caller passes inputs and
 * outputs only; nothing is allocated or freed.
 *   - The first call on a device looks up the array's device address and clears
 *     its flags with a memset queued on `stream` ahead of the kernel (no host or
 *     device synchronisation).  While `stream` is being captured that first call
 *     is refused (H3ENC_ERR_UNSUPPORTED): make it outside any capture.  Later
 *     calls only launch the kernel.
 *   - All calls on a device share the array and it keeps the last call's
 *     contents: calls that overlap on the GPU (other streams, other threads)
 *     race and corrupt each other's results; serialise them.
 *   - A device with more than 160 SMs would need more scratch than the array
 *     holds: the call returns H3ENC_ERR_UNSUPPORTED (message from
 *     h3enc_op_gemm_noalloc_last_error()).
 * Arguments, requirements and other errors are those of h3enc_op_gemm. */
H3ENC_API h3enc_status h3enc_op_gemm_noalloc(const void *A, const void *W, void *C, int32_t M, int32_t N, int32_t K,
                                   int32_t epilogue, const void *R, const void *DS, const int32_t *vis_rank,
                                   int32_t n_vis, int32_t *status, void *stream);

/* Bytes of the fixed scratch array h3enc_op_gemm_noalloc uses. */
H3ENC_API int64_t h3enc_op_gemm_noalloc_scratch_bytes(void);

/* Message of the last h3enc_op_gemm_noalloc error on this thread ("" if none). */
H3ENC_API const char *h3enc_op_gemm_noalloc_last_error(void);

/* Pack gate [I, K] and up [I, K] into W [2I, K] for H3ENC_EPI_SWIGLU: rows
 * [256b, 256b+128) = gate rows [128b, 128b+128), rows [256b+128, 256b+256) =
 * up rows [128b, 128b+128).  Requires I % 128 == 0. */
H3ENC_API h3enc_status h3enc_op_pack_gate_up(const void *gate, const void *up, void *W, int32_t I, int32_t K,
                                   void *stream);

/* Online-FP8 projection (page "vllm-omni ... encoder.py",
 * _validate_encoder_quant_config and the _is_quantized_linear branches): as
 * h3enc_op_gemm with e4m3 operands A [M, K] and W [N, K] (one byte per element,
 * row-major, 16-byte aligned, K % 16 == 0), their fp32 scales sa [M] (per row of
 * A) and sw [N] (per row of W, 16-byte aligned): the product is
 * (A * sa) (W * sw)^T accumulated in fp32 on the tensor cores, then the same
 * epilogues (STORE, RESIDUAL, SWIGLU, RESIDUAL_DS) and the same workspace rules. */
H3ENC_API h3enc_status h3enc_op_gemm_fp8(const void *A, const void *W, const float *sa, const float *sw, void *C,
                               int32_t M, int32_t N, int32_t K, int32_t epilogue, const void *R, const void *DS,
                               const int32_t *vis_rank, int32_t n_vis, void *workspace, int64_t workspace_bytes,
                               int32_t *status, void *stream);

/* Per-row e4m3 quantisation of a bf16 matrix x [rows, cols] (cols % 8 == 0):
 * scale[r] = amax(row r) / 448 in fp32 (1 for an all-zero row), q = e4m3(x * inv)
 * with inv = 448 / amax and the product each rounded once in fp32, then rounded
 * to nearest even, saturating at +-448 (the "fn" variant).  q [rows, cols]
 * bytes; x 16-byte aligned. */
H3ENC_API h3enc_status h3enc_op_quant_rows(const void *x, int32_t rows, int32_t cols, void *q, float *scale,
                                 void *stream);

/* RMSNorm of x [rows, cols] (as h3enc_op_rmsnorm, output rounded to bf16) followed
 * by h3enc_op_quant_rows of that bf16 output: q [rows, cols] e4m3, scale [rows]. */
H3ENC_API h3enc_status h3enc_op_rmsnorm_q8(const void *x, const void *w, void *q, float *scale, int32_t rows,
                                 int32_t cols, float eps, void *stream);

/* y = bf16(w * x / sqrt(mean(x^2) + eps)) per row, fp32 math (page "...
 * encoder.py", MiniMaxH3Qwen3VLRMSNorm).  x, y [rows, cols]; cols % 8 == 0,
 * cols <= 8192; y may equal x. */
H3ENC_API h3enc_status h3enc_op_rmsnorm(const void *x, const void *w, void *y, int32_t rows, int32_t cols,
                              float eps, void *stream);

/* M-RoPE tables (page "... encoder.py", MiniMaxH3Qwen3VLTextRotaryEmbedding and
 * _apply_interleaved_mrope): for j < head_dim/2,
 *   ang = float(positions[axis(j)][s]) * inv_freq[j],  inv_freq[j] = theta^(-2j/head_dim) (fp32),
 *   axis(j) = 1 if j%3==1 and j < 3*section[1]; 2 if j%3==2 and j < 3*section[2]; else 0,
 *   cos_tab[s][j] = cos(ang), sin_tab[s][j] = sin(ang)   (fp32, [S, head_dim/2]). */
H3ENC_API h3enc_status h3enc_op_rope_table(const int32_t *positions, int32_t S, int32_t head_dim, float theta,
                                 const int32_t *section_host, float *cos_tab, float *sin_tab,
                                 void *stream);

/* h3enc_op_rope_table with a choice of layout.  stride == 0: [S, head_dim/2] as above.
 * stride >= S (head_dim % 8 == 0): row-interleaved, the layout the encoder uses,
 *   cos_tab[((j/4) * stride + s) * 4 + j%4] = cos(ang(s, j))   (same for sin_tab),
 * i.e. [head_dim/8][stride][4]: for each group of four frequencies the rows follow one
 * another, so 32 consecutive rows read one group as 512 contiguous bytes.  Rows s >= S of
 * the padding are not written.  Each table holds stride * head_dim/2 floats (16-byte
 * aligned); a stride that is a multiple of 32 keeps every 32-row run on whole lines.
 * INVALID_ARG for 0 < stride < S or head_dim % 8 with stride > 0. */
H3ENC_API h3enc_status h3enc_op_rope_table_ex(const int32_t *positions, int32_t S, int32_t head_dim, float theta,
                                    const int32_t *section_host, int32_t stride, float *cos_tab,
                                    float *sin_tab, void *stream);

/* QKV projection with the per-head q/k RMSNorm and M-RoPE fused into the GEMM
 * epilogue (page "... encoder.py", MiniMaxH3Qwen3VLTextAttention.forward: the
 * q/k/v projections, q_norm/k_norm over head_dim, then _apply_rotary_pos_emb):
 *   qkv = A * W^T with W [(nq + 2*nkv)*d, K] (q rows, then k, then v);
 *   every q head (columns h*d) and k head (columns (nq + g)*d) of qkv becomes
 *   rope(rmsnorm(x, w_q or w_k, eps)) with, for j < d/2,
 *     rope(x)[j] = x[j]*cos[j] - x[j+d/2]*sin[j],  rope(x)[j+d/2] = x[j+d/2]*cos[j] + x[j]*sin[j]
 *   (cos/sin = the fp32 tables of h3enc_op_rope_table, [M, d/2]); v heads are the plain
 *   projection.  C [M, (nq + 2*nkv)*d].  workspace as for h3enc_op_gemm.
 * Requires head_dim in {64, 128} and (nq + 2*nkv)*d % 256 == 0. */
H3ENC_API h3enc_status h3enc_op_gemm_qkv_rope(const void *A, const void *W, void *C, int32_t M, int32_t K,
                                    int32_t n_heads, int32_t n_kv_heads, int32_t head_dim, const void *w_q,
                                    const void *w_k, float eps, const float *cos_tab, const float *sin_tab,
                                    void *workspace, int64_t workspace_bytes, int32_t *status, void *stream);

/* RMSNorm folded into a projection (page "... encoder.py", MiniMaxH3Qwen3VLRMSNorm
 * followed by the projection that reads its output; an algebraic rearrangement the
 * encoder uses when h3enc_config.separate_norm == 0):
 *   rmsnorm(x, g) W^T = diag(1 / sqrt(mean(x^2) + eps)) x (W diag(g))^T.
 * Row statistics are sums of squares over slots of 128 columns, accumulated in fp32 in
 * column order, stored slot-major: ss[s * rows + r] = sum_{c in [128 s, 128 s + 128)} x[r][c]^2.
 *
 * h3enc_op_row_sumsq: ss [cols/128, rows] fp32 of the bf16 matrix x [rows, cols];
 * cols % 128 == 0, x 16-byte aligned. */
H3ENC_API h3enc_status h3enc_op_row_sumsq(const void *x, int32_t rows, int32_t cols, float *ss, void *stream);

/* h3enc_op_fold_cols: W[r][k] = bf16(W[r][k] * gamma[k]) in place (fp32 product rounded
 * to nearest even), W bf16 [rows, cols], gamma bf16 [cols]; cols % 8 == 0, both
 * 16-byte aligned. */
H3ENC_API h3enc_status h3enc_op_fold_cols(void *W, int32_t rows, int32_t cols, const void *gamma, void *stream);

/* h3enc_op_gemm with the folded norm: ss_in [K/128, M] (or NULL): the accumulator of row
 * r is multiplied by 1/sqrt(sum_s ss_in[s][r] / K + eps) (slots added in order) before the
 * epilogue; ss_out [N/128, M] (or NULL; STORE and RESIDUAL only): the row statistics of
 * the bf16 output C, as h3enc_op_row_sumsq would give them.  epilogue: STORE,
 * RESIDUAL or SWIGLU; other arguments as h3enc_op_gemm. */
H3ENC_API h3enc_status h3enc_op_gemm_rms(const void *A, const void *W, void *C, int32_t M, int32_t N, int32_t K,
                                         int32_t epilogue, const void *R, const float *ss_in, float *ss_out,
                                         float eps, void *workspace, int64_t workspace_bytes, int32_t *status,
                                         void *stream);

/* h3enc_op_gemm_qkv_rope reading tables of either layout of h3enc_op_rope_table_ex:
 * cs_stride == 0 for [M, d/2], else the row-interleaved tables of that stride (>= M).
 * ss_in (optional, NULL: none) and in_eps as for h3enc_op_gemm_qkv_rope_rms.  The output is
 * the same, bit for bit, in both layouts; the row-interleaved one is faster (the epilogue's
 * table loads are whole lines). */
H3ENC_API h3enc_status h3enc_op_gemm_qkv_rope_ex(const void *A, const void *W, void *C, int32_t M, int32_t K,
                                       int32_t n_heads, int32_t n_kv_heads, int32_t head_dim, const void *w_q,
                                       const void *w_k, float eps, const float *cos_tab, const float *sin_tab,
                                       int32_t cs_stride, const float *ss_in, float in_eps, void *workspace,
                                       int64_t workspace_bytes, int32_t *status, void *stream);

/* h3enc_op_gemm_qkv_rope with the folded input norm: each row of A * W^T is first
 * multiplied by 1/sqrt(sum_s ss_in[s][r] / K + in_eps) (ss_in [K/128, M], required), then
 * the q/k RMSNorm (eps) and M-RoPE of h3enc_op_gemm_qkv_rope apply. */
H3ENC_API h3enc_status h3enc_op_gemm_qkv_rope_rms(const void *A, const void *W, void *C, int32_t M, int32_t K,
                                                  int32_t n_heads, int32_t n_kv_heads, int32_t head_dim,
                                                  const void *w_q, const void *w_k, float eps,
                                                  const float *cos_tab, const float *sin_tab, const float *ss_in,
                                                  float in_eps, void *workspace, int64_t workspace_bytes,
                                                  int32_t *status, void *stream);

/* ---- vision tower kernels (page "... encoder.py", section "Qwen3-VL vision tower") ----
 * The tower's patch order: per grid, frames, then the m x m blocks row-major, then the
 * patches of a block row-major.  grid_thw: HOST int32 [n_grids, 3] (n_grids <= 64; rows and
 * columns multiples of merge).
 *
 * h3enc_op_layernorm: y = bf16((x - mean) / sqrt(var + eps) * w + b) per row (nn.LayerNorm,
 * biased variance, fp32); x, y [rows, cols] bf16, cols % 8 == 0, cols <= 8192. */
H3ENC_API h3enc_status h3enc_op_layernorm(const void *x, const void *w, const void *b, void *y, int32_t rows,
                                          int32_t cols, float eps, void *stream);

/* h3enc_op_vision_pos_embed (fast_pos_embed_interpolate): out[k] = bf16 of the bilinear
 * sample of the grid_side x grid_side table [grid_side^2, hidden] at patch k: the grid's
 * h x w points evenly spaced from corner to corner (i * (G-1)/(h-1) in double, rounded
 * to fp32), lower corner by truncation, upper clipped to G-1, fp32 weights and
 * products summed corner by corner.  out [n_patches, hidden] bf16. */
H3ENC_API h3enc_status h3enc_op_vision_pos_embed(const void *table, int32_t grid_side, int32_t hidden,
                                                 const int32_t *grid_thw, int32_t n_grids, int32_t merge, void *out,
                                                 void *stream);

/* h3enc_op_vision_rope_table (rot_pos_emb): cos/sin [n_patches, head_dim/2] fp32 of the
 * angles row * inv_freq[j] (j < head_dim/4) and column * inv_freq[j - head_dim/4] (the
 * rest), inv_freq[j] = theta^(-2j/(head_dim/2)) rounded once to fp32; the pairs
 * (j, j + head_dim/2) of q and k rotate by angle j as in h3enc_op_gemm_qkv_rope. */
H3ENC_API h3enc_status h3enc_op_vision_rope_table(const int32_t *grid_thw, int32_t n_grids, int32_t merge,
                                                  int32_t head_dim, float theta, float *cos_tab, float *sin_tab,
                                                  void *stream);

/* h3enc_op_gemm_bias: h3enc_op_gemm with bias [N] (bf16, 16-byte aligned) added to the
 * accumulator; epilogue H3ENC_EPI_STORE (C = bf16(acc + bias)), H3ENC_EPI_RESIDUAL
 * (C = bf16(R + acc + bias)), H3ENC_EPI_GELU_TANH or H3ENC_EPI_GELU_ERF.  Other arguments
 * and requirements as h3enc_op_gemm. */
H3ENC_API h3enc_status h3enc_op_gemm_bias(const void *A, const void *W, void *C, int32_t M, int32_t N, int32_t K,
                                          int32_t epilogue, const void *R, const void *bias, void *workspace,
                                          int64_t workspace_bytes, int32_t *status, void *stream);

/* h3enc_op_gemm_qkv_rope_bias (the vision tower's attention input): qkv = A W^T + bias with
 * W [3 * heads * head_dim, K] (q rows, k rows, v rows), then every q and k head rotated
 * with the fp32 tables cos/sin [M, head_dim/2] (no per-head norm); v heads as they are. */
H3ENC_API h3enc_status h3enc_op_gemm_qkv_rope_bias(const void *A, const void *W, void *C, int32_t M, int32_t K,
                                                   int32_t heads, int32_t head_dim, const void *bias,
                                                   const float *cos_tab, const float *sin_tab, void *workspace,
                                                   int64_t workspace_bytes, int32_t *status, void *stream);

/* h3enc_op_attention_bidir: as h3enc_op_attention with one kv head per q head and no
 * causal mask: every query attends to every key of its segment (the tower's attention
 * inside each frame, scaled_dot_product_attention with is_causal=False). */
H3ENC_API h3enc_status h3enc_op_attention_bidir(const void *qkv, void *o, int32_t S, int32_t heads,
                                                int32_t head_dim, const int32_t *cu_seqlens, int32_t n_seqs,
                                                void *stream);

/* h3enc_op_attention_bidir with a workspace (h3enc_op_attention_workspace_bytes(head_dim)
 * bytes, 16-byte aligned, zero-filled once before its first use and again after a call whose
 * device status reported a timeout; calls sharing it must not overlap on the GPU).  When the persistent kernel's last round of work items would leave
 * most SMs idle, those items are cut into up to 8 ranges of their keys; each range writes
 * its unnormalised output, running maximum and sum to the workspace and the range that
 * finishes last merges them in range order (the same result on every run).  The output
 * equals the plain call's up to fp32 rounding.  0 from the size query: head_dim not 64/128. */
H3ENC_API int64_t h3enc_op_attention_workspace_bytes(int32_t head_dim);
H3ENC_API h3enc_status h3enc_op_attention_bidir_ws(const void *qkv, void *o, int32_t S, int32_t heads,
                                                   int32_t head_dim, const int32_t *cu_seqlens, int32_t n_seqs,
                                                   void *workspace, int64_t workspace_bytes, void *stream);

/* Causal GQA attention over packed sequences (page "... encoder.py",
 * MiniMaxH3Qwen3VLTextAttention.forward: repeat_interleave of K/V, SDPA with
 * is_causal=True, scale 1/sqrt(d)).  Reads q/k/v from qkv [S, (nq+2nkv)*d]
 * (q head h at column h*d, k head g at (nq+g)*d, v head g at (nq+nkv+g)*d),
 * writes o [S, nq*d] (head h at column h*d).  cu_seqlens HOST int32 [n_seqs+1]
 * or NULL (one sequence); n_seqs <= 1024. */
H3ENC_API h3enc_status h3enc_op_attention(const void *qkv, void *o, int32_t S, int32_t n_heads,
                                int32_t n_kv_heads, int32_t head_dim, const int32_t *cu_seqlens,
                                int32_t n_seqs, void *stream);

/* out[s] = table[ids[s]] (bit-exact row copy; page "... encoder.py",
 * embed_tokens / F.embedding).  Ids outside [0, vocab) give a zero row and
 * set status bit 2.  hidden % 8 == 0. */
H3ENC_API h3enc_status h3enc_op_embed(const int32_t *ids, const void *table, int32_t vocab, int32_t hidden,
                            void *out, int32_t S, int32_t *status, void *stream);

/* vis_rank[s] = number of visual rows before s if mask[s] != 0, else -1 (the
 * row of the DeepStack features that boolean-mask assignment gives row s).
 * Sets status bit 4 if the mask holds a count other than n_vis. */
H3ENC_API h3enc_status h3enc_op_vis_rank(const uint8_t *mask, int32_t S, int32_t n_vis, int32_t *vis_rank,
                               int32_t *status, void *stream);

#ifdef __cplusplus
}
#endif
#endif /* H3ENC_OPS_H */
