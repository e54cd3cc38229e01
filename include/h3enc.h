/*
 * h3enc — Qwen3-VL text-decoder prefill ("layer-50 encoder" of MiniMax H3) on
 * one GB300 (sm_103a).  C ABI: plain pointers and sizes, no torch types.
 *
 * What one encode computes (page "vllm-omni vllm_omni/diffusion/models/
 * minimax_h3/encoder.py", MiniMaxH3Qwen3VLTextModel.forward and the classes it
 * calls; the module docstring states the contract):
 *   x = embed_tokens[input_ids]
 *   cos/sin = interleaved 3-D M-RoPE tables of positions[3,S], computed once
 *   for each kept layer l:
 *     x = x + o_proj(attn(rope(q_norm(q)), rope(k_norm(k)), v))      q,k,v of input_layernorm(x)
 *     x = x + down_proj(silu(gate_proj(y)) * up_proj(y)),  y = post_attention_layernorm(x)
 *     if l < num_deepstack: x[visual rows] += deepstack[l]   (row j -> j-th visual row)
 *   out = x  (unnormalised hidden_states[num_layers], bf16 [S, hidden])
 * Attention is causal within each packed sequence (cu_seqlens), GQA with
 * q head h reading kv head h / (n_heads / n_kv_heads), scale 1/sqrt(head_dim).
 *
 * Ownership: the caller owns every input/output buffer and the stream.  The
 * handle owns a copy of the weights (packed for the kernels) and a workspace
 * sized at create from max_tokens; encode calls allocate no device memory and
 * never synchronise the host (h3enc_encode_host excepted: it synchronises, and
 * makes a copy stream on its first DeepStack call and a CUDA graph per call
 * shape).  A handle is used by one host thread at a time.
 *
 * Errors: every argument, shape and completeness error is detected on the
 * host before any launch and returned as a status (h3enc_last_error() has the
 * message).  Errors that only the device can see (token id >= vocab, visual
 * mask count != n_vis, a bounded device wait that ran out) are recorded in a
 * device status word; h3enc_get_status() synchronises and reports them.
 */
#ifndef H3ENC_H
#define H3ENC_H

#include <stdint.h>

#if defined(__GNUC__)
#define H3ENC_API __attribute__((visibility("default")))
#else
#define H3ENC_API
#endif

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
    H3ENC_OK = 0,
    H3ENC_WARN_IGNORED = 1,        /* load_weights: name not used by the kept layers (lm_head, final norm,
                                      layers >= num_layers, vision tower, unknown names) */
    H3ENC_ERR_INVALID_ARG = 2,     /* null pointer, bad size, bad cu_seqlens, bad config */
    H3ENC_ERR_SHAPE = 3,           /* weight shape mismatch; visual-mask count != n_vis (device) */
    H3ENC_ERR_NOT_LOADED = 4,      /* encode before h3enc_finalize_weights succeeded */
    H3ENC_ERR_MISSING_WEIGHTS = 5, /* finalize: a parameter or a fused shard (q/k/v, gate/up) was never loaded */
    H3ENC_ERR_UNSUPPORTED = 6,     /* dtype other than bf16 (e.g. serialized FP8), head_dim not 64/128, ... */
    H3ENC_ERR_CUDA = 7,            /* a CUDA runtime/driver call failed (no device, launch failure) */
    H3ENC_ERR_OOM = 8,             /* device allocation failed */
    H3ENC_ERR_DEVICE_TIMEOUT = 9,  /* a bounded device-side wait ran out (reported by h3enc_get_status) */
    H3ENC_ERR_DEVICE_BOUNDS = 10   /* token id outside [0, vocab) (reported by h3enc_get_status) */
} h3enc_status;

enum { H3ENC_DTYPE_BF16 = 0, H3ENC_DTYPE_F32 = 1, H3ENC_DTYPE_FP8_E4M3 = 2 };

/* Model and capacity.  Shapes of the Qwen3-VL text config (hidden_size,
 * num_attention_heads, num_key_value_heads, head_dim, intermediate_size,
 * vocab_size, rms_norm_eps, rope_theta, mrope_section).  num_layers is the
 * number of decoder layers kept (50 for the layer-50 contract).
 * Requirements of this implementation: head_dim in {64, 128}; hidden and
 * n_heads*head_dim multiples of 64; (n_heads + 2*n_kv_heads)*head_dim and hidden
 * multiples of 256; intermediate a multiple of 128; n_heads % n_kv_heads == 0.
 * vocab == 0 builds an embeddings-only model (h3enc_encode_embeds only). */
typedef struct {
    int32_t num_layers;
    int32_t hidden;
    int32_t n_heads;
    int32_t n_kv_heads;
    int32_t head_dim;
    int32_t intermediate;
    int32_t vocab;
    float rms_eps;
    float rope_theta;
    int32_t mrope_section[3];
    int32_t max_tokens;     /* largest S of one encode (workspace sizing) */
    int32_t max_seqs;       /* largest number of packed sequences, <= 1024 */
    int32_t num_deepstack;  /* largest number of DeepStack levels accepted */
    int32_t linear_fp8;     /* 1: online FP8 linears (page "vllm-omni ... encoder.py",
                               _validate_encoder_quant_config: the bf16 checkpoint is
                               quantised at h3enc_finalize_weights to e4m3 with one fp32
                               scale per output channel, activations to e4m3 with one
                               scale per token on every encode; attention stays bf16).
                               0: plain bf16.  The bf16 weights stay loaded. */
    int32_t separate_norm;  /* bf16 only.  0 (default): the two RMSNorms of a layer run inside
                               the projections that read them (page "... encoder.py",
                               MiniMaxH3Qwen3VLRMSNorm before qkv_proj and gate_up_proj):
                               h3enc_finalize_weights multiplies each norm weight into the
                               K columns of those projections once; every encode then
                               emits per-row sums of squares of the hidden state from the
                               o_proj and down_proj epilogues (and one pass over the layer
                               input), and the QKV and gate/up epilogues scale their rows
                               by 1/sqrt(mean + rms_eps).  The normalised activation is
                               never rounded to bf16 (the folded weights are).  1: a
                               separate RMSNorm kernel writes the bf16 normalised rows
                               before each of the two projections.  With linear_fp8 the
                               norm always runs as its own quantising pass. */
} h3enc_config;

typedef struct h3enc h3enc;

/* Validate cfg, allocate the weight arena and the workspace on the current
 * CUDA device.  *out is NULL on failure. */
H3ENC_API h3enc_status h3enc_create(const h3enc_config *cfg, h3enc **out);

/* Load one checkpoint tensor by its HF name (page "vllm-omni ... encoder.py",
 * MiniMaxH3Qwen3VLEncoder._map_weight_name / load_weights):
 *   model.language_model.embed_tokens.weight                   [vocab, hidden]
 *   model.language_model.layers.{l}.input_layernorm.weight     [hidden]
 *   model.language_model.layers.{l}.post_attention_layernorm.weight [hidden]
 *   model.language_model.layers.{l}.self_attn.{q,k,v}_proj.weight   [n*head_dim, hidden]
 *   model.language_model.layers.{l}.self_attn.o_proj.weight    [hidden, n_heads*head_dim]
 *   model.language_model.layers.{l}.self_attn.{q,k}_norm.weight [head_dim]
 *   model.language_model.layers.{l}.mlp.{gate,up}_proj.weight  [intermediate, hidden]
 *   model.language_model.layers.{l}.mlp.down_proj.weight       [hidden, intermediate]
 * q/k/v are packed into one QKV weight and gate/up into one interleaved
 * weight here.  data: bf16, row-major, host memory (data_on_device=0) or
 * device memory of the handle's device (1); copied, so the caller may free it
 * on return.  Returns H3ENC_WARN_IGNORED for names the kept layers do not use,
 * H3ENC_ERR_SHAPE for a shape mismatch, H3ENC_ERR_UNSUPPORTED for a dtype
 * other than bf16 (the pages accept online FP8 only, never serialized FP8). */
H3ENC_API h3enc_status h3enc_load_weights(h3enc *h, const char *name, const void *data, int32_t dtype,
                                const int64_t *shape, int32_t ndim, int32_t data_on_device);

/* Check that every parameter and every fused shard was loaded (page
 * "... encoder.py", _verify_fused_shards_complete and the missing-parameter
 * check of load_weights) and prepare the kernels' weight descriptors.
 * H3ENC_ERR_MISSING_WEIGHTS lists what is missing in h3enc_last_error(). */
H3ENC_API h3enc_status h3enc_finalize_weights(h3enc *h);

/* One encode, asynchronous on `stream` (a cudaStream_t; NULL = legacy default).
 *   input_ids    device int32 [S]
 *   positions    device int32 [3, S]  (t, h, w rows)
 *   visual_mask  device uint8 [S] (nonzero = visual token) or NULL
 *   deepstack    device bf16 [num_deepstack, n_vis, hidden] or NULL; level l is
 *                added after layer l at the visual rows, row j to the j-th visual row
 *   cu_seqlens   HOST int32 [n_seqs + 1], 0 = cu[0] <= ... <= cu[n_seqs] = S, or NULL
 *                (one sequence); attention is causal within each sequence
 *   out          device bf16 [S, hidden]; the hidden state lives here during the encode
 * S == 0 is a no-op.  Inputs are read-only; the buffers must not overlap out. */
H3ENC_API h3enc_status h3enc_encode(h3enc *h, const int32_t *input_ids, const int32_t *positions,
                          const uint8_t *visual_mask, const void *deepstack, int32_t num_deepstack,
                          int32_t n_vis, const int32_t *cu_seqlens, int32_t n_seqs, int32_t seq_len,
                          void *out, void *stream);

/* As h3enc_encode, with the visual rows' input embeddings replaced by the
 * vision tower's merged features (page "... encoder.py", _encode:
 * inputs_embeds.masked_scatter(mask, visual_embeds)): visual_embeds is device
 * bf16 [n_vis, hidden], row j goes to the j-th visual row; NULL behaves as
 * h3enc_encode.  A visual-mask count other than n_vis is reported by
 * h3enc_get_status (H3ENC_ERR_SHAPE) and those rows keep their token embedding. */
H3ENC_API h3enc_status h3enc_encode_multimodal(h3enc *h, const int32_t *input_ids, const int32_t *positions,
                                     const uint8_t *visual_mask, const void *visual_embeds,
                                     const void *deepstack, int32_t num_deepstack, int32_t n_vis,
                                     const int32_t *cu_seqlens, int32_t n_seqs, int32_t seq_len, void *out,
                                     void *stream);

/* As h3enc_encode, from hidden states instead of token ids, over the layer
 * range [layer_begin, layer_end) (global layer indices: DeepStack level l still
 * follows layer l).  inputs_embeds: device bf16 [S, hidden]; it may equal out. */
H3ENC_API h3enc_status h3enc_encode_embeds(h3enc *h, const void *inputs_embeds, int32_t layer_begin,
                                 int32_t layer_end, const int32_t *positions,
                                 const uint8_t *visual_mask, const void *deepstack,
                                 int32_t num_deepstack, int32_t n_vis, const int32_t *cu_seqlens,
                                 int32_t n_seqs, int32_t seq_len, void *out, void *stream);

/* As h3enc_encode with HOST buffers (ids, positions, mask, deepstack, out):
 * copies the inputs to the handle's device staging buffers, encodes, copies
 * the result back and synchronises `stream`.  Host buffers may be pageable;
 * pinned buffers copy faster.
 * CUDA graphs (h3enc_set_graphs, on by default): the encode reads and writes only
 * the handle's own buffers here, so it is captured into a graph per call shape
 * (seq_len, the cu_seqlens values, n_vis, num_deepstack, whether a mask is given)
 * and replayed: the first call of a shape runs eagerly, the second captures and
 * replays, later ones replay.  Up to 8 shapes are kept (least recently used
 * dropped); loading or finalising weights drops them all.  Calls run eagerly
 * while profiling or layer capture is on, on the legacy or per-thread default
 * stream (NULL), or when `stream` is itself being captured.  The copies stay
 * outside the graph. */
H3ENC_API h3enc_status h3enc_encode_host(h3enc *h, const int32_t *input_ids, const int32_t *positions,
                               const uint8_t *visual_mask, const void *deepstack,
                               int32_t num_deepstack, int32_t n_vis, const int32_t *cu_seqlens,
                               int32_t n_seqs, int32_t seq_len, void *out, void *stream);

/* Record the state after every executed layer: per_layer[l] is a device bf16
 * [max_tokens, hidden] buffer (or NULL to skip layer l), n == num_layers.
 * n == 0 disables capture.  The pointers are kept until changed. */
H3ENC_API h3enc_status h3enc_set_layer_capture(h3enc *h, void *const *per_layer, int32_t n);

/* Synchronise the device, read and clear the device status word.  Returns
 * H3ENC_OK, H3ENC_ERR_DEVICE_TIMEOUT, H3ENC_ERR_DEVICE_BOUNDS or H3ENC_ERR_SHAPE
 * (the first that applies, in that order). */
H3ENC_API h3enc_status h3enc_get_status(h3enc *h);

/* Message of the last error on this handle (or of the last failed create when
 * h is NULL).  Valid until the next call on the handle. */
H3ENC_API const char *h3enc_last_error(const h3enc *h);

H3ENC_API void h3enc_destroy(h3enc *h);

/* ---- multimodal front end (ids -> positions, visual rows, DeepStack layout) ---- */

/* M-RoPE positions [3, S] and the visual mask from token ids (page "vllm-omni
 * ... encoder.py", _get_rope_index with _get_vision_position_ids, and
 * _get_placeholder_mask).  HOST memory in and out.  Tokens equal to
 * image_token_id / video_token_id are visual; consecutive tokens of one kind
 * form a run.  A text run of n tokens at running start c gets (c+i, c+i, c+i)
 * and c += n.  A visual run takes the next grid of its kind (image grids in
 * order; a video of T frames counts as T grids of one frame), whose merged
 * size t * (h/m) * (w/m) (m = spatial_merge_size) must equal the run length,
 * gets (c+f, c+r, c+col) in (f, r, col) row-major order, and c += max(h, w)/m.
 *   image_grid_thw [n_images, 3], video_grid_thw [n_videos, 3] (t, h, w before merging)
 *   positions [3, S] out; visual_mask [S] out (1 = visual) or NULL;
 *   visual_kind [S] out (0 text, 1 image, 2 video) or NULL;
 *   n_image_tokens, n_video_tokens, mrope_delta (max position + 1 - S) out or NULL.
 * H3ENC_ERR_SHAPE if a run does not match its grid or grids run out; the
 * message is in h3enc_frontend_last_error(). */
H3ENC_API h3enc_status h3enc_build_positions(const int32_t *input_ids, int32_t seq_len, int32_t image_token_id,
                                   int32_t video_token_id, const int32_t *image_grid_thw, int32_t n_images,
                                   const int32_t *video_grid_thw, int32_t n_videos,
                                   int32_t spatial_merge_size, int32_t *positions, uint8_t *visual_mask,
                                   uint8_t *visual_kind, int32_t *n_image_tokens, int32_t *n_video_tokens,
                                   int32_t *mrope_delta);

/* DeepStack features of images and videos interleaved in sequence order
 * (page "... encoder.py", _aggregate_deepstack): for every level l,
 * out[l][j] = the next image row if the j-th visual token is an image token,
 * else the next video row.  visual_kind HOST [S] (from h3enc_build_positions);
 * image_feats [levels, n_image_tokens, hidden], video_feats [levels,
 * n_video_tokens, hidden], out [levels, n_image_tokens + n_video_tokens,
 * hidden]: device bf16.  Asynchronous copies on `stream`. */
H3ENC_API h3enc_status h3enc_aggregate_deepstack(const uint8_t *visual_kind, int32_t seq_len,
                                       const void *image_feats, int32_t n_image_tokens, const void *video_feats,
                                       int32_t n_video_tokens, int32_t levels, int32_t hidden, void *out,
                                       void *stream);

/* Message of the last front-end error on this thread. */
H3ENC_API const char *h3enc_frontend_last_error(void);

/* Kernel classes timed by the optional profiler. */
enum {
    H3ENC_K_PREP = 0,     /* embedding gather / input copy, M-RoPE tables, visual ranks */
    H3ENC_K_RMSNORM = 1,
    H3ENC_K_GEMM_QKV = 2,
    H3ENC_K_QUANT = 3,    /* FP8 mode: e4m3 quantisation of the attention and SwiGLU outputs */
    H3ENC_K_ATTN = 4,
    H3ENC_K_GEMM_O = 5,
    H3ENC_K_GEMM_GATE_UP = 6,
    H3ENC_K_GEMM_DOWN = 7,
    H3ENC_K_COUNT = 8
};

/* enable != 0: record a CUDA event pair around every kernel launch (on the
 * launching stream) and accumulate per-class device time.  Resets totals.
 * An encode captured into a CUDA graph while profiling is on carries the event
 * pairs as event-record nodes: each replay records them again, and the next
 * h3enc_get_profile returns the durations of the latest replay (launch counts
 * are those of the capture; the reset then detaches the pairs). */
H3ENC_API h3enc_status h3enc_set_profiling(h3enc *h, int32_t enable);

/* As h3enc_set_profiling, timing only the classes whose bit (1 << class) is set
 * in mask (0 = off); launches of the other classes are still counted. */
H3ENC_API h3enc_status h3enc_set_profiling_classes(h3enc *h, uint32_t mask);

/* Restrict the profiling events to the launches of one decoder layer (0 <= layer <
 * num_layers; -1, the default: every launch).  A sample of identical launches: an
 * event between two launches stops the second from overlapping the first, so timing
 * one layer's launches disturbs an encode far less than timing all of them. */
H3ENC_API h3enc_status h3enc_set_profiling_layer(h3enc *h, int32_t layer);

/* Synchronise and return per-class totals since the last reset: ms[k] and
 * launches[k] (the number of timed launches) for k < n (n <= H3ENC_K_COUNT).
 * Resets totals. */
H3ENC_API h3enc_status h3enc_get_profile(h3enc *h, double *ms, int64_t *launches, int32_t n);

/* Number of kernels this handle has launched since create (a graph replay counts
 * the kernels it runs). */
H3ENC_API int64_t h3enc_launch_count(const h3enc *h);

/* enable (0 or 1): let h3enc_encode_host capture and replay CUDA graphs (default 1).
 * Disabling drops the cached graphs. */
H3ENC_API h3enc_status h3enc_set_graphs(h3enc *h, int32_t enable);

/* Number of captured graphs the handle holds (0..8). */
H3ENC_API int32_t h3enc_graph_count(const h3enc *h);

/* Number of streaming multiprocessors the handle's kernels size their grids by. */
H3ENC_API int32_t h3enc_num_sms(const h3enc *h);

#ifdef __cplusplus
}
#endif
#endif /* H3ENC_H */
