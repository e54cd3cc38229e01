/* h3vis — the Qwen3-VL vision tower on one GB300: pixel patches in, the visual
 * embeddings (one row per merged block of patches) and the DeepStack features
 * out, ready for h3enc_encode_multimodal.
 *
 * Page "vllm-omni vllm_omni/diffusion/models/minimax_h3/encoder.py", section
 * "Qwen3-VL vision tower": MiniMaxH3Qwen3VLVisionModel.forward with
 * MiniMaxH3Qwen3VLVisionPatchEmbed (Conv3d, stride = kernel: a linear over each
 * flattened patch), fast_pos_embed_interpolate, rot_pos_emb,
 * MiniMaxH3Qwen3VLVisionBlock (LayerNorm, packed QKV with bias, 2-D rotary q/k,
 * bidirectional attention inside each frame, projection; LayerNorm, tanh-GELU MLP)
 * and MiniMaxH3Qwen3VLVisionPatchMerger (main merger: LayerNorm then grouping of
 * each m x m block; DeepStack mergers: grouping then LayerNorm; linear, exact
 * GELU, linear).
 *
 * Every call returns an h3enc_status; h3vis_last_error(h) gives the message.
 * Same conventions as h3enc.h: plain pointers, device buffers owned by the
 * caller, asynchronous on the caller's stream, no allocation inside an encode. */
#ifndef H3VIS_H
#define H3VIS_H

#include "h3enc.h"

#ifdef __cplusplus
extern "C" {
#endif

/* Sizes of the tower (the pages read them from the checkpoint's vision config).
 * Requirements of this implementation: hidden, 3*hidden, intermediate and
 * out_hidden multiples of 256; hidden / num_heads in {64, 128};
 * hidden * spatial_merge_size^2 <= 8192 and a multiple of 256;
 * in_channels * temporal_patch_size * patch_size^2 a multiple of 8;
 * num_position_embeddings a perfect square; num_deepstack <= 8 with
 * ascending block indexes below depth; max_patches a multiple of
 * spatial_merge_size^2. */
typedef struct {
    int32_t depth;
    int32_t hidden;
    int32_t num_heads;
    int32_t intermediate;
    int32_t in_channels;
    int32_t patch_size;
    int32_t temporal_patch_size;
    int32_t spatial_merge_size;
    int32_t out_hidden;               /* the text model's hidden size */
    int32_t num_position_embeddings;  /* G * G rows of the learned position table */
    int32_t num_deepstack;
    int32_t deepstack_indexes[8];     /* blocks whose output feeds a DeepStack merger */
    float ln_eps;                     /* 1e-6 on the pages */
    float rope_theta;                 /* 10000 on the pages */
    int32_t max_patches;              /* largest number of patches of one encode */
} h3vis_config;

typedef struct h3vis h3vis;

H3ENC_API h3enc_status h3vis_create(const h3vis_config *cfg, h3vis **out);

/* One checkpoint tensor, bf16, by its HF name: model.visual.patch_embed.proj.
 * {weight [hidden, C, T, P, P] (or [hidden, C*T*P*P]), bias}, model.visual.pos_embed.
 * weight [G*G, hidden], model.visual.blocks.{i}.{norm1,norm2}.{weight,bias},
 * .attn.qkv.{weight [3h, h], bias}, .attn.proj.{weight, bias},
 * .mlp.linear_fc1.{weight [I, h], bias}, .mlp.linear_fc2.{weight [h, I], bias},
 * model.visual.merger.{norm [h], linear_fc1 [4h, 4h], linear_fc2 [out, 4h]}.{weight,
 * bias} and model.visual.deepstack_merger_list.{j}.{norm [4h], linear_fc1,
 * linear_fc2}.{weight, bias} (4h = hidden * spatial_merge_size^2).  Blocks or
 * mergers beyond the configuration are ignored (H3ENC_WARN_IGNORED); a wrong
 * shape is H3ENC_ERR_SHAPE. */
H3ENC_API h3enc_status h3vis_load_weights(h3vis *h, const char *name, const void *data, int32_t dtype,
                                          const int64_t *shape, int32_t ndim, int32_t data_on_device);

/* H3ENC_ERR_MISSING_WEIGHTS (with the missing names) unless every tensor is loaded. */
H3ENC_API h3enc_status h3vis_finalize_weights(h3vis *h);

/* pixel_values: device bf16 [n_patches, C*T*P*P], each patch flattened in (C, T, P, P)
 * order, patches of the grids concatenated in the tower's order (per grid: frames,
 * then m x m blocks row-major, then the block's patches row-major).
 * grid_thw: HOST int32 [n_grids, 3] (frames, patch rows, patch columns; rows and
 * columns multiples of spatial_merge_size; sum of t*h*w = n_patches <= max_patches;
 * n_grids <= 64; frames in all <= 1024).
 * embeds_out: device bf16 [n_patches / m^2, out_hidden] (the merger's output);
 * deepstack_out: device bf16 [num_deepstack, n_patches / m^2, out_hidden] or NULL. */
H3ENC_API h3enc_status h3vis_encode(h3vis *h, const void *pixel_values, int32_t n_patches,
                                    const int32_t *grid_thw, int32_t n_grids, void *embeds_out,
                                    void *deepstack_out, void *stream);

/* Device-side status after the stream (0 = fine; bit 0 = a bounded wait timed out). */
H3ENC_API h3enc_status h3vis_get_status(h3vis *h);
H3ENC_API const char *h3vis_last_error(const h3vis *h);
H3ENC_API int64_t h3vis_launch_count(const h3vis *h);
H3ENC_API void h3vis_destroy(h3vis *h);

#ifdef __cplusplus
}
#endif

#endif /* H3VIS_H */
