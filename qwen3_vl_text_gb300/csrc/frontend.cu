// Multimodal front end of the encoder: token ids -> M-RoPE positions and visual
// mask (host), image + video DeepStack aggregation and visual-embedding merge
// (device copies / gather).
//
// Page "vllm-omni vllm_omni/diffusion/models/minimax_h3/encoder.py":
// _get_rope_index with _get_vision_position_ids (positions), _get_placeholder_mask
// (visual rows are the image / video placeholder ids), _aggregate_deepstack
// (per-level features of images and videos interleaved in sequence order) and
// the masked_scatter of _encode (vision-merger rows replace the placeholder
// embeddings).
#include <cstring>
#include <vector>

#include "../../include/h3enc.h"
#include "common.cuh"
#include "kernels.h"

namespace {

thread_local char g_err[256];

h3enc_status ferr(h3enc_status s, const char *msg) {
    strncpy(g_err, msg, sizeof g_err - 1);
    g_err[sizeof g_err - 1] = 0;
    return s;
}

// One warp per row: rows with vis_rank >= 0 take their row of `src` instead.
__global__ void __launch_bounds__(256) merge_visual_rows_kernel(const int32_t *__restrict__ vis_rank,
                                                                const h3::bf16 *__restrict__ src, int n_vis,
                                                                int hidden, h3::bf16 *out, int S) {
    h3::pdl_trigger();
    h3::pdl_wait();
    const int lane = threadIdx.x & 31;
    const int row = blockIdx.x * 8 + (threadIdx.x >> 5);
    if (row >= S) return;
    const int r = vis_rank[row];
    if (r < 0 || r >= n_vis) return;
    const uint4 *s4 = reinterpret_cast<const uint4 *>(src + (size_t)r * hidden);
    uint4 *d4 = reinterpret_cast<uint4 *>(out + (size_t)row * hidden);
    for (int v = lane; v < (hidden >> 3); v += 32) d4[v] = s4[v];
}

}  // namespace

namespace h3 {
cudaError_t launch_merge_visual_rows(const int32_t *vis_rank, const bf16 *src, int n_vis, int hidden, bf16 *out,
                                     int S, cudaStream_t st) {
    if (S <= 0 || n_vis <= 0) return cudaSuccess;
    cudaLaunchAttribute at[1];
    cudaLaunchConfig_t cfg = pdl_config(dim3((S + 7) / 8), dim3(256), 0, st, at);
    return cudaLaunchKernelEx(&cfg, merge_visual_rows_kernel, vis_rank, src, n_vis, hidden, out, S);
}
}  // namespace h3

extern "C" {

H3ENC_API const char *h3enc_frontend_last_error(void) { return g_err; }

H3ENC_API h3enc_status h3enc_build_positions(const int32_t *input_ids, int32_t seq_len, int32_t image_token_id,
                                             int32_t video_token_id, const int32_t *image_grid_thw,
                                             int32_t n_images, const int32_t *video_grid_thw, int32_t n_videos,
                                             int32_t spatial_merge_size, int32_t *positions,
                                             uint8_t *visual_mask, uint8_t *visual_kind,
                                             int32_t *n_image_tokens, int32_t *n_video_tokens,
                                             int32_t *mrope_delta) {
    g_err[0] = 0;
    if (seq_len < 0 || (seq_len > 0 && (!input_ids || !positions)) || n_images < 0 || n_videos < 0 ||
        (n_images && !image_grid_thw) || (n_videos && !video_grid_thw) || spatial_merge_size < 1)
        return ferr(H3ENC_ERR_INVALID_ARG, "build_positions: bad arguments");
    // grids in encounter order per modality; a video of T frames is T grids of one frame
    std::vector<int> img, vid;
    for (int i = 0; i < n_images; ++i)
        for (int k = 0; k < 3; ++k) img.push_back(image_grid_thw[3 * i + k]);
    for (int i = 0; i < n_videos; ++i)
        for (int f = 0; f < video_grid_thw[3 * i]; ++f) {
            vid.push_back(1);
            vid.push_back(video_grid_thw[3 * i + 1]);
            vid.push_back(video_grid_thw[3 * i + 2]);
        }
    size_t next_img = 0, next_vid = 0;
    int32_t cur = 0, max_pos = -1, n_img_tok = 0, n_vid_tok = 0;
    const int S = seq_len;
    int s = 0;
    while (s < S) {
        const int kind = input_ids[s] == image_token_id ? 1 : input_ids[s] == video_token_id ? 2 : 0;
        int e = s + 1;
        while (e < S && (input_ids[e] == image_token_id ? 1 : input_ids[e] == video_token_id ? 2 : 0) == kind) ++e;
        const int len = e - s;
        if (kind == 0) {
            for (int i = 0; i < len; ++i)
                for (int a = 0; a < 3; ++a) positions[a * S + s + i] = cur + i;
            max_pos = cur + len - 1 > max_pos ? cur + len - 1 : max_pos;
            cur += len;
        } else {
            std::vector<int> &grids = kind == 1 ? img : vid;
            size_t &next = kind == 1 ? next_img : next_vid;
            if (next + 3 > grids.size())
                return ferr(H3ENC_ERR_SHAPE, "build_positions: more visual runs than grids");
            const int t = grids[next], gh = grids[next + 1], gw = grids[next + 2];
            next += 3;
            if (t < 1 || gh < 1 || gw < 1 || gh % spatial_merge_size || gw % spatial_merge_size)
                return ferr(H3ENC_ERR_SHAPE, "build_positions: grid not divisible by the spatial merge size");
            const int lh = gh / spatial_merge_size, lw = gw / spatial_merge_size;
            if ((long long)t * lh * lw != len)
                return ferr(H3ENC_ERR_SHAPE, "build_positions: visual run length differs from its grid");
            int i = 0;
            for (int f = 0; f < t; ++f)
                for (int r = 0; r < lh; ++r)
                    for (int c = 0; c < lw; ++c, ++i) {
                        positions[0 * S + s + i] = cur + f;
                        positions[1 * S + s + i] = cur + r;
                        positions[2 * S + s + i] = cur + c;
                        const int m = cur + (f > r ? (f > c ? f : c) : (r > c ? r : c));
                        max_pos = m > max_pos ? m : max_pos;
                    }
            cur += (gh > gw ? gh : gw) / spatial_merge_size;
            (kind == 1 ? n_img_tok : n_vid_tok) += len;
        }
        for (int i = s; i < e; ++i) {
            if (visual_mask) visual_mask[i] = kind != 0;
            if (visual_kind) visual_kind[i] = (uint8_t)kind;
        }
        s = e;
    }
    if (n_image_tokens) *n_image_tokens = n_img_tok;
    if (n_video_tokens) *n_video_tokens = n_vid_tok;
    if (mrope_delta) *mrope_delta = max_pos + 1 - S;
    return H3ENC_OK;
}

H3ENC_API h3enc_status h3enc_aggregate_deepstack(const uint8_t *visual_kind, int32_t seq_len,
                                                 const void *image_feats, int32_t n_image_tokens,
                                                 const void *video_feats, int32_t n_video_tokens, int32_t levels,
                                                 int32_t hidden, void *out, void *stream) {
    g_err[0] = 0;
    if (seq_len < 0 || levels < 0 || hidden <= 0 || n_image_tokens < 0 || n_video_tokens < 0 ||
        (seq_len > 0 && !visual_kind) || (levels > 0 && (n_image_tokens + n_video_tokens) > 0 && !out) ||
        (n_image_tokens && !image_feats) || (n_video_tokens && !video_feats))
        return ferr(H3ENC_ERR_INVALID_ARG, "aggregate_deepstack: bad arguments");
    int ni = 0, nv = 0;
    for (int s = 0; s < seq_len; ++s) {
        if (visual_kind[s] == 1) ++ni;
        else if (visual_kind[s] == 2) ++nv;
    }
    if (ni != n_image_tokens || nv != n_video_tokens)
        return ferr(H3ENC_ERR_SHAPE, "aggregate_deepstack: feature rows differ from the visual tokens");
    const int nvis = ni + nv;
    const size_t row = (size_t)hidden * sizeof(h3::bf16);
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    int s = 0, ii = 0, vi = 0, j = 0;
    while (s < seq_len) {
        const int kind = visual_kind[s];
        int e = s + 1;
        while (e < seq_len && visual_kind[e] == kind) ++e;
        if (kind != 0) {
            const int len = e - s;
            const char *src = static_cast<const char *>(kind == 1 ? image_feats : video_feats) +
                              (size_t)(kind == 1 ? ii : vi) * row;
            const size_t spitch = (size_t)(kind == 1 ? ni : nv) * row;
            char *dst = static_cast<char *>(out) + (size_t)j * row;
            if (levels > 0) {
                cudaError_t err = cudaMemcpy2DAsync(dst, (size_t)nvis * row, src, spitch, (size_t)len * row, levels,
                                                    cudaMemcpyDeviceToDevice, st);
                if (err != cudaSuccess) return ferr(H3ENC_ERR_CUDA, cudaGetErrorString(err));
            }
            (kind == 1 ? ii : vi) += len;
            j += len;
        }
        s = e;
    }
    return H3ENC_OK;
}

}  // extern "C"
