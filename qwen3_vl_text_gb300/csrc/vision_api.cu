// C ABI of the vision tower (include/h3vis.h) and the op-level entries of its
// kernels (include/h3enc_ops.h).  The encode strings together the projection
// GEMM (bias, GELU and rotary epilogues), the attention kernel with the causal
// mask off, LayerNorm, the position-embedding sampler and the rotary tables.
//
// Page "vllm-omni vllm_omni/diffusion/models/minimax_h3/encoder.py", section
// "Qwen3-VL vision tower": MiniMaxH3Qwen3VLVisionModel.forward.
#include <cstdarg>
#include <cstdio>
#include <cstring>
#include <string>
#include <unordered_map>
#include <vector>

#include "../../include/h3enc_ops.h"
#include "../../include/h3vis.h"
#include "common.cuh"
#include "kernels.h"

using h3::bf16;

namespace {

thread_local std::string g_vis_create_error;

size_t align256(size_t x) { return (x + 255) & ~size_t(255); }

// One checkpoint tensor's place in the arena.
struct Slot {
    bf16 *ptr = nullptr;
    std::vector<int64_t> shape;
    bool loaded = false;
};

struct Block {
    bf16 *n1w, *n1b, *qkv_w, *qkv_b, *proj_w, *proj_b, *n2w, *n2b, *fc1_w, *fc1_b, *fc2_w, *fc2_b;
    CUtensorMap tm_qkv, tm_proj, tm_fc1, tm_fc2;
};

struct Merger {
    bf16 *nw, *nb, *fc1_w, *fc1_b, *fc2_w, *fc2_b;
    CUtensorMap tm_fc1, tm_fc2;
};

}  // namespace

struct h3vis {
    h3vis_config cfg;
    int num_sms = 0, G = 0;
    char *arena = nullptr, *ws = nullptr;
    std::unordered_map<std::string, Slot> slots;
    std::vector<std::string> order;   // names in registration order (missing-weights report)
    bf16 *patch_w = nullptr, *patch_b = nullptr, *pos = nullptr;
    std::vector<Block> blocks;
    Merger merger;
    std::vector<Merger> ds;
    CUtensorMap tm_patch;
    // workspace
    bf16 *x = nullptr, *y = nullptr, *qkv = nullptr, *attn = nullptr, *act = nullptr;
    float *cos_t = nullptr, *sin_t = nullptr, *part = nullptr;
    uint32_t *flags = nullptr;
    void *attn_ws = nullptr;   // attention's key-range partials (a thin last round of items)
    int32_t *status = nullptr;
    CUtensorMap tm_y, tm_attn, tm_act, tm_y4, tm_act4;
    h3::VisionRope rope;
    bool finalized = false;
    std::string err;
    int64_t launches = 0;
};

namespace {

h3enc_status vfail(h3vis *h, h3enc_status s, const char *fmt, ...) {
    char buf[2048];
    va_list ap;
    va_start(ap, fmt);
    vsnprintf(buf, sizeof buf, fmt, ap);
    va_end(ap);
    if (h) h->err = buf; else g_vis_create_error = buf;
    return s;
}

h3enc_status vcuda(h3vis *h, cudaError_t e, const char *what) {
    return vfail(h, e == cudaErrorMemoryAllocation ? H3ENC_ERR_OOM : H3ENC_ERR_CUDA, "%s: %s", what,
                 cudaGetErrorString(e));
}

h3enc_status validate(const h3vis_config *c) {
    if (!c) return vfail(nullptr, H3ENC_ERR_INVALID_ARG, "config is NULL");
    const int m = c->spatial_merge_size;
    const long pd = (long)c->in_channels * c->temporal_patch_size * c->patch_size * c->patch_size;
    if (c->depth < 1 || c->hidden < 1 || c->num_heads < 1 || c->intermediate < 1 || m < 1 || pd < 1 ||
        c->out_hidden < 1 || c->num_position_embeddings < 1 || c->max_patches < 1 || c->num_deepstack < 0 ||
        c->num_deepstack > 8 || !(c->ln_eps > 0.f) || !(c->rope_theta > 0.f))
        return vfail(nullptr, H3ENC_ERR_INVALID_ARG, "config: sizes out of range");
    const int d = c->hidden / c->num_heads, mh = c->hidden * m * m;
    if (c->hidden % c->num_heads || (d != 64 && d != 128))
        return vfail(nullptr, H3ENC_ERR_UNSUPPORTED, "config: head_dim must be 64 or 128");
    if (c->hidden % 256 || c->intermediate % 256 || c->out_hidden % 256 || mh % 256 || mh > 8192 || pd % 8 ||
        c->max_patches % (m * m))
        return vfail(nullptr, H3ENC_ERR_UNSUPPORTED, "config: widths not supported (see h3vis.h)");
    int G = 0;
    while ((G + 1) * (G + 1) <= c->num_position_embeddings) ++G;
    if (G * G != c->num_position_embeddings)
        return vfail(nullptr, H3ENC_ERR_INVALID_ARG, "config: num_position_embeddings is not a square");
    for (int j = 0; j < c->num_deepstack; ++j)
        if (c->deepstack_indexes[j] < 0 || c->deepstack_indexes[j] >= c->depth ||
            (j && c->deepstack_indexes[j] <= c->deepstack_indexes[j - 1]))
            return vfail(nullptr, H3ENC_ERR_INVALID_ARG, "config: deepstack indexes must ascend below depth");
    return H3ENC_OK;
}

// Register a tensor in the arena; returns its pointer.
bf16 *reg(h3vis *h, char *&p, const std::string &name, std::vector<int64_t> shape) {
    size_t n = 1;
    for (int64_t s : shape) n *= (size_t)s;
    Slot sl;
    sl.ptr = reinterpret_cast<bf16 *>(p);
    sl.shape = std::move(shape);
    p += align256(n * 2);
    h->slots[name] = sl;
    h->order.push_back(name);
    return h->slots[name].ptr;
}

// Bytes of the arena (the same walk as the registration, without writing).
size_t arena_bytes(const h3vis_config &c) {
    const size_t h = c.hidden, I = c.intermediate, m = c.spatial_merge_size, mh = h * m * m, o = c.out_hidden;
    const size_t pd = (size_t)c.in_channels * c.temporal_patch_size * c.patch_size * c.patch_size;
    size_t b = align256(h * pd * 2) + align256(h * 2) + align256((size_t)c.num_position_embeddings * h * 2);
    const size_t blk = 4 * align256(h * 2) + align256(3 * h * h * 2) + align256(3 * h * 2) + align256(h * h * 2) +
                       align256(h * 2) + align256(I * h * 2) + align256(I * 2) + align256(h * I * 2) + align256(h * 2);
    b += blk * (size_t)c.depth;
    auto merger = [&](size_t norm) {
        return 2 * align256(norm * 2) + align256(mh * mh * 2) + align256(mh * 2) + align256(o * mh * 2) +
               align256(o * 2);
    };
    return b + merger(h) + (size_t)c.num_deepstack * merger(mh);
}

// The projection GEMM with the tower's epilogues.
cudaError_t gemm(h3vis *h, const CUtensorMap *tA, const CUtensorMap *tW, int M, int N, int K, int epi, bf16 *C,
                 int ldc, const bf16 *R, const bf16 *bias, cudaStream_t st, bool rope = false) {
    h3::GemmPlan p{};
    p.tmA = tA; p.tmW = tW; p.M = M; p.N = N; p.K = K; p.epi = epi;
    p.C = C; p.ldc = ldc; p.R = R; p.bias = bias;
    p.status = h->status;
    p.num_sms = h->num_sms;
    p.part = h->part;
    p.flags = h->flags;
    p.w_static = true;
    if (rope) {
        const int d = h->cfg.hidden / h->cfg.num_heads;
        p.cos_t = h->cos_t; p.sin_t = h->sin_t;
        p.cs_rows = d % 8 == 0 ? h3::cs_stride(M) : 0;   // the tables' layout, as the encode writes them
        p.head_dim = d; p.nq = h->cfg.num_heads; p.nkv = h->cfg.num_heads;
    }
    ++h->launches;
    return h3::launch_gemm(p, st);
}

}  // namespace

extern "C" {

h3enc_status h3vis_create(const h3vis_config *cfg, h3vis **out) {
    if (!out) return vfail(nullptr, H3ENC_ERR_INVALID_ARG, "out is NULL");
    *out = nullptr;
    h3enc_status s = validate(cfg);
    if (s != H3ENC_OK) return s;
    h3vis *h = new h3vis();
    h->cfg = *cfg;
    const h3vis_config &c = h->cfg;
    h->num_sms = h3::device_num_sms();
    if (h->num_sms <= 0) {
        delete h;
        return vfail(nullptr, H3ENC_ERR_CUDA, "no CUDA device");
    }
    while ((h->G + 1) * (h->G + 1) <= c.num_position_embeddings) ++h->G;
    const size_t ab = arena_bytes(c);
    cudaError_t e = cudaMalloc(&h->arena, ab);
    if (e != cudaSuccess) {
        delete h;
        return vfail(nullptr, H3ENC_ERR_OOM, "vision weight arena of %zu bytes: %s", ab, cudaGetErrorString(e));
    }
    const int64_t H = c.hidden, I = c.intermediate, m = c.spatial_merge_size, MH = H * m * m, O = c.out_hidden;
    char *p = h->arena;
    const std::string pre = "model.visual.";
    h->patch_w = reg(h, p, pre + "patch_embed.proj.weight",
                     {H, c.in_channels, c.temporal_patch_size, c.patch_size, c.patch_size});
    h->patch_b = reg(h, p, pre + "patch_embed.proj.bias", {H});
    h->pos = reg(h, p, pre + "pos_embed.weight", {c.num_position_embeddings, H});
    h->blocks.resize(c.depth);
    for (int b = 0; b < c.depth; ++b) {
        const std::string q = pre + "blocks." + std::to_string(b) + ".";
        Block &k = h->blocks[b];
        k.n1w = reg(h, p, q + "norm1.weight", {H});
        k.n1b = reg(h, p, q + "norm1.bias", {H});
        k.n2w = reg(h, p, q + "norm2.weight", {H});
        k.n2b = reg(h, p, q + "norm2.bias", {H});
        k.qkv_w = reg(h, p, q + "attn.qkv.weight", {3 * H, H});
        k.qkv_b = reg(h, p, q + "attn.qkv.bias", {3 * H});
        k.proj_w = reg(h, p, q + "attn.proj.weight", {H, H});
        k.proj_b = reg(h, p, q + "attn.proj.bias", {H});
        k.fc1_w = reg(h, p, q + "mlp.linear_fc1.weight", {I, H});
        k.fc1_b = reg(h, p, q + "mlp.linear_fc1.bias", {I});
        k.fc2_w = reg(h, p, q + "mlp.linear_fc2.weight", {H, I});
        k.fc2_b = reg(h, p, q + "mlp.linear_fc2.bias", {H});
    }
    auto merger = [&](Merger &mg, const std::string &q, int64_t norm) {
        mg.nw = reg(h, p, q + "norm.weight", {norm});
        mg.nb = reg(h, p, q + "norm.bias", {norm});
        mg.fc1_w = reg(h, p, q + "linear_fc1.weight", {MH, MH});
        mg.fc1_b = reg(h, p, q + "linear_fc1.bias", {MH});
        mg.fc2_w = reg(h, p, q + "linear_fc2.weight", {O, MH});
        mg.fc2_b = reg(h, p, q + "linear_fc2.bias", {O});
    };
    merger(h->merger, pre + "merger.", H);
    h->ds.resize(c.num_deepstack);
    for (int j = 0; j < c.num_deepstack; ++j)
        merger(h->ds[j], pre + "deepstack_merger_list." + std::to_string(j) + ".", MH);
    // workspace
    const size_t P = c.max_patches, d = H / c.num_heads;
    const size_t b_x = align256(P * H * 2), b_qkv = align256(P * 3 * H * 2),
                 b_act = align256(P * (size_t)(I > H ? I : H) * 2), b_cs = align256((size_t)h3::cs_stride((int)P) * (d / 2) * 4),
                 b_gemm = align256(h3::gemm_workspace_bytes(h->num_sms)), b_st = 256,
                 b_aw = align256(h3::attention_workspace_bytes(h->num_sms, (int)d));
    const size_t wsz = 3 * b_x + b_qkv + b_act + 2 * b_cs + b_gemm + b_st + b_aw;
    e = cudaMalloc(&h->ws, wsz);
    if (e == cudaSuccess) e = cudaMemset(h->ws, 0, wsz);
    if (e != cudaSuccess) {
        h3vis_destroy(h);
        return vfail(nullptr, H3ENC_ERR_OOM, "vision workspace of %zu bytes: %s", wsz, cudaGetErrorString(e));
    }
    char *w = h->ws;
    h->x = reinterpret_cast<bf16 *>(w); w += b_x;
    h->y = reinterpret_cast<bf16 *>(w); w += b_x;
    h->attn = reinterpret_cast<bf16 *>(w); w += b_x;
    h->qkv = reinterpret_cast<bf16 *>(w); w += b_qkv;
    h->act = reinterpret_cast<bf16 *>(w); w += b_act;
    h->cos_t = reinterpret_cast<float *>(w); w += b_cs;
    h->sin_t = reinterpret_cast<float *>(w); w += b_cs;
    h->part = reinterpret_cast<float *>(w);
    h->flags = reinterpret_cast<uint32_t *>(w + h3::gemm_flags_offset(h->num_sms));
    w += b_gemm;
    h->attn_ws = w;
    w += b_aw;
    h->status = reinterpret_cast<int32_t *>(w);
    const uint32_t ba = (uint32_t)h3::gemm_box_rows_a();
    if (!h3::make_tmap_rows(&h->tm_y, h->y, P, H, ba) || !h3::make_tmap_rows(&h->tm_attn, h->attn, P, H, ba) ||
        !h3::make_tmap_rows(&h->tm_act, h->act, P, I, ba) ||
        !h3::make_tmap_rows(&h->tm_y4, h->y, P / (m * m), MH, ba) ||
        !h3::make_tmap_rows(&h->tm_act4, h->act, P / (m * m), MH, ba)) {
        h3vis_destroy(h);
        return vfail(nullptr, H3ENC_ERR_CUDA, "cuTensorMapEncodeTiled refused a workspace operand");
    }
    h3::make_vision_rope(&h->rope, (int)d, c.rope_theta);
    *out = h;
    return H3ENC_OK;
}

h3enc_status h3vis_load_weights(h3vis *h, const char *name, const void *data, int32_t dtype, const int64_t *shape,
                                int32_t ndim, int32_t data_on_device) {
    if (!h || !name || !data || !shape || ndim < 1) return vfail(h, H3ENC_ERR_INVALID_ARG, "NULL argument");
    auto it = h->slots.find(name);
    if (it == h->slots.end()) {
        vfail(h, H3ENC_WARN_IGNORED, "weight %s has no target in this configuration", name);
        return H3ENC_WARN_IGNORED;
    }
    if (dtype != H3ENC_DTYPE_BF16) return vfail(h, H3ENC_ERR_UNSUPPORTED, "%s: dtype %d is not bf16", name, dtype);
    Slot &sl = it->second;
    size_t want = 1, got = 1;
    for (int64_t s : sl.shape) want *= (size_t)s;
    for (int i = 0; i < ndim; ++i) got *= (size_t)(shape[i] > 0 ? shape[i] : 0);
    bool ok = (size_t)ndim == sl.shape.size();
    for (int i = 0; ok && i < ndim; ++i) ok = shape[i] == sl.shape[i];
    // the patch filter may also come flattened to [hidden, C*T*P*P]
    if (!ok && sl.shape.size() == 5 && ndim == 2) ok = shape[0] == sl.shape[0] && got == want;
    if (!ok) return vfail(h, H3ENC_ERR_SHAPE, "%s: shape mismatch", name);
    cudaError_t e = cudaMemcpy(sl.ptr, data, want * 2, data_on_device ? cudaMemcpyDeviceToDevice
                                                                      : cudaMemcpyHostToDevice);
    if (e != cudaSuccess) return vcuda(h, e, name);
    sl.loaded = true;
    h->finalized = false;
    return H3ENC_OK;
}

h3enc_status h3vis_finalize_weights(h3vis *h) {
    if (!h) return vfail(h, H3ENC_ERR_INVALID_ARG, "NULL handle");
    std::string missing;
    int n = 0;
    for (const auto &name : h->order)
        if (!h->slots[name].loaded) {
            if (n < 20) missing += (missing.empty() ? "" : ", ") + name;
            ++n;
        }
    if (n) return vfail(h, H3ENC_ERR_MISSING_WEIGHTS, "weights not loaded: %d: %s%s", n, missing.c_str(),
                        n > 20 ? ", ..." : "");
    const h3vis_config &c = h->cfg;
    const uint64_t H = c.hidden, I = c.intermediate, m = c.spatial_merge_size, MH = H * m * m, O = c.out_hidden;
    const uint64_t pd = (uint64_t)c.in_channels * c.temporal_patch_size * c.patch_size * c.patch_size;
    const uint32_t bw = (uint32_t)h3::gemm_box_rows_w();
    bool ok = h3::make_tmap_rows(&h->tm_patch, h->patch_w, H, pd, bw);
    for (auto &k : h->blocks)
        ok = ok && h3::make_tmap_rows(&k.tm_qkv, k.qkv_w, 3 * H, H, bw) &&
             h3::make_tmap_rows(&k.tm_proj, k.proj_w, H, H, bw) && h3::make_tmap_rows(&k.tm_fc1, k.fc1_w, I, H, bw) &&
             h3::make_tmap_rows(&k.tm_fc2, k.fc2_w, H, I, bw);
    auto mt = [&](Merger &mg) {
        return h3::make_tmap_rows(&mg.tm_fc1, mg.fc1_w, MH, MH, bw) && h3::make_tmap_rows(&mg.tm_fc2, mg.fc2_w, O, MH, bw);
    };
    ok = ok && mt(h->merger);
    for (auto &mg : h->ds) ok = ok && mt(mg);
    if (!ok) return vfail(h, H3ENC_ERR_CUDA, "cuTensorMapEncodeTiled refused a weight operand");
    h->finalized = true;
    return H3ENC_OK;
}

h3enc_status h3vis_encode(h3vis *h, const void *pixel_values, int32_t n_patches, const int32_t *grid_thw,
                          int32_t n_grids, void *embeds_out, void *deepstack_out, void *stream) {
    if (!h) return vfail(h, H3ENC_ERR_INVALID_ARG, "NULL handle");
    if (!h->finalized) return vfail(h, H3ENC_ERR_NOT_LOADED, "weights not finalized (call h3vis_finalize_weights)");
    const h3vis_config &c = h->cfg;
    if (!pixel_values || !grid_thw || !embeds_out || n_patches < 1 || n_patches > c.max_patches)   // deepstack_out may be NULL
        return vfail(h, H3ENC_ERR_INVALID_ARG, "bad arguments (n_patches %d, max_patches %d)", n_patches,
                     c.max_patches);
    const int m = c.spatial_merge_size;
    h3::VisionGrids gr;
    int n = 0;
    if (!h3::make_vision_grids(&gr, grid_thw, n_grids, m, &n))
        return vfail(h, H3ENC_ERR_INVALID_ARG, "grid_thw: empty grid, more than 64 grids, or rows / columns not "
                                               "divisible by the spatial merge size");
    if (n != n_patches) return vfail(h, H3ENC_ERR_SHAPE, "grid_thw gives %d patches, n_patches is %d", n, n_patches);
    std::vector<int32_t> cu{0};   // one attention segment per frame
    for (int g = 0; g < n_grids; ++g)
        for (int f = 0; f < grid_thw[3 * g]; ++f) cu.push_back(cu.back() + grid_thw[3 * g + 1] * grid_thw[3 * g + 2]);
    if ((int)cu.size() - 1 > h3::kMaxSeqs) return vfail(h, H3ENC_ERR_INVALID_ARG, "more than %d frames", h3::kMaxSeqs);
    if ((reinterpret_cast<uintptr_t>(pixel_values) | reinterpret_cast<uintptr_t>(embeds_out) |
         reinterpret_cast<uintptr_t>(deepstack_out)) & 15)
        return vfail(h, H3ENC_ERR_INVALID_ARG, "device buffers must be 16-byte aligned");
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    const int H = c.hidden, I = c.intermediate, heads = c.num_heads, d = H / heads, MH = H * m * m, O = c.out_hidden;
    const int pd = c.in_channels * c.temporal_patch_size * c.patch_size * c.patch_size;
    const int nm = n / (m * m);
    CUtensorMap tm_px;
    if (!h3::make_tmap_rows(&tm_px, pixel_values, n, pd, h3::gemm_box_rows_a()))
        return vfail(h, H3ENC_ERR_INVALID_ARG, "pixel_values refused by the tensor map (alignment)");
    cudaError_t e;
#define VCHECK(call, what) do { e = (call); ++h->launches; if (e != cudaSuccess) return vcuda(h, e, what); } while (0)
    // patch embedding + sampled position embeddings: x = bf16(pixels W^T + b + pos)
    VCHECK(h3::launch_pos_embed(h->pos, h->G, H, gr, n, h->x, st), "position embeddings");
    e = gemm(h, &tm_px, &h->tm_patch, n, H, pd, h3::EPI_RESIDUAL, h->x, H, h->x, h->patch_b, st);
    if (e != cudaSuccess) return vcuda(h, e, "patch embedding");
    // row-interleaved (head_dim % 8 == 0): the QKV epilogue's warps read them as whole lines
    VCHECK(h3::launch_vision_rope(gr, n, d, h->rope, h->cos_t, h->sin_t, st, d % 8 == 0 ? h3::cs_stride(n) : 0),
           "rotary tables");
    for (int b = 0; b < c.depth; ++b) {
        const Block &k = h->blocks[b];
        VCHECK(h3::launch_layernorm(h->x, k.n1w, k.n1b, h->y, n, H, c.ln_eps, st), "norm1");
        e = gemm(h, &h->tm_y, &k.tm_qkv, n, 3 * H, H, h3::EPI_QKROPE, h->qkv, 3 * H, nullptr, k.qkv_b, st, true);
        if (e != cudaSuccess) return vcuda(h, e, "qkv");
        VCHECK(h3::launch_attention(h->qkv, h->attn, n, heads, heads, d, cu.data(), (int)cu.size() - 1, h->status,
                                    st, nullptr, false, h->attn_ws, h3::attention_workspace_bytes(h->num_sms, d)),
               "attention");
        e = gemm(h, &h->tm_attn, &k.tm_proj, n, H, H, h3::EPI_RESIDUAL, h->x, H, h->x, k.proj_b, st);
        if (e != cudaSuccess) return vcuda(h, e, "proj");
        VCHECK(h3::launch_layernorm(h->x, k.n2w, k.n2b, h->y, n, H, c.ln_eps, st), "norm2");
        e = gemm(h, &h->tm_y, &k.tm_fc1, n, I, H, h3::EPI_GELU_TANH, h->act, I, nullptr, k.fc1_b, st);
        if (e != cudaSuccess) return vcuda(h, e, "fc1");
        e = gemm(h, &h->tm_act, &k.tm_fc2, n, H, I, h3::EPI_RESIDUAL, h->x, H, h->x, k.fc2_b, st);
        if (e != cudaSuccess) return vcuda(h, e, "fc2");
        for (int j = 0; j < c.num_deepstack; ++j) {
            if (c.deepstack_indexes[j] != b || !deepstack_out) continue;
            // DeepStack merger: the m*m patches of a block as one row, LayerNorm over it, fc1, GELU, fc2
            const Merger &mg = h->ds[j];
            VCHECK(h3::launch_layernorm(h->x, mg.nw, mg.nb, h->y, nm, MH, c.ln_eps, st), "deepstack norm");
            e = gemm(h, &h->tm_y4, &mg.tm_fc1, nm, MH, MH, h3::EPI_GELU_ERF, h->act, MH, nullptr, mg.fc1_b, st);
            if (e != cudaSuccess) return vcuda(h, e, "deepstack fc1");
            bf16 *dst = static_cast<bf16 *>(deepstack_out) + (size_t)j * nm * O;
            e = gemm(h, &h->tm_act4, &mg.tm_fc2, nm, O, MH, h3::EPI_STORE, dst, O, nullptr, mg.fc2_b, st);
            if (e != cudaSuccess) return vcuda(h, e, "deepstack fc2");
        }
    }
    // main merger: LayerNorm per patch, then the block's patches as one row, fc1, GELU, fc2
    VCHECK(h3::launch_layernorm(h->x, h->merger.nw, h->merger.nb, h->y, n, H, c.ln_eps, st), "merger norm");
    e = gemm(h, &h->tm_y4, &h->merger.tm_fc1, nm, MH, MH, h3::EPI_GELU_ERF, h->act, MH, nullptr, h->merger.fc1_b, st);
    if (e != cudaSuccess) return vcuda(h, e, "merger fc1");
    e = gemm(h, &h->tm_act4, &h->merger.tm_fc2, nm, O, MH, h3::EPI_STORE, static_cast<bf16 *>(embeds_out), O, nullptr,
             h->merger.fc2_b, st);
    if (e != cudaSuccess) return vcuda(h, e, "merger fc2");
#undef VCHECK
    return H3ENC_OK;
}

h3enc_status h3vis_get_status(h3vis *h) {
    if (!h) return vfail(h, H3ENC_ERR_INVALID_ARG, "NULL handle");
    cudaError_t e = cudaDeviceSynchronize();
    if (e != cudaSuccess) return vcuda(h, e, "device synchronise");
    int32_t st = 0;
    e = cudaMemcpy(&st, h->status, 4, cudaMemcpyDeviceToHost);
    if (e == cudaSuccess) e = cudaMemset(h->status, 0, 4);
    if (e != cudaSuccess) return vcuda(h, e, "status read");
    if (st & 1) {
        // an aborted attention launch may leave key-range arrival counts behind: start them again
        if (h->attn_ws) cudaMemset(h->attn_ws, 0, h3::attention_workspace_bytes(h->num_sms, h->cfg.hidden / h->cfg.num_heads));
        return vfail(h, H3ENC_ERR_DEVICE_TIMEOUT, "a bounded device wait ran out");
    }
    return st ? vfail(h, H3ENC_ERR_CUDA, "device status 0x%x", st) : H3ENC_OK;
}

const char *h3vis_last_error(const h3vis *h) { return h ? h->err.c_str() : g_vis_create_error.c_str(); }

int64_t h3vis_launch_count(const h3vis *h) { return h ? h->launches : 0; }

void h3vis_destroy(h3vis *h) {
    if (!h) return;
    cudaFree(h->arena);
    cudaFree(h->ws);
    delete h;
}

// ---------------------------------------------------------------- op-level entries

h3enc_status h3enc_op_layernorm(const void *x, const void *w, const void *b, void *y, int32_t rows, int32_t cols,
                                float eps, void *stream) {
    if (!x || !w || !b || !y || rows < 0 || cols <= 0 || cols % 8 || cols > 8192)
        return H3ENC_ERR_INVALID_ARG;
    cudaError_t e = h3::launch_layernorm(static_cast<const bf16 *>(x), static_cast<const bf16 *>(w),
                                         static_cast<const bf16 *>(b), static_cast<bf16 *>(y), rows, cols, eps,
                                         static_cast<cudaStream_t>(stream));
    return e == cudaSuccess ? H3ENC_OK : H3ENC_ERR_CUDA;
}

h3enc_status h3enc_op_vision_pos_embed(const void *table, int32_t grid_side, int32_t hidden,
                                       const int32_t *grid_thw, int32_t n_grids, int32_t merge, void *out,
                                       void *stream) {
    h3::VisionGrids gr;
    int n = 0;
    if (!table || !out || grid_side < 1 || hidden <= 0 || hidden % 8 || !grid_thw ||
        !h3::make_vision_grids(&gr, grid_thw, n_grids, merge, &n))
        return H3ENC_ERR_INVALID_ARG;
    cudaError_t e = h3::launch_pos_embed(static_cast<const bf16 *>(table), grid_side, hidden, gr, n,
                                         static_cast<bf16 *>(out), static_cast<cudaStream_t>(stream));
    return e == cudaSuccess ? H3ENC_OK : H3ENC_ERR_CUDA;
}

h3enc_status h3enc_op_vision_rope_table(const int32_t *grid_thw, int32_t n_grids, int32_t merge, int32_t head_dim,
                                        float theta, float *cos_tab, float *sin_tab, void *stream) {
    h3::VisionGrids gr;
    int n = 0;
    if (!grid_thw || !cos_tab || !sin_tab || head_dim < 4 || head_dim % 4 || head_dim > 2 * h3::kMaxHalfDim ||
        !(theta > 0.f) || !h3::make_vision_grids(&gr, grid_thw, n_grids, merge, &n))
        return H3ENC_ERR_INVALID_ARG;
    h3::VisionRope rp;
    h3::make_vision_rope(&rp, head_dim, theta);
    cudaError_t e = h3::launch_vision_rope(gr, n, head_dim, rp, cos_tab, sin_tab, static_cast<cudaStream_t>(stream));
    return e == cudaSuccess ? H3ENC_OK : H3ENC_ERR_CUDA;
}

h3enc_status h3enc_op_gemm_bias(const void *A, const void *W, void *C, int32_t M, int32_t N, int32_t K,
                                int32_t epilogue, const void *R, const void *bias, void *workspace,
                                int64_t workspace_bytes, int32_t *status, void *stream) {
    // epilogue: H3ENC_EPI_STORE, H3ENC_EPI_RESIDUAL, H3ENC_EPI_GELU_TANH or H3ENC_EPI_GELU_ERF
    if (M < 0 || N <= 0 || K <= 0 || N % 256 || K % 8 || !bias ||
        (epilogue != H3ENC_EPI_STORE && epilogue != H3ENC_EPI_RESIDUAL && epilogue != H3ENC_EPI_GELU_TANH &&
         epilogue != H3ENC_EPI_GELU_ERF) || (epilogue == H3ENC_EPI_RESIDUAL && !R))
        return H3ENC_ERR_INVALID_ARG;
    if (M == 0) return H3ENC_OK;
    if (!A || !W || !C) return H3ENC_ERR_INVALID_ARG;
    CUtensorMap ta, tw;
    if (!h3::make_tmap_rows(&ta, A, M, K, h3::gemm_box_rows_a()) || !h3::make_tmap_rows(&tw, W, N, K, h3::gemm_box_rows_w()))
        return H3ENC_ERR_INVALID_ARG;
    h3::GemmPlan p{};
    p.tmA = &ta; p.tmW = &tw; p.M = M; p.N = N; p.K = K; p.epi = epilogue;
    p.C = static_cast<bf16 *>(C); p.ldc = N; p.R = static_cast<const bf16 *>(R); p.bias = static_cast<const bf16 *>(bias);
    p.status = status;
    p.num_sms = h3::device_num_sms();
    if (workspace) {
        if (workspace_bytes < (int64_t)h3::gemm_workspace_bytes(p.num_sms) || (reinterpret_cast<uintptr_t>(workspace) & 255))
            return H3ENC_ERR_INVALID_ARG;
        p.part = static_cast<float *>(workspace);
        p.flags = reinterpret_cast<uint32_t *>(static_cast<char *>(workspace) + h3::gemm_flags_offset(p.num_sms));
    }
    cudaError_t e = h3::launch_gemm(p, static_cast<cudaStream_t>(stream));
    return e == cudaSuccess ? H3ENC_OK : H3ENC_ERR_CUDA;
}

h3enc_status h3enc_op_gemm_qkv_rope_bias(const void *A, const void *W, void *C, int32_t M, int32_t K, int32_t heads,
                                         int32_t head_dim, const void *bias, const float *cos_tab,
                                         const float *sin_tab, void *workspace, int64_t workspace_bytes,
                                         int32_t *status, void *stream) {
    const int64_t N = 3LL * heads * head_dim;
    if (M < 0 || K <= 0 || K % 8 || heads < 1 || (head_dim != 64 && head_dim != 128) || N % 256 || !bias ||
        !cos_tab || !sin_tab)
        return H3ENC_ERR_INVALID_ARG;
    if (M == 0) return H3ENC_OK;
    if (!A || !W || !C) return H3ENC_ERR_INVALID_ARG;
    CUtensorMap ta, tw;
    if (!h3::make_tmap_rows(&ta, A, M, K, h3::gemm_box_rows_a()) || !h3::make_tmap_rows(&tw, W, N, K, h3::gemm_box_rows_w()))
        return H3ENC_ERR_INVALID_ARG;
    h3::GemmPlan p{};
    p.tmA = &ta; p.tmW = &tw; p.M = M; p.N = (int)N; p.K = K; p.epi = h3::EPI_QKROPE;
    p.C = static_cast<bf16 *>(C); p.ldc = (int)N; p.bias = static_cast<const bf16 *>(bias);
    p.cos_t = cos_tab; p.sin_t = sin_tab;
    p.head_dim = head_dim; p.nq = heads; p.nkv = heads;
    p.status = status;
    p.num_sms = h3::device_num_sms();
    if (workspace) {
        if (workspace_bytes < (int64_t)h3::gemm_workspace_bytes(p.num_sms) || (reinterpret_cast<uintptr_t>(workspace) & 255))
            return H3ENC_ERR_INVALID_ARG;
        p.part = static_cast<float *>(workspace);
        p.flags = reinterpret_cast<uint32_t *>(static_cast<char *>(workspace) + h3::gemm_flags_offset(p.num_sms));
    }
    cudaError_t e = h3::launch_gemm(p, static_cast<cudaStream_t>(stream));
    return e == cudaSuccess ? H3ENC_OK : H3ENC_ERR_CUDA;
}

h3enc_status h3enc_op_attention_bidir(const void *qkv, void *o, int32_t S, int32_t heads, int32_t head_dim,
                                      const int32_t *cu_seqlens, int32_t n_seqs, void *stream) {
    if (!qkv || !o || S < 0 || heads < 1 || (head_dim != 64 && head_dim != 128)) return H3ENC_ERR_INVALID_ARG;
    if (cu_seqlens) {
        if (n_seqs < 1 || n_seqs > h3::kMaxSeqs || cu_seqlens[0] != 0 || cu_seqlens[n_seqs] != S)
            return H3ENC_ERR_INVALID_ARG;
        for (int i = 0; i < n_seqs; ++i)
            if (cu_seqlens[i + 1] < cu_seqlens[i]) return H3ENC_ERR_INVALID_ARG;
    }
    cudaError_t e = h3::launch_attention(static_cast<const bf16 *>(qkv), static_cast<bf16 *>(o), S, heads, heads,
                                         head_dim, cu_seqlens, cu_seqlens ? n_seqs : 0, nullptr,
                                         static_cast<cudaStream_t>(stream), nullptr, false);
    return e == cudaSuccess ? H3ENC_OK : H3ENC_ERR_CUDA;
}

int64_t h3enc_op_attention_workspace_bytes(int32_t head_dim) {
    if (head_dim != 64 && head_dim != 128) return 0;
    return (int64_t)h3::attention_workspace_bytes(h3::device_num_sms(), head_dim);
}

h3enc_status h3enc_op_attention_bidir_ws(const void *qkv, void *o, int32_t S, int32_t heads, int32_t head_dim,
                                         const int32_t *cu_seqlens, int32_t n_seqs, void *workspace,
                                         int64_t workspace_bytes, void *stream) {
    if (!qkv || !o || S < 0 || heads < 1 || (head_dim != 64 && head_dim != 128) || !workspace ||
        workspace_bytes < h3enc_op_attention_workspace_bytes(head_dim) || (reinterpret_cast<uintptr_t>(workspace) & 15))
        return H3ENC_ERR_INVALID_ARG;
    if (cu_seqlens) {
        if (n_seqs < 1 || n_seqs > h3::kMaxSeqs || cu_seqlens[0] != 0 || cu_seqlens[n_seqs] != S)
            return H3ENC_ERR_INVALID_ARG;
        for (int i = 0; i < n_seqs; ++i)
            if (cu_seqlens[i + 1] < cu_seqlens[i]) return H3ENC_ERR_INVALID_ARG;
    }
    cudaError_t e = h3::launch_attention(static_cast<const bf16 *>(qkv), static_cast<bf16 *>(o), S, heads, heads,
                                         head_dim, cu_seqlens, cu_seqlens ? n_seqs : 0, nullptr,
                                         static_cast<cudaStream_t>(stream), nullptr, false, workspace,
                                         (size_t)workspace_bytes);
    return e == cudaSuccess ? H3ENC_OK : H3ENC_ERR_CUDA;
}

}  // extern "C"
