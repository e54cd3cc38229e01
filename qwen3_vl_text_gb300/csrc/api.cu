// C ABI of the encoder: handle, weight loading and packing, encode orchestration.
//
// One encode enqueues, on the caller's stream and without host synchronisation:
//   embedding gather (or input copy) -> M-RoPE tables -> visual ranks (if DeepStack)
//   per layer: RMSNorm -> QKV GEMM -> q/k RMSNorm + M-RoPE -> attention ->
//              o GEMM (+residual) -> RMSNorm -> gate/up GEMM (SwiGLU) ->
//              down GEMM (+residual, +DeepStack for layers < levels)
// following MiniMaxH3Qwen3VLTextModel.forward and MiniMaxH3Qwen3VLTextDecoderLayer.
// forward (page "vllm-omni vllm_omni/diffusion/models/minimax_h3/encoder.py").
// The hidden state lives in the caller's output buffer for the whole encode.
#include <algorithm>
#include <cstdarg>
#include <cstdio>
#include <cstdlib>
#include <cstring>
#include <string>
#include <vector>

#include "../../include/h3enc.h"
#include "../../include/h3enc_ops.h"
#include "kernels.h"

#include <nvtx3/nvToolsExt.h>

using h3::bf16;

namespace {

enum { T_IN = 0, T_Q, T_K, T_V, T_QN, T_KN, T_O, T_POST, T_GATE, T_UP, T_DOWN, T_COUNT };
const char *kSuffix[T_COUNT] = {
    "input_layernorm.weight", "self_attn.q_proj.weight", "self_attn.k_proj.weight", "self_attn.v_proj.weight",
    "self_attn.q_norm.weight", "self_attn.k_norm.weight", "self_attn.o_proj.weight",
    "post_attention_layernorm.weight", "mlp.gate_proj.weight", "mlp.up_proj.weight", "mlp.down_proj.weight"};

struct LayerW {
    bf16 *qkv = nullptr, *o = nullptr, *gu = nullptr, *down = nullptr;
    bf16 *in_norm = nullptr, *post_norm = nullptr, *q_norm = nullptr, *k_norm = nullptr;
    CUtensorMap tm_qkv, tm_o, tm_gu, tm_down;
    uint32_t loaded = 0;
    // RMSNorm folded into the projections: shards (bits 1 << T_Q, T_K, T_V, T_GATE, T_UP) whose
    // arena rows already carry their norm weight; a norm reloaded while its projections are
    // folded marks them stale until they are reloaded too
    uint32_t folded = 0;
    bool in_stale = false, post_stale = false;
};

constexpr uint32_t kQKVBits = (1u << T_Q) | (1u << T_K) | (1u << T_V);
constexpr uint32_t kGUBits = (1u << T_GATE) | (1u << T_UP);

thread_local std::string g_create_error;

size_t align256(size_t x) { return (x + 255) & ~size_t(255); }

}  // namespace

struct h3enc {
    h3enc_config cfg;
    int device = 0;
    int num_sms = 0;
    int qkv_out = 0;
    h3::RopeParams rope;
    char *arena = nullptr;
    bf16 *embed = nullptr;
    bool embed_loaded = false;
    std::vector<LayerW> layers;
    char *ws = nullptr;
    bf16 *y = nullptr, *qkv = nullptr, *attn = nullptr, *act = nullptr;
    float *cos_t = nullptr, *sin_t = nullptr;
    int32_t *vis_rank = nullptr, *status = nullptr;
    float *gemm_part = nullptr;      // split-GEMM partials (num_sms x 128 x 256 fp32)
    uint32_t *gemm_flags = nullptr;  // split-GEMM release flags
    int32_t *st_ids = nullptr, *st_pos = nullptr;
    uint8_t *st_mask = nullptr;
    bf16 *st_ds = nullptr, *st_out = nullptr;
    CUtensorMap tm_y, tm_attn, tm_act;
    // RMSNorm folded into the projections (bf16, separate_norm == 0): per-row sums of squares of
    // the hidden state over slots of 128 columns, [hidden / 128][rows of the encode]
    float *row_ss = nullptr;
    // online FP8 (linear_fp8): e4m3 copies of the four projections with per-row scales, e4m3
    // activations with per-token scales
    struct Layer8 {
        uint8_t *qkv, *o, *gu, *down;
        float *s_qkv, *s_o, *s_gu, *s_down;
        CUtensorMap tm_qkv, tm_o, tm_gu, tm_down;
    };
    char *arena8 = nullptr, *ws8 = nullptr;
    std::vector<Layer8> layers8;
    uint8_t *y8 = nullptr, *attn8 = nullptr, *act8 = nullptr;
    float *sy = nullptr, *sattn = nullptr, *sact = nullptr;
    float *amax_attn = nullptr, *amax_act = nullptr;   // per-row |max| published by the producers
    CUtensorMap tm_y8, tm_attn8, tm_act8;
    bool finalized = false;
    std::string err;
    std::vector<void *> capture;
    bool prof = false;
    uint32_t prof_mask = 0;
    int prof_layer = -1;   // time only this decoder layer's launches (-1: every launch)
    int cur_layer = -1;    // the layer encode_core is issuing (-1 outside the layer loop)
    std::vector<cudaEvent_t> ev_pool;
    std::vector<int> ev_class;
    size_t ev_used = 0;
    double ms[H3ENC_K_COUNT] = {0};
    int64_t launches[H3ENC_K_COUNT] = {0};
    int64_t launch_count = 0;
    // h3enc_encode_host's CUDA graphs: one per distinct call shape (every pointer the encode
    // reads or writes is a staging or workspace buffer of the handle, fixed at create), replayed
    // instead of issuing the launches again; least recently used beyond kMaxGraphs is dropped
    struct Graph {
        int S = 0, n_seqs = 0, n_vis = 0, nds = 0;
        bool mask = false;
        std::vector<int32_t> cu;
        cudaGraphExec_t exec = nullptr;   // null until the shape's second call
        bool failed = false;              // its capture failed: it runs eagerly
        bool waits_ds = false;            // it holds a wait for the DeepStack copy
        int64_t launches = 0;             // kernels one replay runs
        uint64_t used = 0;
    };
    static constexpr size_t kMaxGraphs = 8;
    std::vector<Graph> graphs;
    uint64_t graph_tick = 0;
    bool use_graphs = true;
    // h3enc_encode_host's DeepStack copy runs on a stream of its own, so that it lands while
    // the first layer computes; the encode waits for it just before the first DeepStack add
    cudaStream_t copy_st = nullptr;
    cudaEvent_t ds_fork = nullptr, ds_ready = nullptr;
    bool ds_pending = false;   // set while encode_core is to wait for ds_ready
};

namespace {

h3enc_status fail(h3enc *h, h3enc_status s, const char *fmt, ...) {
    char buf[2048];
    va_list ap;
    va_start(ap, fmt);
    vsnprintf(buf, sizeof buf, fmt, ap);
    va_end(ap);
    if (h) h->err = buf; else g_create_error = buf;
    return s;
}

h3enc_status cuda_fail(h3enc *h, cudaError_t e, const char *what) {
    return fail(h, e == cudaErrorMemoryAllocation ? H3ENC_ERR_OOM : H3ENC_ERR_CUDA, "%s: %s", what,
                cudaGetErrorString(e));
}

// Run one kernel launch, timed per class when profiling is on.
// NVTX ranges (encode, layer, launch) for timeline tools; without an attached tool each
// push/pop is a few nanoseconds.  Popped on scope exit, error returns included.
struct NvtxRange {
    explicit NvtxRange(const char *name) { nvtxRangePushA(name); }
    ~NvtxRange() { nvtxRangePop(); }
    NvtxRange(const NvtxRange &) = delete;
    NvtxRange &operator=(const NvtxRange &) = delete;
};
const char *const kClassName[H3ENC_K_COUNT] = {"prep",      "rmsnorm", "gemm_qkv",     "quant",
                                               "attention", "gemm_o",  "gemm_gate_up", "gemm_down"};

// Under stream capture the timing events become event-record nodes of the graph, so every
// replay records them again and the host reads the latest replay's durations.
inline void record_timing_event(cudaEvent_t ev, cudaStream_t st) {
    cudaStreamCaptureStatus cs = cudaStreamCaptureStatusNone;
    if (cudaStreamIsCapturing(st, &cs) != cudaSuccess) cs = cudaStreamCaptureStatusNone;
    cudaEventRecordWithFlags(ev, st, cs == cudaStreamCaptureStatusActive ? cudaEventRecordExternal : 0u);
}

template <class F>
cudaError_t run(h3enc *h, int cls, cudaStream_t st, F &&launch) {
    NvtxRange range(kClassName[cls]);
    size_t e0 = (size_t)-1;
    if (h->prof && (h->prof_mask & (1u << cls)) && (h->prof_layer < 0 || h->prof_layer == h->cur_layer)) {
        if (h->ev_used + 2 > h->ev_pool.size()) {
            for (int i = 0; i < 256; ++i) {
                cudaEvent_t ev;
                if (cudaEventCreate(&ev) != cudaSuccess) break;
                h->ev_pool.push_back(ev);
                h->ev_class.push_back(0);
            }
        }
        if (h->ev_used + 2 <= h->ev_pool.size()) {
            e0 = h->ev_used;
            record_timing_event(h->ev_pool[e0], st);
        } else {
            e0 = (size_t)-1;
        }
    }
    cudaError_t e = launch();
    if (e0 != (size_t)-1) {
        record_timing_event(h->ev_pool[e0 + 1], st);
        h->ev_class[e0] = cls;
        h->ev_used += 2;
        h->launches[cls]++;   // timed launches of the class
    }
    h->launch_count++;
    return e;
}

// bf16 encodes fold the two RMSNorms into the projections unless asked for separate passes;
// the FP8 path quantises the norm's output and keeps its own pass.
bool norm_folded(const h3enc_config &c) { return !c.linear_fp8 && !c.separate_norm; }

// Multiply each layer's input_layernorm weight into the q/k/v rows and its
// post_attention_layernorm weight into the gate/up rows (along K), for the shards not yet
// folded.  A norm changed after its projections were folded cannot be applied to them.
h3enc_status fold_norms(h3enc *h) {
    const h3enc_config &c = h->cfg;
    const int H = c.hidden, qr = c.n_heads * c.head_dim, kr = c.n_kv_heads * c.head_dim;
    std::string stale;
    for (int l = 0; l < c.num_layers; ++l) {
        const LayerW &w = h->layers[l];
        if (w.in_stale && (w.folded & kQKVBits))
            stale += " layers." + std::to_string(l) + ": reload q/k/v_proj (input_layernorm changed)";
        if (w.post_stale && (w.folded & kGUBits))
            stale += " layers." + std::to_string(l) + ": reload gate/up_proj (post_attention_layernorm changed)";
    }
    if (!stale.empty())
        return fail(h, H3ENC_ERR_MISSING_WEIGHTS,
                    "norm weights changed after their projections were folded at finalize:%s", stale.c_str());
    cudaError_t e = cudaSuccess;
    for (auto &w : h->layers) {
        const struct { int bit, r0, r1, blk, parity; const bf16 *g; bf16 *W; } shards[5] = {
            {T_Q, 0, qr, 0, 0, w.in_norm, w.qkv},
            {T_K, qr, qr + kr, 0, 0, w.in_norm, w.qkv},
            {T_V, qr + kr, qr + 2 * kr, 0, 0, w.in_norm, w.qkv},
            {T_GATE, 0, 2 * c.intermediate, 128, 0, w.post_norm, w.gu},   // packed: 128-row blocks
            {T_UP, 0, 2 * c.intermediate, 128, 1, w.post_norm, w.gu},     // alternate gate / up
        };
        for (const auto &sh : shards) {
            if (w.folded & (1u << sh.bit)) continue;
            e = h3::launch_fold_cols(sh.W, H, sh.g, sh.r0, sh.r1, sh.blk, sh.parity, 0);
            if (e != cudaSuccess) return cuda_fail(h, e, "norm fold");
            w.folded |= 1u << sh.bit;
        }
        w.in_stale = w.post_stale = false;
    }
    e = cudaStreamSynchronize(0);
    return e == cudaSuccess ? H3ENC_OK : cuda_fail(h, e, "norm fold");
}

h3enc_status validate_config(const h3enc_config *c) {
    if (!c) return fail(nullptr, H3ENC_ERR_INVALID_ARG, "config is NULL");
    if (c->num_layers < 1 || c->hidden < 1 || c->n_heads < 1 || c->n_kv_heads < 1 || c->intermediate < 1 ||
        c->vocab < 0 || c->max_tokens < 1 || c->max_seqs < 1 || c->max_seqs > h3::kMaxSeqs ||
        c->num_deepstack < 0)
        return fail(nullptr, H3ENC_ERR_INVALID_ARG, "config: sizes out of range");
    if (!(c->rms_eps > 0.f) || !(c->rope_theta > 0.f))
        return fail(nullptr, H3ENC_ERR_INVALID_ARG, "config: rms_eps and rope_theta must be > 0");
    if (c->mrope_section[0] < 0 || c->mrope_section[1] < 0 || c->mrope_section[2] < 0)
        return fail(nullptr, H3ENC_ERR_INVALID_ARG, "config: negative mrope_section");
    if (c->linear_fp8 != 0 && c->linear_fp8 != 1)
        return fail(nullptr, H3ENC_ERR_INVALID_ARG, "config: linear_fp8 must be 0 or 1");
    if (c->separate_norm != 0 && c->separate_norm != 1)
        return fail(nullptr, H3ENC_ERR_INVALID_ARG, "config: separate_norm must be 0 or 1");
    if (c->head_dim != 64 && c->head_dim != 128)
        return fail(nullptr, H3ENC_ERR_UNSUPPORTED, "config: head_dim %d not in {64, 128}", c->head_dim);
    if (c->n_heads % c->n_kv_heads)
        return fail(nullptr, H3ENC_ERR_INVALID_ARG, "config: n_heads %% n_kv_heads != 0");
    const long long qkv = (long long)(c->n_heads + 2 * c->n_kv_heads) * c->head_dim;
    if (c->hidden % 256 || qkv % 256 || (c->n_heads * c->head_dim) % 64 || c->intermediate % 128 ||
        c->hidden > 8192)
        return fail(nullptr, H3ENC_ERR_UNSUPPORTED,
                    "config: need hidden %% 256 == 0 (<= 8192), qkv width %% 256 == 0, n_heads*head_dim %% 64 "
                    "== 0, intermediate %% 128 == 0");
    return H3ENC_OK;
}

struct Sizes {
    size_t qkv, o, gu, down, norm_h, norm_d, layer, embed;
};

Sizes weight_sizes(const h3enc_config &c) {
    Sizes s;
    const size_t H = c.hidden, d = c.head_dim;
    s.qkv = align256((size_t)(c.n_heads + 2 * c.n_kv_heads) * d * H * 2);
    s.o = align256(H * c.n_heads * d * 2);
    s.gu = align256((size_t)2 * c.intermediate * H * 2);
    s.down = align256(H * (size_t)c.intermediate * 2);
    s.norm_h = align256(H * 2);
    s.norm_d = align256(d * 2);
    s.layer = s.qkv + s.o + s.gu + s.down + 2 * s.norm_h + 2 * s.norm_d;
    s.embed = align256((size_t)c.vocab * H * 2);
    return s;
}

bool parse_layer_name(const char *name, int *layer, int *which) {
    static const char kPre[] = "model.language_model.layers.";
    const size_t n = sizeof(kPre) - 1;
    if (strncmp(name, kPre, n) != 0) return false;
    const char *p = name + n;
    if (*p < '0' || *p > '9') return false;
    long l = 0;
    while (*p >= '0' && *p <= '9') {
        l = l * 10 + (*p - '0');
        if (l > 1000000) return false;
        ++p;
    }
    if (*p != '.') return false;
    ++p;
    for (int t = 0; t < T_COUNT; ++t)
        if (strcmp(p, kSuffix[t]) == 0) {
            *layer = (int)l;
            *which = t;
            return true;
        }
    *layer = (int)l;
    *which = -1;
    return true;
}

h3enc_status check_seqs(h3enc *h, const int32_t *cu, int n_seqs, int S) {
    if (!cu) return H3ENC_OK;
    if (n_seqs < 1 || n_seqs > h->cfg.max_seqs)
        return fail(h, H3ENC_ERR_INVALID_ARG, "n_seqs %d outside [1, %d]", n_seqs, h->cfg.max_seqs);
    if (cu[0] != 0 || cu[n_seqs] != S)
        return fail(h, H3ENC_ERR_INVALID_ARG, "cu_seqlens must start at 0 and end at seq_len %d", S);
    for (int i = 0; i < n_seqs; ++i)
        if (cu[i + 1] < cu[i]) return fail(h, H3ENC_ERR_INVALID_ARG, "cu_seqlens decreases at %d", i);
    return H3ENC_OK;
}

h3enc_status check_encode_args(h3enc *h, const void *positions, const uint8_t *mask, const void *ds, int nds,
                               int n_vis, const int32_t *cu, int n_seqs, int S, const void *out) {
    if (!h->finalized) return fail(h, H3ENC_ERR_NOT_LOADED, "weights not finalized (call h3enc_finalize_weights)");
    if (S < 0 || S > h->cfg.max_tokens)
        return fail(h, H3ENC_ERR_INVALID_ARG, "seq_len %d outside [0, max_tokens=%d]", S, h->cfg.max_tokens);
    if (S > 0 && (!positions || !out)) return fail(h, H3ENC_ERR_INVALID_ARG, "positions and out must be non-NULL");
    if (nds < 0 || nds > h->cfg.num_deepstack)
        return fail(h, H3ENC_ERR_INVALID_ARG, "num_deepstack %d outside [0, %d]", nds, h->cfg.num_deepstack);
    if (n_vis < 0 || n_vis > S) return fail(h, H3ENC_ERR_INVALID_ARG, "n_vis %d outside [0, seq_len]", n_vis);
    if (nds > 0 && n_vis > 0 && (!mask || !ds))
        return fail(h, H3ENC_ERR_INVALID_ARG, "DeepStack features need visual_mask and deepstack pointers");
    return check_seqs(h, cu, n_seqs, S);
}

// Online FP8: the e4m3 weight arena (four projections per layer + per-row scales) and
// the e4m3 activation workspace with per-token scales.
h3enc_status create_fp8(h3enc *h) {
    const h3enc_config &c = h->cfg;
    const size_t H = c.hidden, QO = h->qkv_out, AO = (size_t)c.n_heads * c.head_dim, I = c.intermediate;
    const size_t b_qkv = align256(QO * H), b_o = align256(H * AO), b_gu = align256(2 * I * H),
                 b_down = align256(H * I), s_qkv = align256(QO * 4), s_o = align256(H * 4),
                 s_gu = align256(2 * I * 4), s_down = align256(H * 4);
    const size_t per = b_qkv + b_o + b_gu + b_down + s_qkv + s_o + s_gu + s_down;
    cudaError_t e = cudaMalloc(&h->arena8, per * (size_t)c.num_layers);
    if (e != cudaSuccess)
        return fail(h, H3ENC_ERR_OOM, "FP8 weight arena of %zu bytes: %s", per * (size_t)c.num_layers,
                    cudaGetErrorString(e));
    h->layers8.resize(c.num_layers);
    char *p = h->arena8;
    for (auto &w : h->layers8) {
        w.qkv = reinterpret_cast<uint8_t *>(p); p += b_qkv;
        w.o = reinterpret_cast<uint8_t *>(p); p += b_o;
        w.gu = reinterpret_cast<uint8_t *>(p); p += b_gu;
        w.down = reinterpret_cast<uint8_t *>(p); p += b_down;
        w.s_qkv = reinterpret_cast<float *>(p); p += s_qkv;
        w.s_o = reinterpret_cast<float *>(p); p += s_o;
        w.s_gu = reinterpret_cast<float *>(p); p += s_gu;
        w.s_down = reinterpret_cast<float *>(p); p += s_down;
    }
    const size_t T = c.max_tokens;
    const size_t b_y = align256(T * H), b_a = align256(T * AO), b_act = align256(T * I), b_s = align256(T * 4);
    const size_t wsz = b_y + b_a + b_act + 5 * b_s;
    e = cudaMalloc(&h->ws8, wsz);
    if (e != cudaSuccess) return fail(h, H3ENC_ERR_OOM, "FP8 workspace of %zu bytes: %s", wsz, cudaGetErrorString(e));
    p = h->ws8;
    h->y8 = reinterpret_cast<uint8_t *>(p); p += b_y;
    h->attn8 = reinterpret_cast<uint8_t *>(p); p += b_a;
    h->act8 = reinterpret_cast<uint8_t *>(p); p += b_act;
    h->sy = reinterpret_cast<float *>(p); p += b_s;
    h->sattn = reinterpret_cast<float *>(p); p += b_s;
    h->sact = reinterpret_cast<float *>(p); p += b_s;
    h->amax_attn = reinterpret_cast<float *>(p); p += b_s;
    h->amax_act = reinterpret_cast<float *>(p);
    e = cudaMemset(h->ws8, 0, wsz);
    if (e != cudaSuccess) return fail(h, H3ENC_ERR_CUDA, "FP8 workspace clear: %s", cudaGetErrorString(e));
    const uint32_t ba = (uint32_t)h3::gemm_box_rows_a();
    if (!h3::make_tmap_rows_e4m3(&h->tm_y8, h->y8, T, H, ba) ||
        !h3::make_tmap_rows_e4m3(&h->tm_attn8, h->attn8, T, AO, ba) ||
        !h3::make_tmap_rows_e4m3(&h->tm_act8, h->act8, T, I, ba))
        return fail(h, H3ENC_ERR_CUDA, "cuTensorMapEncodeTiled refused an FP8 workspace operand");
    return H3ENC_OK;
}

// Quantise the loaded bf16 projections of every layer (one scale per output row).
h3enc_status finalize_fp8(h3enc *h) {
    const h3enc_config &c = h->cfg;
    const int H = c.hidden, QO = h->qkv_out, AO = c.n_heads * c.head_dim, I = c.intermediate;
    cudaError_t e = cudaDeviceSynchronize();   // weight uploads issued on other streams have landed
    if (e != cudaSuccess) return cuda_fail(h, e, "FP8 weight quantisation (sync)");
    cudaStream_t st;
    e = cudaStreamCreateWithFlags(&st, cudaStreamNonBlocking);
    if (e != cudaSuccess) return cuda_fail(h, e, "FP8 weight quantisation (stream)");
    const uint32_t bw = (uint32_t)h3::gemm_box_rows_w();
    for (int l = 0; l < c.num_layers && e == cudaSuccess; ++l) {
        LayerW &w = h->layers[l];
        h3enc::Layer8 &q = h->layers8[l];
        e = h3::launch_quant_rows(w.qkv, H, QO, H, q.qkv, H, q.s_qkv, st);
        if (e == cudaSuccess) e = h3::launch_quant_rows(w.o, AO, H, AO, q.o, AO, q.s_o, st);
        if (e == cudaSuccess) e = h3::launch_quant_rows(w.gu, H, 2 * I, H, q.gu, H, q.s_gu, st);
        if (e == cudaSuccess) e = h3::launch_quant_rows(w.down, I, H, I, q.down, I, q.s_down, st);
        if (e == cudaSuccess &&
            (!h3::make_tmap_rows_e4m3(&q.tm_qkv, q.qkv, QO, H, bw) || !h3::make_tmap_rows_e4m3(&q.tm_o, q.o, H, AO, bw) ||
             !h3::make_tmap_rows_e4m3(&q.tm_gu, q.gu, 2 * (size_t)I, H, bw) ||
             !h3::make_tmap_rows_e4m3(&q.tm_down, q.down, H, I, bw))) {
            cudaStreamDestroy(st);
            return fail(h, H3ENC_ERR_CUDA, "cuTensorMapEncodeTiled refused an FP8 weight operand");
        }
    }
    const cudaError_t e2 = cudaStreamSynchronize(st);
    cudaStreamDestroy(st);
    if (e != cudaSuccess) return cuda_fail(h, e, "FP8 weight quantisation");
    if (e2 != cudaSuccess) return cuda_fail(h, e2, "FP8 weight quantisation");
    return H3ENC_OK;
}


void drop_graphs(h3enc *h) {
    for (auto &g : h->graphs)
        if (g.exec) cudaGraphExecDestroy(g.exec);
    h->graphs.clear();
}

h3enc_status encode_core(h3enc *h, const int32_t *ids, const bf16 *embeds, int lb, int le, const int32_t *pos,
                         const uint8_t *mask, const bf16 *ds, int nds, int n_vis, const int32_t *cu, int n_seqs,
                         int S, bf16 *out, cudaStream_t st, const bf16 *visual_embeds = nullptr) {
    if (S == 0) return H3ENC_OK;
    NvtxRange encode_range(h->cfg.linear_fp8 ? "h3enc encode (fp8)" : "h3enc encode");
    const h3enc_config &c = h->cfg;
    const int H = c.hidden, d = c.head_dim, nq = c.n_heads, nkv = c.n_kv_heads, I = c.intermediate;
    cudaError_t e;
    if (ids) {
        e = run(h, H3ENC_K_PREP, st, [&] {
            return h3::launch_embed(ids, h->embed, c.vocab, H, out, S, h->status, st);
        });
        if (e != cudaSuccess) return cuda_fail(h, e, "embedding gather");
    } else if (embeds != out) {
        e = cudaMemcpyAsync(out, embeds, (size_t)S * H * 2, cudaMemcpyDeviceToDevice, st);
        if (e != cudaSuccess) return cuda_fail(h, e, "input copy");
    }
    // row-interleaved: the QKV epilogue's warps read them as whole lines
    e = run(h, H3ENC_K_PREP, st,
            [&] { return h3::launch_rope_table(pos, S, h->rope, h->cos_t, h->sin_t, st, h3::cs_stride(S)); });
    if (e != cudaSuccess) return cuda_fail(h, e, "rope table");
    const bool use_ds = nds > 0 && n_vis > 0;
    const bool use_ve = visual_embeds != nullptr && n_vis > 0;
    if (use_ds || use_ve) {
        e = run(h, H3ENC_K_PREP, st,
                [&] { return h3::launch_vis_rank(mask, S, n_vis, h->vis_rank, h->status, st); });
        if (e != cudaSuccess) return cuda_fail(h, e, "visual ranks");
    }
    if (use_ve) {
        // vision-merger rows replace the placeholder embeddings (masked_scatter in sequence order)
        e = run(h, H3ENC_K_PREP, st, [&] {
            return h3::launch_merge_visual_rows(h->vis_rank, visual_embeds, n_vis, H, out, S, st);
        });
        if (e != cudaSuccess) return cuda_fail(h, e, "visual embedding merge");
    }
    const bool f8 = c.linear_fp8 != 0;
    const bool fold = norm_folded(c);
    const int AO = nq * d;
    // folded RMSNorm: the projections read the hidden state itself and scale their rows by the
    // 1/rms its producer's statistics give (here the layer input's, then the o/down epilogues')
    CUtensorMap tm_h;
    if (fold && le > lb) {
        if (!h3::make_tmap_rows(&tm_h, out, S, H, h3::gemm_box_rows_a()))
            return fail(h, H3ENC_ERR_INVALID_ARG, "out must be 16-byte aligned");
        e = run(h, H3ENC_K_RMSNORM, st, [&] { return h3::launch_row_sumsq(out, S, H, h->row_ss, st); });
        if (e != cudaSuccess) return cuda_fail(h, e, "row statistics");
    }
    if (f8 && le > lb) {
        // the quantising passes clear the row maxima after use; start every encode from zeros
        e = cudaMemsetAsync(h->amax_attn, 0, 2 * align256((size_t)c.max_tokens * 4), st);
        if (e != cudaSuccess) return cuda_fail(h, e, "FP8 row maxima clear");
    }
    struct LayerMark {   // the layer being issued, for per-layer profiling; cleared on every exit
        h3enc *h;
        ~LayerMark() { h->cur_layer = -1; }
    } mark{h};
    for (int l = lb; l < le; ++l) {
        h->cur_layer = l;
        char layer_name[32];
        snprintf(layer_name, sizeof layer_name, "layer %d", l);
        NvtxRange layer_range(layer_name);
        LayerW &w = h->layers[l];
        h3enc::Layer8 *w8 = f8 ? &h->layers8[l] : nullptr;
        // input_layernorm (FP8: its bf16 output quantised per token in the same kernel; folded:
        // inside the QKV projection)
        if (!fold) {
            e = run(h, H3ENC_K_RMSNORM, st, [&] {
                return f8 ? h3::launch_rmsnorm_q8(out, w.in_norm, h->y8, h->sy, S, H, c.rms_eps, st)
                          : h3::launch_rmsnorm(out, w.in_norm, h->y, S, H, c.rms_eps, st);
            });
            if (e != cudaSuccess) return cuda_fail(h, e, "input_layernorm");
        }
        h3::GemmPlan p{};
        p.num_sms = h->num_sms;
        p.status = h->status;
        p.part = h->gemm_part;
        p.flags = h->gemm_flags;
        p.M = S;
        p.fp8 = f8;
        p.w_static = true;   // weights change only at load/finalize, never inside an encode
        // QKV projection with q_norm/k_norm and M-RoPE fused into the epilogue
        p.tmA = f8 ? &h->tm_y8 : fold ? &tm_h : &h->tm_y;
        p.ss_in = fold ? h->row_ss : nullptr;
        p.norm_eps = c.rms_eps;
        p.tmW = f8 ? &w8->tm_qkv : &w.tm_qkv;
        p.sa = f8 ? h->sy : nullptr;
        p.sw = f8 ? w8->s_qkv : nullptr;
        p.N = h->qkv_out; p.K = H; p.epi = h3::EPI_QKROPE;
        p.C = h->qkv; p.ldc = h->qkv_out;
        p.wq = w.q_norm; p.wk = w.k_norm; p.cos_t = h->cos_t; p.sin_t = h->sin_t; p.cs_rows = h3::cs_stride(S);
        p.head_dim = d; p.nq = nq; p.nkv = nkv; p.eps = c.rms_eps;
        e = run(h, H3ENC_K_GEMM_QKV, st, [&] { return h3::launch_gemm(p, st); });
        if (e != cudaSuccess) return cuda_fail(h, e, "qkv gemm");
        e = run(h, H3ENC_K_ATTN, st,
                [&] {
                    return h3::launch_attention(h->qkv, h->attn, S, nq, nkv, d, cu, n_seqs, h->status, st,
                                                f8 ? h->amax_attn : nullptr);
                });
        if (e != cudaSuccess) return cuda_fail(h, e, "attention");
        if (f8) {
            e = run(h, H3ENC_K_QUANT, st, [&] {
                return h3::launch_quant_rows_amax(h->attn, AO, S, AO, h->attn8, AO, h->sattn, h->amax_attn, st);
            });
            if (e != cudaSuccess) return cuda_fail(h, e, "attention output quantisation");
        }
        p.wq = p.wk = nullptr; p.cos_t = p.sin_t = nullptr; p.cs_rows = 0;
        p.tmA = f8 ? &h->tm_attn8 : &h->tm_attn;
        p.tmW = f8 ? &w8->tm_o : &w.tm_o;
        p.sa = f8 ? h->sattn : nullptr;
        p.sw = f8 ? w8->s_o : nullptr;
        p.N = H; p.K = AO; p.epi = h3::EPI_RESIDUAL;
        p.C = out; p.ldc = H; p.R = out;
        p.ss_in = nullptr;
        p.ss_out = fold ? h->row_ss : nullptr;   // statistics for the post-attention norm
        e = run(h, H3ENC_K_GEMM_O, st, [&] { return h3::launch_gemm(p, st); });
        if (e != cudaSuccess) return cuda_fail(h, e, "o_proj gemm");
        p.ss_out = nullptr;
        if (!fold) {
            e = run(h, H3ENC_K_RMSNORM, st, [&] {
                return f8 ? h3::launch_rmsnorm_q8(out, w.post_norm, h->y8, h->sy, S, H, c.rms_eps, st)
                          : h3::launch_rmsnorm(out, w.post_norm, h->y, S, H, c.rms_eps, st);
            });
            if (e != cudaSuccess) return cuda_fail(h, e, "post_attention_layernorm");
        }
        p.tmA = f8 ? &h->tm_y8 : fold ? &tm_h : &h->tm_y;
        p.ss_in = fold ? h->row_ss : nullptr;
        p.tmW = f8 ? &w8->tm_gu : &w.tm_gu;
        p.sa = f8 ? h->sy : nullptr;
        p.sw = f8 ? w8->s_gu : nullptr;
        p.N = 2 * I; p.K = H; p.epi = h3::EPI_SWIGLU;
        p.C = h->act; p.ldc = I; p.R = nullptr;
        p.row_amax = f8 ? h->amax_act : nullptr;
        e = run(h, H3ENC_K_GEMM_GATE_UP, st, [&] { return h3::launch_gemm(p, st); });
        if (e != cudaSuccess) return cuda_fail(h, e, "gate/up gemm");
        if (f8) {
            e = run(h, H3ENC_K_QUANT, st,
                    [&] { return h3::launch_quant_rows_amax(h->act, I, S, I, h->act8, I, h->sact, h->amax_act, st); });
            if (e != cudaSuccess) return cuda_fail(h, e, "SwiGLU output quantisation");
        }
        p.tmA = f8 ? &h->tm_act8 : &h->tm_act;
        p.tmW = f8 ? &w8->tm_down : &w.tm_down;
        p.sa = f8 ? h->sact : nullptr;
        p.sw = f8 ? w8->s_down : nullptr;
        p.N = H; p.K = I; p.C = out; p.ldc = H; p.R = out;
        p.ss_in = nullptr;
        p.ss_out = fold && l + 1 < le ? h->row_ss : nullptr;   // statistics for the next input norm
        if (use_ds && l < nds) {
            if (h->ds_pending) {   // the host entry's DeepStack copy, issued on its own stream
                // (inside a capture the wait becomes an event-wait node on the copy's event)
                cudaStreamCaptureStatus cs = cudaStreamCaptureStatusNone;
                e = cudaStreamIsCapturing(st, &cs);
                if (e == cudaSuccess)
                    e = cudaStreamWaitEvent(st, h->ds_ready,
                                            cs == cudaStreamCaptureStatusActive ? cudaEventWaitExternal : 0);
                if (e != cudaSuccess) return cuda_fail(h, e, "DeepStack copy wait");
                h->ds_pending = false;
            }
            p.epi = h3::EPI_RESIDUAL_DS;
            p.DS = ds + (size_t)l * n_vis * H;
            p.vis_rank = h->vis_rank;
            p.n_vis = n_vis;
        } else {
            p.epi = h3::EPI_RESIDUAL;
        }
        e = run(h, H3ENC_K_GEMM_DOWN, st, [&] { return h3::launch_gemm(p, st); });
        if (e != cudaSuccess) return cuda_fail(h, e, "down gemm");
        if (l < (int)h->capture.size() && h->capture[l]) {
            e = cudaMemcpyAsync(h->capture[l], out, (size_t)S * H * 2, cudaMemcpyDeviceToDevice, st);
            if (e != cudaSuccess) return cuda_fail(h, e, "layer capture");
        }
    }
    return H3ENC_OK;
}

}  // namespace

extern "C" {

h3enc_status h3enc_create(const h3enc_config *cfg, h3enc **out) {
    if (!out) return fail(nullptr, H3ENC_ERR_INVALID_ARG, "out is NULL");
    *out = nullptr;
    h3enc_status s = validate_config(cfg);
    if (s != H3ENC_OK) return s;
    h3enc *h = new h3enc();
    h->cfg = *cfg;
    const h3enc_config &c = h->cfg;
    cudaError_t e = cudaGetDevice(&h->device);
    if (e != cudaSuccess) {
        delete h;
        return fail(nullptr, H3ENC_ERR_CUDA, "no CUDA device: %s", cudaGetErrorString(e));
    }
    h->num_sms = h3::device_num_sms();
    h->qkv_out = (c.n_heads + 2 * c.n_kv_heads) * c.head_dim;
    h3::make_rope_params(&h->rope, c.head_dim, c.rope_theta, c.mrope_section);
    const Sizes ws = weight_sizes(c);
    const size_t arena = ws.embed + ws.layer * (size_t)c.num_layers;
    e = cudaMalloc(&h->arena, arena);
    if (e != cudaSuccess) {
        delete h;
        return fail(nullptr, H3ENC_ERR_OOM, "weight arena of %zu bytes: %s", arena, cudaGetErrorString(e));
    }
    char *p = h->arena;
    h->embed = c.vocab ? reinterpret_cast<bf16 *>(p) : nullptr;
    p += ws.embed;
    h->layers.resize(c.num_layers);
    for (auto &w : h->layers) {
        w.qkv = reinterpret_cast<bf16 *>(p); p += ws.qkv;
        w.o = reinterpret_cast<bf16 *>(p); p += ws.o;
        w.gu = reinterpret_cast<bf16 *>(p); p += ws.gu;
        w.down = reinterpret_cast<bf16 *>(p); p += ws.down;
        w.in_norm = reinterpret_cast<bf16 *>(p); p += ws.norm_h;
        w.post_norm = reinterpret_cast<bf16 *>(p); p += ws.norm_h;
        w.q_norm = reinterpret_cast<bf16 *>(p); p += ws.norm_d;
        w.k_norm = reinterpret_cast<bf16 *>(p); p += ws.norm_d;
    }
    const size_t T = c.max_tokens, H = c.hidden;
    const size_t b_y = align256(T * H * 2), b_qkv = align256(T * h->qkv_out * 2),
                 b_attn = align256(T * c.n_heads * c.head_dim * 2), b_act = align256(T * c.intermediate * 2),
                 b_cs = align256((size_t)h3::cs_stride((int)T) * (c.head_dim / 2) * 4), b_rank = align256(T * 4), b_stat = 256,
                 b_ids = align256(T * 4), b_pos = align256(3 * T * 4), b_mask = align256(T),
                 b_ds = align256((size_t)c.num_deepstack * T * H * 2), b_out = b_y,
                 b_gemm = align256(h3::gemm_workspace_bytes(h->num_sms)), b_ss = align256(T * (H / 128) * 4);
    const size_t wsz = b_y + b_qkv + b_attn + b_act + 2 * b_cs + b_rank + b_stat + b_ids + b_pos + b_mask + b_ds +
                       b_out + b_gemm + b_ss;
    e = cudaMalloc(&h->ws, wsz);
    if (e != cudaSuccess) {
        cudaFree(h->arena);
        delete h;
        return fail(nullptr, H3ENC_ERR_OOM, "workspace of %zu bytes: %s", wsz, cudaGetErrorString(e));
    }
    p = h->ws;
    h->y = reinterpret_cast<bf16 *>(p); p += b_y;
    h->qkv = reinterpret_cast<bf16 *>(p); p += b_qkv;
    h->attn = reinterpret_cast<bf16 *>(p); p += b_attn;
    h->act = reinterpret_cast<bf16 *>(p); p += b_act;
    h->cos_t = reinterpret_cast<float *>(p); p += b_cs;
    h->sin_t = reinterpret_cast<float *>(p); p += b_cs;
    h->vis_rank = reinterpret_cast<int32_t *>(p); p += b_rank;
    h->status = reinterpret_cast<int32_t *>(p); p += b_stat;
    h->st_ids = reinterpret_cast<int32_t *>(p); p += b_ids;
    h->st_pos = reinterpret_cast<int32_t *>(p); p += b_pos;
    h->st_mask = reinterpret_cast<uint8_t *>(p); p += b_mask;
    h->st_ds = reinterpret_cast<bf16 *>(p); p += b_ds;
    h->st_out = reinterpret_cast<bf16 *>(p); p += b_out;
    h->gemm_part = reinterpret_cast<float *>(p);
    h->gemm_flags = reinterpret_cast<uint32_t *>(p + h3::gemm_flags_offset(h->num_sms));
    p += b_gemm;
    h->row_ss = reinterpret_cast<float *>(p); p += b_ss;
    e = cudaMemset(h->ws, 0, wsz);
    if (e != cudaSuccess) {
        h3enc_destroy(h);
        return fail(nullptr, H3ENC_ERR_CUDA, "workspace clear: %s", cudaGetErrorString(e));
    }
    if (c.linear_fp8) {
        h3enc_status s8 = create_fp8(h);
        if (s8 != H3ENC_OK) {
            const std::string msg = h->err;
            h3enc_destroy(h);
            return fail(nullptr, s8, "%s", msg.c_str());
        }
    }
    const uint32_t ba = (uint32_t)h3::gemm_box_rows_a();
    if (!h3::make_tmap_rows(&h->tm_y, h->y, T, H, ba) ||
        !h3::make_tmap_rows(&h->tm_attn, h->attn, T, (size_t)c.n_heads * c.head_dim, ba) ||
        !h3::make_tmap_rows(&h->tm_act, h->act, T, c.intermediate, ba)) {
        h3enc_destroy(h);
        return fail(nullptr, H3ENC_ERR_CUDA, "cuTensorMapEncodeTiled refused a workspace operand");
    }
    *out = h;
    return H3ENC_OK;
}

h3enc_status h3enc_load_weights(h3enc *h, const char *name, const void *data, int32_t dtype,
                                const int64_t *shape, int32_t ndim, int32_t data_on_device) {
    if (!h || !name || !data || !shape || ndim < 1) return fail(h, H3ENC_ERR_INVALID_ARG, "NULL argument");
    drop_graphs(h);   // a graph replays the weights as they were when it was captured
    const h3enc_config &c = h->cfg;
    if (strcmp(name, "lm_head.weight") == 0 || strcmp(name, "model.language_model.norm.weight") == 0 ||
        strncmp(name, "model.visual.", 13) == 0)
        return H3ENC_WARN_IGNORED;
    int layer = -1, which = -1;
    const bool is_embed = strcmp(name, "model.language_model.embed_tokens.weight") == 0;
    if (!is_embed) {
        if (!parse_layer_name(name, &layer, &which)) {
            fail(h, H3ENC_WARN_IGNORED, "weight %s has no target parameter", name);
            return H3ENC_WARN_IGNORED;
        }
        if (layer >= c.num_layers) return H3ENC_WARN_IGNORED;
        if (which < 0) {
            fail(h, H3ENC_WARN_IGNORED, "weight %s has no target parameter", name);
            return H3ENC_WARN_IGNORED;
        }
    } else if (c.vocab == 0) {
        return H3ENC_WARN_IGNORED;
    }
    if (dtype == H3ENC_DTYPE_FP8_E4M3)
        return fail(h, H3ENC_ERR_UNSUPPORTED, "%s: serialized FP8 weights are not supported (online FP8 only)", name);
    if (dtype != H3ENC_DTYPE_BF16) return fail(h, H3ENC_ERR_UNSUPPORTED, "%s: dtype %d is not bf16", name, dtype);
    const int64_t H = c.hidden, d = c.head_dim, nq = c.n_heads, nkv = c.n_kv_heads, I = c.intermediate;
    int64_t want[2] = {0, 0};
    int want_nd = 2;
    if (is_embed) { want[0] = c.vocab; want[1] = H; }
    else switch (which) {
        case T_IN: case T_POST: want_nd = 1; want[0] = H; break;
        case T_QN: case T_KN: want_nd = 1; want[0] = d; break;
        case T_Q: want[0] = nq * d; want[1] = H; break;
        case T_K: case T_V: want[0] = nkv * d; want[1] = H; break;
        case T_O: want[0] = H; want[1] = nq * d; break;
        case T_GATE: case T_UP: want[0] = I; want[1] = H; break;
        case T_DOWN: want[0] = H; want[1] = I; break;
    }
    if (ndim != want_nd || shape[0] != want[0] || (want_nd == 2 && shape[1] != want[1]))
        return fail(h, H3ENC_ERR_SHAPE, "%s: shape mismatch (expected [%lld%s%lld])", name, (long long)want[0],
                    want_nd == 2 ? ", " : "", want_nd == 2 ? (long long)want[1] : 0LL);
    const cudaMemcpyKind kind = data_on_device ? cudaMemcpyDeviceToDevice : cudaMemcpyHostToDevice;
    const bf16 *src = static_cast<const bf16 *>(data);
    cudaError_t e = cudaSuccess;
    const size_t n = (size_t)want[0] * (want_nd == 2 ? (size_t)want[1] : 1);
    if (is_embed) {
        e = cudaMemcpy(h->embed, src, n * 2, kind);
        if (e == cudaSuccess) h->embed_loaded = true;
    } else {
        LayerW &w = h->layers[layer];
        bf16 *dst = nullptr;
        switch (which) {
            case T_IN: dst = w.in_norm; break;
            case T_POST: dst = w.post_norm; break;
            case T_QN: dst = w.q_norm; break;
            case T_KN: dst = w.k_norm; break;
            case T_Q: dst = w.qkv; break;
            case T_K: dst = w.qkv + nq * d * H; break;
            case T_V: dst = w.qkv + (nq + nkv) * d * H; break;
            case T_O: dst = w.o; break;
            case T_DOWN: dst = w.down; break;
            default: break;
        }
        if (which == T_GATE || which == T_UP) {
            e = h3::pack_gate_up_rows(src, w.gu, (int)I, (int)H, which == T_UP, kind, 0);
            if (e == cudaSuccess) e = cudaStreamSynchronize(0);
        } else {
            e = cudaMemcpy(dst, src, n * 2, kind);
        }
        if (e == cudaSuccess) {
            w.loaded |= 1u << which;
            w.folded &= ~(1u << which);   // the arena holds the checkpoint's rows again
            if (which == T_IN && (w.folded & kQKVBits)) w.in_stale = true;
            if (which == T_POST && (w.folded & kGUBits)) w.post_stale = true;
        }
    }
    if (e != cudaSuccess) return cuda_fail(h, e, name);
    h->finalized = false;
    return H3ENC_OK;
}

h3enc_status h3enc_finalize_weights(h3enc *h) {
    if (!h) return fail(h, H3ENC_ERR_INVALID_ARG, "NULL handle");
    drop_graphs(h);
    const h3enc_config &c = h->cfg;
    std::string missing, shards;
    int n_missing = 0;
    if (c.vocab && !h->embed_loaded) {
        missing += "model.language_model.embed_tokens.weight";
        ++n_missing;
    }
    for (int l = 0; l < c.num_layers; ++l) {
        const uint32_t m = h->layers[l].loaded;
        for (int t = 0; t < T_COUNT; ++t)
            if (!(m & (1u << t))) {
                if (n_missing < 40) {
                    if (!missing.empty()) missing += ", ";
                    missing += "model.language_model.layers." + std::to_string(l) + "." + kSuffix[t];
                }
                ++n_missing;
            }
        const bool q = m & (1u << T_Q), k = m & (1u << T_K), v = m & (1u << T_V);
        if ((q || k || v) && !(q && k && v))
            shards += " layers." + std::to_string(l) + ".qkv_proj: [" + (q ? "" : "q ") + (k ? "" : "k ") +
                      (v ? "" : "v") + "]";
        const bool g = m & (1u << T_GATE), u = m & (1u << T_UP);
        if ((g || u) && !(g && u))
            shards += " layers." + std::to_string(l) + ".gate_up_proj: [" + (g ? "" : "gate") + (u ? "" : "up") + "]";
    }
    if (n_missing)
        return fail(h, H3ENC_ERR_MISSING_WEIGHTS, "weights not loaded: %d params: %s%s; fused shards missing:%s",
                    n_missing, missing.c_str(), n_missing > 40 ? ", ..." : "", shards.empty() ? " none" : shards.c_str());
    if (norm_folded(c)) {
        h3enc_status sf = fold_norms(h);
        if (sf != H3ENC_OK) return sf;
    }
    const uint32_t bw = (uint32_t)h3::gemm_box_rows_w();
    const size_t H = c.hidden, d = c.head_dim;
    for (auto &w : h->layers) {
        if (!h3::make_tmap_rows(&w.tm_qkv, w.qkv, h->qkv_out, H, bw) ||
            !h3::make_tmap_rows(&w.tm_o, w.o, H, c.n_heads * d, bw) ||
            !h3::make_tmap_rows(&w.tm_gu, w.gu, 2 * (size_t)c.intermediate, H, bw) ||
            !h3::make_tmap_rows(&w.tm_down, w.down, H, c.intermediate, bw))
            return fail(h, H3ENC_ERR_CUDA, "cuTensorMapEncodeTiled refused a weight operand");
    }
    if (c.linear_fp8) {
        h3enc_status s8 = finalize_fp8(h);
        if (s8 != H3ENC_OK) return s8;
    }
    h->finalized = true;
    return H3ENC_OK;
}

h3enc_status h3enc_encode(h3enc *h, const int32_t *input_ids, const int32_t *positions, const uint8_t *visual_mask,
                          const void *deepstack, int32_t num_deepstack, int32_t n_vis, const int32_t *cu_seqlens,
                          int32_t n_seqs, int32_t seq_len, void *out, void *stream) {
    if (!h) return fail(h, H3ENC_ERR_INVALID_ARG, "NULL handle");
    h3enc_status s = check_encode_args(h, positions, visual_mask, deepstack, num_deepstack, n_vis, cu_seqlens,
                                       n_seqs, seq_len, out);
    if (s != H3ENC_OK) return s;
    if (h->cfg.vocab == 0) return fail(h, H3ENC_ERR_UNSUPPORTED, "model has no embedding table (vocab 0)");
    if (seq_len > 0 && !input_ids) return fail(h, H3ENC_ERR_INVALID_ARG, "input_ids is NULL");
    return encode_core(h, input_ids, nullptr, 0, h->cfg.num_layers, positions, visual_mask,
                       static_cast<const bf16 *>(deepstack), num_deepstack, n_vis, cu_seqlens, n_seqs, seq_len,
                       static_cast<bf16 *>(out), static_cast<cudaStream_t>(stream));
}

h3enc_status h3enc_encode_multimodal(h3enc *h, const int32_t *input_ids, const int32_t *positions,
                                     const uint8_t *visual_mask, const void *visual_embeds, const void *deepstack,
                                     int32_t num_deepstack, int32_t n_vis, const int32_t *cu_seqlens, int32_t n_seqs,
                                     int32_t seq_len, void *out, void *stream) {
    if (!h) return fail(h, H3ENC_ERR_INVALID_ARG, "NULL handle");
    h3enc_status s = check_encode_args(h, positions, visual_mask, deepstack, num_deepstack, n_vis, cu_seqlens,
                                       n_seqs, seq_len, out);
    if (s != H3ENC_OK) return s;
    if (h->cfg.vocab == 0) return fail(h, H3ENC_ERR_UNSUPPORTED, "model has no embedding table (vocab 0)");
    if (seq_len > 0 && !input_ids) return fail(h, H3ENC_ERR_INVALID_ARG, "input_ids is NULL");
    if (n_vis > 0 && visual_embeds && !visual_mask)
        return fail(h, H3ENC_ERR_INVALID_ARG, "visual_embeds need a visual_mask");
    return encode_core(h, input_ids, nullptr, 0, h->cfg.num_layers, positions, visual_mask,
                       static_cast<const bf16 *>(deepstack), num_deepstack, n_vis, cu_seqlens, n_seqs, seq_len,
                       static_cast<bf16 *>(out), static_cast<cudaStream_t>(stream),
                       static_cast<const bf16 *>(visual_embeds));
}

h3enc_status h3enc_encode_embeds(h3enc *h, const void *inputs_embeds, int32_t layer_begin, int32_t layer_end,
                                 const int32_t *positions, const uint8_t *visual_mask, const void *deepstack,
                                 int32_t num_deepstack, int32_t n_vis, const int32_t *cu_seqlens, int32_t n_seqs,
                                 int32_t seq_len, void *out, void *stream) {
    if (!h) return fail(h, H3ENC_ERR_INVALID_ARG, "NULL handle");
    h3enc_status s = check_encode_args(h, positions, visual_mask, deepstack, num_deepstack, n_vis, cu_seqlens,
                                       n_seqs, seq_len, out);
    if (s != H3ENC_OK) return s;
    if (layer_begin < 0 || layer_end > h->cfg.num_layers || layer_begin > layer_end)
        return fail(h, H3ENC_ERR_INVALID_ARG, "layer range [%d, %d) outside [0, %d]", layer_begin, layer_end,
                    h->cfg.num_layers);
    if (seq_len > 0 && !inputs_embeds) return fail(h, H3ENC_ERR_INVALID_ARG, "inputs_embeds is NULL");
    return encode_core(h, nullptr, static_cast<const bf16 *>(inputs_embeds), layer_begin, layer_end, positions,
                       visual_mask, static_cast<const bf16 *>(deepstack), num_deepstack, n_vis, cu_seqlens, n_seqs,
                       seq_len, static_cast<bf16 *>(out), static_cast<cudaStream_t>(stream));
}

h3enc_status h3enc_encode_host(h3enc *h, const int32_t *input_ids, const int32_t *positions,
                               const uint8_t *visual_mask, const void *deepstack, int32_t num_deepstack,
                               int32_t n_vis, const int32_t *cu_seqlens, int32_t n_seqs, int32_t seq_len, void *out,
                               void *stream) {
    if (!h) return fail(h, H3ENC_ERR_INVALID_ARG, "NULL handle");
    h3enc_status s = check_encode_args(h, positions, visual_mask, deepstack, num_deepstack, n_vis, cu_seqlens,
                                       n_seqs, seq_len, out);
    if (s != H3ENC_OK) return s;
    if (h->cfg.vocab == 0) return fail(h, H3ENC_ERR_UNSUPPORTED, "model has no embedding table (vocab 0)");
    if (seq_len == 0) return H3ENC_OK;
    if (!input_ids) return fail(h, H3ENC_ERR_INVALID_ARG, "input_ids is NULL");
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    const size_t S = seq_len, H = h->cfg.hidden;
    const bool use_ds = num_deepstack > 0 && n_vis > 0;
    cudaError_t e = cudaSuccess;
    if (use_ds && !h->copy_st) {
        e = cudaStreamCreateWithFlags(&h->copy_st, cudaStreamNonBlocking);
        if (e == cudaSuccess) e = cudaEventCreateWithFlags(&h->ds_fork, cudaEventDisableTiming);
        if (e == cudaSuccess) e = cudaEventCreateWithFlags(&h->ds_ready, cudaEventDisableTiming);
        if (e != cudaSuccess) return cuda_fail(h, e, "copy stream");
    }
    // the DeepStack features (the bulk of the inputs) go first, on the copy stream, once the
    // caller's earlier work on `stream` is done with the staging buffer
    bool ds_waited = !use_ds;   // whether `stream` has been made to wait for that copy
    if (use_ds) {
        e = cudaEventRecord(h->ds_fork, st);
        if (e == cudaSuccess) e = cudaStreamWaitEvent(h->copy_st, h->ds_fork, 0);
        if (e == cudaSuccess)
            e = cudaMemcpyAsync(h->st_ds, deepstack, (size_t)num_deepstack * n_vis * H * 2, cudaMemcpyHostToDevice,
                                h->copy_st);
        if (e == cudaSuccess) e = cudaEventRecord(h->ds_ready, h->copy_st);
        if (e != cudaSuccess) return cuda_fail(h, e, "host-to-device copy");
    }
    // on every way out the host buffer is released only after the copy has read it
    struct DsGuard {
        h3enc *h;
        const bool &waited;
        ~DsGuard() {
            h->ds_pending = false;
            if (!waited) cudaStreamSynchronize(h->copy_st);
        }
    } ds_guard{h, ds_waited};
    e = cudaMemcpyAsync(h->st_ids, input_ids, S * 4, cudaMemcpyHostToDevice, st);
    if (e == cudaSuccess) e = cudaMemcpyAsync(h->st_pos, positions, 3 * S * 4, cudaMemcpyHostToDevice, st);
    if (e == cudaSuccess && visual_mask) e = cudaMemcpyAsync(h->st_mask, visual_mask, S, cudaMemcpyHostToDevice, st);
    if (e != cudaSuccess) return cuda_fail(h, e, "host-to-device copy");
    bool consumed = false;   // the last encode_core made `stream` wait for the DeepStack copy
    auto encode = [&] {
        h->ds_pending = use_ds;
        const h3enc_status r = encode_core(h, h->st_ids, nullptr, 0, h->cfg.num_layers, h->st_pos,
                                           visual_mask ? h->st_mask : nullptr, use_ds ? h->st_ds : nullptr,
                                           num_deepstack, n_vis, cu_seqlens, n_seqs, seq_len, h->st_out, st);
        consumed = use_ds && !h->ds_pending;
        h->ds_pending = false;
        return r;
    };
    // Graphs: the first call of a shape runs eagerly (and so makes every one-time kernel setup);
    // the second captures the encode into a graph, which it and later calls of that shape replay.
    // Eager when profiling or capturing layers (both change what an encode records), on the
    // legacy or per-thread default stream (not capturable), when the caller's stream is itself
    // being captured, or for a shape whose capture failed.
    cudaStreamCaptureStatus cap = cudaStreamCaptureStatusNone;
    const bool graphable = h->use_graphs && !h->prof && h->capture.empty() && st != nullptr &&
                           st != cudaStreamLegacy && st != cudaStreamPerThread &&
                           cudaStreamIsCapturing(st, &cap) == cudaSuccess && cap == cudaStreamCaptureStatusNone;
    h3enc::Graph *g = nullptr;
    if (graphable) {
        const int nseg = cu_seqlens ? n_seqs + 1 : 0;
        for (auto &c : h->graphs)
            if (c.S == seq_len && c.n_seqs == n_seqs && c.n_vis == n_vis && c.nds == num_deepstack &&
                c.mask == (visual_mask != nullptr) && (int)c.cu.size() == nseg &&
                std::equal(c.cu.begin(), c.cu.end(), cu_seqlens))
                g = &c;
        if (!g) {   // a new shape: remember it, run eagerly
            if (h->graphs.size() >= h3enc::kMaxGraphs) {
                auto lru = std::min_element(h->graphs.begin(), h->graphs.end(),
                                            [](const h3enc::Graph &a, const h3enc::Graph &b) { return a.used < b.used; });
                if (lru->exec) cudaGraphExecDestroy(lru->exec);
                h->graphs.erase(lru);
            }
            h3enc::Graph ng;
            ng.S = seq_len;
            ng.n_seqs = n_seqs;
            ng.n_vis = n_vis;
            ng.nds = num_deepstack;
            ng.mask = visual_mask != nullptr;
            if (nseg) ng.cu.assign(cu_seqlens, cu_seqlens + nseg);
            ng.used = ++h->graph_tick;
            h->graphs.push_back(std::move(ng));
        } else {
            g->used = ++h->graph_tick;
            if (!g->exec && !g->failed) {   // the second call of this shape: capture it
                const int64_t before = h->launch_count;
                bool ok = cudaStreamBeginCapture(st, cudaStreamCaptureModeThreadLocal) == cudaSuccess;
                if (ok) {
                    const h3enc_status cs = encode();
                    cudaGraph_t graph = nullptr;
                    ok = cudaStreamEndCapture(st, &graph) == cudaSuccess && cs == H3ENC_OK && graph;
                    cudaGraphExec_t exec = nullptr;
                    if (ok) ok = cudaGraphInstantiate(&exec, graph, 0) == cudaSuccess && exec;
                    if (ok) g->exec = exec;
                    g->waits_ds = consumed;
                    if (graph) cudaGraphDestroy(graph);
                }
                g->launches = h->launch_count - before;
                h->launch_count = before;   // counted when a replay runs them
                if (!ok) {   // this shape stays eager; the eager run below reports any real error
                    (void)cudaGetLastError();
                    g->failed = true;
                    h->err.clear();
                }
            }
            if (!g->exec) g = nullptr;
        }
    }
    if (g) {
        e = cudaGraphLaunch(g->exec, st);   // its wait node takes this call's DeepStack copy
        if (e != cudaSuccess) return cuda_fail(h, e, "graph launch");
        ds_waited = g->waits_ds;
        h->launch_count += g->launches;
    } else {
        s = encode();
        if (s != H3ENC_OK) return s;
        ds_waited = consumed;
    }
    e = cudaMemcpyAsync(out, h->st_out, S * H * 2, cudaMemcpyDeviceToHost, st);
    if (e == cudaSuccess) e = cudaStreamSynchronize(st);
    if (e != cudaSuccess) return cuda_fail(h, e, "device-to-host copy");
    return H3ENC_OK;
}

h3enc_status h3enc_set_layer_capture(h3enc *h, void *const *per_layer, int32_t n) {
    if (!h) return fail(h, H3ENC_ERR_INVALID_ARG, "NULL handle");
    if (n == 0) {
        h->capture.clear();
        return H3ENC_OK;
    }
    if (n != h->cfg.num_layers || !per_layer)
        return fail(h, H3ENC_ERR_INVALID_ARG, "capture needs num_layers=%d pointers", h->cfg.num_layers);
    h->capture.assign(per_layer, per_layer + n);
    return H3ENC_OK;
}

h3enc_status h3enc_get_status(h3enc *h) {
    if (!h) return fail(h, H3ENC_ERR_INVALID_ARG, "NULL handle");
    cudaError_t e = cudaDeviceSynchronize();
    if (e != cudaSuccess) return cuda_fail(h, e, "device synchronise");
    int32_t st = 0;
    e = cudaMemcpy(&st, h->status, 4, cudaMemcpyDeviceToHost);
    if (e == cudaSuccess) e = cudaMemset(h->status, 0, 4);
    if (e != cudaSuccess) return cuda_fail(h, e, "status read");
    if (st & 1) return fail(h, H3ENC_ERR_DEVICE_TIMEOUT, "a bounded device wait ran out");
    if (st & 2) return fail(h, H3ENC_ERR_DEVICE_BOUNDS, "token id outside [0, vocab)");
    if (st & 4) return fail(h, H3ENC_ERR_SHAPE, "visual mask count differs from n_vis");
    return H3ENC_OK;
}

const char *h3enc_last_error(const h3enc *h) { return h ? h->err.c_str() : g_create_error.c_str(); }

void h3enc_destroy(h3enc *h) {
    if (!h) return;
    drop_graphs(h);
    if (h->copy_st) cudaStreamDestroy(h->copy_st);
    if (h->ds_fork) cudaEventDestroy(h->ds_fork);
    if (h->ds_ready) cudaEventDestroy(h->ds_ready);
    for (cudaEvent_t ev : h->ev_pool) cudaEventDestroy(ev);
    if (h->ws8) cudaFree(h->ws8);
    if (h->arena8) cudaFree(h->arena8);
    if (h->ws) cudaFree(h->ws);
    if (h->arena) cudaFree(h->arena);
    delete h;
}

h3enc_status h3enc_set_profiling(h3enc *h, int32_t enable) {
    return h3enc_set_profiling_classes(h, enable ? 0xFFFFFFFFu : 0u);
}

h3enc_status h3enc_set_profiling_classes(h3enc *h, uint32_t mask) {
    if (!h) return fail(h, H3ENC_ERR_INVALID_ARG, "NULL handle");
    h->prof = mask != 0;
    h->prof_mask = mask;
    h->ev_used = 0;
    // reserve event pairs up front so a timed region never creates events
    while (h->prof && h->ev_pool.size() < 16384) {
        cudaEvent_t ev;
        cudaError_t e = cudaEventCreate(&ev);
        if (e != cudaSuccess) return cuda_fail(h, e, "profiling events");
        h->ev_pool.push_back(ev);
        h->ev_class.push_back(0);
    }
    for (int k = 0; k < H3ENC_K_COUNT; ++k) {
        h->ms[k] = 0;
        h->launches[k] = 0;
    }
    return H3ENC_OK;
}

h3enc_status h3enc_set_profiling_layer(h3enc *h, int32_t layer) {
    if (!h || layer < -1 || layer >= h->cfg.num_layers) return fail(h, H3ENC_ERR_INVALID_ARG, "bad layer");
    h->prof_layer = layer;
    return H3ENC_OK;
}

h3enc_status h3enc_get_profile(h3enc *h, double *ms, int64_t *launches, int32_t n) {
    if (!h || n < 0 || n > H3ENC_K_COUNT) return fail(h, H3ENC_ERR_INVALID_ARG, "bad arguments");
    cudaError_t e = cudaDeviceSynchronize();
    if (e != cudaSuccess) return cuda_fail(h, e, "device synchronise");
    for (size_t i = 0; i + 1 < h->ev_used; i += 2) {
        float t = 0.f;
        if (cudaEventElapsedTime(&t, h->ev_pool[i], h->ev_pool[i + 1]) == cudaSuccess) h->ms[h->ev_class[i]] += t;
    }
    h->ev_used = 0;
    for (int k = 0; k < n; ++k) {
        if (ms) ms[k] = h->ms[k];
        if (launches) launches[k] = h->launches[k];
    }
    for (int k = 0; k < H3ENC_K_COUNT; ++k) {
        h->ms[k] = 0;
        h->launches[k] = 0;
    }
    return H3ENC_OK;
}

int64_t h3enc_launch_count(const h3enc *h) { return h ? h->launch_count : 0; }

h3enc_status h3enc_set_graphs(h3enc *h, int32_t enable) {
    if (!h) return fail(h, H3ENC_ERR_INVALID_ARG, "NULL handle");
    if (enable != 0 && enable != 1) return fail(h, H3ENC_ERR_INVALID_ARG, "enable must be 0 or 1");
    h->use_graphs = enable != 0;
    if (!enable) drop_graphs(h);
    return H3ENC_OK;
}

int32_t h3enc_graph_count(const h3enc *h) {
    int32_t n = 0;
    if (h)
        for (const auto &g : h->graphs) n += g.exec != nullptr;
    return n;
}
int32_t h3enc_num_sms(const h3enc *h) { return h ? h->num_sms : 0; }

// ---------------------------------------------------------------- op-level entries

int64_t h3enc_op_gemm_workspace_bytes(void) {
    const int sms = h3::device_num_sms();
    return sms > 0 ? (int64_t)h3::gemm_workspace_bytes(sms) : -1;
}

}  // extern "C"

namespace {

// h3enc_op_gemm and h3enc_op_gemm_rms: the bf16 projection with optional folded-norm row
// statistics in (ss_in) and out (ss_out).
h3enc_status gemm_op(const void *A, const void *W, void *C, int32_t M, int32_t N, int32_t K, int32_t epilogue,
                     const void *R, const void *DS, const int32_t *vis_rank, int32_t n_vis, const float *ss_in,
                     float *ss_out, float norm_eps, void *workspace, int64_t workspace_bytes, int32_t *status,
                     void *stream) {
    if (M < 0 || N <= 0 || K <= 0 || N % 256 || K % 8 || epilogue < 0 || epilogue > 3)
        return fail(nullptr, H3ENC_ERR_INVALID_ARG, "gemm: bad sizes or epilogue");
    if ((ss_in && K % 128) || (ss_out && epilogue == H3ENC_EPI_SWIGLU))
        return fail(nullptr, H3ENC_ERR_INVALID_ARG, "gemm: row statistics need K %% 128 == 0 (in) and a stored "
                                                    "output (out)");
    if (M == 0) return H3ENC_OK;
    if (!A || !W || !C || ((epilogue == H3ENC_EPI_RESIDUAL || epilogue == H3ENC_EPI_RESIDUAL_DS) && !R) ||
        (epilogue == H3ENC_EPI_RESIDUAL_DS && DS && !vis_rank))
        return fail(nullptr, H3ENC_ERR_INVALID_ARG, "gemm: NULL operand");
    CUtensorMap ta, tw;
    if (!h3::make_tmap_rows(&ta, A, M, K, h3::gemm_box_rows_a()) ||
        !h3::make_tmap_rows(&tw, W, N, K, h3::gemm_box_rows_w()))
        return fail(nullptr, H3ENC_ERR_INVALID_ARG, "gemm: operands not 16-byte aligned or driver refused the map");
    h3::GemmPlan p{};
    p.tmA = &ta; p.tmW = &tw; p.M = M; p.N = N; p.K = K; p.epi = epilogue;
    p.C = static_cast<bf16 *>(C);
    p.ldc = epilogue == H3ENC_EPI_SWIGLU ? N / 2 : N;
    p.R = static_cast<const bf16 *>(R);
    p.DS = static_cast<const bf16 *>(DS);
    p.vis_rank = vis_rank;
    p.n_vis = n_vis;
    p.status = status;
    p.num_sms = h3::device_num_sms();
    p.ss_in = ss_in;
    p.ss_out = ss_out;
    p.norm_eps = norm_eps;
    if (workspace) {
        if (workspace_bytes < (int64_t)h3::gemm_workspace_bytes(p.num_sms) ||
            (reinterpret_cast<uintptr_t>(workspace) & 255))
            return fail(nullptr, H3ENC_ERR_INVALID_ARG, "gemm: workspace smaller than h3enc_op_gemm_workspace_bytes() "
                                                        "or not 256-byte aligned");
        p.part = static_cast<float *>(workspace);
        p.flags = reinterpret_cast<uint32_t *>(static_cast<char *>(workspace) +
                                               h3::gemm_flags_offset(p.num_sms));
    }
    cudaError_t e = h3::launch_gemm(p, static_cast<cudaStream_t>(stream));
    return e == cudaSuccess ? H3ENC_OK : cuda_fail(nullptr, e, "gemm launch");
}

}  // namespace

extern "C" {

h3enc_status h3enc_op_gemm(const void *A, const void *W, void *C, int32_t M, int32_t N, int32_t K, int32_t epilogue,
                           const void *R, const void *DS, const int32_t *vis_rank, int32_t n_vis, void *workspace,
                           int64_t workspace_bytes, int32_t *status, void *stream) {
    return gemm_op(A, W, C, M, N, K, epilogue, R, DS, vis_rank, n_vis, nullptr, nullptr, 0.f, workspace,
                   workspace_bytes, status, stream);
}

h3enc_status h3enc_op_gemm_rms(const void *A, const void *W, void *C, int32_t M, int32_t N, int32_t K,
                               int32_t epilogue, const void *R, const float *ss_in, float *ss_out, float eps,
                               void *workspace, int64_t workspace_bytes, int32_t *status, void *stream) {
    if (epilogue == H3ENC_EPI_RESIDUAL_DS)
        return fail(nullptr, H3ENC_ERR_INVALID_ARG, "gemm_rms: epilogue must be STORE, RESIDUAL or SWIGLU");
    return gemm_op(A, W, C, M, N, K, epilogue, R, nullptr, nullptr, 0, ss_in, ss_out, eps, workspace,
                   workspace_bytes, status, stream);
}

h3enc_status h3enc_op_row_sumsq(const void *x, int32_t rows, int32_t cols, float *ss, void *stream) {
    if (!x || !ss || rows < 0 || cols <= 0 || cols % 128 || (reinterpret_cast<uintptr_t>(x) & 15))
        return fail(nullptr, H3ENC_ERR_INVALID_ARG, "row_sumsq: bad args");
    cudaError_t e = h3::launch_row_sumsq(static_cast<const bf16 *>(x), rows, cols, ss,
                                         static_cast<cudaStream_t>(stream));
    return e == cudaSuccess ? H3ENC_OK : cuda_fail(nullptr, e, "row_sumsq launch");
}

h3enc_status h3enc_op_fold_cols(void *W, int32_t rows, int32_t cols, const void *gamma, void *stream) {
    if (!W || !gamma || rows < 0 || cols <= 0 || cols % 8 || (reinterpret_cast<uintptr_t>(W) & 15) ||
        (reinterpret_cast<uintptr_t>(gamma) & 15))
        return fail(nullptr, H3ENC_ERR_INVALID_ARG, "fold_cols: bad args");
    cudaError_t e = h3::launch_fold_cols(static_cast<bf16 *>(W), cols, static_cast<const bf16 *>(gamma), 0, rows, 0,
                                         0, static_cast<cudaStream_t>(stream));
    return e == cudaSuccess ? H3ENC_OK : cuda_fail(nullptr, e, "fold_cols launch");
}

h3enc_status h3enc_op_gemm_trace_next(void *trace, int64_t trace_entries) {
    const int sms = h3::device_num_sms();
    if (!trace || sms <= 0 || trace_entries < (int64_t)sms * 11)
        return fail(nullptr, H3ENC_ERR_INVALID_ARG, "gemm_trace_next: trace needs 11 entries per SM");
    h3::gemm_trace_next(static_cast<unsigned long long *>(trace));
    return H3ENC_OK;
}

h3enc_status h3enc_op_attention_trace_next(void *trace, int64_t trace_entries, int32_t ctas) {
    if (!trace || ctas <= 0 || trace_entries < (int64_t)ctas * h3::attention_trace_fields())
        return fail(nullptr, H3ENC_ERR_INVALID_ARG, "attention_trace_next: trace needs 9 entries per CTA");
    h3::attention_trace_next(static_cast<unsigned long long *>(trace));
    return H3ENC_OK;
}

h3enc_status h3enc_op_pack_gate_up(const void *gate, const void *up, void *W, int32_t I, int32_t K, void *stream) {
    if (!gate || !up || !W || I <= 0 || K <= 0 || I % 128) return fail(nullptr, H3ENC_ERR_INVALID_ARG, "pack: bad args");
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    cudaError_t e = h3::pack_gate_up_rows(static_cast<const bf16 *>(gate), static_cast<bf16 *>(W), I, K, 0,
                                          cudaMemcpyDeviceToDevice, st);
    if (e == cudaSuccess)
        e = h3::pack_gate_up_rows(static_cast<const bf16 *>(up), static_cast<bf16 *>(W), I, K, 1,
                                  cudaMemcpyDeviceToDevice, st);
    return e == cudaSuccess ? H3ENC_OK : cuda_fail(nullptr, e, "pack gate/up");
}

h3enc_status h3enc_op_gemm_fp8(const void *A, const void *W, const float *sa, const float *sw, void *C, int32_t M,
                               int32_t N, int32_t K, int32_t epilogue, const void *R, const void *DS,
                               const int32_t *vis_rank, int32_t n_vis, void *workspace, int64_t workspace_bytes,
                               int32_t *status, void *stream) {
    if (M < 0 || N <= 0 || K <= 0 || N % 256 || K % 16 || epilogue < 0 || epilogue > 3)
        return fail(nullptr, H3ENC_ERR_INVALID_ARG, "gemm_fp8: bad sizes or epilogue");
    if (M == 0) return H3ENC_OK;
    if (!A || !W || !sa || !sw || !C || ((epilogue == H3ENC_EPI_RESIDUAL || epilogue == H3ENC_EPI_RESIDUAL_DS) && !R) ||
        (epilogue == H3ENC_EPI_RESIDUAL_DS && DS && !vis_rank) || (reinterpret_cast<uintptr_t>(sw) & 15))
        return fail(nullptr, H3ENC_ERR_INVALID_ARG, "gemm_fp8: NULL operand or sw not 16-byte aligned");
    CUtensorMap ta, tw;
    if (!h3::make_tmap_rows_e4m3(&ta, A, M, K, h3::gemm_box_rows_a()) ||
        !h3::make_tmap_rows_e4m3(&tw, W, N, K, h3::gemm_box_rows_w()))
        return fail(nullptr, H3ENC_ERR_INVALID_ARG, "gemm_fp8: operands not 16-byte aligned or driver refused the map");
    h3::GemmPlan p{};
    p.tmA = &ta; p.tmW = &tw; p.M = M; p.N = N; p.K = K; p.epi = epilogue;
    p.fp8 = true; p.sa = sa; p.sw = sw;
    p.C = static_cast<bf16 *>(C);
    p.ldc = epilogue == H3ENC_EPI_SWIGLU ? N / 2 : N;
    p.R = static_cast<const bf16 *>(R);
    p.DS = static_cast<const bf16 *>(DS);
    p.vis_rank = vis_rank;
    p.n_vis = n_vis;
    p.status = status;
    p.num_sms = h3::device_num_sms();
    if (workspace) {
        if (workspace_bytes < (int64_t)h3::gemm_workspace_bytes(p.num_sms) ||
            (reinterpret_cast<uintptr_t>(workspace) & 255))
            return fail(nullptr, H3ENC_ERR_INVALID_ARG, "gemm_fp8: workspace smaller than "
                                                        "h3enc_op_gemm_workspace_bytes() or not 256-byte aligned");
        p.part = static_cast<float *>(workspace);
        p.flags = reinterpret_cast<uint32_t *>(static_cast<char *>(workspace) + h3::gemm_flags_offset(p.num_sms));
    }
    cudaError_t e = h3::launch_gemm(p, static_cast<cudaStream_t>(stream));
    return e == cudaSuccess ? H3ENC_OK : cuda_fail(nullptr, e, "gemm_fp8 launch");
}

h3enc_status h3enc_op_quant_rows(const void *x, int32_t rows, int32_t cols, void *q, float *scale, void *stream) {
    if (!x || !q || !scale || rows < 0 || cols <= 0 || cols % 8 || (reinterpret_cast<uintptr_t>(x) & 15) ||
        (reinterpret_cast<uintptr_t>(q) & 7))
        return fail(nullptr, H3ENC_ERR_INVALID_ARG, "quant_rows: bad args");
    cudaError_t e = h3::launch_quant_rows(static_cast<const bf16 *>(x), cols, rows, cols, static_cast<uint8_t *>(q),
                                          cols, scale, static_cast<cudaStream_t>(stream));
    return e == cudaSuccess ? H3ENC_OK : cuda_fail(nullptr, e, "quant_rows launch");
}

h3enc_status h3enc_op_rmsnorm_q8(const void *x, const void *w, void *q, float *scale, int32_t rows, int32_t cols,
                                 float eps, void *stream) {
    if (!x || !w || !q || !scale || rows < 0 || cols <= 0 || cols % 8 || cols > 8192)
        return fail(nullptr, H3ENC_ERR_INVALID_ARG, "rmsnorm_q8: bad args");
    cudaError_t e = h3::launch_rmsnorm_q8(static_cast<const bf16 *>(x), static_cast<const bf16 *>(w),
                                          static_cast<uint8_t *>(q), scale, rows, cols, eps,
                                          static_cast<cudaStream_t>(stream));
    return e == cudaSuccess ? H3ENC_OK : cuda_fail(nullptr, e, "rmsnorm_q8 launch");
}

h3enc_status h3enc_op_rmsnorm(const void *x, const void *w, void *y, int32_t rows, int32_t cols, float eps,
                              void *stream) {
    if (!x || !w || !y || rows < 0 || cols <= 0 || cols % 8 || cols > 8192)
        return fail(nullptr, H3ENC_ERR_INVALID_ARG, "rmsnorm: bad args");
    cudaError_t e = h3::launch_rmsnorm(static_cast<const bf16 *>(x), static_cast<const bf16 *>(w),
                                       static_cast<bf16 *>(y), rows, cols, eps, static_cast<cudaStream_t>(stream));
    return e == cudaSuccess ? H3ENC_OK : cuda_fail(nullptr, e, "rmsnorm launch");
}

h3enc_status h3enc_op_rope_table(const int32_t *positions, int32_t S, int32_t head_dim, float theta,
                                 const int32_t *section_host, float *cos_tab, float *sin_tab, void *stream) {
    if (!positions || !section_host || !cos_tab || !sin_tab || S < 0 || head_dim < 2 || head_dim > 128 ||
        head_dim % 2 || !(theta > 0.f))
        return fail(nullptr, H3ENC_ERR_INVALID_ARG, "rope_table: bad args");
    h3::RopeParams rp;
    h3::make_rope_params(&rp, head_dim, theta, section_host);
    cudaError_t e = h3::launch_rope_table(positions, S, rp, cos_tab, sin_tab, static_cast<cudaStream_t>(stream));
    return e == cudaSuccess ? H3ENC_OK : cuda_fail(nullptr, e, "rope_table launch");
}

h3enc_status h3enc_op_rope_table_ex(const int32_t *positions, int32_t S, int32_t head_dim, float theta,
                                    const int32_t *section_host, int32_t stride, float *cos_tab, float *sin_tab,
                                    void *stream) {
    if (stride == 0) return h3enc_op_rope_table(positions, S, head_dim, theta, section_host, cos_tab, sin_tab, stream);
    if (!positions || !section_host || !cos_tab || !sin_tab || S < 0 || stride < S || head_dim < 8 ||
        head_dim > 128 || head_dim % 8 || !(theta > 0.f) || (reinterpret_cast<uintptr_t>(cos_tab) & 15) ||
        (reinterpret_cast<uintptr_t>(sin_tab) & 15))
        return fail(nullptr, H3ENC_ERR_INVALID_ARG, "rope_table_ex: bad args");
    h3::RopeParams rp;
    h3::make_rope_params(&rp, head_dim, theta, section_host);
    cudaError_t e =
        h3::launch_rope_table(positions, S, rp, cos_tab, sin_tab, static_cast<cudaStream_t>(stream), stride);
    return e == cudaSuccess ? H3ENC_OK : cuda_fail(nullptr, e, "rope_table_ex launch");
}

}  // extern "C"

namespace {

h3enc_status qkv_rope_op(const void *A, const void *W, void *C, int32_t M, int32_t K, int32_t n_heads,
                         int32_t n_kv_heads, int32_t head_dim, const void *w_q, const void *w_k, float eps,
                         const float *cos_tab, const float *sin_tab, const float *ss_in, float in_eps,
                         void *workspace, int64_t workspace_bytes, int32_t *status, void *stream,
                         int32_t cs_stride = 0) {
    const int64_t N = (int64_t)(n_heads + 2 * n_kv_heads) * head_dim;
    if (cs_stride && (cs_stride < M || (reinterpret_cast<uintptr_t>(cos_tab) & 15) ||
                      (reinterpret_cast<uintptr_t>(sin_tab) & 15)))
        return fail(nullptr, H3ENC_ERR_INVALID_ARG, "gemm_qkv_rope: table stride below M or tables misaligned");
    if (ss_in && K % 128)
        return fail(nullptr, H3ENC_ERR_INVALID_ARG, "gemm_qkv_rope: row statistics need K %% 128 == 0");
    if (M < 0 || K <= 0 || K % 8 || n_heads < 1 || n_kv_heads < 1 || (head_dim != 64 && head_dim != 128) ||
        N % 256 || !w_q || !w_k || !cos_tab || !sin_tab)
        return fail(nullptr, H3ENC_ERR_INVALID_ARG, "gemm_qkv_rope: bad sizes or NULL operand");
    if (M == 0) return H3ENC_OK;
    if (!A || !W || !C) return fail(nullptr, H3ENC_ERR_INVALID_ARG, "gemm_qkv_rope: NULL operand");
    CUtensorMap ta, tw;
    if (!h3::make_tmap_rows(&ta, A, M, K, h3::gemm_box_rows_a()) ||
        !h3::make_tmap_rows(&tw, W, N, K, h3::gemm_box_rows_w()))
        return fail(nullptr, H3ENC_ERR_INVALID_ARG, "gemm_qkv_rope: operands not 16-byte aligned");
    h3::GemmPlan p{};
    p.tmA = &ta; p.tmW = &tw; p.M = M; p.N = (int)N; p.K = K; p.epi = h3::EPI_QKROPE;
    p.C = static_cast<bf16 *>(C);
    p.ldc = (int)N;
    p.status = status;
    p.num_sms = h3::device_num_sms();
    p.wq = static_cast<const bf16 *>(w_q); p.wk = static_cast<const bf16 *>(w_k);
    p.cos_t = cos_tab; p.sin_t = sin_tab; p.cs_rows = cs_stride;
    p.head_dim = head_dim; p.nq = n_heads; p.nkv = n_kv_heads; p.eps = eps;
    p.ss_in = ss_in;
    p.norm_eps = in_eps;
    if (workspace) {
        if (workspace_bytes < (int64_t)h3::gemm_workspace_bytes(p.num_sms) ||
            (reinterpret_cast<uintptr_t>(workspace) & 255))
            return fail(nullptr, H3ENC_ERR_INVALID_ARG, "gemm_qkv_rope: workspace too small or misaligned");
        p.part = static_cast<float *>(workspace);
        p.flags = reinterpret_cast<uint32_t *>(static_cast<char *>(workspace) +
                                               h3::gemm_flags_offset(p.num_sms));
    }
    cudaError_t e = h3::launch_gemm(p, static_cast<cudaStream_t>(stream));
    return e == cudaSuccess ? H3ENC_OK : cuda_fail(nullptr, e, "gemm_qkv_rope launch");
}

}  // namespace

extern "C" {

h3enc_status h3enc_op_gemm_qkv_rope(const void *A, const void *W, void *C, int32_t M, int32_t K, int32_t n_heads,
                                    int32_t n_kv_heads, int32_t head_dim, const void *w_q, const void *w_k, float eps,
                                    const float *cos_tab, const float *sin_tab, void *workspace,
                                    int64_t workspace_bytes, int32_t *status, void *stream) {
    return qkv_rope_op(A, W, C, M, K, n_heads, n_kv_heads, head_dim, w_q, w_k, eps, cos_tab, sin_tab, nullptr, 0.f,
                       workspace, workspace_bytes, status, stream);
}

h3enc_status h3enc_op_gemm_qkv_rope_rms(const void *A, const void *W, void *C, int32_t M, int32_t K,
                                        int32_t n_heads, int32_t n_kv_heads, int32_t head_dim, const void *w_q,
                                        const void *w_k, float eps, const float *cos_tab, const float *sin_tab,
                                        const float *ss_in, float in_eps, void *workspace, int64_t workspace_bytes,
                                        int32_t *status, void *stream) {
    if (!ss_in) return fail(nullptr, H3ENC_ERR_INVALID_ARG, "gemm_qkv_rope_rms: ss_in is NULL");
    return qkv_rope_op(A, W, C, M, K, n_heads, n_kv_heads, head_dim, w_q, w_k, eps, cos_tab, sin_tab, ss_in, in_eps,
                       workspace, workspace_bytes, status, stream);
}

h3enc_status h3enc_op_gemm_qkv_rope_ex(const void *A, const void *W, void *C, int32_t M, int32_t K,
                                       int32_t n_heads, int32_t n_kv_heads, int32_t head_dim, const void *w_q,
                                       const void *w_k, float eps, const float *cos_tab, const float *sin_tab,
                                       int32_t cs_stride, const float *ss_in, float in_eps, void *workspace,
                                       int64_t workspace_bytes, int32_t *status, void *stream) {
    if (cs_stride < 0) return fail(nullptr, H3ENC_ERR_INVALID_ARG, "gemm_qkv_rope_ex: negative table stride");
    return qkv_rope_op(A, W, C, M, K, n_heads, n_kv_heads, head_dim, w_q, w_k, eps, cos_tab, sin_tab, ss_in, in_eps,
                       workspace, workspace_bytes, status, stream, cs_stride);
}

h3enc_status h3enc_op_attention(const void *qkv, void *o, int32_t S, int32_t n_heads, int32_t n_kv_heads,
                                int32_t head_dim, const int32_t *cu_seqlens, int32_t n_seqs, void *stream) {
    if (!qkv || !o || S < 0 || n_heads < 1 || n_kv_heads < 1 || n_heads % n_kv_heads ||
        (head_dim != 64 && head_dim != 128))
        return fail(nullptr, H3ENC_ERR_INVALID_ARG, "attention: bad args");
    if (cu_seqlens) {
        if (n_seqs < 1 || n_seqs > h3::kMaxSeqs || cu_seqlens[0] != 0 || cu_seqlens[n_seqs] != S)
            return fail(nullptr, H3ENC_ERR_INVALID_ARG, "attention: bad cu_seqlens");
        for (int i = 0; i < n_seqs; ++i)
            if (cu_seqlens[i + 1] < cu_seqlens[i]) return fail(nullptr, H3ENC_ERR_INVALID_ARG, "attention: bad cu_seqlens");
    }
    cudaError_t e = h3::launch_attention(static_cast<const bf16 *>(qkv), static_cast<bf16 *>(o), S, n_heads,
                                         n_kv_heads, head_dim, cu_seqlens, n_seqs, nullptr,
                                         static_cast<cudaStream_t>(stream));
    return e == cudaSuccess ? H3ENC_OK : cuda_fail(nullptr, e, "attention launch");
}

h3enc_status h3enc_op_embed(const int32_t *ids, const void *table, int32_t vocab, int32_t hidden, void *out, int32_t S,
                            int32_t *status, void *stream) {
    if (!ids || !table || !out || vocab < 1 || hidden < 8 || hidden % 8 || S < 0)
        return fail(nullptr, H3ENC_ERR_INVALID_ARG, "embed: bad args");
    cudaError_t e = h3::launch_embed(ids, static_cast<const bf16 *>(table), vocab, hidden, static_cast<bf16 *>(out), S,
                                     status, static_cast<cudaStream_t>(stream));
    return e == cudaSuccess ? H3ENC_OK : cuda_fail(nullptr, e, "embed launch");
}

h3enc_status h3enc_op_vis_rank(const uint8_t *mask, int32_t S, int32_t n_vis, int32_t *vis_rank, int32_t *status,
                               void *stream) {
    if (!mask || !vis_rank || S < 0) return fail(nullptr, H3ENC_ERR_INVALID_ARG, "vis_rank: bad args");
    cudaError_t e = h3::launch_vis_rank(mask, S, n_vis, vis_rank, status, static_cast<cudaStream_t>(stream));
    return e == cudaSuccess ? H3ENC_OK : cuda_fail(nullptr, e, "vis_rank launch");
}

}  // extern "C"
