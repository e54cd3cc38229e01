"""Plain CPU restatement of the Qwen3-VL text-decoder prefill.

TEST INFRASTRUCTURE ONLY (see the package docstring).  Every function names
the part of the page "vllm-omni vllm_omni/diffusion/models/minimax_h3/
encoder.py" (page 1; page 2 is the same module's API page) that it follows.
Arithmetic is float32 by default (``dtype=np.float64`` for the small pinned
cases); inputs and weights are bf16 values widened exactly.  Nothing is fused,
blocked or reordered beyond what the definition states; numpy ``@`` is the
only library primitive used for contractions.
"""
from __future__ import annotations

import math

import numpy as np

__all__ = [
    "bf16_bits_to_float", "round_to_bf16", "linear", "rms_norm", "rope_inv_freq",
    "mrope_axis_of_pair", "rope_cos_sin", "rotate_half", "apply_rope", "silu",
    "causal_gqa_attention", "deepstack_add", "decoder_layer", "forward", "LayerWeights",
    "layer_weights_from_bits", "STORAGE_POINTS",
]


# ---------------------------------------------------------------------------
# bf16 <-> float (storage format of every tensor on the pages: plain BF16)
# ---------------------------------------------------------------------------

def bf16_bits_to_float(bits: np.ndarray, dtype=np.float32) -> np.ndarray:
    """Exact value of bf16 bit patterns (uint16) as float32/float64."""
    b = np.asarray(bits, dtype=np.uint16).astype(np.uint32) << np.uint32(16)
    return b.view(np.float32).astype(dtype, copy=False)


def round_to_bf16(x: np.ndarray) -> np.ndarray:
    """Round to the nearest bf16 value (ties to even); returns float32 values.

    Used to hand a bf16-typed tensor to the next consumer, exactly as a BF16
    model stores it.
    """
    f = np.asarray(x, dtype=np.float32)
    b = f.view(np.uint32).astype(np.uint64)
    b = (b + 0x7FFF + ((b >> 16) & 1)) >> 16
    return (b.astype(np.uint32) << np.uint32(16)).view(np.float32)


# ---------------------------------------------------------------------------
# elementary steps
# ---------------------------------------------------------------------------

def linear(x: np.ndarray, w: np.ndarray) -> np.ndarray:
    """``F.linear(x, w)``: ``x @ w.T`` with ``w`` stored ``[out, in]`` (no bias).

    Page 1, the QKV / merged-column / row-parallel linear classes (bias=False);
    "Three separate GEMMs" in ``MiniMaxH3Qwen3VLTextAttention.forward``.
    """
    return x @ w.T


def rms_norm(x: np.ndarray, w: np.ndarray, eps: float) -> np.ndarray:
    """RMSNorm over the last axis: ``w * x / sqrt(mean(x**2) + eps)``.

    Page 1, ``MiniMaxH3Qwen3VLRMSNorm`` (variance reduction and scaling in
    float32, gamma of model dtype).  Used as input/post-attention layernorm
    over the hidden size and as q_norm/k_norm over head_dim.
    """
    ms = np.mean(x * x, axis=-1, keepdims=True)
    return x / np.sqrt(ms + x.dtype.type(eps)) * w


def rope_inv_freq(head_dim: int, theta: float) -> np.ndarray:
    """``inv_freq[j] = 1 / theta**(2j/d)``, j = 0..d/2-1, as float32.

    Page 1, ``MiniMaxH3Qwen3VLTextRotaryEmbedding._get_inv_freq`` (the page
    insists the inverse frequencies are float32).  Evaluated in float64 and
    rounded once to float32.
    """
    j = np.arange(0, head_dim, 2, dtype=np.float64)
    return (1.0 / (float(theta) ** (j / head_dim))).astype(np.float32)


def mrope_axis_of_pair(half_dim: int, section) -> np.ndarray:
    """Which position axis (0=T, 1=H, 2=W) drives frequency index j.

    Page 1, ``_apply_interleaved_mrope``: start from the T frequencies, then
    for H (offset 1) and W (offset 2) overwrite indices ``offset, offset+3,
    ...`` below ``3 * section[axis]``.
    """
    axis = np.zeros(half_dim, dtype=np.int64)
    for a, offset in ((1, 1), (2, 2)):
        for j in range(offset, min(3 * int(section[a]), half_dim), 3):
            axis[j] = a
    return axis


def rope_cos_sin(positions: np.ndarray, head_dim: int, theta: float, section, dtype=np.float32):
    """cos/sin tables ``[S, head_dim]`` for interleaved 3-D M-RoPE.

    Page 1, ``MiniMaxH3Qwen3VLTextRotaryEmbedding.forward``:
    ``freqs[a, s, j] = float32(pos[a, s]) * inv_freq[j]`` (a float32 product),
    interleaved per ``mrope_axis_of_pair``, ``emb = cat(freqs, freqs)``.  The
    page casts cos/sin to the activation dtype (bf16); this oracle keeps the
    cosine and sine of the float32 angle at full precision instead.
    """
    pos = np.asarray(positions).astype(np.float32)           # [3, S]
    inv = rope_inv_freq(head_dim, theta)                     # [d/2]
    freqs = pos[:, :, None] * inv[None, None, :]             # [3, S, d/2] float32
    axis = mrope_axis_of_pair(head_dim // 2, section)
    f = freqs[axis, :, np.arange(head_dim // 2)].T           # [S, d/2]
    emb = np.concatenate([f, f], axis=-1).astype(np.float64)
    return np.cos(emb).astype(dtype), np.sin(emb).astype(dtype)


def rotate_half(x: np.ndarray) -> np.ndarray:
    """``cat(-x[..., d/2:], x[..., :d/2])`` (page 1, ``_rotate_half``)."""
    h = x.shape[-1] // 2
    return np.concatenate([-x[..., h:], x[..., :h]], axis=-1)


def apply_rope(x: np.ndarray, cos: np.ndarray, sin: np.ndarray) -> np.ndarray:
    """``x * cos + rotate_half(x) * sin`` for x ``[S, heads, d]``, cos/sin ``[S, d]``.

    Page 1, ``_apply_rotary_pos_emb`` (cos/sin broadcast over heads).
    """
    return x * cos[:, None, :] + rotate_half(x) * sin[:, None, :]


def silu(z: np.ndarray) -> np.ndarray:
    """``z * sigmoid(z)`` (``F.silu`` in page 1, ``MiniMaxH3Qwen3VLTextMLP``)."""
    return z / (1.0 + np.exp(-z))


def causal_gqa_attention(q: np.ndarray, k: np.ndarray, v: np.ndarray, cu_seqlens=None,
                         q_chunk: int = 512) -> np.ndarray:
    """Causal GQA softmax attention, one packed sequence or several.

    q ``[S, nq, d]``, k/v ``[S, nkv, d]`` -> ``[S, nq*d]`` (head-major columns).
    Page 1, ``MiniMaxH3Qwen3VLTextAttention.forward``: K/V repeated with
    ``repeat_interleave(nq // nkv)`` so q head h reads kv head ``h // (nq//nkv)``;
    ``scaled_dot_product_attention(is_causal=True)`` with the default scale
    ``1/sqrt(d)``; output ``transpose(1, 2).reshape(S, nq*d)``.  Segments of
    ``cu_seqlens`` attend only within themselves (block-diagonal causal mask);
    the pages encode one sequence, which is the one-segment case.
    """
    s, nq, d = q.shape
    nkv = k.shape[1]
    group = nq // nkv
    if cu_seqlens is None:
        cu_seqlens = [0, s]
    scale = q.dtype.type(1.0 / math.sqrt(d))
    out = np.zeros((s, nq, d), dtype=q.dtype)
    for a, b in zip(cu_seqlens[:-1], cu_seqlens[1:]):
        a, b = int(a), int(b)
        for h in range(nq):
            g = h // group
            kk = k[a:b, g, :]
            vv = v[a:b, g, :]
            for r0 in range(0, b - a, q_chunk):
                r1 = min(b - a, r0 + q_chunk)
                sc = (q[a + r0:a + r1, h, :] @ kk[:r1].T) * scale          # [rows, keys<r1]
                i = np.arange(r0, r1)[:, None]
                j = np.arange(r1)[None, :]
                sc = np.where(j <= i, sc, -np.inf)
                sc = sc - sc.max(axis=-1, keepdims=True)
                p = np.exp(sc)
                p = p / p.sum(axis=-1, keepdims=True)
                out[a + r0:a + r1, h, :] = p @ vv[:r1]
    return out.reshape(s, nq * d)


def deepstack_add(x: np.ndarray, visual_mask: np.ndarray, feats: np.ndarray) -> np.ndarray:
    """``x[mask, :] = x[mask, :] + feats``: row j of ``feats`` goes to the j-th
    masked position in sequence order (page 1,
    ``MiniMaxH3Qwen3VLTextModel._deepstack_process``)."""
    y = x.copy()
    idx = np.nonzero(np.asarray(visual_mask).astype(bool))[0]
    y[idx, :] = y[idx, :] + feats
    return y


# ---------------------------------------------------------------------------
# layer and model
# ---------------------------------------------------------------------------

class LayerWeights(dict):
    """Float weights of one decoder layer, keyed by the short HF suffix
    (``q_proj``, ``k_proj``, ``v_proj``, ``o_proj``, ``q_norm``, ``k_norm``,
    ``gate_proj``, ``up_proj``, ``down_proj``, ``input_layernorm``,
    ``post_attention_layernorm``)."""


def layer_weights_from_bits(named_bits: dict, dtype=np.float32) -> LayerWeights:
    """Build ``LayerWeights`` from {HF name: bf16 bits}; names are matched on
    their last two components (``self_attn.q_proj.weight`` -> ``q_proj``)."""
    lw = LayerWeights()
    for name, bits in named_bits.items():
        key = name.split(".")[-2]
        lw[key] = bf16_bits_to_float(bits, dtype)
    return lw


STORAGE_POINTS = ("y", "qk_proj", "v", "qk", "attn", "act", "h")


def _store(t: np.ndarray, point: str, storage) -> np.ndarray:
    """Hand tensor ``t`` to the next step: unchanged, or rounded to bf16 when
    ``point`` is in ``storage`` (a set of names from ``STORAGE_POINTS``)."""
    return round_to_bf16(t).astype(t.dtype, copy=False) if storage and point in storage else t


def decoder_layer(x: np.ndarray, w: LayerWeights, cos: np.ndarray, sin: np.ndarray, cfg,
                  cu_seqlens=None, storage=None, fp8=False) -> np.ndarray:
    """One decoder layer (page 1, ``MiniMaxH3Qwen3VLTextDecoderLayer.forward``).

    residual = x; y = input_layernorm(x); attention; x = residual + attn;
    residual = x; y = post_attention_layernorm(x); x = residual + mlp(y).
    Attention (``MiniMaxH3Qwen3VLTextAttention.forward``): q/k/v projections,
    per-head q_norm/k_norm over head_dim, M-RoPE on q and k, causal GQA SDPA,
    o_proj.  MLP (``MiniMaxH3Qwen3VLTextMLP.forward``): down(silu(gate) * up).

    ``storage`` (default None: every tensor exact) names the hand-over points
    rounded to bf16, as a BF16 model stores them: "y" (norm outputs), "qk_proj"
    (q/k projections), "v" (v projection), "qk" (q/k after norm and RoPE),
    "attn" (attention output),
    "act" (SwiGLU output), "h" (residual stream).  With all of them this is the
    rounding floor of a pipeline that keeps exactly those tensors in bf16.

    ``fp8`` runs the four projections as online-FP8 linears (``oracle.fp8``):
    the packed QKV and gate/up projections of the quantised branch are, per output
    channel, the same as the separate q/k/v and gate/up products computed here.
    """
    if fp8:
        from .fp8 import fp8_linear as lin
    else:
        lin = linear
    s = x.shape[0]
    d, nq, nkv = cfg.head_dim, cfg.n_heads, cfg.n_kv_heads
    residual = x
    y = _store(rms_norm(x, w["input_layernorm"], cfg.rms_eps), "y", storage)
    q = _store(lin(y, w["q_proj"]), "qk_proj", storage).reshape(s, nq, d)
    k = _store(lin(y, w["k_proj"]), "qk_proj", storage).reshape(s, nkv, d)
    v = _store(lin(y, w["v_proj"]), "v", storage).reshape(s, nkv, d)
    q = rms_norm(q, w["q_norm"], cfg.rms_eps)
    k = rms_norm(k, w["k_norm"], cfg.rms_eps)
    q = _store(apply_rope(q, cos, sin), "qk", storage)
    k = _store(apply_rope(k, cos, sin), "qk", storage)
    attn = _store(causal_gqa_attention(q, k, v, cu_seqlens), "attn", storage)
    x = _store(residual + lin(attn, w["o_proj"]), "h", storage)
    residual = x
    y = _store(rms_norm(x, w["post_attention_layernorm"], cfg.rms_eps), "y", storage)
    act = _store(silu(lin(y, w["gate_proj"])) * lin(y, w["up_proj"]), "act", storage)
    return _store(residual + lin(act, w["down_proj"]), "h", storage)


def forward(inputs_embeds: np.ndarray, positions: np.ndarray, cfg, get_layer,
            visual_mask=None, deepstack=None, cu_seqlens=None, layers=None,
            capture=None, dtype=np.float32, storage=None, fp8=False) -> np.ndarray:
    """Text-model forward returning the unnormalised last hidden state.

    Page 1, ``MiniMaxH3Qwen3VLTextModel.forward``: cos/sin computed once from
    ``positions [3, S]``; for each kept layer, run the decoder layer, then if
    ``layer_idx < len(deepstack)`` add ``deepstack[layer_idx]`` at the visual
    positions.  No final norm (the encoder returns ``hidden_states[50]``,
    the state after the last kept layer).  ``get_layer(l)`` returns
    ``LayerWeights``; ``layers`` (default ``range(cfg.num_layers)``) allows a
    sub-range with global layer indices; ``capture`` (a list) receives the
    state after every layer; ``storage`` as in ``decoder_layer`` (the
    DeepStack sum is a residual-stream hand-over, point "h"); ``fp8`` as in
    ``decoder_layer``.
    """
    x = np.asarray(inputs_embeds, dtype=dtype)
    cos, sin = rope_cos_sin(positions, cfg.head_dim, cfg.rope_theta, cfg.mrope_section, dtype)
    if layers is None:
        layers = range(cfg.num_layers)
    for l in layers:
        x = decoder_layer(x, get_layer(l), cos, sin, cfg, cu_seqlens, storage, fp8)
        if deepstack is not None and l < len(deepstack):
            x = _store(deepstack_add(x, visual_mask, np.asarray(deepstack[l], dtype=dtype)), "h", storage)
        if capture is not None:
            capture.append(x.copy())
    return x
