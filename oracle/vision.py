"""Plain CPU restatement of the Qwen3-VL vision tower.

TEST INFRASTRUCTURE ONLY (see the package docstring).

Page 1 ("vllm-omni vllm_omni/diffusion/models/minimax_h3/encoder.py"), section
"Qwen3-VL vision tower": ``MiniMaxH3Qwen3VLVisionPatchEmbed`` (Conv3d whose
stride equals its kernel), ``fast_pos_embed_interpolate`` (bilinear lookup in a
square table of learned position embeddings, then the 2x2 merge order),
``rot_pos_emb`` with ``MiniMaxH3Qwen3VLVisionRotaryEmbedding`` (2-D rotary
angles: row frequencies, then column frequencies), ``MiniMaxH3Qwen3VLVisionBlock``
(LayerNorm, attention with a bias-carrying packed QKV, rotary q/k,
bidirectional attention inside each frame, projection; LayerNorm, tanh-GELU
MLP), ``MiniMaxH3Qwen3VLVisionPatchMerger`` (LayerNorm before or after grouping
the 2x2 tokens, then linear, exact GELU, linear) and the model's ``forward``
(DeepStack features from the mergers of the listed blocks).

Arithmetic in float32 by default (float64 for pinned small cases); weights
and inputs are bf16 values widened exactly.  ``storage`` names the hand-over
points rounded to bf16 (the GPU's storage points) for the tolerance floor.
Readings where the pages leave the numerics open: the interpolation weights
and products are kept in fp32 (the page casts the weights to the model dtype
first); LayerNorm uses the biased variance over the last axis in fp32.
"""
from __future__ import annotations

import math

import numpy as np

from .qwen3vl_text import round_to_bf16, rotate_half

__all__ = ["layer_norm", "gelu_tanh", "gelu_erf", "patch_embed", "pos_embed_interpolate", "merge_order",
           "rot_pos_angles", "vision_attention", "vision_block", "patch_merger", "vision_forward",
           "VISION_STORAGE_POINTS"]

VISION_STORAGE_POINTS = ("h", "ln", "qkv", "attn", "act", "merged_ln", "merged_act")


def _store(t: np.ndarray, point: str, storage) -> np.ndarray:
    return round_to_bf16(t).astype(t.dtype, copy=False) if storage and point in storage else t


def layer_norm(x: np.ndarray, w: np.ndarray, b: np.ndarray, eps: float) -> np.ndarray:
    """``nn.LayerNorm`` over the last axis: ``(x - mean) / sqrt(var + eps) * w + b``, with the
    biased variance (mean of squared deviations)."""
    mean = np.mean(x, axis=-1, keepdims=True)
    dev = x - mean
    var = np.mean(dev * dev, axis=-1, keepdims=True)
    return dev / np.sqrt(var + x.dtype.type(eps)) * w + b


def gelu_tanh(x: np.ndarray) -> np.ndarray:
    """The tanh form of GELU the vision MLP uses (``nn.GELU(approximate="tanh")``):
    ``x/2 * (1 + tanh(sqrt(2/pi) * (x + 0.044715 x^3)))``."""
    c = x.dtype.type(math.sqrt(2.0 / math.pi))
    return x.dtype.type(0.5) * x * (1 + np.tanh(c * (x + x.dtype.type(0.044715) * x * x * x)))


def gelu_erf(x: np.ndarray) -> np.ndarray:
    """Exact GELU of the mergers (``nn.GELU()``): ``x * Phi(x)`` with the normal CDF
    ``Phi(x) = (1 + erf(x / sqrt 2)) / 2``."""
    from scipy.special import erf
    return (x * 0.5 * (1.0 + erf(x / np.sqrt(2.0)))).astype(x.dtype, copy=False)


def patch_embed(pixels: np.ndarray, w: np.ndarray, b: np.ndarray) -> np.ndarray:
    """Conv3d with kernel = stride = (T, P, P) over each patch volume [C, T, P, P]: one
    output vector per patch, the dot product of the flattened volume with each flattened
    filter, plus the bias.  pixels [n, C*T*P*P] (the (C, T, P, P) order), w [hidden, C, T, P, P]."""
    return pixels @ w.reshape(w.shape[0], -1).T + b


def merge_order(t: int, h: int, w: int, m: int) -> np.ndarray:
    """(frame, row, column) of every patch in the order the tower keeps them: frames, then
    blocks of m x m patches in row-major block order, then the m x m patches of a block
    row-major (the view/permute of ``fast_pos_embed_interpolate`` and ``rot_pos_emb``)."""
    out = []
    for f in range(t):
        for hb in range(h // m):
            for wb in range(w // m):
                for hi in range(m):
                    for wi in range(m):
                        out.append((f, hb * m + hi, wb * m + wi))
    return np.array(out, dtype=np.int64).reshape(-1, 3)


def pos_embed_interpolate(table: np.ndarray, grids, merge: int) -> np.ndarray:
    """Learned position embeddings of every patch: the square table (G x G rows, G =
    sqrt(rows)) sampled bilinearly at h x w evenly spaced points from corner to corner,
    repeated for every frame, in merge order.  Point (i, j) of a grid sits at table
    coordinates (i (G-1)/(h-1), j (G-1)/(w-1)) (fp32, as ``torch.linspace``), truncated to
    the lower corner, the upper one clipped to G-1."""
    rows = table.shape[0]
    G = int(round(math.sqrt(rows)))
    outs = []
    for t, h, w in grids:
        hs = np.linspace(0, G - 1, h, dtype=np.float32)
        ws = np.linspace(0, G - 1, w, dtype=np.float32)
        grid = np.zeros((h, w, table.shape[1]), dtype=table.dtype)
        for i in range(h):
            h0 = int(hs[i])
            h1 = min(h0 + 1, G - 1)
            dh = np.float32(hs[i] - np.float32(h0))
            for j in range(w):
                w0 = int(ws[j])
                w1 = min(w0 + 1, G - 1)
                dw = np.float32(ws[j] - np.float32(w0))
                c00 = (np.float32(1) - dh) * (np.float32(1) - dw)
                c01 = (np.float32(1) - dh) * dw
                c10 = dh * (np.float32(1) - dw)
                c11 = dh * dw
                grid[i, j] = (table[h0 * G + w0] * c00 + table[h0 * G + w1] * c01 +
                              table[h1 * G + w0] * c10 + table[h1 * G + w1] * c11)
        order = merge_order(t, h, w, merge)
        outs.append(grid[order[:, 1], order[:, 2]])
    return np.concatenate(outs, axis=0)


def rot_pos_angles(grids, head_dim: int, merge: int, theta: float = 10000.0) -> np.ndarray:
    """2-D rotary angles [n, head_dim/2] of every patch in merge order: with the
    ``head_dim/2``-wide rotary embedding (inv_freq[j] = theta^(-2j/(head_dim/2)), fp32),
    the first head_dim/4 angles are row * inv_freq, the next head_dim/4 column * inv_freq
    (fp32 products).  cos/sin of the concatenation (angles, angles) rotate q and k."""
    dim = head_dim // 2
    inv = (1.0 / (np.float64(theta) ** (np.arange(0, dim, 2, dtype=np.float64) / dim))).astype(np.float32)
    outs = []
    for t, h, w in grids:
        order = merge_order(t, h, w, merge)
        r = order[:, 1].astype(np.float32)[:, None] * inv[None, :]
        c = order[:, 2].astype(np.float32)[:, None] * inv[None, :]
        outs.append(np.concatenate([r, c], axis=1).astype(np.float32))
    return np.concatenate(outs, axis=0)


def _rope(x: np.ndarray, ang: np.ndarray) -> np.ndarray:
    """x [n, heads, d] rotated by angles [n, d/2] (pairs j, j + d/2; cos/sin in float64 of
    the fp32 angle, as the text oracle does)."""
    full = np.concatenate([ang, ang], axis=-1).astype(np.float64)
    cos = np.cos(full).astype(x.dtype)[:, None, :]
    sin = np.sin(full).astype(x.dtype)[:, None, :]
    return x * cos + rotate_half(x) * sin


def vision_attention(x, w_qkv, b_qkv, w_proj, b_proj, ang, cu, heads, storage=None):
    """Packed QKV (with bias) -> rotary q/k -> softmax(q k^T / sqrt(d)) v within each
    segment [cu[i], cu[i+1]) (no causal mask) -> projection (with bias)."""
    n, hid = x.shape
    d = hid // heads
    qkv = (x @ w_qkv.T + b_qkv).reshape(n, 3, heads, d)
    q, k, v = qkv[:, 0], qkv[:, 1], qkv[:, 2]
    q = _store(_rope(q, ang), "qkv", storage)
    k = _store(_rope(k, ang), "qkv", storage)
    v = _store(v, "qkv", storage)
    out = np.zeros((n, heads, d), dtype=x.dtype)
    scale = x.dtype.type(1.0 / math.sqrt(d))
    for a, b in zip(cu[:-1], cu[1:]):
        for hh in range(heads):
            s = (q[a:b, hh] @ k[a:b, hh].T) * scale
            s = s - np.max(s, axis=1, keepdims=True)
            p = np.exp(s)
            p = p / np.sum(p, axis=1, keepdims=True)
            out[a:b, hh] = p @ v[a:b, hh]
    o = _store(out.reshape(n, hid), "attn", storage)
    return o @ w_proj.T + b_proj


def vision_block(x, w, ang, cu, cfg, storage=None):
    """``x + attn(LN1(x))`` then ``x + fc2(gelu_tanh(fc1(LN2(x))))``; w maps the block's
    module paths (``norm1.weight`` ...) to arrays."""
    y = _store(layer_norm(x, w["norm1.weight"], w["norm1.bias"], cfg.ln_eps), "ln", storage)
    x = _store(x + vision_attention(y, w["attn.qkv.weight"], w["attn.qkv.bias"], w["attn.proj.weight"],
                                    w["attn.proj.bias"], ang, cu, cfg.num_heads, storage), "h", storage)
    y = _store(layer_norm(x, w["norm2.weight"], w["norm2.bias"], cfg.ln_eps), "ln", storage)
    a = _store(gelu_tanh(y @ w["mlp.linear_fc1.weight"].T + w["mlp.linear_fc1.bias"]), "act", storage)
    return _store(x + (a @ w["mlp.linear_fc2.weight"].T + w["mlp.linear_fc2.bias"]), "h", storage)


def patch_merger(x, w, cfg, postshuffle: bool, storage=None):
    """Group each m x m block's tokens (consecutive in merge order) into one row of width
    hidden * m^2; LayerNorm over hidden before grouping (main merger) or over the grouped
    row after it (DeepStack mergers); then fc1, exact GELU, fc2 (all with bias)."""
    mh = cfg.merged_hidden
    if postshuffle:
        y = layer_norm(x.reshape(-1, mh), w["norm.weight"], w["norm.bias"], cfg.ln_eps)
    else:
        y = layer_norm(x, w["norm.weight"], w["norm.bias"], cfg.ln_eps).reshape(-1, mh)
    y = _store(y, "merged_ln", storage)
    a = _store(gelu_erf(y @ w["linear_fc1.weight"].T + w["linear_fc1.bias"]), "merged_act", storage)
    return a @ w["linear_fc2.weight"].T + w["linear_fc2.bias"]


def vision_forward(pixels: np.ndarray, grids, cfg, weights: dict, storage=None, dtype=np.float32):
    """The tower's forward: returns (merged embeddings [n/m^2, out_hidden], DeepStack
    features, one [n/m^2, out_hidden] per listed block in list order).  ``weights`` maps
    names without the ``model.visual.`` prefix to arrays."""
    W = {k: np.asarray(v, dtype=dtype) for k, v in weights.items()}
    x = patch_embed(np.asarray(pixels, dtype=dtype), W["patch_embed.proj.weight"], W["patch_embed.proj.bias"])
    x = _store(x + pos_embed_interpolate(W["pos_embed.weight"], grids, cfg.spatial_merge_size), "h", storage)
    ang = rot_pos_angles(grids, cfg.head_dim, cfg.spatial_merge_size, cfg.rope_theta)
    cu = [0]
    for t, h, w in grids:   # one attention segment per frame
        for _ in range(t):
            cu.append(cu[-1] + h * w)
    feats = []
    for b in range(cfg.depth):
        blk = {k[len(f"blocks.{b}."):]: v for k, v in W.items() if k.startswith(f"blocks.{b}.")}
        x = vision_block(x, blk, ang, cu, cfg, storage)
        if b in cfg.deepstack_visual_indexes:
            j = cfg.deepstack_visual_indexes.index(b)
            mw = {k[len(f"deepstack_merger_list.{j}."):]: v for k, v in W.items()
                  if k.startswith(f"deepstack_merger_list.{j}.")}
            feats.append(patch_merger(x, mw, cfg, True, storage))
    mw = {k[len("merger."):]: v for k, v in W.items() if k.startswith("merger.")}
    return patch_merger(x, mw, cfg, False, storage), feats
