"""Seeded synthetic workloads for the Qwen3-VL text-decoder prefill (MiniMax H3
layer-50 encoder).

This module is shared by the CPU oracle and the GPU path.  It holds model
shapes, the five benchmark workloads and a counter-based random generator; it
holds none of the decoder's arithmetic.

Every random tensor is a pure function of (seed, tensor name, element index):

    h   = mix32(mix32(idx * 0x61C88647 ^ k1) ^ k2)         (32-bit integer hash)
    out = TABLE[h >> 16]                                   (65536-entry bf16 table)

``TABLE[i]`` is ``bf16(mean + sigma * Phi^-1((i + 0.5) / 65536))``, so a value
is an exact table lookup and the numpy (host, threaded) and torch (any device)
implementations give bit-identical bf16 tensors.  Element rows can be drawn
on their own (``rows=``), which lets the oracle fetch only the embedding rows
a sequence uses.

Shapes follow the HF Qwen3-VL checkpoint layout ``[out_features, in_features]``
("vllm-omni minimax_h3/encoder.py", ``_map_weight_name`` / ``load_weights``).
"""
from __future__ import annotations

import dataclasses
import os
import statistics
import zlib
from concurrent.futures import ThreadPoolExecutor
from functools import lru_cache

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))

__all__ = [
    "ModelConfig", "Workload", "MODELS", "WORKLOADS", "workload",
    "layer_weight_specs", "embed_name", "normal_bf16", "gen_weight",
    "gen_inputs", "bf16_bits_to_torch", "uniform_ints",
    "VisionConfig", "VisionWorkload", "VISION_WORKLOADS", "vision_workload", "vision_weight_specs",
    "gen_vision_inputs",
]

_M32 = 0xFFFFFFFF
_C0 = 0x61C88647  # all multipliers < 2**31 so int64 products never overflow
_C1 = 0x7FEB352D
_C2 = 0x5BD1E995


@dataclasses.dataclass(frozen=True)
class ModelConfig:
    num_layers: int
    hidden: int
    n_heads: int
    n_kv_heads: int
    head_dim: int
    intermediate: int
    vocab: int
    rms_eps: float
    rope_theta: float
    mrope_section: tuple

    @property
    def qkv_out(self) -> int:
        return (self.n_heads + 2 * self.n_kv_heads) * self.head_dim

    def params_per_layer(self) -> int:
        h, d = self.hidden, self.head_dim
        lin = h * self.qkv_out + self.n_heads * d * h + 3 * h * self.intermediate
        return lin + 2 * h + 2 * d


@dataclasses.dataclass(frozen=True)
class Workload:
    name: str
    model: ModelConfig
    seed: int
    # token layout: list of ("text", n) / ("grid", t, h, w) runs, or "varlen"
    runs: tuple = ()
    n_prompts: int = 0
    prompt_len: tuple = (0, 0)
    deepstack_levels: int = 0
    deepstack_sigma: float = 0.0
    embeds_input: bool = False   # one layer fed with N(0,1) hidden input


TINY = ModelConfig(2, 256, 4, 2, 64, 768, 1024, 1e-6, 1e6, (12, 10, 10))
FULL1 = ModelConfig(1, 5120, 64, 8, 128, 25600, 0, 1e-6, 5e6, (24, 20, 20))
FULL50 = ModelConfig(50, 5120, 64, 8, 128, 25600, 151936, 1e-6, 5e6, (24, 20, 20))

MODELS = {"tiny": TINY, "layer": FULL1, "full50": FULL50}

WORKLOADS = {
    0: Workload("tiny-2layer-seq48", TINY, 1000,
                runs=(("text", 8), ("grid", 1, 4, 8), ("text", 8)),
                deepstack_levels=1, deepstack_sigma=0.1),
    1: Workload("one-full-layer-seq512", FULL1, 1001,
                runs=(("text", 512),), embeds_input=True),
    2: Workload("50layer-seq1024-image", FULL50, 1002,
                runs=(("text", 128), ("grid", 1, 24, 32), ("text", 128)),
                deepstack_levels=3, deepstack_sigma=0.5),
    3: Workload("50layer-seq8192-video", FULL50, 1003,
                runs=(("text", 1024), ("grid", 8, 24, 32), ("text", 1024)),
                deepstack_levels=3, deepstack_sigma=0.5),
    4: Workload("50layer-varlen16", FULL50, 1004,
                n_prompts=16, prompt_len=(77, 512)),
}


def workload(i: int) -> Workload:
    return WORKLOADS[i]


# ---------------------------------------------------------------------------
# counter-based generator
# ---------------------------------------------------------------------------

def _keys(seed: int, name: str):
    c = zlib.crc32(name.encode())
    k1 = (c ^ (seed * 0x2545F491)) & _M32
    k2 = (zlib.crc32(name.encode(), seed & _M32) * 0x3C6EF372 + seed) & _M32
    return k1, k2


def _mix32_np(x):
    x ^= x >> np.uint32(16)
    x *= np.uint32(_C1)
    x ^= x >> np.uint32(15)
    x *= np.uint32(_C2)
    x ^= x >> np.uint32(16)
    return x


def _hash_np(idx_u32, k1, k2):
    x = idx_u32 * np.uint32(_C0)
    x ^= np.uint32(k1)
    x = _mix32_np(x)
    x ^= np.uint32(k2)
    return _mix32_np(x)


def _mix32_torch(x):
    x = x ^ (x >> 16)
    x = (x * _C1) & _M32
    x = x ^ (x >> 15)
    x = (x * _C2) & _M32
    return x ^ (x >> 16)


def _hash_torch(idx_i64, k1, k2):
    x = (idx_i64 * _C0) & _M32
    x = _mix32_torch(x ^ k1)
    return _mix32_torch(x ^ k2)


@lru_cache(maxsize=None)
def _table(mean: float, sigma: float) -> np.ndarray:
    """bf16 bit patterns of mean + sigma * Phi^-1((i + 0.5) / 65536)."""
    nd = statistics.NormalDist()
    z = np.array([nd.inv_cdf((i + 0.5) / 65536.0) for i in range(65536)], dtype=np.float64)
    f = (mean + sigma * z).astype(np.float32)
    b = f.view(np.uint32)
    b = (b + (np.uint32(0x7FFF) + ((b >> np.uint32(16)) & np.uint32(1)))) >> np.uint32(16)
    return b.astype(np.uint16)


_CHUNK = 1 << 22


def _threads() -> int:
    return max(1, min(32, os.cpu_count() or 1))


_CLIB = None


def _clib():
    """ctypes handle of _gen.c compiled with gcc (built on first use), or None."""
    global _CLIB
    if _CLIB is not None:
        return _CLIB or None
    import ctypes
    import subprocess
    import tempfile
    src = os.path.join(_HERE, "_gen.c")
    so = os.path.join(_HERE, "_gen.so")
    try:
        if not os.path.exists(so) or os.path.getmtime(so) < os.path.getmtime(src):
            fd, tmp = tempfile.mkstemp(suffix=".so", dir=_HERE)
            os.close(fd)
            subprocess.run(["gcc", "-O3", "-fopenmp", "-shared", "-fPIC", src, "-o", tmp],
                           check=True, capture_output=True)
            os.replace(tmp, so)
        lib = ctypes.CDLL(so)
        u32, u64, i64, p = ctypes.c_uint32, ctypes.c_uint64, ctypes.c_int64, ctypes.c_void_p
        lib.gen_bf16.argtypes = [u32, u32, p, u64, u64, p]
        lib.gen_bf16_rows.argtypes = [u32, u32, p, p, i64, i64, p]
        _CLIB = lib
    except Exception:  # no compiler: numpy formulation of the same hash
        _CLIB = False
    return _CLIB or None


def normal_bf16(seed: int, name: str, shape, mean: float = 0.0, sigma: float = 1.0,
                rows=None, device: str = "cpu"):
    """Seeded bf16 tensor ~ N(mean, sigma^2) (65536-quantile approximation).

    Returns a numpy uint16 array of bf16 bit patterns for ``device='cpu'``,
    or a torch bfloat16 tensor on ``device`` otherwise.  ``rows`` selects rows
    of a 2-D tensor (the values equal those rows of the full tensor).
    """
    shape = tuple(int(s) for s in shape)
    k1, k2 = _keys(seed, name)
    table = _table(float(mean), float(sigma))
    ncol = shape[-1] if len(shape) > 1 else 1
    if device == "cpu":
        lib = _clib()
        if lib is not None:
            if rows is not None:
                rows = np.ascontiguousarray(np.asarray(rows, dtype=np.int64))
                out = np.empty((len(rows), ncol), dtype=np.uint16)
                lib.gen_bf16_rows(k1, k2, table.ctypes.data, rows.ctypes.data, len(rows), ncol,
                                  out.ctypes.data)
                return out
            out = np.empty(shape, dtype=np.uint16)
            lib.gen_bf16(k1, k2, table.ctypes.data, 0, out.size, out.ctypes.data)
            return out
        if rows is not None:
            rows = np.asarray(rows, dtype=np.int64)
            idx = (rows[:, None] * ncol + np.arange(ncol, dtype=np.int64)[None, :]).astype(np.uint32)
            return table[_hash_np(idx, k1, k2) >> np.uint32(16)]
        n = int(np.prod(shape))
        out = np.empty(n, dtype=np.uint16)

        def work(lo):
            hi = min(n, lo + _CHUNK)
            idx = np.arange(lo, hi, dtype=np.uint32)
            out[lo:hi] = table[_hash_np(idx, k1, k2) >> np.uint32(16)]

        starts = range(0, n, _CHUNK)
        if n > 2 * _CHUNK:
            with ThreadPoolExecutor(_threads()) as ex:
                list(ex.map(work, starts))
        else:
            for s in starts:
                work(s)
        return out.reshape(shape)
    import torch
    tab = torch.from_numpy(table.view(np.int16).copy()).to(device)
    if rows is not None:
        r = torch.as_tensor(np.asarray(rows, dtype=np.int64), device=device)
        idx = r[:, None] * ncol + torch.arange(ncol, device=device, dtype=torch.int64)[None, :]
        return tab[_hash_torch(idx, k1, k2) >> 16].view(torch.bfloat16)
    n = int(np.prod(shape))
    out = torch.empty(n, dtype=torch.int16, device=device)
    step = 1 << 26
    for lo in range(0, n, step):
        hi = min(n, lo + step)
        idx = torch.arange(lo, hi, device=device, dtype=torch.int64)
        out[lo:hi] = tab[_hash_torch(idx, k1, k2) >> 16]
    return out.view(torch.bfloat16).reshape(shape)


def uniform_ints(seed: int, name: str, n: int, lo: int, hi: int) -> np.ndarray:
    """n seeded integers uniform in [lo, hi)."""
    k1, k2 = _keys(seed, name)
    h = _hash_np(np.arange(n, dtype=np.uint32), k1, k2).astype(np.uint64)
    return (lo + ((h * np.uint64(hi - lo)) >> np.uint64(32))).astype(np.int64)


def bf16_bits_to_torch(bits: np.ndarray):
    import torch
    return torch.from_numpy(np.ascontiguousarray(bits).view(np.int16)).view(torch.bfloat16)


# ---------------------------------------------------------------------------
# weights
# ---------------------------------------------------------------------------

def embed_name() -> str:
    return "model.language_model.embed_tokens.weight"


def layer_weight_specs(cfg: ModelConfig, layer: int):
    """(HF name, shape, mean, sigma) for every tensor of one decoder layer.

    Linear weights ~ N(0, 0.02); every RMSNorm gamma ~ 1 + N(0, 0.1).
    """
    p = f"model.language_model.layers.{layer}."
    h, d, nq, nkv, i = cfg.hidden, cfg.head_dim, cfg.n_heads, cfg.n_kv_heads, cfg.intermediate
    return [
        (p + "input_layernorm.weight", (h,), 1.0, 0.1),
        (p + "self_attn.q_proj.weight", (nq * d, h), 0.0, 0.02),
        (p + "self_attn.k_proj.weight", (nkv * d, h), 0.0, 0.02),
        (p + "self_attn.v_proj.weight", (nkv * d, h), 0.0, 0.02),
        (p + "self_attn.q_norm.weight", (d,), 1.0, 0.1),
        (p + "self_attn.k_norm.weight", (d,), 1.0, 0.1),
        (p + "self_attn.o_proj.weight", (h, nq * d), 0.0, 0.02),
        (p + "post_attention_layernorm.weight", (h,), 1.0, 0.1),
        (p + "mlp.gate_proj.weight", (i, h), 0.0, 0.02),
        (p + "mlp.up_proj.weight", (i, h), 0.0, 0.02),
        (p + "mlp.down_proj.weight", (h, i), 0.0, 0.02),
    ]


def gen_weight(seed: int, name: str, shape, mean: float, sigma: float, device="cpu", rows=None):
    return normal_bf16(seed, name, shape, mean, sigma, rows=rows, device=device)


# ---------------------------------------------------------------------------
# inputs
# ---------------------------------------------------------------------------

def _layout(w: Workload):
    """positions [3,S] int32, visual mask [S] uint8, cu_seqlens int32.

    Text run of n tokens at running start c: (c+i, c+i, c+i); the start
    advances by n.  A visual grid (t, h, w) (already merged to LLM tokens) at
    start c: (c+f, c+r, c+col) in (f, r, col) row-major order; the start then
    advances by max(h, w) ("vllm-omni minimax_h3/encoder.py",
    ``_get_vision_position_ids`` / ``_get_rope_index``).  Packed prompts
    restart their 1-D positions at 0.
    """
    pos_t, pos_h, pos_w, mask = [], [], [], []
    if w.n_prompts:
        lens = uniform_ints(w.seed, "prompt_lengths", w.n_prompts, w.prompt_len[0], w.prompt_len[1] + 1)
        cu = np.concatenate([[0], np.cumsum(lens)]).astype(np.int32)
        for n in lens:
            a = np.arange(n)
            pos_t.append(a); pos_h.append(a); pos_w.append(a); mask.append(np.zeros(n, np.uint8))
    else:
        cur = 0
        for run in w.runs:
            if run[0] == "text":
                a = np.arange(run[1]) + cur
                pos_t.append(a); pos_h.append(a); pos_w.append(a)
                mask.append(np.zeros(run[1], np.uint8))
                cur += run[1]
            else:
                _, t, gh, gw = run
                f, r, c = np.meshgrid(np.arange(t), np.arange(gh), np.arange(gw), indexing="ij")
                pos_t.append(f.ravel() + cur); pos_h.append(r.ravel() + cur); pos_w.append(c.ravel() + cur)
                mask.append(np.ones(t * gh * gw, np.uint8))
                cur += max(gh, gw)
        s = sum(len(m) for m in mask)
        cu = np.array([0, s], dtype=np.int32)
    positions = np.stack([np.concatenate(pos_t), np.concatenate(pos_h), np.concatenate(pos_w)]).astype(np.int32)
    return positions, np.concatenate(mask), cu


def gen_inputs(w: Workload) -> dict:
    """All per-encode inputs of a workload as numpy arrays (bf16 as uint16 bits)."""
    positions, mask, cu = _layout(w)
    s = positions.shape[1]
    out = {"positions": np.ascontiguousarray(positions), "visual_mask": mask,
           "cu_seqlens": cu, "seq_len": s}
    cfg = w.model
    if w.embeds_input:
        out["inputs_embeds"] = normal_bf16(w.seed, "inputs_embeds", (s, cfg.hidden), 0.0, 1.0)
        out["input_ids"] = None
    else:
        out["input_ids"] = uniform_ints(w.seed, "input_ids", s, 0, cfg.vocab).astype(np.int32)
    n_vis = int(mask.sum())
    out["n_vis"] = n_vis
    if w.deepstack_levels and n_vis:
        out["deepstack"] = normal_bf16(w.seed, "deepstack", (w.deepstack_levels, n_vis, cfg.hidden),
                                       0.0, w.deepstack_sigma)
    else:
        out["deepstack"] = None
    return out


# ---------------------------------------------------------------------------
# vision tower (the producer of the visual embeddings and DeepStack features)
# ---------------------------------------------------------------------------

@dataclasses.dataclass(frozen=True)
class VisionConfig:
    """Sizes of the Qwen3-VL vision tower ("vllm-omni minimax_h3/encoder.py",
    MiniMaxH3Qwen3VLVisionModel and the classes it builds).  The pages take them from
    the checkpoint's config without printing them; the configurations below are
    synthetic (random weights), sized for the kernels (widths multiples of 256)."""
    depth: int
    hidden: int
    num_heads: int
    intermediate: int
    in_channels: int
    patch_size: int
    temporal_patch_size: int
    spatial_merge_size: int
    out_hidden: int
    num_position_embeddings: int
    deepstack_visual_indexes: tuple
    ln_eps: float = 1e-6
    rope_theta: float = 10000.0

    @property
    def head_dim(self) -> int:
        return self.hidden // self.num_heads

    @property
    def patch_dim(self) -> int:
        return self.in_channels * self.temporal_patch_size * self.patch_size * self.patch_size

    @property
    def merged_hidden(self) -> int:
        return self.hidden * self.spatial_merge_size ** 2


@dataclasses.dataclass(frozen=True)
class VisionWorkload:
    name: str
    model: VisionConfig
    seed: int
    grids: tuple   # (t, h, w) patch grids, images and videos in sequence order


VISION_TINY = VisionConfig(depth=3, hidden=256, num_heads=4, intermediate=512, in_channels=3, patch_size=4,
                           temporal_patch_size=2, spatial_merge_size=2, out_hidden=256,
                           num_position_embeddings=64, deepstack_visual_indexes=(0, 1))
VISION_FULL = VisionConfig(depth=24, hidden=1024, num_heads=16, intermediate=4096, in_channels=3, patch_size=16,
                           temporal_patch_size=2, spatial_merge_size=2, out_hidden=5120,
                           num_position_embeddings=2304, deepstack_visual_indexes=(5, 11, 17))

VISION_WORKLOADS = {
    # 8 x 16 patches -> the 4 x 8 merged grid of the tiny text workload
    0: VisionWorkload("vision-tiny-8x16", VISION_TINY, 2000, grids=((1, 8, 16),)),
    # an image and a two-frame video of different sizes: several attention segments
    1: VisionWorkload("vision-tiny-image-video", VISION_TINY, 2001, grids=((1, 12, 8), (2, 8, 8))),
    # one 48 x 64-patch image -> the 24 x 32 merged grid of the seq-1024 workload
    2: VisionWorkload("vision-image-48x64", VISION_FULL, 2002, grids=((1, 48, 64),)),
}


def vision_workload(i: int) -> VisionWorkload:
    return VISION_WORKLOADS[i]


def vision_weight_specs(cfg: VisionConfig):
    """(HF name, shape, mean, sigma) of every vision-tower tensor.  Linear and
    embedding weights and all biases ~ N(0, 0.02); LayerNorm weights ~ 1 + N(0, 0.1),
    LayerNorm biases ~ N(0, 0.1)."""
    p = "model.visual."
    h, i, mh = cfg.hidden, cfg.intermediate, cfg.merged_hidden
    specs = [
        (p + "patch_embed.proj.weight", (h, cfg.in_channels, cfg.temporal_patch_size, cfg.patch_size,
                                         cfg.patch_size), 0.0, 0.02),
        (p + "patch_embed.proj.bias", (h,), 0.0, 0.02),
        (p + "pos_embed.weight", (cfg.num_position_embeddings, h), 0.0, 0.02),
    ]
    for b in range(cfg.depth):
        q = f"{p}blocks.{b}."
        specs += [
            (q + "norm1.weight", (h,), 1.0, 0.1), (q + "norm1.bias", (h,), 0.0, 0.1),
            (q + "attn.qkv.weight", (3 * h, h), 0.0, 0.02), (q + "attn.qkv.bias", (3 * h,), 0.0, 0.02),
            (q + "attn.proj.weight", (h, h), 0.0, 0.02), (q + "attn.proj.bias", (h,), 0.0, 0.02),
            (q + "norm2.weight", (h,), 1.0, 0.1), (q + "norm2.bias", (h,), 0.0, 0.1),
            (q + "mlp.linear_fc1.weight", (i, h), 0.0, 0.02), (q + "mlp.linear_fc1.bias", (i,), 0.0, 0.02),
            (q + "mlp.linear_fc2.weight", (h, i), 0.0, 0.02), (q + "mlp.linear_fc2.bias", (h,), 0.0, 0.02),
        ]
    mergers = [("merger.", h)] + [(f"deepstack_merger_list.{j}.", mh)
                                  for j in range(len(cfg.deepstack_visual_indexes))]
    for m, norm_width in mergers:
        q = p + m
        specs += [
            (q + "norm.weight", (norm_width,), 1.0, 0.1), (q + "norm.bias", (norm_width,), 0.0, 0.1),
            (q + "linear_fc1.weight", (mh, mh), 0.0, 0.02), (q + "linear_fc1.bias", (mh,), 0.0, 0.02),
            (q + "linear_fc2.weight", (cfg.out_hidden, mh), 0.0, 0.02),
            (q + "linear_fc2.bias", (cfg.out_hidden,), 0.0, 0.02),
        ]
    return specs


def gen_vision_inputs(w: VisionWorkload) -> dict:
    """Pixel patches [n_patches, C*T*P*P] (bf16 bits, N(0, 1), flattened in (C, T, P, P)
    order as the patch embedding views them), the grids, and the patch count."""
    cfg = w.model
    n = sum(t * h * ww for t, h, ww in w.grids)
    return {"pixel_values": normal_bf16(w.seed, "pixel_values", (n, cfg.patch_dim), 0.0, 1.0),
            "grid_thw": np.array(w.grids, dtype=np.int32).reshape(-1, 3), "n_patches": n}
