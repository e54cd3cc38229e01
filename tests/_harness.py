"""Shared helpers of the GPU parity tests: build an encoder from the seeded
generator (weights drawn on the device), the matching CPU oracle run (same
weights drawn on the host), and the comparison metrics."""
from __future__ import annotations

import dataclasses

import numpy as np

import oracle as O
import workloads as W


def rel_l2(a, b) -> float:
    a = np.asarray(a, dtype=np.float64)
    b = np.asarray(b, dtype=np.float64)
    return float(np.linalg.norm(a - b) / max(np.linalg.norm(b), 1e-30))


def max_abs_over_rms(a, b) -> float:
    a = np.asarray(a, dtype=np.float64)
    b = np.asarray(b, dtype=np.float64)
    return float(np.max(np.abs(a - b)) / max(np.sqrt(np.mean(b * b)), 1e-30))


# Tensors the GPU path hands between kernels in bf16 (its rounding points).
GPU_STORAGE = frozenset({"y", "v", "qk", "attn", "act", "h"})


# A bar counts as out of reach of bf16 storage when the oracle's own bf16-storage run (rounding
# exactly where the GPU path stores bf16) already sits above FLOOR_REACH x the bar.
FLOOR_REACH = 0.8
FLOOR_REL_SLACK = 1.1      # then the GPU must stay within 1.1x that floor (relative L2) ...
FLOOR_MAX_SLACK = 1.25     # ... and 1.25x its max |diff| / RMS


def _log(rec: dict):
    """Append one parity record as a JSON line to $H3ENC_PARITY_LOG (when set)."""
    import json
    import os
    path = os.environ.get("H3ENC_PARITY_LOG")
    if path:
        with open(path, "a") as f:
            f.write(json.dumps(rec) + "\n")


def parity(what, gpu, ref32, floor, rel_bar, maxabs_bar=None):
    """Tolerance rule of the parity tests.  ``ref32`` is the fp32 oracle.  The GPU passes when
    its relative L2 (and max |diff| / RMS, when ``maxabs_bar`` is given) against ref32 is
    within the stated bar.  Only where a bar is out of reach of bf16 storage does the rule
    fall back on the floor: ``floor`` (an array, or a callable computing it on demand) is the
    same oracle rounding to bf16 at GPU_STORAGE; if its own distance from ref32 exceeds
    FLOOR_REACH x the bar, the GPU must stay within FLOOR_REL_SLACK (FLOOR_MAX_SLACK) x that
    distance.  Every comparison is logged (see ``_log``).  Returns (ok, message)."""
    r = rel_l2(gpu, ref32)
    m = max_abs_over_rms(gpu, ref32) if maxabs_bar is not None else None
    rel_ok = r <= rel_bar
    max_ok = m is None or m <= maxabs_bar
    fl = mf = None
    clause = "bar"
    if not (rel_ok and max_ok) and floor is not None:
        fb = floor() if callable(floor) else floor
        fl = rel_l2(fb, ref32)
        mf = max_abs_over_rms(fb, ref32)
        if not rel_ok and fl > FLOOR_REACH * rel_bar:
            rel_ok = r <= FLOOR_REL_SLACK * fl
            clause = "floor"
        if not max_ok and mf > FLOOR_REACH * maxabs_bar:
            max_ok = m <= FLOOR_MAX_SLACK * mf
            clause = "floor"
    ok = rel_ok and max_ok
    msg = f"{what}: rel {r:.3g} (bar {rel_bar:g}"
    msg += f", bf16 floor {fl:.3g})" if fl is not None else ")"
    if m is not None:
        msg += f"; max/rms {m:.3g} (bar {maxabs_bar:g}" + (f", floor {mf:.3g})" if mf is not None else ")")
    msg += f" [{clause}]"
    _log({"what": what, "rel": r, "max_rms": m, "rel_bar": rel_bar, "max_bar": maxabs_bar, "floor_rel": fl,
          "floor_max_rms": mf, "clause": clause, "ok": ok})
    return ok, msg


def bits_to_f32(bits: np.ndarray) -> np.ndarray:
    """bf16 bit patterns -> float32 (multithreaded via torch; exact)."""
    import torch
    return W.bf16_bits_to_torch(np.ascontiguousarray(bits)).float().numpy()


def t2f(t) -> np.ndarray:
    """torch bf16 tensor (any device) -> float32 numpy."""
    return t.detach().float().cpu().numpy()


def f2bf16_torch(x: np.ndarray, device="cuda"):
    import torch
    return torch.from_numpy(np.ascontiguousarray(x, dtype=np.float32)).to(torch.bfloat16).to(device)


def model_of(wl: W.Workload, num_layers=None):
    m = wl.model
    return m if num_layers is None else dataclasses.replace(m, num_layers=num_layers)


def oracle_layer_getter(wl: W.Workload, cfg):
    def get(l):
        lw = O.LayerWeights()
        for name, shape, mean, sigma in W.layer_weight_specs(cfg, l):
            lw[name.split(".")[-2]] = bits_to_f32(W.gen_weight(wl.seed, name, shape, mean, sigma))
        return lw
    return get


def oracle_embed(wl: W.Workload, cfg, ids: np.ndarray) -> np.ndarray:
    return bits_to_f32(W.gen_weight(wl.seed, W.embed_name(), (cfg.vocab, cfg.hidden), 0.0, 0.02, rows=ids))


def make_encoder(wl: W.Workload, cfg, max_tokens: int, max_seqs: int = 64, fp8: bool = False,
                 separate_norm: bool = False):
    import torch
    from qwen3_vl_text_gb300 import Encoder
    enc = Encoder(cfg, max_tokens=max_tokens, max_seqs=max_seqs, num_deepstack=max(3, wl.deepstack_levels), fp8=fp8,
                  separate_norm=separate_norm)
    for l in range(cfg.num_layers):
        for name, shape, mean, sigma in W.layer_weight_specs(cfg, l):
            enc.load(name, W.gen_weight(wl.seed, name, shape, mean, sigma, device="cuda"))
    if cfg.vocab:
        enc.load(W.embed_name(), W.gen_weight(wl.seed, W.embed_name(), (cfg.vocab, cfg.hidden), 0.0, 0.02,
                                              device="cuda"))
    torch.cuda.synchronize()
    enc.finalize()
    return enc


def device_inputs(inp: dict):
    """Workload inputs as device tensors (ids, positions, mask, deepstack, embeds)."""
    import torch
    dev = {}
    dev["positions"] = torch.from_numpy(inp["positions"]).cuda()
    dev["input_ids"] = None if inp["input_ids"] is None else torch.from_numpy(inp["input_ids"]).cuda()
    dev["visual_mask"] = torch.from_numpy(inp["visual_mask"]).cuda() if inp["n_vis"] else None
    dev["deepstack"] = None if inp["deepstack"] is None else W.bf16_bits_to_torch(inp["deepstack"]).cuda()
    dev["inputs_embeds"] = (None if inp.get("inputs_embeds") is None
                            else W.bf16_bits_to_torch(inp["inputs_embeds"]).cuda())
    return dev


def cu_or_none(inp: dict):
    cu = inp["cu_seqlens"]
    return None if len(cu) == 2 else [int(x) for x in cu]
