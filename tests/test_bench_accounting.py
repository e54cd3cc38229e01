"""The bench's algorithmic work counts, pinned to the weight shapes the workloads load and to
brute-force counts: one encode's FLOPs are 2 x rows x (every projection weight's elements) per
layer plus 4 x heads x head_dim per unmasked (query, key) pair; one vision encode's FLOPs
likewise from the vision weights, with attention over every (query, key) pair of a frame."""
import importlib.util
import os

import numpy as np

import workloads as W

_spec = importlib.util.spec_from_file_location("bench", os.path.join(os.path.dirname(__file__), "..", "bench.py"))
bench = importlib.util.module_from_spec(_spec)
_spec.loader.exec_module(bench)


def _linear_elements(specs, skip=("norm", "bias", "pos_embed", "embed_tokens")):
    return {n: int(np.prod(s)) for n, s, _, _ in specs if len(s) >= 2 and not any(k in n for k in skip)}


def _causal_pairs(cu):
    n = 0
    for a, b in zip(cu[:-1], cu[1:]):
        for i in range(a, b):
            for j in range(a, b):
                n += j <= i
    return n


def test_encode_flops_from_weight_shapes_and_pair_counts():
    for wid in (0, 2):
        wl = W.workload(wid)
        cfg = wl.model
        per_layer = sum(_linear_elements(W.layer_weight_specs(cfg, 0)).values())
        if wid == 2:
            assert per_layer == 487_587_840     # the full-width layer's projection parameters
        for cu in ([0, 48], [0, 1, 17, 40, 48], [0, 1024]):
            S = cu[-1]
            want = cfg.num_layers * (2.0 * S * per_layer + 4.0 * cfg.n_heads * cfg.head_dim * _causal_pairs(cu))
            assert bench.encode_flops(cfg, np.array(cu)) == want
    cfg = W.workload(2).model
    assert abs(bench.encode_flops(cfg, np.array([0, 1024])) / 1e12 - 50.79) < 0.01


def test_vision_flops_from_weight_shapes():
    cfg = W.VISION_TINY
    specs = W.vision_weight_specs(cfg)
    lin = _linear_elements(specs)
    m2 = cfg.spatial_merge_size ** 2
    for grids in ([(1, 4, 4)], [(1, 4, 6), (2, 2, 4)]):
        n = sum(t * h * w for t, h, w in grids)
        total = 0.0
        for name, elems in lin.items():
            rows = n // m2 if "merger" in name else n      # mergers act on the merged rows
            total += 2.0 * rows * elems
        # bidirectional attention inside each frame: every (query, key) pair of the frame
        frame_pairs = sum(t * (h * w) ** 2 for t, h, w in grids)
        total += cfg.depth * 4.0 * cfg.num_heads * (cfg.hidden // cfg.num_heads) * frame_pairs
        assert abs(bench.vision_flops(cfg, grids) - total) <= 1e-9 * total, grids
