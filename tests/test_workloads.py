"""The seeded input generator: determinism, cross-implementation identity and
the workload layouts (token runs, M-RoPE positions, visual masks, packing)."""
import numpy as np
import pytest

import workloads as W


def test_c_numpy_and_torch_formulations_agree():
    torch = pytest.importorskip("torch")
    shape = (513, 77)
    c = W.normal_bf16(5, "blk.w", shape, 0.0, 0.02)
    saved = W._CLIB
    try:
        W._CLIB = False
        n = W.normal_bf16(5, "blk.w", shape, 0.0, 0.02)
    finally:
        W._CLIB = saved
    k1, k2 = W._keys(5, "blk.w")
    idx = torch.arange(shape[0] * shape[1], dtype=torch.int64)
    tab = torch.from_numpy(W._table(0.0, 0.02).view(np.int16).copy())
    t = tab[W._hash_torch(idx, k1, k2) >> 16].numpy().view(np.uint16).reshape(shape)
    assert np.array_equal(c, n) and np.array_equal(c, t)


def test_rows_equal_full_tensor_rows_and_distribution():
    full = W.normal_bf16(9, "emb", (300, 64), 0.0, 0.02)
    rows = [299, 0, 17, 17]
    assert np.array_equal(W.normal_bf16(9, "emb", (300, 64), 0.0, 0.02, rows=rows), full[rows])
    f = (full.astype(np.uint32) << 16).view(np.float32)
    assert abs(f.mean()) < 1e-3 and abs(f.std() - 0.02) < 1e-3
    g = (W.normal_bf16(9, "g", (4096,), 1.0, 0.1).astype(np.uint32) << 16).view(np.float32)
    assert abs(g.mean() - 1.0) < 0.01 and abs(g.std() - 0.1) < 0.01
    assert not np.array_equal(full, W.normal_bf16(9, "emb2", (300, 64), 0.0, 0.02))


def test_tiny_layout_matches_its_description():
    inp = W.gen_inputs(W.workload(0))
    pos, mask = inp["positions"], inp["visual_mask"]
    assert pos.shape == (3, 48) and inp["n_vis"] == 32
    assert pos[:, :8].tolist() == [list(range(8))] * 3
    assert mask.tolist() == [0] * 8 + [1] * 32 + [0] * 8
    vis = pos[:, 8:40]
    assert (vis[0] == 8).all()
    assert vis[1].tolist() == [8 + r for r in range(4) for _ in range(8)]
    assert vis[2].tolist() == [8 + c for _ in range(4) for c in range(8)]
    assert pos[:, 40:].tolist() == [list(range(16, 24))] * 3
    assert inp["deepstack"].shape == (1, 32, 256)
    assert inp["input_ids"].min() >= 0 and inp["input_ids"].max() < 1024


def test_image_and_video_layouts():
    inp = W.gen_inputs(W.workload(2))
    pos = inp["positions"]
    assert inp["seq_len"] == 1024 and inp["n_vis"] == 768
    assert pos[:, 128].tolist() == [128, 128, 128] and pos[:, 128 + 767].tolist() == [128, 151, 159]
    assert pos[:, 896].tolist() == [160, 160, 160] and pos[:, -1].tolist() == [287] * 3
    inp = W.gen_inputs(W.workload(3))
    pos = inp["positions"]
    assert inp["seq_len"] == 8192 and inp["n_vis"] == 6144
    frame = 24 * 32
    assert pos[0, 1024 + 3 * frame] == 1027 and pos[:, 1024 + 6143].tolist() == [1031, 1047, 1055]
    assert pos[:, 7168].tolist() == [1056] * 3


def test_varlen_layout():
    inp = W.gen_inputs(W.workload(4))
    cu = inp["cu_seqlens"]
    lens = np.diff(cu)
    assert len(lens) == 16 and lens.min() >= 77 and lens.max() <= 512
    assert inp["seq_len"] == cu[-1] and inp["n_vis"] == 0 and inp["deepstack"] is None
    pos = inp["positions"]
    for a, b in zip(cu[:-1], cu[1:]):
        assert pos[:, a:b].tolist() == [list(range(b - a))] * 3


def test_weight_specs_cover_one_layer():
    cfg = W.workload(2).model
    specs = W.layer_weight_specs(cfg, 7)
    total = sum(int(np.prod(s)) for _, s, _, _ in specs)
    assert total == cfg.params_per_layer() == 487_587_840 + 2 * 5120 + 2 * 128
