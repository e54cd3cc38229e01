"""Positions and visual rows from token ids (host code, no GPU).

The host helper against the oracle's restatement of the pages' rule on seeded
random layouts (element by element, integers bit-exact), on the empty sequence
and on the malformed layouts both reject, and against the layouts of the
benchmark workloads, which were written from their own description.  The
hand-derived examples live in tests/golden/positions.txt (test_golden.py)."""
import numpy as np
import pytest

import workloads as W


@pytest.fixture(scope="module")
def Q():
    import __graft_entry__
    __graft_entry__._build_module().build()
    import qwen3_vl_text_gb300
    return qwen3_vl_text_gb300


IMG, VID = 151655, 151656


def test_benchmark_image_layout_from_ids(Q):
    wl = W.workload(2)
    inp = W.gen_inputs(wl)
    ids = inp["input_ids"].copy()
    ids[inp["visual_mask"] == 1] = IMG
    ids[inp["visual_mask"] == 0] %= 100000          # no accidental placeholder ids in the text
    pos, mask, kind, ni, nv, _ = Q.h3enc_build_positions(ids, IMG, VID, image_grid_thw=[[1, 48, 64]])
    assert np.array_equal(pos, inp["positions"]) and np.array_equal(mask, inp["visual_mask"]) and ni == 768


def test_run_length_must_match_grid(Q):
    with pytest.raises(Q.H3encError) as e:
        Q.h3enc_build_positions([1] + [IMG] * 7 + [2], IMG, VID, image_grid_thw=[[1, 4, 4]])
    assert e.value.code == 3
    with pytest.raises(Q.H3encError):
        Q.h3enc_build_positions([1] + [IMG] * 4 + [2] + [IMG] * 4, IMG, VID, image_grid_thw=[[1, 4, 4]])
    with pytest.raises(Q.H3encError):
        Q.h3enc_build_positions([IMG] * 4, IMG, VID, image_grid_thw=[[1, 3, 4]])   # 3 not divisible by 2


def _random_layout(rng, merge):
    """Seeded sequence of text runs, images and multi-frame videos (frames split by text)."""
    ids, img, vid = [], [], []
    text = lambda n: ids.extend(int(x) for x in rng.integers(0, 100000, n))
    text(int(rng.integers(0, 4)))
    for _ in range(int(rng.integers(0, 5))):
        gh, gw = merge * int(rng.integers(1, 5)), merge * int(rng.integers(1, 5))
        n = (gh // merge) * (gw // merge)
        if rng.random() < 0.5:
            img.append([1, gh, gw])
            ids.extend([IMG] * n)
        else:
            t = int(rng.integers(1, 4))
            vid.append([t, gh, gw])
            for f in range(t):
                ids.extend([VID] * n)
                if f + 1 < t:
                    text(int(rng.integers(1, 3)))
        text(int(rng.integers(1, 4)))
    return np.array(ids, dtype=np.int64), (img or None), (vid or None)


@pytest.mark.parametrize("merge", [1, 2])
def test_positions_match_the_oracle_on_random_layouts(Q, merge):
    import oracle as O
    rng = np.random.default_rng(4242 + merge)
    for _ in range(300):
        ids, img, vid = _random_layout(rng, merge)
        pos, mask, kind, ni, nv, delta = Q.h3enc_build_positions(ids, IMG, VID, img, vid, spatial_merge_size=merge)
        opos, odelta = O.frontend.rope_index(ids, IMG, VID, img, vid, spatial_merge_size=merge)
        types = O.frontend.token_types(ids, IMG, VID)
        assert np.array_equal(pos, opos) and delta == odelta
        assert np.array_equal(kind, types) and np.array_equal(mask, types != 0)
        assert (ni, nv) == (int((types == 1).sum()), int((types == 2).sum()))


def test_empty_sequence_and_mismatches_agree_with_the_oracle(Q):
    import oracle as O
    pos, mask, kind, ni, nv, delta = Q.h3enc_build_positions(np.zeros(0, dtype=np.int64), IMG, VID)
    opos, odelta = O.frontend.rope_index(np.zeros(0, dtype=np.int64), IMG, VID)
    assert pos.shape == opos.shape == (3, 0) and delta == odelta == 0 and (ni, nv) == (0, 0)
    bad = [
        ([1] + [IMG] * 3 + [2], [[1, 4, 4]], None),            # 3 tokens for a 2 x 2 grid
        ([1] + [VID] * 8, None, [[2, 4, 4]]),                   # two frames with no text between
        ([1] + [IMG] * 4 + [2] + [IMG] * 4, [[1, 4, 4]], None), # a second image with no grid
    ]
    for ids, img, vid in bad:
        with pytest.raises(ValueError):
            O.frontend.rope_index(ids, IMG, VID, img, vid)
        with pytest.raises(Q.H3encError) as e:
            Q.h3enc_build_positions(ids, IMG, VID, img, vid)
        assert e.value.code == 3
