"""Positions and visual rows from token ids (host code, no GPU).

Pinned to a worked example done by hand from the pages' rule (text runs count
up on all three axes; a visual grid counts (frame, row, column) from the
running start, which then advances by max(h, w)/merge), and to the layouts of
the benchmark workloads, which were written from their own description."""
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


def test_hand_worked_image_example(Q):
    # 2 text, an image of grid (1, 4, 8) before a 2x2 merge = 2 x 4 tokens, 2 text
    ids = [5, 6] + [IMG] * 8 + [7, 8]
    pos, mask, kind, ni, nv, delta = Q.h3enc_build_positions(ids, IMG, VID, image_grid_thw=[[1, 4, 8]])
    assert pos[0].tolist() == [0, 1] + [2] * 8 + [6, 7]
    assert pos[1].tolist() == [0, 1] + [2, 2, 2, 2, 3, 3, 3, 3] + [6, 7]
    assert pos[2].tolist() == [0, 1] + [2, 3, 4, 5, 2, 3, 4, 5] + [6, 7]
    assert mask.tolist() == [0, 0] + [1] * 8 + [0, 0]
    assert kind.tolist() == [0, 0] + [1] * 8 + [0, 0]
    assert (ni, nv, delta) == (8, 0, 8 - 12)


def test_hand_worked_video_frames_example(Q):
    # a video of 2 frames (grid (2, 2, 4) -> 2 frames of 1 x 2 tokens), frames separated by a text token
    ids = [1] + [VID] * 2 + [2] + [VID] * 2
    pos, mask, kind, ni, nv, delta = Q.h3enc_build_positions(ids, IMG, VID, video_grid_thw=[[2, 2, 4]])
    # frame 1 at start 1: t 1, h 1, w 1..2; start -> 1 + max(2,4)/2 = 3; text 3; frame 2 at 4
    assert pos.tolist() == [[0, 1, 1, 3, 4, 4], [0, 1, 1, 3, 4, 4], [0, 1, 2, 3, 4, 5]]
    assert kind.tolist() == [0, 2, 2, 0, 2, 2] and (ni, nv) == (0, 4)


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
