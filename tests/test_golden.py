"""Hand-derived fixtures under tests/golden/ (each file names the passage it is
derived from) against the oracle, and where the product has a host-side
counterpart, against it too.  No GPU."""
from pathlib import Path

import numpy as np
import pytest

import oracle as O

GOLDEN = Path(__file__).parent / "golden"
IMG, VID = 151655, 151656
AXIS = {"T": 0, "H": 1, "W": 2}


def read_cases(name):
    """`case:` starts a case; `key: values` lines fill it; `#` lines are comments."""
    cases = []
    for line in (GOLDEN / name).read_text().splitlines():
        line = line.strip()
        if not line or line.startswith("#"):
            continue
        key, _, val = line.partition(":")
        if key == "case":
            cases.append({"case": val.strip()})
        else:
            cases[-1][key] = val.split()
    assert cases, name
    return cases


def ints(v):
    return [int(x) for x in v]


def grids(v):
    return np.array(ints(v), dtype=np.int64).reshape(-1, 3) if v else None


def ids_of(letters):
    return np.array([IMG if c == "I" else VID if c == "V" else 1000 + i for i, c in enumerate(letters)],
                    dtype=np.int64)


@pytest.mark.parametrize("case", read_cases("mrope_axis_tables.txt"), ids=lambda c: c["case"])
def test_mrope_axis_table(case):
    half = int(case["half_dim"][0])
    want = [AXIS[c] for c in case["axes"][0]]
    assert len(want) == half
    assert O.mrope_axis_of_pair(half, ints(case["section"])).tolist() == want


POSITION_CASES = read_cases("positions.txt")


@pytest.mark.parametrize("case", POSITION_CASES, ids=lambda c: c["case"])
def test_positions_oracle(case):
    ids = ids_of(case["ids"])
    pos, delta = O.frontend.rope_index(ids, IMG, VID, grids(case["image_grid_thw"]), grids(case["video_grid_thw"]))
    assert pos.tolist() == [ints(case["t"]), ints(case["h"]), ints(case["w"])]
    assert delta == int(case["delta"][0])
    types = O.frontend.token_types(ids, IMG, VID)
    assert int((types == 1).sum()) == int(case["n_image"][0]) and int((types == 2).sum()) == int(case["n_video"][0])


@pytest.fixture(scope="module")
def Q():
    import __graft_entry__
    __graft_entry__._build_module().build()
    import qwen3_vl_text_gb300
    return qwen3_vl_text_gb300


@pytest.mark.parametrize("case", POSITION_CASES, ids=lambda c: c["case"])
def test_positions_host_helper(Q, case):
    ids = ids_of(case["ids"])
    pos, mask, kind, ni, nv, delta = Q.h3enc_build_positions(ids, IMG, VID, grids(case["image_grid_thw"]),
                                                             grids(case["video_grid_thw"]))
    assert pos.tolist() == [ints(case["t"]), ints(case["h"]), ints(case["w"])]
    assert (ni, nv, delta) == (int(case["n_image"][0]), int(case["n_video"][0]), int(case["delta"][0]))
    assert kind.tolist() == [1 if c == "I" else 2 if c == "V" else 0 for c in case["ids"]]
    assert mask.tolist() == [int(c != "T") for c in case["ids"]]


@pytest.mark.parametrize("case", read_cases("deepstack_order.txt"), ids=lambda c: c["case"])
def test_deepstack_order(case):
    kinds = np.array([{"T": 0, "I": 1, "V": 2}[c] for c in case["kinds"]])
    ni, nv = int((kinds == 1).sum()), int((kinds == 2).sum())
    # row k of the image features holds 1000 + k, row k of the video features 2000 + k
    img = (1000.0 + np.arange(ni, dtype=np.float64))[None, :, None].repeat(2, axis=0)
    vid = (2000.0 + np.arange(nv, dtype=np.float64))[None, :, None].repeat(2, axis=0)
    mask, out = O.frontend.aggregate_deepstack(kinds, img, vid)
    want = [1000 + int(s[1:]) if s[0] == "i" else 2000 + int(s[1:]) for s in case["order"]]
    assert mask.tolist() == (kinds != 0).tolist()
    assert out[0, :, 0].tolist() == want and out[1, :, 0].tolist() == want


@pytest.mark.parametrize("case", read_cases("vision_merge_order.txt"), ids=lambda c: c["case"])
def test_vision_merge_order(case):
    t, h, w = ints(case["grid"])
    want = [[int(v) for v in p.split(",")] for p in case["patches"]]
    assert O.vision.merge_order(t, h, w, int(case["merge"][0])).tolist() == want
