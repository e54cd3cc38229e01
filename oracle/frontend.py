"""Multimodal front end of the encoder, restated for the CPU oracle.

TEST INFRASTRUCTURE ONLY (see the package docstring).

Page 1 ("vllm-omni vllm_omni/diffusion/models/minimax_h3/encoder.py"), the
encoder's ``_encode`` and the helpers it calls before the text model runs:

* token types: image placeholder id -> 1, video placeholder id -> 2, else 0;
* ``_get_rope_index`` / ``_get_vision_position_ids``: M-RoPE positions from
  the ids and the visual grids (a video of T frames counts as T one-frame
  grids; each maximal run of one token type is a text run or one grid);
* ``_get_placeholder_mask`` + ``masked_scatter``: the vision-merger rows
  replace the placeholder embeddings, row j going to the j-th placeholder;
* ``_aggregate_deepstack``: per level, image and video features interleaved
  in the order of their tokens.

Plain Python loops over small host arrays; no code is shared with the
product's host helpers.  Pinned by hand-derived fixtures under
``tests/golden/``.  Reading taken where the pages leave it open: a visual run
whose length differs from its grid, or a run with no grid left, is an error
(the page's concatenation would not fit the sequence), raised as ValueError.
"""
from __future__ import annotations

import numpy as np

__all__ = ["token_types", "rope_index", "vision_position_ids", "placeholder_rows",
           "masked_scatter_rows", "aggregate_deepstack"]


def token_types(input_ids, image_token_id: int, video_token_id: int) -> np.ndarray:
    """0 for text, 1 for an image placeholder, 2 for a video placeholder
    (the ``mm_types`` of ``_encode``)."""
    ids = np.asarray(input_ids).reshape(-1)
    out = np.zeros(ids.shape[0], dtype=np.int64)
    for i, v in enumerate(ids.tolist()):
        if v == image_token_id:
            out[i] = 1
        elif v == video_token_id:
            out[i] = 2
    return out


def vision_position_ids(start: int, grid_thw, temporal_merge: int, spatial_merge: int) -> np.ndarray:
    """Positions [3, t*h*w] of one visual grid after the merges: token k of the
    (frame, row, column) raster gets ``(start + frame, start + row, start + column)``
    (``_get_vision_position_ids``)."""
    t = int(grid_thw[0]) // temporal_merge
    h = int(grid_thw[1]) // spatial_merge
    w = int(grid_thw[2]) // spatial_merge
    cols = []
    for f in range(t):
        for r in range(h):
            for c in range(w):
                cols.append((start + f, start + r, start + c))
    return np.array(cols, dtype=np.int64).reshape(-1, 3).T.copy()


def rope_index(input_ids, image_token_id: int, video_token_id: int, image_grid_thw=None,
               video_grid_thw=None, spatial_merge_size: int = 2):
    """``_get_rope_index`` for one sequence without padding.

    Returns (positions int64 [3, S], mrope_delta = max position + 1 - S).
    """
    types = token_types(input_ids, image_token_id, video_token_id)
    S = types.shape[0]
    grids = {1: [list(map(int, g)) for g in (image_grid_thw if image_grid_thw is not None else [])],
             2: []}
    # a video of T frames is consumed as T grids of a single frame
    for g in (video_grid_thw if video_grid_thw is not None else []):
        for _ in range(int(g[0])):
            grids[2].append([1, int(g[1]), int(g[2])])
    taken = {1: 0, 2: 0}

    # maximal runs of one token type, in order
    runs = []
    s = 0
    while s < S:
        e = s
        while e < S and types[e] == types[s]:
            e += 1
        runs.append((int(types[s]), s, e))
        s = e

    pos = np.zeros((3, S), dtype=np.int64)
    current = 0
    for kind, s, e in runs:
        n = e - s
        if kind == 0:
            for i in range(n):
                pos[:, s + i] = current + i
            current += n
            continue
        if taken[kind] >= len(grids[kind]):
            raise ValueError("a visual run has no grid left")
        g = grids[kind][taken[kind]]
        taken[kind] += 1
        ids3 = vision_position_ids(current, g, 1, spatial_merge_size)
        if ids3.shape[1] != n:
            raise ValueError("a visual run's length differs from its grid")
        pos[:, s:e] = ids3
        current += max(g[1], g[2]) // spatial_merge_size
    delta = (int(pos.max()) + 1 - S) if S else 0
    return pos, delta


def placeholder_rows(input_ids, token_id: int) -> np.ndarray:
    """Sequence indices of the placeholder tokens, in order (``_get_placeholder_mask``)."""
    ids = np.asarray(input_ids).reshape(-1)
    return np.array([i for i, v in enumerate(ids.tolist()) if v == token_id], dtype=np.int64)


def masked_scatter_rows(embeds: np.ndarray, rows: np.ndarray, features: np.ndarray) -> np.ndarray:
    """``embeds.masked_scatter(mask, features)`` with a whole-row mask: feature row j
    replaces embedding row ``rows[j]``; the counts must agree (the page raises otherwise)."""
    rows = np.asarray(rows)
    if rows.shape[0] != features.shape[0]:
        raise ValueError("placeholder tokens and feature rows do not match")
    out = np.array(embeds, copy=True)
    for j, r in enumerate(rows.tolist()):
        out[r, :] = features[j, :]
    return out


def aggregate_deepstack(types, image_feats=None, video_feats=None):
    """``_aggregate_deepstack``: returns (visual mask [S] bool, per-level features
    [levels, n_visual, hidden]) where visual position j (j-th visual token in sequence
    order) takes the next image row if it is an image token, else the next video row.
    With only one modality present its features pass through unchanged."""
    types = np.asarray(types).reshape(-1)
    mask = types != 0
    if image_feats is None and video_feats is None:
        return None, None
    if video_feats is None:
        return types == 1, image_feats
    if image_feats is None:
        return types == 2, video_feats
    levels, hidden = image_feats.shape[0], image_feats.shape[2]
    vis_types = [int(t) for t in types.tolist() if t != 0]
    out = np.zeros((levels, len(vis_types), hidden), dtype=image_feats.dtype)
    i_next = v_next = 0
    for j, t in enumerate(vis_types):
        if t == 1:
            out[:, j, :] = image_feats[:, i_next, :]
            i_next += 1
        else:
            out[:, j, :] = video_feats[:, v_next, :]
            v_next += 1
    if i_next != image_feats.shape[1] or v_next != video_feats.shape[1]:
        raise ValueError("visual tokens and DeepStack feature rows do not match")
    return mask, out
