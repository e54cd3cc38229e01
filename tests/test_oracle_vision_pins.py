"""Pins of the vision-tower oracle (oracle/vision.py) against what the pages and
the mathematics fix, independent of the oracle's own formulas: LayerNorm closed
forms, GELU identities and a numerically integrated normal CDF, Conv3d with
stride = kernel written as a sliding window, bilinear interpolation reproducing
affine tables, the 2-D rotary relative-position property, brute-force
bidirectional attention, and structural identities of the whole tower."""
import math

import numpy as np
import pytest

import oracle as O
import workloads as W

V = O.vision
rng = np.random.default_rng(7)


def test_layer_norm_closed_forms():
    w = rng.normal(1.0, 0.1, 8)
    b = rng.normal(0.0, 0.1, 8)
    # a constant row has no deviation: the output is the bias
    assert np.array_equal(V.layer_norm(np.full((1, 8), 3.25), w, b, 1e-6)[0], b)
    # +-a alternating: mean 0, variance a^2, so each entry is +-a / sqrt(a^2 + eps)
    a = 2.0
    x = np.array([[a, -a] * 4])
    want = np.array([a, -a] * 4) / math.sqrt(a * a + 1e-6) * w + b
    assert np.allclose(V.layer_norm(x, w, b, 1e-6)[0], want, rtol=0, atol=1e-14)
    # invariant to adding a constant; scale invariant when eps is negligible
    y = rng.normal(0, 1, (3, 8))
    assert np.allclose(V.layer_norm(y + 5.0, w, b, 1e-6), V.layer_norm(y, w, b, 1e-6), atol=1e-12)
    assert np.allclose(V.layer_norm(y * 1e3, w, b, 1e-12), V.layer_norm(y, w, b, 1e-12), atol=1e-10)


def test_gelu_forms():
    x = np.linspace(-6, 6, 2001)
    for f in (V.gelu_tanh, V.gelu_erf):
        # x Phi(x) with Phi(x) + Phi(-x) = 1 (tanh odd for the approximate form)
        assert np.allclose(f(x) - f(-x), x, atol=1e-12)
        assert f(np.zeros(1))[0] == 0.0
        assert abs(f(np.array([30.0]))[0] - 30.0) < 1e-9
    # the normal CDF by trapezoidal integration of the density, against gelu_erf / x
    t = np.linspace(-12.0, 3.0, 600001)
    dens = np.exp(-t * t / 2) / math.sqrt(2 * math.pi)
    cdf = np.concatenate([[0.0], np.cumsum((dens[1:] + dens[:-1]) / 2 * np.diff(t))])
    for xv in (-2.5, -1.0, 0.5, 1.0, 2.0, 3.0):
        phi = np.interp(xv, t, cdf)
        assert abs(V.gelu_erf(np.array([xv]))[0] / xv - phi) < 1e-8
    # the tanh form stays within 2e-3 of the exact one; without its cubic term it would not
    err = np.max(np.abs(V.gelu_tanh(x) - V.gelu_erf(x)))
    no_cubic = 0.5 * x * (1 + np.tanh(math.sqrt(2 / math.pi) * x))
    assert err < 2e-3 and np.max(np.abs(no_cubic - V.gelu_erf(x))) > 2e-3


def test_patch_embed_is_a_strided_conv3d():
    C, T, P, hid = 3, 2, 2, 5
    nt, nh, nw = 2, 2, 3   # patches along frames, rows, columns
    vol = rng.normal(0, 1, (C, T * nt, P * nh, P * nw))
    wt = rng.normal(0, 1, (hid, C, T, P, P))
    bias = rng.normal(0, 1, hid)
    # Conv3d with stride = kernel: output (ot, oh, ow) reads the window starting at (ot T, oh P, ow P)
    conv = np.zeros((hid, nt, nh, nw))
    for o in range(hid):
        for ot in range(nt):
            for oh in range(nh):
                for ow in range(nw):
                    win = vol[:, ot * T:(ot + 1) * T, oh * P:(oh + 1) * P, ow * P:(ow + 1) * P]
                    conv[o, ot, oh, ow] = np.sum(win * wt[o]) + bias[o]
    patches = np.stack([vol[:, ot * T:(ot + 1) * T, oh * P:(oh + 1) * P, ow * P:(ow + 1) * P].reshape(-1)
                        for ot in range(nt) for oh in range(nh) for ow in range(nw)])
    got = V.patch_embed(patches, wt, bias)
    assert np.allclose(got, conv.reshape(hid, -1).T, atol=1e-12)


def test_pos_embed_interpolation_is_bilinear():
    G, D = 6, 4
    # an affine table: bilinear interpolation reproduces it exactly at every sample point
    al, be, ga = rng.normal(0, 1, D), rng.normal(0, 1, D), rng.normal(0, 1, D)
    table = np.array([al * r + be * c + ga for r in range(G) for c in range(G)])
    for t, h, w in [(1, 4, 6), (2, 2, 8), (1, 10, 4)]:
        out = V.pos_embed_interpolate(table, [(t, h, w)], 2)
        order = V.merge_order(t, h, w, 2)
        hs = np.linspace(0, G - 1, h, dtype=np.float32).astype(np.float64)
        ws = np.linspace(0, G - 1, w, dtype=np.float32).astype(np.float64)
        want = np.array([al * hs[i] + be * ws[j] + ga for _, i, j in order])
        assert np.allclose(out, want, atol=1e-5), (t, h, w)
    # at the table's own size every sample is a table row; the corners are the table's corners
    tab = rng.normal(0, 1, (G * G, D))
    out = V.pos_embed_interpolate(tab, [(1, G, G)], 2)
    order = V.merge_order(1, G, G, 2)
    assert np.array_equal(out, tab[order[:, 1] * G + order[:, 2]])
    out = V.pos_embed_interpolate(tab, [(1, 2, 2)], 2)   # one block: (0,0) (0,1) (1,0) (1,1)
    assert np.allclose(out[[0, 1, 2, 3]], tab[[0, G - 1, G * G - G, G * G - 1]])


def test_rotary_angles_are_two_dimensional():
    d = 16
    ang = V.rot_pos_angles([(1, 4, 4)], d, 2)
    order = V.merge_order(1, 4, 4, 2)
    inv = 1.0 / (10000.0 ** (np.arange(0, d // 2, 2) / (d // 2)))
    assert np.allclose(ang[:, :d // 4], order[:, 1:2] * inv[None], rtol=1e-6)
    assert np.allclose(ang[:, d // 4:], order[:, 2:3] * inv[None], rtol=1e-6)
    q = rng.normal(0, 1, (len(order), 1, d))
    k = rng.normal(0, 1, (len(order), 1, d))
    rq, rk = V._rope(q, ang), V._rope(k, ang)
    assert np.allclose(np.linalg.norm(rq, axis=-1), np.linalg.norm(q, axis=-1))   # a rotation
    # the score of two patches depends only on their 2-D offset: shift both by (1, 2)
    a = V.rot_pos_angles([(1, 8, 8)], d, 2)
    o8 = V.merge_order(1, 8, 8, 2)
    idx = {(r, c): i for i, (_, r, c) in enumerate(o8)}
    qv, kv = rng.normal(0, 1, (1, 1, d)), rng.normal(0, 1, (1, 1, d))
    for (r1, c1), (r2, c2) in [((0, 0), (2, 3)), ((1, 4), (3, 1))]:
        s1 = np.sum(V._rope(qv, a[[idx[r1, c1]]]) * V._rope(kv, a[[idx[r2, c2]]]))
        s2 = np.sum(V._rope(qv, a[[idx[r1 + 1, c1 + 2]]]) * V._rope(kv, a[[idx[r2 + 1, c2 + 2]]]))
        assert abs(s1 - s2) < 1e-6   # fp32 angles (as the pages build them), float64 rotation


def test_bidirectional_attention_brute_force_and_segments():
    n, heads, d = 7, 2, 4
    hid = heads * d
    x = rng.normal(0, 1, (n, hid))
    wq, bq = rng.normal(0, 0.3, (3 * hid, hid)), rng.normal(0, 0.1, 3 * hid)
    wp, bp = rng.normal(0, 0.3, (hid, hid)), rng.normal(0, 0.1, hid)
    ang = rng.normal(0, 1, (n, d // 2))
    cu = [0, 3, 7]
    got = V.vision_attention(x, wq, bq, wp, bp, ang, cu, heads)
    # loops: each query sees every key of its segment, none outside
    qkv = (x @ wq.T + bq).reshape(n, 3, heads, d)
    q, k, v = V._rope(qkv[:, 0], ang), V._rope(qkv[:, 1], ang), qkv[:, 2]
    o = np.zeros((n, heads, d))
    for s0, s1 in zip(cu[:-1], cu[1:]):
        for i in range(s0, s1):
            for hh in range(heads):
                sc = [float(np.dot(q[i, hh], k[j, hh])) / math.sqrt(d) for j in range(s0, s1)]
                m = max(sc)
                e = [math.exp(s - m) for s in sc]
                o[i, hh] = sum(e[j - s0] / sum(e) * v[j, hh] for j in range(s0, s1))
    assert np.allclose(got, o.reshape(n, hid) @ wp.T + bp, atol=1e-12)
    # packed segments equal separate calls; permuting a segment permutes its outputs
    sep = np.concatenate([V.vision_attention(x[a:b], wq, bq, wp, bp, ang[a:b], [0, b - a], heads)
                          for a, b in zip(cu[:-1], cu[1:])])
    assert np.allclose(got, sep, atol=1e-12)
    perm = np.array([2, 0, 1, 6, 4, 3, 5])
    got_p = V.vision_attention(x[perm], wq, bq, wp, bp, ang[perm], cu, heads)
    assert np.allclose(got_p, got[perm], atol=1e-12)


def _tiny_weights(cfg, seed=3000):
    return {n[len("model.visual."):]: O.bf16_bits_to_float(W.gen_weight(seed, n, s, m, sg), np.float64)
            for n, s, m, sg in W.vision_weight_specs(cfg)}


def test_blocks_with_zero_outputs_are_the_identity():
    cfg = W.VISION_TINY
    ws = _tiny_weights(cfg)
    for k in list(ws):
        if k.endswith(("attn.proj.weight", "attn.proj.bias", "mlp.linear_fc2.weight", "mlp.linear_fc2.bias")):
            ws[k] = np.zeros_like(ws[k])
    grids = [(1, 4, 4)]
    px = rng.normal(0, 1, (16, cfg.patch_dim))
    merged, feats = V.vision_forward(px, grids, cfg, ws, dtype=np.float64)
    x0 = V.patch_embed(px, ws["patch_embed.proj.weight"], ws["patch_embed.proj.bias"]) + \
        V.pos_embed_interpolate(ws["pos_embed.weight"], grids, 2)
    mw = {k[len("merger."):]: v for k, v in ws.items() if k.startswith("merger.")}
    assert np.allclose(merged, V.patch_merger(x0, mw, cfg, False), atol=1e-12)
    d0 = {k[len("deepstack_merger_list.0."):]: v for k, v in ws.items() if k.startswith("deepstack_merger_list.0.")}
    assert np.allclose(feats[0], V.patch_merger(x0, d0, cfg, True), atol=1e-12)
    # a merger with zero linears returns its last bias
    z = dict(mw, **{"linear_fc1.weight": np.zeros_like(mw["linear_fc1.weight"]),
                    "linear_fc2.weight": np.zeros_like(mw["linear_fc2.weight"])})
    assert np.allclose(V.patch_merger(x0, z, cfg, False), np.broadcast_to(mw["linear_fc2.bias"], merged.shape))


def test_vision_float32_tracks_float64():
    w = W.vision_workload(1)
    ws = _tiny_weights(w.model, w.seed)
    px = O.bf16_bits_to_float(W.gen_vision_inputs(w)["pixel_values"], np.float64)
    m64, f64 = V.vision_forward(px, w.grids, w.model, ws, dtype=np.float64)
    m32, f32 = V.vision_forward(px, w.grids, w.model, ws, dtype=np.float32)
    rel = np.linalg.norm(m32 - m64) / np.linalg.norm(m64)
    assert rel < 1e-5 and all(np.linalg.norm(a - b) / np.linalg.norm(b) < 1e-5 for a, b in zip(f32, f64))
