"""Pins of the CPU oracle against values fixed by the pages and by mathematics.

Each test checks one oracle function against something other than itself: a
closed form, a special case that reduces to a textbook result, an invariant,
or brute force on tiny inputs.  Together they are chosen so that a dropped
term, a wrong sign or index, or a transposed operand in the oracle fails at
least one of them.
"""
import math

import numpy as np
import pytest

import oracle as O
import workloads as W

F64 = np.float64


def _rng(seed=0):
    return np.random.default_rng(seed)


# ---------------------------------------------------------------- bf16 storage

def test_bf16_widening_known_patterns():
    bits = np.array([0x3F80, 0xC000, 0x0000, 0x4049, 0x3C00], dtype=np.uint16)
    got = O.bf16_bits_to_float(bits, F64)
    assert got.tolist() == [1.0, -2.0, 0.0, 3.140625, 2.0 ** -7]


def test_bf16_rounding_ties_to_even_and_torch():
    one = 1.0
    x = np.array([one, one + 2 ** -8, one + 3 * 2 ** -8, one + 2 ** -8 + 2 ** -20, -2.0 - 2 ** -7],
                 dtype=np.float32)
    got = O.round_to_bf16(x)
    # 1+2^-8 is a tie between 1 and 1+2^-7 -> even (1); 1+3*2^-8 ties -> 1+2^-6 (even mantissa);
    # the bf16 spacing at 2 is 2^-6, so -2-2^-7 is a tie between -2 and -2-2^-6 -> even (-2)
    assert got.tolist() == [1.0, 1.0, 1.0 + 2 ** -6, 1.0 + 2 ** -7, -2.0]
    torch = pytest.importorskip("torch")
    r = _rng(1).standard_normal(4096).astype(np.float32) * 37.0
    ref = torch.from_numpy(r).to(torch.bfloat16).float().numpy()
    assert np.array_equal(O.round_to_bf16(r), ref)


# ---------------------------------------------------------------- linear

def test_linear_is_x_times_w_transposed():
    # one-hot weight W[a, b] = 1 maps input component b to output component a
    x = _rng(2).standard_normal((3, 5))
    w = np.zeros((7, 5))
    w[6, 1] = 1.0
    y = O.linear(x, w)
    assert y.shape == (3, 7)
    assert np.array_equal(y[:, 6], x[:, 1])
    assert np.count_nonzero(y[:, :6]) == 0


# ---------------------------------------------------------------- RMSNorm

def test_rms_norm_constant_vector():
    n, c, eps = 64, 0.37, 1e-6
    w = 1.0 + 0.1 * _rng(3).standard_normal(n)
    y = O.rms_norm(np.full((1, n), c), w, eps)
    np.testing.assert_allclose(y[0], w * c / math.sqrt(c * c + eps), rtol=1e-14)


def test_rms_norm_one_hot():
    n, a, i, eps = 128, 5.0, 17, 1e-6
    x = np.zeros((1, n))
    x[0, i] = a
    w = np.arange(1, n + 1, dtype=F64)
    y = O.rms_norm(x, w, eps)
    assert y[0, i] == pytest.approx(w[i] * a / math.sqrt(a * a / n + eps), rel=1e-14)
    assert np.count_nonzero(np.delete(y[0], i)) == 0


def test_rms_norm_scale_invariance_and_eps_effect():
    x = _rng(4).standard_normal((4, 256))
    w = np.ones(256)
    np.testing.assert_allclose(O.rms_norm(1000.0 * x, w, 1e-6), O.rms_norm(x, w, 1e-6), rtol=1e-6)
    # eps dominates tiny inputs: y ~ x / sqrt(eps)
    np.testing.assert_allclose(O.rms_norm(1e-9 * x, w, 1e-6), 1e-9 * x / 1e-3, rtol=1e-5)


# ---------------------------------------------------------------- RoPE / M-RoPE

def test_inv_freq_closed_values():
    inv = O.rope_inv_freq(64, 1e6)
    assert inv.dtype == np.float32
    assert inv[0] == 1.0
    assert inv[16] == np.float32(1e-3)         # theta^(-1/2) = 1e-3
    inv = O.rope_inv_freq(128, 5e6)
    assert inv[32] == np.float32(1.0 / math.sqrt(5e6))
    assert inv[63] == np.float32(5e6 ** (-126 / 128))


def test_mrope_axis_tables():
    ax = O.mrope_axis_of_pair(64, (24, 20, 20))
    h = set(range(1, 59, 3))
    w = set(range(2, 60, 3))
    assert set(np.nonzero(ax == 1)[0]) == h and len(h) == 20 and max(h) == 58
    assert set(np.nonzero(ax == 2)[0]) == w and len(w) == 20 and max(w) == 59
    t = set(range(0, 58, 3)) | {60, 61, 62, 63}
    assert set(np.nonzero(ax == 0)[0]) == t and len(t) == 24
    ax = O.mrope_axis_of_pair(32, (12, 10, 10))
    assert np.nonzero(ax == 1)[0].tolist() == [1, 4, 7, 10, 13, 16, 19, 22, 25, 28]
    assert np.nonzero(ax == 2)[0].tolist() == [2, 5, 8, 11, 14, 17, 20, 23, 26, 29]
    assert np.nonzero(ax == 0)[0].tolist() == [0, 3, 6, 9, 12, 15, 18, 21, 24, 27, 30, 31]


def test_mrope_reduces_to_1d_rope():
    p = np.array([0, 1, 7, 300, 4095, 8191])
    pos = np.stack([p, p, p])
    d, theta = 128, 5e6
    cos, sin = O.rope_cos_sin(pos, d, theta, (24, 20, 20), F64)
    for s, ps in enumerate(p):
        for j in range(d // 2):
            ang = float(np.float32(ps) * np.float32(1.0 / theta ** (2 * j / d)))
            assert cos[s, j] == pytest.approx(math.cos(ang), abs=1e-12)
            assert sin[s, j + d // 2] == pytest.approx(math.sin(ang), abs=1e-12)


def test_mrope_axis_independence():
    d = 64
    base = np.array([[5], [5], [5]])
    moved = np.array([[5], [9], [5]])        # only the H position changes
    c0, s0 = O.rope_cos_sin(base, d, 1e6, (12, 10, 10), F64)
    c1, s1 = O.rope_cos_sin(moved, d, 1e6, (12, 10, 10), F64)
    changed = np.nonzero(np.abs(c0[0, :32] - c1[0, :32]) + np.abs(s0[0, :32] - s1[0, :32]) > 0)[0]
    assert changed.tolist() == list(range(1, 30, 3))


def test_rope_is_complex_rotation_by_angle():
    rng = _rng(5)
    s, heads, d = 6, 3, 16
    x = rng.standard_normal((s, heads, d))
    pos = np.stack([np.arange(s) * 3] * 3)
    cos, sin = O.rope_cos_sin(pos, d, 1e4, (3, 3, 2), F64)
    y = O.apply_rope(x, cos, sin)
    half = d // 2
    for si in range(s):
        for j in range(half):
            ang = math.atan2(sin[si, j], cos[si, j])
            z = complex(x[si, 0, j], x[si, 0, j + half]) * complex(math.cos(ang), math.sin(ang))
            assert y[si, 0, j] == pytest.approx(z.real, abs=1e-12)
            assert y[si, 0, j + half] == pytest.approx(z.imag, abs=1e-12)


def test_rope_norm_identity_and_relative_position():
    rng = _rng(6)
    d = 64
    q = rng.standard_normal((1, 1, d))
    k = rng.standard_normal((1, 1, d))
    def rope_at(x, p):
        pos = np.full((3, 1), p)
        c, s = O.rope_cos_sin(pos, d, 1e4, (12, 10, 10), F64)
        return O.apply_rope(x, c, s)[0, 0]
    assert np.array_equal(rope_at(q, 0), q[0, 0])
    for p in (1, 5, 123):
        assert np.linalg.norm(rope_at(q, p)) == pytest.approx(np.linalg.norm(q), rel=1e-12)
    dots = [rope_at(q, m) @ rope_at(k, m - 4) for m in (4, 10, 37, 200)]
    np.testing.assert_allclose(dots, dots[0], rtol=1e-5)


# ---------------------------------------------------------------- attention

def _brute_attention(q, k, v, cu):
    s, nq, d = q.shape
    group = nq // k.shape[1]
    out = np.zeros((s, nq, d))
    for a, b in zip(cu[:-1], cu[1:]):
        for h in range(nq):
            g = h // group
            for i in range(a, b):
                sc = [sum(q[i, h, c] * k[j, g, c] for c in range(d)) / math.sqrt(d) for j in range(a, i + 1)]
                m = max(sc)
                e = [math.exp(t - m) for t in sc]
                z = sum(e)
                for c in range(d):
                    out[i, h, c] = sum(e[j - a] * v[j, g, c] for j in range(a, i + 1)) / z
    return out.reshape(s, nq * d)


def test_attention_brute_force_tiny():
    rng = _rng(7)
    s, nq, nkv, d = 11, 4, 2, 8
    q, k, v = (rng.standard_normal((s, n, d)) for n in (nq, nkv, nkv))
    for cu in ([0, s], [0, 4, 5, s]):
        np.testing.assert_allclose(O.causal_gqa_attention(q, k, v, cu), _brute_attention(q, k, v, cu),
                                   rtol=1e-12, atol=1e-12)


def test_attention_chunking_is_invisible():
    rng = _rng(8)
    s, nq, nkv, d = 37, 4, 1, 8
    q, k, v = (rng.standard_normal((s, n, d)) for n in (nq, nkv, nkv))
    np.testing.assert_allclose(O.causal_gqa_attention(q, k, v, q_chunk=5),
                               O.causal_gqa_attention(q, k, v, q_chunk=512), rtol=1e-11, atol=1e-14)


def test_attention_single_token_returns_v():
    rng = _rng(9)
    q, k, v = rng.standard_normal((1, 4, 8)), rng.standard_normal((1, 2, 8)), rng.standard_normal((1, 2, 8))
    out = O.causal_gqa_attention(q, k, v).reshape(1, 4, 8)
    for h in range(4):
        assert np.allclose(out[0, h], v[0, h // 2], rtol=0, atol=0)


def test_attention_zero_query_is_running_mean():
    rng = _rng(10)
    s = 9
    v = rng.standard_normal((s, 1, 4))
    out = O.causal_gqa_attention(np.zeros((s, 2, 4)), rng.standard_normal((s, 1, 4)), v).reshape(s, 2, 4)
    for i in range(s):
        np.testing.assert_allclose(out[i, 1], v[:i + 1, 0].mean(axis=0), rtol=1e-12)


def test_gqa_equals_mha_with_repeated_kv():
    rng = _rng(11)
    s, nq, nkv, d = 13, 8, 2, 4
    q, k, v = (rng.standard_normal((s, n, d)) for n in (nq, nkv, nkv))
    k_rep, v_rep = np.repeat(k, nq // nkv, axis=1), np.repeat(v, nq // nkv, axis=1)
    np.testing.assert_allclose(O.causal_gqa_attention(q, k, v), O.causal_gqa_attention(q, k_rep, v_rep),
                               rtol=1e-14)


def test_varlen_equals_separate_sequences():
    rng = _rng(12)
    lens = [5, 1, 9]
    cu = np.concatenate([[0], np.cumsum(lens)])
    s = cu[-1]
    q, k, v = (rng.standard_normal((s, n, 4)) for n in (2, 1, 1))
    packed = O.causal_gqa_attention(q, k, v, cu)
    for a, b in zip(cu[:-1], cu[1:]):
        np.testing.assert_allclose(packed[a:b], O.causal_gqa_attention(q[a:b], k[a:b], v[a:b]), rtol=1e-14)


# ---------------------------------------------------------------- SwiGLU / DeepStack

def test_silu_closed_forms():
    z = np.array([0.0, 40.0, -40.0, 1.0])
    y = O.silu(z)
    assert y[0] == 0.0
    assert y[1] == pytest.approx(40.0, rel=1e-15)
    assert abs(y[2]) < 1e-15
    assert y[3] == pytest.approx(1.0 / (1.0 + math.exp(-1.0)), rel=1e-15)


def test_deepstack_row_order_and_zero():
    x = np.zeros((6, 2))
    mask = np.array([0, 1, 0, 1, 1, 0], dtype=np.uint8)
    feats = np.array([[1.0, 2.0], [3.0, 4.0], [5.0, 6.0]])
    y = O.deepstack_add(x, mask, feats)
    assert y.tolist() == [[0, 0], [1, 2], [0, 0], [3, 4], [5, 6], [0, 0]]
    z = _rng(13).standard_normal((6, 2))
    assert np.array_equal(O.deepstack_add(z, mask, np.zeros((3, 2))), z)


# ---------------------------------------------------------------- layer / model

def _tiny_weights(cfg, seed=1000, dtype=F64):
    def get(l):
        return O.layer_weights_from_bits(
            {n: W.gen_weight(seed, n, shp, m, sg) for n, shp, m, sg in W.layer_weight_specs(cfg, l)}, dtype)
    return get


def _tiny_case(dtype=F64):
    wl = W.workload(0)
    cfg = wl.model
    inp = W.gen_inputs(wl)
    emb = O.bf16_bits_to_float(W.gen_weight(wl.seed, W.embed_name(), (cfg.vocab, cfg.hidden), 0.0, 0.02,
                                            rows=inp["input_ids"]), dtype)
    ds = O.bf16_bits_to_float(inp["deepstack"], dtype)
    return wl, cfg, inp, emb, ds


def test_layer_with_zero_output_projections_is_identity():
    cfg = W.workload(0).model
    get = _tiny_weights(cfg)
    w = get(0)
    w["o_proj"] = np.zeros_like(w["o_proj"])
    w["down_proj"] = np.zeros_like(w["down_proj"])
    x = _rng(14).standard_normal((10, cfg.hidden))
    pos = np.stack([np.arange(10)] * 3)
    c, s = O.rope_cos_sin(pos, cfg.head_dim, cfg.rope_theta, cfg.mrope_section, F64)
    assert np.array_equal(O.decoder_layer(x, w, c, s, cfg), x)


def test_single_token_layer_reduces_to_value_path():
    """S=1: softmax over one key is 1, so attention returns v, RoPE and q/k
    never matter.  With zero MLP gate the SwiGLU branch vanishes (silu(0)=0)."""
    cfg = W.workload(0).model
    w = _tiny_weights(cfg)(1)
    w["gate_proj"] = np.zeros_like(w["gate_proj"])
    x = _rng(15).standard_normal((1, cfg.hidden))
    c, s = O.rope_cos_sin(np.array([[3], [4], [5]]), cfg.head_dim, cfg.rope_theta, cfg.mrope_section, F64)
    y = O.decoder_layer(x, w, c, s, cfg)
    # hand-expanded: normalise, take v of each kv head, give it to its q heads, project with o_proj
    xs = x[0]
    xn = xs / math.sqrt(float(np.mean(xs * xs)) + cfg.rms_eps) * w["input_layernorm"]
    v = np.array([sum(w["v_proj"][r, c2] * xn[c2] for c2 in range(cfg.hidden)) for r in range(w["v_proj"].shape[0])])
    heads = [v[(h // 2) * cfg.head_dim:(h // 2 + 1) * cfg.head_dim] for h in range(cfg.n_heads)]
    a = np.concatenate(heads)
    o = np.array([sum(w["o_proj"][r, c2] * a[c2] for c2 in range(a.size)) for r in range(cfg.hidden)])
    np.testing.assert_allclose(y[0], xs + o, rtol=1e-10, atol=1e-12)


def test_causal_prefix_invariance_whole_model():
    wl, cfg, inp, emb, ds = _tiny_case()
    get = _tiny_weights(cfg, wl.seed)
    full = O.forward(emb, inp["positions"], cfg, get, inp["visual_mask"], ds, dtype=F64)
    p = 20
    n_vis_p = int(inp["visual_mask"][:p].sum())
    part = O.forward(emb[:p], inp["positions"][:, :p], cfg, get, inp["visual_mask"][:p],
                     ds[:, :n_vis_p], dtype=F64)
    np.testing.assert_allclose(part, full[:p], rtol=1e-12, atol=1e-12)


def test_packed_model_equals_separate_runs():
    wl, cfg, inp, emb, ds = _tiny_case()
    get = _tiny_weights(cfg, wl.seed)
    cu = [0, 17, 30, 48]
    pos = np.concatenate([np.stack([np.arange(b - a)] * 3) for a, b in zip(cu[:-1], cu[1:])], axis=1)
    packed = O.forward(emb, pos, cfg, get, cu_seqlens=cu, dtype=F64)
    for a, b in zip(cu[:-1], cu[1:]):
        sep = O.forward(emb[a:b], pos[:, a:b], cfg, get, dtype=F64)
        np.testing.assert_allclose(packed[a:b], sep, rtol=1e-11, atol=1e-11)


def test_zero_deepstack_equals_none_and_levels_apply_after_layers():
    wl, cfg, inp, emb, ds = _tiny_case()
    get = _tiny_weights(cfg, wl.seed)
    plain = O.forward(emb, inp["positions"], cfg, get, dtype=F64)
    zero = O.forward(emb, inp["positions"], cfg, get, inp["visual_mask"], np.zeros_like(ds), dtype=F64)
    assert np.array_equal(plain, zero)
    # a level added after the last layer changes exactly the visual rows by exactly the features
    cap = []
    O.forward(emb, inp["positions"], cfg, get, inp["visual_mask"], ds, capture=cap, layers=[0], dtype=F64)
    nods = O.forward(emb, inp["positions"], cfg, get, layers=[0], dtype=F64)
    m = inp["visual_mask"].astype(bool)
    np.testing.assert_allclose(cap[0][m] - nods[m], ds[0], rtol=1e-9, atol=1e-12)
    assert np.array_equal(cap[0][~m], nods[~m])


def test_float32_oracle_tracks_float64():
    wl, cfg, inp, emb, ds = _tiny_case()
    r64 = O.forward(emb, inp["positions"], cfg, _tiny_weights(cfg, wl.seed, F64), inp["visual_mask"], ds,
                    dtype=F64)
    wl, cfg, inp, emb32, ds32 = _tiny_case(np.float32)
    r32 = O.forward(emb32, inp["positions"], cfg, _tiny_weights(cfg, wl.seed, np.float32), inp["visual_mask"],
                    ds32, dtype=np.float32)
    rel = np.linalg.norm(r32 - r64) / np.linalg.norm(r64)
    assert rel < 1e-5


def test_bf16_storage_variant_rounds_only_at_hand_over_points():
    """With every storage point the layer output is bf16-representable; with
    none it is the exact forward; zero output projections keep the identity
    for a bf16-representable input."""
    wl, cfg, inp, emb, ds = _tiny_case(np.float32)
    get = _tiny_weights(cfg, wl.seed, np.float32)
    exact = O.forward(emb, inp["positions"], cfg, get, dtype=np.float32)
    assert np.array_equal(O.forward(emb, inp["positions"], cfg, get, dtype=np.float32, storage=set()), exact)
    allp = O.forward(emb, inp["positions"], cfg, get, dtype=np.float32, storage=set(O.STORAGE_POINTS))
    assert np.array_equal(O.round_to_bf16(allp), allp)
    rel = np.linalg.norm(allp - exact) / np.linalg.norm(exact)
    assert 1e-4 < rel < 3e-2
    w = get(0)
    w["o_proj"] = np.zeros_like(w["o_proj"])
    w["down_proj"] = np.zeros_like(w["down_proj"])
    x = O.round_to_bf16(_rng(16).standard_normal((6, cfg.hidden)).astype(np.float32))
    c, s = O.rope_cos_sin(np.stack([np.arange(6)] * 3), cfg.head_dim, cfg.rope_theta, cfg.mrope_section)
    assert np.array_equal(O.decoder_layer(x, w, c, s, cfg, storage=set(O.STORAGE_POINTS)), x)


# ---------------------------------------------------------------------------
# online-FP8 linears (oracle.fp8)
# ---------------------------------------------------------------------------

def test_e4m3_round_matches_torch_converter():
    """Against torch's independent float8_e4m3fn conversion (round to nearest even) on
    random values across the whole finite range, subnormals and exact ties."""
    torch = pytest.importorskip("torch")
    rng = _rng(40)
    x = np.concatenate([
        rng.standard_normal(20000) * 100.0,
        rng.standard_normal(20000) * 2.0 ** -7,                  # subnormal range
        (np.arange(-4000, 4000) + 0.5) * 2.0 ** -9,              # ties between subnormals
        np.ldexp(1.0 + (np.arange(16) + 0.5) / 8.0, 3),          # ties between normals in [8, 16)
    ]).astype(np.float32)
    x = np.clip(x, -448.0, 448.0)
    ref = torch.from_numpy(x).to(torch.float8_e4m3fn).to(torch.float64).numpy()
    assert np.array_equal(O.fp8.e4m3_round(x), ref)


def test_e4m3_grid_facts():
    r = O.fp8.e4m3_round
    assert r(np.array([448.0]))[0] == 448.0                   # largest finite
    assert r(np.array([600.0, -1e6]))[0] == 448.0 and r(np.array([-1e6]))[0] == -448.0   # saturating
    assert r(np.array([2.0 ** -9]))[0] == 2.0 ** -9           # smallest subnormal
    assert r(np.array([2.0 ** -10]))[0] == 0.0                # tie with 0 -> even (0)
    assert r(np.array([3 * 2.0 ** -10]))[0] == 2.0 ** -8      # tie 1.5 ulp -> even (2 ulp)
    assert r(np.array([1.0 + 2.0 ** -4]))[0] == 1.0           # tie -> even mantissa 000
    assert r(np.array([1.0 + 3 * 2.0 ** -4]))[0] == 1.25      # tie -> even mantissa 010
    assert r(np.array([15.5]))[0] == 16.0                     # rounds up into the next binade
    # the positive finite values from the bit layout: 7 subnormals m/8 * 2^-6, normals (1 + m/8) * 2^(E-7)
    # for E = 1..15 except E = 15, m = 7 (the NaN code of the fn variant): 126 values
    grid = [m / 8 * 2.0 ** -6 for m in range(1, 8)]
    grid += [(1 + m / 8) * 2.0 ** (E - 7) for E in range(1, 16) for m in range(8) if not (E == 15 and m == 7)]
    grid = np.array(sorted(grid))
    assert len(grid) == 126 and grid[-1] == 448.0
    assert np.array_equal(r(grid), grid) and np.array_equal(r(-grid), -grid)
    mid = (grid[:-1] + grid[1:]) / 2                          # every midpoint goes to a neighbour
    got = r(mid)
    assert np.all((got == grid[:-1]) | (got == grid[1:]))
    assert np.all(np.diff(r(np.linspace(-500, 500, 100001))) >= 0)   # monotone


def test_quantize_rows_scales_and_error_bound():
    rng = _rng(41)
    x = O.round_to_bf16(rng.standard_normal((5, 300)).astype(np.float32) * np.array([1e-3, 1, 7, 300, 0])[:, None])
    q, s = O.fp8.quantize_rows(x)
    assert s[4] == 1.0 and np.all(q[4] == 0)                  # zero row
    for i in range(4):
        amax = np.max(np.abs(x[i]))
        assert s[i] == np.float32(amax) / np.float32(448.0)
        assert np.max(np.abs(q[i])) == 448.0                  # the largest element lands on +-448
        deq = q[i] * s[i]
        big = np.abs(x[i]) >= 2.0 ** -6 * s[i]                # normal range of e4m3 after scaling
        assert np.all(np.abs(deq - x[i])[big] <= 2.0 ** -4 * np.abs(x[i])[big] * (1 + 1e-6))
        assert np.all(np.abs(deq - x[i])[~big] <= 2.0 ** -10 * s[i] * (1 + 1e-6))


def test_fp8_linear_is_exact_on_the_grid_and_scales_back():
    """Rows already on the e4m3 grid with amax 448 have scale 1 and quantise to
    themselves: the FP8 linear is then the plain product.  Scaling a row of x or
    of w by a power of two scales the output row / column by it (scales act per row)."""
    rng = _rng(42)
    g = O.fp8.e4m3_round(rng.uniform(-448, 448, (6, 64)))
    g[:, 0] = 448.0
    h = O.fp8.e4m3_round(rng.uniform(-448, 448, (5, 64)))
    h[:, 3] = -448.0
    assert np.array_equal(O.fp8.fp8_linear(g, h), O.linear(g.astype(np.float64), h.astype(np.float64)))
    x = O.round_to_bf16(rng.standard_normal((4, 64)).astype(np.float32))
    w = O.round_to_bf16(rng.standard_normal((3, 64)).astype(np.float32))
    base = O.fp8.fp8_linear(x, w)
    x2 = x.copy(); x2[1] *= 8.0
    w2 = w.copy(); w2[2] *= 0.25
    out = O.fp8.fp8_linear(x2, w2)
    expect = base.copy(); expect[1] *= 8.0; expect[:, 2] *= 0.25
    assert np.array_equal(out, expect)


def test_fp8_layer_tracks_the_bf16_layer():
    """The FP8 tiny model stays within the quantisation error of the exact one
    (e4m3 keeps 3 fraction bits: a few % relative per projection, compounding over
    the 8 projections of the two layers) and does differ from it."""
    wl, cfg, inp, emb, ds = _tiny_case(np.float32)
    get = _tiny_weights(cfg, wl.seed, np.float32)
    exact = O.forward(emb, inp["positions"], cfg, get, inp["visual_mask"], ds, dtype=np.float32)
    q8 = O.forward(emb, inp["positions"], cfg, get, inp["visual_mask"], ds, dtype=np.float32, fp8=True)
    rel = np.linalg.norm(q8 - exact) / np.linalg.norm(exact)
    assert 1e-3 < rel < 1e-1
    # one projection alone: the relative error of a K = 256 product is a few %
    rng = _rng(43)
    x = O.round_to_bf16(rng.standard_normal((32, 256)).astype(np.float32))
    w = O.round_to_bf16(rng.standard_normal((48, 256)).astype(np.float32) * 0.02)
    ref = O.linear(x.astype(np.float64), w.astype(np.float64))
    e1 = np.linalg.norm(O.fp8.fp8_linear(x, w) - ref) / np.linalg.norm(ref)
    assert 5e-3 < e1 < 4e-2


# ---------------------------------------------------------------- whole layer, hand-expanded

def _hand_layer(x, w, pos, cfg, *, qk_norm="before_rope", swap_gate_up=False):
    """One decoder layer written out element by element in float64 Python loops,
    from page 1 (``MiniMaxH3Qwen3VLTextDecoderLayer.forward``,
    ``MiniMaxH3Qwen3VLTextAttention.forward``, ``MiniMaxH3Qwen3VLTextMLP.forward``,
    ``_apply_interleaved_mrope``, ``_rotate_half``): RMSNorm, q/k/v projections,
    per-head q/k RMSNorm with their own weights, then rotate-half RoPE whose
    frequency j is driven by position axis T, H or W, causal GQA softmax
    attention, o_proj and residual; RMSNorm, ``down(silu(gate) * up)`` and
    residual.  ``qk_norm`` ("before_rope", "after_rope", "none") and
    ``swap_gate_up`` plant the mistakes this expansion must tell apart."""
    s, hid = len(x), cfg.hidden
    d, nq, nkv, half = cfg.head_dim, cfg.n_heads, cfg.n_kv_heads, cfg.head_dim // 2
    eps = cfg.rms_eps

    def norm(vec, g):
        r = math.sqrt(sum(t * t for t in vec) / len(vec) + eps)
        return [vec[i] / r * g[i] for i in range(len(vec))]

    def matvec(m, vec):
        return [sum(m[r][c] * vec[c] for c in range(len(vec))) for r in range(len(m))]

    sec = cfg.mrope_section
    axis = []
    for j in range(half):
        if j % 3 == 1 and j < 3 * sec[1]:
            axis.append(1)
        elif j % 3 == 2 and j < 3 * sec[2]:
            axis.append(2)
        else:
            axis.append(0)
    inv = [float(np.float32(1.0 / cfg.rope_theta ** (2.0 * j / d))) for j in range(half)]

    def rope(vec, t):
        out = [0.0] * d
        for j in range(half):
            ang = float(np.float32(np.float32(pos[axis[j]][t]) * np.float32(inv[j])))
            c, sn = math.cos(ang), math.sin(ang)
            out[j] = vec[j] * c - vec[j + half] * sn
            out[j + half] = vec[j + half] * c + vec[j] * sn
        return out

    def head_prep(vec, g, t):
        if qk_norm == "before_rope":
            return rope(norm(vec, g), t)
        if qk_norm == "after_rope":
            return norm(rope(vec, t), g)
        return rope(vec, t)

    wl = {k: v.tolist() for k, v in w.items()}
    qs, ks, vs = [], [], []
    for t in range(s):
        y = norm(x[t], wl["input_layernorm"])
        q, k, v = matvec(wl["q_proj"], y), matvec(wl["k_proj"], y), matvec(wl["v_proj"], y)
        qs.append([head_prep(q[h * d:(h + 1) * d], wl["q_norm"], t) for h in range(nq)])
        ks.append([head_prep(k[g * d:(g + 1) * d], wl["k_norm"], t) for g in range(nkv)])
        vs.append([v[g * d:(g + 1) * d] for g in range(nkv)])
    outs = []
    for t in range(s):
        attn = []
        for h in range(nq):
            g = h // (nq // nkv)
            sc = [sum(qs[t][h][c] * ks[u][g][c] for c in range(d)) / math.sqrt(d) for u in range(t + 1)]
            m = max(sc)
            e = [math.exp(z - m) for z in sc]
            tot = sum(e)
            attn += [sum(e[u] / tot * vs[u][g][c] for u in range(t + 1)) for c in range(d)]
        h1 = [x[t][i] + o for i, o in enumerate(matvec(wl["o_proj"], attn))]
        y2 = norm(h1, wl["post_attention_layernorm"])
        gate, up = matvec(wl["gate_proj"], y2), matvec(wl["up_proj"], y2)
        if swap_gate_up:
            gate, up = up, gate
        act = [gi / (1.0 + math.exp(-gi)) * ui for gi, ui in zip(gate, up)]
        outs.append([h1[i] + dn for i, dn in enumerate(matvec(wl["down_proj"], act))])
    return np.array(outs)


def test_three_token_layer_against_hand_expansion():
    """A 3-token layer with non-zero gate and up weights, strongly non-uniform
    q_norm / k_norm weights and positions that differ on every axis, against the
    loop expansion above.  The same expansion with gate and up swapped, with the
    q/k RMSNorm dropped, or with it applied after the rotation is far from the
    oracle, so each of those mistakes in the oracle would fail here."""
    from types import SimpleNamespace
    cfg = SimpleNamespace(hidden=16, n_heads=4, n_kv_heads=2, head_dim=8, intermediate=12, rms_eps=1e-6,
                          rope_theta=100.0, mrope_section=[2, 1, 1])
    r = _rng(40)
    nq_d, kv_d = cfg.n_heads * cfg.head_dim, cfg.n_kv_heads * cfg.head_dim
    w = O.LayerWeights(
        q_proj=r.standard_normal((nq_d, cfg.hidden)) * 0.4, k_proj=r.standard_normal((kv_d, cfg.hidden)) * 0.4,
        v_proj=r.standard_normal((kv_d, cfg.hidden)) * 0.4, o_proj=r.standard_normal((cfg.hidden, nq_d)) * 0.3,
        gate_proj=r.standard_normal((cfg.intermediate, cfg.hidden)) * 0.5,
        up_proj=r.standard_normal((cfg.intermediate, cfg.hidden)) * 0.5,
        down_proj=r.standard_normal((cfg.hidden, cfg.intermediate)) * 0.3,
        q_norm=1.0 + 0.6 * r.standard_normal(cfg.head_dim), k_norm=1.0 + 0.6 * r.standard_normal(cfg.head_dim),
        input_layernorm=1.0 + 0.2 * r.standard_normal(cfg.hidden),
        post_attention_layernorm=1.0 + 0.2 * r.standard_normal(cfg.hidden))
    x = r.standard_normal((3, cfg.hidden))
    pos = np.array([[0, 3, 5], [0, 1, 7], [0, 4, 2]])       # (t, h, w) per token, all axes distinct
    c, s = O.rope_cos_sin(pos, cfg.head_dim, cfg.rope_theta, cfg.mrope_section, F64)
    got = O.decoder_layer(x, w, c, s, cfg)
    want = _hand_layer(x, w, pos, cfg)
    np.testing.assert_allclose(got, want, rtol=1e-9, atol=1e-10)
    scale = np.linalg.norm(want - x)     # size of what the layer adds
    for kw in ({"swap_gate_up": True}, {"qk_norm": "none"}, {"qk_norm": "after_rope"}):
        wrong = _hand_layer(x, w, pos, cfg, **kw)
        assert np.linalg.norm(wrong - want) > 1e-3 * scale, kw
