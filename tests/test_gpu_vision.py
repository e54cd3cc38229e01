"""The vision tower on the GPU against the oracle (oracle/vision.py), kernel by
kernel through the C ABI, then whole towers, then a tower feeding the text model.

Tolerances as in test_gpu_ops.py (|gpu - ref| <= 2^-7 |ref| + 2^-9 rms(ref) per
element for one rounding to bf16; attention by relative L2 and per row, as the
causal attention test, since P is rounded to bf16); the position-embedding sampler is bit-exact
against the oracle's fp32 arithmetic rounded once; whole towers use the
rule of the text tests (``_harness.parity``: relative L2 <= 2e-2 and max |diff| <=
0.05 RMS, unless the oracle's own bf16-storage run is already past a bar, in which
case within 1.1x / 1.25x of that floor)."""
import dataclasses

import numpy as np
import pytest

import oracle as O
import workloads as W
from _harness import bits_to_f32, make_encoder, oracle_layer_getter, rel_l2, t2f, parity

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu

import qwen3_vl_text_gb300 as Q  # noqa: E402

V = O.vision
EPS = 1e-6


def _bf16(seed, name, shape, mean=0.0, sigma=1.0):
    bits = W.normal_bf16(seed, name, shape, mean, sigma)
    return W.bf16_bits_to_torch(bits).cuda(), bits_to_f32(bits)


def _elementwise_ok(gpu, ref):
    gpu = np.asarray(gpu, np.float64)
    ref = np.asarray(ref, np.float64)
    rms = np.sqrt(np.mean(ref * ref))
    bad = np.abs(gpu - ref) > (2.0 ** -7) * np.abs(ref) + (2.0 ** -9) * rms
    return int(bad.sum()), float(np.max(np.abs(gpu - ref)) / rms)


def _ws():
    return torch.zeros(Q.h3enc_op_gemm_workspace_bytes(), dtype=torch.uint8, device="cuda")


@pytest.mark.parametrize("rows,cols", [(1, 256), (3, 72), (300, 1024), (33, 1536), (7, 2048), (77, 4096), (5, 8192)])
def test_layernorm(rows, cols):
    X, x = _bf16(70, "x", (rows, cols), 0.3, 2.0)
    G, g = _bf16(71, "g", (cols,), 1.0, 0.1)
    B, b = _bf16(72, "b", (cols,), 0.0, 0.1)
    Y = torch.empty_like(X)
    Q.h3enc_op_layernorm(X, G, B, Y, rows, cols, EPS)
    torch.cuda.synchronize()
    bad, worst = _elementwise_ok(t2f(Y), V.layer_norm(x.astype(np.float64), g, b, EPS))
    assert bad == 0, f"{bad} off, worst {worst}"


@pytest.mark.parametrize("grids,G", [(((1, 8, 16),), 8), (((1, 12, 8), (2, 8, 8)), 8), (((1, 48, 64),), 48),
                                     (((1, 2, 2), (3, 4, 6)), 5)])
def test_position_embeddings_bit_exact(grids, G):
    D = 256
    T, t = _bf16(73, "pos", (G * G, D), 0.0, 0.02)
    n = sum(a * b * c for a, b, c in grids)
    out = torch.empty(n, D, dtype=torch.bfloat16, device="cuda")
    Q.h3enc_op_vision_pos_embed(T, G, D, grids, 2, out)
    torch.cuda.synchronize()
    want = O.round_to_bf16(V.pos_embed_interpolate(t.astype(np.float32), grids, 2))
    assert np.array_equal(t2f(out), want)


@pytest.mark.parametrize("d", [64, 128])
def test_rotary_tables(d):
    grids = ((1, 12, 8), (2, 8, 8), (1, 48, 64))
    n = sum(a * b * c for a, b, c in grids)
    c = torch.empty(n, d // 2, device="cuda")
    s = torch.empty_like(c)
    Q.h3enc_op_vision_rope_table(grids, 2, d, 10000.0, c, s)
    torch.cuda.synchronize()
    ang = V.rot_pos_angles(grids, d, 2, 10000.0).astype(np.float64)   # the same fp32 angles
    assert np.max(np.abs(c.cpu().numpy() - np.cos(ang))) < 4e-7
    assert np.max(np.abs(s.cpu().numpy() - np.sin(ang))) < 4e-7


def _shape(case):
    pairs = torch.cuda.get_device_properties(0).multi_processor_count // 2
    if case == "dp":
        return 300, 1024, 512
    return 4 * 256 - 37, (pairs // 4 + 1) * 256, 1536


@pytest.mark.parametrize("case", ["dp", "split"])
@pytest.mark.parametrize("epi", [Q.EPI_STORE, Q.EPI_RESIDUAL, Q.EPI_GELU_TANH, Q.EPI_GELU_ERF])
def test_gemm_bias_epilogues(epi, case):
    M, N, K = _shape(case)
    A, a = _bf16(74, "A", (M, K))
    Wt, w = _bf16(75, "W", (N, K), sigma=0.03)
    Bs, bs = _bf16(76, "bias", (N,), 0.0, 0.5)
    lin = O.linear(a.astype(np.float64), w.astype(np.float64)) + bs
    C = torch.empty(M, N, dtype=torch.bfloat16, device="cuda")
    R = None
    if epi == Q.EPI_RESIDUAL:
        R0, r0 = _bf16(77, "R", (M, N))
        C = R0.clone()
        R = C
        ref = r0 + lin
    elif epi == Q.EPI_GELU_TANH:
        ref = V.gelu_tanh(lin)
    elif epi == Q.EPI_GELU_ERF:
        ref = V.gelu_erf(lin)
    else:
        ref = lin
    Q.h3enc_op_gemm_bias(A, Wt, C, M, N, K, epi, Bs, R=R, workspace=_ws())
    torch.cuda.synchronize()
    bad, worst = _elementwise_ok(t2f(C), ref)
    assert bad == 0, f"{bad} off, worst {worst}"


@pytest.mark.parametrize("grid,split", [((1, 10, 30), False), ((1, 32, 64), True)])
def test_qkv_with_bias_and_2d_rotary(grid, split):
    heads, d = 16, 64
    K = 2048 if split else 512   # split: 96 tiles of 32 k-blocks, a stream-K tail
    M = grid[0] * grid[1] * grid[2]
    N = 3 * heads * d
    A, a = _bf16(78, "A", (M, K))
    Wt, w = _bf16(79, "Wqkv", (N, K), sigma=0.05)
    Bs, bs = _bf16(80, "bqkv", (N,), 0.0, 0.2)
    c = torch.empty(M, d // 2, device="cuda")
    s = torch.empty_like(c)
    Q.h3enc_op_vision_rope_table([grid], 2, d, 10000.0, c, s)
    C = torch.empty(M, N, dtype=torch.bfloat16, device="cuda")
    Q.h3enc_op_gemm_qkv_rope_bias(A, Wt, C, M, K, heads, d, Bs, c, s, workspace=_ws() if split else None)
    torch.cuda.synchronize()
    x = (O.linear(a.astype(np.float64), w.astype(np.float64)) + bs).reshape(M, 3, heads, d)
    ang = V.rot_pos_angles([grid], d, 2)
    ref = np.concatenate([V._rope(x[:, 0], ang).reshape(M, -1), V._rope(x[:, 1], ang).reshape(M, -1),
                          x[:, 2].reshape(M, -1)], axis=1)
    bad, worst = _elementwise_ok(t2f(C), ref)
    assert bad == 0, f"{bad} off, worst {worst}"


def _bidir_case(cu, heads, d, workspace=None):
    S = cu[-1]
    X, x = _bf16(81, "qkv", (S, 3 * heads * d), 0.0, 1.0)
    o = torch.empty(S, heads * d, dtype=torch.bfloat16, device="cuda")
    if workspace is None:
        Q.h3enc_op_attention_bidir(X, o, S, heads, d, cu)
    else:
        Q.h3enc_op_attention_bidir_ws(X, o, S, heads, d, workspace, cu)
    torch.cuda.synchronize()
    return X, x, o


@pytest.mark.parametrize("cu,heads,d,ws", [([0, 96, 160, 224], 4, 64, False), ([0, 1024, 2048], 4, 64, False),
                                           ([0, 200], 4, 64, False),
                                           # more work items than SMs: the last round's pairs run as single
                                           # query tiles; and the same with a pair that has no second tile
                                           # in that range (the split is then refused)
                                           ([0, 3072], 16, 64, False), ([0, 100, 3172], 16, 64, False),
                                           # with a workspace the last round's pairs are cut along the keys
                                           # instead: one segment, two frames, a short segment that limits
                                           # the number of ranges, head_dim 128
                                           ([0, 3072], 16, 64, True), ([0, 1536, 3072], 16, 64, True),
                                           ([0, 384, 4736], 9, 64, True), ([0, 3072], 16, 128, True)])
def test_bidirectional_attention(cu, heads, d, ws):
    S = cu[-1]
    workspace = None
    if ws:
        workspace = torch.zeros(Q.h3enc_op_attention_workspace_bytes(d), dtype=torch.uint8, device="cuda")
    X, x, o = _bidir_case(cu, heads, d, workspace)
    if ws:   # the merge is in range order: the same bits on a second call (counters back at zero)
        o2 = torch.empty_like(o)
        Q.h3enc_op_attention_bidir_ws(X, o2, S, heads, d, workspace, cu)
        torch.cuda.synchronize()
        assert torch.equal(o, o2)
        assert not workspace[-(torch.cuda.get_device_properties(0).multi_processor_count * 32):].any()
    q = x[:, :heads * d].reshape(S, heads, d).astype(np.float64)
    k = x[:, heads * d:2 * heads * d].reshape(S, heads, d).astype(np.float64)
    v = x[:, 2 * heads * d:].reshape(S, heads, d).astype(np.float64)
    ref = np.zeros((S, heads, d))
    for a, b in zip(cu[:-1], cu[1:]):
        for hh in range(heads):
            sc = q[a:b, hh] @ k[a:b, hh].T / np.sqrt(d)
            p = np.exp(sc - sc.max(1, keepdims=True))
            ref[a:b, hh] = (p / p.sum(1, keepdims=True)) @ v[a:b, hh]
    # the bar of the causal attention test: P enters the P.V product rounded to bf16
    got, ref = t2f(o), ref.reshape(S, -1)
    assert rel_l2(got, ref) < 6e-3, f"rel {rel_l2(got, ref):.3g}"
    row_err = np.linalg.norm(got - ref, axis=1) / np.maximum(np.linalg.norm(ref, axis=1), 1e-30)
    assert row_err.max() < 1.5e-2, f"worst row rel {row_err.max():.3g}"


def _tower(w, max_patches=None):
    cfg = w.model
    inp = W.gen_vision_inputs(w)
    enc = Q.VisionEncoder(cfg, max_patches=max_patches or inp["n_patches"])
    for name, shape, mean, sigma in W.vision_weight_specs(cfg):
        enc.load(name, W.gen_weight(w.seed, name, shape, mean, sigma, device="cuda"))
    torch.cuda.synchronize()
    enc.finalize()
    return enc, inp


def _oracle_tower(w, inp, storage=None):
    cfg = w.model
    ws = {n[len("model.visual."):]: bits_to_f32(W.gen_weight(w.seed, n, s, m, sg))
          for n, s, m, sg in W.vision_weight_specs(cfg)}
    return V.vision_forward(bits_to_f32(inp["pixel_values"]), w.grids, cfg, ws, storage=storage)


def _run_tower(enc, w, inp):
    cfg = w.model
    nm = inp["n_patches"] // cfg.spatial_merge_size ** 2
    emb = torch.empty(nm, cfg.out_hidden, dtype=torch.bfloat16, device="cuda")
    ds = torch.empty(len(cfg.deepstack_visual_indexes), nm, cfg.out_hidden, dtype=torch.bfloat16, device="cuda")
    enc.encode(W.bf16_bits_to_torch(inp["pixel_values"]).cuda(), w.grids, emb, ds)
    torch.cuda.synchronize()
    assert enc.status() == 0, Q.h3vis_last_error(enc.handle)
    return emb, ds


@pytest.mark.parametrize("wid", [0, 1])
def test_tiny_tower_against_the_oracle(wid):
    w = W.vision_workload(wid)
    enc, inp = _tower(w, max_patches=256)
    try:
        emb, ds = _run_tower(enc, w, inp)
        again = _run_tower(enc, w, inp)
        assert torch.equal(emb, again[0]) and torch.equal(ds, again[1]), "not deterministic"
    finally:
        enc.close()
    m32, f32 = _oracle_tower(w, inp)
    mbf, fbf = _oracle_tower(w, inp, storage=V.VISION_STORAGE_POINTS)
    ok, msg = parity(f"tower {w.name} merged", t2f(emb), m32, mbf, 2e-2, 0.05)
    assert ok, "merged embeddings: " + msg
    for j in range(len(f32)):
        ok, msg = parity(f"tower {w.name} deepstack {j}", t2f(ds[j]), f32[j], fbf[j], 2e-2, 0.05)
        assert ok, f"deepstack {j}: " + msg


def test_tower_errors():
    w = W.vision_workload(0)
    enc, inp = _tower(w)
    try:
        px = W.bf16_bits_to_torch(inp["pixel_values"]).cuda()
        emb = torch.empty(64, 256, dtype=torch.bfloat16, device="cuda")
        with pytest.raises(Q.H3encError) as e:   # patches do not match the grid
            Q.h3vis_encode(enc.handle, px, inp["n_patches"], [(1, 8, 8)], emb)
        assert e.value.code == 3
        with pytest.raises(Q.H3encError) as e:   # rows not divisible by the merge size
            Q.h3vis_encode(enc.handle, px, inp["n_patches"], [(1, 7, 16)], emb)
        assert e.value.code == 2
        name = "model.visual.blocks.0.attn.qkv.weight"
        with pytest.raises(Q.H3encError) as e:
            enc.load(name, torch.zeros(10, 10, dtype=torch.bfloat16, device="cuda"))
        assert e.value.code == 3
        assert Q.h3vis_load_weights(enc.handle, "model.visual.blocks.9.norm1.weight",
                                    torch.zeros(256, dtype=torch.bfloat16, device="cuda")) == 1
    finally:
        enc.close()


def test_tower_feeds_the_text_model():
    """Tiny tower -> visual embeddings and two DeepStack levels -> the tiny text model's
    multimodal encode, against the oracle chain (vision oracle -> masked scatter ->
    text oracle)."""
    vw = W.vision_workload(0)                 # 8 x 16 patches -> the 4 x 8 visual grid
    tw = W.workload(0)
    cfg = dataclasses.replace(tw.model, vocab=152000)
    tin = W.gen_inputs(tw)
    ids = tin["input_ids"].copy()
    ids[tin["visual_mask"] == 1] = 151655
    venc, vin = _tower(vw)
    tenc = make_encoder(tw, cfg, max_tokens=64)
    try:
        emb, ds = _run_tower(venc, vw, vin)
        S, H = len(ids), cfg.hidden
        out = torch.empty(S, H, dtype=torch.bfloat16, device="cuda")
        Q.h3enc_encode_multimodal(tenc.handle, torch.from_numpy(ids).cuda(), torch.from_numpy(tin["positions"]).cuda(),
                                  torch.from_numpy(tin["visual_mask"]).cuda(), emb, ds, ds.shape[0], emb.shape[0],
                                  None, S, out)
        assert tenc.status() == 0
        got = t2f(out)
    finally:
        venc.close()
        tenc.close()
    m32, f32 = _oracle_tower(vw, vin)
    x0 = bits_to_f32(W.gen_weight(tw.seed, W.embed_name(), (cfg.vocab, H), 0.0, 0.02, rows=ids))
    x0 = O.frontend.masked_scatter_rows(x0, O.frontend.placeholder_rows(ids, 151655), m32)
    get = oracle_layer_getter(tw, cfg)
    ws = [get(l) for l in range(cfg.num_layers)]
    ref = O.forward(x0, tin["positions"], cfg, ws.__getitem__, tin["visual_mask"], np.stack(f32))
    mbf, fbf = _oracle_tower(vw, vin, storage=V.VISION_STORAGE_POINTS)
    xb = O.frontend.masked_scatter_rows(x0, O.frontend.placeholder_rows(ids, 151655), O.round_to_bf16(mbf))
    from _harness import GPU_STORAGE
    refbf = O.forward(xb, tin["positions"], cfg, ws.__getitem__, tin["visual_mask"],
                      O.round_to_bf16(np.stack(fbf)), storage=GPU_STORAGE)
    ok, msg = parity("tower feeding the text model", got, ref, refbf, 2e-2, 0.05)
    assert ok, msg


@pytest.mark.slow
def test_full_size_tower_on_the_48x64_image():
    """The synthetic full-size tower (24 blocks, hidden 1024, 16 heads, DeepStack after
    blocks 5, 11, 17) on one 48 x 64-patch image: every output against the oracle."""
    w = W.vision_workload(2)
    enc, inp = _tower(w)
    try:
        emb, ds = _run_tower(enc, w, inp)
    finally:
        enc.close()
    m32, f32 = _oracle_tower(w, inp)
    mbf, fbf = _oracle_tower(w, inp, storage=V.VISION_STORAGE_POINTS)
    ok, msg = parity(f"tower {w.name} merged", t2f(emb), m32, mbf, 2e-2, 0.05)
    assert ok, "merged embeddings: " + msg
    for j in range(len(f32)):
        ok, msg = parity(f"tower {w.name} deepstack {j}", t2f(ds[j]), f32[j], fbf[j], 2e-2, 0.05)
        assert ok, f"deepstack {j}: " + msg
