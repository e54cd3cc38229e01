"""Whole-encode parity through the C ABI against the CPU oracle.

Bars (from the encoder's contract): per-layer hidden state relative L2 <= 5e-3
when the layer is fed the oracle's bf16-rounded input ("teacher-forced");
final output relative L2 <= 2e-2 and max |diff| <= 0.05 * RMS(out) for free
runs.  Rule (``_harness.parity``): the stated bar, unless the oracle's own
bf16-storage run (rounding exactly where the GPU path stores bf16) is already
past it, in which case the GPU must stay within 1.1x that floor (1.25x for the
max |diff| / RMS).  Bit-exact for determinism and zero DeepStack.  The 50-layer
workloads are in test_gpu_depth.py.
"""
import numpy as np
import pytest

import oracle as O
import workloads as W
from _harness import (GPU_STORAGE, bits_to_f32, cu_or_none, device_inputs, make_encoder, model_of, oracle_embed,
                      oracle_layer_getter, parity, rel_l2, t2f)

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu

import qwen3_vl_text_gb300 as Q  # noqa: E402

LAYER_TOL = 5e-3
FINAL_TOL = 2e-2
MAXABS_TOL = 0.05


def _oracle_inputs(wl, cfg, inp):
    if inp["input_ids"] is not None:
        x0 = oracle_embed(wl, cfg, inp["input_ids"])
    else:
        x0 = bits_to_f32(inp["inputs_embeds"])
    ds = None if inp["deepstack"] is None else bits_to_f32(inp["deepstack"])
    return x0, ds


def _run_gpu(enc, dev, inp, S, capture=None, layer_range=None, embeds=None):
    out = torch.empty(S, enc.model.hidden, dtype=torch.bfloat16, device="cuda")
    if capture is not None:
        Q.h3enc_set_layer_capture(enc.handle, capture)
    nds = 0 if dev["deepstack"] is None else dev["deepstack"].shape[0]
    if embeds is not None or dev["input_ids"] is None:
        lb, le = layer_range if layer_range else (0, enc.model.num_layers)
        Q.h3enc_encode_embeds(enc.handle, embeds if embeds is not None else dev["inputs_embeds"], lb, le,
                              dev["positions"], dev["visual_mask"], dev["deepstack"], nds, inp["n_vis"],
                              cu_or_none(inp), S, out)
    else:
        Q.h3enc_encode(enc.handle, dev["input_ids"], dev["positions"], dev["visual_mask"], dev["deepstack"], nds,
                       inp["n_vis"], cu_or_none(inp), S, out)
    if capture is not None:
        Q.h3enc_set_layer_capture(enc.handle, [])
    assert enc.status() == 0, Q.h3enc_last_error(enc.handle)
    return out


def _check_layers_and_final(wl, cfg, enc, inp, per_layer=True, name=""):
    """Free run vs oracle free run, then every layer teacher-forced."""
    S = inp["seq_len"]
    dev = device_inputs(inp)
    x0, ds = _oracle_inputs(wl, cfg, inp)
    get = oracle_layer_getter(wl, cfg)
    cu = list(inp["cu_seqlens"])
    cap = []
    ws = [get(l) for l in range(cfg.num_layers)]
    ref = O.forward(x0, inp["positions"], cfg, ws.__getitem__, inp["visual_mask"], ds, cu, capture=cap)
    out = t2f(_run_gpu(enc, dev, inp, S))
    ok, msg = parity(f"{name} final", out, ref, lambda: O.forward(
        x0, inp["positions"], cfg, ws.__getitem__, inp["visual_mask"], ds, cu, storage=GPU_STORAGE),
        FINAL_TOL, MAXABS_TOL)
    assert ok, msg
    if not per_layer:
        return
    ins = [x0] + cap[:-1]
    for l in range(cfg.num_layers):
        xin = O.round_to_bf16(ins[l])
        want = O.forward(xin, inp["positions"], cfg, ws.__getitem__, inp["visual_mask"], ds, cu, layers=[l])
        got = t2f(_run_gpu(enc, dev, inp, S, layer_range=(l, l + 1),
                           embeds=torch.from_numpy(xin).to(torch.bfloat16).cuda()))
        ok, msg = parity(f"{name} layer {l} teacher-forced", got, want, lambda: O.forward(
            xin, inp["positions"], cfg, ws.__getitem__, inp["visual_mask"], ds, cu, layers=[l],
            storage=GPU_STORAGE), LAYER_TOL)
        assert ok, msg


@pytest.mark.parametrize("separate_norm", [False, True], ids=["folded_norm", "separate_norm"])
def test_tiny_two_layer_model(separate_norm):
    wl = W.workload(0)
    cfg = wl.model
    enc = make_encoder(wl, cfg, max_tokens=64, separate_norm=separate_norm)
    try:
        _check_layers_and_final(wl, cfg, enc, W.gen_inputs(wl), name=f"tiny ({separate_norm and 'separate' or 'folded'} norm)")
    finally:
        enc.close()


def test_tiny_layer_capture_and_host_entry_match_device_encode():
    wl = W.workload(0)
    cfg = wl.model
    inp = W.gen_inputs(wl)
    S = inp["seq_len"]
    enc = make_encoder(wl, cfg, max_tokens=64)
    try:
        dev = device_inputs(inp)
        caps = [torch.zeros(64, cfg.hidden, dtype=torch.bfloat16, device="cuda") for _ in range(cfg.num_layers)]
        out = _run_gpu(enc, dev, inp, S, capture=caps)
        assert torch.equal(caps[-1][:S], out)
        host_out = torch.empty(S, cfg.hidden, dtype=torch.bfloat16).pin_memory()
        ids = torch.from_numpy(inp["input_ids"])
        pos = torch.from_numpy(inp["positions"])
        mask = torch.from_numpy(inp["visual_mask"])
        ds = W.bf16_bits_to_torch(inp["deepstack"])
        Q.h3enc_encode_host(enc.handle, ids, pos, mask, ds, ds.shape[0], inp["n_vis"], None, S, host_out)
        assert torch.equal(host_out, out.cpu())
        # run twice: deterministic, bit for bit
        assert torch.equal(_run_gpu(enc, dev, inp, S), out)
        # zero DeepStack features equal no DeepStack at all
        z = dict(dev)
        z["deepstack"] = torch.zeros_like(dev["deepstack"])
        nods = dict(dev)
        nods["deepstack"] = None
        assert torch.equal(_run_gpu(enc, z, inp, S), _run_gpu(enc, nods, dict(inp, n_vis=0), S))
        # S = 0 is a no-op
        Q.h3enc_encode(enc.handle, dev["input_ids"], dev["positions"], None, None, 0, 0, None, 0, out)
    finally:
        enc.close()


def test_host_entry_graphs_replay_the_eager_encode():
    """h3enc_encode_host on a stream of its own: the first call of a shape runs eagerly, the
    second captures a CUDA graph, later calls replay it; every output is bit for bit the eager
    one, new input values flow through a replay, a new packing is a new shape, and profiling,
    disabling or reloading weights fall back to (or restart from) eager runs."""
    wl = W.workload(0)
    cfg = wl.model
    inp = W.gen_inputs(wl)
    S = inp["seq_len"]
    enc = make_encoder(wl, cfg, max_tokens=64)
    st = torch.cuda.Stream()
    try:
        ids = torch.from_numpy(inp["input_ids"]).pin_memory()
        pos = torch.from_numpy(inp["positions"]).pin_memory()
        mask = torch.from_numpy(inp["visual_mask"]).pin_memory()
        ds = W.bf16_bits_to_torch(inp["deepstack"]).pin_memory()
        h = enc.handle

        def host(ids_, cu=None):
            out = torch.empty(S, cfg.hidden, dtype=torch.bfloat16).pin_memory()
            n0 = Q.h3enc_launch_count(h)
            Q.h3enc_encode_host(h, ids_, pos, mask, ds, ds.shape[0], inp["n_vis"], cu, S, out, st)
            return out, Q.h3enc_launch_count(h) - n0

        Q.h3enc_set_graphs(h, False)
        ref, n_eager = host(ids)
        ref2, _ = host(ids)
        assert torch.equal(ref, ref2) and n_eager > 0 and Q.h3enc_graph_count(h) == 0
        Q.h3enc_set_graphs(h, True)
        for call in range(4):
            out, n = host(ids)
            assert torch.equal(out, ref), call
            assert n == n_eager, call                      # a replay counts the kernels it runs
            assert Q.h3enc_graph_count(h) == (0 if call == 0 else 1), call
        # other token ids through the same graph: equal to an eager run of them
        ids_b = ((ids.to(torch.int64) * 7 + 3) % cfg.vocab).to(torch.int32).pin_memory()
        out_b, _ = host(ids_b)
        Q.h3enc_set_graphs(h, False)
        want_b, _ = host(ids_b)
        assert torch.equal(out_b, want_b) and not torch.equal(out_b, ref)
        # two packed sequences: another shape, captured on its own second call
        cu = [0, 20, S]
        want_p, _ = host(ids, cu)
        Q.h3enc_set_graphs(h, True)
        for call in range(3):
            out_p, _ = host(ids, cu)
            assert torch.equal(out_p, want_p), call
        assert Q.h3enc_graph_count(h) == 1 and not torch.equal(want_p, ref)
        host(ids)
        host(ids)
        assert Q.h3enc_graph_count(h) == 2
        # profiling on: eager runs, the cached graphs stay
        Q.h3enc_set_profiling(h, True)
        out, _ = host(ids)
        assert torch.equal(out, ref) and Q.h3enc_graph_count(h) == 2
        Q.h3enc_set_profiling(h, False)
        # reloading a weight drops every graph; the handle is finalised again before the next encode
        name, shape, mean, sigma = next(sp for sp in W.layer_weight_specs(cfg, 0) if "o_proj" in sp[0])
        enc.load(name, W.gen_weight(wl.seed, name, shape, mean, sigma, device="cuda"))
        assert Q.h3enc_graph_count(h) == 0
        torch.cuda.synchronize()
        enc.finalize()
        for call in range(3):
            out, _ = host(ids)
            assert torch.equal(out, ref), call
        assert Q.h3enc_graph_count(h) == 1
    finally:
        enc.close()


@pytest.mark.parametrize("separate_norm", [False, True], ids=["folded_norm", "separate_norm"])
def test_one_full_width_layer(separate_norm):
    """One full-width layer at 512 tokens on an N(0,1) hidden input: the free run is the
    teacher-forced run, held to the per-layer bar (no floor) and to the final bars."""
    wl = W.workload(1)
    cfg = wl.model
    inp = W.gen_inputs(wl)
    enc = make_encoder(wl, cfg, max_tokens=inp["seq_len"], separate_norm=separate_norm)
    try:
        dev = device_inputs(inp)
        x0, _ = _oracle_inputs(wl, cfg, inp)
        w = oracle_layer_getter(wl, cfg)(0)
        ref = O.forward(x0, inp["positions"], cfg, lambda _: w)
        out = t2f(_run_gpu(enc, dev, inp, inp["seq_len"]))
        ok, msg = parity(f"one full-width layer ({separate_norm and 'separate' or 'folded'} norm)", out, ref,
                         None, LAYER_TOL, MAXABS_TOL)
        assert ok, msg
    finally:
        enc.close()


@pytest.mark.slow
def test_long_video_layout_one_full_width_layer():
    """The seq-8192 video layout through one full-width layer (DeepStack level 0 after it):
    all 8192 rows, the longest causal rows included; one layer on the oracle's input is the
    teacher-forced case, held to the per-layer bar."""
    wl = W.workload(3)
    cfg = model_of(wl, 1)
    inp = W.gen_inputs(wl)
    enc = make_encoder(wl, cfg, max_tokens=inp["seq_len"])
    try:
        S = inp["seq_len"]
        dev = device_inputs(inp)
        x0, ds = _oracle_inputs(wl, cfg, inp)
        w = oracle_layer_getter(wl, cfg)(0)
        args = (x0, inp["positions"], cfg, lambda _: w, inp["visual_mask"], ds)
        ref = O.forward(*args)
        out = t2f(_run_gpu(enc, dev, inp, S))
        ok, msg = parity("video layout, layer 0, all 8192 rows", out, ref,
                         lambda: O.forward(*args, storage=GPU_STORAGE), LAYER_TOL)
        assert ok, msg
    finally:
        enc.close()


def test_errors_are_reported_before_launch_and_from_the_device():
    wl = W.workload(0)
    cfg = wl.model
    inp = W.gen_inputs(wl)
    S = inp["seq_len"]
    dev = device_inputs(inp)
    enc = Q.Encoder(cfg, max_tokens=64, max_seqs=4, num_deepstack=1)
    try:
        out = torch.empty(S, cfg.hidden, dtype=torch.bfloat16, device="cuda")
        with pytest.raises(Q.H3encError) as e:
            enc.encode(dev["input_ids"], dev["positions"], out)
        assert e.value.code == 4  # NOT_LOADED
        t = torch.zeros(cfg.hidden, dtype=torch.bfloat16, device="cuda")
        assert enc.load("lm_head.weight", t) == 1
        assert enc.load("model.language_model.norm.weight", t) == 1
        assert enc.load("model.language_model.layers.7.input_layernorm.weight", t) == 1  # beyond kept layers
        with pytest.raises(Q.H3encError) as e:
            enc.load("model.language_model.layers.0.input_layernorm.weight",
                     torch.zeros(cfg.hidden + 1, dtype=torch.bfloat16, device="cuda"))
        assert e.value.code == 3
        name = "model.language_model.layers.0.self_attn.q_proj.weight"
        shp = (cfg.n_heads * cfg.head_dim, cfg.hidden)
        fp8 = torch.zeros(shp, dtype=torch.uint8, device="cuda")
        code = Q.lib.h3enc_load_weights(enc.handle, name.encode(), fp8.data_ptr(), 2, (Q._I64 * 2)(*shp), 2, 1)
        assert code == 6 and "online FP8" in Q.h3enc_last_error(enc.handle)
        enc.load(name, torch.zeros(shp, dtype=torch.bfloat16, device="cuda"))
        with pytest.raises(Q.H3encError) as e:
            enc.finalize()
        assert e.value.code == 5
        msg = Q.h3enc_last_error(enc.handle)
        assert "embed_tokens" in msg and "qkv_proj: [k v]" in msg
    finally:
        enc.close()

    enc = make_encoder(wl, cfg, max_tokens=64)
    try:
        out = torch.empty(S, cfg.hidden, dtype=torch.bfloat16, device="cuda")
        with pytest.raises(Q.H3encError) as e:   # S > max_tokens
            Q.h3enc_encode(enc.handle, dev["input_ids"], dev["positions"], None, None, 0, 0, None, 65, out)
        assert e.value.code == 2
        with pytest.raises(Q.H3encError) as e:   # cu_seqlens not ending at S
            Q.h3enc_encode(enc.handle, dev["input_ids"], dev["positions"], None, None, 0, 0, [0, 10, 40], S, out)
        assert e.value.code == 2
        with pytest.raises(Q.H3encError) as e:   # DeepStack without a mask
            Q.h3enc_encode(enc.handle, dev["input_ids"], dev["positions"], None, dev["deepstack"], 1, 32, None, S,
                           out)
        assert e.value.code == 2
        # device-side: visual count mismatch, then an out-of-range token id
        Q.h3enc_encode(enc.handle, dev["input_ids"], dev["positions"], dev["visual_mask"], dev["deepstack"], 1, 31,
                       None, S, out)
        assert enc.status() == 3
        bad = dev["input_ids"].clone()
        bad[3] = cfg.vocab
        Q.h3enc_encode(enc.handle, bad, dev["positions"], None, None, 0, 0, None, S, out)
        assert enc.status() == 10
        assert enc.status() == 0   # read-and-clear
    finally:
        enc.close()


def test_bounded_wait_times_out_into_the_status_and_the_context_survives():
    """Failure detection without a fault: a wait on a flag nothing sets, and one on an
    mbarrier nothing completes, give up after the wait limit and report ST_TIMEOUT;
    a satisfied wait reports nothing; kernels still run afterwards."""
    flag = torch.zeros(1, dtype=torch.int32, device="cuda")
    for use_mbar in (False, True):
        status = torch.zeros(1, dtype=torch.int32, device="cuda")
        Q.h3enc_op_wait_probe(flag, 1, use_mbar, status)
        torch.cuda.synchronize()
        assert int(status.item()) & 1, "the wait did not report its timeout"
    flag.fill_(7)
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    Q.h3enc_op_wait_probe(flag, 7, False, status)
    torch.cuda.synchronize()
    assert int(status.item()) == 0
    # the context is intact: a GEMM still matches its oracle
    A = W.bf16_bits_to_torch(W.normal_bf16(95, "A", (64, 256))).cuda()
    Wt = W.bf16_bits_to_torch(W.normal_bf16(96, "W", (256, 256), 0.0, 0.05)).cuda()
    C = torch.empty(64, 256, dtype=torch.bfloat16, device="cuda")
    Q.h3enc_op_gemm(A, Wt, C, 64, 256, 256, Q.EPI_STORE)
    torch.cuda.synchronize()
    ref = O.linear(t2f(A).astype(np.float64), t2f(Wt).astype(np.float64))
    assert rel_l2(t2f(C), ref) < 5e-3
