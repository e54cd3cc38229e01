"""Online-FP8 linears on the GPU against the oracle's FP8 restatement
(``oracle.fp8``): per-row e4m3 quantisation bit for bit (bytes and scales), the
RMSNorm that emits quantised output, the e4m3 projection GEMM with every
epilogue and the stream-K tail shapes, and the whole FP8 encode."""
import numpy as np
import pytest

import oracle as O
import workloads as W
from _harness import GPU_STORAGE, bits_to_f32, make_encoder, oracle_embed, oracle_layer_getter, rel_l2, t2f, parity

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu

import qwen3_vl_text_gb300 as Q  # noqa: E402


def _bf16(seed, name, shape, mean=0.0, sigma=1.0):
    bits = W.normal_bf16(seed, name, shape, mean, sigma)
    return W.bf16_bits_to_torch(bits).cuda(), bits_to_f32(bits)


def _e4m3_bytes(q: np.ndarray) -> np.ndarray:
    """Grid values -> e4m3 bytes through torch's converter (exact on grid values)."""
    return torch.from_numpy(np.ascontiguousarray(q, dtype=np.float32)).to(torch.float8_e4m3fn).view(torch.uint8).numpy()


def _quant_gpu(x, rows, cols):
    q = torch.empty(rows, cols, dtype=torch.uint8, device="cuda")
    s = torch.empty(rows, dtype=torch.float32, device="cuda")
    Q.h3enc_op_quant_rows(x, rows, cols, q, s)
    return q, s


def _elementwise_ok(gpu, ref):
    gpu = np.asarray(gpu, np.float64)
    ref = np.asarray(ref, np.float64)
    rms = np.sqrt(np.mean(ref * ref))
    bad = np.abs(gpu - ref) > (2.0 ** -7) * np.abs(ref) + (2.0 ** -9) * rms
    return int(bad.sum()), float(np.max(np.abs(gpu - ref)) / rms)


@pytest.mark.parametrize("rows,cols", [(1, 8), (37, 5120), (300, 8192), (5, 25600)])
def test_quant_rows_bit_exact(rows, cols):
    X, x = _bf16(70, "x", (rows, cols), sigma=3.0)
    scale_rows = np.ones(rows, np.float32)
    scale_rows[::3] = 1e-3                      # a spread of magnitudes, a zero row
    X = X * torch.from_numpy(scale_rows).cuda()[:, None].to(torch.bfloat16)
    if rows > 2:
        X[2].zero_()
    x = t2f(X)
    q, s = _quant_gpu(X, rows, cols)
    torch.cuda.synchronize()
    qr, sr = O.fp8.quantize_rows(x)
    assert np.array_equal(s.cpu().numpy(), sr)
    assert np.array_equal(q.cpu().numpy(), _e4m3_bytes(qr))


@pytest.mark.parametrize("rows,cols", [(129, 5120), (7, 256), (3, 1000), (33, 2048), (2, 3072), (2, 4096),
                                       (2, 6144), (2, 7168), (5, 8192)])
def test_rmsnorm_q8_matches_norm_then_quantise(rows, cols):
    """Every register-tile width of the norm pass (8 to 64 values per thread), ragged too."""
    X, x = _bf16(71, "x", (rows, cols), sigma=2.0)
    G, g = _bf16(72, "g", (cols,), 1.0, 0.1)
    q = torch.empty(rows, cols, dtype=torch.uint8, device="cuda")
    s = torch.empty(rows, dtype=torch.float32, device="cuda")
    Q.h3enc_op_rmsnorm_q8(X, G, q, s, rows, cols, 1e-6)
    # the same bf16 norm output from the plain kernel, quantised by the op above, must agree
    Y = torch.empty_like(X)
    Q.h3enc_op_rmsnorm(X, G, Y, rows, cols, 1e-6)
    q2, s2 = _quant_gpu(Y, rows, cols)
    torch.cuda.synchronize()
    same = (q.cpu().numpy() == q2.cpu().numpy()).mean()
    assert same > 0.999 and np.allclose(s.cpu().numpy(), s2.cpu().numpy(), rtol=2e-7, atol=0)
    # and against the oracle: RMSNorm -> bf16 -> per-row e4m3, dequantised
    qr, sr = O.fp8.quantize_rows(O.round_to_bf16(O.rms_norm(x, g, 1e-6)))
    deq = torch.from_numpy(q.cpu().numpy()).view(torch.float8_e4m3fn).double().numpy() * s.cpu().numpy()[:, None]
    ref = qr * sr[:, None]
    assert np.max(np.abs(deq - ref) / (np.abs(ref) + 1e-3 * np.abs(ref).max())) < 0.07


def _stream_k_shape(case, pairs):
    if case == "tail4":
        return 4 * 256 - 37, (pairs // 4 + 1) * 256, 2048
    if case == "span":
        return 4 * 256 - 37, ((pairs + 40) // 4) * 256, 5120
    if case == "nodp":
        return 2 * 256 - 100, 8 * 256, 8192
    return 2 * 256 - 100, 8 * 256, 256


def _workspace():
    return torch.zeros(Q.h3enc_op_gemm_workspace_bytes(), dtype=torch.uint8, device="cuda")


def _deq(q8: np.ndarray, s: np.ndarray) -> np.ndarray:
    return q8 * s.astype(np.float64)[:, None]


@pytest.mark.parametrize("case", ["small", "tail4", "span", "nodp", "few"])
@pytest.mark.parametrize("epi", [Q.EPI_STORE, Q.EPI_RESIDUAL, Q.EPI_SWIGLU])
def test_gemm_fp8_against_dequantised_product(epi, case):
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    M, N, K = (300, 512, 512) if case == "small" else _stream_k_shape(case, sms // 2)
    A, a = _bf16(73, "A", (M, K))
    qa, sa = O.fp8.quantize_rows(a)
    A8, SA = _quant_gpu(A, M, K)
    if epi == Q.EPI_SWIGLU:
        I = N // 2
        G, g = _bf16(74, "G", (I, K), sigma=0.03)
        U, u = _bf16(75, "U", (I, K), sigma=0.03)
        Wp = torch.empty(N, K, dtype=torch.bfloat16, device="cuda")
        Q.h3enc_op_pack_gate_up(G, U, Wp, I, K)
        W8, SW = _quant_gpu(Wp, N, K)
        qg, sg = O.fp8.quantize_rows(g)
        qu, su = O.fp8.quantize_rows(u)
        xa = _deq(qa, sa)
        ref = O.silu(xa @ _deq(qg, sg).T) * (xa @ _deq(qu, su).T)
        C = torch.empty(M, I, dtype=torch.bfloat16, device="cuda")
        R = None
    else:
        Wt, w = _bf16(76, "W", (N, K), sigma=0.03)
        W8, SW = _quant_gpu(Wt, N, K)
        qw, sw = O.fp8.quantize_rows(w)
        ref = _deq(qa, sa) @ _deq(qw, sw).T
        C = torch.empty(M, N, dtype=torch.bfloat16, device="cuda")
        R = None
        if epi == Q.EPI_RESIDUAL:
            R, r = _bf16(77, "R", (M, N))
            C = R
            ref = r + ref
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    Q.h3enc_op_gemm_fp8(A8, W8, SA, SW, C, M, N, K, epi, R=R, workspace=_workspace(), status=status)
    torch.cuda.synchronize()
    assert int(status.item()) == 0
    bad, worst = _elementwise_ok(t2f(C), ref)
    assert bad == 0, f"{bad} elements off, worst {worst}"


def test_fp8_encode_tiny_model_against_fp8_oracle():
    wl = W.workload(0)
    cfg = wl.model
    inp = W.gen_inputs(wl)
    S = inp["seq_len"]
    enc = make_encoder(wl, cfg, max_tokens=64, fp8=True)
    bf = make_encoder(wl, cfg, max_tokens=64)
    try:
        ids = torch.from_numpy(inp["input_ids"]).cuda()
        pos = torch.from_numpy(inp["positions"]).cuda()
        mask = torch.from_numpy(inp["visual_mask"]).cuda()
        ds = W.bf16_bits_to_torch(inp["deepstack"]).cuda()
        out8 = torch.empty(S, cfg.hidden, dtype=torch.bfloat16, device="cuda")
        out16 = torch.empty_like(out8)
        Q.h3enc_encode(enc.handle, ids, pos, mask, ds, ds.shape[0], inp["n_vis"], None, S, out8)
        Q.h3enc_encode(bf.handle, ids, pos, mask, ds, ds.shape[0], inp["n_vis"], None, S, out16)
        again = torch.empty_like(out8)
        Q.h3enc_encode(enc.handle, ids, pos, mask, ds, ds.shape[0], inp["n_vis"], None, S, again)
        torch.cuda.synchronize()
        assert enc.status() == 0, Q.h3enc_last_error(enc.handle)
        assert torch.equal(out8, again)                      # deterministic
    finally:
        enc.close()
        bf.close()
    x0 = oracle_embed(wl, cfg, inp["input_ids"])
    get = oracle_layer_getter(wl, cfg)
    ws = [get(l) for l in range(cfg.num_layers)]
    dsf = bits_to_f32(inp["deepstack"])
    ref8 = O.forward(x0, inp["positions"], cfg, ws.__getitem__, inp["visual_mask"], dsf, fp8=True)
    ref8bf = O.forward(x0, inp["positions"], cfg, ws.__getitem__, inp["visual_mask"], dsf, fp8=True,
                       storage=GPU_STORAGE)
    ok, msg = parity("fp8 tiny encode", t2f(out8), ref8, ref8bf, 2e-2, 0.05)
    assert ok, "fp8 encode vs fp8 oracle: " + msg
    # the FP8 model departs from the bf16 one by its quantisation error, as the oracle's does
    ref = O.forward(x0, inp["positions"], cfg, ws.__getitem__, inp["visual_mask"], dsf)
    e_gpu = rel_l2(t2f(out8), ref)
    e_orc = rel_l2(ref8, ref)
    assert e_gpu < 1.5 * e_orc + 1e-2, (e_gpu, e_orc)
    assert rel_l2(t2f(out16), ref) < e_gpu                 # the bf16 path is the more accurate one


def test_fp8_one_full_width_layer_against_fp8_oracle():
    """One 5120-wide layer (64 q / 8 kv heads, intermediate 25600) at 512 tokens in FP8
    mode: every projection runs the e4m3 GEMM at full size (stream-K tails included)."""
    wl = W.workload(1)
    cfg = wl.model
    inp = W.gen_inputs(wl)
    S = inp["seq_len"]
    enc = make_encoder(wl, cfg, max_tokens=S, fp8=True)
    try:
        x = W.bf16_bits_to_torch(inp["inputs_embeds"]).cuda()
        pos = torch.from_numpy(inp["positions"]).cuda()
        out = torch.empty(S, cfg.hidden, dtype=torch.bfloat16, device="cuda")
        Q.h3enc_encode_embeds(enc.handle, x, 0, cfg.num_layers, pos, None, None, 0, 0, None, S, out)
        torch.cuda.synchronize()
        assert enc.status() == 0, Q.h3enc_last_error(enc.handle)
        got = t2f(out)
    finally:
        enc.close()
    x0 = bits_to_f32(inp["inputs_embeds"])
    w = oracle_layer_getter(wl, cfg)(0)
    ref8 = O.forward(x0, inp["positions"], cfg, lambda _: w, fp8=True)
    ref8bf = O.forward(x0, inp["positions"], cfg, lambda _: w, fp8=True, storage=GPU_STORAGE)
    ok, msg = parity("fp8 one full-width layer", got, ref8, ref8bf, 5e-3)
    assert ok, "fp8 layer vs fp8 oracle: " + msg


@pytest.mark.slow
def test_fp8_packed_prompts_two_full_width_layers():
    """16 packed prompts of 77-512 tokens through two full-width layers in FP8 mode: per-token
    activation scales and block-diagonal attention over cu_seqlens, against the oracle's FP8
    forward on the same packing."""
    import dataclasses
    wl = W.workload(4)
    cfg = dataclasses.replace(wl.model, num_layers=2)
    inp = W.gen_inputs(wl)
    S = inp["seq_len"]
    cu = [int(c) for c in inp["cu_seqlens"]]
    enc = make_encoder(wl, cfg, max_tokens=S, max_seqs=32, fp8=True)
    try:
        ids = torch.from_numpy(inp["input_ids"]).cuda()
        pos = torch.from_numpy(inp["positions"]).cuda()
        out = torch.empty(S, cfg.hidden, dtype=torch.bfloat16, device="cuda")
        Q.h3enc_encode(enc.handle, ids, pos, None, None, 0, 0, cu, S, out)
        torch.cuda.synchronize()
        assert enc.status() == 0, Q.h3enc_last_error(enc.handle)
        got = t2f(out)
    finally:
        enc.close()
    x0 = oracle_embed(wl, cfg, inp["input_ids"])
    get = oracle_layer_getter(wl, cfg)
    ws = [get(l) for l in range(cfg.num_layers)]
    ref8 = O.forward(x0, inp["positions"], cfg, ws.__getitem__, cu_seqlens=cu, fp8=True)
    ref8bf = O.forward(x0, inp["positions"], cfg, ws.__getitem__, cu_seqlens=cu, fp8=True, storage=GPU_STORAGE)
    ok, msg = parity("fp8 packed prompts, 2 layers", got, ref8, ref8bf, 2e-2, 0.05)
    assert ok, "fp8 packed prompts vs fp8 oracle: " + msg
