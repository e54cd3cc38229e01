"""RMSNorm folded into the projections, piece by piece, through the C ABI.

  rmsnorm(x, g) W^T = diag(1 / sqrt(mean(x^2) + eps)) x (W diag(g))^T

(page "vllm-omni ... encoder.py", MiniMaxH3Qwen3VLRMSNorm followed by the
projection reading it).  Row statistics and the weight fold are exact
operations and are compared bit for bit; the scaled projections against the
oracle with the per-kernel tolerance of test_gpu_ops.py; the whole path
against rmsnorm + linear by relative L2 (the fold rounds W diag(g) to bf16
where the separate norm rounds its output instead).  Stream-K shapes cover the
reduction path of the epilogue as well as the data-parallel one.
"""
import numpy as np
import pytest

import oracle as O
import workloads as W
from _harness import bits_to_f32, make_encoder, rel_l2, t2f

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu

import qwen3_vl_text_gb300 as Q  # noqa: E402

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


def _slot_sums(x):
    """Slot-major sums of squares of x [rows, cols], fp32, each slot added in column order
    (a bf16 value squared is exact in fp32, so fused and separate multiply-add agree)."""
    x = np.asarray(x, np.float32)
    rows, cols = x.shape
    out = np.zeros((cols // 128, rows), np.float32)
    for s in range(cols // 128):
        acc = np.zeros(rows, np.float32)
        for c in range(128 * s, 128 * s + 128):
            acc = (acc + x[:, c] * x[:, c]).astype(np.float32)
        out[s] = acc
    return out


def _workspace():
    return torch.zeros(Q.h3enc_op_gemm_workspace_bytes(), dtype=torch.uint8, device="cuda")


def _shape(case):
    """(M, N, K): dp = data-parallel tiles only; split = one wave + 4 tiles shared by all pairs."""
    pairs = torch.cuda.get_device_properties(0).multi_processor_count // 2
    if case == "dp":
        return 300, 1024, 512
    return 4 * 256 - 37, (pairs // 4 + 1) * 256, 2048


@pytest.mark.parametrize("rows,cols", [(1, 128), (300, 5120), (1024, 256)])
def test_row_sumsq_bit_exact(rows, cols):
    X, x = _bf16(40, "x", (rows, cols))
    ss = torch.empty(cols // 128, rows, dtype=torch.float32, device="cuda")
    Q.h3enc_op_row_sumsq(X, rows, cols, ss)
    torch.cuda.synchronize()
    assert np.array_equal(ss.cpu().numpy(), _slot_sums(x))


def test_fold_cols_bit_exact():
    N, K = 384, 5120
    Wt, w = _bf16(41, "W", (N, K), sigma=0.02)
    G, g = _bf16(42, "g", (K,), 1.0, 0.1)
    Q.h3enc_op_fold_cols(Wt, N, K, G)
    torch.cuda.synchronize()
    want = O.round_to_bf16((w.astype(np.float32) * g.astype(np.float32)[None, :]).astype(np.float32))
    assert np.array_equal(t2f(Wt), want)


@pytest.mark.parametrize("case", ["dp", "split"])
@pytest.mark.parametrize("epi", [Q.EPI_STORE, Q.EPI_RESIDUAL])
def test_producer_statistics_are_those_of_the_stored_output(epi, case):
    M, N, K = _shape(case)
    A, _ = _bf16(43, "A", (M, K))
    Wt, _ = _bf16(44, "W", (N, K), sigma=0.03)
    R, _ = _bf16(45, "R", (M, N))
    ws = _workspace()
    plain = R.clone()
    Q.h3enc_op_gemm(A, Wt, plain, M, N, K, epi, R=plain if epi == Q.EPI_RESIDUAL else None, workspace=ws)
    C = R.clone()
    ss = torch.full((N // 128, M), -1.0, dtype=torch.float32, device="cuda")
    Q.h3enc_op_gemm_rms(A, Wt, C, M, N, K, epi, R=C if epi == Q.EPI_RESIDUAL else None, ss_out=ss, workspace=ws)
    torch.cuda.synchronize()
    assert torch.equal(C, plain), "emitting statistics changed the output"
    assert np.array_equal(ss.cpu().numpy(), _slot_sums(t2f(C)))


@pytest.mark.parametrize("case", ["dp", "split"])
@pytest.mark.parametrize("epi", [Q.EPI_STORE, Q.EPI_RESIDUAL, Q.EPI_SWIGLU])
def test_consumer_rows_scaled_by_the_norm(epi, case):
    M, N, K = _shape(case)
    A, a = _bf16(46, "A", (M, K))
    ss = torch.from_numpy(_slot_sums(a)).cuda()
    a64 = a.astype(np.float64)
    r = 1.0 / np.sqrt(np.sum(a64 ** 2, axis=1) / K + EPS)
    ws = _workspace()
    if epi == Q.EPI_SWIGLU:
        I = N // 2
        G, gg = _bf16(47, "G", (I, K), sigma=0.03)
        U, uu = _bf16(48, "U", (I, K), sigma=0.03)
        Wt = torch.empty(N, K, dtype=torch.bfloat16, device="cuda")
        Q.h3enc_op_pack_gate_up(G, U, Wt, I, K)
        gate = r[:, None] * O.linear(a64, gg.astype(np.float64))
        ref = O.silu(gate) * (r[:, None] * O.linear(a64, uu.astype(np.float64)))
        C = torch.empty(M, I, dtype=torch.bfloat16, device="cuda")
        R = None
    else:
        Wt, w = _bf16(49, "W", (N, K), sigma=0.03)
        ref = r[:, None] * O.linear(a64, w.astype(np.float64))
        C = torch.empty(M, N, dtype=torch.bfloat16, device="cuda")
        R = None
        if epi == Q.EPI_RESIDUAL:
            R0, r0 = _bf16(50, "R", (M, N))
            C = R0.clone()
            R = C
            ref = r0 + ref
    Q.h3enc_op_gemm_rms(A, Wt, C, M, N, K, epi, R=R, ss_in=ss, eps=EPS, workspace=ws)
    torch.cuda.synchronize()
    bad, worst = _elementwise_ok(t2f(C), ref)
    assert bad == 0, f"{bad} elements off, worst {worst}"


@pytest.mark.parametrize("case", ["dp", "split"])
def test_folded_norm_matches_norm_then_projection(case):
    """fold(W, g) with the row statistics of x against rmsnorm(x, g) W^T in the oracle."""
    M, N, K = _shape(case)
    X, x = _bf16(51, "x", (M, K))
    Wt, w = _bf16(52, "W", (N, K), sigma=0.03)
    G, g = _bf16(53, "g", (K,), 1.0, 0.1)
    ss = torch.empty(K // 128, M, dtype=torch.float32, device="cuda")
    Q.h3enc_op_row_sumsq(X, M, K, ss)
    Q.h3enc_op_fold_cols(Wt, N, K, G)
    C = torch.empty(M, N, dtype=torch.bfloat16, device="cuda")
    Q.h3enc_op_gemm_rms(X, Wt, C, M, N, K, Q.EPI_STORE, ss_in=ss, eps=EPS, workspace=_workspace())
    torch.cuda.synchronize()
    ref = O.linear(O.rms_norm(x.astype(np.float64), g.astype(np.float64), EPS), w.astype(np.float64))
    # bf16 rounding of the folded weights plus that of the output: well under 2^-8 relative L2
    assert rel_l2(t2f(C), ref) < 4e-3, f"rel {rel_l2(t2f(C), ref):.3g}"


@pytest.mark.parametrize("split", [False, True])
def test_qkv_projection_with_folded_input_norm(split):
    d, nq, nkv = 128, 64, 8
    M, K = (1024, 2048) if split else (300, 512)   # 160 tiles of 32 k-blocks: a stream-K tail
    N = (nq + 2 * nkv) * d
    A, a = _bf16(54, "A", (M, K))
    Wt, w = _bf16(55, "Wqkv", (N, K), sigma=0.05)
    Gq, gq = _bf16(56, "gq", (d,), 1.0, 0.1)
    Gk, gk = _bf16(57, "gk", (d,), 1.0, 0.1)
    ss = torch.from_numpy(_slot_sums(a)).cuda()
    pos = np.stack([np.arange(M) * 3, np.arange(M) * 5 + 1, np.arange(M) * 7 + 2]).astype(np.int32)
    c = torch.empty(M, d // 2, device="cuda")
    s = torch.empty_like(c)
    Q.h3enc_op_rope_table(torch.from_numpy(pos).cuda(), M, d, 5e6, (24, 20, 20), c, s)
    C = torch.empty(M, N, dtype=torch.bfloat16, device="cuda")
    Q.h3enc_op_gemm_qkv_rope_rms(A, Wt, C, M, K, nq, nkv, d, Gq, Gk, EPS, c, s, ss, EPS,
                                 workspace=_workspace() if split else None)
    torch.cuda.synchronize()
    r = 1.0 / np.sqrt(np.sum(a.astype(np.float64) ** 2, axis=1) / K + EPS)
    x = r[:, None] * O.linear(a.astype(np.float64), w.astype(np.float64))
    cos, sin = O.rope_cos_sin(pos, d, 5e6, (24, 20, 20))
    q = O.apply_rope(O.rms_norm(x[:, :nq * d].reshape(M, nq, d), gq, EPS), cos, sin).reshape(M, -1)
    k = O.apply_rope(O.rms_norm(x[:, nq * d:(nq + nkv) * d].reshape(M, nkv, d), gk, EPS), cos, sin).reshape(M, -1)
    ref = np.concatenate([q, k, x[:, (nq + nkv) * d:]], axis=1)
    bad, worst = _elementwise_ok(t2f(C), ref)
    assert bad == 0, f"{bad} elements off, worst {worst}"


def test_reloading_weights_after_the_fold():
    """A projection reloaded after finalize is folded again on the next finalize (same
    encode, bit for bit); a norm reloaded alone is refused until its projections follow."""
    wl = W.workload(0)
    cfg = wl.model
    inp = W.gen_inputs(wl)
    S = inp["seq_len"]
    enc = make_encoder(wl, cfg, max_tokens=64)
    try:
        ids = torch.from_numpy(inp["input_ids"]).cuda()
        pos = torch.from_numpy(inp["positions"]).cuda()

        def encode():
            out = torch.empty(S, cfg.hidden, dtype=torch.bfloat16, device="cuda")
            enc.encode(ids, pos, out)
            torch.cuda.synchronize()
            return out

        want = encode()
        specs = {name: (shape, mean, sigma) for name, shape, mean, sigma in W.layer_weight_specs(cfg, 1)}

        def reload(suffix):
            name = next(n for n in specs if n.endswith(suffix))
            shape, mean, sigma = specs[name]
            enc.load(name, W.gen_weight(wl.seed, name, shape, mean, sigma, device="cuda"))

        reload("self_attn.q_proj.weight")
        reload("mlp.up_proj.weight")
        torch.cuda.synchronize()
        enc.finalize()
        assert torch.equal(encode(), want)
        reload("input_layernorm.weight")
        torch.cuda.synchronize()
        with pytest.raises(Q.H3encError) as e:
            enc.finalize()
        assert "reload q/k/v_proj" in str(e.value)
        for p in ("self_attn.q_proj.weight", "self_attn.k_proj.weight", "self_attn.v_proj.weight"):
            reload(p)
        torch.cuda.synchronize()
        enc.finalize()
        assert torch.equal(encode(), want)
    finally:
        enc.close()
