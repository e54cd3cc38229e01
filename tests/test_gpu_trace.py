"""The profiling hooks (h3enc_op_gemm_trace_next, h3enc_op_attention_trace_next):
a traced launch computes exactly what an untraced one does, its per-CTA stamps are
ordered, and the attention CTAs account for every key tile of the causal work."""
import numpy as np
import pytest

import workloads as W

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu

import qwen3_vl_text_gb300 as Q  # noqa: E402


def _bf16(seed, name, shape, sigma=1.0):
    return W.bf16_bits_to_torch(W.normal_bf16(seed, name, shape, 0.0, sigma)).cuda()


def test_gemm_timeline_is_ordered_and_changes_nothing():
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    M, N, K = 1000, 5120, 2048                 # 80 tiles: full waves plus a stream-K tail
    A, Wt = _bf16(90, "A", (M, K)), _bf16(91, "W", (N, K), 0.03)
    ws = torch.zeros(Q.h3enc_op_gemm_workspace_bytes(), dtype=torch.uint8, device="cuda")
    plain = torch.empty(M, N, dtype=torch.bfloat16, device="cuda")
    traced = torch.empty_like(plain)
    Q.h3enc_op_gemm(A, Wt, plain, M, N, K, Q.EPI_STORE, workspace=ws)
    tr = torch.zeros(sms * 11, dtype=torch.int64, device="cuda")
    Q.h3enc_op_gemm_trace_next(tr)
    Q.h3enc_op_gemm(A, Wt, traced, M, N, K, Q.EPI_STORE, workspace=ws)
    torch.cuda.synchronize()
    assert torch.equal(plain, traced)
    t = tr.view(sms, 11).cpu().numpy()
    ran = t[:, 0] > 0
    assert ran.sum() >= 2
    t = t[ran]
    assert np.all(t[:, 1] >= t[:, 0]) and np.all(t[:, 10] >= t[:, 1])     # start <= ready <= end
    assert np.all(t[:, 5] <= t[:, 10]) and np.all(t[:, 5] >= t[:, 1])     # data-parallel epilogues end in between
    sk = t[:, 6] > 0                                                         # CTAs with a stream-K part
    assert sk.any()
    assert np.all(t[sk, 7] >= t[sk, 6]) and np.all(t[sk, 9] >= t[sk, 7])  # partial written, then reduced
    # an unarmed launch afterwards leaves the buffer alone
    before = tr.clone()
    Q.h3enc_op_gemm(A, Wt, plain, M, N, K, Q.EPI_STORE, workspace=ws)
    torch.cuda.synchronize()
    assert torch.equal(tr, before)


def test_attention_timeline_counts_every_key_tile():
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    S, nq, nkv, d = 1024, 64, 8, 128
    X = _bf16(92, "qkv", (S, (nq + 2 * nkv) * d))
    plain = torch.empty(S, nq * d, dtype=torch.bfloat16, device="cuda")
    traced = torch.empty_like(plain)
    Q.h3enc_op_attention(X, plain, S, nq, nkv, d)
    tr = torch.zeros(sms * 9, dtype=torch.int64, device="cuda")
    Q.h3enc_op_attention_trace_next(tr, sms)
    Q.h3enc_op_attention(X, traced, S, nq, nkv, d)
    torch.cuda.synchronize()
    assert torch.equal(plain, traced)
    t = tr.view(sms, 9).cpu().numpy()
    t = t[t[:, 0] > 0]
    # causal with 8 q heads per kv head: an item is one 128-row query tile of two heads of a
    # kv group, and runs the key tiles up to its own rows
    assert len(t) == min(sms, (nq // 2) * (S // 128))
    assert np.all(t[:, 6] >= t[:, 0])                                        # end after start (ns)
    assert np.all(t[:, 5] >= t[:, 1])                                        # clock stamps ordered
    per_pair = sum(q0 // 128 + 1 for q0 in range(0, S, 128))
    assert int(t[:, 8].sum()) == (nq // 2) * per_pair
    assert int(t[:, 8].max()) <= 8                                           # heavy-first rounds balance
    assert len(set(t[:, 7].tolist())) == len(t)                              # one CTA per SM
