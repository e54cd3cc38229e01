"""The GEMM entry point for callers that cannot allocate device memory.

Some callers of this library cannot call cudaMalloc: code running inside
another framework's allocator callback or after a memory pool has taken the
whole device, plugins that only receive their input and output buffers.
h3enc_op_gemm_noalloc serves them from a fixed scratch array inside the
library instead of a caller workspace.  Same kernel, same schedule: its output
must equal h3enc_op_gemm's with a workspace bit for bit, call after call (the
array keeps the previous call's contents), and meet the CPU oracle at the
per-kernel bound.  The shape puts a partial last wave on the split path (the
only phase that touches the scratch), and the phase timeline checks that the
split ran.  This file sorts last so a stop-at-first-failure run has already
run every other test; it also passes alone in a fresh process.
"""
import numpy as np
import pytest

import oracle as O
import workloads as W

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu

import qwen3_vl_text_gb300 as Q  # noqa: E402

TRACE_STAMPS = 11          # per-CTA entries of the GEMM timeline
STAMP_SPLIT_WRITTEN = 7    # "stream-K partials written"


def _bf16(seed, name, shape, sigma=1.0):
    bits = W.normal_bf16(seed, name, shape, 0.0, sigma)
    return W.bf16_bits_to_torch(bits).cuda(), O.bf16_bits_to_float(bits, np.float64)


def _bad_elements(gpu, ref):
    """Elements outside the per-kernel bound 2^-7 |ref| + 2^-9 RMS(ref)."""
    gpu = gpu.float().cpu().numpy().astype(np.float64)
    rms = np.sqrt(np.mean(ref * ref))
    return int((np.abs(gpu - ref) > 2.0 ** -7 * np.abs(ref) + 2.0 ** -9 * rms).sum())


@pytest.mark.parametrize("epi", [Q.EPI_RESIDUAL, Q.EPI_SWIGLU])
def test_noalloc_gemm_matches_workspace_gemm_twice(epi):
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    assert Q.h3enc_op_gemm_noalloc_scratch_bytes() >= sms * 2 * 128 * 256 * 4
    pairs = sms // 2
    M, N, K = 4 * 256 - 37, (pairs // 4 + 1) * 256, 2048    # one full wave of 256x256 tiles + 4, ragged M
    A, a = _bf16(50, "A", (M, K))
    if epi == Q.EPI_SWIGLU:
        I = N // 2
        G, g = _bf16(51, "G", (I, K), sigma=0.03)
        U, u = _bf16(52, "U", (I, K), sigma=0.03)
        Wt = torch.empty(N, K, dtype=torch.bfloat16, device="cuda")
        Q.h3enc_op_pack_gate_up(G, U, Wt, I, K)
        want = O.silu(O.linear(a, g)) * O.linear(a, u)
        R0 = None
    else:
        Wt, w = _bf16(51, "W", (N, K), sigma=0.03)
        R0, r = _bf16(53, "R", (M, N))
        want = r + O.linear(a, w)
    ldc = N // 2 if epi == Q.EPI_SWIGLU else N

    def fresh():
        return torch.empty(M, ldc, dtype=torch.bfloat16, device="cuda") if R0 is None else R0.clone()

    ws = torch.zeros(Q.h3enc_op_gemm_workspace_bytes(), dtype=torch.uint8, device="cuda")
    ref = fresh()
    Q.h3enc_op_gemm(A, Wt, ref, M, N, K, epi, R=None if R0 is None else ref, workspace=ws)
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    for call in range(2):                    # two calls in a row on the shared array
        out = fresh()
        trace = torch.zeros(sms * TRACE_STAMPS, dtype=torch.int64, device="cuda")
        Q.h3enc_op_gemm_trace_next(trace)
        Q.h3enc_op_gemm_noalloc(A, Wt, out, M, N, K, epi, R=None if R0 is None else out, status=status)
        torch.cuda.synchronize()
        assert int(status.item()) == 0, call
        split_ctas = int((trace.view(sms, TRACE_STAMPS)[:, STAMP_SPLIT_WRITTEN] != 0).sum())
        assert split_ctas > 0, f"call {call}: the split phase did not run, the scratch was not used"
        assert torch.equal(out, ref), f"call {call}: differs from h3enc_op_gemm with a workspace"
        if call == 0:
            assert _bad_elements(out, want) == 0, "outside the per-kernel bound against the oracle"
