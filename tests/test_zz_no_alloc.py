"""The GEMM entry point for callers that cannot allocate device memory.

Some callers of this library cannot call cudaMalloc: code running inside
another framework's allocator callback or after a memory pool has taken the
whole device, plugins that only receive their input and output buffers.
h3enc_op_gemm_noalloc serves them from a fixed scratch array inside the
library instead of a caller workspace.  It must give the same result as
h3enc_op_gemm with a workspace, call after call (the array keeps the previous
call's contents).  This file sorts last so a stop-at-first-failure run has
already run every other test; it also passes alone in a fresh process.
"""
import numpy as np
import pytest

import workloads as W

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu

import qwen3_vl_text_gb300 as Q  # noqa: E402


def _bf16(seed, name, shape, sigma=1.0):
    return W.bf16_bits_to_torch(W.normal_bf16(seed, name, shape, 0.0, sigma)).cuda()


def _close(a, b):
    """The per-element bound of the GEMM parity tests: 2^-7 |ref| + 2^-9 RMS(ref)."""
    a = a.float().cpu().numpy().astype(np.float64)
    b = b.float().cpu().numpy().astype(np.float64)
    rms = np.sqrt(np.mean(b * b))
    return int((np.abs(a - b) > 2.0 ** -7 * np.abs(b) + 2.0 ** -9 * rms).sum())


@pytest.mark.parametrize("epi", [Q.EPI_RESIDUAL, Q.EPI_SWIGLU])
def test_noalloc_gemm_matches_workspace_gemm_twice(epi):
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    assert Q.h3enc_op_gemm_noalloc_scratch_bytes() >= sms * 128 * 256 * 4
    nm = 8
    nn = sms // nm + 1                       # a partial last wave: the split path uses the scratch
    M, N, K = nm * 128 - 5, nn * 256, 1536
    A = _bf16(50, "A", (M, K))
    Wt = _bf16(51, "W", (N, K), sigma=0.03)
    ldc = N // 2 if epi == Q.EPI_SWIGLU else N
    R0 = _bf16(52, "R", (M, ldc)) if epi == Q.EPI_RESIDUAL else None
    ws = torch.zeros(Q.h3enc_op_gemm_workspace_bytes(), dtype=torch.uint8, device="cuda")
    ref = torch.empty(M, ldc, dtype=torch.bfloat16, device="cuda") if R0 is None else R0.clone()
    Q.h3enc_op_gemm(A, Wt, ref, M, N, K, epi, R=None if R0 is None else ref, workspace=ws)
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    for _ in range(2):                       # two calls in a row on the shared array
        out = torch.empty(M, ldc, dtype=torch.bfloat16, device="cuda") if R0 is None else R0.clone()
        Q.h3enc_op_gemm_noalloc(A, Wt, out, M, N, K, epi, R=None if R0 is None else out, status=status)
        torch.cuda.synchronize()
        assert int(status.item()) == 0
        assert _close(out, ref) == 0
