"""Online-FP8 linears of the encoder, restated for the CPU oracle.

TEST INFRASTRUCTURE ONLY (see the package docstring).

Page 1 ("vllm-omni vllm_omni/diffusion/models/minimax_h3/encoder.py"),
``_validate_encoder_quant_config`` and the ``_is_quantized_linear`` branches of
``MiniMaxH3Qwen3VLTextAttention.forward`` / ``MiniMaxH3Qwen3VLTextMLP.forward``:
the encoder accepts online FP8 (the bf16 checkpoint quantised when it is
loaded; serialized FP8 checkpoints are refused), and a quantised QKV or gate/up
projection runs as one packed linear whose output is then split.  The pages do
not spell out the scaling; the reading taken here (and by the CUDA path) is:

* e4m3 values ("fn" variant: no infinities, largest finite 448), round to
  nearest, ties to even, saturating at +-448;
* weights: one fp32 scale per output channel (row of the ``[out, in]``
  matrix), ``scale = amax(row) / 448``;
* activations: one fp32 scale per token (row), computed at run time from the
  bf16 activation the projection receives, same rule;
* ``q = e4m3(x * (448 / amax))``, the reciprocal and the product each rounded
  once in fp32 (a multiply per element instead of a divide); a row of zeros
  gets scale 1 and quantises to zeros;
* ``y = (q_a * s_a) @ (q_w * s_w)^T`` accumulated exactly (float64 here).
"""
from __future__ import annotations

import numpy as np

from .qwen3vl_text import round_to_bf16

__all__ = ["E4M3_MAX", "e4m3_round", "quantize_rows", "fp8_linear"]

E4M3_MAX = 448.0


def e4m3_round(x: np.ndarray) -> np.ndarray:
    """Round to the nearest e4m3 value (ties to even), saturating at +-448.

    e4m3: 1 sign bit, 4 exponent bits (bias 7), 3 mantissa bits; normal numbers
    have 3 fraction bits after the leading one, so inside the binade [2^e, 2^(e+1))
    the spacing is 2^(e-3); below the smallest normal 2^-6 the spacing stays
    2^-9 (subnormals).  Returns float64 values on that grid.
    """
    x = np.asarray(x, dtype=np.float64)
    a = np.abs(x)
    _, e = np.frexp(a)                      # a = m * 2^e, m in [0.5, 1): leading bit 2^(e-1)
    lead = np.maximum(e - 1, -6)            # subnormals share the spacing of the first binade
    step = np.ldexp(1.0, lead - 3)
    q = np.rint(a / step) * step            # a / step is exact (power-of-two scaling); rint ties to even
    q = np.minimum(q, E4M3_MAX)
    return np.copysign(q, x)


def quantize_rows(x: np.ndarray):
    """Per-row quantisation: ``scale = amax / 448`` and ``inv = 448 / amax`` (each one
    fp32 division), ``q = e4m3(x * inv)`` with the product in fp32.
    Returns (q as float64 grid values, scale float32[rows])."""
    x32 = np.asarray(x, dtype=np.float32)
    amax = np.max(np.abs(x32), axis=1)
    pos = amax > 0
    safe = np.where(pos, amax, np.float32(1.0)).astype(np.float32)
    scale = np.where(pos, safe / np.float32(E4M3_MAX), np.float32(1.0)).astype(np.float32)
    inv = np.where(pos, np.float32(E4M3_MAX) / safe, np.float32(1.0)).astype(np.float32)
    q = e4m3_round((x32 * inv[:, None]).astype(np.float32))
    return q, scale


def fp8_linear(x: np.ndarray, w: np.ndarray) -> np.ndarray:
    """``F.linear`` of an online-FP8 projection: the bf16 activation ``x`` and the
    bf16 weight ``w [out, in]`` are each quantised per row, and the product of the
    dequantised operands is formed exactly (float64), returned in ``x``'s dtype."""
    qa, sa = quantize_rows(round_to_bf16(np.asarray(x, dtype=np.float32)))
    qw, sw = quantize_rows(w)
    a = qa * sa.astype(np.float64)[:, None]
    b = qw * sw.astype(np.float64)[:, None]
    return (a @ b.T).astype(np.asarray(x).dtype, copy=False)
