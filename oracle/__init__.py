"""CPU oracle for the Qwen3-VL text-decoder prefill (MiniMax H3 layer-50 encoder).

TEST INFRASTRUCTURE ONLY.  Nothing on the product path imports, links or runs
this package; only ``tests/``, ``__graft_entry__.smoke()`` and ``bench.py``'s
CPU-baseline leg (and its ``--impl reference`` arm) use it.

It is a plain, slow restatement of the forward that the page
"vllm-omni vllm_omni/diffusion/models/minimax_h3/encoder.py" defines
(``MiniMaxH3Qwen3VLTextModel.forward`` and the classes it calls), evaluated in
float32 (or float64) from bf16-rounded weights and inputs.  It shares no code
with the CUDA path.

Parity status of each function is listed in its docstring; every function is
pinned by ``tests/test_oracle_pins.py`` (the front end by the hand-derived
fixtures under ``tests/golden/``) except the end-to-end 50-layer forward
on random weights, whose output has no independent value to compare with
("parity unpinned" beyond the per-step pins and the structural invariants).
"""
from .qwen3vl_text import *  # noqa: F401,F403
from . import fp8  # noqa: F401  (online-FP8 linears)
from . import frontend  # noqa: F401  (token ids -> positions, visual rows, DeepStack order)
from . import vision  # noqa: F401  (the vision tower: visual embeddings and DeepStack features)
