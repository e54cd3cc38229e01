"""The C-ABI library without a GPU: it builds, loads, exports every symbol
the headers declare, and rejects bad configurations before touching CUDA."""
import ctypes
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _declared():
    names = set()
    for f in os.listdir(os.path.join(ROOT, "include")):
        if f.endswith(".h"):
            text = open(os.path.join(ROOT, "include", f)).read()
            names |= set(re.findall(r"^H3ENC_API\s+[\w\s\*]*?\b((?:h3enc|h3vis)_\w+)\s*\(", text, re.M))
    return names


@pytest.fixture(scope="module")
def Q():
    import __graft_entry__
    __graft_entry__._build_module().build()
    import qwen3_vl_text_gb300
    return qwen3_vl_text_gb300


def test_every_declared_symbol_is_exported(Q):
    names = _declared()
    assert len(names) >= 22
    lib = ctypes.CDLL(Q.LIB_PATH)
    missing = [n for n in sorted(names) if not hasattr(lib, n)]
    assert not missing, missing
    assert set(Q._SIGS) == names


def _cfg(Q, **kw):
    c = Q.Config()
    base = dict(num_layers=2, hidden=256, n_heads=4, n_kv_heads=2, head_dim=64, intermediate=768, vocab=1024,
                rms_eps=1e-6, rope_theta=1e6, max_tokens=64, max_seqs=4, num_deepstack=1)
    base.update(kw)
    for k, v in base.items():
        setattr(c, k, v)
    c.mrope_section = (ctypes.c_int32 * 3)(12, 10, 10)
    return c


@pytest.mark.parametrize("kw,code", [
    (dict(num_layers=0), 2), (dict(head_dim=96), 6), (dict(n_heads=3), 2), (dict(hidden=200), 6),
    (dict(intermediate=700), 6), (dict(max_seqs=5000), 2), (dict(rms_eps=0.0), 2), (dict(max_tokens=0), 2),
])
def test_bad_configs_rejected_before_cuda(Q, kw, code):
    with pytest.raises(Q.H3encError) as e:
        Q.h3enc_create(_cfg(Q, **kw))
    assert e.value.code == code
    assert Q.h3enc_last_error(None)


def test_create_without_gpu_reports_cuda_error(Q):
    torch = pytest.importorskip("torch")
    if torch.cuda.is_available():
        pytest.skip("a GPU is present")
    with pytest.raises(Q.H3encError) as e:
        Q.h3enc_create(_cfg(Q))
    assert e.value.code == 7


def test_op_entries_validate_arguments(Q):
    with pytest.raises(Q.H3encError) as e:
        Q.h3enc_op_gemm(16, 16, 16, 4, 100, 64, Q.EPI_STORE, stream=0)      # N not a multiple of 256
    assert e.value.code == 2
    with pytest.raises(Q.H3encError):
        Q.h3enc_op_rmsnorm(16, 16, 16, 4, 8200, 1e-6, stream=0)            # cols > 8192
    with pytest.raises(Q.H3encError):
        Q.h3enc_op_attention(16, 16, 10, 4, 3, 64, stream=0)               # n_heads % n_kv_heads
    with pytest.raises(Q.H3encError):
        Q.h3enc_op_attention(16, 16, 10, 4, 2, 64, [0, 4, 3, 10], stream=0)  # decreasing cu_seqlens
    with pytest.raises(Q.H3encError):
        Q.h3enc_op_pack_gate_up(16, 16, 16, 100, 64, stream=0)              # I % 128
    with pytest.raises(Q.H3encError) as e:
        Q.h3enc_op_rope_table_ex(16, 100, 128, 5e6, (24, 20, 20), 96, 16, 16, stream=0)   # stride < S
    assert e.value.code == 2
    with pytest.raises(Q.H3encError):
        Q.h3enc_op_rope_table_ex(16, 10, 12, 5e6, (2, 2, 2), 32, 16, 16, stream=0)       # head_dim % 8
    with pytest.raises(Q.H3encError) as e:                                              # table stride < M
        Q.h3enc_op_gemm_qkv_rope_ex(16, 16, 16, 100, 512, 4, 2, 64, 16, 16, 1e-6, 16, 16, 64, stream=0)
    assert e.value.code == 2
    assert Q.h3enc_op_attention_workspace_bytes(96) == 0                                # head_dim not 64/128
    with pytest.raises(Q.H3encError) as e:                                              # no workspace
        Q._check(Q.lib.h3enc_op_attention_bidir_ws(16, 16, 256, 4, 64, None, 0, None, 1 << 30, None))
    assert e.value.code == 2


def test_handle_calls_reject_a_null_handle(Q):
    """The graph, profiling and capture switches check their handle before touching CUDA."""
    for call in (lambda: Q.h3enc_set_graphs(None, True), lambda: Q.h3enc_set_profiling(None, True),
                 lambda: Q.h3enc_set_profiling_layer(None, 0)):
        with pytest.raises(Q.H3encError) as e:
            call()
        assert e.value.code == 2
    assert Q.h3enc_graph_count(None) == 0 and Q.h3enc_launch_count(None) == 0
