"""qwen3_vl_text_gb300 — Qwen3-VL text-decoder prefill (MiniMax H3 layer-50
encoder) on one GB300.

Thin ctypes binding over ``libh3enc.so`` (C ABI in ``include/h3enc.h`` and
``include/h3enc_ops.h``): the functions below carry the C names and only
marshal arguments (device pointers from torch tensors, the current CUDA
stream).  Every step of the encode runs in the library's CUDA kernels; if the
library cannot be loaded, importing the binding raises — there is no fallback.
"""
from __future__ import annotations

import ctypes
import os

__all__ = [
    "lib", "H3encError", "Config", "STATUS", "EPI_STORE", "EPI_RESIDUAL", "EPI_SWIGLU", "EPI_RESIDUAL_DS",
    "EPI_GELU_TANH", "EPI_GELU_ERF",
    "h3enc_create", "h3enc_load_weights", "h3enc_finalize_weights", "h3enc_encode", "h3enc_encode_embeds", "h3enc_encode_multimodal",
    "h3enc_encode_host", "h3enc_set_layer_capture", "h3enc_get_status", "h3enc_last_error", "h3enc_destroy",
    "h3enc_set_profiling", "h3enc_set_profiling_classes", "h3enc_set_profiling_layer", "h3enc_get_profile", "h3enc_launch_count", "h3enc_num_sms",
    "h3enc_set_graphs", "h3enc_graph_count",
    "h3enc_build_positions", "h3enc_aggregate_deepstack",
    "h3enc_op_gemm", "h3enc_op_gemm_workspace_bytes", "h3enc_op_gemm_trace_next", "h3enc_op_attention_trace_next", "h3enc_op_gemm_noalloc", "h3enc_op_gemm_noalloc_scratch_bytes", "h3enc_op_pack_gate_up", "h3enc_op_rmsnorm", "h3enc_op_gemm_fp8", "h3enc_op_quant_rows",
    "h3enc_op_rmsnorm_q8", "h3enc_op_wait_probe", "h3enc_op_rope_table", "h3enc_op_rope_table_ex",
    "h3enc_op_gemm_qkv_rope_ex",
    "h3enc_op_gemm_qkv_rope", "h3enc_op_gemm_qkv_rope_rms", "h3enc_op_gemm_rms", "h3enc_op_row_sumsq",
    "h3enc_op_fold_cols", "h3enc_op_layernorm", "h3enc_op_vision_pos_embed", "h3enc_op_vision_rope_table",
    "h3enc_op_gemm_bias", "h3enc_op_gemm_qkv_rope_bias", "h3enc_op_attention_bidir", "VisionConfig",
    "h3enc_op_attention_bidir_ws", "h3enc_op_attention_workspace_bytes",
    "h3vis_create", "h3vis_load_weights", "h3vis_finalize_weights", "h3vis_encode", "h3vis_get_status",
    "h3vis_last_error", "h3vis_launch_count", "h3vis_destroy", "VisionEncoder", "h3enc_op_attention", "h3enc_op_embed", "h3enc_op_vis_rank", "Encoder",
    "KERNEL_CLASSES",
]

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "libh3enc.so")

STATUS = {0: "OK", 1: "WARN_IGNORED", 2: "ERR_INVALID_ARG", 3: "ERR_SHAPE", 4: "ERR_NOT_LOADED",
          5: "ERR_MISSING_WEIGHTS", 6: "ERR_UNSUPPORTED", 7: "ERR_CUDA", 8: "ERR_OOM",
          9: "ERR_DEVICE_TIMEOUT", 10: "ERR_DEVICE_BOUNDS"}
EPI_STORE, EPI_RESIDUAL, EPI_SWIGLU, EPI_RESIDUAL_DS = 0, 1, 2, 3
EPI_GELU_TANH, EPI_GELU_ERF = 5, 6
KERNEL_CLASSES = ["prep", "rmsnorm", "gemm_qkv", "quant", "attention", "gemm_o", "gemm_gate_up", "gemm_down"]


class H3encError(RuntimeError):
    def __init__(self, code: int, msg: str):
        super().__init__(f"h3enc {STATUS.get(code, code)}: {msg}")
        self.code = code


class Config(ctypes.Structure):
    _fields_ = [("num_layers", ctypes.c_int32), ("hidden", ctypes.c_int32), ("n_heads", ctypes.c_int32),
                ("n_kv_heads", ctypes.c_int32), ("head_dim", ctypes.c_int32), ("intermediate", ctypes.c_int32),
                ("vocab", ctypes.c_int32), ("rms_eps", ctypes.c_float), ("rope_theta", ctypes.c_float),
                ("mrope_section", ctypes.c_int32 * 3), ("max_tokens", ctypes.c_int32),
                ("max_seqs", ctypes.c_int32), ("num_deepstack", ctypes.c_int32), ("linear_fp8", ctypes.c_int32),
                ("separate_norm", ctypes.c_int32)]


class VisionConfig(ctypes.Structure):
    _fields_ = [("depth", ctypes.c_int32), ("hidden", ctypes.c_int32), ("num_heads", ctypes.c_int32),
                ("intermediate", ctypes.c_int32), ("in_channels", ctypes.c_int32), ("patch_size", ctypes.c_int32),
                ("temporal_patch_size", ctypes.c_int32), ("spatial_merge_size", ctypes.c_int32),
                ("out_hidden", ctypes.c_int32), ("num_position_embeddings", ctypes.c_int32),
                ("num_deepstack", ctypes.c_int32), ("deepstack_indexes", ctypes.c_int32 * 8),
                ("ln_eps", ctypes.c_float), ("rope_theta", ctypes.c_float), ("max_patches", ctypes.c_int32)]


def _load():
    if not os.path.exists(LIB_PATH):
        raise ImportError(f"{LIB_PATH} is missing: build it with qwen3_vl_text_gb300.build.build()")
    return ctypes.CDLL(LIB_PATH)


lib = _load()

_P, _I32, _I64, _F = ctypes.c_void_p, ctypes.c_int32, ctypes.c_int64, ctypes.c_float
_SIGS = {
    "h3enc_create": ([ctypes.POINTER(Config), ctypes.POINTER(_P)], _I32),
    "h3enc_load_weights": ([_P, ctypes.c_char_p, _P, _I32, ctypes.POINTER(_I64), _I32, _I32], _I32),
    "h3enc_finalize_weights": ([_P], _I32),
    "h3enc_encode": ([_P, _P, _P, _P, _P, _I32, _I32, _P, _I32, _I32, _P, _P], _I32),
    "h3enc_encode_embeds": ([_P, _P, _I32, _I32, _P, _P, _P, _I32, _I32, _P, _I32, _I32, _P, _P], _I32),
    "h3enc_encode_multimodal": ([_P, _P, _P, _P, _P, _P, _I32, _I32, _P, _I32, _I32, _P, _P], _I32),
    "h3enc_encode_host": ([_P, _P, _P, _P, _P, _I32, _I32, _P, _I32, _I32, _P, _P], _I32),
    "h3enc_set_layer_capture": ([_P, ctypes.POINTER(_P), _I32], _I32),
    "h3enc_get_status": ([_P], _I32),
    "h3enc_last_error": ([_P], ctypes.c_char_p),
    "h3enc_destroy": ([_P], None),
    "h3enc_set_profiling": ([_P, _I32], _I32),
    "h3enc_set_profiling_classes": ([_P, ctypes.c_uint32], _I32),
    "h3enc_set_profiling_layer": ([_P, _I32], _I32),
    "h3enc_get_profile": ([_P, ctypes.POINTER(ctypes.c_double), ctypes.POINTER(_I64), _I32], _I32),
    "h3enc_launch_count": ([_P], _I64),
    "h3enc_num_sms": ([_P], _I32),
    "h3enc_set_graphs": ([_P, _I32], _I32),
    "h3enc_graph_count": ([_P], _I32),
    "h3enc_op_gemm": ([_P, _P, _P, _I32, _I32, _I32, _I32, _P, _P, _P, _I32, _P, _I64, _P, _P], _I32),
    "h3enc_op_gemm_workspace_bytes": ([], _I64),
    "h3enc_op_gemm_trace_next": ([_P, _I64], _I32),
    "h3enc_op_attention_trace_next": ([_P, _I64, _I32], _I32),
    "h3enc_build_positions": ([_P, _I32, _I32, _I32, _P, _I32, _P, _I32, _I32, _P, _P, _P, _P, _P, _P], _I32),
    "h3enc_aggregate_deepstack": ([_P, _I32, _P, _I32, _P, _I32, _I32, _I32, _P, _P], _I32),
    "h3enc_frontend_last_error": ([], ctypes.c_char_p),
    "h3enc_op_gemm_noalloc": ([_P, _P, _P, _I32, _I32, _I32, _I32, _P, _P, _P, _I32, _P, _P], _I32),
    "h3enc_op_gemm_noalloc_scratch_bytes": ([], _I64),
    "h3enc_op_gemm_noalloc_last_error": ([], ctypes.c_char_p),
    "h3enc_op_pack_gate_up": ([_P, _P, _P, _I32, _I32, _P], _I32),
    "h3enc_op_rmsnorm": ([_P, _P, _P, _I32, _I32, _F, _P], _I32),
    "h3enc_op_gemm_fp8": ([_P, _P, _P, _P, _P, _I32, _I32, _I32, _I32, _P, _P, _P, _I32, _P, _I64, _P, _P], _I32),
    "h3enc_op_quant_rows": ([_P, _I32, _I32, _P, _P, _P], _I32),
    "h3enc_op_wait_probe": ([_P, ctypes.c_uint32, _I32, _P, _P], _I32),
    "h3enc_op_rmsnorm_q8": ([_P, _P, _P, _P, _I32, _I32, _F, _P], _I32),
    "h3enc_op_rope_table": ([_P, _I32, _I32, _F, ctypes.POINTER(_I32), _P, _P, _P], _I32),
    "h3enc_op_rope_table_ex": ([_P, _I32, _I32, _F, ctypes.POINTER(_I32), _I32, _P, _P, _P], _I32),
    "h3enc_op_gemm_qkv_rope_ex": ([_P, _P, _P, _I32, _I32, _I32, _I32, _I32, _P, _P, _F, _P, _P, _I32, _P, _F, _P,
                                   _I64, _P, _P], _I32),
    "h3enc_op_gemm_qkv_rope_rms": ([_P, _P, _P, _I32, _I32, _I32, _I32, _I32, _P, _P, _F, _P, _P, _P, _F, _P, _I64,
                                    _P, _P], _I32),
    "h3enc_op_gemm_rms": ([_P, _P, _P, _I32, _I32, _I32, _I32, _P, _P, _P, _F, _P, _I64, _P, _P], _I32),
    "h3enc_op_row_sumsq": ([_P, _I32, _I32, _P, _P], _I32),
    "h3enc_op_fold_cols": ([_P, _I32, _I32, _P, _P], _I32),
    "h3enc_op_gemm_qkv_rope": ([_P, _P, _P, _I32, _I32, _I32, _I32, _I32, _P, _P, _F, _P, _P, _P, _I64, _P, _P],
                               _I32),
    "h3enc_op_attention": ([_P, _P, _I32, _I32, _I32, _I32, _P, _I32, _P], _I32),
    "h3enc_op_embed": ([_P, _P, _I32, _I32, _P, _I32, _P, _P], _I32),
    "h3enc_op_vis_rank": ([_P, _I32, _I32, _P, _P, _P], _I32),
    "h3enc_op_layernorm": ([_P, _P, _P, _P, _I32, _I32, _F, _P], _I32),
    "h3enc_op_vision_pos_embed": ([_P, _I32, _I32, _P, _I32, _I32, _P, _P], _I32),
    "h3enc_op_vision_rope_table": ([_P, _I32, _I32, _I32, _F, _P, _P, _P], _I32),
    "h3enc_op_gemm_bias": ([_P, _P, _P, _I32, _I32, _I32, _I32, _P, _P, _P, _I64, _P, _P], _I32),
    "h3enc_op_gemm_qkv_rope_bias": ([_P, _P, _P, _I32, _I32, _I32, _I32, _P, _P, _P, _P, _I64, _P, _P], _I32),
    "h3enc_op_attention_bidir": ([_P, _P, _I32, _I32, _I32, _P, _I32, _P], _I32),
    "h3enc_op_attention_bidir_ws": ([_P, _P, _I32, _I32, _I32, _P, _I32, _P, _I64, _P], _I32),
    "h3enc_op_attention_workspace_bytes": ([_I32], _I64),
    "h3vis_create": ([ctypes.POINTER(VisionConfig), ctypes.POINTER(_P)], _I32),
    "h3vis_load_weights": ([_P, ctypes.c_char_p, _P, _I32, ctypes.POINTER(_I64), _I32, _I32], _I32),
    "h3vis_finalize_weights": ([_P], _I32),
    "h3vis_encode": ([_P, _P, _I32, _P, _I32, _P, _P, _P], _I32),
    "h3vis_get_status": ([_P], _I32),
    "h3vis_last_error": ([_P], ctypes.c_char_p),
    "h3vis_launch_count": ([_P], _I64),
    "h3vis_destroy": ([_P], None),
}
for _name, (_args, _res) in _SIGS.items():
    _fn = getattr(lib, _name)
    _fn.argtypes = _args
    _fn.restype = _res


# ---------------------------------------------------------------- marshalling helpers

def _ptr(t):
    """Device/host address of a tensor, an int address, or None."""
    if t is None:
        return None
    if isinstance(t, int):
        return t
    return t.data_ptr()


def _stream(stream):
    if stream is None:
        import torch
        return torch.cuda.current_stream().cuda_stream
    return stream if isinstance(stream, int) else stream.cuda_stream


def _host_i32(a):
    """ctypes int32 array from a sequence (HOST cu_seqlens / sections)."""
    if a is None:
        return None
    vals = [int(x) for x in a]
    return (ctypes.c_int32 * len(vals))(*vals)


def _check(code, handle=None):
    if code not in (0, 1):
        msg = lib.h3enc_last_error(handle)
        raise H3encError(code, msg.decode() if msg else "")
    return code


# ---------------------------------------------------------------- C-named calls

def h3enc_create(cfg: Config):
    h = _P()
    _check(lib.h3enc_create(ctypes.byref(cfg), ctypes.byref(h)))
    return h.value


def h3enc_load_weights(h, name: str, tensor, data_on_device: bool = True):
    shape = (_I64 * tensor.dim())(*tensor.shape)
    return _check(lib.h3enc_load_weights(h, name.encode(), _ptr(tensor), 0, shape, tensor.dim(),
                                         1 if data_on_device else 0), h)


def h3enc_finalize_weights(h):
    return _check(lib.h3enc_finalize_weights(h), h)


def h3enc_encode(h, input_ids, positions, visual_mask, deepstack, num_deepstack, n_vis, cu_seqlens, seq_len,
                 out, stream=None):
    cu = _host_i32(cu_seqlens)
    n_seqs = len(cu) - 1 if cu is not None else 0
    return _check(lib.h3enc_encode(h, _ptr(input_ids), _ptr(positions), _ptr(visual_mask), _ptr(deepstack),
                                   num_deepstack, n_vis, cu, n_seqs, seq_len, _ptr(out), _stream(stream)), h)


def h3enc_encode_multimodal(h, input_ids, positions, visual_mask, visual_embeds, deepstack, num_deepstack, n_vis,
                            cu_seqlens, seq_len, out, stream=None):
    cu = _host_i32(cu_seqlens)
    n_seqs = len(cu) - 1 if cu is not None else 0
    return _check(lib.h3enc_encode_multimodal(h, _ptr(input_ids), _ptr(positions), _ptr(visual_mask),
                                              _ptr(visual_embeds), _ptr(deepstack), num_deepstack, n_vis, cu,
                                              n_seqs, seq_len, _ptr(out), _stream(stream)), h)


def h3enc_encode_embeds(h, inputs_embeds, layer_begin, layer_end, positions, visual_mask, deepstack,
                        num_deepstack, n_vis, cu_seqlens, seq_len, out, stream=None):
    cu = _host_i32(cu_seqlens)
    n_seqs = len(cu) - 1 if cu is not None else 0
    return _check(lib.h3enc_encode_embeds(h, _ptr(inputs_embeds), layer_begin, layer_end, _ptr(positions),
                                          _ptr(visual_mask), _ptr(deepstack), num_deepstack, n_vis, cu, n_seqs,
                                          seq_len, _ptr(out), _stream(stream)), h)


def h3enc_encode_host(h, input_ids, positions, visual_mask, deepstack, num_deepstack, n_vis, cu_seqlens, seq_len,
                      out, stream=None):
    cu = _host_i32(cu_seqlens)
    n_seqs = len(cu) - 1 if cu is not None else 0
    return _check(lib.h3enc_encode_host(h, _ptr(input_ids), _ptr(positions), _ptr(visual_mask), _ptr(deepstack),
                                        num_deepstack, n_vis, cu, n_seqs, seq_len, _ptr(out), _stream(stream)), h)


def h3enc_build_positions(input_ids, image_token_id, video_token_id, image_grid_thw=None, video_grid_thw=None,
                          spatial_merge_size=2):
    """Host arrays in, (positions int32 [3,S], visual_mask uint8 [S], visual_kind uint8 [S],
    n_image_tokens, n_video_tokens, mrope_delta) out."""
    import numpy as np
    ids = np.ascontiguousarray(input_ids, dtype=np.int32)
    S = ids.shape[0]
    img = None if image_grid_thw is None else np.ascontiguousarray(image_grid_thw, dtype=np.int32).reshape(-1, 3)
    vid = None if video_grid_thw is None else np.ascontiguousarray(video_grid_thw, dtype=np.int32).reshape(-1, 3)
    pos = np.zeros((3, S), dtype=np.int32)
    mask = np.zeros(S, dtype=np.uint8)
    kind = np.zeros(S, dtype=np.uint8)
    ni, nv, delta = ctypes.c_int32(), ctypes.c_int32(), ctypes.c_int32()
    code = lib.h3enc_build_positions(ids.ctypes.data, S, image_token_id, video_token_id,
                                     None if img is None else img.ctypes.data, 0 if img is None else len(img),
                                     None if vid is None else vid.ctypes.data, 0 if vid is None else len(vid),
                                     spatial_merge_size, pos.ctypes.data, mask.ctypes.data, kind.ctypes.data,
                                     ctypes.byref(ni), ctypes.byref(nv), ctypes.byref(delta))
    if code != 0:
        raise H3encError(code, lib.h3enc_frontend_last_error().decode())
    return pos, mask, kind, ni.value, nv.value, delta.value


def h3enc_aggregate_deepstack(visual_kind, image_feats, video_feats, out, stream=None):
    """visual_kind: host uint8 [S]; feats/out: device bf16 [levels, n, hidden] tensors (or None)."""
    import numpy as np
    kind = np.ascontiguousarray(visual_kind, dtype=np.uint8)
    levels, _, hidden = out.shape
    ni = 0 if image_feats is None else int(image_feats.shape[1])
    nv = 0 if video_feats is None else int(video_feats.shape[1])
    code = lib.h3enc_aggregate_deepstack(kind.ctypes.data, kind.shape[0], _ptr(image_feats), ni, _ptr(video_feats),
                                         nv, levels, hidden, _ptr(out), _stream(stream))
    if code != 0:
        raise H3encError(code, lib.h3enc_frontend_last_error().decode())
    return code


def h3enc_set_layer_capture(h, tensors):
    ptrs = (_P * len(tensors))(*[_ptr(t) for t in tensors]) if tensors else None
    return _check(lib.h3enc_set_layer_capture(h, ptrs, len(tensors) if tensors else 0), h)


def h3enc_get_status(h):
    return lib.h3enc_get_status(h)


def h3enc_last_error(h=None) -> str:
    m = lib.h3enc_last_error(h)
    return m.decode() if m else ""


def h3enc_destroy(h):
    lib.h3enc_destroy(h)


def h3enc_set_profiling(h, enable: bool):
    return _check(lib.h3enc_set_profiling(h, 1 if enable else 0), h)


def h3enc_set_profiling_classes(h, classes):
    """Time only the named kernel classes (see KERNEL_CLASSES); [] turns profiling off."""
    mask = 0
    for c in classes:
        mask |= 1 << KERNEL_CLASSES.index(c)
    return _check(lib.h3enc_set_profiling_classes(h, mask), h)


def h3enc_set_profiling_layer(h, layer: int):
    """Time only the given decoder layer's launches (-1: all)."""
    return _check(lib.h3enc_set_profiling_layer(h, layer), h)


def h3enc_get_profile(h):
    n = len(KERNEL_CLASSES)
    ms = (ctypes.c_double * n)()
    cnt = (_I64 * n)()
    _check(lib.h3enc_get_profile(h, ms, cnt, n), h)
    return {k: (ms[i], cnt[i]) for i, k in enumerate(KERNEL_CLASSES)}


def h3enc_launch_count(h) -> int:
    return lib.h3enc_launch_count(h)


def h3enc_num_sms(h) -> int:
    return lib.h3enc_num_sms(h)


def h3enc_set_graphs(h, enable):
    """Let h3enc_encode_host capture and replay one CUDA graph per call shape (default on)."""
    _check(lib.h3enc_set_graphs(h, 1 if enable else 0), h)


def h3enc_graph_count(h) -> int:
    return lib.h3enc_graph_count(h)


def h3enc_op_gemm(A, W, C, M, N, K, epilogue, R=None, DS=None, vis_rank=None, n_vis=0, workspace=None,
                  status=None, stream=None):
    wbytes = 0 if workspace is None else workspace.numel() * workspace.element_size()
    return _check(lib.h3enc_op_gemm(_ptr(A), _ptr(W), _ptr(C), M, N, K, epilogue, _ptr(R), _ptr(DS),
                                    _ptr(vis_rank), n_vis, _ptr(workspace), wbytes, _ptr(status), _stream(stream)))


def h3enc_op_gemm_trace_next(trace):
    """Arm the phase timeline of the next GEMM this thread launches: `trace` is a device int64
    tensor of >= 11 * SMs entries; CTA c writes its 11 stamps (ns) to trace[11c : 11c + 11]."""
    _check(lib.h3enc_op_gemm_trace_next(_ptr(trace), trace.numel()))


def h3enc_op_attention_trace_next(trace, ctas):
    """Arm the per-CTA timeline of the next attention launch on this thread: `trace` is a device
    int64 tensor of >= 9 * ctas entries (ctas = heads * query tiles of 128 rows)."""
    _check(lib.h3enc_op_attention_trace_next(_ptr(trace), trace.numel(), ctas))


def h3enc_op_gemm_workspace_bytes() -> int:
    return lib.h3enc_op_gemm_workspace_bytes()


def h3enc_op_gemm_noalloc(A, W, C, M, N, K, epilogue, R=None, DS=None, vis_rank=None, n_vis=0, status=None,
                          stream=None):
    """h3enc_op_gemm without a workspace argument, for callers that cannot allocate device
    memory: the library's fixed device scratch array is used instead (shared by every call)."""
    code = lib.h3enc_op_gemm_noalloc(_ptr(A), _ptr(W), _ptr(C), M, N, K, epilogue, _ptr(R), _ptr(DS),
                                     _ptr(vis_rank), n_vis, _ptr(status), _stream(stream))
    if code != 0:
        msg = lib.h3enc_op_gemm_noalloc_last_error()
        raise H3encError(code, msg.decode() if msg else "")
    return code


def h3enc_op_gemm_noalloc_scratch_bytes() -> int:
    return lib.h3enc_op_gemm_noalloc_scratch_bytes()


def h3enc_op_pack_gate_up(gate, up, W, I, K, stream=None):
    return _check(lib.h3enc_op_pack_gate_up(_ptr(gate), _ptr(up), _ptr(W), I, K, _stream(stream)))


def h3enc_op_gemm_fp8(A, W, sa, sw, C, M, N, K, epilogue, R=None, DS=None, vis_rank=None, n_vis=0, workspace=None,
                      status=None, stream=None):
    """e4m3 projection: C = epilogue((A * sa) (W * sw)^T); A [M,K] and W [N,K] uint8 e4m3 bytes,
    sa [M] and sw [N] float32."""
    wbytes = 0 if workspace is None else workspace.numel() * workspace.element_size()
    return _check(lib.h3enc_op_gemm_fp8(_ptr(A), _ptr(W), _ptr(sa), _ptr(sw), _ptr(C), M, N, K, epilogue, _ptr(R),
                                        _ptr(DS), _ptr(vis_rank), n_vis, _ptr(workspace), wbytes, _ptr(status),
                                        _stream(stream)))


def h3enc_op_quant_rows(x, rows, cols, q, scale, stream=None):
    return _check(lib.h3enc_op_quant_rows(_ptr(x), rows, cols, _ptr(q), _ptr(scale), _stream(stream)))


def h3enc_op_rmsnorm_q8(x, w, q, scale, rows, cols, eps, stream=None):
    return _check(lib.h3enc_op_rmsnorm_q8(_ptr(x), _ptr(w), _ptr(q), _ptr(scale), rows, cols, eps, _stream(stream)))


def h3enc_op_wait_probe(flag, expect, use_mbarrier, status, stream=None):
    """Bounded-wait self-test: waits for *flag == expect (or on an mbarrier nobody completes);
    a timeout ORs 1 into the device int32 `status`."""
    return _check(lib.h3enc_op_wait_probe(_ptr(flag), expect, 1 if use_mbarrier else 0, _ptr(status),
                                          _stream(stream)))


def h3enc_op_rmsnorm(x, w, y, rows, cols, eps, stream=None):
    return _check(lib.h3enc_op_rmsnorm(_ptr(x), _ptr(w), _ptr(y), rows, cols, eps, _stream(stream)))


def h3enc_op_rope_table(positions, S, head_dim, theta, section, cos_tab, sin_tab, stream=None):
    return _check(lib.h3enc_op_rope_table(_ptr(positions), S, head_dim, theta, _host_i32(section), _ptr(cos_tab),
                                          _ptr(sin_tab), _stream(stream)))


def h3enc_op_rope_table_ex(positions, S, head_dim, theta, section, stride, cos_tab, sin_tab, stream=None):
    return _check(lib.h3enc_op_rope_table_ex(_ptr(positions), S, head_dim, theta, _host_i32(section), stride,
                                             _ptr(cos_tab), _ptr(sin_tab), _stream(stream)))


def h3enc_op_gemm_qkv_rope_ex(A, W, C, M, K, n_heads, n_kv_heads, head_dim, w_q, w_k, eps, cos_tab, sin_tab,
                              cs_stride, ss_in=None, in_eps=0.0, workspace=None, status=None, stream=None):
    wbytes = 0 if workspace is None else workspace.numel() * workspace.element_size()
    return _check(lib.h3enc_op_gemm_qkv_rope_ex(_ptr(A), _ptr(W), _ptr(C), M, K, n_heads, n_kv_heads, head_dim,
                                                _ptr(w_q), _ptr(w_k), eps, _ptr(cos_tab), _ptr(sin_tab), cs_stride,
                                                _ptr(ss_in), in_eps, _ptr(workspace), wbytes, _ptr(status),
                                                _stream(stream)))


def h3enc_op_gemm_qkv_rope(A, W, C, M, K, n_heads, n_kv_heads, head_dim, w_q, w_k, eps, cos_tab, sin_tab,
                           workspace=None, status=None, stream=None):
    wbytes = 0 if workspace is None else workspace.numel() * workspace.element_size()
    return _check(lib.h3enc_op_gemm_qkv_rope(_ptr(A), _ptr(W), _ptr(C), M, K, n_heads, n_kv_heads, head_dim,
                                             _ptr(w_q), _ptr(w_k), eps, _ptr(cos_tab), _ptr(sin_tab),
                                             _ptr(workspace), wbytes, _ptr(status), _stream(stream)))


def h3enc_op_gemm_qkv_rope_rms(A, W, C, M, K, n_heads, n_kv_heads, head_dim, w_q, w_k, eps, cos_tab, sin_tab,
                               ss_in, in_eps, workspace=None, status=None, stream=None):
    wbytes = 0 if workspace is None else workspace.numel() * workspace.element_size()
    return _check(lib.h3enc_op_gemm_qkv_rope_rms(_ptr(A), _ptr(W), _ptr(C), M, K, n_heads, n_kv_heads, head_dim,
                                                 _ptr(w_q), _ptr(w_k), eps, _ptr(cos_tab), _ptr(sin_tab),
                                                 _ptr(ss_in), in_eps, _ptr(workspace), wbytes, _ptr(status),
                                                 _stream(stream)))


def h3enc_op_gemm_rms(A, W, C, M, N, K, epilogue, R=None, ss_in=None, ss_out=None, eps=0.0, workspace=None,
                      status=None, stream=None):
    wbytes = 0 if workspace is None else workspace.numel() * workspace.element_size()
    return _check(lib.h3enc_op_gemm_rms(_ptr(A), _ptr(W), _ptr(C), M, N, K, epilogue, _ptr(R), _ptr(ss_in),
                                        _ptr(ss_out), eps, _ptr(workspace), wbytes, _ptr(status), _stream(stream)))


def h3enc_op_row_sumsq(x, rows, cols, ss, stream=None):
    return _check(lib.h3enc_op_row_sumsq(_ptr(x), rows, cols, _ptr(ss), _stream(stream)))


def h3enc_op_fold_cols(W, rows, cols, gamma, stream=None):
    return _check(lib.h3enc_op_fold_cols(_ptr(W), rows, cols, _ptr(gamma), _stream(stream)))


def h3enc_op_attention(qkv, o, S, n_heads, n_kv_heads, head_dim, cu_seqlens=None, stream=None):
    cu = _host_i32(cu_seqlens)
    n_seqs = len(cu) - 1 if cu is not None else 0
    return _check(lib.h3enc_op_attention(_ptr(qkv), _ptr(o), S, n_heads, n_kv_heads, head_dim, cu, n_seqs,
                                         _stream(stream)))


def h3enc_op_embed(ids, table, vocab, hidden, out, S, status=None, stream=None):
    return _check(lib.h3enc_op_embed(_ptr(ids), _ptr(table), vocab, hidden, _ptr(out), S, _ptr(status),
                                     _stream(stream)))


def h3enc_op_vis_rank(mask, S, n_vis, vis_rank, status=None, stream=None):
    return _check(lib.h3enc_op_vis_rank(_ptr(mask), S, n_vis, _ptr(vis_rank), _ptr(status), _stream(stream)))


def _vcheck(code, handle=None):
    if code not in (0, 1):
        msg = lib.h3vis_last_error(handle)
        raise H3encError(code, msg.decode() if msg else "")
    return code


def h3enc_op_layernorm(x, w, b, y, rows, cols, eps, stream=None):
    return _check(lib.h3enc_op_layernorm(_ptr(x), _ptr(w), _ptr(b), _ptr(y), rows, cols, eps, _stream(stream)))


def _grids(grid_thw):
    g = [int(v) for row in grid_thw for v in row]
    return (ctypes.c_int32 * len(g))(*g), len(g) // 3


def h3enc_op_vision_pos_embed(table, grid_side, hidden, grid_thw, merge, out, stream=None):
    g, n = _grids(grid_thw)
    return _check(lib.h3enc_op_vision_pos_embed(_ptr(table), grid_side, hidden, g, n, merge, _ptr(out),
                                                _stream(stream)))


def h3enc_op_vision_rope_table(grid_thw, merge, head_dim, theta, cos_tab, sin_tab, stream=None):
    g, n = _grids(grid_thw)
    return _check(lib.h3enc_op_vision_rope_table(g, n, merge, head_dim, theta, _ptr(cos_tab), _ptr(sin_tab),
                                                 _stream(stream)))


def h3enc_op_gemm_bias(A, W, C, M, N, K, epilogue, bias, R=None, workspace=None, status=None, stream=None):
    wbytes = 0 if workspace is None else workspace.numel() * workspace.element_size()
    return _check(lib.h3enc_op_gemm_bias(_ptr(A), _ptr(W), _ptr(C), M, N, K, epilogue, _ptr(R), _ptr(bias),
                                         _ptr(workspace), wbytes, _ptr(status), _stream(stream)))


def h3enc_op_gemm_qkv_rope_bias(A, W, C, M, K, heads, head_dim, bias, cos_tab, sin_tab, workspace=None,
                                status=None, stream=None):
    wbytes = 0 if workspace is None else workspace.numel() * workspace.element_size()
    return _check(lib.h3enc_op_gemm_qkv_rope_bias(_ptr(A), _ptr(W), _ptr(C), M, K, heads, head_dim, _ptr(bias),
                                                  _ptr(cos_tab), _ptr(sin_tab), _ptr(workspace), wbytes,
                                                  _ptr(status), _stream(stream)))


def h3enc_op_attention_bidir(qkv, o, S, heads, head_dim, cu_seqlens=None, stream=None):
    cu = _host_i32(cu_seqlens)
    n_seqs = len(cu) - 1 if cu is not None else 0
    return _check(lib.h3enc_op_attention_bidir(_ptr(qkv), _ptr(o), S, heads, head_dim, cu, n_seqs, _stream(stream)))


def h3enc_op_attention_workspace_bytes(head_dim):
    return int(lib.h3enc_op_attention_workspace_bytes(head_dim))


def h3enc_op_attention_bidir_ws(qkv, o, S, heads, head_dim, workspace, cu_seqlens=None, stream=None):
    cu = _host_i32(cu_seqlens)
    n_seqs = len(cu) - 1 if cu is not None else 0
    wbytes = workspace.numel() * workspace.element_size()
    return _check(lib.h3enc_op_attention_bidir_ws(_ptr(qkv), _ptr(o), S, heads, head_dim, cu, n_seqs,
                                                  _ptr(workspace), wbytes, _stream(stream)))


def h3vis_create(cfg: VisionConfig):
    h = _P()
    code = lib.h3vis_create(ctypes.byref(cfg), ctypes.byref(h))
    if code != 0:
        raise H3encError(code, lib.h3vis_last_error(None).decode())
    return h


def h3vis_load_weights(h, name: str, tensor, data_on_device: bool = True):
    shape = (_I64 * tensor.dim())(*tensor.shape)
    return _vcheck(lib.h3vis_load_weights(h, name.encode(), _ptr(tensor), 0, shape, tensor.dim(),
                                          1 if data_on_device else 0), h)


def h3vis_finalize_weights(h):
    return _vcheck(lib.h3vis_finalize_weights(h), h)


def h3vis_encode(h, pixel_values, n_patches, grid_thw, embeds_out, deepstack_out=None, stream=None):
    g, n = _grids(grid_thw)
    return _vcheck(lib.h3vis_encode(h, _ptr(pixel_values), n_patches, g, n, _ptr(embeds_out), _ptr(deepstack_out),
                                    _stream(stream)), h)


def h3vis_get_status(h):
    return lib.h3vis_get_status(h)


def h3vis_last_error(h) -> str:
    m = lib.h3vis_last_error(h)
    return m.decode() if m else ""


def h3vis_launch_count(h) -> int:
    return lib.h3vis_launch_count(h)


def h3vis_destroy(h):
    lib.h3vis_destroy(h)


# ---------------------------------------------------------------- convenience wrappers

class VisionEncoder:
    """Owns one h3vis handle (the vision tower).  ``model`` is any object with the
    vision config attributes (depth, hidden, num_heads, intermediate, in_channels,
    patch_size, temporal_patch_size, spatial_merge_size, out_hidden,
    num_position_embeddings, deepstack_visual_indexes, ln_eps, rope_theta)."""

    def __init__(self, model, max_patches: int):
        c = VisionConfig()
        for f in ("depth", "hidden", "num_heads", "intermediate", "in_channels", "patch_size",
                  "temporal_patch_size", "spatial_merge_size", "out_hidden", "num_position_embeddings",
                  "ln_eps", "rope_theta"):
            setattr(c, f, getattr(model, f))
        idx = list(model.deepstack_visual_indexes)
        c.num_deepstack = len(idx)
        c.deepstack_indexes = (ctypes.c_int32 * 8)(*(idx + [0] * (8 - len(idx))))
        c.max_patches = max_patches
        self.model = model
        self.handle = h3vis_create(c)

    def load(self, name, tensor):
        return h3vis_load_weights(self.handle, name, tensor, tensor.is_cuda)

    def finalize(self):
        return h3vis_finalize_weights(self.handle)

    def encode(self, pixel_values, grid_thw, embeds_out, deepstack_out=None, stream=None):
        return h3vis_encode(self.handle, pixel_values, int(pixel_values.shape[0]), grid_thw, embeds_out,
                            deepstack_out, stream)

    def status(self) -> int:
        return h3vis_get_status(self.handle)

    def close(self):
        if self.handle:
            h3vis_destroy(self.handle)
            self.handle = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass


class Encoder:
    """Owns one h3enc handle.  ``model`` is any object with the Qwen3-VL text
    config attributes (num_layers, hidden, n_heads, n_kv_heads, head_dim,
    intermediate, vocab, rms_eps, rope_theta, mrope_section)."""

    def __init__(self, model, max_tokens: int, max_seqs: int = 64, num_deepstack: int = 3, fp8: bool = False,
                 separate_norm: bool = False):
        c = Config()
        c.num_layers, c.hidden, c.n_heads = model.num_layers, model.hidden, model.n_heads
        c.n_kv_heads, c.head_dim, c.intermediate = model.n_kv_heads, model.head_dim, model.intermediate
        c.vocab, c.rms_eps, c.rope_theta = model.vocab, model.rms_eps, model.rope_theta
        c.mrope_section = (ctypes.c_int32 * 3)(*model.mrope_section)
        c.max_tokens, c.max_seqs, c.num_deepstack = max_tokens, max_seqs, num_deepstack
        c.linear_fp8 = 1 if fp8 else 0
        c.separate_norm = 1 if separate_norm else 0
        self.model = model
        self.handle = h3enc_create(c)

    def load(self, name, tensor):
        return h3enc_load_weights(self.handle, name, tensor, tensor.is_cuda)

    def finalize(self):
        return h3enc_finalize_weights(self.handle)

    def encode(self, input_ids, positions, out, visual_mask=None, deepstack=None, n_vis=0, cu_seqlens=None,
               stream=None):
        nds = 0 if deepstack is None else int(deepstack.shape[0])
        return h3enc_encode(self.handle, input_ids, positions, visual_mask, deepstack, nds, n_vis, cu_seqlens,
                            int(positions.shape[1]), out, stream)

    def encode_embeds(self, inputs_embeds, positions, out, layer_begin=0, layer_end=None, visual_mask=None,
                      deepstack=None, n_vis=0, cu_seqlens=None, stream=None):
        nds = 0 if deepstack is None else int(deepstack.shape[0])
        le = self.model.num_layers if layer_end is None else layer_end
        return h3enc_encode_embeds(self.handle, inputs_embeds, layer_begin, le, positions, visual_mask, deepstack,
                                   nds, n_vis, cu_seqlens, int(positions.shape[1]), out, stream)

    def status(self):
        return h3enc_get_status(self.handle)

    def close(self):
        if self.handle:
            h3enc_destroy(self.handle)
            self.handle = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass
