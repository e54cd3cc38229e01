"""An encode captured into a CUDA graph and replayed on new inputs gives, bit for
bit, what an eager encode gives on the same inputs.  One full-width layer at 512
tokens, so every projection has a stream-K tail: its release flags must get a new
epoch on every replay (the epoch lives in device memory, not in the captured
launch parameters)."""
import pytest

import workloads as W
from _harness import make_encoder

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu

import qwen3_vl_text_gb300 as Q  # noqa: E402


@pytest.mark.parametrize("fp8", [False, True])
def test_encode_replayed_from_a_cuda_graph_matches_eager(fp8):
    wl = W.workload(1)
    cfg = wl.model
    inp = W.gen_inputs(wl)
    S, H = inp["seq_len"], cfg.hidden
    enc = make_encoder(wl, cfg, max_tokens=S, fp8=fp8)
    try:
        pos = torch.from_numpy(inp["positions"]).cuda()
        x_in = torch.empty(S, H, dtype=torch.bfloat16, device="cuda")
        y_out = torch.empty(S, H, dtype=torch.bfloat16, device="cuda")
        inputs = [W.bf16_bits_to_torch(W.normal_bf16(80 + i, "graph_x", (S, H))).cuda() for i in range(3)]

        def encode(x, out):
            Q.h3enc_encode_embeds(enc.handle, x, 0, cfg.num_layers, pos, None, None, 0, 0, None, S, out,
                                  stream=torch.cuda.current_stream())

        eager = []
        for x in inputs:
            o = torch.empty_like(y_out)
            encode(x, o)
            eager.append(o)
        torch.cuda.synchronize()
        x_in.copy_(inputs[0])
        side = torch.cuda.Stream()
        side.wait_stream(torch.cuda.current_stream())
        with torch.cuda.stream(side):
            encode(x_in, y_out)               # warm the launch paths on the capture stream
        torch.cuda.current_stream().wait_stream(side)
        torch.cuda.synchronize()
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g):
            encode(x_in, y_out)
        for rep in range(2):
            for x, want in zip(inputs, eager):
                x_in.copy_(x)
                g.replay()
                torch.cuda.synchronize()
                assert torch.equal(y_out, want), f"replay {rep} differs from the eager encode"
        assert enc.status() == 0, Q.h3enc_last_error(enc.handle)
    finally:
        enc.close()


def test_profiled_graph_replays_time_the_gate_up_launches():
    """Profiling events captured with the encode are graph nodes: after the replays the
    gate/up class reports one duration per layer (the latest replay), the output stays
    the eager one, and the classes not profiled report nothing."""
    wl = W.workload(0)
    cfg = wl.model
    inp = W.gen_inputs(wl)
    S, H = inp["seq_len"], cfg.hidden
    enc = make_encoder(wl, cfg, max_tokens=S)
    try:
        pos = torch.from_numpy(inp["positions"]).cuda()
        x = W.bf16_bits_to_torch(W.normal_bf16(90, "graph_x", (S, H))).cuda()
        want = torch.empty(S, H, dtype=torch.bfloat16, device="cuda")
        got = torch.empty_like(want)
        side = torch.cuda.Stream()

        def encode(out, stream):
            Q.h3enc_encode_embeds(enc.handle, x, 0, cfg.num_layers, pos, None, None, 0, 0, None, S, out,
                                  stream=stream)

        encode(want, torch.cuda.current_stream())
        side.wait_stream(torch.cuda.current_stream())
        encode(got, side)
        torch.cuda.synchronize()
        Q.h3enc_set_profiling_classes(enc.handle, ["gemm_gate_up"])
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=side):
            encode(got, side)
        got.zero_()
        for _ in range(3):
            g.replay()
        torch.cuda.synchronize()
        prof = Q.h3enc_get_profile(enc.handle)
        assert torch.equal(got, want)
        ms, n = prof["gemm_gate_up"]
        assert n == cfg.num_layers and ms > 0.0
        assert all(v[0] == 0.0 for k, v in prof.items() if k != "gemm_gate_up")
        assert enc.status() == 0, Q.h3enc_last_error(enc.handle)
    finally:
        enc.close()


def test_profiling_one_layer_times_one_launch_per_encode():
    wl = W.workload(0)
    cfg = wl.model
    inp = W.gen_inputs(wl)
    S, H = inp["seq_len"], cfg.hidden
    enc = make_encoder(wl, cfg, max_tokens=S)
    try:
        pos = torch.from_numpy(inp["positions"]).cuda()
        x = W.bf16_bits_to_torch(W.normal_bf16(91, "graph_x", (S, H))).cuda()
        out = torch.empty(S, H, dtype=torch.bfloat16, device="cuda")
        Q.h3enc_set_profiling_classes(enc.handle, ["gemm_gate_up", "gemm_down"])
        Q.h3enc_set_profiling_layer(enc.handle, cfg.num_layers - 1)
        for _ in range(3):
            Q.h3enc_encode_embeds(enc.handle, x, 0, cfg.num_layers, pos, None, None, 0, 0, None, S, out)
        prof = Q.h3enc_get_profile(enc.handle)
        assert prof["gemm_gate_up"][1] == 3 and prof["gemm_down"][1] == 3
        assert prof["gemm_gate_up"][0] > 0 and prof["gemm_qkv"] == (0.0, 0)
        with pytest.raises(Q.H3encError):
            Q.h3enc_set_profiling_layer(enc.handle, cfg.num_layers)
        Q.h3enc_set_profiling_layer(enc.handle, -1)
        Q.h3enc_set_profiling_classes(enc.handle, [])
        assert enc.status() == 0
    finally:
        enc.close()
