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
