"""The multimodal front end on the GPU: image + video DeepStack aggregation
(bit-exact row placement) and the encode with vision-merger rows replacing the
placeholder embeddings, driven from token ids through the host position builder."""
import dataclasses

import numpy as np
import pytest

import oracle as O
import workloads as W
from _harness import GPU_STORAGE, bits_to_f32, make_encoder, oracle_layer_getter, t2f, parity

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu

import qwen3_vl_text_gb300 as Q  # noqa: E402

IMG, VID = 151655, 151656


def test_aggregate_deepstack_interleaves_images_and_videos():
    H, levels = 256, 3
    kind = np.array([0] * 3 + [1] * 5 + [0] * 2 + [2] * 4 + [1] * 3 + [2] * 2 + [0], dtype=np.uint8)
    ni, nv = int((kind == 1).sum()), int((kind == 2).sum())
    img_bits = W.normal_bf16(60, "img", (levels, ni, H))
    vid_bits = W.normal_bf16(61, "vid", (levels, nv, H))
    out = torch.empty(levels, ni + nv, H, dtype=torch.bfloat16, device="cuda")
    Q.h3enc_aggregate_deepstack(kind, W.bf16_bits_to_torch(img_bits).cuda(), W.bf16_bits_to_torch(vid_bits).cuda(),
                                out)
    torch.cuda.synchronize()
    mask, expect = O.frontend.aggregate_deepstack(kind, bits_to_f32(img_bits), bits_to_f32(vid_bits))
    assert np.array_equal(mask, kind != 0)
    assert np.array_equal(t2f(out), expect)          # a copy: bit-exact


def _tiny_ids_with_placeholders():
    wl = W.workload(0)
    inp = W.gen_inputs(wl)
    ids = inp["input_ids"].copy()
    ids[inp["visual_mask"] == 1] = IMG      # the 1x4x8 LLM grid = an 8x16 image grid before a 2x2 merge
    return wl, inp, ids


def test_multimodal_encode_from_ids_against_oracle():
    wl, inp, ids = _tiny_ids_with_placeholders()
    cfg = dataclasses.replace(wl.model, vocab=152000)   # the placeholder ids must be valid rows
    pos, mask, kind, ni, nv, _ = Q.h3enc_build_positions(ids, IMG, VID, image_grid_thw=[[1, 8, 16]])
    assert np.array_equal(pos, inp["positions"]) and ni == 32
    S, H = len(ids), cfg.hidden
    vis_bits = W.normal_bf16(62, "visual_embeds", (ni, H), 0.0, 0.05)
    ds_bits = W.normal_bf16(63, "ds_img", (1, ni, H), 0.0, 0.1)
    enc = make_encoder(wl, cfg, max_tokens=64)
    try:
        dev_ids = torch.from_numpy(ids).cuda()
        dev_pos = torch.from_numpy(pos).cuda()
        dev_mask = torch.from_numpy(mask).cuda()
        ve = W.bf16_bits_to_torch(vis_bits).cuda()
        ds = torch.empty(1, ni, H, dtype=torch.bfloat16, device="cuda")
        Q.h3enc_aggregate_deepstack(kind, W.bf16_bits_to_torch(ds_bits).cuda(), None, ds)
        out = torch.empty(S, H, dtype=torch.bfloat16, device="cuda")
        Q.h3enc_encode_multimodal(enc.handle, dev_ids, dev_pos, dev_mask, ve, ds, 1, ni, None, S, out)
        assert enc.status() == 0
        # the same call with the token embeddings as "visual embeddings" is the plain encode, bit for bit
        tok = W.bf16_bits_to_torch(W.gen_weight(wl.seed, W.embed_name(), (cfg.vocab, H), 0.0, 0.02,
                                                rows=ids[mask == 1])).cuda()
        a = torch.empty_like(out)
        b = torch.empty_like(out)
        Q.h3enc_encode_multimodal(enc.handle, dev_ids, dev_pos, dev_mask, tok, ds, 1, ni, None, S, a)
        Q.h3enc_encode(enc.handle, dev_ids, dev_pos, dev_mask, ds, 1, ni, None, S, b)
        torch.cuda.synchronize()
        assert torch.equal(a, b)
        got = t2f(out)
    finally:
        enc.close()
    x0 = bits_to_f32(W.gen_weight(wl.seed, W.embed_name(), (cfg.vocab, H), 0.0, 0.02, rows=ids))
    x0 = O.frontend.masked_scatter_rows(x0, O.frontend.placeholder_rows(ids, IMG), bits_to_f32(vis_bits))
    get = oracle_layer_getter(wl, cfg)
    ws = [get(l) for l in range(cfg.num_layers)]
    dsf = bits_to_f32(ds_bits)
    ref = O.forward(x0, pos, cfg, ws.__getitem__, mask, dsf)
    refbf = O.forward(x0, pos, cfg, ws.__getitem__, mask, dsf, storage=GPU_STORAGE)
    ok, msg = parity("multimodal encode from ids", got, ref, refbf, 2e-2, 0.05)
    assert ok, msg
