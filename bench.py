"""Benchmark: 50-layer Qwen3-VL text-decoder prefill, seq 1024 (128 text + a
1x24x32 image grid + 128 text, DeepStack after layers 0-2), on one GB300.

One step = one full encode (embedding gather, M-RoPE tables, 50 decoder layers)
of one sequence.  Prints ONE JSON line on rank 0:
  value     encoded tokens/s over the whole job, device-timed, inputs resident in HBM
  e2e       the same metric through h3enc_encode_host (host buffers, copies timed)
  roofline  the gate/up projection GEMM (the largest kernel) against measured dense bf16 peak
  cpu_baseline  the CPU oracle on a bounded sample of the same workload
N > 1 (torchrun): every rank encodes its own sequence with its own weight copy
(replicas, no collective on the data path); timing is max over ranks.
``--impl reference`` times the CPU oracle (the reference arm of this tier).
"""
from __future__ import annotations

import argparse
import json
import os
import subprocess
import sys
import threading
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

WORKLOAD_ID = 2
GEMM_GU_CLASS = "gemm_gate_up"
# DRAM bytes (read + write) of one gate/up launch at seq 1024, from an ncu capture of this
# kernel source (dram__bytes_read.sum + dram__bytes_write.sum).
GATE_UP_TRAFFIC_BYTES = 609.4e6
# NVIDIA's dense (no 2:4 sparsity) bf16 tensor rate for one GB300, TFLOP/s: context for the
# measured peaks, which are the denominators of the fractions.
NOMINAL_DENSE_BF16_TFLOPS = 2250.0


def _peaks():
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as f:
            p = json.load(f)
        return float(p["bf16_tflops"]), float(p["bf16_tflops_sustained"]), float(p["hbm_gbs"]), "measured"
    except Exception:
        return 1900.0, 1700.0, 6800.0, "fallback"


def encode_flops(cfg, cu) -> float:
    """Algorithmic FLOPs of one encode: linears 2*S*params + causal attention 4*nq*d*sum L(L+1)/2, per layer."""
    h, d = cfg.hidden, cfg.head_dim
    lin = h * cfg.qkv_out + cfg.n_heads * d * h + 3 * h * cfg.intermediate
    s = int(cu[-1])
    pairs = sum((int(b) - int(a)) * (int(b) - int(a) + 1) // 2 for a, b in zip(cu[:-1], cu[1:]))
    return float(cfg.num_layers) * (2.0 * s * lin + 4.0 * cfg.n_heads * d * pairs)


class Clocks:
    """nvidia-smi samples of SM clock and throttle reasons during the timed region."""
    Q = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.hw_slowdown,"
         "clocks_event_reasons.hw_thermal_slowdown,clocks_event_reasons.sw_thermal_slowdown,"
         "clocks_event_reasons.sw_power_cap")

    def __init__(self, index: int):
        self.index = index
        self.rows = []
        self.proc = None
        self.thread = None

    def start(self):
        try:
            self.proc = subprocess.Popen(["nvidia-smi", "-i", str(self.index), "--query-gpu=" + self.Q,
                                          "--format=csv,noheader,nounits", "-lms", "200"],
                                         stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except Exception:
            self.proc = None
            return
        self.thread = threading.Thread(target=self._read, daemon=True)
        self.thread.start()

    def _read(self):
        for line in self.proc.stdout:
            self.rows.append([x.strip() for x in line.split(",")])

    def stop(self):
        if self.proc is None:
            return None
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except Exception:
            self.proc.kill()
        if self.thread:
            self.thread.join(timeout=2)
        sm = []
        mx = 0.0
        reasons = set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for r in self.rows:
            try:
                sm.append(float(r[1]))
                mx = max(mx, float(r[2]))
                for i, n in enumerate(names):
                    if r[4 + i].lower().startswith("active"):
                        reasons.add(n)
            except Exception:
                pass
        if not sm:
            return None
        sm.sort()
        return {"sm_mhz": sm[len(sm) // 2], "sm_max_mhz": mx, "reasons": sorted(reasons), "samples": len(sm)}


def job_throughput(local_ms: float, units_per_rank: int, steps: int, dist=None, device=None):
    """Whole-job rate of N independent replicas: every rank processed `units_per_rank`
    units per step; the job took as long as its slowest rank (max over ranks).
    Returns (units per second over all ranks, max milliseconds)."""
    ms = float(local_ms)
    world = 1
    if dist is not None and dist.is_initialized():
        import torch
        world = dist.get_world_size()
        t = torch.tensor([ms], dtype=torch.float64, device=device)
        dist.all_reduce(t, op=dist.ReduceOp.MAX)
        ms = float(t.item())
    return world * units_per_rank * steps / (ms / 1e3), ms


class CpuOracleSample:
    """The CPU oracle on the first `layers` decoder layers of the workload: weights drawn once
    (outside any clock), then `run()` returns the seconds one pass takes."""

    def __init__(self, wl, inp, layers):
        import oracle as O
        import workloads as W
        self.O, self.wl, self.inp, self.layers = O, wl, inp, layers
        cfg = wl.model
        if inp["input_ids"] is not None:
            self.x0 = O.bf16_bits_to_float(W.gen_weight(wl.seed, W.embed_name(), (cfg.vocab, cfg.hidden), 0.0, 0.02,
                                                        rows=inp["input_ids"]))
        else:   # a hidden-state input (the one-layer workload)
            self.x0 = O.bf16_bits_to_float(inp["inputs_embeds"])
        self.ds = None if inp["deepstack"] is None else O.bf16_bits_to_float(inp["deepstack"])
        self.mask = inp["visual_mask"] if inp["n_vis"] else None
        self.weights = [O.layer_weights_from_bits({n: W.gen_weight(wl.seed, n, s, m, sg)
                                                   for n, s, m, sg in W.layer_weight_specs(cfg, l)})
                        for l in range(layers)]

    def run(self) -> float:
        t0 = time.perf_counter()
        self.O.forward(self.x0, self.inp["positions"], self.wl.model, lambda l: self.weights[l],
                       self.mask, self.ds, layers=range(self.layers))
        return time.perf_counter() - t0


REF_LAYERS_PER_STEP = 4

# the oracle timed on whole small workloads: (workload id, name)
ORACLE_TIMED = ((0, "tiny_2layer_48tok"), (1, "one_full_layer_512tok"))


def oracle_time(args):
    """One workload through the CPU oracle in this process (its BLAS threads fixed by the caller's
    environment): prints {"seconds": [...], "tokens": S}."""
    import workloads as W
    wl = W.workload(args.oracle_time)
    inp = W.gen_inputs(wl)
    sample = CpuOracleSample(wl, inp, wl.model.num_layers)
    for _ in range(args.warm):
        sample.run()
    ts = [sample.run() for _ in range(args.reps)]
    print(json.dumps({"seconds": ts, "tokens": int(inp["seq_len"])}), flush=True)
    return 0


def oracle_config_timings():
    """The oracle on the tiny 2-layer workload and on one full-width layer at 512 tokens, with all
    host cores and with one thread (BLAS threads set before numpy loads, so each runs in a child
    process): median seconds, tokens/s and, for the full-width layer, GFLOP/s."""
    import workloads as W
    cores = os.cpu_count()
    out = {"cores": cores}
    for wid, name in ORACLE_TIMED:
        wl = W.workload(wid)
        inp = W.gen_inputs(wl)
        flops = encode_flops(wl.model, inp["cu_seqlens"])
        entry = {}
        for label, threads, reps, warm in (("all_cores", cores, 3, 1), ("one_thread", 1, 1, 0)):
            env = dict(os.environ, OMP_NUM_THREADS=str(threads), OPENBLAS_NUM_THREADS=str(threads),
                       MKL_NUM_THREADS=str(threads))
            r = subprocess.run([sys.executable, os.path.abspath(__file__), "--oracle-time", str(wid),
                                "--reps", str(reps), "--warm", str(warm)],
                               env=env, capture_output=True, text=True, timeout=600)
            if r.returncode != 0:
                raise RuntimeError("oracle timing failed: " + r.stderr[-400:])
            d = json.loads(r.stdout.strip().splitlines()[-1])
            ts = sorted(d["seconds"])
            t = ts[len(ts) // 2]
            entry[label] = {"threads": threads, "seconds": t, "tokens_per_s": d["tokens"] / t,
                            "gflops": flops / t / 1e9}
        out[name] = entry
    return out


def workload_config(wl, inp, world) -> dict:
    """The `config` object of both arms' lines: what the workload is, nothing about how it ran."""
    return {"workload": wl.name, "seq_len": int(inp["seq_len"]), "layers": wl.model.num_layers,
            "hidden": wl.model.hidden, "deepstack_levels": wl.deepstack_levels,
            "parallelism": f"replicas x{world}",
            "l2": "no flush: inputs larger than L2 (every step streams each layer's 975 MB of weights)"}


def run_reference(args):
    """The oracle arm: each step runs the first REF_LAYERS_PER_STEP decoder layers of the workload on
    the host cores (a bounded sample of the encode); `ms_per_step` is that measured time, and `value`
    scales it to the 50-layer encode the metric names."""
    rank = int(os.environ.get("RANK", "0"))
    if rank != 0:
        return 0
    import workloads as W
    wl = W.workload(WORKLOAD_ID)
    inp = W.gen_inputs(wl)
    S = inp["seq_len"]
    sample = CpuOracleSample(wl, inp, REF_LAYERS_PER_STEP)
    for _ in range(args.warmup):
        sample.run()
    ts = [sample.run() for _ in range(args.steps)]
    per_step = sum(ts) / len(ts)
    scale = wl.model.num_layers / REF_LAYERS_PER_STEP
    per_encode = per_step * scale
    v = S / per_encode
    cores = os.cpu_count()
    line = {"metric": "encoded tokens/s, 50-layer seq-1024 encode", "value": v, "unit": "tokens/s",
            "impl": "reference", "n_gpus": args.gpus, "steps": args.steps, "warmup": args.warmup,
            "ms_per_step": per_step * 1e3, "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
            "dtype": "f32", "data": "synthetic (seeded random-init weights and inputs)",
            "config": workload_config(wl, inp, 1),
            "layers_timed_per_step": REF_LAYERS_PER_STEP,
            "value_extrapolated_from_layers": REF_LAYERS_PER_STEP,
            "value_note": f"value = seq_len / (ms_per_step x {scale:g}): each step times "
                          f"{REF_LAYERS_PER_STEP} of the {wl.model.num_layers} layers",
            "ms_per_encode_extrapolated": per_encode * 1e3,
            "cpu_baseline": {"value": v, "unit": "tokens/s", "cores": cores, "kind": "oracle",
                             "sample": f"first {REF_LAYERS_PER_STEP} of 50 decoder layers per step (seq 1024), "
                                       f"time x{wl.model.num_layers / REF_LAYERS_PER_STEP:g}"},
            "e2e": {"value": v, "unit": "tokens/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)
    return 0


def run_kernel(args):
    """One kernel of the seq-1024 workload alone, device-timed (for ncu captures and tuning).
    Prints one JSON line with the average launch time and the achieved rate."""
    import numpy as np
    import torch

    import qwen3_vl_text_gb300 as Q
    import workloads as W
    wl = W.workload(WORKLOAD_ID)
    cfg = wl.model
    S = args.seq
    H, I, d, nq, nkv = cfg.hidden, cfg.intermediate, cfg.head_dim, cfg.n_heads, cfg.n_kv_heads
    dev = "cuda"

    def rnd(name, shape, sigma=0.02):
        return W.normal_bf16(7, name, shape, 0.0, sigma, device=dev)

    name = args.kernel
    if name == "gemm_qkv":
        A = rnd("A", (S, H), 1.0)
        Wt = rnd("W", (cfg.qkv_out, H))
        G = rnd("g", (d,), 1.0)
        pos = torch.arange(S, dtype=torch.int32, device=dev).repeat(3, 1).contiguous()
        # the encoder's table layout: row-interleaved, rows padded to a multiple of 32
        stride = (S + 31) // 32 * 32
        c = torch.empty(stride * d // 2, device=dev)
        s_ = torch.empty_like(c)
        Q.h3enc_op_rope_table_ex(pos, S, d, cfg.rope_theta, cfg.mrope_section, stride, c, s_)
        C = torch.empty(S, cfg.qkv_out, dtype=torch.bfloat16, device=dev)
        ws = torch.zeros(Q.h3enc_op_gemm_workspace_bytes(), dtype=torch.uint8, device=dev)
        ss = None
        if args.fold:   # the input RMSNorm folded in: rows scaled by the statistics of A
            ss = torch.empty(H // 128, S, dtype=torch.float32, device=dev)
            Q.h3enc_op_row_sumsq(A, S, H, ss)
        fn = lambda: Q.h3enc_op_gemm_qkv_rope_ex(A, Wt, C, S, H, nq, nkv, d, G, G, 1e-6, c, s_, stride, ss_in=ss,
                                                 in_eps=1e-6, workspace=ws)
        work, unit = 2.0 * S * cfg.qkv_out * H / 1e12, "TFLOP/s"
    elif name.startswith("gemm_"):
        shapes = {"gemm_o": (H, nq * d, Q.EPI_RESIDUAL),
                  "gemm_gate_up": (2 * I, H, Q.EPI_SWIGLU), "gemm_down": (H, I, Q.EPI_RESIDUAL)}
        N, K, epi = shapes[name]
        A = rnd("A", (S, K), 1.0)
        Wt = rnd("W", (N, K))
        C = torch.empty(S, N // 2 if epi == Q.EPI_SWIGLU else N, dtype=torch.bfloat16, device=dev)
        R = C if epi == Q.EPI_RESIDUAL else None
        ws = torch.zeros(Q.h3enc_op_gemm_workspace_bytes(), dtype=torch.uint8, device=dev)
        if args.fp8:
            # e4m3 operands with per-row scales, quantised once outside the timed launches
            A8 = torch.empty(S, K, dtype=torch.uint8, device=dev)
            W8 = torch.empty(N, K, dtype=torch.uint8, device=dev)
            sa = torch.empty(S, dtype=torch.float32, device=dev)
            sw = torch.empty(N, dtype=torch.float32, device=dev)
            Q.h3enc_op_quant_rows(A, S, K, A8, sa)
            Q.h3enc_op_quant_rows(Wt, N, K, W8, sw)
            fn = lambda: Q.h3enc_op_gemm_fp8(A8, W8, sa, sw, C, S, N, K, epi, R=R, workspace=ws)
        elif args.fold and epi == Q.EPI_SWIGLU:   # consumer of the post-attention statistics
            ss = torch.empty(K // 128, S, dtype=torch.float32, device=dev)
            Q.h3enc_op_row_sumsq(A, S, K, ss)
            fn = lambda: Q.h3enc_op_gemm_rms(A, Wt, C, S, N, K, epi, ss_in=ss, eps=1e-6, workspace=ws)
        elif args.fold:   # producer of the next norm's statistics
            ss = torch.empty(N // 128, S, dtype=torch.float32, device=dev)
            fn = lambda: Q.h3enc_op_gemm_rms(A, Wt, C, S, N, K, epi, R=R, ss_out=ss, workspace=ws)
        else:
            fn = lambda: Q.h3enc_op_gemm(A, Wt, C, S, N, K, epi, R=R, workspace=ws)
        work, unit = 2.0 * S * N * K / 1e12, "TFLOP/s"
    elif name == "attention":
        X = rnd("qkv", (S, cfg.qkv_out), 1.0)
        O_ = torch.empty(S, nq * d, dtype=torch.bfloat16, device=dev)
        fn = lambda: Q.h3enc_op_attention(X, O_, S, nq, nkv, d)
        work, unit = 4.0 * nq * d * S * (S + 1) / 2 / 1e12, "TFLOP/s"
    elif name == "rmsnorm":   # x read, y written, gamma read (algorithmic bytes)
        X = rnd("x", (S, H), 1.0)
        G = rnd("g", (H,), 1.0)
        Y = torch.empty_like(X)
        fn = lambda: Q.h3enc_op_rmsnorm(X, G, Y, S, H, 1e-6)
        work, unit = (2.0 * S * H * 2 + 2 * H) / 1e9, "GB/s"
    elif name == "rmsnorm_q8":   # the FP8 path's norm: x read, e4m3 rows + scales written
        X = rnd("x", (S, H), 1.0)
        G = rnd("g", (H,), 1.0)
        Y8 = torch.empty(S, H, dtype=torch.uint8, device=dev)
        sc = torch.empty(S, dtype=torch.float32, device=dev)
        fn = lambda: Q.h3enc_op_rmsnorm_q8(X, G, Y8, sc, S, H, 1e-6)
        work, unit = (S * H * 2 + 2 * H + S * H + 4 * S) / 1e9, "GB/s"
    elif name == "quant_rows":   # e4m3 quantisation of the SwiGLU output [S, I]: read bf16, write bytes
        X = rnd("act", (S, I), 1.0)
        Y8 = torch.empty(S, I, dtype=torch.uint8, device=dev)
        sc = torch.empty(S, dtype=torch.float32, device=dev)
        fn = lambda: Q.h3enc_op_quant_rows(X, S, I, Y8, sc)
        work, unit = (S * I * 2 + S * I + 4 * S) / 1e9, "GB/s"
    elif name == "row_sumsq":   # the folded norm's statistics of the layer input: x read, [H/128, S] written
        X = rnd("x", (S, H), 1.0)
        ss = torch.empty(H // 128, S, dtype=torch.float32, device=dev)
        fn = lambda: Q.h3enc_op_row_sumsq(X, S, H, ss)
        work, unit = (S * H * 2 + 4 * S * (H // 128)) / 1e9, "GB/s"
    elif name == "embed":   # gather of S rows of the 151936 x H table: ids read, rows read and written
        table = rnd("embed", (cfg.vocab, H))
        ids = torch.from_numpy(np.random.default_rng(5).integers(0, cfg.vocab, S).astype(np.int32)).cuda()
        Xo = torch.empty(S, H, dtype=torch.bfloat16, device=dev)
        fn = lambda: Q.h3enc_op_embed(ids, table, cfg.vocab, H, Xo, S)
        work, unit = (4 * S + 2.0 * S * H * 2) / 1e9, "GB/s"
    elif name == "layernorm":   # the vision tower's block norm: x [S, 1024] read, y written, w and b read
        D = W.VISION_FULL.hidden
        X = rnd("x", (S, D), 1.0)
        G = rnd("g", (D,), 1.0)
        B = rnd("b", (D,), 0.1)
        Y = torch.empty_like(X)
        fn = lambda: Q.h3enc_op_layernorm(X, G, B, Y, S, D, 1e-6)
        work, unit = (2.0 * S * D * 2 + 2 * 2 * D) / 1e9, "GB/s"
    elif name == "rope_table":   # positions read, fp32 cos/sin [S, d/2] written
        pos = torch.arange(S, dtype=torch.int32, device=dev).repeat(3, 1).contiguous()
        c = torch.empty(S, d // 2, device=dev)
        s_ = torch.empty_like(c)
        fn = lambda: Q.h3enc_op_rope_table(pos, S, d, cfg.rope_theta, cfg.mrope_section, c, s_)
        work, unit = (3 * 4 * S + 2 * 4 * S * (d // 2)) / 1e9, "GB/s"
    else:
        raise SystemExit("unknown kernel " + name)
    stream = torch.cuda.current_stream()
    for _ in range(args.warmup):
        fn()
    torch.cuda.synchronize()
    ts = []
    flush = torch.empty(256 << 20, dtype=torch.uint8, device=dev)   # 256 MB > L2 between launches
    timeline = args.timeline and (name.startswith("gemm_") or name == "attention")
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    per_cta = 9 if name == "attention" else 11
    trace = torch.zeros(sms * per_cta, dtype=torch.int64, device=dev) if timeline else None
    traces = []
    for _ in range(args.steps):
        flush.zero_()
        if timeline:
            trace.zero_()
        # ~100 us of device sleep: the host enqueues the launch meanwhile, so the start event
        # fires with the launch already queued and the time is the kernel's, not the host's
        torch.cuda._sleep(200_000)
        e0 = torch.cuda.Event(enable_timing=True)
        e1 = torch.cuda.Event(enable_timing=True)
        if timeline:
            if name == "attention":
                Q.h3enc_op_attention_trace_next(trace, sms)
            else:
                Q.h3enc_op_gemm_trace_next(trace)
        e0.record(stream)
        fn()
        e1.record(stream)
        torch.cuda.synchronize()
        ts.append(e0.elapsed_time(e1))
        if timeline:
            traces.append(trace.view(sms, per_cta).cpu().numpy().copy())
    ts.sort()
    ms = ts[len(ts) // 2]
    burst, sustained, hbm, src = _peaks()
    fp8_gemm = bool(args.fp8) and name.startswith("gemm_") and name != "gemm_qkv"
    # e4m3 contractions: the measured bf16 burst peak times the nominal fp8/bf16 ratio (4.5 / 2.25)
    peak = (burst * (2.0 if fp8_gemm else 1.0)) if unit == "TFLOP/s" else hbm
    print(json.dumps({"kernel": name + (" (e4m3)" if fp8_gemm else "") + (" (folded norm)" if args.fold else ""),
                      "seq": S, "ms_median": ms, "ms_min": ts[0], "achieved": work / (ms / 1e3),
                      "work_per_launch": work, "work_unit": "TFLOP" if unit == "TFLOP/s" else "GB",
                      "unit": unit, "peak": peak, "frac": work / (ms / 1e3) / peak,
                      "peak_source": f"{src} {'bf16_tflops' if unit == 'TFLOP/s' else 'hbm_gbs'} (burst)"
                                     + (" x 2 (nominal fp8/bf16)" if fp8_gemm else ""),
                      **({"timeline": kernel_timeline(name, traces)} if timeline else {})}),
          flush=True)
    return 0


def kernel_timeline(name, traces):
    """Medians over the timed launches of the kernel's own per-CTA stamps (µs from the first
    CTA's start; attention's middle stamps are SM cycles, reported as µs at each CTA's mean
    rate between its ns stamps)."""
    import numpy as np
    rows = []
    for t in traces:
        t = t.astype(np.int64)
        t = t[t[:, 0] > 0]
        t0 = t[:, 0].min()
        if name == "attention":
            dur = (t[:, 6] - t[:, 0]) / 1e3
            steps = t[:, 8].astype(np.float64)
            rows.append({"span_us": float(((t[:, 6] - t0) / 1e3).max()),
                         "cta_end_us_median": float(np.median((t[:, 6] - t0) / 1e3)),
                         "key_tiles_per_cta_median": float(np.median(steps)),
                         "us_per_key_tile_median": float(np.median(dur / np.maximum(steps, 1)))})
        else:
            rel = np.where(t > 0, (t - t0) / 1e3, np.nan)
            leaders = ~np.isnan(rel[:, 4])   # the CTAs that issue the MMAs (one per pair)
            rows.append({"span_us": float(np.nanmax(rel[:, 10])),
                         "ready_us_median": float(np.nanmedian(rel[:, 1])),
                         "first_mma_us_median": float(np.nanmedian(rel[leaders, 3])) if leaders.any() else None,
                         "split_acc_ready_us_median": (float(np.nanmedian(rel[:, 6]))
                                                       if not np.all(np.isnan(rel[:, 6])) else None),
                         "last_mma_us_median": float(np.nanmedian(rel[leaders, 4])) if leaders.any() else None,
                         "last_mma_us_min": float(np.nanmin(rel[leaders, 4])) if leaders.any() else None,
                         "last_mma_us_max": float(np.nanmax(rel[leaders, 4])) if leaders.any() else None,
                         "last_tile_epilogue_us_median": float(np.nanmedian(rel[:, 5] - rel[:, 2])),
                         "stream_k_reduce_done_us_max": (float(np.nanmax(rel[:, 9]))
                                                         if not np.all(np.isnan(rel[:, 9])) else None)})
    keys = rows[0].keys()
    return {k: (None if any(r[k] is None for r in rows) else float(np.median([r[k] for r in rows]))) for k in keys}


def vision_flops(cfg, grids) -> float:
    """Algorithmic FLOPs of one vision encode: patch embedding, per block the four linears
    (2 n (4 h^2 + 2 h I)) and bidirectional attention inside each frame (4 heads d L^2 per
    frame of L patches), and the mergers (2 (n/m^2) 4h (4h + out) each)."""
    h, I, m = cfg.hidden, cfg.intermediate, cfg.spatial_merge_size
    n = sum(t * hh * w for t, hh, w in grids)
    frames_sq = sum(t * (hh * w) ** 2 for t, hh, w in grids)
    mh, nm = h * m * m, n // (m * m)
    per_block = 2.0 * n * (4 * h * h + 2 * h * I) + 4.0 * cfg.num_heads * cfg.head_dim * frames_sq
    mergers = (1 + len(cfg.deepstack_visual_indexes)) * 2.0 * nm * mh * (mh + cfg.out_hidden)
    return 2.0 * n * cfg.patch_dim * h + cfg.depth * per_block + mergers


def run_vision(args):
    """The vision tower on one 48 x 64-patch image (the 24 x 32 merged grid of the seq-1024
    text workload), device-timed like the encode; one JSON line."""
    import torch

    import qwen3_vl_text_gb300 as Q
    import workloads as W
    wl = W.vision_workload(2)
    if args.images > 1:   # the same image size, several per encode (one attention segment each)
        import dataclasses
        wl = dataclasses.replace(wl, grids=wl.grids * args.images)
    cfg = wl.model
    inp = W.gen_vision_inputs(wl)
    n = inp["n_patches"]
    nm = n // cfg.spatial_merge_size ** 2
    enc = Q.VisionEncoder(cfg, max_patches=n)
    for name, shape, mean, sigma in W.vision_weight_specs(cfg):
        enc.load(name, W.gen_weight(wl.seed, name, shape, mean, sigma, device="cuda"))
    torch.cuda.synchronize()
    enc.finalize()
    px = W.bf16_bits_to_torch(inp["pixel_values"]).cuda()
    emb = torch.empty(nm, cfg.out_hidden, dtype=torch.bfloat16, device="cuda")
    ds = torch.empty(len(cfg.deepstack_visual_indexes), nm, cfg.out_hidden, dtype=torch.bfloat16, device="cuda")
    stream = torch.cuda.current_stream()

    def step():
        enc.encode(px, wl.grids, emb, ds, stream=stream)

    for _ in range(args.warmup):
        step()
    torch.cuda.synchronize()
    if enc.status() != 0:
        raise RuntimeError("vision status after warm-up: " + Q.h3vis_last_error(enc.handle))
    graph = None
    if not args.eager:
        # one tower encode captured into a CUDA graph and replayed once per step (as the text encode)
        cap = torch.cuda.Stream()
        cap.wait_stream(stream)
        n_cap = Q.h3vis_launch_count(enc.handle)
        graph = torch.cuda.CUDAGraph()
        with torch.cuda.graph(graph, stream=cap):
            enc.encode(px, wl.grids, emb, ds, stream=cap)
        launches_per_step = Q.h3vis_launch_count(enc.handle) - n_cap
        stream.wait_stream(cap)
        graph.replay()
        torch.cuda.synchronize()

    def run_step():
        if graph is not None:
            graph.replay()
        else:
            step()

    clocks = Clocks(int(os.environ.get("LOCAL_RANK", "0")))
    clocks.start()
    time.sleep(0.5)
    torch.cuda.synchronize()
    n0 = Q.h3vis_launch_count(enc.handle)
    e0 = torch.cuda.Event(enable_timing=True)
    e1 = torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    for _ in range(args.steps):
        run_step()
    e1.record(stream)
    torch.cuda.synchronize()
    clk = clocks.stop()
    ms = e0.elapsed_time(e1)
    launches = (launches_per_step * args.steps if graph is not None
                else Q.h3vis_launch_count(enc.handle) - n0)
    if enc.status() != 0:
        raise RuntimeError("vision status after the timed region: " + Q.h3vis_last_error(enc.handle))
    # end to end: pixels copied in from pinned host memory, embeddings and DeepStack features copied out
    h_px = W.bf16_bits_to_torch(inp["pixel_values"]).pin_memory()
    h_emb = torch.empty(emb.shape, dtype=torch.bfloat16).pin_memory()
    h_ds = torch.empty(ds.shape, dtype=torch.bfloat16).pin_memory()
    torch.cuda.synchronize()
    t0 = time.perf_counter()
    for _ in range(args.steps):
        px.copy_(h_px, non_blocking=True)
        run_step()
        h_emb.copy_(emb, non_blocking=True)
        h_ds.copy_(ds, non_blocking=True)
        torch.cuda.current_stream().synchronize()
    e2e_ms = (time.perf_counter() - t0) * 1e3
    burst, sustained, hbm, src = _peaks()
    base, base_name = burst, "bf16_tflops (burst)"   # the higher measured peak; see main()
    flops = vision_flops(cfg, wl.grids)
    tflops = flops * args.steps / (ms / 1e3) / 1e12
    line = {
        "metric": ("vision tower: merged visual tokens/s, " + ("one 48x64-patch image" if args.images == 1
                                                               else f"{args.images} 48x64-patch images per encode")),
        "value": nm * args.steps / (ms / 1e3),
        "unit": "tokens/s", "n_gpus": 1, "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms / args.steps,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "bf16",
        "data": "synthetic (seeded random-init weights and pixels)",
        "config": {"workload": wl.name, "patches": n, "merged_tokens": nm, "depth": cfg.depth, "hidden": cfg.hidden,
                   "heads": cfg.num_heads, "intermediate": cfg.intermediate, "deepstack": len(cfg.deepstack_visual_indexes),
                   "l2": "no flush: each step streams 0.91 GB of weights, far above the 129 MB L2",
                   "launch": "eager (one host launch per kernel)" if graph is None
                             else "CUDA graph of one tower encode, replayed once per step"},
        "images_per_s": args.images * args.steps / (ms / 1e3), "tflops": tflops, "pct_dense_bf16_peak": 100.0 * tflops / base,
        "pct_of_sustained_peak": 100.0 * tflops / sustained,
        "roofline": {"kernel": "whole tower (all launches of one encode)", "bound": "tensor", "achieved": tflops,
                     "peak": base, "unit": "TFLOP/s", "frac": tflops / base,
                     "peak_source": f"{src} {base_name}", "traffic": None},
        "gpu_launches": int(launches),
        "e2e": {"value": nm * args.steps / (e2e_ms / 1e3), "unit": "tokens/s", "h2d_bytes_per_step": int(h_px.numel() * 2),
                "d2h_bytes_per_step": int((h_emb.numel() + h_ds.numel()) * 2)},
        "clocks": clk,
    }
    enc.close()
    if not args.no_cpu_baseline and args.images == 1:
        import oracle as O
        ws = {nme[len("model.visual."):]: O.bf16_bits_to_float(W.gen_weight(wl.seed, nme, sh, mu, sg))
              for nme, sh, mu, sg in W.vision_weight_specs(cfg)}
        pxf = O.bf16_bits_to_float(inp["pixel_values"])
        t0 = time.perf_counter()
        O.vision.vision_forward(pxf, wl.grids, cfg, ws)
        t = time.perf_counter() - t0
        line["cpu_baseline"] = {"value": nm / t, "unit": "tokens/s", "cores": os.cpu_count(), "kind": "oracle",
                                "sample": "one whole tower forward on the same image"}
    print(json.dumps(line), flush=True)
    return 0


def run_multimodal(args):
    """The pages' whole multimodal encode per step: the vision tower on one 48x64-patch image,
    then the 50-layer text encode of the seq-1024 prompt whose 768 image placeholders take the
    tower's embeddings and whose first three layers take its DeepStack features."""
    import torch

    import qwen3_vl_text_gb300 as Q
    import workloads as W
    vw = W.vision_workload(2)
    tw = W.workload(WORKLOAD_ID)
    vcfg, cfg = vw.model, tw.model
    vin, tin = W.gen_vision_inputs(vw), W.gen_inputs(tw)
    S, n_vis = tin["seq_len"], tin["n_vis"]
    venc = Q.VisionEncoder(vcfg, max_patches=vin["n_patches"])
    for name, shape, mean, sigma in W.vision_weight_specs(vcfg):
        venc.load(name, W.gen_weight(vw.seed, name, shape, mean, sigma, device="cuda"))
    enc = Q.Encoder(cfg, max_tokens=S, max_seqs=4, num_deepstack=len(vcfg.deepstack_visual_indexes))
    for l in range(cfg.num_layers):
        for name, shape, mean, sigma in W.layer_weight_specs(cfg, l):
            enc.load(name, W.gen_weight(tw.seed, name, shape, mean, sigma, device="cuda"))
    enc.load(W.embed_name(), W.gen_weight(tw.seed, W.embed_name(), (cfg.vocab, cfg.hidden), 0.0, 0.02,
                                          device="cuda"))
    torch.cuda.synchronize()
    venc.finalize()
    enc.finalize()
    ids_h = tin["input_ids"].copy()
    ids_h[tin["visual_mask"] == 1] = 151655            # the image placeholder id
    ids_h[tin["visual_mask"] == 0] %= 151655
    ids = torch.from_numpy(ids_h).cuda()
    pos = torch.from_numpy(tin["positions"]).cuda()
    mask = torch.from_numpy(tin["visual_mask"]).cuda()
    px = W.bf16_bits_to_torch(vin["pixel_values"]).cuda()
    nds = len(vcfg.deepstack_visual_indexes)
    emb = torch.empty(n_vis, cfg.hidden, dtype=torch.bfloat16, device="cuda")
    ds = torch.empty(nds, n_vis, cfg.hidden, dtype=torch.bfloat16, device="cuda")
    out = torch.empty(S, cfg.hidden, dtype=torch.bfloat16, device="cuda")
    stream = torch.cuda.current_stream()

    def step():
        venc.encode(px, vw.grids, emb, ds, stream=stream)
        Q.h3enc_encode_multimodal(enc.handle, ids, pos, mask, emb, ds, nds, n_vis, None, S, out, stream)

    for _ in range(args.warmup):
        step()
    torch.cuda.synchronize()
    if enc.status() != 0 or venc.status() != 0:
        raise RuntimeError("device status after warm-up")
    clocks = Clocks(int(os.environ.get("LOCAL_RANK", "0")))
    clocks.start()
    time.sleep(0.5)
    torch.cuda.synchronize()
    l0 = Q.h3enc_launch_count(enc.handle) + Q.h3vis_launch_count(venc.handle)
    e0 = torch.cuda.Event(enable_timing=True)
    e1 = torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    for _ in range(args.steps):
        step()
    e1.record(stream)
    torch.cuda.synchronize()
    clk = clocks.stop()
    ms = e0.elapsed_time(e1)
    launches = Q.h3enc_launch_count(enc.handle) + Q.h3vis_launch_count(venc.handle) - l0
    if enc.status() != 0 or venc.status() != 0:
        raise RuntimeError("device status after the timed region")
    # end to end: pixels, ids, positions and mask copied in from pinned memory, the output copied out
    h_px = W.bf16_bits_to_torch(vin["pixel_values"]).pin_memory()
    h_ids = torch.from_numpy(ids_h).pin_memory()
    h_pos = torch.from_numpy(tin["positions"]).pin_memory()
    h_mask = torch.from_numpy(tin["visual_mask"]).pin_memory()
    h_out = torch.empty(S, cfg.hidden, dtype=torch.bfloat16).pin_memory()
    torch.cuda.synchronize()
    t0 = time.perf_counter()
    for _ in range(args.steps):
        px.copy_(h_px, non_blocking=True)
        ids.copy_(h_ids, non_blocking=True)
        pos.copy_(h_pos, non_blocking=True)
        mask.copy_(h_mask, non_blocking=True)
        step()
        h_out.copy_(out, non_blocking=True)
        stream.synchronize()
    e2e_ms = (time.perf_counter() - t0) * 1e3
    burst, sustained, hbm, src = _peaks()
    base, base_name = burst, "bf16_tflops (burst)"   # the higher measured peak; see main()
    flops = encode_flops(cfg, tin["cu_seqlens"]) + vision_flops(vcfg, vw.grids)
    tflops = flops * args.steps / (ms / 1e3) / 1e12
    line = {
        "metric": "multimodal encode (one 48x64-patch image + the seq-1024 prompt): encoded tokens/s",
        "value": S * args.steps / (ms / 1e3), "unit": "tokens/s", "n_gpus": 1, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": ms / args.steps, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "bf16", "data": "synthetic (seeded random-init weights, pixels and ids)",
        "config": {"workload": "vision-image-48x64 + " + tw.name, "seq_len": S, "visual_tokens": n_vis,
                   "launch": "eager (one host launch per kernel)"},
        "tflops": tflops, "pct_dense_bf16_peak": 100.0 * tflops / base,
        "pct_of_sustained_peak": 100.0 * tflops / sustained,
        "roofline": {"kernel": "whole step (vision tower + 50-layer text encode)", "bound": "tensor",
                     "achieved": tflops, "peak": base, "unit": "TFLOP/s", "frac": tflops / base,
                     "peak_source": f"{src} {base_name}", "traffic": None},
        "gpu_launches": int(launches),
        "e2e": {"value": S * args.steps / (e2e_ms / 1e3), "unit": "tokens/s",
                "h2d_bytes_per_step": int(h_px.numel() * 2 + h_ids.numel() * 4 + h_pos.numel() * 4 + h_mask.numel()),
                "d2h_bytes_per_step": int(h_out.numel() * 2)},
        "clocks": clk,
    }
    venc.close()
    enc.close()
    print(json.dumps(line), flush=True)
    return 0


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--kernel", default=None,
                    help="time one kernel alone: gemm_qkv (with the fused q/k norm + M-RoPE), gemm_o, "
                         "gemm_gate_up, gemm_down, attention, rmsnorm, rmsnorm_q8, quant_rows, row_sumsq, embed, "
                         "rope_table, layernorm (the vision tower's, 1024 columns; --seq 3072 for one 48x64 image)")
    ap.add_argument("--seq", type=int, default=1024)
    ap.add_argument("--workload", type=int, default=WORKLOAD_ID, choices=[2, 3, 4],
                    help="2: 50-layer seq-1024 image layout (the headline); 3: seq-8192 video layout; "
                         "4: 16 packed text prompts")
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--timeline", action="store_true",
                    help="with --kernel gemm_* or attention: add the kernel's per-CTA phase timeline")
    ap.add_argument("--separate-norm", action="store_true",
                    help="bf16: run each RMSNorm as its own kernel instead of folding it into the projections")
    ap.add_argument("--vision", action="store_true",
                    help="time the vision tower on one 48x64-patch image instead of the text encode")
    ap.add_argument("--images", type=int, default=1, help="with --vision: images per encode")
    ap.add_argument("--multimodal", action="store_true",
                    help="time the vision tower and the text encode together (one image + the seq-1024 prompt)")
    ap.add_argument("--oracle-time", type=int, default=None, help=argparse.SUPPRESS)
    ap.add_argument("--reps", type=int, default=3, help=argparse.SUPPRESS)
    ap.add_argument("--warm", type=int, default=1, help=argparse.SUPPRESS)
    ap.add_argument("--fold", action="store_true",
                    help="with --kernel: the projection as the folded-norm encode runs it (QKV and gate/up "
                         "scale rows by the norm statistics, o and down emit them)")
    ap.add_argument("--eager", action="store_true",
                    help="launch every kernel from the host in the timed region instead of replaying a "
                         "CUDA graph of the encode")
    ap.add_argument("--cpu-layers", type=int, default=8)
    ap.add_argument("--fp8", action="store_true",
                    help="online-FP8 linears (e4m3 weights per output channel, activations per token); "
                         "attention stays bf16.  Not the headline configuration, which is plain bf16.")
    args = ap.parse_args()
    args.warmup = max(3, args.warmup)
    if args.oracle_time is not None:
        return oracle_time(args)
    if args.vision:
        return run_vision(args)
    if args.multimodal:
        return run_multimodal(args)
    if args.kernel:
        return run_kernel(args)
    if args.impl == "reference":
        return run_reference(args)

    import numpy as np
    import torch

    import qwen3_vl_text_gb300 as Q
    import workloads as W

    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    torch.cuda.set_device(local)
    dist = None
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl")

    wl = W.workload(args.workload)
    headline = args.workload == WORKLOAD_ID
    cfg = wl.model
    inp = W.gen_inputs(wl)
    S = inp["seq_len"]
    cu = [int(x) for x in inp["cu_seqlens"]] if len(inp["cu_seqlens"]) > 2 else None
    n_vis = inp["n_vis"]
    enc = Q.Encoder(cfg, max_tokens=S, max_seqs=max(4, len(inp["cu_seqlens"]) - 1),
                    num_deepstack=max(1, wl.deepstack_levels), fp8=args.fp8, separate_norm=args.separate_norm)
    for l in range(cfg.num_layers):
        for name, shape, mean, sigma in W.layer_weight_specs(cfg, l):
            enc.load(name, W.gen_weight(wl.seed, name, shape, mean, sigma, device="cuda"))
    enc.load(W.embed_name(), W.gen_weight(wl.seed, W.embed_name(), (cfg.vocab, cfg.hidden), 0.0, 0.02,
                                          device="cuda"))
    torch.cuda.synchronize()
    enc.finalize()

    ids = torch.from_numpy(inp["input_ids"]).cuda()
    pos = torch.from_numpy(inp["positions"]).cuda()
    mask = torch.from_numpy(inp["visual_mask"]).cuda() if n_vis else None
    ds = W.bf16_bits_to_torch(inp["deepstack"]).cuda() if inp["deepstack"] is not None else None
    out = torch.empty(S, cfg.hidden, dtype=torch.bfloat16, device="cuda")
    stream = torch.cuda.current_stream()

    def step():
        enc.encode(ids, pos, out, visual_mask=mask, deepstack=ds, n_vis=n_vis, cu_seqlens=cu, stream=stream)

    for _ in range(args.warmup):
        step()
    torch.cuda.synchronize()
    if enc.status() != 0:
        raise RuntimeError("device status after warm-up: " + Q.h3enc_last_error(enc.handle))

    # timed region: events only around one gate/up GEMM per step (the roofline kernel, the middle
    # layer's launch: all 50 are the same work, and an event between two launches stops them
    # overlapping, so timing one disturbs the step far less than timing all)
    Q.h3enc_set_profiling_classes(enc.handle, [GEMM_GU_CLASS])
    Q.h3enc_set_profiling_layer(enc.handle, cfg.num_layers // 2)
    graph = None
    if not args.eager:
        # one encode captured into a CUDA graph (its gate/up event pairs included) and replayed
        # once per step: the same kernels, launched by the graph instead of the host
        cap = torch.cuda.Stream()
        cap.wait_stream(stream)
        enc.encode(ids, pos, out, visual_mask=mask, deepstack=ds, n_vis=n_vis, cu_seqlens=cu, stream=cap)  # warm
        torch.cuda.synchronize()
        Q.h3enc_set_profiling_classes(enc.handle, [GEMM_GU_CLASS])   # drop the warm-up's event pairs
        n_cap = Q.h3enc_launch_count(enc.handle)
        graph = torch.cuda.CUDAGraph()
        with torch.cuda.graph(graph, stream=cap):
            enc.encode(ids, pos, out, visual_mask=mask, deepstack=ds, n_vis=n_vis, cu_seqlens=cu, stream=cap)
        launches_per_step = Q.h3enc_launch_count(enc.handle) - n_cap
        stream.wait_stream(cap)
        graph.replay()
        torch.cuda.synchronize()
        if enc.status() != 0:
            raise RuntimeError("device status after the graph warm-up: " + Q.h3enc_last_error(enc.handle))
    clocks = Clocks(local)
    clocks.start()
    time.sleep(0.5)
    if dist:
        dist.barrier()
    torch.cuda.synchronize()
    n0 = Q.h3enc_launch_count(enc.handle)
    e0 = torch.cuda.Event(enable_timing=True)
    e1 = torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    for _ in range(args.steps):
        if graph is not None:
            graph.replay()
        else:
            step()
    e1.record(stream)
    torch.cuda.synchronize()
    if dist:
        dist.barrier()
    launches = (launches_per_step * args.steps if graph is not None
                else Q.h3enc_launch_count(enc.handle) - n0)
    clk = clocks.stop()
    ms = e0.elapsed_time(e1)
    prof_gu = Q.h3enc_get_profile(enc.handle)[GEMM_GU_CLASS]
    Q.h3enc_set_profiling_classes(enc.handle, [])
    Q.h3enc_set_profiling_layer(enc.handle, -1)
    value, ms = job_throughput(ms, S, args.steps, dist, "cuda")
    if enc.status() != 0:
        raise RuntimeError("device status after the timed region: " + Q.h3enc_last_error(enc.handle))

    # end to end through the host-buffer entry point: pinned inputs in, result out, every step.
    # Right after the timed region and for as many steps, so both see the same power state.
    h_ids = torch.from_numpy(inp["input_ids"]).pin_memory()
    h_pos = torch.from_numpy(inp["positions"]).pin_memory()
    h_mask = torch.from_numpy(inp["visual_mask"]).pin_memory() if n_vis else None
    h_ds = W.bf16_bits_to_torch(inp["deepstack"]).pin_memory() if ds is not None else None
    h_out = torch.empty(S, cfg.hidden, dtype=torch.bfloat16).pin_memory()

    host_stream = torch.cuda.Stream()   # a stream of its own: capturable, unlike the legacy default
    Q.h3enc_set_graphs(enc.handle, graph is not None)   # --eager: the host entry runs eagerly too
    torch.cuda.synchronize()

    def host_step():
        Q.h3enc_encode_host(enc.handle, h_ids, h_pos, h_mask, h_ds, 0 if h_ds is None else h_ds.shape[0], n_vis, cu,
                            S, h_out, host_stream)

    # the entry point runs a new call shape eagerly once, captures it on the second call and
    # replays the graph after that: both happen before the timed calls
    host_step()
    host_step()
    if dist:
        dist.barrier()
    t0 = time.perf_counter()
    e2e_steps = args.steps
    for _ in range(e2e_steps):
        host_step()
    e2e_value, e2e_ms = job_throughput((time.perf_counter() - t0) * 1e3, S, e2e_steps, dist, "cuda")
    h2d = (h_ids.numel() * 4 + h_pos.numel() * 4 + (0 if h_mask is None else h_mask.numel())
           + (0 if h_ds is None else h_ds.numel() * 2))
    d2h = h_out.numel() * 2

    # per-kernel breakdown: the same steps again with an event pair around every launch
    Q.h3enc_set_profiling(enc.handle, True)
    for _ in range(args.steps):
        step()
    prof = Q.h3enc_get_profile(enc.handle)
    Q.h3enc_set_profiling(enc.handle, False)

    burst, sustained, hbm, peak_src = _peaks()
    flops = encode_flops(cfg, inp["cu_seqlens"])
    gu_ms, gu_n = prof_gu
    gu_flops = 2.0 * S * (2 * cfg.intermediate) * cfg.hidden
    gu_achieved = gu_flops / (gu_ms / gu_n / 1e3) / 1e12 if gu_n else 0.0
    # The denominator is the measured burst cuBLAS figure (the higher of the two measured peaks, taken
    # at the maximum SM clock); the fractions of the sustained figure (measured under the power cap at
    # a lower clock) and of NVIDIA's nominal dense rate are reported beside it.  e4m3 contractions
    # take the bf16 figure times the nominal fp8/bf16 dense ratio (4.5 / 2.25).
    f8 = 2.0 if args.fp8 else 1.0
    gu_peak = burst * f8
    line = {
        "metric": (("encoded tokens/s, 50-layer seq-1024 encode" if headline else f"encoded tokens/s, {wl.name}")
                   + (", online FP8 linears" if args.fp8 else "")),
        "value": value, "unit": "tokens/s",
        "n_gpus": world, "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms / args.steps,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
        "dtype": "e4m3 linears, bf16 attention" if args.fp8 else "bf16",
        "data": "synthetic (seeded random-init weights and inputs)",
        "config": workload_config(wl, inp, world),
        "setup": {"sms": Q.h3enc_num_sms(enc.handle),
                  "launch": "eager (one host launch per kernel)" if graph is None
                            else "CUDA graph of one encode, replayed once per step",
                  "rmsnorm": "quantising pass before each projection" if args.fp8
                             else "separate pass before each projection" if args.separate_norm
                             else "folded into the projections (statistics from the o/down epilogues)"},
        "pct_dense_bf16_peak": 100.0 * flops * args.steps / (ms / 1e3) / (burst * 1e12),
        "pct_dense_bf16_peak_basis": f"{peak_src} bf16_tflops (burst cuBLAS, {burst:g} TFLOP/s)",
        "pct_of_sustained_peak": 100.0 * flops * args.steps / (ms / 1e3) / (sustained * 1e12),
        "pct_of_nominal_dense_bf16": 100.0 * flops * args.steps / (ms / 1e3) / (NOMINAL_DENSE_BF16_TFLOPS * 1e12),
        "tflops": flops * args.steps / (ms / 1e3) / 1e12,
        "roofline": {"kernel": "gemm_tcgen05 gate/up + SwiGLU" + (" (e4m3)" if args.fp8 else "")
                               + f", timed at layer {cfg.num_layers // 2} of every step", "bound": "tensor",
                     "achieved": gu_achieved, "peak": gu_peak, "unit": "TFLOP/s", "frac": gu_achieved / gu_peak,
                     "peak_source": f"{peak_src} bf16_tflops (burst)" + (" x 2 (nominal fp8/bf16)" if args.fp8 else ""),
                     "frac_of_sustained": gu_achieved / (sustained * f8),
                     "frac_of_nominal": gu_achieved / (NOMINAL_DENSE_BF16_TFLOPS * f8),
                     "traffic": None if args.fp8 or not headline else GATE_UP_TRAFFIC_BYTES},
        "kernel_ms_per_step": {k: v[0] / args.steps for k, v in prof.items()},
        "kernel_ms_note": "separate pass with an event pair around every launch",
        "gpu_launches": int(launches),
        "e2e": {"value": e2e_value, "unit": "tokens/s", "h2d_bytes_per_step": int(h2d),
                "d2h_bytes_per_step": int(d2h),
                "launch": "h3enc_encode_host: copies in, " + ("the call shape's CUDA graph replayed"
                                                              if graph is not None else "eager launches")
                          + ", copy out, sync"},
        "clocks": clk,
    }
    enc.close()
    if rank == 0 and world == 1 and not args.no_cpu_baseline and not args.fp8 and headline:
        t = CpuOracleSample(wl, inp, args.cpu_layers).run()
        per_encode = t / args.cpu_layers * cfg.num_layers
        line["cpu_baseline"] = {"value": S / per_encode, "unit": "tokens/s", "cores": os.cpu_count(),
                                "kind": "oracle",
                                "sample": f"first {args.cpu_layers} of 50 decoder layers at seq 1024, time scaled x"
                                          f"{cfg.num_layers / args.cpu_layers:g}",
                                "oracle_configs": oracle_config_timings()}
    if rank == 0:
        print(json.dumps(line), flush=True)
    if dist:
        dist.destroy_process_group()
    return 0


if __name__ == "__main__":
    sys.exit(main())
