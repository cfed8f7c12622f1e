#!/usr/bin/env python3
"""Benchmark of the TokenGate pruned-prefill hot path on B300.

One step = one pass of the whole path over one synthetic batch, inputs
resident in HBM: gate MLP scores -> top-K (question kept) -> gather of kept
rows/positions/scores -> the token-gated attention layers above the gate.
For the long-context workload (default) that is 27 layers, each
q/k/v projections -> RoPE + token-gated attention -> output projection with
the residual add; single-layer workloads run one attention layer on seeded
q/k/v.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--workload NAME]
    python bench.py --impl reference ...   (the CPU oracle, bounded sample)

Prints ONE JSON line (rank 0).  ``value`` is gated-attention TFLOP/s:
causal-triangle flops 2*hq*D*T(T+1) per layer over the measured attention
time, summed over ranks.  In the long-context stack RoPE is fused into the
Q/K/V projection, so that time is the attention kernel's; single-layer
workloads add their RoPE call.  ``gate_topk_gather`` gives the GB/s of the
first three steps on algorithmic bytes.  Every call is captured once in a
CUDA graph and replayed, so the device time excludes host launch cost;
``e2e`` instead runs the public Python API with host buffers (copies in the
timed region).  L2 is flushed before every timed step (256 MB written, then
256 MB read).  N > 1 runs independent replicas: the workload is one
sequence and the path has no exchange step.
"""
from __future__ import annotations

import argparse
import json
import os
import statistics
import subprocess
import sys
import threading
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import numpy as np  # noqa: E402

METRIC = "gated-attention TFLOP/s and ms/layer at 16k–128k; gate+top-K+gather GB/s"
UNIT = "TFLOP/s"
DEFAULT_WORKLOAD = "long-128k"


def load_peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        with open(p) as f:
            d = json.load(f)
        return {"hbm_gbs": d["hbm_gbs"], "bf16_tflops": d["bf16_tflops"],
                "bf16_tflops_sustained": d.get("bf16_tflops_sustained"), "source": "measured"}
    return {"hbm_gbs": 6400.0, "bf16_tflops": 1800.0, "bf16_tflops_sustained": 1400.0, "source": "fallback"}


def attention_flops(kept_lens, hq, d):
    """Causal-triangle flops of one layer: QK^T and PV, 2 flops per MAC,
    over the (i, j <= i) pairs: 2 * hq * D * T (T + 1) per sequence."""
    return float(sum(2.0 * hq * d * t * (t + 1) for t in kept_lens))


def path_bytes(shape):
    """Algorithmic HBM bytes of gate + top-K + gather: residuals read once
    (2 d per row), scores written and read (4 + 4 per row), kept ids
    written and read (4 + 4 per kept row), kept rows read and written
    (2 * 2 d per kept row), kept positions and scores written (8 per kept
    row)."""
    n, t, d = shape.n_rows, shape.n_kept, shape.d
    return float(n * 2 * d + n * 8 + t * 8 + t * 4 * d + t * 8)


def masked_path_bytes(shape, n_kept):
    """The same algorithmic bytes for the general prunable-span path, plus
    the mask read twice (counting and selecting, 1 + 1 per row); n_kept is
    that path's kept count."""
    n, d = shape.n_rows, shape.d
    return float(n * 2 * d + n * 8 + 2 * n + n_kept * 8 + n_kept * 4 * d + n_kept * 8)


def measure_masked(P, shape, flush, steps):
    """General prunable spans: the masked gate, top-K and gather on a seeded
    multi-span mask whose prunable share is the workload's document share
    (so the kept count stays close to the workload's), timed like the step:
    one CUDA graph with events between the three calls, L2 flushed first."""
    import torch
    from learned_token_pruning_09_b300 import synth
    tg = P.tg
    frac = float(sum(shape.n_doc)) / max(shape.n_rows, 1)
    mask_h = synth.prunable_spans(shape, frac=frac)
    mask = torch.as_tensor(mask_h).to(P.dev)
    max_len = int(np.diff(shape.cu_seqlens).max())
    kept = torch.empty(shape.n_rows, dtype=torch.int32, device=P.dev)
    cu_kept = torch.empty(shape.batch + 1, dtype=torch.int32, device=P.dev)
    n_prun = torch.empty(shape.batch, dtype=torch.int32, device=P.dev)
    s = torch.empty(shape.n_rows, dtype=torch.float32, device=P.dev)
    ev = [torch.cuda.Event(enable_timing=True, external=True) for _ in range(4)]

    def calls_plain(n_kept):
        tg.tg_gate_score_masked(P.X, mask, P.W1, None, P.W2, P.b2, s_out=s, cu_seqlens=P.cu, topk_ws=P.topk_ws)
        tg.tg_topk_select_masked(s, P.cu, mask, P.kk, max_len, kept_idx=kept, cu_kept=cu_kept, n_prunable=n_prun,
                                 workspace=P.topk_ws)
        tg.tg_gather_kept(P.X, s, P.cu, kept[:n_kept], cu_kept, n_kept, x_kept=P.xk_masked[:n_kept],
                          pos_kept=P.pos_masked[:n_kept], s_kept=P.s_masked[:n_kept])

    def calls(n_kept):
        ev[0].record()
        tg.tg_gate_score_masked(P.X, mask, P.W1, None, P.W2, P.b2, s_out=s, cu_seqlens=P.cu, topk_ws=P.topk_ws)
        ev[1].record()
        tg.tg_topk_select_masked(s, P.cu, mask, P.kk, max_len, kept_idx=kept, cu_kept=cu_kept, n_prunable=n_prun,
                                 workspace=P.topk_ws)
        ev[2].record()
        tg.tg_gather_kept(P.X, s, P.cu, kept[:n_kept], cu_kept, n_kept, x_kept=P.xk_masked[:n_kept],
                          pos_kept=P.pos_masked[:n_kept], s_kept=P.s_masked[:n_kept])
        ev[3].record()

    # the kept count is device data: learn it once, eagerly, then capture
    tg.tg_gate_score_masked(P.X, mask, P.W1, None, P.W2, P.b2, s_out=s)
    tg.tg_topk_select_masked(s, P.cu, mask, P.kk, max_len, kept_idx=kept, cu_kept=cu_kept, n_prunable=n_prun)
    n_kept = int(cu_kept[-1].item())
    P.xk_masked = torch.empty((n_kept, shape.d), dtype=torch.bfloat16, device=P.dev)
    P.pos_masked = torch.empty(n_kept, dtype=torch.int32, device=P.dev)
    P.s_masked = torch.empty(n_kept, dtype=torch.float32, device=P.dev)
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        calls(n_kept)
    per = []
    for i in range(3 + steps):
        flush()
        g.replay()
        torch.cuda.synchronize()
        if i >= 3:
            per.append([ev[k].elapsed_time(ev[k + 1]) for k in range(3)])
    if tg.tg_check_device_status() != tg.TG_OK:
        raise RuntimeError("device status after the masked path: " + tg.lib.tg_last_error_string().decode())
    per = np.array(per).mean(axis=0)
    us = time_calls([lambda: calls_plain(n_kept)], flush, steps)
    byts = masked_path_bytes(shape, n_kept)
    return {"us": us, "gbs": byts / (us * 1e-6) / 1e9, "bytes": byts, "n_kept": n_kept,
            "spans_per_seq": 4, "prunable_rows": int(mask_h.sum()),
            "gate_us": float(per[0]) * 1e3, "topk_us": float(per[1]) * 1e3, "gather_us": float(per[2]) * 1e3}


def measure_attn_bwd(P, shape, flush, steps):
    """The attention backward with respect to s, gain and tau (one layer:
    the step's last, with its own q', K cache, v and a forward o, lse), on a
    seeded upstream gradient dO ~ N(0, 1); one CUDA graph around the call, L2
    flushed before each replay.  Flops are the forward's (S and dP products
    over the causal triangle)."""
    import torch
    tg = P.tg
    L = P.layers[-1]
    T, hq, D = P.T, shape.hq, shape.head_dim
    o = torch.empty((T, hq, D), dtype=torch.bfloat16, device=P.dev)
    lse = torch.empty((hq, T), dtype=torch.float32, device=P.dev)
    tg.tg_gated_attention_rotated(P.q_rot, L["k_cache"], L["v"], P.pos, P.sk, L["gain"], L["tau"], P.cu_kept,
                                  P.max_kept, o=o, lse=lse)
    gen = torch.Generator(device=P.dev)
    gen.manual_seed(20261203)
    d_o = torch.randn((T, hq, D), generator=gen, device=P.dev).to(torch.bfloat16)
    d_s = torch.empty(T, dtype=torch.float32, device=P.dev)
    d_g = torch.empty(hq, dtype=torch.float32, device=P.dev)
    d_t = torch.empty(1, dtype=torch.float32, device=P.dev)
    ws = torch.empty(tg.lib.tg_attention_bwd_workspace_size(T, hq), dtype=torch.uint8, device=P.dev)

    def call():
        tg.tg_gated_attention_bwd(P.q_rot, L["k_cache"], L["v"], o, lse, d_o, P.pos, P.sk, L["gain"], L["tau"],
                                  P.cu_kept, P.max_kept, d_s=d_s, d_gain=d_g, d_tau=d_t, workspace=ws)

    call()
    torch.cuda.synchronize()
    ev = [torch.cuda.Event(enable_timing=True, external=True) for _ in range(2)]
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        ev[0].record()
        call()
        ev[1].record()
    per = []
    for i in range(3 + steps):
        flush()
        g.replay()
        torch.cuda.synchronize()
        if i >= 3:
            per.append(ev[0].elapsed_time(ev[1]))
    if tg.tg_check_device_status() != tg.TG_OK:
        raise RuntimeError("device status after the backward: " + tg.lib.tg_last_error_string().decode())
    ms = float(np.mean(per))
    fl = attention_flops(shape.kept_lens, hq, D)
    return {"ms_per_layer": ms, "tflops": fl / (ms * 1e-3) / 1e12, "gflop_per_layer": fl / 1e9,
            "launches_per_call": 4}


def deltanet_bytes(t, hk, hv, dk, dv):
    """Algorithmic HBM bytes of one gated-delta scan: q and k read (bf16),
    v read and o written (bf16), g and beta read (fp32)."""
    return float(t * (2 * hk * dk * 2 + 2 * hv * dv * 2 + 2 * hv * 4))


def measure_deltanet(dev, flush, steps, peaks, name="deltanet-32k-k4096"):
    """The pruned Gated DeltaNet scan over the kept tokens of a 32k NIAH-like
    context cut to K = 4096 (plus 64 question tokens), one CUDA graph around
    the call, L2 flushed before each replay."""
    import torch
    from learned_token_pruning_09_b300 import synth
    from learned_token_pruning_09_b300 import tokengate as tg
    inp = synth.deltanet_inputs(name)
    cfg = synth.DELTA_SHAPES[name]

    def bf(a):
        return torch.from_numpy(np.ascontiguousarray(a).view(np.int16)).to(dev).view(torch.bfloat16)

    q, k, v = bf(inp["q"]), bf(inp["k"]), bf(inp["v"])
    g = torch.as_tensor(inp["g"]).to(dev)
    beta = torch.as_tensor(inp["beta"]).to(dev)
    cu = torch.as_tensor(inp["cu_kept"]).to(dev)
    o = torch.empty_like(v)
    t = int(inp["cu_kept"][-1])
    nb = len(inp["cu_kept"]) - 1
    ws = torch.empty(tg.tg_gated_delta_scan_workspace_size(t, nb, cfg["hv"], cfg["dk"], cfg["dv"]),
                     dtype=torch.uint8, device=dev)

    def timed(chunked, cu=cu, ws=ws):
        call = lambda: tg.tg_gated_delta_scan(q, k, v, g, beta, cu, o=o, workspace=ws, chunked=chunked)
        call()
        torch.cuda.synchronize()
        graph, evs = capture_step([("scan", call)])
        replay_timed(graph, evs, flush, 3)
        us = float(replay_timed(graph, evs, flush, steps).mean()) * 1e3
        if tg.tg_check_device_status() != tg.TG_OK:
            raise RuntimeError("device status after the scan: " + tg.lib.tg_last_error_string().decode())
        return us

    us = timed(True)
    us_token = timed(False)
    # the same chunks as two launches: padded with empty sequences to more
    # (sequence, head) pairs than the one-launch form takes on any GPU up to
    # 320 SMs; the empty sequences do no work
    n_pad = 160 // cfg["hv"] + 1
    cu_pad = torch.as_tensor(np.concatenate([inp["cu_kept"], np.full(n_pad, t)]).astype(np.int32)).to(dev)
    ws_pad = torch.empty(tg.tg_gated_delta_scan_workspace_size(t, nb + n_pad, cfg["hv"], cfg["dk"], cfg["dv"]),
                         dtype=torch.uint8, device=dev)
    us_two = timed(True, cu_pad, ws_pad)
    byts = deltanet_bytes(t, cfg["hk"], cfg["hv"], cfg["dk"], cfg["dv"])
    return {"workload": name, "tokens": t, "hk": cfg["hk"], "hv": cfg["hv"], "dk": cfg["dk"], "dv": cfg["dv"],
            "form": "chunked (tf32 tensor cores, workspace); per-chunk products and state carry in one cooperative launch when batch x hv <= SMs / 2", "us": us, "gbs": byts / (us * 1e-6) / 1e9,
            "bytes": byts, "frac_of_measured_hbm": byts / (us * 1e-6) / 1e9 / peaks["hbm_gbs"],
            "workspace_bytes": int(ws.numel()), "token_by_token_us": us_token,
            "two_launch_us": us_two,
            "two_launch": "the same chunks in two launches (per-chunk products, then the state carry), forced by "
                          "padding with empty sequences"}


def max_over_ranks(values, device):
    """Each value's maximum over the ranks of the default process group (the
    values unchanged when there is one rank): the slowest rank's time."""
    import torch
    import torch.distributed as dist
    t = torch.tensor([float(v) for v in values], dtype=torch.float64, device=device)
    if dist.is_available() and dist.is_initialized() and dist.get_world_size() > 1:
        dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return [float(x) for x in t.cpu()]


def whole_job_tflops(flops_per_rank, world, max_ms):
    """Whole-job throughput of N replicas: all ranks' flops over the slowest
    rank's time."""
    return flops_per_rank * world / (max_ms * 1e-3) / 1e12


def proj_flops(shape):
    t, d = shape.n_kept, shape.d
    return 2.0 * t * d * (shape.hq + 2 * shape.hkv) * shape.head_dim + 2.0 * t * shape.hq * shape.head_dim * d


# ---------------------------------------------------------------------------
# clocks
# ---------------------------------------------------------------------------


class ClockSampler:
    FIELDS = ("clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, index: int):
        self.index = index
        self.proc = None
        self.lines = []

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.index), f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                 "-lms", "100"], stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self.thread = threading.Thread(target=self._read, daemon=True)
            self.thread.start()
        except OSError:
            self.proc = None

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append(line.strip())

    def stop(self):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        sm, mx, reasons, pw = [], None, set(), []
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for ln in self.lines:
            parts = [p.strip() for p in ln.split(",")]
            if len(parts) < 8:
                continue
            try:
                sm.append(float(parts[0]))
                mx = float(parts[1])
                pw.append(float(parts[2]))
            except ValueError:
                continue
            for nm, v in zip(names, parts[4:8]):
                if v.lower() == "active":
                    reasons.add(nm)
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": mx,
                "reasons": sorted(reasons), "samples": len(sm), "power_w_max": max(pw) if pw else None}


# ---------------------------------------------------------------------------
# inputs
# ---------------------------------------------------------------------------


_RESIDUALS = {}


def make_inputs(shape, with_scores=True):
    from learned_token_pruning_09_b300 import synth
    key = (shape.seed, shape.n_rows, shape.d)     # the budget sweep's three workloads share theirs
    if key not in _RESIDUALS:
        _RESIDUALS.clear()
        _RESIDUALS[key] = synth.residuals(shape)
    inp = {"x": _RESIDUALS[key], "p": synth.gate_weights(shape)}
    if with_scores:
        inp["s_draw"] = synth.score_draws(shape)
    if shape.with_proj:
        inp["layers"] = [synth.layer_params(shape, i) for i in range(shape.n_layers)]
    else:
        inp["ai"] = synth.attention_inputs(shape)
    return inp


def workload_config(shape):
    return {"workload": shape.name, "batch": shape.batch, "n_doc": shape.n_doc, "n_q": shape.n_q,
            "k": shape.k, "kept_tokens": shape.n_kept, "d": shape.d, "gate_h": shape.h, "hq": shape.hq,
            "hkv": shape.hkv, "head_dim": shape.head_dim, "layers_above_gate": shape.n_layers,
            "projections": shape.with_proj, "rope_theta": 1e6,
            "rope": "fused into the Q/K/V projection" if shape.with_proj else "tg_rope_qk before the attention",
            "l2": "flushed before every timed step: 256 MB written, then 256 MB read (no dirty line left)", "parallelism": "replicas"}


# ---------------------------------------------------------------------------
# reference arm / CPU baseline: the oracle on a bounded sample
# ---------------------------------------------------------------------------


def oracle_step_sample(shape, inputs, rng, n_gate_rows=256, n_attn_rows=16):
    """One bounded sample of the workload through the oracle: gate scores of
    ``n_gate_rows`` document rows, top-K over the full score vector, the
    gather, and attention outputs of ``n_attn_rows`` query rows (all heads)
    of one layer (for the stacked workload: layer 0, keys and values
    projected for every kept row).  Returns (seconds, attention flops of the
    sampled rows)."""
    import oracle
    x, p, s_full = inputs["x"], inputs["p"], inputs["s_draw"]
    t0 = time.perf_counter()
    rows = rng.choice(shape.n_doc[0], n_gate_rows, replace=False)
    oracle.gate_score(x, shape.cu_seqlens, shape.n_doc, p["w1"], p["b1"], p["w2"], p["b2"], rows=rows)
    kept, cu_kept = oracle.topk_select(s_full, shape.cu_seqlens, shape.n_doc, shape.k)
    xk, pos, sk = oracle.gather_kept(x, s_full, shape.cu_seqlens, kept, cu_kept)
    t_rows = rng.choice(len(kept), n_attn_rows, replace=False)
    if shape.with_proj:
        lp = inputs["layers"][0]
        oracle.stacked_layer(oracle.bf16_decode(xk), lp["w_qkv"], lp["w_o"], pos, sk, lp["gain"], lp["tau"],
                             cu_kept, shape.hq, shape.hkv, shape.head_dim, rows=t_rows)
    else:
        ai = inputs["ai"]
        oracle.gated_attention(ai["q"], ai["k"], ai["v"], pos, sk, ai["gain"], ai["tau"], cu_kept, rows=t_rows)
    dt = time.perf_counter() - t0
    seq = np.searchsorted(cu_kept, t_rows, side="right") - 1
    visible = t_rows - cu_kept[seq] + 1          # kept rows are in position order
    flops = float(np.sum(4.0 * shape.hq * shape.head_dim * visible))
    return dt, flops


def _openblas():
    """numpy's OpenBLAS, loaded in this process, and its thread-count calls
    (the exported names carry a prefix and suffix in numpy's own build)."""
    import ctypes
    try:
        with open("/proc/self/maps") as f:
            paths = sorted({ln.split()[-1] for ln in f if "openblas" in ln and ln.rstrip().endswith(".so")})
    except OSError:
        return None
    for path in paths:
        lib = ctypes.CDLL(path)
        for pre, suf in (("scipy_", "64_"), ("", "64_"), ("", "")):
            get, put = f"{pre}openblas_get_num_threads{suf}", f"{pre}openblas_set_num_threads{suf}"
            if hasattr(lib, get) and hasattr(lib, put):
                return getattr(lib, get), getattr(lib, put)
    return None


def blas_threads():
    try:
        from threadpoolctl import threadpool_info
        return max([i.get("num_threads", 1) for i in threadpool_info()] + [1])
    except ImportError:
        ob = _openblas()
        return int(ob[0]()) if ob else (os.cpu_count() or 1)


class single_thread:
    """The oracle timed as a single-threaded program: numpy's BLAS pool held
    at one thread while inside (the oracle itself is plain serial code)."""

    def __enter__(self):
        self.lim, self.ob, self.old = None, None, None
        try:
            from threadpoolctl import threadpool_limits
            self.lim = threadpool_limits(limits=1)
        except ImportError:
            self.ob = _openblas()
            if self.ob:
                self.old = int(self.ob[0]())
                self.ob[1](1)
        return self

    def __exit__(self, *exc):
        if self.lim is not None:
            self.lim.restore_original_limits()
        elif self.ob:
            self.ob[1](self.old)
        return False


def cpu_model():
    try:
        with open("/proc/cpuinfo") as f:
            for ln in f:
                if ln.startswith("model name"):
                    return ln.split(":", 1)[1].strip()
    except OSError:
        pass
    return "unknown"


SAMPLE_TEXT = ("gate on 256 document rows, full top-K and gather, then attention outputs of 16 random kept "
               "query rows x all heads of one layer{proj}; value = causal flops of the sampled rows / time")


def run_reference(args, shape):
    rank = int(os.environ.get("RANK", "0"))
    if rank != 0:
        return 0
    inputs = make_inputs(shape)
    rng = np.random.default_rng(0)
    with single_thread():
        for _ in range(args.warmup):
            oracle_step_sample(shape, inputs, rng, 16, 1)
        tot_t, tot_f = 0.0, 0.0
        for _ in range(args.steps):
            dt, fl = oracle_step_sample(shape, inputs, rng)
            tot_t += dt
            tot_f += fl
        cores = blas_threads()
    val = tot_f / tot_t / 1e12
    sample = "per step: " + SAMPLE_TEXT.format(proj=" (with its K/V projections of every kept row)"
                                               if shape.with_proj else "")
    line = {"impl": "reference", "metric": METRIC, "value": val, "unit": UNIT, "n_gpus": args.gpus,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": tot_t / args.steps * 1e3,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
            "data": "synthetic", "config": workload_config(shape),
            "cpu_baseline": {"value": val, "unit": UNIT, "cores": cores, "kind": "oracle",
                             "sample": sample, "cpu": cpu_model()},
            "e2e": {"value": val, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)
    return 0


# ---------------------------------------------------------------------------
# GPU arm
# ---------------------------------------------------------------------------


class Path:
    """Device buffers and the calls of one step, through the public binding."""

    def __init__(self, shape, inputs, dev):
        import torch
        from learned_token_pruning_09_b300 import tokengate as tg
        self.tg, self.shape, self.dev = tg, shape, dev

        def bf(a):
            return torch.from_numpy(np.ascontiguousarray(a).view(np.int16)).to(dev).view(torch.bfloat16)

        def i32(a):
            return torch.as_tensor(np.asarray(a, np.int32)).to(dev)

        self.bf = bf
        p = inputs["p"]
        T, d = shape.n_kept, shape.d
        self.X = bf(inputs["x"])
        self.W1, self.W2, self.b2 = bf(p["w1"]), bf(p["w2"]), p["b2"]
        self.cu, self.nd, self.kk = i32(shape.cu_seqlens), i32(shape.n_doc), i32(shape.k)
        self.T, self.max_nd, self.max_kept = T, max(shape.n_doc), max(shape.kept_lens)
        e = lambda *s, dt=torch.bfloat16: torch.empty(s, dtype=dt, device=dev)
        self.s = e(shape.n_rows, dt=torch.float32)
        self.topk_ws = tg.tg_topk_workspace(shape.batch, dev)
        self.kept = e(T, dt=torch.int32)
        self.cu_kept = e(shape.batch + 1, dt=torch.int32)
        self.xk = e(T, d)
        self.pos = e(T, dt=torch.int32)
        self.sk = e(T, dt=torch.float32)
        hq, hkv, D = shape.hq, shape.hkv, shape.head_dim
        self.q_rot = e(T, hq, D)
        self.layers = []
        if shape.with_proj:
            for lp in inputs["layers"]:
                self.layers.append({
                    "w_qkv": bf(lp["w_qkv"]), "wo": bf(lp["w_o"]), "gain": torch.as_tensor(lp["gain"]).to(dev),
                    "tau": lp["tau"], "k_cache": e(T, hkv, D), "v": e(T, hkv, D)})
            self.o = e(T, hq, D)
        else:
            ai = inputs["ai"]
            self.q, self.k = bf(ai["q"]), bf(ai["k"])
            self.layers.append({"v": bf(ai["v"]), "gain": torch.as_tensor(ai["gain"]).to(dev), "tau": ai["tau"],
                                "k_cache": e(T, hkv, D)})
            self.o = e(T, hq, D)

    # the calls
    def gate(self):
        self.tg.tg_gate_score(self.X, self.cu, self.nd, self.W1, None, self.W2, self.b2, s_out=self.s,
                              topk_ws=self.topk_ws)

    def topk(self):
        self.tg.tg_topk_select(self.s, self.cu, self.nd, self.kk, self.max_nd, self.T, kept_idx=self.kept,
                               cu_kept=self.cu_kept, workspace=self.topk_ws)

    def gather(self):
        self.tg.tg_gather_kept(self.X, self.s, self.cu, self.kept, self.cu_kept, self.T, x_kept=self.xk,
                               pos_kept=self.pos, s_kept=self.sk)

    def proj_qkv(self, i):
        # one GEMM for q, k and v with RoPE in its epilogue: q' into its own
        # buffer, k' into the layer's kept-only K cache
        L, sh = self.layers[i], self.shape
        self.tg.tg_qkv_rope_bf16(self.xk, L["w_qkv"], self.pos, sh.hq, sh.hkv, sh.head_dim, 1e6, q_out=self.q_rot,
                                 k_out=L["k_cache"], v_out=L["v"])

    def rope(self, i):
        # q' into a buffer of its own, k' into the layer's kept-only K cache
        self.tg.tg_rope_qk(self.q, self.k, self.pos, 1e6, self.cu_kept, q_out=self.q_rot,
                           k_out=self.layers[i]["k_cache"])

    def attn(self, i):
        L = self.layers[i]
        self.tg.tg_gated_attention_rotated(self.q_rot, L["k_cache"], L["v"], self.pos, self.sk, L["gain"], L["tau"],
                                           self.cu_kept, self.max_kept, o=self.o)

    def proj_o(self, i):
        L, T = self.layers[i], self.T
        self.tg.tg_linear_bf16(self.o.view(T, -1), L["wo"], residual=self.xk, out=self.xk)

    def segments(self):
        """(name, callable) in step order."""
        segs = [("gate", self.gate), ("topk", self.topk), ("gather", self.gather)]
        for i in range(len(self.layers)):
            if self.shape.with_proj:
                segs.append((f"proj_qkv{i}", lambda i=i: self.proj_qkv(i)))
            else:
                segs.append((f"rope{i}", lambda i=i: self.rope(i)))
            segs.append((f"attn{i}", lambda i=i: self.attn(i)))
            if self.shape.with_proj:
                segs.append((f"proj_o{i}", lambda i=i: self.proj_o(i)))
        return segs

    def launches_per_step(self):
        n = 3
        for _ in self.layers:
            n += 3 if self.shape.with_proj else 2     # qkv (with RoPE), attention, output / RoPE, attention
        return n


class L2Flush:
    """Before every timed step: 256 MB written, then another 256 MB read.
    L2 (126 MB) is then left holding clean lines of a buffer that the timed
    kernels never touch, so they neither hit their own data in L2 nor pay for
    writing back dirty lines of the flush itself."""

    def __init__(self, dev):
        import torch
        self.w = torch.empty(256 * 1024 * 1024, dtype=torch.uint8, device=dev)
        self.r = torch.ones(64 * 1024 * 1024, dtype=torch.int32, device=dev)
        self.out = torch.empty((), dtype=torch.int32, device=dev)

    def __call__(self):
        import torch
        self.w.zero_()
        torch.amax(self.r, dim=0, out=self.out)


def capture_step(segs):
    """The calls of one step captured as one CUDA graph, with a timing event
    recorded before each call and after the last, so that no launch gap sits
    between two kernels and each call's device time can be read back."""
    import torch
    evs = [torch.cuda.Event(enable_timing=True, external=True) for _ in range(len(segs) + 1)]
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph):
        for k, (_, f) in enumerate(segs):
            evs[k].record()
            f()
        evs[-1].record()
    torch.cuda.synchronize()
    return graph, evs


def replay_timed(graph, evs, flush, steps):
    """Replays the step ``steps`` times, L2 flushed before each, and returns
    the per-call device times [steps, calls] in ms."""
    import torch
    per = []
    for _ in range(steps):
        flush()
        graph.replay()
        torch.cuda.synchronize()     # the events are re-recorded by the next replay
        per.append([evs[k].elapsed_time(evs[k + 1]) for k in range(len(evs) - 1)])
    return np.array(per)


def time_calls(calls, flush, steps):
    """Device time (us) of a sequence of calls captured as one CUDA graph with
    events only around the whole sequence, so that consecutive kernels keep
    their programmatic launch edges (a kernel launched early behind its
    predecessor and waiting for it on the device); L2 flushed before each
    replay."""
    graph, evs = capture_step([("calls", lambda: [f() for f in calls])])
    replay_timed(graph, evs, flush, 3)
    return float(replay_timed(graph, evs, flush, steps).mean()) * 1e3


# the other workloads of the metric, each measured as one single-layer step
SIDE_WORKLOADS = ("qwen3-1.7b-16k", "budget-32k-k1024", "budget-32k-k4096", "budget-32k-k8192", "ragged-8")


def measure_workload(name, dev, flush, steps, peaks):
    """One workload's step (gate, top-K, gather, RoPE, token-gated attention
    on seeded q/k/v), captured and timed like the headline step."""
    import torch
    from learned_token_pruning_09_b300 import synth
    shape = synth.ALL_SHAPES[name]()
    P = Path(shape, make_inputs(shape, with_scores=False), dev)
    tg = P.tg
    segs = P.segments()
    for _, f in segs:
        f()
    torch.cuda.synchronize()
    if tg.tg_check_device_status() != tg.TG_OK:
        raise RuntimeError(f"device status ({name}): " + tg.lib.tg_last_error_string().decode())
    graph, evs = capture_step(segs)
    replay_timed(graph, evs, flush, 3)
    seg = dict(zip([n for n, _ in segs], replay_timed(graph, evs, flush, steps).mean(axis=0)))
    if tg.tg_check_device_status() != tg.TG_OK:
        raise RuntimeError(f"device status ({name}): " + tg.lib.tg_last_error_string().decode())
    fl = attention_flops(shape.kept_lens, shape.hq, shape.head_dim)
    attn_ms = seg["rope0"] + seg["attn0"]
    gtg_ms = time_calls([P.gate, P.topk, P.gather], flush, steps) * 1e-3
    byts = path_bytes(shape)
    out = {"batch": shape.batch, "n_rows": shape.n_rows, "kept_tokens": shape.n_kept,
           "attention": {"ms_per_layer": attn_ms, "tflops": fl / (attn_ms * 1e-3) / 1e12,
                         "kernel_ms": seg["attn0"], "kernel_tflops": fl / (seg["attn0"] * 1e-3) / 1e12,
                         "kernel_frac_of_burst": fl / (seg["attn0"] * 1e-3) / 1e12 / peaks["bf16_tflops"],
                         "rope_us": seg["rope0"] * 1e3, "gflop": fl / 1e9},
           "gate_topk_gather": {"us": gtg_ms * 1e3, "gbs": byts / (gtg_ms * 1e-3) / 1e9, "bytes": byts,
                                "frac_of_measured_hbm": byts / (gtg_ms * 1e-3) / 1e9 / peaks["hbm_gbs"],
                                "gate_us": seg["gate"] * 1e3, "topk_us": seg["topk"] * 1e3,
                                "gather_us": seg["gather"] * 1e3,
                                "split": "us: the three calls in one graph; gate/topk/gather_us: each "
                                         "between events (no early launch)"}}
    del P, graph
    torch.cuda.empty_cache()
    return out


def measure_model_ttft(dev, flush, steps):
    """Synthetic time to first token and peak prefill memory of a model with
    Qwen3-1.7B's layout and random weights: TokenGate's pruned prefill
    (gate at layer 1, 27 layers on the kept tokens) against the full prefill
    (every layer on every token), each followed by the first decode step.
    Everything runs eagerly through the public Python API, as a user calls
    it: TTFT is the device time from the first call of the prefill to the
    logits of the first token (host launch gaps included).  Peak prefill
    memory is the most device memory the prefill allocated on top of what
    was allocated before it (the model's weights and inputs, and this
    benchmark's other buffers); ``..._with_weights`` adds the model's own
    weight bytes, the figure a single-model process would see."""
    import torch
    from learned_token_pruning_09_b300 import synth
    from learned_token_pruning_09_b300.model import SyntheticModel
    model = SyntheticModel(synth.model_params_device("qwen3-1.7b", dev), device=dev)
    c = model.cfg
    torch.cuda.synchronize()
    tensors = [t for lp in model.layers for t in lp.values() if isinstance(t, torch.Tensor)]
    tensors += list(model.gate.values()) + [model.final_norm, model.w_lm]
    weights = float(sum(t.numel() * t.element_size() for t in tensors if isinstance(t, torch.Tensor)))
    out = {"model": "Qwen3-1.7B layout, random weights", "layers": c["n_layers"], "gate_layer": c["gate_layer"] + 1,
           "weights_gb": weights / 1e9, "contexts": {}}
    gen = torch.Generator(device=dev)
    gen.manual_seed(synth.BASE_SEED + 51)
    for ctx, (n_doc, n_q, k) in synth.MODEL_CONTEXTS.items():
        n = n_doc + n_q
        x = torch.randn((n, c["d"]), generator=gen, device=dev).to(torch.bfloat16)
        x_new = torch.randn((1, c["d"]), generator=gen, device=dev).to(torch.bfloat16)
        res = {"n_doc": n_doc, "n_q": n_q, "k": k}
        for mode in ("pruned", "full"):
            run = ((lambda: model.prefill(x, [n], [n_doc], [k])) if mode == "pruned"
                   else (lambda: model.prefill_full(x, [n])))
            st = run()
            model.decode(x_new, st)
            del st
            torch.cuda.synchronize()
            ttft, dec, peak = [], [], []
            for _ in range(steps):
                flush()
                torch.cuda.synchronize()
                base = torch.cuda.memory_allocated()
                torch.cuda.reset_peak_memory_stats()
                e = [torch.cuda.Event(enable_timing=True) for _ in range(4)]
                e[0].record()
                st = run()
                e[1].record()
                torch.cuda.synchronize()
                peak.append(torch.cuda.max_memory_allocated() - base)
                e[2].record()
                model.decode(x_new, st)
                e[3].record()
                torch.cuda.synchronize()
                ttft.append(e[0].elapsed_time(e[1]))
                dec.append(e[2].elapsed_time(e[3]))
                del st
            res[mode] = {"ttft_ms": float(np.mean(ttft)), "decode_ms": float(np.mean(dec)),
                         "peak_prefill_gb": float(np.max(peak)) / 1e9,
                         "peak_prefill_gb_with_weights": (float(np.max(peak)) + weights) / 1e9}
            torch.cuda.empty_cache()
        if model_status_bad(model):
            raise RuntimeError("device status after the model runs: " + tg_error())
        res["ttft_speedup"] = res["full"]["ttft_ms"] / res["pruned"]["ttft_ms"]
        res["peak_memory_ratio"] = res["full"]["peak_prefill_gb"] / res["pruned"]["peak_prefill_gb"]
        res["peak_memory_ratio_with_weights"] = (res["full"]["peak_prefill_gb_with_weights"] /
                                                 res["pruned"]["peak_prefill_gb_with_weights"])
        out["contexts"][ctx] = res
        del x, x_new
    del model
    torch.cuda.empty_cache()
    return out


def model_status_bad(model):
    from learned_token_pruning_09_b300 import tokengate as tg
    return tg.tg_check_device_status() != tg.TG_OK


def tg_error():
    from learned_token_pruning_09_b300 import tokengate as tg
    return tg.lib.tg_last_error_string().decode()


def run_gpu(args, shape):
    import torch
    import torch.distributed as dist

    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if world > 1:
        dist.init_process_group("nccl")
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    inputs = make_inputs(shape)
    P = Path(shape, inputs, dev)
    tg = P.tg
    segs = P.segments()
    flush = L2Flush(dev)

    # eager warm-up (initialises the library on this device), then capture
    for _ in range(2):
        for _, f in segs:
            f()
    torch.cuda.synchronize()
    if tg.tg_check_device_status() != tg.TG_OK:
        raise RuntimeError("device status after warm-up: " + tg.lib.tg_last_error_string().decode())
    # The whole step is one CUDA graph, with timing events recorded inside it
    # between the segments, so that no launch gap sits between two kernels.
    names = [n for n, _ in segs]
    graph, evs = capture_step(segs)
    stream = torch.cuda.current_stream()
    replay_timed(graph, evs, flush, max(args.warmup, 3))

    sampler = ClockSampler(local)
    sampler.start()
    time.sleep(0.3)
    if world > 1:
        dist.barrier()
    torch.cuda.synchronize()
    per = replay_timed(graph, evs, flush, args.steps)
    if world > 1:
        dist.barrier()
    clocks = sampler.stop()
    if tg.tg_check_device_status() != tg.TG_OK:
        raise RuntimeError("device status after timed steps: " + tg.lib.tg_last_error_string().decode())

    seg_ms = dict(zip(names, per.mean(axis=0)))
    step_ms = float(per.sum(axis=1).mean())
    # the token-gated attention layer: its RoPE prologue and the attention kernel
    kern_ms = float(sum(v for n, v in seg_ms.items() if n.startswith("attn")))
    rope_ms = float(sum(v for n, v in seg_ms.items() if n.startswith("rope")))
    attn_ms = kern_ms + rope_ms
    proj_ms = float(sum(v for n, v in seg_ms.items() if n.startswith("proj")))
    gtg_ms = time_calls([P.gate, P.topk, P.gather], flush, args.steps) * 1e-3
    nl = len(P.layers)
    step_ms, attn_ms, kern_ms, rope_ms = max_over_ranks([step_ms, attn_ms, kern_ms, rope_ms], dev)
    flops_layer = attention_flops(shape.kept_lens, shape.hq, shape.head_dim)
    tflops_rank = whole_job_tflops(flops_layer * nl, 1, attn_ms)
    kern_tflops = whole_job_tflops(flops_layer * nl, 1, kern_ms)
    value = whole_job_tflops(flops_layer * nl, world, attn_ms)
    byts = path_bytes(shape)
    peaks = load_peaks()

    # ---- general prunable spans (the next row after the path) ----
    masked = measure_masked(P, shape, flush, args.steps)
    masked["frac_of_measured_hbm"] = masked["gbs"] / peaks["hbm_gbs"]
    # ---- attention backward w.r.t. s, gain and tau (the next row after that) ----
    bwd = measure_attn_bwd(P, shape, flush, args.steps)
    bwd["frac_of_burst"] = bwd["tflops"] / peaks["bf16_tflops"]

    # ---- the metric's other workloads, and the synthetic model's TTFT ----
    workloads, model_ttft, deltanet = None, None, None
    if not args.headline_only:
        del graph
        torch.cuda.empty_cache()
        workloads = {n: measure_workload(n, dev, flush, args.steps, peaks) for n in SIDE_WORKLOADS}
        model_ttft = measure_model_ttft(dev, flush, 2)
    deltanet = measure_deltanet(dev, flush, args.steps, peaks)

    # ---- end to end through the public API, host buffers ----
    # Every step copies its inputs from pinned host memory and reads its
    # result back, all inside the timed region.  The next step's inputs travel
    # on a copy stream into a second set of device buffers while this step
    # computes (two input buffer sets, ordered by events); the result is
    # staged into one of two device buffers and read back on the copy stream
    # while the next step computes.
    import torch as _t
    x_h = _t.from_numpy(np.ascontiguousarray(inputs["x"]).view(np.int16)).view(_t.bfloat16).pin_memory()
    inputs_2 = [(lambda b: setattr(P, "X", b), [P.X, _t.empty_like(P.X)], x_h)]
    if not shape.with_proj:
        def v_setter(b):
            P.layers[0]["v"] = b
        for dst, key, setter in ((P.q, "q", lambda b: setattr(P, "q", b)), (P.k, "k", lambda b: setattr(P, "k", b)),
                                 (P.layers[0]["v"], "v", v_setter)):
            host = _t.from_numpy(np.ascontiguousarray(inputs["ai"][key]).view(np.int16)).view(_t.bfloat16).pin_memory()
            inputs_2.append((setter, [dst, _t.empty_like(dst)], host))
    out_dev = P.xk if shape.with_proj else P.o
    out_h = _t.empty(out_dev.shape, dtype=_t.bfloat16).pin_memory()
    kept_h = _t.empty(P.T, dtype=_t.int32).pin_memory()
    h2d = sum(h.numel() * h.element_size() for _, _, h in inputs_2)
    d2h = out_h.numel() * 2 + kept_h.numel() * 4
    copy_stream = _t.cuda.Stream()
    ev_in = [_t.cuda.Event(), _t.cuda.Event()]       # buffer set landed
    ev_free = [_t.cuda.Event(), _t.cuda.Event()]     # the step that read buffer set is done
    stage = [(_t.empty_like(out_dev), _t.empty_like(P.kept)) for _ in range(2)]
    ev_staged = [_t.cuda.Event(), _t.cuda.Event()]   # a step's result staged
    ev_read = [_t.cuda.Event(), _t.cuda.Event()]     # a staged result read back to the host

    def h2d_into(b):
        with _t.cuda.stream(copy_stream):
            copy_stream.wait_event(ev_free[b])
            for _, bufs, host in inputs_2:
                bufs[b].copy_(host, non_blocking=True)
            ev_in[b].record(copy_stream)

    def e2e_run(n):
        h2d_into(0)
        for i in range(n):
            b = i & 1
            if i + 1 < n:
                h2d_into(b ^ 1)
            stream.wait_event(ev_in[b])
            for setter, bufs, _ in inputs_2:
                setter(bufs[b])
            for _, f in segs:
                f()
            ev_free[b].record(stream)
            stream.wait_event(ev_read[b])
            stage[b][0].copy_(out_dev, non_blocking=True)
            stage[b][1].copy_(P.kept, non_blocking=True)
            ev_staged[b].record(stream)
            with _t.cuda.stream(copy_stream):
                copy_stream.wait_event(ev_staged[b])
                out_h.copy_(stage[b][0], non_blocking=True)
                kept_h.copy_(stage[b][1], non_blocking=True)
                ev_read[b].record(copy_stream)
        stream.wait_stream(copy_stream)            # the last read-back is inside the run

    e2e_run(2)
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e2e_steps = max(3, min(args.steps, 10))
    e0.record(stream)
    copy_stream.wait_event(e0)                  # no copy starts before the timed region
    e2e_run(e2e_steps)
    e1.record(stream)
    torch.cuda.synchronize()
    for setter, bufs, _ in inputs_2:
        setter(bufs[0])
    e2e_ms = e0.elapsed_time(e1) / e2e_steps
    e2e_ms, = max_over_ranks([e2e_ms], dev)
    e2e_val = whole_job_tflops(flops_layer * nl, world, e2e_ms)

    # ---- oracle baseline on the host (rank 0, N = 1 only) ----
    cpu = None
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        rng = np.random.default_rng(0)
        tt, ff, ns = 0.0, 0.0, 0
        with single_thread():
            while tt < args.cpu_seconds:
                dt, fl = oracle_step_sample(shape, inputs, rng)
                tt, ff, ns = tt + dt, ff + fl, ns + 1
            cores = blas_threads()
        cpu = {"value": ff / tt / 1e12, "unit": UNIT, "cores": cores, "kind": "oracle",
               "sample": f"{ns} samples, each: " + SAMPLE_TEXT.format(
                   proj=" (with its K/V projections of every kept row)" if shape.with_proj else ""),
               "seconds": tt, "cpu": cpu_model()}

    traffic = None
    tpath = os.path.join(ROOT, "profiles", "traffic.json")
    if os.path.exists(tpath):
        with open(tpath) as f:
            traffic = json.load(f).get(shape.name, {}).get("attn_kernel_dram_bytes_per_launch")

    if rank == 0:
        per_layer = attn_ms / nl
        line = {
            "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world, "steps": args.steps,
            "warmup": max(args.warmup, 3), "ms_per_step": step_ms, "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "bf16", "data": "synthetic",
            "config": workload_config(shape),
            "ms_per_layer": per_layer,
            "attention": {"ms_per_layer": per_layer, "tflops": tflops_rank, "layers": nl,
                          "gflop_per_layer": flops_layer / 1e9,
                          "kernel_ms_per_layer": kern_ms / nl, "kernel_tflops": kern_tflops,
                          "rope_us_per_layer": rope_ms / nl * 1e3},
            "workloads": workloads,
            "model_ttft": model_ttft,
            "gated_deltanet_scan": deltanet,
            "masked_gate_topk_gather": masked,
            "attention_bwd_s_gain_tau": bwd,
            "gate_topk_gather": {"us": gtg_ms * 1e3, "gbs": byts / (gtg_ms * 1e-3) / 1e9, "bytes": byts,
                                 "frac_of_measured_hbm": byts / (gtg_ms * 1e-3) / 1e9 / peaks["hbm_gbs"],
                                 "gate_us": seg_ms["gate"] * 1e3, "topk_us": seg_ms["topk"] * 1e3,
                                 "gather_us": seg_ms["gather"] * 1e3,
                                 "split": "us: the three calls in one graph; gate/topk/gather_us: each "
                                          "between events (no early launch)"},
            "projections": ({"ms_per_step": proj_ms, "tflops": proj_flops(shape) * nl / (proj_ms * 1e-3) / 1e12}
                            if shape.with_proj else None),
            "roofline": {"bound": "tensor", "achieved": kern_tflops, "peak": peaks["bf16_tflops"],
                         "unit": "TFLOP/s", "frac": kern_tflops / peaks["bf16_tflops"], "traffic": traffic,
                         "kernel": "attn_kernel (tg_gated_attention_rotated), mean over the step's launches",
                         "peak_source": peaks["source"] + " burst bf16 (of measured)",
                         "frac_of_sustained": kern_tflops / peaks["bf16_tflops_sustained"]
                         if peaks.get("bf16_tflops_sustained") else None},
            "e2e": {"value": e2e_val, "unit": UNIT, "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
                    "ms_per_step": e2e_ms,
                    "overlap": "each step's host-to-device copy runs on a copy stream into one of two device "
                               "input buffers while the previous step computes; each result is staged on the "
                               "device and read back on the copy stream while the next step computes"},
            "gpu_launches": P.launches_per_step() * args.steps,
            "clocks": clocks,
            "cpu_baseline": cpu,
        }
        print(json.dumps(line), flush=True)
    if world > 1:
        dist.destroy_process_group()
    return 0


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=10)
    ap.add_argument("--warmup", type=int, default=3)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--workload", default=DEFAULT_WORKLOAD)
    ap.add_argument("--layers", type=int, default=None, help="override the stacked workload's layer count")
    ap.add_argument("--cpu-seconds", type=float, default=12.0)
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--headline-only", action="store_true",
                    help="skip the other workloads and the synthetic model's TTFT")
    args = ap.parse_args()
    from learned_token_pruning_09_b300 import synth
    if args.workload not in synth.ALL_SHAPES:
        raise SystemExit(f"unknown workload {args.workload!r}; one of {sorted(synth.ALL_SHAPES)}")
    shape = synth.ALL_SHAPES[args.workload]()
    if args.layers is not None and shape.with_proj:
        shape.n_layers = args.layers
    if args.impl == "reference":
        return run_reference(args, shape)
    return run_gpu(args, shape)


if __name__ == "__main__":
    sys.exit(main())
