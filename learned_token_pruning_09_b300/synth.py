"""Seeded synthetic inputs for the TokenGate pruned-prefill path.

This module draws random numbers and lays them out; it holds none of the
method's arithmetic (no gate, no score transform, no selection, no RoPE, no
attention).  Both the CUDA path and the CPU oracle take their inputs from
here, so a workload is identical on both sides.

The shapes follow the workloads the TokenGate write-ups measure on: Qwen3-1.7B
(hidden 2048, 16 query heads, 8 KV heads, head_dim 128) at batch 1 with a long
document followed by a short question, 16k to 128k tokens ("How does TokenGate
perform on the benchmarks?" and the TL;DR of the MarkTechPost article).  The
task datasets themselves (RepoBench-P, 2WikiMultihopQA, MultiNews, BioDEX,
NIAH) are not used; these draws stand in for their shapes only.

All floating-point tensors are drawn in float32 by numpy's PCG64 and encoded
to bfloat16 by round-to-nearest-even where the path stores bf16.  bf16 arrays
are returned as ``uint16`` bit patterns.
"""
from __future__ import annotations

from dataclasses import dataclass, field
from typing import Dict, List, Optional

import numpy as np

BASE_SEED = 20261202

# ---------------------------------------------------------------------------
# encoding helpers (storage formats, not method arithmetic)
# ---------------------------------------------------------------------------


def f32_to_bf16_bits(a: np.ndarray) -> np.ndarray:
    """Round float32 values to bfloat16 (round-to-nearest-even); return bits."""
    a = np.ascontiguousarray(a, dtype=np.float32)
    u = a.view(np.uint32)
    # the sum wraps only for NaN patterns; the low 16 bits of the shifted sum
    # are the same as those of the unwrapped sum
    rounding = np.uint32(0x7FFF) + ((u >> np.uint32(16)) & np.uint32(1))
    return ((u + rounding) >> np.uint32(16)).astype(np.uint16)


def bf16_bits_to_f32(b: np.ndarray) -> np.ndarray:
    """Decode bfloat16 bit patterns to float32 (exact)."""
    b = np.ascontiguousarray(b, dtype=np.uint16)
    return (b.astype(np.uint32) << np.uint32(16)).view(np.float32)


def _rng(seed_seq: np.random.SeedSequence) -> np.random.Generator:
    return np.random.Generator(np.random.PCG64(seed_seq))


def _normal_bf16(rng: np.random.Generator, shape, std: float = 1.0) -> np.ndarray:
    x = rng.standard_normal(size=shape, dtype=np.float32)
    if std != 1.0:
        x *= np.float32(std)
    return f32_to_bf16_bits(x)


# ---------------------------------------------------------------------------
# workload description
# ---------------------------------------------------------------------------


@dataclass
class Shape:
    """Sizes of one workload (no tensors)."""

    name: str
    n_doc: List[int]          # document tokens per sequence
    n_q: List[int]            # question tokens per sequence
    k: List[int]              # document keep budget per sequence
    d: int                    # hidden size of the gate-layer residual
    h: int                    # gate MLP hidden width
    hq: int                   # query heads
    hkv: int                  # key/value heads
    head_dim: int
    n_layers: int = 1         # token-gated attention layers above the gate
    with_proj: bool = False   # layers carry Q/K/V/O projections
    planted: bool = False     # gate logits carry a planted needle set
    planted_frac: float = 0.02
    tau_fixed: Optional[float] = None
    seed: int = BASE_SEED

    @property
    def batch(self) -> int:
        return len(self.n_doc)

    @property
    def seqlens(self) -> List[int]:
        return [a + b for a, b in zip(self.n_doc, self.n_q)]

    @property
    def cu_seqlens(self) -> np.ndarray:
        return np.concatenate([[0], np.cumsum(self.seqlens)]).astype(np.int32)

    @property
    def n_rows(self) -> int:
        return int(sum(self.seqlens))

    @property
    def k_eff(self) -> List[int]:
        return [min(k, n) for k, n in zip(self.k, self.n_doc)]

    @property
    def kept_lens(self) -> List[int]:
        return [ke + q for ke, q in zip(self.k_eff, self.n_q)]

    @property
    def cu_kept(self) -> np.ndarray:
        return np.concatenate([[0], np.cumsum(self.kept_lens)]).astype(np.int32)

    @property
    def n_kept(self) -> int:
        return int(sum(self.kept_lens))


def tiny(seed_offset: int = 0) -> Shape:
    """Tiny case: 512 document + 32 question tokens, d=256, 4/2 heads, D=64."""
    return Shape("tiny", [512], [32], [128], d=256, h=64, hq=4, hkv=2,
                 head_dim=64, tau_fixed=1.1, seed=BASE_SEED + 0 + seed_offset)


def qwen3_16k() -> Shape:
    """Qwen3-1.7B-shaped single layer: 16,320 document + 64 question tokens."""
    return Shape("qwen3-1.7b-16k", [16320], [64], [2048], d=2048, h=256,
                 hq=16, hkv=8, head_dim=128, seed=BASE_SEED + 1)


def budget_32k(k: int) -> Shape:
    """Budget sweep at 32k: 32,704 document + 64 question tokens, planted logits."""
    assert k in (1024, 4096, 8192)
    return Shape(f"budget-32k-k{k}", [32704], [64], [k], d=2048, h=256,
                 hq=16, hkv=8, head_dim=128, planted=True, seed=BASE_SEED + 2)


def long_128k(n_layers: int = 27) -> Shape:
    """Long context: 131,008 document + 64 question tokens, K=8192, a stack
    of token-gated attention layers with their own projections."""
    return Shape("long-128k", [131008], [64], [8192], d=2048, h=256, hq=16,
                 hkv=8, head_dim=128, n_layers=n_layers, with_proj=True,
                 seed=BASE_SEED + 3)


def ragged_batch() -> Shape:
    """Ragged batch of 8: document lengths U{8192..65536}, 32-128 question
    tokens, keep fraction U[5%, 25%] per sequence (k = floor(frac * n_doc))."""
    ss = np.random.SeedSequence(BASE_SEED + 4)
    rng = _rng(ss.spawn(1)[0])
    n_doc = rng.integers(8192, 65536, size=8, endpoint=True).tolist()
    n_q = rng.integers(32, 128, size=8, endpoint=True).tolist()
    frac = rng.uniform(0.05, 0.25, size=8)
    k = [int(np.floor(f * n)) for f, n in zip(frac, n_doc)]
    return Shape("ragged-8", n_doc, n_q, k, d=2048, h=256, hq=16, hkv=8,
                 head_dim=128, seed=BASE_SEED + 4)


def custom(name: str, n_doc, n_q, k, d=256, h=64, hq=4, hkv=2, head_dim=64,
           seed: int = BASE_SEED + 100, **kw) -> Shape:
    """Any other shape, for edge cases."""
    return Shape(name, list(n_doc), list(n_q), list(k), d=d, h=h, hq=hq,
                 hkv=hkv, head_dim=head_dim, seed=seed, **kw)


# ---------------------------------------------------------------------------
# draws
# ---------------------------------------------------------------------------

# sub-stream ids (stable: adding a stream never changes another's draws)
_S_X, _S_W1, _S_W2, _S_QKV, _S_GAIN, _S_TAU, _S_PLANT, _S_SCORES, _S_LAYERS, _S_SPANS = range(10)


def _stream(shape: Shape, sid: int) -> np.random.Generator:
    ss = np.random.SeedSequence(entropy=shape.seed, spawn_key=(sid,))
    return _rng(ss)


def residuals(shape: Shape) -> np.ndarray:
    """Gate-layer residual stream X [n_rows, d], bf16 ~ N(0, 1)."""
    return _normal_bf16(_stream(shape, _S_X), (shape.n_rows, shape.d))


def gate_weights(shape: Shape) -> Dict[str, object]:
    """Gate MLP parameters d -> h -> 1.  W1 [h, d] ~ N(0, 1/d) (nn.Linear
    layout), w2 [h] ~ N(0, 1/h); both biases zero, as the workloads state."""
    w1 = _normal_bf16(_stream(shape, _S_W1), (shape.h, shape.d), std=1.0 / np.sqrt(shape.d))
    w2 = _normal_bf16(_stream(shape, _S_W2), (shape.h,), std=1.0 / np.sqrt(shape.h))
    return {"w1": w1, "w2": w2, "b1": np.zeros(shape.h, np.float32), "b2": 0.0}


def attention_inputs(shape: Shape, n_kept: Optional[int] = None) -> Dict[str, object]:
    """Per-layer attention inputs for the single-layer workloads:
    q [T, hq, D], k and v [T, hkv, D], bf16 ~ N(0, 1); gain [hq] ~ U(0.5, 2);
    tau = the workload's fixed value, else ~ U(0.9, 1.3)."""
    t = shape.n_kept if n_kept is None else n_kept
    r = _stream(shape, _S_QKV)
    q = _normal_bf16(r, (t, shape.hq, shape.head_dim))
    k = _normal_bf16(r, (t, shape.hkv, shape.head_dim))
    v = _normal_bf16(r, (t, shape.hkv, shape.head_dim))
    gain = _stream(shape, _S_GAIN).uniform(0.5, 2.0, size=shape.hq).astype(np.float32)
    if shape.tau_fixed is not None:
        tau = float(np.float32(shape.tau_fixed))
    else:
        tau = float(np.float32(_stream(shape, _S_TAU).uniform(0.9, 1.3)))
    return {"q": q, "k": k, "v": v, "gain": gain, "tau": tau}


def layer_params(shape: Shape, layer: int) -> Dict[str, object]:
    """Projections and gate parameters of one stacked layer: W_qkv
    [(hq+2 hkv) D, d] and W_o [d, hq D], bf16 ~ N(0, 1/fan_in); gain [hq] ~
    U(0.5, 2); tau ~ U(0.9, 1.3)."""
    ss = np.random.SeedSequence(entropy=shape.seed, spawn_key=(_S_LAYERS, layer))
    r = _rng(ss)
    n_qkv = (shape.hq + 2 * shape.hkv) * shape.head_dim
    n_o_in = shape.hq * shape.head_dim
    w_qkv = _normal_bf16(r, (n_qkv, shape.d), std=1.0 / np.sqrt(shape.d))
    w_o = _normal_bf16(r, (shape.d, n_o_in), std=1.0 / np.sqrt(n_o_in))
    gain = r.uniform(0.5, 2.0, size=shape.hq).astype(np.float32)
    tau = float(np.float32(r.uniform(0.9, 1.3)))
    return {"w_qkv": w_qkv, "w_o": w_o, "gain": gain, "tau": tau}


def planted_logits(shape: Shape) -> np.ndarray:
    """Gate logits with a needle-like structure, per sequence: z ~ N(0, 1)
    except round(frac * n_doc) positions chosen uniformly without replacement
    with z ~ N(3, 1).  Returned as float64 over document rows only, packed in
    sequence order (length sum(n_doc))."""
    r = _stream(shape, _S_PLANT)
    out = []
    for n in shape.n_doc:
        z = r.standard_normal(n)
        m = int(round(shape.planted_frac * n))
        idx = r.choice(n, size=m, replace=False)
        z[idx] = r.normal(3.0, 1.0, size=m)
        out.append(z)
    return np.concatenate(out) if out else np.zeros(0)


def score_draws(shape: Shape, tie_frac: float = 0.05) -> np.ndarray:
    """Non-positive float32 values shaped like gate scores, for testing the
    selector on its own: -|N(0, 4)| per row, with ``tie_frac`` of the document
    rows copied from another row (exact ties) and a few exact -0.0 and +0.0
    values; question rows are +0.0.  Returned over all n_rows."""
    r = _stream(shape, _S_SCORES)
    s = -np.abs(r.normal(0.0, 4.0, size=shape.n_rows)).astype(np.float32)
    cu = shape.cu_seqlens
    for b in range(shape.batch):
        lo, nd = int(cu[b]), shape.n_doc[b]
        if nd > 1:
            m = max(1, int(tie_frac * nd))
            src = r.integers(0, nd, size=m)
            dst = r.integers(0, nd, size=m)
            s[lo + dst] = s[lo + src]
            z = r.integers(0, nd, size=min(4, nd))
            s[lo + z[: len(z) // 2]] = np.float32(-0.0)
            s[lo + z[len(z) // 2:]] = np.float32(0.0)
        s[lo + nd: lo + nd + shape.n_q[b]] = 0.0
    return s


def prunable_spans(shape: Shape, spans_per_seq: int = 4, frac: float = 0.85,
                   seed_offset: int = 0) -> np.ndarray:
    """A per-row prunable mask (uint8 [n_rows]) with several marked spans per
    sequence, the way a prompt template can mark more than one block of
    retrieved text: each sequence's rows are cut at ``2 spans_per_seq - 1``
    random points into alternating fixed / prunable / fixed / ... blocks
    (the first and last blocks fixed), the prunable blocks covering about
    ``frac`` of the sequence.  Sequences shorter than the span count get one
    prunable block in the middle (or none when empty)."""
    r = np.random.default_rng(np.random.SeedSequence(
        [BASE_SEED, _S_SPANS, seed_offset, shape.n_rows, shape.batch]))
    mask = np.zeros(shape.n_rows, dtype=np.uint8)
    cu = shape.cu_seqlens
    for b in range(shape.batch):
        lo, hi = int(cu[b]), int(cu[b + 1])
        n = hi - lo
        if n == 0:
            continue
        if n < 4 * spans_per_seq:
            mask[lo + n // 4: lo + n - n // 4] = 1
            continue
        # fixed blocks share (1 - frac) of the rows, prunable blocks frac
        n_fix = spans_per_seq + 1
        fix_w = r.dirichlet(np.ones(n_fix)) * (1.0 - frac) * n
        prun_w = r.dirichlet(np.ones(spans_per_seq)) * frac * n
        widths = np.empty(2 * spans_per_seq + 1)
        widths[0::2] = fix_w
        widths[1::2] = prun_w
        edges = np.concatenate([[0], np.round(np.cumsum(widths)).astype(np.int64)])
        edges[-1] = n
        for sp in range(spans_per_seq):
            a, e = edges[2 * sp + 1], edges[2 * sp + 2]
            mask[lo + a: lo + e] = 1
    return mask


def budgets(shape: Shape) -> np.ndarray:
    return np.asarray(shape.k, dtype=np.int32)


def n_doc_array(shape: Shape) -> np.ndarray:
    return np.asarray(shape.n_doc, dtype=np.int32)


ALL_SHAPES = {
    "tiny": tiny,
    "qwen3-1.7b-16k": qwen3_16k,
    "budget-32k-k1024": lambda: budget_32k(1024),
    "budget-32k-k4096": lambda: budget_32k(4096),
    "budget-32k-k8192": lambda: budget_32k(8192),
    "long-128k": long_128k,
    "ragged-8": ragged_batch,
}


# ---------------------------------------------------------------------------
# pruned Gated DeltaNet scan inputs
# ---------------------------------------------------------------------------
_S_DELTA = 10

# Kept-token streams of the hybrid model's linear-attention layers: a 32k
# needle-in-a-haystack context (32,704 document + 64 question tokens) cut to
# K = 4,096 kept document tokens, so T = 4,160, batch 1; and a ragged batch.
DELTA_SHAPES = {
    "deltanet-tiny": {"lens": [160], "hk": 2, "hv": 4, "dk": 64, "dv": 64},
    "deltanet-32k-k4096": {"lens": [4160], "hk": 16, "hv": 32, "dk": 128, "dv": 128},
    "deltanet-ragged": {"lens": [1500, 37, 0, 900, 2049], "hk": 4, "hv": 8, "dk": 128, "dv": 128},
}


def deltanet_inputs(name: str) -> Dict[str, object]:
    """Seeded inputs of one gated-delta scan: q, k [T, hk, dk] and v
    [T, hv, dv] bf16 bits ~ N(0, 1); g [T, hv] fp32 log-decays, -g
    log-uniform in [0.005, 0.5] (decays exp(g) in [0.61, 0.995]); beta
    [T, hv] fp32 ~ U(0.05, 0.95); cu_kept [B+1] int32."""
    cfg = DELTA_SHAPES[name]
    lens = cfg["lens"]
    t = int(sum(lens))
    r = np.random.default_rng(np.random.SeedSequence([BASE_SEED, _S_DELTA, t, cfg["hv"], cfg["dk"]]))
    q = _normal_bf16(r, (t, cfg["hk"], cfg["dk"]))
    k = _normal_bf16(r, (t, cfg["hk"], cfg["dk"]))
    v = _normal_bf16(r, (t, cfg["hv"], cfg["dv"]))
    g = (-np.exp(r.uniform(np.log(0.005), np.log(0.5), size=(t, cfg["hv"])))).astype(np.float32)
    beta = r.uniform(0.05, 0.95, size=(t, cfg["hv"])).astype(np.float32)
    cu = np.concatenate([[0], np.cumsum(lens)]).astype(np.int32)
    return {"q": q, "k": k, "v": v, "g": g, "beta": beta, "cu_kept": cu}


# ---------------------------------------------------------------------------
# synthetic Qwen3-style model for the pruned prefill and its decode step
# ---------------------------------------------------------------------------
_S_MODEL = 11

MODEL_CONFIGS = {
    # small enough for the float64 oracle; the layout of the full model
    "model-tiny": {"n_layers": 4, "gate_layer": 1, "d": 128, "ffn": 256, "hq": 4, "hkv": 2, "head_dim": 64,
                   "vocab": 512, "gate_h": 32},
    # Qwen3-1.7B's layout (28 layers, hidden 2048, MLP 6144, 16/8 heads of 128,
    # vocabulary 151,936); TokenGate prunes it at layer 1 counted from one,
    # i.e. index 0 here, so 27 layers run on the kept tokens only
    "qwen3-1.7b": {"n_layers": 28, "gate_layer": 0, "d": 2048, "ffn": 6144, "hq": 16, "hkv": 8, "head_dim": 128,
                   "vocab": 151936, "gate_h": 256},
}

# context lengths of the synthetic time-to-first-token measurement: document
# rows, question rows and the document budget K (the 16k and 128k workloads)
MODEL_CONTEXTS = {"16k": (16320, 64, 2048), "128k": (131008, 64, 8192)}


def model_params(name: str) -> Dict[str, object]:
    """Seeded weights (bf16 bits) of a synthetic model: per layer ln1, ln2,
    q_norm, k_norm ~ 1 + N(0, 0.1^2); w_q, w_k, w_v, w_o, w_gate, w_up,
    w_down ~ N(0, 1/fan_in); layers above the gate get gain ~ U(0.5, 2) and
    tau ~ U(0.9, 1.3); the gate MLP as gate_weights; final norm and an LM
    head ~ N(0, 1/d)."""
    c = MODEL_CONFIGS[name]
    r = np.random.default_rng(np.random.SeedSequence([BASE_SEED, _S_MODEL, c["d"], c["n_layers"]]))
    d, f, hq, hkv, dh = c["d"], c["ffn"], c["hq"], c["hkv"], c["head_dim"]
    norm = lambda n: f32_to_bf16_bits((1.0 + 0.1 * r.standard_normal(n)).astype(np.float32))
    layers = []
    for li in range(c["n_layers"]):
        layers.append({
            "ln1": norm(d), "ln2": norm(d), "q_norm": norm(dh), "k_norm": norm(dh),
            "w_q": _normal_bf16(r, (hq * dh, d), 1.0 / np.sqrt(d)),
            "w_k": _normal_bf16(r, (hkv * dh, d), 1.0 / np.sqrt(d)),
            "w_v": _normal_bf16(r, (hkv * dh, d), 1.0 / np.sqrt(d)),
            "w_o": _normal_bf16(r, (d, hq * dh), 1.0 / np.sqrt(hq * dh)),
            "w_gate": _normal_bf16(r, (f, d), 1.0 / np.sqrt(d)),
            "w_up": _normal_bf16(r, (f, d), 1.0 / np.sqrt(d)),
            "w_down": _normal_bf16(r, (d, f), 1.0 / np.sqrt(f)),
            "gain": r.uniform(0.5, 2.0, size=hq).astype(np.float32),
            "tau": float(np.float32(r.uniform(0.9, 1.3))),
        })
    gate = {"w1": _normal_bf16(r, (c["gate_h"], d), 1.0 / np.sqrt(d)),
            "w2": _normal_bf16(r, (c["gate_h"],), 1.0 / np.sqrt(c["gate_h"])),
            "b1": np.zeros(c["gate_h"], np.float32), "b2": 0.0}
    return {"config": c, "layers": layers, "gate": gate, "final_norm": norm(d),
            "w_lm": _normal_bf16(r, (c["vocab"], d), 1.0 / np.sqrt(d))}


def model_params_device(name: str, device, seed: int = BASE_SEED + 50) -> Dict[str, object]:
    """The same layout and distributions as ``model_params``, drawn on the
    device by torch's seeded generator (the full-size model has 1.4 billion
    weights, too many to draw on the host in a benchmark).  bf16 tensors and
    float32 gains; for timing and memory only, never compared bit for bit."""
    import torch
    c = MODEL_CONFIGS[name]
    g = torch.Generator(device=device)
    g.manual_seed(seed)
    d, f, hq, hkv, dh = c["d"], c["ffn"], c["hq"], c["hkv"], c["head_dim"]

    def normal(shape, std):
        return (torch.randn(shape, generator=g, device=device, dtype=torch.float32) * std).to(torch.bfloat16)

    def norm(n):
        return (1.0 + 0.1 * torch.randn(n, generator=g, device=device, dtype=torch.float32)).to(torch.bfloat16)

    def uniform(n, lo, hi):
        return lo + (hi - lo) * torch.rand(n, generator=g, device=device, dtype=torch.float32)

    layers = []
    for _ in range(c["n_layers"]):
        layers.append({
            "ln1": norm(d), "ln2": norm(d), "q_norm": norm(dh), "k_norm": norm(dh),
            "w_q": normal((hq * dh, d), d ** -0.5), "w_k": normal((hkv * dh, d), d ** -0.5),
            "w_v": normal((hkv * dh, d), d ** -0.5), "w_o": normal((d, hq * dh), (hq * dh) ** -0.5),
            "w_gate": normal((f, d), d ** -0.5), "w_up": normal((f, d), d ** -0.5),
            "w_down": normal((d, f), f ** -0.5),
            "gain": uniform(hq, 0.5, 2.0), "tau": float(uniform(1, 0.9, 1.3).item())})
    gate = {"w1": normal((c["gate_h"], d), d ** -0.5), "w2": normal((c["gate_h"],), c["gate_h"] ** -0.5),
            "b1": torch.zeros(c["gate_h"], device=device), "b2": 0.0}
    return {"config": c, "layers": layers, "gate": gate, "final_norm": norm(d),
            "w_lm": normal((c["vocab"], d), d ** -0.5)}
