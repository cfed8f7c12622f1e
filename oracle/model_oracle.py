"""CPU oracle for a synthetic Qwen3-style pruned prefill and its first decode
step.

TEST INFRASTRUCTURE.  Only ``tests/``, ``__graft_entry__.smoke()`` and the
``cpu_baseline`` / reference leg of ``bench.py`` may import this module; the
product path never calls it and shares no code with it.

It composes the pinned functions of ``tokengate_oracle`` (the gate's GELU and
logsigmoid, the top-K, token-gated attention with RoPE) into the whole
forward pass that TokenGate prunes ("How does TokenGate's learned token
pruning work?", MarkTechPost article: three phases; "What is token-gated
attention?": the bias above the gate).  Everything is float64.  Readings:

* decoder layer (Qwen3 layout): a = RMSNorm(x; ln1); q, k, v = a W_q^T,
  a W_k^T, a W_v^T split per head; q and k normalised per head by RMSNorm
  over the head dimension (weights q_norm, k_norm) before RoPE;
  h = x + attn(q, k, v) W_o^T; m = RMSNorm(h; ln2);
  y = h + (SiLU(m W_gate^T) * (m W_up^T)) W_down^T.
  RMSNorm(x; w) = x / sqrt(mean(x^2) + eps) * w with eps = 1e-6.
* pruned prefill: layers 0..L-1 and the attention of layer L on all N
  tokens; the gate scores the post-attention residual h of layer L; the
  top-K keeps document rows (the question always); the MLP of layer L and
  every layer above it run on the kept rows only, their attention
  token-gated (bias gain_h s_j, temperature tau of each layer); a final
  RMSNorm and the LM head give the logits of the last row of each sequence,
  and the first generated token is their argmax (time to first token ends
  there).
* first decode step: the generated token's input row at position N_b runs
  through every layer; its attention reads the full-length caches in
  layers 0..L (those layers saw every token) and the kept-only caches above
  L, token-gated, with its own score 0 (generated tokens are not
  prunable, as question tokens are not).
"""
from __future__ import annotations

from typing import Dict, List, Optional, Sequence

import numpy as np

from .tokengate_oracle import gated_attention, gelu, logsigmoid, topk_select

__all__ = ["rms_norm", "silu", "swiglu_mlp", "layer_qkv", "attention_block", "dense_layer",
           "pruned_prefill", "decode_step"]

RMS_EPS = 1e-6


def rms_norm(x: np.ndarray, w: np.ndarray, eps: float = RMS_EPS) -> np.ndarray:
    """x / sqrt(mean(x^2) + eps) * w over the last axis."""
    x = np.asarray(x, np.float64)
    return x / np.sqrt(np.mean(x * x, axis=-1, keepdims=True) + eps) * np.asarray(w, np.float64)


def silu(z: np.ndarray) -> np.ndarray:
    """z * sigmoid(z), evaluated without overflow."""
    z = np.asarray(z, np.float64)
    return z * np.exp(-np.logaddexp(0.0, -z))


def swiglu_mlp(m: np.ndarray, p: Dict[str, np.ndarray]) -> np.ndarray:
    """(SiLU(m W_gate^T) * (m W_up^T)) W_down^T."""
    return (silu(m @ p["w_gate"].T) * (m @ p["w_up"].T)) @ p["w_down"].T


def layer_qkv(x: np.ndarray, p: Dict[str, np.ndarray], hq: int, hkv: int, d_head: int):
    """q [T, hq, D], k and v [T, hkv, D] of one layer, q and k normalised
    per head (before RoPE, which the attention applies)."""
    a = rms_norm(x, p["ln1"])
    t = a.shape[0]
    q = (a @ p["w_q"].T).reshape(t, hq, d_head)
    k = (a @ p["w_k"].T).reshape(t, hkv, d_head)
    v = (a @ p["w_v"].T).reshape(t, hkv, d_head)
    return rms_norm(q, p["q_norm"]), rms_norm(k, p["k_norm"]), v


def attention_block(x: np.ndarray, p: Dict[str, np.ndarray], pos: np.ndarray, cu: Sequence[int],
                    hq: int, hkv: int, d_head: int, s: Optional[np.ndarray] = None,
                    gain: Optional[np.ndarray] = None, tau: float = 1.0) -> np.ndarray:
    """h = x + attn W_o^T: plain causal attention (no score bias) unless s
    and gain are given."""
    q, k, v = layer_qkv(x, p, hq, hkv, d_head)
    t = x.shape[0]
    s = np.zeros(t) if s is None else s
    gain = np.zeros(hq) if gain is None else gain
    o, _ = gated_attention(q, k, v, pos, s, gain, tau, cu, q_is_f64=True)
    return x + o.reshape(t, hq * d_head) @ p["w_o"].T


def dense_layer(x, p, pos, cu, hq, hkv, d_head, s=None, gain=None, tau=1.0):
    """One decoder layer (attention block, then the SwiGLU MLP block)."""
    h = attention_block(x, p, pos, cu, hq, hkv, d_head, s, gain, tau)
    return h + swiglu_mlp(rms_norm(h, p["ln2"]), p)


def _positions(cu: Sequence[int]) -> np.ndarray:
    pos = np.zeros(int(cu[-1]), dtype=np.int64)
    for b in range(len(cu) - 1):
        pos[int(cu[b]): int(cu[b + 1])] = np.arange(int(cu[b + 1]) - int(cu[b]))
    return pos


def _gate(h: np.ndarray, is_doc: np.ndarray, gate: Dict[str, np.ndarray]) -> np.ndarray:
    """Gate scores of rows of h (fp32-rounded like the gate's output): the
    gate MLP on document rows, 0 on the others."""
    z = gelu(h @ gate["w1"].T + gate["b1"]) @ gate["w2"] + float(gate["b2"])
    return np.where(is_doc, logsigmoid(z).astype(np.float32), np.float32(0.0))


def pruned_prefill(x0: np.ndarray, layers: List[Dict[str, np.ndarray]], gate: Dict[str, np.ndarray],
                   gate_layer: int, cu_seqlens: Sequence[int], n_doc: Sequence[int], k: Sequence[int],
                   final_norm: np.ndarray, w_lm: np.ndarray, hq: int, hkv: int, d_head: int):
    """The pruned prefill of a packed batch.

    x0 [N, d] float64 input rows; layers: per-layer dicts of float64 weights
    (ln1, w_q, w_k, w_v, q_norm, k_norm, w_o, ln2, w_gate, w_up, w_down,
    gain, tau); gate: w1 [h, d], b1 [h], w2 [h], b2.  Returns a dict with
    logits [B, vocab] of each sequence's last row, next_token [B], the kept
    row ids and cu_kept, the scores s [N], and the caches the decode step
    reads: per layer its k (before RoPE) and v, over all rows in layers
    0..L and over the kept rows above L."""
    x = np.asarray(x0, np.float64)
    cu = np.asarray(cu_seqlens, np.int64)
    pos = _positions(cu)
    caches = []
    for li in range(gate_layer):
        _, kk, vv = layer_qkv(x, layers[li], hq, hkv, d_head)
        caches.append({"k": kk, "v": vv, "rows": np.arange(x.shape[0])})
        x = dense_layer(x, layers[li], pos, cu, hq, hkv, d_head)
    lp = layers[gate_layer]
    _, kk, vv = layer_qkv(x, lp, hq, hkv, d_head)
    caches.append({"k": kk, "v": vv, "rows": np.arange(x.shape[0])})
    h = attention_block(x, lp, pos, cu, hq, hkv, d_head)
    is_doc = np.zeros(x.shape[0], dtype=bool)
    for b in range(len(n_doc)):
        is_doc[int(cu[b]): int(cu[b]) + int(n_doc[b])] = True
    s = _gate(h, is_doc, gate)
    kept, cu_kept = topk_select(s, cu, n_doc, k)
    kept = np.asarray(kept, np.int64)
    hk = h[kept]
    xk = hk + swiglu_mlp(rms_norm(hk, lp["ln2"]), lp)
    pos_k, s_k = pos[kept], s[kept].astype(np.float64)
    for li in range(gate_layer + 1, len(layers)):
        p = layers[li]
        _, kk, vv = layer_qkv(xk, p, hq, hkv, d_head)
        caches.append({"k": kk, "v": vv, "rows": kept})
        xk = dense_layer(xk, p, pos_k, cu_kept, hq, hkv, d_head, s_k, p["gain"], p["tau"])
    last = np.asarray(cu_kept[1:], np.int64) - 1
    logits = rms_norm(xk[last], final_norm) @ w_lm.T
    return {"logits": logits, "next_token": np.argmax(logits, axis=-1), "kept": kept, "cu_kept": cu_kept,
            "s": s, "pos": pos, "caches": caches}


def decode_step(x_new: np.ndarray, prefill: Dict[str, object], layers: List[Dict[str, np.ndarray]],
                gate_layer: int, cu_seqlens: Sequence[int], final_norm: np.ndarray, w_lm: np.ndarray,
                hq: int, hkv: int, d_head: int):
    """The first decode step: x_new [B, d] float64, the input row of each
    sequence's generated token at position N_b.  Its attention reads the
    prefill's caches (all rows in layers 0..L, kept rows above L) plus
    itself.  Returns (logits [B, vocab], hidden [B, d])."""
    cu = np.asarray(cu_seqlens, np.int64)
    nb = len(cu) - 1
    cu_kept = np.asarray(prefill["cu_kept"], np.int64)
    pos_all = prefill["pos"]
    s_all = prefill["s"].astype(np.float64)
    x = np.asarray(x_new, np.float64).copy()
    for li, p in enumerate(layers):
        c = prefill["caches"][li]
        qn, kn, vn = layer_qkv(x, p, hq, hkv, d_head)
        above = li > gate_layer
        seg = cu_kept if above else cu
        out = np.empty((nb, hq * d_head))
        for b in range(nb):
            lo, hi = int(seg[b]), int(seg[b + 1])
            rows = c["rows"][lo:hi]
            n_b = int(cu[b + 1] - cu[b])
            kb = np.concatenate([c["k"][lo:hi], kn[b:b + 1]])
            vb = np.concatenate([c["v"][lo:hi], vn[b:b + 1]])
            qb = np.concatenate([np.zeros((hi - lo, hq, d_head)), qn[b:b + 1]])
            pb = np.concatenate([pos_all[rows], [n_b]])
            if above:
                sb = np.concatenate([s_all[rows], [0.0]])
                gain, tau = p["gain"], p["tau"]
            else:
                sb, gain, tau = np.zeros(hi - lo + 1), np.zeros(hq), 1.0
            o, _ = gated_attention(qb, kb, vb, pb, sb, gain, tau, [0, hi - lo + 1], q_is_f64=True,
                                   rows=np.array([hi - lo]))
            out[b] = o[hi - lo].reshape(hq * d_head)
        h = x + out @ p["w_o"].T
        x = h + swiglu_mlp(rms_norm(h, p["ln2"]), p)
    logits = rms_norm(x, final_norm) @ w_lm.T
    return logits, x
