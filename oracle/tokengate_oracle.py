"""CPU oracle for the TokenGate pruned-prefill path.

TEST INFRASTRUCTURE.  Only ``tests/``, ``__graft_entry__.smoke()`` and the
``cpu_baseline`` / reference leg of ``bench.py`` may import this module.  The
product path (the CUDA library and its binding) never calls it, and it shares
no code with that path: the two meet only at the seeded inputs of
``learned_token_pruning_09_b300.synth``.

Everything here is plain, slow and single-pass, in float64, written from the
TokenGate articles ("How does TokenGate's learned token pruning work?" and
"What is token-gated attention?" in the MarkTechPost article, with the same
facts in the mainews.gr article, section "How it decides what to keep").  The
articles fix the structure (an MLP gate on the post-attention residual at the
gate layer, a top-K over document tokens with the question always kept, layers
above the gate run over the kept tokens only, the kept token's score added as a
bias to the attention logits with a learnable per-head gain and temperature);
the exact algebra that they leave open is taken as follows:

* gate:   z_j = w2 . GELU(W1 x_j + b1) + b2, GELU with the exact erf form;
          s_j = logsigmoid(z_j) for document rows, s_j = 0 for question rows.
* top-K:  per sequence, the K largest s_j among document rows, ties to the
          lower row index, output in ascending row order, then every question
          row.  K larger than the document keeps the whole document.
* attention over kept tokens, per query row i and head h:
          logit_ij = (q'_i . k'_j) / (sqrt(D) tau) + g_h s_j
          over kept j of the same sequence with pos_j <= pos_i; softmax over j;
          o_i = sum_j p_ij v_j.  q' and k' carry rotate-half RoPE at the
          original positions, theta = 1e6; query head h reads KV head
          floor(h / G), G = hq / hkv.
* attention backward (the gradient path from the attention loss to the gate):
          for L = sum dO . o, the derivatives with respect to s_j, g_h and tau,
          from dl_ij = p_ij (dO_i . v_j - sum_j' p_ij' dO_i . v_j').
* pruned Gated DeltaNet (the hybrid model's linear-attention layers, which
          TokenGate also prunes): per value head a state S (d_v x d_k) runs
          the gated delta rule over the KEPT tokens of a sequence, in order,
          S_t = S_{t-1} alpha_t (I - beta_t k_t k_t^T) + beta_t v_t k_t^T,
          o_t = S_t q_t, with alpha_t = exp(g_t), q and k L2-normalised and q
          scaled by 1/sqrt(d_k); a pruned token never updates the state.
* stacked layer (long-context workload): qkv = x W_qkv^T, attention as above,
          x_out = x + o W_o^T.  No norm and no MLP.
* general prunable spans (the prompt template marks the prunable document
          with {state}; several marked spans, anywhere in a sequence): the gate
          scores the prunable rows (0 elsewhere), the top-K budget of a
          sequence goes to its prunable rows, every other row is kept, and the
          kept rows come out in ascending row order.  With the mask equal to
          the document prefix this is the document/question case above.

Every function is pinned by the ``-m "not gpu"`` tests in
``tests/test_oracle_pins.py`` against closed forms, brute force on tiny inputs,
library routines (torch's scaled-dot-product attention in float64 for the
dense-causal special case) and invariants.  Parity is pinned for every
function here; the articles print no intermediate values, so nothing is pinned
to a printed number.
"""
from __future__ import annotations

import heapq
import math
from typing import Optional, Sequence

import numpy as np
from scipy.special import erf as _erf

__all__ = [
    "bf16_decode", "gelu", "logsigmoid", "gate_score", "score_from_logit",
    "topk_select", "gather_kept", "rope", "gated_attention",
    "stacked_layer", "project_qkv", "gate_score_masked", "topk_select_masked",
    "gated_attention_bwd", "gated_delta_scan",
]


def bf16_decode(bits: np.ndarray) -> np.ndarray:
    """bfloat16 bit patterns (uint16) -> float64, exactly."""
    b = np.asarray(bits, dtype=np.uint16).astype(np.uint32) << np.uint32(16)
    return b.view(np.float32).astype(np.float64)


# ---------------------------------------------------------------------------
# gate (MarkTechPost article, "How does TokenGate's learned token pruning
# work?", second phase: an MLP scores every token from its post-attention
# residual at gate layer L)
# ---------------------------------------------------------------------------


def gelu(u: np.ndarray) -> np.ndarray:
    """GELU(u) = u * Phi(u) = 0.5 u (1 + erf(u / sqrt 2))."""
    u = np.asarray(u, dtype=np.float64)
    return 0.5 * u * (1.0 + _erf(u / math.sqrt(2.0)))


def logsigmoid(z: np.ndarray) -> np.ndarray:
    """log(sigmoid(z)) = -log(1 + exp(-z)), evaluated without overflow:
    -log1p(exp(-z)) for z >= 0 and z - log1p(exp(z)) for z < 0."""
    z = np.asarray(z, dtype=np.float64)
    out = np.empty_like(z)
    pos = z >= 0
    out[pos] = -np.log1p(np.exp(-z[pos]))
    zn = z[~pos]
    out[~pos] = zn - np.log1p(np.exp(zn))
    return out


def score_from_logit(z: np.ndarray) -> np.ndarray:
    """Gate score of a document token from its gate logit, rounded to fp32."""
    return logsigmoid(z).astype(np.float32)


def gate_score(x_bits: np.ndarray, cu_seqlens: Sequence[int], n_doc: Sequence[int],
               w1_bits: np.ndarray, b1: Optional[np.ndarray], w2_bits: np.ndarray,
               b2: float, rows: Optional[np.ndarray] = None) -> np.ndarray:
    """Gate scores s [n_rows] float32.

    Document rows: s = logsigmoid(w2 . GELU(W1 x + b1) + b2), computed in
    float64 from the bf16 inputs and rounded once to float32.  Question rows:
    exactly 0.0.  ``rows`` restricts the work to the given row ids (the other
    entries are returned as NaN)."""
    n_rows = np.asarray(x_bits).shape[0]
    is_doc = np.zeros(n_rows, dtype=bool)
    for b in range(len(n_doc)):
        lo = int(cu_seqlens[b])
        is_doc[lo: lo + int(n_doc[b])] = True
    return _gate_on_rows(x_bits, is_doc, w1_bits, b1, w2_bits, b2, rows)


def gate_score_masked(x_bits: np.ndarray, prunable: np.ndarray, w1_bits: np.ndarray,
                      b1: Optional[np.ndarray], w2_bits: np.ndarray, b2: float,
                      rows: Optional[np.ndarray] = None) -> np.ndarray:
    """Gate scores with the prunable rows given by a per-row mask (any
    number of spans, anywhere in a sequence): s = logsigmoid(w2 . GELU(W1 x +
    b1) + b2) on prunable rows, exactly 0 on the others."""
    return _gate_on_rows(x_bits, np.asarray(prunable).astype(bool), w1_bits, b1, w2_bits, b2, rows)


def _gate_on_rows(x_bits, is_doc, w1_bits, b1, w2_bits, b2, rows):
    """The gate MLP on the rows where ``is_doc`` holds, 0 on the others."""
    x_bits = np.asarray(x_bits)
    n_rows = x_bits.shape[0]
    w1 = bf16_decode(w1_bits)                      # [h, d]
    w2 = bf16_decode(w2_bits)                      # [h]
    bias1 = np.zeros(w1.shape[0]) if b1 is None else np.asarray(b1, np.float64)
    want = np.arange(n_rows) if rows is None else np.asarray(rows, np.int64)
    s = np.full(n_rows, np.nan, dtype=np.float32)
    doc_rows = want[is_doc[want]]
    s[want[~is_doc[want]]] = 0.0
    chunk = 8192
    for c in range(0, len(doc_rows), chunk):
        r = doc_rows[c: c + chunk]
        x = bf16_decode(x_bits[r])                 # [m, d]
        u = x @ w1.T + bias1                        # hidden pre-activation
        z = gelu(u) @ w2 + float(b2)                # gate logit
        s[r] = logsigmoid(z).astype(np.float32)
    return s


# ---------------------------------------------------------------------------
# top-K (same section: "a top-K selector keeps the highest-scoring tokens";
# "only the document part of the prompt is prunable, the question is never
# pruned")
# ---------------------------------------------------------------------------


def _rank_key(value: float, index: int):
    """Sort key for 'larger score first, then lower index'.  -0.0 and +0.0
    compare equal (float comparison); NaN ranks after every number,
    including -inf."""
    if math.isnan(value):
        return (1, 0.0, index)
    return (0, -value, index)


def topk_select(s: np.ndarray, cu_seqlens: Sequence[int], n_doc: Sequence[int],
                k: Sequence[int]):
    """Kept rows per sequence.

    Returns (kept_idx int32 [sum T_b], cu_kept int32 [B+1]).  For sequence b
    the kept list is the min(k_b, n_doc_b) document rows with the largest
    score (ties: lower row index first), in ascending row order, followed by
    every question row in order.  Row ids are global (packed) row numbers.
    A min-heap of size K keeps the best candidates while scanning the
    document (heapq.nsmallest over the rank key)."""
    s = np.asarray(s, dtype=np.float32)
    kept, cu = [], [0]
    for b in range(len(n_doc)):
        lo = int(cu_seqlens[b])
        hi = int(cu_seqlens[b + 1])
        nd = int(n_doc[b])
        kb = int(k[b])
        if kb < 0:
            raise ValueError("negative budget")
        ke = min(kb, nd)
        vals = s[lo: lo + nd].tolist()
        best = heapq.nsmallest(ke, range(nd), key=lambda j: _rank_key(vals[j], j))
        doc = sorted(lo + j for j in best)
        kept.extend(doc)
        kept.extend(range(lo + nd, hi))
        cu.append(len(kept))
    return np.asarray(kept, dtype=np.int32), np.asarray(cu, dtype=np.int32)


def topk_select_masked(s: np.ndarray, cu_seqlens: Sequence[int], prunable: np.ndarray,
                       k: Sequence[int]):
    """Kept rows per sequence with general prunable spans.

    Returns (kept_idx int32 [sum T_b], cu_kept int32 [B+1], n_prunable int32
    [B]).  For sequence b: the min(k_b, n_prunable_b) prunable rows with the
    largest score (ties: lower row index first), together with every row that
    is not prunable, all in ascending row order."""
    s = np.asarray(s, dtype=np.float32)
    prunable = np.asarray(prunable).astype(bool)
    kept, cu, n_prun = [], [0], []
    for b in range(len(k)):
        lo = int(cu_seqlens[b])
        hi = int(cu_seqlens[b + 1])
        kb = int(k[b])
        if kb < 0:
            raise ValueError("negative budget")
        cand = [r for r in range(lo, hi) if prunable[r]]
        ke = min(kb, len(cand))
        best = heapq.nsmallest(ke, cand, key=lambda r: _rank_key(float(s[r]), r))
        fixed = [r for r in range(lo, hi) if not prunable[r]]
        kept.extend(sorted(best + fixed))
        cu.append(len(kept))
        n_prun.append(len(cand))
    return (np.asarray(kept, dtype=np.int32), np.asarray(cu, dtype=np.int32),
            np.asarray(n_prun, dtype=np.int32))


# ---------------------------------------------------------------------------
# gather (third phase: "layers above L process only those K tokens and never
# create KV entries for the pruned ones")
# ---------------------------------------------------------------------------


def gather_kept(x_bits: np.ndarray, s: np.ndarray, cu_seqlens: Sequence[int],
                kept_idx: np.ndarray, cu_kept: Sequence[int]):
    """x_kept = X[kept_idx] (bit copies), pos_kept = position of each kept
    row inside its own sequence, s_kept = s[kept_idx]."""
    kept_idx = np.asarray(kept_idx, dtype=np.int64)
    x_kept = np.asarray(x_bits)[kept_idx]
    pos = np.empty(len(kept_idx), dtype=np.int32)
    for b in range(len(cu_kept) - 1):
        a, e = int(cu_kept[b]), int(cu_kept[b + 1])
        pos[a:e] = kept_idx[a:e] - int(cu_seqlens[b])
    s_kept = np.asarray(s, dtype=np.float32)[kept_idx]
    return x_kept, pos, s_kept


# ---------------------------------------------------------------------------
# RoPE at original positions (rotate-half convention, theta = 1e6)
# ---------------------------------------------------------------------------


def rope(x: np.ndarray, pos: np.ndarray, theta: float = 1.0e6) -> np.ndarray:
    """Rotate-half rotary embedding of x [T, H, D] (float64) at positions
    pos [T]: with i < D/2, inv_freq_i = theta^(-2i/D), a = pos * inv_freq_i,
    out[i] = x[i] cos a - x[i + D/2] sin a and
    out[i + D/2] = x[i + D/2] cos a + x[i] sin a."""
    x = np.asarray(x, dtype=np.float64)
    d = x.shape[-1]
    half = d // 2
    inv_freq = theta ** (-2.0 * np.arange(half, dtype=np.float64) / d)
    ang = np.asarray(pos, dtype=np.float64)[:, None] * inv_freq[None, :]   # [T, D/2]
    c = np.cos(ang)[:, None, :]
    sn = np.sin(ang)[:, None, :]
    x1, x2 = x[..., :half], x[..., half:]
    return np.concatenate([x1 * c - x2 * sn, x2 * c + x1 * sn], axis=-1)


# ---------------------------------------------------------------------------
# token-gated attention ("What is token-gated attention?": the kept token's
# score becomes a bias on the attention logits above the gate, refined by a
# learnable per-head gain and a learnable temperature)
# ---------------------------------------------------------------------------


def gated_attention(q_bits: np.ndarray, k_bits: np.ndarray, v_bits: np.ndarray,
                    pos: np.ndarray, s_kept: np.ndarray, gain: np.ndarray,
                    tau: float, cu_kept: Sequence[int], theta: float = 1.0e6,
                    rows: Optional[np.ndarray] = None, q_is_f64: bool = False):
    """Attention over the kept tokens.

    q [T, hq, D], k and v [T, hkv, D] (bf16 bits, or float64 with
    ``q_is_f64``); pos [T] original positions; s_kept [T] gate scores;
    gain [hq]; tau scalar; cu_kept [B+1] sequence boundaries.

    For each requested query row i of sequence b and head h:
      logit_j = (q'_i,h . k'_j,g) / (sqrt(D) tau) + gain_h s_j for every kept
      j of sequence b with pos_j <= pos_i, g = floor(h / (hq / hkv));
      p = softmax(logit); o_i,h = sum_j p_j v_j,g; lse_i,h = log sum_j exp(logit_j).
    Returns (o float64 [T, hq, D], lse float64 [hq, T]); rows not requested
    are NaN."""
    dec = (lambda a: np.asarray(a, np.float64)) if q_is_f64 else bf16_decode
    k, v = dec(k_bits), dec(v_bits)
    t, hq, d = np.asarray(q_bits).shape
    hkv = k.shape[1]
    group = hq // hkv
    pos = np.asarray(pos, dtype=np.int64)
    s_kept = np.asarray(s_kept, dtype=np.float64)
    gain = np.asarray(gain, dtype=np.float64)
    kr = rope(k, pos, theta)
    scale = 1.0 / (math.sqrt(d) * float(tau))
    seq_of = np.empty(t, dtype=np.int64)
    for b in range(len(cu_kept) - 1):
        seq_of[int(cu_kept[b]): int(cu_kept[b + 1])] = b
    want = np.arange(t) if rows is None else np.asarray(rows, dtype=np.int64)
    o = np.full((t, hq, d), np.nan)
    lse = np.full((hq, t), np.nan)
    for i in want:
        qr_i = rope(dec(np.asarray(q_bits)[i:i + 1]), pos[i:i + 1], theta)[0]   # [hq, D]
        b = seq_of[i]
        lo, hi = int(cu_kept[b]), int(cu_kept[b + 1])
        js = np.arange(lo, hi)
        js = js[pos[lo:hi] <= pos[i]]              # causal on original positions
        for h in range(hq):
            g = h // group
            logit = (kr[js, g, :] @ qr_i[h, :]) * scale + gain[h] * s_kept[js]
            m = logit.max()
            e = np.exp(logit - m)
            den = e.sum()
            o[i, h, :] = (e / den) @ v[js, g, :]
            lse[h, i] = m + math.log(den)
    return o, lse


def gated_attention_bwd(q_bits: np.ndarray, k_bits: np.ndarray, v_bits: np.ndarray,
                        pos: np.ndarray, s_kept: np.ndarray, gain: np.ndarray, tau: float,
                        cu_kept: Sequence[int], do_bits: np.ndarray, theta: float = 1.0e6,
                        q_is_f64: bool = False, block: int = 512, scales: bool = False):
    """Gradient of L = sum_{i,h} dO_i,h . o_i,h with respect to the score-side
    parameters of token-gated attention: the kept scores s, the per-head
    gains and the temperature (the path from the attention loss back to the
    gate, "What is token-gated attention?": the score enters the logits as
    gain_h s_j, and the temperature divides q.k).

    Same inputs as ``gated_attention`` plus dO [T, hq, D] (bf16 bits, or
    float64 with ``q_is_f64``).  Per sequence and head h, with the logits
    and P = softmax of ``gated_attention`` (rows over kept keys j with
    pos_j <= pos_i):
      dP_ij = dO_i . v_j,   D_i = sum_j P_ij dP_ij,   dl_ij = P_ij (dP_ij - D_i)
      ds_j   += gain_h sum_i dl_ij
      dgain_h = sum_ij s_j dl_ij
      dtau   += sum_ij dl_ij * (-(q'_i . k'_j) / (sqrt(D) tau^2))
    A key whose score is infinite has P = 0 in every row, and its s_j dl_ij
    terms are taken as 0.  Query rows are taken ``block`` at a time (each row
    is independent).  Returns (ds float64 [T], dgain float64 [hq], dtau).

    With ``scales`` it also returns the magnitudes of the summed terms, the
    natural size of a rounding error in each sum (used by tests for their
    bounds; they change nothing above): sum_h |gain_h| sum_i |dl_ij| per key,
    sum_ij |s_j dl_ij| per head, and sum |dl_ij q'_i . k'_j| / (sqrt(D) tau^2)."""
    dec = (lambda a: np.asarray(a, np.float64)) if q_is_f64 else bf16_decode
    q, k, v, do = dec(q_bits), dec(k_bits), dec(v_bits), dec(do_bits)
    t, hq, d = q.shape
    hkv = k.shape[1]
    group = hq // hkv
    pos = np.asarray(pos, dtype=np.int64)
    s_kept = np.asarray(s_kept, dtype=np.float64)
    gain = np.asarray(gain, dtype=np.float64)
    tau = float(tau)
    qr = rope(q, pos, theta)
    kr = rope(k, pos, theta)
    ds = np.zeros(t)
    dgain = np.zeros(hq)
    dtau = 0.0
    ds_mag = np.zeros(t)
    dg_mag = np.zeros(hq)
    dtau_mag = 0.0
    for b in range(len(cu_kept) - 1):
        lo, hi = int(cu_kept[b]), int(cu_kept[b + 1])
        if hi <= lo:
            continue
        ps = pos[lo:hi]
        s_b = s_kept[lo:hi]
        for h in range(hq):
            g = h // group
            kh, vh = kr[lo:hi, g, :], v[lo:hi, g, :]
            col = np.zeros(hi - lo)          # sum_i dl_ij for this head
            col_mag = np.zeros(hi - lo)
            for r0 in range(lo, hi, block):
                r1 = min(hi, r0 + block)
                qk = qr[r0:r1, h, :] @ kh.T                          # [rows, keys]
                logit = qk / (math.sqrt(d) * tau) + gain[h] * s_b[None, :]
                visible = ps[None, :] <= pos[r0:r1, None]
                logit = np.where(visible, logit, -np.inf)
                m = logit.max(axis=1, keepdims=True)
                m = np.where(np.isfinite(m), m, 0.0)
                e = np.exp(logit - m)
                den = e.sum(axis=1, keepdims=True)
                p = np.divide(e, den, out=np.zeros_like(e), where=den > 0)
                dp = do[r0:r1, h, :] @ vh.T
                delta = (p * dp).sum(axis=1, keepdims=True)
                dl = p * (dp - delta)
                col += dl.sum(axis=0)
                dtau += float((dl * (-qk / (math.sqrt(d) * tau * tau))).sum())
                if scales:
                    col_mag += np.abs(dl).sum(axis=0)
                    dtau_mag += float(np.abs(dl * qk).sum()) / (math.sqrt(d) * tau * tau)
            ds[lo:hi] += gain[h] * col
            use = np.isfinite(s_b) & (col != 0.0)
            dgain[h] += float((s_b[use] * col[use]).sum())
            if scales:
                ds_mag[lo:hi] += abs(gain[h]) * col_mag
                dg_mag[h] += float(np.abs(s_b[use] * col_mag[use]).sum())
    if scales:
        return ds, dgain, dtau, ds_mag, dg_mag, dtau_mag
    return ds, dgain, dtau


# ---------------------------------------------------------------------------
# pruned Gated DeltaNet (TokenGate prunes the Gated DeltaNet layers of the
# hybrid Qwen3.5 model as well as its attention layers; the layer itself is
# the gated delta rule of Gated DeltaNet, Yang, Kautz and Hatamizadeh, 2024)
# ---------------------------------------------------------------------------


def gated_delta_scan(q_bits: np.ndarray, k_bits: np.ndarray, v_bits: np.ndarray, g: np.ndarray,
                     beta: np.ndarray, cu_kept: Sequence[int], scale: Optional[float] = None,
                     initial_state: Optional[np.ndarray] = None, q_is_f64: bool = False,
                     l2_eps: float = 1e-6):
    """The gated delta rule over the kept tokens of each sequence.

    q, k [T, hk, d_k] and v [T, hv, d_v] (bf16 bits, or float64 with
    ``q_is_f64``); g [T, hv] log-decays (alpha = exp(g), g <= 0); beta [T, hv]
    write strengths in [0, 1]; cu_kept [B+1].  Value head h reads q/k head
    h // (hv / hk).  Per sequence and value head, from S = initial_state
    (zero when None), token by token in order:
      k^ = k / sqrt(|k|^2 + eps), q^ = scale q / sqrt(|q|^2 + eps)
      S  = exp(g) (S - beta (S k^) k^T) + beta v k^T
      o  = S q^
    scale defaults to 1 / sqrt(d_k).  Returns (o float64 [T, hv, d_v],
    final states float64 [B, hv, d_v, d_k])."""
    dec = (lambda a: np.asarray(a, np.float64)) if q_is_f64 else bf16_decode
    q, k, v = dec(q_bits), dec(k_bits), dec(v_bits)
    t, hk, dk = q.shape
    hv, dv = v.shape[1], v.shape[2]
    rep = hv // hk
    g = np.asarray(g, np.float64)
    beta = np.asarray(beta, np.float64)
    scale = 1.0 / math.sqrt(dk) if scale is None else float(scale)
    nb = len(cu_kept) - 1
    o = np.zeros((t, hv, dv))
    states = np.zeros((nb, hv, dv, dk))
    for b in range(nb):
        lo, hi = int(cu_kept[b]), int(cu_kept[b + 1])
        for h in range(hv):
            S = np.zeros((dv, dk)) if initial_state is None else np.array(initial_state[b, h], np.float64)
            kh = h // rep
            for i in range(lo, hi):
                kk = k[i, kh] / math.sqrt(float(k[i, kh] @ k[i, kh]) + l2_eps)
                qq = scale * q[i, kh] / math.sqrt(float(q[i, kh] @ q[i, kh]) + l2_eps)
                S = math.exp(g[i, h]) * (S - beta[i, h] * np.outer(S @ kk, kk)) + beta[i, h] * np.outer(v[i, h], kk)
                o[i, h] = S @ qq
            states[b, h] = S
    return o, states


# ---------------------------------------------------------------------------
# stacked layer for the long-context workload
# ---------------------------------------------------------------------------


def project_qkv(x: np.ndarray, w_qkv_bits: np.ndarray, hq: int, hkv: int, d_head: int):
    """qkv = x W_qkv^T split into q [T, hq, D], k [T, hkv, D], v [T, hkv, D]
    (float64; x is float64 [T, d])."""
    w = bf16_decode(w_qkv_bits)
    qkv = np.asarray(x, np.float64) @ w.T
    t = qkv.shape[0]
    nq, nk = hq * d_head, hkv * d_head
    return (qkv[:, :nq].reshape(t, hq, d_head),
            qkv[:, nq:nq + nk].reshape(t, hkv, d_head),
            qkv[:, nq + nk:].reshape(t, hkv, d_head))


def stacked_layer(x: np.ndarray, w_qkv_bits: np.ndarray, w_o_bits: np.ndarray,
                  pos: np.ndarray, s_kept: np.ndarray, gain: np.ndarray, tau: float,
                  cu_kept: Sequence[int], hq: int, hkv: int, d_head: int,
                  theta: float = 1.0e6, rows: Optional[np.ndarray] = None):
    """One token-gated layer above the gate: x_out = x + attn(x W_qkv^T) W_o^T.
    x float64 [T, d].  Keys and values are projected for every kept row;
    outputs are computed for ``rows`` (all by default).  Returns
    (x_out float64 [T, d] with NaN outside ``rows``, o float64 [T, hq, D])."""
    q, k, v = project_qkv(x, w_qkv_bits, hq, hkv, d_head)
    o, _ = gated_attention(q, k, v, pos, s_kept, gain, tau, cu_kept, theta,
                           rows=rows, q_is_f64=True)
    w_o = bf16_decode(w_o_bits)
    t = x.shape[0]
    want = np.arange(t) if rows is None else np.asarray(rows, dtype=np.int64)
    out = np.full_like(np.asarray(x, np.float64), np.nan)
    out[want] = np.asarray(x, np.float64)[want] + o[want].reshape(len(want), hq * d_head) @ w_o.T
    return out, o
