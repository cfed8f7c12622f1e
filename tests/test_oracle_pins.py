"""Pins for the CPU oracle: each test checks the oracle against something
other than itself -- closed forms, brute force written a different way on
tiny inputs, library routines (torch SDPA in float64) and invariants -- so
that a dropped term, a flipped sign, a wrong index or a transposed operand in
``oracle/tokengate_oracle.py`` fails at least one of them."""
import json
import math
import os

import numpy as np
import pytest
import torch

import oracle
from learned_token_pruning_09_b300 import synth

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


# ---------------------------------------------------------------------------
# gate
# ---------------------------------------------------------------------------


def test_logsigmoid_closed_forms():
    ls = oracle.logsigmoid
    assert ls(np.array([0.0]))[0] == pytest.approx(-math.log(2.0), abs=1e-15)
    z = np.linspace(-30, 30, 121)
    # logsigmoid(z) - logsigmoid(-z) = z
    np.testing.assert_allclose(ls(z) - ls(-z), z, atol=1e-12)
    # sigmoid(ln 3) = 3/4
    assert ls(np.array([math.log(3.0)]))[0] == pytest.approx(math.log(0.75), abs=1e-15)
    # tails: no overflow, asymptotes
    assert ls(np.array([800.0]))[0] == 0.0 or abs(ls(np.array([800.0]))[0]) < 1e-300
    assert ls(np.array([-800.0]))[0] == pytest.approx(-800.0, rel=1e-15)
    assert ls(np.array([40.0]))[0] == pytest.approx(-math.exp(-40.0), rel=1e-12)
    assert np.all(ls(z) <= 0.0)


def test_gelu_closed_forms():
    g = oracle.gelu
    assert g(np.array([0.0]))[0] == 0.0
    u = np.linspace(-6, 6, 97)
    # GELU(u) - GELU(-u) = u (since Phi(u) + Phi(-u) = 1)
    np.testing.assert_allclose(g(u) - g(-u), u, atol=1e-14)
    # GELU(1) = Phi(1), the standard normal CDF at 1 (textbook value)
    assert g(np.array([1.0]))[0] == pytest.approx(0.8413447460685429, abs=1e-15)
    # GELU(-1) = -(1 - Phi(1))
    assert g(np.array([-1.0]))[0] == pytest.approx(-0.15865525393145707, abs=1e-15)


def _gate_bruteforce(x, w1, b1, w2, b2):
    """Pure-Python loops with the math module only."""
    out = []
    for row in x:
        z = b2
        for j in range(len(w1)):
            u = b1[j] + sum(w1[j][c] * row[c] for c in range(len(row)))
            z += w2[j] * 0.5 * u * (1.0 + math.erf(u / math.sqrt(2.0)))
        # logsigmoid via log of 1/(1+e^-z)
        out.append(math.log(1.0 / (1.0 + math.exp(-z))))
    return out


def test_gate_matches_bruteforce_tiny():
    rng = np.random.default_rng(7)
    n, d, h = 9, 8, 4
    shape = synth.custom("t", [6], [3], [2], d=d, h=h)
    x = synth.f32_to_bf16_bits(rng.standard_normal((n, d)).astype(np.float32))
    w1 = synth.f32_to_bf16_bits(rng.standard_normal((h, d)).astype(np.float32) * 0.5)
    w2 = synth.f32_to_bf16_bits(rng.standard_normal(h).astype(np.float32))
    b1 = rng.standard_normal(h).astype(np.float32)
    b2 = 0.3
    s = oracle.gate_score(x, shape.cu_seqlens, shape.n_doc, w1, b1, w2, b2)
    xf = synth.bf16_bits_to_f32(x).astype(float).tolist()
    ref = _gate_bruteforce(xf[:6], synth.bf16_bits_to_f32(w1).astype(float).tolist(),
                           b1.astype(float).tolist(),
                           synth.bf16_bits_to_f32(w2).astype(float).tolist(), b2)
    np.testing.assert_allclose(s[:6].astype(float), ref, rtol=1e-6, atol=1e-7)
    assert np.all(s[6:] == 0.0) and not np.any(np.signbit(s[6:]))


def test_gate_zero_w2_gives_logsigmoid_b2():
    shape = synth.custom("t", [40, 7], [5, 2], [4, 4], d=64, h=16)
    x = synth.residuals(shape)
    p = synth.gate_weights(shape)
    w2 = np.zeros(16, dtype=np.uint16)            # bf16 +0.0
    b2 = math.log(3.0)
    s = oracle.gate_score(x, shape.cu_seqlens, shape.n_doc, p["w1"], None, w2, b2)
    cu = shape.cu_seqlens
    for b in range(2):
        doc = s[cu[b]: cu[b] + shape.n_doc[b]]
        np.testing.assert_array_equal(doc, np.float32(math.log(0.75)))
        assert np.all(s[cu[b] + shape.n_doc[b]: cu[b + 1]] == 0.0)


def test_gate_single_hidden_unit_closed_form():
    """h = 1, W1 = e_0, w2 = 1: z = GELU(x_0) exactly."""
    d = 16
    x = synth.f32_to_bf16_bits(np.array([[1.0] + [5.0] * (d - 1),
                                         [-1.0] + [2.0] * (d - 1),
                                         [0.0] * d], dtype=np.float32))
    w1 = synth.f32_to_bf16_bits(np.eye(1, d, dtype=np.float32))
    w2 = synth.f32_to_bf16_bits(np.ones(1, np.float32))
    s = oracle.gate_score(x, [0, 3], [3], w1, None, w2, 0.0)
    phi1 = 0.8413447460685429
    expect = [-math.log1p(math.exp(-phi1)),
              -math.log1p(math.exp(-(-(1 - phi1)))),
              -math.log(2.0)]
    np.testing.assert_allclose(s.astype(float), expect, rtol=1e-7)


def test_gate_rows_subset_consistent():
    shape = synth.custom("t", [50], [6], [8], d=64, h=16)
    x = synth.residuals(shape)
    p = synth.gate_weights(shape)
    full = oracle.gate_score(x, shape.cu_seqlens, shape.n_doc, p["w1"], p["b1"], p["w2"], 0.1)
    rows = np.array([0, 3, 49, 50, 55])
    sub = oracle.gate_score(x, shape.cu_seqlens, shape.n_doc, p["w1"], p["b1"], p["w2"], 0.1, rows=rows)
    np.testing.assert_array_equal(sub[rows], full[rows])


# ---------------------------------------------------------------------------
# top-K
# ---------------------------------------------------------------------------


def _topk_by_rank_counting(s, lo, nd, k):
    """O(n^2) brute force: row j is kept iff fewer than k rows beat it, where
    i beats j when s_i > s_j, or s_i == s_j and i < j."""
    kept = []
    for j in range(nd):
        beaten = 0
        for i in range(nd):
            if s[lo + i] > s[lo + j] or (s[lo + i] == s[lo + j] and i < j):
                beaten += 1
        if beaten < k:
            kept.append(lo + j)
    return kept


@pytest.mark.parametrize("seed", range(6))
def test_topk_matches_rank_counting(seed):
    rng = np.random.default_rng(seed)
    n_doc = rng.integers(0, 60, size=3).tolist()
    n_q = rng.integers(0, 5, size=3).tolist()
    k = rng.integers(0, 70, size=3).tolist()
    shape = synth.custom("t", n_doc, n_q, k)
    cu = shape.cu_seqlens
    # values from a small set -> many exact ties, including -0.0 and +0.0
    pool = np.array([-3.5, -1.0, -0.25, -0.0, 0.0, -7.0], dtype=np.float32)
    s = pool[rng.integers(0, len(pool), size=shape.n_rows)]
    kept, cu_kept = oracle.topk_select(s, cu, n_doc, k)
    expect, ecu = [], [0]
    for b in range(3):
        expect += _topk_by_rank_counting(s, int(cu[b]), n_doc[b], k[b])
        expect += list(range(int(cu[b]) + n_doc[b], int(cu[b + 1])))
        ecu.append(len(expect))
    np.testing.assert_array_equal(kept, expect)
    np.testing.assert_array_equal(cu_kept, ecu)


def test_topk_special_cases():
    # all equal -> the first K document rows
    s = np.full(20, -1.0, np.float32)
    kept, _ = oracle.topk_select(s, [0, 20], [16], [5])
    np.testing.assert_array_equal(kept, [0, 1, 2, 3, 4, 16, 17, 18, 19])
    # a planted set of K distinct maxima -> exactly that set
    rng = np.random.default_rng(3)
    s = -rng.uniform(1, 2, 100).astype(np.float32)
    plant = np.array([97, 5, 44, 60, 12])
    s[plant] = -np.array([0.1, 0.2, 0.3, 0.4, 0.5], np.float32)
    kept, cu = oracle.topk_select(s, [0, 100], [100], [5])
    np.testing.assert_array_equal(kept, np.sort(plant))
    # K >= n_doc keeps the whole document; K = 0 keeps the question only
    kept, cu = oracle.topk_select(s, [0, 100], [90], [1000])
    np.testing.assert_array_equal(kept, np.arange(100))
    kept, cu = oracle.topk_select(s, [0, 100], [90], [0])
    np.testing.assert_array_equal(kept, np.arange(90, 100))
    # +0.0 and -0.0 tie: the lower index wins
    s = np.array([-1.0, 0.0, -0.0, -2.0], np.float32)
    s2 = np.array([-1.0, -0.0, 0.0, -2.0], np.float32)
    assert oracle.topk_select(s, [0, 4], [4], [1])[0].tolist() == [1]
    assert oracle.topk_select(s2, [0, 4], [4], [1])[0].tolist() == [1]
    # NaN ranks after every number
    s = np.array([np.nan, -5.0, np.nan, -9.0], np.float32)
    assert oracle.topk_select(s, [0, 4], [4], [2])[0].tolist() == [1, 3]
    assert oracle.topk_select(s, [0, 4], [4], [3])[0].tolist() == [0, 1, 3]
    s = np.array([np.nan, -np.inf, -1.0, np.nan], np.float32)
    assert oracle.topk_select(s, [0, 4], [4], [2])[0].tolist() == [1, 2]
    assert oracle.topk_select(s, [0, 4], [4], [3])[0].tolist() == [0, 1, 2]
    # empty document
    assert oracle.topk_select(np.zeros(3, np.float32), [0, 3], [0], [4])[0].tolist() == [0, 1, 2]


def test_topk_invariants_on_workload_draws():
    shape = synth.ragged_batch()
    shape = synth.custom("r", [n // 64 for n in shape.n_doc], shape.n_q,
                         [k // 64 for k in shape.k])
    s = synth.score_draws(shape)
    kept, cu_kept = oracle.topk_select(s, shape.cu_seqlens, shape.n_doc, shape.k)
    np.testing.assert_array_equal(cu_kept, shape.cu_kept)
    cu = shape.cu_seqlens
    for b in range(shape.batch):
        ks = kept[cu_kept[b]: cu_kept[b + 1]]
        assert np.all(np.diff(ks) > 0)
        qrows = np.arange(cu[b] + shape.n_doc[b], cu[b + 1])
        assert set(qrows) <= set(ks.tolist())
        doc_kept = ks[ks < cu[b] + shape.n_doc[b]]
        doc_all = np.arange(cu[b], cu[b] + shape.n_doc[b])
        dropped = np.setdiff1d(doc_all, doc_kept)
        if len(doc_kept) and len(dropped):
            assert s[doc_kept].min() >= s[dropped].max()
            # equality only where the index rule applies
            t = s[doc_kept].min()
            eq_kept = doc_kept[s[doc_kept] == t]
            eq_drop = dropped[s[dropped] == t]
            if len(eq_drop):
                assert eq_kept.max() < eq_drop.min()


# ---------------------------------------------------------------------------
# general prunable spans
# ---------------------------------------------------------------------------


@pytest.mark.parametrize("seed", range(4))
def test_masked_select_with_prefix_mask_is_the_document_case(seed):
    """A mask equal to each sequence's document prefix reduces the masked
    selector and gate to the document/question ones (written separately)."""
    rng = np.random.default_rng(100 + seed)
    n_doc = rng.integers(0, 80, size=4).tolist()
    n_q = rng.integers(0, 6, size=4).tolist()
    k = rng.integers(0, 90, size=4).tolist()
    shape = synth.custom("p", n_doc, n_q, k)
    cu = shape.cu_seqlens
    mask = np.zeros(shape.n_rows, np.uint8)
    for b in range(4):
        mask[cu[b]: cu[b] + n_doc[b]] = 1
    s = synth.score_draws(shape)
    kept, cu_kept = oracle.topk_select(s, cu, n_doc, k)
    kept_m, cu_m, n_prun = oracle.topk_select_masked(s, cu, mask, k)
    np.testing.assert_array_equal(kept_m, kept)
    np.testing.assert_array_equal(cu_m, cu_kept)
    np.testing.assert_array_equal(n_prun, n_doc)
    x, p = synth.residuals(shape), synth.gate_weights(shape)
    np.testing.assert_array_equal(
        oracle.gate_score_masked(x, mask, p["w1"], p["b1"], p["w2"], p["b2"]),
        oracle.gate_score(x, cu, n_doc, p["w1"], p["b1"], p["w2"], p["b2"]))


@pytest.mark.parametrize("seed", range(6))
def test_masked_select_matches_rank_counting(seed):
    """Random masks with several spans and many exact ties, against counting
    for each prunable row how many prunable rows of its sequence beat it."""
    rng = np.random.default_rng(200 + seed)
    lens = rng.integers(0, 70, size=3)
    cu = np.concatenate([[0], np.cumsum(lens)]).astype(np.int64)
    n = int(cu[-1])
    mask = (rng.random(n) < 0.6).astype(np.uint8)
    k = rng.integers(0, 50, size=3).tolist()
    pool = np.array([-3.5, -1.0, -0.25, -0.0, 0.0, -7.0], dtype=np.float32)
    s = pool[rng.integers(0, len(pool), size=n)]
    kept, cu_kept, n_prun = oracle.topk_select_masked(s, cu, mask, k)
    expect, ecu = [], [0]
    for b in range(3):
        rows = range(int(cu[b]), int(cu[b + 1]))
        cand = [r for r in rows if mask[r]]
        for r in rows:
            if not mask[r]:
                expect.append(r)
                continue
            beaten = sum(1 for i in cand if s[i] > s[r] or (s[i] == s[r] and i < r))
            if beaten < k[b]:
                expect.append(r)
        ecu.append(len(expect))
        assert n_prun[b] == len(cand)
    np.testing.assert_array_equal(kept, expect)
    np.testing.assert_array_equal(cu_kept, ecu)


def test_masked_select_special_cases():
    s = np.array([-1.0, -2.0, -0.5, -3.0, -0.1, -4.0], np.float32)
    cu = [0, 6]
    # nothing prunable: every row kept, whatever the budget
    none = np.zeros(6, np.uint8)
    assert oracle.topk_select_masked(s, cu, none, [0])[0].tolist() == list(range(6))
    assert oracle.topk_select_masked(s, cu, none, [3])[0].tolist() == list(range(6))
    # everything prunable: K = 0 keeps nothing, K >= n keeps everything
    allp = np.ones(6, np.uint8)
    assert oracle.topk_select_masked(s, cu, allp, [0])[0].tolist() == []
    assert oracle.topk_select_masked(s, cu, allp, [9])[0].tolist() == list(range(6))
    assert oracle.topk_select_masked(s, cu, allp, [2])[0].tolist() == [2, 4]
    # fixed rows interleaved with two spans keep their place in row order
    two = np.array([1, 1, 0, 1, 1, 0], np.uint8)
    assert oracle.topk_select_masked(s, cu, two, [2])[0].tolist() == [0, 2, 4, 5]
    assert oracle.topk_select_masked(s, cu, two, [1])[0].tolist() == [2, 4, 5]


def test_masked_select_invariants_on_span_draws():
    shape = synth.ragged_batch()
    shape = synth.custom("r", [n // 64 for n in shape.n_doc], shape.n_q,
                         [k // 64 for k in shape.k])
    mask = synth.prunable_spans(shape)
    s = synth.score_draws(shape)
    kept, cu_kept, n_prun = oracle.topk_select_masked(s, shape.cu_seqlens, mask, shape.k)
    cu = shape.cu_seqlens
    for b in range(shape.batch):
        ks = kept[cu_kept[b]: cu_kept[b + 1]]
        rows = np.arange(cu[b], cu[b + 1])
        assert np.all(np.diff(ks) > 0)
        fixed = rows[mask[rows] == 0]
        assert set(fixed.tolist()) <= set(ks.tolist())
        prun_kept = ks[mask[ks] == 1]
        assert len(prun_kept) == min(shape.k[b], int(n_prun[b]))
        dropped = np.setdiff1d(rows[mask[rows] == 1], prun_kept)
        if len(prun_kept) and len(dropped):
            assert s[prun_kept].min() >= s[dropped].max()


# ---------------------------------------------------------------------------
# gather
# ---------------------------------------------------------------------------


def test_gather_definition():
    shape = synth.custom("g", [10, 6], [2, 3], [4, 9])
    x = synth.residuals(shape)
    s = synth.score_draws(shape)
    kept, cu_kept = oracle.topk_select(s, shape.cu_seqlens, shape.n_doc, shape.k)
    xk, pos, sk = oracle.gather_kept(x, s, shape.cu_seqlens, kept, cu_kept)
    for i, r in enumerate(kept):
        assert np.array_equal(xk[i], x[r])
        b = 0 if r < shape.cu_seqlens[1] else 1
        assert pos[i] == r - shape.cu_seqlens[b]
        assert sk[i].tobytes() == s[r].tobytes()


# ---------------------------------------------------------------------------
# RoPE
# ---------------------------------------------------------------------------


def _rope_complex(x, pos, theta):
    """Independent form: pair (x_i, x_{i+D/2}) as a complex number times
    exp(j * pos * theta^(-2i/D))."""
    d = x.shape[-1]
    half = d // 2
    z = x[..., :half] + 1j * x[..., half:]
    freq = np.array([theta ** (-(2.0 * i) / d) for i in range(half)])
    rot = np.exp(1j * np.outer(pos, freq))[:, None, :]
    w = z * rot
    return np.concatenate([w.real, w.imag], axis=-1)


def test_rope_pins():
    rng = np.random.default_rng(11)
    x = rng.standard_normal((7, 3, 16))
    pos = np.array([0, 1, 2, 100, 4097, 131071, 65536])
    r = oracle.rope(x, pos, 1.0e6)
    np.testing.assert_allclose(r, _rope_complex(x, pos, 1.0e6), atol=1e-12)
    # position 0 is the identity
    np.testing.assert_array_equal(oracle.rope(x[:1], np.array([0]), 1e6), x[:1])
    # dimension 0 rotates by exactly pos radians
    e = np.zeros((1, 1, 16)); e[0, 0, 0] = 1.0
    r1 = oracle.rope(e, np.array([1]), 1e6)
    assert r1[0, 0, 0] == pytest.approx(math.cos(1.0), abs=1e-15)
    assert r1[0, 0, 8] == pytest.approx(math.sin(1.0), abs=1e-15)
    # relative: <R_p q, R_p' k> depends only on p' - p
    q = rng.standard_normal((1, 1, 16)); k = rng.standard_normal((1, 1, 16))
    a = np.sum(oracle.rope(q, np.array([5]), 1e6) * oracle.rope(k, np.array([12]), 1e6))
    b = np.sum(oracle.rope(q, np.array([1005]), 1e6) * oracle.rope(k, np.array([1012]), 1e6))
    assert a == pytest.approx(b, abs=1e-10)


# ---------------------------------------------------------------------------
# token-gated attention
# ---------------------------------------------------------------------------


def _attn_bruteforce(q, k, v, pos, s, gain, tau, theta):
    """Explicit full masked-softmax matrix with Python loops on tiny
    inputs (single sequence); RoPE through the complex form."""
    t, hq, d = q.shape
    hkv = k.shape[1]
    qr = _rope_complex(q, pos, theta)
    kr = _rope_complex(k, pos, theta)
    o = np.zeros((t, hq, d))
    for h in range(hq):
        g = h * hkv // hq
        for i in range(t):
            logits = []
            for j in range(t):
                if pos[j] <= pos[i]:
                    dot = sum(qr[i, h, c] * kr[j, g, c] for c in range(d))
                    logits.append((j, dot / (math.sqrt(d) * tau) + gain[h] * s[j]))
            mx = max(val for _, val in logits)
            w = [(j, math.exp(val - mx)) for j, val in logits]
            tot = sum(val for _, val in w)
            for j, val in w:
                o[i, h] += val / tot * v[j, g]
    return o


def _rand_qkv(rng, t, hq, hkv, d):
    bf = lambda a: synth.f32_to_bf16_bits(a.astype(np.float32))
    return (bf(rng.standard_normal((t, hq, d))), bf(rng.standard_normal((t, hkv, d))),
            bf(rng.standard_normal((t, hkv, d))))


def test_attention_matches_bruteforce_shuffled_positions():
    rng = np.random.default_rng(5)
    t, hq, hkv, d = 7, 4, 2, 8
    q, k, v = _rand_qkv(rng, t, hq, hkv, d)
    pos = np.array([30, 2, 17, 5, 100, 3, 64])
    s = -rng.uniform(0, 3, t)
    gain = np.array([0.5, 1.0, 1.5, 2.0])
    o, lse = oracle.gated_attention(q, k, v, pos, s, gain, 1.2, [0, t], 1e6)
    ref = _attn_bruteforce(oracle.bf16_decode(q), oracle.bf16_decode(k), oracle.bf16_decode(v),
                           pos, s, gain, 1.2, 1e6)
    np.testing.assert_allclose(o, ref, atol=1e-12)


def _dense_causal_sdpa(q, k, v, pos, theta, tau=1.0):
    """Dense causal attention by torch's scaled_dot_product_attention in
    float64, GQA by repeating KV heads (head h reads KV head h // G)."""
    qr = torch.from_numpy(_rope_complex(q, pos, theta)).permute(1, 0, 2)
    kr = torch.from_numpy(_rope_complex(k, pos, theta)).permute(1, 0, 2)
    vv = torch.from_numpy(v).permute(1, 0, 2)
    g = q.shape[1] // k.shape[1]
    kr = kr.repeat_interleave(g, dim=0)
    vv = vv.repeat_interleave(g, dim=0)
    o = torch.nn.functional.scaled_dot_product_attention(
        qr, kr, vv, is_causal=True, scale=1.0 / (math.sqrt(q.shape[-1]) * tau))
    return o.permute(1, 0, 2).numpy()


@pytest.mark.parametrize("hq,hkv", [(4, 2), (4, 4), (8, 2)])
def test_attention_reduces_to_dense_causal(hq, hkv):
    """K = N, gain 0 (or s = 0) and tau = 1: plain causal attention."""
    rng = np.random.default_rng(hq * 10 + hkv)
    t, d = 40, 16
    q, k, v = _rand_qkv(rng, t, hq, hkv, d)
    pos = np.arange(t)
    s = -rng.uniform(0, 4, t)
    qf, kf, vf = (oracle.bf16_decode(a) for a in (q, k, v))
    o0, _ = oracle.gated_attention(q, k, v, pos, s, np.zeros(hq), 1.0, [0, t], 1e6)
    o1, _ = oracle.gated_attention(q, k, v, pos, np.zeros(t), rng.uniform(0.5, 2, hq), 1.0, [0, t], 1e6)
    ref = _dense_causal_sdpa(qf, kf, vf, pos, 1e6)
    np.testing.assert_allclose(o0, ref, atol=1e-12)
    np.testing.assert_allclose(o1, ref, atol=1e-12)
    # tau: same as zero-bias attention with the softmax scale divided by tau
    o2, _ = oracle.gated_attention(q, k, v, pos, s, np.zeros(hq), 1.7, [0, t], 1e6)
    np.testing.assert_allclose(o2, _dense_causal_sdpa(qf, kf, vf, pos, 1e6, tau=1.7), atol=1e-12)


def test_attention_bias_invariants():
    rng = np.random.default_rng(21)
    t, hq, hkv, d = 24, 2, 1, 16
    q, k, v = _rand_qkv(rng, t, hq, hkv, d)
    pos = np.sort(rng.choice(1000, t, replace=False))
    gain = np.array([0.7, 1.9])
    # a constant score shifts every logit of a row equally: no effect
    c1, _ = oracle.gated_attention(q, k, v, pos, np.full(t, -0.3), gain, 1.1, [0, t])
    c2, _ = oracle.gated_attention(q, k, v, pos, np.full(t, -5.0), gain, 1.1, [0, t])
    np.testing.assert_allclose(c1, c2, atol=1e-12)
    # a key with a huge negative bias drops out: same as removing it
    s = -rng.uniform(0, 1, t)
    s_big = s.copy(); s_big[3] = -1e6
    ob, _ = oracle.gated_attention(q, k, v, pos, s_big, gain, 1.1, [0, t])
    keep = np.array([i for i in range(t) if i != 3])
    orm, _ = oracle.gated_attention(q[keep], k[keep], v[keep], pos[keep], s[keep], gain, 1.1, [0, t - 1])
    np.testing.assert_allclose(ob[keep], orm, atol=1e-12)
    # a larger score means more weight: with q = 0 the output is the
    # score-weighted mean: weights exp(g_h s_j) / sum
    zero = np.zeros_like(q)
    oz, lse = oracle.gated_attention(zero, k, v, pos, s, gain, 1.1, [0, t])
    vf = oracle.bf16_decode(v)
    for h in range(hq):
        w = np.exp(gain[h] * s)
        i = t - 1
        np.testing.assert_allclose(oz[i, h], (w[:, None] * vf[:, 0]).sum(0) / w.sum(), atol=1e-12)
        assert lse[h, i] == pytest.approx(math.log(w.sum()), abs=1e-12)


def test_attention_permutation_and_shift_consistency():
    rng = np.random.default_rng(8)
    t, hq, hkv, d = 20, 4, 2, 16
    q, k, v = _rand_qkv(rng, t, hq, hkv, d)
    pos = np.sort(rng.choice(500, t, replace=False))
    s = -rng.uniform(0, 2, t)
    gain = rng.uniform(0.5, 2, hq)
    o, lse = oracle.gated_attention(q, k, v, pos, s, gain, 0.95, [0, t])
    perm = rng.permutation(t)
    op, lsep = oracle.gated_attention(q[perm], k[perm], v[perm], pos[perm], s[perm], gain, 0.95, [0, t])
    np.testing.assert_allclose(op, o[perm], atol=1e-12)
    np.testing.assert_allclose(lsep, lse[:, perm], atol=1e-12)
    # RoPE is relative: shifting every position leaves the output unchanged
    os_, _ = oracle.gated_attention(q, k, v, pos + 777, s, gain, 0.95, [0, t])
    np.testing.assert_allclose(os_, o, atol=1e-9)


def test_attention_varlen_equals_separate_calls():
    rng = np.random.default_rng(9)
    lens = [5, 11, 1]
    t = sum(lens)
    q, k, v = _rand_qkv(rng, t, 2, 1, 8)
    pos = np.concatenate([np.arange(n) * 3 for n in lens])
    s = -rng.uniform(0, 2, t)
    gain = np.array([1.0, 1.5])
    cu = np.concatenate([[0], np.cumsum(lens)])
    o, _ = oracle.gated_attention(q, k, v, pos, s, gain, 1.0, cu)
    for b in range(3):
        a, e = cu[b], cu[b + 1]
        ob, _ = oracle.gated_attention(q[a:e], k[a:e], v[a:e], pos[a:e], s[a:e], gain, 1.0, [0, e - a])
        np.testing.assert_allclose(o[a:e], ob, atol=1e-13)


def test_attention_golden_orthogonal_example():
    """Hand-derived example (tests/golden/attention_orthogonal.json)."""
    with open(os.path.join(GOLDEN, "attention_orthogonal.json")) as f:
        case = json.load(f)
    q = np.array(case["q"], float)[:, None, :]
    k = np.array(case["k"], float)[:, None, :]
    v = np.array(case["v"], float)[:, None, :]
    o, lse = oracle.gated_attention(q, k, v, np.array(case["pos"]), np.array(case["s"]),
                                    np.array([case["gain"]]), case["tau"], [0, len(case["pos"])],
                                    q_is_f64=True)
    np.testing.assert_allclose(o[:, 0, :], np.array(case["o"]), atol=1e-14)
    np.testing.assert_allclose(lse[0], np.array(case["lse"]), atol=1e-14)


# ---------------------------------------------------------------------------
# stacked layer
# ---------------------------------------------------------------------------


def test_stacked_layer_loops():
    rng = np.random.default_rng(2)
    t, dm, hq, hkv, dh = 6, 8, 2, 1, 4
    x = rng.standard_normal((t, dm))
    wqkv = synth.f32_to_bf16_bits(rng.standard_normal(((hq + 2 * hkv) * dh, dm)).astype(np.float32) * 0.3)
    wo = synth.f32_to_bf16_bits(rng.standard_normal((dm, hq * dh)).astype(np.float32) * 0.3)
    pos = np.array([0, 3, 4, 9, 10, 12])
    s = -rng.uniform(0, 1, t)
    gain = np.array([1.0, 0.6])
    out, o = oracle.stacked_layer(x, wqkv, wo, pos, s, gain, 1.05, [0, t], hq, hkv, dh)
    W = oracle.bf16_decode(wqkv)
    Wo = oracle.bf16_decode(wo)
    qkv = [[sum(x[i][c] * W[r][c] for c in range(dm)) for r in range(W.shape[0])] for i in range(t)]
    qkv = np.array(qkv)
    q = qkv[:, :hq * dh].reshape(t, hq, dh)
    k = qkv[:, hq * dh:(hq + hkv) * dh].reshape(t, hkv, dh)
    v = qkv[:, (hq + hkv) * dh:].reshape(t, hkv, dh)
    oref = _attn_bruteforce(q, k, v, pos, s, gain, 1.05, 1e6)
    np.testing.assert_allclose(o, oref, atol=1e-12)
    flat = oref.reshape(t, hq * dh)
    xref = np.array([[x[i][r] + sum(flat[i][c] * Wo[r][c] for c in range(hq * dh))
                      for r in range(dm)] for i in range(t)])
    np.testing.assert_allclose(out, xref, atol=1e-12)


# ---------------------------------------------------------------------------
# attention backward with respect to s, gain and tau
# ---------------------------------------------------------------------------


def _bwd_case(seed, t=30, hq=4, hkv=2, d=16, cu=None):
    rng = np.random.default_rng(seed)
    q = rng.standard_normal((t, hq, d))
    k = rng.standard_normal((t, hkv, d))
    v = rng.standard_normal((t, hkv, d))
    do = rng.standard_normal((t, hq, d))
    pos = np.cumsum(rng.integers(1, 5, t))
    s = -rng.uniform(0, 3, t)
    gain = rng.uniform(0.5, 2.0, hq)
    cu = [0, t] if cu is None else cu
    return q, k, v, do, pos, s, gain, 1.15, cu


def _loss(q, k, v, do, pos, s, gain, tau, cu):
    o, _ = oracle.gated_attention(q, k, v, pos, s, gain, tau, cu, q_is_f64=True)
    return float((o * do).sum())


@pytest.mark.parametrize("seed,hq,hkv,shuffle", [(1, 4, 2, False), (2, 3, 3, False), (3, 4, 1, False),
                                                 (4, 4, 2, True)])
def test_attention_bwd_matches_central_differences(seed, hq, hkv, shuffle):
    """The backward against central differences of the forward (itself
    pinned to SDPA and brute force): every ds_j, every dgain_h and dtau;
    once with positions out of row order, so that the mask is on positions."""
    q, k, v, do, pos, s, gain, tau, cu = _bwd_case(seed, t=14, hq=hq, hkv=hkv, d=8, cu=[0, 6, 14])
    if shuffle:
        pos = np.random.default_rng(seed).permutation(pos)
    ds, dg, dtau = oracle.gated_attention_bwd(q, k, v, pos, s, gain, tau, cu, do, q_is_f64=True)
    eps = 1e-6
    for j in range(len(s)):
        sp, sm = s.copy(), s.copy()
        sp[j] += eps
        sm[j] -= eps
        fd = (_loss(q, k, v, do, pos, sp, gain, tau, cu) - _loss(q, k, v, do, pos, sm, gain, tau, cu)) / (2 * eps)
        assert abs(fd - ds[j]) < 1e-7 * max(1.0, abs(fd)), (j, fd, ds[j])
    for h in range(hq):
        gp, gm = gain.copy(), gain.copy()
        gp[h] += eps
        gm[h] -= eps
        fd = (_loss(q, k, v, do, pos, s, gp, tau, cu) - _loss(q, k, v, do, pos, s, gm, tau, cu)) / (2 * eps)
        assert abs(fd - dg[h]) < 1e-7 * max(1.0, abs(fd)), (h, fd, dg[h])
    fd = (_loss(q, k, v, do, pos, s, gain, tau + eps, cu) - _loss(q, k, v, do, pos, s, gain, tau - eps, cu)) / (2 * eps)
    assert abs(fd - dtau) < 1e-7 * max(1.0, abs(fd))


def test_attention_bwd_matches_sdpa_autograd():
    """torch autograd through float64 scaled_dot_product_attention with the
    bias g_h s_j and the causal mask as an additive mask, and 1/tau folded
    into the queries."""
    q, k, v, do, pos, s, gain, tau, cu = _bwd_case(7, t=33, hq=6, hkv=2, d=16)
    ds, dg, dtau = oracle.gated_attention_bwd(q, k, v, pos, s, gain, tau, cu, do, q_is_f64=True)
    qr = torch.from_numpy(_rope_complex(q, pos, 1e6)).permute(1, 0, 2)
    kr = torch.from_numpy(_rope_complex(k, pos, 1e6)).permute(1, 0, 2).repeat_interleave(3, dim=0)
    vv = torch.from_numpy(v).permute(1, 0, 2).repeat_interleave(3, dim=0)
    st = torch.tensor(s, requires_grad=True)
    gt = torch.tensor(gain, requires_grad=True)
    tt = torch.tensor(tau, dtype=torch.float64, requires_grad=True)
    pt = torch.from_numpy(pos)
    causal = torch.where(pt[None, :] <= pt[:, None], 0.0, -math.inf).to(torch.float64)
    mask = gt[:, None, None] * st[None, None, :] + causal[None]
    o = torch.nn.functional.scaled_dot_product_attention(qr / tt, kr, vv, attn_mask=mask,
                                                         scale=1.0 / math.sqrt(q.shape[-1]))
    loss = (o.permute(1, 0, 2) * torch.from_numpy(do)).sum()
    loss.backward()
    np.testing.assert_allclose(ds, st.grad.numpy(), rtol=1e-10, atol=1e-12)
    np.testing.assert_allclose(dg, gt.grad.numpy(), rtol=1e-10, atol=1e-12)
    assert abs(dtau - float(tt.grad)) < 1e-10 * max(1.0, abs(dtau))


def test_attention_bwd_two_key_closed_form():
    """One head, two tokens: row 0 sees only itself (p = 1, nothing to
    differentiate); row 1 sees both with p = sigmoid(l1 - l0), so
    dL/dl1 = p0 p1 (a1 - a0), a_j = dO_1 . v_j, dL/dl0 = -dL/dl1."""
    rng = np.random.default_rng(11)
    d = 4
    q, k, v, do = (rng.standard_normal((2, 1, d)) for _ in range(4))
    pos = np.array([0, 1])
    s = np.array([-0.7, -1.9])
    g, tau = 1.3, 0.8
    ds, dg, dtau = oracle.gated_attention_bwd(q, k, v, pos, s, np.array([g]), tau, [0, 2], do, q_is_f64=True)
    qr = oracle.rope(q, pos)
    kr = oracle.rope(k, pos)
    qk = np.array([qr[1, 0] @ kr[0, 0], qr[1, 0] @ kr[1, 0]])
    l = qk / (math.sqrt(d) * tau) + g * s
    p1 = 1.0 / (1.0 + math.exp(l[0] - l[1]))
    p0 = 1.0 - p1
    a = np.array([do[1, 0] @ v[0, 0], do[1, 0] @ v[1, 0]])
    dl1 = p0 * p1 * (a[1] - a[0])
    np.testing.assert_allclose(ds, [-g * dl1, g * dl1], rtol=1e-12)
    np.testing.assert_allclose(dg, [s[1] * dl1 - s[0] * dl1], rtol=1e-12)
    np.testing.assert_allclose(dtau, -(qk[1] * dl1 - qk[0] * dl1) / (math.sqrt(d) * tau * tau), rtol=1e-12)


def test_attention_bwd_invariants():
    q, k, v, do, pos, s, gain, tau, cu = _bwd_case(5, t=40, cu=[0, 17, 17, 40])
    ds, dg, dtau = oracle.gated_attention_bwd(q, k, v, pos, s, gain, tau, cu, do, q_is_f64=True)
    # softmax is shift-invariant: the ds of a sequence sum to zero
    for b in range(len(cu) - 1):
        assert abs(ds[cu[b]:cu[b + 1]].sum()) < 1e-12 * max(1.0, np.abs(ds).max())
    # a score that is constant over every sequence leaves the gains without gradient
    _, dg_c, _ = oracle.gated_attention_bwd(q, k, v, pos, np.full(40, -1.3), gain, tau, cu, do, q_is_f64=True)
    np.testing.assert_allclose(dg_c, 0.0, atol=1e-12)
    # q = 0: the logits do not depend on tau
    _, _, dtau0 = oracle.gated_attention_bwd(np.zeros_like(q), k, v, pos, s, gain, tau, cu, do, q_is_f64=True)
    assert dtau0 == 0.0
    # varlen equals separate calls
    for b in range(len(cu) - 1):
        lo, hi = cu[b], cu[b + 1]
        if hi == lo:
            continue
        dsb, _, _ = oracle.gated_attention_bwd(q[lo:hi], k[lo:hi], v[lo:hi], pos[lo:hi], s[lo:hi], gain, tau,
                                               [0, hi - lo], do[lo:hi], q_is_f64=True)
        np.testing.assert_allclose(ds[lo:hi], dsb, rtol=1e-12, atol=1e-14)
    # the loss is linear in dO
    ds2, dg2, dtau2 = oracle.gated_attention_bwd(q, k, v, pos, s, gain, tau, cu, 2.5 * do, q_is_f64=True)
    np.testing.assert_allclose(ds2, 2.5 * ds, rtol=1e-12, atol=1e-14)
    np.testing.assert_allclose(dg2, 2.5 * dg, rtol=1e-12, atol=1e-14)


def test_attention_bwd_infinite_score_removes_the_key():
    """A key with score -inf is invisible for positive gains: its ds is 0 and
    every other gradient equals the one with that key deleted."""
    q, k, v, do, pos, s, gain, tau, cu = _bwd_case(9, t=20)
    do[7] = 0.0                  # row 7 itself adds no loss term, so it can be deleted
    s2 = s.copy()
    s2[7] = -np.inf
    ds, dg, dtau = oracle.gated_attention_bwd(q, k, v, pos, s2, gain, tau, cu, do, q_is_f64=True)
    keep = np.array([j for j in range(20) if j != 7])
    dsr, dgr, dtaur = oracle.gated_attention_bwd(q[keep], k[keep], v[keep], pos[keep], s[keep], gain, tau,
                                                 [0, 19], do[keep], q_is_f64=True)
    assert ds[7] == 0.0
    np.testing.assert_allclose(ds[keep], dsr, rtol=1e-10, atol=1e-12)
    np.testing.assert_allclose(dg, dgr, rtol=1e-10, atol=1e-12)
    assert abs(dtau - dtaur) < 1e-10 * max(1.0, abs(dtau))


# ---------------------------------------------------------------------------
# pruned Gated DeltaNet (gated delta rule over kept tokens)
# ---------------------------------------------------------------------------


def _unit(a):
    return a / np.linalg.norm(a, axis=-1, keepdims=True)


def test_delta_scan_orthogonal_keys_is_decayed_linear_attention():
    """Mutually orthogonal keys: the erase term never touches earlier content,
    so o_t = sum_{i<=t} exp(G_t - G_i) beta_i (k^_i . q^_t) v_i, G = cumsum(g):
    decayed linear attention, written here as one masked matrix product."""
    rng = np.random.default_rng(1)
    t, dk, dv = 12, 16, 5
    basis = np.linalg.qr(rng.standard_normal((dk, dk)))[0][:t]          # orthonormal rows
    k = (basis * rng.uniform(0.5, 3.0, (t, 1)))[:, None, :]              # any length: k is normalised
    q = rng.standard_normal((t, 1, dk))
    v = rng.standard_normal((t, 1, dv))
    g = -rng.uniform(0.0, 0.7, (t, 1))
    beta = rng.uniform(0.1, 1.0, (t, 1))
    o, _ = oracle.gated_delta_scan(q, k, v, g, beta, [0, t], scale=1.0, q_is_f64=True, l2_eps=0.0)
    G = np.cumsum(g[:, 0])
    mask = np.tril(np.exp(G[:, None] - G[None, :]))
    ref = (mask * (_unit(q[:, 0]) @ _unit(k[:, 0]).T)) @ (beta * v[:, 0])
    np.testing.assert_allclose(o[:, 0], ref, rtol=1e-12, atol=1e-13)


def test_delta_scan_overwrites_a_repeated_key():
    """alpha = 1, beta = 1: writing v2 under the key that holds v1 replaces it
    (the delta rule's overwrite), so the read returns v2 (k^ . q^)."""
    rng = np.random.default_rng(2)
    dk, dv = 8, 4
    key = rng.standard_normal(dk)
    k = np.stack([key, 2.5 * key])[:, None, :]
    q = rng.standard_normal((2, 1, dk))
    v = rng.standard_normal((2, 1, dv))
    o, S = oracle.gated_delta_scan(q, k, v, np.zeros((2, 1)), np.ones((2, 1)), [0, 2], scale=1.0,
                                   q_is_f64=True, l2_eps=0.0)
    kh = _unit(key)
    np.testing.assert_allclose(o[1, 0], v[1, 0] * (kh @ _unit(q[1, 0])), rtol=1e-12, atol=1e-14)
    np.testing.assert_allclose(S[0, 0], np.outer(v[1, 0], kh), rtol=1e-12, atol=1e-14)


def test_delta_scan_matches_unrolled_products():
    """Brute force on a tiny case: S_t = sum_{i<=t} beta_i v_i k^_i^T
    prod_{j=i+1..t} alpha_j (I - beta_j k^_j k^_j^T), the recurrence unrolled
    and multiplied in the other association."""
    rng = np.random.default_rng(3)
    t, dk, dv = 7, 5, 3
    q, k = rng.standard_normal((t, 1, dk)), rng.standard_normal((t, 1, dk))
    v = rng.standard_normal((t, 1, dv))
    g, beta = -rng.uniform(0, 0.5, (t, 1)), rng.uniform(0, 1, (t, 1))
    o, _ = oracle.gated_delta_scan(q, k, v, g, beta, [0, t], scale=0.7, q_is_f64=True, l2_eps=0.0)
    kh, qh = _unit(k[:, 0]), 0.7 * _unit(q[:, 0])
    for tt in range(t):
        S = np.zeros((dv, dk))
        for i in range(tt + 1):
            P = np.eye(dk)
            for j in range(i + 1, tt + 1):
                P = P @ (math.exp(g[j, 0]) * (np.eye(dk) - beta[j, 0] * np.outer(kh[j], kh[j])))
            S += beta[i, 0] * np.outer(v[i, 0], kh[i]) @ P
        # token i's own write carries no alpha_i (S_i = alpha_i (...) + beta_i v_i k_i^T)
        np.testing.assert_allclose(o[tt, 0], S @ qh[tt], rtol=1e-11, atol=1e-13)


def test_delta_scan_pruned_tokens_are_skipped():
    """Running every token with beta = 0 and g = 0 on the pruned ones equals
    running the kept tokens alone: a pruned token never touches the state."""
    rng = np.random.default_rng(4)
    n, hk, hv, dk, dv = 40, 2, 4, 8, 6
    q, k = rng.standard_normal((n, hk, dk)), rng.standard_normal((n, hk, dk))
    v = rng.standard_normal((n, hv, dv))
    g, beta = -rng.uniform(0, 0.5, (n, hv)), rng.uniform(0, 1, (n, hv))
    kept = np.sort(rng.choice(n, 17, replace=False))
    gz, bz = np.zeros_like(g), np.zeros_like(beta)
    gz[kept], bz[kept] = g[kept], beta[kept]
    o_all, s_all = oracle.gated_delta_scan(q, k, v, gz, bz, [0, n], q_is_f64=True)
    o_k, s_k = oracle.gated_delta_scan(q[kept], k[kept], v[kept], g[kept], beta[kept], [0, len(kept)],
                                       q_is_f64=True)
    np.testing.assert_allclose(o_all[kept], o_k, rtol=1e-12, atol=1e-13)
    np.testing.assert_allclose(s_all, s_k, rtol=1e-12, atol=1e-13)


def test_delta_scan_invariants():
    rng = np.random.default_rng(5)
    t, hk, hv, dk, dv = 30, 2, 4, 8, 6
    q, k = rng.standard_normal((t, hk, dk)), rng.standard_normal((t, hk, dk))
    v = rng.standard_normal((t, hv, dv))
    g, beta = -rng.uniform(0, 0.5, (t, hv)), rng.uniform(0, 1, (t, hv))
    cu = [0, 11, 11, 30]
    o, S = oracle.gated_delta_scan(q, k, v, g, beta, cu, q_is_f64=True, l2_eps=0.0)
    # q and k enter only through their directions
    o2, _ = oracle.gated_delta_scan(3.0 * q, 0.25 * k, v, g, beta, cu, q_is_f64=True, l2_eps=0.0)
    np.testing.assert_allclose(o2, o, rtol=1e-11, atol=1e-13)
    # linear in v from a zero state
    o3, S3 = oracle.gated_delta_scan(q, k, -2.0 * v, g, beta, cu, q_is_f64=True, l2_eps=0.0)
    np.testing.assert_allclose(o3, -2.0 * o, rtol=1e-12, atol=1e-13)
    # the default scale is 1/sqrt(d_k), and the output is linear in it
    o4, _ = oracle.gated_delta_scan(q, k, v, g, beta, cu, scale=1.0, q_is_f64=True, l2_eps=0.0)
    np.testing.assert_allclose(o4 / math.sqrt(dk), o, rtol=1e-12, atol=1e-13)
    # value head h reads q/k head h // (hv / hk): heads 2, 3 alone with q/k head 1
    o5, _ = oracle.gated_delta_scan(q[:, 1:], k[:, 1:], v[:, 2:], g[:, 2:], beta[:, 2:], cu, q_is_f64=True,
                                    l2_eps=0.0)
    np.testing.assert_allclose(o5, o[:, 2:], rtol=1e-12, atol=1e-13)
    # an empty sequence keeps its initial (zero) state; varlen equals separate calls
    assert np.all(S[1] == 0.0)
    for b in range(3):
        lo, hi = cu[b], cu[b + 1]
        if hi == lo:
            continue
        ob, sb = oracle.gated_delta_scan(q[lo:hi], k[lo:hi], v[lo:hi], g[lo:hi], beta[lo:hi], [0, hi - lo],
                                         q_is_f64=True, l2_eps=0.0)
        np.testing.assert_allclose(ob, o[lo:hi], rtol=1e-12, atol=1e-13)
        np.testing.assert_allclose(sb[0], S[b], rtol=1e-12, atol=1e-13)


def test_delta_scan_state_continues_across_calls():
    """Two calls, the second started from the first's final state, equal one
    call over the whole sequence (the chunk-to-chunk carry)."""
    rng = np.random.default_rng(6)
    t, dk, dv = 25, 8, 8
    q, k = rng.standard_normal((t, 1, dk)), rng.standard_normal((t, 1, dk))
    v = rng.standard_normal((t, 2, dv))
    g, beta = -rng.uniform(0, 0.5, (t, 2)), rng.uniform(0, 1, (t, 2))
    o, S = oracle.gated_delta_scan(q, k, v, g, beta, [0, t], q_is_f64=True)
    oa, Sa = oracle.gated_delta_scan(q[:9], k[:9], v[:9], g[:9], beta[:9], [0, 9], q_is_f64=True)
    ob, Sb = oracle.gated_delta_scan(q[9:], k[9:], v[9:], g[9:], beta[9:], [0, t - 9], initial_state=Sa,
                                     q_is_f64=True)
    np.testing.assert_allclose(np.concatenate([oa, ob]), o, rtol=1e-12, atol=1e-13)
    np.testing.assert_allclose(Sb, S, rtol=1e-12, atol=1e-13)


def _chunked_delta_scan(q, k, v, g, beta, cu, chunk, scale):
    """The gated delta rule in its chunked (WY) form, derived from the
    recurrence: within a chunk with decays gamma_i = exp(sum_{j<=i} g_j) and
    entering state S0, the pseudo-values u_i = beta_i (v_i - alpha_i S_{i-1}
    k_i) solve (I + A) U = beta V - (beta gamma K) S0^T with
    A_ij = beta_i (gamma_i / gamma_j) k_i . k_j for j < i; then
    O = (gamma Q) S0^T + (M o Q K^T) U (M_ij = gamma_i / gamma_j, j <= i) and
    S <- gamma_C S0 + U^T ((gamma_C / gamma) K)."""
    t, hk, dk = q.shape
    hv, dv = v.shape[1], v.shape[2]
    o = np.zeros((t, hv, dv))
    kh_all = _unit(k)
    qh_all = scale * _unit(q)
    for b in range(len(cu) - 1):
        for h in range(hv):
            S = np.zeros((dv, dk))
            kh = h // (hv // hk)
            for c0 in range(cu[b], cu[b + 1], chunk):
                c1 = min(cu[b + 1], c0 + chunk)
                K, Q, V = kh_all[c0:c1, kh], qh_all[c0:c1, kh], v[c0:c1, h]
                bt = beta[c0:c1, h]
                G = np.cumsum(g[c0:c1, h])
                ratio = np.exp(G[:, None] - G[None, :])
                n = c1 - c0
                A = np.tril(bt[:, None] * ratio * (K @ K.T), -1)
                Tm = np.linalg.solve(np.eye(n) + A, np.eye(n))
                U = Tm @ (bt[:, None] * V) - Tm @ ((bt * np.exp(G))[:, None] * K) @ S.T
                o[c0:c1, h] = (np.exp(G)[:, None] * Q) @ S.T + (np.tril(ratio) * (Q @ K.T)) @ U
                S = np.exp(G[-1]) * S + U.T @ (np.exp(G[-1] - G)[:, None] * K)
    return o


@pytest.mark.parametrize("chunk", [1, 4, 16, 64])
def test_delta_scan_equals_chunked_wy_form(chunk):
    """The recurrence equals its chunked form for any chunk size, on
    sequences that are not multiples of the chunk."""
    rng = np.random.default_rng(7)
    lens = [70, 1, 0, 45]
    cu = np.concatenate([[0], np.cumsum(lens)])
    t, hk, hv, dk, dv = int(cu[-1]), 2, 4, 16, 8
    q, k = rng.standard_normal((t, hk, dk)), rng.standard_normal((t, hk, dk))
    v = rng.standard_normal((t, hv, dv))
    g, beta = -rng.uniform(0, 0.5, (t, hv)), rng.uniform(0, 1, (t, hv))
    o, _ = oracle.gated_delta_scan(q, k, v, g, beta, cu, scale=0.3, q_is_f64=True, l2_eps=0.0)
    oc = _chunked_delta_scan(q, k, v, g, beta, cu, chunk, 0.3)
    np.testing.assert_allclose(oc, o, rtol=1e-10, atol=1e-12)
