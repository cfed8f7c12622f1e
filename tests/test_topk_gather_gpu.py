"""GPU parity of top-K selection and gather against the oracle: bit-exact on
identical fp32 scores, for every workload shape and the edge cases."""
import math

import numpy as np
import pytest
import torch

import oracle
from learned_token_pruning_09_b300 import synth
from tests.helpers import dev_bf16, dev_f32, dev_i32, host_bits

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def tg():
    from learned_token_pruning_09_b300 import tokengate
    return tokengate


def run_topk(tg, s, shape_cu, n_doc, k):
    cu = np.asarray(shape_cu, np.int32)
    seqlens = np.diff(cu)
    n_kept = sum(tg.kept_lengths(seqlens, n_doc, k))
    kept, cu_kept = tg.tg_topk_select(dev_f32(s), dev_i32(cu), dev_i32(n_doc), dev_i32(k),
                                      max(list(n_doc) + [0]), n_kept)
    assert tg.tg_check_device_status() == tg.TG_OK
    return kept.cpu().numpy(), cu_kept.cpu().numpy()


def check_topk(tg, s, cu, n_doc, k):
    kept, cu_kept = run_topk(tg, s, cu, n_doc, k)
    ekept, ecu = oracle.topk_select(s, cu, n_doc, k)
    np.testing.assert_array_equal(cu_kept, ecu)
    np.testing.assert_array_equal(kept, ekept)
    return kept, cu_kept


@pytest.mark.parametrize("name", ["tiny", "qwen3-1.7b-16k", "long-128k", "ragged-8"])
def test_topk_workloads_score_draws(tg, name):
    shape = synth.ALL_SHAPES[name]()
    s = synth.score_draws(shape)
    check_topk(tg, s, shape.cu_seqlens, shape.n_doc, shape.k)


@pytest.mark.parametrize("k", [1024, 4096, 8192])
def test_topk_budget_sweep_planted(tg, k):
    shape = synth.budget_32k(k)
    z = synth.planted_logits(shape)
    s = np.zeros(shape.n_rows, np.float32)
    s[: shape.n_doc[0]] = oracle.score_from_logit(z)
    check_topk(tg, s, shape.cu_seqlens, shape.n_doc, shape.k)


def test_topk_edge_cases(tg):
    rng = np.random.default_rng(1)
    # mixed batch: K=0, K>n_doc, K=n_doc, K=n_doc-1, empty document,
    # empty question, single token, all-equal scores
    n_doc = [0, 1, 7, 300, 300, 1000, 5, 64, 129, 4096]
    n_q = [3, 0, 2, 0, 5, 17, 0, 1, 64, 0]
    k = [4, 1, 0, 300, 299, 1000000, 3, 64, 100, 4095]
    cu = np.concatenate([[0], np.cumsum(np.add(n_doc, n_q))]).astype(np.int32)
    s = -np.abs(rng.normal(0, 3, cu[-1])).astype(np.float32)
    s[cu[7]: cu[7] + 64] = -1.25          # all equal
    # ties, signed zeros, infinities and NaNs
    s[cu[8]: cu[8] + 20] = np.float32(-0.0)
    s[cu[8] + 20: cu[8] + 40] = np.float32(0.0)
    s[cu[8] + 40] = -np.inf
    s[cu[8] + 41] = np.nan
    s[cu[9] + 5] = np.nan
    s[cu[9] + 9] = -np.inf
    check_topk(tg, s, cu, n_doc, k)


def test_topk_large_document_streams_from_global(tg):
    """n_doc beyond the shared-memory capacity of one cluster slice."""
    n = 450_000
    rng = np.random.default_rng(2)
    s = -np.abs(rng.standard_normal(n + 10)).astype(np.float32)
    s[rng.integers(0, n, 5000)] = -0.5    # a tie block straddling the threshold
    check_topk(tg, s, [0, n + 10], [n], [60_000])


def test_topk_all_values_identical_large(tg):
    n = 70_000
    s = np.full(n + 7, -3.0, np.float32)
    kept, _ = check_topk(tg, s, [0, n + 7], [n], [12_345])
    np.testing.assert_array_equal(kept[:12_345], np.arange(12_345))


@pytest.mark.parametrize("name", ["tiny", "qwen3-1.7b-16k", "ragged-8"])
def test_gather_bit_exact(tg, name):
    shape = synth.ALL_SHAPES[name]()
    x = synth.residuals(shape)
    s = synth.score_draws(shape)
    kept, cu_kept = oracle.topk_select(s, shape.cu_seqlens, shape.n_doc, shape.k)
    ex, epos, es = oracle.gather_kept(x, s, shape.cu_seqlens, kept, cu_kept)
    xk, pos, sk = tg.tg_gather_kept(dev_bf16(x), dev_f32(s), dev_i32(shape.cu_seqlens), dev_i32(kept),
                                    dev_i32(cu_kept), len(kept))
    assert tg.tg_check_device_status() == tg.TG_OK
    np.testing.assert_array_equal(host_bits(xk), ex)
    np.testing.assert_array_equal(pos.cpu().numpy(), epos)
    np.testing.assert_array_equal(sk.cpu().numpy().view(np.uint32), es.view(np.uint32))


@pytest.mark.parametrize("d", [8, 72, 4096])
def test_gather_widths_and_rounds(tg, d):
    """Rows of 16 bytes up to 8 KB: at d = 4096 each CTA copies its range in
    several rounds of shared-memory slots; every kept row must land exactly."""
    shape = synth.custom("gather-d%d" % d, [9000, 1, 4000, 131], [3, 0, 50, 2], [5000, 1, 3999, 1],
                         d=d, seed=4242 + d)
    x = synth.residuals(shape)
    s = synth.score_draws(shape)
    kept, cu_kept = oracle.topk_select(s, shape.cu_seqlens, shape.n_doc, shape.k)
    ex, epos, es = oracle.gather_kept(x, s, shape.cu_seqlens, kept, cu_kept)
    xk, pos, sk = tg.tg_gather_kept(dev_bf16(x), dev_f32(s), dev_i32(shape.cu_seqlens), dev_i32(kept),
                                    dev_i32(cu_kept), len(kept))
    assert tg.tg_check_device_status() == tg.TG_OK
    np.testing.assert_array_equal(host_bits(xk), ex)
    np.testing.assert_array_equal(pos.cpu().numpy(), epos)
    np.testing.assert_array_equal(sk.cpu().numpy().view(np.uint32), es.view(np.uint32))


def test_gather_invalid_id_inside_a_long_range(tg):
    """One id outside its sequence, in the middle of a range that takes
    several rounds: it is reported, and every other row is still copied."""
    shape = synth.custom("gather-bad", [20000, 7000], [0, 0], [15000, 6000], d=4096, seed=99)
    x = synth.residuals(shape)
    s = synth.score_draws(shape)
    kept, cu_kept = oracle.topk_select(s, shape.cu_seqlens, shape.n_doc, shape.k)
    bad = 7777
    kept_bad = kept.copy()
    kept_bad[bad] = 20000 + 5                    # a row of the second sequence
    ex, _, _ = oracle.gather_kept(x, s, shape.cu_seqlens, kept, cu_kept)
    xk, _, _ = tg.tg_gather_kept(dev_bf16(x), dev_f32(s), dev_i32(shape.cu_seqlens), dev_i32(kept_bad),
                                 dev_i32(cu_kept), len(kept))
    assert tg.tg_check_device_status() == tg.TG_ERR_DEVICE_INDEX
    got = host_bits(xk)
    rows = np.arange(len(kept)) != bad
    np.testing.assert_array_equal(got[rows], ex[rows])


def test_gather_positions_and_scores_only(tg):
    """Without x (positions alone) and without x_kept (positions and scores):
    no row is copied, and what is written is exact."""
    shape = synth.custom("gather-pos", [3000, 17, 900], [5, 2, 0], [1000, 17, 64], d=64, seed=91)
    x = synth.residuals(shape)
    s = synth.score_draws(shape)
    kept, cu_kept = oracle.topk_select(s, shape.cu_seqlens, shape.n_doc, shape.k)
    _, epos, es = oracle.gather_kept(x, s, shape.cu_seqlens, kept, cu_kept)
    cu, kd, ck = dev_i32(shape.cu_seqlens), dev_i32(kept), dev_i32(cu_kept)
    _, pos, _ = tg.tg_gather_kept(None, None, cu, kd, ck, len(kept), d=64, want=("pos",))
    assert tg.tg_check_device_status() == tg.TG_OK
    np.testing.assert_array_equal(pos.cpu().numpy(), epos)
    xk, pos2, sk = tg.tg_gather_kept(dev_bf16(x), dev_f32(s), cu, kd, ck, len(kept), want=("pos", "s"))
    assert tg.tg_check_device_status() == tg.TG_OK
    assert xk is None
    np.testing.assert_array_equal(pos2.cpu().numpy(), epos)
    np.testing.assert_array_equal(sk.cpu().numpy().view(np.uint32), es.view(np.uint32))


def test_gather_rejects_out_of_sequence_index(tg):
    """A kept id outside its sequence is reported, not read."""
    cu = np.array([0, 10, 20], np.int32)
    s = np.arange(20, dtype=np.float32)
    kept = np.array([1, 2, 15, 12, 19], np.int32)      # 15 belongs to sequence 1
    cu_kept = np.array([0, 3, 5], np.int32)
    x = synth.f32_to_bf16_bits(np.ones((20, 64), np.float32))
    tg.tg_gather_kept(dev_bf16(x), dev_f32(s), dev_i32(cu), dev_i32(kept), dev_i32(cu_kept), 5)
    assert tg.tg_check_device_status() == tg.TG_ERR_DEVICE_INDEX
    assert tg.tg_check_device_status() == tg.TG_OK      # cleared


# ---------------------------------------------------------------------------
# the top-K workspace: the gate's score histograms give the first two radix
# digits (the result must be the same exact selection)
# ---------------------------------------------------------------------------


def gate_then_topk(tg, shape, x, p, ws, gate_calls=1):
    cu, nd = dev_i32(shape.cu_seqlens), dev_i32(shape.n_doc)
    X = dev_bf16(x)
    for _ in range(gate_calls):
        s = tg.tg_gate_score(X, cu, nd, dev_bf16(p["w1"]), None, dev_bf16(p["w2"]), p["b2"], topk_ws=ws)
    kept, cu_kept = tg.tg_topk_select(s, cu, nd, dev_i32(shape.k), max(list(shape.n_doc) + [0]), shape.n_kept,
                                      workspace=ws)
    assert tg.tg_check_device_status() == tg.TG_OK
    return s.cpu().numpy(), kept.cpu().numpy(), cu_kept.cpu().numpy()


@pytest.mark.parametrize("case", ["tiny", "qwen3-1.7b-16k", "edges"])
def test_topk_from_gate_histograms_is_exact(tg, case):
    """Gate with the workspace, then top-K with it: bit-exact against the
    oracle's top-K of the GPU's own scores, including K = 0, K >= n_doc, an
    empty document and one-row documents; the workspace is zero afterwards,
    and a second round on the same workspace is exact again."""
    if case == "edges":
        shape = synth.custom("edges", [0, 1, 300, 300, 1000, 129, 4096, 255, 256],
                             [5, 3, 0, 17, 64, 1, 64, 9, 2], [4, 1, 0, 300, 999, 64, 4000, 1, 255],
                             d=256, h=64, seed=77)
    else:
        shape = synth.ALL_SHAPES[case]()
    x, p = synth.residuals(shape), synth.gate_weights(shape)
    ws = tg.tg_topk_workspace(shape.batch)
    for _ in range(2):
        s, kept, cu_kept = gate_then_topk(tg, shape, x, p, ws)
        ekept, ecu = oracle.topk_select(s, shape.cu_seqlens, shape.n_doc, shape.k)
        np.testing.assert_array_equal(cu_kept, ecu)
        np.testing.assert_array_equal(kept, ekept)
        assert int(ws.count_nonzero()) == 0


def test_topk_stale_histograms_fall_back_exactly(tg):
    """Two gate calls into one workspace before the top-K (the counts then
    exceed n_doc): the selection takes the four radix passes and is still
    exact, and it leaves the workspace zero, so the next round is exact on
    the histogram path again."""
    shape = synth.custom("stale", [3000, 20, 700], [40, 5, 0], [900, 3, 700], d=256, h=64, seed=78)
    x, p = synth.residuals(shape), synth.gate_weights(shape)
    ws = tg.tg_topk_workspace(shape.batch)
    for calls in (2, 1):
        s, kept, cu_kept = gate_then_topk(tg, shape, x, p, ws, gate_calls=calls)
        ekept, ecu = oracle.topk_select(s, shape.cu_seqlens, shape.n_doc, shape.k)
        np.testing.assert_array_equal(kept, ekept)
        np.testing.assert_array_equal(cu_kept, ecu)
        assert int(ws.count_nonzero()) == 0


def test_topk_workspace_without_gate_histograms(tg):
    """A workspace with no gate counts in it (scores from elsewhere): exact."""
    shape = synth.long_128k()
    s = synth.score_draws(shape)
    ws = tg.tg_topk_workspace(shape.batch)
    kept, cu_kept = tg.tg_topk_select(dev_f32(s), dev_i32(shape.cu_seqlens), dev_i32(shape.n_doc),
                                      dev_i32(shape.k), max(shape.n_doc), shape.n_kept, workspace=ws)
    assert tg.tg_check_device_status() == tg.TG_OK
    ekept, ecu = oracle.topk_select(s, shape.cu_seqlens, shape.n_doc, shape.k)
    np.testing.assert_array_equal(kept.cpu().numpy(), ekept)
    assert int(ws.count_nonzero()) == 0


# White-box: the workspace filled on the host with the histograms the gate
# would count (coarse bins of the top 8 bits of each score's order key, fine
# bins of the top 16 bits at the transposed slot ((f & 255) << 8) | (f >> 8)),
# for score vectors the gate would rarely produce: many keys tied in, or
# sharing, the K-th key's 16-bit bin.

def order_keys(s):
    b = np.asarray(s, np.float32).view(np.uint32).copy()
    b[(b & 0x7FFFFFFF) > 0x7F800000] = 0          # NaN
    b[b == 0x80000000] = 0                          # -0 as +0
    return np.where(b & 0x80000000, ~b, b | 0x80000000).astype(np.uint32)


def host_histograms(s, cu, n_doc):
    ws = np.zeros((len(n_doc), 256 + 65536), np.uint32)
    for b, nd in enumerate(n_doc):
        keys = order_keys(s[cu[b]: cu[b] + nd])
        np.add.at(ws[b], keys >> 24, 1)
        f = keys >> 16
        np.add.at(ws[b], 256 + (((f & 255) << 8) | (f >> 8)), 1)
    return ws


def tied_scores(rng, nd, k, n_tied, n_near, contiguous=False):
    """Scores spread evenly over 24,576 of the 16-bit bins (positive floats
    with random bit patterns, about 5 per bin at 131k rows), then n_tied rows
    set to one value v with k - n_tied // 2 other rows above it (so the K-th
    key is v and only some of the ties are taken), and n_near rows set a few
    ulps above or below v (the same 16-bit bin, other keys).  `contiguous`
    puts those rows in one run (one slice of the selector then holds them
    all) instead of scattering them."""
    s = rng.integers(0x10000000, 0x70000000, nd, dtype=np.int64).astype(np.uint32).view(np.float32)
    if contiguous:
        rows = int(rng.integers(0, nd - n_tied - n_near)) + np.arange(n_tied + n_near)
    else:
        rows = rng.choice(nd, n_tied + n_near, replace=False)
    rest = np.setdiff1d(np.arange(nd), rows)
    above = k - n_tied // 2
    v = np.sort(s[rest])[::-1][above]                 # `above` other rows lie strictly above v
    s[rows[:n_tied]] = v
    near = v.view(np.int32) + rng.integers(-3, 4, n_near).astype(np.int32)
    s[rows[n_tied:]] = near.view(np.float32)
    return s


def kth_bin_sizes(s, cu, n_doc, ks):
    out = []
    for b, (nd, k) in enumerate(zip(n_doc, ks)):
        keys = order_keys(s[cu[b]: cu[b] + nd])
        kth = np.sort(keys)[::-1][min(k, nd) - 1]
        out.append(int(np.sum((keys >> 16) == (kth >> 16))))
    return out


@pytest.mark.parametrize("n_tied,n_near,contiguous", [(1, 0, False), (40, 0, False), (200, 30, False),
                                                      (300, 0, False), (2000, 100, False), (200, 0, True),
                                                      (300, 0, True), (3000, 50, True)])
def test_topk_histogram_start_with_ties(tg, n_tied, n_near, contiguous):
    """The first two digits from the histograms, then the last two radix
    passes over many keys in the K-th key's 16-bit bin, exact ties among
    them scattered over the selector's slices or in one run inside one
    slice: bit-exact, ties taken lowest row first across the slices."""
    rng = np.random.default_rng(1000 + n_tied + contiguous)
    n_doc = [131_008, 5_000, 700]
    n_q = [64, 3, 0]
    ks = [8_192, 1_000, 300]
    cu = np.concatenate([[0], np.cumsum(np.array(n_doc) + np.array(n_q))]).astype(np.int32)
    s = np.zeros(int(cu[-1]), np.float32)
    for b in range(3):
        s[cu[b]: cu[b] + n_doc[b]] = tied_scores(rng, n_doc[b], ks[b], min(n_tied, n_doc[b] // 8),
                                                    min(n_near, n_doc[b] // 8), contiguous)
        s[cu[b] + n_doc[b]: cu[b + 1]] = rng.standard_normal(n_q[b])
    print("keys in the K-th key's 16-bit bin:", kth_bin_sizes(s, cu, n_doc, ks))
    ws = torch.from_numpy(host_histograms(s, cu, n_doc).reshape(-1).view(np.uint8)).cuda()
    n_kept = sum(min(k, n) + q for k, n, q in zip(ks, n_doc, n_q))
    kept, cu_kept = tg.tg_topk_select(dev_f32(s), dev_i32(cu), dev_i32(n_doc), dev_i32(ks), max(n_doc), n_kept,
                                      workspace=ws)
    assert tg.tg_check_device_status() == tg.TG_OK
    ekept, ecu = oracle.topk_select(s, cu, n_doc, ks)
    np.testing.assert_array_equal(cu_kept.cpu().numpy(), ecu)
    np.testing.assert_array_equal(kept.cpu().numpy(), ekept)
    assert int(ws.count_nonzero()) == 0
