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
