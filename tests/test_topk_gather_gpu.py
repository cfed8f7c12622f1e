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
