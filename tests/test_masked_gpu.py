"""GPU parity of the general prunable-span path (several marked spans,
anywhere in a sequence) against the oracle: the masked top-K bit-exact on
identical fp32 scores, the masked gate within the gate tolerance with exact
zeros outside the mask, and the prefix mask reproducing the
document/question calls bit for bit."""
import numpy as np
import pytest
import torch

import oracle
from learned_token_pruning_09_b300 import synth
from tests.helpers import dev_bf16, dev_f32, dev_i32

pytestmark = pytest.mark.gpu

GATE_TIGHT = 1e-4


@pytest.fixture(scope="module")
def tg():
    from learned_token_pruning_09_b300 import tokengate
    return tokengate


def dev_u8(a):
    return torch.as_tensor(np.asarray(a, np.uint8)).cuda()


def run_masked_topk(tg, s, cu, mask, k, capacity=None):
    cu = np.asarray(cu, np.int32)
    max_len = int(np.diff(cu).max()) if len(cu) > 1 else 0
    kept, cu_kept, n_prun = tg.tg_topk_select_masked(dev_f32(s), dev_i32(cu), dev_u8(mask), dev_i32(k), max_len,
                                                     kept_capacity=capacity)
    status = tg.tg_check_device_status()
    return kept.cpu().numpy(), cu_kept.cpu().numpy(), n_prun.cpu().numpy(), status


def check_masked_topk(tg, s, cu, mask, k):
    kept, cu_kept, n_prun, status = run_masked_topk(tg, s, cu, mask, k)
    assert status == tg.TG_OK
    ekept, ecu, eprun = oracle.topk_select_masked(s, cu, mask, k)
    np.testing.assert_array_equal(n_prun, eprun)
    np.testing.assert_array_equal(cu_kept, ecu)
    np.testing.assert_array_equal(kept[: ecu[-1]], ekept)


@pytest.mark.parametrize("name", ["tiny", "qwen3-1.7b-16k", "long-128k", "ragged-8"])
def test_masked_topk_workloads(tg, name):
    shape = synth.ALL_SHAPES[name]()
    mask = synth.prunable_spans(shape)
    s = synth.score_draws(shape)
    s[mask == 0] = 0.0              # the masked gate's scores outside the mask
    check_masked_topk(tg, s, shape.cu_seqlens, mask, shape.k)


@pytest.mark.parametrize("name", ["qwen3-1.7b-16k", "ragged-8"])
def test_prefix_mask_equals_document_call(tg, name):
    shape = synth.ALL_SHAPES[name]()
    cu = shape.cu_seqlens
    mask = np.zeros(shape.n_rows, np.uint8)
    for b in range(shape.batch):
        mask[cu[b]: cu[b] + shape.n_doc[b]] = 1
    s = synth.score_draws(shape)
    kept_m, cu_m, n_prun, status = run_masked_topk(tg, s, cu, mask, shape.k)
    assert status == tg.TG_OK
    n_kept = sum(tg.kept_lengths(np.diff(cu), shape.n_doc, shape.k))
    kept, cu_kept = tg.tg_topk_select(dev_f32(s), dev_i32(cu), dev_i32(shape.n_doc), dev_i32(shape.k),
                                      max(shape.n_doc), n_kept)
    np.testing.assert_array_equal(n_prun, shape.n_doc)
    np.testing.assert_array_equal(cu_m, cu_kept.cpu().numpy())
    np.testing.assert_array_equal(kept_m[:n_kept], kept.cpu().numpy())


@pytest.mark.parametrize("case", ["no_prunable", "all_k0", "k_above", "alternating", "single_rows", "ties",
                                  "empty_seq", "wide_slices"])
def test_masked_topk_edge_cases(tg, case):
    rng = np.random.default_rng(hash(case) % 1000)
    if case == "single_rows":
        lens = [1, 1, 2, 1]
    elif case == "empty_seq":
        lens = [0, 300, 0, 5]
    elif case == "wide_slices":
        lens = [70000]              # slices longer than one tile per CTA
    else:
        lens = [1000, 37, 513]
    cu = np.concatenate([[0], np.cumsum(lens)]).astype(np.int32)
    n = int(cu[-1])
    s = -np.abs(rng.normal(0, 3, n)).astype(np.float32)
    mask = (rng.random(n) < 0.7).astype(np.uint8)
    k = [int(max(1, l // 3)) for l in lens]
    if case == "no_prunable":
        mask[:] = 0
    elif case == "all_k0":
        mask[:] = 1
        k = [0] * len(lens)
    elif case == "k_above":
        k = [l + 5 for l in lens]
    elif case == "alternating":
        mask = (np.arange(n) % 2).astype(np.uint8)
    elif case == "ties":
        pool = np.array([-1.0, -2.0, -0.0, 0.0, -0.5], np.float32)
        s = pool[rng.integers(0, len(pool), n)]
    check_masked_topk(tg, s, cu, mask, k)


def test_masked_topk_flags_short_output(tg):
    """kept_capacity below the kept count: the sequences that would overrun
    write nothing and the device status says so."""
    lens = [400, 400]
    cu = np.array([0, 400, 800], np.int32)
    mask = np.zeros(800, np.uint8)
    mask[100:300] = 1
    mask[500:700] = 1
    s = -np.abs(np.random.default_rng(9).normal(0, 1, 800)).astype(np.float32)
    k = [50, 50]
    ekept, ecu, _ = oracle.topk_select_masked(s, cu, mask, k)
    tg.tg_check_device_status()
    _, cu_kept, _, status = run_masked_topk(tg, s, cu, mask, k, capacity=int(ecu[1]) + 10)
    assert status == tg.TG_ERR_DEVICE_INDEX
    assert cu_kept[1] == ecu[1]          # the first sequence fit and was written
    _, _, _, status = run_masked_topk(tg, s, cu, mask, k, capacity=int(ecu[-1]))
    assert status == tg.TG_OK


@pytest.mark.parametrize("name", ["tiny", "qwen3-1.7b-16k"])
def test_masked_gate(tg, name):
    shape = synth.ALL_SHAPES[name]()
    x, p = synth.residuals(shape), synth.gate_weights(shape)
    mask = synth.prunable_spans(shape)
    s = tg.tg_gate_score_masked(dev_bf16(x), dev_u8(mask), dev_bf16(p["w1"]), None, dev_bf16(p["w2"]), p["b2"])
    assert tg.tg_check_device_status() == tg.TG_OK
    s = s.cpu().numpy()
    ref = oracle.gate_score_masked(x, mask, p["w1"], p["b1"], p["w2"], p["b2"])
    assert np.all(s[mask == 0] == 0.0)
    err = np.abs(s.astype(np.float64) - ref.astype(np.float64))
    print(f"{name}: masked gate max |err| = {err.max():.3e}")
    assert err.max() <= GATE_TIGHT


def test_masked_chain_keeps_the_oracle_set(tg):
    """Gate -> top-K -> gather on a multi-span mask, through the masked calls:
    the kept set is the oracle's, up to rows whose score is within 1e-3 of
    the budget threshold (the gate tolerance's near ties)."""
    shape = synth.custom("chain", [6000, 3000], [40, 24], [900, 2000], d=256, h=64)
    x, p = synth.residuals(shape), synth.gate_weights(shape)
    mask = synth.prunable_spans(shape, spans_per_seq=3)
    cu = shape.cu_seqlens
    s_g = tg.tg_gate_score_masked(dev_bf16(x), dev_u8(mask), dev_bf16(p["w1"]), None, dev_bf16(p["w2"]), p["b2"])
    max_len = int(np.diff(cu).max())
    kept, cu_kept, _ = tg.tg_topk_select_masked(s_g, dev_i32(cu), dev_u8(mask), dev_i32(shape.k), max_len)
    n_kept = int(cu_kept[-1])
    xk, pos, sk = tg.tg_gather_kept(dev_bf16(x), s_g, dev_i32(cu), kept[:n_kept], cu_kept, n_kept)
    assert tg.tg_check_device_status() == tg.TG_OK
    s_ref = oracle.gate_score_masked(x, mask, p["w1"], p["b1"], p["w2"], p["b2"])
    ekept, ecu, _ = oracle.topk_select_masked(s_ref, cu, mask, shape.k)
    got = set(kept[:n_kept].cpu().numpy().tolist())
    want = set(ekept.tolist())
    for b in range(shape.batch):
        rows = ekept[ecu[b]: ecu[b + 1]]
        prun_rows = rows[mask[rows] == 1]
        if len(prun_rows) == 0:
            continue
        thr = s_ref[prun_rows].min()
        seq = set(range(int(cu[b]), int(cu[b + 1])))
        for r in (got ^ want) & seq:
            assert mask[r] == 1 and abs(float(s_ref[r]) - float(thr)) < 1e-3, r
    # the gathered rows and positions are those of the kept ids
    k_np = kept[:n_kept].cpu().numpy()
    np.testing.assert_array_equal(xk.cpu().view(torch.int16).numpy().view(np.uint16), np.asarray(x)[k_np])
    b_of = np.searchsorted(cu, k_np, side="right") - 1
    np.testing.assert_array_equal(pos.cpu().numpy(), k_np - cu[b_of])


@pytest.mark.parametrize("name", ["tiny", "qwen3-1.7b-16k", "ragged-8"])
def test_masked_chain_with_the_gate_histograms(tg, name):
    """With the top-K workspace, the masked gate counts each sequence's
    prunable scores and the masked top-K starts from those digits: the same
    scores and the same kept rows, bit for bit, as without the workspace;
    the workspace is zero again afterwards, and a second round gives the same."""
    shape = synth.ALL_SHAPES[name]()
    x, p = synth.residuals(shape), synth.gate_weights(shape)
    mask = synth.prunable_spans(shape)
    cu = np.asarray(shape.cu_seqlens, np.int32)
    max_len = int(np.diff(cu).max())
    X, W1, W2, M, CU, K = dev_bf16(x), dev_bf16(p["w1"]), dev_bf16(p["w2"]), dev_u8(mask), dev_i32(cu), dev_i32(shape.k)
    s0 = tg.tg_gate_score_masked(X, M, W1, None, W2, p["b2"])
    kept0, cu0, _ = tg.tg_topk_select_masked(s0, CU, M, K, max_len)
    ws = tg.tg_topk_workspace(len(cu) - 1)
    for _ in range(2):
        s1 = tg.tg_gate_score_masked(X, M, W1, None, W2, p["b2"], cu_seqlens=CU, topk_ws=ws)
        kept1, cu1, _ = tg.tg_topk_select_masked(s1, CU, M, K, max_len, workspace=ws)
        assert tg.tg_check_device_status() == tg.TG_OK
        assert torch.equal(s0, s1)
        assert torch.equal(cu0, cu1)
        n = int(cu0[-1])
        assert torch.equal(kept0[:n], kept1[:n])
        assert not torch.any(ws)
