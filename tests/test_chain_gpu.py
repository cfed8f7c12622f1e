"""The document path end to end on the GPU, at full size: gate scores, top-K,
gather and token-gated attention, each fed by the previous call's device
output (TokenGate's pruned prefill, MarkTechPost article, "How does
TokenGate's learned token pruning work?").

Against the oracle:
* gate scores within 1e-4 (the spec allows 2e-2);
* the kept set equals the oracle's (its top-K on its own scores) except for
  rows whose oracle score lies within 1e-3 of the oracle's K-th score;
* the gather is exact for the GPU's own kept ids;
* attention on the GPU's kept set equals the oracle's attention on that same
  set (positions and oracle scores of those rows) within 2e-2 + 1e-2 |ref|.
"""
import numpy as np
import pytest
import torch

import oracle
from learned_token_pruning_09_b300 import synth
from tests.helpers import allclose_report, dev_bf16, dev_f32, dev_i32, host_bits, host_f64

pytestmark = pytest.mark.gpu

GATE_TIGHT = 1e-4
TIE_BAND = 1e-3
ATT_ATOL, ATT_RTOL = 2e-2, 1e-2


@pytest.fixture(scope="module")
def tg():
    from learned_token_pruning_09_b300 import tokengate
    return tokengate


def kept_set_differences_are_near_ties(kept_gpu, kept_ref, s_ref, shape):
    """Every row in the symmetric difference of the two kept sets is a
    document row whose oracle score is within TIE_BAND of its sequence's
    K-th oracle score.  Returns the number of differing rows."""
    diff = np.setxor1d(kept_gpu, kept_ref)
    cu = shape.cu_seqlens
    for b in range(shape.batch):
        lo, nd, ke = int(cu[b]), shape.n_doc[b], shape.k_eff[b]
        mine = diff[(diff >= lo) & (diff < int(cu[b + 1]))]
        if len(mine) == 0:
            continue
        assert np.all(mine < lo + nd), "a question row differs"
        s_k = np.sort(s_ref[lo: lo + nd])[::-1][ke - 1]
        assert np.all(np.abs(s_ref[mine] - s_k) < TIE_BAND), (b, mine[:8], s_k)
    return len(diff)


@pytest.mark.parametrize("name", ["qwen3-1.7b-16k", "long-128k", "ragged-8"])
def test_document_chain_end_to_end(tg, name):
    shape = synth.ALL_SHAPES[name]()
    x, p = synth.residuals(shape), synth.gate_weights(shape)
    cu_d, nd_d = dev_i32(shape.cu_seqlens), dev_i32(shape.n_doc)
    X = dev_bf16(x)
    ws = tg.tg_topk_workspace(shape.batch)
    s = tg.tg_gate_score(X, cu_d, nd_d, dev_bf16(p["w1"]), None, dev_bf16(p["w2"]), p["b2"], topk_ws=ws)
    kept, cu_kept = tg.tg_topk_select(s, cu_d, nd_d, dev_i32(shape.k), max(shape.n_doc), shape.n_kept, workspace=ws)
    xk, pos, sk = tg.tg_gather_kept(X, s, cu_d, kept, cu_kept, shape.n_kept)
    ai = synth.attention_inputs(shape)
    o, lse = tg.tg_gated_attention_fwd(dev_bf16(ai["q"]), dev_bf16(ai["k"]), dev_bf16(ai["v"]), pos, sk,
                                       dev_f32(ai["gain"]), ai["tau"], 1e6, cu_kept, max(shape.kept_lens),
                                       want_lse=True)
    assert tg.tg_check_device_status() == tg.TG_OK
    # the top-K cleared the gate's score histograms for the next call
    assert int(ws.count_nonzero()) == 0

    # gate
    s_gpu = s.cpu().numpy()
    s_ref = oracle.gate_score(x, shape.cu_seqlens, shape.n_doc, p["w1"], p["b1"], p["w2"], p["b2"])
    gerr = np.abs(s_gpu.astype(np.float64) - s_ref.astype(np.float64)).max()
    assert gerr <= GATE_TIGHT
    # top-K: the oracle's set up to near ties; the layout is the host's
    kept_gpu = kept.cpu().numpy()
    np.testing.assert_array_equal(cu_kept.cpu().numpy(), shape.cu_kept)
    kept_ref, cu_ref = oracle.topk_select(s_ref, shape.cu_seqlens, shape.n_doc, shape.k)
    n_diff = kept_set_differences_are_near_ties(kept_gpu, kept_ref, s_ref, shape)
    # the GPU's own kept ids are a valid top-K output of the GPU's own scores
    k2, c2 = oracle.topk_select(s_gpu, shape.cu_seqlens, shape.n_doc, shape.k)
    np.testing.assert_array_equal(kept_gpu, k2)
    # gather of those ids, bit for bit
    xk_ref, pos_ref, sk_ref = oracle.gather_kept(x, s_gpu, shape.cu_seqlens, kept_gpu, shape.cu_kept)
    assert np.array_equal(host_bits(xk), xk_ref)
    np.testing.assert_array_equal(pos.cpu().numpy(), pos_ref)
    np.testing.assert_array_equal(sk.cpu().numpy(), sk_ref)
    # attention on the GPU's kept set, the oracle given the same rows and its own scores of them
    rng = np.random.default_rng(11)
    t = shape.n_kept
    rows = np.unique(np.concatenate([np.arange(64), np.arange(t - 64, t), rng.choice(t, 256, replace=False)]))
    ref_o, ref_lse = oracle.gated_attention(ai["q"], ai["k"], ai["v"], pos_ref, s_ref[kept_gpu], ai["gain"],
                                            ai["tau"], shape.cu_kept, rows=rows)
    o_h, lse_h = host_f64(o), lse.cpu().numpy()
    ok, err, exc = allclose_report(o_h[rows], ref_o[rows], ATT_ATOL, ATT_RTOL)
    lerr = np.abs(lse_h[:, rows] - ref_lse[:, rows]).max()
    print(f"{name}: gate |err| {gerr:.2e}; kept-set differences {n_diff}; attention |err| {err:.3e}, "
          f"lse |err| {lerr:.3e}")
    assert ok
    assert lerr <= 2e-2
