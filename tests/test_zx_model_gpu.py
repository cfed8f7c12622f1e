"""GPU parity of the layer calls around the pruned path and of the
synthetic-model runner (pruned prefill + first decode step) against the
fp64 oracle.  Bounds: RMSNorm / SwiGLU within two bf16 roundings; decode
attention as the forward attention (2e-2 + 1e-2|ref|); the runner's logits
within 3% of the largest logit, kept set equal where the oracle's K-th score
gap exceeds 1e-3 (a model of the runner's bf16 rounding points gives 1%)."""
import math

import numpy as np
import pytest
import torch

import oracle
from learned_token_pruning_09_b300 import synth
from tests.helpers import dev_bf16, dev_f32, dev_i32, host_f64

pytestmark = pytest.mark.gpu
bf = lambda a: synth.f32_to_bf16_bits(np.asarray(a, np.float32))


@pytest.fixture(scope="module")
def tg():
    from learned_token_pruning_09_b300 import tokengate
    return tokengate


@pytest.mark.parametrize("rows,d", [(1, 8), (37, 128), (1000, 2048), (4096, 64)])
def test_rms_norm(tg, rows, d):
    rng = np.random.default_rng(rows + d)
    x, w = bf(rng.standard_normal((rows, d)) * 3), bf(1 + 0.1 * rng.standard_normal(d))
    y = host_f64(tg.tg_rms_norm(dev_bf16(x), dev_bf16(w)))
    ref = oracle.model.rms_norm(oracle.bf16_decode(x), oracle.bf16_decode(w))
    assert np.all(np.abs(y - ref) <= 2.0 ** -8 * np.abs(ref) + 1e-6)


@pytest.mark.parametrize("rows,f", [(1, 8), (33, 256), (512, 6144)])
def test_swiglu(tg, rows, f):
    rng = np.random.default_rng(rows + f)
    gu = bf(rng.standard_normal((rows, 2 * f)) * 2)
    y = host_f64(tg.tg_swiglu(dev_bf16(gu)))
    g = oracle.bf16_decode(gu)
    ref = oracle.model.silu(g[:, :f]) * g[:, f:]
    assert np.all(np.abs(y - ref) <= 2.0 ** -8 * np.abs(ref) + 1e-6)


@pytest.mark.parametrize("lens,hq,hkv,d,bias", [([700, 5, 0, 257], 16, 8, 128, True), ([3000], 4, 2, 64, False),
                                                ([1, 300], 8, 1, 128, True)])
def test_decode_attention(tg, lens, hq, hkv, d, bias):
    """The new query of each sequence over its cache and its own key, against
    the oracle's attention of the cache plus the new row (the new row last,
    at position N_b, its score 0)."""
    rng = np.random.default_rng(sum(lens) + hq)
    b = len(lens)
    cu = np.concatenate([[0], np.cumsum(lens)]).astype(np.int32)
    r = int(cu[-1])
    kc, vc = bf(rng.standard_normal((r, hkv, d))), bf(rng.standard_normal((r, hkv, d)))
    qn, kn, vn = bf(rng.standard_normal((b, hq, d))), bf(rng.standard_normal((b, hkv, d))), bf(rng.standard_normal((b, hkv, d)))
    s = -np.abs(rng.normal(0, 2, r)).astype(np.float32)
    gain = rng.uniform(0.5, 2, hq).astype(np.float32)
    tau = 1.1 if bias else 1.0
    pos_c = np.concatenate([np.arange(n) for n in lens]).astype(np.int32)
    pos_n = np.asarray(lens, np.int32)
    # rotate on the GPU as the runner does: the cache at its positions, the new rows at N_b
    # a throwaway q with hkv heads (the RoPE call wants hq a multiple of hkv)
    _, kc_rot = tg.tg_rope_qk(dev_bf16(np.zeros((r, hkv, d), np.uint16)), dev_bf16(kc), dev_i32(pos_c), 1e6,
                              dev_i32(cu))
    q_rot, kn_rot = tg.tg_rope_qk(dev_bf16(qn), dev_bf16(kn), dev_i32(pos_n), 1e6, dev_i32(np.arange(b + 1)))
    o = tg.tg_decode_attention(q_rot, kn_rot, dev_bf16(vn), kc_rot, dev_bf16(vc), dev_i32(cu), max(lens),
                               s_cache=dev_f32(s) if bias else None, gain=dev_f32(gain) if bias else None, tau=tau)
    assert tg.tg_check_device_status() == tg.TG_OK
    o = host_f64(o)
    for i in range(b):
        lo, hi = cu[i], cu[i + 1]
        n = hi - lo
        q_all = np.concatenate([np.zeros((n, hq, d), np.uint16), qn[i:i + 1]])
        k_all = np.concatenate([kc[lo:hi], kn[i:i + 1]])
        v_all = np.concatenate([vc[lo:hi], vn[i:i + 1]])
        p_all = np.concatenate([pos_c[lo:hi], [lens[i]]])
        s_all = np.concatenate([s[lo:hi], [0.0]]) if bias else np.zeros(n + 1)
        g_all = gain if bias else np.zeros(hq)
        ref, _ = oracle.gated_attention(q_all, k_all, v_all, p_all, s_all, g_all, tau, [0, n + 1], rows=np.array([n]))
        assert np.all(np.abs(o[i] - ref[n]) <= 2e-2 + 1e-2 * np.abs(ref[n]))


def test_runner_prefill_and_decode(tg):
    from learned_token_pruning_09_b300.model import SyntheticModel
    m = synth.model_params("model-tiny")
    c = m["config"]
    dec = oracle.bf16_decode
    layers = [{k: (dec(v) if isinstance(v, np.ndarray) and v.dtype == np.uint16 else v) for k, v in lp.items()}
              for lp in m["layers"]]
    gate = {"w1": dec(m["gate"]["w1"]), "w2": dec(m["gate"]["w2"]), "b1": np.zeros(c["gate_h"]), "b2": 0.0}
    rng = np.random.default_rng(0)
    lens, n_doc, k = [60, 45], [52, 40], [12, 9]
    cu = np.concatenate([[0], np.cumsum(lens)])
    x = bf(rng.standard_normal((int(cu[-1]), c["d"])))
    x_new = bf(rng.standard_normal((2, c["d"])))
    model = SyntheticModel(m)
    st = model.prefill(dev_bf16(x), lens, n_doc, k)
    logits = host_f64(st["logits"])
    nxt = host_f64(model.decode(dev_bf16(x_new), st))
    assert tg.tg_check_device_status() == tg.TG_OK
    ref = oracle.model.pruned_prefill(dec(x), layers, gate, c["gate_layer"], cu, n_doc, k, dec(m["final_norm"]),
                                      dec(m["w_lm"]), c["hq"], c["hkv"], c["head_dim"])
    np.testing.assert_array_equal(np.sort(st["kept"].cpu().numpy()), np.sort(ref["kept"]))
    assert np.abs(logits - ref["logits"]).max() <= 0.03 * np.abs(ref["logits"]).max()
    ref_nxt, _ = oracle.model.decode_step(dec(x_new), ref, layers, c["gate_layer"], cu, dec(m["final_norm"]),
                                          dec(m["w_lm"]), c["hq"], c["hkv"], c["head_dim"])
    assert np.abs(nxt - ref_nxt).max() <= 0.03 * np.abs(ref_nxt).max()


def test_runner_full_prefill_and_decode(tg):
    """The full prefill (every layer on every row, no gate) and its decode
    step over full-length caches.  The oracle's pruned prefill with the gate
    at the last layer and the whole document kept is that dense stack: every
    layer runs on every row, none with a score bias."""
    from learned_token_pruning_09_b300.model import SyntheticModel
    m = synth.model_params("model-tiny")
    c = m["config"]
    dec = oracle.bf16_decode
    layers = [{k: (dec(v) if isinstance(v, np.ndarray) and v.dtype == np.uint16 else v) for k, v in lp.items()}
              for lp in m["layers"]]
    gate = {"w1": dec(m["gate"]["w1"]), "w2": dec(m["gate"]["w2"]), "b1": np.zeros(c["gate_h"]), "b2": 0.0}
    rng = np.random.default_rng(1)
    lens = [70, 33, 1]
    cu = np.concatenate([[0], np.cumsum(lens)])
    x = bf(rng.standard_normal((int(cu[-1]), c["d"])))
    x_new = bf(rng.standard_normal((len(lens), c["d"])))
    model = SyntheticModel(m)
    st = model.prefill_full(dev_bf16(x), lens)
    logits = host_f64(st["logits"])
    nxt = host_f64(model.decode(dev_bf16(x_new), st))
    assert tg.tg_check_device_status() == tg.TG_OK
    last = c["n_layers"] - 1
    ref = oracle.model.pruned_prefill(dec(x), layers, gate, last, cu, lens, lens, dec(m["final_norm"]),
                                      dec(m["w_lm"]), c["hq"], c["hkv"], c["head_dim"])
    assert np.abs(logits - ref["logits"]).max() <= 0.03 * np.abs(ref["logits"]).max()
    ref_nxt, _ = oracle.model.decode_step(dec(x_new), ref, layers, last, cu, dec(m["final_norm"]), dec(m["w_lm"]),
                                          c["hq"], c["hkv"], c["head_dim"])
    assert np.abs(nxt - ref_nxt).max() <= 0.03 * np.abs(ref_nxt).max()
