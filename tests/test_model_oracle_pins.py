"""Pins of the synthetic-model oracle (oracle.model): the pruned prefill of a
Qwen3-style stack and its first decode step, composed from the pinned gate,
top-K and token-gated attention.  CPU only."""
import math

import numpy as np
import pytest
import torch
from scipy.special import expit

import oracle
from learned_token_pruning_09_b300 import synth

M = oracle.model


def f64_model(name):
    m = synth.model_params(name)
    dec = oracle.bf16_decode
    layers = []
    for lp in m["layers"]:
        layers.append({key: (dec(val) if isinstance(val, np.ndarray) and val.dtype == np.uint16 else val)
                       for key, val in lp.items()})
    gate = {"w1": dec(m["gate"]["w1"]), "w2": dec(m["gate"]["w2"]), "b1": np.asarray(m["gate"]["b1"], np.float64),
            "b2": m["gate"]["b2"]}
    return m["config"], layers, gate, dec(m["final_norm"]), dec(m["w_lm"])


def test_rms_norm_closed_forms():
    x = np.array([3.0, 4.0])
    np.testing.assert_allclose(M.rms_norm(x, np.ones(2), eps=0.0), x / math.sqrt(12.5), rtol=1e-15)
    c = np.full(6, -2.5)
    w = np.arange(1.0, 7.0)
    np.testing.assert_allclose(M.rms_norm(c, w, eps=0.0), -w, rtol=1e-15)
    rng = np.random.default_rng(0)
    y = rng.standard_normal((5, 9))
    np.testing.assert_allclose(M.rms_norm(7.0 * y, np.ones(9), eps=0.0), M.rms_norm(y, np.ones(9), eps=0.0),
                               rtol=1e-14)
    out = M.rms_norm(y, np.ones(9), eps=0.0)
    np.testing.assert_allclose(np.mean(out * out, axis=-1), 1.0, rtol=1e-14)


def test_silu_closed_forms():
    z = np.linspace(-30, 30, 241)
    np.testing.assert_allclose(M.silu(z), z * expit(z), rtol=1e-14, atol=1e-300)
    np.testing.assert_allclose(M.silu(z) - M.silu(-z), z, rtol=1e-13, atol=1e-13)
    assert M.silu(np.array([0.0]))[0] == 0.0
    assert abs(M.silu(np.array([-800.0]))[0]) < 1e-300


def _torch_layer(x, p, hq, hkv, dh, attn_only=False, theta=1e6):
    """An independent float64 layer: own RMSNorm, RoPE in complex form, SDPA
    with repeated KV heads, torch's SiLU.  One sequence, positions 0..T-1."""
    T = lambda a: torch.from_numpy(np.asarray(a, np.float64))
    xt = T(x)
    n = xt.shape[0]
    rms = lambda a, w: a / torch.sqrt((a * a).mean(-1, keepdim=True) + 1e-6) * T(w)
    a = rms(xt, p["ln1"])
    q = rms((a @ T(p["w_q"]).T).view(n, hq, dh), p["q_norm"])
    k = rms((a @ T(p["w_k"]).T).view(n, hkv, dh), p["k_norm"])
    v = (a @ T(p["w_v"]).T).view(n, hkv, dh)
    half = dh // 2
    ang = torch.arange(n, dtype=torch.float64)[:, None] * theta ** (-2.0 * torch.arange(half, dtype=torch.float64) / dh)
    rot = torch.polar(torch.ones_like(ang), ang)[:, None, :]

    def rope(u):
        zc = torch.complex(u[..., :half], u[..., half:]) * rot
        return torch.cat([zc.real, zc.imag], dim=-1)
    qr, kr = rope(q).permute(1, 0, 2), rope(k).permute(1, 0, 2)
    g = hq // hkv
    o = torch.nn.functional.scaled_dot_product_attention(
        qr, kr.repeat_interleave(g, 0), v.permute(1, 0, 2).repeat_interleave(g, 0), is_causal=True,
        scale=1.0 / math.sqrt(dh))
    h = xt + o.permute(1, 0, 2).reshape(n, hq * dh) @ T(p["w_o"]).T
    if attn_only:
        return h.numpy()
    m = rms(h, p["ln2"])
    y = h + (torch.nn.functional.silu(m @ T(p["w_gate"]).T) * (m @ T(p["w_up"]).T)) @ T(p["w_down"]).T
    return y.numpy()


def test_dense_layer_matches_torch():
    cfg, layers, _, _, _ = f64_model("model-tiny")
    rng = np.random.default_rng(1)
    n = 37
    x = rng.standard_normal((n, cfg["d"]))
    pos = np.arange(n)
    got = M.dense_layer(x, layers[0], pos, [0, n], cfg["hq"], cfg["hkv"], cfg["head_dim"])
    ref = _torch_layer(x, layers[0], cfg["hq"], cfg["hkv"], cfg["head_dim"])
    np.testing.assert_allclose(got, ref, rtol=1e-10, atol=1e-10)


def _prefill(cfg, layers, gate, fn, w_lm, x, cu, n_doc, k):
    return M.pruned_prefill(x, layers, gate, cfg["gate_layer"], cu, n_doc, k, fn, w_lm, cfg["hq"], cfg["hkv"],
                            cfg["head_dim"])


def test_prefill_without_pruning_is_the_dense_model():
    """K >= n_doc and zero gains above the gate: the pruned prefill is the
    dense stack on every token (torch layers), logits at the last row."""
    cfg, layers, gate, fn, w_lm = f64_model("model-tiny")
    for lp in layers:
        lp["gain"] = np.zeros(cfg["hq"])
        lp["tau"] = 1.0
    rng = np.random.default_rng(2)
    n = 40
    x = rng.standard_normal((n, cfg["d"]))
    out = _prefill(cfg, layers, gate, fn, w_lm, x, [0, n], [30], [30])
    assert len(out["kept"]) == n
    y = x
    for lp in layers:
        y = _torch_layer(y, lp, cfg["hq"], cfg["hkv"], cfg["head_dim"])
    ref = M.rms_norm(y[-1:], fn) @ w_lm.T
    np.testing.assert_allclose(out["logits"], ref, rtol=1e-9, atol=1e-9)


def test_gate_reads_the_post_attention_residual_of_its_layer():
    """The prefill's scores are the gate MLP on h = x + attention of layer L,
    with x from the dense layers below it (torch layers)."""
    cfg, layers, gate, fn, w_lm = f64_model("model-tiny")
    rng = np.random.default_rng(3)
    n, nd = 50, 44
    x = rng.standard_normal((n, cfg["d"]))
    out = _prefill(cfg, layers, gate, fn, w_lm, x, [0, n], [nd], [10])
    y = x
    for li in range(cfg["gate_layer"]):
        y = _torch_layer(y, layers[li], cfg["hq"], cfg["hkv"], cfg["head_dim"])
    h = _torch_layer(y, layers[cfg["gate_layer"]], cfg["hq"], cfg["hkv"], cfg["head_dim"], attn_only=True)
    u = h @ gate["w1"].T
    z = (0.5 * u * (1.0 + np.vectorize(math.erf)(u / math.sqrt(2.0)))) @ gate["w2"]
    ref = -np.logaddexp(0.0, -z)
    np.testing.assert_allclose(out["s"][:nd], ref[:nd], rtol=1e-6, atol=1e-6)
    assert np.all(out["s"][nd:] == 0.0)
    assert len(out["kept"]) == 10 + (n - nd)


def _decode_inputs(name, seed, lens, n_doc, k):
    cfg, layers, gate, fn, w_lm = f64_model(name)
    rng = np.random.default_rng(seed)
    cu = np.concatenate([[0], np.cumsum(lens)])
    x = rng.standard_normal((int(cu[-1]), cfg["d"]))
    x_new = rng.standard_normal((len(lens), cfg["d"]))
    return cfg, layers, gate, fn, w_lm, cu, x, x_new


@pytest.mark.parametrize("lens,n_doc,k", [([60], [52], [12]), ([45, 30], [40, 22], [9, 30])])
def test_decode_step_equals_prefill_of_the_extended_prompt(lens, n_doc, k):
    """With pruning and token-gated attention active: one decode step over
    the prefill's caches gives the logits of a pruned prefill of the prompt
    with the new token appended as a question row (its score 0, always kept;
    the document's scores and kept set do not change, attention being
    causal)."""
    cfg, layers, gate, fn, w_lm, cu, x, x_new = _decode_inputs("model-tiny", 4, lens, n_doc, k)
    pre = _prefill(cfg, layers, gate, fn, w_lm, x, cu, n_doc, k)
    logits, _ = M.decode_step(x_new, pre, layers, cfg["gate_layer"], cu, fn, w_lm, cfg["hq"], cfg["hkv"],
                              cfg["head_dim"])
    rows, cu2 = [], [0]
    for b in range(len(lens)):
        rows.append(x[cu[b]:cu[b + 1]])
        rows.append(x_new[b:b + 1])
        cu2.append(cu2[-1] + lens[b] + 1)
    ext = _prefill(cfg, layers, gate, fn, w_lm, np.concatenate(rows), cu2, n_doc, k)
    np.testing.assert_allclose(logits, ext["logits"], rtol=1e-9, atol=1e-9)
    # the kept set of the extended prompt is the prefill's plus the new rows
    assert len(ext["kept"]) == len(pre["kept"]) + len(lens)


def test_decode_step_without_pruning_is_the_dense_model():
    cfg, layers, gate, fn, w_lm, cu, x, x_new = _decode_inputs("model-tiny", 5, [33], [20], [20])
    for lp in layers:
        lp["gain"] = np.zeros(cfg["hq"])
        lp["tau"] = 1.0
    pre = _prefill(cfg, layers, gate, fn, w_lm, x, cu, [20], [20])
    logits, _ = M.decode_step(x_new, pre, layers, cfg["gate_layer"], cu, fn, w_lm, cfg["hq"], cfg["hkv"],
                              cfg["head_dim"])
    y = np.concatenate([x, x_new])
    for lp in layers:
        y = _torch_layer(y, lp, cfg["hq"], cfg["hkv"], cfg["head_dim"])
    np.testing.assert_allclose(logits, M.rms_norm(y[-1:], fn) @ w_lm.T, rtol=1e-9, atol=1e-9)
