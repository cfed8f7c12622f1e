"""GPU parity of the gate MLP, token-gated attention and the projections
against the fp64 oracle.

Tolerances: gate scores within 2e-2 absolute (and, as the fp32 epilogue
allows, within 1e-4 in practice); attention outputs |gpu - ref| <= 2e-2 +
1e-2 |ref| elementwise with bf16 inputs and fp32 accumulation; projections
the same allclose form (one bf16 rounding of the output)."""
import numpy as np
import pytest
import torch

import oracle
from learned_token_pruning_09_b300 import synth
from tests.helpers import allclose_report, dev_bf16, dev_f32, dev_i32, host_bits, host_f64

pytestmark = pytest.mark.gpu

GATE_ATOL = 2e-2
GATE_TIGHT = 1e-4
ATT_ATOL, ATT_RTOL = 2e-2, 1e-2


@pytest.fixture(scope="module")
def tg():
    from learned_token_pruning_09_b300 import tokengate
    return tokengate


def sample_rows(n, rng, k=1024):
    if n <= k:
        return np.arange(n)
    r = np.unique(np.concatenate([np.arange(64), np.arange(n - 64, n), rng.choice(n, k - 128, replace=False)]))
    return r


# ---------------------------------------------------------------------------
# gate
# ---------------------------------------------------------------------------


def run_gate(tg, shape, x, p, b1=None, b2=0.0, w2=None):
    s = tg.tg_gate_score(dev_bf16(x), dev_i32(shape.cu_seqlens), dev_i32(shape.n_doc), dev_bf16(p["w1"]),
                         None if b1 is None else dev_f32(b1), dev_bf16(p["w2"] if w2 is None else w2), b2)
    assert tg.tg_check_device_status() == tg.TG_OK
    return s.cpu().numpy()


@pytest.mark.parametrize("name", ["tiny", "qwen3-1.7b-16k"])
def test_gate_full(tg, name):
    shape = synth.ALL_SHAPES[name]()
    x = synth.residuals(shape)
    p = synth.gate_weights(shape)
    s = run_gate(tg, shape, x, p)
    ref = oracle.gate_score(x, shape.cu_seqlens, shape.n_doc, p["w1"], p["b1"], p["w2"], p["b2"])
    err = np.abs(s.astype(np.float64) - ref.astype(np.float64))
    print(f"{name}: gate max |err| = {err.max():.3e}")
    assert err.max() <= GATE_ATOL
    assert err.max() <= GATE_TIGHT
    nd = shape.n_doc[0]
    assert np.all(s[nd:] == 0.0)


@pytest.mark.parametrize("name", ["long-128k", "ragged-8"])
def test_gate_sampled_full_size(tg, name):
    shape = synth.ALL_SHAPES[name]()
    x = synth.residuals(shape)
    p = synth.gate_weights(shape)
    s = run_gate(tg, shape, x, p)
    rows = sample_rows(shape.n_rows, np.random.default_rng(0), 4096)
    ref = oracle.gate_score(x, shape.cu_seqlens, shape.n_doc, p["w1"], p["b1"], p["w2"], p["b2"], rows=rows)
    err = np.abs(s[rows].astype(np.float64) - ref[rows].astype(np.float64))
    print(f"{name}: gate max |err| over {len(rows)} rows = {err.max():.3e}")
    assert err.max() <= GATE_TIGHT


@pytest.mark.parametrize("h,d", [(16, 64), (48, 192), (256, 256), (128, 1024)])
def test_gate_shapes_biases_ragged_tail(tg, h, d):
    shape = synth.custom("g", [300, 0, 77], [13, 5, 0], [10, 10, 10], d=d, h=h, seed=h + d)
    x = synth.residuals(shape)
    p = synth.gate_weights(shape)
    rng = np.random.default_rng(h)
    b1 = rng.normal(0, 0.5, h).astype(np.float32)
    s = run_gate(tg, shape, x, p, b1=b1, b2=-0.7)
    ref = oracle.gate_score(x, shape.cu_seqlens, shape.n_doc, p["w1"], b1, p["w2"], -0.7)
    np.testing.assert_allclose(s, ref, atol=GATE_TIGHT, rtol=0)


def test_gate_zero_w2_closed_form(tg):
    shape = synth.custom("g", [129], [3], [5], d=128, h=32)
    x = synth.residuals(shape)
    p = synth.gate_weights(shape)
    s = run_gate(tg, shape, x, p, b2=float(np.log(3.0)), w2=np.zeros(32, np.uint16))
    np.testing.assert_allclose(s[:129], np.log(0.75), atol=1e-6)
    assert np.all(s[129:] == 0.0)


# ---------------------------------------------------------------------------
# attention
# ---------------------------------------------------------------------------


def attention_case(shape, pos_mode="topk"):
    """Seeded attention inputs of a workload: kept positions from the
    oracle's top-K on seeded score draws."""
    s_rows = synth.score_draws(shape)
    kept, cu_kept = oracle.topk_select(s_rows, shape.cu_seqlens, shape.n_doc, shape.k)
    _, pos, s_kept = oracle.gather_kept(np.zeros((shape.n_rows, 1), np.uint16), s_rows, shape.cu_seqlens,
                                        kept, cu_kept)
    ai = synth.attention_inputs(shape, n_kept=len(kept))
    return ai, pos, s_kept, cu_kept


def run_attention(tg, ai, pos, s_kept, cu_kept, want_k_cache=False, theta=1e6):
    q, k, v = dev_bf16(ai["q"]), dev_bf16(ai["k"]), dev_bf16(ai["v"])
    kc = torch.empty_like(k) if want_k_cache else None
    max_kept = int(np.diff(cu_kept).max())
    o, lse = tg.tg_gated_attention_fwd(q, k, v, dev_i32(pos), dev_f32(s_kept), dev_f32(ai["gain"]), ai["tau"],
                                       theta, dev_i32(cu_kept), max_kept, want_lse=True, k_cache=kc)
    assert tg.tg_check_device_status() == tg.TG_OK
    return host_f64(o), lse.cpu().numpy(), kc


def check_attention(o, lse, ref_o, ref_lse, rows, label):
    ok, err, exc = allclose_report(o[rows], ref_o[rows], ATT_ATOL, ATT_RTOL)
    lerr = np.nanmax(np.abs(lse[:, rows] - ref_lse[:, rows]))
    print(f"{label}: attention max |err| = {err:.3e} (excess {exc:.3e}), lse max |err| = {lerr:.3e}")
    assert ok
    assert lerr <= 2e-2


@pytest.mark.parametrize("name", ["tiny", "qwen3-1.7b-16k"])
def test_attention_full(tg, name):
    shape = synth.ALL_SHAPES[name]()
    ai, pos, s_kept, cu_kept = attention_case(shape)
    o, lse, _ = run_attention(tg, ai, pos, s_kept, cu_kept)
    rows = np.arange(len(pos)) if name == "tiny" else sample_rows(len(pos), np.random.default_rng(1), 768)
    ref_o, ref_lse = oracle.gated_attention(ai["q"], ai["k"], ai["v"], pos, s_kept, ai["gain"], ai["tau"],
                                            cu_kept, rows=rows)
    check_attention(o, lse, ref_o, ref_lse, rows, name)


@pytest.mark.parametrize("name", ["budget-32k-k1024", "budget-32k-k4096", "budget-32k-k8192", "ragged-8"])
def test_attention_sampled_full_size(tg, name):
    shape = synth.ALL_SHAPES[name]()
    ai, pos, s_kept, cu_kept = attention_case(shape)
    o, lse, _ = run_attention(tg, ai, pos, s_kept, cu_kept)
    rows = sample_rows(len(pos), np.random.default_rng(2), 384)
    # the last row of every sequence sees every kept key
    rows = np.unique(np.concatenate([rows, cu_kept[1:] - 1]))
    ref_o, ref_lse = oracle.gated_attention(ai["q"], ai["k"], ai["v"], pos, s_kept, ai["gain"], ai["tau"],
                                            cu_kept, rows=rows)
    check_attention(o, lse, ref_o, ref_lse, rows, name)


@pytest.mark.parametrize("hq,hkv,d", [(4, 2, 64), (4, 4, 64), (8, 2, 128), (6, 2, 128), (2, 1, 128), (3, 1, 64)])
@pytest.mark.parametrize("lens", [[1], [127, 128, 129], [300, 5, 257]])
def test_attention_heads_and_ragged_tiles(tg, hq, hkv, d, lens):
    rng = np.random.default_rng(hq * 100 + hkv * 10 + d + sum(lens))
    t = sum(lens)
    cu = np.concatenate([[0], np.cumsum(lens)]).astype(np.int32)
    pos = np.concatenate([np.sort(rng.choice(4 * n + 10, n, replace=False)) for n in lens]).astype(np.int32)
    s_kept = -np.abs(rng.normal(0, 2, t)).astype(np.float32)
    bf = lambda a: synth.f32_to_bf16_bits(a.astype(np.float32))
    ai = {"q": bf(rng.standard_normal((t, hq, d))), "k": bf(rng.standard_normal((t, hkv, d))),
          "v": bf(rng.standard_normal((t, hkv, d))), "gain": rng.uniform(0.5, 2, hq).astype(np.float32),
          "tau": 1.07}
    o, lse, kc = run_attention(tg, ai, pos, s_kept, cu, want_k_cache=True)
    rows = np.arange(t)
    ref_o, ref_lse = oracle.gated_attention(ai["q"], ai["k"], ai["v"], pos, s_kept, ai["gain"], ai["tau"], cu)
    check_attention(o, lse, ref_o, ref_lse, rows, f"hq{hq} hkv{hkv} d{d} lens{lens}")
    # the kept-only K cache holds k rotated at the original positions (bf16)
    kref = oracle.rope(oracle.bf16_decode(ai["k"]), pos)
    kgot = host_f64(kc)
    assert np.all(np.abs(kgot - kref) <= 2.0 ** -8 * np.abs(kref) + 1e-6)


def test_attention_large_scores_and_gain(tg):
    """Bias dominating the logits: large gains and very negative scores."""
    rng = np.random.default_rng(5)
    t, hq, hkv, d = 700, 4, 2, 128
    cu = np.array([0, t], np.int32)
    pos = np.arange(t, dtype=np.int32) * 3
    s_kept = np.where(rng.random(t) < 0.3, -40.0, -np.abs(rng.normal(0, 1, t))).astype(np.float32)
    bf = lambda a: synth.f32_to_bf16_bits(a.astype(np.float32))
    ai = {"q": bf(rng.standard_normal((t, hq, d))), "k": bf(rng.standard_normal((t, hkv, d))),
          "v": bf(rng.standard_normal((t, hkv, d))), "gain": np.array([0.0, 0.5, 2.0, 8.0], np.float32),
          "tau": 0.9}
    o, lse, _ = run_attention(tg, ai, pos, s_kept, cu)
    ref_o, ref_lse = oracle.gated_attention(ai["q"], ai["k"], ai["v"], pos, s_kept, ai["gain"], ai["tau"], cu)
    check_attention(o, lse, ref_o, ref_lse, np.arange(t), "large bias")


def test_attention_rejects_unsorted_positions(tg):
    rng = np.random.default_rng(6)
    t = 50
    pos = np.arange(t, dtype=np.int32)
    pos[10], pos[11] = pos[11], pos[10]
    bf = lambda a: synth.f32_to_bf16_bits(a.astype(np.float32))
    ai = {"q": bf(rng.standard_normal((t, 2, 64))), "k": bf(rng.standard_normal((t, 1, 64))),
          "v": bf(rng.standard_normal((t, 1, 64))), "gain": np.ones(2, np.float32), "tau": 1.0}
    q, k, v = dev_bf16(ai["q"]), dev_bf16(ai["k"]), dev_bf16(ai["v"])
    tg.tg_gated_attention_fwd(q, k, v, dev_i32(pos), dev_f32(np.zeros(t)), dev_f32(ai["gain"]), 1.0, 1e6,
                              dev_i32([0, t]), t)
    assert tg.tg_check_device_status() == tg.TG_ERR_DEVICE_INDEX


def _random_attention(rng, lens, hq, hkv, d):
    t = sum(lens)
    cu = np.concatenate([[0], np.cumsum(lens)]).astype(np.int32)
    pos = np.concatenate([np.sort(rng.choice(4 * n + 10, n, replace=False)) for n in lens]).astype(np.int32)
    s_kept = -np.abs(rng.normal(0, 2, t)).astype(np.float32)
    bf = lambda a: synth.f32_to_bf16_bits(a.astype(np.float32))
    ai = {"q": bf(rng.standard_normal((t, hq, d))), "k": bf(rng.standard_normal((t, hkv, d))),
          "v": bf(rng.standard_normal((t, hkv, d))), "gain": rng.uniform(0.5, 2, hq).astype(np.float32),
          "tau": 0.93}
    return ai, pos, s_kept, cu


@pytest.mark.parametrize("hq,hkv,d,lens", [(8, 2, 128, [127, 128, 129]), (3, 1, 64, [300, 5, 257]),
                                           (16, 8, 128, [1000])])
def test_rope_then_rotated_equals_fused_call(tg, hq, hkv, d, lens):
    """tg_rope_qk followed by tg_gated_attention_rotated is the fused call,
    bit for bit, and its k' is the fused call's K cache."""
    ai, pos, s_kept, cu = _random_attention(np.random.default_rng(hq + d + len(lens)), lens, hq, hkv, d)
    q, k, v = dev_bf16(ai["q"]), dev_bf16(ai["k"]), dev_bf16(ai["v"])
    pos_d, s_d, g_d, cu_d = dev_i32(pos), dev_f32(s_kept), dev_f32(ai["gain"]), dev_i32(cu)
    mk = int(max(lens))
    kc = torch.empty_like(k)
    o1, l1 = tg.tg_gated_attention_fwd(q, k, v, pos_d, s_d, g_d, ai["tau"], 1e6, cu_d, mk, want_lse=True, k_cache=kc)
    q2, k2 = tg.tg_rope_qk(q, k, pos_d, 1e6, cu_d)
    o2, l2 = tg.tg_gated_attention_rotated(q2, k2, v, pos_d, s_d, g_d, ai["tau"], cu_d, mk, want_lse=True)
    assert tg.tg_check_device_status() == tg.TG_OK
    assert np.array_equal(host_bits(o1), host_bits(o2))
    assert torch.equal(l1.cpu(), l2.cpu())
    assert np.array_equal(host_bits(kc), host_bits(k2))
    # q' and k' are the oracle's rotation at the original positions, rounded once to bf16
    for got, src in ((q2, ai["q"]), (k2, ai["k"])):
        ref = oracle.rope(oracle.bf16_decode(src), pos)
        assert np.all(np.abs(host_f64(got) - ref) <= 2.0 ** -8 * np.abs(ref) + 1e-6)


@pytest.mark.parametrize("case", ["swap_inside_tile", "swap_across_tiles", "negative"])
def test_rotated_attention_flags_bad_positions(tg, case):
    """Without the RoPE prologue's check, the attention kernel itself flags
    positions that do not strictly increase (its causal tile skipping relies
    on them)."""
    rng = np.random.default_rng(7)
    t, hq, hkv, d = 300, 2, 1, 64
    pos = np.arange(t, dtype=np.int32) * 2
    if case == "swap_inside_tile":
        pos[10], pos[11] = pos[11], pos[10]
    elif case == "swap_across_tiles":
        pos[127], pos[128] = pos[128], pos[127]
    else:
        pos[0] = -5
    bf = lambda a: synth.f32_to_bf16_bits(a.astype(np.float32))
    q, k, v = (dev_bf16(bf(rng.standard_normal(s))) for s in ((t, hq, d), (t, hkv, d), (t, hkv, d)))
    tg.tg_check_device_status()
    tg.tg_gated_attention_rotated(q, k, v, dev_i32(pos), dev_f32(np.zeros(t)), dev_f32(np.ones(hq)), 1.0,
                                  dev_i32([0, t]), t)
    assert tg.tg_check_device_status() == tg.TG_ERR_DEVICE_INDEX
    # well-formed positions leave the status clean
    good = np.arange(t, dtype=np.int32) * 2
    tg.tg_gated_attention_rotated(q, k, v, dev_i32(good), dev_f32(np.zeros(t)), dev_f32(np.ones(hq)), 1.0,
                                  dev_i32([0, t]), t)
    assert tg.tg_check_device_status() == tg.TG_OK


# ---------------------------------------------------------------------------
# projections and the stacked layer
# ---------------------------------------------------------------------------


@pytest.mark.parametrize("m,n,kd", [(1, 16, 64), (300, 48, 128), (1000, 4096, 2048), (257, 2048, 2048),
                                    (129, 272, 64)])
def test_linear(tg, m, n, kd):
    rng = np.random.default_rng(m + n + kd)
    bf = lambda a: synth.f32_to_bf16_bits(a.astype(np.float32))
    a = bf(rng.standard_normal((m, kd)))
    w = bf(rng.standard_normal((n, kd)) / np.sqrt(kd))
    r = bf(rng.standard_normal((m, n)))
    out = host_f64(tg.tg_linear_bf16(dev_bf16(a), dev_bf16(w)))
    ref = oracle.bf16_decode(a) @ oracle.bf16_decode(w).T
    ok, err, _ = allclose_report(out, ref, 1e-2, 1e-2)
    assert ok, err
    out2 = host_f64(tg.tg_linear_bf16(dev_bf16(a), dev_bf16(w), residual=dev_bf16(r)))
    ok, err, _ = allclose_report(out2, ref + oracle.bf16_decode(r), 2e-2, 1e-2)
    assert ok, err
    assert tg.tg_check_device_status() == tg.TG_OK
