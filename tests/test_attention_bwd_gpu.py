"""GPU parity of the attention backward with respect to the kept scores, the
gains and the temperature (tg_gated_attention_bwd) against the fp64 oracle.

The GPU path is the product's: tg_rope_qk (q', k' rounded to bf16), the
forward tg_gated_attention_rotated (o in bf16, lse in fp32), then the
backward.  The oracle differentiates the exact fp64 forward of the raw
inputs, so the bounds cover the forward's bf16 rounding points.  Each output
is a sum of many terms that largely cancel (d_tau most of all), so a bound
relative to the result says little; the bounds are relative to the magnitude
of the summed terms, which the oracle returns with ``scales=True``:
  |d_s_j error|   <= 2^-7  sum_h |g_h| sum_i |dl_ij|          + 1e-4
  |d_gain_h error| <= 2^-11 sum_ij |s_j dl_ij|                + 1e-4
  |d_tau error|   <= 2^-12 sum |dl_ij q'.k'| / (sqrt(D) tau^2) + 1e-3
A numpy model of the GPU's rounding points (q', k' and o in bf16, the rest
exact) on 19 of the cases below gives worst ratios 3.2e-3, 1.7e-4 and 8.8e-5
to those magnitudes; the factors are about 2.5 times that.  The floors cover
exact zeros (a one-token sequence: P = 1 and dP - D vanishes only up to
fp32 rounding)."""
import numpy as np
import pytest
import torch

import oracle
from learned_token_pruning_09_b300 import synth
from tests.helpers import dev_bf16, dev_f32, dev_i32

pytestmark = pytest.mark.gpu

DS_REL, DS_FLOOR = 2.0 ** -7, 1e-4
DG_REL, DG_FLOOR = 2.0 ** -11, 1e-4
DTAU_REL, DTAU_FLOOR = 2.0 ** -12, 1e-3


@pytest.fixture(scope="module")
def tg():
    from learned_token_pruning_09_b300 import tokengate
    return tokengate


def bf(a):
    return synth.f32_to_bf16_bits(np.asarray(a, np.float32))


def run_bwd(tg, ai, do_bits, pos, s_kept, cu, max_kept=None, theta=1e6):
    """The product path: RoPE, forward, backward.  Returns host fp64 arrays."""
    q, k, v = dev_bf16(ai["q"]), dev_bf16(ai["k"]), dev_bf16(ai["v"])
    pos_d, s_d, g_d, cu_d = dev_i32(pos), dev_f32(s_kept), dev_f32(ai["gain"]), dev_i32(cu)
    mk = int(np.diff(cu).max()) if max_kept is None else max_kept
    q_rot, k_rot = tg.tg_rope_qk(q, k, pos_d, theta, cu_d)
    o, lse = tg.tg_gated_attention_rotated(q_rot, k_rot, v, pos_d, s_d, g_d, ai["tau"], cu_d, mk, want_lse=True)
    ds, dg, dtau = tg.tg_gated_attention_bwd(q_rot, k_rot, v, o, lse, dev_bf16(do_bits), pos_d, s_d, g_d, ai["tau"],
                                             cu_d, mk)
    status = tg.tg_check_device_status()
    return ds.double().cpu().numpy(), dg.double().cpu().numpy(), float(dtau.item()), status


def check(got, ref, label):
    ds, dg, dtau = got
    rds, rdg, rdtau, ds_mag, dg_mag, dtau_mag = ref
    err = np.abs(ds - rds)
    lim = DS_REL * ds_mag + DS_FLOOR
    gerr = np.abs(dg - rdg)
    glim = DG_REL * dg_mag + DG_FLOOR
    terr = abs(dtau - rdtau)
    print(f"{label}: d_s max err {err.max(initial=0):.3e} (worst err/bound {(err / lim).max(initial=0):.2f}); "
          f"d_gain max err {gerr.max():.3e} (err/bound {(gerr / glim).max():.2f}); d_tau {dtau:.6e} vs "
          f"{rdtau:.6e} (err/bound {terr / (DTAU_REL * dtau_mag + DTAU_FLOOR):.2f})")
    assert np.all(np.isfinite(ds)) and np.all(np.isfinite(dg)) and np.isfinite(dtau)
    assert np.all(err <= lim)
    assert np.all(gerr <= glim)
    assert terr <= DTAU_REL * dtau_mag + DTAU_FLOOR


def reference(ai, do_bits, pos, s_kept, cu):
    return oracle.gated_attention_bwd(ai["q"], ai["k"], ai["v"], pos, s_kept, ai["gain"], ai["tau"], cu, do_bits,
                                      scales=True)


def workload_case(shape, seed=3):
    """A workload's attention inputs (kept positions from the oracle's top-K
    on seeded scores) and a seeded upstream gradient dO ~ N(0, 1) in bf16."""
    s_rows = synth.score_draws(shape)
    kept, cu_kept = oracle.topk_select(s_rows, shape.cu_seqlens, shape.n_doc, shape.k)
    _, pos, s_kept = oracle.gather_kept(np.zeros((shape.n_rows, 1), np.uint16), s_rows, shape.cu_seqlens,
                                        kept, cu_kept)
    ai = synth.attention_inputs(shape, n_kept=len(kept))
    do_bits = bf(np.random.default_rng(seed).standard_normal(np.asarray(ai["q"]).shape))
    return ai, do_bits, pos, s_kept, cu_kept


@pytest.mark.parametrize("name", ["tiny", "qwen3-1.7b-16k", "long-128k"])
def test_bwd_workloads(tg, name):
    shape = synth.ALL_SHAPES[name]()
    ai, do_bits, pos, s_kept, cu = workload_case(shape)
    got = run_bwd(tg, ai, do_bits, pos, s_kept, cu)
    assert got[3] == tg.TG_OK
    ref = reference(ai, do_bits, pos, s_kept, cu)
    check(got[:3], ref, name)


def random_case(rng, lens, hq, hkv, d, tau=0.93):
    t = sum(lens)
    cu = np.concatenate([[0], np.cumsum(lens)]).astype(np.int32)
    pos = np.concatenate([np.sort(rng.choice(4 * n + 10, n, replace=False)) for n in lens]).astype(np.int32)
    s_kept = -np.abs(rng.normal(0, 2, t)).astype(np.float32)
    ai = {"q": bf(rng.standard_normal((t, hq, d))), "k": bf(rng.standard_normal((t, hkv, d))),
          "v": bf(rng.standard_normal((t, hkv, d))), "gain": rng.uniform(0.5, 2, hq).astype(np.float32),
          "tau": tau}
    do_bits = bf(rng.standard_normal((t, hq, d)))
    return ai, do_bits, pos, s_kept, cu


@pytest.mark.parametrize("hq,hkv,d", [(4, 2, 64), (4, 4, 64), (8, 2, 128), (6, 2, 128), (3, 1, 64), (16, 2, 128)])
@pytest.mark.parametrize("lens", [[1], [127, 128, 129], [300, 0, 5, 257], [700]])
def test_bwd_heads_and_ragged_tiles(tg, hq, hkv, d, lens):
    """GQA group sizes 1, 2, 3, 4 and 8, both head dims, sequences shorter
    than a tile, on and across tile and pair boundaries, and empty."""
    rng = np.random.default_rng(hq * 100 + hkv * 10 + d + sum(lens))
    ai, do_bits, pos, s_kept, cu = random_case(rng, lens, hq, hkv, d)
    got = run_bwd(tg, ai, do_bits, pos, s_kept, cu)
    assert got[3] == tg.TG_OK
    ref = reference(ai, do_bits, pos, s_kept, cu)
    check(got[:3], ref, f"hq{hq} hkv{hkv} d{d} lens{lens}")


def test_bwd_ragged_batch(tg):
    """Several sequences of mixed length in one packed call, with a
    max_kept bound above the longest."""
    rng = np.random.default_rng(44)
    lens = [1500, 37, 900, 2049, 256]
    ai, do_bits, pos, s_kept, cu = random_case(rng, lens, 16, 8, 128, tau=1.2)
    got = run_bwd(tg, ai, do_bits, pos, s_kept, cu, max_kept=2100)
    assert got[3] == tg.TG_OK
    ref = reference(ai, do_bits, pos, s_kept, cu)
    check(got[:3], ref, "ragged batch")


def test_bwd_large_bias_and_zero_gain(tg):
    """The bias dominating the logits (gains up to 8, scores down to -40) and
    a head with zero gain."""
    rng = np.random.default_rng(5)
    t, hq, hkv, d = 700, 4, 2, 128
    ai, do_bits, pos, s_kept, cu = random_case(rng, [t], hq, hkv, d, tau=0.9)
    s_kept = np.where(rng.random(t) < 0.3, -40.0, s_kept).astype(np.float32)
    ai["gain"] = np.array([0.0, 0.5, 2.0, 8.0], np.float32)
    got = run_bwd(tg, ai, do_bits, pos, s_kept, cu)
    assert got[3] == tg.TG_OK
    check(got[:3], reference(ai, do_bits, pos, s_kept, cu), "large bias")


def test_bwd_infinite_scores(tg):
    """Keys with score -inf (positive gains): P = 0 for them, so their d_s is
    exactly 0 and they add nothing to d_gain."""
    rng = np.random.default_rng(6)
    t, hq, hkv, d = 700, 4, 2, 64
    ai, do_bits, pos, s_kept, cu = random_case(rng, [t], hq, hkv, d, tau=1.1)
    s_kept[[3, 200, 650]] = -np.inf
    got = run_bwd(tg, ai, do_bits, pos, s_kept, cu)
    assert got[3] == tg.TG_OK
    check(got[:3], reference(ai, do_bits, pos, s_kept, cu), "infinite scores")
    assert np.all(got[0][[3, 200, 650]] == 0.0)


def test_bwd_is_deterministic_and_sums_to_zero(tg):
    """Fixed reduction order: two calls agree bit for bit; the d_s of every
    sequence sums to about zero (softmax is shift-invariant)."""
    rng = np.random.default_rng(8)
    ai, do_bits, pos, s_kept, cu = random_case(rng, [3000, 1200], 16, 8, 128)
    a = run_bwd(tg, ai, do_bits, pos, s_kept, cu)
    b = run_bwd(tg, ai, do_bits, pos, s_kept, cu)
    assert a[3] == tg.TG_OK and b[3] == tg.TG_OK
    np.testing.assert_array_equal(a[0], b[0])
    np.testing.assert_array_equal(a[1], b[1])
    assert a[2] == b[2]
    for i in range(len(cu) - 1):
        seg = a[0][cu[i]:cu[i + 1]]
        assert abs(seg.sum()) <= 1e-3 * np.abs(seg).sum()


def test_bwd_empty_and_short_max_kept(tg):
    """n_kept = 0 gives zero gradients; a max_kept below a sequence's length
    is flagged on the device."""
    z = torch.zeros((0, 2, 64), dtype=torch.bfloat16, device="cuda")
    zk = torch.zeros((0, 1, 64), dtype=torch.bfloat16, device="cuda")
    lse = torch.zeros((2, 0), dtype=torch.float32, device="cuda")
    e32 = torch.zeros(0, dtype=torch.float32, device="cuda")
    dg = torch.full((2,), 7.0, device="cuda")
    dt = torch.full((1,), 7.0, device="cuda")
    tg.tg_gated_attention_bwd(z, zk, zk, z, lse, z, torch.zeros(0, dtype=torch.int32, device="cuda"), e32,
                              dev_f32([1.0, 1.0]), 1.0, dev_i32([0, 0]), 0, d_gain=dg, d_tau=dt)
    assert tg.tg_check_device_status() == tg.TG_OK
    assert torch.all(dg == 0) and torch.all(dt == 0)
    rng = np.random.default_rng(9)
    ai, do_bits, pos, s_kept, cu = random_case(rng, [600], 2, 1, 64)
    tg.tg_check_device_status()
    *_, status = run_bwd(tg, ai, do_bits, pos, s_kept, cu, max_kept=300)
    assert status == tg.TG_ERR_DEVICE_INDEX
