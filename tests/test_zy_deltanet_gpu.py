"""GPU parity of the pruned Gated DeltaNet scan (tg_gated_delta_scan)
against the fp64 oracle.

The kernel keeps the state in fp32 and rounds o once to bf16, so the bound
on o is the bf16 rounding (2^-9 relative) with a factor of two, plus an
absolute floor of 2e-4 for fp32 error and the approximate exp / rsqrt
(a float32 replay of the kernel's arithmetic on the CPU stays within 4e-8 of
the oracle); the fp32 final state is compared within 1e-4 of its largest
entry.  Continuation and pruning are checked GPU against GPU."""
import numpy as np
import pytest
import torch

import oracle
from learned_token_pruning_09_b300 import synth
from tests.helpers import dev_bf16, dev_f32, dev_i32, host_f64

pytestmark = pytest.mark.gpu

O_RTOL, O_ATOL = 2.0 ** -8, 2e-4
S_REL = 1e-4


@pytest.fixture(scope="module")
def tg():
    from learned_token_pruning_09_b300 import tokengate
    return tokengate


def run_scan(tg, d, initial_state=None, scale=None):
    o, s = tg.tg_gated_delta_scan(dev_bf16(d["q"]), dev_bf16(d["k"]), dev_bf16(d["v"]), dev_f32(d["g"]),
                                  dev_f32(d["beta"]), dev_i32(d["cu_kept"]), scale=scale,
                                  initial_state=None if initial_state is None else dev_f32(initial_state),
                                  want_state=True)
    assert tg.tg_check_device_status() == tg.TG_OK
    return host_f64(o), s.double().cpu().numpy()


def check(o, s, ref_o, ref_s, label):
    err = np.abs(o - ref_o)
    lim = O_RTOL * np.abs(ref_o) + O_ATOL
    serr = np.abs(s - ref_s).max(initial=0.0)
    print(f"{label}: o max err {err.max(initial=0):.3e} (worst err/bound {(err / lim).max(initial=0):.2f}); "
          f"state max err {serr:.3e} of {np.abs(ref_s).max(initial=0):.3e}")
    assert np.all(np.isfinite(o)) and np.all(np.isfinite(s))
    assert np.all(err <= lim)
    assert serr <= S_REL * max(np.abs(ref_s).max(initial=0.0), 1e-6)


@pytest.mark.parametrize("name", ["deltanet-tiny", "deltanet-ragged", "deltanet-32k-k4096"])
def test_scan_workloads(tg, name):
    d = synth.deltanet_inputs(name)
    o, s = run_scan(tg, d)
    ref_o, ref_s = oracle.gated_delta_scan(d["q"], d["k"], d["v"], d["g"], d["beta"], d["cu_kept"])
    check(o, s, ref_o, ref_s, name)


def test_scan_initial_state_and_scale(tg):
    """A given initial state and a non-default scale, against the oracle."""
    d = synth.deltanet_inputs("deltanet-tiny")
    rng = np.random.default_rng(3)
    s0 = rng.standard_normal((1, 4, 64, 64)).astype(np.float32) * 0.1
    o, s = run_scan(tg, d, initial_state=s0, scale=0.3)
    ref_o, ref_s = oracle.gated_delta_scan(d["q"], d["k"], d["v"], d["g"], d["beta"], d["cu_kept"], scale=0.3,
                                           initial_state=s0.astype(np.float64))
    check(o, s, ref_o, ref_s, "initial state")


def test_scan_continues_across_calls(tg):
    """The second half started from the first half's final state gives what
    one call gives (the state passes through memory in fp32)."""
    d = synth.deltanet_inputs("deltanet-tiny")
    o, s = run_scan(tg, d)
    cut = 77
    first = {key: d[key][:cut] for key in ("q", "k", "v", "g", "beta")}
    first["cu_kept"] = np.array([0, cut], np.int32)
    second = {key: d[key][cut:] for key in ("q", "k", "v", "g", "beta")}
    second["cu_kept"] = np.array([0, len(d["g"]) - cut], np.int32)
    oa, sa = run_scan(tg, first)
    ob, sb = run_scan(tg, second, initial_state=sa.astype(np.float32))
    np.testing.assert_allclose(np.concatenate([oa, ob]), o, rtol=0, atol=1e-6)
    np.testing.assert_allclose(sb, s, rtol=0, atol=1e-6)


def test_scan_pruned_tokens_are_skipped(tg):
    """Every token with beta = 0 and g = 0 on the pruned ones gives, at the
    kept tokens, what the kept tokens alone give."""
    d = synth.deltanet_inputs("deltanet-tiny")
    rng = np.random.default_rng(4)
    n = len(d["g"])
    kept = np.sort(rng.choice(n, 61, replace=False))
    full = dict(d)
    full["g"] = np.zeros_like(d["g"])
    full["beta"] = np.zeros_like(d["beta"])
    full["g"][kept] = d["g"][kept]
    full["beta"][kept] = d["beta"][kept]
    o_all, s_all = run_scan(tg, full)
    sub = {key: d[key][kept] for key in ("q", "k", "v", "g", "beta")}
    sub["cu_kept"] = np.array([0, len(kept)], np.int32)
    o_k, s_k = run_scan(tg, sub)
    # a pruned token that touched the state would move o by ~0.1; the bound
    # leaves room for exp(0) evaluated one ulp away from 1 on every pruned token
    np.testing.assert_allclose(o_all[kept], o_k, rtol=0, atol=O_ATOL)
    np.testing.assert_allclose(s_all, s_k, rtol=0, atol=S_REL * max(np.abs(s_k).max(), 1e-6))


def test_scan_rejects_bad_sequences(tg):
    """cu_kept past n_kept is flagged on the device and nothing is read."""
    d = synth.deltanet_inputs("deltanet-tiny")
    bad = dict(d)
    bad["cu_kept"] = np.array([0, len(d["g"]) + 5], np.int32)
    tg.tg_check_device_status()
    tg.tg_gated_delta_scan(dev_bf16(bad["q"]), dev_bf16(bad["k"]), dev_bf16(bad["v"]), dev_f32(bad["g"]),
                           dev_f32(bad["beta"]), dev_i32(bad["cu_kept"]))
    assert tg.tg_check_device_status() == tg.TG_ERR_DEVICE_INDEX
