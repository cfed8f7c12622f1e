"""Failure detection without a GPU fault: every device-side wait in the
tensor-core kernels has a cycle limit.  With the limit set far below a TMA
round trip (200 cycles) the first waits run out; the kernel records
TG_ERR_TIMEOUT in the status word, drains its own copies and MMAs in flight
(with a separate, long limit), frees TMEM and returns.  The host reads the
status, restores the default limit, and the same context computes correct
results again."""
import numpy as np
import pytest
import torch

import oracle
from learned_token_pruning_09_b300 import synth
from tests.helpers import allclose_report, dev_bf16, dev_f32, dev_i32, host_f64

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def tg():
    from learned_token_pruning_09_b300 import tokengate
    yield tokengate
    tokengate.tg_set_watchdog_cycles(0)          # default limit for whatever runs next


def _gate(tg, shape, x, p):
    return tg.tg_gate_score(dev_bf16(x), dev_i32(shape.cu_seqlens), dev_i32(shape.n_doc), dev_bf16(p["w1"]),
                            None, dev_bf16(p["w2"]), p["b2"])


def test_gate_wait_runs_out_then_recovers(tg):
    shape = synth.custom("w", [8000], [64], [100], d=2048, h=256)
    x, p = synth.residuals(shape), synth.gate_weights(shape)
    tg.tg_check_device_status()                  # start clean
    tg.tg_set_watchdog_cycles(200)
    _gate(tg, shape, x, p)
    assert tg.tg_check_device_status() == tg.TG_ERR_TIMEOUT
    tg.tg_set_watchdog_cycles(0)
    s = _gate(tg, shape, x, p).cpu().numpy()
    assert tg.tg_check_device_status() == tg.TG_OK
    rows = np.arange(0, shape.n_rows, 97)
    ref = oracle.gate_score(x, shape.cu_seqlens, shape.n_doc, p["w1"], p["b1"], p["w2"], p["b2"], rows=rows)
    np.testing.assert_allclose(s[rows], ref[rows], atol=1e-4, rtol=0)


def test_attention_wait_runs_out_then_recovers(tg):
    rng = np.random.default_rng(3)
    t, hq, hkv, d = 1500, 16, 8, 128
    bf = lambda a: dev_bf16(synth.f32_to_bf16_bits(a.astype(np.float32)))
    qn = synth.f32_to_bf16_bits(rng.standard_normal((t, hq, d)).astype(np.float32))
    kn = synth.f32_to_bf16_bits(rng.standard_normal((t, hkv, d)).astype(np.float32))
    vn = synth.f32_to_bf16_bits(rng.standard_normal((t, hkv, d)).astype(np.float32))
    pos = np.arange(t, dtype=np.int32) * 2
    s = -np.abs(rng.normal(0, 1, t)).astype(np.float32)
    gain = rng.uniform(0.5, 2, hq).astype(np.float32)
    args = (dev_bf16(qn), dev_bf16(kn), dev_bf16(vn), dev_i32(pos), dev_f32(s), dev_f32(gain), 1.1, 1e6,
            dev_i32([0, t]), t)
    tg.tg_check_device_status()
    tg.tg_set_watchdog_cycles(200)
    tg.tg_gated_attention_fwd(*args)
    assert tg.tg_check_device_status() == tg.TG_ERR_TIMEOUT
    tg.tg_set_watchdog_cycles(0)
    o = tg.tg_gated_attention_fwd(*args)
    assert tg.tg_check_device_status() == tg.TG_OK
    rows = np.arange(0, t, 37)
    ref, _ = oracle.gated_attention(qn, kn, vn, pos, s, gain, 1.1, [0, t], rows=rows)
    ok, err, _ = allclose_report(host_f64(o)[rows], ref[rows], 2e-2, 1e-2)
    assert ok, err


def test_linear_wait_runs_out_then_recovers(tg):
    rng = np.random.default_rng(4)
    a = synth.f32_to_bf16_bits(rng.standard_normal((1000, 2048)).astype(np.float32))
    w = synth.f32_to_bf16_bits((rng.standard_normal((1024, 2048)) / 45).astype(np.float32))
    tg.tg_check_device_status()
    tg.tg_set_watchdog_cycles(200)
    tg.tg_linear_bf16(dev_bf16(a), dev_bf16(w))
    assert tg.tg_check_device_status() == tg.TG_ERR_TIMEOUT
    tg.tg_set_watchdog_cycles(0)
    out = host_f64(tg.tg_linear_bf16(dev_bf16(a), dev_bf16(w)))
    assert tg.tg_check_device_status() == tg.TG_OK
    ref = oracle.bf16_decode(a) @ oracle.bf16_decode(w).T
    ok, err, _ = allclose_report(out, ref, 1e-2, 1e-2)
    assert ok, err


def test_chunked_delta_scan_wait_runs_out_then_recovers(tg):
    """Both kernels of the chunked scan: the per-chunk products wait for each
    MMA past the limit and then for the same MMA with the drain limit; the
    state carry's roles stop, drain their copies and MMAs and free TMEM."""
    d = synth.deltanet_inputs("deltanet-tiny")
    args = (dev_bf16(d["q"]), dev_bf16(d["k"]), dev_bf16(d["v"]), dev_f32(d["g"]), dev_f32(d["beta"]),
            dev_i32(d["cu_kept"]))
    tg.tg_check_device_status()
    tg.tg_set_watchdog_cycles(200)
    tg.tg_gated_delta_scan(*args, chunked=True)
    assert tg.tg_check_device_status() == tg.TG_ERR_TIMEOUT
    tg.tg_set_watchdog_cycles(0)
    o = tg.tg_gated_delta_scan(*args, chunked=True)
    assert tg.tg_check_device_status() == tg.TG_OK
    ref, _ = oracle.gated_delta_scan(d["q"], d["k"], d["v"], d["g"], d["beta"], d["cu_kept"])
    ok, err, _ = allclose_report(host_f64(o), ref, 2e-4, 2.0 ** -8)
    assert ok, err


def test_chunked_delta_scan_two_launches_wait_runs_out_then_recovers(tg):
    """The same for the two-launch form of the chunked scan (the input padded
    with empty sequences to more (sequence, head) pairs than one launch takes
    on any GPU up to 320 SMs)."""
    d = synth.deltanet_inputs("deltanet-tiny")
    t, hv = d["v"].shape[0], d["v"].shape[1]
    cu = np.concatenate([d["cu_kept"], np.full(160 // hv + 1, t)]).astype(np.int32)
    args = (dev_bf16(d["q"]), dev_bf16(d["k"]), dev_bf16(d["v"]), dev_f32(d["g"]), dev_f32(d["beta"]), dev_i32(cu))
    tg.tg_check_device_status()
    tg.tg_set_watchdog_cycles(200)
    tg.tg_gated_delta_scan(*args, chunked=True)
    assert tg.tg_check_device_status() == tg.TG_ERR_TIMEOUT
    tg.tg_set_watchdog_cycles(0)
    o = tg.tg_gated_delta_scan(*args, chunked=True)
    assert tg.tg_check_device_status() == tg.TG_OK
    ref, _ = oracle.gated_delta_scan(d["q"], d["k"], d["v"], d["g"], d["beta"], d["cu_kept"])
    ok, err, _ = allclose_report(host_f64(o), ref, 2e-4, 2.0 ** -8)
    assert ok, err
