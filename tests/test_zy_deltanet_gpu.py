"""GPU parity of the pruned Gated DeltaNet scan (tg_gated_delta_scan)
against the fp64 oracle, in both of its forms: the chunked form on the
tensor cores (tf32 MMAs, with a workspace) and the token-by-token kernel.

Both keep the state in fp32 and round o once to bf16, so the bound on o is
the bf16 rounding (2^-9 relative) with a factor of two, plus an absolute
floor of 2e-4 (a float32 replay of the token-by-token arithmetic stays within
4e-8 of the oracle; a numpy replay of the chunked form's tf32 rounding points
reaches 0.61 of this bound on the three workloads).  The fp32 final state is
compared within 1e-4 of its largest entry for the token-by-token kernel and
within 2e-3 for the chunked form: four units of tf32 rounding (2^-11), the
precision of its products (the replay reaches 4e-4 to 7e-4).  Continuation and
pruning are checked GPU against GPU where the two computations round alike,
and against the oracle otherwise."""
import numpy as np
import pytest
import torch

import oracle
from learned_token_pruning_09_b300 import synth
from tests.helpers import dev_bf16, dev_f32, dev_i32, host_f64

pytestmark = pytest.mark.gpu

O_RTOL, O_ATOL = 2.0 ** -8, 2e-4
S_REL = {False: 1e-4, True: 2e-3}     # by form: token by token, chunked
FORMS = [pytest.param(True, id="chunked"), pytest.param(False, id="recurrent")]


@pytest.fixture(scope="module")
def tg():
    from learned_token_pruning_09_b300 import tokengate
    return tokengate


def run_scan(tg, d, chunked, initial_state=None, scale=None):
    o, s = tg.tg_gated_delta_scan(dev_bf16(d["q"]), dev_bf16(d["k"]), dev_bf16(d["v"]), dev_f32(d["g"]),
                                  dev_f32(d["beta"]), dev_i32(d["cu_kept"]), scale=scale,
                                  initial_state=None if initial_state is None else dev_f32(initial_state),
                                  want_state=True, chunked=chunked)
    assert tg.tg_check_device_status() == tg.TG_OK
    return host_f64(o), s.double().cpu().numpy()


def check(o, s, ref_o, ref_s, label, chunked):
    err = np.abs(o - ref_o)
    lim = O_RTOL * np.abs(ref_o) + O_ATOL
    serr = np.abs(s - ref_s).max(initial=0.0)
    print(f"{label}: o max err {err.max(initial=0):.3e} (worst err/bound {(err / lim).max(initial=0):.2f}); "
          f"state max err {serr:.3e} of {np.abs(ref_s).max(initial=0):.3e}")
    assert np.all(np.isfinite(o)) and np.all(np.isfinite(s))
    assert np.all(err <= lim)
    assert serr <= S_REL[chunked] * max(np.abs(ref_s).max(initial=0.0), 1e-6)


@pytest.mark.parametrize("chunked", FORMS)
@pytest.mark.parametrize("name", ["deltanet-tiny", "deltanet-ragged", "deltanet-32k-k4096"])
def test_scan_workloads(tg, name, chunked):
    d = synth.deltanet_inputs(name)
    o, s = run_scan(tg, d, chunked)
    ref_o, ref_s = oracle.gated_delta_scan(d["q"], d["k"], d["v"], d["g"], d["beta"], d["cu_kept"])
    check(o, s, ref_o, ref_s, name, chunked)


@pytest.mark.parametrize("chunked", FORMS)
def test_scan_initial_state_and_scale(tg, chunked):
    """A given initial state and a non-default scale, against the oracle."""
    d = synth.deltanet_inputs("deltanet-tiny")
    rng = np.random.default_rng(3)
    s0 = rng.standard_normal((1, 4, 64, 64)).astype(np.float32) * 0.1
    o, s = run_scan(tg, d, chunked, initial_state=s0, scale=0.3)
    ref_o, ref_s = oracle.gated_delta_scan(d["q"], d["k"], d["v"], d["g"], d["beta"], d["cu_kept"], scale=0.3,
                                           initial_state=s0.astype(np.float64))
    check(o, s, ref_o, ref_s, "initial state", chunked)


def split_at(d, cut):
    first = {key: d[key][:cut] for key in ("q", "k", "v", "g", "beta")}
    first["cu_kept"] = np.array([0, cut], np.int32)
    second = {key: d[key][cut:] for key in ("q", "k", "v", "g", "beta")}
    second["cu_kept"] = np.array([0, len(d["g"]) - cut], np.int32)
    return first, second


def test_scan_continues_across_calls(tg):
    """The second part started from the first part's final state gives what
    one call gives, exactly, for the token-by-token kernel (the state passes
    through memory in fp32 and both compute the same operations)."""
    d = synth.deltanet_inputs("deltanet-tiny")
    o, s = run_scan(tg, d, False)
    first, second = split_at(d, 77)
    oa, sa = run_scan(tg, first, False)
    ob, sb = run_scan(tg, second, False, initial_state=sa.astype(np.float32))
    np.testing.assert_allclose(np.concatenate([oa, ob]), o, rtol=0, atol=1e-6)
    np.testing.assert_allclose(sb, s, rtol=0, atol=1e-6)


@pytest.mark.parametrize("cut", [64, 77])
def test_scan_chunked_continues_across_calls(tg, cut):
    """The chunked form cut at a chunk boundary and inside a chunk: both parts
    against the oracle's single call.  (Not bit-exact against one call: a
    single call carries the chunks' decay as a scalar factor beside the
    state, a split call starts it over.)"""
    d = synth.deltanet_inputs("deltanet-tiny")
    first, second = split_at(d, cut)
    oa, sa = run_scan(tg, first, True)
    ob, sb = run_scan(tg, second, True, initial_state=sa.astype(np.float32))
    ref_o, ref_s = oracle.gated_delta_scan(d["q"], d["k"], d["v"], d["g"], d["beta"], d["cu_kept"])
    check(np.concatenate([oa, ob]), sb, ref_o, ref_s, f"cut at {cut}", True)


@pytest.mark.parametrize("chunked", FORMS)
def test_scan_pruned_tokens_are_skipped(tg, chunked):
    """Every token with beta = 0 and g = 0 on the pruned ones gives, at the
    kept tokens, what the kept tokens alone give: GPU against GPU for the
    token-by-token kernel; for the chunked form (the two sequences fall into
    different chunks) the full sequence against the oracle of the kept
    tokens alone."""
    d = synth.deltanet_inputs("deltanet-tiny")
    rng = np.random.default_rng(4)
    n = len(d["g"])
    kept = np.sort(rng.choice(n, 61, replace=False))
    full = dict(d)
    full["g"] = np.zeros_like(d["g"])
    full["beta"] = np.zeros_like(d["beta"])
    full["g"][kept] = d["g"][kept]
    full["beta"][kept] = d["beta"][kept]
    o_all, s_all = run_scan(tg, full, chunked)
    sub = {key: d[key][kept] for key in ("q", "k", "v", "g", "beta")}
    sub["cu_kept"] = np.array([0, len(kept)], np.int32)
    if chunked:
        ref_o, ref_s = oracle.gated_delta_scan(sub["q"], sub["k"], sub["v"], sub["g"], sub["beta"], sub["cu_kept"])
        check(o_all[kept], s_all, ref_o, ref_s, "pruned", True)
        return
    o_k, s_k = run_scan(tg, sub, chunked)
    # a pruned token that touched the state would move o by ~0.1; the bound
    # leaves room for exp(0) evaluated one ulp away from 1 on every pruned token
    np.testing.assert_allclose(o_all[kept], o_k, rtol=0, atol=O_ATOL)
    np.testing.assert_allclose(s_all, s_k, rtol=0, atol=S_REL[False] * max(np.abs(s_k).max(), 1e-6))


@pytest.mark.parametrize("chunked", FORMS)
@pytest.mark.parametrize("cu", ["end+5", "far"])
def test_scan_rejects_bad_sequences(tg, chunked, cu):
    """cu_kept past n_kept is flagged on the device and nothing is read or
    written outside the buffers: a sequence ending 5 tokens past the last
    one, and two sequences far past it (whose chunk slots lie beyond the
    workspace's)."""
    d = synth.deltanet_inputs("deltanet-tiny")
    bad = dict(d)
    n = len(d["g"])
    bad["cu_kept"] = (np.array([0, n + 5], np.int32) if cu == "end+5"
                      else np.array([0, 5000, 5100], np.int32))
    tg.tg_check_device_status()
    tg.tg_gated_delta_scan(dev_bf16(bad["q"]), dev_bf16(bad["k"]), dev_bf16(bad["v"]), dev_f32(bad["g"]),
                           dev_f32(bad["beta"]), dev_i32(bad["cu_kept"]), chunked=chunked)
    assert tg.tg_check_device_status() == tg.TG_ERR_DEVICE_INDEX


def test_scan_chunked_edge_shapes(tg):
    """The chunked form on dk = 64 with dv = 16 and 48 (rows of the 128-lane
    state tile left unused), sequences of 1, 63, 64, 65 and 0 tokens, and a
    q/k head shared by three value heads."""
    for dk, dv, hk, hv in ((64, 16, 1, 3), (64, 48, 2, 2), (128, 112, 1, 2)):
        lens = [1, 63, 64, 0, 65, 130]
        t = sum(lens)
        rng = np.random.default_rng(dk + dv)
        d = {"q": synth.f32_to_bf16_bits(rng.standard_normal((t, hk, dk)).astype(np.float32)),
             "k": synth.f32_to_bf16_bits(rng.standard_normal((t, hk, dk)).astype(np.float32)),
             "v": synth.f32_to_bf16_bits(rng.standard_normal((t, hv, dv)).astype(np.float32)),
             "g": (-np.exp(rng.uniform(np.log(0.005), np.log(0.5), (t, hv)))).astype(np.float32),
             "beta": rng.uniform(0.05, 0.95, (t, hv)).astype(np.float32),
             "cu_kept": np.concatenate([[0], np.cumsum(lens)]).astype(np.int32)}
        s0 = rng.standard_normal((len(lens), hv, dv, dk)).astype(np.float32) * 0.1
        o, s = run_scan(tg, d, True, initial_state=s0)
        ref_o, ref_s = oracle.gated_delta_scan(d["q"], d["k"], d["v"], d["g"], d["beta"], d["cu_kept"],
                                               initial_state=s0.astype(np.float64))
        check(o, s, ref_o, ref_s, f"dk {dk} dv {dv} hv {hv}", True)


def test_scan_chunked_many_sequences(tg):
    """300 sequences of 0 to 200 tokens (the per-chunk kernel finds each
    chunk's sequence by a binary search over cu_kept), against the oracle."""
    rng = np.random.default_rng(300)
    lens = rng.integers(0, 201, 300)
    lens[::37] = 0
    t, hk, hv, dk, dv = int(lens.sum()), 1, 2, 64, 32
    d = {"q": synth.f32_to_bf16_bits(rng.standard_normal((t, hk, dk)).astype(np.float32)),
         "k": synth.f32_to_bf16_bits(rng.standard_normal((t, hk, dk)).astype(np.float32)),
         "v": synth.f32_to_bf16_bits(rng.standard_normal((t, hv, dv)).astype(np.float32)),
         "g": (-np.exp(rng.uniform(np.log(0.005), np.log(0.5), (t, hv)))).astype(np.float32),
         "beta": rng.uniform(0.05, 0.95, (t, hv)).astype(np.float32),
         "cu_kept": np.concatenate([[0], np.cumsum(lens)]).astype(np.int32)}
    o, s = run_scan(tg, d, True)
    ref_o, ref_s = oracle.gated_delta_scan(d["q"], d["k"], d["v"], d["g"], d["beta"], d["cu_kept"])
    check(o, s, ref_o, ref_s, "300 sequences", True)


@pytest.mark.parametrize("chunked", FORMS)
def test_scan_without_final_state_gives_the_same_o(tg, chunked):
    """o does not depend on whether the final state is asked for."""
    d = synth.deltanet_inputs("deltanet-ragged")
    args = (dev_bf16(d["q"]), dev_bf16(d["k"]), dev_bf16(d["v"]), dev_f32(d["g"]), dev_f32(d["beta"]),
            dev_i32(d["cu_kept"]))
    o1, _ = tg.tg_gated_delta_scan(*args, want_state=True, chunked=chunked)
    o2 = tg.tg_gated_delta_scan(*args, chunked=chunked)
    assert tg.tg_check_device_status() == tg.TG_OK
    assert torch.equal(o1, o2)


def test_scan_one_launch_and_two_launches_agree(tg):
    """With few (sequence, head) pairs the chunked form runs as one
    cooperative launch, the per-chunk products on some SMs and the state carry
    on others, handing chunks over by flags; with many it runs two launches.
    The arithmetic is the same, so the same chunks padded with empty
    sequences (enough pairs for the two-launch form on any GPU up to 320 SMs)
    give bit-identical outputs: a hand-off that let the state carry read a
    unit before it was complete would show here."""
    d = synth.deltanet_inputs("deltanet-ragged")
    hv = d["v"].shape[1]
    one = run_scan(tg, d, True)
    padded = dict(d)
    n_empty = 160 // hv + 1
    padded["cu_kept"] = np.concatenate([d["cu_kept"], np.full(n_empty, d["cu_kept"][-1])]).astype(np.int32)
    two = run_scan(tg, padded, True)
    nb = len(d["cu_kept"]) - 1
    assert np.array_equal(one[0], two[0])
    assert np.array_equal(one[1], two[1][:nb])
    assert not np.any(two[1][nb:])                # empty sequences keep the zero state


def _random_scan_inputs(rng, lens, hk, hv, dk, dv):
    t = int(sum(lens))
    return {"q": synth.f32_to_bf16_bits(rng.standard_normal((t, hk, dk)).astype(np.float32)),
            "k": synth.f32_to_bf16_bits(rng.standard_normal((t, hk, dk)).astype(np.float32)),
            "v": synth.f32_to_bf16_bits(rng.standard_normal((t, hv, dv)).astype(np.float32)),
            "g": (-np.exp(rng.uniform(np.log(0.005), np.log(0.5), (t, hv)))).astype(np.float32),
            "beta": rng.uniform(0.05, 0.95, (t, hv)).astype(np.float32),
            "cu_kept": np.concatenate([[0], np.cumsum(lens)]).astype(np.int32)}


@pytest.mark.parametrize("extra", [0, 1])
def test_scan_chunked_at_the_one_launch_threshold(tg, extra):
    """batch * hv equal to half the SMs (the largest one-launch shape) and one
    sequence more (two launches), against the oracle."""
    half = torch.cuda.get_device_properties(0).multi_processor_count // 2
    hv, hk, dk, dv = 2, 1, 64, 32
    batch = half // hv + extra
    rng = np.random.default_rng(half + extra)
    lens = rng.integers(1, 140, batch)
    d = _random_scan_inputs(rng, lens, hk, hv, dk, dv)
    o, s = run_scan(tg, d, True)
    ref_o, ref_s = oracle.gated_delta_scan(d["q"], d["k"], d["v"], d["g"], d["beta"], d["cu_kept"])
    check(o, s, ref_o, ref_s, f"batch {batch} x hv {hv} (SMs / 2 = {half})", True)


def test_scan_chunked_workspace_contents_do_not_matter(tg):
    """The same workspace used twice, then filled with 0xFF bytes (every flag
    and every operand set to garbage): the outputs are the same bits each
    time."""
    d = synth.deltanet_inputs("deltanet-ragged")
    args = (dev_bf16(d["q"]), dev_bf16(d["k"]), dev_bf16(d["v"]), dev_f32(d["g"]), dev_f32(d["beta"]),
            dev_i32(d["cu_kept"]))
    t, hv, dv = d["v"].shape
    dk = d["q"].shape[2]
    nb = len(d["cu_kept"]) - 1
    ws = torch.zeros(tg.tg_gated_delta_scan_workspace_size(t, nb, hv, dk, dv), dtype=torch.uint8, device="cuda")
    o1, s1 = tg.tg_gated_delta_scan(*args, want_state=True, workspace=ws)
    o2, s2 = tg.tg_gated_delta_scan(*args, want_state=True, workspace=ws)
    ws.fill_(0xFF)
    o3, s3 = tg.tg_gated_delta_scan(*args, want_state=True, workspace=ws)
    assert tg.tg_check_device_status() == tg.TG_OK
    assert torch.equal(o1, o2) and torch.equal(o1, o3)
    assert torch.equal(s1, s2) and torch.equal(s1, s3)


def test_scan_chunked_dk64_at_scale(tg):
    """dk = dv = 64 on two sequences of ~4k tokens in all, 32 value heads over
    8 q/k heads (64 (sequence, head) pairs: the one-launch form with dk = 64
    at a size that keeps every SM busy), against the oracle."""
    rng = np.random.default_rng(64)
    lens = [2000, 2100]
    d = _random_scan_inputs(rng, lens, 8, 32, 64, 64)
    o, s = run_scan(tg, d, True)
    ref_o, ref_s = oracle.gated_delta_scan(d["q"], d["k"], d["v"], d["g"], d["beta"], d["cu_kept"])
    check(o, s, ref_o, ref_s, "dk 64 at scale", True)
