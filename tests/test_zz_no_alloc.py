"""tg_gated_attention_fwd_noalloc: token-gated attention for callers that
cannot allocate device memory when they call (an engine that plans all of
its device memory at start-up, a plugin under a runtime that owns the
allocator, a plain C program without a scratch buffer).  Its scratch space
is a fixed array inside the library instead of a caller-provided workspace.

The test calls it through the C ABI (ctypes on libtokengate.so) twice in a
row and checks both outputs against tg_gated_attention_fwd with a workspace.
The two run the same kernels on the same inputs, so o and lse must be equal
bit for bit; a wrong offset or an overlap of q' and k' inside the fixed array
would break that.  It also checks that a problem larger than the fixed
scratch is refused.  It sits in a file of its own that pytest collects last."""
import ctypes

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
    f = tokengate.lib.tg_gated_attention_fwd_noalloc
    vp, i32, i64, f32 = ctypes.c_void_p, ctypes.c_int32, ctypes.c_int64, ctypes.c_float
    f.argtypes = [vp, vp, vp, vp, vp, vp, f32, f32, vp, i32, i64, i32, i32, i32, i32, vp, vp, vp, vp]
    f.restype = ctypes.c_int
    tokengate.lib.tg_attention_static_scratch_bytes.argtypes = []
    tokengate.lib.tg_attention_static_scratch_bytes.restype = ctypes.c_size_t
    return tokengate


def _p(t):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def test_noalloc_matches_workspace_entry_point_twice(tg):
    shape = synth.ragged_batch()
    shape = synth.custom("r", [n // 16 for n in shape.n_doc], shape.n_q, [k // 16 for k in shape.k],
                         d=2048, h=256, hq=16, hkv=8, head_dim=128)
    s_rows = synth.score_draws(shape)
    kept, cu_kept = oracle.topk_select(s_rows, shape.cu_seqlens, shape.n_doc, shape.k)
    _, pos, s_kept = oracle.gather_kept(np.zeros((shape.n_rows, 1), np.uint16), s_rows, shape.cu_seqlens,
                                        kept, cu_kept)
    ai = synth.attention_inputs(shape, n_kept=len(kept))
    q, k, v = dev_bf16(ai["q"]), dev_bf16(ai["k"]), dev_bf16(ai["v"])
    pos_d, sk_d, gain_d, cu_d = dev_i32(pos), dev_f32(s_kept), dev_f32(ai["gain"]), dev_i32(cu_kept)
    t, hq, dh = q.shape
    hkv = k.shape[1]
    max_kept = int(np.diff(cu_kept).max())
    o_ref, lse_ref = tg.tg_gated_attention_fwd(q, k, v, pos_d, sk_d, gain_d, ai["tau"], 1e6, cu_d, max_kept,
                                               want_lse=True)
    assert tg.tg_check_device_status() == tg.TG_OK
    stream = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    for call in range(2):
        o = torch.full_like(q, float("nan"))
        lse = torch.full((hq, t), float("nan"), dtype=torch.float32, device=q.device)
        kc = torch.empty_like(k) if call == 1 else None        # both scratch layouts
        rc = tg.lib.tg_gated_attention_fwd_noalloc(
            _p(q), _p(k), _p(v), _p(pos_d), _p(sk_d), _p(gain_d), float(ai["tau"]), 1e6, _p(cu_d),
            cu_d.shape[0] - 1, t, max_kept, hq, hkv, dh, _p(o), _p(lse), _p(kc), stream)
        assert rc == tg.TG_OK, tg.lib.tg_last_error_string().decode()
        assert tg.tg_check_device_status() == tg.TG_OK
        if not torch.equal(o.view(torch.int16), o_ref.view(torch.int16)):
            ok, err, _ = allclose_report(host_f64(o), host_f64(o_ref), 2e-2, 1e-2)
            pytest.fail(f"call {call}: o differs from the workspace call (max |err| {err:.3e}, "
                        f"within the attention tolerance: {ok})")
        assert torch.equal(lse, lse_ref), f"call {call}: lse differs from the workspace call"


def test_noalloc_refuses_problems_beyond_its_scratch(tg):
    cap = int(tg.lib.tg_attention_static_scratch_bytes())
    assert cap == 64 << 20
    hq, hkv, dh = 16, 8, 128
    too_many = cap // (hq * dh * 2) + 1          # q' alone no longer fits
    assert tg.tg_attention_workspace_size(too_many, hq, hkv, dh, True) > cap
    fake = ctypes.c_void_p(256)                  # never dereferenced: refused before any launch
    rc = tg.lib.tg_gated_attention_fwd_noalloc(fake, fake, fake, fake, fake, fake, 1.0, 1e6, fake, 1,
                                               too_many, too_many, hq, hkv, dh, fake, None, fake, None)
    assert rc == tg.TG_ERR_WORKSPACE
    assert b"fixed scratch" in tg.lib.tg_last_error_string()
