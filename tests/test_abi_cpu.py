"""The C-ABI library loads without a GPU, exports every symbol declared in
include/tokengate.h, and rejects invalid arguments on the host before any
CUDA call."""
import ctypes
import os
import re
import subprocess

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "tokengate.h")


@pytest.fixture(scope="module")
def tg():
    from learned_token_pruning_09_b300 import build
    build.build()
    from learned_token_pruning_09_b300 import tokengate
    return tokengate


def declared_symbols():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(tg_[a-z0-9_]+)\s*\(", text)))


def test_header_declares_the_path():
    syms = declared_symbols()
    for s in ("tg_gate_score", "tg_topk_select", "tg_gather_kept", "tg_gated_attention_fwd"):
        assert s in syms


def test_library_exports_every_declared_symbol(tg):
    out = subprocess.run(["nm", "-D", "--defined-only", tg.LIB_PATH], capture_output=True, text=True,
                         check=True).stdout
    exported = set(re.findall(r"\bT (tg_[a-z0-9_]+)\b", out))
    missing = [s for s in declared_symbols() if s not in exported]
    assert not missing, missing
    for s in declared_symbols():
        assert hasattr(tg.lib, s)


def test_version_and_error_string(tg):
    assert "sm_103a" in tg.version()
    assert isinstance(tg.lib.tg_last_error_string(), bytes)


def test_workspace_size(tg):
    ws = tg.tg_attention_workspace_size(8256, 16, 8, 128, True)
    assert ws == ((8256 * 16 * 128 * 2 + 255) // 256) * 256
    ws2 = tg.tg_attention_workspace_size(8256, 16, 8, 128, False)
    assert ws2 == ws + ((8256 * 8 * 128 * 2 + 255) // 256) * 256
    assert tg.tg_attention_workspace_size(0, 16, 8, 128, True) == 0


def _c(v):
    return ctypes.c_void_p(v)


def test_host_validation_rejects_before_launch(tg):
    L = tg.lib
    p = _c(256)      # a fake 16-byte-aligned address: never dereferenced
    # gate: d not a multiple of 64, h out of range, null weights, misalignment
    assert L.tg_gate_score(p, 10, 63, p, p, 1, p, None, p, 0.0, 64, p, None, 0, None) == tg.TG_ERR_INVALID_ARG
    assert L.tg_gate_score(p, 10, 64, p, p, 1, p, None, p, 0.0, 8, p, None, 0, None) == tg.TG_ERR_INVALID_ARG
    assert L.tg_gate_score(p, 10, 64, p, p, 1, p, None, p, 0.0, 272, p, None, 0, None) == tg.TG_ERR_INVALID_ARG
    assert L.tg_gate_score(p, 10, 64, p, p, 1, None, None, p, 0.0, 64, p, None, 0, None) == tg.TG_ERR_INVALID_ARG
    assert L.tg_gate_score(_c(258), 10, 64, p, p, 1, p, None, p, 0.0, 64, p, None, 0, None) == tg.TG_ERR_INVALID_ARG
    assert L.tg_gate_score(p, 10, 64, p, p, 0, p, None, p, 0.0, 64, p, None, 0, None) == tg.TG_ERR_INVALID_ARG
    assert L.tg_gate_score(p, 10, 64, p, p, 1, p, None, p, float("nan"), 64, p, None, 0, None) == tg.TG_ERR_INVALID_ARG
    assert b"multiple of 16" in L.tg_last_error_string() or L.tg_last_error_string()
    # top-K
    assert L.tg_topk_select(p, 10, p, p, p, -1, 5, p, p, None, 0, None) == tg.TG_ERR_INVALID_ARG
    assert L.tg_topk_select(p, 10, p, p, p, 1, -1, p, p, None, 0, None) == tg.TG_ERR_INVALID_ARG
    assert L.tg_topk_select(p, 10, None, p, p, 1, 5, p, p, None, 0, None) == tg.TG_ERR_INVALID_ARG
    assert L.tg_topk_select(p, 10, p, p, p, 0, 5, p, p, None, 0, None) == tg.TG_OK       # empty batch: no-op
    # the top-K workspace (the gate's score histograms): size, alignment, batch limit
    ws = L.tg_topk_workspace_size(3)
    assert ws == 3 * (256 + 65536) * 4
    assert L.tg_topk_workspace_size(0) == 0 and L.tg_topk_workspace_size(65536) == 0
    assert L.tg_topk_select(p, 10, p, p, p, 3, 5, p, p, p, ws - 4, None) == tg.TG_ERR_WORKSPACE
    assert L.tg_topk_select(p, 10, p, p, p, 3, 5, p, p, _c(264), ws, None) == tg.TG_ERR_INVALID_ARG
    assert L.tg_topk_select(p, 10, p, p, p, 70000, 5, p, p, p, ws, None) == tg.TG_ERR_INVALID_ARG
    assert L.tg_gate_score(p, 10, 64, p, p, 3, p, None, p, 0.0, 64, p, p, ws - 4, None) == tg.TG_ERR_WORKSPACE
    assert L.tg_gate_score(p, 10, 64, p, p, 3, p, None, p, 0.0, 64, p, _c(264), ws, None) == tg.TG_ERR_INVALID_ARG
    # general prunable spans
    assert L.tg_gate_score_masked(p, 10, 64, None, p, None, p, 0.0, 64, p, None, 0, None, 0, None) == tg.TG_ERR_INVALID_ARG
    assert L.tg_gate_score_masked(p, 10, 63, p, p, None, p, 0.0, 64, p, None, 0, None, 0, None) == tg.TG_ERR_INVALID_ARG
    assert L.tg_gate_score_masked(p, 0, 64, None, p, None, p, 0.0, 64, p, None, 0, None, 0, None) == tg.TG_OK
    assert L.tg_topk_select_masked(p, 10, p, p, p, 1, -1, 10, p, p, p, None, 0, None) == tg.TG_ERR_INVALID_ARG
    assert L.tg_topk_select_masked(p, 10, p, p, p, 1, 10, -1, p, p, p, None, 0, None) == tg.TG_ERR_INVALID_ARG
    assert L.tg_topk_select_masked(p, 10, p, None, p, 1, 10, 10, p, p, p, None, 0, None) == tg.TG_ERR_INVALID_ARG
    assert L.tg_topk_select_masked(p, 10, p, p, p, 1, 10, 10, p, p, None, None, 0, None) == tg.TG_ERR_INVALID_ARG
    assert L.tg_topk_select_masked(p, 10, p, p, p, 0, 10, 10, p, p, p, None, 0, None) == tg.TG_OK     # empty batch
    # gather
    assert L.tg_gather_kept(p, 10, 12, p, p, p, p, 1, 4, p, p, p, None) == tg.TG_ERR_INVALID_ARG
    assert L.tg_gather_kept(p, 10, 64, p, p, None, p, 1, 4, p, p, p, None) == tg.TG_ERR_INVALID_ARG
    assert L.tg_gather_kept(p, 10, 64, p, p, p, p, 0, 4, p, p, p, None) == tg.TG_ERR_INVALID_ARG
    # attention
    args = dict(q=p, k=p, v=p, pos=p, s=p, g=p, tau=1.0, th=1e6, cu=p, b=1, t=100, mk=100, hq=16, hkv=8, d=128,
                o=p, lse=None, kc=None, ws=p, wsb=1 << 30)

    def attn(**kw):
        a = dict(args, **kw)
        return L.tg_gated_attention_fwd(a["q"], a["k"], a["v"], a["pos"], a["s"], a["g"], a["tau"], a["th"],
                                        a["cu"], a["b"], a["t"], a["mk"], a["hq"], a["hkv"], a["d"], a["o"],
                                        a["lse"], a["kc"], a["ws"], a["wsb"], None)
    assert attn(hq=12, hkv=8) == tg.TG_ERR_INVALID_ARG
    assert attn(d=96) == tg.TG_ERR_UNSUPPORTED
    assert attn(tau=0.0) == tg.TG_ERR_INVALID_ARG
    assert attn(tau=float("inf")) == tg.TG_ERR_INVALID_ARG
    assert attn(wsb=10) == tg.TG_ERR_WORKSPACE
    assert attn(ws=None) == tg.TG_ERR_WORKSPACE
    assert attn(ws=_c(272)) == tg.TG_ERR_INVALID_ARG        # not 256-byte aligned
    assert attn(o=None) == tg.TG_ERR_INVALID_ARG
    assert attn(q=_c(264)) == tg.TG_ERR_INVALID_ARG         # not 16-byte aligned
    assert attn(b=0) == tg.TG_ERR_INVALID_ARG
    assert attn(t=0) == tg.TG_OK                            # nothing to do
    # the two steps of the fused call
    assert L.tg_rope_qk(p, p, p, 1e6, p, 1, 100, 16, 8, 96, p, _c(512), None) == tg.TG_ERR_UNSUPPORTED
    assert L.tg_rope_qk(p, p, p, 0.0, p, 1, 100, 16, 8, 128, p, _c(512), None) == tg.TG_ERR_INVALID_ARG
    assert L.tg_rope_qk(p, p, p, 1e6, p, 1, 100, 16, 8, 128, p, p, None) == tg.TG_ERR_INVALID_ARG  # k_out aliases k
    assert L.tg_rope_qk(p, p, p, 1e6, None, 1, 100, 16, 8, 128, _c(512), _c(768), None) == tg.TG_ERR_INVALID_ARG
    assert L.tg_rope_qk(p, p, p, 1e6, p, 1, 0, 16, 8, 128, _c(512), _c(768), None) == tg.TG_OK
    rot = lambda **kw: L.tg_gated_attention_rotated(
        *(lambda a: (a["q"], a["k"], a["v"], a["pos"], a["s"], a["g"], a["tau"], a["cu"], a["b"], a["t"], a["mk"],
                     a["hq"], a["hkv"], a["d"], a["o"], a["lse"], None))(dict(args, **kw)))
    assert rot(hq=12, hkv=8) == tg.TG_ERR_INVALID_ARG
    assert rot(tau=-1.0) == tg.TG_ERR_INVALID_ARG
    assert rot(v=None) == tg.TG_ERR_INVALID_ARG
    assert rot(k=_c(264)) == tg.TG_ERR_INVALID_ARG
    assert rot(mk=0) == tg.TG_OK
    # attention backward w.r.t. s, gain and tau
    bw = dict(q=p, k=p, v=p, o=p, lse=p, do=p, pos=p, s=p, g=p, tau=1.0, cu=p, b=1, t=100, mk=100, hq=16, hkv=8,
              d=128, ds=p, dg=p, dt=p, ws=p, wsb=1 << 30)

    def bwd(**kw):
        a = dict(bw, **kw)
        return L.tg_gated_attention_bwd(a["q"], a["k"], a["v"], a["o"], a["lse"], a["do"], a["pos"], a["s"], a["g"],
                                        a["tau"], a["cu"], a["b"], a["t"], a["mk"], a["hq"], a["hkv"], a["d"],
                                        a["ds"], a["dg"], a["dt"], a["ws"], a["wsb"], None)
    assert bwd(hq=12, hkv=8) == tg.TG_ERR_INVALID_ARG
    assert bwd(hq=18, hkv=2) == tg.TG_ERR_UNSUPPORTED        # more than 8 query heads per KV head
    assert bwd(hq=512, hkv=64) == tg.TG_ERR_UNSUPPORTED      # more than 256 query heads
    assert bwd(d=96) == tg.TG_ERR_UNSUPPORTED
    assert bwd(tau=0.0) == tg.TG_ERR_INVALID_ARG
    assert bwd(mk=-1) == tg.TG_ERR_INVALID_ARG
    assert bwd(dg=None) == tg.TG_ERR_INVALID_ARG
    assert bwd(ds=None) == tg.TG_ERR_INVALID_ARG
    assert bwd(lse=None) == tg.TG_ERR_INVALID_ARG
    assert bwd(do=_c(264)) == tg.TG_ERR_INVALID_ARG         # not 16-byte aligned
    assert bwd(wsb=10) == tg.TG_ERR_WORKSPACE
    assert bwd(ws=_c(272)) == tg.TG_ERR_INVALID_ARG          # not 256-byte aligned
    assert L.tg_attention_bwd_workspace_size(100, 16) >= 5 * 100 * 16 * 4 + 16 * 64 * 4
    assert L.tg_attention_bwd_workspace_size(0, 16) == 0
    # pruned Gated DeltaNet scan
    sc = dict(q=p, k=p, v=p, g=p, beta=p, cu=p, b=1, t=100, hk=16, hv=32, dk=128, dv=128, scale=0.088,
              s0=None, o=p, s1=None, ws=None, wsb=0)

    def scan(**kw):
        a = dict(sc, **kw)
        return L.tg_gated_delta_scan(a["q"], a["k"], a["v"], a["g"], a["beta"], a["cu"], a["b"], a["t"], a["hk"],
                                     a["hv"], a["dk"], a["dv"], a["scale"], a["s0"], a["o"], a["s1"], a["ws"],
                                     a["wsb"], None)
    assert scan(hv=24) == tg.TG_ERR_INVALID_ARG               # hv not a multiple of hk
    assert scan(dk=96) == tg.TG_ERR_UNSUPPORTED
    assert scan(dv=0) == tg.TG_ERR_INVALID_ARG
    assert scan(scale=0.0) == tg.TG_ERR_INVALID_ARG
    assert scan(scale=float("nan")) == tg.TG_ERR_INVALID_ARG
    assert scan(b=0) == tg.TG_ERR_INVALID_ARG
    assert scan(cu=None) == tg.TG_ERR_INVALID_ARG
    assert scan(beta=None) == tg.TG_ERR_INVALID_ARG
    assert scan(o=None) == tg.TG_ERR_INVALID_ARG
    assert scan(k=_c(264)) == tg.TG_ERR_INVALID_ARG           # not 16-byte aligned
    assert scan(v=_c(264)) == tg.TG_ERR_INVALID_ARG
    assert scan(dv=24) == tg.TG_ERR_INVALID_ARG               # not a multiple of the 16-row blocks
    # the chunked form's workspace: per (chunk slot, value head) the [W2; Qe]
    # and Kd^T images, W1^T, Oloc^T and gamma_C; slots = n_kept / 64 + batch + 1
    wsz = L.tg_gated_delta_scan_workspace_size
    assert wsz(100, 1, 32, 128, 128) == (100 // 64 + 2) * 32 * (128 * 128 * 4 + 128 * 64 * 4 + 2 * 128 * 64 * 4 + 16)
    assert wsz(100, 1, 32, 128, 256) == 0                    # dv > 128: token-by-token kernel only
    assert wsz(100, 1, 32, 96, 128) == 0
    assert wsz(100, 0, 32, 128, 128) == 0
    assert wsz(0, 3, 4, 64, 64) > 0
    assert scan(ws=p, wsb=10) == tg.TG_ERR_WORKSPACE
    assert scan(ws=_c(272), wsb=1 << 40) == tg.TG_ERR_INVALID_ARG   # not 256-byte aligned
    # the layer around the path: norms, SwiGLU, decode attention
    assert L.tg_rms_norm(p, p, 10, 12, 1e-6, p, None) == tg.TG_ERR_INVALID_ARG       # d not a multiple of 8
    assert L.tg_rms_norm(p, p, 10, 64, -1.0, p, None) == tg.TG_ERR_INVALID_ARG       # negative eps
    assert L.tg_rms_norm(p, None, 10, 64, 1e-6, p, None) == tg.TG_ERR_INVALID_ARG
    assert L.tg_rms_norm(_c(264), p, 10, 64, 1e-6, p, None) == tg.TG_ERR_INVALID_ARG  # not 16-byte aligned
    assert L.tg_rms_norm(p, p, 0, 64, 1e-6, p, None) == tg.TG_OK
    assert L.tg_swiglu(p, 10, 12, p, None) == tg.TG_ERR_INVALID_ARG
    assert L.tg_swiglu(p, 10, 64, None, None) == tg.TG_ERR_INVALID_ARG
    assert L.tg_swiglu(p, 0, 64, p, None) == tg.TG_OK
    dargs = dict(q=p, kn=p, vn=p, kc=p, vc=p, cu=p, b=2, rows=100, ml=60, s=None, g=None, tau=1.0, hq=16, hkv=8,
                 d=128, o=p, ws=p, wsb=1 << 30)

    def dec(**kw):
        a = dict(dargs, **kw)
        return L.tg_decode_attention(a["q"], a["kn"], a["vn"], a["kc"], a["vc"], a["cu"], a["b"], a["rows"],
                                     a["ml"], a["s"], a["g"], a["tau"], a["hq"], a["hkv"], a["d"], a["o"], a["ws"],
                                     a["wsb"], None)
    assert dec(hq=12) == tg.TG_ERR_INVALID_ARG
    assert dec(hq=18, hkv=2) == tg.TG_ERR_UNSUPPORTED
    assert dec(d=96) == tg.TG_ERR_UNSUPPORTED
    assert dec(tau=0.0) == tg.TG_ERR_INVALID_ARG
    assert dec(s=p) == tg.TG_ERR_INVALID_ARG                 # s_cache without gain
    assert dec(kc=None) == tg.TG_ERR_INVALID_ARG
    assert dec(wsb=8) == tg.TG_ERR_WORKSPACE
    assert dec(b=0) == tg.TG_OK
    assert L.tg_decode_workspace_size(2, 16, 128, 600) == 2 * 16 * 3 * 130 * 4
    assert L.tg_decode_workspace_size(2, 16, 128, 0) == 2 * 16 * 1 * 130 * 4
    # linear
    assert L.tg_linear_bf16(p, p, None, p, 10, 24, 64, None) == tg.TG_ERR_INVALID_ARG
    assert L.tg_linear_bf16(p, p, None, p, 10, 32, 96, None) == tg.TG_ERR_INVALID_ARG
    assert L.tg_linear_bf16(p, None, None, p, 10, 32, 64, None) == tg.TG_ERR_INVALID_ARG
    assert L.tg_linear_bf16(p, p, None, p, 0, 32, 64, None) == tg.TG_OK
    # the fused Q/K/V projection: head size, kdim, theta and pointers checked on the host
    assert L.tg_qkv_rope_bf16(p, p, 10, 64, 4, 2, 96, p, 1e6, p, p, p, None) == tg.TG_ERR_UNSUPPORTED
    assert L.tg_qkv_rope_bf16(p, p, 10, 96, 4, 2, 64, p, 1e6, p, p, p, None) == tg.TG_ERR_INVALID_ARG
    assert L.tg_qkv_rope_bf16(p, p, 10, 64, 4, 2, 64, p, 0.0, p, p, p, None) == tg.TG_ERR_INVALID_ARG
    assert L.tg_qkv_rope_bf16(p, p, 10, 64, 4, 2, 64, None, 1e6, p, p, p, None) == tg.TG_ERR_INVALID_ARG
    assert L.tg_qkv_rope_bf16(p, p, 10, 64, 0, 2, 64, p, 1e6, p, p, p, None) == tg.TG_ERR_INVALID_ARG
    assert L.tg_qkv_rope_bf16(p, p, 0, 64, 4, 2, 64, p, 1e6, p, p, p, None) == tg.TG_OK


def test_binding_refuses_cpu_tensors(tg):
    import torch
    x = torch.zeros(4, 64, dtype=torch.bfloat16)
    with pytest.raises((ValueError, TypeError)):
        tg.tg_linear_bf16(x, x)
