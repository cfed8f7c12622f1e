"""Python binding of libtokengate.so (C ABI in include/tokengate.h).

Argument marshalling only: each ``tg_*`` function here takes torch CUDA
tensors, checks dtypes/shapes/contiguity, allocates outputs with torch when
the caller passes none, and calls the C entry point of the same name on the
current CUDA stream.  Every step of the path runs in the library's kernels;
there is no fallback: if the library is missing or fails to load, importing
this module raises.
"""
from __future__ import annotations

import ctypes
import os
from typing import Optional, Sequence

import torch

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "libtokengate.so")

TG_OK = 0
TG_ERR_INVALID_ARG = 1
TG_ERR_UNSUPPORTED = 2
TG_ERR_WORKSPACE = 3
TG_ERR_CUDA = 4
TG_ERR_TIMEOUT = 5
TG_ERR_DEVICE_INDEX = 6

_STATUS_NAMES = {0: "TG_OK", 1: "TG_ERR_INVALID_ARG", 2: "TG_ERR_UNSUPPORTED", 3: "TG_ERR_WORKSPACE",
                 4: "TG_ERR_CUDA", 5: "TG_ERR_TIMEOUT", 6: "TG_ERR_DEVICE_INDEX"}


class TokenGateError(RuntimeError):
    def __init__(self, code: int, where: str, msg: str):
        super().__init__(f"{where}: {_STATUS_NAMES.get(code, code)}: {msg}")
        self.code = code


def _load() -> ctypes.CDLL:
    if not os.path.exists(LIB_PATH):
        raise ImportError(f"libtokengate.so is not built ({LIB_PATH}); run "
                          "`python -m learned_token_pruning_09_b300.build`")
    return ctypes.CDLL(LIB_PATH)


lib = _load()

_vp, _i64, _i32, _f32, _sz, _ll = (ctypes.c_void_p, ctypes.c_int64, ctypes.c_int32, ctypes.c_float,
                                   ctypes.c_size_t, ctypes.c_longlong)
_SIGS = {
    "tg_gate_score": [_vp, _i64, _i32, _vp, _vp, _i32, _vp, _vp, _vp, _f32, _i32, _vp, _vp, _sz, _vp],
    "tg_topk_workspace_size": [_i32],
    "tg_topk_select": [_vp, _i64, _vp, _vp, _vp, _i32, _i32, _vp, _vp, _vp, _sz, _vp],
    "tg_gate_score_masked": [_vp, _i64, _i32, _vp, _vp, _vp, _vp, _f32, _i32, _vp, _vp, _i32, _vp, _sz, _vp],
    "tg_topk_select_masked": [_vp, _i64, _vp, _vp, _vp, _i32, _i32, _i64, _vp, _vp, _vp, _vp, _sz, _vp],
    "tg_gather_kept": [_vp, _i64, _i32, _vp, _vp, _vp, _vp, _i32, _i64, _vp, _vp, _vp, _vp],
    "tg_gated_attention_fwd": [_vp, _vp, _vp, _vp, _vp, _vp, _f32, _f32, _vp, _i32, _i64, _i32, _i32, _i32,
                               _i32, _vp, _vp, _vp, _vp, _sz, _vp],
    "tg_rope_qk": [_vp, _vp, _vp, _f32, _vp, _i32, _i64, _i32, _i32, _i32, _vp, _vp, _vp],
    "tg_gated_attention_rotated": [_vp, _vp, _vp, _vp, _vp, _vp, _f32, _vp, _i32, _i64, _i32, _i32, _i32, _i32,
                                   _vp, _vp, _vp],
    "tg_attention_workspace_size": [_i64, _i32, _i32, _i32, _i32],
    "tg_gated_attention_bwd": [_vp, _vp, _vp, _vp, _vp, _vp, _vp, _vp, _vp, _f32, _vp, _i32, _i64, _i32, _i32,
                               _i32, _i32, _vp, _vp, _vp, _vp, _sz, _vp],
    "tg_attention_bwd_workspace_size": [_i64, _i32],
    "tg_rms_norm": [_vp, _vp, _i64, _i32, _f32, _vp, _vp],
    "tg_swiglu": [_vp, _i64, _i32, _vp, _vp],
    "tg_decode_workspace_size": [_i32, _i32, _i32, _i32],
    "tg_decode_attention": [_vp, _vp, _vp, _vp, _vp, _vp, _i32, _i64, _i32, _vp, _vp, _f32, _i32, _i32, _i32, _vp,
                            _vp, _sz, _vp],
    "tg_gated_delta_scan": [_vp, _vp, _vp, _vp, _vp, _vp, _i32, _i64, _i32, _i32, _i32, _i32, _f32, _vp, _vp, _vp,
                            _vp, _sz, _vp],
    "tg_gated_delta_scan_workspace_size": [_i64, _i32, _i32, _i32, _i32],
    "tg_linear_bf16": [_vp, _vp, _vp, _vp, _i64, _i32, _i32, _vp],
    "tg_qkv_rope_bf16": [_vp, _vp, _i64, _i32, _i32, _i32, _i32, _vp, _f32, _vp, _vp, _vp, _vp],
    "tg_check_device_status": [_vp],
    "tg_set_watchdog_cycles": [_ll],
    "tg_last_error_string": [],
    "tg_version": [],
}
for _name, _args in _SIGS.items():
    _f = getattr(lib, _name)
    _f.argtypes = _args
    _f.restype = ctypes.c_int
lib.tg_attention_workspace_size.restype = ctypes.c_size_t
lib.tg_topk_workspace_size.restype = ctypes.c_size_t
lib.tg_attention_bwd_workspace_size.restype = ctypes.c_size_t
lib.tg_decode_workspace_size.restype = ctypes.c_size_t
lib.tg_gated_delta_scan_workspace_size.restype = ctypes.c_size_t
lib.tg_last_error_string.restype = ctypes.c_char_p
lib.tg_version.restype = ctypes.c_char_p
lib.tg_set_watchdog_cycles.restype = None


def _check(code: int, where: str) -> None:
    if code != TG_OK:
        raise TokenGateError(code, where, lib.tg_last_error_string().decode())


def _ptr(t: Optional[torch.Tensor]):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _stream(stream: Optional[torch.cuda.Stream]):
    s = stream if stream is not None else torch.cuda.current_stream()
    return ctypes.c_void_p(s.cuda_stream)


def _need(t: torch.Tensor, dtype: torch.dtype, name: str, ndim: Optional[int] = None) -> None:
    if not isinstance(t, torch.Tensor):
        raise TypeError(f"{name} must be a torch.Tensor")
    if t.dtype != dtype:
        raise TypeError(f"{name} must be {dtype}, got {t.dtype}")
    if not t.is_cuda:
        raise ValueError(f"{name} must be a CUDA tensor")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")
    if ndim is not None and t.dim() != ndim:
        raise ValueError(f"{name} must have {ndim} dims, got {t.dim()}")


def version() -> str:
    return lib.tg_version().decode()


def tg_set_watchdog_cycles(cycles: int) -> None:
    lib.tg_set_watchdog_cycles(int(cycles))


def tg_check_device_status(stream: Optional[torch.cuda.Stream] = None) -> int:
    """Synchronise the stream and return (and clear) the device status code."""
    return lib.tg_check_device_status(_stream(stream))


def tg_topk_workspace(batch: int, device="cuda") -> torch.Tensor:
    """A zero-filled top-K workspace for ``batch`` sequences (the gate's score
    histograms), to pass to both tg_gate_score and tg_topk_select."""
    n = int(lib.tg_topk_workspace_size(int(batch)))
    if n == 0:
        raise ValueError("batch must be in [1, 65535] for a top-K workspace")
    return torch.zeros(n, dtype=torch.uint8, device=device)


def tg_gate_score(x: torch.Tensor, cu_seqlens: torch.Tensor, n_doc: torch.Tensor, w1: torch.Tensor,
                  b1: Optional[torch.Tensor], w2: torch.Tensor, b2: float,
                  s_out: Optional[torch.Tensor] = None, topk_ws: Optional[torch.Tensor] = None,
                  stream=None) -> torch.Tensor:
    """Gate scores s [n_rows] fp32 (logsigmoid of the gate MLP logit for
    document rows, 0 for question rows); with ``topk_ws`` also the score
    histograms that tg_topk_select starts from."""
    _need(x, torch.bfloat16, "x", 2)
    _need(w1, torch.bfloat16, "w1", 2)
    _need(w2, torch.bfloat16, "w2", 1)
    _need(cu_seqlens, torch.int32, "cu_seqlens", 1)
    _need(n_doc, torch.int32, "n_doc", 1)
    if b1 is not None:
        _need(b1, torch.float32, "b1", 1)
    n_rows, d = x.shape
    h = w1.shape[0]
    if w1.shape[1] != d or w2.shape[0] != h:
        raise ValueError("w1 must be [h, d] and w2 [h]")
    if s_out is None:
        s_out = torch.empty(n_rows, dtype=torch.float32, device=x.device)
    _need(s_out, torch.float32, "s_out", 1)
    ws_bytes = 0 if topk_ws is None else topk_ws.numel() * topk_ws.element_size()
    _check(lib.tg_gate_score(_ptr(x), n_rows, d, _ptr(cu_seqlens), _ptr(n_doc), n_doc.shape[0], _ptr(w1),
                             _ptr(b1), _ptr(w2), float(b2), h, _ptr(s_out), _ptr(topk_ws), ws_bytes,
                             _stream(stream)), "tg_gate_score")
    return s_out


def kept_lengths(seqlens: Sequence[int], n_doc: Sequence[int], k: Sequence[int]):
    """Host-side kept length per sequence: min(k, n_doc) + question length."""
    return [min(int(kb), int(nd)) + int(sl) - int(nd) for sl, nd, kb in zip(seqlens, n_doc, k)]


def tg_topk_select(s: torch.Tensor, cu_seqlens: torch.Tensor, n_doc: torch.Tensor, k: torch.Tensor,
                   max_n_doc: int, n_kept: int, kept_idx: Optional[torch.Tensor] = None,
                   cu_kept: Optional[torch.Tensor] = None, workspace: Optional[torch.Tensor] = None, stream=None):
    """Kept row ids [n_kept] int32 and cu_kept [batch+1] int32.  ``n_kept``
    (host) sizes the output: sum over sequences of min(k, n_doc) + n_q.
    ``workspace``: the one given to the tg_gate_score call that produced s
    (see tg_topk_workspace), or None."""
    _need(s, torch.float32, "s", 1)
    for t, nme in ((cu_seqlens, "cu_seqlens"), (n_doc, "n_doc"), (k, "k")):
        _need(t, torch.int32, nme, 1)
    batch = n_doc.shape[0]
    if kept_idx is None:
        kept_idx = torch.empty(max(n_kept, 1), dtype=torch.int32, device=s.device)[:n_kept]
    if cu_kept is None:
        cu_kept = torch.empty(batch + 1, dtype=torch.int32, device=s.device)
    ws_bytes = 0 if workspace is None else workspace.numel() * workspace.element_size()
    _check(lib.tg_topk_select(_ptr(s), s.shape[0], _ptr(cu_seqlens), _ptr(n_doc), _ptr(k), batch,
                              int(max_n_doc), _ptr(kept_idx), _ptr(cu_kept), _ptr(workspace), ws_bytes,
                              _stream(stream)), "tg_topk_select")
    return kept_idx, cu_kept


def tg_gate_score_masked(x: torch.Tensor, prunable: torch.Tensor, w1: torch.Tensor, b1: Optional[torch.Tensor],
                         w2: torch.Tensor, b2: float, s_out: Optional[torch.Tensor] = None,
                         cu_seqlens: Optional[torch.Tensor] = None, topk_ws: Optional[torch.Tensor] = None,
                         stream=None) -> torch.Tensor:
    """Gate scores s [n_rows] fp32 on the rows of a per-row prunable mask
    (uint8 [n_rows], nonzero = prunable), 0 on every other row.  With
    ``topk_ws`` (and ``cu_seqlens``) the gate also counts the masked top-K's
    first two radix digits per sequence."""
    _need(x, torch.bfloat16, "x", 2)
    _need(prunable, torch.uint8, "prunable", 1)
    _need(w1, torch.bfloat16, "w1", 2)
    _need(w2, torch.bfloat16, "w2", 1)
    if b1 is not None:
        _need(b1, torch.float32, "b1", 1)
    n_rows, d = x.shape
    h = w1.shape[0]
    if w1.shape[1] != d or w2.shape[0] != h or prunable.shape[0] != n_rows:
        raise ValueError("w1 must be [h, d], w2 [h] and prunable [n_rows]")
    if s_out is None:
        s_out = torch.empty(n_rows, dtype=torch.float32, device=x.device)
    _need(s_out, torch.float32, "s_out", 1)
    batch = 0
    if topk_ws is not None:
        if cu_seqlens is None:
            raise ValueError("topk_ws needs cu_seqlens")
        _need(cu_seqlens, torch.int32, "cu_seqlens", 1)
        batch = cu_seqlens.shape[0] - 1
    _check(lib.tg_gate_score_masked(_ptr(x), n_rows, d, _ptr(prunable), _ptr(w1), _ptr(b1), _ptr(w2), float(b2), h,
                                    _ptr(s_out), _ptr(cu_seqlens if topk_ws is not None else None), batch,
                                    _ptr(topk_ws), topk_ws.numel() if topk_ws is not None else 0, _stream(stream)),
           "tg_gate_score_masked")
    return s_out


def tg_topk_select_masked(s: torch.Tensor, cu_seqlens: torch.Tensor, prunable: torch.Tensor, k: torch.Tensor,
                          max_len: int, kept_capacity: Optional[int] = None, kept_idx: Optional[torch.Tensor] = None,
                          cu_kept: Optional[torch.Tensor] = None, n_prunable: Optional[torch.Tensor] = None,
                          workspace: Optional[torch.Tensor] = None, stream=None):
    """(kept_idx, cu_kept, n_prunable) with general prunable spans.  kept_idx
    has ``kept_capacity`` entries (default n_rows); its first cu_kept[batch]
    entries are the kept rows.  ``workspace``: the top-K workspace a
    tg_gate_score_masked call filled (its first two digits come from there)."""
    _need(s, torch.float32, "s", 1)
    _need(prunable, torch.uint8, "prunable", 1)
    for t, nme in ((cu_seqlens, "cu_seqlens"), (k, "k")):
        _need(t, torch.int32, nme, 1)
    batch = k.shape[0]
    n_rows = s.shape[0]
    if prunable.shape[0] != n_rows:
        raise ValueError("prunable must be [n_rows]")
    if kept_idx is None:
        cap = n_rows if kept_capacity is None else int(kept_capacity)
        kept_idx = torch.empty(max(cap, 1), dtype=torch.int32, device=s.device)[:cap]
    if cu_kept is None:
        cu_kept = torch.empty(batch + 1, dtype=torch.int32, device=s.device)
    if n_prunable is None:
        n_prunable = torch.empty(batch, dtype=torch.int32, device=s.device)
    _check(lib.tg_topk_select_masked(_ptr(s), n_rows, _ptr(cu_seqlens), _ptr(prunable), _ptr(k), batch,
                                     int(max_len), kept_idx.shape[0], _ptr(kept_idx), _ptr(cu_kept),
                                     _ptr(n_prunable), _ptr(workspace), workspace.numel() if workspace is not None else 0,
                                     _stream(stream)), "tg_topk_select_masked")
    return kept_idx, cu_kept, n_prunable


def tg_gather_kept(x: Optional[torch.Tensor], s: Optional[torch.Tensor], cu_seqlens: torch.Tensor,
                   kept_idx: torch.Tensor, cu_kept: torch.Tensor, n_kept: int, d: Optional[int] = None,
                   x_kept: Optional[torch.Tensor] = None, pos_kept: Optional[torch.Tensor] = None,
                   s_kept: Optional[torch.Tensor] = None, want=("x", "pos", "s"), stream=None):
    """x_kept [n_kept, d] bf16, pos_kept [n_kept] int32, s_kept [n_kept] fp32."""
    _need(cu_seqlens, torch.int32, "cu_seqlens", 1)
    _need(cu_kept, torch.int32, "cu_kept", 1)
    _need(kept_idx, torch.int32, "kept_idx", 1)
    dev = kept_idx.device
    if x is not None:
        _need(x, torch.bfloat16, "x", 2)
        d = x.shape[1]
    n_rows = x.shape[0] if x is not None else (s.shape[0] if s is not None else 0)
    if "x" in want and x_kept is None and x is not None:
        x_kept = torch.empty((n_kept, d), dtype=torch.bfloat16, device=dev)
    if "pos" in want and pos_kept is None:
        pos_kept = torch.empty(n_kept, dtype=torch.int32, device=dev)
    if "s" in want and s_kept is None and s is not None:
        s_kept = torch.empty(n_kept, dtype=torch.float32, device=dev)
    _check(lib.tg_gather_kept(_ptr(x), n_rows, int(d or 8), _ptr(s), _ptr(cu_seqlens), _ptr(kept_idx),
                              _ptr(cu_kept), cu_kept.shape[0] - 1, int(n_kept), _ptr(x_kept), _ptr(pos_kept),
                              _ptr(s_kept), _stream(stream)), "tg_gather_kept")
    return x_kept, pos_kept, s_kept


def tg_attention_workspace_size(n_kept: int, hq: int, hkv: int, head_dim: int, has_k_cache: bool) -> int:
    return int(lib.tg_attention_workspace_size(int(n_kept), hq, hkv, head_dim, 1 if has_k_cache else 0))


def tg_rope_qk(q: torch.Tensor, k: torch.Tensor, pos_kept: torch.Tensor, rope_theta: float, cu_kept: torch.Tensor,
               q_out: Optional[torch.Tensor] = None, k_out: Optional[torch.Tensor] = None, stream=None):
    """(q', k'): q [T, hq, D] and k [T, hkv, D] bf16 rotated by RoPE at pos_kept."""
    _need(q, torch.bfloat16, "q", 3)
    _need(k, torch.bfloat16, "k", 3)
    _need(pos_kept, torch.int32, "pos_kept", 1)
    _need(cu_kept, torch.int32, "cu_kept", 1)
    t, hq, dh = q.shape
    hkv = k.shape[1]
    if k.shape != (t, hkv, dh):
        raise ValueError("k must be [T, hkv, D] matching q")
    q_out = torch.empty_like(q) if q_out is None else q_out
    k_out = torch.empty_like(k) if k_out is None else k_out
    _need(q_out, torch.bfloat16, "q_out", 3)
    _need(k_out, torch.bfloat16, "k_out", 3)
    _check(lib.tg_rope_qk(_ptr(q), _ptr(k), _ptr(pos_kept), float(rope_theta), _ptr(cu_kept), cu_kept.shape[0] - 1,
                          t, hq, hkv, dh, _ptr(q_out), _ptr(k_out), _stream(stream)), "tg_rope_qk")
    return q_out, k_out


def tg_gated_attention_rotated(q_rot: torch.Tensor, k_rot: torch.Tensor, v: torch.Tensor, pos_kept: torch.Tensor,
                               s_kept: torch.Tensor, gain: torch.Tensor, tau: float, cu_kept: torch.Tensor,
                               max_kept: int, o: Optional[torch.Tensor] = None, lse: Optional[torch.Tensor] = None,
                               want_lse: bool = False, stream=None):
    """o [T, hq, D] bf16 (and lse [hq, T] fp32) from q', k' already rotated by tg_rope_qk."""
    _need(q_rot, torch.bfloat16, "q_rot", 3)
    _need(k_rot, torch.bfloat16, "k_rot", 3)
    _need(v, torch.bfloat16, "v", 3)
    _need(pos_kept, torch.int32, "pos_kept", 1)
    _need(s_kept, torch.float32, "s_kept", 1)
    _need(gain, torch.float32, "gain", 1)
    _need(cu_kept, torch.int32, "cu_kept", 1)
    t, hq, dh = q_rot.shape
    hkv = k_rot.shape[1]
    if k_rot.shape != (t, hkv, dh) or v.shape != (t, hkv, dh):
        raise ValueError("k_rot and v must be [T, hkv, D] matching q_rot")
    if o is None:
        o = torch.empty_like(q_rot)
    if lse is None and want_lse:
        lse = torch.empty((hq, t), dtype=torch.float32, device=q_rot.device)
    _check(lib.tg_gated_attention_rotated(_ptr(q_rot), _ptr(k_rot), _ptr(v), _ptr(pos_kept), _ptr(s_kept),
                                          _ptr(gain), float(tau), _ptr(cu_kept), cu_kept.shape[0] - 1, t,
                                          int(max_kept), hq, hkv, dh, _ptr(o), _ptr(lse), _stream(stream)),
           "tg_gated_attention_rotated")
    return (o, lse) if lse is not None else o


def tg_gated_attention_bwd(q_rot: torch.Tensor, k_rot: torch.Tensor, v: torch.Tensor, o: torch.Tensor,
                           lse: torch.Tensor, d_o: torch.Tensor, pos_kept: torch.Tensor, s_kept: torch.Tensor,
                           gain: torch.Tensor, tau: float, cu_kept: torch.Tensor, max_kept: int,
                           d_s: Optional[torch.Tensor] = None, d_gain: Optional[torch.Tensor] = None,
                           d_tau: Optional[torch.Tensor] = None, workspace: Optional[torch.Tensor] = None,
                           stream=None):
    """(d_s [T], d_gain [hq], d_tau [1]) fp32: gradients of sum(d_o * o) with
    respect to the kept scores, the gains and the temperature, from the
    forward's q', k', v, o and lse."""
    _need(q_rot, torch.bfloat16, "q_rot", 3)
    _need(k_rot, torch.bfloat16, "k_rot", 3)
    _need(v, torch.bfloat16, "v", 3)
    _need(o, torch.bfloat16, "o", 3)
    _need(d_o, torch.bfloat16, "d_o", 3)
    _need(lse, torch.float32, "lse", 2)
    _need(pos_kept, torch.int32, "pos_kept", 1)
    _need(s_kept, torch.float32, "s_kept", 1)
    _need(gain, torch.float32, "gain", 1)
    _need(cu_kept, torch.int32, "cu_kept", 1)
    t, hq, dh = q_rot.shape
    hkv = k_rot.shape[1]
    if k_rot.shape != (t, hkv, dh) or v.shape != (t, hkv, dh):
        raise ValueError("k_rot and v must be [T, hkv, D] matching q_rot")
    if o.shape != q_rot.shape or d_o.shape != q_rot.shape or lse.shape != (hq, t):
        raise ValueError("o and d_o must be [T, hq, D] and lse [hq, T]")
    dev = q_rot.device
    if d_s is None:
        d_s = torch.empty(t, dtype=torch.float32, device=dev)
    if d_gain is None:
        d_gain = torch.empty(hq, dtype=torch.float32, device=dev)
    if d_tau is None:
        d_tau = torch.empty(1, dtype=torch.float32, device=dev)
    need = lib.tg_attention_bwd_workspace_size(t, hq)
    if workspace is None:
        workspace = torch.empty(max(need, 1), dtype=torch.uint8, device=dev)
    _check(lib.tg_gated_attention_bwd(_ptr(q_rot), _ptr(k_rot), _ptr(v), _ptr(o), _ptr(lse), _ptr(d_o),
                                      _ptr(pos_kept), _ptr(s_kept), _ptr(gain), float(tau), _ptr(cu_kept),
                                      cu_kept.shape[0] - 1, t, int(max_kept), hq, hkv, dh, _ptr(d_s), _ptr(d_gain),
                                      _ptr(d_tau), _ptr(workspace), workspace.numel(), _stream(stream)),
           "tg_gated_attention_bwd")
    return d_s, d_gain, d_tau


def tg_gated_attention_fwd(q: torch.Tensor, k: torch.Tensor, v: torch.Tensor, pos_kept: torch.Tensor,
                           s_kept: torch.Tensor, gain: torch.Tensor, tau: float, rope_theta: float,
                           cu_kept: torch.Tensor, max_kept: int, o: Optional[torch.Tensor] = None,
                           lse: Optional[torch.Tensor] = None, want_lse: bool = False,
                           k_cache: Optional[torch.Tensor] = None, workspace: Optional[torch.Tensor] = None,
                           stream=None):
    """o [T, hq, D] bf16 (and lse [hq, T] fp32 when requested or given)."""
    _need(q, torch.bfloat16, "q", 3)
    _need(k, torch.bfloat16, "k", 3)
    _need(v, torch.bfloat16, "v", 3)
    _need(pos_kept, torch.int32, "pos_kept", 1)
    _need(s_kept, torch.float32, "s_kept", 1)
    _need(gain, torch.float32, "gain", 1)
    _need(cu_kept, torch.int32, "cu_kept", 1)
    t, hq, dh = q.shape
    hkv = k.shape[1]
    if k.shape != (t, hkv, dh) or v.shape != (t, hkv, dh):
        raise ValueError("k and v must be [T, hkv, D] matching q")
    if o is None:
        o = torch.empty_like(q)
    if lse is None and want_lse:
        lse = torch.empty((hq, t), dtype=torch.float32, device=q.device)
    if k_cache is not None:
        _need(k_cache, torch.bfloat16, "k_cache", 3)
    need = tg_attention_workspace_size(t, hq, hkv, dh, k_cache is not None)
    if workspace is None:
        workspace = torch.empty(max(need, 1), dtype=torch.uint8, device=q.device)
    _check(lib.tg_gated_attention_fwd(_ptr(q), _ptr(k), _ptr(v), _ptr(pos_kept), _ptr(s_kept), _ptr(gain),
                                      float(tau), float(rope_theta), _ptr(cu_kept), cu_kept.shape[0] - 1, t,
                                      int(max_kept), hq, hkv, dh, _ptr(o), _ptr(lse), _ptr(k_cache),
                                      _ptr(workspace), workspace.numel(), _stream(stream)),
           "tg_gated_attention_fwd")
    return (o, lse) if lse is not None else o


def tg_gated_delta_scan_workspace_size(n_kept: int, batch: int, hv: int, dk: int, dv: int) -> int:
    return int(lib.tg_gated_delta_scan_workspace_size(int(n_kept), int(batch), int(hv), int(dk), int(dv)))


def tg_gated_delta_scan(q: torch.Tensor, k: torch.Tensor, v: torch.Tensor, g: torch.Tensor, beta: torch.Tensor,
                        cu_kept: torch.Tensor, scale: Optional[float] = None,
                        initial_state: Optional[torch.Tensor] = None, o: Optional[torch.Tensor] = None,
                        final_state: Optional[torch.Tensor] = None, want_state: bool = False,
                        workspace: Optional[torch.Tensor] = None, chunked: bool = True, stream=None):
    """o [T, hv, dv] bf16 (and the final states [B, hv, dv, dk] fp32 when
    requested or given): the gated delta rule over the kept tokens.
    ``chunked``: the tensor-core chunked form, with ``workspace`` (allocated
    here when None) of tg_gated_delta_scan_workspace_size bytes; False, or a
    shape the chunked form does not take, runs the token-by-token kernel."""
    _need(q, torch.bfloat16, "q", 3)
    _need(k, torch.bfloat16, "k", 3)
    _need(v, torch.bfloat16, "v", 3)
    _need(g, torch.float32, "g", 2)
    _need(beta, torch.float32, "beta", 2)
    _need(cu_kept, torch.int32, "cu_kept", 1)
    t, hk, dk = q.shape
    hv, dv = v.shape[1], v.shape[2]
    batch = cu_kept.shape[0] - 1
    if k.shape != q.shape or v.shape[0] != t or g.shape != (t, hv) or beta.shape != (t, hv):
        raise ValueError("k must match q; v [T, hv, dv]; g and beta [T, hv]")
    if initial_state is not None:
        _need(initial_state, torch.float32, "initial_state", 4)
        if initial_state.shape != (batch, hv, dv, dk):
            raise ValueError("initial_state must be [B, hv, dv, dk]")
    if o is None:
        o = torch.empty((t, hv, dv), dtype=torch.bfloat16, device=q.device)
    if final_state is None and want_state:
        final_state = torch.empty((batch, hv, dv, dk), dtype=torch.float32, device=q.device)
    sc = (1.0 / dk ** 0.5) if scale is None else float(scale)
    ws_bytes = tg_gated_delta_scan_workspace_size(t, batch, hv, dk, dv) if chunked else 0
    if ws_bytes == 0:
        workspace = None
    elif workspace is None:
        workspace = torch.empty(ws_bytes, dtype=torch.uint8, device=q.device)
    _check(lib.tg_gated_delta_scan(_ptr(q), _ptr(k), _ptr(v), _ptr(g), _ptr(beta), _ptr(cu_kept), batch, t, hk, hv,
                                   dk, dv, sc, _ptr(initial_state), _ptr(o), _ptr(final_state), _ptr(workspace),
                                   workspace.numel() if workspace is not None else 0, _stream(stream)),
           "tg_gated_delta_scan")
    return (o, final_state) if final_state is not None else o


def tg_rms_norm(x: torch.Tensor, w: torch.Tensor, eps: float = 1e-6, y: Optional[torch.Tensor] = None,
                stream=None):
    """y = RMSNorm(x) * w over the last dimension (bf16); x of any shape
    whose last dimension is w's length."""
    _need(x, torch.bfloat16, "x")
    _need(w, torch.bfloat16, "w", 1)
    d = w.shape[0]
    if x.shape[-1] != d:
        raise ValueError("the last dimension of x must be len(w)")
    y = torch.empty_like(x) if y is None else y
    _need(y, torch.bfloat16, "y")
    _check(lib.tg_rms_norm(_ptr(x), _ptr(w), x.numel() // d, d, float(eps), _ptr(y), _stream(stream)), "tg_rms_norm")
    return y


def tg_swiglu(gate_up: torch.Tensor, y: Optional[torch.Tensor] = None, stream=None):
    """SiLU(gate_up[:, :f]) * gate_up[:, f:] (bf16 [rows, 2f] -> [rows, f])."""
    _need(gate_up, torch.bfloat16, "gate_up", 2)
    rows, f2 = gate_up.shape
    if f2 % 2:
        raise ValueError("gate_up must have an even number of columns")
    f = f2 // 2
    y = torch.empty((rows, f), dtype=torch.bfloat16, device=gate_up.device) if y is None else y
    _need(y, torch.bfloat16, "y", 2)
    _check(lib.tg_swiglu(_ptr(gate_up), rows, f, _ptr(y), _stream(stream)), "tg_swiglu")
    return y


def tg_decode_attention(q_rot: torch.Tensor, k_new_rot: torch.Tensor, v_new: torch.Tensor, k_cache: torch.Tensor,
                        v_cache: torch.Tensor, cache_cu: torch.Tensor, max_cache_len: int,
                        s_cache: Optional[torch.Tensor] = None, gain: Optional[torch.Tensor] = None,
                        tau: float = 1.0, o: Optional[torch.Tensor] = None,
                        workspace: Optional[torch.Tensor] = None, stream=None):
    """o [B, hq, D] bf16: each sequence's new query over its cache rows and
    its own key (score bias when s_cache and gain are given)."""
    for t_, n_ in ((q_rot, "q_rot"), (k_new_rot, "k_new_rot"), (v_new, "v_new"), (k_cache, "k_cache"),
                   (v_cache, "v_cache")):
        _need(t_, torch.bfloat16, n_, 3)
    _need(cache_cu, torch.int32, "cache_cu", 1)
    if s_cache is not None:
        _need(s_cache, torch.float32, "s_cache", 1)
    if gain is not None:
        _need(gain, torch.float32, "gain", 1)
    b, hq, dh = q_rot.shape
    hkv = k_new_rot.shape[1]
    o = torch.empty_like(q_rot) if o is None else o
    need = lib.tg_decode_workspace_size(b, hq, dh, int(max_cache_len))
    if workspace is None:
        workspace = torch.empty(max(need, 16), dtype=torch.uint8, device=q_rot.device)
    _check(lib.tg_decode_attention(_ptr(q_rot), _ptr(k_new_rot), _ptr(v_new), _ptr(k_cache), _ptr(v_cache),
                                   _ptr(cache_cu), b, k_cache.shape[0], int(max_cache_len), _ptr(s_cache), _ptr(gain),
                                   float(tau), hq, hkv, dh, _ptr(o), _ptr(workspace), workspace.numel(),
                                   _stream(stream)), "tg_decode_attention")
    return o


def tg_linear_bf16(a: torch.Tensor, w: torch.Tensor, residual: Optional[torch.Tensor] = None,
                   out: Optional[torch.Tensor] = None, stream=None) -> torch.Tensor:
    """out = a w^T (+ residual), bf16 [m, n]."""
    _need(a, torch.bfloat16, "a", 2)
    _need(w, torch.bfloat16, "w", 2)
    m, kd = a.shape
    n = w.shape[0]
    if w.shape[1] != kd:
        raise ValueError("w must be [n, k]")
    if residual is not None:
        _need(residual, torch.bfloat16, "residual", 2)
    if out is None:
        out = torch.empty((m, n), dtype=torch.bfloat16, device=a.device)
    _check(lib.tg_linear_bf16(_ptr(a), _ptr(w), _ptr(residual), _ptr(out), m, n, kd, _stream(stream)),
           "tg_linear_bf16")
    return out


def tg_qkv_rope_bf16(x: torch.Tensor, w_qkv: torch.Tensor, pos: torch.Tensor, hq: int, hkv: int, head_dim: int,
                     rope_theta: float = 1.0e6, q_out: Optional[torch.Tensor] = None,
                     k_out: Optional[torch.Tensor] = None, v_out: Optional[torch.Tensor] = None, stream=None):
    """(q', k', v): x w_qkv^T split into q [m, hq, D], k and v [m, hkv, D],
    q and k rotated by RoPE at pos (bf16)."""
    _need(x, torch.bfloat16, "x", 2)
    _need(w_qkv, torch.bfloat16, "w_qkv", 2)
    _need(pos, torch.int32, "pos", 1)
    m, kd = x.shape
    if w_qkv.shape != ((hq + 2 * hkv) * head_dim, kd):
        raise ValueError("w_qkv must be [(hq + 2 hkv) head_dim, k]")
    if pos.shape[0] != m:
        raise ValueError("pos must have one entry per row")
    e = lambda h: torch.empty((m, h, head_dim), dtype=torch.bfloat16, device=x.device)
    q_out = e(hq) if q_out is None else q_out
    k_out = e(hkv) if k_out is None else k_out
    v_out = e(hkv) if v_out is None else v_out
    for t, nm, h in ((q_out, "q_out", hq), (k_out, "k_out", hkv), (v_out, "v_out", hkv)):
        _need(t, torch.bfloat16, nm, 3)
        if tuple(t.shape) != (m, h, head_dim):
            raise ValueError(f"{nm} must be [m, {h}, {head_dim}]")
    _check(lib.tg_qkv_rope_bf16(_ptr(x), _ptr(w_qkv), m, kd, hq, hkv, head_dim, _ptr(pos), float(rope_theta),
                                _ptr(q_out), _ptr(k_out), _ptr(v_out), _stream(stream)), "tg_qkv_rope_bf16")
    return q_out, k_out, v_out
