"""Small conversions shared by the tests (no method arithmetic)."""
import numpy as np
import torch


def dev_bf16(bits: np.ndarray, device="cuda") -> torch.Tensor:
    return torch.from_numpy(np.ascontiguousarray(bits).view(np.int16)).to(device).view(torch.bfloat16)


def dev_i32(a, device="cuda") -> torch.Tensor:
    return torch.as_tensor(np.asarray(a, dtype=np.int32)).to(device)


def dev_f32(a, device="cuda") -> torch.Tensor:
    return torch.as_tensor(np.asarray(a, dtype=np.float32)).to(device)


def host_bits(t: torch.Tensor) -> np.ndarray:
    return t.contiguous().view(torch.int16).cpu().numpy().view(np.uint16)


def host_f64(t: torch.Tensor) -> np.ndarray:
    if t.dtype == torch.bfloat16:
        b = host_bits(t).astype(np.uint32) << np.uint32(16)
        return b.view(np.float32).astype(np.float64)
    return t.double().cpu().numpy()


def allclose_report(got, ref, atol, rtol):
    """Elementwise |got - ref| <= atol + rtol |ref| over finite reference
    entries; returns (ok, max_abs_err, worst_excess)."""
    got = np.asarray(got, np.float64)
    ref = np.asarray(ref, np.float64)
    m = np.isfinite(ref)
    err = np.abs(got[m] - ref[m])
    lim = atol + rtol * np.abs(ref[m])
    ok = bool(np.all(err <= lim)) and bool(np.all(np.isfinite(got[m])))
    return ok, float(err.max(initial=0.0)), float((err - lim).max(initial=-np.inf))
