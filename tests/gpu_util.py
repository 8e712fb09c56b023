"""Helpers shared by the GPU parity tests: device transfer and tolerances."""
import numpy as np
import torch

import workloads as wl


def sv_module():
    from mtp_speculative_decoding_qmv_gb300 import build as b

    b.build()
    import mtp_speculative_decoding_qmv_gb300 as sv

    return sv


def dev():
    return torch.device("cuda:0")


def qmv_to_device(w, s, b, x):
    d = dev()
    wt = torch.from_numpy(np.ascontiguousarray(w).view(np.int32)).to(d)
    st = torch.from_numpy(np.ascontiguousarray(s).view(np.int16)).to(d).view(torch.bfloat16)
    bt = torch.from_numpy(np.ascontiguousarray(b).view(np.int16)).to(d).view(torch.bfloat16)
    if x.dtype == np.uint16:
        xt = torch.from_numpy(np.ascontiguousarray(x).view(np.int16)).to(d).view(torch.bfloat16)
    else:
        xt = torch.from_numpy(np.ascontiguousarray(x, dtype=np.float32)).to(d)
    return wt, st, bt, xt


def assert_qmv_close(y_gpu: np.ndarray, y_ref: np.ndarray, rtol: float = 2e-3):
    """Per element |y - ref| <= rtol * max(|ref|, rms of ref's row): the
    relative-error tolerance with a row-RMS floor for outputs near zero."""
    ref = y_ref.astype(np.float64)
    rms = np.sqrt((ref ** 2).mean(axis=1, keepdims=True))
    bound = rtol * np.maximum(np.abs(ref), rms)
    err = np.abs(y_gpu.astype(np.float64) - ref)
    bad = err > bound
    if bad.any():
        i = np.unravel_index(np.argmax(err / np.maximum(bound, 1e-300)), err.shape)
        raise AssertionError(f"{bad.sum()} of {bad.size} outside tolerance; worst at {i}: "
                             f"gpu {y_gpu[i]!r} ref {y_ref[i]!r} bound {bound[i]:.3g}")
    return float((err / np.maximum(np.abs(ref), rms)).max())


def f32(v: float) -> float:
    """The value a C float parameter carries."""
    return float(np.float32(v))


__all__ = ["sv_module", "dev", "qmv_to_device", "assert_qmv_close", "f32", "wl"]
