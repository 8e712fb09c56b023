"""CPU oracle for the verify-and-accept hot path (float64, plain C via ctypes).

TEST INFRASTRUCTURE ONLY.  Only ``tests/``, ``__graft_entry__.smoke()`` and the
``cpu_baseline`` / ``--impl reference`` legs of ``bench.py`` may import this
package.  The CUDA product path never imports it and shares no code with it.

The arithmetic lives in ``oracle.c`` (one function per step of the path, each
citing the page passage it follows); this module only builds that file with
gcc, loads it and marshals numpy arrays.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
from pathlib import Path

import numpy as np

_HERE = Path(__file__).resolve().parent
_SRC = _HERE / "oracle.c"
_LIB = _HERE / "liboracle.so"

# error-flag bits (same meaning as the product's, defined independently)
FLAG_DRAFT_OUT_OF_RANGE = 1
FLAG_DRAFT_ZERO_Q = 2
FLAG_NONFINITE_LOGIT = 4
FLAG_EMPTY_DIST = 8


def build(force: bool = False) -> Path:
    """Compile oracle.c into liboracle.so with gcc (OpenMP when available)."""
    if _LIB.exists() and not force and _LIB.stat().st_mtime >= _SRC.stat().st_mtime:
        return _LIB
    base = ["gcc", "-O2", "-std=c11", "-ffp-contract=off", "-fno-fast-math", "-fPIC",
            "-shared", str(_SRC), "-o", str(_LIB) + ".tmp", "-lm"]
    try:
        subprocess.run(base[:1] + ["-fopenmp"] + base[1:], check=True, capture_output=True)
    except subprocess.CalledProcessError:
        subprocess.run(base, check=True, capture_output=True)
    os.replace(str(_LIB) + ".tmp", _LIB)
    return _LIB


_lib = None


def lib() -> ctypes.CDLL:
    global _lib
    if _lib is None:
        build()
        L = ctypes.CDLL(str(_LIB))
        P = ctypes.c_void_p
        I = ctypes.c_int
        D = ctypes.c_double
        L.oracle_qmv.argtypes = [P, P, P, P, I, P, I, I, I, I]
        L.oracle_qmv.restype = I
        L.oracle_requantize.argtypes = [P, I, I, P, P, P]
        L.oracle_requantize.restype = I
        L.oracle_filter_row.argtypes = [P, I, D, I, D, P, P, P]
        L.oracle_filter_row.restype = I
        L.oracle_spec_accept.argtypes = [P, P, P, P, P, I, I, I, D, I, D, P, P, P, P]
        L.oracle_spec_accept.restype = I
        L.oracle_gdn_sequential.argtypes = [P, P, P, P, P, P, P, I, I, I, I, I, P]
        L.oracle_gdn_sequential.restype = None
        L.oracle_gdn_capture.argtypes = [P, P, P, P, P, P, I, I, I, I, I, P, P, P, P]
        L.oracle_gdn_capture.restype = None
        L.oracle_gdn_replay.argtypes = [P, P, P, P, P, I, I, I, I, I]
        L.oracle_gdn_replay.restype = None
        L.oracle_conv_capture.argtypes = [P, P, P, I, I, I, I, P]
        L.oracle_conv_capture.restype = None
        L.oracle_conv_replay.argtypes = [P, P, P, I, I, I, I]
        L.oracle_conv_replay.restype = None
        L.oracle_set_threads.argtypes = [I]
        L.oracle_has_openmp.restype = I
        _lib = L
    return _lib


def _ptr(a: np.ndarray | None):
    return None if a is None else a.ctypes.data_as(ctypes.c_void_p)


def _c(a, dtype):
    return np.ascontiguousarray(a, dtype=dtype)


def set_threads(n: int) -> int:
    """Threads the oracle's outer loops may use (1 = single-threaded)."""
    lib().oracle_set_threads(int(n))
    return int(n) if lib().oracle_has_openmp() else 1


# ----------------------------------------------------------------------------
# qmv
# ----------------------------------------------------------------------------
def qmv(w_packed, scales, biases, x, group_size: int = 64) -> np.ndarray:
    """y[M,N] (fp32) = x[M,K] . W^T; W from LSB-first 4-bit nibbles, bf16 s/b.

    ``scales``/``biases`` are bf16 bit patterns (uint16); ``x`` is float32 or
    bf16 bit patterns (uint16 array => bf16).
    """
    w = _c(w_packed, np.uint32)
    s = _c(scales, np.uint16)
    b = _c(biases, np.uint16)
    is_bf16 = np.asarray(x).dtype == np.uint16
    xx = _c(x, np.uint16 if is_bf16 else np.float32)
    M, K = xx.shape
    N = w.shape[0]
    assert w.shape == (N, K // 8) and s.shape == (N, K // group_size) == b.shape
    y = np.empty((M, N), np.float32)
    rc = lib().oracle_qmv(_ptr(w), _ptr(s), _ptr(b), _ptr(xx), int(is_bf16), _ptr(y),
                          M, N, K, group_size)
    if rc:
        raise ValueError("oracle_qmv rejected the shapes")
    return y


def requantize(w_bf16, group_size: int = 64):
    """4-bit affine group-64 requantisation of a bf16 matrix [N, K] (uint16 bit
    patterns): returns (w_packed uint32 [N, K/8], scales, biases uint16 bf16
    bits [N, K/64]) -- the qmv weight layout, min/max affine per group."""
    assert group_size == 64
    w = _c(w_bf16, np.uint16)
    N, K = w.shape
    wp = np.empty((N, K // 8), np.uint32)
    s = np.empty((N, K // 64), np.uint16)
    b = np.empty((N, K // 64), np.uint16)
    if lib().oracle_requantize(_ptr(w), N, K, _ptr(wp), _ptr(s), _ptr(b)):
        raise ValueError("oracle_requantize rejected the shapes")
    return wp, s, b


# ----------------------------------------------------------------------------
# sampling distribution and verify-and-accept
# ----------------------------------------------------------------------------
def filter_row(z, temperature: float, top_k: int, top_p: float):
    """Filtered distribution (float64 [V]) of one logits row; returns (p, flags, topp_margin)."""
    zz = _c(z, np.float32)
    V = zz.shape[0]
    p = np.empty(V, np.float64)
    flags = ctypes.c_int(0)
    margin = ctypes.c_double(0.0)
    lib().oracle_filter_row(_ptr(zz), V, float(temperature), int(top_k), float(top_p), _ptr(p),
                            ctypes.byref(flags), ctypes.byref(margin))
    return p, flags.value, margin.value


def spec_accept(target_logits, draft_logits, draft_tokens, u_accept, u_sample,
                temperature: float, top_k: int, top_p: float):
    """Returns dict(out_tokens [B,K+1], n_accepted [B], err_flags [B], diag [B,3])."""
    tl = _c(target_logits, np.float32)
    B, K1, V = tl.shape
    K = K1 - 1
    dl = _c(draft_logits, np.float32) if draft_logits is not None else np.zeros((B, K, V), np.float32)
    dt = _c(draft_tokens, np.int32)
    ua = _c(u_accept, np.float32)
    us = _c(u_sample, np.float32)
    assert dl.shape == (B, K, V) and dt.shape == (B, K) and ua.shape == (B, K) and us.shape == (B,)
    out = np.empty((B, K + 1), np.int32)
    nacc = np.empty(B, np.int32)
    flags = np.empty(B, np.int32)
    diag = np.empty((B, 3), np.float64)
    rc = lib().oracle_spec_accept(_ptr(tl), _ptr(dl), _ptr(dt), _ptr(ua), _ptr(us), B, K, V,
                                  float(temperature), int(top_k), float(top_p), _ptr(out),
                                  _ptr(nacc), _ptr(flags), _ptr(diag))
    if rc:
        raise ValueError("oracle_spec_accept rejected the arguments")
    return {"out_tokens": out, "n_accepted": nacc, "err_flags": flags, "diag": diag}


# ----------------------------------------------------------------------------
# GatedDeltaNet recurrence and innovation tape
# ----------------------------------------------------------------------------
def gdn_sequential(state, q, k, v, alpha, beta, n_steps=None, want_out: bool = False):
    """Runs n_steps[b] steps of the recurrence from ``state``; returns (state f64, out f64|None)."""
    S = np.array(state, dtype=np.float64, order="C", copy=True)
    B, H, dv, dk = S.shape
    qq, kk, vv = _c(q, np.float32), _c(k, np.float32), _c(v, np.float32)
    T = qq.shape[1]
    aa, bb = _c(alpha, np.float32), _c(beta, np.float32)
    ns = None if n_steps is None else _c(n_steps, np.int32)
    out = np.zeros((B, T, H, dv), np.float64) if want_out else None
    lib().oracle_gdn_sequential(_ptr(S), _ptr(qq), _ptr(kk), _ptr(vv), _ptr(aa), _ptr(bb),
                                _ptr(ns), B, T, H, dk, dv, _ptr(out))
    return S, out


def gdn_capture(state0, q, k, v, alpha, beta):
    """Returns (out [B,T,H,dv] f64, tape dict alpha/e/k in float64)."""
    S0 = _c(state0, np.float32)
    B, H, dv, dk = S0.shape
    qq, kk, vv = _c(q, np.float32), _c(k, np.float32), _c(v, np.float32)
    T = qq.shape[1]
    aa, bb = _c(alpha, np.float32), _c(beta, np.float32)
    out = np.empty((B, T, H, dv), np.float64)
    ta = np.empty((B, T, H), np.float64)
    te = np.empty((B, T, H, dv), np.float64)
    tk = np.empty((B, T, H, dk), np.float64)
    lib().oracle_gdn_capture(_ptr(S0), _ptr(qq), _ptr(kk), _ptr(vv), _ptr(aa), _ptr(bb),
                             B, T, H, dk, dv, _ptr(out), _ptr(ta), _ptr(te), _ptr(tk))
    return out, {"alpha": ta, "e": te, "k": tk}


def gdn_replay(state, tape, n_replay):
    """Applies the first n_replay[b] records of ``tape`` to a float64 copy of ``state``."""
    S = np.array(state, dtype=np.float64, order="C", copy=True)
    B, H, dv, dk = S.shape
    ta, te, tk = (_c(tape[n], np.float64) for n in ("alpha", "e", "k"))
    T = ta.shape[1]
    nr = _c(n_replay, np.int32)
    assert nr.shape == (B,) and (nr >= 0).all() and (nr <= T).all()
    lib().oracle_gdn_replay(_ptr(S), _ptr(ta), _ptr(te), _ptr(tk), _ptr(nr), B, T, H, dk, dv)
    return S


def conv_capture(window, x, weight):
    """Causal depthwise convolution outputs y [B, T, C] (float64) of the T
    verify inputs x [B, T, C] from the committed window [B, W-1, C], with
    weight [W, C]."""
    win = _c(window, np.float64)
    xx = _c(x, np.float64)
    w = _c(weight, np.float64)
    B, T, C = xx.shape
    W = w.shape[0]
    assert win.shape == (B, W - 1, C) and w.shape == (W, C)
    y = np.zeros((B, T, C), np.float64)
    lib().oracle_conv_capture(_ptr(win), _ptr(xx), _ptr(w), B, T, C, W, _ptr(y))
    return y


def conv_replay(window, x, n_replay):
    """The committed window [B, W-1, C] (float64 copy) after the first
    n_replay[b] verify inputs of x [B, T, C]."""
    win = np.array(window, dtype=np.float64, order="C", copy=True)
    xx = _c(x, np.float64)
    B, T, C = xx.shape
    W = win.shape[1] + 1
    nr = _c(n_replay, np.int32)
    assert nr.shape == (B,) and (nr >= 0).all() and (nr <= T).all()
    lib().oracle_conv_replay(_ptr(win), _ptr(xx), _ptr(nr), B, T, C, W)
    return win
