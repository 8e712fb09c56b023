"""GB300 (sm_103a) verify-and-accept hot path of MTP speculative decoding.

A thin binding over libspecverify's C ABI (``include/specverify.h``): each
function here has the C entry point's name, checks and marshals torch
tensors (device, dtype, shape, contiguity) and calls the C function on the
current CUDA stream.  All arithmetic runs in the library's CUDA kernels; if
the library is missing, every call raises -- there is no fallback.

  qmv_smallm        4-bit affine group-64 mat-vec over M = 1..16 verify rows
  spec_accept       fp32 probability-ratio acceptance, residual, bonus token
  gdn_tape_capture  GatedDeltaNet recurrence + innovation tape
  gdn_tape_replay   rebuild the recurrent state over an accepted prefix
"""
from __future__ import annotations

import ctypes
from pathlib import Path

import torch

__all__ = [
    "SvError", "lib", "abi_version", "qmv_smallm", "spec_accept", "spec_accept_workspace_bytes",
    "make_accept_workspace", "gdn_tape_bytes", "gdn_tape_capture", "gdn_tape_replay",
    "set_pdl", "get_pdl", "device_status", "FLAGS", "QmvPlan", "spec_accept_noalloc",
    "spec_accept_noalloc_scratch_bytes", "conv_window_capture", "conv_window_replay",
]

_LIB_PATH = Path(__file__).resolve().parent / "libspecverify.so"

SV_OK, SV_ERR_INVALID_ARG, SV_ERR_UNSUPPORTED, SV_ERR_CUDA, SV_ERR_DEVICE_FLAG = range(5)
SV_F32, SV_BF16 = 0, 1
FLAGS = {"draft_out_of_range": 1, "draft_zero_q": 2, "nonfinite_logit": 4, "empty_dist": 8,
         "replay_range": 16}


class SvError(RuntimeError):
    def __init__(self, status: int, where: str, message: str):
        super().__init__(f"{where}: {message} (status {status})")
        self.status = status


class _Sampling(ctypes.Structure):
    _fields_ = [("temperature", ctypes.c_float), ("top_k", ctypes.c_int),
                ("top_p", ctypes.c_float)]


class _QmvProblem(ctypes.Structure):
    _fields_ = [("w_packed", ctypes.c_void_p), ("scales", ctypes.c_void_p),
                ("biases", ctypes.c_void_p), ("x", ctypes.c_void_p), ("y", ctypes.c_void_p),
                ("N", ctypes.c_int), ("K", ctypes.c_int), ("after", ctypes.c_int),
                ("topk", ctypes.c_void_p)]


_lib = None


def lib() -> ctypes.CDLL:
    """The loaded libspecverify; raises if it has not been built."""
    global _lib
    if _lib is None:
        if not _LIB_PATH.exists():
            raise RuntimeError(
                f"{_LIB_PATH.name} is not built; run `python -m "
                "mtp_speculative_decoding_qmv_gb300.build` (or __graft_entry__.build())")
        L = ctypes.CDLL(str(_LIB_PATH))
        P, I, Z = ctypes.c_void_p, ctypes.c_int, ctypes.c_size_t
        L.sv_abi_version.restype = I
        L.sv_status_string.restype = ctypes.c_char_p
        L.sv_status_string.argtypes = [I]
        L.sv_last_error.restype = ctypes.c_char_p
        L.sv_set_pdl.argtypes = [I]
        L.sv_get_pdl.restype = I
        L.sv_device_status.restype = I
        L.qmv_smallm.argtypes = [P, P, P, P, I, P, I, I, I, I, I, P]
        L.qmv_smallm.restype = I
        L.spec_accept_workspace_bytes.argtypes = [I, I, I]
        L.spec_accept_workspace_bytes.restype = Z
        L.spec_accept.argtypes = [P, P, P, P, P, I, I, I, _Sampling, P, P, P, P, Z, P]
        L.spec_accept.restype = I
        L.spec_accept_lists_workspace_bytes.argtypes = [I, I, I, I]
        L.spec_accept_lists_workspace_bytes.restype = Z
        L.spec_accept_lists_block_bytes.argtypes = [I, I]
        L.spec_accept_lists_block_bytes.restype = Z
        L.spec_accept_lists.argtypes = [P, I, P, P, P, P, I, I, I, _Sampling, P, P, P, P, Z, P]
        L.spec_accept_lists.restype = I
        L.spec_accept_noalloc_scratch_bytes.argtypes = []
        L.spec_accept_noalloc_scratch_bytes.restype = Z
        L.spec_accept_noalloc.argtypes = [P, P, P, P, P, I, I, I, _Sampling, P, P, P, P]
        L.spec_accept_noalloc.restype = I
        L.qmv_plan_device_bytes.argtypes = [ctypes.POINTER(_QmvProblem), I, I, I]
        L.qmv_plan_device_bytes.restype = Z
        L.qmv_plan_create.argtypes = [ctypes.POINTER(_QmvProblem), I, I, I, P, Z,
                                      ctypes.POINTER(P)]
        L.qmv_plan_create.restype = I
        L.qmv_plan_run.argtypes = [P, P]
        L.qmv_plan_run.restype = I
        L.qmv_plan_run_cooperative.argtypes = [P, P]
        L.qmv_plan_run_cooperative.restype = I
        L.qmv_plan_destroy.argtypes = [P]
        L.qmv_plan_destroy.restype = None
        L.qmv_plan_topk_bytes.argtypes = [I, I]
        L.qmv_plan_topk_bytes.restype = Z
        L.qmv_plan_grid.argtypes = [P]
        L.qmv_plan_grid.restype = I
        L.qmv_identity_probe_bytes.argtypes = [I, I, I, I]
        L.qmv_identity_probe_bytes.restype = Z
        L.qmv_identity_probe.argtypes = [P, P, P, I, I, I, I, P, Z, ctypes.POINTER(I), P]
        L.qmv_identity_probe.restype = I
        L.qmv_requantize.argtypes = [P, P, P, P, I, I, P]
        L.qmv_requantize.restype = I
        L.qmv_wide_workspace_bytes.argtypes = [I, I]
        L.qmv_wide_workspace_bytes.restype = Z
        L.qmv_wide.argtypes = [P, P, P, P, P, I, I, I, P, Z, P]
        L.qmv_wide.restype = I
        L.conv_window_capture.argtypes = [P, P, P, I, I, I, I, P, P]
        L.conv_window_capture.restype = I
        L.conv_window_replay.argtypes = [P, P, P, I, I, I, I, I, I, P, P]
        L.conv_window_replay.restype = I
        L.gdn_tape_bytes.argtypes = [I, I, I, I, I]
        L.gdn_tape_bytes.restype = Z
        L.gdn_tape_capture.argtypes = [P, P, P, P, P, P, I, I, I, I, I, P, P, P, P]
        L.gdn_tape_capture.restype = I
        L.gdn_tape_replay.argtypes = [P, P, P, I, I, I, I, I, I, I, P, P]
        L.gdn_tape_replay.restype = I
        _lib = L
    return _lib


def _check(status: int, where: str) -> None:
    if status != SV_OK:
        msg = lib().sv_last_error().decode() or lib().sv_status_string(status).decode()
        raise SvError(status, where, msg)


def _ptr(t: torch.Tensor | None):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _stream(device: torch.device):
    return ctypes.c_void_p(torch.cuda.current_stream(device).cuda_stream)


def _need(t: torch.Tensor, name: str, dtype, shape=None, device=None):
    if not isinstance(t, torch.Tensor):
        raise TypeError(f"{name} must be a torch.Tensor")
    if t.device.type != "cuda":
        raise ValueError(f"{name} must be a CUDA tensor")
    if device is not None and t.device != device:
        raise ValueError(f"{name} is on {t.device}, expected {device}")
    if t.dtype != dtype:
        raise TypeError(f"{name} must be {dtype}, got {t.dtype}")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")
    if shape is not None and tuple(t.shape) != tuple(shape):
        raise ValueError(f"{name} has shape {tuple(t.shape)}, expected {tuple(shape)}")


def abi_version() -> int:
    return lib().sv_abi_version()


def set_pdl(enable: bool) -> None:
    """Programmatic dependent launch for qmv_smallm (see specverify.h)."""
    lib().sv_set_pdl(1 if enable else 0)


def get_pdl() -> bool:
    return bool(lib().sv_get_pdl())


def device_status() -> None:
    """Synchronises and raises SvError if a kernel gave up on a bounded wait."""
    _check(lib().sv_device_status(), "sv_device_status")


# ----------------------------------------------------------------------------
def qmv_smallm(w_packed: torch.Tensor, scales: torch.Tensor, biases: torch.Tensor,
               x: torch.Tensor, y: torch.Tensor | None = None) -> torch.Tensor:
    """y[M, N] (fp32) = x[M, K] . W^T.

    w_packed int32/uint32 view [N, K/8]; scales, biases bf16 [N, K/64] (or
    int16 bit patterns); x fp32 or bf16 [M, K].
    """
    dev = w_packed.device
    N, K8 = w_packed.shape
    K = K8 * 8
    M = x.shape[0]
    wdt = w_packed.dtype
    if wdt not in (torch.int32, torch.uint32):
        raise TypeError("w_packed must be int32 or uint32")
    _need(w_packed, "w_packed", wdt, (N, K8), dev)
    sdt = scales.dtype
    if sdt not in (torch.bfloat16, torch.int16):
        raise TypeError("scales must be bfloat16 (or int16 bit patterns)")
    _need(scales, "scales", sdt, (N, K // 64), dev)
    _need(biases, "biases", sdt, (N, K // 64), dev)
    if x.dtype not in (torch.float32, torch.bfloat16):
        raise TypeError("x must be float32 or bfloat16")
    _need(x, "x", x.dtype, (M, K), dev)
    if y is None:
        y = torch.empty((M, N), dtype=torch.float32, device=dev)
    _need(y, "y", torch.float32, (M, N), dev)
    st = lib().qmv_smallm(_ptr(w_packed), _ptr(scales), _ptr(biases), _ptr(x),
                          SV_BF16 if x.dtype == torch.bfloat16 else SV_F32, _ptr(y),
                          M, N, K, 64, 4, _stream(dev))
    _check(st, "qmv_smallm")
    return y


def qmv_identity_probe(w_packed: torch.Tensor, scales: torch.Tensor, biases: torch.Tensor,
                       M: int, x_dtype: torch.dtype = torch.bfloat16) -> int:
    """Start-up check of block verification for one projection: the number
    of outputs, over three synthetic M-row activation blocks, where the M-row
    qmv_smallm product differs in any bit from the same rows multiplied one at
    a time (0: exact).  Synchronous."""
    dev = w_packed.device
    N, K8 = w_packed.shape
    K = K8 * 8
    if w_packed.dtype not in (torch.int32, torch.uint32):
        raise TypeError("w_packed must be int32 or uint32")
    _need(w_packed, "w_packed", w_packed.dtype, (N, K8), dev)
    if scales.dtype not in (torch.bfloat16, torch.int16):
        raise TypeError("scales must be bfloat16 (or int16 bit patterns)")
    _need(scales, "scales", scales.dtype, (N, K // 64), dev)
    _need(biases, "biases", scales.dtype, (N, K // 64), dev)
    if x_dtype not in (torch.float32, torch.bfloat16):
        raise TypeError("x_dtype must be float32 or bfloat16")
    dt = SV_BF16 if x_dtype == torch.bfloat16 else SV_F32
    nbytes = int(lib().qmv_identity_probe_bytes(M, N, K, dt))
    out = ctypes.c_int(-1)
    if nbytes == 0:  # invalid: the probe itself reports why, before any work
        _check(lib().qmv_identity_probe(_ptr(w_packed), _ptr(scales), _ptr(biases), dt, M, N, K,
                                        None, 0, ctypes.byref(out), _stream(dev)),
               "qmv_identity_probe")
    scratch = torch.empty(nbytes + 256, dtype=torch.uint8, device=dev)
    off = (-scratch.data_ptr()) % 256
    st = lib().qmv_identity_probe(_ptr(w_packed), _ptr(scales), _ptr(biases), dt, M, N, K,
                                  scratch.data_ptr() + off, nbytes, ctypes.byref(out),
                                  _stream(dev))
    _check(st, "qmv_identity_probe")
    return int(out.value)


def qmv_requantize(w: torch.Tensor, out=None):
    """4-bit affine group-64 requantisation of a bf16 matrix [N, K] (the
    drafter's own LM head): returns (w_packed int32 [N, K/8], scales, biases
    bf16 [N, K/64]), the qmv_smallm layout; ``out`` may supply that triple."""
    dev = w.device
    if w.dtype not in (torch.bfloat16, torch.int16):
        raise TypeError("w must be bfloat16 (or int16 bit patterns)")
    if w.dim() != 2:
        raise ValueError("w must be [N, K]")
    N, K = w.shape
    _need(w, "w", w.dtype, (N, K), dev)
    if out is None:
        out = (torch.empty((N, K // 8), dtype=torch.int32, device=dev),
               torch.empty((N, K // 64), dtype=torch.bfloat16, device=dev),
               torch.empty((N, K // 64), dtype=torch.bfloat16, device=dev))
    wp, s, b = out
    _need(wp, "w_packed", torch.int32, (N, K // 8), dev)
    _need(s, "scales", torch.bfloat16, (N, K // 64), dev)
    _need(b, "biases", torch.bfloat16, (N, K // 64), dev)
    _check(lib().qmv_requantize(_ptr(w), _ptr(wp), _ptr(s), _ptr(b), N, K, _stream(dev)),
           "qmv_requantize")
    return wp, s, b


def make_wide_workspace(M: int, K: int, device) -> torch.Tensor:
    """A workspace for qmv_wide with M activation rows of K inputs (256-byte
    aligned: torch's allocator aligns far more)."""
    nbytes = int(lib().qmv_wide_workspace_bytes(M, K))
    if nbytes == 0:
        _check(SV_ERR_INVALID_ARG, "qmv_wide_workspace_bytes")
    return torch.empty(nbytes, dtype=torch.uint8, device=device)


def qmv_wide(w_packed: torch.Tensor, scales: torch.Tensor, biases: torch.Tensor,
             x: torch.Tensor, y: torch.Tensor | None = None,
             workspace: torch.Tensor | None = None) -> torch.Tensor:
    """y[M, N] (fp32) = x[M, K] . W^T on the tcgen05 tensor cores, M <= 128.

    Weight layout of qmv_smallm; x bf16 [M, K], K % 512 == 0.  ``workspace``
    (uint8, from make_wide_workspace) is allocated per call when omitted.
    """
    dev = w_packed.device
    N, K8 = w_packed.shape
    K = K8 * 8
    M = x.shape[0]
    wdt = w_packed.dtype
    if wdt not in (torch.int32, torch.uint32):
        raise TypeError("w_packed must be int32 or uint32")
    _need(w_packed, "w_packed", wdt, (N, K8), dev)
    sdt = scales.dtype
    if sdt not in (torch.bfloat16, torch.int16):
        raise TypeError("scales must be bfloat16 (or int16 bit patterns)")
    _need(scales, "scales", sdt, (N, K // 64), dev)
    _need(biases, "biases", sdt, (N, K // 64), dev)
    if x.dtype not in (torch.bfloat16, torch.int16):
        raise TypeError("x must be bfloat16 (or int16 bit patterns)")
    _need(x, "x", x.dtype, (M, K), dev)
    if y is None:
        y = torch.empty((M, N), dtype=torch.float32, device=dev)
    _need(y, "y", torch.float32, (M, N), dev)
    if workspace is None:
        nbytes = int(lib().qmv_wide_workspace_bytes(M, K))
        workspace = torch.empty(max(nbytes, 1), dtype=torch.uint8, device=dev)
    if workspace.dtype != torch.uint8 or workspace.device != dev or not workspace.is_contiguous():
        raise ValueError("workspace must be a contiguous uint8 tensor on the weights' device")
    st = lib().qmv_wide(_ptr(w_packed), _ptr(scales), _ptr(biases), _ptr(x), _ptr(y), M, N, K,
                        _ptr(workspace), workspace.numel(), _stream(dev))
    _check(st, "qmv_wide")
    return y


class QmvPlan:
    """An ordered list of qmv_smallm problems run by one persistent launch.

    ``problems``: sequence of (w_packed, scales, biases, x, y, after[, topk])
    with the shapes of :func:`qmv_smallm`; ``after`` = True when x is the
    output of an earlier problem of the list.  ``topk`` (at most one problem;
    a uint8 tensor from :func:`make_topk_lists`, y then None) makes that
    problem write per-CTA top-64 lists instead of y.  All x share dtype and M.
    The plan keeps references to every tensor and to its device buffer."""

    def __init__(self, problems):
        if not problems:
            raise ValueError("a plan needs at least one problem")
        x0 = problems[0][3]
        dev = x0.device
        M = x0.shape[0]
        arr = (_QmvProblem * len(problems))()
        dt = SV_BF16 if x0.dtype == torch.bfloat16 else SV_F32
        for i, prob in enumerate(problems):
            w, s_, b_, x, y, after = prob[:6]
            topk = prob[6] if len(prob) > 6 else None
            N, K8 = w.shape
            K = K8 * 8
            _need(w, f"problems[{i}].w_packed", torch.int32, (N, K8), dev)
            _need(s_, f"problems[{i}].scales", torch.bfloat16, (N, K // 64), dev)
            _need(b_, f"problems[{i}].biases", torch.bfloat16, (N, K // 64), dev)
            _need(x, f"problems[{i}].x", x0.dtype, (M, K), dev)
            if topk is None:
                _need(y, f"problems[{i}].y", torch.float32, (M, N), dev)
            else:
                _need(topk, f"problems[{i}].topk", torch.uint8, None, dev)
                if topk.numel() < int(lib().qmv_plan_topk_bytes(M, dt)):
                    raise ValueError(f"problems[{i}].topk is smaller than qmv_plan_topk_bytes")
            arr[i] = _QmvProblem(w.data_ptr(), s_.data_ptr(), b_.data_ptr(), x.data_ptr(),
                                 None if y is None else y.data_ptr(), N, K, 1 if after else 0,
                                 None if topk is None else topk.data_ptr())
        with torch.cuda.device(dev):
            n = int(lib().qmv_plan_device_bytes(arr, len(problems), M, dt))
            if n == 0:  # invalid: qmv_plan_create reports why, with its status
                h = ctypes.c_void_p()
                _check(lib().qmv_plan_create(arr, len(problems), M, dt, None, 0,
                                             ctypes.byref(h)), "qmv_plan_create")
                raise SvError(SV_ERR_INVALID_ARG, "qmv_plan_device_bytes",
                              lib().sv_last_error().decode())
            self.buffer = torch.empty(n + 256, dtype=torch.uint8, device=dev)
            off = (-self.buffer.data_ptr()) % 256
            h = ctypes.c_void_p()
            _check(lib().qmv_plan_create(arr, len(problems), M, dt,
                                         ctypes.c_void_p(self.buffer.data_ptr() + off),
                                         n, ctypes.byref(h)), "qmv_plan_create")
        self._h = h
        self._off, self._nbytes = off, n  # the plan's bytes: buffer[off : off + n]
        self.device = dev
        self.problems = list(problems)  # keep the tensors alive
        self.grid = int(lib().qmv_plan_grid(h))

    def run(self, cooperative: bool = False) -> None:
        """One launch on the current stream; ``cooperative`` guarantees that
        all CTAs are resident together (beside other self-waiting grids)."""
        if cooperative:
            _check(lib().qmv_plan_run_cooperative(self._h, _stream(self.device)),
                   "qmv_plan_run_cooperative")
        else:
            _check(lib().qmv_plan_run(self._h, _stream(self.device)), "qmv_plan_run")

    def close(self) -> None:
        if getattr(self, "_h", None):
            lib().qmv_plan_destroy(self._h)
            self._h = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass


def make_topk_lists(M: int, x_dtype: torch.dtype, device) -> torch.Tensor:
    """A buffer (uint8) for a plan problem's top-64 epilogue: per CTA and row
    64 keys (uint64), then one flag word per CTA and row."""
    dt = SV_BF16 if x_dtype == torch.bfloat16 else SV_F32
    with torch.cuda.device(device):
        n = int(lib().qmv_plan_topk_bytes(M, dt))
    if n == 0:
        _check(SV_ERR_INVALID_ARG, "qmv_plan_topk_bytes")
    return torch.empty(n, dtype=torch.uint8, device=device)


def spec_accept_workspace_bytes(B: int, K: int, V: int) -> int:
    return int(lib().spec_accept_workspace_bytes(B, K, V))


def make_accept_workspace(B: int, K: int, V: int, device) -> torch.Tensor:
    """A zero-filled workspace (uint8) for spec_accept at these sizes."""
    n = spec_accept_workspace_bytes(B, K, V)
    return torch.zeros(max(n, 16), dtype=torch.uint8, device=device)


def spec_accept(target_logits: torch.Tensor, draft_logits: torch.Tensor | None,
                draft_tokens: torch.Tensor, u_accept: torch.Tensor, u_sample: torch.Tensor,
                temperature: float, top_k: int, top_p: float,
                workspace: torch.Tensor | None = None, out_tokens: torch.Tensor | None = None,
                n_accepted: torch.Tensor | None = None, err_flags: torch.Tensor | None = None):
    """Returns (out_tokens [B, K+1] int32, n_accepted [B] int32, err_flags [B] int32)."""
    dev = target_logits.device
    B, K1, V = target_logits.shape
    K = K1 - 1
    _need(target_logits, "target_logits", torch.float32, (B, K + 1, V), dev)
    if draft_logits is not None:
        _need(draft_logits, "draft_logits", torch.float32, (B, K, V), dev)
    _need(draft_tokens, "draft_tokens", torch.int32, (B, K), dev)
    _need(u_accept, "u_accept", torch.float32, (B, K), dev)
    _need(u_sample, "u_sample", torch.float32, (B,), dev)
    if workspace is None:
        workspace = make_accept_workspace(B, K, V, dev)
    _need(workspace, "workspace", torch.uint8, None, dev)
    if out_tokens is None:
        out_tokens = torch.empty((B, K + 1), dtype=torch.int32, device=dev)
    if n_accepted is None:
        n_accepted = torch.empty((B,), dtype=torch.int32, device=dev)
    if err_flags is None:
        err_flags = torch.empty((B,), dtype=torch.int32, device=dev)
    _need(out_tokens, "out_tokens", torch.int32, (B, K + 1), dev)
    _need(n_accepted, "n_accepted", torch.int32, (B,), dev)
    _need(err_flags, "err_flags", torch.int32, (B,), dev)
    samp = _Sampling(float(temperature), int(top_k), float(top_p))
    with torch.cuda.device(dev):
        st = lib().spec_accept(_ptr(target_logits), _ptr(draft_logits), _ptr(draft_tokens),
                               _ptr(u_accept), _ptr(u_sample), B, K, V, samp, _ptr(out_tokens),
                               _ptr(n_accepted), _ptr(err_flags), _ptr(workspace),
                               workspace.numel(), _stream(dev))
    _check(st, "spec_accept")
    return out_tokens, n_accepted, err_flags


def spec_accept_lists(target_lists: torch.Tensor, G: int, V: int,
                      draft_logits: torch.Tensor | None, draft_tokens: torch.Tensor,
                      u_accept: torch.Tensor, u_sample: torch.Tensor, temperature: float,
                      top_k: int, top_p: float, workspace: torch.Tensor | None = None,
                      out_tokens: torch.Tensor | None = None,
                      n_accepted: torch.Tensor | None = None,
                      err_flags: torch.Tensor | None = None):
    """spec_accept with the target rows as per-CTA top-64 lists of a fused LM
    head (a plan problem's ``topk`` buffer, uint8, one block per sequence of
    spec_accept_lists_block_bytes(G, K) bytes).  Same returns as spec_accept."""
    dev = target_lists.device
    B, K = draft_tokens.shape
    _need(target_lists, "target_lists", torch.uint8, None, dev)
    blk = int(lib().spec_accept_lists_block_bytes(G, K))
    if target_lists.numel() < B * blk:
        raise ValueError(f"target_lists holds {target_lists.numel()} bytes, need {B * blk}")
    if draft_logits is not None:
        _need(draft_logits, "draft_logits", torch.float32, (B, K, V), dev)
    _need(draft_tokens, "draft_tokens", torch.int32, (B, K), dev)
    _need(u_accept, "u_accept", torch.float32, (B, K), dev)
    _need(u_sample, "u_sample", torch.float32, (B,), dev)
    if workspace is None:
        n = int(lib().spec_accept_lists_workspace_bytes(B, K, V, int(G)))
        workspace = torch.zeros(max(n, 16), dtype=torch.uint8, device=dev)
    _need(workspace, "workspace", torch.uint8, None, dev)
    if out_tokens is None:
        out_tokens = torch.empty((B, K + 1), dtype=torch.int32, device=dev)
    if n_accepted is None:
        n_accepted = torch.empty((B,), dtype=torch.int32, device=dev)
    if err_flags is None:
        err_flags = torch.empty((B,), dtype=torch.int32, device=dev)
    _need(out_tokens, "out_tokens", torch.int32, (B, K + 1), dev)
    _need(n_accepted, "n_accepted", torch.int32, (B,), dev)
    _need(err_flags, "err_flags", torch.int32, (B,), dev)
    samp = _Sampling(float(temperature), int(top_k), float(top_p))
    with torch.cuda.device(dev):
        st = lib().spec_accept_lists(_ptr(target_lists), int(G), _ptr(draft_logits),
                                     _ptr(draft_tokens), _ptr(u_accept), _ptr(u_sample), B, K,
                                     V, samp, _ptr(out_tokens), _ptr(n_accepted),
                                     _ptr(err_flags), _ptr(workspace), workspace.numel(),
                                     _stream(dev))
    _check(st, "spec_accept_lists")
    return out_tokens, n_accepted, err_flags


def spec_accept_noalloc_scratch_bytes() -> int:
    return int(lib().spec_accept_noalloc_scratch_bytes())


def spec_accept_noalloc(target_logits: torch.Tensor, draft_logits: torch.Tensor | None,
                        draft_tokens: torch.Tensor, u_accept: torch.Tensor,
                        u_sample: torch.Tensor, temperature: float, top_k: int, top_p: float,
                        out_tokens: torch.Tensor, n_accepted: torch.Tensor,
                        err_flags: torch.Tensor | None = None) -> None:
    """spec_accept on the library's fixed device scratch: the caller passes
    every output, so nothing is allocated.  Calls on one device must not
    overlap in time."""
    dev = target_logits.device
    B, K1, V = target_logits.shape
    K = K1 - 1
    _need(target_logits, "target_logits", torch.float32, (B, K + 1, V), dev)
    if draft_logits is not None:
        _need(draft_logits, "draft_logits", torch.float32, (B, K, V), dev)
    _need(draft_tokens, "draft_tokens", torch.int32, (B, K), dev)
    _need(u_accept, "u_accept", torch.float32, (B, K), dev)
    _need(u_sample, "u_sample", torch.float32, (B,), dev)
    _need(out_tokens, "out_tokens", torch.int32, (B, K + 1), dev)
    _need(n_accepted, "n_accepted", torch.int32, (B,), dev)
    if err_flags is not None:
        _need(err_flags, "err_flags", torch.int32, (B,), dev)
    samp = _Sampling(float(temperature), int(top_k), float(top_p))
    # the scratch is looked up on the current device: make it the tensors' one
    with torch.cuda.device(dev):
        st = lib().spec_accept_noalloc(_ptr(target_logits), _ptr(draft_logits),
                                       _ptr(draft_tokens), _ptr(u_accept), _ptr(u_sample), B, K,
                                       V, samp, _ptr(out_tokens), _ptr(n_accepted),
                                       _ptr(err_flags), _stream(dev))
    _check(st, "spec_accept_noalloc")


def gdn_tape_bytes(B: int, T: int, H: int, dk: int, dv: int) -> int:
    return int(lib().gdn_tape_bytes(B, T, H, dk, dv))


def gdn_tape_capture(state0: torch.Tensor, q: torch.Tensor, k: torch.Tensor, v: torch.Tensor,
                     alpha: torch.Tensor, beta: torch.Tensor, tape: torch.Tensor | None = None,
                     out: torch.Tensor | None = None, want_out: bool = True,
                     state_out: torch.Tensor | None = None):
    """Returns (out [B,T,H,dv] fp32 or None, tape fp32 flat); ``state_out``
    [B,H,dv,dk], when given, receives the state after all T tokens."""
    dev = state0.device
    B, H, dv, dk = state0.shape
    T = q.shape[1]
    _need(state0, "state0", torch.float32, (B, H, dv, dk), dev)
    _need(q, "q", torch.float32, (B, T, H, dk), dev)
    _need(k, "k", torch.float32, (B, T, H, dk), dev)
    _need(v, "v", torch.float32, (B, T, H, dv), dev)
    _need(alpha, "alpha", torch.float32, (B, T, H), dev)
    _need(beta, "beta", torch.float32, (B, T, H), dev)
    n = gdn_tape_bytes(B, T, H, dk, dv) // 4
    if tape is None:
        tape = torch.empty(n, dtype=torch.float32, device=dev)
    _need(tape, "tape", torch.float32, (n,), dev)
    if out is None and want_out:
        out = torch.empty((B, T, H, dv), dtype=torch.float32, device=dev)
    if out is not None:
        _need(out, "out", torch.float32, (B, T, H, dv), dev)
    if state_out is not None:
        _need(state_out, "state_out", torch.float32, (B, H, dv, dk), dev)
    st = lib().gdn_tape_capture(_ptr(state0), _ptr(q), _ptr(k), _ptr(v), _ptr(alpha), _ptr(beta),
                                B, T, H, dk, dv, _ptr(out), _ptr(tape), _ptr(state_out),
                                _stream(dev))
    _check(st, "gdn_tape_capture")
    return out, tape


def gdn_tape_replay(state: torch.Tensor, tape: torch.Tensor, n_replay: torch.Tensor, T: int,
                    n_replay_bias: int = 0, err_flags: torch.Tensor | None = None) -> torch.Tensor:
    """Replays n_replay[b % len(n_replay)] + bias records of ``tape`` into
    ``state`` [B, H, dv, dk] in place; returns state."""
    dev = state.device
    B, H, dv, dk = state.shape
    _need(state, "state", torch.float32, (B, H, dv, dk), dev)
    n = gdn_tape_bytes(B, T, H, dk, dv) // 4
    _need(tape, "tape", torch.float32, (n,), dev)
    _need(n_replay, "n_replay", torch.int32, None, dev)
    if n_replay.dim() != 1:
        raise ValueError("n_replay must be 1-D")
    if err_flags is not None:
        _need(err_flags, "err_flags", torch.int32, (B,), dev)
    st = lib().gdn_tape_replay(_ptr(state), _ptr(tape), _ptr(n_replay), n_replay.numel(),
                               int(n_replay_bias), B, T, H, dk, dv, _ptr(err_flags), _stream(dev))
    _check(st, "gdn_tape_replay")
    return state


def conv_window_capture(window: torch.Tensor, x: torch.Tensor, weight: torch.Tensor,
                        y: torch.Tensor | None = None) -> torch.Tensor:
    """Causal depthwise convolution outputs y [B, T, C] (fp32) of x [B, T, C]
    from the committed window [B, W-1, C] (read only), weight [W, C]."""
    dev = x.device
    B, T, C = x.shape
    W = weight.shape[0]
    _need(window, "window", torch.float32, (B, W - 1, C), dev)
    _need(x, "x", torch.float32, (B, T, C), dev)
    _need(weight, "weight", torch.float32, (W, C), dev)
    if y is None:
        y = torch.empty((B, T, C), dtype=torch.float32, device=dev)
    _need(y, "y", torch.float32, (B, T, C), dev)
    _check(lib().conv_window_capture(_ptr(window), _ptr(x), _ptr(weight), B, T, C, W, _ptr(y),
                                     _stream(dev)), "conv_window_capture")
    return y


def conv_window_replay(window: torch.Tensor, x: torch.Tensor, n_replay: torch.Tensor,
                       n_replay_bias: int = 0, err_flags: torch.Tensor | None = None) -> None:
    """Commits the first n_replay[b % len] + bias verify inputs of x [B, T, C]
    into window [B, W-1, C] in place."""
    dev = x.device
    B, T, C = x.shape
    W = window.shape[1] + 1
    _need(window, "window", torch.float32, (B, W - 1, C), dev)
    _need(x, "x", torch.float32, (B, T, C), dev)
    _need(n_replay, "n_replay", torch.int32, None, dev)
    if err_flags is not None:
        _need(err_flags, "err_flags", torch.int32, (B,), dev)
    _check(lib().conv_window_replay(_ptr(window), _ptr(x), _ptr(n_replay), n_replay.numel(),
                                    int(n_replay_bias), B, T, C, W, _ptr(err_flags),
                                    _stream(dev)), "conv_window_replay")
