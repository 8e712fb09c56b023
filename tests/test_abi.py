"""The C ABI boundary, on the host (no GPU): the library loads, exports every
entry point include/specverify.h declares, and rejects invalid arguments
before any launch (every call below returns during host-side validation)."""
import ctypes
import re
from pathlib import Path

import pytest

ROOT = Path(__file__).resolve().parents[1]
HEADER = ROOT / "include" / "specverify.h"


@pytest.fixture(scope="module")
def L():
    from mtp_speculative_decoding_qmv_gb300 import build as b

    b.build()
    import mtp_speculative_decoding_qmv_gb300 as sv

    return sv.lib()


def _declared_functions():
    text = re.sub(r"/\*.*?\*/", "", HEADER.read_text(), flags=re.S)
    text = re.sub(r"#.*", "", text)
    names = []
    for stmt in text.split(";"):
        stmt = " ".join(stmt.split())
        if stmt.startswith("typedef") or "(" not in stmt or "{" in stmt:
            continue
        m = re.search(r"([A-Za-z_]\w*)\s*\(", stmt)
        if m:
            names.append(m.group(1))
    return names


def test_header_declares_the_path():
    names = set(_declared_functions())
    assert {"qmv_smallm", "spec_accept", "gdn_tape_capture", "gdn_tape_replay"} <= names


def test_library_exports_every_declared_symbol(L):
    for name in _declared_functions():
        assert hasattr(L, name), name


def test_abi_version_and_status_strings(L):
    assert L.sv_abi_version() == 2
    assert L.sv_status_string(0) == b"ok"
    assert L.sv_status_string(1) == b"invalid argument"
    assert L.sv_status_string(99) == b"unknown status"


def test_pdl_switch(L):
    L.sv_set_pdl(1)
    assert L.sv_get_pdl() == 1
    L.sv_set_pdl(0)
    assert L.sv_get_pdl() == 0


A = 0x10000  # a 16-byte aligned fake device address; never dereferenced here


def _qmv(L, w=A, s=A + 0x1000000, b=A + 0x2000000, x=A + 0x3000000, dt=1, y=A + 0x4000000,
         M=4, N=64, K=256, gs=64, bits=4):
    return L.qmv_smallm(w, s, b, x, dt, y, M, N, K, gs, bits, None)


@pytest.mark.parametrize("kw,status", [
    ({"K": 100}, 1), ({"K": 0}, 1), ({"M": -1}, 1), ({"gs": 32}, 2), ({"bits": 8}, 2),
    ({"M": 17}, 2), ({"dt": 7}, 1), ({"w": 0}, 1), ({"y": 0}, 1), ({"w": A + 4}, 1),
    ({"x": A + 0x3000008}, 1), ({"y": A + 2}, 1), ({"y": A + 0x3000000}, 1),
])
def test_qmv_rejects(L, kw, status):
    assert _qmv(L, **kw) == status
    assert L.sv_last_error() != b""


def test_qmv_empty_is_a_noop(L):
    assert _qmv(L, M=0) == 0
    assert _qmv(L, N=0) == 0


def _accept(L, tl=A, dl=A + 0x1000000, dt=A + 0x2000000, ua=A + 0x2100000, us=A + 0x2200000,
            B=2, K=3, V=1000, T=0.6, top_k=20, top_p=0.95, out=A + 0x3000000,
            nacc=A + 0x3100000, flags=A + 0x3200000, ws=A + 0x4000000, ws_bytes=None):
    import mtp_speculative_decoding_qmv_gb300 as sv

    if ws_bytes is None:
        ws_bytes = max(L.spec_accept_workspace_bytes(max(B, 0), max(K, 1), max(V, 1)), 16)
    return L.spec_accept(tl, dl, dt, ua, us, B, K, V, sv._Sampling(T, top_k, top_p), out, nacc,
                         flags, ws, ws_bytes, None)


@pytest.mark.parametrize("kw,status", [
    ({"K": 0}, 1), ({"K": 9}, 2), ({"V": 0}, 1), ({"V": 2_000_000}, 2), ({"B": -1}, 1),
    ({"top_k": 0}, 2), ({"top_k": 65}, 2), ({"top_p": 0.0}, 1), ({"top_p": 1.5}, 1),
    ({"T": -1.0}, 1), ({"T": float("nan")}, 1), ({"ws_bytes": 8}, 1), ({"ws": A + 8}, 1),
    ({"tl": 0}, 1), ({"dl": 0}, 1), ({"out": A}, 1), ({"nacc": A + 0x3000000}, 1),
    ({"B": 10000}, 2),
])
def test_accept_rejects(L, kw, status):
    assert _accept(L, **kw) == status


def test_accept_greedy_allows_null_draft_logits_and_empty_batch(L):
    assert _accept(L, B=0) == 0
    # greedy validation passes with draft_logits == NULL (launch not reached: B=0)
    assert _accept(L, B=0, dl=0, T=0.0, top_k=0, top_p=1.0) == 0


def test_workspace_size_is_monotone(L):
    a = L.spec_accept_workspace_bytes(32, 3, 151936)
    assert a > 0 and L.spec_accept_workspace_bytes(64, 3, 151936) > a
    assert L.spec_accept_workspace_bytes(32, 0, 100) == 0


def test_tape_bytes_matches_record_size(L):
    # one record per (b, t, h): alpha + e[dv] + k[dk] fp32 = 1028 bytes at 128/128
    # (T*H = 240 gates per sequence block: already a multiple of 4)
    assert L.gdn_tape_bytes(16, 5, 48, 128, 128) == 16 * 5 * 48 * 1028
    assert L.gdn_tape_bytes(1, 1, 1, 4, 4) == 4 * (8 + 4)
    assert L.gdn_tape_bytes(0, 5, 48, 128, 128) == 0


@pytest.mark.parametrize("kw,status", [
    ({"T": 0}, 1), ({"T": 17}, 2), ({"dk": 130}, 2), ({"dv": 6}, 2), ({"H": 0}, 1),
    ({"state0": 0}, 1), ({"q": A + 4}, 1), ({"tape": A}, 1),
])
def test_capture_rejects(L, kw, status):
    args = dict(state0=A, q=A + 0x1000000, k=A + 0x2000000, v=A + 0x3000000, alpha=A + 0x4000000,
                beta=A + 0x5000000, B=2, T=5, H=4, dk=128, dv=128, out=A + 0x6000000,
                tape=A + 0x7000000, state_out=None)
    args.update(kw)
    st = L.gdn_tape_capture(args["state0"], args["q"], args["k"], args["v"], args["alpha"],
                            args["beta"], args["B"], args["T"], args["H"], args["dk"],
                            args["dv"], args["out"], args["tape"], args["state_out"], None)
    assert st == status


def test_replay_rejects(L):
    assert L.gdn_tape_replay(A, A + 0x1000000, None, 2, 1, 2, 5, 4, 128, 128, None, None) == 1
    assert L.gdn_tape_replay(A, A, A + 0x2000000, 2, 1, 2, 5, 4, 128, 128, None, None) == 1
    assert L.gdn_tape_replay(A + 4, A + 0x1000000, A + 0x2000000, 2, 1, 2, 5, 4, 128, 128, None,
                             None) == 1
    assert L.gdn_tape_replay(A, A + 0x1000000, A + 0x2000000, 3, 1, 2, 5, 4, 128, 128, None,
                             None) == 1  # count > B
    assert L.gdn_tape_replay(A, A + 0x1000000, A + 0x2000000, 0, 1, 2, 5, 4, 128, 128, None,
                             None) == 1  # count < 1
    assert L.gdn_tape_replay(A, A + 0x1000000, A + 0x2000000, 1, 0, 0, 5, 4, 128, 128, None,
                             None) == 0


def test_conv_window_rejects(L):
    win, x, w, y = A, A + 0x1000000, A + 0x2000000, A + 0x3000000
    assert L.conv_window_capture(win, x, w, 2, 5, 64, 1, y, None) == 2   # W < 2
    assert L.conv_window_capture(win, x, w, 2, 5, 64, 9, y, None) == 2   # W > 8
    assert L.conv_window_capture(win, x, w, 2, 65, 64, 4, y, None) == 2  # T > 64
    assert L.conv_window_capture(win, x, w, 2, 0, 64, 4, y, None) == 1   # T < 1
    assert L.conv_window_capture(None, x, w, 2, 5, 64, 4, y, None) == 1
    assert L.conv_window_capture(win, x, w, 2, 5, 64, 4, x, None) == 1   # y overlaps x
    assert L.conv_window_capture(win, x, w, 0, 5, 64, 4, y, None) == 0   # empty batch
    n = A + 0x4000000
    assert L.conv_window_replay(win, x, n, 3, 1, 2, 5, 64, 4, None, None) == 1  # count > B
    assert L.conv_window_replay(win, x, None, 1, 1, 2, 5, 64, 4, None, None) == 1
    assert L.conv_window_replay(win, win, n, 1, 1, 2, 5, 64, 4, None, None) == 1  # window = x
    assert L.conv_window_replay(win + 2, x, n, 1, 1, 2, 5, 64, 4, None, None) == 1
    assert L.conv_window_replay(win, x, n, 1, 1, 0, 5, 64, 4, None, None) == 0


def test_identity_probe_sizes_and_rejects(L):
    # x: 3 blocks of 4 x 512 bf16, y block and y rows 4 x 512 fp32, a counter
    assert L.qmv_identity_probe_bytes(4, 512, 512, 1) == 12288 + 8192 + 8192 + 256
    assert L.qmv_identity_probe_bytes(4, 512, 512, 0) == 24576 + 8192 + 8192 + 256
    assert L.qmv_identity_probe_bytes(17, 512, 512, 1) == 0
    assert L.qmv_identity_probe_bytes(4, 512, 100, 1) == 0
    w, s, b, scr = A, A + 0x1000000, A + 0x2000000, A + 0x3000000
    n = L.qmv_identity_probe_bytes(4, 512, 512, 1)
    out = ctypes.c_int(7)
    assert L.qmv_identity_probe(w, s, b, 1, 0, 512, 512, scr, n, ctypes.byref(out), None) == 2
    assert L.qmv_identity_probe(w, s, b, 1, 17, 512, 512, scr, n, ctypes.byref(out), None) == 2
    assert L.qmv_identity_probe(w, s, b, 1, 4, 512, 96, scr, n, ctypes.byref(out), None) == 1
    assert L.qmv_identity_probe(w, s, b, 7, 4, 512, 512, scr, n, ctypes.byref(out), None) == 1
    assert L.qmv_identity_probe(None, s, b, 1, 4, 512, 512, scr, n, ctypes.byref(out), None) == 1
    assert L.qmv_identity_probe(w, s, b, 1, 4, 512, 512, scr, n, None, None) == 1
    assert L.qmv_identity_probe(w, s, b, 1, 4, 512, 512, scr + 16, n, ctypes.byref(out),
                                None) == 1  # scratch not 256-byte aligned
    assert L.qmv_identity_probe(w, s, b, 1, 4, 512, 512, scr, n - 1, ctypes.byref(out),
                                None) == 1  # scratch too small
    assert L.qmv_identity_probe(w, s, b, 1, 4, 512, 512, w, n, ctypes.byref(out),
                                None) == 1  # scratch overlaps the weights
    assert out.value == 7  # rejected before any work: left unchanged


def test_wide_sizes_and_rejects(L):
    # split group sums: M rows x (2 K/64 rounded up to 128) bf16, 256-byte multiple
    assert L.qmv_wide_workspace_bytes(128, 5120) == 128 * 256 * 2
    assert L.qmv_wide_workspace_bytes(3, 512) == 768
    assert L.qmv_wide_workspace_bytes(129, 512) == 0
    assert L.qmv_wide_workspace_bytes(4, 640) == 0
    w, s, b, x, y, ws = (A + i * 0x1000000 for i in range(6))
    n = L.qmv_wide_workspace_bytes(64, 1024)
    assert L.qmv_wide(w, s, b, x, y, 0, 300, 1024, None, 0, None) == 0  # M = 0: no launch
    assert L.qmv_wide(w, s, b, x, y, 64, 0, 1024, None, 0, None) == 0   # N = 0: no launch
    assert L.qmv_wide(w, s, b, x, y, 129, 300, 1024, ws, n, None) == 2
    assert L.qmv_wide(w, s, b, x, y, 64, 300, 1000, ws, n, None) == 1   # K % 512
    assert L.qmv_wide(w, s, b, x, y, -1, 300, 1024, ws, n, None) == 1
    assert L.qmv_wide(None, s, b, x, y, 64, 300, 1024, ws, n, None) == 1
    assert L.qmv_wide(w, s, b, x, y, 64, 300, 1024, None, n, None) == 1
    assert L.qmv_wide(w + 8, s, b, x, y, 64, 300, 1024, ws, n, None) == 1  # 16-byte alignment
    assert L.qmv_wide(w, s, b, x, y + 2, 64, 300, 1024, ws, n, None) == 1  # 4-byte alignment
    assert L.qmv_wide(w, s, b, x, y, 64, 300, 1024, ws + 16, n, None) == 1  # 256-byte alignment
    assert L.qmv_wide(w, s, b, x, y, 64, 300, 1024, ws, n - 1, None) == 1  # too small
    assert L.qmv_wide(w, s, b, x, x, 64, 300, 1024, ws, n, None) == 1      # y overlaps x
    assert L.qmv_wide(w, s, b, x, y, 64, 300, 1024, x, n, None) == 1       # workspace = x


def test_requantize_rejects(L):
    w, wp, s, b = (A + i * 0x1000000 for i in range(4))
    assert L.qmv_requantize(w, wp, s, b, 0, 128, None) == 0        # N = 0: no launch
    assert L.qmv_requantize(w, wp, s, b, 4, 100, None) == 1        # K % 64
    assert L.qmv_requantize(w, wp, s, b, -1, 128, None) == 1
    assert L.qmv_requantize(None, wp, s, b, 4, 128, None) == 1
    assert L.qmv_requantize(w + 8, wp, s, b, 4, 128, None) == 1    # 16-byte alignment
    assert L.qmv_requantize(w, wp + 2, s, b, 4, 128, None) == 1    # 4-byte alignment
    assert L.qmv_requantize(w, wp, s + 1, b, 4, 128, None) == 1    # 2-byte alignment
    assert L.qmv_requantize(w, w, s, b, 4, 128, None) == 1         # w_packed overlaps w
    assert L.qmv_requantize(w, wp, s, s, 4, 128, None) == 1        # scales = biases


def _accept_lists(L, tl=A, G=304, dl=A + 0x1000000, dt=A + 0x2000000, ua=A + 0x2100000,
                  us=A + 0x2200000, B=2, K=3, V=1000, T=0.6, top_k=20, top_p=0.95,
                  out=A + 0x3000000, nacc=A + 0x3100000, flags=A + 0x3200000, ws=A + 0x4000000,
                  ws_bytes=None):
    import mtp_speculative_decoding_qmv_gb300 as sv

    if ws_bytes is None:
        ws_bytes = max(L.spec_accept_lists_workspace_bytes(max(B, 0), max(K, 1), max(V, 1),
                                                           max(G, 1)), 16)
    return L.spec_accept_lists(tl, G, dl, dt, ua, us, B, K, V, sv._Sampling(T, top_k, top_p),
                               out, nacc, flags, ws, ws_bytes, None)


@pytest.mark.parametrize("kw,status", [
    ({"G": 0}, 2), ({"G": 4096}, 2), ({"tl": 0}, 1), ({"tl": A + 8}, 1), ({"K": 0}, 1),
    ({"top_k": 65}, 2), ({"ws_bytes": 8}, 1), ({"out": A}, 1),
])
def test_accept_lists_rejects(L, kw, status):
    assert _accept_lists(L, **kw) == status


def test_accept_lists_sizes(L):
    # a block per sequence: G x (K+1) x (64 keys x 8 B + one 4-byte flag), 16-byte multiple
    assert L.spec_accept_lists_block_bytes(304, 3) == 304 * 4 * 516
    assert L.spec_accept_lists_block_bytes(3, 1) == (3 * 2 * 516 + 15) // 16 * 16
    assert L.spec_accept_lists_block_bytes(0, 3) == 0
    # one chunk per 32 lists at least: more chunks than a small vocabulary fills
    assert L.spec_accept_lists_workspace_bytes(1, 3, 151936, 304) == \
        L.spec_accept_workspace_bytes(1, 3, 151936)
    assert L.spec_accept_lists_workspace_bytes(1, 3, 1000, 304) > \
        L.spec_accept_workspace_bytes(1, 3, 1000)
    assert _accept_lists(L, B=0) == 0


def test_plan_rejects_two_topk_problems(L):
    import ctypes

    import mtp_speculative_decoding_qmv_gb300 as sv

    arr = (sv._QmvProblem * 2)()
    for i in range(2):
        arr[i] = sv._QmvProblem(A, A + 0x100000, A + 0x200000, A + 0x300000, None, 512, 512, 0,
                                A + 0x1000000 * (i + 1))
    h = ctypes.c_void_p()
    assert L.qmv_plan_create(arr, 2, 4, 1, A + 0x8000000, 1 << 20, ctypes.byref(h)) == 2
    assert b"top-64" in L.sv_last_error()
    arr[0].topk = None   # neither y nor topk: a null output
    arr[1].topk = None
    assert L.qmv_plan_create(arr, 2, 4, 1, A + 0x8000000, 1 << 20, ctypes.byref(h)) == 1
    arr[0].topk = A + 4  # top-k lists must be 8-byte aligned
    assert L.qmv_plan_create(arr, 1, 4, 1, A + 0x8000000, 1 << 20, ctypes.byref(h)) == 1
    assert L.qmv_plan_topk_bytes(0, 1) == 0 and L.qmv_plan_topk_bytes(9, 1) == 0
