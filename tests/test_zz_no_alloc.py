"""spec_accept_noalloc (library-held static scratch) against spec_accept with a
caller workspace, through the C ABI.

Both entry points run the same kernel on the same inputs, so the integer
results (tokens, accepted lengths, flags) must agree exactly.  Each case makes
two noalloc calls in a row on different inputs, so the second one runs on
the scratch the first call left behind.  The file is named to be collected
last: it must pass both alone and after every other GPU test.
"""
import numpy as np
import pytest
import torch

from gpu_util import dev, f32, sv_module, wl

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def sv():
    return sv_module()


def _inputs(stream, B, K, V, sigma, noise):
    tl, dl = wl.accept_logits(stream, B, K, V, sigma=sigma, draft_noise=noise)
    dr = np.argmax(dl, axis=2).astype(np.int32)  # drafts the target often accepts
    ua, us = wl.accept_uniforms(stream, B, K)
    d = dev()
    return [torch.from_numpy(a).to(d) for a in (tl, dl, dr, ua, us)]


def _with_workspace(sv, x, T, top_k, top_p):
    tl, dl, dr, ua, us = x
    out = sv.spec_accept(tl, None if T == 0.0 else dl, dr, ua, us, T, top_k, top_p)
    return [t.cpu().numpy() for t in out]


def _noalloc(sv, x, T, top_k, top_p, outs):
    tl, dl, dr, ua, us = x
    sv.spec_accept_noalloc(tl, None if T == 0.0 else dl, dr, ua, us, T, top_k, top_p, *outs)
    torch.cuda.synchronize()
    return [t.cpu().numpy() for t in outs]


@pytest.mark.parametrize("B,K,V,T,top_k,top_p,sigma,noise", [
    (4, 3, 1000, 0.8, 64, 0.95, 2.0, None),         # tiny vocabulary, independent drafts
    (1, 3, 151936, 0.6, 20, 0.95, 3.0, 0.5),        # LM-head verify, batch 1
    (32, 3, 151936, 0.6, 20, 0.95, 3.0, 0.5),       # batch 32, close to the scratch limit
    (3, 5, 40000, 0.0, 1, 1.0, 2.0, 0.5),           # greedy, ragged last chunk
])
def test_noalloc_matches_workspace_entry_point(sv, B, K, V, T, top_k, top_p, sigma, noise):
    T, top_p = f32(T), f32(top_p)
    assert sv.spec_accept_workspace_bytes(B, K, V) <= sv.spec_accept_noalloc_scratch_bytes()
    d = dev()
    outs = [torch.full((B, K + 1), -7, dtype=torch.int32, device=d),
            torch.full((B,), -7, dtype=torch.int32, device=d),
            torch.full((B,), -7, dtype=torch.int32, device=d)]
    for call, stream in enumerate((900 + B + K, 950 + B + K)):  # two calls in a row
        x = _inputs(stream, B, K, V, sigma, noise)
        ref = _with_workspace(sv, x, T, top_k, top_p)
        got = _noalloc(sv, x, T, top_k, top_p, outs)
        for name, r, g in zip(("out_tokens", "n_accepted", "err_flags"), ref, got):
            np.testing.assert_array_equal(g, r, err_msg=f"call {call}: {name}")
        assert (got[1] >= 0).all() and (got[1] <= K).all()
    sv.device_status()  # raises if a kernel reported a device error


def test_noalloc_shape_changes_on_the_shared_scratch(sv):
    """Calls of different shapes in a row on the one scratch: batch 32 at
    K = 3, then batch 1 at K = 5, then batch 32 at K = 3 again.  Each must
    equal spec_accept on its own fresh workspace, whatever the previous call
    left in the scratch."""
    V, T, top_k, top_p = 151936, f32(0.6), 20, f32(0.95)
    d = dev()
    for call, (B, K) in enumerate([(32, 3), (1, 5), (32, 3)]):
        assert sv.spec_accept_workspace_bytes(B, K, V) <= sv.spec_accept_noalloc_scratch_bytes()
        x = _inputs(970 + call, B, K, V, 3.0, 0.5)
        ref = _with_workspace(sv, x, T, top_k, top_p)
        outs = [torch.full((B, K + 1), -7, dtype=torch.int32, device=d),
                torch.full((B,), -7, dtype=torch.int32, device=d),
                torch.full((B,), -7, dtype=torch.int32, device=d)]
        got = _noalloc(sv, x, T, top_k, top_p, outs)
        for name, r, g in zip(("out_tokens", "n_accepted", "err_flags"), ref, got):
            np.testing.assert_array_equal(g, r, err_msg=f"call {call} (B={B}, K={K}): {name}")
    sv.device_status()


def test_noalloc_rejects_sizes_beyond_the_scratch(sv):
    B, K, V = 64, 8, 151936
    assert sv.spec_accept_workspace_bytes(B, K, V) > sv.spec_accept_noalloc_scratch_bytes()
    tl = torch.zeros((B, K + 1, V), dtype=torch.float32, device=dev())
    outs = [torch.zeros((B, K + 1), dtype=torch.int32, device=dev()),
            torch.zeros((B,), dtype=torch.int32, device=dev()),
            torch.zeros((B,), dtype=torch.int32, device=dev())]
    dl = torch.zeros((B, K, V), dtype=torch.float32, device=dev())
    dr = torch.zeros((B, K), dtype=torch.int32, device=dev())
    ua = torch.zeros((B, K), dtype=torch.float32, device=dev())
    us = torch.zeros((B,), dtype=torch.float32, device=dev())
    with pytest.raises(sv.SvError) as e:
        sv.spec_accept_noalloc(tl, dl, dr, ua, us, 0.6, 20, 0.95, *outs)
    assert e.value.status == 2  # SV_ERR_UNSUPPORTED, nothing launched
    assert "scratch" in str(e.value)
