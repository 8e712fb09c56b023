"""Seeded synthetic inputs for the verify-and-accept hot path.

This module is shared by the tests, the smoke check and the benchmark.  It
holds shapes and random draws only -- none of the method's arithmetic: no
dequantisation, no sampling filter, no recurrence.  Every array comes from
numpy's PCG64 seeded by (MASTER_SEED, stream id, tensor id).

Workload shapes follow the five configurations this project is measured on:
  tiny      one 4-bit linear out=512 in=256 (M=4 fp32 rows); accept over
            V=1000, K=3, B=8, logits ~ N(0, 2)
  mlp       27B-class MLP projections: gate/up 5120->17408, down 17408->5120,
            bf16 rows, M in {1,2,3,4,5,6,8}
  lmhead    LM head 5120->151936, M=4 rows per sequence, 32 sequences; draft
            logits = target logits + N(0, 0.5)
  gdn       GatedDeltaNet tape: B=16, H=48, dk=dv=128, T=5, gates in (0,1),
            L2-normalised keys, accepted prefix ~ U{0..5}
  cycle     64 layers x {q,k,v,o 5120x5120, gate/up 5120->17408,
            down 17408->5120} + LM head, M = K+1, batch 1
"""
from __future__ import annotations

import numpy as np

MASTER_SEED = 20261202

HIDDEN = 5120
INTERMEDIATE = 17408
VOCAB = 151936
N_LAYERS = 64
GDN_HEADS = 48
GDN_DIM = 128
GROUP = 64

# (name, N out, K in) of one decoder layer's projections, in execution order
LAYER_PROJECTIONS = (
    ("q", HIDDEN, HIDDEN),
    ("k", HIDDEN, HIDDEN),
    ("v", HIDDEN, HIDDEN),
    ("o", HIDDEN, HIDDEN),
    ("gate", INTERMEDIATE, HIDDEN),
    ("up", INTERMEDIATE, HIDDEN),
    ("down", HIDDEN, INTERMEDIATE),
)

SAMPLING = {"temperature": 0.6, "top_k": 20, "top_p": 0.95}
GREEDY = {"temperature": 0.0, "top_k": 0, "top_p": 1.0}


def rng(*stream: int) -> np.random.Generator:
    """PCG64 generator for a stream id tuple under the master seed."""
    return np.random.Generator(np.random.PCG64(np.random.SeedSequence([MASTER_SEED, *stream])))


def to_bf16_bits(a: np.ndarray) -> np.ndarray:
    """float32 -> bf16 bit patterns (uint16), round to nearest even (finite inputs)."""
    u = np.ascontiguousarray(a, dtype=np.float32).view(np.uint32).astype(np.uint64)
    u = (u + 0x7FFF + ((u >> 16) & 1)) >> 16
    return u.astype(np.uint16)


def bf16_bits_to_f32(h: np.ndarray) -> np.ndarray:
    """bf16 bit patterns (uint16) -> float32 (exact)."""
    return (np.asarray(h, dtype=np.uint16).astype(np.uint32) << 16).view(np.float32)


# ----------------------------------------------------------------------------
# qmv
# ----------------------------------------------------------------------------
def qmv_weights(stream: int, N: int, K: int, scale_std: float = 0.02):
    """Packed 4-bit weights (uint32 [N, K/8], every nibble uniform on 0..15) and
    bf16 scales / biases [N, K/64] ~ N(0, scale_std)."""
    g = rng(1, stream)
    w = g.integers(0, 2**32, size=(N, K // 8), dtype=np.uint64).astype(np.uint32)
    s = to_bf16_bits(g.normal(0.0, scale_std, size=(N, K // GROUP)).astype(np.float32))
    b = to_bf16_bits(g.normal(0.0, scale_std, size=(N, K // GROUP)).astype(np.float32))
    return w, s, b


def qmv_activations(stream: int, M: int, K: int, dtype: str = "bf16"):
    """Verify rows X [M, K] ~ N(0, 1): float32, or bf16 bit patterns (uint16)."""
    x = rng(2, stream).standard_normal((M, K), dtype=np.float32)
    return to_bf16_bits(x) if dtype == "bf16" else x


# ----------------------------------------------------------------------------
# verify-and-accept
# ----------------------------------------------------------------------------
def accept_logits(stream: int, B: int, K: int, V: int, sigma: float = 2.0,
                  draft_noise: float | None = None):
    """Target logits [B, K+1, V] ~ N(0, sigma); draft logits [B, K, V] are
    independent N(0, sigma) draws, or target[:, :K] + N(0, draft_noise)."""
    g = rng(3, stream)
    tl = (g.standard_normal((B, K + 1, V), dtype=np.float32) * np.float32(sigma))
    if draft_noise is None:
        dl = g.standard_normal((B, K, V), dtype=np.float32) * np.float32(sigma)
    else:
        dl = tl[:, :K, :] + g.standard_normal((B, K, V), dtype=np.float32) * np.float32(draft_noise)
    return np.ascontiguousarray(tl), np.ascontiguousarray(dl)


def accept_uniforms(stream: int, B: int, K: int):
    """u_accept [B, K] and u_sample [B], uniform on [0, 1) in float32."""
    g = rng(4, stream)
    return g.random((B, K), dtype=np.float32), g.random(B, dtype=np.float32)


def uniforms(stream: int, shape) -> np.ndarray:
    """Extra float32 uniforms on [0, 1) (e.g. for drawing draft tokens)."""
    return rng(5, stream).random(shape, dtype=np.float32)


def noise(stream: int, shape, std: float) -> np.ndarray:
    """float32 draws of N(0, std) (e.g. draft logits = target logits + noise)."""
    return (rng(8, stream).standard_normal(shape, dtype=np.float32) * np.float32(std))


# ----------------------------------------------------------------------------
# GatedDeltaNet tape
# ----------------------------------------------------------------------------
def _l2_normalise(a: np.ndarray) -> np.ndarray:
    return (a / np.linalg.norm(a, axis=-1, keepdims=True)).astype(np.float32)


def gdn_inputs(stream: int, B: int, T: int, H: int, dk: int, dv: int, state_std: float = 0.05):
    """Snapshot state0 [B,H,dv,dk] ~ N(0, state_std); q, k [B,T,H,dk] with unit
    L2 norm; v [B,T,H,dv] ~ N(0,1); alpha = exp(-softplus(N(0,1))) and
    beta = 1/(1+exp(-N(0,1))) in (0,1) [B,T,H]; n_replay [B] ~ U{0..T}."""
    g = rng(6, stream)
    s0 = (g.standard_normal((B, H, dv, dk), dtype=np.float32) * np.float32(state_std))
    q = _l2_normalise(g.standard_normal((B, T, H, dk)).astype(np.float32))
    k = _l2_normalise(g.standard_normal((B, T, H, dk)).astype(np.float32))
    v = g.standard_normal((B, T, H, dv), dtype=np.float32)
    a_raw = g.standard_normal((B, T, H))
    alpha = np.exp(-np.logaddexp(0.0, a_raw)).astype(np.float32)
    beta = (1.0 / (1.0 + np.exp(-g.standard_normal((B, T, H))))).astype(np.float32)
    n_replay = g.integers(0, T + 1, size=B).astype(np.int32)
    return {"state0": np.ascontiguousarray(s0), "q": q, "k": k, "v": v,
            "alpha": alpha, "beta": beta, "n_replay": n_replay}


# ----------------------------------------------------------------------------
# short causal convolution windows of a GatedDeltaNet layer
# ----------------------------------------------------------------------------
CONV_WIDTH = 4
CONV_CHANNELS = 3 * GDN_HEADS * GDN_DIM  # q, k, v streams of the 48 heads


def conv_inputs(stream: int, B: int, T: int, C: int, W: int = CONV_WIDTH):
    """Committed window [B, W-1, C] and verify inputs x [B, T, C] ~ N(0, 1),
    weight [W, C] ~ N(0, 1/W) (float32); n_replay [B] ~ U{0..T}."""
    g = rng(7, stream)
    window = g.standard_normal((B, W - 1, C), dtype=np.float32)
    x = g.standard_normal((B, T, C), dtype=np.float32)
    weight = (g.standard_normal((W, C), dtype=np.float32) / np.float32(np.sqrt(W)))
    n_replay = g.integers(0, T + 1, size=B).astype(np.int32)
    return {"window": window, "x": x, "weight": weight, "n_replay": n_replay}
