#!/usr/bin/env python
"""Benchmark of the verify-and-accept hot path on GB300.

Default workload (one step = one verify+accept cycle at draft depth K=3,
M=K+1=4 verify rows, batch 1, 27B-class stack, 4-bit affine g64 weights):
  per layer (64): q, k, v (5120x5120) as one qmv plan, gdn_tape_capture over
      the 4 verify tokens (48 heads, 128 x 128 fp32), o (5120x5120)
      qmv_smallm, gate, up (5120->17408) as one qmv plan, down (17408->5120)
      qmv_smallm
  then the LM head (5120->151936, a qmv plan) whose output is the target
  logits, spec_accept (temperature 0.6, top_k 20, top_p 0.95), and one
  gdn_tape_replay launch committing n_accepted + 1 tape records in all 64
  layers (n_accepted read on the device).
The cycle is captured once as a CUDA graph (programmatic dependent launch
between the qmv kernels) and replayed; its 13.84 GB weight stream is far
larger than L2, so every step streams from HBM.

Prints one JSON line.  --impl reference times the CPU oracle instead
(bounded sample of the same cycle, extrapolated).  --workload mlp | lmhead |
gdn | stream | qmv measure the MLP projections, the LM head + accept batch,
the GDN tape, the weight stream as one plan and one projection shape on
their own.
"""
from __future__ import annotations

import argparse
import json
import os
import statistics
import subprocess
import sys
import tempfile
import time
from pathlib import Path

ROOT = Path(__file__).resolve().parent
if str(ROOT) not in sys.path:
    sys.path.insert(0, str(ROOT))

import workloads as wl  # noqa: E402

METRIC = "qmv_smallm HBM GB/s (% of peak) at M=4; verify+accept cycles/s at K=3"
GROUP = 64
WEIGHT_BYTES = 0.5625  # 4-bit nibble + bf16 scale and bias per 64 weights


def roofline_rate(bandwidth_bytes_per_s: float, bytes_per_step: float) -> float:
    """Upper bound on steps per second when every step streams `bytes_per_step`
    from memory at `bandwidth_bytes_per_s` ("MTP in llama.cpp", section
    "Theoretical maximum tg t/s": decode speed <= bandwidth / active-weight
    bytes)."""
    return bandwidth_bytes_per_s / bytes_per_step


def log(*a):
    print(*a, file=sys.stderr, flush=True)


def measured_peaks():
    p = ROOT / "MEASURED_PEAKS.json"
    if p.exists():
        d = json.loads(p.read_text())
        out = {"hbm_gbs": float(d["hbm_gbs"]), "source": "measured"}
        if "bf16_tflops" in d:
            out["bf16_tflops"] = float(d["bf16_tflops"])
        return out
    return {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "source": "fallback"}


# DRAM bytes (read + written) per algorithmic byte of one qmv_plan launch,
# from the ncu capture of the 4-layer weight-stream plan (bench.py --workload
# stream --layers 4): 1.2925 GB of traffic for 1.2830 GB of algorithmic bytes.
# Re-take it whenever the plan kernel changes.
PLAN_TRAFFIC_RATIO = 1.292530 / 1.283004
E_DRAWS = 16  # seeded draft/uniform draws the end-to-end steps rotate through


def wide_bias_columns(K: int) -> int:
    """Extra MMA input columns qmv_wide spends on the bias term: the split
    group sums (2 K/64 columns) padded to whole two-group stages."""
    groups = -(-2 * (K // GROUP) // 64)
    return 64 * (-(-groups // 2) * 2)


def qmv_bytes(M: int, N: int, K: int) -> int:
    """Algorithmic bytes of one qmv_smallm call: packed nibbles, bf16 scales
    and biases, bf16 rows in, fp32 rows out."""
    return N * K // 2 + 2 * 2 * N * (K // GROUP) + 2 * M * K + 4 * M * N


# ----------------------------------------------------------------------------
# clocks during the timed region
# ----------------------------------------------------------------------------
class ClockSampler:
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.idx = gpu_index
        self.proc = None
        self.path = None

    def __enter__(self):
        fd, self.path = tempfile.mkstemp(suffix=".csv")
        os.close(fd)
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--id={self.idx}", f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "200"],
                stdout=open(self.path, "w"), stderr=subprocess.DEVNULL)
        except (FileNotFoundError, OSError):
            self.proc = None
        time.sleep(0.3)
        return self

    def __exit__(self, *exc):
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()

    def summary(self):
        if self.proc is None or self.path is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        rows = []
        for line in Path(self.path).read_text().splitlines():
            parts = [p.strip() for p in line.split(",")]
            if len(parts) >= 9:
                rows.append(parts)
        os.unlink(self.path)
        if not rows:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["no samples"]}

        def num(v):
            try:
                return float(v)
            except ValueError:
                return None

        sm = [num(r[1]) for r in rows if num(r[1]) is not None]
        mx = [num(r[2]) for r in rows if num(r[2]) is not None]
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[i] for r in rows for i in range(4) if r[5 + i] == "Active"})
        power = [num(r[3]) for r in rows if num(r[3]) is not None]
        return {"sm_mhz": statistics.median(sm) if sm else None,
                "sm_max_mhz": max(mx) if mx else None, "reasons": reasons,
                "samples": len(rows), "power_w_max": max(power) if power else None}


# ----------------------------------------------------------------------------
# the cycle on the GPU
# ----------------------------------------------------------------------------
class Cycle:
    """Device buffers and the launch sequence of one verify+accept cycle."""

    def __init__(self, sv, torch, device, depth: int = 3, layers: int = wl.N_LAYERS,
                 heads: int = wl.GDN_HEADS, dim: int = wl.GDN_DIM, seed: int = 0,
                 layout: str = "plans", weights_from=None, fused_head: bool = False):
        self.sv, self.torch, self.dev = sv, torch, device
        self.layout = layout
        # the LM head writes per-CTA top-64 lists and accept merges them (the
        # logits never go to memory); plan layouts only
        self.fused_head = fused_head and layout in ("plans", "allplans")
        self.K = depth
        self.M = depth + 1
        self.layers = layers
        self.V = wl.VOCAB
        self.heads, self.dim = heads, dim
        g = torch.Generator(device=device)
        g.manual_seed(wl.MASTER_SEED + 17 + seed)
        self.g = g
        self.proj = []  # (w, s, b, x, y)
        if weights_from is None:
            for _ in range(layers):
                for _, N, Kin in wl.LAYER_PROJECTIONS:
                    self.proj.append(self._qmv_buffers(N, Kin))
            self.lm = self._qmv_buffers(self.V, wl.HIDDEN)
        else:  # the same weights at another depth: new activation rows only
            self.proj = [self._rows_for(c) for c in weights_from.proj]
            self.lm = self._rows_for(weights_from.lm)
        self.qmv_calls = self.proj + [self.lm]
        self.qmv_bytes = sum(qmv_bytes(self.M, w.shape[0], w.shape[1] * 8)
                             for (w, _, _, _, _) in self.qmv_calls)
        self.weight_bytes = sum(int(w.numel() * 4 + s.numel() * 2 * 2)
                                for (w, s, _, _, _) in self.qmv_calls)
        # GDN: committed state of every layer, per-layer verify inputs, one tape
        T, H, d = self.M, heads, dim
        f32 = torch.float32
        self.state = torch.randn((layers, H, d, d), generator=g, device=device, dtype=f32) * 0.05

        def unit(shape):
            a = torch.randn(shape, generator=g, device=device, dtype=f32)
            return (a / a.norm(dim=-1, keepdim=True)).contiguous()

        self.gq = [unit((1, T, H, d)) for _ in range(layers)]
        self.gk = [unit((1, T, H, d)) for _ in range(layers)]
        self.gv = [torch.randn((1, T, H, d), generator=g, device=device, dtype=f32)
                   for _ in range(layers)]
        self.galpha = [torch.exp(-torch.nn.functional.softplus(
            torch.randn((1, T, H), generator=g, device=device, dtype=f32))) for _ in range(layers)]
        self.gbeta = [torch.sigmoid(torch.randn((1, T, H), generator=g, device=device, dtype=f32))
                      for _ in range(layers)]
        self.gout = [torch.empty((1, T, H, d), device=device, dtype=f32) for _ in range(layers)]
        blk = sv.gdn_tape_bytes(1, T, H, d, d) // 4
        self.tape = torch.empty(layers * blk, device=device, dtype=f32)
        self.tapes = [self.tape[i * blk:(i + 1) * blk] for i in range(layers)]
        self.gdn_bytes = layers * (H * d * d * 4            # capture reads the snapshot
                                   + T * H * (3 * d + 2) * 4  # q, k, v, alpha, beta
                                   + T * H * d * 4            # outputs
                                   + blk * 4)                 # tape
        # accept: target logits = LM-head output [K+1, V] = [1][K+1][V]
        self.target = self.lm[4].view(1, self.M, self.V)
        self.draft = torch.zeros((1, self.K, self.V), device=device, dtype=f32)
        # the step's small inputs (draft tokens, u_accept, u_sample) and
        # outputs (tokens, accepted count, flags) each in one 4-byte-word
        # buffer, so that a step moves them with one copy each way
        K = self.K
        self.small_in = torch.zeros((2 * K + 1,), device=device, dtype=torch.int32)
        self.draft_tokens = self.small_in[:K].view(1, K)
        self.ua = self.small_in[K:2 * K].view(torch.float32).view(1, K)
        self.us = self.small_in[2 * K:].view(torch.float32)
        ua, us = wl.accept_uniforms(99 + seed, 1, K)
        self.ua.copy_(torch.from_numpy(ua))
        self.us.copy_(torch.from_numpy(us))
        self.ws = sv.make_accept_workspace(1, self.K, self.V, device)
        self.topk = sv.make_topk_lists(self.M, torch.bfloat16, device) if self.fused_head else None
        self.small_out = torch.empty((self.M + 2,), device=device, dtype=torch.int32)
        self.out_tokens = self.small_out[:self.M].view(1, self.M)
        self.n_acc = self.small_out[self.M:self.M + 1]
        self.flags = self.small_out[self.M + 1:]
        self.plans = []
        if layout in ("plans", "allplans"):
            self._make_plans()
        self.qmv_launches = (len(self.plans) + (layers if layout == "plans" else 0)
                             if self.plans else len(self.qmv_calls))
        # + the GatedDeltaNet captures, the replay, and spec_accept: a chunk
        # kernel and a finish kernel on the logits, one kernel on fused lists
        self.launches_per_step = self.qmv_launches + layers + 1 + (1 if self.fused_head else 2)

    def _make_plans(self):
        """Per layer: one plan for q, k, v and one for gate, up (projections
        that read the same input), down as a one-problem plan and o as a
        qmv_smallm launch ("plans"; o follows the GatedDeltaNet capture, whose
        small CTAs leave room for qmv_smallm's to start early), or o as a plan
        too ("allplans"); the LM head as a plan.  Between them sit the
        dependency points of a decoder layer (the GatedDeltaNet capture, then
        o, then down), so each is its own launch, overlapped with its
        predecessor by programmatic dependent launch."""
        QmvPlan = self.sv.QmvPlan
        names = [n for n, _, _ in wl.LAYER_PROJECTIONS]
        n = len(names)
        groups = ((("q", "k", "v"), ("gate", "up"), ("down",)) if self.layout == "plans" else
                  (("q", "k", "v"), ("o",), ("gate", "up"), ("down",)))
        for layer in range(self.layers):
            by = dict(zip(names, self.proj[layer * n:(layer + 1) * n]))
            for grp in groups:
                self.plans.append(QmvPlan([tuple(by[k][:5]) + (False,) for k in grp]))
        if self.fused_head:
            self.plans.append(QmvPlan([tuple(self.lm[:4]) + (None, False, self.topk)]))
            self.head_grid = self.plans[-1].grid
        else:
            self.plans.append(QmvPlan([tuple(self.lm[:5]) + (False,)]))
        self.plan_bytes = sum(qmv_bytes(self.M, w.shape[0], w.shape[1] * 8)
                              for pl in self.plans for (w, *_rest) in pl.problems)
        if self.fused_head:  # the head writes its lists, not M x V logits
            self.plan_bytes += self.topk.numel() - 4 * self.M * self.V

    def _qmv_buffers(self, N, Kin):
        t, g, d = self.torch, self.g, self.dev
        w = t.randint(-(2 ** 31), 2 ** 31 - 1, (N, Kin // 8), generator=g, device=d,
                      dtype=t.int32)
        s = (t.randn((N, Kin // GROUP), generator=g, device=d) * 0.02).to(t.bfloat16)
        b = (t.randn((N, Kin // GROUP), generator=g, device=d) * 0.02).to(t.bfloat16)
        x = t.randn((self.M, Kin), generator=g, device=d).to(t.bfloat16)
        y = t.empty((self.M, N), device=d, dtype=t.float32)
        return (w, s, b, x, y)

    def _rows_for(self, c):
        t = self.torch
        w, s, b = c[:3]
        Kin = w.shape[1] * 8
        x = t.randn((self.M, Kin), generator=self.g, device=self.dev).to(t.bfloat16)
        return (w, s, b, x, t.empty((self.M, w.shape[0]), device=self.dev, dtype=t.float32))

    def prepare_drafts(self, noise: float = 0.5, logit_std: float = 3.0):
        """Once, outside timing: the LM-head input is scaled so that the target
        logits have standard deviation `logit_std` (3: about 70 % of drafts
        accepted per position at T = 0.6, top-k 20, top-p 0.95); draft logits
        = target logits + N(0, noise); drafts = the top token of each row."""
        t = self.torch
        self.run_qmv(self.lm)
        t.cuda.synchronize()
        x = self.lm[3]
        x.copy_((x.float() * (logit_std / float(self.target.std()))).to(x.dtype))
        self.run_qmv(self.lm)
        t.cuda.synchronize()
        z = self.target[:, : self.K].clone()
        z += t.randn(z.shape, generator=self.g, device=self.dev) * noise
        self.draft.copy_(z)
        self.draft_tokens.copy_(self.sample_draft_tokens(1)[0])

    def sample_draft_tokens(self, n: int):
        """n independent draft-token sets [n, 1, K] (int32), each drawn from the
        filtered draft distributions q (T 0.6, top-k 20, top-p 0.95), as the
        ratio test assumes."""
        t = self.torch
        top, idx = (self.draft[0] / 0.6).topk(20, dim=-1)
        q = t.softmax(top, dim=-1)
        keep = (q.cumsum(-1) - q) < 0.95
        q = t.where(keep, q, t.zeros_like(q))
        pick = t.multinomial(q / q.sum(-1, keepdim=True), n, replacement=True,
                             generator=self.g)                      # [K, n]
        return idx.gather(-1, pick).t().reshape(n, 1, self.K).to(t.int32).contiguous()

    def run_qmv(self, c):
        w, s, b, x, y = c
        self.sv.qmv_smallm(w, s, b, x, y)

    def run(self):
        """One cycle: per layer q, k, v -> GatedDeltaNet capture over the
        verify tokens -> o -> gate, up -> down; LM head; spec_accept; one
        tape replay committing the accepted prefix in every layer."""
        self._forward(with_gdn=True)
        self._accept()
        self.sv.gdn_tape_replay(self.state, self.tape, self.n_acc, self.M, n_replay_bias=1)

    def _accept(self):
        if self.fused_head:
            self.sv.spec_accept_lists(self.topk, self.head_grid, self.V, self.draft,
                                      self.draft_tokens, self.ua, self.us, 0.6, 20, 0.95,
                                      workspace=self.ws, out_tokens=self.out_tokens,
                                      n_accepted=self.n_acc, err_flags=self.flags)
        else:
            self.sv.spec_accept(self.target, self.draft, self.draft_tokens, self.ua, self.us,
                                0.6, 20, 0.95, workspace=self.ws, out_tokens=self.out_tokens,
                                n_accepted=self.n_acc, err_flags=self.flags)

    def run_stream_accept(self):
        """The cycle as the weight-stream configuration lists it: every
        projection of every layer, the LM head and spec_accept (no
        GatedDeltaNet tape capture or replay)."""
        self._forward(with_gdn=False)
        self._accept()

    def run_qmv_only(self):
        self._forward(with_gdn=False)

    def run_plans_only(self):
        for pl in self.plans:
            pl.run()

    def _gdn(self, layer):
        self.sv.gdn_tape_capture(self.state[layer:layer + 1], self.gq[layer], self.gk[layer],
                                 self.gv[layer], self.galpha[layer], self.gbeta[layer],
                                 tape=self.tapes[layer], out=self.gout[layer])

    def _forward(self, with_gdn):
        n = len(wl.LAYER_PROJECTIONS)
        for layer in range(self.layers):
            if self.layout == "plans":
                by = dict(zip([m for m, _, _ in wl.LAYER_PROJECTIONS],
                              self.proj[layer * n:(layer + 1) * n]))
                self.plans[3 * layer].run()           # q, k, v
                if with_gdn:
                    self._gdn(layer)
                self.run_qmv(by["o"])
                self.plans[3 * layer + 1].run()       # gate, up
                self.plans[3 * layer + 2].run()       # down
            elif self.layout == "allplans":
                self.plans[4 * layer].run()           # q, k, v
                if with_gdn:
                    self._gdn(layer)
                for i in range(1, 4):                 # o; gate, up; down
                    self.plans[4 * layer + i].run()
            else:
                c = self.proj[layer * n:(layer + 1) * n]
                for i in range(3):  # q, k, v
                    self.run_qmv(c[i])
                if with_gdn:
                    self._gdn(layer)
                for i in range(3, n):  # o, gate, up, down
                    self.run_qmv(c[i])
        if self.plans:
            self.plans[-1].run()
        else:
            self.run_qmv(self.lm)


def capture(torch, fn, stream):
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.stream(stream):
        fn()
        fn()
    torch.cuda.synchronize()
    with torch.cuda.graph(graph, stream=stream):
        fn()
    torch.cuda.synchronize()
    return graph


def time_graph(torch, graph, stream, steps: int, warmup: int, barrier=None):
    with torch.cuda.stream(stream):
        for _ in range(warmup):
            graph.replay()
    torch.cuda.synchronize()
    if barrier:
        barrier()
    start = torch.cuda.Event(enable_timing=True)
    end = torch.cuda.Event(enable_timing=True)
    with torch.cuda.stream(stream):
        start.record(stream)
        for _ in range(steps):
            graph.replay()
        end.record(stream)
    torch.cuda.synchronize()
    if barrier:
        barrier()
    return start.elapsed_time(end)


# ----------------------------------------------------------------------------
# CPU oracle on a bounded sample of the cycle
# ----------------------------------------------------------------------------
def oracle_cycle_sample(depth: int = 3, layer_fraction: float = 1.0, repeats: int = 8,
                        lm_fraction: float = 1.0 / 8, head_fraction: float = 1.0,
                        threads: int | None = None):
    """Times the oracle on a sample of one cycle and extrapolates to a full
    cycle: `layer_fraction` of the rows of one layer's seven projections, run
    `repeats` times (x64/repeats layers), `lm_fraction` of the LM-head rows,
    spec_accept at batch 1 on the full vocabulary, and GDN capture + replay on
    `head_fraction` of one layer's heads (x64 layers), on `threads` host
    threads (default: every core this process may use).  Returns (seconds per
    cycle, sample text, threads)."""
    import numpy as np

    import oracle

    oracle.build()
    threads = oracle.set_threads(threads or len(os.sched_getaffinity(0)))
    M = depth + 1
    t_qmv = 0.0
    for j, (_, N, Kin) in enumerate(wl.LAYER_PROJECTIONS):
        n = max(16, int(N * layer_fraction))
        w, s, b = wl.qmv_weights(700 + j, n, Kin)
        x = wl.qmv_activations(700 + j, M, Kin, "bf16")
        t0 = time.perf_counter()
        for _ in range(repeats):
            oracle.qmv(w, s, b, x)
        t_qmv += (time.perf_counter() - t0) / repeats * (N / n) * wl.N_LAYERS
    n = max(16, int(wl.VOCAB * lm_fraction))
    w, s, b = wl.qmv_weights(720, n, wl.HIDDEN)
    x = wl.qmv_activations(720, M, wl.HIDDEN, "bf16")
    t0 = time.perf_counter()
    logits = oracle.qmv(w, s, b, x)
    t_lm = (time.perf_counter() - t0) * (wl.VOCAB / n)
    tl, dl = wl.accept_logits(721, 1, depth, wl.VOCAB, sigma=3.0, draft_noise=0.5)
    tl[0, :, :n] = logits  # the sampled rows stand in for part of the vocabulary
    dr = np.argmax(dl, axis=2).astype(np.int32)
    ua, us = wl.accept_uniforms(721, 1, depth)
    t0 = time.perf_counter()
    r = oracle.spec_accept(tl, dl, dr, ua, us, float(np.float32(0.6)), 20,
                           float(np.float32(0.95)))
    t_acc = time.perf_counter() - t0
    H = max(1, int(wl.GDN_HEADS * head_fraction))
    g = wl.gdn_inputs(722, 1, M, H, wl.GDN_DIM, wl.GDN_DIM)
    t0 = time.perf_counter()
    _, tape = oracle.gdn_capture(g["state0"], g["q"], g["k"], g["v"], g["alpha"], g["beta"])
    oracle.gdn_replay(g["state0"], tape, np.array([int(r["n_accepted"][0]) + 1], np.int32))
    t_gdn = (time.perf_counter() - t0) * (wl.GDN_HEADS / H) * wl.N_LAYERS
    total = t_qmv + t_lm + t_acc + t_gdn
    sample = (f"oracle on {layer_fraction:g} of the rows of one layer's 7 projections run "
              f"{repeats}x (scaled to 64 layers), {lm_fraction:g} of the LM-head rows, "
              f"spec_accept at batch 1 over the full vocabulary, GDN capture+replay on {H} of "
              f"48 heads of one layer (x64); extrapolated to one full cycle")
    return total, sample, threads


# ----------------------------------------------------------------------------
def dist_env():
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return world, rank, local


def max_over_ranks(torch, seconds: float, world: int, device) -> float:
    """The slowest rank's time (replicas: the job ends when the last one does);
    `seconds` itself on one rank.  All ranks call it."""
    if world <= 1:
        return seconds
    import torch.distributed as dist

    t = torch.tensor([seconds], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def job_rate(units_per_rank: int, world: int, slowest_seconds: float) -> float:
    """Whole-job throughput of `world` replicas, each doing `units_per_rank`
    units: every rank's units over the slowest rank's time (weak scaling)."""
    return units_per_rank * world / slowest_seconds


def run_reference(args):
    """The reference arm: the CPU oracle on the host cores, one bounded
    sample of the cycle per step.  `ms_per_step` is the wall time a sample
    actually took; `value` is the sample's time extrapolated to a full cycle
    (`extrapolated`: true, the scale in `extrapolation`)."""
    world, rank, _ = dist_env()
    if rank != 0:
        return 0
    fractions = dict(layer_fraction=1.0, repeats=1, lm_fraction=1.0 / 64, head_fraction=0.25)
    for _ in range(args.warmup):
        oracle_cycle_sample(args.depth, **fractions)
    per_cycle, wall = [], []
    sample = ""
    threads = 1
    for _ in range(args.steps):
        t0 = time.perf_counter()
        s, sample, threads = oracle_cycle_sample(args.depth, **fractions)
        wall.append(time.perf_counter() - t0)
        per_cycle.append(s)
    t_cycle = statistics.mean(per_cycle)
    t_wall = statistics.mean(wall)
    value = 1.0 / t_cycle
    line = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": "cycles/s",
        "n_gpus": args.gpus, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": t_wall * 1e3, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": cycle_config(args.depth, "plans", world),
        "extrapolated": True,
        "extrapolation": {"seconds_per_sample": t_wall,
                          "seconds_per_cycle_extrapolated": t_cycle,
                          "cycle_per_sample": t_cycle / t_wall,
                          "fractions": fractions,
                          "how": "each step times the oracle on a bounded sample of one cycle "
                                 "(the fractions above of the projections' rows, the LM head "
                                 "and the GatedDeltaNet heads, spec_accept in full); the "
                                 "sample's parts are scaled to a whole cycle"},
        "cpu_baseline": {"value": value, "unit": "cycles/s", "cores": threads,
                         "kind": "oracle", "sample": sample},
        "e2e": {"value": value, "unit": "cycles/s", "h2d_bytes_per_step": 0,
                "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)
    return 0


def workload_name(depth):
    return (f"27B-class verify+accept cycle: draft depth K={depth} (M={depth + 1} verify rows), "
            f"batch 1; 64 layers x {{q,k,v,o 5120x5120; gate,up 5120->17408; down "
            f"17408->5120}} 4-bit affine g64 + GDN tape capture (48 heads, 128x128 fp32) per "
            f"layer; LM head 5120->151936; spec_accept (T=0.6, top_k=20, top_p=0.95); "
            f"one GDN tape replay over all 64 layers")


def cycle_bytes_static(depth: int) -> tuple[int, int]:
    """(weight bytes, algorithmic bytes) of one cycle at draft depth `depth`,
    from the shapes alone: every projection and the LM head (4-bit nibbles,
    bf16 scale and bias per 64, bf16 rows in, fp32 rows out) plus the
    GatedDeltaNet tape work of every layer (snapshot read, verify inputs,
    outputs, tape)."""
    M = depth + 1
    shapes = [(N, K) for _ in range(wl.N_LAYERS) for _, N, K in wl.LAYER_PROJECTIONS]
    shapes.append((wl.VOCAB, wl.HIDDEN))
    weight = sum(N * K // 2 + 2 * 2 * N * (K // GROUP) for N, K in shapes)
    qmv = sum(qmv_bytes(M, N, K) for N, K in shapes)
    T, H, d = M, wl.GDN_HEADS, wl.GDN_DIM
    tape = 4 * (T * H * 2 * d + 4 * ((T * H + 3) // 4))
    gdn = wl.N_LAYERS * (H * d * d * 4 + T * H * (3 * d + 2) * 4 + T * H * d * 4 + tape)
    return weight, qmv + gdn


def cycle_config(depth: int, layout: str = "plans", world: int = 1) -> dict:
    """The workload description both arms of the benchmark print."""
    weight, algo = cycle_bytes_static(depth)
    return {"workload": workload_name(depth), "depth_K": depth, "M": depth + 1, "batch": 1,
            "layers": wl.N_LAYERS, "weight_bytes_per_cycle": weight,
            "algorithmic_bytes_per_cycle": algo,
            "l2": "inputs larger than L2 (13.8 GB weight stream per step)",
            "graph": "one CUDA graph per cycle, PDL between qmv launches",
            "layout": layout,
            "arithmetic": "4-bit weights x bf16 rows on bf16 MMA, fp32 accumulate; "
                          "accept and GDN in fp32",
            "parallelism": "replicas" if world > 1 else "single GPU"}


def run_cycle(args):
    import numpy as np
    import torch

    import mtp_speculative_decoding_qmv_gb300 as sv

    world, rank, local = dist_env()
    if world > 1:
        import torch.distributed as dist

        torch.cuda.set_device(local)
        dist.init_process_group("nccl", device_id=torch.device("cuda", local))
    device = torch.device("cuda", local if world > 1 else 0)
    torch.cuda.set_device(device)

    def barrier():
        if world > 1:
            import torch.distributed as dist

            dist.barrier()

    cpu = cpu1 = None
    if rank == 0 and not args.no_cpu_baseline:
        t, sample, threads = oracle_cycle_sample(args.depth)
        cpu = {"value": 1.0 / t, "unit": "cycles/s", "cores": threads, "kind": "oracle",
               "sample": sample}
        log(f"cpu oracle: {t:.2f} s per cycle (extrapolated) on {threads} threads")
        # the same oracle on one thread, on a smaller sample (about the same
        # wall time)
        t1, sample1, _ = oracle_cycle_sample(args.depth, layer_fraction=1.0 / 4, repeats=1,
                                             lm_fraction=1.0 / 32, head_fraction=0.25,
                                             threads=1)
        cpu1 = {"value": 1.0 / t1, "unit": "cycles/s", "cores": 1, "kind": "oracle",
                "sample": sample1}
        log(f"cpu oracle: {t1:.2f} s per cycle (extrapolated) on 1 thread")

    sv.set_pdl(True)
    cyc = Cycle(sv, torch, device, depth=args.depth, seed=rank, layout=args.layout,
                fused_head=args.lm_head == "fused")
    cyc.prepare_drafts()
    stream = torch.cuda.Stream(device)
    graph = capture(torch, cyc.run, stream)
    qgraph = capture(torch, cyc.run_qmv_only, stream)
    sv.device_status()

    with ClockSampler(device.index if device.index is not None else 0) as clk:
        ms = time_graph(torch, graph, stream, args.steps, args.warmup, barrier)
    clocks = clk.summary()
    per_step_ms = ms / args.steps
    ms = max_over_ranks(torch, ms / 1e3, world, device) * 1e3
    total_cycles = args.steps * world
    value = job_rate(args.steps, world, ms / 1e3)

    # the dominant kernel: the cycle's qmv launches (plans or single
    # projections) as their own graph
    qms = time_graph(torch, qgraph, stream, args.steps, 3)
    qmv_all_gbs = cyc.qmv_bytes / (qms / 1e3 / args.steps) / 1e9
    if cyc.plans:
        # qmv_plan launches (q,k,v, gate,up and down of every layer -- with o
        # too for "allplans" -- and the LM head) in cycle order as their own
        # graph
        pgraph = capture(torch, cyc.run_plans_only, stream)
        pms = time_graph(torch, pgraph, stream, args.steps, 3)
        del pgraph
        n_q, q_bytes, q_ms = len(cyc.plans), cyc.plan_bytes, pms
    else:
        n_q, q_bytes, q_ms = cyc.qmv_launches, cyc.qmv_bytes, qms
    per_launch_s = q_ms / 1e3 / (args.steps * n_q)
    bytes_per_launch = q_bytes / n_q
    achieved = bytes_per_launch / per_launch_s / 1e9
    peaks = measured_peaks()
    # the whole weight stream of the cycle (every projection and the LM head,
    # M rows each) as one plan without waits: the qmv kernel's streaming rate
    stream_plan = sv.QmvPlan([tuple(c[:5]) + (False,) for c in cyc.qmv_calls])
    sgraph = capture(torch, stream_plan.run, stream)
    sms = time_graph(torch, sgraph, stream, args.steps, 3) / args.steps
    stream_gbs = cyc.qmv_bytes / (sms / 1e3) / 1e9
    del sgraph
    stream_plan.close()

    # end to end through the API: drafts/uniforms in from pinned host memory,
    # tokens and accepted length back, every step.  Each step takes the next
    # of E_DRAWS seeded draws of draft tokens and uniforms (a decode loop
    # draws both afresh every cycle), so the accepted lengths reported are a
    # sample mean, not one fixed draw.
    h_draft = cyc.draft.cpu().pin_memory()
    tokens = cyc.sample_draft_tokens(E_DRAWS).cpu().reshape(E_DRAWS, cyc.K)
    uni = [wl.accept_uniforms(1000 + 97 * rank + i, 1, cyc.K) for i in range(E_DRAWS)]
    # per draw, the step's small inputs packed as the device buffer holds them
    h_small = torch.empty((E_DRAWS, 2 * cyc.K + 1), dtype=torch.int32).pin_memory()
    for i, (ua_i, us_i) in enumerate(uni):
        h_small[i, :cyc.K] = tokens[i]
        h_small[i, cyc.K:].view(torch.float32).copy_(
            torch.from_numpy(np.concatenate([ua_i.reshape(-1), us_i.reshape(-1)])))
    h_out = torch.empty_like(cyc.small_out, device="cpu").pin_memory()
    h2d = h_small[0].numel() * 4 + h_draft.numel() * h_draft.element_size()
    d2h = h_out.numel() * 4
    accepted = []

    def e2e_step():
        i = len(accepted) % E_DRAWS
        with torch.cuda.stream(stream):
            cyc.draft.copy_(h_draft, non_blocking=True)
            cyc.small_in.copy_(h_small[i], non_blocking=True)
            graph.replay()
            h_out.copy_(cyc.small_out, non_blocking=True)
        stream.synchronize()
        accepted.append(int(h_out[cyc.M]))

    for _ in range(args.warmup):
        e2e_step()
    barrier()
    t0 = time.perf_counter()
    for _ in range(args.steps):
        e2e_step()
    t_e2e = time.perf_counter() - t0
    barrier()
    t_e2e = max_over_ranks(torch, t_e2e, world, device)
    sv.device_status()

    # the cycle as the weight-stream configuration lists it (projections, LM
    # head, spec_accept; no GatedDeltaNet tape), for comparison
    ngraph = capture(torch, cyc.run_stream_accept, stream)
    nms = time_graph(torch, ngraph, stream, args.steps, args.warmup, barrier)
    nms = max_over_ranks(torch, nms / 1e3, world, device) * 1e3
    no_tape = job_rate(args.steps, world, nms / 1e3)
    del ngraph

    # the same cycle at the configuration's other draft depths (same weights,
    # M = K + 1 rows), each its own graph, timed the same way
    depths = {str(args.depth): value}
    if not args.no_depth_sweep:
        for k in (2, 3, 4, 5):
            if k == args.depth:
                continue
            other = Cycle(sv, torch, device, depth=k, seed=rank, layout=args.layout,
                          fused_head=args.lm_head == "fused",
                          weights_from=cyc)
            other.prepare_drafts()
            og = capture(torch, other.run, stream)
            oms = time_graph(torch, og, stream, args.steps, args.warmup, barrier)
            oms = max_over_ranks(torch, oms / 1e3, world, device) * 1e3
            depths[str(k)] = job_rate(args.steps, world, oms / 1e3)
            del og, other
        sv.device_status()

    launches_per_step = cyc.launches_per_step
    has_plans, qmv_launches = bool(cyc.plans), cyc.qmv_launches
    cyc_qmv_bytes, n_qmv_calls = cyc.qmv_bytes, len(cyc.qmv_calls)
    # the other configurations of the workload, each measured on its own in
    # the same run (rank 0; the cycle's buffers are released first)
    configs, near_ties = None, None
    if rank == 0 and not args.no_configs:
        del graph, qgraph
        cyc_bytes = (cyc.weight_bytes, cyc.qmv_bytes + cyc.gdn_bytes)
        del cyc
        torch.cuda.empty_cache()
        cfg_steps = min(args.steps, 5)
        configs = {
            "mlp_projections": mlp_rates(torch, sv, cfg_steps, 3),
            "lm_head_accept_batch32": lmhead_rates(torch, sv, args.depth, cfg_steps, 3),
            "gdn_tape_batch16": gdn_rates(torch, sv, cfg_steps, 3),
        }
        if not args.no_cpu_baseline:
            # near ties of the accept decisions, from the float64 oracle (CPU leg)
            near_ties = accept_near_ties(torch, sv, args.depth)
    else:
        cyc_bytes = (cyc.weight_bytes, cyc.qmv_bytes + cyc.gdn_bytes)
    if rank != 0:
        return 0
    if cyc_bytes != cycle_bytes_static(args.depth):
        log(f"warning: cycle bytes {cyc_bytes} differ from the static count "
            f"{cycle_bytes_static(args.depth)}")
    cycle_bytes = cyc_bytes[1]
    line = {
        "metric": METRIC, "value": value, "unit": "cycles/s", "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": per_step_ms,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
        "dtype": "bf16", "data": "synthetic",
        "config": cycle_config(args.depth, args.layout, world),
        "cycle_gb_per_s": cycle_bytes / (per_step_ms / 1e3) / 1e9,
        "roofline": {"kernel": "qmv_plan" if has_plans else "qmv_smallm",
                     "bound": "hbm", "achieved": achieved,
                     "peak": peaks["hbm_gbs"], "unit": "GB/s",
                     "frac": achieved / peaks["hbm_gbs"],
                     "traffic": (bytes_per_launch * PLAN_TRAFFIC_RATIO
                                 if has_plans else None),
                     "traffic_source": ("ncu dram__bytes_read.sum + dram__bytes_write.sum of "
                                        "one 4-layer weight-stream plan launch, scaled to this "
                                        "launch size by algorithmic bytes"
                                        if has_plans else None),
                     "peak_source": peaks["source"],
                     "bytes_per_launch": bytes_per_launch,
                     "launch_us": per_launch_s * 1e6,
                     "how": f"the cycle's {n_q} launches of this kernel (M={args.depth + 1}) "
                            f"in cycle order captured as their own graph, CUDA events over "
                            f"{args.steps} replays on the launching stream"},
        "qmv_all": {"value": qmv_all_gbs, "unit": "GB/s", "frac": qmv_all_gbs / peaks["hbm_gbs"],
                    "launches": qmv_launches,
                    "how": "every qmv launch of the cycle (plans and single projections) in "
                           "cycle order as one graph"},
        "qmv_stream": {"value": stream_gbs, "unit": "GB/s", "frac": stream_gbs / peaks["hbm_gbs"],
                       "ms": sms, "bytes": cyc_qmv_bytes,
                       "how": f"all {n_qmv_calls} projections of the cycle (27B-class "
                              f"weight stream, M={args.depth + 1}) as one qmv plan without "
                              f"waits, CUDA events over {args.steps} graph replays"},
        "cycle_roofline": {
            "bound_cycles_per_s": roofline_rate(peaks["hbm_gbs"] * 1e9, cycle_bytes),
            "frac": value / world / roofline_rate(peaks["hbm_gbs"] * 1e9, cycle_bytes),
            "how": "measured HBM bandwidth / algorithmic bytes of one cycle (weights, "
                   "activations, GDN state and tape)"},
        "cpu_baseline": cpu,
        "cpu_baseline_1thread": cpu1,
        "e2e": {"value": total_cycles / t_e2e, "unit": "cycles/s",
                "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h},
        "gpu_launches": launches_per_step * args.steps,
        "clocks": clocks,
        "cycles_per_s_by_depth": {k: depths[k] for k in sorted(depths)},
        "cycles_per_s_without_gdn_tape": no_tape,
        "configs": configs,
        "accept_near_ties": near_ties,
        "acceptance": {"mean_accepted": statistics.mean(accepted) if accepted else None,
                       "depth": args.depth, "draws": min(len(accepted), E_DRAWS),
                       "how": "accepted drafts per cycle over the e2e steps (warm-up "
                              "included), each step a fresh seeded draw of draft "
                              "tokens and uniforms"},
    }
    print(json.dumps(line), flush=True)
    if world > 1:
        import torch.distributed as dist

        dist.destroy_process_group()
    return 0


# ----------------------------------------------------------------------------
# single-config measurements (not the default step)
# ----------------------------------------------------------------------------
def mlp_rates(torch, sv, steps: int, warmup: int, Ms=(1, 2, 3, 4, 5, 6, 8)) -> dict:
    """Configuration 2: the 27B-class MLP verify projections (gate, up
    5120->17408, down 17408->5120), 64 sequences back to back on their own
    weight copies (9.6 GB > L2), per M: as one qmv plan and as separate
    qmv_smallm launches, GB/s against the measured peak and 8 TB/s."""
    dev = torch.device("cuda", 0)
    sv.set_pdl(True)
    g = torch.Generator(device=dev)
    g.manual_seed(wl.MASTER_SEED + 23)
    seqs = 64
    shapes = [(wl.INTERMEDIATE, wl.HIDDEN), (wl.INTERMEDIATE, wl.HIDDEN),
              (wl.HIDDEN, wl.INTERMEDIATE)]
    weights = []
    for _ in range(seqs):
        for N, K in shapes:
            w = torch.randint(-(2 ** 31), 2 ** 31 - 1, (N, K // 8), generator=g, device=dev,
                              dtype=torch.int32)
            s_ = (torch.randn((N, K // GROUP), generator=g, device=dev) * 0.02).to(torch.bfloat16)
            b_ = (torch.randn((N, K // GROUP), generator=g, device=dev) * 0.02).to(torch.bfloat16)
            weights.append((w, s_, b_))
    stream = torch.cuda.Stream(dev)
    per_m, per_m_launch = {}, {}
    for M in Ms:
        xs = {K: torch.randn((M, K), generator=g, device=dev).to(torch.bfloat16)
              for K in (wl.HIDDEN, wl.INTERMEDIATE)}
        ys = [torch.empty((M, w.shape[0]), device=dev) for (w, _, _) in weights]

        def fn():
            for (w, s_, b_), y in zip(weights, ys):
                sv.qmv_smallm(w, s_, b_, xs[w.shape[1] * 8], y)

        nbytes = sum(qmv_bytes(M, w.shape[0], w.shape[1] * 8) for (w, _, _) in weights)
        graph = capture(torch, fn, stream)
        ms = time_graph(torch, graph, stream, steps, warmup)
        per_m_launch[M] = nbytes / (ms / 1e3 / steps) / 1e9
        del graph
        # the same 192 projections as one qmv plan (no dependency points)
        plan = sv.QmvPlan([(w, s_, b_, xs[w.shape[1] * 8], y, False)
                           for (w, s_, b_), y in zip(weights, ys)])
        graph = capture(torch, plan.run, stream)
        ms = time_graph(torch, graph, stream, steps, warmup)
        per_m[M] = nbytes / (ms / 1e3 / steps) / 1e9
        del graph
        plan.close()
        log(f"M={M}: plan {per_m[M]:.0f} GB/s, separate launches {per_m_launch[M]:.0f} GB/s")
    sv.device_status()
    del weights
    peak = measured_peaks()["hbm_gbs"]
    return {"unit": "GB/s",
            "per_M_gbs": per_m,
            "per_M_frac": {m: v / peak for m, v in per_m.items()},
            "per_M_frac_of_8tbs_nominal": {m: v / 8000.0 for m, v in per_m.items()},
            "per_M_gbs_separate_launches": per_m_launch,
            "per_M_frac_separate_launches": {m: v / peak for m, v in per_m_launch.items()},
            "per_M_frac_of_8tbs_nominal_separate_launches":
                {m: v / 8000.0 for m, v in per_m_launch.items()},
            "how": "64 sequences x {gate, up 5120->17408; down 17408->5120} on distinct weight "
                   "copies (9.6 GB), bf16 rows ~N(0,1): one qmv plan per M, and the same 192 "
                   "projections as separate qmv_smallm launches; CUDA events over graph "
                   f"replays ({steps} timed, {warmup} warm-up)"}


def run_mlp(args):
    """27B-class MLP verify projections: gate/up 5120->17408, down 17408->5120,
    64 sequences back to back, each on its own weight copies (9.6 GB > L2),
    for M in 1..8 except 7; qmv_smallm GB/s per M."""
    import torch

    import mtp_speculative_decoding_qmv_gb300 as sv

    r = mlp_rates(torch, sv, args.steps, args.warmup)
    peaks = measured_peaks()
    line = {"metric": METRIC, "value": r["per_M_gbs"][4], "unit": "GB/s", "n_gpus": 1,
            "steps": args.steps, "warmup": args.warmup, "higher_is_better": True,
            "vs_baseline": None, "dtype": "bf16", "data": "synthetic",
            "config": {"workload": "27B-class MLP verify projections: 64 sequences x "
                                   "{gate, up 5120->17408; down 17408->5120}, distinct weight "
                                   "copies (9.6 GB), one qmv plan per M",
                       "l2": "inputs larger than L2"},
            **{k: v for k, v in r.items() if k not in ("unit", "how")},
            "peak": peaks}
    print(json.dumps(line), flush=True)
    return 0


def run_qmv(args):
    """One projection shape (--shape N K) at M = depth + 1, on enough distinct
    weight copies that they stream from HBM (> 300 MB in all), in one CUDA
    graph without PDL; qmv_smallm GB/s.  Also the small case the ncu captures
    of a single qmv_smallm launch run."""
    import torch

    import mtp_speculative_decoding_qmv_gb300 as sv

    dev = torch.device("cuda", 0)
    N, K = args.shape
    M = args.depth + 1
    g = torch.Generator(device=dev)
    g.manual_seed(wl.MASTER_SEED + 37)
    per = qmv_bytes(M, N, K)
    copies = max(4, -(-300_000_000 // per))
    weights = []
    for _ in range(copies):
        w = torch.randint(-(2 ** 31), 2 ** 31 - 1, (N, K // 8), generator=g, device=dev,
                          dtype=torch.int32)
        s_ = (torch.randn((N, K // GROUP), generator=g, device=dev) * 0.02).to(torch.bfloat16)
        b_ = (torch.randn((N, K // GROUP), generator=g, device=dev) * 0.02).to(torch.bfloat16)
        weights.append((w, s_, b_))
    x = torch.randn((M, K), generator=g, device=dev).to(torch.bfloat16)
    y = torch.empty((M, N), device=dev)

    def fn():
        for w, s_, b_ in weights:
            sv.qmv_smallm(w, s_, b_, x, y)

    stream = torch.cuda.Stream(dev)
    graph = capture(torch, fn, stream)
    ms = time_graph(torch, graph, stream, args.steps, args.warmup)
    us = ms / args.steps / copies * 1e3
    gbs = per / (us / 1e6) / 1e9
    peaks = measured_peaks()
    line = {"metric": METRIC, "value": gbs, "unit": "GB/s", "n_gpus": 1, "steps": args.steps,
            "warmup": args.warmup, "higher_is_better": True, "vs_baseline": None,
            "dtype": "bf16", "data": "synthetic",
            "config": {"workload": f"qmv_smallm {K}->{N}, M={M}, {copies} distinct weight "
                                   "copies in one CUDA graph", "l2": "inputs larger than L2"},
            "us_per_call": us, "frac": gbs / peaks["hbm_gbs"], "peak": peaks}
    print(json.dumps(line), flush=True)
    sv.device_status()
    return 0


def run_wide(args):
    """qmv_wide on one wide block (--rows M, default the 128 verify rows of 32
    sequences at K = 3) against --wide-shape N K (default the LM head
    5120 -> 151936), on enough weight copies that they stream from HBM, in one
    CUDA graph; TFLOP/s of the product against the measured bf16 peak.  Also
    the case the ncu captures of the tcgen05 kernel run."""
    import torch

    import mtp_speculative_decoding_qmv_gb300 as sv

    dev = torch.device("cuda", 0)
    N, K = args.wide_shape
    M = args.rows
    g = torch.Generator(device=dev)
    g.manual_seed(wl.MASTER_SEED + 41)
    per = qmv_bytes(M, N, K)
    copies = max(1, -(-300_000_000 // per))
    weights = []
    for _ in range(copies):
        w = torch.randint(-(2 ** 31), 2 ** 31 - 1, (N, K // 8), generator=g, device=dev,
                          dtype=torch.int32)
        s_ = (torch.randn((N, K // GROUP), generator=g, device=dev) * 0.02).to(torch.bfloat16)
        b_ = (torch.randn((N, K // GROUP), generator=g, device=dev) * 0.02).to(torch.bfloat16)
        weights.append((w, s_, b_))
    x = torch.randn((M, K), generator=g, device=dev).to(torch.bfloat16)
    y = torch.empty((M, N), device=dev)
    ws = sv.make_wide_workspace(M, K, dev)

    def fn():
        for w, s_, b_ in weights:
            sv.qmv_wide(w, s_, b_, x, y=y, workspace=ws)

    stream = torch.cuda.Stream(dev)
    graph = capture(torch, fn, stream)
    ms = time_graph(torch, graph, stream, args.steps, args.warmup)
    us = ms / args.steps / copies * 1e3
    peaks = measured_peaks()
    tflops = 2 * M * N * K / (us / 1e6) / 1e12
    n_mma = -(-M // 16) * 16
    issued = 2 * n_mma * N * (2 * K + wide_bias_columns(K)) / (us / 1e6) / 1e12
    line = {"metric": METRIC, "value": tflops, "unit": "TFLOP/s", "n_gpus": 1,
            "steps": args.steps, "warmup": args.warmup, "higher_is_better": True,
            "vs_baseline": None, "dtype": "bf16", "data": "synthetic",
            "config": {"workload": f"qmv_wide {K}->{N}, M={M}, {copies} weight copies in one "
                                   "CUDA graph", "l2": "inputs larger than L2"},
            "us_per_call": us, "gbs": per / (us / 1e6) / 1e9,
            "frac_of_bf16_peak": tflops / peaks["bf16_tflops"],
            "tensor_tflops_issued": issued,
            "issued_frac_of_bf16_peak": issued / peaks["bf16_tflops"],
            "peak": peaks}
    print(json.dumps(line), flush=True)
    sv.device_status()
    return 0


def run_drafthead(args):
    """The drafter's own 4-bit LM head: requantise the bf16 LM head (5120 ->
    151936) with qmv_requantize, then the draft step's logits as qmv_smallm at
    M = 1 on it, beside the bf16 head read by a plain library GEMV (context
    for the draft-time saving the pages report)."""
    import torch

    import mtp_speculative_decoding_qmv_gb300 as sv

    dev = torch.device("cuda", 0)
    g = torch.Generator(device=dev)
    g.manual_seed(wl.MASTER_SEED + 43)
    N, K = wl.VOCAB, wl.HIDDEN
    w16 = (torch.randn((N, K), generator=g, device=dev) * 0.02).to(torch.bfloat16)
    wp = torch.empty((N, K // 8), dtype=torch.int32, device=dev)
    s_ = torch.empty((N, K // GROUP), dtype=torch.bfloat16, device=dev)
    b_ = torch.empty((N, K // GROUP), dtype=torch.bfloat16, device=dev)
    x = torch.randn((1, K), generator=g, device=dev).to(torch.bfloat16)
    y4 = torch.empty((1, N), device=dev)
    y16 = torch.empty((1, N), dtype=torch.bfloat16, device=dev)
    stream = torch.cuda.Stream(dev)

    def requant():
        sv.qmv_requantize(w16, out=(wp, s_, b_))

    def draft4():
        sv.qmv_smallm(wp, s_, b_, x, y4)

    def draft16():
        torch.matmul(x, w16.t(), out=y16)

    requant()
    torch.cuda.synchronize()
    rq = time_graph(torch, capture(torch, requant, stream), stream, args.steps, args.warmup)
    d4 = time_graph(torch, capture(torch, draft4, stream), stream, args.steps, args.warmup)
    d16 = time_graph(torch, capture(torch, draft16, stream), stream, args.steps, args.warmup)
    rq_us, d4_us, d16_us = (t / args.steps * 1e3 for t in (rq, d4, d16))
    peaks = measured_peaks()
    rq_bytes = N * K * 2 + N * K // 2 + 2 * 2 * N * (K // GROUP)
    line = {"metric": METRIC, "value": qmv_bytes(1, N, K) / (d4_us / 1e6) / 1e9, "unit": "GB/s",
            "n_gpus": 1, "steps": args.steps, "warmup": args.warmup, "higher_is_better": True,
            "vs_baseline": None, "dtype": "bf16", "data": "synthetic",
            "config": {"workload": f"draft-only 4-bit LM head {K}->{N}: requantise the bf16 "
                                   "head, then the draft step's logits at M=1",
                       "l2": "inputs larger than L2"},
            "draft_logits_us_4bit": d4_us, "draft_logits_us_bf16_library_gemv": d16_us,
            "draft_lm_head_time_saved": 1.0 - d4_us / d16_us,
            "requantize_us": rq_us,
            "requantize_gbs": rq_bytes / (rq_us / 1e6) / 1e9,
            "requantize_frac": rq_bytes / (rq_us / 1e6) / 1e9 / peaks["hbm_gbs"],
            "frac": qmv_bytes(1, N, K) / (d4_us / 1e6) / 1e9 / peaks["hbm_gbs"],
            "peak": peaks}
    print(json.dumps(line), flush=True)
    sv.device_status()
    return 0


def run_stream(args):
    """The 27B-class verify weight stream (--layers decoder layers of q, k,
    v, o 5120x5120, gate, up 5120->17408, down 17408->5120, plus the LM head
    5120->151936) at M = depth + 1 as ONE qmv plan without dependency waits:
    the qmv kernel's streaming rate.  Also the case the ncu captures of the
    plan kernel run (a few layers)."""
    import torch

    import mtp_speculative_decoding_qmv_gb300 as sv

    dev = torch.device("cuda", 0)
    M = args.depth + 1
    g = torch.Generator(device=dev)
    g.manual_seed(wl.MASTER_SEED + 41)
    shapes = [(N, K) for _ in range(args.layers) for _, N, K in wl.LAYER_PROJECTIONS]
    shapes.append((wl.VOCAB, wl.HIDDEN))
    probs = []
    for N, K in shapes:
        w = torch.randint(-(2 ** 31), 2 ** 31 - 1, (N, K // 8), generator=g, device=dev,
                          dtype=torch.int32)
        s_ = (torch.randn((N, K // GROUP), generator=g, device=dev) * 0.02).to(torch.bfloat16)
        b_ = (torch.randn((N, K // GROUP), generator=g, device=dev) * 0.02).to(torch.bfloat16)
        x = torch.randn((M, K), generator=g, device=dev).to(torch.bfloat16)
        probs.append((w, s_, b_, x, torch.empty((M, N), device=dev), False))
    plan = sv.QmvPlan(probs)
    nbytes = sum(qmv_bytes(M, N, K) for N, K in shapes)
    stream = torch.cuda.Stream(dev)
    graph = capture(torch, plan.run, stream)
    ms = time_graph(torch, graph, stream, args.steps, args.warmup) / args.steps
    gbs = nbytes / (ms / 1e3) / 1e9
    peaks = measured_peaks()
    line = {"metric": METRIC, "value": gbs, "unit": "GB/s", "n_gpus": 1, "steps": args.steps,
            "warmup": args.warmup, "higher_is_better": True, "vs_baseline": None,
            "dtype": "bf16", "data": "synthetic",
            "config": {"workload": f"27B-class weight stream: {args.layers} layers x {{q,k,v,o "
                                   f"5120x5120; gate,up 5120->17408; down 17408->5120}} + LM "
                                   f"head 5120->151936, 4-bit g64, M={M}, one qmv plan",
                       "bytes": nbytes, "grid": plan.grid,
                       "l2": "inputs larger than L2" if nbytes > 3e8 else "small case"},
            "ms_per_step": ms, "frac": gbs / peaks["hbm_gbs"], "peak": peaks}
    print(json.dumps(line), flush=True)
    sv.device_status()
    return 0


def sample_filtered(torch, z, T, top_k, top_p, g):
    """Tokens drawn from the filtered distributions of logits rows z [..., V]
    (temperature, top-k, top-p, renormalise): the drafter's sampling step,
    used to make synthetic drafts (setup only)."""
    top, idx = (z / T).topk(top_k, dim=-1)
    q = torch.softmax(top, dim=-1)
    q = torch.where((q.cumsum(-1) - q) < top_p, q, torch.zeros_like(q))
    flat = (q / q.sum(-1, keepdim=True)).reshape(-1, top_k)
    pick = torch.multinomial(flat, 1, generator=g).view(*q.shape[:-1], 1)
    return idx.gather(-1, pick).squeeze(-1).to(torch.int32)


def lmhead_rates(torch, sv, depth: int, steps: int, warmup: int) -> dict:
    """Configuration 3, LM-head verify + accept: 32 sequences x (M=4 LM-head
    qmv 5120->151936) then one spec_accept over the batch; the LM-head input
    is scaled so the target logits have standard deviation 3, draft = target
    + N(0, 0.5) with drafts sampled from the filtered draft distributions
    (about 70 % accepted per position); T 0.6 / top-k 20 / top-p 0.95, and
    greedy (T = 0).  The batch's rows as one qmv_wide product (the value),
    and as 32 per-sequence problems of one qmv plan."""
    dev = torch.device("cuda", 0)
    sv.set_pdl(True)
    g = torch.Generator(device=dev)
    g.manual_seed(wl.MASTER_SEED + 29)
    B, K, V, H = 32, depth, wl.VOCAB, wl.HIDDEN
    M = K + 1
    w = torch.randint(-(2 ** 31), 2 ** 31 - 1, (V, H // 8), generator=g, device=dev,
                      dtype=torch.int32)
    s_ = (torch.randn((V, H // GROUP), generator=g, device=dev) * 0.02).to(torch.bfloat16)
    b_ = (torch.randn((V, H // GROUP), generator=g, device=dev) * 0.02).to(torch.bfloat16)
    x_all = torch.randn((B * M, H), generator=g, device=dev).to(torch.bfloat16)
    xs = [x_all[i * M:(i + 1) * M] for i in range(B)]  # views: one [B*M, H] block
    logits = torch.empty((B, M, V), device=dev)
    plan = sv.QmvPlan([(w, s_, b_, xs[i], logits[i], False) for i in range(B)])
    plan.run()
    torch.cuda.synchronize()
    c = 3.0 / float(logits.std())
    for x in xs:
        x.copy_((x.float() * c).to(x.dtype))
    plan.run()
    torch.cuda.synchronize()
    draft = (logits[:, :K] + torch.randn((B, K, V), generator=g, device=dev) * 0.5).contiguous()
    tokens = sample_filtered(torch, draft, 0.6, 20, 0.95, g)
    greedy_tokens = draft.argmax(dim=-1).to(torch.int32)
    ua, us = wl.accept_uniforms(31, B, K)
    ua, us = torch.from_numpy(ua).to(dev), torch.from_numpy(us).to(dev)
    ws = sv.make_accept_workspace(B, K, V, dev)
    out = torch.empty((B, M), dtype=torch.int32, device=dev)
    nacc = torch.empty((B,), dtype=torch.int32, device=dev)
    flags = torch.empty((B,), dtype=torch.int32, device=dev)

    def accept():
        sv.spec_accept(logits, draft, tokens, ua, us, 0.6, 20, 0.95, workspace=ws,
                       out_tokens=out, n_accepted=nacc, err_flags=flags)

    # accept timed on its own: three copies of the logits in turn, so that each
    # call streams its inputs from HBM (a greedy call reads 78 MB, which an
    # L2 of 129 MB would otherwise keep from one replay to the next)
    copies = [(logits, draft)] + [(logits.clone(), draft.clone()) for _ in range(2)]

    def accept_copies():
        for lg, dr in copies:
            sv.spec_accept(lg, dr, tokens, ua, us, 0.6, 20, 0.95, workspace=ws,
                           out_tokens=out, n_accepted=nacc, err_flags=flags)

    def accept_greedy_copies():
        for lg, _ in copies:
            sv.spec_accept(lg, None, greedy_tokens, ua, us, 0.0, 1, 1.0, workspace=ws,
                           out_tokens=out, n_accepted=nacc, err_flags=flags)

    def fn():
        plan.run()
        accept()

    # the batch's verify blocks as one M = B (K+1) product on the tcgen05
    # tensor cores: the LM head is streamed once for all sequences
    wws = sv.make_wide_workspace(B * M, H, dev)
    y_all = logits.view(B * M, V)

    def lm_wide():
        sv.qmv_wide(w, s_, b_, x_all, y=y_all, workspace=wws)

    def fn_wide():
        lm_wide()
        accept()

    stream = torch.cuda.Stream(dev)
    ggraph = capture(torch, accept_greedy_copies, stream)
    gms = time_graph(torch, ggraph, stream, steps, warmup) / len(copies)
    n_greedy = nacc.clone()
    graph = capture(torch, fn, stream)
    agraph = capture(torch, accept_copies, stream)
    wgraph = capture(torch, fn_wide, stream)
    lgraph = capture(torch, lm_wide, stream)
    ms_plan = time_graph(torch, graph, stream, steps, warmup)
    ams = time_graph(torch, agraph, stream, steps, warmup) / len(copies)
    ms = time_graph(torch, wgraph, stream, steps, warmup)
    lms = time_graph(torch, lgraph, stream, steps, warmup)
    acc_bytes = B * (2 * K + 1) * V * 4
    n = nacc.cpu().numpy()
    tested = sum(min(int(a) + 1, K) for a in n)
    r = {"value": B / (ms / 1e3 / steps), "unit": "sequence-cycles/s",
            "config": {"workload": f"LM-head verify + accept: batch {B}, K={K} (M={M}) rows "
                                   f"per sequence, 5120->151936 4-bit g64 (the batch's "
                                   f"{B * M} rows as one qmv_wide product), "
                                   f"T=0.6 top_k=20 top_p=0.95, draft = target + N(0, 0.5), "
                                   f"target logits scaled by c to std 3",
                       "c": c},
            "ms_per_step": ms / steps,
            "lm_head_wide": {"kernel": f"qmv_wide, M={B * M} (tcgen05)",
                             "us": lms / steps * 1e3,
                             "gbs": qmv_bytes(B * M, V, H) / (lms / 1e3 / steps) / 1e9,
                             "tflops": 2 * B * M * V * H / (lms / 1e3 / steps) / 1e12,
                             "tensor_tflops_issued":
                                 2 * B * M * V * (2 * H + wide_bias_columns(H))
                                 / (lms / 1e3 / steps) / 1e12},
            "per_sequence_plan": {"sequence_cycles_per_s": B / (ms_plan / 1e3 / steps),
                                  "ms_per_step": ms_plan / steps,
                                  "how": f"{B} M={M} problems in one qmv plan (the LM head "
                                         f"streamed once per sequence), then spec_accept"},
            "qmv_gbs": B * qmv_bytes(M, V, H) / ((ms_plan - ams) / 1e3 / steps) / 1e9,
            "spec_accept_us": ams / steps * 1e3,
            "spec_accept_gbs": acc_bytes / (ams / 1e3 / steps) / 1e9,
            "spec_accept_greedy_us": gms / steps * 1e3,
            "spec_accept_greedy_gbs": B * (K + 1) * V * 4 / (gms / 1e3 / steps) / 1e9,
            "mean_accepted": float(n.mean()),
            "acceptance_rate_per_position": int(n.sum()) / max(tested, 1),
            "logit_scale_c": c,
            "mean_accepted_greedy": float(n_greedy.float().mean().item())}
    plan.close()
    sv.device_status()
    return r


def run_lmhead(args):
    """LM-head verify + accept (configuration 3); see lmhead_rates."""
    import torch

    import mtp_speculative_decoding_qmv_gb300 as sv

    r = lmhead_rates(torch, sv, args.depth, args.steps, args.warmup)
    line = {"metric": METRIC, "value": r["value"], "unit": r["unit"], "n_gpus": 1,
            "steps": args.steps, "warmup": args.warmup, "higher_is_better": True,
            "vs_baseline": None, "dtype": "bf16", "data": "synthetic",
            **{k: v for k, v in r.items() if k not in ("value", "unit")}}
    print(json.dumps(line), flush=True)
    return 0


def gdn_rates(torch, sv, steps: int, warmup: int) -> dict:
    """Configuration 4, the GatedDeltaNet tape: 16 sequences x 48 heads x
    128x128 fp32 state, 5 tokens; capture, then replay of an accepted prefix
    drawn from U{0..5}.  24 independent state copies (1.2 GB) so the timing
    streams from HBM."""
    dev = torch.device("cuda", 0)
    B, T, H, d = 16, 5, wl.GDN_HEADS, wl.GDN_DIM
    x = wl.gdn_inputs(50, B, T, H, d, d)
    copies = 24
    states = [torch.from_numpy(x["state0"]).to(dev) for _ in range(copies)]
    t = {n: torch.from_numpy(x[n]).to(dev) for n in ("q", "k", "v", "alpha", "beta", "n_replay")}
    tapes = [torch.empty(sv.gdn_tape_bytes(B, T, H, d, d) // 4, device=dev) for _ in range(copies)]
    outs = [torch.empty((B, T, H, d), device=dev) for _ in range(copies)]

    def cap():
        for i in range(copies):
            sv.gdn_tape_capture(states[i], t["q"], t["k"], t["v"], t["alpha"], t["beta"],
                                tape=tapes[i], out=outs[i])

    def rep():
        for i in range(copies):
            sv.gdn_tape_replay(states[i], tapes[i], t["n_replay"], T)

    stream = torch.cuda.Stream(dev)
    gc, gr = capture(torch, cap, stream), capture(torch, rep, stream)
    mc = time_graph(torch, gc, stream, steps, warmup) / steps / copies
    mr = time_graph(torch, gr, stream, steps, warmup) / steps / copies
    nb = B * H * d * d * 4
    tape_b = sv.gdn_tape_bytes(B, T, H, d, d)
    cap_bytes = nb + B * T * H * (3 * d + 2) * 4 + B * T * H * d * 4 + tape_b
    n_live = int((x["n_replay"] > 0).sum())
    rep_bytes = n_live * H * d * d * 4 * 2 + tape_b * n_live // B
    sv.device_status()
    peak = measured_peaks()["hbm_gbs"]
    cap_gbs, rep_gbs = cap_bytes / (mc / 1e3) / 1e9, rep_bytes / (mr / 1e3) / 1e9
    return {"capture_us": mc * 1e3, "replay_us": mr * 1e3,
            "capture_gbs": cap_gbs, "replay_gbs": rep_gbs,
            "capture_frac": cap_gbs / peak, "replay_frac": rep_gbs / peak,
            "capture_bytes": cap_bytes, "replay_bytes": rep_bytes,
            "how": "B=16, H=48, dk=dv=128, T=5, prefix ~ U{0..5}; 24 state copies per graph, "
                   "CUDA events, per-call time"}


def run_gdn(args):
    """GatedDeltaNet tape capture/replay (configuration 4); see gdn_rates."""
    import torch

    import mtp_speculative_decoding_qmv_gb300 as sv

    r = gdn_rates(torch, sv, args.steps, args.warmup)
    line = {"metric": "GDN tape capture/replay GB/s", "value": r["capture_gbs"],
            "unit": "GB/s", "n_gpus": 1, "steps": args.steps, "warmup": args.warmup,
            "higher_is_better": True, "vs_baseline": None, "dtype": "f32", "data": "synthetic",
            "config": {"workload": "GDN tape: B=16, H=48, dk=dv=128, T=5, prefix ~ U{0..5}"},
            **{k: v for k, v in r.items() if k != "how"}}
    print(json.dumps(line), flush=True)
    return 0


NEAR_TIE = 1e-5  # |u - p/q|, top-p and inverse-CDF boundary margins counted as near ties


def accept_near_ties(torch, sv, depth: int, seed: int = 77) -> dict:
    """spec_accept on the GPU against the oracle at the LM-head configuration
    (batch 32, V = 151936, draft depth `depth`; target logits ~ N(0, 3),
    draft = target + N(0, 0.5), drafts sampled from the filtered draft
    distributions; T 0.6 / top-k 20 / top-p 0.95), on one seeded draw.
    Counts the sequences whose float64 oracle met a near tie, per class, and
    the sequences whose tokens, accepted length or flags differ outside them
    (the parity bar: zero)."""
    import numpy as np

    import oracle

    oracle.build()
    oracle.set_threads(len(os.sched_getaffinity(0)))
    dev = torch.device("cuda", 0)
    B, K, V = 32, depth, wl.VOCAB
    T, top_k, top_p = float(np.float32(0.6)), 20, float(np.float32(0.95))
    tl, dl = wl.accept_logits(seed, B, K, V, sigma=3.0, draft_noise=0.5)
    g = torch.Generator(device=dev)
    g.manual_seed(wl.MASTER_SEED + seed)
    dr = sample_filtered(torch, torch.from_numpy(dl).to(dev), T, top_k, top_p, g)
    ua, us = wl.accept_uniforms(seed, B, K)
    out, nacc, flags = sv.spec_accept(torch.from_numpy(tl).to(dev), torch.from_numpy(dl).to(dev),
                                      dr, torch.from_numpy(ua).to(dev),
                                      torch.from_numpy(us).to(dev), T, top_k, top_p)
    gpu = [a.cpu().numpy() for a in (out, nacc, flags)]
    t0 = time.perf_counter()
    r = oracle.spec_accept(tl, dl, dr.cpu().numpy(), ua, us, T, top_k, top_p)
    t_oracle = time.perf_counter() - t0
    diag = r["diag"]
    cls = {"accept_ratio": diag[:, 0] < NEAR_TIE, "top_p_boundary": diag[:, 1] < NEAR_TIE,
           "inverse_cdf_boundary": diag[:, 2] < NEAR_TIE}
    near = cls["accept_ratio"] | cls["top_p_boundary"] | cls["inverse_cdf_boundary"]
    ok = ~near
    differ = ((gpu[0] != r["out_tokens"]).any(axis=1) | (gpu[1] != r["n_accepted"]) |
              (gpu[2] != r["err_flags"]))
    return {"sequences": B, "near_tie_margin": NEAR_TIE,
            "near_ties": {k: int(v.sum()) for k, v in cls.items()},
            "near_tie_sequences": int(near.sum()),
            "mismatches_outside_near_ties": int((differ & ok).sum()),
            "mismatches_at_near_ties": int((differ & near).sum()),
            "min_margins": {"accept_ratio": float(diag[:, 0].min()),
                            "top_p_boundary": float(diag[:, 1].min()),
                            "inverse_cdf_boundary": float(diag[:, 2].min())},
            "mean_accepted": float(gpu[1].mean()),
            "oracle_seconds": t_oracle,
            "how": f"one seeded draw (seed {seed}) at the LM-head configuration, the GPU "
                   f"spec_accept against the float64 oracle sequence by sequence; a near tie "
                   f"is a margin below {NEAR_TIE:g} (|u - p/q|, the top-p cumulative sum, the "
                   f"inverse-CDF boundary)"}


def run_conv(args):
    """Short convolution windows of a GatedDeltaNet layer: batch 16, T = 5
    verify tokens, C = 3 x 48 x 128 channels (q, k, v streams), W = 4; the
    capture's outputs and the commit of an accepted prefix ~ U{0..5}."""
    import torch

    import mtp_speculative_decoding_qmv_gb300 as sv

    dev = torch.device("cuda", 0)
    B, T, C, W = 16, 5, wl.CONV_CHANNELS, wl.CONV_WIDTH
    d = wl.conv_inputs(70, B, T, C, W)
    copies = 24  # distinct buffers so that timing streams from HBM
    t = {k: torch.from_numpy(v).to(dev) for k, v in d.items()}
    wins = [t["window"].clone() for _ in range(copies)]
    xs = [t["x"].clone() for _ in range(copies)]
    ys = [torch.empty_like(t["x"]) for _ in range(copies)]

    def cap():
        for i in range(copies):
            sv.conv_window_capture(wins[i], xs[i], t["weight"], y=ys[i])

    def rep():
        for i in range(copies):
            sv.conv_window_replay(wins[i], xs[i], t["n_replay"])

    stream = torch.cuda.Stream(dev)
    gc, gr = capture(torch, cap, stream), capture(torch, rep, stream)
    mc = time_graph(torch, gc, stream, args.steps, args.warmup) / args.steps / copies
    mr = time_graph(torch, gr, stream, args.steps, args.warmup) / args.steps / copies
    cap_bytes = 4 * (B * (W - 1) * C + 2 * B * T * C + W * C)
    n_live = int((d["n_replay"] > 0).sum())
    rep_bytes = 4 * n_live * (2 * (W - 1) * C)  # reads at most W-1 entries, writes W-1
    peaks = measured_peaks()
    line = {"metric": "conv window capture/commit GB/s", "value": cap_bytes / (mc / 1e3) / 1e9,
            "unit": "GB/s", "n_gpus": 1, "steps": args.steps, "warmup": args.warmup,
            "higher_is_better": True, "vs_baseline": None, "dtype": "f32", "data": "synthetic",
            "config": {"workload": f"conv windows: B={B}, T={T}, C={C}, W={W}, prefix ~ U{{0..{T}}}"},
            "capture_us": mc * 1e3, "replay_us": mr * 1e3,
            "capture_frac": cap_bytes / (mc / 1e3) / 1e9 / peaks["hbm_gbs"],
            "replay_gbs": rep_bytes / (mr / 1e3) / 1e9}
    print(json.dumps(line), flush=True)
    sv.device_status()
    return 0


def main(argv=None):
    ap = argparse.ArgumentParser(description=__doc__.split("\n\n")[0])
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20)
    ap.add_argument("--warmup", type=int, default=3)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--depth", type=int, default=3, help="draft depth K (M = K+1)")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-configs", action="store_true",
                    help="cycle: skip the MLP, LM-head + accept and GDN tape sub-measurements")
    ap.add_argument("--no-depth-sweep", action="store_true",
                    help="cycle: skip the draft depths K = 2..5 other than --depth")
    ap.add_argument("--workload", choices=["cycle", "mlp", "lmhead", "gdn", "qmv", "stream",
                                           "conv", "wide", "drafthead"],
                    default="cycle")
    ap.add_argument("--layers", type=int, default=wl.N_LAYERS,
                    help="decoder layers of the --workload stream plan")
    ap.add_argument("--layout", choices=["plans", "allplans", "launches"], default="plans",
                    help="cycle: qmv plans for q,k,v / gate,up / down and qmv_smallm for o "
                         "(plans), plans for every projection (allplans), or one "
                         "qmv_smallm launch per projection (launches)")
    ap.add_argument("--lm-head", choices=["fused", "logits"], default="logits",
                    help="cycle: the LM-head plan writes the logits that spec_accept reads "
                         "(logits), or keeps per-CTA top-64 lists that spec_accept_lists "
                         "merges (fused; the logits never reach memory)")
    ap.add_argument("--shape", type=int, nargs=2, metavar=("N", "K"),
                    default=[wl.INTERMEDIATE, wl.HIDDEN],
                    help="output and input size of the --workload qmv projection")
    ap.add_argument("--wide-shape", type=int, nargs=2, metavar=("N", "K"),
                    default=[wl.VOCAB, wl.HIDDEN],
                    help="output and input size of the --workload wide product")
    ap.add_argument("--rows", type=int, default=128,
                    help="activation rows M of the --workload wide product")
    args = ap.parse_args(argv)
    if args.warmup < 3:
        ap.error("--warmup must be >= 3")
    if args.impl == "reference":
        return run_reference(args)
    return {"cycle": run_cycle, "mlp": run_mlp, "lmhead": run_lmhead, "gdn": run_gdn,
            "qmv": run_qmv, "stream": run_stream, "conv": run_conv, "wide": run_wide,
            "drafthead": run_drafthead}[
        args.workload](args)


if __name__ == "__main__":
    sys.exit(main())
