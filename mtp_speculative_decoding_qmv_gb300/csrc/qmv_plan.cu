// qmv_plan.cu -- an ordered list of 4-bit small-M mat-vecs run by ONE
// persistent launch, sm_103a.
//
// Source: "MTPLX 2.24x faster TPS", section "Layer 0: MLX Runtime" (the verify
// forward runs M = K+1 rows through every 4-bit projection of the target
// model) and "MTP in llama.cpp", section "Theoretical maximum tg t/s" (a
// decode step is bounded by streaming the active weights once at memory
// bandwidth).
//
// A verify forward is hundreds of small projections in a row.  Launched one
// by one, each pays the launch and the latency of its first weight stage
// (several microseconds on this part, as much as streaming a 50 MB
// projection takes), so the weight stream stops at every boundary.  Here the
// whole list is one launch of exactly as many CTAs as fit on the GPU at once
// (not a cooperative launch, which measured ~1.5 us slower per launch; see
// qmv_plan_run for why every CTA still becomes resident):
//  * the list is cut into phases at every problem flagged `after` (its
//    activations are an earlier problem's output); inside a phase the
//    problems are independent;
//  * the (problem, 64-row tile, 512-input stage) work of a phase is laid out
//    flat and every CTA takes one equal contiguous run of it (stream-K
//    style), so every SM has the same number of stages in every phase;
//  * each CTA's producer warp streams the weight stages of all its runs, phase
//    after phase, through the shared-memory ring without ever waiting on
//    other CTAs: the weights of the next phase are in flight while the
//    current phase finishes;
//  * consumers read a phase's activations only after the device-wide count
//    of finished tiles says every tile of the earlier phases has been
//    written (one acquire load by one thread, bounded wait);
//  * a tile whose stages fall in several CTAs' runs is reduced by the last of
//    them to finish, summing the partials in run order -- deterministic;
//  * counters are left at zero by the last CTA / last arriver, so the plan
//    is ready for the next launch.
// The per-group math (nibble widening, bf16 MMA, scale/bias epilogue) is the
// one of qmv_smallm (qmv_common.cuh).
// One problem may carry a top-64 epilogue instead of y: the epilogue warp
// merges each finished tile's values into per-output-row sorted lists of
// (logit, index) keys in shared memory and every CTA writes its lists at the
// end (the fused LM head that spec_accept_lists reads).
#include <algorithm>
#include <cstdlib>
#include <cstring>
#include <new>
#include <vector>

#include "qmv_common.cuh"

namespace sv {
namespace {
using namespace qmv;

constexpr int kPartial = kRows * 8;  // floats per partial tile: 64 rows x 8 columns
constexpr int kPlanCtasPerSm = 2;    // co-resident CTAs per SM (register budget)
constexpr int kEpilogueWarp = kConsumerWarps + 1;   // after the producer warp
constexpr int kPlanThreads = (kConsumerWarps + 2) * 32;
// suspend-time hint of the epilogue warp's waits: it signals tiles that other
// CTAs may be waiting for, so it must resume promptly
constexpr uint32_t kEpilogueSuspendNs = 256;

__device__ unsigned int g_plan_device_error;

// One problem of the plan, in device memory (tensor maps 64-byte aligned).
struct PlanProblem {  // CUtensorMap's own alignment (>= 64 bytes) carries over
  CUtensorMap wmap, smap, bmap;
  const void *x;
  float *y;
  unsigned long long *topk;  // per-CTA top-64 lists instead of y (or null)
  int N, K;
  int tiles, chunks;  // 64-row tiles, 512-input stages
  int chunk_off;      // first flat stage index in its phase
  int tile_off;       // first tile index in its phase
};

struct PlanPhase {
  int first, count;     // problems
  int work;             // stages in the phase (< 2^31)
  int run_q, run_r;     // runs: work = run_q * G + run_r (see run_begin)
  int tiles_before;     // tiles of all earlier phases
  int wait;             // 1: activations are earlier outputs
  int signal;           // 1: a later phase waits for this one's tiles
  int max_splits;       // partial slots per tile
};

// One run of consecutive stages of one tile inside a CTA's range of a
// phase; each CTA's records are contiguous and in order (built on the host).
struct PlanSeg {
  const void *x;        // the problem's activations
  int K;                // the problem's input size
  int p;                // problem
  int tile;             // 64-row tile of the problem
  int c0, c1;           // stages [c0, c1) of the tile
  int split, n_splits;  // this run's place among the runs of the tile
  int tile_in_phase;
  int phase;
  int pad;
};

struct PlanParams {
  const PlanProblem *problems;
  const PlanPhase *phases;
  const PlanSeg *segs;  // [G] first run of each CTA (c0 == c1: none), then the rest
  const int *seg_off;   // [G + 1]: CTA c's later runs are segs[seg_off[c] .. seg_off[c+1])
  float *partials;      // [tiles of a phase][max_splits][kPartial]
  int *tile_count;      // [tiles of a phase] arrivals
  int *done_tiles;      // tiles written (all phases so far)
  int *done_ctas;
  int n_phases;
  int M;
  int stages;
  int topk;  // 1: one problem has the top-64 epilogue (lists in shared memory)
  unsigned long long *topk_out;  // that problem's lists [G][M][64], then flags [G][M]
};

constexpr int kTopK = 64;        // keys kept per CTA and output row by the epilogue
constexpr int kTopKRows = 8;     // M <= 8
// the lists, their flags, and one tile's keys for the merge
constexpr uint32_t kTopKBytes = kTopKRows * kTopK * 8 + kTopKRows * 4 + 64 * 8;
static_assert((kTopKRows * kTopK * 8 + kTopKRows * 4) % 16 == 0, "the tile keys, 16-byte aligned");

struct PlanLayout {
  uint32_t ring, red, topk, bar, total;
};
__host__ __device__ inline PlanLayout plan_layout(int stages, bool topk) {
  PlanLayout L;
  L.ring = (uint32_t)stages * kStageBytesStream;
  L.red = L.ring;
  L.topk = L.red + kRedBytes;
  L.bar = L.topk + (topk ? kTopKBytes : 0u);
  L.bar = (L.bar + 7u) & ~7u;
  L.total = L.bar + (uint32_t)(2 * stages + 2) * 8u + 1024u;
  return L;
}

// Ordered key of a logit: larger float -> larger key; 0 = never kept (NaN,
// +inf, -inf); NaN and +inf also set `nonfinite`.  Equal floats (-0, +0) give
// equal keys; the composite with the inverted index puts the lower index
// first among equal logits.
__device__ __forceinline__ uint32_t topk_logit_key(float v, int &nonfinite) {
  uint32_t u = __float_as_uint(v);
  if ((u & 0x7F800000u) == 0x7F800000u) {
    if ((u & 0x007FFFFFu) != 0 || (u >> 31) == 0) nonfinite = 1;
    return 0u;
  }
  if ((u & 0x7FFFFFFFu) == 0) u = 0;
  return (u & 0x80000000u) ? ~u : (u | 0x80000000u);
}

// One warp merges a tile's values of output row m (lane: rows n0 + lane and
// n0 + lane + 32) into the descending list `list` [kTopK] (shared memory).
// Only values above the list's last key can enter.  Several of them are
// placed at once: every key's place in the merged list is the number of
// larger keys in the list and among the tile's values (keys are distinct:
// one row each), counted against both in shared memory (`tile`, 64 keys),
// and the keys whose place is below kTopK are written there.  A single one
// is inserted by counting the larger entries and shifting the rest down.
__device__ void topk_merge_tile(unsigned long long *list, unsigned long long *tile,
                                unsigned int *flag, float c0, float c1, int n0, int N) {
  const int lane = threadIdx.x & 31;
  int nf = 0;
  const int r0 = n0 + lane, r1 = n0 + lane + 32;
  const uint32_t k0 = r0 < N ? topk_logit_key(c0, nf) : 0u;
  const uint32_t k1 = r1 < N ? topk_logit_key(c1, nf) : 0u;
  if (__any_sync(0xffffffffu, nf) && lane == 0) *flag = 1u;
  unsigned long long e0 = k0 ? ((unsigned long long)k0 << 32) | (0xFFFFFFFFu - (uint32_t)r0) : 0ull;
  unsigned long long e1 = k1 ? ((unsigned long long)k1 << 32) | (0xFFFFFFFFu - (uint32_t)r1) : 0ull;
  unsigned long long l0 = list[lane], l1 = list[lane + 32];
  unsigned long long thr = __shfl_sync(0xffffffffu, l1, 31);
  if (e0 <= thr) e0 = 0ull;
  if (e1 <= thr) e1 = 0ull;
  const int entering = __popc(__ballot_sync(0xffffffffu, e0 != 0ull)) +
                       __popc(__ballot_sync(0xffffffffu, e1 != 0ull));
  if (entering > 1) {
    tile[lane] = e0;
    tile[lane + 32] = e1;
    __syncwarp();
    int p_e0 = 0, p_e1 = 0, p_l0 = lane, p_l1 = lane + 32;  // places in the merged list
#pragma unroll 4
    for (int j = 0; j < kTopK; j += 2) {
      const ulonglong2 t = *reinterpret_cast<const ulonglong2 *>(tile + j);
      const ulonglong2 l = *reinterpret_cast<const ulonglong2 *>(list + j);
      p_e0 += (t.x > e0) + (t.y > e0) + (l.x > e0) + (l.y > e0);
      p_e1 += (t.x > e1) + (t.y > e1) + (l.x > e1) + (l.y > e1);
      p_l0 += (t.x > l0) + (t.y > l0);
      p_l1 += (t.x > l1) + (t.y > l1);
    }
    __syncwarp();  // every read of the list before the first write
    if (l0 != 0ull && p_l0 < kTopK) list[p_l0] = l0;
    if (l1 != 0ull && p_l1 < kTopK) list[p_l1] = l1;
    if (e0 != 0ull && p_e0 < kTopK) list[p_e0] = e0;
    if (e1 != 0ull && p_e1 < kTopK) list[p_e1] = e1;
    __syncwarp();
    return;
  }
  while (__any_sync(0xffffffffu, (e0 | e1) != 0ull)) {
    const unsigned long long g = warp_max_u64(e0 > e1 ? e0 : e1);
    const int pos = __popc(__ballot_sync(0xffffffffu, l0 > g)) +
                    __popc(__ballot_sync(0xffffffffu, l1 > g));
    // shift entries pos.. down one place, g at pos
    unsigned long long p0 = __shfl_up_sync(0xffffffffu, l0, 1);
    unsigned long long p1 = __shfl_up_sync(0xffffffffu, l1, 1);
    const unsigned long long l0_31 = __shfl_sync(0xffffffffu, l0, 31);
    if (lane == 0) p1 = l0_31;
    const unsigned long long n0v = lane < pos ? l0 : (lane == pos ? g : p0);
    const unsigned long long n1v = lane + 32 < pos ? l1 : (lane + 32 == pos ? g : p1);
    l0 = n0v;
    l1 = n1v;
    if (e0 == g) e0 = 0ull;
    if (e1 == g) e1 = 0ull;
    thr = __shfl_sync(0xffffffffu, l1, 31);
    if (e0 <= thr) e0 = 0ull;
    if (e1 <= thr) e1 = 0ull;
  }
  list[lane] = l0;
  list[lane + 32] = l1;
  __syncwarp();
}

__device__ __forceinline__ int atom_add_acq_rel(int *p, int v) {
  int old;
  asm volatile("atom.acq_rel.gpu.global.add.s32 %0, [%1], %2;" : "=r"(old) : "l"(p), "r"(v)
               : "memory");
  return old;
}
__device__ __forceinline__ void red_add_release(int *p, int v) {
  asm volatile("red.release.gpu.global.add.s32 [%0], %1;" ::"l"(p), "r"(v) : "memory");
}
__device__ __forceinline__ int ld_acquire(const int *p) {
  int v;
  asm volatile("ld.acquire.gpu.global.s32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
  return v;
}

// Bounded wait until *p >= target (one thread).  False after the limit.
__device__ bool wait_count(const int *p, int target) {
  if (ld_acquire(p) >= target) return true;
  const unsigned long long t0 = global_timer_ns();
  unsigned ns = 32;
  for (;;) {
    __nanosleep(ns);
    if (ns < 128) ns <<= 1;
    if (ld_acquire(p) >= target) return true;
    if (global_timer_ns() - t0 > kWaitLimitNs) return false;
  }
}

template <bool kXF32>
__device__ __forceinline__ XRaw<kXF32> load_x_l2(const void *xrow, int g, int t) {
  // activations may have been written by other CTAs of this launch: read
  // them at L2 (no stale L1 lines)
  XRaw<kXF32> r;
  if constexpr (!kXF32) {
    const uint4 *p = reinterpret_cast<const uint4 *>(static_cast<const uint16_t *>(xrow) +
                                                     g * 64 + 8 * t);
    r.v[0] = __ldcg(p);
    r.v[1] = __ldcg(p + 4);
  } else {
    const uint4 *p =
        reinterpret_cast<const uint4 *>(static_cast<const float *>(xrow) + g * 64 + 8 * t);
    r.v[0] = __ldcg(p);
    r.v[1] = __ldcg(p + 1);
    r.v[2] = __ldcg(p + 8);
    r.v[3] = __ldcg(p + 9);
  }
  return r;
}

// This CTA's runs: the first at segs[cta] (loaded without waiting for the
// offsets), the later ones from seg_off.
struct RunList {
  const PlanSeg *segs;
  int head, rest, n;
  __device__ RunList(const PlanParams &P, int cta) : segs(P.segs) {
    const PlanSeg &h = P.segs[cta];
    const int first = P.seg_off[cta], last = P.seg_off[cta + 1];
    head = cta;
    rest = first;
    n = (h.c1 > h.c0 ? 1 : 0) + (last - first);
  }
  __device__ const PlanSeg &operator[](int i) const {
    return i == 0 ? segs[head] : segs[rest + i - 1];
  }
};

__device__ __forceinline__ void consumer_bar() {
  asm volatile("bar.sync 1, %0;" ::"r"(kConsumerWarps * 32) : "memory");
}

template <bool kXF32>
__global__ void __launch_bounds__(kPlanThreads, kPlanCtasPerSm)
    qmv_plan_kernel(const PlanParams P) {
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  const uint32_t raw = smem_addr(smem_raw);
  const uint32_t base = raw + ((1024u - (raw & 1023u)) & 1023u);
  uint8_t *smem = smem_raw + (base - raw);
  const int G = gridDim.x, cta = blockIdx.x;
  const int stages = P.stages;
  const PlanLayout L = plan_layout(stages, P.topk != 0);
  const uint32_t full0 = base + L.bar;
  const uint32_t empty0 = full0 + 8u * stages;
  const uint32_t red_full = empty0 + 8u * stages;  // consumers' tile sums are in red
  const uint32_t red_empty = red_full + 8u;        // the epilogue warp has read them
  float *red = reinterpret_cast<float *>(smem + L.red);  // [warp][row * 8 + col]
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  if (threadIdx.x == 0) {
    for (int i = 0; i < stages; ++i) {
      mbar_init_u32(full0 + 8u * i, 1);
      mbar_init_u32(empty0 + 8u * i, kConsumerWarps);
    }
    mbar_init_u32(red_full, kConsumerWarps * 32);
    mbar_init_u32(red_empty, 32);
    fence_mbar_init();
  }
  __syncthreads();
  pdl_launch_dependents();

  if (warp == kConsumerWarps) {
    // ------------------------------ producer ------------------------------
    // weights do not depend on earlier kernels: no griddepcontrol.wait here
    if (lane == 0) {
      const uint64_t policy = l2_policy_evict_first();
      int st = 0, ph = 0;
      long long issued = 0;
      bool ok = true;
      const RunList runs(P, cta);
      for (int i = 0; ok && i < runs.n; ++i) {
        const PlanSeg s = runs[i];
        {
          const PlanProblem &q = P.problems[s.p];
          const int n0 = s.tile * kRows;
          for (int c = s.c0; c < s.c1; ++c) {
            if (issued >= stages && !mbar_wait_u32(empty0 + 8u * st, ph ^ 1)) {
              atomicOr(&g_plan_device_error, 1u);
              ok = false;
              break;
            }
            const uint32_t stage = base + st * kStageBytesStream, bar = full0 + 8u * st;
            const int k0 = c * kStageInputs;
            mbar_arrive_expect_tx_u32(bar, kSbOff + 2 * kRows * 16);
            tma_load_2d(stage, &q.wmap, k0 / 8, n0, bar, policy);
            tma_load_2d(stage + kRows * 128, &q.wmap, k0 / 8 + kBoxWords, n0, bar, policy);
            tma_load_2d(stage + kSbOff, &q.smap, k0 / 64, n0, bar, policy);
            tma_load_2d(stage + kSbOff + kRows * 16, &q.bmap, k0 / 64, n0, bar, policy);
            ++issued;
            if (++st == stages) {
              st = 0;
              ph ^= 1;
            }
          }
        }
      }
      // every copy issued has landed before the CTA may exit (normally the
      // consumers have waited for all of them already)
      for (long long i = std::max(0ll, issued - stages); i < issued; ++i)
        (void)mbar_wait_u32(full0 + 8u * (uint32_t)(i % stages), (uint32_t)((i / stages) & 1));
    }
    __syncwarp();
  } else if (warp == kEpilogueWarp) {
    // ------------------------------ epilogue ------------------------------
    // Per tile run: sum the eight warps' partials in warp order (lane = rows
    // lane and lane + 32, all eight columns), free red, then write y (or
    // this run's partial; the last run of a split tile sums the partials in
    // run order) and count the tile when a later phase waits for it.
    unsigned nseg = 0;
    const float4 *red4 = reinterpret_cast<const float4 *>(red);
    // the top-64 lists of this CTA (empty = key 0) and their non-finite flags
    unsigned long long *tk_list = reinterpret_cast<unsigned long long *>(smem + L.topk);
    unsigned int *tk_flag = reinterpret_cast<unsigned int *>(tk_list + kTopKRows * kTopK);
    unsigned long long *tk_tile =
        reinterpret_cast<unsigned long long *>(tk_flag + kTopKRows);  // 16-byte aligned
    if (P.topk) {
      for (int i = lane; i < kTopKRows * kTopK; i += 32) tk_list[i] = 0ull;
      if (lane < kTopKRows) tk_flag[lane] = 0u;
      __syncwarp();
    }
    pdl_wait();  // y and the plan's counters belong to the preceding kernel until here
    int cur_phase = -1, max_splits = 1, signal = 0;
    const RunList runs(P, cta);
    for (int i = 0; i < runs.n; ++i) {
      const PlanSeg s = runs[i];
      if (s.phase != cur_phase) {
        cur_phase = s.phase;
        max_splits = P.phases[cur_phase].max_splits;
        signal = P.phases[cur_phase].signal;
      }
      {
        if (!mbar_wait_u32(red_full, nseg & 1, kEpilogueSuspendNs))
          atomicOr(&g_plan_device_error, 8u);
        float4 v[4];  // rows lane (v[0], v[1]) and lane + 32 (v[2], v[3]); 8 columns each
#pragma unroll
        for (int i = 0; i < 4; ++i) v[i] = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
        for (int w = 0; w < kConsumerWarps; ++w) {
#pragma unroll
          for (int i = 0; i < 4; ++i) {
            const float4 a = red4[w * (kPartial / 4) + (lane + 32 * (i >> 1)) * 2 + (i & 1)];
            v[i].x += a.x;
            v[i].y += a.y;
            v[i].z += a.z;
            v[i].w += a.w;
          }
        }
        mbar_arrive_u32(red_empty);
        ++nseg;
        const PlanProblem &q = P.problems[s.p];
        const int N = q.N, n0 = s.tile * kRows;
        // A split tile is summed by its first run (split 0): that CTA's run
        // ends with the tile, so it reaches it last and the later runs,
        // which start their CTAs' ranges with it, have usually published
        // their partials already.  They store and count without waiting.
        bool write = true;
        float4 *slots = nullptr;
        if (s.n_splits > 1) {
          slots = reinterpret_cast<float4 *>(P.partials) +
                  (size_t)s.tile_in_phase * max_splits * (kPartial / 4);
          int *count = &P.tile_count[s.tile_in_phase];
          if (s.split > 0) {
#pragma unroll
            for (int i = 0; i < 4; ++i)
              __stcg(&slots[(size_t)s.split * (kPartial / 4) + (lane + 32 * (i >> 1)) * 2 + (i & 1)],
                     v[i]);
            __syncwarp();
            if (lane == 0) red_add_release(count, 1);  // publishes this run's partial
            write = false;
          } else {
            if (lane == 0 && !wait_count(count, s.n_splits - 1))
              atomicOr(&g_plan_device_error, 32u);
            __syncwarp();  // the other lanes read after lane 0's acquire
            // own partial first, then the later runs in run order
#pragma unroll 1
            for (int r = 1; r < s.n_splits; r += 2) {
              float4 a[4], b[4];
              const bool two = r + 1 < s.n_splits;
#pragma unroll
              for (int i = 0; i < 4; ++i) {
                const size_t o = (size_t)(lane + 32 * (i >> 1)) * 2 + (i & 1);
                a[i] = __ldcg(&slots[(size_t)r * (kPartial / 4) + o]);
                b[i] = two ? __ldcg(&slots[(size_t)(r + 1) * (kPartial / 4) + o])
                           : make_float4(0.f, 0.f, 0.f, 0.f);
              }
#pragma unroll
              for (int i = 0; i < 4; ++i) {
                v[i].x += a[i].x;
                v[i].y += a[i].y;
                v[i].z += a[i].z;
                v[i].w += a[i].w;
                if (two) {
                  v[i].x += b[i].x;
                  v[i].y += b[i].y;
                  v[i].z += b[i].z;
                  v[i].w += b[i].w;
                }
              }
            }
          }
        }
        if (write) {
          if (q.topk) {
            // the tile's columns go into this CTA's top-64 lists, not to y
            const float c0[8] = {v[0].x, v[0].y, v[0].z, v[0].w, v[1].x, v[1].y, v[1].z, v[1].w};
            const float c1[8] = {v[2].x, v[2].y, v[2].z, v[2].w, v[3].x, v[3].y, v[3].z, v[3].w};
#pragma unroll
            for (int col = 0; col < 8; ++col)
              if (col < P.M)
                topk_merge_tile(tk_list + col * kTopK, tk_tile, tk_flag + col, c0[col], c1[col],
                                n0, N);
          } else {
#pragma unroll
            for (int h = 0; h < 2; ++h) {
              const int row = n0 + lane + 32 * h;
              if (row < N) {
                const float c[8] = {v[2 * h].x, v[2 * h].y, v[2 * h].z, v[2 * h].w,
                                    v[2 * h + 1].x, v[2 * h + 1].y, v[2 * h + 1].z,
                                    v[2 * h + 1].w};
#pragma unroll
                for (int col = 0; col < 8; ++col)
                  if (col < P.M) q.y[(size_t)col * N + row] = c[col];
              }
            }
          }
          __syncwarp();
          if (lane == 0) {
            if (slots) P.tile_count[s.tile_in_phase] = 0;  // ready for the next launch
            if (signal) red_add_release(P.done_tiles, 1);
          }
        }
      }
    }
    if (P.topk) {
      // every CTA writes its lists (empty ones included) and flags
      unsigned long long *dst = P.topk_out + (size_t)cta * P.M * kTopK;
      for (int i = lane; i < P.M * kTopK; i += 32) dst[i] = tk_list[i];
      unsigned int *fdst =
          reinterpret_cast<unsigned int *>(P.topk_out + (size_t)G * P.M * kTopK) + cta * P.M;
      if (lane < P.M) fdst[lane] = tk_flag[lane];
    }
  } else {
    // ------------------------------ consumers -----------------------------
    const int g8 = lane >> 2, t = lane & 3;
    const int gl = warp;
    const uint32_t ldm_off = ldmatrix_offset(gl, lane);
    const uint32_t sb_off = kSbOff + (uint32_t)(g8 * 16 + gl * 2);
    const int xm = g8 < P.M ? g8 : 0;  // padding columns read row 0, never stored
    const size_t xbytes = kXF32 ? 4 : 2;
    bool ok = true;
    int st = 0, ph = 0;
    unsigned nseg = 0;
    pdl_wait();  // x and the plan's counters belong to the preceding kernel until here
    float acc[kTiles][4];
#pragma unroll
    for (int i = 0; i < kTiles; ++i) acc[i][0] = acc[i][1] = acc[i][2] = acc[i][3] = 0.f;
    const RunList runs(P, cta);
    const int i_end = runs.n;
    int i = 0;
    int cur_phase = -1;
    bool have_x = false;  // xnext holds the first stage of segment i
    XRaw<kXF32> xnext;
    PlanSeg s;
    if (i < i_end) s = runs[0];
    while (i < i_end) {
      if (s.phase != cur_phase) {
        cur_phase = s.phase;
        const PlanPhase &pp = P.phases[cur_phase];
        if (pp.wait) {
          // every tile of the earlier phases is written before x is read
          if (threadIdx.x == 0 && !wait_count(P.done_tiles, pp.tiles_before))
            atomicOr(&g_plan_device_error, 4u);
          consumer_bar();
        }
        have_x = false;
      }
      const void *xrow = static_cast<const uint8_t *>(s.x) + (size_t)xm * s.K * xbytes;
      if (!have_x) xnext = load_x_l2<kXF32>(xrow, s.c0 * kConsumerWarps + gl, t);
      // the next run, for the activation prefetch (same phase only)
      const bool have2 = i + 1 < i_end;
      PlanSeg s2 = s;
      if (have2) s2 = runs[i + 1];
      const bool same = have2 && s2.phase == s.phase;
      int g = s.c0 * kConsumerWarps + gl;
      for (int c = s.c0; c < s.c1; ++c, g += kConsumerWarps) {
        const XRaw<kXF32> xcur = xnext;
        if (c + 1 < s.c1)
          xnext = load_x_l2<kXF32>(xrow, g + kConsumerWarps, t);
        else if (same)
          xnext = load_x_l2<kXF32>(static_cast<const uint8_t *>(s2.x) + (size_t)xm * s2.K * xbytes,
                                   s2.c0 * kConsumerWarps + gl, t);
        if (ok && !warp_wait_stage(full0 + 8u * st, ph)) {
          ok = false;
          if (lane == 0) atomicOr(&g_plan_device_error, 2u);
        }
        if (ok) {
          const uint32_t stage = base + st * kStageBytesStream;
          group_math<kXF32>(acc, stage + ldm_off, xcur, stage + sb_off, 16 * 16, 8 * 16,
                            kRows * 16);
        }
        __syncwarp();
        if (lane == 0) mbar_arrive_u32(empty0 + 8u * st);
        if (++st == stages) {
          st = 0;
          ph ^= 1;
        }
      }
      // hand the run's sums to the epilogue warp: red[warp][row][col]
      if (nseg > 0 && !__all_sync(0xffffffffu, mbar_wait_u32(red_empty, (nseg - 1) & 1)) &&
          lane == 0)
        atomicOr(&g_plan_device_error, 16u);
      float *r = red + warp * kPartial;
#pragma unroll
      for (int rt = 0; rt < kTiles; ++rt) {
        const int r0 = rt * 16 + g8;
        *reinterpret_cast<float2 *>(&r[r0 * 8 + 2 * t]) = make_float2(acc[rt][0], acc[rt][1]);
        *reinterpret_cast<float2 *>(&r[(r0 + 8) * 8 + 2 * t]) =
            make_float2(acc[rt][2], acc[rt][3]);
        acc[rt][0] = acc[rt][1] = acc[rt][2] = acc[rt][3] = 0.f;
      }
      mbar_arrive_u32(red_full);
      ++nseg;
      have_x = same;
      s = s2;
      ++i;
    }
  }

  // the last CTA to finish leaves the tile count at zero for the next launch
  // (a single-phase plan never counts tiles)
  if (P.n_phases > 1) {
    __syncthreads();
    if (threadIdx.x == 0 && atom_add_acq_rel(P.done_ctas, 1) == G - 1) {
      *P.done_tiles = 0;
      *P.done_ctas = 0;
      __threadfence();
    }
  }
}

}  // namespace

unsigned take_device_error_plan() {
  unsigned v = 0, zero = 0;
  cudaMemcpyFromSymbol(&v, g_plan_device_error, sizeof v);
  cudaMemcpyToSymbol(g_plan_device_error, &zero, sizeof zero);
  return v;
}

}  // namespace sv

using namespace sv;

struct sv_qmv_plan {
  int M;
  sv_dtype x_dtype;
  int grid, stages;
  uint32_t smem;
  PlanParams params;
};

namespace {

struct PlanShape {
  std::vector<PlanProblem> probs;
  std::vector<PlanPhase> phases;
  std::vector<int> seg_off;
  std::vector<PlanSeg> segs;
  size_t off_phases, off_seg_off, off_segs, off_partials, off_counts, off_done, total;
  int max_phase_tiles;
};

// Phases, stage offsets and partial slots for `G` CTAs; device buffer layout.
sv_status plan_shape(const sv_qmv_problem *pr, int n, int G, PlanShape &S) {
  S.probs.assign(n, PlanProblem{});
  S.phases.clear();
  int tiles_before = 0;
  S.max_phase_tiles = 1;
  size_t partial_floats = kPartial;
  for (int i = 0; i < n;) {
    PlanPhase ph{};
    ph.first = i;
    ph.wait = (i > 0 && pr[i].after) ? 1 : 0;
    ph.tiles_before = tiles_before;
    long long work = 0;
    int tiles = 0, min_chunks = 1 << 30;
    int j = i;
    do {
      PlanProblem &q = S.probs[j];
      q.N = pr[j].N;
      q.K = pr[j].K;
      q.x = pr[j].x;
      q.y = pr[j].y;
      q.topk = reinterpret_cast<unsigned long long *>(pr[j].topk);
      q.tiles = (q.N + kRows - 1) / kRows;
      q.chunks = q.K / kStageInputs;
      q.chunk_off = (int)work;
      q.tile_off = tiles;
      work += (long long)q.tiles * q.chunks;
      tiles += q.tiles;
      min_chunks = std::min(min_chunks, q.chunks);
      ++j;
    } while (j < n && !pr[j].after);
    ph.count = j - i;
    if (work > (1ll << 30))
      return fail(SV_ERR_UNSUPPORTED, "qmv_plan_create: a phase has more than 2^30 stages");
    ph.work = (int)work;
    ph.run_q = (int)(work / G);
    ph.run_r = (int)(work % G);
    // a tile of C stages meets at most ceil(C / q) + 1 runs of >= q stages
    const long long q_min = work / G;
    int max_chunks = 0;
    for (int k = i; k < j; ++k) max_chunks = std::max(max_chunks, S.probs[k].chunks);
    ph.max_splits = q_min > 0 ? (int)std::min<long long>(G, (max_chunks + q_min - 1) / q_min + 1)
                              : std::min(G, max_chunks);
    partial_floats = std::max(partial_floats, (size_t)tiles * ph.max_splits * kPartial);
    S.max_phase_tiles = std::max(S.max_phase_tiles, tiles);
    tiles_before += tiles;
    S.phases.push_back(ph);
    i = j;
  }
  // every phase but the first waits for all the tiles before it
  for (size_t k = 0; k + 1 < S.phases.size(); ++k) S.phases[k].signal = 1;
  // Each CTA's runs, phase after phase: in a phase of W = q G + r stages CTA
  // c takes [c q + min(c, r), (c+1) q + min(c+1, r)) of the flat (problem,
  // tile, stage) order, so the first r CTAs take q+1 stages and the others q
  // (none when q = 0 and c >= r); the CTAs whose runs meet a tile are
  // consecutive and every one of them holds part of it.
  auto run_begin = [](int c, int q, int r) { return c * q + std::min(c, r); };
  auto owner = [](int j, int q, int r) {
    const int big = r * (q + 1);
    return j < big ? j / (q + 1) : r + (j - big) / q;
  };
  // per CTA, in order; then split into the first run of each CTA (at index
  // c) and the later runs
  std::vector<std::vector<PlanSeg>> per(G);
  for (int c = 0; c < G; ++c) {
    for (int f = 0; f < (int)S.phases.size(); ++f) {
      const PlanPhase &ph = S.phases[f];
      int j = run_begin(c, ph.run_q, ph.run_r);
      const int end = run_begin(c + 1, ph.run_q, ph.run_r);
      int p = ph.first;
      while (j < end) {
        while (j >= S.probs[p].chunk_off + S.probs[p].tiles * S.probs[p].chunks) ++p;
        const PlanProblem &q = S.probs[p];
        PlanSeg g{};
        g.x = q.x;
        g.K = q.K;
        g.p = p;
        const int rel = j - q.chunk_off;
        g.tile = rel / q.chunks;
        g.c0 = rel - g.tile * q.chunks;
        const int tile_start = q.chunk_off + g.tile * q.chunks;
        const int tile_end = tile_start + q.chunks;
        const int seg_end = std::min(tile_end, end);
        g.c1 = g.c0 + (seg_end - j);
        const int first = owner(tile_start, ph.run_q, ph.run_r);
        g.split = c - first;
        g.n_splits = owner(tile_end - 1, ph.run_q, ph.run_r) - first + 1;
        if (g.n_splits > ph.max_splits)
          return fail(SV_ERR_CUDA, "qmv_plan_create: internal split count error");
        g.tile_in_phase = q.tile_off + g.tile;
        g.phase = f;
        per[c].push_back(g);
        j = seg_end;
      }
    }
  }
  S.segs.assign(G, PlanSeg{});  // c0 == c1 == 0: no run
  S.seg_off.assign(G + 1, 0);
  for (int c = 0; c < G; ++c) {
    if (!per[c].empty()) S.segs[c] = per[c][0];
    S.seg_off[c] = (int)S.segs.size();
    for (size_t k = 1; k < per[c].size(); ++k) S.segs.push_back(per[c][k]);
  }
  S.seg_off[G] = (int)S.segs.size();
  if (tiles_before >= (1 << 30))
    return fail(SV_ERR_UNSUPPORTED, "qmv_plan_create: too many tiles");
  auto up = [](size_t v, size_t a) { return (v + a - 1) / a * a; };
  size_t off = up((size_t)n * sizeof(PlanProblem), 256);
  S.off_phases = off;
  off = up(off + S.phases.size() * sizeof(PlanPhase), 256);
  S.off_seg_off = off;
  off = up(off + S.seg_off.size() * sizeof(int), 256);
  S.off_segs = off;
  off = up(off + S.segs.size() * sizeof(PlanSeg), 256);
  S.off_partials = off;
  off = up(off + partial_floats * 4, 256);
  S.off_counts = off;
  off = up(off + (size_t)S.max_phase_tiles * 4, 256);
  S.off_done = off;
  S.total = off + 256;
  return SV_OK;
}

template <bool kXF32>
sv_status plan_config(int dev, bool topk, int &grid, int &stages, uint32_t &smem) {
  int optin = 0, smem_sm = 0, sms = device_sm_count();
  cudaDeviceGetAttribute(&optin, cudaDevAttrMaxSharedMemoryPerBlockOptin, dev);
  cudaDeviceGetAttribute(&smem_sm, cudaDevAttrMaxSharedMemoryPerMultiprocessor, dev);
  cudaFuncAttributes fa = {};
  if (cudaFuncGetAttributes(&fa, qmv_plan_kernel<kXF32>) != cudaSuccess)
    return fail(SV_ERR_CUDA, "qmv_plan: cudaFuncGetAttributes failed");
  if (cudaFuncSetAttribute(qmv_plan_kernel<kXF32>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                           optin - (int)fa.sharedSizeBytes) != cudaSuccess)
    return fail(SV_ERR_CUDA, "qmv_plan: cudaFuncSetAttribute failed: %s",
                cudaGetErrorString(cudaGetLastError()));
  int occ = 0;
  if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&occ, qmv_plan_kernel<kXF32>, kPlanThreads, 0) !=
          cudaSuccess ||
      occ < 1)
    return fail(SV_ERR_CUDA, "qmv_plan: occupancy query failed");
  const int per_sm = std::min(occ, kPlanCtasPerSm);
  // 1 KB per CTA is reserved by the system; static shared memory comes first
  const uint32_t budget = (uint32_t)smem_sm / per_sm - 1024u - (uint32_t)fa.sharedSizeBytes;
  stages = 2;
  const uint32_t cap = std::min<uint32_t>(budget, (uint32_t)optin - (uint32_t)fa.sharedSizeBytes);
  while (stages < 16 && plan_layout(stages + 1, topk).total <= cap) ++stages;
  smem = plan_layout(stages, topk).total;
  if (smem > (uint32_t)optin) return fail(SV_ERR_UNSUPPORTED, "qmv_plan: shared memory");
  int fit = 0;
  if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&fit, qmv_plan_kernel<kXF32>, kPlanThreads,
                                                    smem) != cudaSuccess ||
      fit < 1)
    return fail(SV_ERR_CUDA, "qmv_plan: occupancy query failed");
  grid = std::min(fit, per_sm) * sms;
  return SV_OK;
}

bool has_topk(const sv_qmv_problem *pr, int n) {
  for (int i = 0; i < n; ++i)
    if (pr[i].topk) return true;
  return false;
}

size_t topk_bytes(int grid, int M) {
  return (size_t)grid * M * (kTopK * sizeof(unsigned long long) + sizeof(unsigned int));
}

sv_status validate_problems(const sv_qmv_problem *pr, int n, int M, sv_dtype x_dtype) {
  if (n < 1 || !pr) return fail(SV_ERR_INVALID_ARG, "qmv_plan: need n_problems >= 1");
  if (M < 1 || M > 8) return fail(SV_ERR_UNSUPPORTED, "qmv_plan: M=%d outside [1, 8]", M);
  if (x_dtype != SV_F32 && x_dtype != SV_BF16)
    return fail(SV_ERR_INVALID_ARG, "qmv_plan: unknown x_dtype %d", (int)x_dtype);
  int phase_start = 0, n_topk = 0;
  for (int i = 0; i < n; ++i) {
    const sv_qmv_problem &q = pr[i];
    if (q.N < 1 || q.K < 1)
      return fail(SV_ERR_INVALID_ARG, "qmv_plan: problem %d: need N, K >= 1", i);
    if (q.K % kStageInputs)
      return fail(SV_ERR_UNSUPPORTED, "qmv_plan: problem %d: K=%d is not a multiple of %d", i,
                  q.K, kStageInputs);
    if (q.N > (1 << 30) || q.K > (1 << 30))
      return fail(SV_ERR_INVALID_ARG, "qmv_plan: problem %d too large", i);
    if (!q.w_packed || !q.scales || !q.biases || !q.x || (!q.y && !q.topk))
      return fail(SV_ERR_INVALID_ARG, "qmv_plan: problem %d: null pointer", i);
    if (!aligned(q.w_packed, 16) || !aligned(q.scales, 16) || !aligned(q.biases, 16) ||
        !aligned(q.x, 16) || !aligned(q.y, 4) || !aligned(q.topk, 8))
      return fail(SV_ERR_INVALID_ARG, "qmv_plan: problem %d: misaligned pointer", i);
    if (q.topk && ++n_topk > 1)
      return fail(SV_ERR_UNSUPPORTED, "qmv_plan: more than one problem with a top-64 epilogue");
    const size_t wb = (size_t)q.N * q.K / 2, sbb = (size_t)q.N * (q.K / 64) * 2;
    const size_t xb = (size_t)M * q.K * (x_dtype == SV_F32 ? 4 : 2);
    // the output: y, or the top-64 lists (their size is checked at create)
    const void *out = q.topk ? static_cast<const void *>(q.topk) : q.y;
    const size_t ob = q.topk ? (size_t)1 : (size_t)M * q.N * 4;
    if (overlaps(out, ob, q.w_packed, wb) || overlaps(out, ob, q.scales, sbb) ||
        overlaps(out, ob, q.biases, sbb) || overlaps(out, ob, q.x, xb))
      return fail(SV_ERR_INVALID_ARG, "qmv_plan: problem %d: y overlaps an input", i);
    // an output read later in the same phase would be read before it is written
    if (i == 0 || q.after) phase_start = i;
    for (int j = phase_start; j < i; ++j)
      if (!pr[j].topk && overlaps(pr[j].y, (size_t)M * pr[j].N * 4, q.x, xb))
        return fail(SV_ERR_INVALID_ARG,
                    "qmv_plan: problem %d reads problem %d's output without `after`", i, j);
  }
  return SV_OK;
}

}  // namespace

extern "C" size_t qmv_plan_device_bytes(const sv_qmv_problem *problems, int n_problems, int M,
                                        sv_dtype x_dtype) {
  clear_error();
  if (validate_problems(problems, n_problems, M, x_dtype) != SV_OK) return 0;
  int grid = 0, stages = 0;
  uint32_t smem = 0;
  const int dev = current_device();
  const bool topk = has_topk(problems, n_problems);
  const sv_status st = x_dtype == SV_BF16 ? plan_config<false>(dev, topk, grid, stages, smem)
                                          : plan_config<true>(dev, topk, grid, stages, smem);
  if (st != SV_OK) return 0;
  PlanShape S;
  if (plan_shape(problems, n_problems, grid, S) != SV_OK) return 0;
  return S.total;
}

extern "C" sv_status qmv_plan_create(const sv_qmv_problem *problems, int n_problems, int M,
                                     sv_dtype x_dtype, void *device_buffer, size_t device_bytes,
                                     sv_qmv_plan **plan_out) {
  clear_error();
  if (!plan_out) return fail(SV_ERR_INVALID_ARG, "qmv_plan_create: null plan_out");
  *plan_out = nullptr;
  sv_status st = validate_problems(problems, n_problems, M, x_dtype);
  if (st != SV_OK) return st;
  const int dev = current_device();
  int grid = 0, stages = 0;
  uint32_t smem = 0;
  const bool topk = has_topk(problems, n_problems);
  st = x_dtype == SV_BF16 ? plan_config<false>(dev, topk, grid, stages, smem)
                          : plan_config<true>(dev, topk, grid, stages, smem);
  if (st != SV_OK) return st;
  PlanShape S;
  st = plan_shape(problems, n_problems, grid, S);
  if (st != SV_OK) return st;
  if (!device_buffer || !aligned(device_buffer, 256))
    return fail(SV_ERR_INVALID_ARG, "qmv_plan_create: device_buffer must be 256-byte aligned");
  if (device_bytes < S.total)
    return fail(SV_ERR_INVALID_ARG, "qmv_plan_create: device buffer of %zu bytes, need %zu",
                device_bytes, S.total);
  for (int i = 0; i < n_problems; ++i)
    if (problems[i].topk &&
        overlaps(problems[i].topk, topk_bytes(grid, M), device_buffer, S.total))
      return fail(SV_ERR_INVALID_ARG, "qmv_plan_create: the top-64 buffer overlaps the plan");
  for (int i = 0; i < n_problems; ++i) {
    const sv_qmv_problem &q = problems[i];
    PlanProblem &d = S.probs[i];
    const int groups = q.K / 64;
    st = encode_2d(&d.wmap, CU_TENSOR_MAP_DATA_TYPE_UINT32, q.w_packed, (uint64_t)q.K / 8,
                   (uint64_t)q.N, (uint64_t)q.K / 2, kBoxWords, kRows, CU_TENSOR_MAP_SWIZZLE_128B);
    if (st == SV_OK)
      st = encode_2d(&d.smap, CU_TENSOR_MAP_DATA_TYPE_UINT16, q.scales, (uint64_t)groups,
                     (uint64_t)q.N, (uint64_t)groups * 2, 8, kRows, CU_TENSOR_MAP_SWIZZLE_NONE);
    if (st == SV_OK)
      st = encode_2d(&d.bmap, CU_TENSOR_MAP_DATA_TYPE_UINT16, q.biases, (uint64_t)groups,
                     (uint64_t)q.N, (uint64_t)groups * 2, 8, kRows, CU_TENSOR_MAP_SWIZZLE_NONE);
    if (st != SV_OK) return st;
  }
  // descriptors, phases, then zeroed partial counters and done counters
  std::vector<uint8_t> host(S.off_partials, 0);
  std::memcpy(host.data(), S.probs.data(), S.probs.size() * sizeof(PlanProblem));
  std::memcpy(host.data() + S.off_phases, S.phases.data(), S.phases.size() * sizeof(PlanPhase));
  std::memcpy(host.data() + S.off_seg_off, S.seg_off.data(), S.seg_off.size() * sizeof(int));
  std::memcpy(host.data() + S.off_segs, S.segs.data(), S.segs.size() * sizeof(PlanSeg));
  uint8_t *dbuf = static_cast<uint8_t *>(device_buffer);
  if (cudaMemcpy(dbuf, host.data(), host.size(), cudaMemcpyHostToDevice) != cudaSuccess ||
      cudaMemset(dbuf + S.off_counts, 0, S.total - S.off_counts) != cudaSuccess)
    return fail(SV_ERR_CUDA, "qmv_plan_create: copying the plan to the device failed");
  sv_qmv_plan *plan = new (std::nothrow) sv_qmv_plan;
  if (!plan) return fail(SV_ERR_INVALID_ARG, "qmv_plan_create: out of host memory");
  plan->M = M;
  plan->x_dtype = x_dtype;
  plan->grid = grid;
  plan->stages = stages;
  plan->smem = smem;
  PlanParams &P = plan->params;
  P.problems = reinterpret_cast<const PlanProblem *>(dbuf);
  P.phases = reinterpret_cast<const PlanPhase *>(dbuf + S.off_phases);
  P.seg_off = reinterpret_cast<const int *>(dbuf + S.off_seg_off);
  P.segs = reinterpret_cast<const PlanSeg *>(dbuf + S.off_segs);
  P.partials = reinterpret_cast<float *>(dbuf + S.off_partials);
  P.tile_count = reinterpret_cast<int *>(dbuf + S.off_counts);
  P.done_tiles = reinterpret_cast<int *>(dbuf + S.off_done);
  P.done_ctas = P.done_tiles + 1;
  P.n_phases = (int)S.phases.size();
  P.M = M;
  P.stages = stages;
  P.topk = topk ? 1 : 0;
  P.topk_out = nullptr;
  for (int i = 0; i < n_problems; ++i)
    if (problems[i].topk) P.topk_out = reinterpret_cast<unsigned long long *>(problems[i].topk);
  *plan_out = plan;
  return SV_OK;
}

namespace {
sv_status plan_launch(const sv_qmv_plan *plan, sv_stream_t stream, bool cooperative) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)plan->grid);
  cfg.blockDim = dim3(kPlanThreads);
  cfg.dynamicSmemBytes = plan->smem;
  cfg.stream = reinterpret_cast<cudaStream_t>(stream);
  // The grid is the co-resident count, so every CTA becomes resident as soon
  // as the kernels ahead of it on the device release their SMs, which they do
  // without waiting on this plan; dependents launched early (PDL) start only
  // after every CTA of the plan has started.  The waits between CTAs (phase
  // counts, split tiles) therefore end; each is bounded all the same.  A
  // cooperative launch would guarantee residency outright but measured ~1.5 us
  // slower per launch.
  // A cooperative launch guarantees co-residency outright (for callers that
  // share the device with other grids whose CTAs wait on one another), and
  // is not combined with the programmatic early start.
  cudaLaunchAttribute attr[1];
  int na = 0;
  if (cooperative) {
    attr[na].id = cudaLaunchAttributeCooperative;
    attr[na].val.cooperative = 1;
    ++na;
  } else if (pdl_enabled()) {
    attr[na].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[na].val.programmaticStreamSerializationAllowed = 1;
    ++na;
  }
  cfg.attrs = attr;
  cfg.numAttrs = na;
  const char *what = cooperative ? "qmv_plan_run_cooperative" : "qmv_plan_run";
  const cudaError_t e =
      plan->x_dtype == SV_BF16
          ? cudaLaunchKernelEx(&cfg, qmv_plan_kernel<false>, plan->params)
          : cudaLaunchKernelEx(&cfg, qmv_plan_kernel<true>, plan->params);
  if (e != cudaSuccess) return fail(SV_ERR_CUDA, "%s: launch failed: %s", what, cudaGetErrorString(e));
  return check_launch(what);
}
}  // namespace

extern "C" sv_status qmv_plan_run(const sv_qmv_plan *plan, sv_stream_t stream) {
  clear_error();
  if (!plan) return fail(SV_ERR_INVALID_ARG, "qmv_plan_run: null plan");
  return plan_launch(plan, stream, false);
}

extern "C" sv_status qmv_plan_run_cooperative(const sv_qmv_plan *plan, sv_stream_t stream) {
  clear_error();
  if (!plan) return fail(SV_ERR_INVALID_ARG, "qmv_plan_run_cooperative: null plan");
  return plan_launch(plan, stream, true);
}

extern "C" void qmv_plan_destroy(sv_qmv_plan *plan) { delete plan; }

extern "C" int qmv_plan_grid(const sv_qmv_plan *plan) { return plan ? plan->grid : 0; }

extern "C" size_t qmv_plan_topk_bytes(int M, sv_dtype x_dtype) {
  clear_error();
  if (M < 1 || M > 8 || (x_dtype != SV_F32 && x_dtype != SV_BF16)) {
    fail(SV_ERR_INVALID_ARG, "qmv_plan_topk_bytes: M=%d or dtype %d invalid", M, (int)x_dtype);
    return 0;
  }
  int grid = 0, stages = 0;
  uint32_t smem = 0;
  const int dev = current_device();
  const sv_status st = x_dtype == SV_BF16 ? plan_config<false>(dev, true, grid, stages, smem)
                                          : plan_config<true>(dev, true, grid, stages, smem);
  return st == SV_OK ? topk_bytes(grid, M) : 0;
}
