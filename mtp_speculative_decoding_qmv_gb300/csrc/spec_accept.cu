// spec_accept.cu -- fp32 probability-ratio verification of K drafted tokens
// per sequence, residual resampling and bonus token, sm_103a.
//
// Sources: "MTPLX 2.24x faster TPS", sections "Layer 2: Speculative cycle"
// (Leviathan-Chen acceptance per position in fp32, (p - q)+ residual on the
// first rejection, bonus token when all K are accepted) and "QWEN 3.6 27B @ 63
// TPS" (temperature 0.6, top_p 0.95, top_k 20); "MTP in llama.cpp", section
// "lossless" (temperature 0: accept until the first mismatch with the
// target's argmax, plus one target token).
//
// The distributions are filtered to at most top_k <= 64 tokens, so the only
// vocabulary-wide work is a top-k per logits row: an HBM-bound read of
// (2K+1) rows of V fp32 per sequence.  One kernel does everything:
//  * chunk phase: CTA (chunk, row) reads 16384 logits (coalesced 16-byte
//    streaming loads), bounds the k-th largest from below by the minimum of
//    64 (or 32, 16) group maxima, keeps only elements at or above that bound
//    (typically ~1 % of them) as 64-bit keys (ordered float bits, then lower
//    token id), and writes the chunk's exact top-k sorted to the workspace;
//    chunks of finite logits do the maxima and the bound test in float and
//    build keys only for the kept elements (placed by warp ballots), chunks
//    holding a NaN or an infinity take the same steps on keys throughout:
//    with at most 512 candidates each thread ranks its own by counting the
//    larger keys; otherwise a block radix select finds the k-th key first;
//  * the last CTA of a sequence to finish (CTA barrier, then one acq_rel
//    atomic add by thread 0; no spinning) merges the per-chunk lists of each
//    row (one warp per row,
//    k-way merge) and runs the acceptance for that sequence in one warp:
//    softmax over the kept logits, top-p cut on the descending order,
//    u < p/q test, residual (p - q)+ sampled by inverse CDF in ascending
//    token-id order, bonus token.
// Each call clears the workspace's counter words on the stream before the
// launch, so a workspace needs no preparation and may be reused at any shape.
//
// spec_accept_lists takes the target rows as the per-CTA top-64 lists of a
// fused LM head ("MTP in llama.cpp": one evaluation boundary per cycle, the
// logits never travel through memory): a target row's chunk CTA then merges
// at most 32 of those sorted lists into its top-k instead of reading logits,
// and everything after the chunk phase is the same.
#include <cuda_runtime.h>

#include <algorithm>
#include <cfloat>
#include <cstdint>
#include <mutex>

#include "sv_device.cuh"
#include "sv_internal.h"

namespace sv {
namespace {

constexpr int kThreads = 512;
constexpr int kWarps = kThreads / 32;
constexpr int kChunk = 16384;                  // logits per chunk CTA
constexpr int kPerThread = kChunk / kThreads;  // 32
constexpr int kMaxTopK = 64;
constexpr int kCap = 2048;                     // candidate buffer entries
constexpr int kMaxChunks = 64;                 // V <= 64 * 16384
constexpr int kMaxK = 8;
constexpr int kMaxRows = 2 * kMaxK + 1;
constexpr int kStageBatch = 8;                 // candidate loads per lane in flight
constexpr int kManySequences = 8;              // from here on, three CTAs per SM

typedef unsigned long long u64;

struct AcceptArgs {
  const float *tl, *dl;
  const int32_t *dt;
  const float *ua, *us;
  int B, K, V;
  float temperature;
  int top_k;
  float top_p;
  int32_t *out, *nacc, *flags;
  u64 *cand;      // [B][rows_max][C][kMaxTopK]
  // target rows given as per-CTA top-64 lists of a fused LM head (or null):
  // per sequence, [G][K+1][kMaxTopK] keys then [G][K+1] flag words
  const u64 *tlists;
  long long tstride;  // u64 units per sequence
  int G;
  int *counters;  // [B]
  int *rowflags;  // [B][rows_max]
  int rows;       // rows read per sequence (K+1 greedy, 2K+1 sampling)
  int rows_max;   // 2K+1 (workspace stride)
  int C;          // chunks per row
  int ksel;       // tokens kept per row (1 greedy, top_k otherwise)
  int vec;        // 16-byte loads allowed
  int rows_per_wave;
};

struct WsLayout {
  size_t rowflags, cand, total;
};
// C: chunks per row (ceil(V / kChunk), more for target rows given as lists)
__host__ __device__ inline WsLayout ws_layout_c(int B, int K, size_t C) {
  const size_t rows_max = 2 * (size_t)K + 1;
  WsLayout L;
  L.rowflags = ((size_t)B * 4 + 15) / 16 * 16;
  L.cand = L.rowflags + ((size_t)B * rows_max * 4 + 15) / 16 * 16;
  L.total = L.cand + (size_t)B * rows_max * C * kMaxTopK * 8;
  return L;
}
__host__ __device__ inline WsLayout ws_layout(int B, int K, int V) {
  return ws_layout_c(B, K, ((size_t)V + kChunk - 1) / kChunk);
}
// chunks per row when the target rows come as G per-CTA lists: a chunk CTA
// of a target row merges at most kListsPerChunk lists
constexpr int kListsPerChunk = 32;
__host__ inline int lists_chunks(int V, int G) {
  const int cv = (V + kChunk - 1) / kChunk, cl = (G + kListsPerChunk - 1) / kListsPerChunk;
  return cv > cl ? cv : cl;
}

// ordered key of a logit: larger float -> larger key; 0 marks an excluded
// element (-inf mask, NaN, +inf; NaN and +inf also raise `nonfinite`)
__device__ __forceinline__ uint32_t logit_key(float v, int &nonfinite) {
  uint32_t u = __float_as_uint(v);
  if ((u & 0x7F800000u) == 0x7F800000u) {
    if ((u & 0x007FFFFFu) != 0 || (u >> 31) == 0) nonfinite = 1;
    return 0u;
  }
  if ((u & 0x7FFFFFFFu) == 0) u = 0;  // -0 and +0 compare equal
  return (u & 0x80000000u) ? ~u : (u | 0x80000000u);
}
__device__ __forceinline__ float key_logit(uint32_t k) {
  return __uint_as_float((k & 0x80000000u) ? (k & 0x7FFFFFFFu) : ~k);
}
// composite: key, then the lower token id wins ties
__device__ __forceinline__ u64 composite(uint32_t key, uint32_t idx) {
  return ((u64)key << 32) | (u64)(0xFFFFFFFFu - idx);
}
__device__ __forceinline__ int composite_id(u64 c) { return (int)(0xFFFFFFFFu - (uint32_t)c); }
__device__ __forceinline__ float composite_logit(u64 c) { return key_logit((uint32_t)(c >> 32)); }

struct ChunkSmem {
  u64 buf[kCap];
  u64 top[kMaxTopK];
  unsigned hist[256];
  uint32_t gmax[64];
  float gmaxf[64];
  uint32_t tau;
  float tauf;
  int nc, ntop, done, rem;
  u64 prefix;
  int last;
};

// Exact ksel-th largest among the keys each thread enumerates (all distinct,
// all nonzero): 8-bit radix passes from the top; stops as soon as the whole
// bin at the boundary belongs to the top set.  Returns the threshold T such
// that exactly min(ksel, total) keys are >= T.
template <class Each>
__device__ u64 block_select_threshold(ChunkSmem &S, int ksel, Each each) {
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  u64 prefix = 0, mask = 0;
  int rem = ksel;
  for (int pass = 0; pass < 8; ++pass) {
    const int shift = 56 - 8 * pass;
    for (int i = tid; i < 256; i += kThreads) S.hist[i] = 0;
    __syncthreads();
    each([&](u64 c) {
      if ((c & mask) == prefix) atomicAdd(&S.hist[(c >> shift) & 255u], 1u);
    });
    __syncthreads();
    if (warp == 0) {
      // lane l owns bins 255-8l ... 248-8l (descending)
      unsigned cnt[8], s = 0;
#pragma unroll
      for (int j = 0; j < 8; ++j) {
        cnt[j] = S.hist[255 - 8 * lane - j];
        s += cnt[j];
      }
      unsigned incl = s;
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        unsigned v = __shfl_up_sync(0xffffffffu, incl, o);
        if (lane >= o) incl += v;
      }
      const unsigned total = __shfl_sync(0xffffffffu, incl, 31);
      if (pass == 0 && total <= (unsigned)rem) {  // fewer keys than ksel: keep all
        if (lane == 0) {
          S.prefix = 0;
          S.done = 1;
          S.rem = 0;
        }
      } else {
        unsigned above = incl - s;
        int found = -1;
        unsigned above_at = 0, bin_cnt = 0;
#pragma unroll
        for (int j = 0; j < 8; ++j) {
          if (found < 0 && above < (unsigned)rem && (unsigned)rem <= above + cnt[j]) {
            found = 255 - 8 * lane - j;
            above_at = above;
            bin_cnt = cnt[j];
          }
          above += cnt[j];
        }
        if (found >= 0) {
          S.prefix = prefix | ((u64)found << shift);
          S.rem = rem - (int)above_at;
          S.done = (bin_cnt == (unsigned)(rem - (int)above_at)) ? 1 : 0;
        }
      }
    }
    __syncthreads();
    prefix = S.prefix;
    mask |= (u64)0xFF << shift;
    rem = S.rem;
    const int done = S.done;
    __syncthreads();
    if (done) break;
  }
  return prefix;
}

// Filtered distribution of one merged row held by a warp: entry j (sorted by
// logit, descending) lives in lane j & 31, half j >> 5.
struct RowDist {
  int id[2];
  float p[2];
  int n;  // entries with nonzero probability (0: empty)
};

__device__ RowDist row_dist(const u64 *top, int n, float temperature, float top_p) {
  const int lane = threadIdx.x & 31;
  RowDist D;
  D.n = n;
  float e[2] = {0.f, 0.f};
  const float zmax = n > 0 ? composite_logit(top[0]) : 0.f;
#pragma unroll
  for (int h = 0; h < 2; ++h) {
    const int j = lane + 32 * h;
    D.id[h] = -1;
    if (j < n) {
      D.id[h] = composite_id(top[j]);
      e[h] = expf((composite_logit(top[j]) - zmax) / temperature);
    }
  }
  const float S = warp_sum(e[0] + e[1]);
  D.p[0] = n > 0 ? e[0] / S : 0.f;
  D.p[1] = n > 0 ? e[1] / S : 0.f;
  if (n > 0 && top_p < 1.f) {
    const float c0 = warp_inclusive_scan(D.p[0]);
    const float t0 = __shfl_sync(0xffffffffu, c0, 31);
    const float c1 = warp_inclusive_scan(D.p[1]) + t0;
    const unsigned b0 = __ballot_sync(0xffffffffu, lane < n && c0 >= top_p);
    const unsigned b1 = __ballot_sync(0xffffffffu, lane + 32 < n && c1 >= top_p);
    int cut = n;
    if (b0) cut = __ffs(b0);
    else if (b1) cut = 32 + __ffs(b1);
    const int last = cut - 1;
    const float mass = __shfl_sync(0xffffffffu, last < 32 ? c0 : c1, last & 31);
    D.p[0] = lane < cut ? D.p[0] / mass : 0.f;
    D.p[1] = lane + 32 < cut ? D.p[1] / mass : 0.f;
    D.n = cut;
  }
  return D;
}

// A distribution stored by row_dist's warp (see the finish phase).
__device__ __forceinline__ RowDist stored_dist(const float *dist_p, const int *dist_id,
                                               const int *dist_n, int row) {
  const int lane = threadIdx.x & 31;
  RowDist D;
#pragma unroll
  for (int h = 0; h < 2; ++h) {
    D.p[h] = dist_p[row * 64 + lane + 32 * h];
    D.id[h] = dist_id[row * 64 + lane + 32 * h];
  }
  D.n = dist_n[row];
  return D;
}

__device__ float dist_lookup(const RowDist &D, int token) {
  const unsigned hit0 = __ballot_sync(0xffffffffu, D.id[0] == token && D.p[0] > 0.f);
  const unsigned hit1 = __ballot_sync(0xffffffffu, D.id[1] == token && D.p[1] > 0.f);
  float v = 0.f;
  if (hit0) v = __shfl_sync(0xffffffffu, D.p[0], __ffs(hit0) - 1);
  else if (hit1) v = __shfl_sync(0xffffffffu, D.p[1], __ffs(hit1) - 1);
  return token >= 0 ? v : 0.f;
}

// Smallest token id whose running sum of R (ascending id) exceeds u * sum(R);
// the last token with R > 0 if rounding never crosses; -1 if sum(R) <= 0.
// ids[h], R[h] as in RowDist, the same 64 ids also in shared memory (row_ids,
// read by every lane at once); scratch: 64 floats + 64 ints of warp smem.
__device__ int inverse_cdf_by_id(const int (&ids)[2], const float (&R)[2], float u, float *sR,
                                 int *sId, const int *row_ids) {
  const int lane = threadIdx.x & 31;
  // rank of each of the 64 slots by (token id, slot); id -1 (unused) sorts last
  int rank[2] = {0, 0};
  u64 mykey[2];
#pragma unroll
  for (int h = 0; h < 2; ++h) mykey[h] = ((u64)(uint32_t)ids[h] << 8) | (u64)(lane + 32 * h);
#pragma unroll 8
  for (int src = 0; src < 64; ++src) {
    const int other = row_ids[src];
    const u64 okey = ((u64)(uint32_t)other << 8) | (u64)src;
#pragma unroll
    for (int h = 0; h < 2; ++h) rank[h] += (okey < mykey[h]) ? 1 : 0;
  }
#pragma unroll
  for (int h = 0; h < 2; ++h) {
    sR[rank[h]] = (ids[h] >= 0) ? R[h] : 0.f;
    sId[rank[h]] = ids[h];
  }
  __syncwarp();
  const float r0 = sR[lane], r1 = sR[lane + 32];
  const float c0 = warp_inclusive_scan(r0);
  const float t0 = __shfl_sync(0xffffffffu, c0, 31);
  const float c1 = warp_inclusive_scan(r1) + t0;
  const float Z = __shfl_sync(0xffffffffu, c1, 31);
  int result = -1;
  if (Z > 0.f) {
    const float thr = u * Z;
    const unsigned x0 = __ballot_sync(0xffffffffu, r0 > 0.f && c0 > thr);
    const unsigned x1 = __ballot_sync(0xffffffffu, r1 > 0.f && c1 > thr);
    int pos = -1;
    if (x0) pos = __ffs(x0) - 1;
    else if (x1) pos = 32 + __ffs(x1) - 1;
    else {  // rounding: take the last entry with mass
      const unsigned l0 = __ballot_sync(0xffffffffu, r0 > 0.f);
      const unsigned l1 = __ballot_sync(0xffffffffu, r1 > 0.f);
      pos = l1 ? 32 + 31 - __clz(l1) : 31 - __clz(l0);
    }
    result = sId[pos];
  }
  __syncwarp();
  return result;
}

// kCtasPerSm: co-resident CTAs the register budget is cut for.  Three (40
// registers, a few spilled) hide more load latency when many sequences fill
// the GPU with chunk CTAs (batch 32: 74.0 -> 66.3 us); two keep the finish
// path, which one CTA per sequence runs, free of spills (batch 1: 19.5
// against 20.3 us).
template <int kCtasPerSm>
__global__ void __launch_bounds__(kThreads, kCtasPerSm) spec_accept_kernel(const AcceptArgs a) {
  extern __shared__ __align__(16) uint8_t smem_raw[];
  ChunkSmem &S = *reinterpret_cast<ChunkSmem *>(smem_raw);
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int row_g = blockIdx.y;
  const int b = row_g / a.rows, rloc = row_g % a.rows;
  const int cx = blockIdx.x;
  const int K = a.K, V = a.V;
  const float *row = rloc <= K ? a.tl + ((size_t)b * (K + 1) + rloc) * V
                               : a.dl + ((size_t)b * K + (rloc - K - 1)) * V;
  const int base = cx * kChunk;
  const int ksel = a.ksel;

  if (a.tlists != nullptr && rloc <= K) {
    // ---- target row from the fused LM head: chunk cx merges the per-CTA
    // lists g0..g1-1 of this row into its sorted top-ksel (each list is
    // sorted, so its first ksel keys are all it can contribute)
    const int g0 = (int)((long long)cx * a.G / a.C), g1 = (int)((long long)(cx + 1) * a.G / a.C);
    const int n = g1 - g0;
    const u64 *blk = a.tlists + (size_t)b * a.tstride;
    const unsigned *tfl = reinterpret_cast<const unsigned *>(blk + (size_t)a.G * (K + 1) * kMaxTopK);
    for (int i = tid; i < n * ksel; i += kThreads) {
      const int l = i / ksel, h = i - l * ksel;
      S.buf[i] = __ldcg(blk + ((size_t)(g0 + l) * (K + 1) + rloc) * kMaxTopK + h);
    }
    int nf = 0;
    for (int l = tid; l < n; l += kThreads) nf |= __ldcg(tfl + (size_t)(g0 + l) * (K + 1) + rloc) != 0u;
    const int any_nf = __syncthreads_or(nf);
    if (warp == 0) {
      u64 *dst = a.cand + ((size_t)b * a.rows_max + rloc) * (size_t)a.C * kMaxTopK +
                 (size_t)cx * kMaxTopK;
      int h0 = 0, h1 = 0;  // heads of lists lane and lane + 32
      int j = 0;
      for (; j < ksel; ++j) {
        const u64 v0 = (lane < n && h0 < ksel) ? S.buf[lane * ksel + h0] : 0ull;
        const u64 v1 = (lane + 32 < n && h1 < ksel) ? S.buf[(lane + 32) * ksel + h1] : 0ull;
        const u64 g = warp_max_u64(v0 > v1 ? v0 : v1);
        if (g == 0ull) break;
        if (v0 == g) ++h0;
        else if (v1 == g) ++h1;
        if (lane == 0) dst[j] = g;
      }
      for (int i = j + lane; i < ksel; i += 32) dst[i] = 0ull;  // empty slots
      if (lane == 0 && any_nf)
        atomicOr(&a.rowflags[b * a.rows_max + rloc], SV_FLAG_NONFINITE_LOGIT);
    }
  } else {
  // ---- load the chunk (values past V read as -inf: key 0, never kept) ------
  float v[kPerThread];
  float vsum = 0.f;  // finite iff every value of this thread's share is
  if (a.vec) {
#pragma unroll
    for (int i = 0; i < kPerThread / 4; ++i) {
      const int e = base + 4 * (tid + kThreads * i);
      float4 f = make_float4(-INFINITY, -INFINITY, -INFINITY, -INFINITY);
      if (e < V) {  // V % 4 == 0 on this path
        f = __ldcs(reinterpret_cast<const float4 *>(row + e));
        vsum += (f.x + f.y) + (f.z + f.w);
      }
      v[4 * i + 0] = f.x;
      v[4 * i + 1] = f.y;
      v[4 * i + 2] = f.z;
      v[4 * i + 3] = f.w;
    }
  } else {
#pragma unroll
    for (int i = 0; i < kPerThread; ++i) {
      const int e = base + tid + kThreads * i;
      v[i] = -INFINITY;
      if (e < V) {
        v[i] = __ldcs(row + e);
        vsum += v[i];
      }
    }
  }
  auto index_of = [&](int i) -> uint32_t {
    return a.vec ? (uint32_t)(base + 4 * (tid + kThreads * (i >> 2)) + (i & 3))
                 : (uint32_t)(base + tid + kThreads * i);
  };
  // Rows whose chunk holds a NaN or an infinity (a -inf mask included) take
  // the exact key path below; the others the float path, which keeps the same
  // candidates (the key map is monotone on finite values and maps -0 and +0
  // to one key) and computes keys only for them.
  int nonfinite = 0, dummy = 0;

  // ---- lower bound on the ksel-th largest: min over >= ksel group maxima --
  // (group maxima in float; the same barrier tells whether the chunk is
  // exotic, and only then are key maxima taken, behind one more barrier)
  const int n_groups = ksel <= 16 ? 16 : (ksel <= 32 ? 32 : 64);
  const int tpg = kThreads / n_groups;  // 32, 16 or 8 threads per group
  {
    float fmx = -INFINITY;
#pragma unroll
    for (int i = 0; i < kPerThread; ++i) fmx = fmaxf(fmx, v[i]);
    for (int o = 1; o < tpg; o <<= 1) fmx = fmaxf(fmx, __shfl_xor_sync(0xffffffffu, fmx, o));
    if ((tid % tpg) == 0) S.gmaxf[tid / tpg] = fmx;
  }
  if (tid == 0) S.nc = 0;
  const int exotic = __syncthreads_or(!(fabsf(vsum) <= FLT_MAX));
  if (exotic) {
    uint32_t tmax = 0;
#pragma unroll
    for (int i = 0; i < kPerThread; ++i) tmax = max(tmax, logit_key(v[i], nonfinite));
    for (int o = 1; o < tpg; o <<= 1) tmax = max(tmax, __shfl_xor_sync(0xffffffffu, tmax, o));
    if ((tid % tpg) == 0) S.gmax[tid / tpg] = tmax;
    __syncthreads();
  }
  if (warp == 0) {
    if (!exotic) {  // a group of padding only has maximum -inf
      const float g0 = lane < n_groups ? S.gmaxf[lane] : -INFINITY;
      const float g1 = lane + 32 < n_groups ? S.gmaxf[lane + 32] : -INFINITY;
      const int nz = __popc(__ballot_sync(0xffffffffu, g0 > -INFINITY)) +
                     __popc(__ballot_sync(0xffffffffu, g1 > -INFINITY));
      float mn = INFINITY;
      if (g0 > -INFINITY) mn = fminf(mn, g0);
      if (g1 > -INFINITY) mn = fminf(mn, g1);
      for (int o = 16; o > 0; o >>= 1) mn = fminf(mn, __shfl_xor_sync(0xffffffffu, mn, o));
      if (lane == 0) S.tauf = nz >= ksel ? mn : -FLT_MAX;  // else every finite value
    } else {
      const uint32_t g0 = lane < n_groups ? S.gmax[lane] : 0u;
      const uint32_t g1 = lane + 32 < n_groups ? S.gmax[lane + 32] : 0u;
      const int nz = __popc(__ballot_sync(0xffffffffu, g0 != 0)) +
                     __popc(__ballot_sync(0xffffffffu, g1 != 0));
      uint32_t mn = 0xFFFFFFFFu;
      if (g0) mn = min(mn, g0);
      if (g1) mn = min(mn, g1);
      for (int o = 16; o > 0; o >>= 1) mn = min(mn, __shfl_xor_sync(0xffffffffu, mn, o));
      if (lane == 0) S.tau = nz >= ksel ? mn : 1u;
    }
  }
  __syncthreads();

  // ---- keep the candidates at or above the bound ---------------------------
  if (!exotic) {
    // candidates are rare (~1 %): one ballot per value slot, and only a warp
    // that has some reserves places for them
    const float tauf = S.tauf;
    const unsigned below = (1u << lane) - 1u;
#pragma unroll
    for (int i = 0; i < kPerThread; ++i) {
      const bool keep = v[i] >= tauf;
      const unsigned m = __ballot_sync(0xffffffffu, keep);
      if (m) {
        int wb = 0;
        if (lane == 0) wb = atomicAdd(&S.nc, __popc(m));
        wb = __shfl_sync(0xffffffffu, wb, 0);
        const int pos = wb + __popc(m & below);
        if (keep && pos < kCap) S.buf[pos] = composite(logit_key(v[i], dummy), index_of(i));
      }
    }
  } else {
    const uint32_t tau = S.tau;
    int cnt = 0;
#pragma unroll
    for (int i = 0; i < kPerThread; ++i) cnt += logit_key(v[i], dummy) >= tau ? 1 : 0;
    int incl = cnt;
    for (int o = 1; o < 32; o <<= 1) {
      const int t = __shfl_up_sync(0xffffffffu, incl, o);
      if (lane >= o) incl += t;
    }
    int wbase = 0;
    if (lane == 31) wbase = atomicAdd(&S.nc, incl);
    wbase = __shfl_sync(0xffffffffu, wbase, 31);
    int pos = wbase + incl - cnt;
#pragma unroll
    for (int i = 0; i < kPerThread; ++i) {
      const uint32_t k = logit_key(v[i], dummy);
      if (k >= tau) {
        if (pos < kCap) S.buf[pos] = composite(k, index_of(i));
        ++pos;
      }
    }
  }
  const int any_nonfinite = __syncthreads_or(nonfinite);
  const int nc = S.nc;

  u64 *dst = a.cand + ((size_t)b * a.rows_max + rloc) * (size_t)a.C * kMaxTopK +
             (size_t)cx * kMaxTopK;
  if (nc <= kThreads) {
    // ---- usual case: one candidate per thread; its rank among the (distinct)
    // candidates is its place in the descending top-ksel list
    if (tid < nc) {
      const u64 mine = S.buf[tid];
      int rank = 0;
      for (int j = 0; j < nc; ++j) rank += S.buf[j] > mine ? 1 : 0;
      if (rank < ksel) dst[rank] = mine;
    }
    if (tid >= nc && tid < ksel) dst[tid] = 0;  // empty slots
  } else {
  // ---- exact top-ksel of the chunk -----------------------------------------
  u64 thr;
  if (nc <= kCap) {
    thr = block_select_threshold(S, ksel, [&](auto f) {
      for (int i = tid; i < nc; i += kThreads) f(S.buf[i]);
    });
    if (tid == 0) S.ntop = 0;
    __syncthreads();
    for (int i = tid; i < nc; i += kThreads) {
      const u64 c = S.buf[i];
      if (c >= thr) S.top[atomicAdd(&S.ntop, 1)] = c;
    }
  } else {  // many ties / a flat row: select over the whole chunk
    // (rare) the logits are read again from L2, so that the values need not
    // stay in registers through the selection
    auto key_again = [&](int i) -> uint32_t {
      const int e = (int)index_of(i);
      return e < V ? logit_key(__ldcg(row + e), dummy) : 0u;
    };
    thr = block_select_threshold(S, ksel, [&](auto f) {
#pragma unroll 4
      for (int i = 0; i < kPerThread; ++i) {
        const uint32_t k = key_again(i);
        if (k) f(composite(k, index_of(i)));
      }
    });
    if (tid == 0) S.ntop = 0;
    __syncthreads();
#pragma unroll 4
    for (int i = 0; i < kPerThread; ++i) {
      const uint32_t k = key_again(i);
      if (k) {
        const u64 c = composite(k, index_of(i));
        if (c >= thr) S.top[atomicAdd(&S.ntop, 1)] = c;
      }
    }
  }
  __syncthreads();
  const int ntop = S.ntop;
  // sort descending by rank (keys are distinct) and publish
  u64 mine = 0;
  int rank = 0;
  if (tid < ntop) {
    mine = S.top[tid];
    for (int j = 0; j < ntop; ++j) rank += S.top[j] > mine ? 1 : 0;
  }
  if (tid < ntop) dst[rank] = mine;
  else if (tid < ksel) dst[tid] = 0;  // empty slots
  }
  if (tid == 0 && any_nonfinite) atomicOr(&a.rowflags[b * a.rows_max + rloc], SV_FLAG_NONFINITE_LOGIT);
  }  // chunk of logits

  // ---- the last CTA of this sequence finishes it ---------------------------
  // every thread's candidate stores precede thread 0's release (CTA barrier,
  // then a cumulative acq_rel add); the last CTA acquires the others' lists
  __syncthreads();
  if (tid == 0) {
    int old;
    asm volatile("atom.acq_rel.gpu.global.add.s32 %0, [%1], 1;"
                 : "=r"(old)
                 : "l"(&a.counters[b])
                 : "memory");
    S.last = old == a.rows * a.C - 1;
  }
  __syncthreads();
  if (!S.last) return;

  // merge: one warp per row, rows in waves.  The chunk-phase buffers are dead
  // from here on; this region aliases them.
  u64 *merged = reinterpret_cast<u64 *>(smem_raw);              // [kMaxRows][kMaxTopK]
  int *mcount = reinterpret_cast<int *>(merged + kMaxRows * kMaxTopK);
  // each row's filtered distribution, built by the warp that merged it:
  // entry j at [row][j] (j = lane + 32 h of RowDist), and its support size
  float *dist_p = reinterpret_cast<float *>(mcount + kMaxRows + 1);  // [kMaxRows][64]
  int *dist_id = reinterpret_cast<int *>(dist_p + kMaxRows * 64);    // [kMaxRows][64]
  int *dist_n = dist_id + kMaxRows * 64;                             // [kMaxRows + 1]
  u64 *stage = reinterpret_cast<u64 *>(dist_n + kMaxRows + 1);  // [wave][C*ksel] (8-aligned)
  const int per_row = a.C * ksel;
  for (int r0 = 0; r0 < a.rows; r0 += a.rows_per_wave) {
    const int r = r0 + warp;
    const bool active = warp < a.rows_per_wave && r < a.rows;
    if (active) {
      u64 *st = stage + (size_t)warp * per_row;
      const u64 *src = a.cand + ((size_t)b * a.rows_max + r) * (size_t)a.C * kMaxTopK;
      // the row's lists, kStageBatch loads per lane in flight before their
      // shared-memory stores (a load issued after a store to a possibly
      // aliasing address would wait for it: one round trip per element)
      for (int i0 = 0; i0 < per_row; i0 += 32 * kStageBatch) {
        u64 v[kStageBatch];
#pragma unroll
        for (int u = 0; u < kStageBatch; ++u) {
          const int i = i0 + 32 * u + lane;
          v[u] = i < per_row ? __ldcg(src + (i / ksel) * kMaxTopK + i % ksel) : 0ull;
        }
#pragma unroll
        for (int u = 0; u < kStageBatch; ++u) {
          const int i = i0 + 32 * u + lane;
          if (i < per_row) st[i] = v[u];
        }
      }
      __syncwarp();
      int h0 = 0, h1 = 0;  // heads of lists lane and lane+32
      int j = 0;
      for (; j < ksel; ++j) {
        const u64 v0 = (lane < a.C && h0 < ksel) ? st[lane * ksel + h0] : 0ull;
        const u64 v1 = (lane + 32 < a.C && h1 < ksel) ? st[(lane + 32) * ksel + h1] : 0ull;
        const u64 best = v0 > v1 ? v0 : v1;
        const u64 g = warp_max_u64(best);
        if (g == 0ull) break;
        if (v0 == g) ++h0;
        else if (v1 == g) ++h1;
        if (lane == 0) merged[r * kMaxTopK + j] = g;
      }
      if (lane == 0) mcount[r] = j;
      if (a.temperature != 0.f) {  // the distribution, while the other rows merge
        __syncwarp();
        const RowDist D = row_dist(merged + r * kMaxTopK, j, a.temperature, a.top_p);
#pragma unroll
        for (int h = 0; h < 2; ++h) {
          dist_p[r * 64 + lane + 32 * h] = D.p[h];
          dist_id[r * 64 + lane + 32 * h] = D.id[h];
        }
        if (lane == 0) dist_n[r] = D.n;
      }
    }
    __syncthreads();
  }
  if (warp != 0) return;

  // ---- acceptance for sequence b (one warp) ---------------------------------
  float *sR = reinterpret_cast<float *>(stage);  // 64 floats
  int *sId = reinterpret_cast<int *>(sR + 64);   // 64 ints
  int flags = 0, nacc = 0;
  int emitted = -2;  // -2: none yet
  const bool greedy = a.temperature == 0.f;
  int32_t *out = a.out + (size_t)b * (K + 1);
  for (int j = lane; j <= K; j += 32) out[j] = -1;
  // every position's inputs at once, lane j holding position j (K <= 8):
  // draft token, uniform, and the flags of rows j (target) and K+1+j (draft);
  // lane K the bonus row's flags
  int d_l = 0, f_t = 0, f_d = 0;
  float ua_l = 0.f;
  if (lane < K) {
    d_l = a.dt[(size_t)b * K + lane];
    ua_l = a.ua[(size_t)b * K + lane];
    f_t = __ldcg(&a.rowflags[b * a.rows_max + lane]);
    if (!greedy) f_d = __ldcg(&a.rowflags[b * a.rows_max + K + 1 + lane]);
  } else if (lane == K) {
    f_t = __ldcg(&a.rowflags[b * a.rows_max + K]);
  }
  const float us_b = a.us[b];
  __syncwarp();
  int k = 0;
  for (; k < K; ++k) {
    const int d = __shfl_sync(0xffffffffu, d_l, k);
    const bool d_ok = d >= 0 && d < V;
    flags |= __shfl_sync(0xffffffffu, f_t, k);
    if (greedy) {
      const int am = mcount[k] > 0 ? composite_id(merged[k * kMaxTopK]) : -1;
      if (!d_ok) flags |= SV_FLAG_DRAFT_OUT_OF_RANGE;
      if (d_ok && am >= 0 && d == am) {
        if (lane == 0) out[k] = d;
        ++nacc;
        continue;
      }
      emitted = am;
      break;
    }
    flags |= __shfl_sync(0xffffffffu, f_d, k);
    const RowDist P = stored_dist(dist_p, dist_id, dist_n, k);
    const int qrow = K + 1 + k;
    const RowDist Q = stored_dist(dist_p, dist_id, dist_n, qrow);
    bool accept = false;
    if (!d_ok) {
      flags |= SV_FLAG_DRAFT_OUT_OF_RANGE;
    } else {
      const float qd = dist_lookup(Q, d);
      if (qd == 0.f) {
        flags |= SV_FLAG_DRAFT_ZERO_Q;
      } else {
        const float pd = dist_lookup(P, d);
        accept = __shfl_sync(0xffffffffu, ua_l, k) < pd / qd;
      }
    }
    if (accept) {
      if (lane == 0) out[k] = d;
      ++nacc;
      continue;
    }
    // residual max(0, p - q) over p's support (q's entries read from the
    // stored distribution, all lanes the same address: broadcast)
    float R[2] = {P.p[0], P.p[1]};
#pragma unroll 8
    for (int src = 0; src < 64; ++src) {
      const int qid = dist_id[qrow * 64 + src];
      const float qp = dist_p[qrow * 64 + src];
      if (qid >= 0 && qp > 0.f) {
#pragma unroll
        for (int h = 0; h < 2; ++h)
          if (P.id[h] == qid) R[h] = P.p[h] - qp;
      }
    }
#pragma unroll
    for (int h = 0; h < 2; ++h) R[h] = R[h] > 0.f ? R[h] : 0.f;
    const float Z = warp_sum(R[0] + R[1]);
    if (!(Z > 0.f)) {
      R[0] = P.p[0];
      R[1] = P.p[1];
    }
    emitted = inverse_cdf_by_id(P.id, R, us_b, sR, sId, dist_id + k * 64);
    break;
  }
  if (emitted == -2) {  // all K accepted: bonus from position K+1
    flags |= __shfl_sync(0xffffffffu, f_t, K);
    if (greedy) {
      emitted = mcount[K] > 0 ? composite_id(merged[K * kMaxTopK]) : -1;
    } else {
      const RowDist P = stored_dist(dist_p, dist_id, dist_n, K);
      float R[2] = {P.p[0], P.p[1]};
      emitted = inverse_cdf_by_id(P.id, R, us_b, sR, sId, dist_id + K * 64);
    }
  }
  if (emitted < 0) flags |= SV_FLAG_EMPTY_DIST;
  if (lane == 0) {
    out[nacc] = emitted;
    a.nacc[b] = nacc;
    if (a.flags) a.flags[b] = flags;
    a.counters[b] = 0;  // ready for the next call
  }
  for (int r = lane; r < a.rows_max; r += 32) a.rowflags[b * a.rows_max + r] = 0;
}

}  // namespace

unsigned take_device_error_accept() { return 0u; }  // no bounded waits in this unit

}  // namespace sv

using namespace sv;

extern "C" size_t spec_accept_workspace_bytes(int B, int K, int V) {
  if (B < 0 || K < 1 || V < 1) return 0;
  return ws_layout(B, K, V).total;
}

namespace sv {
namespace {

// Bytes of one sequence's block of per-CTA target lists (G CTAs, K+1 rows):
// keys [G][K+1][kMaxTopK] then flag words [G][K+1], rounded up to 16 bytes.
size_t lists_block_bytes(int G, int K) {
  const size_t b = (size_t)G * (K + 1) * (kMaxTopK * 8 + 4);
  return (b + 15) / 16 * 16;
}

// Both entry points: the target rows come either as logits or (target_lists
// non-null) as the per-CTA lists of a fused LM head.
sv_status accept_impl(const float *target_logits, const u64 *target_lists, int G,
                      const float *draft_logits, const int32_t *draft_tokens,
                      const float *u_accept, const float *u_sample, int B, int K, int V,
                      sv_sampling sampling, int32_t *out_tokens, int32_t *n_accepted,
                      int32_t *err_flags, void *workspace, size_t workspace_bytes,
                      sv_stream_t stream) {
  if (B < 0 || K < 1 || V < 1)
    return fail(SV_ERR_INVALID_ARG, "spec_accept: need B >= 0, K >= 1, V >= 1 (B=%d K=%d V=%d)", B,
                K, V);
  if (K > kMaxK) return fail(SV_ERR_UNSUPPORTED, "spec_accept: K=%d > %d", K, kMaxK);
  if ((long long)V > (long long)kMaxChunks * kChunk)
    return fail(SV_ERR_UNSUPPORTED, "spec_accept: V=%d > %d", V, kMaxChunks * kChunk);
  const bool greedy = sampling.temperature == 0.f;
  if (!(sampling.temperature >= 0.f) || !(sampling.temperature < 3.0e38f))
    return fail(SV_ERR_INVALID_ARG, "spec_accept: temperature must be finite and >= 0");
  if (!greedy) {
    if (sampling.top_k < 1 || sampling.top_k > kMaxTopK)
      return fail(SV_ERR_UNSUPPORTED, "spec_accept: top_k=%d outside [1, %d]", sampling.top_k,
                  kMaxTopK);
    if (!(sampling.top_p > 0.f) || !(sampling.top_p <= 1.f))
      return fail(SV_ERR_INVALID_ARG, "spec_accept: top_p must be in (0, 1]");
  }
  if (B == 0) return SV_OK;
  if ((long long)B * (2 * K + 1) > 65535)
    return fail(SV_ERR_UNSUPPORTED, "spec_accept: B*(2K+1) = %lld > 65535", (long long)B * (2 * K + 1));
  if ((!target_logits && !target_lists) || !draft_tokens || !u_accept || !u_sample ||
      !out_tokens || !n_accepted || !workspace || (!greedy && !draft_logits))
    return fail(SV_ERR_INVALID_ARG, "spec_accept: null pointer");
  if (target_lists) {
    if (G < 1 || G > kListsPerChunk * kMaxChunks)
      return fail(SV_ERR_UNSUPPORTED, "spec_accept_lists: G=%d outside [1, %d]", G,
                  kListsPerChunk * kMaxChunks);
    if (!aligned(target_lists, 16))
      return fail(SV_ERR_INVALID_ARG, "spec_accept_lists: target_lists must be 16-byte aligned");
  }
  const int C = target_lists ? lists_chunks(V, G) : (V + kChunk - 1) / kChunk;
  static_assert(kListsPerChunk * kMaxTopK <= kCap, "a chunk's lists fit the candidate buffer");
  const WsLayout W = ws_layout_c(B, K, (size_t)C);
  if (workspace_bytes < W.total)
    return fail(SV_ERR_INVALID_ARG, "spec_accept: workspace of %zu bytes, need %zu",
                workspace_bytes, W.total);
  if (!aligned(workspace, 16)) return fail(SV_ERR_INVALID_ARG, "spec_accept: workspace must be 16-byte aligned");
  if ((target_logits && !aligned(target_logits, 4)) || (draft_logits && !aligned(draft_logits, 4)) ||
      !aligned(draft_tokens, 4) || !aligned(u_accept, 4) || !aligned(u_sample, 4) ||
      !aligned(out_tokens, 4) || !aligned(n_accepted, 4) || (err_flags && !aligned(err_flags, 4)))
    return fail(SV_ERR_INVALID_ARG, "spec_accept: misaligned pointer");
  const size_t tlb = target_lists ? (size_t)B * lists_block_bytes(G, K) : (size_t)B * (K + 1) * V * 4;
  const size_t dlb = (size_t)B * K * V * 4;
  const size_t ob = (size_t)B * (K + 1) * 4, nb = (size_t)B * 4;
  const void *ins[5] = {target_lists ? static_cast<const void *>(target_lists) : target_logits,
                        draft_logits, draft_tokens, u_accept, u_sample};
  const size_t insb[5] = {tlb, greedy ? 0 : dlb, (size_t)B * K * 4, (size_t)B * K * 4, nb};
  const void *outs[4] = {out_tokens, n_accepted, err_flags, workspace};
  const size_t outsb[4] = {ob, nb, err_flags ? nb : 0, W.total};
  for (int i = 0; i < 4; ++i) {
    for (int j = 0; j < 5; ++j)
      if (overlaps(outs[i], outsb[i], ins[j], insb[j]))
        return fail(SV_ERR_INVALID_ARG, "spec_accept: an output overlaps an input");
    for (int j = i + 1; j < 4; ++j)
      if (overlaps(outs[i], outsb[i], outs[j], outsb[j]))
        return fail(SV_ERR_INVALID_ARG, "spec_accept: outputs overlap");
  }

  AcceptArgs args;
  args.tl = target_logits;
  args.tlists = target_lists;
  args.tstride = target_lists ? (long long)(lists_block_bytes(G, K) / 8) : 0;
  args.G = G;
  args.dl = draft_logits;
  args.dt = draft_tokens;
  args.ua = u_accept;
  args.us = u_sample;
  args.B = B;
  args.K = K;
  args.V = V;
  args.temperature = sampling.temperature;
  args.top_k = sampling.top_k;
  args.top_p = sampling.top_p;
  args.out = out_tokens;
  args.nacc = n_accepted;
  args.flags = err_flags;
  uint8_t *ws = static_cast<uint8_t *>(workspace);
  args.counters = reinterpret_cast<int *>(ws);
  args.rowflags = reinterpret_cast<int *>(ws + W.rowflags);
  args.cand = reinterpret_cast<u64 *>(ws + W.cand);
  args.rows = greedy ? K + 1 : 2 * K + 1;
  args.rows_max = 2 * K + 1;
  args.C = C;
  args.ksel = greedy ? 1 : std::min(sampling.top_k, V);
  args.vec = (V % 4 == 0) && (target_lists || aligned(target_logits, 16)) &&
             (greedy || aligned(draft_logits, 16));
  // final-phase staging: one warp per row, C*ksel keys each, at most 48 KB
  const size_t per_row = (size_t)args.C * args.ksel * 8;
  args.rows_per_wave = (int)std::max<size_t>(
      1, std::min<size_t>({(size_t)args.rows, (size_t)kWarps, (size_t)(48 * 1024) / per_row}));
  const size_t final_bytes = (size_t)kMaxRows * kMaxTopK * 8 + (kMaxRows + 1) * 4 +
                             (size_t)kMaxRows * 64 * 8 + (kMaxRows + 1) * 4 +
                             std::max<size_t>((size_t)args.rows_per_wave * per_row, 64 * 8);
  const size_t smem = std::max(sizeof(ChunkSmem), final_bytes);
  static PerDeviceOnce attrs_once;
  const cudaError_t ce = attrs_once.run([] {
    cudaError_t e = cudaFuncSetAttribute(spec_accept_kernel<2>,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize, 160 * 1024);
    if (e == cudaSuccess)
      e = cudaFuncSetAttribute(spec_accept_kernel<3>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                               160 * 1024);
    return e;
  });
  if (ce != cudaSuccess)
    return fail(SV_ERR_CUDA, "spec_accept: cudaFuncSetAttribute failed: %s", cudaGetErrorString(ce));
  // Counters and row flags start at zero.  Where they sit depends on B and
  // K, and a completed call clears only its own, so a workspace last used at
  // another shape may hold candidate keys there: clear them on the stream.
  if (cudaMemsetAsync(workspace, 0, W.cand, reinterpret_cast<cudaStream_t>(stream)) != cudaSuccess)
    return fail(SV_ERR_CUDA, "spec_accept: clearing the workspace counters failed: %s",
                cudaGetErrorString(cudaGetLastError()));
  dim3 grid((unsigned)args.C, (unsigned)(B * args.rows));
  if (B >= kManySequences)
    spec_accept_kernel<3><<<grid, kThreads, smem, reinterpret_cast<cudaStream_t>(stream)>>>(args);
  else
    spec_accept_kernel<2><<<grid, kThreads, smem, reinterpret_cast<cudaStream_t>(stream)>>>(args);
  return check_launch("spec_accept");
}

}  // namespace
}  // namespace sv

extern "C" sv_status spec_accept(const float *target_logits, const float *draft_logits,
                                 const int32_t *draft_tokens, const float *u_accept,
                                 const float *u_sample, int B, int K, int V, sv_sampling sampling,
                                 int32_t *out_tokens, int32_t *n_accepted, int32_t *err_flags,
                                 void *workspace, size_t workspace_bytes, sv_stream_t stream) {
  clear_error();
  if (!target_logits && B > 0) return fail(SV_ERR_INVALID_ARG, "spec_accept: null pointer");
  return accept_impl(target_logits, nullptr, 0, draft_logits, draft_tokens, u_accept, u_sample,
                     B, K, V, sampling, out_tokens, n_accepted, err_flags, workspace,
                     workspace_bytes, stream);
}

extern "C" size_t spec_accept_lists_workspace_bytes(int B, int K, int V, int G) {
  if (B < 0 || K < 1 || V < 1 || G < 1) return 0;
  return ws_layout_c(B, K, (size_t)lists_chunks(V, G)).total;
}

extern "C" size_t spec_accept_lists_block_bytes(int G, int K) {
  if (G < 1 || K < 1) return 0;
  return lists_block_bytes(G, K);
}

extern "C" sv_status spec_accept_lists(const uint64_t *target_lists, int G,
                                       const float *draft_logits, const int32_t *draft_tokens,
                                       const float *u_accept, const float *u_sample, int B, int K,
                                       int V, sv_sampling sampling, int32_t *out_tokens,
                                       int32_t *n_accepted, int32_t *err_flags, void *workspace,
                                       size_t workspace_bytes, sv_stream_t stream) {
  clear_error();
  if (!target_lists && B > 0) return fail(SV_ERR_INVALID_ARG, "spec_accept_lists: null pointer");
  return accept_impl(nullptr, reinterpret_cast<const u64 *>(target_lists), G, draft_logits,
                     draft_tokens, u_accept, u_sample, B, K, V, sampling, out_tokens, n_accepted,
                     err_flags, workspace, workspace_bytes, stream);
}

// ---- spec_accept_noalloc: the same call on a fixed, statically sized scratch --
//
// For callers that cannot allocate device memory: a plain C host loop that
// links only this library and owns no device allocator, or a decode loop that
// must not call cudaMalloc / cudaFree per step (cudaFree synchronises the
// whole device).  The scratch is one file-scope __device__ array, so there is
// exactly one per device: calls that overlap in time (two streams, two host
// threads) race on it.  The first call on a device looks up the array's
// address; make that first call before any stream capture begins.
namespace sv {
namespace {

constexpr size_t kStaticScratchBytes = size_t(2) << 20;  // 2 MiB
__device__ __align__(256) unsigned char g_accept_scratch[kStaticScratchBytes];

constexpr int kScratchDevices = 64;
std::mutex g_scratch_mu;
void *g_scratch_ptr[kScratchDevices] = {};

// Address of g_accept_scratch on the current device (looked up once per device).
sv_status static_scratch(void **out) {
  int dev = -1;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kScratchDevices)
    return fail(SV_ERR_CUDA, "spec_accept_noalloc: no usable current device");
  std::lock_guard<std::mutex> lock(g_scratch_mu);
  if (!g_scratch_ptr[dev]) {
    void *p = nullptr;
    const cudaError_t e = cudaGetSymbolAddress(&p, g_accept_scratch);
    if (e != cudaSuccess || !p)
      return fail(SV_ERR_CUDA, "spec_accept_noalloc: cudaGetSymbolAddress failed on device %d: %s",
                  dev, cudaGetErrorString(e));
    g_scratch_ptr[dev] = p;
  }
  *out = g_scratch_ptr[dev];
  return SV_OK;
}

}  // namespace
}  // namespace sv

extern "C" size_t spec_accept_noalloc_scratch_bytes(void) { return kStaticScratchBytes; }

extern "C" sv_status spec_accept_noalloc(const float *target_logits, const float *draft_logits,
                                         const int32_t *draft_tokens, const float *u_accept,
                                         const float *u_sample, int B, int K, int V,
                                         sv_sampling sampling, int32_t *out_tokens,
                                         int32_t *n_accepted, int32_t *err_flags,
                                         sv_stream_t stream) {
  clear_error();
  // Sizes spec_accept rejects anyway (and B == 0, a no-op) go straight to it.
  if (B <= 0 || K < 1 || K > kMaxK || V < 1 || (long long)V > (long long)kMaxChunks * kChunk)
    return spec_accept(target_logits, draft_logits, draft_tokens, u_accept, u_sample, B, K, V,
                       sampling, out_tokens, n_accepted, err_flags, nullptr, 0, stream);
  const WsLayout W = ws_layout(B, K, V);
  if (W.total > kStaticScratchBytes)
    return fail(SV_ERR_UNSUPPORTED,
                "spec_accept_noalloc: B=%d K=%d V=%d needs %zu bytes of scratch, the static "
                "scratch holds %zu; use spec_accept with a caller workspace",
                B, K, V, W.total, kStaticScratchBytes);
  void *scratch = nullptr;
  const sv_status st = static_scratch(&scratch);
  if (st != SV_OK) return st;
  // spec_accept clears the counter words it needs on the stream, whatever
  // shape the previous call on the scratch had
  return spec_accept(target_logits, draft_logits, draft_tokens, u_accept, u_sample, B, K, V,
                     sampling, out_tokens, n_accepted, err_flags, scratch, kStaticScratchBytes,
                     stream);
}
