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
// (2K+1) rows of V fp32 per sequence, in chunks of 16384 logits.
//  * chunk selection (chunk_select): the chunk's exact top-k, sorted, as
//    64-bit keys (ordered float bits, then lower token id) in the workspace.
//    The k-th largest of 32 (64 when k > 32) group maxima bounds the chunk's
//    k-th largest from below (k distinct logits reach it); only elements at
//    or above it are kept (typically a few more than k of the 16384), found
//    through the threads whose maximum reaches the bound, and placed by
//    counting larger keys.  Chunks of finite logits work in float and build
//    keys only for kept elements; chunks holding a NaN or +inf work on keys
//    throughout; many kept elements go through a radix select.
//  * finish (finish_sequence), one CTA per sequence: each row's chunk lists
//    merged into its top-k (a warp per row: the top-k of the lists' first
//    few entries bounds the rest from below), softmax over the kept logits,
//    top-p cut on the descending order, and then every position at once (a
//    warp each): the u < p/q test and the residual (p - q)+ sampled by
//    inverse CDF in ascending token-id order; the walk to the first
//    rejection picks the emitted token (the bonus row's sample when all K
//    are accepted).
// Launches: 16-byte-aligned logits go through accept_stream_kernel (a
// persistent CTA per SM, chunks streamed through a ring of bulk copies into
// shared memory, two groups of 256 threads selecting alternate chunks) and
// then accept_finish_kernel (a CTA per sequence).  Other logits, and the
// target lists of a fused LM head, go through spec_accept_kernel, a CTA per
// (chunk, row) whose last CTA of a sequence runs the finish.
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
#include <type_traits>

#include "sv_device.cuh"
#include "sv_internal.h"

namespace sv {
namespace {

constexpr int kThreads = 512;
constexpr int kWarps = kThreads / 32;
constexpr int kChunk = 16384;                  // logits per chunk CTA
constexpr int kPerThread = kChunk / kThreads;  // 32
constexpr int kMaxTopK = 64;
constexpr int kMaxChunks = 64;                 // V <= 64 * 16384
constexpr int kMaxK = 8;
constexpr int kMaxRows = 2 * kMaxK + 1;
constexpr int kStageBatch = 8;                 // candidate loads per lane in flight
constexpr int kFewCandidates = 64;             // packed and ranked by one warp up to here
constexpr int kMergeBuf = 256;                 // per-warp merge keys (else k-way merge)
constexpr int kStreamStages = 3;               // chunks in flight per streaming CTA
constexpr size_t kStreamRingBytes = (size_t)kStreamStages * kChunk * 4;
constexpr int kAccInWords = 2 * kMaxK + kMaxRows + 1 + 6;  // acceptance inputs, 8-byte multiple
static_assert(kAccInWords % 2 == 0, "the staging area after the inputs stays 8-aligned");
static_assert(kPerThread == 32, "a candidate holder's values are one per lane");
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
// max(a, b, c), NaN if any operand is NaN
__device__ __forceinline__ float max3_nan(float a, float b, float c) {
  float d;
  asm("max.NaN.f32 %0, %1, %2, %3;" : "=f"(d) : "f"(a), "f"(b), "f"(c));
  return d;
}
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

// Who selects one chunk: kGT threads (kGW warps) holding kPT logits each.
template <int kGT_, int kPT_>
struct SelGeo {
  static constexpr int kGT = kGT_, kGW = kGT_ / 32, kPT = kPT_;
  static_assert(kGT_ * kPT_ == kChunk && kPT_ % 32 == 0, "a chunk, whole rows of 32 per thread");
};
using CtaGeo = SelGeo<kThreads, kPerThread>;  // a CTA per chunk
using GroupGeo = SelGeo<256, 64>;               // a group of a streaming CTA

// Shared memory of one chunk's selection.  kCapT: candidate buffer entries,
// kSeg of them per warp; kRowsT: candidate holders a warp tests at once.
template <class G, int kCapT, int kRowsT>
struct ChunkSmemT {
  static constexpr int kSeg = kCapT / G::kGW;
  static constexpr int kHolderRows = kRowsT;
  u64 buf[kCapT];
  u64 top[kMaxTopK];
  unsigned hist[256];
  uint32_t gmax[64];
  float gmaxf[64];
  // candidate holders' values, per warp; rows padded by 16 bytes so that the
  // holders' simultaneous 16-byte stores fall in different banks
  float scratch[G::kGW][kRowsT][G::kPT + 4];
  uint32_t tau;               // the bound, as a key (exotic chunks) or a float
  float tauf;
  alignas(16) int wcount[G::kGW];      // candidates each warp found
  alignas(16) u64 few[kFewCandidates + 2];  // the candidates, packed, when few
  int ntop, done, rem;
  u64 prefix;
};
using ChunkSmem = ChunkSmemT<CtaGeo, 2048, 4>;    // a CTA per chunk
using StreamSmem = ChunkSmemT<GroupGeo, 512, 4>;  // each group of a streaming CTA

// Barriers over the threads that select one chunk: the whole CTA, or one of
// the kThreads-thread groups of a CTA (a named barrier).
struct CtaBarrier {
  __device__ __forceinline__ void sync() const { __syncthreads(); }
  __device__ __forceinline__ int sync_or(int p) const { return __syncthreads_or(p); }
};
template <int kCount>
struct GroupBarrier {
  int id;  // 1 + group: barrier 0 is __syncthreads
  __device__ __forceinline__ void sync() const {
    asm volatile("bar.sync %0, %1;" ::"r"(id), "n"(kCount) : "memory");
  }
  __device__ __forceinline__ int sync_or(int p) const {
    int r;
    asm volatile(
        "{\n\t.reg .pred q, o;\n\t"
        "setp.ne.s32 q, %1, 0;\n\t"
        "bar.red.or.pred o, %2, %3, q;\n\t"
        "selp.s32 %0, 1, 0, o;\n\t}"
        : "=r"(r)
        : "r"(p), "r"(id), "n"(kCount)
        : "memory");
    return r;
  }
};

// Exact ksel-th largest among the keys each thread enumerates (all distinct,
// all nonzero): 8-bit radix passes from the top; stops as soon as the whole
// bin at the boundary belongs to the top set.  Returns the threshold T such
// that exactly min(ksel, total) keys are >= T.
template <class G, class Smem, class Bar, class Each>
__device__ u64 block_select_threshold(Smem &S, int ksel, int tid, const Bar &bar, Each each) {
  const int lane = tid & 31, warp = tid >> 5;
  u64 prefix = 0, mask = 0;
  int rem = ksel;
  for (int pass = 0; pass < 8; ++pass) {
    const int shift = 56 - 8 * pass;
    for (int i = tid; i < 256; i += G::kGT) S.hist[i] = 0;
    bar.sync();
    each([&](u64 c) {
      if ((c & mask) == prefix) atomicAdd(&S.hist[(c >> shift) & 255u], 1u);
    });
    bar.sync();
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
    bar.sync();
    prefix = S.prefix;
    mask |= (u64)0xFF << shift;
    rem = S.rem;
    const int done = S.done;
    bar.sync();
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
// ids[h], R[h] as in RowDist: the first n slots hold the row's distinct
// token ids (also in shared memory, row_ids, read by every lane at once), the
// others id -1 and no mass; scratch: 64 floats + 64 ints of warp smem.  The
// slots are placed in ascending id order, the unused ones last.
__device__ int inverse_cdf_by_id(const int (&ids)[2], const float (&R)[2], int n, float u,
                                 float *sR, int *sId, const int *row_ids) {
  const int lane = threadIdx.x & 31;
  // rank of each of the first n slots by token id; the unused ones keep
  // their places past n
  int rank[2] = {lane, lane + 32};
  if (n > 0) {
    int cnt[2] = {0, 0};
#pragma unroll 4
    for (int src = 0; src < n; ++src) {
      const int other = row_ids[src];
#pragma unroll
      for (int h = 0; h < 2; ++h) cnt[h] += (other < ids[h]) ? 1 : 0;
    }
#pragma unroll
    for (int h = 0; h < 2; ++h)
      if (lane + 32 * h < n) rank[h] = cnt[h];
  }
#pragma unroll
  for (int h = 0; h < 2; ++h) {
    const bool live = lane + 32 * h < n;
    sR[rank[h]] = live ? R[h] : 0.f;
    sId[rank[h]] = live ? ids[h] : -1;
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

// Bitonic sort of 64 values held two per lane (element lane in v[0], element
// lane + 32 in v[1]) into descending order.
template <class T>
__device__ __forceinline__ void bitonic64_desc(T (&v)[2], int lane) {
#pragma unroll
  for (int k = 2; k <= 64; k <<= 1) {
#pragma unroll
    for (int j = k >> 1; j > 0; j >>= 1) {
      T o[2];
      if (j == 32) {
        o[0] = v[1];
        o[1] = v[0];
      } else {
        o[0] = __shfl_xor_sync(0xffffffffu, v[0], j);
        o[1] = __shfl_xor_sync(0xffffffffu, v[1], j);
      }
#pragma unroll
      for (int h = 0; h < 2; ++h) {
        const int i = lane + 32 * h;
        // in a block sorted descending (i & k == 0) the lower index of each
        // pair keeps the larger value
        const bool keep_max = ((i & j) == 0) == ((i & k) == 0);
        const T mx = v[h] > o[h] ? v[h] : o[h], mn = v[h] > o[h] ? o[h] : v[h];
        v[h] = keep_max ? mx : mn;
      }
    }
  }
}

// The k-th largest (1-based, counted with multiplicity) of the kN (32 or 64)
// values vals[0, kN) in shared memory (16-byte aligned), by one warp: lane j
// tests vals[j] (and vals[j + 32]), counting the values above it and at or
// above it through broadcast reads, and the value v with (# > v) <= k-1 < (#
// >= v) is the answer.  Every lane returns it.  (The loop is unrolled so
// that all reads are in flight at once.)
template <int kN, class T>
__device__ __forceinline__ T warp_kth_largest(const T *vals, int k) {
  static_assert(sizeof(T) == 4 && (kN == 32 || kN == 64), "32 or 64 32-bit values");
  const int lane = threadIdx.x & 31;
  constexpr int kH = kN / 32;
  T g[kH];
  int gt[kH], ge[kH];
#pragma unroll
  for (int h = 0; h < kH; ++h) {
    g[h] = vals[lane + 32 * h];
    gt[h] = 0;
    ge[h] = 0;
  }
#pragma unroll
  for (int q = 0; q < kN; q += 4) {
    const uint4 w = *reinterpret_cast<const uint4 *>(vals + q);
    const T o[4] = {reinterpret_cast<const T &>(w.x), reinterpret_cast<const T &>(w.y),
                    reinterpret_cast<const T &>(w.z), reinterpret_cast<const T &>(w.w)};
#pragma unroll
    for (int e = 0; e < 4; ++e)
#pragma unroll
      for (int h = 0; h < kH; ++h) {
        gt[h] += o[e] > g[h] ? 1 : 0;
        ge[h] += o[e] >= g[h] ? 1 : 0;
      }
  }
  T r = g[0];
  bool found = false;
#pragma unroll
  for (int h = 0; h < kH; ++h) {
    const unsigned m = __ballot_sync(0xffffffffu, gt[h] <= k - 1 && k - 1 < ge[h]);
    const T v = __shfl_sync(0xffffffffu, g[h], m ? __ffs(m) - 1 : 0);
    if (!found && m) {
      r = v;
      found = true;
    }
  }
  return r;
}
// Order-preserving map of a float (not NaN) to a 32-bit unsigned.
__device__ __forceinline__ uint32_t float_order(float f) {
  const uint32_t u = __float_as_uint(f);
  return (u & 0x80000000u) ? ~u : (u | 0x80000000u);
}

// The exact top-ksel of one chunk of a logits row, sorted descending, into
// dst[0, ksel) (empty slots 0), by kThreads threads (thread index tid, all
// of them behind the barrier bar).  Thread t holds in v[i] the
// logit of token index_at(t, i) (-inf past V).  A CTA may call it for one
// chunk after another: every shared word a call writes was last read, in the
// previous call, before the first barrier of this one.  `extra` (per thread) is OR-ed into the first CTA barrier as bit 1 of its
// vote, and `after_first` runs in every thread right after that barrier with
// the vote.  Returns, in every thread, whether the chunk held a NaN or +inf.
template <class G, class Smem, class Bar, class After>
__device__ int chunk_select(Smem &S, const float (&v)[G::kPT], const float *row, int V, int base,
                            bool vec, int ksel, u64 *dst, int tid, const Bar &bar, int extra,
                            After after_first) {
  constexpr int kGT = G::kGT, kPT = G::kPT, kQ = kPT / 32;
  constexpr int kSeg = Smem::kSeg, kHolderRows = Smem::kHolderRows;
  const int lane = tid & 31, warp = tid >> 5;
  // token id of value slot i of thread t
  auto index_at = [&](int t, int i) -> uint32_t {
    return vec ? (uint32_t)(base + 4 * (t + kGT * (i >> 2)) + (i & 3))
               : (uint32_t)(base + t + kGT * i);
  };
  auto index_of = [&](int i) -> uint32_t { return index_at(tid, i); };
  // slot lane + 32 q of thread t: base + t * t_mul + slot_off[q]
  const int t_mul = vec ? 4 : 1;
  int slot_off[kQ];
#pragma unroll
  for (int q = 0; q < kQ; ++q) {
    const int i = lane + 32 * q;
    slot_off[q] = vec ? 4 * kGT * (i >> 2) + (i & 3) : kGT * i;
  }
  // Chunks holding a NaN or a +inf take the exact key path below; the others
  // the float path, which keeps the same candidates (the key map is monotone
  // on finite values, maps -0 and +0 to one key and -inf, a mask, to the
  // never-kept key 0) and computes keys only for them.  The thread maximum
  // propagates NaN, so one test finds both.
  int nonfinite = 0, dummy = 0;

  // ---- lower bound on the ksel-th largest: the ksel-th largest of the group
  // maxima (ksel distinct logits reach it), 32 groups of threads when
  // ksel <= 32, else 64, found by warp 0.
  const int n_groups = ksel <= 32 ? 32 : 64;
  const int tpg = kGT / n_groups;
  float tmx = v[0];  // this thread's maximum (NaN if it holds one)
#pragma unroll
  for (int i = 1; i + 1 < kPT; i += 2) tmx = max3_nan(tmx, v[i], v[i + 1]);
  tmx = max3_nan(tmx, v[kPT - 1], v[kPT - 1]);
  {
    float fmx = tmx;
    for (int o = 1; o < tpg; o <<= 1) fmx = fmaxf(fmx, __shfl_xor_sync(0xffffffffu, fmx, o));
    if ((tid % tpg) == 0) S.gmaxf[tid / tpg] = fmx;
  }
  const int vote = bar.sync_or((!(tmx <= FLT_MAX) ? 1 : 0) | (extra ? 2 : 0));
  after_first(vote);
  const bool exotic = vote & 1;
  if (exotic) {  // (rare) key maxima, behind one more barrier
    uint32_t tmax = 0;
#pragma unroll
    for (int i = 0; i < kPT; ++i) tmax = max(tmax, logit_key(v[i], nonfinite));
    for (int o = 1; o < tpg; o <<= 1) tmax = max(tmax, __shfl_xor_sync(0xffffffffu, tmax, o));
    if ((tid % tpg) == 0) S.gmax[tid / tpg] = tmax;
    bar.sync();
  }

  if (warp == 0) {
    if (!exotic) {
      float tauf;
      const float g0 = S.gmaxf[lane];
      // groups holding a value above -inf (padding and masks only: -inf)
      const int nz = __popc(__ballot_sync(0xffffffffu, g0 > -INFINITY)) +
                     (n_groups > 32 ? __popc(__ballot_sync(0xffffffffu, S.gmaxf[lane + 32] > -INFINITY))
                                    : 0);
      if (ksel == 1) {  // the largest: one warp reduction on the ordered bits
        const uint32_t mo = __reduce_max_sync(0xffffffffu, float_order(g0));
        tauf = __shfl_sync(0xffffffffu, g0, __ffs(__ballot_sync(0xffffffffu, float_order(g0) == mo)) - 1);
      } else {
        tauf = n_groups == 32 ? warp_kth_largest<32>(S.gmaxf, ksel)
                              : warp_kth_largest<64>(S.gmaxf, ksel);
      }
      if (lane == 0) S.tauf = nz >= ksel ? tauf : -FLT_MAX;  // else every finite value
    } else {
      const int nz = __popc(__ballot_sync(0xffffffffu, S.gmax[lane] != 0u)) +
                     (n_groups > 32 ? __popc(__ballot_sync(0xffffffffu, S.gmax[lane + 32] != 0u)) : 0);
      const uint32_t tau =
          n_groups == 32 ? warp_kth_largest<32>(S.gmax, ksel) : warp_kth_largest<64>(S.gmax, ksel);
      if (lane == 0) S.tau = nz >= ksel ? tau : 1u;  // else every key
    }
  }
  bar.sync();

  // ---- keep the candidates at or above the bound ---------------------------
  // each warp appends its candidates to its own segment of S.buf, without
  // atomics, and publishes how many it found
  u64 *seg = S.buf + warp * kSeg;
  if (!exotic) {
    const float tauf = S.tauf;
    // candidates are rare (a few per warp): only threads whose maximum
    // reaches the bound hold any.  Up to kHolderRows of them at a time put
    // their values in rows of the warp's scratch, and the warp tests the
    // rows, lane l taking slots l, l + 32, ...; each kept value takes a place
    // in the warp's segment with a shared atomic add (a value or two per row:
    // little contention).
    if (lane == 0) S.wcount[warp] = 0;
    __syncwarp();
    unsigned holders = __ballot_sync(0xffffffffu, tmx >= tauf);
    while (holders) {
      const int hrank = __popc(holders & ((1u << lane) - 1u));
      if (((holders >> lane) & 1u) && hrank < kHolderRows) {
        float *row_s = S.scratch[warp][hrank];
#pragma unroll
        for (int i = 0; i < kPT; i += 4)
          *reinterpret_cast<float4 *>(row_s + i) = make_float4(v[i], v[i + 1], v[i + 2], v[i + 3]);
      }
      int th[kHolderRows];  // the batch's holders
#pragma unroll
      for (int h = 0; h < kHolderRows; ++h) {
        th[h] = holders ? __ffs(holders) - 1 : -1;
        holders &= holders - 1u;
      }
      __syncwarp();
#pragma unroll
      for (int h = 0; h < kHolderRows; ++h) {
        if (th[h] < 0) break;  // (warp-uniform)
        const int tb = base + (warp * 32 + th[h]) * t_mul;
#pragma unroll
        for (int q = 0; q < kQ; ++q) {
          const float x = S.scratch[warp][h][lane + 32 * q];
          if (x >= tauf) {
            const int pos = atomicAdd(&S.wcount[warp], 1);
            if (pos < kSeg) seg[pos] = composite(logit_key(x, dummy), (uint32_t)(tb + slot_off[q]));
          }
        }
      }
      __syncwarp();  // rows read before the next batch writes
    }
  } else {
    const uint32_t tau = S.tau;
    int cnt = 0;
#pragma unroll
    for (int i = 0; i < kPT; ++i) cnt += logit_key(v[i], dummy) >= tau ? 1 : 0;
    int incl = cnt;
    for (int o = 1; o < 32; o <<= 1) {
      const int t = __shfl_up_sync(0xffffffffu, incl, o);
      if (lane >= o) incl += t;
    }
    int pos = incl - cnt;
#pragma unroll
    for (int i = 0; i < kPT; ++i) {
      const uint32_t k = logit_key(v[i], dummy);
      if (k >= tau) {
        if (pos < kSeg) seg[pos] = composite(k, index_of(i));
        ++pos;
      }
    }
    if (lane == 31) S.wcount[warp] = incl;
  }
  const int any_nonfinite = bar.sync_or(nonfinite);
  // every warp: the total, its own offset (candidates of lower warps) and
  // whether a segment overflowed, by warp reductions over the warp counts
  const int cl = lane < G::kGW ? S.wcount[lane] : 0;
  const int nc = (int)__reduce_add_sync(0xffffffffu, (unsigned)cl);
  const int before = (int)__reduce_add_sync(0xffffffffu, lane < warp ? (unsigned)cl : 0u);
  const int overflow = (int)__reduce_or_sync(0xffffffffu, cl > kSeg ? 1u : 0u);

  if (nc <= kFewCandidates) {
    // ---- usual case: the candidates packed in S.few, then warp 0 places
    // each by counting the larger ones (keys are distinct)
    const int wc = nc == 0 ? 0 : S.wcount[warp];
    for (int i = lane; i < wc; i += 32) S.few[before + i] = seg[i];
    if (tid < 2) S.few[nc + tid] = 0ull;  // pad: read 16 bytes at a time
    bar.sync();
    if (warp == 0) {
      // keys past nc (stale) are masked; the reads are unrolled so that they
      // are all in flight at once
      auto place = [&](auto n_max) {
        constexpr int kMax = decltype(n_max)::value;
        u64 mine[kMax / 32];
        int rank[kMax / 32];
#pragma unroll
        for (int h = 0; h < kMax / 32; ++h) {
          mine[h] = lane + 32 * h < nc ? S.few[lane + 32 * h] : 0ull;
          rank[h] = 0;
        }
#pragma unroll
        for (int j = 0; j < kMax; j += 2) {
          const ulonglong2 o = *reinterpret_cast<const ulonglong2 *>(&S.few[j]);
          const u64 ox = j < nc ? o.x : 0ull, oy = j + 1 < nc ? o.y : 0ull;
#pragma unroll
          for (int h = 0; h < kMax / 32; ++h) rank[h] += (ox > mine[h] ? 1 : 0) + (oy > mine[h] ? 1 : 0);
        }
#pragma unroll
        for (int h = 0; h < kMax / 32; ++h)
          if (lane + 32 * h < nc && rank[h] < ksel) dst[rank[h]] = mine[h];
      };
      if (nc <= 32) place(std::integral_constant<int, 32>());
      else place(std::integral_constant<int, kFewCandidates>());
      for (int i = lane; i < ksel; i += 32)
        if (i >= nc) dst[i] = 0;  // empty slots
    }
    return any_nonfinite;
  }
  // ---- exact top-ksel of the chunk -----------------------------------------
  u64 thr;
  if (!overflow) {
    const int wc = S.wcount[warp];
    thr = block_select_threshold<G>(S, ksel, tid, bar, [&](auto f) {
      for (int i = lane; i < wc; i += 32) f(seg[i]);
    });
    if (tid == 0) S.ntop = 0;
    bar.sync();
    for (int i = lane; i < wc; i += 32) {
      const u64 c = seg[i];
      if (c >= thr) S.top[atomicAdd(&S.ntop, 1)] = c;
    }
  } else {  // many ties / a flat row: select over the whole chunk
    // (rare) the logits are read again from L2, so that the values need not
    // stay in registers through the selection
    auto key_again = [&](int i) -> uint32_t {
      const int e = (int)index_of(i);
      return e < V ? logit_key(__ldcg(row + e), dummy) : 0u;
    };
    thr = block_select_threshold<G>(S, ksel, tid, bar, [&](auto f) {
#pragma unroll 4
      for (int i = 0; i < kPT; ++i) {
        const uint32_t k = key_again(i);
        if (k) f(composite(k, index_of(i)));
      }
    });
    if (tid == 0) S.ntop = 0;
    bar.sync();
#pragma unroll 4
    for (int i = 0; i < kPT; ++i) {
      const uint32_t k = key_again(i);
      if (k) {
        const u64 c = composite(k, index_of(i));
        if (c >= thr) S.top[atomicAdd(&S.ntop, 1)] = c;
      }
    }
  }
  bar.sync();
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
  // S.top and S.ntop are read until here: the next call's first use of them
  // follows its own barriers
  return any_nonfinite;
}

// ---- finish: merge each row's chunk lists, then the acceptance -------------
// Shared-memory layout of the finish (bytes from the start of its region).
struct FinishLayout {
  size_t merged, mcount, dist_p, dist_id, dist_n, in, pos, cbuf, stage, total;
};
__host__ __device__ inline FinishLayout finish_layout(int rows_per_wave, size_t per_row_bytes) {
  FinishLayout L;
  L.merged = 0;                                            // u64 [kMaxRows][kMaxTopK]
  L.mcount = L.merged + (size_t)kMaxRows * kMaxTopK * 8;   // int [kMaxRows + 1]
  L.dist_p = L.mcount + (kMaxRows + 1) * 4;                // float [kMaxRows][64]
  L.dist_id = L.dist_p + (size_t)kMaxRows * 64 * 4;        // int [kMaxRows][64]
  L.dist_n = L.dist_id + (size_t)kMaxRows * 64 * 4;        // int [kMaxRows + 1]
  L.in = L.dist_n + (kMaxRows + 1) * 4;                    // int [kAccInWords]
  L.pos = L.in + kAccInWords * 4;                          // int [3][kMaxK + 1]
  L.cbuf = (L.pos + 3 * (kMaxK + 1) * 4 + 15) / 16 * 16;   // u64 [rows_per_wave][kMergeBuf]
  L.stage = L.cbuf + (size_t)rows_per_wave * kMergeBuf * 8;  // u64 [rows_per_wave][C*ksel]
  const size_t scratch = (size_t)(kMaxK + 1) * 64 * 8;     // per position: 64 floats + 64 ints
  L.total = L.stage + (rows_per_wave * per_row_bytes > scratch ? rows_per_wave * per_row_bytes
                                                               : scratch);
  return L;
}

// The last steps of sequence b, by one CTA: every row's lists merged into
// its top-ksel (a warp per row, rows in waves) and, when sampling, its
// filtered distribution; then every position's test and the token it would
// emit, in parallel (a warp per position), and the walk to the first
// rejection.  smem: finish_layout(a.rows_per_wave, C * ksel * 8) bytes.
__device__ void finish_sequence(const AcceptArgs &a, int b, uint8_t *smem) {
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int K = a.K, V = a.V, ksel = a.ksel, C = a.C;
  const bool greedy = a.temperature == 0.f;
  const int per_row = C * ksel;
  const FinishLayout FL = finish_layout(a.rows_per_wave, (size_t)per_row * 8);
  u64 *merged = reinterpret_cast<u64 *>(smem + FL.merged);
  int *mcount = reinterpret_cast<int *>(smem + FL.mcount);
  // each row's filtered distribution, built by the warp that merged it:
  // entry j at [row][j] (j = lane + 32 h of RowDist), and its support size
  float *dist_p = reinterpret_cast<float *>(smem + FL.dist_p);
  int *dist_id = reinterpret_cast<int *>(smem + FL.dist_id);
  int *dist_n = reinterpret_cast<int *>(smem + FL.dist_n);
  // the acceptance's inputs: draft tokens [kMaxK], uniforms [kMaxK], row
  // flags [kMaxRows], the sampling uniform
  int *in_d = reinterpret_cast<int *>(smem + FL.in);
  float *in_ua = reinterpret_cast<float *>(in_d + kMaxK);
  int *in_f = reinterpret_cast<int *>(in_ua + kMaxK);
  float *in_us = reinterpret_cast<float *>(in_f + kMaxRows);
  // per position k (K: the bonus row): accepted, the token emitted if the
  // walk stops there, the flags the walk picks up there
  int *pos_acc = reinterpret_cast<int *>(smem + FL.pos);
  int *pos_emit = pos_acc + (kMaxK + 1);
  int *pos_flags = pos_emit + (kMaxK + 1);
  u64 *cbuf = reinterpret_cast<u64 *>(smem + FL.cbuf);
  u64 *stage = reinterpret_cast<u64 *>(smem + FL.stage);

  if (warp == kWarps - 1) {  // loaded while the rows merge (the last warp
                             // merges a row only when 16 rows do)
    if (lane < K) {
      in_d[lane] = a.dt[(size_t)b * K + lane];
      in_ua[lane] = a.ua[(size_t)b * K + lane];
    }
    for (int r = lane; r < a.rows; r += 32) in_f[r] = __ldcg(&a.rowflags[b * a.rows_max + r]);
    if (lane == 0) in_us[0] = a.us[b];
  }

  // subset of every list merged first: its first q entries
  const int q = min(ksel, (3 * ksel + C - 1) / C);
  const int ns = C * q;  // <= 3 ksel + C - 1 < kMergeBuf
  const unsigned below = (1u << lane) - 1u;
  // list and entry of staged key i without an integer division: i < 4096
  // and ksel <= 64 keep (i + 1/2) / ksel at least 1/128 from an integer,
  // far beyond the float product's error
  const float inv_ksel = 1.f / (float)ksel;
  auto list_of = [&](int i) { return (int)(((float)i + 0.5f) * inv_ksel); };
  for (int r0 = 0; r0 < a.rows; r0 += a.rows_per_wave) {
    const int r = r0 + warp;
    const bool active = warp < a.rows_per_wave && r < a.rows;
    if (active) {
      u64 *st = stage + (size_t)warp * per_row;
      u64 *cb = cbuf + (size_t)warp * kMergeBuf;
      u64 *mr = merged + r * kMaxTopK;
      const u64 *src = a.cand + ((size_t)b * a.rows_max + r) * (size_t)C * kMaxTopK;
      // the row's lists, kStageBatch loads per lane in flight before their
      // shared-memory stores (a load issued after a store to a possibly
      // aliasing address would wait for it: one round trip per element);
      // the first q entries of each list also go to cb, contiguously
      for (int i0 = 0; i0 < per_row; i0 += 32 * kStageBatch) {
        u64 v[kStageBatch];
        int lj[kStageBatch];
#pragma unroll
        for (int u = 0; u < kStageBatch; ++u) {
          const int i = i0 + 32 * u + lane;
          const int l = list_of(i);
          lj[u] = l;
          v[u] = i < per_row ? __ldcg(src + l * kMaxTopK + (i - l * ksel)) : 0ull;
        }
#pragma unroll
        for (int u = 0; u < kStageBatch; ++u) {
          const int i = i0 + 32 * u + lane;
          if (i < per_row) {
            st[i] = v[u];
            const int l = lj[u], j = i - l * ksel;
            if (j < q) cb[l * q + j] = v[u];
          }
        }
      }
      if (lane == 0) cb[ns] = 0ull;  // pad: pairs are read 16 bytes at a time
      __syncwarp();
      // The subset's ksel-th largest key T bounds the row's from below.  The
      // subset's keys are ranked by counting larger ones (keys are distinct:
      // one token, one chunk; empty slots, 0, never count), and the top ksel
      // of them are the row's when no list has a key >= T past its first q
      // entries (the usual case: the top ksel rarely take more than q from
      // one list).
      u64 T = 0ull;
      int nnz = 0;  // nonzero keys of the subset
      {
        // every lane's keys of the subset (e = lane + 32 h, h < kH) compared
        // in one pass over it, eight pairs in flight at a time
        auto rank_subset = [&](auto kh_c) {
          constexpr int kH = decltype(kh_c)::value;
          u64 xs[kH];
          int larger[kH];
#pragma unroll
          for (int h = 0; h < kH; ++h) {
            const int e = lane + 32 * h;
            xs[h] = e < ns ? cb[e] : 0ull;
            larger[h] = 0;
            nnz += __popc(__ballot_sync(0xffffffffu, xs[h] != 0ull));
          }
#pragma unroll 8
          for (int f = 0; f < ns; f += 2) {
            const ulonglong2 y = *reinterpret_cast<const ulonglong2 *>(cb + f);
#pragma unroll
            for (int h = 0; h < kH; ++h) larger[h] += (y.x > xs[h] ? 1 : 0) + (y.y > xs[h] ? 1 : 0);
          }
#pragma unroll
          for (int h = 0; h < kH; ++h) {
            if (xs[h] != 0ull && larger[h] < ksel) mr[larger[h]] = xs[h];
            if (xs[h] != 0ull && larger[h] == ksel - 1) T = xs[h];
          }
        };
        switch ((ns + 31) / 32) {  // ns < kMergeBuf = 256
          case 1: rank_subset(std::integral_constant<int, 1>()); break;
          case 2: rank_subset(std::integral_constant<int, 2>()); break;
          case 3: rank_subset(std::integral_constant<int, 3>()); break;
          case 4: rank_subset(std::integral_constant<int, 4>()); break;
          default: rank_subset(std::integral_constant<int, kMergeBuf / 32>()); break;
        }
      }
      T = warp_max_u64(T);  // one lane holds it; 0 if nnz < ksel
      // a key >= T (any nonzero key when T = 0) past the first q entries?
      bool missed = false;
      if (q < ksel)
        for (int l = lane; l < C; l += 32) {
          const u64 x = st[l * ksel + q];
          missed |= x != 0ull && x >= T;
        }
      int j;
      if (!__any_sync(0xffffffffu, missed)) {
        j = min(nnz, ksel);
      } else {
        // (rare) every key >= T competes, typically a few more than ksel
        __syncwarp();
        int nc = 0;
        for (int i0 = 0; i0 < per_row; i0 += 32) {
          const int i = i0 + lane;
          const u64 x = i < per_row ? st[i] : 0ull;
          const bool keep = x != 0ull && x >= T;
          const unsigned m = __ballot_sync(0xffffffffu, keep);
          const int pos = nc + __popc(m & below);
          if (keep && pos < kMergeBuf - 1) cb[pos] = x;
          nc += __popc(m);
        }
        if (nc < kMergeBuf) {
          if (lane == 0) cb[nc] = 0ull;
          __syncwarp();
          for (int e = lane; e < nc; e += 32) {
            const u64 x = cb[e];
            int larger = 0;
#pragma unroll 4
            for (int f = 0; f < nc; f += 2) {
              const ulonglong2 y = *reinterpret_cast<const ulonglong2 *>(cb + f);
              larger += (y.x > x ? 1 : 0) + (y.y > x ? 1 : 0);
            }
            if (larger < ksel) mr[larger] = x;
          }
          j = min(nc, ksel);
        } else {  // (rarer) k-way merge of the lists
          int h0 = 0, h1 = 0;  // heads of lists lane and lane+32
          for (j = 0; j < ksel; ++j) {
            const u64 v0 = (lane < C && h0 < ksel) ? st[lane * ksel + h0] : 0ull;
            const u64 v1 = (lane + 32 < C && h1 < ksel) ? st[(lane + 32) * ksel + h1] : 0ull;
            const u64 best = v0 > v1 ? v0 : v1;
            const u64 g = warp_max_u64(best);
            if (g == 0ull) break;
            if (v0 == g) ++h0;
            else if (v1 == g) ++h1;
            if (lane == 0) mr[j] = g;
          }
        }
      }
      if (lane == 0) mcount[r] = j;
      if (!greedy) {  // the distribution, while the other rows merge
        __syncwarp();
        const RowDist D = row_dist(mr, j, a.temperature, a.top_p);
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

  // ---- every position at once: warp k < K tests draft token k and, if it
  // is rejected, samples the residual (p - q)+ there; warp K the bonus row
  if (warp <= K) {
    const int k = warp;
    int f = in_f[k], acc = 0, emit = -1;
    if (k == K) {
      if (greedy) {
        emit = mcount[K] > 0 ? composite_id(merged[K * kMaxTopK]) : -1;
      } else {
        const RowDist P = stored_dist(dist_p, dist_id, dist_n, K);
        float *sR = reinterpret_cast<float *>(stage) + k * 128;  // 64 floats + 64 ints
        int *sId = reinterpret_cast<int *>(sR + 64);
        float R[2] = {P.p[0], P.p[1]};
        emit = inverse_cdf_by_id(P.id, R, mcount[K], in_us[0], sR, sId, dist_id + K * 64);
      }
    } else {
      const int d = in_d[k];
      const bool d_ok = d >= 0 && d < V;
      if (!d_ok) f |= SV_FLAG_DRAFT_OUT_OF_RANGE;
      if (greedy) {
        const int am = mcount[k] > 0 ? composite_id(merged[k * kMaxTopK]) : -1;
        acc = d_ok && am >= 0 && d == am;
        emit = am;
      } else {
        f |= in_f[K + 1 + k];
        const RowDist P = stored_dist(dist_p, dist_id, dist_n, k);
        const int qrow = K + 1 + k;
        const RowDist Q = stored_dist(dist_p, dist_id, dist_n, qrow);
        if (d_ok) {
          const float qd = dist_lookup(Q, d);
          if (qd == 0.f) {
            f |= SV_FLAG_DRAFT_ZERO_Q;
          } else {
            const float pd = dist_lookup(P, d);
            acc = in_ua[k] < pd / qd;
          }
        }
        if (!acc) {
          // residual max(0, p - q) over p's support (q's entries read from
          // the stored distribution, all lanes the same address: broadcast)
          float R[2] = {P.p[0], P.p[1]};
          const int nq = Q.n;  // entries past it have no mass
#pragma unroll 4
          for (int src = 0; src < nq; ++src) {
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
          float *sR = reinterpret_cast<float *>(stage) + k * 128;
          int *sId = reinterpret_cast<int *>(sR + 64);
          emit = inverse_cdf_by_id(P.id, R, mcount[k], in_us[0], sR, sId, dist_id + k * 64);
        }
      }
    }
    if (lane == 0) {
      pos_acc[k] = acc;
      pos_emit[k] = emit;
      pos_flags[k] = f;
    }
  }
  __syncthreads();
  if (warp != 0) return;

  // ---- the walk: accepted up to the first rejection (or all K, then the
  // bonus), flags of every position it visits
  const unsigned rej = __ballot_sync(0xffffffffu, lane < K && pos_acc[lane] == 0);
  const int stop = rej ? __ffs(rej) - 1 : K;
  int flags = (int)__reduce_or_sync(0xffffffffu, lane <= stop ? (unsigned)pos_flags[lane] : 0u);
  const int emitted = pos_emit[stop];
  if (emitted < 0) flags |= SV_FLAG_EMPTY_DIST;
  int32_t *out = a.out + (size_t)b * (K + 1);
  if (lane <= K) out[lane] = lane < stop ? in_d[lane] : (lane == stop ? emitted : -1);
  if (lane == 0) {
    a.nacc[b] = stop;
    if (a.flags) a.flags[b] = flags;
    a.counters[b] = 0;  // ready for the next call
  }
  for (int r = lane; r < a.rows_max; r += 32) a.rowflags[b * a.rows_max + r] = 0;
}

// Sequence and row of a logits chunk; the row's logits.
__device__ __forceinline__ const float *chunk_row(const AcceptArgs &a, int row_g, int &b,
                                                  int &rloc) {
  b = row_g / a.rows;
  rloc = row_g - b * a.rows;
  const int K = a.K;
  return rloc <= K ? a.tl + ((size_t)b * (K + 1) + rloc) * a.V
                   : a.dl + ((size_t)b * K + (rloc - K - 1)) * a.V;
}
__device__ __forceinline__ u64 *chunk_dst(const AcceptArgs &a, int b, int rloc, int cx) {
  return a.cand + ((size_t)b * a.rows_max + rloc) * (size_t)a.C * kMaxTopK + (size_t)cx * kMaxTopK;
}

// kCtasPerSm: co-resident CTAs the register budget is cut for.  Three (40
// registers) hide more load latency when many sequences fill the GPU with
// chunk CTAs; two keep the finish path, which one CTA per sequence runs,
// free of spills.
//
// One CTA per (chunk, row) of every sequence; the last CTA of a sequence to
// finish (CTA barrier, then one acq_rel atomic add by thread 0; no spinning)
// runs the finish.  Serves the rows given as lists of a fused LM head, and
// logits rows without 16-byte alignment; aligned logits take the streaming
// pair below.
template <int kCtasPerSm>
__global__ void __launch_bounds__(kThreads, kCtasPerSm) spec_accept_kernel(const AcceptArgs a) {
  extern __shared__ __align__(16) uint8_t smem_raw[];
  ChunkSmem &S = *reinterpret_cast<ChunkSmem *>(smem_raw);
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  int b, rloc;
  const float *row = chunk_row(a, blockIdx.y, b, rloc);
  const int cx = blockIdx.x;
  const int K = a.K, V = a.V;
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
      u64 *dst = chunk_dst(a, b, rloc, cx);
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
    // ---- load the chunk (values past V read as -inf: key 0, never kept) ----
    float v[kPerThread];
    if (a.vec) {
#pragma unroll
      for (int i = 0; i < kPerThread / 4; ++i) {
        const int e = base + 4 * (tid + kThreads * i);
        float4 f = make_float4(-INFINITY, -INFINITY, -INFINITY, -INFINITY);
        if (e < V) f = __ldcs(reinterpret_cast<const float4 *>(row + e));  // V % 4 == 0 here
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
        if (e < V) v[i] = __ldcs(row + e);
      }
    }
    const int nf = chunk_select<CtaGeo>(S, v, row, V, base, a.vec != 0, ksel,
                                        chunk_dst(a, b, rloc, cx), tid, CtaBarrier{}, 0,
                                        [](int) {});
    if (tid == 0 && nf) atomicOr(&a.rowflags[b * a.rows_max + rloc], SV_FLAG_NONFINITE_LOGIT);
  }

  // ---- the last CTA of this sequence finishes it ---------------------------
  // every thread's candidate stores precede thread 0's release (CTA barrier,
  // then a cumulative acq_rel add); the last CTA acquires the others' lists
  __syncthreads();
  int last = 0;
  if (tid == 0) {
    int old;
    asm volatile("atom.acq_rel.gpu.global.add.s32 %0, [%1], 1;"
                 : "=r"(old)
                 : "l"(&a.counters[b])
                 : "memory");
    last = old == a.rows * a.C - 1;
  }
  // the decision travels in the barrier's vote, not in shared memory, which
  // the finish reuses from here on
  if (!__syncthreads_or(last)) return;
  finish_sequence(a, b, smem_raw);
}

// ---- streaming pair: every chunk of 16-byte-aligned logits rows, then one
// finish CTA per sequence ------------------------------------------------------
// A persistent CTA per SM runs two groups of kGT threads that select
// alternate chunks of the CTA's sequence (k even, k odd), so that one group's
// barriers and shuffles overlap the other's.  The work order lists every
// row's whole chunks first (sequence-major) and the rows' shorter last chunks
// after them; the 2G group slots (G = gridDim.x, slot p = CTA + G * group)
// take it in rounds of 2G positions, slot p taking position p of even rounds
// and 2G - 1 - p of odd ones, so that the slots that take a position more
// take the shorter chunks.  A slot's positions grow from round to round, and
// chunk k + kStreamStages of a CTA lies rounds after chunk k.  The chunks reach shared memory
// through a ring of kStreamStages slots: chunk k takes slot k % kStreamStages
// as one bulk copy of up to 64 KB that completes on the slot's mbarrier.  A
// group moves a landed chunk to registers, and one of its threads refills the
// slot with chunk k + kStreamStages right after the group's first barrier of
// the selection.  Waits are bounded: a wait that runs out marks the device
// error word, stops the refills, and the CTA runs out its chunks on -inf
// (garbage lists, flagged) and, before returning, waits (bounded again) for
// the copies still in flight.
__device__ unsigned int g_accept_device_error;

constexpr int kStreamGroups = 2;
struct StreamCtl {
  uint64_t full[kStreamStages];      // slot mbarriers
  int4 item[kStreamStages];          // the slot's chunk: position, b, rloc, cx
  unsigned issued[kStreamStages];    // copies started per slot
  unsigned consumed[kStreamStages];  // copies waited for per slot
  int failed;                        // a wait ran out
};
constexpr size_t kStreamSmemBytes =
    kStreamRingBytes + kStreamGroups * sizeof(StreamSmem) + sizeof(StreamCtl);
static_assert(kStreamSmemBytes <= 227 * 1024, "the streaming CTA fits one SM's shared memory");

constexpr int kStreamThreads = kStreamGroups * GroupGeo::kGT;

__global__ void __launch_bounds__(kStreamThreads, 1) accept_stream_kernel(const AcceptArgs a) {
  extern __shared__ __align__(16) uint8_t smem_raw[];
  float *ring = reinterpret_cast<float *>(smem_raw);
  constexpr int kGT = GroupGeo::kGT, kPT = GroupGeo::kPT;
  const int group = threadIdx.x / kGT, tid = threadIdx.x % kGT, warp = tid >> 5;
  StreamSmem &S = reinterpret_cast<StreamSmem *>(smem_raw + kStreamRingBytes)[group];
  StreamCtl &ctl = *reinterpret_cast<StreamCtl *>(smem_raw + kStreamRingBytes +
                                                  kStreamGroups * sizeof(StreamSmem));
  const GroupBarrier<kGT> bar{1 + group};
  const int C = a.C, V = a.V, K = a.K;
  const int n_items = a.B * a.rows * C;
  const int n_full = a.B * a.rows * (C - 1);  // whole chunks (all of them when V % kChunk == 0)
  const int G = gridDim.x;

  // position of the CTA's k-th chunk in the work order
  auto position = [&](int k) {
    const int i = k >> 1, p = blockIdx.x + G * (k & 1);
    return 2 * G * i + ((i & 1) ? 2 * G - 1 - p : p);
  };
  // the chunk at a position: sequence, row, chunk of the row
  auto decode = [&](int pos) {
    int row_g, cx;
    if (pos < n_full) {
      row_g = pos / (C - 1);
      cx = pos - row_g * (C - 1);
    } else {
      row_g = pos - n_full;
      cx = C - 1;
    }
    const int b = row_g / a.rows;
    return make_int4(pos, b, row_g - b * a.rows, cx);
  };
  auto row_of = [&](int b, int rloc) {
    return rloc <= K ? a.tl + ((size_t)b * (K + 1) + rloc) * V
                     : a.dl + ((size_t)b * K + (rloc - K - 1)) * V;
  };

  // (an issuing thread) start the copy of the CTA's k-th chunk into its slot
  auto issue = [&](int k) {
    const int s = k % kStreamStages;
    const int4 it = decode(position(k));
    const int base = it.w * kChunk;
    const uint32_t bytes = (uint32_t)min(kChunk, V - base) * 4u;  // V % 4 == 0: a 16-multiple
    __threadfence_block();  // the slot's previous phase, seen complete, before the record
    ctl.item[s] = it;
    ctl.issued[s] += 1;
    mbar_arrive_expect_tx(&ctl.full[s], bytes);
    // the logits are read once: evict-first in L2, so that the chunk lists
    // written meanwhile stay there for the finish
    bulk_copy_g2s_hint(ring + (size_t)s * kChunk, row_of(it.y, it.z) + base, bytes, &ctl.full[s],
                       l2_policy_evict_first());
  };

  if (threadIdx.x == 0) {
    for (int s = 0; s < kStreamStages; ++s) {
      mbar_init(&ctl.full[s], 1);
      ctl.issued[s] = 0;
      ctl.consumed[s] = 0;
    }
    ctl.failed = 0;
    fence_mbar_init();
    for (int k = 0; k < kStreamStages; ++k)
      if (position(k) < n_items) issue(k);
  }
  __syncthreads();
  pdl_launch_dependents();  // the finish kernel may take SMs as this grid leaves them

  constexpr int kIssuer = 32;  // a thread of the group's warp 1: warp 0 finds the bound meanwhile
  for (int k = group;; k += kStreamGroups) {
    if (position(k) >= n_items) break;  // (the group's positions only grow)
    const int s = k % kStreamStages;
    // warp 0 of the group waits for the slot, and a group barrier passes the
    // landed bytes (and the slot's chunk) on to the rest.  The slot's
    // previous chunk belongs to the other group and its copy may still be
    // landing (copies complete in any order); a parity wait for this chunk's
    // phase would then match the phase before it.  So the wait starts once
    // the slot's record names this chunk (the issuer writes it before
    // starting the copy, after the previous chunk was read): the slot is
    // then in this chunk's phase.
    bool ok = true;
    if (warp == 0 && !*(volatile int *)&ctl.failed) {
      const int want = position(k);
      const volatile int *rec = &ctl.item[s].x;
      if (*rec != want) {
        const unsigned long long t0 = global_timer_ns();
        while (*rec != want)
          if (global_timer_ns() - t0 > kWaitLimitNs) {
            ok = false;
            break;
          }
      }
      __threadfence_block();  // the record before the slot's barrier state
      if (ok) ok = mbar_wait(&ctl.full[s], (uint32_t)(k / kStreamStages) & 1u);
      if (ok && tid == 0) ctl.consumed[s] += 1;
    }
    const int timeout = bar.sync_or(!ok);
    const bool dead = timeout || *(volatile int *)&ctl.failed;
    // after a wait ran out the slot's record may never have been written:
    // the chunk is decoded again (its lists are written, flagged garbage)
    const int4 it = dead ? decode(position(k)) : ctl.item[s];
    const int b = it.y, rloc = it.z, cx = it.w;
    const float *row = row_of(b, rloc);
    const int base = cx * kChunk;
    float v[kPT];
    const float *slot = ring + (size_t)s * kChunk;
    if (!dead && base + kChunk <= V) {  // a whole chunk (all but a row's last)
#pragma unroll
      for (int i = 0; i < kPT / 4; ++i) {
        const float4 f = *reinterpret_cast<const float4 *>(slot + 4 * (tid + kGT * i));
        v[4 * i + 0] = f.x;
        v[4 * i + 1] = f.y;
        v[4 * i + 2] = f.z;
        v[4 * i + 3] = f.w;
      }
    } else {
#pragma unroll
      for (int i = 0; i < kPT / 4; ++i) {
        const int el = 4 * (tid + kGT * i);
        float4 f = make_float4(-INFINITY, -INFINITY, -INFINITY, -INFINITY);
        if (!dead && base + el < V) f = *reinterpret_cast<const float4 *>(slot + el);
        v[4 * i + 0] = f.x;
        v[4 * i + 1] = f.y;
        v[4 * i + 2] = f.z;
        v[4 * i + 3] = f.w;
      }
    }
    const int nf = chunk_select<GroupGeo>(
        S, v, row, V, base, true, a.ksel, chunk_dst(a, b, rloc, cx), tid, bar, timeout,
        [&](int vote) {
          // every thread of the group has read slot s: refill it
          if (vote & 2) {
            if (tid == 0) {
              atomicOr(&g_accept_device_error, 1u);
              *(volatile int *)&ctl.failed = 1;
            }
          } else if (tid == kIssuer && !*(volatile int *)&ctl.failed) {
            if (position(k + kStreamStages) < n_items) {
              asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
              issue(k + kStreamStages);
            }
          }
        });
    if (tid == 0 && nf) atomicOr(&a.rowflags[b * a.rows_max + rloc], SV_FLAG_NONFINITE_LOGIT);
  }
  // copies still in flight (only after a wait ran out) land before the CTA
  // gives up its shared memory, or the bounded wait gives up again
  __syncthreads();
  if (threadIdx.x == 0) {
    for (int s = 0; s < kStreamStages; ++s)
      for (unsigned c = ctl.consumed[s]; c < ctl.issued[s]; ++c)
        if (!mbar_wait(&ctl.full[s], c & 1u)) break;
  }
}

// One CTA per sequence, after the stream kernel.
__global__ void __launch_bounds__(kThreads, 1) accept_finish_kernel(const AcceptArgs a) {
  extern __shared__ __align__(16) uint8_t smem_raw[];
  pdl_wait();  // the lists and row flags are the stream kernel's output
  finish_sequence(a, blockIdx.x, smem_raw);
}

}  // namespace

unsigned take_device_error_accept() {
  unsigned v = 0, zero = 0;
  cudaMemcpyFromSymbol(&v, g_accept_device_error, sizeof v);
  cudaMemcpyToSymbol(g_accept_device_error, &zero, sizeof zero);
  return v;
}

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
  static_assert(kListsPerChunk * kMaxTopK <= ChunkSmem::kSeg * CtaGeo::kGW,
                "a chunk's lists fit the candidate buffer");
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
  const size_t final_bytes = finish_layout(args.rows_per_wave, per_row).total;
  const size_t smem = std::max(sizeof(ChunkSmem), final_bytes);
  const size_t stream_smem = kStreamSmemBytes;
  static PerDeviceOnce attrs_once;
  const cudaError_t ce = attrs_once.run([stream_smem] {
    cudaError_t e = cudaFuncSetAttribute(spec_accept_kernel<2>,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize, 160 * 1024);
    if (e == cudaSuccess)
      e = cudaFuncSetAttribute(spec_accept_kernel<3>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                               160 * 1024);
    if (e == cudaSuccess)
      e = cudaFuncSetAttribute(accept_stream_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                               (int)stream_smem);
    if (e == cudaSuccess)
      e = cudaFuncSetAttribute(accept_finish_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
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
  cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
  if (!target_lists && args.vec) {
    // aligned logits: the streaming kernel (a CTA per SM), then a finish CTA
    // per sequence
    const long long items = (long long)B * args.rows * args.C;
    const int grid = (int)std::min<long long>(items, device_sm_count());
    accept_stream_kernel<<<grid, kStreamThreads, stream_smem, st>>>(args);
    const sv_status ls = check_launch("spec_accept (chunks)");
    if (ls != SV_OK) return ls;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)B);
    cfg.blockDim = dim3(kThreads);
    cfg.dynamicSmemBytes = final_bytes;
    cfg.stream = st;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = pdl_enabled() ? 1 : 0;
    if (cudaLaunchKernelEx(&cfg, accept_finish_kernel, args) != cudaSuccess)
      return fail(SV_ERR_CUDA, "spec_accept (finish): launch failed: %s",
                  cudaGetErrorString(cudaGetLastError()));
    return check_launch("spec_accept (finish)");
  }
  dim3 grid((unsigned)args.C, (unsigned)(B * args.rows));
  if (B >= kManySequences)
    spec_accept_kernel<3><<<grid, kThreads, smem, st>>>(args);
  else
    spec_accept_kernel<2><<<grid, kThreads, smem, st>>>(args);
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
