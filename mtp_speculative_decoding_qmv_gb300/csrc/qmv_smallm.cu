// qmv_smallm.cu -- small-M (1..16 rows) 4-bit affine group-64 quantised mat-vec
// for the target model's verify forward, sm_103a.
//
// Source: "MTPLX 2.24x faster TPS", section "Layer 0: MLX Runtime" (the verify
// forward runs M = K+1 = 3..6 rows, one per drafted position, through the
// 4-bit projections; stock large-M kernels stall on that shape) and the
// "what I had to solve" list of the ai-navigate-news copy, item 3 (MLP
// projections were 51 % of verify time).
//
//   y[m, n] = sum_i x[m, i] * (s[n, i/64] * q[n, i] + b[n, i/64])
//
// The op streams 0.5625 bytes of weight per weight (4-bit nibble + bf16
// scale and bias per 64) and is HBM-bound.  Design:
//  * a CTA owns a tile of 64 output rows and a contiguous run of the K axis
//    in 512-input stages; when there are too few row tiles to fill the GPU,
//    the stages of a tile are split over a thread-block cluster of S CTAs
//    whose partial results meet in the first CTA's shared memory (DSMEM) and
//    are summed there in rank order -- deterministic run to run;
//  * a producer warp streams the CTA's stages through a ring of shared-memory
//    buffers as 2-D tensor-map boxes (cp.async.bulk.tensor, L2 evict-first,
//    completing on the stage's mbarrier): packed weights as 64 rows x 128
//    bytes per 256 inputs (128-byte swizzle), the stage's 8 scales and 8
//    biases per row as 64 x 16 bytes.  Bytes in flight decide the bandwidth
//    (HBM latency under load is microseconds), so the ring holds only those
//    streamed bytes and is sized to fill shared memory at the achieved
//    occupancy; large boxes keep the copy engine far from its per-request
//    limit;
//  * eight consumer warps take one 64-group of each stage (split-K over
//    warps) for all four 16-row MMA tiles, so the per-stage costs of a warp
//    (barrier, activation fragments, sum of x) are spread over 4096 weights;
//    the activation fragments are read from L2 with plain loads issued one
//    stage ahead; warps reduce through shared memory at the end in a fixed
//    order;
//  * each weight is read from shared memory once (ldmatrix on the swizzled
//    box: conflict-free) and used for all M rows: nibbles are widened to
//    bf16 (128 + q, exact) and fed to the tensor cores as the 16-row A
//    operand of mma.m16n8k16 with the (<= 8) activation rows as B.  When K
//    is a multiple of 128 the boxes are byte-expanded (the copy engine leaves
//    a gap after every 8 bytes and ldmatrix.b4x16_p64 widens each nibble to
//    a byte: one byte permute per two weights); otherwise packed boxes are
//    widened with shifts and masks.  The format depends only on K and the
//    weights' alignment, so every M of one matrix shares the arithmetic.
//    Per group D = -128 sum(x) + sum (128 + q) x, the offset being the first
//    MMA's accumulator, and acc += s * D + b * sum(x), with sum(x) taken from
//    an all-ones MMA.  Products are exact, the accumulation is fp32.  CUDA-core FMAs alone cannot keep up with the HBM
//    stream at M >= 2 on this part (4 FMAs + unpack per weight per row
//    against ~3.3 issue slots per streamed weight); the MMA path costs the
//    same at every M.
//  * when K is not a multiple of 512 the scale rows are not 16-byte aligned
//    for the copy engine; the tile's whole scale block is then loaded once
//    (and the K axis is not split);
//  * programmatic dependent launch: the weight stream starts before the
//    preceding kernel on the stream ends; activations are read, and y
//    written, only after griddepcontrol.wait.
#include <algorithm>
#include <atomic>

#include "qmv_common.cuh"

namespace sv {
namespace {
using namespace qmv;

constexpr int kMaxSplits = 8;                      // portable cluster size
// CTAs per SM the register budget is set for: 2 (113 registers a thread) for
// up to 8 activation rows; 1 for 9..16 rows, whose accumulators are twice as
// many
template <int kNT>
constexpr int kMinCtasPerSm = kNT == 1 ? 2 : 1;
__device__ unsigned int g_qmv_device_error;

struct QmvArgs {
  const uint16_t *s;  // [N][K/64] bf16
  const uint16_t *b;  // [N][K/64] bf16
  const void *x;      // [M][K] fp32 or bf16
  float *y;           // [M][N]
  int M, N, K;
  int stages;
  int splits;     // CTAs per row tile (cluster size along K)
  int sb_stream;  // 1: scales/biases stream with the stages; 0: whole tile block once
};

struct Layout {
  uint32_t stage, sb, bar, total;
};

__host__ __device__ inline uint32_t round_up_u32(uint32_t v, uint32_t a) {
  return (v + a - 1) / a * a;
}

// [stages] then, if not streamed, the tile's scale/bias block, then the
// mbarriers.  The end-of-kernel reductions reuse the drained ring (at least
// kRedBytes long per 8 activation rows).  `total` includes 1 KB of
// alignment slack.  p64: byte-expandable weight boxes (K % 128 == 0).
__host__ __device__ inline Layout qmv_layout(int groups, int stages, bool sb_stream, int nt,
                                             bool p64) {
  Layout L;
  L.stage = p64 ? (sb_stream ? kStageBytesP64 : kStageBytesP64Block)
                : (sb_stream ? kStageBytesStream : kStageBytesBlock);
  const uint32_t ring = (uint32_t)stages * L.stage;
  const uint32_t red = kRedBytes * (uint32_t)nt;
  L.sb = (ring > red ? ring : red);
  const uint32_t after = L.sb + (sb_stream ? 0u : round_up_u32(2u * kRows * groups * 2u, 16));
  L.bar = round_up_u32(after, 16);
  L.total = L.bar + (uint32_t)(2 * stages + 1) * 8u + 1024u;
  return L;
}

__device__ __forceinline__ uint32_t cluster_rank() {
  uint32_t r;
  asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
  return r;
}
__device__ __forceinline__ void cluster_sync_all() {
  asm volatile("barrier.cluster.arrive.release.aligned;\n\tbarrier.cluster.wait.acquire.aligned;"
               ::: "memory");
}
__device__ __forceinline__ uint32_t map_shared_to_rank(uint32_t addr, uint32_t rank) {
  uint32_t r;
  asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(r) : "r"(addr), "r"(rank));
  return r;
}
__device__ __forceinline__ void st_cluster_f32(uint32_t addr, float v) {
  asm volatile("st.shared::cluster.f32 [%0], %1;" ::"r"(addr), "f"(v) : "memory");
}

// Producer: expect chunk c's bytes on stage st's barrier and issue its boxes.
// Rows past N, inputs past K and groups past K/64 are zero-filled by the copy
// engine and still counted in the transaction bytes.
template <bool kStream, bool kP64>
__device__ __forceinline__ void issue_stage(const QmvArgs &a, const CUtensorMap *wmap,
                                            const CUtensorMap *smap, const CUtensorMap *bmap,
                                            uint32_t stage_addr, uint32_t bar, int c, int n0,
                                            uint64_t policy) {
  const int k0 = c * kStageInputs;
  const int kn = min(kStageInputs, a.K - k0);
  constexpr int kBoxInputs = kP64 ? kP64BoxInputs : kBoxWords * 8;
  const int boxes = (kn + kBoxInputs - 1) / kBoxInputs;
  // byte-expandable boxes take 8 KB of shared memory for 4 KB transferred
  constexpr uint32_t kBoxSmem = kP64 ? kP64BoxBytes : kRows * 128;
  constexpr uint32_t kBoxTx = kP64 ? kP64BoxTx : kRows * 128;
  const uint32_t bytes = (uint32_t)(boxes * kBoxTx + (kStream ? 2 * kRows * 16 : 0));
  mbar_arrive_expect_tx_u32(bar, bytes);
  for (int bx = 0; bx < boxes; ++bx)
    tma_load_2d(stage_addr + bx * kBoxSmem, wmap,
                kP64 ? k0 + bx * kP64BoxInputs : k0 / 8 + bx * kBoxWords, n0, bar, policy);
  if (kStream) {
    constexpr uint32_t kSb = kP64 ? kP64SbOff : kSbOff;
    tma_load_2d(stage_addr + kSb, smap, k0 / 64, n0, bar, policy);
    tma_load_2d(stage_addr + kSb + kRows * 16, bmap, k0 / 64, n0, bar, policy);
  }
}

// kStream: K % 512 == 0, scales and biases stream with the stages and every
// group of every stage is real; otherwise the tile's whole scale block is
// loaded once and groups past K/64 are skipped.
//
// kNT: 8-row MMA n-tiles of activation rows (1: M <= 8, 2: M <= 16).
// kP64: byte-expandable weight boxes (K % 128 == 0, weights 32-byte aligned);
// otherwise packed boxes widened with shifts and masks.
template <bool kXF32, bool kStream, int kNT, bool kP64>
__global__ void __launch_bounds__(kThreads, kMinCtasPerSm<kNT>)
    qmv_smallm_kernel(const __grid_constant__ CUtensorMap wmap,
                      const __grid_constant__ CUtensorMap smap,
                      const __grid_constant__ CUtensorMap bmap, const QmvArgs a) {
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  // the swizzled boxes need 1024-byte aligned destinations
  const uint32_t raw = smem_addr(smem_raw);
  const uint32_t base = raw + ((1024u - (raw & 1023u)) & 1023u);
  uint8_t *smem = smem_raw + (base - raw);
  const int groups = a.K >> 6;
  const int splits = a.splits;
  const int tile = blockIdx.x / splits;
  const int split = blockIdx.x - tile * splits;
  const int n0 = tile * kRows;
  const int rows = min(kRows, a.N - n0);
  const int n_chunks = (a.K + kStageInputs - 1) / kStageInputs;
  const int c_begin = (int)((long long)split * n_chunks / splits);
  const int c_end = (int)((long long)(split + 1) * n_chunks / splits);
  const int stages = a.stages;
  const Layout L = qmv_layout(groups, stages, kStream, kNT, kP64);
  constexpr int kCols = 8 * kNT;          // activation rows a CTA's sums cover
  constexpr int kParts = 2 * kNT;         // output elements per consumer thread
  const uint32_t full0 = base + L.bar;          // full[i]  = full0 + 8 i
  const uint32_t empty0 = full0 + 8u * stages;  // empty[i] = empty0 + 8 i
  const uint32_t sb_bar = empty0 + 8u * stages;

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  if (threadIdx.x == 0) {
    for (int i = 0; i < stages; ++i) {
      mbar_init_u32(full0 + 8u * i, 1);
      mbar_init_u32(empty0 + 8u * i, kConsumerWarps);
    }
    mbar_init_u32(sb_bar, 32);
    fence_mbar_init();
  }
  __syncthreads();
  pdl_launch_dependents();

  float part[kParts] = {};  // this thread's sums of the tile (consumers)
  bool ok = true;
  if (warp == kConsumerWarps) {
    // ------------------------------ producer ------------------------------
    // Weights, scales and biases do not depend on earlier kernels: no
    // griddepcontrol.wait on this side.
    uint16_t *s_sm = reinterpret_cast<uint16_t *>(smem + L.sb);
    uint16_t *b_sm = s_sm + kRows * groups;
    uint64_t *sb_bar_p = reinterpret_cast<uint64_t *>(smem + (sb_bar - base));
    const uint32_t sb_bytes = (uint32_t)rows * groups * 2;
    if (kStream) {
      mbar_arrive_u32(sb_bar);
    } else if (sb_bytes % 16u == 0) {
      if (lane == 0) {
        mbar_arrive_expect_tx_u32(sb_bar, 2 * sb_bytes);
        bulk_copy_g2s(s_sm, a.s + (size_t)n0 * groups, sb_bytes, sb_bar_p);
        bulk_copy_g2s(b_sm, a.b + (size_t)n0 * groups, sb_bytes, sb_bar_p);
      } else {
        mbar_arrive_u32(sb_bar);
      }
    } else {  // ragged tile whose scale block is not a 16-byte multiple
      for (int i = lane; i < rows * groups; i += 32) {
        s_sm[i] = a.s[(size_t)n0 * groups + i];
        b_sm[i] = a.b[(size_t)n0 * groups + i];
      }
      mbar_arrive_u32(sb_bar);
    }
    if (lane == 0) {
      const uint64_t policy = l2_policy_evict_first();
      int st = 0, ph = 0;  // stage of chunk c and the parity of its previous release
      for (int c = c_begin; c < c_end; ++c) {
        if (c - c_begin >= stages && !mbar_wait_u32(empty0 + 8u * st, ph ^ 1)) {
          atomicOr(&g_qmv_device_error, 1u);
          // let the copies already issued land before the CTA may exit
          for (int i = max(c_begin, c - stages); i < c; ++i)
            (void)mbar_wait_u32(full0 + 8u * ((i - c_begin) % stages),
                                ((i - c_begin) / stages) & 1);
          break;
        }
        issue_stage<kStream, kP64>(a, &wmap, &smap, &bmap, base + st * L.stage, full0 + 8u * st,
                                   c, n0, policy);
        if (++st == stages) {
          st = 0;
          ph ^= 1;
        }
      }
    }
    __syncwarp();
    if (splits == 1) return;
  } else {
    // ------------------------------ consumers -----------------------------
    const int g8 = lane >> 2, t = lane & 3;  // fragment row (= activation row m) and column
    const int gl = warp;  // the stage's group this warp reduces
    uint32_t ldm_off = 0, ldm_off2 = 0;
    if constexpr (kP64)
      ldmatrix_p64_offsets(gl, lane, ldm_off, ldm_off2);
    else
      ldm_off = ldmatrix_offset(gl, lane);
    // scale / bias of rows g8 and g8+8 of tile 0, group gl (streamed layout)
    const uint32_t sb_off = (kP64 ? kP64SbOff : kSbOff) + (uint32_t)(g8 * 16 + gl * 2);
    const uint32_t blk = base + L.sb;  // whole-tile block (not streamed)
    // n-tile nt covers activation rows 8 nt .. 8 nt + 7; lanes of padding
    // columns (m >= M) load nothing (byte-expanded format) or row 0 (packed
    // format); their sums are never stored
    const void *xrow[kNT];
    bool xvalid[kNT];
#pragma unroll
    for (int nt = 0; nt < kNT; ++nt) {
      xvalid[nt] = 8 * nt + g8 < a.M;
      xrow[nt] = static_cast<const uint8_t *>(a.x) +
                 (size_t)(xvalid[nt] ? 8 * nt + g8 : 0) * a.K * (kXF32 ? 4 : 2);
    }
    using XR = typename std::conditional<kP64, XRawP<kXF32>, XRaw<kXF32>>::type;
    auto load = [&](int nt, int grp) -> XR {
      if constexpr (kP64)
        return load_x_p64<kXF32>(xrow[nt], xvalid[nt], grp, t);
      else
        return load_x<kXF32>(xrow[nt], true, grp, t);
    };
    float acc[kNT][kTiles][4];
#pragma unroll
    for (int nt = 0; nt < kNT; ++nt)
#pragma unroll
      for (int i = 0; i < kTiles; ++i)
        acc[nt][i][0] = acc[nt][i][1] = acc[nt][i][2] = acc[nt][i][3] = 0.f;
    // every lane waits (each needs the acquire); the outcome is made warp-uniform
    ok = __all_sync(0xffffffffu, mbar_wait_u32(sb_bar, 0));
    pdl_wait();  // x and y belong to the preceding kernel until here
    int g = c_begin * kConsumerWarps + gl;
    // groups past K/64 (last stage of a ragged K) read a real group's
    // activations; their weights are skipped
    XR xnext[kNT];
#pragma unroll
    for (int nt = 0; nt < kNT; ++nt) xnext[nt] = load(nt, kStream ? g : min(g, groups - 1));
    int st = 0, ph = 0;  // stage of chunk c and the parity of its fill
    for (int c = c_begin; ok && c < c_end; ++c, g += kConsumerWarps) {
      XR xcur[kNT];
#pragma unroll
      for (int nt = 0; nt < kNT; ++nt) xcur[nt] = xnext[nt];
      // next stage's activations: the loads fly during this stage's work
      const int gn = min(g + kConsumerWarps, groups - 1);
#pragma unroll
      for (int nt = 0; nt < kNT; ++nt) xnext[nt] = load(nt, gn);
      if (!warp_wait_stage(full0 + 8u * st, ph)) {
        ok = false;
        break;
      }
      const uint32_t stage = base + st * L.stage;
      // scales/biases: [64][8] scales then [64][8] biases of this stage when
      // streamed, else the tile's whole [64][groups] block
      const uint32_t gb = (uint32_t)groups * 2;
      const bool real = kStream || g < groups;
      const uint32_t sbp = kStream ? stage + sb_off : blk + (uint32_t)(g8 * groups + g) * 2;
      const uint32_t srt = kStream ? 16 * 16 : 16 * gb, sr8 = kStream ? 8 * 16 : 8 * gb;
      const uint32_t sbb = kStream ? kRows * 16 : kRows * gb;
      if (real) {
        if constexpr (kP64) {
          if constexpr (kNT == 1)
            group_math_p64<kXF32>(acc[0], stage + ldm_off, stage + ldm_off2, xcur[0], sbp, srt,
                                  sr8, sbb);
          else
            group_math_p64_x2<kXF32>(acc, stage + ldm_off, stage + ldm_off2, xcur, sbp, srt, sr8,
                                     sbb);
        } else {
          if constexpr (kNT == 1)
            group_math<kXF32>(acc[0], stage + ldm_off, xcur[0], sbp, srt, sr8, sbb);
          else
            group_math_x2<kXF32>(acc, stage + ldm_off, xcur, sbp, srt, sr8, sbb);
        }
      }
      __syncwarp();
      if (lane == 0) mbar_arrive_u32(empty0 + 8u * st);
      if (++st == stages) {
        st = 0;
        ph ^= 1;
      }
    }
    if (!ok && lane == 0) atomicOr(&g_qmv_device_error, 2u);

    // cross-warp reduction in a fixed order, red[warp][row][col] in the drained ring
    float *red = reinterpret_cast<float *>(smem);
    asm volatile("bar.sync 1, %0;" ::"r"(kConsumerWarps * 32) : "memory");
#pragma unroll
    for (int nt = 0; nt < kNT; ++nt) {
#pragma unroll
      for (int rt = 0; rt < kTiles; ++rt) {
        float *p = red + ((size_t)warp * kRows + rt * 16) * kCols + 8 * nt;
        p[g8 * kCols + 2 * t] = acc[nt][rt][0];
        p[g8 * kCols + 2 * t + 1] = acc[nt][rt][1];
        p[(g8 + 8) * kCols + 2 * t] = acc[nt][rt][2];
        p[(g8 + 8) * kCols + 2 * t + 1] = acc[nt][rt][3];
      }
    }
    asm volatile("bar.sync 1, %0;" ::"r"(kConsumerWarps * 32) : "memory");
    // element e = col * 64 + row; thread handles e = tid + 256 h
#pragma unroll
    for (int h = 0; h < kParts; ++h) {
      const int e = threadIdx.x + h * kConsumerWarps * 32;
      const int col = e / kRows, row = e % kRows;
      float v = 0.f;
#pragma unroll
      for (int w = 0; w < kConsumerWarps; ++w) v += red[((size_t)w * kRows + row) * kCols + col];
      part[h] = v;
    }
    if (splits == 1) {
      if (!ok) return;
#pragma unroll
      for (int h = 0; h < kParts; ++h) {
        const int e = threadIdx.x + h * kConsumerWarps * 32;
        const int col = e / kRows, row = e % kRows;  // row fastest: coalesced stores
        if (col < a.M && row < rows) a.y[(size_t)col * a.N + n0 + row] = part[h];
      }
      return;
    }
  }

  // ---- split K: partial tiles meet in the first CTA of the cluster --------
  // (every thread of every CTA of the cluster takes part in both barriers)
  cluster_sync_all();  // all rings drained: the first CTA's ring may be overwritten
  const uint32_t rank = cluster_rank();
  if (warp < kConsumerWarps) {
    const uint32_t slot = map_shared_to_rank(base, 0) + rank * (kRows * kCols * 4);
#pragma unroll
    for (int h = 0; h < kParts; ++h)
      st_cluster_f32(slot + 4u * (threadIdx.x + h * kConsumerWarps * 32), part[h]);
  }
  cluster_sync_all();  // every partial has landed
  if (rank != 0 || warp >= kConsumerWarps) return;
  if (__any_sync(0xffffffffu, !ok)) return;
  const float *slots = reinterpret_cast<const float *>(smem);
#pragma unroll
  for (int h = 0; h < kParts; ++h) {
    const int e = threadIdx.x + h * kConsumerWarps * 32;
    const int col = e / kRows, row = e % kRows;
    float v = 0.f;
    for (int r = 0; r < splits; ++r) v += slots[r * kRows * kCols + e];
    if (col < a.M && row < rows) a.y[(size_t)col * a.N + n0 + row] = v;
  }
}

// Co-resident CTAs per SM allowed by registers and threads (cached per device).
template <bool kXF32, bool kStream, int kNT, bool kP64>
int occupancy_without_smem(int dev) {
  static std::atomic<int> cached[64] = {};
  if (dev < 0 || dev >= 64) return 1;
  int n = cached[dev].load(std::memory_order_relaxed);
  if (n == 0) {
    if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(
            &n, qmv_smallm_kernel<kXF32, kStream, kNT, kP64>, kThreads, 0) != cudaSuccess ||
        n < 1)
      n = 1;
    cached[dev].store(n, std::memory_order_relaxed);
  }
  return n;
}

template <bool kXF32, bool kStream, int kNT, bool kP64>
sv_status launch(const uint32_t *w, QmvArgs args, cudaStream_t stream) {
  static PerDeviceOnce attrs_once;
  const int dev = current_device();
  auto kern = qmv_smallm_kernel<kXF32, kStream, kNT, kP64>;
  int optin = 0;
  cudaDeviceGetAttribute(&optin, cudaDevAttrMaxSharedMemoryPerBlockOptin, dev);
  const cudaError_t ce = attrs_once.run([&] {
    return cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, optin);
  });
  if (ce != cudaSuccess)
    return fail(SV_ERR_CUDA, "qmv_smallm: cudaFuncSetAttribute failed: %s", cudaGetErrorString(ce));
  const int groups = args.K / 64;
  const int tiles = (args.N + kRows - 1) / kRows;
  const int n_chunks = (args.K + kStageInputs - 1) / kStageInputs;
  const int sms = device_sm_count();
  const int occ = occupancy_without_smem<kXF32, kStream, kNT, kP64>(dev);
  // split K over a cluster when the row tiles alone would leave CTA slots
  // idle, as far as the grid still fits in one wave of resident CTAs.  The
  // split decides the fp32 summation order, so it is chosen from the
  // occupancy of the <= 8-row kernel for every M: a row of a 9..16-row call
  // then equals the same row computed alone, bit for bit (at one CTA per SM
  // such a grid may take two waves).
  const int occ_split = occupancy_without_smem<kXF32, kStream, 1, kP64>(dev);
  int splits = 1;
  if (kStream) {
    const int fit = (occ_split * sms) / tiles;
    splits = std::max(1, std::min({fit, kMaxSplits, n_chunks}));
  }
  args.splits = splits;
  const int ctas = tiles * splits;
  // fill shared memory with stages at the occupancy the grid will reach
  const int per_sm = std::max(1, std::min({(ctas + sms - 1) / sms, occ, 8}));
  int smem_sm = 0;
  cudaDeviceGetAttribute(&smem_sm, cudaDevAttrMaxSharedMemoryPerMultiprocessor, dev);
  if (smem_sm <= 0) smem_sm = 228 * 1024;
  const uint32_t budget = (uint32_t)smem_sm / per_sm - 1024u;  // 1 KB reserved per CTA
  const bool sbs = kStream;
  const int per_cta_chunks = (n_chunks + splits - 1) / splits;
  const int max_stages = std::min(32, std::max(2, per_cta_chunks));
  int stages = 2;
  while (stages < max_stages && qmv_layout(groups, stages + 1, sbs, kNT, kP64).total <= budget)
    ++stages;
  Layout L = qmv_layout(groups, stages, sbs, kNT, kP64);
  while (L.total > (uint32_t)optin && stages > 2) L = qmv_layout(groups, --stages, sbs, kNT, kP64);
  if (L.total > (uint32_t)optin)
    return fail(SV_ERR_UNSUPPORTED, "qmv_smallm: K=%d needs %u bytes of shared memory",
                args.K, L.total);
  args.stages = stages;

  CUtensorMap wmap, smap, bmap;
  sv_status st =
      kP64 ? encode_2d(&wmap, CU_TENSOR_MAP_DATA_TYPE_16U4_ALIGN16B, w, (uint64_t)args.K,
                       (uint64_t)args.N, (uint64_t)args.K / 2, kP64BoxInputs, kRows,
                       CU_TENSOR_MAP_SWIZZLE_128B)
           : encode_2d(&wmap, CU_TENSOR_MAP_DATA_TYPE_UINT32, w, (uint64_t)args.K / 8,
                       (uint64_t)args.N, (uint64_t)args.K / 2, kBoxWords, kRows,
                       CU_TENSOR_MAP_SWIZZLE_128B);
  if (st != SV_OK) return st;
  if (sbs) {
    st = encode_2d(&smap, CU_TENSOR_MAP_DATA_TYPE_UINT16, args.s, (uint64_t)groups,
                   (uint64_t)args.N, (uint64_t)groups * 2, 8, kRows, CU_TENSOR_MAP_SWIZZLE_NONE);
    if (st != SV_OK) return st;
    st = encode_2d(&bmap, CU_TENSOR_MAP_DATA_TYPE_UINT16, args.b, (uint64_t)groups,
                   (uint64_t)args.N, (uint64_t)groups * 2, 8, kRows, CU_TENSOR_MAP_SWIZZLE_NONE);
    if (st != SV_OK) return st;
  } else {
    smap = wmap;  // unused
    bmap = wmap;
  }
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)ctas);
  cfg.blockDim = dim3(kThreads);
  cfg.dynamicSmemBytes = L.total;
  cfg.stream = stream;
  cudaLaunchAttribute attr[2];
  int na = 0;
  if (splits > 1) {
    attr[na].id = cudaLaunchAttributeClusterDimension;
    attr[na].val.clusterDim.x = (unsigned)splits;
    attr[na].val.clusterDim.y = 1;
    attr[na].val.clusterDim.z = 1;
    ++na;
  }
  if (pdl_enabled()) {
    attr[na].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[na].val.programmaticStreamSerializationAllowed = 1;
    ++na;
  }
  cfg.attrs = attr;
  cfg.numAttrs = na;
  if (cudaLaunchKernelEx(&cfg, kern, wmap, smap, bmap, args) != cudaSuccess) {
    return fail(SV_ERR_CUDA, "qmv_smallm: launch failed: %s",
                cudaGetErrorString(cudaGetLastError()));
  }
  return check_launch("qmv_smallm");
}

}  // namespace

unsigned take_device_error_qmv() {
  unsigned v = 0, zero = 0;
  cudaMemcpyFromSymbol(&v, g_qmv_device_error, sizeof v);
  cudaMemcpyToSymbol(g_qmv_device_error, &zero, sizeof zero);
  return v;
}

}  // namespace sv

using namespace sv;

extern "C" sv_status qmv_smallm(const uint32_t *w_packed, const uint16_t *scales,
                                const uint16_t *biases, const void *x, sv_dtype x_dtype, float *y,
                                int M, int N, int K, int group_size, int bits,
                                sv_stream_t stream) {
  clear_error();
  if (M < 0 || N < 0 || K <= 0)
    return fail(SV_ERR_INVALID_ARG, "qmv_smallm: need M >= 0, N >= 0, K > 0 (M=%d N=%d K=%d)", M,
                N, K);
  if (group_size != 64 || bits != 4)
    return fail(SV_ERR_UNSUPPORTED, "qmv_smallm: only bits=4, group_size=64 (got %d, %d)", bits,
                group_size);
  if (K % 64 != 0) return fail(SV_ERR_INVALID_ARG, "qmv_smallm: K=%d is not a multiple of 64", K);
  if (M > 16) return fail(SV_ERR_UNSUPPORTED, "qmv_smallm: M=%d > 16", M);
  if (x_dtype != SV_F32 && x_dtype != SV_BF16)
    return fail(SV_ERR_INVALID_ARG, "qmv_smallm: unknown x_dtype %d", (int)x_dtype);
  if (M == 0 || N == 0) return SV_OK;
  if (!w_packed || !scales || !biases || !x || !y)
    return fail(SV_ERR_INVALID_ARG, "qmv_smallm: null pointer");
  if (!aligned(w_packed, 16) || !aligned(scales, 16) || !aligned(biases, 16) || !aligned(x, 16))
    return fail(SV_ERR_INVALID_ARG,
                "qmv_smallm: w_packed, scales, biases and x must be 16-byte aligned");
  if (!aligned(y, 4)) return fail(SV_ERR_INVALID_ARG, "qmv_smallm: y must be 4-byte aligned");
  if ((long long)K > (1ll << 30) || (long long)N * (K / 8) > (1ll << 40) || N > (1 << 30))
    return fail(SV_ERR_INVALID_ARG, "qmv_smallm: N*K too large");
  const size_t wb = (size_t)N * K / 2, sbb = (size_t)N * (K / 64) * 2;
  const size_t xb = (size_t)M * K * (x_dtype == SV_F32 ? 4 : 2), yb = (size_t)M * N * 4;
  if (overlaps(y, yb, w_packed, wb) || overlaps(y, yb, scales, sbb) ||
      overlaps(y, yb, biases, sbb) || overlaps(y, yb, x, xb))
    return fail(SV_ERR_INVALID_ARG, "qmv_smallm: y overlaps an input");

  // scale/bias rows are 16-byte aligned for the copy engine when K % 512 == 0
  QmvArgs args{scales, biases, x, y, M, N, K, 0, 1, K % 512 == 0 ? 1 : 0};
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  const bool bf = x_dtype == SV_BF16;
  // byte-expandable boxes need K % 128 == 0 and 32-byte aligned weights
  // (always so when K % 512 == 0 and the caller's buffer is); the format is a
  // function of (K, w_packed) only, so every M of one weight matrix takes the
  // same per-row arithmetic
  if (K % 128 == 0 && aligned(w_packed, 32)) {
    if (M <= 8) {
      if (args.sb_stream)
        return bf ? launch<false, true, 1, true>(w_packed, args, s)
                  : launch<true, true, 1, true>(w_packed, args, s);
      return bf ? launch<false, false, 1, true>(w_packed, args, s)
                : launch<true, false, 1, true>(w_packed, args, s);
    }
    if (args.sb_stream)
      return bf ? launch<false, true, 2, true>(w_packed, args, s)
                : launch<true, true, 2, true>(w_packed, args, s);
    return bf ? launch<false, false, 2, true>(w_packed, args, s)
              : launch<true, false, 2, true>(w_packed, args, s);
  }
  // K % 128 == 64 (never streamed: K % 512 != 0), or weights only 16-byte aligned
  if (M <= 8) {
    if (args.sb_stream)
      return bf ? launch<false, true, 1, false>(w_packed, args, s)
                : launch<true, true, 1, false>(w_packed, args, s);
    return bf ? launch<false, false, 1, false>(w_packed, args, s)
              : launch<true, false, 1, false>(w_packed, args, s);
  }
  if (args.sb_stream)
    return bf ? launch<false, true, 2, false>(w_packed, args, s)
              : launch<true, true, 2, false>(w_packed, args, s);
  return bf ? launch<false, false, 2, false>(w_packed, args, s)
            : launch<true, false, 2, false>(w_packed, args, s);
}
