// qmv_wide.cu -- the 4-bit affine (group 64) product for wide verify blocks,
// up to 128 activation rows (meant for 17..128; qmv_smallm is the faster
// path at 16 or fewer), on the 5th-generation tensor cores, sm_103a.
//
// Sources: "MTP in llama.cpp", section "Theoretical maximum tg t/s" (the
// verify step streams the quantised weights once per cycle, whatever the
// number of rows) and "MTPLX 2.24x faster TPS", section "Layer 0: MLX
// Runtime" (the verify block's rows go through every 4-bit projection of the
// target model, the LM head included).  Batching the verify blocks of many
// sequences against one LM head (32 sequences x 4 rows = 128 rows) turns the
// mat-vec into a dense contraction: 2 M N K flops against N K / 2 weight
// bytes, about 64 flops per streamed byte at M = 128 -- tensor-core work.
//
//   y[m, n] = sum_i x[m, i] (s[n, g] q[n, i] + b[n, g]),   g = i / 64
//           = sum_i x[m, i] (s q)[n, i]  +  sum_g b[n, g] X[m, g],
//   X[m, g] = sum_{i in g} x[m, i].
//
// s q is a 12-bit product, so it is exactly hi + lo with hi = rn_bf16(s q)
// and lo = s q - hi (both bf16, lo exact); the first sum is two bf16 MMAs over
// the same activation tile.  The bias sum is an MMA too, over extra input
// columns: the "weights" b[n, g] (bf16, exact) against X[m, g] split the same
// way into bf16 hi and lo parts (a small prologue kernel writes them).
// Everything accumulates in fp32 in tensor memory, so no per-group work
// happens outside the tensor cores but the widening of the nibbles.
//
// One persistent CTA per SM, 128 weight rows (the MMA's M) per tile, tiles
// strided over the grid.  Warp roles:
//   warp 13     TMA producer of the packed weights (128 rows x 256 inputs,
//               128-byte swizzle) on its own mbarrier ring;
//   warp 14     TMA producer of the activation stages (64 inputs x rows,
//               128-byte swizzle, the MMA's K-major B operand) on a deep ring:
//               the tiles come from L2, every CTA re-reading them, and each
//               takes ~1.5 us to land;
//   warps 4-11  widen a 64-input group of their 32 rows (two warps per TMEM
//               lane quarter, 32 inputs each) into bf16 hi and -lo and store
//               them into a tensor-memory A stage (tcgen05.st);
//   warp 12     allocates tensor memory and issues tcgen05.mma (A from tensor
//               memory, B from shared memory) into one of two fp32
//               accumulators, releasing stages with tcgen05.commit;
//   warps 0-3   drain a finished accumulator (tcgen05.ld) into y while the
//               next tile accumulates in the other one.
// Every wait is bounded; a wait that gives up sets a device error word and the
// CTA winds down (in-flight copies and MMAs are waited for, bounded, and the
// tensor memory is freed before exit).
#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include <algorithm>
#include <cstdint>

#include "qmv_common.cuh"
#include "sv_device.cuh"
#include "sv_internal.h"

namespace sv {
namespace {

using qmv::encode_2d;
using qmv::tma_load_2d;

constexpr int kTileRows = 128;        // weight rows per tile (MMA M)
constexpr int kMaxRowsX = 128;        // activation rows (MMA N <= 128)
constexpr int kGroup = 64;            // inputs per quantisation group
constexpr int kStageGroups = 2;       // groups per pipeline stage
constexpr int kWBoxWords = 32;        // packed words per weight box row (128 B)
constexpr int kGroupsPerWBox = kWBoxWords * 8 / kGroup;  // 4
constexpr int kXStages = 4;           // activation ring (8 groups): covers the L2 latency
constexpr int kWStages = 4;           // packed-weight ring (16 groups)
constexpr int kAStages = 2;           // tensor-memory A stages (4 groups)
constexpr int kEpiWarps = 4, kDeqWarps = 8;
constexpr int kMmaWarp = kEpiWarps + kDeqWarps;  // 12
constexpr int kWTmaWarp = kMmaWarp + 1;          // 13
constexpr int kXTmaWarp = kWTmaWarp + 1;         // 14
constexpr int kWideThreads = (kXTmaWarp + 1) * 32;  // 480
constexpr uint32_t kTmemCols = 512;
constexpr uint32_t kDCols = 128;                   // one accumulator
constexpr uint32_t kAColBase = 2 * kDCols;         // A stages after the two accumulators
constexpr uint32_t kAGroupCols = 64;               // per group: hi 32 + (-lo) 32 columns
constexpr uint32_t kAStageCols = kStageGroups * kAGroupCols;
constexpr uint32_t kWBoxBytes = kTileRows * 128;   // 16 KB
constexpr uint32_t kXGroupBytes = kMaxRowsX * 128; // 16 KB at 128 rows
constexpr uint32_t kXStageBytes = kStageGroups * kXGroupBytes;
constexpr int kPrepThreads = 256;

static_assert(kAColBase + kAStages * kAStageCols <= kTmemCols, "tensor memory budget");
static_assert(kGroupsPerWBox % kStageGroups == 0, "a weight box holds whole stages");

__device__ unsigned int g_wide_device_error;

// ---- shared memory layout ---------------------------------------------------
struct WideLayout {
  uint32_t x, w, bar, tmem_slot, total;
};
__host__ __device__ inline WideLayout wide_layout() {
  WideLayout L;
  L.x = 0;
  L.w = L.x + kXStages * kXStageBytes;
  L.bar = L.w + kWStages * kWBoxBytes;
  // x_full, x_empty, w_full, w_empty, a_full, a_empty, d_full[2], d_empty[2],
  // mma_done
  const uint32_t nbar = 2 * kXStages + 2 * kWStages + 2 * kAStages + 5;
  L.tmem_slot = L.bar + 8 * nbar;
  L.total = L.tmem_slot + 16;
  return L;
}

struct WideArgs {
  const uint16_t *s, *b;  // [N][G] bf16 scales, biases
  float *y;               // [M][N]
  int M, N, K;
  int G;                  // K / 64 groups (a multiple of 8)
  int E;                  // bias groups: ceil(2 G / 64), rounded up to even
  int n_mma;              // MMA N: M rounded up to 16
};

// ---- tcgen05 ----------------------------------------------------------------
__device__ __forceinline__ void tmem_alloc(uint32_t slot_smem, uint32_t ncols) {
  asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(
                   slot_smem),
               "r"(ncols)
               : "memory");
}
__device__ __forceinline__ void tmem_relinquish() {
  asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
}
__device__ __forceinline__ void tmem_dealloc(uint32_t taddr, uint32_t ncols) {
  asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(ncols)
               : "memory");
}
__device__ __forceinline__ void tc_fence_before() {
  asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
}
__device__ __forceinline__ void tc_fence_after() {
  asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
}
// D[tmem] (+)= A[tmem] * B[smem desc]; kind::f16 with bf16 inputs, fp32 D.
__device__ __forceinline__ void tc_mma_ts(uint32_t d_tmem, uint32_t a_tmem, uint64_t b_desc,
                                          uint32_t idesc, uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\tsetp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], %2, %3, p;\n\t}" ::"r"(d_tmem),
      "r"(a_tmem), "l"(b_desc), "r"(idesc), "r"(accumulate)
      : "memory");
}
// The mbarrier completes one arrival when every tcgen05 operation this thread
// issued before has completed.
__device__ __forceinline__ void tc_commit(uint32_t bar) {
  asm volatile(
      "tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(bar)
      : "memory");
}
__device__ __forceinline__ void tc_st_x16(uint32_t taddr, const uint32_t (&v)[16]) {
  asm volatile(
      "tcgen05.st.sync.aligned.32x32b.x16.b32 [%0], {%1, %2, %3, %4, %5, %6, %7, %8, %9, %10, "
      "%11, %12, %13, %14, %15, %16};" ::"r"(taddr),
      "r"(v[0]), "r"(v[1]), "r"(v[2]), "r"(v[3]), "r"(v[4]), "r"(v[5]), "r"(v[6]), "r"(v[7]),
      "r"(v[8]), "r"(v[9]), "r"(v[10]), "r"(v[11]), "r"(v[12]), "r"(v[13]), "r"(v[14]),
      "r"(v[15])
      : "memory");
}
__device__ __forceinline__ void tc_wait_st() {
  asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory");
}
__device__ __forceinline__ void tc_ld_x32(uint32_t taddr, uint32_t (&v)[32]) {
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x32.b32 {%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, "
      "%11, %12, %13, %14, %15, %16, %17, %18, %19, %20, %21, %22, %23, %24, %25, %26, %27, "
      "%28, %29, %30, %31}, [%32];"
      : "=r"(v[0]), "=r"(v[1]), "=r"(v[2]), "=r"(v[3]), "=r"(v[4]), "=r"(v[5]), "=r"(v[6]),
        "=r"(v[7]), "=r"(v[8]), "=r"(v[9]), "=r"(v[10]), "=r"(v[11]), "=r"(v[12]),
        "=r"(v[13]), "=r"(v[14]), "=r"(v[15]), "=r"(v[16]), "=r"(v[17]), "=r"(v[18]),
        "=r"(v[19]), "=r"(v[20]), "=r"(v[21]), "=r"(v[22]), "=r"(v[23]), "=r"(v[24]),
        "=r"(v[25]), "=r"(v[26]), "=r"(v[27]), "=r"(v[28]), "=r"(v[29]), "=r"(v[30]),
        "=r"(v[31])
      : "r"(taddr)
      : "memory");
}
__device__ __forceinline__ void tc_wait_ld() {
  asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
}

// Shared-memory matrix descriptor of a K-major operand in the 128-byte swizzle
// layout: rows of 128 bytes, 8-row atoms 1024 bytes apart (the stride field),
// start address in 16-byte units; the leading-offset field is unused for this
// layout.  The tile base is 1024-byte aligned; a k16 step inside the atom
// moves the start address by 32 bytes.
__device__ __forceinline__ uint64_t smem_desc_sw128(uint32_t saddr) {
  uint64_t d = 0;
  d |= (uint64_t)((saddr & 0x3FFFFu) >> 4);  // start address
  d |= (uint64_t)1 << 16;                     // leading byte offset (unused), 16 B
  d |= (uint64_t)(1024u >> 4) << 32;          // stride byte offset: 8 rows x 128 B
  d |= (uint64_t)1 << 46;                     // descriptor version
  d |= (uint64_t)2 << 61;                     // 128-byte swizzle
  return d;
}
// Instruction descriptor, kind::f16: fp32 D, bf16 A and B, both K-major,
// M = 128, N = n.
__host__ __device__ constexpr uint32_t idesc_bf16(int n) {
  return (1u << 4)                        // D format: f32
         | (1u << 7)                      // A format: bf16
         | (1u << 10)                     // B format: bf16
         | ((uint32_t)(n >> 3) << 17)     // N / 8
         | ((uint32_t)(kTileRows >> 4) << 24);  // M / 16
}

// Warp-uniform wait: one non-blocking test first (a blocking test costs more
// even when the phase is already complete), then the bounded wait.
__device__ __forceinline__ bool mbar_test_u32(uint32_t bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.test_wait.parity.acquire.cta.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok)
      : "r"(bar), "r"(parity)
      : "memory");
  return ok != 0;
}
// One lane of the (converged) warp.
__device__ __forceinline__ bool elect_one() {
  uint32_t pred = 0;
  asm volatile(
      "{\n\t.reg .pred p;\n\telect.sync _|p, 0xffffffff;\n\tselp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(pred));
  return pred != 0;
}
__device__ __forceinline__ bool warp_wait_fast(uint32_t bar, uint32_t parity) {
  if (__all_sync(0xffffffffu, mbar_test_u32(bar, parity))) return true;
  return qmv::warp_wait_stage(bar, parity);
}

// ---- bf16x2 arithmetic (each a single rounding) ------------------------------
__device__ __forceinline__ uint32_t bf2_sub(uint32_t a, uint32_t b) {
  uint32_t d;
  asm("sub.rn.bf16x2 %0, %1, %2;" : "=r"(d) : "r"(a), "r"(b));
  return d;
}
__device__ __forceinline__ uint32_t bf2_mul(uint32_t a, uint32_t b) {
  uint32_t d;
  asm("mul.rn.bf16x2 %0, %1, %2;" : "=r"(d) : "r"(a), "r"(b));
  return d;
}
__device__ __forceinline__ uint32_t bf2_fma(uint32_t a, uint32_t b, uint32_t c) {
  uint32_t d;
  asm("fma.rn.bf16x2 %0, %1, %2, %3;" : "=r"(d) : "r"(a), "r"(b), "r"(c));
  return d;
}

// 2-D tensor copy with the default L2 policy (the activation tiles are re-read
// by every tile of the grid and should stay in L2).
__device__ __forceinline__ void tma_load_2d_keep(uint32_t dst, const CUtensorMap *map, int x,
                                                 int y, uint32_t bar) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cta.global.mbarrier::complete_tx::bytes "
      "[%0], [%1, {%2, %3}], [%4];" ::"r"(dst),
      "l"(map), "r"(x), "r"(y), "r"(bar)
      : "memory");
}

__device__ __forceinline__ uint4 lds128(uint32_t addr) {
  uint4 v;
  asm volatile("ld.shared.v4.u32 {%0, %1, %2, %3}, [%4];"
               : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
               : "r"(addr));
  return v;
}

// Eight nibbles (inputs 8 w .. 8 w + 7 of the row, LSB first) -> four bf16x2
// pairs of s q in natural input order, split as hi = rn(s q) and
// nlo = hi - s q = -(s q - hi) (exact; the MMA of the lo part negates A).  A
// pair (q_2p, q_2p+1) is widened to bf16 (128 + q) by placing byte p of the
// word and of the word shifted by one nibble in the two halves.
__device__ __forceinline__ void widen_word(uint32_t wd, uint32_t s2, uint32_t ns2, uint32_t *hi,
                                           uint32_t *nlo) {
  const uint32_t t = wd >> 4;
#pragma unroll
  for (int p = 0; p < 4; ++p) {
    const uint32_t sel = (uint32_t)p | ((uint32_t)(4 + p) << 8);
    const uint32_t v = and_or(prmt(wd, t, sel), qmv::kNibbleMask, qmv::kBf16Base);
    const uint32_t q2 = bf2_sub(v, qmv::kBf16Base);  // (q, q') exactly
    const uint32_t h = bf2_mul(s2, q2);
    hi[p] = h;
    nlo[p] = bf2_fma(ns2, q2, h);  // hi - s q, exact
  }
}

// X[m, g] over 64 inputs in ascending order (fp32), written as bf16 hi at
// column g and lo = rn(X - hi) at column G + g of row m of xb [M][Kb]; the
// columns from 2 G to Kb are zero.
__global__ void __launch_bounds__(kPrepThreads) wide_xsum_kernel(const uint16_t *x, uint16_t *xb,
                                                                 int M, int K, int G, int Kb) {
  pdl_launch_dependents();
  pdl_wait();  // x is the preceding kernel's output
  const size_t total = (size_t)M * Kb;
  for (size_t idx = (size_t)blockIdx.x * kPrepThreads + threadIdx.x; idx < total;
       idx += (size_t)gridDim.x * kPrepThreads) {
    const int m = (int)(idx / Kb), j = (int)(idx - (size_t)m * Kb);
    uint16_t out = 0;
    if (j < 2 * G) {
      const int g = j < G ? j : j - G;
      const uint4 *p = reinterpret_cast<const uint4 *>(x + (size_t)m * K + (size_t)g * kGroup);
      uint4 v[8];
#pragma unroll
      for (int u = 0; u < 8; ++u) v[u] = __ldg(p + u);
      float sum = 0.f;
#pragma unroll
      for (int u = 0; u < 8; ++u) {
        const uint32_t w4[4] = {v[u].x, v[u].y, v[u].z, v[u].w};
#pragma unroll
        for (int h = 0; h < 4; ++h) {
          sum += __uint_as_float(w4[h] << 16);
          sum += __uint_as_float(w4[h] & 0xFFFF0000u);
        }
      }
      const __nv_bfloat16 hi = __float2bfloat16_rn(sum);
      out = j < G ? __bfloat16_as_ushort(hi)
                  : __bfloat16_as_ushort(__float2bfloat16_rn(sum - __bfloat162float(hi)));
    }
    xb[idx] = out;
  }
}

// Stages of a tile: two groups each; stage p < G / 2 holds weight groups
// 2p, 2p + 1, the last E / 2 stages the bias columns.  Every role walks the
// same sequence of stages; ring slots and phases advance incrementally.
__global__ void __launch_bounds__(kWideThreads, 1)
    qmv_wide_kernel(const __grid_constant__ CUtensorMap wmap,
                    const __grid_constant__ CUtensorMap xmap,
                    const __grid_constant__ CUtensorMap xbmap, const WideArgs a) {
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  const uint32_t raw = smem_addr(smem_raw);
  const uint32_t base = raw + ((1024u - (raw & 1023u)) & 1023u);
  const WideLayout L = wide_layout();
  const uint32_t xs0 = base + L.x, ws0 = base + L.w;
  const uint32_t x_full = base + L.bar, x_empty = x_full + 8u * kXStages;
  const uint32_t w_full = x_empty + 8u * kXStages, w_empty = w_full + 8u * kWStages;
  const uint32_t a_full = w_empty + 8u * kWStages, a_empty = a_full + 8u * kAStages;
  const uint32_t d_full = a_empty + 8u * kAStages, d_empty = d_full + 16u;
  const uint32_t mma_done = d_empty + 16u;
  const volatile uint32_t *slot =
      reinterpret_cast<const volatile uint32_t *>(smem_raw + (base - raw) + L.tmem_slot);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int tiles = (a.N + kTileRows - 1) / kTileRows;
  const int n_local =
      (int)blockIdx.x < tiles ? (tiles - 1 - (int)blockIdx.x) / (int)gridDim.x + 1 : 0;
  const int Pw = a.G / kStageGroups;             // weight stages per tile
  const int Pt = Pw + a.E / kStageGroups;        // all stages per tile

  if (threadIdx.x == 0) {
    for (int i = 0; i < kXStages; ++i) {
      mbar_init_u32(x_full + 8u * i, 1);
      mbar_init_u32(x_empty + 8u * i, 1);
    }
    for (int i = 0; i < kWStages; ++i) {
      mbar_init_u32(w_full + 8u * i, 1);
      mbar_init_u32(w_empty + 8u * i, kDeqWarps);
    }
    for (int i = 0; i < kAStages; ++i) {
      mbar_init_u32(a_full + 8u * i, kDeqWarps);
      mbar_init_u32(a_empty + 8u * i, 1);
    }
    for (int i = 0; i < 2; ++i) {
      mbar_init_u32(d_full + 8u * i, 1);
      mbar_init_u32(d_empty + 8u * i, kEpiWarps);
    }
    mbar_init_u32(mma_done, 1);
    fence_mbar_init();
  }
  if (warp == kMmaWarp) {
    tmem_alloc(base + L.tmem_slot, kTmemCols);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *slot;
  pdl_launch_dependents();

  if (warp == kWTmaWarp) {
    // --------------------------- weight producer --------------------------
    // weights do not depend on earlier kernels: no griddepcontrol.wait here
    if (lane == 0) {
      const uint64_t wpol = l2_policy_evict_first();
      long long ib = 0;
      uint32_t sw = 0, pw = 0;  // slot and phase of box ib
      bool ok = true;
      for (int t = 0; ok && t < n_local; ++t) {
        const int n0 = ((int)blockIdx.x + t * (int)gridDim.x) * kTileRows;
        for (int j = 0; j < a.G; j += kGroupsPerWBox, ++ib) {
          if (ib >= kWStages && !mbar_wait_u32(w_empty + 8u * sw, pw ^ 1u)) {
            atomicOr(&g_wide_device_error, 1u);
            ok = false;
            break;
          }
          mbar_arrive_expect_tx_u32(w_full + 8u * sw, kWBoxBytes);
          tma_load_2d(ws0 + sw * kWBoxBytes, &wmap, j * 8, n0, w_full + 8u * sw, wpol);
          if (++sw == (uint32_t)kWStages) {
            sw = 0;
            pw ^= 1u;
          }
        }
      }
      // every copy issued has landed before the CTA may exit (normally the
      // consumers have waited for all of them already)
      for (long long k = std::max(0ll, ib - kWStages); k < ib; ++k)
        (void)mbar_wait_u32(w_full + 8u * (uint32_t)(k % kWStages),
                            (uint32_t)((k / kWStages) & 1));
    }
    __syncwarp();
  } else if (warp == kXTmaWarp) {
    // ------------------------- activation producer ------------------------
    if (lane == 0) {
      pdl_wait();  // the activations and their group sums are earlier kernels' output
      long long i = 0;
      uint32_t sx = 0, px = 0;  // slot and phase of stage i
      bool ok = true;
      const uint32_t bytes = (uint32_t)kStageGroups * (uint32_t)a.n_mma * 128u;
      for (int t = 0; ok && t < n_local; ++t) {
        for (int p = 0; p < Pt; ++p, ++i) {
          if (i >= kXStages && !mbar_wait_u32(x_empty + 8u * sx, px ^ 1u)) {
            atomicOr(&g_wide_device_error, 2u);
            ok = false;
            break;
          }
          mbar_arrive_expect_tx_u32(x_full + 8u * sx, bytes);
          const uint32_t dst = xs0 + sx * kXStageBytes;
          for (int g2 = 0; g2 < kStageGroups; ++g2) {
            if (p < Pw)
              tma_load_2d_keep(dst + g2 * kXGroupBytes, &xmap, (kStageGroups * p + g2) * kGroup,
                               0, x_full + 8u * sx);
            else
              tma_load_2d_keep(dst + g2 * kXGroupBytes, &xbmap,
                               (kStageGroups * (p - Pw) + g2) * kGroup, 0, x_full + 8u * sx);
          }
          if (++sx == (uint32_t)kXStages) {
            sx = 0;
            px ^= 1u;
          }
        }
      }
      for (long long k = std::max(0ll, i - kXStages); k < i; ++k)
        (void)mbar_wait_u32(x_full + 8u * (uint32_t)(k % kXStages),
                            (uint32_t)((k / kXStages) & 1));
    }
    __syncwarp();
  } else if (warp == kMmaWarp) {
    // ------------------------------ MMA issuer ----------------------------
    // The whole warp runs the loop (descriptors and addresses stay
    // warp-uniform); one elected lane issues each MMA and commit.
    const uint32_t idesc = idesc_bf16(a.n_mma);
    const uint32_t idesc_neg = idesc | (1u << 13);  // negate A: the stored lo parts are -lo
    uint32_t sa = 0, pa = 0, sx = 0, px = 0;        // slot and phase of the next stage
    bool ok = true;
    for (int t = 0; ok && t < n_local; ++t) {
      const int tb = t & 1;
      if (t >= 2 &&
          !qmv::warp_wait_stage(d_empty + 8u * tb, (uint32_t)(((t >> 1) - 1) & 1))) {
        if (lane == 0) atomicOr(&g_wide_device_error, 4u);
        ok = false;
        break;
      }
      tc_fence_after();
      const uint32_t d = tmem + (uint32_t)tb * kDCols;
      for (int p = 0; p < Pt; ++p) {
        // a_full completes after the activation stage landed (the first
        // widening warp waits for x_full before it arrives): one poll here
        if (!qmv::warp_wait_stage(a_full + 8u * sa, pa)) {
          if (lane == 0) atomicOr(&g_wide_device_error, 8u);
          ok = false;
          break;
        }
        tc_fence_after();
        const uint32_t at = tmem + kAColBase + sa * kAStageCols;
        const uint32_t xb = xs0 + sx * kXStageBytes;
        if (elect_one()) {
#pragma unroll
          for (int g2 = 0; g2 < kStageGroups; ++g2) {
            const uint32_t ag = at + (uint32_t)g2 * kAGroupCols;
            const uint64_t bd = smem_desc_sw128(xb + (uint32_t)g2 * kXGroupBytes);
            if (p < Pw) {
#pragma unroll
              for (int ks = 0; ks < 4; ++ks) {
                tc_mma_ts(d, ag + 8u * ks, bd + 2u * ks, idesc,
                          (p > 0 || g2 > 0 || ks > 0) ? 1u : 0u);
                tc_mma_ts(d, ag + 32u + 8u * ks, bd + 2u * ks, idesc_neg, 1u);
              }
            } else {
#pragma unroll
              for (int ks = 0; ks < 4; ++ks) tc_mma_ts(d, ag + 8u * ks, bd + 2u * ks, idesc, 1u);
            }
          }
          tc_commit(a_empty + 8u * sa);
          tc_commit(x_empty + 8u * sx);
        }
        __syncwarp();
        if (++sa == (uint32_t)kAStages) {
          sa = 0;
          pa ^= 1u;
        }
        if (++sx == (uint32_t)kXStages) {
          sx = 0;
          px ^= 1u;
        }
      }
      if (ok && elect_one()) tc_commit(d_full + 8u * tb);
      __syncwarp();
    }
    // every MMA issued has completed before the tensor memory is freed
    if (elect_one()) {
      tc_commit(mma_done);
      (void)mbar_wait_u32(mma_done, 0);
    }
    __syncwarp();
  } else if (warp >= kEpiWarps) {
    // ------------------------------ widening ------------------------------
    // two warps per TMEM lane quarter, each one half (32 inputs) of every
    // group of its 32 rows; a stage's two groups are widened together (their
    // math interleaved)
    const int qd = warp & 3, hf = (warp - kEpiWarps) >> 2;
    const int r = qd * 32 + lane;
    const uint32_t lane_base = (uint32_t)(qd * 32) << 16;
    const uint32_t arow = tmem + lane_base + kAColBase + 16u * (uint32_t)hf;
    long long i = 0;
    uint32_t sa = 0, pa = 0, sw = 0, pw = 0;  // A slot/phase of stage i, W slot/phase
    uint32_t sx = 0, px = 0;                  // X slot/phase (first widening warp)
    bool ok = true;
    for (int t = 0; ok && t < n_local; ++t) {
      const int n = ((int)blockIdx.x + t * (int)gridDim.x) * kTileRows + r;
      const bool valid = n < a.N;
      const uint16_t *srow = a.s + (size_t)(valid ? n : 0) * a.G;
      const uint16_t *brow = a.b + (size_t)(valid ? n : 0) * a.G;
      uint4 scur = make_uint4(0, 0, 0, 0), snext = make_uint4(0, 0, 0, 0);
      if (valid) snext = __ldg(reinterpret_cast<const uint4 *>(srow));
      for (int p = 0; p < Pt; ++p, ++i) {
        const int j = kStageGroups * p;  // first group of the stage
        uint32_t hi0[16], nlo0[16], hi1[16], nlo1[16];
        if (p < Pw) {
          if ((j & 7) == 0) {
            scur = snext;
            if (valid && j + 8 < a.G)
              snext = __ldg(reinterpret_cast<const uint4 *>(srow + j + 8));
          }
        } else {
          // bias columns k' = 64 e + 32 hf + 2 q (+1): b[n][k' mod G] below 2 G
#pragma unroll
          for (int g2 = 0; g2 < kStageGroups; ++g2) {
            const int kb = kGroup * (j - a.G + g2) + 32 * hf;
#pragma unroll
            for (int q = 0; q < 16; ++q) {
              const int kp = kb + 2 * q;
              uint32_t v = 0;
              if (valid && kp < 2 * a.G)
                v = __ldg(reinterpret_cast<const uint32_t *>(brow + (kp < a.G ? kp : kp - a.G)));
              (g2 == 0 ? hi0 : hi1)[q] = v;
            }
          }
        }
        if (i >= kAStages && !warp_wait_fast(a_empty + 8u * sa, pa ^ 1u)) {
          if (lane == 0) atomicOr(&g_wide_device_error, 16u);
          ok = false;
          break;
        }
        const uint32_t col = arow + sa * kAStageCols;
        if (p < Pw) {
          if ((j & 3) == 0 && !warp_wait_fast(w_full + 8u * sw, pw)) {
            if (lane == 0) atomicOr(&g_wide_device_error, 32u);
            ok = false;
            break;
          }
          tc_fence_after();
          // 16-byte chunks 2 (j % 4) + hf and 2 (j % 4 + 1) + hf of the box row
          const uint32_t rbase = ws0 + sw * kWBoxBytes + (uint32_t)r * 128u;
          const int c0 = 2 * (j & 3) + hf, c1 = c0 + 2;
          const uint4 w0 = lds128(rbase + ((uint32_t)(c0 ^ (r & 7)) << 4));
          const uint4 w1 = lds128(rbase + ((uint32_t)(c1 ^ (r & 7)) << 4));
          const uint32_t sword =
              (j & 4) ? ((j & 2) ? scur.w : scur.z) : ((j & 2) ? scur.y : scur.x);
          const uint32_t s0 = prmt(sword, 0u, 0x1010u), s1 = prmt(sword, 0u, 0x3232u);
          const uint32_t ns0 = s0 ^ 0x80008000u, ns1 = s1 ^ 0x80008000u;
          widen_word(w0.x, s0, ns0, hi0 + 0, nlo0 + 0);
          widen_word(w1.x, s1, ns1, hi1 + 0, nlo1 + 0);
          widen_word(w0.y, s0, ns0, hi0 + 4, nlo0 + 4);
          widen_word(w1.y, s1, ns1, hi1 + 4, nlo1 + 4);
          widen_word(w0.z, s0, ns0, hi0 + 8, nlo0 + 8);
          widen_word(w1.z, s1, ns1, hi1 + 8, nlo1 + 8);
          widen_word(w0.w, s0, ns0, hi0 + 12, nlo0 + 12);
          widen_word(w1.w, s1, ns1, hi1 + 12, nlo1 + 12);
          if ((j & 3) == 2) {  // the box's last stage: its rows are read
            __syncwarp();
            if (lane == 0) mbar_arrive_u32(w_empty + 8u * sw);
            if (++sw == (uint32_t)kWStages) {
              sw = 0;
              pw ^= 1u;
            }
          }
          tc_st_x16(col, hi0);
          tc_st_x16(col + 32u, nlo0);
          tc_st_x16(col + kAGroupCols, hi1);
          tc_st_x16(col + kAGroupCols + 32u, nlo1);
        } else {
          tc_fence_after();
          tc_st_x16(col, hi0);
          tc_st_x16(col + kAGroupCols, hi1);
        }
        tc_wait_st();
        tc_fence_before();
        if (warp == kEpiWarps) {  // the stage's activations too, for the MMA warp
          if (!qmv::warp_wait_stage(x_full + 8u * sx, px)) {
            if (lane == 0) atomicOr(&g_wide_device_error, 128u);
            ok = false;
          }
          if (++sx == (uint32_t)kXStages) {
            sx = 0;
            px ^= 1u;
          }
        }
        __syncwarp();
        if (lane == 0) mbar_arrive_u32(a_full + 8u * sa);
        if (++sa == (uint32_t)kAStages) {
          sa = 0;
          pa ^= 1u;
        }
        if (!ok) break;
      }
    }
  } else {
    // ------------------------------ epilogue ------------------------------
    const uint32_t lane_base = (uint32_t)(warp * 32) << 16;
    bool waited = false;
    for (int t = 0; t < n_local; ++t) {
      const int tb = t & 1;
      if (!qmv::warp_wait_stage(d_full + 8u * tb, (uint32_t)((t >> 1) & 1))) {
        if (lane == 0) atomicOr(&g_wide_device_error, 64u);
        break;
      }
      tc_fence_after();
      if (!waited) {  // y belongs to the preceding kernels until here
        pdl_wait();
        waited = true;
      }
      const int n = ((int)blockIdx.x + t * (int)gridDim.x) * kTileRows + warp * 32 + lane;
      for (int c = 0; c < a.M; c += 32) {
        uint32_t v[32];
        tc_ld_x32(tmem + lane_base + (uint32_t)tb * kDCols + (uint32_t)c, v);
        tc_wait_ld();
        if (n < a.N) {
#pragma unroll
          for (int q = 0; q < 32; ++q)
            if (c + q < a.M) a.y[(size_t)(c + q) * a.N + n] = __uint_as_float(v[q]);
        }
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive_u32(d_empty + 8u * tb);
    }
  }

  tc_fence_before();
  __syncthreads();
  if (warp == kMmaWarp) {
    tc_fence_after();
    tmem_dealloc(tmem, kTmemCols);
  }
}

int wide_bias_stages(int K) {
  const int e = (2 * (K / kGroup) + kGroup - 1) / kGroup;
  return (e + kStageGroups - 1) / kStageGroups * kStageGroups;
}
size_t wide_ws_bytes(int M, int K) {
  const size_t kb = (size_t)wide_bias_stages(K) * kGroup;
  return ((size_t)M * kb * 2 + 255) / 256 * 256;
}

sv_status wide_validate(int M, int N, int K, const char *who) {
  if (M < 0 || N < 0 || K <= 0)
    return fail(SV_ERR_INVALID_ARG, "%s: need M >= 0, N >= 0, K > 0 (M=%d N=%d K=%d)", who, M, N,
                K);
  if (M > kMaxRowsX) return fail(SV_ERR_UNSUPPORTED, "%s: M=%d > %d", who, M, kMaxRowsX);
  if (K % 512 != 0)
    return fail(SV_ERR_INVALID_ARG, "%s: K=%d is not a multiple of 512", who, K);
  if ((long long)K > (1ll << 24) || (long long)N * (K / 8) > (1ll << 40) || N > (1 << 30))
    return fail(SV_ERR_INVALID_ARG, "%s: N*K too large", who);
  return SV_OK;
}

}  // namespace

unsigned take_device_error_wide() {
  unsigned v = 0, zero = 0;
  cudaMemcpyFromSymbol(&v, g_wide_device_error, sizeof v);
  cudaMemcpyToSymbol(g_wide_device_error, &zero, sizeof zero);
  return v;
}

}  // namespace sv

using namespace sv;

extern "C" size_t qmv_wide_workspace_bytes(int M, int K) {
  clear_error();
  if (wide_validate(M, 1, K, "qmv_wide_workspace_bytes") != SV_OK) return 0;
  return wide_ws_bytes(M, K);
}

extern "C" sv_status qmv_wide(const uint32_t *w_packed, const uint16_t *scales,
                              const uint16_t *biases, const uint16_t *x, float *y, int M, int N,
                              int K, void *workspace, size_t workspace_bytes,
                              sv_stream_t stream) {
  clear_error();
  sv_status st = wide_validate(M, N, K, "qmv_wide");
  if (st != SV_OK) return st;
  if (M == 0 || N == 0) return SV_OK;
  if (!w_packed || !scales || !biases || !x || !y || !workspace)
    return fail(SV_ERR_INVALID_ARG, "qmv_wide: null pointer");
  if (!aligned(w_packed, 16) || !aligned(scales, 16) || !aligned(biases, 16) || !aligned(x, 16))
    return fail(SV_ERR_INVALID_ARG,
                "qmv_wide: w_packed, scales, biases and x must be 16-byte aligned");
  if (!aligned(y, 4)) return fail(SV_ERR_INVALID_ARG, "qmv_wide: y must be 4-byte aligned");
  if (!aligned(workspace, 256))
    return fail(SV_ERR_INVALID_ARG, "qmv_wide: workspace must be 256-byte aligned");
  const size_t need = wide_ws_bytes(M, K);
  if (workspace_bytes < need)
    return fail(SV_ERR_INVALID_ARG, "qmv_wide: workspace of %zu bytes, need %zu",
                workspace_bytes, need);
  const size_t wb = (size_t)N * K / 2, sbb = (size_t)N * (K / 64) * 2;
  const size_t xbytes = (size_t)M * K * 2, yb = (size_t)M * N * 4;
  if (overlaps(y, yb, w_packed, wb) || overlaps(y, yb, scales, sbb) ||
      overlaps(y, yb, biases, sbb) || overlaps(y, yb, x, xbytes) ||
      overlaps(y, yb, workspace, need))
    return fail(SV_ERR_INVALID_ARG, "qmv_wide: y overlaps an input or the workspace");
  if (overlaps(workspace, need, x, xbytes) || overlaps(workspace, need, w_packed, wb) ||
      overlaps(workspace, need, scales, sbb) || overlaps(workspace, need, biases, sbb))
    return fail(SV_ERR_INVALID_ARG, "qmv_wide: the workspace overlaps an input");

  const int dev = current_device();
  const int sms = device_sm_count();
  int optin = 0;
  cudaDeviceGetAttribute(&optin, cudaDevAttrMaxSharedMemoryPerBlockOptin, dev);
  const uint32_t smem = wide_layout().total + 1024u;  // + alignment slack
  if (smem > (uint32_t)optin)
    return fail(SV_ERR_UNSUPPORTED, "qmv_wide: needs %u bytes of shared memory", smem);
  static PerDeviceOnce attrs_once;
  const cudaError_t ce = attrs_once.run([&] {
    return cudaFuncSetAttribute(qmv_wide_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                (int)smem);
  });
  if (ce != cudaSuccess)
    return fail(SV_ERR_CUDA, "qmv_wide: cudaFuncSetAttribute failed: %s", cudaGetErrorString(ce));

  WideArgs args{scales, biases, y, M, N, K, K / kGroup, wide_bias_stages(K), (M + 15) / 16 * 16};
  const int kb = args.E * kGroup;
  uint16_t *xb = static_cast<uint16_t *>(workspace);
  CUtensorMap wmap, xmap, xbmap;
  st = encode_2d(&wmap, CU_TENSOR_MAP_DATA_TYPE_UINT32, w_packed, (uint64_t)K / 8, (uint64_t)N,
                 (uint64_t)K / 2, kWBoxWords, kTileRows, CU_TENSOR_MAP_SWIZZLE_128B);
  if (st != SV_OK) return st;
  st = encode_2d(&xmap, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, x, (uint64_t)K, (uint64_t)M,
                 (uint64_t)K * 2, kGroup, (uint32_t)args.n_mma, CU_TENSOR_MAP_SWIZZLE_128B);
  if (st != SV_OK) return st;
  st = encode_2d(&xbmap, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, xb, (uint64_t)kb, (uint64_t)M,
                 (uint64_t)kb * 2, kGroup, (uint32_t)args.n_mma, CU_TENSOR_MAP_SWIZZLE_128B);
  if (st != SV_OK) return st;

  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  const int na = pdl_enabled() ? 1 : 0;

  const size_t prep_total = (size_t)M * kb;
  cudaLaunchConfig_t pc = {};
  pc.gridDim = dim3((unsigned)std::max<size_t>(
      1, std::min<size_t>((prep_total + kPrepThreads - 1) / kPrepThreads, (size_t)sms * 4)));
  pc.blockDim = dim3(kPrepThreads);
  pc.stream = s;
  pc.attrs = attr;
  pc.numAttrs = na;
  if (cudaLaunchKernelEx(&pc, wide_xsum_kernel, x, xb, M, K, args.G, kb) != cudaSuccess)
    return fail(SV_ERR_CUDA, "qmv_wide: prologue launch failed: %s",
                cudaGetErrorString(cudaGetLastError()));
  if ((st = check_launch("qmv_wide (prologue)")) != SV_OK) return st;

  const int tiles = (N + kTileRows - 1) / kTileRows;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)std::min(tiles, sms));
  cfg.blockDim = dim3(kWideThreads);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = s;
  cfg.attrs = attr;
  cfg.numAttrs = na;
  if (cudaLaunchKernelEx(&cfg, qmv_wide_kernel, wmap, xmap, xbmap, args) != cudaSuccess)
    return fail(SV_ERR_CUDA, "qmv_wide: launch failed: %s",
                cudaGetErrorString(cudaGetLastError()));
  return check_launch("qmv_wide");
}
