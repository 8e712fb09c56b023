// qmv_smallm.cu -- small-M (1..8 rows) 4-bit affine group-64 quantised mat-vec
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
//  * one CTA per tile of 16*RT output rows over the whole of K; the grid is
//    sized so the tiles of a typical projection are resident together, and
//    every CTA keeps several KB of weights in flight;
//  * a producer warp streams the tile's rows through a ring of shared-memory
//    stages with bulk async copies (cp.async.bulk, complete_tx on an
//    mbarrier, L2 evict-first), and loads the tile's scales/biases once;
//  * four consumer warps split each 512-input stage (two 64-groups each:
//    split-K over warps) and reduce through shared memory at the end in a
//    fixed order, so results are deterministic;
//  * each weight is read from shared memory once and used for all M rows: the
//    nibbles are widened in registers to bf16 (128 + q, exact) and fed to the
//    tensor cores as the 16-row A operand of mma.m16n8k16 with the (<= 8)
//    activation rows as B; per group the fp32 result is scaled,
//        acc += s * D + (b - 128 s) * sum(x),
//    with sum(x) itself taken from an all-ones MMA.  Products are exact, the
//    accumulation is fp32.  CUDA-core FMAs alone cannot keep up with the
//    HBM stream at M >= 2 on this part (4 FMAs + unpack per weight per row
//    against ~3.3 issue slots per streamed weight), the MMA path costs the
//    same at every M.
//  * programmatic dependent launch: the weight stream may start before the
//    preceding kernel on the stream ends; x is read after griddepcontrol.wait.
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include <algorithm>
#include <cstdint>

#include "sv_device.cuh"
#include "sv_internal.h"

namespace sv {
namespace {

constexpr int kConsumerWarps = 4;
constexpr int kGroupsPerWarp = 2;                                  // per stage
constexpr int kStageInputs = kConsumerWarps * kGroupsPerWarp * 64;  // 512
// Shared-memory bytes of one row of a stage: 256 data + 32 pad, so the
// 64-bit fragment loads of 16 lanes (4 rows x 4 lanes) hit distinct banks.
constexpr int kStageRowBytes = kStageInputs / 2 + 32;
constexpr int kThreads = (kConsumerWarps + 1) * 32;
constexpr uint32_t kBf16One2 = 0x3F803F80u;   // bf16x2 (1, 1)
constexpr uint32_t kNibbleMask = 0x000F000Fu;
constexpr uint32_t kBf16Base = 0x43004300u;   // bf16x2 (128, 128)

__device__ unsigned int g_qmv_device_error;

struct QmvArgs {
  const uint32_t *w;   // [N][K/8]
  const uint16_t *s;   // [N][K/64] bf16
  const uint16_t *b;   // [N][K/64] bf16
  const void *x;       // [M][K] fp32 or bf16
  float *y;            // [M][N]
  int M, N, K;
  int stages;
};

struct Layout {
  size_t sb, red, bar, total;
};

__host__ __device__ inline size_t round_up(size_t v, size_t a) { return (v + a - 1) / a * a; }

__host__ __device__ inline Layout qmv_layout(int rows_cta, int groups, int stages) {
  Layout L;
  L.sb = (size_t)stages * rows_cta * kStageRowBytes;
  L.red = L.sb + round_up((size_t)2 * rows_cta * groups * 2, 16);
  L.bar = L.red + (size_t)kConsumerWarps * rows_cta * 8 * sizeof(float);
  L.total = L.bar + (size_t)(2 * stages + 1) * sizeof(uint64_t);
  return L;
}

// B fragments of one 64-group for the activation row this lane feeds.
// Lane (row m = lane/4, t = lane%4) covers inputs 64g + 16t + [0,16) as two
// 8-input slots; each slot feeds two k16 MMA steps whose k order pairs input
// j with input j+4 -- the order the nibble widening below produces.
template <bool kXF32>
__device__ __forceinline__ void load_b_fragments(const QmvArgs &a, int m, bool valid, int g, int t,
                                                 uint32_t (&hi)[8], uint32_t (&lo)[8]) {
  if constexpr (!kXF32) {
    uint4 v0 = make_uint4(0, 0, 0, 0), v1 = v0;
    if (valid) {
      const uint16_t *p = static_cast<const uint16_t *>(a.x) + (size_t)m * a.K + g * 64 + t * 16;
      v0 = *reinterpret_cast<const uint4 *>(p);
      v1 = *reinterpret_cast<const uint4 *>(p + 8);
    }
    hi[0] = prmt(v0.x, v0.z, 0x5410);  // (x0, x4)
    hi[1] = prmt(v0.x, v0.z, 0x7632);  // (x1, x5)
    hi[2] = prmt(v0.y, v0.w, 0x5410);  // (x2, x6)
    hi[3] = prmt(v0.y, v0.w, 0x7632);  // (x3, x7)
    hi[4] = prmt(v1.x, v1.z, 0x5410);
    hi[5] = prmt(v1.x, v1.z, 0x7632);
    hi[6] = prmt(v1.y, v1.w, 0x5410);
    hi[7] = prmt(v1.y, v1.w, 0x7632);
#pragma unroll
    for (int i = 0; i < 8; ++i) lo[i] = 0;
  } else {
    float v[16];
#pragma unroll
    for (int i = 0; i < 16; ++i) v[i] = 0.f;
    if (valid) {
      const float *p = static_cast<const float *>(a.x) + (size_t)m * a.K + g * 64 + t * 16;
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        const float4 f = reinterpret_cast<const float4 *>(p)[i];
        v[4 * i + 0] = f.x;
        v[4 * i + 1] = f.y;
        v[4 * i + 2] = f.z;
        v[4 * i + 3] = f.w;
      }
    }
    // pair (j, j+4) of each 8-input slot; x = hi + lo with both bf16
#pragma unroll
    for (int slot = 0; slot < 2; ++slot)
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        const float xa = v[8 * slot + j], xb = v[8 * slot + j + 4];
        const __nv_bfloat162 h = __floats2bfloat162_rn(xa, xb);
        const __nv_bfloat162 l =
            __floats2bfloat162_rn(xa - __low2float(h), xb - __high2float(h));
        hi[4 * slot + j] = *reinterpret_cast<const uint32_t *>(&h);
        lo[4 * slot + j] = *reinterpret_cast<const uint32_t *>(&l);
      }
  }
}

// Two k16 MMA steps for one packed word (8 inputs) of rows r and r+8.
// Widening: (w >> 4j) & 0x000F000F | 0x43004300 is the bf16 pair
// (128 + q_j, 128 + q_{j+4}).
template <bool kXF32>
__device__ __forceinline__ void mma_word(float (&d)[4], uint32_t wr, uint32_t wr8,
                                         const uint32_t *hi, const uint32_t *lo) {
  const uint32_t a0 = and_or(wr, kNibbleMask, kBf16Base);
  const uint32_t a0r8 = and_or(wr8, kNibbleMask, kBf16Base);
  const uint32_t a1 = and_or(wr >> 4, kNibbleMask, kBf16Base);
  const uint32_t a1r8 = and_or(wr8 >> 4, kNibbleMask, kBf16Base);
  const uint32_t a2 = and_or(wr >> 8, kNibbleMask, kBf16Base);
  const uint32_t a2r8 = and_or(wr8 >> 8, kNibbleMask, kBf16Base);
  const uint32_t a3 = and_or(wr >> 12, kNibbleMask, kBf16Base);
  const uint32_t a3r8 = and_or(wr8 >> 12, kNibbleMask, kBf16Base);
  mma_bf16_m16n8k16(d, a0, a0r8, a1, a1r8, hi[0], hi[1]);
  mma_bf16_m16n8k16(d, a2, a2r8, a3, a3r8, hi[2], hi[3]);
  if constexpr (kXF32) {
    mma_bf16_m16n8k16(d, a0, a0r8, a1, a1r8, lo[0], lo[1]);
    mma_bf16_m16n8k16(d, a2, a2r8, a3, a3r8, lo[2], lo[3]);
  }
}

template <int RT, bool kXF32>
__global__ void __launch_bounds__(kThreads) qmv_smallm_kernel(const QmvArgs a) {
  extern __shared__ __align__(128) uint8_t smem[];
  constexpr int kRows = 16 * RT;
  const int groups = a.K >> 6;
  const int n0 = blockIdx.x * kRows;
  const int rows = min(kRows, a.N - n0);
  const int n_chunks = (a.K + kStageInputs - 1) / kStageInputs;
  const int stages = a.stages;
  const Layout L = qmv_layout(kRows, groups, stages);
  uint8_t *wst = smem;
  uint16_t *s_sm = reinterpret_cast<uint16_t *>(smem + L.sb);
  uint16_t *b_sm = s_sm + kRows * groups;
  float *red = reinterpret_cast<float *>(smem + L.red);
  uint64_t *full = reinterpret_cast<uint64_t *>(smem + L.bar);
  uint64_t *empty = full + stages;
  uint64_t *sb_bar = empty + stages;

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  if (threadIdx.x == 0) {
    for (int i = 0; i < stages; ++i) {
      mbar_init(&full[i], 1);
      mbar_init(&empty[i], kConsumerWarps);
    }
    mbar_init(sb_bar, 32);
    fence_mbar_init();
  }
  __syncthreads();
  pdl_launch_dependents();

  if (warp == kConsumerWarps) {
    // ------------------------------ producer ------------------------------
    const uint32_t sb_bytes = (uint32_t)rows * groups * 2;
    if (sb_bytes % 16u == 0) {
      if (lane == 0) {
        mbar_arrive_expect_tx(sb_bar, 2 * sb_bytes);
        bulk_copy_g2s(s_sm, a.s + (size_t)n0 * groups, sb_bytes, sb_bar);
        bulk_copy_g2s(b_sm, a.b + (size_t)n0 * groups, sb_bytes, sb_bar);
      } else {
        mbar_arrive(sb_bar);
      }
    } else {  // ragged tile whose scale block is not a 16-byte multiple
      for (int i = lane; i < rows * groups; i += 32) {
        s_sm[i] = a.s[(size_t)n0 * groups + i];
        b_sm[i] = a.b[(size_t)n0 * groups + i];
      }
      mbar_arrive(sb_bar);
    }
    const uint64_t policy = l2_policy_evict_first();
    const size_t row_stride = (size_t)a.K / 2;
    const uint8_t *wbase = reinterpret_cast<const uint8_t *>(a.w) + (size_t)n0 * row_stride;
    int issued = 0;
    bool ok = true;
    for (int c = 0; c < n_chunks; ++c) {
      const int st = c % stages;
      if (c >= stages) {
        int got = 0;
        if (lane == 0) got = mbar_wait(&empty[st], ((c / stages) & 1) ^ 1) ? 1 : 0;
        got = __shfl_sync(0xffffffffu, got, 0);
        if (!got) {
          ok = false;
          break;
        }
      }
      const int k0 = c * kStageInputs;
      const uint32_t rb = (uint32_t)(min(kStageInputs, a.K - k0) / 2);
      if (lane == 0) mbar_arrive_expect_tx(&full[st], rb * (uint32_t)rows);
      __syncwarp();
      uint8_t *dst = wst + (size_t)st * kRows * kStageRowBytes;
      for (int r = lane; r < rows; r += 32)
        bulk_copy_g2s_hint(dst + r * kStageRowBytes, wbase + r * row_stride + k0 / 2, rb,
                           &full[st], policy);
      issued = c + 1;
    }
    if (!ok && lane == 0) {
      atomicOr(&g_qmv_device_error, 1u);
      // let the copies already issued land before the CTA may exit
      for (int c = max(0, issued - stages); c < issued; ++c)
        (void)mbar_wait(&full[c % stages], (c / stages) & 1);
    }
    return;
  }

  // ------------------------------ consumers -------------------------------
  const int r = lane >> 2, t = lane & 3;
  const int m = lane >> 2;  // activation row this lane feeds into B
  const bool m_valid = m < a.M;
  float acc[RT][4];
#pragma unroll
  for (int i = 0; i < RT; ++i) acc[i][0] = acc[i][1] = acc[i][2] = acc[i][3] = 0.f;
  // every lane waits (each needs the acquire); the outcome is made warp-uniform
  bool ok = __all_sync(0xffffffffu, mbar_wait(sb_bar, 0));
  pdl_wait();  // x (and y) belong to the preceding kernel until here
  for (int c = 0; ok && c < n_chunks; ++c) {
    const int st = c % stages;
    if (!__all_sync(0xffffffffu, mbar_wait(&full[st], (c / stages) & 1))) {
      ok = false;
      break;
    }
    const uint8_t *stage = wst + (size_t)st * kRows * kStageRowBytes;
#pragma unroll
    for (int gi = 0; gi < kGroupsPerWarp; ++gi) {
      const int gl = warp * kGroupsPerWarp + gi;
      const int g = c * (kConsumerWarps * kGroupsPerWarp) + gl;
      if (g < groups) {
        uint32_t hi[8], lo[8];
        load_b_fragments<kXF32>(a, m, m_valid, g, t, hi, lo);
        float xs[4] = {0.f, 0.f, 0.f, 0.f};  // sum of x over the group, cols 2t, 2t+1
#pragma unroll
        for (int s = 0; s < 4; ++s) {
          mma_bf16_m16n8k16(xs, kBf16One2, kBf16One2, kBf16One2, kBf16One2, hi[2 * s],
                            hi[2 * s + 1]);
          if constexpr (kXF32)
            mma_bf16_m16n8k16(xs, kBf16One2, kBf16One2, kBf16One2, kBf16One2, lo[2 * s],
                              lo[2 * s + 1]);
        }
#pragma unroll
        for (int rt = 0; rt < RT; ++rt) {
          const int row = rt * 16 + r;
          const uint8_t *rp = stage + row * kStageRowBytes + gl * 32 + t * 8;
          const uint2 w0 = *reinterpret_cast<const uint2 *>(rp);
          const uint2 w8 = *reinterpret_cast<const uint2 *>(rp + 8 * kStageRowBytes);
          float d[4] = {0.f, 0.f, 0.f, 0.f};
          mma_word<kXF32>(d, w0.x, w8.x, hi, lo);
          mma_word<kXF32>(d, w0.y, w8.y, hi + 4, lo + 4);
          const float s0 = bf16_bits_to_float(s_sm[row * groups + g]);
          const float s8 = bf16_bits_to_float(s_sm[(row + 8) * groups + g]);
          const float c0 = fmaf(-128.f, s0, bf16_bits_to_float(b_sm[row * groups + g]));
          const float c8 = fmaf(-128.f, s8, bf16_bits_to_float(b_sm[(row + 8) * groups + g]));
          acc[rt][0] = fmaf(s0, d[0], fmaf(c0, xs[0], acc[rt][0]));
          acc[rt][1] = fmaf(s0, d[1], fmaf(c0, xs[1], acc[rt][1]));
          acc[rt][2] = fmaf(s8, d[2], fmaf(c8, xs[0], acc[rt][2]));
          acc[rt][3] = fmaf(s8, d[3], fmaf(c8, xs[1], acc[rt][3]));
        }
      }
    }
    __syncwarp();
    if (lane == 0) mbar_arrive(&empty[st]);
  }
  if (!ok && lane == 0) atomicOr(&g_qmv_device_error, 2u);

  // cross-warp reduction in a fixed order: red[warp][row][col]
#pragma unroll
  for (int rt = 0; rt < RT; ++rt) {
    float *p = red + ((size_t)warp * kRows + rt * 16) * 8;
    p[r * 8 + 2 * t] = acc[rt][0];
    p[r * 8 + 2 * t + 1] = acc[rt][1];
    p[(r + 8) * 8 + 2 * t] = acc[rt][2];
    p[(r + 8) * 8 + 2 * t + 1] = acc[rt][3];
  }
  asm volatile("bar.sync 1, %0;" ::"r"(kConsumerWarps * 32) : "memory");
  if (!ok) return;
  for (int idx = threadIdx.x; idx < kRows * 8; idx += kConsumerWarps * 32) {
    const int col = idx / kRows, row = idx % kRows;  // row fastest: coalesced stores
    if (col < a.M && row < rows) {
      float v = 0.f;
#pragma unroll
      for (int w = 0; w < kConsumerWarps; ++w) v += red[((size_t)w * kRows + row) * 8 + col];
      a.y[(size_t)col * a.N + n0 + row] = v;
    }
  }
}

template <int RT, bool kXF32>
sv_status launch(const QmvArgs &args, int ctas, size_t smem, cudaStream_t stream) {
  static bool configured[64] = {};
  const int dev = current_device();
  auto kern = qmv_smallm_kernel<RT, kXF32>;
  if (dev >= 0 && dev < 64 && !configured[dev]) {
    int optin = 0;
    cudaDeviceGetAttribute(&optin, cudaDevAttrMaxSharedMemoryPerBlockOptin, dev);
    if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, optin) !=
        cudaSuccess)
      return fail(SV_ERR_CUDA, "qmv_smallm: cudaFuncSetAttribute failed");
    configured[dev] = true;
  }
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)ctas);
  cfg.blockDim = dim3(kThreads);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  if (pdl_enabled()) {
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
  }
  if (cudaLaunchKernelEx(&cfg, kern, args) != cudaSuccess) {
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
  if (M > 8) return fail(SV_ERR_UNSUPPORTED, "qmv_smallm: M=%d > 8", M);
  if (x_dtype != SV_F32 && x_dtype != SV_BF16)
    return fail(SV_ERR_INVALID_ARG, "qmv_smallm: unknown x_dtype %d", (int)x_dtype);
  if (M == 0 || N == 0) return SV_OK;
  if (!w_packed || !scales || !biases || !x || !y)
    return fail(SV_ERR_INVALID_ARG, "qmv_smallm: null pointer");
  if (!aligned(w_packed, 16) || !aligned(scales, 16) || !aligned(biases, 16) || !aligned(x, 16))
    return fail(SV_ERR_INVALID_ARG, "qmv_smallm: w_packed, scales, biases and x must be 16-byte aligned");
  if (!aligned(y, 4)) return fail(SV_ERR_INVALID_ARG, "qmv_smallm: y must be 4-byte aligned");
  if ((long long)N * (K / 8) > (1ll << 40))
    return fail(SV_ERR_INVALID_ARG, "qmv_smallm: N*K too large");
  const size_t wb = (size_t)N * K / 2, sbb = (size_t)N * (K / 64) * 2;
  const size_t xb = (size_t)M * K * (x_dtype == SV_F32 ? 4 : 2), yb = (size_t)M * N * 4;
  if (overlaps(y, yb, w_packed, wb) || overlaps(y, yb, scales, sbb) ||
      overlaps(y, yb, biases, sbb) || overlaps(y, yb, x, xb))
    return fail(SV_ERR_INVALID_ARG, "qmv_smallm: y overlaps an input");

  const int RT = N > 16 ? 2 : 1;
  const int rows_cta = 16 * RT;
  const int groups = K / 64;
  const int ctas = (N + rows_cta - 1) / rows_cta;
  const int n_chunks = (K + kStageInputs - 1) / kStageInputs;
  const int sms = device_sm_count();
  // co-resident CTAs wanted per SM so that one wave covers the grid
  const int per_sm = std::min(8, std::max(1, (ctas + sms - 1) / std::max(1, sms)));
  const size_t budget = (size_t)(220 * 1024) / per_sm;
  const Layout base = qmv_layout(rows_cta, groups, 0);
  const size_t stage_bytes = (size_t)rows_cta * kStageRowBytes + 16;
  int stages = budget > base.total ? (int)((budget - base.total) / stage_bytes) : 2;
  stages = std::max(2, std::min(stages, std::min(16, std::max(2, n_chunks))));
  Layout L = qmv_layout(rows_cta, groups, stages);
  int optin = 0;
  cudaDeviceGetAttribute(&optin, cudaDevAttrMaxSharedMemoryPerBlockOptin, current_device());
  while (L.total > (size_t)optin && stages > 2) L = qmv_layout(rows_cta, groups, --stages);
  if (L.total > (size_t)optin)
    return fail(SV_ERR_UNSUPPORTED, "qmv_smallm: K=%d needs %zu bytes of shared memory", K,
                L.total);

  QmvArgs args{w_packed, scales, biases, x, y, M, N, K, stages};
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  if (RT == 2)
    return x_dtype == SV_BF16 ? launch<2, false>(args, ctas, L.total, s)
                              : launch<2, true>(args, ctas, L.total, s);
  return x_dtype == SV_BF16 ? launch<1, false>(args, ctas, L.total, s)
                            : launch<1, true>(args, ctas, L.total, s);
}
