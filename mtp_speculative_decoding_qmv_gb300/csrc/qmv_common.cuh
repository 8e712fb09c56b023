// qmv_common.cuh -- device and host pieces shared by the two 4-bit small-M
// mat-vec kernels (one projection per launch, and a persistent launch over an
// ordered list of projections): tile geometry, the weight-stage layout, the
// tensor-map copy, and the per-group tensor-core math.
//
//   y[m, n] = sum_i x[m, i] * (s[n, i/64] * q[n, i] + b[n, i/64])
//
// Weights stream through shared memory in stages of 512 inputs x 64 rows
// (two 128-byte-swizzled boxes of 64 rows x 128 bytes) followed, when K is a
// multiple of 512, by the stage's scales [64][8] and biases [64][8] (bf16).
// Each of eight consumer warps reduces one 64-group of a stage for the four
// 16-row MMA tiles: nibbles are widened in registers to bf16 (128 + q,
// exact) and fed to mma.m16n8k16 as A with the (<= 8) activation rows as B;
// per group acc += s * D + (b - 128 s) * sum(x), sum(x) from an all-ones MMA.
#pragma once
#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include <cstdint>
#include <mutex>

#include "sv_device.cuh"
#include "sv_internal.h"

namespace sv {
namespace qmv {

constexpr int kRows = 64;                          // output rows per CTA (4 MMA tiles)
constexpr int kTiles = kRows / 16;
constexpr int kConsumerWarps = 8;                  // one 64-group each per stage
constexpr int kStageInputs = kConsumerWarps * 64;  // 512 inputs per stage
constexpr int kBoxWords = 32;                      // 128-byte box rows = 256 inputs
constexpr int kBoxesPerStage = kStageInputs / (kBoxWords * 8);  // 2
constexpr int kThreads = (kConsumerWarps + 1) * 32;
constexpr uint32_t kBf16One2 = 0x3F803F80u;        // bf16x2 (1, 1)
constexpr uint32_t kNibbleMask = 0x000F000Fu;
constexpr uint32_t kBf16Base = 0x43004300u;        // bf16x2 (128, 128)

// stage: [2 boxes][64 rows x 128 B] (swizzled) then, when streamed, scales
// [64][8] and biases [64][8] (bf16); 1024-byte multiple
constexpr uint32_t kSbOff = kBoxesPerStage * kRows * 128;
constexpr uint32_t kStageBytesStream = (kSbOff + 2 * kRows * 16 + 1023) / 1024 * 1024;
constexpr uint32_t kStageBytesBlock = (kSbOff + 1023) / 1024 * 1024;
constexpr uint32_t kRedBytes = kConsumerWarps * kRows * 8 * 4;  // cross-warp partials

__device__ __forceinline__ void tma_load_2d(uint32_t dst, const CUtensorMap *map, int x, int y,
                                            uint32_t bar, uint64_t policy) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cta.global.mbarrier::complete_tx::bytes.L2::cache_hint "
      "[%0], [%1, {%2, %3}], [%4], %5;" ::"r"(dst),
      "l"(map), "r"(x), "r"(y), "r"(bar), "l"(policy)
      : "memory");
}
__device__ __forceinline__ void ldmatrix_x4(uint32_t (&r)[4], uint32_t addr) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0,%1,%2,%3}, [%4];"
               : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3])
               : "r"(addr));
}
__device__ __forceinline__ uint32_t lds_u16(uint32_t addr) {
  uint16_t v;
  asm volatile("ld.shared.u16 %0, [%1];" : "=h"(v) : "r"(addr));
  return v;
}
// D = A * B with a zero accumulator (the first k16 step of a group).
__device__ __forceinline__ void mma_bf16_zero(float (&d)[4], uint32_t a0, uint32_t a1,
                                              uint32_t a2, uint32_t a3, uint32_t b0,
                                              uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, "
      "{%8,%9}, {%10,%10,%10,%10};"
      : "=f"(d[0]), "=f"(d[1]), "=f"(d[2]), "=f"(d[3])
      : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1), "f"(0.f));
}

// Warp-uniform wait for a stage: one test on the fast path, the bounded wait
// only when the data has not landed yet.  False after the wait limit.
__device__ __forceinline__ bool warp_wait_stage(uint32_t bar, uint32_t parity) {
  if (__all_sync(0xffffffffu, mbar_try_wait_u32(bar, parity))) return true;
  return __all_sync(0xffffffffu, mbar_wait_u32(bar, parity));
}

// Raw activation data of one 64-group for the lane's activation row m: the A
// operand (ldmatrix) gives lane (g = lane/4, t = lane%4) packed words t and
// 4+t of the group, i.e. inputs 8t + [0,8) and 32 + 8t + [0,8), so the lane
// loads those 16 inputs.
template <bool kXF32>
struct XRaw {
  uint4 v[kXF32 ? 4 : 2];
};

template <bool kXF32>
__device__ __forceinline__ XRaw<kXF32> load_x(const void *xrow, bool valid, int g, int t) {
  XRaw<kXF32> r;
#pragma unroll
  for (int i = 0; i < (kXF32 ? 4 : 2); ++i) r.v[i] = make_uint4(0, 0, 0, 0);
  if (valid) {
    if constexpr (!kXF32) {
      const uint16_t *p = static_cast<const uint16_t *>(xrow) + g * 64 + 8 * t;
      r.v[0] = *reinterpret_cast<const uint4 *>(p);
      r.v[1] = *reinterpret_cast<const uint4 *>(p + 32);
    } else {
      const float *p = static_cast<const float *>(xrow) + g * 64 + 8 * t;
      r.v[0] = *reinterpret_cast<const uint4 *>(p);
      r.v[1] = *reinterpret_cast<const uint4 *>(p + 4);
      r.v[2] = *reinterpret_cast<const uint4 *>(p + 32);
      r.v[3] = *reinterpret_cast<const uint4 *>(p + 36);
    }
  }
  return r;
}

// B fragments from the raw activations.  Each packed word feeds two k16 MMA
// steps whose k order pairs input j with input j+4 (the order the nibble
// widening produces), so B takes the same pairs.  fp32 rows become
// x = hi + lo with both parts bf16.
template <bool kXF32>
__device__ __forceinline__ void b_fragments(const XRaw<kXF32> &r, uint32_t (&hi)[8],
                                            uint32_t (&lo)[8]) {
  if constexpr (!kXF32) {
#pragma unroll
    for (int slot = 0; slot < 2; ++slot) {
      const uint4 v = r.v[slot];
      hi[4 * slot + 0] = prmt(v.x, v.z, 0x5410);  // (x0, x4)
      hi[4 * slot + 1] = prmt(v.x, v.z, 0x7632);  // (x1, x5)
      hi[4 * slot + 2] = prmt(v.y, v.w, 0x5410);  // (x2, x6)
      hi[4 * slot + 3] = prmt(v.y, v.w, 0x7632);  // (x3, x7)
    }
#pragma unroll
    for (int i = 0; i < 8; ++i) lo[i] = 0;
  } else {
#pragma unroll
    for (int slot = 0; slot < 2; ++slot) {
      const uint4 u0 = r.v[2 * slot], u1 = r.v[2 * slot + 1];
      const float v[8] = {__uint_as_float(u0.x), __uint_as_float(u0.y), __uint_as_float(u0.z),
                          __uint_as_float(u0.w), __uint_as_float(u1.x), __uint_as_float(u1.y),
                          __uint_as_float(u1.z), __uint_as_float(u1.w)};
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        const __nv_bfloat162 h = __floats2bfloat162_rn(v[j], v[j + 4]);
        const __nv_bfloat162 l =
            __floats2bfloat162_rn(v[j] - __low2float(h), v[j + 4] - __high2float(h));
        hi[4 * slot + j] = *reinterpret_cast<const uint32_t *>(&h);
        lo[4 * slot + j] = *reinterpret_cast<const uint32_t *>(&l);
      }
    }
  }
}

// One 64-group of one stage for the four 16-row tiles of a CTA:
//   acc[rt] += s * D + (b - 128 s) * sum(x)
// `wbase` is the lane's ldmatrix address in the stage for tile 0; the
// lane's scale of row g8 of tile rt is at sb + rt * sb_rt, of row g8+8 at
// + sb_r8, and the biases at + sb_b.
template <bool kXF32>
__device__ __forceinline__ void group_math(float (&acc)[kTiles][4], uint32_t wbase,
                                           const XRaw<kXF32> &xcur, uint32_t sb, uint32_t sb_rt,
                                           uint32_t sb_r8, uint32_t sb_b) {
  uint32_t hi[8], lo[8];
  b_fragments<kXF32>(xcur, hi, lo);
  // words t, 4+t of the group for rows g8 and g8+8 of each MMA tile
  uint32_t w[kTiles][4];
#pragma unroll
  for (int rt = 0; rt < kTiles; ++rt) ldmatrix_x4(w[rt], wbase + rt * 16 * 128);
  // four k16 steps; the tiles' accumulation chains are interleaved so that no
  // MMA waits on the one just issued
  float xs[4];  // sum of x over the group, columns 2t, 2t+1
  float d[kTiles][4];
#pragma unroll
  for (int ks = 0; ks < 4; ++ks) {
    const int wi = (ks >> 1) * 2;  // word t (ks 0,1) or 4+t (ks 2,3)
    const int sh = (ks & 1) * 8;   // nibbles j, j+4 for j = 0,1 or 2,3
    const uint32_t b0 = hi[2 * ks], b1 = hi[2 * ks + 1];
    if (ks == 0)
      mma_bf16_zero(xs, kBf16One2, kBf16One2, kBf16One2, kBf16One2, b0, b1);
    else
      mma_bf16_m16n8k16(xs, kBf16One2, kBf16One2, kBf16One2, kBf16One2, b0, b1);
    if constexpr (kXF32)
      mma_bf16_m16n8k16(xs, kBf16One2, kBf16One2, kBf16One2, kBf16One2, lo[2 * ks],
                        lo[2 * ks + 1]);
#pragma unroll
    for (int rt = 0; rt < kTiles; ++rt) {
      const uint32_t wr = w[rt][wi] >> sh, wr8 = w[rt][wi + 1] >> sh;
      const uint32_t p0 = and_or(wr, kNibbleMask, kBf16Base);
      const uint32_t p0r8 = and_or(wr8, kNibbleMask, kBf16Base);
      const uint32_t p1 = and_or(wr >> 4, kNibbleMask, kBf16Base);
      const uint32_t p1r8 = and_or(wr8 >> 4, kNibbleMask, kBf16Base);
      if (ks == 0)
        mma_bf16_zero(d[rt], p0, p0r8, p1, p1r8, b0, b1);
      else
        mma_bf16_m16n8k16(d[rt], p0, p0r8, p1, p1r8, b0, b1);
      if constexpr (kXF32)
        mma_bf16_m16n8k16(d[rt], p0, p0r8, p1, p1r8, lo[2 * ks], lo[2 * ks + 1]);
    }
  }
#pragma unroll
  for (int rt = 0; rt < kTiles; ++rt) {
    const uint32_t p = sb + rt * sb_rt;
    const float s0 = bf16_bits_to_float(lds_u16(p));
    const float s1 = bf16_bits_to_float(lds_u16(p + sb_r8));
    const float c0 = fmaf(-128.f, s0, bf16_bits_to_float(lds_u16(p + sb_b)));
    const float c1 = fmaf(-128.f, s1, bf16_bits_to_float(lds_u16(p + sb_b + sb_r8)));
    acc[rt][0] = fmaf(s0, d[rt][0], fmaf(c0, xs[0], acc[rt][0]));
    acc[rt][1] = fmaf(s0, d[rt][1], fmaf(c0, xs[1], acc[rt][1]));
    acc[rt][2] = fmaf(s1, d[rt][2], fmaf(c1, xs[0], acc[rt][2]));
    acc[rt][3] = fmaf(s1, d[rt][3], fmaf(c1, xs[1], acc[rt][3]));
  }
}

// Sixteen activation rows (M = 9..16): the same per-group math with two
// 8-column MMA n-tiles, rows 0-7 and 8-15.  Each widened weight fragment
// feeds both n-tiles, so the unpack is paid once per weight whatever M is.
template <bool kXF32>
__device__ __forceinline__ void group_math_x2(float (&acc)[2][kTiles][4], uint32_t wbase,
                                              const XRaw<kXF32> (&xcur)[2], uint32_t sb,
                                              uint32_t sb_rt, uint32_t sb_r8, uint32_t sb_b) {
  uint32_t hi[2][8], lo[2][8];
  b_fragments<kXF32>(xcur[0], hi[0], lo[0]);
  b_fragments<kXF32>(xcur[1], hi[1], lo[1]);
  uint32_t w[kTiles][4];
#pragma unroll
  for (int rt = 0; rt < kTiles; ++rt) ldmatrix_x4(w[rt], wbase + rt * 16 * 128);
  float xs[2][4];  // sum of x over the group per n-tile, columns 2t, 2t+1
  float d[2][kTiles][4];
#pragma unroll
  for (int ks = 0; ks < 4; ++ks) {
    const int wi = (ks >> 1) * 2;
    const int sh = (ks & 1) * 8;
#pragma unroll
    for (int nt = 0; nt < 2; ++nt) {
      if (ks == 0)
        mma_bf16_zero(xs[nt], kBf16One2, kBf16One2, kBf16One2, kBf16One2, hi[nt][2 * ks],
                      hi[nt][2 * ks + 1]);
      else
        mma_bf16_m16n8k16(xs[nt], kBf16One2, kBf16One2, kBf16One2, kBf16One2, hi[nt][2 * ks],
                          hi[nt][2 * ks + 1]);
      if constexpr (kXF32)
        mma_bf16_m16n8k16(xs[nt], kBf16One2, kBf16One2, kBf16One2, kBf16One2, lo[nt][2 * ks],
                          lo[nt][2 * ks + 1]);
    }
#pragma unroll
    for (int rt = 0; rt < kTiles; ++rt) {
      const uint32_t wr = w[rt][wi] >> sh, wr8 = w[rt][wi + 1] >> sh;
      const uint32_t p0 = and_or(wr, kNibbleMask, kBf16Base);
      const uint32_t p0r8 = and_or(wr8, kNibbleMask, kBf16Base);
      const uint32_t p1 = and_or(wr >> 4, kNibbleMask, kBf16Base);
      const uint32_t p1r8 = and_or(wr8 >> 4, kNibbleMask, kBf16Base);
#pragma unroll
      for (int nt = 0; nt < 2; ++nt) {
        if (ks == 0)
          mma_bf16_zero(d[nt][rt], p0, p0r8, p1, p1r8, hi[nt][2 * ks], hi[nt][2 * ks + 1]);
        else
          mma_bf16_m16n8k16(d[nt][rt], p0, p0r8, p1, p1r8, hi[nt][2 * ks], hi[nt][2 * ks + 1]);
        if constexpr (kXF32)
          mma_bf16_m16n8k16(d[nt][rt], p0, p0r8, p1, p1r8, lo[nt][2 * ks], lo[nt][2 * ks + 1]);
      }
    }
  }
#pragma unroll
  for (int rt = 0; rt < kTiles; ++rt) {
    const uint32_t p = sb + rt * sb_rt;
    const float s0 = bf16_bits_to_float(lds_u16(p));
    const float s1 = bf16_bits_to_float(lds_u16(p + sb_r8));
    const float c0 = fmaf(-128.f, s0, bf16_bits_to_float(lds_u16(p + sb_b)));
    const float c1 = fmaf(-128.f, s1, bf16_bits_to_float(lds_u16(p + sb_b + sb_r8)));
#pragma unroll
    for (int nt = 0; nt < 2; ++nt) {
      acc[nt][rt][0] = fmaf(s0, d[nt][rt][0], fmaf(c0, xs[nt][0], acc[nt][rt][0]));
      acc[nt][rt][1] = fmaf(s0, d[nt][rt][1], fmaf(c0, xs[nt][1], acc[nt][rt][1]));
      acc[nt][rt][2] = fmaf(s1, d[nt][rt][2], fmaf(c1, xs[nt][0], acc[nt][rt][2]));
      acc[nt][rt][3] = fmaf(s1, d[nt][rt][3], fmaf(c1, xs[nt][1], acc[nt][rt][3]));
    }
  }
}

// ldmatrix.x4 address offset of `lane` of the warp reducing group gl of a
// stage: lane L reads row ((L >> 3) & 1) * 8 + (L & 7) of an MMA tile, 16-byte
// chunk 2 * (gl % 4) + (L >> 4) of the 128-byte box row, at its swizzled
// position (chunk ^ row % 8).
__device__ __forceinline__ uint32_t ldmatrix_offset(int gl, int lane) {
  const int lrow = ((lane >> 3) & 1) * 8 + (lane & 7);
  const int lchunk = ((gl & 3) << 1) + (lane >> 4);
  return (uint32_t)((gl >> 2) * kRows * 128 + lrow * 128 + ((lchunk ^ (lrow & 7)) << 4));
}

// ---- host -------------------------------------------------------------------
// cuTensorMapEncodeTiled from the driver, found through the runtime (no link
// dependency on libcuda).
typedef CUresult (*EncodeTiledFn)(CUtensorMap *, CUtensorMapDataType, cuuint32_t, void *,
                                  const cuuint64_t *, const cuuint64_t *, const cuuint32_t *,
                                  const cuuint32_t *, CUtensorMapInterleave, CUtensorMapSwizzle,
                                  CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

inline EncodeTiledFn encode_tiled() {
  static EncodeTiledFn fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void *p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault,
                                         &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<EncodeTiledFn>(p);
  });
  return fn;
}

inline sv_status encode_2d(CUtensorMap *map, CUtensorMapDataType dtype, const void *ptr,
                    uint64_t inner, uint64_t rows, uint64_t row_bytes, uint32_t box_inner,
                    uint32_t box_rows, CUtensorMapSwizzle swizzle) {
  EncodeTiledFn enc = encode_tiled();
  if (!enc) return fail(SV_ERR_CUDA, "cuTensorMapEncodeTiled is unavailable");
  const cuuint64_t dims[2] = {(cuuint64_t)inner, (cuuint64_t)rows};
  const cuuint64_t strides[1] = {(cuuint64_t)row_bytes};
  const cuuint32_t box[2] = {box_inner, box_rows};
  const cuuint32_t estr[2] = {1, 1};
  const CUresult r = enc(map, dtype, 2, const_cast<void *>(ptr), dims, strides, box, estr,
                         CU_TENSOR_MAP_INTERLEAVE_NONE, swizzle,
                         CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  if (r != CUDA_SUCCESS)
    return fail(SV_ERR_CUDA, "tensor map encode failed (%d)", (int)r);
  return SV_OK;
}

}  // namespace qmv
}  // namespace sv
