// qmv_common.cuh -- device and host pieces shared by the two 4-bit small-M
// mat-vec kernels (one projection per launch, and a persistent launch over an
// ordered list of projections): tile geometry, the weight-stage layout, the
// tensor-map copy, and the per-group tensor-core math.
//
//   y[m, n] = sum_i x[m, i] * (s[n, i/64] * q[n, i] + b[n, i/64])
//
// Weights stream through shared memory in stages of 512 inputs x 64 rows
// followed, when K is a multiple of 512, by the stage's scales [64][8] and
// biases [64][8] (bf16), in one of two formats:
//  * packed: two 128-byte-swizzled boxes of 64 rows x 128 bytes; nibbles are
//    widened in registers with shifts and masks (bf16 128 + q, exact);
//  * byte-expanded (K % 128 == 0): four boxes written by the copy engine
//    with an 8-byte gap after every 8 data bytes, which ldmatrix widens to
//    one nibble per byte on the way to registers; one byte permute per two
//    weights then gives the bf16 operands.  Twice the shared memory per
//    streamed byte, about half the integer instructions.
// Each consumer warp reduces one 64-group of a stage for 16-row MMA tiles:
// the widened weights are A of mma.m16n8k16, the (<= 8) activation rows B;
// per group D = sum (128 + q) x, and acc += s * D + (b - 128 s) * sum(x)
// for packed stages; byte-expanded stages start D from -128 sum(x) (the
// first MMA's accumulator input) and take acc += s * D + b * sum(x).
// sum(x) comes from an all-ones MMA.
#pragma once
#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include <cstdint>
#include <mutex>
#include <type_traits>

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
// Fetches a tensor-map box into L2 only (no shared memory, no barrier).
__device__ __forceinline__ void tma_prefetch_2d(const CUtensorMap *map, int x, int y) {
  asm volatile("cp.async.bulk.prefetch.tensor.2d.L2.global.tile [%0, {%1, %2}];" ::"l"(map),
               "r"(x), "r"(y)
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

// D = A * B + C with C in other registers than D (no copies of C into D).
__device__ __forceinline__ void mma_bf16_c(float (&d)[4], uint32_t a0, uint32_t a1, uint32_t a2,
                                           uint32_t a3, uint32_t b0, uint32_t b1, float c0,
                                           float c1) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, "
      "{%8,%9}, {%10,%11,%10,%11};"
      : "=f"(d[0]), "=f"(d[1]), "=f"(d[2]), "=f"(d[3])
      : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1), "f"(c0), "f"(c1));
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

// ---- byte-expanded stages (K a multiple of 128) ------------------------------
// The copy engine writes each 128-input x 64-row box of packed nibbles with an
// 8-byte gap after every 8 data bytes (16U4_ALIGN16B, 128-byte swizzle:
// 64 rows x 128 bytes), and ldmatrix.b8x16.b4x16_p64 widens each nibble to
// the low four bits of a byte on the way to registers.  One byte permute with
// 0x43 high bytes then gives two bf16 operands 128 + q: no shifts, no masks.
// A stage is four such boxes (512 inputs) followed by the scales [64][8] and
// biases [64][8]; the copy engine counts only the data bytes (4 KB a box).
constexpr int kP64BoxInputs = 128;
constexpr uint32_t kP64BoxBytes = kRows * 128;              // 8 KB of shared memory
constexpr uint32_t kP64BoxTx = kRows * kP64BoxInputs / 2;   // 4 KB transferred
constexpr int kP64Boxes = kStageInputs / kP64BoxInputs;     // 4
constexpr uint32_t kP64SbOff = kP64Boxes * kP64BoxBytes;
constexpr uint32_t kStageBytesP64 = (kP64SbOff + 2 * kRows * 16 + 1023) / 1024 * 1024;
constexpr uint32_t kStageBytesP64Block = (kP64SbOff + 1023) / 1024 * 1024;
constexpr uint32_t kBf16HiBytes = 0x43434343u;              // 0x43: high byte of bf16 128
constexpr uint32_t kPrmtLo = 0x4140u;                       // bytes 0, 1 -> (128+e0, 128+e1)
constexpr uint32_t kPrmtHi = 0x4342u;                       // bytes 2, 3 -> (128+e2, 128+e3)

__device__ __forceinline__ void ldmatrix_p64_x4(uint32_t (&r)[4], uint32_t addr) {
  asm volatile("ldmatrix.sync.aligned.m8n16.x4.shared.b8x16.b4x16_p64 {%0,%1,%2,%3}, [%4];"
               : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3])
               : "r"(addr));
}

// ldmatrix address offsets of `lane` for group gl of a stage: k16 steps 0, 1
// (first) and 2, 3 (second) of row tile 0; tile rt adds rt * 16 * 128.
// Lane L gives the row (L & 7) + 8 ((L >> 3) & 1) of 16-input chunk
// 4 (gl & 1) + step + (L >> 4) of box gl / 2, at its swizzled position.
__device__ __forceinline__ void ldmatrix_p64_offsets(int gl, int lane, uint32_t &first,
                                                     uint32_t &second) {
  const int row = (lane & 7) + 8 * ((lane >> 3) & 1);
  const int chunk = 4 * (gl & 1) + (lane >> 4);
  const uint32_t base = (uint32_t)(gl >> 1) * kP64BoxBytes + (uint32_t)row * 128;
  first = base + ((uint32_t)(chunk ^ (row & 7)) << 4);
  second = base + ((uint32_t)((chunk + 2) ^ (row & 7)) << 4);
}

// Activations of one 64-group for the lane's activation row: the byte
// expansion gives lane (g, t) inputs 16 s + 4 t + [0, 4) of k16 step s, so the
// lane loads four 4-input pieces (8 bytes each in bf16, 16 in fp32).
template <bool kXF32>
struct XRawP {
  typename std::conditional<kXF32, uint4, uint2>::type v[4];
};

template <bool kXF32>
__device__ __forceinline__ XRawP<kXF32> load_x_p64(const void *xrow, bool valid, int g, int t) {
  XRawP<kXF32> r;
  if constexpr (!kXF32) {
    const uint2 *p = reinterpret_cast<const uint2 *>(static_cast<const uint16_t *>(xrow) + g * 64 + 4 * t);
#pragma unroll
    for (int s = 0; s < 4; ++s) r.v[s] = valid ? p[4 * s] : make_uint2(0, 0);
  } else {
    const uint4 *p = reinterpret_cast<const uint4 *>(static_cast<const float *>(xrow) + g * 64 + 4 * t);
#pragma unroll
    for (int s = 0; s < 4; ++s) r.v[s] = valid ? p[4 * s] : make_uint4(0, 0, 0, 0);
  }
  return r;
}
// Same, read at L2 (activations written by other CTAs of the same launch).
template <bool kXF32>
__device__ __forceinline__ XRawP<kXF32> load_x_p64_l2(const void *xrow, bool valid, int g, int t) {
  XRawP<kXF32> r;
  if constexpr (!kXF32) {
    const uint2 *p = reinterpret_cast<const uint2 *>(static_cast<const uint16_t *>(xrow) + g * 64 + 4 * t);
#pragma unroll
    for (int s = 0; s < 4; ++s) r.v[s] = valid ? __ldcg(p + 4 * s) : make_uint2(0, 0);
  } else {
    const uint4 *p = reinterpret_cast<const uint4 *>(static_cast<const float *>(xrow) + g * 64 + 4 * t);
#pragma unroll
    for (int s = 0; s < 4; ++s) r.v[s] = valid ? __ldcg(p + 4 * s) : make_uint4(0, 0, 0, 0);
  }
  return r;
}

// B fragments of the four k16 steps: step s, register 0 holds inputs
// (4t, 4t+1), register 1 (4t+2, 4t+3) of the step's 16 -- the pairs the byte
// permutes produce.  fp32 rows become x = hi + lo, both bf16.
template <bool kXF32>
__device__ __forceinline__ void b_fragments_p64(const XRawP<kXF32> &r, uint32_t (&hi)[4][2],
                                                uint32_t (&lo)[4][2]) {
#pragma unroll
  for (int s = 0; s < 4; ++s) {
    if constexpr (!kXF32) {
      hi[s][0] = r.v[s].x;
      hi[s][1] = r.v[s].y;
      lo[s][0] = lo[s][1] = 0;
    } else {
      const float v[4] = {__uint_as_float(r.v[s].x), __uint_as_float(r.v[s].y),
                          __uint_as_float(r.v[s].z), __uint_as_float(r.v[s].w)};
#pragma unroll
      for (int j = 0; j < 2; ++j) {
        const __nv_bfloat162 h = __floats2bfloat162_rn(v[2 * j], v[2 * j + 1]);
        const __nv_bfloat162 l =
            __floats2bfloat162_rn(v[2 * j] - __low2float(h), v[2 * j + 1] - __high2float(h));
        hi[s][j] = *reinterpret_cast<const uint32_t *>(&h);
        lo[s][j] = *reinterpret_cast<const uint32_t *>(&l);
      }
    }
  }
}

// Sum of the group's activations, columns 2t, 2t+1 (all-ones A operand).
template <bool kXF32>
__device__ __forceinline__ void group_xsum(float (&xs)[4], const uint32_t (&hi)[4][2],
                                           const uint32_t (&lo)[4][2]) {
  mma_bf16_zero(xs, kBf16One2, kBf16One2, kBf16One2, kBf16One2, hi[0][0], hi[0][1]);
  if constexpr (kXF32)
    mma_bf16_m16n8k16(xs, kBf16One2, kBf16One2, kBf16One2, kBf16One2, lo[0][0], lo[0][1]);
#pragma unroll
  for (int s = 1; s < 4; ++s) {
    mma_bf16_m16n8k16(xs, kBf16One2, kBf16One2, kBf16One2, kBf16One2, hi[s][0], hi[s][1]);
    if constexpr (kXF32)
      mma_bf16_m16n8k16(xs, kBf16One2, kBf16One2, kBf16One2, kBf16One2, lo[s][0], lo[s][1]);
  }
}

// One 64-group of a byte-expanded stage for the four 16-row tiles of a CTA:
//   D = -128 sum(x) + sum_k (128 + q) x    (the offset enters as the first
//                                           MMA's accumulator)
//   acc[rt] += s * D + b * sum(x)
// `w0` / `w2` are the lane's ldmatrix addresses of steps 0-1 / 2-3 for tile
// 0; the lane's scale of row g8 of tile rt is at sb + rt * sb_rt, of row
// g8 + 8 at + sb_r8, and the biases at + sb_b.
template <bool kXF32, bool kPrepared, int kT>
__device__ __forceinline__ void group_math_p64_impl(float (&acc)[kT][4], uint32_t w0,
                                                    uint32_t w2, const XRawP<kXF32> &xcur,
                                                    uint32_t sb, uint32_t sb_rt, uint32_t sb_r8,
                                                    uint32_t sb_b) {
  uint32_t hi[4][2], lo[4][2];
  b_fragments_p64<kXF32>(xcur, hi, lo);
  float xs[4];
  group_xsum<kXF32>(xs, hi, lo);
  const float c0 = -128.f * xs[0], c1 = -128.f * xs[1];
  float d[kT][4];
#pragma unroll
  for (int half = 0; half < 2; ++half) {
    uint32_t w[kT][4];
#pragma unroll
    for (int rt = 0; rt < kT; ++rt) ldmatrix_p64_x4(w[rt], (half ? w2 : w0) + rt * 16 * 128);
    // steps 2 half and 2 half + 1; the tiles' chains are interleaved so no MMA
    // waits on the one just issued
#pragma unroll
    for (int k = 0; k < 2; ++k) {
      const int s = 2 * half + k;
#pragma unroll
      for (int rt = 0; rt < kT; ++rt) {
        const uint32_t r0 = w[rt][2 * k], r8 = w[rt][2 * k + 1];  // rows g8, g8 + 8
        const uint32_t a0 = prmt(r0, kBf16HiBytes, kPrmtLo), a1 = prmt(r8, kBf16HiBytes, kPrmtLo);
        const uint32_t a2 = prmt(r0, kBf16HiBytes, kPrmtHi), a3 = prmt(r8, kBf16HiBytes, kPrmtHi);
        if (s == 0)  // the -128 sum(x) offset enters as the chain's accumulator
          mma_bf16_c(d[rt], a0, a1, a2, a3, hi[0][0], hi[0][1], c0, c1);
        else
          mma_bf16_m16n8k16(d[rt], a0, a1, a2, a3, hi[s][0], hi[s][1]);
        if constexpr (kXF32) mma_bf16_m16n8k16(d[rt], a0, a1, a2, a3, lo[s][0], lo[s][1]);
      }
    }
  }
#pragma unroll
  for (int rt = 0; rt < kT; ++rt) {
    float s0, s1, b0, b1;
    if constexpr (kPrepared) {
      // fp32 (s, s+8, b, b+8) of this lane's rows, 16 bytes at sb + rt * sb_rt
      float4 v;
      asm volatile("ld.shared.v4.f32 {%0,%1,%2,%3}, [%4];"
                   : "=f"(v.x), "=f"(v.y), "=f"(v.z), "=f"(v.w)
                   : "r"(sb + rt * sb_rt));
      s0 = v.x;
      s1 = v.y;
      b0 = v.z;
      b1 = v.w;
    } else {
      const uint32_t p = sb + rt * sb_rt;
      s0 = bf16_bits_to_float(lds_u16(p));
      s1 = bf16_bits_to_float(lds_u16(p + sb_r8));
      b0 = bf16_bits_to_float(lds_u16(p + sb_b));
      b1 = bf16_bits_to_float(lds_u16(p + sb_b + sb_r8));
    }
    acc[rt][0] = fmaf(s0, d[rt][0], fmaf(b0, xs[0], acc[rt][0]));
    acc[rt][1] = fmaf(s0, d[rt][1], fmaf(b0, xs[1], acc[rt][1]));
    acc[rt][2] = fmaf(s1, d[rt][2], fmaf(b1, xs[0], acc[rt][2]));
    acc[rt][3] = fmaf(s1, d[rt][3], fmaf(b1, xs[1], acc[rt][3]));
  }
}
// bf16 scales and biases straight from the stage
template <bool kXF32>
__device__ __forceinline__ void group_math_p64(float (&acc)[kTiles][4], uint32_t w0, uint32_t w2,
                                               const XRawP<kXF32> &xcur, uint32_t sb,
                                               uint32_t sb_rt, uint32_t sb_r8, uint32_t sb_b) {
  group_math_p64_impl<kXF32, false, kTiles>(acc, w0, w2, xcur, sb, sb_rt, sb_r8, sb_b);
}
// fp32 scales and biases prepared per stage (see prepare_sb_p64): the lane's
// four values of tile rt as one 16-byte record at sb + rt * sb_rt
template <bool kXF32, int kT>
__device__ __forceinline__ void group_math_p64_prep(float (&acc)[kT][4], uint32_t w0,
                                                    uint32_t w2, const XRawP<kXF32> &xcur,
                                                    uint32_t sb, uint32_t sb_rt) {
  group_math_p64_impl<kXF32, true, kT>(acc, w0, w2, xcur, sb, sb_rt, 0, 0);
}

// A warp's share of one byte-expanded stage held in registers: the widened
// weight fragments of kT 16-row tiles (k16 steps 0-1 and 2-3) and their
// prepared fp32 (s, s+8, b, b+8) records.  Loading it is all a consumer does
// with the stage's shared memory, so the ring slot can be released before
// the math.
template <int kT>
struct StageRegs {
  uint32_t w[kT][2][4];
  float4 sb[kT];
};

template <int kT>
__device__ __forceinline__ void load_stage_regs(StageRegs<kT> &r, uint32_t w0, uint32_t w2,
                                                uint32_t sb, uint32_t sb_rt) {
#pragma unroll
  for (int rt = 0; rt < kT; ++rt) {
    ldmatrix_p64_x4(r.w[rt][0], w0 + rt * 16 * 128);
    ldmatrix_p64_x4(r.w[rt][1], w2 + rt * 16 * 128);
    asm volatile("ld.shared.v4.f32 {%0,%1,%2,%3}, [%4];"
                 : "=f"(r.sb[rt].x), "=f"(r.sb[rt].y), "=f"(r.sb[rt].z), "=f"(r.sb[rt].w)
                 : "r"(sb + rt * sb_rt));
  }
}

// The group math of group_math_p64 on a stage held in registers.
template <bool kXF32, int kT>
__device__ __forceinline__ void group_math_regs(float (&acc)[kT][4], const StageRegs<kT> &r,
                                                const XRawP<kXF32> &xcur) {
  uint32_t hi[4][2], lo[4][2];
  b_fragments_p64<kXF32>(xcur, hi, lo);
  float xs[4];
  group_xsum<kXF32>(xs, hi, lo);
  const float c0 = -128.f * xs[0], c1 = -128.f * xs[1];
  float d[kT][4];
#pragma unroll
  for (int s = 0; s < 4; ++s) {
#pragma unroll
    for (int rt = 0; rt < kT; ++rt) {
      const uint32_t r0 = r.w[rt][s >> 1][2 * (s & 1)], r8 = r.w[rt][s >> 1][2 * (s & 1) + 1];
      const uint32_t a0 = prmt(r0, kBf16HiBytes, kPrmtLo), a1 = prmt(r8, kBf16HiBytes, kPrmtLo);
      const uint32_t a2 = prmt(r0, kBf16HiBytes, kPrmtHi), a3 = prmt(r8, kBf16HiBytes, kPrmtHi);
      if (s == 0)
        mma_bf16_c(d[rt], a0, a1, a2, a3, hi[0][0], hi[0][1], c0, c1);
      else
        mma_bf16_m16n8k16(d[rt], a0, a1, a2, a3, hi[s][0], hi[s][1]);
      if constexpr (kXF32) mma_bf16_m16n8k16(d[rt], a0, a1, a2, a3, lo[s][0], lo[s][1]);
    }
  }
#pragma unroll
  for (int rt = 0; rt < kT; ++rt) {
    const float4 v = r.sb[rt];
    acc[rt][0] = fmaf(v.x, d[rt][0], fmaf(v.z, xs[0], acc[rt][0]));
    acc[rt][1] = fmaf(v.x, d[rt][1], fmaf(v.z, xs[1], acc[rt][1]));
    acc[rt][2] = fmaf(v.y, d[rt][2], fmaf(v.w, xs[0], acc[rt][2]));
    acc[rt][3] = fmaf(v.y, d[rt][3], fmaf(v.w, xs[1], acc[rt][3]));
  }
}

// The scales [64][8] and biases [64][8] (bf16) of one stage at `raw` written
// as fp32 records (s[r][g], s[r+8][g], b[r][g], b[r+8][g]), r = 16 rt + g8, at
// `out` + 16 ((g * 4 + rt) * 8 + g8): the layout group_math_p64_prep reads
// (a warp's eight lanes of one record index read 128 contiguous bytes).  One
// warp; lane = (rt, g8) handles rows r and r + 8 of every group.
__device__ __forceinline__ void prepare_sb_p64(uint32_t raw, uint32_t out, int lane) {
  const int rt = lane >> 3, g8 = lane & 7, r = 16 * rt + g8;
  uint4 s0, s1, b0, b1;
  asm volatile("ld.shared.v4.u32 {%0,%1,%2,%3}, [%4];"
               : "=r"(s0.x), "=r"(s0.y), "=r"(s0.z), "=r"(s0.w) : "r"(raw + r * 16));
  asm volatile("ld.shared.v4.u32 {%0,%1,%2,%3}, [%4];"
               : "=r"(s1.x), "=r"(s1.y), "=r"(s1.z), "=r"(s1.w) : "r"(raw + (r + 8) * 16));
  asm volatile("ld.shared.v4.u32 {%0,%1,%2,%3}, [%4];"
               : "=r"(b0.x), "=r"(b0.y), "=r"(b0.z), "=r"(b0.w) : "r"(raw + kRows * 16 + r * 16));
  asm volatile("ld.shared.v4.u32 {%0,%1,%2,%3}, [%4];"
               : "=r"(b1.x), "=r"(b1.y), "=r"(b1.z), "=r"(b1.w)
               : "r"(raw + kRows * 16 + (r + 8) * 16));
  const uint32_t sw0[4] = {s0.x, s0.y, s0.z, s0.w}, sw1[4] = {s1.x, s1.y, s1.z, s1.w};
  const uint32_t bw0[4] = {b0.x, b0.y, b0.z, b0.w}, bw1[4] = {b1.x, b1.y, b1.z, b1.w};
#pragma unroll
  for (int g = 0; g < 8; ++g) {
    // group g is the low (even g) or high (odd g) half of word g / 2
    const int wi = g >> 1;
    auto f = [&](uint32_t w) { return __uint_as_float((g & 1) ? (w & 0xFFFF0000u) : (w << 16)); };
    asm volatile("st.shared.v4.f32 [%0], {%1,%2,%3,%4};" ::"r"(out + 16u * ((g * 4 + rt) * 8 + g8)),
                 "f"(f(sw0[wi])), "f"(f(sw1[wi])), "f"(f(bw0[wi])), "f"(f(bw1[wi]))
                 : "memory");
  }
}

// Sixteen activation rows: the same math with two 8-column n-tiles sharing
// every widened weight fragment.
template <bool kXF32>
__device__ __forceinline__ void group_math_p64_x2(float (&acc)[2][kTiles][4], uint32_t w0,
                                                  uint32_t w2, const XRawP<kXF32> (&xcur)[2],
                                                  uint32_t sb, uint32_t sb_rt, uint32_t sb_r8,
                                                  uint32_t sb_b) {
  uint32_t hi[2][4][2], lo[2][4][2];
  float xs[2][4];
#pragma unroll
  for (int nt = 0; nt < 2; ++nt) {
    b_fragments_p64<kXF32>(xcur[nt], hi[nt], lo[nt]);
    group_xsum<kXF32>(xs[nt], hi[nt], lo[nt]);
  }
  float d[2][kTiles][4];
#pragma unroll
  for (int nt = 0; nt < 2; ++nt) {
    const float c0 = -128.f * xs[nt][0], c1 = -128.f * xs[nt][1];
#pragma unroll
    for (int rt = 0; rt < kTiles; ++rt) {
      d[nt][rt][0] = c0;
      d[nt][rt][1] = c1;
      d[nt][rt][2] = c0;
      d[nt][rt][3] = c1;
    }
  }
#pragma unroll
  for (int half = 0; half < 2; ++half) {
    uint32_t w[kTiles][4];
#pragma unroll
    for (int rt = 0; rt < kTiles; ++rt) ldmatrix_p64_x4(w[rt], (half ? w2 : w0) + rt * 16 * 128);
#pragma unroll
    for (int k = 0; k < 2; ++k) {
      const int s = 2 * half + k;
#pragma unroll
      for (int rt = 0; rt < kTiles; ++rt) {
        const uint32_t r0 = w[rt][2 * k], r8 = w[rt][2 * k + 1];
        const uint32_t a0 = prmt(r0, kBf16HiBytes, kPrmtLo), a1 = prmt(r8, kBf16HiBytes, kPrmtLo);
        const uint32_t a2 = prmt(r0, kBf16HiBytes, kPrmtHi), a3 = prmt(r8, kBf16HiBytes, kPrmtHi);
#pragma unroll
        for (int nt = 0; nt < 2; ++nt) {
          mma_bf16_m16n8k16(d[nt][rt], a0, a1, a2, a3, hi[nt][s][0], hi[nt][s][1]);
          if constexpr (kXF32)
            mma_bf16_m16n8k16(d[nt][rt], a0, a1, a2, a3, lo[nt][s][0], lo[nt][s][1]);
        }
      }
    }
  }
#pragma unroll
  for (int rt = 0; rt < kTiles; ++rt) {
    const uint32_t p = sb + rt * sb_rt;
    const float s0 = bf16_bits_to_float(lds_u16(p));
    const float s1 = bf16_bits_to_float(lds_u16(p + sb_r8));
    const float b0 = bf16_bits_to_float(lds_u16(p + sb_b));
    const float b1 = bf16_bits_to_float(lds_u16(p + sb_b + sb_r8));
#pragma unroll
    for (int nt = 0; nt < 2; ++nt) {
      acc[nt][rt][0] = fmaf(s0, d[nt][rt][0], fmaf(b0, xs[nt][0], acc[nt][rt][0]));
      acc[nt][rt][1] = fmaf(s0, d[nt][rt][1], fmaf(b0, xs[nt][1], acc[nt][rt][1]));
      acc[nt][rt][2] = fmaf(s1, d[nt][rt][2], fmaf(b1, xs[nt][0], acc[nt][rt][2]));
      acc[nt][rt][3] = fmaf(s1, d[nt][rt][3], fmaf(b1, xs[nt][1], acc[nt][rt][3]));
    }
  }
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
