// qmv_requant.cu -- a bf16 weight matrix requantised to the 4-bit affine
// group-64 layout of qmv_smallm (the draft-only LM head), sm_103a.
//
// Source: "MTPLX 2.24x faster TPS", section "Layer 0: MLX Runtime": the
// target keeps its LM head at model precision; a separate 4-bit LM head is
// built in memory and used by the drafter only, cutting draft time without
// touching the target's accuracy.  The pages do not print the quantiser; per
// group of 64 inputs of a row it is the min/max affine one:
//   lo = min w, hi = max w (zero extremes as +0),
//   s = rn_bf16((hi - lo) / 15), b = lo,
//   q = 0 if s == 0, else clamp(rint((w - b) / s), 0, 15),
// every step one IEEE fp32 operation (the code is an integer decided by
// floating point, so the steps are fixed, not left to the compiler).
//
// Eight lanes share a group (8 inputs, one packed word each), so a warp
// covers four consecutive groups of the flattened [N][K/64] group index: rows
// are contiguous, so it reads 512 contiguous bytes and writes 128 contiguous
// bytes of packed words.  HBM-bound: 2 bytes in, 0.5625 out per weight.
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include <algorithm>
#include <cstdint>

#include "sv_device.cuh"
#include "sv_internal.h"

namespace sv {
namespace {

constexpr int kReqThreads = 256;
constexpr int kGroupsPerWarp = 4;

__device__ __forceinline__ float bf16_lo(uint32_t w) { return __uint_as_float(w << 16); }
__device__ __forceinline__ float bf16_hi(uint32_t w) { return __uint_as_float(w & 0xFFFF0000u); }

__global__ void __launch_bounds__(kReqThreads)
    requant_kernel(const uint16_t *__restrict__ w, uint32_t *__restrict__ wp,
                   uint16_t *__restrict__ scales, uint16_t *__restrict__ biases,
                   long long n_groups) {
  pdl_launch_dependents();
  pdl_wait();  // the weights may be an earlier kernel's output
  const int lane = threadIdx.x & 31, sub = lane & 7;
  const long long warp0 = ((long long)blockIdx.x * kReqThreads + threadIdx.x) >> 5;
  const long long nwarps = ((long long)gridDim.x * kReqThreads) >> 5;
  for (long long gbase = warp0 * kGroupsPerWarp; gbase < n_groups;
       gbase += nwarps * kGroupsPerWarp) {
    const long long gi = gbase + (lane >> 3);
    const bool ok = gi < n_groups;
    uint4 v = make_uint4(0, 0, 0, 0);
    if (ok) v = __ldcs(reinterpret_cast<const uint4 *>(w + gi * 64) + sub);  // read once
    const float f[8] = {bf16_lo(v.x), bf16_hi(v.x), bf16_lo(v.y), bf16_hi(v.y),
                        bf16_lo(v.z), bf16_hi(v.z), bf16_lo(v.w), bf16_hi(v.w)};
    float lo = f[0], hi = f[0];
#pragma unroll
    for (int j = 1; j < 8; ++j) {
      lo = fminf(lo, f[j]);
      hi = fmaxf(hi, f[j]);
    }
#pragma unroll
    for (int o = 1; o < 8; o <<= 1) {  // within the group's eight lanes
      lo = fminf(lo, __shfl_xor_sync(0xffffffffu, lo, o));
      hi = fmaxf(hi, __shfl_xor_sync(0xffffffffu, hi, o));
    }
    if (lo == 0.0f) lo = 0.0f;  // zero extremes as +0
    if (hi == 0.0f) hi = 0.0f;
    const float step = __fdiv_rn(__fsub_rn(hi, lo), 15.0f);
    const uint16_t s_bits = __bfloat16_as_ushort(__float2bfloat16_rn(step));
    const float s = __uint_as_float((uint32_t)s_bits << 16);
    uint32_t packed = 0;
    if (s != 0.0f) {
#pragma unroll
      for (int j = 0; j < 8; ++j) {
        const float r = rintf(__fdiv_rn(__fsub_rn(f[j], lo), s));
        const uint32_t q = r < 0.0f ? 0u : (r > 15.0f ? 15u : (uint32_t)r);
        packed |= q << (4 * j);
      }
    }
    if (ok) {
      __stcs(wp + gi * 8 + sub, packed);
      if (sub == 0) {
        scales[gi] = s_bits;
        biases[gi] = (uint16_t)(__float_as_uint(lo) >> 16);  // lo is a bf16 value
      }
    }
  }
}

}  // namespace
}  // namespace sv

using namespace sv;

extern "C" sv_status qmv_requantize(const uint16_t *w_bf16, uint32_t *w_packed,
                                    uint16_t *scales, uint16_t *biases, int N, int K,
                                    sv_stream_t stream) {
  clear_error();
  if (N < 0 || K <= 0 || K % 64 != 0)
    return fail(SV_ERR_INVALID_ARG, "qmv_requantize: need N >= 0, K > 0, K %% 64 == 0 (N=%d K=%d)",
                N, K);
  if ((long long)N * K > (1ll << 40))
    return fail(SV_ERR_INVALID_ARG, "qmv_requantize: N*K too large");
  if (N == 0) return SV_OK;
  if (!w_bf16 || !w_packed || !scales || !biases)
    return fail(SV_ERR_INVALID_ARG, "qmv_requantize: null pointer");
  if (!aligned(w_bf16, 16) || !aligned(w_packed, 4) || !aligned(scales, 2) ||
      !aligned(biases, 2))
    return fail(SV_ERR_INVALID_ARG,
                "qmv_requantize: w_bf16 must be 16-byte, w_packed 4-byte, scales and biases "
                "2-byte aligned");
  const size_t wb = (size_t)N * K * 2, pb = (size_t)N * K / 2, sbb = (size_t)N * (K / 64) * 2;
  if (overlaps(w_bf16, wb, w_packed, pb) || overlaps(w_bf16, wb, scales, sbb) ||
      overlaps(w_bf16, wb, biases, sbb) || overlaps(w_packed, pb, scales, sbb) ||
      overlaps(w_packed, pb, biases, sbb) || overlaps(scales, sbb, biases, sbb))
    return fail(SV_ERR_INVALID_ARG, "qmv_requantize: buffers overlap");
  const long long n_groups = (long long)N * (K / 64);
  const long long warps = (n_groups + kGroupsPerWarp - 1) / kGroupsPerWarp;
  const long long want = (warps * 32 + kReqThreads - 1) / kReqThreads;
  const long long cap = (long long)device_sm_count() * 16;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)std::max(1ll, std::min(want, cap)));
  cfg.blockDim = dim3(kReqThreads);
  cfg.stream = reinterpret_cast<cudaStream_t>(stream);
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = pdl_enabled() ? 1 : 0;
  if (cudaLaunchKernelEx(&cfg, requant_kernel, w_bf16, w_packed, scales, biases, n_groups) !=
      cudaSuccess)
    return fail(SV_ERR_CUDA, "qmv_requantize: launch failed: %s",
                cudaGetErrorString(cudaGetLastError()));
  return check_launch("qmv_requantize");
}
