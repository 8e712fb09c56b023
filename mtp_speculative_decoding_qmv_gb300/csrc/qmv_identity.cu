// qmv_identity.cu -- start-up probe: a verify block of M rows through
// qmv_smallm must give, bit for bit, what each row gives alone, sm_103a.
//
// Source: "MTP와 DFlash" (mlxcel manual), section "MTP 정확성 검사": when a
// worker starts, three independent synthetic inputs are pushed through a
// verify block and through the equivalent single-token steps, and block
// verification is used only if the two agree byte for byte; the verdict is
// kept per (model, block width).  Here the check covers the small-M
// projection (the step of the verify forward whose work depends on M): three
// synthetic activation blocks are generated on the device, each is
// multiplied as one M-row block and as M single rows, and the outputs are
// compared as bit patterns on the device.  Keeping the verdict per (weights,
// M) is the caller's part.
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include <cstdint>

#include "sv_device.cuh"
#include "sv_internal.h"

namespace sv {
namespace {

constexpr int kProbeSets = 3;
constexpr int kFillThreads = 256;
constexpr size_t kAlign = 256;

size_t round_up(size_t v) { return (v + kAlign - 1) / kAlign * kAlign; }

// MurmurHash3's 32-bit finaliser (Austin Appleby, public domain): a bijective
// mix of a counter, used only to make reproducible synthetic activations.
__device__ __forceinline__ uint32_t fmix32(uint32_t h) {
  h ^= h >> 16;
  h *= 0x85ebca6bu;
  h ^= h >> 13;
  h *= 0xc2b2ae35u;
  h ^= h >> 16;
  return h;
}

// x[i] = a value in [-2, 2) from the top 24 bits of the mixed index.
template <bool kF32>
__global__ void __launch_bounds__(kFillThreads) probe_fill_kernel(void *x, size_t n) {
  for (size_t i = (size_t)blockIdx.x * kFillThreads + threadIdx.x; i < n;
       i += (size_t)gridDim.x * kFillThreads) {
    const uint32_t h = fmix32((uint32_t)i * 0x9e3779b9u + 0x5bd1e995u);
    const float v = (float)(h >> 8) * (4.0f / 16777216.0f) - 2.0f;
    if (kF32)
      static_cast<float *>(x)[i] = v;
    else
      static_cast<uint16_t *>(x)[i] = __bfloat16_as_ushort(__float2bfloat16_rn(v));
  }
}

// *count += number of i with bits(a[i]) != bits(b[i]).
__global__ void __launch_bounds__(kFillThreads) probe_compare_kernel(const float *a,
                                                                     const float *b, size_t n,
                                                                     unsigned int *count) {
  unsigned int local = 0;
  for (size_t i = (size_t)blockIdx.x * kFillThreads + threadIdx.x; i < n;
       i += (size_t)gridDim.x * kFillThreads)
    local += __float_as_uint(a[i]) != __float_as_uint(b[i]) ? 1u : 0u;
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) local += __shfl_xor_sync(0xffffffffu, local, o);
  if ((threadIdx.x & 31) == 0 && local) atomicAdd(count, local);
}

struct ProbeLayout {
  size_t x, y_block, y_rows, count, total;
};

ProbeLayout probe_layout(int M, int N, int K, sv_dtype x_dtype) {
  ProbeLayout L;
  const size_t es = x_dtype == SV_F32 ? 4 : 2;
  L.x = 0;
  L.y_block = round_up((size_t)kProbeSets * M * K * es);
  L.y_rows = L.y_block + round_up((size_t)M * N * 4);
  L.count = L.y_rows + round_up((size_t)M * N * 4);
  L.total = L.count + kAlign;
  return L;
}

sv_status probe_validate(int M, int N, int K, sv_dtype x_dtype) {
  if (M < 1 || M > 16)
    return fail(SV_ERR_UNSUPPORTED, "qmv_identity_probe: M=%d outside [1, 16]", M);
  if (N < 1 || K < 64 || K % 64 != 0)
    return fail(SV_ERR_INVALID_ARG,
                "qmv_identity_probe: need N >= 1, K >= 64, K %% 64 == 0 (N=%d K=%d)", N, K);
  if (x_dtype != SV_F32 && x_dtype != SV_BF16)
    return fail(SV_ERR_INVALID_ARG, "qmv_identity_probe: unknown x_dtype %d", (int)x_dtype);
  if ((long long)N * K > (1ll << 40) || (long long)kProbeSets * M * K > (1ll << 40))
    return fail(SV_ERR_INVALID_ARG, "qmv_identity_probe: N*K too large");
  return SV_OK;
}

int probe_grid(size_t n) {
  const size_t want = (n + kFillThreads - 1) / kFillThreads;
  const size_t cap = (size_t)device_sm_count() * 8;
  return (int)(want < cap ? (want > 0 ? want : 1) : cap);
}

}  // namespace
}  // namespace sv

using namespace sv;

extern "C" size_t qmv_identity_probe_bytes(int M, int N, int K, sv_dtype x_dtype) {
  clear_error();
  if (probe_validate(M, N, K, x_dtype) != SV_OK) return 0;
  return probe_layout(M, N, K, x_dtype).total;
}

extern "C" sv_status qmv_identity_probe(const uint32_t *w_packed, const uint16_t *scales,
                                        const uint16_t *biases, sv_dtype x_dtype, int M, int N,
                                        int K, void *scratch, size_t scratch_bytes,
                                        int *mismatches, sv_stream_t stream) {
  clear_error();
  sv_status st = probe_validate(M, N, K, x_dtype);
  if (st != SV_OK) return st;
  if (!w_packed || !scales || !biases || !scratch || !mismatches)
    return fail(SV_ERR_INVALID_ARG, "qmv_identity_probe: null pointer");
  if (!aligned(scratch, kAlign))
    return fail(SV_ERR_INVALID_ARG, "qmv_identity_probe: scratch must be 256-byte aligned");
  const ProbeLayout L = probe_layout(M, N, K, x_dtype);
  if (scratch_bytes < L.total)
    return fail(SV_ERR_INVALID_ARG, "qmv_identity_probe: scratch of %zu bytes, need %zu",
                scratch_bytes, L.total);
  const size_t wb = (size_t)N * K / 2, sbb = (size_t)N * (K / 64) * 2;
  if (overlaps(scratch, L.total, w_packed, wb) || overlaps(scratch, L.total, scales, sbb) ||
      overlaps(scratch, L.total, biases, sbb))
    return fail(SV_ERR_INVALID_ARG, "qmv_identity_probe: scratch overlaps the weights");
  *mismatches = -1;

  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  unsigned char *base = static_cast<unsigned char *>(scratch);
  void *x = base + L.x;
  float *y_block = reinterpret_cast<float *>(base + L.y_block);
  float *y_rows = reinterpret_cast<float *>(base + L.y_rows);
  unsigned int *count = reinterpret_cast<unsigned int *>(base + L.count);
  const size_t es = x_dtype == SV_F32 ? 4 : 2;
  const size_t nx = (size_t)kProbeSets * M * K, ny = (size_t)M * N;

  if (cudaMemsetAsync(count, 0, sizeof(unsigned int), s) != cudaSuccess)
    return fail(SV_ERR_CUDA, "qmv_identity_probe: cudaMemsetAsync failed");
  if (x_dtype == SV_F32)
    probe_fill_kernel<true><<<probe_grid(nx), kFillThreads, 0, s>>>(x, nx);
  else
    probe_fill_kernel<false><<<probe_grid(nx), kFillThreads, 0, s>>>(x, nx);
  if ((st = check_launch("qmv_identity_probe (fill)")) != SV_OK) return st;

  for (int set = 0; set < kProbeSets; ++set) {
    const unsigned char *xs = static_cast<const unsigned char *>(x) + (size_t)set * M * K * es;
    st = qmv_smallm(w_packed, scales, biases, xs, x_dtype, y_block, M, N, K, 64, 4, stream);
    for (int m = 0; st == SV_OK && m < M; ++m)
      st = qmv_smallm(w_packed, scales, biases, xs + (size_t)m * K * es, x_dtype,
                      y_rows + (size_t)m * N, 1, N, K, 64, 4, stream);
    if (st != SV_OK) return st;
    probe_compare_kernel<<<probe_grid(ny), kFillThreads, 0, s>>>(y_block, y_rows, ny, count);
    if ((st = check_launch("qmv_identity_probe (compare)")) != SV_OK) return st;
  }
  unsigned int host_count = 0;
  if (cudaMemcpyAsync(&host_count, count, sizeof(host_count), cudaMemcpyDeviceToHost, s) !=
          cudaSuccess ||
      cudaStreamSynchronize(s) != cudaSuccess)
    return fail(SV_ERR_CUDA, "qmv_identity_probe: reading the mismatch count failed");
  *mismatches = (int)host_count;
  return SV_OK;
}
