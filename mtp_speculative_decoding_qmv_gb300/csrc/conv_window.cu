// conv_window.cu -- short causal convolution windows of a GatedDeltaNet layer:
// outputs over the verify tokens, and the commit of an accepted prefix, sm_103a.
//
// Source: "MTP와 DFlash" (mlxcel manual), section "Qwen3.8-Flash-Next
// (qwen4_exp) MTP" (the rollback replays the GatedDeltaNet recurrence and two
// convolution windows over the accepted tokens) and its batched DFlash
// paragraph (linear-attention layers replay the convolution and recurrent
// state over each row's accepted prefix).
//
// Depthwise causal convolution of width W over a channel stream; the state is
// the W-1 most recent inputs of each channel:
//   h(tau) = x[tau][c] (tau >= 0), window[W-1+tau][c] (-(W-1) <= tau < 0)
//   y[t][c] = sum_j weight[j][c] * h(t - (W-1) + j)
// Layouts are time-major (window [B][W-1][C], x, y [B][T][C], weight [W][C]),
// so one thread per (sequence, channel) keeps its window in registers and
// every access of a warp is 32 consecutive channels.  Both kernels move
// memory and do W multiply-adds per output: HBM-bound.
#include <cuda_runtime.h>

#include <cstdint>

#include "sv_device.cuh"
#include "sv_internal.h"

namespace sv {
namespace {

constexpr int kConvThreads = 256;
constexpr int kMaxW = 8;
constexpr int kMaxConvT = 64;

struct ConvArgs {
  const float *window;  // capture: read only
  float *state;         // replay: in/out
  const float *x, *weight;
  float *y;
  const int32_t *n_replay;
  int n_replay_count, n_replay_bias;
  int32_t *err_flags;
  int B, T, C, W;
};

template <int W>
__global__ void __launch_bounds__(kConvThreads) conv_capture_kernel(const ConvArgs a) {
  const int c = blockIdx.x * kConvThreads + threadIdx.x;
  const int b = blockIdx.y;
  pdl_launch_dependents();
  if (c >= a.C) return;
  float w[W], h[W];  // h[j] = h(t - (W-1) + j) for the current t
#pragma unroll
  for (int j = 0; j < W; ++j) w[j] = a.weight[(size_t)j * a.C + c];
  const float *win = a.window + (size_t)b * (W - 1) * a.C + c;
#pragma unroll
  for (int j = 0; j < W - 1; ++j) h[j + 1] = win[(size_t)j * a.C];
  const float *xb = a.x + (size_t)b * a.T * a.C + c;
  float *yb = a.y + (size_t)b * a.T * a.C + c;
  for (int t = 0; t < a.T; ++t) {
#pragma unroll
    for (int j = 0; j < W - 1; ++j) h[j] = h[j + 1];
    h[W - 1] = __ldcs(xb + (size_t)t * a.C);
    float s = 0.f;
#pragma unroll
    for (int j = 0; j < W; ++j) s = fmaf(w[j], h[j], s);
    __stcs(yb + (size_t)t * a.C, s);
  }
}

template <int W>
__global__ void __launch_bounds__(kConvThreads) conv_replay_kernel(const ConvArgs a) {
  const int c = blockIdx.x * kConvThreads + threadIdx.x;
  const int b = blockIdx.y;
  pdl_launch_dependents();
  int L = a.n_replay[b % a.n_replay_count] + a.n_replay_bias;
  const bool clamped = L < 0 || L > a.T;
  L = min(max(L, 0), a.T);
  if (clamped && a.err_flags && blockIdx.x == 0 && threadIdx.x == 0)
    atomicOr(&a.err_flags[b], SV_FLAG_REPLAY_RANGE);
  if (c >= a.C || L == 0) return;
  float *win = a.state + (size_t)b * (W - 1) * a.C + c;
  const float *xb = a.x + (size_t)b * a.T * a.C + c;
  float nw[W - 1];
#pragma unroll
  for (int i = 0; i < W - 1; ++i) {
    const int tau = L - (W - 1) + i;  // a verify input, or an entry of the old window
    nw[i] = tau >= 0 ? xb[(size_t)tau * a.C] : win[(size_t)(W - 1 + tau) * a.C];
  }
#pragma unroll
  for (int i = 0; i < W - 1; ++i) win[(size_t)i * a.C] = nw[i];
}

sv_status conv_validate(const char *who, int B, int T, int C, int W) {
  if (B < 0 || T < 1 || C < 1)
    return fail(SV_ERR_INVALID_ARG, "%s: need B >= 0, T >= 1, C >= 1 (B=%d T=%d C=%d)", who, B, T,
                C);
  if (W < 2 || W > kMaxW)
    return fail(SV_ERR_UNSUPPORTED, "%s: W=%d outside [2, %d]", who, W, kMaxW);
  if (T > kMaxConvT) return fail(SV_ERR_UNSUPPORTED, "%s: T=%d > %d", who, T, kMaxConvT);
  if (B > 65535) return fail(SV_ERR_UNSUPPORTED, "%s: B=%d > 65535", who, B);
  return SV_OK;
}

typedef void (*ConvKernel)(const ConvArgs);

template <int W>
ConvKernel conv_kernel(bool capture) {
  return capture ? conv_capture_kernel<W> : conv_replay_kernel<W>;
}

void conv_launch(bool capture, const ConvArgs &a, cudaStream_t s) {
  const dim3 grid((unsigned)((a.C + kConvThreads - 1) / kConvThreads), (unsigned)a.B);
  ConvKernel k;
  switch (a.W) {
    case 2: k = conv_kernel<2>(capture); break;
    case 3: k = conv_kernel<3>(capture); break;
    case 4: k = conv_kernel<4>(capture); break;
    case 5: k = conv_kernel<5>(capture); break;
    case 6: k = conv_kernel<6>(capture); break;
    case 7: k = conv_kernel<7>(capture); break;
    default: k = conv_kernel<8>(capture); break;
  }
  k<<<grid, kConvThreads, 0, s>>>(a);
}

}  // namespace
}  // namespace sv

using namespace sv;

extern "C" sv_status conv_window_capture(const float *window, const float *x, const float *weight,
                                         int B, int T, int C, int W, float *y,
                                         sv_stream_t stream) {
  clear_error();
  sv_status st = conv_validate("conv_window_capture", B, T, C, W);
  if (st != SV_OK) return st;
  if (B == 0) return SV_OK;
  if (!window || !x || !weight || !y)
    return fail(SV_ERR_INVALID_ARG, "conv_window_capture: null pointer");
  if (!aligned(window, 4) || !aligned(x, 4) || !aligned(weight, 4) || !aligned(y, 4))
    return fail(SV_ERR_INVALID_ARG, "conv_window_capture: misaligned pointer");
  const size_t wb = (size_t)B * (W - 1) * C * 4, xb = (size_t)B * T * C * 4,
               kb = (size_t)W * C * 4;
  if (overlaps(y, xb, window, wb) || overlaps(y, xb, x, xb) || overlaps(y, xb, weight, kb))
    return fail(SV_ERR_INVALID_ARG, "conv_window_capture: y overlaps an input");
  ConvArgs a = {};
  a.window = window;
  a.x = x;
  a.weight = weight;
  a.y = y;
  a.B = B;
  a.T = T;
  a.C = C;
  a.W = W;
  conv_launch(true, a, reinterpret_cast<cudaStream_t>(stream));
  return check_launch("conv_window_capture");
}

extern "C" sv_status conv_window_replay(float *window, const float *x, const int32_t *n_replay,
                                        int n_replay_count, int n_replay_bias, int B, int T, int C,
                                        int W, int32_t *err_flags, sv_stream_t stream) {
  clear_error();
  sv_status st = conv_validate("conv_window_replay", B, T, C, W);
  if (st != SV_OK) return st;
  if (B == 0) return SV_OK;
  if (!window || !x || !n_replay)
    return fail(SV_ERR_INVALID_ARG, "conv_window_replay: null pointer");
  if (n_replay_count < 1 || n_replay_count > B)
    return fail(SV_ERR_INVALID_ARG, "conv_window_replay: n_replay_count=%d outside [1, B=%d]",
                n_replay_count, B);
  if (!aligned(window, 4) || !aligned(x, 4) || !aligned(n_replay, 4) ||
      (err_flags && !aligned(err_flags, 4)))
    return fail(SV_ERR_INVALID_ARG, "conv_window_replay: misaligned pointer");
  const size_t wb = (size_t)B * (W - 1) * C * 4, xb = (size_t)B * T * C * 4;
  if (overlaps(window, wb, x, xb) || overlaps(window, wb, n_replay, (size_t)n_replay_count * 4) ||
      overlaps(err_flags, (size_t)B * 4, window, wb) || overlaps(err_flags, (size_t)B * 4, x, xb))
    return fail(SV_ERR_INVALID_ARG, "conv_window_replay: the window or flags overlap an input");
  ConvArgs a = {};
  a.state = window;
  a.x = x;
  a.n_replay = n_replay;
  a.n_replay_count = n_replay_count;
  a.n_replay_bias = n_replay_bias;
  a.err_flags = err_flags;
  a.B = B;
  a.T = T;
  a.C = C;
  a.W = W;
  conv_launch(false, a, reinterpret_cast<cudaStream_t>(stream));
  return check_launch("conv_window_replay");
}
