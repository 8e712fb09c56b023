// sv_api.cu -- library-wide entry points of libspecverify: ABI version, status
// strings, thread-local error messages, the PDL switch and the device status.
#include <cuda_runtime.h>

#include <atomic>
#include <cstdarg>
#include <cstdio>

#include "sv_internal.h"

namespace sv {
namespace {
thread_local char g_msg[512] = "";
std::atomic<int> g_pdl{0};
std::atomic<int> g_sm_count[64] = {};
}  // namespace

sv_status fail(sv_status st, const char *fmt, ...) {
  va_list ap;
  va_start(ap, fmt);
  std::vsnprintf(g_msg, sizeof g_msg, fmt, ap);
  va_end(ap);
  return st;
}

void clear_error() { g_msg[0] = '\0'; }

bool pdl_enabled() { return g_pdl.load(std::memory_order_relaxed) != 0; }

int current_device() {
  int d = 0;
  if (cudaGetDevice(&d) != cudaSuccess) return -1;
  return d;
}

int device_sm_count() {
  const int d = current_device();
  if (d < 0 || d >= 64) return 1;
  int n = g_sm_count[d].load(std::memory_order_relaxed);
  if (n == 0) {
    cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, d);
    if (n < 1) n = 1;
    g_sm_count[d].store(n, std::memory_order_relaxed);
  }
  return n;
}

sv_status check_launch(const char *what) {
  const cudaError_t e = cudaPeekAtLastError();
  if (e != cudaSuccess) return fail(SV_ERR_CUDA, "%s: %s", what, cudaGetErrorString(e));
  return SV_OK;
}

}  // namespace sv

extern "C" int sv_abi_version(void) { return SV_ABI_VERSION; }

extern "C" const char *sv_status_string(int status) {
  switch (status) {
    case SV_OK: return "ok";
    case SV_ERR_INVALID_ARG: return "invalid argument";
    case SV_ERR_UNSUPPORTED: return "unsupported";
    case SV_ERR_CUDA: return "CUDA error";
    case SV_ERR_DEVICE_FLAG: return "device-side bounded wait gave up";
    default: return "unknown status";
  }
}

extern "C" const char *sv_last_error(void) { return sv::g_msg; }

extern "C" void sv_set_pdl(int enable) { sv::g_pdl.store(enable ? 1 : 0); }

extern "C" int sv_get_pdl(void) { return sv::g_pdl.load(); }

extern "C" sv_status sv_device_status(void) {
  sv::clear_error();
  if (cudaDeviceSynchronize() != cudaSuccess)
    return sv::fail(SV_ERR_CUDA, "sv_device_status: %s", cudaGetErrorString(cudaGetLastError()));
  const unsigned q = sv::take_device_error_qmv();
  const unsigned a = sv::take_device_error_accept();
  const unsigned g = sv::take_device_error_gdn();
  const unsigned p = sv::take_device_error_plan();
  const unsigned w = sv::take_device_error_wide();
  if (q | a | g | p | w)
    return sv::fail(SV_ERR_DEVICE_FLAG,
                    "device error words: qmv=%u accept=%u gdn=%u plan=%u wide=%u", q, a, g, p, w);
  return SV_OK;
}
