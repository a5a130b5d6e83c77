// fa_bwd_noalloc: the backward pass with its scratch memory in a static device array, for
// callers that must not allocate device memory themselves.
//
// Who needs this: code embedded in a host framework that owns every byte of device memory
// (a fixed, pre-planned pool in a serving engine or a plugin host) may not call cudaMalloc,
// and latency-critical callers cannot accept the implicit device synchronisation that
// cudaMalloc/cudaFree may cause. fa_bwd asks them for a workspace; this entry point does
// not. It runs the same kernels as fa_bwd, with the fp32 dQ accumulator (and D, when the
// caller passes none) placed in `g_bwd_scratch` below.
//
// The array lives in every GPU context that loads this library, from load until exit.
// Host code cannot use its name as a device address (it is a host-side stand-in), so the
// first call on each device looks the address up with cudaGetSymbolAddress while that
// device is current, and caches it for that device's context (a call in a new context,
// e.g. after cudaDeviceReset, looks it up again). All calls share the array: the dQ accumulator is
// cleared by every call before use, and calls that overlap on the GPU (other streams,
// other threads) race on it.
#include "fa_internal.h"

namespace fa {
namespace {

// dQ accumulator for up to FA_NOALLOC_MAX_ELEMS elements, then room for D (one float per
// row; rows <= elements / 64 because d >= 64).
constexpr size_t kAccFloats = FA_NOALLOC_MAX_ELEMS;
constexpr size_t kDFloats = FA_NOALLOC_MAX_ELEMS / 64;
constexpr size_t kScratchBytes = (kAccFloats + kDFloats) * sizeof(float);

static __device__ __align__(256) float g_bwd_scratch[kAccFloats + kDFloats];

// Device address of g_bwd_scratch on the current device (nullptr on failure), looked up
// once per device context: a new context (after cudaDeviceReset) places the array anew.
void* scratch_address() {
  static DeviceAddressCache cache;
  return symbol_address_cached(g_bwd_scratch, cache);
}

}  // namespace
}  // namespace fa

extern "C" fa_status_t fa_bwd_noalloc(const void* Q, const void* K, const void* V, const void* O,
                                      const void* dO, const float* LSE, const float* D, void* dQ,
                                      void* dK, void* dV, int B, int H, int N, int d, float scale,
                                      int causal, int dtype, void* stream) {
  const size_t need = fa_bwd_workspace_size(B, H, N, d, dtype);
  const bool plausible = B > 0 && H > 0 && N > 0 && d > 0 && (need > 0 || dtype == FA_DTYPE_FP32);
  if (!plausible)  // let fa_bwd report the precise argument error; it touches no device state
    return fa_bwd(Q, K, V, O, dO, LSE, D, dQ, dK, dV, nullptr, 0, B, H, N, d, scale, causal, dtype,
                  stream);
  const double elems = (double)B * H * N * d;
  if (elems > (double)FA_NOALLOC_MAX_ELEMS) return FA_ERR_WORKSPACE;
  const size_t need_d = D ? 0 : (size_t)B * H * N * sizeof(float);
  if (need > fa::kAccFloats * sizeof(float) || need + need_d > fa::kScratchBytes) return FA_ERR_WORKSPACE;
  void* scratch = fa::scratch_address();
  if (!scratch) return FA_ERR_CUDA;
  // fa_bwd places the accumulator at the start of the workspace and D right after it.
  return fa_bwd(Q, K, V, O, dO, LSE, D, dQ, dK, dV, scratch, fa::kScratchBytes, B, H, N, d, scale, causal,
                dtype, stream);
}
