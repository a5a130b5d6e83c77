// The backward entry functions of the tensor-core path; what they compute is fa_bwd /
// fa_bwd_masked / fa_bwd_bitmask / fa_bwd_dropout in include/fa.h.
//
// dQ is a sum over key tiles, and the 128-key-tile kernel (fa_bwd_wide.cu) gives every key
// tile its own CTA. It computes dQ in one of two ways ("FlashAttention 反向传播" 踩坑二 weighs
// them; both keep fp32 sums and cast to bf16 once, as its 踩坑三 asks):
//   atomic:   each CTA adds its fp32 dQ partials into an accumulator in the workspace; the
//             entry function zeroes it first and one pass here scales it by `scale` and
//             rounds it to bf16 (the masked and dropout instances always take this way);
//   separate: the 128-key-tile kernel gives dK and dV only, and a second kernel over
//             128-query tiles (fa_bwd_dq.cu) recomputes S and dP and accumulates dQ in TMEM.
// fa_set_bwd_dq_mode picks one; by default the atomic way runs (see separate_dq below).
#include <atomic>

#include <cuda_bf16.h>

#include "fa_internal.h"
#include "sm100_ptx.cuh"

namespace fa {
namespace {

using namespace ptx;

// dQ = bf16(scale * dQacc), 8 elements per thread.
__global__ void __launch_bounds__(256) dq_convert_kernel(const float* __restrict__ acc,
                                                        __nv_bfloat16* __restrict__ dq, int64_t n8,
                                                        float scale) {
  const int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
  if (i >= n8) return;
  const float4 a = reinterpret_cast<const float4*>(acc)[2 * i];
  const float4 b = reinterpret_cast<const float4*>(acc)[2 * i + 1];
  uint4 w;
  w.x = pack_bf16(a.x * scale, a.y * scale);
  w.y = pack_bf16(a.z * scale, a.w * scale);
  w.z = pack_bf16(b.x * scale, b.y * scale);
  w.w = pack_bf16(b.z * scale, b.w * scale);
  reinterpret_cast<uint4*>(dq)[i] = w;
}

std::atomic<int> g_dq_mode{FA_BWD_DQ_AUTO};

// The dQ mode for a plain backward. FA_BWD_DQ_AUTO takes the atomic way at every shape: on
// GB300 (preprocess + backward, both modes in one process) the separate pass measured 1.565
// against 1.280 ms at B2 H16 N8192 d128 causal, 0.973 against 0.837 ms at B16 H32 N1024
// d128, 0.346 against 0.270 ms at B4 H16 N2048 d64, 5.800 against 4.697 ms at B1 H8 N32768
// d128 causal and 0.203 against 0.165 ms at B4 H16 N2048 d64 causal. Dropping the dQ
// partials saves the 128-key-tile kernel about a fifth of its time, less than the second
// pass costs, which recomputes S and dP.
bool separate_dq() { return g_dq_mode.load(std::memory_order_relaxed) == FA_BWD_DQ_SEPARATE; }

cudaError_t run_bwd(const void* Q, const void* K, const void* V, const void* dO, const float* LSE, const float* Dv,
                    void* dQ, void* dK, void* dV, float* dQacc, const Shape& s, float scale, bool causal,
                    const BwdVariant& var, int* status, cudaStream_t st) {
  cudaError_t e = cudaMemsetAsync(dQacc, 0, (size_t)s.elems() * sizeof(float), st);
  if (e != cudaSuccess) return e;
  if ((e = tc_bwd_wide(Q, K, V, dO, LSE, Dv, dK, dV, dQacc, s, scale, causal, var, status, st)) != cudaSuccess)
    return e;
  const int64_t n8 = s.elems() / 8;  // d is 64 or 128, so every row is whole groups of 8
  dq_convert_kernel<<<(unsigned)((n8 + 255) / 256), 256, 0, st>>>(dQacc, static_cast<__nv_bfloat16*>(dQ), n8, scale);
  return cudaGetLastError();
}

}  // namespace

int bwd_dq_mode() { return g_dq_mode.load(std::memory_order_relaxed); }
void set_bwd_dq_mode(int mode) { g_dq_mode.store(mode, std::memory_order_relaxed); }

cudaError_t tc_bwd(const void* Q, const void* K, const void* V, const void* dO, const float* LSE,
                   const float* D, void* dQ, void* dK, void* dV, float* dQacc, const Shape& s,
                   float scale, bool causal, int* status, cudaStream_t st) {
  if (separate_dq()) {
    cudaError_t e = tc_bwd_wide(Q, K, V, dO, LSE, D, dK, dV, nullptr, s, scale, causal, BwdVariant{}, status, st);
    if (e != cudaSuccess) return e;
    return tc_bwd_dq(Q, K, V, dO, LSE, D, dQ, s, scale, causal, status, st);
  }
  return run_bwd(Q, K, V, dO, LSE, D, dQ, dK, dV, dQacc, s, scale, causal, BwdVariant{}, status, st);
}

cudaError_t tc_bwd_masked(const void* Q, const void* K, const void* V, const void* dO, const float* LSE,
                          const float* D, void* dQ, void* dK, void* dV, float* dQacc, const Shape& s,
                          float scale, bool causal, const void* mask, int64_t mask_sb, int64_t mask_sh,
                          int64_t mask_srow, int* status, cudaStream_t st) {
  BwdVariant v;
  v.kind = 1;
  v.mask = mask;
  v.sb = mask_sb;
  v.sh = mask_sh;
  v.srow = mask_srow;
  return run_bwd(Q, K, V, dO, LSE, D, dQ, dK, dV, dQacc, s, scale, causal, v, status, st);
}

cudaError_t tc_bwd_bitmask(const void* Q, const void* K, const void* V, const void* dO, const float* LSE,
                           const float* D, void* dQ, void* dK, void* dV, float* dQacc, const Shape& s,
                           float scale, bool causal, const uint32_t* bits, int64_t bits_sb, int64_t bits_sh,
                           int64_t bits_srow, int* status, cudaStream_t st) {
  BwdVariant v;
  v.kind = 3;
  v.mask = bits;
  v.sb = bits_sb;
  v.sh = bits_sh;
  v.srow = bits_srow;
  return run_bwd(Q, K, V, dO, LSE, D, dQ, dK, dV, dQacc, s, scale, causal, v, status, st);
}

cudaError_t tc_bwd_dropout(const void* Q, const void* K, const void* V, const void* dO, const float* LSE,
                           const float* D, void* dQ, void* dK, void* dV, float* dQacc, const Shape& s,
                           float scale, bool causal, uint64_t seed, uint32_t threshold, int* status,
                           cudaStream_t st) {
  BwdVariant v;
  v.kind = 2;
  v.seed = seed;
  v.threshold = threshold;
  return run_bwd(Q, K, V, dO, LSE, D, dQ, dK, dV, dQacc, s, scale, causal, v, status, st);
}

}  // namespace fa
