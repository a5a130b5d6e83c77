// The backward entry functions of the tensor-core path: each zeroes the fp32 dQ accumulator,
// runs the backward kernel (fa_bwd_wide.cu) and converts the accumulator to bf16 dQ; what
// they compute is fa_bwd / fa_bwd_masked / fa_bwd_bitmask / fa_bwd_dropout in include/fa.h.
//
// dQ is a sum over key tiles, and every key tile is a different CTA: the kernel adds each
// tile's fp32 partial into the accumulator, and one pass here scales it by `scale` and
// rounds it to bf16 once ("FlashAttention 反向传播" 踩坑三: fp32 accumulators, a single cast at
// write-back).
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

cudaError_t tc_bwd(const void* Q, const void* K, const void* V, const void* dO, const float* LSE,
                   const float* D, void* dQ, void* dK, void* dV, float* dQacc, const Shape& s,
                   float scale, bool causal, int* status, cudaStream_t st) {
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
