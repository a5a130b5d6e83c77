// Split-KV forward: a few queries (e.g. one decoding step) against a long key / value
// sequence; what it computes is fa_fwd_splitkv in include/fa.h. This file holds the work
// split, the merge and the entry point; the partial states come from the tensor-core
// kernel in fa_splitkv_tc.cu.
//
// The work per head is too small to fill the GPU along the query axis, so the keys are cut
// into pieces processed by separate CTAs, each keeping the online-softmax state (running
// max m, running sum l, un-normalised O) of "flash-attention-v2-sram-tiling" §5 for its
// piece. A second kernel merges the piece states of every query with the rule of
// "知识点13 FlashAttention深度攻略" §4: m = max_s m_s, l = sum_s l_s e^(m_s - m),
// O = sum_s O_s e^(m_s - m) / l. Scores are kept in log2 units (scale * log2 e folded in),
// so every exponential is one ex2.
//
// Work split. K and V of all heads are one contiguous sequence of B*H*N_k rows. It is cut
// into equal contiguous ranges, one per CTA and one CTA per SM, so every SM streams the
// same number of bytes and there is no partial last wave. A range may start or end inside
// a head and may cover the end of one head and the start of the next: each piece of a head
// inside a range is a "segment" and yields one partial state, stored in the slot
// (head, CTA - first CTA of that head).
//
// Causal attention with N_q <= N_k places the queries at the last N_q positions
// (bottom-right alignment): query i hides keys j > i + N_k - N_q.
#include <cuda_bf16.h>

#include <algorithm>

#include "fa_internal.h"
#include "sm100_ptx.cuh"

namespace fa {

namespace {

constexpr int kCtas = 152;          // one CTA per SM of the 152-SM GB300
constexpr int kMinKeysPerCta = 256;
constexpr int kTileKeys = 32;               // CTA ranges are whole multiples of 32 keys
constexpr float kLn2 = 0.6931471805599453f;

struct Layout {
  int64_t L;  // keys per CTA range (a multiple of 32)
  int ctas;   // number of ranges = grid size
  int P;      // partial-state slots per head: the most CTAs one head can touch
};

Layout layout(int64_t heads, int Nk) {
  const int64_t total = heads * Nk;
  int64_t L = std::max<int64_t>((total + kCtas - 1) / kCtas, kMinKeysPerCta);
  L = (L + kTileKeys - 1) / kTileKeys * kTileKeys;
  Layout r;
  r.L = L;
  r.ctas = (int)((total + L - 1) / L);
  r.P = (int)((Nk + L - 1) / L) + 1;
  return r;
}

__device__ __forceinline__ float wmax(float v) {
#pragma unroll
  for (int o = 16; o; o >>= 1) v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, o));
  return v;
}

template <int D>
__global__ void __launch_bounds__(128) splitkv_merge_kernel(const float* __restrict__ part_o,
                                                           const float* __restrict__ part_ml,
                                                           __nv_bfloat16* __restrict__ O, float* __restrict__ LSE,
                                                           int64_t rows, int nq, int Nk, int64_t L, int P) {
  constexpr int C = D / 32;
  const int64_t row = (int64_t)blockIdx.x * 4 + (threadIdx.x >> 5);  // head * nq + qi
  const int lane = threadIdx.x & 31;
  if (row >= rows) return;
  const int64_t head = row / nq, qi = row % nq;
  // the CTAs whose key ranges touch this head wrote slots 0 .. cnt-1
  const int cnt = (int)(((head + 1) * Nk - 1) / L - (head * Nk) / L) + 1;
  const float* ml = part_ml + (head * P * nq + qi) * 2;  // slot s at + s*nq*2
  float M = -INFINITY;
  for (int s = lane; s < cnt; s += 32) M = fmaxf(M, ml[(int64_t)s * nq * 2]);
  M = wmax(M);
  float l = 0.f, o[C];
#pragma unroll
  for (int c = 0; c < C; ++c) o[c] = 0.f;
  for (int s = 0; s < cnt; ++s) {
    const float ms = ml[(int64_t)s * nq * 2];
    if (ms == -INFINITY) continue;  // a piece with no key visible to this query
    const float f = ptx::ex2(ms - M);
    l = fmaf(ml[(int64_t)s * nq * 2 + 1], f, l);
    const float* po = part_o + ((head * P + s) * nq + qi) * D + lane * C;
#pragma unroll
    for (int c = 0; c < C; ++c) o[c] = fmaf(po[c], f, o[c]);
  }
  const float inv = 1.f / l;
  __nv_bfloat16* orow = O + row * D + lane * C;
#pragma unroll
  for (int c = 0; c < C; c += 2) *reinterpret_cast<uint32_t*>(orow + c) = ptx::pack_bf16(o[c] * inv, o[c + 1] * inv);
  if (lane == 0) LSE[row] = (M + log2f(l)) * kLn2;
}

}  // namespace

size_t splitkv_workspace_floats(int64_t heads, int Nq, int Nk, int d) {
  return (size_t)layout(heads, Nk).P * heads * Nq * (d + 2);
}

cudaError_t splitkv_fwd(const void* Q, const void* K, const void* V, void* O, float* LSE, int64_t heads,
                        int Nq, int Nk, int d, float scale, bool causal, float* workspace, int* status,
                        cudaStream_t st) {
  if (d != 64 && d != 128) return cudaErrorInvalidValue;
  const Layout lay = layout(heads, Nk);
  float* part_o = workspace;  // [heads][P][Nq][d], then (m, l) [heads][P][Nq][2]
  float* part_ml = workspace + (size_t)lay.P * heads * Nq * d;
  cudaError_t e = splitkv_tc_partial(Q, K, V, heads, Nq, Nk, d, scale, causal, lay.L, lay.ctas, lay.P, part_o, part_ml,
                                     status, st);
  if (e != cudaSuccess) return e;
  const int64_t rows = heads * Nq;
  const unsigned grid = (unsigned)((rows + 3) / 4);
  if (d == 64)
    splitkv_merge_kernel<64><<<grid, 128, 0, st>>>(part_o, part_ml, static_cast<__nv_bfloat16*>(O), LSE, rows, Nq, Nk,
                                                   lay.L, lay.P);
  else
    splitkv_merge_kernel<128><<<grid, 128, 0, st>>>(part_o, part_ml, static_cast<__nv_bfloat16*>(O), LSE, rows, Nq,
                                                    Nk, lay.L, lay.P);
  return cudaGetLastError();
}

}  // namespace fa
