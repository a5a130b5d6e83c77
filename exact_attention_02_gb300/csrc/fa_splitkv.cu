// Split-KV forward: a few queries (N_q <= 16, e.g. one decoding step) against a long key /
// value sequence; what it computes is fa_fwd_splitkv in include/fa.h.
//
// The work per head is too small to fill the GPU along the query axis, so the keys are
// cut into `splits` chunks processed by separate CTAs, each keeping the online-softmax
// state (running max m, running sum l, un-normalised O) of "flash-attention-v2-sram-
// tiling" §5 for its chunk. A second kernel merges the chunk states of every query with
// the rule of "知识点13 FlashAttention深度攻略" §4: m = max_s m_s,
// l = sum_s l_s e^(m_s - m), O = sum_s O_s e^(m_s - m) / l. Scores are kept in log2 units
// (scale * log2 e folded into q), so every exponential is one ex2.
//
// The kernel reads each key and value row once from HBM and does 4 * N_q * d FLOPs per
// key, so for small N_q it is bound by HBM bandwidth; it runs on the FFMA pipes.
//
// Causal attention with N_q <= N_k places the queries at the last N_q positions
// (bottom-right alignment): query i hides keys j > i + N_k - N_q.
#include <cuda_bf16.h>

#include <algorithm>

#include "fa_internal.h"
#include "sm100_ptx.cuh"

namespace fa {

int splitkv_splits(int64_t heads, int Nk) {
  const int64_t target = 4 * 152;  // about four waves of CTAs on a 152-SM GPU
  const int64_t want = (target + heads - 1) / heads;
  const int64_t most = (Nk + 255) / 256;  // at least 256 keys per chunk
  return (int)std::max<int64_t>(1, std::min(want, most));
}

namespace {

constexpr int kWarps = 4;
constexpr float kLn2 = 0.6931471805599453f;

__device__ __forceinline__ float wmax(float v) {
#pragma unroll
  for (int o = 16; o; o >>= 1) v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, o));
  return v;
}
__device__ __forceinline__ float wsum(float v) {
#pragma unroll
  for (int o = 16; o; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
  return v;
}

struct SplitParams {
  const __nv_bfloat16* Q;
  const __nv_bfloat16* K;
  const __nv_bfloat16* V;
  float* part_o;   // [heads][splits][nq][D]
  float* part_ml;  // [heads][splits][nq][2]
  int nq, Nk, splits, chunk, causal, offset;
  float sl2;  // scale * log2(e)
};

// grid (heads, splits), 4 warps; each warp takes every 4th 32-key group of the chunk.
template <int D, int NQ>
__global__ void __launch_bounds__(kWarps * 32) splitkv_partial_kernel(const SplitParams p) {
  constexpr int C = D / 32;  // output columns per lane
  __shared__ float qs[NQ][D];
  __shared__ float wm[kWarps][NQ], wl[kWarps][NQ];
  __shared__ float wo[kWarps][NQ][D];
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int64_t head = blockIdx.x;
  const int split = blockIdx.y;
  const int nq = p.nq;
  for (int e = threadIdx.x; e < NQ * D; e += blockDim.x) {
    const int qi = e / D;
    qs[qi][e % D] = qi < nq ? __bfloat162float(p.Q[(head * nq + qi) * D + e % D]) * p.sl2 : 0.f;
  }
  __syncthreads();

  const __nv_bfloat16* Kh = p.K + head * p.Nk * D;
  const __nv_bfloat16* Vh = p.V + head * p.Nk * D;
  const int k0 = split * p.chunk;
  const int k1 = min(p.Nk, k0 + p.chunk);
  float m[NQ], lsum[NQ], acc[NQ][C];
#pragma unroll
  for (int qi = 0; qi < NQ; ++qi) {
    m[qi] = -INFINITY;
    lsum[qi] = 0.f;
#pragma unroll
    for (int c = 0; c < C; ++c) acc[qi][c] = 0.f;
  }

  for (int base = k0 + warp * 32; base < k1; base += kWarps * 32) {
    const int key = base + lane;
    const bool valid = key < k1;
    // s[qi] = q_i . k_key (already in log2 units), streaming the key row in 16 B pieces
    float s[NQ];
#pragma unroll
    for (int qi = 0; qi < NQ; ++qi) s[qi] = 0.f;
    const uint4* krow = reinterpret_cast<const uint4*>(Kh + (int64_t)(valid ? key : k0) * D);
#pragma unroll 4
    for (int ch = 0; ch < D / 8; ++ch) {
      const uint4 u = krow[ch];
      const __nv_bfloat162* h = reinterpret_cast<const __nv_bfloat162*>(&u);
      float kf[8];
#pragma unroll
      for (int t = 0; t < 4; ++t) {
        const float2 f = __bfloat1622float2(h[t]);
        kf[2 * t] = f.x;
        kf[2 * t + 1] = f.y;
      }
#pragma unroll
      for (int qi = 0; qi < NQ; ++qi)
        if (qi < nq) {
#pragma unroll
          for (int t = 0; t < 8; ++t) s[qi] = fmaf(qs[qi][ch * 8 + t], kf[t], s[qi]);
        }
    }
    float pq[NQ];
#pragma unroll
    for (int qi = 0; qi < NQ; ++qi) {
      pq[qi] = 0.f;
      if (qi >= nq) continue;
      const bool vis = valid && !(p.causal && key > qi + p.offset);
      const float sv = vis ? s[qi] : -INFINITY;
      const float mnew = fmaxf(m[qi], wmax(sv));
      if (mnew == -INFINITY) continue;  // nothing visible yet for this query (warp-uniform)
      const float corr = ptx::ex2(m[qi] - mnew);
      pq[qi] = vis ? ptx::ex2(sv - mnew) : 0.f;
      lsum[qi] = lsum[qi] * corr + pq[qi];
#pragma unroll
      for (int c = 0; c < C; ++c) acc[qi][c] *= corr;
      m[qi] = mnew;
    }
    // O += p V over the 32 keys of the group; lanes own head-dim columns lane*C .. +C
    const int kend = min(32, k1 - base);
#pragma unroll 4
    for (int kk = 0; kk < kend; ++kk) {
      const __nv_bfloat16* vrow = Vh + (int64_t)(base + kk) * D + lane * C;
      float vf[C];
      if constexpr (C == 4) {
        const uint2 u = *reinterpret_cast<const uint2*>(vrow);
        const float2 a = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&u.x));
        const float2 b = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&u.y));
        vf[0] = a.x, vf[1] = a.y, vf[2] = b.x, vf[3] = b.y;
      } else {
        const float2 a = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(vrow));
        vf[0] = a.x, vf[1] = a.y;
      }
#pragma unroll
      for (int qi = 0; qi < NQ; ++qi)
        if (qi < nq) {
          const float pk = __shfl_sync(0xffffffffu, pq[qi], kk);
#pragma unroll
          for (int c = 0; c < C; ++c) acc[qi][c] = fmaf(pk, vf[c], acc[qi][c]);
        }
    }
  }

  // combine the four warps' states, then write this chunk's (m, l, O) per query
#pragma unroll
  for (int qi = 0; qi < NQ; ++qi) {
    const float l = wsum(lsum[qi]);
    if (lane == 0) {
      wm[warp][qi] = m[qi];
      wl[warp][qi] = l;
    }
#pragma unroll
    for (int c = 0; c < C; ++c) wo[warp][qi][lane * C + c] = acc[qi][c];
  }
  __syncthreads();
  const int64_t slot = (head * p.splits + split) * nq;
  for (int e = threadIdx.x; e < nq * D; e += blockDim.x) {
    const int qi = e / D, col = e % D;
    float M = -INFINITY;
#pragma unroll
    for (int w = 0; w < kWarps; ++w) M = fmaxf(M, wm[w][qi]);
    float o = 0.f, l = 0.f;
    if (M != -INFINITY) {
#pragma unroll
      for (int w = 0; w < kWarps; ++w) {
        const float f = ptx::ex2(wm[w][qi] - M);
        o = fmaf(wo[w][qi][col], f, o);
        l = fmaf(wl[w][qi], f, l);
      }
    }
    p.part_o[(slot + qi) * D + col] = o;
    if (col == 0) {
      p.part_ml[(slot + qi) * 2] = M;
      p.part_ml[(slot + qi) * 2 + 1] = l;
    }
  }
}

// One warp per (head, query): merge the chunk states and write O (bf16) and LSE.
template <int D>
__global__ void __launch_bounds__(128) splitkv_merge_kernel(const float* __restrict__ part_o,
                                                           const float* __restrict__ part_ml,
                                                           __nv_bfloat16* __restrict__ O, float* __restrict__ LSE,
                                                           int64_t rows, int nq, int splits) {
  constexpr int C = D / 32;
  const int64_t row = (int64_t)blockIdx.x * 4 + (threadIdx.x >> 5);  // head * nq + qi
  const int lane = threadIdx.x & 31;
  if (row >= rows) return;
  const int64_t head = row / nq, qi = row % nq;
  const float* ml = part_ml + (head * splits * nq + qi) * 2;  // split s at + s*nq*2
  float M = -INFINITY;
  for (int s = lane; s < splits; s += 32) M = fmaxf(M, ml[(int64_t)s * nq * 2]);
  M = wmax(M);
  float l = 0.f, o[C];
#pragma unroll
  for (int c = 0; c < C; ++c) o[c] = 0.f;
  for (int s = 0; s < splits; ++s) {
    const float ms = ml[(int64_t)s * nq * 2];
    if (ms == -INFINITY) continue;  // a chunk with no visible key
    const float f = ptx::ex2(ms - M);
    l = fmaf(ml[(int64_t)s * nq * 2 + 1], f, l);
    const float* po = part_o + ((head * splits + s) * nq + qi) * D + lane * C;
#pragma unroll
    for (int c = 0; c < C; ++c) o[c] = fmaf(po[c], f, o[c]);
  }
  const float inv = 1.f / l;
  __nv_bfloat16* orow = O + row * D + lane * C;
#pragma unroll
  for (int c = 0; c < C; c += 2) *reinterpret_cast<uint32_t*>(orow + c) = ptx::pack_bf16(o[c] * inv, o[c + 1] * inv);
  if (lane == 0) LSE[row] = (M + log2f(l)) * kLn2;
}

template <int D, int NQ>
cudaError_t launch(const SplitParams& p, int64_t heads, cudaStream_t st) {
  splitkv_partial_kernel<D, NQ><<<dim3((unsigned)heads, p.splits), kWarps * 32, 0, st>>>(p);
  return cudaGetLastError();
}

}  // namespace

size_t splitkv_workspace_floats(int64_t heads, int Nq, int Nk, int d) {
  return (size_t)splitkv_splits(heads, Nk) * heads * Nq * (d + 2);
}

cudaError_t splitkv_fwd(const void* Q, const void* K, const void* V, void* O, float* LSE, int64_t heads,
                        int Nq, int Nk, int d, float scale, bool causal, float* workspace, cudaStream_t st) {
  SplitParams p;
  p.Q = static_cast<const __nv_bfloat16*>(Q);
  p.K = static_cast<const __nv_bfloat16*>(K);
  p.V = static_cast<const __nv_bfloat16*>(V);
  p.nq = Nq;
  p.Nk = Nk;
  p.splits = splitkv_splits(heads, Nk);
  p.chunk = (((Nk + p.splits - 1) / p.splits) + 31) / 32 * 32;
  p.causal = causal ? 1 : 0;
  p.offset = Nk - Nq;
  p.sl2 = scale * 1.4426950408889634f;
  p.part_o = workspace;
  p.part_ml = workspace + (size_t)p.splits * heads * Nq * d;
  cudaError_t e;
  if (d == 64)
    e = Nq == 1 ? launch<64, 1>(p, heads, st) : Nq <= 4 ? launch<64, 4>(p, heads, st) : launch<64, 16>(p, heads, st);
  else
    e = Nq == 1 ? launch<128, 1>(p, heads, st) : Nq <= 4 ? launch<128, 4>(p, heads, st) : launch<128, 16>(p, heads, st);
  if (e != cudaSuccess) return e;
  const int64_t rows = heads * Nq;
  const unsigned grid = (unsigned)((rows + 3) / 4);
  if (d == 64)
    splitkv_merge_kernel<64><<<grid, 128, 0, st>>>(p.part_o, p.part_ml, static_cast<__nv_bfloat16*>(O), LSE, rows,
                                                   Nq, p.splits);
  else
    splitkv_merge_kernel<128><<<grid, 128, 0, st>>>(p.part_o, p.part_ml, static_cast<__nv_bfloat16*>(O), LSE,
                                                    rows, Nq, p.splits);
  return cudaGetLastError();
}

}  // namespace fa
