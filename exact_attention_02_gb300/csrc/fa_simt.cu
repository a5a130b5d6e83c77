// Exact attention on the FFMA pipes: the float32 path (float32 inputs only; bf16 inputs run on
// the tensor-core kernels), and the row-dot D pass for both element types.
//
// One warp owns one query row (forward, dQ) or one key row (dK/dV); each step stages
// 32 keys (or queries) in shared memory, one per lane, so a warp forms 32 scores in
// parallel and merges them into its running statistics with one max and one sum
// reduction. This is the online softmax of "flash-attention-v2-sram-tiling" §5 with
// the un-normalised accumulator of "flash-attention-backpropagation" (Python 演示):
// O is rescaled by exp(m_old - m_new) whenever the row max grows and divided by l
// once at the end. Scores are kept in log2 units (the scale is folded into q, §7).
// The backward rebuilds P = exp(s - LSE) and follows Softmax梯度 / QKV梯度 of
// "flash-attention-backpropagation": dK/dV in one kernel over key rows, dQ in a
// second kernel over query rows, so no accumulator is shared between warps.
#include <cuda_bf16.h>

#include "fa_internal.h"

namespace fa {
namespace {

constexpr int kWarps = 8;   // rows per CTA, one warp each
constexpr int kChunk = 32;  // keys (or queries) staged per step, one per lane
constexpr float kLog2e = 1.4426950408889634f;
constexpr float kLn2 = 0.6931471805599453f;

__device__ __forceinline__ float ldf(const float* p) { return *p; }
__device__ __forceinline__ void stf(float* p, float v) { *p = v; }

__device__ __forceinline__ float warp_max(float v) {
#pragma unroll
  for (int o = 16; o; o >>= 1) v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, o));
  return v;
}
__device__ __forceinline__ float warp_sum(float v) {
#pragma unroll
  for (int o = 16; o; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
  return v;
}

// Shapes: Nq query rows and Nk key/value rows per head; causal hides key j from query i
// when j > i + offset (offset = Nk - Nq: the queries are the last Nq positions).

// Forward: grid = tiles * heads (flattened), block = kWarps warps, warp w -> query row.
template <typename T, int D>
__global__ void __launch_bounds__(kWarps * 32)
simt_fwd_kernel(const T* __restrict__ Q, const T* __restrict__ K, const T* __restrict__ V,
                T* __restrict__ O, float* __restrict__ LSE, int Nq, int Nk, int offset, int tiles,
                float scale, int causal) {
  __shared__ float ks[kChunk][D + 1];
  __shared__ float vs[kChunk][D];
  __shared__ float qs[kWarps][D];
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int64_t head = blockIdx.x / tiles;
  const int row0 = (blockIdx.x % tiles) * kWarps;
  const int row = row0 + warp;
  const bool active = row < Nq;
  const size_t base = (size_t)head * Nq * D, kbase = (size_t)head * Nk * D;
  const float sl2 = scale * kLog2e;
  for (int c = lane; c < D; c += 32)
    qs[warp][c] = active ? ldf(Q + base + (size_t)row * D + c) * sl2 : 0.f;

  float m = -INFINITY, l = 0.f, acc[D / 32];
#pragma unroll
  for (int t = 0; t < D / 32; ++t) acc[t] = 0.f;

  const int kv_end = causal ? min(Nk, row0 + kWarps + offset) : Nk;
  for (int j0 = 0; j0 < kv_end; j0 += kChunk) {
    __syncthreads();
    for (int e = threadIdx.x; e < kChunk * D; e += blockDim.x) {
      const int r = e / D, c = e % D, j = j0 + r;
      float kv = 0.f, vv = 0.f;
      if (j < Nk) {
        kv = ldf(K + kbase + (size_t)j * D + c);
        vv = ldf(V + kbase + (size_t)j * D + c);
      }
      ks[r][c] = kv;
      vs[r][c] = vv;
    }
    __syncthreads();
    const int j = j0 + lane;
    float s = 0.f;
#pragma unroll 16
    for (int c = 0; c < D; ++c) s = fmaf(qs[warp][c], ks[lane][c], s);
    const bool vis = active && j < Nk && (!causal || j <= row + offset);
    s = vis ? s : -INFINITY;
    const float mnew = fmaxf(m, warp_max(s));
    if (mnew == -INFINITY) continue;  // nothing visible yet in this row (warp-uniform)
    const float p = vis ? exp2f(s - mnew) : 0.f;
    const float corr = exp2f(m - mnew);
    l = l * corr + warp_sum(p);
#pragma unroll
    for (int t = 0; t < D / 32; ++t) acc[t] *= corr;
#pragma unroll 8
    for (int jj = 0; jj < kChunk; ++jj) {
      const float pj = __shfl_sync(0xffffffffu, p, jj);
#pragma unroll
      for (int t = 0; t < D / 32; ++t) acc[t] = fmaf(pj, vs[jj][lane + 32 * t], acc[t]);
    }
    m = mnew;
  }
  if (active) {
    const float inv = l > 0.f ? 1.f / l : 0.f;  // a query that sees no key: O = 0, LSE = -inf
#pragma unroll
    for (int t = 0; t < D / 32; ++t) stf(O + base + (size_t)row * D + lane + 32 * t, acc[t] * inv);
    if (lane == 0) LSE[head * Nq + row] = l > 0.f ? (m + log2f(l)) * kLn2 : -INFINITY;
  }
}

// dK, dV: warp w -> key row j; steps over query rows i >= (first key of the CTA) when causal.
template <typename T, int D>
__global__ void __launch_bounds__(kWarps * 32)
simt_bwd_dkdv_kernel(const T* __restrict__ Q, const T* __restrict__ K, const T* __restrict__ V,
                     const T* __restrict__ dO, const float* __restrict__ LSE,
                     const float* __restrict__ Dr, T* __restrict__ dK, T* __restrict__ dV, int Nq,
                     int Nk, int offset, int tiles, float scale, int causal) {
  __shared__ float qs[kChunk][D + 1];
  __shared__ float dos[kChunk][D + 1];
  __shared__ float kr[kWarps][D];
  __shared__ float vr[kWarps][D];
  __shared__ float lse2[kChunk], dd[kChunk];
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int64_t head = blockIdx.x / tiles;
  const int key0 = (blockIdx.x % tiles) * kWarps;
  const int key = key0 + warp;
  const bool active = key < Nk;
  const size_t base = (size_t)head * Nq * D, kbase = (size_t)head * Nk * D;
  const float sl2 = scale * kLog2e;
  for (int c = lane; c < D; c += 32) {
    kr[warp][c] = active ? ldf(K + kbase + (size_t)key * D + c) * sl2 : 0.f;
    vr[warp][c] = active ? ldf(V + kbase + (size_t)key * D + c) : 0.f;
  }
  float dk[D / 32], dv[D / 32];
#pragma unroll
  for (int t = 0; t < D / 32; ++t) dk[t] = dv[t] = 0.f;

  const int i_start = causal ? (max(0, key0 - offset) / kChunk) * kChunk : 0;
  for (int i0 = i_start; i0 < Nq; i0 += kChunk) {
    __syncthreads();
    for (int e = threadIdx.x; e < kChunk * D; e += blockDim.x) {
      const int r = e / D, c = e % D, i = i0 + r;
      float qv = 0.f, dov = 0.f;
      if (i < Nq) {
        qv = ldf(Q + base + (size_t)i * D + c);
        dov = ldf(dO + base + (size_t)i * D + c);
      }
      qs[r][c] = qv;
      dos[r][c] = dov;
    }
    if (threadIdx.x < kChunk) {
      const int i = i0 + threadIdx.x;
      lse2[threadIdx.x] = i < Nq ? LSE[head * Nq + i] * kLog2e : 0.f;
      dd[threadIdx.x] = i < Nq ? Dr[head * Nq + i] : 0.f;
    }
    __syncthreads();
    const int i = i0 + lane;
    float s = 0.f, dp = 0.f;
#pragma unroll 16
    for (int c = 0; c < D; ++c) {
      s = fmaf(qs[lane][c], kr[warp][c], s);
      dp = fmaf(dos[lane][c], vr[warp][c], dp);
    }
    const bool vis = active && i < Nq && (!causal || key <= i + offset);
    const float p = vis ? exp2f(s - lse2[lane]) : 0.f;
    const float ds = p * (dp - dd[lane]);
#pragma unroll 8
    for (int ii = 0; ii < kChunk; ++ii) {
      const float pi = __shfl_sync(0xffffffffu, p, ii);
      const float dsi = __shfl_sync(0xffffffffu, ds, ii);
#pragma unroll
      for (int t = 0; t < D / 32; ++t) {
        dv[t] = fmaf(pi, dos[ii][lane + 32 * t], dv[t]);
        dk[t] = fmaf(dsi, qs[ii][lane + 32 * t], dk[t]);
      }
    }
  }
  if (active) {
#pragma unroll
    for (int t = 0; t < D / 32; ++t) {
      stf(dV + kbase + (size_t)key * D + lane + 32 * t, dv[t]);
      stf(dK + kbase + (size_t)key * D + lane + 32 * t, dk[t] * scale);
    }
  }
}

// dQ: warp w -> query row i; steps over keys j <= (last row of the CTA) when causal.
template <typename T, int D>
__global__ void __launch_bounds__(kWarps * 32)
simt_bwd_dq_kernel(const T* __restrict__ Q, const T* __restrict__ K, const T* __restrict__ V,
                   const T* __restrict__ dO, const float* __restrict__ LSE,
                   const float* __restrict__ Dr, T* __restrict__ dQ, int Nq, int Nk, int offset,
                   int tiles, float scale, int causal) {
  __shared__ float ks[kChunk][D + 1];
  __shared__ float vs[kChunk][D + 1];
  __shared__ float qr[kWarps][D];
  __shared__ float dor[kWarps][D];
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int64_t head = blockIdx.x / tiles;
  const int row0 = (blockIdx.x % tiles) * kWarps;
  const int row = row0 + warp;
  const bool active = row < Nq;
  const size_t base = (size_t)head * Nq * D, kbase = (size_t)head * Nk * D;
  const float sl2 = scale * kLog2e;
  for (int c = lane; c < D; c += 32) {
    qr[warp][c] = active ? ldf(Q + base + (size_t)row * D + c) * sl2 : 0.f;
    dor[warp][c] = active ? ldf(dO + base + (size_t)row * D + c) : 0.f;
  }
  const float lse2 = active ? LSE[head * Nq + row] * kLog2e : 0.f;
  const float drow = active ? Dr[head * Nq + row] : 0.f;
  float dq[D / 32];
#pragma unroll
  for (int t = 0; t < D / 32; ++t) dq[t] = 0.f;

  const int kv_end = causal ? min(Nk, row0 + kWarps + offset) : Nk;
  for (int j0 = 0; j0 < kv_end; j0 += kChunk) {
    __syncthreads();
    for (int e = threadIdx.x; e < kChunk * D; e += blockDim.x) {
      const int r = e / D, c = e % D, j = j0 + r;
      float kv = 0.f, vv = 0.f;
      if (j < Nk) {
        kv = ldf(K + kbase + (size_t)j * D + c);
        vv = ldf(V + kbase + (size_t)j * D + c);
      }
      ks[r][c] = kv;
      vs[r][c] = vv;
    }
    __syncthreads();
    const int j = j0 + lane;
    float s = 0.f, dp = 0.f;
#pragma unroll 16
    for (int c = 0; c < D; ++c) {
      s = fmaf(qr[warp][c], ks[lane][c], s);
      dp = fmaf(dor[warp][c], vs[lane][c], dp);
    }
    const bool vis = active && j < Nk && (!causal || j <= row + offset);
    const float p = vis ? exp2f(s - lse2) : 0.f;
    const float ds = p * (dp - drow);
#pragma unroll 8
    for (int jj = 0; jj < kChunk; ++jj) {
      const float dsj = __shfl_sync(0xffffffffu, ds, jj);
#pragma unroll
      for (int t = 0; t < D / 32; ++t) dq[t] = fmaf(dsj, ks[jj][lane + 32 * t], dq[t]);
    }
  }
  if (active) {
#pragma unroll
    for (int t = 0; t < D / 32; ++t) stf(dQ + base + (size_t)row * D + lane + 32 * t, dq[t] * scale);
  }
}

// D_i = sum_c dO_ic O_ic. A thread handles kItems 16-byte pieces of O and of dO, kStride
// threads apart, and issues all of their loads before the first use, so each thread keeps
// 2 * kItems loads in flight (one piece each measured 0.74 of the HBM copy rate). The G
// threads that cover one row (G = row bytes / 16, a power of two <= 32) are consecutive
// lanes of a warp and reduce by shuffles.
constexpr int kPreItems = 4;
constexpr int kPreThreads = 256;

template <typename T, int D>
__global__ void __launch_bounds__(kPreThreads)
preprocess_kernel(const T* __restrict__ O, const T* __restrict__ dO, float* __restrict__ Dr,
                  int64_t rows) {
  constexpr int kVec = 16 / sizeof(T);
  constexpr int G = D / kVec;
  const int64_t pieces = rows * G;
  const int64_t stride = (int64_t)gridDim.x * kPreThreads;  // a multiple of 32: lanes keep their rows
  const int64_t tid = (int64_t)blockIdx.x * kPreThreads + threadIdx.x;
  uint4 a[kPreItems], b[kPreItems];
#pragma unroll
  for (int u = 0; u < kPreItems; ++u) {
    const int64_t i = tid + u * stride;
    if (i < pieces) {
      a[u] = *reinterpret_cast<const uint4*>(O + i * kVec);
      b[u] = *reinterpret_cast<const uint4*>(dO + i * kVec);
    } else {
      a[u] = b[u] = make_uint4(0, 0, 0, 0);
    }
  }
#pragma unroll
  for (int u = 0; u < kPreItems; ++u) {
    float acc = 0.f;
    if constexpr (sizeof(T) == 2) {
      const __nv_bfloat162* pa = reinterpret_cast<const __nv_bfloat162*>(&a[u]);
      const __nv_bfloat162* pb = reinterpret_cast<const __nv_bfloat162*>(&b[u]);
#pragma unroll
      for (int v = 0; v < 4; ++v) {
        const float2 fa = __bfloat1622float2(pa[v]);
        const float2 fb = __bfloat1622float2(pb[v]);
        acc = fmaf(fa.x, fb.x, acc);
        acc = fmaf(fa.y, fb.y, acc);
      }
    } else {
      const float* pa = reinterpret_cast<const float*>(&a[u]);
      const float* pb = reinterpret_cast<const float*>(&b[u]);
#pragma unroll
      for (int v = 0; v < 4; ++v) acc = fmaf(pa[v], pb[v], acc);
    }
#pragma unroll
    for (int o = G / 2; o; o >>= 1) acc += __shfl_xor_sync(0xffffffffu, acc, o);
    const int64_t i = tid + u * stride;
    if (i < pieces && i % G == 0) Dr[i / G] = acc;
  }
}

template <typename T, int D>
cudaError_t launch_fwd(const void* Q, const void* K, const void* V, void* O, float* LSE,
                       const Shape& s, float scale, bool causal, cudaStream_t st) {
  const int tiles = (s.N + kWarps - 1) / kWarps;
  const int64_t grid = (int64_t)tiles * s.heads();
  const int offset = causal ? s.keys() - s.N : 0;
  simt_fwd_kernel<T, D><<<(unsigned)grid, kWarps * 32, 0, st>>>(
      (const T*)Q, (const T*)K, (const T*)V, (T*)O, LSE, s.N, s.keys(), offset, tiles, scale, causal ? 1 : 0);
  return cudaGetLastError();
}

template <typename T, int D>
cudaError_t launch_bwd(const void* Q, const void* K, const void* V, const void* dO,
                       const float* LSE, const float* Dr, void* dQ, void* dK, void* dV,
                       const Shape& s, float scale, bool causal, cudaStream_t st) {
  const int qtiles = (s.N + kWarps - 1) / kWarps, ktiles = (s.keys() + kWarps - 1) / kWarps;
  const int offset = causal ? s.keys() - s.N : 0;
  simt_bwd_dkdv_kernel<T, D><<<(unsigned)((int64_t)ktiles * s.heads()), kWarps * 32, 0, st>>>(
      (const T*)Q, (const T*)K, (const T*)V, (const T*)dO, LSE, Dr, (T*)dK, (T*)dV, s.N, s.keys(), offset,
      ktiles, scale, causal ? 1 : 0);
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  simt_bwd_dq_kernel<T, D><<<(unsigned)((int64_t)qtiles * s.heads()), kWarps * 32, 0, st>>>(
      (const T*)Q, (const T*)K, (const T*)V, (const T*)dO, LSE, Dr, (T*)dQ, s.N, s.keys(), offset, qtiles, scale,
      causal ? 1 : 0);
  return cudaGetLastError();
}

template <typename T, int D>
cudaError_t launch_pre(const void* O, const void* dO, float* Dr, const Shape& s, cudaStream_t st) {
  constexpr int G = D / (16 / sizeof(T));
  const int64_t pieces = s.rows() * G;
  const int64_t per_block = (int64_t)kPreThreads * kPreItems;
  const int64_t grid = (pieces + per_block - 1) / per_block;
  preprocess_kernel<T, D><<<(unsigned)grid, kPreThreads, 0, st>>>((const T*)O, (const T*)dO, Dr, s.rows());
  return cudaGetLastError();
}

}  // namespace

cudaError_t simt_fwd(const void* Q, const void* K, const void* V, void* O, float* LSE,
                     const Shape& s, float scale, bool causal, cudaStream_t st) {
  return s.d == 64 ? launch_fwd<float, 64>(Q, K, V, O, LSE, s, scale, causal, st)
                   : launch_fwd<float, 128>(Q, K, V, O, LSE, s, scale, causal, st);
}

cudaError_t simt_bwd(const void* Q, const void* K, const void* V, const void* dO,
                     const float* LSE, const float* D, void* dQ, void* dK, void* dV,
                     const Shape& s, float scale, bool causal, cudaStream_t st) {
  return s.d == 64 ? launch_bwd<float, 64>(Q, K, V, dO, LSE, D, dQ, dK, dV, s, scale, causal, st)
                   : launch_bwd<float, 128>(Q, K, V, dO, LSE, D, dQ, dK, dV, s, scale, causal, st);
}

cudaError_t preprocess_d(const void* O, const void* dO, float* D, const Shape& s, bool bf16,
                         cudaStream_t st) {
  if (bf16)
    return s.d == 64 ? launch_pre<__nv_bfloat16, 64>(O, dO, D, s, st)
                     : launch_pre<__nv_bfloat16, 128>(O, dO, D, s, st);
  return s.d == 64 ? launch_pre<float, 64>(O, dO, D, s, st) : launch_pre<float, 128>(O, dO, D, s, st);
}

}  // namespace fa
