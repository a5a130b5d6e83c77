// Split-KV forward: a few queries (e.g. one decoding step) against a long key / value
// sequence; what it computes is fa_fwd_splitkv in include/fa.h. This file holds the work
// split, the FFMA partial kernel (d = 64, up to 16 queries) and the merge; with d = 128 the
// partial states come from the tensor-core kernel in fa_splitkv_tc.cu instead.
//
// The work per head is too small to fill the GPU along the query axis, so the keys are cut
// into pieces processed by separate CTAs, each keeping the online-softmax state (running
// max m, running sum l, un-normalised O) of "flash-attention-v2-sram-tiling" §5 for its
// piece. A second kernel merges the piece states of every query with the rule of
// "知识点13 FlashAttention深度攻略" §4: m = max_s m_s, l = sum_s l_s e^(m_s - m),
// O = sum_s O_s e^(m_s - m) / l. Scores are kept in log2 units (scale * log2 e folded into
// q), so every exponential is one ex2.
//
// Work split. K and V of all heads are one contiguous sequence of B*H*N_k rows. It is cut
// into equal contiguous ranges, one per CTA and one CTA per SM, so every SM streams the
// same number of bytes and there is no partial last wave. A range may start or end inside
// a head and may cover the end of one head and the start of the next: each piece of a head
// inside a range is a "segment" and yields one partial state, stored in the slot
// (head, CTA - first CTA of that head).
//
// Pipeline. One producer thread streams 32-key tiles of K and V into a ring of shared-
// memory stages with TMA (3-D maps [heads, N_k, d], 128-byte swizzle, rows past the end of
// a head read as zeros). Four consumer warps take the tiles round-robin, each keeping its
// own online-softmax state; at the end of a segment the four states are merged through
// shared memory. For q.k a lane owns one key and walks its row in 16-byte chunks; the
// swizzle puts the chunks of 8 consecutive rows in 8 different bank groups, so these reads
// are free of bank conflicts. For p.V a lane owns d/32 output columns of every query.
//
// Each key and value row is read once from HBM and costs 4 * N_q * d FLOPs on the FFMA
// pipes, so the kernel is bound by HBM bandwidth for N_q up to about 8; at N_q = 16 the
// FFMA pipes become the limit.
//
// Causal attention with N_q <= N_k places the queries at the last N_q positions
// (bottom-right alignment): query i hides keys j > i + N_k - N_q.
#include <cuda_bf16.h>

#include <algorithm>

#include "fa_internal.h"
#include "sm100_ptx.cuh"
#include "tma_host.h"

namespace fa {

namespace {

constexpr int kCtas = 152;          // one CTA per SM of the 152-SM GB300
constexpr int kMinKeysPerCta = 256;
constexpr int kTileKeys = 32;
constexpr int kConsumerWarps = 4;
constexpr int kThreads = (kConsumerWarps + 1) * 32;  // + one producer warp
constexpr int kSmemBudget = 200 * 1024;
constexpr float kLn2 = 0.6931471805599453f;

struct Layout {
  int64_t L;  // keys per CTA range (multiple of the tile)
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

template <int D>
struct Cfg {
  static constexpr int kBoxes = D / 64;                  // 64-column TMA boxes per row
  static constexpr int kBoxBytes = kTileKeys * 128;      // 32 rows x 64 bf16
  static constexpr int kTileBytes = kBoxes * kBoxBytes;  // one tile of K (or of V)
  static constexpr int kStageBytes = 2 * kTileBytes;     // K and V
  static constexpr int C = D / 32;                       // output columns per lane
};

// Stage ring first (1024-byte aligned for the swizzle), then the consumers' buffers.
// The stage count is a multiple of the consumer-warp count, so a stage is always filled
// for the same warp; that warp has waited on the stage's previous fill before it waits on
// the next, so the parity of the full barrier is never two phases behind.
template <int D, int NQ>
struct Smem {
  using G = Cfg<D>;
  static constexpr int kExtra = kConsumerWarps * NQ * D * 4 + NQ * D * 4 + kConsumerWarps * kTileKeys * NQ * 4 +
                                2 * kConsumerWarps * NQ * 4 + 1024;
  static constexpr int kStages = (kSmemBudget - kExtra) / G::kStageBytes / kConsumerWarps * kConsumerWarps;
  static_assert(kStages >= kConsumerWarps && kStages % kConsumerWarps == 0, "stage ring");
  static constexpr int kWo = kStages * G::kStageBytes;              // [warps][NQ][D] f32
  static constexpr int kQs = kWo + kConsumerWarps * NQ * D * 4;     // [NQ][D] f32, scaled q
  static constexpr int kPs = kQs + NQ * D * 4;                      // [warps][32][NQ] f32
  static constexpr int kWm = kPs + kConsumerWarps * kTileKeys * NQ * 4;
  static constexpr int kWl = kWm + kConsumerWarps * NQ * 4;
  static constexpr int kBar = (kWl + kConsumerWarps * NQ * 4 + 7) / 8 * 8;  // full[S], empty[S]
  static constexpr int kAbort = kBar + 2 * kStages * 8;
  static constexpr int kBytes = kAbort + 16;
  static constexpr int kAlloc = kBytes + 1024;  // slack to align the stages to 1024 bytes
};

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
__device__ __forceinline__ void consumers_sync() {
  asm volatile("bar.sync 1, %0;" ::"n"(kConsumerWarps * 32) : "memory");
}

struct SplitParams {
  const __nv_bfloat16* Q;
  float* part_o;   // [heads][P][nq][D]
  float* part_ml;  // [heads][P][nq][2]: (m in log2 units, l)
  int64_t total;   // heads * Nk
  int64_t L;
  int nq, Nk, P, causal, offset;
  float sl2;  // scale * log2(e)
  int* status;
};

template <int D, int NQ>
__global__ void __launch_bounds__(kThreads, 1)
splitkv_partial_kernel(const __grid_constant__ CUtensorMap tmK, const __grid_constant__ CUtensorMap tmV,
                       const SplitParams p) {
  using G = Cfg<D>;
  using S = Smem<D, NQ>;
  constexpr int kStages = S::kStages;
  constexpr int C = G::C;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  float* wo = reinterpret_cast<float*>(smem + S::kWo);
  float* qs = reinterpret_cast<float*>(smem + S::kQs);
  float* wm = reinterpret_cast<float*>(smem + S::kWm);
  float* wl = reinterpret_cast<float*>(smem + S::kWl);
  uint64_t* full = reinterpret_cast<uint64_t*>(smem + S::kBar);
  uint64_t* empty = full + kStages;
  volatile int* abort = reinterpret_cast<volatile int*>(smem + S::kAbort);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  if (threadIdx.x == 0) {
    for (int s = 0; s < kStages; ++s) {
      ptx::mbar_init(&full[s], 1);
      ptx::mbar_init(&empty[s], 1);
    }
    *abort = 0;
    ptx::fence_mbar_init();
  }
  __syncthreads();

  const int64_t g_begin = (int64_t)blockIdx.x * p.L;
  const int64_t g_end = min(p.total, g_begin + p.L);
  const int nq = p.nq;
  int issued = 0;

  if (warp == kConsumerWarps) {
    // ---------------------------------------------------------------- producer
    if (lane == 0) {
      ptx::prefetch_tmap(&tmK);
      ptx::prefetch_tmap(&tmV);
      bool ok = true;
      int seq = 0;
      for (int64_t g = g_begin; g < g_end && ok;) {
        const int64_t h = g / p.Nk;
        const int k0 = (int)(g - h * p.Nk);
        const int k1 = (int)(k0 + (g_end - g) < (int64_t)p.Nk ? k0 + (g_end - g) : p.Nk);
        for (int kt = k0; kt < k1; kt += kTileKeys, ++seq) {
          const int b = seq % kStages;
          if (seq >= kStages && !(ok = ptx::mbar_wait(&empty[b], ((seq / kStages) - 1) & 1, p.status, abort)))
            break;
          uint8_t* st = smem + b * G::kStageBytes;
          ptx::mbar_expect_tx(&full[b], G::kStageBytes);
#pragma unroll
          for (int x = 0; x < G::kBoxes; ++x) {
            ptx::tma_load_3d(st + x * G::kBoxBytes, &tmK, &full[b], x * 64, kt, (int)h);
            ptx::tma_load_3d(st + G::kTileBytes + x * G::kBoxBytes, &tmV, &full[b], x * 64, kt, (int)h);
          }
        }
        g += k1 - k0;
      }
      issued = seq;
    }
  } else {
    // ---------------------------------------------------------------- consumers
    float* ps = reinterpret_cast<float*>(smem + S::kPs) + warp * kTileKeys * NQ;
    bool ok = true;
    int seq = 0;
    for (int64_t g = g_begin; g < g_end;) {
      const int64_t h = g / p.Nk;
      const int k0 = (int)(g - h * p.Nk);
      const int k1 = (int)(k0 + (g_end - g) < (int64_t)p.Nk ? k0 + (g_end - g) : p.Nk);
      for (int e = threadIdx.x; e < NQ * D; e += kConsumerWarps * 32) {
        const int qi = e / D;
        qs[e] = qi < nq ? __bfloat162float(p.Q[(h * nq + qi) * D + e % D]) * p.sl2 : 0.f;
      }
      consumers_sync();
      float qr[NQ == 1 ? D : 1];  // the single query lives in registers
      if constexpr (NQ == 1) {
#pragma unroll
        for (int c = 0; c < D; ++c) qr[c] = qs[c];
      }
      float m[NQ], lsum[NQ], acc[NQ][C];
#pragma unroll
      for (int qi = 0; qi < NQ; ++qi) {
        m[qi] = -INFINITY;
        lsum[qi] = 0.f;
#pragma unroll
        for (int c = 0; c < C; ++c) acc[qi][c] = 0.f;
      }

      for (int kt = k0; kt < k1; kt += kTileKeys, ++seq) {
        if ((seq & (kConsumerWarps - 1)) != warp) continue;
        const int b = seq % kStages;
        if (ok) ok = __all_sync(0xffffffffu, ptx::mbar_wait(&full[b], (seq / kStages) & 1, p.status, abort));
        if (!ok) continue;
        const uint8_t* ks = smem + b * G::kStageBytes;
        const uint8_t* vs = ks + G::kTileBytes;

        // s = q . k for this lane's key, its row read in 16-byte chunks (chunk c of row r
        // sits at chunk position c ^ (r % 8) of the row's 128-byte line)
        float s[NQ];
#pragma unroll
        for (int qi = 0; qi < NQ; ++qi) s[qi] = 0.f;
#pragma unroll(NQ == 1 ? D / 8 : 2)  // q of a single query is indexed statically
        for (int c = 0; c < D / 8; ++c) {
          const uint4 u = *reinterpret_cast<const uint4*>(ks + (c >> 3) * G::kBoxBytes + lane * 128 +
                                                          (((c & 7) ^ (lane & 7)) << 4));
          const __nv_bfloat162* hv = reinterpret_cast<const __nv_bfloat162*>(&u);
          float kf[8];
#pragma unroll
          for (int t = 0; t < 4; ++t) {
            const float2 f = __bfloat1622float2(hv[t]);
            kf[2 * t] = f.x;
            kf[2 * t + 1] = f.y;
          }
          if constexpr (NQ == 1) {
#pragma unroll
            for (int t = 0; t < 8; ++t) s[0] = fmaf(qr[c * 8 + t], kf[t], s[0]);
          } else {
#pragma unroll
            for (int qi = 0; qi < NQ; ++qi)
              if (qi < nq) {
                const float4 a = *reinterpret_cast<const float4*>(qs + qi * D + c * 8);
                const float4 bq = *reinterpret_cast<const float4*>(qs + qi * D + c * 8 + 4);
                s[qi] = fmaf(a.x, kf[0], s[qi]);
                s[qi] = fmaf(a.y, kf[1], s[qi]);
                s[qi] = fmaf(a.z, kf[2], s[qi]);
                s[qi] = fmaf(a.w, kf[3], s[qi]);
                s[qi] = fmaf(bq.x, kf[4], s[qi]);
                s[qi] = fmaf(bq.y, kf[5], s[qi]);
                s[qi] = fmaf(bq.z, kf[6], s[qi]);
                s[qi] = fmaf(bq.w, kf[7], s[qi]);
              }
          }
        }

        // online softmax over the warp's 32 keys; p goes to shared memory for p.V
        const int key = kt + lane;
        const bool valid = key < k1;
#pragma unroll
        for (int qi = 0; qi < NQ; ++qi) {
          float pq = 0.f;
          if (qi < nq) {
            const bool vis = valid && !(p.causal && key > qi + p.offset);
            const float sv = vis ? s[qi] : -INFINITY;
            const float mnew = fmaxf(m[qi], wmax(sv));
            if (mnew != -INFINITY) {  // warp-uniform: some key so far is visible to this query
              const float corr = ptx::ex2(m[qi] - mnew);
              pq = vis ? ptx::ex2(sv - mnew) : 0.f;
              lsum[qi] = fmaf(lsum[qi], corr, pq);
#pragma unroll
              for (int c = 0; c < C; ++c) acc[qi][c] *= corr;
              m[qi] = mnew;
            }
          }
          ps[lane * NQ + qi] = pq;
        }
        __syncwarp();

        // O += p V over the tile's keys; lane owns columns lane*C .. lane*C + C - 1
        const int kend = min(kTileKeys, k1 - kt);
        const int vbox = (lane * C) / 64;
        const int vbyte = (lane * C * 2) & 127;  // byte offset inside the 128-byte line
        const uint8_t* vcol = vs + vbox * G::kBoxBytes + (vbyte & 15);
        const int vchunk = vbyte >> 4;
#pragma unroll 4
        for (int kk = 0; kk < kend; ++kk) {
          const uint8_t* vrow = vcol + kk * 128 + ((vchunk ^ (kk & 7)) << 4);
          float vf[C];
          if constexpr (C == 4) {
            const uint2 u = *reinterpret_cast<const uint2*>(vrow);
            const float2 a = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&u.x));
            const float2 bb = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&u.y));
            vf[0] = a.x, vf[1] = a.y, vf[2] = bb.x, vf[3] = bb.y;
          } else {
            const float2 a = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(vrow));
            vf[0] = a.x, vf[1] = a.y;
          }
          float pk[NQ];
          if constexpr (NQ == 1) {
            pk[0] = ps[kk];
          } else {
#pragma unroll
            for (int j = 0; j < NQ; j += 4) {
              const float4 t = *reinterpret_cast<const float4*>(ps + kk * NQ + j);
              pk[j] = t.x, pk[j + 1] = t.y, pk[j + 2] = t.z, pk[j + 3] = t.w;
            }
          }
#pragma unroll
          for (int qi = 0; qi < NQ; ++qi)
            if (qi < nq) {
#pragma unroll
              for (int c = 0; c < C; ++c) acc[qi][c] = fmaf(pk[qi], vf[c], acc[qi][c]);
            }
        }
        __syncwarp();  // every lane is done with this stage and with ps
        if (lane == 0) ptx::mbar_arrive(&empty[b]);
      }

      // end of the segment: merge the four warps' states and write this CTA's slot
#pragma unroll
      for (int qi = 0; qi < NQ; ++qi) {
        const float l = wsum(lsum[qi]);
        if (lane == 0) {
          wm[warp * NQ + qi] = m[qi];
          wl[warp * NQ + qi] = l;
        }
#pragma unroll
        for (int c = 0; c < C; ++c) wo[(warp * NQ + qi) * D + lane * C + c] = acc[qi][c];
      }
      consumers_sync();
      const int slot = (int)(blockIdx.x - (h * p.Nk) / p.L);
      const int64_t base = (h * p.P + slot) * nq;
      for (int e = threadIdx.x; e < nq * D; e += kConsumerWarps * 32) {
        const int qi = e / D, col = e % D;
        float M = -INFINITY;
#pragma unroll
        for (int w = 0; w < kConsumerWarps; ++w) M = fmaxf(M, wm[w * NQ + qi]);
        float o = 0.f, l = 0.f;
        if (M != -INFINITY) {
#pragma unroll
          for (int w = 0; w < kConsumerWarps; ++w) {
            const float f = ptx::ex2(wm[w * NQ + qi] - M);
            o = fmaf(wo[(w * NQ + qi) * D + col], f, o);
            l = fmaf(wl[w * NQ + qi], f, l);
          }
        }
        p.part_o[(base + qi) * D + col] = o;
        if (col == 0) {
          p.part_ml[(base + qi) * 2] = M;
          p.part_ml[(base + qi) * 2 + 1] = l;
        }
      }
      consumers_sync();  // wo, wm, wl and qs are reused by the next segment
      g += k1 - k0;
    }
  }

  __syncthreads();
  // After a failed wait, let the copies still in flight land before the CTA's shared
  // memory is released (bounded waits, no abort: these copies were issued).
  if (warp == kConsumerWarps && lane == 0 && *abort) {
    for (int seq = max(0, issued - kStages); seq < issued; ++seq)
      ptx::mbar_wait(&full[seq % kStages], (seq / kStages) & 1, p.status, nullptr);
  }
}

// One warp per (head, query): merge the head's partial states and write O (bf16) and LSE.
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

template <int D, int NQ>
cudaError_t launch_partial(const CUtensorMap& mk, const CUtensorMap& mv, const SplitParams& p, int ctas,
                           cudaStream_t st) {
  using S = Smem<D, NQ>;
  static_assert(S::kAlloc <= 227 * 1024, "shared memory budget");
  static const bool attr = cudaFuncSetAttribute(splitkv_partial_kernel<D, NQ>,
                                                cudaFuncAttributeMaxDynamicSharedMemorySize,
                                                S::kAlloc) == cudaSuccess;
  if (!attr) return cudaErrorInvalidConfiguration;
  splitkv_partial_kernel<D, NQ><<<ctas, kThreads, S::kAlloc, st>>>(mk, mv, p);
  return cudaGetLastError();
}

template <int D>
cudaError_t launch_d(const CUtensorMap& mk, const CUtensorMap& mv, const SplitParams& p, int ctas,
                     cudaStream_t st) {
  if (p.nq == 1) return launch_partial<D, 1>(mk, mv, p, ctas, st);
  if (p.nq <= 4) return launch_partial<D, 4>(mk, mv, p, ctas, st);
  if (p.nq <= 8) return launch_partial<D, 8>(mk, mv, p, ctas, st);
  return launch_partial<D, 16>(mk, mv, p, ctas, st);
}

}  // namespace

size_t splitkv_workspace_floats(int64_t heads, int Nq, int Nk, int d) {
  return (size_t)layout(heads, Nk).P * heads * Nq * (d + 2);
}

cudaError_t splitkv_fwd(const void* Q, const void* K, const void* V, void* O, float* LSE, int64_t heads,
                        int Nq, int Nk, int d, float scale, bool causal, float* workspace, int* status,
                        cudaStream_t st) {
  const Layout lay = layout(heads, Nk);
  SplitParams p;
  p.Q = static_cast<const __nv_bfloat16*>(Q);
  p.total = heads * Nk;
  p.L = lay.L;
  p.nq = Nq;
  p.Nk = Nk;
  p.P = lay.P;
  p.causal = causal ? 1 : 0;
  p.offset = Nk - Nq;
  p.sl2 = scale * 1.4426950408889634f;
  p.status = status;
  p.part_o = workspace;
  p.part_ml = workspace + (size_t)lay.P * heads * Nq * d;
  cudaError_t e;
  if (d == 128) {  // the tensor-core partial kernel (same partial states)
    e = splitkv_tc_partial(Q, K, V, heads, Nq, Nk, scale, causal, workspace, status, st);
  } else {
    CUtensorMap mk, mv;
    if (!make_map_bf16_3d(&mk, K, heads, Nk, d, kTileKeys) || !make_map_bf16_3d(&mv, V, heads, Nk, d, kTileKeys))
      return cudaErrorInvalidValue;
    e = launch_d<64>(mk, mv, p, lay.ctas, st);
  }
  if (e != cudaSuccess) return e;
  const int64_t rows = heads * Nq;
  const unsigned grid = (unsigned)((rows + 3) / 4);
  if (d == 64)
    splitkv_merge_kernel<64><<<grid, 128, 0, st>>>(p.part_o, p.part_ml, static_cast<__nv_bfloat16*>(O), LSE, rows,
                                                   Nq, Nk, lay.L, lay.P);
  else
    splitkv_merge_kernel<128><<<grid, 128, 0, st>>>(p.part_o, p.part_ml, static_cast<__nv_bfloat16*>(O), LSE,
                                                    rows, Nq, Nk, lay.L, lay.P);
  return cudaGetLastError();
}

}  // namespace fa
