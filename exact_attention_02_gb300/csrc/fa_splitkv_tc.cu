// Split-KV forward on the tensor cores, for 2..64 queries against a long key/value
// sequence (d = 128): the same partial states and merge as fa_splitkv.cu, with the two
// products of each 128-key tile on tcgen05.
//
// Work split: as in fa_splitkv.cu, one CTA per SM takes an equal contiguous range of the
// flattened (head, key) sequence; each piece of a head inside the range is a segment with
// its own partial state (m, l, O) per query, merged afterwards by splitkv_merge_kernel.
//
// Per 128-key tile (keys on the MMA's M side, queries on N, padded to 64 with zero rows):
//   S^T = K Q^T           M = 128 keys, N = 64, K = d: one TMEM accumulator [keys x queries]
//   softmax               4 warps, one thread per key (= TMEM lane): scores in log2 units,
//                         masked keys -inf; per query a running max m_q, refreshed only when
//                         some score exceeds it by more than 2^8 (then O^T and the row sums
//                         are rescaled); p = 2^(s - m_q) <= 256 written as bf16 P^T rows to
//                         a 128-byte-swizzled shared-memory tile
//   O^T += V^T P^T        M = 128 (d), N = 64, K = 128 keys: A = the V tile read MN-major,
//                         B = P^T (MN-major), accumulator O^T [d x queries] in TMEM
// Row sums stay per thread (64 partial sums) and are reduced once per segment. An N = 64
// product costs the same issue slot as N = 16, so the padding costs nothing.
//
// Roles: warps 0-3 softmax and epilogue, warp 4 TMA producer, warp 5 MMA issuer.
// Rows: K/V through 3-D maps [heads, N_k, d] (rows past the end of a head read as zeros),
// Q through [heads, N_q, d] with 64-row boxes (rows past N_q read as zeros).
#include <cuda_bf16.h>

#include <algorithm>

#include "fa_internal.h"
#include "sm100_ptx.cuh"
#include "tma_host.h"

namespace fa {
namespace {

using namespace ptx;

constexpr int kCtas = 152;
constexpr int kMinKeys = 256;
constexpr int BN = 128;  // keys per tile
constexpr int D = 128;
constexpr int NQP = 64;  // queries padded to the MMA's N
constexpr int kThreads = 192;
constexpr int kLoadWarp = 4, kMmaWarp = 5;
constexpr float kThreshold = 8.f;

constexpr int kBoxBytes = BN * 128;           // [128 rows x 64 bf16]
constexpr int kTileBytes = 2 * kBoxBytes;     // one K or V tile (d = 128)
constexpr int kQBox = NQP * 128;              // [64 rows x 64 bf16]
constexpr int kQBytes = 2 * kQBox;
constexpr int kPBytes = BN * NQP * 2;         // P^T [128 keys x 64 queries] bf16
constexpr int kKStages = 3, kVStages = 2;  // K is read a tile before V, so it gets the deeper ring
constexpr int kKOff = 0;
constexpr int kVOff = kKOff + kKStages * kTileBytes;
constexpr int kQOff = kVOff + kVStages * kTileBytes;
constexpr int kPOff = kQOff + kQBytes;
constexpr int kCorrOff = kPOff + 2 * kPBytes;       // float[64] rescale factors
constexpr int kMOff = kCorrOff + 4 * NQP;           // float[64] running max per query (log2 units)
constexpr int kRedOff = kMOff + 4 * NQP;            // float[4][64] cross-warp scratch
constexpr int kFlagOff = kRedOff + 4 * 4 * NQP;     // int[2][4] per-warp flags, by tile parity
constexpr int kSmemBytes = kFlagOff + 32 + 1024;
static_assert(kSmemBytes <= 227 * 1024, "shared memory");

constexpr uint32_t kColS0 = 0, kColO = 2 * NQP;  // S buffers [0,128), O^T [128,192)
constexpr uint32_t kTmemCols = 256;

struct Layout {
  int64_t L;
  int ctas;
  int P;
};
Layout layout(int64_t heads, int Nk) {
  const int64_t total = heads * Nk;
  int64_t L = std::max<int64_t>((total + kCtas - 1) / kCtas, kMinKeys);
  L = (L + 31) / 32 * 32;
  Layout r;
  r.L = L;
  r.ctas = (int)((total + L - 1) / L);
  r.P = (int)((Nk + L - 1) / L) + 1;
  return r;
}

struct TcParams {
  float* part_o;   // [heads][P][nq][D]
  float* part_ml;  // [heads][P][nq][2]
  int64_t total, L;
  int nq, Nk, P, causal, offset;
  float sl2;
  int* status;
};

struct Ctl {
  uint64_t k_full[kKStages], v_full[kVStages], k_empty[kKStages], v_empty[kVStages];
  uint64_t q_full, q_empty, s_full[2], p_full[2], pv_done[2], o_free, drain;
  uint32_t tmem_base;
  int abort;
};

__device__ __forceinline__ void softmax_sync() { asm volatile("bar.sync 1, 128;" ::: "memory"); }

// Segment iteration shared by every role: segment (head h, keys [k0, k1)).
struct SegIter {
  int64_t g, g_end, Nk;
  __device__ bool next(int64_t& h, int& k0, int& k1) {
    if (g >= g_end) return false;
    h = g / Nk;
    k0 = (int)(g - h * Nk);
    const int64_t rem = g_end - g;
    k1 = (int)(k0 + rem < Nk ? k0 + rem : Nk);
    g += k1 - k0;
    return true;
  }
};

__global__ void __launch_bounds__(kThreads, 1)
splitkv_tc_kernel(const __grid_constant__ CUtensorMap tmK, const __grid_constant__ CUtensorMap tmV,
                  const __grid_constant__ CUtensorMap tmQ, const TcParams p) {
  extern __shared__ uint8_t smem_raw[];
  __shared__ Ctl ctl;
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int64_t g_begin = (int64_t)blockIdx.x * p.L;
  const int64_t g_end = min(p.total, g_begin + p.L);

  if (threadIdx.x == 0) {
    for (int s = 0; s < kKStages; ++s) {
      mbar_init(&ctl.k_full[s], 1);
      mbar_init(&ctl.k_empty[s], 1);
    }
    for (int s = 0; s < kVStages; ++s) {
      mbar_init(&ctl.v_full[s], 1);
      mbar_init(&ctl.v_empty[s], 1);
    }
    mbar_init(&ctl.q_full, 1);
    mbar_init(&ctl.q_empty, 1);
    for (int b = 0; b < 2; ++b) {
      mbar_init(&ctl.s_full[b], 1);
      mbar_init(&ctl.p_full[b], 4);  // one arrival per softmax warp
    }
    mbar_init(&ctl.pv_done[0], 1);
    mbar_init(&ctl.pv_done[1], 1);
    mbar_init(&ctl.o_free, 4);
    mbar_init(&ctl.drain, 1);
    ctl.abort = 0;
    fence_mbar_init();
  }
  if (warp == kMmaWarp) tmem_alloc(&ctl.tmem_base, kTmemCols);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = ctl.tmem_base;
  volatile int* abort = &ctl.abort;

  if (warp == kLoadWarp) {
    // ---------------------------------------------------------------- TMA producer
    // Lane 0 streams Q and K, lane 1 streams V: a K slot frees a tile before the V slot of
    // the same tile, so the two rings advance independently.
    if (lane < 2) {
      const bool kq = lane == 0;
      if (kq) {
        prefetch_tmap(&tmK);
        prefetch_tmap(&tmQ);
      } else {
        prefetch_tmap(&tmV);
      }
      constexpr int kMaxStages = kKStages > kVStages ? kKStages : kVStages;
      const int stages = kq ? kKStages : kVStages;
      uint64_t* full = kq ? ctl.k_full : ctl.v_full;
      uint64_t* empty = kq ? ctl.k_empty : ctl.v_empty;
      const CUtensorMap* map = kq ? &tmK : &tmV;
      uint8_t* ring = smem + (kq ? kKOff : kVOff);
      SegIter it{g_begin, g_end, p.Nk};
      int64_t h;
      int k0, k1, seg = 0, t = 0, last[kMaxStages], last_q = -1;
      for (int s = 0; s < kMaxStages; ++s) last[s] = -1;
      bool ok = true;
      while (ok && it.next(h, k0, k1)) {
        if (kq) {  // Q of this head, once the previous segment's S products have read the old one
          if (seg > 0 && !(ok = mbar_wait(&ctl.q_empty, (seg - 1) & 1, p.status, abort))) break;
          mbar_expect_tx(&ctl.q_full, kQBytes);
          for (int b = 0; b < 2; ++b) tma_load_3d(smem + kQOff + b * kQBox, &tmQ, &ctl.q_full, b * 64, 0, (int)h);
          last_q = seg;
        }
        for (int kt = k0; ok && kt < k1; kt += BN, ++t) {
          const int s = t % stages;
          if (t >= stages && !(ok = mbar_wait(&empty[s], ((t / stages) - 1) & 1, p.status, abort))) break;
          mbar_expect_tx(&full[s], kTileBytes);
          for (int b = 0; b < 2; ++b)
            tma_load_3d(ring + s * kTileBytes + b * kBoxBytes, map, &full[s], b * 64, kt, (int)h);
          last[s] = t;
        }
        ++seg;
      }
      // every issued copy lands before the CTA may exit
      if (last_q >= 0) mbar_wait(&ctl.q_full, last_q & 1, p.status, nullptr);
      for (int s = 0; s < stages; ++s)
        if (last[s] >= 0) mbar_wait(&full[s], (last[s] / stages) & 1, p.status, nullptr);
    }
  } else if (warp == kMmaWarp) {
    // ---------------------------------------------------------------- MMA issuer
    if (lane == 0) {
      constexpr uint32_t idS = idesc_bf16(BN, NQP, false, false);  // S^T: A = K, B = Q, both K-major
      constexpr uint32_t idO = idesc_bf16(D, NQP, true, true);     // O^T: A = V^T, B = P^T, MN-major
      const uint64_t dK0 = sdesc_sw128(smem_u32(smem + kKOff), 16, 1024);
      const uint64_t dQ0 = sdesc_sw128(smem_u32(smem + kQOff), 16, 1024);
      const uint64_t dV0 = sdesc_sw128(smem_u32(smem + kVOff), kBoxBytes, 1024);
      const uint64_t dP0 = sdesc_sw128(smem_u32(smem + kPOff), kPBytes, 1024);
      auto issue_S = [&](int t) {
        const uint32_t ko = (t % kKStages) * kTileBytes;
#pragma unroll
        for (int k = 0; k < D / 16; ++k) {
          const uint32_t off = (k / 4) * kBoxBytes + (k % 4) * 32, qoff = (k / 4) * kQBox + (k % 4) * 32;
          mma_ss(tmem + kColS0 + (t & 1) * NQP, sdesc_add(dK0, ko + off), sdesc_add(dQ0, qoff), idS, k > 0);
        }
      };
      auto issue_PV = [&](int t, bool acc) {
        const uint32_t vo = (t % kVStages) * kTileBytes, po = (t & 1) * kPBytes;
#pragma unroll
        for (int k = 0; k < BN / 16; ++k)
          mma_ss(tmem + kColO, sdesc_add(dV0, vo + k * 2048), sdesc_add(dP0, po + k * 2048), idO,
                 (acc || k > 0) ? 1u : 0u);
      };
      SegIter it{g_begin, g_end, p.Nk};
      int64_t h;
      int k0, k1, seg = 0, t = 0;
      bool ok = true;
      while (ok && it.next(h, k0, k1)) {
        const int n = (k1 - k0 + BN - 1) / BN;  // tiles in this segment: t .. t + n - 1
        if (!(ok = mbar_wait(&ctl.q_full, seg & 1, p.status, abort))) break;
        if (!(ok = mbar_wait(&ctl.k_full[t % kKStages], (t / kKStages) & 1, p.status, abort))) break;
        tc_fence_after();
        issue_S(t);
        mma_commit(&ctl.k_empty[t % kKStages]);
        mma_commit(&ctl.s_full[t & 1]);
        for (int i = 0; i < n; ++i, ++t) {
          if (i + 1 < n) {  // S of the next tile into the other buffer (read out by tile t-1's softmax)
            if (t >= 1 && !(ok = mbar_wait(&ctl.p_full[(t + 1) & 1], ((t - 1) >> 1) & 1, p.status, abort))) break;
            if (!(ok = mbar_wait(&ctl.k_full[(t + 1) % kKStages], ((t + 1) / kKStages) & 1, p.status, abort)))
              break;
            tc_fence_after();
            issue_S(t + 1);
            mma_commit(&ctl.k_empty[(t + 1) % kKStages]);
            mma_commit(&ctl.s_full[(t + 1) & 1]);
          } else {
            mma_commit(&ctl.q_empty);  // every S of the segment is issued: Q may be replaced
          }
          if (!(ok = mbar_wait(&ctl.p_full[t & 1], (t >> 1) & 1, p.status, abort))) break;
          if (!(ok = mbar_wait(&ctl.v_full[t % kVStages], (t / kVStages) & 1, p.status, abort))) break;
          if (i == 0 && seg > 0 && !(ok = mbar_wait(&ctl.o_free, (seg - 1) & 1, p.status, abort))) break;
          tc_fence_after();
          issue_PV(t, i > 0);
          mma_commit(&ctl.v_empty[t % kVStages]);
          mma_commit(&ctl.pv_done[t & 1]);
        }
        ++seg;
      }
      // every MMA retires before TMEM is released
      mma_commit(&ctl.drain);
      mbar_wait(&ctl.drain, 0, p.status, nullptr);
    }
  } else {
    // ---------------------------------------------------------------- softmax + epilogue
    const int r = warp * 32 + lane;  // TMEM lane: key of the tile in S^T, head-dim row in O^T
    const uint32_t lane_off = (uint32_t)(warp * 32) << 16;
    float* corr = reinterpret_cast<float*>(smem + kCorrOff);
    float* mrow = reinterpret_cast<float*>(smem + kMOff);  // uniform over the threads
    float* red = reinterpret_cast<float*>(smem + kRedOff);
    int* flags = reinterpret_cast<int*>(smem + kFlagOff);
    const int nq = p.nq;
    SegIter it{g_begin, g_end, p.Nk};
    int64_t h;
    int k0, k1, t = 0;
    bool ok = true;
    // After a failed (timed-out) wait the loops keep their shape, skipping the waits and the
    // TMEM accesses, so that every softmax warp still reaches every named barrier.
    while (it.next(h, k0, k1)) {
      const int n = (k1 - k0 + BN - 1) / BN;
      if (r < NQP) mrow[r] = -INFINITY;
      float l[NQP];
#pragma unroll
      for (int q = 0; q < NQP; ++q) l[q] = 0.f;
      softmax_sync();
      for (int i = 0; i < n; ++i, ++t) {
        if (ok) ok = __all_sync(0xffffffffu, mbar_wait(&ctl.s_full[t & 1], (t >> 1) & 1, p.status, abort));
        float x[NQP];
        if (ok) {
          tc_fence_after();
          tmem_ld32x2(tmem + lane_off + kColS0 + (t & 1) * NQP, tmem + lane_off + kColS0 + (t & 1) * NQP + 32,
                      *reinterpret_cast<float(*)[32]>(&x[0]), *reinterpret_cast<float(*)[32]>(&x[32]));
        } else {
#pragma unroll
          for (int q = 0; q < NQP; ++q) x[q] = 0.f;
        }
        const int key = k0 + i * BN + r;
        const bool kin = key < k1;
        bool grow = false;
#pragma unroll
        for (int q = 0; q < NQP; ++q) {
          const bool vis = ok && kin && q < nq && !(p.causal && key > q + p.offset);
          x[q] = vis ? x[q] * p.sl2 : -INFINITY;
          grow |= x[q] > mrow[q] + kThreshold;
        }
        // does any score of the tile exceed its query's reference max by the threshold?
        grow = __any_sync(0xffffffffu, grow);
        int* fl = flags + (t & 1) * 4;
        if (lane == 0) fl[warp] = grow ? 1 : 0;
        softmax_sync();
        if ((fl[0] | fl[1] | fl[2] | fl[3]) != 0) {  // uniform over the four warps
          // exact column maxima of the tile: warp reduction, then across the warps
#pragma unroll
          for (int q = 0; q < NQP; ++q) {
            float v = x[q];
#pragma unroll
            for (int o = 16; o; o >>= 1) v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, o));
            if (lane == 0) red[warp * NQP + q] = v;
          }
          softmax_sync();
          if (r < NQP) {
            const float mx = fmaxf(fmaxf(red[r], red[NQP + r]), fmaxf(red[2 * NQP + r], red[3 * NQP + r]));
            const float mo = mrow[r], mn = fmaxf(mo, mx);
            corr[r] = mn > mo ? ex2(mo - mn) : 1.f;  // mo = -inf gives 0: nothing accumulated yet
            mrow[r] = mn;
          }
          softmax_sync();
#pragma unroll
          for (int q = 0; q < NQP; ++q) l[q] *= corr[q];
          if (i > 0 && ok) {
            // O^T (lane = head-dim row) is rescaled once the previous tile's PV has finished
            ok = __all_sync(0xffffffffu,
                            mbar_wait(&ctl.pv_done[(t - 1) & 1], ((t - 1) >> 1) & 1, p.status, abort));
            if (ok) {
              tc_fence_after();
              float ov[NQP];
              tmem_ld32x2(tmem + lane_off + kColO, tmem + lane_off + kColO + 32,
                          *reinterpret_cast<float(*)[32]>(&ov[0]), *reinterpret_cast<float(*)[32]>(&ov[32]));
#pragma unroll
              for (int c = 0; c < NQP; c += 16) {
                uint32_t w[16];
#pragma unroll
                for (int u = 0; u < 16; ++u) w[u] = __float_as_uint(ov[c + u] * corr[c + u]);
                tmem_st16(tmem + lane_off + kColO + c, w);
              }
              tmem_wait_st();
            }
          }
        }
        // The P^T buffer of this tile was last read by PV(t - 2).
        if (t >= 2 && ok)
          ok = __all_sync(0xffffffffu, mbar_wait(&ctl.pv_done[t & 1], ((t - 2) >> 1) & 1, p.status, abort));
        // p = 2^(x - m) <= 2^threshold; P^T row r of the tile: 128 bytes, 128-byte swizzle
        uint8_t* prow = smem + kPOff + (t & 1) * kPBytes + r * 128;
#pragma unroll
        for (int c = 0; c < NQP / 8; ++c) {
          uint32_t w[4];
#pragma unroll
          for (int u = 0; u < 4; ++u) {
            const int q = c * 8 + 2 * u;
            const float m0 = mrow[q], m1 = mrow[q + 1];
            const float p0 = ex2(x[q] - (m0 == -INFINITY ? 0.f : m0));
            const float p1 = ex2(x[q + 1] - (m1 == -INFINITY ? 0.f : m1));
            l[q] += p0;
            l[q + 1] += p1;
            w[u] = pack_bf16(p0, p1);
          }
          *reinterpret_cast<uint4*>(prow + ((c ^ (r & 7)) << 4)) = make_uint4(w[0], w[1], w[2], w[3]);
        }
        fence_proxy_async_smem();
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(&ctl.p_full[t & 1]);
      }
      // ---- end of segment: reduce the row sums, read O^T, write this CTA's partial state
      const int tl = t - 1;  // the segment's last tile
      if (ok) ok = __all_sync(0xffffffffu, mbar_wait(&ctl.pv_done[tl & 1], (tl >> 1) & 1, p.status, abort));
#pragma unroll
      for (int q = 0; q < NQP; ++q) {
        float v = l[q];
#pragma unroll
        for (int o = 16; o; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
        if (lane == 0) red[warp * NQP + q] = v;
      }
      softmax_sync();
      const int slot = (int)(blockIdx.x - (h * p.Nk) / p.L);
      const int64_t base = (h * p.P + slot) * nq;
      if (r < nq) {
        p.part_ml[(base + r) * 2] = mrow[r];
        p.part_ml[(base + r) * 2 + 1] = red[r] + red[NQP + r] + red[2 * NQP + r] + red[3 * NQP + r];
      }
      if (ok) {
        tc_fence_after();
        float ov[NQP];
        tmem_ld32x2(tmem + lane_off + kColO, tmem + lane_off + kColO + 32, *reinterpret_cast<float(*)[32]>(&ov[0]),
                    *reinterpret_cast<float(*)[32]>(&ov[32]));
#pragma unroll
        for (int q = 0; q < NQP; ++q)
          if (q < nq) p.part_o[(base + q) * D + r] = ov[q];
      }
      tc_fence_before();
      softmax_sync();  // red[], mrow[] and O^T are free for the next segment
      if (lane == 0) mbar_arrive(&ctl.o_free);
    }
  }

  tc_fence_before();
  __syncthreads();
  if (warp == kMmaWarp) {
    tc_fence_after();
    tmem_dealloc(tmem, kTmemCols);
  }
}

}  // namespace

size_t splitkv_tc_workspace_floats(int64_t heads, int Nq, int Nk) {
  return (size_t)layout(heads, Nk).P * heads * Nq * (D + 2);
}

int splitkv_tc_partials(int64_t heads, int Nk, int64_t* L) {
  const Layout lay = layout(heads, Nk);
  *L = lay.L;
  return lay.P;
}

cudaError_t splitkv_tc_partial(const void* Q, const void* K, const void* V, int64_t heads, int Nq, int Nk,
                               float scale, bool causal, float* workspace, int* status, cudaStream_t st) {
  const Layout lay = layout(heads, Nk);
  CUtensorMap mk, mv, mq;
  if (!make_map_bf16_3d(&mk, K, heads, Nk, D, BN) || !make_map_bf16_3d(&mv, V, heads, Nk, D, BN) ||
      !make_map_bf16_3d(&mq, Q, heads, Nq, D, NQP))
    return cudaErrorInvalidValue;
  static const bool attr =
      cudaFuncSetAttribute(splitkv_tc_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, kSmemBytes) ==
      cudaSuccess;
  if (!attr) return cudaErrorInvalidConfiguration;
  TcParams p;
  p.part_o = workspace;
  p.part_ml = workspace + (size_t)lay.P * heads * Nq * D;
  p.total = heads * Nk;
  p.L = lay.L;
  p.nq = Nq;
  p.Nk = Nk;
  p.P = lay.P;
  p.causal = causal ? 1 : 0;
  p.offset = Nk - Nq;
  p.sl2 = scale * 1.4426950408889634f;
  p.status = status;
  splitkv_tc_kernel<<<lay.ctas, kThreads, kSmemBytes, st>>>(mk, mv, mq, p);
  return cudaGetLastError();
}

}  // namespace fa
