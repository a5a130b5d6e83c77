// Split-KV forward on the tensor cores, for 1..64 queries against a long key/value
// sequence (d = 64 or 128): the same partial states and merge as fa_splitkv.cu, with the
// two products of each key tile on tcgen05.
//
// Work split (chosen by fa_splitkv.cu): one CTA per SM takes an equal contiguous range of L
// keys of the flattened (head, key) sequence; each piece of a head inside the range is a
// segment with its own partial state (m, l, O) per query, stored in slot (head, CTA - first
// CTA of the head) and merged afterwards by splitkv_merge_kernel.
//
// Per 128 keys of a tile (keys on the MMA's M side, queries on N, padded to 64 with zero rows):
//   S^T = K Q^T           M = 128 keys, N = 64, K = d: one TMEM accumulator [keys x queries]
//   softmax               one thread per (key = TMEM lane, query group): scores in log2
//                         units, masked keys -inf; per query a running max m_q, refreshed
//                         only when some score exceeds it by more than 2^8 (then O^T and the
//                         row sums are rescaled); p = 2^(s - m_q) <= 256 written as bf16 P^T
//                         rows to a 128-byte-swizzled shared-memory tile. m_q starts at the
//                         finite -1e30, so no score needs a test for -inf: the first visible
//                         score always triggers a refresh, and a masked one gives 2^-inf = 0.
//                         A tile that no key bound or causal rule touches for the group skips
//                         the masking altogether.
//   O^T += V^T P^T        M = 128 (d), N = 64, K = 128 keys: A = the V tile read MN-major,
//                         B = P^T (MN-major), accumulator O^T [d x queries] in TMEM
// Row sums stay per thread (64 partial sums) and are reduced once per segment. An N = 64
// product costs the same issue slot as N = 16, so the padding costs nothing.
//
// Roles: warps 0-7 softmax and epilogue, warp 8 TMA producer (lane 0 Q and K, lane 1 V),
// warp 9 MMA issuer. The softmax warps form two groups of four; group g owns the query
// columns g*C .. g*C + C - 1 (C = 8, 16 or 32, the smallest with 2C >= N_q), keeps their
// running maxima and synchronises on its own named barrier. Warp w reads TMEM lanes
// 32*(w%4)..+31, so both groups see every key. A group without queries sits out, and the
// barriers it would arrive on count only the groups that have queries.
// Rows: K/V through 3-D maps [heads, N_k, d] (rows past the end of a head read as zeros),
// Q through [heads, N_q, d] with 64-row boxes (rows past N_q read as zeros).
// A tile is 32 KB of K (or V): 128 keys at d = 128; 256 keys at d = 64, as one 64-column
// box, where S^T is two M = 128 products (4 k-steps each) and each softmax thread owns
// keys r and 128 + r, so a d = 64 tile carries as many bytes per synchronisation as a
// d = 128 one. At d = 64, O^T += V^T P^T stays an M = 128 product whose second 64-row
// atom reads 16 KB further into shared memory; those rows land in O^T lanes 64..127,
// which nothing reads (each output row depends only on its own row of V^T).
#include <cuda_bf16.h>

#include <algorithm>

#include "fa_internal.h"
#include "sm100_ptx.cuh"
#include "tma_host.h"

namespace fa {
namespace {

using namespace ptx;

constexpr int BN = 128;  // keys per S^T product (the MMA's M)
constexpr int NQP = 64;  // queries padded to the MMA's N
constexpr int kSoftThreads = 256;  // two groups of four softmax warps
constexpr int kThreads = kSoftThreads + 64;
constexpr int kLoadWarp = 8, kMmaWarp = 9;
constexpr float kThreshold = 8.f;
constexpr float kNegM0 = 1e30f;  // -m of a query before its first visible score

constexpr int kBoxBytes = BN * 128;           // [128 rows x 64 bf16]
constexpr int kQBox = NQP * 128;              // [64 rows x 64 bf16]
constexpr int kMaxStages = 8;

// Shared-memory layout by head dimension (1024-byte aligned base).
template <int D>
struct Cfg {
  static constexpr int kBoxes = D / 64;                // 64-column boxes per row
  // A tile is 32 KB of K (or V): 128 keys at d = 128, 256 keys at d = 64, where S^T takes
  // two M = 128 products (keys 0..127 and 128..255) and each softmax thread two keys.
  static constexpr int kHalves = D == 64 ? 2 : 1;
  static constexpr int kTileKeys = BN * kHalves;
  static constexpr int kBoxBytesT = kTileKeys * 128;   // one 64-column box of a tile
  static constexpr int kTile = kBoxes * kBoxBytesT;    // one K or V stage
  static constexpr int kPTile = kTileKeys * NQP * 2;   // P^T [tile keys x 64 queries] bf16
  static constexpr int kPBufs = 2;                     // P^T buffers
  // K is read a tile before V, so it gets the deeper ring where shared memory allows (at
  // d = 64 the two P^T tiles of 32 KB leave room for two stages of each)
  static constexpr int kKStages = D == 64 ? 2 : 3;
  static constexpr int kVStages = 2;
  static constexpr int kSCols = kHalves * NQP;         // TMEM columns of one S^T buffer
  static constexpr uint32_t kColO = 2 * kSCols;        // O^T after the two S^T buffers
  static constexpr uint32_t kTmemCols = kColO + NQP <= 256 ? 256 : 512;
  static constexpr int kQBytes = kBoxes * kQBox;
  static constexpr int kKOff = 0;
  static constexpr int kVOff = kKOff + kKStages * kTile;
  static constexpr int kQOff = kVOff + kVStages * kTile;
  static constexpr int kPOff = kQOff + kQBytes;
  static constexpr int kCorrOff = kPOff + kPBufs * kPTile;  // float[64] rescale factors
  static constexpr int kNmOff = kCorrOff + 4 * NQP;      // float[64] -m per query (log2 units)
  static constexpr int kNmtOff = kNmOff + 4 * NQP;       // float[64] -(m + threshold) per query
  static constexpr int kRedOff = kNmtOff + 4 * NQP;      // float[4][64] cross-warp scratch
  static constexpr int kFlagOff = kRedOff + 4 * 4 * NQP; // int[2][8] per-warp flags, by tile parity
  static constexpr int kSmemBytes = kFlagOff + 64 + 1024;
  static_assert(kKStages <= kMaxStages && kVStages <= kMaxStages, "stages");
  static_assert(kSmemBytes <= 227 * 1024, "shared memory");
  // the second 64-row atom of V^T (kBoxBytes past each k-step's rows) stays inside the
  // allocation, also for the last k-step of the last V stage
  static_assert(kVOff + (kVStages - 1) * kTile + kBoxBytes + kBoxBytesT <= kSmemBytes - 1024, "V^T atom");
};

constexpr uint32_t kColS0 = 0;  // S^T buffers, then O^T (Cfg::kColO)

struct TcParams {
  float* part_o;   // [heads][P][nq][d]
  float* part_ml;  // [heads][P][nq][2]
  int64_t total, L;
  int nq, Nk, P, causal, offset;
  float sl2;
  int* status;
};

struct Ctl {
  uint64_t k_full[kMaxStages], v_full[kMaxStages], k_empty[kMaxStages], v_empty[kMaxStages];
  uint64_t q_full, q_empty, s_full[2], p_full[2], pv_done[2], o_free, drain;
  uint32_t tmem_base;
  int abort;
};

// Named barrier of softmax group g (barrier 0 is __syncthreads).
__device__ __forceinline__ void group_sync(int g) { asm volatile("bar.sync %0, 128;" ::"r"(1 + g) : "memory"); }

// kN consecutive fp32 columns of this thread's TMEM lane (kN = 8, 16 or 32); the load and
// its wait form one statement, so no use of the values is scheduled before they arrive.
template <int kN>
__device__ __forceinline__ void tmem_ld_cols(uint32_t ta, float (&v)[kN]) {
  static_assert(kN == 8 || kN == 16 || kN == 32, "columns");
  if constexpr (kN == 32) {
    tmem_ld32(ta, v);
  } else if constexpr (kN == 16) {
    tmem_ld16(ta, *reinterpret_cast<uint32_t(*)[16]>(&v[0]));
  } else {
    uint32_t* r = reinterpret_cast<uint32_t*>(v);
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x8.b32 {%0,%1,%2,%3,%4,%5,%6,%7}, [%8];\n"
        "tcgen05.wait::ld.sync.aligned;"
        : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7])
        : "r"(ta)
        : "memory");
  }
}

// Store kN consecutive 32-bit columns of this thread's TMEM lane (no wait).
template <int kN>
__device__ __forceinline__ void tmem_st_cols(uint32_t ta, const uint32_t (&w)[kN]) {
  if constexpr (kN == 8) {
    asm volatile("tcgen05.st.sync.aligned.32x32b.x8.b32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8};" ::"r"(ta), "r"(w[0]),
                 "r"(w[1]), "r"(w[2]), "r"(w[3]), "r"(w[4]), "r"(w[5]), "r"(w[6]), "r"(w[7])
                 : "memory");
  } else {
#pragma unroll
    for (int c = 0; c < kN; c += 16) tmem_st16(ta + c, *reinterpret_cast<const uint32_t(*)[16]>(&w[c]));
  }
}

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

template <int D, int kCols>
__global__ void __launch_bounds__(kThreads, 1)
splitkv_tc_kernel(const __grid_constant__ CUtensorMap tmK, const __grid_constant__ CUtensorMap tmV,
                  const __grid_constant__ CUtensorMap tmQ, const TcParams p) {
  using C = Cfg<D>;
  extern __shared__ uint8_t smem_raw[];
  __shared__ Ctl ctl;
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int64_t g_begin = (int64_t)blockIdx.x * p.L;
  const int64_t g_end = min(p.total, g_begin + p.L);
  const uint32_t groups = (uint32_t)((p.nq + kCols - 1) / kCols);  // softmax groups with queries: 1 or 2

  if (threadIdx.x == 0) {
    for (int s = 0; s < C::kKStages; ++s) {
      mbar_init(&ctl.k_full[s], 1);
      mbar_init(&ctl.k_empty[s], 1);
    }
    for (int s = 0; s < C::kVStages; ++s) {
      mbar_init(&ctl.v_full[s], 1);
      mbar_init(&ctl.v_empty[s], 1);
    }
    mbar_init(&ctl.q_full, 1);
    mbar_init(&ctl.q_empty, 1);
    for (int b = 0; b < 2; ++b) {
      mbar_init(&ctl.s_full[b], 1);
      mbar_init(&ctl.p_full[b], 4 * groups);  // one arrival per softmax warp with queries
    }
    mbar_init(&ctl.pv_done[0], 1);
    mbar_init(&ctl.pv_done[1], 1);
    mbar_init(&ctl.o_free, 4 * groups);
    mbar_init(&ctl.drain, 1);
    ctl.abort = 0;
    fence_mbar_init();
  }
  if (warp == kMmaWarp) tmem_alloc(&ctl.tmem_base, C::kTmemCols);
  if (threadIdx.x < kSoftThreads) {
    // P^T columns no group writes (queries past 2C) stay zero for every PV product
    for (int i = threadIdx.x; i < C::kPBufs * C::kPTile / 16; i += kSoftThreads)
      reinterpret_cast<uint4*>(smem + C::kPOff)[i] = make_uint4(0u, 0u, 0u, 0u);
    fence_proxy_async_smem();
  }
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
      const int stages = kq ? C::kKStages : C::kVStages;
      uint64_t* full = kq ? ctl.k_full : ctl.v_full;
      uint64_t* empty = kq ? ctl.k_empty : ctl.v_empty;
      const CUtensorMap* map = kq ? &tmK : &tmV;
      uint8_t* ring = smem + (kq ? C::kKOff : C::kVOff);
      SegIter it{g_begin, g_end, p.Nk};
      int64_t h;
      int k0, k1, seg = 0, t = 0, last[kMaxStages], last_q = -1;
      for (int s = 0; s < kMaxStages; ++s) last[s] = -1;
      bool ok = true;
      while (ok && it.next(h, k0, k1)) {
        if (kq) {  // Q of this head, once the previous segment's S products have read the old one
          if (seg > 0 && !(ok = mbar_wait(&ctl.q_empty, (seg - 1) & 1, p.status, abort))) break;
          mbar_expect_tx(&ctl.q_full, C::kQBytes);
          for (int b = 0; b < D / 64; ++b) tma_load_3d(smem + C::kQOff + b * kQBox, &tmQ, &ctl.q_full, b * 64, 0, (int)h);
          last_q = seg;
        }
        for (int kt = k0; ok && kt < k1; kt += C::kTileKeys, ++t) {
          const int s = t % stages;
          if (t >= stages && !(ok = mbar_wait(&empty[s], ((t / stages) - 1) & 1, p.status, abort))) break;
          mbar_expect_tx(&full[s], C::kTile);
          for (int b = 0; b < D / 64; ++b)
            tma_load_3d(ring + s * C::kTile + b * C::kBoxBytesT, map, &full[s], b * 64, kt, (int)h);
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
      // O^T: A = V^T (M = 128 rows of d, zero past d = 64), B = P^T, both MN-major
      constexpr uint32_t idO = idesc_bf16(128, NQP, true, true);
      const uint64_t dK0 = sdesc_sw128(smem_u32(smem + C::kKOff), 16, 1024);
      const uint64_t dQ0 = sdesc_sw128(smem_u32(smem + C::kQOff), 16, 1024);
      const uint64_t dV0 = sdesc_sw128(smem_u32(smem + C::kVOff), kBoxBytes, 1024);
      const uint64_t dP0 = sdesc_sw128(smem_u32(smem + C::kPOff), C::kPTile, 1024);
      auto issue_S = [&](int t) {
        const uint32_t ko = (t % C::kKStages) * C::kTile;
#pragma unroll
        for (int hb = 0; hb < C::kHalves; ++hb)  // keys 128*hb .. +127 of the tile
#pragma unroll
          for (int k = 0; k < D / 16; ++k) {
            const uint32_t off = (k / 4) * C::kBoxBytesT + hb * (BN * 128) + (k % 4) * 32,
                           qoff = (k / 4) * kQBox + (k % 4) * 32;
            mma_ss(tmem + kColS0 + (t & 1) * C::kSCols + hb * NQP, sdesc_add(dK0, ko + off), sdesc_add(dQ0, qoff),
                   idS, k > 0);
          }
      };
      auto issue_PV = [&](int t, bool acc) {
        const uint32_t vo = (t % C::kVStages) * C::kTile, po = (t % C::kPBufs) * C::kPTile;
#pragma unroll
        for (int k = 0; k < C::kTileKeys / 16; ++k)
          mma_ss(tmem + C::kColO, sdesc_add(dV0, vo + k * 2048), sdesc_add(dP0, po + k * 2048), idO,
                 (acc || k > 0) ? 1u : 0u);
      };
      SegIter it{g_begin, g_end, p.Nk};
      int64_t h;
      int k0, k1, seg = 0, t = 0;
      bool ok = true;
      while (ok && it.next(h, k0, k1)) {
        const int n = (k1 - k0 + C::kTileKeys - 1) / C::kTileKeys;  // tiles in this segment: t .. t + n - 1
        if (!(ok = mbar_wait(&ctl.q_full, seg & 1, p.status, abort))) break;
        if (!(ok = mbar_wait(&ctl.k_full[t % C::kKStages], (t / C::kKStages) & 1, p.status, abort))) break;
        tc_fence_after();
        issue_S(t);
        mma_commit(&ctl.k_empty[t % C::kKStages]);
        mma_commit(&ctl.s_full[t & 1]);
        for (int i = 0; i < n; ++i, ++t) {
          if (i + 1 < n) {  // S of the next tile into the other buffer (read out by tile t-1's softmax)
            if (t >= 1 && !(ok = mbar_wait(&ctl.p_full[(t + 1) & 1], ((t - 1) >> 1) & 1, p.status, abort))) break;
            if (!(ok = mbar_wait(&ctl.k_full[(t + 1) % C::kKStages], ((t + 1) / C::kKStages) & 1, p.status, abort)))
              break;
            tc_fence_after();
            issue_S(t + 1);
            mma_commit(&ctl.k_empty[(t + 1) % C::kKStages]);
            mma_commit(&ctl.s_full[(t + 1) & 1]);
          } else {
            mma_commit(&ctl.q_empty);  // every S of the segment is issued: Q may be replaced
          }
          if (!(ok = mbar_wait(&ctl.p_full[t & 1], (t >> 1) & 1, p.status, abort))) break;
          if (!(ok = mbar_wait(&ctl.v_full[t % C::kVStages], (t / C::kVStages) & 1, p.status, abort))) break;
          if (i == 0 && seg > 0 && !(ok = mbar_wait(&ctl.o_free, (seg - 1) & 1, p.status, abort))) break;
          tc_fence_after();
          issue_PV(t, i > 0);
          mma_commit(&ctl.v_empty[t % C::kVStages]);
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
    const int g = warp >> 2, wq = warp & 3;  // softmax group, TMEM lane quarter
    const int r = wq * 32 + lane;            // TMEM lane: key of the tile in S^T, head-dim row in O^T
    const uint32_t lane_off = (uint32_t)(wq * 32) << 16;
    const int q0 = g * kCols;                // the group's first query column
    float* corr = reinterpret_cast<float*>(smem + C::kCorrOff);
    float* nm = reinterpret_cast<float*>(smem + C::kNmOff);    // uniform over the group's threads
    float* nmt = reinterpret_cast<float*>(smem + C::kNmtOff);
    const float sl2 = p.sl2;
    const float2 sl2x2 = make_float2(sl2, sl2);
    float* red = reinterpret_cast<float*>(smem + C::kRedOff);
    int* flags = reinterpret_cast<int*>(smem + C::kFlagOff);
    const int nq = p.nq;
    if (q0 < nq) {
      SegIter it{g_begin, g_end, p.Nk};
      int64_t h;
      int k0, k1, t = 0;
      bool ok = true;
      // After a failed (timed-out) wait the loops keep their shape, skipping the waits and
      // the TMEM accesses, so that every warp of the group still reaches every named barrier.
      while (it.next(h, k0, k1)) {
        const int n = (k1 - k0 + C::kTileKeys - 1) / C::kTileKeys;
        if (r < kCols) {
          nm[q0 + r] = kNegM0;
          nmt[q0 + r] = kNegM0;  // -(m + threshold) rounds to the same value
        }
        float l[kCols];
#pragma unroll
        for (int q = 0; q < kCols; ++q) l[q] = 0.f;
        group_sync(g);
        for (int i = 0; i < n; ++i, ++t) {
          if (ok) ok = __all_sync(0xffffffffu, mbar_wait(&ctl.s_full[t & 1], (t >> 1) & 1, p.status, abort));
          // x[hb] holds the raw scores q.k of key 128*hb + r of the tile; masked ones become
          // -inf (scaled: still -inf)
          float x[C::kHalves][kCols];
#pragma unroll
          for (int hb = 0; hb < C::kHalves; ++hb) {
            if (ok) {
              tc_fence_after();
              tmem_ld_cols<kCols>(tmem + lane_off + kColS0 + (t & 1) * C::kSCols + hb * NQP + q0, x[hb]);
            } else {
#pragma unroll
              for (int q = 0; q < kCols; ++q) x[hb][q] = 0.f;
            }
          }
          const int kb = k0 + i * C::kTileKeys;  // first key of the tile
          const bool full = ok && kb + C::kTileKeys <= k1 && q0 + kCols <= nq &&
                            (!p.causal || kb + C::kTileKeys - 1 <= q0 + p.offset);
          if (!full) {
#pragma unroll
            for (int hb = 0; hb < C::kHalves; ++hb) {
              const int key = kb + hb * BN + r;
              const bool kin = key < k1;
#pragma unroll
              for (int q = 0; q < kCols; ++q) {
                const int qg = q0 + q;
                const bool vis = ok && kin && qg < nq && !(p.causal && key > qg + p.offset);
                x[hb][q] = vis ? x[hb][q] : -INFINITY;
              }
            }
          }
          // does any score of the tile exceed its query's reference max by the threshold?
          const float4* nmt4 = reinterpret_cast<const float4*>(nmt + q0);
          float e = -INFINITY;
#pragma unroll
          for (int hb = 0; hb < C::kHalves; ++hb)
#pragma unroll
            for (int q = 0; q < kCols; q += 4) {
              const float4 t4 = nmt4[q / 4];
              const float2 a = ffma2(make_float2(x[hb][q], x[hb][q + 1]), sl2x2, make_float2(t4.x, t4.y));
              const float2 b = ffma2(make_float2(x[hb][q + 2], x[hb][q + 3]), sl2x2, make_float2(t4.z, t4.w));
              e = fmax3(e, a.x, a.y);
              e = fmax3(e, b.x, b.y);
            }
          const bool grow = __any_sync(0xffffffffu, e > 0.f);
          int* fl = flags + (t & 1) * 8 + 4 * g;
          if (lane == 0) fl[wq] = grow ? 1 : 0;
          group_sync(g);
          if ((fl[0] | fl[1] | fl[2] | fl[3]) != 0) {  // uniform over the group
            // exact column maxima of the tile: warp reduction, then across the group's warps
#pragma unroll
            for (int q = 0; q < kCols; ++q) {
              float v = x[0][q];
#pragma unroll
              for (int hb = 1; hb < C::kHalves; ++hb) v = fmaxf(v, x[hb][q]);
              v *= sl2;
#pragma unroll
              for (int o = 16; o; o >>= 1) v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, o));
              if (lane == 0) red[wq * NQP + q0 + q] = v;
            }
            group_sync(g);
            if (r < kCols) {
              const int qg = q0 + r;
              const float mx = fmaxf(fmaxf(red[qg], red[NQP + qg]), fmaxf(red[2 * NQP + qg], red[3 * NQP + qg]));
              const float mo = -nm[qg], mn = fmaxf(mo, mx);
              corr[qg] = mn > mo ? ex2(mo - mn) : 1.f;  // mo = -1e30 gives 0: nothing accumulated yet
              nm[qg] = -mn;
              nmt[qg] = -(mn + kThreshold);
            }
            group_sync(g);
#pragma unroll
            for (int q = 0; q < kCols; ++q) l[q] *= corr[q0 + q];
            if (i > 0 && ok) {
              // the group's O^T columns (lane = head-dim row) are rescaled once the previous
              // tile's PV has finished
              ok = __all_sync(0xffffffffu,
                              mbar_wait(&ctl.pv_done[(t - 1) & 1], ((t - 1) >> 1) & 1, p.status, abort));
              if (ok) {
                tc_fence_after();
                float ov[kCols];
                tmem_ld_cols<kCols>(tmem + lane_off + C::kColO + q0, ov);
                uint32_t w[kCols];
#pragma unroll
                for (int q = 0; q < kCols; ++q) w[q] = __float_as_uint(ov[q] * corr[q0 + q]);
                tmem_st_cols<kCols>(tmem + lane_off + C::kColO + q0, w);
                tmem_wait_st();
              }
            }
          }
          // The P^T buffer of this tile was last read by PV(t - kPBufs).
          if (t >= C::kPBufs && ok)
            ok = __all_sync(0xffffffffu, mbar_wait(&ctl.pv_done[(t - C::kPBufs) & 1], ((t - C::kPBufs) >> 1) & 1,
                                                   p.status, abort));
          // p = 2^(s - m) <= 2^threshold; the group's 2C bytes of P^T rows 128*hb + r
          // (128-byte swizzle; those rows share r's position in their group of 8)
          const float4* nm4 = reinterpret_cast<const float4*>(nm + q0);
#pragma unroll
          for (int hb = 0; hb < C::kHalves; ++hb) {
            uint8_t* prow = smem + C::kPOff + (t % C::kPBufs) * C::kPTile + (hb * BN + r) * 128;
#pragma unroll
            for (int c = 0; c < kCols / 8; ++c) {
              uint32_t w[4];
#pragma unroll
              for (int u = 0; u < 4; ++u) {
                const int q = c * 8 + 2 * u;
                const float4 m4 = nm4[q / 4];
                const float2 a = ffma2(make_float2(x[hb][q], x[hb][q + 1]), sl2x2,
                                       (u & 1) ? make_float2(m4.z, m4.w) : make_float2(m4.x, m4.y));
                const float p0 = ex2(a.x), p1 = ex2(a.y);
                const float2 ls = fadd2(make_float2(l[q], l[q + 1]), make_float2(p0, p1));
                l[q] = ls.x;
                l[q + 1] = ls.y;
                w[u] = pack_bf16(p0, p1);
              }
              const int chunk = q0 / 8 + c;
              *reinterpret_cast<uint4*>(prow + ((chunk ^ (r & 7)) << 4)) = make_uint4(w[0], w[1], w[2], w[3]);
            }
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
        for (int q = 0; q < kCols; ++q) {
          float v = l[q];
#pragma unroll
          for (int o = 16; o; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
          if (lane == 0) red[wq * NQP + q0 + q] = v;
        }
        group_sync(g);
        const int slot = (int)(blockIdx.x - (h * p.Nk) / p.L);
        const int64_t base = (h * p.P + slot) * nq;
        if (r < kCols && q0 + r < nq) {
          const int qg = q0 + r;
          const float m = -nm[qg];
          p.part_ml[(base + qg) * 2] = m <= -0.5f * kNegM0 ? -INFINITY : m;  // no visible key: -inf
          p.part_ml[(base + qg) * 2 + 1] = red[qg] + red[NQP + qg] + red[2 * NQP + qg] + red[3 * NQP + qg];
        }
        if (ok) {
          tc_fence_after();
          float ov[kCols];
          tmem_ld_cols<kCols>(tmem + lane_off + C::kColO + q0, ov);  // warp-collective: every lane loads
          if (r < D) {  // O^T lanes past d hold V^T's zero rows
#pragma unroll
            for (int q = 0; q < kCols; ++q)
              if (q0 + q < nq) p.part_o[(base + q0 + q) * D + r] = ov[q];
          }
        }
        tc_fence_before();
        group_sync(g);  // red[], nm[], nmt[] and the group's O^T columns are free for the next segment
        if (lane == 0) mbar_arrive(&ctl.o_free);
      }
    }
  }

  // The producer and MMA roles run on single lanes: they rejoin the rest of their warps
  // first, so that the barrier below (which counts whole warps) holds until every role is done.
  __syncwarp();
  tc_fence_before();
  __syncthreads();
  if (warp == kMmaWarp) {
    tc_fence_after();
    tmem_dealloc(tmem, C::kTmemCols);
  }
}

template <int D, int kCols>
cudaError_t launch(const CUtensorMap& mk, const CUtensorMap& mv, const CUtensorMap& mq, const TcParams& p, int ctas,
                   cudaStream_t st) {
  static const bool attr = cudaFuncSetAttribute(splitkv_tc_kernel<D, kCols>,
                                                cudaFuncAttributeMaxDynamicSharedMemorySize, Cfg<D>::kSmemBytes) == cudaSuccess;
  if (!attr) return cudaErrorInvalidConfiguration;
  splitkv_tc_kernel<D, kCols><<<ctas, kThreads, Cfg<D>::kSmemBytes, st>>>(mk, mv, mq, p);
  return cudaGetLastError();
}

template <int D>
cudaError_t launch_d(const CUtensorMap& mk, const CUtensorMap& mv, const CUtensorMap& mq, const TcParams& p, int ctas,
                     cudaStream_t st) {
  if (p.nq <= 16) return launch<D, 8>(mk, mv, mq, p, ctas, st);
  if (p.nq <= 32) return launch<D, 16>(mk, mv, mq, p, ctas, st);
  return launch<D, 32>(mk, mv, mq, p, ctas, st);
}

}  // namespace

cudaError_t splitkv_tc_partial(const void* Q, const void* K, const void* V, int64_t heads, int Nq, int Nk, int d,
                               float scale, bool causal, int64_t L, int ctas, int P, float* part_o, float* part_ml,
                               int* status, cudaStream_t st) {
  if (d != 64 && d != 128) return cudaErrorInvalidValue;
  CUtensorMap mk, mv, mq;
  const int tile_keys = d == 64 ? Cfg<64>::kTileKeys : Cfg<128>::kTileKeys;
  if (!make_map_bf16_3d(&mk, K, heads, Nk, d, tile_keys) || !make_map_bf16_3d(&mv, V, heads, Nk, d, tile_keys) ||
      !make_map_bf16_3d(&mq, Q, heads, Nq, d, NQP))
    return cudaErrorInvalidValue;
  TcParams p;
  p.part_o = part_o;
  p.part_ml = part_ml;
  p.total = heads * Nk;
  p.L = L;
  p.nq = Nq;
  p.Nk = Nk;
  p.P = P;
  p.causal = causal ? 1 : 0;
  p.offset = Nk - Nq;
  p.sl2 = scale * 1.4426950408889634f;
  p.status = status;
  return d == 64 ? launch_d<64>(mk, mv, mq, p, ctas, st) : launch_d<128>(mk, mv, mq, p, ctas, st);
}

}  // namespace fa
