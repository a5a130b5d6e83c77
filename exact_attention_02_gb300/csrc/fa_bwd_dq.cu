// Attention backward, dQ alone, on 128-query tiles (head dimension 64 or 128; bf16 in, fp32
// accumulate): the separate dQ pass of fa_bwd. The 128-key-tile kernel (fa_bwd_wide.cu),
// run without its dQ partials, supplies dK and dV; this kernel supplies dQ.
//
// Method ("flash-attention-backpropagation", QKV梯度: dQ = dS K / sqrt(d); "FlashAttention
// 反向传播" 踩坑二 weighs one recompute per tile for all three gradients against a second
// pass for dQ): one CTA owns a 128-row query tile of one head and loops over the key tiles
// the tile sees, recomputing S and dP for each:
//   S   = Q_i K_j^T                  [queries x keys]  tcgen05, A, B from smem (K-major)
//   dP  = dO_i V_j^T                 [queries x keys]  tcgen05
//   P   = exp2(S * scale*log2e - LSE*log2e)            softmax warps
//   dS  = P * (dP - D)                                 softmax warps, bf16 into TMEM
//   dQ_i += dS K_j                   A = dS from TMEM, B = K_j (MN-major), fp32 in TMEM
// and scale * dQ_i is rounded to bf16 once, when the last key tile is in. dQ never leaves
// the chip in fp32: no accumulator in global memory, no atomic additions, no clearing or
// conversion pass, and the result does not depend on the order in which CTAs run.
//
// Queries sit on the TMEM lanes. TMEM: S [0,128), dP [128,256), dQ [256,256+d), dS (bf16
// pairs) [384,448). The softmax warps release S and dP as soon as they have loaded them, so
// S(j+1) and dP(j+1) run while they work on tile j; dQ(j) needs only finish before dS(j+1)
// is stored. Issue order: S(0) dP(0) | S(j+1) dP(j+1) | dQ(j) | ...
//
// CTA = 10 warps: 0-7 softmax (two warpgroups over key columns 0-63 and 64-127 of each
// tile; a thread owns one query row = TMEM lane), which also write dQ at the end; 8 TMA
// producer; 9 MMA issuer. Shared memory: Q_i and dO_i (once), a ring of K_j and one of V_j
// tiles. K_j is read by S(j) and dQ(j), V_j only by dP(j), so V's slots free a product
// earlier and K takes one stage more at d = 128 (3 K + 2 V: 224 KB).
//
// Query and key lengths as in the 128-key-tile kernel: causal is bottom-right aligned
// (query i hides keys j > i + Nk - Nq), keys past the end of a head arrive as zero rows and
// are masked, queries past the end get P = 0 and are not stored.
#include <cuda_bf16.h>

#include "fa_internal.h"
#include "sm100_ptx.cuh"
#include "tma_host.h"

namespace fa {
namespace {

using namespace ptx;

constexpr int BQ = 128;  // queries per CTA
constexpr int BN = 128;  // keys per tile
constexpr int kThreads = 320;
constexpr int kLoadWarp = 8;
constexpr int kMmaWarp = 9;
constexpr float kLog2e = 1.4426950408889634f;
constexpr int kBox = 128 * 128;  // one [128 rows x 64 columns] bf16 box, 128-byte swizzle
constexpr uint32_t kTmemCols = 512;

struct DqCtl {
  uint64_t q_full;
  uint64_t k_full[4], v_full[4], k_empty[4], v_empty[4];
  uint64_t st_full;   // S(j) and dP(j) have run
  uint64_t s_free;    // the softmax warps have loaded S(j) and dP(j) (256 arrivals)
  uint64_t ds_full;   // dS(j) is in TMEM (256 arrivals)
  uint64_t dq_done;   // dQ(j) has run (its dS columns may be overwritten)
  uint64_t dq_final;  // every dQ product has run
  uint64_t drain;
  uint32_t tmem_base;
  int abort;
};

template <int D>
struct DqCfg {
  static constexpr int kBoxes = D / 64;         // 64-column boxes per row
  static constexpr int kRowTile = 128 * D * 2;  // a [128 rows x D] bf16 tile
  static constexpr int kKStages = D == 128 ? 3 : 4;
  static constexpr int kVStages = D == 128 ? 2 : 4;
  static constexpr int kQOff = 0;
  static constexpr int kDOOff = kRowTile;
  static constexpr int kKOff = 2 * kRowTile;
  static constexpr int kVOff = kKOff + kKStages * kRowTile;
  static constexpr int kCtlOff = kVOff + kVStages * kRowTile;
  static constexpr int kSmemBytes = kCtlOff + (int)sizeof(DqCtl);
  static_assert(kSmemBytes <= 227 * 1024, "shared-memory budget");
  static_assert(kKStages <= 4 && kVStages <= 4, "barrier arrays");
  static constexpr uint32_t kColS = 0, kColDP = 128, kColDQ = 256, kColDS = 384;
  static_assert(kColDQ + D <= kColDS && kColDS + 64 <= kTmemCols, "TMEM budget");
};

struct DqParams {
  const float* LSE;
  const float* Dvec;
  __nv_bfloat16* dQ;
  int* status;
  int Nq, Nk;
  int heads;
  int qtiles;
  int kvtiles;
  int causal;
  int offset;  // causal: query i hides keys j > i + offset
  float scale;
  float sl2;   // scale * log2(e)
};

template <int D, bool kTail>
__global__ void __launch_bounds__(kThreads, 1)
fa_bwd_dq_kernel(const __grid_constant__ CUtensorMap tmQ, const __grid_constant__ CUtensorMap tmK,
                 const __grid_constant__ CUtensorMap tmV, const __grid_constant__ CUtensorMap tmdO,
                 const DqParams p) {
  using C = DqCfg<D>;
  extern __shared__ __align__(1024) uint8_t smem[];
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  // The swizzled operand layout needs a 1024-byte aligned base; the runtime provides it for
  // this declaration, and the kernel refuses to run (status word) if it did not.
  if ((smem_u32(smem) & 1023u) != 0) {
    if (threadIdx.x == 0 && p.status) atomicExch(p.status, 3 /* FA_ERR_CUDA */);
    return;
  }
  DqCtl& ctl = *reinterpret_cast<DqCtl*>(smem + C::kCtlOff);

  int qt, head;
  if (p.causal) {  // query tiles near the end see the most keys: launch them first
    qt = p.qtiles - 1 - (int)(blockIdx.x / p.heads);
    head = (int)(blockIdx.x % p.heads);
  } else {
    qt = (int)(blockIdx.x % p.qtiles);
    head = (int)(blockIdx.x / p.qtiles);
  }
  const int qrow_base = head * p.Nq;
  // key tiles the tile sees: causal, up to the limit of its last query (none when even that
  // query sees no key, which only happens with more queries than keys)
  int nk = p.kvtiles;
  if (p.causal) {
    const int lim = min((qt + 1) * BQ, p.Nq) - 1 + p.offset;
    nk = lim < 0 ? 0 : min(p.kvtiles, lim / BN + 1);
  }
  if (nk == 0) {  // no query of the tile sees a key: dQ = 0
    const int q = qt * BQ + (int)threadIdx.x;
    if (threadIdx.x < BQ && q < p.Nq) {
      uint4* dst = reinterpret_cast<uint4*>(p.dQ + (size_t)(qrow_base + q) * D);
#pragma unroll
      for (int u = 0; u < D / 8; ++u) dst[u] = make_uint4(0, 0, 0, 0);
    }
    return;
  }

  if (threadIdx.x == 0) {
    mbar_init(&ctl.q_full, 1);
    for (int s = 0; s < 4; ++s) {
      mbar_init(&ctl.k_full[s], 1);
      mbar_init(&ctl.v_full[s], 1);
      mbar_init(&ctl.k_empty[s], 1);
      mbar_init(&ctl.v_empty[s], 1);
    }
    mbar_init(&ctl.st_full, 1);
    mbar_init(&ctl.s_free, 256);
    mbar_init(&ctl.ds_full, 256);
    mbar_init(&ctl.dq_done, 1);
    mbar_init(&ctl.dq_final, 1);
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
    if (lane == 0) {
      prefetch_tmap(&tmQ);
      prefetch_tmap(&tmK);
      prefetch_tmap(&tmV);
      prefetch_tmap(&tmdO);
      // Test hook of the failure path: never arm Q/dO, so the MMA thread's wait for them
      // runs out (see StatusBlock); off unless a test sets it.
      const bool skip_q = injected(p.status, kInjectBwd);
      if (!skip_q) {
        mbar_expect_tx(&ctl.q_full, 2 * C::kRowTile);
        for (int b = 0; b < C::kBoxes; ++b) {
          tma_load_3d(smem + C::kQOff + b * kBox, &tmQ, &ctl.q_full, b * 64, qt * BQ, head);
          tma_load_3d(smem + C::kDOOff + b * kBox, &tmdO, &ctl.q_full, b * 64, qt * BQ, head);
        }
      }
      int last_k[4] = {-1, -1, -1, -1}, last_v[4] = {-1, -1, -1, -1};
      for (int j = 0; j < nk; ++j) {
        const int sk = j % C::kKStages, sv = j % C::kVStages;
        // K_j's slot frees once dQ(j - stages) has run, V_j's once dP(j - stages) has
        if (j >= C::kKStages && !mbar_wait(&ctl.k_empty[sk], ((j / C::kKStages) - 1) & 1, p.status, abort)) break;
        mbar_expect_tx(&ctl.k_full[sk], C::kRowTile);
        for (int b = 0; b < C::kBoxes; ++b)
          tma_load_3d(smem + C::kKOff + sk * C::kRowTile + b * kBox, &tmK, &ctl.k_full[sk], b * 64, j * BN, head);
        last_k[sk] = j;
        if (j >= C::kVStages && !mbar_wait(&ctl.v_empty[sv], ((j / C::kVStages) - 1) & 1, p.status, abort)) break;
        mbar_expect_tx(&ctl.v_full[sv], C::kRowTile);
        for (int b = 0; b < C::kBoxes; ++b)
          tma_load_3d(smem + C::kVOff + sv * C::kRowTile + b * kBox, &tmV, &ctl.v_full[sv], b * 64, j * BN, head);
        last_v[sv] = j;
      }
      // every issued copy must land before the CTA may exit
      if (!skip_q) mbar_wait(&ctl.q_full, 0, p.status, nullptr);
      for (int s = 0; s < 4; ++s) {
        if (last_k[s] >= 0) mbar_wait(&ctl.k_full[s], (last_k[s] / C::kKStages) & 1, p.status, nullptr);
        if (last_v[s] >= 0) mbar_wait(&ctl.v_full[s], (last_v[s] / C::kVStages) & 1, p.status, nullptr);
      }
    }
  } else if (warp == kMmaWarp) {
    if (lane == 0) {
      constexpr uint32_t idS = idesc_bf16(BQ, BN, false, false);  // S, dP
      constexpr uint32_t idQ = idesc_bf16(BQ, D, false, true);    // dQ (B MN-major)
      const uint64_t dQk = sdesc_sw128(smem_u32(smem + C::kQOff), 16, 1024);
      const uint64_t dOk = sdesc_sw128(smem_u32(smem + C::kDOOff), 16, 1024);
      const uint64_t dKk = sdesc_sw128(smem_u32(smem + C::kKOff), 16, 1024);     // K_j, K-major
      const uint64_t dKmn = sdesc_sw128(smem_u32(smem + C::kKOff), kBox, 1024);  // K_j, MN-major
      const uint64_t dVk = sdesc_sw128(smem_u32(smem + C::kVOff), 16, 1024);
      // K = d: 16 columns (32 bytes) per step inside a box, the next box after 4 steps
      auto issue_SdP = [&](int sk, int sv) {
#pragma unroll
        for (int k = 0; k < D / 16; ++k) {
          const uint32_t off = (k / 4) * kBox + (k % 4) * 32;
          mma_ss(tmem + C::kColS, sdesc_add(dQk, off), sdesc_add(dKk, sk * C::kRowTile + off), idS, k > 0);
        }
#pragma unroll
        for (int k = 0; k < D / 16; ++k) {
          const uint32_t off = (k / 4) * kBox + (k % 4) * 32;
          mma_ss(tmem + C::kColDP, sdesc_add(dOk, off), sdesc_add(dVk, sv * C::kRowTile + off), idS, k > 0);
        }
      };
      // K = keys: 16 keys per step, 8 TMEM columns of packed dS and 16 rows (2048 bytes) of K_j
      auto issue_dQ = [&](int sk, bool acc) {
#pragma unroll
        for (int k = 0; k < BN / 16; ++k)
          mma_ts(tmem + C::kColDQ, tmem + C::kColDS + k * 8, sdesc_add(dKmn, sk * C::kRowTile + k * 2048), idQ,
                 (acc || k > 0) ? 1u : 0u);
      };
      bool ok = mbar_wait(&ctl.q_full, 0, p.status, abort) && mbar_wait(&ctl.k_full[0], 0, p.status, abort) &&
                mbar_wait(&ctl.v_full[0], 0, p.status, abort);
      if (ok) {
        tc_fence_after();
        issue_SdP(0, 0);
        mma_commit(&ctl.st_full);
        mma_commit(&ctl.v_empty[0]);
      }
      for (int j = 0; ok && j < nk; ++j) {
        const int sk = j % C::kKStages;
        if (j + 1 < nk) {  // S(j+1), dP(j+1) over the columns the softmax warps have loaded
          const int sk1 = (j + 1) % C::kKStages, sv1 = (j + 1) % C::kVStages;
          if (!(ok = mbar_wait(&ctl.s_free, j & 1, p.status, abort))) break;
          if (!(ok = mbar_wait(&ctl.k_full[sk1], ((j + 1) / C::kKStages) & 1, p.status, abort))) break;
          if (!(ok = mbar_wait(&ctl.v_full[sv1], ((j + 1) / C::kVStages) & 1, p.status, abort))) break;
          tc_fence_after();
          issue_SdP(sk1, sv1);
          mma_commit(&ctl.st_full);
          mma_commit(&ctl.v_empty[sv1]);
        }
        if (!(ok = mbar_wait(&ctl.ds_full, j & 1, p.status, abort))) break;
        tc_fence_after();
        issue_dQ(sk, j > 0);
        mma_commit(&ctl.dq_done);
        mma_commit(&ctl.k_empty[sk]);
      }
      mma_commit(&ctl.dq_final);
      mma_commit(&ctl.drain);
      mbar_wait(&ctl.drain, 0, p.status, nullptr);
    }
  } else {
    // ---------------- softmax-backward warpgroups and the dQ epilogue ----------------
    const int wg = warp >> 2;
    const int r = (warp & 3) * 32 + lane;  // TMEM lane = query row in the tile
    const int q = qt * BQ + r;             // query row in the head
    const bool qin = !kTail || q < p.Nq;
    const uint32_t lane_off = (uint32_t)((warp & 3) * 32) << 16;
    // rows past the end of the head: LSE = +inf gives P = 0
    const float lse = qin ? p.LSE[qrow_base + q] : INFINITY;
    const float dq_d = qin ? p.Dvec[qrow_base + q] : 0.f;
    const float2 sl2 = make_float2(p.sl2, p.sl2);
    const float2 nl = make_float2(-lse * kLog2e, -lse * kLog2e);
    const float2 dvec = make_float2(dq_d, dq_d);
    const float2 minus1 = make_float2(-1.f, -1.f);
    bool ok = true;
    for (int j = 0; ok && j < nk; ++j) {
      ok = __all_sync(0xffffffffu, mbar_wait(&ctl.st_full, j & 1, p.status, abort));
      if (!ok) break;
      tc_fence_after();
      // some key of the tile is past the causal limit of some query, or past the end of the head
      const bool edge = (p.causal && j * BN + BN - 1 > qt * BQ + p.offset) || (kTail && j * BN + BN > p.Nk);
      const int lim = min(p.causal ? q + p.offset : 0x7fffffff, p.Nk - 1);  // last visible key
      uint32_t pk[32];
#pragma unroll
      for (int c = 0; c < 2; ++c) {
        const int c0 = wg * 64 + c * 32;  // first key column of this chunk
        float sv[32], dp[32];
        tmem_ld32x2(tmem + lane_off + C::kColS + c0, tmem + lane_off + C::kColDP + c0, sv, dp);
        if (c == 1) {  // S(j), dP(j) are in registers: S(j+1), dP(j+1) may overwrite them
          tc_fence_before();
          mbar_arrive(&ctl.s_free);
        }
#pragma unroll
        for (int u = 0; u < 16; ++u) {
          const float2 x = ffma2(make_float2(sv[2 * u], sv[2 * u + 1]), sl2, nl);
          float2 pr = make_float2(ex2(x.x), ex2(x.y));
          if (edge) {
            const int key = j * BN + c0 + 2 * u;
            if (key > lim) pr.x = 0.f;
            if (key + 1 > lim) pr.y = 0.f;
          }
          const float2 ds = fmul2(pr, ffma2(dvec, minus1, make_float2(dp[2 * u], dp[2 * u + 1])));
          pk[16 * c + u] = pack_bf16(ds.x, ds.y);
        }
      }
      if (j > 0) {  // dQ(j-1) must have read the dS columns
        ok = __all_sync(0xffffffffu, mbar_wait(&ctl.dq_done, (j - 1) & 1, p.status, abort));
        if (!ok) break;
        tc_fence_after();
      }
      tmem_st16(tmem + lane_off + C::kColDS + wg * 32, *reinterpret_cast<const uint32_t(*)[16]>(&pk[0]));
      tmem_st16(tmem + lane_off + C::kColDS + wg * 32 + 16, *reinterpret_cast<const uint32_t(*)[16]>(&pk[16]));
      tmem_wait_st();
      tc_fence_before();
      mbar_arrive(&ctl.ds_full);
    }
    if (ok) ok = __all_sync(0xffffffffu, mbar_wait(&ctl.dq_final, 0, p.status, abort));
    if (ok) {
      // dQ of query row r; warpgroup wg writes columns wg*D/2 .. wg*D/2 + D/2 - 1
      tc_fence_after();
      __nv_bfloat16* dst = p.dQ + (size_t)(qrow_base + q) * D;
#pragma unroll 1
      for (int c0 = wg * (D / 2); c0 < wg * (D / 2) + D / 2; c0 += 32) {
        float v[32];
        tmem_ld32(tmem + lane_off + C::kColDQ + c0, v);
        uint4 w[4];
        uint32_t* wu = reinterpret_cast<uint32_t*>(w);
#pragma unroll
        for (int u = 0; u < 16; ++u) wu[u] = pack_bf16(v[2 * u] * p.scale, v[2 * u + 1] * p.scale);
        if (qin) {
          uint4* d4 = reinterpret_cast<uint4*>(dst + c0);
#pragma unroll
          for (int u = 0; u < 4; ++u) d4[u] = w[u];
        }
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
    tmem_dealloc(tmem, kTmemCols);
  }
}

template <int D>
cudaError_t launch_dq(const void* Q, const void* K, const void* V, const void* dO, const float* LSE,
                      const float* Dv, void* dQ, const Shape& s, float scale, bool causal, int* status,
                      cudaStream_t st) {
  using C = DqCfg<D>;
  CUtensorMap mq, mk, mv, mdo;
  const int64_t heads = s.heads();
  if (!make_map_bf16_3d(&mq, Q, heads, s.N, D, BQ) || !make_map_bf16_3d(&mk, K, heads, s.keys(), D, BN) ||
      !make_map_bf16_3d(&mv, V, heads, s.keys(), D, BN) || !make_map_bf16_3d(&mdo, dO, heads, s.N, D, BQ))
    return cudaErrorInvalidValue;
  static bool attr = [] {
    return cudaFuncSetAttribute(fa_bwd_dq_kernel<D, false>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                C::kSmemBytes) == cudaSuccess &&
           cudaFuncSetAttribute(fa_bwd_dq_kernel<D, true>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                C::kSmemBytes) == cudaSuccess;
  }();
  if (!attr) return cudaErrorInvalidConfiguration;
  DqParams p;
  p.LSE = LSE;
  p.Dvec = Dv;
  p.dQ = static_cast<__nv_bfloat16*>(dQ);
  p.status = status;
  p.Nq = s.N;
  p.Nk = s.keys();
  p.heads = (int)heads;
  p.qtiles = (s.N + BQ - 1) / BQ;
  p.kvtiles = (s.keys() + BN - 1) / BN;
  p.causal = causal ? 1 : 0;
  p.offset = causal ? s.keys() - s.N : 0;
  p.scale = scale;
  p.sl2 = scale * kLog2e;
  const int64_t grid = (int64_t)p.qtiles * p.heads;
  if (s.N % BQ != 0 || s.keys() % BN != 0)
    fa_bwd_dq_kernel<D, true><<<(unsigned)grid, kThreads, C::kSmemBytes, st>>>(mq, mk, mv, mdo, p);
  else
    fa_bwd_dq_kernel<D, false><<<(unsigned)grid, kThreads, C::kSmemBytes, st>>>(mq, mk, mv, mdo, p);
  return cudaGetLastError();
}

}  // namespace

cudaError_t tc_bwd_dq(const void* Q, const void* K, const void* V, const void* dO, const float* LSE,
                      const float* Dv, void* dQ, const Shape& s, float scale, bool causal, int* status,
                      cudaStream_t st) {
  if (s.d == 64) return launch_dq<64>(Q, K, V, dO, LSE, Dv, dQ, s, scale, causal, status, st);
  if (s.d == 128) return launch_dq<128>(Q, K, V, dO, LSE, Dv, dQ, s, scale, causal, status, st);
  return cudaErrorInvalidValue;
}

}  // namespace fa
