// Attention backward on the tcgen05 tensor cores (bf16 in, fp32 accumulate); what it
// computes is fa_bwd in include/fa.h.
//
// Method ("flash-attention-backpropagation", 反向总览 / Softmax梯度 / QKV梯度): the
// outer loop runs over key/value tiles (one 128-key tile per CTA), the inner loop over
// 64-row query tiles; P is rebuilt from the forward's LSE, and one recompute of each
// (i, j) tile yields dV, dK and dQ together (the single-recompute loop the Ascend page
// "FlashAttention 反向传播" recommends over one pass per gradient). All accumulators are
// fp32 and are rounded to bf16 once, on write-back.
//
// Working in the transposed frame puts the 128 keys of the CTA on the 128 TMEM lanes:
//   S^T  = K_j Q_i^T          [keys x queries]   tcgen05, A,B = smem (K-major)
//   dP^T = V_j dO_i^T         [keys x queries]   tcgen05
//   P^T  = exp2(S^T * scale*log2e - LSE_i*log2e), masked (causal: key > query)
//   dS^T = P^T * (dP^T - D_i)                     softmax warps, one thread per key
//   dV_j += P^T dO_i          TMEM accumulator    A = P^T from TMEM
//   dK_j += dS^T Q_i          TMEM accumulator    A = dS^T from TMEM
//   dQ_i^T = K_j^T dS^T            (lanes = head dim)   A = K_j (MN-major), B = dS^T (smem, MN-major)
// and the dQ partials are added into an fp32 accumulator in global memory (red.add); a
// last pass scales it by `scale` and rounds to bf16. dQ^T is always an M = 128 product:
// at d = 64 its second 64-row atom of K^T reads the V tile that follows K in shared
// memory, and those rows land in TMEM lanes 64..127, which the dQ warps do not read.
//
// TMEM (512 columns): dV | dK | 2 buffers of (S^T | dP^T). Each softmax warpgroup
// writes its bf16 P^T over the S^T columns it has just read and its bf16 dS^T over the
// dP^T columns it has just read; the dQ partial of a tile then reuses its S^T columns
// once dV has consumed P^T. Query tiles are BQ = 64 rows, which leaves room for two
// buffers, so the softmax of tile i+1 overlaps the MMAs of tile i.
//
// CTA = 14 warps: 0-7 softmax (two warpgroups splitting the query columns), 8-11 dQ
// reduction + dK/dV epilogue, 12 TMA producer, 13 MMA issuer.
//
// Masks and dropout (kVar): the additive mask adds M log2(e) to each exponent; the
// boolean mask (packed bits, as the forward reads them) and dropout zero P for hidden or
// dropped keys, so their dS is 0 as well; kept dropout weights are scaled by 256 / (256 - t).
//
// Query and key lengths: Nq query rows against Nk key/value rows per head (Nq = Nk for
// fa_bwd); causal is bottom-right aligned (query i hides keys j > i + Nk - Nq), so a key
// tile starts at the first query tile that sees any of its keys (with this alignment every
// key is seen by the last query; a tile that no query saw would get dK = dV = 0). Queries
// that see no key (Nq > Nk) have LSE = -inf from the
// forward; every one of their keys is hidden by the causal rule, so their P is 0.
// Any lengths: Q/K/V/dO are read through [heads, rows, d] tensor maps (rows past the end of
// a head arrive as zeros), queries past the end get LSE = +inf (P = 0), and dQ/dK/dV rows
// past the end are neither accumulated nor stored.
#include <cuda_bf16.h>

#include "fa_internal.h"
#include "philox.cuh"
#include "sm100_ptx.cuh"
#include "tma_host.h"

namespace fa {
namespace {

using namespace ptx;

constexpr int BN = 128;  // keys per CTA
constexpr int kThreads = 448;
constexpr int kDqWarp0 = 8;
constexpr int kLoadWarp = 12;
constexpr int kMmaWarp = 13;
constexpr float kLog2e = 1.4426950408889634f;

struct BwdCtl {
  uint64_t kv_full, stage_full[3], stage_empty[3];
  uint64_t s_full[2], sm_done[2], dq_full, dq_empty, kv_done, drain;
  uint32_t tmem_base;
  int abort;
};

template <int D>
struct BwdCfg {
  static constexpr int BQ = 64;                      // queries per tile
  static constexpr int NB = 2;                       // S^T/dP^T buffers in TMEM
  static constexpr int kCols = BQ / 2;               // query columns per softmax warpgroup
  static constexpr int kBoxes = D / 64;              // 64-column boxes per row
  static constexpr int kKVBytes = BN * D * 2;        // K_j or V_j
  static constexpr int kQBox = BQ * 128;             // one [BQ x 64] box of Q_i / dO_i
  static constexpr int kQBytes = BQ * D * 2;
  static constexpr int kStages = 3;
  static constexpr int kDsBytes = BN * BQ * 2;       // dS^T [keys x queries] bf16, two buffers
  // shared-memory layout (1024-byte aligned base; control block last)
  static constexpr int kKOff = 0;
  static constexpr int kVOff = kKOff + kKVBytes;
  static constexpr int kStageOff = kVOff + kKVBytes;
  static constexpr int kStageBytes = 2 * kQBytes;    // Q_i then dO_i
  static constexpr int kDsOff = kStageOff + kStages * kStageBytes;
  static constexpr int kVecOff = kDsOff + 2 * kDsBytes;  // LSE_i, D_i per stage
  static constexpr int kVecBytes = 2 * BQ * 4;
  static constexpr int kCtlOff = kVecOff + kStages * kVecBytes;
  static constexpr int kSmemBytes = kCtlOff + (int)sizeof(BwdCtl);
  // TMEM columns
  static constexpr uint32_t kColDV = 0;
  static constexpr uint32_t kColDK = D;
  __device__ static constexpr uint32_t colS(int b) { return 2 * D + b * 2 * BQ; }
  __device__ static constexpr uint32_t colDP(int b) { return 2 * D + b * 2 * BQ + BQ; }
  static constexpr uint32_t kTmemCols = 512;
  static_assert(2 * D + NB * 2 * BQ <= 512, "TMEM budget");
  // the dQ^T partial (BQ columns) reuses a buffer's S^T columns; at d = 64 the M = 128
  // dQ^T product reads its second atom of K^T from the V tile right after K
  static_assert(kVOff == kKOff + kKVBytes || D == 128, "V follows K");
  static_assert(kSmemBytes <= 227 * 1024, "shared-memory budget");
};

struct BwdParams {
  const float* LSE;
  const float* Dvec;
  float* dQacc;
  __nv_bfloat16* dK;
  __nv_bfloat16* dV;
  int* status;
  int Nq;      // query rows per head
  int Nk;      // key / value rows per head
  int heads;
  int kvtiles;
  int qtiles;
  int causal;
  int offset;  // causal: query i hides keys j > i + offset (offset = Nk - Nq, bottom-right)
  float scale;
  float sl2;  // scale * log2(e)
  // additive mask (kMask): element (b, h, i, j) at mask[b*mask_sb + h*mask_sh + i*mask_srow + j]
  const __nv_bfloat16* mask;
  // boolean mask (kVar == 3): visibility bits, word (b, h, i, j / 32) at
  // bits[b*mask_sb + h*mask_sh + i*mask_srow + j / 32] (the same strides, in 32-bit words)
  const uint32_t* bits;
  int64_t mask_sb, mask_sh, mask_srow;
  int H;
  // dropout (kVar == 2): Philox key, keep threshold and the scale of a kept weight
  uint32_t seed_lo, seed_hi, drop_tt;  // drop_tt: the keep threshold in all four bytes
  float drop_scale;
};

// Transpose of a 32 x 32 bit matrix held one row per lane: on return lane T holds bit c =
// bit T of lane c's row. Five butterfly stages; the stage of width s swaps, between lanes
// l and l ^ s, the s-bit groups whose position differs from the lane in bit s.
__device__ __forceinline__ uint32_t transpose32(uint32_t x, int lane) {
  constexpr uint32_t kLow[5] = {0x0000FFFFu, 0x00FF00FFu, 0x0F0F0F0Fu, 0x33333333u, 0x55555555u};
#pragma unroll
  for (int k = 0; k < 5; ++k) {
    const int s = 16 >> k;
    const uint32_t m = kLow[k];  // bit positions p with (p & s) == 0
    const uint32_t y = __shfl_xor_sync(0xffffffffu, x, s);
    x = (lane & s) ? ((x & ~m) | ((y & ~m) >> s)) : ((x & m) | ((y & m) << s));
  }
  return x;
}

__device__ __forceinline__ void bulk_load(void* dst, const void* src, uint32_t bytes, uint64_t* bar) {
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(
          smem_u32(dst)),
      "l"(reinterpret_cast<uint64_t>(src)), "r"(bytes), "r"(smem_u32(bar))
      : "memory");
}

// TMEM column of the packed bf16 operand for query block k (16 queries) when each of the
// two softmax warpgroups packs its kCols queries into the first kCols/2 columns of its
// half of the buffer.
template <int kCols>
__device__ __forceinline__ uint32_t packed_col(uint32_t base, int k) {
  return base + (k / (kCols / 16)) * kCols + (k % (kCols / 16)) * 8;
}

// kTail: N is not a multiple of the tiles, so the partial-tile guards are compiled in; the
// instance for whole tiles carries none of them.
// kVar: 0 plain, 1 additive mask, 2 dropout, 3 boolean mask (packed bits).
template <int D, bool kTail, int kVar>
__global__ void __launch_bounds__(kThreads, 1)
fa_bwd_tc_kernel(const __grid_constant__ CUtensorMap tmQ, const __grid_constant__ CUtensorMap tmK,
                 const __grid_constant__ CUtensorMap tmV, const __grid_constant__ CUtensorMap tmdO,
                 const BwdParams p) {
  using C = BwdCfg<D>;
  constexpr bool kMask = kVar == 1;
  constexpr bool kDrop = kVar == 2;
  constexpr bool kBits = kVar == 3;
  constexpr int BQ = C::BQ;
  extern __shared__ __align__(1024) uint8_t smem[];
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  // The swizzled operand layout needs a 1024-byte aligned base; the runtime provides it
  // for this declaration, and the kernel refuses to run (status word) if it did not.
  if ((smem_u32(smem) & 1023u) != 0) {
    if (threadIdx.x == 0 && p.status) atomicExch(p.status, 3 /* FA_ERR_CUDA */);
    return;
  }
  BwdCtl& ctl = *reinterpret_cast<BwdCtl*>(smem + C::kCtlOff);

  int kt, head;
  if (p.causal) {  // key tiles near the start see the most queries: launch them first
    kt = (int)(blockIdx.x / p.heads);
    head = (int)(blockIdx.x % p.heads);
  } else {
    kt = (int)(blockIdx.x % p.kvtiles);
    head = (int)(blockIdx.x / p.kvtiles);
  }
  const int qrow_base = head * p.Nq;  // LSE, D and dQ rows of the head
  const int krow_base = head * p.Nk;  // dK and dV rows of the head
  // causal: the first query tile holding a query that sees key kt * BN (query + offset >= key)
  const int q_first = p.causal ? max(0, kt * BN - p.offset) / BQ : 0;
  const int nq = p.qtiles - q_first;
  if (nq <= 0) {
    // No query sees a key of this tile (causal with more keys past the last query's limit
    // than the tile start): dK = dV = 0 for its rows, nothing else to do.
    if (threadIdx.x < BN && kt * BN + (int)threadIdx.x < p.Nk) {
      const size_t row = (size_t)krow_base + kt * BN + threadIdx.x;
      uint4* dk = reinterpret_cast<uint4*>(p.dK + row * D);
      uint4* dv = reinterpret_cast<uint4*>(p.dV + row * D);
#pragma unroll
      for (int u = 0; u < D / 8; ++u) dk[u] = dv[u] = make_uint4(0, 0, 0, 0);
    }
    return;
  }

  if (threadIdx.x == 0) {
    mbar_init(&ctl.kv_full, 1);
    for (int s = 0; s < C::kStages; ++s) {
      mbar_init(&ctl.stage_full[s], 1);
      mbar_init(&ctl.stage_empty[s], 1);
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(&ctl.s_full[b], 1);
      mbar_init(&ctl.sm_done[b], 256);
    }
    mbar_init(&ctl.dq_full, 1);
    mbar_init(&ctl.dq_empty, 128);
    mbar_init(&ctl.kv_done, 1);
    mbar_init(&ctl.drain, 1);
    ctl.abort = 0;
    fence_mbar_init();
  }
  if (warp == kMmaWarp) tmem_alloc(&ctl.tmem_base, C::kTmemCols);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = ctl.tmem_base;
  volatile int* abort = &ctl.abort;
  uint8_t* sK = smem + C::kKOff;
  uint8_t* sV = smem + C::kVOff;

  if (warp == kLoadWarp) {
    // Lane 0 drives the TMA copies and the barriers. LSE_i and D_i of a full tile whose
    // rows start 16-byte aligned arrive by bulk copy with the stage; otherwise (the last,
    // partial tile of a head, or N not a multiple of 4) the warp stages them with
    // bounds-checked loads before lane 0 arms the stage: queries past the end of the
    // head get LSE = +inf and D = 0, so their P and dS are exactly zero.
    if (lane == 0) {
      prefetch_tmap(&tmQ);
      prefetch_tmap(&tmK);
      prefetch_tmap(&tmV);
      prefetch_tmap(&tmdO);
      mbar_expect_tx(&ctl.kv_full, 2 * C::kKVBytes);
      for (int b = 0; b < C::kBoxes; ++b) {
        tma_load_3d(sK + b * (BN * 128), &tmK, &ctl.kv_full, b * 64, kt * BN, head);
        tma_load_3d(sV + b * (BN * 128), &tmV, &ctl.kv_full, b * 64, kt * BN, head);
      }
    }
    int last[3] = {-1, -1, -1};
    // Test hook of the failure path: never arm the first Q/dO stage, so the MMA thread's
    // wait for it runs out (see StatusBlock); off unless a test sets it.
    const bool skip_first = injected(p.status, kInjectBwd);
    // When every tile of the head takes the bulk path, lane 0 runs the loop alone.
    const bool all_bulk = !kTail || ((p.Nq % BQ) == 0 && (p.Nq % 4) == 0);
    for (int it = 0; it < nq && (lane == 0 || !all_bulk); ++it) {
      const int s = it % C::kStages;
      bool ok = true;
      if (lane == 0 && it >= C::kStages)
        ok = mbar_wait(&ctl.stage_empty[s], ((it / C::kStages) - 1) & 1, p.status, abort);
      if (!all_bulk) ok = __shfl_sync(0xffffffffu, ok ? 1 : 0, 0) != 0;
      if (!ok) break;
      const int q0 = (q_first + it) * BQ;  // first query of the tile, within the head
      uint8_t* st = smem + C::kStageOff + s * C::kStageBytes;
      float* vec = reinterpret_cast<float*>(smem + C::kVecOff + s * C::kVecBytes);
      const bool bulk = !kTail || (q0 + BQ <= p.Nq && (p.Nq % 4) == 0);
      if (!bulk) {
        for (int c = lane; c < BQ; c += 32) {
          const bool in = q0 + c < p.Nq;
          vec[c] = in ? p.LSE[qrow_base + q0 + c] : INFINITY;
          vec[BQ + c] = in ? p.Dvec[qrow_base + q0 + c] : 0.f;
        }
        __syncwarp();
      }
      if (it == 0 && skip_first) continue;
      if (lane == 0) {
        mbar_expect_tx(&ctl.stage_full[s], C::kStageBytes + (bulk ? C::kVecBytes : 0));
        for (int b = 0; b < C::kBoxes; ++b) {
          tma_load_3d(st + b * C::kQBox, &tmQ, &ctl.stage_full[s], b * 64, q0, head);
          tma_load_3d(st + C::kQBytes + b * C::kQBox, &tmdO, &ctl.stage_full[s], b * 64, q0, head);
        }
        if (bulk) {
          bulk_load(vec, p.LSE + qrow_base + q0, BQ * 4, &ctl.stage_full[s]);
          bulk_load(vec + BQ, p.Dvec + qrow_base + q0, BQ * 4, &ctl.stage_full[s]);
        }
      }
      last[s] = it;
    }
    if (lane == 0) {
      mbar_wait(&ctl.kv_full, 0, p.status, nullptr);
      for (int s = 0; s < C::kStages; ++s)
        if (last[s] >= 0) mbar_wait(&ctl.stage_full[s], (last[s] / C::kStages) & 1, p.status, nullptr);
    }
  } else if (warp == kMmaWarp) {
    if (lane == 0) {
      constexpr uint32_t idSP = idesc_bf16(BN, BQ, false, false);   // S^T, dP^T
      constexpr uint32_t idKV = idesc_bf16(BN, D, false, true);     // dV, dK
      constexpr uint32_t idQ = idesc_bf16(128, BQ, true, true);    // dQ^T: M = 128 rows of the head dim
      const uint32_t aK = smem_u32(sK), aV = smem_u32(sV);
      const uint32_t aStage = smem_u32(smem + C::kStageOff);
      const uint32_t aDs = smem_u32(smem + C::kDsOff);
      // Base descriptors; each MMA below only advances the start address.
      const uint64_t dK_k = sdesc_sw128(aK, 16, 1024);            // K_j, K-major (rows = keys)
      const uint64_t dK_mn = sdesc_sw128(aK, BN * 128, 1024);     // K_j read as K_j^T / MN-major
      const uint64_t dV_k = sdesc_sw128(aV, 16, 1024);
      auto stage_desc = [&](int s, bool dO, bool mn) {
        const uint32_t a = aStage + s * C::kStageBytes + (dO ? C::kQBytes : 0);
        return mn ? sdesc_sw128(a, C::kQBox, 1024) : sdesc_sw128(a, 16, 1024);
      };
      auto issue_S = [&](int s, int b) {
        const uint64_t qd = stage_desc(s, false, false);
#pragma unroll
        for (int k = 0; k < D / 16; ++k)
          mma_ss(tmem + C::colS(b), sdesc_add(dK_k, (k / 4) * (BN * 128) + (k % 4) * 32),
                 sdesc_add(qd, (k / 4) * C::kQBox + (k % 4) * 32), idSP, k > 0);
      };
      auto issue_dP = [&](int s, int b) {
        const uint64_t od = stage_desc(s, true, false);
#pragma unroll
        for (int k = 0; k < D / 16; ++k)
          mma_ss(tmem + C::colDP(b), sdesc_add(dV_k, (k / 4) * (BN * 128) + (k % 4) * 32),
                 sdesc_add(od, (k / 4) * C::kQBox + (k % 4) * 32), idSP, k > 0);
      };
      auto issue_dV_dK = [&](int it, int b, int s, bool which_dk) {
        // dV += P^T dO_i or dK += dS^T Q_i (K = queries; A = packed bf16 in TMEM)
        const uint64_t bd = stage_desc(s, !which_dk, true);
        const uint32_t acc_col = which_dk ? C::kColDK : C::kColDV;
        const uint32_t a_col = which_dk ? C::colDP(b) : C::colS(b);
#pragma unroll
        for (int k = 0; k < BQ / 16; ++k)
          mma_ts(tmem + acc_col, packed_col<C::kCols>(tmem + a_col, k), sdesc_add(bd, k * 2048), idKV,
                 (it > 0 || k > 0) ? 1u : 0u);
      };
      auto issue_dQ = [&](int b, int dsbuf) {
        // dQ partial (K = keys) over this buffer's S^T columns (P^T was read by dV, in
        // issue order).
        const uint64_t dsd = sdesc_sw128(aDs + dsbuf * C::kDsBytes, BN * 128, 1024);
#pragma unroll
        for (int k = 0; k < BN / 16; ++k)
          mma_ss(tmem + C::colS(b), sdesc_add(dK_mn, k * 2048), sdesc_add(dsd, k * 2048), idQ, k > 0);
      };
      bool ok = mbar_wait(&ctl.kv_full, 0, p.status, abort);
      // Issue order per tile i (buffer b = i % 2):
      //   dV(i), S(i+1), dK(i), dQ(i), dP(i+2)
      // S(i+1) lands in the columns that held the partial dQ(i-1); placing dP(i+1) and
      // dV(i) ahead of it gives the dQ warpgroup time to read that partial out, and the
      // softmax of tile i+1 runs while dK(i), dQ(i) and dP(i+2) execute.
      if (ok && nq > 0 && (ok = mbar_wait(&ctl.stage_full[0], 0, p.status, abort))) {
        tc_fence_after();
        issue_S(0, 0);
        issue_dP(0, 0);
        mma_commit(&ctl.s_full[0]);
      }
      if (ok && nq > 1 && (ok = mbar_wait(&ctl.stage_full[1], 0, p.status, abort))) {
        tc_fence_after();
        issue_dP(1, 1);
      }
      for (int it = 0; ok && it < nq; ++it) {
        const int s = it % C::kStages;
        const int b = it & 1;
        if (!(ok = mbar_wait(&ctl.sm_done[b], (it / 2) & 1, p.status, abort))) break;
        tc_fence_after();
        issue_dV_dK(it, b, s, false);
        // The previous partial dQ(i-1) sits in buffer b^1's S^T columns; it must have been
        // read out before S(i+1) overwrites them (and before dQ(i) is handed off, so the
        // two hand-off barriers stay one phase apart).
        if (it > 0 && !(ok = mbar_wait(&ctl.dq_empty, (it - 1) & 1, p.status, abort))) break;
        tc_fence_after();
        if (it + 1 < nq) {
          issue_S((it + 1) % C::kStages, b ^ 1);  // stage it+1 was waited for with dP(i+1)
          mma_commit(&ctl.s_full[b ^ 1]);
        }
        issue_dV_dK(it, b, s, true);
        issue_dQ(b, it & 1);
        mma_commit(&ctl.dq_full);
        if constexpr (D != 128) mma_commit(&ctl.stage_empty[s]);  // at d = 128 the dQ warps free it
        if (it + 2 < nq) {
          const int s2 = (it + 2) % C::kStages;
          if (!(ok = mbar_wait(&ctl.stage_full[s2], ((it + 2) / C::kStages) & 1, p.status, abort))) break;
          tc_fence_after();
          issue_dP(s2, b);  // dP^T columns of buffer b: dS^T was read by dK above (issue order)
        }
      }
      mma_commit(&ctl.kv_done);
      mma_commit(&ctl.drain);
      mbar_wait(&ctl.drain, 0, p.status, nullptr);
    }
  } else if (warp < kDqWarp0) {
    // ---------------- softmax-backward warpgroups ----------------
    constexpr int kCols = C::kCols;
    const int wg = warp >> 2;
    const int r = (warp & 3) * 32 + lane;         // key row in the tile = TMEM lane
    const int key = kt * BN + r;
    const uint32_t lane_off = (uint32_t)((warp & 3) * 32) << 16;
    const float2 sl2 = make_float2(p.sl2, p.sl2);
    const float2 neg_log2e = make_float2(-kLog2e, -kLog2e);
    const float2 minus1 = make_float2(-1.f, -1.f);
    // kBits: the warp's 32 keys are one word of each query's row. Lane L reads the word of
    // query (tile start + this warpgroup's first column + L), one tile ahead, so that the
    // load's latency hides behind the current tile.
    static_assert(!kBits || kCols == 32, "one 32-query chunk per tile");
    const int kword = (kt * BN + (warp & 3) * 32) >> 5;
    const uint32_t* bcol =
        kBits ? p.bits + (int64_t)(head / p.H) * p.mask_sb + (int64_t)(head % p.H) * p.mask_sh + kword : nullptr;
    auto bits_word = [&](int it) -> uint32_t {
      const int q = (q_first + it) * BQ + wg * kCols + lane;
      return (it < nq && (!kTail || (q < p.Nq && kword * 32 < p.Nk))) ? bcol[(int64_t)q * p.mask_srow] : 0u;
    };
    uint32_t bword = kBits ? bits_word(0) : 0u;
    bool ok = true;
    for (int it = 0; ok && it < nq; ++it) {
      const int s = it % C::kStages;
      const int b = it % C::NB;
      const uint32_t bcur = bword;
      if constexpr (kBits) bword = bits_word(it + 1);
      ok = __all_sync(0xffffffffu, mbar_wait(&ctl.s_full[b], (it / C::NB) & 1, p.status, abort));
      if (!ok) break;
      tc_fence_after();
      const float* vec = reinterpret_cast<const float*>(smem + C::kVecOff + s * C::kVecBytes);
      const int q0 = (q_first + it) * BQ;
      // some key of the tile exceeds the limit of some query of the tile
      const bool diag = p.causal && q0 + p.offset < kt * BN + BN - 1;
      uint8_t* dsrow = smem + C::kDsOff + (it & 1) * C::kDsBytes + r * 128;
#pragma unroll
      for (int ch = 0; ch < kCols / 32; ++ch) {
        const int c0 = wg * kCols + ch * 32;  // first query column of this chunk
        // kMask: M(query, this key) * log2(e) for the chunk's 32 queries; across the warp
        // each load reads 32 consecutive keys of one mask row. Issued before the TMEM loads
        // so that their latency overlaps.
        float mk[kMask ? 32 : 1];
        if constexpr (kMask) {
          const __nv_bfloat16* mcol = p.mask + (int64_t)(head / p.H) * p.mask_sb +
                                      (int64_t)(head % p.H) * p.mask_sh + key;
#pragma unroll
          for (int c = 0; c < 32; ++c) {
            const int q = q0 + c0 + c;
            mk[c] = (!kTail || (key < p.Nk && q < p.Nq))
                        ? __bfloat162float(mcol[(int64_t)q * p.mask_srow]) * kLog2e
                        : 0.f;
          }
        }
        // kDrop: keep bits of this thread's key against the chunk's 32 queries. Lane L draws
        // the bits of query (chunk start + L) against the warp's 32 keys (2 Philox blocks of
        // 16 keys); transposing that 32 x 32 bit block leaves lane T with bit c =
        // keep(query c, key T).
        uint32_t kbits = 0;
        if constexpr (kDrop) {
          const uint32_t i = (uint32_t)(q0 + c0 + lane);
          const uint32_t blk0 = (uint32_t)((kt * BN + (warp & 3) * 32) >> 4);
          const uint32_t row = rng::keep16(blk0, i, (uint32_t)head, p.seed_lo, p.seed_hi, p.drop_tt) |
                               (rng::keep16(blk0 + 1, i, (uint32_t)head, p.seed_lo, p.seed_hi, p.drop_tt) << 16);
          kbits = transpose32(row, lane);
        }
        // kBits: transposing the 32 lanes' words (prefetched above) leaves lane T with
        // bit c = visible(query c of the chunk, key T).
        const uint32_t vbits = kBits ? transpose32(bcur, lane) : 0u;
        float sv[32], dp[32];
        tmem_ld32x2(tmem + lane_off + C::colS(b) + c0, tmem + lane_off + C::colDP(b) + c0, sv, dp);
        // -LSE*log2(e) and D for the 32 columns, loaded as 16-byte vectors up front
        float2 nl[16], dv[16];
#pragma unroll
        for (int u = 0; u < 8; ++u) {
          const float4 a = *reinterpret_cast<const float4*>(vec + c0 + 4 * u);
          const float4 b = *reinterpret_cast<const float4*>(vec + BQ + c0 + 4 * u);
          nl[2 * u] = fmul2(make_float2(a.x, a.y), neg_log2e);
          nl[2 * u + 1] = fmul2(make_float2(a.z, a.w), neg_log2e);
          if constexpr (kMask || kBits) {  // a query with no visible key (LSE = -inf) has P = 0
            if (a.x == -INFINITY) nl[2 * u].x = -INFINITY;
            if (a.y == -INFINITY) nl[2 * u].y = -INFINITY;
            if (a.z == -INFINITY) nl[2 * u + 1].x = -INFINITY;
            if (a.w == -INFINITY) nl[2 * u + 1].y = -INFINITY;
          }
          dv[2 * u] = make_float2(b.x, b.y);
          dv[2 * u + 1] = make_float2(b.z, b.w);
        }
        uint32_t pk[16], dk[16];
#pragma unroll
        for (int u = 0; u < 16; ++u) {
          const int c = c0 + 2 * u;
          float2 x = ffma2(make_float2(sv[2 * u], sv[2 * u + 1]), sl2, nl[u]);
          if constexpr (kMask) x = fadd2(x, make_float2(mk[2 * u], mk[2 * u + 1]));
          float2 pr = make_float2(ex2(x.x), ex2(x.y));
          if constexpr (kBits) {  // a hidden key has P = 0, and so dS = 0
            if (!((vbits >> (2 * u)) & 1u)) pr.x = 0.f;
            if (!((vbits >> (2 * u + 1)) & 1u)) pr.y = 0.f;
          }
          if (diag) {
            if (key > q0 + c + p.offset) pr.x = 0.f;
            if (key > q0 + c + 1 + p.offset) pr.y = 0.f;
          }
          float2 dd;
          if constexpr (kDrop) {  // dP of a dropped key is 0; a kept one is scaled
            const bool k0 = (kbits >> (2 * u)) & 1u, k1 = (kbits >> (2 * u + 1)) & 1u;
            dd = make_float2(k0 ? fmaf(dp[2 * u], p.drop_scale, -dv[u].x) : -dv[u].x,
                             k1 ? fmaf(dp[2 * u + 1], p.drop_scale, -dv[u].y) : -dv[u].y);
            pk[u] = pack_bf16(k0 ? pr.x : 0.f, k1 ? pr.y : 0.f);  // dV takes the kept weights
          } else {
            dd = ffma2(dv[u], minus1, make_float2(dp[2 * u], dp[2 * u + 1]));
            pk[u] = pack_bf16(pr.x, pr.y);
          }
          const float2 dsv = fmul2(pr, dd);
          dk[u] = pack_bf16(dsv.x, dsv.y);
        }
        // bf16 P^T over S^T and dS^T over dP^T, in columns this warpgroup has already read
        tmem_st16(tmem + lane_off + C::colS(b) + wg * kCols + ch * 16, pk);
        tmem_st16(tmem + lane_off + C::colDP(b) + wg * kCols + ch * 16, dk);
        // dS^T row r, columns c0..c0+31: four 16-byte chunks of a 128-byte swizzled row
        // (atom column c0 / 64, chunk (c0 % 64) / 8 + u, XOR (r % 8)).
        uint8_t* atom = dsrow + (c0 / 64) * (BN * 128);
#pragma unroll
        for (int u = 0; u < 4; ++u) {
          const int chunk = ((c0 % 64) / 8 + u) ^ (r & 7);
          *reinterpret_cast<uint4*>(atom + chunk * 16) =
              make_uint4(dk[4 * u], dk[4 * u + 1], dk[4 * u + 2], dk[4 * u + 3]);
        }
      }
      tmem_wait_st();
      fence_proxy_async_smem();
      tc_fence_before();
      mbar_arrive(&ctl.sm_done[b]);
    }
  } else if (warp < kLoadWarp) {
    // ---------------- dQ reduction, then the dK/dV epilogue ----------------
    const int r = (warp & 3) * 32 + lane;  // TMEM lane
    const uint32_t lane_off = (uint32_t)((warp & 3) * 32) << 16;
    bool ok = true;
    for (int it = 0; ok && it < nq; ++it) {
      ok = __all_sync(0xffffffffu, mbar_wait(&ctl.dq_full, it & 1, p.status, abort));
      if (!ok) break;
      tc_fence_after();
      // dq_full(i) follows every MMA that reads the Q/dO stage of tile i (S, dP, dV, dK), so
      // at d = 128 one dQ thread frees that stage here instead of a separate MMA commit: one
      // commit fewer per tile, measured 1% faster at d = 128 (and 2% slower at d = 64).
      if (D == 128 && warp == kDqWarp0 && lane == 0) mbar_arrive(&ctl.stage_empty[it % C::kStages]);
      const int q0 = qrow_base + (q_first + it) * BQ;
      const int nvalid = p.Nq - (q_first + it) * BQ;  // queries of the tile inside the head
      const uint32_t colQ = C::colS(it % C::NB);
      // lane = head-dim index r; columns = the BQ queries of the tile, released as soon as
      // they are in registers
      static_assert(BQ == 64, "one 64-column drain per tile");
      float v[BQ];
      tmem_ld32x2(tmem + lane_off + colQ, tmem + lane_off + colQ + 32, *reinterpret_cast<float(*)[32]>(&v[0]),
                  *reinterpret_cast<float(*)[32]>(&v[32]));
      tc_fence_before();
      mbar_arrive(&ctl.dq_empty);
      // At d = 64, TMEM lanes 64..127 (the warps with warp % 4 >= 2) hold no head-dim row:
      // those warps skip the reductions, a branch that is uniform over each warp.
      if (D == 128 || r < D) {
        float* dst = p.dQacc + (size_t)q0 * D + r;
        // Keep the bound test out of the reduction loop: a predicate inside it makes the
        // compiler serialise the reductions (measured 1.7x slower backward). Both loops
        // unroll fully, so v stays in registers: a partial unroll indexes v at run time
        // and moves it to local memory (2-4% slower backward).
        if (!kTail || BQ <= nvalid) {
#pragma unroll
          for (int c = 0; c < BQ; ++c) atomicAdd(dst + (size_t)c * D, v[c]);
        } else {  // the last, partial tile of a head
#pragma unroll
          for (int c = 0; c < BQ; ++c)
            if (c < nvalid) atomicAdd(dst + (size_t)c * D, v[c]);
        }
      }
    }
    if (ok) ok = __all_sync(0xffffffffu, mbar_wait(&ctl.kv_done, 0, p.status, abort));
    if (ok) {
      tc_fence_after();
      const size_t row = (size_t)krow_base + kt * BN + r;
      const bool in = !kTail || kt * BN + r < p.Nk;  // key rows past the end are not stored
#pragma unroll 1
      for (int c0 = 0; c0 < D; c0 += 32) {
        float v[32];
        uint4 w[4];
        uint32_t* wu = reinterpret_cast<uint32_t*>(w);
        tmem_ld32(tmem + lane_off + C::kColDV + c0, v);
        const float vs = kDrop ? p.drop_scale : 1.f;  // kept weights entered dV unscaled
#pragma unroll
        for (int u = 0; u < 16; ++u) wu[u] = pack_bf16(v[2 * u] * vs, v[2 * u + 1] * vs);
        uint4* dv = reinterpret_cast<uint4*>(p.dV + row * D + c0);
        if (in) {
#pragma unroll
          for (int u = 0; u < 4; ++u) dv[u] = w[u];
        }
        tmem_ld32(tmem + lane_off + C::kColDK + c0, v);
#pragma unroll
        for (int u = 0; u < 16; ++u) wu[u] = pack_bf16(v[2 * u] * p.scale, v[2 * u + 1] * p.scale);
        uint4* dk = reinterpret_cast<uint4*>(p.dK + row * D + c0);
        if (in) {
#pragma unroll
          for (int u = 0; u < 4; ++u) dk[u] = w[u];
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
    tmem_dealloc(tmem, C::kTmemCols);
  }
}

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

struct MaskArg {
  const void* ptr = nullptr;
  int64_t sb = 0, sh = 0, srow = 0;
};

struct DropArg {
  uint64_t seed = 0;
  uint32_t t = 0;
};

// The 64-query-tile kernel: every call with a mask or dropout.
template <int D, int kVar>
cudaError_t launch_narrow(const void* Q, const void* K, const void* V, const void* dO, const float* LSE,
                          const float* Dv, void* dQ, void* dK, void* dV, float* dQacc, const Shape& s,
                          float scale, bool causal, const MaskArg& mask, const DropArg& drop, int* status,
                          cudaStream_t st) {
  using C = BwdCfg<D>;
  CUtensorMap mq, mk, mv, mdo;
  const int64_t heads = s.heads();
  if (!make_map_bf16_3d(&mq, Q, heads, s.N, D, C::BQ) || !make_map_bf16_3d(&mk, K, heads, s.keys(), D, BN) ||
      !make_map_bf16_3d(&mv, V, heads, s.keys(), D, BN) || !make_map_bf16_3d(&mdo, dO, heads, s.N, D, C::BQ))
    return cudaErrorInvalidValue;
  static bool attr = [] {
    return cudaFuncSetAttribute(fa_bwd_tc_kernel<D, false, kVar>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                C::kSmemBytes) == cudaSuccess &&
           cudaFuncSetAttribute(fa_bwd_tc_kernel<D, true, kVar>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                C::kSmemBytes) == cudaSuccess;
  }();
  if (!attr) return cudaErrorInvalidConfiguration;
  cudaError_t e = cudaMemsetAsync(dQacc, 0, (size_t)s.elems() * sizeof(float), st);
  if (e != cudaSuccess) return e;
  BwdParams p;
  p.LSE = LSE;
  p.Dvec = Dv;
  p.dQacc = dQacc;
  p.dK = static_cast<__nv_bfloat16*>(dK);
  p.dV = static_cast<__nv_bfloat16*>(dV);
  p.status = status;
  p.Nq = s.N;
  p.Nk = s.keys();
  p.heads = (int)s.heads();
  p.kvtiles = (s.keys() + BN - 1) / BN;
  p.qtiles = (s.N + C::BQ - 1) / C::BQ;
  p.causal = causal ? 1 : 0;
  p.offset = causal ? s.keys() - s.N : 0;
  p.scale = scale;
  p.sl2 = scale * kLog2e;
  p.mask = static_cast<const __nv_bfloat16*>(mask.ptr);
  p.bits = static_cast<const uint32_t*>(mask.ptr);
  p.mask_sb = mask.sb;
  p.mask_sh = mask.sh;
  p.mask_srow = mask.srow;
  p.H = s.H;
  p.seed_lo = (uint32_t)(drop.seed & 0xFFFFFFFFu);
  p.seed_hi = (uint32_t)(drop.seed >> 32);
  p.drop_tt = drop.t * 0x01010101u;
  p.drop_scale = (float)(256.0 / (256.0 - (double)drop.t));
  const int64_t grid = (int64_t)p.kvtiles * p.heads;
  if (s.N % 128 != 0 || s.keys() % 128 != 0)
    fa_bwd_tc_kernel<D, true, kVar><<<(unsigned)grid, kThreads, C::kSmemBytes, st>>>(mq, mk, mv, mdo, p);
  else
    fa_bwd_tc_kernel<D, false, kVar><<<(unsigned)grid, kThreads, C::kSmemBytes, st>>>(mq, mk, mv, mdo, p);
  if ((e = cudaGetLastError()) != cudaSuccess) return e;
  const int64_t n8 = s.elems() / 8;
  dq_convert_kernel<<<(unsigned)((n8 + 255) / 256), 256, 0, st>>>(dQacc, static_cast<__nv_bfloat16*>(dQ),
                                                                  n8, scale);
  return cudaGetLastError();
}

template <int D, int kVar>
cudaError_t launch(const void* Q, const void* K, const void* V, const void* dO, const float* LSE,
                   const float* Dv, void* dQ, void* dK, void* dV, float* dQacc, const Shape& s,
                   float scale, bool causal, const MaskArg& mask, const DropArg& drop, int* status,
                   cudaStream_t st) {
  if constexpr (kVar == 0) {
    // no mask or dropout: the 128-query-tile kernel (fa_bwd_wide.cu)
    cudaError_t e = cudaMemsetAsync(dQacc, 0, (size_t)s.elems() * sizeof(float), st);
    if (e != cudaSuccess) return e;
    if ((e = tc_bwd_wide(Q, K, V, dO, LSE, Dv, dK, dV, dQacc, s, scale, causal, status, st)) != cudaSuccess) return e;
    const int64_t n8 = s.elems() / 8;
    dq_convert_kernel<<<(unsigned)((n8 + 255) / 256), 256, 0, st>>>(dQacc, static_cast<__nv_bfloat16*>(dQ), n8, scale);
    return cudaGetLastError();
  } else {
    return launch_narrow<D, kVar>(Q, K, V, dO, LSE, Dv, dQ, dK, dV, dQacc, s, scale, causal, mask, drop, status, st);
  }
}

}  // namespace

cudaError_t tc_bwd(const void* Q, const void* K, const void* V, const void* dO, const float* LSE,
                   const float* D, void* dQ, void* dK, void* dV, float* dQacc, const Shape& s,
                   float scale, bool causal, int* status, cudaStream_t st) {
  const MaskArg none;
  const DropArg nodrop;
  return s.d == 64
             ? launch<64, 0>(Q, K, V, dO, LSE, D, dQ, dK, dV, dQacc, s, scale, causal, none, nodrop, status, st)
             : launch<128, 0>(Q, K, V, dO, LSE, D, dQ, dK, dV, dQacc, s, scale, causal, none, nodrop, status, st);
}

cudaError_t tc_bwd_masked(const void* Q, const void* K, const void* V, const void* dO, const float* LSE,
                          const float* D, void* dQ, void* dK, void* dV, float* dQacc, const Shape& s,
                          float scale, bool causal, const void* mask, int64_t mask_sb, int64_t mask_sh,
                          int64_t mask_srow, int* status, cudaStream_t st) {
  MaskArg m;
  m.ptr = mask;
  m.sb = mask_sb;
  m.sh = mask_sh;
  m.srow = mask_srow;
  const DropArg nodrop;
  return s.d == 64
             ? launch<64, 1>(Q, K, V, dO, LSE, D, dQ, dK, dV, dQacc, s, scale, causal, m, nodrop, status, st)
             : launch<128, 1>(Q, K, V, dO, LSE, D, dQ, dK, dV, dQacc, s, scale, causal, m, nodrop, status, st);
}

cudaError_t tc_bwd_bitmask(const void* Q, const void* K, const void* V, const void* dO, const float* LSE,
                           const float* D, void* dQ, void* dK, void* dV, float* dQacc, const Shape& s,
                           float scale, bool causal, const uint32_t* bits, int64_t bits_sb, int64_t bits_sh,
                           int64_t bits_srow, int* status, cudaStream_t st) {
  MaskArg m;
  m.ptr = bits;
  m.sb = bits_sb;
  m.sh = bits_sh;
  m.srow = bits_srow;
  const DropArg nodrop;
  return s.d == 64
             ? launch<64, 3>(Q, K, V, dO, LSE, D, dQ, dK, dV, dQacc, s, scale, causal, m, nodrop, status, st)
             : launch<128, 3>(Q, K, V, dO, LSE, D, dQ, dK, dV, dQacc, s, scale, causal, m, nodrop, status, st);
}

cudaError_t tc_bwd_dropout(const void* Q, const void* K, const void* V, const void* dO, const float* LSE,
                           const float* D, void* dQ, void* dK, void* dV, float* dQacc, const Shape& s,
                           float scale, bool causal, uint64_t seed, uint32_t threshold, int* status,
                           cudaStream_t st) {
  const MaskArg none;
  DropArg dr;
  dr.seed = seed;
  dr.t = threshold;
  return s.d == 64
             ? launch<64, 2>(Q, K, V, dO, LSE, D, dQ, dK, dV, dQacc, s, scale, causal, none, dr, status, st)
             : launch<128, 2>(Q, K, V, dO, LSE, D, dQ, dK, dV, dQacc, s, scale, causal, none, dr, status, st);
}

}  // namespace fa
