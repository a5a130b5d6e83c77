// Attention backward on 128-query tiles, head dimension 64 or 128 (bf16 in, fp32 accumulate);
// what it computes is fa_bwd in include/fa.h, and fa_bwd_masked, fa_bwd_bitmask and
// fa_bwd_dropout with their mask or dropout (the kVar instances).
//
// Method ("flash-attention-backpropagation", 反向总览 / Softmax梯度 / QKV梯度; the single
// recompute per tile of "FlashAttention 反向传播" 踩坑二): a work item is a 128-key tile of
// one head, whose CTA loops over the 128-row query tiles that see it; P is rebuilt from the
// forward's LSE, and each recompute of a tile feeds dV, dK and dQ.
//
// Keys sit on the 128 TMEM lanes, so dV and dK accumulate in TMEM:
//   S^T  = K_j Q_i^T                 [keys x queries]  tcgen05, A, B from smem (K-major)
//   dP^T = V_j dO_i^T                [keys x queries]  tcgen05
//   P^T  = exp2(S^T * scale*log2e - LSE_i*log2e)       softmax warps, phase A
//   dS^T = P^T * (dP^T - D_i)                          softmax warps, phase B
//   dV_j += P^T dO_i                 A = P^T from TMEM (bf16, packed over S^T)
//   dK_j += dS^T Q_i                 A = dS^T from smem (K-major)
//   dQ_i^T = K_j^T dS^T              [head dim x queries]  A = K_j (MN-major), B = dS^T (MN-major)
// and every dQ partial is added into an fp32 accumulator in global memory (red.add); a
// last pass scales it by `scale` and rounds it to bf16 (fa_bwd_tc.cu).
//
// Every product is M = 128, N = 128: a tcgen05.mma of that shape runs at the full math
// rate, while the N = 64 products of 64-query tiles are bound by shared-memory operand
// reads. The price is TMEM room: dV | dK | S^T | dP^T fill the 512 columns, so there is one
// S^T and one dP^T buffer. The softmax is therefore split in two phases, so that the
// tensor core always has a product that does not wait for it:
//   phase A (needs S^T):  P^T, written over S^T in TMEM (dV reads it from there);
//   phase B (needs dP^T): dS^T, written to shared memory only (dK and dQ read it there),
//                         which frees the dP^T columns for the dQ^T partial.
// Issue order for tile i (all products of a tile after its own inputs, in this order):
//   S(i+1) | dK(i) dQ(i) | dV(i+1) | dP(i+1)
// so phase A of tile i+1 runs beside dK(i) and dQ(i), the softmax warps read the dQ(i)
// partial out of the dP^T columns beside dV(i+1), and phase B of tile i+1 runs beside S(i+2).
// At d = 64 the dQ^T partial has TMEM columns of its own (dV and dK take 64 each, which
// leaves 128 free), and the separate dQ mode has no dQ product at all: there nothing waits
// for the dP^T columns but dP itself, and the order is
//   S(i+1) | dK(i) dQ(i) | dP(i+1) | dV(i+1)
// so that phase B of tile i+1, which needs only dP(i+1), runs beside dV(i+1) and S(i+2).
//
// CTA = 10 warps: 0-7 softmax (two warpgroups over query columns 0-63 and 64-127; a thread
// owns one key row = TMEM lane), which also read the dQ^T partials out of TMEM (between
// phases A and B, when they would otherwise wait) and write dK and dV at the end; 8 TMA
// producer; 9 MMA issuer. Shared memory: K, V (32 KB each), two Q/dO stages (64 KB each),
// dS^T (32 KB) and LSE/D per stage.
//
// Persistent: one CTA per SM runs (key tile, head) items one after another, so that each
// item's fixed costs overlap the previous item's end. While the softmax warps read out the
// last dQ^T partial and store dK and dV, the producer loads the next item's first Q/dO stage
// and (once the last products have read them) its K and V, and the tensor core computes its
// first S^T and dP^T; only dV and dK of the new item wait for the accumulators to be read.
//
// Masks and dropout (kVar, "知识点13" §7: both are fused into the softmax step): the additive
// mask adds M log2(e) to each exponent; the boolean mask (packed bits, as the forward reads
// them) and dropout zero P for hidden or dropped keys, so their dS is 0 as well; dV takes only
// the kept weights, scaled by 256 / (256 - t) in its epilogue, and a dropped key's dP is 0.
//
// Query and key lengths: Nq query rows against Nk key rows per head,
// causal bottom-right aligned (query i hides keys j > i + Nk - Nq); rows past the end of a
// head arrive as zeros from the tensor maps, queries past the end get LSE = +inf (P = 0),
// and rows past the end are neither accumulated nor stored.
#include <cuda_bf16.h>

#include <atomic>

#include "fa_internal.h"
#include "philox.cuh"
#include "sm100_ptx.cuh"
#include "tma_host.h"

namespace fa {
namespace {

using namespace ptx;

constexpr int BN = 128;  // keys per CTA
constexpr int BQ = 128;  // queries per tile
constexpr int kThreads = 320;
constexpr int kLoadWarp = 8;
constexpr int kMmaWarp = 9;
constexpr int kStages = 2;
constexpr float kLog2e = 1.4426950408889634f;

constexpr int kBox = 128 * 128;  // one [128 rows x 64 columns] bf16 box, 128-byte swizzle
constexpr int kVecBytes = 2 * BQ * 4;
constexpr uint32_t kTmemCols = 512;

struct WideCtl {
  uint64_t kv_full, q_full[kStages], do_full[kStages], q_empty[kStages], do_empty[kStages];
  uint64_t s_full, dp_full, p_done, ds_done, dq_full, dq_empty, kv_done, dv_final, acc_empty, drain;
  uint32_t tmem_base;
  int abort;
};

// Sizes and places for head dimension D (64 or 128).
template <int D>
struct WideCfg {
  static constexpr int kBoxes = D / 64;         // 64-column boxes per row
  static constexpr int kRowTile = 128 * D * 2;  // a [128 rows x D] bf16 tile: K_j, V_j, Q_i or dO_i
  // Shared memory (1024-byte aligned base; control block last). V follows K: at d = 64 the
  // M = 128 dQ^T product reads V's rows as the second 64-row atom of K^T, and those result
  // rows land in TMEM lanes 64-127, which nobody reads.
  static constexpr int kKOff = 0;
  static constexpr int kVOff = kKOff + kRowTile;
  static constexpr int kStageOff = kVOff + kRowTile;  // stage s: Q_i at + s * 2 * kRowTile, dO_i after it
  static constexpr int kDsOff = kStageOff + kStages * 2 * kRowTile;
  static constexpr int kVecOff = kDsOff + 2 * kBox;   // dS^T is [128 keys x 128 queries]; then LSE_i, D_i
  static constexpr int kCtlOff = kVecOff + kStages * kVecBytes;
  static constexpr int kSmemBytes = kCtlOff + (int)sizeof(WideCtl);
  static_assert(kSmemBytes <= 227 * 1024, "shared-memory budget");
  static_assert(D == 128 || kVOff == kKOff + kBox, "V follows K");
  // TMEM columns: dV | dK | S^T (then P^T, bf16 pairs, in the first half of each 64) |
  // dP^T (then, at d = 128, the dQ^T partial) | at d = 64, the dQ^T partial
  static constexpr uint32_t kColDV = 0;
  static constexpr uint32_t kColDK = D;
  static constexpr uint32_t kColS = 2 * D;
  static constexpr uint32_t kColDP = 2 * D + 128;
  static constexpr bool kSepDQ = kColDP + 256 <= kTmemCols;  // room for dQ^T beside dP^T
  static constexpr uint32_t kColDQ = kSepDQ ? kColDP + 128 : kColDP;
  static_assert(kColDQ + 128 <= kTmemCols, "TMEM budget");
};

struct WideParams {
  const float* LSE;
  const float* Dvec;
  float* dQacc;
  __nv_bfloat16* dK;
  __nv_bfloat16* dV;
  int* status;
  int Nq, Nk;
  int heads;
  int kvtiles;
  int qtiles;
  int causal;
  int offset;  // causal: query i hides keys j > i + offset
  float scale;
  float sl2;   // scale * log2(e)
};

// The arguments of the mask and dropout instances, a kernel argument of their own: with them in
// WideParams the plain instance measured 3% slower, same source and registers otherwise.
struct VarParams {
  // additive mask (kVar == 1): element (b, h, i, j) at mask[b*mask_sb + h*mask_sh + i*mask_srow + j]
  const __nv_bfloat16* mask;
  // boolean mask (kVar == 3): visibility bits, word (b, h, i, j / 32) at
  // bits[b*mask_sb + h*mask_sh + i*mask_srow + j / 32] (the same strides, in 32-bit words)
  const uint32_t* bits;
  int64_t mask_sb, mask_sh, mask_srow;
  int H;
  // dropout (kVar == 2): Philox key, keep threshold (in all four bytes) and a kept weight's scale
  uint32_t seed_lo, seed_hi, drop_tt;
  float drop_scale;
};

// Transpose of a 32 x 32 bit matrix held one row per lane: on return lane T holds bit c =
// bit T of lane c's row. Five butterfly stages; the stage of width s swaps, between lanes l
// and l ^ s, the s-bit groups whose position differs from the lane in bit s.
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

// TMEM column of the packed bf16 P^T for query block k (16 queries): each softmax
// warpgroup packs its 64 queries into the first 32 columns of its 64-column half.
__device__ __forceinline__ uint32_t packed_col(uint32_t base, int k) { return base + (k / 4) * 64 + (k % 4) * 8; }

// 10 warps put at most 3 warps on each of the SM's four sub-partitions (16 K registers each),
// which allows 168 registers per thread: a softmax thread holds its 64 weights from phase A
// to phase B and, between the two, a 64-column row of the dQ partial.
// kVar: 0 plain, 1 additive mask, 2 dropout, 3 boolean mask (packed bits). kDQ: the dQ^T
// partials are computed and added into the accumulator; without them the kernel gives dK and
// dV only, and the separate dQ pass (fa_bwd_dq.cu) gives dQ.
template <int D, bool kTail, int kVar, bool kDQ>
__global__ void __launch_bounds__(kThreads, 1)
fa_bwd_wide_kernel(const __grid_constant__ CUtensorMap tmQ, const __grid_constant__ CUtensorMap tmK,
                   const __grid_constant__ CUtensorMap tmV, const __grid_constant__ CUtensorMap tmdO,
                   const WideParams p, const VarParams pv) {
  using C = WideCfg<D>;
  constexpr bool kMask = kVar == 1;
  constexpr bool kDrop = kVar == 2;
  constexpr bool kBits = kVar == 3;
  constexpr uint32_t kColDV = C::kColDV, kColDK = C::kColDK, kColS = C::kColS, kColDP = C::kColDP, kColDQ = C::kColDQ;
  extern __shared__ __align__(1024) uint8_t smem[];
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  // The swizzled operand layout needs a 1024-byte aligned base; the runtime provides it for
  // this declaration, and the kernel refuses to run (status word) if it did not.
  if ((smem_u32(smem) & 1023u) != 0) {
    if (threadIdx.x == 0 && p.status) atomicExch(p.status, 3 /* FA_ERR_CUDA */);
    return;
  }
  WideCtl& ctl = *reinterpret_cast<WideCtl*>(smem + C::kCtlOff);

  // Work items are (key tile, head) pairs, w = 0 .. items-1. Causal: key tiles near the start
  // see the most queries and come first. Each CTA (one per SM) takes the items
  // b, 2G-1-b, 2G+b, 4G-1-b, ... (G CTAs): every round of G items runs in the other direction,
  // so that the heavier items of one round and the lighter ones of the next land on the same SM.
  const int items = p.kvtiles * p.heads;
  const int G = (int)gridDim.x, b = (int)blockIdx.x;
  auto item_of = [&](int r) { return r * G + ((r & 1) ? G - 1 - b : b); };
  auto decode = [&](int w, int& kt, int& head) {
    if (p.causal) {
      kt = w / p.heads;
      head = w % p.heads;
    } else {
      kt = w % p.kvtiles;
      head = w / p.kvtiles;
    }
  };
  // causal: the first query tile holding a query that sees key kt * BN (query + offset >= key)
  auto q_first_of = [&](int kt) { return p.causal ? max(0, kt * BN - p.offset) / BQ : 0; };

  if (threadIdx.x == 0) {
    mbar_init(&ctl.kv_full, 1);
    for (int s = 0; s < kStages; ++s) {
      mbar_init(&ctl.q_full[s], 1);
      mbar_init(&ctl.do_full[s], 1);
      mbar_init(&ctl.q_empty[s], 1);
      mbar_init(&ctl.do_empty[s], 1);
    }
    mbar_init(&ctl.s_full, 1);
    mbar_init(&ctl.dp_full, 1);
    mbar_init(&ctl.p_done, 256);
    mbar_init(&ctl.ds_done, 256);
    mbar_init(&ctl.dq_full, 1);
    mbar_init(&ctl.dq_empty, 256);
    mbar_init(&ctl.kv_done, 1);
    mbar_init(&ctl.dv_final, 1);
    mbar_init(&ctl.acc_empty, 256);
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

  // Every barrier of a query tile counts tiles over all items of the CTA (g below), and kv_full,
  // kv_done and acc_empty count the CTA's items (ni).
  if (warp == kLoadWarp) {
    // Lane 0 drives the copies and barriers. LSE_i and D_i of a whole tile whose rows start
    // 16-byte aligned arrive by bulk copy with Q_i; otherwise (the last, partial tile of a
    // head, or Nq not a multiple of 4) the warp stages them with bounds-checked loads:
    // queries past the end of the head get LSE = +inf and D = 0, so P = dS = 0.
    if (lane == 0) {
      prefetch_tmap(&tmQ);
      prefetch_tmap(&tmK);
      prefetch_tmap(&tmV);
      prefetch_tmap(&tmdO);
    }
    int last_q[kStages] = {-1, -1}, last_do[kStages] = {-1, -1}, last_kv = -1;
    // Test hook of the failure path: never arm the first Q stage, so the MMA thread's wait
    // for it runs out (see StatusBlock); off unless a test sets it.
    const bool skip_first = injected(p.status, kInjectBwd);
    const bool all_bulk = !kTail || ((p.Nq % BQ) == 0 && (p.Nq % 4) == 0);
    bool ok = true;
    int g = 0, ni = 0;
    for (int r = 0; ok && (lane == 0 || !all_bulk); ++r) {
      const int w = item_of(r);
      if (w >= items) break;
      int kt, head;
      decode(w, kt, head);
      const int q_first = q_first_of(kt);
      const int nq = p.qtiles - q_first;
      if (nq <= 0) continue;
      const int qrow_base = head * p.Nq;
      // K_j and V_j once the products of the previous item that read them have run; after the
      // first item, behind this item's first Q/dO stage, whose slot frees earlier
      auto load_kv = [&]() {
        if (lane == 0) {
          if (ni > 0 && !mbar_wait(&ctl.kv_done, (ni - 1) & 1, p.status, abort)) {
            ok = false;
          } else {
            mbar_expect_tx(&ctl.kv_full, 2 * C::kRowTile);
            for (int bx = 0; bx < C::kBoxes; ++bx) {
              tma_load_3d(smem + C::kKOff + bx * kBox, &tmK, &ctl.kv_full, bx * 64, kt * BN, head);
              tma_load_3d(smem + C::kVOff + bx * kBox, &tmV, &ctl.kv_full, bx * 64, kt * BN, head);
            }
            last_kv = ni;
          }
        }
        if (!all_bulk) ok = __shfl_sync(0xffffffffu, ok ? 1 : 0, 0) != 0;
      };
      if (ni == 0) load_kv();
      for (int it = 0; ok && it < nq; ++it) {
        const int gi = g + it;
        const int s = gi % kStages;
        const uint32_t par = ((gi / kStages) - 1) & 1;
        // Q_i's slot (and its LSE/D) frees once dK of the tile two back has run.
        if (lane == 0 && gi >= kStages) ok = mbar_wait(&ctl.q_empty[s], par, p.status, abort);
        if (!all_bulk) ok = __shfl_sync(0xffffffffu, ok ? 1 : 0, 0) != 0;
        if (!ok) break;
        const int q0 = (q_first + it) * BQ;  // first query of the tile, within the head
        uint8_t* st = smem + C::kStageOff + s * 2 * C::kRowTile;
        float* vec = reinterpret_cast<float*>(smem + C::kVecOff + s * kVecBytes);
        const bool bulk = !kTail || (q0 + BQ <= p.Nq && (p.Nq % 4) == 0);
        if (!bulk) {
          for (int c = lane; c < BQ; c += 32) {
            const bool in = q0 + c < p.Nq;
            vec[c] = in ? p.LSE[qrow_base + q0 + c] : INFINITY;
            vec[BQ + c] = in ? p.Dvec[qrow_base + q0 + c] : 0.f;
          }
          __syncwarp();
        }
        if (lane == 0) {
          if (gi > 0 || !skip_first) {
            mbar_expect_tx(&ctl.q_full[s], C::kRowTile + (bulk ? kVecBytes : 0));
            for (int bx = 0; bx < C::kBoxes; ++bx) tma_load_3d(st + bx * kBox, &tmQ, &ctl.q_full[s], bx * 64, q0, head);
            if (bulk) {
              bulk_load(vec, p.LSE + qrow_base + q0, BQ * 4, &ctl.q_full[s]);
              bulk_load(vec + BQ, p.Dvec + qrow_base + q0, BQ * 4, &ctl.q_full[s]);
            }
            last_q[s] = gi;
          }
          // dO_i's slot frees once dV of the tile two back has run (earlier than Q's).
          if (gi >= kStages && !mbar_wait(&ctl.do_empty[s], par, p.status, abort)) ok = false;
          if (ok) {
            mbar_expect_tx(&ctl.do_full[s], C::kRowTile);
            for (int bx = 0; bx < C::kBoxes; ++bx)
              tma_load_3d(st + C::kRowTile + bx * kBox, &tmdO, &ctl.do_full[s], bx * 64, q0, head);
            last_do[s] = gi;
          }
        }
        if (!all_bulk) ok = __shfl_sync(0xffffffffu, ok ? 1 : 0, 0) != 0;
        if (ok && it == 0 && ni > 0) load_kv();
      }
      g += nq;
      ++ni;
    }
    if (lane == 0) {  // every issued copy must land before the CTA may exit
      if (last_kv >= 0) mbar_wait(&ctl.kv_full, last_kv & 1, p.status, nullptr);
      for (int s = 0; s < kStages; ++s) {
        if (last_q[s] >= 0) mbar_wait(&ctl.q_full[s], (last_q[s] / kStages) & 1, p.status, nullptr);
        if (last_do[s] >= 0) mbar_wait(&ctl.do_full[s], (last_do[s] / kStages) & 1, p.status, nullptr);
      }
    }
  } else if (warp == kMmaWarp) {
    if (lane == 0) {
      constexpr uint32_t idSP = idesc_bf16(BN, BQ, false, false);  // S^T, dP^T
      constexpr uint32_t idKV = idesc_bf16(BN, D, false, true);    // dV, dK (B MN-major)
      constexpr uint32_t idQ = idesc_bf16(128, BQ, true, true);    // dQ^T (A and B MN-major), M = 128
      const uint32_t aStage = smem_u32(smem + C::kStageOff);
      // Base descriptors; each MMA below only advances the start address.
      const uint64_t dKk = sdesc_sw128(smem_u32(smem + C::kKOff), 16, 1024);     // K_j, K-major
      const uint64_t dKmn = sdesc_sw128(smem_u32(smem + C::kKOff), kBox, 1024);  // K_j^T, MN-major
      const uint64_t dVk = sdesc_sw128(smem_u32(smem + C::kVOff), 16, 1024);
      const uint64_t dSk = sdesc_sw128(smem_u32(smem + C::kDsOff), 16, 1024);    // dS^T as A, K-major
      const uint64_t dSmn = sdesc_sw128(smem_u32(smem + C::kDsOff), kBox, 1024); // dS^T as B, MN-major
      auto stage_k = [&](int s, bool dO) {
        return sdesc_sw128(aStage + s * 2 * C::kRowTile + (dO ? C::kRowTile : 0), 16, 1024);
      };
      auto stage_mn = [&](int s, bool dO) {
        return sdesc_sw128(aStage + s * 2 * C::kRowTile + (dO ? C::kRowTile : 0), kBox, 1024);
      };
      // K = d: 16 columns (32 bytes) per step inside a box, the next box after 4 steps
      auto issue_S = [&](int s) {
        const uint64_t qd = stage_k(s, false);
#pragma unroll
        for (int k = 0; k < D / 16; ++k)
          mma_ss(tmem + kColS, sdesc_add(dKk, (k / 4) * kBox + (k % 4) * 32), sdesc_add(qd, (k / 4) * kBox + (k % 4) * 32),
                 idSP, k > 0);
      };
      auto issue_dP = [&](int s) {
        const uint64_t od = stage_k(s, true);
#pragma unroll
        for (int k = 0; k < D / 16; ++k)
          mma_ss(tmem + kColDP, sdesc_add(dVk, (k / 4) * kBox + (k % 4) * 32),
                 sdesc_add(od, (k / 4) * kBox + (k % 4) * 32), idSP, k > 0);
      };
      // K = queries: 16 rows (2048 bytes) of the MN-major dO_i / Q_i per step
      auto issue_dV = [&](bool first, int s) {
        const uint64_t bd = stage_mn(s, true);
#pragma unroll
        for (int k = 0; k < BQ / 16; ++k)
          mma_ts(tmem + kColDV, packed_col(tmem + kColS, k), sdesc_add(bd, k * 2048), idKV, (!first || k > 0) ? 1u : 0u);
      };
      auto issue_dK = [&](bool first, int s) {
        const uint64_t bd = stage_mn(s, false);
#pragma unroll
        for (int k = 0; k < BQ / 16; ++k)
          mma_ss(tmem + kColDK, sdesc_add(dSk, (k / 4) * kBox + (k % 4) * 32), sdesc_add(bd, k * 2048), idKV,
                 (!first || k > 0) ? 1u : 0u);
      };
      // K = keys: 16 rows (2048 bytes) of K_j and of dS^T per step
      auto issue_dQ = [&]() {
#pragma unroll
        for (int k = 0; k < BN / 16; ++k)
          mma_ss(tmem + kColDQ, sdesc_add(dKmn, k * 2048), sdesc_add(dSmn, k * 2048), idQ, k > 0);
      };
      bool ok = true;
      int g = 0, ni = 0;
      for (int r = 0; ok; ++r) {
        const int w = item_of(r);
        if (w >= items) break;
        int kt, head;
        decode(w, kt, head);
        const int nq = p.qtiles - q_first_of(kt);
        if (nq <= 0) continue;
        // prologue: S(0), dP(0), dV(0) of the item
        const int s0 = g % kStages;
        const uint32_t par0 = (g / kStages) & 1;
        if (!(ok = mbar_wait(&ctl.kv_full, ni & 1, p.status, abort))) break;
        if (!(ok = mbar_wait(&ctl.q_full[s0], par0, p.status, abort))) break;
        tc_fence_after();
        issue_S(s0);
        mma_commit(&ctl.s_full);
        if (!(ok = mbar_wait(&ctl.do_full[s0], par0, p.status, abort))) break;
        if constexpr (kDQ && !C::kSepDQ) {  // the previous item's last dQ^T partial is out of the dP^T columns
          if (g > 0 && !(ok = mbar_wait(&ctl.dq_empty, (g - 1) & 1, p.status, abort))) break;
        }
        tc_fence_after();
        issue_dP(s0);
        mma_commit(&ctl.dp_full);
        if (!(ok = mbar_wait(&ctl.p_done, g & 1, p.status, abort))) break;
        // dV and dK of the previous item have been read out of TMEM
        if (ni > 0 && !(ok = mbar_wait(&ctl.acc_empty, (ni - 1) & 1, p.status, abort))) break;
        tc_fence_after();
        issue_dV(true, s0);
        mma_commit(&ctl.do_empty[s0]);  // dP(0) and dV(0), the readers of dO(0), issued
        if (nq == 1) mma_commit(&ctl.dv_final);  // the item's last dV product
        for (int it = 0; ok && it < nq; ++it) {
          const int gi = g + it;
          const int s = gi % kStages, s1 = (gi + 1) % kStages;
          const bool next = it + 1 < nq;
          const uint32_t par1 = ((gi + 1) / kStages) & 1;
          // S(i+1) over the S^T columns: P^T(i) was read by dV(i), issued before
          if (next) {
            if (!(ok = mbar_wait(&ctl.q_full[s1], par1, p.status, abort))) break;
            tc_fence_after();
            issue_S(s1);
            mma_commit(&ctl.s_full);
          }
          // dK(i) and dQ(i) read dS^T(i) from shared memory; dQ^T(i) lands in the dP^T
          // columns, which phase B of tile i has read, or in columns of its own, which the
          // softmax warps have emptied of the previous partial
          if (!(ok = mbar_wait(&ctl.ds_done, gi & 1, p.status, abort))) break;
          tc_fence_after();
          issue_dK(it == 0, s);
          mma_commit(&ctl.q_empty[s]);
          if constexpr (kDQ) {
            if (C::kSepDQ && gi > 0) {
              if (!(ok = mbar_wait(&ctl.dq_empty, (gi - 1) & 1, p.status, abort))) break;
              tc_fence_after();
            }
            issue_dQ();
            mma_commit(&ctl.dq_full);
          }
          // dP(i+1) ahead of dV(i+1) where nothing else occupies the dP^T columns; with the dQ^T
          // partial there, dP(i+1) would wait for its read-out, and dV(i+1) goes first (dP first
          // measured 2% slower at d = 128)
          constexpr bool kDPFirst = C::kSepDQ || !kDQ;
          if (kDPFirst && next) {
            if (!(ok = mbar_wait(&ctl.do_full[s1], par1, p.status, abort))) break;
            tc_fence_after();
            issue_dP(s1);
            mma_commit(&ctl.dp_full);
            if (!(ok = mbar_wait(&ctl.p_done, (gi + 1) & 1, p.status, abort))) break;
            tc_fence_after();
            issue_dV(false, s1);
            mma_commit(&ctl.do_empty[s1]);  // dP(i+1) and dV(i+1), the readers of dO(i+1), issued
            if (it + 2 == nq) mma_commit(&ctl.dv_final);
          } else if (next) {
            // dV(i+1) reads P^T(i+1) from TMEM and dO(i+1) from its stage: both must be in
            if (!(ok = mbar_wait(&ctl.p_done, (gi + 1) & 1, p.status, abort))) break;
            if (!(ok = mbar_wait(&ctl.do_full[s1], par1, p.status, abort))) break;
            tc_fence_after();
            issue_dV(false, s1);
            if (it + 2 == nq) mma_commit(&ctl.dv_final);
            // dP(i+1) once the softmax warps have read the dQ^T(i) partial out of its columns
            if constexpr (kDQ && !C::kSepDQ) {
              if (!(ok = mbar_wait(&ctl.dq_empty, gi & 1, p.status, abort))) break;
              tc_fence_after();
            }
            issue_dP(s1);
            mma_commit(&ctl.dp_full);
            mma_commit(&ctl.do_empty[s1]);  // dV(i+1) and dP(i+1), the readers of dO(i+1), issued
          }
        }
        if (!ok) break;
        mma_commit(&ctl.kv_done);  // every product of the item: K_j, V_j and dV, dK are free to read
        g += nq;
        ++ni;
      }
      mma_commit(&ctl.drain);
      mbar_wait(&ctl.drain, 0, p.status, nullptr);
    }
  } else {
    // ---------------- softmax-backward warpgroups, dQ read-out, dK/dV epilogue ----------------
    const int wg = warp >> 2;
    const int r = (warp & 3) * 32 + lane;  // TMEM lane: the key row (S^T, dP^T, dV, dK), or the
                                           // head-dim index (the dQ^T partial)
    const uint32_t lane_off = (uint32_t)((warp & 3) * 32) << 16;
    const float2 sl2 = make_float2(p.sl2, p.sl2);
    const float2 neg_log2e = make_float2(-kLog2e, -kLog2e);
    const float2 minus1 = make_float2(-1.f, -1.f);
    uint8_t* dsrow = smem + C::kDsOff + r * 128;
    // The dQ^T partial of tile j: lane = head-dim index r, columns = the tile's queries; this
    // warpgroup takes its 64 columns and releases them as soon as they are in registers (dP of
    // the next tile, or at d = 64 its dQ, waits for that). It adds the first 32 into the fp32
    // accumulator at once and holds the other 32 for phase B of the next tile (16 after each of
    // its two chunks): spread out this way, the reductions slow the tensor core's operand reads
    // less than in one burst.
    float held[32];
    float* held_dst = nullptr;
    int held_valid = 0;
    // red.add of 32 columns (queries) of one head-dim row; the bound test stays out of the
    // reduction loop (a predicate inside it serialises the reductions), and both loops unroll
    // fully so the values stay in registers.
    auto add32 = [&](float* dst, const float* v, int nvalid) {
      if (!kTail || 32 <= nvalid) {
#pragma unroll
        for (int c = 0; c < 32; ++c) atomicAdd(dst + (size_t)c * D, v[c]);
      } else {  // the last, partial tile of a head
#pragma unroll
        for (int c = 0; c < 32; ++c)
          if (c < nvalid) atomicAdd(dst + (size_t)c * D, v[c]);
      }
    };
    // red.add of 16 of the held columns (part 0: columns 0-15, part 1: 16-31)
    auto flush_held = [&](int part) {
      if (!held_dst) return;
      float* dst = held_dst + (size_t)(16 * part) * D;
      const int nvalid = held_valid - 16 * part;
      if (!kTail || 16 <= nvalid) {
#pragma unroll
        for (int c = 0; c < 16; ++c) atomicAdd(dst + (size_t)c * D, held[16 * part + c]);
      } else {
#pragma unroll
        for (int c = 0; c < 16; ++c)
          if (c < nvalid) atomicAdd(dst + (size_t)c * D, held[16 * part + c]);
      }
      if (part == 1) held_dst = nullptr;
    };
    // At d = 64 only TMEM lanes 0-63 hold head-dim rows: the warps of lanes 64-127 load their
    // (unused) lanes too, but add nothing (a test that is uniform over each warp).
    const bool dq_rows = (warp & 3) * 32 < D;
    int q_first = 0, qrow_base = 0;
    // partial j of the current item, the CTA's tile gj
    auto read_out_dq = [&](int j, int gj) -> bool {
      if (!__all_sync(0xffffffffu, mbar_wait(&ctl.dq_full, gj & 1, p.status, abort))) return false;
      tc_fence_after();
      float v[32];
      tmem_ld32x2(tmem + lane_off + kColDQ + wg * 64, tmem + lane_off + kColDQ + wg * 64 + 32, v, held);
      tc_fence_before();
      mbar_arrive(&ctl.dq_empty);
      if (!dq_rows) return true;
      const int qh = (q_first + j) * BQ + wg * 64;  // first query of this half, within the head
      float* dst = p.dQacc + (size_t)(qrow_base + qh) * D + r;
      add32(dst, v, p.Nq - qh);
      held_dst = dst + (size_t)32 * D;
      held_valid = p.Nq - qh - 32;
      return true;
    };
    bool ok = true;
    int g = 0, ni = 0;
    for (int rr = 0; ok; ++rr) {
      const int w = item_of(rr);
      if (w >= items) break;
      int kt, head;
      decode(w, kt, head);
      q_first = q_first_of(kt);
      const int nq = p.qtiles - q_first;
      qrow_base = head * p.Nq;
      const int krow_base = head * p.Nk;
      if (nq <= 0) {  // no query sees these keys: dK = dV = 0
        if (threadIdx.x < BN && kt * BN + (int)threadIdx.x < p.Nk) {
          const size_t row = (size_t)krow_base + kt * BN + threadIdx.x;
          uint4* dk = reinterpret_cast<uint4*>(p.dK + row * D);
          uint4* dv = reinterpret_cast<uint4*>(p.dV + row * D);
#pragma unroll
          for (int u = 0; u < D / 8; ++u) dk[u] = dv[u] = make_uint4(0, 0, 0, 0);
        }
        continue;
      }
      const int key = kt * BN + r;
      // kBits: the warp's 32 keys are one word of each query's row. For chunk ch, lane L reads the
      // word of query (tile start + wg * 64 + ch * 32 + L), one tile ahead, so that the load's
      // latency hides behind the current tile.
      const int kword = (kt * BN + (warp & 3) * 32) >> 5;
      const uint32_t* bcol =
          kBits ? pv.bits + (int64_t)(head / pv.H) * pv.mask_sb + (int64_t)(head % pv.H) * pv.mask_sh + kword : nullptr;
      auto bits_word = [&](int it, int ch) -> uint32_t {
        const int q = (q_first + it) * BQ + wg * 64 + ch * 32 + lane;
        return (it < nq && (!kTail || (q < p.Nq && kword * 32 < p.Nk))) ? bcol[(int64_t)q * pv.mask_srow] : 0u;
      };
      uint32_t bword[2] = {0u, 0u};
      if constexpr (kBits) {
        bword[0] = bits_word(0, 0);
        bword[1] = bits_word(0, 1);
      }
      for (int it = 0; ok && it < nq; ++it) {
        const int gi = g + it;
        const float* vec = reinterpret_cast<const float*>(smem + C::kVecOff + (gi % kStages) * kVecBytes);
        uint32_t bcur[2] = {bword[0], bword[1]};
        if constexpr (kBits) {
          bword[0] = bits_word(it + 1, 0);
          bword[1] = bits_word(it + 1, 1);
        }
        uint32_t kbits[2] = {0u, 0u};  // kDrop: keep bits of this key against each chunk's 32 queries
        const int q0 = (q_first + it) * BQ;
        // some key of the tile exceeds the limit of some query of the tile
        const bool diag = p.causal && q0 + p.offset < kt * BN + BN - 1;
        // ---- phase A: P^T = exp2(S^T * scale * log2e - LSE * log2e), over S^T in TMEM
        ok = __all_sync(0xffffffffu, mbar_wait(&ctl.s_full, gi & 1, p.status, abort));
        if (!ok) break;
        tc_fence_after();
        float pr[64];  // this row's P for the warpgroup's 64 queries, kept for phase B
#pragma unroll
        for (int ch = 0; ch < 2; ++ch) {
          const int c0 = wg * 64 + ch * 32;  // first query column of this chunk
          // kMask: M(query, this key) * log2(e) for the chunk's 32 queries (across the warp each
          // load reads 32 consecutive keys of one mask row), issued before the TMEM load
          float mk[kMask ? 32 : 1];
          if constexpr (kMask) {
            const __nv_bfloat16* mcol = pv.mask + (int64_t)(head / pv.H) * pv.mask_sb + (int64_t)(head % pv.H) * pv.mask_sh + key;
#pragma unroll
            for (int c = 0; c < 32; ++c) {
              const int q = q0 + c0 + c;
              mk[c] = (!kTail || (key < p.Nk && q < p.Nq)) ? __bfloat162float(mcol[(int64_t)q * pv.mask_srow]) * kLog2e : 0.f;
            }
          }
          // kDrop: lane L draws the keep bits of query (chunk start + L) against the warp's 32
          // keys (two Philox blocks of 16 keys); the transpose leaves lane T with bit c =
          // keep(query c of the chunk, key T). kBits: the same transpose of the prefetched words.
          if constexpr (kDrop) {
            const uint32_t i = (uint32_t)(q0 + c0 + lane);
            const uint32_t blk0 = (uint32_t)((kt * BN + (warp & 3) * 32) >> 4);
            const uint32_t row = rng::keep16(blk0, i, (uint32_t)head, pv.seed_lo, pv.seed_hi, pv.drop_tt) |
                                 (rng::keep16(blk0 + 1, i, (uint32_t)head, pv.seed_lo, pv.seed_hi, pv.drop_tt) << 16);
            kbits[ch] = transpose32(row, lane);
          }
          const uint32_t vbits = kBits ? transpose32(bcur[ch], lane) : 0u;
          float sv[32];
          tmem_ld32(tmem + lane_off + kColS + c0, sv);
          uint32_t pk[16];
          if constexpr (kVar == 0) {
#pragma unroll
            for (int u = 0; u < 16; ++u) {
              const int c = c0 + 2 * u;
              const float2 lse = *reinterpret_cast<const float2*>(vec + c);
              const float2 x = ffma2(make_float2(sv[2 * u], sv[2 * u + 1]), sl2, fmul2(lse, neg_log2e));
              float2 pv = make_float2(ex2(x.x), ex2(x.y));
              if (diag) {
                if (key > q0 + c + p.offset) pv.x = 0.f;
                if (key > q0 + c + 1 + p.offset) pv.y = 0.f;
              }
              pr[ch * 32 + 2 * u] = pv.x;
              pr[ch * 32 + 2 * u + 1] = pv.y;
              pk[u] = pack_bf16(pv.x, pv.y);
            }
          } else {
#pragma unroll
          for (int u = 0; u < 16; ++u) {
            const int c = c0 + 2 * u;
            const float2 lse = *reinterpret_cast<const float2*>(vec + c);
            float2 nl = fmul2(lse, neg_log2e);
            if constexpr (kMask || kBits) {  // a query with no visible key (LSE = -inf) has P = 0
              if (lse.x == -INFINITY) nl.x = -INFINITY;
              if (lse.y == -INFINITY) nl.y = -INFINITY;
            }
            float2 x = ffma2(make_float2(sv[2 * u], sv[2 * u + 1]), sl2, nl);
            if constexpr (kMask) x = fadd2(x, make_float2(mk[2 * u], mk[2 * u + 1]));
            float2 pv = make_float2(ex2(x.x), ex2(x.y));
            if constexpr (kBits) {  // a hidden key has P = 0, and so dS = 0
              if (!((vbits >> (2 * u)) & 1u)) pv.x = 0.f;
              if (!((vbits >> (2 * u + 1)) & 1u)) pv.y = 0.f;
            }
            if (diag) {
              if (key > q0 + c + p.offset) pv.x = 0.f;
              if (key > q0 + c + 1 + p.offset) pv.y = 0.f;
            }
            pr[ch * 32 + 2 * u] = pv.x;
            pr[ch * 32 + 2 * u + 1] = pv.y;
            if constexpr (kDrop) {  // dV takes the kept weights (scaled by c in its epilogue)
              const uint32_t kb = kbits[ch] >> (2 * u);
              pk[u] = pack_bf16((kb & 1u) ? pv.x : 0.f, (kb & 2u) ? pv.y : 0.f);
            } else {
              pk[u] = pack_bf16(pv.x, pv.y);
            }
          }
          }
          tmem_st16(tmem + lane_off + kColS + wg * 64 + ch * 16, pk);
        }
        tmem_wait_st();
        tc_fence_before();
        mbar_arrive(&ctl.p_done);
        // ---- the previous tile's dQ^T partial, while dK/dQ of that tile and dV of this one run
        if constexpr (kDQ) {
          if (it > 0 && !(ok = read_out_dq(it - 1, gi - 1))) break;
        }
        // ---- phase B: dS^T = P^T * (dP^T - D), to shared memory only
        ok = __all_sync(0xffffffffu, mbar_wait(&ctl.dp_full, gi & 1, p.status, abort));
        if (!ok) break;
        tc_fence_after();
#pragma unroll
        for (int ch = 0; ch < 2; ++ch) {
          const int c0 = wg * 64 + ch * 32;
          float dp[32];
          tmem_ld32(tmem + lane_off + kColDP + c0, dp);
          uint32_t dk[16];
#pragma unroll
          for (int u = 0; u < 16; ++u) {
            float2 dd;
            if constexpr (kDrop) {  // dP of a dropped key is 0; a kept one is scaled
              const float2 dvec = *reinterpret_cast<const float2*>(vec + BQ + c0 + 2 * u);
              const uint32_t kb = kbits[ch] >> (2 * u);
              dd = make_float2((kb & 1u) ? fmaf(dp[2 * u], pv.drop_scale, -dvec.x) : -dvec.x,
                               (kb & 2u) ? fmaf(dp[2 * u + 1], pv.drop_scale, -dvec.y) : -dvec.y);
            } else {
              dd = ffma2(*reinterpret_cast<const float2*>(vec + BQ + c0 + 2 * u), minus1,
                         make_float2(dp[2 * u], dp[2 * u + 1]));
            }
            const float2 ds = fmul2(make_float2(pr[ch * 32 + 2 * u], pr[ch * 32 + 2 * u + 1]), dd);
            dk[u] = pack_bf16(ds.x, ds.y);
          }
          // dS^T row r, query columns c0..c0+31: four 16-byte chunks of a 128-byte swizzled
          // row (box c0 / 64, chunk (c0 % 64) / 8 + u, XOR (r % 8))
          uint8_t* atom = dsrow + (c0 / 64) * kBox;
#pragma unroll
          for (int u = 0; u < 4; ++u) {
            const int chunk = ((c0 % 64) / 8 + u) ^ (r & 7);
            *reinterpret_cast<uint4*>(atom + chunk * 16) = make_uint4(dk[4 * u], dk[4 * u + 1], dk[4 * u + 2], dk[4 * u + 3]);
          }
          if (ch == 0) flush_held(0);
        }
        fence_proxy_async_smem();
        tc_fence_before();
        mbar_arrive(&ctl.ds_done);
        flush_held(1);
      }
      // dV is final once the item's last dV product has run (before dK and dQ of the last tile):
      // store it while those run
      const size_t row = (size_t)krow_base + kt * BN + r;
      const bool in = !kTail || kt * BN + r < p.Nk;  // key rows past the end are not stored
      if (ok) ok = __all_sync(0xffffffffu, mbar_wait(&ctl.dv_final, ni & 1, p.status, abort));
      if (!ok) break;
      tc_fence_after();
#pragma unroll 1
      for (int c0 = wg * (D / 2); c0 < wg * (D / 2) + D / 2; c0 += 32) {
        float v[32];
        uint4 wv[4];
        uint32_t* wu = reinterpret_cast<uint32_t*>(wv);
        tmem_ld32(tmem + lane_off + kColDV + c0, v);
        if constexpr (kDrop) {  // kept weights entered dV unscaled
#pragma unroll
          for (int u = 0; u < 16; ++u) wu[u] = pack_bf16(v[2 * u] * pv.drop_scale, v[2 * u + 1] * pv.drop_scale);
        } else {
#pragma unroll
          for (int u = 0; u < 16; ++u) wu[u] = pack_bf16(v[2 * u], v[2 * u + 1]);
        }
        uint4* dv = reinterpret_cast<uint4*>(p.dV + row * D + c0);
        if (in) {
#pragma unroll
          for (int u = 0; u < 4; ++u) dv[u] = wv[u];
        }
      }
      if constexpr (kDQ) {
        if (ok) ok = read_out_dq(nq - 1, g + nq - 1);
      }
      if (ok) {
        flush_held(0);
        flush_held(1);
      }
      if (ok) ok = __all_sync(0xffffffffu, mbar_wait(&ctl.kv_done, ni & 1, p.status, abort));
      if (!ok) break;
      // dK of key row r; warpgroup wg writes columns wg*D/2 .. wg*D/2 + D/2 - 1
      tc_fence_after();
#pragma unroll 1
      for (int c0 = wg * (D / 2); c0 < wg * (D / 2) + D / 2; c0 += 32) {
        float v[32];
        uint4 wv[4];
        uint32_t* wu = reinterpret_cast<uint32_t*>(wv);
        tmem_ld32(tmem + lane_off + kColDK + c0, v);
#pragma unroll
        for (int u = 0; u < 16; ++u) wu[u] = pack_bf16(v[2 * u] * p.scale, v[2 * u + 1] * p.scale);
        uint4* dk = reinterpret_cast<uint4*>(p.dK + row * D + c0);
        if (in) {
#pragma unroll
          for (int u = 0; u < 4; ++u) dk[u] = wv[u];
        }
      }
      // the next item's dV and dK may overwrite the accumulators
      tc_fence_before();
      mbar_arrive(&ctl.acc_empty);
      g += nq;
      ++ni;
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

// Streaming multiprocessors of the current device (looked up once per device).
int sm_count() {
  static std::atomic<int> cached[64] = {};
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return 1;
  int n = cached[dev].load(std::memory_order_relaxed);
  if (n <= 0) {
    if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || n <= 0) return 1;
    cached[dev].store(n, std::memory_order_relaxed);
  }
  return n;
}

template <int D, int kVar, bool kDQ>
cudaError_t launch_wide(const void* Q, const void* K, const void* V, const void* dO, const float* LSE,
                        const float* Dv, void* dK, void* dV, float* dQacc, const Shape& s, float scale, bool causal,
                        const BwdVariant& var, int* status, cudaStream_t st) {
  using C = WideCfg<D>;
  CUtensorMap mq, mk, mv, mdo;
  const int64_t heads = s.heads();
  if (!make_map_bf16_3d(&mq, Q, heads, s.N, D, BQ) || !make_map_bf16_3d(&mk, K, heads, s.keys(), D, BN) ||
      !make_map_bf16_3d(&mv, V, heads, s.keys(), D, BN) || !make_map_bf16_3d(&mdo, dO, heads, s.N, D, BQ))
    return cudaErrorInvalidValue;
  static bool attr = [] {
    return cudaFuncSetAttribute(fa_bwd_wide_kernel<D, false, kVar, kDQ>,
                                cudaFuncAttributeMaxDynamicSharedMemorySize, C::kSmemBytes) == cudaSuccess &&
           cudaFuncSetAttribute(fa_bwd_wide_kernel<D, true, kVar, kDQ>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                C::kSmemBytes) == cudaSuccess;
  }();
  if (!attr) return cudaErrorInvalidConfiguration;
  WideParams p;
  p.LSE = LSE;
  p.Dvec = Dv;
  p.dQacc = dQacc;
  p.dK = static_cast<__nv_bfloat16*>(dK);
  p.dV = static_cast<__nv_bfloat16*>(dV);
  p.status = status;
  p.Nq = s.N;
  p.Nk = s.keys();
  p.heads = (int)heads;
  p.kvtiles = (s.keys() + BN - 1) / BN;
  p.qtiles = (s.N + BQ - 1) / BQ;
  p.causal = causal ? 1 : 0;
  p.offset = causal ? s.keys() - s.N : 0;
  p.scale = scale;
  p.sl2 = scale * kLog2e;
  VarParams pv;
  pv.mask = static_cast<const __nv_bfloat16*>(var.mask);
  pv.bits = static_cast<const uint32_t*>(var.mask);
  pv.mask_sb = var.sb;
  pv.mask_sh = var.sh;
  pv.mask_srow = var.srow;
  pv.H = s.H;
  pv.seed_lo = (uint32_t)(var.seed & 0xFFFFFFFFu);
  pv.seed_hi = (uint32_t)(var.seed >> 32);
  pv.drop_tt = var.threshold * 0x01010101u;
  pv.drop_scale = (float)(256.0 / (256.0 - (double)var.threshold));
  // one CTA per SM (the shared memory allows no second), each running items until none is left
  const int64_t items = (int64_t)p.kvtiles * p.heads;
  const int64_t grid = items < sm_count() ? items : sm_count();
  if (s.N % BQ != 0 || s.keys() % BN != 0)
    fa_bwd_wide_kernel<D, true, kVar, kDQ><<<(unsigned)grid, kThreads, C::kSmemBytes, st>>>(mq, mk, mv, mdo, p, pv);
  else
    fa_bwd_wide_kernel<D, false, kVar, kDQ><<<(unsigned)grid, kThreads, C::kSmemBytes, st>>>(mq, mk, mv, mdo, p, pv);
  return cudaGetLastError();
}

template <int D>
cudaError_t launch_wide_var(const void* Q, const void* K, const void* V, const void* dO, const float* LSE,
                            const float* Dv, void* dK, void* dV, float* dQacc, const Shape& s, float scale,
                            bool causal, const BwdVariant& var, int* status, cudaStream_t st) {
  if (!dQacc) {  // dK and dV only: the plain instance; dQ comes from the separate pass
    if (var.kind != 0) return cudaErrorInvalidValue;
    return launch_wide<D, 0, false>(Q, K, V, dO, LSE, Dv, dK, dV, dQacc, s, scale, causal, var, status, st);
  }
  switch (var.kind) {
    case 0: return launch_wide<D, 0, true>(Q, K, V, dO, LSE, Dv, dK, dV, dQacc, s, scale, causal, var, status, st);
    case 1: return launch_wide<D, 1, true>(Q, K, V, dO, LSE, Dv, dK, dV, dQacc, s, scale, causal, var, status, st);
    case 2: return launch_wide<D, 2, true>(Q, K, V, dO, LSE, Dv, dK, dV, dQacc, s, scale, causal, var, status, st);
    case 3: return launch_wide<D, 3, true>(Q, K, V, dO, LSE, Dv, dK, dV, dQacc, s, scale, causal, var, status, st);
  }
  return cudaErrorInvalidValue;
}

}  // namespace

cudaError_t tc_bwd_wide(const void* Q, const void* K, const void* V, const void* dO, const float* LSE,
                        const float* Dv, void* dK, void* dV, float* dQacc, const Shape& s, float scale, bool causal,
                        const BwdVariant& var, int* status, cudaStream_t st) {
  if (s.d == 64) return launch_wide_var<64>(Q, K, V, dO, LSE, Dv, dK, dV, dQacc, s, scale, causal, var, status, st);
  if (s.d == 128) return launch_wide_var<128>(Q, K, V, dO, LSE, Dv, dK, dV, dQacc, s, scale, causal, var, status, st);
  return cudaErrorInvalidValue;
}

}  // namespace fa
