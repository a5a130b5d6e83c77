// Attention forward on the 5th-generation tensor cores (tcgen05 + TMEM + TMA), bf16 in,
// fp32 accumulate; what it computes is fa_fwd in include/fa.h.
//
// Method ("flash-attention-v2-sram-tiling" §4-§7): Q is cut into 128-row tiles, K/V
// stream past in 128-row tiles, and each query row keeps a running max m and sum l
// (the online softmax of §5, merged as in "知识点13" section 4). S and P never leave
// the chip: S = Q K^T lands in TMEM, the softmax warps turn it into P (bf16) in place,
// and O += P V accumulates in TMEM. The 1/sqrt(d) scale and log2(e) are folded into a
// single multiplier so every exponential is one FFMA + one ex2 (§7, scale folding).
//
// CTA = two 128-row Q tiles of one head (rows 256*pair .. +255), 10 warps (11 at d = 64):
//   warps 0-3  softmax for Q tile 0 (one thread per row = one TMEM lane)
//   warps 4-7  softmax for Q tile 1
//   warp 8     TMA producer: Q once, then K_j / V_j into a ring of shared-memory stages
//   warp 9     MMA issuer (one thread): S_t = Q_t K_j^T, O_t += P_t V_j (at d = 64, warp 9
//              issues tile 0's products and an eleventh warp tile 1's)
// The two tiles ping-pong: while one warpgroup exponentiates S_0, the tensor core works
// on tile 1, and the other way round.
//
// TMEM (512 columns x 128 lanes): S_0 [0,128), S_1 [128,256), O_0 [256,256+d),
// O_1 [256+d, 256+2d). At d = 128 P_t (bf16 pairs) overwrites the first 64 columns of S_t,
// so S_t(j+1) waits for PV_t(j), and each Q tile's chain per K tile is softmax, then PV and
// S on the tensor core, then softmax again. At d = 64 the 128 columns left over hold P_0
// [384,448) and P_1 [448,512): the softmax warps release S_t as soon as they have loaded it,
// S_t(j+1) runs while they exponentiate S_t(j), and PV_t(j) needs only finish before
// P_t(j+1) is stored (or O_t rescaled), so the tensor core leaves the softmax's chain; with
// one issuer per tile, neither tile's products then wait behind the other's.
//
// Lazy rescale: O and l are rescaled only when the row max grows by more than 8 (log2
// units); otherwise P uses the stale max (values <= 2^8). The result is exact because
// O and l always share the same reference max, and O / l cancels it.
//
// FP8 (e4m3) instance: Q, K and V arrive as e4m3 bytes with one dequantisation factor per
// tensor. S = Q K^T and O += P V run as kind::f8f6f4 MMAs (K = 32 per instruction); the
// factors of Q and K are folded into the exponent multiplier and V's into the epilogue.
// P is rounded to e4m3 (4 per TMEM column). Its rescale threshold is 4 and it is stored
// as 16 p, so the stored values stay in (0, 256] and every p >= 2^-10 of the running
// max lies in e4m3's normal range (relative rounding error <= 2^-4); the factor 16 cancels
// in O / l and is taken out of the LSE.
//
// Additive mask instance (kMask): an [N, N] bf16 mask M per head (broadcast over batch or
// heads by zero strides) is added to the scaled scores ("知识点13" section 7 fuses the mask
// into the softmax step). Each softmax thread streams its row's 128 mask values for the
// next K tile into registers while the current tile is processed, and folds them into S
// as S + M / scale, so the exponent multiplier turns them into (scale q.k + M) log2 e.
// Rows with no visible key so far keep m = -inf and exponentiate against 0; a row with
// no visible key at all stores O = 0 and LSE = -inf.
//
// Boolean mask instance (kVar == 3): the same mask restricted to 0 (visible) and -inf
// (hidden), packed one bit per key: bit j % 32 of word j / 32 of a query's row. A softmax
// thread prefetches its row's 128 bits for the next K tile (one 16-byte load, against 256
// bytes of bf16 mask) and sets the scores of hidden keys to -inf before the row max, as
// the causal diagonal does; rows without a visible key behave as with the additive mask.
//
// Dropout instance (kVar == 2): the same section of "知识点13" fuses dropout into the
// softmax step. Each softmax thread draws the keep bits of its row for the next K tile
// (8 Philox calls of 16 keys, see philox.cuh) while the tile's S is being computed, stores
// p only for kept keys (row sums l still take every p) and scales O by 256 / (256 - t).
//
// Query and key lengths: Nq query rows against Nk key/value rows per head (Nq = Nk for
// fa_fwd). Causal is bottom-right aligned: query i hides keys j > i + Nk - Nq ("知识点13"
// 代码手撕 gives the square rule j > i; the offset places the queries at the end of the
// sequence, as when a prefill continues a cached prefix), so Q tile t sees the K tiles up to
// the limit of its last query, and only the tiles that cross that limit mask anything.
// With Nq > Nk the first Nq - Nk queries see no key: they get O = 0 and LSE = -inf.
// Any lengths: Q/K/V are read through [heads, rows, d] tensor maps, so rows past the end of
// a head arrive as zeros; keys past the end are masked and rows past the end are not stored.
#include <cuda_bf16.h>

#include "fa_internal.h"
#include "philox.cuh"
#include "sm100_ptx.cuh"
#include "tma_host.h"

namespace fa {
namespace {

using namespace ptx;

constexpr int BM = 128;  // query rows per Q tile
constexpr int BN = 128;  // keys per K/V tile
constexpr int kLoadWarp = 8;
constexpr int kMmaWarp = 9;  // and, with one issuer per Q tile, warp 10
constexpr float kLn2 = 0.6931471805599453f;
constexpr int kBoxBytes = BM * 128;  // one [128 rows x 128 bytes] swizzled box

// F8: e4m3 operands (1 byte) instead of bf16 (2 bytes).
template <int D, bool F8>
struct FwdCfg {
  static constexpr int kRowBytes = D * (F8 ? 1 : 2);
  static_assert(kRowBytes % 128 == 0, "rows are whole 128-byte swizzle lines");
  static constexpr int kBoxes = kRowBytes / 128;
  static constexpr int kBoxElems = F8 ? 128 : 64;  // elements per 128-byte box row
  static constexpr int kTileBytes = BM * kRowBytes;
  static constexpr int kKStep = F8 ? 32 : 16;  // K elements per MMA = 32 bytes of a row
  static constexpr int kSSteps = D / kKStep;   // MMAs per S tile (K = head dim)
  static constexpr int kPVSteps = BN / kKStep; // MMAs per PV (K = keys)
  static constexpr float kThreshold = F8 ? 4.f : 8.f;  // lazy-rescale threshold (log2 units)
  static constexpr float kPShift = F8 ? 4.f : 0.f;     // P is stored as 2^kPShift p
  // Ring depths. A third K (or V) stage with 256-byte rows measured slower than two of
  // each: the loads are limited by L2-to-SM bandwidth, not by how far ahead they start.
  static constexpr int kKStages = kRowBytes == 256 ? 2 : 4;
  static constexpr int kVStages = kRowBytes == 256 ? 2 : 4;
  static constexpr int kQOff = 0;
  static constexpr int kKOff = kQOff + 2 * kTileBytes;
  static constexpr int kVOff = kKOff + kKStages * kTileBytes;
  static constexpr int kSmemBytes = kVOff + kVStages * kTileBytes + 1024;
  static_assert(kKStages <= 4 && kVStages <= 4, "barrier arrays");
  static_assert(kSmemBytes + 256 <= 227 * 1024, "shared memory per CTA");
  __device__ static constexpr uint32_t colS(int t) { return t ? 128u : 0u; }
  __device__ static constexpr uint32_t colO(int t) { return t ? 256u + D : 256u; }
  // P in columns of its own (d = 64: 2 x (128 S + 64 O + 64 P) = 512 columns)
  static constexpr bool kSepP = D == 64 && !F8;
  // With P in columns of its own, each Q tile gets an MMA issuer of its own (warps 9 and 10),
  // so that neither tile's products wait behind the other's in one issue order: 11% faster at
  // d = 64. At d = 128 the same split measured 28-42% slower: there S(j+1) follows PV(j) in
  // each tile, and the one issuer's fixed order keeps the two tiles' softmax phases apart.
  static constexpr bool kTwoIssuers = kSepP;
  static constexpr int kThreads = kTwoIssuers ? 352 : 320;
  __device__ static constexpr uint32_t colP(int t) { return kSepP ? 384u + 64u * t : colS(t); }
  static constexpr uint32_t kTmemCols = 512;
};

struct FwdParams {
  __nv_bfloat16* O;
  float* LSE;
  int* status;
  int Nq;       // query rows per head
  int Nk;       // key / value rows per head
  int heads;
  int qtiles;
  int kvtiles;
  int pairs;
  int causal;
  int offset;   // causal: query i hides keys j > i + offset (offset = Nk - Nq, bottom-right)
  int hides;    // some query may see no key at all (causal with Nq > Nk)
  float sl2;      // scale * log2(e) (* the Q and K factors for e4m3)
  float o_scale;  // V's factor for e4m3, else 1
  // additive mask (kMask): element (b, h, i, j) at mask[b*mask_sb + h*mask_sh + i*mask_srow + j]
  const __nv_bfloat16* mask;
  // boolean mask (kVar == 3): visibility bits, word (b, h, i, j / 32) at
  // bits[b*mask_sb + h*mask_sh + i*mask_srow + j / 32] (the same strides, in 32-bit words)
  const uint32_t* bits;
  int64_t mask_sb, mask_sh, mask_srow;
  int H;
  float inv_scale;  // 1 / scale: M joins the raw scores as M / scale
  // dropout (kVar == 2): Philox key, keep threshold and the scale of a kept weight
  uint32_t seed_lo, seed_hi, drop_tt;  // drop_tt: the keep threshold in all four bytes
  float drop_scale;
};

struct FwdCtl {
  uint64_t q_full;
  uint64_t k_full[4], v_full[4], k_empty[4], v_empty[4];
  uint64_t s_full[2], p_full[2], o_full[2];
  uint64_t s_free[2], pv_done[2];  // P in columns of its own: S_t loaded; PV_t(j) retired
  uint64_t drain;
  uint32_t tmem_base;
  int abort;
};

// kVar: 0 plain, 1 additive mask, 2 dropout, 3 boolean mask (packed bits).
template <int D, bool F8, int kVar>
__global__ void __launch_bounds__(FwdCfg<D, F8>::kThreads, 1)
fa_fwd_tc_kernel(const __grid_constant__ CUtensorMap tmQ, const __grid_constant__ CUtensorMap tmK,
                 const __grid_constant__ CUtensorMap tmV, const FwdParams p) {
  using C = FwdCfg<D, F8>;
  constexpr bool kMask = kVar == 1;
  constexpr bool kDrop = kVar == 2;
  constexpr bool kBits = kVar == 3;
  constexpr bool kHides = kMask || kBits;  // a row may have no visible key
  static_assert(!(F8 && kVar), "the e4m3 instance has no mask or dropout");
  extern __shared__ uint8_t smem_raw[];
  __shared__ FwdCtl ctl;
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

  int pair, head;
  if (p.causal) {  // heaviest pairs first
    pair = p.pairs - 1 - (int)(blockIdx.x / p.heads);
    head = (int)(blockIdx.x % p.heads);
  } else {
    pair = (int)(blockIdx.x % p.pairs);
    head = (int)(blockIdx.x / p.pairs);
  }
  const int qt0 = 2 * pair;
  const bool act1 = qt0 + 1 < p.qtiles;
  // K/V tiles Q tile qt sees: causal, up to the limit of its last query (none when even
  // that query sees no key, which only happens with more queries than keys)
  auto kv_tiles_of = [&](int qt) {
    if (!p.causal) return p.kvtiles;
    const int lim = min((qt + 1) * BM, p.Nq) - 1 + p.offset;
    return lim < 0 ? 0 : min(p.kvtiles, lim / BN + 1);
  };
  const int nkv0 = kv_tiles_of(qt0);
  const int nkv1 = act1 ? kv_tiles_of(qt0 + 1) : 0;
  const int nkv = max(nkv0, nkv1);
  const int row_base = head * p.Nq;
  if (nkv == 0) {
    // No query of this CTA sees a key: O = 0 and LSE = -inf, nothing else to do.
    if (warp < 8) {
      const int qrow = (qt0 + (warp >> 2)) * BM + (warp & 3) * 32 + lane;
      if ((warp >> 2) == 0 || act1) {
        if (qrow < p.Nq) {
          uint4* dst = reinterpret_cast<uint4*>(p.O + (size_t)(row_base + qrow) * D);
#pragma unroll
          for (int u = 0; u < D / 8; ++u) dst[u] = make_uint4(0, 0, 0, 0);
          p.LSE[row_base + qrow] = -INFINITY;
        }
      }
    }
    return;
  }

  if (threadIdx.x == 0) {
    mbar_init(&ctl.q_full, 1);
    for (int s = 0; s < 4; ++s) {
      mbar_init(&ctl.k_full[s], 1);
      mbar_init(&ctl.v_full[s], 1);
      mbar_init(&ctl.k_empty[s], C::kTwoIssuers && act1 ? 2 : 1);  // one arrival per issuer
      mbar_init(&ctl.v_empty[s], C::kTwoIssuers && act1 ? 2 : 1);
    }
    for (int t = 0; t < 2; ++t) {
      mbar_init(&ctl.s_full[t], 1);
      mbar_init(&ctl.p_full[t], 128);
      mbar_init(&ctl.o_full[t], 1);
      mbar_init(&ctl.s_free[t], 128);
      mbar_init(&ctl.pv_done[t], 1);
    }
    mbar_init(&ctl.drain, C::kTwoIssuers && act1 ? 2 : 1);
    ctl.abort = 0;
    fence_mbar_init();
  }
  if (warp == kMmaWarp) tmem_alloc(&ctl.tmem_base, C::kTmemCols);
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
      mbar_expect_tx(&ctl.q_full, (act1 ? 2 : 1) * C::kTileBytes);
      for (int t = 0; t < (act1 ? 2 : 1); ++t)
        for (int b = 0; b < C::kBoxes; ++b)
          tma_load_3d(smem + C::kQOff + (t * C::kBoxes + b) * kBoxBytes, &tmQ, &ctl.q_full, b * C::kBoxElems,
                      (qt0 + t) * BM, head);
      int last_k[4] = {-1, -1, -1, -1}, last_v[4] = {-1, -1, -1, -1};
      // Test hook of the failure path: never arm K_0, so the MMA thread's wait for it runs
      // out (see StatusBlock); off unless a test sets it.
      const bool skip_k0 = injected(p.status, kInjectFwd);
      // K_j's slot frees once the S products that read K_{j-stages} have run, V_j's once
      // the PV products have: K is read a whole tile earlier than V, so it loads earlier.
      for (int j = 0; j < nkv; ++j) {
        const int sk = j % C::kKStages, sv = j % C::kVStages;
        if (j >= C::kKStages && !mbar_wait(&ctl.k_empty[sk], ((j / C::kKStages) - 1) & 1, p.status, abort))
          break;
        if (j > 0 || !skip_k0) {
          mbar_expect_tx(&ctl.k_full[sk], C::kTileBytes);
          for (int b = 0; b < C::kBoxes; ++b)
            tma_load_3d(smem + C::kKOff + (sk * C::kBoxes + b) * kBoxBytes, &tmK, &ctl.k_full[sk],
                        b * C::kBoxElems, j * BN, head);
          last_k[sk] = j;
        }
        if (j >= C::kVStages && !mbar_wait(&ctl.v_empty[sv], ((j / C::kVStages) - 1) & 1, p.status, abort))
          break;
        mbar_expect_tx(&ctl.v_full[sv], C::kTileBytes);
        for (int b = 0; b < C::kBoxes; ++b)
          tma_load_3d(smem + C::kVOff + (sv * C::kBoxes + b) * kBoxBytes, &tmV, &ctl.v_full[sv], b * C::kBoxElems,
                      j * BN, head);
        last_v[sv] = j;
      }
      // Every issued copy must land before the CTA may exit.
      mbar_wait(&ctl.q_full, 0, p.status, nullptr);
      for (int s = 0; s < 4; ++s) {
        if (last_k[s] >= 0) mbar_wait(&ctl.k_full[s], (last_k[s] / C::kKStages) & 1, p.status, nullptr);
        if (last_v[s] >= 0) mbar_wait(&ctl.v_full[s], (last_v[s] / C::kVStages) & 1, p.status, nullptr);
      }
    }
  } else if (warp == kMmaWarp && !C::kTwoIssuers) {
    // One issuer for both Q tiles: S_t(j+1) right after PV_t(j), tile 0 first.
    if (lane == 0) {
      constexpr uint32_t idS = F8 ? idesc_e4m3(BM, BN, false, false) : idesc_bf16(BM, BN, false, false);
      constexpr uint32_t idO = F8 ? idesc_e4m3(BM, D, false, true) : idesc_bf16(BM, D, false, true);
      const uint32_t sQ = smem_u32(smem + C::kQOff);
      const uint32_t sK = smem_u32(smem + C::kKOff);
      const uint32_t sV = smem_u32(smem + C::kVOff);
      // Base descriptors; each MMA below only advances the start address.
      const uint64_t dQ0 = sdesc_sw128(sQ, 16, 1024);
      const uint64_t dK0 = sdesc_sw128(sK, 16, 1024);
      const uint64_t dV0 = sdesc_sw128(sV, kBoxBytes, 1024);
      auto issue_S = [&](int t, int s) {
        const uint32_t qo = t * C::kBoxes * kBoxBytes, ko = s * C::kBoxes * kBoxBytes;
#pragma unroll
        for (int k = 0; k < C::kSSteps; ++k) {  // 32 bytes of each row per step
          const uint32_t off = (k / 4) * kBoxBytes + (k % 4) * 32;
          if constexpr (F8)
            mma_ss_f8(tmem + C::colS(t), sdesc_add(dQ0, qo + off), sdesc_add(dK0, ko + off), idS, k > 0);
          else
            mma_ss(tmem + C::colS(t), sdesc_add(dQ0, qo + off), sdesc_add(dK0, ko + off), idS, k > 0);
        }
      };
      auto issue_PV = [&](int t, int s, bool acc) {
        const uint32_t vo = s * C::kBoxes * kBoxBytes;
        // K step = kKStep keys: 8 TMEM columns of packed P, kKStep 128-byte rows of V
#pragma unroll
        for (int k = 0; k < C::kPVSteps; ++k) {
          if constexpr (F8)
            mma_ts_f8(tmem + C::colO(t), tmem + C::colP(t) + k * 8, sdesc_add(dV0, vo + k * C::kKStep * 128), idO,
                      (acc || k > 0) ? 1u : 0u);
          else
            mma_ts(tmem + C::colO(t), tmem + C::colP(t) + k * 8, sdesc_add(dV0, vo + k * C::kKStep * 128), idO,
                   (acc || k > 0) ? 1u : 0u);
        }
      };
      bool ok = mbar_wait(&ctl.q_full, 0, p.status, abort) && mbar_wait(&ctl.k_full[0], 0, p.status, abort);
      if (ok) {
        tc_fence_after();
        if (nkv0 > 0) {
          issue_S(0, 0);
          mma_commit(&ctl.s_full[0]);
        }
        if (nkv1 > 0) {
          issue_S(1, 0);
          mma_commit(&ctl.s_full[1]);
        }
        mma_commit(&ctl.k_empty[0]);
      }
      for (int j = 0; ok && j < nkv; ++j) {
        const int s = j % C::kVStages;
        bool k_next = false;
        ok = mbar_wait(&ctl.v_full[s], (j / C::kVStages) & 1, p.status, abort);
        for (int t = 0; ok && t < 2; ++t) {
          const int nk = t ? nkv1 : nkv0;
          if (j >= nk) continue;
          if (!(ok = mbar_wait(&ctl.p_full[t], j & 1, p.status, abort))) break;
          tc_fence_after();
          issue_PV(t, s, j > 0);
          if (j + 1 < nk) {
            if (!k_next) {
              const int s2 = (j + 1) % C::kKStages;
              if (!(ok = mbar_wait(&ctl.k_full[s2], ((j + 1) / C::kKStages) & 1, p.status, abort))) break;
              tc_fence_after();
              k_next = true;
            }
            issue_S(t, (j + 1) % C::kKStages);
            mma_commit(&ctl.s_full[t]);
          } else {
            mma_commit(&ctl.o_full[t]);
          }
        }
        if (k_next) mma_commit(&ctl.k_empty[(j + 1) % C::kKStages]);  // every S of K_{j+1} issued
        mma_commit(&ctl.v_empty[s]);
      }
      // All MMAs must retire before TMEM is released.
      mma_commit(&ctl.drain);
      mbar_wait(&ctl.drain, 0, p.status, nullptr);
    }
  } else if (C::kTwoIssuers && (warp == kMmaWarp || warp == kMmaWarp + 1)) {
    // Issuer of Q tile t: S_t(j+1) as soon as the softmax warps have loaded S_t(j), then PV_t(j)
    // once P_t(j) is in. Each K/V stage is freed by one arrival per issuer; an issuer whose tile
    // sees fewer K/V tiles than its partner still arrives for the rest, each after that tile's
    // copy has landed (so never twice within one phase).
    const int t = warp - kMmaWarp;
    const int nk = t ? nkv1 : nkv0;
    if (lane == 0 && (t == 0 || act1)) {
      constexpr uint32_t idS = idesc_bf16(BM, BN, false, false);
      constexpr uint32_t idO = idesc_bf16(BM, D, false, true);
      // Base descriptors; each MMA below only advances the start address.
      const uint64_t dQ0 = sdesc_sw128(smem_u32(smem + C::kQOff) + t * C::kBoxes * kBoxBytes, 16, 1024);
      const uint64_t dK0 = sdesc_sw128(smem_u32(smem + C::kKOff), 16, 1024);
      const uint64_t dV0 = sdesc_sw128(smem_u32(smem + C::kVOff), kBoxBytes, 1024);
      const uint32_t colS = C::colS(t), colO = C::colO(t), colP = C::colP(t);
      auto issue_S = [&](int s) {
        const uint32_t ko = s * C::kBoxes * kBoxBytes;
#pragma unroll
        for (int k = 0; k < C::kSSteps; ++k) {  // 32 bytes of each row per step
          const uint32_t off = (k / 4) * kBoxBytes + (k % 4) * 32;
          mma_ss(tmem + colS, sdesc_add(dQ0, off), sdesc_add(dK0, ko + off), idS, k > 0);
        }
      };
      auto issue_PV = [&](int s, bool acc) {
        const uint32_t vo = s * C::kBoxes * kBoxBytes;
        // K step = kKStep keys: 8 TMEM columns of packed P, kKStep 128-byte rows of V
#pragma unroll
        for (int k = 0; k < C::kPVSteps; ++k)
          mma_ts(tmem + colO, tmem + colP + k * 8, sdesc_add(dV0, vo + k * C::kKStep * 128), idO,
                 (acc || k > 0) ? 1u : 0u);
      };
      auto k_wait = [&](int j) {
        return mbar_wait(&ctl.k_full[j % C::kKStages], (j / C::kKStages) & 1, p.status, abort);
      };
      bool ok = mbar_wait(&ctl.q_full, 0, p.status, abort) && k_wait(0);
      if (ok) {
        tc_fence_after();
        if (nk > 0) {
          issue_S(0);
          mma_commit(&ctl.s_full[t]);
          mma_commit(&ctl.k_empty[0]);
        } else {
          mbar_arrive(&ctl.k_empty[0]);
        }
      }
      for (int j = 0; ok && j < nkv; ++j) {
        const int s = j % C::kVStages, s2 = (j + 1) % C::kKStages;
        const bool mine = j < nk, next_mine = j + 1 < nk;
        if (j + 1 < nkv) {
          if (next_mine && !(ok = mbar_wait(&ctl.s_free[t], j & 1, p.status, abort))) break;
          if (!(ok = k_wait(j + 1))) break;
          if (next_mine) {
            tc_fence_after();
            issue_S(s2);
            mma_commit(&ctl.s_full[t]);
            mma_commit(&ctl.k_empty[s2]);
          } else {
            mbar_arrive(&ctl.k_empty[s2]);
          }
        }
        if (!(ok = mbar_wait(&ctl.v_full[s], (j / C::kVStages) & 1, p.status, abort))) break;
        if (mine) {
          if (!(ok = mbar_wait(&ctl.p_full[t], j & 1, p.status, abort))) break;
          tc_fence_after();
          issue_PV(s, j > 0);
          mma_commit(&ctl.pv_done[t]);
          if (!next_mine) mma_commit(&ctl.o_full[t]);
          mma_commit(&ctl.v_empty[s]);
        } else {
          mbar_arrive(&ctl.v_empty[s]);
        }
      }
      // All MMAs must retire before TMEM is released.
      mma_commit(&ctl.drain);
      mbar_wait(&ctl.drain, 0, p.status, nullptr);
    }
  } else {
    // ---------------- softmax warpgroups ----------------
    const int t = warp >> 2;
    const int nk = t ? nkv1 : nkv0;
    const int r = (warp & 3) * 32 + lane;       // row in the tile = TMEM lane
    const int qrow = (qt0 + t) * BM + r;        // query row in the head
    const uint32_t lane_off = (uint32_t)((warp & 3) * 32) << 16;
    const uint32_t tS = tmem + lane_off + C::colS(t);
    const uint32_t tO = tmem + lane_off + C::colO(t);
    const uint32_t tP = tmem + lane_off + C::colP(t);
    const float sl2 = p.sl2;
    float m = -INFINITY, l = 0.f;
    bool ok = nk > 0;
    // kMask: this row's mask values for the K tile about to be processed, 8 bf16 per
    // 16-byte load (rows of the mask are 16-byte aligned and padded to a multiple of 8);
    // rows and columns past the end of the head load nothing.
    uint4 mreg[kMask ? BN / 8 : 1];
    const __nv_bfloat16* mrow = nullptr;
    if constexpr (kMask) {
      if (qrow < p.Nq)
        mrow = p.mask + (int64_t)(head / p.H) * p.mask_sb + (int64_t)(head % p.H) * p.mask_sh +
               (int64_t)qrow * p.mask_srow;
#pragma unroll
      for (int c8 = 0; c8 < BN / 8; ++c8)
        mreg[c8] = (mrow && 8 * c8 < p.Nk && nk > 0) ? ld_global_v4_ordered(mrow + 8 * c8) : make_uint4(0, 0, 0, 0);
    }
    // kBits: this row's visibility bits for the K tile about to be processed (words
    // 4j .. 4j+3 of the row; rows hold at least 4 words per K tile of the head).
    uint4 breg = make_uint4(0, 0, 0, 0);
    const uint32_t* brow = nullptr;
    if constexpr (kBits) {
      if (qrow < p.Nq)
        brow = p.bits + (int64_t)(head / p.H) * p.mask_sb + (int64_t)(head % p.H) * p.mask_sh +
               (int64_t)qrow * p.mask_srow;
      if (brow && nk > 0) breg = ld_global_v4_ordered(brow);
    }
    // tcgen05.ld/st are warp-collective (.sync.aligned): every branch that guards one
    // is made uniform across the warp, including the outcome of each bounded wait.
    for (int j = 0; ok && j < nk; ++j) {
      // kDrop: keep bits of this row against the tile's 128 keys (bit c of word c / 32),
      // drawn before waiting for S so that the work overlaps the S product
      uint32_t keep[kDrop ? BN / 32 : 1];
      if constexpr (kDrop) {
#pragma unroll
        for (int w = 0; w < BN / 32; ++w) keep[w] = 0;
#pragma unroll
        for (int c16 = 0; c16 < BN / 16; ++c16)
          keep[c16 / 2] |= rng::keep16((uint32_t)(j * (BN / 16) + c16), (uint32_t)qrow, (uint32_t)head, p.seed_lo,
                                       p.seed_hi, p.drop_tt)
                           << (16 * (c16 % 2));
      }
      ok = __all_sync(0xffffffffu, mbar_wait(&ctl.s_full[t], j & 1, p.status, abort));
      if (!ok) break;
      tc_fence_after();
      float sv[BN];
      if constexpr (!kMask) {
        tmem_ld32x2(tS, tS + 32, *reinterpret_cast<float(*)[32]>(&sv[0]), *reinterpret_cast<float(*)[32]>(&sv[32]));
        tmem_ld32x2(tS + 64, tS + 96, *reinterpret_cast<float(*)[32]>(&sv[64]),
                    *reinterpret_cast<float(*)[32]>(&sv[96]));
      } else {
        // 32 columns at a time, each folded with its mask values at once, so the mask
        // registers free up as the scores arrive (the row and the prefetched mask do not
        // fit in registers together)
#pragma unroll
        for (int q = 0; q < BN / 32; ++q) {
          tmem_ld32(tS + 32 * q, *reinterpret_cast<float(*)[32]>(&sv[32 * q]));
#pragma unroll
          for (int c8 = 4 * q; c8 < 4 * q + 4; ++c8) {  // s += M / scale
            const uint32_t w[4] = {mreg[c8].x, mreg[c8].y, mreg[c8].z, mreg[c8].w};
#pragma unroll
            for (int u = 0; u < 4; ++u) {
              const float lo = __uint_as_float(w[u] << 16), hi = __uint_as_float(w[u] & 0xFFFF0000u);
              sv[8 * c8 + 2 * u] = fmaf(lo, p.inv_scale, sv[8 * c8 + 2 * u]);
              sv[8 * c8 + 2 * u + 1] = fmaf(hi, p.inv_scale, sv[8 * c8 + 2 * u + 1]);
            }
          }
        }
      }
      if constexpr (C::kSepP) {  // S_t is in registers: the next S may overwrite it
        tc_fence_before();
        mbar_arrive(&ctl.s_free[t]);
      }
      // kBits: keys whose bit is clear are hidden. (Skipping this for tiles whose bits are
      // all set measured 17% slower: the branch costs registers the loop needs.)
      if constexpr (kBits) {
        const uint32_t bw[4] = {breg.x, breg.y, breg.z, breg.w};
#pragma unroll
        for (int c = 0; c < BN; ++c)
          if (!((bw[c / 32] >> (c % 32)) & 1u)) sv[c] = -INFINITY;
      }
      // Hidden keys: key > query + offset (causal), and keys past the end of the head in
      // its last, partial tile (their rows were read as zeros). Keep columns c <= lim. With
      // Nq <= Nk and no mask every row keeps at least key 0 of its first tile visible.
      // (The test is tile-uniform: only the tiles that cross the limit of the tile's first
      // query, or the end of the keys, compute a per-row limit.)
      const bool diag = p.causal && j * BN + BN - 1 > (qt0 + t) * BM + p.offset;
      const int valid = p.Nk - j * BN;
      if (diag || valid < BN) {
        const int lim = min(diag ? qrow + p.offset - j * BN : BN - 1, valid - 1);
#pragma unroll
        for (int c = 0; c < BN; ++c)
          if (c > lim) sv[c] = -INFINITY;
      }
      // row max: four independent chains of 3-input max over columns 0..BN-1
      static_assert(BN % 8 == 0, "the chains take 8 columns per step");
      float mx0 = fmaxf(sv[0], sv[1]), mx1 = fmaxf(sv[2], sv[3]), mx2 = fmaxf(sv[4], sv[5]),
            mx3 = fmaxf(sv[6], sv[7]);
#pragma unroll
      for (int c = 8; c < BN; c += 8) {
        mx0 = fmax3(mx0, sv[c], sv[c + 1]);
        mx1 = fmax3(mx1, sv[c + 2], sv[c + 3]);
        mx2 = fmax3(mx2, sv[c + 4], sv[c + 5]);
        mx3 = fmax3(mx3, sv[c + 6], sv[c + 7]);
      }
      const float mx = fmaxf(fmaxf(mx0, mx1), fmaxf(mx2, mx3));
      const float m_new = fmaxf(m, mx * sl2);
      const bool grow = m_new > m + C::kThreshold;
      if (C::kSepP && j > 0) {  // PV_t(j-1) must have read P_t and added into O_t
        ok = __all_sync(0xffffffffu, mbar_wait(&ctl.pv_done[t], (j - 1) & 1, p.status, abort));
        if (!ok) break;
        tc_fence_after();
      }
      if (__any_sync(0xffffffffu, grow)) {
        const float corr = grow ? ex2(m - m_new) : 1.f;
        l *= corr;
        if (j > 0) {
#pragma unroll 1
          for (int c0 = 0; c0 < D; c0 += 32) {
            float ov[32];
            tmem_ld32(tO + c0, ov);
            uint32_t w0[16], w1[16];
#pragma unroll
            for (int u = 0; u < 16; ++u) {
              w0[u] = __float_as_uint(ov[u] * corr);
              w1[u] = __float_as_uint(ov[16 + u] * corr);
            }
            tmem_st16(tO + c0, w0);
            tmem_st16(tO + c0 + 16, w1);
          }
        }
        if (grow) m = m_new;
      }
      const float2 sl2v = make_float2(sl2, sl2);
      // a row with no visible key so far (only possible with a mask) exponentiates
      // against 0: its scores are all -inf, so every p is 0
      const float m_use = ((kHides || p.hides) && m == -INFINITY) ? 0.f : m;
      const float2 neg_m = make_float2(C::kPShift - m_use, C::kPShift - m_use);
      float2 rs0 = make_float2(0.f, 0.f), rs1 = make_float2(0.f, 0.f);
      if constexpr (!F8) {
#pragma unroll
        for (int q = 0; q < BN / 32; ++q) {
          uint32_t pk[16];
#pragma unroll
          for (int u = 0; u < 16; ++u) {
            const float2 x = ffma2(make_float2(sv[32 * q + 2 * u], sv[32 * q + 2 * u + 1]), sl2v, neg_m);
            const float2 pr = make_float2(ex2(x.x), ex2(x.y));
            if (u & 1)
              rs1 = fadd2(rs1, pr);
            else
              rs0 = fadd2(rs0, pr);
            if constexpr (kDrop) {  // dropped keys contribute no weight to O
              const uint32_t kb = keep[q] >> (2 * u);
              pk[u] = pack_bf16((kb & 1u) ? pr.x : 0.f, (kb & 2u) ? pr.y : 0.f);
            } else {
              pk[u] = pack_bf16(pr.x, pr.y);
            }
          }
          tmem_st16(tP + 16 * q, pk);
        }
      } else {
#pragma unroll
        for (int q = 0; q < BN / 64; ++q) {
          uint32_t pk[16];  // 64 keys, four e4m3 per column
#pragma unroll
          for (int u = 0; u < 16; ++u) {
            const float* v4 = &sv[64 * q + 4 * u];
            const float2 x0 = ffma2(make_float2(v4[0], v4[1]), sl2v, neg_m);
            const float2 x1 = ffma2(make_float2(v4[2], v4[3]), sl2v, neg_m);
            const float2 p0 = make_float2(ex2(x0.x), ex2(x0.y));
            const float2 p1 = make_float2(ex2(x1.x), ex2(x1.y));
            rs0 = fadd2(rs0, p0);
            rs1 = fadd2(rs1, p1);
            pk[u] = pack_e4m3x4(p0.x, p0.y, p1.x, p1.y);
          }
          tmem_st16(tP + 16 * q, pk);
        }
      }
      l += (rs0.x + rs0.y) + (rs1.x + rs1.y);
      if constexpr (kBits)  // the next tile's bits land while its S is computed
        breg = (brow && j + 1 < nk) ? ld_global_v4_ordered(brow + 4 * (j + 1)) : make_uint4(0, 0, 0, 0);
      if constexpr (kMask) {  // the next tile's mask lands while its S is computed
#pragma unroll
        for (int c8 = 0; c8 < BN / 8; ++c8) {
          const int col = (j + 1) * BN + 8 * c8;
          mreg[c8] = (mrow && col < p.Nk && j + 1 < nk) ? ld_global_v4_ordered(mrow + col) : make_uint4(0, 0, 0, 0);
        }
      }
      tmem_wait_st();
      tc_fence_before();
      mbar_arrive(&ctl.p_full[t]);
    }
    if (ok) ok = __all_sync(0xffffffffu, mbar_wait(&ctl.o_full[t], 0, p.status, abort));
    if (ok) {
      tc_fence_after();
      const float inv_l = (!(kHides || p.hides) || l > 0.f) ? (kDrop ? p.drop_scale : p.o_scale) / l : 0.f;  // no visible key: O = 0
      __nv_bfloat16* orow = p.O + (size_t)(row_base + qrow) * D;
#pragma unroll 1
      for (int c0 = 0; c0 < D; c0 += 32) {
        float ov[32];
        tmem_ld32(tO + c0, ov);
        uint4 w[4];
        uint32_t* wu = reinterpret_cast<uint32_t*>(w);
#pragma unroll
        for (int u = 0; u < 16; ++u) wu[u] = pack_bf16(ov[2 * u] * inv_l, ov[2 * u + 1] * inv_l);
        uint4* dst = reinterpret_cast<uint4*>(orow + c0);
        if (qrow < p.Nq) {  // rows past the end of the head belong to no query
#pragma unroll
          for (int u = 0; u < 4; ++u) dst[u] = w[u];
        }
      }
      if (qrow < p.Nq) p.LSE[row_base + qrow] = (m - C::kPShift + log2f(l)) * kLn2;
    } else if (nk == 0 && qrow < p.Nq) {
      // this Q tile sees no key (its CTA partner does): O = 0, LSE = -inf
      uint4* dst = reinterpret_cast<uint4*>(p.O + (size_t)(row_base + qrow) * D);
#pragma unroll
      for (int u = 0; u < D / 8; ++u) dst[u] = make_uint4(0, 0, 0, 0);
      p.LSE[row_base + qrow] = -INFINITY;
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

struct MaskArg {
  const void* ptr = nullptr;
  int64_t sb = 0, sh = 0, srow = 0;
};

struct DropArg {
  uint64_t seed = 0;
  uint32_t t = 0;
};

template <int D, bool F8, int kVar>
cudaError_t launch(const void* Q, const void* K, const void* V, void* O, float* LSE, const Shape& s,
                   float scale, float sl2, float o_scale, bool causal, const MaskArg& mask, const DropArg& drop,
                   int* status, cudaStream_t st) {
  using C = FwdCfg<D, F8>;
  CUtensorMap mq, mk, mv;
  const int64_t heads = s.heads();
  bool maps;
  if constexpr (F8)
    maps = make_map_u8_3d(&mq, Q, heads, s.N, D, BM) && make_map_u8_3d(&mk, K, heads, s.keys(), D, BN) &&
           make_map_u8_3d(&mv, V, heads, s.keys(), D, BN);
  else
    maps = make_map_bf16_3d(&mq, Q, heads, s.N, D, BM) && make_map_bf16_3d(&mk, K, heads, s.keys(), D, BN) &&
           make_map_bf16_3d(&mv, V, heads, s.keys(), D, BN);
  if (!maps) return cudaErrorInvalidValue;
  static bool attr = [] {
    return cudaFuncSetAttribute(fa_fwd_tc_kernel<D, F8, kVar>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                C::kSmemBytes) == cudaSuccess;
  }();
  if (!attr) return cudaErrorInvalidConfiguration;
  FwdParams p;
  p.O = static_cast<__nv_bfloat16*>(O);
  p.LSE = LSE;
  p.status = status;
  p.Nq = s.N;
  p.Nk = s.keys();
  p.heads = (int)s.heads();
  p.qtiles = (s.N + BM - 1) / BM;
  p.kvtiles = (s.keys() + BN - 1) / BN;
  p.pairs = (p.qtiles + 1) / 2;
  p.causal = causal ? 1 : 0;
  p.offset = causal ? s.keys() - s.N : 0;
  p.hides = causal && s.N > s.keys() ? 1 : 0;
  p.sl2 = sl2;
  p.o_scale = o_scale;
  p.mask = static_cast<const __nv_bfloat16*>(mask.ptr);
  p.bits = static_cast<const uint32_t*>(mask.ptr);
  p.mask_sb = mask.sb;
  p.mask_sh = mask.sh;
  p.mask_srow = mask.srow;
  p.H = s.H;
  p.inv_scale = 1.f / scale;
  p.seed_lo = (uint32_t)(drop.seed & 0xFFFFFFFFu);
  p.seed_hi = (uint32_t)(drop.seed >> 32);
  p.drop_tt = drop.t * 0x01010101u;
  p.drop_scale = (float)(256.0 / (256.0 - (double)drop.t));
  const int64_t grid = (int64_t)p.pairs * p.heads;
  fa_fwd_tc_kernel<D, F8, kVar><<<(unsigned)grid, C::kThreads, C::kSmemBytes, st>>>(mq, mk, mv, p);
  return cudaGetLastError();
}

constexpr float kLog2e = 1.4426950408889634f;

}  // namespace

cudaError_t tc_fwd(const void* Q, const void* K, const void* V, void* O, float* LSE, const Shape& s,
                   float scale, bool causal, int* status, cudaStream_t st) {
  const MaskArg none;
  const DropArg nodrop;
  return s.d == 64
             ? launch<64, false, 0>(Q, K, V, O, LSE, s, scale, scale * kLog2e, 1.f, causal, none, nodrop, status, st)
             : launch<128, false, 0>(Q, K, V, O, LSE, s, scale, scale * kLog2e, 1.f, causal, none, nodrop, status, st);
}

cudaError_t tc_fwd_masked(const void* Q, const void* K, const void* V, void* O, float* LSE, const Shape& s,
                          float scale, bool causal, const void* mask, int64_t mask_sb, int64_t mask_sh,
                          int64_t mask_srow, int* status, cudaStream_t st) {
  MaskArg m;
  m.ptr = mask;
  m.sb = mask_sb;
  m.sh = mask_sh;
  m.srow = mask_srow;
  const DropArg nodrop;
  return s.d == 64
             ? launch<64, false, 1>(Q, K, V, O, LSE, s, scale, scale * kLog2e, 1.f, causal, m, nodrop, status, st)
             : launch<128, false, 1>(Q, K, V, O, LSE, s, scale, scale * kLog2e, 1.f, causal, m, nodrop, status, st);
}

cudaError_t tc_fwd_bitmask(const void* Q, const void* K, const void* V, void* O, float* LSE, const Shape& s,
                           float scale, bool causal, const uint32_t* bits, int64_t bits_sb, int64_t bits_sh,
                           int64_t bits_srow, int* status, cudaStream_t st) {
  MaskArg m;
  m.ptr = bits;
  m.sb = bits_sb;
  m.sh = bits_sh;
  m.srow = bits_srow;
  const DropArg nodrop;
  return s.d == 64
             ? launch<64, false, 3>(Q, K, V, O, LSE, s, scale, scale * kLog2e, 1.f, causal, m, nodrop, status, st)
             : launch<128, false, 3>(Q, K, V, O, LSE, s, scale, scale * kLog2e, 1.f, causal, m, nodrop, status, st);
}

cudaError_t tc_fwd_dropout(const void* Q, const void* K, const void* V, void* O, float* LSE, const Shape& s,
                           float scale, bool causal, uint64_t seed, uint32_t threshold, int* status,
                           cudaStream_t st) {
  const MaskArg none;
  DropArg dr;
  dr.seed = seed;
  dr.t = threshold;
  return s.d == 64
             ? launch<64, false, 2>(Q, K, V, O, LSE, s, scale, scale * kLog2e, 1.f, causal, none, dr, status, st)
             : launch<128, false, 2>(Q, K, V, O, LSE, s, scale, scale * kLog2e, 1.f, causal, none, dr, status, st);
}

cudaError_t tc_fwd_fp8(const void* Q, const void* K, const void* V, void* O, float* LSE, const Shape& s,
                       float scale, bool causal, float q_descale, float k_descale, float v_descale,
                       int* status, cudaStream_t st) {
  const MaskArg none;
  const DropArg nodrop;
  return launch<128, true, 0>(Q, K, V, O, LSE, s, scale, scale * kLog2e * q_descale * k_descale, v_descale,
                              causal, none, nodrop, status, st);
}

}  // namespace fa
