// Internal declarations shared by the library's translation units (not part of the ABI).
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include <mutex>

#include "../../include/fa.h"

namespace fa {

// Sizes of one call, validated on the host. N is the number of query rows per head; Nk,
// when set (> 0), the number of key/value rows, which is otherwise N as well.
struct Shape {
  int B, H, N, d;
  int Nk = 0;
  int keys() const { return Nk > 0 ? Nk : N; }
  int64_t heads() const { return (int64_t)B * H; }
  int64_t rows() const { return heads() * N; }
  int64_t elems() const { return rows() * d; }
  int64_t key_elems() const { return heads() * keys() * d; }
};

// Device status word: bounded waits that give up write FA_ERR_DEVICE_TIMEOUT here.
// Defined in fa_api.cu; kernels in other units reach it through this pointer, which
// fa_api.cu resolves once per device context.
int* device_status_ptr();

// Unique ID of the calling thread's current CUDA context (0 if there is none or the
// query fails).
unsigned long long current_context_id();

// Device addresses of a __device__ variable, one per device, each valid for the context it
// was looked up in: a lookup is repeated when the device's current context has changed
// (after cudaDeviceReset, symbols move with the new context).
struct DeviceAddressCache {
  static constexpr int kDevices = 64;
  struct Entry {
    void* ptr = nullptr;
    unsigned long long ctx = 0;
  };
  std::mutex mu;
  Entry entry[kDevices];
};

// The current device's address of `symbol` (a __device__ variable of the calling
// translation unit, passed as its host-side stand-in), from `cache` when its context is
// unchanged; nullptr on failure.
void* symbol_address_cached(const void* symbol, DeviceAddressCache& cache);

// ---- exact FFMA path (fa_simt.cu): float32 inputs only (bf16 runs on the tensor cores) ----
cudaError_t simt_fwd(const void* Q, const void* K, const void* V, void* O, float* LSE,
                     const Shape& s, float scale, bool causal, cudaStream_t st);
cudaError_t simt_bwd(const void* Q, const void* K, const void* V, const void* dO,
                     const float* LSE, const float* D, void* dQ, void* dK, void* dV,
                     const Shape& s, float scale, bool causal, cudaStream_t st);

// ---- tcgen05 tensor-core path (bf16, d in {64, 128}, N % 128 == 0) ----
cudaError_t tc_fwd(const void* Q, const void* K, const void* V, void* O, float* LSE, const Shape& s,
                   float scale, bool causal, int* status, cudaStream_t st);
// bf16 forward with an additive bf16 mask: element (b, h, i, j) at
// mask[b*mask_sb + h*mask_sh + i*mask_srow + j] (strides in elements, multiples of 8).
cudaError_t tc_fwd_masked(const void* Q, const void* K, const void* V, void* O, float* LSE, const Shape& s,
                          float scale, bool causal, const void* mask, int64_t mask_sb, int64_t mask_sh,
                          int64_t mask_srow, int* status, cudaStream_t st);
// bf16 forward with a boolean mask packed one bit per key: query i sees key j iff bit j % 32
// of word bits[b*bits_sb + h*bits_sh + i*bits_srow + j / 32] is set (strides in 32-bit words,
// multiples of 4; rows hold at least 4 words per 128-key tile).
cudaError_t tc_fwd_bitmask(const void* Q, const void* K, const void* V, void* O, float* LSE, const Shape& s,
                           float scale, bool causal, const uint32_t* bits, int64_t bits_sb, int64_t bits_sh,
                           int64_t bits_srow, int* status, cudaStream_t st);
// bf16 forward with dropout: Philox-4x32-10 keep bits keyed by `seed`, kept iff the 8-bit
// uniform is >= threshold; kept weights scaled by 256 / (256 - threshold).
cudaError_t tc_fwd_dropout(const void* Q, const void* K, const void* V, void* O, float* LSE, const Shape& s,
                           float scale, bool causal, uint64_t seed, uint32_t threshold, int* status,
                           cudaStream_t st);
// e4m3 Q, K, V (d = 128) with per-tensor dequantisation factors; O bf16, LSE fp32.
cudaError_t tc_fwd_fp8(const void* Q, const void* K, const void* V, void* O, float* LSE, const Shape& s,
                       float scale, bool causal, float q_descale, float k_descale, float v_descale,
                       int* status, cudaStream_t st);
// dQacc: fp32 [B*H*N, d] workspace; zeroed, accumulated and converted inside the call.
cudaError_t tc_bwd(const void* Q, const void* K, const void* V, const void* dO, const float* LSE,
                   const float* D, void* dQ, void* dK, void* dV, float* dQacc, const Shape& s,
                   float scale, bool causal, int* status, cudaStream_t st);

// What a backward call adds to plain attention: an additive bf16 mask or a packed boolean
// mask (pointer and strides, as for tc_fwd_masked / tc_fwd_bitmask), or dropout (Philox key
// and keep threshold, as for tc_fwd_dropout).
struct BwdVariant {
  int kind = 0;  // 0 plain, 1 additive mask, 2 dropout, 3 boolean mask (packed bits)
  const void* mask = nullptr;
  int64_t sb = 0, sh = 0, srow = 0;
  uint64_t seed = 0;
  uint32_t threshold = 0;
};

// The backward kernel alone (no zeroing, no convert), on 128-query tiles (fa_bwd_wide.cu;
// d = 64 or 128): dQacc must be zero on entry and receives the unscaled fp32 dQ sums. With
// dQacc null (plain attention only) it computes dK and dV alone.
cudaError_t tc_bwd_wide(const void* Q, const void* K, const void* V, const void* dO, const float* LSE,
                        const float* Dv, void* dK, void* dV, float* dQacc, const Shape& s, float scale, bool causal,
                        const BwdVariant& var, int* status, cudaStream_t st);

// The separate dQ pass (fa_bwd_dq.cu; d = 64 or 128, plain attention): dQ in bf16, written
// directly, from the same inputs as tc_bwd_wide.
cudaError_t tc_bwd_dq(const void* Q, const void* K, const void* V, const void* dO, const float* LSE,
                      const float* Dv, void* dQ, const Shape& s, float scale, bool causal, int* status,
                      cudaStream_t st);

// How tc_bwd computes dQ (fa_set_bwd_dq_mode): FA_BWD_DQ_AUTO, _ATOMIC or _SEPARATE.
int bwd_dq_mode();
void set_bwd_dq_mode(int mode);

// The backward with the additive mask of tc_fwd_masked.
cudaError_t tc_bwd_masked(const void* Q, const void* K, const void* V, const void* dO, const float* LSE,
                          const float* D, void* dQ, void* dK, void* dV, float* dQacc, const Shape& s,
                          float scale, bool causal, const void* mask, int64_t mask_sb, int64_t mask_sh,
                          int64_t mask_srow, int* status, cudaStream_t st);

// The backward with the boolean mask of tc_fwd_bitmask.
cudaError_t tc_bwd_bitmask(const void* Q, const void* K, const void* V, const void* dO, const float* LSE,
                           const float* D, void* dQ, void* dK, void* dV, float* dQacc, const Shape& s,
                           float scale, bool causal, const uint32_t* bits, int64_t bits_sb, int64_t bits_sh,
                           int64_t bits_srow, int* status, cudaStream_t st);

// The backward with the dropout of tc_fwd_dropout (same seed and threshold).
cudaError_t tc_bwd_dropout(const void* Q, const void* K, const void* V, const void* dO, const float* LSE,
                           const float* D, void* dQ, void* dK, void* dV, float* dQacc, const Shape& s,
                           float scale, bool causal, uint64_t seed, uint32_t threshold, int* status,
                           cudaStream_t st);

// ---- split-KV forward for few queries (fa_splitkv.cu): bf16, d = 64 or 128, Nq <= 64 ----
size_t splitkv_workspace_floats(int64_t heads, int Nq, int Nk, int d);
cudaError_t splitkv_fwd(const void* Q, const void* K, const void* V, void* O, float* LSE, int64_t heads,
                        int Nq, int Nk, int d, float scale, bool causal, float* workspace, int* status,
                        cudaStream_t st);

// tcgen05 partial kernel (fa_splitkv_tc.cu): ctas CTA ranges of L keys each over the
// flattened (head, key) sequence; writes part_o [heads][P][Nq][d] and part_ml
// [heads][P][Nq][2] = (m in log2 units, l), merged by fa_splitkv.cu.
cudaError_t splitkv_tc_partial(const void* Q, const void* K, const void* V, int64_t heads, int Nq, int Nk, int d,
                               float scale, bool causal, int64_t L, int ctas, int P, float* part_o, float* part_ml,
                               int* status, cudaStream_t st);

// ---- memory-bound helpers (fa_simt.cu) ----
cudaError_t preprocess_d(const void* O, const void* dO, float* D, const Shape& s, bool bf16,
                         cudaStream_t st);

}  // namespace fa
