// C ABI entry points: argument checks, dispatch to the kernels, status reporting.
#include <math.h>
#include <mutex>

#include "fa_internal.h"
#include "sm100_ptx.cuh"

namespace fa {

// Per device: the status word (0 or FA_ERR_DEVICE_TIMEOUT) and the failure-path test hooks.
__device__ ptx::StatusBlock g_device_block;

unsigned long long current_context_id() {
  using GetCurrent = CUresult (*)(CUcontext*);
  using GetId = CUresult (*)(CUcontext, unsigned long long*);
  static const GetCurrent get_current = [] {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q{};
    return cudaGetDriverEntryPointByVersion("cuCtxGetCurrent", &p, 12000, cudaEnableDefault, &q) == cudaSuccess &&
                   q == cudaDriverEntryPointSuccess
               ? reinterpret_cast<GetCurrent>(p)
               : nullptr;
  }();
  static const GetId get_id = [] {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q{};
    return cudaGetDriverEntryPointByVersion("cuCtxGetId", &p, 12000, cudaEnableDefault, &q) == cudaSuccess &&
                   q == cudaDriverEntryPointSuccess
               ? reinterpret_cast<GetId>(p)
               : nullptr;
  }();
  CUcontext ctx = nullptr;
  unsigned long long id = 0;
  if (!get_current || !get_id || get_current(&ctx) != CUDA_SUCCESS || !ctx || get_id(ctx, &id) != CUDA_SUCCESS)
    return 0;
  return id;
}

void* symbol_address_cached(const void* symbol, DeviceAddressCache& cache) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= DeviceAddressCache::kDevices) return nullptr;
  std::lock_guard<std::mutex> lock(cache.mu);
  DeviceAddressCache::Entry& e = cache.entry[dev];
  const unsigned long long ctx = current_context_id();
  if (e.ptr && ctx != 0 && ctx == e.ctx) return e.ptr;
  // First use on this device, or a new context (e.g. after cudaDeviceReset): look it up.
  // The lookup makes the device's primary context current if none was.
  void* p = nullptr;
  if (cudaGetSymbolAddress(&p, symbol) != cudaSuccess) return nullptr;
  e.ptr = p;
  e.ctx = current_context_id();
  return p;
}

int* device_status_ptr() {
  static DeviceAddressCache cache;
  void* block = symbol_address_cached(&g_device_block, cache);
  return block ? &static_cast<ptx::StatusBlock*>(block)->status : nullptr;
}

namespace {

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

// Checks sizes, dtype and scale. s.N is the query length; s.keys() the key length (s.Nk
// is 0 for the square entry points, which makes it N as well; a negative s.Nk is invalid).
fa_status_t check_shape(const Shape& s, int dtype, float* scale) {
  if (s.B < 1 || s.H < 1 || s.N < 1 || s.d < 1 || s.Nk < 0) return FA_ERR_INVALID_ARG;
  if (dtype != FA_DTYPE_BF16 && dtype != FA_DTYPE_FP32) return FA_ERR_INVALID_ARG;
  // B*H*N*d must be representable; keep B*H below 2^31 and the element count < 2^60.
  const int64_t bh = (int64_t)s.B * s.H;
  const int64_t longest = s.N > s.keys() ? s.N : s.keys();
  if (bh >= (int64_t(1) << 31)) return FA_ERR_INVALID_ARG;
  if (bh * longest > (int64_t(1) << 50) || bh * longest * s.d > (int64_t(1) << 60)) return FA_ERR_INVALID_ARG;
  if (scale && !(isfinite(*scale) && *scale > 0.f)) return FA_ERR_INVALID_ARG;
  if (s.d != 64 && s.d != 128) return FA_ERR_UNSUPPORTED;
  // TMA coordinates are 32-bit row indices into the [B*H*rows, d] views.
  if (dtype == FA_DTYPE_BF16 && bh * longest > INT32_MAX) return FA_ERR_UNSUPPORTED;
  if (dtype == FA_DTYPE_FP32 && longest > 4096) return FA_ERR_UNSUPPORTED;
  return FA_OK;
}

fa_status_t check_ptrs(std::initializer_list<const void*> ps) {
  for (const void* p : ps)
    if (!p || !aligned16(p)) return FA_ERR_INVALID_ARG;
  return FA_OK;
}

fa_status_t from_cuda(cudaError_t e) { return e == cudaSuccess ? FA_OK : FA_ERR_CUDA; }

}  // namespace
}  // namespace fa

using fa::Shape;

namespace fa {
namespace {
fa_status_t fwd_common(const void* Q, const void* K, const void* V, void* O, float* LSE, const Shape& s,
                       float scale, int causal, int dtype, void* stream) {
  fa_status_t r = check_shape(s, dtype, &scale);
  if (r != FA_OK) return r;
  if ((r = check_ptrs({Q, K, V, O, LSE})) != FA_OK) return r;
  if (causal != 0 && causal != 1) return FA_ERR_INVALID_ARG;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  if (dtype == FA_DTYPE_BF16) {
    int* status = device_status_ptr();
    if (!status) return FA_ERR_CUDA;
    return from_cuda(tc_fwd(Q, K, V, O, LSE, s, scale, causal == 1, status, st));
  }
  return from_cuda(simt_fwd(Q, K, V, O, LSE, s, scale, causal == 1, st));
}
}  // namespace
}  // namespace fa

extern "C" fa_status_t fa_fwd_rect(const void* Q, const void* K, const void* V, void* O, float* LSE, int B,
                                   int H, int Nq, int Nk, int d, float scale, int causal, int dtype,
                                   void* stream) {
  if (Nk < 1) return FA_ERR_INVALID_ARG;
  Shape s{B, H, Nq, d};
  s.Nk = Nk;
  return fa::fwd_common(Q, K, V, O, LSE, s, scale, causal, dtype, stream);
}

extern "C" fa_status_t fa_fwd(const void* Q, const void* K, const void* V, void* O, float* LSE,
                              int B, int H, int N, int d, float scale, int causal, int dtype,
                              void* stream) {
  return fa::fwd_common(Q, K, V, O, LSE, Shape{B, H, N, d}, scale, causal, dtype, stream);
}

extern "C" fa_status_t fa_fwd_fp8(const void* Q, const void* K, const void* V, void* O, float* LSE,
                                  int B, int H, int N, int d, float scale, int causal, float q_descale,
                                  float k_descale, float v_descale, void* stream) {
  const Shape s{B, H, N, d};
  // The bf16 checks cover sizes, scale and the 32-bit row limit; d is narrower here.
  fa_status_t r = fa::check_shape(s, FA_DTYPE_BF16, &scale);
  if (r != FA_OK) return r;
  for (float f : {q_descale, k_descale, v_descale})
    if (!(isfinite(f) && f > 0.f)) return FA_ERR_INVALID_ARG;
  if (causal != 0 && causal != 1) return FA_ERR_INVALID_ARG;
  if ((r = fa::check_ptrs({Q, K, V, O, LSE})) != FA_OK) return r;
  if (d != 128) return FA_ERR_UNSUPPORTED;
  int* status = fa::device_status_ptr();
  if (!status) return FA_ERR_CUDA;
  return fa::from_cuda(fa::tc_fwd_fp8(Q, K, V, O, LSE, s, scale, causal == 1, q_descale, k_descale, v_descale,
                                      status, static_cast<cudaStream_t>(stream)));
}

extern "C" fa_status_t fa_bwd_preprocess(const void* O, const void* dO, float* D, int B, int H,
                                         int N, int d, int dtype, void* stream) {
  const Shape s{B, H, N, d};
  fa_status_t r = fa::check_shape(s, dtype, nullptr);
  if (r != FA_OK) return r;
  if ((r = fa::check_ptrs({O, dO, D})) != FA_OK) return r;
  return fa::from_cuda(
      fa::preprocess_d(O, dO, D, s, dtype == FA_DTYPE_BF16, static_cast<cudaStream_t>(stream)));
}

extern "C" size_t fa_bwd_workspace_size(int B, int H, int N, int d, int dtype) {
  const Shape s{B, H, N, d};
  if (fa::check_shape(s, dtype, nullptr) != FA_OK) return 0;
  return dtype == FA_DTYPE_BF16 ? (size_t)s.elems() * sizeof(float) : 0;
}

namespace fa {
namespace {

struct Mask {
  const void* ptr;
  int64_t sb, sh, srow;
};

// The mask's rows are read in 16-byte pieces: the base must be 16-byte aligned, every
// stride a non-negative multiple of 8 elements, and each row must hold N rounded up to 8.
fa_status_t check_mask(const Mask& m, const Shape& s, int dtype) {
  if (!m.ptr || !aligned16(m.ptr)) return FA_ERR_INVALID_ARG;
  if (m.sb < 0 || m.sh < 0 || m.sb % 8 || m.sh % 8 || m.srow % 8) return FA_ERR_INVALID_ARG;
  if (m.srow < ((int64_t)s.N + 7) / 8 * 8) return FA_ERR_INVALID_ARG;
  if (dtype != FA_DTYPE_BF16) return FA_ERR_UNSUPPORTED;
  return FA_OK;
}

// Packed visibility bits: each 128-key tile of a row is read as one 16-byte piece, so the
// base must be 16-byte aligned, every stride a non-negative multiple of 4 words, and each
// row must hold 4 words per 128-key tile of the head.
fa_status_t check_bits(const Mask& m, const Shape& s, int dtype) {
  if (!m.ptr || !aligned16(m.ptr)) return FA_ERR_INVALID_ARG;
  if (m.sb < 0 || m.sh < 0 || m.sb % 4 || m.sh % 4 || m.srow % 4) return FA_ERR_INVALID_ARG;
  if (m.srow < ((int64_t)s.N + 127) / 128 * 4) return FA_ERR_INVALID_ARG;
  if (dtype != FA_DTYPE_BF16) return FA_ERR_UNSUPPORTED;
  return FA_OK;
}

struct Drop {
  uint64_t seed;
  uint32_t t;  // keep iff the 8-bit uniform >= t
};

// Dropout probability p in [0, 1) -> 8-bit keep threshold round(p * 256), at most 255.
fa_status_t drop_threshold(float p, int dtype, uint32_t* t) {
  if (!(isfinite(p) && p >= 0.f && p < 1.f)) return FA_ERR_INVALID_ARG;
  if (dtype != FA_DTYPE_BF16) return FA_ERR_UNSUPPORTED;
  const double r = floor((double)p * 256.0 + 0.5);
  *t = (uint32_t)(r > 255.0 ? 255.0 : r);
  return FA_OK;
}

fa_status_t bwd_common(const void* Q, const void* K, const void* V, const void* O, const void* dO,
                       const float* LSE, const float* D, void* dQ, void* dK, void* dV, void* workspace,
                       size_t workspace_bytes, int B, int H, int N, int d, float scale, int causal, int dtype,
                       const Mask* mask, const Drop* drop, void* stream, const Mask* bits = nullptr, int Nk = 0) {
  Shape s{B, H, N, d};
  s.Nk = Nk;
  fa_status_t r = check_shape(s, dtype, &scale);
  if (r != FA_OK) return r;
  if ((r = check_ptrs({Q, K, V, O, dO, LSE, dQ, dK, dV})) != FA_OK) return r;
  if (D && !aligned16(D)) return FA_ERR_INVALID_ARG;
  if (causal != 0 && causal != 1) return FA_ERR_INVALID_ARG;
  if (mask && (r = check_mask(*mask, s, dtype)) != FA_OK) return r;
  if (bits && (r = check_bits(*bits, s, dtype)) != FA_OK) return r;
  const size_t need = fa_bwd_workspace_size(B, H, N, d, dtype);
  const size_t need_d = D ? 0 : (size_t)s.rows() * sizeof(float);
  if (need + need_d > 0) {
    if (!workspace || workspace_bytes < need + need_d) return FA_ERR_WORKSPACE;
    if (!aligned16(workspace)) return FA_ERR_INVALID_ARG;
  }
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  const bool bf16 = dtype == FA_DTYPE_BF16;
  if (!D) {
    float* Dw = reinterpret_cast<float*>(static_cast<char*>(workspace) + need);
    if ((r = from_cuda(preprocess_d(O, dO, Dw, s, bf16, st))) != FA_OK) return r;
    D = Dw;
  }
  if (bf16) {
    int* status = device_status_ptr();
    if (!status) return FA_ERR_CUDA;
    float* acc = static_cast<float*>(workspace);
    if (mask)
      return from_cuda(tc_bwd_masked(Q, K, V, dO, LSE, D, dQ, dK, dV, acc, s, scale, causal == 1, mask->ptr,
                                     mask->sb, mask->sh, mask->srow, status, st));
    if (bits)
      return from_cuda(tc_bwd_bitmask(Q, K, V, dO, LSE, D, dQ, dK, dV, acc, s, scale, causal == 1,
                                      static_cast<const uint32_t*>(bits->ptr), bits->sb, bits->sh, bits->srow,
                                      status, st));
    if (drop)
      return from_cuda(tc_bwd_dropout(Q, K, V, dO, LSE, D, dQ, dK, dV, acc, s, scale, causal == 1, drop->seed,
                                      drop->t, status, st));
    return from_cuda(tc_bwd(Q, K, V, dO, LSE, D, dQ, dK, dV, acc, s, scale, causal == 1, status, st));
  }
  return from_cuda(simt_bwd(Q, K, V, dO, LSE, D, dQ, dK, dV, s, scale, causal == 1, st));
}

}  // namespace
}  // namespace fa

extern "C" fa_status_t fa_bwd(const void* Q, const void* K, const void* V, const void* O,
                              const void* dO, const float* LSE, const float* D, void* dQ,
                              void* dK, void* dV, void* workspace, size_t workspace_bytes, int B,
                              int H, int N, int d, float scale, int causal, int dtype,
                              void* stream) {
  return fa::bwd_common(Q, K, V, O, dO, LSE, D, dQ, dK, dV, workspace, workspace_bytes, B, H, N, d, scale, causal,
                        dtype, nullptr, nullptr, stream);
}

extern "C" size_t fa_bwd_rect_workspace_size(int B, int H, int Nq, int Nk, int d, int dtype) {
  if (Nk < 1) return 0;
  Shape s{B, H, Nq, d};
  s.Nk = Nk;
  if (fa::check_shape(s, dtype, nullptr) != FA_OK) return 0;
  return dtype == FA_DTYPE_BF16 ? (size_t)s.elems() * sizeof(float) : 0;
}

extern "C" fa_status_t fa_bwd_rect(const void* Q, const void* K, const void* V, const void* O, const void* dO,
                                   const float* LSE, const float* D, void* dQ, void* dK, void* dV, void* workspace,
                                   size_t workspace_bytes, int B, int H, int Nq, int Nk, int d, float scale,
                                   int causal, int dtype, void* stream) {
  if (Nk < 1) return FA_ERR_INVALID_ARG;
  return fa::bwd_common(Q, K, V, O, dO, LSE, D, dQ, dK, dV, workspace, workspace_bytes, B, H, Nq, d, scale, causal,
                        dtype, nullptr, nullptr, stream, nullptr, Nk);
}

extern "C" fa_status_t fa_fwd_masked(const void* Q, const void* K, const void* V, void* O, float* LSE,
                                     const void* mask, long long mask_stride_b, long long mask_stride_h,
                                     long long mask_stride_row, int B, int H, int N, int d, float scale,
                                     int causal, int dtype, void* stream) {
  const Shape s{B, H, N, d};
  fa_status_t r = fa::check_shape(s, dtype, &scale);
  if (r != FA_OK) return r;
  if ((r = fa::check_ptrs({Q, K, V, O, LSE})) != FA_OK) return r;
  if (causal != 0 && causal != 1) return FA_ERR_INVALID_ARG;
  const fa::Mask m{mask, mask_stride_b, mask_stride_h, mask_stride_row};
  if ((r = fa::check_mask(m, s, dtype)) != FA_OK) return r;
  int* status = fa::device_status_ptr();
  if (!status) return FA_ERR_CUDA;
  return fa::from_cuda(fa::tc_fwd_masked(Q, K, V, O, LSE, s, scale, causal == 1, mask, m.sb, m.sh, m.srow, status,
                                         static_cast<cudaStream_t>(stream)));
}

extern "C" fa_status_t fa_bwd_masked(const void* Q, const void* K, const void* V, const void* O,
                                     const void* dO, const float* LSE, const float* D, void* dQ, void* dK,
                                     void* dV, const void* mask, long long mask_stride_b,
                                     long long mask_stride_h, long long mask_stride_row, void* workspace,
                                     size_t workspace_bytes, int B, int H, int N, int d, float scale, int causal,
                                     int dtype, void* stream) {
  const fa::Mask m{mask, mask_stride_b, mask_stride_h, mask_stride_row};
  return fa::bwd_common(Q, K, V, O, dO, LSE, D, dQ, dK, dV, workspace, workspace_bytes, B, H, N, d, scale, causal,
                        dtype, &m, nullptr, stream);
}

extern "C" fa_status_t fa_fwd_bitmask(const void* Q, const void* K, const void* V, void* O, float* LSE,
                                      const void* bits, long long bits_stride_b, long long bits_stride_h,
                                      long long bits_stride_row, int B, int H, int N, int d, float scale,
                                      int causal, int dtype, void* stream) {
  const Shape s{B, H, N, d};
  fa_status_t r = fa::check_shape(s, dtype, &scale);
  if (r != FA_OK) return r;
  if ((r = fa::check_ptrs({Q, K, V, O, LSE})) != FA_OK) return r;
  if (causal != 0 && causal != 1) return FA_ERR_INVALID_ARG;
  const fa::Mask m{bits, bits_stride_b, bits_stride_h, bits_stride_row};
  if ((r = fa::check_bits(m, s, dtype)) != FA_OK) return r;
  int* status = fa::device_status_ptr();
  if (!status) return FA_ERR_CUDA;
  return fa::from_cuda(fa::tc_fwd_bitmask(Q, K, V, O, LSE, s, scale, causal == 1, static_cast<const uint32_t*>(bits),
                                          m.sb, m.sh, m.srow, status, static_cast<cudaStream_t>(stream)));
}

extern "C" fa_status_t fa_bwd_bitmask(const void* Q, const void* K, const void* V, const void* O,
                                      const void* dO, const float* LSE, const float* D, void* dQ, void* dK,
                                      void* dV, const void* bits, long long bits_stride_b,
                                      long long bits_stride_h, long long bits_stride_row, void* workspace,
                                      size_t workspace_bytes, int B, int H, int N, int d, float scale, int causal,
                                      int dtype, void* stream) {
  const fa::Mask m{bits, bits_stride_b, bits_stride_h, bits_stride_row};
  return fa::bwd_common(Q, K, V, O, dO, LSE, D, dQ, dK, dV, workspace, workspace_bytes, B, H, N, d, scale, causal,
                        dtype, nullptr, nullptr, stream, &m);
}

extern "C" fa_status_t fa_fwd_dropout(const void* Q, const void* K, const void* V, void* O, float* LSE, int B,
                                      int H, int N, int d, float scale, int causal, float p_drop,
                                      unsigned long long seed, int dtype, void* stream) {
  const Shape s{B, H, N, d};
  fa_status_t r = fa::check_shape(s, dtype, &scale);
  if (r != FA_OK) return r;
  if ((r = fa::check_ptrs({Q, K, V, O, LSE})) != FA_OK) return r;
  if (causal != 0 && causal != 1) return FA_ERR_INVALID_ARG;
  uint32_t t = 0;
  if ((r = fa::drop_threshold(p_drop, dtype, &t)) != FA_OK) return r;
  int* status = fa::device_status_ptr();
  if (!status) return FA_ERR_CUDA;
  return fa::from_cuda(fa::tc_fwd_dropout(Q, K, V, O, LSE, s, scale, causal == 1, (uint64_t)seed, t, status,
                                          static_cast<cudaStream_t>(stream)));
}

extern "C" fa_status_t fa_bwd_dropout(const void* Q, const void* K, const void* V, const void* O,
                                      const void* dO, const float* LSE, const float* D, void* dQ, void* dK,
                                      void* dV, void* workspace, size_t workspace_bytes, int B, int H, int N, int d,
                                      float scale, int causal, float p_drop, unsigned long long seed, int dtype,
                                      void* stream) {
  fa::Drop dr{(uint64_t)seed, 0};
  const fa_status_t r = fa::drop_threshold(p_drop, dtype, &dr.t);
  if (r != FA_OK) return r;
  return fa::bwd_common(Q, K, V, O, dO, LSE, D, dQ, dK, dV, workspace, workspace_bytes, B, H, N, d, scale, causal,
                        dtype, nullptr, &dr, stream);
}

namespace {
fa_status_t check_splitkv(int B, int H, int Nq, int Nk, int d, float scale, int causal, int dtype) {
  if (B < 1 || H < 1 || Nq < 1 || Nk < 1 || d < 1) return FA_ERR_INVALID_ARG;
  if (dtype != FA_DTYPE_BF16 && dtype != FA_DTYPE_FP32) return FA_ERR_INVALID_ARG;
  if (!(isfinite(scale) && scale > 0.f)) return FA_ERR_INVALID_ARG;
  if (causal != 0 && causal != 1) return FA_ERR_INVALID_ARG;
  if ((int64_t)B * H >= (int64_t(1) << 31) || (int64_t)B * H * Nk > (int64_t(1) << 50)) return FA_ERR_INVALID_ARG;
  if (causal && Nq > Nk) return FA_ERR_INVALID_ARG;
  if (dtype != FA_DTYPE_BF16 || (d != 64 && d != 128) || Nq > 64) return FA_ERR_UNSUPPORTED;
  return FA_OK;
}
}  // namespace

extern "C" size_t fa_fwd_splitkv_workspace_size(int B, int H, int Nq, int Nk, int d, int dtype) {
  if (check_splitkv(B, H, Nq, Nk, d, 1.f, 0, dtype) != FA_OK) return 0;
  return fa::splitkv_workspace_floats((int64_t)B * H, Nq, Nk, d) * sizeof(float);
}

extern "C" fa_status_t fa_fwd_splitkv(const void* Q, const void* K, const void* V, void* O, float* LSE,
                                      int B, int H, int Nq, int Nk, int d, float scale, int causal,
                                      int dtype, void* workspace, size_t workspace_bytes, void* stream) {
  fa_status_t r = check_splitkv(B, H, Nq, Nk, d, scale, causal, dtype);
  if (r != FA_OK) return r;
  if ((r = fa::check_ptrs({Q, K, V, O, LSE})) != FA_OK) return r;
  const size_t need = fa_fwd_splitkv_workspace_size(B, H, Nq, Nk, d, dtype);
  if (!workspace || workspace_bytes < need) return FA_ERR_WORKSPACE;
  if (!fa::aligned16(workspace)) return FA_ERR_INVALID_ARG;
  int* status = fa::device_status_ptr();
  if (!status) return FA_ERR_CUDA;
  return fa::from_cuda(fa::splitkv_fwd(Q, K, V, O, LSE, (int64_t)B * H, Nq, Nk, d, scale, causal == 1,
                                       static_cast<float*>(workspace), status, static_cast<cudaStream_t>(stream)));
}

extern "C" const char* fa_get_error_string(fa_status_t status) {
  switch (status) {
    case FA_OK: return "FA_OK";
    case FA_ERR_INVALID_ARG: return "FA_ERR_INVALID_ARG: null/misaligned pointer or bad size, scale or flag";
    case FA_ERR_UNSUPPORTED: return "FA_ERR_UNSUPPORTED: valid arguments outside what is implemented (d, N, dtype)";
    case FA_ERR_CUDA: return "FA_ERR_CUDA: a CUDA call or kernel launch failed";
    case FA_ERR_DEVICE_TIMEOUT: return "FA_ERR_DEVICE_TIMEOUT: a bounded device-side wait gave up";
    case FA_ERR_WORKSPACE: return "FA_ERR_WORKSPACE: workspace missing or smaller than fa_bwd_workspace_size()";
  }
  return "unknown fa_status_t";
}

extern "C" fa_status_t fa_get_last_device_status(void) {
  int* p = fa::device_status_ptr();
  if (!p) return FA_ERR_CUDA;
  int v = 0;
  if (cudaMemcpy(&v, p, sizeof(int), cudaMemcpyDeviceToHost) != cudaSuccess) return FA_ERR_CUDA;
  if (v != 0) {
    const int zero = 0;
    if (cudaMemcpy(p, &zero, sizeof(int), cudaMemcpyHostToDevice) != cudaSuccess) return FA_ERR_CUDA;
  }
  return v == 0 ? FA_OK : static_cast<fa_status_t>(v);
}

extern "C" fa_status_t fa_set_bwd_dq_mode(int mode) {
  if (mode != FA_BWD_DQ_AUTO && mode != FA_BWD_DQ_ATOMIC && mode != FA_BWD_DQ_SEPARATE) return FA_ERR_INVALID_ARG;
  fa::set_bwd_dq_mode(mode);
  return FA_OK;
}

extern "C" int fa_get_bwd_dq_mode(void) { return fa::bwd_dq_mode(); }

extern "C" fa_status_t fa_test_inject_timeout(int which, unsigned long long wait_limit_ns) {
  if (which != 0 && which != fa::ptx::kInjectFwd && which != fa::ptx::kInjectBwd) return FA_ERR_INVALID_ARG;
  int* p = fa::device_status_ptr();
  if (!p) return FA_ERR_CUDA;
  fa::ptx::StatusBlock* b = reinterpret_cast<fa::ptx::StatusBlock*>(p);
  if (cudaMemcpy(&b->inject, &which, sizeof(int), cudaMemcpyHostToDevice) != cudaSuccess ||
      cudaMemcpy(&b->limit_ns, &wait_limit_ns, sizeof(unsigned long long), cudaMemcpyHostToDevice) != cudaSuccess)
    return FA_ERR_CUDA;
  return FA_OK;
}
