/*
 * fa.h — C ABI of the exact-attention library (GB300, sm_103a).
 *
 * Exact scaled-dot-product attention over contiguous [B, H, N, d] tensors, with no
 * N x N matrix in device memory: the forward pass keeps O and one float per query
 * row (LSE); the backward pass rebuilds the attention weights from LSE.
 *
 * Sources (web pages, by title and section):
 *   "flash-attention-backpropagation" (aiqz.cc): 前向台账 (row max m, row sum l),
 *       反向总览 (P rebuilt from the forward's statistics), Softmax梯度 (D, dP, dS),
 *       QKV梯度 (dV, dQ, dK accumulated block by block).
 *   "flash-attention-v2-sram-tiling" (aiqz.cc): §1 (Attention = softmax(QK^T/sqrt d)V),
 *       §4 (tiling), §5 (online softmax), §6 (recompute and fusion), §7 (scale folding,
 *       row-parallel work split).
 *   "知识点13 FlashAttention深度攻略" (blog.xiaohack.org): 代码手撕 (causal mask j > i).
 *
 * Conventions shared by every entry point
 *   Layout   Q, K, V, O, dO, dQ, dK, dV: contiguous row-major [B, H, N, d]; all share
 *            one element type (dtype). LSE and D: contiguous float32 [B, H, N].
 *   dtype    FA_DTYPE_BF16 (tensor-core path) or FA_DTYPE_FP32 (exact FFMA path).
 *   Shapes   B, H, N >= 1 (any N: partial last tiles are handled); d in {64, 128}.
 *            bf16: B*H*N < 2^31. fp32: N <= 4096. B*H < 2^31.
 *   scale    finite and > 0; scores are s_ij = scale * q_i . k_j (1/sqrt(d) on the pages).
 *   causal   0: every key is visible. 1: key j is hidden from query i when j > i.
 *   Pointers device pointers (cudaMalloc or torch), 16-byte aligned, non-overlapping
 *            between inputs and outputs. The caller owns every buffer and the stream.
 *   stream   a cudaStream_t passed as void* (NULL = legacy default stream). Every call
 *            only enqueues work on it and returns; nothing synchronises.
 *   Errors   Arguments are checked on the host before anything is launched: a bad
 *            argument returns FA_ERR_INVALID_ARG or FA_ERR_UNSUPPORTED and touches no
 *            buffer. A failed launch returns FA_ERR_CUDA. A device-side wait that runs
 *            out of time records FA_ERR_DEVICE_TIMEOUT in a device status word, which
 *            fa_get_last_device_status() reads after the caller synchronises.
 */
#ifndef FA_GB300_H
#define FA_GB300_H

#include <stddef.h>

#if defined(__GNUC__)
#define FA_API __attribute__((visibility("default")))
#else
#define FA_API
#endif

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
  FA_OK = 0,
  FA_ERR_INVALID_ARG = 1,    /* null pointer, bad size/scale/alignment */
  FA_ERR_UNSUPPORTED = 2,    /* valid but not implemented (d, N, dtype combination) */
  FA_ERR_CUDA = 3,           /* a CUDA runtime/driver call failed */
  FA_ERR_DEVICE_TIMEOUT = 4, /* a bounded device-side wait gave up */
  FA_ERR_WORKSPACE = 5       /* workspace missing or too small */
} fa_status_t;

typedef enum { FA_DTYPE_BF16 = 0, FA_DTYPE_FP32 = 1 } fa_dtype_t;

/*
 * fa_fwd — attention forward.
 *   O_i   = sum_j P_ij V_j,  P_ij = exp(s_ij - m_i) / l_i over the visible keys j,
 *   LSE_i = m_i + ln(l_i),   m_i = max_j s_ij,  l_i = sum_j exp(s_ij - m_i).
 * ("flash-attention-v2-sram-tiling" §1, §4, §5; "flash-attention-backpropagation" 前向台账.)
 * In:  Q, K, V [B,H,N,d] dtype.   Out: O [B,H,N,d] dtype, LSE [B,H,N] float32.
 * LSE is natural-log, in units of the scaled scores; it replaces the pages' (m, l) pair.
 */
FA_API fa_status_t fa_fwd(const void* Q, const void* K, const void* V, void* O, float* LSE,
                   int B, int H, int N, int d, float scale, int causal, int dtype,
                   void* stream);

/*
 * fa_bwd_preprocess — D_i = sum_c dO_ic * O_ic ("flash-attention-backpropagation",
 * Softmax梯度). In: O, dO [B,H,N,d] dtype. Out: D [B,H,N] float32.
 */
FA_API fa_status_t fa_bwd_preprocess(const void* O, const void* dO, float* D,
                              int B, int H, int N, int d, int dtype, void* stream);

/*
 * fa_bwd_workspace_size — bytes of device workspace fa_bwd needs for these sizes
 * (the float32 dQ accumulator of the bf16 path; 0 for fp32). Returns 0 for
 * arguments fa_bwd would reject.
 */
FA_API size_t fa_bwd_workspace_size(int B, int H, int N, int d, int dtype);

/*
 * fa_bwd — attention backward from the forward's O and LSE.
 *   P_ij  = exp(s_ij - LSE_i)          (P rebuilt, 反向总览 / 数值稳定)
 *   dV_j  = sum_i P_ij dO_i            (QKV梯度)
 *   dP_ij = dO_i . V_j,  dS_ij = P_ij (dP_ij - D_i)     (Softmax梯度)
 *   dQ_i  = scale sum_j dS_ij K_j,  dK_j = scale sum_i dS_ij Q_i   (QKV梯度)
 * In:  Q, K, V, O, dO [B,H,N,d] dtype; LSE [B,H,N] float32 from fa_fwd; D [B,H,N]
 *      float32 from fa_bwd_preprocess, or NULL, in which case fa_bwd computes it
 *      first into the workspace (the size query then includes room for it).
 * Out: dQ, dK, dV [B,H,N,d] dtype (overwritten).
 * workspace: device buffer of at least fa_bwd_workspace_size(...) bytes (plus
 *      4*B*H*N bytes when D is NULL); its contents on entry do not matter.
 */
FA_API fa_status_t fa_bwd(const void* Q, const void* K, const void* V, const void* O,
                   const void* dO, const float* LSE, const float* D,
                   void* dQ, void* dK, void* dV, void* workspace, size_t workspace_bytes,
                   int B, int H, int N, int d, float scale, int causal, int dtype,
                   void* stream);

/*
 * fa_set_bwd_dq_mode / fa_get_bwd_dq_mode — how the bf16 backward without mask or dropout
 * (fa_bwd, fa_bwd_rect, fa_bwd_noalloc) computes dQ, the one gradient that sums over key
 * tiles ("FlashAttention 反向传播" 踩坑二: one recompute per tile for all three gradients, or
 * a second pass for dQ; "flash-attention-v2-sram-tiling" §7 counts the cost of split
 * sums). Both modes keep fp32 sums and round to bf16 once (踩坑三); they agree to bf16
 * rounding, not bit for bit.
 *   FA_BWD_DQ_ATOMIC   (1): each 128-key tile adds its fp32 dQ partials into the workspace
 *                           with atomic additions, then one pass scales and rounds them.
 *   FA_BWD_DQ_SEPARATE (2): dK and dV from the key-tile kernel alone, then a kernel over
 *                           128-query tiles recomputes S and dP and accumulates dQ on chip;
 *                           dQ does not depend on the order of any additions.
 *   FA_BWD_DQ_AUTO     (0, the default): the atomic mode, the faster of the two at every
 *                           shape measured on GB300 (the separate pass costs 16-28% more).
 * The setting is process-wide and applies to calls made after it; masked and dropout
 * backward calls always use the atomic mode. fa_set_bwd_dq_mode returns
 * FA_ERR_INVALID_ARG for any other value; fa_get_bwd_dq_mode returns the setting.
 */
typedef enum { FA_BWD_DQ_AUTO = 0, FA_BWD_DQ_ATOMIC = 1, FA_BWD_DQ_SEPARATE = 2 } fa_bwd_dq_mode_t;
FA_API fa_status_t fa_set_bwd_dq_mode(int mode);
FA_API int fa_get_bwd_dq_mode(void);

/*
 * fa_fwd_rect / fa_bwd_rect — fa_fwd / fa_bwd with Nq query rows against Nk key/value rows
 * per head (cross-attention, or a prefill of Nq new tokens that continues a cached prefix
 * of Nk - Nq tokens: "flash-attention-v2-sram-tiling" 场景二 serves long documents against
 * a key/value cache; "知识点13 FlashAttention深度攻略" 代码手撕 tiles the query and key ranges
 * separately, with min() tails). fa_fwd and fa_bwd are the case Nq = Nk.
 * causal: the queries are the last Nq positions of the sequence (bottom-right alignment):
 *      query i hides keys j > i + Nk - Nq. With Nq = Nk this is the rule of fa_fwd. With
 *      Nq > Nk the first Nq - Nk queries see no key: they get O = 0 and LSE = -inf, their
 *      dQ rows are 0 and they add nothing to dK or dV.
 * In:  Q, dO [B,H,Nq,d]; K, V [B,H,Nk,d] (dtype); LSE, D [B,H,Nq] float32 (D from
 *      fa_bwd_preprocess on O, dO with N = Nq, or NULL as for fa_bwd).
 * Out: O, dQ [B,H,Nq,d]; dK, dV [B,H,Nk,d] (dtype); LSE [B,H,Nq] float32.
 * Shapes: Nq, Nk >= 1; the limits of fa_fwd apply to the longer of the two (bf16:
 *      B*H*max(Nq, Nk) < 2^31; fp32: max(Nq, Nk) <= 4096).
 * workspace: at least fa_bwd_rect_workspace_size(...) bytes (the float32 dQ accumulator,
 *      4*B*H*Nq*d bytes for bf16), plus 4*B*H*Nq bytes when D is NULL. The remaining
 *      arguments and errors are those of fa_fwd and fa_bwd.
 */
FA_API fa_status_t fa_fwd_rect(const void* Q, const void* K, const void* V, void* O, float* LSE,
                               int B, int H, int Nq, int Nk, int d, float scale, int causal, int dtype,
                               void* stream);
FA_API size_t fa_bwd_rect_workspace_size(int B, int H, int Nq, int Nk, int d, int dtype);
FA_API fa_status_t fa_bwd_rect(const void* Q, const void* K, const void* V, const void* O,
                               const void* dO, const float* LSE, const float* D,
                               void* dQ, void* dK, void* dV, void* workspace, size_t workspace_bytes,
                               int B, int H, int Nq, int Nk, int d, float scale, int causal, int dtype,
                               void* stream);

/*
 * fa_bwd_noalloc — fa_bwd for callers that must not allocate device memory.
 * The pages have no counterpart: this is a packaging of fa_bwd, not a step of the method.
 * Some callers cannot call cudaMalloc: code hosted by a framework that owns all device
 * memory through a fixed, pre-planned pool (serving engines, plugin hosts) may not
 * allocate outside it, and latency-critical paths cannot take the implicit device
 * synchronisation cudaMalloc/cudaFree may bring. This entry point takes no workspace: its
 * scratch (the fp32 dQ accumulator, and D when D is NULL) is a static device array inside
 * the library, FA_NOALLOC_MAX_ELEMS floats plus FA_NOALLOC_MAX_ELEMS/64 floats (32.5 MiB),
 * held by every GPU that loads the library until the process exits. It allocates nothing.
 * Arguments and results are those of fa_bwd (without workspace / workspace_bytes).
 * Limits: B*H*N*d <= FA_NOALLOC_MAX_ELEMS, else FA_ERR_WORKSPACE and nothing runs.
 * First call on a device: looks up the array's device address (cudaGetSymbolAddress) with
 * that device current and caches it for the device's current context (a first call in a
 * new context, e.g. after cudaDeviceReset, looks it up again); make that first call before
 * any stream capture.
 * Sharing: all calls use the same array. Each call clears the accumulator before use, so
 * leftovers of earlier calls do not leak into results, but calls that overlap on the GPU
 * (concurrent streams or threads) race on the array and must be serialised by the caller.
 */
#define FA_NOALLOC_MAX_ELEMS (8u * 1024u * 1024u)
FA_API fa_status_t fa_bwd_noalloc(const void* Q, const void* K, const void* V, const void* O,
                           const void* dO, const float* LSE, const float* D,
                           void* dQ, void* dK, void* dV,
                           int B, int H, int N, int d, float scale, int causal, int dtype,
                           void* stream);

/*
 * fa_fwd_splitkv — forward for a few queries against a long key/value sequence (a
 * decoding step against a cache): same outputs as fa_fwd, with N_q query rows and N_k
 * key/value rows per head. The keys are split into chunks handled in parallel, each
 * keeping the online-softmax state (m, l, un-normalised O) of "flash-attention-v2-sram-
 * tiling" §5; the chunk states are merged with the rule of "知识点13" §4
 * (m = max m_s, l = sum l_s e^(m_s - m), O = sum O_s e^(m_s - m) / l).
 * In:  Q [B,H,N_q,d], K and V [B,H,N_k,d] bf16.  Out: O [B,H,N_q,d] bf16, LSE [B,H,N_q] fp32.
 * causal: the queries are the last N_q positions (requires N_q <= N_k): query i hides
 *      keys j > i + N_k - N_q. causal = 0: every key is visible.
 * Supported: bf16; d = 64 or 128 with 1 <= N_q <= 64 (else
 *      FA_ERR_UNSUPPORTED); any N_k >= 1. Both products of each 128-key tile run on the
 *      tensor cores.
 * workspace: device buffer of at least fa_fwd_splitkv_workspace_size(...) bytes (fp32
 *      chunk states); its contents on entry do not matter.
 */
FA_API size_t fa_fwd_splitkv_workspace_size(int B, int H, int Nq, int Nk, int d, int dtype);
FA_API fa_status_t fa_fwd_splitkv(const void* Q, const void* K, const void* V, void* O, float* LSE,
                           int B, int H, int Nq, int Nk, int d, float scale, int causal, int dtype,
                           void* workspace, size_t workspace_bytes, void* stream);

/*
 * fa_fwd_masked / fa_bwd_masked — fa_fwd / fa_bwd with an additive mask M added to the
 * scaled scores ("知识点13 FlashAttention深度攻略" §7 算子融合优化: the mask is applied inside
 * the fused softmax step):
 *      s_ij = scale * q_i . k_j + M_ij,   then the causal rule (if causal) as for fa_fwd.
 * mask: bf16 (dtype must be FA_DTYPE_BF16, else FA_ERR_UNSUPPORTED), device pointer,
 *      16-byte aligned. Element M(b, h, i, j) is read at
 *      mask[b * mask_stride_b + h * mask_stride_h + i * mask_stride_row + j]
 *      (strides in elements; 0 broadcasts over batch or heads). Every stride must be a
 *      non-negative multiple of 8 and mask_stride_row >= N rounded up to 8 (rows are read
 *      in 16-byte pieces; the padding is never used). The caller owns the mask; it is read
 *      by both calls and never written. Entries are finite or -inf (-inf hides the key).
 * A query whose every key is hidden has no softmax: it gets O = 0 and LSE = -inf, and it
 *      contributes nothing to dK or dV (its dQ row is 0).
 * The remaining arguments, layouts, workspace and errors are those of fa_fwd and fa_bwd;
 *      pass the same mask, scale and causal flag to both.
 */
FA_API fa_status_t fa_fwd_masked(const void* Q, const void* K, const void* V, void* O, float* LSE,
                                 const void* mask, long long mask_stride_b, long long mask_stride_h,
                                 long long mask_stride_row, int B, int H, int N, int d, float scale,
                                 int causal, int dtype, void* stream);
FA_API fa_status_t fa_bwd_masked(const void* Q, const void* K, const void* V, const void* O,
                                 const void* dO, const float* LSE, const float* D, void* dQ, void* dK,
                                 void* dV, const void* mask, long long mask_stride_b,
                                 long long mask_stride_h, long long mask_stride_row, void* workspace,
                                 size_t workspace_bytes, int B, int H, int N, int d, float scale,
                                 int causal, int dtype, void* stream);

/*
 * fa_fwd_bitmask / fa_bwd_bitmask — fa_fwd_masked / fa_bwd_masked for a boolean mask, whose
 * entries are 0 (the key is visible) or -inf (hidden), stored one bit per key: the same
 * result as the additive mask with those entries, at 1/16 of its bytes.
 * bits: 32-bit words (dtype must be FA_DTYPE_BF16, else FA_ERR_UNSUPPORTED), device
 *      pointer, 16-byte aligned. Query i of head (b, h) sees key j iff bit (j % 32) of word
 *      bits[b * bits_stride_b + h * bits_stride_h + i * bits_stride_row + j / 32]
 *      is 1 (and, when causal, j <= i). Strides are in words, 0 broadcasts over batch or
 *      heads; every stride must be a non-negative multiple of 4, and bits_stride_row at
 *      least 4 * ceil(N / 128): each 128-key tile of a row is read as one 16-byte piece.
 *      Bits of keys j >= N are never used. The caller owns the words; both calls read
 *      them and never write them; pass the same words, scale and causal flag to both.
 * A query with no visible key gets O = 0 and LSE = -inf, as with fa_fwd_masked.
 * The remaining arguments, layouts, workspace and errors are those of fa_fwd_masked and
 *      fa_bwd_masked.
 */
FA_API fa_status_t fa_fwd_bitmask(const void* Q, const void* K, const void* V, void* O, float* LSE,
                                  const void* bits, long long bits_stride_b, long long bits_stride_h,
                                  long long bits_stride_row, int B, int H, int N, int d, float scale,
                                  int causal, int dtype, void* stream);
FA_API fa_status_t fa_bwd_bitmask(const void* Q, const void* K, const void* V, const void* O,
                                  const void* dO, const float* LSE, const float* D, void* dQ, void* dK,
                                  void* dV, const void* bits, long long bits_stride_b,
                                  long long bits_stride_h, long long bits_stride_row, void* workspace,
                                  size_t workspace_bytes, int B, int H, int N, int d, float scale,
                                  int causal, int dtype, void* stream);

/*
 * fa_fwd_dropout / fa_bwd_dropout — fa_fwd / fa_bwd with dropout on the attention weights
 * ("知识点13 FlashAttention深度攻略" §7 算子融合优化: dropout is fused into the softmax step):
 *      O = (P o K c) V,  P = softmax of the scores, K the 0/1 keep matrix, c its scale.
 * LSE is the undropped softmax's. The backward is the exact gradient of that O for the
 *      same K: pass the same p_drop and seed to both calls (and D from the dropped O).
 * Keep bits: Philox-4x32-10 (Salmon et al., "Parallel random numbers: as easy as 1, 2, 3",
 *      SC 2011). Element (query i, key j) of head h = b*H + head takes byte j % 4 of word
 *      (j % 16) / 4 of Philox(counter (j / 16, i, h, 0), key (seed & 0xffffffff,
 *      seed >> 32)); the key is kept iff that byte >= t = min(255, round(p_drop * 256)),
 *      and c = 256 / (256 - t): the probability is quantised to a multiple of 2^-8 and
 *      every weight keeps its expected value exactly.
 * p_drop: finite, 0 <= p_drop < 1 (else FA_ERR_INVALID_ARG); dtype must be FA_DTYPE_BF16
 *      (else FA_ERR_UNSUPPORTED). The remaining arguments are those of fa_fwd / fa_bwd.
 */
FA_API fa_status_t fa_fwd_dropout(const void* Q, const void* K, const void* V, void* O, float* LSE, int B,
                                  int H, int N, int d, float scale, int causal, float p_drop,
                                  unsigned long long seed, int dtype, void* stream);
FA_API fa_status_t fa_bwd_dropout(const void* Q, const void* K, const void* V, const void* O,
                                  const void* dO, const float* LSE, const float* D, void* dQ, void* dK,
                                  void* dV, void* workspace, size_t workspace_bytes, int B, int H, int N,
                                  int d, float scale, int causal, float p_drop, unsigned long long seed,
                                  int dtype, void* stream);

/*
 * fa_fwd_fp8 — the forward of fa_fwd on 8-bit inputs ("flash-attention" (data.6616ai.com),
 * 参考答案: FlashAttention-3 runs on FP8; "知识点13" 前沿研究方向: mixed precision with FP8).
 * In:  Q, K, V [B,H,N,d] as e4m3 bytes (OCP FP8 E4M3: 1 sign, 4 exponent bits with bias 7,
 *      3 mantissa bits, subnormals, no infinities, S.1111.111 = NaN), each with one
 *      dequantisation factor: the value of element x is q_descale * e4m3(x) (k_descale,
 *      v_descale likewise).
 * Out: O [B,H,N,d] bf16 and LSE [B,H,N] fp32, for the scores s_ij = scale * q_i . k_j of the
 *      dequantised values: exactly what fa_fwd returns for those values, except that the
 *      attention weights are rounded to e4m3 before they multiply V (scores, running
 *      statistics, LSE and the accumulation of O stay fp32). For every weight >= 2^-10 of
 *      its row's largest the rounding error is <= 2^-4 of the weight; smaller weights may
 *      lose up to their whole value.
 * Supported: d = 128 (else FA_ERR_UNSUPPORTED); any N >= 1; causal 0 or 1 as for fa_fwd.
 * q_descale, k_descale, v_descale, scale: finite and > 0, else FA_ERR_INVALID_ARG.
 */
FA_API fa_status_t fa_fwd_fp8(const void* Q, const void* K, const void* V, void* O, float* LSE,
                              int B, int H, int N, int d, float scale, int causal, float q_descale,
                              float k_descale, float v_descale, void* stream);

/*
 * fa_fwd_bwd_host — forward and backward of tensors that live in host memory: the
 * copies to and from the device overlap the kernels. The heads (independent of one
 * another) are cut into contiguous groups: `chunks` equal ones (at most 16 and at most
 * B*H), or with chunks = 0 five groups in the ratio 1:2:2:2:1 when B*H >= 8 (the first
 * group's copy-in and the last one's copy-out overlap no kernel, so they are the small
 * ones) and up to 4 equal groups otherwise;
 * each group is copied in (Q, K, V, dO), run through fa_fwd, fa_bwd_preprocess and fa_bwd,
 * and copied out (O, LSE, dQ, dK, dV) on three internal streams, with three device slots
 * in `workspace` in rotation, so one group's copies run while another's kernels do.
 * In:  Q, K, V, dO host [B,H,N,d] bf16 (page-locked memory, e.g. cudaHostAlloc, lets
 *      the copies run asynchronously; pageable memory works but serialises them).
 * Out: O host [B,H,N,d] bf16, LSE host [B,H,N] fp32, dQ, dK, dV host [B,H,N,d] bf16.
 * workspace: device buffer of at least fa_fwd_bwd_host_workspace_size(...) bytes,
 *      256-byte aligned; its contents on entry do not matter.
 * stream: the work starts after what is already queued on `stream`, and `stream` waits
 *      for all of it: the outputs are in host memory once `stream` has been synchronised.
 *      The call itself does not block.
 * Supported: bf16, d in {64, 128}, causal 0/1, B*H*N < 2^31 (else FA_ERR_UNSUPPORTED).
 * Errors: as for fa_fwd / fa_bwd. A failure returned after some work was enqueued leaves
 *      that work running, but `stream` still waits for all of it: synchronise `stream`
 *      before freeing or reusing the buffers.
 */
FA_API size_t fa_fwd_bwd_host_workspace_size(int B, int H, int N, int d, int dtype, int chunks);
FA_API fa_status_t fa_fwd_bwd_host(const void* Q, const void* K, const void* V, const void* dO, void* O,
                                   float* LSE, void* dQ, void* dK, void* dV, void* workspace,
                                   size_t workspace_bytes, int B, int H, int N, int d, float scale,
                                   int causal, int dtype, int chunks, void* stream);

/* Text for a status code (static storage; never NULL). */
FA_API const char* fa_get_error_string(fa_status_t status);

/*
 * fa_get_last_device_status — reads and clears the device status word of the
 * current device. Call it after synchronising the streams the library ran on.
 * Returns FA_OK, FA_ERR_DEVICE_TIMEOUT, or FA_ERR_CUDA if the read itself failed.
 */
FA_API fa_status_t fa_get_last_device_status(void);

/*
 * fa_test_inject_timeout — for tests of the failure path only; not part of the method (the
 * pages have no counterpart). Every device-side wait of the tensor-core kernels is bounded
 * (4 s by default); when a wait gives up, the kernel records FA_ERR_DEVICE_TIMEOUT in the
 * device status word, stops its other roles, waits (bounded) for its own copies and
 * products in flight, releases its tensor memory and returns. This call lets a test
 * exercise that path on the current device without faulting or hanging the GPU:
 *   which = 1: in the next fa_fwd (bf16) launches, the first CTA never arms its first K
 *              tile, so the MMA thread's wait for it runs out;
 *   which = 2: the same for the first Q/dO tile of fa_bwd (bf16);
 *   which = 0: off (the normal state).
 * wait_limit_ns: the wait limit in force while set (0 restores the default of 4 s).
 * The call synchronises with the device (it writes device memory with cudaMemcpy). Results
 * of calls made while an injection is on are undefined; turn it off before any other use.
 * Returns FA_ERR_INVALID_ARG for another `which`, FA_ERR_CUDA if the write fails.
 */
FA_API fa_status_t fa_test_inject_timeout(int which, unsigned long long wait_limit_ns);

#ifdef __cplusplus
}
#endif
#endif /* FA_GB300_H */
