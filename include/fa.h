/*
 * fa.h -- C ABI of the GB300 (sm_103a) stabilised BF16 FlashAttention library.
 *
 * The library computes softmax attention O = softmax(scale * Q K^T) V and its
 * gradients with hand-written tcgen05/TMA kernels.  It follows these pages:
 *
 *   [ijyty]  ijyty.com/news/896914 (BF16 FlashAttention numerical stability):
 *            §2.1 tiled online softmax -- running row max m, running sum l,
 *            O rescaled by exp(m_prev - m), P~ = exp(S - m), O += P~ V,
 *            final O = diag(l)^-1 O; §3.1 delta = rowsum(dO o O) in the
 *            backward; §4.1/§4.2 the stabilised safe softmax (a repeated row
 *            maximum moves the shift to beta*rm for rm > 0 or to 0 for rm < 0;
 *            beta in [1.1, 1.5], 1.25 recommended); §6.1 the fix carries over
 *            to FP8 with dynamic scaling factors; §7.1 the monitor
 *            (S == rowmax(S)).sum().
 *   [jsqmd]  "Flash Attention低精度训练稳定性优化实践" §3.2: QK^T accumulated in
 *            FP32, softmax in FP32, the product with V in BF16; §3.3 the
 *            running max / log-sum-exp bookkeeping.
 *   [cnnet]  "FlashAttention 训练时为什么会梯度爆炸？" §2: the backward recomputes
 *            the forward's probabilities from Q, K, V instead of storing them;
 *            §3.1 Attention(Q,K,V) = softmax(QK^T / sqrt(d_k)) V; §3.3 an
 *            overflow check on the backward's gradients.
 *   [web578] "為什么BF16的FlashAttention會把訓練「炸掉」？" mechanism 2: detect a
 *            repeated row maximum and shift so the exponent at the maximum is
 *            strictly below 1.
 *
 * Conventions shared by every entry point
 *   - Tensors q, k, v, o, dO, dq, dk, dv are BF16, contiguous [B, H, N, d]
 *     row-major (d fastest).  lse and delta are FP32 [B, H, N].  All are
 *     DEVICE pointers, 16-byte aligned, owned by the caller.
 *   - d must be 64 or 128; N >= 1; B, H >= 1; B*H*N < 2^31.
 *   - scale must be finite and > 0 (the pages advise choosing it by
 *     experiment rather than fixing 1/sqrt(d) [jsqmd §5], so it is explicit).
 *   - causal != 0 means query i sees keys j <= i (top-left aligned).
 *   - lse is the natural-log logsumexp of the scaled logits scale*q.k.
 *   - Calls are asynchronous on `stream` (a cudaStream_t; NULL = legacy
 *     default stream).  The return value reports argument and launch errors
 *     only; errors raised on the device (a bounded wait that timed out, a
 *     non-finite output) are read with fa_device_status() or
 *     fa_device_report_read().
 *   - The library allocates nothing per call.  It keeps one 64-byte status
 *     record per device (fa_device_report), allocated on first use.
 *     fa_bwd_noalloc uses a separate, static record of its own, read with
 *     fa_bwd_noalloc_status().
 */
#ifndef FA_H_
#define FA_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
  FA_OK = 0,
  FA_ERR_INVALID_ARG = 1,   /* null pointer, bad size, misaligned pointer, bad scale/beta */
  FA_ERR_UNSUPPORTED = 2,   /* valid but not implemented (e.g. d not in {64, 128}) */
  FA_ERR_CUDA = 3,          /* a CUDA runtime/driver call failed; see fa_last_error() */
  FA_ERR_TIMEOUT = 4,       /* (fa_device_status) a kernel's bounded wait ran out */
  FA_ERR_DEVICE_BOUNDS = 5, /* (fa_device_status) a device-side index or layout check fired */
  FA_WARN_NONFINITE = 6     /* (fa_device_status) an output (O, LSE, dQ, dK or dV) held NaN or Inf */
} fa_status;

/* Which output a non-finite count of fa_device_report belongs to. */
enum { FA_OUT_O = 0, FA_OUT_LSE = 1, FA_OUT_DQ = 2, FA_OUT_DK = 3, FA_OUT_DV = 4, FA_NUM_OUTPUTS = 5 };

/* Bits of fa_device_report.flags. */
enum { FA_DEVFLAG_TIMEOUT = 1, FA_DEVFLAG_BOUNDS = 2, FA_DEVFLAG_NONFINITE = 4 };

/*
 * What the kernels recorded on the device since the record was last read (the NaN monitor
 * of [ijyty §7.1] and [jsqmd §5], per output; the overflow check in the backward that
 * [cnnet §3.3] describes for CANN 8.0).
 *   flags        : FA_DEVFLAG_* bits
 *   bounds_site  : builds with FA_DEBUG_BOUNDS: the site id of the first failed index
 *                  check (0 = none); bounds_value: the index that check saw
 *   nonfinite[i] : how many entries of output i (FA_OUT_*) were written as NaN or Inf,
 *                  counted on the stored values (BF16 for O, dQ, dK, dV; FP32 for LSE)
 */
typedef struct {
  uint32_t flags;
  uint32_t bounds_site;
  int64_t bounds_value;
  uint64_t nonfinite[FA_NUM_OUTPUTS];
  uint64_t reserved;
} fa_device_report;

/* Shift branch codes written to fa_row_stats.row_branch. */
enum { FA_BRANCH_RM = 0, FA_BRANCH_BETA = 1, FA_BRANCH_ZERO = 2 };

/*
 * Optional per-row statistics of the forward ([ijyty §7.1] monitor; [jsqmd §5]
 * "watch the max/min of the softmax input").  Each pointer is a device array
 * of B*H*N entries or NULL (not written).
 *   row_max_raw : rm, the largest visible raw score q.k (before scale)
 *   row_ties    : rs, how many visible keys reach rm exactly (FP32 equality), all modes
 *   row_branch  : which shift the stabilised rule chose (FA_BRANCH_*); 0 in plain mode
 *   row_ones    : how many visible BF16 P~ entries of the row were exactly 1.0
 *   row_min_raw : the smallest visible raw score of the row
 */
typedef struct {
  float* row_max_raw;
  int32_t* row_ties;
  int8_t* row_branch;
  int32_t* row_ones;
  float* row_min_raw;
} fa_row_stats;

/*
 * fa_fwd -- attention forward ([ijyty §2.1], [cnnet §3.1]).
 *   q, k, v : inputs, BF16 [B,H,N,d]
 *   o       : output, BF16 [B,H,N,d]
 *   lse     : output, FP32 [B,H,N]
 *   stable  : 0 = plain safe softmax (m = running row max);
 *             1 = stabilised shift [ijyty §4.1] with a running tie count over
 *                 all visible keys seen so far (m = beta*rm if rm > 0 and the
 *                 maximum repeats, 0 if rm < 0 and it repeats, else rm);
 *             2 = the block-local reading of [ijyty §4.2]: each block of 128
 *                 keys applies the same rule to its own max and tie count, and
 *                 the row keeps the largest shift seen so far (depends on the
 *                 block width; row_branch reports the block that set the shift);
 *   beta    : shift factor for stable = 1, 2; finite and >= 1 (ignored when stable = 0)
 *   stats   : optional per-row statistics (NULL = none)
 * Returns FA_OK, FA_ERR_INVALID_ARG, FA_ERR_UNSUPPORTED or FA_ERR_CUDA.
 */
int fa_fwd(const void* q, const void* k, const void* v, void* o, float* lse, int B, int H, int N, int d,
           int causal, float scale, int stable, float beta, const fa_row_stats* stats, void* stream);

/*
 * fa_quantize_fp8 -- dynamic per-tensor FP8 scaling ([ijyty §6.1]: the stabilised
 * shift carries over to FP8 when paired with dynamic scaling factors; the page gives no
 * formula, this is the usual amax rule).
 *   x        : input, BF16, n elements (any shape, contiguous), device, 16-byte aligned
 *   x8       : output, E4M3 codes (1 byte each), n elements, device, 16-byte aligned
 *   descale  : output, one FP32 on the device: amax(|x|) / 448 (1 if x is all zero)
 *   x8[i] = E4M3(x[i] / descale) -- FP32 division, round to nearest even, saturating at
 *   +-448 -- so x is represented by x8 * descale.  Four launches on `stream`; descale is
 *   used as the amax scratch until the last one.  NaN or Inf in x give a NaN or Inf descale.
 * Returns FA_OK, FA_ERR_INVALID_ARG or FA_ERR_CUDA.
 */
int fa_quantize_fp8(const void* x, size_t n, void* x8, float* descale, void* stream);

/*
 * fa_fwd_fp8 -- the forward of fa_fwd with E4M3 inputs ([ijyty §6.1], FP8 with dynamic
 * scaling).  Q K^T and P~ V run as E4M3 x E4M3 tensor-core products with FP32
 * accumulation; the softmax runs in FP32 as in fa_fwd.
 *   q8, k8, v8 : E4M3 codes, [B,H,N,d] contiguous, device, 16-byte aligned
 *   descale    : device FP32[3] = the per-tensor scales of Q, K, V (fa_quantize_fp8's
 *                outputs); the inputs are q8 * descale[0], k8 * descale[1], v8 * descale[2]
 *   o, lse     : as fa_fwd (O in BF16, lse of the dequantised scores)
 *   the raw scores, the row maximum, the tie count and the shift rule are those of the
 *   dequantised scores (q8 dq).(k8 dk); P~ is multiplied by 2^8 and rounded to E4M3 for the
 *   P~V product; stats->row_max_raw / row_min_raw are in dequantised units and
 *   stats->row_ones counts P~ entries whose E4M3 value is exactly 1.0 (2^8 after scaling).
 *   d must be 64 or 128 (FA_ERR_UNSUPPORTED otherwise).
 * Returns FA_OK, FA_ERR_INVALID_ARG, FA_ERR_UNSUPPORTED or FA_ERR_CUDA.
 */
int fa_fwd_fp8(const void* q8, const void* k8, const void* v8, const float* descale, void* o, float* lse,
               int B, int H, int N, int d, int causal, float scale, int stable, float beta,
               const fa_row_stats* stats, void* stream);

/*
 * fa_bwd_workspace_size -- bytes of device scratch fa_bwd needs: an FP32
 * [B,H,N,d] dQ accumulator, then lse*log2(e) and delta as FP32 [B,H,N_pad]
 * (N_pad = N rounded up to a multiple of 128; the padding holds lse = +inf
 * and delta = 0), each part rounded up to 256 bytes.  Returns 0 for invalid
 * sizes.
 */
size_t fa_bwd_workspace_size(int B, int H, int N, int d);

/*
 * fa_bwd -- attention backward by recomputation ([cnnet §2], [ijyty §3.1]).
 *   q, k, v, o, lse, dO : forward inputs/outputs and the output gradient
 *   dq, dk, dv          : outputs, BF16 [B,H,N,d]
 *   delta_out           : optional FP32 [B,H,N] copy of delta = rowsum(dO o O) (NULL = none)
 *   workspace           : caller-owned device scratch of at least
 *                         fa_bwd_workspace_size(B,H,N,d) bytes, 256-byte aligned;
 *                         its contents on entry do not matter
 * The backward uses only o and lse from the forward, so it is the same for
 * plain and stabilised forwards.
 * Returns FA_OK, FA_ERR_INVALID_ARG, FA_ERR_UNSUPPORTED or FA_ERR_CUDA.
 */
int fa_bwd(const void* q, const void* k, const void* v, const void* o, const float* lse, const void* dO,
           void* dq, void* dk, void* dv, float* delta_out, int B, int H, int N, int d, int causal,
           float scale, void* workspace, size_t workspace_bytes, void* stream);

/*
 * fa_bwd_staged -- the same computation as fa_bwd, split into its three
 * device stages so a caller can schedule or time them separately.  Same
 * arguments as fa_bwd plus `stages`, a bit mask:
 *   FA_BWD_PREPROCESS  delta = rowsum(dO o O) and zeroing of the FP32 dQ accumulator
 *   FA_BWD_MAIN        the recomputing kernel: dK, dV and the dQ accumulator
 *   FA_BWD_DQ_CONVERT  dq = bf16(scale * dQ accumulator)
 * The stages must run in this order on the same workspace (the accumulator
 * lives there between calls); fa_bwd(...) == fa_bwd_staged(..., FA_BWD_ALL).
 */
enum { FA_BWD_PREPROCESS = 1, FA_BWD_MAIN = 2, FA_BWD_DQ_CONVERT = 4, FA_BWD_ALL = 7 };

int fa_bwd_staged(const void* q, const void* k, const void* v, const void* o, const float* lse, const void* dO,
                  void* dq, void* dk, void* dv, float* delta_out, int B, int H, int N, int d, int causal,
                  float scale, void* workspace, size_t workspace_bytes, void* stream, int stages);

/*
 * fa_bwd_noalloc -- the backward of fa_bwd for callers that cannot allocate device
 * memory.  (The pages have no counterpart; this is a deployment variant.)
 *
 * Some callers cannot call cudaMalloc: a plugin or custom operator inside a host
 * application that owns the device-memory budget and forbids allocations outside
 * its pool, or a latency-critical path where cudaMalloc/cudaFree would
 * synchronise the device.  This entry point allocates nothing: the backward's
 * scratch (the FP32 dQ accumulator and delta) lives in a fixed file-scope device
 * array of FA_NOALLOC_SCRATCH_BYTES (32 MiB) that every GPU loading the library
 * holds until the process exits.  The caller still passes all inputs and outputs.
 *   - Arguments, layouts and results are those of fa_bwd without the workspace.
 *   - Problems whose scratch, fa_bwd_workspace_size(B,H,N,d), exceeds 32 MiB are
 *     rejected with FA_ERR_INVALID_ARG and a message (e.g. B*H*N*d up to about
 *     8M elements at d = 128).
 *   - The first call on a device looks up the array's device address
 *     (cudaGetSymbolAddress, with that device current); make that first call before
 *     any stream capture.
 *   - Every call on a device shares the one array and the library zeroes what must
 *     start at zero on each call; calls that overlap on the GPU (different streams,
 *     or host threads racing) race on the scratch and give wrong results: serialise
 *     them.
 *   - What its kernels record on the device (a bounded wait that timed out, an index
 *     check, non-finite gradients) goes to a static status record of its own, not the
 *     one fa_device_status() reads: read it with fa_bwd_noalloc_status().
 * Returns FA_OK, FA_ERR_INVALID_ARG, FA_ERR_UNSUPPORTED or FA_ERR_CUDA (argument and
 * launch errors; device-side errors come from fa_bwd_noalloc_status()).
 */
#define FA_NOALLOC_SCRATCH_BYTES (32u * 1024u * 1024u)

int fa_bwd_noalloc(const void* q, const void* k, const void* v, const void* o, const float* lse, const void* dO,
                   void* dq, void* dk, void* dv, float* delta_out, int B, int H, int N, int d, int causal,
                   float scale, void* stream);

/*
 * fa_bwd_noalloc_status -- synchronise `stream`, then read and clear the status record
 * that fa_bwd_noalloc's kernels write on the current device.  Allocates nothing (the
 * record is a static device variable; its address was looked up by the first
 * fa_bwd_noalloc call on the device, or is looked up here).  `out` may be NULL; when
 * given, it receives the record as it was before clearing.
 * Returns FA_OK, FA_ERR_TIMEOUT, FA_ERR_DEVICE_BOUNDS or FA_WARN_NONFINITE (in that
 * order of precedence), or FA_ERR_CUDA if the synchronisation or the copy fails.
 */
int fa_bwd_noalloc_status(void* stream, fa_device_report* out);

/*
 * fa_device_status -- synchronise `stream`, then return and clear the current
 * device's status record: FA_OK, FA_ERR_TIMEOUT, FA_ERR_DEVICE_BOUNDS or
 * FA_WARN_NONFINITE (in that order of precedence; FA_ERR_CUDA if the
 * synchronisation itself fails).  FA_WARN_NONFINITE is the NaN monitor of
 * [jsqmd §5] / [ijyty §7.1]: some output written since the last read held a
 * NaN or an Inf (e.g. from non-finite inputs); the call itself completed.
 */
int fa_device_status(void* stream);

/*
 * fa_device_report_read -- the same as fa_device_status, and also copies the record
 * (flags, first failed index check, non-finite count per output) into `out` (non-NULL)
 * before it is cleared, so a caller can tell which output held NaN or Inf and how many
 * entries did.
 */
int fa_device_report_read(void* stream, fa_device_report* out);

/* Message for the last non-OK return on the calling thread ("" if none). */
const char* fa_last_error(void);

/* Library version string. */
const char* fa_version(void);

#ifdef __cplusplus
}
#endif

#endif /* FA_H_ */
