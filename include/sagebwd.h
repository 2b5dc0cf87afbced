/*
 * sagebwd.h -- C ABI of the GB300 (sm_103a) SageBwd attention library.
 *
 * SageBwd is the trainable INT8 attention of "SageBwd: A Trainable Low-bit
 * Attention" (Abstract): its forward and backward quantize six of the seven
 * attention matmuls to INT8 -- forward S = Q K^T and O = P V, backward S
 * recompute, dV = P^T dO, dQ = dS K and dK = dS^T Q -- and keep only
 * dP = dO V^T in 16-bit floating point ("SageAttention3: Microscaling FP4
 * Attention for Inference and An Exploration of 8-Bit Training", summary
 * page, Approach, and the "Measured effects" row on leaving dO V^T
 * unquantized).
 * K is smoothed by subtracting its per-channel mean over tokens (SageBwd
 * Abstract, finding (iv)); QK-norm, where used, is applied by the caller.
 *
 * Quantization granularity (the pages leave it open; this library's choice):
 *   Q, K, V, dO : one FP32 scale per 128-token block of a head (all d
 *                 channels): a = max|x|, scale = a/127,
 *                 code = clamp(rint(x * 127/a), -127, 127), half to even;
 *   forward P~  : per query row and 128-key tile, code = rint(127*2^(t-tmax));
 *   backward P  : per key and 128-query tile, scale = max P / 127;
 *   backward dS : one scale per 128 x 128 tile, scale = max|dS| / 127.
 * Optional channel balancing (balance_qk = 1; off by default, this library's
 * addition after SmoothQuant, listed under "Builds on" of the SageBwd page):
 * per (batch, kv head, channel) an exponent
 *   e = clamp(floor((E(aQ) - E(aK)) / 2), -126, 126)   (0 if aQ or aK is 0),
 * with aQ the channel's max |Q| over the kv head's query heads and all
 * tokens, aK its max |K - mean_K| (|K| without smoothing), E(a) = floor(log2 a);
 * Q's channel is multiplied by 2^-e and K's (after smoothing) by 2^e before
 * the block quantizers, which leaves Q K^T unchanged exactly and evens out
 * channel outliers between the two operands; dQ is multiplied by 2^-e and
 * dK by 2^e when they are converted to BF16.
 * Q/K sub-scales (qk_subexp = 1: this library's default Q/K granularity, which
 * the Python binding and the benchmark select unless told otherwise; 0 keeps
 * one scale per block, the plainest reading): each 8-channel group of a
 * 128-token block of Q and of K keeps the block scale and is refined by 2^k,
 * k = clamp(floor(log2(block max / group max)), 0, 8) (0 if the group max is
 * below 2^-100): stored value rint(x * 127/max * 2^k) * 2^-k, exact in BF16
 * (x_q of sagebwd_quantize then holds such values for Q and K).  Channel
 * outliers then cost precision only in their own group: on inputs with 1% of
 * the channels scaled x20 the plain mode misses cosine similarity 0.995 (O) /
 * 0.99 (dQ, dK) against exact attention and this mode meets it; on inputs
 * without channel outliers (QK-normed, or roughly Gaussian per channel) every
 * k is 0 and both modes give the same codes.  (The
 * SageBwd pages fix INT8 per-block quantization of Q and K, Abstract, but no
 * block shape; the sub-scales are a power-of-two refinement inside the block.)
 * Optional dS sub-scales (ds_subexp = 1; off by default, this library's finer
 * dS granularity): the tile keeps its scale max|dS| / 127, and each key's codes
 * within a group of 32 queries of the tile are refined by 2^k,
 * k = clamp(floor(log2(tile max / group max)), 0, 8) (0 if the group max is
 * below 2^-100): code = rint(dS * 127/max * 2^k), operand value code * 2^-k,
 * exact in BF16, read as is by dK = dS^T Q and dQ = dS K (their FP32 sums are
 * then no longer exact integers, but rounding there is at the 2^-24 level).
 * Optional Q-smoothing (smooth_q = 1; off by default; the SageBwd page calls
 * it optional with limited benefit, Abstract, finding (iv)): each 128-token
 * block of each query head subtracts its FP32 channel means mean_Q (exact sum
 * over the block's tokens, divided, rounded to FP32) before quantizing, and
 * the logits gain the FP32 term mean_Q(block of i) . K'_k (K' the K that the
 * quantizer sees: K - mean_K with smooth_k), so S = Q K'^T is unchanged up to
 * quantization.  The backward adds the same term to the recomputed S and, for
 * dK = dS^T (Q - mean_Q + mean_Q), the block mean's share: per tile
 * scale * s_dS * (sum over the tile's queries of the dS codes) * mean_Q.  dQ
 * needs no correction.  Not combined with balance_qk (SAGEBWD_ERR_UNSUPPORTED);
 * sagebwd_quantize returns SAGEBWD_ERR_UNSUPPORTED for Q under it (its codes
 * come with block means, which only sagebwd_fwd_quantize stores).
 * The INT8 codes are held as integer-valued BF16 and multiplied on the
 * tensor cores with FP32 accumulation, which is exact for these tiles
 * (|sum| <= 128 * 127^2 < 2^24).
 * FP8 variant (fp8 = 1; the pages compare INT8 with FP8 SageBwd, "SageAttention3 ... 8-Bit
 * Training" summary page, Measured effects): every quantizer of the method stores the FP8 E4M3
 * rounding (to nearest even, saturating at 448) of its value scaled to 448 instead of an INT8 code,
 * with the same granularity (Q, K, V, dO per 128-token block, scale max/448; forward P~ per row and
 * key tile, E4M3 of 448 * 2^(t - tmax); backward P per key and query tile, scale max/448; dS per
 * tile, scale max/448); dP = dO V^T stays BF16.  Not with qk_subexp, ds_subexp, balance_qk,
 * smooth_q, the BF16 attribution flags or SAGEBWD_FLAG_DEBUG_DUMP (SAGEBWD_ERR_UNSUPPORTED).
 *
 * Conventions for every entry point:
 *   - Tensors are row-major contiguous. Q, dO, O, dQ: BF16 [B][Hq][N][d];
 *     K, V, dK, dV: BF16 [B][Hkv][N][d]; LSE: FP32 [B][Hq][N].
 *     Query head h reads kv head h / (Hq / Hkv) (grouped-query attention).
 *   - Every pointer is a DEVICE pointer owned by the caller, 16-byte aligned.
 *     The library allocates, frees and synchronizes nothing (except
 *     sagebwd_check_status, which synchronizes the given stream), keeps no
 *     state between calls beyond read-only caches (driver entry points, SM
 *     counts, the query heads per backward CTA chosen for a shape) and the
 *     static scratch array of sagebwd_quantize_k_noalloc, and launches only
 *     on the given stream.
 *   - Supported: d in {64, 128}; Hq % Hkv == 0; N >= 1; B, Hq, Hkv >= 1.
 *   - Errors are returned before any launch for bad arguments; a launch
 *     failure returns SAGEBWD_ERR_CUDA.  Kernels bound every wait; a wait
 *     that runs out records SAGEBWD_ERR_TIMEOUT in the status word kept in
 *     the workspace, read with sagebwd_check_status.  No C++ exception
 *     crosses this interface.
 */
#ifndef SAGEBWD_H_
#define SAGEBWD_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
  SAGEBWD_OK = 0,
  SAGEBWD_ERR_INVALID_ARG = 1, /* null pointer, bad sizes, Hq % Hkv != 0 */
  SAGEBWD_ERR_UNSUPPORTED = 2, /* head dim other than 64 / 128, or a size beyond the int32 index range */
  SAGEBWD_ERR_MISALIGNED = 3,  /* a pointer not 16-byte aligned */
  SAGEBWD_ERR_CUDA = 4,        /* a CUDA runtime call or launch failed */
  SAGEBWD_ERR_TIMEOUT = 5,     /* a kernel's bounded wait ran out (device status word) */
  SAGEBWD_ERR_SCRATCH_LIMIT = 6 /* the problem needs more than the fixed scratch of sagebwd_quantize_k_noalloc */
} sagebwd_status;

/* Which operand sagebwd_quantize handles. */
enum { SAGEBWD_Q = 0, SAGEBWD_K = 1, SAGEBWD_V = 2, SAGEBWD_DO = 3 };

/* sagebwd_problem.flags */
#define SAGEBWD_FLAG_DROP_ONE_LOAD 0x1u /* fault injection: the forward kernel skips one K-tile load and the
                                           backward kernel the dO^ load of each CTA's second tile, so
                                           their bounded waits run out and the call reports
                                           SAGEBWD_ERR_TIMEOUT */
#define SAGEBWD_FLAG_DEBUG_DUMP 0x2u    /* parity checking: the attention kernels also write every tile's
                                           INT8-semantics operands and raw tensor-core products into the
                                           workspace (layout at sagebwd_debug_dump_offset; small problems
                                           only; not with ds_subexp or smooth_q) */
/* Error attribution ("SageBwd: A Trainable Low-bit Attention", Abstract, finding (ii): the backward's
 * error comes mainly from dS; "SageAttention3 ... 8-Bit Training" summary, Measured effects: the dO V^T
 * row): each flag makes one quantizer keep its scale but store the BF16 rounding (to nearest even) of
 * the scaled value, x * 127/max, instead of its INT8 code, so that comparing runs with one flag set
 * shows how much of the error that quantizer carries.  Q^ and K^ then carry no sub-scales.  Not with
 * ds_subexp, smooth_q or SAGEBWD_FLAG_DEBUG_DUMP (SAGEBWD_ERR_UNSUPPORTED). */
#define SAGEBWD_FLAG_BF16_Q 0x10u   /* Q^ */
#define SAGEBWD_FLAG_BF16_K 0x20u   /* K^ */
#define SAGEBWD_FLAG_BF16_V 0x40u   /* V^ */
#define SAGEBWD_FLAG_BF16_DO 0x80u  /* dO^ */
#define SAGEBWD_FLAG_BF16_PF 0x100u /* forward P~ (per row and key tile) */
#define SAGEBWD_FLAG_BF16_PB 0x200u /* backward P^T (per key and query tile) */
#define SAGEBWD_FLAG_BF16_DS 0x400u /* backward dS (per tile) */
#define SAGEBWD_FLAGS_BF16 0x7F0u

typedef struct {
  int32_t B, Hq, Hkv, N, d;
  int32_t causal;       /* 1: key k visible to query i iff k <= i (top-left aligned); 0: all keys */
  int32_t smooth_k;     /* 1: subtract the per-channel mean of K over tokens before quantizing (the method) */
  int32_t balance_qk;   /* 1: power-of-two Q/K channel balancing before quantizing (see above); 0 in the method */
  int32_t ds_subexp;    /* 1: dS sub-scales per key and 32-query group (see above); 0: one dS scale per tile */
  int32_t qk_subexp;    /* 1 (recommended default): Q/K sub-scales per 8-channel group of each block (see
                           above); 0: one scale per block */
  int32_t smooth_q;     /* 1: Q-smoothing, block means of Q subtracted (see above); 0: plain Q (the default) */
  uint32_t flags;       /* SAGEBWD_FLAG_* (0 in normal use) */
  float softmax_scale;  /* <= 0 selects 1/sqrt(d) */
  uint32_t wait_timeout_ms; /* bound of every in-kernel wait; 0 selects 2000 ms */
  int32_t fp8;          /* 1: the FP8 variant (see above); 0: INT8, the method */
} sagebwd_problem;

/* Bytes of the `saved` buffer that sagebwd_fwd fills and sagebwd_bwd reads:
 * the quantized Q, K, V (integer-valued BF16, same shapes as the inputs),
 * their FP32 block scales, the FP32 mean of K [B*Hkv][d], the int32
 * balancing exponents [B*Hkv][d] (written only with balance_qk) and, with
 * smooth_q, the FP32 block means of Q [B*Hq][ceil(N/128)][d] and the FP32
 * logit terms mean_Q . K' [B*Hq][ceil(N/128)][128 * ceil(N/128)] (in base-2
 * units, times scale * log2 e), each section starting on a 256-byte
 * boundary, and with fp8 the same E4M3 values as bytes for the FP8 tensor cores: Q [B*Hq][N][d],
 * K [B*Hkv][N][d] and V transposed per head [B*Hkv][d][128 * ceil(N/128)] (zero past N).  Returns 0
 * for an invalid problem. */
size_t sagebwd_saved_bytes(const sagebwd_problem* prob);

/* Bytes of workspace for pass 0 (forward, sagebwd_fwd / sagebwd_quantize) or
 * pass 1 (backward, sagebwd_bwd).  The workspace holds the status word first,
 * then scratch (K-mean partial sums, and with balance_qk the per-block channel
 * maxima of Q and K; D = rowsum(dO*O), the quantized dO and its scales, the
 * FP32 dQ, dK and dV accumulators, and with smooth_q a small ring of dS column
 * sums per backward CTA; with SAGEBWD_FLAG_DEBUG_DUMP the dump follows).
 * Contents need no initialisation and are
 * not meaningful between calls, except the status word. */
size_t sagebwd_workspace_bytes(const sagebwd_problem* prob, int pass);

/* Quantize one operand ("SageBwd", Abstract: INT8 quantization; K-smoothing).
 *   which  : SAGEBWD_Q / _K / _V / _DO; x has that operand's shape.  With
 *            balance_qk the codes of Q and K depend on both tensors: Q and K
 *            then return SAGEBWD_ERR_UNSUPPORTED (use sagebwd_fwd_quantize).
 *   x_q    : BF16 output, same shape, integer values in [-127, 127] (for Q and K
 *            with qk_subexp: such integers times 2^-k, k in [0, 8]).
 *   scales : FP32 [B*H][ceil(N/128)] block scales.
 *   k_mean : FP32 [B*Hkv][d] channel means when which == SAGEBWD_K and
 *            smooth_k == 1 (then required), else ignored (may be NULL).
 *   ws     : forward workspace (sagebwd_workspace_bytes(prob, 0)).       */
sagebwd_status sagebwd_quantize(const sagebwd_problem* prob, int which, const void* x, void* x_q, float* scales,
                                float* k_mean, void* ws, void* stream);

/* Forward: quantize Q, K (smoothed, balanced as selected), V into `saved`, then the fused
 * attention forward with online softmax ("SageBwd", Abstract; FlashAttention
 * lineage listed under "Builds on").
 *   o   : BF16 [B][Hq][N][d] output.
 *   lse : FP32 [B][Hq][N], natural-log log-sum-exp of each row of the scores
 *         the kernel softmaxes, scale * Q (K - mean_K)^T (with smooth_k = 1 this
 *         differs from the LSE of scale * Q K^T by -scale * Q_i . mean_K).
 *   saved : sagebwd_saved_bytes(prob) bytes, read back by sagebwd_bwd.
 *   ws  : sagebwd_workspace_bytes(prob, 0) bytes.                          */
sagebwd_status sagebwd_fwd(const sagebwd_problem* prob, const void* q, const void* k, const void* v, void* o,
                           float* lse, void* saved, void* ws, void* stream);

/* Backward ("SageBwd: A Trainable Low-bit Attention", Abstract: the INT8 S
 * recompute and the INT8 products dV = P^T dO, dQ = dS K, dK = dS^T Q; the
 * "SageAttention3 ... 8-Bit Training" summary page, Approach: dP = dO V^T kept
 * in 16-bit floating point; D = rowsum(dO * O) and dS = P (dP - D) from the
 * FlashAttention-2 backward listed under "Builds on"): D and the quantized dO,
 * then the fused backward (S recompute, dV = P^T dO, dP = dO V^T in BF16,
 * dS = P (dP - D), dK = dS^T Q, dQ = dS K) and the FP32 -> BF16 conversion of dQ.
 *   q, k, v, o, dO : the forward's inputs and output and the gradient of o.
 *   lse, saved     : exactly as produced by sagebwd_fwd for these inputs.
 *   dq : BF16 [B][Hq][N][d]; dk, dv : BF16 [B][Hkv][N][d] (summed over the
 *        query heads of each kv head).
 *   ws : sagebwd_workspace_bytes(prob, 1) bytes.                            */
sagebwd_status sagebwd_bwd(const sagebwd_problem* prob, const void* q, const void* k, const void* v, const void* o,
                           const void* dO, const float* lse, const void* saved, void* dq, void* dk, void* dv, void* ws,
                           void* stream);

/* The same two passes split into the library's kernel stages, for callers
 * that schedule or time them separately.  Calling the stages in this order,
 * on one stream, is exactly sagebwd_fwd / sagebwd_bwd.
 *   sagebwd_fwd_quantize  : K mean (and the balancing exponents) and the
 *                           Q, K, V quantization into `saved`.  With
 *                           K-smoothing (and no balancing) its later launches
 *                           are programmatic dependents of the earlier ones
 *                           (CUDA's programmatic stream serialization): Q and V
 *                           are quantized while K's mean is computed.  The
 *                           stage's first launch, and every launch after the
 *                           stage, are ordinary stream-ordered launches.
 *   sagebwd_fwd_attention : the fused forward kernel on `saved` -> o, lse.
 *   sagebwd_bwd_prepare   : D = rowsum(dO * O), quantized dO, zeroed dQ
 *                           accumulator and, when they are used, dK and dV
 *                           accumulators (all in the backward workspace).
 *   sagebwd_bwd_attention : the fused backward kernel -> the FP32 dQ, dK, dV
 *                           accumulators in the workspace; when one CTA covers
 *                           all query heads of a kv head (the library's choice
 *                           of query heads per CTA, e.g. always with Hq == Hkv)
 *                           and balance_qk is 0, it writes BF16 dk, dv itself
 *                           and the dK / dV accumulators are not used.
 *   sagebwd_bwd_finish    : the accumulators -> BF16 dq and, unless the
 *                           attention stage wrote them, dk, dv (times 2^-e
 *                           and 2^e with balance_qk; `saved` holds e).
 * The three backward stages must see the same problem (they take the same
 * decision on dk, dv).                                                      */
sagebwd_status sagebwd_fwd_quantize(const sagebwd_problem* prob, const void* q, const void* k, const void* v,
                                    void* saved, void* ws, void* stream);
sagebwd_status sagebwd_fwd_attention(const sagebwd_problem* prob, const void* saved, void* o, float* lse, void* ws,
                                     void* stream);
sagebwd_status sagebwd_bwd_prepare(const sagebwd_problem* prob, const void* o, const void* dO, void* ws,
                                   void* stream);
sagebwd_status sagebwd_bwd_attention(const sagebwd_problem* prob, const void* v, const void* dO, const float* lse,
                                     const void* saved, void* dk, void* dv, void* ws, void* stream);
sagebwd_status sagebwd_bwd_finish(const sagebwd_problem* prob, const void* saved, void* dq, void* dk, void* dv,
                                  void* ws, void* stream);

/* K quantization (K-smoothing mean + per-block codes), like
 * sagebwd_quantize(prob, SAGEBWD_K, ...), for callers that cannot allocate
 * device memory -- an operator hook handed only its input and output tensors,
 * code that runs where cudaMalloc is not allowed or would synchronize the
 * device, a process whose memory belongs to a pool it cannot draw from at that
 * point.  It takes no workspace: the FP64 channel sums of the K-mean pass go to
 * a fixed 8 MiB array compiled into the library, which every GPU that loads
 * the library keeps until the process exits.  (The SageBwd pages have no
 * counterpart of this entry point.)
 *   - balance_qk must be 0 (K's codes would depend on Q): else
 *     SAGEBWD_ERR_UNSUPPORTED.
 *   - Limit: B * Hkv * ceil(N/128) * d <= 1048576 (e.g. B=2, Hkv=30, N=17776,
 *     d=64 needs 533760); larger problems return SAGEBWD_ERR_SCRATCH_LIMIT
 *     before any launch.  With smooth_k == 0 no scratch is used.
 *   - The first call on a device looks up the array's device address
 *     (cudaGetSymbolAddress) with that device current; make that first call
 *     before any stream capture.  The address is kept per device and context:
 *     after cudaDeviceReset the next call looks it up again (and that call,
 *     too, should come before any capture).  It allocates nothing at any time.
 *   - All calls share the one array: calls that can overlap on the GPU (other
 *     streams, other host threads) race and must be serialized by the caller.
 *     Every partial sum is written before it is read, so the array needs no
 *     clearing between calls.
 *   k, k_q, scales, k_mean: as for sagebwd_quantize with which == SAGEBWD_K. */
sagebwd_status sagebwd_quantize_k_noalloc(const sagebwd_problem* prob, const void* k, void* k_q, float* scales,
                                          float* k_mean, void* stream);

/* Synchronize `stream` and return the status word in `ws` (SAGEBWD_OK or
 * SAGEBWD_ERR_TIMEOUT); *detail (optional) receives the raw word, whose bits
 * 8..15 name the wait that ran out. */
sagebwd_status sagebwd_check_status(const void* ws, void* stream, int32_t* detail);

const char* sagebwd_status_string(sagebwd_status s);

/* Byte offset inside the pass-0 (forward) or pass-1 (backward) workspace of the
 * debug dump written under SAGEBWD_FLAG_DEBUG_DUMP; 0 when the flag is not set
 * or the problem is invalid.  One record per 128 x 128 tile (b, query head h,
 * query block i, key block j), at index ((b*Hq + h)*nb + i)*nb + j, nb =
 * ceil(N/128); records of tiles a causal problem skips are not written.
 * Forward record (T_f = 128*128*4 + 128*128*2 + 128*d*4 bytes):
 *   FP32 S_int [128 queries][128 keys] = Q^ K^T of the stored values, as accumulated (integers
 *   without Q/K sub-scales; with them sums of (code 2^-k)(code 2^-k') products, which FP32 need
 *   not hold exactly);
 *   BF16 P~ codes [128 queries][128 keys];  FP32 [P^ V^] [128 queries][d].
 * Backward record (T_b = 2*128*128*2 + 3*128*d*4 bytes):
 *   BF16 P^T codes [128 keys][128 queries];  BF16 dS codes [128 keys][128 queries];
 *   FP32 [P^T dO^] [128 keys][d];  FP32 [dS^T Q^] [128 keys][d];  FP32 [dS K^] [128 queries][d].
 * The workspace of a flagged problem is that much larger; a problem whose dump
 * would exceed 2^31 bytes is refused (SAGEBWD_ERR_UNSUPPORTED). */
size_t sagebwd_debug_dump_offset(const sagebwd_problem* prob, int pass);

/* Library version, as major*10000 + minor*100 + patch. */
int32_t sagebwd_version(void);

#ifdef __cplusplus
}
#endif

#endif /* SAGEBWD_H_ */
