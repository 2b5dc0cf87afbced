// Host/device declarations shared by the translation units of libsagebwd.
#pragma once
#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <cstddef>
#include <cstdint>

#include "../../include/sagebwd.h"

namespace sagebwd {

constexpr int kBlk = 128;                            // tokens per quantization block and per tile
// What a quantizer stores: the INT8 code (the method), the BF16 rounding of the scaled value (error
// attribution), or the FP8 E4M3 rounding of the value scaled to 448 (the FP8 variant); the last two
// are exact in the BF16 operand carrier.
enum ValueMode { kValInt8 = 0, kValBf16 = 1, kValFp8 = 2 };
constexpr float kFp8Max = 448.f;                     // largest finite E4M3 value
constexpr float kLog2_448 = 8.8073549220576041f;     // log2(448)
constexpr float kLog2e = 1.4426950408889634f;        // log2(e)
constexpr float kLn2 = 0.69314718055994531f;         // ln(2)
constexpr float kLog2_127 = 6.9886846867721655f;     // log2(127)
constexpr uint64_t kDefaultTimeoutNs = 2000000000ull;
// A quantization group (block, P^T row, dS tile) whose largest magnitude is
// below 2^-120 quantizes to zero codes with scale 0, so that 127/max never
// overflows FP32.
constexpr float kMinGroupMax = 7.52316384526264e-37f;  // 2^-120
// The same rule for the FP8 variant, whose 448/max overflows FP32 already below ~2^-119.2.
constexpr float kMinGroupMaxFp8 = 3.00926553810506e-36f;  // 2^-118

// Status word codes written by kernels (low byte = sagebwd_status, bits 8..15 = wait site).
__host__ __device__ constexpr int status_timeout(int site) { return (int)SAGEBWD_ERR_TIMEOUT | (site << 8); }

inline int nblocks(int N) { return (N + kBlk - 1) / kBlk; }

// ------------------------------------------------------------------ quantize
struct QuantJob {
  const __nv_bfloat16* x;  // [BH][N][d]
  __nv_bfloat16* xq;       // [BH][N][d] integer-valued codes
  float* scale;            // [BH][nb]
  const float* mean;       // [BH][d] or nullptr
  int BH;
  const int* bexp;         // [B*Hkv][d] channel balancing exponents, or nullptr
  int bexp_group;          // heads per exponent row: Hq/Hkv for Q, 1 for K
  int bexp_sign;           // -1: x times 2^-e (Q); +1: x times 2^e (K)
  int subexp;              // 1: power-of-two sub-scales per 8-channel group of each block (Q/K option)
  float* bmean;            // [BH][nb][d] or nullptr: Q-smoothing, each block's channel means subtracted
                           // first (and written here)
  int vmode;               // ValueMode: INT8 code (0), BF16 of x * 127/max (1), E4M3 of x * 448/max (2)
  // FP8 variant only (else nullptr): the same E4M3 values as bytes, for the FP8 tensor cores
  uint8_t* x8;             // [BH][N][d]
  uint8_t* x8t;            // [BH][d][128 nb]: each head's values transposed (tokens contiguous), zero past N
  double* part;            // non-null: this job only writes the FP64 channel sums of each block [BH][nb][d]
                           // (the K-mean pass), no codes
};
struct QuantParams {
  QuantJob job[3];
  int njobs;
  int block_start[4];  // prefix sums of BH * nb over the jobs
  int N, d, nb;
  int* status;         // cleared by block 0 when clear_status
  int clear_status;
};
// pdl: launched as a programmatic dependent of the previous grid in the stream (the blocks of a
// job with a mean wait for that grid; the others may run beside it).
cudaError_t launch_quantize(const QuantParams& p, cudaStream_t s, bool pdl = false);
cudaError_t launch_kmean(const __nv_bfloat16* k, double* part, float* mean, int BH, int N, int d, int* status,
                         int clear_status, cudaStream_t s);
// The second half of the K-mean pass alone: mean[bh][c] = (sum of the block sums) / N.
cudaError_t launch_kmean_final(const double* part, float* mean, int BH, int N, int d, cudaStream_t s,
                               bool pdl = false);
// Channel statistics of Q and K for the channel balancing: per (b, kv head,
// channel) the K mean (smooth) and the balancing exponent.
struct StatsParams {
  const __nv_bfloat16* q;  // [B*Hq][N][d]
  const __nv_bfloat16* k;  // [B*Hkv][N][d]
  double* ksum;            // [B*Hkv][nb][d] partial sums (scratch)
  float* kmax;             // [B*Hkv][nb][d] partial maxima (scratch)
  float* kmin;             // [B*Hkv][nb][d] partial minima (scratch)
  float* qmax;             // [B*Hq][nb][d] partial max |Q| (scratch)
  float* mean;             // [B*Hkv][d] K channel means (written when smooth)
  int* bexp;               // [B*Hkv][d] balancing exponents
  int BHq, BHk, G, N, d, nb, smooth;
  int* status;             // cleared by the first block
};
cudaError_t launch_qk_stats(const StatsParams& p, cudaStream_t s);
// Q-smoothing's logit terms bias[bhq][ib][k] = c0 * (mean_Q(bhq, ib) . K'_k), K' = K - mean_K
// (kmean non-null) or K, for every key k < 128 * nb (0 past N); causal: only ib >= k / 128.
struct QBiasParams {
  const __nv_bfloat16* k;  // [B*Hkv][N][d]
  const float* kmean;      // [B*Hkv][d] or nullptr
  const float* qmean;      // [B*Hq][nb][d]
  float* bias;             // [B*Hq][nb][128 nb]
  int BHq, G, N, d, nb, causal;
  float c0;
};
cudaError_t launch_qsmooth_bias(const QBiasParams& p, cudaStream_t s);

// ------------------------------------------------------------------ backward helpers
struct PrepParams {
  const __nv_bfloat16* o;   // [BHq][N][d]
  const __nv_bfloat16* dO;  // [BHq][N][d]
  float* D;                 // [BHq][N]
  __nv_bfloat16* dOq;       // [BHq][N][d]
  float* sdo;               // [BHq][nb]
  float* dq_acc;            // [BHq][N][d], zeroed
  float* dk_acc;            // [BHk][N][d], zeroed
  float* dv_acc;            // [BHk][N][d], zeroed
  int BH, BHk, N, d, nb;
  int* status;
  int vmode;                // ValueMode of the dO quantizer
};
cudaError_t launch_bwd_prep(const PrepParams& p, cudaStream_t s);
// FP32 gradient accumulators -> BF16 outputs, up to three arrays in one launch.
struct ConvertJob {
  const float* acc;
  __nv_bfloat16* out;
  size_t n;          // elements, a multiple of 4
  const int* bexp;   // nullptr, or [B*Hkv][d] balancing exponents: out = acc * 2^(sign * e)
  int sign;          // -1 for dQ, +1 for dK
  int group;         // heads per exponent row (Hq/Hkv for dQ, 1 for dK)
  int N, d;
};
cudaError_t launch_grad_convert(const ConvertJob* jobs, int njobs, cudaStream_t s);

// ------------------------------------------------------------------ attention kernels
struct FwdParams {
  int B, Hq, Hkv, N, nb, G;
  float c0;  // softmax_scale * log2(e), FP32
  const float* sq;
  const float* sk;
  const float* sv;
  __nv_bfloat16* o;
  float* lse;
  const float* qbias;  // Q-smoothing logit terms [BHq][nb][128 nb] (base 2), or nullptr
  int* status;
  uint64_t timeout_ns;
  uint32_t flags;
};
// The debug-dump instantiation (SAGEBWD_FLAG_DEBUG_DUMP) takes this extension: one record per
// tile, layout as documented at sagebwd_debug_dump_offset.
struct FwdDumpParams : FwdParams {
  uint8_t* dump;
};
// dump == nullptr selects the plain (or Q-smoothing) instantiations.  f8: the FP8 variant on the
// FP8 tensor cores (tq, tk over the E4M3 bytes of Q^, K^ [BH][N][d], tv over V^ transposed
// [BHk][d][128 nb]; p.flags must carry kFlagFp8Codes).
cudaError_t launch_fwd(const CUtensorMap& tq, const CUtensorMap& tk, const CUtensorMap& tv, const FwdDumpParams& p,
                       int d, int causal, int f8, cudaStream_t s);

// Kept at 128 bytes: a larger parameter block made ptxas spill in the d = 64 kernels.
struct BwdParams {
  int B, Hq, Hkv, N, nb, G;
  float c0;        // softmax_scale * log2(e)
  float sc;        // softmax_scale
  const float* sq;  // [BHq][nb]
  const float* sk;  // [BHk][nb]
  const float* sdo; // [BHq][nb]
  const float* lse; // [BHq][N]
  const float* D;   // [BHq][N]
  int HS;           // query heads per CTA (a divisor of G)
  uint32_t flags;   // SAGEBWD_FLAG_* | kBwdDirectDKDV
  float* dq_acc;    // [BHq][N][d]
  // dK, dV destinations [BHk][N][d]: FP32 accumulators (added into), or, with kBwdDirectDKDV
  // (one CTA covers all G query heads of its key block and no factor follows), the BF16 outputs
  void* dk_dst;
  void* dv_dst;
  int* status;
  uint64_t timeout_ns;
};
constexpr uint32_t kBwdDirectDKDV = 1u << 31;
// FwdParams.flags / BwdParams.flags: the FP8 variant's codes (set by the library, not by callers)
constexpr uint32_t kFlagFp8Codes = 1u << 30;
static_assert(sizeof(BwdParams) <= 128, "backward parameter block above 128 bytes");
// The Q-smoothing instantiations take these extra tables: the logit terms [BHq][nb][128 nb], the
// block means of Q [BHq][nb][d], and scratch for the per-slice column sums of the dS codes
// [grid][2][4][128].
struct BwdQsmParams : BwdParams {
  const float* qbias;
  const float* qmean;
  float* cs_part;
  uint8_t* dump;  // debug dump (plain instantiation only), or nullptr
};
struct BwdDumpParams : BwdParams {
  uint8_t* dump;
};
// p.qbias == nullptr selects the plain instantiations (which take only the BwdParams part).
cudaError_t launch_bwd(const CUtensorMap& tq, const CUtensorMap& tk, const CUtensorMap& tv, const CUtensorMap& tdo,
                       const CUtensorMap& tdoq, const CUtensorMap& tdq, const BwdQsmParams& p, int d, int causal,
                       int ds_subexp, cudaStream_t s);
// Query heads per backward CTA: the divisor of G whose CTAs, dispatched longest
// first onto `sms` multiprocessors, finish soonest (ties: more heads per CTA).
int bwd_heads_per_cta(int B, int Hkv, int G, int nb, int causal, int sms);

}  // namespace sagebwd
