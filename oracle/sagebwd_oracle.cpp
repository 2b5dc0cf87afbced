// SageBwd CPU oracle.  TEST INFRASTRUCTURE ONLY: the tests, the smoke check
// and the bench's CPU baseline call this; the product path never does.
// It shares no code with the CUDA library.
//
// What it computes (sources):
//  * "SageBwd: A Trainable Low-bit Attention", Abstract: a trainable INT8
//    attention whose forward and backward quantize six of the seven attention
//    matmuls; K-smoothing (subtracting the mean of K over tokens) is kept;
//    the score gradient dS is the main error source.
//  * "SageAttention3: Microscaling FP4 Attention for Inference and An
//    Exploration of 8-Bit Training" (summary page), Approach and the
//    "Measured effects" row on leaving dO.V^T unquantized: the product is the
//    one matmul left in 16/64-bit floating point.
//  * FlashAttention / FlashAttention-2 (listed under "Builds on" of the SageBwd
//    page): the forward keeps the log-sum-exp of each query row, and the
//    backward uses D_i = rowsum(dO_i * O_i) and dS = P * (dP - D).
//
// The pages fix no block size, scale rule or rounding mode.  The readings
// implemented here (one per function below) are:
//  * every quantized operand of Q, K, V, dO is cut into blocks of 128 tokens
//    (all d channels), one scale per block: a = max|x|, s = a/127,
//    code = clamp(rint(x * (127/a)), -127, 127); a block whose max is below
//    2^-120 (zero, or so small that 127/a would overflow FP32) gives codes 0
//    and s = 0; the scale arithmetic is IEEE FP32;
//  * K is smoothed by its FP32 channel mean over all N tokens (sum taken in
//    FP64, divided by N in FP64, rounded once to FP32), K' = K - mean in FP32;
//  * forward P~: per query row and 128-key tile, code = rint(127*2^(t - tmax))
//    with tmax the row maximum inside the tile (so the tile's scale is
//    2^(tmax - m)/127 relative to the running maximum m); the softmax
//    denominator is summed from the unquantized P~;
//  * backward P (for dV = P^T dO): per key and 128-query tile, scale
//    max_i P / 127;  backward dS: one scale per 128 x 128 tile, max|dS|/127,
//    one code matrix shared by dK = dS^T Q and dQ = dS K;
//  * dP = dO V^T uses the BF16 inputs, accumulated here in FP64;
//  * no correction term for the gradient through the K mean (each row of dS
//    sums to zero, so the mean's gradient vanishes);
//  * ablation int8_dp (off by default): dP = dO V^T from the INT8 codes of dO
//    and V, the variant the pages' ablation rejects;
//  * optional Q-smoothing (smooth_q, off by default; the pages call it optional
//    with limited benefit in pre-training, SageBwd Abstract, finding (iv)): each
//    128-token block of Q subtracts its channel means before quantizing, and
//    S gains mean_Q . K'^T in FP32; dK gains (sum over the block's queries of
//    dS) times mean_Q (see qsmooth_bias);
//  * ablation fp8 (off by default): every quantizer produces FP8 E4M3 values
//    with scale max/448 instead of INT8 codes (the pages compare INT8 with FP8
//    SageBwd, "SageAttention3 ..." summary, Measured effects);
//  * optional Q/K sub-scales (qk_subexp, off by default; the library's own
//    finer Q/K granularity): a power-of-two refinement per 8-channel group of
//    each 128-token block (see quant_block);
//  * optional dS sub-scales (ds_subexp, off by default; the library's own
//    finer dS granularity): a power-of-two refinement per key and 32-query
//    group inside each tile, baked into the BF16 operand values (see
//    ds_subexp_of);
//  * optional channel balancing (balance_qk, off by default; the library's
//    own addition, after SmoothQuant, listed under "Builds on" of the SageBwd
//    page): per (batch, kv head, channel) an exponent e moves magnitude
//    between Q and K before their block quantizers -- Q's channel times 2^-e,
//    K's (smoothed) channel times 2^e -- which leaves Q K^T unchanged exactly;
//    dQ is multiplied by 2^-e and dK by 2^e at the end.  See balance_exponents.
//
// Every floating-point quantity that decides an integer code is rounded to
// FP32 exactly where the GPU path computes it in FP32 (Mode::F below); every
// other sum and product is FP64.  With exact_codes = 1 the quantizers keep
// their scales but skip rint and clamp and no FP32 rounding happens: the whole
// pipeline must then reproduce exact FP64 attention, which is what pins its
// structure (scales, masks, tile bookkeeping) in the tests.
#include <algorithm>
#include <cmath>
#include <cstdint>
#include <cstring>
#include <limits>
#include <vector>
#ifdef _OPENMP
#include <omp.h>
#endif

extern "C" {
typedef struct {
  int32_t B, Hq, Hkv, N, d;
  int32_t causal;       // 1: key k is visible to query i iff k <= i (top-left aligned, N_q == N_k)
  int32_t smooth_k;     // 1: subtract the per-channel mean of K before quantizing it
  int32_t balance_qk;   // 1: power-of-two channel balancing of Q and K before quantizing them
  int32_t exact_codes;  // 1: quantizers keep their scales but neither round nor clamp; no FP32 rounding
  int32_t threads;      // <= 0: OpenMP default
  uint32_t exact_mask;  // error attribution: bit set = that quantizer keeps its scale but skips rint/clamp
                        // (bit 0 Q, 1 K, 2 V, 3 dO, 4 P~ forward, 5 P^T backward, 6 dS); FP32 rounding stays
  int32_t int8_dp;      // ablation: dP = dO V^T from the INT8 codes of dO and V instead of BF16 operands
  int32_t ds_subexp;    // 1: dS codes carry a power-of-two sub-scale per (key, 32-query group) of a tile
  int32_t qk_subexp;    // 1: Q and K codes carry a power-of-two sub-scale per (block, 8-channel group)
  int32_t fp8;          // ablation: every quantizer produces FP8 E4M3 values (scale max/448) instead of INT8
  int32_t smooth_q;     // 1: Q-smoothing (block mean of Q subtracted before quantizing, mean . K' added to S)
  int32_t l_from_codes; // planted misreading, for the tests only: the softmax denominator summed from the
                        // dequantized P~ codes instead of the unquantized P~ (the reading kept here, r8)
  uint32_t bf16_mask;   // error attribution (same bit order as exact_mask): that quantizer keeps its scale
                        // but stores the BF16 rounding of the scaled value instead of its INT8 code
  double softmax_scale;  // <= 0: 1/sqrt(d)
} oracle_problem;
}

namespace {

constexpr int BLK = 128;  // tokens per quantization block and per tile
constexpr double kLog2e = 1.4426950408889634073599246810019;
constexpr double kLn2 = 0.69314718055994530941723212145818;
const double kInf = std::numeric_limits<double>::infinity();

inline double bf16_to_double(uint16_t h) {
  uint32_t u = (uint32_t)h << 16;
  float f;
  std::memcpy(&f, &u, 4);
  return (double)f;
}

// Which quantizer a code belongs to (bit index of exact_mask).
enum Quantizer { QZ_Q = 0, QZ_K = 1, QZ_V = 2, QZ_DO = 3, QZ_PF = 4, QZ_PB = 5, QZ_DS = 6 };

// Arithmetic of the quantized algorithm.  F() is an FP32 rounding point (the
// GPU computes that value in FP32); Q() turns a scaled value into its integer
// code: round to nearest, ties to even (C nearbyint in the default mode), then
// clamp to [-127, 127].  Codes are stored as doubles: every integer product
// sum here stays far below 2^53, so it is exact.
// FP8 E4M3 (4 exponent bits, bias 7, 3 mantissa bits, no infinities, largest
// finite 448): round to nearest, ties to even, saturating at 448.  Normal
// numbers of binary exponent E (>= -6) have spacing 2^(E-3); below 2^-6 the
// subnormal spacing is 2^-9.
double round_e4m3(double v) {
  const double a = std::fabs(v);
  if (a == 0.0) return 0.0;
  int e = 0;
  std::frexp(a, &e);  // a = f 2^e, f in [0.5, 1): binary exponent e - 1
  const double q = std::ldexp(1.0, std::max(e - 1, -6) - 3);
  const double r = std::min(448.0, std::nearbyint(a / q) * q);
  return std::copysign(r, v);
}

// Round to BF16 (8 significant bits), to nearest with ties to even, from the FP32 value of v.
double round_bf16(double v) {
  const float f = (float)v;
  uint32_t u;
  std::memcpy(&u, &f, 4);
  if ((u & 0x7F800000u) == 0x7F800000u) return v;  // inf / nan unchanged
  u = (u + 0x7FFFu + ((u >> 16) & 1u)) & 0xFFFF0000u;
  float r;
  std::memcpy(&r, &u, 4);
  return (double)r;
}

struct Mode {
  bool fp32;       // false only in the exact_codes pin mode
  uint32_t exact;  // bit set: that quantizer does not round
  uint32_t bf16 = 0;      // bit set: that quantizer rounds to BF16 instead of to an INT8 code
  bool fp8 = false;       // the FP8 ablation: E4M3 values instead of INT8 codes
  double qmax = 127.0;    // largest code: 127 (INT8) or 448 (E4M3)
  // A quantization group (block, P^T row, dS tile) whose largest magnitude is below this gets
  // all-zero codes and scale 0, so that qmax/max stays finite in FP32: 2^-120 for INT8 codes,
  // 2^-118 for E4M3 values (448/max overflows below ~2^-119.2)
  double min_group() const { return fp8 ? std::ldexp(1.0, -118) : std::ldexp(1.0, -120); }
  double F(double x) const { return fp32 ? (double)(float)x : x; }
  double Q(int which, double x) const {
    if (exact & (1u << which)) return x;
    if (bf16 & (1u << which)) return round_bf16(x);
    if (fp8) return round_e4m3(x);
    const double r = std::nearbyint(x);
    return std::min(127.0, std::max(-127.0, r));
  }
};
inline Mode mode_of(const oracle_problem* p) {
  Mode m = p->exact_codes ? Mode{false, 0x7Fu} : Mode{true, p->exact_mask};
  m.bf16 = p->exact_codes ? 0u : p->bf16_mask;
  if (p->fp8) {
    m.fp8 = true;
    m.qmax = 448.0;
  }
  return m;
}

inline int nblocks(int N) { return (N + BLK - 1) / BLK; }
inline double scale_of(const oracle_problem* p) {
  return p->softmax_scale > 0 ? p->softmax_scale : 1.0 / std::sqrt((double)p->d);
}
inline void set_threads(const oracle_problem* p) {
#ifdef _OPENMP
  if (p->threads > 0) omp_set_num_threads(p->threads);
#else
  (void)p;
#endif
}

// One quantized tensor [BH][N][d]: codes, one scale per (bh, 128-token block), optional channel mean.
struct QTensor {
  int BH = 0, N = 0, d = 0;
  std::vector<double> codes;
  std::vector<double> scale;  // [BH][nblocks]
  std::vector<double> mean;   // [BH][d] (K only)
  std::vector<double> bmean;  // [BH][nblocks][d] block means (Q-smoothing only)
  std::vector<double> val;    // [BH][N][d] the values the quantizer saw (K under Q-smoothing only)
  double c(int bh, int n, int ch) const { return codes[((size_t)bh * N + n) * d + ch]; }
  double s(int bh, int blk) const { return scale[(size_t)bh * nblocks(N) + blk]; }
  double bm(int bh, int blk, int ch) const { return bmean[((size_t)bh * nblocks(N) + blk) * d + ch]; }
  double v(int bh, int n, int ch) const { return val[((size_t)bh * N + n) * d + ch]; }
};

// Power-of-two sub-scale exponent of a group inside a quantization group
// (the library's reading for the optional sub-scales): the largest integer k
// <= log2(amax / gmax), clamped to [0, kSubMax], and 0 when gmax is below
// 2^-100; from the binary exponents and fractions, so exact.
constexpr int kSubMax = 8;
int subexp_of(double amax, double gmax) {
  if (gmax < std::ldexp(1.0, -100)) return 0;
  int ea = 0, eg = 0;
  const double fa = std::frexp(amax, &ea), fg = std::frexp(gmax, &eg);
  const int k = ea - eg - (fa < fg ? 1 : 0);
  return std::min(kSubMax, std::max(0, k));
}

// Per-block absmax quantizer (the build's reading: 128 tokens x d channels,
// symmetric, scale a/127, round to nearest even, clamp to +-127).  With
// subexp (Q and K under qk_subexp) each group of 8 channels of the block
// (all its rows) is refined by 2^k, k = subexp_of(block max, group max): the
// value is code * 2^-k with code = rint(x * inv * 2^k), exact in BF16, and
// the block scale a/127 dequantizes it as before.
constexpr int kChanGroup = 8;
void quant_block(const Mode& M, int which, const double* x, int count, double* codes, double* scale, int d = 0,
                 bool subexp = false) {
  double a = 0;
  for (int e = 0; e < count; ++e) a = std::max(a, std::fabs(x[e]));
  if (a < M.min_group()) {
    for (int e = 0; e < count; ++e) codes[e] = 0;
    *scale = 0;
    return;
  }
  const double inv = M.F(M.qmax / a);
  *scale = M.F(a / M.qmax);
  if (!subexp) {
    for (int e = 0; e < count; ++e) codes[e] = M.Q(which, M.F(x[e] * inv));
    return;
  }
  const int rows = count / d;
  for (int c0 = 0; c0 < d; c0 += kChanGroup) {
    double g = 0;
    for (int r = 0; r < rows; ++r)
      for (int c = c0; c < c0 + kChanGroup; ++c) g = std::max(g, std::fabs(x[(size_t)r * d + c]));
    const double f = std::ldexp(1.0, subexp_of(a, g));
    for (int r = 0; r < rows; ++r)
      for (int c = c0; c < c0 + kChanGroup; ++c) {
        const size_t e = (size_t)r * d + c;
        codes[e] = M.Q(which, M.F(x[e] * inv) * f) / f;
      }
  }
}

// FP32 channel means of one head's tokens [N][d] ("SageBwd: A Trainable
// Low-bit Attention", Abstract: K-smoothing): FP64 sum, FP64 divide, one
// FP32 rounding.
void channel_mean(const Mode& M, const uint16_t* xb, int N, int d, double* mu) {
  for (int ch = 0; ch < d; ++ch) {
    double sum = 0;
    for (int n = 0; n < N; ++n) sum += bf16_to_double(xb[(size_t)n * d + ch]);
    mu[ch] = M.F(sum / (double)N);
  }
}

// Quantize a BF16 tensor [BH][N][d]; with smooth, first subtract the channel
// mean over all N tokens (K-smoothing).  With fac, every value (after the
// smoothing) is then multiplied by its channel's factor
// (*fac)[(bh / fac_group) * d + ch], rounded to FP32, before the block
// quantizer sees it (channel balancing).
// block_smooth (Q-smoothing): each block first subtracts its own channel means
// (FP64 sum over the block's valid tokens, divided in FP64, rounded to FP32),
// kept in out.bmean.  keep_vals keeps the values the quantizer saw in out.val.
void quantize_tensor(const Mode& M, int which, const uint16_t* x, int BH, int N, int d, bool smooth, QTensor& out,
                     const std::vector<double>* fac = nullptr, int fac_group = 1, bool subexp = false,
                     bool block_smooth = false, bool keep_vals = false) {
  out.BH = BH;
  out.N = N;
  out.d = d;
  const int nb = nblocks(N);
  out.codes.assign((size_t)BH * N * d, 0);
  out.scale.assign((size_t)BH * nb, 0.0);
  out.mean.assign(smooth ? (size_t)BH * d : 0, 0.0);
  out.bmean.assign(block_smooth ? (size_t)BH * nb * d : 0, 0.0);
  out.val.assign(keep_vals ? (size_t)BH * N * d : 0, 0.0);
#pragma omp parallel for schedule(dynamic)
  for (int bh = 0; bh < BH; ++bh) {
    const uint16_t* xb = x + (size_t)bh * N * d;
    std::vector<double> mu(d, 0.0);
    if (smooth) {
      channel_mean(M, xb, N, d, mu.data());
      std::copy(mu.begin(), mu.end(), out.mean.begin() + (size_t)bh * d);
    }
    const double* f = fac ? fac->data() + (size_t)(bh / fac_group) * d : nullptr;
    std::vector<double> vals((size_t)BLK * d);
    for (int blk = 0; blk < nb; ++blk) {
      const int n0 = blk * BLK, rows = std::min(BLK, N - n0);
      for (int r = 0; r < rows; ++r)
        for (int ch = 0; ch < d; ++ch) {
          const double v = bf16_to_double(xb[(size_t)(n0 + r) * d + ch]);
          double val = smooth ? M.F(v - mu[ch]) : v;
          if (f) val = M.F(val * f[ch]);
          vals[(size_t)r * d + ch] = val;
          if (keep_vals) out.val[((size_t)bh * N + n0 + r) * d + ch] = val;
        }
      if (block_smooth) {
        double* bm = &out.bmean[((size_t)bh * nb + blk) * d];
        for (int ch = 0; ch < d; ++ch) {
          double sum = 0;
          for (int r = 0; r < rows; ++r) sum += vals[(size_t)r * d + ch];
          bm[ch] = M.F(sum / (double)rows);
        }
        for (int r = 0; r < rows; ++r)
          for (int ch = 0; ch < d; ++ch) vals[(size_t)r * d + ch] = M.F(vals[(size_t)r * d + ch] - bm[ch]);
      }
      quant_block(M, which, vals.data(), rows * d, &out.codes[((size_t)bh * N + n0) * d], &out.scale[(size_t)bh * nb + blk],
                  d, subexp);
    }
  }
}

// floor(a / 2) for any sign of a.
inline int floor_half(int a) { return a >= 0 ? a / 2 : -((1 - a) / 2); }

// Channel balancing exponents, one per (batch, kv head, channel) [B*Hkv][d]
// (the library's reading, after SmoothQuant's migration of magnitude from
// activations to weights): with
//   aQ = max |Q| of the channel over the G query heads of the kv head and
//        all N tokens,
//   aK = max |K'| of the channel over all N tokens, K' the K the quantizer
//        sees (K minus its FP32 channel mean, rounded to FP32, when smoothing),
// the exponent is e = floor((E(aQ) - E(aK)) / 2), E(a) = floor(log2 a) (the
// binary exponent), clamped to [-126, 126] so that 2^e and 2^-e are normal
// FP32 numbers, and 0 when aQ or aK is zero.  Scaling Q by 2^-e and K' by 2^e
// leaves both channel maxima within a factor 4 of sqrt(aQ * aK).
std::vector<int> balance_exponents(const Mode& M, const oracle_problem* p, const uint16_t* q, const uint16_t* k) {
  const int N = p->N, d = p->d, G = p->Hq / p->Hkv, BHk = p->B * p->Hkv;
  std::vector<int> e((size_t)BHk * d, 0);
#pragma omp parallel for schedule(dynamic)
  for (int bhk = 0; bhk < BHk; ++bhk) {
    const uint16_t* kb = k + (size_t)bhk * N * d;
    std::vector<double> mu(d, 0.0);
    if (p->smooth_k) channel_mean(M, kb, N, d, mu.data());
    const int b = bhk / p->Hkv, hk = bhk % p->Hkv;
    for (int ch = 0; ch < d; ++ch) {
      double ak = 0, aq = 0;
      for (int n = 0; n < N; ++n) {
        const double v = bf16_to_double(kb[(size_t)n * d + ch]);
        ak = std::max(ak, std::fabs(p->smooth_k ? M.F(v - mu[ch]) : v));
      }
      for (int h = hk * G; h < (hk + 1) * G; ++h) {
        const uint16_t* qb = q + ((size_t)b * p->Hq + h) * N * d;
        for (int n = 0; n < N; ++n) aq = std::max(aq, std::fabs(bf16_to_double(qb[(size_t)n * d + ch])));
      }
      if (aq > 0 && ak > 0) {
        int eq = 0, ek = 0;
        std::frexp(aq, &eq);  // a = m 2^E with m in [0.5, 1): floor(log2 a) = E - 1 on both sides
        std::frexp(ak, &ek);
        e[(size_t)bhk * d + ch] = std::min(126, std::max(-126, floor_half(eq - ek)));
      }
    }
  }
  return e;
}

// Q and K as the attention consumes them: Q plain, K smoothed (smooth_k), both
// channel-balanced (balance_qk).  fq / fk (optional) receive the per
// (b, kv head, channel) factors 2^-e and 2^e (all 1 without balancing).
void quantize_qk(const Mode& M, const oracle_problem* p, const uint16_t* q, const uint16_t* k, QTensor& qq,
                 QTensor& kq, std::vector<int>* exps = nullptr, std::vector<double>* fq = nullptr,
                 std::vector<double>* fk = nullptr) {
  const size_t nf = (size_t)p->B * p->Hkv * p->d;
  std::vector<int> e = p->balance_qk ? balance_exponents(M, p, q, k) : std::vector<int>(nf, 0);
  std::vector<double> f_q(nf), f_k(nf);
  for (size_t i = 0; i < nf; ++i) {
    f_q[i] = std::ldexp(1.0, -e[i]);
    f_k[i] = std::ldexp(1.0, e[i]);
  }
  const int G = p->Hq / p->Hkv;
  quantize_tensor(M, QZ_Q, q, p->B * p->Hq, p->N, p->d, false, qq, p->balance_qk ? &f_q : nullptr, G,
                  p->qk_subexp != 0, p->smooth_q != 0);
  quantize_tensor(M, QZ_K, k, p->B * p->Hkv, p->N, p->d, p->smooth_k != 0, kq, p->balance_qk ? &f_k : nullptr, 1,
                  p->qk_subexp != 0, false, p->smooth_q != 0);
  if (exps) *exps = std::move(e);
  if (fq) *fq = std::move(f_q);
  if (fk) *fk = std::move(f_k);
}

inline bool visible(const oracle_problem* p, int i, int k) { return k < p->N && (!p->causal || k <= i); }

// Q-smoothing's correction of S for query block ib and key k, in base 2:
// c0 * (mean_Q(ib) . K'_k), the dot product in FP64 rounded to FP32 (K' the
// unquantized K the quantizer saw); 0 without Q-smoothing.
inline double qsmooth_bias(const Mode& M, const oracle_problem* p, const QTensor& qq, const QTensor& kq, int bhq,
                           int ib, int bhk, int k, double c0) {
  if (!p->smooth_q) return 0.0;
  double b = 0;
  for (int ch = 0; ch < p->d; ++ch) b += qq.bm(bhq, ib, ch) * kq.v(bhk, k, ch);
  return M.F(M.F(b) * c0);
}

// Base-2 logits of one query row against one 128-key tile:
// t_k = S_int * (sQ sK) * (scale log2 e) with S_int = Q^_i . K^_k, the row's
// FP32 logit of S = Q K^T; -inf where the key is masked.  Returns the tile's
// row maximum (-inf when every key of the tile is masked).
double fwd_tile_logits(const Mode& M, const oracle_problem* p, const QTensor& qq, const QTensor& kq, int b, int h,
                       int i, int jb, double c0, double* t /* indexed by key */) {
  const int N = p->N, d = p->d, G = p->Hq / p->Hkv, hk = h / G;
  const int bhq = b * p->Hq + h, bhk = b * p->Hkv + hk, ib = i / BLK;
  const double qks = M.F(M.F(qq.s(bhq, ib) * kq.s(bhk, jb)) * c0);
  double tmax = -kInf;
  for (int k = jb * BLK; k < std::min(N, (jb + 1) * BLK); ++k) {
    if (!visible(p, i, k)) {
      t[k] = -kInf;
      continue;
    }
    double s = 0;
    for (int ch = 0; ch < d; ++ch) s += qq.c(bhq, i, ch) * kq.c(bhk, k, ch);
    t[k] = M.F(M.F(s * qks) + qsmooth_bias(M, p, qq, kq, bhq, ib, bhk, k, c0));
    tmax = std::max(tmax, t[k]);
  }
  return tmax;
}

// Code of P~ for one key: rint(127 * 2^(t - tmax)), tmax the row maximum of its tile.
inline double fwd_p_code(const Mode& M, double t, double tmax) {
  return M.Q(QZ_PF, M.F(M.qmax * M.F(std::exp2(M.F(t - tmax)))));
}

// Forward of the quantized algorithm for query row i of head h, written as the
// definition rather than as the online recurrence: the per-tile quantization
// of P~ depends only on the tile's own row maximum, so the result equals what
// an online-softmax kernel computes for any order of the key tiles.
//   O_i = sum_j 2^(tmax_j - m)/127 * sV_j * sum_{k in j} code(P~)_k V^_k  /  l
//   l   = sum_k 2^(t_k - m)   (unquantized P~),   m = max_j tmax_j
//   LSE = (m + log2 l) ln 2
void fwd_row(const Mode& M, const oracle_problem* p, const QTensor& qq, const QTensor& kq, const QTensor& vq, int b,
             int h, int i, double c0, double* o_row, double* lse_out, std::vector<double>& t, std::vector<double>& acc) {
  const int N = p->N, d = p->d, G = p->Hq / p->Hkv, hk = h / G, nb = nblocks(N);
  const int bhk = b * p->Hkv + hk;
  const int jb_end = p->causal ? i / BLK : nb - 1;
  std::vector<double> tmax(jb_end + 1, -kInf);
  for (int jb = 0; jb <= jb_end; ++jb) tmax[jb] = fwd_tile_logits(M, p, qq, kq, b, h, i, jb, c0, t.data());
  double m = -kInf;
  for (int jb = 0; jb <= jb_end; ++jb) m = std::max(m, tmax[jb]);
  double l = 0;
  if (p->l_from_codes) {
    // the misreading the tests plant: l from the codes, sum_j 2^(tmax_j - m)/127 * sum_k code_k
    for (int jb = 0; jb <= jb_end; ++jb) {
      if (tmax[jb] == -kInf) continue;
      double cs = 0;
      for (int k = jb * BLK; k < std::min(N, (jb + 1) * BLK); ++k)
        if (t[k] != -kInf) cs += fwd_p_code(M, t[k], tmax[jb]);
      l += std::exp2(tmax[jb] - m) / M.qmax * cs;
    }
  } else {
    for (int k = 0; k < std::min(N, (jb_end + 1) * BLK); ++k)
      if (t[k] != -kInf) l += std::exp2(t[k] - m);
  }
  std::fill(acc.begin(), acc.end(), 0.0);
  for (int jb = 0; jb <= jb_end; ++jb) {
    if (tmax[jb] == -kInf) continue;
    const double w = std::exp2(tmax[jb] - m) / M.qmax * vq.s(bhk, jb);
    for (int ch = 0; ch < d; ++ch) {
      double s = 0;
      for (int k = jb * BLK; k < std::min(N, (jb + 1) * BLK); ++k) {
        if (t[k] == -kInf) continue;
        s += fwd_p_code(M, t[k], tmax[jb]) * vq.c(bhk, k, ch);
      }
      acc[ch] += w * s;
    }
  }
  for (int ch = 0; ch < d; ++ch) o_row[ch] = acc[ch] / l;
  *lse_out = (m + std::log2(l)) * kLn2;
}

void fwd_impl(const oracle_problem* p, const uint16_t* q, const uint16_t* k, const uint16_t* v, double* o, double* lse,
              const uint8_t* qsel) {
  const Mode M = mode_of(p);
  QTensor qq, kq, vq;
  quantize_qk(M, p, q, k, qq, kq);
  quantize_tensor(M, QZ_V, v, p->B * p->Hkv, p->N, p->d, false, vq);
  const double c0 = M.F(scale_of(p) * kLog2e);
  const int N = p->N, d = p->d, nb = nblocks(N);
  const long rows = (long)p->B * p->Hq * N;
#pragma omp parallel
  {
    std::vector<double> t(N), acc(d);
#pragma omp for schedule(dynamic, 16)
    for (long r = 0; r < rows; ++r) {
      const int i = (int)(r % N);
      const int bh = (int)(r / N);
      if (qsel && !qsel[(size_t)bh * nb + i / BLK]) continue;
      fwd_row(M, p, qq, kq, vq, bh / p->Hq, bh % p->Hq, i, c0, o + (size_t)r * d, lse + r, t, acc);
    }
  }
}

// One 128 x 128 backward tile (query block ib, key block jb, query head h):
// everything that the three quantized backward products of the tile consume.
struct BwdTile {
  int i0 = 0, k0 = 0, ni = 0, nk = 0;
  std::vector<double> pt;   // code(P^T)[k][i]
  std::vector<double> spc;  // scale of row k of P^T
  std::vector<double> ds;   // code(dS)[i][k]
  double sds = 0;                       // scale of the dS tile
};

// dS sub-scales (the library's reading, ds_subexp): the tile's codes keep the
// one FP32 scale max|dS| / 127, and each key's codes within a group of
// kSubGroup consecutive queries of the tile are refined by 2^k, k = the
// largest integer <= log2(tile max / group max), at most kSubMax, 0 when the
// group max is below 2^-100: code = rint(dS * inv * 2^k), value = code * 2^-k
// (exact in BF16: a 7-bit integer times a power of two).  Both products that
// read dS (dK = dS^T Q, dQ = dS K) use these values, so the sub-scale needs no
// dequantization step of its own.
constexpr int kSubGroup = 32;
int ds_subexp_of(const std::vector<double>& dS, int ni, int a0, int c, double amax) {
  double g = 0;
  for (int a = a0; a < std::min(ni, a0 + kSubGroup); ++a) g = std::max(g, std::fabs(dS[(size_t)a * BLK + c]));
  return subexp_of(amax, g);
}

void bwd_tile(const Mode& M, const oracle_problem* p, const QTensor& qq, const QTensor& kq, const uint16_t* v,
              const uint16_t* dO, const double* o, const double* lse, int b, int h, int ib, int jb, double c0,
              double l2e, BwdTile& T, const QTensor* doq = nullptr, const QTensor* vq = nullptr) {
  const int N = p->N, d = p->d, G = p->Hq / p->Hkv, hk = h / G;
  const int bhq = b * p->Hq + h, bhk = b * p->Hkv + hk;
  T.i0 = ib * BLK;
  T.k0 = jb * BLK;
  T.ni = std::min(BLK, N - T.i0);
  T.nk = std::min(BLK, N - T.k0);
  std::vector<double> P((size_t)BLK * BLK, 0.0), dS((size_t)BLK * BLK, 0.0);
  const double qks = M.F(M.F(qq.s(bhq, ib) * kq.s(bhk, jb)) * c0);
  for (int a = 0; a < T.ni; ++a) {
    const int i = T.i0 + a;
    const size_t qrow = ((size_t)bhq * N + i) * d;
    double D = 0;  // D_i = rowsum(dO_i * O_i)
    for (int ch = 0; ch < d; ++ch) D += bf16_to_double(dO[qrow + ch]) * o[qrow + ch];
    const double L = M.F(M.F(lse[(size_t)bhq * N + i]) * l2e);  // LSE in base 2
    for (int c = 0; c < T.nk; ++c) {
      const int kk = T.k0 + c;
      if (!visible(p, i, kk)) continue;
      double s = 0;
      for (int ch = 0; ch < d; ++ch) s += qq.c(bhq, i, ch) * kq.c(bhk, kk, ch);
      const double tt = M.F(M.F(s * qks) + qsmooth_bias(M, p, qq, kq, bhq, ib, bhk, kk, c0));
      const double pp = M.F(std::exp2(M.F(tt - L)));  // normalized probability
      // dP = dO V^T: the product kept in high precision (BF16 inputs, FP64 sum here);
      // the int8_dp ablation takes it from the dO and V codes instead (the pages' ablation of
      // leaving this product unquantized, run the other way round).
      double dp = 0;
      if (doq && vq) {
        for (int ch = 0; ch < d; ++ch) dp += doq->c(bhq, i, ch) * vq->c(bhk, kk, ch);
        dp *= doq->s(bhq, ib) * vq->s(bhk, jb);
      } else {
        const size_t vrow = ((size_t)bhk * N + kk) * d;
        for (int ch = 0; ch < d; ++ch) dp += bf16_to_double(dO[qrow + ch]) * bf16_to_double(v[vrow + ch]);
      }
      P[(size_t)a * BLK + c] = pp;
      dS[(size_t)a * BLK + c] = M.F(pp * (dp - D));
    }
  }
  // P^T quantized per key row over the tile's queries.
  T.pt.assign((size_t)BLK * BLK, 0);
  T.spc.assign(BLK, 0.0);
  for (int c = 0; c < T.nk; ++c) {
    double cmax = 0;
    for (int a = 0; a < T.ni; ++a) cmax = std::max(cmax, P[(size_t)a * BLK + c]);
    if (cmax < M.min_group()) continue;
    const double inv = M.F(M.qmax / cmax);
    T.spc[c] = M.F(cmax / M.qmax);
    for (int a = 0; a < T.ni; ++a) T.pt[(size_t)c * BLK + a] = M.Q(QZ_PB, M.F(P[(size_t)a * BLK + c] * inv));
  }
  // dS quantized with one scale for the whole tile (and, with ds_subexp, a
  // power-of-two sub-scale per key and group of 32 queries).
  T.ds.assign((size_t)BLK * BLK, 0);
  double amax = 0;
  for (int a = 0; a < T.ni; ++a)
    for (int c = 0; c < T.nk; ++c) amax = std::max(amax, std::fabs(dS[(size_t)a * BLK + c]));
  T.sds = 0;
  if (amax >= M.min_group()) {
    const double inv = M.F(M.qmax / amax);
    T.sds = M.F(amax / M.qmax);
    for (int a = 0; a < T.ni; ++a)
      for (int c = 0; c < T.nk; ++c) {
        const double x = M.F(dS[(size_t)a * BLK + c] * inv);
        if (!p->ds_subexp) {
          T.ds[(size_t)a * BLK + c] = M.Q(QZ_DS, x);
        } else {
          const int k = ds_subexp_of(dS, T.ni, a / kSubGroup * kSubGroup, c, amax);
          const double f = std::ldexp(1.0, k);
          T.ds[(size_t)a * BLK + c] = M.Q(QZ_DS, x * f) / f;  // a code times 2^-k
        }
      }
  }
}

void bwd_impl(const oracle_problem* p, const uint16_t* q, const uint16_t* k, const uint16_t* v, const double* o,
              const uint16_t* dO, const double* lse, double* dq, double* dk, double* dv, const uint8_t* qsel,
              const uint8_t* ksel) {
  const Mode M = mode_of(p);
  QTensor qq, kq, dq8, vq;
  std::vector<double> fq, fk;  // channel balancing factors, undone on dQ and dK at the end
  quantize_qk(M, p, q, k, qq, kq, nullptr, &fq, &fk);
  quantize_tensor(M, QZ_DO, dO, p->B * p->Hq, p->N, p->d, false, dq8);
  if (p->int8_dp) quantize_tensor(M, QZ_V, v, p->B * p->Hkv, p->N, p->d, false, vq);
  const QTensor* dp_do = p->int8_dp ? &dq8 : nullptr;
  const QTensor* dp_v = p->int8_dp ? &vq : nullptr;
  const double sc = scale_of(p);
  const double c0 = M.F(sc * kLog2e);
  const double l2e = M.F(kLog2e);
  const int N = p->N, d = p->d, nb = nblocks(N), G = p->Hq / p->Hkv;
  // dK, dV: one task per (b, kv head, key block), summed over the G query heads.
  const long ktasks = (long)p->B * p->Hkv * nb;
#pragma omp parallel
  {
    BwdTile T;
    std::vector<double> accv((size_t)BLK * d), acck((size_t)BLK * d);
#pragma omp for schedule(dynamic)
    for (long task = 0; task < ktasks; ++task) {
      if (ksel && !ksel[task]) continue;
      const int jb = (int)(task % nb), bhk = (int)(task / nb), b = bhk / p->Hkv, hk = bhk % p->Hkv;
      std::fill(accv.begin(), accv.end(), 0.0);
      std::fill(acck.begin(), acck.end(), 0.0);
      for (int h = hk * G; h < (hk + 1) * G; ++h) {
        const int bhq = b * p->Hq + h;
        for (int ib = p->causal ? jb : 0; ib < nb; ++ib) {
          bwd_tile(M, p, qq, kq, v, dO, o, lse, b, h, ib, jb, c0, l2e, T, dp_do, dp_v);
          for (int c = 0; c < T.nk; ++c)
            for (int ch = 0; ch < d; ++ch) {
              double sv = 0, sk = 0;
              for (int a = 0; a < T.ni; ++a) {
                sv += T.pt[(size_t)c * BLK + a] * dq8.c(bhq, T.i0 + a, ch);  // P^T dO
                sk += T.ds[(size_t)a * BLK + c] * qq.c(bhq, T.i0 + a, ch);   // dS^T Q
              }
              accv[(size_t)c * d + ch] += T.spc[c] * dq8.s(bhq, ib) * sv;
              acck[(size_t)c * d + ch] += sc * T.sds * qq.s(bhq, ib) * sk;
            }
          if (p->smooth_q)  // dK = dS^T (Q_s + mean_Q): the block mean's share, from the same dS values
            for (int c = 0; c < T.nk; ++c) {
              double colsum = 0;
              for (int a = 0; a < T.ni; ++a) colsum += T.ds[(size_t)a * BLK + c];
              for (int ch = 0; ch < d; ++ch) acck[(size_t)c * d + ch] += sc * T.sds * colsum * qq.bm(bhq, ib, ch);
            }
        }
      }
      for (int c = 0; c < std::min(BLK, N - jb * BLK); ++c)
        for (int ch = 0; ch < d; ++ch) {
          const size_t idx = ((size_t)bhk * N + jb * BLK + c) * d + ch;
          dv[idx] = accv[(size_t)c * d + ch];
          dk[idx] = acck[(size_t)c * d + ch] * fk[(size_t)bhk * d + ch];  // dK = dS^T (Q 2^-e) 2^e
        }
    }
  }
  // dQ: one task per (b, query head, query block).
  const long qtasks = (long)p->B * p->Hq * nb;
#pragma omp parallel
  {
    BwdTile T;
    std::vector<double> accq((size_t)BLK * d);
#pragma omp for schedule(dynamic)
    for (long task = 0; task < qtasks; ++task) {
      if (qsel && !qsel[task]) continue;
      const int ib = (int)(task % nb), bhq = (int)(task / nb), b = bhq / p->Hq, h = bhq % p->Hq;
      const int bhk = b * p->Hkv + h / G;
      std::fill(accq.begin(), accq.end(), 0.0);
      for (int jb = 0; jb <= (p->causal ? ib : nb - 1); ++jb) {
        bwd_tile(M, p, qq, kq, v, dO, o, lse, b, h, ib, jb, c0, l2e, T, dp_do, dp_v);
        for (int a = 0; a < T.ni; ++a)
          for (int ch = 0; ch < d; ++ch) {
            double s = 0;
            for (int c = 0; c < T.nk; ++c) s += T.ds[(size_t)a * BLK + c] * kq.c(bhk, T.k0 + c, ch);  // dS K
            accq[(size_t)a * d + ch] += sc * T.sds * kq.s(bhk, jb) * s;
          }
      }
      for (int a = 0; a < std::min(BLK, N - ib * BLK); ++a)
        for (int ch = 0; ch < d; ++ch)  // dQ = dS (K' 2^e) 2^-e
          dq[((size_t)bhq * N + ib * BLK + a) * d + ch] = accq[(size_t)a * d + ch] * fq[(size_t)bhk * d + ch];
    }
  }
}

}  // namespace

extern "C" {

int oracle_check_problem(const oracle_problem* p) {
  if (!p || p->B < 1 || p->Hq < 1 || p->Hkv < 1 || p->N < 1 || p->d < 1) return 1;
  if (p->Hq % p->Hkv != 0) return 1;
  if (p->fp8 && (p->ds_subexp || p->qk_subexp)) return 1;  // sub-scales are defined for INT8 codes
  if (p->smooth_q && p->balance_qk) return 1;               // not defined together
  return 0;
}

// Quantize one BF16 tensor [BH][N][d]: integer codes (int8), FP32 block scales
// [BH][ceil(N/128)], and (smooth only) the FP32 channel means [BH][d].
int oracle_quantize(const oracle_problem* p, const uint16_t* x, int BH, int smooth, int8_t* codes, float* scales,
                    float* mean) {
  if (oracle_check_problem(p)) return 1;
  set_threads(p);
  QTensor qt;
  quantize_tensor(Mode{true, 0}, QZ_Q, x, BH, p->N, p->d, smooth != 0, qt);
  for (size_t e = 0; e < qt.codes.size(); ++e) codes[e] = (int8_t)qt.codes[e];
  for (size_t e = 0; e < qt.scale.size(); ++e) scales[e] = (float)qt.scale[e];
  if (smooth && mean)
    for (size_t e = 0; e < qt.mean.size(); ++e) mean[e] = (float)qt.mean[e];
  return 0;
}

// Same, without rounding: codes are x/s as FP64 (exact_codes pipeline), for pins.
int oracle_quantize_exact(const oracle_problem* p, const uint16_t* x, int BH, int smooth, double* codes,
                          double* scales, double* mean) {
  if (oracle_check_problem(p)) return 1;
  set_threads(p);
  QTensor qt;
  quantize_tensor(Mode{false, 0x7Fu}, QZ_Q, x, BH, p->N, p->d, smooth != 0, qt);
  std::copy(qt.codes.begin(), qt.codes.end(), codes);
  std::copy(qt.scale.begin(), qt.scale.end(), scales);
  if (smooth && mean) std::copy(qt.mean.begin(), qt.mean.end(), mean);
  return 0;
}

// Q and K as the forward quantizes them (K-smoothing, channel balancing and
// sub-scales as the problem selects): the operand values (integer codes, or
// code * 2^-k with qk_subexp) as FP32, FP32 block scales, the FP32 K channel
// means [B*Hkv][d] (smooth_k) and the balancing exponents [B*Hkv][d] (all 0
// unless balance_qk).  mean and exps may be NULL.
int oracle_quantize_qk(const oracle_problem* p, const uint16_t* q, const uint16_t* k, float* qc, float* qs,
                       float* kc, float* ks, float* mean, int32_t* exps) {
  if (oracle_check_problem(p)) return 1;
  set_threads(p);
  QTensor qq, kq;
  std::vector<int> e;
  Mode M{true, 0};
  M.bf16 = p->bf16_mask & ((1u << QZ_Q) | (1u << QZ_K));  // the attribution mode, where it applies to Q and K
  if (p->fp8) {  // the FP8 variant's E4M3 values
    M.fp8 = true;
    M.qmax = 448.0;
  }
  quantize_qk(M, p, q, k, qq, kq, &e);
  for (size_t i = 0; i < qq.codes.size(); ++i) qc[i] = (float)qq.codes[i];
  for (size_t i = 0; i < qq.scale.size(); ++i) qs[i] = (float)qq.scale[i];
  for (size_t i = 0; i < kq.codes.size(); ++i) kc[i] = (float)kq.codes[i];
  for (size_t i = 0; i < kq.scale.size(); ++i) ks[i] = (float)kq.scale[i];
  if (mean && p->smooth_k)
    for (size_t i = 0; i < kq.mean.size(); ++i) mean[i] = (float)kq.mean[i];
  if (exps)
    for (size_t i = 0; i < e.size(); ++i) exps[i] = e[i];
  return 0;
}

// Q-smoothing's quantities as the forward uses them (smooth_q problems): the FP32 block
// means of Q [B*Hq][nb][d] and the base-2 logit terms [B*Hq][nb][N] of qsmooth_bias.
int oracle_qsmooth_terms(const oracle_problem* p, const uint16_t* q, const uint16_t* k, float* qmean, float* bias) {
  if (oracle_check_problem(p) || !p->smooth_q) return 1;
  set_threads(p);
  const Mode M = mode_of(p);
  QTensor qq, kq;
  quantize_qk(M, p, q, k, qq, kq);
  const double c0 = M.F(scale_of(p) * kLog2e);
  const int N = p->N, nb = nblocks(N), G = p->Hq / p->Hkv;
  for (size_t i = 0; i < qq.bmean.size(); ++i) qmean[i] = (float)qq.bmean[i];
#pragma omp parallel for schedule(dynamic)
  for (int bhq = 0; bhq < p->B * p->Hq; ++bhq) {
    const int bhk = (bhq / p->Hq) * p->Hkv + (bhq % p->Hq) / G;
    for (int ib = 0; ib < nb; ++ib)
      for (int key = 0; key < N; ++key)
        bias[((size_t)bhq * nb + ib) * N + key] = (float)qsmooth_bias(M, p, qq, kq, bhq, ib, bhk, key, c0);
  }
  return 0;
}

// Quantized forward.  o: FP64 [B][Hq][N][d]; lse: FP64 [B][Hq][N] (natural log).
// qsel (optional): [B*Hq][ceil(N/128)] flags; unselected query blocks are not written.
int oracle_fwd(const oracle_problem* p, const uint16_t* q, const uint16_t* k, const uint16_t* v, double* o,
               double* lse, const uint8_t* qsel) {
  if (oracle_check_problem(p)) return 1;
  set_threads(p);
  fwd_impl(p, q, k, v, o, lse, qsel);
  return 0;
}

// Quantized backward.  o: the forward output as FP64 values (the caller passes
// the forward's result, rounded to BF16 when it mirrors the library's call);
// lse: the forward's LSE.  qsel selects the dQ query blocks [B*Hq][nb], ksel
// the dK/dV key blocks [B*Hkv][nb]; NULL selects all.
int oracle_bwd(const oracle_problem* p, const uint16_t* q, const uint16_t* k, const uint16_t* v, const double* o,
               const uint16_t* dO, const double* lse, double* dq, double* dk, double* dv, const uint8_t* qsel,
               const uint8_t* ksel) {
  if (oracle_check_problem(p)) return 1;
  set_threads(p);
  bwd_impl(p, q, k, v, o, dO, lse, dq, dk, dv, qsel, ksel);
  return 0;
}

// Exact FP64 softmax attention (the full-precision reference for the cosine
// similarity criteria): S = scale * Q K^T, P = softmax(S), O = P V.
int oracle_exact_fwd(const oracle_problem* p, const uint16_t* q, const uint16_t* k, const uint16_t* v, double* o,
                     double* lse, const uint8_t* qsel) {
  if (oracle_check_problem(p)) return 1;
  set_threads(p);
  const int N = p->N, d = p->d, G = p->Hq / p->Hkv, nb = nblocks(N);
  const double sc = scale_of(p);
  const long rows = (long)p->B * p->Hq * N;
#pragma omp parallel
  {
    std::vector<double> s(N);
#pragma omp for schedule(dynamic, 16)
    for (long r = 0; r < rows; ++r) {
      const int i = (int)(r % N), bhq = (int)(r / N), b = bhq / p->Hq, h = bhq % p->Hq;
      if (qsel && !qsel[(size_t)bhq * nb + i / BLK]) continue;
      const int bhk = b * p->Hkv + h / G;
      double m = -kInf;
      for (int kk = 0; kk < N; ++kk) {
        if (!visible(p, i, kk)) continue;
        double acc = 0;
        for (int ch = 0; ch < d; ++ch)
          acc += bf16_to_double(q[(size_t)r * d + ch]) * bf16_to_double(k[((size_t)bhk * N + kk) * d + ch]);
        s[kk] = sc * acc;
        m = std::max(m, s[kk]);
      }
      double l = 0;
      for (int kk = 0; kk < N; ++kk) {
        s[kk] = visible(p, i, kk) ? std::exp(s[kk] - m) : 0.0;  // unnormalized probability
        l += s[kk];
      }
      for (int ch = 0; ch < d; ++ch) {
        double acc = 0;
        for (int kk = 0; kk < N; ++kk) acc += s[kk] * bf16_to_double(v[((size_t)bhk * N + kk) * d + ch]);
        o[(size_t)r * d + ch] = acc / l;
      }
      lse[r] = m + std::log(l);
    }
  }
  return 0;
}

// Exact FP64 attention backward given the exact forward's O and LSE:
// P = exp(S - LSE), dV = P^T dO, dP = dO V^T, D = rowsum(dO * O),
// dS = P * (dP - D), dQ = scale * dS K, dK = scale * dS^T Q (GQA: summed over
// the query heads that share a kv head).
int oracle_exact_bwd(const oracle_problem* p, const uint16_t* q, const uint16_t* k, const uint16_t* v,
                     const double* o, const uint16_t* dO, const double* lse, double* dq, double* dk, double* dv,
                     const uint8_t* qsel, const uint8_t* ksel) {
  if (oracle_check_problem(p)) return 1;
  set_threads(p);
  const int N = p->N, d = p->d, G = p->Hq / p->Hkv, nb = nblocks(N);
  const double sc = scale_of(p);
  // D_i = rowsum(dO_i * O_i) for every query row.
  std::vector<double> Dv((size_t)p->B * p->Hq * N);
#pragma omp parallel for schedule(static)
  for (long r = 0; r < (long)Dv.size(); ++r) {
    double D = 0;
    for (int ch = 0; ch < d; ++ch) D += bf16_to_double(dO[(size_t)r * d + ch]) * o[(size_t)r * d + ch];
    Dv[r] = D;
  }
  auto Dval = [&](int bhq, int i) { return Dv[(size_t)bhq * N + i]; };
  auto P_dS = [&](int bhq, int bhk, int i, int kk, double D, double* Pout) {
    double s = 0, dp = 0;
    for (int ch = 0; ch < d; ++ch) {
      s += bf16_to_double(q[((size_t)bhq * N + i) * d + ch]) * bf16_to_double(k[((size_t)bhk * N + kk) * d + ch]);
      dp += bf16_to_double(dO[((size_t)bhq * N + i) * d + ch]) * bf16_to_double(v[((size_t)bhk * N + kk) * d + ch]);
    }
    const double P = std::exp(sc * s - lse[(size_t)bhq * N + i]);
    *Pout = P;
    return P * (dp - D);
  };
  const long krows = (long)p->B * p->Hkv * N;
#pragma omp parallel
  {
    std::vector<double> av(d), ak(d);
#pragma omp for schedule(dynamic, 16)
    for (long r = 0; r < krows; ++r) {
      const int kk = (int)(r % N), bhk = (int)(r / N), b = bhk / p->Hkv, hk = bhk % p->Hkv;
      if (ksel && !ksel[(size_t)bhk * nb + kk / BLK]) continue;
      std::fill(av.begin(), av.end(), 0.0);
      std::fill(ak.begin(), ak.end(), 0.0);
      for (int h = hk * G; h < (hk + 1) * G; ++h) {
        const int bhq = b * p->Hq + h;
        for (int i = 0; i < N; ++i) {
          if (!visible(p, i, kk)) continue;
          double P;
          const double dS = P_dS(bhq, bhk, i, kk, Dval(bhq, i), &P);
          for (int ch = 0; ch < d; ++ch) {
            av[ch] += P * bf16_to_double(dO[((size_t)bhq * N + i) * d + ch]);
            ak[ch] += sc * dS * bf16_to_double(q[((size_t)bhq * N + i) * d + ch]);
          }
        }
      }
      for (int ch = 0; ch < d; ++ch) {
        dv[(size_t)r * d + ch] = av[ch];
        dk[(size_t)r * d + ch] = ak[ch];
      }
    }
  }
  const long qrows = (long)p->B * p->Hq * N;
#pragma omp parallel
  {
    std::vector<double> aq(d);
#pragma omp for schedule(dynamic, 16)
    for (long r = 0; r < qrows; ++r) {
      const int i = (int)(r % N), bhq = (int)(r / N), b = bhq / p->Hq, h = bhq % p->Hq;
      if (qsel && !qsel[(size_t)bhq * nb + i / BLK]) continue;
      const int bhk = b * p->Hkv + h / G;
      const double D = Dval(bhq, i);
      std::fill(aq.begin(), aq.end(), 0.0);
      for (int kk = 0; kk < N; ++kk) {
        if (!visible(p, i, kk)) continue;
        double P;
        const double dS = P_dS(bhq, bhk, i, kk, D, &P);
        for (int ch = 0; ch < d; ++ch) aq[ch] += sc * dS * bf16_to_double(k[((size_t)bhk * N + kk) * d + ch]);
      }
      for (int ch = 0; ch < d; ++ch) dq[(size_t)r * d + ch] = aq[ch];
    }
  }
  return 0;
}

// Codes of P~ of one forward tile (query block ib, key block jb, head h):
// codes [128][128] (row = query ib*128+a, col = key jb*128+c; 0 where masked
// or outside N) and the tile's row maxima tmax [128] (base-2 logits; -inf
// where the row sees no key or lies outside N).
int oracle_fwd_tile(const oracle_problem* p, const uint16_t* q, const uint16_t* k, int b, int h, int ib, int jb,
                    int32_t* codes, double* tmax) {
  if (oracle_check_problem(p) || p->exact_codes) return 1;
  set_threads(p);
  const Mode M = mode_of(p);
  QTensor qq, kq;
  quantize_qk(M, p, q, k, qq, kq);
  const double c0 = M.F(scale_of(p) * kLog2e);
  std::vector<double> t(p->N);
  for (int a = 0; a < BLK; ++a) {
    const int i = ib * BLK + a;
    tmax[a] = -kInf;
    for (int c = 0; c < BLK; ++c) codes[a * BLK + c] = 0;
    if (i >= p->N) continue;
    tmax[a] = fwd_tile_logits(M, p, qq, kq, b, h, i, jb, c0, t.data());
    for (int c = 0; c < BLK; ++c) {
      const int kk = jb * BLK + c;
      if (kk < p->N && t[kk] != -kInf) codes[a * BLK + c] = (int32_t)fwd_p_code(M, t[kk], tmax[a]);
    }
  }
  return 0;
}

// Everything the quantized backward of one tile consumes: pt [128][128] codes
// of P^T (row = key), spc [128] their per-key scales, ds [128][128] the dS
// operand values (row = query): integer codes, or code * 2^-k with ds_subexp,
// *sds the tile's dS scale.  o, lse: the forward's outputs.
int oracle_bwd_tile(const oracle_problem* p, const uint16_t* q, const uint16_t* k, const uint16_t* v, const double* o,
                    const uint16_t* dO, const double* lse, int b, int h, int ib, int jb, int32_t* pt, double* spc,
                    double* ds, double* sds) {
  if (oracle_check_problem(p) || p->exact_codes) return 1;
  set_threads(p);
  const Mode M = mode_of(p);
  QTensor qq, kq;
  quantize_qk(M, p, q, k, qq, kq);
  BwdTile T;
  bwd_tile(M, p, qq, kq, v, dO, o, lse, b, h, ib, jb, M.F(scale_of(p) * kLog2e), M.F(kLog2e), T);
  for (size_t e = 0; e < T.pt.size(); ++e) pt[e] = (int32_t)T.pt[e];
  std::copy(T.spc.begin(), T.spc.end(), spc);
  std::copy(T.ds.begin(), T.ds.end(), ds);  // integer codes; with ds_subexp code * 2^-k
  *sds = T.sds;
  return 0;
}

// FP8 E4M3 rounding of n values (the fp8 ablation's element rounding), for pins.
int oracle_round_e4m3(const double* x, double* y, int64_t n) {
  for (int64_t i = 0; i < n; ++i) y[i] = round_e4m3(x[i]);
  return 0;
}

int oracle_max_threads(void) {
#ifdef _OPENMP
  return omp_get_max_threads();
#else
  return 1;
#endif
}

}  // extern "C"
