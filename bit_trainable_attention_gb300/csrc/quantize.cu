// HBM-bound kernels of the SageBwd path: the K channel mean, the per-block
// absmax INT8 quantizer (Q, K, V and dO), the backward preprocess
// (D = rowsum(dO * O) with the dO quantization) and the FP32 -> BF16 dQ
// conversion.  Loads and stores are 16-byte vectors along d; one CTA owns one
// 128-token block of one head, so the block's absmax never leaves the CTA.
//
// Quantizer ("SageBwd: A Trainable Low-bit Attention", Abstract: INT8
// attention with K-smoothing; the block size and scale rule are this
// library's reading): a = max|x| over a 128 x d block, inv = 127/a and
// s = a/127 in IEEE FP32, code = clamp(rint(x * inv), -127, 127); a block
// whose max is below 2^-120 (zero, or so small that 127/a would overflow)
// gives codes 0 and s = 0.  K first subtracts its channel mean over all
// N tokens, summed in FP64 in a fixed order (deterministic) and rounded once
// to FP32.
//
// Optional channel balancing (the library's addition, after SmoothQuant,
// listed under "Builds on" of the SageBwd page): per (batch, kv head, channel)
// e = clamp(floor((E(aQ) - E(aK)) / 2), -126, 126), E the binary exponent of
// the channel's max |Q| over the kv head's query heads and of its max
// |K - mean|; Q's channel is multiplied by 2^-e and K's by 2^e (one exact FP32
// multiply, after the smoothing) before the block quantizer.
#include "ptx.cuh"
#include "sagebwd_internal.h"

namespace sagebwd {
namespace {

constexpr int kThreads = 256;

__device__ __forceinline__ void unpack8(const uint4& u, float (&f)[8]) {
  const uint32_t w[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
  for (int e = 0; e < 4; ++e) {
    f[2 * e] = __uint_as_float(w[e] << 16);
    f[2 * e + 1] = __uint_as_float(w[e] & 0xFFFF0000u);
  }
}

// codes are integers in [-127, 127]: the BF16 conversion is exact
__device__ __forceinline__ uint32_t pack2(float a, float b) {
  __nv_bfloat162 h = __floats2bfloat162_rn(a, b);
  return *reinterpret_cast<uint32_t*>(&h);
}

__device__ __forceinline__ float quant_code(float x, float inv) {
  float c = rintf(__fmul_rn(x, inv));
  return fminf(127.f, fmaxf(-127.f, c));
}

// Block-wide max of non-negative values; every thread gets the result.
__device__ __forceinline__ float block_max(float v, float* red) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, o));
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  __syncthreads();  // red may still be read from a previous use
  if (lane == 0) red[warp] = v;
  __syncthreads();
  float m = red[0];
#pragma unroll
  for (int w = 1; w < kThreads / 32; ++w) m = fmaxf(m, red[w]);
  return m;
}

// 2^e as an FP32 number, for -126 <= e <= 127 (built from the IEEE 754 fields).
__device__ __forceinline__ float exp2_int(int e) { return __int_as_float((127 + e) << 23); }

// floor(log2 a) for a finite a > 0, read off the IEEE 754 fields (subnormals:
// the position of the leading mantissa bit).
__device__ __forceinline__ int binary_exponent(float a) {
  const uint32_t u = __float_as_uint(a);
  const int biased = (int)((u >> 23) & 0xFFu);
  return biased ? biased - 127 : (31 - __clz((int)u)) - 149;
}

// Exact channel sums of one thread's rows (u: RPL 16-byte vectors of 8 BF16
// channels; rows past N were loaded as zeros).  FP32 additions are checked
// with Knuth's error-free TwoSum (s = a + b, err = (a - (s - (s - a))) +
// (b - (s - a))); when none of them rounded, the FP32 sums are exact and only
// they are widened to FP64 -- FP64 is slow on this GPU.  A thread whose values
// span too wide a range for that re-sums its rows in FP64.  The result is the
// exact sum either way (for BF16 inputs of ordinary range, where the FP64
// additions that follow are exact too).
template <int RPL>
__device__ __forceinline__ void exact_row_sums(const uint4 (&u)[RPL], double (&acc)[8]) {
  float sum[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
  bool exact = true;
#pragma unroll
  for (int i = 0; i < RPL; ++i) {
    float f[8];
    unpack8(u[i], f);
#pragma unroll
    for (int e = 0; e < 8; ++e) {
      const float t = __fadd_rn(sum[e], f[e]);
      const float bv = __fsub_rn(t, sum[e]);
      const float err = __fadd_rn(__fsub_rn(sum[e], __fsub_rn(t, bv)), __fsub_rn(f[e], bv));
      exact = exact && (err == 0.f);
      sum[e] = t;
    }
  }
  if (exact) {
#pragma unroll
    for (int e = 0; e < 8; ++e) acc[e] = (double)sum[e];
  } else {
#pragma unroll
    for (int e = 0; e < 8; ++e) acc[e] = 0.0;
#pragma unroll
    for (int i = 0; i < RPL; ++i) {
      float f[8];
      unpack8(u[i], f);
#pragma unroll
      for (int e = 0; e < 8; ++e) acc[e] += (double)f[e];
    }
  }
}

// Quantize the 128 x D block (bh, blk) of one tensor.  V8 = D / 8 16-byte vectors per row;
// a thread keeps one 8-channel group (kThreads is a multiple of V8) over PER rows, holds
// the raw vectors in registers and unpacks them twice (absmax pass, code pass), which keeps
// the register count low enough for several CTAs per SM.
// fac (optional): the channel balancing factors of this head's channels, in shared memory.
// gred (non-null: Q/K sub-scales): shared scratch [kThreads / 32][D / 8] for the maxima of the
// 8-channel groups; each group's codes are then refined by 2^k (see below).
// BM (Q-smoothing): the block's own channel means are subtracted instead of a head-wide mean
// and written to bmean[bh][blk][D]; mred / smean are shared scratch [kThreads / 32][D] / [D]
// for them.
// vmode (uniform over the CTA): kValInt8 the codes as above; kValBf16 (error attribution) the block
// keeps its scale but stores the BF16 rounding (to nearest even) of x * inv instead of the code (no
// sub-scales); kValFp8 (the FP8 variant) scale = a/448, inv = 448/a and the stored value is the
// E4M3 rounding (to nearest even, saturating) of x * inv, held exactly in BF16.
// x8 / x8t (kValFp8 only, optional): the E4M3 values also as bytes, [BH][N][D] and transposed
// [BH][D][128 nb] (through the shared tile t8 [D][128]; zero past N).
template <int D, bool BM = false>
__device__ void quantize_block(const __nv_bfloat16* __restrict__ x, __nv_bfloat16* __restrict__ xq,
                               float* __restrict__ scale, const float* __restrict__ mean, int bh, int blk, int N,
                               int nb, float* red, const float* fac = nullptr, float* gred = nullptr,
                               float* __restrict__ bmean = nullptr, double* mred = nullptr, float* smean = nullptr,
                               int vmode = kValInt8, uint8_t* __restrict__ x8 = nullptr,
                               uint8_t* __restrict__ x8t = nullptr, uint8_t* t8 = nullptr) {
  constexpr int V8 = D / 8, RL = kThreads / V8;
  constexpr int PER = kBlk / RL;  // rows (16-byte vectors) per thread
  static_assert(kThreads % V8 == 0 && kBlk % RL == 0, "thread layout");
  const int row0 = blk * kBlk;
  const size_t base = ((size_t)bh * N + row0) * D;
  const int c8 = threadIdx.x % V8, rl = threadIdx.x / V8;
  float mu[8], fc[8];
#pragma unroll
  for (int k = 0; k < 8; ++k) {
    mu[k] = mean != nullptr ? mean[c8 * 8 + k] : 0.f;
    fc[k] = fac != nullptr ? fac[c8 * 8 + k] : 1.f;
  }
  const bool sub = BM || mean != nullptr;
  // x - mean, then times the balancing factor (each an FP32 rounding), as configured
  auto load = [&](const uint4& u, float (&v)[8]) {
    unpack8(u, v);
    if (sub) {
#pragma unroll
      for (int k = 0; k < 8; ++k) v[k] = __fsub_rn(v[k], mu[k]);
    }
    if (fac != nullptr) {
#pragma unroll
      for (int k = 0; k < 8; ++k) v[k] = __fmul_rn(v[k], fc[k]);
    }
  };
  uint4 raw[PER];
#pragma unroll
  for (int e = 0; e < PER; ++e) {
    const int r = rl + e * RL;
    raw[e] = row0 + r < N ? *reinterpret_cast<const uint4*>(x + base + (size_t)r * D + c8 * 8)
                          : make_uint4(0u, 0u, 0u, 0u);
  }
  if constexpr (BM) {
    // Q-smoothing: the channel sums of the block's valid rows (rows past N were loaded as
    // zeros), exact (FP32 checked by TwoSum, else FP64; the FP64 combination across row lanes
    // and warps is exact for BF16 inputs of ordinary range), divided in FP64 and rounded to FP32
    double acc[8];
    exact_row_sums<PER>(raw, acc);
#pragma unroll
    for (int o = V8; o < 32; o <<= 1) {
#pragma unroll
      for (int k = 0; k < 8; ++k) acc[k] += __shfl_xor_sync(0xffffffffu, acc[k], o);
    }
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    if (lane < V8) {
#pragma unroll
      for (int k = 0; k < 8; ++k) mred[warp * D + lane * 8 + k] = acc[k];
    }
    __syncthreads();
    if (threadIdx.x < D) {
      double sum = 0.0;
#pragma unroll
      for (int w = 0; w < kThreads / 32; ++w) sum += mred[w * D + threadIdx.x];
      const float m = __double2float_rn(sum / (double)min(kBlk, N - row0));
      smean[threadIdx.x] = m;
      bmean[((size_t)bh * nb + blk) * D + threadIdx.x] = m;
    }
    __syncthreads();
#pragma unroll
    for (int k = 0; k < 8; ++k) mu[k] = smean[c8 * 8 + k];
  }
  float amax = 0.f;
#pragma unroll
  for (int e = 0; e < PER; ++e) {
    if (row0 + rl + e * RL < N) {
      float v[8];
      load(raw[e], v);
#pragma unroll
      for (int k = 0; k < 8; ++k) amax = fmaxf(amax, fabsf(v[k]));
    }
  }
  float gmax = amax;  // this thread's part of its 8-channel group's maximum
  const float a = block_max(amax, red);
  const bool live = a >= (vmode == kValFp8 ? kMinGroupMaxFp8 : kMinGroupMax);
  const float qmax = vmode == kValFp8 ? kFp8Max : 127.f;
  const float inv = live ? __fdiv_rn(qmax, a) : 0.f;
  if (vmode != kValInt8) {
#pragma unroll
    for (int e = 0; e < PER; ++e) {
      const int r = rl + e * RL;
      const bool valid = row0 + r < N;
      float v[8];
      if (valid) {
        load(raw[e], v);
#pragma unroll
        for (int q = 0; q < 8; ++q) v[q] = __fmul_rn(v[q], inv);
      } else {
#pragma unroll
        for (int q = 0; q < 8; ++q) v[q] = 0.f;
      }
      if (valid) {
        const uint4 out =
            vmode == kValBf16
                ? make_uint4(pack2(v[0], v[1]), pack2(v[2], v[3]), pack2(v[4], v[5]), pack2(v[6], v[7]))
                : make_uint4(e4m3x2_bf16x2(v[0], v[1]), e4m3x2_bf16x2(v[2], v[3]), e4m3x2_bf16x2(v[4], v[5]),
                             e4m3x2_bf16x2(v[6], v[7]));
        *reinterpret_cast<uint4*>(xq + base + (size_t)r * D + c8 * 8) = out;
      }
      if (vmode == kValFp8 && (x8 != nullptr || x8t != nullptr)) {
        const uint32_t b01 = e4m3x2_bytes(v[0], v[1]), b23 = e4m3x2_bytes(v[2], v[3]);
        const uint32_t b45 = e4m3x2_bytes(v[4], v[5]), b67 = e4m3x2_bytes(v[6], v[7]);
        if (x8 != nullptr && valid)
          *reinterpret_cast<uint2*>(x8 + base + (size_t)r * D + c8 * 8) =
              make_uint2(b01 | (b23 << 16), b45 | (b67 << 16));
        if (x8t != nullptr) {
          const uint32_t b[4] = {b01, b23, b45, b67};
#pragma unroll
          for (int q = 0; q < 8; ++q) t8[(c8 * 8 + q) * kBlk + r] = (uint8_t)(b[q >> 1] >> (8 * (q & 1)));
        }
      }
    }
    if (vmode == kValFp8 && x8t != nullptr) {
      // the transposed tile [D][128 tokens] as 16-byte rows pieces (rows past N were written as zero)
      __syncthreads();
      for (int i = threadIdx.x; i < D * (kBlk / 16); i += kThreads) {
        const int c = i / (kBlk / 16), v16 = i % (kBlk / 16);
        *reinterpret_cast<uint4*>(x8t + ((size_t)bh * D + c) * ((size_t)nb * kBlk) + row0 + v16 * 16) =
            *reinterpret_cast<const uint4*>(t8 + c * kBlk + v16 * 16);
      }
    }
  } else if (gred != nullptr) {
    // Q/K sub-scales: the group's maximum over the block's rows (the lanes that share c8,
    // then the warps), k = floor(log2(a / group max)) in [0, 8] (0 below 2^-100); the
    // codes are rint(x * inv * 2^k) and the stored values code * 2^-k, rounded onto that
    // grid directly by adding and subtracting 1.5 * 2^(23-k) (ties to even)
#pragma unroll
    for (int o = V8; o < 32; o <<= 1) gmax = fmaxf(gmax, __shfl_xor_sync(0xffffffffu, gmax, o));
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    if (lane < V8) gred[warp * V8 + lane] = gmax;
    __syncthreads();
    float g = 0.f;
#pragma unroll
    for (int w = 0; w < kThreads / 32; ++w) g = fmaxf(g, gred[w * V8 + c8]);
    int k = 0;
    if (live && g >= 0x1p-100f) {
      const uint32_t ua = __float_as_uint(a), ug = __float_as_uint(g);
      k = min(8, (int)(ua >> 23) - (int)(ug >> 23) - ((ua & 0x7FFFFFu) < (ug & 0x7FFFFFu) ? 1 : 0));
    }
    const float mg = __int_as_float(((127 + 23 - k) << 23) | 0x400000);
#pragma unroll
    for (int e = 0; e < PER; ++e) {
      const int r = rl + e * RL;
      if (row0 + r < N) {
        float v[8];
        load(raw[e], v);
#pragma unroll
        for (int q = 0; q < 8; ++q) v[q] = __fsub_rn(__fadd_rn(__fmul_rn(v[q], inv), mg), mg);
        const uint4 out = make_uint4(pack2(v[0], v[1]), pack2(v[2], v[3]), pack2(v[4], v[5]), pack2(v[6], v[7]));
        *reinterpret_cast<uint4*>(xq + base + (size_t)r * D + c8 * 8) = out;
      }
    }
  } else {
#pragma unroll
    for (int e = 0; e < PER; ++e) {
      const int r = rl + e * RL;
      if (row0 + r < N) {
        float v[8];
        load(raw[e], v);
        uint4 out;
        out.x = pack2(quant_code(v[0], inv), quant_code(v[1], inv));
        out.y = pack2(quant_code(v[2], inv), quant_code(v[3], inv));
        out.z = pack2(quant_code(v[4], inv), quant_code(v[5], inv));
        out.w = pack2(quant_code(v[6], inv), quant_code(v[7], inv));
        *reinterpret_cast<uint4*>(xq + base + (size_t)r * D + c8 * 8) = out;
      }
    }
  }
  if (threadIdx.x == 0) scale[(size_t)bh * nb + blk] = live ? __fdiv_rn(a, qmax) : 0.f;
}

// The exact FP64 channel sums of one 128-token block of one head (rows past N add nothing):
// part[bh][blk][D], four rows per lane at a time (exact_row_sums), then across the row lanes.
template <int D>
__device__ void block_channel_sums(const __nv_bfloat16* __restrict__ k, double* __restrict__ part, int bh, int blk,
                                   int N, int nb, double* red) {
  constexpr int V8 = D / 8, RL = kThreads / V8, RPL = kBlk / RL, G = 4;
  const int c8 = threadIdx.x % V8, rl = threadIdx.x / V8;
  double acc[8] = {0, 0, 0, 0, 0, 0, 0, 0};
#pragma unroll
  for (int g = 0; g < RPL; g += G) {
    uint4 u[G];
#pragma unroll
    for (int i = 0; i < G; ++i) {
      const int r = blk * kBlk + rl + (g + i) * RL;
      u[i] = r < N ? *reinterpret_cast<const uint4*>(k + ((size_t)bh * N + r) * D + c8 * 8)
                   : make_uint4(0u, 0u, 0u, 0u);
    }
    double s[8];
    exact_row_sums<G>(u, s);
#pragma unroll
    for (int e = 0; e < 8; ++e) acc[e] += s[e];
  }
#pragma unroll
  for (int e = 0; e < 8; ++e) red[rl * D + c8 * 8 + e] = acc[e];
  __syncthreads();
  if (threadIdx.x < D) {
    double t = 0;
#pragma unroll
    for (int q = 0; q < RL; ++q) t += red[q * D + threadIdx.x];
    part[((size_t)bh * nb + blk) * D + threadIdx.x] = t;
  }
}

template <int D, bool BM>
__global__ void __launch_bounds__(kThreads, BM ? 2 : 4) quantize_kernel(const QuantParams p) {
  __shared__ float red[kThreads / 32];
  __shared__ float fac[D];
  __shared__ float gred[kThreads / 32 * (D / 8)];
  if (p.clear_status && blockIdx.x == 0 && threadIdx.x == 0) *p.status = 0;
  pdl_trigger();
  int j = 0;
  while (j + 1 < p.njobs && (int)blockIdx.x >= p.block_start[j + 1]) ++j;
  const int local = blockIdx.x - p.block_start[j];
  const QuantJob& job = p.job[j];
  const int bh = local / p.nb;
  if (job.part != nullptr) {  // the K-mean pass's block sums, beside the other operands' codes
    __shared__ double sred[(kThreads / (D / 8)) * D];
    block_channel_sums<D>(job.x, job.part, bh, local % p.nb, p.N, p.nb, sred);
    return;
  }
  const float* mean = job.mean != nullptr ? job.mean + (size_t)bh * D : nullptr;  // this head's channel means
  // launched as a dependent of the kernel that computes the means: only the blocks that subtract
  // them wait for it
  if (mean != nullptr) pdl_wait();
  if (job.bexp != nullptr) {
    if (threadIdx.x < D) fac[threadIdx.x] = exp2_int(job.bexp_sign * job.bexp[(bh / job.bexp_group) * D + threadIdx.x]);
    __syncthreads();  // quantize_block reads fac only after this
  }
  if constexpr (BM) {
    __shared__ double mred[kThreads / 32 * D];
    __shared__ float smean[D];
    if (job.bmean != nullptr) {
      quantize_block<D, true>(job.x, job.xq, job.scale, mean, bh, local % p.nb, p.N, p.nb, red,
                              job.bexp != nullptr ? fac : nullptr, job.subexp ? gred : nullptr, job.bmean, mred,
                              smean, job.vmode);
      return;
    }
  }
  if (job.vmode == kValFp8) {
    __shared__ __align__(16) uint8_t t8[D * kBlk];  // transposed E4M3 tile
    quantize_block<D>(job.x, job.xq, job.scale, mean, bh, local % p.nb, p.N, p.nb, red, nullptr, nullptr, nullptr,
                      nullptr, nullptr, kValFp8, job.x8, job.x8t, t8);
    return;
  }
  quantize_block<D>(job.x, job.xq, job.scale, mean, bh, local % p.nb, p.N, p.nb, red,
                    job.bexp != nullptr ? fac : nullptr, job.subexp ? gred : nullptr, nullptr, nullptr, nullptr,
                    job.vmode);
}

// Channel statistics of one 128-token block of one head.  Blocks with
// blockIdx.y < BHk read K: FP64 channel sums (exact for BF16 inputs of
// ordinary range) and channel max / min; the others read Q: channel max |Q|,
// in FP32 only.  Every thread loads its RPL rows up front (16-byte vectors,
// rows past N skipped), then the row lanes are combined in shared memory.
template <int D>
__device__ __forceinline__ void k_stats_block(const StatsParams& p, int bh, int blk, uint8_t* smem) {
  constexpr int V8 = D / 8, RL = kThreads / V8, RPL = kBlk / RL;  // row lanes, rows per lane
  double(*sred)[D] = reinterpret_cast<double(*)[D]>(smem);
  float(*xred)[D] = reinterpret_cast<float(*)[D]>(smem + sizeof(double) * RL * D);
  float(*nred)[D] = reinterpret_cast<float(*)[D]>(smem + (sizeof(double) + sizeof(float)) * RL * D);
  const int c8 = threadIdx.x % V8, rl = threadIdx.x / V8;
  uint4 u[RPL];
#pragma unroll
  for (int i = 0; i < RPL; ++i) {
    const int r = blk * kBlk + rl + i * RL;
    u[i] = r < p.N ? *reinterpret_cast<const uint4*>(p.k + ((size_t)bh * p.N + r) * D + c8 * 8)
                   : make_uint4(0u, 0u, 0u, 0u);
  }
  double sum[8];
  exact_row_sums<RPL>(u, sum);
  float mx[8], mn[8];
#pragma unroll
  for (int e = 0; e < 8; ++e) {
    mx[e] = -INFINITY;
    mn[e] = INFINITY;
  }
#pragma unroll
  for (int i = 0; i < RPL; ++i) {
    if (blk * kBlk + rl + i * RL >= p.N) continue;
    float f[8];
    unpack8(u[i], f);
#pragma unroll
    for (int e = 0; e < 8; ++e) {
      mx[e] = fmaxf(mx[e], f[e]);
      mn[e] = fminf(mn[e], f[e]);
    }
  }
#pragma unroll
  for (int e = 0; e < 8; ++e) {
    sred[rl][c8 * 8 + e] = sum[e];
    xred[rl][c8 * 8 + e] = mx[e];
    nred[rl][c8 * 8 + e] = mn[e];
  }
  __syncthreads();
  if (threadIdx.x < D) {
    const int c = threadIdx.x;
    double s = 0;
    float a = -INFINITY, b = INFINITY;
#pragma unroll
    for (int q = 0; q < RL; ++q) {
      s += sred[q][c];
      a = fmaxf(a, xred[q][c]);
      b = fminf(b, nred[q][c]);
    }
    const size_t o = ((size_t)bh * p.nb + blk) * D + c;
    p.ksum[o] = s;
    p.kmax[o] = a;
    p.kmin[o] = b;
  }
}

template <int D>
__device__ __forceinline__ void q_absmax_block(const StatsParams& p, int bh, int blk, uint8_t* smem) {
  constexpr int V8 = D / 8, RL = kThreads / V8, RPL = kBlk / RL;
  float(*xred)[D] = reinterpret_cast<float(*)[D]>(smem);
  const int c8 = threadIdx.x % V8, rl = threadIdx.x / V8;
  uint4 u[RPL];
#pragma unroll
  for (int i = 0; i < RPL; ++i) {
    const int r = blk * kBlk + rl + i * RL;
    u[i] = r < p.N ? *reinterpret_cast<const uint4*>(p.q + ((size_t)bh * p.N + r) * D + c8 * 8)
                   : make_uint4(0u, 0u, 0u, 0u);  // |0| never raises a maximum
  }
  float mx[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
#pragma unroll
  for (int i = 0; i < RPL; ++i) {
    float f[8];
    unpack8(u[i], f);
#pragma unroll
    for (int e = 0; e < 8; ++e) mx[e] = fmaxf(mx[e], fabsf(f[e]));
  }
#pragma unroll
  for (int e = 0; e < 8; ++e) xred[rl][c8 * 8 + e] = mx[e];
  __syncthreads();
  if (threadIdx.x < D) {
    float a = 0.f;
#pragma unroll
    for (int q = 0; q < RL; ++q) a = fmaxf(a, xred[q][threadIdx.x]);
    p.qmax[((size_t)bh * p.nb + blk) * D + threadIdx.x] = a;
  }
}

template <int D>
__global__ void __launch_bounds__(kThreads) qk_stats_partial_kernel(const StatsParams p) {
  constexpr int RL = kThreads / (D / 8);
  __shared__ __align__(16) uint8_t smem[(sizeof(double) + 2 * sizeof(float)) * RL * D];
  if (blockIdx.x == 0 && blockIdx.y == 0 && threadIdx.x == 0) *p.status = 0;
  if ((int)blockIdx.y < p.BHk)
    k_stats_block<D>(p, blockIdx.y, blockIdx.x, smem);
  else
    q_absmax_block<D>(p, blockIdx.y - p.BHk, blockIdx.x, smem);
}

// Per (b, kv head): the K channel means and the balancing exponents.  A CTA
// takes 32 channels; its 8 warps reduce interleaved slices of the per-block
// partials, then warp 0 combines the slices in a fixed order.  The K side of
// the rule is max_n |fl(K_n - mean)|, which equals
// max(fl(Kmax - mean), fl(mean - Kmin)) because rounding is monotonic and
// symmetric.
constexpr int kFinalSlices = 32;
__global__ void __launch_bounds__(kFinalSlices * 32) qk_stats_final_kernel(const StatsParams p) {
  __shared__ double ssum[kFinalSlices][32];
  __shared__ float smax[kFinalSlices][32], smin[kFinalSlices][32], sq[kFinalSlices][32];
  const int bhk = blockIdx.x, lane = threadIdx.x & 31, sl = threadIdx.x >> 5;
  const int c = blockIdx.y * 32 + lane;
  double s = 0;
  float kx = -INFINITY, kn = INFINITY, aq = 0.f;
#pragma unroll 4
  for (int b = sl; b < p.nb; b += kFinalSlices) {
    const size_t o = ((size_t)bhk * p.nb + b) * p.d + c;
    s += p.ksum[o];
    kx = fmaxf(kx, p.kmax[o]);
    kn = fminf(kn, p.kmin[o]);
  }
  const int nq = p.G * p.nb;  // the kv head's query heads are consecutive: row (bhk * G + g) * nb + b
#pragma unroll 4
  for (int m = sl; m < nq; m += kFinalSlices) aq = fmaxf(aq, p.qmax[((size_t)bhk * nq + m) * p.d + c]);
  ssum[sl][lane] = s;
  smax[sl][lane] = kx;
  smin[sl][lane] = kn;
  sq[sl][lane] = aq;
  __syncthreads();
  if (sl != 0) return;
  for (int q = 1; q < kFinalSlices; ++q) {
    s += ssum[q][lane];
    kx = fmaxf(kx, smax[q][lane]);
    kn = fminf(kn, smin[q][lane]);
    aq = fmaxf(aq, sq[q][lane]);
  }
  float ak;
  if (p.smooth) {
    const float mu = (float)(s / (double)p.N);
    p.mean[(size_t)bhk * p.d + c] = mu;
    ak = fmaxf(__fsub_rn(kx, mu), __fsub_rn(mu, kn));
  } else {
    ak = fmaxf(kx, -kn);
  }
  int e = 0;
  if (aq > 0.f && ak > 0.f) {
    e = (binary_exponent(aq) - binary_exponent(ak)) >> 1;  // arithmetic shift: floor of the half
    e = min(126, max(-126, e));
  }
  p.bexp[(size_t)bhk * p.d + c] = e;
}

// Channel sums of K over one 128-token block, in FP64 (exact for BF16 inputs of
// ordinary range), reduced across threads in a fixed order.
template <int D>
__global__ void __launch_bounds__(kThreads) kmean_partial_kernel(const __nv_bfloat16* __restrict__ k,
                                                                 double* __restrict__ part, int N, int nb,
                                                                 int* status, int clear_status) {
  constexpr int V8 = D / 8, RL = kThreads / V8;  // row lanes
  __shared__ double red[RL][D];
  if (clear_status && blockIdx.x == 0 && blockIdx.y == 0 && threadIdx.x == 0) *status = 0;
  const int bh = blockIdx.y, blk = blockIdx.x;
  constexpr int RPL = kBlk / RL;  // rows per lane, all loaded up front
  const int c8 = threadIdx.x % V8, rl = threadIdx.x / V8;
  uint4 u[RPL];
#pragma unroll
  for (int i = 0; i < RPL; ++i) {
    const int r = blk * kBlk + rl + i * RL;
    u[i] = r < N ? *reinterpret_cast<const uint4*>(k + ((size_t)bh * N + r) * D + c8 * 8)
                 : make_uint4(0u, 0u, 0u, 0u);  // adds 0
  }
  double acc[8];
  exact_row_sums<RPL>(u, acc);
#pragma unroll
  for (int e = 0; e < 8; ++e) red[rl][c8 * 8 + e] = acc[e];
  __syncthreads();
  if (threadIdx.x < D) {
    double s = 0;
#pragma unroll
    for (int q = 0; q < RL; ++q) s += red[q][threadIdx.x];
    part[((size_t)bh * nb + blk) * D + threadIdx.x] = s;
  }
}

// Per head: the FP32 channel means from the per-block FP64 sums.  A CTA takes 32
// channels; its warps sum interleaved slices of the blocks, warp 0 combines
// the slices in a fixed order.
__global__ void __launch_bounds__(kFinalSlices * 32) kmean_final_kernel(const double* __restrict__ part,
                                                                        float* __restrict__ mean, int N, int nb,
                                                                        int d) {
  __shared__ double ssum[kFinalSlices][32];
  pdl_trigger();
  pdl_wait();  // the block sums, when launched as a dependent of their kernel
  const int bh = blockIdx.x, lane = threadIdx.x & 31, sl = threadIdx.x >> 5;
  const int c = blockIdx.y * 32 + lane;
  double s = 0;
#pragma unroll 4
  for (int b = sl; b < nb; b += kFinalSlices) s += part[((size_t)bh * nb + b) * d + c];
  ssum[sl][lane] = s;
  __syncthreads();
  if (sl != 0) return;
  for (int q = 1; q < kFinalSlices; ++q) s += ssum[q][lane];
  mean[(size_t)bh * d + c] = (float)(s / (double)N);
}

// Backward preprocess for one 128-query block: D_i = sum_c dO[i,c] O[i,c]
// (FP32), the dO block quantization, and zeroing the block's rows of the FP32
// dQ accumulator.
// Q-smoothing's logit terms ("SageBwd: A Trainable Low-bit Attention", Abstract, finding
// (iv); the library's reading of the optional Q-smoothing): with Q = (Q - mean_Q) + mean_Q per
// 128-token block, S = Q K'^T gains mean_Q(block of i) . K'_k, which depends on the query only
// through its block.  CTA (key block jb, query head bhq) writes, for every query block ib that
// sees key block jb, c0 * (mean_Q(bhq, ib) . K'_k) for its 128 keys, K' = K - mean_K (one FP32
// rounding each; K itself without smoothing), 0 past N.  Thread t holds keys 2 (t/2) and
// 2 (t/2) + 1 over channel half t % 2 in registers; the means of kQB query blocks at a time are
// staged in shared memory (broadcast reads, 8 FMAs per 16-byte load), each (key, block) sums its
// half in one FP32 chain, and the two halves are added with a lane shuffle.
constexpr int kQB = 8;
template <int D>
__global__ void __launch_bounds__(kBlk) qsmooth_bias_kernel(const QBiasParams p) {
  constexpr int DH = D / 2;
  __shared__ float4 msm[kQB * D / 4];
  // causal: key block jb sees nb - jb query blocks; blocks are dispatched in launch order with
  // blockIdx.x fastest, so the longest (small jb) go first
  const int jb = blockIdx.y, bhq = blockIdx.x;
  const int pair = threadIdx.x >> 1, half = threadIdx.x & 1;
  const int key0 = jb * kBlk + 2 * pair;
  const int bhk = bhq / p.G;  // b Hq + h -> b Hkv + h / G
  const size_t np = (size_t)p.nb * kBlk;
  float kr[2][DH];
#pragma unroll
  for (int u = 0; u < 2; ++u) {
    const bool live = key0 + u < p.N;
#pragma unroll
    for (int v = 0; v < DH / 8; ++v) {
      float f[8];
      if (live) {
        unpack8(*reinterpret_cast<const uint4*>(p.k + ((size_t)bhk * p.N + key0 + u) * D + half * DH + v * 8), f);
      } else {
#pragma unroll
        for (int e = 0; e < 8; ++e) f[e] = 0.f;
      }
#pragma unroll
      for (int e = 0; e < 8; ++e) {
        const int ch = half * DH + v * 8 + e;
        kr[u][v * 8 + e] = p.kmean != nullptr ? __fsub_rn(f[e], p.kmean[(size_t)bhk * D + ch]) : f[e];
      }
    }
  }
  const float4* mg = reinterpret_cast<const float4*>(p.qmean + (size_t)bhq * p.nb * D);
  const int mykey = key0 + half;  // the key this thread writes
  for (int ib0 = p.causal ? jb : 0; ib0 < p.nb; ib0 += kQB) {
    const int nq = min(kQB, p.nb - ib0);
    __syncthreads();  // the previous chunk's means have been read
    for (int e = threadIdx.x; e < nq * D / 4; e += kBlk) msm[e] = mg[(size_t)ib0 * D / 4 + e];
    __syncthreads();
    float acc[kQB][2];
#pragma unroll
    for (int q = 0; q < kQB; ++q) acc[q][0] = acc[q][1] = 0.f;
#pragma unroll
    for (int c4 = 0; c4 < DH / 4; ++c4) {
#pragma unroll
      for (int q = 0; q < kQB; ++q) {
        const float4 m = msm[q * D / 4 + half * DH / 4 + c4];  // rows past nq hold stale values; not stored
#pragma unroll
        for (int u = 0; u < 2; ++u) {
          acc[q][u] = fmaf(m.x, kr[u][4 * c4], acc[q][u]);
          acc[q][u] = fmaf(m.y, kr[u][4 * c4 + 1], acc[q][u]);
          acc[q][u] = fmaf(m.z, kr[u][4 * c4 + 2], acc[q][u]);
          acc[q][u] = fmaf(m.w, kr[u][4 * c4 + 3], acc[q][u]);
        }
      }
    }
#pragma unroll
    for (int q = 0; q < kQB; ++q) {
      // channel half 0 + half 1 of key 2 pair + half (the partner holds the other half)
      const float mine = half ? acc[q][1] : acc[q][0];
      const float other = __shfl_xor_sync(0xffffffffu, half ? acc[q][0] : acc[q][1], 1);
      const float dot = half == 0 ? mine + other : other + mine;
      if (q < nq) p.bias[((size_t)bhq * p.nb + ib0 + q) * np + mykey] = mykey < p.N ? __fmul_rn(dot, p.c0) : 0.f;
    }
  }
}

template <int D>
__global__ void __launch_bounds__(kThreads) bwd_prep_kernel(const PrepParams p) {
  __shared__ float red[kThreads / 32];
  if (blockIdx.x == 0 && blockIdx.y == 0 && threadIdx.x == 0) *p.status = 0;
  constexpr int V8 = D / 8;
  constexpr int PER = kBlk * V8 / kThreads;
  const int bh = blockIdx.y, blk = blockIdx.x;
  const int row0 = blk * kBlk;
  const size_t base = ((size_t)bh * p.N + row0) * D;
  // D = rowsum(dO * O): V8 consecutive threads share a row (V8 divides 32).
#pragma unroll
  for (int e = 0; e < PER; ++e) {
    const int idx = threadIdx.x + e * kThreads;
    const int r = idx / V8, c8 = idx % V8;
    float s = 0.f;
    if (row0 + r < p.N) {
      float a[8], b[8];
      unpack8(*reinterpret_cast<const uint4*>(p.dO + base + (size_t)r * D + c8 * 8), a);
      unpack8(*reinterpret_cast<const uint4*>(p.o + base + (size_t)r * D + c8 * 8), b);
#pragma unroll
      for (int k = 0; k < 8; ++k) s = fmaf(a[k], b[k], s);
      float4* z = reinterpret_cast<float4*>(p.dq_acc + base + (size_t)r * D + c8 * 8);
      z[0] = make_float4(0.f, 0.f, 0.f, 0.f);
      z[1] = make_float4(0.f, 0.f, 0.f, 0.f);
      if (bh < p.BHk) {  // the kv heads' dK / dV accumulators (BHk <= BH)
        float4* zk = reinterpret_cast<float4*>(p.dk_acc + base + (size_t)r * D + c8 * 8);
        float4* zv = reinterpret_cast<float4*>(p.dv_acc + base + (size_t)r * D + c8 * 8);
        zk[0] = zk[1] = zv[0] = zv[1] = make_float4(0.f, 0.f, 0.f, 0.f);
      }
    }
#pragma unroll
    for (int o = V8 / 2; o > 0; o >>= 1) s += __shfl_xor_sync(0xffffffffu, s, o);
    if (c8 == 0 && row0 + r < p.N) p.D[(size_t)bh * p.N + row0 + r] = s;
  }
  quantize_block<D>(p.dO, p.dOq, p.sdo, nullptr, bh, blk, p.N, p.nb, red, nullptr, nullptr, nullptr, nullptr,
                    nullptr, p.vmode);
}

struct ConvertJobs {
  ConvertJob job[3];
  int njobs;
};
__global__ void grad_convert_kernel(const ConvertJobs J) {
  for (int k = 0; k < J.njobs; ++k) {
    const ConvertJob& job = J.job[k];
    const float4* acc = reinterpret_cast<const float4*>(job.acc);
    uint2* out = reinterpret_cast<uint2*>(job.out);
    const size_t n4 = job.n / 4;
    const size_t row_elems = (size_t)job.N * job.d;
    const size_t stride = (size_t)gridDim.x * blockDim.x;
    constexpr int U = 4;  // vectors in flight per thread
    for (size_t i0 = (size_t)blockIdx.x * blockDim.x + threadIdx.x; i0 < n4; i0 += U * stride) {
      float4 v[U];
#pragma unroll
      for (int u = 0; u < U; ++u) {
        const size_t i = i0 + u * stride;
        if (i < n4) v[u] = acc[i];
      }
#pragma unroll
      for (int u = 0; u < U; ++u) {
        const size_t i = i0 + u * stride;
        if (i >= n4) continue;
        if (job.bexp != nullptr) {  // undo the channel balancing: exact power-of-two factors
          const size_t e0 = 4 * i;
          const int c = (int)(e0 % job.d);
          const int* ex = job.bexp + (e0 / row_elems / job.group) * job.d + c;
          v[u].x = __fmul_rn(v[u].x, exp2_int(job.sign * ex[0]));
          v[u].y = __fmul_rn(v[u].y, exp2_int(job.sign * ex[1]));
          v[u].z = __fmul_rn(v[u].z, exp2_int(job.sign * ex[2]));
          v[u].w = __fmul_rn(v[u].w, exp2_int(job.sign * ex[3]));
        }
        out[i] = make_uint2(pack2(v[u].x, v[u].y), pack2(v[u].z, v[u].w));
      }
    }
  }
}

}  // namespace

// Launch with the programmatic-serialization attribute when pdl is set (the kernel may start
// while the previous grid in the stream runs; it waits for it where it reads its results).
template <typename... Args>
cudaError_t launch_ex(void (*kernel)(Args...), dim3 grid, dim3 block, bool pdl, cudaStream_t s, Args... args) {
  cudaLaunchConfig_t cfg{};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = 0;
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = pdl ? 1 : 0;
  return cudaLaunchKernelEx(&cfg, kernel, args...);
}

cudaError_t launch_quantize(const QuantParams& p, cudaStream_t s, bool pdl) {
  const int blocks = p.block_start[p.njobs];
  if (blocks == 0) return cudaSuccess;
  bool bm = false;  // Q-smoothing's block means: a separate instantiation
  for (int j = 0; j < p.njobs; ++j) bm = bm || p.job[j].bmean != nullptr;
  auto kernel = p.d == 64 ? (bm ? quantize_kernel<64, true> : quantize_kernel<64, false>)
                          : (bm ? quantize_kernel<128, true> : quantize_kernel<128, false>);
  return launch_ex(kernel, dim3(blocks), dim3(kThreads), pdl, s, p);
}

cudaError_t launch_kmean_final(const double* part, float* mean, int BH, int N, int d, cudaStream_t s, bool pdl) {
  return launch_ex(kmean_final_kernel, dim3(BH, d / 32), dim3(kFinalSlices * 32), pdl, s, part, mean, N, nblocks(N),
                   d);
}

cudaError_t launch_kmean(const __nv_bfloat16* k, double* part, float* mean, int BH, int N, int d, int* status,
                         int clear_status, cudaStream_t s) {
  const int nb = nblocks(N);
  dim3 grid(nb, BH);
  if (d == 64)
    kmean_partial_kernel<64><<<grid, kThreads, 0, s>>>(k, part, N, nb, status, clear_status);
  else
    kmean_partial_kernel<128><<<grid, kThreads, 0, s>>>(k, part, N, nb, status, clear_status);
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  kmean_final_kernel<<<dim3(BH, d / 32), kFinalSlices * 32, 0, s>>>(part, mean, N, nb, d);
  return cudaGetLastError();
}

cudaError_t launch_qk_stats(const StatsParams& p, cudaStream_t s) {
  dim3 grid(p.nb, p.BHk + p.BHq);
  if (p.d == 64)
    qk_stats_partial_kernel<64><<<grid, kThreads, 0, s>>>(p);
  else
    qk_stats_partial_kernel<128><<<grid, kThreads, 0, s>>>(p);
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  qk_stats_final_kernel<<<dim3(p.BHk, p.d / 32), kFinalSlices * 32, 0, s>>>(p);
  return cudaGetLastError();
}

cudaError_t launch_bwd_prep(const PrepParams& p, cudaStream_t s) {
  dim3 grid(p.nb, p.BH);
  if (p.d == 64)
    bwd_prep_kernel<64><<<grid, kThreads, 0, s>>>(p);
  else
    bwd_prep_kernel<128><<<grid, kThreads, 0, s>>>(p);
  return cudaGetLastError();
}

cudaError_t launch_grad_convert(const ConvertJob* jobs, int njobs, cudaStream_t s) {
  ConvertJobs J{};
  size_t n4 = 0;
  for (int k = 0; k < njobs && k < 3; ++k) {
    J.job[k] = jobs[k];
    n4 = J.job[k].n / 4 > n4 ? J.job[k].n / 4 : n4;
  }
  J.njobs = njobs < 3 ? njobs : 3;
  if (n4 == 0) return cudaSuccess;
  int dev = 0, sms = 148;
  cudaGetDevice(&dev);
  cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  const size_t want = (n4 + 255) / 256;
  const int blocks = (int)(want < (size_t)sms * 8 ? want : (size_t)sms * 8);
  grad_convert_kernel<<<blocks, 256, 0, s>>>(J);
  return cudaGetLastError();
}

cudaError_t launch_qsmooth_bias(const QBiasParams& p, cudaStream_t s) {
  const dim3 grid(p.BHq, p.nb);
  if (p.d == 64)
    qsmooth_bias_kernel<64><<<grid, kBlk, 0, s>>>(p);
  else
    qsmooth_bias_kernel<128><<<grid, kBlk, 0, s>>>(p);
  return cudaGetLastError();
}

}  // namespace sagebwd
