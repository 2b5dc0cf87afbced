// Fused SageBwd attention forward on sm_103a ("SageBwd: A Trainable Low-bit
// Attention", Abstract: INT8 S = Q K^T and O = P V; FlashAttention-style
// online softmax with the LSE kept for the backward).
//
// One CTA computes two 128-row query tiles (t = 0, 1) of one head, so that the
// softmax of one tile overlaps the tensor-core work of the other.  Warp roles:
//   warps 0-3 / 4-7  softmax warpgroup of tile 0 / 1: thread r owns query row r
//                    (TMEM lane r) and keeps that row of the running output in
//                    FP32 registers
//   warp 8           TMA producer: both Q^ tiles once, K^_j and V^_j through rings
//   warp 9           TMEM allocation and the single MMA-issuing thread
//   warps 10-11      idle (complete the third warpgroup, which gives its
//                    registers to the softmax warpgroups: 384 threads launch with
//                    168 registers each; 128 * kRegsLow + 256 * kRegsHigh <= 384 * 168)
// TMEM: tile t owns S_t [256t, 256t+128) and O_t [256t+128, 256t+128+d).  The
// quantized P~ codes are written over S_t (packed BF16, columns [256t, 256t+64))
// and feed O_t = P^_t V^_j as the A operand straight from TMEM.
// MMA order per key tile j: S_0(j), S_1(j), then P^_0 V^_j, P^_1 V^_j; S_t(j+1)
// waits until P^_t V^_j has consumed the codes that share its columns.
//
// Softmax of tile j for one row (FP32, base-2 logits t = S_int * sQ sK scale log2e):
//   tmax  = max_k t_k over the visible keys of the row in the tile
//   code  = rint(2^(t - tmax + log2 127)) in [0, 127]   (P~ quantized per row and tile)
//   m'    = max(m, tmax),  alpha = 2^(m - m'),  r = 2^(tmax - m')
//   l     = l alpha + (r/127) sum_k 2^(t - tmax + log2 127)   (unquantized P~)
//   O    <- O alpha + (r/127) sV_j [P^ V^]_j   (dequantization per tile, applied one
//           tile late, once the P V product has landed)
// Epilogue: O / l as BF16, LSE = (m + log2 l) ln 2.
#include "kernel_common.cuh"

namespace sagebwd {
namespace {

constexpr int kFThreads = 384;
constexpr uint32_t kFRegsLaunch = 168, kFRegsLow = 40, kFRegsHigh = 232;
static_assert(128 * kFRegsLow + 256 * kFRegsHigh <= kFThreads * kFRegsLaunch, "register split exceeds the launch");

template <int D>
struct FwdCfg {
  static constexpr int NS = 2;             // K / V stages
  static constexpr int TILE = 128 * D * 2;  // one Q^ / K^ / V^ tile (bytes)
  static constexpr int OFF_Q = 0;           // two Q^ tiles
  static constexpr int OFF_K = OFF_Q + 2 * TILE;
  static constexpr int OFF_V = OFF_K + NS * TILE;
  static constexpr int OFF_BAR = OFF_V + NS * TILE;
  static constexpr int NBAR = 1 + 4 * NS + 2 * 4 + 1;
  static constexpr int SMEM = OFF_BAR + NBAR * 8 + 16 + 1024;
  static_assert(SMEM <= 232448, "shared memory beyond the per-CTA limit");
  __host__ __device__ static constexpr int col_s(int t) { return 256 * t; }
  __host__ __device__ static constexpr int col_o(int t) { return 256 * t + 128; }
};

enum FwdSite { kSiteQ = 1, kSiteKFull, kSiteKEmpty, kSiteVFull, kSiteVEmpty, kSiteSFull, kSitePFull, kSitePVDone,
               kSiteOEmpty };

template <int D, bool CAUSAL>
__global__ void __launch_bounds__(kFThreads, 1)
    fwd_kernel(const __grid_constant__ CUtensorMap tmQ, const __grid_constant__ CUtensorMap tmK,
               const __grid_constant__ CUtensorMap tmV, const FwdParams p) {
  using C = FwdCfg<D>;
  constexpr int NS = C::NS;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = align1024(smem_raw);
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + C::OFF_BAR);
  uint64_t* bar_q = bars;
  uint64_t* bar_k_full = bar_q + 1;
  uint64_t* bar_k_empty = bar_k_full + NS;
  uint64_t* bar_v_full = bar_k_empty + NS;
  uint64_t* bar_v_empty = bar_v_full + NS;
  uint64_t* bar_s_full = bar_v_empty + NS;  // [2] S_t in TMEM
  uint64_t* bar_p_full = bar_s_full + 2;    // [2] codes of P~_t in TMEM (softmax)
  uint64_t* bar_pv_done = bar_p_full + 2;   // [2] P^_t V^ in TMEM (and the codes consumed)
  uint64_t* bar_o_empty = bar_pv_done + 2;  // [2] O_t folded into registers (softmax)
  uint64_t* bar_final = bar_o_empty + 2;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(bar_final + 1);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int BH = p.B * p.Hq;
  const int npairs = (p.nb + 1) / 2;
  const int L = blockIdx.x;
  const int pr = CAUSAL ? (npairs - 1 - L / BH) : (L / BH);  // causal: longest rows first
  const int bhq = L % BH;
  const int b = bhq / p.Hq, h = bhq % p.Hq;
  const int bhk = b * p.Hkv + h / p.G;
  int nkb[2];
#pragma unroll
  for (int t = 0; t < 2; ++t) {
    const int qb = 2 * pr + t;
    nkb[t] = qb >= p.nb ? 0 : (CAUSAL ? qb + 1 : p.nb);
  }
  const int nkb_max = nkb[0] > nkb[1] ? nkb[0] : nkb[1];

  if (tid == 0) {
    mbar_init(bar_q, 1);
    for (int s = 0; s < NS; ++s) {
      mbar_init(bar_k_full + s, 1);
      mbar_init(bar_k_empty + s, 1);
      mbar_init(bar_v_full + s, 1);
      mbar_init(bar_v_empty + s, 1);
    }
    for (int t = 0; t < 2; ++t) {
      mbar_init(bar_s_full + t, 1);
      mbar_init(bar_p_full + t, 128);
      mbar_init(bar_pv_done + t, 1);
      mbar_init(bar_o_empty + t, 128);
    }
    mbar_init(bar_final, 1);
    *abort_flag = 0;
    fence_mbar_init();
  }
  if (warp == 9) {
    tmem_alloc(tmem_slot, 512);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  const WaitCtx wc{abort_flag, p.status, p.timeout_ns};

  if (warp >= 8) {
    setmaxnreg_dec<kFRegsLow>();
    if (warp == 8 && lane == 0) {
      // ---------------------------------------------------------- TMA producer
      int k_issued[NS], v_issued[NS];
      for (int s = 0; s < NS; ++s) k_issued[s] = v_issued[s] = 0;
      const int nq = (nkb[0] > 0) + (nkb[1] > 0);
      mbar_arrive_expect_tx(bar_q, nq * C::TILE);
      for (int t = 0; t < 2; ++t)
        if (nkb[t] > 0)
          for (int c = 0; c < D / 64; ++c)
            tma_load_3d(smem + C::OFF_Q + t * C::TILE + c * 16384, &tmQ, bar_q, c * 64, (2 * pr + t) * kBlk, bhq);
      for (int j = 0; j < nkb_max; ++j) {
        const int s = j % NS, n = j / NS;
        if (j >= NS && !wait1(wc, bar_k_empty + s, (n - 1) & 1, kSiteKEmpty)) break;
        if (!((p.flags & SAGEBWD_FLAG_DROP_ONE_LOAD) && j == 1)) {  // fault injection skips one load
          mbar_arrive_expect_tx(bar_k_full + s, C::TILE);
          for (int c = 0; c < D / 64; ++c)
            tma_load_3d(smem + C::OFF_K + s * C::TILE + c * 16384, &tmK, bar_k_full + s, c * 64, j * kBlk, bhk);
          k_issued[s] = n + 1;
        }
        if (j >= NS && !wait1(wc, bar_v_empty + s, (n - 1) & 1, kSiteVEmpty)) break;
        mbar_arrive_expect_tx(bar_v_full + s, C::TILE);
        for (int c = 0; c < D / 64; ++c)
          tma_load_3d(smem + C::OFF_V + s * C::TILE + c * 16384, &tmV, bar_v_full + s, c * 64, j * kBlk, bhk);
        v_issued[s] = n + 1;
      }
      // Copies still in flight must land before the CTA's shared memory is released.
      drain(bar_q, 0, p.timeout_ns);
      for (int s = 0; s < NS; ++s) {
        if (k_issued[s]) drain(bar_k_full + s, (k_issued[s] - 1) & 1, p.timeout_ns);
        if (v_issued[s]) drain(bar_v_full + s, (v_issued[s] - 1) & 1, p.timeout_ns);
      }
    } else if (warp == 9 && lane == 0) {
      // ---------------------------------------------------------- MMA issuer
      const uint32_t idS = idesc_bf16_f32(128, 128, false, false);
      const uint32_t idO = idesc_bf16_f32(128, D, false, true);
      bool ok = wait1(wc, bar_q, 0, kSiteQ);
      for (int j = 0; ok && j < nkb_max; ++j) {
        const int s = j % NS;
        if (!wait1(wc, bar_k_full + s, (j / NS) & 1, kSiteKFull)) break;
        const uint32_t kdesc = sdesc_sw128_lo(smem_u32(smem + C::OFF_K + s * C::TILE), 16);
#pragma unroll
        for (int t = 0; t < 2; ++t) {
          if (j >= nkb[t]) continue;
          // S_t(j) overwrites the columns that held P^_t(j-1): wait until P^_t(j-1) V^ is done
          if (j >= 1 && !wait1(wc, bar_pv_done + t, (j - 1) & 1, kSitePVDone)) {
            ok = false;
            break;
          }
          tc_fence_after();
          const uint32_t qdesc = sdesc_sw128_lo(smem_u32(smem + C::OFF_Q + t * C::TILE), 16);
          if constexpr (D == 128)
            umma_chain8_kk(tmem + C::col_s(t), sdesc_from_lo(qdesc), sdesc_from_lo(kdesc), idS);
          else
            umma_chain4_kk(tmem + C::col_s(t), sdesc_from_lo(qdesc), sdesc_from_lo(kdesc), idS);
          umma_commit(bar_s_full + t);
        }
        if (!ok) break;
        umma_commit(bar_k_empty + s);
        if (!wait1(wc, bar_v_full + s, (j / NS) & 1, kSiteVFull)) break;
        const uint32_t vdesc = sdesc_sw128_lo(smem_u32(smem + C::OFF_V + s * C::TILE), 16384);
#pragma unroll
        for (int t = 0; t < 2; ++t) {
          if (j >= nkb[t]) continue;
          if (!wait1(wc, bar_p_full + t, j & 1, kSitePFull)) {
            ok = false;
            break;
          }
          if (j >= 1 && !wait1(wc, bar_o_empty + t, (j - 1) & 1, kSiteOEmpty)) {
            ok = false;
            break;
          }
          tc_fence_after();
          // O_t = P^_t V^_j: A = the codes in TMEM (K = 128 keys = 64 packed columns, 8 per
          // K step), B = V^_j [key][d] read MN-major
#pragma unroll
          for (int kk = 0; kk < 8; ++kk)
            umma_ts(tmem + C::col_o(t), tmem + C::col_s(t) + kk * 8, sdesc_from_lo(vdesc + kk * 128), idO, kk > 0);
          umma_commit(bar_pv_done + t);
        }
        if (!ok) break;
        umma_commit(bar_v_empty + s);
      }
      // Every MMA issued above must complete before TMEM is released.
      umma_commit(bar_final);
      drain(bar_final, 0, p.timeout_ns);
    }
  } else {
    setmaxnreg_inc<kFRegsHigh>();
    // ------------------------------------------------------------ softmax / correction
    const int t = warp >> 2;  // query tile of this warpgroup
    const int r = tid & 127;  // query row within the tile == TMEM lane
    const int qb = 2 * pr + t;
    const int i = qb * kBlk + r;
    const int nk = nkb[t];
    const uint32_t lane_base = (uint32_t)((warp & 3) * 32) << 16;
    const uint32_t s_addr = tmem + lane_base + C::col_s(t);
    const uint32_t o_addr = tmem + lane_base + C::col_o(t);
    const float sQv = nk > 0 ? p.sq[(size_t)bhq * p.nb + qb] : 0.f;
    float m = -INFINITY, l = 0.f;
    float o_acc[D];
#pragma unroll
    for (int c = 0; c < D; ++c) o_acc[c] = 0.f;
    float pend_alpha = 0.f, pend_w = 0.f;
    bool ok = true;

    // Fold tile jj's P V product into the running output.
    auto fold = [&](int jj, float a, float w) -> bool {
      if (!waitw(wc, bar_pv_done + t, jj & 1, kSitePVDone)) return false;
      tc_fence_after();
#pragma unroll
      for (int c0 = 0; c0 < D; c0 += 32) {
        uint32_t v[32];
        tmem_ld32(o_addr + c0, v);
        tmem_ld_wait();
#pragma unroll
        for (int e = 0; e < 32; ++e) o_acc[c0 + e] = fmaf(w, __uint_as_float(v[e]), o_acc[c0 + e] * a);
      }
      tc_fence_before();
      mbar_arrive(bar_o_empty + t);
      return true;
    };

    for (int j = 0; j < nk; ++j) {
      if (!waitw(wc, bar_s_full + t, j & 1, kSiteSFull)) {
        ok = false;
        break;
      }
      tc_fence_after();
      const float sKv = p.sk[(size_t)bhk * p.nb + j];
      const float sVv = p.sv[(size_t)bhk * p.nb + j];
      const float qks = __fmul_rn(__fmul_rn(sQv, sKv), p.c0);
      const int k0 = j * kBlk;
      const bool need_mask = (CAUSAL && j == qb) || (k0 + kBlk > p.N);
      const int kvis = need_mask ? (min(p.N, CAUSAL ? i + 1 : p.N) - k0) : kBlk;  // visible keys of this row
      // pass 1: row maximum of S_int over the visible keys
      float smax = -INFINITY;
#pragma unroll
      for (int c0 = 0; c0 < 128; c0 += 32) {
        uint32_t v[32];
        tmem_ld32(s_addr + c0, v);
        tmem_ld_wait();
#pragma unroll
        for (int e = 0; e < 32; ++e) {
          const float sv = __uint_as_float(v[e]);
          smax = fmaxf(smax, (need_mask && c0 + e >= kvis) ? -INFINITY : sv);
        }
      }
      const float tmax = __fmul_rn(smax, qks);
      const float m_new = fmaxf(m, tmax);
      const float alpha = ex2_approx(m - m_new);
      const float rj = ex2_approx(tmax - m_new);
      const float bias = kLog2_127 - tmax;
      // pass 2: codes of P~ written over the S columns already read (chunk c of 32 keys
      // -> 16 packed columns starting at 16c), and the unquantized row sum
      float usum = 0.f;
#pragma unroll
      for (int c0 = 0; c0 < 128; c0 += 32) {
        uint32_t v[32];
        tmem_ld32(s_addr + c0, v);
        tmem_ld_wait();
        uint32_t pk[16];
#pragma unroll
        for (int e = 0; e < 32; e += 2) {
          float u0 = ex2_approx(fmaf(__uint_as_float(v[e]), qks, bias));
          float u1 = ex2_approx(fmaf(__uint_as_float(v[e + 1]), qks, bias));
          if (need_mask) {
            if (c0 + e >= kvis) u0 = 0.f;
            if (c0 + e + 1 >= kvis) u1 = 0.f;
          }
          usum += u0 + u1;
          pk[e >> 1] = pack_int_bf16x2(rint_small(u0), rint_small(u1));
        }
        tmem_st16(s_addr + (c0 >> 1), pk);
      }
      tmem_st_wait();
      tc_fence_before();
      mbar_arrive(bar_p_full + t);
      const float w_l = rj * (1.f / 127.f);
      l = fmaf(w_l, usum, l * alpha);
      m = m_new;
      if (j >= 1 && !fold(j - 1, pend_alpha, pend_w)) {
        ok = false;
        break;
      }
      pend_alpha = alpha;
      pend_w = w_l * sVv;
    }
    if (ok && nk > 0) ok = fold(nk - 1, pend_alpha, pend_w);
    if (ok && nk > 0 && !*abort_flag && i < p.N) {
      const float inv_l = 1.f / l;
      uint4* dst = reinterpret_cast<uint4*>(p.o + ((size_t)bhq * p.N + i) * D);
#pragma unroll
      for (int c = 0; c < D; c += 8) {
        uint4 u;
        u.x = pack_bf16x2(o_acc[c] * inv_l, o_acc[c + 1] * inv_l);
        u.y = pack_bf16x2(o_acc[c + 2] * inv_l, o_acc[c + 3] * inv_l);
        u.z = pack_bf16x2(o_acc[c + 4] * inv_l, o_acc[c + 5] * inv_l);
        u.w = pack_bf16x2(o_acc[c + 6] * inv_l, o_acc[c + 7] * inv_l);
        dst[c / 8] = u;
      }
      p.lse[(size_t)bhq * p.N + i] = (m + log2f(l)) * kLn2;
    }
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 9) {
    tc_fence_after();
    tmem_dealloc(tmem, 512);
  }
}

template <int D, bool CAUSAL>
cudaError_t launch_fwd_t(const CUtensorMap& tq, const CUtensorMap& tk, const CUtensorMap& tv, const FwdParams& p,
                         cudaStream_t s) {
  using C = FwdCfg<D>;
  auto kern = fwd_kernel<D, CAUSAL>;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, C::SMEM);
  if (e != cudaSuccess) return e;
  const int grid = (p.nb + 1) / 2 * p.B * p.Hq;
  kern<<<grid, kFThreads, C::SMEM, s>>>(tq, tk, tv, p);
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_fwd(const CUtensorMap& tq, const CUtensorMap& tk, const CUtensorMap& tv, const FwdParams& p, int d,
                       int causal, cudaStream_t s) {
  if (d == 64) return causal ? launch_fwd_t<64, true>(tq, tk, tv, p, s) : launch_fwd_t<64, false>(tq, tk, tv, p, s);
  return causal ? launch_fwd_t<128, true>(tq, tk, tv, p, s) : launch_fwd_t<128, false>(tq, tk, tv, p, s);
}

}  // namespace sagebwd
