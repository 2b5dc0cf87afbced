// Fused SageBwd attention forward on sm_103a ("SageBwd: A Trainable Low-bit
// Attention", Abstract: INT8 S = Q K^T and O = P V; FlashAttention-style
// online softmax with the LSE kept for the backward).
//
// One CTA computes one 128-row query tile of one head.  Warp roles:
//   warps 0-3  softmax / correction: thread r owns query row r (TMEM lane r)
//   warp 4     TMA producer: Q^ once, then K^_j and V^_j through a ring of stages
//   warp 5     TMEM allocation and the single MMA-issuing thread
// Per key tile j the MMA thread issues S_j = Q^ K^_j^T (integer-valued BF16,
// FP32 accumulation, exact) into one of two TMEM S buffers, then the
// previous tile's O_j-1 = P^_j-1 V^_j-1 into one of two TMEM O buffers, so the
// softmax of tile j overlaps the tensor-core work of tiles j and j-1.
//
// Softmax of tile j (FP32, base-2 logits t = S_int * sQ sK scale log2e):
//   tmax  = max_k t_k over the visible keys of the row in the tile
//   code  = rint(2^(t - tmax + log2 127)) in [0, 127]   (P~ quantized per row
//           and tile; written as the A operand of the P V product)
//   m'    = max(m, tmax),  alpha = 2^(m - m'),  r = 2^(tmax - m')
//   l     = l alpha + (r/127) sum_k 2^(t - tmax + log2 127)  (unquantized P~)
//   O    <- O alpha + (r/127) sV_j [P^ V^]_j   (dequantization per tile;
//           applied one tile late, when the P V product has landed)
// Epilogue: O / l as BF16, LSE = (m + log2 l) ln 2.
#include "kernel_common.cuh"

namespace sagebwd {
namespace {

template <int D>
struct FwdCfg {
  static constexpr int NS = D == 128 ? 2 : 3;  // K / V stages
  static constexpr int NP = D == 128 ? 1 : 2;  // P^ buffers
  static constexpr int TILE = 128 * D * 2;     // one Q^/K^/V^ tile (bytes)
  static constexpr int PTILE = 128 * 128 * 2;  // one P^ tile
  static constexpr int OFF_Q = 0;
  static constexpr int OFF_K = OFF_Q + TILE;
  static constexpr int OFF_V = OFF_K + NS * TILE;
  static constexpr int OFF_P = OFF_V + NS * TILE;
  static constexpr int OFF_BAR = OFF_P + NP * PTILE;
  static constexpr int NBAR = 1 + 4 * NS + 2 + 2 + 2 * NP + 2 + 2 + 1;
  static constexpr int SMEM = OFF_BAR + NBAR * 8 + 16 + 1024;
};

enum FwdSite { kSiteQ = 1, kSiteKFull, kSiteKEmpty, kSiteVFull, kSiteVEmpty, kSiteSFull, kSiteSEmpty,
               kSitePFull, kSitePEmpty, kSiteOFull, kSiteOEmpty };

template <int D, bool CAUSAL>
__global__ void __launch_bounds__(192, 1)
    fwd_kernel(const __grid_constant__ CUtensorMap tmQ, const __grid_constant__ CUtensorMap tmK,
               const __grid_constant__ CUtensorMap tmV, const FwdParams p) {
  using C = FwdCfg<D>;
  constexpr int NS = C::NS, NP = C::NP;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = align1024(smem_raw);
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + C::OFF_BAR);
  uint64_t* bar_q = bars;
  uint64_t* bar_k_full = bar_q + 1;
  uint64_t* bar_k_empty = bar_k_full + NS;
  uint64_t* bar_v_full = bar_k_empty + NS;
  uint64_t* bar_v_empty = bar_v_full + NS;
  uint64_t* bar_s_full = bar_v_empty + NS;
  uint64_t* bar_s_empty = bar_s_full + 2;
  uint64_t* bar_p_full = bar_s_empty + 2;
  uint64_t* bar_p_empty = bar_p_full + NP;
  uint64_t* bar_o_full = bar_p_empty + NP;
  uint64_t* bar_o_empty = bar_o_full + 2;
  uint64_t* bar_final = bar_o_empty + 2;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(bar_final + 1);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int BH = p.B * p.Hq;
  const int L = blockIdx.x;
  const int qb = CAUSAL ? (p.nb - 1 - L / BH) : (L / BH);  // causal: longest rows first
  const int bhq = L % BH;
  const int b = bhq / p.Hq, h = bhq % p.Hq;
  const int bhk = b * p.Hkv + h / p.G;
  const int q0 = qb * kBlk;
  const int nkb = CAUSAL ? qb + 1 : p.nb;

  if (tid == 0) {
    mbar_init(bar_q, 1);
    for (int s = 0; s < NS; ++s) {
      mbar_init(bar_k_full + s, 1);
      mbar_init(bar_k_empty + s, 1);
      mbar_init(bar_v_full + s, 1);
      mbar_init(bar_v_empty + s, 1);
    }
    for (int s = 0; s < 2; ++s) {
      mbar_init(bar_s_full + s, 1);
      mbar_init(bar_s_empty + s, 128);
      mbar_init(bar_o_full + s, 1);
      mbar_init(bar_o_empty + s, 128);
    }
    for (int s = 0; s < NP; ++s) {
      mbar_init(bar_p_full + s, 128);
      mbar_init(bar_p_empty + s, 1);
    }
    mbar_init(bar_final, 1);
    *abort_flag = 0;
    fence_mbar_init();
  }
  if (warp == 5) {
    tmem_alloc(tmem_slot, 512);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  const WaitCtx wc{abort_flag, p.status, p.timeout_ns};

  if (warp == 4) {
    // ------------------------------------------------------------ TMA producer
    if (lane == 0) {
      int k_issued[NS], v_issued[NS];
      for (int s = 0; s < NS; ++s) k_issued[s] = v_issued[s] = 0;
      mbar_arrive_expect_tx(bar_q, C::TILE);
      for (int c = 0; c < D / 64; ++c) tma_load_3d(smem + C::OFF_Q + c * 16384, &tmQ, bar_q, c * 64, q0, bhq);
      for (int j = 0; j < nkb; ++j) {
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
    }
  } else if (warp == 5) {
    // ------------------------------------------------------------ MMA issuer
    if (lane == 0) {
      const uint32_t idS = idesc_bf16_f32(128, 128, false, false);
      const uint32_t idO = idesc_bf16_f32(128, D, false, true);
      bool ok = wait1(wc, bar_q, 0, kSiteQ);
      const uint32_t sQ = smem_u32(smem + C::OFF_Q);
      for (int j = 0; ok && j <= nkb; ++j) {
        if (j < nkb) {
          const int s = j % NS, sb = j & 1;
          if (!wait1(wc, bar_k_full + s, (j / NS) & 1, kSiteKFull)) break;
          if (j >= 2 && !wait1(wc, bar_s_empty + sb, ((j >> 1) - 1) & 1, kSiteSEmpty)) break;
          tc_fence_after();
          const uint32_t sK = smem_u32(smem + C::OFF_K + s * C::TILE);
#pragma unroll
          for (int kk = 0; kk < D / 16; ++kk) {
            const uint32_t off = (kk >> 2) * 16384 + (kk & 3) * 32;
            umma_ss(tmem + sb * 128, sdesc_sw128(sQ + off, 16, 1024), sdesc_sw128(sK + off, 16, 1024), idS, kk > 0);
          }
          umma_commit(bar_s_full + sb);
          umma_commit(bar_k_empty + s);
        }
        if (j >= 1) {
          const int jj = j - 1, s = jj % NS, ob = jj & 1, pb = jj % NP;
          if (!wait1(wc, bar_p_full + pb, (jj / NP) & 1, kSitePFull)) break;
          if (!wait1(wc, bar_v_full + s, (jj / NS) & 1, kSiteVFull)) break;
          if (jj >= 2 && !wait1(wc, bar_o_empty + ob, ((jj >> 1) - 1) & 1, kSiteOEmpty)) break;
          tc_fence_after();
          const uint32_t sP = smem_u32(smem + C::OFF_P + pb * C::PTILE);
          const uint32_t sV = smem_u32(smem + C::OFF_V + s * C::TILE);
#pragma unroll
          for (int kk = 0; kk < 8; ++kk) {
            umma_ss(tmem + 256 + ob * D, sdesc_sw128(sP + (kk >> 2) * 16384 + (kk & 3) * 32, 16, 1024),
                    sdesc_sw128(sV + kk * 2048, 16384, 1024), idO, kk > 0);
          }
          umma_commit(bar_o_full + ob);
          umma_commit(bar_v_empty + s);
          umma_commit(bar_p_empty + pb);
        }
      }
      // Every MMA issued above must complete before TMEM is released.
      umma_commit(bar_final);
      drain(bar_final, 0, p.timeout_ns);
    }
  } else {
    // ------------------------------------------------------------ softmax / correction
    const int r = tid;  // query row within the tile == TMEM lane
    const int i = q0 + r;
    const uint32_t lane_base = (uint32_t)(warp * 32) << 16;
    const float sQv = p.sq[(size_t)bhq * p.nb + qb];
    float m = -INFINITY, l = 0.f;
    float o_acc[D];
#pragma unroll
    for (int c = 0; c < D; ++c) o_acc[c] = 0.f;
    float pend_alpha = 0.f, pend_w = 0.f;
    bool ok = true;

    // Fold tile t's P V product into the running output.
    auto fold = [&](int t, float a, float w) -> bool {
      const int ob = t & 1;
      if (!waitw(wc, bar_o_full + ob, (t >> 1) & 1, kSiteOFull)) return false;
      tc_fence_after();
#pragma unroll
      for (int c0 = 0; c0 < D; c0 += 32) {
        uint32_t v[32];
        tmem_ld32(tmem + lane_base + 256 + ob * D + c0, v);
        tmem_ld_wait();
#pragma unroll
        for (int e = 0; e < 32; ++e) o_acc[c0 + e] = fmaf(w, __uint_as_float(v[e]), o_acc[c0 + e] * a);
      }
      tc_fence_before();
      mbar_arrive(bar_o_empty + ob);
      return true;
    };

    for (int j = 0; j < nkb; ++j) {
      const int sb = j & 1;
      if (!waitw(wc, bar_s_full + sb, (j >> 1) & 1, kSiteSFull)) {
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
      const uint32_t s_addr = tmem + lane_base + sb * 128;
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
      const int pb = j % NP;
      if (j >= NP && !waitw(wc, bar_p_empty + pb, ((j / NP) - 1) & 1, kSitePEmpty)) {
        ok = false;
        break;
      }
      // pass 2: codes of P~ into the swizzled A tile, and the unquantized row sum
      const uint32_t p_base = smem_u32(smem + C::OFF_P + pb * C::PTILE);
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
          pk[e >> 1] = pack_bf16x2(rint_f32(u0), rint_f32(u1));
        }
#pragma unroll
        for (int q = 0; q < 4; ++q)
          st_shared_v4(p_base + sw128_offset(r, (c0 >> 3) + q), pk[4 * q], pk[4 * q + 1], pk[4 * q + 2],
                       pk[4 * q + 3]);
      }
      tc_fence_before();
      mbar_arrive(bar_s_empty + sb);
      fence_proxy_async_smem();
      mbar_arrive(bar_p_full + pb);
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
    if (ok) ok = fold(nkb - 1, pend_alpha, pend_w);
    if (ok && !*abort_flag && i < p.N) {
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
  if (warp == 5) {
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
  const int grid = p.nb * p.B * p.Hq;
  kern<<<grid, 192, C::SMEM, s>>>(tq, tk, tv, p);
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_fwd(const CUtensorMap& tq, const CUtensorMap& tk, const CUtensorMap& tv, const FwdParams& p, int d,
                       int causal, cudaStream_t s) {
  if (d == 64) return causal ? launch_fwd_t<64, true>(tq, tk, tv, p, s) : launch_fwd_t<64, false>(tq, tk, tv, p, s);
  return causal ? launch_fwd_t<128, true>(tq, tk, tv, p, s) : launch_fwd_t<128, false>(tq, tk, tv, p, s);
}

}  // namespace sagebwd
