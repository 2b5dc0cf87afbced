// Fused SageBwd attention backward on sm_103a ("SageBwd: A Trainable Low-bit
// Attention", Abstract: INT8 S recompute, dV = P^T dO, dQ = dS K,
// dK = dS^T Q; "SageAttention3 ... 8-Bit Training" summary, Approach: dO V^T
// kept in 16-bit floating point; FlashAttention-2 backward structure with
// D = rowsum(dO * O) and dS = P (dP - D)).
//
// One CTA owns one 128-key block j of one kv head and loops over the G query
// heads of that kv head and their 128-query blocks i, so dK_j and dV_j are
// summed in registers and written once; dQ is accumulated across CTAs with
// FP32 reductions into the workspace.  Warp roles:
//   warps 0-15       four compute warpgroups: thread (w, r) owns key row r
//                    (TMEM lane r), query columns [32w, 32w+32) of the tile and
//                    output columns [w d/4, (w+1) d/4) of dK, dV, dQ
//   warp 16          TMA producer (K^_j, V_j once; Q^_i, dO_i, dO^_i per tile)
//   warp 17          TMEM allocation and the MMA-issuing thread
//   warps 18-19      idle (they complete the fifth warpgroup, which gives its
//                    registers to the compute warpgroups: 640 threads launch
//                    with 96 registers each; the producer warpgroup drops to
//                    kRegsLow, the compute warpgroups rise to kRegsHigh)
// Per tile (TMEM columns: S^T [0,128), dP^T [128,256), dV [256,256+d),
// dK [256+d,256+2d), dQ [0,d) reusing S^T once it is consumed):
//   MMA   S^T = K^_j Q^_i^T (integer-valued BF16, exact)  dP^T = V_j dO_i^T (BF16)
//   pass 1  P = 2^(S sQ sK scale log2e - LSE_i log2e), dS = P (dP - D_i); both
//           written back to TMEM in place; row max of P, tile max of |dS|
//   pass 2  code(P^T) per key row (scale max P / 127), code(dS) per tile
//           (scale max|dS| / 127) into swizzled shared-memory A operands
//   MMA   dK = dS^T Q^_i, dQ = dS K^_j, dV = P^T dO^_i (all exact integer products)
//   pass 3  dequantize: dV += sP sdO [.], dK += scale sdS sQ [.],
//           dQ_acc += scale sdS sK [.] (FP32 reduction to global)
#include "kernel_common.cuh"

namespace sagebwd {
namespace {

template <int D>
struct BwdCfg {
  static constexpr int NS = D == 128 ? 1 : 2;  // stages of the per-tile operands
  static constexpr int TILE = 128 * D * 2;
  static constexpr int PTILE = 128 * 128 * 2;
  static constexpr int OFF_K = 0;
  static constexpr int OFF_V = OFF_K + TILE;
  static constexpr int OFF_Q = OFF_V + TILE;
  static constexpr int OFF_DO = OFF_Q + NS * TILE;
  static constexpr int OFF_DOQ = OFF_DO + NS * TILE;
  static constexpr int OFF_PT = OFF_DOQ + NS * TILE;
  static constexpr int OFF_DST = OFF_PT + PTILE;
  static constexpr int OFF_VEC = OFF_DST + PTILE;  // L2[128], Dv[128], pmax bits[128], am[16]
  static constexpr int OFF_BAR = OFF_VEC + (128 + 128 + 128 + 16) * 4;
  static constexpr int NBAR = 1 + 6 * NS + 4 + 2 + 1;
  static constexpr int BYTES = OFF_BAR + NBAR * 8 + 16;
  // The tiles need a 1024-byte aligned base; the D = 128 layout leaves no room for padding.
  static constexpr int SMEM = BYTES + 1024 <= 232448 ? BYTES + 1024 : BYTES;
  static constexpr int C_S = 0, C_DP = 128, C_DV = 256, C_DK = 256 + D, C_DQ = 0;
  static_assert(BYTES <= 232448, "shared memory beyond the per-CTA limit");
};

constexpr int kNWG = 4;                      // compute warpgroups
constexpr int kCompute = kNWG * 128;          // compute threads
constexpr int kThreads = kCompute + 128;      // + the producer / MMA warpgroup
constexpr int kQC = 128 / kNWG;               // query columns per compute thread
constexpr uint32_t kRegsLaunch = 96, kRegsLow = 32, kRegsHigh = 112;
static_assert(128 * kRegsLow + kCompute * kRegsHigh <= kThreads * kRegsLaunch, "register split exceeds the launch");

enum BwdSite { bSiteKV = 16, bSiteQFull, bSiteQEmpty, bSiteDOFull, bSiteDOEmpty, bSiteDOQFull, bSiteDOQEmpty,
               bSiteSDP, bSiteDSReady, bSiteAcc, bSiteTmemFree, bSiteAlign, bSiteC1, bSiteC2 };

template <int D, bool CAUSAL>
__global__ void __launch_bounds__(kThreads, 1)
    bwd_kernel(const __grid_constant__ CUtensorMap tmQ, const __grid_constant__ CUtensorMap tmK,
               const __grid_constant__ CUtensorMap tmV, const __grid_constant__ CUtensorMap tmDO,
               const __grid_constant__ CUtensorMap tmDOQ, const BwdParams p) {
  using C = BwdCfg<D>;
  constexpr int NS = C::NS;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = align1024(smem_raw);
  if (C::SMEM == C::BYTES && smem != smem_raw) {
    // no room to realign: report instead of computing on a misaligned layout
    if (threadIdx.x == 0) atomicCAS(p.status, 0, status_timeout(bSiteAlign));
    return;
  }
  float* L2v = reinterpret_cast<float*>(smem + C::OFF_VEC);
  float* Dv = L2v + 128;
  int* pmx = reinterpret_cast<int*>(Dv + 128);  // [128] row maxima of P (P >= 0: float bits order as ints)
  float* am = reinterpret_cast<float*>(pmx + 128);  // [16] per-warp maxima of |dS|
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + C::OFF_BAR);
  uint64_t* bar_kv = bars;
  uint64_t* bar_q_full = bar_kv + 1;
  uint64_t* bar_q_empty = bar_q_full + NS;
  uint64_t* bar_do_full = bar_q_empty + NS;
  uint64_t* bar_do_empty = bar_do_full + NS;
  uint64_t* bar_doq_full = bar_do_empty + NS;
  uint64_t* bar_doq_empty = bar_doq_full + NS;
  uint64_t* bar_sdp = bar_doq_empty + NS;
  uint64_t* bar_ds_ready = bar_sdp + 1;
  uint64_t* bar_acc = bar_ds_ready + 1;
  uint64_t* bar_tmem_free = bar_acc + 1;
  uint64_t* bar_c1 = bar_tmem_free + 1;  // compute threads: LSE / D of the tile stored
  uint64_t* bar_c2 = bar_c1 + 1;         // compute threads: row and tile maxima stored
  uint64_t* bar_final = bar_c2 + 1;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(bar_final + 1);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int BHk = p.B * p.Hkv;
  const int L = blockIdx.x;
  const int j = L / BHk;  // causal: small j has the most query blocks, scheduled first
  const int bhk = L % BHk;
  const int b = bhk / p.Hkv, hk = bhk % p.Hkv;
  const int k0 = j * kBlk;
  const int ib0 = CAUSAL ? j : 0;
  const int nq = p.nb - ib0;
  const int T = p.G * nq;

  if (tid == 0) {
    mbar_init(bar_kv, 1);
    for (int s = 0; s < NS; ++s) {
      mbar_init(bar_q_full + s, 1);
      mbar_init(bar_q_empty + s, 1);
      mbar_init(bar_do_full + s, 1);
      mbar_init(bar_do_empty + s, 1);
      mbar_init(bar_doq_full + s, 1);
      mbar_init(bar_doq_empty + s, 1);
    }
    mbar_init(bar_sdp, 1);
    mbar_init(bar_ds_ready, kCompute);
    mbar_init(bar_acc, 1);
    mbar_init(bar_tmem_free, kCompute);
    mbar_init(bar_c1, kCompute);
    mbar_init(bar_c2, kCompute);
    mbar_init(bar_final, 1);
    *abort_flag = 0;
    fence_mbar_init();
  }
  if (warp == 17) {
    tmem_alloc(tmem_slot, 512);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  const WaitCtx wc{abort_flag, p.status, p.timeout_ns};
  if (warp >= 16) {
    setmaxnreg_dec<kRegsLow>();
    if (warp == 16 && lane == 0) {
      // ---------------------------------------------------------- TMA producer
      int q_iss[NS], do_iss[NS], doq_iss[NS];
      for (int s = 0; s < NS; ++s) q_iss[s] = do_iss[s] = doq_iss[s] = 0;
      mbar_arrive_expect_tx(bar_kv, 2 * C::TILE);
      for (int c = 0; c < D / 64; ++c) {
        tma_load_3d(smem + C::OFF_K + c * 16384, &tmK, bar_kv, c * 64, k0, bhk);
        tma_load_3d(smem + C::OFF_V + c * 16384, &tmV, bar_kv, c * 64, k0, bhk);
      }
      for (int it = 0; it < T; ++it) {
        const int s = it % NS, n = it / NS;
        const int bhq = b * p.Hq + hk * p.G + it / nq;
        const int i0 = (ib0 + it % nq) * kBlk;
        // dO is released first (after dP), then Q^ (after dK), then dO^ (after dV)
        if (it >= NS && !wait1(wc, bar_do_empty + s, (n - 1) & 1, bSiteDOEmpty)) break;
        mbar_arrive_expect_tx(bar_do_full + s, C::TILE);
        for (int c = 0; c < D / 64; ++c)
          tma_load_3d(smem + C::OFF_DO + s * C::TILE + c * 16384, &tmDO, bar_do_full + s, c * 64, i0, bhq);
        do_iss[s] = n + 1;
        if (it >= NS && !wait1(wc, bar_q_empty + s, (n - 1) & 1, bSiteQEmpty)) break;
        mbar_arrive_expect_tx(bar_q_full + s, C::TILE);
        for (int c = 0; c < D / 64; ++c)
          tma_load_3d(smem + C::OFF_Q + s * C::TILE + c * 16384, &tmQ, bar_q_full + s, c * 64, i0, bhq);
        q_iss[s] = n + 1;
        if (it >= NS && !wait1(wc, bar_doq_empty + s, (n - 1) & 1, bSiteDOQEmpty)) break;
        mbar_arrive_expect_tx(bar_doq_full + s, C::TILE);
        for (int c = 0; c < D / 64; ++c)
          tma_load_3d(smem + C::OFF_DOQ + s * C::TILE + c * 16384, &tmDOQ, bar_doq_full + s, c * 64, i0, bhq);
        doq_iss[s] = n + 1;
      }
      drain(bar_kv, 0, p.timeout_ns);
      for (int s = 0; s < NS; ++s) {
        if (q_iss[s]) drain(bar_q_full + s, (q_iss[s] - 1) & 1, p.timeout_ns);
        if (do_iss[s]) drain(bar_do_full + s, (do_iss[s] - 1) & 1, p.timeout_ns);
        if (doq_iss[s]) drain(bar_doq_full + s, (doq_iss[s] - 1) & 1, p.timeout_ns);
      }
    } else if (warp == 17 && lane == 0) {
      // ---------------------------------------------------------- MMA issuer
      const uint32_t idSS = idesc_bf16_f32(128, 128, false, false);  // S^T, dP^T
      const uint32_t idKM = idesc_bf16_f32(128, D, false, true);     // dK, dV: A K-major, B MN-major
      const uint32_t idQM = idesc_bf16_f32(128, D, true, true);      // dQ: A MN-major, B MN-major
      const uint32_t sK = smem_u32(smem + C::OFF_K), sV = smem_u32(smem + C::OFF_V);
      const uint32_t sPT = smem_u32(smem + C::OFF_PT), sDST = smem_u32(smem + C::OFF_DST);
      bool ok = wait1(wc, bar_kv, 0, bSiteKV);
      for (int it = 0; ok && it < T; ++it) {
        const int s = it % NS;
        const uint32_t ph = (it / NS) & 1;
        const uint32_t sQ = smem_u32(smem + C::OFF_Q + s * C::TILE);
        const uint32_t sDO = smem_u32(smem + C::OFF_DO + s * C::TILE);
        const uint32_t sDOQ = smem_u32(smem + C::OFF_DOQ + s * C::TILE);
        if (!wait1(wc, bar_q_full + s, ph, bSiteQFull)) break;
        if (!wait1(wc, bar_do_full + s, ph, bSiteDOFull)) break;
        if (it >= 1 && !wait1(wc, bar_tmem_free, (it - 1) & 1, bSiteTmemFree)) break;
        tc_fence_after();
#pragma unroll
        for (int kk = 0; kk < D / 16; ++kk) {
          const uint32_t off = (kk >> 2) * 16384 + (kk & 3) * 32;
          umma_ss(tmem + C::C_S, sdesc_sw128(sK + off, 16, 1024), sdesc_sw128(sQ + off, 16, 1024), idSS, kk > 0);
        }
#pragma unroll
        for (int kk = 0; kk < D / 16; ++kk) {
          const uint32_t off = (kk >> 2) * 16384 + (kk & 3) * 32;
          umma_ss(tmem + C::C_DP, sdesc_sw128(sV + off, 16, 1024), sdesc_sw128(sDO + off, 16, 1024), idSS, kk > 0);
        }
        umma_commit(bar_sdp);
        umma_commit(bar_do_empty + s);
        if (!wait1(wc, bar_ds_ready, it & 1, bSiteDSReady)) break;
        if (!wait1(wc, bar_doq_full + s, ph, bSiteDOQFull)) break;
        tc_fence_after();
        // dK = dS^T Q^  (A: dS^T tile [key][query], K-major; B: Q^ [query][d], MN-major)
#pragma unroll
        for (int kk = 0; kk < 8; ++kk)
          umma_ss(tmem + C::C_DK, sdesc_sw128(sDST + (kk >> 2) * 16384 + (kk & 3) * 32, 16, 1024),
                  sdesc_sw128(sQ + kk * 2048, 16384, 1024), idKM, kk > 0);
        umma_commit(bar_q_empty + s);
        // dQ = dS K^  (A: the same dS^T tile read MN-major as [query][key]; B: K^ [key][d], MN-major)
#pragma unroll
        for (int kk = 0; kk < 8; ++kk)
          umma_ss(tmem + C::C_DQ, sdesc_sw128(sDST + kk * 2048, 16384, 1024), sdesc_sw128(sK + kk * 2048, 16384, 1024),
                  idQM, kk > 0);
        // dV = P^T dO^  (A: P^T tile [key][query], K-major; B: dO^ [query][d], MN-major)
#pragma unroll
        for (int kk = 0; kk < 8; ++kk)
          umma_ss(tmem + C::C_DV, sdesc_sw128(sPT + (kk >> 2) * 16384 + (kk & 3) * 32, 16, 1024),
                  sdesc_sw128(sDOQ + kk * 2048, 16384, 1024), idKM, kk > 0);
        umma_commit(bar_doq_empty + s);
        umma_commit(bar_acc);
      }
      umma_commit(bar_final);
      drain(bar_final, 0, p.timeout_ns);
    }
  } else {
    setmaxnreg_inc<kRegsHigh>();
    // ------------------------------------------------------------ compute warpgroups
    constexpr int DC = D / kNWG;       // output columns per thread
    const int w = warp >> 2;           // compute warpgroup 0..kNWG-1
    const int r = tid & 127;           // key row == TMEM lane
    const int ct = tid;                // index among the compute threads
    const uint32_t lane_base = (uint32_t)((warp & 3) * 32) << 16;
    const int kglob = k0 + r;
    const bool key_ok = kglob < p.N;
    const float sKv = p.sk[(size_t)bhk * p.nb + j];
    float dv_run[DC], dk_run[DC];
#pragma unroll
    for (int c = 0; c < DC; ++c) dv_run[c] = dk_run[c] = 0.f;

    for (int it = 0; it < T; ++it) {
      const int bhq = b * p.Hq + hk * p.G + it / nq;
      const int ib = ib0 + it % nq;
      const int i0 = ib * kBlk;
      // LSE (base 2) and D of the tile's queries; +inf / 0 past N
      {
        const int q = ct & 127;
        const bool in = i0 + q < p.N;
        if (ct < 128)
          L2v[q] = in ? __fmul_rn(p.lse[(size_t)bhq * p.N + i0 + q], kLog2e) : INFINITY;
        else if (ct < 256)
          Dv[q] = in ? p.D[(size_t)bhq * p.N + i0 + q] : 0.f;
        else if (ct < 384)
          pmx[q] = 0;
      }
      // (an mbarrier rather than bar.sync, so that this wait is bounded too)
      mbar_arrive(bar_c1);
      if (!waitw(wc, bar_c1, it & 1, bSiteC1)) break;
      const float qks = __fmul_rn(__fmul_rn(p.sq[(size_t)bhq * p.nb + ib], sKv), p.c0);
      const bool diag = CAUSAL && ib == j;
      if (!waitw(wc, bar_sdp, it & 1, bSiteSDP)) break;
      tc_fence_after();
      // pass 1
      float pmax = 0.f, amax = 0.f;
#pragma unroll
      for (int c0 = 0; c0 < kQC; c0 += 8) {
        const int col = kQC * w + c0;  // query column within the tile
        uint32_t sv[8], dpv[8];        // S -> P and dP -> dS, converted in place
        tmem_ld8(tmem + lane_base + C::C_S + col, sv);
        tmem_ld8(tmem + lane_base + C::C_DP + col, dpv);
        tmem_ld_wait();
#pragma unroll
        for (int e = 0; e < 8; ++e) {
          float pr = ex2_approx(fmaf(__uint_as_float(sv[e]), qks, -L2v[col + e]));
          if (!key_ok || (diag && col + e < r)) pr = 0.f;
          const float ds = pr * (__uint_as_float(dpv[e]) - Dv[col + e]);
          pmax = fmaxf(pmax, pr);
          amax = fmaxf(amax, fabsf(ds));
          sv[e] = __float_as_uint(pr);
          dpv[e] = __float_as_uint(ds);
        }
        tmem_st8(tmem + lane_base + C::C_S + col, sv);
        tmem_st8(tmem + lane_base + C::C_DP + col, dpv);
      }
      tmem_st_wait();
      atomicMax(pmx + r, __float_as_int(pmax));
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, o));
      if (lane == 0) am[warp] = amax;
      mbar_arrive(bar_c2);
      if (!waitw(wc, bar_c2, it & 1, bSiteC2)) break;
      const float cmax = __int_as_float(pmx[r]);
      float a = am[0];
#pragma unroll
      for (int q = 1; q < kCompute / 32; ++q) a = fmaxf(a, am[q]);
      const bool p_live = cmax >= kMinGroupMax, d_live = a >= kMinGroupMax;
      const float invP = p_live ? __fdiv_rn(127.f, cmax) : 0.f;
      const float sPc = p_live ? __fdiv_rn(cmax, 127.f) : 0.f;
      const float invA = d_live ? __fdiv_rn(127.f, a) : 0.f;
      const float sDS = d_live ? __fdiv_rn(a, 127.f) : 0.f;
      // pass 2: codes into the swizzled A tiles (row = key r, 16-byte chunk = 8 queries)
      const uint32_t pt_base = smem_u32(smem + C::OFF_PT), ds_base = smem_u32(smem + C::OFF_DST);
#pragma unroll
      for (int c0 = 0; c0 < kQC; c0 += 8) {
        const int col = kQC * w + c0;
        uint32_t pv[8], dsv[8];
        tmem_ld8(tmem + lane_base + C::C_S + col, pv);
        tmem_ld8(tmem + lane_base + C::C_DP + col, dsv);
        tmem_ld_wait();
#pragma unroll
        for (int e = 0; e < 8; e += 2) {
          pv[e >> 1] = pack_bf16x2(rint_f32(__fmul_rn(__uint_as_float(pv[e]), invP)),
                                   rint_f32(__fmul_rn(__uint_as_float(pv[e + 1]), invP)));
          dsv[e >> 1] = pack_bf16x2(rint_f32(__fmul_rn(__uint_as_float(dsv[e]), invA)),
                                    rint_f32(__fmul_rn(__uint_as_float(dsv[e + 1]), invA)));
        }
        const uint32_t off = sw128_offset(r, col >> 3);
        st_shared_v4(pt_base + off, pv[0], pv[1], pv[2], pv[3]);
        st_shared_v4(ds_base + off, dsv[0], dsv[1], dsv[2], dsv[3]);
      }
      tc_fence_before();
      fence_proxy_async_smem();
      mbar_arrive(bar_ds_ready);
      if (!waitw(wc, bar_acc, it & 1, bSiteAcc)) break;
      tc_fence_after();
      // pass 3: dequantize the three integer tiles
      const float fv = __fmul_rn(sPc, p.sdo[(size_t)bhq * p.nb + ib]);
      const float fk = __fmul_rn(__fmul_rn(p.sc, sDS), p.sq[(size_t)bhq * p.nb + ib]);
      const float fq = __fmul_rn(__fmul_rn(p.sc, sDS), sKv);
      const int qrow = i0 + r;  // dQ tile: lane r is query row i0 + r
      float* dq_dst = p.dq_acc + ((size_t)bhq * p.N + qrow) * D + w * DC;
#pragma unroll
      for (int c0 = 0; c0 < DC; c0 += 16) {
        uint32_t v[16];
        tmem_ld16(tmem + lane_base + C::C_DV + w * DC + c0, v);
        tmem_ld_wait();
#pragma unroll
        for (int e = 0; e < 16; ++e) dv_run[c0 + e] = fmaf(fv, __uint_as_float(v[e]), dv_run[c0 + e]);
        tmem_ld16(tmem + lane_base + C::C_DK + w * DC + c0, v);
        tmem_ld_wait();
#pragma unroll
        for (int e = 0; e < 16; ++e) dk_run[c0 + e] = fmaf(fk, __uint_as_float(v[e]), dk_run[c0 + e]);
        tmem_ld16(tmem + lane_base + C::C_DQ + w * DC + c0, v);
        tmem_ld_wait();
        if (qrow < p.N) {
#pragma unroll
          for (int e = 0; e < 16; e += 4)
            red_add_v4_f32(dq_dst + c0 + e, fq * __uint_as_float(v[e]), fq * __uint_as_float(v[e + 1]),
                           fq * __uint_as_float(v[e + 2]), fq * __uint_as_float(v[e + 3]));
        }
      }
      tc_fence_before();
      mbar_arrive(bar_tmem_free);
    }
    if (!*abort_flag && key_ok) {
      uint4* dkd = reinterpret_cast<uint4*>(p.dk + ((size_t)bhk * p.N + kglob) * D + w * DC);
      uint4* dvd = reinterpret_cast<uint4*>(p.dv + ((size_t)bhk * p.N + kglob) * D + w * DC);
#pragma unroll
      for (int c = 0; c < DC; c += 8) {
        dkd[c / 8] = make_uint4(pack_bf16x2(dk_run[c], dk_run[c + 1]), pack_bf16x2(dk_run[c + 2], dk_run[c + 3]),
                                pack_bf16x2(dk_run[c + 4], dk_run[c + 5]), pack_bf16x2(dk_run[c + 6], dk_run[c + 7]));
        dvd[c / 8] = make_uint4(pack_bf16x2(dv_run[c], dv_run[c + 1]), pack_bf16x2(dv_run[c + 2], dv_run[c + 3]),
                                pack_bf16x2(dv_run[c + 4], dv_run[c + 5]), pack_bf16x2(dv_run[c + 6], dv_run[c + 7]));
      }
    }
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 17) {
    tc_fence_after();
    tmem_dealloc(tmem, 512);
  }
}

template <int D, bool CAUSAL>
cudaError_t launch_bwd_t(const CUtensorMap& tq, const CUtensorMap& tk, const CUtensorMap& tv, const CUtensorMap& tdo,
                         const CUtensorMap& tdoq, const BwdParams& p, cudaStream_t s) {
  using C = BwdCfg<D>;
  auto kern = bwd_kernel<D, CAUSAL>;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, C::SMEM);
  if (e != cudaSuccess) return e;
  const int grid = p.nb * p.B * p.Hkv;
  kern<<<grid, kThreads, C::SMEM, s>>>(tq, tk, tv, tdo, tdoq, p);
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_bwd(const CUtensorMap& tq, const CUtensorMap& tk, const CUtensorMap& tv, const CUtensorMap& tdo,
                       const CUtensorMap& tdoq, const BwdParams& p, int d, int causal, cudaStream_t s) {
  if (d == 64)
    return causal ? launch_bwd_t<64, true>(tq, tk, tv, tdo, tdoq, p, s)
                  : launch_bwd_t<64, false>(tq, tk, tv, tdo, tdoq, p, s);
  return causal ? launch_bwd_t<128, true>(tq, tk, tv, tdo, tdoq, p, s)
                : launch_bwd_t<128, false>(tq, tk, tv, tdo, tdoq, p, s);
}

}  // namespace sagebwd
