// Fused SageBwd attention backward on sm_103a ("SageBwd: A Trainable Low-bit
// Attention", Abstract: INT8 S recompute, dV = P^T dO, dQ = dS K,
// dK = dS^T Q; "SageAttention3 ... 8-Bit Training" summary, Approach: dO V^T
// kept in 16-bit floating point; FlashAttention-2 backward structure with
// D = rowsum(dO * O) and dS = P (dP - D)).
//
// One CTA owns one 128-key block j of one kv head and loops over HS of the G
// query heads of that kv head and their 128-query blocks i.  dK_j and dV_j are
// summed in registers over those tiles and added once into FP32 accumulators;
// dQ is accumulated across CTAs by TMA bulk reduce-adds into an FP32 workspace.
// CTAs are numbered longest first (causal: small j has the most query blocks),
// and HS is chosen on the host so that this list balances over the SMs.
// Warp roles:
//   warps 0-15   four compute warpgroups: thread (w, r) owns key row r
//                (TMEM lane r), query columns [32w, 32w+32) of the tile and
//                output columns [w d/4, (w+1) d/4) of dK, dV, dQ
//   warp 16      TMA producer (K^_j, V_j once; dO_i, Q^_i, dO^_i per tile)
//   warp 17      TMEM allocation and the MMA-issuing thread
//   warp 18      dQ reducer: bulk reduce-add of each staged dQ tile
//   warp 19      idle (completes the fifth warpgroup: 640 threads launch with
//                96 registers each; that warpgroup drops to kRegsLow and the
//                compute warpgroups rise to kRegsHigh)
// TMEM columns: S^T [0,128), dP^T [128,256), dV [256,256+d), dK [256+d,256+2d),
// dQ [0,d) (reusing S^T once P is consumed).
// Per tile i (MMAs in issue order; the compute passes between them):
//   pass 1  P = 2^(S sQ sK scale log2e - LSE_i log2e), dS = P (dP - D_i), both
//           written back to TMEM in place; row max of P, tile max of |dS|
//   pass 2a code(P^T) per key row (scale max P / 127) -> shared A tile
//     MMA  dV = P^T dO^_i
//   pass 2b code(dS) per tile (scale max|dS| / 127) -> shared A tile
//     MMA  dK = dS^T Q^_i, dQ = dS K^_j
//     MMA  next tile's dP^T = V_j dO_i+1^T (BF16), then S^T = K^_j Q^_i+1^T once
//          the dQ tile has been read (they overlap pass 3)
//   pass 3  dequantize: dQ tile * scale sdS sK -> FP32 staging tile (reduced
//           into global by the reducer warp); dV += sP sdO [.], dK += scale sdS sQ [.]
#include <functional>
#include <queue>
#include <vector>

#include "kernel_common.cuh"

namespace sagebwd {
namespace {

constexpr int kNWG = 4;                      // compute warpgroups
constexpr int kCompute = kNWG * 128;          // compute threads
constexpr int kThreads = kCompute + 128;      // + the producer / MMA / reducer warpgroup
constexpr int kQC = 128 / kNWG;               // query columns per compute thread
constexpr uint32_t kRegsLaunch = 96, kRegsLow = 64, kRegsHigh = 104;
static_assert(128 * kRegsLow + kCompute * kRegsHigh <= kThreads * kRegsLaunch, "register split exceeds the launch");

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
  static constexpr int OFF_PT = OFF_DOQ + NS * TILE;  // P^T codes; with dS^T: the dQ staging tile
  static constexpr int OFF_DST = OFF_PT + PTILE;
  static constexpr int OFF_VEC = OFF_DST + PTILE;  // L2[128], Dv[128], pmax bits[128], am[16]
  static constexpr int OFF_BAR = OFF_VEC + (128 + 128 + 128 + 16) * 4;
  static constexpr int NBAR = 1 + 6 * NS + 12 + 1;
  static constexpr int BYTES = OFF_BAR + NBAR * 8 + 16;
  // The tiles need a 1024-byte aligned base; the d = 128 layout leaves no room for padding.
  static constexpr int SMEM = BYTES + 1024 <= 232448 ? BYTES + 1024 : BYTES;
  static constexpr int C_S = 0, C_DP = 128, C_DV = 256, C_DK = 256 + D, C_DQ = 0;
  static_assert(BYTES <= 232448, "shared memory beyond the per-CTA limit");
  static_assert(128 * D * 4 <= 2 * PTILE, "the FP32 dQ staging tile must fit in the two code tiles");
};

enum BwdSite { bSiteKV = 16, bSiteQFull, bSiteQEmpty, bSiteDOFull, bSiteDOEmpty, bSiteDOQFull, bSiteDOQEmpty,
               bSiteSDP, bSitePTReady, bSiteDSReady, bSiteAccV, bSiteAccQ, bSiteDQRead, bSiteTmemFree, bSiteDQStaged,
               bSiteStagingFree, bSiteStagingFree2, bSiteC1, bSiteC2, bSiteAlign };

template <int D, bool CAUSAL>
__global__ void __launch_bounds__(kThreads, 1)
    bwd_kernel(const __grid_constant__ CUtensorMap tmQ, const __grid_constant__ CUtensorMap tmK,
               const __grid_constant__ CUtensorMap tmV, const __grid_constant__ CUtensorMap tmDO,
               const __grid_constant__ CUtensorMap tmDOQ, const __grid_constant__ CUtensorMap tmDQ,
               const BwdParams p) {
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
  int* pmx = reinterpret_cast<int*>(Dv + 128);      // [128] row maxima of P (P >= 0: float bits order as ints)
  float* am = reinterpret_cast<float*>(pmx + 128);  // [16] per-warp maxima of |dS|
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + C::OFF_BAR);
  uint64_t* bar_kv = bars;
  uint64_t* bar_q_full = bar_kv + 1;
  uint64_t* bar_q_empty = bar_q_full + NS;
  uint64_t* bar_do_full = bar_q_empty + NS;
  uint64_t* bar_do_empty = bar_do_full + NS;
  uint64_t* bar_doq_full = bar_do_empty + NS;
  uint64_t* bar_doq_empty = bar_doq_full + NS;
  uint64_t* bar_sdp = bar_doq_empty + NS;          // S^T and dP^T of the tile are in TMEM
  uint64_t* bar_pt_ready = bar_sdp + 1;            // P^T codes written (compute)
  uint64_t* bar_ds_ready = bar_pt_ready + 1;       // dS codes written, P / dS reads done (compute)
  uint64_t* bar_acc_v = bar_ds_ready + 1;          // dV tile in TMEM
  uint64_t* bar_acc_q = bar_acc_v + 1;             // dK and dQ tiles in TMEM
  uint64_t* bar_dq_read = bar_acc_q + 1;           // dQ tile read out of TMEM (compute)
  uint64_t* bar_tmem_free = bar_dq_read + 1;       // dV, dK tiles read out of TMEM (compute)
  uint64_t* bar_dq_staged = bar_tmem_free + 1;     // FP32 dQ tile written to the staging tile (compute)
  uint64_t* bar_staging_free = bar_dq_staged + 1;  // staging half in the P^T tile read by the reduce (reducer)
  uint64_t* bar_staging_free2 = bar_staging_free + 1;  // staging half in the dS^T tile read (reducer)
  uint64_t* bar_c1 = bar_staging_free2 + 1;        // compute threads: LSE / D of the tile stored
  uint64_t* bar_c2 = bar_c1 + 1;                   // compute threads: row and tile maxima stored
  uint64_t* bar_final = bar_c2 + 1;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(bar_final + 1);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int BHk = p.B * p.Hkv;
  const int NG = p.G / p.HS;  // head groups per kv head
  const int L = blockIdx.x;
  const int j = L / (BHk * NG);  // causal: small j has the most query blocks, scheduled first
  const int bhk = (L / NG) % BHk;
  const int b = bhk / p.Hkv, hk = bhk % p.Hkv;
  const int hq0 = hk * p.G + (L % NG) * p.HS;  // first query head of this CTA
  const int k0 = j * kBlk;
  const int ib0 = CAUSAL ? j : 0;
  const int nq = p.nb - ib0;
  const int T = p.HS * nq;

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
    mbar_init(bar_pt_ready, kCompute);
    mbar_init(bar_ds_ready, kCompute);
    mbar_init(bar_acc_v, 1);
    mbar_init(bar_acc_q, 1);
    mbar_init(bar_dq_read, kCompute);
    mbar_init(bar_tmem_free, kCompute);
    mbar_init(bar_dq_staged, kCompute);
    mbar_init(bar_staging_free, 1);
    mbar_init(bar_staging_free2, 1);
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
        const int bhq = b * p.Hq + hq0 + it / nq;
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
      // Descriptor low words are built once per buffer; the chained MMAs add the per-K-step
      // offsets (no carry: shared addresses stay below 2^18).
      const uint32_t dK_k = sdesc_sw128_lo(smem_u32(smem + C::OFF_K), 16);
      const uint32_t dK_mn = sdesc_sw128_lo(smem_u32(smem + C::OFF_K), 16384);
      const uint32_t dV_k = sdesc_sw128_lo(smem_u32(smem + C::OFF_V), 16);
      const uint32_t dPT_k = sdesc_sw128_lo(smem_u32(smem + C::OFF_PT), 16);
      const uint32_t dDS_k = sdesc_sw128_lo(smem_u32(smem + C::OFF_DST), 16);
      const uint32_t dDS_mn = sdesc_sw128_lo(smem_u32(smem + C::OFF_DST), 16384);
      auto dQ_k = [&](int st) { return sdesc_sw128_lo(smem_u32(smem + C::OFF_Q + st * C::TILE), 16); };
      auto dQ_mn = [&](int st) { return sdesc_sw128_lo(smem_u32(smem + C::OFF_Q + st * C::TILE), 16384); };
      auto dDO_k = [&](int st) { return sdesc_sw128_lo(smem_u32(smem + C::OFF_DO + st * C::TILE), 16); };
      auto dDOQ_mn = [&](int st) { return sdesc_sw128_lo(smem_u32(smem + C::OFF_DOQ + st * C::TILE), 16384); };
      auto chain_kk = [&](uint32_t d_col, uint32_t a_lo, uint32_t b_lo, uint32_t idesc) {
        if constexpr (D == 128)
          umma_chain8_kk(tmem + d_col, sdesc_from_lo(a_lo), sdesc_from_lo(b_lo), idesc);
        else
          umma_chain4_kk(tmem + d_col, sdesc_from_lo(a_lo), sdesc_from_lo(b_lo), idesc);
      };
      auto issue_dp = [&](int s) {
        chain_kk(C::C_DP, dV_k, dDO_k(s), idSS);
        umma_commit(bar_do_empty + s);
      };
      auto issue_s = [&](int s) {
        chain_kk(C::C_S, dK_k, dQ_k(s), idSS);
        umma_commit(bar_sdp);  // also covers the dP^T issued before it
      };
      bool ok = wait1(wc, bar_kv, 0, bSiteKV) && wait1(wc, bar_do_full, 0, bSiteDOFull) &&
                wait1(wc, bar_q_full, 0, bSiteQFull);
      if (ok) {
        tc_fence_after();
        issue_dp(0);
        issue_s(0);
      }
      for (int it = 0; ok && it < T; ++it) {
        const int s = it % NS;
        const uint32_t ph = (it / NS) & 1;
        // dV = P^T dO^  (A: P^T tile [key][query], K-major; B: dO^ [query][d], MN-major)
        if (!wait1(wc, bar_pt_ready, it & 1, bSitePTReady)) break;
        if (!wait1(wc, bar_doq_full + s, ph, bSiteDOQFull)) break;
        if (it >= 1 && !wait1(wc, bar_tmem_free, (it - 1) & 1, bSiteTmemFree)) break;
        tc_fence_after();
        umma_chain8_km(tmem + C::C_DV, sdesc_from_lo(dPT_k), sdesc_from_lo(dDOQ_mn(s)), idKM);
        umma_commit(bar_doq_empty + s);
        umma_commit(bar_acc_v);
        // dK = dS^T Q^  (A: dS^T tile [key][query], K-major; B: Q^ [query][d], MN-major)
        if (!wait1(wc, bar_ds_ready, it & 1, bSiteDSReady)) break;
        tc_fence_after();
        umma_chain8_km(tmem + C::C_DK, sdesc_from_lo(dDS_k), sdesc_from_lo(dQ_mn(s)), idKM);
        umma_commit(bar_q_empty + s);
        // dQ = dS K^  (A: the same dS^T tile read MN-major as [query][key]; B: K^ [key][d], MN-major)
        umma_chain8_mm(tmem + C::C_DQ, sdesc_from_lo(dDS_mn), sdesc_from_lo(dK_mn), idQM);
        umma_commit(bar_acc_q);
        // the next tile's dP^T now (its columns are free), its S^T once the dQ tile is read
        if (it + 1 < T) {
          const int s2 = (it + 1) % NS;
          const uint32_t ph2 = ((it + 1) / NS) & 1;
          if (!wait1(wc, bar_do_full + s2, ph2, bSiteDOFull)) break;
          tc_fence_after();
          issue_dp(s2);
          if (!wait1(wc, bar_q_full + s2, ph2, bSiteQFull)) break;
          if (!wait1(wc, bar_dq_read, it & 1, bSiteDQRead)) break;
          tc_fence_after();
          issue_s(s2);
        }
      }
      // Every MMA issued above must complete before TMEM is released.
      umma_commit(bar_final);
      drain(bar_final, 0, p.timeout_ns);
    } else if (warp == 18 && lane == 0) {
      // ---------------------------------------------------------- dQ reducer
      // The FP32 dQ tile is staged as D/32 boxes of [128 rows][32 floats]: the first half of
      // the boxes in the P^T code tile, the second half in the dS^T code tile.  Each half is
      // its own bulk group, so the P^T tile is released as soon as its half has been read.
      const uint8_t* staging = smem + C::OFF_PT;
      const uint8_t* staging2 = smem + C::OFF_DST;
      for (int it = 0; it < T; ++it) {
        if (!wait1(wc, bar_dq_staged, it & 1, bSiteDQStaged)) break;
        const int bhq = b * p.Hq + hq0 + it / nq;
        const int i0 = (ib0 + it % nq) * kBlk;
#pragma unroll
        for (int bx = 0; bx < D / 64; ++bx) tma_reduce_add_3d(&tmDQ, staging + bx * 16384, bx * 32, i0, bhq);
        bulk_commit_group();
#pragma unroll
        for (int bx = D / 64; bx < D / 32; ++bx)
          tma_reduce_add_3d(&tmDQ, staging2 + (bx - D / 64) * 16384, bx * 32, i0, bhq);
        bulk_commit_group();
        bulk_wait_group_read<1>();
        mbar_arrive(bar_staging_free);
        bulk_wait_group_read<0>();
        mbar_arrive(bar_staging_free2);
      }
      bulk_wait_group0();
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
    const uint32_t pt_base = smem_u32(smem + C::OFF_PT), ds_base = smem_u32(smem + C::OFF_DST);
    uint64_t dv_run[DC / 2], dk_run[DC / 2];  // packed FP32 pairs (columns c, c + 1)
#pragma unroll
    for (int c = 0; c < DC / 2; ++c) dv_run[c] = dk_run[c] = 0ull;

    // Per-tile LSE (base 2) / D values (stored negated: they enter as addends) and
    // block scales, loaded one tile ahead so that their global-memory latency hides
    // behind the current tile.
    const int q_own = ct & 127;
    auto tile_vec = [&](int t) -> float {
      const int bq = b * p.Hq + hq0 + t / nq;
      const int row = (ib0 + t % nq) * kBlk + q_own;
      const bool in = row < p.N;
      if (ct < 128) return in ? -__fmul_rn(p.lse[(size_t)bq * p.N + row], kLog2e) : -INFINITY;
      if (ct < 256) return in ? -p.D[(size_t)bq * p.N + row] : 0.f;
      return 0.f;
    };
    auto tile_sq = [&](int t) { return p.sq[(size_t)(b * p.Hq + hq0 + t / nq) * p.nb + ib0 + t % nq]; };
    auto tile_sdo = [&](int t) { return p.sdo[(size_t)(b * p.Hq + hq0 + t / nq) * p.nb + ib0 + t % nq]; };
    float pf_vec = tile_vec(0), pf_sq = tile_sq(0), pf_sdo = tile_sdo(0);

    for (int it = 0; it < T; ++it) {
      const int ib = ib0 + it % nq;
      // -LSE (base 2) and -D of the tile's queries (-inf / 0 past N); reset the row maxima
      if (ct < 128)
        L2v[q_own] = pf_vec;
      else if (ct < 256)
        Dv[q_own] = pf_vec;
      else if (ct < 384)
        pmx[q_own] = 0;
      const float sQt = pf_sq, sdOt = pf_sdo;
      if (it + 1 < T) {
        pf_vec = tile_vec(it + 1);
        pf_sq = tile_sq(it + 1);
        pf_sdo = tile_sdo(it + 1);
      }
      // (mbarriers rather than bar.sync, so that these waits are bounded too)
      mbar_arrive(bar_c1);
      if (!waitw(wc, bar_c1, it & 1, bSiteC1)) break;
      const float qks = __fmul_rn(__fmul_rn(sQt, sKv), p.c0);
      const bool diag = CAUSAL && ib == j;
      if (!waitw(wc, bar_sdp, it & 1, bSiteSDP)) break;
      tc_fence_after();
      // pass 1
      float pmax = 0.f, amax = 0.f;
      const float2 qks2 = make_float2(qks, qks);
      const bool masked = diag || (k0 + kBlk > p.N);
#pragma unroll
      for (int c0 = 0; c0 < kQC; c0 += 8) {
        const int col = kQC * w + c0;  // query column within the tile
        uint32_t sv[8], dpv[8];        // S -> P and dP -> dS, converted in place
        tmem_ld8(tmem + lane_base + C::C_S + col, sv);
        tmem_ld8(tmem + lane_base + C::C_DP + col, dpv);
        tmem_ld_wait();
#pragma unroll
        for (int e4 = 0; e4 < 8; e4 += 4) {
          const float4 l4 = *reinterpret_cast<const float4*>(L2v + col + e4);  // -LSE log2 e
          const float4 d4 = *reinterpret_cast<const float4*>(Dv + col + e4);   // -D
#pragma unroll
          for (int e2 = 0; e2 < 4; e2 += 2) {
            const int e = e4 + e2;
            const float2 nl = e2 == 0 ? make_float2(l4.x, l4.y) : make_float2(l4.z, l4.w);
            const float2 nd = e2 == 0 ? make_float2(d4.x, d4.y) : make_float2(d4.z, d4.w);
            const float2 x = ffma2(make_float2(__uint_as_float(sv[e]), __uint_as_float(sv[e + 1])), qks2, nl);
            float2 pr = make_float2(ex2_approx(x.x), ex2_approx(x.y));
            if (masked) {
              if (!key_ok || (diag && col + e < r)) pr.x = 0.f;
              if (!key_ok || (diag && col + e + 1 < r)) pr.y = 0.f;
            }
            const float2 ds =
                fmul2(pr, fadd2(make_float2(__uint_as_float(dpv[e]), __uint_as_float(dpv[e + 1])), nd));
            pmax = fmax3(pmax, pr.x, pr.y);
            amax = fmax3(amax, fabsf(ds.x), fabsf(ds.y));
            sv[e] = __float_as_uint(pr.x);
            sv[e + 1] = __float_as_uint(pr.y);
            dpv[e] = __float_as_uint(ds.x);
            dpv[e + 1] = __float_as_uint(ds.y);
          }
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
      // hardware reciprocal (<= 2 ulp) rather than IEEE division: these scales only
      // decide codes of this tile and dequantize it; a code at a rounding tie may differ
      const float invP = p_live ? __fdividef(127.f, cmax) : 0.f;
      const float sPc = p_live ? cmax * (1.f / 127.f) : 0.f;
      const float invA = d_live ? __fdividef(127.f, a) : 0.f;
      const float sDS = d_live ? a * (1.f / 127.f) : 0.f;
      const float2 invP2 = make_float2(invP, invP), invA2 = make_float2(invA, invA);
      // codes = rint(x) by adding and removing 1.5 * 2^23 (exact for |x| < 2^22)
      const float2 kMagic2 = make_float2(12582912.0f, 12582912.0f), kNegMagic2 = make_float2(-12582912.0f, -12582912.0f);
      // the code tiles double as the dQ staging tile: wait until the last reduce has read its half
      if (it >= 1 && !waitw(wc, bar_staging_free, (it - 1) & 1, bSiteStagingFree)) break;
      // pass 2a: codes of P^T into the swizzled A tile (row = key r, 16-byte chunk = 8 queries)
      {
#pragma unroll
        for (int h = 0; h < kQC; h += 16) {
          uint32_t pv[16];
          tmem_ld16(tmem + lane_base + C::C_S + kQC * w + h, pv);
          tmem_ld_wait();
#pragma unroll
          for (int e = 0; e < 16; e += 2) {
            const float2 cd = fadd2(
                fadd2(fmul2(make_float2(__uint_as_float(pv[e]), __uint_as_float(pv[e + 1])), invP2), kMagic2), kNegMagic2);
            pv[e >> 1] = pack_int_bf16x2(cd.x, cd.y);
          }
          st_shared_v4(pt_base + sw128_offset(r, ((kQC * w + h) >> 3)), pv[0], pv[1], pv[2], pv[3]);
          st_shared_v4(pt_base + sw128_offset(r, ((kQC * w + h) >> 3) + 1), pv[4], pv[5], pv[6], pv[7]);
        }
      }
      fence_proxy_async_smem();
      mbar_arrive(bar_pt_ready);
      // pass 2b: codes of dS (one scale per tile)
      if (it >= 1 && !waitw(wc, bar_staging_free2, (it - 1) & 1, bSiteStagingFree2)) break;
      {
#pragma unroll
        for (int h = 0; h < kQC; h += 16) {
          uint32_t dsv[16];
          tmem_ld16(tmem + lane_base + C::C_DP + kQC * w + h, dsv);
          tmem_ld_wait();
#pragma unroll
          for (int e = 0; e < 16; e += 2) {
            const float2 cd = fadd2(
                fadd2(fmul2(make_float2(__uint_as_float(dsv[e]), __uint_as_float(dsv[e + 1])), invA2), kMagic2),
                kNegMagic2);
            dsv[e >> 1] = pack_int_bf16x2(cd.x, cd.y);
          }
          st_shared_v4(ds_base + sw128_offset(r, ((kQC * w + h) >> 3)), dsv[0], dsv[1], dsv[2], dsv[3]);
          st_shared_v4(ds_base + sw128_offset(r, ((kQC * w + h) >> 3) + 1), dsv[4], dsv[5], dsv[6], dsv[7]);
        }
      }
      tc_fence_before();
      fence_proxy_async_smem();
      mbar_arrive(bar_ds_ready);
      // pass 3: dV first (its MMA finishes first), then dQ (frees the S^T columns for
      // the next tile), then dK
      const float fv = __fmul_rn(sPc, sdOt);
      const float fk = __fmul_rn(__fmul_rn(p.sc, sDS), sQt);
      const float fq = __fmul_rn(__fmul_rn(p.sc, sDS), sKv);
      const uint64_t fv2 = pack_f32x2(fv, fv), fk2 = pack_f32x2(fk, fk);
      const float2 fq2 = make_float2(fq, fq);
      if (!waitw(wc, bar_acc_v, it & 1, bSiteAccV)) break;
      tc_fence_after();
#pragma unroll
      for (int c0 = 0; c0 < DC; c0 += 16) {
        uint32_t v[16];
        tmem_ld16(tmem + lane_base + C::C_DV + w * DC + c0, v);
        tmem_ld_wait();
#pragma unroll
        for (int e = 0; e < 16; e += 2) ffma2_acc(dv_run[(c0 + e) >> 1], fv2, v[e], v[e + 1]);
      }
      if (!waitw(wc, bar_acc_q, it & 1, bSiteAccQ)) break;
      tc_fence_after();
      // dQ tile (lane r = query row i0 + r) -> scaled FP32 staging tile, D/32 boxes of
      // [128 rows][32 floats] with the 128-byte swizzle, reduced into global by the reducer warp
#pragma unroll
      for (int c0 = 0; c0 < DC; c0 += 16) {
        uint32_t v[16];
        tmem_ld16(tmem + lane_base + C::C_DQ + w * DC + c0, v);
        tmem_ld_wait();
#pragma unroll
        for (int c4 = 0; c4 < 16; c4 += 4) {
          const int col = w * DC + c0 + c4;
          const int box = col >> 5;  // boxes [0, D/64) in the P^T tile, the rest in the dS^T tile
          const uint32_t box_base = box < D / 64 ? pt_base + box * 16384 : ds_base + (box - D / 64) * 16384;
          const uint32_t off = (uint32_t)(r * 128 + ((((col & 31) >> 2) ^ (r & 7)) << 4));
          const float2 q01 = fmul2(fq2, make_float2(__uint_as_float(v[c4]), __uint_as_float(v[c4 + 1])));
          const float2 q23 = fmul2(fq2, make_float2(__uint_as_float(v[c4 + 2]), __uint_as_float(v[c4 + 3])));
          st_shared_v4(box_base + off, __float_as_uint(q01.x), __float_as_uint(q01.y), __float_as_uint(q23.x),
                       __float_as_uint(q23.y));
        }
      }
      tc_fence_before();
      mbar_arrive(bar_dq_read);
      fence_proxy_async_smem();
      mbar_arrive(bar_dq_staged);
#pragma unroll
      for (int c0 = 0; c0 < DC; c0 += 16) {
        uint32_t v[16];
        tmem_ld16(tmem + lane_base + C::C_DK + w * DC + c0, v);
        tmem_ld_wait();
#pragma unroll
        for (int e = 0; e < 16; e += 2) ffma2_acc(dk_run[(c0 + e) >> 1], fk2, v[e], v[e + 1]);
      }
      tc_fence_before();
      mbar_arrive(bar_tmem_free);
    }
    if (!*abort_flag && key_ok) {
      // this CTA's share of dK_j, dV_j (row kglob, columns [w DC, (w+1) DC)) into the FP32 sums
      float* dka = p.dk_acc + ((size_t)bhk * p.N + kglob) * D + w * DC;
      float* dva = p.dv_acc + ((size_t)bhk * p.N + kglob) * D + w * DC;
#pragma unroll
      for (int c = 0; c < DC; c += 4) {
        const int h = c >> 1;
        red_add_v4_f32(dka + c, lo_f32(dk_run[h]), hi_f32(dk_run[h]), lo_f32(dk_run[h + 1]), hi_f32(dk_run[h + 1]));
        red_add_v4_f32(dva + c, lo_f32(dv_run[h]), hi_f32(dv_run[h]), lo_f32(dv_run[h + 1]), hi_f32(dv_run[h + 1]));
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
                         const CUtensorMap& tdoq, const CUtensorMap& tdq, const BwdParams& p, cudaStream_t s) {
  using C = BwdCfg<D>;
  auto kern = bwd_kernel<D, CAUSAL>;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, C::SMEM);
  if (e != cudaSuccess) return e;
  const int grid = p.nb * p.B * p.Hkv * (p.G / p.HS);
  kern<<<grid, kThreads, C::SMEM, s>>>(tq, tk, tv, tdo, tdoq, tdq, p);
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_bwd(const CUtensorMap& tq, const CUtensorMap& tk, const CUtensorMap& tv, const CUtensorMap& tdo,
                       const CUtensorMap& tdoq, const CUtensorMap& tdq, const BwdParams& p, int d, int causal,
                       cudaStream_t s) {
  if (d == 64)
    return causal ? launch_bwd_t<64, true>(tq, tk, tv, tdo, tdoq, tdq, p, s)
                  : launch_bwd_t<64, false>(tq, tk, tv, tdo, tdoq, tdq, p, s);
  return causal ? launch_bwd_t<128, true>(tq, tk, tv, tdo, tdoq, tdq, p, s)
                : launch_bwd_t<128, false>(tq, tk, tv, tdo, tdoq, tdq, p, s);
}

// Longest-processing-time list schedule of the backward CTAs (one per key block,
// kv head and group of HS query heads, in launch order) on `sms` SMs, for each
// divisor HS of G; a CTA costs its tiles plus one tile of setup and drain.
int bwd_heads_per_cta(int B, int Hkv, int G, int nb, int causal, int sms) {
  if (sms < 1) sms = 1;
  int best_hs = G;
  double best = -1.0;
  for (int hs = G; hs >= 1; --hs) {
    if (G % hs) continue;
    const long long per_j = (long long)B * Hkv * (G / hs);
    std::priority_queue<double, std::vector<double>, std::greater<double>> load;
    for (int m = 0; m < sms; ++m) load.push(0.0);
    double makespan = 0.0;
    for (int j = 0; j < nb; ++j) {
      const double cost = (double)hs * (causal ? nb - j : nb) + 1.0;
      for (long long c = 0; c < per_j; ++c) {
        const double t = load.top() + cost;
        load.pop();
        load.push(t);
        if (t > makespan) makespan = t;
      }
    }
    if (best < 0.0 || makespan < best * 0.995) {  // a smaller HS must win by more than noise
      best = makespan;
      best_hs = hs;
    }
  }
  return best_hs;
}

}  // namespace sagebwd
