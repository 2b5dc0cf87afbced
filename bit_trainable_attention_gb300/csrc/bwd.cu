// Fused SageBwd attention backward on sm_103a ("SageBwd: A Trainable Low-bit
// Attention", Abstract: INT8 S recompute, dV = P^T dO, dQ = dS K,
// dK = dS^T Q; "SageAttention3 ... 8-Bit Training" summary, Approach: dO V^T
// kept in 16-bit floating point; FlashAttention-2 backward structure with
// D = rowsum(dO * O) and dS = P (dP - D)).
//
// One CTA owns one 128-key block j of one kv head and loops over HS of the G
// query heads of that kv head and their 128-query blocks i (the tiles).  dK_j
// and dV_j are summed in registers over those tiles and added once into FP32
// accumulators; dQ is accumulated across CTAs by TMA bulk reduce-adds into an
// FP32 workspace.  CTAs are numbered longest first (causal: small j has the
// most query blocks), and HS is chosen on the host so that this list balances
// over the SMs.
//
// Warp roles (the work of one tile flows S -> A while the tensor core already
// computes the next tile's S^T and dP^T); SWG softmax warpgroups, SWG = 2 on
// d = 128 (640 threads) and 4 on d = 64 (896 threads):
//   warps [0, 4 SWG)          softmax warpgroups S: thread (s, r) owns key row r
//               (TMEM lane r) and queries [QPT s, QPT s + QPT) of the tile, QPT =
//               128 / SWG: P, dS, the codes of P^T (row scale: the slices of a row
//               exchange their maxima through shared memory) written to TMEM as the
//               A operand of dV, and the codes of dS (tile scale) written to shared
//               memory.  d = 128 in three passes: P from S^T (before dP^T is waited
//               for); dS with the P^T codes; the dS codes.  d = 64 in the order P and
//               dS; the P^T codes; the dS codes.
//   next 8 warps  accumulator warpgroups A (two): thread (a, r) owns output
//               columns [a d/2, (a+1) d/2) of row r of dV and dK (FP32 sums in
//               registers) and of the dQ tile it scales into the staging tile
//   last 4 warps  TMA producer of K^, V, dO; TMEM allocation and the MMA-issuing
//               thread; dQ reducer (bulk reduce-add of each staged half); TMA
//               producer of Q^, dO^
// Registers (setmaxnreg from the launch count): d = 128 launch 96, S 64, A 160,
// control 32 (128 * 32 + 256 * 64 + 256 * 160 = 640 * 96); d = 64 launch 72,
// S 64, A 104, control 40.
// TMEM columns: S^T / P [0,128), dP^T / dS [128,256), dV [256,256+d), dK
// [256+d,256+2d).  d = 128: dQ reuses the dV columns once they are read and the
// P^T codes sit in the first 64 dK columns until dV has read them; d = 64: dQ
// [384,448), P^T codes [448,512).
// MMA order per tile i (each waits for what it overwrites or reads):
//   S^T(i+1) = K^_j Q^_i+1^T                 once the P of tile i has been coded
//   dV(i) = P^T codes (TMEM) x dO^_i         while the dS of tile i is coded
//   dP^T(i+1) = V_j dO_i+1^T (BF16)          once the dS of tile i has been coded
//   dK(i) = dS^T Q^_i, dQ(i) = dS K^_j       from the shared dS code tile
// (d = 128 issues dK(i) before dP^T(i+1): the next tile's second pass needs both), so
// the softmax warpgroups of d = 128 start the next tile as soon as S^T(i+1) (committed
// with dV(i)) is there, and those of d = 64 once dP^T(i+1) is.
// With Q-smoothing (QSM) the recomputed logits gain the precomputed term mean_Q(block i) . K'_r
// of the thread's key (one scalar per thread and tile, folded into -LSE), each softmax thread
// sums its dS operand values over its queries, and the accumulator warpgroups add the block
// mean's share of dK = dS^T (Q - mean_Q + mean_Q): scale s_dS (column sum) mean_Q(block i).
// The per-slice column sums go through a small global scratch ring (two tile parities); there
// is no shared memory left for them on d = 128.
// Shared memory at d = 128 has room for one dO, dO^ stage and two Q^ stages, so
// the FP32 dQ staging tile of tile i borrows the dO tile (dO_i+1 has been read by
// dP^T(i+1) by then) and the dS code tile (after dK(i), dQ(i)); d = 64
// double-buffers everything and has its own.
#include <functional>
#include <queue>
#include <vector>

#include "kernel_common.cuh"

namespace sagebwd {
namespace {

constexpr int kDSubMax = 8;  // largest dS sub-scale exponent

// d = 64 layout: softmax warpgroups and the register split (softmax, accumulator, control)
constexpr int kSwg64 = 4;
constexpr uint32_t kRegS64 = 64, kRegA64 = 104, kRegC64 = 40;

template <int D>
struct BwdCfg {
  static constexpr bool ALIAS = D == 128;     // staging tile borrowed from dO and the dS codes
  static constexpr int NS = D == 128 ? 1 : 2;  // dO, dO^ stages (Q^ always has two)
  static constexpr int TILE = 128 * D * 2;
  static constexpr int CTILE = 128 * 128 * 2;  // dS code tile
  // registers per thread after setmaxnreg: softmax, accumulator and control warpgroups.  On
  // d = 128 the accumulators need 160 (fewer spill more and cost more than the control roles
  // gain); on d = 64 the control roles get 64, which removes their spills (bwd 5% faster).
  static constexpr uint32_t REG_S = D == 128 ? 64 : kRegS64, REG_A = D == 128 ? 160 : kRegA64,
                            REG_C = D == 128 ? 32 : kRegC64;
  // softmax warpgroups: on d = 128 two (64 query columns per thread); on d = 64, where the
  // tensor work per tile halves but the softmax work does not, four (32 columns per thread)
  static constexpr int SWG = D == 128 ? 2 : kSwg64;
  static constexpr int QPT = 128 / SWG;                  // query columns per softmax thread
  static constexpr int S_WARPS = 4 * SWG, A_WARP0 = S_WARPS, C_WARP0 = S_WARPS + 8;
  static constexpr int THREADS = 32 * (C_WARP0 + 4);
  static constexpr uint32_t REGS_LAUNCH = (65536 / THREADS) / 8 * 8 > 96 ? 96 : (65536 / THREADS) / 8 * 8;
  static_assert(128 * REG_C + 128 * SWG * REG_S + 256 * REG_A <= THREADS * REGS_LAUNCH,
                "register split exceeds the launch");
  static constexpr int OFF_K = 0;
  static constexpr int OFF_V = OFF_K + TILE;
  static constexpr int OFF_Q = OFF_V + TILE;
  static constexpr int OFF_DO = OFF_Q + 2 * TILE;
  static constexpr int OFF_DOQ = OFF_DO + NS * TILE;
  static constexpr int OFF_DST = OFF_DOQ + NS * TILE;
  static constexpr int OFF_STG = OFF_DST + CTILE;  // own staging tile (d = 64 only)
  static constexpr int OFF_VEC = OFF_STG + (ALIAS ? 0 : 128 * D * 4);
  // Softmax passes per tile.  SPLIT (d = 128): P from S^T alone, then dS once dP^T is there (its
  // MMA runs behind the first pass); the row maxima of P are combined by an atomic maximum on the bit
  // patterns (P >= 0 orders like its unsigned bits) in one slot per row.  Otherwise (d = 64) P and dS
  // in one pass after both products, each slice's row maxima in a slot of its own.
  static constexpr bool SPLIT = D == 128;
  static_assert(SPLIT || SWG > 2, "the fused pass exchanges the row maxima of P among more than two slices");
  static constexpr int PM_FLOATS = SPLIT ? 128 : 128 * SWG;
  // -LSE log2 e [128], -D [128], P^T scale x sdO per row [2][128], |dS| maxima [S_WARPS] (read
  // as 16-byte vectors), dS scale [2], row maxima of P [PM_FLOATS]
  static constexpr int VEC_FLOATS = 128 + 128 + 256 + 2 + S_WARPS + PM_FLOATS;
  static constexpr int OFF_BAR = OFF_VEC + ((VEC_FLOATS * 4 + 15) / 16) * 16;
  static constexpr int NBAR = 1 + 4 + 4 * NS + 19;
  static constexpr int BYTES = OFF_BAR + NBAR * 8 + 16;
  // The tiles need a 1024-byte aligned base; the d = 128 layout leaves no room for padding.
  static constexpr int SMEM = BYTES + 1024 <= 232448 ? BYTES + 1024 : BYTES;
  static constexpr int C_S = 0, C_DP = 128, C_DV = 256, C_DK = 256 + D, C_DQ = ALIAS ? C_DV : 256 + 2 * D,
                       C_PC = ALIAS ? C_DK : 448;  // P^T codes (64 packed columns)
  static_assert(BYTES <= 232448, "shared memory beyond the per-CTA limit");
  static_assert(ALIAS ? (128 * D * 4 == NS * TILE + CTILE) : true, "the staging halves must fill dO and dS codes");
  // FP32 dQ staging: D/32 boxes of [128 rows][32 floats] (16 KB, 128-byte swizzle)
  __host__ __device__ static constexpr int stg_box(int b) {
    return ALIAS ? (b < D / 64 ? OFF_DO + b * 16384 : OFF_DST + (b - D / 64) * 16384) : OFF_STG + b * 16384;
  }
};

enum BwdSite { bSiteKV = 16, bSiteQFull, bSiteQEmpty, bSiteDOFull, bSiteDOEmpty, bSiteDOQFull, bSiteDOQEmpty,
               bSiteS, bSitePTReady, bSiteDSReady, bSiteAccV, bSiteAccQ, bSiteAccK, bSiteTmemFreeV, bSiteDVQFree,
               bSiteTmemFreeK, bSiteStaged, bSiteStgFree, bSiteC1, bSiteC2, bSiteC3, bSiteAlign, bSiteDP };

// The plain instantiations take BwdParams (128 bytes), the Q-smoothing ones BwdQsmParams, the
// debug-dump one (DBG) BwdDumpParams.
template <bool QSM, bool DBG>
struct BwdParamsOf {
  using type = BwdParams;
};
template <>
struct BwdParamsOf<true, false> {
  using type = BwdQsmParams;
};
template <>
struct BwdParamsOf<false, true> {
  using type = BwdDumpParams;
};

// Debug dump record of one tile: P^T codes and dS codes (BF16 [128 keys][128 queries]), then the
// raw FP32 tile products [P^T dO^], [dS^T Q^] ([128 keys][D]) and [dS K^] ([128 queries][D]).
template <int D>
struct BwdDump {
  static constexpr size_t PT = 0, DS = 128 * 128 * 2, DV = 2 * 128 * 128 * 2, DK = DV + 128 * D * 4,
                          DQ = DK + 128 * D * 4, BYTES = DQ + 128 * D * 4;
};
// Maximum of the per-warp maxima am[0, NW) (16-byte aligned shared memory, NW a multiple of 4).
template <int NW>
__device__ __forceinline__ float max_of_warps(const float* am) {
  static_assert(NW % 4 == 0, "whole vectors");
  float a = 0.f;  // the maxima are of absolute values
#pragma unroll
  for (int q = 0; q < NW; q += 4) {
    const float4 v = ld_shared_v4_f32(smem_u32(am + q));
    a = fmax3(a, fmax3(v.x, v.y, v.z), v.w);
  }
  return a;
}
// Write 4 consecutive 32-bit words (16 bytes, 16-byte aligned) to global memory.
__device__ __forceinline__ void dump4(uint8_t* dst, const uint32_t* w) {
  *reinterpret_cast<uint4*>(dst) = make_uint4(w[0], w[1], w[2], w[3]);
}
// Write 16 consecutive 32-bit words (64 bytes, 16-byte aligned) to global memory.
__device__ __forceinline__ void dump16(uint8_t* dst, const uint32_t* w) {
  uint4* d4 = reinterpret_cast<uint4*>(dst);
#pragma unroll
  for (int k = 0; k < 4; ++k) d4[k] = make_uint4(w[4 * k], w[4 * k + 1], w[4 * k + 2], w[4 * k + 3]);
}

// VAR: kValBf16 (error attribution, SAGEBWD_FLAG_BF16_PB / _DS in p.flags) the P^T and / or dS
// operands are the BF16 rounding of the scaled values instead of their integer codes; kValFp8 (the
// FP8 variant) both are the E4M3 rounding of the values scaled to 448 (scales max / 448).
template <int D, bool CAUSAL, bool DSX, bool QSM, bool DBG, int VAR = kValInt8>
__global__ void __launch_bounds__(BwdCfg<D>::THREADS, 1)
    bwd_kernel(const __grid_constant__ CUtensorMap tmQ, const __grid_constant__ CUtensorMap tmK,
               const __grid_constant__ CUtensorMap tmV, const __grid_constant__ CUtensorMap tmDO,
               const __grid_constant__ CUtensorMap tmDOQ, const __grid_constant__ CUtensorMap tmDQ,
               const typename BwdParamsOf<QSM, DBG>::type p) {
  using C = BwdCfg<D>;
  constexpr int NS = C::NS;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = align1024(smem_raw);
  if (C::SMEM == C::BYTES && smem != smem_raw) {
    // no room to realign: report instead of computing on a misaligned layout
    if (threadIdx.x == 0) atomicCAS(p.status, 0, status_timeout(bSiteAlign));
    return;
  }
  float* L2v = reinterpret_cast<float*>(smem + C::OFF_VEC);  // -LSE_q log2 e of the tile's queries
  float* Dv = L2v + 128;                                      // -D_q
  float* fv_ring = Dv + 128;                                  // [2][128] sP_row * sdO per tile parity
  float* am = fv_ring + 256;                                    // [S_WARPS] per-warp maxima of |dS| (16-B aligned)
  float* sds_ring = am + C::S_WARPS;                            // [2] dS scale per tile parity
  uint32_t* pm = reinterpret_cast<uint32_t*>(sds_ring + 2);     // row maxima of P (bits; PM_FLOATS)
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + C::OFF_BAR);
  uint64_t* bar_kv = bars;
  uint64_t* bar_q_full = bar_kv + 1;              // [2]
  uint64_t* bar_q_empty = bar_q_full + 2;         // [2]
  uint64_t* bar_do_full = bar_q_empty + 2;        // [NS]
  uint64_t* bar_do_empty = bar_do_full + NS;      // [NS]
  uint64_t* bar_doq_full = bar_do_empty + NS;     // [NS]
  uint64_t* bar_doq_empty = bar_doq_full + NS;    // [NS] (own staging only)
  uint64_t* bar_s = bar_doq_empty + NS;           // S^T of the tile in TMEM
  uint64_t* bar_dp = bar_s + 1;                   // dP^T of the tile in TMEM
  uint64_t* bar_pt_ready = bar_dp + 1;            // P^T codes in TMEM, P read, row scales stored (S)
  // [2] by tile parity (phase = tile / 2): dS codes in shared memory, dS read, dS scale stored
  // (S).  Two, so that no waiter can miss a phase: the one after next needs every role's work
  // on the tile after this one.
  uint64_t* bar_ds_ready = bar_pt_ready + 1;
  uint64_t* bar_acc_v = bar_ds_ready + 2;         // dV tile in TMEM
  uint64_t* bar_acc_q = bar_acc_v + 1;            // dQ tile in TMEM
  uint64_t* bar_acc_k = bar_acc_q + 1;            // dK tile in TMEM (dS codes no longer read)
  uint64_t* bar_tmem_free_v = bar_acc_k + 1;      // dV tile read (A; gates the aliased dQ)
  uint64_t* bar_dvq_free = bar_tmem_free_v + 1;   // dV and dQ tiles read (A)
  uint64_t* bar_tmem_free_k = bar_dvq_free + 1;   // dK tile read (A)
  uint64_t* bar_staged = bar_tmem_free_k + 1;     // [2] staging half h written (A warpgroup h)
  uint64_t* bar_stg_free = bar_staged + 2;        // [2] staging half h read by the reduce (reducer)
  uint64_t* bar_c1 = bar_stg_free + 2;            // S: the tile's -LSE / -D vectors stored
  uint64_t* bar_c2 = bar_c1 + 1;                  // S: row maxima of P combined
  uint64_t* bar_c3 = bar_c2 + 1;                  // S: |dS| maxima stored
  uint64_t* bar_final = bar_c3 + 1;
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
  auto tile_bhq = [&](int t) { return b * p.Hq + hq0 + t / nq; };
  auto tile_ib = [&](int t) { return ib0 + t % nq; };
  // The same walk without a division per tile: (query head within the CTA's heads, query block)
  // of tile t + 1 from that of tile t, for the roles that need them every tile.
  struct TilePos {
    int h, ib;
  };
  auto next_pos = [&](TilePos t) {
    if (++t.ib == ib0 + nq) {
      t.ib = ib0;
      ++t.h;
    }
    return t;
  };
  auto pos_bhq = [&](TilePos t) { return b * p.Hq + hq0 + t.h; };
  // debug dump record of tile t (DBG instantiation only)
  auto dump_rec = [&](int t) -> uint8_t* {
    if constexpr (DBG)
      return p.dump + (((size_t)tile_bhq(t) * p.nb + tile_ib(t)) * p.nb + j) * BwdDump<D>::BYTES;
    else
      return nullptr;
  };

  if (tid == 0) {
    mbar_init(bar_kv, 1);
    for (int s = 0; s < 2; ++s) {
      mbar_init(bar_q_full + s, 1);
      mbar_init(bar_q_empty + s, 1);
      mbar_init(bar_staged + s, 128);
      mbar_init(bar_stg_free + s, 1);
    }
    for (int s = 0; s < NS; ++s) {
      mbar_init(bar_do_full + s, 1);
      mbar_init(bar_do_empty + s, 1);
      mbar_init(bar_doq_full + s, 1);
      mbar_init(bar_doq_empty + s, 1);
    }
    mbar_init(bar_s, 1);
    mbar_init(bar_dp, 1);
    mbar_init(bar_pt_ready, 128 * C::SWG);
    mbar_init(bar_ds_ready, 128 * C::SWG);
    mbar_init(bar_ds_ready + 1, 128 * C::SWG);
    mbar_init(bar_acc_v, 1);
    mbar_init(bar_acc_q, 1);
    mbar_init(bar_acc_k, 1);
    mbar_init(bar_tmem_free_v, 256);
    mbar_init(bar_dvq_free, 256);
    mbar_init(bar_tmem_free_k, 256);
    mbar_init(bar_c1, 128 * C::SWG);
    mbar_init(bar_c2, 128 * C::SWG);
    mbar_init(bar_c3, 128 * C::SWG);
    mbar_init(bar_final, 1);
    *abort_flag = 0;
    fence_mbar_init();
  }
  if (tid < 128) pm[tid] = 0u;
  constexpr int W_LOAD = C::C_WARP0, W_MMA = C::C_WARP0 + 1, W_RED = C::C_WARP0 + 2, W_LOAD2 = C::C_WARP0 + 3;
  if (warp == W_MMA) {
    tmem_alloc(tmem_slot, 512);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  const WaitCtx wc{abort_flag, p.status, p.timeout_ns};

  if (warp >= C::C_WARP0) {
    setmaxnreg_to<C::REG_C, C::REGS_LAUNCH>();
    if (warp == W_LOAD && lane == 0) {
      // ---------------------------------------------------------- TMA producer: K^, V, dO
      // (the dO slot is released late on d = 128, where it holds tile it-2's dQ staging
      // half 0; Q^ and dO^ have their own producer so that they never queue behind it)
      int do_iss[NS];
      for (int s = 0; s < NS; ++s) do_iss[s] = 0;
      mbar_arrive_expect_tx(bar_kv, 2 * C::TILE);
      for (int c = 0; c < D / 64; ++c) {
        tma_load_3d(smem + C::OFF_K + c * 16384, &tmK, bar_kv, c * 64, k0, bhk);
        tma_load_3d(smem + C::OFF_V + c * 16384, &tmV, bar_kv, c * 64, k0, bhk);
      }
      TilePos pos{0, ib0};
      for (int it = 0; it < T; ++it, pos = next_pos(pos)) {
        const int s = it % NS, n = it / NS;
        if (C::ALIAS) {
          if (it == 1 && !wait1(wc, bar_do_empty, 0, bSiteDOEmpty)) break;
          if (it >= 2 && !wait1(wc, bar_stg_free, (it - 2) & 1, bSiteStgFree)) break;
        } else {
          if (it >= NS && !wait1(wc, bar_do_empty + s, (n - 1) & 1, bSiteDOEmpty)) break;
        }
        mbar_arrive_expect_tx(bar_do_full + s, C::TILE);
        for (int c = 0; c < D / 64; ++c)
          tma_load_3d(smem + C::OFF_DO + s * C::TILE + c * 16384, &tmDO, bar_do_full + s, c * 64,
                      pos.ib * kBlk, pos_bhq(pos));
        do_iss[s] = n + 1;
      }
      // Copies still in flight must land before the CTA's shared memory is released.
      drain(bar_kv, 0, p.timeout_ns);
      for (int s = 0; s < NS; ++s)
        if (do_iss[s]) drain(bar_do_full + s, (do_iss[s] - 1) & 1, p.timeout_ns);
    } else if (warp == W_LOAD2 && lane == 0) {
      // ---------------------------------------------------------- TMA producer: Q^, dO^
      int q_iss[2] = {0, 0}, doq_iss[NS];
      for (int s = 0; s < NS; ++s) doq_iss[s] = 0;
      TilePos pos{0, ib0};
      for (int it = 0; it < T; ++it, pos = next_pos(pos)) {
        const int s = it % NS, n = it / NS, sq = it & 1, nq2 = it >> 1;
        const int bhq = pos_bhq(pos), i0 = pos.ib * kBlk;
        if (it >= 2 && !wait1(wc, bar_q_empty + sq, (nq2 - 1) & 1, bSiteQEmpty)) break;
        mbar_arrive_expect_tx(bar_q_full + sq, C::TILE);
        for (int c = 0; c < D / 64; ++c)
          tma_load_3d(smem + C::OFF_Q + sq * C::TILE + c * 16384, &tmQ, bar_q_full + sq, c * 64, i0, bhq);
        q_iss[sq] = nq2 + 1;
        if (it >= NS && !wait1(wc, bar_doq_empty + s, (n - 1) & 1, bSiteDOQEmpty)) break;
        if (!((p.flags & SAGEBWD_FLAG_DROP_ONE_LOAD) && it == 1)) {  // fault injection skips one load
          mbar_arrive_expect_tx(bar_doq_full + s, C::TILE);
          for (int c = 0; c < D / 64; ++c)
            tma_load_3d(smem + C::OFF_DOQ + s * C::TILE + c * 16384, &tmDOQ, bar_doq_full + s, c * 64, i0, bhq);
          doq_iss[s] = n + 1;
        }
      }
      for (int s = 0; s < 2; ++s)
        if (q_iss[s]) drain(bar_q_full + s, (q_iss[s] - 1) & 1, p.timeout_ns);
      for (int s = 0; s < NS; ++s)
        if (doq_iss[s]) drain(bar_doq_full + s, (doq_iss[s] - 1) & 1, p.timeout_ns);
    } else if (warp == W_MMA && lane == 0) {
      // ---------------------------------------------------------- MMA issuer
      const uint32_t idSS = idesc_bf16_f32(128, 128, false, false);  // S^T, dP^T
      const uint32_t idKM = idesc_bf16_f32(128, D, false, true);     // dK (SS), dV (TS): B MN-major
      const uint32_t idQM = idesc_bf16_f32(128, D, true, true);      // dQ: A MN-major, B MN-major
      // Descriptor low words (the chained MMAs add the per-K-step offsets; no carry:
      // shared addresses stay below 2^18).
      const uint32_t dK_k = sdesc_sw128_lo(smem_u32(smem + C::OFF_K), 16);
      const uint32_t dK_mn = sdesc_sw128_lo(smem_u32(smem + C::OFF_K), 16384);
      const uint32_t dV_k = sdesc_sw128_lo(smem_u32(smem + C::OFF_V), 16);
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
      bool ok = wait1(wc, bar_kv, 0, bSiteKV) && wait1(wc, bar_q_full, 0, bSiteQFull) &&
                wait1(wc, bar_do_full, 0, bSiteDOFull);
      if (ok) {
        tc_fence_after();
        chain_kk(C::C_S, dK_k, dQ_k(0), idSS);
        if (C::SPLIT) umma_commit(bar_s);  // (d = 64 waits for S^T and dP^T together: bar_dp)
        chain_kk(C::C_DP, dV_k, dDO_k(0), idSS);
        umma_commit(bar_dp);
        umma_commit(bar_do_empty);
      }
      for (int it = 0; ok && it < T; ++it) {
        const int s = it % NS;
        const uint32_t ph = (it / NS) & 1;
        const bool next = it + 1 < T;
        // S^T of the next tile once the P of this tile has been read into codes
        if (!wait1(wc, bar_pt_ready, it & 1, bSitePTReady)) break;
        if (next) {
          const int sq = (it + 1) & 1;
          if (!wait1(wc, bar_q_full + sq, ((it + 1) >> 1) & 1, bSiteQFull)) break;
          tc_fence_after();
          chain_kk(C::C_S, dK_k, dQ_k(sq), idSS);
        }
        // dV = P^T dO^: A = the P^T codes in TMEM (row = key, 128 queries = 64 packed
        // columns, 8 per K step), B = dO^ [query][d] read MN-major; it runs while the
        // softmax warpgroups code dS
        if (!wait1(wc, bar_doq_full + s, ph, bSiteDOQFull)) break;
        if (it >= 1 && !wait1(wc, bar_dvq_free, (it - 1) & 1, bSiteDVQFree)) break;
        tc_fence_after();
        {
          const uint32_t bdesc = dDOQ_mn(s);
#pragma unroll
          for (int kk = 0; kk < 8; ++kk)
            umma_ts(tmem + C::C_DV, tmem + C::C_PC + kk * 8, sdesc_from_lo(bdesc + kk * 128), idKM, kk > 0);
        }
        umma_commit(bar_acc_v);
        umma_commit(bar_doq_empty + s);
        if (C::SPLIT && next) umma_commit(bar_s);  // S^T(i+1), issued before dV(i)
        // Once dS is coded: dP^T of the next tile (its columns are free), dK(i) and dQ(i).  On d = 128
        // dK(i) goes first: the next tile's second pass needs both dP^T(i+1) and dK(i) read (the
        // P^T codes share the dK columns), and dK(i) waits behind nothing; on d = 64 the next tile
        // starts with dP^T(i+1).
        if (!wait1(wc, bar_ds_ready + (it & 1), (it >> 1) & 1, bSiteDSReady)) break;
        auto issue_dp = [&]() -> bool {
          if (!next) return true;
          const int s2 = (it + 1) % NS;
          if (!wait1(wc, bar_do_full + s2, ((it + 1) / NS) & 1, bSiteDOFull)) return false;
          tc_fence_after();
          chain_kk(C::C_DP, dV_k, dDO_k(s2), idSS);
          umma_commit(bar_dp);
          if (!C::ALIAS) umma_commit(bar_do_empty + s2);
          return true;
        };
        // dK = dS^T Q^  (A: dS^T codes [key][query], K-major; B: Q^ [query][d], MN-major);
        // on d = 128 it overwrites the P^T codes, so dV must have read them
        auto issue_dk = [&]() -> bool {
          if (C::ALIAS && !wait1(wc, bar_acc_v, it & 1, bSiteAccV)) return false;
          if (it >= 1 && !wait1(wc, bar_tmem_free_k, (it - 1) & 1, bSiteTmemFreeK)) return false;
          tc_fence_after();
          umma_chain8_km(tmem + C::C_DK, sdesc_from_lo(dDS_k), sdesc_from_lo(dQ_mn(it & 1)), idKM);
          if (C::SPLIT) {
            umma_commit(bar_acc_k);
            umma_commit(bar_q_empty + (it & 1));
          }
          return true;
        };
        // dQ = dS K^  (A: the dS^T code tile read MN-major as [query][key]; B: K^ [key][d], MN-major)
        auto issue_dq = [&]() -> bool {
          if (C::ALIAS && !wait1(wc, bar_tmem_free_v, it & 1, bSiteTmemFreeV)) return false;
          tc_fence_after();
          umma_chain8_mm(tmem + C::C_DQ, sdesc_from_lo(dDS_mn), sdesc_from_lo(dK_mn), idQM);
          if (!C::SPLIT) {  // d = 64: dK(i)'s barriers too (one commit point fewer per tile)
            umma_commit(bar_acc_k);
            umma_commit(bar_q_empty + (it & 1));
          }
          umma_commit(bar_acc_q);
          return true;
        };
        if (!(C::SPLIT ? issue_dk() && issue_dp() && issue_dq() : issue_dp() && issue_dk() && issue_dq())) break;
      }
      // Every MMA issued above must complete before TMEM is released.
      umma_commit(bar_final);
      drain(bar_final, 0, p.timeout_ns);
    } else if (warp == W_RED && lane == 0) {
      // ---------------------------------------------------------- dQ reducer
      // Half h of the FP32 dQ tile (columns [h d/2, (h+1) d/2)) is staged by accumulator
      // warpgroup h.  Half 1 goes first: on d = 128 it occupies the dS code tile that the
      // softmax warpgroups need next; both reduces run at once and each half is released
      // as soon as its own read has finished.
      TilePos pos{0, ib0};
      for (int it = 0; it < T; ++it, pos = next_pos(pos)) {
        const int bhq = pos_bhq(pos), i0 = pos.ib * kBlk;
        if (!wait1(wc, bar_staged + 1, it & 1, bSiteStaged)) break;
#pragma unroll
        for (int bx = D / 64; bx < D / 32; ++bx) tma_reduce_add_3d(&tmDQ, smem + C::stg_box(bx), bx * 32, i0, bhq);
        bulk_commit_group();
        if (!wait1(wc, bar_staged, it & 1, bSiteStaged)) break;
#pragma unroll
        for (int bx = 0; bx < D / 64; ++bx) tma_reduce_add_3d(&tmDQ, smem + C::stg_box(bx), bx * 32, i0, bhq);
        bulk_commit_group();
        bulk_wait_group_read<1>();
        mbar_arrive(bar_stg_free + 1);
        bulk_wait_group_read<0>();
        mbar_arrive(bar_stg_free);
      }
      bulk_wait_group0();
    }
  } else if (warp < C::S_WARPS) {
    setmaxnreg_to<C::REG_S, C::REGS_LAUNCH>();
    // ------------------------------------------------------------ softmax warpgroups
    constexpr int QPT = C::QPT;        // query columns per thread
    const int ws = warp >> 2;          // query slice [QPT ws, QPT ws + QPT)
    const int r = tid & 127;           // key row == TMEM lane
    const int qc0 = QPT * ws;          // first query column of this thread
    const uint32_t lane_base = (uint32_t)((warp & 3) * 32) << 16;
    const uint32_t s_addr = tmem + lane_base + C::C_S + qc0, dp_addr = tmem + lane_base + C::C_DP + qc0;
    const uint32_t pc_addr = tmem + lane_base + C::C_PC + qc0 / 2;
    const bool key_ok = k0 + r < p.N;
    const float sKv = p.sk[(size_t)bhk * p.nb + j];
    const uint32_t ds_base = smem_u32(smem + C::OFF_DST);
    const uint32_t l2v_s = smem_u32(L2v), dv_s = smem_u32(Dv);
    // Per tile: half 0 stores -LSE (base 2) of query r, half 1 stores -D (-inf / 0
    // past N); loaded one tile ahead so that their latency hides behind the current tile.
    auto tile_vec = [&](TilePos t) -> float {
      const int row = t.ib * kBlk + r;
      if (row >= p.N) return ws == 0 ? -INFINITY : 0.f;
      const size_t idx = (size_t)pos_bhq(t) * p.N + row;
      return ws == 0 ? -__fmul_rn(p.lse[idx], kLog2e) : -p.D[idx];
    };
    auto tile_sq = [&](TilePos t) { return p.sq[(size_t)pos_bhq(t) * p.nb + t.ib]; };
    auto tile_sdo = [&](TilePos t) { return p.sdo[(size_t)pos_bhq(t) * p.nb + t.ib]; };
    // Q-smoothing: the logit term mean_Q(tile's query block) . K'_r of this thread's key
    auto tile_bias = [&](TilePos t) -> float {
      if constexpr (QSM)
        return p.qbias[((size_t)pos_bhq(t) * p.nb + t.ib) * ((size_t)p.nb * kBlk) + k0 + r];
      else
        return 0.f;
    };
    TilePos pos{0, ib0};  // tile it (tile it + 1 once the prefetch below has advanced it)
    // (only slices 0 and 1 store the vectors, only slice 0 the row factor that needs sdO)
    float pf_vec = ws < 2 ? tile_vec(pos) : 0.f, pf_sq = tile_sq(pos), pf_sdo = ws == 0 ? tile_sdo(pos) : 0.f,
          pf_bias = tile_bias(pos);
    const float2 kMagic2 = make_float2(12582912.0f, 12582912.0f), kNegMagic2 = make_float2(-12582912.0f, -12582912.0f);

    for (int it = 0; it < T; ++it) {
      const int ib = pos.ib;
      // the vectors of the previous tile were last read before its c2 (d = 64) or c3 (d = 128)
      if (ws < 2) (ws == 0 ? L2v : Dv)[r] = pf_vec;
      const float sQt = pf_sq, sdOt = pf_sdo, bk = pf_bias;
      pos = next_pos(pos);
      if (it + 1 < T) {
        if (ws < 2) pf_vec = tile_vec(pos);
        pf_sq = tile_sq(pos);
        if (ws == 0) pf_sdo = tile_sdo(pos);
        if (QSM) pf_bias = tile_bias(pos);
      }
      mbar_arrive(bar_c1);
      if (!waitw(wc, bar_c1, it & 1, bSiteC1)) break;
      const float qks = __fmul_rn(__fmul_rn(sQt, sKv), p.c0);
      const float2 qks2 = make_float2(qks, qks);
      const bool diag = CAUSAL && ib == j;
      const bool masked = diag || (k0 + kBlk > p.N);
      float invA = 0.f, magic_lo = 12582912.0f, magic_hi = 12582912.0f;  // the dS code parameters
      if constexpr (C::SPLIT) {
        // d = 128: P first from S^T alone (its barrier is committed with dV(i-1)'s), dP^T waited
        // for only then
        if (!waitw(wc, bar_s, it & 1, bSiteS)) break;
        tc_fence_after();
        // pass 1: P = 2^(S sQ sK scale log2e - LSE log2e), written over S^T in place, and this
        // thread's share of its row maximum; the next chunk's TMEM load is in flight while a chunk
        // is computed.  dP^T is not read yet: its MMA runs behind this pass.
        float pmax = 0.f;
        {
          uint32_t sv[2][8];
          tmem_ld8(s_addr, sv[0]);
#pragma unroll
          for (int c = 0; c < QPT / 8; ++c) {
            const int cur = c & 1;
            tmem_ld_wait_regs(sv[cur]);
            if (c + 1 < QPT / 8) tmem_ld8(s_addr + (c + 1) * 8, sv[cur ^ 1]);
#pragma unroll
            for (int e4 = 0; e4 < 8; e4 += 4) {
              const int q = qc0 + c * 8 + e4;  // query column within the tile
              const float4 l4 = ld_shared_v4_f32(l2v_s + q * 4);
#pragma unroll
              for (int e2 = 0; e2 < 4; e2 += 2) {
                const int e = e4 + e2;
                float2 nl = e2 == 0 ? make_float2(l4.x, l4.y) : make_float2(l4.z, l4.w);
                if (QSM) nl = fadd2(nl, make_float2(bk, bk));
                const float2 x =
                    ffma2(make_float2(__uint_as_float(sv[cur][e]), __uint_as_float(sv[cur][e + 1])), qks2, nl);
                float2 pr = make_float2(ex2_approx(x.x), ex2_approx(x.y));
                if (masked) {
                  if (!key_ok || (diag && q + e2 < r)) pr.x = 0.f;
                  if (!key_ok || (diag && q + e2 + 1 < r)) pr.y = 0.f;
                }
                pmax = fmax3(pmax, pr.x, pr.y);
                sv[cur][e] = __float_as_uint(pr.x);
                sv[cur][e + 1] = __float_as_uint(pr.y);
              }
            }
            tmem_st8(s_addr + c * 8, sv[cur]);
          }
        }
        // row maximum of P over the slices: the maximum of the bit patterns (P >= 0 orders like
        // its unsigned bits) in a slot that was cleared after every slice had read the previous
        // tile's value (and before this tile's c1)
        atomicMax(pm + r, __float_as_uint(pmax));
        tmem_st_wait();
        mbar_arrive(bar_c2);
        if (!waitw(wc, bar_c2, it & 1, bSiteC2)) break;
        pmax = __uint_as_float(pm[r]);
        constexpr float kMinMax = VAR == kValFp8 ? kMinGroupMaxFp8 : kMinGroupMax;
        constexpr float kQMax = VAR == kValFp8 ? kFp8Max : 127.f;
        // hardware reciprocal (<= 2 ulp) rather than IEEE division: these scales only
        // decide codes of this tile and dequantize it; a code at a rounding tie may differ
        const bool p_live = pmax >= kMinMax;
        const float invP = p_live ? __fdividef(kQMax, pmax) : 0.f;
        const float sPc = p_live ? pmax * (1.f / kQMax) : 0.f;
        if (ws == 0) fv_ring[(it & 1) * 128 + r] = __fmul_rn(sPc, sdOt);
        // pass 2: dS = P (dP - D), written over dP^T in place, with this thread's maxima of |dS|,
        // and the codes of P^T (row scale; 8 queries -> 4 packed columns) over the previous tile's
        // codes: dV(i-1) must have read them (d = 64), and on d = 128, where they share the dK
        // columns, dK(i-1) must have been read too (which implies the former)
        if (it >= 1 && !(C::ALIAS ? waitw(wc, bar_tmem_free_k, (it - 1) & 1, bSiteTmemFreeK)
                                  : waitw(wc, bar_acc_v, (it - 1) & 1, bSiteAccV)))
          break;
        if (!waitw(wc, bar_dp, it & 1, bSiteDP)) break;
        tc_fence_after();
        // amax: |dS| maximum of this thread's first 32 queries, amax_hi: of its last 32 (the
        // two sub-scale groups; without sub-scales one maximum covers all 64)
        float amax = 0.f, amax_hi = 0.f;
        {
          const float2 invP2 = make_float2(invP, invP);
          const bool pt_bf16 = VAR == kValBf16 && (p.flags & SAGEBWD_FLAG_BF16_PB);
          uint32_t pv[2][8], dpv[2][8];
          tmem_ld8(s_addr, pv[0]);
          tmem_ld8(dp_addr, dpv[0]);
#pragma unroll
          for (int c = 0; c < QPT / 8; ++c) {
            const int cur = c & 1;
            tmem_ld_wait_regs(pv[cur]);
            tmem_ld_wait_regs(dpv[cur]);
            if (c + 1 < QPT / 8) {
              tmem_ld8(s_addr + (c + 1) * 8, pv[cur ^ 1]);
              tmem_ld8(dp_addr + (c + 1) * 8, dpv[cur ^ 1]);
            }
            uint32_t pk[4];
#pragma unroll
            for (int e4 = 0; e4 < 8; e4 += 4) {
              const float4 d4 = ld_shared_v4_f32(dv_s + (qc0 + c * 8 + e4) * 4);
#pragma unroll
              for (int e2 = 0; e2 < 4; e2 += 2) {
                const int e = e4 + e2;
                const float2 nd = e2 == 0 ? make_float2(d4.x, d4.y) : make_float2(d4.z, d4.w);
                const float2 pr = make_float2(__uint_as_float(pv[cur][e]), __uint_as_float(pv[cur][e + 1]));
                const float2 ds = fmul2(
                    pr, fadd2(make_float2(__uint_as_float(dpv[cur][e]), __uint_as_float(dpv[cur][e + 1])), nd));
                if (DSX && c >= 4)
                  amax_hi = fmax3(amax_hi, fabsf(ds.x), fabsf(ds.y));
                else
                  amax = fmax3(amax, fabsf(ds.x), fabsf(ds.y));
                dpv[cur][e] = __float_as_uint(ds.x);
                dpv[cur][e + 1] = __float_as_uint(ds.y);
                const float2 sc2 = fmul2(pr, invP2);
                if (VAR == kValFp8) {
                  pk[e >> 1] = e4m3x2_bf16x2(sc2.x, sc2.y);
                } else if (pt_bf16) {
                  pk[e >> 1] = pack_bf16x2(sc2.x, sc2.y);
                } else {
                  const float2 cd = fadd2(fadd2(sc2, kMagic2), kNegMagic2);
                  pk[e >> 1] = pack_int_bf16x2(cd.x, cd.y);
                }
              }
            }
            tmem_st8(dp_addr + c * 8, dpv[cur]);
            tmem_st4(pc_addr + c * 4, pk);
            if constexpr (DBG) dump4(dump_rec(it) + BwdDump<D>::PT + ((size_t)r * 128 + qc0 + c * 8) * 2, pk);
          }
        }
        tmem_st_wait();
        tc_fence_before();
        mbar_arrive(bar_pt_ready);
        // tile maximum of |dS| over the softmax warps
        const float amax_lo = amax;
        if (DSX) amax = fmaxf(amax, amax_hi);
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, o));
        if (lane == 0) am[warp] = amax;
        mbar_arrive(bar_c3);
        if (!waitw(wc, bar_c3, it & 1, bSiteC3)) break;
        // every slice has read the row maximum of P: clear it for the next tile
        if (ws == 0) pm[r] = 0u;
        const float a = max_of_warps<C::S_WARPS>(am);
        const bool d_live = a >= kMinMax;
        invA = d_live ? __fdividef(kQMax, a) : 0.f;
        const float sDS = d_live ? a * (1.f / kQMax) : 0.f;
        // dS sub-scales: group g of this thread's key gets k = floor(log2(a / max_g)) in
        // [0, 8] (0 below 2^-100), from the binary exponents and fractions; its operand values
        // are rint(dS * invA * 2^k) * 2^-k (a code times 2^-k, exact in BF16).  Adding and
        // subtracting 1.5 * 2^(23-k), whose unit in the last place is 2^-k, rounds to that
        // grid directly (ties to even), so the sub-scale costs no instruction per element.
        if (DSX) {
          auto subexp = [&](float g) -> int {
            if (!(g >= 0x1p-100f)) return 0;
            const uint32_t ua = __float_as_uint(a), ug = __float_as_uint(g);
            const int k = (int)(ua >> 23) - (int)(ug >> 23) - ((ua & 0x7FFFFFu) < (ug & 0x7FFFFFu) ? 1 : 0);
            return min(k, kDSubMax);
          };
          magic_lo = __int_as_float(((127 + 23 - subexp(amax_lo)) << 23) | 0x400000);
          magic_hi = __int_as_float(((127 + 23 - subexp(amax_hi)) << 23) | 0x400000);
        }
        if (tid == 0) sds_ring[it & 1] = sDS;
      } else {
        // d = 64: S^T and dP^T together (its dP^T product is short and done by the time S^T is)
        float* pmf = reinterpret_cast<float*>(pm);  // [SWG][128] row maxima of P per slice
        if (!waitw(wc, bar_dp, it & 1, bSiteDP)) break;  // (its commit follows S^T's MMAs too)
        tc_fence_after();
        // pass 1: P = 2^(S sQ sK scale log2e - LSE log2e), dS = P (dP - D), written back in
        // place; the next chunk's TMEM loads are in flight while a chunk is computed
        // amax: |dS| maximum of this thread's first 32 queries, amax_hi: of its last 32 (the
        // two sub-scale groups; without sub-scales one maximum covers all 64)
        float pmax = 0.f, amax = 0.f, amax_hi = 0.f;
        {
          uint32_t sv[2][8], dpv[2][8];
          tmem_ld8(s_addr, sv[0]);
          tmem_ld8(dp_addr, dpv[0]);
#pragma unroll
          for (int c = 0; c < QPT / 8; ++c) {
            const int cur = c & 1;
            tmem_ld_wait_regs(sv[cur]);
            tmem_ld_wait_regs(dpv[cur]);
            if (c + 1 < QPT / 8) {
              tmem_ld8(s_addr + (c + 1) * 8, sv[cur ^ 1]);
              tmem_ld8(dp_addr + (c + 1) * 8, dpv[cur ^ 1]);
            }
#pragma unroll
            for (int e4 = 0; e4 < 8; e4 += 4) {
              const int q = qc0 + c * 8 + e4;  // query column within the tile
              const float4 l4 = ld_shared_v4_f32(l2v_s + q * 4);
              const float4 d4 = ld_shared_v4_f32(dv_s + q * 4);
#pragma unroll
              for (int e2 = 0; e2 < 4; e2 += 2) {
                const int e = e4 + e2;
                float2 nl = e2 == 0 ? make_float2(l4.x, l4.y) : make_float2(l4.z, l4.w);
                if (QSM) nl = fadd2(nl, make_float2(bk, bk));
                const float2 nd = e2 == 0 ? make_float2(d4.x, d4.y) : make_float2(d4.z, d4.w);
                const float2 x =
                    ffma2(make_float2(__uint_as_float(sv[cur][e]), __uint_as_float(sv[cur][e + 1])), qks2, nl);
                float2 pr = make_float2(ex2_approx(x.x), ex2_approx(x.y));
                if (masked) {
                  if (!key_ok || (diag && q + e2 < r)) pr.x = 0.f;
                  if (!key_ok || (diag && q + e2 + 1 < r)) pr.y = 0.f;
                }
                const float2 ds = fmul2(
                    pr, fadd2(make_float2(__uint_as_float(dpv[cur][e]), __uint_as_float(dpv[cur][e + 1])), nd));
                pmax = fmax3(pmax, pr.x, pr.y);
                if (DSX && c >= 4)
                  amax_hi = fmax3(amax_hi, fabsf(ds.x), fabsf(ds.y));
                else
                  amax = fmax3(amax, fabsf(ds.x), fabsf(ds.y));
                sv[cur][e] = __float_as_uint(pr.x);
                sv[cur][e + 1] = __float_as_uint(pr.y);
                dpv[cur][e] = __float_as_uint(ds.x);
                dpv[cur][e + 1] = __float_as_uint(ds.y);
              }
            }
            tmem_st8(s_addr + c * 8, sv[cur]);
            tmem_st8(dp_addr + c * 8, dpv[cur]);
          }
        }
        tmem_st_wait();
        // tile maximum of |dS| over the 8 softmax warps; row maximum of P over the two halves:
        // half 0 publishes its maximum, half 1 combines and publishes the row's
        const float amax_lo = amax;
        if (DSX) amax = fmaxf(amax, amax_hi);
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, o));
        if (lane == 0) am[warp] = amax;
        pmf[ws * 128 + r] = pmax;
        mbar_arrive(bar_c2);
        if (!waitw(wc, bar_c2, it & 1, bSiteC2)) break;
        // every slice reads all partial maxima (the next tile writes them only after its c1)
        pmax = pmf[r];
#pragma unroll
        for (int q = 1; q < C::SWG; ++q) pmax = fmaxf(pmax, pmf[q * 128 + r]);
        const float a = max_of_warps<C::S_WARPS>(am);
        constexpr float kMinMax = VAR == kValFp8 ? kMinGroupMaxFp8 : kMinGroupMax;
        const bool p_live = pmax >= kMinMax, d_live = a >= kMinMax;
        // hardware reciprocal (<= 2 ulp) rather than IEEE division: these scales only
        // decide codes of this tile and dequantize it; a code at a rounding tie may differ
        constexpr float kQMax = VAR == kValFp8 ? kFp8Max : 127.f;
        const float invP = p_live ? __fdividef(kQMax, pmax) : 0.f;
        const float sPc = p_live ? pmax * (1.f / kQMax) : 0.f;
        invA = d_live ? __fdividef(kQMax, a) : 0.f;
        const float sDS = d_live ? a * (1.f / kQMax) : 0.f;
        // dS sub-scales: group g of this thread's key gets k = floor(log2(a / max_g)) in
        // [0, 8] (0 below 2^-100), from the binary exponents and fractions; its operand values
        // are rint(dS * invA * 2^k) * 2^-k (a code times 2^-k, exact in BF16).  Adding and
        // subtracting 1.5 * 2^(23-k), whose unit in the last place is 2^-k, rounds to that
        // grid directly (ties to even), so the sub-scale costs no instruction per element.
        if (DSX) {
          auto subexp = [&](float g) -> int {
            if (!(g >= 0x1p-100f)) return 0;
            const uint32_t ua = __float_as_uint(a), ug = __float_as_uint(g);
            const int k = (int)(ua >> 23) - (int)(ug >> 23) - ((ua & 0x7FFFFFu) < (ug & 0x7FFFFFu) ? 1 : 0);
            return min(k, kDSubMax);
          };
          magic_lo = __int_as_float(((127 + 23 - subexp(amax_lo)) << 23) | 0x400000);
          magic_hi = __int_as_float(((127 + 23 - subexp(amax_hi)) << 23) | 0x400000);
        }
        if (ws == 0) fv_ring[(it & 1) * 128 + r] = __fmul_rn(sPc, sdOt);
        if (tid == 0) sds_ring[it & 1] = sDS;
        // pass 2a: codes of P^T (row scale), 32 queries -> 16 packed columns, over the previous
        // tile's codes: dV(i-1) must have read them (d = 64), and on d = 128, where they share
        // the dK columns, dK(i-1) must have been read too (which implies the former)
        if (it >= 1 && !(C::ALIAS ? waitw(wc, bar_tmem_free_k, (it - 1) & 1, bSiteTmemFreeK)
                                  : waitw(wc, bar_acc_v, (it - 1) & 1, bSiteAccV)))
          break;
        tc_fence_after();
        {
          const float2 invP2 = make_float2(invP, invP);
          const bool pt_bf16 = VAR == kValBf16 && (p.flags & SAGEBWD_FLAG_BF16_PB);
#pragma unroll
          for (int c0 = 0; c0 < QPT; c0 += 32) {
            uint32_t v[32];
            tmem_ld32(s_addr + c0, v);
            tmem_ld_wait();
            uint32_t pk[16];
#pragma unroll
            for (int e = 0; e < 32; e += 2) {
              const float2 sc2 = fmul2(make_float2(__uint_as_float(v[e]), __uint_as_float(v[e + 1])), invP2);
              if (VAR == kValFp8) {
                pk[e >> 1] = e4m3x2_bf16x2(sc2.x, sc2.y);
              } else if (pt_bf16) {
                pk[e >> 1] = pack_bf16x2(sc2.x, sc2.y);
              } else {
                const float2 cd = fadd2(fadd2(sc2, kMagic2), kNegMagic2);
                pk[e >> 1] = pack_int_bf16x2(cd.x, cd.y);
              }
            }
            if constexpr (DBG) dump16(dump_rec(it) + BwdDump<D>::PT + ((size_t)r * 128 + qc0 + c0) * 2, pk);
            tmem_st16(pc_addr + (c0 >> 1), pk);
          }
        }
        tmem_st_wait();
        tc_fence_before();
        mbar_arrive(bar_pt_ready);
      }
      // pass 3: codes of dS (tile scale) into the shared A tile [key r][query], 16-byte
      // chunk = 8 queries, 128-byte swizzle, over the previous tile's codes: dK(i-1) and
      // dQ(i-1) must have read them (d = 64), and on d = 128 the tile is then the previous
      // tile's dQ staging half 1 until the reducer has read it (which implies the former)
      if (it >= 1 && !(C::ALIAS ? waitw(wc, bar_stg_free + 1, (it - 1) & 1, bSiteStgFree)
                                : waitw(wc, bar_acc_q, (it - 1) & 1, bSiteAccQ)))
        break;
      // Q-smoothing on d = 64: the accumulator warpgroups have finished tile i-1 (so they read the
      // column sums of tile i-2 from this parity's slot, and waited for tile i-1's dS release
      // before this tile's can complete); on d = 128 the staging wait above implies both
      if (QSM && !C::ALIAS && it >= 1 && !waitw(wc, bar_dvq_free, (it - 1) & 1, bSiteDVQFree)) break;
      float2 csum = make_float2(0.f, 0.f);  // this thread's sum of its dS operand values (exact in FP32)
      {
        const bool ds_bf16 = VAR == kValBf16 && (p.flags & SAGEBWD_FLAG_BF16_DS);
#pragma unroll
        for (int c0 = 0; c0 < QPT; c0 += 32) {
          const float2 invA2 = make_float2(invA, invA);
          const float mg = c0 == 0 ? magic_lo : magic_hi;
          const float2 magic2 = make_float2(mg, mg), neg_magic2 = make_float2(-mg, -mg);
          uint32_t v[32];
          tmem_ld32(dp_addr + c0, v);
          tmem_ld_wait();
#pragma unroll
          for (int e = 0; e < 32; e += 2) {
            const float2 sc2 = fmul2(make_float2(__uint_as_float(v[e]), __uint_as_float(v[e + 1])), invA2);
            if (VAR == kValFp8) {
              v[e >> 1] = e4m3x2_bf16x2(sc2.x, sc2.y);
              continue;
            }
            if (ds_bf16) {
              v[e >> 1] = pack_bf16x2(sc2.x, sc2.y);
              continue;
            }
            const float2 cd = fadd2(fadd2(sc2, magic2), neg_magic2);
            if (QSM) csum = fadd2(csum, cd);
            v[e >> 1] = pack_int_bf16x2(cd.x, cd.y);
          }
          if constexpr (DBG) dump16(dump_rec(it) + BwdDump<D>::DS + ((size_t)r * 128 + qc0 + c0) * 2, v);
#pragma unroll
          for (int h = 0; h < 4; ++h)
            st_shared_v4(ds_base + sw128_offset(r, ((qc0 + c0) >> 3) + h), v[4 * h], v[4 * h + 1], v[4 * h + 2],
                         v[4 * h + 3]);
        }
      }
      if constexpr (QSM) p.cs_part[(((size_t)blockIdx.x * 2 + (it & 1)) * C::SWG + ws) * 128 + r] = csum.x + csum.y;
      tc_fence_before();
      fence_proxy_async_smem();
      mbar_arrive(bar_ds_ready + (it & 1));
    }
  } else {
    setmaxnreg_to<C::REG_A, C::REGS_LAUNCH>();
    // ------------------------------------------------------------ accumulator warpgroups
    constexpr int DH = D / 2;           // output columns per thread
    const int wa = (warp - C::A_WARP0) >> 2;  // accumulator warpgroup 0 / 1
    const int r = tid & 127;            // key row == TMEM lane
    const uint32_t lane_base = (uint32_t)((warp & 3) * 32) << 16;
    const int kglob = k0 + r;
    const float sKv = p.sk[(size_t)bhk * p.nb + j];
    uint64_t dv_run[DH / 2], dk_run[DH / 2];  // packed FP32 pairs (columns c, c + 1)
#pragma unroll
    for (int c = 0; c < DH / 2; ++c) dv_run[c] = dk_run[c] = 0ull;
    TilePos apos{0, ib0};
    float sq_next = p.sq[(size_t)pos_bhq(apos) * p.nb + apos.ib];

    for (int it = 0; it < T; ++it) {
      const float sQt = sq_next;
      const TilePos cur = apos;  // this tile
      apos = next_pos(apos);
      if (it + 1 < T) sq_next = p.sq[(size_t)pos_bhq(apos) * p.nb + apos.ib];
      // Q-smoothing: this warpgroup's half of mean_Q(tile's query block) into L1 now, read at
      // the end of the tile (a quarter of a line per lane group: lanes 0..DH/32-1 of each warp)
      if constexpr (QSM && C::ALIAS) {  // (on d = 64 the prefetch measured slower)
        if (lane < DH / 32)
          prefetch_l1(p.qmean + ((size_t)pos_bhq(cur) * p.nb + cur.ib) * D + wa * DH + lane * 32);
      }
      if (!waitw(wc, bar_acc_v, it & 1, bSiteAccV)) break;
      // the row scales of P were stored before the P^T codes were released
      if (!waitw(wc, bar_pt_ready, it & 1, bSitePTReady)) break;
      tc_fence_after();
      const float fv = fv_ring[(it & 1) * 128 + r];
      // the dS scale and the factors of the dK and dQ tiles: on d = 64 stored with the row scales
      // of P, on d = 128 only before the dS codes are released (read after dK(i) below)
      float sDS = 0.f, fk = 0.f, fq = 0.f;
      if constexpr (!C::SPLIT) {
        sDS = sds_ring[it & 1];
        fk = __fmul_rn(__fmul_rn(p.sc, sDS), sQt);
        fq = __fmul_rn(__fmul_rn(p.sc, sDS), sKv);
      }
      {
        const uint64_t fv2 = pack_f32x2(fv, fv);
#pragma unroll
        for (int c0 = 0; c0 < DH; c0 += 16) {
          uint32_t v[16];
          tmem_ld16(tmem + lane_base + C::C_DV + wa * DH + c0, v);
          tmem_ld_wait_regs(v);
          if constexpr (DBG) dump16(dump_rec(it) + BwdDump<D>::DV + ((size_t)r * D + wa * DH + c0) * 4, v);
#pragma unroll
          for (int e = 0; e < 16; e += 2) ffma2_acc(dv_run[(c0 + e) >> 1], fv2, v[e], v[e + 1]);
        }
      }
      if (C::ALIAS) {
        tc_fence_before();
        mbar_arrive(bar_tmem_free_v);
      }
      if (!waitw(wc, bar_acc_k, it & 1, bSiteAccK)) break;
      if constexpr (C::SPLIT) {
        if (!waitw(wc, bar_ds_ready + (it & 1), (it >> 1) & 1, bSiteDSReady)) break;
        sDS = sds_ring[it & 1];
        fk = __fmul_rn(__fmul_rn(p.sc, sDS), sQt);
        fq = __fmul_rn(__fmul_rn(p.sc, sDS), sKv);
      }
      tc_fence_after();
      {
        const uint64_t fk2 = pack_f32x2(fk, fk);
#pragma unroll
        for (int c0 = 0; c0 < DH; c0 += 16) {
          uint32_t v[16];
          tmem_ld16(tmem + lane_base + C::C_DK + wa * DH + c0, v);
          tmem_ld_wait_regs(v);
          if constexpr (DBG) dump16(dump_rec(it) + BwdDump<D>::DK + ((size_t)r * D + wa * DH + c0) * 4, v);
#pragma unroll
          for (int e = 0; e < 16; e += 2) ffma2_acc(dk_run[(c0 + e) >> 1], fk2, v[e], v[e + 1]);
        }
      }
      tc_fence_before();
      mbar_arrive(bar_tmem_free_k);
      if constexpr (QSM) {
        // Q-smoothing, while dQ(i) runs: dK_r += scale s_dS (sum over the tile's queries of the dS
        // operand values) mean_Q(block i); the slices' column sums were stored before dS was
        // released (on d = 128 waited for above)
        if (!C::SPLIT && !waitw(wc, bar_ds_ready + (it & 1), (it >> 1) & 1, bSiteDSReady)) break;
        const float* cs = p.cs_part + ((size_t)blockIdx.x * 2 + (it & 1)) * C::SWG * 128 + r;
        float colsum = cs[0];
#pragma unroll
        for (int q = 1; q < C::SWG; ++q) colsum += cs[q * 128];
        const float wcs = __fmul_rn(__fmul_rn(p.sc, sDS), colsum);
        const uint64_t w2 = pack_f32x2(wcs, wcs);
        const float4* mq =
            reinterpret_cast<const float4*>(p.qmean + ((size_t)pos_bhq(cur) * p.nb + cur.ib) * D + wa * DH);
#pragma unroll
        for (int c = 0; c < DH; c += 4) {
          const float4 m = __ldg(mq + c / 4);
          ffma2_acc(dk_run[c >> 1], w2, __float_as_uint(m.x), __float_as_uint(m.y));
          ffma2_acc(dk_run[(c >> 1) + 1], w2, __float_as_uint(m.z), __float_as_uint(m.w));
        }
      }
      // dQ tile (lane r = query row i0 + r) -> scaled FP32 staging half wa: boxes of
      // [128 rows][32 floats] with the 128-byte swizzle, reduced into global by the reducer
      // (on d = 128 half 0 overwrites dO_i+1, which dP^T(i+1) has read, and half 1 the dS
      // codes, which dK(i) and dQ(i) have read)
      if (!waitw(wc, bar_acc_q, it & 1, bSiteAccQ)) break;
      if (!C::ALIAS && it >= 1 && !waitw(wc, bar_stg_free + wa, (it - 1) & 1, bSiteStgFree)) break;
      tc_fence_after();
      {
        const float2 fq2 = make_float2(fq, fq);
#pragma unroll
        for (int c0 = 0; c0 < DH; c0 += 16) {
          uint32_t v[16];
          tmem_ld16(tmem + lane_base + C::C_DQ + wa * DH + c0, v);
          tmem_ld_wait_regs(v);
          if constexpr (DBG) dump16(dump_rec(it) + BwdDump<D>::DQ + ((size_t)r * D + wa * DH + c0) * 4, v);
#pragma unroll
          for (int c4 = 0; c4 < 16; c4 += 4) {
            const int col = wa * DH + c0 + c4;
            const uint32_t box_base = smem_u32(smem + C::stg_box(col >> 5));
            const uint32_t off = (uint32_t)(r * 128 + ((((col & 31) >> 2) ^ (r & 7)) << 4));
            const float2 q01 = fmul2(fq2, make_float2(__uint_as_float(v[c4]), __uint_as_float(v[c4 + 1])));
            const float2 q23 = fmul2(fq2, make_float2(__uint_as_float(v[c4 + 2]), __uint_as_float(v[c4 + 3])));
            st_shared_v4(box_base + off, __float_as_uint(q01.x), __float_as_uint(q01.y), __float_as_uint(q23.x),
                         __float_as_uint(q23.y));
          }
        }
      }
      fence_proxy_async_smem();
      mbar_arrive(bar_staged + wa);
      tc_fence_before();
      mbar_arrive(bar_dvq_free);
    }
    if (!*abort_flag && kglob < p.N) {
      const size_t row = ((size_t)bhk * p.N + kglob) * D + wa * DH;
      if (p.flags & kBwdDirectDKDV) {
        // the only CTA of this key block: dK_j, dV_j (row kglob, columns [wa d/2, (wa+1) d/2))
        // rounded to BF16 as the conversion kernel would round the FP32 sums
        uint4* dko = reinterpret_cast<uint4*>(static_cast<__nv_bfloat16*>(p.dk_dst) + row);
        uint4* dvo = reinterpret_cast<uint4*>(static_cast<__nv_bfloat16*>(p.dv_dst) + row);
#pragma unroll
        for (int c = 0; c < DH; c += 8) {
          const int h = c >> 1;
          dko[c / 8] = make_uint4(pack_bf16x2(lo_f32(dk_run[h]), hi_f32(dk_run[h])),
                                  pack_bf16x2(lo_f32(dk_run[h + 1]), hi_f32(dk_run[h + 1])),
                                  pack_bf16x2(lo_f32(dk_run[h + 2]), hi_f32(dk_run[h + 2])),
                                  pack_bf16x2(lo_f32(dk_run[h + 3]), hi_f32(dk_run[h + 3])));
          dvo[c / 8] = make_uint4(pack_bf16x2(lo_f32(dv_run[h]), hi_f32(dv_run[h])),
                                  pack_bf16x2(lo_f32(dv_run[h + 1]), hi_f32(dv_run[h + 1])),
                                  pack_bf16x2(lo_f32(dv_run[h + 2]), hi_f32(dv_run[h + 2])),
                                  pack_bf16x2(lo_f32(dv_run[h + 3]), hi_f32(dv_run[h + 3])));
        }
      } else {
        // this CTA's share of dK_j, dV_j into the FP32 sums
        float* dka = static_cast<float*>(p.dk_dst) + row;
        float* dva = static_cast<float*>(p.dv_dst) + row;
#pragma unroll
        for (int c = 0; c < DH; c += 4) {
          const int h = c >> 1;
          red_add_v4_f32(dka + c, lo_f32(dk_run[h]), hi_f32(dk_run[h]), lo_f32(dk_run[h + 1]),
                         hi_f32(dk_run[h + 1]));
          red_add_v4_f32(dva + c, lo_f32(dv_run[h]), hi_f32(dv_run[h]), lo_f32(dv_run[h + 1]),
                         hi_f32(dv_run[h + 1]));
        }
      }
    }
  }
  tc_fence_before();
  __syncthreads();
  if (warp == W_MMA) {
    tc_fence_after();
    tmem_dealloc(tmem, 512);
  }
}

template <int D, bool CAUSAL, bool DSX>
cudaError_t launch_bwd_t(const CUtensorMap& tq, const CUtensorMap& tk, const CUtensorMap& tv, const CUtensorMap& tdo,
                         const CUtensorMap& tdoq, const CUtensorMap& tdq, const BwdQsmParams& p, cudaStream_t s) {
  using C = BwdCfg<D>;
  const int grid = p.nb * p.B * p.Hkv * (p.G / p.HS);
  if (p.qbias != nullptr) {
    auto kern = bwd_kernel<D, CAUSAL, DSX, true, false>;
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, C::SMEM);
    if (e != cudaSuccess) return e;
    kern<<<grid, C::THREADS, C::SMEM, s>>>(tq, tk, tv, tdo, tdoq, tdq, p);
  } else if (p.dump != nullptr) {
    if (DSX) return cudaErrorInvalidValue;  // the dump covers the plain instantiation only
    auto kern = bwd_kernel<D, CAUSAL, false, false, true>;
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, C::SMEM);
    if (e != cudaSuccess) return e;
    BwdDumpParams dp;
    static_cast<BwdParams&>(dp) = static_cast<const BwdParams&>(p);
    dp.dump = p.dump;
    kern<<<grid, C::THREADS, C::SMEM, s>>>(tq, tk, tv, tdo, tdoq, tdq, dp);
  } else if (p.flags & (SAGEBWD_FLAG_BF16_PB | SAGEBWD_FLAG_BF16_DS | kFlagFp8Codes)) {
    if (DSX) return cudaErrorInvalidValue;  // these cover the plain instantiation only
    auto kern = (p.flags & kFlagFp8Codes) ? bwd_kernel<D, CAUSAL, false, false, false, kValFp8>
                                          : bwd_kernel<D, CAUSAL, false, false, false, kValBf16>;
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, C::SMEM);
    if (e != cudaSuccess) return e;
    kern<<<grid, C::THREADS, C::SMEM, s>>>(tq, tk, tv, tdo, tdoq, tdq, static_cast<const BwdParams&>(p));
  } else {
    auto kern = bwd_kernel<D, CAUSAL, DSX, false, false>;
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, C::SMEM);
    if (e != cudaSuccess) return e;
    kern<<<grid, C::THREADS, C::SMEM, s>>>(tq, tk, tv, tdo, tdoq, tdq, static_cast<const BwdParams&>(p));
  }
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_bwd(const CUtensorMap& tq, const CUtensorMap& tk, const CUtensorMap& tv, const CUtensorMap& tdo,
                       const CUtensorMap& tdoq, const CUtensorMap& tdq, const BwdQsmParams& p, int d, int causal,
                       int ds_subexp, cudaStream_t s) {
#define SAGEBWD_BWD_CASE(D_, C_)                                                                  \
  if (d == D_ && (causal != 0) == C_)                                                             \
    return ds_subexp ? launch_bwd_t<D_, C_, true>(tq, tk, tv, tdo, tdoq, tdq, p, s)              \
                     : launch_bwd_t<D_, C_, false>(tq, tk, tv, tdo, tdoq, tdq, p, s);
  SAGEBWD_BWD_CASE(64, true)
  SAGEBWD_BWD_CASE(64, false)
  SAGEBWD_BWD_CASE(128, true)
  SAGEBWD_BWD_CASE(128, false)
#undef SAGEBWD_BWD_CASE
  return cudaErrorInvalidValue;
}

// Longest-processing-time list schedule of the backward CTAs (one per key block,
// kv head and group of HS query heads, in launch order) on `sms` SMs, for each
// divisor HS of G; a CTA costs its tiles plus four tiles of setup and drain (TMEM
// allocation, the K^ / V loads, the pipeline fill and the last tile's products and
// epilogue) -- the value whose predicted order and gaps match the backward measured
// with HS = 1, 2, 3 on the 16K-token GQA 6:1 workload (3.162, 3.145, 3.191 ms).
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
      const double cost = (double)hs * (causal ? nb - j : nb) + 4.0;
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
