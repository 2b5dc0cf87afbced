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
//                    168 registers each; 128 * LOW + 256 * HIGH <= 384 * 168)
// TMEM: tile t owns S_t [256t, 256t+128) and O_t [256t+128, 256t+128+d).  The
// quantized P~ codes (packed BF16, 64 columns) feed O_t = P^_t V^_j as the A operand
// straight from TMEM.  d = 128: they are written over S_t (columns [256t, 256t+64)),
// and the MMA order is S_0(0), S_1(0), then per key tile j: P^_0 V^_j, S_0(j+1),
// P^_1 V^_j, S_1(j+1), S_t(j+1) waiting until P^_t V^_j has consumed the codes that
// share its columns.  d = 64: they have their own columns [256t+192, 256t+256), so
// S_t(j+1) is issued as soon as the softmax has read S_t(j), before P^_t V^_j, and the
// softmax folds P^_t V^_j in after its first pass over S_t(j+1).  Either way the
// softmax of one tile runs while the tensor core serves the other.
//
// Softmax of tile j for one row (FP32, base-2 logits t = S_int * sQ sK scale log2e):
//   tmax  = max_k t_k over the visible keys of the row in the tile
//   code  = rint(2^(t - tmax + log2 127)) in [0, 127]   (P~ quantized per row and tile)
//   The output and row sum are kept relative to a reference m_ref (raised to tmax,
//   with a rescale by a = 2^(m_ref - tmax), only when tmax > m_ref + 8), r = 2^(tmax - m_ref):
//   l     = l a + (r/127) sum_k 2^(t - tmax + log2 127)   (unquantized P~)
//   O    <- O a + (r/127) sV_j [P^ V^]_j   (dequantization per tile, applied one
//           tile late, once the P V product has landed)
// With Q-smoothing the logits gain a term per key of the tile, mean_Q(query block) . K'_k
// (base 2, precomputed), copied next to V_j and added with the same FMA: t = S_int sQ sK c0 + b_k;
// pass 1 writes t back over S_int, and pass 2 then adds log2 127 - tmax.
// Epilogue: O / l as BF16, LSE = (m_ref + log2 l) ln 2.  The quotient does not depend
// on the reference, so this is the online softmax of the definition.
#include "kernel_common.cuh"

namespace sagebwd {
namespace {

constexpr int kFThreads = 384;
constexpr uint32_t kFRegsLaunch = 168;
// registers per thread after setmaxnreg: control warps (producer, MMA) and softmax
// warpgroups.  Measured on d = 128 (long-context workload): 40 / 232 0.846 ms, 56 / 224
// 0.825 ms (before the scale prefetch; 0.820 ms after it), 64 / 216 0.815 ms (ptxas: 128 B of
// spill stores per thread against 240 B at 56 / 224), 96 / 200 0.820 ms; on d = 64, 88 / 208
// (0.478 ms against 0.496 ms at 40 / 232 on the 8K-token GQA workload).
template <int D>
struct FwdRegs {
  static constexpr uint32_t LOW = D == 128 ? 64 : 88, HIGH = D == 128 ? 216 : 208;
  static_assert(128 * LOW + 256 * HIGH <= kFThreads * kFRegsLaunch, "register split exceeds the launch");
};

// F8: the FP8 variant on the FP8 tensor cores (1-byte E4M3 tiles: Q^, K^ [128 tokens][D], V^
// transposed [D][128 keys]; three K / V stages).
template <int D, bool F8 = false>
struct FwdCfg {
  static constexpr int NS = F8 ? 3 : 2;                 // K / V stages
  static constexpr int TILE = 128 * D * (F8 ? 1 : 2);  // one Q^ / K^ / V^ tile (bytes)
  static constexpr int OFF_Q = 0;           // two Q^ tiles
  static constexpr int OFF_K = OFF_Q + 2 * TILE;
  static constexpr int OFF_V = OFF_K + NS * TILE;
  static constexpr int OFF_BIAS = OFF_V + NS * TILE;  // Q-smoothing logit terms [NS][2 tiles][128]
  static constexpr int OFF_BAR = OFF_BIAS + NS * 2 * 512;
  static constexpr int NBAR = 1 + 4 * NS + 2 * 4 + 1;
  static constexpr int SMEM = OFF_BAR + NBAR * 8 + 16 + 1024;
  static_assert(SMEM <= 232448, "shared memory beyond the per-CTA limit");
  __host__ __device__ static constexpr int col_s(int t) { return 256 * t; }
  __host__ __device__ static constexpr int col_o(int t) { return 256 * t + 128; }
  // D = 64 leaves 64 columns per tile free after S_t and O_t: the codes of P~ get their own
  // columns there, so S_t(j+1) need not wait for P^_t V^_j (SEPC); D = 128 writes them over S_t.
  static constexpr bool SEPC = D == 64;
  __host__ __device__ static constexpr int col_c(int t) { return SEPC ? 256 * t + 192 : 256 * t; }
};

enum FwdSite { kSiteQ = 1, kSiteKFull, kSiteKEmpty, kSiteVFull, kSiteVEmpty, kSiteSFull, kSitePFull, kSitePVDone,
               kSiteOEmpty };

// The debug-dump instantiation (DBG) takes FwdDumpParams; one record per tile: the raw FP32
// S_int [128 queries][128 keys], the P~ codes (BF16 [128 queries][128 keys]) and the raw FP32
// [P^ V^] [128 queries][D].
template <bool DBG>
struct FwdParamsOf {
  using type = FwdParams;
};
template <>
struct FwdParamsOf<true> {
  using type = FwdDumpParams;
};
template <int D>
struct FwdDump {
  static constexpr size_t S = 0, PC = 128 * 128 * 4, PV = PC + 128 * 128 * 2, BYTES = PV + 128 * D * 4;
};
// Write 16 consecutive 32-bit words (64 bytes, 16-byte aligned) to global memory.
__device__ __forceinline__ void fdump16(uint8_t* dst, const uint32_t* w) {
  uint4* d4 = reinterpret_cast<uint4*>(dst);
#pragma unroll
  for (int k = 0; k < 4; ++k) d4[k] = make_uint4(w[4 * k], w[4 * k + 1], w[4 * k + 2], w[4 * k + 3]);
}

// VAR (ValueMode of the P~ operand): kValInt8 its integer code rint(127 * 2^(t - tmax)); kValBf16
// (error attribution, SAGEBWD_FLAG_BF16_PF) the BF16 rounding of 127 * 2^(t - tmax); kValFp8 (the
// FP8 variant) the E4M3 rounding of 448 * 2^(t - tmax), dequantized by 2^(tmax - m) / 448.
// F8 (with VAR == kValFp8): the same values as E4M3 bytes on the FP8 tensor cores (tcgen05.mma
// kind::f8f6f4, K = 32 per instruction): S from the byte tiles of Q^ and K^, O = P^ V^ with the P~
// bytes packed four per TMEM column and V^ read from its transposed tile (all operands K-major).
template <int D, bool CAUSAL, bool QSM, bool DBG, int VAR = kValInt8, bool F8 = false>
__global__ void __launch_bounds__(kFThreads, 1)
    fwd_kernel(const __grid_constant__ CUtensorMap tmQ, const __grid_constant__ CUtensorMap tmK,
               const __grid_constant__ CUtensorMap tmV, const typename FwdParamsOf<DBG>::type p) {
  static_assert(!F8 || (VAR == kValFp8 && !QSM && !DBG), "the FP8 tensor-core path is the FP8 variant only");
  using C = FwdCfg<D, F8>;
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
    setmaxnreg_dec<FwdRegs<D>::LOW>();
    if (warp == 8 && lane == 0) {
      // ---------------------------------------------------------- TMA producer
      int k_issued[NS], v_issued[NS];
      for (int s = 0; s < NS; ++s) k_issued[s] = v_issued[s] = 0;
      const int nq = (nkb[0] > 0) + (nkb[1] > 0);
      mbar_arrive_expect_tx(bar_q, nq * C::TILE);
      for (int t = 0; t < 2; ++t)
        if (nkb[t] > 0) {
          if constexpr (F8)
            tma_load_3d(smem + C::OFF_Q + t * C::TILE, &tmQ, bar_q, 0, (2 * pr + t) * kBlk, bhq);
          else
            for (int c = 0; c < D / 64; ++c)
              tma_load_3d(smem + C::OFF_Q + t * C::TILE + c * 16384, &tmQ, bar_q, c * 64, (2 * pr + t) * kBlk, bhq);
        }
      for (int j = 0; j < nkb_max; ++j) {
        const int s = j % NS, n = j / NS;
        if (j >= NS && !wait1(wc, bar_k_empty + s, (n - 1) & 1, kSiteKEmpty)) break;
        if (!((p.flags & SAGEBWD_FLAG_DROP_ONE_LOAD) && j == 1)) {  // fault injection skips one load
          mbar_arrive_expect_tx(bar_k_full + s, C::TILE);
          if constexpr (F8)
            tma_load_3d(smem + C::OFF_K + s * C::TILE, &tmK, bar_k_full + s, 0, j * kBlk, bhk);
          else
            for (int c = 0; c < D / 64; ++c)
              tma_load_3d(smem + C::OFF_K + s * C::TILE + c * 16384, &tmK, bar_k_full + s, c * 64, j * kBlk, bhk);
          k_issued[s] = n + 1;
        }
        if (j >= NS && !wait1(wc, bar_v_empty + s, (n - 1) & 1, kSiteVEmpty)) break;
        // Q-smoothing: the logit terms of tile j for each query tile that reads it ride on the
        // V stage, which is released only after both tiles' codes of key tile j are written
        const int nbias = QSM ? (j < nkb[0]) + (j < nkb[1]) : 0;
        mbar_arrive_expect_tx(bar_v_full + s, C::TILE + nbias * 512);
        if constexpr (F8)  // the transposed V^ tile [D][128 keys]
          tma_load_3d(smem + C::OFF_V + s * C::TILE, &tmV, bar_v_full + s, j * kBlk, 0, bhk);
        else
          for (int c = 0; c < D / 64; ++c)
            tma_load_3d(smem + C::OFF_V + s * C::TILE + c * 16384, &tmV, bar_v_full + s, c * 64, j * kBlk, bhk);
        if (QSM) {
          for (int t = 0; t < 2; ++t)
            if (j < nkb[t])
              bulk_load_1d(smem + C::OFF_BIAS + (s * 2 + t) * 512,
                           p.qbias + ((size_t)bhq * p.nb + 2 * pr + t) * ((size_t)p.nb * kBlk) + (size_t)j * kBlk, 512,
                           bar_v_full + s);
        }
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
      const uint32_t idS = F8 ? idesc_e4m3_f32(128, 128) : idesc_bf16_f32(128, 128, false, false);
      const uint32_t idO = F8 ? idesc_e4m3_f32(128, D) : idesc_bf16_f32(128, D, false, true);
      // FP8 tiles: rows of D bytes (128-byte swizzle for D = 128, 64-byte for D = 64; 8-row stride
      // 8 D bytes); the transposed V^ tile has 128-byte rows
      constexpr uint32_t kF8Swz = D == 128 ? kSwizzle128B : kSwizzle64B;
      // S_t = Q^_t K^_j^T into TMEM columns [col_s(t), col_s(t) + 128)
      auto issue_s = [&](int t, uint32_t kdesc) {
        const uint32_t qaddr = smem_u32(smem + C::OFF_Q + t * C::TILE);
        if constexpr (F8) {
#pragma unroll
          for (int kk = 0; kk < D / 32; ++kk)  // 32 bytes of the K dimension per MMA
            umma_f8_ss(tmem + C::col_s(t), sdesc_kmajor(qaddr + kk * 32, 8 * D, kF8Swz),
                       sdesc_kmajor(kdesc + kk * 32, 8 * D, kF8Swz), idS, kk > 0);
        } else {
          const uint32_t qdesc = sdesc_sw128_lo(qaddr, 16);
          if constexpr (D == 128)
            umma_chain8_kk(tmem + C::col_s(t), sdesc_from_lo(qdesc), sdesc_from_lo(kdesc), idS);
          else
            umma_chain4_kk(tmem + C::col_s(t), sdesc_from_lo(qdesc), sdesc_from_lo(kdesc), idS);
        }
        umma_commit(bar_s_full + t);
      };
      // FP8: issue_s takes the K^ tile's shared address, the BF16 path its descriptor low word
      auto k_arg = [&](int st) -> uint32_t {
        const uint32_t a = smem_u32(smem + C::OFF_K + st * C::TILE);
        return F8 ? a : sdesc_sw128_lo(a, 16);
      };
      bool ok = wait1(wc, bar_q, 0, kSiteQ) && wait1(wc, bar_k_full, 0, kSiteKFull);
      if (ok) {
        tc_fence_after();
        const uint32_t kdesc = k_arg(0);
        for (int t = 0; t < 2; ++t)
          if (nkb[t] > 0) issue_s(t, kdesc);
        umma_commit(bar_k_empty);
      }
      // Per key tile j: P^_0 V^_j, S_0(j+1), P^_1 V^_j, S_1(j+1), so that the tensor
      // core works on one tile while the softmax warpgroup of the other runs.  With separate
      // code columns (D = 64) S_t(j+1) goes first, as soon as the softmax has read S_t(j).
      for (int j = 0; ok && j < nkb_max; ++j) {
        const int s = j % NS, s1 = (j + 1) % NS;
        if (!wait1(wc, bar_v_full + s, (j / NS) & 1, kSiteVFull)) break;
        const uint32_t vaddr = smem_u32(smem + C::OFF_V + s * C::TILE);
        const uint32_t vdesc = sdesc_sw128_lo(vaddr, 16384);
        const uint32_t kdesc = k_arg(s1);
        bool k_ready = false;
#pragma unroll
        for (int t = 0; t < 2; ++t) {
          if (j < nkb[t]) {
            if (!wait1(wc, bar_p_full + t, j & 1, kSitePFull)) {
              ok = false;
              break;
            }
            if (C::SEPC && j + 1 < nkb[t]) {
              if (!k_ready && !wait1(wc, bar_k_full + s1, ((j + 1) / NS) & 1, kSiteKFull)) {
                ok = false;
                break;
              }
              k_ready = true;
              tc_fence_after();
              issue_s(t, kdesc);  // S_t(j) has been read: its columns are free
            }
            if (j >= 1 && !wait1(wc, bar_o_empty + t, (j - 1) & 1, kSiteOEmpty)) {
              ok = false;
              break;
            }
            tc_fence_after();
            if constexpr (F8) {
              // O_t = P^_t V^_j: A = the E4M3 bytes in TMEM (128 keys = 32 columns, 8 per K step of
              // 32), B = the transposed V^_j [d][key], K-major (32 bytes per K step)
#pragma unroll
              for (int kk = 0; kk < 4; ++kk)
                umma_f8_ts(tmem + C::col_o(t), tmem + C::col_c(t) + kk * 8,
                           sdesc_kmajor(vaddr + kk * 32, 1024, kSwizzle128B), idO, kk > 0);
            } else {
              // O_t = P^_t V^_j: A = the codes in TMEM (128 keys = 64 packed columns, 8 per
              // K step), B = V^_j [key][d] read MN-major
#pragma unroll
              for (int kk = 0; kk < 8; ++kk)
                umma_ts(tmem + C::col_o(t), tmem + C::col_c(t) + kk * 8, sdesc_from_lo(vdesc + kk * 128), idO,
                        kk > 0);
            }
            umma_commit(bar_pv_done + t);
          }
          if (!C::SEPC && j + 1 < nkb[t]) {
            if (!k_ready && !wait1(wc, bar_k_full + s1, ((j + 1) / NS) & 1, kSiteKFull)) {
              ok = false;
              break;
            }
            k_ready = true;
            // S_t(j+1) overwrites the code columns: P^_t V^_j must have read them
            if (!wait1(wc, bar_pv_done + t, j & 1, kSitePVDone)) {
              ok = false;
              break;
            }
            tc_fence_after();
            issue_s(t, kdesc);
          }
        }
        if (!ok) break;
        umma_commit(bar_v_empty + s);
        if (k_ready) umma_commit(bar_k_empty + s1);
      }
      // Every MMA issued above must complete before TMEM is released.
      umma_commit(bar_final);
      drain(bar_final, 0, p.timeout_ns);
    }
  } else {
    setmaxnreg_inc<FwdRegs<D>::HIGH>();
    // ------------------------------------------------------------ softmax / correction
    const int t = warp >> 2;  // query tile of this warpgroup
    const int r = tid & 127;  // query row within the tile == TMEM lane
    const int qb = 2 * pr + t;
    const int i = qb * kBlk + r;
    const int nk = nkb[t];
    const uint32_t lane_base = (uint32_t)((warp & 3) * 32) << 16;
    const uint32_t s_addr = tmem + lane_base + C::col_s(t);
    const uint32_t o_addr = tmem + lane_base + C::col_o(t);
    const uint32_t c_addr = tmem + lane_base + C::col_c(t);  // the codes of P~
    const float sQv = nk > 0 ? p.sq[(size_t)bhq * p.nb + qb] : 0.f;
    // The running output and sum are kept relative to a reference maximum m_ref that
    // only moves when a tile's maximum exceeds it by more than 2^8; the result is the
    // same ratio, and the rescale of the output is skipped on most tiles.
    float m_ref = -INFINITY, l = 0.f;
    uint64_t o_acc[D / 2];
#pragma unroll
    for (int c = 0; c < D / 2; ++c) o_acc[c] = 0ull;
    float pend_a = 1.f, pend_w = 0.f;
    bool ok = true;

    // Fold tile jj's P V product into the running output: o = o * a + w * [P^ V^]_jj.
    // debug dump record of key tile jj of this warpgroup's query tile (DBG instantiation only)
    auto dump_rec = [&](int jj) -> uint8_t* {
      if constexpr (DBG)
        return p.dump + (((size_t)bhq * p.nb + qb) * p.nb + jj) * FwdDump<D>::BYTES;
      else
        return nullptr;
    };
    auto fold = [&](int jj, float a, float w) -> bool {
      if (!waitw(wc, bar_pv_done + t, jj & 1, kSitePVDone)) return false;
      tc_fence_after();
      if (__any_sync(0xffffffffu, a != 1.f)) {
        const uint64_t a2 = pack_f32x2(a, a);
#pragma unroll
        for (int c = 0; c < D / 2; ++c) fmul2_acc(o_acc[c], a2);
      }
      const uint64_t w2 = pack_f32x2(w, w);
#pragma unroll
      for (int c0 = 0; c0 < D; c0 += 32) {
        uint32_t v[32];
        tmem_ld32(o_addr + c0, v);
        tmem_ld_wait();
        if constexpr (DBG) {
          fdump16(dump_rec(jj) + FwdDump<D>::PV + ((size_t)r * D + c0) * 4, v);
          fdump16(dump_rec(jj) + FwdDump<D>::PV + ((size_t)r * D + c0 + 16) * 4, v + 16);
        }
#pragma unroll
        for (int e = 0; e < 32; e += 2)
          ffma2_acc(o_acc[(c0 + e) >> 1], w2, v[e], v[e + 1]);
      }
      tc_fence_before();
      mbar_arrive(bar_o_empty + t);
      return true;
    };

    // the K and V block scales, loaded one key tile ahead (their latency hides behind a tile)
    float pf_sk = nk > 0 ? p.sk[(size_t)bhk * p.nb] : 0.f, pf_sv = nk > 0 ? p.sv[(size_t)bhk * p.nb] : 0.f;
    for (int j = 0; j < nk; ++j) {
      const float sKv = pf_sk, sVv = pf_sv;
      if (j + 1 < nk) {
        pf_sk = p.sk[(size_t)bhk * p.nb + j + 1];
        pf_sv = p.sv[(size_t)bhk * p.nb + j + 1];
      }
      // the previous tile's product lands while S_t(j) is computed (with separate code columns it
      // is folded after pass 1, since S_t(j) was issued before P^_t V^_(j-1))
      if (!C::SEPC && j >= 1 && !fold(j - 1, pend_a, pend_w)) {
        ok = false;
        break;
      }
      if (!waitw(wc, bar_s_full + t, j & 1, kSiteSFull)) {
        ok = false;
        break;
      }
      tc_fence_after();
      const float qks = __fmul_rn(__fmul_rn(sQv, sKv), p.c0);
      const int k0 = j * kBlk;
      const bool need_mask = (CAUSAL && j == qb) || (k0 + kBlk > p.N);
      const int kvis = need_mask ? (min(p.N, CAUSAL ? i + 1 : p.N) - k0) : kBlk;  // visible keys of this row
      const float2 qks2 = make_float2(qks, qks);
      // Q-smoothing: this tile's logit terms mean_Q . K'_k (base 2), one per key, in shared memory
      const float* bsm = reinterpret_cast<const float*>(smem + C::OFF_BIAS + ((j % NS) * 2 + t) * 512);
      float tmax;
      if constexpr (QSM) {
        // pass 1: row maximum of t = S_int sQ sK c0 + bias over the visible keys
        if (!waitw(wc, bar_v_full + (j % NS), (j / NS) & 1, kSiteVFull)) {
          ok = false;
          break;
        }
        float xmax = -INFINITY;
#pragma unroll
        for (int c0 = 0; c0 < 128; c0 += 32) {
          uint32_t v[32];
          tmem_ld32(s_addr + c0, v);
          tmem_ld_wait();
#pragma unroll
          for (int e = 0; e < 32; e += 4) {
            const float4 b4 = *reinterpret_cast<const float4*>(bsm + c0 + e);
            const float2 x01 = ffma2(make_float2(__uint_as_float(v[e]), __uint_as_float(v[e + 1])), qks2,
                                     make_float2(b4.x, b4.y));
            const float2 x23 = ffma2(make_float2(__uint_as_float(v[e + 2]), __uint_as_float(v[e + 3])), qks2,
                                     make_float2(b4.z, b4.w));
            if (need_mask) {
              xmax = fmax3(xmax, c0 + e < kvis ? x01.x : -INFINITY, c0 + e + 1 < kvis ? x01.y : -INFINITY);
              xmax = fmax3(xmax, c0 + e + 2 < kvis ? x23.x : -INFINITY, c0 + e + 3 < kvis ? x23.y : -INFINITY);
            } else {
              xmax = fmax3(xmax, x01.x, x01.y);
              xmax = fmax3(xmax, x23.x, x23.y);
            }
            v[e] = __float_as_uint(x01.x);
            v[e + 1] = __float_as_uint(x01.y);
            v[e + 2] = __float_as_uint(x23.x);
            v[e + 3] = __float_as_uint(x23.y);
          }
          // the logits replace S_int in TMEM, so that pass 2 only adds the row's offset
          tmem_st16(s_addr + c0, *reinterpret_cast<const uint32_t(*)[16]>(v));
          tmem_st16(s_addr + c0 + 16, *reinterpret_cast<const uint32_t(*)[16]>(v + 16));
        }
        tmem_st_wait();
        tmax = xmax;
      } else {
        // pass 1: row maximum of S_int over the visible keys
        float smax = -INFINITY;
        if (need_mask) {
#pragma unroll
          for (int c0 = 0; c0 < 128; c0 += 32) {
            uint32_t v[32];
            tmem_ld32(s_addr + c0, v);
            tmem_ld_wait();
#pragma unroll
            for (int e = 0; e < 32; e += 2)
              smax = fmax3(smax, c0 + e < kvis ? __uint_as_float(v[e]) : -INFINITY,
                           c0 + e + 1 < kvis ? __uint_as_float(v[e + 1]) : -INFINITY);
            if constexpr (DBG) {
              fdump16(dump_rec(j) + FwdDump<D>::S + ((size_t)r * 128 + c0) * 4, v);
              fdump16(dump_rec(j) + FwdDump<D>::S + ((size_t)r * 128 + c0 + 16) * 4, v + 16);
            }
          }
        } else {
#pragma unroll
          for (int c0 = 0; c0 < 128; c0 += 32) {
            uint32_t v[32];
            tmem_ld32(s_addr + c0, v);
            tmem_ld_wait();
#pragma unroll
            for (int e = 0; e < 32; e += 2) smax = fmax3(smax, __uint_as_float(v[e]), __uint_as_float(v[e + 1]));
            if constexpr (DBG) {
              fdump16(dump_rec(j) + FwdDump<D>::S + ((size_t)r * 128 + c0) * 4, v);
              fdump16(dump_rec(j) + FwdDump<D>::S + ((size_t)r * 128 + c0 + 16) * 4, v + 16);
            }
          }
        }
        tmax = __fmul_rn(smax, qks);
      }
      float a = 1.f;
      if (tmax > m_ref + 8.f) {
        a = ex2_approx(m_ref - tmax);
        m_ref = tmax;
      }
      const float rj = ex2_approx(tmax - m_ref);
      // separate code columns: fold tile j-1's product now (it ran behind S_t(j)), before pass 2
      // writes this tile's codes over the columns it read
      if (C::SEPC && j >= 1 && !fold(j - 1, pend_a, pend_w)) {
        ok = false;
        break;
      }
      constexpr float kQLog2 = VAR == kValFp8 ? kLog2_448 : kLog2_127, kQInv = VAR == kValFp8 ? 1.f / kFp8Max : 1.f / 127.f;
      const float bias = kQLog2 - tmax;
      // pass 2: codes of P~ written over the S columns already read (chunk c of 32 keys
      // -> 16 packed columns starting at 16c), and the unquantized row sum
      const float2 bias2 = make_float2(bias, bias);
      const float2 mg = make_float2(12582912.0f, 12582912.0f), nmg = make_float2(-12582912.0f, -12582912.0f);
      float2 usum = make_float2(0.f, 0.f);
#pragma unroll
      for (int c0 = 0; c0 < 128; c0 += 32) {
        uint32_t v[32];
        tmem_ld32(s_addr + c0, v);
        tmem_ld_wait();
        uint32_t pk[16];
        uint32_t pb[8];  // F8: the chunk's 32 E4M3 bytes, four per word
#pragma unroll
        for (int e = 0; e < 32; e += 2) {
          const float2 x = QSM ? fadd2(make_float2(__uint_as_float(v[e]), __uint_as_float(v[e + 1])), bias2)
                               : ffma2(make_float2(__uint_as_float(v[e]), __uint_as_float(v[e + 1])), qks2, bias2);
          float2 u = make_float2(ex2_approx(x.x), ex2_approx(x.y));
          if (need_mask) {
            if (c0 + e >= kvis) u.x = 0.f;
            if (c0 + e + 1 >= kvis) u.y = 0.f;
          }
          usum = fadd2(usum, u);
          if constexpr (F8) {
            const uint32_t b2 = e4m3x2_bytes(u.x, u.y);
            if (e & 2)
              pb[e >> 2] |= b2 << 16;
            else
              pb[e >> 2] = b2;
          } else if constexpr (VAR == kValBf16) {
            pk[e >> 1] = pack_bf16x2(u.x, u.y);
          } else if constexpr (VAR == kValFp8) {
            pk[e >> 1] = e4m3x2_bf16x2(u.x, u.y);
          } else {
            // round to the nearest integer (ties to even) with the 1.5 * 2^23 constant
            const float2 cd = fadd2(fadd2(u, mg), nmg);
            pk[e >> 1] = pack_int_bf16x2(cd.x, cd.y);
          }
        }
        if constexpr (DBG) fdump16(dump_rec(j) + FwdDump<D>::PC + ((size_t)r * 128 + c0) * 2, pk);
        if constexpr (F8)
          tmem_st8(c_addr + (c0 >> 2), pb);
        else
          tmem_st16(c_addr + (c0 >> 1), pk);
      }
      tmem_st_wait();
      tc_fence_before();
      mbar_arrive(bar_p_full + t);
      const float w_l = rj * kQInv;
      l = fmaf(w_l, usum.x + usum.y, l * a);
      pend_a = a;
      pend_w = w_l * sVv;
    }
    if (ok && nk > 0) ok = fold(nk - 1, pend_a, pend_w);
    if (ok && nk > 0 && !*abort_flag && i < p.N) {
      const float inv_l = 1.f / l;
      uint4* dst = reinterpret_cast<uint4*>(p.o + ((size_t)bhq * p.N + i) * D);
#pragma unroll
      for (int c = 0; c < D / 2; c += 4) {
        uint4 u;
        u.x = pack_bf16x2(lo_f32(o_acc[c]) * inv_l, hi_f32(o_acc[c]) * inv_l);
        u.y = pack_bf16x2(lo_f32(o_acc[c + 1]) * inv_l, hi_f32(o_acc[c + 1]) * inv_l);
        u.z = pack_bf16x2(lo_f32(o_acc[c + 2]) * inv_l, hi_f32(o_acc[c + 2]) * inv_l);
        u.w = pack_bf16x2(lo_f32(o_acc[c + 3]) * inv_l, hi_f32(o_acc[c + 3]) * inv_l);
        dst[c / 4] = u;
      }
      p.lse[(size_t)bhq * p.N + i] = (m_ref + log2f(l)) * kLn2;
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
cudaError_t launch_fwd_t(const CUtensorMap& tq, const CUtensorMap& tk, const CUtensorMap& tv, const FwdDumpParams& p,
                         int f8, cudaStream_t s) {
  using C = FwdCfg<D>;
  const int grid = (p.nb + 1) / 2 * p.B * p.Hq;
  if (f8) {
    if (p.qbias != nullptr || p.dump != nullptr || !(p.flags & kFlagFp8Codes)) return cudaErrorInvalidValue;
    auto kern = fwd_kernel<D, CAUSAL, false, false, kValFp8, true>;
    constexpr int smem = FwdCfg<D, true>::SMEM;
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
    if (e != cudaSuccess) return e;
    kern<<<grid, kFThreads, smem, s>>>(tq, tk, tv, static_cast<const FwdParams&>(p));
  } else if (p.dump != nullptr) {
    if (p.qbias != nullptr) return cudaErrorInvalidValue;  // the dump covers the plain instantiation only
    auto kern = fwd_kernel<D, CAUSAL, false, true>;
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, C::SMEM);
    if (e != cudaSuccess) return e;
    kern<<<grid, kFThreads, C::SMEM, s>>>(tq, tk, tv, p);
  } else if (p.flags & (SAGEBWD_FLAG_BF16_PF | kFlagFp8Codes)) {
    if (p.qbias != nullptr) return cudaErrorInvalidValue;  // these cover the plain instantiation only
    auto kern = (p.flags & kFlagFp8Codes) ? fwd_kernel<D, CAUSAL, false, false, kValFp8>
                                          : fwd_kernel<D, CAUSAL, false, false, kValBf16>;
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, C::SMEM);
    if (e != cudaSuccess) return e;
    kern<<<grid, kFThreads, C::SMEM, s>>>(tq, tk, tv, static_cast<const FwdParams&>(p));
  } else {
    auto kern = p.qbias != nullptr ? fwd_kernel<D, CAUSAL, true, false> : fwd_kernel<D, CAUSAL, false, false>;
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, C::SMEM);
    if (e != cudaSuccess) return e;
    kern<<<grid, kFThreads, C::SMEM, s>>>(tq, tk, tv, static_cast<const FwdParams&>(p));
  }
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_fwd(const CUtensorMap& tq, const CUtensorMap& tk, const CUtensorMap& tv, const FwdDumpParams& p,
                       int d, int causal, int f8, cudaStream_t s) {
  if (d == 64)
    return causal ? launch_fwd_t<64, true>(tq, tk, tv, p, f8, s) : launch_fwd_t<64, false>(tq, tk, tv, p, f8, s);
  return causal ? launch_fwd_t<128, true>(tq, tk, tv, p, f8, s) : launch_fwd_t<128, false>(tq, tk, tv, p, f8, s);
}

}  // namespace sagebwd
