// C ABI of libsagebwd: argument checks, buffer layouts, TMA tensor maps and
// the launch sequence of each entry point.  All device memory belongs to the
// caller; nothing here allocates, frees or synchronizes (except
// sagebwd_check_status).
#include <cudaTypedefs.h>

#include <atomic>
#include <cmath>
#include <mutex>

#include "sagebwd_internal.h"

using namespace sagebwd;

namespace {

constexpr size_t kAlign = 256;
inline size_t align_up(size_t x) { return (x + kAlign - 1) / kAlign * kAlign; }

bool problem_ok(const sagebwd_problem* p) {
  return p && p->B >= 1 && p->Hq >= 1 && p->Hkv >= 1 && p->N >= 1 && p->d >= 1 && p->Hq % p->Hkv == 0;
}

sagebwd_status check_problem(const sagebwd_problem* p) {
  if (!problem_ok(p)) return SAGEBWD_ERR_INVALID_ARG;
  if (p->d != 64 && p->d != 128) return SAGEBWD_ERR_UNSUPPORTED;
  // int32 element indices inside the kernels, and grid limits
  const double elems = (double)p->B * p->Hq * p->N * p->d;
  if (elems >= 2147483648.0) return SAGEBWD_ERR_UNSUPPORTED;
  if ((double)nblocks(p->N) * p->B * p->Hq >= 2147483647.0) return SAGEBWD_ERR_UNSUPPORTED;
  if (p->smooth_q && p->balance_qk) return SAGEBWD_ERR_UNSUPPORTED;  // not defined together
  if (p->smooth_q && nblocks(p->N) > 65535) return SAGEBWD_ERR_UNSUPPORTED;  // logit-term grid limit
  // the FP8 variant: block scales without sub-scales, no balancing, Q-smoothing, attribution or dump
  if (p->fp8 && (p->qk_subexp || p->ds_subexp || p->balance_qk || p->smooth_q ||
                 (p->flags & (SAGEBWD_FLAGS_BF16 | SAGEBWD_FLAG_DEBUG_DUMP))))
    return SAGEBWD_ERR_UNSUPPORTED;
  if (p->fp8 != 0 && p->fp8 != 1) return SAGEBWD_ERR_INVALID_ARG;
  // the attribution instantiations cover the kernels without dS sub-scales, Q-smoothing and the dump
  if ((p->flags & SAGEBWD_FLAGS_BF16) && (p->ds_subexp || p->smooth_q || (p->flags & SAGEBWD_FLAG_DEBUG_DUMP)))
    return SAGEBWD_ERR_UNSUPPORTED;
  if (p->flags & SAGEBWD_FLAG_DEBUG_DUMP) {
    // the dump covers the kernels without dS sub-scales and Q-smoothing, at most 2^31 bytes
    if (p->ds_subexp || p->smooth_q) return SAGEBWD_ERR_UNSUPPORTED;
    const double nb = nblocks(p->N);
    if ((double)p->B * p->Hq * nb * nb * (98304.0 + 1536.0 * p->d) >= 2147483648.0) return SAGEBWD_ERR_UNSUPPORTED;
  }
  return SAGEBWD_OK;
}

bool aligned16(const void* ptr) { return (reinterpret_cast<uintptr_t>(ptr) & 15u) == 0; }

struct SavedLayout {
  size_t q, k, v, sq, sk, sv, mu, be, qm, qb, q8, k8, v8t, total;
};
SavedLayout saved_layout(const sagebwd_problem* p) {
  const size_t nb = (size_t)nblocks(p->N);
  const size_t qe = (size_t)p->B * p->Hq * p->N * p->d, ke = (size_t)p->B * p->Hkv * p->N * p->d;
  SavedLayout L;
  size_t off = 0;
  L.q = off; off += align_up(qe * 2);
  L.k = off; off += align_up(ke * 2);
  L.v = off; off += align_up(ke * 2);
  L.sq = off; off += align_up((size_t)p->B * p->Hq * nb * 4);
  L.sk = off; off += align_up((size_t)p->B * p->Hkv * nb * 4);
  L.sv = off; off += align_up((size_t)p->B * p->Hkv * nb * 4);
  L.mu = off; off += align_up((size_t)p->B * p->Hkv * p->d * 4);
  L.be = off; off += align_up((size_t)p->B * p->Hkv * p->d * 4);
  L.qm = L.qb = L.q8 = L.k8 = L.v8t = 0;
  if (p->smooth_q) {  // block means of Q, and the logit terms mean_Q . K' per (query head, query block, key)
    L.qm = off; off += align_up((size_t)p->B * p->Hq * nb * p->d * 4);
    L.qb = off; off += align_up((size_t)p->B * p->Hq * nb * nb * kBlk * 4);
  }
  if (p->fp8) {  // the E4M3 values as bytes for the FP8 forward: Q, K row-major, V transposed per head
    L.q8 = off; off += align_up(qe);
    L.k8 = off; off += align_up(ke);
    L.v8t = off; off += align_up((size_t)p->B * p->Hkv * p->d * nb * kBlk);
  }
  L.total = off;
  return L;
}

// Workspace: [status word | pass scratch].
struct WsLayout {
  size_t status, kpart, kmax, kmin, qmax, D, dOq, sdo, dqacc, dkacc, dvacc, cs, dump, total;
};
WsLayout ws_layout(const sagebwd_problem* p, int pass) {
  const size_t nb = (size_t)nblocks(p->N);
  WsLayout L{};
  size_t off = 0;
  L.status = off; off += kAlign;
  if (pass == 0) {
    L.kpart = off; off += align_up((size_t)p->B * p->Hkv * nb * p->d * 8);
    if (p->balance_qk) {
      L.kmax = off; off += align_up((size_t)p->B * p->Hkv * nb * p->d * 4);
      L.kmin = off; off += align_up((size_t)p->B * p->Hkv * nb * p->d * 4);
      L.qmax = off; off += align_up((size_t)p->B * p->Hq * nb * p->d * 4);
    }
  } else {
    const size_t qe = (size_t)p->B * p->Hq * p->N * p->d;
    L.D = off; off += align_up((size_t)p->B * p->Hq * p->N * 4);
    L.dOq = off; off += align_up(qe * 2);
    L.sdo = off; off += align_up((size_t)p->B * p->Hq * nb * 4);
    L.dqacc = off; off += align_up(qe * 4);
    const size_t ke = (size_t)p->B * p->Hkv * p->N * p->d;
    L.dkacc = off; off += align_up(ke * 4);
    L.dvacc = off; off += align_up(ke * 4);
    // Q-smoothing: per backward CTA (at most one per query head and key block) a ring of
    // two tile parities x four softmax slices x 128 keys of dS column sums
    if (p->smooth_q) {
      L.cs = off; off += align_up((size_t)p->B * p->Hq * nb * 2 * 4 * 128 * 4);
    }
  }
  if (p->flags & SAGEBWD_FLAG_DEBUG_DUMP) {
    // one record per (b, query head, query block, key block): forward 128*128*(4 + 2) + 128*d*4
    // bytes, backward 2*128*128*2 + 3*128*d*4 bytes
    const size_t rec = pass == 0 ? 98304 + (size_t)512 * p->d : 65536 + (size_t)1536 * p->d;
    L.dump = off; off += align_up((size_t)p->B * p->Hq * nb * nb * rec);
  }
  L.total = off;
  return L;
}

template <class T>
T* at(void* base, size_t off) {
  return reinterpret_cast<T*>(static_cast<uint8_t*>(base) + off);
}
template <class T>
const T* at(const void* base, size_t off) {
  return reinterpret_cast<const T*>(static_cast<const uint8_t*>(base) + off);
}

PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
  static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* f = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &f, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(f);
  });
  return fn;
}

// 3-D map over a BF16 [BH][N][d] tensor: box = 64 channels x 128 tokens x 1
// head, 128-byte swizzle; tokens past N read as zero.
bool make_map(CUtensorMap* m, const void* base, int BH, int N, int d) {
  auto fn = encode_fn();
  if (!fn) return false;
  cuuint64_t dims[3] = {(cuuint64_t)d, (cuuint64_t)N, (cuuint64_t)BH};
  cuuint64_t strides[2] = {(cuuint64_t)d * 2, (cuuint64_t)N * d * 2};
  cuuint32_t box[3] = {64, 128, 1};
  cuuint32_t es[3] = {1, 1, 1};
  return fn(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(base), dims, strides, box, es,
            CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
            CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// 3-D map over an FP32 [BH][N][d] tensor for reduce-adds: box = 32 channels x
// 128 tokens x 1 head, 128-byte swizzle; rows past N are not written.
bool make_map_f32(CUtensorMap* m, const void* base, int BH, int N, int d) {
  auto fn = encode_fn();
  if (!fn) return false;
  cuuint64_t dims[3] = {(cuuint64_t)d, (cuuint64_t)N, (cuuint64_t)BH};
  cuuint64_t strides[2] = {(cuuint64_t)d * 4, (cuuint64_t)N * d * 4};
  cuuint32_t box[3] = {32, 128, 1};
  cuuint32_t es[3] = {1, 1, 1};
  return fn(m, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 3, const_cast<void*>(base), dims, strides, box, es,
            CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
            CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// 3-D map over a byte tensor [outer][mid][inner] (E4M3 values): box = box_inner bytes x box_mid x 1,
// swizzle of box_inner bytes (128 or 64); rows past mid read as zero.
bool make_map_u8(CUtensorMap* m, const void* base, int outer, int mid, int inner, int box_inner, int box_mid) {
  auto fn = encode_fn();
  if (!fn) return false;
  cuuint64_t dims[3] = {(cuuint64_t)inner, (cuuint64_t)mid, (cuuint64_t)outer};
  cuuint64_t strides[2] = {(cuuint64_t)inner, (cuuint64_t)inner * mid};
  cuuint32_t box[3] = {(cuuint32_t)box_inner, (cuuint32_t)box_mid, 1};
  cuuint32_t es[3] = {1, 1, 1};
  const CUtensorMapSwizzle swz = box_inner == 128 ? CU_TENSOR_MAP_SWIZZLE_128B : CU_TENSOR_MAP_SWIZZLE_64B;
  return fn(m, CU_TENSOR_MAP_DATA_TYPE_UINT8, 3, const_cast<void*>(base), dims, strides, box, es,
            CU_TENSOR_MAP_INTERLEAVE_NONE, swz, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
            CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

float softmax_scale_of(const sagebwd_problem* p) {
  return p->softmax_scale > 0.f ? p->softmax_scale : (float)(1.0 / std::sqrt((double)p->d));
}
float c0_of(const sagebwd_problem* p) {
  // scale * log2(e), formed in FP64 and rounded once
  return (float)((double)softmax_scale_of(p) * 1.4426950408889634073599246810019);
}
uint64_t timeout_of(const sagebwd_problem* p) {
  return p->wait_timeout_ms ? (uint64_t)p->wait_timeout_ms * 1000000ull : kDefaultTimeoutNs;
}

sagebwd_status cuda_status(cudaError_t e) { return e == cudaSuccess ? SAGEBWD_OK : SAGEBWD_ERR_CUDA; }

// What the quantizer selected by its attribution flag stores (ValueMode).
int vmode_of(const sagebwd_problem* p, uint32_t bf16_flag) {
  return p->fp8 ? kValFp8 : ((p->flags & bf16_flag) ? kValBf16 : kValInt8);
}
// Flags the attention kernels get: the caller's, plus the FP8 variant's code rounding.
uint32_t kernel_flags(const sagebwd_problem* p) { return p->flags | (p->fp8 ? kFlagFp8Codes : 0u); }

#define SB_CHECK(expr)                          \
  do {                                          \
    const sagebwd_status st_ = (expr);          \
    if (st_ != SAGEBWD_OK) return st_;          \
  } while (0)

sagebwd_status need(bool ok, sagebwd_status err) { return ok ? SAGEBWD_OK : err; }

sagebwd_status check_ptrs(std::initializer_list<const void*> ptrs) {
  for (const void* p : ptrs) {
    if (p == nullptr) return SAGEBWD_ERR_INVALID_ARG;
    if (!aligned16(p)) return SAGEBWD_ERR_MISALIGNED;
  }
  return SAGEBWD_OK;
}

sagebwd_status fwd_quantize_impl(const sagebwd_problem* p, const void* q, const void* k, const void* v, void* saved,
                                 void* ws, cudaStream_t st) {
  const SavedLayout S = saved_layout(p);
  const WsLayout W = ws_layout(p, 0);
  int* status = at<int>(ws, W.status);
  const int nb = nblocks(p->N);
  const float* mean = p->smooth_k ? at<float>(saved, S.mu) : nullptr;
  const int* bexp = nullptr;
  if (p->balance_qk) {
    StatsParams sp{};
    sp.q = static_cast<const __nv_bfloat16*>(q);
    sp.k = static_cast<const __nv_bfloat16*>(k);
    sp.ksum = at<double>(ws, W.kpart);
    sp.kmax = at<float>(ws, W.kmax);
    sp.kmin = at<float>(ws, W.kmin);
    sp.qmax = at<float>(ws, W.qmax);
    sp.mean = at<float>(saved, S.mu);
    sp.bexp = at<int>(saved, S.be);
    sp.BHq = p->B * p->Hq;
    sp.BHk = p->B * p->Hkv;
    sp.G = p->Hq / p->Hkv;
    sp.N = p->N;
    sp.d = p->d;
    sp.nb = nb;
    sp.smooth = p->smooth_k ? 1 : 0;
    sp.status = status;
    SB_CHECK(cuda_status(launch_qk_stats(sp, st)));
    bexp = at<int>(saved, S.be);
  }
  const int G = p->Hq / p->Hkv;
  QuantParams qp{};
  qp.job[0] = {static_cast<const __nv_bfloat16*>(q), at<__nv_bfloat16>(saved, S.q), at<float>(saved, S.sq), nullptr,
               p->B * p->Hq, bexp, G, -1, p->qk_subexp ? 1 : 0, p->smooth_q ? at<float>(saved, S.qm) : nullptr,
               vmode_of(p, SAGEBWD_FLAG_BF16_Q)};
  qp.job[1] = {static_cast<const __nv_bfloat16*>(k), at<__nv_bfloat16>(saved, S.k), at<float>(saved, S.sk), mean,
               p->B * p->Hkv, bexp, 1, 1, p->qk_subexp ? 1 : 0, nullptr, vmode_of(p, SAGEBWD_FLAG_BF16_K)};
  qp.job[2] = {static_cast<const __nv_bfloat16*>(v), at<__nv_bfloat16>(saved, S.v), at<float>(saved, S.sv), nullptr,
               p->B * p->Hkv, nullptr, 1, 1, 0, nullptr, vmode_of(p, SAGEBWD_FLAG_BF16_V)};
  if (p->fp8) {  // the bytes the FP8 forward reads
    qp.job[0].x8 = at<uint8_t>(saved, S.q8);
    qp.job[1].x8 = at<uint8_t>(saved, S.k8);
    qp.job[2].x8t = at<uint8_t>(saved, S.v8t);
  }
  qp.N = p->N;
  qp.d = p->d;
  qp.nb = nb;
  qp.status = status;
  auto launch_jobs = [&](std::initializer_list<QuantJob> jobs, int clear, bool pdl = false) -> sagebwd_status {
    QuantParams lp = qp;
    lp.njobs = 0;
    lp.block_start[0] = 0;
    for (const QuantJob& j : jobs) {
      lp.job[lp.njobs] = j;
      lp.block_start[lp.njobs + 1] = lp.block_start[lp.njobs] + j.BH * nb;
      ++lp.njobs;
    }
    lp.clear_status = clear;
    return cuda_status(launch_quantize(lp, st, pdl));
  };
  if (p->smooth_k && !p->balance_qk) {
    // K-smoothing: K's block sums, then the channel means (a small kernel), then one launch of the
    // Q, V and K codes.  The last two are programmatic dependents of the launch before them: the Q
    // and V blocks run while the sums and means are computed, and only the K blocks (last in the
    // grid) wait for the means.
    QuantJob jsum{};
    jsum.x = static_cast<const __nv_bfloat16*>(k);
    jsum.BH = p->B * p->Hkv;
    jsum.part = at<double>(ws, W.kpart);
    SB_CHECK(launch_jobs({jsum}, 1));
    SB_CHECK(cuda_status(launch_kmean_final(at<double>(ws, W.kpart), at<float>(saved, S.mu), p->B * p->Hkv, p->N,
                                            p->d, st, true)));
    SB_CHECK(launch_jobs({qp.job[0], qp.job[2], qp.job[1]}, 0, true));
  } else {
    SB_CHECK(launch_jobs({qp.job[0], qp.job[1], qp.job[2]}, p->balance_qk ? 0 : 1));
  }
  if (p->smooth_q) {
    QBiasParams bp{};
    bp.k = static_cast<const __nv_bfloat16*>(k);
    bp.kmean = mean;
    bp.qmean = at<float>(saved, S.qm);
    bp.bias = at<float>(saved, S.qb);
    bp.BHq = p->B * p->Hq;
    bp.G = G;
    bp.N = p->N;
    bp.d = p->d;
    bp.nb = nb;
    bp.causal = p->causal ? 1 : 0;
    bp.c0 = c0_of(p);
    SB_CHECK(cuda_status(launch_qsmooth_bias(bp, st)));
  }
  return SAGEBWD_OK;
}

sagebwd_status fwd_attention_impl(const sagebwd_problem* p, const void* saved, void* o, float* lse, void* ws,
                                  cudaStream_t st) {
  const SavedLayout S = saved_layout(p);
  const WsLayout W = ws_layout(p, 0);
  CUtensorMap tq, tk, tv;
  if (p->fp8) {  // the FP8 tensor cores read the E4M3 bytes (V transposed per head)
    const int nb = nblocks(p->N);
    if (!make_map_u8(&tq, at<uint8_t>(saved, S.q8), p->B * p->Hq, p->N, p->d, p->d, 128) ||
        !make_map_u8(&tk, at<uint8_t>(saved, S.k8), p->B * p->Hkv, p->N, p->d, p->d, 128) ||
        !make_map_u8(&tv, at<uint8_t>(saved, S.v8t), p->B * p->Hkv, p->d, nb * kBlk, 128, p->d))
      return SAGEBWD_ERR_CUDA;
  } else if (!make_map(&tq, at<uint8_t>(saved, S.q), p->B * p->Hq, p->N, p->d) ||
             !make_map(&tk, at<uint8_t>(saved, S.k), p->B * p->Hkv, p->N, p->d) ||
             !make_map(&tv, at<uint8_t>(saved, S.v), p->B * p->Hkv, p->N, p->d)) {
    return SAGEBWD_ERR_CUDA;
  }
  FwdDumpParams fp{};
  fp.B = p->B;
  fp.Hq = p->Hq;
  fp.Hkv = p->Hkv;
  fp.N = p->N;
  fp.nb = nblocks(p->N);
  fp.G = p->Hq / p->Hkv;
  fp.c0 = c0_of(p);
  fp.sq = at<float>(saved, S.sq);
  fp.sk = at<float>(saved, S.sk);
  fp.sv = at<float>(saved, S.sv);
  fp.o = static_cast<__nv_bfloat16*>(o);
  fp.lse = lse;
  fp.qbias = p->smooth_q ? at<float>(saved, S.qb) : nullptr;
  fp.dump = (p->flags & SAGEBWD_FLAG_DEBUG_DUMP) ? at<uint8_t>(ws, W.dump) : nullptr;
  fp.status = at<int>(ws, W.status);
  fp.timeout_ns = timeout_of(p);
  fp.flags = kernel_flags(p);
  return cuda_status(launch_fwd(tq, tk, tv, fp, p->d, p->causal, p->fp8, st));
}

// Query heads per backward CTA for this shape on the current device, memoised
// (the list schedule behind it costs more host time than a launch).
int heads_per_cta(const sagebwd_problem* p) {
  struct Key {
    int B, Hkv, G, nb, causal, sms;
    bool operator==(const Key& o) const {
      return B == o.B && Hkv == o.Hkv && G == o.G && nb == o.nb && causal == o.causal && sms == o.sms;
    }
  };
  static std::mutex mu;
  static Key keys[16];
  static int vals[16];
  static int used = 0, next = 0;
  static std::atomic<int> sm_count[64];  // per device, queried once (zero until then)
  int dev = 0, sms = 148;
  cudaGetDevice(&dev);
  if (dev >= 0 && dev < 64 && sm_count[dev].load(std::memory_order_relaxed) > 0) {
    sms = sm_count[dev].load(std::memory_order_relaxed);
  } else {
    cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    if (dev >= 0 && dev < 64) sm_count[dev].store(sms, std::memory_order_relaxed);
  }
  const Key k{p->B, p->Hkv, p->Hq / p->Hkv, nblocks(p->N), p->causal ? 1 : 0, sms};
  std::lock_guard<std::mutex> lock(mu);
  for (int i = 0; i < used; ++i)
    if (keys[i] == k) return vals[i];
  const int hs = bwd_heads_per_cta(k.B, k.Hkv, k.G, k.nb, k.causal, k.sms);
  keys[next] = k;
  vals[next] = hs;
  next = (next + 1) % 16;
  if (used < 16) ++used;
  return hs;
}

// dK, dV go straight to their BF16 outputs when each key block has a single CTA
// (all G query heads of a kv head in one CTA) and no factor follows (channel
// balancing multiplies dK at the conversion): no FP32 accumulators to zero,
// reduce or convert.
bool direct_dkdv(const sagebwd_problem* p, int hs) { return !p->balance_qk && hs == p->Hq / p->Hkv; }

sagebwd_status bwd_prepare_impl(const sagebwd_problem* p, const void* o, const void* dO, void* ws, cudaStream_t st,
                                int hs) {
  const WsLayout W = ws_layout(p, 1);
  PrepParams pp{};
  pp.o = static_cast<const __nv_bfloat16*>(o);
  pp.dO = static_cast<const __nv_bfloat16*>(dO);
  pp.D = at<float>(ws, W.D);
  pp.dOq = at<__nv_bfloat16>(ws, W.dOq);
  pp.sdo = at<float>(ws, W.sdo);
  pp.dq_acc = at<float>(ws, W.dqacc);
  pp.dk_acc = at<float>(ws, W.dkacc);
  pp.dv_acc = at<float>(ws, W.dvacc);
  pp.BH = p->B * p->Hq;
  pp.BHk = direct_dkdv(p, hs) ? 0 : p->B * p->Hkv;  // the dK / dV accumulators to zero
  pp.N = p->N;
  pp.d = p->d;
  pp.nb = nblocks(p->N);
  pp.status = at<int>(ws, W.status);
  pp.vmode = vmode_of(p, SAGEBWD_FLAG_BF16_DO);
  return cuda_status(launch_bwd_prep(pp, st));
}

sagebwd_status bwd_attention_impl(const sagebwd_problem* p, const void* v, const void* dO, const float* lse,
                                  const void* saved, void* dk, void* dv, void* ws, cudaStream_t st, int hs) {
  const SavedLayout S = saved_layout(p);
  const WsLayout W = ws_layout(p, 1);
  CUtensorMap tq, tk, tv, tdo, tdoq, tdq;
  if (!make_map(&tq, at<uint8_t>(saved, S.q), p->B * p->Hq, p->N, p->d) ||
      !make_map(&tk, at<uint8_t>(saved, S.k), p->B * p->Hkv, p->N, p->d) ||
      !make_map(&tv, v, p->B * p->Hkv, p->N, p->d) || !make_map(&tdo, dO, p->B * p->Hq, p->N, p->d) ||
      !make_map(&tdoq, at<uint8_t>(ws, W.dOq), p->B * p->Hq, p->N, p->d) ||
      !make_map_f32(&tdq, at<uint8_t>(ws, W.dqacc), p->B * p->Hq, p->N, p->d))
    return SAGEBWD_ERR_CUDA;
  BwdQsmParams bp{};
  bp.B = p->B;
  bp.Hq = p->Hq;
  bp.Hkv = p->Hkv;
  bp.N = p->N;
  bp.nb = nblocks(p->N);
  bp.G = p->Hq / p->Hkv;
  bp.c0 = c0_of(p);
  bp.sc = softmax_scale_of(p);
  bp.sq = at<float>(saved, S.sq);
  bp.sk = at<float>(saved, S.sk);
  bp.sdo = at<float>(ws, W.sdo);
  bp.lse = lse;
  bp.D = at<float>(ws, W.D);
  bp.HS = hs;
  bp.dq_acc = at<float>(ws, W.dqacc);
  const bool direct = direct_dkdv(p, hs);
  bp.dk_dst = direct ? dk : static_cast<void*>(at<float>(ws, W.dkacc));
  bp.dv_dst = direct ? dv : static_cast<void*>(at<float>(ws, W.dvacc));
  if (p->smooth_q) {
    bp.qbias = at<float>(saved, S.qb);
    bp.qmean = at<float>(saved, S.qm);
    bp.cs_part = at<float>(ws, W.cs);
  }
  bp.dump = (p->flags & SAGEBWD_FLAG_DEBUG_DUMP) ? at<uint8_t>(ws, W.dump) : nullptr;
  bp.status = at<int>(ws, W.status);
  bp.timeout_ns = timeout_of(p);
  bp.flags = (kernel_flags(p) & ~kBwdDirectDKDV) | (direct ? kBwdDirectDKDV : 0u);
  return cuda_status(launch_bwd(tq, tk, tv, tdo, tdoq, tdq, bp, p->d, p->causal, p->ds_subexp ? 1 : 0, st));
}

sagebwd_status bwd_finish_impl(const sagebwd_problem* p, const void* saved, void* dq, void* dk, void* dv, void* ws,
                               cudaStream_t st, int hs) {
  const WsLayout W = ws_layout(p, 1);
  const size_t nq = (size_t)p->B * p->Hq * p->N * p->d, nk = (size_t)p->B * p->Hkv * p->N * p->d;
  // with channel balancing: dQ = dS (K 2^e) 2^-e and dK = dS^T (Q 2^-e) 2^e
  const int* bexp = p->balance_qk ? at<int>(saved, saved_layout(p).be) : nullptr;
  const ConvertJob jobs[3] = {
      {at<float>(ws, W.dqacc), static_cast<__nv_bfloat16*>(dq), nq, bexp, -1, p->Hq / p->Hkv, p->N, p->d},
      {at<float>(ws, W.dkacc), static_cast<__nv_bfloat16*>(dk), nk, bexp, 1, 1, p->N, p->d},
      {at<float>(ws, W.dvacc), static_cast<__nv_bfloat16*>(dv), nk, nullptr, 1, 1, p->N, p->d}};
  return cuda_status(launch_grad_convert(jobs, direct_dkdv(p, hs) ? 1 : 3, st));  // dK, dV written directly
}

}  // namespace

extern "C" {

size_t sagebwd_saved_bytes(const sagebwd_problem* prob) {
  if (check_problem(prob) != SAGEBWD_OK) return 0;
  return saved_layout(prob).total;
}

size_t sagebwd_workspace_bytes(const sagebwd_problem* prob, int pass) {
  if (check_problem(prob) != SAGEBWD_OK || (pass != 0 && pass != 1)) return 0;
  return ws_layout(prob, pass).total;
}

sagebwd_status sagebwd_quantize(const sagebwd_problem* prob, int which, const void* x, void* x_q, float* scales,
                                float* k_mean, void* ws, void* stream) {
  SB_CHECK(check_problem(prob));
  SB_CHECK(need(which >= SAGEBWD_Q && which <= SAGEBWD_DO, SAGEBWD_ERR_INVALID_ARG));
  // balanced Q and K codes depend on both tensors: only sagebwd_fwd_quantize makes them
  SB_CHECK(need(!(prob->balance_qk && (which == SAGEBWD_Q || which == SAGEBWD_K)), SAGEBWD_ERR_UNSUPPORTED));
  // Q-smoothing's block means have no output here: only sagebwd_fwd_quantize makes those Q codes
  SB_CHECK(need(!(prob->smooth_q && which == SAGEBWD_Q), SAGEBWD_ERR_UNSUPPORTED));
  const bool smooth = which == SAGEBWD_K && prob->smooth_k;
  SB_CHECK(check_ptrs({x, x_q, scales, ws}));
  if (smooth) SB_CHECK(check_ptrs({k_mean}));
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  const WsLayout W = ws_layout(prob, 0);
  int* status = at<int>(ws, W.status);
  const int heads = (which == SAGEBWD_K || which == SAGEBWD_V) ? prob->Hkv : prob->Hq;
  const int BH = prob->B * heads, nb = nblocks(prob->N);
  if (smooth)
    SB_CHECK(cuda_status(launch_kmean(static_cast<const __nv_bfloat16*>(x), at<double>(ws, W.kpart), k_mean, BH,
                                      prob->N, prob->d, status, 1, st)));
  QuantParams qp{};
  qp.job[0] = {static_cast<const __nv_bfloat16*>(x), static_cast<__nv_bfloat16*>(x_q), scales,
               smooth ? k_mean : nullptr, BH, nullptr, 1, 1,
               (prob->qk_subexp && (which == SAGEBWD_Q || which == SAGEBWD_K)) ? 1 : 0};
  qp.job[0].vmode = vmode_of(prob, SAGEBWD_FLAG_BF16_Q << which);
  qp.njobs = 1;
  qp.block_start[0] = 0;
  qp.block_start[1] = BH * nb;
  qp.N = prob->N;
  qp.d = prob->d;
  qp.nb = nb;
  qp.status = status;
  qp.clear_status = smooth ? 0 : 1;
  return cuda_status(launch_quantize(qp, st));
}

sagebwd_status sagebwd_fwd_quantize(const sagebwd_problem* prob, const void* q, const void* k, const void* v,
                                    void* saved, void* ws, void* stream) {
  SB_CHECK(check_problem(prob));
  SB_CHECK(check_ptrs({q, k, v, saved, ws}));
  return fwd_quantize_impl(prob, q, k, v, saved, ws, static_cast<cudaStream_t>(stream));
}

sagebwd_status sagebwd_fwd_attention(const sagebwd_problem* prob, const void* saved, void* o, float* lse, void* ws,
                                     void* stream) {
  SB_CHECK(check_problem(prob));
  SB_CHECK(check_ptrs({saved, o, lse, ws}));
  return fwd_attention_impl(prob, saved, o, lse, ws, static_cast<cudaStream_t>(stream));
}

sagebwd_status sagebwd_fwd(const sagebwd_problem* prob, const void* q, const void* k, const void* v, void* o,
                           float* lse, void* saved, void* ws, void* stream) {
  SB_CHECK(check_problem(prob));
  SB_CHECK(check_ptrs({q, k, v, o, lse, saved, ws}));
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  SB_CHECK(fwd_quantize_impl(prob, q, k, v, saved, ws, st));
  return fwd_attention_impl(prob, saved, o, lse, ws, st);
}

sagebwd_status sagebwd_bwd_prepare(const sagebwd_problem* prob, const void* o, const void* dO, void* ws,
                                   void* stream) {
  SB_CHECK(check_problem(prob));
  SB_CHECK(check_ptrs({o, dO, ws}));
  return bwd_prepare_impl(prob, o, dO, ws, static_cast<cudaStream_t>(stream), heads_per_cta(prob));
}

sagebwd_status sagebwd_bwd_attention(const sagebwd_problem* prob, const void* v, const void* dO, const float* lse,
                                     const void* saved, void* dk, void* dv, void* ws, void* stream) {
  SB_CHECK(check_problem(prob));
  SB_CHECK(check_ptrs({v, dO, lse, saved, dk, dv, ws}));
  return bwd_attention_impl(prob, v, dO, lse, saved, dk, dv, ws, static_cast<cudaStream_t>(stream),
                            heads_per_cta(prob));
}

sagebwd_status sagebwd_bwd_finish(const sagebwd_problem* prob, const void* saved, void* dq, void* dk, void* dv,
                                  void* ws, void* stream) {
  SB_CHECK(check_problem(prob));
  SB_CHECK(check_ptrs({saved, dq, dk, dv, ws}));
  return bwd_finish_impl(prob, saved, dq, dk, dv, ws, static_cast<cudaStream_t>(stream), heads_per_cta(prob));
}

sagebwd_status sagebwd_bwd(const sagebwd_problem* prob, const void* q, const void* k, const void* v, const void* o,
                           const void* dO, const float* lse, const void* saved, void* dq, void* dk, void* dv, void* ws,
                           void* stream) {
  SB_CHECK(check_problem(prob));
  SB_CHECK(check_ptrs({q, k, v, o, dO, lse, saved, dq, dk, dv, ws}));
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  const int hs = heads_per_cta(prob);
  SB_CHECK(bwd_prepare_impl(prob, o, dO, ws, st, hs));
  SB_CHECK(bwd_attention_impl(prob, v, dO, lse, saved, dk, dv, ws, st, hs));
  return bwd_finish_impl(prob, saved, dq, dk, dv, ws, st, hs);
}

sagebwd_status sagebwd_check_status(const void* ws, void* stream, int32_t* detail) {
  if (ws == nullptr) return SAGEBWD_ERR_INVALID_ARG;
  int32_t word = 0;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  if (cudaMemcpyAsync(&word, ws, sizeof(word), cudaMemcpyDeviceToHost, st) != cudaSuccess)
    return SAGEBWD_ERR_CUDA;
  if (cudaStreamSynchronize(st) != cudaSuccess) return SAGEBWD_ERR_CUDA;
  if (detail) *detail = word;
  return (word & 0xFF) == 0 ? SAGEBWD_OK : static_cast<sagebwd_status>(word & 0xFF);
}

const char* sagebwd_status_string(sagebwd_status s) {
  switch (s) {
    case SAGEBWD_OK: return "ok";
    case SAGEBWD_ERR_INVALID_ARG: return "invalid argument";
    case SAGEBWD_ERR_UNSUPPORTED: return "unsupported problem (head dim must be 64 or 128; sizes within int32)";
    case SAGEBWD_ERR_MISALIGNED: return "pointer not 16-byte aligned";
    case SAGEBWD_ERR_CUDA: return "CUDA runtime error";
    case SAGEBWD_ERR_TIMEOUT: return "a kernel wait timed out";
    case SAGEBWD_ERR_SCRATCH_LIMIT: return "problem too large for the fixed scratch of sagebwd_quantize_k_noalloc";
  }
  return "unknown status";
}

size_t sagebwd_debug_dump_offset(const sagebwd_problem* prob, int pass) {
  if (check_problem(prob) != SAGEBWD_OK || (pass != 0 && pass != 1) || !(prob->flags & SAGEBWD_FLAG_DEBUG_DUMP))
    return 0;
  return ws_layout(prob, pass).dump;
}

int32_t sagebwd_version(void) { return 100; }

}  // extern "C"
