// K quantization with K-smoothing that needs no caller workspace.
//
// sagebwd_quantize(SAGEBWD_K, ...) keeps the FP64 per-block channel sums of K
// (the scratch of its mean pass) in the caller's workspace.  Some callers have
// no way to provide one: a framework plugin or operator hook that is handed
// only its input and output tensors, code that runs where cudaMalloc is not
// permitted or would synchronize the device at the wrong moment, or a process
// whose memory is all owned by a pool it cannot draw from at that point.  This
// entry point serves them with a fixed scratch array compiled into the
// library: every GPU that loads the library reserves it (8 MiB) until the
// process exits.
#include <cudaTypedefs.h>

#include <mutex>

#include "sagebwd_internal.h"

namespace {

// Room for 2^20 FP64 partial sums: B * Hkv * ceil(N / 128) * d <= 1048576.
constexpr size_t kScratchDoubles = size_t(1) << 20;
static __device__ __align__(256) double g_kmean_scratch[kScratchDoubles];

constexpr int kMaxDevices = 64;
std::mutex g_lock;
double* g_scratch_ptr[kMaxDevices] = {};
unsigned long long g_scratch_ctx[kMaxDevices] = {};  // id of the context the address belongs to

// Unique id of the calling thread's current CUDA context (the driver never reuses one within a
// process), or 0 when it cannot be read.
unsigned long long current_context_id() {
  using GetCurrent = CUresult (*)(CUcontext*);
  using GetId = CUresult (*)(CUcontext, unsigned long long*);
  static GetCurrent get_current = nullptr;
  static GetId get_id = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* f = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuCtxGetCurrent", &f, 12000, cudaEnableDefault, &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      get_current = reinterpret_cast<GetCurrent>(f);
    if (cudaGetDriverEntryPointByVersion("cuCtxGetId", &f, 12000, cudaEnableDefault, &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      get_id = reinterpret_cast<GetId>(f);
  });
  CUcontext ctx = nullptr;
  unsigned long long id = 0;
  if (get_current == nullptr || get_id == nullptr || get_current(&ctx) != CUDA_SUCCESS || ctx == nullptr ||
      get_id(ctx, &id) != CUDA_SUCCESS)
    return 0;
  return id;
}

// Device address of the scratch array in the current device's context, looked up once per device and
// context (the host-side symbol is only a stand-in and must not reach a kernel).  A context that was
// destroyed (cudaDeviceReset) and created again has a new id, so the address is looked up again; when
// the id cannot be read the address is looked up on every call.
double* scratch_on_current_device() {
  int dev = -1;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return nullptr;
  std::lock_guard<std::mutex> guard(g_lock);
  const unsigned long long ctx = current_context_id();
  if (g_scratch_ptr[dev] != nullptr && ctx != 0 && ctx == g_scratch_ctx[dev]) return g_scratch_ptr[dev];
  void* ptr = nullptr;
  if (cudaGetSymbolAddress(&ptr, g_kmean_scratch) != cudaSuccess) return nullptr;
  g_scratch_ptr[dev] = static_cast<double*>(ptr);
  g_scratch_ctx[dev] = current_context_id();  // the lookup made the runtime's context current
  return g_scratch_ptr[dev];
}

}  // namespace

extern "C" sagebwd_status sagebwd_quantize_k_noalloc(const sagebwd_problem* prob, const void* k, void* k_q,
                                                     float* scales, float* k_mean, void* stream) {
  using namespace sagebwd;
  if (prob == nullptr || prob->B < 1 || prob->Hq < 1 || prob->Hkv < 1 || prob->N < 1 || prob->Hq % prob->Hkv != 0)
    return SAGEBWD_ERR_INVALID_ARG;
  if (prob->d != 64 && prob->d != 128) return SAGEBWD_ERR_UNSUPPORTED;
  if (prob->balance_qk) return SAGEBWD_ERR_UNSUPPORTED;  // balanced K codes depend on Q
  if (prob->fp8 && prob->qk_subexp) return SAGEBWD_ERR_UNSUPPORTED;  // E4M3 values carry no sub-scales
  if ((double)prob->B * prob->Hkv * prob->N * prob->d >= 2147483648.0) return SAGEBWD_ERR_UNSUPPORTED;
  const bool smooth = prob->smooth_k != 0;
  for (const void* ptr : {k, (const void*)k_q, (const void*)scales}) {
    if (ptr == nullptr) return SAGEBWD_ERR_INVALID_ARG;
    if (reinterpret_cast<uintptr_t>(ptr) & 15u) return SAGEBWD_ERR_MISALIGNED;
  }
  if (smooth) {
    if (k_mean == nullptr) return SAGEBWD_ERR_INVALID_ARG;
    if (reinterpret_cast<uintptr_t>(k_mean) & 15u) return SAGEBWD_ERR_MISALIGNED;
  }
  const int BH = prob->B * prob->Hkv, nb = nblocks(prob->N);
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  if (smooth) {
    if ((size_t)BH * nb * prob->d > kScratchDoubles) return SAGEBWD_ERR_SCRATCH_LIMIT;
    double* scratch = scratch_on_current_device();
    if (scratch == nullptr) return SAGEBWD_ERR_CUDA;
    // every partial sum is written before it is read: the scratch needs no clearing
    if (launch_kmean(static_cast<const __nv_bfloat16*>(k), scratch, k_mean, BH, prob->N, prob->d, nullptr, 0, st) !=
        cudaSuccess)
      return SAGEBWD_ERR_CUDA;
  }
  QuantParams qp{};
  qp.job[0] = {static_cast<const __nv_bfloat16*>(k), static_cast<__nv_bfloat16*>(k_q), scales,
               smooth ? k_mean : nullptr, BH, nullptr, 1, 1, prob->qk_subexp ? 1 : 0};
  qp.job[0].vmode = prob->fp8 ? kValFp8 : ((prob->flags & SAGEBWD_FLAG_BF16_K) ? kValBf16 : kValInt8);
  qp.njobs = 1;
  qp.block_start[0] = 0;
  qp.block_start[1] = BH * nb;
  qp.N = prob->N;
  qp.d = prob->d;
  qp.nb = nb;
  qp.status = nullptr;
  qp.clear_status = 0;
  return launch_quantize(qp, st) == cudaSuccess ? SAGEBWD_OK : SAGEBWD_ERR_CUDA;
}
