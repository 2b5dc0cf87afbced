// Thin inline-PTX wrappers for the sm_103a features the SageBwd kernels use:
// mbarriers (with bounded waits), TMA tile loads, tcgen05 MMA / TMEM access,
// and the shared-memory / instruction descriptors of the 5th-generation
// tensor cores.  Everything here is a one-instruction wrapper or a bit-field
// packer; no arithmetic of the attention method lives in this file.
#pragma once
#include <cstdint>
#include <cuda.h>

namespace sagebwd {

__device__ __forceinline__ uint32_t smem_u32(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ uint64_t globaltimer_ns() {
  uint64_t t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
}

// ---------------------------------------------------------------- mbarrier
__device__ __forceinline__ void mbar_init(uint64_t* bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(bar)), "r"(count) : "memory");
}
__device__ __forceinline__ void fence_mbar_init() {
  asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}
__device__ __forceinline__ void mbar_arrive(uint64_t* bar) {
  asm volatile("mbarrier.arrive.release.cta.shared::cta.b64 _, [%0];" ::"r"(smem_u32(bar)) : "memory");
}
__device__ __forceinline__ void mbar_arrive_expect_tx(uint64_t* bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.release.cta.shared::cta.b64 _, [%0], %1;" ::"r"(smem_u32(bar)),
               "r"(bytes)
               : "memory");
}
__device__ __forceinline__ bool mbar_try_wait(uint64_t* bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.try_wait.parity.acquire.cta.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}\n"
      : "=r"(ok)
      : "r"(smem_u32(bar)), "r"(parity)
      : "memory");
  return ok != 0;
}
// Wait for the phase with the given parity to complete, giving up after
// limit_ns nanoseconds of %globaltimer.  Returns false on timeout; the caller
// then records the failure and leaves its loop instead of spinning forever.
__device__ __forceinline__ bool mbar_wait(uint64_t* bar, uint32_t parity, uint64_t limit_ns) {
  if (mbar_try_wait(bar, parity)) return true;
  const uint64_t t0 = globaltimer_ns();
  while (true) {
    if (mbar_try_wait(bar, parity)) return true;
    if (globaltimer_ns() - t0 > limit_ns) return false;
  }
}

// ---------------------------------------------------------------- fences
__device__ __forceinline__ void fence_proxy_async_smem() {
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}
__device__ __forceinline__ void named_bar_sync(uint32_t id, uint32_t nthreads) {
  asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(nthreads) : "memory");
}

// Warpgroup register reallocation: every thread of the warpgroup executes it.
template <uint32_t N>
__device__ __forceinline__ void setmaxnreg_inc() {
  asm volatile("setmaxnreg.inc.sync.aligned.u32 %0;" ::"n"(N));
}
template <uint32_t N>
__device__ __forceinline__ void setmaxnreg_dec() {
  asm volatile("setmaxnreg.dec.sync.aligned.u32 %0;" ::"n"(N));
}

// Move a warpgroup from the launch's per-thread register count to `To`: a
// decrease releases registers to the pool, an increase waits for them; an
// increase must never name a count below the current one, nor a decrease above it.
template <uint32_t To, uint32_t Launch>
__device__ __forceinline__ void setmaxnreg_to() {
  if constexpr (To < Launch)
    setmaxnreg_dec<To>();
  else if constexpr (To > Launch)
    setmaxnreg_inc<To>();
}

// Prefetch the 128-byte line holding p into L1 (no register result, never faults the thread).
__device__ __forceinline__ void prefetch_l1(const void* p) {
  asm volatile("prefetch.global.L1 [%0];" ::"l"(reinterpret_cast<uint64_t>(p)));
}

// ---------------------------------------------------------------- TMA
__device__ __forceinline__ void tma_prefetch_desc(const CUtensorMap* map) {
  asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(map)) : "memory");
}
// 3-D tiled load: coordinates are (x = innermost element, y, z).  The caller
// guarantees x * element_size is a multiple of 16 bytes.
__device__ __forceinline__ void tma_load_3d(void* smem_dst, const CUtensorMap* map, uint64_t* bar, int x, int y,
                                            int z) {
  asm volatile(
      "cp.async.bulk.tensor.3d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
      " [%0], [%1, {%3, %4, %5}], [%2];" ::"r"(smem_u32(smem_dst)),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(smem_u32(bar)), "r"(x), "r"(y), "r"(z)
      : "memory");
}
__device__ __forceinline__ void tma_load_2d(void* smem_dst, const CUtensorMap* map, uint64_t* bar, int x, int y) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
      " [%0], [%1, {%3, %4}], [%2];" ::"r"(smem_u32(smem_dst)),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(smem_u32(bar)), "r"(x), "r"(y)
      : "memory");
}
// 1-D bulk copy global -> shared, completing on an mbarrier: both addresses 16-byte aligned,
// bytes a multiple of 16.
__device__ __forceinline__ void bulk_load_1d(void* smem_dst, const void* gsrc, uint32_t bytes, uint64_t* bar) {
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(
          smem_u32(smem_dst)),
      "l"(reinterpret_cast<uint64_t>(gsrc)), "r"(bytes), "r"(smem_u32(bar))
      : "memory");
}

// 3-D tiled reduce-add of a shared-memory tile into global memory (element
// type from the tensor map), tracked by the issuing thread's bulk group.
__device__ __forceinline__ void tma_reduce_add_3d(const CUtensorMap* map, const void* smem_src, int x, int y, int z) {
  asm volatile(
      "cp.reduce.async.bulk.tensor.3d.global.shared::cta.add.tile.bulk_group [%0, {%2, %3, %4}], [%1];" ::"l"(
          reinterpret_cast<uint64_t>(map)),
      "r"(smem_u32(smem_src)), "r"(x), "r"(y), "r"(z)
      : "memory");
}
__device__ __forceinline__ void bulk_commit_group() { asm volatile("cp.async.bulk.commit_group;" ::: "memory"); }
// Wait until at most N committed bulk groups of this thread are still READING their shared-memory sources.
template <int N>
__device__ __forceinline__ void bulk_wait_group_read() {
  asm volatile("cp.async.bulk.wait_group.read %0;" ::"n"(N) : "memory");
}
// Wait until every committed bulk group of this thread has completed.
__device__ __forceinline__ void bulk_wait_group0() { asm volatile("cp.async.bulk.wait_group 0;" ::: "memory"); }

// ---------------------------------------------------------------- tcgen05
__device__ __forceinline__ void tmem_alloc(uint32_t* smem_result, uint32_t ncols) {
  asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(smem_u32(smem_result)),
               "r"(ncols)
               : "memory");
}
__device__ __forceinline__ void tmem_relinquish() {
  asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
}
__device__ __forceinline__ void tmem_dealloc(uint32_t taddr, uint32_t ncols) {
  asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(ncols) : "memory");
}
__device__ __forceinline__ void tc_fence_before() { asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory"); }
__device__ __forceinline__ void tc_fence_after() { asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory"); }

// D(tmem) (+)= A(smem) * B(smem), 16-bit operands, FP32 accumulator.
__device__ __forceinline__ void umma_ss(uint32_t d_tmem, uint64_t a_desc, uint64_t b_desc, uint32_t idesc,
                                        uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\tsetp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}\n" ::"r"(d_tmem),
      "l"(a_desc), "l"(b_desc), "r"(idesc), "r"(accumulate)
      : "memory");
}
// D(tmem) (+)= A(tmem) * B(smem).
__device__ __forceinline__ void umma_ts(uint32_t d_tmem, uint32_t a_tmem, uint64_t b_desc, uint32_t idesc,
                                        uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\tsetp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], %2, %3, p;\n\t}\n" ::"r"(d_tmem),
      "r"(a_tmem), "l"(b_desc), "r"(idesc), "r"(accumulate)
      : "memory");
}
// D(tmem) (+)= A(smem) * B(smem), FP8 E4M3 operands (kind::f8f6f4, K = 32 per instruction).
__device__ __forceinline__ void umma_f8_ss(uint32_t d_tmem, uint64_t a_desc, uint64_t b_desc, uint32_t idesc,
                                           uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\tsetp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::f8f6f4 [%0], %1, %2, %3, p;\n\t}\n" ::"r"(d_tmem),
      "l"(a_desc), "l"(b_desc), "r"(idesc), "r"(accumulate)
      : "memory");
}
// D(tmem) (+)= A(tmem) * B(smem), FP8 E4M3 operands; A packs four values per 32-bit column.
__device__ __forceinline__ void umma_f8_ts(uint32_t d_tmem, uint32_t a_tmem, uint64_t b_desc, uint32_t idesc,
                                           uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\tsetp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::f8f6f4 [%0], [%1], %2, %3, p;\n\t}\n" ::"r"(d_tmem),
      "r"(a_tmem), "l"(b_desc), "r"(idesc), "r"(accumulate)
      : "memory");
}
// ---------------------------------------------------------------- chained MMAs
// One K loop of tcgen05.mma kind::f16 in a single asm block (the first MMA
// overwrites D, the rest accumulate), so the issuing thread spends about three
// instructions per MMA.  The descriptors advance in 16-byte units of the start
// address: a K-major 128-byte-swizzled operand by 32 bytes per K step of 16
// (and to the next 16 KB sub-tile every four steps), an MN-major one by 16
// rows of 128 bytes.
// 8 K steps, A and B K-major.
__device__ __forceinline__ void umma_chain8_kk(uint32_t d_tmem, uint64_t a_desc, uint64_t b_desc, uint32_t idesc) {
  asm volatile(
      "{\n\t.reg .pred p0, p1;\n\t.reg .b64 ra, rb;\n\t"
      "setp.ne.b32 p0, 0, 0;\n\tsetp.eq.b32 p1, 0, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p0;\n\t"
      "add.s64 ra, %1, 2;\n\tadd.s64 rb, %2, 2;\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], ra, rb, %3, p1;\n\t"
      "add.s64 ra, %1, 4;\n\tadd.s64 rb, %2, 4;\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], ra, rb, %3, p1;\n\t"
      "add.s64 ra, %1, 6;\n\tadd.s64 rb, %2, 6;\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], ra, rb, %3, p1;\n\t"
      "add.s64 ra, %1, 1024;\n\tadd.s64 rb, %2, 1024;\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], ra, rb, %3, p1;\n\t"
      "add.s64 ra, %1, 1026;\n\tadd.s64 rb, %2, 1026;\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], ra, rb, %3, p1;\n\t"
      "add.s64 ra, %1, 1028;\n\tadd.s64 rb, %2, 1028;\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], ra, rb, %3, p1;\n\t"
      "add.s64 ra, %1, 1030;\n\tadd.s64 rb, %2, 1030;\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], ra, rb, %3, p1;\n\t"
      "}\n" ::"r"(d_tmem), "l"(a_desc), "l"(b_desc), "r"(idesc)
      : "memory");
}
// 4 K steps, A and B K-major.
__device__ __forceinline__ void umma_chain4_kk(uint32_t d_tmem, uint64_t a_desc, uint64_t b_desc, uint32_t idesc) {
  asm volatile(
      "{\n\t.reg .pred p0, p1;\n\t.reg .b64 ra, rb;\n\t"
      "setp.ne.b32 p0, 0, 0;\n\tsetp.eq.b32 p1, 0, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p0;\n\t"
      "add.s64 ra, %1, 2;\n\tadd.s64 rb, %2, 2;\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], ra, rb, %3, p1;\n\t"
      "add.s64 ra, %1, 4;\n\tadd.s64 rb, %2, 4;\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], ra, rb, %3, p1;\n\t"
      "add.s64 ra, %1, 6;\n\tadd.s64 rb, %2, 6;\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], ra, rb, %3, p1;\n\t"
      "}\n" ::"r"(d_tmem), "l"(a_desc), "l"(b_desc), "r"(idesc)
      : "memory");
}
// 8 K steps, A K-major, B MN-major.
__device__ __forceinline__ void umma_chain8_km(uint32_t d_tmem, uint64_t a_desc, uint64_t b_desc, uint32_t idesc) {
  asm volatile(
      "{\n\t.reg .pred p0, p1;\n\t.reg .b64 ra, rb;\n\t"
      "setp.ne.b32 p0, 0, 0;\n\tsetp.eq.b32 p1, 0, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p0;\n\t"
      "add.s64 ra, %1, 2;\n\tadd.s64 rb, %2, 128;\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], ra, rb, %3, p1;\n\t"
      "add.s64 ra, %1, 4;\n\tadd.s64 rb, %2, 256;\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], ra, rb, %3, p1;\n\t"
      "add.s64 ra, %1, 6;\n\tadd.s64 rb, %2, 384;\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], ra, rb, %3, p1;\n\t"
      "add.s64 ra, %1, 1024;\n\tadd.s64 rb, %2, 512;\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], ra, rb, %3, p1;\n\t"
      "add.s64 ra, %1, 1026;\n\tadd.s64 rb, %2, 640;\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], ra, rb, %3, p1;\n\t"
      "add.s64 ra, %1, 1028;\n\tadd.s64 rb, %2, 768;\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], ra, rb, %3, p1;\n\t"
      "add.s64 ra, %1, 1030;\n\tadd.s64 rb, %2, 896;\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], ra, rb, %3, p1;\n\t"
      "}\n" ::"r"(d_tmem), "l"(a_desc), "l"(b_desc), "r"(idesc)
      : "memory");
}
// 8 K steps, A and B MN-major.
__device__ __forceinline__ void umma_chain8_mm(uint32_t d_tmem, uint64_t a_desc, uint64_t b_desc, uint32_t idesc) {
  asm volatile(
      "{\n\t.reg .pred p0, p1;\n\t.reg .b64 ra, rb;\n\t"
      "setp.ne.b32 p0, 0, 0;\n\tsetp.eq.b32 p1, 0, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p0;\n\t"
      "add.s64 ra, %1, 128;\n\tadd.s64 rb, %2, 128;\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], ra, rb, %3, p1;\n\t"
      "add.s64 ra, %1, 256;\n\tadd.s64 rb, %2, 256;\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], ra, rb, %3, p1;\n\t"
      "add.s64 ra, %1, 384;\n\tadd.s64 rb, %2, 384;\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], ra, rb, %3, p1;\n\t"
      "add.s64 ra, %1, 512;\n\tadd.s64 rb, %2, 512;\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], ra, rb, %3, p1;\n\t"
      "add.s64 ra, %1, 640;\n\tadd.s64 rb, %2, 640;\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], ra, rb, %3, p1;\n\t"
      "add.s64 ra, %1, 768;\n\tadd.s64 rb, %2, 768;\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], ra, rb, %3, p1;\n\t"
      "add.s64 ra, %1, 896;\n\tadd.s64 rb, %2, 896;\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], ra, rb, %3, p1;\n\t"
      "}\n" ::"r"(d_tmem), "l"(a_desc), "l"(b_desc), "r"(idesc)
      : "memory");
}

// Arrive once on `bar` when every tcgen05 op issued so far by this thread has completed.
__device__ __forceinline__ void umma_commit(uint64_t* bar) {
  asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(
                   smem_u32(bar))
               : "memory");
}

// Instruction descriptor for kind::f16 with BF16 A/B and FP32 D.
// Bit layout (PTX ISA, tcgen05 instruction descriptor): [4,6) D format
// (1 = F32), [7,10) A format (1 = BF16), [10,13) B format (1 = BF16),
// 15 A major (1 = MN), 16 B major (1 = MN), [17,23) N>>3, [24,29) M>>4.
__host__ __device__ constexpr uint32_t idesc_bf16_f32(int M, int N, bool a_mn_major, bool b_mn_major) {
  return (1u << 4) | (1u << 7) | (1u << 10) | ((a_mn_major ? 1u : 0u) << 15) | ((b_mn_major ? 1u : 0u) << 16) |
         ((uint32_t)(N >> 3) << 17) | ((uint32_t)(M >> 4) << 24);
}

// Instruction descriptor for kind::f8f6f4 with E4M3 A/B (format 0) and FP32 D, both K-major.
__host__ __device__ constexpr uint32_t idesc_e4m3_f32(int M, int N) {
  return (1u << 4) | ((uint32_t)(N >> 3) << 17) | ((uint32_t)(M >> 4) << 24);
}
// Swizzle modes of the tcgen05 shared-memory descriptor (bits [61,64)).
constexpr uint32_t kSwizzle128B = 2, kSwizzle64B = 4;
// K-major descriptor with a given 8-row stride and swizzle mode (leading byte offset unused: 16).
__device__ __forceinline__ uint64_t sdesc_kmajor(uint32_t saddr, uint32_t sbo_bytes, uint32_t swizzle) {
  uint64_t d = 0;
  d |= (uint64_t)((saddr >> 4) & 0x3FFFu);
  d |= (uint64_t)(16u >> 4) << 16;
  d |= (uint64_t)((sbo_bytes >> 4) & 0x3FFFu) << 32;
  d |= (uint64_t)1u << 46;
  d |= (uint64_t)swizzle << 61;
  return d;
}
// Shared-memory matrix descriptor (tcgen05 layout): [0,14) start>>4,
// [16,30) leading byte offset>>4, [32,46) stride byte offset>>4,
// [46,48) version = 1, [61,64) swizzle mode (2 = 128-byte swizzle).
__device__ __forceinline__ uint64_t sdesc_sw128(uint32_t saddr, uint32_t lbo_bytes, uint32_t sbo_bytes) {
  uint64_t d = 0;
  d |= (uint64_t)((saddr >> 4) & 0x3FFFu);
  d |= (uint64_t)((lbo_bytes >> 4) & 0x3FFFu) << 16;
  d |= (uint64_t)((sbo_bytes >> 4) & 0x3FFFu) << 32;
  d |= (uint64_t)1u << 46;
  d |= (uint64_t)2u << 61;
  return d;
}

// Low 32 bits of a 128-byte-swizzle descriptor (start address and leading byte
// offset); the high half is the same for every descriptor with a 1024-byte
// stride offset, see sdesc_sw128_hi.
__device__ __forceinline__ uint32_t sdesc_sw128_lo(uint32_t saddr, uint32_t lbo_bytes) {
  return ((saddr >> 4) & 0x3FFFu) | (((lbo_bytes >> 4) & 0x3FFFu) << 16);
}
__host__ __device__ constexpr uint32_t sdesc_sw128_hi() { return (1024u >> 4) | (1u << 14) | (2u << 29); }
__device__ __forceinline__ uint64_t sdesc_from_lo(uint32_t lo) {
  return ((uint64_t)sdesc_sw128_hi() << 32) | lo;
}

// ---------------------------------------------------------------- programmatic dependent launch
// A grid launched with the programmatic-serialization attribute may start before the grid ahead
// of it in the stream has finished; pdl_wait blocks until that grid has completed and its memory
// is visible (a no-op for a grid launched without the attribute).  pdl_trigger lets the next such
// grid start once every CTA of this one has issued it (or exited).
__device__ __forceinline__ void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
__device__ __forceinline__ void pdl_trigger() { asm volatile("griddepcontrol.launch_dependents;" ::: "memory"); }

// ---------------------------------------------------------------- TMEM ld / st
__device__ __forceinline__ void tmem_ld8(uint32_t taddr, uint32_t (&r)[8]) {
  asm volatile("tcgen05.ld.sync.aligned.32x32b.x8.b32 {%0,%1,%2,%3,%4,%5,%6,%7}, [%8];"
               : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7])
               : "r"(taddr));
}
__device__ __forceinline__ void tmem_st8(uint32_t taddr, const uint32_t (&r)[8]) {
  asm volatile("tcgen05.st.sync.aligned.32x32b.x8.b32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8};" ::"r"(taddr), "r"(r[0]),
               "r"(r[1]), "r"(r[2]), "r"(r[3]), "r"(r[4]), "r"(r[5]), "r"(r[6]), "r"(r[7])
               : "memory");
}
__device__ __forceinline__ void tmem_st4(uint32_t taddr, const uint32_t (&r)[4]) {
  asm volatile("tcgen05.st.sync.aligned.32x32b.x4.b32 [%0], {%1,%2,%3,%4};" ::"r"(taddr), "r"(r[0]), "r"(r[1]),
               "r"(r[2]), "r"(r[3])
               : "memory");
}
#define SB_R8(i) "=r"(r[i + 0]), "=r"(r[i + 1]), "=r"(r[i + 2]), "=r"(r[i + 3]), "=r"(r[i + 4]), "=r"(r[i + 5]), \
                 "=r"(r[i + 6]), "=r"(r[i + 7])
// 32 lanes x 32 bits, 16 consecutive columns: thread t of the warp gets lane (base + t), cols [c, c+16).
__device__ __forceinline__ void tmem_ld16(uint32_t taddr, uint32_t (&r)[16]) {
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x16.b32 "
      "{%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15}, [%16];"
      : SB_R8(0), SB_R8(8)
      : "r"(taddr));
}
__device__ __forceinline__ void tmem_ld32(uint32_t taddr, uint32_t (&r)[32]) {
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x32.b32 "
      "{%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,"
      "%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31}, [%32];"
      : SB_R8(0), SB_R8(8), SB_R8(16), SB_R8(24)
      : "r"(taddr));
}
#undef SB_R8
__device__ __forceinline__ void tmem_ld_wait() { asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory"); }

#define SB_W8(i) "r"(r[i + 0]), "r"(r[i + 1]), "r"(r[i + 2]), "r"(r[i + 3]), "r"(r[i + 4]), "r"(r[i + 5]), \
                 "r"(r[i + 6]), "r"(r[i + 7])
__device__ __forceinline__ void tmem_st16(uint32_t taddr, const uint32_t (&r)[16]) {
  asm volatile(
      "tcgen05.st.sync.aligned.32x32b.x16.b32 [%0], "
      "{%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16};" ::"r"(taddr),
      SB_W8(0), SB_W8(8)
      : "memory");
}
#undef SB_W8
// tcgen05.wait::ld naming the destination registers of the loads it waits for,
// so that the compiler cannot schedule a use of them above the wait.
__device__ __forceinline__ void tmem_ld_wait_regs(uint32_t (&r)[16]) {
  asm volatile("tcgen05.wait::ld.sync.aligned;"
               : "+r"(r[0]), "+r"(r[1]), "+r"(r[2]), "+r"(r[3]), "+r"(r[4]), "+r"(r[5]), "+r"(r[6]), "+r"(r[7]),
                 "+r"(r[8]), "+r"(r[9]), "+r"(r[10]), "+r"(r[11]), "+r"(r[12]), "+r"(r[13]), "+r"(r[14]), "+r"(r[15])
               :
               : "memory");
}
__device__ __forceinline__ void tmem_ld_wait_regs(uint32_t (&r)[8]) {
  asm volatile("tcgen05.wait::ld.sync.aligned;"
               : "+r"(r[0]), "+r"(r[1]), "+r"(r[2]), "+r"(r[3]), "+r"(r[4]), "+r"(r[5]), "+r"(r[6]), "+r"(r[7])
               :
               : "memory");
}
__device__ __forceinline__ void tmem_st_wait() { asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory"); }

// ---------------------------------------------------------------- scalar helpers
__device__ __forceinline__ float ex2_approx(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}
// Round to nearest integer, ties to even (the C rint() of the default mode).
__device__ __forceinline__ float rint_f32(float x) {
  float y;
  asm("cvt.rni.f32.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}
// Packed FP32 on sm_100-class parts: one instruction performs two IEEE
// round-to-nearest operations on a register pair, so the elementwise softmax
// work costs half the issue slots.  Each lane's result equals the scalar op's.
__device__ __forceinline__ float2 ffma2(float2 a, float2 b, float2 c) {
  float2 d;
  asm("{\n\t.reg .b64 ra, rb, rc, rd;\n\tmov.b64 ra, {%2, %3};\n\tmov.b64 rb, {%4, %5};\n\tmov.b64 rc, {%6, %7};\n\t"
      "fma.rn.f32x2 rd, ra, rb, rc;\n\tmov.b64 {%0, %1}, rd;\n\t}"
      : "=f"(d.x), "=f"(d.y)
      : "f"(a.x), "f"(a.y), "f"(b.x), "f"(b.y), "f"(c.x), "f"(c.y));
  return d;
}
__device__ __forceinline__ float2 fadd2(float2 a, float2 b) {
  float2 d;
  asm("{\n\t.reg .b64 ra, rb, rd;\n\tmov.b64 ra, {%2, %3};\n\tmov.b64 rb, {%4, %5};\n\t"
      "add.rn.f32x2 rd, ra, rb;\n\tmov.b64 {%0, %1}, rd;\n\t}"
      : "=f"(d.x), "=f"(d.y)
      : "f"(a.x), "f"(a.y), "f"(b.x), "f"(b.y));
  return d;
}
__device__ __forceinline__ float2 fmul2(float2 a, float2 b) {
  float2 d;
  asm("{\n\t.reg .b64 ra, rb, rd;\n\tmov.b64 ra, {%2, %3};\n\tmov.b64 rb, {%4, %5};\n\t"
      "mul.rn.f32x2 rd, ra, rb;\n\tmov.b64 {%0, %1}, rd;\n\t}"
      : "=f"(d.x), "=f"(d.y)
      : "f"(a.x), "f"(a.y), "f"(b.x), "f"(b.y));
  return d;
}
// A register pair holding two FP32 lanes (lo, hi), for accumulators that stay packed.
__device__ __forceinline__ uint64_t pack_f32x2(float lo, float hi) {
  uint64_t r;
  asm("mov.b64 %0, {%1, %2};" : "=l"(r) : "f"(lo), "f"(hi));
  return r;
}
__device__ __forceinline__ float lo_f32(uint64_t x) { return __uint_as_float(static_cast<uint32_t>(x)); }
__device__ __forceinline__ float hi_f32(uint64_t x) { return __uint_as_float(static_cast<uint32_t>(x >> 32)); }
// acc = w2 * (v0, v1) + acc, lane by lane
__device__ __forceinline__ void ffma2_acc(uint64_t& acc, uint64_t w2, uint32_t v0, uint32_t v1) {
  asm("{\n\t.reg .b64 rv;\n\tmov.b64 rv, {%2, %3};\n\tfma.rn.f32x2 %0, %1, rv, %0;\n\t}"
      : "+l"(acc)
      : "l"(w2), "r"(v0), "r"(v1));
}
// acc = acc * a2, lane by lane
__device__ __forceinline__ void fmul2_acc(uint64_t& acc, uint64_t a2) {
  asm("mul.rn.f32x2 %0, %0, %1;" : "+l"(acc) : "l"(a2));
}
// Three-input maximum (one instruction on sm_100-class parts).
__device__ __forceinline__ float fmax3(float a, float b, float c) {
  float d;
  asm("max.f32 %0, %1, %2, %3;" : "=f"(d) : "f"(a), "f"(b), "f"(c));
  return d;
}
// Two floats rounded to FP8 E4M3 (to nearest even, saturating at +-448) and returned as bf16x2
// (lo = a, hi = b): E4M3 values convert exactly to FP16, FP32 and BF16.
__device__ __forceinline__ uint32_t e4m3x2_bf16x2(float a, float b) {
  uint16_t e;
  asm("cvt.rn.satfinite.e4m3x2.f32 %0, %2, %1;" : "=h"(e) : "f"(a), "f"(b));
  uint32_t h;
  asm("cvt.rn.f16x2.e4m3x2 %0, %1;" : "=r"(h) : "h"(e));
  float lo, hi;
  asm("{\n\t.reg .b16 l, u;\n\tmov.b32 {l, u}, %2;\n\tcvt.f32.f16 %0, l;\n\tcvt.f32.f16 %1, u;\n\t}"
      : "=f"(lo), "=f"(hi)
      : "r"(h));
  uint32_t r;
  asm("cvt.rn.bf16x2.f32 %0, %2, %1;" : "=r"(r) : "f"(lo), "f"(hi));
  return r;
}
// Two floats rounded to FP8 E4M3 (to nearest even, saturating) as two bytes (lo = a, hi = b).
__device__ __forceinline__ uint32_t e4m3x2_bytes(float a, float b) {
  uint16_t e;
  asm("cvt.rn.satfinite.e4m3x2.f32 %0, %2, %1;" : "=h"(e) : "f"(a), "f"(b));
  return (uint32_t)e;
}
// Pack two floats into bf16x2 (lo = a, hi = b), round to nearest even.
__device__ __forceinline__ uint32_t pack_bf16x2(float a, float b) {
  uint32_t r;
  asm("cvt.rn.bf16x2.f32 %0, %2, %1;" : "=r"(r) : "f"(a), "f"(b));
  return r;
}
// A 16-byte shared load kept in program order (volatile), so that an unrolled loop
// does not hoist all of its loads ahead and run out of registers.
__device__ __forceinline__ float4 ld_shared_v4_f32(uint32_t addr) {
  float4 v;
  asm volatile("ld.shared.v4.f32 {%0,%1,%2,%3}, [%4];" : "=f"(v.x), "=f"(v.y), "=f"(v.z), "=f"(v.w) : "r"(addr));
  return v;
}
__device__ __forceinline__ void st_shared_v4(uint32_t addr, uint32_t a, uint32_t b, uint32_t c, uint32_t d) {
  asm volatile("st.shared.v4.b32 [%0], {%1,%2,%3,%4};" ::"r"(addr), "r"(a), "r"(b), "r"(c), "r"(d) : "memory");
}
__device__ __forceinline__ void red_add_v4_f32(float* gptr, float a, float b, float c, float d) {
  asm volatile("red.global.add.v4.f32 [%0], {%1,%2,%3,%4};" ::"l"(gptr), "f"(a), "f"(b), "f"(c), "f"(d)
               : "memory");
}

}  // namespace sagebwd
