// PTX wrappers shared by the tcgen05 kernels (MLA and many-row GQA):
// mbarriers with bounded waits, TMA tile copies, shared-memory matrix and
// instruction descriptors for tcgen05.mma kind::f16 (bf16 in, fp32 out),
// tcgen05 MMA issue / commit / fences, TMEM loads and stores, and the bf16
// packing of P. Internal linkage: every translation unit gets its own copy.
#pragma once

#include <cuda.h>
#include <cudaTypedefs.h>
#include <cuda_bf16.h>
#include <stdint.h>

#include <mutex>

#include "dcp_internal.cuh"

namespace dcp {
namespace {

// Polls before a wait gives up. A build may lower it (-DDCP_SPIN_LIMIT=n) to
// exercise the expiry path: every kernel then aborts at its first wait that
// is not already satisfied, raises DCP_DEVERR_TIMEOUT and returns.
#ifndef DCP_SPIN_LIMIT
#define DCP_SPIN_LIMIT (1u << 24)
#endif
constexpr uint32_t kSpinLimit = DCP_SPIN_LIMIT;

__device__ __forceinline__ uint32_t saddr(const void* p) { return static_cast<uint32_t>(__cvta_generic_to_shared(p)); }

__device__ __forceinline__ uint32_t cluster_rank() {
  uint32_t r;
  asm volatile("mov.u32 %0, %%cluster_ctarank;\n" : "=r"(r));
  return r;
}
__device__ __forceinline__ void bar_init(uint32_t b, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;\n" ::"r"(b), "r"(count));
}
__device__ __forceinline__ void bar_arrive(uint32_t b) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];\n" ::"r"(b) : "memory");
}
__device__ __forceinline__ void bar_arrive_tx(uint32_t b, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;\n" ::"r"(b), "r"(bytes) : "memory");
}
__device__ __forceinline__ bool bar_try(uint32_t b, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n .reg .pred p;\n mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n selp.u32 %0, 1, 0, p;\n}\n"
      : "=r"(ok) : "r"(b), "r"(parity) : "memory");
  return ok != 0;
}
__device__ __forceinline__ bool bar_try_cluster(uint32_t b, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n .reg .pred p;\n mbarrier.try_wait.parity.acquire.cluster.shared::cta.b64 p, [%1], %2;\n"
      " selp.u32 %0, 1, 0, p;\n}\n"
      : "=r"(ok) : "r"(b), "r"(parity) : "memory");
  return ok != 0;
}
// Non-blocking probe: unlike try_wait, test_wait never suspends the thread,
// so a loop polling several barriers reacts to whichever completes first.
__device__ __forceinline__ bool bar_test(uint32_t b, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n .reg .pred p;\n mbarrier.test_wait.parity.shared::cta.b64 p, [%1], %2;\n selp.u32 %0, 1, 0, p;\n}\n"
      : "=r"(ok) : "r"(b), "r"(parity) : "memory");
  return ok != 0;
}
// Poll by a whole warp: true only if every lane saw the phase complete, so
// the warp's control flow stays uniform.
__device__ __forceinline__ bool bar_test_warp(uint32_t b, uint32_t parity) {
  return __all_sync(0xffffffffu, bar_test(b, parity));
}
// Bounded wait. Returns false if the kernel is aborting (this wait expired, or
// another role's did): the caller then stops.
__device__ __noinline__ bool wait_bar(uint32_t b, uint32_t parity, volatile int* abort_flag, int32_t* err,
                                      bool cluster_scope = false) {
  for (uint32_t i = 0; i < kSpinLimit; ++i) {
    if (cluster_scope ? bar_try_cluster(b, parity) : bar_try(b, parity)) return true;
    if ((i & 63u) == 63u && *abort_flag) return false;
  }
  *abort_flag = 1;
  raise_flag(err, DCP_DEVERR_TIMEOUT);
  return false;
}
// Warp-uniform bounded wait: the warp proceeds only if every lane's wait
// succeeded, so the .sync.aligned TMEM accesses that follow always run with
// the whole warp (and an abort leaves the warp together).
__device__ __forceinline__ bool wait_warp(uint32_t b, uint32_t parity, volatile int* abort_flag, int32_t* err,
                                          bool cluster_scope = false) {
  const bool ok = wait_bar(b, parity, abort_flag, err, cluster_scope);
  return __all_sync(0xffffffffu, ok);
}
// Bounded wait that ignores the abort flag (teardown drains: copies and MMAs
// already issued always complete). Polled, so the bound is a poll count.
__device__ __forceinline__ void drain_bar(uint32_t b, uint32_t parity) {
  for (uint32_t i = 0; i < (1u << 22); ++i)
    if (bar_test(b, parity)) return;
}

__device__ __forceinline__ void tma_load(uint32_t dst, const CUtensorMap* map, int x, int y, uint32_t bar) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes [%0], [%1, {%2, %3}], [%4];\n"
      ::"r"(dst), "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y), "r"(bar) : "memory");
}

// The same tile copy delivered to the same shared-memory offset of every CTA
// of the cluster in cta_mask, each of whose mbarriers at offset `bar`
// receives the bytes that land in that CTA.
__device__ __forceinline__ void tma_load_mc(uint32_t dst, const CUtensorMap* map, int x, int y, uint32_t bar,
                                            uint16_t cta_mask) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes.multicast::cluster"
      " [%0], [%1, {%2, %3}], [%4], %5;\n"
      ::"r"(dst), "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y), "r"(bar), "h"(cta_mask) : "memory");
}
// All threads of every CTA of the cluster meet here (release / acquire).
__device__ __forceinline__ void cluster_sync() {
  asm volatile("barrier.cluster.arrive.release.aligned;\nbarrier.cluster.wait.acquire.aligned;\n" ::: "memory");
}

// Plain bulk copy of `bytes` contiguous bytes (a multiple of 16, both
// addresses 16-byte aligned) into this CTA's shared memory.
__device__ __forceinline__ void bulk_load(uint32_t dst, const void* src, uint32_t bytes, uint32_t bar) {
  asm volatile("cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];\n"
               ::"r"(dst), "l"(src), "r"(bytes), "r"(bar) : "memory");
}

// Pull `bytes` (a multiple of 16, 16-byte aligned) of global memory into L2.
__device__ __forceinline__ void l2_prefetch(const void* src, uint32_t bytes) {
  asm volatile("cp.async.bulk.prefetch.L2.global [%0], %1;\n" ::"l"(src), "r"(bytes) : "memory");
}

// Shared-memory matrix descriptor: 128-byte swizzle, 8-row groups 1024 B apart.
// lbo is the byte stride between 64-element atoms along M/N for MN-major
// operands (unused for K-major ones).
__device__ __forceinline__ uint64_t sdesc(uint32_t addr, uint32_t lbo) {
  uint64_t d = (uint64_t)((addr >> 4) & 0x3FFF);
  d |= (uint64_t)((lbo >> 4) & 0x3FFF) << 16;
  d |= (uint64_t)(1024 >> 4) << 32;
  d |= 1ull << 46;   // descriptor version for tcgen05
  d |= 2ull << 61;   // 128-byte swizzle
  return d;
}
// Instruction descriptor, kind::f16: bf16 A/B (fp16 with f16 set), fp32 accumulate.
__host__ __device__ constexpr uint32_t idesc(int M, int N, int b_mn_major, bool f16 = false) {
  return (1u << 4) | (f16 ? 0u : (1u << 7) | (1u << 10)) | ((uint32_t)b_mn_major << 16) |
         ((uint32_t)(N >> 3) << 17) | ((uint32_t)(M >> 4) << 24);
}
// D (+)= A . B with A and B in shared memory; the whole warp calls, one elected lane issues
__device__ __forceinline__ void mma_ss(uint32_t d, uint64_t a, uint64_t b, uint32_t id, int accumulate) {
  asm volatile(
      "{\n .reg .pred p, e;\n elect.sync _|e, 0xffffffff;\n setp.ne.b32 p, %4, 0;\n"
      " @e tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n}\n"
      ::"r"(d), "l"(a), "l"(b), "r"(id), "r"(accumulate));
}
// D (+)= A . B with A read from tensor memory
__device__ __forceinline__ void mma_ts(uint32_t d, uint32_t a_tmem, uint64_t b, uint32_t id, int accumulate) {
  asm volatile(
      "{\n .reg .pred p, e;\n elect.sync _|e, 0xffffffff;\n setp.ne.b32 p, %4, 0;\n"
      " @e tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], %2, %3, p;\n}\n"
      ::"r"(d), "r"(a_tmem), "l"(b), "r"(id), "r"(accumulate));
}
__device__ __forceinline__ void mma_commit(uint32_t bar) {
  asm volatile("{\n .reg .pred e;\n elect.sync _|e, 0xffffffff;\n"
               " @e tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];\n}\n" ::"r"(bar)
               : "memory");
}
// As mma_commit, arriving on the mbarrier at offset `bar` of every CTA in cta_mask.
__device__ __forceinline__ void mma_commit_mc(uint32_t bar, uint16_t cta_mask) {
  asm volatile("{\n .reg .pred e;\n elect.sync _|e, 0xffffffff;\n"
               " @e tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.multicast::cluster.b64 [%0], %1;\n}\n"
               ::"r"(bar), "h"(cta_mask) : "memory");
}
__device__ __forceinline__ void tc_fence_before() { asm volatile("tcgen05.fence::before_thread_sync;\n" ::: "memory"); }
__device__ __forceinline__ void tc_fence_after() { asm volatile("tcgen05.fence::after_thread_sync;\n" ::: "memory"); }
__device__ __forceinline__ void tmem_wait_ld() { asm volatile("tcgen05.wait::ld.sync.aligned;\n" ::: "memory"); }
__device__ __forceinline__ void tmem_wait_st() { asm volatile("tcgen05.wait::st.sync.aligned;\n" ::: "memory"); }
__device__ __forceinline__ void tmem_ld32(uint32_t taddr, uint32_t* r) {
  asm volatile("tcgen05.ld.sync.aligned.32x32b.x32.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31}, [%32];\n"
               : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15]), "=r"(r[16]), "=r"(r[17]), "=r"(r[18]), "=r"(r[19]), "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]), "=r"(r[24]), "=r"(r[25]), "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]), "=r"(r[31])
               : "r"(taddr));
}
__device__ __forceinline__ void tmem_st32(uint32_t taddr, const uint32_t* r) {
  asm volatile("tcgen05.st.sync.aligned.32x32b.x32.b32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31,%32};\n"
               :: "r"(taddr), "r"(r[0]), "r"(r[1]), "r"(r[2]), "r"(r[3]), "r"(r[4]), "r"(r[5]), "r"(r[6]), "r"(r[7]), "r"(r[8]), "r"(r[9]), "r"(r[10]), "r"(r[11]), "r"(r[12]), "r"(r[13]), "r"(r[14]), "r"(r[15]), "r"(r[16]), "r"(r[17]), "r"(r[18]), "r"(r[19]), "r"(r[20]), "r"(r[21]), "r"(r[22]), "r"(r[23]), "r"(r[24]), "r"(r[25]), "r"(r[26]), "r"(r[27]), "r"(r[28]), "r"(r[29]), "r"(r[30]), "r"(r[31]) : "memory");
}
__device__ __forceinline__ void tmem_st16(uint32_t taddr, const uint32_t* r) {
  asm volatile(
      "tcgen05.st.sync.aligned.32x32b.x16.b32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16};\n"
      ::"r"(taddr), "r"(r[0]), "r"(r[1]), "r"(r[2]), "r"(r[3]), "r"(r[4]), "r"(r[5]), "r"(r[6]), "r"(r[7]),
      "r"(r[8]), "r"(r[9]), "r"(r[10]), "r"(r[11]), "r"(r[12]), "r"(r[13]), "r"(r[14]), "r"(r[15])
      : "memory");
}
__device__ __forceinline__ void st_shared_v4(uint32_t a, uint32_t x, uint32_t y, uint32_t z, uint32_t w) {
  asm volatile("st.shared.v4.b32 [%0], {%1, %2, %3, %4};\n" ::"r"(a), "r"(x), "r"(y), "r"(z), "r"(w) : "memory");
}
// 2^x on the SFU, denormal results flushed to zero
__device__ __forceinline__ float ex2_ftz(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;\n" : "=f"(y) : "f"(x));
  return y;
}
// Packed fp32 pairs (one instruction for two lanes of work) and three-input
// extrema, to thin the softmax warps' instruction streams.
__device__ __forceinline__ unsigned long long f2pack(float a, float b) {
  unsigned long long r;
  asm("mov.b64 %0, {%1, %2};" : "=l"(r) : "f"(a), "f"(b));
  return r;
}
__device__ __forceinline__ void f2unpack(unsigned long long r, float& a, float& b) {
  asm("mov.b64 {%0, %1}, %2;" : "=f"(a), "=f"(b) : "l"(r));
}
__device__ __forceinline__ unsigned long long ffma2(unsigned long long a, unsigned long long b, unsigned long long c) {
  unsigned long long d;
  asm("fma.rn.f32x2 %0, %1, %2, %3;" : "=l"(d) : "l"(a), "l"(b), "l"(c));
  return d;
}
__device__ __forceinline__ unsigned long long fadd2(unsigned long long a, unsigned long long b) {
  unsigned long long d;
  asm("add.rn.f32x2 %0, %1, %2;" : "=l"(d) : "l"(a), "l"(b));
  return d;
}
__device__ __forceinline__ float max3f(float a, float b, float c) {
  float d;
  asm("max.f32 %0, %1, %2, %3;" : "=f"(d) : "f"(a), "f"(b), "f"(c));
  return d;
}
__device__ __forceinline__ float min3f(float a, float b, float c) {
  float d;
  asm("min.f32 %0, %1, %2, %3;" : "=f"(d) : "f"(a), "f"(b), "f"(c));
  return d;
}
// maximum (MAX) or minimum of 32 or 64 fp32 bit patterns, as a tree of
// three-input extrema (17 / 32 instructions instead of 31 / 63)
template <int N, bool MAX>
__device__ __forceinline__ float ext_tree(const uint32_t* v) {
  static_assert(N == 32 || N == 64, "32 or 64 values");
  auto e3 = [](float a, float b, float c) { return MAX ? max3f(a, b, c) : min3f(a, b, c); };
  auto e2 = [](float a, float b) { return MAX ? fmaxf(a, b) : fminf(a, b); };
  auto f = [&](int i) { return __uint_as_float(v[i]); };
  if constexpr (N == 64) {
    float t[22], u[8];
#pragma unroll
    for (int i = 0; i < 21; ++i) t[i] = e3(f(3 * i), f(3 * i + 1), f(3 * i + 2));
    t[21] = f(63);
#pragma unroll
    for (int i = 0; i < 7; ++i) u[i] = e3(t[3 * i], t[3 * i + 1], t[3 * i + 2]);
    u[7] = t[21];
    return e3(e3(u[0], u[1], u[2]), e3(u[3], u[4], u[5]), e2(u[6], u[7]));
  } else {
    float t[11];
#pragma unroll
    for (int i = 0; i < 10; ++i) t[i] = e3(f(3 * i), f(3 * i + 1), f(3 * i + 2));
    t[10] = e2(f(30), f(31));
    return e2(e3(e3(t[0], t[1], t[2]), e3(t[3], t[4], t[5]), e3(t[6], t[7], t[8])), e2(t[9], t[10]));
  }
}

// bf16 pair (x0 in the low half), round to nearest even
__device__ __forceinline__ uint32_t pack_bf16(float x0, float x1) {
  const __nv_bfloat162 h = __floats2bfloat162_rn(x0, x1);
  return *reinterpret_cast<const uint32_t*>(&h);
}
// P as two bf16 terms without conversion instructions (they share the SFU's
// issue rate with ex2): hi = x rounded to bf16 (half-way cases up, which for
// x >= 0 moves hi by at most half an ulp: |x - hi| <= 2^-8 |x|), taken as the
// top 16 bits of x + 2^15 (as bits) with a byte permute; lo = the remainder
// x - hi (exact in fp32) truncated to bf16, so |x - hi - lo| < 2^-15 |x|.
// Pairs: x0 in the low half of each word. For finite x >= 0 below 2^127.
__device__ __forceinline__ void split_p_bf16(float x0, float x1, uint32_t& hi, uint32_t& lo) {
  const uint32_t u0 = __float_as_uint(x0) + 0x8000u, u1 = __float_as_uint(x1) + 0x8000u;
  hi = __byte_perm(u0, u1, 0x7632);
  const float r0 = x0 - __uint_as_float(u0 & 0xFFFF0000u);
  const float r1 = x1 - __uint_as_float(u1 & 0xFFFF0000u);
  lo = __byte_perm(__float_as_uint(r0), __float_as_uint(r1), 0x7632);
}
// bf16 pair of the rounding residuals x - bf16(x)
__device__ __forceinline__ uint32_t residual_bf16(float x0, float x1) {
  const __nv_bfloat162 h = __floats2bfloat162_rn(x0, x1);
  const float2 hf = __bfloat1622float2(h);
  return pack_bf16(x0 - hf.x, x1 - hf.y);
}

// cuTensorMapEncodeTiled from the driver, looked up once.
inline PFN_cuTensorMapEncodeTiled_v12000 tensor_map_encoder() {
  static std::once_flag once;
  static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
  std::call_once(once, [] {
    void* f = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &f, 12000, cudaEnableDefault, &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(f);
  });
  return fn;
}

}  // namespace
}  // namespace dcp
