// common.cuh -- device helpers shared by the libvarlen_ssm kernels (sm_103a).
#pragma once

#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include <algorithm>

#include "kernels.h"

namespace vssm {

constexpr float kLog2e = 1.4426950408889634f;

// Device checks of the VSSM_CHECKS=1 build: VSSM_CHECKED(cond, status) is
// cond, and when cond fails it ORs kStatusDeviceCheck into *status, so that
// the caller can skip the access it guards; in the ordinary build it is the
// constant true and costs nothing.  Nothing traps.
__device__ __forceinline__ bool device_check(bool cond, int* status) {
  if (!cond && status) atomicOr(status, kStatusDeviceCheck);
  return cond;
}
#if VSSM_CHECKS
#define VSSM_CHECKED(cond, status) ::vssm::device_check((cond), (status))
#else
#define VSSM_CHECKED(cond, status) true
#endif

// look-back flag values
enum : int { kFlagNone = 0, kFlagAggregate = 1, kFlagInclusive = 2 };

// ------------------------------------------------------------------ I/O types
__device__ __forceinline__ float to_f(float v) { return v; }
__device__ __forceinline__ float to_f(__nv_bfloat16 v) { return __bfloat162float(v); }

template <typename T> __device__ __forceinline__ T from_f(float v);
template <> __device__ __forceinline__ float from_f<float>(float v) { return v; }
template <> __device__ __forceinline__ __nv_bfloat16 from_f<__nv_bfloat16>(float v) {
  return __float2bfloat16_rn(v);
}

// ------------------------------------------------------------------ math
// 2^x on the MUFU unit (PTX ex2.approx, flush-to-zero): exp(x) = ex2(x * log2 e).
__device__ __forceinline__ float ex2(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

__device__ __forceinline__ float sigmoidf_fast(float x) {
  return __fdividef(1.0f, 1.0f + ex2(-x * kLog2e));
}

// SiLU(x) = x * sigmoid(x)
__device__ __forceinline__ float siluf(float x) { return x * sigmoidf_fast(x); }

// 2^x's inverse on the MUFU unit (PTX lg2.approx, flush-to-zero).
__device__ __forceinline__ float lg2(float x) {
  float y;
  asm("lg2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

// softplus(x) = log(1 + e^x) = max(x, 0) + log1p(e), e = e^-|x| in (0, 1], and
// its derivative sigmoid(x) = 1 / (1 + e) for x >= 0, e / (1 + e) below.
// log1p(e) = ln 2 * log2(1 + e) for e >= 1/32 (one MUFU lg2: relative error
// of a few 1e-6 there), and the series e - e^2/2 + e^3/3 - e^4/4 below 1/32
// (truncation error under e^4 / 5 < 2e-7 relative).  Three MUFU operations
// for both values.
__device__ __forceinline__ float softplus_sig(float x, float* sig) {
  const float e = ex2(-fabsf(x) * kLog2e);
  const float ope = 1.0f + e;
  const float series = e * fmaf(e, fmaf(e, fmaf(e, -0.25f, 0.33333334f), -0.5f), 1.0f);
  const float l1p = e >= 0.03125f ? lg2(ope) * 0.6931471805599453f : series;
  const float r = __fdividef(1.0f, ope);  // MUFU reciprocal, relative error ~2^-22
  *sig = x >= 0.0f ? r : e * r;
  return fmaxf(x, 0.0f) + l1p;
}

__device__ __forceinline__ float softplusf(float x) {
  float s;
  return softplus_sig(x, &s);
}

// ------------------------------------------------------------------ packed FP32 pairs
// Two lanes of FP32 per instruction (fma/mul.rn.f32x2): the FMA pipe does the
// same work, but the pair costs one issue slot.  Each component is rounded
// exactly as the scalar instruction would round it.
__device__ __forceinline__ float2 splat2(float v) { return make_float2(v, v); }
__device__ __forceinline__ float2 mul2(float2 a, float2 b) { return __fmul2_rn(a, b); }
__device__ __forceinline__ float2 fma2(float2 a, float2 b, float2 c) { return __ffma2_rn(a, b, c); }
__device__ __forceinline__ float2 ex2x2(float2 x) { return make_float2(ex2(x.x), ex2(x.y)); }

// Loads N fp32 values (16-byte aligned shared memory) as N/2 pairs.
template <int N>
__device__ __forceinline__ void lds_pairs(float2 (&v)[N / 2], const float* p) {
#pragma unroll
  for (int i = 0; i < N / 2; i += 2) {
    const float4 q = *reinterpret_cast<const float4*>(p + 2 * i);
    v[i] = make_float2(q.x, q.y);
    v[i + 1] = make_float2(q.z, q.w);
  }
}

// ------------------------------------------------------------------ timers, memory order
__device__ __forceinline__ uint64_t globaltimer_ns() {
  uint64_t t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
}

__device__ __forceinline__ int ld_acquire_gpu(const int* p) {
  int v;
  asm volatile("ld.acquire.gpu.global.b32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
  return v;
}

__device__ __forceinline__ void st_release_gpu(int* p, int v) {
  asm volatile("st.release.gpu.global.b32 [%0], %1;" ::"l"(p), "r"(v) : "memory");
}

__device__ __forceinline__ void st_relaxed_gpu(int* p, int v) {
  asm volatile("st.relaxed.gpu.global.b32 [%0], %1;" ::"l"(p), "r"(v) : "memory");
}

// Orders this thread's earlier memory accesses before its later ones, for
// observers anywhere on the GPU.
__device__ __forceinline__ void fence_acq_rel_gpu() { asm volatile("fence.acq_rel.gpu;" ::: "memory"); }

// Spin (with backoff) until *flag != 0 or `limit_ns` passes.  Returns the flag
// value, or 0 after a timeout (the caller records the error and carries on).
__device__ __forceinline__ int wait_flag(const int* flag, uint64_t limit_ns) {
  int v = ld_acquire_gpu(flag);
  if (v != 0) return v;
  const uint64_t t0 = globaltimer_ns();
  unsigned backoff = 32;
  for (;;) {
    __nanosleep(backoff);
    v = ld_acquire_gpu(flag);
    if (v != 0) return v;
    if (globaltimer_ns() - t0 > limit_ns) return 0;
    if (backoff < 1024) backoff <<= 1;
  }
}

// Sleeps about `ns` nanoseconds (a test knob's delay; always ends).
__device__ __forceinline__ void sleep_ns(uint64_t ns) {
  const uint64_t t0 = globaltimer_ns();
  while (globaltimer_ns() - t0 < ns) __nanosleep(1000);
}

// A carry word that holds no value yet: the all-ones NaN.  The caller fills a
// carry array with it before the launch.  FP32 arithmetic never yields it (a
// NaN result is the canonical 0x7fffffff) and st_carry turns it into that NaN
// all the same, so a carry word is its own flag: each 32-bit half of a 64-bit
// access is single-copy atomic, and a reader sees either kCarryUnset or the
// whole value, with no fence on either side.
constexpr unsigned kCarryUnset = 0xffffffffu;

__device__ __forceinline__ float2 ld_carry(const float2* p) {
  unsigned x, y;
  asm volatile("ld.relaxed.gpu.global.v2.b32 {%0, %1}, [%2];" : "=r"(x), "=r"(y) : "l"(p) : "memory");
  return make_float2(__uint_as_float(x), __uint_as_float(y));
}

__device__ __forceinline__ bool carry_set(float2 v) {
  return __float_as_uint(v.x) != kCarryUnset && __float_as_uint(v.y) != kCarryUnset;
}

__device__ __forceinline__ void st_carry(float2* p, float2 v) {
  unsigned x = __float_as_uint(v.x), y = __float_as_uint(v.y);
  x = x == kCarryUnset ? 0x7fffffffu : x;
  y = y == kCarryUnset ? 0x7fffffffu : y;
  asm volatile("st.relaxed.gpu.global.v2.b32 [%0], {%1, %2};" ::"l"(p), "r"(x), "r"(y) : "memory");
}

// The same for one 32-bit carry word.
__device__ __forceinline__ float ld_carry1(const float* p) {
  unsigned x;
  asm volatile("ld.relaxed.gpu.global.b32 %0, [%1];" : "=r"(x) : "l"(p) : "memory");
  return __uint_as_float(x);
}

__device__ __forceinline__ bool carry_set1(float v) { return __float_as_uint(v) != kCarryUnset; }

__device__ __forceinline__ void st_carry1(float* p, float v) {
  unsigned x = __float_as_uint(v);
  x = x == kCarryUnset ? 0x7fffffffu : x;
  asm volatile("st.relaxed.gpu.global.b32 [%0], %1;" ::"l"(p), "r"(x) : "memory");
}

// Warp-wide wait on one look-back slot whose carry words are their own flags
// and whose aggregate is announced by `flag`.  Returns kFlagInclusive once
// every lane's carry word holds a value (the value in *v), kFlagAggregate once
// every lane has acquired the aggregate flag, kFlagNone after `limit_ns`.  The
// result is the same in every lane.
__device__ __forceinline__ int wait_carry(const float2* carry, const int* flag, uint64_t limit_ns,
                                          float2* v) {
  const uint64_t t0 = globaltimer_ns();
  unsigned backoff = 32;
  for (;;) {
    *v = ld_carry(carry);
    if (__all_sync(0xffffffffu, carry_set(*v))) return kFlagInclusive;
    if (__all_sync(0xffffffffu, ld_acquire_gpu(flag) == kFlagAggregate)) return kFlagAggregate;
    if (__shfl_sync(0xffffffffu, globaltimer_ns() - t0 > limit_ns, 0)) return kFlagNone;
    __nanosleep(backoff);
    if (backoff < 1024) backoff <<= 1;
  }
}

// The same for a 128-bit carry (four 32-bit words, each single-copy atomic).
__device__ __forceinline__ float4 ld_carry4(const float4* p) {
  unsigned x, y, z, w;
  asm volatile("ld.relaxed.gpu.global.v4.b32 {%0, %1, %2, %3}, [%4];"
               : "=r"(x), "=r"(y), "=r"(z), "=r"(w) : "l"(p) : "memory");
  return make_float4(__uint_as_float(x), __uint_as_float(y), __uint_as_float(z), __uint_as_float(w));
}

__device__ __forceinline__ bool carry_set4(float4 v) {
  return __float_as_uint(v.x) != kCarryUnset && __float_as_uint(v.y) != kCarryUnset &&
         __float_as_uint(v.z) != kCarryUnset && __float_as_uint(v.w) != kCarryUnset;
}

__device__ __forceinline__ void st_carry4(float4* p, float4 v) {
  unsigned x = __float_as_uint(v.x), y = __float_as_uint(v.y), z = __float_as_uint(v.z), w = __float_as_uint(v.w);
  x = x == kCarryUnset ? 0x7fffffffu : x;
  y = y == kCarryUnset ? 0x7fffffffu : y;
  z = z == kCarryUnset ? 0x7fffffffu : z;
  w = w == kCarryUnset ? 0x7fffffffu : w;
  asm volatile("st.relaxed.gpu.global.v4.b32 [%0], {%1, %2, %3, %4};" ::"l"(p), "r"(x), "r"(y), "r"(z), "r"(w)
               : "memory");
}

// wait_carry for 128-bit carries.
__device__ __forceinline__ int wait_carry4(const float4* carry, const int* flag, uint64_t limit_ns,
                                           float4* v) {
  const uint64_t t0 = globaltimer_ns();
  unsigned backoff = 32;
  for (;;) {
    *v = ld_carry4(carry);
    if (__all_sync(0xffffffffu, carry_set4(*v))) return kFlagInclusive;
    if (__all_sync(0xffffffffu, ld_acquire_gpu(flag) == kFlagAggregate)) return kFlagAggregate;
    if (__shfl_sync(0xffffffffu, globaltimer_ns() - t0 > limit_ns, 0)) return kFlagNone;
    __nanosleep(backoff);
    if (backoff < 1024) backoff <<= 1;
  }
}

// ------------------------------------------------------------------ mbarrier + TMA
__device__ __forceinline__ uint32_t smem_u32(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ void mbar_init(uint64_t* bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(bar)), "r"(count) : "memory");
}

__device__ __forceinline__ void fence_mbar_init() {
  asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint64_t* bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_u32(bar)),
               "r"(bytes)
               : "memory");
}

// Arrival without data (completes the phase once every expected byte is in).
__device__ __forceinline__ void mbar_arrive(uint64_t* bar) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_u32(bar)) : "memory");
}

__device__ __forceinline__ bool mbar_try_wait(uint64_t* bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok)
      : "r"(smem_u32(bar)), "r"(parity)
      : "memory");
  return ok != 0;
}

// After a copy wait has been reported as timed out, a CTA waits this much
// longer for the copy before it leaves, so that no copy it requested is still
// writing into its shared memory once another CTA may own that memory.
constexpr unsigned long long kCopyDrainNs = 1ull << 30;

// Wait for phase `parity` of the barrier; gives up after limit_ns (returns false).
__device__ __forceinline__ bool mbar_wait(uint64_t* bar, uint32_t parity, uint64_t limit_ns) {
  if (mbar_try_wait(bar, parity)) return true;
  const uint64_t t0 = globaltimer_ns();
  for (;;) {
    if (mbar_try_wait(bar, parity)) return true;
    if (globaltimer_ns() - t0 > limit_ns) return false;
  }
}

// 2-D tiled TMA load of box (x = inner coordinate, y = row) into shared memory.
__device__ __forceinline__ void tma_load_2d(void* dst, const CUtensorMap* map, int x, int y,
                                            uint64_t* bar) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
      " [%0], [%1, {%2, %3}], [%4];" ::"r"(smem_u32(dst)),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y), "r"(smem_u32(bar))
      : "memory");
}

// 1-D bulk copy global -> shared (both 16-byte aligned, bytes % 16 == 0).
__device__ __forceinline__ void bulk_load_1d(void* dst, const void* src, uint32_t bytes,
                                             uint64_t* bar) {
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::
          "r"(smem_u32(dst)),
      "l"(src), "r"(bytes), "r"(smem_u32(bar))
      : "memory");
}

// ------------------------------------------------------------------ tensor memory (TMEM)
// Tensor memory is 128 lanes x 512 columns of 32-bit words per SM.  A CTA
// allocates columns (a power of two >= 32) with one warp; warp w of the CTA
// can then read and write the lanes 32 (w % 4) .. 32 (w % 4) + 31 of those
// columns, one lane per thread (the .32x32b shape).  Loads and stores are
// asynchronous: tcgen05.wait::ld / wait::st complete them.  The waits below
// name the registers involved as in-out operands, so that the compiler can
// neither read a loaded register before the wait nor reuse a stored one
// before the store has taken it.
__device__ __forceinline__ void tmem_alloc128(uint32_t* dst) {  // warp-collective
  asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], 128;" ::"r"(smem_u32(dst))
               : "memory");
  asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
}

__device__ __forceinline__ void tmem_dealloc128(uint32_t taddr) {  // warp-collective
  asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, 128;" ::"r"(taddr) : "memory");
}

__device__ __forceinline__ void tmem_fence_before_sync() {
  asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
}

__device__ __forceinline__ void tmem_fence_after_sync() {
  asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
}

// 16 consecutive columns of this thread's lane.
__device__ __forceinline__ void tmem_st16(uint32_t taddr, const uint32_t (&v)[16]) {
  asm volatile(
      "tcgen05.st.sync.aligned.32x32b.x16.b32 [%0], {%1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, "
      "%13, %14, %15, %16};" ::"r"(taddr),
      "r"(v[0]), "r"(v[1]), "r"(v[2]), "r"(v[3]), "r"(v[4]), "r"(v[5]), "r"(v[6]), "r"(v[7]), "r"(v[8]),
      "r"(v[9]), "r"(v[10]), "r"(v[11]), "r"(v[12]), "r"(v[13]), "r"(v[14]), "r"(v[15])
      : "memory");
}

__device__ __forceinline__ void tmem_wait_st16(uint32_t (&v)[16]) {
  asm volatile("tcgen05.wait::st.sync.aligned;"
               : "+r"(v[0]), "+r"(v[1]), "+r"(v[2]), "+r"(v[3]), "+r"(v[4]), "+r"(v[5]), "+r"(v[6]),
                 "+r"(v[7]), "+r"(v[8]), "+r"(v[9]), "+r"(v[10]), "+r"(v[11]), "+r"(v[12]), "+r"(v[13]),
                 "+r"(v[14]), "+r"(v[15])
               :
               : "memory");
}

__device__ __forceinline__ void tmem_ld16(uint32_t taddr, uint32_t (&v)[16]) {
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x16.b32 {%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, "
      "%13, %14, %15}, [%16];"
      : "=r"(v[0]), "=r"(v[1]), "=r"(v[2]), "=r"(v[3]), "=r"(v[4]), "=r"(v[5]), "=r"(v[6]), "=r"(v[7]),
        "=r"(v[8]), "=r"(v[9]), "=r"(v[10]), "=r"(v[11]), "=r"(v[12]), "=r"(v[13]), "=r"(v[14]), "=r"(v[15])
      : "r"(taddr)
      : "memory");
}

__device__ __forceinline__ void tmem_wait_ld16(uint32_t (&v)[16]) {
  asm volatile("tcgen05.wait::ld.sync.aligned;"
               : "+r"(v[0]), "+r"(v[1]), "+r"(v[2]), "+r"(v[3]), "+r"(v[4]), "+r"(v[5]), "+r"(v[6]),
                 "+r"(v[7]), "+r"(v[8]), "+r"(v[9]), "+r"(v[10]), "+r"(v[11]), "+r"(v[12]), "+r"(v[13]),
                 "+r"(v[14]), "+r"(v[15])
               :
               : "memory");
}

__device__ __forceinline__ void tmem_alloc256(uint32_t* dst) {  // warp-collective
  asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], 256;" ::"r"(smem_u32(dst))
               : "memory");
  asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
}

__device__ __forceinline__ void tmem_dealloc256(uint32_t taddr) {  // warp-collective
  asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, 256;" ::"r"(taddr) : "memory");
}

// 32 consecutive columns of this thread's lane.
__device__ __forceinline__ void tmem_st32(uint32_t taddr, const uint32_t (&v)[32]) {
  asm volatile(
      "tcgen05.st.sync.aligned.32x32b.x32.b32 [%0], {%1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, "
      "%13, %14, %15, %16, %17, %18, %19, %20, %21, %22, %23, %24, %25, %26, %27, %28, %29, %30, %31, %32};" ::
          "r"(taddr),
      "r"(v[0]), "r"(v[1]), "r"(v[2]), "r"(v[3]), "r"(v[4]), "r"(v[5]), "r"(v[6]), "r"(v[7]), "r"(v[8]),
      "r"(v[9]), "r"(v[10]), "r"(v[11]), "r"(v[12]), "r"(v[13]), "r"(v[14]), "r"(v[15]), "r"(v[16]),
      "r"(v[17]), "r"(v[18]), "r"(v[19]), "r"(v[20]), "r"(v[21]), "r"(v[22]), "r"(v[23]), "r"(v[24]),
      "r"(v[25]), "r"(v[26]), "r"(v[27]), "r"(v[28]), "r"(v[29]), "r"(v[30]), "r"(v[31])
      : "memory");
}

__device__ __forceinline__ void tmem_wait_st32(uint32_t (&v)[32]) {
  asm volatile("tcgen05.wait::st.sync.aligned;"
               : "+r"(v[0]), "+r"(v[1]), "+r"(v[2]), "+r"(v[3]), "+r"(v[4]), "+r"(v[5]), "+r"(v[6]),
                 "+r"(v[7]), "+r"(v[8]), "+r"(v[9]), "+r"(v[10]), "+r"(v[11]), "+r"(v[12]), "+r"(v[13]),
                 "+r"(v[14]), "+r"(v[15]), "+r"(v[16]), "+r"(v[17]), "+r"(v[18]), "+r"(v[19]),
                 "+r"(v[20]), "+r"(v[21]), "+r"(v[22]), "+r"(v[23]), "+r"(v[24]), "+r"(v[25]),
                 "+r"(v[26]), "+r"(v[27]), "+r"(v[28]), "+r"(v[29]), "+r"(v[30]), "+r"(v[31])
               :
               : "memory");
}

// Waits for every earlier tensor-memory store of this thread to complete.
__device__ __forceinline__ void tmem_wait_st() { asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory"); }

__device__ __forceinline__ void tmem_ld32(uint32_t taddr, uint32_t (&v)[32]) {
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x32.b32 {%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, "
      "%13, %14, %15, %16, %17, %18, %19, %20, %21, %22, %23, %24, %25, %26, %27, %28, %29, %30, %31}, [%32];"
      : "=r"(v[0]), "=r"(v[1]), "=r"(v[2]), "=r"(v[3]), "=r"(v[4]), "=r"(v[5]), "=r"(v[6]), "=r"(v[7]),
        "=r"(v[8]), "=r"(v[9]), "=r"(v[10]), "=r"(v[11]), "=r"(v[12]), "=r"(v[13]), "=r"(v[14]), "=r"(v[15]),
        "=r"(v[16]), "=r"(v[17]), "=r"(v[18]), "=r"(v[19]), "=r"(v[20]), "=r"(v[21]), "=r"(v[22]),
        "=r"(v[23]), "=r"(v[24]), "=r"(v[25]), "=r"(v[26]), "=r"(v[27]), "=r"(v[28]), "=r"(v[29]),
        "=r"(v[30]), "=r"(v[31])
      : "r"(taddr)
      : "memory");
}

__device__ __forceinline__ void tmem_wait_ld32(uint32_t (&v)[32]) {
  asm volatile("tcgen05.wait::ld.sync.aligned;"
               : "+r"(v[0]), "+r"(v[1]), "+r"(v[2]), "+r"(v[3]), "+r"(v[4]), "+r"(v[5]), "+r"(v[6]),
                 "+r"(v[7]), "+r"(v[8]), "+r"(v[9]), "+r"(v[10]), "+r"(v[11]), "+r"(v[12]), "+r"(v[13]),
                 "+r"(v[14]), "+r"(v[15]), "+r"(v[16]), "+r"(v[17]), "+r"(v[18]), "+r"(v[19]),
                 "+r"(v[20]), "+r"(v[21]), "+r"(v[22]), "+r"(v[23]), "+r"(v[24]), "+r"(v[25]),
                 "+r"(v[26]), "+r"(v[27]), "+r"(v[28]), "+r"(v[29]), "+r"(v[30]), "+r"(v[31])
               :
               : "memory");
}

// Barrier over `count` threads (a multiple of 32) on named barrier `id` (1..15).
__device__ __forceinline__ void named_barrier(int id, int count) {
  asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(count) : "memory");
}

// 4 consecutive io values as floats (16-byte or 8-byte aligned).
__device__ __forceinline__ float4 ld_io4(const float* p) { return *reinterpret_cast<const float4*>(p); }
__device__ __forceinline__ float4 ld_io4(const __nv_bfloat16* p) {
  const uint2 q = *reinterpret_cast<const uint2*>(p);
  return make_float4(__uint_as_float(q.x << 16), __uint_as_float(q.x & 0xffff0000u),
                     __uint_as_float(q.y << 16), __uint_as_float(q.y & 0xffff0000u));
}

// ------------------------------------------------------------------ pairs of io values
__device__ __forceinline__ float2 ld_io2(const float* p) { return *reinterpret_cast<const float2*>(p); }
__device__ __forceinline__ float2 ld_io2(const __nv_bfloat16* p) {
  return __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(p));
}
__device__ __forceinline__ void st_io2(float* p, float2 v) { *reinterpret_cast<float2*>(p) = v; }
__device__ __forceinline__ void st_io2(__nv_bfloat16* p, float2 v) {
  *reinterpret_cast<__nv_bfloat162*>(p) = __float22bfloat162_rn(v);
}

// ------------------------------------------------------------------ vector loads of N values
// Loads N consecutive io values from shared memory (16-byte aligned) as floats.
template <int N>
__device__ __forceinline__ void lds_row(float (&v)[N], const float* p) {
  static_assert(N % 4 == 0, "N must be a multiple of 4");
#pragma unroll
  for (int i = 0; i < N; i += 4) {
    const float4 q = *reinterpret_cast<const float4*>(p + i);
    v[i] = q.x; v[i + 1] = q.y; v[i + 2] = q.z; v[i + 3] = q.w;
  }
}

template <int N>
__device__ __forceinline__ void lds_row(float (&v)[N], const __nv_bfloat16* p) {
  static_assert(N % 8 == 0, "N must be a multiple of 8 for bf16");
#pragma unroll
  for (int i = 0; i < N; i += 8) {
    const uint4 q = *reinterpret_cast<const uint4*>(p + i);
    const __nv_bfloat162* h = reinterpret_cast<const __nv_bfloat162*>(&q);
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      const float2 f = __bfloat1622float2(h[j]);
      v[i + 2 * j] = f.x;
      v[i + 2 * j + 1] = f.y;
    }
  }
}

// Widens `count` bf16 values staged in shared memory into an fp32 copy (all
// threads of the block take part; the caller synchronises before reading).
// For fp32 I/O the staged values are used as they are.
template <typename T>
__device__ __forceinline__ const float* widen_rows(const T* src, float* dst, int count, int tid,
                                                   int nthreads) {
  if constexpr (sizeof(T) == 4) {
    return reinterpret_cast<const float*>(src);
  } else {
    int done = 0;  // values widened by the 16-byte path
    if (((reinterpret_cast<uintptr_t>(src) | reinterpret_cast<uintptr_t>(dst)) & 15u) == 0) {
      // 8 values per 16-byte load; a bf16 is the upper half of the float it rounds
      const uint4* s8 = reinterpret_cast<const uint4*>(src);
      float4* d4 = reinterpret_cast<float4*>(dst);
      for (int i = tid; i < count / 8; i += nthreads) {
        const uint4 q = s8[i];
        d4[2 * i] = make_float4(__uint_as_float(q.x << 16), __uint_as_float(q.x & 0xffff0000u),
                                __uint_as_float(q.y << 16), __uint_as_float(q.y & 0xffff0000u));
        d4[2 * i + 1] = make_float4(__uint_as_float(q.z << 16), __uint_as_float(q.z & 0xffff0000u),
                                    __uint_as_float(q.w << 16), __uint_as_float(q.w & 0xffff0000u));
      }
      done = count & ~7;
    }
    const __nv_bfloat162* s2 = reinterpret_cast<const __nv_bfloat162*>(src);
    float2* d2 = reinterpret_cast<float2*>(dst);
    for (int i = done / 2 + tid; i < count / 2; i += nthreads) d2[i] = __bfloat1622float2(s2[i]);
    return dst;
  }
}

// ------------------------------------------------------------------ launch shape
// CTAs of `kernel` that fit on one SM at once, from its registers and shared
// memory and the SM's limits.  The kernels that allocate tensor memory use
// this instead of the runtime's occupancy query, which answers 1 for them
// (it cannot know how many columns a CTA takes); their callers cap the count
// by the columns each CTA allocates.
template <typename K>
inline cudaError_t resident_ctas_per_sm(K kernel, int threads, size_t smem, int* per_sm) {
  cudaFuncAttributes fa;
  int dev = 0, regs_sm = 0, smem_sm = 0, reserved = 0, thr_sm = 0, blk_sm = 0;
  cudaError_t e = cudaFuncGetAttributes(&fa, kernel);
  if (e == cudaSuccess) e = cudaGetDevice(&dev);
  if (e == cudaSuccess) e = cudaDeviceGetAttribute(&regs_sm, cudaDevAttrMaxRegistersPerMultiprocessor, dev);
  if (e == cudaSuccess) e = cudaDeviceGetAttribute(&smem_sm, cudaDevAttrMaxSharedMemoryPerMultiprocessor, dev);
  if (e == cudaSuccess) e = cudaDeviceGetAttribute(&reserved, cudaDevAttrReservedSharedMemoryPerBlock, dev);
  if (e == cudaSuccess) e = cudaDeviceGetAttribute(&thr_sm, cudaDevAttrMaxThreadsPerMultiProcessor, dev);
  if (e == cudaSuccess) e = cudaDeviceGetAttribute(&blk_sm, cudaDevAttrMaxBlocksPerMultiprocessor, dev);
  if (e != cudaSuccess) return e;
  const int warps = (threads + 31) / 32;
  const int regs_warp = (fa.numRegs * 32 + 255) / 256 * 256;  // allocated per warp in units of 256
  int n = blk_sm;
  if (regs_warp > 0) n = std::min(n, regs_sm / (regs_warp * warps));
  n = std::min(n, smem_sm / (int)(smem + fa.sharedSizeBytes + (size_t)reserved));
  n = std::min(n, thr_sm / threads);
  *per_sm = n;
  return cudaSuccess;
}

// The current device's SM count (1 when the query fails).
inline int device_sm_count() {
  int dev = 0, n_sm = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || cudaDeviceGetAttribute(&n_sm, cudaDevAttrMultiProcessorCount, dev) !=
                                                 cudaSuccess || n_sm < 1)
    return 1;
  return n_sm;
}

// Blocks of a grid-stride kernel of 256-thread blocks over `work` items: one
// item per thread, at most the 8 blocks per SM that fill the device once.
inline int64_t grid_stride_blocks(int64_t work) {
  const int64_t cap = (int64_t)device_sm_count() * 8;
  const int64_t b = (work + 255) / 256;
  return b < cap ? b : cap;
}

// Grid of a persistent kernel: as many CTAs as fit on the device at once (all
// SMs x resident CTAs per SM), never more than there are work items.  With
// max_per_sm > 0 the count per SM comes from resident_ctas_per_sm and is
// capped at max_per_sm.
template <typename K>
inline cudaError_t persistent_grid(K kernel, int threads, size_t smem, int64_t items, int* grid,
                                   int max_per_sm = 0) {
  int dev = 0, n_sm = 0, per_sm = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e == cudaSuccess) e = cudaDeviceGetAttribute(&n_sm, cudaDevAttrMultiProcessorCount, dev);
  if (e == cudaSuccess)
    e = max_per_sm > 0 ? resident_ctas_per_sm(kernel, threads, smem, &per_sm)
                       : cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, kernel, threads, smem);
  if (e != cudaSuccess) return e;
  if (max_per_sm > 0 && per_sm > max_per_sm) per_sm = max_per_sm;
  const int64_t cap = (int64_t)(per_sm > 0 ? per_sm : 1) * (n_sm > 0 ? n_sm : 1);
  *grid = (int)(items < cap ? items : cap);
  return cudaSuccess;
}

}  // namespace vssm
