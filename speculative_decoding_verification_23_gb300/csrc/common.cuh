// Device helpers shared by the verification kernels: inline PTX for
// mbarriers, 1-D TMA bulk copies, cluster (DSMEM) access, and warp
// reductions.  Every wait here is bounded (a cycle-count limit):
// a wait that runs out returns false and the caller records an error status
// instead of spinning forever.
#pragma once

#include <cstdint>
#include <cuda_runtime.h>
#include <cuda_bf16.h>

#include "spec_internal.h"   // kTagShift

namespace sv {

// Per-request status bits (the same values as spec_verify.h).
constexpr int kStatusBadToken = 1;
constexpr int kStatusBadParam = 2;
constexpr int kStatusBadLogits = 4;
constexpr int kStatusBadK = 8;
constexpr int kStatusTimeout = 16;

constexpr int kMaxK = 32;

__device__ __forceinline__ uint32_t smem_u32(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

// ---------------------------------------------------------------- mbarrier
__device__ __forceinline__ void mbar_init(uint64_t* bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(bar)), "r"(count) : "memory");
}

__device__ __forceinline__ void fence_mbar_init() {
  asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}

__device__ __forceinline__ void mbar_arrive(uint64_t* bar) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_u32(bar)) : "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint64_t* bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_u32(bar)), "r"(bytes)
               : "memory");
}

// Arrive (release, cluster scope) on the barrier at the same shared-memory
// offset in CTA `rank` of this cluster.
__device__ __forceinline__ void mbar_arrive_remote(uint64_t* bar, uint32_t rank) {
  uint32_t remote;
  asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(remote) : "r"(smem_u32(bar)), "r"(rank));
  asm volatile("mbarrier.arrive.release.cluster.shared::cluster.b64 _, [%0];" ::"r"(remote) : "memory");
}

__device__ __forceinline__ bool mbar_test(uint64_t* bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{ .reg .pred p; mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2; selp.u32 %0, 1, 0, p; }"
      : "=r"(ok)
      : "r"(smem_u32(bar)), "r"(parity)
      : "memory");
  return ok != 0;
}

__device__ __forceinline__ bool mbar_test_cluster(uint64_t* bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{ .reg .pred p; mbarrier.try_wait.parity.acquire.cluster.shared::cta.b64 p, [%1], %2; selp.u32 %0, 1, 0, p; }"
      : "=r"(ok)
      : "r"(smem_u32(bar)), "r"(parity)
      : "memory");
  return ok != 0;
}

// Bounded waits: true once the phase with `parity` has completed, false if
// the limit (in SM clock cycles, a few seconds at any clock) ran out first.
constexpr long long kWaitLimitCycles = 4000000000ll;

__device__ __forceinline__ bool mbar_wait(uint64_t* bar, uint32_t parity) {
  if (mbar_test(bar, parity)) return true;
  const long long t0 = clock64();
  for (;;) {
    if (mbar_test(bar, parity)) return true;
    if (clock64() - t0 > kWaitLimitCycles) return false;
  }
}

__device__ __forceinline__ bool mbar_wait_cluster(uint64_t* bar, uint32_t parity) {
  if (mbar_test_cluster(bar, parity)) return true;
  const long long t0 = clock64();
  for (;;) {
    if (mbar_test_cluster(bar, parity)) return true;
    if (clock64() - t0 > kWaitLimitCycles) return false;
  }
}

// The fills a producer put into a ring of at most 32 slots (bit s: slot s
// filled at least once; parity bit s: the phase of its last fill).  A
// producer whose wait ran out stops issuing and, before its CTA may exit,
// waits (bounded) for the copies it already started to land.
struct RingFills {
  uint32_t filled = 0, par = 0;
  __device__ __forceinline__ void note(uint32_t slot, uint32_t phase) {
    filled |= 1u << slot;
    par = (par & ~(1u << slot)) | ((phase & 1u) << slot);
  }
  __device__ __forceinline__ void drain(uint64_t* full, int nslots) const {
    for (int s = 0; s < nslots; ++s)
      if ((filled >> s) & 1u) (void)mbar_wait(&full[s], (par >> s) & 1u);
  }
};

// ------------------------------------------- arrival counters, call-tagged
// A request's arrival counter is one 64-bit word: the calling launch's tag
// in the high 40 bits, that launch's arrivals in the low 24.  A word with
// any other tag (an earlier call's, or whatever the memory held) counts as
// no arrival yet, so the counters need no initial value and no clearing
// launch between calls.  Returns the arrivals of this launch before this
// one.
//
// An arrival that reads another tag first resets the word to (tag, 0) with
// one compare-and-swap against the value it read; then every arrival adds
// one.  Only this launch's arrivals write the word while it runs, and each
// writes it with this launch's tag, so a failed reset means the word already
// carries the tag, and no add lands on a stale word.  No retry loop: under
// many simultaneous arrivals a loop of exchanges costs quadratically many
// atomics at one address.
__device__ __forceinline__ int tagged_arrive(unsigned long long* ctr, unsigned long long tag) {
  const unsigned long long v = *reinterpret_cast<volatile unsigned long long*>(ctr);
  if ((v >> kTagShift) != tag) atomicCAS(ctr, v, tag << kTagShift);
  const unsigned long long old = atomicAdd(ctr, 1ull);
  return (int)(old & ((1ull << kTagShift) - 1ull));
}

// Position in the ring: slot index and the parity of its current use.
struct RingCursor {
  uint32_t slot = 0, phase = 0;
  __device__ __forceinline__ void advance(int nslots) {
    if (++slot == (uint32_t)nslots) {
      slot = 0;
      phase ^= 1u;
    }
  }
};

// ------------------------------------------------------ TMA bulk (1-D) copy
// Global -> this CTA's shared memory, completion signalled on `bar` as
// transaction bytes.  dst, src and bytes must be multiples of 16.
__device__ __forceinline__ void bulk_g2s(void* dst, const void* src, uint32_t bytes, uint64_t* bar,
                                         uint64_t policy) {
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes.L2::cache_hint [%0], [%1], %2, [%3], %4;" ::"r"(
          smem_u32(dst)),
      "l"(src), "r"(bytes), "r"(smem_u32(bar)), "l"(policy)
      : "memory");
}

__device__ __forceinline__ uint64_t l2_policy_evict_first() {
  uint64_t p;
  asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(p));
  return p;
}

__device__ __forceinline__ uint64_t l2_policy_evict_last() {
  uint64_t p;
  asm volatile("createpolicy.fractional.L2::evict_last.b64 %0, 1.0;" : "=l"(p));
  return p;
}

// ------------------------------------------------------------- clusters
__device__ __forceinline__ uint32_t cluster_rank() {
  uint32_t r;
  asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
  return r;
}

__device__ __forceinline__ uint32_t cluster_size() {
  uint32_t r;
  asm volatile("mov.u32 %0, %%cluster_nctarank;" : "=r"(r));
  return r;
}

__device__ __forceinline__ void cluster_sync_all() {
  asm volatile("barrier.cluster.arrive.release.aligned;\n\tbarrier.cluster.wait.acquire.aligned;" ::: "memory");
}

__device__ __forceinline__ uint32_t map_rank(const void* p, uint32_t rank) {
  uint32_t r;
  asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(r) : "r"(smem_u32(p)), "r"(rank));
  return r;
}

__device__ __forceinline__ void st_remote_f64(uint32_t addr, double v) {
  asm volatile("st.shared::cluster.f64 [%0], %1;" ::"r"(addr), "d"(v) : "memory");
}

__device__ __forceinline__ double ld_remote_f64(uint32_t addr) {
  double v;
  asm volatile("ld.shared::cluster.f64 %0, [%1];" : "=d"(v) : "r"(addr) : "memory");
  return v;
}

__device__ __forceinline__ float ld_remote_f32(uint32_t addr) {
  float v;
  asm volatile("ld.shared::cluster.f32 %0, [%1];" : "=f"(v) : "r"(addr) : "memory");
  return v;
}

__device__ __forceinline__ void fence_acq_rel_cluster() {
  asm volatile("fence.acq_rel.cluster;" ::: "memory");
}

// Named barrier over the first `nthreads` threads (warps 0..nthreads/32-1).
__device__ __forceinline__ void named_sync(int id, int nthreads) {
  asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(nthreads) : "memory");
}

// ------------------------------------------------------------- numerics
__device__ __forceinline__ float ex2(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

__device__ __forceinline__ float warp_sum(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
  return v;
}

__device__ __forceinline__ double warp_sum_d(double v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
  return v;
}

__device__ __forceinline__ float warp_max(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, o));
  return v;
}

__device__ __forceinline__ int warp_or(int v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v |= __shfl_xor_sync(0xffffffffu, v, o);
  return v;
}

// Inclusive prefix sum across the warp (lane order).
__device__ __forceinline__ float warp_incl_scan(float v, int lane) {
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    float t = __shfl_up_sync(0xffffffffu, v, o);
    if (lane >= o) v += t;
  }
  return v;
}

__device__ __forceinline__ double warp_incl_scan_d(double v, int lane) {
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    double t = __shfl_up_sync(0xffffffffu, v, o);
    if (lane >= o) v += t;
  }
  return v;
}

// Repetition penalty of one logit (CTRL convention), correctly rounded fp32.
__device__ __forceinline__ float penalize(float z, float alpha) {
  return z > 0.f ? __fdiv_rn(z, alpha) : __fmul_rn(z, alpha);
}

// 4 consecutive logits from shared memory, converted to fp32.
__device__ __forceinline__ void load4(const float* p, float* z) {
  float4 v = *reinterpret_cast<const float4*>(p);
  z[0] = v.x; z[1] = v.y; z[2] = v.z; z[3] = v.w;
}

__device__ __forceinline__ void load4(const __nv_bfloat16* p, float* z) {
  uint2 v = *reinterpret_cast<const uint2*>(p);
  z[0] = __uint_as_float(v.x << 16);
  z[1] = __uint_as_float(v.x & 0xffff0000u);
  z[2] = __uint_as_float(v.y << 16);
  z[3] = __uint_as_float(v.y & 0xffff0000u);
}

template <typename T>
__device__ __forceinline__ float to_f32(T v);
template <>
__device__ __forceinline__ float to_f32<float>(float v) { return v; }
template <>
__device__ __forceinline__ float to_f32<__nv_bfloat16>(__nv_bfloat16 v) { return __bfloat162float(v); }

__device__ __forceinline__ bool is_bad_logit(float z) {  // NaN or +inf
  return !(z < __int_as_float(0x7f800000));
}

}  // namespace sv
