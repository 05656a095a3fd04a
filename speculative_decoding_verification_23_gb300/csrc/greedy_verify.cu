// Greedy longest-prefix verification for GB300 (sm_103a)
// ("Adaptive-SpecDecode-Lab" README, section "实现": the target verifies
// [last committed, d1..dK] in one forward; the longest prefix of drafts that
// equal the target's argmax is accepted; the first mismatch is replaced by
// the target's argmax (correction), and a fully matched draft earns the
// argmax of the last row (bonus)).
//
// One CTA per (target row, 8192-token chunk): a single pass over the chunk
// with 16-byte read-only loads, the repetition penalty applied through a
// shared-memory bitmap of the row's penalised tokens, and a (value, lowest
// index) argmax.  The partial argmaxes go to the workspace; the last CTA of a
// request (an atomic counter) reduces them per row and emits the tokens.
// The argmax is exact: fp32 comparisons of the penalised logits, lowest id on
// ties, so the result is bit-identical to any correct argmax.
#include "common.cuh"
#include "spec_internal.h"

namespace sv {

namespace {

__device__ __forceinline__ bool better(float v, int i, float bv, int bi) {
  return v > bv || (v == bv && i < bi);
}

// 8 consecutive logits from global memory (16 B for bf16, 32 B for fp32).
__device__ __forceinline__ void ldg8(const __nv_bfloat16* p, float* z) {
  uint4 v;
  asm volatile("ld.global.nc.L1::no_allocate.v4.u32 {%0,%1,%2,%3}, [%4];"
               : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
               : "l"(p));
  z[0] = __uint_as_float(v.x << 16); z[1] = __uint_as_float(v.x & 0xffff0000u);
  z[2] = __uint_as_float(v.y << 16); z[3] = __uint_as_float(v.y & 0xffff0000u);
  z[4] = __uint_as_float(v.z << 16); z[5] = __uint_as_float(v.z & 0xffff0000u);
  z[6] = __uint_as_float(v.w << 16); z[7] = __uint_as_float(v.w & 0xffff0000u);
}

__device__ __forceinline__ void ldg8(const float* p, float* z) {
  float4 a, b;
  asm volatile("ld.global.nc.L1::no_allocate.v4.f32 {%0,%1,%2,%3}, [%4];"
               : "=f"(a.x), "=f"(a.y), "=f"(a.z), "=f"(a.w)
               : "l"(p));
  asm volatile("ld.global.nc.L1::no_allocate.v4.f32 {%0,%1,%2,%3}, [%4];"
               : "=f"(b.x), "=f"(b.y), "=f"(b.z), "=f"(b.w)
               : "l"(p + 4));
  z[0] = a.x; z[1] = a.y; z[2] = a.z; z[3] = a.w;
  z[4] = b.x; z[5] = b.y; z[6] = b.z; z[7] = b.w;
}

}  // namespace

template <typename T>
__global__ void __launch_bounds__(kGreedyThreads) greedy_verify_kernel(const __grid_constant__ GreedyParams P) {
  __shared__ uint32_t bitmap[kGreedyChunk / 32];
  __shared__ float s_val[kGreedyThreads / 32];
  __shared__ int s_idx[kGreedyThreads / 32];
  __shared__ int s_flags;
  __shared__ int s_last;

  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int row = blockIdx.x / P.nck;
  const int ck = blockIdx.x % P.nck;
  // request of this target row: largest b with off_b = cu_draft[b] + b <= row
  int lo = 0, hi = P.B;
  while (hi - lo > 1) {
    const int mid = (lo + hi) >> 1;
    if (__ldg(P.cu_draft + mid) + mid <= row) lo = mid; else hi = mid;
  }
  const int b = lo;
  const int d0 = __ldg(P.cu_draft + b);
  const int K = __ldg(P.cu_draft + b + 1) - d0;
  const int i = row - (d0 + b);
  const int c0 = ck * kGreedyChunk;
  const int c1 = min(P.V, c0 + kGreedyChunk);
  const float alpha = P.rep_penalty ? __ldg(P.rep_penalty + b) : 1.f;
  int flags = 0;
  if (K < 0 || K > P.max_k || i < 0 || i > K) flags |= kStatusBadK;
  if (!(alpha > 0.f) || !(alpha < INFINITY)) flags |= kStatusBadParam;
  const int h0 = P.cu_hist ? __ldg(P.cu_hist + b) : 0;
  const int h1 = P.cu_hist ? __ldg(P.cu_hist + b + 1) : 0;
  const int npre = (i >= 0 && i <= K) ? i : 0;
  const bool pen = !(flags & kStatusBadParam) && alpha != 1.f && (h1 > h0 || npre > 0);

  // the chunk's logits, loaded first so that the loads are in flight while
  // the penalty bitmap is built: thread owns 8-element groups g = tid + 256*j
  const T* rowp = static_cast<const T*>(P.target) + (size_t)row * P.ld_t;
  float best = -INFINITY;
  int bidx = 0x7fffffff;
  constexpr int kGroups = kGreedyChunk / 8 / kGreedyThreads;  // 4
  float z[kGroups][8];
#pragma unroll
  for (int j = 0; j < kGroups; ++j) {
    const int g0 = c0 + 8 * (tid + kGreedyThreads * j);
    if (g0 + 8 <= c1) {
      ldg8(rowp + g0, z[j]);
    } else if (g0 < c1) {  // ragged end of the row: no read past V
#pragma unroll
      for (int e = 0; e < 8; ++e) z[j][e] = g0 + e < c1 ? to_f32<T>(rowp[g0 + e]) : -INFINITY;
    }
  }
  if (tid == 0) s_flags = 0;
  for (int w = tid; w < kGreedyChunk / 32; w += kGreedyThreads) bitmap[w] = 0u;
  __syncthreads();
  for (int j = h0 + tid; j < h1; j += kGreedyThreads) {
    const int t = __ldg(P.hist + j);
    if (t < 0 || t >= P.V) flags |= kStatusBadToken;
    else if (pen && t >= c0 && t < c1) atomicOr(&bitmap[(t - c0) >> 5], 1u << ((t - c0) & 31));
  }
  const int kread = (K >= 0 && K <= P.max_k && K <= kMaxK) ? K : 0;
  for (int j = tid; j < kread; j += kGreedyThreads) {
    const int t = __ldg(P.draft_tokens + d0 + j);
    if (t < 0 || t >= P.V) flags |= kStatusBadToken;
    else if (pen && j < npre && t >= c0 && t < c1) atomicOr(&bitmap[(t - c0) >> 5], 1u << ((t - c0) & 31));
  }
  __syncthreads();

#pragma unroll
  for (int j = 0; j < kGroups; ++j) {
    const int l0 = 8 * (tid + kGreedyThreads * j);  // offset within the chunk
    const int g0 = c0 + l0;
    if (g0 >= c1) continue;
    uint32_t m = pen ? (bitmap[l0 >> 5] >> (l0 & 31)) & 0xFFu : 0u;
#pragma unroll
    for (int e = 0; e < 8; ++e) {
      float v = z[j][e];
      if (g0 + e >= c1) continue;
      if (m & (1u << e)) v = penalize(v, alpha);
      if (is_bad_logit(v)) flags |= kStatusBadLogits;
      if (better(v, g0 + e, best, bidx)) { best = v; bidx = g0 + e; }
    }
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
    const float ov = __shfl_xor_sync(0xffffffffu, best, o);
    const int oi = __shfl_xor_sync(0xffffffffu, bidx, o);
    if (better(ov, oi, best, bidx)) { best = ov; bidx = oi; }
  }
  flags = warp_or(flags);
  if (lane == 0) {
    s_val[warp] = best;
    s_idx[warp] = bidx;
    if (flags) atomicOr(&s_flags, flags);
  }
  __syncthreads();
  if (tid == 0) {
    float bv = s_val[0];
    int bi = s_idx[0];
    for (int w = 1; w < kGreedyThreads / 32; ++w)
      if (better(s_val[w], s_idx[w], bv, bi)) { bv = s_val[w]; bi = s_idx[w]; }
    GreedyPartial gp;
    gp.val = bv; gp.idx = bi; gp.flags = s_flags; gp.pad = 0;
    P.partials[(size_t)row * P.nck + ck] = gp;
    __threadfence();
    const int target = (K + 1) * P.nck;
    const int old = tagged_arrive(P.counters + b, P.tag);
    s_last = K >= 0 && old == target - 1;
  }
  __syncthreads();
  if (!s_last) return;
  __threadfence();
  // ---- finalize request b: argmax per row, then the prefix match
  __shared__ int g_arg[kMaxK + 1];
  __shared__ int g_flags;
  const bool k_ok = K <= P.max_k && K <= kMaxK;
  if (tid == 0) g_flags = k_ok ? 0 : kStatusBadK;
  __syncthreads();
  for (int r = warp; k_ok && r <= K; r += kGreedyThreads / 32) {
    float bv = -INFINITY;
    int bi = 0x7fffffff, fl = 0;
    const GreedyPartial* pp = P.partials + (size_t)(d0 + b + r) * P.nck;
    for (int j = lane; j < P.nck; j += 32) {
      const float v = __ldcg(&pp[j].val);
      const int ix = __ldcg(&pp[j].idx);
      fl |= __ldcg(&pp[j].flags);
      if (better(v, ix, bv, bi)) { bv = v; bi = ix; }
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
      const float ov = __shfl_xor_sync(0xffffffffu, bv, o);
      const int oi = __shfl_xor_sync(0xffffffffu, bi, o);
      if (better(ov, oi, bv, bi)) { bv = ov; bi = oi; }
    }
    fl = warp_or(fl);
    if (lane == 0) {
      g_arg[r] = bi;
      if (fl) atomicOr(&g_flags, fl);
    }
  }
  __syncthreads();
  if (warp == 0) {
    const int st = g_flags;
    const int off = d0 + b;
    const int xl = (!st && lane < K) ? __ldg(P.draft_tokens + d0 + lane) : -1;
    const unsigned mism = __ballot_sync(0xffffffffu, !st && lane < K && g_arg[lane] != xl);
    const int j = mism ? __ffs(mism) - 1 : K;
    for (int s = lane; s <= K; s += 32) {
      int tok = -1;
      if (!st) tok = s < j ? __ldg(P.draft_tokens + d0 + s) : (s == j ? g_arg[j] : -1);
      P.out_tokens[off + s] = tok;
    }
    if (lane == 0) {
      P.out_accepted[b] = st ? -1 : j;
      if (P.out_status) P.out_status[b] = st;
    }
  }
}

template __global__ void greedy_verify_kernel<float>(const __grid_constant__ GreedyParams);
template __global__ void greedy_verify_kernel<__nv_bfloat16>(const __grid_constant__ GreedyParams);

}  // namespace sv

namespace sv {

// Host launcher: one CTA per (target row, chunk).
int launch_greedy_verify(const GreedyParams& P, bool bf16, cudaStream_t stream) {
  const long long rows = (long long)P.total + P.B;
  const long long grid = rows * P.nck;
  if (grid <= 0) return 0;
  if (grid > 0x7fffffffLL) return -1;
  if (bf16)
    greedy_verify_kernel<__nv_bfloat16><<<(unsigned)grid, kGreedyThreads, 0, stream>>>(P);
  else
    greedy_verify_kernel<float><<<(unsigned)grid, kGreedyThreads, 0, stream>>>(P);
  return cudaGetLastError() == cudaSuccess ? 0 : -1;
}

}  // namespace sv
