// Draft confidence for early stopping ("Adaptive-SpecDecode-Lab" README,
// section "Confidence-guided early stop": after each draft token the drafter
// reads its top-1 probability from the logits it already has and stops
// proposing below a threshold; the low-confidence token is still verified).
//
// conf_i = max_v q_i(v), q_i the draft distribution of row i after the
// repetition penalty (history plus the drafts before row i) and the
// temperature: conf = 1 / sum_v 2^((z'_v - max z') c), c = log2(e)/T.
// k_eff_b = i + 1 for the first row i of request b with conf_i < threshold,
// else K_b.
//
// One CTA per (draft row, 8192-token chunk): 16-byte read-only loads, the
// penalty from a shared-memory bitmap of the chunk's penalised tokens, the
// chunk's exact maximum and the sum of 2^((z' - max) c) over it.  The
// partials go to the workspace; the last CTA of a request (an atomic
// counter) combines them per row and writes conf and k_eff.  B extra CTAs
// report the requests without drafts.  The bound is HBM: every draft logit
// is read once.
#include "common.cuh"
#include "spec_internal.h"

namespace sv {

namespace {

__device__ __forceinline__ void ldg8c(const __nv_bfloat16* p, float* z) {
  uint4 v;
  asm volatile("ld.global.nc.L1::no_allocate.v4.u32 {%0,%1,%2,%3}, [%4];"
               : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
               : "l"(p));
  z[0] = __uint_as_float(v.x << 16); z[1] = __uint_as_float(v.x & 0xffff0000u);
  z[2] = __uint_as_float(v.y << 16); z[3] = __uint_as_float(v.y & 0xffff0000u);
  z[4] = __uint_as_float(v.z << 16); z[5] = __uint_as_float(v.z & 0xffff0000u);
  z[6] = __uint_as_float(v.w << 16); z[7] = __uint_as_float(v.w & 0xffff0000u);
}

__device__ __forceinline__ void ldg8c(const float* p, float* z) {
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

// Request scalars: temperature factor and the validity bits they imply.
__device__ __forceinline__ int conf_params(const ConfParams& P, int b, float& c, float& alpha) {
  const float T_ = P.temperature ? __ldg(P.temperature + b) : 1.f;
  alpha = P.rep_penalty ? __ldg(P.rep_penalty + b) : 1.f;
  int flags = 0;
  if (!(T_ > 0.f) || !(T_ < INFINITY) || !(alpha > 0.f) || !(alpha < INFINITY)) flags |= kStatusBadParam;
  c = __fdiv_rn(1.44269504088896341f, flags ? 1.f : T_);
  return flags;
}

}  // namespace

template <typename T>
__global__ void __launch_bounds__(kGreedyThreads) confidence_kernel(const __grid_constant__ ConfParams P) {
  __shared__ uint32_t bitmap[kGreedyChunk / 32];
  __shared__ float s_red[kGreedyThreads / 32];
  __shared__ int s_flags;
  __shared__ int s_last;
  __shared__ float s_conf[kMaxK];

  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int n_row_ctas = P.total * P.nck;

  if ((int)blockIdx.x >= n_row_ctas) {
    // one CTA per request: requests without drafts, or with an invalid
    // draft count, are finished here (the row CTAs finish the others)
    const int b = blockIdx.x - n_row_ctas;
    const int d0 = __ldg(P.cu_draft + b);
    const int K = __ldg(P.cu_draft + b + 1) - d0;
    const bool bad_k = K < 0 || K > P.max_k || K > kMaxK;
    if (K != 0 && !bad_k) return;
    float c, alpha;
    int flags = conf_params(P, b, c, alpha) | (bad_k ? kStatusBadK : 0);
    if (bad_k)
      for (int r = max(d0, 0) + tid; r < min(d0 + K, P.total); r += kGreedyThreads) P.out_conf[r] = NAN;
    const int h0 = P.cu_hist ? __ldg(P.cu_hist + b) : 0;
    const int h1 = P.cu_hist ? __ldg(P.cu_hist + b + 1) : 0;
    for (int j = h0 + tid; j < h1; j += kGreedyThreads) {
      const int t = __ldg(P.hist + j);
      if (t < 0 || t >= P.V) flags |= kStatusBadToken;
    }
    flags = warp_or(flags);
    if (tid == 0) s_flags = 0;
    __syncthreads();
    if (lane == 0 && flags) atomicOr(&s_flags, flags);
    __syncthreads();
    if (tid == 0) {
      P.out_k_eff[b] = s_flags ? -1 : 0;
      if (P.out_status) P.out_status[b] = s_flags;
    }
    return;
  }

  const int d = blockIdx.x / P.nck;  // draft row
  const int ck = blockIdx.x % P.nck;
  // request of this draft row: the largest b with cu_draft[b] <= d
  int lo = 0, hi = P.B;
  while (hi - lo > 1) {
    const int mid = (lo + hi) >> 1;
    if (__ldg(P.cu_draft + mid) <= d) lo = mid; else hi = mid;
  }
  const int b = lo;
  const int d0 = __ldg(P.cu_draft + b);
  const int K = __ldg(P.cu_draft + b + 1) - d0;
  const int i = d - d0;
  const int c0 = ck * kGreedyChunk;
  const int c1 = min(P.V, c0 + kGreedyChunk);
  float c, alpha;
  int flags = conf_params(P, b, c, alpha);
  if (K < 0 || K > P.max_k || K > kMaxK || i < 0 || i >= K) flags |= kStatusBadK;
  const int h0 = P.cu_hist ? __ldg(P.cu_hist + b) : 0;
  const int h1 = P.cu_hist ? __ldg(P.cu_hist + b + 1) : 0;
  const int npre = (i >= 0 && i < K) ? i : 0;
  const bool pen = !(flags & kStatusBadParam) && alpha != 1.f && (h1 > h0 || npre > 0);

  // the chunk's logits, loaded first so that the loads are in flight while
  // the penalty bitmap is built: thread owns 8-element groups g = tid + 256*j
  const T* rowp = static_cast<const T*>(P.draft) + (size_t)d * P.ld_d;
  constexpr int kGroups = kGreedyChunk / 8 / kGreedyThreads;  // 4
  float z[kGroups][8];
#pragma unroll
  for (int j = 0; j < kGroups; ++j) {
    const int g0 = c0 + 8 * (tid + kGreedyThreads * j);
    if (g0 + 8 <= c1) {
      ldg8c(rowp + g0, z[j]);
    } else {
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

  float mx = -INFINITY;
#pragma unroll
  for (int j = 0; j < kGroups; ++j) {
    const int l0 = 8 * (tid + kGreedyThreads * j);
    const uint32_t m = (pen && c0 + l0 < c1) ? (bitmap[l0 >> 5] >> (l0 & 31)) & 0xFFu : 0u;
#pragma unroll
    for (int e = 0; e < 8; ++e) {
      if (m & (1u << e)) z[j][e] = penalize(z[j][e], alpha);
      if (is_bad_logit(z[j][e])) flags |= kStatusBadLogits;
      mx = fmaxf(mx, z[j][e]);
    }
  }
  mx = warp_max(mx);
  if (lane == 0) s_red[warp] = mx;
  __syncthreads();
  mx = s_red[0];
  for (int w = 1; w < kGreedyThreads / 32; ++w) mx = fmaxf(mx, s_red[w]);
  __syncthreads();
  // sum of 2^((z' - mx) c) over the chunk (0 when the chunk is all -inf)
  float s = 0.f;
  if (mx > -INFINITY && mx < INFINITY) {
    const float cm = mx * c;
#pragma unroll
    for (int j = 0; j < kGroups; ++j)
#pragma unroll
      for (int e = 0; e < 8; ++e) s += ex2(fmaf(z[j][e], c, -cm));
  }
  s = warp_sum(s);
  flags = warp_or(flags);
  if (lane == 0) {
    s_red[warp] = s;
    if (flags) atomicOr(&s_flags, flags);
  }
  __syncthreads();
  if (tid == 0) {
    float st = 0.f;
    for (int w = 0; w < kGreedyThreads / 32; ++w) st += s_red[w];
    ConfPartial cp;
    cp.m = mx;
    cp.s = st;
    cp.flags = s_flags;
    cp.pad = 0;
    P.partials[(size_t)d * P.nck + ck] = cp;
    __threadfence();
    const int target = kread * P.nck;
    const int old = atomicAdd(P.counters + b, 1);
    s_last = (K == kread) && (old == target - 1);
  }
  __syncthreads();
  if (!s_last) return;

  // ---- last CTA of the request: per row, combine the chunks; then k_eff
  __threadfence();
  for (int r = warp; r < K; r += kGreedyThreads / 32) {
    const ConfPartial* pr = P.partials + (size_t)(d0 + r) * P.nck;
    float m = -INFINITY, sum = 0.f;
    int f = 0;
    for (int k = lane; k < P.nck; k += 32) {
      const float mk = __ldcg(&pr[k].m);
      f |= __ldcg(&pr[k].flags);
      m = fmaxf(m, mk);
    }
    m = warp_max(m);
    if (m > -INFINITY && m < INFINITY) {
      const float cm = m * c;
      for (int k = lane; k < P.nck; k += 32) {
        const float mk = __ldcg(&pr[k].m), sk = __ldcg(&pr[k].s);
        if (mk > -INFINITY) sum += sk * ex2(fmaf(mk, c, -cm));
      }
    }
    sum = warp_sum(sum);
    f = warp_or(f);
    if (!(sum > 0.f) || !(sum < INFINITY)) f |= kStatusBadLogits;
    if (lane == 0) {
      s_conf[r] = __fdiv_rn(1.f, sum);
      if (f) atomicOr(&s_flags, f);
    }
  }
  __syncthreads();
  if (tid == 0) {
    const int st = s_flags;
    int k_eff = K;
    for (int r = 0; r < K; ++r)
      if (s_conf[r] < P.threshold) {
        k_eff = r + 1;
        break;
      }
    P.out_k_eff[b] = st ? -1 : k_eff;
    if (P.out_status) P.out_status[b] = st;
  }
  for (int r = tid; r < K; r += kGreedyThreads) P.out_conf[d0 + r] = s_flags ? NAN : s_conf[r];
}

int launch_confidence(const ConfParams& P, bool bf16, cudaStream_t stream) {
  const long long grid = (long long)P.total * P.nck + P.B;
  if (grid <= 0) return 0;
  if (grid > 0x7fffffffLL) return -2;
  if (bf16) confidence_kernel<__nv_bfloat16><<<(unsigned)grid, kGreedyThreads, 0, stream>>>(P);
  else confidence_kernel<float><<<(unsigned)grid, kGreedyThreads, 0, stream>>>(P);
  return cudaGetLastError() == cudaSuccess ? 0 : -7;
}

}  // namespace sv
