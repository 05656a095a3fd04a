// Device helpers of the streaming kernels (pipe_verify.cu, and the draft
// confidence kernel in confidence.cu): a row staged in shared memory as
// 2 KB warp segments, the penalised positions of a segment, and the hot
// loops of pass 1 (softmax statistics: a running reference and the sum of
// 2^(z'c - ref)) and pass 2 (the residual mass of max(p - q, 0)), with
// their online combines.
#pragma once

#include <cstdint>
#include <cuda_runtime.h>
#include <cuda_bf16.h>

#include "common.cuh"

namespace sv {

namespace {

constexpr float kLim = 18446744073709551616.0f;  // 2^64

__device__ __forceinline__ void fence_proxy_async_smem() {
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

__device__ __forceinline__ int warp_incl_scan_i(int v, int lane) {
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const int t = __shfl_up_sync(0xffffffffu, v, o);
    if (lane >= o) v += t;
  }
  return v;
}

// 16 bytes of a staged row as fp32: 8 bf16 or 4 fp32 values, in token order.
__device__ __forceinline__ void cvt16(const uint4& v, float (&z)[8]) {
  z[0] = __uint_as_float(v.x << 16);
  z[1] = __uint_as_float(v.x & 0xffff0000u);
  z[2] = __uint_as_float(v.y << 16);
  z[3] = __uint_as_float(v.y & 0xffff0000u);
  z[4] = __uint_as_float(v.z << 16);
  z[5] = __uint_as_float(v.z & 0xffff0000u);
  z[6] = __uint_as_float(v.w << 16);
  z[7] = __uint_as_float(v.w & 0xffff0000u);
}
__device__ __forceinline__ void cvt16(const uint4& v, float (&z)[4]) {
  z[0] = __uint_as_float(v.x);
  z[1] = __uint_as_float(v.y);
  z[2] = __uint_as_float(v.z);
  z[3] = __uint_as_float(v.w);
}

template <typename T>
struct Vec {
  static constexpr int N = 16 / (int)sizeof(T);  // values per 16-byte vector
};

template <typename T>
__device__ __forceinline__ T neg_inf();
template <>
__device__ __forceinline__ float neg_inf<float>() { return -INFINITY; }
template <>
__device__ __forceinline__ __nv_bfloat16 neg_inf<__nv_bfloat16>() { return __ushort_as_bfloat16((unsigned short)0xFF80u); }

// A warp segment is 2048 bytes of one row: lane l holds the 16-byte
// vectors j*32 + l (j = 0..3), i.e. tokens (j*32 + l)*N + e of the segment.
__device__ __forceinline__ void lds_seg(const unsigned char* seg, int lane, uint4 (&v)[4]) {
#pragma unroll
  for (int j = 0; j < 4; ++j) v[j] = *reinterpret_cast<const uint4*>(seg + (j * 32 + lane) * 16);
}

template <int N>
__device__ __forceinline__ void mask_tail(float (&z)[4][N], int lane, int nvalid) {
#pragma unroll
  for (int j = 0; j < 4; ++j)
#pragma unroll
    for (int e = 0; e < N; ++e)
      if ((j * 32 + lane) * N + e >= nvalid) z[j][e] = -INFINITY;
}

// Calls f(o) for every penalised position o of segment s (offset within
// the segment): lane l takes bitmap word s*wps + l (l < wps), its set bits
// one by one.  Returns whether the segment has any (warp-uniform).
template <typename F>
__device__ __forceinline__ bool for_penalised(const uint32_t* bm, int s, int wps, int lane, F&& f) {
  uint32_t w = lane < wps ? bm[s * wps + lane] : 0u;
  if (!__any_sync(0xffffffffu, w != 0u)) return false;
  while (w) {
    const int bit = __ffs(w) - 1;
    w &= w - 1;
    f(32 * lane + bit);
  }
  return true;
}

// Pass-1 statistics of one row segment for one lane: the running reference
// `ref` (units of z'c) only moves up, when a segment's sum of 2^(z'c - ref)
// would exceed 2^64 (and on the first segment with a finite value); `run`
// accumulates the sums.  NaN or +inf logits make `run` NaN, which the
// combine reports as invalid logits.
template <int N>
__device__ __forceinline__ void stats_row(const float (&z)[4][N], float c, float& ref, float& run) {
  const float2 c2 = make_float2(c, c);
  float2 nr = make_float2(-ref, -ref);
  float2 acc = make_float2(0.f, 0.f);
#pragma unroll
  for (int j = 0; j < 4; ++j)
#pragma unroll
    for (int e = 0; e < N; e += 2) {
      const float2 y = __ffma2_rn(make_float2(z[j][e], z[j][e + 1]), c2, nr);
      acc = __fadd2_rn(acc, make_float2(ex2(y.x), ex2(y.y)));
    }
  float s = acc.x + acc.y;
  if (!(s <= kLim)) {
    float mx = -INFINITY;
#pragma unroll
    for (int j = 0; j < 4; ++j)
#pragma unroll
      for (int e = 0; e < N; ++e) mx = fmaxf(mx, z[j][e]);
    if (mx > -INFINITY) {
      const float nref = mx * c;
      if (nref > ref) {
        run *= ex2(ref - nref);
        ref = nref;
      }
      nr = make_float2(-ref, -ref);
      acc = make_float2(0.f, 0.f);
#pragma unroll
      for (int j = 0; j < 4; ++j)
#pragma unroll
        for (int e = 0; e < N; e += 2) {
          const float2 y = __ffma2_rn(make_float2(z[j][e], z[j][e + 1]), c2, nr);
          acc = __fadd2_rn(acc, make_float2(ex2(y.x), ex2(y.y)));
        }
      s = acc.x + acc.y;
    } else if (mx == -INFINITY) {
      s = 0.f;  // nothing finite in this segment while the reference is unset
    }
  }
  run += s;
}

// Group A: statistics of NR rows of one warp segment of a ring slot.
template <typename T, int NR>
__device__ __forceinline__ void seg_stats(const unsigned char* seg, int row_bytes, int lane, int nvalid, float c,
                                          float (&ref)[2], float (&run)[2]) {
  constexpr int N = Vec<T>::N;
  uint4 v[NR][4];
#pragma unroll
  for (int r = 0; r < NR; ++r) lds_seg(seg + r * row_bytes, lane, v[r]);
#pragma unroll
  for (int r = 0; r < NR; ++r) {
    float z[4][N];
#pragma unroll
    for (int j = 0; j < 4; ++j) cvt16(v[r][j], z[j]);
    if (nvalid < 128 * N) mask_tail<N>(z, lane, nvalid);
    stats_row<N>(z, c, ref[r], run[r]);
  }
}

// Group B: this lane's share of one segment's residual mass sum max(p-q, 0)
// (BONUS: of p), p = 2^(z'c - Mp) / Sp and q = 2^(z'c - Mq) / Sq.
template <typename T, bool BONUS>
__device__ __forceinline__ float seg_resid(const unsigned char* seg, int row_bytes, int lane, int nvalid, float c,
                                           float Mp, float Mq, float ip, float iq) {
  constexpr int N = Vec<T>::N;
  uint4 vp[4], vq[4];
  lds_seg(seg, lane, vp);
  if (!BONUS) lds_seg(seg + row_bytes, lane, vq);
  float zp[4][N], zq[4][N];
#pragma unroll
  for (int j = 0; j < 4; ++j) {
    cvt16(vp[j], zp[j]);
    if (!BONUS) cvt16(vq[j], zq[j]);
  }
  if (nvalid < 128 * N) {
    mask_tail<N>(zp, lane, nvalid);
    if (!BONUS) mask_tail<N>(zq, lane, nvalid);
  }
  const float2 c2 = make_float2(c, c), np2 = make_float2(-Mp, -Mp), nq2 = make_float2(-Mq, -Mq);
  const float2 ip2 = make_float2(ip, ip), iq2 = make_float2(iq, iq), m1 = make_float2(-1.f, -1.f);
  float2 acc = make_float2(0.f, 0.f);
#pragma unroll
  for (int j = 0; j < 4; ++j)
#pragma unroll
    for (int e = 0; e < N; e += 2) {
      const float2 yp = __ffma2_rn(make_float2(zp[j][e], zp[j][e + 1]), c2, np2);
      const float2 p = __fmul2_rn(make_float2(ex2(yp.x), ex2(yp.y)), ip2);
      if (BONUS) {
        acc = __fadd2_rn(acc, p);
      } else {
        const float2 yq = __ffma2_rn(make_float2(zq[j][e], zq[j][e + 1]), c2, nq2);
        const float2 q = __fmul2_rn(make_float2(ex2(yq.x), ex2(yq.y)), iq2);
        const float2 d = __ffma2_rn(q, m1, p);
        acc = __fadd2_rn(acc, make_float2(fmaxf(d.x, 0.f), fmaxf(d.y, 0.f)));
      }
    }
  return acc.x + acc.y;
}

// The same probability and residual for one token (bit-identical to the
// packed arithmetic above, component by component).
__device__ __forceinline__ float prob_of(float z, float c, float M, float inv) {
  return __fmul_rn(ex2(fmaf(z, c, -M)), inv);
}
__device__ __forceinline__ float resid_of(float p, float q) { return fmaxf(fmaf(q, -1.f, p), 0.f); }

// (reference, sum) of a warp from its lanes'.
__device__ __forceinline__ float2 warp_combine(float ref, float s) {
  const float M = warp_max(ref);
  const float t = (ref > -INFINITY) ? s * ex2(ref - M) : s;
  return make_float2(M, warp_sum(t));
}

__device__ __forceinline__ void combine_into(float2 v, float& M, float& S) {
  // S is kept relative to M; v = (ref, sum)
  if (v.x > M) {
    S = (M > -INFINITY ? S * ex2(M - v.x) : S) + v.y;
    M = v.x;
  } else {
    S += (v.x > -INFINITY) ? v.y * ex2(v.x - M) : v.y;
  }
}

// Online (reference, sum) update with one value v (units of z'c).
__device__ __forceinline__ void online_add(float v, float& ref, float& s) {
  if (v > -INFINITY) {
    if (v > ref) {
      s = (ref > -INFINITY ? s * ex2(ref - v) : 0.f) + 1.f;
      ref = v;
    } else {
      s += ex2(v - ref);
    }
  }
}

}  // namespace

}  // namespace sv
