// Device helpers shared by the two sampling kernels (the cluster/resident
// kernel in sample_verify.cu and the pipelined streaming kernel in
// pipe_verify.cu): work-item decoding, per-request validity, the
// 256-token chunk layout used for direct global reads, probability and
// residual arithmetic, and the fp64 chunk scan.
#pragma once

#include "common.cuh"
#include "spec_internal.h"

namespace sv {

struct Item {
  int b, i, K;
  int tgt_row, dft_row;
  bool bonus;
  bool rows_ok;
};

__device__ __forceinline__ Item decode_item(const SampleParams& P, int item) {
  Item it;
  if (item < P.total) {
    int lo = 0, hi = P.B;
    while (hi - lo > 1) {
      const int mid = (lo + hi) >> 1;
      if (__ldg(P.cu_draft + mid) <= item) lo = mid; else hi = mid;
    }
    it.b = lo;
    it.i = item - __ldg(P.cu_draft + lo);
    it.bonus = false;
    it.tgt_row = item + lo;
    it.dft_row = item;
    it.rows_ok = true;
  } else {
    const int b = item - P.total;
    const int c0 = __ldg(P.cu_draft + b), c1 = __ldg(P.cu_draft + b + 1);
    it.b = b;
    it.i = c1 - c0;
    it.bonus = true;
    it.rows_ok = (c0 >= 0 && c0 <= c1 && c1 <= P.total);
    it.tgt_row = it.rows_ok ? c1 + b : b;
    it.dft_row = -1;
  }
  it.K = __ldg(P.cu_draft + it.b + 1) - __ldg(P.cu_draft + it.b);
  return it;
}

// Validity of a request's scalars (read the same way by producer and consumers).
__device__ __forceinline__ bool item_params_ok(const SampleParams& P, int b) {
  const float T_ = P.temperature ? __ldg(P.temperature + b) : 1.f;
  const float alpha = P.rep_penalty ? __ldg(P.rep_penalty + b) : 1.f;
  const float tp = P.top_p ? __ldg(P.top_p + b) : 1.f;
  const float D = P.tv_budget ? __ldg(P.tv_budget + b) : 0.f;
  return (T_ > 0.f) && (T_ < INFINITY) && (alpha > 0.f) && (alpha < INFINITY) && (tp > 0.f) && (tp <= 1.f) &&
         (D >= 0.f) && (D <= 1.f);
}

// Top-p radix passes an item makes: 4 when it filters, else 0.
template <bool TOPP>
__device__ __forceinline__ int radix_passes(const SampleParams& P, int b) {
  if constexpr (!TOPP) {
    return 0;
  } else {
    return (item_params_ok(P, b) && __ldg(P.top_p + b) < 1.f) ? 4 : 0;
  }
}

// Element j (0..7) of a lane within a 256-token chunk: 4l+j, then 128+4l+j-4.
__device__ __forceinline__ int lane_elem(int lane, int j) { return j < 4 ? 4 * lane + j : 128 + 4 * lane + (j - 4); }

// The same 8 logits read straight from global memory (used once per item by
// the streaming variant's candidate search).  Loads first, then conversion,
// so that callers can issue the loads of several rows back to back.
template <typename T>
__device__ __forceinline__ void global_raw(const T* slice_row, int ib, int lane, int len, T* raw) {
#pragma unroll
  for (int j = 0; j < 8; ++j) {
    const int idx = ib + lane_elem(lane, j);
    raw[j] = slice_row[idx < len ? idx : 0];
  }
}

template <typename T>
__device__ __forceinline__ void convert_raw(const T* raw, int ib, int lane, int len, const uint32_t* bitmap, bool pen,
                                            float alpha, float* z) {
#pragma unroll
  for (int j = 0; j < 8; ++j) {
    const int idx = ib + lane_elem(lane, j);
    z[j] = idx < len ? to_f32<T>(raw[j]) : -INFINITY;
    if (pen && idx < len && ((bitmap[idx >> 5] >> (idx & 31)) & 1u)) z[j] = penalize(z[j], alpha);
  }
}

template <typename T>
__device__ __forceinline__ void global_logits(const T* slice_row, int ib, int lane, int len, const uint32_t* bitmap,
                                              bool pen, float alpha, float* z) {
  T raw[8];
  global_raw<T>(slice_row, ib, lane, len, raw);
  convert_raw<T>(raw, ib, lane, len, bitmap, pen, alpha, z);
}

// Order-preserving map of an fp32 logit to an unsigned key (ties stay ties).
__device__ __forceinline__ uint32_t order_key(float z) {
  const uint32_t u = __float_as_uint(z);
  return (u & 0x80000000u) ? ~u : (u | 0x80000000u);
}

// How a value becomes a probability.  Resident variant without top-p: the
// store holds e = 2^(z'c - ref_k) and p = e * fac_k, fac_k = 2^(ref_k - M)/S.
// Otherwise the value is the penalised logit z' itself (resident top-p
// store, or any streamed logit) and p = [key(z') >= tau] 2^(z'c - M) / kept;
// cutting the nucleus on exact logit keys keeps equal logits together.
struct RowProb {
  uint32_t tau_key;  // keep key(z') >= tau_key (0 keeps every token)
  float c, mc;       // log2(e)/T and the row reference M (units of z'c)
  float invs;        // 1 / kept mass
  double kept;       // kept mass, in units of 2^(z'c - M)
};

// Probability modes: kPE = stored e times its chunk factor (resident, no
// top-p); kPZ = logit, no top-p; kPZT = logit with the top-p cut.
enum { kPE = 0, kPZ = 1, kPZT = 2 };

template <int MODE>
__device__ __forceinline__ float prob1(float s, float fac, const RowProb& rp) {
  if constexpr (MODE == kPE) {
    return s * fac;
  } else if constexpr (MODE == kPZ) {
    return ex2(fmaf(s, rp.c, -rp.mc)) * rp.invs;
  } else {
    return order_key(s) >= rp.tau_key ? ex2(fmaf(s, rp.c, -rp.mc)) * rp.invs : 0.f;
  }
}

// The same for a lane's 8 values, in packed fp32x2 arithmetic (bit-identical
// to prob1 element by element).
template <int MODE>
__device__ __forceinline__ void probs8(const float* s, float fac, const RowProb& rp, float* p) {
  if constexpr (MODE == kPE) {
    const float2 f2 = make_float2(fac, fac);
#pragma unroll
    for (int j = 0; j < 8; j += 2) {
      const float2 r = __fmul2_rn(make_float2(s[j], s[j + 1]), f2);
      p[j] = r.x;
      p[j + 1] = r.y;
    }
  } else {
    const float2 c2 = make_float2(rp.c, rp.c), m2 = make_float2(-rp.mc, -rp.mc);
    const float2 i2 = make_float2(rp.invs, rp.invs);
#pragma unroll
    for (int j = 0; j < 8; j += 2) {
      const float2 y = __ffma2_rn(make_float2(s[j], s[j + 1]), c2, m2);
      const float2 r = __fmul2_rn(make_float2(ex2(y.x), ex2(y.y)), i2);
      p[j] = r.x;
      p[j + 1] = r.y;
    }
    if constexpr (MODE == kPZT) {
#pragma unroll
      for (int j = 0; j < 8; ++j)
        if (order_key(s[j]) < rp.tau_key) p[j] = 0.f;
    }
  }
}

// r = max(p - q, 0) for 8 values; returns their sum.
__device__ __forceinline__ float resid8(const float* p, const float* q, float* r) {
  const float2 m1 = make_float2(-1.f, -1.f);
  float2 acc = make_float2(0.f, 0.f);
#pragma unroll
  for (int j = 0; j < 8; j += 2) {
    const float2 d = __ffma2_rn(make_float2(q[j], q[j + 1]), m1, make_float2(p[j], p[j + 1]));
    r[j] = fmaxf(d.x, 0.f);
    r[j + 1] = fmaxf(d.y, 0.f);
    acc = __fadd2_rn(acc, make_float2(r[j], r[j + 1]));
  }
  return acc.x + acc.y;
}

__device__ __forceinline__ float sum8(const float* v) {
  float2 a = __fadd2_rn(make_float2(v[0], v[1]), make_float2(v[2], v[3]));
  const float2 b = __fadd2_rn(make_float2(v[4], v[5]), make_float2(v[6], v[7]));
  a = __fadd2_rn(a, b);
  return a.x + a.y;
}

// Warp 0 of every CTA: the chunk sums seg[0..nch) summed in fp64 over lane
// blocks of consecutive chunks, then scanned across lanes.  Every use (the
// CTA total exchanged over the cluster and the owner's search) takes this
// one order of summation.
__device__ __forceinline__ double seg_block_scan(const float* seg, int nch, int lane, int& k0, int& k1,
                                                 double& block, double& incl) {
  const int bl = (nch + 31) / 32;
  k0 = min(nch, lane * bl);
  k1 = min(nch, k0 + bl);
  double s = 0.0;
  for (int k = k0; k < k1; ++k) s += (double)seg[k];
  block = s;
  incl = warp_incl_scan_d(s, lane);
  return __shfl_sync(0xffffffffu, incl, 31);
}

__device__ __forceinline__ void exps8(const float* z, float c, float refc, float* e) {
  const float2 c2 = make_float2(c, c), nr = make_float2(-refc, -refc);
#pragma unroll
  for (int j = 0; j < 8; j += 2) {
    const float2 y = __ffma2_rn(make_float2(z[j], z[j + 1]), c2, nr);
    e[j] = ex2(y.x);
    e[j + 1] = ex2(y.y);
  }
}

__device__ __forceinline__ float max8(const float* z) {
  float m = fmaxf(fmaxf(z[0], z[1]), fmaxf(z[2], z[3]));
  return fmaxf(m, fmaxf(fmaxf(z[4], z[5]), fmaxf(z[6], z[7])));
}

// Streaming pass-1 statistics of one chunk of NR rows with a per-lane running
// reference (no warp-wide step in the hot loop): each lane keeps refc, the
// running maximum of z'c it has seen when a chunk would overflow (sum above
// 2^64; first set from the lane's first chunk), and Ssum of 2^(z'c - refc).
template <int NR>
__device__ __forceinline__ void chunk_stats_lane(float (&z)[2][8], float c, float* refc, bool& have_ref, float* Ssum) {
  const float kLim = 18446744073709551616.0f;  // 2^64
  if (!have_ref) {
#pragma unroll
    for (int r = 0; r < NR; ++r) {
      const float mx = max8(z[r]);
      refc[r] = (mx > -INFINITY) ? mx * c : 0.f;
    }
    have_ref = true;
  }
#pragma unroll
  for (int r = 0; r < NR; ++r) {
    float e[8];
    exps8(z[r], c, refc[r], e);
    float s = sum8(e);
    if (!(s <= kLim)) {  // rare and lane-local
      const float mx = max8(z[r]);
      const float nref = (mx > -INFINITY) ? mx * c : 0.f;
      if (nref > refc[r]) {
        Ssum[r] *= ex2(refc[r] - nref);
        refc[r] = nref;
      }
      exps8(z[r], c, refc[r], e);
      s = sum8(e);
    }
    Ssum[r] += s;
  }
}

}  // namespace sv
