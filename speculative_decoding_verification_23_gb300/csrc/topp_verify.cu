// Top-p path of mentored speculative sampling ("What I Gave Up to Make
// Speculative Decoding Faster", section "A knob for accepting more draft
// tokens", with both distributions filtered by top-p as in the "Speculative
// Decoding" note, section "Warum eine Korrektur noetig ist").
//
// Row-cut kernel: one persistent CTA per SM takes logical rows r =
// blockIdx.x + j * gridDim.x.  A producer warp streams each row through a
// ring of 16 KB TMA bulk copies; 16 consumer warps make one pass over it:
//  - the row's maximum M of z'c and its mass S = sum 2^(z'c - M), each thread
//    keeping a running reference that it lowers its sum to when it rises;
//  - the candidates: every token within kCutWindow (log2 units) of the
//    running maximum, as (index, z') pairs in shared memory.  The running
//    maximum never exceeds M, so every token within the window of M is
//    among them.
// The cut is then an exact select on the order keys of z': the largest key
// whose upper set holds top_p * S, by histograms of mass over key ranges,
// each level narrowing the range 1024-fold, and a sort of the last few.  It
// reads the candidates when the window holds the cut (the common case),
// else the row from global memory again (the window missed, or the
// candidates overflowed).  The kept tokens go to a pool as a list.
//
// Finish kernel: one CTA per request.  Status, then for each position
// p~(x) and q~(x) from the row records and two gathers, d = TV(p~, q~) =
// sum over p's list of max(p~ - q~, 0), theta, pi(x) and the acceptance
// test; then the residual or bonus draw in token order over the list.
// Rows without a list are scanned in full.
#include <cstdint>
#include <cuda_runtime.h>
#include <cuda_bf16.h>

#include "common.cuh"
#include "spec_internal.h"
#include "topp_internal.h"

namespace sv {
namespace {

// ------------------------------------------------------------ shared layout
constexpr int kOffCand = kCutSlots * kCutChunkBytes;
constexpr int kOffBits = kOffCand + kCutCand * 8;
constexpr int kOffHm = kOffBits + kCutMaxV / 8;
constexpr int kOffHc = kOffHm + kCutBins * 4;
constexpr int kOffBars = kOffHc + kCutBins * 4;
constexpr int kOffMisc = kOffBars + 2 * kCutSlots * 8;

struct CutMisc {
  double dred[kCutConsumerWarps];
  float wM[kCutConsumerWarps];
  float wS[kCutConsumerWarps];
  unsigned kred[kCutConsumerWarps];
  int ired[kCutConsumerWarps];
  int ired2[kCutConsumerWarps];
  double above;          // mass above the current key range
  int ncand, over, bad, cta_max;
  int abort;             // a bounded wait ran out in this CTA
  int snap[2];           // abort, as all consumer warps read it after a barrier
  int bstar, nsmall, nlist;
  unsigned klo, khi;
  unsigned tau_key;
  float M, S;
  double Sk;
  int n_upper, done, dense;
};
constexpr int kCutSmem = kOffMisc + (int)sizeof(CutMisc);
static_assert(kCutSmem <= 232448, "shared memory of the row-cut kernel");
static_assert(kOffBars % 8 == 0 && kOffMisc % 8 == 0, "alignment");

constexpr int kConsumerBar = 1;
__device__ __forceinline__ void csync() { named_sync(kConsumerBar, kCutConsumers); }

// Order-preserving int image of a float (for atomicMax in shared memory).
__device__ __forceinline__ int fkey_i(float f) {
  const int i = __float_as_int(f);
  return i >= 0 ? i : i ^ 0x7fffffff;
}
__device__ __forceinline__ float fval_i(int k) { return __int_as_float(k >= 0 ? k : k ^ 0x7fffffff); }

// Order-preserving unsigned key of an fp32 logit (equal logits, equal keys).
__device__ __forceinline__ uint32_t okey(float z) {
  const uint32_t u = __float_as_uint(z);
  return (u & 0x80000000u) ? ~u : (u | 0x80000000u);
}
__device__ __forceinline__ float okey_val(uint32_t k) {
  return __uint_as_float((k & 0x80000000u) ? (k & 0x7fffffffu) : ~k);
}

// Merge two (reference, sum) pairs, the sum relative to 2^reference.
__device__ __forceinline__ void ref_merge(float& M, float& S, float m, float s) {
  if (!(m > -INFINITY)) return;
  if (!(M > -INFINITY)) {
    M = m;
    S = s;
    return;
  }
  if (m > M) {
    S = S * ex2(M - m) + s;
    M = m;
  } else {
    S += s * ex2(m - M);
  }
}

// The request and row of logical row r (rows in request order), by binary
// search over the requests' first rows 2 cu_draft[b] + b; the logits row
// (target row, or draft row + NT); false when r does not map to a row of a
// consistent request.
struct RowMap {
  int b, i, kind, src, K;
};
__device__ __forceinline__ bool map_row(const ToppParams& P, int r, RowMap& m) {
  int lo = 0, hi = P.B - 1;
  while (lo < hi) {
    const int mid = (lo + hi + 1) >> 1;
    if (2 * __ldg(P.cu_draft + mid) + mid <= r) lo = mid;
    else hi = mid - 1;
  }
  const int b = lo;
  const int d0 = __ldg(P.cu_draft + b), d1 = __ldg(P.cu_draft + b + 1);
  m.b = b;
  m.K = d1 - d0;
  const int off = r - (2 * d0 + b);
  m.i = off >> 1;
  m.kind = off & 1;
  if (d0 < 0 || d1 < d0 || d1 > P.total || off < 0 || m.i > m.K || (m.kind && m.i >= m.K)) return false;
  m.src = m.kind ? P.NT + d0 + m.i : d0 + b + m.i;
  return true;
}

template <typename T>
__device__ __forceinline__ const unsigned char* logits_row(const ToppParams& P, int src) {
  if (src < P.NT)
    return reinterpret_cast<const unsigned char*>(P.target) + (size_t)src * (size_t)P.ld_t * sizeof(T);
  return reinterpret_cast<const unsigned char*>(P.draft) + (size_t)(src - P.NT) * (size_t)P.ld_d * sizeof(T);
}

__device__ __forceinline__ bool request_params_ok(const ToppParams& P, int b) {
  const float T = __ldg(P.temperature + b);
  const float alpha = P.rep_penalty ? __ldg(P.rep_penalty + b) : 1.f;
  const float tp = __ldg(P.top_p + b);
  const float D = __ldg(P.tv_budget + b);
  return T > 0.f && T < INFINITY && alpha > 0.f && alpha < INFINITY && tp > 0.f && tp <= 1.f && D >= 0.f &&
         D <= 1.f;
}

// The bytes a row's copies cover: V logits rounded up to 16 bytes (inside
// the row's padded stride, which the host checks is a multiple of 16 bytes).
__device__ __forceinline__ int row_bytes(const ToppParams& P, int es) { return (P.V * es + 15) & ~15; }

// Bounded wait on a ring barrier; gives up at once when this CTA has
// aborted, and aborts it when the limit runs out.
__device__ __forceinline__ bool cut_wait(uint64_t* bar, uint32_t parity, CutMisc* ms) {
  if (mbar_test(bar, parity)) return true;
  const long long t0 = clock64();
  for (;;) {
    if (mbar_test(bar, parity)) return true;
    if (*reinterpret_cast<volatile int*>(&ms->abort)) return false;
    if (clock64() - t0 > kWaitLimitCycles) {
      atomicExch(&ms->abort, 1);
      return false;
    }
  }
}

// ------------------------------------------------------------ the producer
// The ring holds kCutSlots chunks (96 KB), too few bytes in flight for an
// SM's share of HBM bandwidth at the latency of a loaded memory system.  So
// the producer also prefetches into L2 the chunk kCutPrefetch positions
// ahead of the one it copies (384 KB ahead), before it waits for a free
// slot: the copies then mostly read L2, and the prefetches keep HBM busy
// while the consumers select a row's cut.
constexpr int kCutPrefetch = 24;

__device__ __forceinline__ void prefetch_l2(const void* p, uint32_t bytes) {
  asm volatile("cp.async.bulk.prefetch.L2.global [%0], %1;" ::"l"(p), "r"(bytes) : "memory");
}

// A position in this CTA's chunk sequence (rows blockIdx.x + j gridDim.x,
// chunks 0 .. nch - 1 of each).
struct ChunkCursor {
  int r = 0, ch = 0;
  const unsigned char* src = nullptr;
  template <typename T>
  __device__ __forceinline__ void start(const ToppParams& P, int row) {
    r = row;
    ch = 0;
    RowMap m;
    src = r < P.NR ? logits_row<T>(P, map_row(P, r, m) ? m.src : 0) : nullptr;
  }
  template <typename T>
  __device__ __forceinline__ void next(const ToppParams& P, int nch) {
    if (++ch == nch) start<T>(P, r + (int)gridDim.x);
  }
};

template <typename T>
__device__ void cut_producer(const ToppParams& P, unsigned char* ring, uint64_t* full, uint64_t* empty, CutMisc* ms,
                             int lane) {
  if (lane != 0) return;
  const uint64_t pol = l2_policy_evict_first();
  const int rb = row_bytes(P, (int)sizeof(T));
  const int nch = (rb + kCutChunkBytes - 1) / kCutChunkBytes;
  auto chunk_bytes = [&](int ch) { return (uint32_t)min(kCutChunkBytes, rb - ch * kCutChunkBytes); };
  RingFills fills;
  ChunkCursor cur, pre;
  cur.start<T>(P, blockIdx.x);
  pre.start<T>(P, blockIdx.x);
  for (int i = 0; i < kCutPrefetch && pre.r < P.NR; ++i) {
    prefetch_l2(pre.src + (size_t)pre.ch * kCutChunkBytes, chunk_bytes(pre.ch));
    pre.next<T>(P, nch);
  }
  for (int k = 0; cur.r < P.NR; ++k) {
    if (pre.r < P.NR) {
      prefetch_l2(pre.src + (size_t)pre.ch * kCutChunkBytes, chunk_bytes(pre.ch));
      pre.next<T>(P, nch);
    }
    const int s = k % kCutSlots;
    if (k >= kCutSlots && !cut_wait(empty + s, (uint32_t)((k / kCutSlots - 1) & 1), ms)) break;
    const uint32_t bytes = chunk_bytes(cur.ch);
    mbar_arrive_expect_tx(full + s, bytes);
    bulk_g2s(ring + (size_t)s * kCutChunkBytes, cur.src + (size_t)cur.ch * kCutChunkBytes, bytes, full + s, pol);
    fills.note((uint32_t)s, (uint32_t)((k / kCutSlots) & 1));
    cur.next<T>(P, nch);
  }
  // nothing may land in shared memory after the CTA exits
  fills.drain(full, kCutSlots);
}

// ------------------------------------------------------------ the consumers
// Elements of a 16-byte vector as fp32.
template <typename T>
struct Vec;
template <>
struct Vec<float> {
  static constexpr int N = 4;
  __device__ static void cvt(const uint4& v, float (&z)[8]) {
    z[0] = __uint_as_float(v.x);
    z[1] = __uint_as_float(v.y);
    z[2] = __uint_as_float(v.z);
    z[3] = __uint_as_float(v.w);
  }
};
template <>
struct Vec<__nv_bfloat16> {
  static constexpr int N = 8;
  __device__ static void cvt(const uint4& v, float (&z)[8]) {
    z[0] = __uint_as_float(v.x << 16);
    z[1] = __uint_as_float(v.x & 0xffff0000u);
    z[2] = __uint_as_float(v.y << 16);
    z[3] = __uint_as_float(v.y & 0xffff0000u);
    z[4] = __uint_as_float(v.z << 16);
    z[5] = __uint_as_float(v.z & 0xffff0000u);
    z[6] = __uint_as_float(v.w << 16);
    z[7] = __uint_as_float(v.w & 0xffff0000u);
  }
};

// One row's setting, the same in every consumer thread.
struct RowCtx {
  RowMap m;
  bool mapped, usable, pen;
  float c, alpha, tp;
};

// The penalised logits of a 16-byte vector whose first token is t0
// (tokens >= V read as -inf); `bad` collects NaN and +inf of real tokens.
template <typename T>
__device__ __forceinline__ void pen_vec(const uint4& raw, int t0, const RowCtx& x, const uint32_t* bits, int V,
                                        float (&z)[8], bool& bad) {
  constexpr int N = Vec<T>::N;
  Vec<T>::cvt(raw, z);
  uint32_t w = 0;
  if (x.pen && t0 < V) w = bits[t0 >> 5] >> (t0 & 31);
#pragma unroll
  for (int j = 0; j < N; ++j) {
    if (t0 + j < V) {
      bad |= is_bad_logit(z[j]);
      if ((w >> j) & 1u) z[j] = penalize(z[j], x.alpha);
    } else {
      z[j] = -INFINITY;
    }
  }
}

// Block-wide (consumer threads) reductions through the shared scratch.
__device__ __forceinline__ unsigned cmin_u(unsigned v, CutMisc* ms, int cw, int lane) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v = min(v, __shfl_xor_sync(0xffffffffu, v, o));
  if (lane == 0) ms->kred[cw] = v;
  csync();
  unsigned t = 0xffffffffu;
#pragma unroll
  for (int w = 0; w < kCutConsumerWarps; ++w) t = min(t, ms->kred[w]);
  csync();
  return t;
}
__device__ __forceinline__ unsigned cmax_u(unsigned v, CutMisc* ms, int cw, int lane) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v = max(v, __shfl_xor_sync(0xffffffffu, v, o));
  if (lane == 0) ms->kred[cw] = v;
  csync();
  unsigned t = 0u;
#pragma unroll
  for (int w = 0; w < kCutConsumerWarps; ++w) t = max(t, ms->kred[w]);
  csync();
  return t;
}

// Visits every token of the select's source with (index, penalised logit):
// the candidates (from shared memory), or the whole row (from global
// memory, eight 16-byte loads in flight per thread).
template <typename T, bool GLOBAL, typename F>
__device__ __forceinline__ void visit(const ToppParams& P, const RowCtx& x, const int2* cand, int ncand,
                                      const uint32_t* bits, int ct, F&& f) {
  if constexpr (!GLOBAL) {
    for (int j = ct; j < ncand; j += kCutConsumers) {
      const int2 e = cand[j];
      f(e.x, __int_as_float(e.y));
    }
  } else {
    constexpr int N = Vec<T>::N;
    constexpr int kDepth = 8;
    const uint4* row = reinterpret_cast<const uint4*>(logits_row<T>(P, x.m.src));
    const int nv = row_bytes(P, (int)sizeof(T)) / 16;
    for (int v0 = ct; v0 < nv; v0 += kDepth * kCutConsumers) {
      uint4 raw[kDepth];
#pragma unroll
      for (int q = 0; q < kDepth; ++q) {
        const int v = v0 + q * kCutConsumers;
        raw[q] = v < nv ? __ldcg(row + v) : make_uint4(0u, 0u, 0u, 0u);
      }
#pragma unroll
      for (int q = 0; q < kDepth; ++q) {
        const int v = v0 + q * kCutConsumers;
        if (v >= nv) break;
        float z[8];
        bool bad = false;
        pen_vec<T>(raw[q], v * N, x, bits, P.V, z, bad);
#pragma unroll
        for (int j = 0; j < N; ++j)
          if (v * N + j < P.V) f(v * N + j, z[j]);
      }
    }
  }
}

// One level of the select: a histogram of mass (2^(z'c - M)) and count
// over the bins that `binf` assigns (-1: not in this level), then the first
// bin from the top whose inclusive mass, with `above` before the first
// bin, reaches the target.  Every consumer thread gets the same result.
struct BinPick {
  int b;          // the bin (-1: none reaches the target)
  int lastb;      // the last bin with tokens
  double above;   // mass before bin b (with the level's `above`)
  int n_above;    // tokens before bin b (with the level's count)
  int cnt;        // tokens in bin b
  double mass;    // their mass
};

template <typename T, bool GLOBAL, typename BinF>
__device__ BinPick pick_bin(const ToppParams& P, const RowCtx& x, const int2* cand, int ncand, float M,
                            double target, double above, int n_above, float* hm, int* hc, const uint32_t* bits,
                            CutMisc* ms, int ct, int cw, int lane, BinF&& binf) {
  for (int j = ct; j < kCutBins; j += kCutConsumers) {
    hm[j] = 0.f;
    hc[j] = 0;
  }
  csync();
  visit<T, GLOBAL>(P, x, cand, ncand, bits, ct, [&](int, float z) {
    const int bin = binf(z);
    if (bin < 0) return;
    atomicAdd(hm + bin, ex2(__fmul_rn(z, x.c) - M));
    atomicAdd(hc + bin, 1);
  });
  csync();
  static_assert(kCutBins == 2 * kCutConsumers, "two bins per consumer thread");
  const double m0 = (double)hm[2 * ct], m1 = (double)hm[2 * ct + 1];
  const int c0 = hc[2 * ct], c1 = hc[2 * ct + 1];
  const double incl = warp_incl_scan_d(m0 + m1, lane);
  int cincl = c0 + c1;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const int t = __shfl_up_sync(0xffffffffu, cincl, o);
    if (lane >= o) cincl += t;
  }
  if (lane == 31) {
    ms->dred[cw] = incl;
    ms->ired[cw] = cincl;
  }
  csync();
  double wbase = 0.0;
  int cbase = 0;
  for (int w = 0; w < cw; ++w) {
    wbase += ms->dred[w];
    cbase += ms->ired[w];
  }
  const double excl = above + wbase + incl - (m0 + m1);
  const int cexcl = n_above + cbase + cincl - (c0 + c1);
  int pick = 0x7fffffff;
  if (excl + m0 >= target && c0 > 0) pick = 2 * ct;
  else if (excl + m0 + m1 >= target && c1 > 0) pick = 2 * ct + 1;
  int last = c1 > 0 ? 2 * ct + 1 : (c0 > 0 ? 2 * ct : -1);
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
    pick = min(pick, __shfl_xor_sync(0xffffffffu, pick, o));
    last = max(last, __shfl_xor_sync(0xffffffffu, last, o));
  }
  if (lane == 0) {
    ms->kred[cw] = (unsigned)pick;
    ms->ired2[cw] = last;
  }
  csync();
  BinPick r;
  int b = 0x7fffffff;
  r.lastb = -1;
  for (int w = 0; w < kCutConsumerWarps; ++w) {
    b = min(b, (int)ms->kred[w]);
    r.lastb = max(r.lastb, ms->ired2[w]);
  }
  r.b = b == 0x7fffffff ? -1 : b;
  csync();
  // the owner of the chosen bin (or of the last one) publishes what lies above it
  const int ob = r.b >= 0 ? r.b : r.lastb;
  if (ob >= 0 && ob >> 1 == ct) {
    ms->above = (ob & 1) ? excl + m0 : excl;
    ms->n_upper = (ob & 1) ? cexcl + c0 : cexcl;
    ms->bstar = (ob & 1) ? c1 : c0;
    ms->Sk = (ob & 1) ? m1 : m0;
  }
  csync();
  r.above = ms->above;
  r.n_above = ms->n_upper;
  r.cnt = ms->bstar;
  r.mass = ms->Sk;
  csync();
  return r;
}

// The cut among at most 32 tokens (those `inb` accepts), with `above` the
// mass and `n_above` the count of the tokens of higher keys: the tokens
// sorted by key, ties walked together.  Sets ms->tau_key, ms->Sk and
// ms->n_upper (an upper bound on the kept count).
template <typename T, bool GLOBAL, typename InB>
__device__ void small_cut(const ToppParams& P, const RowCtx& x, const int2* cand, int ncand, float M, double target,
                          double above, int n_above, float* hm, int* hc, const uint32_t* bits, CutMisc* ms, int ct,
                          int cw, int lane, InB&& inb) {
  if (ct == 0) ms->nsmall = 0;
  csync();
  unsigned* sk = reinterpret_cast<unsigned*>(hc);
  float* smass = hm;
  visit<T, GLOBAL>(P, x, cand, ncand, bits, ct, [&](int, float z) {
    if (!inb(z)) return;
    const int s = atomicAdd(&ms->nsmall, 1);
    if (s < 32) {
      sk[s] = okey(z);
      smass[s] = ex2(__fmul_rn(z, x.c) - M);
    }
  });
  csync();
  if (cw == 0) {
    const int n = min(ms->nsmall, 32);
    const unsigned k = lane < n ? sk[lane] : 0u;
    const double w = lane < n ? (double)smass[lane] : 0.0;
    double grp = 0.0, hi_mass = 0.0;
    for (int j = 0; j < n; ++j) {
      const unsigned kj = __shfl_sync(0xffffffffu, k, j);
      const double wj = __shfl_sync(0xffffffffu, w, j);
      if (lane < n) {
        if (kj == k) grp += wj;
        else if (kj > k) hi_mass += wj;
      }
    }
    // a key is the cut when its upper set (itself included) reaches the
    // target and the keys above it do not; the lowest key if none does
    const double upto = above + hi_mass + grp;
    const bool is_cut = lane < n && upto >= target && above + hi_mass < target;
    const unsigned cm = __ballot_sync(0xffffffffu, is_cut);
    unsigned best;
    double bsk;
    if (cm) {
      const int L = __ffs(cm) - 1;
      best = __shfl_sync(0xffffffffu, k, L);
      bsk = __shfl_sync(0xffffffffu, upto, L);
    } else {
      unsigned mk = lane < n ? k : 0xffffffffu;
      double tot = lane < n ? w : 0.0;
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) {
        mk = min(mk, __shfl_xor_sync(0xffffffffu, mk, o));
        tot += __shfl_xor_sync(0xffffffffu, tot, o);
      }
      best = mk;
      bsk = above + tot;
    }
    if (lane == 0) {
      ms->tau_key = best;
      ms->Sk = bsk;
      ms->n_upper = n_above + n;
    }
  }
  csync();
}

// The exact cut over the tokens of a source that `inr` accepts, with the
// mass and count of higher tokens given: levels of 1024 bins over shrinking
// ranges of the order keys of z' (each level narrows the range 1024-fold),
// until one key or at most 32 tokens remain.  When rounding leaves the
// target out of reach, down to the lowest token.
template <typename T, bool GLOBAL, typename InR>
__device__ void key_levels(const ToppParams& P, const RowCtx& x, const int2* cand, int ncand, float M, double target,
                           double above, int n_above, float* hm, int* hc, const uint32_t* bits, CutMisc* ms, int ct,
                           int cw, int lane, InR&& inr) {
  unsigned klo = 0xffffffffu, khi = 0u;
  visit<T, GLOBAL>(P, x, cand, ncand, bits, ct, [&](int, float z) {
    if (z > -INFINITY && inr(z)) {
      klo = min(klo, okey(z));
      khi = max(khi, okey(z));
    }
  });
  klo = cmin_u(klo, ms, cw, lane);
  khi = cmax_u(khi, ms, cw, lane);
  for (int level = 0; level < 6 && klo <= khi; ++level) {
    const unsigned long long range = (unsigned long long)(khi - klo) + 1ull;
    const unsigned lo = klo, hi = khi;
    auto kbin = [&](float z) -> int {
      const uint32_t kz = okey(z);
      if (kz < lo || kz > hi || !inr(z)) return -1;
      return (int)(((unsigned long long)(hi - kz) * (unsigned long long)kCutBins) / range);
    };
    BinPick bp = pick_bin<T, GLOBAL>(P, x, cand, ncand, M, target, above, n_above, hm, hc, bits, ms, ct, cw, lane,
                                     kbin);
    const int b = bp.b >= 0 ? bp.b : bp.lastb;
    const unsigned lo_off = (unsigned)(((unsigned long long)b * range + kCutBins - 1) / kCutBins);
    const unsigned hi_off = (unsigned)(((unsigned long long)(b + 1) * range + kCutBins - 1) / kCutBins) - 1u;
    const unsigned nkhi = hi - lo_off, nklo = hi - hi_off;
    above = bp.above;
    n_above = bp.n_above;
    if (nklo == nkhi) {
      // one key: every token of it is kept, however many tie
      if (ct == 0) {
        ms->tau_key = nkhi;
        ms->Sk = above + bp.mass;
        ms->n_upper = n_above + bp.cnt;
      }
      csync();
      return;
    }
    if (bp.cnt <= 32) {
      small_cut<T, GLOBAL>(P, x, cand, ncand, M, target, above, n_above, hm, hc, bits, ms, ct, cw, lane,
                           [&](float z) {
                             const uint32_t kz = okey(z);
                             return kz >= nklo && kz <= nkhi && inr(z);
                           });
      return;
    }
    klo = nklo;
    khi = nkhi;
  }
  // the key ranges shrink 1024-fold a level, so the loop ends in small_cut
  if (ct == 0) {
    ms->tau_key = klo;
    ms->Sk = target;
    ms->n_upper = n_above;
  }
  csync();
}

// The cut from the candidates: a first level of 1024 bins uniform in z'c
// over the window [M - kCutWindow, M], then the tokens of the chosen bin.
// False when the window's mass is short of the target (the cut lies below
// it).
template <typename T>
__device__ bool select_window(const ToppParams& P, const RowCtx& x, const int2* cand, int ncand, float M,
                              double target, float* hm, int* hc, const uint32_t* bits, CutMisc* ms, int ct, int cw,
                              int lane) {
  const float ylo = M - kCutWindow;
  const float scale = (float)kCutBins / kCutWindow;
  auto ybin = [=](float z) -> int {
    const float y = __fmul_rn(z, x.c);
    if (!(y >= ylo)) return -1;
    return min(kCutBins - 1, (int)((M - y) * scale));
  };
  const BinPick bp = pick_bin<T, false>(P, x, cand, ncand, M, target, 0.0, 0, hm, hc, bits, ms, ct, cw, lane, ybin);
  if (bp.b < 0) return false;
  const int b = bp.b;
  auto inb = [=](float z) { return ybin(z) == b; };
  if (bp.cnt <= 32)
    small_cut<T, false>(P, x, cand, ncand, M, target, bp.above, bp.n_above, hm, hc, bits, ms, ct, cw, lane, inb);
  else
    key_levels<T, false>(P, x, cand, ncand, M, target, bp.above, bp.n_above, hm, hc, bits, ms, ct, cw, lane, inb);
  return true;
}

// The consumer warps (consumer thread ct = 0..511, warp cw = 0..15): per
// row the penalty bitmap, the streaming pass, then the cut and the list.
template <typename T>
__device__ void cut_consumers(const ToppParams& P, unsigned char* smem, uint64_t* full, uint64_t* empty,
                              CutMisc* ms, int ct, int cw, int lane) {
  constexpr int N = Vec<T>::N;
  const int rb = row_bytes(P, (int)sizeof(T));
  const int nch = (rb + kCutChunkBytes - 1) / kCutChunkBytes;
  int2* cand = reinterpret_cast<int2*>(smem + kOffCand);
  uint32_t* bits = reinterpret_cast<uint32_t*>(smem + kOffBits);
  float* hm = reinterpret_cast<float*>(smem + kOffHm);
  int* hc = reinterpret_cast<int*>(smem + kOffHc);
  const unsigned tag32 = (unsigned)P.tag;
  const int tpc = kCutChunkBytes / (int)sizeof(T);   // tokens per chunk
  // this CTA's share of the pool, taken row by row
  const int pool_per = P.pool_cap / (int)gridDim.x;
  const int pool0 = (int)blockIdx.x * pool_per;
  int pool_used = 0;
  int k = 0;          // chunks taken from the ring
  int par = 0;        // which abort snapshot this row reads
  for (int r = blockIdx.x; r < P.NR; r += gridDim.x, par ^= 1) {
    RowCtx x;
    x.mapped = map_row(P, r, x.m);
    const int b = x.m.b;
    x.usable = x.mapped && request_params_ok(P, b);
    x.alpha = P.rep_penalty ? __ldg(P.rep_penalty + b) : 1.f;
    x.tp = __ldg(P.top_p + b);
    x.c = x.usable ? (float)(1.4426950408889634 / (double)__ldg(P.temperature + b)) : 1.f;
    x.pen = x.usable && x.alpha != 1.f;
    // the previous row's readers of the candidates, bitmap and scratch are done
    csync();
    if (ct == 0) {
      ms->ncand = 0;
      ms->bad = 0;
      ms->cta_max = fkey_i(-INFINITY);
      ms->snap[par] = *reinterpret_cast<volatile int*>(&ms->abort);
    }
    if (x.pen)
      for (int j = ct; j < (P.V + 31) / 32; j += kCutConsumers) bits[j] = 0u;
    csync();
    if (ms->snap[par]) break;            // every consumer warp reads the same snapshot
    if (x.pen) {
      // the row's penalty set: its request's history and the drafts before it
      int h0 = 0, h1 = 0;
      if (P.cu_hist) {
        h0 = __ldg(P.cu_hist + b);
        h1 = __ldg(P.cu_hist + b + 1);
        if (h0 < 0 || h1 < h0) h1 = h0;
      }
      for (int j = h0 + ct; j < h1; j += kCutConsumers) {
        const int t = __ldg(P.hist + j);
        if (t >= 0 && t < P.V) atomicOr(bits + (t >> 5), 1u << (t & 31));
      }
      const int d0 = __ldg(P.cu_draft + b);
      for (int j = ct; j < x.m.i; j += kCutConsumers) {
        const int t = __ldg(P.draft_tokens + d0 + j);
        if (t >= 0 && t < P.V) atomicOr(bits + (t >> 5), 1u << (t & 31));
      }
      csync();
    }
    // ---- the streaming pass
    const float inv_c = 1.f / x.c;     // the candidate bound's margin covers its rounding
    float rt = -INFINITY, st = 0.f;
    bool bad = false;
    for (int ch = 0; ch < nch; ++ch, ++k) {
      const int s = k % kCutSlots;
      (void)cut_wait(full + s, (uint32_t)((k / kCutSlots) & 1), ms);   // an abort drops the row below
      const uint4* slot = reinterpret_cast<const uint4*>(smem + (size_t)s * kCutChunkBytes);
      const int nvec = min(kCutChunkBytes, rb - ch * kCutChunkBytes) / 16;
      const uint4 zero4 = make_uint4(0u, 0u, 0u, 0u);
      const uint4 v0 = ct < nvec ? slot[ct] : zero4;
      const uint4 v1 = ct + kCutConsumers < nvec ? slot[ct + kCutConsumers] : zero4;
      __syncwarp();
      if (lane == 0) mbar_arrive(empty + s);
      const int tok0 = ch * tpc;
      float z[2][8];
      if (!x.pen && tok0 + tpc <= P.V) {
        // the common chunk: every token real, no penalty (NaN and +inf show
        // in the row's mass and maximum, checked once per row)
        Vec<T>::cvt(v0, z[0]);
        Vec<T>::cvt(v1, z[1]);
      } else {
        pen_vec<T>(v0, tok0 + ct * N, x, bits, P.V, z[0], bad);
        pen_vec<T>(v1, tok0 + (ct + kCutConsumers) * N, x, bits, P.V, z[1], bad);
      }
      float zm2[2];
#pragma unroll
      for (int h = 0; h < 2; ++h) {
        float a = fmaxf(z[h][0], z[h][1]), b2 = fmaxf(z[h][2], z[h][3]);
        if constexpr (N == 8) {
          a = fmaxf(a, fmaxf(z[h][4], z[h][5]));
          b2 = fmaxf(b2, fmaxf(z[h][6], z[h][7]));
        }
        zm2[h] = fmaxf(a, b2);
      }
      const float zm = fmaxf(zm2[0], zm2[1]);
      const float vm = __fmul_rn(zm, x.c);      // the chunk's largest z'c (c > 0: the product keeps the order)
      if (ch == 0) {
        // the first chunk's maximum primes the CTA's, so that the first
        // chunk does not take most of its tokens as candidates
        const float wmax = warp_max(vm);
        if (lane == 0 && wmax > -INFINITY) atomicMax(&ms->cta_max, fkey_i(wmax));
        csync();
      }
      if (vm > rt) {
        st *= ex2(rt - vm);
        rt = vm;
      }
      if (rt > -INFINITY) {
        const float nrt = -rt;
        float acc[2] = {0.f, 0.f};
#pragma unroll
        for (int h = 0; h < 2; ++h)
#pragma unroll
          for (int j = 0; j < N; ++j) acc[j & 1] += ex2(fmaf(z[h][j], x.c, nrt));
        st += acc[0] + acc[1];
      } else {
        // nothing above -inf yet in this thread: a NaN would skip the sum
#pragma unroll
        for (int h = 0; h < 2; ++h)
#pragma unroll
          for (int j = 0; j < N; ++j) bad |= z[h][j] != z[h][j];
      }
      // candidates: within the window of the running maximum (this thread's,
      // or the CTA's as the threads have published it; neither exceeds M),
      // tested on z' against a bound a little below thr / c, so that every
      // token with z'c >= thr (as the select computes z'c) is taken
      const float cm = fval_i(*reinterpret_cast<volatile int*>(&ms->cta_max));
      if (rt > cm) atomicMax(&ms->cta_max, fkey_i(rt));
      const float thr = fmaxf(rt, cm) - kCutWindow;
      const float tz = thr * inv_c;
      const float zthr = tz - (fabsf(tz) * 1e-5f + 1e-30f);
      int kt = 0;
#pragma unroll
      for (int h = 0; h < 2; ++h)
#pragma unroll
        for (int j = 0; j < N; ++j) kt += (z[h][j] >= zthr && z[h][j] > -INFINITY) ? 1 : 0;
      if (__ballot_sync(0xffffffffu, kt > 0)) {
        int incl = kt;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
          const int t = __shfl_up_sync(0xffffffffu, incl, o);
          if (lane >= o) incl += t;
        }
        int base = 0;
        if (lane == 31) base = atomicAdd(&ms->ncand, incl);
        base = __shfl_sync(0xffffffffu, base, 31);
        int pos = base + incl - kt;
#pragma unroll
        for (int h = 0; h < 2; ++h)
#pragma unroll
          for (int j = 0; j < N; ++j)
            if (z[h][j] >= zthr && z[h][j] > -INFINITY) {
              if (pos < kCutCand)
                cand[pos] = make_int2(tok0 + (ct + h * kCutConsumers) * N + j, __float_as_int(z[h][j]));
              ++pos;
            }
      }
    }
    // ---- the row's maximum and mass
    float M = rt, S = st;
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
      const float m2 = __shfl_xor_sync(0xffffffffu, M, o), s2 = __shfl_xor_sync(0xffffffffu, S, o);
      ref_merge(M, S, m2, s2);
    }
    if (lane == 0) {
      ms->wM[cw] = M;
      ms->wS[cw] = S;
    }
    if (__any_sync(0xffffffffu, bad) && lane == 0) atomicOr(&ms->bad, 1);
    csync();
    if (ct == 0) ms->snap[par] = *reinterpret_cast<volatile int*>(&ms->abort);
    M = -INFINITY;
    S = 0.f;
    for (int w = 0; w < kCutConsumerWarps; ++w) ref_merge(M, S, ms->wM[w], ms->wS[w]);
    const bool rbad = ms->bad != 0 || !(M > -INFINITY) || !(M < INFINITY) || !(S >= 0.f);
    const int ncand = ms->ncand;
    csync();
    if (ms->snap[par]) break;            // a wait ran out: the row is not recorded
    if (!x.mapped) continue;
    CutRow rec;
    rec.M = M;
    rec.tau = -INFINITY;
    rec.Sk = S;
    rec.n = -1;
    rec.off = 0;
    rec.flags = rbad ? kStatusBadLogits : 0;
    rec.S = S;
    rec.tag = tag32;
    if (x.usable && !rbad && x.tp < 1.f) {
      const double target = (double)x.tp * (double)S;
      bool win = ncand <= kCutCand;
      if (win) win = select_window<T>(P, x, cand, ncand, M, target, hm, hc, bits, ms, ct, cw, lane);
      if (!win) {
        key_levels<T, true>(P, x, cand, ncand, M, target, 0.0, 0, hm, hc, bits, ms, ct, cw, lane,
                            [](float) { return true; });
        rec.flags |= kCutViaRow;
      }
      const unsigned tk = ms->tau_key;
      rec.tau = okey_val(tk);
      rec.Sk = (float)ms->Sk;
      const int nup = ms->n_upper;
      // the kept list, in this CTA's share of the pool (every thread keeps
      // the same count); a set that does not fit is not listed
      if (nup <= kCutListMax && pool_used + nup <= pool_per) {
        const int off = pool0 + pool_used;
        if (ct == 0) ms->nlist = 0;
        csync();
        auto put = [&](int v, float z) {
          if (okey(z) >= tk) {
            const int q = atomicAdd(&ms->nlist, 1);
            if (q < nup) P.pool[off + q] = v;
          }
        };
        if (win) visit<T, false>(P, x, cand, ncand, bits, ct, put);
        else visit<T, true>(P, x, cand, ncand, bits, ct, put);
        csync();
        rec.n = min(ms->nlist, nup);
        rec.off = off;
        pool_used += rec.n;
      }
    }
    if (ct == 0) P.rows[r] = rec;
  }
}

// A CTA whose rows end early (a wait ran out) still takes part in nothing
// else: the finish kernel reports its requests as timed out.
template <typename T>
__global__ void __launch_bounds__(kCutThreads, 1) topp_cut_kernel(const __grid_constant__ ToppParams P) {
  extern __shared__ __align__(128) unsigned char smem[];
  uint64_t* full = reinterpret_cast<uint64_t*>(smem + kOffBars);
  uint64_t* empty = full + kCutSlots;
  CutMisc* ms = reinterpret_cast<CutMisc*>(smem + kOffMisc);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  if (threadIdx.x == 0) {
    for (int s = 0; s < kCutSlots; ++s) {
      mbar_init(full + s, 1);
      mbar_init(empty + s, kCutConsumerWarps);
    }
    ms->abort = 0;
    ms->snap[0] = ms->snap[1] = 0;
    ms->over = 0;
    fence_mbar_init();
  }
  __syncthreads();
  // a cu_draft that is not a valid packing: nothing is read, every request
  // reports SPEC_STATUS_BAD_K
  int bad = 0;
  if (threadIdx.x == 0 && (__ldg(P.cu_draft) != 0 || __ldg(P.cu_draft + P.B) != P.total)) bad = 1;
  for (int b = threadIdx.x; b < P.B; b += blockDim.x)
    if (__ldg(P.cu_draft + b + 1) < __ldg(P.cu_draft + b)) bad = 1;
  if (bad) atomicOr(&ms->over, 1);
  __syncthreads();
  const bool broken = ms->over != 0;
  if (blockIdx.x == 0 && threadIdx.x == 0) *P.broken = (P.tag << 1) | (broken ? 1ull : 0ull);
  if (broken) return;
  if (warp == 0) cut_producer<T>(P, smem, full, empty, ms, lane);
  else cut_consumers<T>(P, smem, full, empty, ms, threadIdx.x - 32, warp - 1, lane);
}

// ------------------------------------------------------------ finish kernel
struct FinMisc {
  double dred[kFinThreads / 32];
  int ired[kFinThreads / 32];
  int st;
  float px, qx;
};

template <typename T>
__device__ __forceinline__ float raw_logit(const ToppParams& P, int src, int v) {
  return to_f32<T>(__ldg(reinterpret_cast<const T*>(logits_row<T>(P, src)) + v));
}

// p~(v) of a token with penalised logit z under its row's record.
__device__ __forceinline__ float kept_prob(float z, const CutRow& R, float c) {
  return z >= R.tau ? __fdiv_rn(ex2(__fmul_rn(z, c) - R.M), R.Sk) : 0.f;
}

__device__ __forceinline__ double fin_sum(double v, FinMisc& fm, int lane, int warp) {
  v = warp_sum_d(v);
  if (lane == 0) fm.dred[warp] = v;
  __syncthreads();
  double t = 0.0;
#pragma unroll
  for (int w = 0; w < kFinThreads / 32; ++w) t += fm.dred[w];
  __syncthreads();
  return t;
}

// What a draw or a sum weighs at token v: p~(v), or max(p~(v) - q~(v), 0)
// with a draft row; z' is the penalised logit under the position's set.
struct Weigh {
  const ToppParams* P;
  CutRow rp, rq;
  int src_p, src_q;     // src_q < 0: weigh p~ alone
  float c, alpha;
  bool pen;
  const uint32_t* pbits;
  template <typename T>
  __device__ __forceinline__ float at(int v) const {
    const bool pv = pen && ((pbits[v >> 5] >> (v & 31)) & 1u);
    float zp = raw_logit<T>(*P, src_p, v);
    if (pv) zp = penalize(zp, alpha);
    const float p = kept_prob(zp, rp, c);
    if (src_q < 0) return p;
    float zq = raw_logit<T>(*P, src_q, v);
    if (pv) zq = penalize(zq, alpha);
    return fmaxf(p - kept_prob(zq, rq, c), 0.f);
  }
};

// Sum of the weights over p's kept tokens (its list, or every token).
template <typename T>
__device__ double weigh_sum(const ToppParams& P, const Weigh& w, FinMisc& fm, int tid, int lane, int warp) {
  double s = 0.0;
  if (w.rp.n >= 0) {
    for (int e = tid; e < w.rp.n; e += kFinThreads) s += (double)w.template at<T>(__ldg(P.pool + w.rp.off + e));
  } else {
    for (int v = tid; v < P.V; v += kFinThreads) s += (double)w.template at<T>(v);
  }
  return fin_sum(s, fm, lane, warp);
}

// Inverse CDF in token-id order over p's kept tokens: the smallest v whose
// inclusive prefix of weights exceeds u * (their sum); the last token with
// weight if rounding leaves none.  Thread t walks the tokens of bitmap
// words [t wpt, (t+1) wpt): the list's tokens (marked in `mark`), or all.
template <typename T>
__device__ int draw_tokens(const ToppParams& P, const Weigh& w, float u, uint32_t* mark, FinMisc& fm, int tid,
                           int lane, int warp) {
  const int W = (P.V + 31) / 32;
  const bool listed = w.rp.n >= 0;
  if (listed) {
    for (int j = tid; j < W; j += kFinThreads) mark[j] = 0u;
    __syncthreads();
    for (int e = tid; e < w.rp.n; e += kFinThreads) {
      const int v = __ldg(P.pool + w.rp.off + e);
      atomicOr(mark + (v >> 5), 1u << (v & 31));
    }
    __syncthreads();
  }
  const int wpt = (W + kFinThreads - 1) / kFinThreads;
  const int w0 = tid * wpt, w1 = min(W, w0 + wpt);
  auto word = [&](int j) -> uint32_t {
    if (listed) return mark[j];
    const int n = P.V - 32 * j;
    return n >= 32 ? 0xffffffffu : ((1u << n) - 1u);
  };
  double loc = 0.0;
  int lastv = -1;
  for (int j = w0; j < w1; ++j)
    for (uint32_t m = word(j); m; m &= m - 1) {
      const int v = 32 * j + __ffs(m) - 1;
      const float x = w.template at<T>(v);
      loc += (double)x;
      if (x > 0.f) lastv = v;
    }
  // exclusive prefix of the threads' sums, and the total
  double incl = warp_incl_scan_d(loc, lane);
  if (lane == 31) fm.dred[warp] = incl;
  int lv = lastv;
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) lv = max(lv, __shfl_xor_sync(0xffffffffu, lv, o));
  if (lane == 0) fm.ired[warp] = lv;
  __syncthreads();
  double base = 0.0, tot = 0.0;
  int last = -1;
  for (int k = 0; k < kFinThreads / 32; ++k) {
    if (k < warp) base += fm.dred[k];
    tot += fm.dred[k];
    last = max(last, fm.ired[k]);
  }
  __syncthreads();
  const double t = (double)u * tot;
  const double excl = base + incl - loc;
  if (tid == 0) fm.st = -1;
  __syncthreads();
  if (excl <= t && t < excl + loc) {
    // this thread's range holds t (the ranges are disjoint); if rounding
    // keeps the walk below t, its last token with weight
    double acc = excl;
    int found = -1;
    for (int j = w0; j < w1 && found < 0; ++j)
      for (uint32_t m = word(j); m; m &= m - 1) {
        const int v = 32 * j + __ffs(m) - 1;
        acc += (double)w.template at<T>(v);
        if (acc > t) {
          found = v;
          break;
        }
      }
    atomicMax(&fm.st, found >= 0 ? found : lastv);
  }
  __syncthreads();
  const int tok = fm.st >= 0 ? fm.st : last;
  __syncthreads();
  return tok;
}

template <typename T>
__global__ void __launch_bounds__(kFinThreads) topp_finish_kernel(const __grid_constant__ ToppParams P) {
  extern __shared__ __align__(16) uint32_t fsm[];
  __shared__ FinMisc fm;
  const int b = blockIdx.x, tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int W = (P.V + 31) / 32;
  uint32_t* pbits = fsm;
  uint32_t* mark = fsm + W;
  const int d0 = __ldg(P.cu_draft + b), d1 = __ldg(P.cu_draft + b + 1);
  const bool rows_ok = d0 >= 0 && d1 >= d0 && d1 <= P.total;
  const int K = d1 - d0, off = d0 + b, base = 2 * d0 + b;
  const bool tv_only = P.mode == kModeTvOnly;
  const unsigned long long bw = __ldcg(P.broken);
  const unsigned tag32 = (unsigned)P.tag;
  if (tid == 0) fm.st = 0;
  __syncthreads();
  int s = 0;
  if ((bw >> 1) != P.tag) {
    s = kStatusTimeout;                 // the row-cut kernel did not run for this call
  } else if (bw & 1ull) {
    s = kStatusBadK;                    // cu_draft is not a valid packing
  } else {
    const float T_ = __ldg(P.temperature + b);
    const float alpha = P.rep_penalty ? __ldg(P.rep_penalty + b) : 1.f;
    const float tp = __ldg(P.top_p + b);
    const float D = __ldg(P.tv_budget + b);
    int h0 = 0, h1 = 0;
    if (P.cu_hist) {
      h0 = __ldg(P.cu_hist + b);
      h1 = __ldg(P.cu_hist + b + 1);
    }
    if (tid == 0) {
      if (K > P.max_k || K > kMaxK) s |= kStatusBadK;
      if (!(T_ > 0.f && T_ < INFINITY && alpha > 0.f && alpha < INFINITY && tp > 0.f && tp <= 1.f && D >= 0.f &&
            D <= 1.f))
        s |= kStatusBadParam;
      if (h0 < 0 || h1 < h0) s |= kStatusBadToken;
    }
    if (h0 >= 0 && h1 >= h0)
      for (int j = h0 + tid; j < h1; j += kFinThreads) {
        const int t = __ldg(P.hist + j);
        if (t < 0 || t >= P.V) s |= kStatusBadToken;
      }
    for (int j = tid; j < K; j += kFinThreads) {
      const int t = __ldg(P.draft_tokens + d0 + j);
      if (t < 0 || t >= P.V) s |= kStatusBadToken;
    }
    for (int j = tid; j <= 2 * K; j += kFinThreads) {
      const CutRow R = P.rows[base + j];
      s |= R.tag != tag32 ? kStatusTimeout : (R.flags & kCutStatusMask);
    }
  }
  if (s) atomicOr(&fm.st, s);
  __syncthreads();
  const int st = fm.st;
  __syncthreads();
  if (st) {
    if (tv_only) {
      if (rows_ok)
        for (int p = d0 + tid; p < d1; p += kFinThreads) {
          P.out_tv[p] = NAN;
          P.out_theta[p] = NAN;
          if (P.out_px) P.out_px[p] = NAN;
          if (P.out_qx) P.out_qx[p] = NAN;
        }
    } else {
      if (rows_ok)
        for (int j = tid; j <= K; j += kFinThreads) P.out_tokens[off + j] = -1;
      if (tid == 0) {
        P.out_accepted[b] = -1;
        if (P.out_status) P.out_status[b] = st;
      }
    }
    return;
  }
  const float c = (float)(1.4426950408889634 / (double)__ldg(P.temperature + b));
  const float alpha = P.rep_penalty ? __ldg(P.rep_penalty + b) : 1.f;
  const bool pen = alpha != 1.f;
  const float D = __ldg(P.tv_budget + b);
  if (pen) {
    for (int j = tid; j < W; j += kFinThreads) pbits[j] = 0u;
    __syncthreads();
    if (P.cu_hist)
      for (int j = __ldg(P.cu_hist + b) + tid; j < __ldg(P.cu_hist + b + 1); j += kFinThreads) {
        const int t = __ldg(P.hist + j);
        atomicOr(pbits + (t >> 5), 1u << (t & 31));
      }
    __syncthreads();
  }
  Weigh w;
  w.P = &P;
  w.c = c;
  w.alpha = alpha;
  w.pen = pen;
  w.pbits = pbits;
  int j = K;
  double Rj = 0.0;
  for (int i = 0; i < K; ++i) {
    w.rp = P.rows[base + 2 * i];
    w.rq = P.rows[base + 2 * i + 1];
    w.src_p = off + i;
    w.src_q = P.NT + d0 + i;
    const int x = __ldg(P.draft_tokens + d0 + i);
    if (tid == 0) {
      const bool pv = pen && ((pbits[x >> 5] >> (x & 31)) & 1u);
      float zp = raw_logit<T>(P, w.src_p, x), zq = raw_logit<T>(P, w.src_q, x);
      if (pv) {
        zp = penalize(zp, alpha);
        zq = penalize(zq, alpha);
      }
      fm.px = kept_prob(zp, w.rp, c);
      fm.qx = kept_prob(zq, w.rq, c);
    }
    const double dsum = weigh_sum<T>(P, w, fm, tid, lane, warp);   // its barriers publish px, qx
    const float px = fm.px, qx = fm.qx;
    const float d = (float)fmin(fmax(dsum, 0.0), 1.0);
    const float theta = d <= D ? 1.f : __fdiv_rn(D, d);
    const float pi = fmaf(theta, qx, (1.f - theta) * px);
    if (tv_only) {
      if (tid == 0) {
        P.out_tv[d0 + i] = d;
        P.out_theta[d0 + i] = theta;
        if (P.out_px) P.out_px[d0 + i] = px;
        if (P.out_qx) P.out_qx[d0 + i] = qx;
      }
    } else if (!(__ldg(P.uniforms + off + i) * qx < pi)) {
      j = i;
      Rj = dsum;
      break;
    }
    // x_i joins the penalty set of the later positions
    __syncthreads();
    if (pen && tid == 0) atomicOr(pbits + (x >> 5), 1u << (x & 31));
    __syncthreads();
  }
  if (tv_only) return;
  const float ufin = __ldg(P.uniforms + off + K);
  int tok = -1;
  if (j < K) {
    // the residual of position j, or p~_j when the residual has no mass
    if (!(Rj > 0.0)) w.src_q = -1;
    tok = draw_tokens<T>(P, w, ufin, mark, fm, tid, lane, warp);
  } else if (!(P.flags & 1u)) {
    w.rp = P.rows[base + 2 * K];
    w.src_p = off + K;
    w.src_q = -1;
    tok = draw_tokens<T>(P, w, ufin, mark, fm, tid, lane, warp);
  }
  for (int s2 = tid; s2 <= K; s2 += kFinThreads) {
    int o = -1;
    if (s2 < j) o = __ldg(P.draft_tokens + d0 + s2);
    else if (s2 == j) o = tok;
    P.out_tokens[off + s2] = o;
  }
  if (tid == 0) {
    P.out_accepted[b] = j;
    if (P.out_status) P.out_status[b] = 0;
  }
}

template <typename T>
int launch_topp_t(const ToppParams& P, int num_sms, cudaStream_t stream) {
  auto cut = topp_cut_kernel<T>;
  auto fin = topp_finish_kernel<T>;
  const int fin_smem = 2 * ((P.V + 31) / 32) * 4;
  if (cudaFuncSetAttribute(cut, cudaFuncAttributeMaxDynamicSharedMemorySize, kCutSmem) != cudaSuccess ||
      cudaFuncSetAttribute(fin, cudaFuncAttributeMaxDynamicSharedMemorySize, fin_smem) != cudaSuccess) {
    cudaGetLastError();
    return -1;
  }
  const int grid = max(1, min(num_sms, P.NR));
  cut<<<grid, kCutThreads, kCutSmem, stream>>>(P);
  fin<<<P.B, kFinThreads, fin_smem, stream>>>(P);
  if (cudaGetLastError() != cudaSuccess) return -1;
  return 0;
}

}  // namespace

int topp_cut_smem_bytes() { return kCutSmem; }

int launch_topp_verify(const ToppParams& P, bool bf16, int num_sms, cudaStream_t stream) {
  return bf16 ? launch_topp_t<__nv_bfloat16>(P, num_sms, stream) : launch_topp_t<float>(P, num_sms, stream);
}

}  // namespace sv
