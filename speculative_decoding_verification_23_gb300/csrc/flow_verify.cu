// Dataflow streaming kernel of mentored speculative sampling without top-p
// ("What I Gave Up to Make Speculative Decoding Faster", section "A knob for
// accepting more draft tokens"), for batches with more work items than SMs.
//
// A work item is one draft position (target row + draft row) or one bonus
// row.  Each of its two passes is cut into tasks of one vocabulary chunk
// (about 15k tokens of each row):
//   pass 1: per consumer warp ("unit") the softmax statistics of its lines,
//           i.e. a reference and the sum of 2^(z'c - ref) per row (z' the
//           penalised logit, c = log2(e)/T), and the draft token's logits;
//   pass 2: per unit the mass of max(p - q, 0) with the item's normalisers.
// One CTA per SM takes tasks from a single global counter in a fixed order:
// pass-1 tasks of item k + lag are interleaved with pass-2 tasks of item k,
// so the whole GPU works on a few dozen items at a time, every SM does the
// same share, and an item's rows are still in L2 when pass 2 reads them.
//
// Warp roles of a CTA:
//   consumers (kFlowConsumers, in groups of kFlowUnits that take alternate
//       slots): one unit of their group's task each;
//   flow warp: claims the next tasks, issues their TMA bulk copies, and
//       counts every finished task for its item (release);
//   two setup warps: a task's penalty bitmap (the request's history bitmap,
//       built by flow_prep_kernel, plus the drafts before the row) and, for
//       pass 2, the item's normalisers, combined from the pass-1 units once
//       the item's pass-1 count is complete;
//   tail warp: the items k = CTA, CTA + grid, ... in pass-1 list order, each
//       once its count is complete.  A position: TV d = total residual mass,
//       theta, p(x), q(x), pi(x), the acceptance decision.  The last item of
//       a request finalises it: first rejection, the inverse-CDF correction
//       (or bonus) searched in the owning unit, the tokens.
// Every wait is bounded; a wait that runs out records SPEC_STATUS_TIMEOUT.

#include "common.cuh"
#include "spec_internal.h"
#include "verify_common.cuh"

namespace sv {

namespace {

constexpr int kNC = kFlowConsumers;
constexpr int kWarpF = kNC;          // flow warp (claims, copies, counts)
constexpr int kWarpS = kNC + 1;      // setup warps kWarpS, kWarpS + 1
constexpr int kWarpT = kNC + 3;      // tail warp
constexpr int kTails = 1;
constexpr int kFlowWarps = kNC + 3 + kTails;
constexpr int kFlowThreads = 32 * kFlowWarps;

extern __shared__ __align__(128) unsigned char flow_smem[];

struct FSmem {
  const FlowLayout& L;
  __device__ __forceinline__ explicit FSmem(const FlowLayout& l) : L(l) {}
  __device__ __forceinline__ unsigned char* slot(int s) const { return flow_smem + L.off_ring + s * L.slot_bytes; }
  __device__ __forceinline__ uint32_t* bm(int s) const {
    return reinterpret_cast<uint32_t*>(flow_smem + L.off_bm + s * L.bm_words * 4);
  }
  __device__ __forceinline__ FlowHdr* hdr(int s) const { return reinterpret_cast<FlowHdr*>(flow_smem + L.off_hdr) + s; }
  __device__ __forceinline__ int* cu() const { return reinterpret_cast<int*>(flow_smem + L.off_cu); }
  __device__ __forceinline__ float* tw(int t) const {
    return reinterpret_cast<float*>(flow_smem + L.off_tw + t * align_up_i(L.nu * 4, 16));
  }
  __device__ __forceinline__ uint64_t* bars() const { return reinterpret_cast<uint64_t*>(flow_smem + L.off_bar); }
  // per slot: flow warp + setup warp -> consumers (task ready, tx bytes
  // landed); flow warp -> setup warp (task claimed); consumers -> flow warp
  // (task done, slot free)
  __device__ __forceinline__ uint64_t* full(int s) const { return bars() + s; }
  __device__ __forceinline__ uint64_t* claim(int s) const { return bars() + kFlowSlots + s; }
  __device__ __forceinline__ uint64_t* done(int s) const { return bars() + 2 * kFlowSlots + s; }
};

template <typename T>
__device__ __forceinline__ T neg_inf_t();
template <>
__device__ __forceinline__ float neg_inf_t<float>() { return -INFINITY; }
template <>
__device__ __forceinline__ __nv_bfloat16 neg_inf_t<__nv_bfloat16>() {
  return __ushort_as_bfloat16((unsigned short)0xFF80u);
}

__device__ __forceinline__ void fence_proxy_async_smem() {
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

__device__ __forceinline__ int atom_add_acq_rel(int* p, int v) {
  int old;
  asm volatile("atom.acq_rel.gpu.global.add.s32 %0, [%1], %2;" : "=r"(old) : "l"(p), "r"(v) : "memory");
  return old;
}

__device__ __forceinline__ int ld_acquire(const int* p) {
  int v;
  asm volatile("ld.acquire.gpu.global.s32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
  return v;
}

__device__ __forceinline__ void red_release_add(int* p, int v) {
  asm volatile("red.release.gpu.global.add.s32 [%0], %1;" ::"l"(p), "r"(v) : "memory");
}

__device__ __forceinline__ void flag_error(const SampleParams& P, int bits) { atomicOr(P.F.ctl + 1, bits); }

// Bounded wait of a whole warp: every lane waits (each lane's own acquire of
// the phase), then the lanes vote, so that a wait that ran out for any lane
// ends the warp's loop in all of them.
__device__ __forceinline__ bool warp_wait(const SampleParams& P, uint64_t* bar, uint32_t parity, bool& to) {
  bool ok = !to && mbar_wait(bar, parity);
  ok = __all_sync(0xffffffffu, ok);
  if (!ok && !to) {
    to = true;
    if ((threadIdx.x & 31) == 0) flag_error(P, kStatusTimeout);
  }
  return ok;
}

// Task s of the fixed sequence.  Pass-1 tasks run over the bonus rows
// first (they need no pass 2, and a request is finalised as soon as its
// last position is decided), then over the draft positions; the first
// `lag` items' pass-1 tasks come alone, then pass-1 tasks of list item
// k + lag alternate with pass-2 tasks of position k, then whatever remains
// of either list.
__device__ __forceinline__ void flow_task(const SampleParams& P, int s, int& type, int& item, int& chunk) {
  const int nck = P.FL.nck;
  const int NA = P.n_items * nck, NB = P.n_p2 * nck;
  const int G = min(P.FL.lag_items * nck, NA);
  int a = -1, bb = -1;
  if (s < G) {
    a = s;
  } else {
    const int t = s - G;
    const int np = min(NA - G, NB);
    if (t < 2 * np) {
      if (t & 1) bb = t >> 1;
      else a = G + (t >> 1);
    } else {
      const int r = t - 2 * np;
      if (NA - G > NB) a = G + np + r;
      else bb = np + r;
    }
  }
  if (a >= 0) {
    type = 1;
    const int k = a / nck;
    chunk = a - k * nck;
    // list order: the n_items - n_p2 bonus rows (items n_p2 ..), then the positions
    const int nb = P.n_items - P.n_p2;
    item = k < nb ? P.n_p2 + k : k - nb;
  } else {
    type = 2;
    item = bb / nck;
    chunk = bb - item * nck;
  }
}

__device__ __forceinline__ int n_tasks(const SampleParams& P) { return (P.n_items + P.n_p2) * P.FL.nck; }

__device__ __forceinline__ const int* cu_of(const SampleParams& P, const FSmem& S) {
  return P.B + 1 <= 1024 ? S.cu() : P.cu_draft;
}

// The work item's request, position and rows (the decoding of pdecode),
// found by the whole warp: the last request b in [0, B) with cu[b] <= item,
// 32 candidates per step.
__device__ __forceinline__ Item pdecode_w(const SampleParams& P, const int* cu, int item, int lane) {
  if (item >= P.total) return pdecode(P, cu, item);
  int lo = 0, hi = P.B;
  while (hi - lo > 1) {
    const int step = (hi - lo + 31) >> 5;
    const int idx = lo + lane * step;
    const unsigned msk = __ballot_sync(0xffffffffu, idx < hi && cu[idx] <= item);
    lo += (msk ? 31 - __clz(msk) : 0) * step;
    hi = min(hi, lo + step);
  }
  Item it;
  it.b = lo;
  it.i = item - cu[lo];
  it.bonus = false;
  it.tgt_row = item + lo;
  it.dft_row = item;
  it.rows_ok = true;
  it.K = cu[lo + 1] - cu[lo];
  return it;
}

// Lines [l0, l1) of the chunk (within the slot) that position wp handles.
__device__ __forceinline__ void unit_lines(int wp, int nlines, int& l0, int& l1) {
  l0 = (wp * nlines) / kFlowUnits;
  l1 = ((wp + 1) * nlines) / kFlowUnits;
}

// ------------------------------------------------------------ flow warp
// A task decoded for its bulk copies.
struct Fill {
  int task;          // -1: no more tasks
  int type, item;
  int tgt_row, dft_row;  // dft_row < 0 for a bonus row
  int lo;
  uint32_t bytes;    // per row
};

template <typename T>
__device__ __forceinline__ Fill decode_fill(const SampleParams& P, const int* cu, int s, int lane) {
  Fill f;
  f.task = -1;
  if (s >= n_tasks(P)) return f;
  f.task = s;
  int chunk;
  flow_task(P, s, f.type, f.item, chunk);
  const Item it = pdecode_w(P, cu, f.item, lane);
  f.tgt_row = it.tgt_row;
  f.dft_row = it.bonus ? -1 : it.dft_row;
  f.lo = chunk * P.FL.lpc;
  const int ntok = min(P.FL.lpc * 256, P.V - f.lo * 256);
  f.bytes = (uint32_t)((ntok * (int)sizeof(T) + 15) & ~15);
  return f;
}

// Claims tasks in sequence order from one global counter (blocks of two,
// the next block claimed ahead), issues their bulk copies into free slots,
// and counts every finished task for its item (a release add: the units it
// wrote are visible to whoever sees the count).  Slots finished meanwhile
// are taken in one batch.
template <typename T>
__device__ void flow_warp(const SampleParams& P, const FSmem& S, int lane) {
  const FlowLayout& L = P.FL;
  const uint64_t keep = l2_policy_evict_last(), drop = l2_policy_evict_first();
  const int* cu = cu_of(P, S);
  bool to = false;
  int stops = 0;  // stop headers written (one for each setup warp)
  // lane 0: claimed tasks [cb, ce) and the next block's claim in flight;
  // all lanes: the decoded next task
  int cb = 0, ce = 0, nb0 = 0;
  if (lane == 0) {
    cb = atomicAdd(P.F.ctl, 2);
    ce = cb + 2;
    nb0 = atomicAdd(P.F.ctl, 2);
  }
  Fill nx = decode_fill<T>(P, cu, __shfl_sync(0xffffffffu, cb, 0), lane);
  // slot n % kFlowSlots gets the next claimed task (or a stop)
  auto fill = [&](int n) {
    const int slot = n % kFlowSlots;
    if (lane == 0) {
      FlowHdr& h = *S.hdr(slot);
      if (nx.task >= 0) {
        h.task = nx.task;
        unsigned char* dst = S.slot(slot);
        // rows read again by pass 2 stay in L2; the rest may go
        const uint64_t pol = (nx.type == 1 && nx.item < P.n_p2) ? keep : drop;
        const bool two = nx.dft_row >= 0;
        mbar_arrive_expect_tx(S.full(slot), two ? 2 * nx.bytes : nx.bytes);
        bulk_g2s(dst, static_cast<const unsigned char*>(P.target) + ((size_t)nx.tgt_row * P.ld_t + (size_t)nx.lo * 256) * sizeof(T),
                 nx.bytes, S.full(slot), pol);
        if (two)
          bulk_g2s(dst + L.row_bytes,
                   static_cast<const unsigned char*>(P.draft) + ((size_t)nx.dft_row * P.ld_d + (size_t)nx.lo * 256) * sizeof(T),
                   nx.bytes, S.full(slot), pol);
        mbar_arrive(S.claim(slot));
        // the next task: claimed ahead, decoded below (off the refill path)
        if (++cb == ce) {
          cb = nb0;
          ce = cb + 2;
          nb0 = atomicAdd(P.F.ctl, 2);
        }
      } else {
        h.task = -1;
        mbar_arrive(S.full(slot));
        mbar_arrive(S.claim(slot));
        ++stops;
      }
    }
    stops = __shfl_sync(0xffffffffu, stops, 0);
    if (nx.task >= 0) nx = decode_fill<T>(P, cu, __shfl_sync(0xffffffffu, cb, 0), lane);
  };
  int nfill = 0;
  while (nfill < kFlowSlots && stops < 2) fill(nfill++);
  for (int n = 0;;) {
    if (!warp_wait(P, S.done(n % kFlowSlots), (uint32_t)(n / kFlowSlots) & 1u, to)) break;
    int nb = 1;
    if (lane == 0)
      while (n + nb < nfill && mbar_test(S.done((n + nb) % kFlowSlots), (uint32_t)((n + nb) / kFlowSlots) & 1u))
        ++nb;
    nb = __shfl_sync(0xffffffffu, nb, 0);
    int task = -1, type = 0, item = 0;
    if (lane < nb) {
      const int slot = (n + lane) % kFlowSlots;
      // this lane's own acquire of the (already completed) phase
      mbar_test(S.done(slot), (uint32_t)((n + lane) / kFlowSlots) & 1u);
      const FlowHdr& h = *S.hdr(slot);
      task = h.task;
      type = h.type;
      item = h.item;
    }
    __syncwarp();
    // refill the finished slots first, then count their tasks
    for (int k = 0; k < nb && stops < 2; ++k) fill(nfill++);
    if (lane < nb && task >= 0) red_release_add(P.F.cnt + (size_t)(type - 1) * P.n_items + item, 1);
    if (__ballot_sync(0xffffffffu, lane < nb && task < 0) || to) break;
    n += nb;
  }
}

// ---------------------------------------------------- item normalisers
__device__ __forceinline__ void combine_pair(float2 v, float& M, float& S) {
  // S is kept relative to M; v = (ref, sum)
  if (v.x > M) {
    S = (M > -INFINITY ? S * ex2(M - v.x) : S) + v.y;
    M = v.x;
  } else {
    S += (v.x > -INFINITY) ? v.y * ex2(v.x - M) : v.y;
  }
}

// An item's pass-1 statistics from its unit records, warp-wide, in one
// fixed order (so every caller gets the same bits): per row the reference
// M (units of z'c) and 1/S; ok is false for logits that are NaN or +inf or
// leave no mass.  rows = 1 (bonus) leaves the draft row at (0, 1).
__device__ __forceinline__ bool item_norms(const SampleParams& P, int item, int rows, int lane, float& M0, float& i0,
                                           float& M1, float& i1) {
  const float4* rec = P.F.p1 + (size_t)item * P.FL.nu;
  constexpr int kPer = 8;
  float4 r[kPer];
#pragma unroll
  for (int q = 0; q < kPer; ++q)
    r[q] = lane + 32 * q < P.FL.nu ? __ldcg(rec + lane + 32 * q) : make_float4(-INFINITY, 0.f, -INFINITY, 0.f);
  float S0 = 0.f, S1 = 0.f;
  M0 = -INFINITY;
  M1 = -INFINITY;
#pragma unroll
  for (int q = 0; q < kPer; ++q) {
    combine_pair(make_float2(r[q].x, r[q].y), M0, S0);
    combine_pair(make_float2(r[q].z, r[q].w), M1, S1);
  }
  for (int u = lane + 32 * kPer; u < P.FL.nu; u += 32) {
    const float4 rr = __ldcg(rec + u);
    combine_pair(make_float2(rr.x, rr.y), M0, S0);
    combine_pair(make_float2(rr.z, rr.w), M1, S1);
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
    const float a = __shfl_xor_sync(0xffffffffu, M0, o), b = __shfl_xor_sync(0xffffffffu, S0, o);
    const float c = __shfl_xor_sync(0xffffffffu, M1, o), d = __shfl_xor_sync(0xffffffffu, S1, o);
    combine_pair(make_float2(a, b), M0, S0);
    combine_pair(make_float2(c, d), M1, S1);
  }
  M0 = __shfl_sync(0xffffffffu, M0, 0);
  S0 = __shfl_sync(0xffffffffu, S0, 0);
  M1 = __shfl_sync(0xffffffffu, M1, 0);
  S1 = __shfl_sync(0xffffffffu, S1, 0);
  bool ok = (S0 > 0.f) && (S0 < INFINITY) && (M0 < INFINITY);
  if (rows == 2) ok = ok && (S1 > 0.f) && (S1 < INFINITY) && (M1 < INFINITY);
  i0 = ok ? __fdiv_rn(1.f, S0) : 1.f;
  i1 = ok && rows == 2 ? __fdiv_rn(1.f, S1) : 1.f;
  if (!ok) M0 = 0.f;
  if (!ok || rows != 2) M1 = 0.f;
  return ok;
}

// ---------------------------------------------------------------- setup
// Everything a task's consumers need besides the rows: the slot's penalty
// bitmap and, for pass 2, the item's normalisers.  The global loads of a
// task (scalars, bitmap words, earlier drafts, normalisers) are issued
// together.
template <typename T>
__device__ void setup(const SampleParams& P, const FSmem& S, int j, int lane) {
  const FlowLayout& L = P.FL;
  const int* cu = cu_of(P, S);
  bool to = false;
  for (int n = j;; n += 2) {
    const int slot = n % kFlowSlots;
    if (!warp_wait(P, S.claim(slot), (uint32_t)(n / kFlowSlots) & 1u, to)) break;
    FlowHdr& h = *S.hdr(slot);
    const int s = h.task;
    if (s < 0) {
      __syncwarp();
      if (lane == 0) mbar_arrive(S.full(slot));
      break;
    }
    int type, item, chunk;
    flow_task(P, s, type, item, chunk);
    const Item it = pdecode_w(P, cu, item, lane);
    const int lo = chunk * L.lpc;
    const int nl = min(L.lpc, L.nlines - lo);
    const int t0 = lo * 256, t1 = (lo + nl) * 256;
    // loads that need nothing but the task
    const uint4* src = reinterpret_cast<const uint4*>(P.F.hbm + (size_t)it.b * P.F.hbm_words + (size_t)lo * 8);
    uint4 wv[4];
#pragma unroll
    for (int q = 0; q < 4; ++q)
      wv[q] = (lane + 32 * q < 2 * nl) ? __ldg(src + lane + 32 * q) : make_uint4(0u, 0u, 0u, 0u);
    const int d0 = cu[it.b];
    const int npre = it.bonus ? (it.rows_ok ? it.K : 0) : it.i;
    const int ptok = lane < npre ? __ldg(P.draft_tokens + d0 + lane) : -1;
    const Scalars sc = item_scalars(P, it, item, cu);
    if (sc.pen) {
      uint32_t* bm = S.bm(slot);
      const bool hist = sc.h1 > sc.h0;
#pragma unroll
      for (int q = 0; q < 4; ++q)
        if (lane + 32 * q < 2 * nl) reinterpret_cast<uint4*>(bm)[lane + 32 * q] = hist ? wv[q] : make_uint4(0u, 0u, 0u, 0u);
      for (int q = lane + 128; q < 2 * nl; q += 32)
        reinterpret_cast<uint4*>(bm)[q] = hist ? __ldg(src + q) : make_uint4(0u, 0u, 0u, 0u);
      __syncwarp();
      if (ptok >= t0 && ptok < t1 && ptok < P.V) atomicOr(&bm[(ptok - t0) >> 5], 1u << (ptok & 31));
      for (int q = lane + 32; q < npre; q += 32) {
        const int tok = __ldg(P.draft_tokens + d0 + q);
        if (tok >= t0 && tok < t1 && tok < P.V) atomicOr(&bm[(tok - t0) >> 5], 1u << (tok & 31));
      }
    }
    float4 a = make_float4(0.f, 1.f, 0.f, 1.f);
    if (type == 2) {
      // the item's normalisers, once all its pass-1 tasks are counted
      int late = 0;
      if (lane == 0) {
        const int* c1 = P.F.cnt + item;
        const long long t0c = clock64();
        while (ld_acquire(c1) < L.nck) {
          if (clock64() - t0c > kWaitLimitCycles) {
            late = 1;
            flag_error(P, kStatusTimeout);
            break;
          }
        }
      }
      if (__shfl_sync(0xffffffffu, late, 0)) to = true;
      __syncwarp();
      item_norms(P, item, 2, lane, a.x, a.y, a.z, a.w);
    }
    if (lane == 0) {
      h.type = type;
      h.item = item;
      h.chunk = chunk;
      h.lo_line = lo;
      h.nlines = nl;
      h.nrows = sc.nrows;
      h.pen = sc.pen ? 1 : 0;
      h.x = sc.x;
      h.c = sc.c;
      h.alpha = sc.alpha;
      h.Mt = a.x;
      h.it = a.y;
      h.Md = a.z;
      h.id = a.w;
    }
    __syncwarp();
    if (lane == 0) mbar_arrive(S.full(slot));
    if (to) break;
  }
}

// ------------------------------------------------------------ consumers
// One 256-token line of a staged row as 8 fp32 values per lane: bf16 lane l
// holds tokens 8l..8l+7; fp32 lane l holds 4l..4l+3 and 128+4l..128+4l+3.
template <typename T>
__device__ __forceinline__ void line_vals(const unsigned char* row, int line, int lane, float (&z)[8]) {
  if constexpr (sizeof(T) == 2) {
    const uint4 v = *reinterpret_cast<const uint4*>(row + line * 512 + lane * 16);
    z[0] = __uint_as_float(v.x << 16);
    z[1] = __uint_as_float(v.x & 0xffff0000u);
    z[2] = __uint_as_float(v.y << 16);
    z[3] = __uint_as_float(v.y & 0xffff0000u);
    z[4] = __uint_as_float(v.z << 16);
    z[5] = __uint_as_float(v.z & 0xffff0000u);
    z[6] = __uint_as_float(v.w << 16);
    z[7] = __uint_as_float(v.w & 0xffff0000u);
  } else {
    const uint4 a = *reinterpret_cast<const uint4*>(row + line * 1024 + lane * 16);
    const uint4 b = *reinterpret_cast<const uint4*>(row + line * 1024 + 512 + lane * 16);
    z[0] = __uint_as_float(a.x);
    z[1] = __uint_as_float(a.y);
    z[2] = __uint_as_float(a.z);
    z[3] = __uint_as_float(a.w);
    z[4] = __uint_as_float(b.x);
    z[5] = __uint_as_float(b.y);
    z[6] = __uint_as_float(b.z);
    z[7] = __uint_as_float(b.w);
  }
}

template <typename T>
__device__ __forceinline__ int line_tok(int lane, int e) {
  if constexpr (sizeof(T) == 2) return 8 * lane + e;
  else return e < 4 ? 4 * lane + e : 128 + 4 * lane + (e - 4);
}

// Tokens at or past V (the row's last line) become -inf.
template <typename T>
__device__ __forceinline__ void mask_line(float (&z)[8], int line_tok0, int lane, int V) {
#pragma unroll
  for (int e = 0; e < 8; ++e)
    if (line_tok0 + line_tok<T>(lane, e) >= V) z[e] = -INFINITY;
}

__device__ __forceinline__ float2 exp_sum8(const float (&z)[8], float2 c2, float2 nr, float2 acc) {
#pragma unroll
  for (int e = 0; e < 8; e += 2) {
    const float2 y = __ffma2_rn(make_float2(z[e], z[e + 1]), c2, nr);
    acc = __fadd2_rn(acc, make_float2(ex2(y.x), ex2(y.y)));
  }
  return acc;
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

__device__ __forceinline__ void combine_into(float2 v, float& M, float& S) {
  // S is kept relative to M; v = (ref, sum)
  if (v.x > M) {
    S = (M > -INFINITY ? S * ex2(M - v.x) : S) + v.y;
    M = v.x;
  } else {
    S += (v.x > -INFINITY) ? v.y * ex2(v.x - M) : v.y;
  }
}

// (reference, sum) of a warp from its lanes'.
__device__ __forceinline__ float2 warp_combine(float ref, float s) {
  const float M = warp_max(ref);
  const float t = (ref > -INFINITY) ? s * ex2(ref - M) : s;
  return make_float2(M, warp_sum(t));
}

// A lane's (reference, sum) of one row over lines [l0, l1), recomputed from
// its maximum (the slow path of a unit whose sums left the fp32 range).
template <typename T>
__device__ __noinline__ float2 lane_stats_exact(const unsigned char* row, int l0, int l1, int lane, int tok0, int V,
                                                float c) {
  float mx = -INFINITY;
  for (int ln = l0; ln < l1; ++ln) {
    float z[8];
    line_vals<T>(row, ln, lane, z);
    mask_line<T>(z, tok0 + (ln - l0) * 256, lane, V);
    for (int e = 0; e < 8; ++e) mx = fmaxf(mx, z[e]);
  }
  if (!(mx > -INFINITY)) return make_float2(-INFINITY, 0.f);
  const float ref = mx * c;
  float2 acc = make_float2(0.f, 0.f);
  for (int ln = l0; ln < l1; ++ln) {
    float z[8];
    line_vals<T>(row, ln, lane, z);
    mask_line<T>(z, tok0 + (ln - l0) * 256, lane, V);
    acc = exp_sum8(z, make_float2(c, c), make_float2(-ref, -ref), acc);
  }
  return make_float2(ref, acc.x + acc.y);
}

// Calls f(o) for every penalised position o (offset within the chunk) of
// lines [l0, l1): lane l takes bitmap words l, l + 32, ... of the lines and
// their set bits one by one (a word rarely holds more than one).  Returns
// whether there were any.
template <typename F>
__device__ __forceinline__ bool for_penalised(const uint32_t* bm, int l0, int l1, int lane, F&& f) {
  const int w1 = l1 * 8;
  bool any = false;
  for (int wb = l0 * 8; wb < w1; wb += 32) {
    uint32_t w = wb + lane < w1 ? bm[wb + lane] : 0u;
    if (!__any_sync(0xffffffffu, w != 0u)) continue;
    any = true;
    while (w) {
      f((wb + lane) * 32 + __ffs(w) - 1);
      w &= w - 1;
    }
  }
  return any;
}

// Pass 1 of one unit: per row the warp's (reference, sum) into p1[item][unit].
// The reference is the warp's maximum over its first line (units of z'c);
// a sum that leaves the fp32 range (or a first line without a finite value)
// sends the unit through the exact per-lane path.
template <typename T>
__device__ __forceinline__ void pass1_unit(const SampleParams& P, const FlowHdr& h, unsigned char* base,
                                           const uint32_t* bm, int l0, int l1, int unit, int lane) {
  const FlowLayout& L = P.FL;
  const int nr = h.nrows;
  unsigned char* row0 = base;
  unsigned char* row1 = base + L.row_bytes;
  const int tok0 = (h.lo_line + l0) * 256;      // first token of the unit
  const int tok1 = min((h.lo_line + l1) * 256, P.V);
  const float c = h.c;
  float pref[2] = {-INFINITY, -INFINITY}, psum[2] = {0.f, 0.f};
  bool bad = false;
  if (h.x >= tok0 && h.x < tok1) {
    // the draft token's raw logits, before any patch
    if (lane == 0) {
      const int o = h.x - h.lo_line * 256;
      P.F.xz[h.item] = make_float2(to_f32<T>(reinterpret_cast<const T*>(row0)[o]),
                                   to_f32<T>(reinterpret_cast<const T*>(row1)[o]));
    }
    __syncwarp();
  }
  if (h.pen) {
    // penalised positions: their exact softmax terms, then out of the stream
    bool wrote = false;
    const float alpha = h.alpha;
    const bool any = for_penalised(bm, l0, l1, lane, [&](int o) {
      T* pp = reinterpret_cast<T*>(row0) + o;
      T* qq = reinterpret_cast<T*>(row1) + o;
      const float zp = to_f32<T>(*pp);
      const float zq = nr == 2 ? to_f32<T>(*qq) : 0.f;
      if (is_bad_logit(zp) || (nr == 2 && is_bad_logit(zq))) bad = true;
      const float yp = penalize(zp, alpha) * c;
      const float yq = penalize(zq, alpha) * c;
      *pp = neg_inf_t<T>();
      if (nr == 2) *qq = neg_inf_t<T>();
      online_add(yp, pref[0], psum[0]);
      if (nr == 2) online_add(yq, pref[1], psum[1]);
      wrote = true;
    });
    if (any) {
      if (wrote) fence_proxy_async_smem();
      __syncwarp();
    }
  }
  float M[2] = {-INFINITY, -INFINITY}, Sw[2] = {0.f, 0.f};
  if (l1 > l0) {
    const bool tail = tok0 + (l1 - l0) * 256 > P.V;  // the unit holds the row's last, partial line
    const float2 c2 = make_float2(c, c);
    float zt[8], zd[8];
    line_vals<T>(row0, l0, lane, zt);
    if (nr == 2) line_vals<T>(row1, l0, lane, zd);
    if (tail && l1 - l0 == 1) {
      mask_line<T>(zt, tok0, lane, P.V);
      if (nr == 2) mask_line<T>(zd, tok0, lane, P.V);
    }
    float m0 = max8(zt), m1 = nr == 2 ? max8(zd) : -INFINITY;
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
      m0 = fmaxf(m0, __shfl_xor_sync(0xffffffffu, m0, o));
      m1 = fmaxf(m1, __shfl_xor_sync(0xffffffffu, m1, o));
    }
    M[0] = m0 * c;
    M[1] = m1 * c;
    const float2 n0 = make_float2(-M[0], -M[0]), n1 = make_float2(-M[1], -M[1]);
    float2 a0 = exp_sum8(zt, c2, n0, make_float2(0.f, 0.f));
    float2 a1 = make_float2(0.f, 0.f);
    if (nr == 2) {
      a1 = exp_sum8(zd, c2, n1, a1);
#pragma unroll 2
      for (int ln = l0 + 1; ln < l1; ++ln) {
        line_vals<T>(row0, ln, lane, zt);
        line_vals<T>(row1, ln, lane, zd);
        if (tail && ln == l1 - 1) {
          mask_line<T>(zt, tok0 + (ln - l0) * 256, lane, P.V);
          mask_line<T>(zd, tok0 + (ln - l0) * 256, lane, P.V);
        }
        a0 = exp_sum8(zt, c2, n0, a0);
        a1 = exp_sum8(zd, c2, n1, a1);
      }
    } else {
#pragma unroll 2
      for (int ln = l0 + 1; ln < l1; ++ln) {
        line_vals<T>(row0, ln, lane, zt);
        if (tail && ln == l1 - 1) mask_line<T>(zt, tok0 + (ln - l0) * 256, lane, P.V);
        a0 = exp_sum8(zt, c2, n0, a0);
      }
    }
    float r0 = a0.x + a0.y, r1 = a1.x + a1.y;
    if (pref[0] > -INFINITY) r0 += psum[0] * ex2(pref[0] - M[0]);
    if (pref[1] > -INFINITY) r1 += psum[1] * ex2(pref[1] - M[1]);
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
      r0 += __shfl_xor_sync(0xffffffffu, r0, o);
      r1 += __shfl_xor_sync(0xffffffffu, r1, o);
    }
    Sw[0] = r0;
    Sw[1] = r1;
    // out of range or NaN (a first line without a finite value, an extreme
    // spread of logits within the unit, or invalid logits): per-lane
    // references from each lane's maximum
#pragma unroll
    for (int r = 0; r < 2; ++r) {
      if (r < nr && !(Sw[r] < INFINITY)) {
        const float2 e = lane_stats_exact<T>(r ? row1 : row0, l0, l1, lane, tok0, P.V, c);
        float Ml = e.x, Sl = e.y;
        combine_into(make_float2(pref[r], psum[r]), Ml, Sl);
        const float2 wv = warp_combine(Ml, Sl);
        M[r] = wv.x;
        Sw[r] = wv.y;
      }
    }
    if (nr != 2) {
      M[1] = -INFINITY;
      Sw[1] = 0.f;
    }
  }
  if (__any_sync(0xffffffffu, bad)) Sw[0] = NAN;
  if (lane == 0) __stcg(P.F.p1 + (size_t)h.item * L.nu + unit, make_float4(M[0], Sw[0], M[1], Sw[1]));
}

__device__ __forceinline__ float prob_of(float z, float c, float M, float inv) {
  return __fmul_rn(ex2(fmaf(z, c, -M)), inv);
}
__device__ __forceinline__ float resid_of(float p, float q) { return fmaxf(fmaf(q, -1.f, p), 0.f); }

// Residual mass max(p-q, 0) of the 8 values of one line (bit-identical to
// prob_of / resid_of element by element).
__device__ __forceinline__ float2 resid_sum8(const float (&zt)[8], const float (&zd)[8], float2 c2, float2 nmt,
                                             float2 nmd, float2 it2, float2 id2, float2 acc) {
  const float2 m1 = make_float2(-1.f, -1.f);
#pragma unroll
  for (int e = 0; e < 8; e += 2) {
    const float2 yp = __ffma2_rn(make_float2(zt[e], zt[e + 1]), c2, nmt);
    const float2 yq = __ffma2_rn(make_float2(zd[e], zd[e + 1]), c2, nmd);
    const float2 p = __fmul2_rn(make_float2(ex2(yp.x), ex2(yp.y)), it2);
    const float2 q = __fmul2_rn(make_float2(ex2(yq.x), ex2(yq.y)), id2);
    const float2 d = __ffma2_rn(q, m1, p);
    acc = __fadd2_rn(acc, make_float2(fmaxf(d.x, 0.f), fmaxf(d.y, 0.f)));
  }
  return acc;
}

// Pass 2 of one unit (draft positions only): its residual mass into p2[item][unit].
template <typename T>
__device__ __forceinline__ void pass2_unit(const SampleParams& P, const FlowHdr& h, unsigned char* base,
                                           const uint32_t* bm, int l0, int l1, int unit, int lane) {
  const FlowLayout& L = P.FL;
  unsigned char* row0 = base;
  unsigned char* row1 = base + L.row_bytes;
  const int tok0 = (h.lo_line + l0) * 256;
  const float c = h.c, Mt = h.Mt, it = h.it, Md = h.Md, id = h.id;
  float extra = 0.f;
  if (h.pen) {
    bool wrote = false;
    const float alpha = h.alpha;
    const bool any = for_penalised(bm, l0, l1, lane, [&](int o) {
      T* pp = reinterpret_cast<T*>(row0) + o;
      T* qq = reinterpret_cast<T*>(row1) + o;
      const float zp = to_f32<T>(*pp), zq = to_f32<T>(*qq);
      const float p = prob_of(penalize(zp, alpha), c, Mt, it);
      const float q = prob_of(penalize(zq, alpha), c, Md, id);
      *pp = neg_inf_t<T>();
      *qq = neg_inf_t<T>();
      extra += resid_of(p, q);
      wrote = true;
    });
    if (any) {
      if (wrote) fence_proxy_async_smem();
      __syncwarp();
    }
  }
  const bool tail = tok0 + (l1 - l0) * 256 > P.V;
  const float2 c2 = make_float2(c, c), nmt = make_float2(-Mt, -Mt), nmd = make_float2(-Md, -Md);
  const float2 it2 = make_float2(it, it), id2 = make_float2(id, id);
  float2 acc = make_float2(0.f, 0.f);
#pragma unroll 2
  for (int ln = l0; ln < l1; ++ln) {
    float zt[8], zd[8];
    line_vals<T>(row0, ln, lane, zt);
    line_vals<T>(row1, ln, lane, zd);
    if (tail && ln == l1 - 1) {
      mask_line<T>(zt, tok0 + (ln - l0) * 256, lane, P.V);
      mask_line<T>(zd, tok0 + (ln - l0) * 256, lane, P.V);
    }
    acc = resid_sum8(zt, zd, c2, nmt, nmd, it2, id2, acc);
  }
  const float m = warp_sum(acc.x + acc.y + extra);
  if (lane == 0) __stcg(P.F.p2 + (size_t)h.item * L.nu + unit, m);
}

template <typename T>
__device__ void consumer(const SampleParams& P, const FSmem& S, int w, int lane) {
  bool to = false;
  const int g = w / kFlowUnits, wg = w % kFlowUnits;
  for (int n = g;; n += kFlowConsumers / kFlowUnits) {
    const int slot = n % kFlowSlots;
    if (!warp_wait(P, S.full(slot), (uint32_t)(n / kFlowSlots) & 1u, to)) break;
    const FlowHdr& h = *S.hdr(slot);
    if (h.task < 0) {
      __syncwarp();
      if (lane == 0) mbar_arrive(S.done(slot));
      break;
    }
    // the position rotates with the chunk so that the longer units spread
    // over all warps of the group
    const int wp = (wg + h.chunk) % kFlowUnits;
    int l0, l1;
    unit_lines(wp, h.nlines, l0, l1);
    const int unit = h.chunk * kFlowUnits + wp;
    if (h.type == 1) pass1_unit<T>(P, h, S.slot(slot), S.bm(slot), l0, l1, unit, lane);
    else pass2_unit<T>(P, h, S.slot(slot), S.bm(slot), l0, l1, unit, lane);
    __syncwarp();
    if (lane == 0) mbar_arrive(S.done(slot));
  }
}

// ------------------------------------------------------------ tail jobs
// Records one item's status; the last item of its request to finish
// finalises the request.
template <typename T>
__device__ void request_done(const SampleParams& P, const FSmem& S, int t, const Item& it, int item, int flags,
                             int lane);

// What both kinds of item job need: scalars, the status bits of the item
// (tokens, parameters, logits) and the normalisers.
struct ItemInfo {
  Item it;
  Scalars sc;
  int d0, npre, ptok;  // earlier drafts: lane q < npre holds draft q (ptok)
  float M0, i0, M1, i1;
  float2 xz;
  int flags;
  bool ok;
};

__device__ __forceinline__ ItemInfo item_info(const SampleParams& P, const int* cu, int item, int lane) {
  ItemInfo f;
  f.it = pdecode_w(P, cu, item, lane);
  f.d0 = cu[f.it.b];
  f.npre = f.it.bonus ? (f.it.rows_ok ? f.it.K : 0) : f.it.i;
  // loads that need only the item, issued together
  f.ptok = lane < f.npre ? __ldg(P.draft_tokens + f.d0 + lane) : -1;
  const int rfl = __ldcg(P.F.rflags + f.it.b);
  f.xz = f.it.bonus ? make_float2(0.f, 0.f) : __ldcg(P.F.xz + item);
  f.sc = item_scalars(P, f.it, item, cu);
  f.ok = item_norms(P, item, f.sc.nrows, lane, f.M0, f.i0, f.M1, f.i1);
  int fl = (lane < f.npre && (f.ptok < 0 || f.ptok >= P.V)) ? kStatusBadToken : 0;
  for (int q = lane + 32; q < f.npre; q += 32) {
    const int tok = __ldg(P.draft_tokens + f.d0 + q);
    if (tok < 0 || tok >= P.V) fl |= kStatusBadToken;
  }
  f.flags = f.sc.flags | rfl | (f.ok ? 0 : kStatusBadLogits) | warp_or(fl);
  return f;
}

// A position's p(x) and q(x) (x may be penalised itself).
__device__ __forceinline__ void item_pq(const SampleParams& P, const ItemInfo& f, int lane, float& px, float& qx) {
  px = 0.f;
  qx = 0.f;
  const Scalars& sc = f.sc;
  if (f.it.bonus || sc.x < 0 || sc.x >= P.V || !f.ok) return;
  bool in = sc.pen && __any_sync(0xffffffffu, lane < f.npre && f.ptok == sc.x);
  for (int q = lane + 32; q < f.npre; q += 32) in |= __ldg(P.draft_tokens + f.d0 + q) == sc.x;
  if (sc.pen && sc.h1 > sc.h0) in |= (__ldg(P.F.hbm + (size_t)sc.b * P.F.hbm_words + (sc.x >> 5)) >> (sc.x & 31)) & 1u;
  const bool xpen = sc.pen && __any_sync(0xffffffffu, in);
  px = prob_of(xpen ? penalize(f.xz.x, sc.alpha) : f.xz.x, sc.c, f.M0, f.i0);
  qx = prob_of(xpen ? penalize(f.xz.y, sc.alpha) : f.xz.y, sc.c, f.M1, f.i1);
}

// Records one item's status; the last item of its request to finish
// finalises the request.
template <typename T>
__device__ void request_done(const SampleParams& P, const FSmem& S, const Item& it, int item, int flags, int lane);

// A bonus row: its status, then the request's count.
template <typename T>
__device__ void bonus_job(const SampleParams& P, const FSmem& S, int item, int lane) {
  const ItemInfo f = item_info(P, cu_of(P, S), item, lane);
  request_done<T>(P, S, f.it, item, f.flags, lane);
}

// A draft position: TV d, theta, pi(x), the acceptance decision (or, in
// TV-only mode, the outputs).
template <typename T>
__device__ void p2_job(const SampleParams& P, const FSmem& S, int item, int lane) {
  const FlowLayout& L = P.FL;
  double r = 0.0;
  for (int u = lane; u < L.nu; u += 32) r += (double)__ldcg(P.F.p2 + (size_t)item * L.nu + u);
  const ItemInfo f = item_info(P, cu_of(P, S), item, lane);
  const Scalars& sc = f.sc;
  float px, qx;
  item_pq(P, f, lane, px, qx);
  const int flags = f.flags;
  const double R = warp_sum_d(r);
  const double tv = fmin(R, 1.0);
  double theta = 1.0;
  if (tv > (double)sc.D) theta = (double)__fdiv_rn(sc.D, (float)tv);
  const double pi = (1.0 - theta) * (double)px + theta * (double)qx;
  if (P.mode != kModeSample) {
    if (lane == 0) {
      const bool bad = flags != 0;
      P.out_tv[item] = bad ? NAN : (float)tv;
      if (P.out_theta) P.out_theta[item] = bad ? NAN : (float)theta;
      if (P.out_px) P.out_px[item] = bad ? NAN : px;
      if (P.out_qx) P.out_qx[item] = bad ? NAN : qx;
    }
    return;
  }
  const float u_acc = sc.uniforms_ok ? __ldg(P.uniforms + sc.off + f.it.i) : 0.f;
  const int acc = ((double)u_acc * (double)qx < pi) ? 1 : 0;
  if (lane == 0) {
    ItemResult* res = P.results + item;
    res->acc = acc;
    res->cand = -1;
    res->tv = (float)tv;
    res->theta = (float)theta;
    res->px = px;
    res->qx = qx;
    res->pad[0] = __float_as_int((float)R);
  }
  request_done<T>(P, S, f.it, item, flags, lane);
}

// Warp-wide owner search over per-unit masses seg[0..n) (fp64 blocks of
// consecutive units per lane, then a lane scan): the first unit with mass
// whose inclusive prefix exceeds t = u * total, and t minus the prefix
// before it; if rounding leaves t out of reach, the last unit with mass
// (take_last).  Returns the total mass.
__device__ __forceinline__ double owner_search(const float* seg, int n, double u, int lane, int& ks, double& rem,
                                               bool& take_last) {
  int k0, k1;
  double blk, inc;
  const double R = seg_block_scan(seg, n, lane, k0, k1, blk, inc);
  const double t = u * R;
  ks = -1;
  rem = 0.0;
  take_last = false;
  const unsigned mh = __ballot_sync(0xffffffffu, blk > 0.0 && inc > t);
  if (mh) {
    const int L0 = __ffs(mh) - 1;
    int kk = -1;
    double rr = 0.0;
    bool tl = false;
    if (lane == L0) {
      double cum = inc - blk;
      int klast = -1;
      for (int k = k0; k < k1; ++k) {
        const double sg = (double)seg[k];
        if (sg > 0.0) {
          if (cum + sg > t) {
            kk = k;
            rr = t - cum;
            break;
          }
          klast = k;
        }
        cum += sg;
      }
      if (kk < 0) {
        kk = klast;
        tl = true;
      }
    }
    ks = __shfl_sync(0xffffffffu, kk, L0);
    rem = __shfl_sync(0xffffffffu, rr, L0);
    take_last = __shfl_sync(0xffffffffu, (int)tl, L0) != 0;
  }
  if (ks < 0) {
    const unsigned mp = __ballot_sync(0xffffffffu, blk > 0.0);
    if (mp) {
      const int L1 = 31 - __clz(mp);
      int kl = -1;
      if (lane == L1)
        for (int k = k1 - 1; k >= k0; --k)
          if (seg[k] > 0.f) {
            kl = k;
            break;
          }
      ks = __shfl_sync(0xffffffffu, kl, L1);
    }
    take_last = true;
  }
  return R;
}

// Inverse CDF within tokens [t0, t1) of an item's rows (warp-wide): the
// first token whose inclusive prefix of w exceeds rem, w = max(p-q, 0) or p
// (ponly); with take_last, or if rounding leaves no such token, the last
// token with w > 0.  Lane l takes LT consecutive tokens of each piece of
// 32*LT.  Returns -1 if the range has no mass.
template <typename T>
__device__ int search_range(const SampleParams& P, const Scalars& sc, const T* gp, const T* gq, bool ponly, int t0,
                            int t1, double rem, bool take_last, float Mt, float it, float Md, float id, int lane) {
  constexpr int N = 16 / (int)sizeof(T);
  constexpr int LT = 4 * N;  // 32 (bf16) or 16 (fp32) tokens per lane
  const int xl = (lane < sc.npre && sc.pen) ? __ldg(P.draft_tokens + sc.d0 + lane) : -1;
  const bool hist = sc.pen && sc.h1 > sc.h0;
  const uint32_t* hb = P.F.hbm + (size_t)sc.b * P.F.hbm_words;
  int found = -1, last_any = -1;
  double cum = 0.0;
  for (int base0 = t0; base0 < t1; base0 += 32 * LT) {
    const int base = base0 + lane * LT;
    uint32_t pm = 0;
    if (sc.pen) {
      if (hist && base < t1) {
        const uint32_t wv = __ldg(hb + (base >> 5));
        pm = LT == 32 ? wv : (wv >> (base & 31)) & ((1u << LT) - 1u);
      }
      for (int q = 0; q < sc.npre && q < 32; ++q) {
        const int tok = __shfl_sync(0xffffffffu, xl, q);
        if (tok >= base && tok < base + LT) pm |= 1u << (tok - base);
      }
    }
    float w[LT];
    float ls = 0.f;
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      const bool in = base + j * N < t1;
      const uint4 vp = in ? __ldg(reinterpret_cast<const uint4*>(gp + base + j * N)) : make_uint4(0u, 0u, 0u, 0u);
      const uint4 vq = (in && !ponly) ? __ldg(reinterpret_cast<const uint4*>(gq + base + j * N))
                                      : make_uint4(0u, 0u, 0u, 0u);
      float zp[8], zq[8];
      if constexpr (N == 8) {
        zp[0] = __uint_as_float(vp.x << 16); zp[1] = __uint_as_float(vp.x & 0xffff0000u);
        zp[2] = __uint_as_float(vp.y << 16); zp[3] = __uint_as_float(vp.y & 0xffff0000u);
        zp[4] = __uint_as_float(vp.z << 16); zp[5] = __uint_as_float(vp.z & 0xffff0000u);
        zp[6] = __uint_as_float(vp.w << 16); zp[7] = __uint_as_float(vp.w & 0xffff0000u);
        zq[0] = __uint_as_float(vq.x << 16); zq[1] = __uint_as_float(vq.x & 0xffff0000u);
        zq[2] = __uint_as_float(vq.y << 16); zq[3] = __uint_as_float(vq.y & 0xffff0000u);
        zq[4] = __uint_as_float(vq.z << 16); zq[5] = __uint_as_float(vq.z & 0xffff0000u);
        zq[6] = __uint_as_float(vq.w << 16); zq[7] = __uint_as_float(vq.w & 0xffff0000u);
      } else {
        zp[0] = __uint_as_float(vp.x); zp[1] = __uint_as_float(vp.y);
        zp[2] = __uint_as_float(vp.z); zp[3] = __uint_as_float(vp.w);
        zq[0] = __uint_as_float(vq.x); zq[1] = __uint_as_float(vq.y);
        zq[2] = __uint_as_float(vq.z); zq[3] = __uint_as_float(vq.w);
      }
#pragma unroll
      for (int e = 0; e < N; ++e) {
        const int i = j * N + e;
        float a = zp[e], bq = zq[e];
        if ((pm >> i) & 1u) {
          a = penalize(a, sc.alpha);
          bq = penalize(bq, sc.alpha);
        }
        float v = 0.f;
        if (base + i < t1) {
          const float p = prob_of(a, sc.c, Mt, it);
          v = ponly ? p : resid_of(p, prob_of(bq, sc.c, Md, id));
        }
        w[i] = v;
        ls += v;
      }
    }
    const float incl = warp_incl_scan(ls, lane);
    const float excl = incl - ls;
    const float tot = __shfl_sync(0xffffffffu, incl, 31);
    // last token with mass in this piece (kept for the fallback)
    {
      const unsigned mp = __ballot_sync(0xffffffffu, ls > 0.f);
      if (mp) {
        const int L1 = 31 - __clz(mp);
        int jj = -1;
        if (lane == L1) {
#pragma unroll
          for (int i = 0; i < LT; ++i)
            if (w[i] > 0.f) jj = i;
        }
        jj = __shfl_sync(0xffffffffu, jj, L1);
        last_any = base0 + L1 * LT + jj;
      }
    }
    if (!take_last) {
      const double r = rem - cum;
      const unsigned m = __ballot_sync(0xffffffffu, ((double)incl > r) && ((double)excl <= r) && ls > 0.f);
      if (m) {
        const int L0 = __ffs(m) - 1;
        int jj = -1;
        if (lane == L0) {
          double cc = (double)excl;
          int lastpos = -1;
#pragma unroll
          for (int i = 0; i < LT; ++i) {
            if (jj < 0) {
              cc += (double)w[i];
              if (w[i] > 0.f) {
                lastpos = i;
                if (cc > r) jj = i;
              }
            }
          }
          if (jj < 0) jj = lastpos;
        }
        jj = __shfl_sync(0xffffffffu, jj, L0);
        if (jj >= 0) {
          found = base0 + L0 * LT + jj;
          break;
        }
      }
    }
    cum += (double)tot;
  }
  return found >= 0 ? found : last_any;
}

// The correction or bonus token of an item: inverse CDF at u_fin of the
// residual (or of p with ponly), first the owning unit, then the token.
template <typename T>
__device__ int item_candidate(const SampleParams& P, const FSmem& S, int item, bool ponly, float u_fin, int lane) {
  const FlowLayout& L = P.FL;
  const int* cu = cu_of(P, S);
  const Item it = pdecode_w(P, cu, item, lane);
  const Scalars sc = item_scalars(P, it, item, cu);
  float4 a;
  item_norms(P, item, it.bonus ? 1 : 2, lane, a.x, a.y, a.z, a.w);
  float* tw = S.tw(0);
  for (int u = lane; u < L.nu; u += 32) {
    float m;
    if (ponly) {
      const float4 r = __ldcg(P.F.p1 + (size_t)item * L.nu + u);
      m = (r.x > -INFINITY) ? __fmul_rn(r.y * ex2(r.x - a.x), a.y) : 0.f;
    } else {
      m = __ldcg(P.F.p2 + (size_t)item * L.nu + u);
    }
    tw[u] = m;
  }
  __syncwarp();
  int ks;
  double rem;
  bool take_last;
  owner_search(tw, L.nu, (double)u_fin, lane, ks, rem, take_last);
  __syncwarp();
  if (ks < 0) return -1;
  const int chunk = ks / kFlowUnits, wp = ks - chunk * kFlowUnits;
  const int lo = chunk * L.lpc, nl = min(L.lpc, L.nlines - lo);
  int l0, l1;
  unit_lines(wp, nl, l0, l1);
  const int t0 = (lo + l0) * 256, t1 = min((lo + l1) * 256, P.V);
  const T* gp = static_cast<const T*>(P.target) + (size_t)it.tgt_row * P.ld_t;
  const T* gq = it.bonus ? gp : static_cast<const T*>(P.draft) + (size_t)it.dft_row * P.ld_d;
  return search_range<T>(P, sc, gp, gq, ponly, t0, t1, rem, take_last, a.x, a.y, a.z, a.w, lane);
}

template <typename T>
__device__ void request_done(const SampleParams& P, const FSmem& S, const Item& it, int item, int flags, int lane) {
  const int b = it.b, K = it.K;
  int fin = 0;
  if (lane == 0) {
    P.inval[(size_t)item * kMaxCluster] = flags;
    const int old = atom_add_acq_rel(P.F.req + b, 1);
    fin = (old == K) && K >= 0 && it.rows_ok;
  }
  if (!__shfl_sync(0xffffffffu, fin, 0)) return;
  const int* cu = cu_of(P, S);
  const int d0 = cu[b], off = d0 + b;
  int st = 0;
  for (int j = lane; j < K + 1; j += 32) {
    const int item_j = j < K ? d0 + j : P.total + b;
    st |= __ldcg(P.inval + (size_t)item_j * kMaxCluster);
  }
  st = warp_or(st);
  int acc = 1;
  if (lane < K) acc = __ldcg(&P.results[d0 + lane].acc);
  const unsigned rej = __ballot_sync(0xffffffffu, lane < K && acc == 0);
  const int jrej = rej ? __ffs(rej) - 1 : K;
  const bool nobonus = (P.flags & 1u) != 0;
  int last = -1;
  if (!st) {
    const float u_fin = __ldg(P.uniforms + off + K);
    if (jrej < K) {
      const float R = __int_as_float(__ldcg(&P.results[d0 + jrej].pad[0]));
      last = item_candidate<T>(P, S, d0 + jrej, !(R > 0.f), u_fin, lane);
    } else if (!nobonus) {
      last = item_candidate<T>(P, S, P.total + b, true, u_fin, lane);
    }
  }
  for (int s = lane; s <= K; s += 32) {
    int tok;
    if (st) tok = -1;
    else if (s < jrej) tok = __ldg(P.draft_tokens + d0 + s);
    else if (s == jrej) tok = last;
    else tok = -1;
    P.out_tokens[off + s] = tok;
  }
  if (lane == 0) {
    P.out_accepted[b] = st ? -1 : jrej;
    if (P.out_status) P.out_status[b] = st;
  }
}

// The items k = CTA, CTA + grid, ... of the pass-1 list (bonus rows first),
// each once its last pass (pass 1 of a bonus row, pass 2 of a position) has
// counted every chunk.
template <typename T>
__device__ void tail(const SampleParams& P, const FSmem& S, int lane) {
  const int nbon = P.n_items - P.n_p2;
  for (int k = blockIdx.x; k < P.n_items; k += gridDim.x) {
    const int item = k < nbon ? P.n_p2 + k : k - nbon;
    const bool bonus = item >= P.n_p2;
    const int* c = P.F.cnt + (bonus ? 0 : P.n_items) + item;
    int late = 0;
    if (lane == 0) {
      const long long t0 = clock64();
      while (ld_acquire(c) < P.FL.nck) {
        if (clock64() - t0 > kWaitLimitCycles) {
          late = 1;
          flag_error(P, kStatusTimeout);
          break;
        }
      }
    }
    if (__shfl_sync(0xffffffffu, late, 0)) break;
    if (bonus) bonus_job<T>(P, S, item, lane);
    else p2_job<T>(P, S, item, lane);
  }
}

// ---------------------------------------------------------------- kernels
template <typename T>
__global__ void __launch_bounds__(kFlowThreads, 1) flow_verify_kernel(const __grid_constant__ SampleParams P) {
  const FlowLayout& L = P.FL;
  const FSmem S(L);
  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int tid = threadIdx.x;
  if (tid == 0) {
    for (int s = 0; s < kFlowSlots; ++s) {
      mbar_init(S.full(s), 2);
      mbar_init(S.claim(s), 1);
      mbar_init(S.done(s), kFlowUnits);
    }
    fence_mbar_init();
  }
  if (P.B + 1 <= 1024)
    for (int i = tid; i <= P.B; i += kFlowThreads) S.cu()[i] = __ldg(P.cu_draft + i);
  __syncthreads();

  if (warp < kNC) {
    consumer<T>(P, S, warp, lane);
  } else if (warp == kWarpF) {
    flow_warp<T>(P, S, lane);
  } else if (warp < kWarpT) {
    setup<T>(P, S, warp - kWarpS, lane);
  } else {
    tail<T>(P, S, lane);
  }
  __syncthreads();
  // the last CTA to finish reports a run that lost a wait: every request
  // gets the timeout status (some may never have been finalised)
  __shared__ int last;
  if (tid == 0) {
    __threadfence();
    last = atomicAdd(P.F.ctl + 2, 1) == (int)gridDim.x - 1 && ld_acquire(P.F.ctl + 1) != 0;
  }
  __syncthreads();
  if (last && P.mode == kModeSample) {
    for (int b = tid; b < P.B; b += kFlowThreads) {
      P.out_accepted[b] = -1;
      if (P.out_status) P.out_status[b] = kStatusTimeout;
    }
  }
}

// Per request: the status bits of its history tokens and, when the
// repetition penalty applies, its history bitmap; the extra CTAs clear the
// counters and item records of the main kernel.
__global__ void __launch_bounds__(256) flow_prep_kernel(const __grid_constant__ SampleParams P) {
  const int tid = threadIdx.x;
  if ((int)blockIdx.x < P.B) {
    const int b = blockIdx.x;
    const int h0 = P.cu_hist ? __ldg(P.cu_hist + b) : 0;
    const int h1 = P.cu_hist ? __ldg(P.cu_hist + b + 1) : 0;
    const float alpha = P.rep_penalty ? __ldg(P.rep_penalty + b) : 1.f;
    const bool pen = item_params_ok(P, b) && alpha != 1.f && h1 > h0;
    uint32_t* bm = P.F.hbm + (size_t)b * P.F.hbm_words;
    if (pen)
      for (int q = tid; q < P.F.hbm_words / 4; q += blockDim.x)
        reinterpret_cast<uint4*>(bm)[q] = make_uint4(0u, 0u, 0u, 0u);
    __syncthreads();
    int flags = 0;
    for (int j = h0 + tid; j < h1; j += blockDim.x) {
      const int tok = __ldg(P.hist + j);
      if (tok < 0 || tok >= P.V) flags |= kStatusBadToken;
      else if (pen) atomicOr(&bm[tok >> 5], 1u << (tok & 31));
    }
    flags = __syncthreads_or(flags);
    if (tid == 0) P.F.rflags[b] = flags ? kStatusBadToken : 0;
  } else {
    const int nz = gridDim.x - P.B;
    for (int q = ((int)blockIdx.x - P.B) * blockDim.x + tid; q < P.F.zero_words; q += nz * blockDim.x)
      P.F.zero[q] = 0;
  }
}

}  // namespace

int launch_flow_verify(SampleParams& P, bool bf16, int num_sms, cudaStream_t stream) {
  const int smem = P.FL.total;
  const long long ntask = (long long)(P.n_items + P.n_p2) * P.FL.nck;
  if (ntask <= 0) return 0;
  const int grid = (int)(ntask < num_sms ? ntask : num_sms);
  // pass-2 lag: about kFlowLagRings rings of tasks across the GPU, so that
  // an item's pass-1 tasks have finished (and been combined) before its
  // pass-2 tasks are claimed
  // (counted past the bonus rows, which lead the pass-1 list)
  P.FL.lag_items = (P.n_items - P.n_p2) + (kFlowLagRings * grid * kFlowSlots) / (2 * P.FL.nck) + 2;
  const int nz = (P.F.zero_words + 2047) / 2048;
  flow_prep_kernel<<<P.B + (nz < 64 ? nz : 64), 256, 0, stream>>>(P);
  if (cudaGetLastError() != cudaSuccess) return -7;
  if (bf16) {
    auto kern = flow_verify_kernel<__nv_bfloat16>;
    if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, smem) != cudaSuccess) {
      cudaGetLastError();
      return -8;
    }
    kern<<<grid, kFlowThreads, smem, stream>>>(P);
  } else {
    auto kern = flow_verify_kernel<float>;
    if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, smem) != cudaSuccess) {
      cudaGetLastError();
      return -8;
    }
    kern<<<grid, kFlowThreads, smem, stream>>>(P);
  }
  if (cudaGetLastError() != cudaSuccess) return -7;
  return 0;
}

}  // namespace sv
