// Split-vocabulary sampling kernel of mentored speculative sampling without
// top-p ("What I Gave Up to Make Speculative Decoding Faster", section "A
// knob for accepting more draft tokens"; D = 0 is the lossless rule of the
// "Speculative Decoding" note, section "Warum eine Korrektur noetig ist").
//
// One persistent CTA per SM; every logit row is cut into `nseg` vocabulary
// segments and unit u = (row u / nseg, segment u % nseg) goes to CTA
// u mod gridDim in that order, so the CTAs stay within one row-width of each
// other and each reads the same number of bytes (+-1 unit).
//
// Pass 1 (every row, every logit read once): softmax statistics per
// (unit, warp): a reference and the sum of 2^(z'c - ref), z' the penalised
// logit, c = log2(e)/T.  When a row's last unit is in, the decider warp of
// the CTA that owns the row combines it; when a request's last row is in,
// the owner of the request takes its decisions from pass-1 quantities
// alone wherever they are fixed:
//   theta = min(1, D/d) lies in [D, min(1, D/(q(x)-p(x)))] because
//   q(x) - p(x) <= d <= 1, so pi(x) = p(x) + theta (q(x) - p(x)) is bounded
//   by p + D (q - p) and min(q, p + D) when q(x) > p(x), and pi(x) >= q(x)
//   when p(x) >= q(x).  A uniform outside the bounds (with a relative margin
//   far above the fp32 error) fixes the acceptance test without d.
// Pass 2 (a "job"): only for the positions whose test the bounds leave open
// before the first certain rejection, and for that rejection itself (its
// residual draw).  A job re-reads the position's two rows in half-segment
// units, unit g of the job list going to CTA g mod gridDim, and sums
// max(p - q, 0) per (unit, warp); its last unit gives d = TV(p, q), theta,
// pi(x) and the exact decision.  The finisher warp of the request's owner
// then draws the correction from the residual's (unit, warp) masses and one
// re-read range, or the bonus token from the last target row's pass-1
// masses, and writes the tokens.
//
// Warp roles: warp 0 producer (TMA bulk copies into a 6-slot ring; slot s
// feeds consumer group s mod 3), warp 1 recorder (stores the consumers'
// partials, counts units, finds published second-pass units for the
// producer), warp 2 decider (row combines, decisions, second passes' ends),
// warp 3 finisher (draws and tokens), warps 4.. consumers in 3 groups of 8.
// Every wait is bounded; a wait that runs out raises a global abort flag,
// everyone leaves, and the last CTA marks unfinished requests
// SPEC_STATUS_TIMEOUT.

#include "common.cuh"
#include "spec_internal.h"
#include "seg_internal.h"
#include "stream_common.cuh"

namespace sv {

namespace {

extern __shared__ __align__(128) unsigned char seg_smem[];

constexpr int seg_al16(int x) { return (x + 15) / 16 * 16; }
constexpr int kOffBars = kSegSlots * kSegSlotBytes;                     // full[kSegSlots], empty[kSegSlots]
constexpr int kOffRec = seg_al16(kOffBars + 2 * kSegSlots * 8);        // unit records (kSegRecN)
constexpr int kOffMisc = seg_al16(kOffRec + kSegRecN * (int)sizeof(SegUnitRec));  // control words
constexpr int kSegJq = 64;                                              // second-pass candidates found, not yet issued
constexpr int kOffJq = seg_al16(kOffMisc + 64);                         // their job entries (kSegJq, 8 bytes each)
// Claimed pass-1 units queued for the producer, with their geometry.
struct SegSteal {
  unsigned long long logits, bits, desc;   // global addresses
  int u, tok0, n, pad;
};
constexpr int kSegSq = 32;
constexpr int kStealChunk = 8;                                          // pass-1 units per claim
constexpr int kStealAhead = 16;                                         // queued claimed units kept ahead
constexpr int kStealLead = 8;                                           // dealt units left when claiming starts
static_assert(kStealAhead <= kSegSq && kStealChunk <= 32, "claims fit the queue and a warp");
constexpr int kOffSq = kOffJq + kSegJq * 8;                             // the claimed units (kSegSq)
constexpr int kSegFq = 64;                                              // requests ready for their tokens
constexpr int kOffFq = kOffSq + kSegSq * (int)sizeof(SegSteal);         // their indices (kSegFq)
constexpr int kDrawBytes = 4096;                                         // a draw's staged logits (both rows of a pair)
constexpr int kOffDraw = kOffFq + kSegFq * 4;                           // [2]: the finisher's and the decider's draw areas
constexpr int kDrawArea = kDrawBytes + 256 + 16;                        // logits, penalty words, mbarrier + phase
constexpr int kOffCu = kOffDraw + 2 * kDrawArea;                        // cu_draft copy (B + 1 <= kSegCuCap)
constexpr int kSegSmem = kOffCu + kSegCuCap * 4;
static_assert(kSegSlotBytes % 128 == 0 && kOffBars % 8 == 0 && kOffRec % 16 == 0 && kOffJq % 16 == 0 &&
                  kOffSq % 16 == 0 && kOffFq % 16 == 0 && kOffDraw % 16 == 0 && kDrawArea % 16 == 0 &&
                  kOffCu % 16 == 0,
              "shared-memory regions keep the alignment of their widest access");


// ------------------------------------------------------------------ PTX
__device__ __forceinline__ void mbar_expect(uint64_t* bar, uint32_t bytes) {
  asm volatile("mbarrier.expect_tx.relaxed.cta.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(bar)), "r"(bytes)
               : "memory");
}
__device__ __forceinline__ void st_rel_cta(unsigned* p, unsigned v) {
  asm volatile("st.release.cta.shared::cta.u32 [%0], %1;" ::"r"(smem_u32(p)), "r"(v) : "memory");
}
__device__ __forceinline__ unsigned ld_acq_cta(const unsigned* p) {
  unsigned v;
  asm volatile("ld.acquire.cta.shared::cta.u32 %0, [%1];" : "=r"(v) : "r"(smem_u32(p)) : "memory");
  return v;
}
__device__ __forceinline__ unsigned atom_add_gpu(unsigned* p, unsigned v) {
  unsigned o;
  asm volatile("atom.acq_rel.gpu.global.add.u32 %0, [%1], %2;" : "=r"(o) : "l"(p), "r"(v) : "memory");
  return o;
}
__device__ __forceinline__ void red_add_gpu(unsigned* p, unsigned v) {
  asm volatile("red.release.gpu.global.add.u32 [%0], %1;" ::"l"(p), "r"(v) : "memory");
}
__device__ __forceinline__ unsigned ld_acq_gpu(const unsigned* p) {
  unsigned v;
  asm volatile("ld.acquire.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
  return v;
}
__device__ __forceinline__ void st_rel_gpu64(void* p, unsigned long long v) {
  asm volatile("st.release.gpu.global.u64 [%0], %1;" ::"l"(p), "l"(v) : "memory");
}
__device__ __forceinline__ void fence_proxy_async_global() {
  asm volatile("fence.proxy.async.global;" ::: "memory");
}

// Records other CTAs wrote in this launch are read through L2 (__ldcg).
__device__ __forceinline__ SegRowDesc ld_desc(const SegRowDesc* p) {
  SegRowDesc d;
  const int4* s = reinterpret_cast<const int4*>(p);
  int4* o = reinterpret_cast<int4*>(&d);
#pragma unroll
  for (int j = 0; j < (int)(sizeof(SegRowDesc) / 16); ++j) o[j] = __ldcg(s + j);
  return d;
}
__device__ __forceinline__ SegRowStat ld_stat(const SegRowStat* p) {
  const float4 v = __ldcg(reinterpret_cast<const float4*>(p));
  SegRowStat r;
  r.M = v.x;
  r.S = v.y;
  r.px = v.z;
  r.flags = __float_as_int(v.w);
  return r;
}
__device__ __forceinline__ SegPos ld_pos(const SegPos* p) {
  SegPos r;
  const int4* s = reinterpret_cast<const int4*>(p);
  int4* o = reinterpret_cast<int4*>(&r);
  o[0] = __ldcg(s);
  o[1] = __ldcg(s + 1);
  return r;
}
__device__ __forceinline__ SegJobDesc ld_job(const SegJobDesc* p) {
  const float4 v = __ldcg(reinterpret_cast<const float4*>(p));
  SegJobDesc r;
  r.Lp = v.x;
  r.Lq = v.y;
  r.fp = v.z;
  r.fq = v.w;
  return r;
}

// ------------------------------------------------------------- shared state
struct Ring {
  __device__ unsigned char* slot(int s) const { return seg_smem + (size_t)s * kSegSlotBytes; }
  __device__ uint64_t* full() const { return reinterpret_cast<uint64_t*>(seg_smem + kOffBars); }
  __device__ uint64_t* empty() const { return full() + kSegSlots; }
  __device__ SegUnitRec* rec(int k) const {
    return reinterpret_cast<SegUnitRec*>(seg_smem + kOffRec) + (k % kSegRecN);
  }
  __device__ unsigned* misc() const { return reinterpret_cast<unsigned*>(seg_smem + kOffMisc); }
  __device__ unsigned long long* jq() const { return reinterpret_cast<unsigned long long*>(seg_smem + kOffJq); }
  __device__ int* fq() const { return reinterpret_cast<int*>(seg_smem + kOffFq); }
  __device__ SegSteal* sq() const { return reinterpret_cast<SegSteal*>(seg_smem + kOffSq); }
  __device__ int* cu() const { return reinterpret_cast<int*>(seg_smem + kOffCu); }
  __device__ unsigned char* draw_area(int i) const { return seg_smem + kOffDraw + i * kDrawArea; }
};

__device__ __forceinline__ SegUnitHdr* hdr_of(unsigned char* slot) {
  return reinterpret_cast<SegUnitHdr*>(slot + kSegHdrOff);
}

__device__ __forceinline__ bool aborted(const SegParams& P) {
  return *reinterpret_cast<volatile const unsigned*>(P.ctl + kCtlAbort) != 0u;
}
__device__ __forceinline__ void raise_abort(const SegParams& P) { atomicExch(P.ctl + kCtlAbort, 1u); }

// One try of an mbarrier phase that may suspend the thread for up to
// `ns` nanoseconds (it resumes early once the phase completes), so that a
// waiting warp takes no issue slots from the working ones.
__device__ __forceinline__ bool mbar_try(uint64_t* bar, uint32_t parity, uint32_t ns) {
  uint32_t ok;
  asm volatile(
      "{ .reg .pred p; mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2, %3; selp.u32 %0, 1, 0, p; }"
      : "=r"(ok)
      : "r"(smem_u32(bar)), "r"(parity), "r"(ns)
      : "memory");
  return ok != 0;
}

// Bounded wait on an mbarrier phase; false if it ran out or another CTA
// raised the abort flag.
__device__ __forceinline__ bool ring_wait(const SegParams& P, uint64_t* bar, uint32_t parity) {
  if (mbar_try(bar, parity, 20000u)) return true;
  const long long t0 = clock64();
  for (int n = 1;; ++n) {
    if (mbar_try(bar, parity, 20000u)) return true;
    if ((n & 3) == 0 && aborted(P)) return false;
    if (clock64() - t0 > P.wait_limit) {
      raise_abort(P);
      return false;
    }
  }
}

// Bounded poll of a global word until pred(value) holds.
template <typename F>
__device__ __forceinline__ bool poll_gpu(const SegParams& P, const unsigned* p, F&& pred) {
  if (pred(ld_acq_gpu(p))) return true;
  const long long t0 = clock64();
  for (;;) {
    __nanosleep(128);
    if (pred(ld_acq_gpu(p))) return true;
    if (aborted(P)) return false;
    if (clock64() - t0 > P.wait_limit) {
      raise_abort(P);
      return false;
    }
  }
}

// ---------------------------------------------------------------- arithmetic
// (reference, sum) pairs, the sum relative to 2^reference.
__device__ __forceinline__ void pair_merge(float& M, float& S, float m, float s) {
  if (s == 0.f) return;
  if (S == 0.f) {
    M = m;
    S = s;
    return;
  }
  const float nm = fmaxf(M, m);
  S = S * ex2(M - nm) + s * ex2(m - nm);
  M = nm;
}

__device__ __forceinline__ void warp_pair(float& M, float& S) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
    const float m = __shfl_xor_sync(0xffffffffu, M, o);
    const float s = __shfl_xor_sync(0xffffffffu, S, o);
    pair_merge(M, S, m, s);
  }
}

__device__ __forceinline__ bool params_ok(float T, float alpha, float D) {
  return T > 0.f && T < INFINITY && alpha > 0.f && alpha < INFINITY && D >= 0.f && D <= 1.f;
}

// The acceptance test from pass-1 quantities: 1 certain accept, 0 certain
// reject, 2 needs d.  The thresholds are on u (the test is u < pi(x)/q(x));
// the margin of 1e-5 relative is far above the fp32 error of p(x)/q(x).
__device__ __forceinline__ int bound_decision(float px, float qx, float D, float u) {
  if (!(qx > 0.f) || !(px >= 0.f) || !(qx < INFINITY) || !(px < INFINITY)) return 2;
  if (px >= qx) return u < 1.f - 1e-5f ? 1 : 2;
  const float lo = __fdiv_rn(fmaf(D, qx - px, px), qx);     // theta = D: d <= 1
  const float hi = fminf(1.f, __fdiv_rn(px + D, qx));        // theta <= D / (q(x) - p(x))
  if (u < lo - (1e-5f * lo + 1e-9f)) return 1;
  if (u > hi + (1e-5f * hi + 1e-9f)) return 0;
  return 2;
}

// ------------------------------------------------------------ prologue
// Request b's prologue, by the CTA's warps 1 .. kSegThreads / 32 - 1 (`tid` in
// 0 .. kPrepThreads-1; the producer warp is busy with the first copies):
// status bits, the history bitmap (every token of the request's history)
// and the descriptors of the request's rows.  With alpha = 1 the penalty is
// the identity and the set stays empty.  `sh` is a shared word for the
// status bits.
constexpr int kPrepThreads = kSegThreads - 32;
constexpr int kPrepBar = 15;

__device__ __forceinline__ void prep_sync() { named_sync(kPrepBar, kPrepThreads); }

__device__ void prep_request(const SegParams& P, int b, int tid, unsigned* sh) {
  const int lane = tid & 31;
  const int d0 = __ldg(P.cu_draft + b), d1 = __ldg(P.cu_draft + b + 1);
  const int K = d1 - d0;
  const bool rows_ok = d0 >= 0 && d1 >= d0 && d1 <= P.total;
  const float T = __ldg(P.temperature + b);
  const float alpha = P.rep_penalty ? __ldg(P.rep_penalty + b) : 1.f;
  const float D = __ldg(P.tv_budget + b);
  const bool pok = params_ok(T, alpha, D);
  const bool pen = pok && alpha != 1.f;
  int h0 = 0, h1 = 0;
  bool hist_ok = true;
  if (P.cu_hist) {
    h0 = __ldg(P.cu_hist + b);
    h1 = __ldg(P.cu_hist + b + 1);
    if (h0 < 0 || h1 < h0) {
      hist_ok = false;
      h1 = h0;
    }
  }
  const int words = P.g.bm_bytes / 4;
  uint32_t* bm = P.bitmap + (size_t)b * words;
  if (tid == 0) {
    int st = 0;
    if (!rows_ok) {
      atomicOr(P.ctl + kCtlBroken, 1u);
      st |= kStatusBadK;
    }
    if (K > P.max_k) st |= kStatusBadK;
    if (!pok) st |= kStatusBadParam;
    if (!hist_ok) st |= kStatusBadToken;
    *sh = (unsigned)st;
  }
  uint4* bm4 = reinterpret_cast<uint4*>(bm);
  for (int j = tid; j < words / 4; j += kPrepThreads) bm4[j] = make_uint4(0u, 0u, 0u, 0u);
  prep_sync();
  // history tokens (loads first, then the bits) and the drafts' range check
  unsigned bad = 0;
  for (int j0 = h0; j0 < h1; j0 += 2 * kPrepThreads) {
    int t[2];
#pragma unroll
    for (int q = 0; q < 2; ++q) {
      const int j = j0 + q * kPrepThreads + tid;
      t[q] = j < h1 ? __ldg(P.hist + j) : 0;
    }
#pragma unroll
    for (int q = 0; q < 2; ++q) {
      if (j0 + q * kPrepThreads + tid >= h1) continue;
      if (t[q] < 0 || t[q] >= P.V) bad = 1;
      else if (pen) atomicOr(bm + (t[q] >> 5), 1u << (t[q] & 31));
    }
  }
  if (rows_ok)
    for (int k = tid; k < K; k += kPrepThreads) {
      const int t = __ldg(P.draft_tokens + d0 + k);
      if (t < 0 || t >= P.V) bad = 1;
    }
  if (__any_sync(0xffffffffu, bad) && lane == 0) atomicOr(sh, (unsigned)kStatusBadToken);
  prep_sync();
  if (tid >= 32) return;
  // warp 1: the request's drafts (lane k holds x_k; K <= 32 for a valid request)
  const int st = (int)*sh;
  if (lane == 0) P.req_status[b] = st;
  if (!rows_ok) return;
  int x = -1;
  if (lane < K) x = __ldg(P.draft_tokens + d0 + lane);
  const bool xok = x >= 0 && x < P.V;
  // x_k in the history (the bitmap is complete: read through L2)
  const bool inh = pen && xok && ((__ldcg(bm + (x >> 5)) >> (x & 31)) & 1u);
  // x_k's first occurrence among the drafts
  bool first = xok;
  const int kk = K < 32 ? K : 32;
  for (int j = 0; j < kk; ++j) {
    const int e = __shfl_sync(0xffffffffu, x, j);
    if (j < lane && e == x) first = false;
  }
  const float c = pok ? (float)(1.4426950408889634 / (double)T) : 1.f;
  const float a = pok ? alpha : 1.f;
  const int off = d0 + b;
  // row i's extras: the drafts before it that are not in the history, each once
  SegRowDesc d;
  d.b = b;
  d.i = lane;
  d.kind = 0;
  d.x = (lane < K && xok) ? x : -1;
  d.x_pen = (lane < K) && inh;
  d.n_extra = 0;
  d.c = c;
  d.alpha = a;
  d.src = 0;
  d.pad[0] = d.pad[1] = d.pad[2] = 0;
#pragma unroll
  for (int k = 0; k < kSegMaxExtras; ++k) d.extras[k] = -1;
  for (int j = 0; j < kk; ++j) {
    const int e = __shfl_sync(0xffffffffu, x, j);
    const bool ein = __shfl_sync(0xffffffffu, (int)inh, j) != 0;
    const bool efirst = __shfl_sync(0xffffffffu, (int)first, j) != 0;
    if (pen && j < lane && efirst && !ein) d.extras[d.n_extra++] = e;
    if (pen && j < lane && e == d.x && d.x >= 0) d.x_pen = 1;
  }
  // rows in request order: target i at base + 2i, draft i at base + 2i + 1,
  // the bonus row at base + 2K
  const int base = 2 * d0 + b;
  for (int i = lane; i <= K; i += 32) {
    if (i >= 32) {        // only invalid requests (K > max_k) get here: no penalty bookkeeping
      d.i = i;
      d.x = -1;
      d.x_pen = 0;
      d.n_extra = 0;
    }
    d.kind = 0;
    d.src = off + i;
    P.rowdesc[base + 2 * i] = d;
    if (i < K) {
      P.posdesc[d0 + i] = d;
      d.kind = 1;
      d.src = P.NT + d0 + i;
      P.rowdesc[base + 2 * i + 1] = d;
    }
  }
}

// ------------------------------------------------------------ the producer
// Row r's logits: target row r (r < NT) or draft row r - NT.
template <typename T>
__device__ __forceinline__ const unsigned char* row_ptr(const SegParams& P, int r) {
  if (r < P.NT) return static_cast<const unsigned char*>(P.target) + (size_t)r * P.ld_t * sizeof(T);
  return static_cast<const unsigned char*>(P.draft) + (size_t)(r - P.NT) * P.ld_d * sizeof(T);
}

__device__ __forceinline__ uint32_t tma_bytes(int n, int es) { return (uint32_t)((n * es + 15) & ~15); }

// Logical row r (rows in request order) -> its request and its logits row
// (target row t, or draft row k as NT + k), by binary search over the
// requests' first rows 2 cu_draft[b] + b.  `cu` is cu_draft (a shared-memory
// copy when it fits).  Rows of an inconsistent cu_draft map to row 0 (such a
// batch streams nothing once the prologue has seen it).
__device__ __forceinline__ int2 row_src(const SegParams& P, const int* cu, int r) {
  int lo = 0, hi = P.B;
  while (hi - lo > 1) {
    const int mid = (lo + hi) >> 1;
    if (2 * cu[mid] + mid <= r) lo = mid;
    else hi = mid;
  }
  const int b = lo, d0 = cu[b], K = cu[b + 1] - d0;
  const int j = r - (2 * d0 + b);
  int src;
  if (d0 < 0 || K < 0 || j < 0 || j > 2 * K) src = 0;
  else if (j == 2 * K) src = d0 + b + K;
  else if (j & 1) src = P.NT + d0 + (j >> 1);
  else src = d0 + b + (j >> 1);
  if (src < 0 || src >= P.NR) src = 0;
  return make_int2(b, src);
}

// Pass-1 units: u = 0 .. NR * nseg - 1 in row order.  The first ones, in
// whole waves of gridDim (kDealtNum / kDealtDen of the waves when there are
// at least kDealtDen), are dealt out: CTA c takes u = c + ks * gridDim.x, so
// that all CTAs sweep the rows together (requests complete in order).  The
// rest go to whichever CTA claims them first (a global counter), in chunks
// of kStealChunk: CTAs that ran slower take fewer of them, which evens out
// the end of the pass.
constexpr int kDealtNum = 3, kDealtDen = 4;
__device__ __forceinline__ int dealt_units(const SegParams& P) {
  const long long U = (long long)P.NR * P.g.nseg;
  const long long waves = (U + gridDim.x - 1) / gridDim.x;
  const long long own = waves >= kDealtDen ? waves * kDealtNum / kDealtDen : waves;
  return (int)(own * gridDim.x < U ? own * gridDim.x : U);
}
__device__ __forceinline__ int static_units(const SegParams& P) {
  const long long D = dealt_units(P);
  return (long long)blockIdx.x < D ? (int)((D - 1 - blockIdx.x) / gridDim.x + 1) : 0;
}
__device__ __forceinline__ int unit_of(int ks) { return (int)blockIdx.x + ks * (int)gridDim.x; }

// The wait for the producer's copies in flight before its CTA exits: a fixed
// bound (about two seconds), whatever wait limit the call runs with.
constexpr long long kSegDrainCycles = 4000000000ll;

// Producer state, the same in every lane of warp 0.
struct Prod {
  uint32_t filled = 0;    // slots filled at least once (bit s)
  uint32_t par = 0;       // parity of each slot's last fill (bit s)
  int rec_seen = 0;       // records the recorder had taken when last looked
  __device__ __forceinline__ void fill(int k) {
    const int s = k % kSegSlots;
    filled |= 1u << s;
    par = (par & ~(1u << s)) | ((uint32_t)((k / kSegSlots) & 1) << s);
  }
};

// Unit k may go into the ring: the recorder has taken the record unit
// k - kSegRecN left, and the consumers have released the slot.  Waited by
// lane 0; every lane gets the outcome (false: a wait ran out).
__device__ __forceinline__ bool wait_slot(const SegParams& P, const Ring& R, Prod& st, int k, int lane) {
  bool ok = true;
  if (k >= kSegRecN && st.rec_seen <= k - kSegRecN) {
    if (lane == 0) {
      const long long t0 = clock64();
      while ((int)ld_acq_cta(R.misc() + 1) <= k - kSegRecN) {
        if (aborted(P) || clock64() - t0 > P.wait_limit) {
          raise_abort(P);
          ok = false;
          break;
        }
        __nanosleep(32);
      }
      st.rec_seen = (int)ld_acq_cta(R.misc() + 1);
    }
    st.rec_seen = __shfl_sync(0xffffffffu, st.rec_seen, 0);
  }
  if (k >= kSegSlots && lane == 0 && ok) {
    const int s = k % kSegSlots;
    ok = ring_wait(P, R.empty() + s, (uint32_t)((k / kSegSlots - 1) & 1));
  }
  return __shfl_sync(0xffffffffu, ok, 0) != 0;
}

// Whether an mbarrier phase has completed, without waiting for it.
__device__ __forceinline__ bool mbar_done(uint64_t* bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{ .reg .pred p; mbarrier.test_wait.parity.shared::cta.b64 p, [%1], %2; selp.u32 %0, 1, 0, p; }"
      : "=r"(ok)
      : "r"(smem_u32(bar)), "r"(parity)
      : "memory");
  return ok != 0;
}

// Arrive on a full barrier, raising the bytes it waits for first.
__device__ __forceinline__ void mbar_arrive_expect(uint64_t* bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.release.cta.shared::cta.b64 _, [%0], %1;" ::"r"(smem_u32(bar)), "r"(bytes)
               : "memory");
}

// The slot header and the unit record of ring unit k (plain stores: the
// slot's arrival releases them to the consumers, and the recorder reads the
// record only after the consumers have counted the unit done).
__device__ __forceinline__ void put_unit(const Ring& R, int k, int kind, int id, int part, int tok0, int n) {
  unsigned char* slot = R.slot(k % kSegSlots);
  SegUnitHdr* h = hdr_of(slot);
  *reinterpret_cast<int4*>(h) = make_int4(kind, id, part, tok0);
  h->n = n;
  *reinterpret_cast<int4*>(R.rec(k)) = make_int4(kind, id, part, 0);
}

// Pass-1 unit geometry: static unit ks of this CTA is unit u =
// blockIdx.x + ks * gridDim.x, i.e. segment u % nseg of logical row
// u / nseg.  Lane l of the producer holds the geometry of static unit
// 32 j + l of the current batch j of 32, and issues that unit.
struct RowUnit {
  const unsigned char* logits;   // the segment's first logit
  const unsigned char* bits;     // the segment's penalty bits (its request's bitmap)
  const SegRowDesc* desc;        // the row's descriptor
  int u, tok0, n;                // n < 0: no such unit
};

template <typename T>
__device__ __forceinline__ RowUnit row_unit(const SegParams& P, const int* cu, int ks, int n_static) {
  RowUnit x{};
  x.n = -1;
  if (ks >= n_static) return x;
  x.u = unit_of(ks);
  const int r = x.u / P.g.nseg, sg = x.u - r * P.g.nseg;
  x.tok0 = sg * P.g.seg;
  x.n = min(P.g.seg, P.V - x.tok0);
  const int2 bs = row_src(P, cu, r);
  x.logits = row_ptr<T>(P, bs.y) + (size_t)x.tok0 * sizeof(T);
  x.bits = reinterpret_cast<const unsigned char*>(P.bitmap) + (size_t)bs.x * P.g.bm_bytes + (size_t)sg * (P.g.seg / 8);
  x.desc = P.rowdesc + r;
  return x;
}

// The logits copy of a pass-1 unit (ring unit k), ahead of the rest.
template <typename T>
__device__ __forceinline__ void issue_row_logits(const Ring& R, int k, const RowUnit& x, uint64_t pol) {
  const int s = k % kSegSlots;
  put_unit(R, k, kUnitRow, x.u, 0, x.tok0, x.n);
  const uint32_t bytes = tma_bytes(x.n, sizeof(T));
  mbar_expect(R.full() + s, bytes);
  bulk_g2s(R.slot(s), x.logits, bytes, R.full() + s, pol);
}

// A pass-1 unit as ring unit k: the logits (unless already on their way),
// the penalty bits and the row descriptor, with the slot's single arrival
// first (it raises the bytes the slot waits for).
template <typename T>
__device__ __forceinline__ void issue_row(const SegParams& P, const Ring& R, int k, const RowUnit& x,
                                          bool logits_issued, uint64_t pol_s, uint64_t pol_k) {
  const int s = k % kSegSlots;
  unsigned char* slot = R.slot(s);
  if (!logits_issued) put_unit(R, k, kUnitRow, x.u, 0, x.tok0, x.n);
  const uint32_t lb = logits_issued ? 0u : tma_bytes(x.n, sizeof(T));
  const uint32_t bmb = (uint32_t)(P.g.seg / 8);
  mbar_arrive_expect(R.full() + s, lb + bmb + (uint32_t)sizeof(SegRowDesc));
  if (lb) bulk_g2s(slot, x.logits, lb, R.full() + s, pol_s);
  bulk_g2s(slot + kSegLogitBytes, x.bits, bmb, R.full() + s, pol_k);
  bulk_g2s(slot + kSegDescOff, x.desc, (uint32_t)sizeof(SegRowDesc), R.full() + s, pol_k);
}

// Pass-2 unit: half-segment `part` of position p (request b).
template <typename T>
__device__ __forceinline__ void issue_pair(const SegParams& P, const Ring& R, int k, int p, int b, int part,
                                           uint64_t pol_s, uint64_t pol_k) {
  const int s = k % kSegSlots;
  unsigned char* slot = R.slot(s);
  const int sg = part >> 1, hh = part & 1;
  const int half = P.g.seg / 2;
  const int tok0 = sg * P.g.seg + hh * half;
  const int n = max(0, min(half, P.V - tok0));
  put_unit(R, k, kUnitPair, p, part, tok0, n);
  const uint32_t bytes = tma_bytes(n, sizeof(T));
  const uint32_t bmb = (uint32_t)(half / 8);
  mbar_arrive_expect(R.full() + s, 2 * bytes + bmb + (uint32_t)(sizeof(SegRowDesc) + sizeof(SegJobDesc)));
  if (bytes) {
    bulk_g2s(slot, row_ptr<T>(P, p + b) + (size_t)tok0 * sizeof(T), bytes, R.full() + s, pol_s);
    bulk_g2s(slot + kSegLogitBytes / 2, row_ptr<T>(P, P.NT + p) + (size_t)tok0 * sizeof(T), bytes, R.full() + s,
             pol_s);
  }
  bulk_g2s(slot + kSegLogitBytes,
           reinterpret_cast<const unsigned char*>(P.bitmap) + (size_t)b * P.g.bm_bytes + (size_t)tok0 / 8, bmb,
           R.full() + s, pol_k);
  bulk_g2s(slot + kSegDescOff, P.posdesc + p, (uint32_t)sizeof(SegRowDesc), R.full() + s, pol_k);
  bulk_g2s(slot + kSegDescOff + sizeof(SegRowDesc), P.jobdesc + p, (uint32_t)sizeof(SegJobDesc), R.full() + s,
           pol_k);
}

__device__ __forceinline__ void issue_stop(const Ring& R, int k) {
  const int s = k % kSegSlots;
  hdr_of(R.slot(s))->kind = kUnitStop;
  mbar_arrive(R.full() + s);
}

// cu_draft as the producer reads it: the shared-memory copy when it fits.
__device__ __forceinline__ const int* cu_of(const SegParams& P, const Ring& R) {
  return P.B + 1 <= kSegCuCap ? R.cu() : P.cu_draft;
}

// Pass-1 units whose logits copies start before the prologue's end: more
// of them only slow the prologue's own loads.
constexpr int kSegPre = 3;

// The producer warp, before the prologue: caches cu_draft, computes the
// geometry of its first 32 static units (lane l: unit l) and starts the
// logits copies of the first kSegPre of them, one lane each.  Returns how
// many copies it started.
template <typename T>
__device__ int producer_prefetch(const SegParams& P, const Ring& R, Prod& st, RowUnit& mine, int lane) {
  if (P.B + 1 <= kSegCuCap)
    for (int j = lane; j <= P.B; j += 32) R.cu()[j] = __ldg(P.cu_draft + j);
  __syncwarp();
  const int n_static = static_units(P);
  const int pre = min(n_static, kSegPre);
  mine = row_unit<T>(P, cu_of(P, R), lane, n_static);
  if (lane < pre) issue_row_logits<T>(R, lane, mine, l2_policy_evict_first());
  for (int k = 0; k < pre; ++k) st.fill(k);
  return pre;
}

__device__ __forceinline__ unsigned ld_relaxed_gpu(const unsigned* p) {
  unsigned v;
  asm volatile("ld.relaxed.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
  return v;
}

__device__ __forceinline__ unsigned long long ld_relaxed_gpu64(const void* p) {
  unsigned long long v;
  asm volatile("ld.relaxed.gpu.global.u64 %0, [%1];" : "=l"(v) : "l"(p) : "memory");
  return v;
}

// The producer warp: puts units into the ring in order.  Static (pass-1)
// units go in as their slots come free, each issued by the lane that holds
// its geometry; second-pass units go ahead of them as soon as the recorder
// has queued one.  At the end, one stop per consumer group.
template <typename T>
__device__ void producer(const SegParams& P, const Ring& R, Prod& st, RowUnit mine, int pre, int lane) {
  const int G = gridDim.x;
  const int n_static = static_units(P);
  const int* cu = cu_of(P, R);
  const uint64_t pol_s = l2_policy_evict_first(), pol_k = l2_policy_evict_last();
  // every CTA's prologue is done: descriptors and bitmaps exist
  bool ok = true;
  if (lane == 0) ok = poll_gpu(P, P.ctl + kCtlPrepDone, [G](unsigned v) { return v >= (unsigned)G; });
  ok = __shfl_sync(0xffffffffu, ok, 0) != 0;
  fence_proxy_async_global();
  const bool broken = ok && ld_acq_gpu(P.ctl + kCtlBroken) != 0u;
  // the job list is cleared and may be watched (misc[5], for the recorder)
  if (lane == 0 && ok && !broken) st_rel_cta(R.misc() + 5, 1u);
  int k = 0;        // units put into the ring (static and second-pass)
  int real = 0;     // of which real units (the rest are stops)
  int stops = 0;    // stop units in the ring (one per group ends the consumers)
  long long t_idle = clock64();   // the last unit issued (bounds the wait for jobs)
  if (ok && !broken) {
    const unsigned upj = (unsigned)P.g.upj;
    int ks = 0;               // static units issued
    // Second-pass units: this CTA's candidates g = blockIdx.x + c * G of the
    // job list (unit g: part g % upj of job g / upj), taken in order c =
    // 0, 1, ...  The recorder warp watches the job list and queues each
    // candidate's entry once published (misc[8] counts them); the producer
    // issues no global load while static units remain, so that none of its
    // releases waits on one.
    unsigned head = 0;        // candidates issued
    unsigned shead = 0;       // claimed pass-1 units issued
    if (pre > 0) {
      // first the prefetched units (ring units 0 .. pre-1, their slots
      // fresh): penalty bits, descriptors and arrivals, one lane each
      if (lane < pre) issue_row<T>(P, R, lane, mine, true, pol_s, pol_k);
      k = ks = pre;
    }
    for (;;) {
      const unsigned tail = *reinterpret_cast<volatile unsigned*>(R.misc() + 8);
      if (head < tail) {
        (void)ld_acq_cta(R.misc() + 8);      // the queued entry and its job's descriptors
        const unsigned long long e0 = R.jq()[head % kSegJq];
        ok = wait_slot(P, R, st, k, lane);
        if (!ok) break;
        if (lane == 0)
          issue_pair<T>(P, R, k, (int)(e0 & 0xffffffffull) - 1, (int)(e0 >> 32),
                        (int)((blockIdx.x + head * (unsigned)G) % upj), pol_s, pol_k);
        st.fill(k);
        ++k;
        ++head;
        if (lane == 0) st_rel_cta(R.misc() + 9, head);   // the queue entry is free again
        t_idle = clock64();
        continue;
      }
      if (ks < n_static) {
        if ((ks & 31) == 0 && ks > 0) mine = row_unit<T>(P, cu, ks + lane, n_static);
        // the next units whose slots are free and whose records the
        // recorder has taken (to the end of this batch of 32) go in
        // together, one lane each; with none free, wait for the first
        const int lim = min(min(kSegSlots, n_static - ks), 32 - (ks & 31));
        const int kk = k + lane;
        bool fr = false;
        if (lane < lim)
          fr = (kk < kSegRecN || st.rec_seen > kk - kSegRecN) &&
               (kk < kSegSlots || mbar_done(R.empty() + kk % kSegSlots, (uint32_t)((kk / kSegSlots - 1) & 1)));
        const unsigned fm = __ballot_sync(0xffffffffu, fr);
        int n = fm == 0xffffffffu ? 32 : __ffs(~fm) - 1;
        if (n == 0) {
          ok = wait_slot(P, R, st, k, lane);
          if (!ok) break;
          n = 1;
        }
        __syncwarp();     // the slots' releases, seen by the testing lanes, before the copies
        if (((lane - ks) & 31) < n) issue_row<T>(P, R, k + ((lane - ks) & 31), mine, false, pol_s, pol_k);
        for (int j = 0; j < n; ++j) st.fill(k + j);
        k += n;
        ks += n;
        if (lane == 0) *reinterpret_cast<volatile unsigned*>(R.misc() + 13) = (unsigned)ks;   // for the claims
        t_idle = clock64();
        continue;
      }
      // then the claimed pass-1 units the recorder queued (misc[6]), those
      // whose slots are free together, one lane each
      const unsigned stail = *reinterpret_cast<volatile unsigned*>(R.misc() + 6);
      if (shead < stail) {
        (void)ld_acq_cta(R.misc() + 6);
        const int lim = min((int)(stail - shead), kSegSlots);
        const int kk = k + lane;
        bool fr = false;
        if (lane < lim)
          fr = (kk < kSegRecN || st.rec_seen > kk - kSegRecN) &&
               (kk < kSegSlots || mbar_done(R.empty() + kk % kSegSlots, (uint32_t)((kk / kSegSlots - 1) & 1)));
        const unsigned fm = __ballot_sync(0xffffffffu, fr);
        int n = fm == 0xffffffffu ? 32 : __ffs(~fm) - 1;
        if (n == 0) {
          ok = wait_slot(P, R, st, k, lane);
          if (!ok) break;
          n = 1;
        }
        __syncwarp();
        if (lane < n) {
          const SegSteal e = R.sq()[(shead + lane) % kSegSq];
          RowUnit x;
          x.logits = reinterpret_cast<const unsigned char*>(e.logits);
          x.bits = reinterpret_cast<const unsigned char*>(e.bits);
          x.desc = reinterpret_cast<const SegRowDesc*>(e.desc);
          x.u = e.u;
          x.tok0 = e.tok0;
          x.n = e.n;
          issue_row<T>(P, R, k + lane, x, false, pol_s, pol_k);
        }
        for (int j = 0; j < n; ++j) st.fill(k + j);
        k += n;
        shead += n;
        __syncwarp();
        if (lane == 0) st_rel_cta(R.misc() + 14, shead);   // the queue entries are free again
        t_idle = clock64();
        continue;
      }
      // dealt units done and nothing queued: finished once no claimed
      // pass-1 unit will come (misc[15]), every request is decided and the
      // next candidate lies past the jobs reserved
      bool done = false;
      if (lane == 0) {
        const unsigned jg = (blockIdx.x + head * (unsigned)G) / upj;
        if (ld_acq_cta(R.misc() + 15) != 0u && shead == ld_acq_cta(R.misc() + 6) &&
            (jg >= (unsigned)P.total ||
             (ld_acq_gpu(P.ctl + kCtlDecided) >= (unsigned)P.B && jg >= ld_acq_gpu(P.ctl + kCtlJobTail))))
          done = true;
        else if (aborted(P)) ok = false;
        else if (clock64() - t_idle > P.wait_limit) {
          // bounded: the wait ends with the job or with every request decided
          raise_abort(P);
          ok = false;
        }
      }
      done = __shfl_sync(0xffffffffu, done, 0) != 0;
      ok = __shfl_sync(0xffffffffu, ok, 0) != 0;
      if (done || !ok) break;
      __nanosleep(100);
    }
    real = k;
  } else {
    // nothing to stream: the prefetched slots become stops once their bytes land
    if (lane == 0)
      for (int j = 0; j < pre; ++j) {
        hdr_of(R.slot(j))->kind = kUnitStop;
        mbar_arrive(R.full() + j);
      }
    stops = pre;
    k = pre;
  }
  if (lane == 0) {
    R.misc()[0] = (unsigned)real;          // units the recorder will see
    R.misc()[4] = (ok && !broken) ? 0u : 1u;  // rows and requests will not complete
    st_rel_cta(R.misc() + 2, 1u);
  }
  // one stop per group (each group leaves at the first stop it claims)
  for (int j = k; stops < kSegGroups; ++j, ++stops) {
    if (!wait_slot(P, R, st, j, lane)) break;
    if (lane == 0) issue_stop(R, j);
    st.fill(j);
  }
  // nothing may land in shared memory after the CTA exits
  if (lane == 0)
    for (int s2 = 0; s2 < kSegSlots; ++s2)
      if ((st.filled >> s2) & 1u) {
        const long long t0 = clock64();
        while (!mbar_test(R.full() + s2, (st.par >> s2) & 1u) && clock64() - t0 < kSegDrainCycles) {
        }
      }
  __syncwarp();
}

// ------------------------------------------------------------ the consumers
// A consumer warp owns a contiguous range of each unit (pass 1: wr tokens
// of one row; pass 2: wr2 tokens of both rows), and lane l a contiguous run
// of it (64 bf16 / 32 fp32 tokens in pass 1, half that per row in pass 2):
// 128 or 64 bytes, so that the run's penalty bits are one word of the
// slot's bitmap.  A lane reads its 16-byte vectors in the order m ^ L (L
// from the lane index), which keeps the eight lanes of every quarter-warp
// on distinct banks.
//
// Penalised tokens: before it loads its run, a lane reads each of its
// penalised tokens (the bits of its run in the slot's bitmap, plus the
// row's extras), adds that token's penalised term to a side sum and
// overwrites the token with -inf in the slot; the hot loop then sums the
// run as it stands.  Every lane touches only its own run.

template <int N>
__device__ __forceinline__ uint32_t neg_word();
template <>
__device__ __forceinline__ uint32_t neg_word<8>() { return 0xFF80FF80u; }
template <>
__device__ __forceinline__ uint32_t neg_word<4>() { return 0xFF800000u; }

// Elements e >= keep of a vector become -inf.
template <int N>
__device__ __forceinline__ void mask_vec(uint4& v, int keep) {
  uint32_t* w = reinterpret_cast<uint32_t*>(&v);
#pragma unroll
  for (int e = 0; e < N; ++e) {
    if (e < keep) continue;
    if constexpr (N == 8) {
      const uint32_t m = (e & 1) ? 0xFFFF0000u : 0x0000FFFFu;
      w[e >> 1] = (w[e >> 1] & ~m) | (0xFF80FF80u & m);
    } else {
      w[e] = 0xFF800000u;
    }
  }
}

template <typename T>
__device__ __forceinline__ float ldz(const unsigned char* p) {
  return to_f32<T>(*reinterpret_cast<const T*>(p));
}

// A logit of the slot becomes -inf.
template <typename T>
__device__ __forceinline__ void set_neg_inf(unsigned char* p) {
  if constexpr (sizeof(T) == 2) *reinterpret_cast<uint16_t*>(p) = 0xFF80u;
  else *reinterpret_cast<uint32_t*>(p) = 0xFF800000u;
}

// 16 bytes of shared memory at a 32-bit shared-window address.  Volatile
// with a memory clobber: no load moves past the slot's release, nor ahead of
// the lane's own -inf stores.
__device__ __forceinline__ uint4 lds16(uint32_t a) {
  uint4 v;
  asm volatile("ld.shared.v4.u32 {%0, %1, %2, %3}, [%4];"
               : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
               : "r"(a)
               : "memory");
  return v;
}

// Penalty bits of a lane's run of `bits` tokens (64, 32 or 16) starting at
// bit `bit0` of the slot's bitmap (bit0 a multiple of `bits`), with the
// row's extras (drafts before the row outside the history) folded in.
// Tokens of the warp's range are [first_tok, first_tok + wn); lane l's run
// starts at first_tok + l * bits.
template <int BITS>
__device__ __forceinline__ unsigned long long run_bits(const unsigned char* bm, int bit0, const SegRowDesc* d,
                                                       int first_tok, int wn, int lane) {
  unsigned long long pm = 0;
  if (lane * BITS < wn) {
    if constexpr (BITS == 64) pm = *reinterpret_cast<const unsigned long long*>(bm + bit0 / 8);
    else if constexpr (BITS == 32) pm = *reinterpret_cast<const uint32_t*>(bm + bit0 / 8);
    else pm = *reinterpret_cast<const uint16_t*>(bm + bit0 / 8);
  }
  const int ne = d->n_extra;
  if (ne > 0) {
    const int e = lane < ne ? d->extras[lane] : -1;
    const int rel = e - first_tok;
    unsigned hit = __ballot_sync(0xffffffffu, e >= 0 && rel >= 0 && rel < wn);
    while (hit) {
      const int kk = __ffs(hit) - 1;
      hit &= hit - 1;
      const int rk = __shfl_sync(0xffffffffu, rel, kk);
      if (lane == rk / BITS) pm |= 1ull << (rk % BITS);
    }
  }
  return pm;
}

// The lane's run (VPL vectors at shared address `run`, `ln` valid tokens)
// into registers, vector m of the result being the run's vector m ^ L;
// tokens past `ln` read as -inf.  A lane with no tokens (ln == 0) reads a
// whole run's worth of the slot beyond its warp's range (still inside the
// slot) and the caller drops its sum: the lanes of a full unit then all
// take the same path.
template <int N, int VPL>
__device__ __forceinline__ void load_run(uint4 (&v)[VPL], uint32_t run, int L, int ln) {
  if (ln == N * VPL || ln == 0) {
    const uint32_t sw = run | ((uint32_t)L << 4);
#pragma unroll
    for (int m = 0; m < VPL; ++m) v[m] = lds16(sw ^ ((uint32_t)m << 4));
  } else {
    const uint32_t NW = neg_word<N>();
#pragma unroll
    for (int m = 0; m < VPL; ++m) {
      const int vi = m ^ L;
      v[m] = make_uint4(NW, NW, NW, NW);
      if (vi * N < ln) {
        v[m] = lds16(run + (uint32_t)vi * 16u);
        if (vi * N + N > ln) mask_vec<N>(v[m], ln - vi * N);
      }
    }
  }
}

// Sum of 2^(z c) over the 8 (bf16) or 4 (fp32) logits of a vector.
template <int N>
__device__ __forceinline__ float2 vec_exp_sum(const uint4& v, float2 c2, float2 acc) {
  float z[N];
  cvt16(v, z);
  const float2 z2 = make_float2(0.f, 0.f);
#pragma unroll
  for (int e = 0; e < N; e += 2) {
    const float2 y = __ffma2_rn(make_float2(z[e], z[e + 1]), c2, z2);
    acc = __fadd2_rn(acc, make_float2(ex2(y.x), ex2(y.y)));
  }
  return acc;
}

// A per-lane sum of 2^(z'c) (reference 0) is trusted inside [2^-100, 2^100]:
// a row's total then stays far inside fp32.  Outside it (or NaN), the
// warp's partial is flagged and the recorder recomputes that range with the
// range's largest logit as the reference.
constexpr float kSumHi = 1.2676506002282294e30f;   // 2^100
constexpr float kSumLo = 7.888609052210118e-31f;   // 2^-100

// Pass 1 of one unit for consumer warp w (0..7 of its group): the sum of
// 2^(z'c) over the warp's tokens, and the row's draft-token logit.  All
// reads of the slot come first (the draft token, the penalised tokens, the
// lane's run into registers); the slot goes back to the producer
// (`release`) before the arithmetic.
template <typename T, typename Rel>
__device__ __forceinline__ void unit_row(const SegParams& P, unsigned char* slot, const SegUnitHdr& h, int w,
                                         int lane, SegUnitRec* rc, Rel&& release) {
  constexpr int N = Vec<T>::N;
  constexpr int VPL = 8;                   // vectors per lane
  constexpr int TPL = N * VPL;             // tokens per lane: 64 bf16, 32 fp32
  const SegRowDesc* d = reinterpret_cast<const SegRowDesc*>(slot + kSegDescOff);
  const float c = d->c, alpha = d->alpha;
  const int wt0 = w * P.g.wr;
  const int wn = max(0, min(P.g.wr, h.n - wt0));
  const int ln = max(0, min(TPL, wn - lane * TPL));   // this lane's tokens
  const unsigned char* run = slot + (size_t)(wt0 + lane * TPL) * sizeof(T);
  // the draft token's logit (row r's draft token lies in one lane's run)
  if (d->x >= 0) {
    const int rel = d->x - h.tok0 - wt0;
    if (rel >= 0 && rel < wn && lane == rel / TPL) {
      float z = ldz<T>(run + (size_t)(rel % TPL) * sizeof(T));
      if (d->x_pen) z = penalize(z, alpha);
      rc->zx = z;
      rc->has_zx = 1;
    }
  }
  // penalised tokens: their own terms, then -inf in the slot
  const unsigned long long pm = run_bits<TPL>(slot + kSegLogitBytes, wt0 + lane * TPL, d, h.tok0 + wt0, wn, lane);
  float side = 0.f;
  for (unsigned long long mm = pm; mm; mm &= mm - 1) {
    const int e = __ffsll((long long)mm) - 1;
    if (e < ln) {
      unsigned char* q = const_cast<unsigned char*>(run) + (size_t)e * sizeof(T);
      side += ex2(__fmul_rn(penalize(ldz<T>(q), alpha), c));
      set_neg_inf<T>(q);
    }
  }
  uint4 v[VPL];
  load_run<N, VPL>(v, (uint32_t)__cvta_generic_to_shared(run), lane & 7, ln);
  release();
  const float2 c2 = make_float2(c, c);
  float2 a0 = make_float2(0.f, 0.f), a1 = make_float2(0.f, 0.f);
#pragma unroll
  for (int m = 0; m < VPL; m += 2) {
    a0 = vec_exp_sum<N>(v[m], c2, a0);
    a1 = vec_exp_sum<N>(v[m + 1], c2, a1);
  }
  const float s = ln > 0 ? (a0.x + a0.y) + (a1.x + a1.y) + side : 0.f;
  // a lane outside the trusted range flags the warp's partial (S < 0)
  const bool bad = __any_sync(0xffffffffu, !(s <= kSumHi) || (s < kSumLo && ln > 0));
  const float S = warp_sum(s);
  if (lane == 0) rc->r[w] = bad ? make_float2(0.f, -1.f) : make_float2(0.f, S);
}

// Residual terms of two packed token pairs in units of fp: max(p - q, 0) / fp
// with p = 2^(zp c - Lp) fp and q = 2^(zq c - Lq) fq, as max(eq * -r + ep, 0)
// (ep, eq the two powers, r = fq / fp) in one fused step.  Rows that agree
// give exactly 0 whichever way the compiler schedules it.
__device__ __forceinline__ float2 pair_terms(float2 zp, float2 zq, float2 c2, float2 np2, float2 nq2, float2 mr2) {
  const float2 a = __ffma2_rn(zp, c2, np2);
  const float2 bq = __ffma2_rn(zq, c2, nq2);
  const float2 df = __ffma2_rn(make_float2(ex2(bq.x), ex2(bq.y)), mr2, make_float2(ex2(a.x), ex2(a.y)));
  return make_float2(fmaxf(df.x, 0.f), fmaxf(df.y, 0.f));
}

// One token's residual term in units of fp, as pair_terms computes it.
__device__ __forceinline__ float pair_term(float zp, float zq, float c, float Lp, float Lq, float r) {
  return fmaxf(__fmaf_rn(ex2(fmaf(zq, c, -Lq)), -r, ex2(fmaf(zp, c, -Lp))), 0.f);
}

// Pass 2 of one half-segment unit for consumer warp w: the warp's share of
// sum max(p - q, 0), p = 2^(z'c - Lp) fp, q = 2^(z'c - Lq) fq (summed in
// units of fp, then scaled).
template <typename T, typename Rel>
__device__ __forceinline__ void unit_pair(const SegParams& P, unsigned char* slot, const SegUnitHdr& h, int w,
                                          int lane, SegUnitRec* rc, Rel&& release) {
  constexpr int N = Vec<T>::N;
  constexpr int VPL = 4;                   // vectors per lane and row
  constexpr int TPL = N * VPL;             // tokens per lane: 32 bf16, 16 fp32
  const SegRowDesc* d = reinterpret_cast<const SegRowDesc*>(slot + kSegDescOff);
  const SegJobDesc* jd = reinterpret_cast<const SegJobDesc*>(slot + kSegDescOff + sizeof(SegRowDesc));
  const float c = d->c, alpha = d->alpha, Lp = jd->Lp, Lq = jd->Lq, fp = jd->fp;
  const float r = __fdiv_rn(jd->fq, fp);
  const int wt0 = w * P.g.wr2;
  const int wn = max(0, min(P.g.wr2, h.n - wt0));
  const int ln = max(0, min(TPL, wn - lane * TPL));
  const unsigned char* rp = slot + (size_t)(wt0 + lane * TPL) * sizeof(T);
  const unsigned char* rq = rp + kSegLogitBytes / 2;
  // penalised tokens: their own residual terms, then -inf in both rows
  const unsigned long long pm = run_bits<TPL>(slot + kSegLogitBytes, wt0 + lane * TPL, d, h.tok0 + wt0, wn, lane);
  float side = 0.f;
  for (unsigned long long mm = pm; mm; mm &= mm - 1) {
    const int e = __ffsll((long long)mm) - 1;
    if (e < ln) {
      unsigned char* qp = const_cast<unsigned char*>(rp) + (size_t)e * sizeof(T);
      unsigned char* qq = const_cast<unsigned char*>(rq) + (size_t)e * sizeof(T);
      side += pair_term(penalize(ldz<T>(qp), alpha), penalize(ldz<T>(qq), alpha), c, Lp, Lq, r);
      set_neg_inf<T>(qp);
      set_neg_inf<T>(qq);
    }
  }
  // the lane's run of both rows into registers, then the slot goes back
  uint4 vp[VPL], vq[VPL];
  const uint32_t sp = (uint32_t)__cvta_generic_to_shared(rp);
  load_run<N, VPL>(vp, sp, (lane >> 1) & 3, ln);
  load_run<N, VPL>(vq, sp + (uint32_t)(kSegLogitBytes / 2), (lane >> 1) & 3, ln);
  release();
  const float2 c2 = make_float2(c, c), np2 = make_float2(-Lp, -Lp), nq2 = make_float2(-Lq, -Lq);
  const float2 mr2 = make_float2(-r, -r);
  float2 acc = make_float2(0.f, 0.f);
#pragma unroll
  for (int m = 0; m < VPL; ++m) {
    float zp[N], zq[N];
    cvt16(vp[m], zp);
    cvt16(vq[m], zq);
#pragma unroll
    for (int e = 0; e < N; e += 2)
      acc = __fadd2_rn(acc, pair_terms(make_float2(zp[e], zp[e + 1]), make_float2(zq[e], zq[e + 1]), c2, np2, nq2,
                                       mr2));
  }
  const float S = warp_sum(ln > 0 ? acc.x + acc.y + side : 0.f) * fp;
  if (lane == 0) rc->r[w] = make_float2(S, 0.f);
}

// Group g's warps take units g, g + kSegGroups, ...: each warp its own share
// of every such unit, at its own pace (no barrier between the group's
// warps); the slot goes back to the producer once all of them have read it.
template <typename T>
__device__ void consumer(const SegParams& P, const Ring& R, int cw, int lane) {
  const int grp = cw / kSegGroupWarps, w = cw % kSegGroupWarps;
  for (int k = grp;; k += kSegGroups) {
    const int s = k % kSegSlots;
    if (!ring_wait(P, R.full() + s, (uint32_t)((k / kSegSlots) & 1))) break;
    unsigned char* slot = R.slot(s);
    const SegUnitHdr h = *hdr_of(slot);
    if (h.kind == kUnitStop) break;
    // the slot goes back to the producer as soon as the warp has read it
    auto release = [&]() {
      __syncwarp();
      if (lane == 0) mbar_arrive(R.empty() + s);
    };
    SegUnitRec* rc = R.rec(k);
    if (h.kind == kUnitRow) unit_row<T>(P, slot, h, w, lane, rc, release);
    else unit_pair<T>(P, slot, h, w, lane, rc, release);
    __syncwarp();
    if (lane == 0) {
      __threadfence_block();
      atomicAdd(&rc->ndone, 1u);
    }
  }
}

// ------------------------------------------------------------ draws and records
// Inverse CDF inside the token range [a, a + n) (a a multiple of 32) of a
// row, or of the residual max(p - q, 0) of a row pair: the smallest v whose
// prefix mass (from a) exceeds t; the last token with mass if t is out of
// reach.  The per-token arithmetic is that of the streaming passes.
// A lane's 32 consecutive tokens t0 .. t0+31 of a row (t0 a multiple of 32):
// vector loads, each only where it starts before `end` (a vector that starts
// inside the row ends inside its padded stride).
template <typename T>
struct Run32 {
  static constexpr int NV = 32 * (int)sizeof(T) / 16;   // 4 (bf16) or 8 (fp32) vectors
  uint4 v[NV];
  __device__ __forceinline__ void load(const T* row, int t0, int end) {
    constexpr int N = Vec<T>::N;
#pragma unroll
    for (int q = 0; q < NV; ++q)
      v[q] = t0 + q * N < end ? __ldcg(reinterpret_cast<const uint4*>(row + t0) + q) : make_uint4(0u, 0u, 0u, 0u);
  }
  __device__ __forceinline__ float at(int j) const {   // j a compile-time index after unrolling
    constexpr int N = Vec<T>::N;
    const uint32_t* w = reinterpret_cast<const uint32_t*>(&v[j / N]);
    if constexpr (N == 8) {
      const uint32_t x = w[(j % N) >> 1];
      return __uint_as_float((j & 1) ? (x & 0xffff0000u) : (x << 16));
    } else {
      return __uint_as_float(w[j % N]);
    }
  }
};

template <typename T, bool PAIR>
__device__ __forceinline__ float draw_term(float zp, float zq, bool pen, const SegRowDesc& d, float Lp, float fp,
                                           float Lq, float fq) {
  if (pen) zp = penalize(zp, d.alpha);
  if (!PAIR) return __fmul_rn(ex2(fmaf(zp, d.c, -Lp)), fp);
  if (pen) zq = penalize(zq, d.alpha);
  return __fmul_rn(pair_term(zp, zq, d.c, Lp, Lq, __fdiv_rn(fq, fp)), fp);
}

// A warp's staging area for one draw: the range's logits (a row's range at
// `p`, or both rows' at `p` and `q`), its penalty words, and the mbarrier the
// bulk copies complete on, with the parity of its next phase.
struct DrawBuf {
  unsigned char* p;
  unsigned char* q;
  uint32_t* bits;
  uint64_t* bar;
  unsigned* phase;
};

__device__ __forceinline__ DrawBuf draw_buf(const Ring& R, int i) {
  unsigned char* area = R.draw_area(i);
  DrawBuf db;
  db.p = area;
  db.q = area + kDrawBytes / 2;
  db.bits = reinterpret_cast<uint32_t*>(area + kDrawBytes);
  db.bar = reinterpret_cast<uint64_t*>(area + kDrawBytes + 256);
  db.phase = reinterpret_cast<unsigned*>(area + kDrawBytes + 256 + 8);
  return db;
}

// Inverse CDF inside the token range [a, a + n) (a a multiple of 32) of a
// row, or of the residual max(p - q, 0) of a row pair: the smallest v whose
// prefix mass (from a) exceeds t; the last token with mass if t is out of
// reach.  p = 2^(z'c - Lp) * fp and q = 2^(z'c - Lq) * fq, as in the
// streaming passes.  The range (at most kDrawBytes per row) comes into the
// warp's DrawBuf with one bulk copy per row, its penalty words with plain
// loads alongside; the walk then reads shared memory only.
template <typename T, bool PAIR>
__device__ int range_draw(const SegParams& P, const DrawBuf& db, int rp_row, int rq_row, int a, int n,
                          const SegRowDesc& d, float Lp, float fp, float Lq, float fq, int b, double t, int lane) {
  const uint32_t bytes = tma_bytes(n, sizeof(T));
  unsigned par = 0;
  if (lane == 0) {
    par = *db.phase;
    mbar_arrive_expect(db.bar, PAIR ? 2 * bytes : bytes);
    const uint64_t pol = l2_policy_evict_first();
    bulk_g2s(db.p, row_ptr<T>(P, rp_row) + (size_t)a * sizeof(T), bytes, db.bar, pol);
    if (PAIR) bulk_g2s(db.q, row_ptr<T>(P, rq_row) + (size_t)a * sizeof(T), bytes, db.bar, pol);
  }
  // penalty words of the range, with the row's extras
  const uint32_t* bm = P.bitmap + (size_t)b * (P.g.bm_bytes / 4) + (a >> 5);
  const int nw = (n + 31) >> 5;
  for (int w = lane; w < nw; w += 32) db.bits[w] = __ldcg(bm + w);
  __syncwarp();
  if (lane < d.n_extra) {
    const int e = d.extras[lane] - a;
    if (e >= 0 && e < n) atomicOr(db.bits + (e >> 5), 1u << (e & 31));
  }
  par = __shfl_sync(0xffffffffu, par, 0);
  bool ok = true;
  if (lane == 0) {
    ok = ring_wait(P, db.bar, par);
    *db.phase = par ^ 1u;
  }
  ok = __shfl_sync(0xffffffffu, (int)ok, 0) != 0;
  __syncwarp();
  if (!ok) return -1;
  auto zp_at = [&](int i) { return ldz<T>(db.p + (size_t)i * sizeof(T)); };
  auto zq_at = [&](int i) { return PAIR ? ldz<T>(db.q + (size_t)i * sizeof(T)) : 0.f; };
  int found = -1, lastpos = -1;
  double carry = 0.0;
  for (int base = 0; base < n && found < 0; base += 1024) {
    const int t0 = base + 32 * lane;
    const int cnt = max(0, min(32, n - t0));
    const uint32_t pw = cnt > 0 ? db.bits[t0 >> 5] : 0u;
    // the lane's 32 terms summed in fp32 with compensation (the part has
    // little fp64 throughput); the warp's prefix in fp64
    float ls = 0.f, lc = 0.f;
    int mylast = -1;
    for (int j = 0; j < cnt; ++j) {
      const float r = draw_term<T, PAIR>(zp_at(t0 + j), zq_at(t0 + j), (pw >> j) & 1u, d, Lp, fp, Lq, fq);
      const float y = __fsub_rn(r, lc), tt = __fadd_rn(ls, y);
      lc = __fsub_rn(__fsub_rn(tt, ls), y);
      ls = tt;
      if (r > 0.f) mylast = a + t0 + j;
    }
    const double lsum = (double)ls;
    const double incl = warp_incl_scan_d(lsum, lane);
    const double tot = __shfl_sync(0xffffffffu, incl, 31);
    const unsigned hit = __ballot_sync(0xffffffffu, carry + incl > t);
    if (hit) {
      // lane L's run again, one token per lane: the terms' prefix in token
      // order (a warp scan) against what is left of t after the lanes before
      // L; rounding can leave it short, and then the run's last token with
      // mass is the draw
      const int L = __ffs(hit) - 1;
      const int tL = __shfl_sync(0xffffffffu, t0, L), cL = __shfl_sync(0xffffffffu, cnt, L);
      const uint32_t pL = __shfl_sync(0xffffffffu, pw, L);
      const double rest = t - (carry + __shfl_sync(0xffffffffu, incl - lsum, L));
      const float r = lane < cL ? draw_term<T, PAIR>(zp_at(tL + lane), zq_at(tL + lane), (pL >> lane) & 1u, d, Lp, fp,
                                                     Lq, fq)
                                : 0.f;
      const float pre = warp_incl_scan(r, lane);
      const unsigned over = __ballot_sync(0xffffffffu, lane < cL && (double)pre > rest);
      found = over ? a + tL + __ffs(over) - 1 : __shfl_sync(0xffffffffu, mylast, L);
    }
    int ml = mylast;
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) ml = max(ml, __shfl_xor_sync(0xffffffffu, ml, o));
    if (ml >= 0) lastpos = ml;
    carry += tot;
  }
  __syncwarp();     // the buffer is free again once every lane is done with it
  return found >= 0 ? found : lastpos;
}

// The owning part of a draw over `nparts` (<= 512) part masses (mass(j) for
// part j) at t = u * total: returns the part, sets *before to the mass
// before it and *total to the total mass.  The masses go to the warp's draw
// area (as doubles, at most kDrawBytes), lane l summing parts
// l*per .. l*per + per - 1; the lane that holds t walks its parts again.
template <typename F>
__device__ int owning_part(int nparts, F&& mass, double u, double* before, double* total, const DrawBuf& db,
                           int lane) {
  double* m = reinterpret_cast<double*>(db.p);
  for (int j = lane; j < nparts; j += 32) m[j] = mass(j);
  __syncwarp();
  const int per = (nparts + 31) / 32;
  const int j0 = min(lane * per, nparts), j1 = min(j0 + per, nparts);
  double ls = 0.0;
  int lp = -1;
  for (int j = j0; j < j1; ++j) {
    ls += m[j];
    if (m[j] > 0.0) lp = j;
  }
  const double incl = warp_incl_scan_d(ls, lane);
  const double tot = __shfl_sync(0xffffffffu, incl, 31);
  *total = tot;
  const double t = u * tot;
  const unsigned hit = __ballot_sync(0xffffffffu, incl > t && ls > 0.0);
  int part = -1;
  double bef = 0.0;
  if (hit) {
    const int L = __ffs(hit) - 1;
    if (lane == L) {
      // this lane's first part that takes t, and its last part with mass
      double acc = incl - ls, lb = 0.0;
      for (int j = j0; j < j1; ++j) {
        if (m[j] > 0.0) {
          if (part < 0 && acc + m[j] > t) {
            part = j;
            bef = acc;
          }
          lb = acc;
        }
        acc += m[j];
      }
      if (part < 0) {       // rounding: the lane's last part with mass
        part = lp;
        bef = lb;
      }
    }
    part = __shfl_sync(0xffffffffu, part, L);
    bef = __shfl_sync(0xffffffffu, bef, L);
  } else {
    // t out of reach (rounding): the last part with mass
    const unsigned has = __ballot_sync(0xffffffffu, lp >= 0);
    if (has) {
      const int L = 31 - __clz(has);
      double lb = 0.0;
      if (lane == L) {
        double acc = incl - ls;
        for (int j = j0; j < lp; ++j) acc += m[j];
        lb = acc;
      }
      part = __shfl_sync(0xffffffffu, lp, L);
      bef = __shfl_sync(0xffffffffu, lb, L);
    }
  }
  __syncwarp();     // the draw area is free again
  *before = bef;
  return part;
}

// A row's log2 normaliser M + log2 S as an fp32 value Lf and a factor f with
// 2^(y - M) / S = 2^(y - Lf) * f: f = 2^(Lf - M) / S makes up for the
// rounding of Lf, so that y - Lf stays small for the tokens that carry the
// mass (their exponent keeps its precision) and no probability is scaled.
// fp32 throughout: the part has little fp64 throughput.
__device__ __forceinline__ void split_norm(float M, float S, float* Lf, float* f) {
  const float L = M + log2f(S);
  *Lf = L;
  *f = exp2f(L - M) / S;
}

// The pass-1 partial of unit u, warp w, recomputed from global memory when
// the consumers flagged it: the range's largest penalised logit (units of
// z'c) as the reference, and the sum of 2^(z'c - reference).
template <typename T>
__device__ float2 fixup_partial(const SegParams& P, int u, int w, int lane) {
  const int r = u / P.g.nseg, sg = u % P.g.nseg;
  const SegRowDesc d = ld_desc(P.rowdesc + r);
  const int a = sg * P.g.seg + w * P.g.wr;
  const int n = min(P.g.wr, P.V - a);
  if (n <= 0) return make_float2(0.f, 0.f);
  const T* row = reinterpret_cast<const T*>(row_ptr<T>(P, d.src));
  const uint32_t* bm = P.bitmap + (size_t)d.b * (P.g.bm_bytes / 4);
  float mx = -INFINITY, sum = 0.f;
  for (int pass = 0; pass < 2; ++pass) {
    for (int base = a; base < a + n; base += 1024) {
      const int t0 = base + 32 * lane;
      const int end = a + n;
      const int cnt = max(0, min(32, end - t0));
      Run32<T> rv;
      rv.load(row, t0, end);
      uint32_t pw = cnt > 0 ? __ldcg(bm + (t0 >> 5)) : 0u;
      for (int k = 0; k < d.n_extra; ++k) {
        const int e = d.extras[k];
        if (e >= t0 && e < t0 + 32) pw |= 1u << (e - t0);
      }
#pragma unroll
      for (int j = 0; j < 32; ++j) {
        if (j < cnt) {
          float z = rv.at(j);
          if ((pw >> j) & 1u) z = penalize(z, d.alpha);
          if (pass == 0) mx = fmaxf(mx, z);
          else sum += ex2(fmaf(z, d.c, -mx * d.c));
        }
      }
    }
    if (pass == 0) {
      mx = warp_max(mx);
      if (!(mx > -INFINITY)) return make_float2(0.f, 0.f);   // nothing finite (NaN makes the sum NaN below)
    }
  }
  return make_float2(mx * d.c, warp_sum(sum));
}

// Draw from p of target row r (the bonus token, or a rejection whose
// residual mass is 0) with uniform u, from the row's pass-1 masses.
template <typename T>
__device__ int draw_from_p(const SegParams& P, const DrawBuf& db, int r, float u, int lane) {
  const SegRowStat rs = ld_stat(P.rowstat + r);
  const float2* pp = P.part1 + (size_t)r * P.g.nseg * kSegGroupWarps;
  const float M = rs.M, S = rs.S;
  auto mass = [&](int j) -> double {
    const float2 v = __ldcg(pp + j);
    return v.y == 0.f ? 0.0 : (double)(v.y * exp2f(v.x - M) / S);
  };
  double before, total;
  const int part = owning_part(P.g.nseg * kSegGroupWarps, mass, (double)u, &before, &total, db, lane);
  if (part < 0) return -1;
  const SegRowDesc d = ld_desc(P.rowdesc + r);
  const int a = (part / kSegGroupWarps) * P.g.seg + (part % kSegGroupWarps) * P.g.wr;
  const int n = min(P.g.wr, P.V - a);
  float L, f;
  split_norm(M, S, &L, &f);
  return range_draw<T, false>(P, db, d.src, -1, a, n, d, L, f, 0.f, 0.f, d.b, (double)u * total - before, lane);
}

// Draw from the residual max(p - q, 0) of position p with uniform u, from
// the position's pass-2 masses; -2 if the residual mass is 0.
template <typename T>
__device__ int draw_residual(const SegParams& P, const DrawBuf& db, int p, int b, float u, int lane) {
  const float* pp = P.part2 + (size_t)p * P.g.upj * kSegGroupWarps;
  auto mass = [&](int j) -> double { return (double)__ldcg(pp + j); };
  double before, total;
  const int part = owning_part(P.g.upj * kSegGroupWarps, mass, (double)u, &before, &total, db, lane);
  if (!(total > 0.0)) return -2;
  if (part < 0) return -1;
  const SegJobDesc jd = ld_job(P.jobdesc + p);
  const SegRowDesc d = ld_desc(P.posdesc + p);
  const int h = part / kSegGroupWarps, w = part % kSegGroupWarps;
  const int a = (h >> 1) * P.g.seg + (h & 1) * (P.g.seg / 2) + w * P.g.wr2;
  const int n = min(P.g.wr2, P.V - a);
  return range_draw<T, true>(P, db, p + b, P.NT + p, a, n, d, jd.Lp, jd.fp, jd.Lq, jd.fq, b, (double)u * total - before,
                             lane);
}

// Emits request b's tokens once every decision it needs is known: the
// accepted prefix up to the first rejection j, then the draw from the
// residual of j (from p_j if that residual has no mass), or the bonus token
// from the last target row when every draft is accepted.
template <typename T>
__device__ void finalize(const SegParams& P, const DrawBuf& db, int b, int lane) {
  const int d0 = __ldg(P.cu_draft + b), K = __ldg(P.cu_draft + b + 1) - d0, off = d0 + b;
  bool acc = true;
  if (lane < K) {
    const SegPos ps = ld_pos(P.pos + d0 + lane);
    acc = ps.state == 1 || (ps.state == 2 && ps.acc);
  }
  const unsigned rej = __ballot_sync(0xffffffffu, lane < K && !acc);
  const int j = rej ? __ffs(rej) - 1 : K;
  const float ufin = __ldg(P.uniforms + off + K);
  const int base = 2 * d0 + b;      // the request's first row
  int tok = -1;
  if (j < K) {
    tok = draw_residual<T>(P, db, d0 + j, b, ufin, lane);
    if (tok == -2) tok = draw_from_p<T>(P, db, base + 2 * j, ufin, lane);
  } else if (!(P.flags & 1u)) {
    tok = draw_from_p<T>(P, db, base + 2 * K, ufin, lane);
  }
  for (int s = lane; s <= K; s += 32) {
    int o = -1;
    if (s < j) o = __ldg(P.draft_tokens + d0 + s);
    else if (s == j) o = tok;
    P.out_tokens[off + s] = o;
  }
  if (lane == 0) {
    P.out_accepted[b] = j;
    if (P.out_status) P.out_status[b] = 0;
    P.req_done[b] = 1u;
  }
}

// The request's rows are all in: status, the decisions pass 1 fixes, and
// the jobs (second passes) for the rest.  Returns the positions whose job
// the caller then waits for (0: the request is finished).
template <typename T>
__device__ unsigned request_decide(const SegParams& P, int b, int lane, bool& ready) {
  ready = false;
  const int d0 = __ldg(P.cu_draft + b), K = __ldg(P.cu_draft + b + 1) - d0, off = d0 + b;
  const int base = 2 * d0 + b;      // the request's first row
  int st = __ldcg(P.req_status + b);
  int fl = 0;
  for (int j = lane; j <= 2 * K; j += 32) fl |= ld_stat(P.rowstat + base + j).flags;
  st |= warp_or(fl);
  const bool tv_only = P.mode == kModeTvOnly;
  unsigned need = 0;
  if (st == 0 && K > 0) {
    const float D = __ldg(P.tv_budget + b);
    int state = 1;
    if (lane < K) {
      const SegRowStat sp = ld_stat(P.rowstat + base + 2 * lane), sq = ld_stat(P.rowstat + base + 2 * lane + 1);
      state = tv_only ? 2 : bound_decision(sp.px, sq.px, D, __ldg(P.uniforms + off + lane));
      SegPos ps;
      ps.state = state;
      ps.px = sp.px;
      ps.qx = sq.px;
      ps.acc = 0;
      ps.d = 0.f;
      ps.theta = 0.f;
      ps.b = b;
      ps.pad = 0;
      P.pos[d0 + lane] = ps;
    }
    const unsigned kmask = K >= 32 ? 0xffffffffu : ((1u << K) - 1u);
    const unsigned rej = __ballot_sync(0xffffffffu, state == 0) & kmask;
    const unsigned und = __ballot_sync(0xffffffffu, state == 2) & kmask;
    const int js = rej ? __ffs(rej) - 1 : K;
    const unsigned below = js >= 32 ? 0xffffffffu : ((1u << js) - 1u);
    // undecided tests before the first certain rejection, and that
    // rejection's residual
    need = tv_only ? kmask : ((und & below) | (js < K ? (1u << js) : 0u));
    if (need) {
      if ((need >> lane) & 1u) {
        const SegRowStat sp = ld_stat(P.rowstat + base + 2 * lane), sq = ld_stat(P.rowstat + base + 2 * lane + 1);
        SegJobDesc jd;
        split_norm(sp.M, sp.S, &jd.Lp, &jd.fp);
        split_norm(sq.M, sq.S, &jd.Lq, &jd.fq);
        P.jobdesc[d0 + lane] = jd;
        fence_proxy_async_global();
      }
      __syncwarp();
      if (lane == 0) {
        P.req_need[b] = (unsigned)__popc(need);
        unsigned slot = atom_add_gpu(P.ctl + kCtlJobTail, (unsigned)__popc(need));
        for (unsigned m = need; m; m &= m - 1) {
          const int i = __ffs(m) - 1;
          const unsigned long long e =
              (unsigned long long)(unsigned)(d0 + i + 1) | ((unsigned long long)(unsigned)b << 32);
          st_rel_gpu64(P.jobs + 2 * slot++, e);
        }
      }
      __syncwarp();
    }
  }
  if (!need) {
    if (st != 0) {
      if (tv_only) {
        for (int i = lane; i < K; i += 32) {
          P.out_tv[d0 + i] = NAN;
          P.out_theta[d0 + i] = NAN;
          if (P.out_px) P.out_px[d0 + i] = NAN;
          if (P.out_qx) P.out_qx[d0 + i] = NAN;
        }
      } else {
        for (int s = lane; s <= K; s += 32) P.out_tokens[off + s] = -1;
        if (lane == 0) {
          P.out_accepted[b] = -1;
          if (P.out_status) P.out_status[b] = st;
        }
      }
      if (lane == 0) P.req_done[b] = 1u;
    } else if (!tv_only) {
      ready = true;       // every decision is known: the tokens can be drawn
    } else if (lane == 0) {
      P.req_done[b] = 1u;
    }
  }
  __syncwarp();
  if (lane == 0) red_add_gpu(P.ctl + kCtlDecided, 1u);
  return need;
}

// Row r's units are all in: its statistics and the probability of its
// draft token; then one more row of its request is in.
template <typename T>
__device__ void row_combine(const SegParams& P, int r, int lane) {
  const int np = P.g.nseg * kSegGroupWarps;
  const float2* pp = P.part1 + (size_t)r * np;
  float M = 0.f, S = 0.f;
  for (int j0 = 0; j0 < np; j0 += 256) {
    float2 v[8];
#pragma unroll
    for (int q = 0; q < 8; ++q) {
      const int j = j0 + q * 32 + lane;
      v[q] = j < np ? __ldcg(pp + j) : make_float2(0.f, 0.f);
    }
#pragma unroll
    for (int q = 0; q < 8; ++q) pair_merge(M, S, v[q].x, v[q].y);
  }
  const int b = __ldcg(&P.rowdesc[r].b), x = __ldcg(&P.rowdesc[r].x);
  const float c = __ldcg(&P.rowdesc[r].c);
  const float zx = x >= 0 ? __ldcg(P.zx + r) : 0.f;
  warp_pair(M, S);
  int flags = 0;
  if (!(S > 0.f) || !(S < INFINITY)) flags = kStatusBadLogits;
  float px = 0.f;
  if (x >= 0 && flags == 0) px = exp2f(fmaf(zx, c, -M)) / S;
  if (lane == 0) {
    SegRowStat rs;
    rs.M = M;
    rs.S = S;
    rs.px = px;
    rs.flags = flags;
    P.rowstat[r] = rs;
    red_add_gpu(P.req_rows + b, 1u);
  }
}

// Position p's pass-2 units are all in: d = TV(p, q) (the residual mass),
// theta = min(1, D/d) (1 when d <= D), pi(x) and the acceptance test.
template <typename T>
__device__ void job_finish(const SegParams& P, int p, int lane) {
  const int np = P.g.upj * kSegGroupWarps;
  const float* pp = P.part2 + (size_t)p * np;
  double s = 0.0;
  for (int j0 = 0; j0 < np; j0 += 256) {
    float v[8];
#pragma unroll
    for (int q = 0; q < 8; ++q) {
      const int j = j0 + q * 32 + lane;
      v[q] = j < np ? __ldcg(pp + j) : 0.f;
    }
#pragma unroll
    for (int q = 0; q < 8; ++q) s += (double)v[q];
  }
  s = warp_sum_d(s);
  const SegPos ps = ld_pos(P.pos + p);
  const int b = ps.b;
  const float d = (float)fmin(fmax(s, 0.0), 1.0);
  const float D = __ldg(P.tv_budget + b);
  const float theta = d <= D ? 1.f : __fdiv_rn(D, d);
  const float pi = fmaf(theta, ps.qx, (1.f - theta) * ps.px);
  if (lane == 0) {
    if (P.mode == kModeTvOnly) {
      P.out_tv[p] = d;
      P.out_theta[p] = theta;
      if (P.out_px) P.out_px[p] = ps.px;
      if (P.out_qx) P.out_qx[p] = ps.qx;
    } else {
      const float u = __ldg(P.uniforms + p + b);
      P.pos[p].acc = (u * ps.qx < pi) ? 1 : 0;
      P.pos[p].d = d;
      P.pos[p].theta = theta;
    }
  }
  __syncwarp();
}

// Items of this CTA (i-th item = c + i * G) handled once ready, polled 8 at
// a time in one round trip; `done` marks the window's handled items.
struct Owned {
  int n = 0;        // items owned
  int next = 0;     // first item not yet handled
  unsigned done = 0;  // handled items among next .. next + 31
  __device__ void advance() {
    while (next < n && (done & 1u)) {
      done >>= 1;
      ++next;
    }
  }
};

// The recorder warp: takes each unit its consumers have finished (in ring
// order), recomputes the partials they flagged, stores the partials (and the
// captured draft-token logit) to global memory and counts the unit against
// its row (pass 1) or position (pass 2).  It never waits on other CTAs, so
// the producer's record ring keeps moving.
template <typename T>
__device__ void recorder(const SegParams& P, const Ring& R, int lane) {
  int k = 0;
  long long t_last = clock64();
  // the producer's second-pass candidates (see the producer): lane j loads
  // the job entry of candidate cb + j; the published ones, in order, are
  // queued for the producer
  const unsigned G = gridDim.x, upj = (unsigned)P.g.upj, njob = (unsigned)P.total;
  const int* cu = cu_of(P, R);
  const int dealt = dealt_units(P), n_dealt = static_units(P), n_units = P.NR * P.g.nseg;
  unsigned stail = 0;       // claimed pass-1 units queued
  bool steal_done = dealt >= n_units;
  if (steal_done && lane == 0) st_rel_cta(R.misc() + 15, 1u);
  unsigned cb = 0, jtail = 0;
  unsigned long long ent = 0;
  bool pend = false, jq_done = false;
  for (;;) {
    bool progress = false;
    // 1. units finished by all their warps, in ring order
    // record slot i counts kSegGroupWarps per use: unit k is done once its
    // slot's count reaches kSegGroupWarps * (k / kSegRecN + 1)
    const bool fin = ld_acq_cta(&R.rec(k + lane)->ndone) ==
                     (unsigned)(kSegGroupWarps * ((k + lane) / kSegRecN + 1));
    const unsigned fm = __ballot_sync(0xffffffffu, fin);
    const int done = k + (fm == 0xffffffffu ? 32 : __ffs(~fm) - 1);
    const int nd = min(done - k, 32);
    if (nd > 0) {
      progress = true;
      // the units' results go to global memory (lane w: warp w's partial) ...
      for (int j = 0; j < nd; ++j) {
        const SegUnitRec* rc = R.rec(k + j);
        const int kind = rc->kind, id = rc->id;
        float2 v = make_float2(0.f, 0.f);
        if (lane < kSegGroupWarps) v = rc->r[lane];
        // partials the consumers could not trust are recomputed here
        unsigned fx = __ballot_sync(0xffffffffu, kind == kUnitRow && lane < kSegGroupWarps && v.y < 0.f);
        while (fx) {
          const int L = __ffs(fx) - 1;
          fx &= fx - 1;
          const float2 f = fixup_partial<T>(P, id, L, lane);
          if (lane == L) v = f;
        }
        if (lane < kSegGroupWarps) {
          if (kind == kUnitRow) P.part1[(size_t)id * kSegGroupWarps + lane] = v;
          else P.part2[((size_t)id * P.g.upj + rc->part) * kSegGroupWarps + lane] = v.x;
        } else if (lane == kSegGroupWarps && kind == kUnitRow && rc->has_zx) {
          P.zx[id / P.g.nseg] = rc->zx;
        }
      }
      __syncwarp();
      // ... then each counts against its row or position (fire and forget)
      if (lane < nd) {
        const SegUnitRec* rc = R.rec(k + lane);
        red_add_gpu(rc->kind == kUnitRow ? P.row_cnt + rc->id / P.g.nseg : P.job_cnt + rc->id, 1u);
      }
      __syncwarp();
      k += nd;
      if (lane == 0) st_rel_cta(R.misc() + 1, (unsigned)k);
    }
    // 2. second-pass candidates: last round's published entries join the
    //    queue (as far as it has room), then the next window is loaded
    //    (once every CTA has cleared its part of the job list: misc[5])
    if (!jq_done && ld_acq_cta(R.misc() + 5) != 0u) {
      if (pend) {
        const unsigned jg = (blockIdx.x + (cb + lane) * G) / upj;
        const bool pub = jg < njob && (unsigned)(ent & 0xffffffffull) != 0u;
        const unsigned pm = __ballot_sync(0xffffffffu, pub);
        int n = pm == 0xffffffffu ? 32 : __ffs(~pm) - 1;
        n = min(n, kSegJq - (int)(jtail - ld_acq_cta(R.misc() + 9)));
        if (n > 0) {
          asm volatile("fence.acq_rel.gpu;" ::: "memory");   // each entry's release happens before the queue's
          if (lane < n) R.jq()[(jtail + lane) % kSegJq] = ent;
          __syncwarp();
          jtail += n;
          cb += n;
          if (lane == 0) st_rel_cta(R.misc() + 8, jtail);
        }
        pend = false;
      }
      if ((blockIdx.x + cb * G) / upj >= njob || ld_acq_cta(R.misc() + 2) != 0u) {
        jq_done = true;       // no candidate left, or the producer has finished
      } else {
        const unsigned jg = (blockIdx.x + (cb + lane) * G) / upj;
        ent = jg < njob ? ld_relaxed_gpu64(P.jobs + 2 * jg) : 0ull;
        pend = true;
      }
    }
    // 3. pass-1 units past the dealt ones: once the producer's dealt units
    //    are nearly issued (misc[13]), claim kStealChunk at a time while the
    //    queue holds fewer than kStealAhead; lane j works out the geometry
    //    of the j-th
    if (!steal_done && stail - ld_acq_cta(R.misc() + 14) + kStealChunk <= (unsigned)kStealAhead &&
        (int)*reinterpret_cast<volatile unsigned*>(R.misc() + 13) + kStealLead >= n_dealt) {
      int u0 = 0;
      if (lane == 0) u0 = dealt + (int)atom_add_gpu(P.ctl + kCtlSteal, (unsigned)kStealChunk);
      u0 = __shfl_sync(0xffffffffu, u0, 0);
      const int n = max(0, min(kStealChunk, n_units - u0));
      if (lane < n) {
        const int u = u0 + lane, r = u / P.g.nseg, sg = u - r * P.g.nseg;
        const int2 bs = row_src(P, cu, r);
        SegSteal e;
        e.tok0 = sg * P.g.seg;
        e.n = min(P.g.seg, P.V - e.tok0);
        e.u = u;
        e.pad = 0;
        e.logits = reinterpret_cast<unsigned long long>(row_ptr<T>(P, bs.y) + (size_t)e.tok0 * sizeof(T));
        e.bits = reinterpret_cast<unsigned long long>(reinterpret_cast<const unsigned char*>(P.bitmap) +
                                                      (size_t)bs.x * P.g.bm_bytes + (size_t)sg * (P.g.seg / 8));
        e.desc = reinterpret_cast<unsigned long long>(P.rowdesc + r);
        R.sq()[(stail + lane) % kSegSq] = e;
      }
      __syncwarp();
      if (n > 0) {
        if (lane == 0) st_rel_cta(R.misc() + 6, stail + (unsigned)n);
        stail += (unsigned)n;
        progress = true;
      }
      if (n < kStealChunk) {
        steal_done = true;
        if (lane == 0) st_rel_cta(R.misc() + 15, 1u);   // no more claimed pass-1 units
      }
    }
    if (progress) {
      t_last = clock64();
      continue;
    }
    // done once the producer has published its unit count and all are in
    if (ld_acq_cta(R.misc() + 2) != 0u && (int)R.misc()[0] == k) break;
    if (aborted(P)) break;
    if (clock64() - t_last > P.wait_limit) {
      raise_abort(P);
      break;
    }
    __nanosleep(64);
  }
}

// A request whose decisions are all known goes to the finisher warp, which
// draws its last token and emits its tokens; with the queue full, the
// decider does it itself.
template <typename T>
__device__ __forceinline__ void queue_final(const SegParams& P, const Ring& R, unsigned& tail, int b, int lane) {
  if (tail - ld_acq_cta(R.misc() + 11) >= (unsigned)kSegFq) {
    finalize<T>(P, draw_buf(R, 1), b, lane);
    return;
  }
  __syncwarp();
  if (lane == 0) {
    R.fq()[tail % kSegFq] = b;
    st_rel_cta(R.misc() + 10, tail + 1);   // the request's decisions and its entry, then the count
  }
  ++tail;
}

// The finisher warp: the requests the decider queued, in order; done once
// the decider has finished (misc[12]) and the queue is empty.
template <typename T>
__device__ void finisher(const SegParams& P, const Ring& R, int lane) {
  unsigned head = 0;
  long long t_last = clock64();
  for (;;) {
    if (head < ld_acq_cta(R.misc() + 10)) {
      finalize<T>(P, draw_buf(R, 0), R.fq()[head % kSegFq], lane);
      ++head;
      __syncwarp();
      if (lane == 0) st_rel_cta(R.misc() + 11, head);
      t_last = clock64();
      continue;
    }
    if (ld_acq_cta(R.misc() + 12) != 0u && head == ld_acq_cta(R.misc() + 10)) break;
    if (aborted(P)) break;
    if (clock64() - t_last > P.wait_limit) {
      raise_abort(P);
      break;
    }
    __nanosleep(200);
  }
}

// The decider warp: for the rows and requests this CTA owns (the i-th is
// c + i * gridDim), combines a row once all its units are counted, decides a
// request once all its rows are combined, waits for its positions' second
// passes, finishes those and emits the tokens.
template <typename T>
__device__ void decider(const SegParams& P, const Ring& R, int lane) {
  const int G = gridDim.x, c = blockIdx.x;
  const int* cu = cu_of(P, R);
  Owned rows, reqs;
  int jp = -1, jb = -1;     // a position of an owned request waiting for its second pass (per lane)
  unsigned fq_tail = 0;     // requests handed to the finisher
  rows.n = c < P.NR ? (P.NR - 1 - c) / G + 1 : 0;
  reqs.n = c < P.B ? (P.B - 1 - c) / G + 1 : 0;
  // nothing completes when cu_draft is not a valid packing
  if (!poll_gpu(P, P.ctl + kCtlPrepDone, [G](unsigned v) { return v >= (unsigned)G; })) return;
  if (ld_acq_gpu(P.ctl + kCtlBroken) != 0u) return;
  long long t_last = clock64();
  for (;;) {
    bool progress = false;
    // 2-4. one round trip of relaxed loads: the next owned rows (lanes
    //      0..7), the next owned requests (lanes 8..15) and the positions
    //      waiting for their second pass (any lane)
    const int ri = rows.next + lane, qi = reqs.next + lane - 8;
    const bool c_row = lane < 8 && ri < rows.n && !((rows.done >> lane) & 1u);
    const bool c_req = lane >= 8 && lane < 16 && qi < reqs.n && !((reqs.done >> (lane - 8)) & 1u);
    const int qb = c + qi * G;
    unsigned v_row = 0, v_req = 0, v_job = 0;
    int Kq = 0;
    if (c_row) v_row = ld_relaxed_gpu(P.row_cnt + c + ri * G);
    if (c_req) {
      Kq = cu[qb + 1] - cu[qb];
      v_req = ld_relaxed_gpu(P.req_rows + qb);
    }
    if (jp >= 0) v_job = ld_relaxed_gpu(P.job_cnt + jp);
    unsigned rm = __ballot_sync(0xffffffffu, c_row && v_row == (unsigned)P.g.nseg);
    unsigned qm = __ballot_sync(0xffffffffu, c_req && v_req == (unsigned)(2 * Kq + 1)) >> 8;
    unsigned jm = __ballot_sync(0xffffffffu, jp >= 0 && v_job == (unsigned)P.g.upj);
    if (rm | qm | jm) {
      progress = true;
      asm volatile("fence.acq_rel.gpu;" ::: "memory");   // the counts' releases happen before what follows
    }
    // rows whose units are all in
    rows.done |= rm;
    while (rm) {
      const int L = __ffs(rm) - 1;
      rm &= rm - 1;
      row_combine<T>(P, c + (rows.next + L) * G, lane);
    }
    rows.advance();
    // requests whose rows are all combined (while the wait list has room for
    // all of a request's positions)
    {
      int room = __popc(__ballot_sync(0xffffffffu, jp < 0));
      while (qm) {
        const int L = __ffs(qm) - 1;
        qm &= qm - 1;
        const int KL = __shfl_sync(0xffffffffu, Kq, 8 + L);
        if (min(KL, 32) > room) break;    // decided later, once jobs have finished
        reqs.done |= 1u << L;
        const int bb = c + (reqs.next + L) * G;
        bool ready;
        const unsigned need = request_decide<T>(P, bb, lane, ready);
        if (ready) queue_final<T>(P, R, fq_tail, bb, lane);
        if (need) {
          // the request's positions with a job join the wait list
          const int d0 = cu[bb];
          const unsigned freem = __ballot_sync(0xffffffffu, jp < 0);
          unsigned nm = need, fm = freem;
          while (nm) {
            const int i = __ffs(nm) - 1;
            nm &= nm - 1;
            const int f = __ffs(fm) - 1;
            fm &= fm - 1;
            if (lane == f) {
              jp = d0 + i;
              jb = bb;
            }
          }
          room -= __popc(need);
        }
      }
      reqs.advance();
    }
    // positions whose second pass is complete; a request whose last one this
    // is gets its tokens
    while (jm) {
      const int L = __ffs(jm) - 1;
      jm &= jm - 1;
      const int p = __shfl_sync(0xffffffffu, jp, L);
      const int b = __shfl_sync(0xffffffffu, jb, L);
      job_finish<T>(P, p, lane);
      if (lane == L) jp = -1;
      const bool more = __ballot_sync(0xffffffffu, jp >= 0 && jb == b) != 0u;
      if (!more) {
        if (P.mode == kModeTvOnly) {
          if (lane == 0) P.req_done[b] = 1u;
        } else {
          queue_final<T>(P, R, fq_tail, b, lane);
        }
      }
    }
    if (progress) {
      t_last = clock64();
      continue;
    }
    if (rows.next >= rows.n && reqs.next >= reqs.n && !__any_sync(0xffffffffu, jp >= 0)) break;
    if (aborted(P)) break;
    if (clock64() - t_last > P.wait_limit) {
      raise_abort(P);
      break;
    }
    __nanosleep(100);
  }
}

template <typename T>
__global__ void __launch_bounds__(kSegThreads, 1) seg_verify_kernel(const __grid_constant__ SegParams P) {
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  Ring R;
  if (threadIdx.x == 0) {
    for (int s = 0; s < kSegSlots; ++s) {
      mbar_init(R.full() + s, 1);
      mbar_init(R.empty() + s, kSegGroupWarps);
    }
    for (int i = 0; i < 2; ++i) {
      const DrawBuf db = draw_buf(R, i);
      mbar_init(db.bar, 1);
      *db.phase = 0u;
    }
    fence_mbar_init();
  }
  if (threadIdx.x < 16) R.misc()[threadIdx.x] = 0u;
  for (int i = threadIdx.x; i < kSegRecN; i += blockDim.x) R.rec(i)->ndone = 0u;
  __syncthreads();
  Prod st;
  RowUnit mine{};
  int pre = 0;
  if (warp == 0) pre = producer_prefetch<T>(P, R, st, mine, lane);
  // the prologue: request b on CTA b mod gridDim (warps 1 and up; warp 0 has
  // started the first copies)
  if (blockIdx.x == 0 && threadIdx.x == 0) {
    if (__ldg(P.cu_draft) != 0 || __ldg(P.cu_draft + P.B) != P.total) atomicOr(P.ctl + kCtlBroken, 1u);
  }
  // this CTA's stripe of the per-call counters, before the grid-wide wait
  // that ends the prologue (nothing reads or writes them before it)
  {
    const size_t n16 = P.zero_bytes / 16;
    uint4* z = reinterpret_cast<uint4*>(P.zero);
    for (size_t i = (size_t)blockIdx.x * blockDim.x + threadIdx.x; i < n16; i += (size_t)gridDim.x * blockDim.x)
      z[i] = make_uint4(0u, 0u, 0u, 0u);
  }
  if (warp >= 1)
    for (int b = blockIdx.x; b < P.B; b += gridDim.x) {
      prep_request(P, b, threadIdx.x - 32, R.misc() + 7);
      prep_sync();
    }
  fence_proxy_async_global();
  __syncthreads();
  if (threadIdx.x == 0) {
    __threadfence();
    red_add_gpu(P.ctl + kCtlPrepDone, 1u);
  }
  if (warp == 0) {
    producer<T>(P, R, st, mine, pre, lane);
  } else if (warp == 1) {
    recorder<T>(P, R, lane);
  } else if (warp == 2) {
    decider<T>(P, R, lane);
    __syncwarp();
    if (lane == 0) st_rel_cta(R.misc() + 12, 1u);   // the finisher's queue is complete
  } else if (warp == 3) {
    finisher<T>(P, R, lane);
  } else {
    consumer<T>(P, R, warp - kSegCtlWarps, lane);
  }
  __syncthreads();
  if (threadIdx.x == 0) {
    __threadfence();
    const unsigned old = atom_add_gpu(P.ctl + kCtlExited, 1u);
    R.misc()[3] = (old + 1u == gridDim.x) ? 1u : 0u;
  }
  __syncthreads();
  if (R.misc()[3]) {
    // the last CTA: requests left unfinished (a wait ran out, or cu_draft
    // is not a valid packing) are reported
    __threadfence();
    const bool ab = aborted(P);
    for (int b = threadIdx.x; b < P.B; b += blockDim.x) {
      if (__ldcg(P.req_done + b)) continue;
      const int d0 = __ldg(P.cu_draft + b), d1 = __ldg(P.cu_draft + b + 1);
      const bool rows_ok = d0 >= 0 && d1 >= d0 && d1 <= P.total;
      if (P.mode == kModeTvOnly) {
        if (rows_ok)
          for (int p = d0; p < d1; ++p) {
            P.out_tv[p] = NAN;
            P.out_theta[p] = NAN;
          }
        continue;
      }
      if (rows_ok)
        for (int s = 0; s <= d1 - d0; ++s) P.out_tokens[d0 + b + s] = -1;
      P.out_accepted[b] = -1;
      if (P.out_status) P.out_status[b] = ab ? kStatusTimeout : kStatusBadK;
    }
    // every other CTA has left: the control words go back to zero for the
    // next call
    __syncthreads();
    if (threadIdx.x < kCtlWords) P.ctl[threadIdx.x] = 0u;
  }
}

}  // namespace

// Control words of the kernel (kCtlWords per device), zero between calls.
// One call at a time uses them: a launch takes every SM for its cooperative
// grid, so a second one starts only after the first has left.
__device__ unsigned g_seg_ctl[kCtlWords];

int seg_smem_bytes() { return kSegSmem; }

unsigned* seg_ctl_address() {
  void* p = nullptr;
  if (cudaGetSymbolAddress(&p, g_seg_ctl) != cudaSuccess) {
    cudaGetLastError();
    return nullptr;
  }
  return static_cast<unsigned*>(p);
}

int launch_seg_verify(const SegParams& P, bool bf16, int num_sms, cudaStream_t stream) {
  auto kern = bf16 ? seg_verify_kernel<__nv_bfloat16> : seg_verify_kernel<float>;
  if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, kSegSmem) != cudaSuccess) {
    cudaGetLastError();
    return -1;
  }
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)num_sms);
  cfg.blockDim = dim3(kSegThreads);
  cfg.dynamicSmemBytes = kSegSmem;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeCooperative;
  attr[0].val.cooperative = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  if (cudaLaunchKernelEx(&cfg, kern, P) != cudaSuccess) {
    cudaGetLastError();
    return -1;
  }
  return 0;
}

}  // namespace sv
