// Pipelined streaming kernel of mentored speculative sampling without top-p
// ("What I Gave Up to Make Speculative Decoding Faster", section "A knob for
// accepting more draft tokens"), for batches with more work items than SMs.
//
// A work item is one draft position (target row + draft row) or one bonus
// row, as in the cluster kernel.  One CTA per SM loops over its items
// (item k of CTA c is c + k * gridDim.x); its warps have six roles:
//   group A streaming warps (kPipeWarpsA): pass 1 of item k from a TMA ring
//       fed from HBM (L2 policy evict_last): per lane a running reference and
//       the sum of 2^(z'c - ref), z' the penalised logit, c = log2(e)/T;
//   group A setup warp: the penalty bitmap of item k+1 (history plus the
//       drafts before the row), then item k's combine: (M, 1/S) per row,
//       p(x) and q(x);
//   group B streaming warps (kPipeWarpsB): pass 2 of item k-1 from a second
//       ring that re-reads the rows (L2 hits, evict_first): the mass of
//       max(p-q, 0) (or of p for a bonus row) per segment;
//   group B tail warp: for item k-2 the prefix over segments (TV d = total
//       residual mass), theta, pi(x), the acceptance decision, the
//       inverse-CDF candidate and the request's finalisation;
//   two producer warps (lane 0 issues the bulk copies of one ring each).
// Only ring A reads HBM, so HBM keeps streaming while the per-item serial
// steps run on the setup and tail warps.  Per-item state (bitmap, hand-off
// block, segment masses) is triple-buffered; mbarriers order the roles.
//
// Repetition penalty: before a streaming warp reads its segment of a ring
// slot, the lanes holding bitmap words with set bits take the penalised
// positions out of the stream (-inf) after adding their exact terms: group A
// their softmax terms, group B their residuals.  The hot loops never test
// the penalty.
//
// A rejected position whose residual mass is exactly zero (its correction
// is then drawn from p) leaves the pipeline; all compute warps recompute such
// items at the end with direct global loads ("deferred").

#include "common.cuh"
#include "spec_internal.h"
#include "stream_common.cuh"
#include "verify_common.cuh"

namespace sv {

namespace {

constexpr int kNA = kPipeWarpsA;
constexpr int kNB = kPipeWarpsB;
constexpr int kNC = kNA + kNB + 2;             // compute warps (streaming + setup + tail)
constexpr int kThreadsA = kNA * 32;
constexpr int kThreadsB = kNB * 32;
constexpr int kThreadsC = kNC * 32;
constexpr int kPipeThreads = kThreadsC + 64;   // + producer warps A and B
constexpr int kBarA = 1, kBarB = 2, kBarC = 3;  // named barriers of the groups

extern __shared__ __align__(128) unsigned char pipe_smem[];

// Shared-memory regions, addressed from the layout in parameter space (no
// table of pointers that would have to live in local memory).
struct PSmem {
  const PipeLayout& L;
  __device__ __forceinline__ explicit PSmem(const PipeLayout& l) : L(l) {}
  __device__ __forceinline__ unsigned char* at(int off) const { return pipe_smem + off; }
  __device__ __forceinline__ unsigned char* ring_a() const { return at(L.off_ring_a); }
  __device__ __forceinline__ unsigned char* ring_b() const { return at(L.off_ring_b); }
  // item buffer kb's penalty bitmap (the slow path uses buffer 0)
  __device__ __forceinline__ uint32_t* bm(int kb) const {
    return reinterpret_cast<uint32_t*>(at(L.off_bm + kb * align_up_i(L.bm_words * 4, 16)));
  }
  // slow path: 256-token chunk sums
  __device__ __forceinline__ float* part() const { return reinterpret_cast<float*>(at(L.off_part)); }
  // item buffer kb: [nseg] segment residual mass
  __device__ __forceinline__ float* segt(int kb) const {
    return reinterpret_cast<float*>(at(L.off_segt + kb * align_up_i(L.nseg * 4, 16)));
  }
  // cu_draft copy (when B + 1 <= kPipeCuCap)
  __device__ __forceinline__ int* cu() const { return reinterpret_cast<int*>(at(L.off_cu)); }
  __device__ __forceinline__ PipeStats* stats(int kb) const {
    return reinterpret_cast<PipeStats*>(at(L.off_stats + kb * align_up_i((int)sizeof(PipeStats), 16)));
  }
  // misc: [compute warps][2] slow-path warp partials (up to 64), then scalars
  __device__ __forceinline__ float2* cwp() const { return reinterpret_cast<float2*>(at(L.off_misc)); }
  // mi: [0] group B status bits, [1] B deferral, [2] B finalize flag,
  //     [3] slow finalize flag, [4] slow: draw from p
  __device__ __forceinline__ int* mi() const { return reinterpret_cast<int*>(at(L.off_misc + 576)); }
  __device__ __forceinline__ uint32_t* defer() const { return reinterpret_cast<uint32_t*>(at(L.off_defer)); }
  __device__ __forceinline__ uint64_t* bars() const { return reinterpret_cast<uint64_t*>(at(L.off_bar)); }
  __device__ __forceinline__ uint64_t* full_a() const { return bars(); }
  __device__ __forceinline__ uint64_t* empty_a() const { return bars() + L.slots_a; }
  __device__ __forceinline__ uint64_t* full_b() const { return bars() + 2 * L.slots_a; }
  __device__ __forceinline__ uint64_t* empty_b() const { return bars() + 2 * L.slots_a + L.slots_b; }
  // [kPipeBufs] each: setup warp -> A streaming warps: the item's penalty
  // list is built; A streaming warps -> setup warp: pass 1 done; setup warp
  // -> B streaming warps and producer B: statistics combined; B streaming
  // warps -> tail warp: pass 2 done; tail warp and producer B -> setup warp:
  // the item's buffers are free again
  __device__ __forceinline__ uint64_t* list_ready() const { return bars() + 2 * L.slots_a + 2 * L.slots_b; }
  __device__ __forceinline__ uint64_t* pass1_done() const { return list_ready() + kPipeBufs; }
  __device__ __forceinline__ uint64_t* stats_full() const { return list_ready() + 2 * kPipeBufs; }
  __device__ __forceinline__ uint64_t* pass2_done() const { return list_ready() + 3 * kPipeBufs; }
  __device__ __forceinline__ uint64_t* buf_free() const { return list_ready() + 4 * kPipeBufs; }
  // A streaming warps -> tail warp: their share of the last item's pass 2 is done
  __device__ __forceinline__ uint64_t* pass2a_done() const { return list_ready() + 5 * kPipeBufs; }
};


// Records one item's status; the last item of its request to finish writes
// the request's tokens (first rejected position's candidate, or the bonus).
// `tg` is the thread's index in the calling group of `nthr` threads (named
// barrier `bar`); the group's warp 0 writes.
__device__ __forceinline__ void finish_item(const SampleParams& P, const Item& it, int item, int flags, int tg, int bar,
                                            int nthr, int* shflag) {
  const int b = it.b, K = it.K;
  if (tg == 0) {
    P.inval[(size_t)item * kMaxCluster] = flags;
    __threadfence();
    const int old = tagged_arrive(P.counters + b, P.tag);
    *shflag = (old == K) && K >= 0 && it.rows_ok;
  }
  if (bar >= 0) named_sync(bar, nthr);
  else __syncwarp();
  if (*shflag && tg < 32) {
    const int lane = tg;
    __threadfence();
    const int d0 = __ldg(P.cu_draft + b), off = d0 + b;
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
    int last;
    if (jrej < K) last = __ldcg(&P.results[d0 + jrej].cand);
    else last = nobonus ? -1 : __ldcg(&P.results[P.total + b].cand);
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
}

// Items of this CTA (item k is blockIdx.x + k * gridDim.x).
__device__ __forceinline__ int n_local_items(const SampleParams& P) {
  return (int)blockIdx.x < P.n_items ? (P.n_items - (int)blockIdx.x + (int)gridDim.x - 1) / (int)gridDim.x : 0;
}

// The last item's pass 2 is shared: ring B / group B take the even
// positions of its (reversed) stage order, ring A / group A the odd ones,
// once group A has no pass 1 left.
__device__ __forceinline__ bool b_skips(int k, int n_local, int stn) { return k == n_local - 1 && (stn & 1); }

// cu_draft as the kernel reads it: the shared-memory copy when it fits.
__device__ __forceinline__ const int* cu_ptr(const SampleParams& P, const PSmem& S) {
  return P.B + 1 <= kPipeCuCap ? S.cu() : P.cu_draft;
}

// The work item's request, position and rows (the same decoding as
// decode_item, reading cu_draft through `cu`).
__device__ __forceinline__ Item pdecode(const SampleParams& P, const int* cu, int item) {
  Item it;
  if (item < P.total) {
    int lo = 0, hi = P.B;
    while (hi - lo > 1) {
      const int mid = (lo + hi) >> 1;
      if (cu[mid] <= item) lo = mid;
      else hi = mid;
    }
    it.b = lo;
    it.i = item - cu[lo];
    it.bonus = false;
    it.tgt_row = item + lo;
    it.dft_row = item;
    it.rows_ok = true;
  } else {
    const int b = item - P.total;
    const int c0 = cu[b], c1 = cu[b + 1];
    it.b = b;
    it.i = c1 - c0;
    it.bonus = true;
    it.rows_ok = (c0 >= 0 && c0 <= c1 && c1 <= P.total);
    it.tgt_row = it.rows_ok ? c1 + b : b;
    it.dft_row = -1;
  }
  it.K = cu[it.b + 1] - cu[it.b];
  return it;
}

// Per-request scalars and the status bits that follow from them.
struct Scalars {
  int b, K, d0, off, nrows, x, flags;
  float alpha, c, D;
  bool params_ok, pen, uniforms_ok;
  int h0, h1, npre;
};

__device__ __forceinline__ Scalars item_scalars(const SampleParams& P, const Item& it, int item, const int* cu) {
  Scalars s;
  s.b = it.b;
  s.K = it.K;
  s.d0 = cu[it.b];
  s.off = s.d0 + it.b;
  s.nrows = it.bonus ? 1 : 2;
  s.flags = 0;
  if (!it.rows_ok || s.K < 0 || s.K > P.max_k || s.K > kMaxK) s.flags |= kStatusBadK;
  const float T_ = P.temperature ? __ldg(P.temperature + s.b) : 1.f;
  s.alpha = P.rep_penalty ? __ldg(P.rep_penalty + s.b) : 1.f;
  s.D = P.tv_budget ? __ldg(P.tv_budget + s.b) : 0.f;
  s.params_ok = item_params_ok(P, s.b);
  if (!s.params_ok) s.flags |= kStatusBadParam;
  // invalid scalars are reported; the statistics then use T = 1, no penalty
  s.c = __fdiv_rn(1.44269504088896341f, s.params_ok ? T_ : 1.f);
  s.x = it.bonus ? -1 : __ldg(P.draft_tokens + item);
  if (!it.bonus && (s.x < 0 || s.x >= P.V)) s.flags |= kStatusBadToken;
  s.h0 = P.cu_hist ? __ldg(P.cu_hist + s.b) : 0;
  s.h1 = P.cu_hist ? __ldg(P.cu_hist + s.b + 1) : 0;
  s.npre = it.bonus ? (it.rows_ok ? s.K : 0) : it.i;
  s.pen = s.params_ok && s.alpha != 1.f && (s.h1 > s.h0 || s.npre > 0);
  s.uniforms_ok = !(s.flags & kStatusBadK);
  return s;
}

// Marks the penalty set of a request row in `bm` (if pen) and reports
// out-of-range tokens; threads t of nt.
__device__ __forceinline__ int mark_penalty_set(const SampleParams& P, const Scalars& s, uint32_t* bm, int t, int nt) {
  int flags = 0;
  // eight loads in flight per thread before their bits are set
  for (int j0 = s.h0 + t; j0 < s.h1; j0 += 8 * nt) {
    int tok[8];
#pragma unroll
    for (int q = 0; q < 8; ++q) tok[q] = j0 + q * nt < s.h1 ? __ldg(P.hist + j0 + q * nt) : 0;
#pragma unroll
    for (int q = 0; q < 8; ++q) {
      if (j0 + q * nt >= s.h1) continue;
      if (tok[q] < 0 || tok[q] >= P.V) flags |= kStatusBadToken;
      else if (s.pen) atomicOr(&bm[tok[q] >> 5], 1u << (tok[q] & 31));
    }
  }
  for (int j = t; j < s.npre; j += nt) {
    const int tok = __ldg(P.draft_tokens + s.d0 + j);
    if (tok < 0 || tok >= P.V) flags |= kStatusBadToken;
    else if (s.pen) atomicOr(&bm[tok >> 5], 1u << (tok & 31));
  }
  return flags;
}

// ------------------------------------------------------------ producers
template <typename T, bool IS_A>
__device__ __forceinline__ void producer(const SampleParams& P, const PipeLayout& L, const PSmem& S) {
  const uint64_t pol = IS_A ? l2_policy_evict_last() : l2_policy_evict_first();
  constexpr int es = (int)sizeof(T);
  const int stage = (IS_A ? kNA : kNB) * L.seg;
  const int nst = IS_A ? L.nst_a : L.nst_b;
  const int nslots = IS_A ? L.slots_a : L.slots_b;
  const int slot_bytes = IS_A ? L.slot_a : L.slot_b;
  unsigned char* ring = IS_A ? S.ring_a() : S.ring_b();
  uint64_t* full = IS_A ? S.full_a() : S.full_b();
  uint64_t* empty = IS_A ? S.empty_a() : S.empty_b();
  RingCursor rc;
  RingFills fills;
  bool to = false;   // a wait ran out: nothing more is issued (the consumers' own waits then run out)
  int k = 0;
  const int* cu = cu_ptr(P, S);
  const int n_local = n_local_items(P);
  for (int item = blockIdx.x; item < P.n_items && !to; item += gridDim.x, ++k) {
    const Item it = pdecode(P, cu, item);
    if (!IS_A) {
      // pass 2 of item k starts once its statistics are combined (the rows
      // are then in L2)
      const int kb = k % kPipeBufs;
      if (!mbar_wait(&S.stats_full()[kb], (uint32_t)(k / kPipeBufs) & 1u)) {
        to = true;
        break;
      }
      mbar_arrive(&S.buf_free()[kb]);  // this warp has seen item k's statistics
    }
    const unsigned char* rowp = static_cast<const unsigned char*>(P.target) + (size_t)it.tgt_row * P.ld_t * es;
    const unsigned char* rowq =
        it.bonus ? rowp : static_cast<const unsigned char*>(P.draft) + (size_t)it.dft_row * P.ld_d * es;
    for (int st = 0; st < nst; ++st) {
      if (!IS_A && b_skips(k, n_local, st)) continue;
      const uint32_t slot = rc.slot, phase = rc.phase;
      // first use of a slot: the phase "before" its first completes at once
      if (!mbar_wait(&empty[slot], rc.phase ^ 1u)) {
        to = true;
        break;
      }
      rc.advance(nslots);
      fills.note(slot, phase);
      // ring B takes the stages in reverse: the lines ring A read last are
      // re-read first, while they are the least likely to have left L2
      const int sx = IS_A ? st : nst - 1 - st;
      const int n = min(stage, P.V - sx * stage);
      const uint32_t bytes = (uint32_t)((n * es + 15) & ~15);
      unsigned char* dst = ring + (size_t)slot * slot_bytes;
      mbar_arrive_expect_tx(&full[slot], it.bonus ? bytes : 2 * bytes);
      bulk_g2s(dst, rowp + (size_t)sx * stage * es, bytes, &full[slot], pol);
      if (!it.bonus) bulk_g2s(dst + (size_t)stage * es, rowq + (size_t)sx * stage * es, bytes, &full[slot], pol);
    }
  }
  if (IS_A && n_local > 0 && !to) {
    // ring A then carries the last item's odd pass-2 stages (a re-read, in
    // ring B's reversed order), once its statistics are combined
    const int kl = n_local - 1;
    if (!mbar_wait(&S.stats_full()[kl % kPipeBufs], (uint32_t)(kl / kPipeBufs) & 1u)) to = true;
    const Item it = pdecode(P, cu, blockIdx.x + kl * gridDim.x);
    const unsigned char* rowp = static_cast<const unsigned char*>(P.target) + (size_t)it.tgt_row * P.ld_t * es;
    const unsigned char* rowq =
        it.bonus ? rowp : static_cast<const unsigned char*>(P.draft) + (size_t)it.dft_row * P.ld_d * es;
    const uint64_t pol2 = l2_policy_evict_first();
    for (int st = 1; st < L.nst_b && !to; st += 2) {
      const uint32_t slot = rc.slot, phase = rc.phase;
      if (!mbar_wait(&empty[slot], rc.phase ^ 1u)) {
        to = true;
        break;
      }
      rc.advance(nslots);
      fills.note(slot, phase);
      const int sx = L.nst_b - 1 - st;
      const int n = min(stage, P.V - sx * stage);
      const uint32_t bytes = (uint32_t)((n * es + 15) & ~15);
      unsigned char* dst = ring + (size_t)slot * slot_bytes;
      mbar_arrive_expect_tx(&full[slot], it.bonus ? bytes : 2 * bytes);
      bulk_g2s(dst, rowp + (size_t)sx * stage * es, bytes, &full[slot], pol2);
      if (!it.bonus) bulk_g2s(dst + (size_t)stage * es, rowq + (size_t)sx * stage * es, bytes, &full[slot], pol2);
    }
  }
  // after a wait ran out: the copies already started land before the CTA
  // may exit (the consumers' own waits run out and mark their items)
  if (to) fills.drain(full, nslots);
}

// Pass 2 of segment s_id of item buffer kb from a staged ring segment (both
// rows, kNB * kPipeSegBytes apart): the penalised tokens' exact residuals
// (or p), their copies -inf, then the segment's mass of max(p-q, 0) (or of
// p for a bonus row) to segt.
template <typename T>
__device__ __forceinline__ void pass2_seg(const SampleParams& P, const PipeLayout& L, const PSmem& S, int kb,
                                          const Item& it, const Scalars& sc, unsigned char* seg, int s_id, int lane) {
  const int SEG = L.seg;
  const int wps = SEG / 32;
  const int row_bytes = kNB * kPipeSegBytes;
  const PipeStats& st = *S.stats(kb);
  const float Mp = st.M[0], Mq = st.M[1], ip = st.inv[0], iq = st.inv[1];
  float extra = 0.f;
  if (st.pen) {
    // penalised positions: their exact residual (or p), then out of the
    // stream (-inf)
    const bool two = sc.nrows == 2;
    bool wrote = false;
    const bool any = for_penalised(S.bm(kb), s_id, wps, lane, [&](int o) {
      T* pp = reinterpret_cast<T*>(seg) + o;
      T* qq = reinterpret_cast<T*>(seg + row_bytes) + o;
      const float p = prob_of(penalize(to_f32<T>(*pp), sc.alpha), sc.c, Mp, ip);
      extra += it.bonus ? p : resid_of(p, prob_of(penalize(to_f32<T>(*qq), sc.alpha), sc.c, Mq, iq));
      *pp = neg_inf<T>();
      if (two) *qq = neg_inf<T>();
      wrote = true;
    });
    if (any) {
      if (wrote) fence_proxy_async_smem();
      __syncwarp();
    }
  }
  const int nvalid = min(SEG, P.V - s_id * SEG);
  const float v = it.bonus ? seg_resid<T, true>(seg, row_bytes, lane, nvalid, sc.c, Mp, Mq, ip, iq)
                           : seg_resid<T, false>(seg, row_bytes, lane, nvalid, sc.c, Mp, Mq, ip, iq);
  const float tot = warp_sum(v + extra);
  if (lane == 0) S.segt(kb)[s_id] = tot;
}

static_assert(kPipeWarpsA == kPipeWarpsB, "the rings share a stage size");

// ------------------------------------------------------------- group A
// Streaming warps: pass 1 of each item over ring A.  Before reading a
// segment the lanes copy the penalised positions' raw logits into the list
// and overwrite them with -inf; each lane keeps a running reference and the
// sum of 2^(z'c - ref); the warp's (reference, sum) per row goes to the setup
// warp.
template <typename T>
__device__ __forceinline__ void a_stream(const SampleParams& P, const PipeLayout& L, const PSmem& S, int wa, int lane) {
  const int SEG = L.seg;
  const int row_bytes = kNA * kPipeSegBytes;
  const int* cu = cu_ptr(P, S);
  RingCursor rc;
  bool timeout = false;
  int k = 0;
  for (int item = blockIdx.x; item < P.n_items; item += gridDim.x, ++k) {
    const int kb = k % kPipeBufs;
    PipeStats& st = *S.stats(kb);
    const Item it = pdecode(P, cu, item);
    const Scalars sc = item_scalars(P, it, item, cu);
    if (!timeout && !mbar_wait(&S.list_ready()[kb], (uint32_t)(k / kPipeBufs) & 1u)) timeout = true;
    const bool pen = st.pen != 0;
    const int wps = SEG / 32;
    float ref[2] = {-INFINITY, -INFINITY}, run[2] = {0.f, 0.f};
    float pref[2] = {-INFINITY, -INFINITY}, psum[2] = {0.f, 0.f};
    int pflags = 0;
    for (int stn = 0; stn < L.nst_a; ++stn) {
      const uint32_t slot = rc.slot;
      if (!timeout && !mbar_wait(&S.full_a()[slot], rc.phase)) timeout = true;
      rc.advance(L.slots_a);
      const int s_id = stn * kNA + wa;
      if (s_id < L.nseg) {
        unsigned char* seg = S.ring_a() + (size_t)slot * L.slot_a + wa * kPipeSegBytes;
        const int base = s_id * SEG;
        if (sc.x >= base && sc.x < base + SEG) {
          // the draft token's raw logits, before any patch
          if (lane == 0) {
            st.xz[0] = to_f32<T>(reinterpret_cast<const T*>(seg)[sc.x - base]);
            st.xz[1] = to_f32<T>(reinterpret_cast<const T*>(seg + row_bytes)[sc.x - base]);
          }
          __syncwarp();
        }
        if (pen) {
          // penalised positions: add their exact terms, then take them out
          // of the stream (-inf)
          const bool two = sc.nrows == 2;
          bool wrote = false;
          const bool any = for_penalised(S.bm(kb), s_id, wps, lane, [&](int o) {
            T* pp = reinterpret_cast<T*>(seg) + o;
            T* qq = reinterpret_cast<T*>(seg + row_bytes) + o;
            const float zp = to_f32<T>(*pp), zq = two ? to_f32<T>(*qq) : 0.f;
            if (is_bad_logit(zp) || (two && is_bad_logit(zq))) pflags |= kStatusBadLogits;
            online_add(penalize(zp, sc.alpha) * sc.c, pref[0], psum[0]);
            if (two) online_add(penalize(zq, sc.alpha) * sc.c, pref[1], psum[1]);
            *pp = neg_inf<T>();
            if (two) *qq = neg_inf<T>();
            wrote = true;
          });
          if (any) {
            if (wrote) fence_proxy_async_smem();
            __syncwarp();
          }
        }
        const int nvalid = min(SEG, P.V - base);
        if (sc.nrows == 2) seg_stats<T, 2>(seg, row_bytes, lane, nvalid, sc.c, ref, run);
        else seg_stats<T, 1>(seg, row_bytes, lane, nvalid, sc.c, ref, run);
      }
      __syncwarp();
      if (lane == 0) mbar_arrive(&S.empty_a()[slot]);
    }
#pragma unroll
    for (int r = 0; r < 2; ++r) {
      // the lane's stream terms and its penalised tokens' terms, then the warp's
      float M = ref[r], Sl = run[r];
      combine_into(make_float2(pref[r], psum[r]), M, Sl);
      const float2 wv = warp_combine(M, Sl);
      if (lane == 0) st.wp[wa][r] = wv;
    }
    pflags = warp_or(pflags);
    if (lane == 0) st.aflags[wa] = pflags | (timeout ? kStatusTimeout : 0);
    __syncwarp();
    if (lane == 0) mbar_arrive(&S.pass1_done()[kb]);
  }
  const int n_local = n_local_items(P);
  if (n_local > 0) {
    // the odd positions of the last item's pass 2, from ring A
    const int kl = n_local - 1;
    const int kb = kl % kPipeBufs;
    const int item = blockIdx.x + kl * gridDim.x;
    const Item it = pdecode(P, cu, item);
    const Scalars sc = item_scalars(P, it, item, cu);
    if (!timeout && !mbar_wait(&S.stats_full()[kb], (uint32_t)(kl / kPipeBufs) & 1u)) timeout = true;
    for (int st = 1; st < L.nst_b; st += 2) {
      const uint32_t slot = rc.slot;
      if (!timeout && !mbar_wait(&S.full_a()[slot], rc.phase)) timeout = true;
      rc.advance(L.slots_a);
      const int s_id = (L.nst_b - 1 - st) * kNA + wa;
      if (s_id < L.nseg)
        pass2_seg<T>(P, L, S, kb, it, sc, S.ring_a() + (size_t)slot * L.slot_a + wa * kPipeSegBytes, s_id, lane);
      __syncwarp();
      if (lane == 0) mbar_arrive(&S.empty_a()[slot]);
    }
    if (lane == 0 && timeout) atomicOr(&S.stats(kb)->flags, kStatusTimeout);
    __syncwarp();
    if (lane == 0) mbar_arrive(&S.pass2a_done()[0]);
  }
}

// Group A's setup warp, per item k: the penalty list of item k+1 (bitmap,
// then compaction into a list sorted by segment), then item k's softmax
// combine with the penalised tokens' exact terms, p(x), q(x) and the
// penalised tokens' residual mass per segment.
template <typename T>
__device__ __forceinline__ void a_setup(const SampleParams& P, const PipeLayout& L, const PSmem& S, int lane) {
  const int SEG = L.seg;
  const int wshift = __ffs(SEG / 32) - 1;  // log2(bitmap words per segment)
  const int* cu = cu_ptr(P, S);
  bool timeout = false;
  const int n_local = (int)blockIdx.x < P.n_items ? (P.n_items - (int)blockIdx.x + (int)gridDim.x - 1) / (int)gridDim.x : 0;

  auto build = [&](int k) {
    const int item = blockIdx.x + k * gridDim.x;
    const int kb = k % kPipeBufs;
    const Item it = pdecode(P, cu, item);
    const Scalars sc = item_scalars(P, it, item, cu);
    // buffer kb is free once item k-3's tail and producer B are done with it
    if (!timeout && !mbar_wait(&S.buf_free()[kb], ((uint32_t)(k / kPipeBufs) & 1u) ^ 1u)) timeout = true;
    PipeStats& st = *S.stats(kb);
    uint32_t* bm = S.bm(kb);
    if (sc.pen)
      for (int q = lane; q < L.bm_words / 4; q += 32) reinterpret_cast<uint4*>(bm)[q] = make_uint4(0u, 0u, 0u, 0u);
    __syncwarp();
    int flags = sc.flags | mark_penalty_set(P, sc, bm, lane, 32) | (timeout ? kStatusTimeout : 0);
    flags = warp_or(flags);
    if (lane == 0) {
      st.flags = flags;
      st.pen = sc.pen ? 1 : 0;
    }
    __syncwarp();
    if (lane == 0) mbar_arrive(&S.list_ready()[kb]);
  };

  auto combine = [&](int k) {
    const int item = blockIdx.x + k * gridDim.x;
    const int kb = k % kPipeBufs;
    const Item it = pdecode(P, cu, item);
    const Scalars sc = item_scalars(P, it, item, cu);
    PipeStats& st = *S.stats(kb);
    if (!timeout && !mbar_wait(&S.pass1_done()[kb], (uint32_t)(k / kPipeBufs) & 1u)) timeout = true;
    int flags = st.flags | (timeout ? kStatusTimeout : 0);
    for (int w = 0; w < kNA; ++w) flags |= st.aflags[w];
    float M[2] = {0.f, 0.f}, inv[2] = {1.f, 1.f};
    float px = 0.f, qx = 0.f;
    {
      float Ssum[2];
#pragma unroll
      for (int r = 0; r < 2; ++r) {
        M[r] = -INFINITY;
        Ssum[r] = 0.f;
        for (int w = 0; w < kNA; ++w) combine_into(st.wp[w][r], M[r], Ssum[r]);
      }
#pragma unroll
      for (int r = 0; r < 2; ++r)
        if (r < sc.nrows && (!(Ssum[r] > 0.f) || !(Ssum[r] < INFINITY) || !(M[r] < INFINITY)))
          flags |= kStatusBadLogits;
      const bool ok_stats = !(flags & kStatusBadLogits);
#pragma unroll
      for (int r = 0; r < 2; ++r) {
        const bool use = ok_stats && r < sc.nrows;
        inv[r] = use ? __fdiv_rn(1.f, Ssum[r]) : 1.f;
        if (!use) M[r] = 0.f;
      }
      if (lane == 0 && !it.bonus && sc.x >= 0 && sc.x < P.V && ok_stats) {
        // p(x), q(x) (x may be penalised itself)
        const bool xpen = st.pen && ((S.bm(kb)[sc.x >> 5] >> (sc.x & 31)) & 1u);
        const float zp = xpen ? penalize(st.xz[0], sc.alpha) : st.xz[0];
        const float zq = xpen ? penalize(st.xz[1], sc.alpha) : st.xz[1];
        px = prob_of(zp, sc.c, M[0], inv[0]);
        qx = prob_of(zq, sc.c, M[1], inv[1]);
      }
    }
    if (lane == 0) {
      st.M[0] = M[0];
      st.M[1] = M[1];
      st.inv[0] = inv[0];
      st.inv[1] = inv[1];
      st.px = px;
      st.qx = qx;
      st.flags = flags;
    }
    __syncwarp();
    if (lane == 0) mbar_arrive(&S.stats_full()[kb]);
  };

  if (n_local > 0) build(0);
  for (int k = 0; k < n_local; ++k) {
    if (k + 1 < n_local) build(k + 1);
    combine(k);
  }
}

// Inverse CDF within segment s (warp-wide): the first token whose inclusive
// prefix of w exceeds rem, w = max(p-q, 0) or p (ponly); `take_last` or no
// such token: the segment's last token with w > 0.  Returns -1 if none.
template <typename T>
__device__ __forceinline__ int search_segment(const SampleParams& P, const PipeLayout& L, const uint32_t* bm,
                                              const T* gp, const T* gq, bool ponly, int s, double rem, bool take_last,
                                              float c, float alpha, float Mp, float Mq, float ip, float iq, int lane) {
  constexpr int N = Vec<T>::N;
  constexpr int LT = 4 * N;  // tokens per lane, contiguous
  const int sbase = s * L.seg;
  const int base = sbase + lane * LT;
  // this lane's penalised tokens (bitmap bits base .. base + LT - 1)
  uint32_t pm = 0;
  if (bm) {
    const uint32_t w = bm[base >> 5];
    pm = LT == 32 ? w : (w >> (base & 31)) & ((1u << LT) - 1u);
  }
  uint4 vp[4], vq[4];
#pragma unroll
  for (int j = 0; j < 4; ++j) {
    const bool in = base + j * N < P.V;
    vp[j] = in ? __ldg(reinterpret_cast<const uint4*>(gp + base + j * N)) : make_uint4(0u, 0u, 0u, 0u);
    vq[j] = (in && !ponly) ? __ldg(reinterpret_cast<const uint4*>(gq + base + j * N)) : make_uint4(0u, 0u, 0u, 0u);
  }
  float w[LT];
  float ls = 0.f;
#pragma unroll
  for (int j = 0; j < 4; ++j) {
    float zp[N], zq[N];
    cvt16(vp[j], zp);
    cvt16(vq[j], zq);
#pragma unroll
    for (int e = 0; e < N; ++e) {
      const int i = j * N + e;
      float a = zp[e], bq = zq[e];
      if ((pm >> i) & 1u) {
        a = penalize(a, alpha);
        bq = penalize(bq, alpha);
      }
      float v = 0.f;
      if (base + i < P.V) {
        const float p = prob_of(a, c, Mp, ip);
        v = ponly ? p : resid_of(p, prob_of(bq, c, Mq, iq));
      }
      w[i] = v;
      ls += v;
    }
  }
  const float incl = warp_incl_scan(ls, lane);
  const float excl = incl - ls;
  int found = -1;
  if (!take_last) {
    const unsigned m = __ballot_sync(0xffffffffu, ((double)incl > rem) && ((double)excl <= rem) && ls > 0.f);
    if (m) {
      const int L0 = __ffs(m) - 1;
      int jj = -1;
      if (lane == L0) {
        double cum = (double)excl;
        int lastpos = -1;
#pragma unroll
        for (int i = 0; i < LT; ++i) {
          if (jj < 0) {
            cum += (double)w[i];
            if (w[i] > 0.f) {
              lastpos = i;
              if (cum > rem) jj = i;
            }
          }
        }
        if (jj < 0) jj = lastpos;
      }
      jj = __shfl_sync(0xffffffffu, jj, L0);
      if (jj >= 0) found = sbase + L0 * LT + jj;
    }
  }
  if (found < 0) {
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
      found = sbase + L1 * LT + jj;
    }
  }
  return found;
}

// Warp-wide owner search over per-unit masses seg[0..n) (fp64 blocks of
// consecutive units per lane, then a lane scan): the first unit with mass
// whose inclusive prefix exceeds t, and t minus the prefix before it; if
// rounding leaves t out of reach, the last unit with mass (take_last).
// Returns the total mass.
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

// ------------------------------------------------------------- group B

// Streaming warps: pass 2 of each item over ring B with the setup warp's
// normalisers; per lane and segment the sum of max(p-q, 0) (or p for a bonus
// row); then the segment masses for the tail warp.
template <typename T>
__device__ __forceinline__ void b_stream(const SampleParams& P, const PipeLayout& L, const PSmem& S, int wb, int lane) {
  const int* cu = cu_ptr(P, S);
  const int n_local = n_local_items(P);
  RingCursor rc;
  bool timeout = false;
  int k = 0;
  for (int item = blockIdx.x; item < P.n_items; item += gridDim.x, ++k) {
    const int kb = k % kPipeBufs;
    PipeStats& st = *S.stats(kb);
    const Item it = pdecode(P, cu, item);
    const Scalars sc = item_scalars(P, it, item, cu);
    if (!timeout && !mbar_wait(&S.stats_full()[kb], (uint32_t)(k / kPipeBufs) & 1u)) timeout = true;
    {
      for (int stn = 0; stn < L.nst_b; ++stn) {
        if (b_skips(k, n_local, stn)) continue;
        const uint32_t slot = rc.slot;
        if (!timeout && !mbar_wait(&S.full_b()[slot], rc.phase)) timeout = true;
        rc.advance(L.slots_b);
        const int s_id = (L.nst_b - 1 - stn) * kNB + wb;  // stages in reverse (producer B)
        if (s_id < L.nseg)
          pass2_seg<T>(P, L, S, kb, it, sc, S.ring_b() + (size_t)slot * L.slot_b + wb * kPipeSegBytes, s_id, lane);
        __syncwarp();
        if (lane == 0) mbar_arrive(&S.empty_b()[slot]);
      }
      if (lane == 0 && timeout) atomicOr(&st.flags, kStatusTimeout);
    }
    __syncwarp();
    if (lane == 0) mbar_arrive(&S.pass2_done()[kb]);
  }
}

// Group B's tail warp, per item: the prefix over segments (TV d = total
// residual mass), theta, pi(x), the acceptance decision, the inverse-CDF
// candidate and the request's finalisation; then the item's buffers go back
// to the setup warp.
template <typename T>
__device__ __forceinline__ void b_tail(const SampleParams& P, const PipeLayout& L, const PSmem& S, int lane) {
  const int* cu = cu_ptr(P, S);
  bool timeout = false;
  int k = 0;
  for (int item = blockIdx.x; item < P.n_items; item += gridDim.x, ++k) {
    const int kb = k % kPipeBufs;
    const PipeStats& st = *S.stats(kb);
    const Item it = pdecode(P, cu, item);
    const Scalars sc = item_scalars(P, it, item, cu);
    const T* gp = static_cast<const T*>(P.target) + (size_t)it.tgt_row * P.ld_t;
    const T* gq = it.bonus ? gp : static_cast<const T*>(P.draft) + (size_t)it.dft_row * P.ld_d;
    float u_acc = 0.f, u_fin = 0.f;
    if (P.mode == kModeSample && sc.uniforms_ok) {
      u_fin = __ldg(P.uniforms + sc.off + sc.K);
      if (!it.bonus) u_acc = __ldg(P.uniforms + sc.off + it.i);
    }
    if (!timeout && !mbar_wait(&S.pass2_done()[kb], (uint32_t)(k / kPipeBufs) & 1u)) timeout = true;
    if (k == n_local_items(P) - 1 && !timeout && !mbar_wait(&S.pass2a_done()[0], 0u)) timeout = true;
    {
      const int flags = st.flags | (timeout ? kStatusTimeout : 0);
      const float Mp = st.M[0], Mq = st.M[1], ip = st.inv[0], iq = st.inv[1];
      const float px = st.px, qx = st.qx;
      int ks;
      double rem;
      bool take_last;
      const double R = owner_search(S.segt(kb), L.nseg, (double)u_fin, lane, ks, rem, take_last);
      const double tv = it.bonus ? 0.0 : fmin(R, 1.0);
      double theta = 1.0;
      if (tv > (double)sc.D) theta = (double)__fdiv_rn(sc.D, (float)tv);
      int acc = 1;
      if (!it.bonus) {
        const double pi = (1.0 - theta) * (double)px + theta * (double)qx;
        acc = ((double)u_acc * (double)qx < pi) ? 1 : 0;
      }
      const bool sample = P.mode == kModeSample;
      const bool need_cand = sample && flags == 0 && (it.bonus ? !(P.flags & 1u) : acc == 0);
      bool deferred = false;
      int cand = -1;
      if (need_cand) {
        if (!it.bonus && !(R > 0.0)) {
          deferred = true;  // correction from p: recomputed by the slow path
        } else if (ks >= 0) {
          cand = search_segment<T>(P, L, st.pen ? S.bm(kb) : nullptr, gp, gq, it.bonus, ks, rem, take_last, sc.c,
                                   sc.alpha, Mp, Mq, ip, iq, lane);
        }
      }
      if (lane == 0) {
        if (deferred) {
          S.defer()[k >> 5] |= 1u << (k & 31);
        } else if (sample) {
          ItemResult* res = P.results + item;
          res->acc = acc;
          res->cand = cand;
          res->tv = (float)tv;
          res->theta = (float)theta;
          res->px = px;
          res->qx = qx;
        } else {
          const bool bad = flags != 0;
          P.out_tv[item] = bad ? NAN : (float)tv;
          if (P.out_theta) P.out_theta[item] = bad ? NAN : (float)theta;
          if (P.out_px) P.out_px[item] = bad ? NAN : px;
          if (P.out_qx) P.out_qx[item] = bad ? NAN : qx;
        }
      }
      if (sample && !deferred) finish_item(P, it, item, flags, lane, -1, 32, &S.mi()[2]);
    }
    __syncwarp();
    if (lane == 0) mbar_arrive(&S.buf_free()[kb]);
  }
}

// ------------------------------------------------------------- slow path
// One deferred item with all compute warps and direct global loads: the
// same method in 256-token chunks (penalty from a bitmap).
template <typename T>
__device__ __forceinline__ void slow_item(const SampleParams& P, const PipeLayout& L, const PSmem& S, int item, int warp, int lane) {
  constexpr int NW = kNC, NT = kThreadsC;
  const int tid = warp * 32 + lane;
  const int* cu = cu_ptr(P, S);
  const Item it = pdecode(P, cu, item);
  const Scalars sc = item_scalars(P, it, item, cu);
  const int V = P.V;
  const int nch = (V + kChunk - 1) / kChunk;
  const T* gp = static_cast<const T*>(P.target) + (size_t)it.tgt_row * P.ld_t;
  const T* gq = it.bonus ? gp : static_cast<const T*>(P.draft) + (size_t)it.dft_row * P.ld_d;
  if (tid == 0) S.mi()[0] = 0;
  int flags = sc.flags | mark_penalty_set(P, sc, S.bm(0), tid, NT);
  named_sync(kBarC, NT);

  // pass 1
  float refc[2] = {0.f, 0.f}, Ssum[2] = {0.f, 0.f};
  bool have_ref = false;
  for (int kk = warp; kk < nch; kk += NW) {
    float z[2][8];
    global_logits<T>(gp, kk * kChunk, lane, V, S.bm(0), sc.pen, sc.alpha, z[0]);
    if (sc.nrows == 2) {
      global_logits<T>(gq, kk * kChunk, lane, V, S.bm(0), sc.pen, sc.alpha, z[1]);
      chunk_stats_lane<2>(z, sc.c, refc, have_ref, Ssum);
    } else {
      chunk_stats_lane<1>(z, sc.c, refc, have_ref, Ssum);
    }
  }
#pragma unroll
  for (int r = 0; r < 2; ++r) {
    const float ref = have_ref && r < sc.nrows ? refc[r] : -INFINITY;
    const float2 wv = warp_combine(ref, ref > -INFINITY ? Ssum[r] : 0.f);
    if (lane == 0) S.cwp()[warp * 2 + r] = wv;
  }
  named_sync(kBarC, NT);
  float M[2], Sr[2], inv[2];
#pragma unroll
  for (int r = 0; r < 2; ++r) {
    M[r] = -INFINITY;
    Sr[r] = 0.f;
    for (int w = 0; w < NW; ++w) combine_into(S.cwp()[w * 2 + r], M[r], Sr[r]);
  }
#pragma unroll
  for (int r = 0; r < 2; ++r)
    if (r < sc.nrows && (!(Sr[r] > 0.f) || !(Sr[r] < INFINITY) || !(M[r] < INFINITY))) flags |= kStatusBadLogits;
  const bool ok_stats = !(flags & kStatusBadLogits);
  RowProb rp[2];
#pragma unroll
  for (int r = 0; r < 2; ++r) {
    const bool use = ok_stats && r < sc.nrows;
    inv[r] = use ? __fdiv_rn(1.f, Sr[r]) : 1.f;
    if (!use) M[r] = 0.f;
    rp[r].tau_key = 0u;
    rp[r].c = sc.c;
    rp[r].mc = M[r];
    rp[r].invs = inv[r];
    rp[r].kept = 1.0;
  }

  // pass 2 (ponly: chunk sums of p instead of the residual)
  float* seg = S.part();
  bool ponly = it.bonus;
  double R = 0.0;
  int ks = -1;
  double rem = 0.0;
  bool take_last = false;
  float px = 0.f, qx = 0.f;
  double tv = 0.0, theta = 1.0;
  int acc = 1;
  for (int attempt = 0; attempt < 2; ++attempt) {
    for (int kk = warp; kk < nch; kk += NW) {
      float z[8], pp[8];
      global_logits<T>(gp, kk * kChunk, lane, V, S.bm(0), sc.pen, sc.alpha, z);
      probs8<kPZ>(z, 0.f, rp[0], pp);
      float s;
      if (ponly) {
        s = sum8(pp);
      } else {
        float zq[8], qq[8], rr[8];
        global_logits<T>(gq, kk * kChunk, lane, V, S.bm(0), sc.pen, sc.alpha, zq);
        probs8<kPZ>(zq, 0.f, rp[1], qq);
        s = resid8(pp, qq, rr);
      }
      s = warp_sum(s);
      if (lane == 0) seg[kk] = s;
    }
    named_sync(kBarC, NT);
    if (warp == 0) {
      const float uf = (P.mode == kModeSample && sc.uniforms_ok) ? __ldg(P.uniforms + sc.off + sc.K) : 0.f;
      R = owner_search(seg, nch, (double)uf, lane, ks, rem, take_last);
      if (attempt == 0 && lane == 0) {
        if (!it.bonus && sc.x >= 0 && sc.x < V && ok_stats) {
          float zp = to_f32<T>(gp[sc.x]), zq = to_f32<T>(gq[sc.x]);
          if (sc.pen && ((S.bm(0)[sc.x >> 5] >> (sc.x & 31)) & 1u)) {
            zp = penalize(zp, sc.alpha);
            zq = penalize(zq, sc.alpha);
          }
          px = prob_of(zp, sc.c, M[0], inv[0]);
          qx = prob_of(zq, sc.c, M[1], inv[1]);
        }
        tv = it.bonus ? 0.0 : fmin(R, 1.0);
        if (tv > (double)sc.D) theta = (double)sc.D / tv;
        if (!it.bonus) {
          const float ua = (P.mode == kModeSample && sc.uniforms_ok) ? __ldg(P.uniforms + sc.off + it.i) : 0.f;
          const double pi = (1.0 - theta) * (double)px + theta * (double)qx;
          acc = ((double)ua * (double)qx < pi) ? 1 : 0;
        }
        S.mi()[4] = (P.mode == kModeSample && !it.bonus && acc == 0 && !(R > 0.0) && ok_stats) ? 1 : 0;
      }
    }
    named_sync(kBarC, NT);
    if (attempt == 0 && S.mi()[4]) {
      ponly = true;  // no residual mass: the correction is drawn from p
      continue;
    }
    break;
  }

  // candidate (warp 0): the owning chunk, then the lane and element
  if (warp == 0) acc = __shfl_sync(0xffffffffu, acc, 0);
  const bool need_cand =
      P.mode == kModeSample && flags == 0 && ok_stats && (it.bonus ? !(P.flags & 1u) : acc == 0);
  if (warp == 0) {
    int found = -1;
    if (need_cand && ks >= 0) {
      const int ib = ks * kChunk;
      float w[8];
      {
        float zp[8], pp[8];
        global_logits<T>(gp, ib, lane, V, S.bm(0), sc.pen, sc.alpha, zp);
        probs8<kPZ>(zp, 0.f, rp[0], pp);
        if (ponly) {
#pragma unroll
          for (int j = 0; j < 8; ++j) w[j] = pp[j];
        } else {
          float zq[8], qq[8];
          global_logits<T>(gq, ib, lane, V, S.bm(0), sc.pen, sc.alpha, zq);
          probs8<kPZ>(zq, 0.f, rp[1], qq);
          resid8(pp, qq, w);
        }
      }
      if (!take_last) {
        for (int half = 0; half < 2 && found < 0; ++half) {
          const float* wh = w + 4 * half;
          const float ls = (wh[0] + wh[1]) + (wh[2] + wh[3]);
          const float incl = warp_incl_scan(ls, lane);
          const float excl = incl - ls;
          const bool hit = ((double)incl > rem) && ((double)excl <= rem) && ls > 0.f;
          const unsigned m = __ballot_sync(0xffffffffu, hit);
          if (m) {
            const int L0 = __ffs(m) - 1;
            int jj = -1;
            if (lane == L0) {
              double cum = (double)excl;
              for (int j = 0; j < 4; ++j) {
                cum += (double)wh[j];
                if (wh[j] > 0.f && cum > rem) {
                  jj = j;
                  break;
                }
              }
              if (jj < 0)
                for (int j = 3; j >= 0; --j)
                  if (wh[j] > 0.f) {
                    jj = j;
                    break;
                  }
            }
            jj = __shfl_sync(0xffffffffu, jj, L0);
            found = ib + 128 * half + 4 * L0 + jj;
          } else {
            rem -= (double)__shfl_sync(0xffffffffu, incl, 31);
          }
        }
      }
      if (found < 0) {
        for (int half = 1; half >= 0 && found < 0; --half) {
          int lj = -1;
          for (int j = 3; j >= 0; --j)
            if (w[4 * half + j] > 0.f) {
              lj = j;
              break;
            }
          const unsigned m = __ballot_sync(0xffffffffu, lj >= 0);
          if (m) {
            const int L0 = 31 - __clz(m);
            lj = __shfl_sync(0xffffffffu, lj, L0);
            found = ib + 128 * half + 4 * L0 + lj;
          }
        }
      }
    }
    if (lane == 0) {
      if (P.mode == kModeSample) {
        ItemResult* res = P.results + item;
        res->acc = acc;
        res->cand = found;
        res->tv = (float)tv;
        res->theta = (float)theta;
        res->px = px;
        res->qx = qx;
      } else {
        const bool bad = flags != 0;
        P.out_tv[item] = bad ? NAN : (float)tv;
        if (P.out_theta) P.out_theta[item] = bad ? NAN : (float)theta;
        if (P.out_px) P.out_px[item] = bad ? NAN : px;
        if (P.out_qx) P.out_qx[item] = bad ? NAN : qx;
      }
    }
  }
  {
    const int f = warp_or(flags);
    if (lane == 0 && f) atomicOr(&S.mi()[0], f);
  }
  named_sync(kBarC, NT);
  flags = S.mi()[0];
  if (P.mode == kModeSample) finish_item(P, it, item, flags, tid, kBarC, NT, &S.mi()[3]);
  // clear the bitmap for the next deferred item
  if (sc.pen) {
    for (int j = sc.h0 + tid; j < sc.h1; j += NT) {
      const int t = __ldg(P.hist + j);
      if (t >= 0 && t < V) S.bm(0)[t >> 5] = 0u;
    }
    for (int j = tid; j < sc.npre; j += NT) {
      const int t = __ldg(P.draft_tokens + sc.d0 + j);
      if (t >= 0 && t < V) S.bm(0)[t >> 5] = 0u;
    }
  }
  named_sync(kBarC, NT);
}

// ---------------------------------------------------------------- kernel
template <typename T>
__global__ void __launch_bounds__(kPipeThreads, 1) pipe_verify_kernel(const __grid_constant__ SampleParams P) {
  const PipeLayout& L = P.PL;
  const PSmem S(L);
  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int tid = threadIdx.x;
  if (tid == 0) {
    for (int s = 0; s < L.slots_a; ++s) {
      mbar_init(&S.full_a()[s], 1);
      mbar_init(&S.empty_a()[s], kNA);
    }
    for (int s = 0; s < L.slots_b; ++s) {
      mbar_init(&S.full_b()[s], 1);
      mbar_init(&S.empty_b()[s], kNB);
    }
    for (int i = 0; i < kPipeBufs; ++i) {
      mbar_init(&S.list_ready()[i], 1);
      mbar_init(&S.pass1_done()[i], kNA);
      mbar_init(&S.stats_full()[i], 1);
      mbar_init(&S.pass2_done()[i], kNB);
      mbar_init(&S.buf_free()[i], 2);
    }
    mbar_init(&S.pass2a_done()[0], kNA);
    fence_mbar_init();
  }
  for (int w = tid; w < kPipeMaxIters / 32; w += kPipeThreads) S.defer()[w] = 0u;
  if (P.B + 1 <= kPipeCuCap)
    for (int i = tid; i <= P.B; i += kPipeThreads) S.cu()[i] = __ldg(P.cu_draft + i);
  if (tid < 16) S.mi()[tid] = 0;
  __syncthreads();

  if (warp < kNA) {
    a_stream<T>(P, L, S, warp, lane);
  } else if (warp == kNA) {
    a_setup<T>(P, L, S, lane);
  } else if (warp < kNA + 1 + kNB) {
    b_stream<T>(P, L, S, warp - kNA - 1, lane);
  } else if (warp == kNA + 1 + kNB) {
    b_tail<T>(P, L, S, lane);
  } else {
    if (lane == 0) {
      if (warp == kNC) producer<T, true>(P, L, S);
      else producer<T, false>(P, L, S);
    }
    return;
  }
  // deferred items of this CTA, after the pipeline has drained (bitmap 0
  // serves their penalty sets)
  named_sync(kBarC, kThreadsC);
  for (int q = tid; q < L.bm_words; q += kThreadsC) S.bm(0)[q] = 0u;
  named_sync(kBarC, kThreadsC);
  int k = 0;
  for (int item = blockIdx.x; item < P.n_items; item += gridDim.x, ++k)
    if ((S.defer()[k >> 5] >> (k & 31)) & 1u) slow_item<T>(P, L, S, item, warp, lane);
}

}  // namespace

// Layout for the pipelined kernel (-1 if it does not fit `max_smem`).
int choose_pipe_layout(int V, int elem_bytes, int max_smem, PipeLayout* out) {
  for (int slots_a = kPipeSlotsA; slots_a >= 2; --slots_a) {
    const PipeLayout L = make_pipe_layout(V, elem_bytes, slots_a, kPipeSlotsB);
    if (L.total <= max_smem) {
      *out = L;
      return 0;
    }
  }
  return -1;
}

int launch_pipe_verify(SampleParams& P, bool bf16, int num_sms, cudaStream_t stream) {
  const int smem = P.PL.total;
  const int grid = P.n_items < num_sms ? P.n_items : num_sms;
  if (grid <= 0) return 0;
  P.C = 1;
  P.n_clusters = grid;
  if (bf16) {
    auto kern = pipe_verify_kernel<__nv_bfloat16>;
    if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, smem) != cudaSuccess) {
      cudaGetLastError();
      return -8;
    }
    kern<<<grid, kPipeThreads, smem, stream>>>(P);
  } else {
    auto kern = pipe_verify_kernel<float>;
    if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, smem) != cudaSuccess) {
      cudaGetLastError();
      return -8;
    }
    kern<<<grid, kPipeThreads, smem, stream>>>(P);
  }
  if (cudaGetLastError() != cudaSuccess) return -7;
  return 0;
}

}  // namespace sv
