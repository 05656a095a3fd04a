// Fused mentored speculative sampling for GB300 (sm_103a).
//
// A thread-block cluster of C CTAs (C = 1 .. 16) handles one work item at a
// time: a draft position (target row i and draft row i of a request) or a
// request's bonus row (target row K).  Each CTA owns a contiguous slice of
// the vocabulary.  A producer warp streams the CTA's slice of both rows from
// global memory into a shared-memory ring with 1-D TMA bulk copies (one
// slot = one stage: the CTA's next 256 tokens per consumer warp of the target
// row followed by the same tokens of the draft row); 16 consumer warps work on the slots.  Per item:
//
//   pass 1  repetition penalty and temperature; running (reference, sum) of
//           e = 2^(z'c - ref) per row, c = log2(e)/T: one exponential per
//           logit.  The resident variant also keeps e (or, with top-p, the
//           penalised logit z') of every token in shared memory.
//   sync 1  (max, sum) of both rows: warps -> CTA -> cluster through DSMEM.
//   top-p   (optional) a mass-weighted radix select over the exact logit
//           keys, four 8-bit digits, each histogram reduced over the cluster.
//   pass 2  r = max(p - q, 0) summed per 256-token chunk (bonus rows: p).
//           The resident variant reads its shared-memory copy; the streaming
//           variant re-reads the slice (an L2 hit: it was read moments ago)
//           and recomputes p and q.  TV d = sum r ("What I Gave Up to Make
//           Speculative Decoding Faster", "A knob for accepting more draft
//           tokens": d = 1/2 sum|p-q|, equal to sum max(p-q, 0) for two
//           distributions).
//   sync 2  chunk and CTA prefix sums of r across the cluster.
//   decide  theta = min(1, D/d); pi(x) = (1-theta) p(x) + theta q(x); accept
//           iff u q(x) < pi(x); the residual candidate = inverse CDF of r at
//           u_fin, found by the CTA, chunk and lane that hold it.  Bonus rows
//           take the inverse CDF of p.
//   emit    the last CTA to finish a request (an atomic counter) scans the K
//           acceptance flags with a warp ballot and writes the tokens.
//
// Acceptance and correction are evaluated speculatively at every position;
// the uniforms are assigned per position, so this equals evaluating them in
// order and stopping at the first rejection.  The resident variant reads
// each logit from HBM once and suits small batches (few items, many CTAs
// each); the streaming variant keeps about one item per SM in flight and
// suits large batches.
#include "common.cuh"
#include "spec_internal.h"
#include "verify_common.cuh"

namespace sv {

namespace {


struct Shared {
  unsigned char* ring;
  float* e;          // [2][slice] (resident variant)
  uint32_t* bitmap;  // [nch * 8]
  float* refc;       // [2][nch]   (resident variant)
  float* fac;        // [2][nch]   (resident variant)
  float* seg;        // [nch]
  float2* wpart;     // [2][16]
  double* xchg;      // [2][C][kXchgDoubles]
  float* hist;       // [2 buf][2 rows][256]
  float* tot;        // [2 rows][256]
  double* misc_d;    // 16 doubles
  int* misc_i;       // 16 ints
  float* misc_f;     // 16 floats
  uint64_t* full;
  uint64_t* empty;
  uint64_t* csync;   // [2]
};

__device__ __forceinline__ Shared carve(unsigned char* smem, const SmemLayout& L) {
  Shared S;
  S.ring = smem;
  S.e = reinterpret_cast<float*>(smem + L.off_e);
  S.bitmap = reinterpret_cast<uint32_t*>(smem + L.off_bitmap);
  S.refc = reinterpret_cast<float*>(smem + L.off_refc);
  S.fac = reinterpret_cast<float*>(smem + L.off_fac);
  S.seg = reinterpret_cast<float*>(smem + L.off_seg);
  S.wpart = reinterpret_cast<float2*>(smem + L.off_wpart);
  S.xchg = reinterpret_cast<double*>(smem + L.off_xchg);
  S.hist = reinterpret_cast<float*>(smem + L.off_hist);
  S.tot = reinterpret_cast<float*>(smem + L.off_tot);
  S.misc_d = reinterpret_cast<double*>(smem + L.off_misc);
  S.misc_i = reinterpret_cast<int*>(smem + L.off_misc + 128);
  S.misc_f = reinterpret_cast<float*>(smem + L.off_misc + 192);
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + L.off_bar);
  S.full = bars;
  S.empty = bars + L.nslots;
  S.csync = bars + 2 * L.nslots;
  return S;
}

// Barrier over the consumer warps only (the producer warp keeps streaming).
template <int NCT>
__device__ __forceinline__ void consumer_sync() { named_sync(1, NCT); }

// misc_i: [0] status bits of the item found by this CTA, [2] finalize flag,
// [4] owner CTA of the final draw, [5] owner takes the last positive token,
// [8 + row] selected top-p digit.
// misc_d: [0] p(x), [1] q(x), [4..7] top-p mass above / in the selected bin,
// [10..13] (M, S) of both rows, [14] R, [15] this CTA's prefix of R.
// misc_f: [0], [2] 1/S per row, [4 + row] 1/kept mass.
constexpr int kMiFlags = 0, kMiFinalize = 2;
constexpr int kMdPx = 0, kMdQx = 1;

struct ClusterPhase {
  uint32_t cph = 0;  // cluster exchanges done by this CTA
  bool failed = false;
};

__device__ __forceinline__ double* xchg_slot(const Shared& S, int C, uint32_t buf, int c) {
  return S.xchg + ((size_t)buf * C + c) * kXchgDoubles;
}

// Warp 0 publishes up to four doubles into exchange slot [buf][rank] of every
// CTA of the cluster: lane c writes CTA c and then arrives (release, cluster
// scope) on CTA c's csync[buf], so the C pushes proceed in parallel.  Every
// consumer thread then waits on its own csync[buf]; afterwards
// S.xchg[buf][c][*] holds the values of CTA c.  The caller makes any other
// shared-memory data it wants visible (fence + CTA barrier) beforehand.
// Two alternating barriers and buffers keep consecutive exchanges apart.
__device__ __forceinline__ bool cluster_exchange(const Shared& S, ClusterPhase& ph, int C, uint32_t rank,
                                                 int nvals, double a0, double a1, double a2, double a3) {
  const uint32_t buf = ph.cph & 1u;
  const uint32_t parity = (ph.cph >> 1) & 1u;
  const int lane = threadIdx.x & 31;
  if (threadIdx.x < 32 && lane < C) {
    const uint32_t base = map_rank(xchg_slot(S, C, buf, (int)rank), (uint32_t)lane);
    if (nvals > 0) st_remote_f64(base, a0);
    if (nvals > 1) st_remote_f64(base + 8u, a1);
    if (nvals > 2) st_remote_f64(base + 16u, a2);
    if (nvals > 3) st_remote_f64(base + 24u, a3);
    mbar_arrive_remote(&S.csync[buf], (uint32_t)lane);
  }
  const bool ok = ph.failed ? false : mbar_wait_cluster(&S.csync[buf], parity);
  if (!ok) ph.failed = true;  // after one timeout, stop waiting
  ph.cph++;
  return ok;
}

// Warp-parallel log-sum combine of up to 16 (ref, sum) pairs per row: lane l
// holds pair (l & 15) of row (l >> 4).  Every lane of a row's half-warp gets
// M = max ref and S = sum_j S_j 2^(ref_j - M) (fp64 accumulation, one exp2f
// per lane).
__device__ __forceinline__ void halfwarp_combine(float ref, double s, float& M, double& Ssum) {
  float m = ref;
#pragma unroll
  for (int o = 8; o > 0; o >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, o));
  double v = (ref > -INFINITY && m > -INFINITY) ? s * (double)exp2f(ref - m) : 0.0;
#pragma unroll
  for (int o = 8; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
  M = m;
  Ssum = v;
}


// A lane's 8 logits of chunk `ib` (slice offset) of a staged row, in fp32,
// -inf past the live length, penalised where the bitmap says so.
template <typename T>
__device__ __forceinline__ void stage_logits(const T* chunk, int ib, int lane, int len, const uint32_t* bitmap,
                                             bool pen, float alpha, float* z) {
  load4(chunk + 4 * lane, z);
  load4(chunk + 128 + 4 * lane, z + 4);
  if (ib + kChunk > len) {
#pragma unroll
    for (int j = 0; j < 8; ++j)
      if (ib + lane_elem(lane, j) >= len) z[j] = -INFINITY;
  }
  if (pen && __any_sync(0xffffffffu, bitmap[(ib >> 5) + (lane & 7)] != 0u)) {
    const uint32_t wa = bitmap[(ib >> 5) + (lane >> 3)];
    const uint32_t wb = bitmap[(ib >> 5) + 4 + (lane >> 3)];
    const uint32_t sh = 4u * (lane & 7);
    uint32_t m = ((wa >> sh) & 0xFu) | (((wb >> sh) & 0xFu) << 4);
    while (m) {
      const int j = __ffs(m) - 1;
      m &= m - 1;
      float v = z[0];
#pragma unroll
      for (int jj = 1; jj < 8; ++jj)
        if (jj == j) v = z[jj];
      v = penalize(v, alpha);
#pragma unroll
      for (int jj = 0; jj < 8; ++jj)
        if (jj == j) z[jj] = v;
    }
  }
}

// A lane's 8 raw values of a staged chunk, as loaded (converted later).
template <typename T>
struct Raw8;
template <>
struct Raw8<__nv_bfloat16> {
  uint2 a, b;
};
template <>
struct Raw8<float> {
  float4 a, b;
};

__device__ __forceinline__ void load_raw8(const __nv_bfloat16* chunk, int lane, Raw8<__nv_bfloat16>& r) {
  r.a = *reinterpret_cast<const uint2*>(chunk + 4 * lane);
  r.b = *reinterpret_cast<const uint2*>(chunk + 128 + 4 * lane);
}
__device__ __forceinline__ void load_raw8(const float* chunk, int lane, Raw8<float>& r) {
  r.a = *reinterpret_cast<const float4*>(chunk + 4 * lane);
  r.b = *reinterpret_cast<const float4*>(chunk + 128 + 4 * lane);
}
__device__ __forceinline__ void cvt_raw8(const Raw8<__nv_bfloat16>& r, float* z) {
  z[0] = __uint_as_float(r.a.x << 16); z[1] = __uint_as_float(r.a.x & 0xffff0000u);
  z[2] = __uint_as_float(r.a.y << 16); z[3] = __uint_as_float(r.a.y & 0xffff0000u);
  z[4] = __uint_as_float(r.b.x << 16); z[5] = __uint_as_float(r.b.x & 0xffff0000u);
  z[6] = __uint_as_float(r.b.y << 16); z[7] = __uint_as_float(r.b.y & 0xffff0000u);
}
__device__ __forceinline__ void cvt_raw8(const Raw8<float>& r, float* z) {
  z[0] = r.a.x; z[1] = r.a.y; z[2] = r.a.z; z[3] = r.a.w;
  z[4] = r.b.x; z[5] = r.b.y; z[6] = r.b.z; z[7] = r.b.w;
}

// Both rows of a staged chunk (row 1 at +row_stride elements; only row 0
// when nrows == 1): every shared-memory load is issued first, then the
// conversion; the tail mask and the repetition penalty are rare,
// warp-uniform branches.
template <typename T>
__device__ __forceinline__ void stage_chunk2(const T* chunk, int row_stride, int nrows, int ib, int lane, int len,
                                             const uint32_t* bitmap, bool pen, float alpha, float (&z)[2][8]) {
  Raw8<T> r0, r1;
  load_raw8(chunk, lane, r0);
  if (nrows == 2) load_raw8(chunk + row_stride, lane, r1);
  const uint32_t pw = pen ? bitmap[(ib >> 5) + (lane & 7)] : 0u;
  cvt_raw8(r0, z[0]);
  if (nrows == 2) cvt_raw8(r1, z[1]);
  if (ib + kChunk > len) {
#pragma unroll
    for (int j = 0; j < 8; ++j)
      if (ib + lane_elem(lane, j) >= len) z[0][j] = z[1][j] = -INFINITY;
  }
  if (pen && __any_sync(0xffffffffu, pw != 0u)) {
    const uint32_t wa = bitmap[(ib >> 5) + (lane >> 3)];
    const uint32_t wb = bitmap[(ib >> 5) + 4 + (lane >> 3)];
    const uint32_t sh = 4u * (lane & 7);
    uint32_t m = ((wa >> sh) & 0xFu) | (((wb >> sh) & 0xFu) << 4);
    while (m) {
      const int j = __ffs(m) - 1;
      m &= m - 1;
      float v0 = z[0][0], v1 = z[1][0];
#pragma unroll
      for (int jj = 1; jj < 8; ++jj)
        if (jj == j) { v0 = z[0][jj]; v1 = z[1][jj]; }
      v0 = penalize(v0, alpha);
      v1 = penalize(v1, alpha);
#pragma unroll
      for (int jj = 0; jj < 8; ++jj)
        if (jj == j) { z[0][jj] = v0; z[1][jj] = v1; }
    }
  }
}


// The lane's 8 stored values of chunk k (resident e-array); `fill` past the
// live length.
__device__ __forceinline__ void load_e8(const float* e_row, int k, int lane, int len, float fill, float* v) {
  const int ib = k * kChunk;
  if (ib + kChunk <= len) {
    load4(e_row + ib + 4 * lane, v);
    load4(e_row + ib + 128 + 4 * lane, v + 4);
  } else {
#pragma unroll
    for (int j = 0; j < 8; ++j) {
      const int idx = ib + lane_elem(lane, j);
      v[j] = idx < len ? e_row[idx] : fill;
    }
  }
}


// Pass-1 statistics of one chunk of NR rows (1 or 2) for one warp: per row a
// running reference refc (warp-uniform, units of z'c) and a lane sum Ssum of
// 2^(z'c - refc).  A reference starts at the row's first chunk maximum and
// only moves up, when a chunk would overflow (sum above 2^64).  e receives
// the chunk's 2^(z'c - refc).
template <int NR>
__device__ __forceinline__ void chunk_stats_n(float (&z)[2][8], float c, float* refc, bool& have_ref, float* Ssum,
                                              float (&e)[2][8]) {
  const float kLim = 18446744073709551616.0f;  // 2^64
  if (!have_ref) {
#pragma unroll
    for (int r = 0; r < NR; ++r) {
      const float mx = warp_max(max8(z[r]));
      refc[r] = (mx > -INFINITY) ? mx * c : 0.f;
    }
    have_ref = true;
  }
  float s[NR];
#pragma unroll
  for (int r = 0; r < NR; ++r) {
    exps8(z[r], c, refc[r], e[r]);
    s[r] = sum8(e[r]);
  }
  bool bad = false;
#pragma unroll
  for (int r = 0; r < NR; ++r) bad |= !(s[r] <= kLim);
  if (__any_sync(0xffffffffu, bad)) {
#pragma unroll
    for (int r = 0; r < NR; ++r) {
      if (__any_sync(0xffffffffu, !(s[r] <= kLim))) {
        const float mx = warp_max(max8(z[r]));
        const float nref = (mx > -INFINITY) ? mx * c : 0.f;
        if (nref > refc[r]) {
          Ssum[r] *= ex2(refc[r] - nref);
          refc[r] = nref;
        }
        exps8(z[r], c, refc[r], e[r]);
        s[r] = sum8(e[r]);
      }
    }
  }
#pragma unroll
  for (int r = 0; r < NR; ++r) Ssum[r] += s[r];
}


// Waits for the next ring slot (consumer side); returns the slot index.
__device__ __forceinline__ uint32_t next_full(const Shared& S, const SmemLayout& L, RingCursor& rc, bool& timeout) {
  const uint32_t slot = rc.slot;
  if (!timeout && !mbar_wait(&S.full[slot], rc.phase)) timeout = true;  // after one timeout, stop waiting
  rc.advance(L.nslots);
  return slot;
}

__device__ __forceinline__ void release_slot(const Shared& S, uint32_t slot, int lane) {
  __syncwarp();
  if (lane == 0) mbar_arrive(&S.empty[slot]);
}

}  // namespace

// -------------------------------------------------------------------- kernel
template <typename T, bool TOPP, bool RESIDENT>
__global__ void __launch_bounds__(((RESIDENT ? kResidentWarps : kStreamWarps) + 1) * 32, RESIDENT ? 1 : kStreamCtasPerSm)
    sample_verify_kernel(const __grid_constant__ SampleParams P) {
  constexpr int NW = RESIDENT ? kResidentWarps : kStreamWarps;  // consumer warps
  constexpr int NCT = NW * 32;                                    // consumer threads
  constexpr int STAGE = NW * kChunk;                              // tokens of each row per slot
  extern __shared__ __align__(128) unsigned char smem[];
  const SmemLayout& L = P.L;
  Shared S = carve(smem, L);
  const int C = P.C;
  const uint32_t rank = cluster_rank();
  const int cluster_id = blockIdx.x / C;
  const int v0 = (int)rank * L.slice;
  const int len = max(0, min(L.slice, P.V - v0));
  const int nst = (len + STAGE - 1) / STAGE;
  const int nch = (len + kChunk - 1) / kChunk;
  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int tid = threadIdx.x;
  constexpr bool kFromE = RESIDENT && !TOPP;  // stored values are e, not logits

  if (tid == 0) {
    for (int s = 0; s < L.nslots; ++s) {
      mbar_init(&S.full[s], 1);
      mbar_init(&S.empty[s], NW);
    }
    mbar_init(&S.csync[0], C);
    mbar_init(&S.csync[1], C);
    fence_mbar_init();
  }
  cluster_sync_all();

  if (warp == NW) {
    // ------------------------------------------------------------ producer
    if (lane == 0 && len > 0) {
      const uint64_t keep_policy = l2_policy_evict_last();
      const uint64_t drop_policy = l2_policy_evict_first();
      const int es = (int)sizeof(T);
      RingCursor rc;
      bool ptimeout = false;
      for (int item = cluster_id; item < P.n_items; item += P.n_clusters) {
        const Item it = decode_item(P, item);
        const unsigned char* rowp =
            static_cast<const unsigned char*>(P.target) + ((size_t)it.tgt_row * P.ld_t + v0) * es;
        const unsigned char* rowq =
            it.bonus ? rowp : static_cast<const unsigned char*>(P.draft) + ((size_t)it.dft_row * P.ld_d + v0) * es;
        // pass 1; the streaming variant then re-reads for the radix passes and pass 2
        const int npass = RESIDENT ? 1 : 2 + radix_passes<TOPP>(P, it.b);
        for (int pass = 0; pass < npass; ++pass) {
          const uint64_t pol = (RESIDENT || pass == npass - 1) ? drop_policy : keep_policy;
          for (int st = 0; st < nst; ++st) {
            const uint32_t slot = rc.slot;
            // first use of a slot: the phase "before" its first completes at once
            if (!ptimeout && !mbar_wait(&S.empty[slot], rc.phase ^ 1u)) ptimeout = true;  // consumers see their own
            rc.advance(L.nslots);
            const int n = min(STAGE, len - st * STAGE);
            const uint32_t bytes = (uint32_t)((n * es + 15) & ~15);
            unsigned char* dst = S.ring + (size_t)slot * L.slot_bytes;
            mbar_arrive_expect_tx(&S.full[slot], it.bonus ? bytes : 2 * bytes);
            bulk_g2s(dst, rowp + (size_t)st * STAGE * es, bytes, &S.full[slot], pol);
            if (!it.bonus)
              bulk_g2s(dst + (size_t)STAGE * es, rowq + (size_t)st * STAGE * es, bytes, &S.full[slot], pol);
          }
        }
      }
    }
    __syncwarp();
  } else {
    // ----------------------------------------------------------- consumers
    ClusterPhase ph;
    RingCursor seq;
    bool timeout = false;
    for (int item = cluster_id; item < P.n_items; item += P.n_clusters) {
      const Item it = decode_item(P, item);
      const int b = it.b;
      const int K = it.K;
      const int d0 = __ldg(P.cu_draft + b);
      const int off = d0 + b;
      const int nrows = it.bonus ? 1 : 2;
      int flags = 0;
      if (!it.rows_ok || K < 0 || K > P.max_k || K > kMaxK) flags |= kStatusBadK;
      const float T_ = P.temperature ? __ldg(P.temperature + b) : 1.f;
      const float alpha = P.rep_penalty ? __ldg(P.rep_penalty + b) : 1.f;
      const float tp = P.top_p ? __ldg(P.top_p + b) : 1.f;
      const float D = P.tv_budget ? __ldg(P.tv_budget + b) : 0.f;
      const bool params_ok = item_params_ok(P, b);
      if (!params_ok) flags |= kStatusBadParam;
      // invalid scalars are reported as such; the statistics then use T = 1
      // and no penalty so that they raise no other flag
      const float c = __fdiv_rn(1.44269504088896341f, params_ok ? T_ : 1.f);  // log2(e)/T
      const int x = it.bonus ? -1 : __ldg(P.draft_tokens + item);
      if (!it.bonus && (x < 0 || x >= P.V)) flags |= kStatusBadToken;
      const int h0 = P.cu_hist ? __ldg(P.cu_hist + b) : 0;
      const int h1 = P.cu_hist ? __ldg(P.cu_hist + b + 1) : 0;
      const int npre = it.bonus ? (it.rows_ok ? K : 0) : it.i;  // drafts before this row
      const bool pen = params_ok && (alpha != 1.f) && ((h1 > h0) || npre > 0) && len > 0;
      const int nrad = radix_passes<TOPP>(P, b);
      const T* gp_row = static_cast<const T*>(P.target) + (size_t)it.tgt_row * P.ld_t + v0;
      const T* gq_row = it.bonus ? gp_row : static_cast<const T*>(P.draft) + (size_t)it.dft_row * P.ld_d + v0;

      // ---- penalty set of this row within the CTA slice; token validity
      const bool cpen = pen;
      if (tid == 0) S.misc_i[kMiFlags] = 0;
      if (cpen)
        for (int w = tid; w < L.nch * 8; w += NCT) S.bitmap[w] = 0u;
      consumer_sync<NCT>();
      for (int j = h0 + tid; j < h1; j += NCT) {
        const int t = __ldg(P.hist + j);
        if (t < 0 || t >= P.V) flags |= kStatusBadToken;
        else if (cpen && t >= v0 && t < v0 + len) atomicOr(&S.bitmap[(t - v0) >> 5], 1u << ((t - v0) & 31));
      }
      for (int j = tid; j < npre; j += NCT) {
        const int t = __ldg(P.draft_tokens + d0 + j);
        if (t < 0 || t >= P.V) flags |= kStatusBadToken;
        else if (cpen && t >= v0 && t < v0 + len) atomicOr(&S.bitmap[(t - v0) >> 5], 1u << ((t - v0) & 31));
      }
      consumer_sync<NCT>();

      // ---- pass 1: statistics of both rows (resident: also keep the values)
      {
        float refc[2] = {0.f, 0.f}, Ssum[2] = {0.f, 0.f};
        bool have_ref = false;
        for (int st = 0; st < nst; ++st) {
          const uint32_t slot = next_full(S, L, seq, timeout);
          const int k = st * NW + warp;
          if (k < nch) {
            const int ib = k * kChunk;
            const T* base = reinterpret_cast<const T*>(S.ring + (size_t)slot * L.slot_bytes) + warp * kChunk;
            float z[2][8];
            stage_chunk2<T>(base, STAGE, nrows, ib, lane, len, S.bitmap, cpen, alpha, z);
            if constexpr (RESIDENT) {
              float e[2][8];
              if (nrows == 2) chunk_stats_n<2>(z, c, refc, have_ref, Ssum, e);
              else chunk_stats_n<1>(z, c, refc, have_ref, Ssum, e);
              // the store holds e, or z' with top-p; row capacity is L.slice
              for (int r = 0; r < nrows; ++r) {
                float* dst = S.e + (size_t)r * L.slice + ib;
                const float* sv8 = TOPP ? z[r] : e[r];
                if (ib + 4 * lane < L.slice)
                  *reinterpret_cast<float4*>(dst + 4 * lane) = make_float4(sv8[0], sv8[1], sv8[2], sv8[3]);
                if (ib + 128 + 4 * lane < L.slice)
                  *reinterpret_cast<float4*>(dst + 128 + 4 * lane) = make_float4(sv8[4], sv8[5], sv8[6], sv8[7]);
                if (lane == 0) S.refc[r * L.nch + k] = refc[r];
              }
            } else {
              if (nrows == 2) chunk_stats_lane<2>(z, c, refc, have_ref, Ssum);
              else chunk_stats_lane<1>(z, c, refc, have_ref, Ssum);
            }
          }
          release_slot(S, slot, lane);
        }
        for (int r = 0; r < 2; ++r) {
          if constexpr (RESIDENT) {
            const float Sw = warp_sum(Ssum[r]);
            if (lane == 0)
              S.wpart[r * kMaxConsumerWarps + warp] = make_float2(have_ref && r < nrows ? refc[r] : -INFINITY, Sw);
          } else {
            // combine the lanes' (reference, sum) pairs
            const float ref = have_ref && r < nrows ? refc[r] : -INFINITY;
            const float Mw = warp_max(ref);
            const double v = (ref > -INFINITY && Mw > -INFINITY) ? (double)Ssum[r] * (double)exp2f(ref - Mw) : 0.0;
            const double Sw = warp_sum_d(v);
            if (lane == 0) S.wpart[r * kMaxConsumerWarps + warp] = make_float2(Mw, (float)Sw);
          }
        }
      }
      consumer_sync<NCT>();

      // ---- sync 1: (M, S) per row, warps -> CTA -> cluster
      {
        double a0 = 0.0, a1 = 0.0, a2 = 0.0, a3 = 0.0;
        if (warp == 0) {
          const int r = lane >> 4, w = lane & 15;
          const float2 v = (r < nrows && w < NW) ? S.wpart[r * kMaxConsumerWarps + w] : make_float2(-INFINITY, 0.f);
          float M;
          double Ssum;
          halfwarp_combine(v.x, (double)v.y, M, Ssum);
          a0 = __shfl_sync(0xffffffffu, (double)M, 0);
          a1 = __shfl_sync(0xffffffffu, Ssum, 0);
          a2 = __shfl_sync(0xffffffffu, (double)M, 16);
          a3 = __shfl_sync(0xffffffffu, Ssum, 16);
        }
        if (!cluster_exchange(S, ph, C, rank, 4, a0, a1, a2, a3)) timeout = true;
      }
      if (warp == 0) {
        const uint32_t buf = (ph.cph - 1) & 1u;
        const int r = lane >> 4, cc = lane & 15;
        float ref = -INFINITY;
        double s = 0.0;
        if (cc < C) {
          const double* xs = xchg_slot(S, C, buf, cc);
          ref = (float)xs[2 * r];
          s = xs[2 * r + 1];
        }
        float M;
        double Ssum;
        halfwarp_combine(ref, s, M, Ssum);
        if (cc == 0) {
          S.misc_d[10 + 2 * r] = (double)M;
          S.misc_d[11 + 2 * r] = Ssum;
          S.misc_f[2 * r] = (float)(1.0 / Ssum);
        }
      }
      consumer_sync<NCT>();
      double Mr[2], Sr[2];
      float invS[2];
      for (int r = 0; r < 2; ++r) {
        Mr[r] = S.misc_d[10 + 2 * r];
        Sr[r] = S.misc_d[11 + 2 * r];
        invS[r] = S.misc_f[2 * r];
      }
      for (int r = 0; r < nrows; ++r)
        if (!(Sr[r] > 0.0) || !(Sr[r] < INFINITY) || !(Mr[r] < INFINITY)) flags |= kStatusBadLogits;
      const bool ok_stats = !(flags & kStatusBadLogits);

      // ---- chunk factors fac_k = 2^(ref_k - M) / S (resident e store)
      if constexpr (kFromE) {
        for (int j = tid; j < nrows * nch; j += NCT) {
          const int r = j / nch, k = j % nch;
          S.fac[r * L.nch + k] = ok_stats ? exp2f(S.refc[r * L.nch + k] - (float)Mr[r]) * invS[r] : 0.f;
        }
        consumer_sync<NCT>();
      }

      RowProb rp[2];
      for (int r = 0; r < 2; ++r) {
        rp[r].tau_key = 0u;
        rp[r].c = c;
        rp[r].mc = (float)(ok_stats && Mr[r] > -INFINITY ? Mr[r] : 0.0);
        rp[r].kept = (ok_stats && r < nrows) ? Sr[r] : 1.0;
        rp[r].invs = (ok_stats && r < nrows) ? invS[r] : 1.f;
      }

      // ---- top-p: tau per row by a mass-weighted radix select over the exact
      // logit keys, four 8-bit digits, MSB first: the largest key whose upper
      // set {key >= tau} holds at least top_p of the mass (the "Speculative
      // Decoding" note: both p and q include top-p)
      if constexpr (TOPP) {
        if (nrad > 0) {
          const bool work = ok_stats;
          uint32_t prefix[2] = {0u, 0u};
          double above[2] = {0.0, 0.0};
          const double target[2] = {(double)tp * Sr[0], (double)tp * Sr[1]};
          double kept[2] = {Sr[0], Sr[1]};
          for (int pass = 0; pass < 4; ++pass) {
            const int shift = 24 - 8 * pass;
            const uint32_t hb = ph.cph & 1u;
            float* hist = S.hist + hb * 512;
            for (int j = tid; j < 512; j += NCT) hist[j] = 0.f;
            consumer_sync<NCT>();
            auto accumulate = [&](const float* zv, int r) {
#pragma unroll
              for (int j = 0; j < 8; ++j) {
                const uint32_t key = order_key(zv[j]);
                const bool match = pass == 0 || (key >> (shift + 8)) == (prefix[r] >> (shift + 8));
                if (match) {
                  const float w = ex2(fmaf(zv[j], c, -rp[r].mc));
                  if (w > 0.f) atomicAdd(&hist[r * 256 + ((key >> shift) & 255u)], w);
                }
              }
            };
            if constexpr (RESIDENT) {
              if (work)
                for (int r = 0; r < nrows; ++r)
                  for (int k = warp; k < nch; k += NW) {
                    float zv[8];
                    load_e8(S.e + (size_t)r * L.slice, k, lane, len, -INFINITY, zv);
                    accumulate(zv, r);
                  }
            } else {
              for (int st = 0; st < nst; ++st) {
                const uint32_t slot = next_full(S, L, seq, timeout);
                const int k = st * NW + warp;
                if (work && k < nch)
                  for (int r = 0; r < nrows; ++r) {
                    const T* chunk = reinterpret_cast<const T*>(S.ring + (size_t)slot * L.slot_bytes) +
                                     r * STAGE + warp * kChunk;
                    float zv[8];
                    stage_logits<T>(chunk, k * kChunk, lane, len, S.bitmap, cpen, alpha, zv);
                    accumulate(zv, r);
                  }
                release_slot(S, slot, lane);
              }
            }
            fence_acq_rel_cluster();
            consumer_sync<NCT>();
            if (!cluster_exchange(S, ph, C, rank, 0, 0.0, 0.0, 0.0, 0.0)) timeout = true;
            for (int j = tid; j < 512; j += NCT) {  // gather the C histograms: (row, bin)
              const int r = j >> 8, bin = j & 255;
              double s = 0.0;
              if (r < nrows)
                for (int cc = 0; cc < C; ++cc)
                  s += (double)ld_remote_f32(map_rank(&hist[r * 256 + bin], (uint32_t)cc));
              S.tot[r * 256 + bin] = (float)s;
            }
            consumer_sync<NCT>();
            if (warp < nrows) {
              // lane owns bins [8*lane, 8*lane+8): the largest digit d with
              // above + mass(bins >= d) >= target
              const int r = warp;
              double lsum = 0.0;
              for (int j = 0; j < 8; ++j) lsum += (double)S.tot[r * 256 + 8 * lane + j];
              double incl = lsum;  // mass of this lane's block and every block above it
              for (int o = 1; o < 32; o <<= 1) {
                const double t = __shfl_down_sync(0xffffffffu, incl, o);
                if (lane + o < 32) incl += t;
              }
              const double excl = incl - lsum;
              const double need = target[r] - above[r];
              const unsigned m = __ballot_sync(0xffffffffu, (excl < need) && (excl + lsum >= need));
              int dsel = 0;
              double cum = 0.0, bm = 0.0;
              if (m) {
                const int L0 = 31 - __clz(m);
                cum = __shfl_sync(0xffffffffu, excl, L0);
                dsel = 8 * L0;
                for (int j = 7; j >= 0; --j) {
                  const double v = (double)S.tot[r * 256 + 8 * L0 + j];
                  if (cum + v >= need) { dsel = 8 * L0 + j; bm = v; break; }
                  cum += v;
                }
              } else {
                // rounding left the target out of reach: keep everything down
                // to the lowest non-empty bin
                for (int j = 255; j >= 0; --j) {
                  const double v = (double)S.tot[r * 256 + j];
                  if (v > 0.0) { dsel = j; bm = v; }
                }
                cum = 0.0;
                for (int j = 255; j > dsel; --j) cum += (double)S.tot[r * 256 + j];
              }
              if (lane == 0) {
                S.misc_i[8 + r] = dsel;
                S.misc_d[4 + 2 * r] = above[r] + cum;
                S.misc_d[5 + 2 * r] = bm;
              }
            }
            consumer_sync<NCT>();
            for (int r = 0; r < nrows; ++r) {
              prefix[r] |= ((uint32_t)S.misc_i[8 + r]) << shift;
              above[r] = S.misc_d[4 + 2 * r];
              kept[r] = above[r] + S.misc_d[5 + 2 * r];
            }
            if (tid == 0)
              for (int r = 0; r < nrows; ++r) S.misc_f[4 + r] = (float)(1.0 / kept[r]);
            consumer_sync<NCT>();
          }
          if (work)
            for (int r = 0; r < nrows; ++r) {
              rp[r].tau_key = prefix[r];
              rp[r].kept = kept[r];
              rp[r].invs = S.misc_f[4 + r];
            }
        }
      }

      // ---- resident: p(x), q(x) from the stored values (the pass-2 formula)
      constexpr int kMode = TOPP ? kPZT : (RESIDENT ? kPE : kPZ);
      const float efill = kMode == kPE ? 0.f : -INFINITY;  // a stored value of zero probability
      if (RESIDENT && !it.bonus && tid == 0 && x >= v0 && x < v0 + len && ok_stats) {
        const int j = x - v0, k = j / kChunk;
        S.misc_d[kMdPx] = (double)prob1<kMode>(S.e[j], kFromE ? S.fac[k] : 0.f, rp[0]);
        S.misc_d[kMdQx] = (double)prob1<kMode>(S.e[(size_t)L.slice + j], kFromE ? S.fac[L.nch + k] : 0.f, rp[1]);
      }

      // ---- pass 2: per-chunk sums of r = max(p - q, 0) (positions) or p (bonus)
      const double u_fin = P.mode == kModeSample ? (double)__ldg(P.uniforms + off + K) : 0.0;
      bool cdf_of_p = it.bonus;
      if constexpr (RESIDENT) {
        for (int k = warp; k < nch; k += NW) {
          float ep[8], pp[8];
          load_e8(S.e, k, lane, len, efill, ep);
          probs8<kMode>(ep, kFromE ? S.fac[k] : 0.f, rp[0], pp);
          float s;
          if (it.bonus) {
            s = sum8(pp);
          } else {
            float eq[8], qq[8], rr[8];
            load_e8(S.e + L.slice, k, lane, len, efill, eq);
            probs8<kMode>(eq, kFromE ? S.fac[L.nch + k] : 0.f, rp[1], qq);
            s = resid8(pp, qq, rr);
          }
          s = warp_sum(s);
          if (lane == 0) S.seg[k] = s;
        }
      } else {
        for (int st = 0; st < nst; ++st) {
          const uint32_t slot = next_full(S, L, seq, timeout);
          const int k = st * NW + warp;
          if (k < nch) {
            const int ib = k * kChunk;
            const T* base = reinterpret_cast<const T*>(S.ring + (size_t)slot * L.slot_bytes) + warp * kChunk;
            float zz[2][8], pp[8];
            stage_chunk2<T>(base, STAGE, nrows, ib, lane, len, S.bitmap, cpen, alpha, zz);
            const float* zp = zz[0];
            float s;
            if (it.bonus) {
              probs8<kMode>(zp, 0.f, rp[0], pp);
              s = sum8(pp);
            } else {
              const float* zq = zz[1];
              float qq[8], rr[8];
              probs8<kMode>(zp, 0.f, rp[0], pp);
              probs8<kMode>(zq, 0.f, rp[1], qq);
              s = resid8(pp, qq, rr);
              // the lane holding x records p(x), q(x)
              const int jx = x - v0 - ib;
              if (ok_stats && jx >= 0 && jx < kChunk) {
                const int owner_lane = jx < 128 ? (jx >> 2) : ((jx - 128) >> 2);
                const int jj = jx < 128 ? (jx & 3) : 4 + ((jx - 128) & 3);
                if (lane == owner_lane) {
                  float px = 0.f, qx = 0.f;
#pragma unroll
                  for (int j = 0; j < 8; ++j)
                    if (j == jj) { px = pp[j]; qx = qq[j]; }
                  S.misc_d[kMdPx] = (double)px;
                  S.misc_d[kMdQx] = (double)qx;
                }
              }
            }
            s = warp_sum(s);
            if (lane == 0) S.seg[k] = s;
          }
          release_slot(S, slot, lane);
        }
      }
      consumer_sync<NCT>();

      // ---- sync 2: CTA totals, cluster prefix, owner of the final draw
      double R = 0.0, Pc = 0.0;
      int owner = -1;
      bool take_last = false;
      for (int attempt = 0; attempt < 2; ++attempt) {
        double Rc = 0.0;
        if (warp == 0) {
          int k0, k1;
          double blk, inc;
          Rc = seg_block_scan(S.seg, nch, lane, k0, k1, blk, inc);
        }
        if (!cluster_exchange(S, ph, C, rank, 1, Rc, 0.0, 0.0, 0.0)) timeout = true;
        if (warp == 0) {
          // lane c: mass of CTA c; prefix sums, total, owner of u_fin * R
          const uint32_t buf = (ph.cph - 1) & 1u;
          const double rc = lane < C ? xchg_slot(S, C, buf, lane)[0] : 0.0;
          const double inc = warp_incl_scan_d(rc, lane);
          const double tot = __shfl_sync(0xffffffffu, inc, 31);
          const double t = u_fin * tot;
          const unsigned hit = __ballot_sync(0xffffffffu, lane < C && rc > 0.0 && inc > t);
          const unsigned pos = __ballot_sync(0xffffffffu, lane < C && rc > 0.0);
          if (lane == 0) {
            S.misc_d[14] = tot;
            S.misc_i[4] = hit ? __ffs(hit) - 1 : (pos ? 31 - __clz(pos) : -1);
            S.misc_i[5] = hit ? 0 : 1;
          }
          if (lane == (int)rank) S.misc_d[15] = inc - rc;
        }
        consumer_sync<NCT>();
        R = S.misc_d[14];
        Pc = S.misc_d[15];
        owner = S.misc_i[4];
        take_last = S.misc_i[5] != 0;
        if (attempt == 0 && !cdf_of_p && !(R > 0.0) && P.mode == kModeSample && ok_stats) {
          // no residual mass (only reachable when q(x) = 0): draw from p; the
          // chunk sums of p come from the resident store or from global memory
          cdf_of_p = true;
          for (int k = warp; k < nch; k += NW) {
            float v[8], pp[8];
            if constexpr (RESIDENT) {
              load_e8(S.e, k, lane, len, efill, v);
            } else {
              global_logits<T>(gp_row, k * kChunk, lane, len, S.bitmap, cpen, alpha, v);
            }
            probs8<kMode>(v, kFromE ? S.fac[k] : 0.f, rp[0], pp);
            const float s = warp_sum(sum8(pp));
            if (lane == 0) S.seg[k] = s;
          }
          consumer_sync<NCT>();
          continue;
        }
        break;
      }

      // ---- decisions
      const double tv = (it.bonus || cdf_of_p) ? 0.0 : fmin(R, 1.0);
      double theta = 1.0;  // fp64 division by one thread only
      if (tid == 0) theta = (tv <= (double)D) ? 1.0 : (double)D / tv;
      const bool x_owner = !it.bonus && x >= v0 && x < v0 + len;
      double pv = 0.0, qv = 0.0;
      if (x_owner && tid == 0) {
        pv = S.misc_d[kMdPx];
        qv = S.misc_d[kMdQx];
        const double pi = (1.0 - theta) * pv + theta * qv;
        const double u = P.mode == kModeSample ? (double)__ldg(P.uniforms + off + it.i) : 0.0;
        if (P.results) {
          ItemResult* res = P.results + item;
          res->acc = (u * qv < pi) ? 1 : 0;
          res->px = (float)pv;
          res->qx = (float)qv;
        }
      }
      if (!it.bonus && tid == 0 && rank == 0 && P.results) {
        P.results[item].tv = (float)tv;
        P.results[item].theta = (float)theta;
      }

      // ---- candidate: inverse CDF at u_fin within the owning CTA: the lane
      // block, then the chunk, then the lane and element that hold it
      if (P.mode == kModeSample && ok_stats && owner == (int)rank && warp == 0) {
        const double tl = u_fin * R - Pc;
        int k0, k1;
        double blk, inc;
        seg_block_scan(S.seg, nch, lane, k0, k1, blk, inc);
        const double exc = inc - blk;
        int ks = -1;
        double rem = 0.0;
        bool tl_last = take_last;
        const unsigned mh = __ballot_sync(0xffffffffu, !take_last && blk > 0.0 && inc > tl);
        if (mh) {
          const int L0 = __ffs(mh) - 1;
          if (lane == L0) {
            double cum = exc;
            int klast = -1;
            for (int k = k0; k < k1; ++k) {
              const double sg = (double)S.seg[k];
              if (sg > 0.0) {
                if (cum + sg > tl) { ks = k; rem = tl - cum; break; }
                klast = k;
              }
              cum += sg;
            }
            if (ks < 0) ks = klast;  // rounding: the block's last chunk with mass
          }
          ks = __shfl_sync(0xffffffffu, ks, L0);
          rem = __shfl_sync(0xffffffffu, rem, L0);
          tl_last = false;
          if (ks >= 0 && rem <= 0.0 && (double)S.seg[ks] <= 0.0) tl_last = true;
        }
        if (ks < 0) {
          // the last chunk with mass
          const unsigned mp = __ballot_sync(0xffffffffu, blk > 0.0);
          if (mp) {
            const int L1 = 31 - __clz(mp);
            int kl = -1;
            if (lane == L1)
              for (int k = k1 - 1; k >= k0; --k)
                if (S.seg[k] > 0.f) { kl = k; break; }
            ks = __shfl_sync(0xffffffffu, kl, L1);
          }
          tl_last = true;
        }
        int found = -1;
        if (ks >= 0) {
          float w[8];
          const int ib = ks * kChunk;
          {
            float vp[8], pp[8], vq[8];
            if constexpr (RESIDENT) {
              load_e8(S.e, ks, lane, len, efill, vp);
              if (!cdf_of_p) load_e8(S.e + L.slice, ks, lane, len, efill, vq);
            } else {
              T rawp[8], rawq[8];
              global_raw<T>(gp_row, ib, lane, len, rawp);
              if (!cdf_of_p) global_raw<T>(gq_row, ib, lane, len, rawq);
              convert_raw<T>(rawp, ib, lane, len, S.bitmap, cpen, alpha, vp);
              if (!cdf_of_p) convert_raw<T>(rawq, ib, lane, len, S.bitmap, cpen, alpha, vq);
            }
            probs8<kMode>(vp, kFromE ? S.fac[ks] : 0.f, rp[0], pp);
            if (cdf_of_p) {
#pragma unroll
              for (int j = 0; j < 8; ++j) w[j] = pp[j];
            } else {
              float qq[8];
              probs8<kMode>(vq, kFromE ? S.fac[L.nch + ks] : 0.f, rp[1], qq);
              resid8(pp, qq, w);
            }
          }
          if (!tl_last) {
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
                    if (wh[j] > 0.f && cum > rem) { jj = j; break; }
                  }
                  if (jj < 0)
                    for (int j = 3; j >= 0; --j)
                      if (wh[j] > 0.f) { jj = j; break; }
                }
                jj = __shfl_sync(0xffffffffu, jj, L0);
                found = ib + 128 * half + 4 * L0 + jj;
              } else {
                rem -= (double)__shfl_sync(0xffffffffu, incl, 31);
              }
            }
          }
          if (found < 0) {
            // the last element with positive mass in the chunk
            for (int half = 1; half >= 0 && found < 0; --half) {
              int lj = -1;
              for (int j = 3; j >= 0; --j)
                if (w[4 * half + j] > 0.f) { lj = j; break; }
              const unsigned m = __ballot_sync(0xffffffffu, lj >= 0);
              if (m) {
                const int L0 = 31 - __clz(m);
                lj = __shfl_sync(0xffffffffu, lj, L0);
                found = ib + 128 * half + 4 * L0 + lj;
              }
            }
          }
        }
        if (lane == 0) P.results[item].cand = found >= 0 ? v0 + found : -1;
      }

      // ---- status of this CTA's share of the item; arrival count
      if (timeout) flags |= kStatusTimeout;
      flags = warp_or(flags);
      if (lane == 0 && flags) atomicOr(&S.misc_i[kMiFlags], flags);
      __threadfence();
      consumer_sync<NCT>();
      if (P.mode == kModeTvOnly && tid == 0) {
        // every CTA checks the same scalars, tokens and row statistics, so its
        // flags are the request's
        const bool bad = S.misc_i[kMiFlags] != 0;
        if (rank == 0) {
          P.out_tv[item] = bad ? NAN : (float)tv;
          if (P.out_theta) P.out_theta[item] = bad ? NAN : (float)theta;
        }
        if (x_owner) {
          if (P.out_px) P.out_px[item] = bad ? NAN : (float)pv;
          if (P.out_qx) P.out_qx[item] = bad ? NAN : (float)qv;
        } else if (rank == 0 && !(x >= 0 && x < P.V)) {
          if (P.out_px) P.out_px[item] = NAN;
          if (P.out_qx) P.out_qx[item] = NAN;
        }
      }
      if (P.mode == kModeSample) {
        if (tid == 0) {
          P.inval[(size_t)item * kMaxCluster + rank] = S.misc_i[kMiFlags];
          __threadfence();
          const int target = C * (K + 1);
          const int old = tagged_arrive(P.counters + b, P.tag);
          S.misc_i[kMiFinalize] = (old == target - 1) && K >= 0 && it.rows_ok;
        }
        consumer_sync<NCT>();
        if (S.misc_i[kMiFinalize] && warp == 0) {
          __threadfence();
          int st = 0;
          for (int j = lane; j < (K + 1) * C; j += 32) {
            const int ii = j / C, cc = j % C;
            const int item_j = ii < K ? d0 + ii : P.total + b;
            st |= __ldcg(P.inval + (size_t)item_j * kMaxCluster + cc);
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
      consumer_sync<NCT>();
    }
  }
  // no CTA may leave while others can still read its shared memory
  cluster_sync_all();
}

namespace {

template <typename T, bool TOPP, bool RESIDENT>
int launch_t(SampleParams& P, cudaStream_t stream) {
  auto kern = sample_verify_kernel<T, TOPP, RESIDENT>;
  const int smem = P.L.total;
  if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, smem) != cudaSuccess) {
    cudaGetLastError();
    return -8;
  }
  if (P.C > 8 && cudaFuncSetAttribute(kern, cudaFuncAttributeNonPortableClusterSizeAllowed, 1) != cudaSuccess) {
    cudaGetLastError();
    return -8;
  }
  cudaLaunchConfig_t cfg = {};
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = P.C;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cfg.blockDim = dim3(((RESIDENT ? kResidentWarps : kStreamWarps) + 1) * 32);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = stream;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  // clusters resident at once (cached per device and configuration)
  static thread_local int cached_dev = -1, cached_C = 0, cached_smem = 0, cached_n = 0;
  int dev = 0;
  cudaGetDevice(&dev);
  if (dev != cached_dev || cached_C != P.C || cached_smem != smem) {
    cfg.gridDim = dim3(P.C);
    int n = 0;
    if (cudaOccupancyMaxActiveClusters(&n, kern, &cfg) != cudaSuccess || n <= 0) {
      cudaGetLastError();
      return -8;
    }
    cached_dev = dev; cached_C = P.C; cached_smem = smem; cached_n = n;
  }
  P.n_clusters = P.n_items < cached_n ? P.n_items : cached_n;
  if (P.n_clusters <= 0) return 0;
  cfg.gridDim = dim3(P.n_clusters * P.C);
  if (cudaLaunchKernelEx(&cfg, kern, P) != cudaSuccess) {
    cudaGetLastError();
    return -7;
  }
  return 0;
}

}  // namespace

// Resident layout: the smallest cluster (1..16) whose slice fits.
int choose_resident_layout(int V, int elem_bytes, bool topp, int max_smem, int* C_out, SmemLayout* L_out) {
  for (int C = 1; C <= kMaxCluster; C *= 2) {
    const SmemLayout L = make_resident_layout(V, C, elem_bytes, topp);
    if (L.total <= max_smem) {
      *C_out = C;
      *L_out = L;
      return 0;
    }
  }
  return -1;
}

// Streaming layout for cluster size C (-1 if it does not fit).
int choose_stream_layout(int V, int C, int elem_bytes, bool topp, int max_smem, int smem_per_sm,
                         SmemLayout* L_out) {
  const SmemLayout L = make_stream_layout(V, C, elem_bytes, topp, max_smem, smem_per_sm);
  if (L.total <= 0) return -1;
  *L_out = L;
  return 0;
}

int launch_sample_verify(SampleParams& P, bool bf16, bool topp, cudaStream_t stream) {
  const bool res = P.L.resident != 0;
  if (bf16) {
    if (topp) return res ? launch_t<__nv_bfloat16, true, true>(P, stream) : launch_t<__nv_bfloat16, true, false>(P, stream);
    return res ? launch_t<__nv_bfloat16, false, true>(P, stream) : launch_t<__nv_bfloat16, false, false>(P, stream);
  }
  if (topp) return res ? launch_t<float, true, true>(P, stream) : launch_t<float, true, false>(P, stream);
  return res ? launch_t<float, false, true>(P, stream) : launch_t<float, false, false>(P, stream);
}

}  // namespace sv
