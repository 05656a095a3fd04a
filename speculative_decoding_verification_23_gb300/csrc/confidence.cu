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
//
// Batches with at least one draft row per SM take the pipelined kernel
// instead (conf_pipe_kernel below): one CTA per SM streams whole rows
// through a TMA ring, so that the loads never wait on a CTA's serial steps.
#include "common.cuh"
#include "spec_internal.h"
#include "conf_internal.h"
#include "stream_common.cuh"

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
    const int old = tagged_arrive(P.counters + b, P.tag);
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

// ------------------------------------------------------------- pipelined
// One CTA per SM; draft row k of CTA c is row c + k * gridDim.x.  Warps:
//   streaming warps (kConfWarps): stage st of a row is segments
//       st * kConfWarps + w (2 KB each) in one ring slot; warp w keeps per
//       lane a running reference, the sum of 2^(z'c - ref) and the largest
//       z' (z' the penalised logit, c = log2(e)/T);
//   setup warp: the penalty bitmap of row k+1 (all compute warps build
//       row 0's together at the start), then row k's combine:
//       conf = 2^(max z' * c - M) / S with M the largest reference and S
//       the sum relative to it, the row's status bits, and the request's
//       k_eff once its last row is done (an atomic counter per request);
//   producer warp: lane 0 issues one bulk copy per stage (evict_first:
//       every logit is read once).
// The penalised positions leave the stream as in the sampling kernels: the
// lanes holding their bitmap words add their exact terms and overwrite them
// with -inf before the hot loop reads the segment.

namespace {

constexpr int kCW = kConfWarps;
constexpr int kConfThreads = (kCW + 2) * 32;

extern __shared__ __align__(128) unsigned char conf_smem[];

struct CSmem {
  const ConfLayout& L;
  __device__ __forceinline__ explicit CSmem(const ConfLayout& l) : L(l) {}
  __device__ __forceinline__ unsigned char* at(int off) const { return conf_smem + off; }
  __device__ __forceinline__ unsigned char* ring() const { return at(L.off_ring); }
  __device__ __forceinline__ uint32_t* bm(int kb) const {
    return reinterpret_cast<uint32_t*>(at(L.off_bm + kb * align_up_i(L.bm_words * 4, 16)));
  }
  __device__ __forceinline__ ConfStats* stats(int kb) const {
    return reinterpret_cast<ConfStats*>(at(L.off_stats + kb * align_up_i((int)sizeof(ConfStats), 16)));
  }
  __device__ __forceinline__ int* cu() const { return reinterpret_cast<int*>(at(L.off_cu)); }
  __device__ __forceinline__ uint64_t* bars() const { return reinterpret_cast<uint64_t*>(at(L.off_bar)); }
  __device__ __forceinline__ uint64_t* full() const { return bars(); }
  __device__ __forceinline__ uint64_t* empty() const { return bars() + L.slots; }
  // [kConfBufs] each: setup warp -> streaming warps: the row's bitmap is
  // built; streaming warps -> setup warp: the row is streamed
  __device__ __forceinline__ uint64_t* bm_ready() const { return bars() + 2 * L.slots; }
  __device__ __forceinline__ uint64_t* row_done() const { return bm_ready() + kConfBufs; }
};

__device__ __forceinline__ const int* conf_cu(const ConfParams& P, const CSmem& S) {
  return S.L.cu_ints ? S.cu() : P.cu_draft;
}

// Rows of this CTA.
__device__ __forceinline__ int conf_n_local(const ConfParams& P) {
  return (int)blockIdx.x < P.total ? (P.total - (int)blockIdx.x + (int)gridDim.x - 1) / (int)gridDim.x : 0;
}

// Draft row d: its request, position and scalars.
struct CRow {
  int b, d0, K, i, h0, h1, flags;
  float c, alpha;
  bool valid;  // the request's draft count is valid and d is one of its rows
  bool pen;    // the repetition penalty applies to the row
};

__device__ __forceinline__ CRow conf_row(const ConfParams& P, const int* cu, int d) {
  CRow r;
  int lo = 0, hi = P.B;  // the largest b with cu_draft[b] <= d
  while (hi - lo > 1) {
    const int mid = (lo + hi) >> 1;
    if (cu[mid] <= d) lo = mid;
    else hi = mid;
  }
  r.b = lo;
  r.d0 = cu[lo];
  r.K = cu[lo + 1] - r.d0;
  r.i = d - r.d0;
  r.valid = r.K >= 0 && r.K <= P.max_k && r.K <= kMaxK && r.i >= 0 && r.i < r.K;
  r.flags = conf_params(P, r.b, r.c, r.alpha) | (r.valid ? 0 : kStatusBadK);
  r.h0 = P.cu_hist ? __ldg(P.cu_hist + r.b) : 0;
  r.h1 = P.cu_hist ? __ldg(P.cu_hist + r.b + 1) : 0;
  r.pen = !(r.flags & kStatusBadParam) && r.alpha != 1.f && (r.h1 > r.h0 || (r.valid && r.i > 0));
  return r;
}

// Row d's penalty set (history plus the drafts before the row) into bm when
// the penalty applies; reports out-of-range tokens of the history and the
// row's own draft token (the request's rows together cover all its drafts).
// Thread t of nt.
__device__ __forceinline__ int conf_mark(const ConfParams& P, const CRow& r, int d, uint32_t* bm, int t, int nt) {
  int flags = 0;
  // eight loads in flight per thread before their bits are set
  for (int j0 = r.h0 + t; j0 < r.h1; j0 += 8 * nt) {
    int tok[8];
#pragma unroll
    for (int q = 0; q < 8; ++q) tok[q] = j0 + nt * q < r.h1 ? __ldg(P.hist + j0 + nt * q) : 0;
#pragma unroll
    for (int q = 0; q < 8; ++q) {
      if (j0 + nt * q >= r.h1) continue;
      if (tok[q] < 0 || tok[q] >= P.V) flags |= kStatusBadToken;
      else if (r.pen) atomicOr(&bm[tok[q] >> 5], 1u << (tok[q] & 31));
    }
  }
  const int npre = r.valid ? r.i : 0;
  for (int j = t; j < npre; j += nt) {
    const int tk = __ldg(P.draft_tokens + r.d0 + j);
    if (r.pen && tk >= 0 && tk < P.V) atomicOr(&bm[tk >> 5], 1u << (tk & 31));
  }
  if (t == 0) {
    const int x = __ldg(P.draft_tokens + d);
    if (x < 0 || x >= P.V) flags |= kStatusBadToken;
  }
  return flags;
}

// One staged 2 KB segment for one lane: the largest value and the pass-1
// statistics (reference, sum of 2^(z'c - ref)).
template <typename T>
__device__ __forceinline__ void seg_stats_max(const unsigned char* seg, int lane, int nvalid, float c, float& ref,
                                              float& run, float& zmax) {
  constexpr int N = Vec<T>::N;
  uint4 v[4];
  lds_seg(seg, lane, v);
  float z[4][N];
#pragma unroll
  for (int j = 0; j < 4; ++j) cvt16(v[j], z[j]);
  if (nvalid < 128 * N) mask_tail<N>(z, lane, nvalid);
  float m0 = zmax, m1 = -INFINITY;
#pragma unroll
  for (int j = 0; j < 4; ++j)
#pragma unroll
    for (int e = 0; e < N; e += 2) {
      m0 = fmaxf(m0, z[j][e]);
      m1 = fmaxf(m1, z[j][e + 1]);
    }
  zmax = fmaxf(m0, m1);
  stats_row<N>(z, c, ref, run);
}

template <typename T>
__device__ __forceinline__ void conf_stream(const ConfParams& P, const CSmem& S, int w, int lane) {
  const ConfLayout& L = S.L;
  const int SEG = L.seg, wps = SEG / 32;
  const int n_local = conf_n_local(P);
  RingCursor rc;
  bool to = false;
  for (int k = 0; k < n_local; ++k) {
    const int kb = k % kConfBufs;
    if (!to && !mbar_wait(&S.bm_ready()[kb], (uint32_t)(k / kConfBufs) & 1u)) to = true;
    ConfStats& st = *S.stats(kb);
    const bool pen = st.pen != 0;
    const float c = st.c, alpha = st.alpha;
    float ref = -INFINITY, run = 0.f, pref = -INFINITY, psum = 0.f, zmax = -INFINITY;
    int pflags = 0;
    for (int stn = 0; stn < L.nst; ++stn) {
      const uint32_t slot = rc.slot;
      if (!to && !mbar_wait(&S.full()[slot], rc.phase)) to = true;
      rc.advance(L.slots);
      const int s_id = stn * kCW + w;
      if (s_id < L.nseg) {
        unsigned char* seg = S.ring() + (size_t)slot * L.slot_bytes + w * 2048;
        if (pen) {
          // penalised positions: their exact terms, then out of the stream
          bool wrote = false;
          const bool any = for_penalised(S.bm(kb), s_id, wps, lane, [&](int o) {
            T* pp = reinterpret_cast<T*>(seg) + o;
            const float z = to_f32<T>(*pp);
            if (is_bad_logit(z)) pflags |= kStatusBadLogits;
            const float zp = penalize(z, alpha);
            zmax = fmaxf(zmax, zp);
            online_add(zp * c, pref, psum);
            *pp = neg_inf<T>();
            wrote = true;
          });
          if (any) {
            if (wrote) fence_proxy_async_smem();
            __syncwarp();
          }
        }
        seg_stats_max<T>(seg, lane, min(SEG, P.V - s_id * SEG), c, ref, run, zmax);
      }
      __syncwarp();
      if (lane == 0) mbar_arrive(&S.empty()[slot]);
    }
    combine_into(make_float2(pref, psum), ref, run);
    const float2 wv = warp_combine(ref, run);
    zmax = warp_max(zmax);
    pflags = warp_or(pflags);
    if (lane == 0) {
      st.wp[w] = wv;
      st.zmax[w] = zmax;
      st.wflags[w] = pflags | (to ? kStatusTimeout : 0);
    }
    __syncwarp();
    if (lane == 0) mbar_arrive(&S.row_done()[kb]);
  }
}

template <typename T>
__device__ __forceinline__ void conf_setup(const ConfParams& P, const CSmem& S, int lane) {
  const ConfLayout& L = S.L;
  const int* cu = conf_cu(P, S);
  const int n_local = conf_n_local(P);
  bool to = false;

  auto build = [&](int k) {
    // buffer k % kConfBufs was last used by row k - 2, combined already
    const int d = blockIdx.x + k * gridDim.x;
    const int kb = k % kConfBufs;
    const CRow r = conf_row(P, cu, d);
    uint32_t* bm = S.bm(kb);
    if (r.pen)
      for (int q = lane; q < L.bm_words / 4; q += 32) reinterpret_cast<uint4*>(bm)[q] = make_uint4(0u, 0u, 0u, 0u);
    __syncwarp();
    const int flags = warp_or(r.flags | conf_mark(P, r, d, bm, lane, 32));
    ConfStats& st = *S.stats(kb);
    if (lane == 0) {
      st.flags = flags;
      st.pen = r.pen ? 1 : 0;
      st.c = r.c;
      st.alpha = r.alpha;
    }
    __syncwarp();
    if (lane == 0) mbar_arrive(&S.bm_ready()[kb]);
  };

  auto combine = [&](int k) {
    const int d = blockIdx.x + k * gridDim.x;
    const int kb = k % kConfBufs;
    const CRow r = conf_row(P, cu, d);
    if (!to && !mbar_wait(&S.row_done()[kb], (uint32_t)(k / kConfBufs) & 1u)) to = true;
    const ConfStats& st = *S.stats(kb);
    const float2 v = lane < kCW ? st.wp[lane] : make_float2(-INFINITY, 0.f);
    const float2 t = warp_combine(v.x, v.y);  // (M, S)
    const float zm = warp_max(lane < kCW ? st.zmax[lane] : -INFINITY);
    int flags = st.flags | (to ? kStatusTimeout : 0) | warp_or(lane < kCW ? st.wflags[lane] : 0);
    if (!(t.y > 0.f) || !(t.y < INFINITY) || !(t.x < INFINITY) || !(zm < INFINITY)) flags |= kStatusBadLogits;
    const float conf = flags ? NAN : __fdiv_rn(ex2(fmaf(zm, r.c, -t.x)), t.y);
    int last = 0;
    if (lane == 0 && r.valid) {
      P.out_conf[d] = conf;
      ConfPartial cp;
      cp.m = conf;
      cp.s = 0.f;
      cp.flags = flags;
      cp.pad = 0;
      P.partials[d] = cp;
      __threadfence();
      last = tagged_arrive(P.counters + r.b, P.tag) == r.K - 1;
    }
    if (__shfl_sync(0xffffffffu, last, 0)) {
      // the request's last row: status and the confidence-stopped count
      __threadfence();
      int f = 0;
      float cf = 0.f;
      if (lane < r.K) {
        f = __ldcg(&P.partials[r.d0 + lane].flags);
        cf = __ldcg(&P.partials[r.d0 + lane].m);
      }
      f = warp_or(f);
      const unsigned below = __ballot_sync(0xffffffffu, lane < r.K && cf < P.threshold);
      if (lane == 0) {
        P.out_k_eff[r.b] = f ? -1 : (below ? __ffs(below) : r.K);
        if (P.out_status) P.out_status[r.b] = f;
      }
      if (f && lane < r.K) P.out_conf[r.d0 + lane] = NAN;
    }
  };

  // row 0's set was built by all compute warps
  if (n_local > 0 && lane == 0) mbar_arrive(&S.bm_ready()[0]);
  for (int k = 0; k < n_local; ++k) {
    if (k + 1 < n_local) build(k + 1);
    combine(k);
  }

  // requests without drafts, or with an invalid draft count (their rows
  // wrote nothing)
  for (int b = blockIdx.x; b < P.B; b += gridDim.x) {
    const int d0 = cu[b];
    const int K = cu[b + 1] - d0;
    const bool bad_k = K < 0 || K > P.max_k || K > kMaxK;
    if (K != 0 && !bad_k) continue;
    float c, alpha;
    int flags = conf_params(P, b, c, alpha) | (bad_k ? kStatusBadK : 0);
    if (bad_k)
      for (int r = max(d0, 0) + lane; r < min(d0 + K, P.total); r += 32) P.out_conf[r] = NAN;
    const int h0 = P.cu_hist ? __ldg(P.cu_hist + b) : 0;
    const int h1 = P.cu_hist ? __ldg(P.cu_hist + b + 1) : 0;
    for (int j = h0 + lane; j < h1; j += 32) {
      const int t = __ldg(P.hist + j);
      if (t < 0 || t >= P.V) flags |= kStatusBadToken;
    }
    flags = warp_or(flags);
    if (lane == 0) {
      P.out_k_eff[b] = flags ? -1 : 0;
      if (P.out_status) P.out_status[b] = flags;
    }
  }
}

template <typename T>
__device__ __forceinline__ void conf_producer(const ConfParams& P, const CSmem& S) {
  const ConfLayout& L = S.L;
  constexpr int es = (int)sizeof(T);
  const uint64_t pol = l2_policy_evict_first();
  const int stage = kCW * L.seg;  // tokens per stage
  const int n_local = conf_n_local(P);
  RingCursor rc;
  RingFills fills;
  bool to = false;   // a wait ran out: nothing more is issued (the compute warps' own waits then run out)
  for (int k = 0; k < n_local && !to; ++k) {
    const int d = blockIdx.x + k * gridDim.x;
    const unsigned char* row = static_cast<const unsigned char*>(P.draft) + (size_t)d * P.ld_d * es;
    for (int st = 0; st < L.nst; ++st) {
      const uint32_t slot = rc.slot, phase = rc.phase;
      // first use of a slot: the phase "before" its first completes at once
      if (!mbar_wait(&S.empty()[slot], rc.phase ^ 1u)) {
        to = true;
        break;
      }
      rc.advance(L.slots);
      fills.note(slot, phase);
      // the row's padded stride (a multiple of 16 bytes) covers the rounding
      const int n = min(stage, P.V - st * stage);
      const uint32_t bytes = (uint32_t)((n * es + 15) & ~15);
      mbar_arrive_expect_tx(&S.full()[slot], bytes);
      bulk_g2s(S.ring() + (size_t)slot * L.slot_bytes, row + (size_t)st * stage * es, bytes, &S.full()[slot], pol);
    }
  }
  // after a wait ran out: the copies already started land before the CTA
  // may exit
  if (to) fills.drain(S.full(), L.slots);
}

template <typename T>
__global__ void __launch_bounds__(kConfThreads, 1) conf_pipe_kernel(const __grid_constant__ ConfParams P) {
  const ConfLayout& L = P.CL;
  const CSmem S(L);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31, tid = threadIdx.x;
  if (tid == 0) {
    for (int s = 0; s < L.slots; ++s) {
      mbar_init(&S.full()[s], 1);
      mbar_init(&S.empty()[s], kCW);
    }
    for (int i = 0; i < kConfBufs; ++i) {
      mbar_init(&S.bm_ready()[i], 1);
      mbar_init(&S.row_done()[i], kCW);
    }
    fence_mbar_init();
  }
  for (int i = tid; i < L.cu_ints; i += kConfThreads) S.cu()[i] = __ldg(P.cu_draft + i);
  __syncthreads();
  if (warp <= kCW && conf_n_local(P) > 0) {
    // the first row's penalty set, by all compute warps while the producer
    // fills the ring (the setup warp builds the later ones alone)
    constexpr int nt = (kCW + 1) * 32;
    const CRow r = conf_row(P, conf_cu(P, S), blockIdx.x);
    ConfStats& st = *S.stats(0);
    if (r.pen)
      for (int q = tid; q < L.bm_words / 4; q += nt) reinterpret_cast<uint4*>(S.bm(0))[q] = make_uint4(0u, 0u, 0u, 0u);
    if (tid == 0) {
      st.flags = r.flags;
      st.pen = r.pen ? 1 : 0;
      st.c = r.c;
      st.alpha = r.alpha;
    }
    named_sync(1, nt);
    const int f = warp_or(conf_mark(P, r, blockIdx.x, S.bm(0), tid, nt));
    if (lane == 0 && f) atomicOr(&st.flags, f);
    named_sync(1, nt);
  }
  if (warp < kCW) conf_stream<T>(P, S, warp, lane);
  else if (warp == kCW) conf_setup<T>(P, S, lane);
  else if (lane == 0) conf_producer<T>(P, S);
}

}  // namespace

// Layout of the pipelined kernel (-1 if it does not fit `max_smem`).
int choose_conf_layout(int V, int elem_bytes, int B, int max_smem, ConfLayout* out) {
  for (int slots = kConfSlots; slots >= 2; --slots) {
    const ConfLayout L = make_conf_layout(V, elem_bytes, slots, B);
    if (L.total <= max_smem) {
      *out = L;
      return 0;
    }
  }
  return -1;
}

int launch_conf_pipe(const ConfParams& P, bool bf16, int num_sms, cudaStream_t stream) {
  const int smem = P.CL.total;
  const int grid = P.total < 1 ? 1 : (P.total < num_sms ? P.total : num_sms);
  if (bf16) {
    auto kern = conf_pipe_kernel<__nv_bfloat16>;
    if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, smem) != cudaSuccess) {
      cudaGetLastError();
      return -8;
    }
    kern<<<grid, kConfThreads, smem, stream>>>(P);
  } else {
    auto kern = conf_pipe_kernel<float>;
    if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, smem) != cudaSuccess) {
      cudaGetLastError();
      return -8;
    }
    kern<<<grid, kConfThreads, smem, stream>>>(P);
  }
  return cudaGetLastError() == cudaSuccess ? 0 : -7;
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
