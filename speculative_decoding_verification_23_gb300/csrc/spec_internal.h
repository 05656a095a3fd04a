// Internal parameter blocks and workspace layout shared by the entry points
// (spec_verify.cu) and the kernels.  Host and device code.
#pragma once

#include <cstddef>
#include <cstdint>

#include <vector_types.h>

namespace sv {

// Call-tagged arrival counters (tagged_arrive): bits of a counter word below
// the call's tag, i.e. the most arrivals one call may count.
constexpr int kTagShift = 24;

// ----------------------------------------------------------------- sampling
constexpr int kChunk = 256;                 // tokens per warp-chunk (8 per lane)
// Consumer warps per CTA: the resident variant runs one 16-warp CTA per SM;
// the streaming variant runs two 8-warp CTAs per SM, so that one CTA's
// per-item synchronisation overlaps the other's streaming.  Each CTA also
// has one producer warp.  A ring slot carries kChunk tokens per consumer warp
// of each row.
constexpr int kResidentWarps = 16;
constexpr int kStreamWarps = 16;
constexpr int kMaxConsumerWarps = 16;
constexpr int kResidentRingBytes = 64 * 1024;
constexpr int kStreamRingMaxBytes = 192 * 1024;
constexpr int kStreamCtasPerSm = 1;
constexpr int kXchgDoubles = 8;             // per CTA per exchange buffer
constexpr int kMaxCluster = 16;

enum SampleMode : int { kModeSample = 0, kModeTvOnly = 1 };

struct ItemResult {       // one per work item (a draft position or a bonus row)
  int acc;                // acceptance flag (positions)
  int cand;               // residual candidate (positions) / bonus token
  float tv, theta, px, qx;
  int pad[2];
};

// Shared memory of the sampling kernel.  A ring slot holds one stage: the
// CTA's next `stage` tokens of the target row followed by the same tokens of
// the draft row.  The resident variant also keeps one fp32 value per token
// of its slice of both rows (the e-array); the streaming variant re-reads
// the rows through the ring instead.
struct SmemLayout {
  int slice;      // token ids per CTA (multiple of 64)
  int nch;        // chunks per CTA slice (ceil(slice / 256))
  int nw;         // consumer warps
  int stage;      // tokens of each row per slot (nw * 256)
  int nslots;     // ring slots
  int slot_bytes;
  int resident;
  int off_e, off_bitmap, off_refc, off_fac, off_seg, off_wpart, off_xchg, off_hist, off_tot, off_misc, off_bar;
  int total;
};

__host__ __device__ inline int align_up_i(int x, int a) { return (x + a - 1) / a * a; }

// Everything but the ring and the e-array, from `off` on.
inline int layout_tail(SmemLayout& L, int off, int C, bool topp) {
  L.off_bitmap = off;   off += L.nch * 8 * 4;   // 8 words per 256-token chunk
  L.off_refc = off;     off += L.resident ? align_up_i(2 * L.nch * 4, 16) : 0;
  L.off_fac = off;      off += L.resident ? align_up_i(2 * L.nch * 4, 16) : 0;
  L.off_seg = off;      off += align_up_i(L.nch * 4, 16);
  L.off_wpart = off;    off += 2 * kMaxConsumerWarps * 8;
  L.off_xchg = off;     off += 2 * C * kXchgDoubles * 8;
  L.off_hist = off;     off += topp ? 2 * 2 * 256 * 4 : 0;
  L.off_tot = off;      off += topp ? 2 * 256 * 4 : 0;
  L.off_misc = off;     off += 256;
  L.off_bar = off;      off += (2 * L.nslots + 2) * 8;  // full, empty, csync[2]
  return align_up_i(off, 128);
}

// Resident variant for cluster size C: 64 KB ring + the e-array.
inline SmemLayout make_resident_layout(int V, int C, int elem_bytes, bool topp) {
  SmemLayout L{};
  L.resident = 1;
  L.nw = kResidentWarps;
  L.stage = L.nw * kChunk;
  L.slice = align_up_i((V + C - 1) / C, 64);
  L.nch = (L.slice + kChunk - 1) / kChunk;
  L.slot_bytes = 2 * L.stage * elem_bytes;
  L.nslots = kResidentRingBytes / L.slot_bytes;
  L.off_e = kResidentRingBytes;
  L.total = layout_tail(L, L.off_e + 2 * L.slice * 4, C, topp);
  return L;
}

// Streaming variant: the deepest ring (whole slots, at most 96 KB, at least
// 2 slots) such that two CTAs fit in one SM's `smem_per_sm` and one in
// `max_smem`; total = 0 if none does.
inline SmemLayout make_stream_layout(int V, int C, int elem_bytes, bool topp, int max_smem, int smem_per_sm) {
  SmemLayout L{};
  L.resident = 0;
  L.nw = kStreamWarps;
  L.stage = L.nw * kChunk;
  L.slice = align_up_i((V + C - 1) / C, 64);
  L.nch = (L.slice + kChunk - 1) / kChunk;
  L.slot_bytes = 2 * L.stage * elem_bytes;
  const int budget = smem_per_sm / kStreamCtasPerSm - 1024;  // the driver reserves ~1 KB per CTA
  for (int ns = kStreamRingMaxBytes / L.slot_bytes; ns >= 2; --ns) {
    L.nslots = ns;
    L.off_e = ns * L.slot_bytes;
    L.total = layout_tail(L, L.off_e, C, topp);
    if (L.total <= max_smem && L.total <= budget) return L;
  }
  L.total = 0;
  return L;
}

// ------------------------------------------- pipelined streaming sampling
// One CTA per SM, persistent over its items.  Four warp roles: group A's
// streaming warps compute pass-1 statistics of item k from HBM while group
// B's streaming warps run pass 2 (an L2 re-read) of item k-1; group A's setup
// warp builds the penalty list of item k+1 and combines item k's statistics,
// group B's tail warp takes the decisions and the candidate of item k-2.
// Each streaming group has its own TMA producer warp and ring.
constexpr int kPipeWarpsA = 8;        // group A streaming warps (+ 1 setup warp)
constexpr int kPipeWarpsB = 8;        // group B streaming warps (+ 1 tail warp)
constexpr int kPipeBufs = 3;          // per-item buffers in flight
constexpr int kPipeSegBytes = 2048;   // one row's bytes per warp per stage (64 per lane)
constexpr int kPipeCuCap = 1024;      // cu_draft entries cached in shared memory (B + 1 <= this)
constexpr int kPipeMaxIters = 8192;   // items per CTA (deferred-item bits)
constexpr int kPipeSlotsA = 3;        // ring slots of group A (HBM stream) ...
constexpr int kPipeSlotsB = 2;        // ... and of group B (L2 re-read)

// One item's hand-offs between the roles.
struct PipeStats {
  float2 wp[kPipeWarpsA][2];  // per A streaming warp and row: (reference, sum) of pass 1
  int aflags[kPipeWarpsA];    // status bits seen by each A streaming warp
  float M[2], inv[2];         // per row: reference and 1 / softmax sum (units of z'c)
  float px, qx;               // p(x), q(x) of the draft token
  float xz[2];                // raw logits of the draft token (captured from the ring)
  int flags;                  // status bits of the item
  int pen;                    // the repetition penalty applies (bitmap kb holds the set)
};

struct PipeLayout {
  int seg;              // tokens of a row per warp segment (kPipeSegBytes / elem bytes)
  int nseg;             // segments per row
  int nst_a, nst_b;     // stages per row (group A / group B)
  int slots_a, slots_b;
  int slot_a, slot_b;   // bytes per ring slot
  int bm_words;         // bitmap words (nseg * seg / 32)
  int off_ring_a, off_ring_b, off_bm, off_part, off_segt, off_stats, off_misc,
      off_defer, off_cu, off_bar;
  int total;
};

inline PipeLayout make_pipe_layout(int V, int elem_bytes, int slots_a, int slots_b) {
  PipeLayout L{};
  L.seg = kPipeSegBytes / elem_bytes;
  L.nseg = (V + L.seg - 1) / L.seg;
  L.nst_a = (L.nseg + kPipeWarpsA - 1) / kPipeWarpsA;
  L.nst_b = (L.nseg + kPipeWarpsB - 1) / kPipeWarpsB;
  L.slots_a = slots_a;
  L.slots_b = slots_b;
  L.slot_a = 2 * kPipeWarpsA * kPipeSegBytes;
  L.slot_b = 2 * kPipeWarpsB * kPipeSegBytes;
  L.bm_words = L.nseg * L.seg / 32;
  const int segv = align_up_i(L.nseg * 4, 16);
  int off = 0;
  L.off_ring_a = off;  off += slots_a * L.slot_a;
  L.off_ring_b = off;  off += slots_b * L.slot_b;
  L.off_bm = off;      off += kPipeBufs * align_up_i(L.bm_words * 4, 16);  // one penalty bitmap per item buffer
  L.off_part = off;    off += align_up_i((V + 255) / 256 * 4, 16);  // slow path: 256-token chunk sums
  L.off_segt = off;    off += kPipeBufs * segv;
  L.off_stats = off;   off += kPipeBufs * align_up_i((int)sizeof(PipeStats), 16);
  L.off_misc = off;    off += 1024;
  L.off_defer = off;   off += kPipeMaxIters / 8;
  L.off_cu = off;      off += kPipeCuCap * 4;
  L.off_bar = off;     off += (2 * slots_a + 2 * slots_b + 5 * kPipeBufs + 1) * 8;
  L.total = align_up_i(off, 128);
  return L;
}

struct SampleParams {
  const void* target;
  long long ld_t;
  const void* draft;
  long long ld_d;
  const int* cu_draft;
  const int* draft_tokens;
  const int* cu_hist;
  const int* hist;
  const float* temperature;
  const float* rep_penalty;
  const float* top_p;
  const float* tv_budget;
  const float* uniforms;
  int B, V, total, max_k;
  unsigned flags;
  int mode;
  // outputs
  int* out_tokens;
  int* out_accepted;
  int* out_status;
  float* out_tv;
  float* out_theta;
  float* out_px;
  float* out_qx;
  // workspace
  unsigned long long* counters;   // [B] call-tagged arrivals (tagged_arrive)
  unsigned long long tag;         // this call's tag
  ItemResult* results;   // [total + B]
  int* inval;            // [(total + B) * kMaxCluster]
  // geometry
  int C;
  int n_items;
  int n_clusters;
  SmemLayout L;
  PipeLayout PL;   // pipelined streaming kernel only
};

// ------------------------------------------------------------------- greedy
constexpr int kGreedyThreads = 256;
constexpr int kGreedyChunk = 8192;   // elements per CTA

struct GreedyPartial {
  float val;
  int idx;
  int flags;
  int pad;
};

struct GreedyParams {
  const void* target;
  long long ld_t;
  const int* cu_draft;
  const int* draft_tokens;
  const int* cu_hist;
  const int* hist;
  const float* rep_penalty;
  int B, V, total, max_k;
  int nck;               // chunks per row
  int* out_tokens;
  int* out_accepted;
  int* out_status;
  unsigned long long* counters;   // [B] call-tagged arrivals (tagged_arrive)
  unsigned long long tag;         // this call's tag
  GreedyPartial* partials;  // [(total + B) * nck]
};

// -------------------------------------------------------------- workspace
struct WorkspaceLayout {
  size_t off_counters, off_results, off_inval, off_partials, total;
};

inline size_t align_up_z(size_t x, size_t a) { return (x + a - 1) / a * a; }

inline WorkspaceLayout make_workspace_layout(int B, int total, int V) {
  WorkspaceLayout W{};
  size_t items = (size_t)total + (size_t)B;
  size_t nck = ((size_t)V + kGreedyChunk - 1) / kGreedyChunk;
  W.off_counters = 0;
  size_t off = align_up_z((size_t)B * 8, 256);
  W.off_results = off;
  off = align_up_z(off + items * sizeof(ItemResult), 256);
  W.off_inval = off;
  off = align_up_z(off + items * kMaxCluster * 4, 256);
  W.off_partials = off;
  off = align_up_z(off + items * nck * sizeof(GreedyPartial), 256);
  W.total = off;
  return W;
}

}  // namespace sv
