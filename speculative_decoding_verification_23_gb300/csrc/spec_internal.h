// Internal parameter blocks and workspace layout shared by the entry points
// (spec_verify.cu) and the kernels.  Host and device code.
#pragma once

#include <cstddef>
#include <cstdint>

#include <vector_types.h>

namespace sv {

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
  L.off_bar = off;     off += (2 * slots_a + 2 * slots_b + 5 * kPipeBufs) * 8;
  L.total = align_up_i(off, 128);
  return L;
}


// ---------------------------------------- dataflow streaming sampling kernel
// Each pass over a work item's rows is cut into tasks of one vocabulary
// chunk; every CTA (one per SM) takes tasks from one global counter, so the
// whole GPU works on a few items at a time.  Pass-2 tasks of an item are
// placed `lag_items` items behind its pass-1 tasks, so its rows are still in
// L2 when they are read again.
constexpr int kFlowConsumers = 16;      // streaming warps per CTA, in groups of kFlowUnits
constexpr int kFlowUnits = 8;           // warps (units) per task; groups take alternate slots
constexpr int kFlowSlots = 4;           // ring slots, one task each
constexpr int kFlowSlotBytes = 51200;   // two rows of one chunk
constexpr int kFlowLagRings = 5;        // pass-2 lag, in GPU-wide rings of tasks

// Per ring slot: the task and everything its consumers need.
struct FlowHdr {
  int task;       // index in the task sequence, -1 = no more tasks
  int type;       // 1 = pass 1, 2 = pass 2
  int item, chunk;
  int lo_line;    // first 256-token line of the chunk
  int nlines;     // lines in the chunk
  int nrows;      // 2 (draft position) or 1 (bonus row)
  int pen;        // the repetition penalty applies (slot bitmap holds the set)
  int x;          // draft token (-1 for a bonus row)
  float c;        // log2(e) / T
  float alpha;    // repetition penalty
  float Mt, it, Md, id;  // pass 2: per row reference and 1 / sum
  int pad[3];
};

struct FlowLayout {
  int lpc;         // lines (256 tokens) per chunk
  int nlines;      // lines per row
  int nck;         // chunks per row
  int nu;          // units per row (nck * kFlowUnits): one consumer warp's lines of a chunk
  int row_bytes;   // one row of a slot
  int slot_bytes;  // two rows
  int bm_words;    // penalty bitmap words per slot (lpc * 8)
  int lag_items;   // pass-2 lag in items
  int off_ring, off_bm, off_hdr, off_cu, off_tw, off_bar;
  int total;
};

inline FlowLayout make_flow_layout(int V, int elem_bytes) {
  FlowLayout L{};
  const int maxl = kFlowSlotBytes / (2 * 256 * elem_bytes);
  L.nlines = (V + 255) / 256;
  L.nck = (L.nlines + maxl - 1) / maxl;
  L.lpc = (L.nlines + L.nck - 1) / L.nck;
  L.nu = L.nck * kFlowUnits;
  L.row_bytes = L.lpc * 256 * elem_bytes;
  L.slot_bytes = 2 * L.row_bytes;
  L.bm_words = L.lpc * 8;
  int off = 0;
  L.off_ring = off;  off += kFlowSlots * L.slot_bytes;
  L.off_bm = off;    off += kFlowSlots * L.bm_words * 4;
  L.off_hdr = off;   off += kFlowSlots * (int)sizeof(FlowHdr);
  L.off_cu = off;    off += 1024 * 4;                                  // cu_draft copy (B + 1 <= 1024)
  L.off_tw = off;    off += align_up_i(L.nu * 4, 16);                  // tail warp's unit masses
  L.off_bar = off;   off += 3 * kFlowSlots * 8;
  L.total = align_up_i(off, 128);
  return L;
}

// Global workspace of the dataflow kernel (part of the caller's workspace).
struct FlowWs {
  uint32_t* hbm;      // [B][hbm_words] history bitmaps
  int hbm_words;
  int* rflags;        // [B] status bits of the history tokens
  int* zero;          // start of the region cleared before each launch:
  int zero_words;     //   req[B], cnt[2][n_items], ctl[8]
  int* req;           // [B] decided items per request
  int* cnt;           // [2][n_items] finished pass-1 / pass-2 tasks per item
  int* ctl;           // [0] next task, [1] error bits, [2] CTAs done
  float4* p1;         // [n_items][nu] pass-1 (reference, sum) per unit: target, draft
  float* p2;          // [n_items][nu] pass-2 residual mass per unit
  float2* xz;         // [n_items] raw logits of the draft token (target, draft)
};

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
  int* counters;         // [B]
  ItemResult* results;   // [total + B]
  int* inval;            // [(total + B) * kMaxCluster]
  // geometry
  int C;
  int n_items;
  int n_clusters;
  SmemLayout L;
  PipeLayout PL;   // pipelined streaming kernel only
  FlowLayout FL;   // dataflow kernel only
  FlowWs F;        // dataflow kernel only
  int n_p2;        // items with a pass 2 (draft positions)
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
  int* counters;         // [B]
  GreedyPartial* partials;  // [(total + B) * nck]
};

// ------------------------------------------------------ draft confidence
struct ConfPartial {
  float m;    // chunk maximum of the penalised logits
  float s;    // sum over the chunk of 2^((z' - m) c)
  int flags;
  int pad;
};

struct ConfParams {
  const void* draft;
  long long ld_d;
  const int* cu_draft;
  const int* draft_tokens;
  const int* cu_hist;
  const int* hist;
  const float* temperature;
  const float* rep_penalty;
  int B, V, total, max_k;
  int nck;                 // chunks per row
  float threshold;
  float* out_conf;         // [total]
  int* out_k_eff;          // [B]
  int* out_status;         // [B] or null
  int* counters;           // [B]
  ConfPartial* partials;   // [total * nck]
};

// -------------------------------------------------------------- workspace
struct WorkspaceLayout {
  size_t off_counters, off_results, off_inval, off_partials;
  size_t off_hbm, off_rflags, off_zero, off_p1, off_p2, off_xz;  // dataflow kernel
  int hbm_words, nu, zero_words;
  size_t total;
};

inline size_t align_up_z(size_t x, size_t a) { return (x + a - 1) / a * a; }

inline WorkspaceLayout make_workspace_layout(int B, int total, int V) {
  WorkspaceLayout W{};
  size_t items = (size_t)total + (size_t)B;
  size_t nck = ((size_t)V + kGreedyChunk - 1) / kGreedyChunk;
  W.off_counters = 0;
  size_t off = align_up_z((size_t)B * 4, 256);
  W.off_results = off;
  off = align_up_z(off + items * sizeof(ItemResult), 256);
  W.off_inval = off;
  off = align_up_z(off + items * kMaxCluster * 4, 256);
  W.off_partials = off;
  off = align_up_z(off + items * nck * sizeof(GreedyPartial), 256);
  // dataflow kernel: units per row of the finer (fp32) chunking covers both dtypes
  const FlowLayout f4 = make_flow_layout(V, 4), f2 = make_flow_layout(V, 2);
  W.nu = f4.nu > f2.nu ? f4.nu : f2.nu;
  W.hbm_words = align_up_i((V + 31) / 32, 8);
  W.off_hbm = off;
  off = align_up_z(off + (size_t)B * W.hbm_words * 4, 256);
  W.off_rflags = off;
  off = align_up_z(off + (size_t)B * 4, 256);
  W.off_zero = off;
  const size_t zw = (size_t)B + 2 * items + 8;
  W.zero_words = (int)zw;
  off = align_up_z(off + zw * 4, 256);
  W.off_p1 = off;
  off = align_up_z(off + items * W.nu * 16, 256);
  W.off_p2 = off;
  off = align_up_z(off + items * W.nu * 4, 256);
  W.off_xz = off;
  off = align_up_z(off + items * 8, 256);
  W.total = off;
  return W;
}

}  // namespace sv
