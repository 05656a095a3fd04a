// Split-vocabulary sampling kernel (seg_verify.cu): parameter block, record
// types and layouts shared by the host code and the kernel.
//
// Work is cut into units of one vocabulary segment of one logit row (pass 1)
// or half a segment of a target/draft row pair (pass 2).  Units are spread
// over one persistent CTA per SM; every record below lives in the caller's
// workspace (or the fixed scratch of spec_verify_sample_static).
#pragma once

#include <cstddef>
#include <cstdint>

namespace sv {

constexpr int kSegGroupWarps = 8;                  // consumer warps per group (one unit at a time)
constexpr int kSegGroups = 3;                      // unit k goes to group k % kSegGroups
constexpr int kSegConsumers = kSegGroups * kSegGroupWarps;
constexpr int kSegCtlWarps = 4;                    // producer, recorder, decider and finisher warps
constexpr int kSegThreads = (kSegConsumers + kSegCtlWarps) * 32;
constexpr int kSegSlots = 6;                       // TMA ring slots
static_assert(kSegSlots % kSegGroups == 0, "slot k % kSegSlots belongs to group k % kSegGroups");
constexpr int kSegLogitBytes = 30720;              // logit bytes per slot (one segment of one row)
constexpr int kSegBmBytes = kSegLogitBytes / 2 / 8;  // penalty bits of a bf16 segment
constexpr int kSegDescOff = kSegLogitBytes + kSegBmBytes;
constexpr int kSegMaxExtras = 32;
constexpr int kSegRecN = 64;                       // unit records between producer and finisher
constexpr int kSegCuCap = 1024;                    // cu_draft entries cached in shared memory
constexpr int kSegMaxSegs = 32;                    // segments per row (a draw scans <= 16 * kSegMaxSegs parts)

// Unit kinds in a slot header.
enum : int { kUnitStop = 0, kUnitRow = 1, kUnitPair = 2 };

// One per logit row, written by the kernel's prologue.  Rows are numbered
// request by request (request b's rows start at 2 cu_draft[b] + b): target
// row i at 2i, draft row i at 2i + 1, the bonus row (target row K_b) last.
// The penalty set of a row is its request's history (a bitmap per request)
// plus `extras`: the drafts before the row that are not in the history,
// each once.
struct SegRowDesc {
  int b;          // request
  int i;          // position within the request (K_b for the bonus row)
  int kind;       // 0 target row, 1 draft row
  int x;          // the row's draft token x_i (-1 for a bonus row)
  int x_pen;      // x_i is in the row's penalty set
  int n_extra;
  float c;        // log2(e) / T
  float alpha;    // repetition penalty (1 = none)
  int src;        // the logits: target row src (< total + B) or draft row src - (total + B)
  int pad[3];
  int extras[kSegMaxExtras];
};
static_assert(sizeof(SegRowDesc) == 176, "row descriptor size");

// Per position that needs the second pass: the rows' log2 normalisers as
// fp32 values and factors, p(v) = 2^(z'(v) c - Lp) fp and
// q(v) = 2^(z'(v) c - Lq) fq (the factors carry what rounding the
// normalisers to fp32 dropped).
struct SegJobDesc {
  float Lp, Lq;
  float fp, fq;
};
static_assert(sizeof(SegJobDesc) == 16, "job descriptor size");

// Per row after pass 1: softmax statistics (S relative to the reference M,
// both in units of z'c) and the probability of the row's draft token.
struct SegRowStat {
  float M, S, px;
  int flags;
};

// Per position.
struct SegPos {
  int state;      // 0 certain reject, 1 certain accept, 2 undecided (from pass 1)
  float px, qx;
  int acc;        // the decision after the second pass
  float d, theta; // TV and theta after the second pass
  int b, pad;
};

// Slot header written by the producer (generic stores) before it arrives on
// the slot's full barrier.
struct SegUnitHdr {
  int kind;
  int id;         // pass 1: unit index u (row = u / nseg); pass 2: position p
  int part;       // pass 2: half-segment index h (segment h / 2, half h % 2)
  int tok0;       // first token of the unit
  int n;          // tokens in the unit
  int pad[3];
};

// Per unit in flight (a ring of kSegRecN in shared memory): what the
// producer issued, and the consumers' results, which the finisher stores.
struct SegUnitRec {
  int kind, id, part, has_zx;
  float zx;
  unsigned ndone;             // consumer warps done with the unit
  int pad[2];
  float2 r[kSegGroupWarps];   // pass 1: (reference, sum) per warp; pass 2: .x = residual mass per warp
};

constexpr int kSegHdrOff = kSegDescOff + (int)sizeof(SegRowDesc) + (int)sizeof(SegJobDesc);
constexpr int kSegSlotBytes = ((kSegHdrOff + (int)sizeof(SegUnitHdr)) + 127) / 128 * 128;

// Control words at the start of the zeroed region.
enum : int {
  kCtlPrepDone = 0,  // CTAs done with the prologue
  kCtlBroken,        // cu_draft is not a valid packing: every request is invalid
  kCtlJobTail,       // jobs reserved
  kCtlClaim,         // second-pass units claimed
  kCtlDecided,       // requests decided after pass 1
  kCtlExited,        // CTAs finished
  kCtlAbort,         // a bounded wait ran out somewhere
  kCtlSteal,         // pass-1 units past the dealt ones claimed
  kCtlWords = 16
};

// Vocabulary segmentation for a row of V tokens with `es`-byte logits.
struct SegGeom {
  int seg;        // tokens per segment (multiple of 512)
  int nseg;       // segments per row
  int wr;         // tokens per consumer warp in pass 1 (seg / 8)
  int wr2;        // tokens per consumer warp in pass 2 (seg / 16)
  int upj;        // pass-2 units per position (2 * nseg)
  int bm_bytes;   // penalty bitmap bytes per request (nseg * seg / 8)
};

__host__ __device__ inline SegGeom make_seg_geom(int V, int es) {
  SegGeom g{};
  const int max_tok = kSegLogitBytes / es;       // 15360 bf16, 7680 fp32 (multiples of 512)
  g.nseg = (V + max_tok - 1) / max_tok;
  if (g.nseg < 1) g.nseg = 1;
  const int per = (V + g.nseg - 1) / g.nseg;
  g.seg = (per + 511) / 512 * 512;     // pass-2 warp ranges stay multiples of 32 tokens
  g.wr = g.seg / kSegGroupWarps;
  g.wr2 = g.seg / (2 * kSegGroupWarps);
  g.upj = 2 * g.nseg;
  g.bm_bytes = g.nseg * g.seg / 8;
  return g;
}

// Workspace regions of the kernel (offsets in bytes, 256-byte aligned).
struct SegWorkspace {
  size_t off_zero, zero_bytes;    // counters the kernel clears at its start (from off_jobs)
  size_t off_ctl, off_row_cnt, off_req_rows, off_req_pend, off_job_cnt, off_jobs, off_req_done;
  size_t off_bitmap, off_rowdesc, off_part1, off_rowstat, off_zx, off_pos, off_part2, off_jobdesc, off_req_status,
      off_req_need, off_posdesc;
  size_t total;
};

inline size_t seg_align(size_t x) { return (x + 255) / 256 * 256; }

inline SegWorkspace make_seg_workspace(int B, int total, int V, int es) {
  const SegGeom g = make_seg_geom(V, es);
  const size_t NR = 2 * (size_t)total + (size_t)B;
  SegWorkspace w{};
  size_t off = 0;
  w.off_zero = off;
  w.off_ctl = off;        off += kCtlWords * 4;
  w.off_jobs = off;       off += (size_t)total * 8;     // 64-bit entries: 8-byte aligned (ctl is 64 bytes)
  w.off_row_cnt = off;    off += NR * 4;
  w.off_req_rows = off;   off += (size_t)B * 4;
  w.off_req_pend = off;   off += (size_t)B * 4;
  w.off_req_done = off;   off += (size_t)B * 4;
  w.off_job_cnt = off;    off += (size_t)total * 4;
  off = seg_align(off);
  w.zero_bytes = off - w.off_zero;
  w.off_bitmap = off;     off = seg_align(off + (size_t)B * g.bm_bytes);
  w.off_rowdesc = off;    off = seg_align(off + NR * sizeof(SegRowDesc));
  w.off_part1 = off;      off = seg_align(off + NR * g.nseg * kSegGroupWarps * 8);
  w.off_rowstat = off;    off = seg_align(off + NR * sizeof(SegRowStat));
  w.off_zx = off;         off = seg_align(off + NR * 4);
  w.off_pos = off;        off = seg_align(off + (size_t)total * sizeof(SegPos));
  w.off_part2 = off;      off = seg_align(off + (size_t)total * g.upj * kSegGroupWarps * 4);
  w.off_jobdesc = off;    off = seg_align(off + (size_t)total * sizeof(SegJobDesc));
  w.off_req_status = off; off = seg_align(off + (size_t)B * 4);
  w.off_req_need = off;   off = seg_align(off + (size_t)B * 4);
  w.off_posdesc = off;    off = seg_align(off + (size_t)total * sizeof(SegRowDesc));
  w.total = off;
  return w;
}

struct SegParams {
  // inputs (as in spec_args)
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
  const float* tv_budget;
  const float* uniforms;
  int B, V, total, max_k;
  unsigned flags;
  int mode;                 // kModeSample or kModeTvOnly
  // outputs
  int* out_tokens;
  int* out_accepted;
  int* out_status;
  float* out_tv;
  float* out_theta;
  float* out_px;
  float* out_qx;
  // geometry
  SegGeom g;
  int NT;                   // target rows (total + B); draft row k is physical row NT + k
  int NR;                   // all rows
  long long wait_limit;     // cycles a bounded wait may spin
  // control words: a per-device array, zero between calls (the call's last
  // CTA clears it before it exits)
  unsigned* ctl;
  // workspace
  unsigned char* zero;      // the per-call counters [zero, zero + zero_bytes): cleared by the CTAs
  size_t zero_bytes;        // before the prologue's grid-wide wait (a multiple of 16)
  unsigned* row_cnt;
  unsigned* req_rows;
  unsigned* req_pend;
  unsigned* req_done;
  unsigned* job_cnt;
  int* jobs;                // [2 * total] published jobs: (position + 1, request); 0 = not yet written
  uint32_t* bitmap;         // [B][bm_bytes / 4]
  SegRowDesc* rowdesc;      // [NR], rows in request order
  SegRowDesc* posdesc;      // [total]: position p's target-row descriptor (second pass)
  float2* part1;            // [NR * nseg][8]: (reference, sum) per pass-1 unit and warp
  SegRowStat* rowstat;      // [NR]
  float* zx;                // [NR]: penalised logit of the row's draft token
  SegPos* pos;              // [total]
  float* part2;             // [total][upj][8]: residual mass per pass-2 unit and warp
  SegJobDesc* jobdesc;      // [total]
  int* req_status;          // [B]
  unsigned* req_need;       // [B] jobs a request waits for
};

}  // namespace sv
