// Top-p sampling path (topp_verify.cu): parameter block, per-row record and
// workspace layout shared by the host code and the two kernels.
//
// Nucleus sampling keeps, in each target and draft row, the smallest set of
// most probable tokens whose mass reaches top_p, ties at the cut included,
// and renormalises ("Speculative Decoding" note: both p and q pass through
// top-p before the test).  With the logit scales that language models
// produce the kept set is small (tens to a few thousand tokens), so the path
// has two kernels:
//  - the row-cut kernel reads every row once from HBM and leaves, per row,
//    its maximum, its mass, the cut value tau and the list of kept tokens;
//  - the finish kernel takes each request's decisions, TV distances and
//    draws from those lists alone, gathering the other row's logits at the
//    listed tokens (a filtered row is zero off its list).
// A row whose list does not fit its CTA's share of the pool (or a request
// with top_p = 1) is not listed, and the finish kernel scans its rows in
// full.
#pragma once

#include <cstddef>
#include <cstdint>

namespace sv {

constexpr int kCutConsumerWarps = 16;
constexpr int kCutThreads = (kCutConsumerWarps + 1) * 32;   // warp 0 produces
constexpr int kCutConsumers = kCutConsumerWarps * 32;
constexpr int kCutChunkBytes = 16384;                      // one TMA copy, one ring slot
constexpr int kCutSlots = 6;
constexpr int kCutCand = 10240;                            // candidate (index, logit) entries
constexpr int kCutMaxV = 262144;                           // penalty bitmap capacity (tokens)
constexpr int kCutBins = 1024;                             // select histogram bins
constexpr float kCutWindow = 13.f;                         // candidate window below the row max (log2 units)
constexpr int kCutPoolPerRow = 1024;                       // kept-list entries per row, on average
constexpr int kCutPoolMax = 1 << 23;                       // pool entries at most
constexpr int kCutListMax = 32768;                         // a longer kept set is not listed (dense)
constexpr int kFinThreads = 256;
constexpr int kCutViaRow = 1 << 16;                        // a record flag, not a status bit
constexpr int kCutStatusMask = 0xffff;

// Per logical row (request order: request b's rows start at 2 cu_draft[b] + b;
// target row i at 2i, draft row i at 2i + 1, the bonus row at 2K).
// p(v) = [z'(v) >= tau] 2^(z'(v) c - M) / Sk, z' the penalised logit.
struct CutRow {
  float M;        // largest z'c of the row (log2 units)
  float tau;      // the cut: keep z' >= tau (-inf keeps every token)
  float Sk;       // kept mass, in units of 2^(z'c - M)
  int n;          // kept tokens listed in the pool; -1: not listed (dense)
  int off;        // the list's first pool entry
  int flags;      // kStatusBadLogits; kCutViaRow: the cut was selected over the row in global memory
  float S;        // the row's whole mass, in units of 2^(z'c - M)
  unsigned tag;   // low 32 bits of the writing call's tag (a row the call left unwritten keeps another)
};
static_assert(sizeof(CutRow) == 32, "row record size");

struct ToppParams {
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
  int mode;              // kModeSample or kModeTvOnly
  int NT, NR;            // target rows (total + B), logical rows (2 total + B)
  int* out_tokens;
  int* out_accepted;
  int* out_status;
  float* out_tv;
  float* out_theta;
  float* out_px;
  float* out_qx;
  CutRow* rows;                  // [NR]
  int* pool;                     // kept token lists; CTA c of the row-cut grid fills
                                 // [c, c + 1) * (pool_cap / gridDim) in row order
  unsigned long long* broken;    // (tag << 1) | (cu_draft is not a valid packing)
  unsigned long long tag;        // the call's tag (rows carry its low 32 bits)
  int pool_cap;                  // pool entries
};

struct ToppWorkspace {
  size_t off_rows, off_ctr, off_pool, total;   // off_ctr: the `broken` word
  int pool_cap;
};

inline ToppWorkspace make_topp_workspace(int B, int total, int V) {
  (void)V;
  ToppWorkspace W{};
  const size_t NR = 2 * (size_t)total + (size_t)B;
  auto al = [](size_t x) { return (x + 255) / 256 * 256; };
  W.off_rows = 0;
  W.off_ctr = al(NR * sizeof(CutRow));
  W.off_pool = W.off_ctr + 256;
  size_t cap = NR * (size_t)kCutPoolPerRow;
  if (cap > (size_t)kCutPoolMax) cap = kCutPoolMax;
  W.pool_cap = (int)cap;
  W.total = al(W.off_pool + cap * 4);
  return W;
}

}  // namespace sv
