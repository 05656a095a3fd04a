// Parameter block and shared-memory layout of the draft-confidence kernels
// (confidence.cu); the host entry point fills them (spec_verify.cu).
#pragma once

#include "spec_internal.h"

namespace sv {

// ------------------------------------------------------ draft confidence
// Chunked kernel: one partial per (row, chunk).  Pipelined kernel: one per
// row, m holding the row's confidence (s and pad unused).
struct ConfPartial {
  float m;    // chunk maximum of the penalised logits
  float s;    // sum over the chunk of 2^((z' - m) c)
  int flags;  // status bits
  int pad;
};

// Pipelined variant (batches with at least one draft row per SM): one CTA
// per SM loops over its rows; 16 streaming warps take one 2 KB segment of
// the row per stage from a TMA ring, a setup warp builds the next row's
// penalty bitmap and combines the current row, a producer warp fills the
// ring.
constexpr int kConfWarps = 16;   // streaming warps (+ setup + producer)
constexpr int kConfBufs = 2;     // per-row buffers (bitmap, hand-off block): row k streams while row k+1's is built
constexpr int kConfSlots = 5;    // ring slots (one stage of a row each), at most

// One row's hand-offs between the streaming warps and the setup warp.
struct ConfStats {
  float2 wp[kConfWarps];   // per streaming warp: (reference, sum) of 2^(z'c - ref)
  float zmax[kConfWarps];  // per streaming warp: the largest penalised logit
  int wflags[kConfWarps];  // status bits seen by each streaming warp
  int flags;               // status bits of the row
  int pen;                 // the repetition penalty applies (bitmap kb holds the set)
  float c, alpha;          // the row's log2(e)/T and penalty
};

struct ConfLayout {
  int seg;         // tokens per warp segment (2048 bytes)
  int nseg;        // segments per row
  int nst;         // stages per row
  int slots;       // ring slots
  int slot_bytes;  // kConfWarps * 2048
  int bm_words;    // bitmap words per buffer (nseg * seg / 32)
  int cu_ints;     // cu_draft entries cached in shared memory (0: read from global memory)
  int off_ring, off_bm, off_stats, off_cu, off_bar;
  int total;
};

inline ConfLayout make_conf_layout(int V, int elem_bytes, int slots, int B) {
  ConfLayout L{};
  L.seg = 2048 / elem_bytes;
  L.nseg = (V + L.seg - 1) / L.seg;
  L.nst = (L.nseg + kConfWarps - 1) / kConfWarps;
  L.slots = slots;
  L.slot_bytes = kConfWarps * 2048;
  L.bm_words = L.nseg * L.seg / 32;
  L.cu_ints = B + 1 <= 1024 ? B + 1 : 0;
  int off = 0;
  L.off_ring = off;   off += slots * L.slot_bytes;
  L.off_bm = off;     off += kConfBufs * align_up_i(L.bm_words * 4, 16);
  L.off_stats = off;  off += kConfBufs * align_up_i((int)sizeof(ConfStats), 16);
  L.off_cu = off;     off += align_up_i(L.cu_ints * 4, 16);
  L.off_bar = off;    off += (2 * slots + 2 * kConfBufs) * 8;
  L.total = align_up_i(off, 128);
  return L;
}

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
  unsigned long long* counters;   // [B] call-tagged arrivals (tagged_arrive)
  unsigned long long tag;         // this call's tag
  ConfPartial* partials;   // [total * nck]
  ConfLayout CL;           // pipelined variant only
};

}  // namespace sv
