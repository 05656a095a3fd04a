/*
 * spec_verify.h — C ABI of the GB300 (sm_103a) speculative-decoding
 * verification library (libspecverify.so).
 *
 * The library runs the step that follows the target model's verify forward:
 * for every request it turns target logits [K+1, V] and draft logits [K, V]
 * into the emitted tokens of that round.
 *
 *   spec_verify_sample  mentored speculative sampling ("What I Gave Up to
 *                       Make Speculative Decoding Faster", section "A knob
 *                       for accepting more draft tokens"): p and q after
 *                       repetition penalty and temperature (and top-p, as in
 *                       the "Speculative Decoding" note, section "Warum eine
 *                       Korrektur noetig ist"); d = TV(p,q) = 1/2 sum|p-q|;
 *                       theta = min(1, D/d) (1 when d = 0);
 *                       pi = (1-theta) p + theta q; accept x ~ q with
 *                       probability min(1, pi(x)/q(x)); keep the prefix up
 *                       to the first rejection; replace the rejected token
 *                       by a draw from the normalised residual max(p-q, 0);
 *                       after a fully accepted draft, a bonus token from p.
 *                       D = 0 is lossless speculative sampling.
 *   spec_verify_greedy  greedy longest-prefix verification
 *                       ("Adaptive-SpecDecode-Lab" README, section "实现"):
 *                       argmax of each penalised target row, prefix match
 *                       against the drafts, the target's argmax as the
 *                       correction on the first mismatch, or as the bonus
 *                       when every draft matches.
 *   spec_tv_budget      the per-position quantities alone: d, theta, p(x),
 *                       q(x) ("What I Gave Up to Make Speculative Decoding
 *                       Faster", section "A knob for accepting more draft
 *                       tokens": the total variation d between the
 *                       processed target and draft rows, and the mixing
 *                       weight theta = min(1, D/d) it sets).
 *
 * Conventions shared by every entry point
 * ---------------------------------------
 * Memory: every pointer is caller-owned DEVICE memory (except `args`, which
 * is a host struct).  The library never allocates or frees memory and never
 * synchronises the device; all work is enqueued on `stream` and completes
 * asynchronously.  Inputs are only read; outputs are only written.
 *
 * Batch layout (packed ragged rows): request b has K_b = cu_draft[b+1] -
 * cu_draft[b] drafts (0 <= K_b <= max_k <= 32).  Its draft rows are
 * cu_draft[b] .. cu_draft[b+1]-1 of draft_logits; its target rows are
 * off_b .. off_b + K_b of target_logits with off_b = cu_draft[b] + b (row
 * off_b + i scores the token after [last committed, d_1..d_i]).
 * cu_draft must be non-decreasing with cu_draft[0] = 0 and
 * cu_draft[B] = total_drafts.
 *
 * Logits: row-major, `ld` elements between rows (ld >= V), fp32 or bf16.
 * Each buffer must start on a 16-byte boundary, ld * sizeof(dtype) must be a
 * multiple of 16, and the buffer must hold rows * ld elements (entries
 * V .. ld-1 of a row are padding and are never used; they may be read).
 *
 * Per-request scalars [B] (fp32): temperature T > 0, repetition penalty
 * alpha > 0 (NULL = 1, no penalty), top_p in (0,1] (NULL = 1, no filter),
 * TV budget D in [0,1].  Repetition penalty: for every distinct token t of
 * the request's history plus the drafts preceding the row,
 * z'_t = z_t/alpha if z_t > 0 else z_t*alpha (fp32, correctly rounded);
 * then z'' = z'/T.  Top-p keeps every token whose probability is at least
 * tau, tau being the probability at which the descending cumulative mass
 * first reaches top_p, and renormalises; it is applied to p and q
 * separately, before they are compared.
 *
 * Uniforms [total_drafts + B] in [0,1): u[off_b + i] (i < K_b) is the
 * acceptance draw of draft i; u[off_b + K_b] is the final draw (correction
 * or bonus).  Draws are inverse-CDF in token-id order: the smallest v whose
 * inclusive prefix mass exceeds u * (total mass).
 *
 * Outputs: out_tokens [total_drafts + B], request b writing slots
 * off_b .. off_b + K_b: the accepted drafts, then the correction or bonus,
 * then -1.  out_accepted [B] = number of accepted drafts.
 * out_status [B] (may be NULL) = 0, or an OR of SPEC_STATUS_* for invalid
 * per-request data; such a request's tokens and accepted count are -1.
 *
 * Return value: SPEC_OK (0) once the work is enqueued, or a negative
 * SPEC_ERR_* from the host-side checks (nothing is enqueued then) or from
 * the launch.  No entry point ever traps on the device.
 *
 * Workspace: spec_workspace_bytes(B, total_drafts, V) bytes of device
 * memory, at least 256-byte aligned.  Its contents need no initialisation
 * and every call is one kernel launch: the split-vocabulary sampling kernel
 * clears its counters itself at its start; the other kernels count each
 * request's arrivals on a 64-bit word tagged with the call (a process-wide
 * call number in [1, 2^40)), and a word with another tag counts as zero.
 * Under stream capture the tag would replay with the graph, so a captured
 * call also captures a cudaMemsetAsync of its B counter words (tag 0).
 * Calls that share one workspace must be ordered (same stream, or
 * synchronised).
 */
#ifndef SPEC_VERIFY_H
#define SPEC_VERIFY_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* A CUDA stream handle (cudaStream_t / CUstream); NULL = legacy stream. */
typedef struct CUstream_st *spec_stream_t;

enum { SPEC_F32 = 0, SPEC_BF16 = 1 };

enum {
  SPEC_OK = 0,
  SPEC_ERR_NULL = -1,        /* a required pointer is NULL                 */
  SPEC_ERR_SHAPE = -2,       /* B, V, total_drafts or ld out of range      */
  SPEC_ERR_DTYPE = -3,       /* dtype is not SPEC_F32 / SPEC_BF16          */
  SPEC_ERR_K_TOO_LARGE = -4, /* max_k > SPEC_MAX_K                         */
  SPEC_ERR_WORKSPACE = -5,   /* workspace NULL, misaligned or too small    */
  SPEC_ERR_ALIGN = -6,       /* logits not 16-byte aligned / ld*size % 16  */
  SPEC_ERR_LAUNCH = -7,      /* the CUDA launch failed                     */
  SPEC_ERR_DEVICE = -8,      /* no usable device, or V too large for it    */
  SPEC_ERR_STATIC_SCRATCH = -9 /* spec_verify_sample_static: the batch needs
                                  more than SPEC_STATIC_SCRATCH_BYTES        */
};

/* out_status bits */
enum {
  SPEC_STATUS_BAD_TOKEN = 1,  /* a draft or history token outside [0,V)       */
  SPEC_STATUS_BAD_PARAM = 2,  /* T <= 0, alpha <= 0, top_p not in (0,1],
                                 D not in [0,1], or NaN                      */
  SPEC_STATUS_BAD_LOGITS = 4, /* NaN or +inf logit (sampling: or a row whose
                                 logits are all -inf)                        */
  SPEC_STATUS_BAD_K = 8,      /* K_b < 0, K_b > max_k, or cu_draft broken     */
  SPEC_STATUS_TIMEOUT = 16    /* an internal wait ran out (not expected)     */
};

#define SPEC_MAX_K 32
/* flags: emit no bonus token after a fully accepted draft (the mentored-
   decoding engine's behaviour; "Even full acceptance did not buy a
   speedup").  out_tokens slot off_b + K_b is then -1 in that case. */
#define SPEC_NO_BONUS 1u
/* flags, sampling only: kernel strategy hints (results agree with the
   definition either way; fp32 rounding may differ in the last bits).
   RESIDENT keeps each CTA's slice of both rows in shared memory and reads
   every logit once; it suits batches whose work items (sum K_b + B) all fit
   in one wave of clusters.  SPLIT (without top-p) cuts every row into
   vocabulary segments spread over all SMs: one read of each logit for the
   softmax statistics, and a second read of only the rows of positions whose
   decision those statistics leave open.  STREAMING without top-p names the
   pipelined kernel (about one work item per SM in flight, each item's
   second pass re-read from L2); with top-p, the cluster kernel's streaming
   variant.  Without a hint: RESIDENT when the batch fits in one wave, else
   SPLIT (rows of at most 32 segments: V <= 491520 bf16, 245760 fp32).
   With top-p and no RESIDENT or STREAMING hint (SPLIT included), the top-p
   path: a row-cut kernel reads every row once and keeps each row's exact
   nucleus as a token list, and a finish kernel decides and draws from the
   lists (V <= 262144, and the buffer large enough for its records: always
   for a workspace). */
#define SPEC_PREFER_RESIDENT 2u
#define SPEC_PREFER_STREAMING 4u
#define SPEC_PREFER_SPLIT 8u

typedef struct {
  int32_t B;             /* requests, >= 1                                   */
  int32_t V;             /* vocabulary, >= 1                                 */
  int32_t total_drafts;  /* sum of K_b = cu_draft[B]                         */
  int32_t max_k;         /* upper bound on every K_b, <= SPEC_MAX_K          */
  int32_t dtype;         /* SPEC_F32 or SPEC_BF16 (both logit buffers)        */
  const int32_t *cu_draft;     /* [B+1]                                      */
  const void *target_logits;   /* [total_drafts + B, ld_target]              */
  int64_t ld_target;
  const void *draft_logits;    /* [total_drafts, ld_draft]; unused by greedy */
  int64_t ld_draft;
  const int32_t *draft_tokens; /* [total_drafts]                             */
  const int32_t *cu_hist;      /* [B+1] or NULL (no history)                 */
  const int32_t *hist_tokens;  /* [cu_hist[B]] or NULL                       */
  const float *temperature;    /* [B]; unused by greedy                      */
  const float *rep_penalty;    /* [B] or NULL                                */
  const float *top_p;          /* [B] or NULL; unused by greedy              */
  const float *tv_budget;      /* [B]; unused by greedy                      */
  const float *uniforms;       /* [total_drafts + B]; sampling only          */
  uint32_t flags;              /* SPEC_NO_BONUS | SPEC_PREFER_*              */
} spec_args;

/* Workspace size in bytes for a batch (covers all three entry points). */
size_t spec_workspace_bytes(int32_t B, int32_t total_drafts, int32_t V);

/* Mentored speculative sampling (see above).  Needs temperature, tv_budget
   and uniforms. */
int spec_verify_sample(const spec_args *args, int32_t *out_tokens, int32_t *out_accepted,
                       int32_t *out_status, void *workspace, size_t ws_bytes, spec_stream_t stream);

/* Greedy longest-prefix verification (see above).  Reads target_logits,
   draft_tokens, history and rep_penalty only.  The argmax compares the fp32
   penalised logits and takes the lowest token id on exact ties. */
int spec_verify_greedy(const spec_args *args, int32_t *out_tokens, int32_t *out_accepted,
                       int32_t *out_status, void *workspace, size_t ws_bytes, spec_stream_t stream);

/* Per-position mentored-decoding quantities ("What I Gave Up to Make
   Speculative Decoding Faster", section "A knob for accepting more draft
   tokens"), [total_drafts] each: out_tv = d = TV(p_i, q_i) = sum_v
   max(p_i(v) - q_i(v), 0), out_theta = theta_i = min(1, D_b / d) (1 when
   d <= D_b), out_p_at_draft = p_i(x_i), out_q_at_draft = q_i(x_i) (the last
   two may be NULL).  p_i and q_i are the target and draft rows after the
   repetition penalty, the temperature and top-p, as for sampling.  Invalid
   positions get NaN.  Reads no uniforms.  Same workspace as sampling. */
int spec_tv_budget(const spec_args *args, float *out_tv, float *out_theta, float *out_p_at_draft,
                   float *out_q_at_draft, void *workspace, size_t ws_bytes, spec_stream_t stream);

/* Draft confidence for early stopping ("Adaptive-SpecDecode-Lab" README,
 * section "Confidence-guided early stop": after each draft token the drafter
 * reads its top-1 probability from the logits it already has and stops
 * proposing below a threshold; that low-confidence token is still verified).
 *
 * For every draft row i of request b: out_conf[cu_draft[b] + i] =
 * max_v q_i(v), with q_i the draft distribution after the repetition penalty
 * (history plus the drafts before row i) and the temperature (top-p does not
 * enter).  out_k_eff[b] = i + 1 for the first row with confidence below
 * `threshold`, else K_b: the drafts a confidence-stopped drafter would have
 * proposed.  Reads draft_logits, cu_draft, draft_tokens, history,
 * temperature (NULL = 1) and rep_penalty; not the target logits.
 * out_status [B] (may be NULL) as for sampling; an invalid request gets
 * out_k_eff = -1 and NaN confidences.  One pass over the draft logits
 * (HBM-bound).  Same workspace as the other entry points. */
int spec_draft_confidence(const spec_args *args, float threshold, float *out_conf, int32_t *out_k_eff,
                          int32_t *out_status, void *workspace, size_t ws_bytes, spec_stream_t stream);

/* Fixed-scratch variant of spec_verify_sample: no workspace argument.
 *
 * The method has no counterpart to this call.  It serves callers that cannot
 * hand the library a workspace: a serving loop that planned all of its
 * device memory up front and has nothing left to give out per call, or a
 * caller for which a cudaMalloc at the point of the call (it may synchronise
 * the device) is not acceptable.
 *
 * Arguments, checks, kernels and results are those of spec_verify_sample;
 * the workspace is replaced by one buffer per device that the library holds
 * as a file-scope __device__ array of SPEC_STATIC_SCRATCH_BYTES (8 MiB).  The
 * call allocates and frees nothing.
 *
 * Size limit: the batch needs the scratch of the kernel the call runs.
 * Without top-p (the split-vocabulary kernel) that is about 160 bytes per
 * logit row (2 total_drafts + B rows), 64 bytes per row and vocabulary
 * segment (segments of 15360 bf16 or 7680 fp32 logits), V/8 bytes of
 * penalty bitmap per request and 64 bytes per vocabulary segment and draft;
 * for B = 64, K = 8, V = 152064 it is 2.4 MiB in bf16 and 3.3 MiB in fp32.
 * With top-p the top-p path needs 32 bytes per logical row and 4 KiB of
 * kept-token lists per row (B = 256, total_drafts = 1152: 10.5 MiB, over
 * the scratch); when that does not fit, the cluster kernel serves the
 * batch, with 96 bytes per work item
 * (total_drafts + B).  A batch that does not fit returns
 * SPEC_ERR_STATIC_SCRATCH and enqueues nothing.
 *
 * Zeroing: as for the workspace entry point (the split-vocabulary kernel
 * clears its counters at its start; the cluster kernel's counters are
 * call-tagged, cleared only under stream capture); everything else in the
 * buffer is written before it is read.
 *
 * Address: every call looks the buffer up with cudaGetSymbolAddress for the
 * current device (a host-side lookup that allocates nothing).  The first
 * call on a device may load the library's device code; make it outside any
 * stream capture.  A failed lookup returns SPEC_ERR_DEVICE.
 *
 * Races: all calls on one device share the buffer.  They must be ordered
 * (one stream, or synchronised); two calls in flight at once, on two streams
 * or from two host threads, race and corrupt each other's results. */
#define SPEC_STATIC_SCRATCH_BYTES (8u << 20)
int spec_verify_sample_static(const spec_args *args, int32_t *out_tokens, int32_t *out_accepted,
                              int32_t *out_status, spec_stream_t stream);

/* A static description of a return code. */
const char *spec_status_string(int code);

/* Diagnostic hook: the bound, in SM clock cycles, on every wait of the
   split-vocabulary sampling kernel (SPEC_PREFER_SPLIT, and the default
   without top-p).  Each wait that runs out sets a global abort flag; every
   CTA then stops, and the requests left unfinished get
   SPEC_STATUS_TIMEOUT (tokens -1, accepted -1) while the call itself still
   returns SPEC_OK.  cycles <= 0 restores the default of 4e9 cycles (about
   two seconds).  Process-wide; applies to calls launched afterwards.
   Returns the previous bound.  The wait for copies in flight before a CTA
   exits keeps its own fixed bound of about two seconds. */
int64_t spec_set_wait_cycles(int64_t cycles);

#ifdef __cplusplus
}
#endif
#endif /* SPEC_VERIFY_H */
