// C ABI of libspecverify.so: host-side validation, workspace layout and
// launches.  No entry point allocates, frees or synchronises; all device
// work is enqueued on the caller's stream.
#include <cstdint>
#include <atomic>
#include <cstring>

#include <cuda_runtime.h>
#include <nvtx3/nvToolsExt.h>

#include "spec_verify.h"
#include "spec_internal.h"
#include "conf_internal.h"
#include "seg_internal.h"
#include "topp_internal.h"

namespace sv {
int choose_resident_layout(int V, int elem_bytes, bool topp, int max_smem, int* C_out, SmemLayout* L_out);
int choose_stream_layout(int V, int C, int elem_bytes, bool topp, int max_smem, int smem_per_sm,
                         SmemLayout* L_out);
int launch_sample_verify(SampleParams& P, bool bf16, bool topp, cudaStream_t stream);
int launch_greedy_verify(const GreedyParams& P, bool bf16, cudaStream_t stream);
int choose_pipe_layout(int V, int elem_bytes, int max_smem, PipeLayout* out);
int launch_pipe_verify(SampleParams& P, bool bf16, int num_sms, cudaStream_t stream);
int launch_confidence(const ConfParams& P, bool bf16, cudaStream_t stream);
int choose_conf_layout(int V, int elem_bytes, int B, int max_smem, ConfLayout* out);
int launch_conf_pipe(const ConfParams& P, bool bf16, int num_sms, cudaStream_t stream);
int launch_seg_verify(const SegParams& P, bool bf16, int num_sms, cudaStream_t stream);
int launch_topp_verify(const ToppParams& P, bool bf16, int num_sms, cudaStream_t stream);
int topp_cut_smem_bytes();
int seg_smem_bytes();
unsigned* seg_ctl_address();
}  // namespace sv

namespace {

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

int elem_bytes(int dtype) { return dtype == SPEC_BF16 ? 2 : 4; }

// Checks shared by all entry points.  `need_draft`: draft logits are read.
int check_common(const spec_args* a, bool need_draft) {
  if (!a) return SPEC_ERR_NULL;
  if (a->dtype != SPEC_F32 && a->dtype != SPEC_BF16) return SPEC_ERR_DTYPE;
  if (a->B < 1 || a->V < 1 || a->total_drafts < 0 || a->max_k < 0) return SPEC_ERR_SHAPE;
  if (a->max_k > SPEC_MAX_K) return SPEC_ERR_K_TOO_LARGE;
  if ((long long)a->total_drafts > (long long)a->B * a->max_k) return SPEC_ERR_SHAPE;
  if (!a->cu_draft || !a->target_logits) return SPEC_ERR_NULL;
  if (a->total_drafts > 0 && !a->draft_tokens) return SPEC_ERR_NULL;
  if (a->cu_hist && !a->hist_tokens) return SPEC_ERR_NULL;
  const int es = elem_bytes(a->dtype);
  if (a->ld_target < a->V) return SPEC_ERR_SHAPE;
  if (!aligned16(a->target_logits) || (a->ld_target * es) % 16 != 0) return SPEC_ERR_ALIGN;
  if (need_draft && a->total_drafts > 0) {
    if (!a->draft_logits) return SPEC_ERR_NULL;
    if (a->ld_draft < a->V) return SPEC_ERR_SHAPE;
    if (!aligned16(a->draft_logits) || (a->ld_draft * es) % 16 != 0) return SPEC_ERR_ALIGN;
  }
  return SPEC_OK;
}

int check_workspace(const spec_args* a, const void* ws, size_t ws_bytes) {
  if (!ws) return SPEC_ERR_WORKSPACE;
  if ((reinterpret_cast<uintptr_t>(ws) & 255u) != 0) return SPEC_ERR_WORKSPACE;
  if (ws_bytes < spec_workspace_bytes(a->B, a->total_drafts, a->V)) return SPEC_ERR_WORKSPACE;
  return SPEC_OK;
}

int device_props(int* max_smem, int* num_sms, int* smem_per_sm = nullptr) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) { cudaGetLastError(); return SPEC_ERR_DEVICE; }
  int per_sm = 0;
  if (cudaDeviceGetAttribute(max_smem, cudaDevAttrMaxSharedMemoryPerBlockOptin, dev) != cudaSuccess ||
      cudaDeviceGetAttribute(num_sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess ||
      cudaDeviceGetAttribute(&per_sm, cudaDevAttrMaxSharedMemoryPerMultiprocessor, dev) != cudaSuccess) {
    cudaGetLastError();
    return SPEC_ERR_DEVICE;
  }
  if (smem_per_sm) *smem_per_sm = per_sm;
  return SPEC_OK;
}

void fill_sample_inputs(sv::SampleParams& P, const spec_args* a) {
  std::memset(&P, 0, sizeof(P));
  P.target = a->target_logits;
  P.ld_t = a->ld_target;
  P.draft = a->draft_logits;
  P.ld_d = a->ld_draft;
  P.cu_draft = a->cu_draft;
  P.draft_tokens = a->draft_tokens;
  P.cu_hist = a->cu_hist;
  P.hist = a->hist_tokens;
  P.temperature = a->temperature;
  P.rep_penalty = a->rep_penalty;
  P.top_p = a->top_p;
  P.tv_budget = a->tv_budget;
  P.uniforms = a->uniforms;
  P.B = a->B;
  P.V = a->V;
  P.total = a->total_drafts;
  P.max_k = a->max_k;
  P.flags = a->flags;
}

// An NVTX range around each entry point's host work and launches (named
// after the entry point), for timelines taken with a profiler; without one
// attached the push and pop do nothing.
struct NvtxRange {
  explicit NvtxRange(const char* name) { nvtxRangePushA(name); }
  ~NvtxRange() { nvtxRangePop(); }
  NvtxRange(const NvtxRange&) = delete;
  NvtxRange& operator=(const NvtxRange&) = delete;
};

// Default bound on every wait of the split-vocabulary kernel, in SM clock
// cycles (about two seconds at any clock this part runs); the calls use
// g_seg_wait_limit, which spec_set_wait_cycles changes.
constexpr long long kSegWaitLimit = 4000000000ll;
std::atomic<long long> g_seg_wait_limit{kSegWaitLimit};

// Tags of the calls whose kernels count arrivals with tagged_arrive: one per
// call, in [1, 2^40).  Outside stream capture a call takes a fresh tag and
// enqueues nothing but its kernel.  Under capture the tag would be replayed
// with the graph, so the call captures a clear of its B counters instead and
// uses tag 0, which a cleared word carries.
std::atomic<unsigned long long> g_call_tag{0};

int call_tag(unsigned long long* counters, int B, cudaStream_t s, unsigned long long* tag) {
  cudaStreamCaptureStatus cs = cudaStreamCaptureStatusNone;
  if (cudaStreamIsCapturing(s, &cs) != cudaSuccess) {
    cudaGetLastError();
    return SPEC_ERR_LAUNCH;
  }
  if (cs != cudaStreamCaptureStatusNone) {
    if (cudaMemsetAsync(counters, 0, (size_t)B * sizeof(unsigned long long), s) != cudaSuccess) {
      cudaGetLastError();
      return SPEC_ERR_LAUNCH;
    }
    *tag = 0;
    return SPEC_OK;
  }
  const unsigned long long span = (1ull << (64 - sv::kTagShift)) - 1ull;
  *tag = g_call_tag.fetch_add(1, std::memory_order_relaxed) % span + 1ull;
  return SPEC_OK;
}

// The split-vocabulary kernel can serve sampling without top-p when a row
// has at most kSegMaxSegs segments (V <= 491520 bf16, 245760 fp32).
bool seg_fits(const spec_args* a) {
  return !a->top_p && sv::make_seg_geom(a->V, elem_bytes(a->dtype)).nseg <= sv::kSegMaxSegs;
}

// It does when asked for, and by default for batches the resident cluster
// kernel would not take in one wave (`resident_pick`: the choice made
// without hints).  SPEC_PREFER_RESIDENT and SPEC_PREFER_STREAMING keep the
// kernels they name.
// TV-only calls need the second pass over every position, which the
// pipelined kernel serves from L2 (its two passes over a row run back to
// back), so they take the split kernel only when asked for it.
bool use_seg(const spec_args* a, bool resident_pick, bool tv_only) {
  if (!seg_fits(a)) return false;
  if (a->flags & SPEC_PREFER_SPLIT) return true;
  if (a->flags & (SPEC_PREFER_RESIDENT | SPEC_PREFER_STREAMING)) return false;
  return !resident_pick && !tv_only;
}

// The split-vocabulary kernel (no top-p): sampling or the TV quantities.
int run_seg(const sv::SampleParams& S, const spec_args* a, void* ws, int num_sms, int max_smem,
            cudaStream_t stream) {
  if (sv::seg_smem_bytes() > max_smem) return SPEC_ERR_DEVICE;
  const int es = elem_bytes(a->dtype);
  const sv::SegWorkspace W = sv::make_seg_workspace(a->B, a->total_drafts, a->V, es);
  unsigned char* w = static_cast<unsigned char*>(ws);
  sv::SegParams P;
  std::memset(&P, 0, sizeof(P));
  P.target = a->target_logits;
  P.ld_t = a->ld_target;
  P.draft = a->draft_logits;
  P.ld_d = a->ld_draft;
  P.cu_draft = a->cu_draft;
  P.draft_tokens = a->draft_tokens;
  P.cu_hist = a->cu_hist;
  P.hist = a->hist_tokens;
  P.temperature = a->temperature;
  P.rep_penalty = a->rep_penalty;
  P.tv_budget = a->tv_budget;
  P.uniforms = S.uniforms;
  P.B = a->B;
  P.V = a->V;
  P.total = a->total_drafts;
  P.max_k = a->max_k;
  P.flags = a->flags;
  P.mode = S.mode;
  P.out_tokens = S.out_tokens;
  P.out_accepted = S.out_accepted;
  P.out_status = S.out_status;
  P.out_tv = S.out_tv;
  P.out_theta = S.out_theta;
  P.out_px = S.out_px;
  P.out_qx = S.out_qx;
  P.g = sv::make_seg_geom(a->V, es);
  P.NT = a->total_drafts + a->B;
  P.NR = 2 * a->total_drafts + a->B;
  P.wait_limit = g_seg_wait_limit.load(std::memory_order_relaxed);
  P.ctl = sv::seg_ctl_address();
  if (!P.ctl) return SPEC_ERR_DEVICE;
  P.zero = w + W.off_jobs;
  P.zero_bytes = W.zero_bytes - (W.off_jobs - W.off_zero);
  P.row_cnt = reinterpret_cast<unsigned*>(w + W.off_row_cnt);
  P.req_rows = reinterpret_cast<unsigned*>(w + W.off_req_rows);
  P.req_pend = reinterpret_cast<unsigned*>(w + W.off_req_pend);
  P.req_done = reinterpret_cast<unsigned*>(w + W.off_req_done);
  P.job_cnt = reinterpret_cast<unsigned*>(w + W.off_job_cnt);
  P.jobs = reinterpret_cast<int*>(w + W.off_jobs);
  P.bitmap = reinterpret_cast<uint32_t*>(w + W.off_bitmap);
  P.rowdesc = reinterpret_cast<sv::SegRowDesc*>(w + W.off_rowdesc);
  P.part1 = reinterpret_cast<float2*>(w + W.off_part1);
  P.rowstat = reinterpret_cast<sv::SegRowStat*>(w + W.off_rowstat);
  P.zx = reinterpret_cast<float*>(w + W.off_zx);
  P.pos = reinterpret_cast<sv::SegPos*>(w + W.off_pos);
  P.part2 = reinterpret_cast<float*>(w + W.off_part2);
  P.jobdesc = reinterpret_cast<sv::SegJobDesc*>(w + W.off_jobdesc);
  P.req_status = reinterpret_cast<int*>(w + W.off_req_status);
  P.req_need = reinterpret_cast<unsigned*>(w + W.off_req_need);
  P.posdesc = reinterpret_cast<sv::SegRowDesc*>(w + W.off_posdesc);
  return sv::launch_seg_verify(P, a->dtype == SPEC_BF16, num_sms, stream) == 0 ? SPEC_OK : SPEC_ERR_LAUNCH;
}

// The top-p path (row-cut and finish kernels) serves top-p batches unless a
// cluster kernel is asked for, when its records fit the buffer the call has
// (a workspace is always large enough; the fixed scratch may not be) and V
// fits its penalty bitmap.
bool use_topp(const spec_args* a, size_t ws_bytes, int max_smem) {
  if (!a->top_p || (a->flags & (SPEC_PREFER_RESIDENT | SPEC_PREFER_STREAMING))) return false;
  if (a->V > sv::kCutMaxV || sv::topp_cut_smem_bytes() > max_smem) return false;
  return sv::make_topp_workspace(a->B, a->total_drafts, a->V).total <= ws_bytes;
}

int run_topp(const sv::SampleParams& S, const spec_args* a, void* ws, int num_sms, cudaStream_t stream) {
  const sv::ToppWorkspace W = sv::make_topp_workspace(a->B, a->total_drafts, a->V);
  unsigned char* w = static_cast<unsigned char*>(ws);
  sv::ToppParams P;
  std::memset(&P, 0, sizeof(P));
  P.target = a->target_logits;
  P.ld_t = a->ld_target;
  P.draft = a->draft_logits;
  P.ld_d = a->ld_draft;
  P.cu_draft = a->cu_draft;
  P.draft_tokens = a->draft_tokens;
  P.cu_hist = a->cu_hist;
  P.hist = a->hist_tokens;
  P.temperature = a->temperature;
  P.rep_penalty = a->rep_penalty;
  P.top_p = a->top_p;
  P.tv_budget = a->tv_budget;
  P.uniforms = S.uniforms;
  P.B = a->B;
  P.V = a->V;
  P.total = a->total_drafts;
  P.max_k = a->max_k;
  P.flags = a->flags;
  P.mode = S.mode;
  P.NT = a->total_drafts + a->B;
  P.NR = 2 * a->total_drafts + a->B;
  P.out_tokens = S.out_tokens;
  P.out_accepted = S.out_accepted;
  P.out_status = S.out_status;
  P.out_tv = S.out_tv;
  P.out_theta = S.out_theta;
  P.out_px = S.out_px;
  P.out_qx = S.out_qx;
  P.rows = reinterpret_cast<sv::CutRow*>(w + W.off_rows);
  P.broken = reinterpret_cast<unsigned long long*>(w + W.off_ctr);
  P.pool = reinterpret_cast<int*>(w + W.off_pool);
  P.pool_cap = W.pool_cap;
  const int rc = call_tag(P.broken, 1, stream, &P.tag);
  if (rc) return rc;
  return sv::launch_topp_verify(P, a->dtype == SPEC_BF16, num_sms, stream) == 0 ? SPEC_OK : SPEC_ERR_LAUNCH;
}

// Picks the kernel variant.  Resident (each logit read once, values kept in
// the shared memory of a C-CTA cluster) when every work item gets its own
// cluster in one wave; otherwise the split-vocabulary kernel without top-p
// and the cluster kernel's streaming variant with top-p.  SPEC_PREFER_*
// flags override the choice; SPEC_PREFER_STREAMING without top-p names the
// pipelined kernel (one CTA per SM, pass 1 of the next item overlapping
// pass 2 of the current one).
int run_sample(sv::SampleParams& P, const spec_args* a, void* ws, size_t ws_bytes, cudaStream_t stream) {
  int max_smem = 0, num_sms = 0, smem_per_sm = 0;
  int rc = device_props(&max_smem, &num_sms, &smem_per_sm);
  if (rc) return rc;
  const bool topp = a->top_p != nullptr;
  if (topp && use_topp(a, ws_bytes, max_smem)) return run_topp(P, a, ws, num_sms, stream);
  const int es = elem_bytes(a->dtype);
  int C_res = 0;
  sv::SmemLayout L_res{}, L_str{};
  const bool res_ok = sv::choose_resident_layout(a->V, es, topp, max_smem, &C_res, &L_res) == 0;
  int C_str = 1;
  while (C_str <= sv::kMaxCluster &&
         sv::choose_stream_layout(a->V, C_str, es, topp, max_smem, smem_per_sm, &L_str) != 0)
    C_str *= 2;
  const bool str_ok = C_str <= sv::kMaxCluster;
  const bool resident_pick = res_ok && (!str_ok || (long long)P.n_items * C_res <= num_sms);
  if (use_seg(a, resident_pick, P.mode == sv::kModeTvOnly)) return run_seg(P, a, ws, num_sms, max_smem, stream);
  bool resident;
  if ((a->flags & SPEC_PREFER_RESIDENT) && res_ok) resident = true;
  else if ((a->flags & SPEC_PREFER_STREAMING) && str_ok) resident = false;
  else resident = resident_pick;
  sv::PipeLayout L_pipe{};
  const bool pipe_ok = !topp && sv::choose_pipe_layout(a->V, es, max_smem, &L_pipe) == 0 &&
                       (long long)P.n_items <= (long long)num_sms * sv::kPipeMaxIters;
  if (!resident && !str_ok && !pipe_ok) return SPEC_ERR_SHAPE;
  const sv::WorkspaceLayout W = sv::make_workspace_layout(a->B, a->total_drafts, a->V);
  unsigned char* w = static_cast<unsigned char*>(ws);
  P.counters = reinterpret_cast<unsigned long long*>(w + W.off_counters);
  P.results = reinterpret_cast<sv::ItemResult*>(w + W.off_results);
  P.inval = reinterpret_cast<int*>(w + W.off_inval);
  P.tag = 0;
  if (P.mode == sv::kModeSample) {
    rc = call_tag(P.counters, a->B, stream, &P.tag);
    if (rc) return rc;
  }
  if (!resident && pipe_ok) {
    P.PL = L_pipe;
    return sv::launch_pipe_verify(P, a->dtype == SPEC_BF16, num_sms, stream);
  }
  P.C = resident ? C_res : C_str;
  P.L = resident ? L_res : L_str;
  return sv::launch_sample_verify(P, a->dtype == SPEC_BF16, topp, stream);
}

// ---- fixed device scratch of spec_verify_sample_static
// One buffer per device, placed by the CUDA runtime when this module loads;
// no call of this library allocates it.  Its address is looked up on every
// call (cudaGetSymbolAddress with the caller's device current): a host-side
// lookup that allocates nothing, and stays right after a device reset
// reloads the module.
static __device__ __align__(256) unsigned char g_static_scratch[SPEC_STATIC_SCRATCH_BYTES];

int static_scratch_address(void** out) {
  void* p = nullptr;
  if (cudaGetSymbolAddress(&p, g_static_scratch) != cudaSuccess || !p) {
    cudaGetLastError();
    return SPEC_ERR_DEVICE;
  }
  *out = p;
  return SPEC_OK;
}

// Scratch the sampling call needs: the cluster kernels' counters, results
// and flags, or the split-vocabulary kernel's records when it may serve the
// batch (the larger of the two then, as the choice between them depends on
// the device).
size_t sample_scratch_bytes(const spec_args* a) {
  const size_t n = sv::make_workspace_layout(a->B, a->total_drafts, a->V).off_partials;
  if (!seg_fits(a) || (a->flags & (SPEC_PREFER_RESIDENT | SPEC_PREFER_STREAMING))) return n;
  const size_t m = sv::make_seg_workspace(a->B, a->total_drafts, a->V, elem_bytes(a->dtype)).total;
  return m > n ? m : n;
}

}  // namespace

extern "C" {

size_t spec_workspace_bytes(int32_t B, int32_t total_drafts, int32_t V) {
  if (B < 0 || total_drafts < 0 || V < 0) return 0;
  size_t n = sv::make_workspace_layout(B, total_drafts, V).total;
  for (int es : {2, 4}) {
    const size_t m = sv::make_seg_workspace(B, total_drafts, V, es).total;
    if (m > n) n = m;
  }
  const size_t t = sv::make_topp_workspace(B, total_drafts, V).total;
  return t > n ? t : n;
}

int spec_verify_sample(const spec_args* a, int32_t* out_tokens, int32_t* out_accepted, int32_t* out_status,
                       void* workspace, size_t ws_bytes, spec_stream_t stream) {
  NvtxRange nvtx("spec_verify_sample");
  int rc = check_common(a, true);
  if (rc) return rc;
  if (!out_tokens || !out_accepted || !a->temperature || !a->tv_budget || !a->uniforms) return SPEC_ERR_NULL;
  rc = check_workspace(a, workspace, ws_bytes);
  if (rc) return rc;
  sv::SampleParams P;
  fill_sample_inputs(P, a);
  P.mode = sv::kModeSample;
  P.out_tokens = out_tokens;
  P.out_accepted = out_accepted;
  P.out_status = out_status;
  P.n_items = a->total_drafts + a->B;
  return run_sample(P, a, workspace, ws_bytes, reinterpret_cast<cudaStream_t>(stream));
}

int spec_verify_sample_static(const spec_args* a, int32_t* out_tokens, int32_t* out_accepted, int32_t* out_status,
                              spec_stream_t stream) {
  NvtxRange nvtx("spec_verify_sample_static");
  int rc = check_common(a, true);
  if (rc) return rc;
  if (!out_tokens || !out_accepted || !a->temperature || !a->tv_budget || !a->uniforms) return SPEC_ERR_NULL;
  if (sample_scratch_bytes(a) > SPEC_STATIC_SCRATCH_BYTES) return SPEC_ERR_STATIC_SCRATCH;
  void* scratch = nullptr;
  rc = static_scratch_address(&scratch);
  if (rc) return rc;
  sv::SampleParams P;
  fill_sample_inputs(P, a);
  P.mode = sv::kModeSample;
  P.out_tokens = out_tokens;
  P.out_accepted = out_accepted;
  P.out_status = out_status;
  P.n_items = a->total_drafts + a->B;
  return run_sample(P, a, scratch, SPEC_STATIC_SCRATCH_BYTES, reinterpret_cast<cudaStream_t>(stream));
}

int spec_tv_budget(const spec_args* a, float* out_tv, float* out_theta, float* out_p_at_draft,
                   float* out_q_at_draft, void* workspace, size_t ws_bytes, spec_stream_t stream) {
  NvtxRange nvtx("spec_tv_budget");
  int rc = check_common(a, true);
  if (rc) return rc;
  if (!out_tv || !out_theta || !a->temperature || !a->tv_budget) return SPEC_ERR_NULL;
  rc = check_workspace(a, workspace, ws_bytes);
  if (rc) return rc;
  if (a->total_drafts == 0) return SPEC_OK;
  sv::SampleParams P;
  fill_sample_inputs(P, a);
  P.mode = sv::kModeTvOnly;
  P.uniforms = nullptr;
  P.out_tv = out_tv;
  P.out_theta = out_theta;
  P.out_px = out_p_at_draft;
  P.out_qx = out_q_at_draft;
  P.n_items = a->total_drafts;
  return run_sample(P, a, workspace, ws_bytes, reinterpret_cast<cudaStream_t>(stream));
}

int spec_verify_greedy(const spec_args* a, int32_t* out_tokens, int32_t* out_accepted, int32_t* out_status,
                       void* workspace, size_t ws_bytes, spec_stream_t stream) {
  NvtxRange nvtx("spec_verify_greedy");
  int rc = check_common(a, false);
  if (rc) return rc;
  if (!out_tokens || !out_accepted) return SPEC_ERR_NULL;
  rc = check_workspace(a, workspace, ws_bytes);
  if (rc) return rc;
  const cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  int max_smem = 0, num_sms = 0;
  rc = device_props(&max_smem, &num_sms);
  if (rc) return rc;
  const sv::WorkspaceLayout W = sv::make_workspace_layout(a->B, a->total_drafts, a->V);
  unsigned char* w = static_cast<unsigned char*>(workspace);
  sv::GreedyParams P;
  std::memset(&P, 0, sizeof(P));
  P.target = a->target_logits;
  P.ld_t = a->ld_target;
  P.cu_draft = a->cu_draft;
  P.draft_tokens = a->draft_tokens;
  P.cu_hist = a->cu_hist;
  P.hist = a->hist_tokens;
  P.rep_penalty = a->rep_penalty;
  P.B = a->B;
  P.V = a->V;
  P.total = a->total_drafts;
  P.max_k = a->max_k;
  P.nck = (a->V + sv::kGreedyChunk - 1) / sv::kGreedyChunk;
  P.out_tokens = out_tokens;
  P.out_accepted = out_accepted;
  P.out_status = out_status;
  P.counters = reinterpret_cast<unsigned long long*>(w + W.off_counters);
  P.partials = reinterpret_cast<sv::GreedyPartial*>(w + W.off_partials);
  rc = call_tag(P.counters, a->B, s, &P.tag);
  if (rc) return rc;
  return sv::launch_greedy_verify(P, a->dtype == SPEC_BF16, s) == 0 ? SPEC_OK : SPEC_ERR_LAUNCH;
}

int spec_draft_confidence(const spec_args* a, float threshold, float* out_conf, int32_t* out_k_eff,
                          int32_t* out_status, void* workspace, size_t ws_bytes, spec_stream_t stream) {
  NvtxRange nvtx("spec_draft_confidence");
  if (!a) return SPEC_ERR_NULL;
  if (a->dtype != SPEC_F32 && a->dtype != SPEC_BF16) return SPEC_ERR_DTYPE;
  if (a->B < 1 || a->V < 1 || a->total_drafts < 0 || a->max_k < 0) return SPEC_ERR_SHAPE;
  if (a->max_k > SPEC_MAX_K) return SPEC_ERR_K_TOO_LARGE;
  if ((long long)a->total_drafts > (long long)a->B * a->max_k) return SPEC_ERR_SHAPE;
  if (!a->cu_draft || !out_k_eff) return SPEC_ERR_NULL;
  if (a->cu_hist && !a->hist_tokens) return SPEC_ERR_NULL;
  const int es = elem_bytes(a->dtype);
  if (a->total_drafts > 0) {
    if (!a->draft_logits || !a->draft_tokens || !out_conf) return SPEC_ERR_NULL;
    if (a->ld_draft < a->V) return SPEC_ERR_SHAPE;
    if (!aligned16(a->draft_logits) || (a->ld_draft * es) % 16 != 0) return SPEC_ERR_ALIGN;
  }
  int rc = check_workspace(a, workspace, ws_bytes);
  if (rc) return rc;
  int max_smem = 0, num_sms = 0;
  rc = device_props(&max_smem, &num_sms);
  if (rc) return rc;
  const cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  const sv::WorkspaceLayout W = sv::make_workspace_layout(a->B, a->total_drafts, a->V);
  unsigned char* w = static_cast<unsigned char*>(workspace);
  sv::ConfParams P;
  std::memset(&P, 0, sizeof(P));
  P.draft = a->draft_logits;
  P.ld_d = a->ld_draft;
  P.cu_draft = a->cu_draft;
  P.draft_tokens = a->draft_tokens;
  P.cu_hist = a->cu_hist;
  P.hist = a->hist_tokens;
  P.temperature = a->temperature;
  P.rep_penalty = a->rep_penalty;
  P.B = a->B;
  P.V = a->V;
  P.total = a->total_drafts;
  P.max_k = a->max_k;
  P.nck = (a->V + sv::kGreedyChunk - 1) / sv::kGreedyChunk;
  P.threshold = threshold;
  P.out_conf = out_conf;
  P.out_k_eff = out_k_eff;
  P.out_status = out_status;
  P.counters = reinterpret_cast<unsigned long long*>(w + W.off_counters);
  P.partials = reinterpret_cast<sv::ConfPartial*>(w + W.off_partials);
  rc = call_tag(P.counters, a->B, s, &P.tag);
  if (rc) return rc;
  // at least one draft row per SM: the pipelined kernel (whole rows per
  // CTA); smaller batches spread each row over 8192-token chunks
  if (a->total_drafts >= num_sms && sv::choose_conf_layout(a->V, es, a->B, max_smem, &P.CL) == 0)
    rc = sv::launch_conf_pipe(P, a->dtype == SPEC_BF16, num_sms, s);
  else
    rc = sv::launch_confidence(P, a->dtype == SPEC_BF16, s);
  return rc == 0 ? SPEC_OK : (rc == -2 ? SPEC_ERR_SHAPE : SPEC_ERR_LAUNCH);
}

int64_t spec_set_wait_cycles(int64_t cycles) {
  const long long v = cycles > 0 ? (long long)cycles : kSegWaitLimit;
  return (int64_t)g_seg_wait_limit.exchange(v, std::memory_order_relaxed);
}

const char* spec_status_string(int code) {
  switch (code) {
    case SPEC_OK: return "ok";
    case SPEC_ERR_NULL: return "a required pointer is NULL";
    case SPEC_ERR_SHAPE: return "B, V, total_drafts or ld out of range";
    case SPEC_ERR_DTYPE: return "unsupported dtype";
    case SPEC_ERR_K_TOO_LARGE: return "max_k exceeds SPEC_MAX_K (32)";
    case SPEC_ERR_WORKSPACE: return "workspace missing, misaligned or too small";
    case SPEC_ERR_ALIGN: return "logits must be 16-byte aligned with ld*sizeof(dtype) a multiple of 16";
    case SPEC_ERR_LAUNCH: return "CUDA launch failed";
    case SPEC_ERR_DEVICE: return "no usable CUDA device (needs sm_103a) or V too large";
    case SPEC_ERR_STATIC_SCRATCH:
      return "batch needs more than the fixed scratch of spec_verify_sample_static (SPEC_STATIC_SCRATCH_BYTES)";
    default: return "unknown status";
  }
}

}  // extern "C"
