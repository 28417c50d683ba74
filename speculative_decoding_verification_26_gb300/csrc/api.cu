// api.cu -- the C ABI declared in include/spec_verify.h.
//
// Host side only: argument checks, workspace layout, and the two launches of
// one call on the caller's stream:
//   plan_kernel    (1 CTA)        resets counters, settles requests with bad
//                                 arguments, builds the row schedule;
//   verify_kernel  (persistent)   streams the needed logit rows, decides each
//                                 position as soon as its rows are in, and
//                                 runs each request's final draw.
// The second launch uses programmatic dependent launch, so its start-up
// overlaps the plan kernel; it waits on griddepcontrol.wait before reading
// the schedule.  The plan kernel is launched without it, so it starts only
// after all earlier work on the stream (which may be producing the inputs).
#include <cuda_runtime.h>

#include <atomic>
#include <cstdint>
#include <mutex>

#include "common.cuh"

using namespace sv;

namespace {

thread_local uint64_t g_launches = 0;
std::atomic<long long> g_wait_limit{kWaitLimitCycles};   // spec_set_wait_limit
thread_local cudaEvent_t g_prof_begin = nullptr, g_prof_end = nullptr;

struct DevState {
  bool ready = false;
  int ctas = 0;       // resident verify CTAs on the device (SMs x CTAs per SM, at most 2 per SM)
  int status = SPEC_OK;
};
constexpr int kMaxDevices = 64;
DevState g_dev[kMaxDevices];
std::mutex g_mu;

int device_state(int* ctas) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return SPEC_ERR_CUDA;
  if (dev < 0 || dev >= kMaxDevices) return SPEC_ERR_UNSUPPORTED;
  std::lock_guard<std::mutex> lk(g_mu);
  DevState& d = g_dev[dev];
  if (!d.ready) {
    int major = 0, minor = 0, n = 0;
    if (cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
      return SPEC_ERR_CUDA;
    if (major != 10 || minor != 3) {
      d.status = SPEC_ERR_UNSUPPORTED;   // the library carries sm_103a code only
    } else {
      cudaError_t e = configure_kernels();
      int per_sm = 0;
      if (e == cudaSuccess) e = verify_blocks_per_sm(&per_sm);
      if (e != cudaSuccess) return SPEC_ERR_CUDA;
      if (per_sm < 1) {
        d.status = SPEC_ERR_UNSUPPORTED;
      } else {
        d.status = SPEC_OK;
        n *= per_sm < 2 ? per_sm : 2;
      }
    }
    d.ctas = n;
    d.ready = true;
  }
  *ctas = d.ctas;
  return d.status;
}

bool sizes_ok(int B, int G, int V) {
  if (B < 1 || B > SPEC_MAX_B || G < 0 || G > SPEC_MAX_G || V < 2 || V >= (1 << 28)) return false;
  // work items, draw-queue and deferred-queue entries are counted in 32 bits
  const long long ce = chunk_elems(SPEC_F32), se = stage_elems(SPEC_F32);
  const long long rows = (long long)B * (2 * G + 1);
  const long long nch = (V + ce - 1) / ce, nres = (V + se - 1) / se;
  return rows * nch < (1ll << 31) && (long long)B * (kMaxDrawRounds * nres + 2 * G * nch + 2) < (1ll << 31);
}

bool aligned(const void* p, size_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }

struct Call {
  int mode;
  const void* target;
  const void* draft;
  int dtype, B, G, V;
  const int32_t* draft_tokens;
  const int32_t* gamma;
  const float* temperature;
  const float* uniforms;
  int32_t* accept_len;
  int32_t* tokens;
  int32_t* status;
  float* signals;
  float* row_signals;
  float* accept_prob;
  void* workspace;
  size_t workspace_bytes;
  cudaStream_t stream;
};

int run(const Call& c) {
  if (!sizes_ok(c.B, c.G, c.V) || (c.dtype != SPEC_F32 && c.dtype != SPEC_BF16)) return SPEC_ERR_INVALID_ARG;
  const size_t es = c.dtype == SPEC_BF16 ? 2 : 4;
  const bool greedy = c.mode == MODE_GREEDY, sample = c.mode == MODE_SAMPLE, sig = c.mode == MODE_SIGNALS;
  // required pointers
  if (!sig && (!c.target || !c.accept_len || !c.tokens)) return SPEC_ERR_INVALID_ARG;
  if (!sig && c.G > 0 && !c.draft_tokens) return SPEC_ERR_INVALID_ARG;
  if ((sample || sig) && c.G > 0 && !c.draft) return SPEC_ERR_INVALID_ARG;
  if (!greedy && !c.temperature) return SPEC_ERR_INVALID_ARG;
  if ((sample || c.mode == MODE_ONEHOT) && !c.uniforms) return SPEC_ERR_INVALID_ARG;
  if (sig && !c.signals) return SPEC_ERR_INVALID_ARG;
  if (!aligned(c.target, es) || !aligned(c.draft, es)) return SPEC_ERR_INVALID_ARG;
  const void* ptrs4[] = {c.draft_tokens, c.gamma, c.temperature, c.uniforms, c.accept_len, c.tokens,
                         c.status, c.signals, c.row_signals, c.accept_prob};
  for (const void* p : ptrs4)
    if (!aligned(p, 4)) return SPEC_ERR_INVALID_ARG;
  const Layout L = make_layout(c.B, c.G, c.V, c.dtype);
  if (!c.workspace || c.workspace_bytes < L.total) return SPEC_ERR_WORKSPACE;
  if (!aligned(c.workspace, 256)) return SPEC_ERR_INVALID_ARG;
  int ctas = 0;
  const int ds = device_state(&ctas);
  if (ds != SPEC_OK) return ds;

  unsigned char* ws = static_cast<unsigned char*>(c.workspace);
  Params P{};
  P.target = static_cast<const unsigned char*>(c.target);
  P.draft = static_cast<const unsigned char*>(c.draft);
  P.dtype = c.dtype; P.B = c.B; P.G = c.G; P.V = c.V; P.mode = c.mode;
  P.signals_on = sig ? 1 : (sample && c.signals ? 1 : 0);
  P.draft_tokens = c.draft_tokens; P.gamma = c.gamma; P.temperature = c.temperature; P.uniforms = c.uniforms;
  P.accept_len = c.accept_len; P.tokens = c.tokens; P.status = c.status;
  P.signals = c.signals; P.row_signals = c.row_signals; P.accept_prob = c.accept_prob;
  P.hdr = reinterpret_cast<Header*>(ws + L.hdr);
  P.req_flags = reinterpret_cast<int*>(ws + L.req_flags);
  P.known_reject = reinterpret_cast<int*>(ws + L.known_reject);
  P.row_list = reinterpret_cast<int*>(ws + L.row_list);
  P.req_scale = reinterpret_cast<float*>(ws + L.req_scale);
  P.req_scale_lo = reinterpret_cast<float*>(ws + L.req_scale_lo);
  P.req_ks = reinterpret_cast<float*>(ws + L.req_ks);
  P.req_gam = reinterpret_cast<int*>(ws + L.req_gam);
  P.req_status = reinterpret_cast<int*>(ws + L.req_status);
  P.req_fin = reinterpret_cast<unsigned*>(ws + L.req_fin);
  P.cparts = reinterpret_cast<tword*>(ws + L.cparts);
  P.dsum = reinterpret_cast<tword*>(ws + L.dsum);
  P.gsum = reinterpret_cast<tword*>(ws + L.gsum);
  P.dd = reinterpret_cast<tword*>(ws + L.dd);
  P.dq = reinterpret_cast<tword*>(ws + L.dq);
  P.claim = reinterpret_cast<tword*>(ws + L.claim);
  P.defq = reinterpret_cast<tword*>(ws + L.defq);
  P.nrows = L.nrows; P.nch = L.nch; P.nres = L.nres; P.dq_cap = L.dq_cap; P.def_cap = L.def_cap;
  // Lookahead: greedy and sample calls read every row in position-major order
  // and skip the rows past a decided reject (a dependency per position, a
  // read issued only once the position before is accepted, would put a full
  // pipeline latency on every step of a long chain).  A one-hot call reads
  // the target rows of positions 0 and 1 up front and the row of position
  // i + 2 once position i is accepted (its drafts are rejected early: most
  // later rows are not needed).
  P.lookahead = c.mode == MODE_ONEHOT ? 2 : c.G + 1;
  P.aligned_rows = ((size_t)c.V * es) % 16 == 0 && aligned(c.target, 16) && aligned(c.draft, 16);
  P.wait_limit = g_wait_limit.load(std::memory_order_relaxed);
  // Rows a draw may read again (positions 0 .. keep_pos, both models in the
  // full-q mode) are loaded with an evict-last L2 policy, as long as they
  // fill at most 3/4 of the 129 MB L2 of a GB300; the draw then reads them
  // from L2.  Calls without draws keep nothing.
  P.keep_pos = -1;
  if (sample || c.mode == MODE_ONEHOT) {
    const double per_pos = (double)c.B * (sample ? 2 : 1) * c.V * es;
    const double budget = 0.75 * 129.0 * 1024 * 1024;
    for (int j = 0; j <= c.G && (j + 1) * per_pos <= budget; ++j) P.keep_pos = j;
  }

  // persistent grid: every CTA resident at once (two per SM), never more
  // CTAs than work items
  const long long max_items = (long long)c.B * (2 * c.G + 1) * L.nch;
  const int grid1 = (int)(max_items < (long long)ctas ? max_items : (long long)ctas);
  const cudaEvent_t pb = g_prof_begin, pe = g_prof_end;
  g_prof_begin = g_prof_end = nullptr;
  cudaError_t e = launch_plan(P, c.stream);
  if (e == cudaSuccess) {
    ++g_launches;
    if (pb) e = cudaEventRecord(pb, c.stream);
  }
  if (e == cudaSuccess) e = launch_verify(P, grid1 > 0 ? grid1 : 1, c.stream, pb == nullptr);
  if (e == cudaSuccess) {
    ++g_launches;
    if (pe) e = cudaEventRecord(pe, c.stream);
  }
  return e == cudaSuccess ? SPEC_OK : SPEC_ERR_CUDA;
}

// Library-owned scratch of spec_verify_sample_static (one per device: a
// __device__ variable lives in each context that loads the module).
static __device__ __align__(256) unsigned char g_static_ws[SPEC_STATIC_WORKSPACE_BYTES];

// Device address of g_static_ws on the current device, looked up once per
// device with that device current.
void* g_static_addr[kMaxDevices] = {};

int static_workspace(void** out) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return SPEC_ERR_CUDA;
  if (dev < 0 || dev >= kMaxDevices) return SPEC_ERR_UNSUPPORTED;
  std::lock_guard<std::mutex> lk(g_mu);
  if (!g_static_addr[dev]) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_static_ws) != cudaSuccess || p == nullptr) return SPEC_ERR_CUDA;
    g_static_addr[dev] = p;
  }
  *out = g_static_addr[dev];
  return SPEC_OK;
}

}  // namespace

extern "C" {

size_t spec_workspace_bytes(int B, int G, int V) {
  if (!sizes_ok(B, G, V)) return 0;
  const Layout a = make_layout(B, G, V, SPEC_F32), b = make_layout(B, G, V, SPEC_BF16);
  return a.total > b.total ? a.total : b.total;
}

const char* spec_status_string(int code) {
  switch (code) {
    case SPEC_OK: return "ok";
    case SPEC_ERR_INVALID_ARG: return "invalid argument";
    case SPEC_ERR_WORKSPACE: return "workspace missing or too small";
    case SPEC_ERR_CUDA: return "CUDA launch or runtime error";
    case SPEC_ERR_UNSUPPORTED: return "device is not sm_103";
    default: break;
  }
  return "unknown code";
}

const char* spec_request_status_string(int bit) {
  switch (bit) {
    case SPEC_ST_OK: return "ok";
    case SPEC_ST_NONFINITE: return "non-finite logits in a row that was read";
    case SPEC_ST_BAD_TOKEN: return "draft token outside [0, V)";
    case SPEC_ST_BAD_GAMMA: return "gamma outside [0, G]";
    case SPEC_ST_ZERO_RESIDUAL: return "residual mass rounded to zero; drew from p";
    case SPEC_ST_GUARDED: return "near-tie draw taken again in extended precision (informational)";
    case SPEC_ST_TIMEOUT: return "internal wait timed out";
    case SPEC_ST_BAD_TEMPERATURE: return "temperature not positive and finite";
    case SPEC_ST_BAD_UNIFORM: return "uniform outside [0, 1)";
    default: break;
  }
  return "unknown status bit";
}

uint64_t spec_launch_count(void) { return g_launches; }

int spec_set_wait_limit(long long cycles) {
  g_wait_limit.store(cycles > 0 ? cycles : kWaitLimitCycles, std::memory_order_relaxed);
  return SPEC_OK;
}

int spec_profile_next_call(void* begin_event, void* end_event) {
  g_prof_begin = static_cast<cudaEvent_t>(begin_event);
  g_prof_end = static_cast<cudaEvent_t>(end_event);
  return SPEC_OK;
}

int spec_verify_greedy(const void* target_logits, int dtype, int B, int G, int V, const int32_t* draft_tokens,
                       const int32_t* gamma, int32_t* accept_len, int32_t* tokens, int32_t* status,
                       void* workspace, size_t workspace_bytes, spec_stream_t stream) {
  Call c{MODE_GREEDY, target_logits, nullptr, dtype, B, G, V, draft_tokens, gamma, nullptr, nullptr,
         accept_len, tokens, status, nullptr, nullptr, nullptr, workspace, workspace_bytes,
         reinterpret_cast<cudaStream_t>(stream)};
  return run(c);
}

int spec_verify_sample(const void* target_logits, const void* draft_logits, int dtype, int B, int G, int V,
                       const int32_t* draft_tokens, const int32_t* gamma, const float* temperature,
                       const float* uniforms, int32_t* accept_len, int32_t* tokens, float* signals,
                       float* accept_prob, int32_t* status, void* workspace, size_t workspace_bytes,
                       spec_stream_t stream) {
  Call c{MODE_SAMPLE, target_logits, draft_logits, dtype, B, G, V, draft_tokens, gamma, temperature, uniforms,
         accept_len, tokens, status, signals, nullptr, accept_prob, workspace, workspace_bytes,
         reinterpret_cast<cudaStream_t>(stream)};
  return run(c);
}

int spec_verify_sample_static(const void* target_logits, const void* draft_logits, int dtype, int B, int G,
                              int V, const int32_t* draft_tokens, const int32_t* gamma, const float* temperature,
                              const float* uniforms, int32_t* accept_len, int32_t* tokens, float* signals,
                              float* accept_prob, int32_t* status, spec_stream_t stream) {
  // size checks first: nothing touches the device when they fail
  const size_t need = spec_workspace_bytes(B, G, V);
  if (need == 0) return SPEC_ERR_INVALID_ARG;
  if (need > (size_t)SPEC_STATIC_WORKSPACE_BYTES) return SPEC_ERR_WORKSPACE;
  void* ws = nullptr;
  const int rc = static_workspace(&ws);
  if (rc != SPEC_OK) return rc;
  Call c{MODE_SAMPLE, target_logits, draft_logits, dtype, B, G, V, draft_tokens, gamma, temperature, uniforms,
         accept_len, tokens, status, signals, nullptr, accept_prob, ws, (size_t)SPEC_STATIC_WORKSPACE_BYTES,
         reinterpret_cast<cudaStream_t>(stream)};
  return run(c);
}

int spec_verify_onehot(const void* target_logits, int dtype, int B, int G, int V, const int32_t* draft_tokens,
                       const int32_t* gamma, const float* temperature, const float* uniforms, int32_t* accept_len,
                       int32_t* tokens, float* accept_prob, int32_t* status, void* workspace,
                       size_t workspace_bytes, spec_stream_t stream) {
  Call c{MODE_ONEHOT, target_logits, nullptr, dtype, B, G, V, draft_tokens, gamma, temperature, uniforms,
         accept_len, tokens, status, nullptr, nullptr, accept_prob, workspace, workspace_bytes,
         reinterpret_cast<cudaStream_t>(stream)};
  return run(c);
}

int spec_divergence_stats(const void* target_logits, const void* draft_logits, int dtype, int B, int G, int V,
                          const int32_t* gamma, const float* temperature, float* stats, int32_t* status,
                          spec_stream_t stream) {
  if (!sizes_ok(B, G, V) || (dtype != SPEC_F32 && dtype != SPEC_BF16)) return SPEC_ERR_INVALID_ARG;
  const size_t es = dtype == SPEC_BF16 ? 2 : 4;
  if (!temperature || (G > 0 && (!target_logits || !draft_logits || !stats))) return SPEC_ERR_INVALID_ARG;
  if (!aligned(target_logits, es) || !aligned(draft_logits, es)) return SPEC_ERR_INVALID_ARG;
  const void* ptrs4[] = {gamma, temperature, stats, status};
  for (const void* p : ptrs4)
    if (!aligned(p, 4)) return SPEC_ERR_INVALID_ARG;
  int ctas = 0;
  const int ds = device_state(&ctas);
  if (ds != SPEC_OK) return ds;
  const cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  if (status && cudaMemsetAsync(status, 0, sizeof(int32_t) * (size_t)B, s) != cudaSuccess) return SPEC_ERR_CUDA;
  if (G == 0) return SPEC_OK;
  int dev = 0, nsm = 0;
  if (cudaGetDevice(&dev) != cudaSuccess ||
      cudaDeviceGetAttribute(&nsm, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
    return SPEC_ERR_CUDA;
  DivParams P{};
  P.target = static_cast<const unsigned char*>(target_logits);
  P.draft = static_cast<const unsigned char*>(draft_logits);
  P.dtype = dtype; P.B = B; P.G = G; P.V = V;
  P.aligned = ((size_t)V * es) % 16 == 0 && aligned(target_logits, 16) && aligned(draft_logits, 16);
  P.gamma = gamma; P.temperature = temperature; P.stats = stats; P.status = status;
  const long long pairs = (long long)B * G;
  const int grid = (int)(pairs < (long long)nsm ? pairs : (long long)nsm);
  if (launch_divergence(P, grid, s) != cudaSuccess) return SPEC_ERR_CUDA;
  ++g_launches;
  return SPEC_OK;
}

int spec_filter_top_k_top_p(void* logits, int dtype, int n, int V, const int32_t* top_k, const float* top_p,
                            const float* temperature, int32_t* status, spec_stream_t stream) {
  if (n < 1 || V < 2 || V >= (1 << 28) || !logits || (dtype != SPEC_F32 && dtype != SPEC_BF16))
    return SPEC_ERR_INVALID_ARG;
  const size_t es = dtype == SPEC_BF16 ? 2 : 4;
  if (!aligned(logits, es)) return SPEC_ERR_INVALID_ARG;
  const void* ptrs4[] = {top_k, top_p, temperature, status};
  for (const void* p : ptrs4)
    if (!aligned(p, 4)) return SPEC_ERR_INVALID_ARG;
  int ctas = 0;
  const int ds = device_state(&ctas);
  if (ds != SPEC_OK) return ds;
  FiltParams P{};
  P.logits = static_cast<unsigned char*>(logits);
  P.dtype = dtype; P.n = n; P.V = V;
  P.top_k = top_k; P.top_p = top_p; P.temperature = temperature; P.status = status;
  const int grid = n < ctas ? n : ctas;   // one row per resident CTA at a time (two per SM)
  if (launch_filter(P, grid > 0 ? grid : 1, reinterpret_cast<cudaStream_t>(stream)) != cudaSuccess)
    return SPEC_ERR_CUDA;
  ++g_launches;
  return SPEC_OK;
}

int spec_gamma_select(const float* signals, const float* comp, const float* model, int B, int32_t* gamma_star,
                      float* expected, spec_stream_t stream) {
  if (B < 1 || B > SPEC_MAX_B || !signals || !model || !gamma_star) return SPEC_ERR_INVALID_ARG;
  if (!aligned(signals, 16)) return SPEC_ERR_INVALID_ARG;
  const void* ptrs4[] = {comp, model, gamma_star, expected};
  for (const void* p : ptrs4)
    if (!aligned(p, 4)) return SPEC_ERR_INVALID_ARG;
  int ctas = 0;
  const int ds = device_state(&ctas);
  if (ds != SPEC_OK) return ds;
  if (launch_gamma_select(signals, comp, model, B, gamma_star, expected, reinterpret_cast<cudaStream_t>(stream)) !=
      cudaSuccess)
    return SPEC_ERR_CUDA;
  ++g_launches;
  return SPEC_OK;
}

int spec_draft_signals(const void* draft_logits, int dtype, int B, int G, int V, const int32_t* gamma,
                       const float* temperature, float* signals, float* row_signals, int32_t* status,
                       void* workspace, size_t workspace_bytes, spec_stream_t stream) {
  Call c{MODE_SIGNALS, nullptr, draft_logits, dtype, B, G, V, nullptr, gamma, temperature, nullptr,
         nullptr, nullptr, status, signals, row_signals, nullptr, workspace, workspace_bytes,
         reinterpret_cast<cudaStream_t>(stream)};
  return run(c);
}

}  // extern "C"
