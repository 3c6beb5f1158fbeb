// Host runtime of libriver.so: the C ABI declared in include/river.h.
//
// Owns the model (weights in the kernels' layouts), the exit river, the
// shared KV cache with its per-step device state, and the CUDA graph that
// replays one decode step with a single launch.  Every step of the path runs
// in the kernels of this library; the host only validates arguments and
// enqueues launches.
#include <algorithm>
#include <atomic>
#include <cmath>
#include <cstdarg>
#include <cstdio>
#include <cstring>
#include <string>
#include <vector>

#include "internal.h"

using namespace river;

namespace {

thread_local std::string g_err;

rl_status fail(rl_status s, const char* fmt, ...) {
  char buf[512];
  va_list ap;
  va_start(ap, fmt);
  vsnprintf(buf, sizeof(buf), fmt, ap);
  va_end(ap);
  g_err = buf;
  return s;
}

// Allocation-failure injection (rl_debug_fail_allocations): the number of
// library allocations that may still succeed; negative = no injection.
std::atomic<long long> g_alloc_budget{-1};

// True when the next allocation must fail (and counts the one that may not).
bool alloc_injected_failure() {
  long long b = g_alloc_budget.load();
  while (b >= 0) {
    if (b == 0) return true;
    if (g_alloc_budget.compare_exchange_weak(b, b - 1)) return false;
  }
  return false;
}

#define RL_CUDA(call)                                                                    \
  do {                                                                                   \
    cudaError_t e_ = (call);                                                             \
    if (e_ != cudaSuccess) return fail(RL_ERR_CUDA, "%s: %s", #call, cudaGetErrorString(e_)); \
  } while (0)

#define RL_LAUNCHED()                                                                    \
  do {                                                                                   \
    cudaError_t e_ = cudaGetLastError();                                                 \
    if (e_ != cudaSuccess) return fail(RL_ERR_CUDA, "kernel launch: %s", cudaGetErrorString(e_)); \
  } while (0)

struct Linear {
  bf16* w = nullptr;        // [N][Kp]
  bf16* wt = nullptr;       // the same weights unit-tiled for the persistent step kernel
  uint32_t* qw = nullptr;   // [N][Kp/8]
  __half2* sz = nullptr;    // [N][Kp/128]
  unsigned char* qwt = nullptr;  // W4 + (s, z) in the fused kernel's unit-tiled layout
  int N = 0, K = 0, Kp = 0;
  int view_base = 0;        // first rl linear index this fused matrix maps to
  const int2* rowmap = nullptr;
  CUtensorMap tm;           // TMA map of w for the tensor-core GEMM (128 x 64 boxes)
  unsigned char* qtc = nullptr;  // W4 + (s, z) in the tensor-core GEMM's k-block layout
  // backbone offloading: w and wt live in host memory (w_host / wt points
  // there); w points into the model's device staging buffer
  bool offloaded = false;
  const bf16* w_host = nullptr;
};

struct Layer {
  Linear qkv, o, gu, dn;
  float* g_attn = nullptr;
  float* g_ffn = nullptr;
};

}  // namespace

struct rl_model {
  rl_config cfg;
  int L, d, Hq, Hkv, hd, F, V;
  int Kd, Ko, Kf, Nqkv;
  std::vector<Layer> layers;
  bf16* embed = nullptr;
  bf16* lm_head = nullptr;  // [V][Kd]
  bf16* lm_head_t = nullptr;  // unit-tiled copy
  CUtensorMap tm_lm;          // TMA map of lm_head for the tensor-core GEMM
  bool step_ok = false;       // the persistent step kernel can be launched cooperatively
  float* g_final = nullptr;
  float* inv_freq = nullptr;
  int2* map_qkv = nullptr;
  int2* map_gu = nullptr;
  int2* map_id = nullptr;
  bool quantized = false;
  std::vector<NSView> views;  // [L][7]
  NSView* d_views = nullptr;
  std::vector<void*> allocs;
  int sm_count = 0;
  size_t bytes = 0;

  template <typename T>
  rl_status alloc(T** p, size_t n) {
    void* q = nullptr;
    if (n == 0) n = 1;
    if (alloc_injected_failure()) return fail(RL_ERR_OOM, "cudaMalloc(%zu bytes): injected failure", n * sizeof(T));
    cudaError_t e = cudaMalloc(&q, n * sizeof(T));
    if (e != cudaSuccess) {
      cudaGetLastError();
      return fail(RL_ERR_OOM, "cudaMalloc(%zu bytes): %s", n * sizeof(T), cudaGetErrorString(e));
    }
    allocs.push_back(q);
    bytes += n * sizeof(T);
    *p = static_cast<T*>(q);
    return RL_OK;
  }
  // backbone offloading (rl_model_offload_backbone)
  int offload_from = -1;          // first offloaded layer (0-based), -1: none
  bf16* stage = nullptr;          // device buffer one offloaded layer's [N][Kp] weights are staged in
  std::vector<void*> host_allocs; // pinned host memory of the offloaded layers
  size_t host_bytes = 0;
  int epoch = 0;                  // bumped when weight pointers move (decode graphs are captured again)
  ~rl_model() {
    for (void* p : allocs) cudaFree(p);
    for (void* p : host_allocs) cudaFreeHost(p);
  }
  // Releases one device allocation made by alloc().
  void release(void* p, size_t nbytes) {
    for (size_t i = 0; i < allocs.size(); ++i)
      if (allocs[i] == p) {
        cudaFree(p);
        allocs.erase(allocs.begin() + (long)i);
        bytes -= nbytes;
        return;
      }
  }
};

namespace {

struct GraphKey {
  int B = -1, mode = -1;
  float tau = 0.f;
  const int* sched = nullptr;
  int sched_len = 0;
  const int* tokens = nullptr;
  float* logits = nullptr;
  int* next = nullptr;
  int* exit = nullptr;
  float* min_cos = nullptr;
  float* trace = nullptr;
  int prof = 0;  // 0 off, 1 event records, 2 + per-CTA timeline
  bool fused = false;
  bool step = false;
  long long wait = 0;  // rl_kv_set_wait_limit
  int epoch = 0;       // the model's weight-placement epoch
  bool operator==(const GraphKey& o) const {
    return B == o.B && mode == o.mode && tau == o.tau && sched == o.sched &&
           sched_len == o.sched_len && tokens == o.tokens && logits == o.logits &&
           next == o.next && exit == o.exit && min_cos == o.min_cos && trace == o.trace &&
           prof == o.prof && fused == o.fused && step == o.step && wait == o.wait &&
           epoch == o.epoch;
  }
};

// One profiled launch: kind, layer, algorithmic bytes of either path.
struct ProfRec {
  int kind = 0, layer = 0;
  bool gemv = false, attn = false;
  double bytes_bf = 0, bytes_w4 = 0;
  int phase = -1;      // >= 0: a phase of the persistent step kernel (timeline record)
};

}  // namespace

struct rl_kv {
  rl_model* m = nullptr;
  int maxB = 0, Tmax = 0;
  std::vector<bf16*> K, V;     // per-layer views into one allocation each
  CUtensorMap tmk, tmv;        // all layers' K / V as one 2-D tensor [L*maxB*Hkv*Tmax][hd], 16-row boxes
  CUtensorMap tmk64, tmv64;    // the same, 64-row boxes (streaming decode attention)
  bool tm_ok = false;
  DevState* st = nullptr;
  int host_pos = 0, host_step = 0;
  // decode workspace
  float* h[3] = {nullptr, nullptr, nullptr};
  bf16 *x_attn = nullptr, *x_ffn = nullptr, *o = nullptr, *u = nullptr;
  float *xs_attn = nullptr, *xs_ffn = nullptr, *xs_o = nullptr, *xs_u = nullptr;
  float* q = nullptr;
  float2* rope_cs = nullptr;  // (cos, sin) of pos * inv_freq[i], [Tmax][hd/2]
  float* part = nullptr;
  int nchunks_cap = 1;
  float* cosbuf = nullptr;
  // fused small-batch decode workspace (stream-K partials, tickets, argmax)
  float* ws = nullptr;
  unsigned* tile_ticket = nullptr;
  unsigned* cta_ticket = nullptr;
  unsigned* attn_ticket = nullptr;
  float* tc_ws = nullptr;             // split-K partial tiles of the tensor-core GEMM
  size_t tc_ws_floats = 0;
  unsigned* tc_ticket = nullptr;      // per output tile, zero between launches
  int tc_ticket_n = 0;
  float* am_val = nullptr;
  int* am_idx = nullptr;
  float* st_mid = nullptr;  // per-tile |h_mid|^2 of the O projection's output [d/16][8]
  float* st_end = nullptr;  // per-tile (|h_out|^2, <h_in,h_out>, |h_in|^2) of the layer [d/16][8][3]
  bool use_fused = true;
  int path_pref = RL_PATH_AUTO;  // rl_kv_set_decode_path
  long long wait_limit = 0;      // rl_kv_set_wait_limit (0: the kernels' own limits)
  // persistent step kernel
  bool use_step = true;
  unsigned* bars = nullptr;           // per-CTA phase flags [n_bars], 128 bytes apart
  size_t n_bars = 0;
  unsigned* tctr = nullptr;           // per-phase tile counters [nph_cap]
  PhaseDesc* d_ph = nullptr;          // phase descriptors [nph_cap]
  std::vector<PhaseDesc> h_ph;        // host copy of what d_ph holds
  int nph_cap = 0;
  float* part_s = nullptr;            // attention partials [min(maxB,8)][Hq][part_cap][hd+4]
  int part_cap = 0;
  unsigned long long* tl = nullptr;   // per-phase timeline (profiling) [2][nph_cap]
  unsigned long long* tl2 = nullptr;  // per-CTA timeline (profiling level 2) [nph_cap][grid][kTl2]
  bool timeline = false;
  int nph_last = 0;
  int n_tile_ticket = 0;
  // buffers of the host-pointer entry point
  int* d_tok = nullptr;
  int* d_next = nullptr;
  int* d_exit = nullptr;
  float* d_logits = nullptr;
  float* d_mincos = nullptr;
  float* trace = nullptr;
  // decode graph
  cudaGraphExec_t exec = nullptr;
  GraphKey key;
  // step path: the captured graph, its kernel node and the arguments captured
  // (a new token pointer only updates the node's parameters)
  cudaGraph_t graph = nullptr;
  cudaGraphNode_t step_node = nullptr;
  StepArgs step_args;
  // live profiling
  bool profiling = false;
  std::vector<cudaEvent_t> ev;
  std::vector<ProfRec> recs;
  int nrec = 0;
  int* d_paths = nullptr;
  int prof_pos = 0, prof_B = 1;
  std::vector<void*> allocs;

  template <typename T>
  rl_status alloc(T** p, size_t n) {
    void* q = nullptr;
    if (n == 0) n = 1;
    if (alloc_injected_failure()) return fail(RL_ERR_OOM, "cudaMalloc(%zu bytes): injected failure", n * sizeof(T));
    cudaError_t e = cudaMalloc(&q, n * sizeof(T));
    if (e != cudaSuccess) {
      cudaGetLastError();
      return fail(RL_ERR_OOM, "cudaMalloc(%zu bytes): %s", n * sizeof(T), cudaGetErrorString(e));
    }
    e = cudaMemset(q, 0, n * sizeof(T));
    if (e != cudaSuccess) return fail(RL_ERR_CUDA, "cudaMemset: %s", cudaGetErrorString(e));
    allocs.push_back(q);
    *p = static_cast<T*>(q);
    return RL_OK;
  }
  ~rl_kv() {
    if (exec) cudaGraphExecDestroy(exec);
    if (graph) cudaGraphDestroy(graph);
    for (cudaEvent_t e : ev) cudaEventDestroy(e);
    for (void* p : allocs) cudaFree(p);
  }
};

namespace {

#define RL_TRY(expr)                  \
  do {                                \
    rl_status s_ = (expr);            \
    if (s_ != RL_OK) return s_;       \
  } while (0)

cudaStream_t as_stream(rl_stream_t s) { return static_cast<cudaStream_t>(s); }

// Internal row order of the fused QKV matrix: per head, 16-row tile j holds
// dims 8j..8j+7 and hd/2+8j..hd/2+8j+7, so each RoPE pair (i, i + hd/2)
// lands in one tile.  Source 0/1/2 = wq/wk/wv.
std::vector<int2> qkv_rowmap(int Hq, int Hkv, int hd) {
  std::vector<int2> m;
  const int heads = Hq + 2 * Hkv;
  for (int r = 0; r < heads * hd; ++r) {
    const int head = r / hd, i = r % hd, j = i / 16, rr = i % 16;
    const int dim = rr < 8 ? 8 * j + rr : hd / 2 + 8 * j + rr - 8;
    if (head < Hq)
      m.push_back(make_int2(0, head * hd + dim));
    else if (head < Hq + Hkv)
      m.push_back(make_int2(1, (head - Hq) * hd + dim));
    else
      m.push_back(make_int2(2, (head - Hq - Hkv) * hd + dim));
  }
  return m;
}

// Internal row order of the fused gate/up matrix: tile j = gate rows
// 8j..8j+7 then up rows 8j..8j+7 (SwiGLU pairs in one tile).
std::vector<int2> gu_rowmap(int F) {
  std::vector<int2> m;
  for (int r = 0; r < 2 * F; ++r) {
    const int j = r / 16, rr = r % 16;
    m.push_back(rr < 8 ? make_int2(0, 8 * j + rr) : make_int2(1, 8 * j + rr - 8));
  }
  return m;
}

rl_status upload_map(rl_model* m, const std::vector<int2>& h, int2** d) {
  RL_TRY(m->alloc(d, h.size()));
  RL_CUDA(cudaMemcpy(*d, h.data(), h.size() * sizeof(int2), cudaMemcpyHostToDevice));
  return RL_OK;
}

rl_status validate_config(const rl_config* c) {
  if (!c) return fail(RL_ERR_INVALID_ARG, "config is NULL");
  if (c->n_layers < 1 || c->d_model < 16 || c->n_q_heads < 1 || c->n_kv_heads < 1 ||
      c->ffn_dim < 8 || c->vocab < 16)
    return fail(RL_ERR_INVALID_ARG, "non-positive or too small dimension in config");
  if (c->head_dim != 64 && c->head_dim != 128)
    return fail(RL_ERR_UNSUPPORTED, "head_dim must be 64 or 128 (got %d)", c->head_dim);
  if (c->n_q_heads % c->n_kv_heads != 0 || c->n_q_heads / c->n_kv_heads > 8)
    return fail(RL_ERR_UNSUPPORTED, "n_q_heads must be a multiple (<= 8x) of n_kv_heads");
  if (c->d_model % 16 || c->ffn_dim % 8 || c->vocab % 16)
    return fail(RL_ERR_UNSUPPORTED, "d_model and vocab must be multiples of 16, ffn_dim of 8");
  if (c->d_model > 12288) return fail(RL_ERR_UNSUPPORTED, "d_model > 12288");
  if (c->group_size != kGroup) return fail(RL_ERR_UNSUPPORTED, "group_size must be 128");
  if (!(c->rms_eps > 0.f) || !(c->rope_theta > 0.f))
    return fail(RL_ERR_INVALID_ARG, "rms_eps and rope_theta must be positive");
  return RL_OK;
}

int decode_nchunks(const rl_model* m, int B, int Tmax) {
  int n = (2 * m->sm_count + B * m->Hkv - 1) / (B * m->Hkv);
  const int cap = (Tmax + 63) / 64;
  if (n > cap) n = cap;
  if (n > 64) n = 64;
  if (n < 1) n = 1;
  return n;
}

GemvArgs gemv_base(const rl_model* m, const Linear& lin, int w4_mode, const DevState* st,
                   int layer_no) {
  GemvArgs a;
  memset(&a, 0, sizeof(a));
  a.w = lin.w;
  a.qw = lin.qw;
  a.qtc = lin.qtc;
  a.sz = lin.sz;
  a.N = lin.N;
  a.Kp = lin.Kp;
  a.w4_mode = w4_mode;
  a.exit_layer = st ? &st->exit_layer : nullptr;
  a.layer_no = layer_no;
  return a;
}

struct StepIO {
  const int* tokens;
  int B, T;  // T = 1 for decode
  const rl_exit_policy* pol;
  float* logits;
  int* next;
  int* exit;
  float* min_cos;
  bool prefill;  // rows are B sequences of T prompt tokens at positions 0..T-1
};

// Event records around launches when the cache has profiling switched on.
struct Prof {
  rl_kv* kv;
  cudaStream_t s;
  bool on;
  int n = 0;
  void begin() {
    if (on && n < (int)kv->recs.size())
      cudaEventRecordWithFlags(kv->ev[2 * n], s, cudaEventRecordExternal);
  }
  int* slot() { return (on && n < (int)kv->recs.size()) ? kv->d_paths + n : nullptr; }
  void end(int kind, int layer, double bytes_bf, double bytes_w4, bool gemv, bool attn = false) {
    if (!on || n >= (int)kv->recs.size()) return;
    // External records become event-record nodes when the step is captured.
    cudaEventRecordWithFlags(kv->ev[2 * n + 1], s, cudaEventRecordExternal);
    ProfRec& r = kv->recs[n];
    r.kind = kind;
    r.layer = layer;
    r.gemv = gemv;
    r.attn = attn;
    r.bytes_bf = bytes_bf;
    r.bytes_w4 = bytes_w4;
    ++n;
  }
};

double bytes_bf16(const Linear& l) { return (double)l.N * l.K * 2.0; }
double bytes_w4(const Linear& l) {
  return (double)l.N * l.K / 2.0 + (double)l.N * ((l.K + kGroup - 1) / kGroup) * 4.0;
}

// Enqueue one full pass of the decode path (T == 1) or of the prefill
// (T > 1, buffers passed in `ws`).
struct Work {
  float* h[3];
  bf16 *x_attn, *x_ffn, *o, *u;
  float *xs_attn, *xs_ffn, *xs_o, *xs_u;
  float* q;
  float* part;
  int nchunks;
  float* cosbuf;
};

// Below this many tokens the GEMV's weight stream is the whole cost and the
// tensor-core GEMM gains nothing.
constexpr int kTcMinTokens = 16;

// One projection over a.B tokens: the bf16 weights on the tensor cores (or
// the GEMV for a few tokens), the exit river's W4 weights in the dequantising
// GEMV; which of the two runs is decided on the device.
rl_status project(const rl_model* m, rl_kv* kv, const CUtensorMap& tm, GemvArgs a, cudaStream_t s) {
  a.tc_ws = kv->tc_ws;
  a.tc_ws_floats = kv->tc_ws_floats;
  a.tc_ticket = kv->tc_ticket;
  a.tc_ticket_n = kv->tc_ticket_n;
  a.first_wait = kv->wait_limit;
  if (a.B >= kTcMinTokens) {
    // the tensor-core GEMM runs bf16 layers and, when the projection has
    // enough output tiles, the W4 exit-river layers (dequantised in shared
    // memory); otherwise the dequantising GEMV runs the W4 layers
    a.tc_w4 = a.qtc != nullptr && tc_gemm_runs_w4(a.N, a.B, m->sm_count);
    RL_CUDA(launch_gemm_tc(tm, a, m->sm_count, s));
    if (a.w4_mode == W4_OFF || a.tc_w4) return RL_OK;
    a.w4_only = 1;
  }
  launch_gemv(a, m->sm_count, s);
  RL_LAUNCHED();
  return RL_OK;
}

// An offloaded layer's [N][Kp] weights into the device staging buffer, unless
// the device-side exit state says the layer runs on the exit river.
rl_status stage_layer(const rl_model* m, rl_kv* kv, int l, int w4mode, cudaStream_t s) {
  const Layer& ly = m->layers[l];
  if (!ly.qkv.offloaded) return RL_OK;
  const int* ex = w4mode == W4_BY_LAYER ? &kv->st->exit_layer : nullptr;
  for (const Linear* lin : {&ly.qkv, &ly.o, &ly.gu, &ly.dn}) {
    launch_stage_weights(lin->w_host, const_cast<bf16*>(lin->w), (size_t)lin->N * lin->Kp * 2, ex, l + 1,
                         m->sm_count, s);
    RL_LAUNCHED();
  }
  return RL_OK;
}

rl_status enqueue_pass(rl_model* m, rl_kv* kv, const StepIO& io, const Work& w, cudaStream_t s) {
  const int L = m->L, d = m->d;
  Prof pf{kv, s, kv->profiling && !io.prefill};
  const bool prefill = io.prefill;
  const int T = io.T;
  const int M = prefill ? io.B * io.T : io.B;  // rows (tokens) in this pass
  const int Gd = m->Kd / kGroup, Go = m->Ko / kGroup, Gf = m->Kf / kGroup;
  const int w4mode = m->quantized ? W4_BY_LAYER : W4_OFF;
  const int mode = io.pol->mode;
  const float tau = io.pol->tau;

  RowNormArgs emb;
  memset(&emb, 0, sizeof(emb));
  emb.tokens = io.tokens;
  emb.embed = m->embed;
  emb.vocab = m->V;
  emb.h_out = w.h[0];
  emb.rows = M;
  emb.d = d;
  emb.g = m->layers[0].g_attn;
  emb.eps = m->cfg.rms_eps;
  emb.x = w.x_attn;
  emb.ldx = m->Kd;
  emb.xsum = w.xs_attn;
  emb.ldxs = Gd;
  emb.L = L;
  emb.mode = mode;
  emb.tau = tau;
  emb.st = kv->st;
  emb.schedule = io.pol->d_schedule;
  emb.schedule_len = io.pol->schedule_len > 0 ? io.pol->schedule_len : 1;
  emb.use_step_index = prefill ? 0 : 1;
  emb.trace = kv->trace;
  emb.trace_layer = 0;
  emb.trace_maxB = kv->maxB;
  emb.trace_T = prefill ? T : 0;
  pf.begin();
  launch_rownorm(emb, s);
  RL_LAUNCHED();
  pf.end(RL_K_EMBED, 0, 0, 0, false);

  int cur = 0;
  for (int l = 0; l < L; ++l) {
    const Layer& ly = m->layers[l];
    const int mid = (cur + 1) % 3, nxt = (cur + 2) % 3;
    RL_TRY(stage_layer(m, kv, l, w4mode, s));
    // QKV + RoPE + KV append
    {
      GemvArgs a = gemv_base(m, ly.qkv, w4mode, kv->st, l + 1);
      a.x = w.x_attn;
      a.ldx = m->Kd;
      a.xsum = w.xs_attn;
      a.ldxs = Gd;
      a.B = M;
      a.epi = EPI_QKV_ROPE;
      a.q_out = w.q;
      a.kc = kv->K[l];
      a.vc = kv->V[l];
      a.maxB = kv->maxB;
      a.Tmax = kv->Tmax;
      a.Hq = m->Hq;
      a.Hkv = m->Hkv;
      a.hd = m->hd;
      a.pos_ptr = &kv->st->pos;
      a.T_prefill = prefill ? T : 0;
      a.col_base = 0;
      a.inv_freq = m->inv_freq;
      a.rope_cs = kv->rope_cs;
      a.err = &kv->st->err;
      pf.begin();
      a.path_out = pf.slot();
      RL_TRY(project(m, kv, ly.qkv.tm, a, s));
      pf.end(RL_K_QKV, l + 1, bytes_bf16(ly.qkv), bytes_w4(ly.qkv), true);
    }
    // attention over the shared cache
    AttnArgs at;
    memset(&at, 0, sizeof(at));
    at.q = w.q;
    at.kc = kv->K[l];
    at.vc = kv->V[l];
    at.maxB = kv->maxB;
    at.Tmax = kv->Tmax;
    at.Hq = m->Hq;
    at.Hkv = m->Hkv;
    at.hd = m->hd;
    at.nq = M;
    at.T_prefill = prefill ? T : 0;
    at.pos_ptr = &kv->st->pos;
    at.nchunks = w.nchunks;
    at.part = w.part;
    at.o = w.o;
    at.ldo = m->Ko;
    pf.begin();
    if (prefill && kv->tm_ok && attn_prefill_supported(m->Hq / m->Hkv, m->hd)) {
      // the prompt: causal flash-style attention on the tensor cores
      AttnPrefillArgs ap;
      memset(&ap, 0, sizeof(ap));
      ap.tmk64 = kv->tmk64;
      ap.tmv64 = kv->tmv64;
      ap.layer_row0 = l * kv->maxB * m->Hkv * kv->Tmax;
      ap.q = w.q;
      ap.T = T;
      ap.Hq = m->Hq;
      ap.Hkv = m->Hkv;
      ap.Tmax = kv->Tmax;
      ap.nseq = io.B;
      ap.o = w.o;
      ap.ldo = m->Ko;
      ap.err = &kv->st->err;
      RL_CUDA(launch_attn_prefill(ap, m->Hq / m->Hkv, m->hd, s));
    } else if (prefill) {
      launch_attention(at, s);
    } else if (kv->tm_ok && attn_stream_supported(m->Hq / m->Hkv, m->hd)) {
      // decode: persistent CTAs stream the chunks (TMA ring, tensor cores),
      // then the chunks are merged
      at.nchunks = decode_attention_chunks(M, m->Hkv, kv->Tmax, m->sm_count);
      AttnStreamArgs as;
      memset(&as, 0, sizeof(as));
      as.tmk = kv->tmk;
      as.tmv = kv->tmv;
      as.tmk64 = kv->tmk64;
      as.tmv64 = kv->tmv64;
      as.layer_row0 = l * kv->maxB * m->Hkv * kv->Tmax;
      as.q = w.q;
      as.pos_ptr = &kv->st->pos;
      as.Tmax = kv->Tmax;
      as.Hq = m->Hq;
      as.Hkv = m->Hkv;
      as.nq = M;
      as.nchunks = at.nchunks;
      attn_stream_smem(&as.nslot);
      as.part = w.part;
      as.err = &kv->st->err;
      RL_CUDA(launch_attn_stream(as, m->Hq / m->Hkv, m->hd, m->sm_count, s));
      launch_attention_combine(at, s);
    } else {
      // decode: chunks of <= 128 positions staged in shared memory, the last
      // CTA of each (sequence, KV head) combines them (one launch)
      at.nchunks = decode_attention_chunks(M, m->Hkv, kv->Tmax, m->sm_count);
      at.ticket = kv->attn_ticket;
      RL_CUDA(launch_attention_fused(at, false, s));
    }
    RL_LAUNCHED();
    pf.end(RL_K_ATTN, l + 1, 0, 0, false, true);
    if (M <= kTcW4AllTokens) {  // the W4 GEMV's zero-point term needs the group sums
      pf.begin();
      launch_group_sums(w.o, m->Ko, m->Ko, M, w.xs_o, Go, s);
      RL_LAUNCHED();
      pf.end(RL_K_GSUM, l + 1, 0, 0, false);
    }
    // O projection + residual
    {
      GemvArgs a = gemv_base(m, ly.o, w4mode, kv->st, l + 1);
      a.x = w.o;
      a.ldx = m->Ko;
      a.xsum = w.xs_o;
      a.ldxs = Go;
      a.B = M;
      a.epi = EPI_RESID;
      a.out = w.h[mid];
      a.ldo = d;
      a.resid = w.h[cur];
      a.ldr = d;
      a.err = &kv->st->err;
      pf.begin();
      a.path_out = pf.slot();
      RL_TRY(project(m, kv, ly.o.tm, a, s));
      pf.end(RL_K_O, l + 1, bytes_bf16(ly.o), bytes_w4(ly.o), true);
    }
    // pre-FFN RMSNorm
    RowNormArgs n2;
    memset(&n2, 0, sizeof(n2));
    n2.h_out = w.h[mid];
    n2.rows = M;
    n2.d = d;
    n2.g = ly.g_ffn;
    n2.eps = m->cfg.rms_eps;
    n2.x = w.x_ffn;
    n2.ldx = m->Kd;
    n2.xsum = w.xs_ffn;
    n2.ldxs = Gd;
    n2.st = kv->st;
    pf.begin();
    launch_rownorm(n2, s);
    RL_LAUNCHED();
    pf.end(RL_K_NORM, l + 1, 0, 0, false);
    // gate/up + SwiGLU
    {
      GemvArgs a = gemv_base(m, ly.gu, w4mode, kv->st, l + 1);
      a.x = w.x_ffn;
      a.ldx = m->Kd;
      a.xsum = w.xs_ffn;
      a.ldxs = Gd;
      a.B = M;
      a.epi = EPI_SWIGLU;
      a.out_h = w.u;
      a.ldoh = m->Kf;
      a.err = &kv->st->err;
      pf.begin();
      a.path_out = pf.slot();
      RL_TRY(project(m, kv, ly.gu.tm, a, s));
      pf.end(RL_K_GU, l + 1, bytes_bf16(ly.gu), bytes_w4(ly.gu), true);
    }
    if (M <= kTcW4AllTokens) {
      pf.begin();
      launch_group_sums(w.u, m->Kf, m->Kf, M, w.xs_u, Gf, s);
      RL_LAUNCHED();
      pf.end(RL_K_GSUM, l + 1, 0, 0, false);
    }
    // down + residual
    {
      GemvArgs a = gemv_base(m, ly.dn, w4mode, kv->st, l + 1);
      a.x = w.u;
      a.ldx = m->Kf;
      a.xsum = w.xs_u;
      a.ldxs = Gf;
      a.B = M;
      a.epi = EPI_RESID;
      a.out = w.h[nxt];
      a.ldo = d;
      a.resid = w.h[mid];
      a.ldr = d;
      a.err = &kv->st->err;
      pf.begin();
      a.path_out = pf.slot();
      RL_TRY(project(m, kv, ly.dn.tm, a, s));
      pf.end(RL_K_DOWN, l + 1, bytes_bf16(ly.dn), bytes_w4(ly.dn), true);
    }
    // layer end: cosine, batch-min, tau compare, next RMSNorm
    RowNormArgs le;
    memset(&le, 0, sizeof(le));
    le.h_in = w.h[cur];
    le.h_out = w.h[nxt];
    le.rows = M;
    le.d = d;
    le.g = (l + 1 < L) ? m->layers[l + 1].g_attn : m->g_final;
    le.eps = m->cfg.rms_eps;
    le.x = w.x_attn;
    le.ldx = m->Kd;
    le.xsum = w.xs_attn;
    le.ldxs = Gd;
    le.cosbuf = w.cosbuf;
    le.layer_no = l + 1;
    le.L = L;
    le.mode = mode;
    le.tau = tau;
    le.min_cos_out = io.min_cos;
    le.exit_out = io.exit;
    le.st = kv->st;
    le.set_pos = prefill ? T : -1;
    le.set_step = prefill ? 0 : -1;
    le.trace = kv->trace;
    le.trace_layer = l + 1;
    le.trace_maxB = kv->maxB;
    le.trace_T = prefill ? T : 0;
    pf.begin();
    launch_rownorm(le, s);
    RL_LAUNCHED();
    pf.end(RL_K_LAYER_END, l + 1, 0, 0, false);
    cur = nxt;
  }
  // final RMSNorm was applied by the last layer end (gain g_final) into x_attn.
  {
    GemvArgs a = gemv_base(m, Linear(), W4_OFF, nullptr, 0);
    a.w = m->lm_head;
    a.N = m->V;
    a.Kp = m->Kd;
    const int last = prefill ? T - 1 : 0;
    const int stride = prefill ? T : 1;
    a.x = w.x_attn + (size_t)last * m->Kd;
    a.ldx = m->Kd * stride;
    a.B = io.B;
    a.epi = EPI_STORE;
    a.out = io.logits;
    a.ldo = m->V;
    a.err = &kv->st->err;
    pf.begin();
    a.path_out = pf.slot();
    RL_TRY(project(m, kv, m->tm_lm, a, s));
    const double lm = (double)m->V * m->d * 2.0;
    pf.end(RL_K_LM_HEAD, 0, lm, lm, true);
  }
  if (io.next) {
    pf.begin();
    launch_argmax(io.logits, m->V, m->V, io.B, io.next, s);
    RL_LAUNCHED();
    pf.end(RL_K_ARGMAX, 0, 0, 0, false);
  }
  if (pf.on) kv->nrec = pf.n;
  return RL_OK;
}

// Fused small-batch decode pass (B <= 8): five kernels per layer plus the
// LM head, chained with programmatic dependent launch.
rl_status enqueue_decode_fused(rl_model* m, rl_kv* kv, const StepIO& io, int nchunks,
                               cudaStream_t s) {
  const int L = m->L, d = m->d, B = io.B;
  Prof pf{kv, s, kv->profiling};
  const bool pdl = !pf.on;  // event records between kernels would break the programmatic edges
  const int w4mode = m->quantized ? W4_BY_LAYER : W4_OFF;
  const int tiles_d = d / 16;
  auto base = [&](const Linear& lin, int layer_no) {
    FusedArgs a;
    memset(&a, 0, sizeof(a));
    a.w = lin.w;
    a.qwt = lin.qwt;
    a.N = lin.N;
    a.Kp = lin.Kp;
    a.w4_mode = w4mode;
    a.layer_no = layer_no;
    a.st = kv->st;
    a.B = B;
    a.d = d;
    a.eps = m->cfg.rms_eps;
    a.L = L;
    a.mode = io.pol->mode;
    a.tau = io.pol->tau;
    a.schedule = io.pol->d_schedule;
    a.schedule_len = io.pol->schedule_len > 0 ? io.pol->schedule_len : 1;
    a.trace_maxB = kv->maxB;
    a.ws = kv->ws;
    a.tile_ticket = kv->tile_ticket;
    a.cta_ticket = kv->cta_ticket;
    return a;
  };
  int cur = 0;
  for (int l = 0; l < L; ++l) {
    const Layer& ly = m->layers[l];
    const int mid = (cur + 1) % 3, nxt = (cur + 2) % 3;
    RL_TRY(stage_layer(m, kv, l, w4mode, s));
    // QKV: exit decision of layer l (l >= 1), RMSNorm scale, projection, RoPE, KV append
    {
      FusedArgs a = base(ly.qkv, l + 1);
      if (l == 0) {
        a.xmode = X_EMBED;
        a.tokens = io.tokens;
        a.embed = m->embed;
        a.vocab = m->V;
        a.gain_embed = ly.g_attn;
        a.h_store = kv->h[0];
        a.step_begin = 1;
        a.trace = kv->trace;
        a.trace_layer = 0;
      } else {
        a.xmode = X_SCALED;
        a.xg = kv->x_attn;
        a.ldxg = m->Kd;
        a.stats_in = kv->st_end;
        a.stats_tiles = tiles_d;
        a.stats_k = 3;
        a.dec_layer = l;
        a.min_cos_out = io.min_cos;
      }
      a.epi = EPI_QKV_ROPE;
      a.q_out = kv->q;
      a.kc = kv->K[l];
      a.vc = kv->V[l];
      a.maxB = kv->maxB;
      a.Tmax = kv->Tmax;
      a.Hq = m->Hq;
      a.Hkv = m->Hkv;
      a.hd = m->hd;
      a.inv_freq = m->inv_freq;
      pf.begin();
      a.path_out = pf.slot();
      RL_CUDA(launch_gemv_fused(a, m->sm_count, pdl && l > 0, s));
      pf.end(RL_K_QKV, l + 1, bytes_bf16(ly.qkv), bytes_w4(ly.qkv), true);
    }
    {
      AttnArgs at;
      memset(&at, 0, sizeof(at));
      at.q = kv->q;
      at.kc = kv->K[l];
      at.vc = kv->V[l];
      at.maxB = kv->maxB;
      at.Tmax = kv->Tmax;
      at.Hq = m->Hq;
      at.Hkv = m->Hkv;
      at.hd = m->hd;
      at.nq = B;
      at.pos_ptr = &kv->st->pos;
      at.nchunks = nchunks;
      at.part = kv->part;
      at.o = kv->o;
      at.ldo = m->Ko;
      at.ticket = kv->attn_ticket;
      pf.begin();
      RL_CUDA(launch_attention_fused(at, pdl, s));
      pf.end(RL_K_ATTN, l + 1, 0, 0, false, true);
    }
    {  // O projection + residual; x' and |h_mid|^2 partials for the FFN norm
      FusedArgs a = base(ly.o, l + 1);
      a.xmode = X_COPY;
      a.xg = kv->o;
      a.ldxg = m->Ko;
      a.epi = EPI_RESID;
      a.out = kv->h[mid];
      a.ldo = d;
      a.resid = kv->h[cur];
      a.ldr = d;
      a.gnext = ly.g_ffn;
      a.xnext = kv->x_ffn;
      a.ldxnext = m->Kd;
      a.stats_out = kv->st_mid;
      a.stats_k_out = 1;
      pf.begin();
      a.path_out = pf.slot();
      RL_CUDA(launch_gemv_fused(a, m->sm_count, pdl, s));
      pf.end(RL_K_O, l + 1, bytes_bf16(ly.o), bytes_w4(ly.o), true);
    }
    {  // gate/up + SwiGLU
      FusedArgs a = base(ly.gu, l + 1);
      a.xmode = X_SCALED;
      a.xg = kv->x_ffn;
      a.ldxg = m->Kd;
      a.stats_in = kv->st_mid;
      a.stats_tiles = tiles_d;
      a.stats_k = 1;
      a.epi = EPI_SWIGLU;
      a.out_h = kv->u;
      a.ldoh = m->Kf;
      pf.begin();
      a.path_out = pf.slot();
      RL_CUDA(launch_gemv_fused(a, m->sm_count, pdl, s));
      pf.end(RL_K_GU, l + 1, bytes_bf16(ly.gu), bytes_w4(ly.gu), true);
    }
    {  // down + residual; x' and layer-end partials for the next layer
      FusedArgs a = base(ly.dn, l + 1);
      a.xmode = X_COPY;
      a.xg = kv->u;
      a.ldxg = m->Kf;
      a.epi = EPI_RESID;
      a.out = kv->h[nxt];
      a.ldo = d;
      a.resid = kv->h[mid];
      a.ldr = d;
      a.gnext = (l + 1 < L) ? m->layers[l + 1].g_attn : m->g_final;
      a.xnext = kv->x_attn;
      a.ldxnext = m->Kd;
      a.stats_out = kv->st_end;
      a.stats_k_out = 3;
      a.h_in = kv->h[cur];
      a.trace = kv->trace;
      a.trace_layer = l + 1;
      pf.begin();
      a.path_out = pf.slot();
      RL_CUDA(launch_gemv_fused(a, m->sm_count, pdl, s));
      pf.end(RL_K_DOWN, l + 1, bytes_bf16(ly.dn), bytes_w4(ly.dn), true);
    }
    cur = nxt;
  }
  {
    // LM head: min cosine of layer L, final RMSNorm scale, logits, argmax, end of step
    Linear lm;
    lm.w = m->lm_head;
    lm.N = m->V;
    lm.K = m->d;
    lm.Kp = m->Kd;
    FusedArgs a = base(lm, 0);
    a.w4_mode = W4_OFF;
    a.xmode = X_SCALED;
    a.xg = kv->x_attn;
    a.ldxg = m->Kd;
    a.stats_in = kv->st_end;
    a.stats_tiles = tiles_d;
    a.stats_k = 3;
    a.dec_layer = L;
    a.min_cos_out = io.min_cos;
    a.epi = EPI_LMHEAD;
    a.out = io.logits;
    a.ldo = m->V;
    a.am_val = kv->am_val;
    a.am_idx = kv->am_idx;
    a.next_token = io.next;
    a.exit_out = io.exit;
    pf.begin();
    a.path_out = pf.slot();
    RL_CUDA(launch_gemv_fused(a, m->sm_count, pdl, s));
    const double lmb = (double)m->V * m->d * 2.0;
    pf.end(RL_K_LM_HEAD, 0, lmb, lmb, true);
  }
  if (pf.on) kv->nrec = pf.n;
  return RL_OK;
}

// Zero the cross-CTA counters of the decode kernels (after an aborted step,
// or when the position is rewound).
rl_status reset_sync_words(rl_kv* kv, cudaStream_t s) {
  RL_CUDA(cudaMemsetAsync(kv->bars, 0, kv->n_bars * sizeof(unsigned), s));
  RL_CUDA(cudaMemsetAsync(kv->tctr, 0, (size_t)kv->nph_cap * sizeof(unsigned), s));
  RL_CUDA(cudaMemsetAsync(kv->tile_ticket, 0, (size_t)kv->n_tile_ticket * sizeof(unsigned), s));
  RL_CUDA(cudaMemsetAsync(kv->attn_ticket, 0, (size_t)kv->maxB * kv->m->Hkv * sizeof(unsigned), s));
  RL_CUDA(cudaMemsetAsync(kv->cta_ticket, 0, sizeof(unsigned), s));
  RL_CUDA(cudaMemsetAsync(kv->tc_ticket, 0, (size_t)kv->tc_ticket_n * sizeof(unsigned), s));
  return RL_OK;
}

// ---------------------------------------------------------------------------
// Persistent step kernel: phase descriptors, fit test, launch.
// ---------------------------------------------------------------------------
int step_kmax(const rl_model* m) { return std::max(std::max(m->Kd, m->Ko), m->Kf); }

// Tile scheduling of a projection with `ntiles` 16-row tiles over `grid`
// CTAs: claimed at run time from a shared counter when there are at least
// four tiles per CTA (the faster CTAs take more), else assigned round-robin.
int step_split(int ntiles, int upt, int grid) {
  (void)upt;
  return ntiles >= 4 * grid ? 1 : 0;
}

bool step_fits_model(const rl_model* m, int B) {
  if (!m->step_ok || B < 1 || B > kFusedMaxB || m->d % 16) return false;
  const int rep = m->Hq / m->Hkv;
  if ((rep != 1 && rep != 2 && rep != 4) || (m->hd != 64 && m->hd != 128)) return false;
  int ns = 0;
  const size_t smem = step_smem_bytes(B, step_kmax(m), step_kmax(m) / kGroup, &ns);
  return smem && decode_step_occupancy(smem) >= 1;
}

bool step_fits(const rl_model* m, const rl_kv* kv, int B) {
  if (!m->step_ok || !kv->tm_ok || !kv->part_s || B < 1 || B > kFusedMaxB || B > kv->maxB || m->d % 16)
    return false;
  const int rep = m->Hq / m->Hkv;
  if ((rep != 1 && rep != 2 && rep != 4) || (m->hd != 64 && m->hd != 128)) return false;
  if (6 * m->L + 1 > kv->nph_cap) return false;
  int ns = 0;
  const size_t smem = step_smem_bytes(B, step_kmax(m), step_kmax(m) / kGroup, &ns);
  if (!smem) return false;
  return decode_step_occupancy(smem) >= 1;
}

bool fused_fits(const rl_model* m, int B);

// The kernels a decode step of batch B runs: the persistent step kernel, the
// fused five-launches-per-layer path, or the generic path (any batch); -1
// when the path the cache was told to use cannot run this batch.
int decode_path(const rl_model* m, const rl_kv* kv, int B) {
  const bool step = kv->use_step && step_fits(m, kv, B);
  const bool fused = kv->use_fused && fused_fits(m, B);
  switch (kv->path_pref) {
    case RL_PATH_STEP: return step ? RL_PATH_STEP : -1;
    case RL_PATH_FUSED: return fused ? RL_PATH_FUSED : -1;
    case RL_PATH_GENERIC: return RL_PATH_GENERIC;
    default: return step ? RL_PATH_STEP : (fused ? RL_PATH_FUSED : RL_PATH_GENERIC);
  }
}

std::vector<PhaseDesc> build_step_phases(rl_model* m, rl_kv* kv, const StepIO& io) {
  const int L = m->L, d = m->d, grid = m->sm_count;
  const int tiles_d = d / 16;
  std::vector<PhaseDesc> ph;
  auto gemv = [&](const Linear& lin, int layer_no) {
    PhaseDesc p;
    memset(&p, 0, sizeof(p));
    p.kind = PH_GEMV;
    p.layer_no = layer_no;
    p.wt = lin.wt;
    p.wt_sys = lin.offloaded ? 1 : 0;
    p.qwt = m->quantized ? lin.qwt : nullptr;
    p.N = lin.N;
    p.Kp = lin.Kp;
    p.split = step_split(lin.N / 16, (lin.Kp + 1023) / 1024, grid);
    return p;
  };
  int cur = 0;
  for (int l = 0; l < L; ++l) {
    const Layer& ly = m->layers[l];
    const int mid = (cur + 1) % 3, nxt = (cur + 2) % 3;
    {  // QKV: exit decision of layer l, RMSNorm scale, projection, RoPE, KV append
      PhaseDesc p = gemv(ly.qkv, l + 1);
      if (l == 0) {
        p.xmode = X_EMBED;
        p.trace = kv->trace;
        p.trace_layer = 0;
      } else {
        p.xmode = X_SCALED;
        p.xg = kv->x_attn;
        p.ldxg = m->Kd;
        p.stats_in = kv->st_end;
        p.stats_tiles = tiles_d;
        p.stats_k = 3;
        p.dec_layer = l;
      }
      p.epi = EPI_QKV_ROPE;
      p.q_out = kv->q;
      p.kc = kv->K[l];
      p.vc = kv->V[l];
      ph.push_back(p);
    }
    {  // attention
      PhaseDesc p;
      memset(&p, 0, sizeof(p));
      p.kind = PH_ATTN;
      p.layer_no = l + 1;
      p.q_out = kv->q;
      p.kc = kv->K[l];
      p.vc = kv->V[l];
      p.o_out = kv->o;
      p.ldo_attn = m->Ko;
      ph.push_back(p);  // the last CTA of each (sequence, KV head) merges its chunks
    }
    {  // O + residual; x' and |h_mid|^2 partials for the FFN norm
      PhaseDesc p = gemv(ly.o, l + 1);
      p.xmode = X_COPY;
      p.xg = kv->o;
      p.ldxg = m->Ko;
      p.epi = EPI_RESID;
      p.out = kv->h[mid];
      p.ldo = d;
      p.resid = kv->h[cur];
      p.ldr = d;
      p.gnext = ly.g_ffn;
      p.xnext = kv->x_ffn;
      p.ldxnext = m->Kd;
      p.stats_out = kv->st_mid;
      p.stats_k_out = 1;
      ph.push_back(p);
    }
    {  // gate/up + SwiGLU
      PhaseDesc p = gemv(ly.gu, l + 1);
      p.xmode = X_SCALED;
      p.xg = kv->x_ffn;
      p.ldxg = m->Kd;
      p.stats_in = kv->st_mid;
      p.stats_tiles = tiles_d;
      p.stats_k = 1;
      p.epi = EPI_SWIGLU;
      p.out_h = kv->u;
      p.ldoh = m->Kf;
      ph.push_back(p);
    }
    {  // down + residual; x' and layer-end partials for the next layer
      PhaseDesc p = gemv(ly.dn, l + 1);
      p.xmode = X_COPY;
      p.xg = kv->u;
      p.ldxg = m->Kf;
      p.epi = EPI_RESID;
      p.out = kv->h[nxt];
      p.ldo = d;
      p.resid = kv->h[mid];
      p.ldr = d;
      p.gnext = (l + 1 < L) ? m->layers[l + 1].g_attn : m->g_final;
      p.xnext = kv->x_attn;
      p.ldxnext = m->Kd;
      p.stats_out = kv->st_end;
      p.stats_k_out = 3;
      p.h_in = kv->h[cur];
      p.trace = kv->trace;
      p.trace_layer = l + 1;
      ph.push_back(p);
    }
    cur = nxt;
  }
  {  // LM head: min cosine of layer L, final RMSNorm scale, logits, argmax
    Linear lm;
    lm.wt = m->lm_head_t;
    lm.N = m->V;
    lm.K = m->d;
    lm.Kp = m->Kd;
    PhaseDesc p = gemv(lm, 0);
    p.qwt = nullptr;
    p.split = 0;
    p.xmode = X_SCALED;
    p.xg = kv->x_attn;
    p.ldxg = m->Kd;
    p.stats_in = kv->st_end;
    p.stats_tiles = tiles_d;
    p.stats_k = 3;
    p.dec_layer = L;
    p.epi = EPI_LMHEAD;
    p.out = io.logits;
    p.ldo = m->V;
    ph.push_back(p);
  }
  return ph;
}

// Make the device descriptors match this call (synchronously, outside any
// capture; waits for earlier work on `s` that may still read them).
rl_status prepare_step_phases(rl_model* m, rl_kv* kv, const StepIO& io, cudaStream_t s) {
  std::vector<PhaseDesc> ph = build_step_phases(m, kv, io);
  if ((int)ph.size() > kv->nph_cap) return fail(RL_ERR_UNSUPPORTED, "too many phases");
  if (ph.size() == kv->h_ph.size() && memcmp(ph.data(), kv->h_ph.data(), ph.size() * sizeof(PhaseDesc)) == 0)
    return RL_OK;
  RL_CUDA(cudaStreamSynchronize(s));
  RL_CUDA(cudaMemcpy(kv->d_ph, ph.data(), ph.size() * sizeof(PhaseDesc), cudaMemcpyHostToDevice));
  kv->h_ph.swap(ph);
  return RL_OK;
}

rl_status enqueue_decode_step(rl_model* m, rl_kv* kv, const StepIO& io, cudaStream_t s) {
  const int B = io.B;
  StepArgs a;
  memset(&a, 0, sizeof(a));
  a.ph = kv->d_ph;
  a.nph = (int)kv->h_ph.size();
  a.st = kv->st;
  a.B = B;
  a.L = m->L;
  a.d = m->d;
  a.Hq = m->Hq;
  a.Hkv = m->Hkv;
  a.hd = m->hd;
  a.Tmax = kv->Tmax;
  a.vocab = m->V;
  a.eps = m->cfg.rms_eps;
  a.mode = io.pol->mode;
  a.tau = io.pol->tau;
  a.schedule = io.pol->d_schedule;
  a.schedule_len = io.pol->schedule_len > 0 ? io.pol->schedule_len : 1;
  a.tokens = io.tokens;
  a.embed = m->embed;
  a.gain_embed = m->layers[0].g_attn;
  a.h_store = kv->h[0];
  a.trace_maxB = kv->maxB;
  a.inv_freq = m->inv_freq;
  a.min_cos_out = io.min_cos;
  a.next_token = io.next;
  a.exit_out = io.exit;
  a.am_val = kv->am_val;
  a.am_idx = kv->am_idx;
  a.cta_ticket = kv->cta_ticket;
  a.bars = kv->bars;
  a.tctr = kv->tctr;
  a.ws = kv->ws;
  a.tile_ticket = kv->tile_ticket;
  a.part = kv->part_s;
  a.attn_ticket = kv->attn_ticket;
  a.part_cap = kv->part_cap;
  a.rope_cs = kv->rope_cs;
  a.tmk = kv->tmk;
  a.tmv = kv->tmv;
  a.kv_rows_layer = kv->maxB * m->Hkv * kv->Tmax;
  a.xs_row_bytes = step_kmax(m) * 2 + 64;
  a.gmax = step_kmax(m) / kGroup;
  a.bar_wait = kv->wait_limit;
  const size_t smem = step_smem_bytes(B, step_kmax(m), a.gmax, &a.nslot);
  if (!smem) return fail(RL_ERR_UNSUPPORTED, "step kernel does not fit");
  const bool prof = kv->profiling;
  if (prof) {
    a.tl = kv->tl;
    RL_CUDA(cudaMemsetAsync(kv->tl, 0xff, (size_t)a.nph * 8, s));
    RL_CUDA(cudaMemsetAsync(kv->tl + a.nph, 0, (size_t)a.nph * 8, s));
    if (kv->timeline) {
      a.tl2 = kv->tl2;
      RL_CUDA(cudaMemsetAsync(kv->tl2, 0, (size_t)a.nph * m->sm_count * kTl2 * 8, s));
    }
    cudaEventRecordWithFlags(kv->ev[0], s, cudaEventRecordExternal);
  }
  kv->step_args = a;
  // a CTA may take more than one attention chunk once B x KV heads x
  // 128-position chunks of the cache's longest context exceed the grid
  const bool multi = (long long)B * m->Hkv * ((kv->Tmax + 127) / 128) > m->sm_count;
  RL_CUDA(launch_decode_step(a, m->sm_count, smem, multi, m->offload_from >= 0, s));
  if (prof) {
    cudaEventRecordWithFlags(kv->ev[1], s, cudaEventRecordExternal);
    kv->nph_last = a.nph;
    kv->nrec = -1;  // marks a step-kernel profile
  }
  return RL_OK;
}

// The fused path holds each projection's activations in shared memory.
bool fused_fits(const rl_model* m, int B) {
  if (B > kFusedMaxB || m->d % 16) return false;
  FusedArgs a;
  memset(&a, 0, sizeof(a));
  a.B = B;
  const int kps[3] = {m->Kd, m->Ko, m->Kf};
  for (int kp : kps) {
    a.Kp = kp;
    if (fused_smem_bytes(a) > 220 * 1024) return false;
  }
  return true;
}

Work decode_work(rl_kv* kv, int B) {
  Work w;
  for (int i = 0; i < 3; ++i) w.h[i] = kv->h[i];
  w.x_attn = kv->x_attn;
  w.x_ffn = kv->x_ffn;
  w.o = kv->o;
  w.u = kv->u;
  w.xs_attn = kv->xs_attn;
  w.xs_ffn = kv->xs_ffn;
  w.xs_o = kv->xs_o;
  w.xs_u = kv->xs_u;
  w.q = kv->q;
  w.part = kv->part;
  w.nchunks = decode_nchunks(kv->m, B, kv->Tmax);
  w.cosbuf = kv->cosbuf;
  return w;
}

rl_status check_policy(const rl_model* m, const rl_exit_policy* p) {
  if (!p) return fail(RL_ERR_INVALID_ARG, "policy is NULL");
  if (p->mode == RL_EXIT_TAU) {
    if (!(p->tau == p->tau)) return fail(RL_ERR_INVALID_ARG, "tau is NaN");
    if (p->tau <= 1.0f && !m->quantized)
      return fail(RL_ERR_STATE, "tau <= 1 can exit: call rl_quantize_exit_layers first");
    return RL_OK;
  }
  if (p->mode == RL_EXIT_FORCED) {
    if (!p->d_schedule || p->schedule_len < 1)
      return fail(RL_ERR_INVALID_ARG, "forced policy needs d_schedule and schedule_len >= 1");
    if (!m->quantized)
      return fail(RL_ERR_STATE, "forced exits need the exit river: call rl_quantize_exit_layers");
    return RL_OK;
  }
  return fail(RL_ERR_INVALID_ARG, "unknown policy mode %d", p->mode);
}

bool is_capturable(cudaStream_t s) {
  return s != nullptr && s != cudaStreamLegacy && s != cudaStreamPerThread;
}

}  // namespace

extern "C" {

const char* rl_version(void) { return "libriver 0.1 (sm_103a)"; }

const char* rl_last_error(void) { return g_err.c_str(); }

rl_status rl_model_create(const rl_config* cfg, const rl_weights* wts, rl_stream_t stream,
                          rl_model** out) {
  if (!out) return fail(RL_ERR_INVALID_ARG, "out is NULL");
  *out = nullptr;
  RL_TRY(validate_config(cfg));
  if (!wts || !wts->embed || !wts->lm_head || !wts->g_final || !wts->layers)
    return fail(RL_ERR_INVALID_ARG, "weights: NULL pointer");
  for (int l = 0; l < cfg->n_layers; ++l) {
    const rl_layer_weights& lw = wts->layers[l];
    if (!lw.wq || !lw.wk || !lw.wv || !lw.wo || !lw.wg || !lw.wu || !lw.wd || !lw.g_attn || !lw.g_ffn)
      return fail(RL_ERR_INVALID_ARG, "weights of layer %d: NULL pointer", l);
  }
  cudaStream_t s = as_stream(stream);
  rl_model* m = new rl_model();
  m->cfg = *cfg;
  m->L = cfg->n_layers;
  m->d = cfg->d_model;
  m->Hq = cfg->n_q_heads;
  m->Hkv = cfg->n_kv_heads;
  m->hd = cfg->head_dim;
  m->F = cfg->ffn_dim;
  m->V = cfg->vocab;
  m->Kd = round_up(m->d, kGroup);
  m->Ko = round_up(m->Hq * m->hd, kGroup);
  m->Kf = round_up(m->F, kGroup);
  m->Nqkv = (m->Hq + 2 * m->Hkv) * m->hd;
  int dev = 0;
  cudaGetDevice(&dev);
  cudaDeviceGetAttribute(&m->sm_count, cudaDevAttrMultiProcessorCount, dev);
  if (m->sm_count < 1) m->sm_count = 1;
  gemv_fused_setup();
  attention_setup();
  attn_stream_setup();
  decode_step_setup();
  if (!tc_gemm_available()) {
    delete m;
    return fail(RL_ERR_CUDA, "the driver does not export cuTensorMapEncodeTiled");
  }
  {
    cudaError_t e = tc_gemm_init();
    if (e != cudaSuccess) {
      delete m;
      return fail(RL_ERR_CUDA, "tensor-core GEMM setup: %s", cudaGetErrorString(e));
    }
  }
  {
    int coop = 0;
    cudaDeviceGetAttribute(&coop, cudaDevAttrCooperativeLaunch, dev);
    // one consumer thread per CTA polls that CTA's phase flag: grid <= 256
    m->step_ok = coop != 0 && m->sm_count <= 256;
  }

  auto bail = [&](rl_status st) {
    delete m;
    return st;
  };
#define M_TRY(expr)                     \
  do {                                  \
    rl_status s_ = (expr);              \
    if (s_ != RL_OK) return bail(s_);   \
  } while (0)
#define M_CUDA(call)                                                                      \
  do {                                                                                    \
    cudaError_t e_ = (call);                                                              \
    if (e_ != cudaSuccess)                                                                \
      return bail(fail(RL_ERR_CUDA, "%s: %s", #call, cudaGetErrorString(e_)));            \
  } while (0)

  M_TRY(upload_map(m, qkv_rowmap(m->Hq, m->Hkv, m->hd), &m->map_qkv));
  M_TRY(upload_map(m, gu_rowmap(m->F), &m->map_gu));
  {
    const int n = std::max(m->d, m->V);
    std::vector<int2> id(n);
    for (int i = 0; i < n; ++i) id[i] = make_int2(0, i);
    M_TRY(upload_map(m, id, &m->map_id));
  }

  auto make_linear = [&](Linear& lin, int N, int K, int view_base, const int2* map,
                         GatherSrcs src) -> rl_status {
    lin.N = N;
    lin.K = K;
    lin.Kp = round_up(K, kGroup);
    lin.view_base = view_base;
    lin.rowmap = map;
    RL_TRY(m->alloc(&lin.w, (size_t)N * lin.Kp));
    launch_gather_rows(lin.w, lin.Kp, N, K, map, src, K, s);
    RL_LAUNCHED();
    if (!make_weight_tmap(&lin.tm, lin.w, N, lin.Kp))
      return fail(RL_ERR_CUDA, "tensor map of a %d x %d weight could not be encoded", N, lin.Kp);
    RL_TRY(m->alloc(&lin.wt, (size_t)N * lin.Kp));
    launch_bf16_tile_layout(lin.w, N, lin.Kp, lin.wt, s);
    RL_LAUNCHED();
    return RL_OK;
  };

  m->layers.resize(m->L);
  for (int l = 0; l < m->L; ++l) {
    const rl_layer_weights& lw = wts->layers[l];
    Layer& ly = m->layers[l];
    GatherSrcs qkv = {{(const bf16*)lw.wq, (const bf16*)lw.wk, (const bf16*)lw.wv}};
    GatherSrcs o = {{(const bf16*)lw.wo, nullptr, nullptr}};
    GatherSrcs gu = {{(const bf16*)lw.wg, (const bf16*)lw.wu, nullptr}};
    GatherSrcs dn = {{(const bf16*)lw.wd, nullptr, nullptr}};
    M_TRY(make_linear(ly.qkv, m->Nqkv, m->d, RL_WQ, m->map_qkv, qkv));
    M_TRY(make_linear(ly.o, m->d, m->Hq * m->hd, RL_WO, m->map_id, o));
    M_TRY(make_linear(ly.gu, 2 * m->F, m->d, RL_WG, m->map_gu, gu));
    M_TRY(make_linear(ly.dn, m->d, m->F, RL_WD, m->map_id, dn));
    M_TRY(m->alloc(&ly.g_attn, m->d));
    M_TRY(m->alloc(&ly.g_ffn, m->d));
    launch_bf16_to_f32((const bf16*)lw.g_attn, ly.g_attn, m->d, s);
    launch_bf16_to_f32((const bf16*)lw.g_ffn, ly.g_ffn, m->d, s);
  }
  M_TRY(m->alloc(&m->embed, (size_t)m->V * m->d));
  M_CUDA(cudaMemcpyAsync(m->embed, wts->embed, (size_t)m->V * m->d * sizeof(bf16),
                         cudaMemcpyDeviceToDevice, s));
  M_TRY(m->alloc(&m->lm_head, (size_t)m->V * m->Kd));
  launch_gather_rows(m->lm_head, m->Kd, m->V, m->d, m->map_id,
                     GatherSrcs{{(const bf16*)wts->lm_head, nullptr, nullptr}}, m->d, s);
  if (!make_weight_tmap(&m->tm_lm, m->lm_head, m->V, m->Kd))
    return bail(fail(RL_ERR_CUDA, "tensor map of the LM head could not be encoded"));
  M_TRY(m->alloc(&m->lm_head_t, (size_t)m->V * m->Kd));
  launch_bf16_tile_layout(m->lm_head, m->V, m->Kd, m->lm_head_t, s);
  M_TRY(m->alloc(&m->g_final, m->d));
  launch_bf16_to_f32((const bf16*)wts->g_final, m->g_final, m->d, s);
  {
    std::vector<float> inv(m->hd / 2);
    for (int i = 0; i < m->hd / 2; ++i)
      inv[i] = (float)std::pow((double)m->cfg.rope_theta, -2.0 * i / (double)m->hd);
    M_TRY(m->alloc(&m->inv_freq, inv.size()));
    M_CUDA(cudaMemcpyAsync(m->inv_freq, inv.data(), inv.size() * sizeof(float),
                           cudaMemcpyHostToDevice, s));
  }
  M_CUDA(cudaGetLastError());
  M_CUDA(cudaStreamSynchronize(s));
#undef M_TRY
#undef M_CUDA
  *out = m;
  return RL_OK;
}

void rl_model_destroy(rl_model* m) { delete m; }

}  // extern "C"

namespace {

// Device storage of the exit river: the interchange views (original row
// order) and, per fused matrix, the W4 layout; `fill` writes them (the
// quantizer, or the views uploaded from a file), then the unit-tiled copies.
template <typename Fill>
rl_status build_exit_river_allocs(rl_model* m, cudaStream_t s, Fill fill);

// Builds the exit river; on any failure every allocation it made is released
// and the model is left as it was (no exit river).
template <typename Fill>
rl_status build_exit_river(rl_model* m, cudaStream_t s, Fill fill) {
  const size_t mark = m->allocs.size();
  const size_t bytes0 = m->bytes;
  const rl_status st = build_exit_river_allocs(m, s, fill);
  if (st == RL_OK) return RL_OK;
  cudaStreamSynchronize(s);  // nothing enqueued may still use what is freed
  cudaGetLastError();
  for (size_t i = mark; i < m->allocs.size(); ++i) cudaFree(m->allocs[i]);
  m->allocs.resize(mark);
  m->bytes = bytes0;
  m->views.clear();
  m->d_views = nullptr;
  for (Layer& ly : m->layers)
    for (Linear* lin : {&ly.qkv, &ly.o, &ly.gu, &ly.dn}) {
      lin->qw = nullptr;
      lin->sz = nullptr;
      lin->qwt = nullptr;
      lin->qtc = nullptr;
    }
  m->quantized = false;
  return st;
}

template <typename Fill>
rl_status build_exit_river_allocs(rl_model* m, cudaStream_t s, Fill fill) {
  const int L = m->L;
  m->views.assign((size_t)L * 7, NSView{});
  const int outs[7] = {m->Hq * m->hd, m->Hkv * m->hd, m->Hkv * m->hd, m->d, m->F, m->F, m->d};
  const int ins[7] = {m->d, m->d, m->d, m->Hq * m->hd, m->d, m->d, m->F};
  for (int l = 0; l < L; ++l)
    for (int i = 0; i < 7; ++i) {
      NSView& v = m->views[(size_t)l * 7 + i];
      v.N = outs[i];
      v.K = ins[i];
      const int G = (ins[i] + kGroup - 1) / kGroup;
      RL_TRY(m->alloc(&v.q, (size_t)v.N * (v.K / 8)));
      RL_TRY(m->alloc(&v.s, (size_t)v.N * G));
      RL_TRY(m->alloc(&v.z, (size_t)v.N * G));
    }
  RL_TRY(m->alloc(&m->d_views, m->views.size()));
  RL_CUDA(cudaMemcpyAsync(m->d_views, m->views.data(), m->views.size() * sizeof(NSView),
                          cudaMemcpyHostToDevice, s));
  for (int l = 0; l < L; ++l) {
    Layer& ly = m->layers[l];
    Linear* lins[4] = {&ly.qkv, &ly.o, &ly.gu, &ly.dn};
    for (Linear* lin : lins) {
      RL_TRY(m->alloc(&lin->qw, (size_t)lin->N * (lin->Kp / 8)));
      RL_TRY(m->alloc(&lin->sz, (size_t)lin->N * (lin->Kp / kGroup)));
    }
  }
  RL_TRY(fill());
  for (int l = 0; l < L; ++l) {
    Layer& ly = m->layers[l];
    Linear* lins[4] = {&ly.qkv, &ly.o, &ly.gu, &ly.dn};
    for (Linear* lin : lins) {
      RL_TRY(m->alloc(&lin->qwt, w4_tiled_bytes(lin->N, lin->Kp)));
      launch_w4_tile_layout(lin->qw, lin->sz, lin->N, lin->Kp, lin->qwt, s);
      RL_LAUNCHED();
      RL_TRY(m->alloc(&lin->qtc, w4_tc_bytes(lin->N, lin->Kp)));
      launch_w4_tc_layout(lin->qw, lin->sz, lin->N, lin->Kp, lin->qtc, s);
      RL_LAUNCHED();
    }
  }
  RL_CUDA(cudaStreamSynchronize(s));
  m->quantized = true;
  return RL_OK;
}

constexpr char kExitMagic[8] = {'R', 'L', 'W', '4', 'E', 'X', 'I', 'T'};
constexpr uint32_t kExitVersion = 1;

void exit_header(const rl_model* m, uint32_t (&h)[8]) {
  const uint32_t v[8] = {kExitVersion, (uint32_t)m->L, (uint32_t)m->d, (uint32_t)m->Hq,
                         (uint32_t)m->Hkv, (uint32_t)m->hd, (uint32_t)m->F, (uint32_t)kGroup};
  for (int i = 0; i < 8; ++i) h[i] = v[i];
}

}  // namespace

extern "C" {

}  // extern "C"

namespace {

rl_status quantize_exit_river(rl_model* m, const HqqParams* hqq, cudaStream_t s) {
  return build_exit_river(m, s, [&]() -> rl_status {
    for (int l = 0; l < m->L; ++l) {
      Layer& ly = m->layers[l];
      Linear* lins[4] = {&ly.qkv, &ly.o, &ly.gu, &ly.dn};
      for (Linear* lin : lins) {
        launch_quantize(lin->w, lin->N, lin->K, lin->Kp, lin->qw, lin->sz, lin->rowmap,
                        m->d_views + (size_t)l * 7 + lin->view_base, hqq, s);
        RL_LAUNCHED();
      }
    }
    return RL_OK;
  });
}

}  // namespace

extern "C" {

rl_status rl_quantize_exit_layers(rl_model* m, rl_stream_t stream) {
  if (!m) return fail(RL_ERR_INVALID_ARG, "model is NULL");
  if (m->quantized) return RL_OK;
  return quantize_exit_river(m, nullptr, as_stream(stream));
}

rl_status rl_quantize_exit_layers_hqq(rl_model* m, int32_t iters, double lp_norm, double beta,
                                      double kappa, rl_stream_t stream) {
  if (!m) return fail(RL_ERR_INVALID_ARG, "model is NULL");
  if (iters < 0 || iters > 1000 || !(lp_norm > 0.0 && lp_norm <= 2.0) || !(beta > 0.0) ||
      !(kappa >= 1.0) || !(kappa < 1e3))
    return fail(RL_ERR_INVALID_ARG,
                "HQQ settings: iters in [0, 1000], lp_norm in (0, 2], beta > 0, kappa in [1, 1000)");
  if (m->quantized) return fail(RL_ERR_STATE, "the exit river is already built");
  HqqParams hp;
  hp.iters = iters;
  hp.p = lp_norm;
  hp.beta = beta;
  hp.kappa = kappa;
  return quantize_exit_river(m, &hp, as_stream(stream));
}

rl_status rl_exit_kv_cosine(const rl_model* m, int32_t layer, const float* d_h, int32_t B,
                            float* d_cos, rl_stream_t stream) {
  if (!m || !d_h || !d_cos) return fail(RL_ERR_INVALID_ARG, "NULL argument");
  if (layer < 0 || layer >= m->L) return fail(RL_ERR_INVALID_ARG, "layer %d outside [0, %d)", layer, m->L);
  if (B < 1 || B > 65535 / (2 * m->Hkv)) return fail(RL_ERR_INVALID_ARG, "B=%d out of range", B);
  if (!m->quantized) return fail(RL_ERR_STATE, "exit river not built");
  const Linear& q = m->layers[layer].qkv;
  // an offloaded layer's weights are read from host memory (plain loads)
  RL_CUDA(launch_exit_kv_cosine(d_h, B, m->d, m->layers[layer].g_attn, q.offloaded ? q.w_host : q.w, q.qw,
                                q.sz, q.Kp, m->Hq, m->Hkv, m->hd, d_cos, as_stream(stream)));
  return RL_OK;
}

rl_status rl_save_exit_layers(const rl_model* m, const char* path) {
  if (!m || !path) return fail(RL_ERR_INVALID_ARG, "NULL argument");
  if (!m->quantized) return fail(RL_ERR_STATE, "exit river not built");
  FILE* f = fopen(path, "wb");
  if (!f) return fail(RL_ERR_INVALID_ARG, "cannot open %s for writing", path);
  uint32_t h[8];
  exit_header(m, h);
  bool ok = fwrite(kExitMagic, 1, 8, f) == 8 && fwrite(h, 4, 8, f) == 8;
  std::vector<uint32_t> q;
  std::vector<uint16_t> sc, zr;
  for (size_t i = 0; ok && i < m->views.size(); ++i) {
    const NSView& v = m->views[i];
    const size_t nq = (size_t)v.N * (v.K / 8), ng = (size_t)v.N * ((v.K + kGroup - 1) / kGroup);
    q.resize(nq);
    sc.resize(ng);
    zr.resize(ng);
    if (cudaMemcpy(q.data(), v.q, nq * 4, cudaMemcpyDeviceToHost) != cudaSuccess ||
        cudaMemcpy(sc.data(), v.s, ng * 2, cudaMemcpyDeviceToHost) != cudaSuccess ||
        cudaMemcpy(zr.data(), v.z, ng * 2, cudaMemcpyDeviceToHost) != cudaSuccess) {
      fclose(f);
      return fail(RL_ERR_CUDA, "copying the exit river to the host failed");
    }
    const uint32_t nk[2] = {(uint32_t)v.N, (uint32_t)v.K};
    ok = fwrite(nk, 4, 2, f) == 2 && fwrite(q.data(), 4, nq, f) == nq && fwrite(sc.data(), 2, ng, f) == ng &&
         fwrite(zr.data(), 2, ng, f) == ng;
  }
  ok = (fclose(f) == 0) && ok;
  if (!ok) return fail(RL_ERR_INVALID_ARG, "writing %s failed", path);
  return RL_OK;
}

rl_status rl_load_exit_layers(rl_model* m, const char* path, rl_stream_t stream) {
  if (!m || !path) return fail(RL_ERR_INVALID_ARG, "NULL argument");
  if (m->quantized) return fail(RL_ERR_STATE, "exit river already built");
  // read and check the whole file on the host first: a bad file leaves the model unchanged
  FILE* f = fopen(path, "rb");
  if (!f) return fail(RL_ERR_INVALID_ARG, "cannot open %s", path);
  char magic[8];
  uint32_t h[8], want[8];
  exit_header(m, want);
  bool ok = fread(magic, 1, 8, f) == 8 && memcmp(magic, kExitMagic, 8) == 0 && fread(h, 4, 8, f) == 8 &&
            memcmp(h, want, sizeof(h)) == 0;
  if (!ok) {
    fclose(f);
    return fail(RL_ERR_INVALID_ARG, "%s is not an exit river of this model's shape", path);
  }
  const int L = m->L;
  const int outs[7] = {m->Hq * m->hd, m->Hkv * m->hd, m->Hkv * m->hd, m->d, m->F, m->F, m->d};
  const int ins[7] = {m->d, m->d, m->d, m->Hq * m->hd, m->d, m->d, m->F};
  std::vector<std::vector<uint32_t>> q((size_t)L * 7);
  std::vector<std::vector<uint16_t>> sc((size_t)L * 7), zr((size_t)L * 7);
  for (int i = 0; ok && i < L * 7; ++i) {
    uint32_t nk[2];
    const int N = outs[i % 7], K = ins[i % 7];
    ok = fread(nk, 4, 2, f) == 2 && nk[0] == (uint32_t)N && nk[1] == (uint32_t)K;
    if (!ok) break;
    const size_t nq = (size_t)N * (K / 8), ng = (size_t)N * ((K + kGroup - 1) / kGroup);
    q[i].resize(nq);
    sc[i].resize(ng);
    zr[i].resize(ng);
    ok = fread(q[i].data(), 4, nq, f) == nq && fread(sc[i].data(), 2, ng, f) == ng &&
         fread(zr[i].data(), 2, ng, f) == ng;
  }
  char extra;
  ok = ok && fread(&extra, 1, 1, f) == 0;  // nothing may follow
  fclose(f);
  if (!ok) return fail(RL_ERR_INVALID_ARG, "%s is truncated or does not match the model", path);
  cudaStream_t s = as_stream(stream);
  return build_exit_river(m, s, [&]() -> rl_status {
    for (int i = 0; i < L * 7; ++i) {
      const NSView& v = m->views[i];
      RL_CUDA(cudaMemcpyAsync(v.q, q[i].data(), q[i].size() * 4, cudaMemcpyHostToDevice, s));
      RL_CUDA(cudaMemcpyAsync(v.s, sc[i].data(), sc[i].size() * 2, cudaMemcpyHostToDevice, s));
      RL_CUDA(cudaMemcpyAsync(v.z, zr[i].data(), zr[i].size() * 2, cudaMemcpyHostToDevice, s));
    }
    for (int l = 0; l < L; ++l) {
      Layer& ly = m->layers[l];
      Linear* lins[4] = {&ly.qkv, &ly.o, &ly.gu, &ly.dn};
      for (Linear* lin : lins) {
        launch_w4_from_views(lin->N, lin->K, lin->Kp, lin->qw, lin->sz, lin->rowmap,
                             m->d_views + (size_t)l * 7 + lin->view_base, s);
        RL_LAUNCHED();
      }
    }
    RL_CUDA(cudaStreamSynchronize(s));  // the host arrays are freed on return
    return RL_OK;
  });
}

rl_status rl_exit_layer_view(const rl_model* m, int32_t layer, int32_t which,
                             const uint32_t** qweight, const uint16_t** scales,
                             const uint16_t** zeros, int32_t* n_rows, int32_t* n_cols) {
  if (!m) return fail(RL_ERR_INVALID_ARG, "model is NULL");
  if (!m->quantized) return fail(RL_ERR_STATE, "exit river not built");
  if (layer < 0 || layer >= m->L || which < 0 || which > 6)
    return fail(RL_ERR_INVALID_ARG, "layer %d / linear %d out of range", layer, which);
  const NSView& v = m->views[(size_t)layer * 7 + which];
  if (qweight) *qweight = v.q;
  if (scales) *scales = v.s;
  if (zeros) *zeros = v.z;
  if (n_rows) *n_rows = v.N;
  if (n_cols) *n_cols = v.K;
  return RL_OK;
}

rl_status rl_kv_cache_alloc(const rl_model* mc, int32_t max_batch, int32_t max_seq, rl_kv** out) {
  if (!mc || !out) return fail(RL_ERR_INVALID_ARG, "NULL argument");
  *out = nullptr;
  if (max_batch < 1 || max_batch > 1024 || max_seq < 1)
    return fail(RL_ERR_INVALID_ARG, "max_batch must be in [1, 1024] and max_seq >= 1");
  rl_model* m = const_cast<rl_model*>(mc);
  rl_kv* kv = new rl_kv();
  kv->m = m;
  kv->maxB = max_batch;
  kv->Tmax = max_seq;
  auto bail = [&](rl_status st) {
    delete kv;
    return st;
  };
#define K_TRY(expr)                   \
  do {                                \
    rl_status s_ = (expr);            \
    if (s_ != RL_OK) return bail(s_); \
  } while (0)
  const size_t per_layer = (size_t)max_batch * m->Hkv * max_seq * m->hd;
  kv->K.resize(m->L);
  kv->V.resize(m->L);
  {
    bf16 *k_all = nullptr, *v_all = nullptr;
    K_TRY(kv->alloc(&k_all, per_layer * m->L));
    K_TRY(kv->alloc(&v_all, per_layer * m->L));
    for (int l = 0; l < m->L; ++l) {
      kv->K[l] = k_all + per_layer * l;
      kv->V[l] = v_all + per_layer * l;
    }
    // the decode attention reads K / V chunks by TMA: 16- and 64-row x 64-dim boxes
    const long long rows = (long long)m->L * max_batch * m->Hkv * max_seq;
    kv->tm_ok = rows < (1ll << 31) && (m->hd == 64 || m->hd == 128) &&
                make_tmap_bf16(&kv->tmk, k_all, m->hd, (int)rows, m->hd, 16) &&
                make_tmap_bf16(&kv->tmv, v_all, m->hd, (int)rows, m->hd, 16) &&
                make_tmap_bf16(&kv->tmk64, k_all, m->hd, (int)rows, m->hd, 64) &&
                make_tmap_bf16(&kv->tmv64, v_all, m->hd, (int)rows, m->hd, 64);
  }
  K_TRY(kv->alloc(&kv->st, 1));
  const int B = max_batch;
  for (int i = 0; i < 3; ++i) K_TRY(kv->alloc(&kv->h[i], (size_t)B * m->d));
  K_TRY(kv->alloc(&kv->x_attn, (size_t)B * m->Kd));
  K_TRY(kv->alloc(&kv->x_ffn, (size_t)B * m->Kd));
  K_TRY(kv->alloc(&kv->o, (size_t)B * m->Ko));
  K_TRY(kv->alloc(&kv->u, (size_t)B * m->Kf));
  K_TRY(kv->alloc(&kv->xs_attn, (size_t)B * (m->Kd / kGroup)));
  K_TRY(kv->alloc(&kv->xs_ffn, (size_t)B * (m->Kd / kGroup)));
  K_TRY(kv->alloc(&kv->xs_o, (size_t)B * (m->Ko / kGroup)));
  K_TRY(kv->alloc(&kv->xs_u, (size_t)B * (m->Kf / kGroup)));
  K_TRY(kv->alloc(&kv->q, (size_t)B * m->Hq * m->hd));
  int ncap = 1;
  for (int b = 1; b <= B; ++b) {
    ncap = std::max(ncap, b * decode_nchunks(m, b, max_seq));
    ncap = std::max(ncap, b * decode_attention_chunks(b, m->Hkv, max_seq, m->sm_count));
  }
  if (decode_attention_chunks(1, m->Hkv, max_seq, m->sm_count) > 256)
    return bail(fail(RL_ERR_UNSUPPORTED, "max_seq %d exceeds the decode attention limit (32768)", max_seq));
  kv->nchunks_cap = ncap;
  K_TRY(kv->alloc(&kv->part, (size_t)ncap * m->Hq * (m->hd + 2)));
  K_TRY(kv->alloc(&kv->cosbuf, (size_t)B));
  {
    const int sm = m->sm_count;
    const int max_tiles = std::max(std::max(m->Nqkv, 2 * m->F), std::max(m->d, m->V)) / 16 + 1;
    K_TRY(kv->alloc(&kv->ws, (size_t)sm * 2 * 128));
    K_TRY(kv->alloc(&kv->tile_ticket, (size_t)max_tiles));
    kv->n_tile_ticket = max_tiles;
    K_TRY(kv->alloc(&kv->cta_ticket, 1));
    K_TRY(kv->alloc(&kv->attn_ticket, (size_t)B * m->Hkv));
    kv->tc_ws_floats = (size_t)4 * sm * 64 * 128;  // split-K partial tiles (~20 MB at 152 SMs)
    K_TRY(kv->alloc(&kv->tc_ws, kv->tc_ws_floats));
    kv->tc_ticket_n = 1024;
    K_TRY(kv->alloc(&kv->tc_ticket, (size_t)kv->tc_ticket_n));
    K_TRY(kv->alloc(&kv->am_val, (size_t)sm * kFusedMaxB));
    K_TRY(kv->alloc(&kv->am_idx, (size_t)sm * kFusedMaxB));
    K_TRY(kv->alloc(&kv->st_mid, (size_t)(m->d / 16) * 8));
    K_TRY(kv->alloc(&kv->st_end, (size_t)(m->d / 16) * 8 * 3));
  }
  {
    // persistent step kernel: phase counters, descriptors, attention partials
    kv->nph_cap = 6 * m->L + 2;
    kv->n_bars = (size_t)m->sm_count * 32;
    K_TRY(kv->alloc(&kv->bars, kv->n_bars));
    K_TRY(kv->alloc(&kv->tctr, (size_t)kv->nph_cap));
    K_TRY(kv->alloc(&kv->d_ph, (size_t)kv->nph_cap));
    const int CH = 128;  // positions per attention chunk
    const int need = (max_seq + CH - 1) / CH;
    kv->part_cap = std::min(256, need + m->sm_count + 1);
    if (need <= 256) {
      const int bs = std::min(B, kFusedMaxB);
      K_TRY(kv->alloc(&kv->part_s, (size_t)bs * m->Hq * kv->part_cap * (m->hd + 4)));
    } else {
      kv->part_cap = 0;  // context too long for the step kernel's chunking: fused path
    }
  }
  K_TRY(kv->alloc(&kv->d_tok, (size_t)B));
  K_TRY(kv->alloc(&kv->d_next, (size_t)B));
  K_TRY(kv->alloc(&kv->d_exit, 1));
  K_TRY(kv->alloc(&kv->d_logits, (size_t)B * m->V));
  K_TRY(kv->alloc(&kv->d_mincos, (size_t)m->L));
  K_TRY(kv->alloc(&kv->rope_cs, (size_t)max_seq * (m->hd / 2)));
  launch_rope_table(m->inv_freq, m->hd / 2, max_seq, kv->rope_cs, 0);
  {
    cudaError_t e = cudaStreamSynchronize(0);
    if (e != cudaSuccess) return bail(fail(RL_ERR_CUDA, "RoPE table: %s", cudaGetErrorString(e)));
  }
#undef K_TRY
  *out = kv;
  return RL_OK;
}

rl_status rl_kv_cache_free(rl_kv* kv) {
  delete kv;
  return RL_OK;
}

rl_status rl_kv_view(const rl_kv* kv, int32_t layer, const void** d_k, const void** d_v) {
  if (!kv) return fail(RL_ERR_INVALID_ARG, "kv is NULL");
  if (layer < 0 || layer >= kv->m->L) return fail(RL_ERR_INVALID_ARG, "layer out of range");
  if (d_k) *d_k = kv->K[layer];
  if (d_v) *d_v = kv->V[layer];
  return RL_OK;
}

rl_status rl_kv_position(const rl_kv* kv, int32_t* pos, int32_t* decode_step) {
  if (!kv) return fail(RL_ERR_INVALID_ARG, "kv is NULL");
  if (pos) *pos = kv->host_pos;
  if (decode_step) *decode_step = kv->host_step;
  return RL_OK;
}

rl_status rl_kv_set_position(rl_kv* kv, int32_t pos, int32_t decode_step, rl_stream_t stream) {
  if (!kv) return fail(RL_ERR_INVALID_ARG, "kv is NULL");
  if (pos < 0 || pos > kv->Tmax || decode_step < 0)
    return fail(RL_ERR_INVALID_ARG, "position %d outside [0, %d] or negative step", pos, kv->Tmax);
  launch_set_state(kv->st, pos, decode_step, as_stream(stream));
  RL_LAUNCHED();
  RL_TRY(reset_sync_words(kv, as_stream(stream)));
  kv->host_pos = pos;
  kv->host_step = decode_step;
  return RL_OK;
}

rl_status rl_kv_set_wait_limit(rl_kv* kv, int64_t polls) {
  if (!kv) return fail(RL_ERR_INVALID_ARG, "kv is NULL");
  if (polls < 0) return fail(RL_ERR_INVALID_ARG, "polls must be >= 0");
  kv->wait_limit = polls;
  return RL_OK;
}

rl_status rl_debug_fail_allocations(int64_t after) {
  g_alloc_budget.store(after < 0 ? -1 : after);
  return RL_OK;
}

rl_status rl_kv_set_decode_path(rl_kv* kv, int32_t path) {
  if (!kv) return fail(RL_ERR_INVALID_ARG, "kv is NULL");
  if (path < RL_PATH_AUTO || path > RL_PATH_GENERIC) return fail(RL_ERR_INVALID_ARG, "unknown path %d", path);
  kv->path_pref = path;
  return RL_OK;
}

int32_t rl_kv_decode_path(const rl_kv* kv, int32_t B) {
  if (!kv || B < 1 || B > kv->maxB) return -1;
  return decode_path(kv->m, kv, B);
}

rl_status rl_kv_set_trace(rl_kv* kv, float* d_hidden) {
  if (!kv) return fail(RL_ERR_INVALID_ARG, "kv is NULL");
  kv->trace = d_hidden;
  return RL_OK;
}

rl_status rl_prefill(rl_model* m, rl_kv* kv, const int32_t* d_tokens, int32_t B, int32_t T,
                     const rl_exit_policy* policy, float* d_logits, int32_t* d_next_token,
                     int32_t* d_exit_layer, float* d_min_cos, rl_stream_t stream) {
  if (!m || !kv || !d_tokens || !d_logits || !d_exit_layer)
    return fail(RL_ERR_INVALID_ARG, "NULL argument");
  if (kv->m != m) return fail(RL_ERR_INVALID_ARG, "kv cache belongs to another model");
  if (B < 1 || T < 1) return fail(RL_ERR_INVALID_ARG, "B and T must be >= 1");
  if (B > kv->maxB || T > kv->Tmax)
    return fail(RL_ERR_CAPACITY, "B=%d > max_batch=%d or T=%d > max_seq=%d", B, kv->maxB, T,
                kv->Tmax);
  RL_TRY(check_policy(m, policy));
  cudaStream_t s = as_stream(stream);
  const size_t M = (size_t)B * T;
  const int Gd = m->Kd / kGroup, Go = m->Ko / kGroup, Gf = m->Kf / kGroup;
  // stream-ordered workspace for the B*T token rows
  const size_t n_h = M * m->d, n_xd = M * m->Kd, n_xo = M * m->Ko, n_xf = M * m->Kf;
  const size_t bytes = 3 * n_h * 4 + 2 * n_xd * 2 + n_xo * 2 + n_xf * 2 +
                       M * (2 * Gd + Go + Gf) * 4 + M * m->Hq * m->hd * 4 +
                       M * m->Hq * (m->hd + 2) * 4 + M * 4 + 32 * 256;  // + alignment slack of the carve-up
  char* base = nullptr;
  if (alloc_injected_failure()) return fail(RL_ERR_OOM, "prefill workspace: injected allocation failure");
  RL_CUDA(cudaMallocAsync((void**)&base, bytes, s));
  RL_CUDA(cudaMemsetAsync(base, 0, bytes, s));
  char* p = base;
  auto take = [&](size_t nbytes) {
    char* r = p;
    p += (nbytes + 255) / 256 * 256;
    return r;
  };
  Work w;
  for (int i = 0; i < 3; ++i) w.h[i] = (float*)take(n_h * 4);
  w.x_attn = (bf16*)take(n_xd * 2);
  w.x_ffn = (bf16*)take(n_xd * 2);
  w.o = (bf16*)take(n_xo * 2);
  w.u = (bf16*)take(n_xf * 2);
  w.xs_attn = (float*)take(M * Gd * 4);
  w.xs_ffn = (float*)take(M * Gd * 4);
  w.xs_o = (float*)take(M * Go * 4);
  w.xs_u = (float*)take(M * Gf * 4);
  w.q = (float*)take(M * m->Hq * m->hd * 4);
  w.part = (float*)take(M * m->Hq * (m->hd + 2) * 4);
  w.nchunks = 1;
  w.cosbuf = (float*)take(M * 4);
  if ((size_t)(p - base) > bytes) return fail(RL_ERR_CUDA, "prefill workspace sizing");
  StepIO io{d_tokens, B, T, policy, d_logits, d_next_token, d_exit_layer, d_min_cos, true};
  RL_TRY(reset_sync_words(kv, s));
  rl_status st = enqueue_pass(m, kv, io, w, s);
  cudaFreeAsync(base, s);
  if (st != RL_OK) return st;
  kv->host_pos = T;
  kv->host_step = 0;
  return RL_OK;
}

rl_status rl_decode_step(rl_model* m, rl_kv* kv, const int32_t* d_tokens, int32_t B,
                         const rl_exit_policy* policy, float* d_logits, int32_t* d_next_token,
                         int32_t* d_exit_layer, float* d_min_cos, rl_stream_t stream) {
  if (!m || !kv || !d_tokens || !d_logits || !d_exit_layer)
    return fail(RL_ERR_INVALID_ARG, "NULL argument");
  if (kv->m != m) return fail(RL_ERR_INVALID_ARG, "kv cache belongs to another model");
  if (B < 1) return fail(RL_ERR_INVALID_ARG, "B must be >= 1");
  if (B > kv->maxB || B > kMaxBatch)
    return fail(RL_ERR_CAPACITY, "B=%d > max_batch=%d (or > %d)", B, kv->maxB, kMaxBatch);
  if (kv->host_pos + 1 > kv->Tmax)
    return fail(RL_ERR_CAPACITY, "KV cache full: position %d, max_seq %d", kv->host_pos, kv->Tmax);
  RL_TRY(check_policy(m, policy));
  cudaStream_t s = as_stream(stream);
  StepIO io{d_tokens, B, 1, policy, d_logits, d_next_token, d_exit_layer, d_min_cos, false};
  const Work w = decode_work(kv, B);
  kv->prof_pos = kv->host_pos;
  kv->prof_B = B;
  const int path = decode_path(m, kv, B);
  if (path < 0) return fail(RL_ERR_UNSUPPORTED, "the requested decode path does not fit batch %d", B);
  const bool step = path == RL_PATH_STEP;
  const bool fused = path == RL_PATH_FUSED;
  auto enqueue = [&]() -> rl_status {
    if (step) return enqueue_decode_step(m, kv, io, s);
    if (fused) return enqueue_decode_fused(m, kv, io, decode_attention_chunks(B, m->Hkv, kv->Tmax, m->sm_count), s);
    return enqueue_pass(m, kv, io, w, s);
  };
  if (!is_capturable(s)) {
    if (step) RL_TRY(prepare_step_phases(m, kv, io, s));
    RL_TRY(enqueue());
  } else {
    GraphKey key;
    key.B = B;
    key.mode = policy->mode;
    key.tau = policy->tau;
    key.sched = policy->d_schedule;
    key.sched_len = policy->schedule_len;
    key.tokens = step ? nullptr : d_tokens;  // step path: a new token pointer is a parameter update
    key.logits = d_logits;
    key.next = d_next_token;
    key.exit = d_exit_layer;
    key.min_cos = d_min_cos;
    key.trace = kv->trace;
    key.prof = kv->profiling ? (kv->timeline ? 2 : 1) : 0;
    key.fused = fused;
    key.step = step;
    key.wait = kv->wait_limit;
    key.epoch = m->epoch;
    if (!kv->exec || !(key == kv->key)) {
      if (step) RL_TRY(prepare_step_phases(m, kv, io, s));
      cudaGraph_t g = nullptr;
      RL_CUDA(cudaStreamBeginCapture(s, cudaStreamCaptureModeThreadLocal));
      rl_status st = enqueue();
      cudaError_t e = cudaStreamEndCapture(s, &g);
      if (st != RL_OK) {
        if (g) cudaGraphDestroy(g);
        return st;
      }
      if (e != cudaSuccess) return fail(RL_ERR_CUDA, "graph capture: %s", cudaGetErrorString(e));
      if (kv->exec && (step || kv->graph)) {
        // the step path keeps its graph (for node updates): instantiate afresh
        cudaGraphExecDestroy(kv->exec);
        kv->exec = nullptr;
      }
      if (kv->graph) {
        cudaGraphDestroy(kv->graph);
        kv->graph = nullptr;
        kv->step_node = nullptr;
      }
      if (kv->exec) {
        cudaGraphExecUpdateResultInfo info;
        if (cudaGraphExecUpdate(kv->exec, g, &info) != cudaSuccess) {
          cudaGetLastError();
          cudaGraphExecDestroy(kv->exec);
          kv->exec = nullptr;
        }
      }
      if (!kv->exec) {
        e = cudaGraphInstantiate(&kv->exec, g, 0);
        if (e != cudaSuccess) {
          cudaGraphDestroy(g);
          kv->exec = nullptr;
          return fail(RL_ERR_CUDA, "graph instantiate: %s", cudaGetErrorString(e));
        }
      }
      if (step) {
        size_t nn = 0;
        RL_CUDA(cudaGraphGetNodes(g, nullptr, &nn));
        std::vector<cudaGraphNode_t> nodes(nn);
        RL_CUDA(cudaGraphGetNodes(g, nodes.data(), &nn));
        for (cudaGraphNode_t nd : nodes) {
          cudaGraphNodeType t;
          RL_CUDA(cudaGraphNodeGetType(nd, &t));
          if (t == cudaGraphNodeTypeKernel) kv->step_node = nd;
        }
        kv->graph = g;
        if (!kv->step_node) return fail(RL_ERR_CUDA, "decode-step graph holds no kernel node");
      } else {
        cudaGraphDestroy(g);
      }
      kv->key = key;
    } else if (step && kv->step_node && kv->step_args.tokens != d_tokens) {
      StepArgs a2 = kv->step_args;
      a2.tokens = d_tokens;
      cudaKernelNodeParams kp;
      RL_CUDA(cudaGraphKernelNodeGetParams(kv->step_node, &kp));
      void* args[1] = {&a2};
      kp.kernelParams = args;
      kp.extra = nullptr;
      RL_CUDA(cudaGraphExecKernelNodeSetParams(kv->exec, kv->step_node, &kp));
      kv->step_args = a2;
    }
    RL_CUDA(cudaGraphLaunch(kv->exec, s));
  }
  kv->host_pos += 1;
  kv->host_step += 1;
  return RL_OK;
}

rl_status rl_decode_step_host(rl_model* m, rl_kv* kv, const int32_t* h_tokens, int32_t B,
                              const rl_exit_policy* policy, float* h_logits,
                              int32_t* h_next_token, int32_t* h_exit_layer, float* h_min_cos,
                              rl_stream_t stream) {
  if (!m || !kv || !h_tokens || !h_next_token || !h_exit_layer)
    return fail(RL_ERR_INVALID_ARG, "NULL argument");
  if (B < 1 || B > kv->maxB) return fail(RL_ERR_CAPACITY, "B=%d outside [1, max_batch]", B);
  cudaStream_t s = as_stream(stream);
  RL_CUDA(cudaMemcpyAsync(kv->d_tok, h_tokens, (size_t)B * 4, cudaMemcpyHostToDevice, s));
  RL_TRY(rl_decode_step(m, kv, kv->d_tok, B, policy, kv->d_logits, kv->d_next, kv->d_exit,
                        kv->d_mincos, stream));
  RL_CUDA(cudaMemcpyAsync(h_next_token, kv->d_next, (size_t)B * 4, cudaMemcpyDeviceToHost, s));
  RL_CUDA(cudaMemcpyAsync(h_exit_layer, kv->d_exit, 4, cudaMemcpyDeviceToHost, s));
  if (h_logits)
    RL_CUDA(cudaMemcpyAsync(h_logits, kv->d_logits, (size_t)B * m->V * 4, cudaMemcpyDeviceToHost, s));
  if (h_min_cos)
    RL_CUDA(cudaMemcpyAsync(h_min_cos, kv->d_mincos, (size_t)m->L * 4, cudaMemcpyDeviceToHost, s));
  RL_CUDA(cudaStreamSynchronize(s));
  return RL_OK;
}

rl_status rl_sync(rl_model* m, rl_kv* kv, rl_stream_t stream) {
  (void)m;
  RL_CUDA(cudaStreamSynchronize(as_stream(stream)));
  RL_CUDA(cudaGetLastError());
  if (kv) {
    int err = 0;
    RL_CUDA(cudaMemcpy(&err, &kv->st->err, sizeof(int), cudaMemcpyDeviceToHost));
    if (err) {
      RL_CUDA(cudaMemset(&kv->st->err, 0, sizeof(int)));
      RL_TRY(reset_sync_words(kv, as_stream(stream)));
      RL_CUDA(cudaStreamSynchronize(as_stream(stream)));
      return fail(RL_ERR_DEVICE, "device error word 0x%x (%s%s%s%s)", err,
                  (err & RL_DEVERR_TOKEN) ? "token id out of range " : "",
                  (err & RL_DEVERR_CAPACITY) ? "kv capacity " : "",
                  (err & RL_DEVERR_SCHEDULE) ? "schedule entry out of range " : "",
                  (err & RL_DEVERR_TIMEOUT) ? "a bounded wait in a kernel timed out" : "");
    }
  }
  return RL_OK;
}

rl_status rl_kv_set_profiling(rl_kv* kv, int32_t enable) {
  if (!kv) return fail(RL_ERR_INVALID_ARG, "kv is NULL");
  if (enable && kv->ev.empty()) {
    const int cap = 12 * kv->m->L + 8;
    kv->recs.assign(cap, ProfRec());
    kv->ev.assign(2 * cap, nullptr);
    for (auto& e : kv->ev) RL_CUDA(cudaEventCreate(&e));
    RL_TRY(kv->alloc(&kv->d_paths, (size_t)cap));
    RL_TRY(kv->alloc(&kv->tl, (size_t)2 * kv->nph_cap));
  }
  if (enable >= 2 && !kv->tl2)
    RL_TRY(kv->alloc(&kv->tl2, (size_t)kv->nph_cap * kv->m->sm_count * kTl2));
  kv->profiling = enable != 0;
  kv->timeline = enable >= 2;
  return RL_OK;
}

rl_status rl_kv_timeline(rl_kv* kv, rl_stream_t stream, int64_t cap, uint64_t* out, int32_t* nphase,
                         int32_t* nctas, int32_t* nstamps) {
  if (!kv || !out || !nphase || !nctas || !nstamps) return fail(RL_ERR_INVALID_ARG, "NULL argument");
  if (!kv->tl2 || kv->nrec != -1) return fail(RL_ERR_STATE, "no per-CTA timeline recorded");
  RL_CUDA(cudaStreamSynchronize(as_stream(stream)));
  const int64_t need = (int64_t)kv->nph_last * kv->m->sm_count * kTl2;
  if (cap < need) return fail(RL_ERR_INVALID_ARG, "timeline buffer too small");
  RL_CUDA(cudaMemcpy(out, kv->tl2, (size_t)need * 8, cudaMemcpyDeviceToHost));
  *nphase = kv->nph_last;
  *nctas = kv->m->sm_count;
  *nstamps = kTl2;
  return RL_OK;
}

rl_status rl_kv_profile(rl_kv* kv, rl_stream_t stream, int32_t cap, int32_t* kinds,
                        int32_t* layers, int32_t* paths, float* ms, double* bytes, int32_t* n) {
  if (!kv || !n) return fail(RL_ERR_INVALID_ARG, "NULL argument");
  RL_CUDA(cudaStreamSynchronize(as_stream(stream)));
  if (kv->nrec == -1) {
    // persistent step kernel: one record per phase (first start .. last end
    // over CTAs, from the in-kernel timeline), then the whole kernel (events)
    const rl_model* m = kv->m;
    const int nph = kv->nph_last;
    std::vector<unsigned long long> tl((size_t)2 * nph);
    RL_CUDA(cudaMemcpy(tl.data(), kv->tl, tl.size() * 8, cudaMemcpyDeviceToHost));
    DevState hs;
    RL_CUDA(cudaMemcpy(&hs, kv->st, sizeof(hs), cudaMemcpyDeviceToHost));
    const int e = hs.exit_layer;
    int cnt = 0;
    double total = 0;
    for (int p = 0; p < nph && cnt < cap; ++p, ++cnt) {
      const PhaseDesc& d = kv->h_ph[p];
      int kind = RL_K_LM_HEAD;
      double b = 0;
      int path = -1;
      if (d.kind == PH_ATTN) {
        kind = RL_K_ATTN;
        b = 2.0 * kv->prof_B * m->Hkv * (double)(kv->prof_pos + 1) * m->hd * 2.0;
      } else {
        if (d.layer_no > 0)
          kind = d.epi == EPI_QKV_ROPE ? RL_K_QKV
                 : d.epi == EPI_SWIGLU ? RL_K_GU
                 : d.stats_k_out == 3  ? RL_K_DOWN
                                       : RL_K_O;
        path = (d.qwt && d.layer_no > e) ? 1 : 0;
        b = path ? (double)d.N * d.Kp / 2.0 + (double)d.N * (d.Kp / kGroup) * 4.0
                 : (double)d.N * d.Kp * 2.0;
      }
      total += b;
      const double t = tl[(size_t)nph + p] > tl[p] ? (double)(tl[(size_t)nph + p] - tl[p]) * 1e-6 : 0.0;
      if (kinds) kinds[cnt] = kind;
      if (layers) layers[cnt] = d.layer_no;
      if (paths) paths[cnt] = path;
      if (ms) ms[cnt] = (float)t;
      if (bytes) bytes[cnt] = b;
    }
    if (cnt < cap) {
      float t = 0.f;
      RL_CUDA(cudaEventElapsedTime(&t, kv->ev[0], kv->ev[1]));
      if (kinds) kinds[cnt] = RL_K_STEP;
      if (layers) layers[cnt] = 0;
      if (paths) paths[cnt] = -1;
      if (ms) ms[cnt] = t;
      if (bytes) bytes[cnt] = total;
      ++cnt;
    }
    *n = cnt;
    return RL_OK;
  }
  const int cnt = std::min(kv->nrec, (int)cap);
  std::vector<int> hp(kv->nrec > 0 ? kv->nrec : 1, 0);
  if (kv->nrec > 0)
    RL_CUDA(cudaMemcpy(hp.data(), kv->d_paths, kv->nrec * sizeof(int), cudaMemcpyDeviceToHost));
  const rl_model* m = kv->m;
  for (int i = 0; i < cnt; ++i) {
    const ProfRec& r = kv->recs[i];
    float t = 0.f;
    RL_CUDA(cudaEventElapsedTime(&t, kv->ev[2 * i], kv->ev[2 * i + 1]));
    const int path = r.gemv ? hp[i] : -1;
    double b = path == 1 ? r.bytes_w4 : r.bytes_bf;
    if (r.attn)  // K and V rows 0..p of every sequence
      b = 2.0 * kv->prof_B * m->Hkv * (double)(kv->prof_pos + 1) * m->hd * 2.0;
    if (kinds) kinds[i] = r.kind;
    if (layers) layers[i] = r.layer;
    if (paths) paths[i] = path;
    if (ms) ms[i] = t;
    if (bytes) bytes[i] = b;
  }
  *n = cnt;
  return RL_OK;
}

int32_t rl_decode_kernel_count(const rl_model* m, int32_t B) {
  if (!m || B < 1) return 0;
  if (step_fits_model(m, B)) return 1;  // one persistent kernel per step
  // offloaded layers: four staging launches each on the other paths
  const int stage = m->offload_from >= 0 ? 4 * (m->L - m->offload_from) : 0;
  if (fused_fits(m, B))  // fused path: QKV, attention, O, gate/up, down; LM head
    return m->L * 5 + 1 + stage;
  // per layer: QKV, attention (stream + combine, or one fused launch), group
  // sums (up to kTcW4AllTokens tokens), O, RMSNorm, gate/up, group sums, down,
  // layer end
  const int attn = attn_stream_supported(m->Hq / m->Hkv, m->hd) ? 2 : 1;
  const int gsum = B <= kTcW4AllTokens ? 2 : 0;
  return 1 + m->L * (6 + gsum + attn) + 1 + 1 + stage;
}

rl_status rl_model_offload_backbone(rl_model* m, int32_t first_layer, rl_stream_t stream) {
  if (!m) return fail(RL_ERR_INVALID_ARG, "model is NULL");
  if (first_layer < 0 || first_layer > m->L)
    return fail(RL_ERR_INVALID_ARG, "first_layer %d outside [0, %d]", first_layer, m->L);
  if (!m->quantized) return fail(RL_ERR_STATE, "build the exit river before offloading the backbone");
  if (m->offload_from >= 0) return fail(RL_ERR_STATE, "the backbone is already offloaded");
  if (first_layer == m->L) return RL_OK;
  cudaStream_t s = as_stream(stream);
  RL_CUDA(cudaStreamSynchronize(s));
  // the staging buffer: one layer's four [N][Kp] matrices
  const Layer& l0 = m->layers[first_layer];
  size_t stage_elems = 0;
  for (const Linear* lin : {&l0.qkv, &l0.o, &l0.gu, &l0.dn}) stage_elems += (size_t)lin->N * lin->Kp;
  bf16* stage = nullptr;
  RL_TRY(m->alloc(&stage, stage_elems));
  // host copies first: nothing is released until every layer has its copy
  struct Move { Linear* lin; bf16* hw; bf16* hwt; size_t off; };
  std::vector<Move> moves;
  auto undo = [&](rl_status st) {
    for (Move& mv : moves) {
      cudaFreeHost(mv.hw);
      cudaFreeHost(mv.hwt);
    }
    m->release(stage, stage_elems * sizeof(bf16));
    return st;
  };
  for (int l = first_layer; l < m->L; ++l) {
    Layer& ly = m->layers[l];
    size_t off = 0;
    for (Linear* lin : {&ly.qkv, &ly.o, &ly.gu, &ly.dn}) {
      const size_t nb = (size_t)lin->N * lin->Kp * sizeof(bf16);
      Move mv{lin, nullptr, nullptr, off};
      off += (size_t)lin->N * lin->Kp;
      if (alloc_injected_failure() || cudaHostAlloc((void**)&mv.hw, nb, cudaHostAllocMapped) != cudaSuccess) {
        cudaGetLastError();
        return undo(fail(RL_ERR_OOM, "pinned host memory for layer %d", l + 1));
      }
      if (alloc_injected_failure() || cudaHostAlloc((void**)&mv.hwt, nb, cudaHostAllocMapped) != cudaSuccess) {
        cudaGetLastError();
        cudaFreeHost(mv.hw);
        return undo(fail(RL_ERR_OOM, "pinned host memory for layer %d", l + 1));
      }
      moves.push_back(mv);
      if (cudaMemcpy(mv.hw, lin->w, nb, cudaMemcpyDeviceToHost) != cudaSuccess ||
          cudaMemcpy(mv.hwt, lin->wt, nb, cudaMemcpyDeviceToHost) != cudaSuccess) {
        cudaGetLastError();
        return undo(fail(RL_ERR_CUDA, "copying layer %d to host memory", l + 1));
      }
    }
  }
  // device addresses of the host copies (the same as the host ones with
  // unified addressing), the staging buffer's tensor maps
  for (Move& mv : moves) {
    void *dw = nullptr, *dwt = nullptr;
    if (cudaHostGetDevicePointer(&dw, mv.hw, 0) != cudaSuccess ||
        cudaHostGetDevicePointer(&dwt, mv.hwt, 0) != cudaSuccess) {
      cudaGetLastError();
      return undo(fail(RL_ERR_CUDA, "device address of pinned host memory"));
    }
    CUtensorMap tm;
    if (!make_weight_tmap(&tm, stage + mv.off, mv.lin->N, mv.lin->Kp))
      return undo(fail(RL_ERR_CUDA, "tensor map of the staging buffer"));
    Linear& lin = *mv.lin;
    const size_t nb = (size_t)lin.N * lin.Kp * sizeof(bf16);
    m->release(lin.w, nb);
    m->release(lin.wt, nb);
    lin.w_host = static_cast<const bf16*>(dw);
    lin.wt = static_cast<bf16*>(dwt);
    lin.w = stage + mv.off;
    lin.tm = tm;
    lin.offloaded = true;
    m->host_allocs.push_back(mv.hw);
    m->host_allocs.push_back(mv.hwt);
    m->host_bytes += 2 * nb;
  }
  m->stage = stage;
  m->offload_from = first_layer;
  ++m->epoch;
  return RL_OK;
}

rl_status rl_model_memory(const rl_model* m, uint64_t* device_bytes, uint64_t* host_bytes) {
  if (!m) return fail(RL_ERR_INVALID_ARG, "model is NULL");
  if (device_bytes) *device_bytes = m->bytes;
  if (host_bytes) *host_bytes = m->host_bytes;
  return RL_OK;
}

}  // extern "C"

namespace river {

LmHeadView lm_head_view(const rl_model* m) {
  LmHeadView v;
  v.w = m->lm_head;
  v.g_final = m->g_final;
  v.V = m->V;
  v.d = m->d;
  v.Kd = m->Kd;
  v.L = m->L;
  v.sm_count = m->sm_count;
  v.eps = m->cfg.rms_eps;
  return v;
}

rl_status set_error(rl_status s, const char* msg) { return fail(s, "%s", msg); }

}  // namespace river
