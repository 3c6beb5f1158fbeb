// Internal declarations shared by the kernels and the host runtime of
// libriver.so.  Nothing here is part of the C ABI (see include/river.h).
#pragma once

#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "river.h"

namespace river {

// Programmatic dependent launch for the many-launch decode path: a kernel
// launched with launch_pdl is set up while its predecessor in the stream
// finishes and calls pdl_wait() (the predecessor has completed and its
// writes are visible) before it reads anything; launched without the
// attribute the wait is a no-op.  No kernel triggers its successor early:
// an early trigger let the next kernel's CTAs hold SMs that the current
// kernel's later waves needed, and the batch-32 step got slower.
__device__ __forceinline__ void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
template <typename... KArgs, typename... Args>
inline cudaError_t launch_pdl(void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem, cudaStream_t s,
                              Args... args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kernel, args...);
}

typedef __nv_bfloat16 bf16;

constexpr int kGroup = 128;     // quantization group along K
constexpr int kMaxBatch = 64;   // decode batch handled by one GEMV launch

inline int round_up(int x, int m) { return (x + m - 1) / m * m; }

// ---------------------------------------------------------------------------
// Per-cache device state.  All kernels of one step read/write it; it never
// returns to the host during a step.
// ---------------------------------------------------------------------------
struct DevState {
  int pos;          // next KV slot to write (shared by all sequences)
  int step;         // decode-step counter since the last prefill (forced schedules)
  int exit_layer;   // exit layer e of the current step: layers l > e use the exit river
  int err;          // RL_DEVERR_* bits, sticky until rl_sync
  unsigned int ticket;  // last-arriver counter of the row-norm kernel (reset by the last CTA)
  unsigned int pad[3];
};

// ---------------------------------------------------------------------------
// GEMV / small-batch GEMM: y[b][n] = sum_k x[b][k] * W[n][k] on bf16 weights
// or on W4 weights (q - z) * s, chosen on the device per layer.
// ---------------------------------------------------------------------------
enum GemvEpilogue {
  EPI_STORE = 0,     // out[b][n] = y
  EPI_RESID = 1,     // out[b][n] = resid[b][n] + y
  EPI_SWIGLU = 2,    // rows interleaved per 16-row tile (8 gate, 8 up): out_h[b][j] = silu(g) * u
  EPI_QKV_ROPE = 3,  // rows permuted per head (RoPE pairs in one tile); RoPE + KV append
  EPI_LMHEAD = 4,    // logits + argmax (fused decode path only)
};

enum W4Mode { W4_OFF = 0, W4_ON = 1, W4_BY_LAYER = 2 };

struct GemvArgs {
  const bf16* w;          // bf16 [N][Kp] row-major (K zero-padded to Kp)
  const uint32_t* qw;     // W4 [N][Kp/8], nibble for k at bits 4*(k%8)
  const __half2* sz;      // W4 (scale, zero) per (row, group) [N][Kp/128]
  int N, Kp;              // N % 16 == 0, Kp % 128 == 0
  int w4_mode;            // W4Mode
  const int* exit_layer;  // W4_BY_LAYER: W4 path iff layer_no > *exit_layer
  int layer_no;           // 1-based
  const bf16* x;          // activations [B][ldx] bf16 (zero beyond K)
  int ldx;
  const float* xsum;      // per (b, group) sum of x, [B][ldxs] (W4 path only)
  int ldxs;
  int B;                  // columns (tokens) in this launch; k_gemv walks them 64 at a time
  int epi;
  float* out; int ldo;            // STORE / RESID
  const float* resid; int ldr;    // RESID
  bf16* out_h; int ldoh;          // SWIGLU
  // EPI_QKV_ROPE
  float* q_out;           // [tokens][Hq*hd] fp32
  bf16* kc; bf16* vc;     // layer cache base, [maxB][Hkv][Tmax][hd]
  int maxB, Tmax, Hq, Hkv, hd;
  const int* pos_ptr;     // decode: slot for every column
  int T_prefill;          // >0: column c is token (col_base + c) = seq*T + t at position t
  int col_base;
  const float* inv_freq;  // [hd/2]
  const float2* rope_cs;  // nullable: (cos, sin) of pos * inv_freq[i], [Tmax][hd/2]
  int* err;
  int* path_out;          // nullable: CTA 0 records the path taken (0 bf16, 1 W4)
  int w4_only;            // k_gemv: return at once unless the W4 path is taken
  // k_gemm_tc split-K (few output tiles): fp32 partial tiles and per-tile tickets
  float* tc_ws; size_t tc_ws_floats; unsigned* tc_ticket; int tc_ticket_n;
  int ksplit;             // set by launch_gemm_tc
  int tc_w4;              // k_gemm_tc runs the W4 path too (else it returns at once for W4 layers)
  const unsigned char* qtc;  // W4 in the tensor-core GEMM's k-block layout (w4_tc_bytes), or null
  long long first_wait;   // k_gemm_tc: polls of the epilogue's accumulator wait (0: the default)
};

void launch_gemv(const GemvArgs& a, int sm_count, cudaStream_t s);

// ---------------------------------------------------------------------------
// Tensor-core GEMM (tcgen05 + TMA) over many tokens (see gemm_tc.cu): the
// GemvArgs' bf16 weights against B tokens of x (no 64-column limit), the same
// epilogues; returns at once when the layer takes the W4 path.
// ---------------------------------------------------------------------------
bool tc_gemm_available();
cudaError_t tc_gemm_init();
bool make_tmap_bf16(CUtensorMap* map, const void* base, int inner, int rows, int ld, int box_rows);
bool make_weight_tmap(CUtensorMap* map, const bf16* w, int N, int Kp);
// W4 words and (scale, zero) pairs in the tensor-core GEMM's k-block layout.
size_t w4_tc_bytes(int N, int Kp);
void launch_w4_tc_layout(const uint32_t* qw, const __half2* sz, int N, int Kp, void* out, cudaStream_t s);
int tc_pick_bn(int N, int M, int sm_count);
// a.qtc: the layer's exit copy in the k-block layout (launch_w4_tc_layout), or null.
cudaError_t launch_gemm_tc(const CUtensorMap& tmW, const GemvArgs& a, int sm_count, cudaStream_t s);
// Whether the tensor-core GEMM also runs a W4 layer of this shape: always
// above kTcW4AllTokens tokens, else when the projection has at least half as
// many output tiles as SMs (narrower ones run on the dequantising GEMV, which
// needs the activations' per-group sums).
constexpr int kTcW4AllTokens = 32;
bool tc_gemm_runs_w4(int N, int B, int sm_count);
// (cos, sin) of pos * inv_freq[i] for pos < Tmax, i < half: [Tmax][half].
void launch_rope_table(const float* inv_freq, int half, int Tmax, float2* out, cudaStream_t s);

// ---------------------------------------------------------------------------
// Fused small-batch decode GEMV (B <= 8): norm / exit decision / embedding in
// the prologue, stream-K main loop, fused epilogues (see gemv_fused.cu).
// ---------------------------------------------------------------------------
// Activations of a fused projection: X_COPY = bf16 rows copied as they are;
// X_SCALED = bf16 rows x' = h * gain written by the producing epilogue, scaled
// per column by 1/sqrt(mean(h^2) + eps) from per-tile partial sums (and, with
// three partials per tile, the previous layer's exit decision);
// X_EMBED = the token embedding gathered and normalised in the prologue.
enum XMode { X_COPY = 1, X_SCALED = 2, X_EMBED = 3 };
constexpr int kFusedMaxB = 8;

struct FusedArgs {
  const bf16* w;          // bf16 [N][Kp] row-major
  const void* qwt;        // W4 in the unit-tiled layout (w4_tiled_bytes)
  int N, Kp;
  int w4_mode; int layer_no;
  DevState* st;
  int B;
  int xmode;
  const bf16* xg; int ldxg;                 // activations [B][ldxg], zero beyond K
  const float* stats_in; int stats_tiles; int stats_k;  // X_SCALED: [tiles][8][stats_k]
  int d; float eps;
  int dec_layer;                            // layer whose exit decision is taken here (0: none)
  int L; int mode; float tau; const int* schedule; int schedule_len; int step_begin;
  float* min_cos_out;
  const int* tokens; const bf16* embed; int vocab; const float* gain_embed; float* h_store;
  int epi;
  float* out; int ldo; const float* resid; int ldr; bf16* out_h; int ldoh;
  const float* gnext; bf16* xnext; int ldxnext;          // RESID: x' = h * gnext for the next norm
  float* stats_out; int stats_k_out; const float* h_in;  // RESID: per-tile partial sums
  float* trace; int trace_layer; int trace_maxB;
  float* q_out; bf16* kc; bf16* vc; int maxB, Tmax, Hq, Hkv, hd; const float* inv_freq;
  float* am_val; int* am_idx; int* next_token; int* exit_out;
  float* ws; unsigned* tile_ticket; unsigned* cta_ticket;
  int* path_out;
};

size_t fused_smem_bytes(const FusedArgs& a);
size_t w4_tiled_bytes(int N, int Kp);
void launch_w4_tile_layout(const uint32_t* qw, const __half2* sz, int N, int Kp, void* out,
                           cudaStream_t s);
int fused_grid(const FusedArgs& a, int sm_count);
void gemv_fused_setup();
cudaError_t launch_gemv_fused(const FusedArgs& a, int sm_count, bool pdl, cudaStream_t s);

// ---------------------------------------------------------------------------
// Row kernels: embedding, RMSNorm, cosine, batch-min exit decision.
// ---------------------------------------------------------------------------
struct RowNormArgs {
  // embedding mode (tokens != nullptr): h_out[r] = embed[tokens[r]]
  const int* tokens; const bf16* embed; int vocab;
  const float* h_in;      // residual entering the layer (cosine), nullable
  float* h_out;           // residual leaving the layer [rows][d]
  int rows, d;
  const float* g;         // gain of the next RMSNorm [d], nullable (no x written)
  float eps;
  bf16* x; int ldx;       // normalized bf16 output
  float* xsum; int ldxs;  // per-group sums of x
  // decision (when h_in != nullptr)
  float* cosbuf;          // [rows]
  int layer_no, L;
  int mode; float tau;    // RL_EXIT_TAU / RL_EXIT_FORCED
  float* min_cos_out;     // [L], nullable
  int* exit_out;          // written at layer L, nullable
  DevState* st;
  int set_pos;            // at layer L: st->pos = set_pos (>= 0) or st->pos + 1 (< 0)
  int set_step;           // at layer L: st->step = set_step (>= 0) or st->step + 1 (< 0)
  // step begin (embedding mode, CTA 0): initialize st->exit_layer
  const int* schedule; int schedule_len; int use_step_index;
  // trace of the last position of each sequence
  float* trace; int trace_layer; int trace_maxB; int trace_T;
};

void launch_rownorm(const RowNormArgs& a, cudaStream_t s);

void launch_group_sums(const bf16* x, int ldx, int Kp, int B, float* xsum, int ldxs,
                       cudaStream_t s);

void launch_argmax(const float* logits, int ld, int V, int B, int* out, cudaStream_t s);

// ---------------------------------------------------------------------------
// Attention over the shared KV cache.
// ---------------------------------------------------------------------------
struct AttnArgs {
  const float* q;         // [nq][Hq*hd] (RoPE applied)
  const bf16* kc; const bf16* vc;  // [maxB][Hkv][Tmax][hd]
  int maxB, Tmax, Hq, Hkv, hd;
  int nq;                 // query rows
  int T_prefill;          // >0: row r is sequence r/T at position r%T; else row b at *pos_ptr
  const int* pos_ptr;
  int nchunks;            // context split per (row, kv head)
  float* part;            // [nq][Hq][nchunks][hd + 2]
  bf16* o; int ldo;       // [nq][ldo] output, head h at h*hd
  unsigned* ticket;       // fused kernel: [nq][Hkv] last-arriver counters (zero between launches)
};

void launch_attention(const AttnArgs& a, cudaStream_t s);
// Single-kernel decode attention: partials + combine by the last CTA per (row, KV head).
cudaError_t launch_attention_fused(const AttnArgs& a, bool pdl, cudaStream_t s);
void attention_setup();

// Streaming decode attention (any batch): persistent CTAs, K/V chunks and
// query rows by TMA into a shared-memory ring, tensor-core chunks; writes the
// chunk partials [nq][Hq][nchunks][hd + 2] that k_attn_combine merges.
struct AttnStreamArgs {
  CUtensorMap tmk, tmv;   // every layer's K / V cache as one 2-D tensor [rows][hd], 16 x 64 boxes
  CUtensorMap tmk64, tmv64;  // the same tensors, 64 x 64 boxes
  int layer_row0;         // first row of this layer: layer * maxB * Hkv * Tmax
  const float* q;         // [nq][Hq][hd] (RoPE applied)
  const int* pos_ptr;
  int Tmax, Hq, Hkv, nq, nchunks, nslot;
  float* part;            // [nq][Hq][nchunks][hd + 2]
  int* err;
};
size_t attn_stream_smem(int* nslot);
void attn_stream_setup();
bool attn_stream_supported(int rep, int hd);
cudaError_t launch_attn_stream(const AttnStreamArgs& a, int rep, int hd, int grid, cudaStream_t s);
// Causal prompt attention on the tensor cores (attn_prefill.cu): query row
// (seq, t) of q [nseq*T][Hq*hd] attends to cache rows 0..t of its sequence;
// o [nseq*T][ldo] bf16.
struct AttnPrefillArgs {
  CUtensorMap tmk64, tmv64;  // every layer's K / V cache as one 2-D tensor [rows][hd], 64 x 64 boxes
  int layer_row0;            // first row of this layer: layer * maxB * Hkv * Tmax
  const float* q;
  int T, Hq, Hkv, Tmax, nseq;
  bf16* o;
  int ldo;
  int* err;
};
bool attn_prefill_supported(int rep, int hd);
cudaError_t launch_attn_prefill(const AttnPrefillArgs& a, int rep, int hd, cudaStream_t s);

// The combine half of launch_attention: merge a.nchunks partials into a.o.
void launch_attention_combine(const AttnArgs& a, cudaStream_t s);
// Context chunks per (sequence, KV head) of the fused decode attention (<= 256
// supported by its merge; <= 128 positions per chunk).
int decode_attention_chunks(int B, int Hkv, int Tmax, int sm_count);

// ---------------------------------------------------------------------------
// Weight preparation and quantization.
// ---------------------------------------------------------------------------
// Up to three source matrices [rows][src_ld]; rowmap[r] = (source, source row).
struct GatherSrcs { const bf16* p[3]; };

void launch_gather_rows(bf16* dst, int ldd, int N, int K, const int2* rowmap, GatherSrcs srcs,
                        int src_ld, cudaStream_t s);
void launch_set_state(DevState* st, int pos, int step, cudaStream_t s);
void launch_bf16_to_f32(const bf16* src, float* dst, int n, cudaStream_t s);

struct NSView { uint32_t* q; uint16_t* s; uint16_t* z; int N; int K; };

// HQQ zero-point refinement settings (float64, as the iteration computes).
struct HqqParams {
  int iters = 0;
  double p = 0.7, beta = 10.0, kappa = 1.01;
};

// Quantize the library's bf16 copy w [N][Kp] (K real inputs) into the
// internal W4 layout (qw, sz) and the interchange views: row r goes to
// views[rowmap[r].x] at row rowmap[r].y.  hqq == nullptr: min-max rounding;
// otherwise min-max followed by the HQQ refinement of every group's zero.
void launch_quantize(const bf16* w, int N, int K, int Kp, uint32_t* qw, __half2* sz,
                     const int2* rowmap, const NSView* views, const HqqParams* hqq, cudaStream_t s);
// Exit-vs-backbone K/V cosine per (sequence, K/V, KV head) of residual rows
// h [B][d] entering a layer: w [N][Kp] bf16 and (qw, sz) W4 of its fused QKV
// matrix, g its attention RMSNorm gain; out [B][2][Hkv].
cudaError_t launch_exit_kv_cosine(const float* h, int B, int d, const float* g, const bf16* w,
                                  const uint32_t* qw, const __half2* sz, int Kp, int Hq, int Hkv,
                                  int hd, float* out, cudaStream_t s);

// Offloaded backbone layers: copy `bytes` (a multiple of 16) from host memory
// into the device staging buffer, unless *exit_layer says layer layer_no runs
// on the exit river (exit_layer == nullptr: always copy).
void launch_stage_weights(const void* src, void* dst, size_t bytes, const int* exit_layer, int layer_no,
                          int sm_count, cudaStream_t s);

// The internal W4 layout (qw, sz) of a fused matrix from interchange views
// that already hold the exit layer (rl_load_exit_layers).
void launch_w4_from_views(int N, int K, int Kp, uint32_t* qw, __half2* sz, const int2* rowmap,
                          const NSView* views, cudaStream_t s);


// ---------------------------------------------------------------------------
// Persistent decode step (B <= 8): one cooperative kernel runs every phase of
// a decode step -- per layer QKV (+RoPE, KV append, exit decision), attention,
// O, gate/up, down; then the LM head -- with grid-wide phase barriers.  The
// weight stream of a CTA runs ahead across phase boundaries: it depends only
// on the weight path, never on this step's activations.
// ---------------------------------------------------------------------------
enum PhaseKind { PH_GEMV = 0, PH_ATTN = 1 };

struct PhaseDesc {
  int kind;                   // PH_GEMV / PH_ATTN
  int layer_no;               // 1..L; 0 = LM head (always the bf16 weights)
  // GEMV weights
  const bf16* wt;             // bf16 unit-tiled (see k_bf16_tile_layout)
  int wt_sys;                 // 1: wt is in host memory (an offloaded backbone layer)
  const unsigned char* qwt;   // W4 unit-tiled, nullptr if there is no exit-river copy
  int N, Kp, split;           // split: tiles claimed at run time (else round-robin)
  // activations
  int xmode;                  // X_COPY / X_SCALED / X_EMBED
  const bf16* xg;
  int ldxg;
  const float* stats_in;
  int stats_tiles, stats_k;
  int dec_layer;              // > 0: exit decision of layer dec_layer in the prologue
  // epilogue
  int epi;
  float* out;
  int ldo;
  const float* resid;
  int ldr;
  bf16* out_h;
  int ldoh;
  const float* gnext;
  bf16* xnext;
  int ldxnext;
  float* stats_out;
  int stats_k_out;
  const float* h_in;
  float* trace;
  int trace_layer;
  float* q_out;               // QKV output / attention input [B][Hq*hd] fp32
  bf16* kc;                   // layer's K cache [maxB][Hkv][Tmax][hd]
  bf16* vc;
  bf16* o_out;                // attention output [B][ldo_attn] bf16
  int ldo_attn;
};

struct StepArgs {
  CUtensorMap tmk, tmv;       // every layer's K / V cache as one 2-D tensor [rows][hd], 16 x 64 boxes, 128 B swizzle
  int kv_rows_layer;          // rows of one layer's cache: maxB * Hkv * Tmax
  const PhaseDesc* ph;
  int nph;
  DevState* st;
  int B, L, d, Hq, Hkv, hd, Tmax, vocab;
  float eps;
  int mode;
  float tau;
  const int* schedule;
  int schedule_len;
  const int* tokens;
  const bf16* embed;
  const float* gain_embed;
  float* h_store;
  int trace_maxB;
  const float* inv_freq;
  const float2* rope_cs;      // (cos, sin) of pos * inv_freq[i], [Tmax][hd/2], the same sincosf values
  float* min_cos_out;
  int* next_token;
  int* exit_out;
  float* am_val;
  int* am_idx;
  unsigned* cta_ticket;
  unsigned* bars;             // [grid * 32] per-CTA phase flags (128 B apart), zero at step start
  unsigned* tctr;             // [nph] tiles handed out per projection phase, zero at step start
  float* ws;                  // stream-K partial tiles [grid][2][128]
  unsigned* tile_ticket;      // [max tiles]
  float* part;                // attention partials [B][Hq][part_cap][hd + 2]
  unsigned* attn_ticket;      // [B][Hkv]
  int part_cap;
  int nslot;                  // weight ring slots
  int xs_row_bytes;           // activation row stride in shared memory
  int gmax;                   // max 128-input groups over the phases
  unsigned long long* tl;     // optional timeline: [nph] first starts, then [nph] last ends
  unsigned long long* tl2;    // optional per-CTA timeline [nph][grid][kTl2] (globaltimer ns)
  long long bar_wait;         // polls of a grid-barrier wait before it gives up (0: the default)
};
// Stamps of the per-CTA timeline, per (phase, CTA).
enum Tl2Stamp {
  TL2_BAR = 0,     // consumers: previous phase complete (grid barrier passed)
  TL2_X = 1,       // consumers: activation rows in shared memory (attention: first chunk)
  TL2_W = 2,       // consumers: first weight unit in shared memory
  TL2_CDONE = 3,   // consumers: last tile / chunk computed
  TL2_ARRIVE = 4,  // epilogues done, arrival at the phase counter
  TL2_P0 = 5,      // producer: first copy of the phase issued
  TL2_P1 = 6,      // producer: last copy of the phase issued
  TL2_RED = 7,     // reducer: RMSNorm scale / exit decision ready
  kTl2 = 8
};

// Shared memory the step kernel needs (0 if it does not fit).
size_t step_smem_bytes(int B, int kmax, int gmax, int* nslot);
// multi: the instantiation for contexts where a CTA may take several
// attention chunks (see k_decode_step)
// multi: a CTA may take more than one attention chunk; wide: the model has
// offloaded layers (the producer warp reads them with all its lanes).
cudaError_t launch_decode_step(const StepArgs& a, int grid, size_t smem, bool multi, bool wide, cudaStream_t s);
void decode_step_setup();
int decode_step_occupancy(size_t smem);  // resident CTAs per SM at this shared-memory size
// Attention chunks per (sequence, KV head) for context `ctx` (identical on host and device).
// Chunks of the context per (sequence, KV head) in the step kernel: as few
// as its 128-position slots allow while every CTA takes at most one chunk (a
// chunk's warps run 16 positions each, so longer chunks cost no latency and
// the merge combines fewer partials); beyond one chunk per CTA, the rounds of
// chunks are spread over the whole grid.
__host__ __device__ inline int step_attn_chunks(int ctx, int B, int Hkv, int hd, int grid, int cap) {
  const int CH = 128;  // positions per chunk
  const int n_min = (ctx + CH - 1) / CH;
  const int items = B * Hkv * n_min;
  const int per = (items + grid - 1) / grid;
  int n = per == 1 ? n_min : (per * grid) / (B * Hkv);
  if (n < n_min) n = n_min;
  if (n > ctx) n = ctx;
  if (n > cap) n = cap;
  if (n < 1) n = 1;
  return n;
}
// bf16 weights [N][Kp] -> the unit-tiled layout of the step kernel.
void launch_bf16_tile_layout(const bf16* w, int N, int Kp, bf16* out, cudaStream_t s);

// ---------------------------------------------------------------------------
// What the allocation-free LM-head entry point needs from the model, and the
// runtime's error message setter (both defined in api.cu).
// ---------------------------------------------------------------------------
struct LmHeadView {
  const bf16* w;          // LM head [V][Kd]
  const float* g_final;   // final RMSNorm gain [d]
  int V, d, Kd, L, sm_count;
  float eps;
};
LmHeadView lm_head_view(const rl_model* m);
rl_status set_error(rl_status s, const char* msg);

}  // namespace river
