/*
 * river.h -- C ABI of libriver.so, the GB300 (sm_103a) decode hot path of the
 * River-LLM "KV-shared exit river".
 *
 * Method (River-LLM explainer page, "River-LLM: Large Language Model Seamless
 * Exit Based on KV Share"):
 *   section 三  every decoder layer gets a training-free W4A16 copy, the exit
 *               layer; exit layer l writes its K/V into backbone layer l's own
 *               cache slot, so later tokens never meet a missing cache entry.
 *   section 四  state-transition similarity: cosine of the hidden state entering
 *               vs leaving layer l; the minimum over all tokens processed
 *               together is compared with tau; once it exceeds tau, layers
 *               l+1..L run on the exit river (no later layer is checked).
 *   section 五  prefill takes one sequence-level decision, generation one per
 *               decode step.
 * Format of the exit layers: asymmetric 4-bit weights in groups of 128
 * consecutive inputs, fp16 scale and zero per group, eight nibbles per
 * uint32 (nibble for input k at bits 4*(k%8)).
 *
 * Conventions for every entry point
 *   - Pointers named d_* are DEVICE pointers owned by the caller; h_* are host
 *     pointers owned by the caller.  Objects (rl_model, rl_kv) are owned by the
 *     library and released with their destroy/free call.
 *   - Streams are cudaStream_t passed as rl_stream_t (NULL = legacy default
 *     stream).  Calls that take a stream enqueue work on it and return without
 *     waiting, unless stated otherwise.
 *   - Every call returns rl_status.  Argument errors are detected on the host
 *     before anything is enqueued and leave all state unchanged; the message is
 *     available from rl_last_error() (thread-local).  Errors found on the device
 *     (token id out of range, KV capacity, bad schedule entry) set a device
 *     error word that rl_sync() reports as RL_ERR_DEVICE; the offending write is
 *     skipped, never performed out of bounds.  No call aborts the process.
 *   - Weights and activations are bf16 on the device; logits, cosines and the
 *     residual stream are fp32.
 */
#ifndef RIVER_H
#define RIVER_H

#include <stdint.h>

#if defined(__GNUC__)
#define RL_API __attribute__((visibility("default")))
#else
#define RL_API
#endif

#ifdef __cplusplus
extern "C" {
#endif

typedef struct rl_model rl_model;
typedef struct rl_kv rl_kv;
typedef void* rl_stream_t; /* cudaStream_t */

typedef enum {
  RL_OK = 0,
  RL_ERR_INVALID_ARG = 1, /* bad pointer, shape or policy; nothing enqueued */
  RL_ERR_OOM = 2,         /* device allocation failed */
  RL_ERR_CUDA = 3,        /* a CUDA runtime call failed; see rl_last_error() */
  RL_ERR_CAPACITY = 4,    /* position would reach max_seq, or batch > max_batch */
  RL_ERR_STATE = 5,       /* e.g. exit river used before rl_quantize_exit_layers */
  RL_ERR_DEVICE = 6,      /* device error word set (reported by rl_sync) */
  RL_ERR_UNSUPPORTED = 7  /* shape outside what the kernels handle */
} rl_status;

/* Device error word bits (rl_sync returns RL_ERR_DEVICE if any is set). */
enum {
  RL_DEVERR_TOKEN = 1,    /* a token id was outside [0, vocab); row 0 used instead */
  RL_DEVERR_CAPACITY = 2, /* KV position >= max_seq; K/V write skipped */
  RL_DEVERR_SCHEDULE = 4, /* forced schedule entry outside [0, L]; clamped */
  RL_DEVERR_TIMEOUT = 8   /* a bounded wait inside a kernel gave up; outputs invalid */
};

/* Decoder shape (Llama-style).  Requirements: head_dim in {64, 128};
 * n_q_heads % n_kv_heads == 0; d_model, ffn_dim multiples of 16;
 * group_size == 128; n_q_heads * head_dim == d_model is not required. */
typedef struct {
  int32_t n_layers, d_model, n_q_heads, n_kv_heads, head_dim, ffn_dim, vocab, group_size;
  float rms_eps, rope_theta;
} rl_config;

/* One decoder layer's weights: device pointers to bf16, linear weights
 * row-major [out][in]: wq [Hq*hd][d], wk/wv [Hkv*hd][d], wo [d][Hq*hd],
 * wg/wu [F][d], wd [d][F]; g_attn/g_ffn are the RMSNorm gains [d]. */
typedef struct {
  const void *wq, *wk, *wv, *wo, *wg, *wu, *wd, *g_attn, *g_ffn;
} rl_layer_weights;

/* embed [V][d], lm_head [V][d], g_final [d] (bf16, device); layers: HOST
 * array of n_layers entries. */
typedef struct {
  const void *embed, *lm_head, *g_final;
  const rl_layer_weights* layers;
} rl_weights;

/* Which linear of a layer (rl_exit_layer_view). */
enum { RL_WQ = 0, RL_WK = 1, RL_WV = 2, RL_WO = 3, RL_WG = 4, RL_WU = 5, RL_WD = 6 };

/* Exit policy (explainer section 四).
 *   RL_EXIT_TAU:    exit after the first layer l < L whose batch-minimum cosine
 *                   is strictly greater than tau; tau > 1 never exits.
 *   RL_EXIT_FORCED: exit layer e taken from d_schedule (device int32, values in
 *                   [0, L]; e = L is full depth, e = 0 runs every layer on the
 *                   exit river).  Decode step i (counted from the last prefill)
 *                   uses d_schedule[i % schedule_len]; prefill uses d_schedule[0].
 * "Exit layer e" = number of layers run on the backbone; layers e+1..L run on
 * the exit river. */
enum { RL_EXIT_TAU = 0, RL_EXIT_FORCED = 1 };
typedef struct {
  int32_t mode;
  float tau;
  const int32_t* d_schedule;
  int32_t schedule_len;
} rl_exit_policy;

/* Library version string (static storage). */
RL_API const char* rl_version(void);

/* Thread-local message of the last failed call on this thread ("" if none). */
RL_API const char* rl_last_error(void);

/* Create a model on the current CUDA device.  Copies every weight into the
 * library's own layout (the caller may free its buffers once the stream has
 * reached this point).  Synchronous with respect to `stream`. */
RL_API rl_status rl_model_create(const rl_config* cfg, const rl_weights* w, rl_stream_t stream,
                          rl_model** out);
RL_API void rl_model_destroy(rl_model* m);

/* quantize_exit_layers (explainer section 三): build the exit river, one W4A16
 * copy of each layer's seven linears, by min-max round-to-nearest per group of
 * 128 inputs:  s = fp16((max-min)/15) (1.0 if max == min or it rounds to 0),
 * z = fp16(-min/s), q = clamp(rint(w/s + z), 0, 15), all in IEEE fp32.  A
 * ragged last group (inputs not a multiple of 128) covers the remainder.
 * Norm gains are shared with the backbone.  Enqueued on `stream`. */
RL_API rl_status rl_quantize_exit_layers(rl_model* m, rl_stream_t stream);

/* quantize_exit_layers with HQQ's zero-point refinement (explainer section
 * 六 names HQQ, which needs no calibration data, as the exit layers'
 * quantizer; half-quadratic quantization, Badri and Shaji 2023).  The
 * min-max scale above stays; each group's zero point z is refined by `iters`
 * alternations, in float64 with every operation rounded once:
 *   q = clamp(rint(w/s + z), 0, 15),  r = w - s(q - z),
 *   e = sign(r) max(|r| - |r|^(lp_norm-1)/beta, 0)   (0 where r == 0),
 *   z = mean over the group of q - (w - e)/s,  beta *= kappa.
 * The stored zero is the fp16 value (min-max's or an iteration's, rounded
 * once from float64) whose stored codes give the lowest sum |w - s(q - z)|^p
 * over the group (ties keep the earlier); codes follow the min-max rule with
 * it, so the packed format and every other entry point are unchanged.  The
 * method's usual settings: iters 20, lp_norm 0.7, beta 10, kappa 1.01.
 * RL_ERR_INVALID_ARG for iters outside [0, 1000], lp_norm outside (0, 2],
 * beta <= 0 (infinity allowed: no shrinkage) or kappa outside [1, 1000);
 * RL_ERR_STATE if the exit river is already built.  Enqueued on `stream`;
 * returns once the exit river is ready. */
RL_API rl_status rl_quantize_exit_layers_hqq(rl_model* m, int32_t iters, double lp_norm, double beta,
                                             double kappa, rl_stream_t stream);

/* Read-only device views of one exit linear in the interchange format:
 * qweight [N][K/8] uint32, scales [N][ceil(K/128)] fp16 bits,
 * zeros [N][ceil(K/128)] fp16 bits, rows in the caller's original order.
 * Valid until rl_model_destroy.  RL_ERR_STATE before quantization. */
RL_API rl_status rl_exit_layer_view(const rl_model* m, int32_t layer, int32_t which_linear,
                             const uint32_t** qweight, const uint16_t** scales,
                             const uint16_t** zeros, int32_t* n_rows, int32_t* n_cols);

/* Backbone offloading (explainer section 五: once the exit river is built,
 * deep backbone layers run only on the steps that do not exit before them,
 * so their weights can live in host memory).  Moves the bf16 backbone
 * weights of layers first_layer..L-1 (0-based) to pinned host memory (the
 * Grace CPU's, reached over NVLink-C2C on GB300) and frees their device
 * copies; the exit river, embedding, norms and LM head stay on the device,
 * plus one device buffer the size of one layer's backbone weights.  A step
 * reads an offloaded layer's weights from host memory only when it runs that
 * layer on the backbone: the persistent step kernel copies them straight
 * into its ring; the other paths (prefill, batches) first copy the layer
 * into the device buffer, a copy skipped on the device when the layer runs
 * on the exit river.  Results are unchanged; such steps are slower by the
 * host-memory transfer.  Needs the exit river (RL_ERR_STATE otherwise; it is
 * built from the device copies), once per model (RL_ERR_STATE after);
 * first_layer == L offloads nothing.  RL_ERR_OOM if pinned host memory runs
 * out (nothing is moved then).  Waits for `stream`; decode graphs captured
 * before are captured again at their next step. */
RL_API rl_status rl_model_offload_backbone(rl_model* m, int32_t first_layer, rl_stream_t stream);

/* Device and pinned host bytes the model holds (weights, exit river,
 * staging), excluding every rl_kv. */
RL_API rl_status rl_model_memory(const rl_model* m, uint64_t* device_bytes, uint64_t* host_bytes);

/* Exit-vs-backbone K/V similarity, a diagnostic (explainer section 三: the
 * K/V an exit layer writes into the backbone's slot stays close to what the
 * backbone layer would have written).  For B residual rows d_h [B][d_model]
 * (fp32, device, caller-owned) entering layer `layer` (0-based), both weight
 * sets of that layer project the same RMSNorm'd row to K and V; d_cos
 * [B][2][n_kv_heads] (fp32, device, caller-owned) receives, per sequence, the
 * cosine between the exit layer's and the backbone layer's K (index 0) and V
 * (index 1) of every KV head.  RoPE rotates both keys of a head alike at any
 * position, so the result does not depend on the position.  RL_ERR_STATE
 * before the exit river is built; RL_ERR_INVALID_ARG for a bad layer, batch
 * or pointer.  Enqueued on `stream`. */
RL_API rl_status rl_exit_kv_cosine(const rl_model* m, int32_t layer, const float* d_h, int32_t B,
                                   float* d_cos, rl_stream_t stream);

/* Save / load the exit river in the published packing (per layer and linear,
 * in RL_WQ .. RL_WD order: qweight [N][K/8] u32, scales and zeros [N][G] fp16
 * bits).  File: the 8 bytes "RLW4EXIT", u32 version (1), u32 n_layers,
 * d_model, n_q_heads, n_kv_heads, head_dim, ffn_dim, group_size, then per
 * (layer, linear) u32 N, u32 K and the three arrays; host byte order.
 * rl_save_exit_layers needs a built exit river (RL_ERR_STATE otherwise) and
 * returns when the file is written.  rl_load_exit_layers builds the exit
 * river from such a file instead of rl_quantize_exit_layers (a model's exit
 * river is built once: RL_ERR_STATE if it exists); a file that cannot be read
 * or does not match the model's shape returns RL_ERR_INVALID_ARG and leaves
 * the model unchanged.  It returns when the exit river is ready.  Not on the
 * pages (section 三 builds exit layers in under a minute); it skips the
 * quantizer for a model whose exit layers were already built. */
RL_API rl_status rl_save_exit_layers(const rl_model* m, const char* path);
RL_API rl_status rl_load_exit_layers(rl_model* m, const char* path, rl_stream_t stream);

/* kv_cache_alloc: one shared cache per layer (explainer sections 三, 六: exit
 * and backbone layers use the same slots; no duplicate cache), bf16
 * K and V each [max_batch][n_kv_heads][max_seq][head_dim], plus the decode
 * workspace for up to max_batch sequences.  Position starts at 0. */
RL_API rl_status rl_kv_cache_alloc(const rl_model* m, int32_t max_batch, int32_t max_seq, rl_kv** out);
RL_API rl_status rl_kv_cache_free(rl_kv* kv);

/* Device pointers of layer `layer`'s K and V cache (layout above). */
RL_API rl_status rl_kv_view(const rl_kv* kv, int32_t layer, const void** d_k, const void** d_v);

/* Host-side view of the next write position (all sequences share it). */
RL_API rl_status rl_kv_position(const rl_kv* kv, int32_t* pos, int32_t* decode_step);

/* Rewind/advance the write position and the decode-step counter used by
 * forced schedules.  Slots >= pos are simply overwritten later.  Enqueued on
 * `stream`. */
RL_API rl_status rl_kv_set_position(rl_kv* kv, int32_t pos, int32_t decode_step, rl_stream_t stream);

/* Optional debug trace: when d_hidden is non-NULL, every later prefill/decode
 * call writes the fp32 residual stream of the last position of each sequence
 * after the embedding and after every layer: d_hidden [L+1][max_batch][d].
 * NULL switches it off. */
RL_API rl_status rl_kv_set_trace(rl_kv* kv, float* d_hidden);

/* Which kernels run a decode step.  RL_PATH_STEP: one persistent cooperative
 * kernel per step (batch <= 8, shapes whose activations and weight ring fit in
 * shared memory, GQA ratio 1, 2 or 4, head_dim 64 or 128); RL_PATH_FUSED: five
 * launches per layer plus the LM head (batch <= 8); RL_PATH_GENERIC: eight
 * to eleven launches per layer (tensor-core GEMMs from 16 tokens, streaming
 * attention), any batch.  RL_PATH_AUTO (default) takes the first that
 * fits, in that order.  A forced path that does not fit a call's batch makes
 * that rl_decode_step return RL_ERR_UNSUPPORTED.  The math is the same on
 * every path (explainer sections 三, 四); they differ in rounding order only. */
enum { RL_PATH_AUTO = 0, RL_PATH_STEP = 1, RL_PATH_FUSED = 2, RL_PATH_GENERIC = 3 };
RL_API rl_status rl_kv_set_decode_path(rl_kv* kv, int32_t path);
/* The path a decode step of batch B would take (-1: none fits the forced path,
 * or bad arguments). */
RL_API int32_t rl_kv_decode_path(const rl_kv* kv, int32_t B);

/* prefill (explainer section 五, sequence-level exit): run d_tokens [B][T]
 * (device int32) at positions 0..T-1, resetting the cache position to 0 and the
 * decode-step counter to 0; one exit decision for all B*T tokens.
 * Outputs (device, caller-owned): d_logits [B][vocab] fp32 of the last
 * position; d_next_token [B] (greedy argmax, ties to the lowest id; may be
 * NULL); d_exit_layer [1]; d_min_cos [L] (batch-minimum cosine of every layer;
 * may be NULL).  Requires B <= max_batch and T < max_seq. */
RL_API rl_status rl_prefill(rl_model* m, rl_kv* kv, const int32_t* d_tokens, int32_t B, int32_t T,
                     const rl_exit_policy* policy, float* d_logits, int32_t* d_next_token,
                     int32_t* d_exit_layer, float* d_min_cos, rl_stream_t stream);

/* decode_step (explainer sections 四, 五: token-level exit per generation
 * step, minimum over the batch): one token per sequence, d_tokens [B], at the
 * current position p; writes K/V slot p of every layer (backbone or exit
 * layer, same slot) and advances p.  Outputs as rl_prefill.  The step runs as
 * one CUDA graph launch (captured on the first call for a given batch, policy
 * and set of buffers); the exit decision never returns to the host.
 * RL_ERR_CAPACITY if p + 1 > max_seq. */
RL_API rl_status rl_decode_step(rl_model* m, rl_kv* kv, const int32_t* d_tokens, int32_t B,
                         const rl_exit_policy* policy, float* d_logits, int32_t* d_next_token,
                         int32_t* d_exit_layer, float* d_min_cos, rl_stream_t stream);

/* decode_step with HOST buffers (end-to-end form): copies h_tokens [B] to the
 * device, runs rl_decode_step, copies back h_next_token [B], h_exit_layer [1]
 * and, if non-NULL, h_logits [B][vocab] and h_min_cos [L], then waits for the
 * stream.  Host buffers should be pinned for asynchronous copies. */
RL_API rl_status rl_decode_step_host(rl_model* m, rl_kv* kv, const int32_t* h_tokens, int32_t B,
                              const rl_exit_policy* policy, float* h_logits,
                              int32_t* h_next_token, int32_t* h_exit_layer, float* h_min_cos,
                              rl_stream_t stream);

/* Wait for `stream`, then report and clear the device error word of `kv`
 * (RL_ERR_DEVICE with the bits in rl_last_error()); kv may be NULL. */
RL_API rl_status rl_sync(rl_model* m, rl_kv* kv, rl_stream_t stream);

/* Kernel kinds reported by rl_kv_profile. */
enum {
  RL_K_EMBED = 0,      /* embedding gather + first RMSNorm (+ step begin) */
  RL_K_QKV = 1,        /* fused QKV projection + RoPE + KV append (GEMV kernel) */
  RL_K_ATTN = 2,       /* decode attention over the shared cache (split + combine) */
  RL_K_GSUM = 3,       /* per-group activation sums for the W4 path */
  RL_K_O = 4,          /* O projection + residual (GEMV kernel) */
  RL_K_NORM = 5,       /* pre-FFN RMSNorm */
  RL_K_GU = 6,         /* fused gate/up projection + SwiGLU (GEMV kernel) */
  RL_K_DOWN = 7,       /* down projection + residual (GEMV kernel) */
  RL_K_LAYER_END = 8,  /* cosine, batch-min, tau compare, next RMSNorm */
  RL_K_LM_HEAD = 9,    /* LM head (GEMV kernel) */
  RL_K_ARGMAX = 10,
  RL_K_STEP = 11       /* the whole persistent decode-step kernel (B <= 8); the
                          phase records before it come from its in-kernel timeline:
                          first start to last end of each phase over all CTAs */
};

/* Live per-kernel timing of decode steps: when enabled, the captured decode
 * graph also holds CUDA event records around every kernel (a little slower;
 * use it for a separate measurement pass).  rl_kv_profile waits for `stream`
 * and returns, for the last decode step, up to `cap` records: kind, the layer
 * (1-based, 0 outside layers), the path the GEMV kernels took (0 = bf16
 * backbone, 1 = W4 exit river, -1 = not a projection), milliseconds, and the
 * algorithmic bytes of the launch (weights and scales of the chosen path;
 * K/V rows 0..p for attention).  *n receives the record count. */
RL_API rl_status rl_kv_set_profiling(rl_kv* kv, int32_t enable);
RL_API rl_status rl_kv_profile(rl_kv* kv, rl_stream_t stream, int32_t cap, int32_t* kinds,
                               int32_t* layers, int32_t* paths, float* ms, double* bytes,
                               int32_t* n);

/* Per-CTA timeline of the last profiled decode step of the persistent step
 * kernel (rl_kv_set_profiling(kv, 2) records it; level 1 does not).  Waits for
 * `stream`, then copies into the host buffer `out` (capacity `cap` entries)
 * the globaltimer stamps, in nanoseconds, laid out [phase][CTA][stamp]: for
 * each phase of the step and each CTA, *nstamps values (0 = the event did not
 * happen on that CTA): 0 previous phase complete, 1 activation rows (or the
 * first attention chunk) in shared memory, 2 first weight unit in shared
 * memory, 3 last tile computed, 4 arrival at the phase counter, 5 / 6 first /
 * last weight copy issued by the producer, 7 RMSNorm scale and exit decision
 * ready.  RL_ERR_STATE if the last step did not record one; RL_ERR_INVALID_ARG
 * if `cap` < phases x CTAs x stamps.  Measurement only: not part of the
 * method (the pages time only whole decode steps). */
RL_API rl_status rl_kv_timeline(rl_kv* kv, rl_stream_t stream, int64_t cap, uint64_t* out,
                                int32_t* nphase, int32_t* nctas, int32_t* nstamps);

/* Failure injection for tests (the pages describe no failure handling; these
 * make the library's own failure paths run without faulting a GPU).
 *
 * rl_kv_set_wait_limit: from the next decode step or prefill on `kv` (a
 * decode graph is captured again), the persistent step kernel's grid-wide
 * phase barrier and the tensor-core GEMM's first accumulator wait give up
 * after `polls` polls (0 restores the kernels' own limits, about a second
 * or more).  A wait that gives up sets RL_DEVERR_TIMEOUT; the kernel then
 * finishes its phases without computing, waits (with its own limits) for
 * every copy and tensor-core operation it issued, frees its tensor memory
 * and exits, so rl_sync reports RL_ERR_DEVICE and the context stays usable.
 * The step's outputs and its K/V slot are then invalid: rewind the position
 * (rl_kv_set_position) and run the step again.
 *
 * rl_debug_fail_allocations: the next `after` device allocations made by
 * the library succeed and every later one fails as if cudaMalloc had
 * (RL_ERR_OOM), until it is called with a negative value (the default: no
 * injection).  Process-wide; not thread-safe with respect to concurrent
 * allocating calls. */
RL_API rl_status rl_kv_set_wait_limit(rl_kv* kv, int64_t polls);
RL_API rl_status rl_debug_fail_allocations(int64_t after);

/* Number of kernels one decode step launches for batch B (for launch
 * accounting); 0 on bad arguments. */
RL_API int32_t rl_decode_kernel_count(const rl_model* m, int32_t B);

/* rl_lm_head_static: final RMSNorm + LM head + greedy argmax of B residual
 * rows, for callers that must not allocate device memory.  The pages have no
 * counterpart to this call: it is the decode step's last kernel offered on
 * its own, with all of its working memory in one fixed static device array
 * inside the library (about 209 KiB), so the call allocates nothing and needs
 * no rl_kv.  Callers that cannot allocate: code running while another
 * framework captures a CUDA graph (an allocation is not capturable), serving
 * loops with a fixed memory pool, and latency-critical paths where
 * cudaMalloc / cudaFree would synchronise the device.
 *   d_h          [B][d_model] fp32 residual rows (device, caller-owned)
 *   d_logits     [B][vocab] fp32 out (device, caller-owned)
 *   d_next_token [B] int32 out, ties to the lowest id (device; may be NULL)
 *   d_err        [1] int32 out: RL_DEVERR_* bits of this call (device; may be NULL)
 * Limits: 1 <= B <= 8, d_model <= 8192, vocab and d_model multiples of 16,
 * and the B rows must fit in the kernel's shared memory next to its weight
 * ring: B * (2*Kp + 64 + Kp/32) <= 115,712 bytes with Kp = d_model rounded up
 * to 128, i.e. every B <= 8 up to d_model 7040, and B <= 6 at d_model 8192.
 * Beyond them the call returns RL_ERR_UNSUPPORTED and enqueues nothing.
 * The first call on each device resolves the array's device address with that
 * device current; make that first call before any stream capture on the
 * device.  Every call shares the one array: calls that overlap on the GPU
 * (different streams or threads) race on it; calls on one stream are safe. */
RL_API rl_status rl_lm_head_static(const rl_model* m, const float* d_h, int32_t B,
                                   float* d_logits, int32_t* d_next_token, int32_t* d_err,
                                   rl_stream_t stream);

#ifdef __cplusplus
}
#endif
#endif /* RIVER_H */
