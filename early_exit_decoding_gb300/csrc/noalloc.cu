// rl_lm_head_static: the decode step's last kernel (final RMSNorm, LM head,
// greedy argmax) for callers that must not allocate device memory.
//
// Who cannot allocate: code that runs while another framework captures a
// CUDA graph (cudaMalloc is not a capturable operation, and a capture that
// meets one is invalidated), serving loops that own a fixed device-memory
// pool and forbid allocation after start-up, and latency-critical paths where
// cudaMalloc / cudaFree would synchronise the device.  This entry point needs
// no rl_kv: all of its working memory is one file-scope static device array,
// whose size is fixed when the library is loaded.
//
// Limits: batch <= 8 rows, d_model <= 8192, at most 1024 CTAs in the LM-head
// launch (one per streaming multiprocessor at most), and the rows must fit in
// shared memory beside the GEMV kernel's weight ring: B * (2*Kp + 64 + Kp/32)
// <= 115,712 bytes (Kp = d_model rounded up to 128), so batch 8 up to
// d_model 7040 and batch 6 at d_model 8192.  Larger requests are rejected
// with RL_ERR_UNSUPPORTED before anything is enqueued.
//
// Every call shares the one array: two calls that overlap on the GPU (on
// different streams, or on different host threads) race on it and may
// return wrong results.  Calls on one stream are ordered and safe.
#include <cstring>
#include <mutex>

#include "internal.h"

namespace river {

namespace {

constexpr int kStaticMaxB = kFusedMaxB;  // rows per call
constexpr int kStaticMaxD = 8192;        // d_model (rounded up to 128)
constexpr int kStaticMaxGrid = 1024;     // CTAs of the LM-head launch

// Scratch layout, byte offsets from the start of the array (each 256-aligned).
constexpr size_t kOffX = 0;  // bf16 x' rows [kStaticMaxB][kStaticMaxD]
constexpr size_t kOffStats = kOffX + (size_t)kStaticMaxB * kStaticMaxD * 2;  // f32 [D/16][8]
constexpr size_t kOffAmVal = kOffStats + (size_t)(kStaticMaxD / 16) * 8 * 4;  // f32 [grid][8]
constexpr size_t kOffAmIdx = kOffAmVal + (size_t)kStaticMaxGrid * 8 * 4;      // i32 [grid][8]
constexpr size_t kOffTicket = kOffAmIdx + (size_t)kStaticMaxGrid * 8 * 4;     // u32
constexpr size_t kOffState = kOffTicket + 256;                                // DevState
constexpr size_t kScratchBytes = kOffState + 256;                             // 213,504 bytes

static __device__ __align__(256) unsigned char g_lm_scratch[kScratchBytes];

// Device address of g_lm_scratch per device, resolved once per device.
constexpr int kMaxDevices = 64;
std::mutex g_mu;
unsigned char* g_ptr[kMaxDevices] = {};

// x'[b][k] = bf16(h[b][k] * g[k]) (zero beyond d) and the per-16-row-tile
// sums of h^2 that the LM-head kernel turns into the RMSNorm scale.  Block 0
// also clears what must start at zero: the CTA ticket and the device state.
__global__ void k_lm_static_prep(const float* __restrict__ h, int ldh, const float* __restrict__ g,
                                 int d, int Kp, unsigned char* __restrict__ scratch) {
  const int b = blockIdx.x;
  bf16* x = reinterpret_cast<bf16*>(scratch + kOffX) + (size_t)b * Kp;
  float* stats = reinterpret_cast<float*>(scratch + kOffStats);
  const float* hb = h + (size_t)b * ldh;
  for (int t = threadIdx.x; t < Kp / 16; t += blockDim.x) {
    float ss = 0.f;
    for (int i = 0; i < 16; ++i) {
      const int k = t * 16 + i;
      float v = 0.f, xv = 0.f;
      if (k < d) {
        v = hb[k];
        xv = v * g[k];
      }
      ss += v * v;
      x[k] = __float2bfloat16_rn(xv);
    }
    if (t < d / 16) stats[(size_t)t * 8 + b] = ss;
  }
  if (b == 0 && threadIdx.x == 0) {
    *reinterpret_cast<unsigned int*>(scratch + kOffTicket) = 0u;
    DevState* st = reinterpret_cast<DevState*>(scratch + kOffState);
    st->pos = 0;
    st->step = 0;
    st->exit_layer = 0;
    st->err = 0;
    st->ticket = 0u;
  }
}

__global__ void k_lm_static_status(const unsigned char* __restrict__ scratch, int32_t* err) {
  *err = reinterpret_cast<const DevState*>(scratch + kOffState)->err;
}

}  // namespace

}  // namespace river

using namespace river;

extern "C" rl_status rl_lm_head_static(const rl_model* m, const float* d_h, int32_t B,
                                       float* d_logits, int32_t* d_next_token, int32_t* d_err,
                                       rl_stream_t stream) {
  if (!m || !d_h || !d_logits) return set_error(RL_ERR_INVALID_ARG, "NULL argument");
  const LmHeadView v = lm_head_view(m);
  if (B < 1 || B > kStaticMaxB)
    return set_error(RL_ERR_UNSUPPORTED, "rl_lm_head_static: batch must be in [1, 8]");
  if (v.Kd > kStaticMaxD)
    return set_error(RL_ERR_UNSUPPORTED, "rl_lm_head_static: d_model above 8192");
  if (v.d % 16 || v.V % 16)
    return set_error(RL_ERR_UNSUPPORTED, "rl_lm_head_static: d_model and vocab must be multiples of 16");

  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) {
    cudaGetLastError();
    return set_error(RL_ERR_CUDA, "rl_lm_head_static: no current device");
  }
  unsigned char* scratch = nullptr;
  {
    // Set-up, once per device, with that device current.  The first call on a
    // device must come before any stream capture on it: resolving the symbol
    // can load the module, which a capturing stream does not allow.
    std::lock_guard<std::mutex> lock(g_mu);
    if (!g_ptr[dev]) {
      void* p = nullptr;
      const cudaError_t e = cudaGetSymbolAddress(&p, g_lm_scratch);
      if (e != cudaSuccess || !p) {
        cudaGetLastError();
        return set_error(RL_ERR_CUDA, "rl_lm_head_static: cudaGetSymbolAddress failed");
      }
      g_ptr[dev] = static_cast<unsigned char*>(p);
    }
    scratch = g_ptr[dev];
  }

  FusedArgs a;
  memset(&a, 0, sizeof(a));
  a.w = v.w;
  a.N = v.V;
  a.Kp = v.Kd;
  a.w4_mode = W4_OFF;
  a.layer_no = 0;
  a.st = reinterpret_cast<DevState*>(scratch + kOffState);
  a.B = B;
  a.xmode = X_SCALED;
  a.xg = reinterpret_cast<const bf16*>(scratch + kOffX);
  a.ldxg = v.Kd;
  a.stats_in = reinterpret_cast<const float*>(scratch + kOffStats);
  a.stats_tiles = v.d / 16;
  a.stats_k = 1;
  a.d = v.d;
  a.eps = v.eps;
  a.dec_layer = 0;  // no exit decision here
  a.L = v.L;
  a.mode = RL_EXIT_TAU;
  a.tau = 2.f;
  a.schedule_len = 1;
  a.epi = EPI_LMHEAD;
  a.out = d_logits;
  a.ldo = v.V;
  a.am_val = reinterpret_cast<float*>(scratch + kOffAmVal);
  a.am_idx = reinterpret_cast<int*>(scratch + kOffAmIdx);
  a.next_token = d_next_token;
  a.cta_ticket = reinterpret_cast<unsigned*>(scratch + kOffTicket);
  // Whole 16-row tiles per CTA: no tile is split, so the split-tile merge
  // (ws, tile_ticket) is never reached.
  a.ws = nullptr;
  a.tile_ticket = nullptr;
  if (fused_grid(a, v.sm_count) > kStaticMaxGrid)
    return set_error(RL_ERR_UNSUPPORTED, "rl_lm_head_static: more than 1024 CTAs");
  if (fused_smem_bytes(a) > 220 * 1024)
    return set_error(RL_ERR_UNSUPPORTED, "rl_lm_head_static: rows do not fit in shared memory");

  cudaStream_t s = static_cast<cudaStream_t>(stream);
  k_lm_static_prep<<<B, 256, 0, s>>>(d_h, v.d, v.g_final, v.d, v.Kd, scratch);
  cudaError_t e = cudaGetLastError();
  if (e == cudaSuccess) e = launch_gemv_fused(a, v.sm_count, false, s);
  if (e == cudaSuccess && d_err) {
    k_lm_static_status<<<1, 1, 0, s>>>(scratch, d_err);
    e = cudaGetLastError();
  }
  if (e != cudaSuccess) return set_error(RL_ERR_CUDA, cudaGetErrorString(e));
  return RL_OK;
}
