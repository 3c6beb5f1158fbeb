// Exit-vs-backbone K/V similarity (River-LLM explainer, section 三: an exit
// layer writes K/V into the backbone's own cache slot, and what it writes
// stays close to what the backbone layer would have written there).
//
// For residual rows h entering a layer, both weight sets project the same
// normalised row x = h / rms(h) * g_attn to K and V; the cosine between the
// two, per sequence and KV head, is the diagnostic.  The RMSNorm factor is
// one positive scalar per row and RoPE rotates both keys of a head by the
// same orthogonal map at any position, so neither changes the cosine: the
// kernel projects x' = h * g_attn and skips RoPE.  The fused QKV matrix holds
// each head's rows contiguously (dims permuted within the head, the same way
// for both weight sets), so a head's cosine is taken over its rows as stored.
//
// One CTA per (sequence, K or V, KV head); one warp per output row at a time.
#include "internal.h"

namespace river {

namespace {

constexpr int kKvcThreads = 256;

__global__ void __launch_bounds__(kKvcThreads) k_exit_kv_cosine(
    const float* __restrict__ h, int d, const float* __restrict__ g, const bf16* __restrict__ w,
    const uint32_t* __restrict__ qw, const __half2* __restrict__ sz, int Kp, int Hq, int Hkv,
    int hd, float* __restrict__ out) {
  extern __shared__ float xs[];  // x' = h * g, zero beyond d: [Kp]
  __shared__ float red[3][kKvcThreads / 32];
  const int hk = blockIdx.x % Hkv, which = (blockIdx.x / Hkv) & 1, b = blockIdx.x / (2 * Hkv);
  for (int k = threadIdx.x; k < Kp; k += blockDim.x)
    xs[k] = k < d ? h[(size_t)b * d + k] * g[k] : 0.f;
  __syncthreads();
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31, G = Kp / kGroup;
  const int row0 = (Hq + which * Hkv + hk) * hd;
  float pbe = 0.f, pbb = 0.f, pee = 0.f;
  for (int j = warp; j < hd; j += kKvcThreads / 32) {
    const int r = row0 + j;
    const bf16* wr = w + (size_t)r * Kp;
    const uint32_t* qr = qw + (size_t)r * (Kp / 8);
    float yb = 0.f, ye = 0.f;
    for (int c = lane; c < Kp / 8; c += 32) {  // 8 inputs per lane and step
      const uint4 wv = *reinterpret_cast<const uint4*>(wr + c * 8);
      const uint32_t q = qr[c];
      const __half2 s_z = sz[(size_t)r * G + (c * 8) / kGroup];
      const float s = __low2float(s_z), z = __high2float(s_z);
      const __nv_bfloat162* w2 = reinterpret_cast<const __nv_bfloat162*>(&wv);
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        const float2 f = __bfloat1622float2(w2[i]);
        const float x0 = xs[c * 8 + 2 * i], x1 = xs[c * 8 + 2 * i + 1];
        yb += f.x * x0 + f.y * x1;
        const float q0 = (float)((q >> (8 * i)) & 0xFu), q1 = (float)((q >> (8 * i + 4)) & 0xFu);
        ye += (q0 - z) * s * x0 + (q1 - z) * s * x1;
      }
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
      yb += __shfl_xor_sync(0xffffffffu, yb, o);
      ye += __shfl_xor_sync(0xffffffffu, ye, o);
    }
    pbe += yb * ye;
    pbb += yb * yb;
    pee += ye * ye;
  }
  if (lane == 0) {
    red[0][warp] = pbe;
    red[1][warp] = pbb;
    red[2][warp] = pee;
  }
  __syncthreads();
  if (threadIdx.x == 0) {
    float be = 0.f, bb = 0.f, ee = 0.f;
    for (int i = 0; i < kKvcThreads / 32; ++i) {
      be += red[0][i];
      bb += red[1][i];
      ee += red[2][i];
    }
    out[blockIdx.x] = be / fmaxf(sqrtf(bb) * sqrtf(ee), 1e-12f);
  }
}

}  // namespace

cudaError_t launch_exit_kv_cosine(const float* h, int B, int d, const float* g, const bf16* w,
                                  const uint32_t* qw, const __half2* sz, int Kp, int Hq, int Hkv,
                                  int hd, float* out, cudaStream_t s) {
  const size_t smem = (size_t)Kp * sizeof(float);
  if (smem > 48 * 1024) {
    const cudaError_t e = cudaFuncSetAttribute(k_exit_kv_cosine,
                                               cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
  }
  k_exit_kv_cosine<<<B * 2 * Hkv, kKvcThreads, smem, s>>>(h, d, g, w, qw, sz, Kp, Hq, Hkv, hd, out);
  return cudaGetLastError();
}

}  // namespace river
