// quantize_exit_layers: build the exit river (River-LLM explainer, section
// 三: each exit layer is a training-free copy of the backbone layer's
// parameters, shrunk to 4-bit weights with 16-bit activations).
//
// Per group of 128 consecutive inputs of a row (the last group of a row whose
// width is not a multiple of 128 covers the remainder), min-max
// round-to-nearest with a float zero point, each step one IEEE fp32 operation
// (no contraction) and fp16 rounding where the value is stored:
//   s = fp16((max - min) / 15), or 1.0 if max == min or s rounds to 0
//   z = fp16(-min / s)
//   q = clamp(rint(w / s + z), 0, 15)       rint: round half to even
// One warp per (row, group); lane l holds inputs 4l..4l+3 of the group.
#include <float.h>

#include "internal.h"

namespace river {

namespace {

__global__ void k_quantize(const bf16* __restrict__ w, int N, int K, int Kp,
                           uint32_t* __restrict__ qw, __half2* __restrict__ sz,
                           const int2* __restrict__ rowmap, const NSView* __restrict__ views) {
  const int G = Kp / kGroup;
  const long long wid = ((long long)blockIdx.x * blockDim.x + threadIdx.x) >> 5;
  const int lane = threadIdx.x & 31;
  if (wid >= (long long)N * G) return;
  const int r = (int)(wid / G), gi = (int)(wid % G);
  const int k0 = gi * kGroup + 4 * lane;

  float v[4];
  bool valid[4];
  float mn = FLT_MAX, mx = -FLT_MAX;
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    valid[i] = (k0 + i) < K;
    v[i] = valid[i] ? __bfloat162float(w[(size_t)r * Kp + k0 + i]) : 0.f;
    if (valid[i]) {
      mn = fminf(mn, v[i]);
      mx = fmaxf(mx, v[i]);
    }
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
    mn = fminf(mn, __shfl_xor_sync(0xffffffffu, mn, o));
    mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, o));
  }
  __half s = __float2half_rn(__fdiv_rn(__fsub_rn(mx, mn), 15.0f));
  if (mx == mn || __half2float(s) == 0.0f) s = __float2half_rn(1.0f);
  const float sf = __half2float(s);
  const __half z = __float2half_rn(__fdiv_rn(-mn, sf));
  const float zf = __half2float(z);

  uint32_t v16 = 0;
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    uint32_t q = 0;
    if (valid[i]) {
      const float t = rintf(__fadd_rn(__fdiv_rn(v[i], sf), zf));
      q = (uint32_t)fminf(fmaxf(t, 0.0f), 15.0f);
    }
    v16 |= q << (4 * i);
  }
  const uint32_t hi = __shfl_down_sync(0xffffffffu, v16, 1);
  const int2 m = rowmap[r];
  const NSView view = views[m.x];
  if ((lane & 1) == 0) {
    const uint32_t word = v16 | (hi << 16);
    const int wi = gi * 16 + lane / 2;  // word index within the row
    qw[(size_t)r * (Kp / 8) + wi] = word;
    if (wi < K / 8) view.q[(size_t)m.y * (K / 8) + wi] = word;
  }
  if (lane == 0) {
    sz[(size_t)r * G + gi] = __halves2half2(s, z);
    const int Gv = (K + kGroup - 1) / kGroup;
    view.s[(size_t)m.y * Gv + gi] = __half_as_ushort(s);
    view.z[(size_t)m.y * Gv + gi] = __half_as_ushort(z);
  }
}

// The internal W4 layout of one fused matrix from the interchange views (the
// inverse of the view writes in k_quantize): row r from views[rowmap[r].x]
// row rowmap[r].y, words past K/8 zero, (scale, zero) per group.
__global__ void k_w4_from_views(int N, int K, int Kp, uint32_t* __restrict__ qw, __half2* __restrict__ sz,
                                const int2* __restrict__ rowmap, const NSView* __restrict__ views) {
  const int r = blockIdx.x;
  if (r >= N) return;
  const int2 m = rowmap[r];
  const NSView v = views[m.x];
  const int W = Kp / 8, Wv = K / 8, G = Kp / kGroup;
  for (int wi = threadIdx.x; wi < W; wi += blockDim.x)
    qw[(size_t)r * W + wi] = wi < Wv ? v.q[(size_t)m.y * Wv + wi] : 0u;
  for (int gi = threadIdx.x; gi < G; gi += blockDim.x)
    sz[(size_t)r * G + gi] = __halves2half2(__ushort_as_half(v.s[(size_t)m.y * G + gi]),
                                            __ushort_as_half(v.z[(size_t)m.y * G + gi]));
}

}  // namespace

void launch_quantize(const bf16* w, int N, int K, int Kp, uint32_t* qw, __half2* sz,
                     const int2* rowmap, const NSView* views, cudaStream_t s) {
  const long long warps = (long long)N * (Kp / kGroup);
  const long long blocks = (warps * 32 + 255) / 256;
  k_quantize<<<(unsigned)blocks, 256, 0, s>>>(w, N, K, Kp, qw, sz, rowmap, views);
}

void launch_w4_from_views(int N, int K, int Kp, uint32_t* qw, __half2* sz, const int2* rowmap,
                          const NSView* views, cudaStream_t s) {
  if (N > 0) k_w4_from_views<<<N, 128, 0, s>>>(N, K, Kp, qw, sz, rowmap, views);
}

}  // namespace river
