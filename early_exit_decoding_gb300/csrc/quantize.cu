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
//
// HQQ refinement (explainer section 六 names HQQ as the exit layers'
// quantizer; Badri and Shaji, "Half-Quadratic Quantization of Large Machine
// Learning Models", 2023): the min-max scale stays, and the zero point of
// each group is moved to lower sum |w - s (q - z)|^p (p < 1) by alternating,
// in float64 with every operation rounded once (no contraction):
//   q = clamp(rint(w / s + z), 0, 15),  r = w - s (q - z)
//   e = sign(r) max(|r| - |r|^(p-1) / beta, 0)        (0 where r == 0)
//   z = (sum over the group of q - (w - e) / s) / n,   beta *= kappa
// for a fixed number of iterations.  The stored zero is the fp16 value (the
// min-max one or an iteration's, rounded once from float64) whose stored
// codes give the lowest sum |w - s (q - z)|^p over the group, ties keeping
// the earlier; the codes then follow the min-max rule with that zero.
#include <float.h>

#include "internal.h"

namespace river {

namespace {

__device__ __forceinline__ double warp_sum_f64(double v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v = __dadd_rn(v, __shfl_xor_sync(0xffffffffu, v, o));
  return v;
}

// Stored code of input v for scale sf and zero zf (fp32, one rounding each).
__device__ __forceinline__ float code_of(float v, float sf, float zf) {
  const float t = rintf(__fadd_rn(__fdiv_rn(v, sf), zf));
  return fminf(fmaxf(t, 0.0f), 15.0f);
}

// sum over the group of |w - s (q - z)|^p with the stored codes of zero z16.
__device__ __forceinline__ double group_lp_error(const float (&v)[4], const bool (&valid)[4], float sf,
                                                 __half z16, double p) {
  const float zf = __half2float(z16);
  const double s64 = (double)sf, z64 = (double)zf;
  double acc = 0.0;
#pragma unroll
  for (int i = 0; i < 4; ++i)
    if (valid[i]) {
      const double q = (double)code_of(v[i], sf, zf);
      const double r = __dsub_rn((double)v[i], __dmul_rn(s64, __dsub_rn(q, z64)));
      acc = __dadd_rn(acc, pow(fabs(r), p));
    }
  return warp_sum_f64(acc);
}

template <bool kHqq>
__global__ void k_quantize(const bf16* __restrict__ w, int N, int K, int Kp,
                           uint32_t* __restrict__ qw, __half2* __restrict__ sz,
                           const int2* __restrict__ rowmap, const NSView* __restrict__ views,
                           HqqParams hp) {
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
  __half z = __float2half_rn(__fdiv_rn(-mn, sf));
  if (kHqq) {
    int n = 0;
#pragma unroll
    for (int i = 0; i < 4; ++i) n += valid[i] ? 1 : 0;
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) n += __shfl_xor_sync(0xffffffffu, n, o);
    const double s64 = (double)sf, pm1 = __dsub_rn(hp.p, 1.0);
    double zz = (double)__half2float(z), beta = hp.beta;
    __half best = z;
    double best_err = group_lp_error(v, valid, sf, z, hp.p);
    for (int it = 0; it < hp.iters; ++it) {
      double part = 0.0;
#pragma unroll
      for (int i = 0; i < 4; ++i)
        if (valid[i]) {
          const double wv = (double)v[i];
          const double q = fmin(fmax(rint(__dadd_rn(__ddiv_rn(wv, s64), zz)), 0.0), 15.0);
          const double r = __dsub_rn(wv, __dmul_rn(s64, __dsub_rn(q, zz)));
          const double ar = fabs(r);
          double e = 0.0;
          if (ar > 0.0) {
            const double sh = fmax(__dsub_rn(ar, __ddiv_rn(pow(ar, pm1), beta)), 0.0);
            e = r < 0.0 ? -sh : sh;
          }
          part = __dadd_rn(part, __dsub_rn(q, __ddiv_rn(__dsub_rn(wv, e), s64)));
        }
      zz = __ddiv_rn(warp_sum_f64(part), (double)n);
      beta = __dmul_rn(beta, hp.kappa);
      const __half zc = __double2half(zz);
      const double err = group_lp_error(v, valid, sf, zc, hp.p);
      if (err < best_err) {
        best_err = err;
        best = zc;
      }
    }
    z = best;
  }
  const float zf = __half2float(z);

  uint32_t v16 = 0;
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    uint32_t q = 0;
    if (valid[i]) q = (uint32_t)code_of(v[i], sf, zf);
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
                     const int2* rowmap, const NSView* views, const HqqParams* hqq, cudaStream_t s) {
  const long long warps = (long long)N * (Kp / kGroup);
  const long long blocks = (warps * 32 + 255) / 256;
  if (hqq)
    k_quantize<true><<<(unsigned)blocks, 256, 0, s>>>(w, N, K, Kp, qw, sz, rowmap, views, *hqq);
  else
    k_quantize<false><<<(unsigned)blocks, 256, 0, s>>>(w, N, K, Kp, qw, sz, rowmap, views, HqqParams{});
}

void launch_w4_from_views(int N, int K, int Kp, uint32_t* qw, __half2* sz, const int2* rowmap,
                          const NSView* views, cudaStream_t s) {
  if (N > 0) k_w4_from_views<<<N, 128, 0, s>>>(N, K, Kp, qw, sz, rowmap, views);
}

}  // namespace river
