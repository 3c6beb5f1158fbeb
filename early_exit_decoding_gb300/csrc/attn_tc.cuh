// Tensor-core attention over one chunk of K/V rows staged in shared memory
// by TMA (16-row x 64-dim boxes, 128-byte swizzle): shared by the persistent
// decode-step kernel and the streaming decode-attention kernel.
#pragma once

#include "dev_common.cuh"

namespace river {
namespace attn {

using namespace dev;

// Byte offset of 16-byte chunk c of K/V row r in an attention chunk staged by
// TMA with the 128-byte swizzle: 64-dim halves of 128 rows x 128 bytes at
// 16 KB apart, chunk c & 7 of a row stored at (c & 7) ^ (r & 7).
__device__ __forceinline__ uint32_t kv_off(int r, int c) {
  return (uint32_t)((c >> 3) * 16384 + r * 128 + (((c & 7) ^ (r & 7)) << 4));
}

// A operand of m16n8k16 for one 16-dim k-step of q (rows = the REP query
// heads; rows >= REP zero) from q staged in shared memory (fp32 [REP][HDC],
// scaled by 1/sqrt(hd)), split into bf16 hi + lo parts: a[0..1] = a0 hi / lo,
// a[2..3] = a2 hi / lo.
template <int REP, int HDC>
__device__ __forceinline__ void q_frag(const float* qs, int ks, int g, int t, uint32_t (&a)[4],
                                       float qscale = 1.f) {
  float2 lo = make_float2(0.f, 0.f), hi = lo;
  if (g < REP) {
    lo = *reinterpret_cast<const float2*>(qs + g * HDC + ks * 16 + 2 * t);
    hi = *reinterpret_cast<const float2*>(qs + g * HDC + ks * 16 + 8 + 2 * t);
    lo.x *= qscale;
    lo.y *= qscale;
    hi.x *= qscale;
    hi.y *= qscale;
  }
  split_bf16x2(lo.x, lo.y, a[0], a[1]);
  split_bf16x2(hi.x, hi.y, a[2], a[3]);
}

// One warp's share of an attention chunk on the tensor cores: positions
// j0 .. j0 + jn - 1 (jn <= 16; two 8-position n-tiles) against the REP query
// heads of one KV head.  S = q K^T and O = P V run as m16n8k16 MMAs (q and P
// split into bf16 hi + lo: fp32-level accuracy; q from shared memory, times
// qscale); K / V
// fragments come from the
// swizzled chunk by ldmatrix (V transposed), conflict free.  After S, a
// barrier of the consumer warps (every warp is done reading K) frees the K
// rows, which then hold the warps' partials: per head (max, sum, o[hd]) at w0,
// o written 64 dims at a time.
template <int REP, int HDC>
__device__ __forceinline__ void attn_warp_tc(const unsigned char* Ks, const unsigned char* Vs, int j0, int jn,
                                             const float* qs, int lane, float* w0, float qscale = 1.f) {
  constexpr int WS = 2 + HDC;
  const int g = lane >> 2, t = lane & 3;
  const int mi = lane >> 3, ri = lane & 7;
  float sacc[2][4];
#pragma unroll
  for (int n = 0; n < 2; ++n)
#pragma unroll
    for (int i = 0; i < 4; ++i) sacc[n][i] = 0.f;
  if (jn > 0) {  // uniform over the warp
    // S: ldmatrix x4 = K rows j0 .. j0 + 15 x 16 dims -> b0 / b1 of both n-tiles
    const uint32_t kb = smem_u32(Ks);
    const int row = j0 + (mi >> 1) * 8 + ri;
#pragma unroll
    for (int ks = 0; ks < HDC / 16; ++ks) {
      uint32_t kf[4], qa[4];
      ldsm_x4(kf, kb + kv_off(row, ks * 2 + (mi & 1)));
      q_frag<REP, HDC>(qs, ks, g, t, qa, qscale);
#pragma unroll
      for (int n = 0; n < 2; ++n) {
        mma_bf16(sacc[n], qa[0], 0u, qa[2], 0u, kf[2 * n], kf[2 * n + 1]);
        mma_bf16(sacc[n], qa[1], 0u, qa[3], 0u, kf[2 * n], kf[2 * n + 1]);
      }
    }
  }
  // row g's scores at positions 2t, 2t + 1 (n-tile 0) and 8 + 2t, 9 + 2t (n-tile 1)
  const float sv[4] = {sacc[0][0], sacc[0][1], sacc[1][0], sacc[1][1]};
  const int pidx[4] = {2 * t, 2 * t + 1, 8 + 2 * t, 9 + 2 * t};
  float m = -FLT_MAX;
#pragma unroll
  for (int i = 0; i < 4; ++i)
    if (pidx[i] < jn) m = fmaxf(m, sv[i]);
  m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, 1));
  m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, 2));
  float pv[4], l = 0.f;
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    pv[i] = pidx[i] < jn ? __expf(sv[i] - m) : 0.f;
    l += pv[i];
  }
  l += __shfl_xor_sync(0xffffffffu, l, 1);
  l += __shfl_xor_sync(0xffffffffu, l, 2);
  uint32_t pa0h, pa0l, pa2h, pa2l;
  split_bf16x2(pv[0], pv[1], pa0h, pa0l);
  split_bf16x2(pv[2], pv[3], pa2h, pa2l);
  dev::named_sync(1, 8 * 32);  // K is no longer read: the partials may overlay it
  float* wr = w0 + g * WS;
  if (g < REP && t == 0) {
    wr[0] = m;
    wr[1] = l;
  }
  // O = P V, 64 dims at a time: ldmatrix x4 trans = V rows j0 .. j0 + 15 x 16
  // dims -> b0 / b1 of two 8-dim n-tiles
  const uint32_t vb = smem_u32(Vs);
  const int vrow = j0 + (mi & 1) * 8 + ri;
#pragma unroll
  for (int hh = 0; hh < HDC / 64; ++hh) {
    float o[8][4];
#pragma unroll
    for (int n = 0; n < 8; ++n)
#pragma unroll
      for (int i = 0; i < 4; ++i) o[n][i] = 0.f;
    if (jn > 0) {
#pragma unroll
      for (int nd = 0; nd < 8; nd += 2) {
        uint32_t vf[4];
        ldsm_x4_t(vf, vb + kv_off(vrow, hh * 8 + nd + (mi >> 1)));
#pragma unroll
        for (int h = 0; h < 2; ++h) {
          mma_bf16(o[nd + h], pa0h, 0u, pa2h, 0u, vf[2 * h], vf[2 * h + 1]);
          mma_bf16(o[nd + h], pa0l, 0u, pa2l, 0u, vf[2 * h], vf[2 * h + 1]);
        }
      }
    }
    if (g < REP) {
#pragma unroll
      for (int nd = 0; nd < 8; ++nd) {
        wr[2 + hh * 64 + nd * 8 + 2 * t] = o[nd][0];
        wr[2 + hh * 64 + nd * 8 + 2 * t + 1] = o[nd][1];
      }
    }
  }
}

}  // namespace attn
}  // namespace river
