// Tensor-core attention over one chunk of K/V rows staged in shared memory
// by TMA (boxes of 16 or 64 rows x 64 dims, 128-byte swizzle): shared by the
// persistent decode-step kernel and the streaming decode-attention kernel.
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

// Softmax weights of one warp's NB x 16 positions, as A operands of the
// P V MMAs (bf16 hi + lo of rows g, k-columns 2t, 2t + 1 and 8 + 2t, 9 + 2t
// of each 16-position block), with the warp's running max and sum.
template <int NB>
struct PFrag {
  uint32_t h0[NB], l0[NB], h2[NB], l2[NB];
  float m, l;
};

// S = q K^T for positions j0 .. j0 + jn - 1 of the chunk (16-position blocks
// b < NB; a block with no valid position is skipped, so rows past the staged
// boxes are never read), then the warp's online-softmax max, weights and sum.
// K fragments by ldmatrix from the swizzled chunk, q from shared memory split
// into bf16 hi + lo (fp32-level accuracy), times qscale.
template <int REP, int HDC, int NB>
__device__ __forceinline__ void attn_scores(const unsigned char* Ks, int j0, int jn, const float* qs,
                                            int lane, float qscale, PFrag<NB>& p) {
  const int g = lane >> 2, t = lane & 3;
  const int mi = lane >> 3, ri = lane & 7;
  float sacc[NB][2][4];
#pragma unroll
  for (int b = 0; b < NB; ++b)
#pragma unroll
    for (int n = 0; n < 2; ++n)
#pragma unroll
      for (int i = 0; i < 4; ++i) sacc[b][n][i] = 0.f;
  if (jn > 0) {  // uniform over the warp
    const uint32_t kb = smem_u32(Ks);
#pragma unroll
    for (int ks = 0; ks < HDC / 16; ++ks) {
      uint32_t qa[4];
      q_frag<REP, HDC>(qs, ks, g, t, qa, qscale);
#pragma unroll
      for (int b = 0; b < NB; ++b) {
        if (jn > 16 * b) {
          // ldmatrix x4 = K rows of the block x 16 dims -> b0 / b1 of both n-tiles
          uint32_t kf[4];
          ldsm_x4(kf, kb + kv_off(j0 + 16 * b + (mi >> 1) * 8 + ri, ks * 2 + (mi & 1)));
#pragma unroll
          for (int n = 0; n < 2; ++n) {
            mma_bf16(sacc[b][n], qa[0], 0u, qa[2], 0u, kf[2 * n], kf[2 * n + 1]);
            mma_bf16(sacc[b][n], qa[1], 0u, qa[3], 0u, kf[2 * n], kf[2 * n + 1]);
          }
        }
      }
    }
  }
  // row g's scores at positions 16b + 8n + 2t + {0, 1}
  float m = -FLT_MAX;
#pragma unroll
  for (int b = 0; b < NB; ++b)
#pragma unroll
    for (int n = 0; n < 2; ++n)
#pragma unroll
      for (int i = 0; i < 2; ++i)
        if (16 * b + 8 * n + 2 * t + i < jn) m = fmaxf(m, sacc[b][n][i]);
  m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, 1));
  m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, 2));
  float l = 0.f;
#pragma unroll
  for (int b = 0; b < NB; ++b) {
    float pv[2][2];
#pragma unroll
    for (int n = 0; n < 2; ++n)
#pragma unroll
      for (int i = 0; i < 2; ++i) {
        pv[n][i] = 16 * b + 8 * n + 2 * t + i < jn ? __expf(sacc[b][n][i] - m) : 0.f;
        l += pv[n][i];
      }
    split_bf16x2(pv[0][0], pv[0][1], p.h0[b], p.l0[b]);
    split_bf16x2(pv[1][0], pv[1][1], p.h2[b], p.l2[b]);
  }
  l += __shfl_xor_sync(0xffffffffu, l, 1);
  l += __shfl_xor_sync(0xffffffffu, l, 2);
  p.m = m;
  p.l = l;
}

// O = P V over the same positions, 64 dims at a time (ldmatrix x4 trans = V
// rows of a block x 16 dims -> b0 / b1 of two 8-dim n-tiles); row g's
// (max, sum, o[hd]) written at wr (rows g >= REP write nothing).
template <int REP, int HDC, int NB>
__device__ __forceinline__ void attn_values(const unsigned char* Vs, int j0, int jn, const PFrag<NB>& p,
                                            int lane, float* wr) {
  const int g = lane >> 2, t = lane & 3;
  const int mi = lane >> 3, ri = lane & 7;
  if (g < REP && t == 0) {
    wr[0] = p.m;
    wr[1] = p.l;
  }
  const uint32_t vb = smem_u32(Vs);
#pragma unroll
  for (int hh = 0; hh < HDC / 64; ++hh) {
    float o[8][4];
#pragma unroll
    for (int n = 0; n < 8; ++n)
#pragma unroll
      for (int i = 0; i < 4; ++i) o[n][i] = 0.f;
#pragma unroll
    for (int b = 0; b < NB; ++b) {
      if (jn > 16 * b) {
        const int vrow = j0 + 16 * b + (mi & 1) * 8 + ri;
#pragma unroll
        for (int nd = 0; nd < 8; nd += 2) {
          uint32_t vf[4];
          ldsm_x4_t(vf, vb + kv_off(vrow, hh * 8 + nd + (mi >> 1)));
#pragma unroll
          for (int h = 0; h < 2; ++h) {
            mma_bf16(o[nd + h], p.h0[b], 0u, p.h2[b], 0u, vf[2 * h], vf[2 * h + 1]);
            mma_bf16(o[nd + h], p.l0[b], 0u, p.l2[b], 0u, vf[2 * h], vf[2 * h + 1]);
          }
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

// One warp's share of an attention chunk (positions j0 .. j0 + jn - 1, jn <=
// 16) in the persistent step kernel: after S a barrier of the eight consumer
// warps (every warp is done reading K) frees the K rows, which then hold the
// warps' partials: per head (max, sum, o[hd]) at w0.
template <int REP, int HDC>
__device__ __forceinline__ void attn_warp_tc(const unsigned char* Ks, const unsigned char* Vs, int j0, int jn,
                                             const float* qs, int lane, float* w0, float qscale = 1.f) {
  PFrag<1> p;
  attn_scores<REP, HDC, 1>(Ks, j0, jn, qs, lane, qscale, p);
  dev::named_sync(1, 8 * 32);  // K is no longer read: the partials may overlay it
  attn_values<REP, HDC, 1>(Vs, j0, jn, p, lane, w0 + (lane >> 2) * (2 + HDC));
}

}  // namespace attn
}  // namespace river
