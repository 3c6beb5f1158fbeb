// Grouped-query attention over the shared per-layer KV cache.
//
// The cache is the backbone's own (River-LLM explainer, section 三: the exit
// layer writes and reads the same slots), one contiguous bf16
// [maxB][Hkv][Tmax][hd] array per layer.  A query at position p attends to
// positions 0..p.  Each CTA takes one (query row, KV head, context chunk),
// reads every K and V row of its chunk once for all Hq/Hkv query heads that
// share the KV head, and keeps an online softmax (running max and sum);
// a combine kernel merges the chunks (split-context "flash decoding").
#include <float.h>

#include "internal.h"

namespace river {

namespace {

constexpr int kThreads = 128;
constexpr int kMaxRep = 8;

template <int HD>
__global__ void __launch_bounds__(kThreads) k_attn_partial(AttnArgs a) {
  const int c = blockIdx.x, hk = blockIdx.y, row = blockIdx.z;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int rep = a.Hq / a.Hkv;
  int seq, pos;
  if (a.T_prefill > 0) {
    seq = row / a.T_prefill;
    pos = row % a.T_prefill;
  } else {
    seq = row;
    pos = *a.pos_ptr;
  }
  int ctx = pos + 1;
  if (ctx > a.Tmax) ctx = a.Tmax;
  int clen = (ctx + a.nchunks - 1) / a.nchunks;
  if (clen < 64) clen = 64;
  const int start = c * clen;
  const int end = min(start + clen, ctx);

  __shared__ float qs[kMaxRep][HD];
  __shared__ float ps[kMaxRep][kThreads];
  __shared__ float red[kMaxRep][kThreads / 32];

  const float scale = rsqrtf((float)HD);
  for (int i = tid; i < rep * HD; i += kThreads) {
    const int h = i / HD, dd = i % HD;
    qs[h][dd] = a.q[(size_t)row * a.Hq * HD + (hk * rep + h) * HD + dd] * scale;
  }
  __syncthreads();

  constexpr int kSlotsMax = kMaxRep * HD / 2 / kThreads;  // (h, dim-pair) slots per thread
  float2 acc[kSlotsMax > 0 ? kSlotsMax : 1];
#pragma unroll
  for (int i = 0; i < (kSlotsMax > 0 ? kSlotsMax : 1); ++i) acc[i] = make_float2(0.f, 0.f);
  float m_run[kMaxRep], l_run[kMaxRep];
#pragma unroll
  for (int h = 0; h < kMaxRep; ++h) {
    m_run[h] = -FLT_MAX;
    l_run[h] = 0.f;
  }
  const size_t head_base = ((size_t)seq * a.Hkv + hk) * a.Tmax;
  const bf16* kbase = a.kc + head_base * HD;
  const bf16* vbase = a.vc + head_base * HD;
  const int nslots = rep * HD / 2;

  for (int sb = start; sb < end; sb += kThreads) {
    const int j = sb + tid;
    const bool valid = j < end;
    float sc[kMaxRep];
#pragma unroll
    for (int h = 0; h < kMaxRep; ++h) sc[h] = 0.f;
    if (valid) {
      const uint4* kr = reinterpret_cast<const uint4*>(kbase + (size_t)j * HD);
#pragma unroll 4
      for (int v = 0; v < HD / 8; ++v) {
        const uint4 w = kr[v];
        const __nv_bfloat162* e = reinterpret_cast<const __nv_bfloat162*>(&w);
#pragma unroll
        for (int i = 0; i < 4; ++i) {
          const float2 f = __bfloat1622float2(e[i]);
#pragma unroll
          for (int h = 0; h < kMaxRep; ++h) {
            if (h < rep) sc[h] += f.x * qs[h][8 * v + 2 * i] + f.y * qs[h][8 * v + 2 * i + 1];
          }
        }
      }
    }
    // block max per head
#pragma unroll
    for (int h = 0; h < kMaxRep; ++h) {
      if (h >= rep) break;
      float v = valid ? sc[h] : -FLT_MAX;
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, o));
      if (lane == 0) red[h][warp] = v;
    }
    __syncthreads();
    float alpha[kMaxRep];
#pragma unroll
    for (int h = 0; h < kMaxRep; ++h) {
      if (h >= rep) break;
      float bm = red[h][0];
#pragma unroll
      for (int w = 1; w < kThreads / 32; ++w) bm = fmaxf(bm, red[h][w]);
      const float mnew = fmaxf(m_run[h], bm);
      alpha[h] = __expf(m_run[h] - mnew);
      m_run[h] = mnew;
      ps[h][tid] = valid ? __expf(sc[h] - mnew) : 0.f;
    }
    __syncthreads();
    // block sum per head
#pragma unroll
    for (int h = 0; h < kMaxRep; ++h) {
      if (h >= rep) break;
      float v = ps[h][tid];
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
      if (lane == 0) red[h][warp] = v;
    }
    __syncthreads();
#pragma unroll
    for (int h = 0; h < kMaxRep; ++h) {
      if (h >= rep) break;
      float bs = 0.f;
#pragma unroll
      for (int w = 0; w < kThreads / 32; ++w) bs += red[h][w];
      l_run[h] = l_run[h] * alpha[h] + bs;
    }
    // P V
    const int nvalid = min(kThreads, end - sb);
#pragma unroll
    for (int si = 0; si < (kSlotsMax > 0 ? kSlotsMax : 1); ++si) {
      const int s = tid + si * kThreads;
      if (s >= nslots) break;
      const int h = s / (HD / 2), dp = s % (HD / 2);
      float2 o = acc[si];
      float al = 1.f;
#pragma unroll
      for (int hh = 0; hh < kMaxRep; ++hh)
        if (hh == h) al = alpha[hh];
      o.x *= al;
      o.y *= al;
      const __nv_bfloat162* vp =
          reinterpret_cast<const __nv_bfloat162*>(vbase + (size_t)sb * HD) + dp;
      for (int i = 0; i < nvalid; ++i) {
        const float p = ps[h][i];
        const float2 v = __bfloat1622float2(vp[(size_t)i * (HD / 2)]);
        o.x += p * v.x;
        o.y += p * v.y;
      }
      acc[si] = o;
    }
    __syncthreads();
  }

  // write partials: o (unnormalised), m, l
  float* part = a.part + ((size_t)row * a.Hq + hk * rep) * a.nchunks * (HD + 2);
#pragma unroll
  for (int si = 0; si < (kSlotsMax > 0 ? kSlotsMax : 1); ++si) {
    const int s = tid + si * kThreads;
    if (s >= nslots) break;
    const int h = s / (HD / 2), dp = s % (HD / 2);
    float* p = part + ((size_t)h * a.nchunks + c) * (HD + 2);
    p[2 * dp] = acc[si].x;
    p[2 * dp + 1] = acc[si].y;
  }
  if (tid < rep) {
    float mm = -FLT_MAX, ll = 0.f;
#pragma unroll
    for (int h = 0; h < kMaxRep; ++h)
      if (h == tid) {
        mm = m_run[h];
        ll = l_run[h];
      }
    float* p = part + ((size_t)tid * a.nchunks + c) * (HD + 2);
    p[HD] = start < end ? mm : -FLT_MAX;
    p[HD + 1] = start < end ? ll : 0.f;
  }
}

template <int HD>
__global__ void __launch_bounds__(HD) k_attn_combine(AttnArgs a) {
  const int hq = blockIdx.x, row = blockIdx.y, dd = threadIdx.x;
  const float* part = a.part + ((size_t)row * a.Hq + hq) * a.nchunks * (HD + 2);
  float M = -FLT_MAX;
  for (int c = 0; c < a.nchunks; ++c) {
    const float* p = part + (size_t)c * (HD + 2);
    if (p[HD + 1] > 0.f) M = fmaxf(M, p[HD]);
  }
  float num = 0.f, den = 0.f;
  for (int c = 0; c < a.nchunks; ++c) {
    const float* p = part + (size_t)c * (HD + 2);
    const float l = p[HD + 1];
    if (l > 0.f) {
      const float w = __expf(p[HD] - M);
      num += w * p[dd];
      den += w * l;
    }
  }
  const float v = den > 0.f ? num / den : 0.f;
  a.o[(size_t)row * a.ldo + hq * HD + dd] = __float2bfloat16_rn(v);
}

}  // namespace

void launch_attention(const AttnArgs& a, cudaStream_t s) {
  dim3 g1(a.nchunks, a.Hkv, a.nq);
  dim3 g2(a.Hq, a.nq);
  if (a.hd == 64) {
    k_attn_partial<64><<<g1, kThreads, 0, s>>>(a);
    k_attn_combine<64><<<g2, 64, 0, s>>>(a);
  } else {
    k_attn_partial<128><<<g1, kThreads, 0, s>>>(a);
    k_attn_combine<128><<<g2, 128, 0, s>>>(a);
  }
}

}  // namespace river
