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
__device__ __forceinline__ void attn_partial_body(const AttnArgs& a) {
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
  {
    float qv[kMaxRep * HD / kThreads];  // all loads first, then the stores
#pragma unroll
    for (int q = 0; q < kMaxRep * HD / kThreads; ++q) {
      const int i = tid + q * kThreads;
      qv[q] = i < rep * HD ? a.q[(size_t)row * a.Hq * HD + hk * rep * HD + i] : 0.f;
    }
#pragma unroll
    for (int q = 0; q < kMaxRep * HD / kThreads; ++q) {
      const int i = tid + q * kThreads;
      if (i < rep * HD) qs[i / HD][i % HD] = qv[q] * scale;
    }
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
      uint4 kw[HD / 8];  // the whole K row in flight at once
#pragma unroll
      for (int v = 0; v < HD / 8; ++v) kw[v] = kr[v];
#pragma unroll
      for (int v = 0; v < HD / 8; ++v) {
        const uint4 w = kw[v];
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
    for (int h = 0; h < kMaxRep; ++h) alpha[h] = 1.f;
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
    // P V: eight positions per batch, all their V loads in flight together
    const int nvalid = min(kThreads, end - sb);
    constexpr int NS = (kSlotsMax > 0 ? kSlotsMax : 1);
    int sh[NS];
#pragma unroll
    for (int si = 0; si < NS; ++si) {
      const int s = tid + si * kThreads;
      sh[si] = s < nslots ? s / (HD / 2) : -1;
      if (sh[si] >= 0) {
        float al = 1.f;
#pragma unroll
        for (int hh = 0; hh < kMaxRep; ++hh)
          if (hh == sh[si]) al = alpha[hh];
        acc[si].x *= al;
        acc[si].y *= al;
      }
    }
    const __nv_bfloat162* vrow = reinterpret_cast<const __nv_bfloat162*>(vbase + (size_t)sb * HD);
    for (int i0 = 0; i0 < nvalid; i0 += 8) {
      __nv_bfloat162 vv[NS][8];
#pragma unroll
      for (int si = 0; si < NS; ++si)
#pragma unroll
        for (int q = 0; q < 8; ++q)
          if (sh[si] >= 0 && i0 + q < nvalid)
            vv[si][q] = vrow[(size_t)(i0 + q) * (HD / 2) + (tid + si * kThreads) % (HD / 2)];
#pragma unroll
      for (int si = 0; si < NS; ++si) {
        if (sh[si] < 0) continue;
#pragma unroll
        for (int q = 0; q < 8; ++q) {
          if (i0 + q < nvalid) {
            const float p = ps[sh[si]][i0 + q];
            const float2 v = __bfloat1622float2(vv[si][q]);
            acc[si].x += p * v.x;
            acc[si].y += p * v.y;
          }
        }
      }
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
__global__ void __launch_bounds__(kThreads) k_attn_partial(AttnArgs a) {
  attn_partial_body<HD>(a);
}

__device__ __forceinline__ void grid_dep_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
__device__ __forceinline__ void grid_dep_launch() { asm volatile("griddepcontrol.launch_dependents;" :::); }

// Decode attention in one kernel.  CTA (chunk c, KV head, sequence) owns
// context positions [start, end).  Rows before the current position are
// final before the projection kernel that precedes this one finishes (only
// row `pos` is being written), so they are copied into shared memory with
// cp.async BEFORE the programmatic-dependent-launch wait; after the wait only
// q and row `pos` are fetched.  Each K/V row is read once for all Hq/Hkv query
// heads of the group.  The last CTA of each (sequence, KV head) to finish
// merges the chunks (split-context "flash decoding"); no CTA waits on another.
constexpr int kCH = 128;  // max positions per CTA

template <int HD>
__global__ void __launch_bounds__(kThreads) k_attn_decode(AttnArgs a) {
  constexpr int RSK = HD * 2 + 16;  // padded smem row: conflict-free row-per-thread reads
  extern __shared__ __align__(16) unsigned char kvs[];  // K rows, then V rows
  unsigned char* Ks = kvs;
  unsigned char* Vs = kvs + kCH * RSK;
  __shared__ float qs[kMaxRep][HD];
  __shared__ float ps[kMaxRep][kCH];
  __shared__ float red[kMaxRep][kThreads / 32];
  __shared__ float mstat[kMaxRep][2];
  __shared__ int s_last;

  const int c = blockIdx.x, hk = blockIdx.y, b = blockIdx.z;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int rep = a.Hq / a.Hkv;
  const int nch = a.nchunks;
  const int pos = *a.pos_ptr;  // set by the previous step: stable before the wait
  int ctx = pos + 1;
  if (ctx > a.Tmax) ctx = a.Tmax;
  const int clen = (ctx + nch - 1) / nch;  // <= kCH by the chunk-count rule
  const int start = c * clen;
  const int end = min(start + clen, ctx);
  const int n = end > start ? end - start : 0;
  const size_t head_base = ((size_t)b * a.Hkv + hk) * a.Tmax;
  const bf16* kb = a.kc + head_base * HD;
  const bf16* vb = a.vc + head_base * HD;

  // ---- before the wait: rows start .. min(end, pos) - 1 -----------------------
  const int npre = max(0, min(end, pos) - start);
  for (int idx = tid; idx < npre * (HD / 8); idx += kThreads) {
    const int r = idx / (HD / 8), ch = idx % (HD / 8);
    const uint32_t dk = (uint32_t)__cvta_generic_to_shared(Ks + r * RSK + ch * 16);
    const uint32_t dv = (uint32_t)__cvta_generic_to_shared(Vs + r * RSK + ch * 16);
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(dk),
                 "l"(kb + (size_t)(start + r) * HD + ch * 8) : "memory");
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(dv),
                 "l"(vb + (size_t)(start + r) * HD + ch * 8) : "memory");
  }
  asm volatile("cp.async.commit_group;" ::: "memory");
  grid_dep_wait();
  grid_dep_launch();

  // ---- after the wait: q and the row being written this step ------------------
  const float scale = rsqrtf((float)HD);
  {
    float qv[kMaxRep * HD / kThreads];
#pragma unroll
    for (int q = 0; q < kMaxRep * HD / kThreads; ++q) {
      const int i = tid + q * kThreads;
      qv[q] = i < rep * HD ? a.q[(size_t)b * a.Hq * HD + hk * rep * HD + i] : 0.f;
    }
    if (pos >= start && pos < end && tid < HD / 8) {
      const int r = pos - start;
      *reinterpret_cast<uint4*>(Ks + r * RSK + tid * 16) =
          *reinterpret_cast<const uint4*>(kb + (size_t)pos * HD + tid * 8);
      *reinterpret_cast<uint4*>(Vs + r * RSK + tid * 16) =
          *reinterpret_cast<const uint4*>(vb + (size_t)pos * HD + tid * 8);
    }
#pragma unroll
    for (int q = 0; q < kMaxRep * HD / kThreads; ++q) {
      const int i = tid + q * kThreads;
      if (i < rep * HD) qs[i / HD][i % HD] = qv[q] * scale;
    }
  }
  asm volatile("cp.async.wait_all;" ::: "memory");
  __syncthreads();

  // ---- scores: one position per thread ------------------------------------------
  float sc[kMaxRep];
#pragma unroll
  for (int h = 0; h < kMaxRep; ++h) sc[h] = -FLT_MAX;
  if (tid < n) {
#pragma unroll
    for (int h = 0; h < kMaxRep; ++h) sc[h] = 0.f;
#pragma unroll 4
    for (int v = 0; v < HD / 8; ++v) {
      const uint4 w = *reinterpret_cast<const uint4*>(Ks + tid * RSK + v * 16);
      const __nv_bfloat162* e = reinterpret_cast<const __nv_bfloat162*>(&w);
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        const float2 f = __bfloat1622float2(e[i]);
#pragma unroll
        for (int h = 0; h < kMaxRep; ++h)
          if (h < rep) sc[h] += f.x * qs[h][8 * v + 2 * i] + f.y * qs[h][8 * v + 2 * i + 1];
      }
    }
  }
  // block max and sum per head
#pragma unroll
  for (int h = 0; h < kMaxRep; ++h) {
    if (h >= rep) break;
    float v = sc[h];
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, o));
    if (lane == 0) red[h][warp] = v;
  }
  __syncthreads();
  if (tid < rep) {
    float m = red[tid][0];
#pragma unroll
    for (int w = 1; w < kThreads / 32; ++w) m = fmaxf(m, red[tid][w]);
    mstat[tid][0] = m;
  }
  __syncthreads();
#pragma unroll
  for (int h = 0; h < kMaxRep; ++h) {
    if (h >= rep) break;
    const float p = tid < n ? __expf(sc[h] - mstat[h][0]) : 0.f;
    if (tid < kCH) ps[h][tid] = p;
    float v = p;
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
    if (lane == 0) red[h][warp] = v;
  }
  __syncthreads();
  if (tid < rep) {
    float l = 0.f;
#pragma unroll
    for (int w = 0; w < kThreads / 32; ++w) l += red[tid][w];
    mstat[tid][1] = l;
  }
  // ---- P V: thread owns (head, dim pair) slots ----------------------------------
  constexpr int NS = kMaxRep * HD / 2 / kThreads;
  float2 acc[NS];
#pragma unroll
  for (int si = 0; si < NS; ++si) acc[si] = make_float2(0.f, 0.f);
  const int nslots = rep * HD / 2;
  for (int j = 0; j < n; ++j) {
#pragma unroll
    for (int si = 0; si < NS; ++si) {
      const int s2 = tid + si * kThreads;
      if (s2 < nslots) {
        const int h = s2 / (HD / 2), dp = s2 % (HD / 2);
        const float p = ps[h][j];
        const float2 v = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(Vs + j * RSK + dp * 4));
        acc[si].x += p * v.x;
        acc[si].y += p * v.y;
      }
    }
  }
  __syncthreads();
  // ---- partials: o (unnormalised), running max, sum ------------------------------
  float* part = a.part + ((size_t)b * a.Hq + hk * rep) * nch * (HD + 2);
#pragma unroll
  for (int si = 0; si < NS; ++si) {
    const int s2 = tid + si * kThreads;
    if (s2 < nslots) {
      const int h = s2 / (HD / 2), dp = s2 % (HD / 2);
      float* p = part + ((size_t)h * nch + c) * (HD + 2);
      p[2 * dp] = acc[si].x;
      p[2 * dp + 1] = acc[si].y;
    }
  }
  if (tid < rep) {
    float* p = part + ((size_t)tid * nch + c) * (HD + 2);
    p[HD] = n > 0 ? mstat[tid][0] : -FLT_MAX;
    p[HD + 1] = n > 0 ? mstat[tid][1] : 0.f;
  }
  __threadfence();
  __syncthreads();
  if (tid == 0)
    s_last = atomicAdd(&a.ticket[(size_t)b * a.Hkv + hk], 1u) == (unsigned int)(nch - 1);
  __syncthreads();
  if (!s_last) return;
  __threadfence();
  // ---- merge (last CTA of this sequence and KV head) ----------------------------
  float2* ml = reinterpret_cast<float2*>(kvs);           // [rep][nch]
  float* wc = reinterpret_cast<float*>(kvs) + 2 * kMaxRep * 256;  // [rep][nch]
  for (int i = tid; i < rep * nch; i += kThreads) {
    const int h = i / nch, cc = i % nch;
    const float* p = a.part + (((size_t)b * a.Hq + hk * rep + h) * nch + cc) * (HD + 2);
    ml[i] = make_float2(__ldcg(p + HD), __ldcg(p + HD + 1));
  }
  __syncthreads();
  if (tid < rep) {
    float M = -FLT_MAX, den = 0.f;
    for (int cc = 0; cc < nch; ++cc)
      if (ml[tid * nch + cc].y > 0.f) M = fmaxf(M, ml[tid * nch + cc].x);
    for (int cc = 0; cc < nch; ++cc) {
      const float2 v = ml[tid * nch + cc];
      const float w = v.y > 0.f ? __expf(v.x - M) : 0.f;
      wc[tid * nch + cc] = w;
      den += w * v.y;
    }
    const float inv = den > 0.f ? 1.f / den : 0.f;
    for (int cc = 0; cc < nch; ++cc) wc[tid * nch + cc] *= inv;
  }
  __syncthreads();
  // every thread owns OPT outputs and issues the loads of all of them for a
  // batch of chunks at once
  constexpr int OPT = kMaxRep * HD / kThreads;
  constexpr int CB = OPT <= 4 ? 16 : 8;
  float num[OPT];
#pragma unroll
  for (int o = 0; o < OPT; ++o) num[o] = 0.f;
  for (int c0 = 0; c0 < nch; c0 += CB) {
    float v[OPT][CB];
#pragma unroll
    for (int o = 0; o < OPT; ++o) {
      const int i = tid + o * kThreads;
      const int h = i / HD, dd = i % HD;
      const float* p = a.part + ((size_t)b * a.Hq + hk * rep + h) * nch * (HD + 2) + dd;
#pragma unroll
      for (int q = 0; q < CB; ++q)
        v[o][q] = (i < rep * HD && c0 + q < nch) ? __ldcg(p + (size_t)(c0 + q) * (HD + 2)) : 0.f;
    }
#pragma unroll
    for (int o = 0; o < OPT; ++o) {
      const int i = tid + o * kThreads;
      const int h = i < rep * HD ? i / HD : 0;
#pragma unroll
      for (int q = 0; q < CB; ++q)
        if (c0 + q < nch) num[o] += wc[h * nch + c0 + q] * v[o][q];
    }
  }
#pragma unroll
  for (int o = 0; o < OPT; ++o) {
    const int i = tid + o * kThreads;
    if (i < rep * HD) {
      const int h = i / HD, dd = i % HD;
      a.o[(size_t)b * a.ldo + (hk * rep + h) * HD + dd] = __float2bfloat16_rn(num[o]);
    }
  }
  if (tid == 0) a.ticket[(size_t)b * a.Hkv + hk] = 0u;
}

// Merge of one (row, query head)'s chunk partials: M = the largest chunk
// maximum (a block reduction over the chunks, read in parallel), then the
// weights w_c = exp(m_c - M) of up to kCombBlk chunks at a time are staged in
// shared memory and thread dd sums w_c o_c[dd] and w_c l_c in chunk order
// (independent loads, so the chunk loop runs at L2 throughput, not latency).
constexpr int kCombBlk = 512;

template <int HD>
__global__ void __launch_bounds__(HD) k_attn_combine(AttnArgs a) {
  pdl_wait();
  __shared__ float s_w[kCombBlk], s_l[kCombBlk];
  __shared__ float s_red[HD / 32];
  const int hq = blockIdx.x, row = blockIdx.y, dd = threadIdx.x;
  const int nch = a.nchunks;
  const float* part = a.part + ((size_t)row * a.Hq + hq) * nch * (HD + 2);
  float M = -FLT_MAX;
  for (int c = dd; c < nch; c += HD) {
    const float* p = part + (size_t)c * (HD + 2);
    if (p[HD + 1] > 0.f) M = fmaxf(M, p[HD]);
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) M = fmaxf(M, __shfl_xor_sync(0xffffffffu, M, o));
  if ((dd & 31) == 0) s_red[dd >> 5] = M;
  __syncthreads();
#pragma unroll
  for (int w = 0; w < HD / 32; ++w) M = fmaxf(M, s_red[w]);
  float num = 0.f, den = 0.f;
  for (int c0 = 0; c0 < nch; c0 += kCombBlk) {
    const int nb = min(kCombBlk, nch - c0);
    __syncthreads();  // the previous block's weights have been used
    for (int c = dd; c < nb; c += HD) {
      const float* p = part + (size_t)(c0 + c) * (HD + 2);
      const float l = p[HD + 1];
      s_l[c] = l;
      s_w[c] = l > 0.f ? __expf(p[HD] - M) : 0.f;
    }
    __syncthreads();
    const float* pd = part + (size_t)c0 * (HD + 2) + dd;
#pragma unroll 8
    for (int c = 0; c < nb; ++c) {
      num += s_w[c] * pd[(size_t)c * (HD + 2)];
      den += s_w[c] * s_l[c];
    }
  }
  const float v = den > 0.f ? num / den : 0.f;
  a.o[(size_t)row * a.ldo + hq * HD + dd] = __float2bfloat16_rn(v);
}

}  // namespace

void attention_setup() {
  cudaFuncSetAttribute(k_attn_decode<128>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                       2 * kCH * (128 * 2 + 16));
  cudaFuncSetAttribute(k_attn_decode<64>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                       2 * kCH * (64 * 2 + 16));
  cudaFuncSetAttribute(k_attn_decode<128>, cudaFuncAttributePreferredSharedMemoryCarveout,
                       cudaSharedmemCarveoutMaxShared);
  cudaFuncSetAttribute(k_attn_decode<64>, cudaFuncAttributePreferredSharedMemoryCarveout,
                       cudaSharedmemCarveoutMaxShared);
}

int decode_attention_chunks(int B, int Hkv, int Tmax, int sm_count) {
  // at most kCH positions per CTA; otherwise about two CTAs per SM, >= 32 positions each
  const int need = (Tmax + kCH - 1) / kCH;
  int n = (2 * sm_count + B * Hkv - 1) / (B * Hkv);
  const int cap32 = (Tmax + 31) / 32;
  if (n > cap32) n = cap32;
  if (n < need) n = need;
  if (n < 1) n = 1;
  return n;
}

cudaError_t launch_attention_fused(const AttnArgs& a, bool pdl, cudaStream_t s) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(a.nchunks, a.Hkv, a.nq);
  cfg.blockDim = dim3(kThreads);
  cfg.dynamicSmemBytes = 0;
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = pdl ? 1 : 0;
  if (a.hd == 64) {
    cfg.dynamicSmemBytes = 2 * kCH * (64 * 2 + 16);
    return cudaLaunchKernelEx(&cfg, k_attn_decode<64>, a);
  }
  cfg.dynamicSmemBytes = 2 * kCH * (128 * 2 + 16);
  return cudaLaunchKernelEx(&cfg, k_attn_decode<128>, a);
}

void launch_attention_combine(const AttnArgs& a, cudaStream_t s) {
  dim3 g2(a.Hq, a.nq);
  if (a.hd == 64)
    launch_pdl(k_attn_combine<64>, g2, dim3(64), 0, s, a);
  else
    launch_pdl(k_attn_combine<128>, g2, dim3(128), 0, s, a);
}

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
