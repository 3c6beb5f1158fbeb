// Row kernels of the decode/prefill path.
//
// k_rownorm is the layer-end kernel: for every token it computes the
// state-transition similarity of the layer (cosine of the residual entering
// vs leaving it, River-LLM explainer section 四), the next RMSNorm (bf16
// activations plus their per-group sums for the W4 path), and -- in the last
// CTA to finish, chosen by an atomic ticket, so no CTA ever waits -- the
// minimum over all tokens processed together and the tau compare that sets
// the step's exit layer on the device.  Once the exit layer is below L no
// later layer is checked (section 四: similarity rises with depth).
#include <float.h>

#include "internal.h"

namespace river {

namespace {

constexpr int kThreads = 256;

__device__ __forceinline__ float warp_sum(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
  return v;
}

__device__ __forceinline__ float warp_min(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v = fminf(v, __shfl_xor_sync(0xffffffffu, v, o));
  return v;
}

// Block-wide sum of three values (fixed order: per warp, then warp 0).
__device__ __forceinline__ void block_sum3(float& a, float& b, float& c) {
  __shared__ float sh[3][kThreads / 32];
  const int w = threadIdx.x >> 5, l = threadIdx.x & 31;
  a = warp_sum(a);
  b = warp_sum(b);
  c = warp_sum(c);
  if (l == 0) {
    sh[0][w] = a;
    sh[1][w] = b;
    sh[2][w] = c;
  }
  __syncthreads();
  if (w == 0) {
    a = l < kThreads / 32 ? sh[0][l] : 0.f;
    b = l < kThreads / 32 ? sh[1][l] : 0.f;
    c = l < kThreads / 32 ? sh[2][l] : 0.f;
    a = warp_sum(a);
    b = warp_sum(b);
    c = warp_sum(c);
    if (l == 0) {
      sh[0][0] = a;
      sh[1][0] = b;
      sh[2][0] = c;
    }
  }
  __syncthreads();
  a = sh[0][0];
  b = sh[1][0];
  c = sh[2][0];
  __syncthreads();
}

__global__ void __launch_bounds__(kThreads) k_rownorm(RowNormArgs a) {
  pdl_wait();
  extern __shared__ float hrow[];  // d fp32 values of this row
  __shared__ int s_last;
  const int r = blockIdx.x;
  const int tid = threadIdx.x;
  const int d = a.d;
  float* hout = a.h_out + (size_t)r * d;

  if (a.tokens != nullptr) {
    int tok = a.tokens[r];
    if (tok < 0 || tok >= a.vocab) {
      if (tid == 0) atomicOr(&a.st->err, RL_DEVERR_TOKEN);
      tok = 0;
    }
    const bf16* e = a.embed + (size_t)tok * d;
    for (int k = tid; k < d; k += kThreads) {
      const float v = __bfloat162float(e[k]);
      hrow[k] = v;
      hout[k] = v;
    }
    if (r == 0 && tid == 0) {
      // Step begin: the exit layer of this call.
      int e_l = a.L;
      if (a.mode == RL_EXIT_FORCED) {
        const int idx = a.use_step_index ? (a.st->step % a.schedule_len) : 0;
        e_l = a.schedule[idx];
        if (e_l < 0 || e_l > a.L) {
          atomicOr(&a.st->err, RL_DEVERR_SCHEDULE);
          e_l = e_l < 0 ? 0 : a.L;
        }
      }
      a.st->exit_layer = e_l;
    }
  }
  float ss_out = 0.f, dot = 0.f, ss_in = 0.f;
  const float* hin = a.h_in ? a.h_in + (size_t)r * d : nullptr;
  if (a.tokens != nullptr) {
    __syncthreads();
    for (int k = tid; k < d; k += kThreads) {
      const float v = hrow[k];
      ss_out += v * v;
      if (hin) {
        const float u = hin[k];
        dot += u * v;
        ss_in += u * u;
      }
    }
  } else {
    // one pass over the row (and the layer's input row), four values a load
    const float4* h4 = reinterpret_cast<const float4*>(hout);
    const float4* i4 = reinterpret_cast<const float4*>(hin);
    float4* s4 = reinterpret_cast<float4*>(hrow);
    for (int k = tid; k < d / 4; k += kThreads) {
      const float4 v = h4[k];
      s4[k] = v;
      ss_out += v.x * v.x + v.y * v.y + v.z * v.z + v.w * v.w;
      if (hin) {
        const float4 u = i4[k];
        dot += u.x * v.x + u.y * v.y + u.z * v.z + u.w * v.w;
        ss_in += u.x * u.x + u.y * u.y + u.z * u.z + u.w * u.w;
      }
    }
  }
  block_sum3(ss_out, dot, ss_in);  // its barriers also publish hrow

  if (a.g != nullptr) {
    const float den = sqrtf(ss_out / (float)d + a.eps);
    bf16* x = a.x + (size_t)r * a.ldx;
    for (int k8 = tid; k8 < d / 8; k8 += kThreads) {
      const float4 h0 = reinterpret_cast<const float4*>(hrow)[2 * k8];
      const float4 h1 = reinterpret_cast<const float4*>(hrow)[2 * k8 + 1];
      const float4 g0 = reinterpret_cast<const float4*>(a.g)[2 * k8];
      const float4 g1 = reinterpret_cast<const float4*>(a.g)[2 * k8 + 1];
      const __nv_bfloat162 b0 = __floats2bfloat162_rn(h0.x / den * g0.x, h0.y / den * g0.y);
      const __nv_bfloat162 b1 = __floats2bfloat162_rn(h0.z / den * g0.z, h0.w / den * g0.w);
      const __nv_bfloat162 b2 = __floats2bfloat162_rn(h1.x / den * g1.x, h1.y / den * g1.y);
      const __nv_bfloat162 b3 = __floats2bfloat162_rn(h1.z / den * g1.z, h1.w / den * g1.w);
      uint4 pk;
      pk.x = *reinterpret_cast<const uint32_t*>(&b0);
      pk.y = *reinterpret_cast<const uint32_t*>(&b1);
      pk.z = *reinterpret_cast<const uint32_t*>(&b2);
      pk.w = *reinterpret_cast<const uint32_t*>(&b3);
      *reinterpret_cast<uint4*>(x + (size_t)k8 * 8) = pk;
      // keep the rounded values for the group sums
      const float2 f0 = __bfloat1622float2(b0), f1 = __bfloat1622float2(b1);
      const float2 f2 = __bfloat1622float2(b2), f3 = __bfloat1622float2(b3);
      reinterpret_cast<float4*>(hrow)[2 * k8] = make_float4(f0.x, f0.y, f1.x, f1.y);
      reinterpret_cast<float4*>(hrow)[2 * k8 + 1] = make_float4(f2.x, f2.y, f3.x, f3.y);
    }
    __syncthreads();
    const int w = tid >> 5, l = tid & 31;
    const int G = (d + kGroup - 1) / kGroup;
    for (int gi = w; gi < G; gi += kThreads / 32) {
      float s = 0.f;
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        const int k = gi * kGroup + 4 * l + i;
        if (k < d) s += hrow[k];
      }
      s = warp_sum(s);
      if (l == 0) a.xsum[(size_t)r * a.ldxs + gi] = s;
    }
    __syncthreads();
    // restore the residual values for the trace below
    if (a.trace) {
      for (int k = tid; k < d; k += kThreads) hrow[k] = hout[k];
      __syncthreads();
    }
  }

  if (a.trace != nullptr) {
    const bool last_pos = a.trace_T <= 0 || (r % a.trace_T) == a.trace_T - 1;
    if (last_pos) {
      const int seq = a.trace_T > 0 ? r / a.trace_T : r;
      float* tr = a.trace + ((size_t)a.trace_layer * a.trace_maxB + seq) * d;
      for (int k = tid; k < d; k += kThreads) tr[k] = hout[k];
    }
  }

  if (hin == nullptr) return;

  if (tid == 0) {
    const float den = fmaxf(sqrtf(ss_in) * sqrtf(ss_out), 1e-12f);
    a.cosbuf[r] = dot / den;
  }
  // Last-arriver reduction: no CTA waits for another.
  __threadfence();
  __syncthreads();
  if (tid == 0) {
    const unsigned int t = atomicAdd(&a.st->ticket, 1u);
    s_last = (t == (unsigned int)(a.rows - 1));
  }
  __syncthreads();
  if (!s_last) return;
  __threadfence();
  float m = FLT_MAX;
  for (int i = tid; i < a.rows; i += kThreads) m = fminf(m, __ldcg(a.cosbuf + i));
  m = warp_min(m);
  __shared__ float sm[kThreads / 32];
  if ((tid & 31) == 0) sm[tid >> 5] = m;
  __syncthreads();
  if (tid == 0) {
    for (int w = 1; w < kThreads / 32; ++w) m = fminf(m, sm[w]);
    m = fminf(m, sm[0]);
    if (a.min_cos_out) a.min_cos_out[a.layer_no - 1] = m;
    DevState* st = a.st;
    if (a.mode == RL_EXIT_TAU && st->exit_layer == a.L && a.layer_no < a.L && m > a.tau)
      st->exit_layer = a.layer_no;
    if (a.layer_no == a.L) {
      if (a.exit_out) a.exit_out[0] = st->exit_layer;
      st->pos = a.set_pos >= 0 ? a.set_pos : st->pos + 1;
      st->step = a.set_step >= 0 ? a.set_step : st->step + 1;
    }
    st->ticket = 0u;
    __threadfence();
  }
}

__global__ void k_group_sums(const bf16* __restrict__ x, int ldx, int Kp, int B,
                             float* __restrict__ xsum, int ldxs) {
  pdl_wait();
  const int G = Kp / kGroup;
  const int wid = (blockIdx.x * blockDim.x + threadIdx.x) >> 5;
  const int l = threadIdx.x & 31;
  if (wid >= B * G) return;
  const int b = wid / G, gi = wid % G;
  const bf16* p = x + (size_t)b * ldx + gi * kGroup + 4 * l;
  float s = 0.f;
#pragma unroll
  for (int i = 0; i < 4; ++i) s += __bfloat162float(p[i]);
  s = warp_sum(s);
  if (l == 0) xsum[(size_t)b * ldxs + gi] = s;
}

__global__ void __launch_bounds__(1024) k_argmax(const float* __restrict__ logits, int ld, int V,
                                                 int* __restrict__ out) {
  pdl_wait();
  const int b = blockIdx.x;
  const float* p = logits + (size_t)b * ld;
  float best = -FLT_MAX;
  int bi = 0x7fffffff;
  // four values a load, four loads in flight; each thread scans its indices
  // in increasing order, so a tie keeps the smaller index (V % 4 == 0)
  const float4* p4 = reinterpret_cast<const float4*>(p);
  const int n4 = V >> 2, step = blockDim.x;
  auto take = [&](float v, int i) {
    if (v > best || (v == best && i < bi)) {
      best = v;
      bi = i;
    }
  };
  int c = threadIdx.x;
  for (; c + 3 * step < n4; c += 4 * step) {
    float4 q[4];
#pragma unroll
    for (int j = 0; j < 4; ++j) q[j] = p4[c + j * step];
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      const int i = 4 * (c + j * step);
      take(q[j].x, i);
      take(q[j].y, i + 1);
      take(q[j].z, i + 2);
      take(q[j].w, i + 3);
    }
  }
  for (; c < n4; c += step) {
    const float4 q = p4[c];
    take(q.x, 4 * c);
    take(q.y, 4 * c + 1);
    take(q.z, 4 * c + 2);
    take(q.w, 4 * c + 3);
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
    const float ov = __shfl_xor_sync(0xffffffffu, best, o);
    const int oi = __shfl_xor_sync(0xffffffffu, bi, o);
    if (ov > best || (ov == best && oi < bi)) {
      best = ov;
      bi = oi;
    }
  }
  __shared__ float sv[32];
  __shared__ int si[32];
  const int w = threadIdx.x >> 5, l = threadIdx.x & 31;
  if (l == 0) {
    sv[w] = best;
    si[w] = bi;
  }
  __syncthreads();
  if (threadIdx.x == 0) {
    const int nw = blockDim.x / 32;
    for (int i = 1; i < nw; ++i)
      if (sv[i] > best || (sv[i] == best && si[i] < bi)) {
        best = sv[i];
        bi = si[i];
      }
    out[b] = bi == 0x7fffffff ? 0 : bi;
  }
}

__global__ void k_gather_rows(bf16* __restrict__ dst, int ldd, int K, const int2* __restrict__ map,
                              GatherSrcs srcs, int src_ld) {
  const int r = blockIdx.x;
  const int2 m = map[r];
  const bf16* s = srcs.p[m.x] + (size_t)m.y * src_ld;
  bf16* o = dst + (size_t)r * ldd;
  const bf16 zero = __float2bfloat16_rn(0.f);
  for (int k = threadIdx.x; k < ldd; k += blockDim.x) o[k] = k < K ? s[k] : zero;
}

__global__ void k_set_state(DevState* st, int pos, int step) {
  st->pos = pos;
  st->step = step;
}

__global__ void k_bf16_to_f32(const bf16* __restrict__ s, float* __restrict__ d, int n) {
  const int i = blockIdx.x * blockDim.x + threadIdx.x;
  if (i < n) d[i] = __bfloat162float(s[i]);
}

}  // namespace

void launch_rownorm(const RowNormArgs& a, cudaStream_t s) {
  launch_pdl(k_rownorm, dim3(a.rows), dim3(kThreads), a.d * sizeof(float), s, a);
}

void launch_group_sums(const bf16* x, int ldx, int Kp, int B, float* xsum, int ldxs,
                       cudaStream_t s) {
  const int warps = B * (Kp / kGroup);
  const int blocks = (warps * 32 + 255) / 256;
  launch_pdl(k_group_sums, dim3(blocks), dim3(256), 0, s, x, ldx, Kp, B, xsum, ldxs);
}

void launch_argmax(const float* logits, int ld, int V, int B, int* out, cudaStream_t s) {
  launch_pdl(k_argmax, dim3(B), dim3(1024), 0, s, logits, ld, V, out);
}

void launch_gather_rows(bf16* dst, int ldd, int N, int K, const int2* rowmap, GatherSrcs srcs,
                        int src_ld, cudaStream_t s) {
  k_gather_rows<<<N, 256, 0, s>>>(dst, ldd, K, rowmap, srcs, src_ld);
}

void launch_set_state(DevState* st, int pos, int step, cudaStream_t s) {
  k_set_state<<<1, 1, 0, s>>>(st, pos, step);
}

void launch_bf16_to_f32(const bf16* src, float* dst, int n, cudaStream_t s) {
  k_bf16_to_f32<<<(n + 255) / 256, 256, 0, s>>>(src, dst, n);
}

}  // namespace river
