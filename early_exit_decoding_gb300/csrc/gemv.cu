// Dual-path decode GEMV: one kernel streams either a layer's bf16 backbone
// weights or its W4A16 exit-layer copy, picked on the device from the step's
// exit layer (River-LLM explainer, section 四: once the similarity exceeds
// tau the remaining layers run on the exit river; no host round trip).
//
// Data path (sm_103a):
//   * weights are read once, 16 B per lane (ld.global.nc, L1 no-allocate),
//     straight into mma.sync m16n8k16 A fragments: the K index that each
//     fragment slot stands for is permuted so that one lane's 32 consecutive
//     inputs of a row form its slots for a whole 128-input group (a
//     reduction may visit K in any order as long as x is visited the same
//     way), so no shared-memory staging or shuffles are needed;
//   * W4 nibbles become bf16 (128 + q) with one shift and one LOP3 per pair;
//     the group's scale/zero are applied once per group:
//         sum_k (q_k - z) s x_k = s * (sum_k (128 + q_k) x_k - (128 + z) sum_k x_k);
//   * the batch (decode tokens) is the MMA's N dimension, 8 columns per tile;
//   * the 8 warps of a CTA split K by groups; partial tiles are summed in
//     shared memory and the epilogue (residual, SwiGLU, RoPE + KV append)
//     runs on the finished 16-row tile.
#include "internal.h"

namespace river {

namespace {

constexpr int kWarps = 8;

__device__ __forceinline__ uint4 ldg_stream(const void* p) {
  uint4 r;
  asm volatile("ld.global.nc.L1::no_allocate.v4.u32 {%0,%1,%2,%3}, [%4];"
               : "=r"(r.x), "=r"(r.y), "=r"(r.z), "=r"(r.w)
               : "l"(p));
  return r;
}

__device__ __forceinline__ uint4 ldg_x(const void* p) {
  return __ldg(reinterpret_cast<const uint4*>(p));
}

__device__ __forceinline__ void mma_bf16(float (&d)[4], uint32_t a0, uint32_t a1, uint32_t a2,
                                         uint32_t a3, uint32_t b0, uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 "
      "{%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, {%0,%1,%2,%3};"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}

__device__ __forceinline__ uint32_t u4get(const uint4& v, int i) {
  return i == 0 ? v.x : (i == 1 ? v.y : (i == 2 ? v.z : v.w));
}

// Accumulates one 16-row tile's partial sums over this warp's groups.
// Lane (g = lane/4, t = lane%4) owns rows g and g+8 and, in group gi, the
// 32 inputs gi*128 + 32t .. +31.
template <int NT, bool W4>
__device__ __forceinline__ void tile_partial(const GemvArgs& a, int rt, int cb, int warp, int lane,
                                             float (&y)[NT][4]) {
  const int g = lane >> 2, t = lane & 3;
  const int r0 = rt * 16 + g, r1 = r0 + 8;
  const int G = a.Kp >> 7;
#pragma unroll
  for (int j = 0; j < NT; ++j)
#pragma unroll
    for (int i = 0; i < 4; ++i) y[j][i] = 0.f;

  for (int gi = warp; gi < G; gi += kWarps) {
    if constexpr (W4) {
      const int wpr = a.Kp >> 3;  // uint32 words per row
      const uint4 wa = ldg_stream(a.qw + (size_t)r0 * wpr + gi * 16 + 4 * t);
      const uint4 wb = ldg_stream(a.qw + (size_t)r1 * wpr + gi * 16 + 4 * t);
      float acc[NT][4];
#pragma unroll
      for (int j = 0; j < NT; ++j)
#pragma unroll
        for (int i = 0; i < 4; ++i) acc[j][i] = 0.f;
#pragma unroll
      for (int m = 0; m < 4; ++m) {
        const uint32_t va = u4get(wa, m), vb = u4get(wb, m);
        uint4 X[NT];
#pragma unroll
        for (int j = 0; j < NT; ++j) {
          const int col = cb + j * 8 + g;
          X[j] = col < a.B ? ldg_x(a.x + (size_t)col * a.ldx + gi * 128 + 32 * t + 8 * m)
                           : make_uint4(0, 0, 0, 0);
        }
#pragma unroll
        for (int h = 0; h < 2; ++h) {
          // slot pairs: (nibble h, h+4) and (nibble h+2, h+6) of the word
          const uint32_t A0 = ((va >> (4 * h)) & 0x000F000Fu) | 0x43004300u;
          const uint32_t A1 = ((vb >> (4 * h)) & 0x000F000Fu) | 0x43004300u;
          const uint32_t A2 = ((va >> (4 * h + 8)) & 0x000F000Fu) | 0x43004300u;
          const uint32_t A3 = ((vb >> (4 * h + 8)) & 0x000F000Fu) | 0x43004300u;
          const uint32_t sel = h ? 0x7632u : 0x5410u;
#pragma unroll
          for (int j = 0; j < NT; ++j) {
            const uint32_t B0 = __byte_perm(X[j].x, X[j].z, sel);
            const uint32_t B1 = __byte_perm(X[j].y, X[j].w, sel);
            mma_bf16(acc[j], A0, A1, A2, A3, B0, B1);
          }
        }
      }
      const int gpr = a.Kp >> 7;
      const float2 sz0 = __half22float2(a.sz[(size_t)r0 * gpr + gi]);
      const float2 sz1 = __half22float2(a.sz[(size_t)r1 * gpr + gi]);
      const float o0 = 128.f + sz0.y, o1 = 128.f + sz1.y;
#pragma unroll
      for (int j = 0; j < NT; ++j) {
        const int c0 = cb + j * 8 + 2 * t, c1 = c0 + 1;
        const float xs0 = c0 < a.B ? a.xsum[(size_t)c0 * a.ldxs + gi] : 0.f;
        const float xs1 = c1 < a.B ? a.xsum[(size_t)c1 * a.ldxs + gi] : 0.f;
        y[j][0] += sz0.x * (acc[j][0] - o0 * xs0);
        y[j][1] += sz0.x * (acc[j][1] - o0 * xs1);
        y[j][2] += sz1.x * (acc[j][2] - o1 * xs0);
        y[j][3] += sz1.x * (acc[j][3] - o1 * xs1);
      }
    } else {
      const bf16* pa = a.w + (size_t)r0 * a.Kp + gi * 128 + 32 * t;
      const bf16* pb = a.w + (size_t)r1 * a.Kp + gi * 128 + 32 * t;
      uint4 wa[4], wb[4];
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        wa[i] = ldg_stream(pa + 8 * i);
        wb[i] = ldg_stream(pb + 8 * i);
      }
#pragma unroll
      for (int hq = 0; hq < 4; ++hq) {  // 16-byte quarter of the lane's 64 bytes
        uint4 X[NT];
#pragma unroll
        for (int j = 0; j < NT; ++j) {
          const int col = cb + j * 8 + g;
          X[j] = col < a.B ? ldg_x(a.x + (size_t)col * a.ldx + gi * 128 + 32 * t + 8 * hq)
                           : make_uint4(0, 0, 0, 0);
        }
#pragma unroll
        for (int e = 0; e < 2; ++e) {  // step s = 2*hq + e: inputs 32t + 4s .. +3
          const uint32_t A0 = u4get(wa[hq], 2 * e), A2 = u4get(wa[hq], 2 * e + 1);
          const uint32_t A1 = u4get(wb[hq], 2 * e), A3 = u4get(wb[hq], 2 * e + 1);
#pragma unroll
          for (int j = 0; j < NT; ++j)
            mma_bf16(y[j], A0, A1, A2, A3, u4get(X[j], 2 * e), u4get(X[j], 2 * e + 1));
        }
      }
    }
  }
}

__device__ __forceinline__ float silu_f(float v) { return v / (1.f + __expf(-v)); }

// Epilogue on a finished tile: tile[r][c] holds output row rt*16 + r for
// column cb + c (< B).
template <int NT>
__device__ void epilogue(const GemvArgs& a, int rt, int cb, const float (*tile)[NT * 8]) {
  const int tid = threadIdx.x;
  const int ncol = min(NT * 8, a.B - cb);
  if (a.epi == EPI_STORE || a.epi == EPI_RESID) {
    for (int idx = tid; idx < 16 * ncol; idx += blockDim.x) {
      const int c = idx / 16, r = idx % 16;
      const int n = rt * 16 + r;
      const size_t gc = (size_t)(cb + c);
      float v = tile[r][c];
      if (a.epi == EPI_RESID) v += a.resid[gc * a.ldr + n];
      a.out[gc * a.ldo + n] = v;
    }
    return;
  }
  if (a.epi == EPI_SWIGLU) {
    for (int idx = tid; idx < 8 * ncol; idx += blockDim.x) {
      const int c = idx / 8, r = idx % 8;
      const float gv = tile[r][c], uv = tile[r + 8][c];
      a.out_h[(size_t)(cb + c) * a.ldoh + rt * 8 + r] = __float2bfloat16_rn(silu_f(gv) * uv);
    }
    return;
  }
  // EPI_QKV_ROPE: internal row rt*16 + r; within a head, tile j holds dims
  // 8j..8j+7 (rows 0..7) and hd/2 + 8j .. (rows 8..15).
  const int hd = a.hd, half = hd / 2;
  const int row0 = rt * 16;
  const int head_all = row0 / hd;
  const int jt = (row0 % hd) / 16;
  for (int idx = tid; idx < 8 * ncol; idx += blockDim.x) {
    const int c = idx / 8, r = idx % 8;
    const int dim = 8 * jt + r;
    int seq, pos, qrow;
    if (a.T_prefill > 0) {
      const int tok = a.col_base + cb + c;
      seq = tok / a.T_prefill;
      pos = tok % a.T_prefill;
      qrow = tok;
    } else {
      seq = cb + c;
      pos = *a.pos_ptr;
      qrow = cb + c;
    }
    float lo = tile[r][c], hi = tile[r + 8][c];
    if (head_all < a.Hq + a.Hkv) {  // q or k head: rotate
      float sn, cs;
      if (a.rope_cs != nullptr && pos >= 0 && pos < a.Tmax) {
        const float2 cs_sn = a.rope_cs[(size_t)pos * half + dim];
        cs = cs_sn.x;
        sn = cs_sn.y;
      } else {
        sincosf((float)pos * a.inv_freq[dim], &sn, &cs);
      }
      const float nlo = lo * cs - hi * sn;
      const float nhi = hi * cs + lo * sn;
      lo = nlo;
      hi = nhi;
    }
    if (head_all < a.Hq) {
      float* q = a.q_out + (size_t)qrow * a.Hq * hd + head_all * hd;
      q[dim] = lo;
      q[dim + half] = hi;
    } else {
      if (pos < 0 || pos >= a.Tmax) {
        if (idx == 0) atomicOr(a.err, RL_DEVERR_CAPACITY);
        continue;
      }
      const bool is_k = head_all < a.Hq + a.Hkv;
      const int hk = is_k ? head_all - a.Hq : head_all - a.Hq - a.Hkv;
      bf16* cache = is_k ? a.kc : a.vc;
      bf16* dst = cache + (((size_t)seq * a.Hkv + hk) * a.Tmax + pos) * hd;
      dst[dim] = __float2bfloat16_rn(lo);
      dst[dim + half] = __float2bfloat16_rn(hi);
    }
  }
}

template <int NT>
__global__ void __launch_bounds__(kWarps * 32) k_gemv(GemvArgs a) {
  pdl_wait();
  __shared__ float4 red[kWarps][NT][32];
  __shared__ float tile[16][NT * 8];
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  bool w4 = a.w4_mode == W4_ON;
  if (a.w4_mode == W4_BY_LAYER) w4 = a.layer_no > *a.exit_layer;
  if (a.w4_only && !w4) return;  // the tensor-core GEMM ran the bf16 weights
  if (a.path_out != nullptr && blockIdx.x == 0 && threadIdx.x == 0) *a.path_out = w4 ? 1 : 0;
  const int ntiles = a.N / 16;
  const int nitems = ntiles * ((a.B + NT * 8 - 1) / (NT * 8));
  for (int item = blockIdx.x; item < nitems; item += gridDim.x) {
    const int rt = item % ntiles, cb = (item / ntiles) * NT * 8;
    float y[NT][4];
    if (w4)
      tile_partial<NT, true>(a, rt, cb, warp, lane, y);
    else
      tile_partial<NT, false>(a, rt, cb, warp, lane, y);
#pragma unroll
    for (int j = 0; j < NT; ++j) red[warp][j][lane] = make_float4(y[j][0], y[j][1], y[j][2], y[j][3]);
    __syncthreads();
    for (int idx = threadIdx.x; idx < 16 * NT * 8; idx += blockDim.x) {
      const int r = idx / (NT * 8), c = idx % (NT * 8);
      const int j = c / 8, cc = c % 8;
      const int ln = (r % 8) * 4 + cc / 2;
      const int comp = (r >= 8 ? 2 : 0) + (cc & 1);
      float s = 0.f;
#pragma unroll
      for (int w = 0; w < kWarps; ++w) {
        const float4 v = red[w][j][ln];
        s += comp == 0 ? v.x : (comp == 1 ? v.y : (comp == 2 ? v.z : v.w));
      }
      tile[r][c] = s;
    }
    __syncthreads();
    epilogue<NT>(a, rt, cb, tile);
    __syncthreads();
  }
}

}  // namespace

void launch_gemv(const GemvArgs& a, int sm_count, cudaStream_t s) {
  const int ntiles = a.N / 16 * ((a.B + kMaxBatch - 1) / kMaxBatch);
  int grid = sm_count * 4;
  if (grid > ntiles) grid = ntiles;
  if (grid < 1) grid = 1;
  const int nt = (a.B + 7) / 8;
  if (nt <= 1)
    launch_pdl(k_gemv<1>, dim3(grid), dim3(kWarps * 32), 0, s, a);
  else if (nt <= 2)
    launch_pdl(k_gemv<2>, dim3(grid), dim3(kWarps * 32), 0, s, a);
  else if (nt <= 4)
    launch_pdl(k_gemv<4>, dim3(grid), dim3(kWarps * 32), 0, s, a);
  else
    launch_pdl(k_gemv<8>, dim3(grid), dim3(kWarps * 32), 0, s, a);
}

}  // namespace river
