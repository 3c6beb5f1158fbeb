// Fused decode projection for small batches (B <= 8): one kernel per linear
// of a layer, with the work around it folded in.  Warp roles in a CTA:
//
//  * producer warp: streams the weights through a shared-memory ring with
//    bulk asynchronous copies (cp.async.bulk, completion counted on
//    mbarriers).  When the layer's weight path -- bf16 backbone or W4 exit
//    river (River-LLM explainer, section 四: after the exit the remaining
//    layers run on the exit river) -- is already fixed, the copies start
//    BEFORE the programmatic-dependent-launch wait and overlap the previous
//    kernel;
//  * eight consumer warps: mma.sync on the staged weights, the 128-input
//    groups of a 16-row tile spread over the warps, with four independent
//    accumulators per warp so the tensor-core latency pipelines;
//  * reducer warp: sums the eight partial tiles (double-buffered hand-off, no
//    block-wide barrier in the consumers' loop) and runs the epilogue --
//    residual add (+ x' = h * gain and per-tile partial sums for the next
//    RMSNorm and the exit decision), SwiGLU, RoPE + append to the shared KV
//    cache, or logits + argmax.  A tile split between CTAs (stream-K) is
//    completed by the last reducer to arrive (atomic ticket; partials summed
//    in CTA order, so results are deterministic and no CTA waits on another).
//
// Activations arrive as bf16 rows x' = h * gain written by the producing
// epilogue (one bulk copy per row).  RMSNorm's per-token scale
// 1/sqrt(mean(h^2) + eps) factors out of the dot products and is applied in
// the epilogue; it comes from the per-tile partial sums.  For QKV and the LM
// head those partials also give the state-transition cosine of the previous
// layer (residual entering vs leaving it), whose batch minimum is compared
// with tau to fix the step's exit layer (section 四); every CTA computes the
// same decision, CTA 0 records it.
//
// Every mbarrier wait is bounded; on timeout the kernel records
// RL_DEVERR_TIMEOUT, drains its own copies (bounded) and exits.
#include <float.h>

#include "internal.h"

namespace river {

namespace {

constexpr int NC = 8;                    // consumer warps
constexpr int WP = NC;                   // producer warp index
constexpr int kThreads = (NC + 2) * 32;  // + producer + reducer
constexpr int KU = 1024;                 // inputs per work unit (8 groups of 128)
constexpr int RSB = KU * 2 + 64;         // bf16 stage row stride (bytes), 64 mod 128
constexpr int STAGE_B = 16 * RSB;        // bf16 stage bytes
constexpr int STAGE_W = 16 * 512 + 512;  // W4 stage: 16 rows x 512 B nibbles + 16 x 8 (s,z)
constexpr int RING = 3 * STAGE_B;        // ring bytes (3 bf16 stages or 11 W4 stages)
constexpr int SMAX = RING / STAGE_W;     // max stages
constexpr long long kSpin = 1LL << 20;   // bounded mbarrier polls

__device__ __forceinline__ uint32_t smem_u32(const void* p) {
  return (uint32_t)__cvta_generic_to_shared(p);
}
__device__ __forceinline__ void mbar_init(uint64_t* b, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(b)), "r"(count) : "memory");
}
__device__ __forceinline__ void mbar_expect_tx(uint64_t* b, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_u32(b)),
               "r"(bytes)
               : "memory");
}
__device__ __forceinline__ void mbar_arrive(uint64_t* b) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_u32(b)) : "memory");
}
__device__ __forceinline__ bool mbar_try(uint64_t* b, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n .reg .pred p;\n mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n"
      " selp.u32 %0, 1, 0, p;\n}\n"
      : "=r"(ok)
      : "r"(smem_u32(b)), "r"(parity)
      : "memory");
  return ok != 0;
}
// Bounded wait: false on timeout.
__device__ __forceinline__ bool mbar_wait(uint64_t* b, uint32_t parity) {
  for (long long i = 0; i < kSpin; ++i)
    if (mbar_try(b, parity)) return true;
  return false;
}
__device__ __forceinline__ void bulk_g2s(void* dst, const void* src, uint32_t bytes, uint64_t* bar) {
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(
          smem_u32(dst)),
      "l"(src), "r"(bytes), "r"(smem_u32(bar))
      : "memory");
}
__device__ __forceinline__ void grid_dep_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
__device__ __forceinline__ void grid_dep_launch() {
  asm volatile("griddepcontrol.launch_dependents;" :::);
}
__device__ __forceinline__ void consumer_sync() {
  asm volatile("bar.sync 1, %0;" ::"n"(NC * 32) : "memory");
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
__device__ __forceinline__ float f4get(const float4& v, int i) {
  return i == 0 ? v.x : (i == 1 ? v.y : (i == 2 ? v.z : v.w));
}

__device__ __forceinline__ float warp_sum(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
  return v;
}

// CTA owning unit x under the tile partition c0(c) = floor(ntiles*c/grid)*UPT.
__device__ __forceinline__ int chunk_owner(long long x, long long ntiles, int UPT, int grid) {
  const long long tile = x / UPT;
  int c = (int)((tile * grid) / ntiles);
  while (c + 1 < grid && (ntiles * (c + 1)) / grid <= tile) ++c;
  while (c > 0 && (ntiles * c) / grid > tile) --c;
  return c;
}

__device__ __forceinline__ float silu_f(float v) { return v / (1.f + __expf(-v)); }

}  // namespace

__global__ void __launch_bounds__(kThreads, 2) k_gemv_fused(FusedArgs a) {
  extern __shared__ __align__(128) unsigned char smem[];
  __shared__ __align__(8) uint64_t full[SMAX], empty[SMAX], xbar, rfull[2], rempty[2];
  __shared__ float s_col[8][3];
  __shared__ float s_rs[8];
  __shared__ float s_freq[64];
  __shared__ int s_path, s_last;
  __shared__ volatile int s_abort;

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int g = lane >> 2, t = lane & 3;
  const int B = a.B;
  const int G = a.Kp >> 7;
  const int UPT = (a.Kp + KU - 1) / KU;  // units per 16-row tile
  const int ntiles = a.N >> 4;
  const int grid = gridDim.x, cta = blockIdx.x;
  // Whole 16-row tiles per CTA, spread evenly: no tile is shared between CTAs,
  // so no tile ever needs a cross-CTA merge (the stream-K merge below then
  // never triggers; it stays for grids that split tiles).
  const long long c0 = ((long long)ntiles * cta / grid) * UPT;
  const long long c1 = ((long long)ntiles * (cta + 1) / grid) * UPT;
  const int nunits = (int)(c1 - c0);
  const int first_tile = (int)(c0 / UPT);
  const int ntl = nunits > 0 ? (int)((c1 - 1) / UPT) - first_tile + 1 : 0;  // tiles touched
  const int RSX = a.Kp * 2 + 64;  // activation row stride (bytes), 64 mod 128
  const bool scaled = a.xmode != X_COPY;

  unsigned char* ring = smem;
  unsigned char* xs = smem + RING;
  size_t off = RING + (size_t)B * RSX;
  float* xsum = reinterpret_cast<float*>(smem + off);
  off += (((size_t)B * G * 4) + 15) & ~(size_t)15;
  float4* red = reinterpret_cast<float4*>(smem + off);  // [2][NC][32]

  if (tid == 0) {
    for (int i = 0; i < SMAX; ++i) {
      mbar_init(&full[i], 1);
      mbar_init(&empty[i], NC);
    }
    mbar_init(&xbar, 1);
    for (int i = 0; i < 2; ++i) {
      mbar_init(&rfull[i], NC);
      mbar_init(&rempty[i], 1);
    }
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    s_abort = 0;
  }
  if (tid < 8) s_rs[tid] = 1.f;
  __syncthreads();

  // ---- weight path known before the wait? ------------------------------------
  int e_pre = a.L;
  bool certain = true;
  if (a.w4_mode == W4_BY_LAYER) {
    if (a.step_begin) {
      if (a.mode == RL_EXIT_FORCED) {
        e_pre = a.schedule[a.st->step % a.schedule_len];
        e_pre = e_pre < 0 ? 0 : (e_pre > a.L ? a.L : e_pre);
      }
    } else {
      e_pre = a.st->exit_layer;
      // a tau decision taken in this kernel may still move the exit layer
      if (a.dec_layer > 0 && a.mode == RL_EXIT_TAU && e_pre == a.L && a.dec_layer < a.L)
        certain = false;
    }
  }
  const bool w4_pre = a.w4_mode == W4_BY_LAYER && a.layer_no > e_pre;

  // Producer: one lane issues the copies of unit i into ring slot i % S.
  auto issue = [&](bool w4p, int i, int S) {
    const int slot = i % S;
    const long long u = c0 + i;
    const int tl = (int)(u / UPT), uk = (int)(u % UPT);
    const int k0 = uk * KU;
    const int kn = min(KU, a.Kp - k0);
    unsigned char* st = ring + (size_t)slot * (w4p ? STAGE_W : STAGE_B);
    if (w4p) {
      const unsigned char* src =
          reinterpret_cast<const unsigned char*>(a.qwt) + ((size_t)tl * UPT + uk) * STAGE_W;
      mbar_expect_tx(&full[slot], STAGE_W);
      bulk_g2s(st, src, STAGE_W, &full[slot]);
    } else {
      const uint32_t rowb = (uint32_t)kn * 2;
      mbar_expect_tx(&full[slot], 16 * rowb);
      const bf16* src = a.w + (size_t)tl * 16 * a.Kp + k0;
      for (int r = 0; r < 16; ++r)
        bulk_g2s(st + r * RSB, src + (size_t)r * a.Kp, rowb, &full[slot]);
    }
  };

  int issued = 0;
  if (warp == WP && lane == 0 && certain) {
    const int S = w4_pre ? SMAX : RING / STAGE_B;
    for (; issued < nunits && issued < S; ++issued) issue(w4_pre, issued, S);
  }
  const int pos = a.st->pos;  // written by the previous step: stable before the wait

  grid_dep_wait();
  grid_dep_launch();

  // ---- activations ------------------------------------------------------------
  if (warp == WP) {
    if (lane == 0 && a.xmode != X_EMBED) {
      mbar_expect_tx(&xbar, (uint32_t)B * a.Kp * 2);
      for (int b = 0; b < B; ++b)
        bulk_g2s(xs + (size_t)b * RSX, a.xg + (size_t)b * a.ldxg, (uint32_t)a.Kp * 2, &xbar);
    }
  } else if (warp < NC) {
    const int ct = tid;  // consumer thread 0..255
    if (a.epi == EPI_QKV_ROPE && ct < a.hd / 2) s_freq[ct] = a.inv_freq[ct];
    if (a.xmode == X_SCALED) {
      // warp b sums the per-tile partials of column b (all loads in one batch)
      if (warp < B) {
        float acc[3] = {0.f, 0.f, 0.f};
        for (int t0 = 0; t0 < a.stats_tiles; t0 += 32 * 4) {
          float v[4][3];
#pragma unroll
          for (int q = 0; q < 4; ++q) {
            const int tt = t0 + q * 32 + lane;
#pragma unroll
            for (int j = 0; j < 3; ++j)
              v[q][j] = (tt < a.stats_tiles && j < a.stats_k)
                            ? a.stats_in[((size_t)tt * 8 + warp) * a.stats_k + j]
                            : 0.f;
          }
#pragma unroll
          for (int q = 0; q < 4; ++q)
#pragma unroll
            for (int j = 0; j < 3; ++j) acc[j] += v[q][j];
        }
#pragma unroll
        for (int j = 0; j < 3; ++j) acc[j] = warp_sum(acc[j]);
        if (lane == 0) {
          s_col[warp][0] = acc[0];
          s_col[warp][1] = acc[1];
          s_col[warp][2] = acc[2];
        }
      }
    } else if (a.xmode == X_EMBED) {
      // gather the token rows; x' = bf16(e * gain) into shared memory
      const int d = a.d;
      const int nch = d >> 3;  // 8-element chunks per row
      for (int b = 0; b < B; ++b) {
        const int tok_raw = a.tokens[b];
        const int tok = (tok_raw < 0 || tok_raw >= a.vocab) ? 0 : tok_raw;
        if (cta == 0 && ct == 0 && (tok_raw < 0 || tok_raw >= a.vocab))
          atomicOr(&a.st->err, RL_DEVERR_TOKEN);
        float ss = 0.f;
        constexpr int PER = 4;  // chunks per thread per batch (d <= 8192)
        for (int q0 = 0; q0 < nch; q0 += NC * 32 * PER) {
          uint4 e[PER];
          float4 g0[PER], g1[PER];
#pragma unroll
          for (int q = 0; q < PER; ++q) {
            const int ch = q0 + q * NC * 32 + ct;
            if (ch < nch) {
              e[q] = *reinterpret_cast<const uint4*>(a.embed + (size_t)tok * d + ch * 8);
              g0[q] = *reinterpret_cast<const float4*>(a.gain_embed + ch * 8);
              g1[q] = *reinterpret_cast<const float4*>(a.gain_embed + ch * 8 + 4);
            }
          }
#pragma unroll
          for (int q = 0; q < PER; ++q) {
            const int ch = q0 + q * NC * 32 + ct;
            if (ch >= nch) continue;
            const __nv_bfloat162* ev = reinterpret_cast<const __nv_bfloat162*>(&e[q]);
            const float gg[8] = {g0[q].x, g0[q].y, g0[q].z, g0[q].w,
                                 g1[q].x, g1[q].y, g1[q].z, g1[q].w};
            float hv[8];
            uint32_t xw[4];
#pragma unroll
            for (int i = 0; i < 4; ++i) {
              const float2 f = __bfloat1622float2(ev[i]);
              hv[2 * i] = f.x;
              hv[2 * i + 1] = f.y;
              ss += f.x * f.x + f.y * f.y;
              const __nv_bfloat162 xb = __floats2bfloat162_rn(f.x * gg[2 * i], f.y * gg[2 * i + 1]);
              xw[i] = *reinterpret_cast<const uint32_t*>(&xb);
            }
            *reinterpret_cast<uint4*>(xs + (size_t)b * RSX + ch * 16) =
                make_uint4(xw[0], xw[1], xw[2], xw[3]);
            if (cta == 0) {
              float* hs = a.h_store + (size_t)b * d + ch * 8;
              *reinterpret_cast<float4*>(hs) = make_float4(hv[0], hv[1], hv[2], hv[3]);
              *reinterpret_cast<float4*>(hs + 4) = make_float4(hv[4], hv[5], hv[6], hv[7]);
              if (a.trace) {
                float* tr = a.trace + ((size_t)a.trace_layer * a.trace_maxB + b) * d + ch * 8;
                *reinterpret_cast<float4*>(tr) = make_float4(hv[0], hv[1], hv[2], hv[3]);
                *reinterpret_cast<float4*>(tr + 4) = make_float4(hv[4], hv[5], hv[6], hv[7]);
              }
            }
          }
        }
        for (int k = d + ct; k < a.Kp; k += NC * 32)  // zero padding beyond d
          reinterpret_cast<bf16*>(xs + (size_t)b * RSX)[k] = __float2bfloat16_rn(0.f);
        ss = warp_sum(ss);
        if (lane == 0) red[warp * 32 + b] = make_float4(ss, 0.f, 0.f, 0.f);
      }
      consumer_sync();
      if (ct < B) {
        float sum = 0.f;
        for (int w = 0; w < NC; ++w) sum += red[w * 32 + ct].x;
        s_col[ct][0] = sum;
      }
    }
    consumer_sync();
    if (ct == 0) {
      int e = e_pre;
      if (a.step_begin && a.mode == RL_EXIT_FORCED) {
        const int raw = a.schedule[a.st->step % a.schedule_len];
        if ((raw < 0 || raw > a.L) && cta == 0) atomicOr(&a.st->err, RL_DEVERR_SCHEDULE);
      }
      if (a.xmode == X_SCALED && a.dec_layer > 0 && a.stats_k == 3) {
        float m = FLT_MAX;
        for (int b = 0; b < B; ++b) {
          const float ss = s_col[b][0], dot = s_col[b][1], ssp = s_col[b][2];
          m = fminf(m, dot / fmaxf(sqrtf(ssp) * sqrtf(ss), 1e-12f));
        }
        if (a.mode == RL_EXIT_TAU && e == a.L && a.dec_layer < a.L && m > a.tau) e = a.dec_layer;
        if (cta == 0 && a.min_cos_out) a.min_cos_out[a.dec_layer - 1] = m;
      }
      if (cta == 0 && a.w4_mode != W4_OFF && (a.step_begin || a.dec_layer > 0)) a.st->exit_layer = e;
      s_path = (a.w4_mode == W4_BY_LAYER && a.layer_no > e) ? 1 : 0;
      if (scaled)
        for (int b = 0; b < B; ++b) s_rs[b] = 1.f / sqrtf(s_col[b][0] / (float)a.d + a.eps);
    }
  }
  __syncthreads();
  const bool w4 = s_path != 0;
  const int S = w4 ? SMAX : RING / STAGE_B;
  if (a.path_out && cta == 0 && tid == 0) *a.path_out = w4 ? 1 : 0;

  if (warp == WP) {
    // ---- producer: keep the ring full ----------------------------------------
    if (lane == 0) {
      for (int i = issued; i < nunits; ++i) {
        const int slot = i % S;
        if (s_abort || (i >= S && !mbar_wait(&empty[slot], ((i / S) - 1) & 1))) {
          if (!s_abort) atomicOr(&a.st->err, RL_DEVERR_TIMEOUT);
          s_abort = 1;
          break;
        }
        issue(w4, i, S);
        issued = i + 1;
      }
    }
  } else if (warp < NC) {
    // ---- consumers ----------------------------------------------------------------
    if (a.xmode != X_EMBED && !mbar_wait(&xbar, 0)) {
      if (lane == 0) atomicOr(&a.st->err, RL_DEVERR_TIMEOUT);
      s_abort = 1;
    }
    if (w4) {  // per-group sums of the bf16 activations
      for (int gw = warp; gw < B * G; gw += NC) {
        const int b = gw / G, gi = gw % G;
        const uint2 v = *reinterpret_cast<const uint2*>(xs + (size_t)b * RSX + (gi * 128 + 4 * lane) * 2);
        const float2 f0 = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&v.x));
        const float2 f1 = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&v.y));
        const float s2 = warp_sum((f0.x + f0.y) + (f1.x + f1.y));
        if (lane == 0) xsum[b * G + gi] = s2;
      }
      consumer_sync();
    }
    float y[4][4];
#pragma unroll
    for (int j = 0; j < 4; ++j)
#pragma unroll
      for (int i = 0; i < 4; ++i) y[j][i] = 0.f;
    int tcount = 0;
    // column g of the MMA reads activation row min(g, B-1): columns >= B are
    // computed on a duplicate row and discarded, with no divergent branch
    const unsigned char* xrow = xs + (size_t)(g < B ? g : B - 1) * RSX;

    for (int i = 0; i < nunits; ++i) {
      const int slot = i % S;
      bool ok = s_abort == 0 && mbar_wait(&full[slot], (i / S) & 1);
      if (!ok && s_abort == 0) {
        if (lane == 0) atomicOr(&a.st->err, RL_DEVERR_TIMEOUT);
        s_abort = 1;
      }
      const long long u = c0 + i;
      const int uk = (int)(u % UPT);
      const int gi = uk * 8 + warp;  // this warp's group
      const unsigned char* st = ring + (size_t)slot * (w4 ? STAGE_W : STAGE_B);
      if (ok && gi < G) {
        if (w4) {
          // Lane t's word m holds the eight nibbles of input chunk 4m + t of
          // the group (inputs gi*128 + 32m + 8t .. +7); odd rows have their
          // 64-byte halves swapped in the tiled layout.
          const int cw = warp * 4 + t;
          const uint4 wa = *reinterpret_cast<const uint4*>(st + g * 512 + ((cw ^ ((g & 1) << 2)) * 16));
          const uint4 wb = *reinterpret_cast<const uint4*>(st + (g + 8) * 512 +
                                                           ((cw ^ (((g + 8) & 1) << 2)) * 16));
          const uint32_t* szs = reinterpret_cast<const uint32_t*>(st + 16 * 512);
          const uint32_t s0 = szs[g * 8 + (warp ^ (g >> 2))];
          const uint32_t s1 = szs[(g + 8) * 8 + (warp ^ ((g + 8) >> 2))];
          float acc[4][4];
#pragma unroll
          for (int m = 0; m < 4; ++m)
#pragma unroll
            for (int q = 0; q < 4; ++q) acc[m][q] = 0.f;
#pragma unroll
          for (int m = 0; m < 4; ++m) {
            const uint32_t va = u4get(wa, m), vb = u4get(wb, m);
            const uint4 X = *reinterpret_cast<const uint4*>(xrow + (gi * 128 + 32 * m + 8 * t) * 2);
#pragma unroll
            for (int h = 0; h < 2; ++h) {
              const uint32_t A0 = ((va >> (4 * h)) & 0x000F000Fu) | 0x43004300u;
              const uint32_t A1 = ((vb >> (4 * h)) & 0x000F000Fu) | 0x43004300u;
              const uint32_t A2 = ((va >> (4 * h + 8)) & 0x000F000Fu) | 0x43004300u;
              const uint32_t A3 = ((vb >> (4 * h + 8)) & 0x000F000Fu) | 0x43004300u;
              const uint32_t sel = h ? 0x7632u : 0x5410u;
              mma_bf16(acc[m], A0, A1, A2, A3, __byte_perm(X.x, X.z, sel), __byte_perm(X.y, X.w, sel));
            }
          }
          __half2 h0, h1;
          *reinterpret_cast<uint32_t*>(&h0) = s0;
          *reinterpret_cast<uint32_t*>(&h1) = s1;
          const float2 sz0 = __half22float2(h0), sz1 = __half22float2(h1);
          const float xs0 = 2 * t < B ? xsum[(2 * t) * G + gi] : 0.f;
          const float xs1 = 2 * t + 1 < B ? xsum[(2 * t + 1) * G + gi] : 0.f;
          const float o0 = 128.f + sz0.y, o1 = 128.f + sz1.y;
          const float a0 = (acc[0][0] + acc[1][0]) + (acc[2][0] + acc[3][0]);
          const float a1 = (acc[0][1] + acc[1][1]) + (acc[2][1] + acc[3][1]);
          const float a2 = (acc[0][2] + acc[1][2]) + (acc[2][2] + acc[3][2]);
          const float a3 = (acc[0][3] + acc[1][3]) + (acc[2][3] + acc[3][3]);
          y[0][0] += sz0.x * (a0 - o0 * xs0);
          y[0][1] += sz0.x * (a1 - o0 * xs1);
          y[0][2] += sz1.x * (a2 - o1 * xs0);
          y[0][3] += sz1.x * (a3 - o1 * xs1);
        } else {
          // lane t holds the 8-element chunks 4 i4 + t (i4 = 0..3) of the group
#pragma unroll
          for (int i4 = 0; i4 < 4; ++i4) {
            const int cb = warp * 16 + 4 * i4 + t;  // 16-byte chunk within the unit row
            const uint4 wa = *reinterpret_cast<const uint4*>(st + g * RSB + cb * 16);
            const uint4 wb = *reinterpret_cast<const uint4*>(st + (g + 8) * RSB + cb * 16);
            const uint4 X = *reinterpret_cast<const uint4*>(xrow + (uk * KU + cb * 8) * 2);
#pragma unroll
            for (int e = 0; e < 2; ++e)
              mma_bf16(y[i4], u4get(wa, 2 * e), u4get(wb, 2 * e), u4get(wa, 2 * e + 1),
                       u4get(wb, 2 * e + 1), u4get(X, 2 * e), u4get(X, 2 * e + 1));
          }
        }
      }
      __syncwarp();
      if (lane == 0) mbar_arrive(&empty[slot]);
      if (u + 1 == c1 || (u + 1) % UPT == 0) {
        // hand the tile's partial sums to the reducer warp (double buffered)
        const int buf = tcount & 1;
        if (tcount >= 2 && !mbar_wait(&rempty[buf], ((tcount >> 1) - 1) & 1)) s_abort = 1;
        float4 v;
        v.x = (y[0][0] + y[1][0]) + (y[2][0] + y[3][0]);
        v.y = (y[0][1] + y[1][1]) + (y[2][1] + y[3][1]);
        v.z = (y[0][2] + y[1][2]) + (y[2][2] + y[3][2]);
        v.w = (y[0][3] + y[1][3]) + (y[2][3] + y[3][3]);
        red[(buf * NC + warp) * 32 + lane] = v;
#pragma unroll
        for (int j = 0; j < 4; ++j)
#pragma unroll
          for (int q = 0; q < 4; ++q) y[j][q] = 0.f;
        __syncwarp();
        if (lane == 0) mbar_arrive(&rfull[buf]);
        ++tcount;
      }
    }
  } else {
    // ---- reducer warp: tile sums and epilogues ---------------------------------------
    // Lane l holds tile values (r, c) = (l/8 + 4k, l%8), k = 0..3; rows r and
    // r + 8 (k and k + 2) sit in the same lane.
    const int c = lane & 7, rb = lane >> 3;
    float amv = -FLT_MAX;
    int ami = 0x7fffffff;
    for (int tc = 0; tc < ntl; ++tc) {
      const int tl = first_tile + tc;
      const int buf = tc & 1;
      // epilogue inputs that do not depend on the tile sums: fetch first
      float res[4] = {0.f, 0.f, 0.f, 0.f}, hin[4] = {0.f, 0.f, 0.f, 0.f}, gn[4] = {0.f, 0.f, 0.f, 0.f};
      if (a.epi == EPI_RESID && c < B) {
#pragma unroll
        for (int k = 0; k < 4; ++k) {
          const int n = tl * 16 + rb + 4 * k;
          res[k] = a.resid[(size_t)c * a.ldr + n];
          if (a.h_in) hin[k] = a.h_in[(size_t)c * a.d + n];
          if (a.gnext) gn[k] = a.gnext[n];
        }
      }
      if (s_abort || !mbar_wait(&rfull[buf], (tc >> 1) & 1)) {
        if (!s_abort && lane == 0) atomicOr(&a.st->err, RL_DEVERR_TIMEOUT);
        s_abort = 1;
        break;
      }
      float tv[4];
#pragma unroll
      for (int k = 0; k < 4; ++k) {
        const int r = rb + 4 * k;
        const int ln = (r & 7) * 4 + (c >> 1);
        const int comp = (r >= 8 ? 2 : 0) + (c & 1);
        float sum = 0.f;
#pragma unroll
        for (int w = 0; w < NC; ++w) sum += f4get(red[(buf * NC + w) * 32 + ln], comp);
        tv[k] = sum;
      }
      __syncwarp();
      if (lane == 0) mbar_arrive(&rempty[buf]);
      // tile split between CTAs: last reducer to arrive completes it
      const long long tc0 = (long long)tl * UPT, tc1 = tc0 + UPT;
      bool do_epi = true;
      if (tc0 < c0 || tc1 > c1) {
        const int slot = tl == first_tile ? 0 : 1;
        float* wsp = a.ws + ((size_t)cta * 2 + slot) * 128;
#pragma unroll
        for (int k = 0; k < 4; ++k) wsp[lane + 32 * k] = tv[k];
        __threadfence();
        __syncwarp();
        const int oa = chunk_owner(tc0, ntiles, UPT, grid), ob = chunk_owner(tc1 - 1, ntiles, UPT, grid);
        unsigned int last = 0;
        if (lane == 0) last = atomicAdd(&a.tile_ticket[tl], 1u) == (unsigned int)(ob - oa);
        last = __shfl_sync(0xffffffffu, last, 0);
        do_epi = last != 0;
        if (do_epi) {
          __threadfence();
#pragma unroll
          for (int k = 0; k < 4; ++k) tv[k] = 0.f;
          for (int o = oa; o <= ob; ++o) {
            const int ft = (int)(((long long)ntiles * o) / grid);
            const float* p = a.ws + ((size_t)o * 2 + (tl == ft ? 0 : 1)) * 128;
#pragma unroll
            for (int k = 0; k < 4; ++k) tv[k] += __ldcg(p + lane + 32 * k);
          }
          if (lane == 0) a.tile_ticket[tl] = 0u;
        }
      }
      if (!do_epi) continue;
      if (a.epi == EPI_RESID) {
        float s0 = 0.f, s1 = 0.f, s2 = 0.f;
        if (c < B) {
#pragma unroll
          for (int k = 0; k < 4; ++k) {
            const int n = tl * 16 + rb + 4 * k;
            const float v = tv[k] + res[k];
            a.out[(size_t)c * a.ldo + n] = v;
            if (a.trace) a.trace[((size_t)a.trace_layer * a.trace_maxB + c) * a.ldo + n] = v;
            if (a.xnext) a.xnext[(size_t)c * a.ldxnext + n] = __float2bfloat16_rn(v * gn[k]);
            s0 += v * v;
            s1 += v * hin[k];
            s2 += hin[k] * hin[k];
          }
        }
        if (a.stats_out) {  // per-tile partial sums of column c: |h|^2, <h_in, h>, |h_in|^2
#pragma unroll
          for (int o = 8; o < 32; o <<= 1) {
            s0 += __shfl_xor_sync(0xffffffffu, s0, o);
            s1 += __shfl_xor_sync(0xffffffffu, s1, o);
            s2 += __shfl_xor_sync(0xffffffffu, s2, o);
          }
          if (lane < 8 && c < B) {
            float* so = a.stats_out + ((size_t)tl * 8 + c) * a.stats_k_out;
            so[0] = s0;
            if (a.stats_k_out == 3) {
              so[1] = s1;
              so[2] = s2;
            }
          }
        }
      } else if (a.epi == EPI_STORE) {
        if (c < B)
#pragma unroll
          for (int k = 0; k < 4; ++k)
            a.out[(size_t)c * a.ldo + tl * 16 + rb + 4 * k] = tv[k] * s_rs[c];
      } else if (a.epi == EPI_SWIGLU) {
        if (c < B) {
          const float rs = s_rs[c];
#pragma unroll
          for (int k = 0; k < 2; ++k) {
            const float gv = tv[k] * rs, uv = tv[k + 2] * rs;
            a.out_h[(size_t)c * a.ldoh + tl * 8 + rb + 4 * k] = __float2bfloat16_rn(silu_f(gv) * uv);
          }
        }
      } else if (a.epi == EPI_QKV_ROPE) {
        if (c < B) {
          const int hd = a.hd, half = hd >> 1;
          const int row0 = tl * 16;
          const int head_all = row0 / hd;
          const float rs = s_rs[c];
#pragma unroll
          for (int k = 0; k < 2; ++k) {
            const int r = rb + 4 * k;
            const int dim = 8 * ((row0 % hd) >> 4) + r;
            float lo = tv[k] * rs, hi = tv[k + 2] * rs;
            if (head_all < a.Hq + a.Hkv) {
              float sn, cs;
              sincosf((float)pos * s_freq[dim], &sn, &cs);
              const float nlo = lo * cs - hi * sn, nhi = hi * cs + lo * sn;
              lo = nlo;
              hi = nhi;
            }
            if (head_all < a.Hq) {
              float* q = a.q_out + (size_t)c * a.Hq * hd + head_all * hd;
              q[dim] = lo;
              q[dim + half] = hi;
            } else if (pos >= 0 && pos < a.Tmax) {
              const bool is_k = head_all < a.Hq + a.Hkv;
              const int hk = is_k ? head_all - a.Hq : head_all - a.Hq - a.Hkv;
              bf16* dst = (is_k ? a.kc : a.vc) + (((size_t)c * a.Hkv + hk) * a.Tmax + pos) * hd;
              dst[dim] = __float2bfloat16_rn(lo);
              dst[dim + half] = __float2bfloat16_rn(hi);
            } else if (r == 0 && c == 0) {
              atomicOr(&a.st->err, RL_DEVERR_CAPACITY);
            }
          }
        }
      } else {  // EPI_LMHEAD: logits and this lane's running argmax of column c
        if (c < B) {
          const float rs = s_rs[c];
#pragma unroll
          for (int k = 0; k < 4; ++k) {
            const int n = tl * 16 + rb + 4 * k;
            const float v = tv[k] * rs;
            a.out[(size_t)c * a.ldo + n] = v;
            if (v > amv || (v == amv && n < ami)) {
              amv = v;
              ami = n;
            }
          }
        }
      }
    }
    if (a.epi == EPI_LMHEAD) {
#pragma unroll
      for (int o = 8; o < 32; o <<= 1) {
        const float ov = __shfl_xor_sync(0xffffffffu, amv, o);
        const int oi = __shfl_xor_sync(0xffffffffu, ami, o);
        if (ov > amv || (ov == amv && oi < ami)) {
          amv = ov;
          ami = oi;
        }
      }
      if (lane < 8) {
        a.am_val[(size_t)cta * 8 + lane] = amv;
        a.am_idx[(size_t)cta * 8 + lane] = ami;
      }
    }
  }

  // ---- drain: never leave the CTA with copies in flight ------------------------
  __syncthreads();
  if (warp == WP && lane == 0 && s_abort) {
    for (int i = issued - S < 0 ? 0 : issued - S; i < issued; ++i) mbar_wait(&full[i % S], (i / S) & 1);
  }

  // ---- LM head: argmax over CTAs (last arriver), end of the step ---------------
  if (a.epi == EPI_LMHEAD) {
    __threadfence();
    __syncthreads();
    if (tid == 0) s_last = atomicAdd(a.cta_ticket, 1u) == (unsigned int)(grid - 1);
    __syncthreads();
    if (s_last) {
      __threadfence();
      if (warp < B) {  // warp b reduces column b over all CTAs, loads batched
        float bv = -FLT_MAX;
        int bi = 0x7fffffff;
        for (int o0 = 0; o0 < grid; o0 += 32 * 8) {
          float v[8];
          int ix[8];
#pragma unroll
          for (int q = 0; q < 8; ++q) {
            const int o = o0 + q * 32 + lane;
            v[q] = o < grid ? __ldcg(a.am_val + (size_t)o * 8 + warp) : -FLT_MAX;
            ix[q] = o < grid ? __ldcg(a.am_idx + (size_t)o * 8 + warp) : 0x7fffffff;
          }
#pragma unroll
          for (int q = 0; q < 8; ++q)
            if (v[q] > bv || (v[q] == bv && ix[q] < bi)) {
              bv = v[q];
              bi = ix[q];
            }
        }
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) {
          const float ov = __shfl_xor_sync(0xffffffffu, bv, o);
          const int oi = __shfl_xor_sync(0xffffffffu, bi, o);
          if (ov > bv || (ov == bv && oi < bi)) {
            bv = ov;
            bi = oi;
          }
        }
        if (lane == 0 && a.next_token) a.next_token[warp] = bi == 0x7fffffff ? 0 : bi;
      }
      if (tid == 0) {
        DevState* st = a.st;
        if (a.exit_out) a.exit_out[0] = st->exit_layer;
        st->pos = st->pos + 1;
        st->step = st->step + 1;
        *a.cta_ticket = 0u;
        __threadfence();
      }
    }
  }
}

size_t fused_smem_bytes(const FusedArgs& a) {
  const int G = a.Kp / 128;
  size_t off = RING + (size_t)a.B * (a.Kp * 2 + 64);
  off += (((size_t)a.B * G * 4) + 15) & ~(size_t)15;
  off += (size_t)2 * NC * 32 * 16;
  return off;
}

int fused_grid(const FusedArgs& a, int sm_count) {
  const int ntiles = a.N / 16;
  return ntiles < sm_count ? ntiles : sm_count;
}

size_t w4_tiled_bytes(int N, int Kp) {
  return (size_t)(N / 16) * ((Kp + KU - 1) / KU) * STAGE_W;
}

void gemv_fused_setup() {
  cudaFuncSetAttribute(k_gemv_fused, cudaFuncAttributeMaxDynamicSharedMemorySize, 220 * 1024);
  // one shared-memory carveout for every decode kernel: switching the L1 /
  // shared split between consecutive kernels would drain the SMs
  cudaFuncSetAttribute(k_gemv_fused, cudaFuncAttributePreferredSharedMemoryCarveout,
                       cudaSharedmemCarveoutMaxShared);
}

cudaError_t launch_gemv_fused(const FusedArgs& a, int sm_count, bool pdl, cudaStream_t s) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(fused_grid(a, sm_count));
  cfg.blockDim = dim3(kThreads);
  cfg.dynamicSmemBytes = fused_smem_bytes(a);
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = pdl ? 1 : 0;
  return cudaLaunchKernelEx(&cfg, k_gemv_fused, a);
}

// ---------------------------------------------------------------------------
// W4 copy in the unit-tiled layout the ring consumes.  For 16-row tile T and
// 1024-input unit u, one contiguous STAGE_W block: 16 rows x 512 bytes of
// nibbles, then 16 x 8 (scale, zero) pairs.  Within a row, the 64 bytes of
// group w hold its 16 words transposed (position 4t + m <- word 4m + t), so
// lane t of the consuming fragment reads input chunks 4m + t; odd rows store
// their 16-byte chunk c at c ^ 4 (swapped 64-byte halves).  (s, z) of row r,
// group w sits at r*8 + (w ^ (r >> 2)).  Padding beyond Kp is zero.  These
// permutations keep every shared-memory read of the consumer bank-conflict
// free.
// ---------------------------------------------------------------------------
__global__ void k_w4_tile_layout(const uint32_t* __restrict__ qw, const __half2* __restrict__ sz,
                                 int N, int Kp, unsigned char* __restrict__ out) {
  const int G = Kp / 128, UPT = (Kp + KU - 1) / KU;
  const long long blk = blockIdx.x;  // one block per (tile, unit)
  const int tl = (int)(blk / UPT), uk = (int)(blk % UPT);
  unsigned char* dst = out + blk * STAGE_W;
  for (int idx = threadIdx.x; idx < 16 * 128; idx += blockDim.x) {  // words of the unit
    const int r = idx >> 7, wd = idx & 127;                         // destination word in the row
    const int grp = wd >> 4, p = wd & 15, tt = p >> 2, m = p & 3;   // position p = 4t + m
    const int src_word = uk * 128 + grp * 16 + 4 * m + tt;          // word 4m + t of the group
    uint32_t v = 0;
    if (uk * 8 + grp < G) v = qw[(size_t)(tl * 16 + r) * (Kp / 8) + src_word];
    const int chunk = wd >> 2, within = wd & 3;
    reinterpret_cast<uint32_t*>(dst + r * 512 + ((chunk ^ ((r & 1) << 2)) * 16))[within] = v;
  }
  for (int idx = threadIdx.x; idx < 16 * 8; idx += blockDim.x) {
    const int r = idx >> 3, w = idx & 7;
    const int gi = uk * 8 + w;
    __half2 v = __floats2half2_rn(0.f, 0.f);
    if (gi < G) v = sz[(size_t)(tl * 16 + r) * G + gi];
    reinterpret_cast<__half2*>(dst + 16 * 512)[r * 8 + (w ^ (r >> 2))] = v;
  }
}

void launch_w4_tile_layout(const uint32_t* qw, const __half2* sz, int N, int Kp, void* out,
                           cudaStream_t s) {
  const long long blocks = (long long)(N / 16) * ((Kp + KU - 1) / KU);
  k_w4_tile_layout<<<(unsigned)blocks, 256, 0, s>>>(qw, sz, N, Kp, static_cast<unsigned char*>(out));
}

}  // namespace river
