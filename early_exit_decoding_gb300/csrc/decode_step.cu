// Persistent decode step for small batches (B <= 8): ONE cooperative kernel
// per decode step runs every phase -- for each layer QKV (+ exit decision,
// RoPE, KV append), attention (the last CTA of each KV head merges its chunks), O (+ residual), gate/up (+ SwiGLU), down
// (+ residual, next RMSNorm input, cosine partials); then the LM head (+
// greedy argmax).  River-LLM explainer, section 四: the batch-minimum cosine of
// a layer's input and output residual decides, once, that the remaining
// layers run on the W4A16 exit river; section 三: those layers write K/V into
// the backbone's own cache slot.
//
// One CTA per SM, warp-specialised:
//   * producer warp: streams, through a ring of shared-memory slots, every
//     weight unit (16 rows x 1024 inputs bf16, or four 16 x 1024 W4 units with
//     their scales/zeros, one bulk copy each) and every K/V chunk this CTA will
//     consume in the whole step, in consumption order.  None of that depends on
//     this step's activations, so the stream runs ahead across phase
//     boundaries; it only waits for free slots and -- in tau mode, before the
//     exit -- for this CTA's exit decision of the previous layer, which picks
//     bf16 or W4 weights for the next one;
//   * eight consumer warps: wait for the previous phase (grid-wide arrival
//     counter); reduce the norm / cosine statistics while the phase's
//     activation rows arrive; run mma.sync on the staged weights, each warp on
//     its own 128 inputs of every unit, keeping per-warp partial tiles in
//     shared memory; every few tiles, all 256 threads sum the partials (fixed
//     order: deterministic) and run the epilogue in parallel.
// A CTA takes the 16-row tiles cta, cta + grid, ... of each projection.  Every
// wait is bounded: on timeout the kernel sets RL_DEVERR_TIMEOUT and winds down
// without touching more memory.
#include <type_traits>

#include "dev_common.cuh"
#include "attn_tc.cuh"

namespace river {

namespace {

using namespace dev;
using namespace attn;

constexpr int NC = 8;                     // consumer warps
constexpr int WP = NC;                    // producer warp
constexpr int kThreads = (NC + 1) * 32;
constexpr int KU = 1024;                  // inputs per unit
constexpr int STAGE_W = 16 * 512 + 512;   // one W4 unit: 16 rows x 512 B nibbles + 16 x 8 (s, z)
constexpr int W4U = 4;                    // W4 units per ring slot
constexpr int SLOT_B = W4U * STAGE_W;     // 34816 bytes (>= 32 KB bf16 unit, >= K+V chunk)
constexpr int kMaxSlots = 8;
constexpr int kCHP = 128;                 // positions per attention chunk
constexpr int kAttnHalf = 16384;          // V offset in a one-slot chunk (head_dim 64)
constexpr long long kSpin = 1LL << 20;     // mbarrier polls
constexpr long long kSpinBar = 1LL << 24;  // grid-barrier polls (each with a short sleep)
// kWide producer's slot wait, in ns of %globaltimer: a whole warp polling
// spends a poll budget far faster than one lane, and with layers read from
// host memory a slot can stay taken for milliseconds at a phase boundary
constexpr unsigned long long kWaitNsWide = 4000000000ull;
constexpr int kBarCons = 1;                // named barrier: consumer warps
constexpr int kStaticSmem = 12 * 1024;     // upper bound of the kernel's static shared memory

// Position in the ring of shared-memory slots: slot index and how many times
// the ring has wrapped (the mbarrier phase parity), advanced without divisions.
struct RingPos {
  int slot, round;
  __device__ __forceinline__ void next(int ns) {
    if (++slot == ns) {
      slot = 0;
      ++round;
    }
  }
};

// Timeline of a profiled step: tl[p] = first start of phase p over CTAs,
// tl[nph + p] = last end.
__device__ __forceinline__ void tl_mark(unsigned long long* tl, int nph, int p, int which) {
  if (!tl) return;
  unsigned long long t;
  asm volatile("mov.u64 %0, %globaltimer;" : "=l"(t));
  if (which == 0)
    atomicMin(tl + p, t);
  else
    atomicMax(tl + nph + p, t);
}

// Per-CTA timeline stamp (profiling only).
__device__ __forceinline__ void tl2_mark(unsigned long long* tl2, int grid, int p, int cta, int k) {
  if (!tl2) return;
  unsigned long long t;
  asm volatile("mov.u64 %0, %globaltimer;" : "=l"(t));
  tl2[((size_t)p * grid + cta) * kTl2 + k] = t;
}

// One W4 unit of the step kernel's consumer warp: this warp's 128-input group
// gi of 16 weight rows (stage `st`) against the activation rows.  Lane t's word
// m holds the eight nibbles of input chunk 4m + t of the group; odd rows have
// their 64-byte halves swapped.  Each nibble field, masked in place, is the bit
// pattern of the subnormal fp16 q * 2^-24 (fields at bits 4..7 read
// 16 q * 2^-24): one AND per operand register, exact products in the MMA.  The
// activations are fp16, scaled and reordered per 8-input chunk as (x0,x4),
// (x2,x6), (x1,x5), (x3,x7), each group scaled by 2^k; xsum holds per
// (row, group) the input sum and 2^-k.
__device__ __forceinline__ void w4_unit(const unsigned char* st, int gi, const unsigned char* xrow,
                                        const float* xsum, int B, int G, int warp, int g, int t,
                                        float (&y)[4]) {
  const int cw = warp * 4 + t;
  const uint4 wa = *reinterpret_cast<const uint4*>(st + g * 512 + ((cw ^ ((g & 1) << 2)) * 16));
  const uint4 wb = *reinterpret_cast<const uint4*>(st + (g + 8) * 512 + ((cw ^ (((g + 8) & 1) << 2)) * 16));
  const uint32_t* szs = reinterpret_cast<const uint32_t*>(st + 16 * 512);
  const uint32_t s0 = szs[g * 8 + (warp ^ (g >> 2))];
  const uint32_t s1 = szs[(g + 8) * 8 + (warp ^ ((g + 8) >> 2))];
  float c1[4], c2[4];
#pragma unroll
  for (int q = 0; q < 4; ++q) c1[q] = c2[q] = 0.f;
#pragma unroll
  for (int m = 0; m < 4; ++m) {
    const uint32_t va = u4get(wa, m), vb = u4get(wb, m), ha = va >> 8, hb = vb >> 8;
    const uint4 X = *reinterpret_cast<const uint4*>(xrow + (gi * 128 + 32 * m + 8 * t) * 2);
    mma_f16(c1, va & 0x000F000Fu, vb & 0x000F000Fu, ha & 0x000F000Fu, hb & 0x000F000Fu, X.x, X.y);
    mma_f16(c2, va & 0x00F000F0u, vb & 0x00F000F0u, ha & 0x00F000F0u, hb & 0x00F000F0u, X.z, X.w);
  }
  __half2 h0, h1;
  *reinterpret_cast<uint32_t*>(&h0) = s0;
  *reinterpret_cast<uint32_t*>(&h1) = s1;
  const float2 sz0 = __half22float2(h0), sz1 = __half22float2(h1);
  const float2* xs2 = reinterpret_cast<const float2*>(xsum);
  const float2 xa = 2 * t < B ? xs2[(2 * t) * G + gi] : make_float2(0.f, 0.f);
  const float2 xb = 2 * t + 1 < B ? xs2[(2 * t + 1) * G + gi] : make_float2(0.f, 0.f);
  // sum_k (q_k - z) s x_k = s 2^24 2^-k (c1 + c2 / 16) - s z sum_k x_k
  const float p0 = sz0.x * 16777216.f, p1 = sz1.x * 16777216.f;
  const float q0 = sz0.x * sz0.y, q1 = sz1.x * sz1.y;
  float av[4];
#pragma unroll
  for (int c = 0; c < 4; ++c) av[c] = c1[c] + 0.0625f * c2[c];
  y[0] = fmaf(p0 * xa.y, av[0], fmaf(-q0, xa.x, y[0]));
  y[1] = fmaf(p0 * xb.y, av[1], fmaf(-q0, xb.x, y[1]));
  y[2] = fmaf(p1 * xa.y, av[2], fmaf(-q1, xa.x, y[2]));
  y[3] = fmaf(p1 * xb.y, av[3], fmaf(-q1, xb.x, y[3]));
}

}  // namespace

// kMulti: the attention may give a CTA more than one chunk (contexts where
// B x KV heads x 128-position chunks exceed the grid); each CTA then takes
// consecutive chunks, and two chunks of one head group are folded into one
// partial before the merge.  Otherwise chunks are dealt round-robin (one per
// CTA at the contexts that instantiation is launched for).
// kWide: the model has offloaded layers, whose units the producer warp reads
// from host memory with 16-byte copies of all 32 lanes (one lane issuing
// them reaches ~91 GB/s over the whole GPU).  The whole warp then walks the
// copy schedule; otherwise lane 0 alone does (the warp-wide walk measured
// 1-2 % slower on resident models, which keep the single-lane one).
template <bool kMulti, bool kWide>
__global__ void __launch_bounds__(kThreads, 1) k_decode_step(const __grid_constant__ StepArgs a) {
  extern __shared__ __align__(128) unsigned char smem[];
  __shared__ __align__(8) uint64_t full[kMaxSlots], empty[kMaxSlots], xbar;
  __shared__ __align__(16) PhaseDesc cdesc;  // consumers' copy of the current phase
  __shared__ float s_col[8][3];              // per column: the phase's reduced statistics
  __shared__ float s_stw[NC][24];            // per warp partial statistics
  __shared__ float s_rs[8];
  __shared__ float s_freq[64];
  __shared__ volatile int s_e;    // exit layer as far as this CTA knows it
  __shared__ volatile int s_dec;  // last layer whose exit decision this CTA has taken
  __shared__ volatile int s_abort;
  __shared__ int s_pos, s_last, s_merge;
  __shared__ __align__(16) float s_mrg[4 * NC];  // LM-head argmax scratch: per half warp (value, index)

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int g = lane >> 2, t = lane & 3;
  const int grid = gridDim.x, cta = blockIdx.x;
  const int B = a.B, NS = a.nslot, RSX = a.xs_row_bytes;
  // the ring starts on a 1024-byte boundary (128-byte-swizzled TMA destinations)
  unsigned char* ring = smem + ((1024u - (smem_u32(smem) & 1023u)) & 1023u);
  unsigned char* xs = ring + (size_t)NS * SLOT_B;
  float* xsum = reinterpret_cast<float*>(xs + (size_t)B * RSX);
  float4* red = reinterpret_cast<float4*>(reinterpret_cast<unsigned char*>(xsum) +
                                          ((((size_t)B * a.gmax * 8) + 15) & ~(size_t)15));
  float* redf = reinterpret_cast<float*>(red);

  if (tid == 0) {
    for (int i = 0; i < NS; ++i) {
      mbar_init(&full[i], 1);
      mbar_init(&empty[i], NC);
    }
    mbar_init(&xbar, 1);
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    s_abort = 0;
    s_pos = a.st->pos;
    int e = a.L;
    if (a.mode == RL_EXIT_FORCED) {
      e = a.schedule[a.st->step % a.schedule_len];
      e = e < 0 ? 0 : (e > a.L ? a.L : e);
    }
    s_e = e;
    s_dec = 0;
  }
  if (tid < 8) s_rs[tid] = 1.f;
  if (tid < 64) s_freq[tid] = tid < a.hd / 2 ? a.inv_freq[tid] : 0.f;
  __syncthreads();

  if (warp == WP) {
    // ================================ producer ===================================
    // (kWide: every lane walks the same schedule; lane 0 waits for slots and
    // issues the bulk and tensor copies; decisions that read shared state are
    // lane 0's, broadcast.)
    if (kWide || lane == 0) {
      const bool l0 = !kWide || lane == 0;
      auto uni = [&](bool v) -> bool {
        if constexpr (kWide) return __shfl_sync(0xffffffffu, (int)v, 0) != 0;
        return v;
      };
      RingPos rp{0, 0};
      int issued = 0;
      int e_known = s_e;
      auto take_slot = [&]() -> bool {
        if (rp.round == 0) return true;
        bool ok = true;
        if (l0) {
          if (s_abort) {
            ok = false;
          } else if (!(kWide ? mbar_wait_for(&empty[rp.slot], (uint32_t)((rp.round - 1) & 1), kWaitNsWide)
                             : mbar_wait(&empty[rp.slot], (uint32_t)((rp.round - 1) & 1), kSpin))) {
            atomicOr(&a.st->err, RL_DEVERR_TIMEOUT);
            s_abort = 1;
            ok = false;
          } else {
            // consumers that aborted free slots without waiting for their
            // copies: never issue into such a slot (the arrival orders their
            // abort flag before it)
            ok = !s_abort;
          }
        }
        return uni(ok);
      };
      for (int p = 0; p < a.nph && !uni(s_abort); ++p) {
        const PhaseDesc* D = a.ph + p;
        bool first_copy = true;
        auto stamp_copy = [&]() {
          if (!a.tl2 || !l0) return;
          if (first_copy) tl2_mark(a.tl2, grid, p, cta, TL2_P0);
          first_copy = false;
          tl2_mark(a.tl2, grid, p, cta, TL2_P1);
        };
        if (D->kind == PH_GEMV) {
          const int layer_no = D->layer_no;
          const unsigned char* qwt = D->qwt;
          const bf16* wt = D->wt;
          const bool wt_sys = D->wt_sys != 0;
          const int N = D->N, Kp = D->Kp;
          bool w4 = false;
          if (qwt && layer_no > 0) {
            if (a.mode == RL_EXIT_TAU && e_known >= a.L && layer_no >= 2) {
              // the weight path of this layer waits for the exit decision of the previous one
              bool decided = true;
              int e_now = 0;
              if (l0) {
                long long i = 0;
                while (s_dec < layer_no - 1 && !s_abort && i < kSpinBar) {
                  __nanosleep(64);
                  ++i;
                }
                decided = s_dec >= layer_no - 1;
                if (!decided) {
                  if (!s_abort) atomicOr(&a.st->err, RL_DEVERR_TIMEOUT);
                  s_abort = 1;
                }
                e_now = s_e;
              }
              if (!uni(decided)) break;
              if constexpr (kWide)
                e_known = __shfl_sync(0xffffffffu, e_now, 0);
              else
                e_known = e_now;
            }
            w4 = layer_no > e_known;
          }
          // whole 16-row tiles cta, cta + grid, ... (the consumers walk the same list)
          const int UPT = (Kp + KU - 1) / KU, ntiles = N >> 4;
          for (int tl = cta; tl < ntiles && !uni(s_abort); tl += grid) {
            if (w4) {
              for (int s0 = 0; s0 < UPT; s0 += W4U) {
                if (!take_slot()) break;
                const int ns = min(W4U, UPT - s0);
                const int slot = rp.slot;
                if (l0) {
                  mbar_expect_tx(&full[slot], (uint32_t)(ns * STAGE_W));
                  bulk_g2s(ring + (size_t)slot * SLOT_B, qwt + ((size_t)tl * UPT + s0) * STAGE_W,
                           (uint32_t)(ns * STAGE_W), &full[slot]);
                }
                stamp_copy();
                rp.next(NS);
                ++issued;
              }
            } else {
              for (int uk = 0; uk < UPT; ++uk) {
                if (!take_slot()) break;
                const int k0 = uk * KU, kn = min(KU, Kp - k0);
                const int slot = rp.slot;
                const uint32_t bytes = (uint32_t)(16 * kn * 2);
                const unsigned char* src =
                    reinterpret_cast<const unsigned char*>(wt + (size_t)tl * 16 * Kp + (size_t)16 * k0);
                unsigned char* dst = ring + (size_t)slot * SLOT_B;
                if (wt_sys) {
                  // an offloaded layer's unit from host memory: 16-byte copies on
                  // the load path
                  if constexpr (kWide) {
                    // by every lane, waited for here (the host link, not the
                    // wait, bounds these units); lane 0's arrival after every
                    // lane's copies have landed is the slot's one expected one
                    for (uint32_t o = (uint32_t)lane * 16; o < bytes; o += 32 * 16) cp_async16(dst + o, src + o);
                    asm volatile("cp.async.wait_all;" ::: "memory");
                    __syncwarp();
                    if (l0) mbar_arrive(&full[slot]);
                  } else {
                    // lane 0 alone: their landing is the slot's one expected arrival
                    for (uint32_t o = 0; o < bytes; o += 16) cp_async16(dst + o, src + o);
                    cp_async_mbar_arrive(&full[slot]);
                  }
                } else if (l0) {
                  mbar_expect_tx(&full[slot], bytes);
                  bulk_g2s(dst, src, bytes, &full[slot]);
                }
                stamp_copy();
                rp.next(NS);
                ++issued;
              }
            }
          }
        } else if (D->kind == PH_ATTN) {
          // attention: the chunk's K and V rows by TMA in 16-row boxes of 64
          // dims (128-byte swizzle), every row a warp may read (ceil16 of the
          // chunk); the row at this step's position is rewritten by the
          // consumers once it has landed.  head_dim 64: K and V in one slot (V
          // at 16 KB); head_dim 128: K in one slot, V in the next, each as two
          // 64-dim halves 16 KB apart.
          const int pos = s_pos, hd = a.hd, Hkv = a.Hkv;
          const int ctx = min(pos + 1, a.Tmax);
          const int nch = step_attn_chunks(ctx, B, Hkv, hd, grid, a.part_cap);
          const int clen = (ctx + nch - 1) / nch;
          const int nitems = B * Hkv * nch;
          const bool two = hd * 2 * kCHP > kAttnHalf;
          const int halves = hd / 64;
          const int lrow0 = (D->layer_no - 1) * a.kv_rows_layer;
          // kMulti: CTA c takes the consecutive chunks c*per .. c*per + per - 1
          // (mostly of one head group), so every group's last chunk ends in the
          // last round; else chunks c, c + grid, ...
          const int per = kMulti ? (nitems + grid - 1) / grid : 1;
          const int it0 = kMulti ? cta * per : cta, it_end = kMulti ? min(nitems, cta * per + per) : nitems;
          for (int it = it0; it < it_end && !uni(s_abort); it += kMulti ? 1 : grid) {
            const int b = it / (Hkv * nch), rr = it % (Hkv * nch), hk = rr / nch, ch = rr % nch;
            const int start = ch * clen, end = min(start + clen, ctx);
            const int n = min(kCHP, max(0, end - start));
            const int nbox = (n + 15) >> 4;
            const int row0 = lrow0 + (b * Hkv + hk) * a.Tmax + start;
            const uint32_t bytes = (uint32_t)(nbox * 2048 * halves);  // per tensor (K or V)
            auto load = [&](const CUtensorMap* tm, unsigned char* dst, uint64_t* bar) {
              for (int h = 0; h < halves; ++h)
                for (int i = 0; i < nbox; ++i) tma_load_2d(dst + h * 16384 + i * 2048, tm, h * 64, row0 + 16 * i, bar);
            };
            if (!take_slot()) break;
            const int sk = rp.slot;
            rp.next(NS);
            ++issued;
            stamp_copy();
            if (!two) {
              if (l0) {
                mbar_expect_tx(&full[sk], 2 * bytes);
                load(&a.tmk, ring + (size_t)sk * SLOT_B, &full[sk]);
                load(&a.tmv, ring + (size_t)sk * SLOT_B + kAttnHalf, &full[sk]);
              }
            } else {
              if (l0) {
                mbar_expect_tx(&full[sk], bytes);
                load(&a.tmk, ring + (size_t)sk * SLOT_B, &full[sk]);
              }
              if (!take_slot()) break;
              const int sv = rp.slot;
              rp.next(NS);
              ++issued;
              if (l0) {
                mbar_expect_tx(&full[sv], bytes);
                load(&a.tmv, ring + (size_t)sv * SLOT_B, &full[sv]);
              }
            }
          }
        }
      }
      // never leave with copies in flight: this lane's host-memory copies,
      // and (lane 0) the last NS issued units
      if constexpr (kWide) asm volatile("cp.async.wait_all;" ::: "memory");
      if (l0 && s_abort)
        for (int u = issued - NS < 0 ? 0 : issued - NS; u < issued; ++u)
          mbar_wait(&full[u % NS], (uint32_t)((u / NS) & 1), kSpin);
    }
  } else {
    // ================================ consumers ==================================
    const int ct = tid;
    RingPos rc{0, 0};
    uint32_t xpar = 0;
    float amv = -FLT_MAX;  // LM head: running argmax of this thread's outputs
    int ami = 0x7fffffff;
    for (int p = 0; p < a.nph; ++p) {
      {
        const int* src = reinterpret_cast<const int*>(a.ph + p);
        int* dst = reinterpret_cast<int*>(&cdesc);
        for (int i = ct; i < (int)(sizeof(PhaseDesc) / 4); i += NC * 32) dst[i] = __ldg(src + i);
      }
      if (p > 0 && ct < grid && !s_abort) {
        // every CTA has finished phase p - 1: thread j waits for CTA j's flag
        // (CTA j stores p after its phase p - 1; flags sit 128 bytes apart)
        const unsigned* fp = a.bars + (size_t)ct * 32;
        const long long lim = a.bar_wait > 0 ? a.bar_wait : kSpinBar;
        bool arrived = false;
        for (long long i = 0; i < lim && !arrived; ++i) arrived = ld_acquire(fp) >= (unsigned)p;
        if (!arrived) {
          atomicOr(&a.st->err, RL_DEVERR_TIMEOUT);
          s_abort = 1;
        }
        if (ct == 0) fence_proxy_async();  // the phase's bulk copies read other CTAs' writes
      }
      named_sync(kBarCons, NC * 32);
      if (ct == 0) {
        tl_mark(a.tl, a.nph, p, 0);
        tl2_mark(a.tl2, grid, p, cta, TL2_BAR);
      }
      const PhaseDesc& D = cdesc;

      if (D.kind == PH_GEMV) {
        const int Kp = D.Kp, G = Kp >> 7;
        // ---- activation rows (bulk copy), concurrently with the statistics ----
        // (issued and waited for even after an abort: the CTA never leaves
        // with a copy in flight)
        if (D.xmode != X_EMBED && ct == 0) {
          mbar_expect_tx(&xbar, (uint32_t)B * Kp * 2);
          for (int b = 0; b < B; ++b)
            bulk_g2s(xs + (size_t)b * RSX, D.xg + (size_t)b * D.ldxg, (uint32_t)Kp * 2, &xbar);
        }
        if (D.xmode == X_EMBED) {
          // gather the token rows; x' = bf16(e * gain) into shared memory
          const int d = a.d, nchk = d >> 3;
          for (int b = 0; b < B; ++b) {
            const int tok_raw = a.tokens[b];
            const int tok = (tok_raw < 0 || tok_raw >= a.vocab) ? 0 : tok_raw;
            if (cta == 0 && ct == 0 && (tok_raw < 0 || tok_raw >= a.vocab))
              atomicOr(&a.st->err, RL_DEVERR_TOKEN);
            float ss = 0.f;
            constexpr int PER = 4;
            for (int q0 = 0; q0 < nchk; q0 += NC * 32 * PER) {
              uint4 e[PER];
              float4 g0[PER], g1[PER];
#pragma unroll
              for (int q = 0; q < PER; ++q) {
                const int ch = q0 + q * NC * 32 + ct;
                if (ch < nchk) {
                  e[q] = *reinterpret_cast<const uint4*>(a.embed + (size_t)tok * d + ch * 8);
                  g0[q] = *reinterpret_cast<const float4*>(a.gain_embed + ch * 8);
                  g1[q] = *reinterpret_cast<const float4*>(a.gain_embed + ch * 8 + 4);
                }
              }
#pragma unroll
              for (int q = 0; q < PER; ++q) {
                const int ch = q0 + q * NC * 32 + ct;
                if (ch >= nchk) continue;
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
                  if (D.trace) {
                    float* tr = D.trace + ((size_t)D.trace_layer * a.trace_maxB + b) * d + ch * 8;
                    *reinterpret_cast<float4*>(tr) = make_float4(hv[0], hv[1], hv[2], hv[3]);
                    *reinterpret_cast<float4*>(tr + 4) = make_float4(hv[4], hv[5], hv[6], hv[7]);
                  }
                }
              }
            }
            for (int k = d + ct; k < Kp; k += NC * 32)
              reinterpret_cast<bf16*>(xs + (size_t)b * RSX)[k] = __float2bfloat16_rn(0.f);
            fence_proxy_async_smem();  // later phases bulk-copy into these bytes
            ss = warp_sum(ss);
            if (lane == 0) red[warp * 32 + b] = make_float4(ss, 0.f, 0.f, 0.f);
          }
          named_sync(kBarCons, NC * 32);
          if (ct < B) {
            float sum = 0.f;
            for (int w = 0; w < NC; ++w) sum += red[w * 32 + ct].x;
            s_col[ct][0] = sum;
          }
        }
        // ---- statistics of the producing phase (X_SCALED): per column sums of its
        // per-tile partials (|h|^2; with three partials also <h_in, h> and
        // |h_in|^2).  The loads are issued now; the reduction waits for the first
        // epilogue unless the exit decision is needed first (tau mode, not yet
        // exited: it picks this layer's weights).
        const int sk = D.stats_k;
        const bool scaled = D.xmode == X_SCALED;
        const bool regs = scaled && B * sk <= 6 && D.stats_tiles <= NC * 32;
        float pv[6];
#pragma unroll
        for (int i = 0; i < 6; ++i) pv[i] = 0.f;
        if (regs && ct < D.stats_tiles) {
          const float* sp = D.stats_in + (size_t)ct * 8 * sk;
#pragma unroll
          for (int i = 0; i < 6; ++i)
            if (i < B * sk) pv[i] = __ldcg(sp + i);
        }
        // (1) per-warp partial sums into s_stw (no barrier)
        auto stats_partials = [&]() {
          if (regs) {
#pragma unroll
            for (int i = 0; i < 6; ++i)
              if (i < B * sk) {
                const float v = warp_sum(pv[i]);
                if (lane == 0) s_stw[warp][(i / sk) * 3 + i % sk] = v;
              }
          } else {
            float acc[kFusedMaxB][3];
#pragma unroll
            for (int b = 0; b < kFusedMaxB; ++b)
#pragma unroll
              for (int j = 0; j < 3; ++j) acc[b][j] = 0.f;
            for (int tt = ct; tt < D.stats_tiles; tt += NC * 32) {
              const float* sp = D.stats_in + (size_t)tt * 8 * sk;
#pragma unroll
              for (int b = 0; b < kFusedMaxB; ++b)
#pragma unroll
                for (int j = 0; j < 3; ++j)
                  if (b < B && j < sk) acc[b][j] += __ldcg(sp + b * sk + j);
            }
#pragma unroll
            for (int b = 0; b < kFusedMaxB; ++b)
#pragma unroll
              for (int j = 0; j < 3; ++j)
                if (b < B && j < sk) {
                  const float v = warp_sum(acc[b][j]);
                  if (lane == 0) s_stw[warp][b * 3 + j] = v;
                }
          }
        };
        // (2) after a barrier: column sums in a fixed order (the same in every thread)
        auto col_sum = [&](int b, int j) {
          float sum = 0.f;
#pragma unroll
          for (int w = 0; w < NC; ++w) sum += s_stw[w][b * 3 + j];
          return sum;
        };
        auto col_rs = [&](int b) { return 1.f / sqrtf(col_sum(b, 0) / (float)a.d + a.eps); };
        // (3) thread 0: RMSNorm scales and the exit decision of layer dec_layer
        // (batch minimum of the cosine between the residual entering and leaving it)
        auto stats_decide = [&]() {
          for (int b = 0; b < B; ++b) s_rs[b] = col_rs(b);
          if (D.dec_layer > 0 && sk == 3) {
            float m = FLT_MAX;
            for (int b = 0; b < B; ++b)
              m = fminf(m, col_sum(b, 1) / fmaxf(sqrtf(col_sum(b, 2)) * sqrtf(col_sum(b, 0)), 1e-12f));
            int e = s_e;
            if (a.mode == RL_EXIT_TAU && e == a.L && D.dec_layer < a.L && m > a.tau) e = D.dec_layer;
            s_e = e;
            if (cta == 0) {
              if (a.min_cos_out) a.min_cos_out[D.dec_layer - 1] = m;
              a.st->exit_layer = e;
            }
            __threadfence_block();
            s_dec = D.dec_layer;
          }
          tl2_mark(a.tl2, grid, p, cta, TL2_RED);
        };
        bool stats_pending = scaled;
        if (D.xmode == X_EMBED) {
          named_sync(kBarCons, NC * 32);
          if (ct == 0) {  // step begin
            if (a.mode == RL_EXIT_FORCED && cta == 0) {
              const int raw = a.schedule[a.st->step % a.schedule_len];
              if (raw < 0 || raw > a.L) atomicOr(&a.st->err, RL_DEVERR_SCHEDULE);
            }
            if (cta == 0) a.st->exit_layer = s_e;
            for (int b = 0; b < B; ++b) s_rs[b] = 1.f / sqrtf(s_col[b][0] / (float)a.d + a.eps);
          }
          named_sync(kBarCons, NC * 32);
        } else if (scaled && (!regs || (a.mode == RL_EXIT_TAU && s_e == a.L && D.dec_layer > 0 && D.dec_layer < a.L && sk == 3))) {
          stats_partials();
          named_sync(kBarCons, NC * 32);
          if (ct == 0) stats_decide();
          named_sync(kBarCons, NC * 32);
          stats_pending = false;
        }
        const bool w4 = D.qwt && D.layer_no > 0 && D.layer_no > s_e;
        const int ntiles = D.N >> 4, UPT = (Kp + KU - 1) / KU;
        const int nt = cta < ntiles ? (ntiles - cta + grid - 1) / grid : 0;  // this CTA's tiles
        // flush batches: TB tiles of per-warp partials in shared memory; an
        // epilogue round covers R outputs (a multiple of 16 B, so a thread keeps
        // its column c in every round and 16 consecutive lanes hold one tile column)
        const int TB = max(1, 16 / B);
        const int R = ((NC * 32) / (16 * B)) * 16 * B;
        const int my_c = (ct >> 4) % B, my_r = ct & 15;
        // residual epilogues: this thread's inputs of the first round, fetched now
        float pre_res = 0.f, pre_hin = 0.f, pre_gn = 0.f;
        float2 pre_cs = make_float2(1.f, 0.f);  // QKV: (cos, sin) of this thread's first-round RoPE pair
        if (D.epi == EPI_QKV_ROPE && my_r < 8 && ct < R && ct < min(TB, nt) * 16 * B) {
          const int row0 = (cta + (ct / (16 * B)) * grid) * 16;
          const int pos = s_pos;
          if (row0 / a.hd < a.Hq + a.Hkv && pos >= 0 && pos < a.Tmax)
            pre_cs = __ldg(a.rope_cs + (size_t)pos * (a.hd >> 1) + 8 * ((row0 % a.hd) >> 4) + my_r);
        }
        if (D.epi == EPI_RESID && ct < R && ct < min(TB, nt) * 16 * B) {
          const int n = (cta + (ct / (16 * B)) * grid) * 16 + my_r;
          pre_res = __ldcg(D.resid + (size_t)my_c * D.ldr + n);
          if (D.h_in) pre_hin = __ldcg(D.h_in + (size_t)my_c * a.d + n);
          if (D.gnext) pre_gn = D.gnext[n];
        }
        if (D.xmode != X_EMBED) {
          if (!mbar_wait(&xbar, xpar, kSpin)) {
            if (lane == 0) atomicOr(&a.st->err, RL_DEVERR_TIMEOUT);
            s_abort = 1;
          }
          xpar ^= 1u;
        }
        if (ct == 0) tl2_mark(a.tl2, grid, p, cta, TL2_X);
        if (w4) {
          // The W4 MMAs run in fp16.  Each 128-input group of every activation
          // row is scaled by its own power of two 2^k (largest |x| of the group
          // just below 2^15: exact, and bf16 values in the fp16 normal range
          // convert exactly), converted to fp16 in place and reordered per
          // 8-input chunk as (x0,x4), (x2,x6), (x1,x5), (x3,x7) to match the
          // nibble fields the MMA reads; xsum[b][group] = (sum of the group's
          // inputs, 2^-k).  The 16 chunks of a group sit in 16 consecutive
          // lanes: group max and sum take four shuffles each, no block barrier.
          const int nchk = Kp >> 3;
          float2* xs2 = reinterpret_cast<float2*>(xsum);
          for (int c0 = 0; c0 < nchk; c0 += NC * 32) {
            const int ch = c0 + ct;
            const bool on = ch < nchk;  // nchk is a multiple of 16: groups are all on or all off
            for (int b = 0; b < B; ++b) {
              uint4* cp = reinterpret_cast<uint4*>(xs + (size_t)b * RSX + (on ? ch : 0) * 16);
              float f[8];
              float mx = 0.f;
              if (on) {
                const uint4 v = *cp;
                const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
                for (int i = 0; i < 4; ++i) {
                  const float2 ff = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&w[i]));
                  f[2 * i] = ff.x;
                  f[2 * i + 1] = ff.y;
                  mx = fmaxf(mx, fmaxf(fabsf(ff.x), fabsf(ff.y)));
                }
              }
#pragma unroll
              for (int o = 1; o < 16; o <<= 1) mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, o));
              int e = 0;
              if (mx > 0.f) frexpf(mx, &e);  // mx < 2^e
              const int k = min(max(15 - e, -120), 120);
              const float sc = ldexpf(1.f, k);
              float sum = 0.f;
              if (on) {
#pragma unroll
                for (int i = 0; i < 8; ++i) f[i] *= sc;
                sum = ((f[0] + f[1]) + (f[2] + f[3])) + ((f[4] + f[5]) + (f[6] + f[7]));
                const __half2 p0 = __floats2half2_rn(f[0], f[4]), p1 = __floats2half2_rn(f[2], f[6]);
                const __half2 p2 = __floats2half2_rn(f[1], f[5]), p3 = __floats2half2_rn(f[3], f[7]);
                *cp = make_uint4(*reinterpret_cast<const uint32_t*>(&p0), *reinterpret_cast<const uint32_t*>(&p1),
                                 *reinterpret_cast<const uint32_t*>(&p2), *reinterpret_cast<const uint32_t*>(&p3));
              }
#pragma unroll
              for (int o = 1; o < 16; o <<= 1) sum += __shfl_xor_sync(0xffffffffu, sum, o);
              const float inv = ldexpf(1.f, -k);
              if (on && (ct & 15) == 0) xs2[b * G + (ch >> 4)] = make_float2(sum * inv, inv);
            }
          }
          fence_proxy_async_smem();  // a later phase's bulk copy rewrites these bytes
          named_sync(kBarCons, NC * 32);
        }
        // MMA column g reads activation row min(g, B-1); columns >= B are dropped
        const unsigned char* xrow = xs + (size_t)(g < B ? g : B - 1) * RSX;
        bool first_w = true;

        // epilogue of a batch of nb tiles starting at tile t_first (all consumer threads)
        auto flush = [&](int nb, int t_first, bool first_batch) {
          // deferred statistics: warp partials, then (after the batch barrier)
          // every epilogue thread sums its own column's scale; thread 0 decides
          const bool fresh = stats_pending;
          if (fresh) stats_partials();
          named_sync(kBarCons, NC * 32);
          if (fresh) {
            stats_pending = false;
            if (ct == 0) stats_decide();
          }
          const float rsv = scaled ? col_rs(my_c) : s_rs[my_c];
          const int nout = nb * 16 * B;
          const int rounds = (nout + R - 1) / R;
          for (int rd = 0; rd < rounds; ++rd) {
            const int i = rd * R + ct;
            const bool act = ct < R && i < nout;
            const int tb = act ? i / (16 * B) : 0;
            const int tl = t_first + tb * grid;
            float v = 0.f;
            if (act) {
#pragma unroll
              for (int w = 0; w < NC; ++w) v += redf[((tb * NC + w) * B + my_c) * 16 + my_r];
            }
            if (D.epi == EPI_RESID) {
              float s0 = 0.f, s1 = 0.f, s2 = 0.f;
              if (act) {
                const int n = tl * 16 + my_r;
                float res = pre_res, hin = pre_hin, gn = pre_gn;
                if (!(first_batch && rd == 0)) {
                  res = __ldcg(D.resid + (size_t)my_c * D.ldr + n);
                  hin = D.h_in ? __ldcg(D.h_in + (size_t)my_c * a.d + n) : 0.f;
                  gn = D.gnext ? D.gnext[n] : 0.f;
                }
                const float val = v + res;
                D.out[(size_t)my_c * D.ldo + n] = val;
                if (D.trace) D.trace[((size_t)D.trace_layer * a.trace_maxB + my_c) * D.ldo + n] = val;
                if (D.xnext) D.xnext[(size_t)my_c * D.ldxnext + n] = __float2bfloat16_rn(val * gn);
                s0 = val * val;
                s1 = val * hin;
                s2 = hin * hin;
              }
              if (D.stats_out) {
#pragma unroll
                for (int o = 1; o < 16; o <<= 1) {
                  s0 += __shfl_xor_sync(0xffffffffu, s0, o);
                  s1 += __shfl_xor_sync(0xffffffffu, s1, o);
                  s2 += __shfl_xor_sync(0xffffffffu, s2, o);
                }
                if (act && my_r == 0) {
                  float* so = D.stats_out + ((size_t)tl * 8 + my_c) * D.stats_k_out;
                  so[0] = s0;
                  if (D.stats_k_out == 3) {
                    so[1] = s1;
                    so[2] = s2;
                  }
                }
              }
            } else if (D.epi == EPI_SWIGLU) {
              // rows r < 8 of a tile are gate rows, r + 8 the matching up rows
              const float up = __shfl_down_sync(0xffffffffu, v, 8);
              if (act && my_r < 8) {
                const float rs = rsv;
                D.out_h[(size_t)my_c * D.ldoh + tl * 8 + my_r] = __float2bfloat16_rn(silu_f(v * rs) * (up * rs));
              }
            } else if (D.epi == EPI_QKV_ROPE) {
              // rows r and r + 8 of a tile are one RoPE pair (dims dim, dim + hd/2)
              const float hv = __shfl_down_sync(0xffffffffu, v, 8);
              if (act && my_r < 8) {
                const int hd = a.hd, half = hd >> 1;
                const int row0 = tl * 16;
                const int head_all = row0 / hd;
                const float rs = rsv;
                const int pos = s_pos;
                const int dim = 8 * ((row0 % hd) >> 4) + my_r;
                float lo = v * rs, hi = hv * rs;
                if (head_all < a.Hq + a.Hkv) {
                  float sn, cs;
                  if (first_batch && rd == 0 && pos >= 0 && pos < a.Tmax) {
                    cs = pre_cs.x;
                    sn = pre_cs.y;
                  } else {
                    sincosf((float)pos * s_freq[dim], &sn, &cs);
                  }
                  const float nlo = lo * cs - hi * sn, nhi = hi * cs + lo * sn;
                  lo = nlo;
                  hi = nhi;
                }
                if (head_all < a.Hq) {
                  float* q = D.q_out + (size_t)my_c * a.Hq * hd + head_all * hd;
                  q[dim] = lo;
                  q[dim + half] = hi;
                } else if (pos >= 0 && pos < a.Tmax) {
                  const bool is_k = head_all < a.Hq + a.Hkv;
                  const int hk = is_k ? head_all - a.Hq : head_all - a.Hq - a.Hkv;
                  bf16* dst = (is_k ? D.kc : D.vc) + (((size_t)my_c * a.Hkv + hk) * a.Tmax + pos) * hd;
                  dst[dim] = __float2bfloat16_rn(lo);
                  dst[dim + half] = __float2bfloat16_rn(hi);
                } else if (my_r == 0 && my_c == 0) {
                  atomicOr(&a.st->err, RL_DEVERR_CAPACITY);
                }
              }
            } else if (D.epi == EPI_LMHEAD) {
              if (act) {
                const int n = tl * 16 + my_r;
                const float val = v * rsv;
                D.out[(size_t)my_c * D.ldo + n] = val;
                if (val > amv || (val == amv && n < ami)) {
                  amv = val;
                  ami = n;
                }
              }
            } else {  // EPI_STORE
              if (act) D.out[(size_t)my_c * D.ldo + tl * 16 + my_r] = v * rsv;
            }
          }
          named_sync(kBarCons, NC * 32);
        };

        int nb = 0, t_first = cta;
        bool first_batch = true;
        for (int tl = cta; tl < ntiles; tl += grid) {
          // the ring slot of the next unit(s), waited for
          auto take = [&](bool& ok) -> const unsigned char* {
            const int slot = rc.slot;
            ok = s_abort == 0 && mbar_wait(&full[slot], (uint32_t)(rc.round & 1), kSpin);
            if (!ok && s_abort == 0) {
              if (lane == 0) atomicOr(&a.st->err, RL_DEVERR_TIMEOUT);
              s_abort = 1;
            }
            if (first_w && ct == 0) tl2_mark(a.tl2, grid, p, cta, TL2_W);
            first_w = false;
            return ring + (size_t)slot * SLOT_B;
          };
          auto release = [&]() {
            __syncwarp();
            if (lane == 0) mbar_arrive(&empty[rc.slot]);
            rc.next(NS);
          };
          float v0, v1, v2, v3;
          if (w4) {
            // W4 units, two at a time: independent MMA chains interleave
            float y[2][4];
#pragma unroll
            for (int j = 0; j < 2; ++j)
#pragma unroll
              for (int i = 0; i < 4; ++i) y[j][i] = 0.f;
            for (int uk = 0; uk < UPT; uk += W4U) {
              bool ok;
              const unsigned char* sb = take(ok);
              const int ns = min(W4U, UPT - uk);
              for (int s = 0; s < ns; s += 2) {
                const int ga = (uk + s) * 8 + warp, gb = ga + 8;
                const bool on_a = ok && ga < G, on_b = ok && s + 1 < ns && gb < G;
                if (on_b) {
                  w4_unit(sb + (size_t)s * STAGE_W, ga, xrow, xsum, B, G, warp, g, t, y[0]);
                  w4_unit(sb + (size_t)(s + 1) * STAGE_W, gb, xrow, xsum, B, G, warp, g, t, y[1]);
                } else if (on_a) {
                  w4_unit(sb + (size_t)s * STAGE_W, ga, xrow, xsum, B, G, warp, g, t, y[0]);
                }
              }
              release();
            }
            v0 = y[0][0] + y[1][0];
            v1 = y[0][1] + y[1][1];
            v2 = y[0][2] + y[1][2];
            v3 = y[0][3] + y[1][3];
          } else {
            float y[2][4];
#pragma unroll
            for (int j = 0; j < 2; ++j)
#pragma unroll
              for (int i = 0; i < 4; ++i) y[j][i] = 0.f;
            for (int uk = 0; uk < UPT; ++uk) {
              bool ok;
              const unsigned char* sb = take(ok);
              // bf16 unit: 16 rows of kn inputs; 16-byte chunk c of row r at
              // c ^ 4 (r & 1): the 8 lanes of a quarter warp (rows 2q, 2q+1,
              // chunks c0..c0+3) hit 8 different 16-byte bank groups
              const int gi = uk * 8 + warp;  // this warp's 128 inputs of the unit
              if (ok && gi < G) {
                const int k0 = uk * KU, kn = min(KU, Kp - k0), RS = kn * 2;
                const int sw = (g & 1) << 2;
#pragma unroll
                for (int i4 = 0; i4 < 4; ++i4) {
                  const int cb = warp * 16 + 4 * i4 + t;
                  const uint4 wa = *reinterpret_cast<const uint4*>(sb + g * RS + ((cb ^ sw) << 4));
                  const uint4 wb = *reinterpret_cast<const uint4*>(sb + (g + 8) * RS + ((cb ^ sw) << 4));
                  const uint4 X = *reinterpret_cast<const uint4*>(xrow + (k0 + cb * 8) * 2);
#pragma unroll
                  for (int e = 0; e < 2; ++e)
                    mma_bf16(y[i4 & 1], u4get(wa, 2 * e), u4get(wb, 2 * e), u4get(wa, 2 * e + 1),
                             u4get(wb, 2 * e + 1), u4get(X, 2 * e), u4get(X, 2 * e + 1));
                }
              }
              release();
            }
            v0 = y[0][0] + y[1][0];
            v1 = y[0][1] + y[1][1];
            v2 = y[0][2] + y[1][2];
            v3 = y[0][3] + y[1][3];
          }
          // this warp's partial tile -> the batch buffer ([tile][warp][column][row])
          {
            float* rw = redf + (size_t)(nb * NC + warp) * B * 16;
            if (2 * t < B) {
              rw[(2 * t) * 16 + g] = v0;
              rw[(2 * t) * 16 + g + 8] = v2;
            }
            if (2 * t + 1 < B) {
              rw[(2 * t + 1) * 16 + g] = v1;
              rw[(2 * t + 1) * 16 + g + 8] = v3;
            }
          }
          if (++nb == TB || tl + grid >= ntiles) {
            flush(nb, t_first, first_batch);
            first_batch = false;
            t_first = tl + grid;
            nb = 0;
          }
        }
        if (stats_pending) {  // a CTA without tiles still takes the decision
          stats_partials();
          named_sync(kBarCons, NC * 32);
          if (ct == 0) stats_decide();
        }
        if (D.epi == EPI_LMHEAD) {
          // this CTA's argmax per column: 16-lane groups, then one thread per column
#pragma unroll
          for (int o = 1; o < 16; o <<= 1) {
            const float ov = __shfl_xor_sync(0xffffffffu, amv, o);
            const int oi = __shfl_xor_sync(0xffffffffu, ami, o);
            if (ov > amv || (ov == amv && oi < ami)) {
              amv = ov;
              ami = oi;
            }
          }
          float* sv = s_mrg;
          int* si = reinterpret_cast<int*>(s_mrg + 2 * NC);
          if (my_r == 0) {
            sv[ct >> 4] = ct < R ? amv : -FLT_MAX;
            si[ct >> 4] = ct < R ? ami : 0x7fffffff;
          }
          named_sync(kBarCons, NC * 32);
          if (ct < B) {
            float bv = -FLT_MAX;
            int bi = 0x7fffffff;
            for (int h = 0; h < 2 * NC; ++h)
              if (h % B == ct && (sv[h] > bv || (sv[h] == bv && si[h] < bi))) {
                bv = sv[h];
                bi = si[h];
              }
            a.am_val[(size_t)cta * 8 + ct] = bv;
            a.am_idx[(size_t)cta * 8 + ct] = bi;
          }
        }
      } else if (D.kind == PH_ATTN) {
        // ---- attention over this CTA's chunks: partial (max, sum, o) per chunk ----
        const int pos = s_pos, hd = a.hd, Hkv = a.Hkv, Hq = a.Hq, rep = Hq / Hkv;
        const int ctx = min(pos + 1, a.Tmax);
        const int nch = step_attn_chunks(ctx, B, Hkv, hd, grid, a.part_cap);
        const int clen = (ctx + nch - 1) / nch;
        const int nitems = B * Hkv * nch;
        const bool two = hd * 2 * kCHP > kAttnHalf;
        const float scale = rsqrtf((float)hd);
        const int WS = 2 + hd;
        if (clen > kCHP && cta == 0 && ct == 0) atomicOr(&a.st->err, RL_DEVERR_CAPACITY);
        auto run = [&](auto rep_c, auto dpl_c) {
          constexpr int REP = decltype(rep_c)::value, DPL = decltype(dpl_c)::value, HDC = 32 * DPL;
          // q of an item, scaled by 1/sqrt(hd), staged in the (idle) activation
          // buffer: loaded before the chunk is waited for
          float* qs = reinterpret_cast<float*>(xs);
          auto load_q = [&](int it) {
            const int b = it / (Hkv * nch), hk = (it % (Hkv * nch)) / nch;
            const float4* qg = reinterpret_cast<const float4*>(D.q_out + (size_t)b * Hq * HDC + (size_t)hk * REP * HDC);
            for (int i = ct; i < REP * HDC / 4; i += NC * 32) {
              float4 v = __ldcg(qg + i);
              v.x *= scale;
              v.y *= scale;
              v.z *= scale;
              v.w *= scale;
              reinterpret_cast<float4*>(qs)[i] = v;
            }
          };
          const int per = kMulti ? (nitems + grid - 1) / grid : 1;  // the producer's order
          const int it0 = kMulti ? cta * per : cta, it_end = kMulti ? min(nitems, cta * per + per) : nitems;
          // two chunks per CTA, of one head group (an even chunk count): the
          // first one's partial is kept in shared memory and folded into the
          // second, so a head group has nch / 2 partials to merge
          const bool pair = kMulti && per == 2 && (nch & 1) == 0;
          const int npart = pair ? nch / 2 : nch;
          for (int it = it0; it < it_end; it += kMulti ? 1 : grid) {
            const bool first = pair && it == it0;
            load_q(it);
            const int b = it / (Hkv * nch), rr = it % (Hkv * nch), hk = rr / nch, ch = rr % nch;
            const int start = ch * clen, end = min(start + clen, ctx);
            const int n = min(kCHP, max(0, end - start));
            // the row written by this step's QKV phase: loads issued before the wait
            const size_t head_base = ((size_t)b * Hkv + hk) * a.Tmax;
            const bool has_new = pos >= start && pos < start + n && ct < HDC / 8;
            uint4 kv_new = make_uint4(0u, 0u, 0u, 0u), vv_new = kv_new;
            if (has_new) {
              kv_new = __ldcg(reinterpret_cast<const uint4*>(D.kc + (head_base + pos) * HDC) + ct);
              vv_new = __ldcg(reinterpret_cast<const uint4*>(D.vc + (head_base + pos) * HDC) + ct);
            }
            const int slot = rc.slot;
            bool ok = s_abort == 0 && mbar_wait(&full[slot], (uint32_t)(rc.round & 1), kSpin);
            rc.next(NS);
            int slot_v = slot;
            if (two) {
              slot_v = rc.slot;
              ok = ok && mbar_wait(&full[slot_v], (uint32_t)(rc.round & 1), kSpin);
              rc.next(NS);
            }
            if (!ok && s_abort == 0) {
              if (lane == 0) atomicOr(&a.st->err, RL_DEVERR_TIMEOUT);
              s_abort = 1;
            }
            if (it == it0 && ct == 0) tl2_mark(a.tl2, grid, p, cta, TL2_X);
            unsigned char* Ks = ring + (size_t)slot * SLOT_B;
            unsigned char* Vs = two ? ring + (size_t)slot_v * SLOT_B : Ks + kAttnHalf;
            if (ok && has_new) {  // 16-byte chunk ct of the row, into its swizzled place
              const int rw = pos - start;
              *reinterpret_cast<uint4*>(Ks + kv_off(rw, ct)) = kv_new;
              *reinterpret_cast<uint4*>(Vs + kv_off(rw, ct)) = vv_new;
              fence_proxy_async_smem();  // the slot is refilled by bulk copies later
            }
            named_sync(kBarCons, NC * 32);
            // per-warp scores, softmax and P V on the tensor cores, 16 positions
            // per warp; the warps' partials overlay the K rows
            float* wb = reinterpret_cast<float*>(Ks);
            const int nn = ok ? n : 0;
            const int j0 = warp * 16, jn = max(0, min(16, nn - j0));
            attn_warp_tc<REP, HDC>(Ks, Vs, j0, jn, qs, lane, wb + (size_t)warp * REP * WS);
            named_sync(kBarCons, NC * 32);
            // combine the eight warps (online-softmax rescale) into this chunk's
            // partial; partial rows of PS floats (o[hd], max, sum, 2 pad: 16-byte rows)
            constexpr int PS = HDC + 4;
            float* part = a.part + ((size_t)b * Hq + (size_t)hk * REP) * a.part_cap * PS;
            float* keep = redf;  // a pair's first partial: [3][REP * HDC] numerator, max, sum
            for (int i = ct; i < REP * HDC; i += NC * 32) {
              const int h = i / HDC, dd = i % HDC;
              float M = -FLT_MAX;
#pragma unroll
              for (int w = 0; w < NC; ++w) M = fmaxf(M, wb[(w * REP + h) * WS]);
              float num = 0.f, den = 0.f;
#pragma unroll
              for (int w = 0; w < NC; ++w) {
                const float* ww = wb + (w * REP + h) * WS;
                const float f = ww[1] > 0.f ? __expf(ww[0] - M) : 0.f;
                num += f * ww[2 + dd];
                den += f * ww[1];
              }
              if (first) {
                keep[i] = num;
                keep[REP * HDC + i] = M;
                keep[2 * REP * HDC + i] = den;
                continue;
              }
              if (pair) {  // fold in the pair's first chunk (it precedes this one)
                const float n1 = keep[i], M1 = keep[REP * HDC + i], d1 = keep[2 * REP * HDC + i];
                if (d1 > 0.f) {
                  if (den > 0.f) {
                    const float Mn = fmaxf(M1, M);
                    const float a1 = __expf(M1 - Mn), a2 = __expf(M - Mn);
                    num = n1 * a1 + num * a2;
                    den = d1 * a1 + den * a2;
                    M = Mn;
                  } else {
                    num = n1;
                    den = d1;
                    M = M1;
                  }
                }
              }
              float* pp = part + ((size_t)h * a.part_cap + (pair ? ch >> 1 : ch)) * PS;
              pp[dd] = num;
              if (dd == 0) {
                pp[HDC] = den > 0.f ? M : -FLT_MAX;
                pp[HDC + 1] = den;
              }
            }
            fence_proxy_async_smem();  // the warps' partials overlay the slot, refilled by bulk copies
            named_sync(kBarCons, NC * 32);
            if (first) {  // no partial of its own: free the slots, go on to the second chunk
              if (lane == 0) {
                mbar_arrive(&empty[slot]);
                if (two) mbar_arrive(&empty[slot_v]);
              }
              continue;
            }
            // ---- the last CTA to finish a chunk of (b, hk) merges its chunks ----
            // (release: this CTA's partial writes, ordered by the barrier above,
            // before the ticket; acquire: every other chunk's partial after it)
            if (ct == 0) {
              const unsigned tk = atom_add_acq_rel(a.attn_ticket + b * Hkv + hk, 1u);
              s_merge = tk == (unsigned)(npart - 1);
            }
            named_sync(kBarCons, NC * 32);
            const bool merge = s_merge;
            // the partials are in global memory: this item's slot(s) are free
            if (lane == 0) {
              mbar_arrive(&empty[slot]);
              if (two) mbar_arrive(&empty[slot_v]);
            }
            if (merge) {
              // every thread merges its own outputs (head h, dim dd) from the
              // chunks' partials in L2, a round's loads all in flight at once:
              // no shared memory, no barrier
              const float* hp = a.part + ((size_t)b * Hq + (size_t)hk * REP) * a.part_cap * PS;
              constexpr int NOUT = (REP * HDC + NC * 32 - 1) / (NC * 32);
#pragma unroll
              for (int k = 0; k < NOUT; ++k) {
                const int i = ct + k * NC * 32;
                if (i < REP * HDC) {
                  const int h = i / HDC, dd = i % HDC;
                  const float* ph = hp + (size_t)h * a.part_cap * PS;
                  float M = -FLT_MAX, num = 0.f, den = 0.f;
                  for (int c0 = 0; c0 < npart; c0 += 8) {
                    float vm[8], vl[8], vo[8];
#pragma unroll
                    for (int j = 0; j < 8; ++j) {
                      const bool in = c0 + j < npart;
                      const float* pc = ph + (size_t)(c0 + j) * PS;
                      vm[j] = in ? __ldcg(pc + HDC) : -FLT_MAX;
                      vl[j] = in ? __ldcg(pc + HDC + 1) : 0.f;
                      vo[j] = in ? __ldcg(pc + dd) : 0.f;
                    }
                    // chunks in order, rescaled to the running maximum
                    float Mn = M;
#pragma unroll
                    for (int j = 0; j < 8; ++j)
                      if (vl[j] > 0.f) Mn = fmaxf(Mn, vm[j]);
                    const float al = __expf(M - Mn);
                    num *= al;
                    den *= al;
#pragma unroll
                    for (int j = 0; j < 8; ++j) {
                      const float f = vl[j] > 0.f ? __expf(vm[j] - Mn) : 0.f;
                      num += f * vo[j];
                      den += f * vl[j];
                    }
                    M = Mn;
                  }
                  D.o_out[(size_t)b * D.ldo_attn + (size_t)(hk * REP + h) * HDC + dd] =
                      __float2bfloat16_rn(den > 0.f ? num / den : 0.f);
                }
              }
              if (ct == 0) a.attn_ticket[b * Hkv + hk] = 0u;  // next step starts from zero
            }
          }
        };
        using I1 = std::integral_constant<int, 1>;
        using I2 = std::integral_constant<int, 2>;
        using I4 = std::integral_constant<int, 4>;
        switch (rep * 8 + (hd >> 5)) {
          case 1 * 8 + 2: run(I1{}, I2{}); break;
          case 2 * 8 + 2: run(I2{}, I2{}); break;
          case 4 * 8 + 2: run(I4{}, I2{}); break;
          case 1 * 8 + 4: run(I1{}, I4{}); break;
          case 2 * 8 + 4: run(I2{}, I4{}); break;
          default: run(I4{}, I4{}); break;
        }
      }
      // ---- end of phase: this CTA's writes are done; arrive ----
      if (ct == 0) tl2_mark(a.tl2, grid, p, cta, TL2_CDONE);
      named_sync(kBarCons, NC * 32);
      if (ct == 0) {
        tl_mark(a.tl, a.nph, p, 1);
        tl2_mark(a.tl2, grid, p, cta, TL2_ARRIVE);
        // the release orders every write of this CTA's phase (made before the
        // barrier above) before the arrival
        if (p + 1 < a.nph) st_release(a.bars + (size_t)cta * 32, (unsigned)(p + 1));
      }
    }
  }

  // ---- end of step: argmax over CTAs and the state update, by the last CTA ----
  __threadfence();
  __syncthreads();
  if (tid == 0) s_last = atomicAdd(a.cta_ticket, 1u) == (unsigned int)(grid - 1);
  __syncthreads();
  if (!s_last) return;
  __threadfence();
  if (warp < B) {
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
  for (int i = tid; i < grid; i += kThreads) a.bars[(size_t)i * 32] = 0u;
  for (int i = tid; i < a.nph; i += kThreads) a.tctr[i] = 0u;
  if (tid == 0) {
    DevState* st = a.st;
    if (a.exit_out) a.exit_out[0] = st->exit_layer;
    st->pos = st->pos + 1;
    st->step = st->step + 1;
    *a.cta_ticket = 0u;
  }
  __threadfence();
}

size_t step_smem_bytes(int B, int kmax, int gmax, int* nslot) {
  const size_t xs = (size_t)B * (kmax * 2 + 64);
  const size_t xsum = (((size_t)B * gmax * 8) + 15) & ~(size_t)15;
  const size_t red = (size_t)2 * NC * 32 * 16;
  const size_t budget = 227 * 1024 - kStaticSmem;
  const size_t fixed = xs + xsum + red + 1024;  // + alignment of the ring
  if (fixed >= budget) return 0;
  int ns = (int)((budget - fixed) / SLOT_B);
  if (ns > 6) ns = 6;
  if (ns < 3) return 0;
  if (nslot) *nslot = ns;
  return (size_t)ns * SLOT_B + fixed;
}

int decode_step_occupancy(size_t smem) {
  int n = 0;
  if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, k_decode_step<false, false>, kThreads, smem) !=
      cudaSuccess) {
    cudaGetLastError();
    return 0;
  }
  return n;
}

void decode_step_setup() {
  for (auto k : {k_decode_step<false, false>, k_decode_step<true, false>, k_decode_step<false, true>,
                 k_decode_step<true, true>}) {
    cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, 227 * 1024 - kStaticSmem);
    cudaFuncSetAttribute(k, cudaFuncAttributePreferredSharedMemoryCarveout, cudaSharedmemCarveoutMaxShared);
  }
}

cudaError_t launch_decode_step(const StepArgs& a, int grid, size_t smem, bool multi, bool wide, cudaStream_t s) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(grid);
  cfg.blockDim = dim3(kThreads);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeCooperative;  // all CTAs resident: they wait on one another
  attr[0].val.cooperative = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  if (wide)
    return multi ? cudaLaunchKernelEx(&cfg, k_decode_step<true, true>, a)
                 : cudaLaunchKernelEx(&cfg, k_decode_step<false, true>, a);
  return multi ? cudaLaunchKernelEx(&cfg, k_decode_step<true, false>, a)
               : cudaLaunchKernelEx(&cfg, k_decode_step<false, false>, a);
}

// ---------------------------------------------------------------------------
// bf16 weights [N][Kp] -> unit-tiled: for 16-row tile T and 1024-input unit u
// (kn = min(1024, Kp - 1024u) inputs), 16 rows of kn inputs stored
// contiguously at T*16*Kp + 16*1024*u elements, 16-byte chunk c of row r at
// chunk position c ^ (4 * (r & 1)): one bulk copy per unit, conflict-free reads.
// ---------------------------------------------------------------------------
__global__ void k_bf16_tile_layout(const bf16* __restrict__ w, int N, int Kp, bf16* __restrict__ out) {
  const int UPT = (Kp + KU - 1) / KU;
  const long long blk = blockIdx.x;
  const int tl = (int)(blk / UPT), uk = (int)(blk % UPT);
  const int k0 = uk * KU, kn = min(KU, Kp - k0), nch = kn / 8;
  unsigned char* dst = reinterpret_cast<unsigned char*>(out + (size_t)tl * 16 * Kp + (size_t)16 * k0);
  for (int idx = threadIdx.x; idx < 16 * nch; idx += blockDim.x) {
    const int r = idx / nch, c = idx % nch;
    const uint4 v = *reinterpret_cast<const uint4*>(w + (size_t)(tl * 16 + r) * Kp + k0 + c * 8);
    *reinterpret_cast<uint4*>(dst + (size_t)r * kn * 2 + ((c ^ ((r & 1) << 2)) * 16)) = v;
  }
}

void launch_bf16_tile_layout(const bf16* w, int N, int Kp, bf16* out, cudaStream_t s) {
  const long long blocks = (long long)(N / 16) * ((Kp + KU - 1) / KU);
  k_bf16_tile_layout<<<(unsigned)blocks, 256, 0, s>>>(w, N, Kp, out);
}

}  // namespace river

