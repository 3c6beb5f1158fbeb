// Tensor-core GEMM for the many-token passes (prefill, large decode
// batches): out[t][n] = sum_k W[n][k] x[t][k] with the backbone's bf16
// weights, on the 5th-generation tensor cores (tcgen05, accumulators in
// tensor memory), operands brought in by TMA.
//
// The projection is computed "swap-AB": the MMA's M side is 128 weight rows
// (output features), its N side is BN tokens, so one kernel serves a
// 32-token decode batch (BN = 32) and a 2048-token prompt (BN = 256) alike,
// and the epilogue reads one feature per TMEM lane, i.e. 32 consecutive
// features per warp, which makes every output store a coalesced row segment.
// The epilogues are the decode GEMV's (store, residual add, SwiGLU on the
// interleaved gate/up rows, RoPE + K/V append on the permuted QKV rows; the
// row orders put each rotate-half / gate-up pair 8 rows apart, so a pair sits
// in one warp and is exchanged with one shuffle).
//
// The weights of exit layers are W4 (River-LLM explainer, section 四: the
// device-side exit layer picks the path): eight more warps dequantise each
// 128 x 64 weight block, (q - z) * s rounded to bf16, straight into the
// 128-byte-swizzled shared-memory layout the TMA would have written, and the
// MMAs run as for the backbone's bf16 weights.  The packed words and the
// rows' (scale, zero) pairs of a block come from the W4 copy in this
// kernel's k-block layout (w4_tc_bytes), one bulk copy per block.  At decode
// batch sizes a W4 launch is bound by its chain of ring hand-offs and its
// per-unit epilogue rather than by its quarter-size weight bytes; up to 32
// tokens a narrow W4 projection (fewer output tiles than half the SMs) runs
// faster on the dequantising GEMV, which takes it (tc_gemm_runs_w4).
//
// When the output tiles are fewer than the SMs (a decode batch's narrow
// projections), K is split: unit u = (tile, split), each split accumulates
// its contiguous range of 64-input blocks and writes the fp32 tile to a
// workspace; the last of the tile's CTAs (ticket) sums the splits in split
// order and runs the epilogue, so the result does not depend on timing.
//
// Persistent CTAs (one per SM) walk the units; 512 threads in 16 warps:
// warps 0 and 15 issue the TMA loads (bf16: the 128 x 64 weight tiles and
// the BN x 64 token tiles of a STAGES-deep ring; W4: the token tiles and the
// W4 blocks, see kW4NA), warp 1 owns the tensor-memory allocation (two
// BN-column fp32 accumulators) and its lane 0 issues the MMAs; the epilogue
// warps (2..9 for bf16 layers, 2..5 for W4) run the epilogue of one tile
// while the MMAs of the next fill the other accumulator (warp w reads TMEM
// lanes 32 (w % 4) .. +31); for W4 layers warps 6..13 dequantise.  Every
// wait is bounded; a wait that runs out sets RL_DEVERR_TIMEOUT and the CTA
// winds down (all MMAs retired, all copies landed, tensor memory freed).
#include <algorithm>

#include <cuda.h>
#include <cudaTypedefs.h>

#include "dev_common.cuh"
#include "internal.h"

namespace river {

namespace {

using dev::smem_u32;

constexpr int kThreadsTc = 512;  // 16 warps: TMA, MMA, epilogue / W4 dequantising warps, TMA
constexpr int kBM = 128;           // weight rows per tile (MMA M)
constexpr int kBK = 64;            // K per stage: one 128-byte swizzle row of bf16
constexpr int kABytes = kBM * kBK * 2;
constexpr long long kSpinTc = 1ll << 20;

using dev::tma_load_2d;

__device__ __forceinline__ void tma_prefetch_map(const CUtensorMap* map) {
  asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(map)) : "memory");
}

// Shared-memory matrix descriptor of a K-major tile written by TMA with the
// 128-byte swizzle: rows of 128 bytes, 8-row (1024-byte) swizzle atoms
// stacked along M/N (stride byte offset 1024), the tile base 1024-aligned.
__device__ __forceinline__ uint64_t sw128_desc(uint32_t saddr) {
  uint64_t d = 0;
  d |= (uint64_t)((saddr & 0x3FFFFu) >> 4);        // start address
  d |= (uint64_t)1 << 16;                          // leading byte offset (unused here)
  d |= (uint64_t)(1024 >> 4) << 32;                // stride byte offset
  d |= (uint64_t)1 << 46;                          // descriptor version
  d |= (uint64_t)2 << 61;                          // 128-byte swizzle
  return d;
}

// Instruction descriptor, kind::f16: fp32 accumulate, bf16 A and B, both
// K-major, shape M x N.
__host__ __device__ constexpr uint32_t idesc_bf16(int M, int N) {
  return (1u << 4) | (1u << 7) | (1u << 10) | ((uint32_t)(N >> 3) << 17) |
         ((uint32_t)(M >> 4) << 24);
}

__device__ __forceinline__ void mma_tc(uint32_t tmem_d, uint64_t adesc, uint64_t bdesc,
                                       uint32_t idesc, uint32_t accum) {
  asm volatile(
      "{\n .reg .pred p;\n setp.ne.b32 p, %4, 0;\n"
      " tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n}\n" ::"r"(tmem_d),
      "l"(adesc), "l"(bdesc), "r"(idesc), "r"(accum)
      : "memory");
}

// Arrives on `bar` once every MMA this thread issued before has completed.
__device__ __forceinline__ void mma_commit(uint64_t* bar) {
  asm volatile(
      "tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(
          smem_u32(bar))
      : "memory");
}

__device__ __forceinline__ void tc_fence_before() {
  asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
}
__device__ __forceinline__ void tc_fence_after() {
  asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
}

// 32 lanes x 16 consecutive fp32 columns: thread i of the warp gets lane
// (taddr lane + i), columns taddr col .. +15.
__device__ __forceinline__ void tmem_ld16(uint32_t taddr, float (&v)[16]) {
  uint32_t r[16];
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x16.b32 "
      "{%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15}, [%16];"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]),
        "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]),
        "=r"(r[14]), "=r"(r[15])
      : "r"(taddr));
  asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
#pragma unroll
  for (int i = 0; i < 16; ++i) v[i] = __uint_as_float(r[i]);
}

// SiLU for the gate/up epilogue (fast reciprocal: the product is rounded to
// bf16 right after).
__device__ __forceinline__ float silu_fast(float v) { return __fdividef(v, 1.f + __expf(-v)); }

// Epilogue of one 16-column chunk: this thread's feature row R (< N when
// `row_ok`) for launch columns col0 .. col0 + 15 (those < B), read from the
// accumulator at `taddr`.  All 32 lanes of the warp call it together (the
// gate/up and rotate-half partners, 8 rows apart, are exchanged by shuffles).
// TM: the values come from the accumulator at `taddr`; otherwise from `vin`.
template <bool TM>
__device__ __forceinline__ void epi_chunk(const GemvArgs& a, int R, bool row_ok, int lane,
                                          int col0, uint32_t taddr, const float* vin = nullptr) {
  const int nc = min(16, a.B - col0);
  float v[16];
  auto fetch = [&]() {
    if constexpr (TM) {
      tmem_ld16(taddr, v);
    } else {
#pragma unroll
      for (int j = 0; j < 16; ++j) v[j] = vin[j];
    }
  };
  if (a.epi == EPI_RESID) {
    float r[16];  // residual loads issued before the accumulator read
#pragma unroll
    for (int j = 0; j < 16; ++j)
      r[j] = (row_ok && j < nc) ? __ldg(a.resid + (size_t)(col0 + j) * a.ldr + R) : 0.f;
    fetch();
    if (row_ok) {
#pragma unroll
      for (int j = 0; j < 16; ++j)
        if (j < nc) a.out[(size_t)(col0 + j) * a.ldo + R] = v[j] + r[j];
    }
    return;
  }
  fetch();
  if (a.epi == EPI_STORE) {
    if (row_ok) {
#pragma unroll
      for (int j = 0; j < 16; ++j)
        if (j < nc) a.out[(size_t)(col0 + j) * a.ldo + R] = v[j];
    }
    return;
  }
  float o[16];
#pragma unroll
  for (int j = 0; j < 16; ++j) o[j] = __shfl_xor_sync(0xffffffffu, v[j], 8);
  const bool low = (lane & 8) == 0;
  if (a.epi == EPI_SWIGLU) {
    if (row_ok && low) {
      bf16* dst = a.out_h + (R >> 4) * 8 + (R & 7);
#pragma unroll
      for (int j = 0; j < 16; ++j)
        if (j < nc) dst[(size_t)(col0 + j) * a.ldoh] = __float2bfloat16_rn(silu_fast(v[j]) * o[j]);
    }
    return;
  }
  // EPI_QKV_ROPE: row R of head R / hd holds dim 8 jt + (R % 8) (+ hd/2 in
  // the upper half of its 16-row tile), jt = (R % hd) / 16.
  if (!row_ok) return;
  const int hd = a.hd, half = hd / 2;
  const int head_all = R / hd;
  const int dim0 = 8 * ((R % hd) >> 4) + (R & 7);
  const int dim = low ? dim0 : dim0 + half;
  const bool rot = head_all < a.Hq + a.Hkv;
  const bool is_q = head_all < a.Hq;
  const bool is_k = !is_q && rot;
  const int hk = is_q ? 0 : (is_k ? head_all - a.Hq : head_all - a.Hq - a.Hkv);
  bf16* cache = is_k ? a.kc : a.vc;
  if (a.T_prefill <= 0) {
    // decode: every column is at the same position, so its (cos, sin) is
    // loaded once (not once per column behind the column's stores)
    const int pos = __ldg(a.pos_ptr);
    const bool in_cache = pos >= 0 && pos < a.Tmax;
    float sn = 0.f, cs = 1.f;
    if (rot) {
      if (a.rope_cs != nullptr && in_cache) {
        const float2 t = __ldg(a.rope_cs + (size_t)pos * half + dim0);
        cs = t.x;
        sn = t.y;
      } else {
        sincosf((float)pos * a.inv_freq[dim0], &sn, &cs);
      }
    }
#pragma unroll
    for (int j = 0; j < 16; ++j) {
      if (j >= nc) break;
      const int c = col0 + j;
      float x = v[j];
      if (rot) x = low ? x * cs - o[j] * sn : x * cs + o[j] * sn;
      if (is_q)
        a.q_out[(size_t)c * a.Hq * hd + head_all * hd + dim] = x;
      else if (!in_cache)
        atomicOr(a.err, RL_DEVERR_CAPACITY);
      else
        cache[(((size_t)c * a.Hkv + hk) * a.Tmax + pos) * hd + dim] = __float2bfloat16_rn(x);
    }
    return;
  }
  // prefill: every column is a token at its own position; the (cos, sin) of
  // the 16 columns are loaded first (independent loads, in flight together),
  // then the rotations and stores
  float2 csn[16];
#pragma unroll
  for (int j = 0; j < 16; ++j) {
    const int tok = a.col_base + col0 + j;
    const int pos = tok - (tok / a.T_prefill) * a.T_prefill;
    csn[j] = make_float2(1.f, 0.f);
    if (rot && j < nc && pos < a.Tmax) {
      if (a.rope_cs != nullptr) {
        csn[j] = __ldg(a.rope_cs + (size_t)pos * half + dim0);
      } else {
        float sn, cs;
        sincosf((float)pos * a.inv_freq[dim0], &sn, &cs);
        csn[j] = make_float2(cs, sn);
      }
    }
  }
#pragma unroll
  for (int j = 0; j < 16; ++j) {
    if (j >= nc) break;
    const int tok = a.col_base + col0 + j;
    const int seq = tok / a.T_prefill, pos = tok - seq * a.T_prefill;
    const bool in_cache = pos < a.Tmax;
    float x = v[j];
    if (rot) x = low ? x * csn[j].x - o[j] * csn[j].y : x * csn[j].x + o[j] * csn[j].y;
    if (is_q) {
      a.q_out[(size_t)tok * a.Hq * hd + head_all * hd + dim] = x;
    } else if (!in_cache) {
      atomicOr(a.err, RL_DEVERR_CAPACITY);
    } else {
      cache[(((size_t)seq * a.Hkv + hk) * a.Tmax + pos) * hd + dim] = __float2bfloat16_rn(x);
    }
  }
}

// Warp roles: 0 and 15 TMA producers, 1 MMA issuer; bf16 layers: warps
// 2 .. 9 run the epilogue; W4 layers: warps 2 .. 5 run the epilogue and warps
// 6 .. 13 dequantise, as two sets of four that take alternate k-blocks (a set
// covers the 128 rows of its k-block, one row per thread), so one set's waits
// and bookkeeping overlap the other's arithmetic.
constexpr int kEpiWarps = 8;   // bf16 layers
constexpr int kEpiWarpsW4 = 4;
constexpr int kDqWarps = 8;    // W4 layers: two sets of kDqSet
constexpr int kDqSet = 4;
constexpr int kDqWarp0 = 2 + kEpiWarpsW4;
constexpr int kQWBytes = 128 * 32;  // one W4 block's packed words: 128 rows x 8 words
constexpr int kW4Blk = kQWBytes + 512;  // + the rows' (scale, zero) pairs: one k-block of w4_tc
// W4 layers carve the same shared memory into three rings: NA dequantised
// weight tiles (made on chip), TS token tiles, and WS stages of packed words
// with their (scale, zero) pairs, one contiguous block of the w4_tc layout per
// k-block (one bulk copy; read from the row-major words, the same bytes came
// as 32-byte pieces of 128 rows and DRAM delivered them at a fraction of its
// bandwidth).  The packed words run WS k-blocks ahead of the token tiles.
// The MMAs of k-block g free its token tile and its dequantised tile at once:
// one commit per k-block to kdone[g % KD], KD = max(TS, NA) (a waiter never
// lags the MMAs by KD k-blocks, so the parity it waits for is unambiguous).
template <int BN>
constexpr int kW4NA = BN >= 256 ? 2 : (BN >= 128 ? 3 : 6);
template <int BN>
constexpr int kW4TS = BN >= 256 ? 3 : (BN >= 128 ? 4 : 8);
template <int BN>
constexpr int kW4WS = 12;
template <int BN>
constexpr int kW4KD = kW4TS<BN> > kW4NA<BN> ? kW4TS<BN> : kW4NA<BN>;
constexpr int kW4MaxNA = 6, kW4MaxWS = 12, kW4MaxKD = 8;
template <int BN>
constexpr int w4_smem_bytes() {
  return kW4NA<BN> * kABytes + kW4TS<BN> * BN * kBK * 2 + kW4WS<BN> * kW4Blk;
}
template <int BN>
constexpr bool w4_rings_ok() {
  return kW4NA<BN> <= kW4MaxNA && kW4WS<BN> <= kW4MaxWS && kW4KD<BN> <= kW4MaxKD && kW4TS<BN> <= 8 &&
         w4_smem_bytes<BN>() + 1024 <= 215 * 1024;
}
static_assert(w4_rings_ok<32>() && w4_rings_ok<64>() && w4_rings_ok<128>() && w4_rings_ok<256>(),
              "W4 rings must fit the shared memory");


// Persistent: CTA b takes tiles b, b + grid, ...; tile t covers weight rows
// (t / tiles_m) * 128 .. +127 and tokens (t % tiles_m) * BN .. +BN-1, so the
// CTAs running at one time share weight tiles in L2.  Two accumulators in
// tensor memory: the epilogue of tile i overlaps the MMAs of tile i + 1.
template <int BN, int STAGES>
__global__ void __launch_bounds__(kThreadsTc, 1)
    k_gemm_tc(const __grid_constant__ CUtensorMap tmW, const __grid_constant__ CUtensorMap tmX,
              const GemvArgs a) {
  pdl_wait();
  constexpr int kBBytes = BN * kBK * 2;
  constexpr uint32_t kTmemCols = 2 * BN;
  bool w4 = a.w4_mode == W4_ON;
  if (a.w4_mode == W4_BY_LAYER) w4 = a.layer_no > *a.exit_layer;
  if (w4 && (a.qtc == nullptr || !a.tc_w4)) return;  // the dequantising GEMV runs this W4 layer
  if (a.path_out != nullptr && blockIdx.x == 0 && threadIdx.x == 0) *a.path_out = w4 ? 1 : 0;

  extern __shared__ unsigned char smem_dyn[];
  unsigned char* smem =
      reinterpret_cast<unsigned char*>((reinterpret_cast<uintptr_t>(smem_dyn) + 1023) & ~(uintptr_t)1023);
  unsigned char* sA = smem;
  unsigned char* sB = smem + STAGES * kABytes;
  __shared__ __align__(8) uint64_t full[STAGES], empty[STAGES], afull[STAGES], acc_full[2], acc_empty[2],
      mma_done, kdone[kW4MaxKD], wfull[kW4MaxWS], wempty[kW4MaxWS];
  __shared__ uint32_t tmem_base;
  __shared__ volatile int s_fail;
  __shared__ volatile int s_last;

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int tiles_m = (a.B + BN - 1) / BN;
  const int ntiles = ((a.N + kBM - 1) / kBM) * tiles_m;
  const int nk = a.Kp / kBK;
  // work units: (tile t, split sp) = u = t * S + sp covers k-blocks kb0(u) .. kb1(u) - 1
  const int S = a.tc_ws != nullptr && a.ksplit > 1 ? a.ksplit : 1;
  const int nunits = ntiles * S;
  auto kb0_of = [&](int u) { return nk * (u % S) / S; };
  auto kb1_of = [&](int u) { return nk * (u % S + 1) / S; };
  // W4 rings (see kW4NA): dequantised tiles sA, token tiles sT, blocks of
  // packed words and (scale, zero) pairs sQW
  constexpr int NA = kW4NA<BN>, TS = kW4TS<BN>, WS = kW4WS<BN>, KD = kW4KD<BN>;
  unsigned char* sT = smem + NA * kABytes;
  unsigned char* sQW = sT + TS * kBBytes;
  // A CTA's k-blocks in order: unit u = blockIdx.x, blockIdx.x + grid, ...,
  // k-blocks kb0(u) .. kb1(u) - 1 of each.  The walk keeps the unit's weight
  // row n0, token m0 and k-block range, so a step costs no division (the
  // issuing threads' per-k-block work bounds a decode batch's GEMM).
  struct Walk {
    int u, kb, kbe, n0, m0;
  };
  auto walk_unit = [&](Walk& w) {
    const int t = w.u / S;
    w.n0 = (t / tiles_m) * kBM;
    w.m0 = (t % tiles_m) * BN;
    w.kb = kb0_of(w.u);
    w.kbe = kb1_of(w.u);
  };
  auto walk_first = [&]() {
    Walk w{(int)blockIdx.x, 0, 0, 0, 0};
    if (w.u < nunits) walk_unit(w);
    return w;
  };
  auto walk_next = [&](Walk& w) {
    if (++w.kb == w.kbe) {
      w.u += gridDim.x;
      if (w.u < nunits) walk_unit(w);
    }
  };
  int nkb = 0;  // k-blocks this CTA runs
  for (int u = blockIdx.x; u < nunits; u += gridDim.x) nkb += kb1_of(u) - kb0_of(u);

  if (threadIdx.x == 0) {
    for (int i = 0; i < STAGES; ++i) {
      dev::mbar_init(&full[i], w4 ? 1 : 2);  // bf16: the weight tile's and the token tile's producers
      dev::mbar_init(&empty[i], 1);
      dev::mbar_init(&afull[i], kDqSet);
    }
    for (int i = 0; i < kW4MaxKD; ++i) dev::mbar_init(&kdone[i], 1);
    for (int i = 0; i < kW4MaxWS; ++i) {
      dev::mbar_init(&wfull[i], 1);
      dev::mbar_init(&wempty[i], kDqSet);
    }
    for (int i = 0; i < 2; ++i) {
      dev::mbar_init(&acc_full[i], 1);
      dev::mbar_init(&acc_empty[i], w4 ? kEpiWarpsW4 : kEpiWarps);
    }
    dev::mbar_init(&mma_done, 1);
    s_fail = 0;
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    tma_prefetch_map(&tmW);
    tma_prefetch_map(&tmX);
  }
  if (warp == 1) {
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(
                     smem_u32(&tmem_base)),
                 "r"(kTmemCols)
                 : "memory");
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = tmem_base;

  if (warp == 0 || warp == kThreadsTc / 32 - 1) {
    // Two TMA producer warps.  bf16: warp 0 the weight tiles, the last warp
    // the token tiles, both into stage s of the STAGES ring (full[s] expects
    // both) once the MMAs of its previous round completed.  W4: warp 0 the
    // token tiles into the TS ring (freed by the MMAs), the last warp the
    // packed-word blocks into the WS ring (freed by the dequantising warps as
    // soon as they have read them), WS k-blocks ahead.  Each waits only for
    // consumers of inputs issued before, so they cannot stall each other.
    // (Issuing from several lanes of the warp, each k-block from lane
    // g mod 4, was measured: no faster at decode batches, and a 512-token
    // prompt's gate/up took 56 instead of 42 us.)
    const bool words = w4 && warp != 0;
    const int NSL = words ? WS : (w4 ? TS : STAGES);
    constexpr int NI = 1;
    if (lane < NI) {
      uint64_t* fb = words ? wfull : full;
      uint64_t* eb = words ? wempty : empty;
      Walk w = walk_first();
      for (int j = 0; j < lane && j < nkb; ++j) walk_next(w);
      int g = lane;
      for (; g < nkb; g += NI) {
        const int s = g % NSL, r = g / NSL;
        // the slot's previous k-block g - NSL must be done (W4 tokens: its MMAs, kdone)
        const bool free = r == 0 || (w4 && !words ? dev::mbar_wait(&kdone[(g - NSL) % KD], ((g - NSL) / KD) & 1, kSpinTc)
                                                  : dev::mbar_wait(&eb[s], (r - 1) & 1, kSpinTc));
        if (!free) {
          s_fail = 1;
          break;
        }
        if (words) {  // the block's packed W4 words and (scale, zero) pairs
          dev::mbar_expect_tx(&fb[s], kW4Blk);
          dev::bulk_g2s(sQW + s * kW4Blk, a.qtc + ((size_t)(w.n0 / kBM) * nk + w.kb) * kW4Blk, kW4Blk, &fb[s]);
        } else if (w4) {
          dev::mbar_expect_tx(&fb[s], kBBytes);
          tma_load_2d(sT + s * kBBytes, &tmX, w.kb * kBK, w.m0, &fb[s]);
        } else if (warp == 0) {
          dev::mbar_expect_tx(&fb[s], kABytes);
          tma_load_2d(sA + s * kABytes, &tmW, w.kb * kBK, w.n0, &fb[s]);
        } else {
          dev::mbar_expect_tx(&fb[s], kBBytes);
          tma_load_2d(sB + s * kBBytes, &tmX, w.kb * kBK, w.m0, &fb[s]);
        }
        for (int j = 0; j < NI; ++j) walk_next(w);
      }
      // the CTA may not exit with copies in flight: wait (bounded) for the
      // last ones this lane issued
      for (int g2 = g - NI; g2 >= 0 && g2 > g - NI - NSL; g2 -= NI)
        dev::mbar_wait(&fb[g2 % NSL], (g2 / NSL) & 1, kSpinTc);
    }
  } else if (warp == 1) {
    if (lane == 0) {  // MMA issuer
      const uint32_t idesc = idesc_bf16(kBM, BN);
      const int NSL = w4 ? TS : STAGES;
      int i = 0;
      int s = 0, sa = 0, kd = 0;  // token (bf16: whole) stage, W4 dequantised tile and kdone
      uint32_t par = 0, pa = 0;   // their phase parities
      bool ok = true;
      for (int uu = blockIdx.x; uu < nunits && ok; uu += gridDim.x, ++i) {
        const int acc = i & 1, u = i >> 1;
        if (u > 0 && !dev::mbar_wait(&acc_empty[acc], (u - 1) & 1, kSpinTc)) {
          s_fail = 1;
          break;
        }
        tc_fence_after();
        const uint32_t d = tmem + (uint32_t)(acc * BN);
        const int kbs = kb0_of(uu), kbe = kb1_of(uu);
        for (int kb = kbs; kb < kbe; ++kb) {
          // bf16: stage s of the one ring; W4: token tile s of TS, dequantised tile sa of NA
          if (!dev::mbar_wait(&full[s], par, kSpinTc) || (w4 && !dev::mbar_wait(&afull[sa], pa, kSpinTc))) {
            s_fail = 1;
            ok = false;
            break;
          }
          tc_fence_after();
          const uint64_t ad = sw128_desc(smem_u32(sA + (w4 ? sa : s) * kABytes));
          const uint64_t bd = sw128_desc(smem_u32((w4 ? sT : sB) + s * kBBytes));
#pragma unroll
          for (int k = 0; k < kBK / 16; ++k)  // 16 bf16 = 32 bytes = 2 in the address field
            mma_tc(d, ad + 2 * k, bd + 2 * k, idesc, (kb != kbs || k != 0) ? 1u : 0u);
          if (w4) {
            mma_commit(&kdone[kd]);  // frees its token tile and its dequantised tile
            if (++kd == KD) kd = 0;
            if (++sa == NA) {
              sa = 0;
              pa ^= 1u;
            }
          } else {
            mma_commit(&empty[s]);
          }
          if (++s == NSL) {
            s = 0;
            par ^= 1u;
          }
        }
        mma_commit(&acc_full[acc]);
      }
      // every MMA has completed before tensor memory is released
      mma_commit(&mma_done);
      dev::mbar_wait(&mma_done, 0, kSpinTc);
    }
  } else if (w4 && warp >= kDqWarp0 && warp < kDqWarp0 + kDqWarps) {
    // W4 dequantising warps: thread r writes weight row n0 + r of every 128 x 64
    // block, 8 chunks of 8 bf16 at chunk position c ^ (r & 7) (128-byte swizzle).
    // The producer TMA-loads each block's packed words (128 rows x 32 bytes)
    // WS blocks ahead; each thread copies its row's (scale, zero) WS - 1 blocks
    // ahead with cp.async.  A nibble q becomes the weight without an integer
    // conversion: placed at bits 10..13 of 0x46000000 it is the float
    // v = 8192 + q, and fma(v, s, c) with c = -(8192 + z) s rounded once gives
    // (q - z) s within s 2^-10 (8192 + z is exact: z is an fp16 in [0, 16)).
    {
      const int set = (warp - kDqWarp0) / kDqSet;
      const int r = threadIdx.x - (kDqWarp0 + set * kDqSet) * 32;
      // this set's k-blocks are g = set, set + 2, ...
      for (int g = set; g < nkb; g += 2) {
        const int sw = g % WS;
        const bool landed = dev::mbar_wait(&wfull[sw], (g / WS) & 1, kSpinTc);  // its words too
        const unsigned char* blk = sQW + sw * kW4Blk;
        const uint4 w0 = *reinterpret_cast<const uint4*>(blk + r * 32);
        const uint4 w1 = *reinterpret_cast<const uint4*>(blk + r * 32 + 16);
        const float2 zs = __half22float2(*reinterpret_cast<const __half2*>(blk + kQWBytes + r * 4));
        // every lane has read the stage: its words may be overwritten (a stage
        // whose copy did not land is never handed back)
        const bool all_landed = __all_sync(0xffffffffu, landed);
        if (all_landed && (threadIdx.x & 31) == 0) dev::mbar_arrive(&wempty[sw]);
        // dequantised tile sa was last read by the MMAs of k-block g - NA
        const int sa = g % NA;
        const bool got = all_landed && (g < NA || dev::mbar_wait(&kdone[(g - NA) % KD], ((g - NA) / KD) & 1, kSpinTc));
        if (!__all_sync(0xffffffffu, got)) {  // the same decision in every lane
          s_fail = 1;
          break;
        }
        unsigned char* dst = sA + sa * kABytes + r * 128;
        const uint32_t wv[8] = {w0.x, w0.y, w0.z, w0.w, w1.x, w1.y, w1.z, w1.w};
        const float sc = zs.x, c0 = -(8192.f + zs.y) * zs.x;
#pragma unroll
        for (int c = 0; c < 8; ++c) {  // chunk c: inputs 8c .. 8c + 7 = the nibbles of word c
          uint32_t pk[4];
#pragma unroll
          for (int e = 0; e < 4; ++e) {
            // nibble 2e sits at bits 8e, nibble 2e + 1 at 8e + 4: move each to bit 10
            const int sh0 = 8 * e - 10, sh1 = 8 * e - 6;
            const uint32_t b0 = sh0 < 0 ? wv[c] << -sh0 : wv[c] >> sh0;
            const uint32_t b1 = sh1 < 0 ? wv[c] << -sh1 : wv[c] >> sh1;
            const float v0 = __uint_as_float((b0 & 0x3C00u) | 0x46000000u);
            const float v1 = __uint_as_float((b1 & 0x3C00u) | 0x46000000u);
            const __nv_bfloat162 b2 = __floats2bfloat162_rn(fmaf(v0, sc, c0), fmaf(v1, sc, c0));
            pk[e] = *reinterpret_cast<const uint32_t*>(&b2);
          }
          *reinterpret_cast<uint4*>(dst + ((c ^ (r & 7)) << 4)) = make_uint4(pk[0], pk[1], pk[2], pk[3]);
        }
        dev::fence_proxy_async_smem();  // generic writes before the MMAs' reads
        __syncwarp();
        if ((threadIdx.x & 31) == 0) dev::mbar_arrive(&afull[sa]);
      }
    }
  } else if (warp >= 2 && warp < 2 + (w4 ? kEpiWarpsW4 : kEpiWarps)) {
    // epilogue warps: lane quarter warp % 4; bf16: column half (warp - 2) / 4,
    // W4 (four warps): every column
    const int q = warp & 3, h = (warp - 2) >> 2;
    const int nthr = (w4 ? kEpiWarpsW4 : kEpiWarps) * 32;
    const int c_lo = w4 ? 0 : h * (BN / 32), c_hi = w4 ? BN / 16 : (h + 1) * (BN / 32);
    int i = 0;
    for (int u = blockIdx.x; u < nunits; u += gridDim.x, ++i) {
      const int t = u / S;
      const int acc = i & 1, ua = i >> 1;
      const int n0 = (t / tiles_m) * kBM, m0 = (t % tiles_m) * BN;
      // (a wait limit below the default only shortens this wait: every wait
      // that keeps MMAs or copies from outliving the CTA keeps its own)
      const bool got = a.first_wait > 0 ? dev::mbar_poll(&acc_full[acc], ua & 1, a.first_wait)
                                        : dev::mbar_wait(&acc_full[acc], ua & 1, kSpinTc);
      if (!got) s_fail = 1;
      if (S > 1) {
        // every epilogue warp takes the same decision after the barrier (a wait
        // that ran out in one warp stops all of them)
        dev::named_sync(2, nthr);
        if (s_fail) break;
      } else if (!got) {
        break;
      }
      tc_fence_after();
      const int R = n0 + 32 * q + lane;
      const bool row_ok = R < a.N;
      const uint32_t tacc = tmem + ((uint32_t)(32 * q) << 16) + (uint32_t)(acc * BN);
      if (S == 1) {
#pragma unroll 1
        for (int c16 = c_lo; c16 < c_hi; ++c16) {
          const int col0 = m0 + c16 * 16;
          if (col0 >= a.B) break;
          epi_chunk<true>(a, R, row_ok, lane, col0, tacc + (uint32_t)(c16 * 16));
        }
        tc_fence_before();
        __syncwarp();
        if (lane == 0) dev::mbar_arrive(&acc_empty[acc]);
        continue;
      }
      // split K: this unit's fp32 partial tile -> ws[u][column][128 rows]
      float* wsu = a.tc_ws + (size_t)u * BN * kBM;
#pragma unroll 1
      for (int c16 = c_lo; c16 < c_hi; ++c16) {
        float v[16];
        tmem_ld16(tacc + (uint32_t)(c16 * 16), v);
#pragma unroll
        for (int j = 0; j < 16; ++j) wsu[(size_t)(c16 * 16 + j) * kBM + 32 * q + lane] = v[j];
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) dev::mbar_arrive(&acc_empty[acc]);
      // the last unit of tile t to finish sums the partials in split order and
      // runs the epilogue (release: the partial stores before the ticket,
      // ordered by the barrier; acquire: the other units' partials after it)
      dev::named_sync(2, nthr);
      if (warp == 2 && lane == 0) s_last = dev::atom_add_acq_rel(a.tc_ticket + t, 1u) == (unsigned)(S - 1);
      dev::named_sync(2, nthr);
      if (s_last) {
        const float* wst = a.tc_ws + (size_t)t * S * BN * kBM;
#pragma unroll 1
        for (int c16 = c_lo; c16 < c_hi; ++c16) {
          const int col0 = m0 + c16 * 16;
          if (col0 >= a.B) break;
          // the splits' partials summed in split order; the loads of four
          // splits are in flight at a time (one L2 round trip per four)
          float v[16];
#pragma unroll
          for (int j = 0; j < 16; ++j) v[j] = 0.f;
          for (int sp0 = 0; sp0 < S; sp0 += 4) {
            float t[4][16];
#pragma unroll
            for (int i = 0; i < 4; ++i) {
              const float* p = wst + ((size_t)(sp0 + i) * BN + c16 * 16) * kBM + 32 * q + lane;
#pragma unroll
              for (int j = 0; j < 16; ++j) t[i][j] = sp0 + i < S ? __ldcg(p + (size_t)j * kBM) : 0.f;
            }
#pragma unroll
            for (int i = 0; i < 4; ++i)
              if (sp0 + i < S) {
#pragma unroll
                for (int j = 0; j < 16; ++j) v[j] += t[i][j];
              }
          }
          epi_chunk<false>(a, R, row_ok, lane, col0, 0u, v);
        }
        dev::named_sync(2, nthr);
        if (warp == 2 && lane == 0) a.tc_ticket[t] = 0u;  // the next launch starts from zero
      }
      dev::named_sync(2, nthr);
    }
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem), "r"(kTmemCols)
                 : "memory");
  }
  if (threadIdx.x == 0 && s_fail && a.err != nullptr) atomicOr(a.err, RL_DEVERR_TIMEOUT);
}

template <int BN, int STAGES>
constexpr int tc_smem_bytes() {
  return (STAGES * (kABytes + BN * kBK * 2) > w4_smem_bytes<BN>() ? STAGES * (kABytes + BN * kBK * 2)
                                                                   : w4_smem_bytes<BN>()) +
         1024;
}

PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
  static PFN_cuTensorMapEncodeTiled_v12000 fn = [] {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) !=
            cudaSuccess ||
        q != cudaDriverEntryPointSuccess)
      p = nullptr;
    return reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
  }();
  return fn;
}

template <int BN, int STAGES>
cudaError_t set_smem_attr() {
  return cudaFuncSetAttribute(k_gemm_tc<BN, STAGES>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                              tc_smem_bytes<BN, STAGES>());
}

// K splits for a decode batch's projection (memory-bound: every unit streams
// its 128 weight rows x its share of K): the split count whose makespan,
// waves x (a unit's fixed cost + 1 / S of a whole tile's stream), is lowest.
// The fixed cost (pipeline fill, partial tile store and reduction; about
// 1.5 us) is taken relative to a tile's stream of 128 rows x K bf16 at about
// 45 GB/s per SM.  At least 4 k-blocks per split; partial tiles within the
// workspace; a split must gain 3 % over the next smaller one.
int tc_pick_split(int tiles, int nk, int sm_count, size_t tile_floats, size_t ws_floats) {
  const double fixed = 1.5e-6 * 45e9 / (128.0 * 64 * 2 * nk);
  auto cost = [&](int S) {
    const int waves = (tiles * S + sm_count - 1) / sm_count;
    return waves * (fixed + 1.0 / S);
  };
  int best = 1;
  double best_cost = cost(1);
  for (int S = 2; S <= 32 && S <= nk / 4; ++S) {
    if ((size_t)tiles * S * tile_floats > ws_floats) break;
    const double c = cost(S);
    if (c < 0.97 * best_cost) {
      best = S;
      best_cost = c;
    }
  }
  return best;
}

// K splits of a prompt's projection with a long reduction (at least 128
// k-blocks) whose 128-token tiles fill at most half the SMs: as many units
// per tile as the SMs hold, each at least 64 k-blocks (0: no split, the tile
// width by tc_pick_bn).  Measured on the 512-token prompt of the Llama-3.2-1B
// shape (bf16 layers): the down projection (K 8192, 64 tiles) from one
// 64-token-tile unit per SM to two 128-token-tile units per tile took the
// prompt from 3.30 to 3.15 ms; projections with K 2048 (32 k-blocks) only
// lost with a split.  A layer the device finds on the W4 path takes the same
// units.
int tc_prompt_split(const GemvArgs& a, int sm_count) {
  const int nk = a.Kp / kBK;
  if (a.B <= 64 || nk < 128 || a.tc_ws == nullptr) return 0;
  const int tiles = ((a.N + kBM - 1) / kBM) * ((a.B + 127) / 128);
  if (2 * tiles > sm_count || tiles > a.tc_ticket_n) return 0;
  const int S = std::min(sm_count / tiles, nk / 64);
  if (S < 2 || (size_t)tiles * S * 128 * kBM > a.tc_ws_floats) return 0;
  return S;
}

// split > 0: that many K splits (tc_prompt_split); else the decode batch's rule
template <int BN, int STAGES>
cudaError_t launch_tc(const CUtensorMap& tmW, const GemvArgs& a, int sm_count,
                      cudaStream_t s, int split = 0) {
  constexpr int smem = tc_smem_bytes<BN, STAGES>();
  CUtensorMap tmX;
  if (!make_tmap_bf16(&tmX, a.x, a.Kp, a.B, a.ldx, BN)) return cudaErrorInvalidValue;
  const int tiles = ((a.N + kBM - 1) / kBM) * ((a.B + BN - 1) / BN);
  GemvArgs b = a;
  b.ksplit = split > 0 ? split
             : BN <= 64 && a.tc_ws != nullptr && tiles <= a.tc_ticket_n
                 ? tc_pick_split(tiles, a.Kp / kBK, sm_count, (size_t)BN * kBM, a.tc_ws_floats)
                 : 1;
  const int S = b.ksplit;
  int grid = tiles * S;
  if (grid > sm_count) grid = sm_count;
  return launch_pdl(k_gemm_tc<BN, STAGES>, dim3(grid), dim3(kThreadsTc), (size_t)smem, s, tmW, tmX,
                    b);
}

__global__ void k_rope_table(const float* inv_freq, int half, int n, float2* out) {
  const int i = blockIdx.x * blockDim.x + threadIdx.x;
  if (i >= n) return;
  const int pos = i / half, dim = i - pos * half;
  float sn, cs;
  sincosf((float)pos * inv_freq[dim], &sn, &cs);
  out[i] = make_float2(cs, sn);
}

}  // namespace

void launch_rope_table(const float* inv_freq, int half, int Tmax, float2* out, cudaStream_t s) {
  const int n = half * Tmax;
  if (n > 0) k_rope_table<<<(n + 255) / 256, 256, 0, s>>>(inv_freq, half, n, out);
}

bool tc_gemm_available() { return encode_fn() != nullptr; }

// Shared-memory opt-in of every instantiation (once per process and device,
// before any launch or graph capture).
cudaError_t tc_gemm_init() {
  cudaError_t e = set_smem_attr<256, 4>();
  if (e == cudaSuccess) e = set_smem_attr<128, 6>();
  if (e == cudaSuccess) e = set_smem_attr<64, 8>();
  if (e == cudaSuccess) e = set_smem_attr<32, 8>();
  return e;
}

// 2-D bf16 tensor map over rows x inner (row stride ld elements), boxes of
// 64 inner elements (128 bytes, 128-byte swizzle) x box_rows rows; reads
// outside the tensor fill zeros.
bool make_tmap_bf16(CUtensorMap* map, const void* base, int inner, int rows, int ld, int box_rows) {
  PFN_cuTensorMapEncodeTiled_v12000 fn = encode_fn();
  if (fn == nullptr || base == nullptr || inner <= 0 || rows <= 0 || box_rows <= 0 || box_rows > 256)
    return false;
  if ((reinterpret_cast<uintptr_t>(base) & 15) != 0 || ((size_t)ld * 2) % 16 != 0 || inner % kBK != 0)
    return false;
  const cuuint64_t dims[2] = {(cuuint64_t)inner, (cuuint64_t)rows};
  const cuuint64_t strides[1] = {(cuuint64_t)ld * 2};
  const cuuint32_t box[2] = {(cuuint32_t)kBK, (cuuint32_t)box_rows};
  const cuuint32_t estr[2] = {1, 1};
  return fn(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(base), dims, strides, box,
            estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
            CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// W4 copy in the tensor-core GEMM's k-block layout: for 128-row tile T and
// 64-input k-block kb, one contiguous kW4Blk-byte block at (T * Kp/64 + kb):
// the 128 rows' 8 packed words (row r at 32 r), then each row's (scale, zero)
// pair of the block's group (kb / 2) at kQWBytes + 4 r.  Rows past N are zero.
size_t w4_tc_bytes(int N, int Kp) { return (size_t)((N + kBM - 1) / kBM) * (Kp / kBK) * kW4Blk; }

__global__ void k_w4_tc_layout(const uint32_t* __restrict__ qw, const __half2* __restrict__ sz, int N,
                               int Kp, unsigned char* __restrict__ out) {
  const int nk = Kp / kBK, G = Kp / 128;
  const long long blk = blockIdx.x;  // one CTA per (tile, k-block)
  const int T = (int)(blk / nk), kb = (int)(blk % nk);
  unsigned char* dst = out + blk * kW4Blk;
  for (int i = threadIdx.x; i < kBM * 8; i += blockDim.x) {
    const int r = i >> 3, wd = i & 7, R = T * kBM + r;
    reinterpret_cast<uint32_t*>(dst)[i] = R < N ? qw[(size_t)R * (Kp / 8) + kb * 8 + wd] : 0u;
  }
  for (int r = threadIdx.x; r < kBM; r += blockDim.x) {
    const int R = T * kBM + r;
    reinterpret_cast<__half2*>(dst + kQWBytes)[r] = R < N ? sz[(size_t)R * G + kb / 2] : __floats2half2_rn(0.f, 0.f);
  }
}

void launch_w4_tc_layout(const uint32_t* qw, const __half2* sz, int N, int Kp, void* out, cudaStream_t s) {
  const long long blocks = (long long)((N + kBM - 1) / kBM) * (Kp / kBK);
  if (blocks > 0)
    k_w4_tc_layout<<<(unsigned)blocks, 256, 0, s>>>(qw, sz, N, Kp, static_cast<unsigned char*>(out));
}

bool make_weight_tmap(CUtensorMap* map, const bf16* w, int N, int Kp) {
  return make_tmap_bf16(map, w, Kp, N, Kp, kBM);
}

// Token tile: the width whose estimated makespan (tiles per CTA x the tile's
// time, from the MMA efficiency measured per width on GB300) is smallest.
int tc_pick_bn(int N, int M, int sm_count) {
  // a decode batch: one token tile (split K fills the SMs), since an MMA of
  // 128 x 32 x 16 costs about as long as one of 128 x 64 x 16
  if (M <= 64) return M <= 32 ? 32 : 64;
  static const int widths[4] = {256, 128, 64, 32};
  static const float eff[4] = {1.0f, 0.65f, 0.35f, 0.2f};
  const int tn = (N + kBM - 1) / kBM;
  int best = 32;
  float best_cost = 1e30f;
  for (int i = 0; i < 4; ++i) {
    const int bn = widths[i];
    if (bn > 32 && bn / 2 >= M) continue;  // more than half the tile would be padding
    const int tiles = tn * ((M + bn - 1) / bn);
    const float cost = (float)((tiles + sm_count - 1) / sm_count) * bn / eff[i];
    if (cost < best_cost) {
      best_cost = cost;
      best = bn;
    }
  }
  return best;
}

bool tc_gemm_runs_w4(int N, int B, int sm_count) {
  if (B > kTcW4AllTokens) return true;
  const int bn = tc_pick_bn(N, B, sm_count);
  const int tiles = ((N + kBM - 1) / kBM) * ((B + bn - 1) / bn);
  return 2 * tiles >= sm_count;
}

cudaError_t launch_gemm_tc(const CUtensorMap& tmW, const GemvArgs& a, int sm_count,
                           cudaStream_t s) {
  if (a.B <= 0 || a.N <= 0) return cudaSuccess;
  const int split = tc_prompt_split(a, sm_count);
  if (split > 0) return launch_tc<128, 6>(tmW, a, sm_count, s, split);
  switch (tc_pick_bn(a.N, a.B, sm_count)) {
    case 256: return launch_tc<256, 4>(tmW, a, sm_count, s);
    case 128: return launch_tc<128, 6>(tmW, a, sm_count, s);
    case 64: return launch_tc<64, 8>(tmW, a, sm_count, s);
    default: return launch_tc<32, 8>(tmW, a, sm_count, s);
  }
}

}  // namespace river
