// Streaming decode attention for any batch (River-LLM explainer, section 三:
// every layer, backbone or exit river, reads the backbone's own K/V slots).
//
// One persistent CTA per SM walks the (sequence, KV head, chunk of <= 128
// positions) items.  A producer lane TMA-loads each chunk's K and V rows
// (64-row boxes, 16-row boxes for the tail, 64 dims at a time with the
// 128-byte swizzle, from tensor maps that cover every layer's cache) and the
// item's query rows into a ring of shared-memory slots, running ahead of the
// consumers.  The eight consumer warps form two groups of four that take
// alternate items, so one group's softmax, combine and stores overlap the
// other's loads and MMAs; a warp runs 32 positions of its group's chunk on
// the tensor cores (attn::attn_scores / attn_values: q K^T and P V as
// m16n8k16 MMAs) and releases the K rows (then the V rows) the moment it has
// read them.  The group combines its warps' online-softmax partials in its
// own shared-memory area and writes the chunk's (o, max, sum) partial;
// k_attn_combine then merges the chunks.  Every wait is bounded: a wait that
// runs out sets RL_DEVERR_TIMEOUT and the kernel winds down.
#include "attn_tc.cuh"
#include "dev_common.cuh"

namespace river {

namespace {

using namespace dev;
using namespace attn;

constexpr int kNCW = 8;                      // consumer warps
constexpr int kNG = 2;                       // consumer groups, one item each
constexpr int kGW = kNCW / kNG;              // warps per group
constexpr int kNB = 128 / (16 * kGW);        // 16-position blocks per warp
constexpr int kThreadsS = (kNCW + 1) * 32;   // + the producer warp
constexpr int kSlotS = 34816;                // 32 KB of K (+ V) rows + the query rows
constexpr int kQOff = 32768;                 // query rows inside a slot
constexpr int kMaxSlotsS = 6;
constexpr int kPartS = kNG * kGW * 4 * (2 + 128) * 4;  // the groups' partials (REP <= 4, hd <= 128)
constexpr long long kSpinS = 1LL << 22;

template <int REP, int HDC>
__global__ void __launch_bounds__(kThreadsS, 1) k_attn_stream(const __grid_constant__ AttnStreamArgs a) {
  pdl_wait();
  constexpr bool TWO = HDC == 128;  // K and V rows in separate slots
  constexpr int WS = 2 + HDC;
  constexpr int SPI = TWO ? 2 : 1;  // slots per item
  extern __shared__ __align__(128) unsigned char smem[];
  __shared__ __align__(8) uint64_t full[kMaxSlotsS], empty[kMaxSlotsS];
  __shared__ int s_pos;
  __shared__ volatile int s_abort;
  unsigned char* ring = smem + ((1024u - (smem_u32(smem) & 1023u)) & 1023u);
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int NS = a.nslot;
  if (tid == 0) {
    for (int i = 0; i < NS; ++i) {
      mbar_init(&full[i], 1);
      mbar_init(&empty[i], kGW);
    }
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    s_pos = *a.pos_ptr;
    s_abort = 0;
  }
  __syncthreads();
  const int pos = s_pos;
  const int ctx = min(pos + 1, a.Tmax);
  const int nch = a.nchunks;
  // chunk starts on 16-row boundaries (whole TMA boxes); clen <= 128 because
  // nch >= ceil(Tmax / 128)
  const int clen = (((ctx + nch - 1) / nch) + 15) & ~15;
  const int nitems = a.nq * a.Hkv * nch;
  const int grid = gridDim.x, cta = blockIdx.x;
  auto item_rows = [&](int it, int& b, int& hk, int& ch, int& start) {
    b = it / (a.Hkv * nch);
    const int rr = it % (a.Hkv * nch);
    hk = rr / nch;
    ch = rr % nch;
    start = ch * clen;
    return min(128, max(0, min(start + clen, ctx) - start));
  };

  // Group g owns slots g * NSG .. g * NSG + NSG - 1 and consumes the CTA's
  // items k = g, g + kNG, ...: its slot uses (SPI per item) fill its slots in
  // order, so a wait on a use always follows the wait on that slot's previous
  // use and the parity of the phase it waits for is never ambiguous.
  const int NSG = NS / kNG;

  if (warp == kNCW) {
    // ================================ producer ===================================
    if (lane == 0) {
      int issued[kNG] = {};
      auto take = [&](int g) -> int {
        const int u = issued[g], s = g * NSG + u % NSG, round = u / NSG;
        if (round > 0 && !mbar_wait(&empty[s], (uint32_t)((round - 1) & 1), kSpinS)) {
          atomicOr(a.err, RL_DEVERR_TIMEOUT);
          s_abort = 1;
          return -1;
        }
        ++issued[g];
        return s;
      };
      for (int k = 0, it = cta; it < nitems && !s_abort; ++k, it += grid) {
        const int g = k % kNG;
        int b, hk, ch, start;
        const int n = item_rows(it, b, hk, ch, start);
        const int n64 = n >> 6, n16 = ((n & 63) + 15) >> 4;
        const int row0 = a.layer_row0 + (b * a.Hkv + hk) * a.Tmax + start;
        const uint32_t kvb = (uint32_t)((n64 * 64 + n16 * 16) * 128 * (HDC / 64));  // K or V bytes
        const uint32_t qb = (uint32_t)(REP * HDC * 4);
        auto load = [&](const CUtensorMap* tm64, const CUtensorMap* tm16, unsigned char* dst, uint64_t* bar) {
          for (int h = 0; h < HDC / 64; ++h) {
            for (int i = 0; i < n64; ++i) tma_load_2d(dst + h * 16384 + i * 8192, tm64, h * 64, row0 + 64 * i, bar);
            for (int i = 0; i < n16; ++i)
              tma_load_2d(dst + h * 16384 + n64 * 8192 + i * 2048, tm16, h * 64, row0 + 64 * n64 + 16 * i, bar);
          }
        };
        const int sk = take(g);
        if (sk < 0) break;
        unsigned char* ks = ring + (size_t)sk * kSlotS;
        mbar_expect_tx(&full[sk], kvb * (TWO ? 1 : 2) + qb);
        load(&a.tmk64, &a.tmk, ks, &full[sk]);
        if (!TWO) load(&a.tmv64, &a.tmv, ks + 16384, &full[sk]);
        bulk_g2s(ks + kQOff, a.q + ((size_t)b * a.Hq + (size_t)hk * REP) * HDC, qb, &full[sk]);
        if (TWO) {
          const int sv = take(g);
          if (sv < 0) break;
          mbar_expect_tx(&full[sv], kvb);
          load(&a.tmv64, &a.tmv, ring + (size_t)sv * kSlotS, &full[sv]);
        }
      }
      // never leave with copies in flight
      if (s_abort)
        for (int g = 0; g < kNG; ++g)
          for (int u = max(0, issued[g] - NSG); u < issued[g]; ++u)
            mbar_wait(&full[g * NSG + u % NSG], (uint32_t)((u / NSG) & 1), kSpinS);
    }
  } else {
    // ================================ consumers ==================================
    const int grp = warp / kGW, gw = warp % kGW, gt = tid - grp * kGW * 32;
    float* wb = reinterpret_cast<float*>(ring + (size_t)NS * kSlotS) + (size_t)grp * kGW * REP * WS;
    const float scale = rsqrtf((float)HDC);
    for (int kg = 0, it = cta + grp * grid; it < nitems; ++kg, it += kNG * grid) {
      int b, hk, ch, start;
      const int n = item_rows(it, b, hk, ch, start);
      const int uk = SPI * kg, sk = grp * NSG + uk % NSG;
      const int uv = uk + SPI - 1, sv = grp * NSG + uv % NSG;
      bool ok = !s_abort && mbar_wait(&full[sk], (uint32_t)((uk / NSG) & 1), kSpinS);
      if (!ok && !s_abort) {
        if (lane == 0) atomicOr(a.err, RL_DEVERR_TIMEOUT);
        s_abort = 1;
      }
      const unsigned char* Ks = ring + (size_t)sk * kSlotS;
      const int j0 = gw * 16 * kNB;
      int jn = ok ? max(0, min(16 * kNB, n - j0)) : 0;
      PFrag<kNB> p;
      attn_scores<REP, HDC, kNB>(Ks, j0, jn, reinterpret_cast<const float*>(Ks + kQOff), lane, scale, p);
      if (TWO) {
        __syncwarp();
        if (lane == 0) mbar_arrive(&empty[sk]);  // this warp is done with the K rows and q
        ok = ok && !s_abort && mbar_wait(&full[sv], (uint32_t)((uv / NSG) & 1), kSpinS);
        if (!ok && !s_abort) {
          if (lane == 0) atomicOr(a.err, RL_DEVERR_TIMEOUT);
          s_abort = 1;
        }
        if (!ok) jn = 0;
      }
      const unsigned char* Vs = TWO ? ring + (size_t)sv * kSlotS : Ks + 16384;
      attn_values<REP, HDC, kNB>(Vs, j0, jn, p, lane, wb + (size_t)(gw * REP + (lane >> 2)) * WS);
      __syncwarp();
      if (lane == 0) mbar_arrive(&empty[sv]);  // done with the V rows (and, one slot, K)
      named_sync(1 + grp, kGW * 32);
      // combine the group's warps into the chunk's partial: [b][Hq][nch][hd + 2]
      float* part = a.part + ((size_t)b * a.Hq + (size_t)hk * REP) * nch * (HDC + 2);
      for (int i = gt; i < REP * HDC; i += kGW * 32) {
        const int h = i / HDC, dd = i % HDC;
        float M = -FLT_MAX;
#pragma unroll
        for (int w = 0; w < kGW; ++w) M = fmaxf(M, wb[(w * REP + h) * WS]);
        float num = 0.f, den = 0.f;
#pragma unroll
        for (int w = 0; w < kGW; ++w) {
          const float* ww = wb + (w * REP + h) * WS;
          const float f = ww[1] > 0.f ? __expf(ww[0] - M) : 0.f;
          num += f * ww[2 + dd];
          den += f * ww[1];
        }
        float* pp = part + ((size_t)h * nch + ch) * (HDC + 2);
        pp[dd] = num;
        if (dd == 0) {
          pp[HDC] = den > 0.f ? M : -FLT_MAX;
          pp[HDC + 1] = den;
        }
      }
      named_sync(1 + grp, kGW * 32);  // the partials area is rewritten by the group's next item
    }
  }
}

template <int REP, int HDC>
cudaError_t launch_one(const AttnStreamArgs& a, int grid, size_t smem, cudaStream_t s) {
  return launch_pdl(k_attn_stream<REP, HDC>, dim3(grid), dim3(kThreadsS), smem, s, a);
}

template <int REP, int HDC>
void setup_one(size_t smem) {
  cudaFuncSetAttribute(k_attn_stream<REP, HDC>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
}

}  // namespace

size_t attn_stream_smem(int* nslot) {
  if (nslot) *nslot = kMaxSlotsS;
  return (size_t)kMaxSlotsS * kSlotS + kPartS + 1024;
}

void attn_stream_setup() {
  const size_t smem = attn_stream_smem(nullptr);
  setup_one<1, 64>(smem);
  setup_one<2, 64>(smem);
  setup_one<4, 64>(smem);
  setup_one<1, 128>(smem);
  setup_one<2, 128>(smem);
  setup_one<4, 128>(smem);
}

bool attn_stream_supported(int rep, int hd) {
  return (rep == 1 || rep == 2 || rep == 4) && (hd == 64 || hd == 128);
}

cudaError_t launch_attn_stream(const AttnStreamArgs& a, int rep, int hd, int grid, cudaStream_t s) {
  const size_t smem = attn_stream_smem(nullptr);
  switch (rep * 1000 + hd) {
    case 1064: return launch_one<1, 64>(a, grid, smem, s);
    case 2064: return launch_one<2, 64>(a, grid, smem, s);
    case 4064: return launch_one<4, 64>(a, grid, smem, s);
    case 1128: return launch_one<1, 128>(a, grid, smem, s);
    case 2128: return launch_one<2, 128>(a, grid, smem, s);
    case 4128: return launch_one<4, 128>(a, grid, smem, s);
    default: return cudaErrorInvalidValue;
  }
}

}  // namespace river
