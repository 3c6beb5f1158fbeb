// Streaming decode attention for any batch (River-LLM explainer, section 三:
// every layer, backbone or exit river, reads the backbone's own K/V slots).
//
// One persistent CTA per SM walks the (sequence, KV head, chunk of <= 128
// positions) items.  A producer lane TMA-loads each chunk's K and V rows
// (16-row x 64-dim boxes, 128-byte swizzle, from the one tensor map that
// covers every layer's cache) and the item's query rows into a ring of
// shared-memory slots, running ahead of the consumers; eight consumer warps
// run the chunk on the tensor cores (attn::attn_warp_tc: q K^T and P V as
// m16n8k16 MMAs, 16 positions per warp), combine the warps' online-softmax
// partials and write the chunk's (o, max, sum) partial; k_attn_combine then
// merges the chunks.  Every wait is bounded: a wait that runs out sets
// RL_DEVERR_TIMEOUT and the kernel winds down.
#include "attn_tc.cuh"
#include "dev_common.cuh"

namespace river {

namespace {

using namespace dev;
using namespace attn;

constexpr int kNCW = 8;                      // consumer warps
constexpr int kThreadsS = (kNCW + 1) * 32;   // + the producer warp
constexpr int kSlotS = 34816;                // 32 KB of K (+ V) rows + the query rows
constexpr int kQOff = 32768;                 // query rows inside a slot
constexpr int kMaxSlotsS = 6;
constexpr long long kSpinS = 1LL << 22;

template <int REP, int HDC>
__global__ void __launch_bounds__(kThreadsS, 1) k_attn_stream(const __grid_constant__ AttnStreamArgs a) {
  constexpr bool TWO = HDC == 128;  // K and V rows in separate slots
  constexpr int WS = 2 + HDC;
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
      mbar_init(&empty[i], kNCW);
    }
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    s_pos = *a.pos_ptr;
    s_abort = 0;
  }
  __syncthreads();
  const int pos = s_pos;
  const int ctx = min(pos + 1, a.Tmax);
  const int nch = a.nchunks;
  const int clen = (ctx + nch - 1) / nch;
  const int nitems = a.nq * a.Hkv * nch;
  const int grid = gridDim.x, cta = blockIdx.x;

  if (warp == kNCW) {
    // ================================ producer ===================================
    if (lane == 0) {
      int slot = 0, round = 0, issued = 0;
      auto take = [&]() -> int {
        if (round > 0 && !mbar_wait(&empty[slot], (uint32_t)((round - 1) & 1), kSpinS)) {
          atomicOr(a.err, RL_DEVERR_TIMEOUT);
          s_abort = 1;
          return -1;
        }
        const int s = slot;
        if (++slot == NS) {
          slot = 0;
          ++round;
        }
        ++issued;
        return s;
      };
      for (int it = cta; it < nitems && !s_abort; it += grid) {
        const int b = it / (a.Hkv * nch), rr = it % (a.Hkv * nch), hk = rr / nch, ch = rr % nch;
        const int start = ch * clen, n = min(128, max(0, min(start + clen, ctx) - start));
        const int nbox = (n + 15) >> 4;
        const int row0 = a.layer_row0 + (b * a.Hkv + hk) * a.Tmax + start;
        const uint32_t kvb = (uint32_t)(nbox * 2048 * (HDC / 64));  // K or V bytes
        const uint32_t qb = (uint32_t)(REP * HDC * 4);
        auto load = [&](const CUtensorMap* tm, unsigned char* dst, uint64_t* bar) {
          for (int h = 0; h < HDC / 64; ++h)
            for (int i = 0; i < nbox; ++i) tma_load_2d(dst + h * 16384 + i * 2048, tm, h * 64, row0 + 16 * i, bar);
        };
        const int sk = take();
        if (sk < 0) break;
        unsigned char* ks = ring + (size_t)sk * kSlotS;
        mbar_expect_tx(&full[sk], kvb * (TWO ? 1 : 2) + qb);
        load(&a.tmk, ks, &full[sk]);
        if (!TWO) load(&a.tmv, ks + 16384, &full[sk]);
        bulk_g2s(ks + kQOff, a.q + ((size_t)b * a.Hq + (size_t)hk * REP) * HDC, qb, &full[sk]);
        if (TWO) {
          const int sv = take();
          if (sv < 0) break;
          mbar_expect_tx(&full[sv], kvb);
          load(&a.tmv, ring + (size_t)sv * kSlotS, &full[sv]);
        }
      }
      // never leave with copies in flight
      if (s_abort)
        for (int u = issued - NS < 0 ? 0 : issued - NS; u < issued; ++u)
          mbar_wait(&full[u % NS], (uint32_t)((u / NS) & 1), kSpinS);
    }
  } else {
    // ================================ consumers ==================================
    const int ct = tid;
    int slot = 0, round = 0;
    const float scale = rsqrtf((float)HDC);
    for (int it = cta; it < nitems; it += grid) {
      const int b = it / (a.Hkv * nch), rr = it % (a.Hkv * nch), hk = rr / nch, ch = rr % nch;
      const int start = ch * clen, n = min(128, max(0, min(start + clen, ctx) - start));
      const int sk = slot;
      bool ok = !s_abort && mbar_wait(&full[sk], (uint32_t)(round & 1), kSpinS);
      if (++slot == NS) {
        slot = 0;
        ++round;
      }
      int sv = sk;
      if (TWO) {
        sv = slot;
        ok = ok && mbar_wait(&full[sv], (uint32_t)(round & 1), kSpinS);
        if (++slot == NS) {
          slot = 0;
          ++round;
        }
      }
      if (!ok && !s_abort) {
        if (lane == 0) atomicOr(a.err, RL_DEVERR_TIMEOUT);
        s_abort = 1;
      }
      unsigned char* Ks = ring + (size_t)sk * kSlotS;
      unsigned char* Vs = TWO ? ring + (size_t)sv * kSlotS : Ks + 16384;
      const float* qs = reinterpret_cast<const float*>(Ks + kQOff);
      float* wb = reinterpret_cast<float*>(Ks);  // the warps' partials overlay the K rows
      const int nn = ok ? n : 0;
      const int j0 = warp * 16, jn = max(0, min(16, nn - j0));
      attn_warp_tc<REP, HDC>(Ks, Vs, j0, jn, qs, lane, wb + (size_t)warp * REP * WS, scale);
      named_sync(1, kNCW * 32);
      // combine the eight warps into the chunk's partial: [b][Hq][nch][hd + 2]
      float* part = a.part + ((size_t)b * a.Hq + (size_t)hk * REP) * nch * (HDC + 2);
      for (int i = ct; i < REP * HDC; i += kNCW * 32) {
        const int h = i / HDC, dd = i % HDC;
        float M = -FLT_MAX;
#pragma unroll
        for (int w = 0; w < kNCW; ++w) M = fmaxf(M, wb[(w * REP + h) * WS]);
        float num = 0.f, den = 0.f;
#pragma unroll
        for (int w = 0; w < kNCW; ++w) {
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
      fence_proxy_async_smem();  // the slot is refilled by bulk copies
      named_sync(1, kNCW * 32);
      if (lane == 0) {
        mbar_arrive(&empty[sk]);
        if (TWO) mbar_arrive(&empty[sv]);
      }
    }
  }
}

template <int REP, int HDC>
cudaError_t launch_one(const AttnStreamArgs& a, int grid, size_t smem, cudaStream_t s) {
  k_attn_stream<REP, HDC><<<grid, kThreadsS, smem, s>>>(a);
  return cudaGetLastError();
}

template <int REP, int HDC>
void setup_one(size_t smem) {
  cudaFuncSetAttribute(k_attn_stream<REP, HDC>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
}

}  // namespace

size_t attn_stream_smem(int* nslot) {
  if (nslot) *nslot = kMaxSlotsS;
  return (size_t)kMaxSlotsS * kSlotS + 1024;
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
