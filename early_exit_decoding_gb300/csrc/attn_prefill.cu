// Causal prompt attention on the tensor cores (River-LLM explainer, section
// 五: the prompt is one pass whose layers all write the shared cache; the
// attention of prompt position p reads the cache rows 0..p of its sequence).
//
// One CTA per (block of query positions, KV head, sequence).  Its 128 query
// rows are the block's positions x the Hq/Hkv query heads that share the KV
// head (row r = position r / REP, head r % REP), so every K/V row staged in
// shared memory serves all of them.  A producer lane TMA-loads the K and V
// rows of 64-position key blocks (64-row x 64-dim boxes, 128-byte swizzle)
// into a ring; each of eight consumer warps owns 16 query rows and keeps a
// flash-style online softmax over the key blocks:
//   S = q K^T   (m16n8k16 MMAs; q split into bf16 high + low parts so the
//                products keep fp32-level accuracy, K is bf16 and exact)
//   causal mask, running max and sum, rescale of the output accumulator
//   O += P V    (P from the S accumulators, split into bf16 high + low)
// and writes O / sum in bf16 to the attention output rows.  Key blocks past
// the block's last position are never loaded.  Every wait is bounded; a wait
// that runs out sets RL_DEVERR_TIMEOUT and the CTA finishes without
// computing, after the copies it issued have landed.
#include <float.h>

#include "dev_common.cuh"
#include "internal.h"

namespace river {

namespace {

using namespace dev;

constexpr int kPfWarps = 8;                     // consumer warps
constexpr int kPfThreads = (kPfWarps + 1) * 32;  // + producer warp
constexpr int kPfRows = kPfWarps * 16;           // query rows per CTA
constexpr int kKB = 64;                          // key positions per block
constexpr int kPfStages = 3;
constexpr long long kPfSpin = 1ll << 20;

// Byte offset of 16-byte chunk c of row r in a 64-row block staged by TMA
// with the 128-byte swizzle (64-dim halves of 64 rows x 128 bytes, 8 KB apart).
__device__ __forceinline__ uint32_t blk_off(int r, int c) {
  return (uint32_t)((c >> 3) * (kKB * 128) + r * 128 + (((c & 7) ^ (r & 7)) << 4));
}

// Byte offset of 16-byte chunk c of query row r (HDC dims of bf16 per row),
// XOR-swizzled so the eight rows an ldmatrix reads sit in distinct banks.
template <int HDC>
__device__ __forceinline__ uint32_t q_off(int r, int c) {
  return (uint32_t)(r * HDC * 2 + ((c ^ (r & 7)) << 4));
}

template <int REP, int HDC>
__global__ void __launch_bounds__(kPfThreads, 1) k_attn_prefill(const __grid_constant__ AttnPrefillArgs a) {
  constexpr int QB = kPfRows / REP;  // query positions per CTA
  constexpr int KVB = kKB * HDC * 2;  // bytes of one K (or V) block
  constexpr int STAGE = 2 * KVB;
  extern __shared__ __align__(1024) unsigned char smem_raw[];
  __shared__ __align__(8) uint64_t full[kPfStages], empty[kPfStages];
  __shared__ int s_fail;
  unsigned char* smem = smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);
  unsigned char* ring = smem;                               // [stages][K block, V block]
  unsigned char* qhi = ring + kPfStages * STAGE;            // bf16 [128][HDC], swizzled
  unsigned char* qlo = qhi + kPfRows * HDC * 2;

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int nqb = (a.T + QB - 1) / QB;
  const int qb = nqb - 1 - (int)blockIdx.x;  // the longest rows first
  const int hk = blockIdx.y, seq = blockIdx.z;
  const int q0 = qb * QB;
  const int qlast = min(q0 + QB, a.T) - 1;   // last query position of the CTA
  const int nkb = qlast / kKB + 1;           // key blocks 0 .. nkb - 1
  const int row0 = a.layer_row0 + (seq * a.Hkv + hk) * a.Tmax;

  if (tid == 0) {
    for (int i = 0; i < kPfStages; ++i) {
      mbar_init(&full[i], 1);
      mbar_init(&empty[i], kPfWarps);
    }
    s_fail = 0;
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  }
  // the CTA's query rows, times 1/sqrt(hd), as bf16 high + low parts
  const float scale = rsqrtf((float)HDC);
  for (int i = tid; i < kPfRows * (HDC / 8); i += kPfThreads) {
    const int r = i / (HDC / 8), c = i % (HDC / 8);
    const int pos = q0 + r / REP, h = r % REP;
    float v[8];
    if (pos < a.T) {
      const float4* src = reinterpret_cast<const float4*>(
          a.q + ((size_t)(seq * a.T + pos) * a.Hq + (size_t)(hk * REP + h)) * HDC + c * 8);
      const float4 x0 = __ldg(src), x1 = __ldg(src + 1);
      v[0] = x0.x; v[1] = x0.y; v[2] = x0.z; v[3] = x0.w;
      v[4] = x1.x; v[5] = x1.y; v[6] = x1.z; v[7] = x1.w;
    } else {
#pragma unroll
      for (int j = 0; j < 8; ++j) v[j] = 0.f;
    }
    uint32_t hi[4], lo[4];
#pragma unroll
    for (int j = 0; j < 4; ++j) split_bf16x2(v[2 * j] * scale, v[2 * j + 1] * scale, hi[j], lo[j]);
    *reinterpret_cast<uint4*>(qhi + q_off<HDC>(r, c)) = make_uint4(hi[0], hi[1], hi[2], hi[3]);
    *reinterpret_cast<uint4*>(qlo + q_off<HDC>(r, c)) = make_uint4(lo[0], lo[1], lo[2], lo[3]);
  }
  __syncthreads();

  if (warp == kPfWarps) {
    // ------------------------------ producer ---------------------------------
    if (lane == 0) {
      int issued = 0;
      for (int kb = 0; kb < nkb; ++kb, ++issued) {
        const int st = kb % kPfStages, n = kb / kPfStages;
        if (n > 0 && !mbar_wait(&empty[st], (uint32_t)((n - 1) & 1), kPfSpin)) {
          s_fail = 1;
          break;
        }
        mbar_expect_tx(&full[st], (uint32_t)STAGE);
        unsigned char* ks = ring + st * STAGE;
#pragma unroll
        for (int hf = 0; hf < HDC / 64; ++hf) {
          tma_load_2d(ks + hf * (kKB * 128), &a.tmk64, hf * 64, row0 + kb * kKB, &full[st]);
          tma_load_2d(ks + KVB + hf * (kKB * 128), &a.tmv64, hf * 64, row0 + kb * kKB, &full[st]);
        }
      }
      // never leave with copies in flight
      for (int u = issued - kPfStages < 0 ? 0 : issued - kPfStages; u < issued; ++u)
        mbar_wait(&full[u % kPfStages], (uint32_t)((u / kPfStages) & 1), kPfSpin);
    }
  } else {
    // ------------------------------ consumers --------------------------------
    const int g = lane >> 2, t = lane & 3, mi = lane >> 3, ri = lane & 7;
    const int rA = warp * 16 + g, rB = rA + 8;       // this lane's two query rows
    const int pA = q0 + rA / REP, pB = q0 + rB / REP;  // their positions
    const int wlast = min(q0 + (warp * 16 + 15) / REP, a.T - 1);  // the warp's last position
    float o[HDC / 8][4];
#pragma unroll
    for (int n = 0; n < HDC / 8; ++n)
#pragma unroll
      for (int i = 0; i < 4; ++i) o[n][i] = 0.f;
    float mA = -FLT_MAX, mB = -FLT_MAX, lA = 0.f, lB = 0.f;
    const uint32_t qh = smem_u32(qhi), ql = smem_u32(qlo);
    for (int kb = 0; kb < nkb; ++kb) {
      const int st = kb % kPfStages;
      const bool ok = s_fail == 0 && mbar_wait(&full[st], (uint32_t)((kb / kPfStages) & 1), kPfSpin);
      if (!ok) s_fail = 1;
      const int k0 = kb * kKB;
      if (ok && k0 <= wlast) {  // blocks past the warp's last position add nothing
        const uint32_t kbase = smem_u32(ring + st * STAGE), vbase = kbase + KVB;
        // ---- S = q K^T over the block's 64 keys: 8 n-tiles of 8 keys ----
        float s[8][4];
#pragma unroll
        for (int n = 0; n < 8; ++n)
#pragma unroll
          for (int i = 0; i < 4; ++i) s[n][i] = 0.f;
#pragma unroll
        for (int ks = 0; ks < HDC / 16; ++ks) {
          uint32_t ah[4], al[4];
          const int qr = warp * 16 + (mi & 1) * 8 + ri, qc = ks * 2 + (mi >> 1);
          ldsm_x4(ah, qh + q_off<HDC>(qr, qc));
          ldsm_x4(al, ql + q_off<HDC>(qr, qc));
#pragma unroll
          for (int b = 0; b < 4; ++b) {  // 16 keys: b0 / b1 of two n-tiles
            uint32_t kf[4];
            ldsm_x4(kf, kbase + blk_off(16 * b + (mi >> 1) * 8 + ri, ks * 2 + (mi & 1)));
#pragma unroll
            for (int h = 0; h < 2; ++h) {
              mma_bf16(s[2 * b + h], ah[0], ah[1], ah[2], ah[3], kf[2 * h], kf[2 * h + 1]);
              mma_bf16(s[2 * b + h], al[0], al[1], al[2], al[3], kf[2 * h], kf[2 * h + 1]);
            }
          }
        }
        // ---- causal mask, online softmax ----
        float bA = -FLT_MAX, bB = -FLT_MAX;
#pragma unroll
        for (int n = 0; n < 8; ++n)
#pragma unroll
          for (int i = 0; i < 2; ++i) {
            const int key = k0 + 8 * n + 2 * t + i;
            if (key > pA) s[n][i] = -FLT_MAX;
            if (key > pB) s[n][2 + i] = -FLT_MAX;
            bA = fmaxf(bA, s[n][i]);
            bB = fmaxf(bB, s[n][2 + i]);
          }
        bA = fmaxf(bA, __shfl_xor_sync(0xffffffffu, bA, 1));
        bA = fmaxf(bA, __shfl_xor_sync(0xffffffffu, bA, 2));
        bB = fmaxf(bB, __shfl_xor_sync(0xffffffffu, bB, 1));
        bB = fmaxf(bB, __shfl_xor_sync(0xffffffffu, bB, 2));
        const float nA = fmaxf(mA, bA), nB = fmaxf(mB, bB);
        // a row with no valid key yet keeps max -FLT_MAX and weight 0
        const float cA = nA == -FLT_MAX ? 1.f : __expf(mA - nA);
        const float cB = nB == -FLT_MAX ? 1.f : __expf(mB - nB);
        mA = nA;
        mB = nB;
        lA *= cA;
        lB *= cB;
#pragma unroll
        for (int n = 0; n < HDC / 8; ++n) {
          o[n][0] *= cA;
          o[n][1] *= cA;
          o[n][2] *= cB;
          o[n][3] *= cB;
        }
#pragma unroll
        for (int n = 0; n < 8; ++n)
#pragma unroll
          for (int i = 0; i < 2; ++i) {
            s[n][i] = s[n][i] == -FLT_MAX ? 0.f : __expf(s[n][i] - mA);
            s[n][2 + i] = s[n][2 + i] == -FLT_MAX ? 0.f : __expf(s[n][2 + i] - mB);
            lA += s[n][i];
            lB += s[n][2 + i];
          }
        // ---- O += P V: 4 steps of 16 keys ----
#pragma unroll
        for (int kk = 0; kk < 4; ++kk) {
          uint32_t ph[4], pl[4];
          split_bf16x2(s[2 * kk][0], s[2 * kk][1], ph[0], pl[0]);          // row g, keys 2t
          split_bf16x2(s[2 * kk][2], s[2 * kk][3], ph[1], pl[1]);          // row g + 8
          split_bf16x2(s[2 * kk + 1][0], s[2 * kk + 1][1], ph[2], pl[2]);  // row g, keys 8 + 2t
          split_bf16x2(s[2 * kk + 1][2], s[2 * kk + 1][3], ph[3], pl[3]);  // row g + 8
          const int vrow = 16 * kk + (mi & 1) * 8 + ri;
#pragma unroll
          for (int nd = 0; nd < HDC / 8; nd += 2) {  // 16 dims: two n-tiles
            uint32_t vf[4];
            ldsm_x4_t(vf, vbase + blk_off(vrow, nd + (mi >> 1)));
#pragma unroll
            for (int h = 0; h < 2; ++h) {
              mma_bf16(o[nd + h], ph[0], ph[1], ph[2], ph[3], vf[2 * h], vf[2 * h + 1]);
              mma_bf16(o[nd + h], pl[0], pl[1], pl[2], pl[3], vf[2 * h], vf[2 * h + 1]);
            }
          }
        }
      }
      __syncwarp();
      if (lane == 0) mbar_arrive(&empty[st]);
    }
    // ---- O / sum -> bf16 output rows ----
    lA += __shfl_xor_sync(0xffffffffu, lA, 1);
    lA += __shfl_xor_sync(0xffffffffu, lA, 2);
    lB += __shfl_xor_sync(0xffffffffu, lB, 1);
    lB += __shfl_xor_sync(0xffffffffu, lB, 2);
    const float iA = lA > 0.f ? 1.f / lA : 0.f, iB = lB > 0.f ? 1.f / lB : 0.f;
    const int hA = rA % REP, hB = rB % REP;
    bf16* oA = a.o + (size_t)(seq * a.T + pA) * a.ldo + (size_t)(hk * REP + hA) * HDC;
    bf16* oB = a.o + (size_t)(seq * a.T + pB) * a.ldo + (size_t)(hk * REP + hB) * HDC;
#pragma unroll
    for (int n = 0; n < HDC / 8; ++n) {
      if (pA < a.T)
        *reinterpret_cast<__nv_bfloat162*>(oA + 8 * n + 2 * t) = __floats2bfloat162_rn(o[n][0] * iA, o[n][1] * iA);
      if (pB < a.T)
        *reinterpret_cast<__nv_bfloat162*>(oB + 8 * n + 2 * t) = __floats2bfloat162_rn(o[n][2] * iB, o[n][3] * iB);
    }
  }
  __syncthreads();
  if (tid == 0 && s_fail && a.err) atomicOr(a.err, RL_DEVERR_TIMEOUT);
}

template <int REP, int HDC>
constexpr size_t pf_smem() {
  return 1024 + (size_t)kPfStages * 2 * kKB * HDC * 2 + 2 * (size_t)kPfRows * HDC * 2;
}

template <int REP, int HDC>
cudaError_t launch_pf(const AttnPrefillArgs& a, cudaStream_t s) {
  constexpr size_t smem = pf_smem<REP, HDC>();
  static bool init = false;
  if (!init) {
    const cudaError_t e = cudaFuncSetAttribute(k_attn_prefill<REP, HDC>,
                                               cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
    init = true;
  }
  constexpr int QB = kPfRows / REP;
  const dim3 grid((a.T + QB - 1) / QB, a.Hkv, a.nseq);
  k_attn_prefill<REP, HDC><<<grid, kPfThreads, smem, s>>>(a);
  return cudaGetLastError();
}

}  // namespace

bool attn_prefill_supported(int rep, int hd) {
  return (rep == 1 || rep == 2 || rep == 4 || rep == 8) && (hd == 64 || hd == 128);
}

cudaError_t launch_attn_prefill(const AttnPrefillArgs& a, int rep, int hd, cudaStream_t s) {
  switch (rep * 1000 + hd) {
    case 1064: return launch_pf<1, 64>(a, s);
    case 2064: return launch_pf<2, 64>(a, s);
    case 4064: return launch_pf<4, 64>(a, s);
    case 8064: return launch_pf<8, 64>(a, s);
    case 1128: return launch_pf<1, 128>(a, s);
    case 2128: return launch_pf<2, 128>(a, s);
    case 4128: return launch_pf<4, 128>(a, s);
    case 8128: return launch_pf<8, 128>(a, s);
    default: return cudaErrorInvalidValue;
  }
}

}  // namespace river
