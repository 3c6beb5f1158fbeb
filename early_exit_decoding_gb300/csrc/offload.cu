// Backbone offloading (River-LLM explainer, section 五: deep backbone layers
// are rarely run once the exit river is in place, so their weights can live
// in host memory and be fetched only on the steps that run them).
//
// On GB300 the host memory is the Grace CPU's, reached over NVLink-C2C.  The
// persistent decode-step kernel reads an offloaded layer's unit-tiled weights
// straight from there (16-byte cp.async copies into its ring, only for the
// layers a step runs on the backbone); the other paths (prefill, the fused
// and generic decode) read weights through TMA tensor maps or bulk copies
// from device memory, so before each offloaded layer a staging kernel copies
// its [N][Kp] weights into one device buffer shared by all offloaded layers
// -- and does nothing when the device-side exit state says the layer runs on
// the exit river.
#include "internal.h"

namespace river {

namespace {

__global__ void k_stage_weights(const uint4* __restrict__ src, uint4* __restrict__ dst, size_t n16,
                                const int* __restrict__ exit_layer, int layer_no) {
  if (exit_layer && layer_no > *exit_layer) return;  // the layer runs on its W4 exit copy
  const size_t stride = (size_t)gridDim.x * blockDim.x;
  for (size_t i = (size_t)blockIdx.x * blockDim.x + threadIdx.x; i < n16; i += stride) dst[i] = src[i];
}

}  // namespace

void launch_stage_weights(const void* src, void* dst, size_t bytes, const int* exit_layer, int layer_no,
                          int sm_count, cudaStream_t s) {
  k_stage_weights<<<4 * sm_count, 256, 0, s>>>(static_cast<const uint4*>(src), static_cast<uint4*>(dst),
                                                bytes / 16, exit_layer, layer_no);
}

}  // namespace river
