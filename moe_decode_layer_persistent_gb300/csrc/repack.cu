// repack.cu -- NVFP4 weight scale factors, re-laid out once at layer creation
// for the block-scaled tensor-core MMA.
//
// In:  scales [G][N][K/16] (one E4M3 byte per 16 inputs, the caller's layout).
// Out: [G][N/128][KB][4][512]: for every 128-row tile and every K-block of 256
//      inputs, four 512-byte chunks (64 inputs each) in the MMA's scale-factor
//      layout (row m, sub-block j at byte (m%32)*16 + (m/32)*4 + j).  Inputs
//      past K read as scale 0.
#include "host_util.h"

namespace mk {

__global__ void k_sf_repack(const uint8_t* __restrict__ in, uint8_t* __restrict__ out, int G,
                            int N, int K16, int KB) {
  const int NT = N / 128;
  const size_t total = static_cast<size_t>(G) * NT * KB * 2048;
  for (size_t i = blockIdx.x * static_cast<size_t>(blockDim.x) + threadIdx.x; i < total;
       i += static_cast<size_t>(gridDim.x) * blockDim.x) {
    const uint32_t within = static_cast<uint32_t>(i % 2048);
    size_t rest = i / 2048;
    const int kb = static_cast<int>(rest % KB);
    rest /= KB;
    const int nt = static_cast<int>(rest % NT);
    const size_t g = rest / NT;
    const uint32_t c = within / 512, a = within % 512;
    const uint32_t m = a / 16 + 32 * ((a % 16) / 4), j = a % 4;
    const int k16 = kb * 16 + static_cast<int>(c * 4 + j);
    uint8_t v = 0;
    if (k16 < K16) v = in[(g * N + static_cast<size_t>(nt) * 128 + m) * K16 + k16];
    out[i] = v;
  }
}

mk_status launch_sf_repack(const void* in, void* out, int G, int N, int K, cudaStream_t s) {
  if (N % 128 != 0 || K % 64 != 0) return MK_ERR_INVALID_ARG;
  const int K16 = K / 16, KB = (K + 255) / 256;
  k_sf_repack<<<1024, 256, 0, s>>>(static_cast<const uint8_t*>(in), static_cast<uint8_t*>(out),
                                   G, N, K16, KB);
  MK_CUDA_TRY(cudaGetLastError());
  return MK_OK;
}

size_t sf_repacked_bytes(int G, int N, int K) {
  return static_cast<size_t>(G) * (N / 128) * ((K + 255) / 256) * 2048;
}

}  // namespace mk
