// Instantiations of the CUDA-core attention kernel for __half elements at
// chunk sizes 16 and 32 (one translation unit per element type and chunk-size pair
// keeps the build parallel).
#include "attn_simt.cuh"

namespace pst {

cudaError_t launch_attn_simt_f16_small(int D, int C, int g, const AttnParams& p, int grid, cudaStream_t s) {
  return launch_simt_dc<__half, 16, 32>(D, C, g, p, grid, s);
}

}  // namespace pst
