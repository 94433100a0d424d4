// Instantiations of the CUDA-core attention kernel for __half elements (one
// translation unit per element type keeps the build parallel).
#include "attn_simt.cuh"

namespace pst {

cudaError_t launch_attn_simt_f16(int D, int C, int g, const AttnParams& p, int grid, cudaStream_t s) {
  return launch_simt_dc<__half>(D, C, g, p, grid, s);
}

}  // namespace pst
