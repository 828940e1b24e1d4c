// gemm_skinny_bf16.cu -- the skinny-path kernels with bf16 output.
#include "gemm_skinny.cuh"

namespace hg {

cudaError_t launch_skinny_bf16(int nu, int nb, const CUtensorMap &tmX, const CUtensorMap &tmW,
                               const SkinnyParams &p, int grid, cudaStream_t s) {
    return launch_skinny_typed<OUT_BF16>(nu, nb, tmX, tmW, p, grid, s);
}

}  // namespace hg
