// gemm_pair_f32.cu -- the CTA-pair GEMM kernels with f32 output.
#include "gemm_pair.cuh"

namespace hg {

cudaError_t launch_pair_f32(int pn, int ks, bool ts, const CUtensorMap &tmA, const CUtensorMap &tmB,
                            const CUtensorMap &tmC, const TiledParams &p, int grid, cudaStream_t s) {
    return launch_pair_typed<OUT_F32>(pn, ks, ts, tmA, tmB, tmC, p, grid, s);
}

}  // namespace hg
