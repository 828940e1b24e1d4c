// gemm_pair_bf16.cu -- the CTA-pair GEMM kernels with bf16 output.
#include "gemm_pair.cuh"

namespace hg {

cudaError_t launch_pair_bf16(int pn, int ks, bool ts, const CUtensorMap &tmA, const CUtensorMap &tmB,
                             const CUtensorMap &tmC, const TiledParams &p, int grid, cudaStream_t s) {
    return launch_pair_typed<OUT_BF16>(pn, ks, ts, tmA, tmB, tmC, p, grid, s);
}

int pair_max_active_pairs_bf16() { return max_pairs_typed<OUT_BF16>(); }

}  // namespace hg
