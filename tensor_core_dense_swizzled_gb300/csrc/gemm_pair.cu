// gemm_pair.cu -- public entry points of the CTA-pair GEMM (gemm_pair.cuh);
// the kernels are instantiated per output type in gemm_pair_{f16,bf16,f32}.cu.
#include "gemm_pair.cuh"

namespace hg {

int pair_stages(int ks) { return ks == 1 ? PairCfg<256, 1>::STAGES : PairCfg<256, 2>::STAGES; }

int pair_max_active_pairs() { return pair_max_active_pairs_bf16(); }

cudaError_t launch_pair(int pn, int ks, int out, bool tma_store, const CUtensorMap &tmA,
                        const CUtensorMap &tmB, const CUtensorMap &tmC, const TiledParams &p,
                        int grid, cudaStream_t stream) {
    switch (out) {
        case OUT_F16: return launch_pair_f16(pn, ks, tma_store, tmA, tmB, tmC, p, grid, stream);
        case OUT_BF16: return launch_pair_bf16(pn, ks, tma_store, tmA, tmB, tmC, p, grid, stream);
        case OUT_F32: return launch_pair_f32(pn, ks, tma_store, tmA, tmB, tmC, p, grid, stream);
        default: return cudaErrorInvalidValue;
    }
}

}  // namespace hg
