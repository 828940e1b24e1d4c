// gemm_skinny.cu -- public entry points of the skinny-path GEMM
// (gemm_skinny.cuh); the kernels are instantiated per output type in
// gemm_skinny_{f16,bf16,f32}.cu.
#include "gemm_skinny.cuh"

namespace hg {

int skinny_stages(int nu, int nb) { return nu == 16 ? stages_nb<16>(nb) : stages_nb<32>(nb); }

cudaError_t launch_skinny(int nu, int nb, int out, const CUtensorMap &tmX, const CUtensorMap &tmW,
                          const SkinnyParams &p, int grid, cudaStream_t stream) {
    switch (out) {
        case OUT_F16: return launch_skinny_f16(nu, nb, tmX, tmW, p, grid, stream);
        case OUT_BF16: return launch_skinny_bf16(nu, nb, tmX, tmW, p, grid, stream);
        case OUT_F32: return launch_skinny_f32(nu, nb, tmX, tmW, p, grid, stream);
        default: return cudaErrorInvalidValue;
    }
}

}  // namespace hg
