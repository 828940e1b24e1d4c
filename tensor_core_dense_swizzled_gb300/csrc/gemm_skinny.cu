// gemm_skinny.cu -- the HBM-bound path for decode-shaped GEMMs (small M).
//
// With M <= 32 the product moves about 2*K*N bytes of B for 2*M*K*N FLOP, an
// arithmetic intensity near M FLOP/byte -- far below the ridge point, so the
// kernel is bound by streaming B from HBM ("tensor-cores-cutlass-and-cute",
// section 四.1 and the self-test of section 九 classify kernels by intensity
// against the ridge point).  The tensor core still does the arithmetic, but
// the design goal is bytes in flight and DRAM-friendly access, not MMA rate:
//
//   * swap A and B: compute C^T = B^T . A^T so that the large dimension N
//     fills the 128-row side of the MMA and M (padded to NU = 16 or 32 with
//     TMA zero fill) is the MMA's N.  B^T is read MN-major straight from the
//     row-major K x N B (64-column blocks); A^T is read K-major from the
//     row-major M x K A.
//   * a work unit covers NT x 128 consecutive columns of C (NT MMAs per
//     16-deep K step), so every K row of B is read in runs of NT x 256
//     contiguous bytes;
//   * split K into `split` ranges so that batch * split * ceil(N / (128 NT))
//     work units fill every SM with a balanced number of units; each
//     persistent CTA runs a deep ring of stages (about 200 KB in flight).
//   * fixup: every unit writes its fp32 partials (NU x 128 per 128-column
//     sub-tile) to workspace; for each 32-column quarter of a sub-tile, the
//     epilogue warp that arrives last at that quarter's counter sums the
//     partials in split order 0, 1, ... (so the result does not depend on
//     arrival order), converts, writes C and resets the counter for the next
//     run.  No warp waits on another at an unbounded barrier.
#include "kernels.h"
#include "ptx.cuh"
#include "tile_common.cuh"
#include "watchdog.cuh"

namespace hg {
namespace {

constexpr int BK = 64;
constexpr int TN = 128;  // columns of C per MMA (= MMA M)
constexpr int NUM_THREADS = 192;
constexpr int EPI_WARPS = 4;

constexpr uint32_t pow2_at_least(uint32_t x) {
    uint32_t p = 32;
    while (p < x) p <<= 1;
    return p;
}

template <int NU, int NT>
struct SkinnyCfg {
    static_assert(NU == 16 || NU == 32, "padded M");
    static_assert(NT == 1 || NT == 2 || NT == 4, "128-column sub-tiles per unit");
    static constexpr int W_BLOCKS = 2 * NT;          // 64-column blocks of B per stage
    static constexpr uint32_t W_BLOCK = BK * 128;    // 64 k x 64 n
    static constexpr uint32_t W_BYTES = W_BLOCKS * W_BLOCK;
    static constexpr uint32_t X_BYTES = NU * BK * 2;  // A tile: NU rows x 64 k
    static constexpr uint32_t TX_BYTES = W_BYTES + X_BYTES;
    static constexpr int STAGES_FIT = (232448 - 2048) / (W_BYTES + X_BYTES);
    static constexpr int STAGES = STAGES_FIT > 12 ? 12 : STAGES_FIT;
    static constexpr uint32_t TMEM_STRIDE = NT * NU;  // columns per accumulator buffer
    static constexpr uint32_t TMEM_COLS = pow2_at_least(2 * TMEM_STRIDE);
    static constexpr int SMEM_W = 0;
    static constexpr int SMEM_X = SMEM_W + STAGES * W_BYTES;
    static constexpr int SMEM_BAR = SMEM_X + STAGES * X_BYTES;
    static constexpr int NUM_BARS = 2 * STAGES + 4 + 1;
    static constexpr int SMEM_MISC = SMEM_BAR + NUM_BARS * 8;
    static constexpr int SMEM_TOTAL = SMEM_MISC + 16 + 1024;
    static_assert(SMEM_TOTAL <= 232448, "shared memory budget");
};

__device__ __forceinline__ void unit_coords(const SkinnyParams &p, int u, int &b, int &s, int &nt) {
    const int per_batch = p.split * p.num_tiles;
    b = u / per_batch;
    const int r = u - b * per_batch;
    s = r / p.num_tiles;  // split index varies slowest: concurrent units read adjacent columns
    nt = r - s * p.num_tiles;
}

template <int NU, int NT, int OUT>
__global__ void __launch_bounds__(NUM_THREADS, 1)
    hgemm_skinny_kernel(const __grid_constant__ CUtensorMap tmX,
                        const __grid_constant__ CUtensorMap tmW, const SkinnyParams p) {
    using Cfg = SkinnyCfg<NU, NT>;
    extern __shared__ uint8_t smem_raw[];
    const uint32_t raw = smem_u32(smem_raw);
    uint8_t *smem = smem_raw + ((1024u - (raw & 1023u)) & 1023u);
    const uint32_t sbase = smem_u32(smem);
    const uint32_t sW = sbase + Cfg::SMEM_W;
    const uint32_t sX = sbase + Cfg::SMEM_X;
    const uint32_t bar0 = sbase + Cfg::SMEM_BAR;
    auto full = [&](int s) { return bar0 + 8u * s; };
    auto empty = [&](int s) { return bar0 + 8u * (Cfg::STAGES + s); };
    auto tfull = [&](int b) { return bar0 + 8u * (2 * Cfg::STAGES + b); };
    auto tempty = [&](int b) { return bar0 + 8u * (2 * Cfg::STAGES + 2 + b); };
    const uint32_t drain = bar0 + 8u * (2 * Cfg::STAGES + 4);
    volatile uint32_t *tmem_slot = reinterpret_cast<volatile uint32_t *>(smem + Cfg::SMEM_MISC);
    volatile int32_t *abort_flag = reinterpret_cast<volatile int32_t *>(smem + Cfg::SMEM_MISC + 4);

    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;

    if (threadIdx.x == 0) {
        for (int s = 0; s < Cfg::STAGES; ++s) {
            mbar_init(full(s), 1);
            mbar_init(empty(s), 1);
        }
        for (int b = 0; b < 2; ++b) {
            mbar_init(tfull(b), 1);
            mbar_init(tempty(b), EPI_WARPS);
        }
        mbar_init(drain, 1);
        *abort_flag = 0;
        fence_mbar_init();
        prefetch_tmap(&tmX);
        prefetch_tmap(&tmW);
    }
    if (warp == 1) {
        tmem_alloc(smem_u32(const_cast<uint32_t *>(tmem_slot)), Cfg::TMEM_COLS);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem_base = *tmem_slot;
    const WaitCtl wc{abort_flag, p.err, p.timeout_ns};
    // The next kernel of the stream may be scheduled now; it waits for this
    // one to complete before it reads memory (griddep_wait below).
    if (threadIdx.x == 0) griddep_launch_dependents();

    if (warp == 0) {
        // ------------------------------------------------------------ TMA producer
        if (lane == 0) {
            // Nothing this kernel reads may be read before the previous kernel
            // of the stream has completed (dependent launches).
            griddep_wait();
            int stage = 0;
            uint32_t phase = 0;
            int issued = 0;
            bool ok = true;
            for (int u = blockIdx.x; ok && u < p.units; u += gridDim.x) {
                int b, s, nt;
                unit_coords(p, u, b, s, nt);
                const int kb0 = s * p.kb_per_split;
                const int kb1 = min(p.num_kb, kb0 + p.kb_per_split);
                for (int kb = kb0; kb < kb1; ++kb) {
                    if (!wait_bounded(empty(stage), phase ^ 1u, wc,
                                      timeout_code(ROLE_PRODUCER, stage))) {
                        ok = false;
                        break;
                    }
                    mbar_arrive_expect_tx(full(stage), Cfg::TX_BYTES);
#pragma unroll
                    for (int j = 0; j < Cfg::W_BLOCKS; ++j)
                        tma_load_3d(sW + stage * Cfg::W_BYTES + j * Cfg::W_BLOCK, &tmW, full(stage),
                                    nt * (NT * TN) + j * 64, kb * BK, b);
                    tma_load_3d(sX + stage * Cfg::X_BYTES, &tmX, full(stage), kb * BK, 0, b);
                    ++issued;
                    if (++stage == Cfg::STAGES) {
                        stage = 0;
                        phase ^= 1u;
                    }
                }
            }
            const int pending = issued < Cfg::STAGES ? issued : Cfg::STAGES;
            for (int i = 0; i < pending; ++i) {
                if (stage == 0) {
                    stage = Cfg::STAGES - 1;
                    phase ^= 1u;
                } else {
                    --stage;
                }
                wait_bounded(full(stage), phase, wc, 0, /*honor_abort=*/false);
            }
        }
    } else if (warp == 1) {
        // ------------------------------------------------------------ MMA issuer
        if (lane == 0) {
            int stage = 0;
            uint32_t phase = 0;
            bool ok = true;
            int local = 0;
            for (int u = blockIdx.x; ok && u < p.units; u += gridDim.x, ++local) {
                int b, s, nt;
                unit_coords(p, u, b, s, nt);
                const int kb0 = s * p.kb_per_split;
                const int kb1 = min(p.num_kb, kb0 + p.kb_per_split);
                const int buf = local & 1;
                const uint32_t tph = (local >> 1) & 1;
                if (!wait_bounded(tempty(buf), tph ^ 1u, wc, timeout_code(ROLE_MMA, 0x100 + buf))) {
                    ok = false;
                    break;
                }
                tc_fence_after();
                const uint32_t d0 = tmem_base + buf * Cfg::TMEM_STRIDE;
                for (int kb = kb0; kb < kb1; ++kb) {
                    if (!wait_bounded(full(stage), phase, wc, timeout_code(ROLE_MMA, stage))) {
                        ok = false;
                        break;
                    }
                    tc_fence_after();
                    const uint32_t w0 = sW + stage * Cfg::W_BYTES;
                    const uint32_t x0 = sX + stage * Cfg::X_BYTES;
#pragma unroll
                    for (int k = 0; k < BK / 16; ++k) {
                        const uint64_t bd = sdesc_sw128(x0 + k * 32, 16, 1024);  // MMA B = A^T, K-major
#pragma unroll
                        for (int j = 0; j < NT; ++j) {
                            // MMA A = columns j*128 .. j*128+127 of the B tile, MN-major
                            const uint64_t ad = sdesc_sw128(
                                w0 + 2 * j * Cfg::W_BLOCK + k * 16 * 128, Cfg::W_BLOCK, 1024);
                            umma_f16(d0 + j * NU, ad, bd, p.idesc, (kb > kb0 || k > 0) ? 1u : 0u);
                        }
                    }
                    umma_commit(empty(stage));
                    if (++stage == Cfg::STAGES) {
                        stage = 0;
                        phase ^= 1u;
                    }
                }
                if (!ok) break;
                umma_commit(tfull(buf));
            }
            umma_commit(drain);
            wait_bounded(drain, 0, wc, 0, /*honor_abort=*/false);
        }
    } else {
        // ------------------------------------------------------------ epilogue + fixup
        const int q = warp & 3;
        int local = 0;
        const int num_n128 = (p.N + TN - 1) / TN;
        for (int u = blockIdx.x; u < p.units; u += gridDim.x, ++local) {
            int b, s, nt;
            unit_coords(p, u, b, s, nt);
            const int buf = local & 1;
            const uint32_t tph = (local >> 1) & 1;
            if (!wait_bounded_warp(tfull(buf), tph, wc, timeout_code(ROLE_EPILOGUE, buf))) break;
            tc_fence_after();
            const uint32_t tq =
                tmem_base + (static_cast<uint32_t>(q * 32) << 16) + buf * Cfg::TMEM_STRIDE;
            uint32_t v[NT][NU];
#pragma unroll
            for (int j = 0; j < NT; ++j) {
                if constexpr (NU == 16) {
                    tmem_ld16(tq + j * NU, v[j]);
                } else {
                    tmem_ld32(tq + j * NU, v[j]);
                }
            }
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(tempty(buf));

            const int nl = q * 32 + lane;  // column within a 128-column sub-tile
            const int64_t cbase = static_cast<int64_t>(b) * p.strideC;
#pragma unroll
            for (int j = 0; j < NT; ++j) {
                const int n128 = nt * NT + j;
                if (n128 >= num_n128) break;  // sub-tile entirely past N (warp-uniform)
                const int n = n128 * TN + nl;
                if (p.split == 1) {
                    if (n < p.N) {
#pragma unroll
                        for (int m = 0; m < NU; ++m)
                            if (m < p.M)
                                store_one<OUT>(p.C, cbase + static_cast<int64_t>(m) * p.ldc + n,
                                               __uint_as_float(v[j][m]));
                    }
                    continue;
                }
                const int64_t ctr = (static_cast<int64_t>(b) * num_n128 + n128) * EPI_WARPS + q;
                float *part = p.partials +
                              ((static_cast<int64_t>(b) * p.split + s) * num_n128 + n128) *
                                  (static_cast<int64_t>(NU) * TN);
#pragma unroll
                for (int m = 0; m < NU; ++m) __stcg(part + m * TN + nl, __uint_as_float(v[j][m]));
                __threadfence();
                __syncwarp();
                int last = 0;
                if (lane == 0) last = (atomicAdd(p.counters + ctr, 1) == p.split - 1) ? 1 : 0;
                last = __shfl_sync(0xFFFFFFFFu, last, 0);
                if (last) {
                    __threadfence();
                    const int64_t stride_split = static_cast<int64_t>(num_n128) * NU * TN;
                    const float *p0 = p.partials +
                                      (static_cast<int64_t>(b) * p.split * num_n128 + n128) * (NU * TN);
                    if (n < p.N) {
                        for (int m = 0; m < p.M && m < NU; ++m) {
                            float acc = 0.f;
                            for (int ss = 0; ss < p.split; ++ss)
                                acc += __ldcg(p0 + ss * stride_split + m * TN + nl);
                            store_one<OUT>(p.C, cbase + static_cast<int64_t>(m) * p.ldc + n, acc);
                        }
                    }
                    if (lane == 0) p.counters[ctr] = 0;  // ready for the next run
                }
            }
        }
    }

    __syncwarp();
    tc_fence_before();
    __syncthreads();
    if (warp == 1) {
        tc_fence_after();
        tmem_dealloc(tmem_base, Cfg::TMEM_COLS);
    }
}

template <int NU, int NT, int OUT>
cudaError_t launch_impl(const CUtensorMap &tmX, const CUtensorMap &tmW, const SkinnyParams &p,
                        int grid, cudaStream_t stream) {
    auto kern = hgemm_skinny_kernel<NU, NT, OUT>;
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         SkinnyCfg<NU, NT>::SMEM_TOTAL);
    if (e != cudaSuccess) return e;
    return launch_dependent(kern, grid, NUM_THREADS, SkinnyCfg<NU, NT>::SMEM_TOTAL, stream, tmX,
                            tmW, p);
}

template <int NU, int NT>
cudaError_t launch_out(int out, const CUtensorMap &tmX, const CUtensorMap &tmW,
                       const SkinnyParams &p, int grid, cudaStream_t s) {
    switch (out) {
        case OUT_F16: return launch_impl<NU, NT, OUT_F16>(tmX, tmW, p, grid, s);
        case OUT_BF16: return launch_impl<NU, NT, OUT_BF16>(tmX, tmW, p, grid, s);
        case OUT_F32: return launch_impl<NU, NT, OUT_F32>(tmX, tmW, p, grid, s);
        default: return cudaErrorInvalidValue;
    }
}

template <int NU>
cudaError_t launch_nt(int nt, int out, const CUtensorMap &tmX, const CUtensorMap &tmW,
                      const SkinnyParams &p, int grid, cudaStream_t s) {
    switch (nt) {
        case 1: return launch_out<NU, 1>(out, tmX, tmW, p, grid, s);
        case 2: return launch_out<NU, 2>(out, tmX, tmW, p, grid, s);
        case 4: return launch_out<NU, 4>(out, tmX, tmW, p, grid, s);
        default: return cudaErrorInvalidValue;
    }
}

}  // namespace

int skinny_stages(int nu, int nt) {
    if (nu == 16)
        return nt == 1 ? SkinnyCfg<16, 1>::STAGES
                       : (nt == 2 ? SkinnyCfg<16, 2>::STAGES : SkinnyCfg<16, 4>::STAGES);
    return nt == 1 ? SkinnyCfg<32, 1>::STAGES
                   : (nt == 2 ? SkinnyCfg<32, 2>::STAGES : SkinnyCfg<32, 4>::STAGES);
}

cudaError_t launch_skinny(int nu, int nt, int out, const CUtensorMap &tmX, const CUtensorMap &tmW,
                          const SkinnyParams &p, int grid, cudaStream_t stream) {
    if (nu == 16) return launch_nt<16>(nt, out, tmX, tmW, p, grid, stream);
    if (nu == 32) return launch_nt<32>(nt, out, tmX, tmW, p, grid, stream);
    return cudaErrorInvalidValue;
}

}  // namespace hg
