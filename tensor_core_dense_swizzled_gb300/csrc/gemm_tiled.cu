// gemm_tiled.cu -- persistent, warp-specialised tcgen05 GEMM for sm_103a.
//
// C_b = A_b . B_b with A (M x K) and B (K x N) row-major, fp16/bf16 inputs,
// fp32 accumulation in tensor memory, fp32/fp16/bf16 output.
//
// Structure (the Blackwell form of "tensor-cores-cutlass-and-cute" section 五.3,
// warp specialisation with full/empty barrier pairs around a stage ring):
//   warp 0, one thread   TMA producer: for every 64-deep K block waits until
//                        the stage is empty, arms full[stage] with the byte
//                        count (section 五.1) and issues one A box (128 x 64)
//                        and ceil(BN/64) B boxes (64 x 64) into 128-byte-
//                        swizzled shared memory.
//   warp 1, one thread   MMA issuer: waits full[stage], issues four
//                        tcgen05.mma (K = 16 each) that read A and B from
//                        shared memory through descriptors (section 五.2) and
//                        accumulate into a TMEM buffer, then tcgen05.commit
//                        frees the stage.  After a tile's last K block it
//                        commits tfull[buf].
//   warps 2-5 (or 2-9)   epilogue: wait tfull[buf], tcgen05.ld 32-column
//                        chunks (lane = output row), convert, stage each
//                        32-row x 128-byte piece in 128-byte-swizzled shared
//                        memory and TMA-store it (section 四.5's point that
//                        the epilogue should write full sectors), or write C
//                        with predicated coalesced stores when C is not
//                        16-byte aligned.  They release TMEM (tempty[buf]) as
//                        soon as the last chunk is in registers.  With
//                        eight epilogue warps (EW = 8: products with few K
//                        blocks, where draining the accumulator bounds the
//                        tile, e.g. batched S = Q K^T with K = 128), two
//                        warps share each TMEM lane quarter, one per half of
//                        the tile's 32-column chunks.
// Two TMEM accumulator buffers let the epilogue of tile i overlap the main
// loop of tile i+1 -- the effect "ping-pong" consumers buy on Hopper
// (section 五.3).  The CTA loops over tiles (persistent; grid <= SM count) in
// grouped order so that concurrently running CTAs share A and B in L2
// (section 四.5 lists tile order as one of the gaps).
//
// Operand layouts in shared memory (both from TMA with SWIZZLE_128B, which is
// the hardware form of the XOR swizzle of section 三.5: 16-byte chunk c of row
// r goes to chunk c ^ (r & 7)):
//   A: K-major, 128 rows x 128 bytes (64 k); descriptor SBO = 1024.
//   B: MN-major (B is K x N row-major, so N is contiguous): ceil(BN/64) blocks of
//      64 k-rows x 128 bytes (64 n); descriptor LBO = 8192 (next n block),
//      SBO = 1024 (next 8 k).  The k-th MMA of a stage starts 16 rows
//      (2048 bytes) further.
// Ragged M/N/K edges are handled by TMA: loads zero-fill outside the tensor
// and stores clip to it.
#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include "kernels.h"
#include "ptx.cuh"
#include "tile_common.cuh"
#include "watchdog.cuh"

namespace hg {
namespace {

constexpr int BM = 128;
constexpr int BK = 64;
constexpr int STG_BYTES = EPI_STG_BYTES;
constexpr int STG_BUFS = EPI_STG_BUFS;

// EW: epilogue warps (4 or 8); warp 0 TMA, warp 1 MMA, warps 2 .. EW + 1 epilogue.
template <int BN, int EW = 4>
struct TiledCfg {
    static_assert(BN == 128 || BN == 192 || BN == 224 || BN == 256, "tile N");
    static_assert(EW == 4 || EW == 8, "epilogue warps");
    static constexpr int THREADS = 32 * (2 + EW);
    static constexpr int B_BLOCKS = (BN + 63) / 64;  // 64-column blocks of B per stage
    static constexpr uint32_t A_BYTES = BM * BK * 2;
    static constexpr uint32_t B_BLOCK = BK * 128;  // 64 k-rows x 64 n (128 bytes)
    static constexpr uint32_t B_BYTES = B_BLOCKS * B_BLOCK;
    static constexpr uint32_t TX_BYTES = A_BYTES + B_BYTES;
    static constexpr int STG_TOTAL = EW * STG_BUFS * STG_BYTES;
    // as many stages as fit next to the epilogue staging (227 KB per CTA)
    static constexpr int STAGES = (232448 - STG_TOTAL - 2048) / (A_BYTES + B_BYTES);
    static constexpr uint32_t TMEM_STRIDE = BN <= 128 ? 128 : 256;  // column offset of buffer 1
    static constexpr uint32_t TMEM_COLS = 2 * TMEM_STRIDE;          // two fp32 accumulators
    static constexpr int SMEM_A = 0;
    static constexpr int SMEM_B = SMEM_A + STAGES * A_BYTES;
    static constexpr int SMEM_C = SMEM_B + STAGES * B_BYTES;
    static constexpr int SMEM_BAR = SMEM_C + STG_TOTAL;
    static constexpr int NUM_BARS = 2 * STAGES + 4 + 1;
    static constexpr int SMEM_MISC = SMEM_BAR + NUM_BARS * 8;
    static constexpr int SMEM_TOTAL = SMEM_MISC + 16 + 1024;  // + alignment slack
    static_assert(SMEM_TOTAL <= 232448, "shared memory budget");
};

__device__ __forceinline__ void tile_coords(const TiledParams &p, int t, int &b, int &mt, int &nt) {
    grouped_tile(t, p.num_m, p.num_n, p.group_m, b, mt, nt);
}

// Debug checks (p.debug): walks this CTA's tiles before any role starts and
// checks that each tile and its coordinates lie inside the problem (with
// p.debug == 2, CTA 0's first tile is moved past the last, which the check
// must catch).  On a failure it records it in the error word and the CTA
// does no work at all.
__device__ __noinline__ bool tiled_sequence_ok(const TiledParams &p) {
    if (p.num_kb < 1) return invariant_failed(p.err, invariant_code(KERNEL_TILED, CHECK_KRANGE));
    for (int t0 = blockIdx.x; t0 < p.tiles; t0 += gridDim.x) {
        const int t = (p.debug == 2 && blockIdx.x == 0 && t0 == 0) ? t0 + p.tiles : t0;
        if (t < 0 || t >= p.tiles)
            return invariant_failed(p.err, invariant_code(KERNEL_TILED, CHECK_TILE));
        int b, mt, nt;
        tile_coords(p, t, b, mt, nt);
        if (b < 0 || b >= p.batch || mt < 0 || mt >= p.num_m || nt < 0 || nt >= p.num_n)
            return invariant_failed(p.err, invariant_code(KERNEL_TILED, CHECK_TILE));
    }
    return true;
}

// F8: 8-bit inputs (kind::f8f6f4), K blocks of 128 elements, both operands
// K-major.
template <int BN, int OUT, bool TMA_STORE, bool EPI, bool F8 = false, int EW = 4>
__global__ void __launch_bounds__(32 * (2 + EW), 1)
    hgemm_tiled_kernel(const __grid_constant__ CUtensorMap tmA,
                       const __grid_constant__ CUtensorMap tmB,
                       const __grid_constant__ CUtensorMap tmC, const TiledParams p) {
    constexpr int BKE = F8 ? 128 : 64;  // elements per K block (128 bytes either way)
    using Cfg = TiledCfg<BN, EW>;
    extern __shared__ uint8_t smem_raw[];
    const uint32_t raw = smem_u32(smem_raw);
    uint8_t *smem = smem_raw + ((1024u - (raw & 1023u)) & 1023u);
    const uint32_t sbase = smem_u32(smem);
    const uint32_t sA = sbase + Cfg::SMEM_A;
    const uint32_t sB = sbase + Cfg::SMEM_B;
    const uint32_t sC = sbase + Cfg::SMEM_C;
    const uint32_t bar0 = sbase + Cfg::SMEM_BAR;
    auto full = [&](int s) { return bar0 + 8u * s; };
    auto empty = [&](int s) { return bar0 + 8u * (Cfg::STAGES + s); };
    auto tfull = [&](int b) { return bar0 + 8u * (2 * Cfg::STAGES + b); };
    auto tempty = [&](int b) { return bar0 + 8u * (2 * Cfg::STAGES + 2 + b); };
    const uint32_t drain = bar0 + 8u * (2 * Cfg::STAGES + 4);
    volatile uint32_t *tmem_slot = reinterpret_cast<volatile uint32_t *>(smem + Cfg::SMEM_MISC);
    volatile int32_t *abort_flag = reinterpret_cast<volatile int32_t *>(smem + Cfg::SMEM_MISC + 4);
    volatile int32_t *skip_all = reinterpret_cast<volatile int32_t *>(smem + Cfg::SMEM_MISC + 8);

    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;

    if (threadIdx.x == 0) {
        for (int s = 0; s < Cfg::STAGES; ++s) {
            mbar_init(full(s), 1);
            mbar_init(empty(s), 1);
        }
        for (int b = 0; b < 2; ++b) {
            mbar_init(tfull(b), 1);
            mbar_init(tempty(b), EW);
        }
        mbar_init(drain, 1);
        *abort_flag = 0;
        *skip_all = p.debug && !tiled_sequence_ok(p) ? 1 : 0;
        fence_mbar_init();
        prefetch_tmap(&tmA);
        prefetch_tmap(&tmB);
        if (TMA_STORE) prefetch_tmap(&tmC);
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
    // first tile of this CTA; past the last when the debug checks failed
    const int t_first = *skip_all ? p.tiles : static_cast<int>(blockIdx.x);
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
            for (int t = t_first; ok && t < p.tiles; t += gridDim.x) {
                int b, mt, nt;
                tile_coords(p, t, b, mt, nt);
                for (int kb = 0; kb < p.num_kb; ++kb) {
                    if (!wait_bounded(empty(stage), phase ^ 1u, wc,
                                      timeout_code(ROLE_PRODUCER, stage))) {
                        ok = false;
                        break;
                    }
                    if (p.withhold_kb && blockIdx.x == 0 && t == 0 && kb == p.withhold_kb - 1) {
                        // Abort-path testing: this stage is never armed or
                        // loaded, so the MMA issuer's wait on full[stage]
                        // expires; it is still counted as issued, and the
                        // teardown's wait on it is bounded as well.
                        ++issued;
                        if (++stage == Cfg::STAGES) {
                            stage = 0;
                            phase ^= 1u;
                        }
                        continue;
                    }
                    mbar_arrive_expect_tx(full(stage), Cfg::TX_BYTES);
                    tma_load_3d(sA + stage * Cfg::A_BYTES, &tmA, full(stage), kb * BKE, mt * BM, b);
                    // 64 x 64 blocks of B: (n, k) MN-major, or (k, n) K-major
                    // when B is stored N x K (the blocks stack into BN rows)
#pragma unroll
                    for (int j = 0; j < Cfg::B_BLOCKS; ++j) {
                        if (p.b_kmajor)
                            tma_load_3d(sB + stage * Cfg::B_BYTES + j * Cfg::B_BLOCK, &tmB,
                                        full(stage), kb * BKE, nt * BN + j * 64, b);
                        else
                            tma_load_3d(sB + stage * Cfg::B_BYTES + j * Cfg::B_BLOCK, &tmB,
                                        full(stage), nt * BN + j * 64, kb * BK, b);
                    }
                    ++issued;
                    if (++stage == Cfg::STAGES) {
                        stage = 0;
                        phase ^= 1u;
                    }
                }
            }
            // Teardown: no TMA write into this CTA's shared memory may still be
            // in flight.  On the normal path these phases completed long ago.
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
            for (int t = t_first; ok && t < p.tiles; t += gridDim.x, ++local) {
                const int buf = local & 1;
                const uint32_t tph = (local >> 1) & 1;
                if (!wait_bounded(tempty(buf), tph ^ 1u, wc, timeout_code(ROLE_MMA, 0x100 + buf))) {
                    ok = false;
                    break;
                }
                tc_fence_after();
                const uint32_t d_tmem = tmem_base + buf * Cfg::TMEM_STRIDE;
                for (int kb = 0; kb < p.num_kb; ++kb) {
                    if (!wait_bounded(full(stage), phase, wc, timeout_code(ROLE_MMA, stage))) {
                        ok = false;
                        break;
                    }
                    tc_fence_after();
                    const uint32_t a0 = sA + stage * Cfg::A_BYTES;
                    const uint32_t b0 = sB + stage * Cfg::B_BYTES;
#pragma unroll
                    for (int k = 0; k < BK / 16; ++k) {
                        const uint64_t ad = sdesc_sw128(a0 + k * 32, 16, 1024);
                        const uint64_t bd = p.b_kmajor
                                                ? sdesc_sw128(b0 + k * 32, 16, 1024)
                                                : sdesc_sw128(b0 + k * 16 * 128, Cfg::B_BLOCK, 1024);
                        if constexpr (F8)
                            umma_f8(d_tmem, ad, bd, p.idesc, (kb | k) != 0 ? 1u : 0u);
                        else
                            umma_f16(d_tmem, ad, bd, p.idesc, (kb | k) != 0 ? 1u : 0u);
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
            // Teardown: every MMA issued has completed before TMEM is freed.
            umma_commit(drain);
            wait_bounded(drain, 0, wc, 0, /*honor_abort=*/false);
        }
    } else {
        // ------------------------------------------------------------ epilogue
        const int q = warp & 3;   // TMEM lane quarter this warp may read
        const int ew = warp - 2;  // staging slot
        const uint32_t stg = sC + ew * STG_BUFS * STG_BYTES;
        // chunks [c_lo, c_hi) of the tile's 32-column chunks are this warp's
        constexpr int NCH = BN / 32;
        const int half = EW == 8 ? ew >> 2 : 0;
        const int c_lo = EW == 8 && half ? (NCH + 1) / 2 : 0;
        const int c_hi = EW == 8 && !half ? (NCH + 1) / 2 : NCH;
        const EpiArgs epi{&tmC, p.C, p.ldc, p.strideC, p.M, p.N, p.ep};
        int sbuf = 0;
        int local = 0;
        for (int t = t_first; t < p.tiles; t += gridDim.x, ++local) {
            int b, mt, nt;
            tile_coords(p, t, b, mt, nt);
            const int buf = local & 1;
            const uint32_t tph = (local >> 1) & 1;
            const int row0 = mt * BM + q * 32;
            const int col0 = nt * BN;
            if constexpr (EPI) prefetch_c_prev<OUT>(epi, row0 + lane, col0 + 32 * c_lo, 32 * (c_hi - c_lo), b);
            if (!wait_bounded_warp(tfull(buf), tph, wc, timeout_code(ROLE_EPILOGUE, buf))) break;
            tc_fence_after();
            const uint32_t tbase =
                tmem_base + (static_cast<uint32_t>(q * 32) << 16) + buf * Cfg::TMEM_STRIDE;
            drain_accumulator<OUT, TMA_STORE, BN, false, EPI>(
                tbase, stg, sbuf, row0, col0, b, epi,
                [&] {
                    if (lane == 0) mbar_arrive(tempty(buf));
                },
                nullptr, c_lo, c_hi);
        }
        if (TMA_STORE && lane == 0) bulk_wait<0>();
    }

    __syncwarp();
    tc_fence_before();
    __syncthreads();
    if (warp == 1) {
        tc_fence_after();
        tmem_dealloc(tmem_base, Cfg::TMEM_COLS);
    }
}

template <int BN, int OUT, bool TS, bool EPI, bool F8 = false, int EW = 4>
cudaError_t launch_impl(const CUtensorMap &tmA, const CUtensorMap &tmB, const CUtensorMap &tmC,
                        const TiledParams &p, int grid, cudaStream_t stream) {
    using Cfg = TiledCfg<BN, EW>;
    auto kern = hgemm_tiled_kernel<BN, OUT, TS, EPI, F8, EW>;
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         Cfg::SMEM_TOTAL);
    if (e != cudaSuccess) return e;
    return launch_dependent(kern, grid, Cfg::THREADS, Cfg::SMEM_TOTAL, stream, tmA, tmB, tmC, p);
}

template <int BN, int OUT>
cudaError_t launch_ts(bool ts, const CUtensorMap &tmA, const CUtensorMap &tmB,
                      const CUtensorMap &tmC, const TiledParams &p, int grid, cudaStream_t s) {
    // p.f8: 8-bit inputs (tile widths 128 and 256 only); p.ep.on: the
    // fused-epilogue variant
    if constexpr (BN == 128 || BN == 256) {
        if (p.f8) {
            if (p.epi_warps != 4) return cudaErrorInvalidValue;
            if (p.ep.on)
                return ts ? launch_impl<BN, OUT, true, true, true>(tmA, tmB, tmC, p, grid, s)
                          : launch_impl<BN, OUT, false, true, true>(tmA, tmB, tmC, p, grid, s);
            return ts ? launch_impl<BN, OUT, true, false, true>(tmA, tmB, tmC, p, grid, s)
                      : launch_impl<BN, OUT, false, false, true>(tmA, tmB, tmC, p, grid, s);
        }
    } else {
        if (p.f8) return cudaErrorInvalidValue;
    }
    if constexpr (BN == 128 || BN == 256) {
        // eight epilogue warps: 16-bit inputs, tile widths 128 and 256
        if (p.epi_warps == 8) {
            if (p.ep.on)
                return ts ? launch_impl<BN, OUT, true, true, false, 8>(tmA, tmB, tmC, p, grid, s)
                          : launch_impl<BN, OUT, false, true, false, 8>(tmA, tmB, tmC, p, grid, s);
            return ts ? launch_impl<BN, OUT, true, false, false, 8>(tmA, tmB, tmC, p, grid, s)
                      : launch_impl<BN, OUT, false, false, false, 8>(tmA, tmB, tmC, p, grid, s);
        }
    }
    if (p.epi_warps != 4) return cudaErrorInvalidValue;
    if (p.ep.on)
        return ts ? launch_impl<BN, OUT, true, true>(tmA, tmB, tmC, p, grid, s)
                  : launch_impl<BN, OUT, false, true>(tmA, tmB, tmC, p, grid, s);
    return ts ? launch_impl<BN, OUT, true, false>(tmA, tmB, tmC, p, grid, s)
              : launch_impl<BN, OUT, false, false>(tmA, tmB, tmC, p, grid, s);
}

template <int BN>
cudaError_t launch_out(int out, bool ts, const CUtensorMap &tmA, const CUtensorMap &tmB,
                       const CUtensorMap &tmC, const TiledParams &p, int grid, cudaStream_t s) {
    switch (out) {
        case OUT_F16: return launch_ts<BN, OUT_F16>(ts, tmA, tmB, tmC, p, grid, s);
        case OUT_BF16: return launch_ts<BN, OUT_BF16>(ts, tmA, tmB, tmC, p, grid, s);
        case OUT_F32: return launch_ts<BN, OUT_F32>(ts, tmA, tmB, tmC, p, grid, s);
        default: return cudaErrorInvalidValue;
    }
}

}  // namespace

int tiled_smem_bytes(int bn, int epi_warps) {
    if (epi_warps == 8) {
        switch (bn) {
            case 128: return TiledCfg<128, 8>::SMEM_TOTAL;
            case 256: return TiledCfg<256, 8>::SMEM_TOTAL;
            default: return 0;
        }
    }
    switch (bn) {
        case 128: return TiledCfg<128>::SMEM_TOTAL;
        case 192: return TiledCfg<192>::SMEM_TOTAL;
        case 224: return TiledCfg<224>::SMEM_TOTAL;
        case 256: return TiledCfg<256>::SMEM_TOTAL;
        default: return 0;
    }
}

int tiled_stages(int bn, int epi_warps) {
    if (epi_warps == 8) {
        switch (bn) {
            case 128: return TiledCfg<128, 8>::STAGES;
            case 256: return TiledCfg<256, 8>::STAGES;
            default: return 0;
        }
    }
    switch (bn) {
        case 128: return TiledCfg<128>::STAGES;
        case 192: return TiledCfg<192>::STAGES;
        case 224: return TiledCfg<224>::STAGES;
        case 256: return TiledCfg<256>::STAGES;
        default: return 0;
    }
}

cudaError_t launch_tiled(int bn, int out, bool tma_store, const CUtensorMap &tmA,
                         const CUtensorMap &tmB, const CUtensorMap &tmC, const TiledParams &p,
                         int grid, cudaStream_t stream) {
    switch (bn) {
        case 128: return launch_out<128>(out, tma_store, tmA, tmB, tmC, p, grid, stream);
        case 192: return launch_out<192>(out, tma_store, tmA, tmB, tmC, p, grid, stream);
        case 224: return launch_out<224>(out, tma_store, tmA, tmB, tmC, p, grid, stream);
        case 256: return launch_out<256>(out, tma_store, tmA, tmB, tmC, p, grid, stream);
        default: return cudaErrorInvalidValue;
    }
}

}  // namespace hg
