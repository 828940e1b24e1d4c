// gemm_pair.cu -- persistent tcgen05 GEMM on CTA pairs (cta_group::2).
//
// Same product as gemm_tiled.cu (C_b = A_b . B_b, row-major, fp16/bf16 in,
// fp32 accumulate), with 256 x 256 output tiles computed by a cluster of two
// CTAs on two SMs.  The even CTA (rank 0, the "leader") issues every MMA;
// one `tcgen05.mma.cta_group::2` (M = 256, N = 256, K = 16) reads rows
// 0..127 of the A tile and columns 0..127 of the B tile from the leader's
// shared memory and rows 128..255 / columns 128..255 from the odd CTA's, and
// leaves rows 0..127 of the accumulator in the leader's TMEM and rows
// 128..255 in the odd CTA's.  Per K block each CTA therefore stages 16 KB of
// A and 16 KB of B -- two thirds of what one CTA computing 128 x 256 on its
// own stages (16 KB + 32 KB) -- which cuts the L2 -> SM traffic per FLOP by a
// third and leaves room for six stages instead of four.  This is the pairing
// "tensor-cores-cutlass-and-cute" section 六.5 shows as a 2 x 1 x 1 cluster
// sharing B (there with TMA multicast and wgmma; here with the pair MMA).
//
// Barriers (all in shared memory, same offsets in both CTAs):
//   full[s]    leader only: armed by the leader's producer with the bytes of
//              BOTH CTAs' stage s (64 KB); each CTA's TMA load counts its
//              bytes on the leader's barrier (.cta_group::2 loads).
//   empty[s]   both CTAs: the leader's MMA thread commits with a multicast to
//              both once the stage's MMAs are done; each producer waits on
//              its own before overwriting its half of the stage.
//   tfull[b]   both CTAs: multicast commit after a tile's last K block.
//   tempty[b]  leader only, 8 arrivals: the 4 epilogue warps of each CTA
//              (the odd CTA's arrive remotely, cluster-scope release).
//   drain      leader only: MMA completion before TMEM is freed.
// Every wait is bounded (watchdog.cuh).  Both CTAs walk the same tile
// sequence, so their loops have equal trip counts, and both end at a
// cluster barrier before TMEM is freed and the CTAs exit (no CTA leaves
// while its peer may still signal it).
#include "kernels.h"
#include "ptx.cuh"
#include "tile_common.cuh"
#include "watchdog.cuh"

namespace hg {
namespace {

constexpr int BM = 128;       // rows per CTA (256 per pair)
constexpr int BK = 64;
constexpr int NUM_THREADS = 192;
constexpr int EPI_WARPS = 4;

// PN = columns per pair tile (256 or 224); each CTA stages PN/2 columns of B
// in two 64-column blocks (the second partly used when PN = 224).
template <int PN>
struct PairCfg {
    static_assert(PN == 256 || PN == 224, "pair tile N");
    static constexpr int BNH = PN / 2;
    static constexpr int B_BLOCKS = (BNH + 63) / 64;
    static constexpr uint32_t A_BYTES = BM * BK * 2;     // 16 KB
    static constexpr uint32_t B_BLOCK = BK * 128;        // 64 k x 64 n
    static constexpr uint32_t B_BYTES = B_BLOCKS * B_BLOCK;  // 16 KB
    static constexpr uint32_t STAGE_BYTES = A_BYTES + B_BYTES;
    static constexpr uint32_t TX_BYTES = 2 * STAGE_BYTES;      // both CTAs
    static constexpr int STG_TOTAL = EPI_WARPS * EPI_STG_BUFS * EPI_STG_BYTES;
    static constexpr int STAGES = (232448 - STG_TOTAL - 2048) / STAGE_BYTES;
    static constexpr uint32_t TMEM_STRIDE = 256;
    static constexpr uint32_t TMEM_COLS = 512;
    static constexpr int SMEM_A = 0;
    static constexpr int SMEM_B = SMEM_A + STAGES * A_BYTES;
    static constexpr int SMEM_C = SMEM_B + STAGES * B_BYTES;
    static constexpr int SMEM_BAR = SMEM_C + STG_TOTAL;
    static constexpr int NUM_BARS = 2 * STAGES + 4 + 1;
    static constexpr int SMEM_MISC = SMEM_BAR + NUM_BARS * 8;
    static constexpr int SMEM_TOTAL = SMEM_MISC + 16 + 1024;
    static_assert(SMEM_TOTAL <= 232448, "shared memory budget");
};

// Work unit u -> tile t and K-block range [kb0, kb1).  `half` is -1 for a
// whole tile, else the K half (0 or 1) of a split tail tile.
__device__ __forceinline__ void pair_unit(const TiledParams &p, int u, int &t, int &kb0, int &kb1,
                                          int &half) {
    if (u < p.full_tiles || p.tail_split == 1) {
        t = u;
        kb0 = 0;
        kb1 = p.num_kb;
        half = -1;
        return;
    }
    const int v = u - p.full_tiles;
    t = p.full_tiles + (v >> 1);
    half = v & 1;
    const int mid = p.num_kb >> 1;
    kb0 = half ? mid : 0;
    kb1 = half ? p.num_kb : mid;
}

// Bounded spin on a global flag set (with release) by another CTA.
__device__ __forceinline__ bool wait_flag_bounded(const int32_t *flag, const WaitCtl &c,
                                                  int32_t code) {
    const uint64_t t0 = globaltimer_ns();
    for (uint32_t it = 0; it < kMaxWaitIterations; ++it) {
        int32_t v;
        asm volatile("ld.acquire.gpu.global.b32 %0, [%1];" : "=r"(v) : "l"(flag) : "memory");
        if (v) return true;
        if (*c.abort_flag) return false;
        if (globaltimer_ns() - t0 > c.timeout_ns) break;
    }
    atomicCAS(c.err, 0, code);
    *c.abort_flag = 1;
    return false;
}

// Bounded wait with cluster-scope acquire (for barriers the peer CTA arrives on).
__device__ __forceinline__ bool wait_bounded_cluster(uint32_t bar, uint32_t parity, const WaitCtl &c,
                                                     int32_t code) {
    if (mbar_try_wait_cluster(bar, parity)) return true;
    const uint64_t t0 = globaltimer_ns();
    for (uint32_t it = 0; it < kMaxWaitIterations; ++it) {
        if (mbar_try_wait_cluster(bar, parity)) return true;
        if (*c.abort_flag) return false;
        if (globaltimer_ns() - t0 > c.timeout_ns) break;
    }
    atomicCAS(c.err, 0, code);
    *c.abort_flag = 1;
    return false;
}

template <int PN, int OUT, bool TMA_STORE>
__global__ void __launch_bounds__(NUM_THREADS, 1)
    hgemm_pair_kernel(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB,
                      const __grid_constant__ CUtensorMap tmC, const TiledParams p) {
    using Cfg = PairCfg<PN>;
    constexpr int BNH = Cfg::BNH;
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

    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    const uint32_t rank = cluster_ctarank();
    const int pair = blockIdx.x >> 1;
    const int npairs = gridDim.x >> 1;

    if (threadIdx.x == 0) {
        for (int s = 0; s < Cfg::STAGES; ++s) {
            mbar_init(full(s), 1);
            mbar_init(empty(s), 1);
        }
        for (int b = 0; b < 2; ++b) {
            mbar_init(tfull(b), 1);
            mbar_init(tempty(b), 2 * EPI_WARPS);
        }
        mbar_init(drain, 1);
        *abort_flag = 0;
        fence_mbar_init();
        prefetch_tmap(&tmA);
        prefetch_tmap(&tmB);
        if (TMA_STORE) prefetch_tmap(&tmC);
    }
    if (warp == 1) {
        tmem_alloc_pair(smem_u32(const_cast<uint32_t *>(tmem_slot)), Cfg::TMEM_COLS);
        tmem_relinquish_pair();
    }
    tc_fence_before();
    cluster_sync();  // barriers of both CTAs initialised, TMEM allocated in both
    tc_fence_after();
    const uint32_t tmem_base = *tmem_slot;
    const WaitCtl wc{abort_flag, p.err, p.timeout_ns};
    // The next kernel of the stream may be scheduled now; it waits for this
    // one to complete before it reads memory (griddep_wait below).
    if (threadIdx.x == 0) griddep_launch_dependents();

    if (warp == 0) {
        // ------------------------------------------------------------ TMA producer (both CTAs)
        if (lane == 0) {
            // Nothing this kernel reads may be read before the previous kernel
            // of the stream has completed (dependent launches).
            griddep_wait();
            int stage = 0;
            uint32_t phase = 0;
            int issued = 0;
            bool ok = true;
            for (int u = pair; ok && u < p.units; u += npairs) {
                int t, kb0, kb1, half;
                pair_unit(p, u, t, kb0, kb1, half);
                int b, mt, nt;
                grouped_tile(t, p.num_m, p.num_n, p.group_m, b, mt, nt);
                const int m0 = mt * (2 * BM) + static_cast<int>(rank) * BM;
                const int n0 = nt * PN + static_cast<int>(rank) * BNH;
                for (int kb = kb0; kb < kb1; ++kb) {
                    if (!wait_bounded(empty(stage), phase ^ 1u, wc,
                                      timeout_code(ROLE_PRODUCER, stage))) {
                        ok = false;
                        break;
                    }
                    const uint32_t fb = mapa_shared(full(stage), 0);  // the leader's full[stage]
                    if (rank == 0) mbar_arrive_expect_tx(full(stage), Cfg::TX_BYTES);
                    tma_load_3d_pair(sA + stage * Cfg::A_BYTES, &tmA, fb, kb * BK, m0, b);
#pragma unroll
                    for (int j = 0; j < Cfg::B_BLOCKS; ++j)
                        tma_load_3d_pair(sB + stage * Cfg::B_BYTES + j * Cfg::B_BLOCK, &tmB, fb,
                                         n0 + j * 64, kb * BK, b);
                    ++issued;
                    if (++stage == Cfg::STAGES) {
                        stage = 0;
                        phase ^= 1u;
                    }
                }
            }
            // Teardown: no TMA write into this CTA's shared memory may still be
            // in flight.  The leader sees its full barriers complete (they count
            // both CTAs' bytes); the odd CTA sees its empty barriers complete
            // (the MMA consumed the stage, so its bytes had landed).
            const int pending = issued < Cfg::STAGES ? issued : Cfg::STAGES;
            for (int i = 0; i < pending; ++i) {
                if (stage == 0) {
                    stage = Cfg::STAGES - 1;
                    phase ^= 1u;
                } else {
                    --stage;
                }
                if (rank == 0)
                    wait_bounded(full(stage), phase, wc, 0, /*honor_abort=*/false);
                else
                    wait_bounded(empty(stage), phase, wc, 0, /*honor_abort=*/false);
            }
        }
    } else if (warp == 1) {
        // ------------------------------------------------------------ MMA issuer (leader)
        if (rank == 0 && lane == 0) {
            int stage = 0;
            uint32_t phase = 0;
            bool ok = true;
            int local = 0;
            for (int u = pair; ok && u < p.units; u += npairs, ++local) {
                int t, kb0, kb1, half;
                pair_unit(p, u, t, kb0, kb1, half);
                const int buf = local & 1;
                const uint32_t tph = (local >> 1) & 1;
                if (!wait_bounded_cluster(tempty(buf), tph ^ 1u, wc,
                                          timeout_code(ROLE_MMA, 0x100 + buf))) {
                    ok = false;
                    break;
                }
                tc_fence_after();
                const uint32_t d_tmem = tmem_base + buf * Cfg::TMEM_STRIDE;
                for (int kb = kb0; kb < kb1; ++kb) {
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
                        const uint64_t bd = sdesc_sw128(b0 + k * 16 * 128, Cfg::B_BLOCK, 1024);
                        umma_f16_pair(d_tmem, ad, bd, p.idesc, (kb > kb0 || k > 0) ? 1u : 0u);
                    }
                    umma_commit_pair(empty(stage), 0x3);
                    if (++stage == Cfg::STAGES) {
                        stage = 0;
                        phase ^= 1u;
                    }
                }
                if (!ok) break;
                umma_commit_pair(tfull(buf), 0x3);
            }
            umma_commit_pair(drain, 0x1);
            wait_bounded(drain, 0, wc, 0, /*honor_abort=*/false);
        }
    } else {
        // ------------------------------------------------------------ epilogue (both CTAs)
        const int q = warp & 3;
        const int ew = warp - 2;
        const uint32_t stg = sC + ew * EPI_STG_BUFS * EPI_STG_BYTES;
        float *stg_f =
            reinterpret_cast<float *>(smem + Cfg::SMEM_C + ew * EPI_STG_BUFS * EPI_STG_BYTES);
        const EpiArgs epi{&tmC, p.C, p.ldc, p.strideC, p.M, p.N};
        int sbuf = 0;
        int local = 0;
        for (int u = pair; u < p.units; u += npairs, ++local) {
            int t, kb0, kb1, half;
            pair_unit(p, u, t, kb0, kb1, half);
            int b, mt, nt;
            grouped_tile(t, p.num_m, p.num_n, p.group_m, b, mt, nt);
            const int buf = local & 1;
            const uint32_t tph = (local >> 1) & 1;
            if (!wait_bounded_warp(tfull(buf), tph, wc, timeout_code(ROLE_EPILOGUE, buf))) break;
            tc_fence_after();
            const uint32_t tbase =
                tmem_base + (static_cast<uint32_t>(q * 32) << 16) + buf * Cfg::TMEM_STRIDE;
            const int row0 = mt * (2 * BM) + static_cast<int>(rank) * BM + q * 32;
            const int col0 = nt * PN;
            const uint32_t release_bar = mapa_shared(tempty(buf), 0);
            auto release = [&] {
                if (lane == 0) mbar_arrive_cluster(release_bar);
            };
            if (half < 0) {
                drain_accumulator<OUT, TMA_STORE, PN>(tbase, stg, stg_f, sbuf, row0, col0, b, epi,
                                                      release);
                continue;
            }
            // Split tail tile: its two K halves run on two pairs at the same
            // time.  Each half owns half of the 32-column chunks of every warp's
            // 32 rows: it spills the chunks the other half owns (fp32) and
            // raises that half's flag, then waits (bounded) for its own flag and
            // stores own + other for the chunks it owns.  Neither side waits
            // before spilling, so both waits end; every output element is one
            // two-term fp32 sum, which commutes, so the result does not depend
            // on which half finishes first.  The reader clears its flag.
            constexpr int NCH = PN / 32;
            constexpr int HCH = (NCH + 1) / 2;  // chunks owned by half 0
            const int slot = ((t - p.full_tiles) * 2 + static_cast<int>(rank)) * EPI_WARPS + q;
            int32_t *flags = p.tail_sync + 2 * slot;          // flags[h]: region of half h ready
            float *region = p.partials + static_cast<int64_t>(slot) * (2 * 4 * 1024);
            const int other = half ^ 1;
            const int own_lo = half ? HCH : 0, own_hi = half ? NCH : HCH;
            const int oth_lo = other ? HCH : 0, oth_hi = other ? NCH : HCH;
            spill_accumulator(tbase, region + other * (4 * 1024), oth_lo, oth_hi);
            __threadfence();
            __syncwarp();
            if (lane == 0)
                asm volatile("st.release.gpu.global.b32 [%0], %1;" ::"l"(flags + other), "r"(1)
                             : "memory");
            int ok = 1;
            if (lane == 0)
                ok = wait_flag_bounded(flags + half, wc, timeout_code(ROLE_EPILOGUE, 0x200 + slot)) ? 1 : 0;
            ok = __shfl_sync(0xFFFFFFFFu, ok, 0);
            __syncwarp();
            if (!ok) {
                tc_fence_before();
                release();
                break;
            }
            drain_accumulator<OUT, TMA_STORE, PN, true>(tbase, stg, stg_f, sbuf, row0, col0, b, epi,
                                                        release, region + half * (4 * 1024),
                                                        own_lo, own_hi);
            if (lane == 0) flags[half] = 0;  // read: ready for the next run
        }
        if (TMA_STORE && lane == 0) bulk_wait<0>();
    }

    __syncwarp();
    tc_fence_before();
    cluster_sync();  // neither CTA frees TMEM or exits while its peer may still signal it
    if (warp == 1) {
        tc_fence_after();
        tmem_dealloc_pair(tmem_base, Cfg::TMEM_COLS);
    }
}

template <int PN, int OUT, bool TS>
cudaError_t launch_impl(const CUtensorMap &tmA, const CUtensorMap &tmB, const CUtensorMap &tmC,
                        const TiledParams &p, int grid, cudaStream_t stream) {
    auto kern = hgemm_pair_kernel<PN, OUT, TS>;
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         PairCfg<PN>::SMEM_TOTAL);
    if (e != cudaSuccess) return e;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(static_cast<unsigned>(grid), 1, 1);
    cfg.blockDim = dim3(NUM_THREADS, 1, 1);
    cfg.dynamicSmemBytes = PairCfg<PN>::SMEM_TOTAL;
    cfg.stream = stream;
    cudaLaunchAttribute attr[2];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = 2;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[1].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 2;
    return cudaLaunchKernelEx(&cfg, kern, tmA, tmB, tmC, p);
}

template <int OUT, bool TS>
int max_pairs_impl() {
    auto kern = hgemm_pair_kernel<256, OUT, TS>;
    if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             PairCfg<256>::SMEM_TOTAL) != cudaSuccess)
        return 0;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(2, 1, 1);
    cfg.blockDim = dim3(NUM_THREADS, 1, 1);
    cfg.dynamicSmemBytes = PairCfg<256>::SMEM_TOTAL;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = 2;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    int n = 0;
    if (cudaOccupancyMaxActiveClusters(&n, kern, &cfg) != cudaSuccess) return 0;
    return n;
}

template <int PN, int OUT>
cudaError_t launch_ts(bool ts, const CUtensorMap &tmA, const CUtensorMap &tmB,
                      const CUtensorMap &tmC, const TiledParams &p, int grid, cudaStream_t s) {
    return ts ? launch_impl<PN, OUT, true>(tmA, tmB, tmC, p, grid, s)
              : launch_impl<PN, OUT, false>(tmA, tmB, tmC, p, grid, s);
}

template <int PN>
cudaError_t launch_out(int out, bool ts, const CUtensorMap &tmA, const CUtensorMap &tmB,
                       const CUtensorMap &tmC, const TiledParams &p, int grid, cudaStream_t s) {
    switch (out) {
        case OUT_F16: return launch_ts<PN, OUT_F16>(ts, tmA, tmB, tmC, p, grid, s);
        case OUT_BF16: return launch_ts<PN, OUT_BF16>(ts, tmA, tmB, tmC, p, grid, s);
        case OUT_F32: return launch_ts<PN, OUT_F32>(ts, tmA, tmB, tmC, p, grid, s);
        default: return cudaErrorInvalidValue;
    }
}

}  // namespace

int pair_stages() { return PairCfg<256>::STAGES; }

int pair_max_active_pairs() { return max_pairs_impl<OUT_BF16, true>(); }

cudaError_t launch_pair(int pn, int out, bool tma_store, const CUtensorMap &tmA,
                        const CUtensorMap &tmB, const CUtensorMap &tmC, const TiledParams &p,
                        int grid, cudaStream_t stream) {
    if (pn == 256) return launch_out<256>(out, tma_store, tmA, tmB, tmC, p, grid, stream);
    if (pn == 224) return launch_out<224>(out, tma_store, tmA, tmB, tmC, p, grid, stream);
    return cudaErrorInvalidValue;
}

}  // namespace hg
