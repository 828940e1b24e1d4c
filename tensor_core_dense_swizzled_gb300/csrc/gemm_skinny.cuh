#pragma once
// gemm_skinny.cuh -- the HBM-bound path for decode-shaped GEMMs (small M):
// the kernel template and its launchers, instantiated per output type by
// gemm_skinny_f16.cu, gemm_skinny_bf16.cu and gemm_skinny_f32.cu.
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
//   * a work unit covers NB x 64 consecutive columns of C (NT = ceil(NB / 2)
//     MMAs of 128 columns per 16-deep K step), so every K row of B is read in
//     runs of NB x 128 contiguous bytes.  With NB odd the last MMA's upper 64
//     rows read whatever follows the stage in shared memory and are never
//     stored: the tensor core is idle on this path anyway, and 192-column
//     units put 150 CTAs on 8 x 28672 (as cuBLAS does on GB300, grid 150
//     of 192 x 8 tiles) where 256-column units leave 40 SMs idle;
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

template <int NU, int NB>
struct SkinnyCfg {
    static_assert(NU == 16 || NU == 32, "padded M");
    static_assert(NB == 2 || NB == 3 || NB == 4 || NB == 6 || NB == 8, "64-column blocks per unit");
    static constexpr int NT = (NB + 1) / 2;          // 128-column MMAs per K step
    static constexpr int W_BLOCKS = NB;              // 64-column blocks of B per stage
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

// Stores the final value of C[m][n] (element idx of C), through the fused
// epilogue when it is on.
template <int OUT, bool EPI>
__device__ __forceinline__ void store_epi(const SkinnyParams &p, int64_t idx, int m, int n, float acc) {
    if constexpr (EPI) {
        const EpiParams &ep = p.ep;
        const float rs = ep.row_scale ? __ldg(ep.row_scale + m) : 1.f;
        const float cs = ep.col_scale ? __ldg(ep.col_scale + n) : 1.f;
        const float bias = ep.bias ? __ldg(ep.bias + n) : 0.f;
        const float prev = ep.beta != 0.f ? load_one<OUT>(p.C, idx) : 0.f;
        acc = epi_value(ep, acc, rs, cs, bias, prev);
    }
    store_one<OUT>(p.C, idx, acc);
}

// One piece of a CTA's work: K blocks [kb0, kb1) of column tile nt of batch
// b.  The tile's K range is cut into nseg pieces; this is piece seg (pieces
// are numbered in K order, and partials are summed in that order).
struct SkPiece {
    int b, nt, kb0, kb1, seg, nseg;
};

// The sequence of pieces a CTA runs (the producer, the MMA issuer and the
// epilogue walk the same sequence).  Split mode: units blockIdx.x,
// + gridDim.x, ...; unit (b, s, nt) is K split s of tile nt.  Deal mode
// (p.deal): the steps are dealt in equal contiguous ranges, step order
// (batch, tile, K block) with the K block fastest.
struct SkinnySched {
    int u, s, s_end, q, r;
    __device__ __forceinline__ explicit SkinnySched(const SkinnyParams &p) {
        u = blockIdx.x;
        s = s_end = q = r = 0;
        if (p.deal) {
            const int total = p.batch * p.num_tiles * p.num_kb;
            const int c = blockIdx.x, g = gridDim.x;
            q = total / g;  // >= 1: the grid is at most the number of steps
            r = total % g;
            s = c * q + min(c, r);
            s_end = s + q + (c < r ? 1 : 0);
        }
    }
    // CTA whose range holds step `step` (ranges of q + 1 steps, then of q).
    __device__ __forceinline__ int owner(int step) const {
        const int big = r * (q + 1);
        return step < big ? step / (q + 1) : r + (step - big) / q;
    }
    __device__ __forceinline__ bool next(const SkinnyParams &p, SkPiece &w) {
        if (p.deal) {
            if (s >= s_end) return false;
            const int g = s / p.num_kb;
            w.kb0 = s - g * p.num_kb;
            w.kb1 = min(p.num_kb, w.kb0 + (s_end - s));
            s += w.kb1 - w.kb0;
            w.b = g / p.num_tiles;
            w.nt = g - w.b * p.num_tiles;
            const int first = owner(g * p.num_kb);
            w.seg = owner(g * p.num_kb + w.kb0) - first;
            w.nseg = owner(g * p.num_kb + p.num_kb - 1) - first + 1;
            return true;
        }
        if (u >= p.units) return false;
        int sidx;
        unit_coords(p, u, w.b, sidx, w.nt);
        w.kb0 = sidx * p.kb_per_split;
        w.kb1 = min(p.num_kb, w.kb0 + p.kb_per_split);
        w.seg = sidx;
        w.nseg = p.split;
        u += gridDim.x;
        return true;
    }
};

// Debug checks (p.debug): walks this CTA's whole piece sequence before any
// role starts and checks that every piece's batch entry, column tile, K range
// and segment lie inside the problem (with p.debug == 2, CTA 0's first piece
// is moved past the last column tile, which the check must catch).  On a
// failure it records it in the error word and the CTA does no work at all.
__device__ __noinline__ bool skinny_sequence_ok(const SkinnyParams &p) {
    SkinnySched sched(p);
    SkPiece w;
    bool first = true;
    while (sched.next(p, w)) {
        if (p.debug == 2 && first && blockIdx.x == 0) w.nt += p.num_tiles;
        first = false;
        if (w.b < 0 || w.b >= p.batch || w.nt < 0 || w.nt >= p.num_tiles)
            return invariant_failed(p.err, invariant_code(KERNEL_SKINNY, CHECK_TILE));
        if (w.kb0 < 0 || w.kb0 >= w.kb1 || w.kb1 > p.num_kb)
            return invariant_failed(p.err, invariant_code(KERNEL_SKINNY, CHECK_KRANGE));
        if (w.seg < 0 || w.seg >= w.nseg || w.nseg > p.split)
            return invariant_failed(p.err, invariant_code(KERNEL_SKINNY, CHECK_PIECE));
    }
    return true;
}

// F8: 8-bit inputs (kind::f8f6f4), K blocks of 128 elements, both operands
// K-major.
template <int NU, int NB, int OUT, bool EPI, bool F8 = false>
__global__ void __launch_bounds__(NUM_THREADS, 1)
    hgemm_skinny_kernel(const __grid_constant__ CUtensorMap tmX,
                        const __grid_constant__ CUtensorMap tmW, const SkinnyParams p) {
    constexpr int BKE = F8 ? 128 : 64;  // elements per K block (128 bytes either way)
    using Cfg = SkinnyCfg<NU, NB>;
    constexpr int NT = Cfg::NT;
    constexpr int UW = NB * 64;  // columns of C per work unit
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
            mbar_init(tempty(b), EPI_WARPS);
        }
        mbar_init(drain, 1);
        *abort_flag = 0;
        *skip_all = p.debug && !skinny_sequence_ok(p) ? 1 : 0;
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
    const bool run = *skip_all == 0;
    // The next kernel of the stream may be scheduled now; it waits for this
    // one to complete before it reads memory (griddep_wait below).
    if (threadIdx.x == 0) griddep_launch_dependents();

    if (warp == 0) {
        // ------------------------------------------------------------ TMA producer
        if (lane == 0) {
            // Ask L2 for this CTA's first p.prefetch stages of B while the
            // previous kernel of the stream may still run (a dependent launch
            // starts on SMs the previous kernel has left): the ramp of this
            // kernel then overlaps the previous one's last CTAs, when DRAM is
            // under-used.  L2 is where the GPU's memory is coherent, so data
            // the previous kernel still writes is not read stale: nothing
            // reaches shared memory before griddep_wait.
            {
                SkinnySched pre(p);
                SkPiece w;
                int n = 0;
                while (n < p.prefetch && pre.next(p, w)) {
                    for (int kb = w.kb0; kb < w.kb1 && n < p.prefetch; ++kb, ++n)
                        for (int j = 0; j < Cfg::W_BLOCKS; ++j)
                            if (p.b_kmajor)
                                tma_prefetch_3d(&tmW, kb * BKE, w.nt * UW + j * 64, w.b);
                            else
                                tma_prefetch_3d(&tmW, w.nt * UW + j * 64, kb * BK, w.b);
                }
            }
            // Nothing this kernel reads may reach shared memory before the
            // previous kernel of the stream has completed (dependent launches).
            griddep_wait();
            int stage = 0;
            uint32_t phase = 0;
            int issued = 0;
            bool ok = run;
            SkinnySched sched(p);
            SkPiece w;
            while (ok && sched.next(p, w)) {
                const int b = w.b, nt = w.nt;
                for (int kb = w.kb0; kb < w.kb1; ++kb) {
                    if (!wait_bounded(empty(stage), phase ^ 1u, wc,
                                      timeout_code(ROLE_PRODUCER, stage))) {
                        ok = false;
                        break;
                    }
                    if (p.b_kmajor && kb + 1 < w.kb1) {
                        // B stored N x K: a stage holds 128 bytes of each of
                        // UW rows.  Two stages are filled together, row block
                        // by row block, so that the two 128-byte pieces of a
                        // row are requested back to back (DRAM serves them
                        // from one open row).  On 8 x 28672 x 4096 bf16 this
                        // took 44.1 us to 40.7 us; groups of three stages
                        // measured 42.0 us.
                        const int stage2 = stage + 1 == Cfg::STAGES ? 0 : stage + 1;
                        const uint32_t phase2 = stage + 1 == Cfg::STAGES ? phase ^ 1u : phase;
                        if (!wait_bounded(empty(stage2), phase2 ^ 1u, wc,
                                          timeout_code(ROLE_PRODUCER, stage2))) {
                            ok = false;
                            break;
                        }
                        mbar_arrive_expect_tx(full(stage), Cfg::TX_BYTES);
                        mbar_arrive_expect_tx(full(stage2), Cfg::TX_BYTES);
#pragma unroll
                        for (int j = 0; j < Cfg::W_BLOCKS; ++j) {
                            tma_load_3d(sW + stage * Cfg::W_BYTES + j * Cfg::W_BLOCK, &tmW, full(stage),
                                        kb * BKE, nt * UW + j * 64, b);
                            tma_load_3d(sW + stage2 * Cfg::W_BYTES + j * Cfg::W_BLOCK, &tmW, full(stage2),
                                        (kb + 1) * BKE, nt * UW + j * 64, b);
                        }
                        tma_load_3d(sX + stage * Cfg::X_BYTES, &tmX, full(stage), kb * BKE, 0, b);
                        tma_load_3d(sX + stage2 * Cfg::X_BYTES, &tmX, full(stage2), (kb + 1) * BKE, 0, b);
                        issued += 2;
                        ++kb;
                        stage = stage2;
                        phase = phase2;
                        if (++stage == Cfg::STAGES) {
                            stage = 0;
                            phase ^= 1u;
                        }
                        continue;
                    }
                    mbar_arrive_expect_tx(full(stage), Cfg::TX_BYTES);
#pragma unroll
                    for (int j = 0; j < Cfg::W_BLOCKS; ++j) {
                        // 64 x 64 blocks of B: (n, k) MN-major, or (k, n) when B is
                        // stored N x K (blocks stack into rows = columns of C)
                        if (p.b_kmajor)
                            tma_load_3d(sW + stage * Cfg::W_BYTES + j * Cfg::W_BLOCK, &tmW,
                                        full(stage), kb * BKE, nt * UW + j * 64, b);
                        else
                            tma_load_3d(sW + stage * Cfg::W_BYTES + j * Cfg::W_BLOCK, &tmW,
                                        full(stage), nt * UW + j * 64, kb * BK, b);
                    }
                    tma_load_3d(sX + stage * Cfg::X_BYTES, &tmX, full(stage), kb * BKE, 0, b);
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
            bool ok = run;
            int local = 0;
            SkinnySched sched(p);
            SkPiece w;
            for (; ok && sched.next(p, w); ++local) {
                const int kb0 = w.kb0, kb1 = w.kb1;
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
                            // (with NB odd, the last one's upper 64 columns are
                            // the shared memory after the stage: never stored)
                            const uint64_t ad =
                                p.b_kmajor
                                    ? sdesc_sw128(w0 + 2 * j * Cfg::W_BLOCK + k * 32, 16, 1024)
                                    : sdesc_sw128(w0 + 2 * j * Cfg::W_BLOCK + k * 16 * 128,
                                                  Cfg::W_BLOCK, 1024);
                            if constexpr (F8)
                                umma_f8(d0 + j * NU, ad, bd, p.idesc, (kb > kb0 || k > 0) ? 1u : 0u);
                            else
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
        const int num_sub = p.num_tiles * NT;  // 128-column sub-tiles: NT per unit
        SkinnySched sched(p);
        SkPiece w;
        for (; run && sched.next(p, w); ++local) {
            const int b = w.b, nt = w.nt;
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
                const int col0 = nt * UW + j * TN;  // first column of sub-tile j
                if (col0 >= p.N) break;             // sub-tile entirely past N (warp-uniform)
                const int sub = nt * NT + j;
                const int n = col0 + nl;
                // the column is in this unit and in C (with NB odd, the last
                // sub-tile holds 64 columns of the unit)
                const bool in = (j * TN + nl < UW) && n < p.N;
                if (w.nseg == 1) {
                    if (in) {
#pragma unroll
                        for (int m = 0; m < NU; ++m)
                            if (m < p.M)
                                store_epi<OUT, EPI>(p, cbase + static_cast<int64_t>(m) * p.ldc + n, m, n,
                                               __uint_as_float(v[j][m]));
                    }
                    continue;
                }
                const int64_t ctr = (static_cast<int64_t>(b) * num_sub + sub) * EPI_WARPS + q;
                float *part = p.partials +
                              ((static_cast<int64_t>(b) * p.split + w.seg) * num_sub + sub) *
                                  (static_cast<int64_t>(NU) * TN);
#pragma unroll
                for (int m = 0; m < NU; ++m) __stcg(part + m * TN + nl, __uint_as_float(v[j][m]));
                __threadfence();
                __syncwarp();
                int last = 0;
                if (lane == 0) last = (atomicAdd(p.counters + ctr, 1) == w.nseg - 1) ? 1 : 0;
                last = __shfl_sync(0xFFFFFFFFu, last, 0);
                if (last) {
                    __threadfence();
                    const int64_t stride_split = static_cast<int64_t>(num_sub) * NU * TN;
                    const float *p0 = p.partials +
                                      (static_cast<int64_t>(b) * p.split * num_sub + sub) * (NU * TN);
                    if (in) {
                        // Sum in split order 0, 1, ... (deterministic).  The NU
                        // rows of one split are independent loads issued
                        // together, so the fixup costs one L2 round trip per
                        // split (row by row it was NU x split dependent round
                        // trips, which outlasted the next unit's main loop).
                        float acc[NU];
#pragma unroll
                        for (int m = 0; m < NU; ++m) acc[m] = 0.f;
                        for (int ss = 0; ss < w.nseg; ++ss) {
                            const float *ps = p0 + ss * stride_split + nl;
                            float t[NU];
#pragma unroll
                            for (int m = 0; m < NU; ++m)
                                t[m] = (m < p.M) ? __ldcg(ps + m * TN) : 0.f;
#pragma unroll
                            for (int m = 0; m < NU; ++m) acc[m] += t[m];
                        }
#pragma unroll
                        for (int m = 0; m < NU; ++m)
                            if (m < p.M)
                                store_epi<OUT, EPI>(p, cbase + static_cast<int64_t>(m) * p.ldc + n, m, n,
                                               acc[m]);
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

template <int NU, int NB, int OUT, bool EPI, bool F8 = false>
cudaError_t launch_impl(const CUtensorMap &tmX, const CUtensorMap &tmW, const SkinnyParams &p,
                        int grid, cudaStream_t stream) {
    auto kern = hgemm_skinny_kernel<NU, NB, OUT, EPI, F8>;
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         SkinnyCfg<NU, NB>::SMEM_TOTAL);
    if (e != cudaSuccess) return e;
    return launch_dependent(kern, grid, NUM_THREADS, SkinnyCfg<NU, NB>::SMEM_TOTAL, stream, tmX,
                            tmW, p);
}

template <int NU, int NB, int OUT>
cudaError_t launch_epi(const CUtensorMap &tmX, const CUtensorMap &tmW, const SkinnyParams &p,
                       int grid, cudaStream_t s) {
    if constexpr (NB == 2 || NB == 4) {  // 8-bit inputs: 128- and 256-column units
        if (p.f8)
            return p.ep.on ? launch_impl<NU, NB, OUT, true, true>(tmX, tmW, p, grid, s)
                           : launch_impl<NU, NB, OUT, false, true>(tmX, tmW, p, grid, s);
    } else {
        if (p.f8) return cudaErrorInvalidValue;
    }
    return p.ep.on ? launch_impl<NU, NB, OUT, true>(tmX, tmW, p, grid, s)
                   : launch_impl<NU, NB, OUT, false>(tmX, tmW, p, grid, s);
}

template <int NU, int OUT>
cudaError_t launch_nb(int nb, const CUtensorMap &tmX, const CUtensorMap &tmW,
                      const SkinnyParams &p, int grid, cudaStream_t s) {
    switch (nb) {
        case 2: return launch_epi<NU, 2, OUT>(tmX, tmW, p, grid, s);
        case 3: return launch_epi<NU, 3, OUT>(tmX, tmW, p, grid, s);
        case 4: return launch_epi<NU, 4, OUT>(tmX, tmW, p, grid, s);
        case 6: return launch_epi<NU, 6, OUT>(tmX, tmW, p, grid, s);
        case 8: return launch_epi<NU, 8, OUT>(tmX, tmW, p, grid, s);
        default: return cudaErrorInvalidValue;
    }
}

// All variants of one output type; each output type is instantiated in its
// own translation unit (gemm_skinny_f16.cu, ...) so that they compile in
// parallel.
template <int OUT>
cudaError_t launch_skinny_typed(int nu, int nb, const CUtensorMap &tmX, const CUtensorMap &tmW,
                                const SkinnyParams &p, int grid, cudaStream_t s) {
    if (nu == 16) return launch_nb<16, OUT>(nb, tmX, tmW, p, grid, s);
    if (nu == 32) return launch_nb<32, OUT>(nb, tmX, tmW, p, grid, s);
    return cudaErrorInvalidValue;
}

template <int NU>
int stages_nb(int nb) {
    switch (nb) {
        case 2: return SkinnyCfg<NU, 2>::STAGES;
        case 3: return SkinnyCfg<NU, 3>::STAGES;
        case 4: return SkinnyCfg<NU, 4>::STAGES;
        case 6: return SkinnyCfg<NU, 6>::STAGES;
        case 8: return SkinnyCfg<NU, 8>::STAGES;
        default: return 0;
    }
}

}  // namespace

cudaError_t launch_skinny_f16(int nu, int nb, const CUtensorMap &tmX, const CUtensorMap &tmW,
                              const SkinnyParams &p, int grid, cudaStream_t s);
cudaError_t launch_skinny_bf16(int nu, int nb, const CUtensorMap &tmX, const CUtensorMap &tmW,
                               const SkinnyParams &p, int grid, cudaStream_t s);
cudaError_t launch_skinny_f32(int nu, int nb, const CUtensorMap &tmX, const CUtensorMap &tmW,
                              const SkinnyParams &p, int grid, cudaStream_t s);

}  // namespace hg
