#pragma once
// gemm_pair.cuh -- persistent tcgen05 GEMM on CTA pairs (cta_group::2): the
// kernel template and its launchers, instantiated per output type by
// gemm_pair_f16.cu, gemm_pair_bf16.cu and gemm_pair_f32.cu.
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
//   empty[s]   both CTAs: the leader's MMA thread commits to each CTA's
//              barrier (two point-to-point commits) once the stage's MMAs
//              are done; each producer waits on its own before overwriting
//              its half of the stage.
//   tfull[b]   both CTAs: the same two commits after a tile's last K block.
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
// KS = 64-wide K blocks per pipeline stage.  One thread issues every MMA of
// the pair, and each stage costs it a barrier wait and a commit on top of
// its 4 x KS MMAs; with KS = 1 that overhead (about 240 of 576 cycles per
// stage, measured on GB300) left the tensor pipe idle about 11 % of the
// time, so stages hold two K blocks: 3 stages of 64 KB per CTA, the same
// bytes in flight as 6 of 32 KB.
template <int PN, int KS>
struct PairCfg {
    static_assert(PN == 256 || PN == 224, "pair tile N");
    static_assert(KS == 1 || KS == 2, "K blocks per stage");
    static constexpr int BNH = PN / 2;
    static constexpr int B_BLOCKS = (BNH + 63) / 64;
    static constexpr uint32_t A_SUB = BM * BK * 2;            // 16 KB per K block
    static constexpr uint32_t B_BLOCK = BK * 128;             // 64 k x 64 n
    static constexpr uint32_t B_SUB = B_BLOCKS * B_BLOCK;     // 16 KB per K block
    static constexpr uint32_t A_BYTES = KS * A_SUB;
    static constexpr uint32_t B_BYTES = KS * B_SUB;
    // B of a stage: 64-column block j holds its KS x 64 K rows contiguously
    // (128-byte rows), block j at j * B_COLS -- the order a 4-D box
    // (64 n, KS x 64 k, B_BLOCKS) lands in; K block s of block j is at
    // j * B_COLS + s * B_BLOCK.
    static constexpr uint32_t B_COLS = KS * B_BLOCK;
    static constexpr uint32_t SUB_BYTES = A_SUB + B_SUB;
    static constexpr uint32_t STAGE_BYTES = A_BYTES + B_BYTES;
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

// One piece of a pair's work: K steps [ks0, ks1) of tile t, and what the
// epilogue does with the accumulator.
enum PieceRole : int {
    PIECE_WHOLE = -1,  // the whole K range: store C
    PIECE_HALF0 = 0,   // K half 0 / 1 of a split tail tile; the other half runs
    PIECE_HALF1 = 1,   //   on another pair at the same time (symmetric exchange)
    PIECE_CLOSE = 2,   // stream-K: the first K steps of a tile whose remaining
                       //   steps the next pair ran first; add its partial, store C
    PIECE_SPILL = 3,   // stream-K: the last K steps of a tile; publish the partial
    PIECE_PART = 4,    // first-wave dealing: piece seg of nseg of a tile; publish the
                       //   partial, the last piece to arrive sums them all and stores C
};
struct Piece {
    int t, ks0, ks1, role;
    int slot;       // PIECE_HALF0/1: index of the split tile among the split tiles
    int seg, nseg;  // PIECE_PART
};

// Most pieces a tile dealt in the first wave may be cut into.
constexpr int MAX_SEG = 4;

// The sequence of pieces a pair runs; the producer, the MMA issuer and the
// epilogue of both CTAs walk the same sequence.
//
// Unit mode (p.stream_k == 0): units pair, pair + npairs, ... in raster
// order, so that the pairs of a wave work on neighbouring tiles at the same
// K step and share their operand blocks in L2.  With p.tail_split == 2 the
// T = tiles - full_tiles tiles that do not fill a wave are split in two K
// halves, and those 2T <= pairs half units come FIRST (units 0 .. 2T - 1,
// tiles 0 .. T - 1), the whole tiles T .. tiles - 1 after them.  The two
// halves of a tile run at the same time on two pairs and exchange partials
// through global memory; a release/acquire hand-over between SMs took about
// 4.5 us on GB300, which the first wave hides behind the next whole tile
// (with the halves last it was exposed at the end of the kernel).
// First-wave dealing (p.stream_k == 2): the K steps of tiles 0 ..
// full_tiles - 1 (the tiles that do not fill a wave) are dealt to all pairs
// as contiguous, equal ranges (to one step) and run FIRST; then whole tiles
// full_tiles + pair, + npairs, ...  Every pair gets the same work.  A dealt
// tile cut into pieces on consecutive pairs is combined by its last piece
// to arrive (PIECE_PART: no waiting), while the next whole tiles run.
// Stream-K mode (p.stream_k == 1): whole tiles below p.full_tiles first,
// then the K steps of the last S = tiles -
// full_tiles tiles (pairs <= S < 2 pairs) are dealt to the pairs as
// contiguous, equal ranges (to one step), so every pair ends at the same
// time.  Each range is at least num_ks long, so a tile is cut at most once:
// its last steps are the FIRST piece of the next pair's range (run at the
// start, PIECE_SPILL) and its first steps the LAST piece of this pair's range
// (run at the end, PIECE_CLOSE); the closer finds its partner's partial
// published long before it needs it.  (Dealing all tiles this way spreads
// the pairs over the whole raster at unrelated K steps: 8192^3 ran 14 %
// slower than whole tiles, from L2 misses.)
struct PairSched {
    int u;
    int s, s_end, q, r;
    __device__ __forceinline__ PairSched(const TiledParams &p, int num_ks, int pair, int npairs) {
        u = pair;
        s = s_end = q = r = 0;
        if (p.stream_k) {
            // mode 1: the last tiles - full_tiles tiles; mode 2: tiles
            // 0 .. full_tiles - 1, dealt before the whole tiles
            const int total = (p.stream_k == 2 ? p.full_tiles : p.tiles - p.full_tiles) * num_ks;
            q = total / npairs;
            r = total % npairs;
            s = pair * q + min(pair, r);
            s_end = s + q + (pair < r ? 1 : 0);
            if (p.stream_k == 2) u = p.full_tiles + pair;
        }
    }
    // Pair whose dealt range holds step `step` (ranges of q + 1 steps, then of q).
    __device__ __forceinline__ int owner(int step) const {
        const int big = r * (q + 1);
        return step < big ? step / (q + 1) : r + (step - big) / q;
    }
    __device__ __forceinline__ bool next(const TiledParams &p, int num_ks, int npairs, Piece &w) {
        if (p.stream_k == 2) {
            if (s < s_end) {
                w.t = s / num_ks;
                w.ks0 = s - w.t * num_ks;
                w.ks1 = min(num_ks, w.ks0 + (s_end - s));
                s += w.ks1 - w.ks0;
                if (w.ks0 == 0 && w.ks1 == num_ks) {
                    w.role = PIECE_WHOLE;
                } else {
                    w.role = PIECE_PART;
                    const int first = owner(w.t * num_ks);
                    w.seg = owner(w.t * num_ks + w.ks0) - first;
                    w.nseg = owner(w.t * num_ks + num_ks - 1) - first + 1;
                }
                return true;
            }
            if (u >= p.tiles) return false;
            w.t = u;
            w.ks0 = 0;
            w.ks1 = num_ks;
            w.role = PIECE_WHOLE;
            u += npairs;
            return true;
        }
        if (p.stream_k == 1 && u >= p.full_tiles) {
            if (s >= s_end) return false;
            const int r = s / num_ks;
            w.t = p.full_tiles + r;
            w.ks0 = s - r * num_ks;
            w.ks1 = min(num_ks, w.ks0 + (s_end - s));
            s += w.ks1 - w.ks0;
            w.role = (w.ks0 == 0 && w.ks1 == num_ks) ? PIECE_WHOLE
                     : w.ks0 == 0                    ? PIECE_CLOSE
                                                     : PIECE_SPILL;
            return true;
        }
        if (!p.stream_k && u >= p.units) return false;
        const int halves = (p.stream_k || p.tail_split == 1) ? 0 : p.units - p.full_tiles;  // 2T
        if (u < halves) {
            w.t = u >> 1;
            w.slot = u >> 1;
            w.role = u & 1;
            const int mid = num_ks >> 1;
            w.ks0 = w.role ? mid : 0;
            w.ks1 = w.role ? num_ks : mid;
        } else {
            w.t = u - (halves >> 1);
            w.ks0 = 0;
            w.ks1 = num_ks;
            w.role = PIECE_WHOLE;
        }
        u += npairs;
        return true;
    }
};

// Debug checks (p.debug): walks this CTA's whole piece sequence with the
// schedule's own code, before any role starts, and checks that every piece's
// tile, coordinates, K range and segment lie inside the problem (with
// p.debug == 2, pair 0's first piece is given a tile past the last, which the
// check must catch).  On a failure it records it in the error word and the
// CTA does no work at all.  Checking up front keeps the roles' loops as they
// are: a check inside them cost the kernel 1-3 % on GB300.
__device__ __noinline__ bool pair_sequence_ok(const TiledParams &p, int num_ks, int pair, int npairs) {
    PairSched sched(p, num_ks, pair, npairs);
    Piece w;
    bool first = true;
    while (sched.next(p, num_ks, npairs, w)) {
        if (p.debug == 2 && first && pair == 0) w.t += p.tiles;
        first = false;
        if (w.t < 0 || w.t >= p.tiles)
            return invariant_failed(p.err, invariant_code(KERNEL_PAIR, CHECK_TILE));
        int b, mt, nt;
        grouped_tile(w.t, p.num_m, p.num_n, p.group_m, b, mt, nt);
        if (b < 0 || b >= p.batch || mt < 0 || mt >= p.num_m || nt < 0 || nt >= p.num_n)
            return invariant_failed(p.err, invariant_code(KERNEL_PAIR, CHECK_TILE));
        if (w.ks0 < 0 || w.ks0 >= w.ks1 || w.ks1 > num_ks)
            return invariant_failed(p.err, invariant_code(KERNEL_PAIR, CHECK_KRANGE));
        if (w.role == PIECE_PART && (w.seg < 0 || w.seg >= w.nseg || w.nseg > p.max_seg))
            return invariant_failed(p.err, invariant_code(KERNEL_PAIR, CHECK_PIECE));
    }
    return true;
}

// Bounded spin on a global flag set (with release) by another CTA.  Polls
// with relaxed loads; the fence after the load that sees the flag makes the
// pair an acquire (one fence instead of one per poll).
__device__ __forceinline__ bool wait_flag_bounded(const int32_t *flag, const WaitCtl &c,
                                                  int32_t code) {
    const uint64_t t0 = globaltimer_ns();
    for (uint32_t it = 0; it < kMaxWaitIterations; ++it) {
        int32_t v;
        asm volatile("ld.relaxed.gpu.global.b32 %0, [%1];" : "=r"(v) : "l"(flag) : "memory");
        if (v) {
            asm volatile("fence.acq_rel.gpu;" ::: "memory");
            return true;
        }
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

// F8: 8-bit inputs (kind::f8f6f4), K blocks of 128 elements (the same 128
// bytes per staged row), both operands K-major.
template <int PN, int KS, int OUT, bool TMA_STORE, bool EPI, bool F8 = false>
__global__ void __launch_bounds__(NUM_THREADS, 1)
    hgemm_pair_kernel(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB,
                      const __grid_constant__ CUtensorMap tmC, const TiledParams p) {
    constexpr int BKE = F8 ? 128 : 64;  // elements per K block (128 bytes either way)
    using Cfg = PairCfg<PN, KS>;
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
    volatile int32_t *skip_all = reinterpret_cast<volatile int32_t *>(smem + Cfg::SMEM_MISC + 8);

    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    const uint32_t rank = cluster_ctarank();
    const int pair = blockIdx.x >> 1;
    const int npairs = gridDim.x >> 1;
    const int num_ks = (p.num_kb + KS - 1) / KS;  // pipeline steps per tile

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
        *skip_all = p.debug && !pair_sequence_ok(p, num_ks, pair, npairs) ? 1 : 0;
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
    const bool run = *skip_all == 0;  // both CTAs of a pair walk the same pieces: same answer
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
            bool ok = run;
            PairSched sched(p, num_ks, pair, npairs);
            Piece w;
            while (ok && sched.next(p, num_ks, npairs, w)) {
                int b, mt, nt;
                grouped_tile(w.t, p.num_m, p.num_n, p.group_m, b, mt, nt);
                const int m0 = mt * (2 * BM) + static_cast<int>(rank) * BM;
                const int n0 = nt * PN + static_cast<int>(rank) * BNH;
                for (int ks = w.ks0; ks < w.ks1; ++ks) {
                    if (!wait_bounded(empty(stage), phase ^ 1u, wc,
                                      timeout_code(ROLE_PRODUCER, stage))) {
                        ok = false;
                        break;
                    }
                    const uint32_t fb = mapa_shared(full(stage), 0);  // the leader's full[stage]
                    const uint32_t dA = sA + stage * Cfg::A_BYTES;
                    const uint32_t dB = sB + stage * Cfg::B_BYTES;
                    if (p.wide_boxes) {
                        // One copy per operand (each TMA instruction costs the
                        // issuing thread ~90 cycles, which adds to the stage's
                        // latency).  The boxes are whole even past the last K
                        // block (zero-filled), so the bytes are the stage's.
                        if (rank == 0) mbar_arrive_expect_tx(full(stage), 2u * Cfg::STAGE_BYTES);
                        tma_load_4d_pair(dA, &tmA, fb, 0, m0, ks * KS, b);
                        if (p.b_kmajor)  // B stored N x K: the same view as A's
                            tma_load_4d_pair(dB, &tmB, fb, 0, n0, ks * KS, b);
                        else
                            tma_load_4d_pair(dB, &tmB, fb, 0, ks * KS * BK, n0 / 64, b);
                    } else {
                        // K blocks of this step that exist (the last step of an
                        // odd count has one); the leader arms for both CTAs' bytes.
                        const int nsub = min(KS, p.num_kb - ks * KS);
                        if (rank == 0)
                            mbar_arrive_expect_tx(full(stage), 2u * nsub * Cfg::SUB_BYTES);
#pragma unroll
                        for (int s = 0; s < KS; ++s) {
                            if (s >= nsub) break;
                            const int kb = ks * KS + s;
                            tma_load_3d_pair(dA + s * Cfg::A_SUB, &tmA, fb, kb * BKE, m0, b);
                            if (p.b_kmajor) {
                                // K-major: 64-row blocks j of K block s stacked, so
                                // the CTA's 128 rows of B are contiguous
#pragma unroll
                                for (int j = 0; j < Cfg::B_BLOCKS; ++j)
                                    tma_load_3d_pair(dB + s * Cfg::B_SUB + j * Cfg::B_BLOCK, &tmB, fb,
                                                     kb * BKE, n0 + j * 64, b);
                            } else {
#pragma unroll
                                for (int j = 0; j < Cfg::B_BLOCKS; ++j)
                                    tma_load_3d_pair(dB + j * Cfg::B_COLS + s * Cfg::B_BLOCK, &tmB,
                                                     fb, n0 + j * 64, kb * BK, b);
                            }
                        }
                    }
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
            bool ok = run;
            int local = 0;
            // Completion signals go to each CTA's barrier by its cluster
            // address: the barriers sit at the same offsets in both CTAs, so
            // one mapa per CTA of the barrier block gives them all.
            const uint32_t own_bars = mapa_shared(bar0, 0);
            const uint32_t peer_bars = mapa_shared(bar0, 1);
            auto commit_both = [&](uint32_t bar) {
                umma_commit_pair_to(own_bars + (bar - bar0));
                umma_commit_pair_to(peer_bars + (bar - bar0));
            };
            PairSched sched(p, num_ks, pair, npairs);
            Piece w;
            for (; ok && sched.next(p, num_ks, npairs, w); ++local) {
                const int ks0 = w.ks0, ks1 = w.ks1;
                const int buf = local & 1;
                const uint32_t tph = (local >> 1) & 1;
                if (!wait_bounded_cluster(tempty(buf), tph ^ 1u, wc,
                                          timeout_code(ROLE_MMA, 0x100 + buf))) {
                    ok = false;
                    break;
                }
                tc_fence_after();
                const uint32_t d_tmem = tmem_base + buf * Cfg::TMEM_STRIDE;
                const uint64_t adesc0 = sdesc_sw128(sA, 16, 1024);
                // B MN-major: 64-column blocks B_COLS apart, 2 KB per 16 K rows;
                // K-major (stored N x K): rows of 128 bytes, 32 bytes per 16 K
                const bool bk = p.b_kmajor != 0;
                const uint64_t bdesc0 =
                    bk ? sdesc_sw128(sB, 16, 1024) : sdesc_sw128(sB, Cfg::B_COLS, 1024);
                for (int ks = ks0; ks < ks1; ++ks) {
                    if (!wait_bounded(full(stage), phase, wc, timeout_code(ROLE_MMA, stage))) {
                        ok = false;
                        break;
                    }
                    tc_fence_after();
                    const int nsub = min(KS, p.num_kb - ks * KS);
                    // Descriptors: those of stage 0 plus the byte offset / 16 in
                    // the start-address field (shared-memory offsets stay below
                    // 256 KB, so the add cannot carry out of the field).  One
                    // thread issues every MMA; rebuilding each descriptor cost
                    // it more than the MMA's own issue.
                    const uint64_t a_st = adesc0 + ((stage * Cfg::A_BYTES) >> 4);
                    const uint64_t b_st = bdesc0 + ((stage * Cfg::B_BYTES) >> 4);
                    const uint32_t acc0 = ks > ks0 ? 1u : 0u;
#pragma unroll
                    for (int s = 0; s < KS; ++s) {
                        if (s >= nsub) break;
#pragma unroll
                        for (int k = 0; k < BK / 16; ++k) {
                            const uint64_t ad = a_st + ((s * Cfg::A_SUB + k * 32) >> 4);
                            const uint64_t bd =
                                b_st + (bk ? ((s * Cfg::B_SUB + k * 32) >> 4)
                                           : ((s * Cfg::B_BLOCK + k * 16 * 128) >> 4));
                            if constexpr (F8)
                                umma_f8_pair(d_tmem, ad, bd, p.idesc, (s > 0 || k > 0) ? 1u : acc0);
                            else
                                umma_f16_pair(d_tmem, ad, bd, p.idesc, (s > 0 || k > 0) ? 1u : acc0);
                        }
                    }
                    commit_both(empty(stage));
                    if (++stage == Cfg::STAGES) {
                        stage = 0;
                        phase ^= 1u;
                    }
                }
                if (!ok) break;
                commit_both(tfull(buf));
            }
            umma_commit_pair_to(own_bars + (drain - bar0));
            wait_bounded(drain, 0, wc, 0, /*honor_abort=*/false);
        }
    } else {
        // ------------------------------------------------------------ epilogue (both CTAs)
        const int q = warp & 3;
        const int ew = warp - 2;
        const uint32_t stg = sC + ew * EPI_STG_BUFS * EPI_STG_BYTES;
        const EpiArgs epi{&tmC, p.C, p.ldc, p.strideC, p.M, p.N, p.ep};
        int sbuf = 0;
        int local = 0;
        constexpr int NCH = PN / 32;  // 32-column chunks of a warp's accumulator rows
        PairSched sched(p, num_ks, pair, npairs);
        Piece w;
        while (run && sched.next(p, num_ks, npairs, w)) {
            const int t = w.t;
            int b, mt, nt;
            grouped_tile(t, p.num_m, p.num_n, p.group_m, b, mt, nt);
            const int buf = local & 1;
            const uint32_t tph = (local >> 1) & 1;
            ++local;
            const int row0 = mt * (2 * BM) + static_cast<int>(rank) * BM + q * 32;
            const int col0 = nt * PN;
            if constexpr (EPI) prefetch_c_prev<OUT>(epi, row0 + lane, col0, PN, b);
            if (!wait_bounded_warp(tfull(buf), tph, wc, timeout_code(ROLE_EPILOGUE, buf))) break;
            tc_fence_after();
            const uint32_t tbase =
                tmem_base + (static_cast<uint32_t>(q * 32) << 16) + buf * Cfg::TMEM_STRIDE;
            const uint32_t release_bar = mapa_shared(tempty(buf), 0);
            auto release = [&] {
                if (lane == 0) mbar_arrive_cluster(release_bar);
            };
            if (w.role == PIECE_WHOLE) {
                drain_accumulator<OUT, TMA_STORE, PN, false, EPI>(tbase, stg, sbuf, row0, col0, b, epi,
                                                      release);
                continue;
            }
            if (w.role == PIECE_PART) {
                // First-wave dealing: every piece publishes its fp32 partial
                // (layout [tile][seg][CTA][warp][NCH chunks]) and counts itself
                // on the (tile, CTA, warp) counter with an acquire-release
                // atomic; the piece that arrives last sums the nseg partials in
                // segment order and stores C.  Nothing waits for anything.
                const int cidx = (w.t * 2 + static_cast<int>(rank)) * EPI_WARPS + q;
                int32_t *ctr = p.tail_sync + cidx;
                const int64_t seg_stride = static_cast<int64_t>(2 * EPI_WARPS) * NCH * 1024;
                const float *parts =
                    p.partials + ((static_cast<int64_t>(w.t) * p.max_seg * 2 + rank) * EPI_WARPS + q) *
                                     (NCH * 1024);
                spill_accumulator(tbase, const_cast<float *>(parts) + w.seg * seg_stride, 0, NCH);
                tc_fence_before();
                __syncwarp();
                release();  // TMEM read: the MMA may move on
                __syncwarp();  // every lane's stores before lane 0's release (cumulative)
                int last = 0;
                if (lane == 0) {
                    int old;
                    asm volatile("atom.add.acq_rel.gpu.global.s32 %0, [%1], 1;"
                                 : "=r"(old)
                                 : "l"(ctr)
                                 : "memory");
                    last = old == w.nseg - 1 ? 1 : 0;
                }
                last = __shfl_sync(0xFFFFFFFFu, last, 0);
                __syncwarp();  // lane 0's acquire before every lane's loads
                if (last) {
                    drain_partials<OUT, TMA_STORE, PN, MAX_SEG, EPI>(parts, seg_stride, w.nseg, stg,
                                                                sbuf, row0, col0, b, epi);
                    if (lane == 0) *ctr = 0;  // ready for the next run
                }
                continue;
            }
            if (w.role >= PIECE_CLOSE) {
                // Stream-K cut tile.  Slot k belongs to the cut at the start of
                // pair k's range: pair k spills there (its first piece), pair
                // k - 1 closes from there (its last piece).  One fp32 region of
                // NCH x 32 x 32 and one flag per (slot, CTA, warp).
                const int slot = w.role == PIECE_SPILL ? pair : pair + 1;
                const int idx = (slot * 2 + static_cast<int>(rank)) * EPI_WARPS + q;
                int32_t *flag = p.tail_sync + idx;
                float *region = p.partials + static_cast<int64_t>(idx) * (NCH * 1024);
                if (w.role == PIECE_SPILL) {
                    spill_accumulator(tbase, region, 0, NCH);
                    tc_fence_before();
                    __syncwarp();
                    release();  // TMEM read: the MMA may move on
                    // the warp barrier orders every lane's stores before lane
                    // 0's release (release is cumulative)
                    __syncwarp();
                    if (lane == 0)
                        asm volatile("st.release.gpu.global.b32 [%0], %1;" ::"l"(flag), "r"(1)
                                     : "memory");
                    continue;
                }
                int ok = 1;
                if (lane == 0)
                    ok = wait_flag_bounded(flag, wc, timeout_code(ROLE_EPILOGUE, 0x200 + idx)) ? 1 : 0;
                ok = __shfl_sync(0xFFFFFFFFu, ok, 0);
                __syncwarp();
                if (!ok) {
                    tc_fence_before();
                    release();
                    break;
                }
                drain_accumulator<OUT, TMA_STORE, PN, true, EPI>(tbase, stg, sbuf, row0, col0, b,
                                                            epi, release, region, 0, NCH);
                if (lane == 0) *flag = 0;  // read: ready for the next run
                continue;
            }
            const int half = w.role;
            // Split tail tile: its two K halves run on two pairs at the same
            // time.  Each half owns half of the 32-column chunks of every warp's
            // 32 rows: it spills the chunks the other half owns (fp32) and
            // raises that half's flag, then waits (bounded) for its own flag and
            // stores own + other for the chunks it owns.  Neither side waits
            // before spilling, so both waits end; every output element is one
            // two-term fp32 sum, which commutes, so the result does not depend
            // on which half finishes first.  The reader clears its flag.
            constexpr int HCH = (NCH + 1) / 2;  // chunks owned by half 0
            const int slot = (w.slot * 2 + static_cast<int>(rank)) * EPI_WARPS + q;
            int32_t *flags = p.tail_sync + 2 * slot;          // flags[h]: region of half h ready
            float *region = p.partials + static_cast<int64_t>(slot) * (2 * 4 * 1024);
            const int other = half ^ 1;
            const int own_lo = half ? HCH : 0, own_hi = half ? NCH : HCH;
            const int oth_lo = other ? HCH : 0, oth_hi = other ? NCH : HCH;
            spill_accumulator(tbase, region + other * (4 * 1024), oth_lo, oth_hi);
            __syncwarp();  // every lane's stores before lane 0's release (cumulative)
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
            drain_accumulator<OUT, TMA_STORE, PN, true, EPI>(tbase, stg, sbuf, row0, col0, b, epi,
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

template <int PN, int KS, int OUT, bool TS, bool EPI, bool F8 = false>
cudaError_t launch_impl(const CUtensorMap &tmA, const CUtensorMap &tmB, const CUtensorMap &tmC,
                        const TiledParams &p, int grid, cudaStream_t stream) {
    auto kern = hgemm_pair_kernel<PN, KS, OUT, TS, EPI, F8>;
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         PairCfg<PN, KS>::SMEM_TOTAL);
    if (e != cudaSuccess) return e;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(static_cast<unsigned>(grid), 1, 1);
    cfg.blockDim = dim3(NUM_THREADS, 1, 1);
    cfg.dynamicSmemBytes = PairCfg<PN, KS>::SMEM_TOTAL;
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

// All variants of one output type: pn, K blocks per stage, TMA store, fused
// epilogue (p.ep.on).  Each output type is instantiated in its own
// translation unit (gemm_pair_f16.cu, ...) so that they compile in parallel.
template <int OUT>
cudaError_t launch_pair_typed(int pn, int ks, bool ts, const CUtensorMap &tmA,
                              const CUtensorMap &tmB, const CUtensorMap &tmC, const TiledParams &p,
                              int grid, cudaStream_t s) {
    const int v = (pn == 256 ? 0 : 8) | (ks == 2 ? 0 : 4) | (ts ? 0 : 2) | (p.ep.on ? 1 : 0);
    if ((pn != 256 && pn != 224) || (ks != 1 && ks != 2)) return cudaErrorInvalidValue;
    if (p.f8) {  // 8-bit inputs: 256 x 256 tiles, two K blocks per stage only
        switch (v) {
            case 0: return launch_impl<256, 2, OUT, true, false, true>(tmA, tmB, tmC, p, grid, s);
            case 1: return launch_impl<256, 2, OUT, true, true, true>(tmA, tmB, tmC, p, grid, s);
            case 2: return launch_impl<256, 2, OUT, false, false, true>(tmA, tmB, tmC, p, grid, s);
            case 3: return launch_impl<256, 2, OUT, false, true, true>(tmA, tmB, tmC, p, grid, s);
            default: return cudaErrorInvalidValue;
        }
    }
    switch (v) {
        case 0: return launch_impl<256, 2, OUT, true, false>(tmA, tmB, tmC, p, grid, s);
        case 1: return launch_impl<256, 2, OUT, true, true>(tmA, tmB, tmC, p, grid, s);
        case 2: return launch_impl<256, 2, OUT, false, false>(tmA, tmB, tmC, p, grid, s);
        case 3: return launch_impl<256, 2, OUT, false, true>(tmA, tmB, tmC, p, grid, s);
        case 4: return launch_impl<256, 1, OUT, true, false>(tmA, tmB, tmC, p, grid, s);
        case 5: return launch_impl<256, 1, OUT, true, true>(tmA, tmB, tmC, p, grid, s);
        case 6: return launch_impl<256, 1, OUT, false, false>(tmA, tmB, tmC, p, grid, s);
        case 7: return launch_impl<256, 1, OUT, false, true>(tmA, tmB, tmC, p, grid, s);
        case 8: return launch_impl<224, 2, OUT, true, false>(tmA, tmB, tmC, p, grid, s);
        case 9: return launch_impl<224, 2, OUT, true, true>(tmA, tmB, tmC, p, grid, s);
        case 10: return launch_impl<224, 2, OUT, false, false>(tmA, tmB, tmC, p, grid, s);
        case 11: return launch_impl<224, 2, OUT, false, true>(tmA, tmB, tmC, p, grid, s);
        case 12: return launch_impl<224, 1, OUT, true, false>(tmA, tmB, tmC, p, grid, s);
        case 13: return launch_impl<224, 1, OUT, true, true>(tmA, tmB, tmC, p, grid, s);
        case 14: return launch_impl<224, 1, OUT, false, false>(tmA, tmB, tmC, p, grid, s);
        case 15: return launch_impl<224, 1, OUT, false, true>(tmA, tmB, tmC, p, grid, s);
        default: return cudaErrorInvalidValue;
    }
}

// Co-resident 2-CTA clusters of the pair kernel.  Every variant uses the
// same shared memory (192 KB of stages), so one gives the count for all.
template <int OUT>
int max_pairs_typed() {
    auto kern = hgemm_pair_kernel<256, 2, OUT, true, false>;
    if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             PairCfg<256, 2>::SMEM_TOTAL) != cudaSuccess)
        return 0;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(2, 1, 1);
    cfg.blockDim = dim3(NUM_THREADS, 1, 1);
    cfg.dynamicSmemBytes = PairCfg<256, 2>::SMEM_TOTAL;
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

}  // namespace

// Per-output-type entry points (gemm_pair_f16.cu, gemm_pair_bf16.cu,
// gemm_pair_f32.cu).
cudaError_t launch_pair_f16(int pn, int ks, bool ts, const CUtensorMap &tmA, const CUtensorMap &tmB,
                            const CUtensorMap &tmC, const TiledParams &p, int grid, cudaStream_t s);
cudaError_t launch_pair_bf16(int pn, int ks, bool ts, const CUtensorMap &tmA, const CUtensorMap &tmB,
                             const CUtensorMap &tmC, const TiledParams &p, int grid, cudaStream_t s);
cudaError_t launch_pair_f32(int pn, int ks, bool ts, const CUtensorMap &tmA, const CUtensorMap &tmB,
                            const CUtensorMap &tmC, const TiledParams &p, int grid, cudaStream_t s);
int pair_max_active_pairs_bf16();

}  // namespace hg
