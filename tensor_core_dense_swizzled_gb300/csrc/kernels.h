// kernels.h -- parameter blocks and host launchers of libhgemm's kernels.
// Shared by the kernel translation units and the C-ABI layer (api.cpp); no
// device code here.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <stdint.h>

namespace hg {

enum OutType : int { OUT_F16 = 0, OUT_BF16 = 1, OUT_F32 = 2 };

// Instruction descriptor of tcgen05.mma .kind::f16 with an fp32 accumulator:
//   bits 4-5 D format (1 = f32), 7-9 A format, 10-12 B format (0 = f16,
//   1 = bf16), 15 A major (0 = K, 1 = MN), 16 B major, 17-22 N >> 3,
//   24-28 M >> 4.
constexpr uint32_t idesc_f16(uint32_t ab_bf16, uint32_t a_mn, uint32_t b_mn,
                                                 uint32_t m, uint32_t n) {
    return (1u << 4) | (ab_bf16 << 7) | (ab_bf16 << 10) | (a_mn << 15) | (b_mn << 16) |
           ((n >> 3) << 17) | ((m >> 4) << 24);
}

// Instruction descriptor of tcgen05.mma .kind::f8f6f4 with an fp32
// accumulator: the same fields as idesc_f16, A / B formats 0 = E4M3,
// 1 = E5M2.
constexpr uint32_t idesc_f8(uint32_t a_fmt, uint32_t b_fmt, uint32_t a_mn, uint32_t b_mn,
                            uint32_t m, uint32_t n) {
    return (1u << 4) | (a_fmt << 7) | (b_fmt << 10) | (a_mn << 15) | (b_mn << 16) |
           ((n >> 3) << 17) | ((m >> 4) << 24);
}

// Elements per 128-byte K block: 64 of a 16-bit type, 128 of an 8-bit one.
constexpr int kblock_elems(bool f8) { return f8 ? 128 : 64; }

// Fused epilogue of the final values of C (see hgemm_epilogue_t):
// D = act(alpha * rs[i] * cs[j] * acc + beta * C_prev + bias[j]).  `on` = 0:
// D = acc (nothing else is read).
struct EpiParams {
    float alpha, beta;
    const float *bias, *row_scale, *col_scale;
    int32_t act;  // 0 none, 1 ReLU, 2 GELU
    int32_t on;
};

// Persistent tiled kernel: 128 x BN output tiles, BK = 64, TMEM accumulators.
struct TiledParams {
    int32_t M, N, K, batch;
    int32_t num_m, num_n, num_kb;  // tiles along M, N; 64-wide K blocks
    int32_t tiles;                 // batch * num_m * num_n
    int32_t group_m;               // raster: m-tiles per group (L2 reuse)
    uint32_t idesc;                // tcgen05 instruction descriptor
    void *C;                       // generic (non-TMA) epilogue only
    int64_t ldc, strideC;
    int32_t *err;                  // device error word
    uint64_t timeout_ns;
    // Pair kernel only: work units.  Tiles [0, full_tiles) are one unit each;
    // each of the remaining tiles - full_tiles "tail" tiles is split into
    // tail_split (1 or 2) K halves, so that the last, partial wave finishes
    // in half a tile time.  units = full_tiles + (tiles - full_tiles) * tail_split.
    int32_t full_tiles, tail_split, units;
    float *partials;               // [tail][rank][warp][chunk][32 rows][32 cols] fp32
    int32_t *tail_sync;            // [tail][rank][warp][2]: arrival counter, ready flag (zero between runs)
    // Pair kernel only: 1 when the A and B maps are the 4-D views that load a
    // whole stage of each operand with one copy (see launch_pair).
    int32_t wide_boxes;
    // Pair kernel only: 2 = first-wave dealing (see max_seg); 1 = stream-K
    // schedule (tiles >= pairs): tiles below
    // full_tiles run whole, the K steps of the rest (pairs <= rest < 2 pairs)
    // are dealt to the pairs in equal contiguous ranges; cut tiles meet
    // through partials / tail_sync slots indexed by pair ([pair][rank][warp]:
    // PN / 32 chunks of 32 x 32 fp32, one flag).
    int32_t stream_k;
    // Pair kernel, stream_k == 2 (first-wave dealing of tiles 0 .. full_tiles
    // - 1): partials [tile][max_seg][rank][warp][PN / 32 chunks][32 x 32]
    // fp32, tail_sync = counters [tile][rank][warp] (zero between runs).
    int32_t max_seg;
    EpiParams ep;
    // 1: B is stored N x K (K contiguous) and staged K-major; 0: K x N,
    // staged MN-major.
    int32_t b_kmajor;
    // 1: 8-bit inputs (E4M3 / E5M2, both operands K-major); a K block is 128
    // elements (num_kb counts those).
    int32_t f8;
    // Single-CTA tiled kernel only: epilogue warps, 4 or 8 (8: two warps per
    // TMEM lane quarter, each draining half of the tile's columns; 16-bit
    // inputs and tile widths 128 / 256).
    int32_t epi_warps;
    // Single-CTA tiled kernel, abort-path testing only: 0 off; k >= 1 leaves
    // the stage of K block k - 1 of CTA 0's first tile unarmed (no
    // expect_tx, no copies), so the MMA issuer's bounded wait on it expires.
    int32_t withhold_kb;
    // Invariant checks (debug_checks): 0 off, 1 on, 2 on with an out-of-range
    // tile planted in the first work item of CTA 0 / pair 0.
    int32_t debug;
};

// Skinny kernel: C^T = B^T . A^T, NB x 64 output columns of C per work
// unit (NT = ceil(NB / 2) sub-tiles of 128 columns), split-K.  Partials and
// counters are indexed by sub-tile (num_tiles x NT of them).
struct SkinnyParams {
    int32_t M, N, K, batch;
    int32_t num_tiles;    // NB x 64-wide column tiles (work units along N): ceil(N / (64 NB))
    int32_t num_kb;       // 64-wide K blocks in total
    int32_t split;        // K splits
    int32_t kb_per_split; // K blocks per split (last split may have fewer)
    int32_t units;        // batch * split * num_tiles
    uint32_t idesc;
    void *C;
    int64_t ldc, strideC;
    float *partials;      // [batch][split][num_tiles x NT][NU][128] fp32 (split > 1)
    int32_t *counters;    // [batch][num_tiles x NT][4] arrival counters (one per epilogue warp), zero between runs
    int32_t *err;
    uint64_t timeout_ns;
    // 1: stream-K dealing -- the batch x num_tiles x num_kb (tile, K block)
    // steps are dealt to the CTAs as equal contiguous ranges, so every SM
    // streams the same number of bytes; a tile cut into several pieces is
    // summed by the last piece to arrive.  `split` is then the most pieces a
    // tile can be cut into (the partials' stride) and kb_per_split unused.
    int32_t deal;
    // Stages of B each CTA asks L2 for before waiting on the previous kernel.
    int32_t prefetch;
    EpiParams ep;
    // 1: B is stored N x K (K contiguous): the MMA's A operand (B^T) is
    // staged K-major, rows = columns of C; 0: K x N, staged MN-major.
    int32_t b_kmajor;
    // 1: 8-bit inputs (K-major only); K blocks of 128 elements.
    int32_t f8;
    // Invariant checks, as TiledParams::debug.
    int32_t debug;
};

// Shared memory the tiled kernel needs for a given BN (bytes, incl. alignment slack).
int tiled_smem_bytes(int bn, int epi_warps);
int tiled_stages(int bn, int epi_warps);
int skinny_stages(int nu, int nb);

// Launchers return cudaSuccess or the launch error.  `out` is an OutType.
cudaError_t launch_tiled(int bn, int out, bool tma_store, const CUtensorMap &tmA,
                         const CUtensorMap &tmB, const CUtensorMap &tmC, const TiledParams &p,
                         int grid, cudaStream_t stream);

// nu = padded M (16 or 32); nb = 64-column blocks per work unit (2, 3, 4, 6, 8).
cudaError_t launch_skinny(int nu, int nb, int out, const CUtensorMap &tmA, const CUtensorMap &tmB,
                          const SkinnyParams &p, int grid, cudaStream_t stream);

// CTA-pair kernel (cta_group::2): 256 x pn tiles, TiledParams with num_m
// counting 256-row tiles and num_n pn-column tiles; `grid` = 2 x pairs.
// ks = 64-wide K blocks per pipeline stage (1 or 2).
//
// Maps: with p.wide_boxes == 0, tmA is the 3-D (K, M, batch) map with
// 64 x 128 boxes and tmB the 3-D (N, K, batch) map with 64 x 64 boxes (both
// 128-byte swizzled), loaded box by box.  With p.wide_boxes == 1 (pn = 256,
// K and N multiples of 64) they are 4-D views that split the contiguous
// dimension in 64-element blocks: tmA (64, M, K / 64, batch) with boxes
// 64 x 128 x ks, tmB (64, K, N / 64, batch) with boxes 64 x 64 ks x 2, so one
// copy per operand fills a stage.
int pair_stages(int ks);
int pair_max_active_pairs();  // co-resident 2-CTA clusters on the current device (0 on error)
// pn = columns per pair tile: 256 or 224 (112 B columns per CTA).
cudaError_t launch_pair(int pn, int ks, int out, bool tma_store, const CUtensorMap &tmA,
                        const CUtensorMap &tmB, const CUtensorMap &tmC, const TiledParams &p,
                        int grid, cudaStream_t stream);

// One operand copy: a batch of rows x cols 16-bit matrices (leading
// dimension ld_src, batch stride stride_src, any 2-byte alignment) into dst
// with leading dimension ld_dst (a multiple of 8, >= cols) and batch stride
// stride_dst (16-byte aligned).
struct Repack16Job {
    const void *src;
    int64_t ld_src, stride_src;
    void *dst;
    int64_t ld_dst, stride_dst, rows, cols, batch;
};

// Runs one or two operand copies in a single launch.
cudaError_t launch_repack16(const Repack16Job *jobs, int njobs, int num_sms, cudaStream_t stream);

// Writes zeros into a batch of rows x cols blocks of `elem_bytes`-byte elements.
cudaError_t launch_zero_fill(void *C, int64_t ldc, int64_t strideC, int64_t rows, int64_t cols,
                             int64_t batch, int elem_bytes, int num_sms, cudaStream_t stream);

// K = 0 with a fused epilogue: D = act(beta * C_prev + bias) over the
// batch of rows x cols blocks of C.  `out` is an OutType.
cudaError_t launch_epilogue_fill(void *C, int64_t ldc, int64_t strideC, int64_t rows,
                                 int64_t cols, int64_t batch, int out, const EpiParams &ep,
                                 int num_sms, cudaStream_t stream);

// One-warp kernel waiting on an mbarrier nothing signals (watchdog self-test).
cudaError_t launch_watchdog_selftest(int32_t *err, uint64_t timeout_ns, cudaStream_t stream);

// Attention forward (attention.cu): O = softmax(scale Q K^T [causal]) V with
// Q [bh][sq][128], K, V [bh][skv][128], O [bh][sq][128], 16-bit, dense.
// One CTA per 128-query tile, two per SM; the tensor maps cover Q, K and V
// as (128 elements, rows, bh) with 64 x 128 boxes for Q and 64 x 64 for K, V.
struct AttnParams {
    int32_t bh, sq, skv;  // heads x batch, query rows, key rows
    int32_t nqt;          // query tiles per head: ceil(sq / 128)
    int32_t causal;       // key j allowed for query i when j <= i + skv - sq
    float scale_log2;     // softmax scale x log2(e), > 0
    uint32_t idesc_s;     // S = Q K^T: M 128, N 64 keys, both K-major
    uint32_t idesc_o;     // O += P V: M 128, N 128, P from TMEM, V MN-major
    void *O;
    int32_t *err;
    uint64_t timeout_ns;
};

cudaError_t launch_attention(bool bf16, const CUtensorMap &tmQ, const CUtensorMap &tmK,
                             const CUtensorMap &tmV, const AttnParams &p, cudaStream_t stream);

}  // namespace hg
