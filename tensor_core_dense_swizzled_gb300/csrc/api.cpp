// api.cpp -- the C ABI of libhgemm (declared in include/hgemm.h).
//
// Host side only: argument validation, the choice of execution path, the
// device workspace, TMA tensor-map encoding and kernel launches.  The checks
// mirror the host wrapper of the Ampere kernel in
// "tensor-cores-cutlass-and-cute" section 四.4 (device, dtype, shape and
// layout are checked before any pointer is reinterpreted), widened to the
// strided, batched and ragged cases the library accepts.
#include <cuda.h>
#include <cuda_runtime.h>
#include <cudaTypedefs.h>

#include <cmath>
#include <cstdarg>
#include <cstdint>
#include <cstdio>
#include <cstdlib>
#include <cstring>
#include <map>
#include <memory>
#include <mutex>
#include <string>
#include <tuple>

#include "hgemm.h"
#include "internal.h"
#include "kernels.h"

namespace {

constexpr uint64_t kDefaultTimeoutNs = 2000000000ull;  // 2 s per pipeline wait
constexpr int64_t kMaxDim = (1ll << 31) - 1;
constexpr int kMaxHostChunks = 4;  // row chunks of the hgemm_run_host pipeline

thread_local std::string g_detail;

hgemm_status_t fail(hgemm_status_t s, const char *fmt, ...) {
    char buf[512];
    va_list ap;
    va_start(ap, fmt);
    vsnprintf(buf, sizeof(buf), fmt, ap);
    va_end(ap);
    g_detail = buf;
    return s;
}

hgemm_status_t cuda_fail(cudaError_t e, const char *what) {
    return fail(e == cudaErrorMemoryAllocation ? HGEMM_ERR_OOM : HGEMM_ERR_CUDA, "%s: %s (%s)", what,
                cudaGetErrorName(e), cudaGetErrorString(e));
}

PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
    static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
    static std::once_flag once;
    std::call_once(once, [] {
        void *p = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault,
                                             &q) == cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
    });
    return fn;
}

inline int64_t round_up(int64_t x, int64_t m) { return (x + m - 1) / m * m; }
inline int64_t ceil_div(int64_t x, int64_t m) { return (x + m - 1) / m; }
inline bool aligned16(const void *p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }
inline int out_bytes(hgemm_dtype_t d) { return d == HGEMM_F32 ? 4 : 2; }
inline bool is_f8(hgemm_dtype_t d) { return d == HGEMM_E4M3 || d == HGEMM_E5M2; }
inline int in_bytes(hgemm_dtype_t d) { return is_f8(d) ? 1 : 2; }
// Elements per K block: 128 bytes of the input type (one swizzled row).
inline int kblock(hgemm_dtype_t d) { return is_f8(d) ? 128 : 64; }
inline int out_type(hgemm_dtype_t d) {
    return d == HGEMM_F32 ? hg::OUT_F32 : (d == HGEMM_BF16 ? hg::OUT_BF16 : hg::OUT_F16);
}

// Encodes a 3-D tiled map over a row-major [batch][rows][cols] array with the
// given element size, leading dimension and batch stride (elements).
hgemm_status_t encode_3d(CUtensorMap *map, const void *base, CUtensorMapDataType dt, int esize,
                         int64_t cols, int64_t rows, int64_t batch, int64_t ld, int64_t stride,
                         uint32_t box_cols, uint32_t box_rows,
                         CUtensorMapSwizzle swz = CU_TENSOR_MAP_SWIZZLE_128B,
                         CUtensorMapL2promotion promo = CU_TENSOR_MAP_L2_PROMOTION_L2_256B) {
    auto fn = encode_fn();
    if (!fn) return fail(HGEMM_ERR_CUDA, "cuTensorMapEncodeTiled is not available from the driver");
    int64_t bstride = stride * esize;
    if (batch == 1) bstride = round_up(rows * ld * esize, 16);
    cuuint64_t dims[3] = {static_cast<cuuint64_t>(cols), static_cast<cuuint64_t>(rows),
                          static_cast<cuuint64_t>(batch)};
    cuuint64_t strides[2] = {static_cast<cuuint64_t>(ld * esize), static_cast<cuuint64_t>(bstride)};
    cuuint32_t box[3] = {box_cols, box_rows, 1};
    cuuint32_t estr[3] = {1, 1, 1};
    CUresult r = fn(map, dt, 3, const_cast<void *>(base), dims, strides, box, estr,
                    CU_TENSOR_MAP_INTERLEAVE_NONE, swz, promo,
                    CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    if (r != CUDA_SUCCESS)
        return fail(HGEMM_ERR_CUDA,
                    "cuTensorMapEncodeTiled failed (%d): dims %lld x %lld x %lld, ld %lld, "
                    "stride %lld, box %u x %u",
                    static_cast<int>(r), static_cast<long long>(cols), static_cast<long long>(rows),
                    static_cast<long long>(batch), static_cast<long long>(ld),
                    static_cast<long long>(stride), box_cols, box_rows);
    return HGEMM_OK;
}

// 4-D view of a row-major rows x cols operand whose contiguous dimension is
// a multiple of blk = 128 bytes / esize elements (64 16-bit or 128 8-bit),
// split in blk-element blocks: dims (blk, rows, cols / blk, batch), strides
// ld (rows), 128 bytes (blocks), stride (batch); box blk x box_rows x
// box_blocks; 128-byte swizzle, zero fill outside.  A (M x K) with
// box_blocks = K blocks per stage and B (K x N) with box_rows = K rows per
// stage, box_blocks = 64-column blocks per CTA.
hgemm_status_t encode_split_4d(CUtensorMap *map, const void *base, CUtensorMapDataType dt,
                               int esize, int64_t cols, int64_t rows, int64_t batch, int64_t ld,
                               int64_t stride, uint32_t box_rows, uint32_t box_blocks) {
    auto fn = encode_fn();
    if (!fn) return fail(HGEMM_ERR_CUDA, "cuTensorMapEncodeTiled is not available from the driver");
    const int64_t blk = 128 / esize;
    int64_t bstride = stride * esize;
    if (batch == 1) bstride = round_up(rows * ld * esize, 16);
    cuuint64_t dims[4] = {static_cast<cuuint64_t>(blk), static_cast<cuuint64_t>(rows),
                          static_cast<cuuint64_t>(cols / blk), static_cast<cuuint64_t>(batch)};
    cuuint64_t strides[3] = {static_cast<cuuint64_t>(ld * esize), 128,
                             static_cast<cuuint64_t>(bstride)};
    cuuint32_t box[4] = {static_cast<cuuint32_t>(blk), box_rows, box_blocks, 1};
    cuuint32_t estr[4] = {1, 1, 1, 1};
    CUresult r = fn(map, dt, 4, const_cast<void *>(base), dims, strides, box, estr,
                    CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                    CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    if (r != CUDA_SUCCESS)
        return fail(HGEMM_ERR_CUDA, "cuTensorMapEncodeTiled (4-D view) failed (%d)", static_cast<int>(r));
    return HGEMM_OK;
}

}  // namespace

struct hgemm_plan_s {
    int64_t M, N, K, lda, ldb, ldc, batch, sA, sB, sC;
    hgemm_dtype_t din, dout;
    hgemm_options_t opt;
    int device, num_sms;
    int path;
    // tiled path
    int bn;
    int epi_warps = 4;     // single-CTA tiled kernel: epilogue warps of plain runs (4 or 8)
    int epi_warps_ep = 4;  // the same for runs with the fused epilogue
    bool pair;  // 256 x 256 tiles on CTA pairs (cta_group::2)
    // pair path: tiles [0, full_tiles) whole, the tail split in tail_split K halves
    int64_t ptiles = 0, full_tiles = 0, units = 0;
    int tail_split = 1;
    int pair_ks = 2;  // pair path: 64-wide K blocks per pipeline stage
    bool wide = false;  // pair path: A/B maps are the 4-D one-copy-per-stage views
    int stream_k = 0;  // pair path: 1 stream-K of the last waves, 2 first-wave dealing (see plan_create)
    int max_seg = 0;   // stream_k == 2: most pieces a dealt tile is cut into
    // skinny path
    int nu, nb, split, kb_per;  // padded M, 64-column blocks per unit, K splits
    bool skinny_deal = false;   // stream-K dealing (split = most pieces per tile)
    int grid;
    bool ld_repack_a, ld_repack_b;  // forced by leading dimension / stride
    bool ldc_tma;                   // C's ld / stride allow TMA stores
    uint64_t timeout_ns;
    // workspace: [err 256 B][counters][partials][A copy][B copy]
    char *ws = nullptr;
    size_t ws_bytes = 0, off_counters = 0, off_partials = 0, off_apack = 0, off_bpack = 0;
    size_t apack_bytes = 0, bpack_bytes = 0;
    bool have_apack = false, have_bpack = false;  // workspace holds room for the copy
    int64_t lda_p = 0, ldb_p = 0, sA_p = 0, sB_p = 0;
    // host-buffer (end-to-end) staging
    char *dA = nullptr, *dB = nullptr, *dC = nullptr;
    size_t dA_bytes = 0, dB_bytes = 0, dC_bytes = 0;
    // hgemm_run_host pipeline (see host_pipeline): row chunks of A and C run
    // as plans of their own on the caller's stream while the next chunk's
    // rows of A arrive on s_in and finished rows of C leave on s_out
    hgemm_plan_s *sub[kMaxHostChunks] = {};  // chunk i's plan (chunks of equal rows share one)
    bool sub_own[kMaxHostChunks] = {};       // sub[i] is owned (first chunk of its size)
    int64_t chunk_r0[kMaxHostChunks + 1] = {};  // chunk i: rows [chunk_r0[i], chunk_r0[i + 1])
    int nchunks = 0;
    cudaStream_t s_in = nullptr, s_out = nullptr;
    cudaEvent_t ev_start = nullptr, ev_done = nullptr;
    cudaEvent_t ev_a[kMaxHostChunks] = {}, ev_c[kMaxHostChunks] = {};
    // tensor-map cache
    const void *okA = nullptr, *okB = nullptr;  // the last A, B, C that passed
    const void *okC = nullptr;                  //   check_device_pointer, and the
    const float *okBias = nullptr, *okRow = nullptr, *okCol = nullptr;  // epilogue's vectors
    const void *mA = nullptr, *mB = nullptr;
    void *mC = nullptr;
    bool maps_ok = false;
    CUtensorMap tmA, tmB, tmC;
};

namespace {

int64_t span_elems(int64_t rows, int64_t cols, int64_t ld, int64_t batch, int64_t stride) {
    if (rows == 0 || cols == 0) return 0;
    return (batch - 1) * stride + (rows - 1) * ld + cols;
}

hgemm_status_t validate(int64_t M, int64_t N, int64_t K, int64_t lda, int64_t ldb, int64_t ldc,
                        int64_t batch, int64_t sA, int64_t sB, int64_t sC, bool trans_b, hgemm_dtype_t din,
                        hgemm_dtype_t dout) {
    if (din != HGEMM_F16 && din != HGEMM_BF16 && !is_f8(din))
        return fail(HGEMM_ERR_INVALID_ARG,
                    "dtype_in must be HGEMM_F16, HGEMM_BF16, HGEMM_E4M3 or HGEMM_E5M2 (got %d)",
                    static_cast<int>(din));
    if (dout != HGEMM_F16 && dout != HGEMM_BF16 && dout != HGEMM_F32)
        return fail(HGEMM_ERR_INVALID_ARG, "dtype_out must be HGEMM_F32, HGEMM_F16 or HGEMM_BF16 (got %d)",
                    static_cast<int>(dout));
    if (M < 0 || N < 0 || K < 0)
        return fail(HGEMM_ERR_INVALID_ARG, "negative size M=%lld N=%lld K=%lld",
                    static_cast<long long>(M), static_cast<long long>(N), static_cast<long long>(K));
    if (batch < 1) return fail(HGEMM_ERR_INVALID_ARG, "batch must be >= 1 (got %lld)", static_cast<long long>(batch));
    if (M > kMaxDim || N > kMaxDim || K > kMaxDim || batch > kMaxDim)
        return fail(HGEMM_ERR_UNSUPPORTED, "sizes above 2^31-1 are not supported");
    if (M > 0 && K > 0 && lda < K)
        return fail(HGEMM_ERR_INVALID_ARG, "lda (%lld) < K (%lld)", static_cast<long long>(lda), static_cast<long long>(K));
    if (K > 0 && N > 0 && !trans_b && ldb < N)
        return fail(HGEMM_ERR_INVALID_ARG, "ldb (%lld) < N (%lld)", static_cast<long long>(ldb), static_cast<long long>(N));
    if (K > 0 && N > 0 && trans_b && ldb < K)
        return fail(HGEMM_ERR_INVALID_ARG, "ldb (%lld) < K (%lld) with trans_b (B stored N x K)",
                    static_cast<long long>(ldb), static_cast<long long>(K));
    if (M > 0 && N > 0 && ldc < N)
        return fail(HGEMM_ERR_INVALID_ARG, "ldc (%lld) < N (%lld)", static_cast<long long>(ldc), static_cast<long long>(N));
    if (batch > 1 && (sA < 0 || sB < 0 || sC < 0))
        return fail(HGEMM_ERR_INVALID_ARG, "negative batch stride");
    if (batch > 1 && M > 0 && N > 0 && sC < (M - 1) * ldc + N)
        return fail(HGEMM_ERR_INVALID_ARG, "strideC (%lld) makes the batches of C overlap",
                    static_cast<long long>(sC));
    {
        // every byte count derived from a span (staging buffers, copies,
        // tensor-map strides) must fit comfortably in 64 bits
        auto span_bytes = [](int64_t rows, int64_t cols, int64_t ld, int64_t nb, int64_t stride, int eb) {
            if (rows == 0 || cols == 0) return static_cast<__int128>(0);
            return (static_cast<__int128>(nb - 1) * stride + static_cast<__int128>(rows - 1) * ld + cols) * eb;
        };
        const __int128 kMaxSpan = static_cast<__int128>(1) << 60;
        const int ib = in_bytes(din), ob = out_bytes(dout);
        const int64_t nb = batch > 1 ? batch : 1;
        if (span_bytes(M, K, lda, nb, batch > 1 ? sA : 0, ib) > kMaxSpan ||
            span_bytes(trans_b ? N : K, trans_b ? K : N, ldb, nb, batch > 1 ? sB : 0, ib) > kMaxSpan ||
            span_bytes(M, N, ldc, nb, batch > 1 ? sC : 0, ob) > kMaxSpan)
            return fail(HGEMM_ERR_UNSUPPORTED, "an operand spans more than 2^60 bytes (leading dimension or "
                                               "batch stride too large)");
    }
    const int64_t tiles = batch * ceil_div(M, 128) * ceil_div(N, 128);
    if (tiles > kMaxDim) return fail(HGEMM_ERR_UNSUPPORTED, "too many output tiles");
    if (is_f8(din) && M > 0 && N > 0 && K > 0) {
        // 8-bit operands are read in place (no aligned copy is made): both
        // contiguous along K, rows and batches on 16-byte boundaries
        if (!trans_b)
            return fail(HGEMM_ERR_UNSUPPORTED, "8-bit inputs need B stored N x K (trans_b = 1)");
        if (lda % 16 != 0 || ldb % 16 != 0)
            return fail(HGEMM_ERR_UNSUPPORTED, "8-bit inputs need lda and ldb multiples of 16 (got %lld, %lld)",
                        static_cast<long long>(lda), static_cast<long long>(ldb));
        if (batch > 1 && (sA % 16 != 0 || sB % 16 != 0))
            return fail(HGEMM_ERR_UNSUPPORTED, "8-bit inputs need strideA and strideB multiples of 16");
    }
    return HGEMM_OK;
}

// Picks the split count for the skinny path: the smallest split whose units
// fill the persistent grid to >= 90% (units per wave), else the best found.
// Splitting K is a last resort: on GB300 the 8 x 28672 x 4096 product ran at
// 39.4 us unsplit (112 CTAs, 256-column units) against 60-95 us with 2 to 8
// splits over all 152 SMs.  Unsplit, the CTAs sweep the same K rows of B
// together and consume whole DRAM rows; split, they read several distant K
// ranges at once.  So K is split only when the unsplit units would leave
// more than 40 % of the SMs idle (small N), and then just enough.
int choose_split(int64_t work_tiles, int num_kb, int num_sms) {
    if (work_tiles * 10 >= static_cast<int64_t>(num_sms) * 6) return 1;
    int best = 1;
    double best_eff = 0;
    for (int s = 1; s <= 16 && s <= num_kb; ++s) {
        const int kb_per = static_cast<int>(ceil_div(num_kb, s));
        const int s_eff = static_cast<int>(ceil_div(num_kb, kb_per));
        if (s_eff != s) continue;
        if (s > 1 && kb_per < 4) break;
        const int64_t units = work_tiles * s;
        const int64_t waves = ceil_div(units, num_sms);
        const double eff = static_cast<double>(units) / static_cast<double>(waves * num_sms);
        if (eff > best_eff + 1e-9) {
            best_eff = eff;
            best = s;
        }
        if (eff >= 0.9) return s;
    }
    return best;
}

// Picks the tile width of the tiled path.  A persistent CTA processes its
// tiles in rounds ("waves") of one tile per SM.  The main loop is bound by
// delivering operands to shared memory, so a tile costs about the bytes it
// stages per K block (16 KB of A plus 8 KB per 64-column block of B), not
// its width: on GB300 at 4096^3, 128 x 224 tiles (4 B blocks, 4 waves) ran
// at 98.3 us against 91.1 us for 128 x 256 (3.4 waves), and 128 x 192 at
// 104.5 us.  Ties go to the wider tile.
int choose_tile_n(int64_t batch, int64_t M, int64_t N, int sms, bool f8) {
    static const int cands[] = {256, 224, 192, 128};
    int best = 256;
    double best_t = 1e300;
    for (int bn : cands) {
        if (f8 && bn != 256 && bn != 128) continue;  // the 8-bit kernels built
        const int64_t tiles = batch * ceil_div(M, 128) * ceil_div(N, bn);
        const int64_t waves = ceil_div(tiles, sms);
        const double t = static_cast<double>(waves) * (16 + 8 * ((bn + 63) / 64));
        if (t < best_t - 1e-9) {
            best_t = t;
            best = bn;
        }
    }
    return best;
}

// Debugging overrides from the environment, read at every plan creation and
// applied only where the caller's options leave the field at its default:
//   HGEMM_DEBUG=1          debug_checks = 1 (kernel invariant checks)
//   HGEMM_TIMEOUT_NS=<n>   the watchdog limit of every pipeline wait
//   HGEMM_FORCE_CONFIG=    pair | single | single:<tile_n> | skinny: the kernel
//                          (CTA pairs, single-CTA tiles, the skinny path)
// An unrecognised value is ignored.
void apply_env_overrides(hgemm_options_t &opt) {
    if (const char *v = std::getenv("HGEMM_DEBUG"))
        if (opt.debug_checks == 0 && std::atoi(v) != 0) opt.debug_checks = 1;
    if (const char *v = std::getenv("HGEMM_TIMEOUT_NS")) {
        const long long ns = std::atoll(v);
        if (opt.timeout_ns == 0 && ns > 0) opt.timeout_ns = static_cast<uint64_t>(ns);
    }
    if (const char *v = std::getenv("HGEMM_FORCE_CONFIG")) {
        if (opt.force_path == 0 && opt.cta_pair == 0) {
            if (std::strcmp(v, "pair") == 0) {
                opt.force_path = HGEMM_PATH_TILED;
                opt.cta_pair = 1;
            } else if (std::strncmp(v, "single", 6) == 0) {
                opt.force_path = HGEMM_PATH_TILED;
                opt.cta_pair = 2;
                if (v[6] == ':' && opt.tile_n == 0) opt.tile_n = std::atoi(v + 7);
            } else if (std::strcmp(v, "skinny") == 0) {
                opt.force_path = HGEMM_PATH_SKINNY;
            }
        }
    }
}

hgemm_status_t alloc_workspace(hgemm_plan_s *p) {
    size_t off = 256;  // error word (+ padding)
    p->off_counters = off;
    size_t counters = 0, partials = 0;
    if (p->path == HGEMM_PATH_SKINNY) {
        // 128-column sub-tiles: ceil(nb / 2) per work unit
        const int64_t num_n = ceil_div(p->N, 64 * p->nb) * ((p->nb + 1) / 2);
        counters = static_cast<size_t>(p->batch * num_n) * 4 * sizeof(int32_t);
        if (p->split > 1)
            partials = static_cast<size_t>(p->batch) * p->split * num_n * p->nu * 128 * sizeof(float);
    }
    if (p->path == HGEMM_PATH_TILED && p->pair && p->stream_k == 2) {
        // per dealt tile: counters [tile][CTA][warp]; partials
        // [tile][max_seg][CTA][warp][bn / 32 chunks of 32 x 32 fp32]
        counters = static_cast<size_t>(p->full_tiles * 2 * 4) * sizeof(int32_t);
        partials = static_cast<size_t>(p->full_tiles * p->max_seg * 2 * 4 * (p->bn / 32) * 1024) *
                   sizeof(float);
    }
    if (p->path == HGEMM_PATH_TILED && p->pair && p->stream_k == 1) {
        // per pair (the cut at the start of its range): 2 CTAs x 4 epilogue
        // warps, each with one flag and bn / 32 chunks of 32 x 32 fp32
        const int64_t slots = p->grid / 2;
        counters = static_cast<size_t>(slots * 2 * 4) * sizeof(int32_t);
        partials = static_cast<size_t>(slots * 2 * 4 * (p->bn / 32) * 1024) * sizeof(float);
    }
    if (p->path == HGEMM_PATH_TILED && p->pair && p->tail_split > 1) {
        // per tail tile: 2 CTAs x 4 epilogue warps, each with two flags and two
        // regions of up to 4 chunks of 32 rows x 32 fp32 columns (one region
        // per K half, holding the chunks that half stores)
        const int64_t tail = p->ptiles - p->full_tiles;
        counters = static_cast<size_t>(tail * 2 * 4 * 2) * sizeof(int32_t);
        partials = static_cast<size_t>(tail * 2 * 4 * 2 * 4 * 1024) * sizeof(float);
    }
    off = static_cast<size_t>(round_up(static_cast<int64_t>(off + counters), 256));
    p->off_partials = off;
    off = static_cast<size_t>(round_up(static_cast<int64_t>(off + partials), 256));
    if (p->path == HGEMM_PATH_TILED || p->path == HGEMM_PATH_SKINNY) {
        // aligned copies of A and B; allocated whenever a copy can be needed
        // (by the leading dimension now, or by a misaligned pointer later).
        // The tiled path pads their rows to whole 128-byte blocks: the copy
        // writes zeros past the last column, so the pair kernel's one-copy-
        // per-stage views apply to a copied operand whatever K and N are.
        const int64_t pad = p->path == HGEMM_PATH_TILED ? kblock(p->din) : 8;
        p->lda_p = round_up(p->K, pad);
        p->sA_p = p->M * p->lda_p;
        // B stored K x N, or N x K with trans_b: rows x cols of the stored matrix
        p->ldb_p = round_up(p->opt.trans_b ? p->K : p->N, pad);
        p->sB_p = (p->opt.trans_b ? p->N : p->K) * p->ldb_p;
        p->apack_bytes = static_cast<size_t>(p->batch * p->sA_p * in_bytes(p->din));
        p->bpack_bytes = static_cast<size_t>(p->batch * p->sB_p * in_bytes(p->din));
    }
    p->ws_bytes = off;
    p->off_apack = p->off_bpack = 0;
    if (p->ld_repack_a || p->opt.force_repack) {
        p->off_apack = p->ws_bytes;
        p->ws_bytes = static_cast<size_t>(round_up(static_cast<int64_t>(p->ws_bytes + p->apack_bytes), 256));
        p->have_apack = true;
    }
    if (p->ld_repack_b || p->opt.force_repack) {
        p->off_bpack = p->ws_bytes;
        p->ws_bytes = static_cast<size_t>(round_up(static_cast<int64_t>(p->ws_bytes + p->bpack_bytes), 256));
        p->have_bpack = true;
    }
    cudaError_t e = cudaMalloc(reinterpret_cast<void **>(&p->ws), p->ws_bytes);
    if (e != cudaSuccess) {
        p->ws = nullptr;
        return cuda_fail(e, "cudaMalloc(workspace)");
    }
    e = cudaMemset(p->ws, 0, p->off_partials);  // error word + counters start at zero
    if (e != cudaSuccess) return cuda_fail(e, "cudaMemset(workspace)");
    return HGEMM_OK;
}

// Grows the workspace when a run needs an operand copy the plan did not
// foresee (a misaligned base pointer).  Synchronous; happens at most once per
// operand and plan.
hgemm_status_t ensure_pack(hgemm_plan_s *p, bool need_a, bool need_b) {
    const bool add_a = need_a && !p->have_apack;
    const bool add_b = need_b && !p->have_bpack;
    if (!add_a && !add_b) return HGEMM_OK;
    size_t need = p->ws_bytes;
    size_t off_a = p->off_apack, off_b = p->off_bpack;
    if (add_a) {
        off_a = need;
        need = static_cast<size_t>(round_up(static_cast<int64_t>(need + p->apack_bytes), 256));
    }
    if (add_b) {
        off_b = need;
        need = static_cast<size_t>(round_up(static_cast<int64_t>(need + p->bpack_bytes), 256));
    }
    char *nws = nullptr;
    cudaError_t e = cudaDeviceSynchronize();
    if (e != cudaSuccess) return cuda_fail(e, "cudaDeviceSynchronize");
    e = cudaMalloc(reinterpret_cast<void **>(&nws), need);
    if (e != cudaSuccess) return cuda_fail(e, "cudaMalloc(workspace)");
    e = cudaMemcpy(nws, p->ws, p->off_partials, cudaMemcpyDeviceToDevice);
    if (e != cudaSuccess) {
        cudaFree(nws);
        return cuda_fail(e, "cudaMemcpy(workspace)");
    }
    cudaFree(p->ws);
    p->ws = nws;
    p->ws_bytes = need;
    p->off_apack = off_a;
    p->off_bpack = off_b;
    p->have_apack = p->have_apack || add_a;
    p->have_bpack = p->have_bpack || add_b;
    p->maps_ok = false;
    return HGEMM_OK;
}

hgemm_status_t plan_create(hgemm_plan_t *out, int64_t M, int64_t N, int64_t K, int64_t lda,
                           int64_t ldb, int64_t ldc, int64_t batch, int64_t sA, int64_t sB,
                           int64_t sC, hgemm_dtype_t din, hgemm_dtype_t dout,
                           const hgemm_options_t *options) {
    if (!out) return fail(HGEMM_ERR_INVALID_ARG, "plan pointer is NULL");
    *out = nullptr;
    if (options && (options->trans_b < 0 || options->trans_b > 1))
        return fail(HGEMM_ERR_INVALID_ARG, "trans_b must be 0 or 1");
    hgemm_status_t st = validate(M, N, K, lda, ldb, ldc, batch, sA, sB, sC,
                                 options && options->trans_b, din, dout);
    if (st != HGEMM_OK) return st;
    hgemm_options_t opt{};
    if (options) opt = *options;
    apply_env_overrides(opt);
    if (opt.force_path != 0 && opt.force_path != HGEMM_PATH_TILED && opt.force_path != HGEMM_PATH_SKINNY)
        return fail(HGEMM_ERR_INVALID_ARG, "force_path must be 0, HGEMM_PATH_TILED or HGEMM_PATH_SKINNY");
    if (opt.tile_n != 0 && opt.tile_n != 128 && opt.tile_n != 192 && opt.tile_n != 224 &&
        opt.tile_n != 256)
        return fail(HGEMM_ERR_INVALID_ARG, "tile_n must be 0, 128, 192, 224 or 256");
    if (opt.split_k < 0) return fail(HGEMM_ERR_INVALID_ARG, "split_k must be >= 0");
    if (opt.skinny_tile_n != 0 && opt.skinny_tile_n != 128 && opt.skinny_tile_n != 192 &&
        opt.skinny_tile_n != 256 && opt.skinny_tile_n != 384 && opt.skinny_tile_n != 512)
        return fail(HGEMM_ERR_INVALID_ARG, "skinny_tile_n must be 0, 128, 192, 256, 384 or 512");
    if (opt.cta_pair < 0 || opt.cta_pair > 2)
        return fail(HGEMM_ERR_INVALID_ARG, "cta_pair must be 0, 1 or 2");
    if (opt.pair_k_blocks < 0 || opt.pair_k_blocks > 2)
        return fail(HGEMM_ERR_INVALID_ARG, "pair_k_blocks must be 0, 1 or 2");
    if (opt.tail_mode < 0 || opt.tail_mode > 4)
        return fail(HGEMM_ERR_INVALID_ARG, "tail_mode must be 0, 1, 2, 3 or 4");
    if (opt.skinny_stream_k < 0 || opt.skinny_stream_k > 2)
        return fail(HGEMM_ERR_INVALID_ARG, "skinny_stream_k must be 0, 1 or 2");
    if (opt.group_m < 0 || opt.group_m > 4096)
        return fail(HGEMM_ERR_INVALID_ARG, "group_m must be in [0, 4096]");
    if (opt.tiled_epi_warps != 0 && opt.tiled_epi_warps != 4 && opt.tiled_epi_warps != 8)
        return fail(HGEMM_ERR_INVALID_ARG, "tiled_epi_warps must be 0, 4 or 8");
    if (opt.skinny_prefetch < -1 || opt.skinny_prefetch > 64)
        return fail(HGEMM_ERR_INVALID_ARG, "skinny_prefetch must be in [-1, 64]");
    if (opt.debug_checks < 0 || opt.debug_checks > 2)
        return fail(HGEMM_ERR_INVALID_ARG, "debug_checks must be 0, 1 or 2");
    if (opt.debug_withhold_kb < 0)
        return fail(HGEMM_ERR_INVALID_ARG, "debug_withhold_kb must be >= 0");
    if (opt.cta_pair == 1 && opt.tile_n != 0 && opt.tile_n != 256 && opt.tile_n != 224)
        return fail(HGEMM_ERR_INVALID_ARG, "CTA-pair tiles are 256 x 256 or 256 x 224 (tile_n 0, 256 or 224)");
    if (is_f8(din) && M > 0 && N > 0 && K > 0) {
        if (opt.force_repack)
            return fail(HGEMM_ERR_UNSUPPORTED, "8-bit inputs are never copied (force_repack)");
        if (opt.tile_n != 0 && opt.tile_n != 128 && opt.tile_n != 256)
            return fail(HGEMM_ERR_UNSUPPORTED, "8-bit inputs: tile_n must be 0, 128 or 256");
        if (opt.pair_k_blocks == 1)
            return fail(HGEMM_ERR_UNSUPPORTED, "8-bit inputs: pair_k_blocks must be 0 or 2");
        if (opt.skinny_tile_n != 0 && opt.skinny_tile_n != 128 && opt.skinny_tile_n != 256)
            return fail(HGEMM_ERR_UNSUPPORTED, "8-bit inputs: skinny_tile_n must be 0, 128 or 256");
    }
    if (opt.force_path == HGEMM_PATH_SKINNY && M > 32)
        return fail(HGEMM_ERR_UNSUPPORTED, "the skinny path handles M <= 32 (got %lld)", static_cast<long long>(M));

    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return fail(HGEMM_ERR_NO_DEVICE, "no CUDA device: %s", cudaGetErrorString(e));
    int major = 0, minor = 0, sms = 0;
    cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev);
    cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev);
    cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    if (major != 10 || minor != 3)
        return fail(HGEMM_ERR_NO_DEVICE, "libhgemm is built for sm_103a; device %d is sm_%d%d", dev,
                    major, minor);

    hgemm_plan_s *p = new (std::nothrow) hgemm_plan_s();
    if (!p) return fail(HGEMM_ERR_OOM, "host allocation failed");
    p->M = M; p->N = N; p->K = K;
    p->lda = lda; p->ldb = ldb; p->ldc = ldc; p->batch = batch;
    p->sA = batch > 1 ? sA : 0;
    p->sB = batch > 1 ? sB : 0;
    p->sC = batch > 1 ? sC : 0;
    p->din = din; p->dout = dout; p->opt = opt;
    p->device = dev; p->num_sms = sms;
    p->timeout_ns = opt.timeout_ns ? opt.timeout_ns : kDefaultTimeoutNs;
    p->bn = 0; p->nu = 0; p->nb = 2; p->split = 1; p->kb_per = 0; p->grid = 0;
    p->pair = false;

    if (M == 0 || N == 0) {
        p->path = HGEMM_PATH_EMPTY;
    } else if (K == 0) {
        p->path = HGEMM_PATH_ZERO_FILL;
    } else if (opt.force_path == HGEMM_PATH_SKINNY || (opt.force_path == 0 && M <= 32)) {
        p->path = HGEMM_PATH_SKINNY;
    } else {
        p->path = HGEMM_PATH_TILED;
    }

    const int ob = out_bytes(dout);
    const int ib = in_bytes(din);
    p->ld_repack_a = (lda * ib) % 16 != 0 || (batch > 1 && (p->sA * ib) % 16 != 0);
    p->ld_repack_b = (ldb * ib) % 16 != 0 || (batch > 1 && (p->sB * ib) % 16 != 0);
    // TMA stores write whole 16-byte chunks: a row whose byte length is not a
    // multiple of 16 would have the elements after column N-1 overwritten (up
    // to the next 16-byte boundary, past the end of the last row too), so the
    // TMA-store epilogue also needs N * sizeof(out) to be a multiple of 16.
    p->ldc_tma = (ldc * ob) % 16 == 0 && (N * ob) % 16 == 0 &&
                 (batch == 1 || (p->sC * ob) % 16 == 0) && !opt.force_generic_store;

    const int num_kb = static_cast<int>(ceil_div(K, kblock(din)));
    if (p->path == HGEMM_PATH_TILED) {
        p->bn = opt.tile_n ? opt.tile_n : choose_tile_n(batch, M, N, sms, is_f8(din));
        const int64_t tiles = batch * ceil_div(M, 128) * ceil_div(N, p->bn);
        p->grid = static_cast<int>(tiles < sms ? tiles : sms);
        p->pair = false;
        if (opt.cta_pair == 1 || (opt.cta_pair == 0 && (opt.tile_n == 0 || opt.tile_n == 256))) {
            const int max_pairs = hg::pair_max_active_pairs();
            if (opt.cta_pair == 1 && max_pairs < 1) {
                delete p;
                return fail(HGEMM_ERR_UNSUPPORTED, "no 2-CTA cluster fits on this device");
            }
            // 256 x 224 pair tiles (4 exact waves at 4096^2) measured no
            // faster than 256 x 256 (87.5 us both): they stage the same bytes.
            // They stay available through tile_n = 224.
            const int pn = opt.tile_n == 224 ? 224 : 256;
            const int64_t ptiles = batch * ceil_div(M, 256) * ceil_div(N, pn);
            // Against single CTAs (see choose_tile_n): a pair tile stages
            // 32 KB per CTA per K block for 128 x pn outputs per SM; a
            // single-CTA tile 16 KB + 8 KB per 64 columns.  Pairs win on a
            // strict gain and only for K long enough to be tensor-bound (a
            // short K leaves the product bound by writing C, where smaller
            // single-CTA tiles spread the stores better).
            const double t_single = static_cast<double>(ceil_div(tiles, sms)) *
                                    (16 + 8 * ((p->bn + 63) / 64));
            const double t_pair = max_pairs > 0 ? static_cast<double>(ceil_div(ptiles, max_pairs)) * 32
                                                : 1e300;
            if (opt.cta_pair == 1 || (t_pair < t_single && M > 128 && N > 128 && K >= 512)) {
                p->pair = true;
                p->bn = pn;
                p->ptiles = ptiles;
                p->full_tiles = ptiles;
                p->units = ptiles;
                p->tail_split = 1;
                // Tail: the last, partial wave of T = ptiles mod pairs tiles
                // would leave the other pairs idle for a whole tile time.
                //  - 2T <= pairs: those T tiles are split in two K halves run
                //    by two pairs at once, in the first wave (their exchange
                //    hides behind the next tile): 4096^3 (256 tiles, 76 pairs)
                //    runs 3.5 tile times instead of 4.
                //  - otherwise, with at least one full wave: stream-K (equal
                //    K-step ranges for the last one-and-a-bit waves).  Where
                //    both apply, the halves measured faster (4096^3: 85.7 us
                //    against 88.7 us, interleaved on one GB300): the dealt
                //    ranges run at unrelated K steps and lose L2 reuse.
                const int64_t T = ptiles % max_pairs;
                p->pair_ks = opt.pair_k_blocks ? opt.pair_k_blocks : 2;
                const int64_t num_steps = ceil_div(num_kb, p->pair_ks);
                const bool can_sk = T > 0 && ptiles >= max_pairs;
                const bool can_halves = T > 0 && 2 * T <= max_pairs && num_steps >= 2;
                // first-wave dealing: the T * num_steps steps cover every pair
                // and cut no tile into more than MAX_SEG (4) pieces
                const int64_t dealt = T * num_steps;
                const int64_t dq = dealt / max_pairs;
                const int64_t segs = dq > 0 ? (num_steps - 1) / dq + 2 : 0;
                const bool can_deal = T > 0 && dq >= 1 && segs <= 4;
                int mode = opt.no_tail_split ? 1 : opt.tail_mode;
                if (mode == 0) mode = can_halves ? 2 : 3;
                if (mode == 4 && !can_deal) mode = can_halves ? 2 : 3;
                if (mode == 4) {
                    p->stream_k = 2;
                    p->full_tiles = T;  // tiles 0 .. T-1 are dealt
                    p->max_seg = static_cast<int>(segs < max_pairs ? segs : max_pairs);
                    p->units = max_pairs;  // every pair takes part
                } else if (mode == 3 && can_sk) {
                    p->stream_k = 1;
                    // all waves but the last one and a bit run whole tiles
                    p->full_tiles = (ptiles / max_pairs - 1) * max_pairs;
                } else if (mode >= 2 && can_halves) {
                    p->tail_split = 2;
                    p->full_tiles = ptiles - T;
                    p->units = p->full_tiles + 2 * T;
                }
                p->grid = static_cast<int>(2 * (p->units < max_pairs ? p->units : max_pairs));
            }
        }
        if (!p->pair) {
            // Eight epilogue warps for the fused epilogue on products with
            // few K blocks per tile, where the epilogue's arithmetic and its
            // reads of C bound a tile (batched S = Q K^T, 64 x 1024 x 1024 x
            // 128, on GB300: + bias + GELU 100.7 -> 73.3 us, + beta C + bias
            // + ReLU 204.7 -> 138.0 us).  Plain products keep four: there the
            // stores are DRAM-bound and eight warps ran slower (53.2 ->
            // 56.4 us).
            const bool can8 = !is_f8(din) && (p->bn == 128 || p->bn == 256);
            if (opt.tiled_epi_warps == 8 && !can8) {
                delete p;
                return fail(HGEMM_ERR_UNSUPPORTED,
                            "eight epilogue warps need 16-bit inputs and tile width 128 or 256");
            }
            p->epi_warps = opt.tiled_epi_warps ? opt.tiled_epi_warps : 4;
            p->epi_warps_ep = opt.tiled_epi_warps ? opt.tiled_epi_warps : (can8 && num_kb <= 16 ? 8 : 4);
        }
    } else if (p->path == HGEMM_PATH_SKINNY) {
        p->nu = M <= 16 ? 16 : 32;
        p->nb = opt.skinny_tile_n ? opt.skinny_tile_n / 64 : hg::pick_skinny_nb(N, batch, sms);
        if (is_f8(din) && p->nb != 2 && p->nb != 4) p->nb = 4;  // the 8-bit kernels built
        const int64_t work = batch * ceil_div(N, 64 * p->nb);
        const int64_t steps = work * num_kb;
        // Deal mode (stream-K, on request only): every SM streams an equal
        // share of the (tile, K block) steps.  On 8 x 28672 x 4096 it ran
        // 45-54 us against 38.5 us for 112 unsplit 256-column units: the
        // unsplit units read each row of B together (112 x 512 contiguous
        // bytes) while dealt ranges read unrelated rows at once.
        const bool deal = opt.skinny_stream_k == 2;
        if (deal && steps < (int64_t(1) << 30)) {
            p->skinny_deal = true;
            p->grid = static_cast<int>(steps < sms ? steps : sms);
            const int64_t q = steps / p->grid;
            // a tile's num_kb steps meet at most (num_kb - 1) / q + 2 ranges
            const int64_t segs = (num_kb - 1) / q + 2;
            p->split = static_cast<int>(segs < p->grid ? segs : p->grid);
            p->kb_per = 0;
        } else {
            int split = opt.split_k ? opt.split_k : choose_split(work, num_kb, sms);
            if (split > num_kb) split = num_kb;
            if (split < 1) split = 1;
            p->kb_per = static_cast<int>(ceil_div(num_kb, split));
            p->split = static_cast<int>(ceil_div(num_kb, p->kb_per));  // no empty split
            const int64_t units = work * p->split;
            p->grid = static_cast<int>(units < sms ? units : sms);
        }
    }
    if (opt.debug_withhold_kb > 0 &&
        (p->path != HGEMM_PATH_TILED || p->pair || is_f8(din) || opt.debug_withhold_kb > num_kb)) {
        delete p;
        return fail(HGEMM_ERR_UNSUPPORTED,
                    "debug_withhold_kb applies to the single-CTA tiled kernel, 16-bit inputs, "
                    "k <= ceil(K / 64)");
    }
    st = alloc_workspace(p);
    if (st != HGEMM_OK) {
        if (p->ws) cudaFree(p->ws);
        delete p;
        return st;
    }
    *out = p;
    return HGEMM_OK;
}

// Extents of the pair kernel's 4-D views of A and B: an operand read from
// its aligned copy may be viewed up to the next 128-byte block of its
// contiguous dimension (the copy holds zeros there, which add nothing to the
// product; extra columns of B only make accumulator columns that are never
// stored).  The views need those extents to be whole blocks.
struct WideDims {
    int64_t ka, kb, nb;  // A's K, B's K (trans_b) or N (otherwise)
    bool ok;
};
WideDims wide_dims(const hgemm_plan_s *p, bool packed_a, bool packed_b) {
    const int64_t bke = kblock(p->din);
    const bool tb = p->opt.trans_b != 0;
    WideDims w;
    w.ka = packed_a ? round_up(p->K, bke) : p->K;
    w.kb = tb && packed_b ? round_up(p->K, bke) : p->K;
    w.nb = !tb && packed_b ? round_up(p->N, 64) : p->N;
    w.ok = p->path == HGEMM_PATH_TILED && p->pair && p->bn == 256 && w.ka % bke == 0 &&
           (tb ? w.kb % bke == 0 : w.nb % 64 == 0);
    if (packed_a && w.ka > p->lda_p) w.ok = false;
    if (packed_b && (tb ? w.kb : w.nb) > p->ldb_p) w.ok = false;
    return w;
}

hgemm_status_t encode_maps(hgemm_plan_s *p, const void *A, const void *B, void *C, bool tma_store) {
    if (p->maps_ok && A == p->mA && B == p->mB && C == p->mC) return HGEMM_OK;
    const CUtensorMapDataType dt = is_f8(p->din)         ? CU_TENSOR_MAP_DATA_TYPE_UINT8
                                   : p->din == HGEMM_BF16 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16
                                                          : CU_TENSOR_MAP_DATA_TYPE_FLOAT16;
    // every staged row is one 128-byte K block: 64 16-bit or 128 8-bit elements
    const int ib = in_bytes(p->din);
    const int bke = kblock(p->din);
    const bool packed_a = p->have_apack && A == p->ws + p->off_apack;
    const bool packed_b = p->have_bpack && B == p->ws + p->off_bpack;
    const int64_t lda = packed_a ? p->lda_p : p->lda;
    const int64_t sA = packed_a ? p->sA_p : p->sA;
    const int64_t ldb = packed_b ? p->ldb_p : p->ldb;
    const int64_t sB = packed_b ? p->sB_p : p->sB;
    hgemm_status_t st;
    if (p->path == HGEMM_PATH_TILED) {
        // Pair tiles 256 wide with K and N multiples of 64 (or operands read
        // from their zero-padded copies, wide_dims): the 4-D views (one copy
        // per operand per stage); otherwise, or if the driver rejects them,
        // the 3-D maps.
        // B stored N x K (trans_b) is staged K-major like A: its 4-D view
        // splits K the same way (128 rows of B per CTA), and needs only K to
        // be a multiple of 64.
        const bool tb = p->opt.trans_b != 0;
        const WideDims wd = wide_dims(p, packed_a, packed_b);
        p->wide = false;
        if (wd.ok) {
            p->wide = encode_split_4d(&p->tmA, A, dt, ib, wd.ka, p->M, p->batch, lda, sA, 128,
                                      static_cast<uint32_t>(p->pair_ks)) == HGEMM_OK &&
                      (tb ? encode_split_4d(&p->tmB, B, dt, ib, wd.kb, p->N, p->batch, ldb, sB, 128,
                                            static_cast<uint32_t>(p->pair_ks))
                          : encode_split_4d(&p->tmB, B, dt, ib, wd.nb, p->K, p->batch, ldb, sB,
                                            static_cast<uint32_t>(64 * p->pair_ks), 2)) == HGEMM_OK;
        }
        if (!p->wide) {
            st = encode_3d(&p->tmA, A, dt, ib, p->K, p->M, p->batch, lda, sA,
                           static_cast<uint32_t>(bke), 128);
            if (st != HGEMM_OK) return st;
            // boxes of 64 rows of B either way: (n, k) MN-major 64 x 64, (k, n)
            // K-major one K block x 64
            st = tb ? encode_3d(&p->tmB, B, dt, ib, p->K, p->N, p->batch, ldb, sB,
                                static_cast<uint32_t>(bke), 64)
                    : encode_3d(&p->tmB, B, dt, ib, p->N, p->K, p->batch, ldb, sB, 64, 64);
            if (st != HGEMM_OK) return st;
        }
        if (tma_store) {
            const CUtensorMapDataType ct = p->dout == HGEMM_F32   ? CU_TENSOR_MAP_DATA_TYPE_FLOAT32
                                           : p->dout == HGEMM_BF16 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16
                                                                   : CU_TENSOR_MAP_DATA_TYPE_FLOAT16;
            // 32 x 32 pieces: 128-byte rows (fp32) or 64-byte rows (fp16/bf16)
            const int ob = out_bytes(p->dout);
            st = encode_3d(&p->tmC, C, ct, ob, p->N, p->M, p->batch, p->ldc, p->sC, 32, 32,
                           ob == 4 ? CU_TENSOR_MAP_SWIZZLE_128B : CU_TENSOR_MAP_SWIZZLE_64B);
            if (st != HGEMM_OK) return st;
        } else {
            std::memset(&p->tmC, 0, sizeof(p->tmC));
        }
    } else {
        st = encode_3d(&p->tmA, A, dt, ib, p->K, p->M, p->batch, lda, sA, static_cast<uint32_t>(bke),
                       static_cast<uint32_t>(p->nu));
        if (st != HGEMM_OK) return st;
        // streamed once: 128-byte L2 fills (256-byte promotion measured 1.3 %
        // slower on 8 x 28672 x 4096)
        st = p->opt.trans_b
                 ? encode_3d(&p->tmB, B, dt, ib, p->K, p->N, p->batch, ldb, sB,
                             static_cast<uint32_t>(bke), 64, CU_TENSOR_MAP_SWIZZLE_128B,
                             CU_TENSOR_MAP_L2_PROMOTION_L2_128B)
                 : encode_3d(&p->tmB, B, dt, ib, p->N, p->K, p->batch, ldb, sB, 64, 64,
                             CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_128B);
        if (st != HGEMM_OK) return st;
        std::memset(&p->tmC, 0, sizeof(p->tmC));
    }
    p->mA = A; p->mB = B; p->mC = C;
    p->maps_ok = true;
    return HGEMM_OK;
}

hgemm_status_t plan_run(hgemm_plan_s *p, const void *A, const void *B, void *C, cudaStream_t s,
                        const hg::EpiParams &ep = hg::EpiParams{1.f, 0.f, nullptr, nullptr, nullptr, 0, 0}) {
    if (p->path == HGEMM_PATH_EMPTY) return HGEMM_OK;
    if (!C) return fail(HGEMM_ERR_INVALID_ARG, "C is NULL");
    const int ob = out_bytes(p->dout);
    if ((reinterpret_cast<uintptr_t>(C) % ob) != 0) return fail(HGEMM_ERR_INVALID_ARG, "C is not element-aligned");
    int cur = -1;
    cudaGetDevice(&cur);
    if (cur != p->device)
        return fail(HGEMM_ERR_INVALID_ARG, "plan was created on device %d but device %d is current", p->device, cur);
    if (C != p->okC) {  // checked once per pointer
        hgemm_status_t pst = hg::check_device_pointer(C, p->device, "C");
        if (pst != HGEMM_OK) return pst;
        p->okC = C;
    }
    cudaError_t e;
    if (p->path == HGEMM_PATH_ZERO_FILL) {
        if (ep.on) {
            e = hg::launch_epilogue_fill(C, p->ldc, p->sC, p->M, p->N, p->batch, out_type(p->dout),
                                         ep, p->num_sms, s);
            return e == cudaSuccess ? HGEMM_OK : cuda_fail(e, "epilogue launch");
        }
        e = hg::launch_zero_fill(C, p->ldc, p->sC, p->M, p->N, p->batch, ob, p->num_sms, s);
        return e == cudaSuccess ? HGEMM_OK : cuda_fail(e, "zero-fill launch");
    }
    if (!A || !B) return fail(HGEMM_ERR_INVALID_ARG, "A or B is NULL");
    if (A != p->okA || B != p->okB) {  // checked once per pointer pair
        hgemm_status_t pst = hg::check_device_pointer(A, p->device, "A");
        if (pst == HGEMM_OK) pst = hg::check_device_pointer(B, p->device, "B");
        if (pst != HGEMM_OK) return pst;
        p->okA = A;
        p->okB = B;
    }
    if (in_bytes(p->din) == 2 &&
        ((reinterpret_cast<uintptr_t>(A) & 1) || (reinterpret_cast<uintptr_t>(B) & 1)))
        return fail(HGEMM_ERR_INVALID_ARG, "A or B is not element-aligned");
    if (is_f8(p->din) && (!aligned16(A) || !aligned16(B)))
        return fail(HGEMM_ERR_UNSUPPORTED, "8-bit A and B must be 16-byte aligned (no copy is made)");

    const bool pack_a = p->ld_repack_a || p->opt.force_repack || !aligned16(A);
    const bool pack_b = p->ld_repack_b || p->opt.force_repack || !aligned16(B);
    hgemm_status_t st = ensure_pack(p, pack_a, pack_b);
    if (st != HGEMM_OK) return st;
    const void *Ae = A;
    const void *Be = B;
    hg::Repack16Job jobs[2];
    int njobs = 0;
    if (pack_a) {
        jobs[njobs++] = hg::Repack16Job{A, p->lda, p->sA, p->ws + p->off_apack, p->lda_p,
                                        p->sA_p, p->M, p->K, p->batch};
        Ae = p->ws + p->off_apack;
    }
    if (pack_b) {
        jobs[njobs++] = hg::Repack16Job{B, p->ldb, p->sB, p->ws + p->off_bpack, p->ldb_p,
                                        p->sB_p, p->opt.trans_b ? p->N : p->K,
                                        p->opt.trans_b ? p->K : p->N, p->batch};
        Be = p->ws + p->off_bpack;
    }
    if (njobs > 0) {  // both copies in one launch
        e = hg::launch_repack16(jobs, njobs, p->num_sms, s);
        if (e != cudaSuccess) return cuda_fail(e, "operand copy launch");
    }
    int32_t *err = reinterpret_cast<int32_t *>(p->ws);
    const uint32_t bf = p->din == HGEMM_BF16 ? 1u : 0u;
    const bool f8 = is_f8(p->din);
    const uint32_t f8fmt = p->din == HGEMM_E5M2 ? 1u : 0u;  // kind::f8f6f4 codes: E4M3 0, E5M2 1
    if (p->path == HGEMM_PATH_TILED) {
        const bool ts = p->ldc_tma && aligned16(C);
        st = encode_maps(p, Ae, Be, C, ts);
        if (st != HGEMM_OK) return st;
        hg::TiledParams tp{};
        tp.M = static_cast<int32_t>(p->M);
        tp.N = static_cast<int32_t>(p->N);
        tp.K = static_cast<int32_t>(p->K);
        tp.batch = static_cast<int32_t>(p->batch);
        tp.num_m = static_cast<int32_t>(ceil_div(p->M, p->pair ? 256 : 128));
        tp.num_n = static_cast<int32_t>(ceil_div(p->N, p->bn));
        tp.num_kb = static_cast<int32_t>(ceil_div(p->K, kblock(p->din)));
        tp.tiles = tp.batch * tp.num_m * tp.num_n;
        // Raster groups: 16 m-tiles, or 8 for pair tiles when there are at
        // least 32 m-tiles.  On GB300 at 8192^3 (32 m-tiles) groups of 8 read
        // 0.94 GB from DRAM per launch against 1.15 GB with 16 (2.09 GB with
        // 32), in the same time; at 4096^3 (16 m-tiles) 8 read 86 MB against
        // 71 MB, also in the same time.
        tp.group_m = p->opt.group_m ? p->opt.group_m : (p->pair && tp.num_m >= 32 ? 8 : 16);
        // B MN-major (stored K x N, N contiguous) or K-major (trans_b: N x K)
        tp.idesc = f8 ? hg::idesc_f8(f8fmt, f8fmt, 0, 0, p->pair ? 256 : 128, static_cast<uint32_t>(p->bn))
                      : hg::idesc_f16(bf, 0, p->opt.trans_b ? 0 : 1, p->pair ? 256 : 128,
                                      static_cast<uint32_t>(p->bn));
        tp.f8 = f8 ? 1 : 0;
        tp.b_kmajor = p->opt.trans_b ? 1 : 0;
        tp.C = C;
        tp.ep = ep;
        tp.epi_warps = ep.on ? p->epi_warps_ep : p->epi_warps;
        tp.ldc = p->ldc;
        tp.strideC = p->sC;
        tp.err = err;
        tp.timeout_ns = p->timeout_ns;
        tp.full_tiles = static_cast<int32_t>(p->pair ? p->full_tiles : tp.tiles);
        tp.tail_split = p->pair ? p->tail_split : 1;
        tp.units = static_cast<int32_t>(p->pair ? p->units : tp.tiles);
        tp.wide_boxes = p->wide ? 1 : 0;
        tp.stream_k = p->stream_k;
        tp.max_seg = p->max_seg;
        tp.partials = reinterpret_cast<float *>(p->ws + p->off_partials);
        tp.tail_sync = reinterpret_cast<int32_t *>(p->ws + p->off_counters);
        tp.withhold_kb = p->pair ? 0 : p->opt.debug_withhold_kb;
        tp.debug = p->opt.debug_checks;
        if (p->pair)
            e = hg::launch_pair(p->bn, p->pair_ks, out_type(p->dout), ts, p->tmA, p->tmB, p->tmC, tp,
                                p->grid, s);
        else
            e = hg::launch_tiled(p->bn, out_type(p->dout), ts, p->tmA, p->tmB, p->tmC, tp, p->grid, s);
        return e == cudaSuccess ? HGEMM_OK : cuda_fail(e, "tiled kernel launch");
    }
    // skinny
    st = encode_maps(p, Ae, Be, C, false);
    if (st != HGEMM_OK) return st;
    hg::SkinnyParams sp{};
    sp.M = static_cast<int32_t>(p->M);
    sp.N = static_cast<int32_t>(p->N);
    sp.K = static_cast<int32_t>(p->K);
    sp.batch = static_cast<int32_t>(p->batch);
    sp.num_tiles = static_cast<int32_t>(ceil_div(p->N, 64 * p->nb));
    sp.num_kb = static_cast<int32_t>(ceil_div(p->K, kblock(p->din)));
    sp.split = p->split;
    sp.kb_per_split = p->kb_per;
    sp.units = sp.batch * sp.split * sp.num_tiles;
    sp.deal = p->skinny_deal ? 1 : 0;
    // default none: on 8 x 28672 x 4096, 4 or 8 stages measured the same as
    // none (38.4-38.7 us back to back), 16 and more slower
    // Automatic (0): 4 stages for 8-bit inputs, whose units stream half the
    // bytes of 16-bit ones, so the first loads' latency weighs twice (GB300,
    // 8 x 28672 x 4096 E4M3: 22.2 us against 23.2 us; 8 stages 23.7 us); none
    // for 16-bit inputs (no change at 4 or 8 stages, slower from 16).
    sp.prefetch = p->opt.skinny_prefetch > 0    ? p->opt.skinny_prefetch
                  : p->opt.skinny_prefetch == 0 ? (is_f8(p->din) ? 4 : 0)
                                                : 0;
    // the MMA's A operand is B^T: MN-major from a K x N B, K-major from an
    // N x K B (trans_b)
    sp.idesc = f8 ? hg::idesc_f8(f8fmt, f8fmt, 0, 0, 128, static_cast<uint32_t>(p->nu))
                  : hg::idesc_f16(bf, p->opt.trans_b ? 0 : 1, 0, 128, static_cast<uint32_t>(p->nu));
    sp.f8 = f8 ? 1 : 0;
    sp.b_kmajor = p->opt.trans_b ? 1 : 0;
    sp.debug = p->opt.debug_checks;
    sp.C = C;
    sp.ep = ep;
    sp.ldc = p->ldc;
    sp.strideC = p->sC;
    sp.partials = reinterpret_cast<float *>(p->ws + p->off_partials);
    sp.counters = reinterpret_cast<int32_t *>(p->ws + p->off_counters);
    sp.err = err;
    sp.timeout_ns = p->timeout_ns;
    e = hg::launch_skinny(p->nu, p->nb, out_type(p->dout), p->tmA, p->tmB, sp, p->grid, s);
    return e == cudaSuccess ? HGEMM_OK : cuda_fail(e, "skinny kernel launch");
}

// Reads the plan's device error word (the plan's stream must be idle):
// HGEMM_ERR_TIMEOUT with the role and barrier when a watchdog fired, after
// clearing the word and any split-K counters the aborted run left behind.
hgemm_status_t read_error_word(hgemm_plan_s *p) {
    if (!p->ws) return HGEMM_OK;
    int32_t word = 0;
    cudaError_t e = cudaMemcpy(&word, p->ws, sizeof(word), cudaMemcpyDeviceToHost);
    if (e != cudaSuccess) return cuda_fail(e, "reading the device error word");
    if (word == 0) return HGEMM_OK;
    cudaMemset(p->ws, 0, p->off_partials);
    return hg::status_from_error_word(word);
}

// ---------------------------------------------------------------- one-shot cache
//
// One plan per (device, arguments, stream): a plan must not run on two streams
// at once (its workspace is shared), so callers on different streams get
// plans of their own.  Each entry's lock keeps two host threads that use the
// same stream from updating the plan's cached tensor maps at the same time;
// their runs are ordered by the stream itself.

using CacheKey = std::tuple<int, int64_t, int64_t, int64_t, int64_t, int64_t, int64_t, int64_t,
                            int64_t, int64_t, int64_t, int, int, uintptr_t>;
struct CacheEntry {
    hgemm_plan_s *plan = nullptr;
    std::mutex mu;
};
std::mutex g_cache_mu;
std::map<CacheKey, std::unique_ptr<CacheEntry>> g_cache;

}  // namespace

extern "C" {

hgemm_status_t hgemm_plan_create(hgemm_plan_t *plan, int64_t M, int64_t N, int64_t K, int64_t lda,
                                 int64_t ldb, int64_t ldc, int64_t batch, int64_t strideA,
                                 int64_t strideB, int64_t strideC, hgemm_dtype_t dtype_in,
                                 hgemm_dtype_t dtype_out) {
    return plan_create(plan, M, N, K, lda, ldb, ldc, batch, strideA, strideB, strideC, dtype_in,
                       dtype_out, nullptr);
}

hgemm_status_t hgemm_plan_create_ex(hgemm_plan_t *plan, int64_t M, int64_t N, int64_t K,
                                    int64_t lda, int64_t ldb, int64_t ldc, int64_t batch,
                                    int64_t strideA, int64_t strideB, int64_t strideC,
                                    hgemm_dtype_t dtype_in, hgemm_dtype_t dtype_out,
                                    const hgemm_options_t *options) {
    return plan_create(plan, M, N, K, lda, ldb, ldc, batch, strideA, strideB, strideC, dtype_in,
                       dtype_out, options);
}

hgemm_status_t hgemm_run(hgemm_plan_t plan, const void *A, const void *B, void *C, void *stream) {
    if (!plan) return fail(HGEMM_ERR_INVALID_ARG, "plan is NULL");
    return plan_run(plan, A, B, C, static_cast<cudaStream_t>(stream));
}

hgemm_status_t hgemm_run_ex(hgemm_plan_t plan, const void *A, const void *B, void *C, void *stream,
                            const hgemm_epilogue_t *epilogue) {
    if (!plan) return fail(HGEMM_ERR_INVALID_ARG, "plan is NULL");
    hg::EpiParams ep{1.f, 0.f, nullptr, nullptr, nullptr, 0, 0};
    if (epilogue) {
        if (epilogue->activation < HGEMM_ACT_NONE || epilogue->activation > HGEMM_ACT_GELU_TANH)
            return fail(HGEMM_ERR_INVALID_ARG, "unknown activation %d", epilogue->activation);
        if (!std::isfinite(epilogue->alpha) || !std::isfinite(epilogue->beta))
            return fail(HGEMM_ERR_INVALID_ARG, "alpha and beta must be finite");
        ep.alpha = epilogue->alpha;
        ep.beta = epilogue->beta;
        ep.bias = epilogue->bias;
        ep.row_scale = epilogue->row_scale;
        ep.col_scale = epilogue->col_scale;
        ep.act = epilogue->activation;
        ep.on = 1;
        // the epilogue's vectors are read by the kernels too: device memory
        // of the plan's GPU, checked once per pointer set
        if (ep.bias != plan->okBias || ep.row_scale != plan->okRow || ep.col_scale != plan->okCol) {
            const struct {
                const float *ptr;
                const char *name;
            } vecs[3] = {{ep.bias, "bias"}, {ep.row_scale, "row_scale"}, {ep.col_scale, "col_scale"}};
            for (const auto &v : vecs) {
                if (!v.ptr) continue;
                hgemm_status_t st = hg::check_device_pointer(v.ptr, plan->device, v.name);
                if (st != HGEMM_OK) return st;
            }
            plan->okBias = ep.bias;
            plan->okRow = ep.row_scale;
            plan->okCol = ep.col_scale;
        }
    }
    return plan_run(plan, A, B, C, static_cast<cudaStream_t>(stream), ep);
}

}  // extern "C"

namespace {

// hgemm_run_host in row chunks: worth it for one large product (batch 1, M
// >= 1024, A and C together >= 16 MB), where the host link, not the kernel,
// sets the time.  M is cut into up to four chunks of a multiple of 256 rows
// (so every chunk starts 16-byte aligned whenever the rows are).  r0[i] is the
// first row of chunk i, r0[n] = M.  (Splitting the last 256 rows off as a
// fifth chunk, to shorten what is left after the last rows of A arrive,
// measured slower on GB300: 4096^3 0.486 against 0.471 ms per call -- a
// 256-row product takes nearly as long as a whole wave.)
bool host_chunking(const hgemm_plan_s *p, int64_t *r0, int &n) {
    if (p->path != HGEMM_PATH_TILED || p->batch != 1 || p->M < 1024 || p->opt.debug_withhold_kb)
        return false;
    const double bytes = static_cast<double>(p->M) * p->K * in_bytes(p->din) +
                         static_cast<double>(p->M) * p->N * out_bytes(p->dout);
    if (bytes < 16e6) return false;
    const int64_t rows = round_up(ceil_div(p->M, 4), 256);
    n = 0;
    for (int64_t r = 0; r < p->M; r += rows) r0[n++] = r;
    r0[n] = p->M;
    return n >= 2;
}

// Copies rows [r0, r0 + rows) of C (batch 1) from the device staging buffer
// to the host on stream s; only the N columns of each row.
cudaError_t copy_c_rows(hgemm_plan_s *p, void *C_host, int64_t r0, int64_t rows, cudaStream_t s) {
    const int ob = out_bytes(p->dout);
    const size_t off = static_cast<size_t>(r0 * p->ldc) * ob;
    if (p->ldc == p->N)
        return cudaMemcpyAsync(static_cast<char *>(C_host) + off, p->dC + off,
                               static_cast<size_t>(rows * p->N) * ob, cudaMemcpyDeviceToHost, s);
    return cudaMemcpy2DAsync(static_cast<char *>(C_host) + off, static_cast<size_t>(p->ldc) * ob,
                             p->dC + off, static_cast<size_t>(p->ldc) * ob,
                             static_cast<size_t>(p->N) * ob, static_cast<size_t>(rows),
                             cudaMemcpyDeviceToHost, s);
}

// The chunked hgemm_run_host.  Three streams: s_in copies B, then the rows of
// A chunk by chunk; the caller's stream runs chunk i's product (a plan of its
// own over rows [r0, r0 + rows) of the staging buffers) once its rows of A
// have arrived; s_out copies chunk i's rows of C back once its product is
// done.  So the copies in, the products and the copies out of different
// chunks overlap (host-to-device and device-to-host use the link's two
// directions).  Everything is ordered after the caller's earlier work on
// `s` (ev_start) and before its later work (ev_done).
hgemm_status_t host_pipeline(hgemm_plan_s *p, const void *A_host, const void *B_host, void *C_host,
                             cudaStream_t s, size_t b_bytes) {
    const int ib = in_bytes(p->din);
    cudaError_t e = cudaSuccess;
    if (!p->s_in) {
        if ((e = cudaStreamCreateWithFlags(&p->s_in, cudaStreamNonBlocking)) != cudaSuccess ||
            (e = cudaStreamCreateWithFlags(&p->s_out, cudaStreamNonBlocking)) != cudaSuccess ||
            (e = cudaEventCreateWithFlags(&p->ev_start, cudaEventDisableTiming)) != cudaSuccess ||
            (e = cudaEventCreateWithFlags(&p->ev_done, cudaEventDisableTiming)) != cudaSuccess)
            return cuda_fail(e, "host pipeline streams");
        for (int i = 0; i < kMaxHostChunks; ++i)
            if ((e = cudaEventCreateWithFlags(&p->ev_a[i], cudaEventDisableTiming)) != cudaSuccess ||
                (e = cudaEventCreateWithFlags(&p->ev_c[i], cudaEventDisableTiming)) != cudaSuccess)
                return cuda_fail(e, "host pipeline events");
    }
    for (int i = 0; i < p->nchunks; ++i) {  // the chunks' plans, made on first use
        if (p->sub[i]) continue;
        const int64_t rows = p->chunk_r0[i + 1] - p->chunk_r0[i];
        for (int j = 0; j < i; ++j)
            if (p->chunk_r0[j + 1] - p->chunk_r0[j] == rows) p->sub[i] = p->sub[j];
        if (p->sub[i]) continue;
        hgemm_status_t st = plan_create(&p->sub[i], rows, p->N, p->K, p->lda, p->ldb, p->ldc, 1, 0, 0,
                                        0, p->din, p->dout, &p->opt);
        if (st != HGEMM_OK) return st;
        p->sub_own[i] = true;
    }
    auto drain = [&] {  // on a failure after work was enqueued: let it finish
        cudaStreamSynchronize(p->s_in);
        cudaStreamSynchronize(p->s_out);
        cudaStreamSynchronize(s);
    };
    if ((e = cudaEventRecord(p->ev_start, s)) != cudaSuccess ||
        (e = cudaStreamWaitEvent(p->s_in, p->ev_start, 0)) != cudaSuccess ||
        (e = cudaStreamWaitEvent(p->s_out, p->ev_start, 0)) != cudaSuccess)
        return cuda_fail(e, "host pipeline ordering");
    if ((e = cudaMemcpyAsync(p->dB, B_host, b_bytes, cudaMemcpyHostToDevice, p->s_in)) != cudaSuccess) {
        drain();
        return cuda_fail(e, "copy B to device");
    }
    for (int i = 0; i < p->nchunks; ++i) {
        const int64_t r0 = p->chunk_r0[i];
        const int64_t rows = p->chunk_r0[i + 1] - r0;
        const size_t off = static_cast<size_t>(r0 * p->lda) * ib;
        const size_t len = static_cast<size_t>(span_elems(rows, p->K, p->lda, 1, 0)) * ib;
        if ((e = cudaMemcpyAsync(p->dA + off, static_cast<const char *>(A_host) + off, len,
                                 cudaMemcpyHostToDevice, p->s_in)) != cudaSuccess ||
            (e = cudaEventRecord(p->ev_a[i], p->s_in)) != cudaSuccess) {
            drain();
            return cuda_fail(e, "copy A to device");
        }
    }
    const int ob = out_bytes(p->dout);
    for (int i = 0; i < p->nchunks; ++i) {
        const int64_t r0 = p->chunk_r0[i];
        const int64_t rows = p->chunk_r0[i + 1] - r0;
        hgemm_plan_s *sub = p->sub[i];
        if ((e = cudaStreamWaitEvent(s, p->ev_a[i], 0)) != cudaSuccess) {
            drain();
            return cuda_fail(e, "host pipeline ordering");
        }
        hgemm_status_t st = plan_run(sub, p->dA + static_cast<size_t>(r0 * p->lda) * ib, p->dB,
                                     p->dC + static_cast<size_t>(r0 * p->ldc) * ob, s);
        if (st != HGEMM_OK) {
            drain();
            return st;
        }
        if ((e = cudaEventRecord(p->ev_c[i], s)) != cudaSuccess ||
            (e = cudaStreamWaitEvent(p->s_out, p->ev_c[i], 0)) != cudaSuccess ||
            (e = copy_c_rows(p, C_host, r0, rows, p->s_out)) != cudaSuccess) {
            drain();
            return cuda_fail(e, "copy C to host");
        }
    }
    if ((e = cudaEventRecord(p->ev_done, p->s_out)) != cudaSuccess ||
        (e = cudaStreamWaitEvent(s, p->ev_done, 0)) != cudaSuccess) {
        drain();
        return cuda_fail(e, "host pipeline ordering");
    }
    if ((e = cudaStreamSynchronize(s)) != cudaSuccess) return cuda_fail(e, "cudaStreamSynchronize");
    // the products ran: a watchdog timeout left C incomplete
    for (int i = 0; i < p->nchunks; ++i) {
        if (!p->sub_own[i]) continue;
        hgemm_status_t st = read_error_word(p->sub[i]);
        if (st != HGEMM_OK) return st;
    }
    return HGEMM_OK;
}

void free_plan(hgemm_plan_s *plan) {
    if (plan->ws) cudaFree(plan->ws);
    if (plan->dA) cudaFree(plan->dA);
    if (plan->dB) cudaFree(plan->dB);
    if (plan->dC) cudaFree(plan->dC);
    for (int i = 0; i < kMaxHostChunks; ++i)
        if (plan->sub_own[i]) free_plan(plan->sub[i]);
    if (plan->s_in) cudaStreamDestroy(plan->s_in);
    if (plan->s_out) cudaStreamDestroy(plan->s_out);
    if (plan->ev_start) cudaEventDestroy(plan->ev_start);
    if (plan->ev_done) cudaEventDestroy(plan->ev_done);
    for (int i = 0; i < kMaxHostChunks; ++i) {
        if (plan->ev_a[i]) cudaEventDestroy(plan->ev_a[i]);
        if (plan->ev_c[i]) cudaEventDestroy(plan->ev_c[i]);
    }
    delete plan;
}

}  // namespace

extern "C" {

hgemm_status_t hgemm_run_host(hgemm_plan_t plan, const void *A_host, const void *B_host, void *C_host,
                              void *stream) {
    if (!plan) return fail(HGEMM_ERR_INVALID_ARG, "plan is NULL");
    hgemm_plan_s *p = plan;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    if (p->path == HGEMM_PATH_EMPTY) return HGEMM_OK;
    if (!C_host || (p->path != HGEMM_PATH_ZERO_FILL && (!A_host || !B_host)))
        return fail(HGEMM_ERR_INVALID_ARG, "host pointer is NULL");
    const int ob = out_bytes(p->dout);
    const int ib = in_bytes(p->din);
    const size_t a_bytes = static_cast<size_t>(span_elems(p->M, p->K, p->lda, p->batch, p->sA)) * ib;
    const size_t b_bytes =
        static_cast<size_t>(p->opt.trans_b ? span_elems(p->N, p->K, p->ldb, p->batch, p->sB)
                                           : span_elems(p->K, p->N, p->ldb, p->batch, p->sB)) * ib;
    const size_t c_bytes = static_cast<size_t>(span_elems(p->M, p->N, p->ldc, p->batch, p->sC)) * ob;
    cudaError_t e;
    auto grow = [&](char **buf, size_t *have, size_t want) -> cudaError_t {
        if (*have >= want) return cudaSuccess;
        if (*buf) cudaFree(*buf);
        *buf = nullptr;
        *have = 0;
        cudaError_t r = cudaMalloc(reinterpret_cast<void **>(buf), want < 16 ? 16 : want);
        if (r == cudaSuccess) *have = want;
        return r;
    };
    if ((e = grow(&p->dA, &p->dA_bytes, a_bytes)) != cudaSuccess) return cuda_fail(e, "cudaMalloc(A staging)");
    if ((e = grow(&p->dB, &p->dB_bytes, b_bytes)) != cudaSuccess) return cuda_fail(e, "cudaMalloc(B staging)");
    if ((e = grow(&p->dC, &p->dC_bytes, c_bytes)) != cudaSuccess) return cuda_fail(e, "cudaMalloc(C staging)");
    if (host_chunking(p, p->chunk_r0, p->nchunks))
        return host_pipeline(p, A_host, B_host, C_host, s, b_bytes);
    if (p->path != HGEMM_PATH_ZERO_FILL) {
        if ((e = cudaMemcpyAsync(p->dA, A_host, a_bytes, cudaMemcpyHostToDevice, s)) != cudaSuccess)
            return cuda_fail(e, "copy A to device");
        if ((e = cudaMemcpyAsync(p->dB, B_host, b_bytes, cudaMemcpyHostToDevice, s)) != cudaSuccess)
            return cuda_fail(e, "copy B to device");
    }
    hgemm_status_t st = plan_run(p, p->dA, p->dB, p->dC, s);
    if (st != HGEMM_OK) return st;
    // copy back only the M x N block of each batch: host elements between rows stay intact.
    // Batches stacked at the row pitch (strideC = M * ldc) are one 2-D copy of batch * M
    // rows, and rows without padding (ldc = N) one contiguous copy.
    const bool stacked = p->batch == 1 || p->sC == p->M * p->ldc;
    if (stacked && p->ldc == p->N) {
        e = cudaMemcpyAsync(C_host, p->dC, static_cast<size_t>(p->batch * p->M * p->N) * ob,
                            cudaMemcpyDeviceToHost, s);
        if (e != cudaSuccess) return cuda_fail(e, "copy C to host");
    } else {
        const int64_t copies = stacked ? 1 : p->batch;
        const int64_t rows = stacked ? p->batch * p->M : p->M;
        for (int64_t b = 0; b < copies; ++b) {
            const size_t off = static_cast<size_t>(b * p->sC) * ob;
            e = cudaMemcpy2DAsync(static_cast<char *>(C_host) + off, static_cast<size_t>(p->ldc) * ob,
                                  p->dC + off, static_cast<size_t>(p->ldc) * ob,
                                  static_cast<size_t>(p->N) * ob, static_cast<size_t>(rows),
                                  cudaMemcpyDeviceToHost, s);
            if (e != cudaSuccess) return cuda_fail(e, "copy C to host");
        }
    }
    e = cudaStreamSynchronize(s);
    if (e != cudaSuccess) return cuda_fail(e, "cudaStreamSynchronize");
    // the product ran: a watchdog timeout left C incomplete
    return read_error_word(p);
}

hgemm_status_t hgemm_check(hgemm_plan_t plan, void *stream) {
    if (!plan) return fail(HGEMM_ERR_INVALID_ARG, "plan is NULL");
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    cudaError_t e = cudaStreamSynchronize(s);
    if (e != cudaSuccess) return cuda_fail(e, "stream reports an error");
    return read_error_word(plan);
}

hgemm_status_t hgemm_plan_destroy(hgemm_plan_t plan) {
    if (!plan) return HGEMM_OK;
    free_plan(plan);
    return HGEMM_OK;
}

hgemm_status_t hgemm_plan_get_info(hgemm_plan_t plan, hgemm_plan_info_t *info) {
    if (!plan || !info) return fail(HGEMM_ERR_INVALID_ARG, "plan or info is NULL");
    hgemm_plan_info_t r{};
    r.path = plan->path;
    r.tile_k = kblock(plan->din);
    r.split_k = 1;
    if (plan->path == HGEMM_PATH_TILED) {
        r.tile_m = plan->pair ? 256 : 128;
        r.tile_n = plan->bn;
        r.stages = plan->pair ? hg::pair_stages(plan->pair_ks) : hg::tiled_stages(plan->bn, plan->epi_warps);
        r.epi_warps = plan->pair ? 4 : plan->epi_warps;
        r.epi_warps_epilogue = plan->pair ? 4 : plan->epi_warps_ep;
        if (plan->pair) r.tile_k = kblock(plan->din) * plan->pair_ks;
        r.tma_store = plan->ldc_tma ? 1 : 0;
    } else if (plan->path == HGEMM_PATH_SKINNY) {
        r.tile_m = plan->nu;
        r.tile_n = 64 * plan->nb;
        r.stages = hg::skinny_stages(plan->nu, plan->nb);
        r.split_k = plan->split;
    }
    r.grid = plan->grid;
    const bool busy = plan->path == HGEMM_PATH_TILED || plan->path == HGEMM_PATH_SKINNY;
    r.repack_a = (busy && (plan->ld_repack_a || plan->opt.force_repack)) ? 1 : 0;
    r.repack_b = (busy && (plan->ld_repack_b || plan->opt.force_repack)) ? 1 : 0;
    r.kernels_per_run = plan->path == HGEMM_PATH_EMPTY ? 0 : 1 + ((r.repack_a || r.repack_b) ? 1 : 0);
    if (plan->path == HGEMM_PATH_ZERO_FILL) r.kernels_per_run = 1;
    r.workspace_bytes = static_cast<int64_t>(plan->ws_bytes);
    int64_t r0[kMaxHostChunks + 1];
    int nchunks = 1;
    r.host_chunks = host_chunking(plan, r0, nchunks) ? nchunks : 1;
    r.tail_split = plan->path == HGEMM_PATH_TILED && plan->pair ? plan->tail_split : 1;
    r.trans_b = plan->opt.trans_b;
    r.stream_k = plan->path == HGEMM_PATH_TILED && plan->pair ? plan->stream_k
                 : plan->path == HGEMM_PATH_SKINNY && plan->skinny_deal ? 1
                                                                       : 0;
    // before the first run: as the plan's own copies (leading dimensions)
    // decide; after it: what the last run used
    r.wide_boxes = plan->maps_ok ? (plan->wide ? 1 : 0)
                                 : (wide_dims(plan, r.repack_a != 0, r.repack_b != 0).ok ? 1 : 0);
    *info = r;
    return HGEMM_OK;
}

hgemm_status_t hgemm(const void *A, const void *B, void *C, int64_t M, int64_t N, int64_t K,
                     int64_t lda, int64_t ldb, int64_t ldc, int64_t batch, int64_t strideA,
                     int64_t strideB, int64_t strideC, hgemm_dtype_t dtype_in,
                     hgemm_dtype_t dtype_out, void *stream) {
    int dev = 0;
    cudaGetDevice(&dev);
    CacheKey key{dev, M, N, K, lda, ldb, ldc, batch, batch > 1 ? strideA : 0,
                 batch > 1 ? strideB : 0, batch > 1 ? strideC : 0, static_cast<int>(dtype_in),
                 static_cast<int>(dtype_out), reinterpret_cast<uintptr_t>(stream)};
    CacheEntry *entry = nullptr;
    {
        std::lock_guard<std::mutex> g(g_cache_mu);
        auto it = g_cache.find(key);
        if (it != g_cache.end()) {
            entry = it->second.get();
        } else {
            hgemm_plan_s *p = nullptr;
            hgemm_status_t st = plan_create(&p, M, N, K, lda, ldb, ldc, batch, strideA, strideB,
                                            strideC, dtype_in, dtype_out, nullptr);
            if (st != HGEMM_OK) return st;
            auto e = std::make_unique<CacheEntry>();
            e->plan = p;
            entry = e.get();
            g_cache[key] = std::move(e);
        }
    }
    std::lock_guard<std::mutex> g(entry->mu);
    return plan_run(entry->plan, A, B, C, static_cast<cudaStream_t>(stream));
}

hgemm_status_t hgemm_cache_clear(void) {
    std::lock_guard<std::mutex> g(g_cache_mu);
    for (auto &kv : g_cache) hgemm_plan_destroy(kv.second->plan);
    g_cache.clear();
    return HGEMM_OK;
}

hgemm_status_t hgemm_watchdog_selftest(uint64_t timeout_ns, void *stream, int32_t *device_code) {
    if (!device_code) return fail(HGEMM_ERR_INVALID_ARG, "device_code is NULL");
    *device_code = 0;
    int32_t *err = nullptr;
    cudaError_t e = cudaMalloc(reinterpret_cast<void **>(&err), sizeof(int32_t));
    if (e != cudaSuccess) return cuda_fail(e, "cudaMalloc(error word)");
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    e = cudaMemsetAsync(err, 0, sizeof(int32_t), s);
    if (e == cudaSuccess) e = hg::launch_watchdog_selftest(err, timeout_ns, s);
    if (e == cudaSuccess) e = cudaMemcpyAsync(device_code, err, sizeof(int32_t), cudaMemcpyDeviceToHost, s);
    if (e == cudaSuccess) e = cudaStreamSynchronize(s);
    cudaFree(err);
    if (e != cudaSuccess) return cuda_fail(e, "watchdog self-test");
    if (*device_code != 0) return fail(HGEMM_ERR_TIMEOUT, "watchdog fired (code 0x%08x)", static_cast<uint32_t>(*device_code));
    return HGEMM_OK;
}

const char *hgemm_status_string(hgemm_status_t s) {
    switch (s) {
        case HGEMM_OK: return "HGEMM_OK";
        case HGEMM_ERR_INVALID_ARG: return "HGEMM_ERR_INVALID_ARG";
        case HGEMM_ERR_UNSUPPORTED: return "HGEMM_ERR_UNSUPPORTED";
        case HGEMM_ERR_NO_DEVICE: return "HGEMM_ERR_NO_DEVICE";
        case HGEMM_ERR_CUDA: return "HGEMM_ERR_CUDA";
        case HGEMM_ERR_OOM: return "HGEMM_ERR_OOM";
        case HGEMM_ERR_TIMEOUT: return "HGEMM_ERR_TIMEOUT";
        case HGEMM_ERR_INTERNAL: return "HGEMM_ERR_INTERNAL";
        default: return "HGEMM_ERR_UNKNOWN";
    }
}

const char *hgemm_last_error_detail(void) { return g_detail.c_str(); }

int32_t hgemm_version(void) { return 100; }

}  // extern "C"

// ---------------------------------------------------------------- internal helpers
// Thin wrappers over the helpers above for other translation units of the
// library (noalloc.cu); declared in internal.h.
namespace hg {

hgemm_status_t encode_map_3d(CUtensorMap *map, const void *base, int bf16, int64_t cols,
                             int64_t rows, int64_t ld, uint32_t box_cols, uint32_t box_rows) {
    return encode_3d(map, base,
                     bf16 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16 : CU_TENSOR_MAP_DATA_TYPE_FLOAT16, 2,
                     cols, rows, 1, ld, 0, box_cols, box_rows);
}

hgemm_status_t encode_map_batched(CUtensorMap *map, const void *base, int bf16, int64_t cols,
                                  int64_t rows, int64_t batch, int64_t ld, int64_t stride,
                                  uint32_t box_cols, uint32_t box_rows) {
    return encode_3d(map, base,
                     bf16 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16 : CU_TENSOR_MAP_DATA_TYPE_FLOAT16, 2,
                     cols, rows, batch, ld, stride, box_cols, box_rows);
}

int pick_split(int64_t work_tiles, int num_kb, int num_sms) {
    return choose_split(work_tiles, num_kb, num_sms);
}

int pick_skinny_nb(int64_t N, int64_t batch, int num_sms) {
    // Columns per work unit: each K row of B is read in runs of 128 x nb
    // contiguous bytes, and the units of one wave read the same rows.
    // Measured on 8 x 28672 x 4096 (back to back, best of 5): 256-column
    // units (112 CTAs) 37.8-38.5 us; 192-column units (150 CTAs, the grid
    // cuBLAS uses) 40.2 us; 384 with split 2 44.4 us; 128-column units
    // unsplit 49.4 us (224 units = 1.5 waves); 512-column units 49.5 us
    // (only 56 CTAs busy).  Narrow products keep 128 columns so that more
    // units exist, and split K to fill the SMs.
    (void)batch;
    (void)num_sms;
    return N >= 4096 ? 4 : 2;
}

hgemm_status_t set_error_detail(hgemm_status_t s, const char *msg) { return fail(s, "%s", msg); }

hgemm_status_t check_device_pointer(const void *ptr, int device, const char *what) {
    cudaPointerAttributes a{};
    cudaError_t e = cudaPointerGetAttributes(&a, ptr);
    if (e != cudaSuccess) {
        cudaGetLastError();  // the query's error is not the caller's
        return fail(HGEMM_ERR_INVALID_ARG, "%s (%p) is not a pointer CUDA knows: %s", what, ptr,
                    cudaGetErrorString(e));
    }
    if (a.type == cudaMemoryTypeManaged) return HGEMM_OK;
    if (a.type == cudaMemoryTypeDevice && a.device == device) return HGEMM_OK;
    if (a.type == cudaMemoryTypeDevice)
        return fail(HGEMM_ERR_INVALID_ARG, "%s (%p) is memory of device %d, not of the plan's device %d",
                    what, ptr, a.device, device);
    return fail(HGEMM_ERR_INVALID_ARG, "%s (%p) is host memory; device pointers are required "
                "(hgemm_run_host takes host buffers)", what, ptr);
}

hgemm_status_t status_from_error_word(int32_t word) {
    if (word == 0) return HGEMM_OK;
    const unsigned role = (static_cast<uint32_t>(word) >> 16) & 0xFFu;
    const unsigned idx = static_cast<uint32_t>(word) & 0xFFFFu;
    if ((static_cast<uint32_t>(word) & 0xC0000000u) == 0x40000000u) {
        static const char *kernels[] = {"?", "single-CTA tiled", "CTA-pair", "skinny"};
        static const char *checks[] = {"?", "tile outside the output", "K range outside K",
                                       "piece outside its tile"};
        return fail(HGEMM_ERR_INTERNAL, "device invariant check failed: %s kernel, %s (code 0x%08x)",
                    role < 4 ? kernels[role] : "?", idx < 4 ? checks[idx] : "?",
                    static_cast<uint32_t>(word));
    }
    static const char *names[] = {"?", "TMA producer", "MMA issuer", "epilogue", "drain", "self-test"};
    return fail(HGEMM_ERR_TIMEOUT, "device wait timed out: role %s, barrier %u (code 0x%08x)",
                role < 6 ? names[role] : "?", idx, static_cast<uint32_t>(word));
}

}  // namespace hg
