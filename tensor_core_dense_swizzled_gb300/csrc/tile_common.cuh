// tile_common.cuh -- device helpers shared by the tiled GEMM kernels: the
// grouped tile raster, 16-byte shared-memory stores for the epilogue staging,
// and the fp32 -> fp16/bf16 conversions (round to nearest even, as the
// "tensor-cores-cutlass-and-cute" Ampere epilogue does with
// __floats2bfloat162_rn, section 四.3).
#pragma once

#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <stdint.h>

#include "kernels.h"
#include "ptx.cuh"

namespace hg {

// Tile t of a batch of num_m x num_n tiles, in groups of `group_m` m-tiles:
// within a group the m index runs fastest, so the tiles that concurrently
// running CTAs work on share a few rows of A and columns of B in L2
// (tile order is one of the gaps listed in "tensor-cores-cutlass-and-cute"
// section 四.5).
__device__ __forceinline__ void grouped_tile(int t, int num_m, int num_n, int group_m, int &b,
                                             int &mt, int &nt) {
    const int per_batch = num_m * num_n;
    b = t / per_batch;
    const int r = t - b * per_batch;
    const int span = group_m * num_n;
    const int g = r / span;
    const int first_m = g * group_m;
    const int gsz = min(num_m - first_m, group_m);
    const int rr = r - g * span;
    mt = first_m + rr % gsz;
    nt = rr / gsz;
}

__device__ __forceinline__ void st_shared_v4(uint32_t addr, uint32_t a, uint32_t b, uint32_t c,
                                             uint32_t d) {
    asm volatile("st.shared.v4.b32 [%0], {%1, %2, %3, %4};" ::"r"(addr), "r"(a), "r"(b), "r"(c),
                 "r"(d)
                 : "memory");
}

__device__ __forceinline__ void st_shared_b32(uint32_t addr, uint32_t v) {
    asm volatile("st.shared.b32 [%0], %1;" ::"r"(addr), "r"(v) : "memory");
}

__device__ __forceinline__ uint32_t ld_shared_b32(uint32_t addr) {
    uint32_t v;
    asm volatile("ld.shared.b32 %0, [%1];" : "=r"(v) : "r"(addr) : "memory");
    return v;
}

template <int OUT>
__device__ __forceinline__ uint32_t pack2(uint32_t lo, uint32_t hi) {
    const float a = __uint_as_float(lo), b = __uint_as_float(hi);
    if constexpr (OUT == OUT_BF16) {
        __nv_bfloat162 h = __floats2bfloat162_rn(a, b);
        return *reinterpret_cast<uint32_t *>(&h);
    } else {
        __half2 h = __floats2half2_rn(a, b);
        return *reinterpret_cast<uint32_t *>(&h);
    }
}

template <int OUT>
__device__ __forceinline__ void store_one(void *C, int64_t idx, float v) {
    if constexpr (OUT == OUT_F32) {
        static_cast<float *>(C)[idx] = v;
    } else if constexpr (OUT == OUT_BF16) {
        static_cast<__nv_bfloat16 *>(C)[idx] = __float2bfloat16_rn(v);
    } else {
        static_cast<__half *>(C)[idx] = __float2half_rn(v);
    }
}

// Launches `kern` on `stream` with programmatic stream serialization: the
// kernel may be scheduled while the previous kernel of the stream finishes;
// it calls griddep_wait() before reading memory (see ptx.cuh).
template <typename Kernel, typename... Args>
cudaError_t launch_dependent(Kernel kern, int grid, int threads, int smem, cudaStream_t stream,
                             const Args &...args) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(static_cast<unsigned>(grid), 1, 1);
    cfg.blockDim = dim3(static_cast<unsigned>(threads), 1, 1);
    cfg.dynamicSmemBytes = static_cast<size_t>(smem);
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, kern, args...);
}

// Epilogue staging: each epilogue warp owns EPI_STG_BUFS x EPI_STG_BYTES of
// shared memory, used as pieces of 32 rows x 32 columns: two of 4 KB for fp32
// output, four of 2 KB for fp16/bf16 (more TMA stores in flight: the drain
// of a tile waits on stores still reading their pieces).
constexpr int EPI_STG_BYTES = 4096;
constexpr int EPI_STG_BUFS = 2;
template <int OUT>
struct EpiPiece {
    static constexpr int BYTES = OUT == OUT_F32 ? 4096 : 2048;
};

struct EpiArgs {
    const CUtensorMap *tmC;  // TMA-store path
    void *C;                 // predicated-store path; C's previous values (beta != 0)
    int64_t ldc, strideC;
    int32_t M, N;
    EpiParams ep;
};

// tanh via the hardware approximation (MUFU, relative error about 2^-11).
__device__ __forceinline__ float tanh_approx(float x) {
    float y;
    asm("tanh.approx.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}

// GELU in the erf form, x * Phi(x) = 0.5 x (1 + erf(x / sqrt 2)), with erf
// from Abramowitz & Stegun, Handbook of Mathematical Functions, formula
// 7.1.26: for z >= 0, erf(z) = 1 - q(z), q = (a1 t + ... + a5 t^5) e^(-z^2),
// t = 1 / (1 + p z), absolute error <= 1.5e-7 (plus fp32 rounding and the
// SFU's ex2 and the reciprocal); erf is odd.
__device__ __forceinline__ float gelu_erf(float x) {
    const float z = fabsf(x) * 0.70710678118654752f;
    float t;
    asm("rcp.approx.ftz.f32 %0, %1;" : "=f"(t) : "f"(fmaf(0.3275911f, z, 1.f)));
    float poly = fmaf(1.061405429f, t, -1.453152027f);
    poly = fmaf(poly, t, 1.421413741f);
    poly = fmaf(poly, t, -0.284496736f);
    poly = fmaf(poly, t, 0.254829592f);
    poly *= t;
    float e;
    asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(e) : "f"(-z * z * 1.4426950408889634f));
    const float q = poly * e;  // 1 - erf(|x| / sqrt 2)
    return 0.5f * x * (x >= 0.f ? 2.f - q : q);
}

// Activation of the fused epilogue: 1 ReLU; 2 GELU in the erf form
// x * Phi(x) = 0.5 x (1 + erf(x / sqrt 2)); 3 GELU in the tanh form
// 0.5 x (1 + tanh(sqrt(2 / pi) (x + 0.044715 x^3))).
__device__ __forceinline__ float epi_act(float x, int act) {
    if (act == 1) return fmaxf(x, 0.f);
    if (act == 2) return gelu_erf(x);
    if (act == 3) {
        const float u = 0.7978845608028654f * fmaf(0.044715f * x, x * x, x);
        return 0.5f * x * (1.f + tanh_approx(u));
    }
    return x;
}

// D = act(alpha * rs * cs * acc + beta * c_prev + bias), fp32.
__device__ __forceinline__ float epi_value(const EpiParams &ep, float acc, float rs, float cs,
                                           float bias, float c_prev) {
    float t = ep.alpha * rs * cs * acc;
    if (ep.beta != 0.f) t = fmaf(ep.beta, c_prev, t);
    return epi_act(t + bias, ep.act);
}

template <int OUT>
__device__ __forceinline__ float load_one(const void *C, int64_t idx) {
    if constexpr (OUT == OUT_F32) {
        return static_cast<const float *>(C)[idx];
    } else if constexpr (OUT == OUT_BF16) {
        return __bfloat162float(static_cast<const __nv_bfloat16 *>(C)[idx]);
    } else {
        return __half2float(static_cast<const __half *>(C)[idx]);
    }
}

// Unpacks two 16-bit values of the output type to floats.
template <int OUT>
__device__ __forceinline__ void unpack2(uint32_t w, float &lo, float &hi) {
    if constexpr (OUT == OUT_BF16) {
        __nv_bfloat162 h = *reinterpret_cast<__nv_bfloat162 *>(&w);
        lo = __low2float(h);
        hi = __high2float(h);
    } else {
        __half2 h = *reinterpret_cast<__half2 *>(&w);
        lo = __low2float(h);
        hi = __high2float(h);
    }
}

// Applies the fused epilogue to one lane's 32 values of row `row`, columns
// col .. col+31 (lane = row; the TMA-store path: rows of C are 16-byte
// multiples and so is N * sizeof(out), so C's previous values are read as
// 16-byte vectors that never cross column N).  The column vectors are read
// once per chunk, element l by lane l, and handed to every lane by shuffles.
template <int OUT>
__device__ __forceinline__ void epi_row(uint32_t (&v)[32], int row, int col, int b,
                                        const EpiArgs &e) {
    const EpiParams &ep = e.ep;
    const int lane = threadIdx.x & 31;
    const bool row_in = row < e.M;
    const float rs = (ep.row_scale && row_in) ? __ldg(ep.row_scale + row) : 1.f;
    const bool lin = col + lane < e.N;
    const float cs_l = (ep.col_scale && lin) ? __ldg(ep.col_scale + col + lane) : 1.f;
    const float bias_l = (ep.bias && lin) ? __ldg(ep.bias + col + lane) : 0.f;
    const float arow = ep.alpha * rs;
    if (ep.beta != 0.f) {
        // C's previous values: every load of the chunk issued before any is
        // used (one memory round trip per chunk)
        const int64_t off = static_cast<int64_t>(b) * e.strideC + static_cast<int64_t>(row) * e.ldc + col;
        uint4 raw[OUT == OUT_F32 ? 8 : 4];
        constexpr int NV = OUT == OUT_F32 ? 8 : 4;  // 16-byte vectors per 32 columns
        constexpr int EPV = 32 / NV;                // elements per vector
#pragma unroll
        for (int q = 0; q < NV; ++q) {
            raw[q] = make_uint4(0u, 0u, 0u, 0u);
            if (row_in && col + EPV * q < e.N)
                raw[q] = *(reinterpret_cast<const uint4 *>(static_cast<const char *>(e.C) +
                                                           off * (OUT == OUT_F32 ? 4 : 2)) + q);
        }
#pragma unroll
        for (int q = 0; q < NV; ++q) {
            float prev[EPV];
            if constexpr (OUT == OUT_F32) {
                prev[0] = __uint_as_float(raw[q].x);
                prev[1] = __uint_as_float(raw[q].y);
                prev[2] = __uint_as_float(raw[q].z);
                prev[3] = __uint_as_float(raw[q].w);
            } else {
                unpack2<OUT>(raw[q].x, prev[0], prev[1]);
                unpack2<OUT>(raw[q].y, prev[2], prev[3]);
                unpack2<OUT>(raw[q].z, prev[4], prev[5]);
                unpack2<OUT>(raw[q].w, prev[6], prev[7]);
            }
#pragma unroll
            for (int j = 0; j < EPV; ++j) {
                const int jj = EPV * q + j;
                const float cs = __shfl_sync(0xFFFFFFFFu, cs_l, jj);
                const float bias = __shfl_sync(0xFFFFFFFFu, bias_l, jj);
                const float t = fmaf(ep.beta, prev[j], arow * cs * __uint_as_float(v[jj]));
                v[jj] = __float_as_uint(epi_act(t + bias, ep.act));
            }
        }
    } else {
#pragma unroll
        for (int jj = 0; jj < 32; ++jj) {
            const float cs = __shfl_sync(0xFFFFFFFFu, cs_l, jj);
            const float bias = __shfl_sync(0xFFFFFFFFu, bias_l, jj);
            v[jj] = __float_as_uint(epi_act(arow * cs * __uint_as_float(v[jj]) + bias, ep.act));
        }
    }
}

// beta != 0: asks L2 for C's previous values of row `row`, columns col0 ..
// col0 + ncols - 1 (clipped to the matrix), while the accumulator of the tile
// is still being computed, so that the epilogue's reads of them hit L2
// instead of waiting on DRAM chunk by chunk.
template <int OUT>
__device__ __forceinline__ void prefetch_c_prev(const EpiArgs &e, int row, int col0, int ncols, int b) {
    if (e.ep.beta == 0.f || row >= e.M) return;
    constexpr int OB = OUT == OUT_F32 ? 4 : 2;
    const int cols = min(ncols, e.N - col0);
    if (cols <= 0) return;
    const char *rowp = static_cast<const char *>(e.C) +
                       (static_cast<int64_t>(b) * e.strideC + static_cast<int64_t>(row) * e.ldc + col0) * OB;
    for (int off = 0; off < cols * OB; off += 128)
        asm volatile("prefetch.global.L2 [%0];" ::"l"(rowp + off));
}

// Converts 32 fp32 columns (chunk c of a warp's 32 rows, lane = row) and
// stores them into C: TMA_STORE through the warp's swizzled staging pieces
// (fp32 rows of 128 bytes: chunk j of row r at j ^ (r & 7); fp16/bf16 rows of
// 64 bytes: chunk j at j ^ ((r >> 1) & 3), the 64-byte-row swizzle of
// "tensor-cores-cutlass-and-cute" section 三.5) and one TMA store by lane 0
// -- the C map clips rows >= M and columns >= N (it is only used when
// N * sizeof(out) is a multiple of 16 bytes); otherwise the 32 x 32 piece is
// transposed through shared memory (element (r, c) at r*32 + (c ^ r):
// conflict-free both ways) and lane l writes column l of every row with
// predicated, coalesced stores.
// EPI: the fused epilogue (e.ep) is applied first; a separate kernel variant
// so that plain products carry none of its code or registers.
template <int OUT, bool TMA_STORE, bool EPI>
__device__ __forceinline__ void store_chunk(uint32_t (&v)[32], int c, uint32_t stg, int &sbuf, int row0, int col0, int b,
                                            const EpiArgs &e) {
    const int lane = threadIdx.x & 31;
    if constexpr (TMA_STORE) {
        if constexpr (EPI) epi_row<OUT>(v, row0 + lane, col0 + c * 32, b, e);
        constexpr int PIECE = EpiPiece<OUT>::BYTES;
        constexpr int NPIECE = EPI_STG_BUFS * EPI_STG_BYTES / PIECE;
        if (lane == 0) bulk_wait_read<NPIECE - 1>();
        __syncwarp();
        const uint32_t piece = stg + sbuf * PIECE;
        if constexpr (OUT == OUT_F32) {
            const uint32_t row_addr = piece + lane * 128;
#pragma unroll
            for (int j = 0; j < 8; ++j)
                st_shared_v4(row_addr + ((j ^ (lane & 7)) << 4), v[4 * j], v[4 * j + 1],
                             v[4 * j + 2], v[4 * j + 3]);
        } else {
            uint32_t pk[16];
#pragma unroll
            for (int i = 0; i < 16; ++i) pk[i] = pack2<OUT>(v[2 * i], v[2 * i + 1]);
            const uint32_t row_addr = piece + lane * 64;
#pragma unroll
            for (int j = 0; j < 4; ++j)
                st_shared_v4(row_addr + ((j ^ ((lane >> 1) & 3)) << 4), pk[4 * j], pk[4 * j + 1],
                             pk[4 * j + 2], pk[4 * j + 3]);
        }
        fence_proxy_async_smem();
        __syncwarp();
        if (lane == 0) {
            tma_store_3d(e.tmC, piece, col0 + c * 32, row0, b);
            bulk_commit();
        }
        sbuf = (sbuf + 1 == NPIECE) ? 0 : sbuf + 1;
    } else {
        // The piece goes through the warp's staging area transposed (element
        // (r, c) at r*32 + (c ^ r), conflict-free both ways), so that lane l
        // then holds column l of the 32 rows and each store instruction writes
        // one row's 32 consecutive elements.  Rows are handled in groups of
        // 16 (8 with the fused epilogue): a group's values (and its previous
        // C values) are all read before its first store -- as far as the
        // compiler knows a store to C may alias a later load, so loads and
        // stores interleaved row by row ran as 32 dependent round trips
        // (about 12 us per 128 x 256 tile on GB300, against 3.4 us for the
        // TMA-store path).
        __syncwarp();
#pragma unroll
        for (int j = 0; j < 32; ++j) st_shared_b32(stg + 4u * (lane * 32 + (j ^ lane)), v[j]);
        __syncwarp();
        const int col = col0 + c * 32 + lane;
        const int nrows = min(32, e.M - row0);  // rows of the piece inside C
        const bool live = col < e.N && nrows > 0;
        constexpr int OB = OUT == OUT_F32 ? 4 : 2;
        char *p0 = live ? static_cast<char *>(e.C) + (static_cast<int64_t>(b) * e.strideC +
                                                      static_cast<int64_t>(row0) * e.ldc + col) * OB
                        : nullptr;
        const int64_t rstep = e.ldc * OB;
        float cs = 1.f, bias = 0.f;
        if constexpr (EPI) {
            if (live && e.ep.col_scale) cs = __ldg(e.ep.col_scale + col);
            if (live && e.ep.bias) bias = __ldg(e.ep.bias + col);
        }
        constexpr int GR = EPI ? 8 : 16;  // rows per group (registers)
#pragma unroll
        for (int g = 0; g < 32; g += GR) {
            float x[GR];
#pragma unroll
            for (int r = 0; r < GR; ++r)
                x[r] = __uint_as_float(ld_shared_b32(stg + 4u * ((g + r) * 32 + (lane ^ (g + r)))));
            if (!live) continue;
            if constexpr (EPI) {
                const EpiParams &ep = e.ep;
                float rs[GR], prev[GR];
#pragma unroll
                for (int r = 0; r < GR; ++r) {
                    const bool in = g + r < nrows;
                    rs[r] = (ep.row_scale && in) ? __ldg(ep.row_scale + row0 + g + r) : 1.f;
                    prev[r] = (ep.beta != 0.f && in) ? load_one<OUT>(p0 + (g + r) * rstep, 0) : 0.f;
                }
#pragma unroll
                for (int r = 0; r < GR; ++r)
                    if (g + r < nrows)
                        store_one<OUT>(p0 + (g + r) * rstep, 0, epi_value(ep, x[r], rs[r], cs, bias, prev[r]));
            } else {
#pragma unroll
                for (int r = 0; r < GR; ++r)
                    if (g + r < nrows) store_one<OUT>(p0 + (g + r) * rstep, 0, x[r]);
            }
        }
    }
}

// One epilogue warp drains its 32 TMEM lanes (output rows row0..row0+31) x
// NCOLS fp32 columns of one accumulator, starting at TMEM address `tbase`,
// into C columns col0.. of batch b.  `release()` runs once the last column
// is in registers, so the MMA issuer can reuse the accumulator while the
// stores drain.
//
// Each 32-column chunk is stored by store_chunk.
//
// ADD: `addend` holds another fp32 partial of the same 32 rows in the layout
// spill_accumulator writes; it is added to the accumulator (own + addend)
// before the conversion.
template <int OUT, bool TMA_STORE, int NCOLS, bool ADD = false, bool EPI = false, typename Release>
__device__ __forceinline__ void drain_accumulator(uint32_t tbase, uint32_t stg,
                                                  int &sbuf, int row0, int col0, int b,
                                                  const EpiArgs &e, Release release,
                                                  const float *addend = nullptr, int c_lo = 0,
                                                  int c_hi = NCOLS / 32) {
    static_assert(NCOLS % 32 == 0, "32-column pieces");
    const int lane = threadIdx.x & 31;
    // Chunks [c_lo, c_hi) of the accumulator; `addend` holds chunk c_lo first.
    // ADD: the addend of chunk c+1 is loaded while chunk c is processed, so
    // only the first L2 round trip is exposed.
    float4 nxt[ADD ? 8 : 1];
    if constexpr (ADD) {
        const float4 *src = reinterpret_cast<const float4 *>(addend) + lane;
#pragma unroll
        for (int j = 0; j < 8; ++j) nxt[j] = __ldcg(src + j * 32);
    }
    // TMEM loads run one chunk ahead: chunk c+1 is in flight while chunk c is
    // converted, staged and stored.
    uint32_t v[32], vn[32];
    tmem_ld32_issue(tbase + c_lo * 32, vn);
#pragma unroll 1
    for (int c = c_lo; c < c_hi; ++c) {
        tmem_ld32_wait(vn);
#pragma unroll
        for (int i = 0; i < 32; ++i) v[i] = vn[i];
        if (c + 1 < c_hi) {
            tmem_ld32_issue(tbase + (c + 1) * 32, vn);
        } else {
            tc_fence_before();
            __syncwarp();
            release();
        }
        if constexpr (ADD) {
            float4 cur[8];
#pragma unroll
            for (int j = 0; j < 8; ++j) cur[j] = nxt[j];
            if (c + 1 < c_hi) {
                const float4 *src =
                    reinterpret_cast<const float4 *>(addend + (c + 1 - c_lo) * 1024) + lane;
#pragma unroll
                for (int j = 0; j < 8; ++j) nxt[j] = __ldcg(src + j * 32);
            }
#pragma unroll
            for (int j = 0; j < 8; ++j) {
                const float4 a = cur[j];
                v[4 * j] = __float_as_uint(__uint_as_float(v[4 * j]) + a.x);
                v[4 * j + 1] = __float_as_uint(__uint_as_float(v[4 * j + 1]) + a.y);
                v[4 * j + 2] = __float_as_uint(__uint_as_float(v[4 * j + 2]) + a.z);
                v[4 * j + 3] = __float_as_uint(__uint_as_float(v[4 * j + 3]) + a.w);
            }
        }
        store_chunk<OUT, TMA_STORE, EPI>(v, c, stg, sbuf, row0, col0, b, e);
    }
}

// Sums nseg fp32 partials of one warp's 32 rows x NCOLS columns, stored in
// the spill_accumulator layout at parts + s * seg_stride (s = 0 .. nseg-1),
// in the order s = 0, 1, ... (so the result does not depend on which piece
// arrived last), and stores the sum into C like drain_accumulator.  Each
// chunk is summed in two passes of 16 columns; all segments' loads of a pass
// are issued before any is used (two L2 round trips per chunk, 64 registers
// of loads in flight).  nseg <= MAXSEG.
template <int OUT, bool TMA_STORE, int NCOLS, int MAXSEG, bool EPI = false>
__device__ __forceinline__ void drain_partials(const float *parts, int64_t seg_stride, int nseg,
                                               uint32_t stg, int &sbuf, int row0,
                                               int col0, int b, const EpiArgs &e) {
    const int lane = threadIdx.x & 31;
#pragma unroll 1
    for (int c = 0; c < NCOLS / 32; ++c) {
        uint32_t v[32];
#pragma unroll
        for (int h = 0; h < 2; ++h) {
            float4 t[MAXSEG][4];
#pragma unroll
            for (int s = 0; s < MAXSEG; ++s) {
                if (s < nseg) {
                    const float4 *src =
                        reinterpret_cast<const float4 *>(parts + s * seg_stride + c * 1024) + lane;
#pragma unroll
                    for (int j = 0; j < 4; ++j) t[s][j] = __ldcg(src + (4 * h + j) * 32);
                }
            }
#pragma unroll
            for (int j = 0; j < 4; ++j) {
                float4 a = t[0][j];
#pragma unroll
                for (int s = 1; s < MAXSEG; ++s) {
                    if (s < nseg) {
                        a.x += t[s][j].x;
                        a.y += t[s][j].y;
                        a.z += t[s][j].z;
                        a.w += t[s][j].w;
                    }
                }
                const int q = 4 * (4 * h + j);
                v[q] = __float_as_uint(a.x);
                v[q + 1] = __float_as_uint(a.y);
                v[q + 2] = __float_as_uint(a.z);
                v[q + 3] = __float_as_uint(a.w);
            }
        }
        store_chunk<OUT, TMA_STORE, EPI>(v, c, stg, sbuf, row0, col0, b, e);
    }
}

// Writes one warp's 32 TMEM lanes x NCOLS fp32 columns to global memory,
// bypassing L1, as float4s indexed [chunk][j][lane] (chunk = 32 columns,
// j = which 4 of them, lane = row): every warp-wide store covers 512
// contiguous bytes.  (A row-per-lane layout made each store touch 32 cache
// lines and took twice as long as the whole epilogue.)  Only chunks
// [c_lo, c_hi) are written, chunk c_lo first; TMEM is not released (the
// caller still reads its other chunks).
__device__ __forceinline__ void spill_accumulator(uint32_t tbase, float *dst, int c_lo, int c_hi) {
    const int lane = threadIdx.x & 31;
#pragma unroll 1
    for (int c = c_lo; c < c_hi; ++c) {
        uint32_t v[32];
        tmem_ld32(tbase + c * 32, v);
        float4 *out = reinterpret_cast<float4 *>(dst + (c - c_lo) * 1024) + lane;
#pragma unroll
        for (int j = 0; j < 8; ++j)
            __stcg(out + j * 32, make_float4(__uint_as_float(v[4 * j]), __uint_as_float(v[4 * j + 1]),
                                        __uint_as_float(v[4 * j + 2]), __uint_as_float(v[4 * j + 3])));
    }
}

}  // namespace hg
