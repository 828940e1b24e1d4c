// attention.cu -- fused attention forward on tcgen05 for sm_103a.
//
// O = softmax(scale * Q K^T [causal]) V per (batch x head, query row), the
// block "post_1787550000" builds its tensor-core work toward (sections 1-2:
// S = Q K^T and O = P V moved onto the tensor cores with the softmax between
// them, P = softmax(S) fed to the second product without leaving the chip;
// "hgemm_mma_m16n8k16_mma2x4_warp4x4_kernel" section 2 on the row-wise max
// and sum of S and the accumulator of one product becoming the operand of
// the next).  Head dimension 128, fp16 or bf16 in and out, fp32 scores,
// probabilities rounded to the input type for the second product (as the
// register hand-over of the pages does), fp32 accumulation.
//
// One CTA computes a 128-row query tile of one head, streaming keys and
// values in blocks of 64 rows; two CTAs share an SM (96 KB of shared memory
// and 256 TMEM columns each), so that one CTA's softmax runs while the
// other's products occupy the tensor core, and one CTA's start-up and
// epilogue hide behind the other's main loop.
//   warp 0, one thread   TMA: the Q tile once, then K_j and V_j into a ring
//                        of two stages (separate full / empty barriers for K
//                        and V, so S_j can start before V_j lands).
//   warp 1, one thread   MMA for the scores: S_j = Q K_j^T into TMEM buffer
//                        j % 2 (8 MMAs of K = 16 over the head dimension,
//                        N = 64 keys).
//   warp 2, one thread   MMA for the output: once the softmax warps have
//                        written P_j, O += P_j V_j (4 MMAs of 16 keys,
//                        N = 128) with P read straight from TMEM -- the
//                        Blackwell form of the pages' register hand-over: P
//                        never touches shared memory.  Issuing a tcgen05.mma
//                        costs its thread about as long as a 64-key MMA
//                        runs, so the two products get a thread each.
//   warps 3-6            online softmax, one query row per thread (the TMEM
//                        lane of its row): tcgen05.ld the 64 scores of S_j,
//                        mask, take the row max, form p = 2^(s * scale *
//                        log2 e - m) with the SFU's ex2, sum the row, rescale
//                        O in TMEM when the reference max moved, and
//                        tcgen05.st P (16-bit pairs) over the first 32
//                        columns of S_j's buffer.  After the last block:
//                        O / l, rounded to the output type, stored to global
//                        memory.
// A buffer's next S (block j + 2) is issued only once P_j V_j has completed,
// since P_j lives in it; a K or V stage is reloaded once the S, or the P V,
// that read it has completed (their own barriers say so).
//
// The reference max m is raised only when a block's max exceeds it by more
// than 8 (in log2 units): p then stays <= 2^8, and O and l, always scaled by
// the same 2^-m, give the same quotient O / l as with the running max, while
// the O rescale (a TMEM load / multiply / store of the warp's 32 rows, after
// waiting for the previous P V) happens only when some row of the warp
// raised its reference.
//
// Every wait is bounded (watchdog.cuh); a timeout records its code in the
// error word, the CTA's roles leave their loops, the MMA thread waits for
// its MMAs and the producer for its copies, and TMEM is freed.
#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "kernels.h"
#include "ptx.cuh"
#include "tile_common.cuh"
#include "watchdog.cuh"

namespace hg {
namespace {

constexpr int ATT_THREADS = 224;               // warp 0 TMA, warps 1-2 MMA, warps 3-6 softmax
constexpr int ATT_BN = 64;                     // keys per block
constexpr uint32_t ATT_QTILE = 128 * 128 * 2;  // Q: 128 rows x 128 16-bit elements
constexpr uint32_t ATT_QHALF = ATT_QTILE / 2;  // one 64-element column block of Q
constexpr uint32_t ATT_KTILE = ATT_BN * 128 * 2;   // K or V block: 64 rows x 128 elements
constexpr uint32_t ATT_KHALF = ATT_KTILE / 2;      // one 64-element column block
constexpr int ATT_STAGES = 2;                  // K / V ring depth

// shared memory, from a 1024-byte-aligned base
constexpr uint32_t SM_Q = 0;
constexpr uint32_t SM_K = SM_Q + ATT_QTILE;
constexpr uint32_t SM_V = SM_K + ATT_STAGES * ATT_KTILE;
constexpr uint32_t SM_BAR = SM_V + ATT_STAGES * ATT_KTILE;
// barriers: q_full, k_full[2], v_full[2], s_full[2], pv_done[2], p_full[2],
// o_final, drain[2]
constexpr int ATT_NBAR = 1 + 2 * ATT_STAGES + 2 + 2 + 2 + 1 + 2;
constexpr uint32_t SM_MISC = SM_BAR + 8 * ATT_NBAR;
constexpr uint32_t ATT_SMEM = SM_MISC + 16 + 1024;  // + alignment slack

// TMEM columns: S / P buffers at 0 and 64, O at 128 (256 allocated)
constexpr uint32_t TM_S = 0;
constexpr uint32_t TM_O = 128;
constexpr uint32_t TM_COLS = 256;

// (d0, d1) = (a0 * b0 + c0, a1 * b1 + c1): one fma.rn.f32x2, each lane
// rounded as fmaf rounds it.
__device__ __forceinline__ void ffma2(float &d0, float &d1, float a0, float a1, float b0, float b1,
                                      float c0, float c1) {
    asm("{\n\t.reg .b64 pa, pb, pc, pd;\n\t"
        "mov.b64 pa, {%2, %3};\n\tmov.b64 pb, {%4, %5};\n\tmov.b64 pc, {%6, %7};\n\t"
        "fma.rn.f32x2 pd, pa, pb, pc;\n\tmov.b64 {%0, %1}, pd;\n\t}"
        : "=f"(d0), "=f"(d1)
        : "f"(a0), "f"(a1), "f"(b0), "f"(b1), "f"(c0), "f"(c1));
}

// (d0, d1) = (a0 + b0, a1 + b1): one add.rn.f32x2.
__device__ __forceinline__ void fadd2(float &d0, float &d1, float a0, float a1, float b0, float b1) {
    asm("{\n\t.reg .b64 pa, pb, pd;\n\t"
        "mov.b64 pa, {%2, %3};\n\tmov.b64 pb, {%4, %5};\n\t"
        "add.rn.f32x2 pd, pa, pb;\n\tmov.b64 {%0, %1}, pd;\n\t}"
        : "=f"(d0), "=f"(d1)
        : "f"(a0), "f"(a1), "f"(b0), "f"(b1));
}

// max(a, b, c) in one instruction.
__device__ __forceinline__ float fmax3(float a, float b, float c) {
    float d;
    asm("max.f32 %0, %1, %2, %3;" : "=f"(d) : "f"(a), "f"(b), "f"(c));
    return d;
}

__device__ __forceinline__ float u2f(uint32_t x) { return __uint_as_float(x); }
__device__ __forceinline__ uint32_t f2u(float x) { return __float_as_uint(x); }

template <bool BF16>
__global__ void __launch_bounds__(ATT_THREADS, 2)
    attention_fwd_kernel(const __grid_constant__ CUtensorMap tmQ, const __grid_constant__ CUtensorMap tmK,
                         const __grid_constant__ CUtensorMap tmV, const AttnParams p) {
    constexpr int OUT = BF16 ? OUT_BF16 : OUT_F16;
    extern __shared__ uint8_t smem_raw[];
    const uint32_t raw = smem_u32(smem_raw);
    uint8_t *smem = smem_raw + ((1024u - (raw & 1023u)) & 1023u);
    const uint32_t sbase = smem_u32(smem);
    const uint32_t sQ = sbase + SM_Q, sK = sbase + SM_K, sV = sbase + SM_V;
    const uint32_t bar0 = sbase + SM_BAR;
    const uint32_t q_full = bar0;
    // Every [2] barrier entry below completes once per use of its stage or
    // buffer, in order, and no waiter can fall two phases behind an entry
    // (each wait names the event the entry's next phase needs).
    auto k_full = [&](int s) { return bar0 + 8u * (1 + s); };
    auto v_full = [&](int s) { return bar0 + 8u * (3 + s); };
    auto s_full = [&](int b) { return bar0 + 8u * (5 + b); };   // S_j done (also: K_j read)
    auto pv_done = [&](int b) { return bar0 + 8u * (7 + b); };  // P_j V_j done (also: V_j read)
    auto p_full = [&](int b) { return bar0 + 8u * (9 + b); };
    const uint32_t o_final = bar0 + 8u * 11;
    auto drain = [&](int r) { return bar0 + 8u * (12 + r); };
    volatile uint32_t *tmem_slot = reinterpret_cast<volatile uint32_t *>(smem + SM_MISC);
    volatile int32_t *abort_flag = reinterpret_cast<volatile int32_t *>(smem + SM_MISC + 4);

    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    // query tiles in descending order: under the causal mask the longest
    // tiles start first
    const int qt = p.nqt - 1 - static_cast<int>(blockIdx.x) / p.bh;
    const int bh = static_cast<int>(blockIdx.x) % p.bh;
    const int q0 = qt * 128;
    // key blocks this tile reads: the last row q0 + 127 sees keys up to
    // q0 + 127 + skv - sq under the causal mask
    int kv_end = p.skv;
    if (p.causal) kv_end = min(p.skv, q0 + 128 + (p.skv - p.sq));
    const int nkv = (kv_end + ATT_BN - 1) / ATT_BN;

    if (threadIdx.x == 0) {
        mbar_init(q_full, 1);
        for (int b = 0; b < 2; ++b) {
            mbar_init(k_full(b), 1);
            mbar_init(v_full(b), 1);
            mbar_init(s_full(b), 1);
            mbar_init(pv_done(b), 1);
            mbar_init(p_full(b), 4);
            mbar_init(drain(b), 1);
        }
        mbar_init(o_final, 1);
        *abort_flag = 0;
        fence_mbar_init();
        prefetch_tmap(&tmQ);
        prefetch_tmap(&tmK);
        prefetch_tmap(&tmV);
    }
    if (warp == 1) {
        tmem_alloc(smem_u32(const_cast<uint32_t *>(tmem_slot)), TM_COLS);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem_base = *tmem_slot;
    const WaitCtl wc{abort_flag, p.err, p.timeout_ns};

    if (warp == 0) {
        // ------------------------------------------------------------ TMA producer
        if (lane == 0) {
            mbar_arrive_expect_tx(q_full, ATT_QTILE);
            tma_load_3d(sQ, &tmQ, q_full, 0, q0, bh);
            tma_load_3d(sQ + ATT_QHALF, &tmQ, q_full, 64, q0, bh);
            int issued_k = 0, issued_v = 0;
            for (int j = 0; j < nkv; ++j) {
                const int s = j & 1;
                const uint32_t ph = static_cast<uint32_t>(j >> 1) & 1u;
                if (j >= 2 && !wait_bounded(s_full(s), ph ^ 1u, wc, timeout_code(ROLE_PRODUCER, s))) break;
                mbar_arrive_expect_tx(k_full(s), ATT_KTILE);
                tma_load_3d(sK + s * ATT_KTILE, &tmK, k_full(s), 0, j * ATT_BN, bh);
                tma_load_3d(sK + s * ATT_KTILE + ATT_KHALF, &tmK, k_full(s), 64, j * ATT_BN, bh);
                ++issued_k;
                if (j >= 2 && !wait_bounded(pv_done(s), ph ^ 1u, wc, timeout_code(ROLE_PRODUCER, 2 + s))) break;
                mbar_arrive_expect_tx(v_full(s), ATT_KTILE);
                tma_load_3d(sV + s * ATT_KTILE, &tmV, v_full(s), 0, j * ATT_BN, bh);
                tma_load_3d(sV + s * ATT_KTILE + ATT_KHALF, &tmV, v_full(s), 64, j * ATT_BN, bh);
                ++issued_v;
            }
            // copies still in flight land before the CTA leaves (immediate on
            // the normal path: the MMAs consumed them)
            wait_bounded(q_full, 0, wc, 0, /*honor_abort=*/false);
            for (int j = max(0, issued_k - ATT_STAGES); j < issued_k; ++j)
                wait_bounded(k_full(j & 1), static_cast<uint32_t>(j >> 1) & 1u, wc, 0, false);
            for (int j = max(0, issued_v - ATT_STAGES); j < issued_v; ++j)
                wait_bounded(v_full(j & 1), static_cast<uint32_t>(j >> 1) & 1u, wc, 0, false);
        }
    } else if (warp == 1) {
        // ------------------------------------------------------------ MMA: scores
        if (lane == 0) {
            bool ok = wait_bounded(q_full, 0, wc, timeout_code(ROLE_MMA, 0x200));
            const uint64_t qdesc = sdesc_sw128(sQ, 16, 1024);
            for (int j = 0; ok && j < nkv; ++j) {
                const int s = j & 1;
                if (!wait_bounded(k_full(s), static_cast<uint32_t>(j >> 1) & 1u, wc,
                                  timeout_code(ROLE_MMA, s)))
                    break;
                // buffer s holds P_{j-2} until P_{j-2} V_{j-2} has completed
                if (j >= 2 && !wait_bounded(pv_done(s), static_cast<uint32_t>((j - 2) >> 1) & 1u, wc,
                                            timeout_code(ROLE_MMA, 0x100 + s)))
                    break;
                tc_fence_after();
                const uint64_t kdesc = sdesc_sw128(sK + s * ATT_KTILE, 16, 1024);
                const uint32_t tS = tmem_base + TM_S + 64u * s;
#pragma unroll
                for (int kk = 0; kk < 8; ++kk) {
                    const uint32_t qoff = (kk >> 2) * ATT_QHALF + (kk & 3) * 32;
                    const uint32_t koff = (kk >> 2) * ATT_KHALF + (kk & 3) * 32;
                    umma_f16(tS, qdesc + (qoff >> 4), kdesc + (koff >> 4), p.idesc_s, kk > 0 ? 1u : 0u);
                }
                umma_commit(s_full(s));
            }
            umma_commit(drain(0));
            wait_bounded(drain(0), 0, wc, 0, /*honor_abort=*/false);
        }
    } else if (warp == 2) {
        // ------------------------------------------------------------ MMA: output
        if (lane == 0) {
            const uint32_t tO = tmem_base + TM_O;
            bool ok = true;
            // O += P_t V_t: P from TMEM (8 columns per 16 keys); V MN-major
            // (two 64-column blocks 8 KB apart, 2 KB per 16 keys)
            for (int t = 0; t < nkv; ++t) {
                const int ts = t & 1;
                const uint32_t ph = static_cast<uint32_t>(t >> 1) & 1u;
                if (!wait_bounded(p_full(ts), ph, wc, timeout_code(ROLE_MMA, 0x300 + ts)) ||
                    !wait_bounded(v_full(ts), ph, wc, timeout_code(ROLE_MMA, 0x302 + ts))) {
                    ok = false;
                    break;
                }
                tc_fence_after();
                const uint64_t vdesc = sdesc_sw128(sV + ts * ATT_KTILE, ATT_KHALF, 1024);
                const uint32_t tP = tmem_base + TM_S + 64u * ts;
#pragma unroll
                for (int kk = 0; kk < ATT_BN / 16; ++kk)
                    umma_f16_tmem_a(tO, tP + 8u * kk, vdesc + ((kk * 2048u) >> 4), p.idesc_o,
                                    (t > 0 || kk > 0) ? 1u : 0u);
                umma_commit(pv_done(ts));
            }
            if (ok) umma_commit(o_final);
            umma_commit(drain(1));
            wait_bounded(drain(1), 0, wc, 0, /*honor_abort=*/false);
        }
    } else {
        // ------------------------------------------------------------ softmax warps
        const uint32_t quarter = static_cast<uint32_t>(warp & 3);
        const int row = static_cast<int>(quarter) * 32 + lane;
        const uint32_t lane_addr = (quarter * 32u) << 16;
        const int qi = q0 + row;
        int lim = p.skv;  // keys < lim are allowed for this row
        if (p.causal) lim = min(lim, qi + 1 + (p.skv - p.sq));
        const float c = p.scale_log2;
        float m_ref = -INFINITY, l = 0.f;
        bool ok = true;
        uint32_t sv[64];
        for (int j = 0; j < nkv; ++j) {
            const int b = j & 1;
            const uint32_t tS = tmem_base + lane_addr + TM_S + 64u * b;
            if (!wait_bounded_warp(s_full(b), static_cast<uint32_t>(j >> 1) & 1u, wc,
                                   timeout_code(ROLE_EPILOGUE, b))) {
                ok = false;
                break;
            }
            tc_fence_after();
            tmem_ld64(tS, sv);
            const int kbase = j * ATT_BN;
            if (kbase + ATT_BN > lim) {
#pragma unroll
                for (int i = 0; i < 64; ++i)
                    if (kbase + i >= lim) sv[i] = f2u(-INFINITY);
            }
            // row max and sum in 8 independent partials (short dependency
            // chains: few warps share an SM sub-partition), with three-input
            // max and packed fp32 pairs to halve the instruction count
            float pm[8];
#pragma unroll
            for (int t = 0; t < 8; ++t) pm[t] = fmaxf(u2f(sv[t]), u2f(sv[t + 8]));
#pragma unroll
            for (int i = 16; i < 64; i += 16)
#pragma unroll
                for (int t = 0; t < 8; ++t) pm[t] = fmax3(pm[t], u2f(sv[i + t]), u2f(sv[i + 8 + t]));
            float mx = fmax3(fmax3(pm[0], pm[1], pm[2]), fmax3(pm[3], pm[4], pm[5]), fmaxf(pm[6], pm[7]));
            mx *= c;
            float alpha = 1.f;
            const bool raise = mx > m_ref + 8.f;
            if (raise) {
                alpha = ex2_approx(m_ref - mx);
                m_ref = mx;
            }
            float ps[8];
#pragma unroll
            for (int t = 0; t < 8; ++t) ps[t] = 0.f;
            uint32_t pk[32];  // P as 16-bit pairs, key 2i in the low half of pk[i]
#pragma unroll
            for (int i = 0; i < 64; i += 2) {
                float a0, a1;
                ffma2(a0, a1, u2f(sv[i]), u2f(sv[i + 1]), c, c, -m_ref, -m_ref);
                const float e0 = ex2_approx(a0);
                const float e1 = ex2_approx(a1);
                fadd2(ps[i & 7], ps[(i & 7) + 1], ps[i & 7], ps[(i & 7) + 1], e0, e1);
                pk[i / 2] = pack2<OUT>(f2u(e0), f2u(e1));
            }
            const float sum = ((ps[0] + ps[1]) + (ps[2] + ps[3])) + ((ps[4] + ps[5]) + (ps[6] + ps[7]));
            l = l * alpha + sum;
            if (j >= 1 && __any_sync(0xFFFFFFFFu, raise)) {
                // O must hold every earlier block before it is rescaled
                if (!wait_bounded_warp(pv_done((j - 1) & 1), static_cast<uint32_t>((j - 1) >> 1) & 1u, wc,
                                       timeout_code(ROLE_EPILOGUE, 0x10))) {
                    ok = false;
                    break;
                }
                tc_fence_after();
#pragma unroll 1
                for (int q = 0; q < 4; ++q) {
                    uint32_t o[32];
                    tmem_ld32(tmem_base + lane_addr + TM_O + 32u * q, o);
#pragma unroll
                    for (int i = 0; i < 32; ++i) o[i] = f2u(u2f(o[i]) * alpha);
                    tmem_st32(tmem_base + lane_addr + TM_O + 32u * q, o);
                }
            }
            // P over the first 32 columns of the buffer (its scores are in
            // registers already)
            tmem_st32(tS, pk);
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(p_full(b));
        }
        if (ok && wait_bounded_warp(o_final, 0, wc, timeout_code(ROLE_EPILOGUE, 0x11))) {
            tc_fence_after();
            const float inv = 1.f / l;
            const bool store = qi < p.sq;
            uint8_t *orow = static_cast<uint8_t *>(p.O) +
                            (static_cast<int64_t>(bh) * p.sq + (store ? qi : 0)) * 256;
#pragma unroll 1
            for (int q = 0; q < 4; ++q) {
                uint32_t o[32];
                tmem_ld32(tmem_base + lane_addr + TM_O + 32u * q, o);
                if (store) {
                    uint4 *dst = reinterpret_cast<uint4 *>(orow + q * 64);
#pragma unroll
                    for (int t = 0; t < 4; ++t) {
                        uint4 v;
                        v.x = pack2<OUT>(f2u(u2f(o[8 * t]) * inv), f2u(u2f(o[8 * t + 1]) * inv));
                        v.y = pack2<OUT>(f2u(u2f(o[8 * t + 2]) * inv), f2u(u2f(o[8 * t + 3]) * inv));
                        v.z = pack2<OUT>(f2u(u2f(o[8 * t + 4]) * inv), f2u(u2f(o[8 * t + 5]) * inv));
                        v.w = pack2<OUT>(f2u(u2f(o[8 * t + 6]) * inv), f2u(u2f(o[8 * t + 7]) * inv));
                        dst[t] = v;
                    }
                }
            }
        }
    }

    tc_fence_before();
    __syncthreads();
    if (warp == 1) {
        tc_fence_after();
        tmem_dealloc(tmem_base, TM_COLS);
    }
}

}  // namespace

cudaError_t launch_attention(bool bf16, const CUtensorMap &tmQ, const CUtensorMap &tmK,
                             const CUtensorMap &tmV, const AttnParams &p, cudaStream_t stream) {
    auto kern = bf16 ? attention_fwd_kernel<true> : attention_fwd_kernel<false>;
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         static_cast<int>(ATT_SMEM));
    if (e != cudaSuccess) return e;
    const unsigned grid = static_cast<unsigned>(p.bh) * static_cast<unsigned>(p.nqt);
    kern<<<grid, ATT_THREADS, ATT_SMEM, stream>>>(tmQ, tmK, tmV, p);
    return cudaGetLastError();
}

}  // namespace hg
