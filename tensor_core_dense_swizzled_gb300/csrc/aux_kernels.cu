// aux_kernels.cu -- small HBM-bound helpers around the GEMM kernels.
//
//   repack16   copies a 16-bit operand whose base, leading dimension or batch
//              stride is not 16-byte aligned into an aligned workspace copy
//              (leading dimension rounded up to whole 128-byte blocks for the
//              tiled kernels, to 8 elements for the skinny kernels; padding
//              written as zeros), so that TMA can read it.  TMA needs 16-byte-aligned global addresses and
//              strides; the pages state the same 16-byte requirement for
//              cp.async / ldmatrix rows ("tensor-cores-cutlass-and-cute",
//              section 四.3 notes, and the 16-byte stride checks quoted from
//              vLLM in section 六.6).
//   zero_fill  writes the empty sum (K == 0) into C.
//   watchdog   a one-warp kernel whose only wait can never complete: the
//              bounded wait must give up and report.
// All loops are grid-stride loops over a grid sized to the SM count.
#include <stdint.h>

#include "kernels.h"
#include "ptx.cuh"
#include "tile_common.cuh"
#include "watchdog.cuh"

namespace hg {
namespace {

// Copies rows of up to two 16-bit operands (one launch for A and B) into
// 16-byte aligned rows.  The work is split into tasks of one row and a
// segment of 32 * SEG_U destination chunks of 8 elements (16 bytes); one
// warp per task, grid-stride, so that a long row keeps several warps busy.
// Counting aligned 16-byte granules from the one holding the row's first
// element, destination chunk c is source granules c and c+1 shifted right
// by the row's misalignment mis (0..7 elements).  Lane l loads granules
// c0 + l + 32u (u < SEG_U) of its segment -- all loads of the task are in
// flight together -- and takes granule c+1 from lane l+1's register of the
// same u, or, for lane 31, from lane 0's register of u+1 (the granule after
// the segment is loaded by lane 31 alone), so every granule is read once
// and every load and store is a full 16 bytes.  mis is the same for every
// lane of a task: it selects a body specialised for it, in which each output
// word is one funnel shift (or a plain move when mis is even; mis == 0 needs
// no second granule).  A granule is read only if it holds at least one
// element of the row, so nothing outside the row's own granules is touched.
// Elements past `cols` in the last chunk are written as zero (row padding
// that TMA never reads).
constexpr int SEG_U = 4;

template <int MIS>
__device__ __forceinline__ void repack_segment(const uint4 *g, uint16_t *d, int64_t c0, int64_t last,
                                               int64_t nch, int64_t cols, int lane) {
    constexpr int WS = MIS >> 1, ODD = MIS & 1;
    uint4 x[SEG_U];
#pragma unroll
    for (int u = 0; u < SEG_U; ++u) {
        const int64_t c = c0 + lane + 32 * u;
        x[u] = c <= last ? __ldg(g + c) : make_uint4(0, 0, 0, 0);
    }
    uint4 after = make_uint4(0, 0, 0, 0);  // the granule after the segment (lane 31)
    if (MIS != 0 && lane == 31 && c0 + 32 * SEG_U <= last) after = __ldg(g + c0 + 32 * SEG_U);
#pragma unroll
    for (int u = 0; u < SEG_U; ++u) {
        const int64_t c = c0 + lane + 32 * u;
        uint32_t w[8] = {x[u].x, x[u].y, x[u].z, x[u].w, 0, 0, 0, 0};
        if constexpr (MIS != 0) {
            const uint4 nb = u + 1 < SEG_U ? x[u + 1] : x[u];
            w[4] = __shfl_down_sync(0xFFFFFFFFu, x[u].x, 1);
            w[5] = __shfl_down_sync(0xFFFFFFFFu, x[u].y, 1);
            w[6] = __shfl_down_sync(0xFFFFFFFFu, x[u].z, 1);
            w[7] = __shfl_down_sync(0xFFFFFFFFu, x[u].w, 1);
            const uint32_t b0 = __shfl_sync(0xFFFFFFFFu, nb.x, 0);
            const uint32_t b1 = __shfl_sync(0xFFFFFFFFu, nb.y, 0);
            const uint32_t b2 = __shfl_sync(0xFFFFFFFFu, nb.z, 0);
            const uint32_t b3 = __shfl_sync(0xFFFFFFFFu, nb.w, 0);
            if (lane == 31) {
                if (u + 1 < SEG_U) {
                    w[4] = b0; w[5] = b1; w[6] = b2; w[7] = b3;
                } else {
                    w[4] = after.x; w[5] = after.y; w[6] = after.z; w[7] = after.w;
                }
            }
        }
        if (c >= nch) continue;  // after the shuffles: every lane takes part in them
        uint32_t o[4];
#pragma unroll
        for (int i = 0; i < 4; ++i)
            o[i] = ODD ? __funnelshift_r(w[i + WS], w[i + WS + 1], 16) : w[i + WS];
        if (c * 8 + 8 > cols) {  // the row's last chunk: zero the padding
#pragma unroll
            for (int i = 0; i < 4; ++i) {
                const int64_t e = c * 8 + 2 * i;  // column of o[i]'s low half
                if (e >= cols) o[i] = 0;
                else if (e + 1 >= cols) o[i] &= 0xFFFFu;
            }
        }
        *reinterpret_cast<uint4 *>(d + c * 8) = make_uint4(o[0], o[1], o[2], o[3]);
    }
}

__global__ void repack16_kernel(const Repack16Job j0, const Repack16Job j1, int njobs) {
    griddep_wait();  // the source may be the previous kernel's output
    if (threadIdx.x == 0) griddep_launch_dependents();
    constexpr int SEG = 32 * SEG_U;
    const int64_t segs0 = ((j0.ld_dst >> 3) + SEG - 1) / SEG;
    const int64_t segs1 = ((j1.ld_dst >> 3) + SEG - 1) / SEG;
    const int64_t tasks0 = j0.batch * j0.rows * segs0;
    const int64_t total = tasks0 + (njobs > 1 ? j1.batch * j1.rows * segs1 : 0);
    const int wpb = blockDim.x >> 5;
    const int lane = threadIdx.x & 31;
    for (int64_t t = static_cast<int64_t>(blockIdx.x) * wpb + (threadIdx.x >> 5); t < total;
         t += static_cast<int64_t>(gridDim.x) * wpb) {
        const bool second = t >= tasks0;
        const Repack16Job &j = second ? j1 : j0;
        const int64_t segs = second ? segs1 : segs0;
        const int64_t tt = second ? t - tasks0 : t;
        const int64_t rr = tt / segs, seg = tt - rr * segs;
        const int64_t b = rr / j.rows, r = rr - b * j.rows;
        const uint16_t *s = static_cast<const uint16_t *>(j.src) + b * j.stride_src + r * j.ld_src;
        uint16_t *d = static_cast<uint16_t *>(j.dst) + b * j.stride_dst + r * j.ld_dst;
        const uintptr_t sa = reinterpret_cast<uintptr_t>(s);
        const int mis = static_cast<int>((sa & 15u) >> 1);
        const uint4 *g = reinterpret_cast<const uint4 *>(sa - (sa & 15u));
        const int64_t last = (mis + j.cols - 1) >> 3;  // granule of the row's last element
        const int64_t nch = j.ld_dst >> 3, c0 = seg * SEG;
        switch (mis) {
            case 0: repack_segment<0>(g, d, c0, last, nch, j.cols, lane); break;
            case 1: repack_segment<1>(g, d, c0, last, nch, j.cols, lane); break;
            case 2: repack_segment<2>(g, d, c0, last, nch, j.cols, lane); break;
            case 3: repack_segment<3>(g, d, c0, last, nch, j.cols, lane); break;
            case 4: repack_segment<4>(g, d, c0, last, nch, j.cols, lane); break;
            case 5: repack_segment<5>(g, d, c0, last, nch, j.cols, lane); break;
            case 6: repack_segment<6>(g, d, c0, last, nch, j.cols, lane); break;
            default: repack_segment<7>(g, d, c0, last, nch, j.cols, lane); break;
        }
    }
}

__global__ void zero_fill_kernel(char *C, int64_t ldc, int64_t strideC, int64_t rows, int64_t cols,
                                 int64_t batch, int elem_bytes) {
    const int64_t total = batch * rows * cols;
    for (int64_t idx = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x; idx < total;
         idx += static_cast<int64_t>(gridDim.x) * blockDim.x) {
        const int64_t j = idx % cols;
        const int64_t rb = idx / cols;
        const int64_t i = rb % rows;
        const int64_t b = rb / rows;
        char *e = C + (b * strideC + i * ldc + j) * elem_bytes;
        if (elem_bytes == 4)
            *reinterpret_cast<uint32_t *>(e) = 0u;
        else
            *reinterpret_cast<uint16_t *>(e) = 0u;
    }
}

// K = 0 with a fused epilogue: the product is an empty sum, so
// D = act(beta * C_prev + bias) (scales multiply zero).
template <int OUT>
__global__ void epilogue_fill_kernel(void *C, int64_t ldc, int64_t strideC, int64_t rows,
                                     int64_t cols, int64_t batch, EpiParams ep) {
    const int64_t total = batch * rows * cols;
    for (int64_t idx = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x; idx < total;
         idx += static_cast<int64_t>(gridDim.x) * blockDim.x) {
        const int64_t j = idx % cols;
        const int64_t rb = idx / cols;
        const int64_t i = rb % rows;
        const int64_t b = rb / rows;
        const int64_t e = b * strideC + i * ldc + j;
        const float bias = ep.bias ? __ldg(ep.bias + j) : 0.f;
        const float prev = ep.beta != 0.f ? load_one<OUT>(C, e) : 0.f;
        store_one<OUT>(C, e, epi_value(ep, 0.f, 1.f, 1.f, bias, prev));
    }
}

__global__ void watchdog_selftest_kernel(int32_t *err, uint64_t timeout_ns) {
    __shared__ __align__(8) uint64_t bar;
    __shared__ int32_t abort_flag;
    if (threadIdx.x == 0) {
        mbar_init(smem_u32(&bar), 1);
        abort_flag = 0;
        fence_mbar_init();
    }
    __syncthreads();
    const WaitCtl wc{&abort_flag, err, timeout_ns};
    if (threadIdx.x == 0) {
        // phase 0 never completes: nothing arrives on `bar`
        (void)wait_bounded(smem_u32(&bar), 0, wc, timeout_code(ROLE_SELFTEST, 0));
    }
    __syncthreads();
}

int grid_for(int64_t total, int threads, int num_sms) {
    const int64_t blocks = (total + threads - 1) / threads;
    const int64_t cap = static_cast<int64_t>(num_sms) * 8;
    return static_cast<int>(blocks < 1 ? 1 : (blocks < cap ? blocks : cap));
}

}  // namespace

cudaError_t launch_repack16(const Repack16Job *jobs, int njobs, int num_sms, cudaStream_t stream) {
    if (njobs < 1 || njobs > 2) return cudaErrorInvalidValue;
    int64_t tasks = 0;  // (row, segment) tasks, as repack16_kernel counts them
    for (int i = 0; i < njobs; ++i) {
        const Repack16Job &j = jobs[i];
        if (j.ld_dst % 8 != 0 || (reinterpret_cast<uintptr_t>(j.dst) & 15) != 0 ||
            j.stride_dst % 8 != 0 || (reinterpret_cast<uintptr_t>(j.src) & 1) != 0 || j.rows < 1 ||
            j.cols < 1 || j.ld_dst < j.cols)
            return cudaErrorInvalidValue;
        tasks += j.batch * j.rows * (((j.ld_dst >> 3) + 32 * SEG_U - 1) / (32 * SEG_U));
    }
    // 8 warps per block, 4 blocks per SM: on GB300 the copy of two
    // 4095 x 4095 operands ran 24.9 us this way, 27.1 us with 8 blocks per SM
    // and 36.8 us with one warp per whole row
    const int threads = 256;
    const int64_t blocks = (tasks + 7) / 8;  // one warp per task
    const int64_t cap = static_cast<int64_t>(num_sms) * 4;
    const int grid = static_cast<int>(blocks < cap ? blocks : cap);
    return launch_dependent(repack16_kernel, grid, threads, 0, stream, jobs[0],
                            njobs > 1 ? jobs[1] : jobs[0], njobs);
}

cudaError_t launch_zero_fill(void *C, int64_t ldc, int64_t strideC, int64_t rows, int64_t cols,
                             int64_t batch, int elem_bytes, int num_sms, cudaStream_t stream) {
    const int64_t total = batch * rows * cols;
    if (total == 0) return cudaSuccess;
    zero_fill_kernel<<<grid_for(total, 256, num_sms), 256, 0, stream>>>(
        static_cast<char *>(C), ldc, strideC, rows, cols, batch, elem_bytes);
    return cudaGetLastError();
}

cudaError_t launch_epilogue_fill(void *C, int64_t ldc, int64_t strideC, int64_t rows,
                                 int64_t cols, int64_t batch, int out, const EpiParams &ep,
                                 int num_sms, cudaStream_t stream) {
    const int64_t total = batch * rows * cols;
    if (total == 0) return cudaSuccess;
    const int grid = grid_for(total, 256, num_sms);
    switch (out) {
        case OUT_F16: epilogue_fill_kernel<OUT_F16><<<grid, 256, 0, stream>>>(C, ldc, strideC, rows, cols, batch, ep); break;
        case OUT_BF16: epilogue_fill_kernel<OUT_BF16><<<grid, 256, 0, stream>>>(C, ldc, strideC, rows, cols, batch, ep); break;
        case OUT_F32: epilogue_fill_kernel<OUT_F32><<<grid, 256, 0, stream>>>(C, ldc, strideC, rows, cols, batch, ep); break;
        default: return cudaErrorInvalidValue;
    }
    return cudaGetLastError();
}

cudaError_t launch_watchdog_selftest(int32_t *err, uint64_t timeout_ns, cudaStream_t stream) {
    watchdog_selftest_kernel<<<1, 32, 0, stream>>>(err, timeout_ns);
    return cudaGetLastError();
}

}  // namespace hg
