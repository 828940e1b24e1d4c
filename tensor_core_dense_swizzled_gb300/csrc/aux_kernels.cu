// aux_kernels.cu -- small HBM-bound helpers around the GEMM kernels.
//
//   repack16   copies a 16-bit operand whose base, leading dimension or batch
//              stride is not 16-byte aligned into an aligned workspace copy
//              (leading dimension rounded up to 8 elements), so that TMA can
//              read it.  TMA needs 16-byte-aligned global addresses and
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

__device__ __forceinline__ uint32_t select8(const uint32_t (&w)[8], int k) {
    uint32_t r = w[0];
#pragma unroll
    for (int t = 1; t < 8; ++t) r = (k == t) ? w[t] : r;
    return r;
}

// Copies rows of up to two 16-bit operands (one launch for A and B) into
// 16-byte aligned rows.  One warp per row; lane l writes destination chunks
// l, l+32, ... of 8 elements (16 bytes).  Counting aligned 16-byte granules
// from the one holding the row's first element, destination chunk c is
// source granules c and c+1 shifted right by the row's misalignment (0..7
// elements), so every load and store is a full 16 bytes.  A granule is read
// only if it holds at least one element of the row, so nothing outside the
// row's own granules is touched.  Elements past `cols` in the last chunk are
// written as zero (row padding that TMA never reads).
__global__ void repack16_kernel(const Repack16Job j0, const Repack16Job j1, int njobs) {
    griddep_wait();  // the source may be the previous kernel's output
    if (threadIdx.x == 0) griddep_launch_dependents();
    const int64_t rows0 = j0.batch * j0.rows;
    const int64_t total = rows0 + (njobs > 1 ? j1.batch * j1.rows : 0);
    const int wpb = blockDim.x >> 5;
    const int lane = threadIdx.x & 31;
    for (int64_t row = static_cast<int64_t>(blockIdx.x) * wpb + (threadIdx.x >> 5); row < total;
         row += static_cast<int64_t>(gridDim.x) * wpb) {
        const bool second = row >= rows0;
        const int64_t rr = second ? row - rows0 : row;
        const int64_t rows = second ? j1.rows : j0.rows;
        const int64_t cols = second ? j1.cols : j0.cols;
        const int64_t ld_dst = second ? j1.ld_dst : j0.ld_dst;
        const int64_t b = rr / rows, r = rr - (rr / rows) * rows;
        const uint16_t *s = static_cast<const uint16_t *>(second ? j1.src : j0.src) +
                            b * (second ? j1.stride_src : j0.stride_src) +
                            r * (second ? j1.ld_src : j0.ld_src);
        uint16_t *d = static_cast<uint16_t *>(second ? j1.dst : j0.dst) +
                      b * (second ? j1.stride_dst : j0.stride_dst) + r * ld_dst;
        const uintptr_t sa = reinterpret_cast<uintptr_t>(s);
        const int mis = static_cast<int>((sa & 15u) >> 1);
        const uint4 *g = reinterpret_cast<const uint4 *>(sa - (sa & 15u));
        const int64_t last = (mis + cols - 1) >> 3;  // granule of the row's last element
        const int ws = mis >> 1, odd = mis & 1;
        const int64_t nch = ld_dst >> 3;
        for (int64_t c = lane; c < nch; c += 32) {
            uint32_t w[8] = {0, 0, 0, 0, 0, 0, 0, 0};
            if (c <= last) {
                const uint4 x = __ldg(g + c);
                w[0] = x.x; w[1] = x.y; w[2] = x.z; w[3] = x.w;
            }
            if (c + 1 <= last) {
                const uint4 y = __ldg(g + c + 1);
                w[4] = y.x; w[5] = y.y; w[6] = y.z; w[7] = y.w;
            }
            uint32_t o[4];
#pragma unroll
            for (int i = 0; i < 4; ++i) {
                const uint32_t lo = select8(w, i + ws), hi = select8(w, i + ws + 1);
                o[i] = odd ? __funnelshift_r(lo, hi, 16) : lo;
                const int64_t e = c * 8 + 2 * i;  // column of o[i]'s low half
                if (e >= cols) o[i] = 0;
                else if (e + 1 >= cols) o[i] &= 0xFFFFu;
            }
            *reinterpret_cast<uint4 *>(d + c * 8) = make_uint4(o[0], o[1], o[2], o[3]);
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
    int64_t rows = 0;
    for (int i = 0; i < njobs; ++i) {
        const Repack16Job &j = jobs[i];
        if (j.ld_dst % 8 != 0 || (reinterpret_cast<uintptr_t>(j.dst) & 15) != 0 ||
            j.stride_dst % 8 != 0 || (reinterpret_cast<uintptr_t>(j.src) & 1) != 0 || j.rows < 1 ||
            j.cols < 1 || j.ld_dst < j.cols)
            return cudaErrorInvalidValue;
        rows += j.batch * j.rows;
    }
    const int threads = 256;  // 8 warps, one row each
    const int64_t blocks = (rows + 7) / 8;
    const int64_t cap = static_cast<int64_t>(num_sms) * 8;
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
