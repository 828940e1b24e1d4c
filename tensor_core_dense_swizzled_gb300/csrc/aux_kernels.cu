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
#include "watchdog.cuh"

namespace hg {
namespace {

// One thread writes one aligned 16-byte chunk (8 elements) of a destination
// row; the source reads are 2-byte loads with no alignment assumption.
__global__ void repack16_kernel(const uint16_t *__restrict__ src, int64_t ld_src, int64_t stride_src,
                                uint16_t *__restrict__ dst, int64_t ld_dst, int64_t stride_dst,
                                int64_t rows, int64_t cols, int64_t batch) {
    const int64_t chunks = ld_dst / 8;
    const int64_t total = batch * rows * chunks;
    for (int64_t idx = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x; idx < total;
         idx += static_cast<int64_t>(gridDim.x) * blockDim.x) {
        const int64_t c8 = idx % chunks;
        const int64_t rb = idx / chunks;
        const int64_t r = rb % rows;
        const int64_t b = rb / rows;
        const uint16_t *s = src + b * stride_src + r * ld_src + c8 * 8;
        uint32_t w[4];
#pragma unroll
        for (int e = 0; e < 4; ++e) {
            const int64_t col = c8 * 8 + 2 * e;
            const uint32_t lo = (col < cols) ? s[2 * e] : 0u;
            const uint32_t hi = (col + 1 < cols) ? s[2 * e + 1] : 0u;
            w[e] = lo | (hi << 16);
        }
        uint4 *d = reinterpret_cast<uint4 *>(dst + b * stride_dst + r * ld_dst + c8 * 8);
        *d = make_uint4(w[0], w[1], w[2], w[3]);
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

cudaError_t launch_repack16(const void *src, int64_t ld_src, int64_t stride_src, void *dst,
                            int64_t ld_dst, int64_t stride_dst, int64_t rows, int64_t cols,
                            int64_t batch, int num_sms, cudaStream_t stream) {
    if (ld_dst % 8 != 0 || (reinterpret_cast<uintptr_t>(dst) & 15) != 0 || stride_dst % 8 != 0)
        return cudaErrorInvalidValue;
    const int64_t total = batch * rows * (ld_dst / 8);
    if (total == 0) return cudaSuccess;
    repack16_kernel<<<grid_for(total, 256, num_sms), 256, 0, stream>>>(
        static_cast<const uint16_t *>(src), ld_src, stride_src, static_cast<uint16_t *>(dst),
        ld_dst, stride_dst, rows, cols, batch);
    return cudaGetLastError();
}

cudaError_t launch_zero_fill(void *C, int64_t ldc, int64_t strideC, int64_t rows, int64_t cols,
                             int64_t batch, int elem_bytes, int num_sms, cudaStream_t stream) {
    const int64_t total = batch * rows * cols;
    if (total == 0) return cudaSuccess;
    zero_fill_kernel<<<grid_for(total, 256, num_sms), 256, 0, stream>>>(
        static_cast<char *>(C), ldc, strideC, rows, cols, batch, elem_bytes);
    return cudaGetLastError();
}

cudaError_t launch_watchdog_selftest(int32_t *err, uint64_t timeout_ns, cudaStream_t stream) {
    watchdog_selftest_kernel<<<1, 32, 0, stream>>>(err, timeout_ns);
    return cudaGetLastError();
}

}  // namespace hg
