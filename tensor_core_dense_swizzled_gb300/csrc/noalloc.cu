// noalloc.cu -- hgemm_skinny_noalloc: the small-M (decode-shaped) product
// with no device memory allocation at all.
//
// Who needs it.  The planned API (hgemm_plan_create / hgemm_run) allocates
// its split-K workspace with cudaMalloc when a plan is made.  Some callers
// cannot do that: a host framework that owns every device allocation and
// hands a plugin only its input and output buffers, a server whose device
// memory is budgeted once at start-up and may not grow afterwards, or a
// latency-critical loop where cudaMalloc's implicit device synchronisation
// is not acceptable.  This entry point serves them: the caller passes A, B
// and C, and the split-K partial sums, arrival counters and error word live
// in a fixed array compiled into the library.
//
// The array.  `g_scratch` below is a file-scope __device__ array of
// kScratchBytes (8 MiB).  Every GPU that loads the library holds one copy of
// it until the process exits.  In host code the name `g_scratch` is only a
// host-side stand-in for the symbol, never a device address: the first call
// on each device looks up the real address with cudaGetSymbolAddress (with
// that device current) and caches it, keyed by the device's current CUDA
// context, so make that first call before any stream capture.  A new context
// on the device (after cudaDeviceReset, say) reloads the module and may move
// the array: the next call sees the new context's id and looks the address
// up again (when the driver cannot report a context id, every call looks it
// up, which is a cheap host call).  All calls on a device share the one
// array and it keeps the last call's contents: each call clears the error
// word and the counters (cudaMemsetAsync on the caller's stream) before its
// kernel runs, and the partial sums need no clearing because every one is
// written before it is read.  Calls that overlap on the GPU (two streams, or two host threads
// without ordering) race on the array and give wrong results: order them.
//
// Limits.  M <= 32, batch 1, and A and B must be directly readable by TMA
// (16-byte aligned base pointers, leading dimensions a multiple of 8
// elements), because this entry point cannot make aligned copies.  The split
// count is the planned path's; it is lowered when the partial sums would not
// fit in the array, and a request that does not fit even unsplit is refused
// with HGEMM_ERR_UNSUPPORTED.  A device watchdog timeout is recorded in the
// array's error word; hgemm_skinny_noalloc_check reads and clears it (the
// next product clears it too, before its kernel runs).
#include <cuda.h>
#include <cuda_runtime.h>
#include <cudaTypedefs.h>

#include <cstdio>
#include <mutex>

#include "hgemm.h"
#include "internal.h"
#include "kernels.h"

namespace {

constexpr size_t kScratchBytes = size_t(8) << 20;  // 8 MiB per device
constexpr size_t kErrBytes = 256;                  // error word + padding
constexpr int kMaxDevices = 64;
constexpr uint64_t kTimeoutNs = 2000000000ull;

static __device__ __align__(256) unsigned char g_scratch[kScratchBytes];

// The address of g_scratch found on a device, and the id of the context it
// was found in.
struct ScratchAddr {
    bool valid;
    unsigned long long ctx_id;
    void *ptr;
};
std::mutex g_mu;
ScratchAddr g_scratch_dev[kMaxDevices] = {};

// Unique id of the calling thread's current CUDA context (cuCtxGetId, reached
// through the runtime's driver entry points); false when there is no current
// context or the driver cannot say.
bool current_context_id(unsigned long long *id) {
    static PFN_cuCtxGetCurrent_v4000 get_current = nullptr;
    static PFN_cuCtxGetId_v12000 get_id = nullptr;
    static std::once_flag once;
    std::call_once(once, [] {
        void *p = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuCtxGetCurrent", &p, 4000, cudaEnableDefault, &q) ==
                cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            get_current = reinterpret_cast<PFN_cuCtxGetCurrent_v4000>(p);
        p = nullptr;
        if (cudaGetDriverEntryPointByVersion("cuCtxGetId", &p, 12000, cudaEnableDefault, &q) ==
                cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            get_id = reinterpret_cast<PFN_cuCtxGetId_v12000>(p);
    });
    if (!get_current || !get_id) return false;
    CUcontext ctx = nullptr;
    if (get_current(&ctx) != CUDA_SUCCESS || ctx == nullptr) return false;
    return get_id(ctx, id) == CUDA_SUCCESS;
}

// Device address of g_scratch on `dev` (which must be current), looked up
// once per context of that device.
hgemm_status_t scratch_address(int dev, unsigned char **out) {
    std::lock_guard<std::mutex> lock(g_mu);
    if (dev < 0 || dev >= kMaxDevices)
        return hg::set_error_detail(HGEMM_ERR_UNSUPPORTED, "device ordinal too large");
    ScratchAddr &slot = g_scratch_dev[dev];
    unsigned long long id = 0;
    if (slot.valid && current_context_id(&id) && id == slot.ctx_id) {
        *out = static_cast<unsigned char *>(slot.ptr);
        return HGEMM_OK;
    }
    void *p = nullptr;
    cudaError_t e = cudaGetSymbolAddress(&p, g_scratch);  // also makes the context current
    if (e != cudaSuccess || p == nullptr) {
        char msg[256];
        snprintf(msg, sizeof(msg), "cudaGetSymbolAddress(scratch) failed: %s", cudaGetErrorString(e));
        return hg::set_error_detail(HGEMM_ERR_CUDA, msg);
    }
    // keyed by the context it belongs to; not kept when no id is available
    slot.valid = current_context_id(&id);
    slot.ctx_id = id;
    slot.ptr = p;
    *out = static_cast<unsigned char *>(p);
    return HGEMM_OK;
}

inline int64_t ceil_div(int64_t x, int64_t m) { return (x + m - 1) / m; }
inline int64_t round256(int64_t x) { return (x + 255) / 256 * 256; }

}  // namespace

extern "C" hgemm_status_t hgemm_skinny_noalloc(const void *A, const void *B, void *C, int64_t M,
                                               int64_t N, int64_t K, int64_t lda, int64_t ldb,
                                               int64_t ldc, hgemm_dtype_t dtype_in,
                                               hgemm_dtype_t dtype_out, void *stream) {
    using hg::set_error_detail;
    if (dtype_in != HGEMM_F16 && dtype_in != HGEMM_BF16)
        return set_error_detail(HGEMM_ERR_INVALID_ARG, "dtype_in must be HGEMM_F16 or HGEMM_BF16");
    if (dtype_out != HGEMM_F16 && dtype_out != HGEMM_BF16 && dtype_out != HGEMM_F32)
        return set_error_detail(HGEMM_ERR_INVALID_ARG, "dtype_out must be HGEMM_F32, HGEMM_F16 or HGEMM_BF16");
    if (M < 0 || N < 0 || K < 0) return set_error_detail(HGEMM_ERR_INVALID_ARG, "negative size");
    if (M > 32)
        return set_error_detail(HGEMM_ERR_UNSUPPORTED, "hgemm_skinny_noalloc handles M <= 32");
    if (N > (int64_t(1) << 31) - 1 || K > (int64_t(1) << 31) - 1)
        return set_error_detail(HGEMM_ERR_UNSUPPORTED, "sizes above 2^31-1 are not supported");
    if (M == 0 || N == 0) return HGEMM_OK;
    if (ldc < N) return set_error_detail(HGEMM_ERR_INVALID_ARG, "ldc < N");
    if (K > 0 && (lda < K || ldb < N)) return set_error_detail(HGEMM_ERR_INVALID_ARG, "lda < K or ldb < N");
    if (!C) return set_error_detail(HGEMM_ERR_INVALID_ARG, "C is NULL");
    const int ob = dtype_out == HGEMM_F32 ? 4 : 2;
    if (reinterpret_cast<uintptr_t>(C) % ob != 0)
        return set_error_detail(HGEMM_ERR_INVALID_ARG, "C is not element-aligned");

    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return set_error_detail(HGEMM_ERR_NO_DEVICE, "no CUDA device");
    int major = 0, minor = 0, sms = 0;
    cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev);
    cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev);
    cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    if (major != 10 || minor != 3)
        return set_error_detail(HGEMM_ERR_NO_DEVICE, "libhgemm is built for sm_103a");
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    const int out = dtype_out == HGEMM_F32 ? hg::OUT_F32 : (dtype_out == HGEMM_BF16 ? hg::OUT_BF16 : hg::OUT_F16);

    hgemm_status_t cst = hg::check_device_pointer(C, dev, "C");
    if (cst != HGEMM_OK) return cst;
    if (K == 0) {  // the empty sum
        e = hg::launch_zero_fill(C, ldc, 0, M, N, 1, ob, sms, s);
        if (e != cudaSuccess) return set_error_detail(HGEMM_ERR_CUDA, cudaGetErrorString(e));
        return HGEMM_OK;
    }
    if (!A || !B) return set_error_detail(HGEMM_ERR_INVALID_ARG, "A or B is NULL");
    {
        hgemm_status_t pst = hg::check_device_pointer(A, dev, "A");
        if (pst == HGEMM_OK) pst = hg::check_device_pointer(B, dev, "B");
        if (pst != HGEMM_OK) return pst;
    }
    if ((reinterpret_cast<uintptr_t>(A) & 15) || (reinterpret_cast<uintptr_t>(B) & 15) ||
        (lda * 2) % 16 || (ldb * 2) % 16)
        return set_error_detail(HGEMM_ERR_UNSUPPORTED,
                                "hgemm_skinny_noalloc needs 16-byte aligned A and B with leading "
                                "dimensions a multiple of 8 elements (it cannot make aligned copies)");

    // scratch layout: [error word][counters: num_n x 4][partials: split x num_n x NU x 128 fp32]
    // (num_n = 128-column sub-tiles; a work unit of nb 64-column blocks covers
    // ceil(nb / 2) of them)
    const int nu = M <= 16 ? 16 : 32;
    const int nb = hg::pick_skinny_nb(N, 1, sms);
    const int64_t num_tiles = ceil_div(N, 64 * nb);
    const int64_t num_n = num_tiles * ((nb + 1) / 2);
    const int num_kb = static_cast<int>(ceil_div(K, 64));
    const int64_t counter_bytes = round256(num_n * 4 * static_cast<int64_t>(sizeof(int32_t)));
    int split = hg::pick_split(num_tiles, num_kb, sms);
    auto partial_bytes = [&](int sp) -> int64_t {
        return sp > 1 ? sp * num_n * nu * 128 * static_cast<int64_t>(sizeof(float)) : 0;
    };
    while (split > 1 && static_cast<int64_t>(kErrBytes) + counter_bytes + partial_bytes(split) >
                            static_cast<int64_t>(kScratchBytes))
        --split;
    if (static_cast<int64_t>(kErrBytes) + counter_bytes + partial_bytes(split) >
        static_cast<int64_t>(kScratchBytes))
        return set_error_detail(HGEMM_ERR_UNSUPPORTED,
                                "N is too large for the 8 MiB scratch array of hgemm_skinny_noalloc");
    const int kb_per = static_cast<int>(ceil_div(num_kb, split));
    split = static_cast<int>(ceil_div(num_kb, kb_per));

    unsigned char *scratch = nullptr;
    hgemm_status_t st = scratch_address(dev, &scratch);
    if (st != HGEMM_OK) return st;

    CUtensorMap tmX, tmW;
    const int bf = dtype_in == HGEMM_BF16 ? 1 : 0;
    st = hg::encode_map_3d(&tmX, A, bf, K, M, lda, 64, static_cast<uint32_t>(nu));
    if (st != HGEMM_OK) return st;
    st = hg::encode_map_3d(&tmW, B, bf, N, K, ldb, 64, 64);
    if (st != HGEMM_OK) return st;

    // the error word and the counters must start at zero
    e = cudaMemsetAsync(scratch, 0, kErrBytes + counter_bytes, s);
    if (e != cudaSuccess) return set_error_detail(HGEMM_ERR_CUDA, cudaGetErrorString(e));

    hg::SkinnyParams sp{};
    sp.M = static_cast<int32_t>(M);
    sp.N = static_cast<int32_t>(N);
    sp.K = static_cast<int32_t>(K);
    sp.batch = 1;
    sp.num_tiles = static_cast<int32_t>(num_tiles);
    sp.num_kb = num_kb;
    sp.split = split;
    sp.kb_per_split = kb_per;
    sp.units = static_cast<int32_t>(num_tiles * split);
    sp.idesc = hg::idesc_f16(static_cast<uint32_t>(bf), 1, 0, 128, static_cast<uint32_t>(nu));
    sp.C = C;
    sp.ldc = ldc;
    sp.strideC = 0;
    sp.err = reinterpret_cast<int32_t *>(scratch);
    sp.counters = reinterpret_cast<int32_t *>(scratch + kErrBytes);
    sp.partials = reinterpret_cast<float *>(scratch + kErrBytes + counter_bytes);
    sp.timeout_ns = kTimeoutNs;
    const int grid = static_cast<int>(sp.units < sms ? sp.units : sms);
    e = hg::launch_skinny(nu, nb, out, tmX, tmW, sp, grid, s);
    if (e != cudaSuccess) return set_error_detail(HGEMM_ERR_CUDA, cudaGetErrorString(e));
    return HGEMM_OK;
}

extern "C" hgemm_status_t hgemm_skinny_noalloc_check(void *stream) {
    cudaError_t e = cudaStreamSynchronize(static_cast<cudaStream_t>(stream));
    if (e != cudaSuccess) return hg::set_error_detail(HGEMM_ERR_CUDA, cudaGetErrorString(e));
    int dev = 0;
    e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return hg::set_error_detail(HGEMM_ERR_NO_DEVICE, "no CUDA device");
    unsigned char *scratch = nullptr;
    hgemm_status_t st = scratch_address(dev, &scratch);
    if (st != HGEMM_OK) return st;
    int32_t word = 0;
    e = cudaMemcpy(&word, scratch, sizeof(word), cudaMemcpyDeviceToHost);
    if (e != cudaSuccess) return hg::set_error_detail(HGEMM_ERR_CUDA, cudaGetErrorString(e));
    if (word == 0) return HGEMM_OK;
    e = cudaMemset(scratch, 0, sizeof(word));
    if (e != cudaSuccess) return hg::set_error_detail(HGEMM_ERR_CUDA, cudaGetErrorString(e));
    return hg::status_from_error_word(word);
}
