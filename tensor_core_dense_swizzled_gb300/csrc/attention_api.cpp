// attention_api.cpp -- the C ABI of the fused attention forward (declared in
// include/hgemm.h): argument checks, the plan's workspace, tensor maps and
// the launch of attention.cu's kernel.
#include <cuda.h>
#include <cuda_runtime.h>

#include <cmath>
#include <cstdarg>
#include <cstdint>
#include <cstdio>
#include <cstring>
#include <new>

#include "hgemm.h"
#include "internal.h"
#include "kernels.h"

namespace {

constexpr uint64_t kAttnTimeoutNs = 2000000000ull;  // 2 s per pipeline wait
constexpr int64_t kMax32 = (1ll << 31) - 1;

hgemm_status_t afail(hgemm_status_t s, const char *fmt, ...) {
    char buf[512];
    va_list ap;
    va_start(ap, fmt);
    vsnprintf(buf, sizeof(buf), fmt, ap);
    va_end(ap);
    return hg::set_error_detail(s, buf);
}

hgemm_status_t acuda(cudaError_t e, const char *what) {
    return afail(e == cudaErrorMemoryAllocation ? HGEMM_ERR_OOM : HGEMM_ERR_CUDA, "%s: %s (%s)", what,
                 cudaGetErrorName(e), cudaGetErrorString(e));
}

inline bool aligned16(const void *p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

}  // namespace

struct hgemm_attn_plan_s {
    int64_t bh, sq, skv, d;
    float scale;
    int causal;
    hgemm_dtype_t dt;
    int device, num_sms;
    int32_t *err = nullptr;  // device error word (256 B)
    // host-buffer staging
    char *dQ = nullptr, *dK = nullptr, *dV = nullptr, *dO = nullptr;
    // the last Q, K, V, O that passed check_device_pointer
    const void *okQ = nullptr, *okK = nullptr, *okV = nullptr, *okO = nullptr;
    // tensor-map cache
    const void *mQ = nullptr, *mK = nullptr, *mV = nullptr;
    bool maps_ok = false;
    CUtensorMap tmQ, tmK, tmV;
};

namespace {

int64_t q_bytes(const hgemm_attn_plan_s *p) { return p->bh * p->sq * p->d * 2; }
int64_t kv_bytes(const hgemm_attn_plan_s *p) { return p->bh * p->skv * p->d * 2; }

hgemm_status_t attn_run(hgemm_attn_plan_s *p, const void *Q, const void *K, const void *V, void *O,
                        cudaStream_t s) {
    if (p->sq == 0) return HGEMM_OK;
    if (!O || !aligned16(O)) return afail(HGEMM_ERR_INVALID_ARG, "O is NULL or not 16-byte aligned");
    int cur = -1;
    cudaGetDevice(&cur);
    if (cur != p->device)
        return afail(HGEMM_ERR_INVALID_ARG, "plan was created on device %d but device %d is current",
                     p->device, cur);
    if (O != p->okO) {  // checked once per pointer
        hgemm_status_t st = hg::check_device_pointer(O, p->device, "O");
        if (st != HGEMM_OK) return st;
        p->okO = O;
    }
    cudaError_t e;
    if (p->skv == 0) {  // the empty sum
        e = hg::launch_zero_fill(O, p->d, 0, p->bh * p->sq, p->d, 1, 2, p->num_sms, s);
        return e == cudaSuccess ? HGEMM_OK : acuda(e, "zero-fill launch");
    }
    if (!Q || !K || !V) return afail(HGEMM_ERR_INVALID_ARG, "Q, K or V is NULL");
    if (!(Q == p->okQ && K == p->okK && V == p->okV)) {  // once per pointer set
        hgemm_status_t st = hg::check_device_pointer(Q, p->device, "Q");
        if (st == HGEMM_OK) st = hg::check_device_pointer(K, p->device, "K");
        if (st == HGEMM_OK) st = hg::check_device_pointer(V, p->device, "V");
        if (st != HGEMM_OK) return st;
        p->okQ = Q; p->okK = K; p->okV = V;
    }
    if (!aligned16(Q) || !aligned16(K) || !aligned16(V))
        return afail(HGEMM_ERR_INVALID_ARG, "Q, K and V must be 16-byte aligned");
    const int bf = p->dt == HGEMM_BF16 ? 1 : 0;
    if (!(p->maps_ok && Q == p->mQ && K == p->mK && V == p->mV)) {
        hgemm_status_t st;
        st = hg::encode_map_batched(&p->tmQ, Q, bf, p->d, p->sq, p->bh, p->d, p->sq * p->d, 64, 128);
        if (st != HGEMM_OK) return st;
        // K and V stream in blocks of 64 rows
        st = hg::encode_map_batched(&p->tmK, K, bf, p->d, p->skv, p->bh, p->d, p->skv * p->d, 64, 64);
        if (st != HGEMM_OK) return st;
        st = hg::encode_map_batched(&p->tmV, V, bf, p->d, p->skv, p->bh, p->d, p->skv * p->d, 64, 64);
        if (st != HGEMM_OK) return st;
        p->mQ = Q; p->mK = K; p->mV = V;
        p->maps_ok = true;
    }
    hg::AttnParams ap{};
    ap.bh = static_cast<int32_t>(p->bh);
    ap.sq = static_cast<int32_t>(p->sq);
    ap.skv = static_cast<int32_t>(p->skv);
    ap.nqt = static_cast<int32_t>((p->sq + 127) / 128);
    ap.causal = p->causal;
    ap.scale_log2 = static_cast<float>(static_cast<double>(p->scale) * 1.4426950408889634);
    // S = Q K^T (N = 64 keys): both operands K-major; O += P V: P from
    // tensor memory, V MN-major
    ap.idesc_s = hg::idesc_f16(static_cast<uint32_t>(bf), 0, 0, 128, 64);
    ap.idesc_o = hg::idesc_f16(static_cast<uint32_t>(bf), 0, 1, 128, 128);
    ap.O = O;
    ap.err = p->err;
    ap.timeout_ns = kAttnTimeoutNs;
    e = hg::launch_attention(bf != 0, p->tmQ, p->tmK, p->tmV, ap, s);
    return e == cudaSuccess ? HGEMM_OK : acuda(e, "attention kernel launch");
}

}  // namespace

extern "C" {

hgemm_status_t hgemm_attention_plan_create(hgemm_attn_plan_t *plan, int64_t batch_heads,
                                           int64_t seq_q, int64_t seq_kv, int64_t head_dim,
                                           float scale, int causal, hgemm_dtype_t dtype) {
    if (!plan) return afail(HGEMM_ERR_INVALID_ARG, "plan pointer is NULL");
    *plan = nullptr;
    if (dtype != HGEMM_F16 && dtype != HGEMM_BF16)
        return afail(HGEMM_ERR_INVALID_ARG, "attention dtype must be HGEMM_F16 or HGEMM_BF16 (got %d)",
                     static_cast<int>(dtype));
    if (batch_heads < 1 || seq_q < 0 || seq_kv < 0 || head_dim < 1)
        return afail(HGEMM_ERR_INVALID_ARG, "bad sizes: batch_heads %lld, seq_q %lld, seq_kv %lld, head_dim %lld",
                     static_cast<long long>(batch_heads), static_cast<long long>(seq_q),
                     static_cast<long long>(seq_kv), static_cast<long long>(head_dim));
    if (!(std::isfinite(scale) && scale > 0.f))
        return afail(HGEMM_ERR_INVALID_ARG, "scale must be finite and > 0");
    if (causal != 0 && causal != 1) return afail(HGEMM_ERR_INVALID_ARG, "causal must be 0 or 1");
    if (causal && seq_q > seq_kv)
        return afail(HGEMM_ERR_INVALID_ARG, "causal attention needs seq_q <= seq_kv (%lld > %lld)",
                     static_cast<long long>(seq_q), static_cast<long long>(seq_kv));
    if (head_dim != 128) return afail(HGEMM_ERR_UNSUPPORTED, "head_dim must be 128 (got %lld)",
                                      static_cast<long long>(head_dim));
    if (seq_q > kMax32 || seq_kv > kMax32 || batch_heads > kMax32 ||
        batch_heads * ((seq_q + 127) / 128) > kMax32)
        return afail(HGEMM_ERR_UNSUPPORTED, "sizes above 2^31-1 are not supported");
    // the byte sizes of Q / O and of K / V (staging buffers, copies) must fit
    // comfortably in 64 bits: batch_heads x seq x 128 x 2 bytes <= 2^60
    if (batch_heads > ((1ll << 52) / (seq_q > seq_kv ? (seq_q > 0 ? seq_q : 1) : (seq_kv > 0 ? seq_kv : 1))))
        return afail(HGEMM_ERR_UNSUPPORTED, "batch_heads x sequence length too large (over 2^60 bytes)");

    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return afail(HGEMM_ERR_NO_DEVICE, "no CUDA device: %s", cudaGetErrorString(e));
    int major = 0, minor = 0, sms = 0;
    cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev);
    cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev);
    cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    if (major != 10 || minor != 3)
        return afail(HGEMM_ERR_NO_DEVICE, "libhgemm is built for sm_103a; device %d is sm_%d%d", dev,
                     major, minor);
    hgemm_attn_plan_s *p = new (std::nothrow) hgemm_attn_plan_s();
    if (!p) return afail(HGEMM_ERR_OOM, "host allocation failed");
    p->bh = batch_heads; p->sq = seq_q; p->skv = seq_kv; p->d = head_dim;
    p->scale = scale; p->causal = causal; p->dt = dtype;
    p->device = dev; p->num_sms = sms;
    e = cudaMalloc(reinterpret_cast<void **>(&p->err), 256);
    if (e == cudaSuccess) e = cudaMemset(p->err, 0, 256);
    if (e != cudaSuccess) {
        if (p->err) cudaFree(p->err);
        delete p;
        return acuda(e, "cudaMalloc(attention workspace)");
    }
    *plan = p;
    return HGEMM_OK;
}

hgemm_status_t hgemm_attention_run(hgemm_attn_plan_t plan, const void *Q, const void *K,
                                   const void *V, void *O, void *stream) {
    if (!plan) return afail(HGEMM_ERR_INVALID_ARG, "plan is NULL");
    return attn_run(plan, Q, K, V, O, static_cast<cudaStream_t>(stream));
}

hgemm_status_t hgemm_attention_run_host(hgemm_attn_plan_t plan, const void *Q_host,
                                        const void *K_host, const void *V_host, void *O_host,
                                        void *stream) {
    if (!plan) return afail(HGEMM_ERR_INVALID_ARG, "plan is NULL");
    hgemm_attn_plan_s *p = plan;
    if (p->sq == 0) return HGEMM_OK;
    if (!O_host || (p->skv > 0 && (!Q_host || !K_host || !V_host)))
        return afail(HGEMM_ERR_INVALID_ARG, "host pointer is NULL");
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    const size_t qb = static_cast<size_t>(q_bytes(p)), kb = static_cast<size_t>(kv_bytes(p));
    cudaError_t e = cudaSuccess;
    if (!p->dO) {
        e = cudaMalloc(reinterpret_cast<void **>(&p->dO), qb);
        if (e == cudaSuccess && kb > 0) e = cudaMalloc(reinterpret_cast<void **>(&p->dQ), qb);
        if (e == cudaSuccess && kb > 0) e = cudaMalloc(reinterpret_cast<void **>(&p->dK), kb);
        if (e == cudaSuccess && kb > 0) e = cudaMalloc(reinterpret_cast<void **>(&p->dV), kb);
        if (e != cudaSuccess) return acuda(e, "cudaMalloc(attention staging)");
    }
    if (kb > 0) {
        if ((e = cudaMemcpyAsync(p->dQ, Q_host, qb, cudaMemcpyHostToDevice, s)) != cudaSuccess ||
            (e = cudaMemcpyAsync(p->dK, K_host, kb, cudaMemcpyHostToDevice, s)) != cudaSuccess ||
            (e = cudaMemcpyAsync(p->dV, V_host, kb, cudaMemcpyHostToDevice, s)) != cudaSuccess)
            return acuda(e, "copy Q, K, V to device");
    }
    hgemm_status_t st = attn_run(p, p->dQ, p->dK, p->dV, p->dO, s);
    if (st != HGEMM_OK) return st;
    if ((e = cudaMemcpyAsync(O_host, p->dO, qb, cudaMemcpyDeviceToHost, s)) != cudaSuccess)
        return acuda(e, "copy O to host");
    if ((e = cudaStreamSynchronize(s)) != cudaSuccess) return acuda(e, "cudaStreamSynchronize");
    return HGEMM_OK;
}

hgemm_status_t hgemm_attention_check(hgemm_attn_plan_t plan, void *stream) {
    if (!plan) return afail(HGEMM_ERR_INVALID_ARG, "plan is NULL");
    cudaError_t e = cudaStreamSynchronize(static_cast<cudaStream_t>(stream));
    if (e != cudaSuccess) return acuda(e, "stream reports an error");
    int32_t word = 0;
    e = cudaMemcpy(&word, plan->err, sizeof(word), cudaMemcpyDeviceToHost);
    if (e != cudaSuccess) return acuda(e, "reading the device error word");
    if (word != 0) {
        cudaMemset(plan->err, 0, sizeof(word));
        return afail(HGEMM_ERR_TIMEOUT, "attention: device wait timed out (code 0x%08x)",
                     static_cast<uint32_t>(word));
    }
    return HGEMM_OK;
}

hgemm_status_t hgemm_attention_plan_destroy(hgemm_attn_plan_t plan) {
    if (!plan) return HGEMM_OK;
    if (plan->err) cudaFree(plan->err);
    if (plan->dQ) cudaFree(plan->dQ);
    if (plan->dK) cudaFree(plan->dK);
    if (plan->dV) cudaFree(plan->dV);
    if (plan->dO) cudaFree(plan->dO);
    delete plan;
    return HGEMM_OK;
}

}  // extern "C"
