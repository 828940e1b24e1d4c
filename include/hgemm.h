/*
 * hgemm.h -- C ABI of libhgemm: half-precision tensor-core GEMM on GB300
 * (sm_103a).
 *
 * The operation (defined in "hgemm_mma_m16n8k16_mma2x4_warp4x4_kernel",
 * section 1.1: C = A x B with A[M x K] and B[K x N] both row-major, C row-major;
 * fp32 accumulation as in "tensor-cores-cutlass-and-cute", section 四.1):
 *
 *     C_b[i][j] = sum_{k<K} A_b[i][k] * B_b[k][j]      for b < batch
 *
 * with fp16 or bf16 inputs, fp32 accumulation, and fp32, fp16 or bf16
 * output (fp32 -> fp16/bf16 rounds to nearest even).  Element (i,k) of A_b is at
 * A + b*strideA + i*lda + k, element (k,j) of B_b at B + b*strideB + k*ldb + j,
 * and element (i,j) of C_b at C + b*strideC + i*ldc + j.  All leading
 * dimensions and strides count elements, not bytes.  hgemm_run overwrites C;
 * hgemm_run_ex adds a fused epilogue (alpha, beta times C's previous value,
 * scales, bias, activation; declared below).  The argument checks follow the
 * host wrapper of the
 * "tensor-cores-cutlass-and-cute" Ampere kernel (section 四.4): a bad dtype or
 * shape is refused, never reinterpreted.
 *
 * Ownership.  The caller owns A, B, C and the stream.  A plan owns its device
 * workspace (error word, split-K partials, aligned copies of misaligned
 * operands) and its cached TMA descriptors; hgemm_plan_destroy frees them.
 * A plan is bound to the CUDA device that is current when it is created, and
 * one plan must not run on two streams, or from two host threads, at once (its
 * workspace and cached descriptors are shared); the one-shot hgemm() keeps a
 * plan per stream for this reason.
 *
 * Errors.  Every entry point returns a status and never aborts, exits or
 * prints.  hgemm_last_error_detail() gives a message for the calling thread's
 * last failure.  Kernel launches are asynchronous: a device-side watchdog
 * timeout surfaces at hgemm_check().  Operand pointers of the device-memory
 * entry points must point into device memory of the plan's GPU (or managed
 * memory): each run asks cudaPointerGetAttributes about a pointer the first
 * time it sees it and refuses host memory, another GPU's memory or an
 * unknown address with HGEMM_ERR_INVALID_ARG, before anything is launched.
 *
 * Alignment.  Pointers must be element-aligned.  When a base pointer is
 * 16-byte aligned and its leading dimension and batch stride are multiples of
 * 16 bytes, the operand is read by TMA in place; otherwise it is first copied
 * into an aligned workspace buffer (rows padded with zeros to whole 64-element
 * blocks on the tiled path, to 8 elements on the skinny path).  A misaligned C
 * is written with predicated stores instead of TMA stores.  Nothing is refused
 * for alignment.
 */
#ifndef HGEMM_H
#define HGEMM_H

#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
    HGEMM_F16 = 0,  /* IEEE binary16 */
    HGEMM_BF16 = 1, /* bfloat16 */
    HGEMM_F32 = 2,  /* IEEE binary32 (output only) */
    HGEMM_E4M3 = 3, /* 8-bit float, 1-4-3 bits, bias 7, no infinities, S.1111.111 is NaN
                       (input only) */
    HGEMM_E5M2 = 4  /* 8-bit float, 1-5-2 bits, bias 15, IEEE-style infinities and NaNs
                       (input only) */
} hgemm_dtype_t;

typedef enum {
    HGEMM_OK = 0,
    HGEMM_ERR_INVALID_ARG = 1, /* null pointer with work to do, negative size, ld too short, bad dtype */
    HGEMM_ERR_UNSUPPORTED = 2, /* well-formed request this build does not implement */
    HGEMM_ERR_NO_DEVICE = 3,   /* no CUDA device, or not an sm_103 device */
    HGEMM_ERR_CUDA = 4,        /* a CUDA runtime/driver call failed (see detail) */
    HGEMM_ERR_OOM = 5,         /* device or host allocation failed */
    HGEMM_ERR_TIMEOUT = 6,     /* a device-side wait ran out of time (kernel aborted cleanly) */
    HGEMM_ERR_INTERNAL = 7     /* a device-side invariant check failed (debug_checks; the kernel
                                  stopped before using the offending work item) */
} hgemm_status_t;

/* Execution paths a plan can take (hgemm_plan_info_t.path). */
enum {
    HGEMM_PATH_EMPTY = 0,     /* M == 0 or N == 0: nothing to do */
    HGEMM_PATH_ZERO_FILL = 1, /* K == 0: C is set to zero (the empty sum) */
    HGEMM_PATH_TILED = 2,     /* persistent TMA + tcgen05 kernel, 128 x BN tiles */
    HGEMM_PATH_SKINNY = 3     /* small M: swap-AB, split-K, weights streamed from HBM */
};

typedef struct hgemm_plan_s *hgemm_plan_t;

/* Optional knobs for hgemm_plan_create_ex; zero-initialise and set what you
 * need.  They exist for testing and tuning: the defaults are what
 * hgemm_plan_create picks. */
typedef struct {
    int force_path;           /* 0: automatic; HGEMM_PATH_TILED or HGEMM_PATH_SKINNY to force */
    int force_generic_store;  /* 1: predicated st.global epilogue even when C suits TMA */
    int force_repack;         /* 1: copy A and B to aligned workspace even when aligned */
    int tile_n;               /* 0: automatic; 128, 192, 224 or 256 (tiled path) */
    int split_k;              /* 0: automatic; >= 1 (skinny path) */
    uint64_t timeout_ns;      /* 0: default (2 s); device watchdog for each pipeline wait */
    int cta_pair;             /* tiled path: 0 automatic, 1 force 256 x 256 tiles on CTA pairs
                                 (tcgen05 cta_group::2), 2 force single-CTA 128 x tile_n tiles */
    int skinny_tile_n;        /* skinny path: 0 automatic, or 128 / 192 / 256 / 384 / 512 columns of C per
                                 work unit */
    int no_tail_split;        /* CTA pairs: 1 runs whole tiles only, so the last partial wave of
                                 tiles stays whole (no stream-K, no K halves) */
    int pair_k_blocks;        /* CTA pairs: 0 automatic (2), or 1 / 2 64-wide K blocks per pipeline
                                 stage (tile_k of the plan info is 64 x this) */
    int tail_mode;            /* CTA pairs, the tiles that do not fill a wave: 0 automatic; 1 whole
                                 tiles; 2 K halves of each such tile, run by two pairs in the
                                 first wave (needs 2 x tail tiles <= pairs); 3 stream-K over the
                                 last waves (needs tiles >= pairs); 4 their K steps dealt to all
                                 pairs in the first wave (needs tail steps >= pairs, at most 4
                                 pieces per tile).  A forced mode whose condition fails falls
                                 back to 2, then 3, then 1. */
    int skinny_stream_k;      /* skinny path: 0 automatic (off), 1 off, 2 on: the (tile, K block)
                                 steps are dealt to the SMs in equal contiguous ranges */
    int skinny_prefetch;      /* skinny path: stages of B each CTA asks L2 for before it waits on
                                 the previous kernel of the stream; 0 automatic (4 for 8-bit
                                 inputs, none for 16-bit), -1 none */
    int group_m;              /* tiled path: m-tiles per raster group (tiles run m-fastest within a
                                 group of group_m tile rows); 0 automatic (16; 8 for CTA-pair
                                 tiles when M spans at least 32 of them) */
    int trans_b;              /* 0: B is K x N row-major (element (k, j) at B + k*ldb + j); 1: B is
                                 stored N x K row-major (element (k, j) at B + j*ldb + k, ldb >= K),
                                 i.e. C = A . B_stored^T -- a linear layer's weight, or attention's
                                 S = Q K^T with K stored [seq][dim] */
    int tiled_epi_warps;      /* single-CTA tiled path, warps that drain the accumulators: 0
                                 automatic (4; 8 for runs with the fused epilogue when the
                                 inputs are 16-bit, the tile 128 or 256 wide and K <= 1024), 4,
                                 or 8 (16-bit inputs and tile widths 128 / 256 only, else
                                 HGEMM_ERR_UNSUPPORTED) */
    int debug_withhold_kb;    /* testing the abort path only: 0 off; k >= 1 makes CTA 0 of the
                                 single-CTA tiled kernel leave the pipeline stage of K block k of
                                 its first tile unarmed and unloaded, so the MMA issuer's wait on it
                                 runs out after timeout_ns; the run then leaves C incomplete and
                                 hgemm_check returns HGEMM_ERR_TIMEOUT.  k <= ceil(K / 64); plans
                                 that take another kernel (CTA pairs, skinny, 8-bit inputs) get
                                 HGEMM_ERR_UNSUPPORTED */
    int debug_checks;         /* 0: off unless the environment variable HGEMM_DEBUG is set to a
                                 non-zero value; 1: before its roles start, every CTA walks its
                                 whole sequence of work items with the scheduler's own code and
                                 checks their invariants (tile and coordinates inside the output,
                                 K range inside K, piece inside its tile); on a violation it
                                 records it in the device error word and does no work at all:
                                 hgemm_check then returns HGEMM_ERR_INTERNAL.  No trap, no assert.
                                 (A CTA pair whose K-half or stream-K partner stopped this way
                                 waits for it until the watchdog limit.)  2: testing the check
                                 only -- the first work item of CTA 0 (or CTA pair 0) is given a
                                 tile index past the last tile, which the check must catch */
} hgemm_options_t;

/* Read-only description of what a plan will launch. */
typedef struct {
    int path;             /* HGEMM_PATH_* */
    int tile_m, tile_n, tile_k;
    int stages;           /* shared-memory pipeline depth */
    int split_k;          /* K splits (skinny path), else 1 */
    int grid;             /* CTAs of the main kernel (persistent: <= SM count) */
    int repack_a;         /* 1: A is copied to an aligned workspace first */
    int repack_b;         /* 1: B likewise */
    int tma_store;        /* 1: TMA-store epilogue; 0: predicated st.global */
    int kernels_per_run;  /* kernel launches one hgemm_run makes */
    int64_t workspace_bytes;
    int tail_split;       /* CTA pairs: 2 when the last partial wave's tiles run as two K halves */
    int wide_boxes;       /* CTA pairs: 1 when each pipeline stage of A and of B is one TMA copy
                             (4-D views; 256-wide tiles, K and N multiples of 64, or the
                             operand read from its zero-padded aligned copy).  Before the
                             first run: as the leading dimensions decide; after it: what
                             the last run used */
    int trans_b;          /* the plan's B layout (hgemm_options_t.trans_b) */
    int stream_k;         /* K steps dealt in equal contiguous ranges: CTA pairs 1 (tail_mode 3)
                             or 2 (tail_mode 4), the skinny path 1 (skinny_stream_k; split_k is
                             then the most pieces a column tile is cut into) */
    int epi_warps;        /* tiled path: warps draining the accumulators in plain runs (4 or 8;
                             CTA pairs 4), else 0 */
    int epi_warps_epilogue; /* the same for runs with the fused epilogue (hgemm_run_ex) */
    int host_chunks;      /* hgemm_run_host: row chunks whose copies in, products and copies out
                             overlap (batch 1, M >= 1024, A and C >= 16 MB together), or 1 */
} hgemm_plan_info_t;

/* Creates a plan for C_b = A_b . B_b, b < batch.
 *   M, N, K          >= 0.  M == 0 or N == 0 makes an empty plan; K == 0 a
 *                    plan that writes zeros.
 *   lda >= K, ldb >= N, ldc >= N (elements; checked only when that operand
 *                    has rows to read or write).
 *   batch >= 1; strideA/B/C (elements) are used only when batch > 1 and must
 *                    then be >= 0.
 *   dtype_in  in {HGEMM_F16, HGEMM_BF16, HGEMM_E4M3, HGEMM_E5M2} (applies to
 *                    both A and B).
 *   dtype_out in {HGEMM_F32, HGEMM_F16, HGEMM_BF16}.
 * 8-bit inputs (HGEMM_E4M3 / HGEMM_E5M2) are multiplied exactly and summed in
 * fp32 like the 16-bit ones, at the tensor cores' 8-bit rate: the
 * "tensor-cores-cutlass-and-cute" page lists FP8 e4m3 with fp32
 * accumulation among the tensor-core input types, notes that an instruction
 * consumes a fixed number of bytes along K (so twice the K of a 16-bit type),
 * and takes K blocks of 128 one-byte elements where bf16 takes 64 (its
 * section on vLLM's FP8 kernels).  They take the
 * layout those units read without a copy, and anything else is
 * HGEMM_ERR_UNSUPPORTED: B stored N x K (options.trans_b = 1, so both
 * operands are contiguous along K); lda and ldb multiples of 16; with
 * batch > 1, strideA and strideB multiples of 16; A and B 16-byte aligned
 * (checked by hgemm_run); no force_repack; tile_n 0, 128 or 256,
 * pair_k_blocks 0 or 2, skinny_tile_n 0, 128 or 256.  Per-tensor or
 * per-channel dequantisation scales go in the epilogue (alpha, row_scale,
 * col_scale of hgemm_run_ex).
 * Validation needs no GPU; on valid arguments the current device must be an
 * sm_103 GPU (else HGEMM_ERR_NO_DEVICE).  Device workspace is allocated here.
 * On success *plan receives a handle the caller must destroy. */
hgemm_status_t hgemm_plan_create(hgemm_plan_t *plan, int64_t M, int64_t N, int64_t K,
                                 int64_t lda, int64_t ldb, int64_t ldc, int64_t batch,
                                 int64_t strideA, int64_t strideB, int64_t strideC,
                                 hgemm_dtype_t dtype_in, hgemm_dtype_t dtype_out);

/* As hgemm_plan_create, with options (NULL = defaults). */
hgemm_status_t hgemm_plan_create_ex(hgemm_plan_t *plan, int64_t M, int64_t N, int64_t K,
                                    int64_t lda, int64_t ldb, int64_t ldc, int64_t batch,
                                    int64_t strideA, int64_t strideB, int64_t strideC,
                                    hgemm_dtype_t dtype_in, hgemm_dtype_t dtype_out,
                                    const hgemm_options_t *options);

/* Enqueues the product on `stream` (a cudaStream_t; NULL = legacy default
 * stream).  A, B, C are device pointers laid out as the plan says.  Returns
 * once the kernels are enqueued; the result is ready when the stream is.
 * INVALID_ARG for a null pointer when the plan has work to do. */
hgemm_status_t hgemm_run(hgemm_plan_t plan, const void *A, const void *B, void *C, void *stream);

/* Fused epilogue: the kernels write, for every element of C,
 *
 *     D[i][j] = act(alpha * rs[i] * cs[j] * (A.B)[i][j] + beta * C[i][j] + bias[j])
 *
 * (C on the right is the value C held before the call), rounded once to the
 * output type.  The terms follow the bias / ReLU / GELU epilogues the pages
 * list among cuBLASLt's features ("tensor-cores-cutlass-and-cute", its
 * comparison with cuBLAS); scale, add, then activate.  All arithmetic is
 * fp32.  Vectors are device fp32 arrays shared by every batch entry; NULL
 * means rs = 1, cs = 1, bias = 0.  beta == 0 leaves C unread (it may hold
 * anything, NaN included). */
typedef enum {
    HGEMM_ACT_NONE = 0,
    HGEMM_ACT_RELU = 1, /* max(x, 0) */
    HGEMM_ACT_GELU = 2, /* x * Phi(x) = 0.5 x (1 + erf(x / sqrt 2)); erf by Abramowitz &
                           Stegun 7.1.26 (absolute error <= 1.5e-7) */
    HGEMM_ACT_GELU_TANH = 3 /* 0.5 x (1 + tanh(sqrt(2/pi) (x + 0.044715 x^3))), the tanh form
                               (tanh from the hardware approximation) */
} hgemm_activation_t;

typedef struct {
    float alpha;            /* scales the product */
    float beta;             /* scales C's previous value; 0: C is not read */
    const float *bias;      /* N values added per column, or NULL */
    const float *row_scale; /* M values scaling row i of the product, or NULL */
    const float *col_scale; /* N values scaling column j of the product, or NULL */
    int activation;         /* hgemm_activation_t, applied last */
} hgemm_epilogue_t;

/* hgemm_run with a fused epilogue (NULL: plain product, as hgemm_run).
 * INVALID_ARG for an unknown activation or non-finite alpha / beta. */
hgemm_status_t hgemm_run_ex(hgemm_plan_t plan, const void *A, const void *B, void *C, void *stream,
                            const hgemm_epilogue_t *epilogue);

/* End-to-end variant for operands in HOST memory (pinned memory is fastest):
 * copies A and B to plan-owned device buffers on `stream`, runs the product,
 * copies the M x N block(s) of C back into the host buffer (elements outside
 * the block are left untouched), and synchronises `stream` before returning.
 * A large product (plan info host_chunks > 1) runs in row chunks: B and then
 * the rows of A chunk by chunk are copied in on a second stream, each chunk's
 * product runs on `stream` as soon as its rows have arrived, and its rows of
 * C are copied out on a third stream as soon as it is done, so copies in,
 * products and copies out overlap.  The streams and the chunks' plans are
 * made on the first such call and kept by the plan; all the work is ordered
 * after what was queued on `stream` before the call.
 * It then reads the plan's device error word as hgemm_check does: after a
 * watchdog timeout it returns HGEMM_ERR_TIMEOUT (C_host is then incomplete)
 * and clears the word.  The device buffers are allocated on the first call
 * and kept by the plan. */
hgemm_status_t hgemm_run_host(hgemm_plan_t plan, const void *A_host, const void *B_host,
                              void *C_host, void *stream);

/* Synchronises `stream` and reads the plan's device error word.  Returns
 * HGEMM_ERR_TIMEOUT if a pipeline wait of an earlier hgemm_run ran out of
 * time (the kernel then left C incomplete but released all its resources),
 * HGEMM_ERR_CUDA if the stream reports a CUDA error, else HGEMM_OK.  The
 * error word is cleared on read. */
hgemm_status_t hgemm_check(hgemm_plan_t plan, void *stream);

/* Frees the plan's workspace; the caller must make sure no hgemm_run of it
 * is still executing.  NULL is accepted. */
hgemm_status_t hgemm_plan_destroy(hgemm_plan_t plan);

/* Fills *info with what the plan launches. */
hgemm_status_t hgemm_plan_get_info(hgemm_plan_t plan, hgemm_plan_info_t *info);

/* One-shot product: looks up (or creates and keeps) a plan for these
 * arguments and this stream in a process-wide cache, then runs it on
 * `stream`.  Each stream gets a plan (and workspace) of its own, so one-shot
 * calls may run on several streams and from several host threads at once.
 * Cached plans live until hgemm_cache_clear() or process exit. */
hgemm_status_t hgemm(const void *A, const void *B, void *C, int64_t M, int64_t N, int64_t K,
                     int64_t lda, int64_t ldb, int64_t ldc, int64_t batch, int64_t strideA,
                     int64_t strideB, int64_t strideC, hgemm_dtype_t dtype_in,
                     hgemm_dtype_t dtype_out, void *stream);

/* Destroys every cached one-shot plan (the caller makes sure none is running). */
hgemm_status_t hgemm_cache_clear(void);

/* Watchdog self-test: launches a one-warp kernel that waits, with the same
 * bounded wait the GEMM pipeline uses, on an mbarrier that nothing signals.
 * The wait must give up after `timeout_ns` and report it.  On return
 * *device_code holds the error word the kernel wrote (non-zero when the
 * watchdog fired) and the status is HGEMM_ERR_TIMEOUT in that case. */
hgemm_status_t hgemm_watchdog_selftest(uint64_t timeout_ns, void *stream, int32_t *device_code);

/* Allocation-free product for small M (no counterpart on the source pages:
 * it exists for callers, not for the method).  The same swap-AB split-K
 * kernel as the planned skinny path, for callers that may not allocate
 * device memory: a host framework that owns every allocation and hands over
 * only input and output buffers, a process whose device memory is budgeted
 * at start-up, or a latency-critical loop where cudaMalloc's implicit
 * synchronisation is not acceptable.  It calls no cudaMalloc, cudaFree or
 * allocating library routine.
 *   A: M x K (lda), B: K x N (ldb), C: M x N (ldc), row-major, batch 1,
 *   device pointers; M <= 32; A and B 16-byte aligned with lda and ldb
 *   multiples of 8 elements (no aligned copies can be made);
 *   dtype_in in {F16, BF16}, dtype_out in {F32, F16, BF16}; enqueued on
 *   `stream`, asynchronous.
 * Its split-K partial sums, counters and error word live in one 8 MiB
 * __device__ array inside the library, held by every GPU that loads it until
 * the process exits.  The first call on each device (and the first after
 * the device gets a new CUDA context) looks up that array's device address;
 * make the first call before any stream capture.  Every call
 * shares the array: calls that overlap on the GPU race and must be ordered.
 * The split count is lowered to fit the array; a request that does not fit
 * even unsplit returns HGEMM_ERR_UNSUPPORTED, as do misaligned operands and
 * M > 32.  A device watchdog timeout is not returned here (the kernel runs
 * after the call returns): hgemm_skinny_noalloc_check reports it. */
hgemm_status_t hgemm_skinny_noalloc(const void *A, const void *B, void *C, int64_t M, int64_t N,
                                    int64_t K, int64_t lda, int64_t ldb, int64_t ldc,
                                    hgemm_dtype_t dtype_in, hgemm_dtype_t dtype_out, void *stream);

/* Status of the last hgemm_skinny_noalloc product on the current device, the
 * allocation-free counterpart of hgemm_check: synchronises `stream` (the
 * stream that product used), reads the array's device error word and clears
 * it.  HGEMM_OK, or HGEMM_ERR_TIMEOUT when a device wait of that product
 * timed out (C is then incomplete; the detail names the role and barrier).
 * Allocates nothing.  Call it after the product and before the next
 * hgemm_skinny_noalloc on the device, which clears the word before its
 * kernel runs. */
hgemm_status_t hgemm_skinny_noalloc_check(void *stream);

/* ---------------------------------------------------------------- attention
 *
 * Fused attention forward: the block the "post_1787550000" experiment builds
 * its tensor-core work toward (its sections 1-2: the products S = Q K^T and
 * O = P V of a FlashAttention kernel on the tensor cores, the softmax of S
 * between them, P handed to the second product without a trip through
 * memory, and a causal mask), with the row-wise max and sum of S the
 * "hgemm_mma_m16n8k16_mma2x4_warp4x4_kernel" page describes (its section 2).
 * For every head b < batch_heads and query row i < seq_q:
 *
 *     O[b][i] = sum_j p_j V[b][j] / sum_j p_j,
 *     p_j     = exp(scale * Q[b][i] . K[b][j] - max_j(...)),
 *
 * over the allowed keys j: every j < seq_kv, or with `causal`
 * j <= i + seq_kv - seq_q (the last query row sees every key).
 *   Q  [batch_heads][seq_q][head_dim], K and V [batch_heads][seq_kv][head_dim],
 *   O  [batch_heads][seq_q][head_dim]: dense row-major device arrays of
 *      `dtype` (HGEMM_F16 or HGEMM_BF16, O included), 16-byte aligned.
 * Scores and softmax are fp32; the probabilities are rounded to `dtype` for
 * the product with V, which accumulates in fp32; O is rounded once.
 * head_dim must be 128 (else HGEMM_ERR_UNSUPPORTED); scale finite and > 0;
 * causal needs seq_q <= seq_kv, so that every row has a key (else
 * HGEMM_ERR_INVALID_ARG).  seq_q == 0 does nothing; seq_kv == 0 writes
 * zeros (the empty sum).  Plans own a small device workspace (the error
 * word), cached TMA descriptors and the staging buffers of
 * hgemm_attention_run_host; as with GEMM plans, one plan must not run on two
 * streams or from two host threads at once: give each its own plan. */
typedef struct hgemm_attn_plan_s *hgemm_attn_plan_t;

hgemm_status_t hgemm_attention_plan_create(hgemm_attn_plan_t *plan, int64_t batch_heads,
                                           int64_t seq_q, int64_t seq_kv, int64_t head_dim,
                                           float scale, int causal, hgemm_dtype_t dtype);

/* Enqueues the attention forward on `stream` (device pointers; returns once
 * enqueued).  INVALID_ARG for a null or misaligned pointer. */
hgemm_status_t hgemm_attention_run(hgemm_attn_plan_t plan, const void *Q, const void *K,
                                   const void *V, void *O, void *stream);

/* As hgemm_attention_run with Q, K, V and O in host memory: copies the
 * inputs to plan-owned device buffers, runs, copies O back and synchronises
 * `stream`. */
hgemm_status_t hgemm_attention_run_host(hgemm_attn_plan_t plan, const void *Q_host,
                                        const void *K_host, const void *V_host, void *O_host,
                                        void *stream);

/* Synchronises `stream` and reads the plan's device error word, as
 * hgemm_check does for GEMM plans (HGEMM_ERR_TIMEOUT after a watchdog
 * timeout; the word is cleared on read). */
hgemm_status_t hgemm_attention_check(hgemm_attn_plan_t plan, void *stream);

/* Frees the plan (NULL accepted); no run of it may still be executing. */
hgemm_status_t hgemm_attention_plan_destroy(hgemm_attn_plan_t plan);

const char *hgemm_status_string(hgemm_status_t status);
const char *hgemm_last_error_detail(void);

/* Library version as MAJOR*10000 + MINOR*100 + PATCH. */
int32_t hgemm_version(void);

#ifdef __cplusplus
}
#endif

#endif /* HGEMM_H */
