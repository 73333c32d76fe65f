/*
 * sdpa_math.h -- C ABI of the GB300 (sm_103a) materialised-probability
 * scaled-dot-product-attention forward.
 *
 * The operation is the SDPA "math" backend forward that returns both the
 * output and the full attention-probability map (FlagOS-OP PR #10
 * "feat: add sdpa_math operator", overview: aten::_scaled_dot_product_attention_math
 * returning (out, attn_probs)):
 *
 *     S = scale * Q K^T  (+ additive mask | -inf where a bool mask is false
 *                         | -inf above the diagonal when causal)
 *     P = softmax(S)  along the key axis          P: [B, Hq, Sq, Skv]
 *     O = P V                                     O: [B, Hq, Sq, Dv]
 *
 * with the semantics fixed by that page ("semantics" item of the overview):
 *   - is_causal together with a mask is an error;
 *   - a bool mask means -inf masking (True keeps a key, False removes it),
 *     aligned with F.scaled_dot_product_attention;
 *   - a row whose keys are all masked gives P = 0 and O = 0 (not NaN);
 *   - grouped-query attention needs Hq divisible by Hkv (query head h reads
 *     key/value head h / (Hq/Hkv)); otherwise an error;
 *   - no dropout (dropout_p = 0).
 * Causal masking is top-left aligned: key j is visible to query i iff j <= i.
 *
 * Layout and ownership (all calls):
 *   - Every tensor is a logical rank-4 array described by sdpa_tensor: a data
 *     pointer (DEVICE memory for sdpa_math_fwd*), a dtype, four extents and
 *     four strides counted in ELEMENTS.  The innermost stride must be 1 (the
 *     page's "_d1(): only stride(-1) == 1 is required", micro-optimisation
 *     item of the 2026-10-02 update); the other strides are free, so
 *     transposed [B,S,H,D] storage is accepted without a copy.  Inputs may
 *     be broadcast views (stride 0 over a batch, head or row dimension, as
 *     torch's expand() makes); the tensor-core families that read 128-row
 *     TMA tiles serve batch and head broadcasts and leave broadcast rows to
 *     the other families.  Outputs must not overlap themselves: a stride-0
 *     dimension of extent > 1 in out, probs, dq, dk or dv is an error.
 *   - The caller owns every buffer and the stream.  The library allocates no
 *     device memory per call and keeps no pointer after the call returns.
 *   - out and probs are written in full (every element, including the zeros
 *     above a causal diagonal and the zeros of fully masked rows); their prior
 *     contents are irrelevant.  They must not alias the inputs or each other.
 *   - Calls are asynchronous on `stream` (a cudaStream_t; NULL = the legacy
 *     default stream).  A call returns after enqueuing its kernels.
 *
 * Errors: every argument check happens on the host before any launch; on a
 * non-OK status nothing was enqueued and sdpa_math_last_error() returns a
 * message (thread-local).  Launch failures return SDPA_ERR_CUDA.
 */
#ifndef SDPA_MATH_H
#define SDPA_MATH_H

#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

#define SDPA_MATH_ABI_VERSION 1

/* Same type as cudaStream_t (struct CUstream_st *), without needing CUDA headers. */
typedef struct CUstream_st *sdpa_stream_t;

typedef enum {
    SDPA_OK = 0,
    SDPA_ERR_INVALID_ARGUMENT = 1, /* shape / dtype / stride / semantics violation */
    SDPA_ERR_UNSUPPORTED = 2,      /* valid request outside what is built (D > 256, dtype) */
    SDPA_ERR_CUDA = 3,             /* a CUDA runtime call or launch failed */
    SDPA_ERR_TIMEOUT = 4           /* a bounded device-side wait gave up (see sdpa_math_device_status) */
} sdpa_status;

typedef enum {
    SDPA_F32 = 0,
    SDPA_F16 = 1,
    SDPA_BF16 = 2,
    SDPA_BOOL = 3 /* one byte per element, 0 = false, anything else = true */
} sdpa_dtype;

typedef enum {
    SDPA_MASK_NONE = 0,
    SDPA_MASK_BOOL = 1,    /* mask dtype SDPA_BOOL: false -> -inf */
    SDPA_MASK_ADDITIVE = 2 /* mask dtype = the q dtype or SDPA_F32: added to scale*QK^T */
} sdpa_mask_kind;

/* Kernel families.  AUTO chooses by counting live score tiles (see sdpa_math_plan). */
typedef enum {
    SDPA_VARIANT_AUTO = 0,
    SDPA_VARIANT_SIMT = 1,       /* CUDA-core kernel: any dtype, D <= 256, any layout */
    SDPA_VARIANT_TC_TWOPASS = 2, /* tcgen05: row-LSE sweep, then exact P = exp(S - lse) and P V */
    SDPA_VARIANT_TC_FUSED = 3,   /* tcgen05: one sweep, the whole score row block kept in TMEM */
    SDPA_VARIANT_DECODE = 4,     /* few query rows per KV head: KV split across a CTA cluster */
    SDPA_VARIANT_TC_PAIRED = 5,  /* TC_TWOPASS with two query tiles per CTA sharing each K/V load */
    SDPA_VARIANT_SPLIT = 6,      /* few query rows, long key sequence: keys split over a cluster of up
                                    to 16 CTAs, scores kept on chip, V streamed (split-KV) */
    SDPA_VARIANT_TC_DECODE = 7,  /* few query rows, D = Dv = 128, f16/bf16: the cluster split of SPLIT
                                    with S^T = K Q^T and O^T = V^T P^T on the tensor cores, K / V by TMA */
    SDPA_VARIANT_TC_ONESWEEP = 8 /* tcgen05, one Q K^T sweep: the live key tiles of a 128-row block
                                    split over a cluster of up to 8 CTAs (4 tiles each, so at most
                                    32 tiles = 4096 keys per row block), exp2(S - tile max) kept in
                                    TMEM, row LSE by DSMEM, then P = that * exp2(max - lse) */
} sdpa_variant;

typedef struct {
    void *data;          /* base pointer (device memory for the fwd calls) */
    sdpa_dtype dtype;
    int64_t shape[4];    /* logical extents */
    int64_t stride[4];   /* in elements; stride[3] must be 1 when shape[3] > 1 */
} sdpa_tensor;

/*
 * sdpa_math_fwd -- (O, P) forward.
 *
 *   q     [B, Hq,  Sq,  D ]  f32 | f16 | bf16
 *   k     [B, Hkv, Skv, D ]  same dtype as q
 *   v     [B, Hkv, Skv, Dv]  same dtype as q
 *   mask  NULL iff mask_kind == SDPA_MASK_NONE; otherwise [Bm, Hm, Sq, Skv]
 *         with Bm in {1, B} and Hm in {1, Hq} (size-1 extents broadcast).
 *   is_causal  nonzero = top-left causal masking; must be 0 when a mask is given.
 *   scale      multiplier of Q K^T (finite).  The usual choice is 1/sqrt(D).
 *   out   [B, Hq, Sq, Dv]   written, dtype of q
 *   probs [B, Hq, Sq, Skv]  written, dtype of q (the materialised P)
 *   stream     cudaStream_t to enqueue on.
 *
 * Returns SDPA_ERR_INVALID_ARGUMENT for: a NULL tensor or data pointer (when
 * the tensor has elements), a negative extent, dtype mismatch among
 * q/k/v/out/probs, B mismatch, K and V disagreeing on Skv or Hkv, q and k
 * disagreeing on D, Hq % Hkv != 0, causal together with a mask, a mask shape
 * outside {1,B} x {1,Hq} x Sq x Skv, a mask dtype not allowed for its kind,
 * an innermost stride != 1, out or probs with the wrong shape or with a
 * stride-0 dimension of extent > 1, a data pointer not aligned to its
 * element size, or a non-finite scale.  Returns
 * SDPA_ERR_UNSUPPORTED for D or Dv > 256 or an input dtype that is not
 * f32/f16/bf16.
 */
sdpa_status sdpa_math_fwd(const sdpa_tensor *q, const sdpa_tensor *k, const sdpa_tensor *v,
                          const sdpa_tensor *mask, sdpa_mask_kind mask_kind, int is_causal,
                          float scale, sdpa_tensor *out, sdpa_tensor *probs,
                          sdpa_stream_t stream);

/*
 * sdpa_math_fwd_ex -- sdpa_math_fwd with a forced kernel family and an
 * optional row log-sum-exp output (the exact-P identity of the page's
 * "P800 exact-P fast path" update: P = exp(scale*QK^T - LSE)).
 *
 *   variant  SDPA_VARIANT_AUTO, or a family to force (a test / profiling hook,
 *            the analogue of the page's SDPA_MATH_FUSED=on/off/auto switch).
 *            A forced family that cannot serve the request returns
 *            SDPA_ERR_UNSUPPORTED with a message saying why.
 *   lse      NULL, or a DEVICE pointer to B*Hq*Sq contiguous floats written with
 *            the natural-log LSE of each row ([B, Hq, Sq] order), -inf for a
 *            fully masked row.
 */
sdpa_status sdpa_math_fwd_ex(const sdpa_tensor *q, const sdpa_tensor *k, const sdpa_tensor *v,
                             const sdpa_tensor *mask, sdpa_mask_kind mask_kind, int is_causal,
                             float scale, sdpa_tensor *out, sdpa_tensor *probs, float *lse,
                             sdpa_variant variant, sdpa_stream_t stream);

/* Host-only planning result (no CUDA call is made). */
typedef struct {
    sdpa_variant variant;     /* family AUTO would launch */
    int64_t live_score_tiles; /* 128x128 score tiles left after causal truncation, all (b, h) */
    int64_t launches;         /* kernels the call enqueues */
} sdpa_plan;

/*
 * sdpa_math_plan -- validate exactly like sdpa_math_fwd and report the kernel
 * family the call would use.  AUTO's rule, in order: fp32 -> SIMT; at most 16
 * query rows per KV head -> DECODE while a 1/8 key chunk fits it, else
 * TC_DECODE (D = Dv = 128, f16/bf16), else SPLIT; otherwise the tensor-core
 * families, chosen by the number of score tiles that survive causal truncation
 * rather than by area (the page's fusion criterion, "single-kernel fusion
 * (small shapes)" update): TC_FUSED while every 128-row block keeps at most
 * two live 128-key tiles (Skv <= 256, or causal with Sq <= 256), then TC_PAIRED (two query
 * tiles per CTA) for calls without a causal mask when the paired grid still
 * gives about one CTA per SM, else TC_TWOPASS; SIMT when none accepts the
 * layout.  `requested` is the variant the caller would pass to
 * sdpa_math_fwd_ex (AUTO = let the rule choose).  Data pointers are checked
 * for NULL and alignment but never dereferenced; the only CUDA call is a
 * query of the current device's SM count (nothing is enqueued).
 */
sdpa_status sdpa_math_plan(const sdpa_tensor *q, const sdpa_tensor *k, const sdpa_tensor *v,
                           const sdpa_tensor *mask, sdpa_mask_kind mask_kind, int is_causal,
                           float scale, const sdpa_tensor *out, const sdpa_tensor *probs,
                           sdpa_variant requested, sdpa_plan *plan);

/*
 * sdpa_math_device_status -- synchronise `stream`, then read and clear the
 * library's device error word.  Every device-side wait of the tensor-core
 * kernels has an iteration limit; a wait that runs out records itself there
 * and the kernel returns early (freeing its tensor memory) instead of hanging.
 * Returns SDPA_OK, SDPA_ERR_TIMEOUT (with the location in the message) or
 * SDPA_ERR_CUDA.
 */
sdpa_status sdpa_math_device_status(sdpa_stream_t stream);

/*
 * sdpa_math_bwd -- gradients of the (O, P) forward for q, k and v when both
 * outputs carry a gradient (FlagOS-OP PR #10: the overview's A1 item, where
 * the gradient flows through dout and dprobs; "2026-10-07 update: P800 fused
 * backward", where dprobs goes through the exact softmax Jacobian of the
 * materialised map and GQA gradients are reduced back to the KV heads):
 *     dP = dout V^T + dprobs,   dS = P * (dP - rowsum(P * dP))
 *     dq = scale dS K,   dk = scale dS^T Q,   dv = P^T dout
 * with dk and dv summed over the query heads of each KV head.
 *
 *   q, k, v  the forward's inputs ([B,Hq,Sq,D], [B,Hkv,Skv,D], [B,Hkv,Skv,Dv]);
 *   probs    the forward's P [B,Hq,Sq,Skv] (it already holds the mask and the
 *            causal zeros, so neither is passed again; masked keys and fully
 *            masked rows get no gradient);
 *   dout     [B,Hq,Sq,Dv]; dprobs [B,Hq,Sq,Skv], or NULL for no gradient
 *            through P;
 *   dq, dk, dv  outputs with the shapes of q, k, v, fully overwritten;
 *   rowsum   caller-owned DEVICE buffer of B*Hq*Sq floats, written with
 *            rowsum(P * dP) per row ([B, Hq, Sq] order); the library
 *            allocates nothing.
 * All tensors share one dtype (f32 / f16 / bf16, fp32 accumulation), device
 * pointers, unit innermost stride; D, Dv <= 256.  Asynchronous on `stream`.
 * Errors as sdpa_math_fwd (argument checks on the host before any launch).
 * f16 / bf16 calls with D == Dv in {64, 128} and 16-byte aligned rows run on
 * the tensor cores (two kernels: per query tile dq and rowsum, then per key
 * tile dk and dv; dS is rounded to the input dtype as an MMA operand); every
 * other call runs on two CUDA-core kernels with fp32 dS.
 */
sdpa_status sdpa_math_bwd(const sdpa_tensor *q, const sdpa_tensor *k, const sdpa_tensor *v,
                          const sdpa_tensor *probs, const sdpa_tensor *dout, const sdpa_tensor *dprobs,
                          float scale, sdpa_tensor *dq, sdpa_tensor *dk, sdpa_tensor *dv, float *rowsum,
                          sdpa_stream_t stream);

/*
 * sdpa_math_bwd_ex -- sdpa_math_bwd with the kernel family chosen by the
 * caller: SDPA_VARIANT_AUTO (as sdpa_math_bwd), SDPA_VARIANT_SIMT (the
 * CUDA-core kernels, any supported shape) or SDPA_VARIANT_TC_TWOPASS (the
 * tensor-core kernels; SDPA_ERR_UNSUPPORTED with the reason when the call
 * does not meet their conditions).  Any other value is SDPA_ERR_INVALID_ARGUMENT.
 */
sdpa_status sdpa_math_bwd_ex(const sdpa_tensor *q, const sdpa_tensor *k, const sdpa_tensor *v,
                             const sdpa_tensor *probs, const sdpa_tensor *dout, const sdpa_tensor *dprobs,
                             float scale, sdpa_tensor *dq, sdpa_tensor *dk, sdpa_tensor *dv, float *rowsum,
                             sdpa_variant variant, sdpa_stream_t stream);

/*
 * sdpa_math_bwd_noalloc -- sdpa_math_bwd for callers that cannot allocate
 * device memory.  (The pages have no counterpart of this call; it is an
 * addition of this library.)
 *
 * sdpa_math_bwd needs a B*Hq*Sq float buffer from the caller to carry the
 * per-row sums from its first kernel to its second.  Some callers cannot
 * provide one: code hosted inside a framework that hands out all device
 * memory from its own pre-planned pool and forbids side allocations, or a
 * real-time path that must not call cudaMalloc after start-up because the
 * call can block and synchronise the device.  This entry point takes no such
 * buffer.  It uses a fixed array in the library's own device memory instead
 * (SDPA_BWD_NOALLOC_MAX_ROWS floats, 4 MiB, held by every GPU that loads the
 * library until the process exits) and allocates nothing: no cudaMalloc, no
 * cudaFree, no allocating library routine.
 *
 * Arguments, semantics, kernels and results are those of sdpa_math_bwd with
 * an internal rowsum buffer (the per-row sums are not returned).  The caller
 * still owns q, k, v, probs, dout, dprobs, dq, dk, dv and the stream.
 *
 *   - Size limit: B*Hq*Sq (the query rows of q) must not exceed
 *     SDPA_BWD_NOALLOC_MAX_ROWS; larger calls return SDPA_ERR_UNSUPPORTED
 *     before anything is enqueued.
 *   - Set-up: the first call on each device looks up the array's device
 *     address (with that device current) and keeps it for later calls; make
 *     that first call before any stream capture.  A failed look-up returns
 *     SDPA_ERR_CUDA.
 *   - Sharing: every call on a device uses the same array, and it keeps the
 *     last call's contents.  Nothing in it needs to start at zero (each call
 *     writes every row it later reads).  Two calls whose kernels overlap on
 *     the GPU (for example on two streams without ordering between them)
 *     race on the array and give wrong gradients: order such calls.
 * Other errors as sdpa_math_bwd.
 */
#define SDPA_BWD_NOALLOC_MAX_ROWS (1 << 20)
sdpa_status sdpa_math_bwd_noalloc(const sdpa_tensor *q, const sdpa_tensor *k, const sdpa_tensor *v,
                                  const sdpa_tensor *probs, const sdpa_tensor *dout, const sdpa_tensor *dprobs,
                                  float scale, sdpa_tensor *dq, sdpa_tensor *dk, sdpa_tensor *dv,
                                  sdpa_stream_t stream);

/*
 * sdpa_math_selftest_wait -- diagnostic for the failure path above.  Enqueues
 * on `stream` one single-thread kernel that waits, through the same bounded
 * mbarrier wait the tensor-core kernels use, on a barrier nothing ever
 * arrives at.  The wait runs out after about one second, records role 15 in
 * the device error word and the kernel returns; no fault, no hang.  A
 * following sdpa_math_device_status(stream) then returns SDPA_ERR_TIMEOUT.
 * Returns SDPA_OK, or SDPA_ERR_CUDA if the launch fails.
 */
sdpa_status sdpa_math_selftest_wait(sdpa_stream_t stream);

/* Message for the last non-OK status returned on this thread ("" if none). */
const char *sdpa_math_last_error(void);

/* SDPA_MATH_ABI_VERSION of the loaded library. */
int sdpa_math_abi_version(void);

#ifdef __cplusplus
}
#endif

#endif /* SDPA_MATH_H */
