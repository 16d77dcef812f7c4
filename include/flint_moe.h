/*
 * flint_moe.h -- C ABI of the Flint mixture-of-experts FFN layer for B300
 * (sm_103a).
 *
 * The layer (RecursiveSI/flint, vLLM recipe page, "Overview": a
 * mixture-of-experts model with 256 experts, top-6 sigmoid routing plus a
 * shared expert; neoteo.com "Model kodujacy Flint", specification table: six
 * routed experts per token plus one shared expert that is always active):
 *
 *   l[t,e] = sum_h x[t,h] Wr[e,h] + b[e]                (router, fp32 accumulate)
 *   S_t    = 6 experts with the largest l[t,e]          (equal logits: lower index)
 *   w[t,j] = sigmoid(l[t,S_tj]) / sum_j' sigmoid(l[t,S_tj'])
 *   y[t]   = sum_j w[t,j] FFN_{S_tj}(x_t) + FFN_shared(x_t)
 *   FFN(x) = Wd (silu(Wg x) * (Wu x)),  silu(z) = z / (1 + exp(-z))
 *
 * The pages give the expert count, top-6, the sigmoid and the shared expert.
 * They do not give the hidden size, the expert width, the activation or the
 * weight normalisation; this library fixes H = 2048, I = 512, SwiGLU experts,
 * weights renormalised to sum to one and an unweighted shared expert (those
 * sizes reproduce the pages' 39.8B total / ~2.5B active parameter counts).
 *
 * Memory: every pointer below is a DEVICE pointer unless marked "host".  All
 * matrices are row-major [out][in] (each row contiguous along the reduced
 * dimension).  bf16 = IEEE binary32's upper 16 bits.  Device buffers must be
 * 16-byte aligned.
 *
 * Errors: every call returns a flint_status_t.  Arguments are checked on the
 * host before anything is launched.  Kernels report device-side problems
 * (a bounded wait that ran out, an expert index out of range) in a status
 * word in mapped host memory; the next call on the handle, flint_moe_route_only
 * (which synchronises) and flint_moe_destroy return it.  No kernel traps.
 */
#ifndef FLINT_MOE_H
#define FLINT_MOE_H

#include <stdint.h>
#include <cuda_runtime_api.h>

#if defined(__GNUC__)
#define FLINT_API __attribute__((visibility("default")))
#else
#define FLINT_API
#endif

#ifdef __cplusplus
extern "C" {
#endif

#define FLINT_HIDDEN 2048      /* H: model width                           */
#define FLINT_INTER 512        /* I: expert intermediate width (routed and shared) */
#define FLINT_EXPERTS 256      /* E: routed experts                        */
#define FLINT_TOPK 6           /* k: routed experts per token              */
#define FLINT_CHUNK 8192       /* tokens per internal chunk of a forward   */
#define FLINT_DECODE_MAX_T 32  /* T <= this takes the weight-streaming path */

typedef struct flint_moe* flint_moe_t;

typedef enum {
    FLINT_BF16 = 0,   /* bf16 expert weights, copied into an owned layout  */
    FLINT_NVFP4 = 1   /* NVFP4 (W4A16) expert weights, repacked and owned   */
} flint_dtype_t;

typedef enum {
    FLINT_OK = 0,
    FLINT_ERR_INVALID_ARG = 1,     /* null / misaligned pointer, bad T, bad dtype     */
    FLINT_ERR_CUDA = 2,            /* a CUDA runtime or driver call failed            */
    FLINT_ERR_OOM = 3,             /* device allocation failed in create              */
    FLINT_ERR_DEVICE_TIMEOUT = 4,  /* a bounded device wait ran out (kernel returned) */
    FLINT_ERR_DEVICE_BADINDEX = 5, /* a kernel saw an expert/token index out of range */
    FLINT_ERR_UNSUPPORTED = 6,     /* no sm_103a device, or an unsupported request    */
    FLINT_ERR_INTERNAL = 7         /* a kernel's internal capacity check failed: a
                                      library defect, not a caller error (the grid
                                      sizes are chosen so that it cannot happen) */
} flint_status_t;

/* One NVFP4 matrix [R][K] (RecursiveSI/flint vLLM recipe page, "Overview":
 * the NVFP4 checkpoint is run as W4A16).  packed[R][K/2]: E2M1 codes, the
 * even column in the low nibble; block_scales[R][K/16]: one E4M3 code per 16
 * consecutive columns; tensor_scale: fp32.  The weight is
 * e2m1(q) * e4m3(s_block) * tensor_scale.  The struct itself lives in host
 * memory; packed and block_scales are device pointers. */
typedef struct {
    const uint8_t* packed;
    const uint8_t* block_scales;
    float tensor_scale;
} flint_nvfp4_t;

/* Build a layer handle on the current device.
 *   out        host: receives the handle.
 *   router_W   bf16 [256][2048].
 *   router_b   fp32 [256] per-expert logit bias, or NULL for none.
 *   gate_up_W  host array of 256 entries, one per routed expert.
 *              FLINT_BF16: device pointer to bf16 [1024][2048], rows 0..511
 *              the gate projection, rows 512..1023 the up projection.
 *              FLINT_NVFP4: host pointer to a flint_nvfp4_t of shape [1024][2048].
 *   down_W     host array of 256 entries: bf16 [2048][512], or flint_nvfp4_t*.
 *   shared_W   host array {gate_up, down} of the shared expert, same rules.
 *   dtype      FLINT_BF16 or FLINT_NVFP4 (the router stays bf16 either way).
 * Ownership: bf16 expert weights are read during create only: the handle
 * owns a copy of every expert matrix cut into 16 KiB tensor-core operand
 * tiles (1.6 GB per layer), which both the decode and the many-token path
 * read, and the caller may free its buffers on return.  While create runs,
 * the caller's bf16 experts and the handle's copy both exist, so the peak
 * device footprint of a layer is twice its expert bytes (3.2 GB) until the
 * caller frees its own buffers.  The router (bf16,
 * both dtypes) is borrowed: it stays alive and unchanged until destroy.  The
 * handle owns a workspace for FLINT_CHUNK tokens (about 310 MB).  NVFP4
 * weights are repacked into a layout the handle owns (1.77 MB per
 * expert, no bf16 copy); the caller may free its buffers on return.
 * Synchronises the device.
 * Errors: INVALID_ARG, OOM, CUDA, UNSUPPORTED (device is not sm_103). */
FLINT_API flint_status_t flint_moe_create(flint_moe_t* out, const void* router_W, const float* router_b,
                                const void* const* gate_up_W, const void* const* down_W,
                                const void* const* shared_W, flint_dtype_t dtype);

/* y = layer(x) for T >= 1 tokens.
 *   x  bf16 [T][2048], y bf16 [T][2048] (fully overwritten); x and y must not
 *   overlap.  Runs asynchronously on stream s; allocates nothing; capturable in
 *   a CUDA graph.  T <= 32 takes the weight-streaming decode kernels
 *   (FLINT_NVFP4: W4A16, the codes dequantised into the MMA fragments), larger
 *   T the grouped tensor-core path in chunks of FLINT_CHUNK tokens
 *   (FLINT_NVFP4: the weight tiles dequantised to bf16 in shared memory).  One
 *   handle serves one stream at a time (the workspace is per handle).
 * Errors: INVALID_ARG (null, misaligned, T < 1), CUDA (launch failed), or a
 * device status left by an earlier call. */
FLINT_API flint_status_t flint_moe_forward(flint_moe_t h, const void* x, int T, void* y, cudaStream_t s);

/* n layers applied in order, y[l] = layer_l(x[l]) for l = 0 .. n-1, with the
 * result of n flint_moe_forward calls on one stream (cross-layer decode; the
 * recipe page's low-latency decode path and the mrchatgpt.org article's decode
 * megakernel, section 4, name the idea).
 *   layers  host array of n handles, all of one dtype, on one device.
 *   x, y    host arrays of n device pointers, bf16 [T][2048] each; x[l] and
 *           y[l] must not overlap.  Layer l reads x[l] only after every
 *           earlier layer has written its y, so x[l + 1] may be y[l] (a
 *           chained stack) or any other buffer.
 *   T       tokens per layer, T >= 1.
 * T <= FLINT_STACK_MAX_T (bf16 or NVFP4 layers): ONE persistent kernel
 * launch per FLINT_STACK_MAX_LAYERS layers (one CTA per SM walks the layers;
 * grid-wide device-scope barriers separate a layer's phases, each wait
 * bounded).  The launch needs every SM of the device: do not run other
 * kernels beside it.  Larger T: n flint_moe_forward calls.
 * Asynchronous on s, allocates nothing, capturable in a CUDA graph.  Scratch:
 * layers[0]'s workspace, so layers[0] must not be used on another stream
 * meanwhile; device errors are reported in layers[0]'s status word.
 * Errors: INVALID_ARG (null, misaligned, overlapping x[l]/y[l], mixed
 * dtypes or devices), CUDA, or a device status left by an earlier call. */
#define FLINT_STACK_MAX_T 8
#define FLINT_STACK_MAX_LAYERS 64
FLINT_API flint_status_t flint_moe_forward_layers(const flint_moe_t* layers, int n, const void* const* x, int T,
                                                  void* const* y, cudaStream_t s);

/* Routing alone, for testing (synchronises s before returning).
 *   x       bf16 [T][2048] or NULL.
 *   logits  fp32 [T][256].  If x is NULL, logits is the INPUT: the router
 *           matrix and bias are skipped and selection runs on these values.
 *           If x is non-NULL, logits may be NULL or receives the router's fp32
 *           logits (bias included).
 *   idx     int32 [T][6] chosen experts, in decreasing logit order (equal
 *           logits: lower index first).
 *   w       fp32 [T][6] renormalised sigmoid weights, same order.
 *   offsets int32 [257] or NULL: offsets[e] = number of (token, slot) pairs
 *           choosing an expert below e; offsets[256] = 6T.
 *   gather_idx int32 [6T] or NULL: pair ids t*6+j grouped by expert, in
 *           increasing pair id within an expert (a stable counting sort).
 *   T       1 <= T <= FLINT_CHUNK.
 * Errors: INVALID_ARG, CUDA, or a device status. */
FLINT_API flint_status_t flint_moe_route_only(flint_moe_t h, const void* x, float* logits, int T,
                                    int32_t* idx, float* w, int32_t* offsets,
                                    int32_t* gather_idx, cudaStream_t s);

/* Synchronise the device, release everything the handle owns and return the
 * last device status.  NULL is accepted (returns FLINT_OK). */
FLINT_API flint_status_t flint_moe_destroy(flint_moe_t h);

/* Kernels of one forward that flint_moe_set_kernel_events can time. */
typedef enum {
    FLINT_KERNEL_ROUTER = 0,   /* router logits (T <= 32) / router GEMM + top-6 (T > 32) */
    FLINT_KERNEL_GATE_UP = 1,  /* expert gate/up projections + SwiGLU                  */
    FLINT_KERNEL_DOWN = 2,     /* expert down projections (T <= 32: with the combine)  */
    FLINT_KERNEL_COMBINE = 3   /* weighted combine (T > 32 only)                       */
} flint_kernel_t;

/* Profiling hook: while set, every flint_moe_forward on h records `start`
 * on its stream immediately before launching the kernel `kernel`
 * (a flint_kernel_t) and `stop` immediately after it, so that
 * cudaEventElapsedTime(start, stop) is that kernel's duration (for a forward
 * of several FLINT_CHUNK chunks: the last chunk's).  The events (created by
 * the caller, timing enabled) must outlive the setting.  An event recorded
 * between two kernels removes their programmatic-launch overlap, so a hooked
 * forward is slower than an unhooked one: for measurement only.  Not for
 * use during stream capture (the records would not become graph nodes).
 * kernel = -1 clears the hook (events may then be NULL).
 * Errors: INVALID_ARG (null handle, unknown kernel, null event). */
FLINT_API flint_status_t flint_moe_set_kernel_events(flint_moe_t h, int kernel, cudaEvent_t start,
                                                     cudaEvent_t stop);

/* Human-readable name of a status code (static storage). */
FLINT_API const char* flint_status_string(flint_status_t st);

/* The expert permutation of flint_moe_route_only (offsets and gather_idx,
 * same definitions and results) computed from a given routing, without a
 * layer handle and without allocating any device memory.  The pages define
 * no such call: it exists for callers that must not allocate at routing time
 * (allocator-free serving loops, external memory pools).
 *   idx        int32 [T][6] expert ids in 0..255 (device).
 *   offsets    int32 [257] (device), as in flint_moe_route_only.
 *   gather_idx int32 [6T] (device), as in flint_moe_route_only.
 *   T          1 <= T <= FLINT_CHUNK; a larger T is rejected with
 *              FLINT_ERR_INVALID_ARG, because the scratch is a fixed device
 *              array sized for FLINT_CHUNK tokens (327,936 bytes).
 * The scratch is one array per device shared by every call: calls that
 * overlap in time (two streams, two host threads) race on it and must be
 * serialised by the caller.  The first call on a device looks up the array's
 * address on that device (cudaGetSymbolAddress).  Every call ends by
 * reading the scratch's status word back to the host and synchronising s.
 * Errors: INVALID_ARG, CUDA, DEVICE_BADINDEX (an id in idx outside 0..255;
 * outputs are then unspecified). */
FLINT_API flint_status_t flint_permute_static(const int32_t* idx, int T, int32_t* offsets,
                                              int32_t* gather_idx, cudaStream_t s);

/* ---- 4-bit output layer --------------------------------------------------
 * The pages report that Flint's output layer (lm_head) was quantised to 4
 * bits as well and is run from the NVFP4 checkpoint (mrchatgpt.org article,
 * section 4, the quantisation item; qantcore.space review, section 04, the
 * quantised variants).  The vocabulary size V is not on the pages: any
 * positive multiple of 16 is accepted.  A decode step's logits are
 *   logits[t][v] = sum_h x[t][h] * W[v][h],  W[v][h] = e2m1 * e4m3 * s_tensor,
 * computed by one weight-streaming kernel (W read once per call). */
typedef struct flint_lm_head* flint_lm_head_t;
#define FLINT_LM_HEAD_MAX_T 32

/* Build an output-layer handle on the current device.
 *   out  host: receives the handle (NULL on failure).
 *   W    host pointer to a flint_nvfp4_t of shape [V][2048] (device data).
 *   V    rows of W, a positive multiple of 16.
 * The handle repacks W into memory it owns (V x 1152 bytes) and keeps no
 * reference to W's buffers: the caller may free them on return.
 * Errors: INVALID_ARG (null pointer, V not a positive multiple of 16),
 * UNSUPPORTED (no sm_103 device), OOM, CUDA. */
FLINT_API flint_status_t flint_lm_head_create(flint_lm_head_t* out, const flint_nvfp4_t* W, int V);

/* Logits of T tokens, enqueued on stream s (asynchronous).
 *   x       bf16 [T][2048], device, 16-byte aligned.
 *   T       1 <= T <= FLINT_LM_HEAD_MAX_T.
 *   logits  fp32 [T][V], device, 16-byte aligned, fully overwritten; must not
 *           overlap x.
 * Errors: INVALID_ARG, CUDA; DEVICE_TIMEOUT when an earlier call's bounded
 * wait gave up (its outputs are then unspecified; the error is reported
 * once, by the next call on the handle or by destroy). */
FLINT_API flint_status_t flint_lm_head_forward(flint_lm_head_t h, const void* x, int T, float* logits,
                                               cudaStream_t s);

/* Synchronise the device, release the handle and report a pending device
 * status.  NULL is a no-op. */
FLINT_API flint_status_t flint_lm_head_destroy(flint_lm_head_t h);

/* Test hook: launch one kernel that waits on a device flag nothing sets,
 * with a wait limit of timeout_ns nanoseconds of %globaltimer; returns
 * FLINT_ERR_DEVICE_TIMEOUT when the bounded wait gives up as designed.
 * Synchronises s. */
FLINT_API flint_status_t flint_debug_bounded_wait(uint64_t timeout_ns, cudaStream_t s);

#ifdef __cplusplus
}
#endif

#endif /* FLINT_MOE_H */
