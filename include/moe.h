/*
 * moe.h — C ABI of libmoe.so: one top-k Mixture-of-Experts layer on one GB300
 * (sm_103a).
 *
 * The layer. Every decoder layer of Muse Spark is a Mixture-of-Experts layer
 * in which each token picks 8 of 256 experts ("How SGLang-TorchTPU
 * accelerated an 816B-parameter MoE on TPU v7", section "Introduction");
 * per-expert outputs are combined after the experts run ("TensorSharp Muse
 * Spark benchmark", section "Performance"); partial sums of expert outputs
 * are kept in fp32 because bf16 partial sums cost quality (same page, section
 * "Answer quality"). The pages leave the gate and FFN open; this library
 * computes, per token t with bf16 input x[t, 0:d]:
 *
 *   logit[e] = sum_c x[c] * Wr[e, c]  (fp32 accumulate) + bias[e]
 *   p        = softmax(logit) over all E experts (fp32)
 *   ids[0:k] = the k largest p, ties to the lower expert id, by descending p
 *   w[j]     = p[ids[j]] / sum_j' p[ids[j']]
 *   h_j      = silu(Wg[ids[j]] x) * (Wu[ids[j]] x)
 *   y        = sum_j w[j] * (Wd[ids[j]] h_j)   (fp32, j ascending) -> bf16
 *
 * Conventions for every call:
 *  - Pointers named *_host are host memory; every other pointer is device
 *    memory owned by the caller, 16-byte aligned, and must stay valid for as
 *    long as the layer or the enqueued work uses it. The library allocates no
 *    device memory: scratch lives in the caller's workspace.
 *  - `stream` is a cudaStream_t passed as void* (NULL: the legacy default
 *    stream). All device work is enqueued on it, in order; calls return
 *    without waiting for the GPU unless stated otherwise.
 *  - bf16 tensors are raw bf16 bits, row-major, innermost index last.
 *  - Argument errors are detected on the host before any work is enqueued
 *    (MOE_ERR_INVALID_ARG / MOE_ERR_UNSUPPORTED); launch failures return
 *    MOE_ERR_CUDA; conditions detected by a kernel (a bounded wait that ran
 *    out, an index out of range) set an error word in the workspace that
 *    moe_get_device_status() reports.
 *  - A layer object is not thread-safe; distinct layers may be used from
 *    distinct threads. Two calls on one layer must not overlap on the GPU
 *    (they share the workspace): issue them on one stream.
 */
#ifndef MOE_H_
#define MOE_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
    MOE_OK = 0,
    MOE_ERR_INVALID_ARG = 1,  /* null pointer, misaligned pointer, T out of range */
    MOE_ERR_UNSUPPORTED = 2,  /* shape or format this library does not implement */
    MOE_ERR_CUDA = 3,         /* a CUDA runtime call or launch failed */
    MOE_ERR_DEVICE = 4,       /* a kernel flagged an out-of-range index */
    MOE_ERR_TIMEOUT = 5       /* a kernel's bounded wait ran out */
} moe_status;

/* Expert weight format. NVFP4 ("How SGLang-TorchTPU accelerated an
 * 816B-parameter MoE on TPU v7", section "Results and interpretation", runs
 * experts as NVFP4 weights): 16-element blocks along the contraction index,
 * each element an E2M1 code, each block one E4M3 scale, each tensor (one
 * matrix of one expert) one fp32 scale: w = e2m1 * e4m3 * s_tensor. */
typedef enum { MOE_W_BF16 = 0, MOE_W_NVFP4 = 1 } moe_wfmt;

typedef struct moe_layer moe_layer;

/* Layer description. Shapes: E experts, hidden size d, expert width I, k
 * experts per token, at most max_tokens tokens per call.
 * Supported: 1 <= k <= 8, k <= E <= 256, d and I multiples of 64, d <= 8192,
 * I <= 4096, 1 <= max_tokens <= 65536. */
typedef struct {
    int d, E, top_k, I, max_tokens;
    moe_wfmt fmt;
    const void *w_router;     /* [E, d] bf16 */
    const float *router_bias; /* [E] fp32, or NULL for no bias */
    /* MOE_W_BF16 experts (NULL otherwise) */
    const void *w_gate;       /* [E, I, d] bf16 */
    const void *w_up;         /* [E, I, d] bf16 */
    const void *w_down;       /* [E, d, I] bf16 */
    /* MOE_W_NVFP4 experts (NULL otherwise). Two E2M1 codes per byte, the low
     * nibble holding the lower contraction index; E4M3 scales one per 16. */
    const uint8_t *q_gate, *q_up; /* [E, I, d/2] */
    const uint8_t *q_down;        /* [E, d, I/2] */
    const uint8_t *s_gate, *s_up; /* [E, I, d/16] */
    const uint8_t *s_down;        /* [E, d, I/16] */
    const float *g_gate, *g_up, *g_down; /* [E] per-tensor fp32 scales */
    /* 0: the plain weighted sum. 1: each expert's output is RMS-normalised
     * (Y / sqrt(mean(Y^2) + 1e-6), no learned scale) before the weighted sum,
     * a reading of "Muse Spark normalises each expert's output, then combines"
     * ("TensorSharp Muse Spark benchmark", section "Performance"). */
    int expert_out_norm;
    /* bf16 experts only. 0: w_gate and w_up are separate [E, I, d] tensors.
     * 1: w_gate points to one [E, I, 2, d] tensor holding gate row i then up
     * row i of each expert (the fused gate/up projection, interleaved by row)
     * and w_up is ignored; the small-batch kernels then fetch a row pair as one
     * contiguous copy. */
    int gate_up_interleaved;
} moe_layer_desc;

/* Bytes of device workspace the layer needs (for max_tokens). No GPU work. */
moe_status moe_workspace_size(const moe_layer_desc *desc, size_t *bytes);

/* Create a layer over caller-owned weights and workspace (ws_bytes at least
 * moe_workspace_size; 256-byte aligned). Zeroes the workspace's control words
 * with a synchronous cudaMemset on the current device; *out receives a
 * host-side handle freed by moe_layer_destroy. */
moe_status moe_layer_create(const moe_layer_desc *desc, void *workspace, size_t ws_bytes,
                            moe_layer **out);

/* Routing and token permutation only (router, softmax, top-k, renormalise,
 * then the permutation). x [T, d] bf16. Outputs (device):
 *   ids [T, k] int32 (descending weight), w [T, k] fp32 (sums to 1 per token),
 *   counts [E] int32, offsets [E+1] int32 (exclusive prefix sum of counts),
 *   perm [T*k] int32: perm[offsets[e] + r] = the r-th smallest token id routed
 *   to expert e, pos [T, k] int32: the row of (t, j) in that order.
 * Any output pointer may be NULL to skip it. 1 <= T <= max_tokens. */
moe_status moe_route(moe_layer *layer, const void *x, int T, int32_t *ids, float *w,
                     int32_t *counts, int32_t *offsets, int32_t *perm, int32_t *pos,
                     void *stream);

/* Layer forward: out [T, d] bf16 = MoE(x). out must not alias x. */
moe_status moe_forward(moe_layer *layer, const void *x, void *out, int T, void *stream);

/* out = bf16(res + MoE(x)) with the residual added in fp32. out may alias res
 * but not x. Used between stacked layers (pre-norm residual block). */
moe_status moe_forward_residual(moe_layer *layer, const void *x, const void *res, void *out,
                                int T, void *stream);

/* End-to-end forward from host memory: copies x_host [T, d] bf16 into the
 * workspace, runs moe_forward, copies the result to out_host [T, d] bf16 and
 * waits for the stream. Page-locked host buffers give asynchronous copies. */
moe_status moe_forward_host(moe_layer *layer, const void *x_host, void *out_host, int T,
                            void *stream);

/* Expert outputs of the last forward on this layer, before the weighted sum:
 * Y [T*k, d] fp32, row pos[t, j] holding expert ids[t, j] applied to token t
 * (pos from moe_route on the same x). For parity checks of every slot. After
 * a large-batch forward the outputs were kept in bf16 (the grouped GEMMs'
 * output precision) and are widened to fp32 here. */
moe_status moe_debug_expert_outputs(moe_layer *layer, float *Y, int T, void *stream);

/* Small-batch (T <= 16) kernel choice. Both compute the same layer in one
 * persistent launch; they differ in where the expert FFNs run:
 *   MOE_DECODE_CUDA_CORES: each weight row is multiplied by the tokens on the
 *     CUDA cores as it streams in (suits one token with bf16 weights, where
 *     the stream alone sets the pace);
 *   MOE_DECODE_TENSOR_CORES: 128 weight rows at a time are the M operand of
 *     tcgen05.mma and the tokens the N = 16 operand, NVFP4 codes widened into
 *     tensor memory on the way (suits several tokens or NVFP4 weights);
 *   MOE_DECODE_AUTO (default): the tensor cores for bf16 experts and 8 or
 *     more tokens, else the CUDA cores.
 * The tensor-core kernel needs d % 128 == 0 and no expert_out_norm; where a
 * layer does not meet that, the CUDA-core kernel runs whatever the choice.
 * Stacks follow the choice of their first layer. */
enum { MOE_DECODE_AUTO = 0, MOE_DECODE_CUDA_CORES = 1, MOE_DECODE_TENSOR_CORES = 2 };
moe_status moe_set_decode_path(moe_layer *layer, int path);

/* Routing records of the last forward or route on this layer, as the
 * kernels left them in the workspace (no recomputation): the fields of
 * moe_route, same layouts; any output pointer may be NULL. A forward of
 * T <= 16 tokens leaves the records its single decode launch computed and
 * published; a larger forward leaves those of the large-batch routing
 * kernels, or, where it runs in chunks of 16 tokens, those of its last
 * chunk. T must be the last call's token count. For parity checks of the
 * routing each forward path uses. */
moe_status moe_debug_route_records(moe_layer *layer, int T, int32_t *ids, float *w, int32_t *counts,
                                   int32_t *offsets, int32_t *perm, int32_t *pos, void *stream);

/* Test hook for the device-side failure detection. While hold != 0, every
 * cross-CTA wait of this layer's single-launch decode kernels (T <= 16, and
 * moe_stack_forward on a stack whose first layer is this one) waits for
 * something that never comes: a grid barrier for one arrival more than the
 * grid provides, the hand-off of the router's logits for a tag no CTA
 * writes. Its bounded wait (1.5 s) runs out:
 * the launch unwinds without computing the experts, leaves `out` undefined
 * and sets the timeout bit that moe_get_device_status() reports as
 * MOE_ERR_TIMEOUT. hold = 0 restores normal operation; the next call runs
 * normally (the launch that gave up resets its counters on exit). Enqueued on
 * `stream` (one 4-byte host-to-device copy). */
moe_status moe_debug_hold_grid_barrier(moe_layer *layer, int hold, void *stream);

/* Row-wise RMSNorm without a learned scale: out = x / sqrt(mean(x^2) + eps),
 * x and out [T, d] bf16 (out may alias x), fp32 arithmetic. */
moe_status moe_rmsnorm(const void *x, void *out, int T, int d, float eps, void *stream);

/* NVFP4 quantiser for n tensors of shape [rows, K] (bf16, contiguous):
 *   s_t = amax|W| / (6*448) (1 for an all-zero tensor),
 *   block scale = E4M3((amax_block / 6) / s_t), code = E2M1(w / (scale * s_t)),
 * round-to-nearest-even, saturating. Outputs q [n, rows, K/2], s [n, rows, K/16],
 * g [n] fp32 (g is also used as the amax accumulator). K multiple of 32. */
moe_status moe_quantize_nvfp4(const void *W, int n, int rows, int K, uint8_t *q, uint8_t *s,
                              float *g, void *stream);

/* Waits for `stream`, then reads and clears the layer's device error word:
 * MOE_OK, MOE_ERR_DEVICE or MOE_ERR_TIMEOUT. */
moe_status moe_get_device_status(moe_layer *layer, void *stream);

/* Number of kernel launches the last forward/route on this layer enqueued. */
int moe_last_launch_count(const moe_layer *layer);

/* Per-kernel timing for measurement. After moe_profile_begin(layer, n), each
 * of the next n forwards on the layer also records a CUDA event on its stream
 * before each of its kernels and one after the last (host-side event objects;
 * no device memory). moe_profile_end waits for those events and writes
 * ms[f * max_kernels + i] = duration of kernel i of recorded forward f, and
 * the counts, then stops recording. */
moe_status moe_profile_begin(moe_layer *layer, int max_forwards);
moe_status moe_profile_end(moe_layer *layer, float *ms_host, int max_kernels, int *n_forwards,
                           int *n_kernels);

/* The pages have no counterpart to this call; it serves callers that cannot
 * allocate device memory (a plugin inside an inference server or engine that
 * owns all device memory and hands it only input and output buffers, or a
 * real-time loop that forbids allocation after start-up).
 *
 * Same result as moe_forward on the CUDA-core small-batch kernel
 * (MOE_DECODE_CUDA_CORES) for 1 <= T <= 16 tokens, with no layer object
 * and no workspace: the scratch lives in one static device array of
 * MOE_STATIC_SCRATCH_BYTES that every GPU which loads libmoe.so holds until
 * the process exits. The call allocates nothing (no cudaMalloc, no
 * allocating library routine). desc is read on the host during the call only;
 * its max_tokens is ignored (the shape is checked as if it were T). x [T, d]
 * and out [T, d] are bf16 device buffers of the caller.
 * - Every call, with the caller's device and context current, looks up the
 *   array's device address in that context (cudaGetSymbolAddress; nothing is
 *   cached, so a new context after cudaDeviceReset, or a context of the
 *   caller's own on the same device, gets its own copy of the array). The
 *   first call in a process may load the library's device code: make it
 *   before any stream capture.
 * - Every call shares the one array and clears its control words at the start
 *   (an async memset on `stream`): calls that overlap on the GPU race, so
 *   issue them on one stream or otherwise order them.
 * - Shapes whose scratch exceeds MOE_STATIC_SCRATCH_BYTES, or whose tokens do
 *   not fit in shared memory beside the weight ring, return
 *   MOE_ERR_UNSUPPORTED; T outside [1, 16] returns MOE_ERR_INVALID_ARG; both
 *   before any GPU work.
 * - Device-side error bits (a bounded wait that ran out) are not reported:
 *   the next call clears them. After such an event `out` is undefined; a
 *   caller that needs the check uses moe_forward and moe_get_device_status. */
#define MOE_STATIC_SCRATCH_BYTES (8u << 20)
moe_status moe_forward_static_scratch(const moe_layer_desc *desc, const void *x, void *out, int T,
                                      void *stream);

/* Stacked layers in one launch (the persistent multi-layer decode kernel
 * the pages' megakernel idea suggests, "How SGLang-TorchTPU accelerated an
 * 816B-parameter MoE on TPU v7", section "Key optimisations"). For
 * l = 0 .. n_layers-1:
 *     x_{l+1} = x_l + MoE_l(RMSNorm(x_l)),   x_0 = x,   out = x_n,
 * RMSNorm without a gain, eps as given, its output rounded to bf16 (the
 * arithmetic of moe_rmsnorm), the sum rounded to bf16 (moe_forward_residual).
 * - moe_stack_create: 1 <= n_layers <= 64 layers of equal d, E, top_k, I and
 *   weight format, without expert_out_norm, whose max_tokens >= 1. It writes
 *   the layers' weight pointers (not the weights) into layers[0]'s workspace
 *   once (a synchronous copy); the stack then runs on that workspace, so the
 *   stack and layers[0] must not run at the same time. The layers must
 *   outlive the stack.
 * - moe_stack_forward: T in [1, 8] and <= layers[0]'s max_tokens; x, out bf16
 *   [T, d] device buffers (out may alias x). layer_out, if not NULL, receives
 *   every layer's output, [n_layers, T, d] bf16. One launch, no host sync.
 *   Errors as for moe_forward. */
typedef struct moe_stack moe_stack;
moe_status moe_stack_create(moe_layer *const *layers, int n_layers, moe_stack **out);
moe_status moe_stack_forward(moe_stack *stack, const void *x, void *out, int T, float eps, void *layer_out,
                             void *stream);
/* End-to-end stack forward from host memory: copies x_host [T, d] bf16 into
 * layers[0]'s workspace, runs moe_stack_forward, copies the result to
 * out_host [T, d] bf16 and waits for the stream. Page-locked host buffers
 * give asynchronous copies. */
moe_status moe_stack_forward_host(moe_stack *stack, const void *x_host, void *out_host, int T, float eps,
                                  void *stream);
moe_status moe_stack_destroy(moe_stack *stack);

moe_status moe_layer_destroy(moe_layer *layer);

const char *moe_status_string(moe_status s);

#ifdef __cplusplus
}
#endif

#endif /* MOE_H_ */
