// static_scratch.cu — the decode forward for callers that cannot allocate
// device memory.
//
// Some callers cannot call cudaMalloc: a plugin inside a host application
// (an inference server or engine) that owns all device memory and hands the
// plugin only its input and output buffers, or a real-time loop in which
// allocating after start-up is forbidden. moe_forward_static_scratch() gives
// them the small-batch layer forward (T <= 16) without a caller workspace:
// its scratch (routing records, h, expert outputs, control words) lives in
// the file-scope device array below, which every GPU that loads this library
// holds until the process exits.
#include <cuda_runtime.h>
#include <stdint.h>

#include "common.cuh"

namespace {

using namespace moe;

// Scratch of the static-scratch forward, shared by every call on a device.
static __device__ __align__(256) unsigned char g_static_scratch[MOE_STATIC_SCRATCH_BYTES];

bool aligned16(const void *p) { return ((uintptr_t)p & 15u) == 0; }

// Set-up, done on every call with the caller's device and context current:
// the host-side name g_static_scratch is only a stand-in, so the kernel gets
// the array's device address in the current context (a lookup, no
// allocation). Nothing is cached, so a context created later (after
// cudaDeviceReset, or the caller's own context on the same device) gets its
// own module's address, and concurrent host threads share no state.
moe_status device_setup(void **scratch, int *num_sms) {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return MOE_ERR_CUDA;
    void *ptr = nullptr;
    if (cudaGetSymbolAddress(&ptr, g_static_scratch) != cudaSuccess || !ptr) return MOE_ERR_CUDA;
    int sms = 0;
    if (cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || sms < 1)
        return MOE_ERR_CUDA;
    *scratch = ptr;
    *num_sms = sms;
    return MOE_OK;
}

}  // namespace

extern "C" moe_status moe_forward_static_scratch(const moe_layer_desc *desc, const void *x, void *out, int T,
                                                 void *stream) {
    if (!desc) return MOE_ERR_INVALID_ARG;
    // the shape checks of a layer sized for exactly T tokens (desc->max_tokens
    // is not used); no GPU work
    moe_layer_desc shape = *desc;
    shape.max_tokens = T < 1 ? 1 : T;
    size_t ignore = 0;
    moe_status s = moe_workspace_size(&shape, &ignore);
    if (s != MOE_OK) return s;
    if (!x || !out || !aligned16(x) || !aligned16(out) || x == out || T < 1 || T > 16 || !desc->w_router ||
        !aligned16(desc->w_router))
        return MOE_ERR_INVALID_ARG;
    if (desc->fmt == MOE_W_BF16) {
        const void *wu = desc->gate_up_interleaved ? desc->w_gate : desc->w_up;
        if (!desc->w_gate || !wu || !desc->w_down || !aligned16(desc->w_gate) || !aligned16(wu) ||
            !aligned16(desc->w_down))
            return MOE_ERR_INVALID_ARG;
    } else {
        const void *p[] = {desc->q_gate, desc->q_up, desc->q_down, desc->s_gate, desc->s_up,
                           desc->s_down, desc->g_gate, desc->g_up,  desc->g_down};
        for (const void *q : p)
            if (!q || !aligned16(q)) return MOE_ERR_INVALID_ARG;
    }
    const Workspace need = workspace_layout(nullptr, desc->d, desc->E, desc->top_k, desc->I, T);
    if (need.bytes > MOE_STATIC_SCRATCH_BYTES) return MOE_ERR_UNSUPPORTED;
    // the tokens' rows sit in shared memory next to a ring of at least two stages
    if ((size_t)T * desc->d * 2 + 2 * (4 * (size_t)desc->d * 2) + 4096 > 227 * 1024) return MOE_ERR_UNSUPPORTED;

    void *scratch = nullptr;
    int num_sms = 0;
    s = device_setup(&scratch, &num_sms);
    if (s != MOE_OK) return s;

    LayerDev L{};
    L.d = desc->d;
    L.E = desc->E;
    L.k = desc->top_k;
    L.I = desc->I;
    L.max_T = T;
    L.fmt = desc->fmt;
    L.wr = (const uint16_t *)desc->w_router;
    L.bias = desc->router_bias;
    L.wg = (const uint16_t *)desc->w_gate;
    L.wu = desc->gate_up_interleaved ? L.wg + desc->d : (const uint16_t *)desc->w_up;
    L.gu_ld = desc->gate_up_interleaved ? 2 * (int64_t)desc->d : desc->d;
    L.wd = (const uint16_t *)desc->w_down;
    L.qg = desc->q_gate;
    L.qu = desc->q_up;
    L.qd = desc->q_down;
    L.sg = desc->s_gate;
    L.su = desc->s_up;
    L.sd = desc->s_down;
    L.gg = desc->g_gate;
    L.gu = desc->g_up;
    L.gd = desc->g_down;
    L.num_sms = num_sms;
    L.expert_norm = desc->expert_out_norm ? 1 : 0;
    const Workspace ws = workspace_layout(scratch, L.d, L.E, L.k, L.I, T);

    cudaStream_t st = (cudaStream_t)stream;
    // the array keeps the previous call's contents: the control words (error
    // bits, counters, the logits' epoch) and the tagged logits start at zero
    // (with the epoch back at 0, a tag left by an earlier call could match)
    if (cudaMemsetAsync(ws.ctrl, 0, control_bytes(ws, L.E), st) != cudaSuccess) return MOE_ERR_CUDA;
    // the same single-launch layer kernel moe_forward runs for T <= 16
    const cudaError_t e = launch_decode_fused(L, ws, (const uint16_t *)x, nullptr, (uint16_t *)out, T, st);
    return e == cudaSuccess ? MOE_OK : MOE_ERR_CUDA;
}
