// q4moe_noalloc.cu -- q4moe_gate_up_swiglu_noalloc: the fused call for
// callers that cannot allocate device memory.
//
// The fast tensor-core path wants scratch memory (the routed activations
// copied once into grouped order, which the GEMM then reads through TMA).
// q4moe_gate_up_swiglu_ex takes that scratch from the caller; some callers
// have none to give -- a plugin running inside a host engine that owns every
// byte of GPU memory through its own pool, code held to a fixed memory
// budget, or a latency-critical decode loop that must never risk the device
// synchronisation an allocation can cause.  For them this entry point uses a
// fixed scratch array that lives in the library itself: a file-scope
// __device__ array, which exists once on every GPU that loads the library
// and stays there until the process exits.  Nothing here calls cudaMalloc,
// cudaFree or any allocating routine.
#include <climits>
#include <cstdio>
#include <mutex>

#include "q4moe_internal.cuh"

namespace {

// The scratch: bf16 grouped activations [M][H], at most
// Q4MOE_NOALLOC_SCRATCH_BYTES.  Host code must not use the name as an
// address (it is only a host-side stand-in for the device symbol); the
// device address comes from cudaGetSymbolAddress below.
static __device__ __align__(256) unsigned char
    g_noalloc_scratch[Q4MOE_NOALLOC_SCRATCH_BYTES];

constexpr int kMaxDevices = 64;
void *g_scratch_ptr[kMaxDevices];
std::mutex g_scratch_mutex;

// Device address of the scratch on the current device, looked up once per
// device (the first call on each device does it).
int scratch_address(void **out) {
    int dev = 0;
    cudaError_t err = cudaGetDevice(&dev);
    if (err != cudaSuccess)
        return q4moe::report_error(Q4MOE_ERR_CUDA, "cudaGetDevice failed");
    if (dev < 0 || dev >= kMaxDevices)
        return q4moe::report_error(Q4MOE_ERR_DEVICE,
                                   "device ordinal out of range");
    std::lock_guard<std::mutex> lock(g_scratch_mutex);
    if (g_scratch_ptr[dev] == nullptr) {
        void *p = nullptr;
        err = cudaGetSymbolAddress(&p, g_noalloc_scratch);
        if (err != cudaSuccess || p == nullptr) {
            char msg[160];
            snprintf(msg, sizeof msg,
                     "cudaGetSymbolAddress(scratch) failed: %s",
                     cudaGetErrorString(err));
            return q4moe::report_error(Q4MOE_ERR_CUDA, msg);
        }
        g_scratch_ptr[dev] = p;
    }
    *out = g_scratch_ptr[dev];
    return Q4MOE_OK;
}

}  // namespace

extern "C" int q4moe_gate_up_swiglu_noalloc(
    const void *x, const q4moe_slabs_t *expert_slabs,
    const int32_t *row_offsets_per_expert, const int32_t *token_to_expert_map,
    int64_t M, int64_t H, int64_t I, void *out, cudaStream_t stream) {
    if (M < 0 || H < 0)
        return q4moe::report_error(Q4MOE_ERR_INVALID_ARG,
                                   "M and H must be non-negative");
    // bound M and H before forming M * H * 2 (no int64 overflow): beyond
    // these the scratch could never hold the rows anyway
    if (M > INT32_MAX || H > (INT64_C(1) << 24) ||
        (M > 0 && M * H > (INT64_C(1) << 40)))
        return q4moe::report_error(
            Q4MOE_ERR_INVALID_ARG,
            "q4moe_gate_up_swiglu_noalloc: M * H exceeds the library's "
            "fixed scratch");
    const int64_t need = q4moe_workspace_bytes(M, H);
    if (need > (int64_t)Q4MOE_NOALLOC_SCRATCH_BYTES) {
        char msg[200];
        snprintf(msg, sizeof msg,
                 "q4moe_gate_up_swiglu_noalloc: M*H*2 = %lld bytes exceeds "
                 "the library's fixed scratch of %lld bytes; use "
                 "q4moe_gate_up_swiglu_ex with a workspace",
                 (long long)need, (long long)Q4MOE_NOALLOC_SCRATCH_BYTES);
        return q4moe::report_error(Q4MOE_ERR_INVALID_ARG, msg);
    }
    void *scratch = nullptr;
    const int rc = scratch_address(&scratch);
    if (rc != Q4MOE_OK)
        return rc;
    q4moe_options_t opts{};
    opts.workspace = scratch;
    opts.workspace_bytes = (int64_t)Q4MOE_NOALLOC_SCRATCH_BYTES;
    return q4moe_gate_up_swiglu_ex(x, expert_slabs, row_offsets_per_expert,
                                   token_to_expert_map, M, H, I, out, &opts,
                                   stream);
}
