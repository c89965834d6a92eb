// q4moe_group.cu -- token -> expert grouping (a stable counting sort of the
// routed (token, slot) pairs by expert id), run by one thread block.
//
// The pages hand each expert slot its own [M, H] row block (page 52,
// streamed-experts.ts, Glm52CanonicalMetalExecutor.execute); this kernel
// builds those row lists for every expert in one pass:
//   1. histogram of expert ids in shared memory;
//   2. exclusive scan -> row_offsets;
//   3. pairs taken 1024 at a time in order; within a chunk each pair's rank
//      among equal ids is (pairs of that id in earlier warps) + (earlier
//      lanes of its own warp with that id, from __match_any_sync), so rows
//      of one expert keep the token order.
#include "q4moe_internal.cuh"

namespace q4moe {
namespace {

constexpr int kThreads = 1024;
constexpr int kWarps = kThreads / 32;

__global__ void __launch_bounds__(kThreads, 1)
group_rows_kernel(const int32_t *__restrict__ topk, int32_t pairs, int32_t k,
                  int32_t E, int32_t *__restrict__ row_offsets,
                  int32_t *__restrict__ token_of_row,
                  int32_t *__restrict__ row_of_pair,
                  unsigned int *__restrict__ status) {
    extern __shared__ int32_t smem[];
    int32_t *s_base = smem;             // [E]   next free row of expert e
    int32_t *s_warp = smem + E;         // [kWarps][E] per-warp counts/bases
    __shared__ int32_t s_warp_sums[kWarps];
    __shared__ int s_bad;

    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    for (int e = tid; e < E; e += kThreads)
        s_base[e] = 0;
    if (tid == 0)
        s_bad = 0;
    __syncthreads();

    // 1. histogram
    for (int32_t q = tid; q < pairs; q += kThreads) {
        const int32_t e = topk[q];
        if (e >= 0 && e < E)
            atomicAdd(&s_base[e], 1);
        else
            s_bad = 1;
    }
    __syncthreads();

    // 2. exclusive scan over E <= kThreads counts (one per thread)
    const int32_t c = tid < E ? s_base[tid] : 0;
    int32_t incl = c;
#pragma unroll
    for (int d = 1; d < 32; d <<= 1) {
        const int32_t v = __shfl_up_sync(0xffffffffu, incl, d);
        if (lane >= d)
            incl += v;
    }
    if (lane == 31)
        s_warp_sums[warp] = incl;
    __syncthreads();
    if (warp == 0) {
        int32_t w = s_warp_sums[lane];
        int32_t wi = w;
#pragma unroll
        for (int d = 1; d < 32; d <<= 1) {
            const int32_t v = __shfl_up_sync(0xffffffffu, wi, d);
            if (lane >= d)
                wi += v;
        }
        s_warp_sums[lane] = wi - w;  // exclusive prefix of warp totals
    }
    __syncthreads();
    const int32_t excl = s_warp_sums[warp] + incl - c;
    if (tid < E) {
        s_base[tid] = excl;
        row_offsets[tid] = excl;
    }
    if (tid == E - 1 || (E == 0 && tid == 0))
        row_offsets[E] = excl + c;
    if (tid == 0 && s_bad)
        atomicOr(status, Q4MOE_DEV_BAD_EXPERT_ID);
    __syncthreads();

    // 3. stable scatter, one chunk of kThreads pairs at a time
    const unsigned lt_mask = (1u << lane) - 1u;
    for (int32_t c0 = 0; c0 < pairs; c0 += kThreads) {
        for (int j = tid; j < kWarps * E; j += kThreads)
            s_warp[j] = 0;
        __syncthreads();
        const int32_t q = c0 + tid;
        int32_t e = -1;
        if (q < pairs) {
            e = topk[q];
            if (e < 0 || e >= E)
                e = -1;
        }
        const unsigned peers = __match_any_sync(0xffffffffu, e);
        const int rank = __popc(peers & lt_mask);
        if (e >= 0 && rank == 0)
            s_warp[warp * E + e] = __popc(peers);
        __syncthreads();
        for (int ee = tid; ee < E; ee += kThreads) {
            int32_t run = s_base[ee];
            for (int w = 0; w < kWarps; ++w) {
                const int32_t n = s_warp[w * E + ee];
                s_warp[w * E + ee] = run;
                run += n;
            }
            s_base[ee] = run;
        }
        __syncthreads();
        if (q < pairs) {
            if (e >= 0) {
                const int32_t row = s_warp[warp * E + e] + rank;
                token_of_row[row] = q / k;
                row_of_pair[q] = row;
            } else {
                row_of_pair[q] = -1;
            }
        }
        __syncthreads();
    }
}

}  // namespace

cudaError_t launch_group_rows(const int32_t *topk, int64_t pairs, int32_t k,
                              int32_t E, int32_t *row_offsets,
                              int32_t *token_of_row, int32_t *row_of_pair,
                              unsigned int *status, cudaStream_t s) {
    const size_t smem = sizeof(int32_t) * (size_t)E * (1 + kWarps);
    cudaError_t err = cudaFuncSetAttribute(
        group_rows_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
        (int)smem);
    if (err != cudaSuccess)
        return err;
    group_rows_kernel<<<1, kThreads, smem, s>>>(
        topk, (int32_t)pairs, k, E, row_offsets, token_of_row, row_of_pair,
        status);
    count_launches(1);
    return cudaGetLastError();
}

}  // namespace q4moe
