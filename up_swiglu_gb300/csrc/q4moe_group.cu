// q4moe_group.cu -- token -> expert grouping (a stable counting sort of the
// routed (token, slot) pairs by expert id), run by one thread block.
//
// The pages hand each expert slot its own [M, H] row block (page 52,
// streamed-experts.ts, Glm52CanonicalMetalExecutor.execute); this kernel
// builds those row lists for every expert in one pass over the pairs:
//   1. each warp owns one contiguous segment of the pairs and counts its
//      experts 32 pairs at a time (__match_any_sync groups equal ids; the
//      lowest lane of a group adds the group's size);
//   2. per expert, an exclusive scan over the warps, then over the experts,
//      turns the counts into each warp's first row for that expert and into
//      row_offsets;
//   3. each warp walks its segment again, giving a pair the row
//      base + (earlier lanes with the same id); segments are in pair order,
//      so rows of one expert keep the token order.
#include <algorithm>

#include "q4moe_internal.cuh"

namespace q4moe {
namespace {

constexpr int kThreads = 1024;
constexpr int kWarps = kThreads / 32;
constexpr int kBatch = 16;   // ids each lane loads at once

// kMulti = false: one block groups all pairs and writes row_offsets.
// kMulti = true: block b groups its segment [b*seg, min(pairs, (b+1)*seg))
// into rows starting, for each expert e, at the base that
// group_scan_kernel left at row_of_pair[b*seg + e] (read before anything is
// written there).
template <bool kMulti>
__global__ void __launch_bounds__(kThreads, 1)
group_rows_kernel(const int32_t *__restrict__ topk, int32_t pairs,
                  int32_t seg, int32_t k, int32_t E,
                  int32_t *__restrict__ row_offsets,
                  int32_t *__restrict__ token_of_row,
                  int32_t *__restrict__ row_of_pair,
                  unsigned int *__restrict__ status) {
    extern __shared__ int32_t smem[];
    int32_t *s_cnt = smem;              // [kWarps][E] counts, then bases
    int32_t *s_tot = smem + kWarps * E; // [E] first row of each expert
    __shared__ int32_t s_warp_sums[kWarps];
    __shared__ int s_bad;

    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const unsigned lt_mask = (1u << lane) - 1u;
    const int32_t b0q = kMulti ? (int32_t)blockIdx.x * seg : 0;
    const int32_t bq1 = kMulti ? min(pairs, b0q + seg) : pairs;
    grid_dependency_wait();
    for (int j = tid; j < kWarps * E; j += kThreads)
        s_cnt[j] = 0;
    if (kMulti)
        for (int e = tid; e < E; e += kThreads)
            s_tot[e] = row_of_pair[b0q + e];
    if (tid == 0)
        s_bad = 0;
    __syncthreads();

    const int32_t wseg = (bq1 - b0q + kWarps - 1) / kWarps;
    const int32_t q0 = min(bq1, b0q + warp * wseg), q1 = min(bq1, q0 + wseg);
    int32_t *cnt = s_cnt + warp * E;

    // 1. per-warp counts; each lane loads kBatch ids before using any, so a
    //    warp waits for one memory latency per 32*kBatch pairs
    for (int32_t b0 = q0; b0 < q1; b0 += 32 * kBatch) {
        int32_t ids[kBatch];
#pragma unroll
        for (int i = 0; i < kBatch; ++i) {
            const int32_t q = b0 + i * 32 + lane;
            ids[i] = q < q1 ? topk[q] : -1;
        }
#pragma unroll
        for (int i = 0; i < kBatch; ++i) {
            int32_t e = ids[i];
            if (b0 + i * 32 + lane < q1 && (e < 0 || e >= E)) {
                e = -1;
                s_bad = 1;
            }
            const unsigned peers = __match_any_sync(0xffffffffu, e);
            if (e >= 0 && (peers & lt_mask) == 0)
                cnt[e] += __popc(peers);
            __syncwarp();
        }
    }
    __syncthreads();

    // 2. per expert: each warp's first row (scan over warps), then (one
    //    block) the offsets (scan over experts; E <= kThreads, one per
    //    thread)
    int32_t tot = 0;
    for (int e = tid; e < E; e += kThreads) {
        int32_t run = 0;
        for (int w = 0; w < kWarps; ++w) {
            const int32_t n = s_cnt[w * E + e];
            s_cnt[w * E + e] = run;
            run += n;
        }
        tot = run;
    }
    if (!kMulti) {
        int32_t incl = tot;
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
            const int32_t w = s_warp_sums[lane];
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
        const int32_t excl = s_warp_sums[warp] + incl - tot;
        if (tid < E) {
            s_tot[tid] = excl;
            row_offsets[tid] = excl;
            if (tid == E - 1)
                row_offsets[E] = excl + tot;
        }
    }
    if (tid == 0 && s_bad)
        atomicOr(status, Q4MOE_DEV_BAD_EXPERT_ID);
    __syncthreads();

    // 3. stable scatter (the ids are read again, kBatch per lane at once)
    for (int32_t b0 = q0; b0 < q1; b0 += 32 * kBatch) {
        int32_t ids[kBatch];
#pragma unroll
        for (int i = 0; i < kBatch; ++i) {
            const int32_t q = b0 + i * 32 + lane;
            ids[i] = q < q1 ? topk[q] : -1;
        }
#pragma unroll
        for (int i = 0; i < kBatch; ++i) {
            const int32_t q = b0 + i * 32 + lane;
            int32_t e = ids[i];
            if (e < 0 || e >= E)
                e = -1;
            const unsigned peers = __match_any_sync(0xffffffffu, e);
            const int rank = __popc(peers & lt_mask);
            int32_t row = -1;
            if (e >= 0)
                row = s_tot[e] + cnt[e] + rank;
            __syncwarp();
            if (e >= 0 && rank == 0)
                cnt[e] += __popc(peers);
            __syncwarp();
            if (q < q1) {
                row_of_pair[q] = row;
                if (row >= 0)
                    token_of_row[row] = q / k;
            }
        }
    }
}

// Multi-block pass 1: block b counts the experts of its segment and leaves
// the counts at row_of_pair[b*seg + e] (its own segment, at least E long).
__global__ void __launch_bounds__(kThreads)
group_count_kernel(const int32_t *__restrict__ topk, int32_t pairs,
                   int32_t seg, int32_t E, int32_t *__restrict__ row_of_pair) {
    extern __shared__ int32_t s_c[];
    grid_dependency_wait();
    for (int e = threadIdx.x; e < E; e += blockDim.x)
        s_c[e] = 0;
    __syncthreads();
    const int32_t q0 = (int32_t)blockIdx.x * seg, q1 = min(pairs, q0 + seg);
    for (int32_t q = q0 + threadIdx.x; q < q1; q += blockDim.x) {
        const int32_t e = topk[q];
        if (e >= 0 && e < E)
            atomicAdd(&s_c[e], 1);
    }
    __syncthreads();
    for (int e = threadIdx.x; e < E; e += blockDim.x)
        row_of_pair[q0 + e] = s_c[e];
}

// Multi-block pass 2 (one block): per expert, the exclusive scan of the
// blocks' counts; over experts, the offsets; the counts become each
// (block, expert)'s first row.  Warp w sums a slice of the blocks.
__global__ void __launch_bounds__(kThreads, 1)
group_scan_kernel(int32_t nblk, int32_t seg, int32_t E,
                  int32_t *__restrict__ row_offsets,
                  int32_t *__restrict__ row_of_pair) {
    extern __shared__ int32_t s_part[];  // [kWarps][E] slice sums, then bases
    __shared__ int32_t s_warp_sums[kWarps];
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int bpw = (nblk + kWarps - 1) / kWarps;
    const int b0 = min(nblk, warp * bpw), b1 = min(nblk, b0 + bpw);
    grid_dependency_wait();
    for (int e = lane; e < E; e += 32) {
        int32_t sum = 0;
        for (int b = b0; b < b1; ++b)
            sum += row_of_pair[b * seg + e];
        s_part[warp * E + e] = sum;
    }
    __syncthreads();
    int32_t tot = 0;
    for (int e = tid; e < E; e += kThreads) {
        int32_t run = 0;
        for (int w = 0; w < kWarps; ++w) {
            const int32_t n = s_part[w * E + e];
            s_part[w * E + e] = run;
            run += n;
        }
        tot = run;
    }
    int32_t incl = tot;
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
        const int32_t w = s_warp_sums[lane];
        int32_t wi = w;
#pragma unroll
        for (int d = 1; d < 32; d <<= 1) {
            const int32_t v = __shfl_up_sync(0xffffffffu, wi, d);
            if (lane >= d)
                wi += v;
        }
        s_warp_sums[lane] = wi - w;
    }
    __syncthreads();
    const int32_t excl = s_warp_sums[warp] + incl - tot;
    if (tid < E) {
        row_offsets[tid] = excl;
        if (tid == E - 1)
            row_offsets[E] = excl + tot;
        for (int w = 0; w < kWarps; ++w)
            s_part[w * E + tid] += excl;
    }
    __syncthreads();
    for (int e = lane; e < E; e += 32) {
        int32_t run = s_part[warp * E + e];
        for (int b = b0; b < b1; ++b) {
            const int32_t n = row_of_pair[b * seg + e];
            row_of_pair[b * seg + e] = run;
            run += n;
        }
    }
}

}  // namespace

cudaError_t launch_group_rows(const int32_t *topk, int64_t pairs, int32_t k,
                              int32_t E, int32_t *row_offsets,
                              int32_t *token_of_row, int32_t *row_of_pair,
                              unsigned int *status, int num_sms,
                              cudaStream_t s) {
    const size_t smem = sizeof(int32_t) * (size_t)E * (1 + kWarps);
    // Large inputs: one block per SM-sized segment of at least
    // max(E, 1024) pairs; the segment of the last block must still hold E
    // counts.
    int32_t nblk = (int32_t)std::min<int64_t>(
        num_sms, pairs / std::max<int32_t>(E, 1024));
    int32_t seg = 0;
    for (; nblk >= 8; --nblk) {
        seg = (int32_t)((pairs + nblk - 1) / nblk);
        if (seg >= E && (int64_t)(nblk - 1) * seg + E <= pairs)
            break;
    }
    cudaError_t err;
    if (nblk >= 8) {
        const size_t scan_smem = sizeof(int32_t) * (size_t)E * kWarps;
        if ((err = cudaFuncSetAttribute(
                 group_rows_kernel<true>,
                 cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem)) !=
                cudaSuccess ||
            (err = cudaFuncSetAttribute(
                 group_scan_kernel,
                 cudaFuncAttributeMaxDynamicSharedMemorySize,
                 (int)scan_smem)) != cudaSuccess)
            return err;
        if ((err = launch_pdl(group_count_kernel, dim3(nblk), dim3(kThreads),
                              sizeof(int32_t) * (size_t)E, s, topk,
                              (int32_t)pairs, seg, E, row_of_pair)) !=
                cudaSuccess ||
            (err = launch_pdl(group_scan_kernel, dim3(1), dim3(kThreads),
                              scan_smem, s, nblk, seg, E, row_offsets,
                              row_of_pair)) != cudaSuccess)
            return err;
        return launch_pdl(group_rows_kernel<true>, dim3(nblk), dim3(kThreads),
                          smem, s, topk, (int32_t)pairs, seg, k, E,
                          row_offsets, token_of_row, row_of_pair, status);
    }
    err = cudaFuncSetAttribute(group_rows_kernel<false>,
                               cudaFuncAttributeMaxDynamicSharedMemorySize,
                               (int)smem);
    if (err != cudaSuccess)
        return err;
    return launch_pdl(group_rows_kernel<false>, dim3(1), dim3(kThreads), smem,
                      s, topk, (int32_t)pairs, 0, k, E, row_offsets,
                      token_of_row, row_of_pair, status);
}

}  // namespace q4moe
