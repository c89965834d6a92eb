// q4moe_matvec.cu -- grouped Q4 gate/up + SwiGLU matvec for experts with few
// rows (decode / speculative verify widths).
//
// launch_matvec picks the first version the call allows (the TMA version
// with a fixed unit height and the generic version are batch-invariant: a
// row's result does not depend on the other rows of the call):
//   q4moe_matvec_lat.cu  one expert, 1 to 8 grouped rows, gate/up, not in
//                        batch-invariant calls (laid out for latency);
//   q4moe_matvec_tma.cu  slabs at base + e * stride, H % 256 == 0,
//                        I % 16 == 0, 16-byte aligned weight sections
//                        (weights moved by TMA);
//   q4moe_matvec_mma.cu  also a per-expert pointer table, H % 128 == 0
//                        (weights moved by per-thread cp.async);
//   this generic version otherwise.
//
// Generic version: any H % 8 == 0, I % 4 == 0.  One warp owns one output
// row i of one expert and up to 8 of the expert's grouped rows at a time,
// so every packed word it loads serves all of them (the shared-row idea of
// the pages' trellis GATEUP_SHARED_M_SOURCE, page 57, gate-up.ts); lanes
// stride over the row's words as the page's GATE_UP_SOURCE does (page 52),
// accumulate gate and up in f32, and meet in a shuffle reduction.
//
// The down projection (page 52, DOWN_SOURCE) uses the TMA version when it
// can (its K, the MLP's intermediate size, % 256 == 0, output rows % 16 ==
// 0, slabs at base + e * stride), else the generic down kernel below (any
// K % 8 == 0): one warp per output row, one matrix, no tail.
#include "q4moe_internal.cuh"
#include "q4moe_sm100.cuh"

namespace q4moe {
namespace {

constexpr int kWarpsPerBlock = 4;
constexpr int kRowsPerWarp = 4;
constexpr int kRowsPerBlock = kWarpsPerBlock * kRowsPerWarp;
constexpr int kChunk = 8;

__device__ __forceinline__ float warp_sum(float v) {
#pragma unroll
    for (int d = 16; d > 0; d >>= 1)
        v += __shfl_xor_sync(0xffffffffu, v, d);
    return v;
}

// Weight `place` of packed word w: nibble place minus 8 (Q4, 8 per word)
// or signed byte place (Q8, 4 per word), as f32.
template <bool kQ8>
__device__ __forceinline__ float weight_at(uint32_t w, int place) {
    if (kQ8)
        return (float)(int)(int8_t)(w >> (8 * place));
    return (float)((int)((w >> (4 * place)) & 0xFu) - 8);
}

// The activations matching word w of a row: 8 bf16 (Q4) or 4 (Q8).
template <bool kQ8>
__device__ __forceinline__ void load_acts(const uint16_t *row, int64_t w,
                                          uint32_t (&v)[4]) {
    if (kQ8) {
        const uint2 t = *reinterpret_cast<const uint2 *>(row + w * 4);
        v[0] = t.x;
        v[1] = t.y;
        v[2] = v[3] = 0;
    } else {
        const uint4 t = *reinterpret_cast<const uint4 *>(row + w * 8);
        v[0] = t.x;
        v[1] = t.y;
        v[2] = t.z;
        v[3] = t.w;
    }
}

template <bool kQ8>
__global__ void __launch_bounds__(kWarpsPerBlock * 32)
matvec_generic_kernel(GateUpArgs a) {
    constexpr int kPer = kQ8 ? 4 : 8;            // weights per 32-bit word
    __shared__ int32_t s_off[Q4MOE_MAX_EXPERTS + 1];
    grid_dependency_wait();
    if (!stage_row_offsets(a, s_off))
        return;
    const int32_t mvmax = matvec_limit(a, s_off);
    const int e = blockIdx.y;
    const int32_t r0 = s_off[e], r1 = s_off[e + 1];
    const int32_t rows = r1 - r0;
    if (rows == 0 || rows > mvmax)
        return;
    const uint8_t *slab = expert_slab(a, e);
    if (slab == nullptr)
        return;
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const int64_t words = a.H / kPer;
    const float *gs = reinterpret_cast<const float *>(slab + a.gate_s_off);
    const float *us = reinterpret_cast<const float *>(slab + a.up_s_off);

    for (int rr = 0; rr < kRowsPerWarp; ++rr) {
        const int64_t i = (int64_t)blockIdx.x * kRowsPerBlock +
                          warp * kRowsPerWarp + rr;
        if (i >= a.I)
            break;
        const uint32_t *gw = reinterpret_cast<const uint32_t *>(
                                 slab + a.gate_w_off) + i * words;
        const uint32_t *uw = reinterpret_cast<const uint32_t *>(
                                 slab + a.up_w_off) + i * words;
        for (int32_t p0 = r0; p0 < r1; p0 += kChunk) {
            const int nt = min(kChunk, r1 - p0);
            int64_t tok[kChunk];
#pragma unroll
            for (int j = 0; j < kChunk; ++j)
                tok[j] = j < nt ? row_token(a, p0 + j) : -1;
            float ag[kChunk], au[kChunk];
#pragma unroll
            for (int j = 0; j < kChunk; ++j)
                ag[j] = au[j] = 0.0f;
            for (int64_t w = lane; w < words; w += 32) {
                const uint32_t g = gw[w], u = uw[w];
#pragma unroll
                for (int j = 0; j < kChunk; ++j) {
                    if (tok[j] < 0)
                        continue;
                    uint32_t xw[4];
                    load_acts<kQ8>(a.x + tok[j] * a.H, w, xw);
#pragma unroll
                    for (int place = 0; place < kPer; ++place) {
                        const float xf = bf16_f32(
                            (xw[place >> 1] >> (16 * (place & 1))) & 0xFFFFu);
                        ag[j] = __fmaf_rn(weight_at<kQ8>(g, place), xf, ag[j]);
                        au[j] = __fmaf_rn(weight_at<kQ8>(u, place), xf, au[j]);
                    }
                }
            }
#pragma unroll
            for (int j = 0; j < kChunk; ++j) {
                const float G = warp_sum(ag[j]);
                const float U = warp_sum(au[j]);
                if (lane == j && tok[j] >= 0) {
                    const float g32 = __fmul_rn(G, gs[i]);
                    const float u32 = __fmul_rn(U, us[i]);
                    const int64_t o = (int64_t)(p0 + j) * a.I + i;
                    a.out[o] = swiglu_out(a.sigmoid, g32, u32);
                    if (a.gate_f32)
                        a.gate_f32[o] = g32;
                    if (a.up_f32)
                        a.up_f32[o] = u32;
                }
            }
        }
    }
}

// Down projection, generic: warp per output row h (a.I of them) of one
// expert, lanes over the row's K/8 words, up to 8 grouped rows of mid at a
// time; out = bf16(sum * scale).
template <bool kQ8>
__global__ void __launch_bounds__(kWarpsPerBlock * 32)
down_generic_kernel(GateUpArgs a) {
    constexpr int kPer = kQ8 ? 4 : 8;
    __shared__ int32_t s_off[Q4MOE_MAX_EXPERTS + 1];
    grid_dependency_wait();
    if (!stage_row_offsets(a, s_off))
        return;
    const int32_t mvmax = matvec_limit(a, s_off);
    const int e = blockIdx.y;
    const int32_t r0 = s_off[e], r1 = s_off[e + 1];
    const int32_t rows = r1 - r0;
    if (rows == 0 || rows > mvmax)
        return;
    const uint8_t *slab = expert_slab(a, e);
    if (slab == nullptr)
        return;
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const int64_t words = a.H / kPer;
    const float *ds = reinterpret_cast<const float *>(slab + a.gate_s_off);
    for (int rr = 0; rr < kRowsPerWarp; ++rr) {
        const int64_t h = (int64_t)blockIdx.x * kRowsPerBlock +
                          warp * kRowsPerWarp + rr;
        if (h >= a.I)
            break;
        const uint32_t *dw = reinterpret_cast<const uint32_t *>(
                                 slab + a.gate_w_off) + h * words;
        for (int32_t p0 = r0; p0 < r1; p0 += kChunk) {
            const int nt = min(kChunk, r1 - p0);
            float acc[kChunk];
#pragma unroll
            for (int j = 0; j < kChunk; ++j)
                acc[j] = 0.0f;
            for (int64_t w = lane; w < words; w += 32) {
                const uint32_t q = dw[w];
#pragma unroll
                for (int j = 0; j < kChunk; ++j) {
                    if (j >= nt)
                        continue;
                    uint32_t mw[4];
                    load_acts<kQ8>(a.x + (int64_t)(p0 + j) * a.H, w, mw);
#pragma unroll
                    for (int place = 0; place < kPer; ++place) {
                        const float mf = bf16_f32(
                            (mw[place >> 1] >> (16 * (place & 1))) & 0xFFFFu);
                        acc[j] = __fmaf_rn(weight_at<kQ8>(q, place), mf,
                                           acc[j]);
                    }
                }
            }
#pragma unroll
            for (int j = 0; j < kChunk; ++j) {
                const float D = warp_sum(acc[j]);
                if (lane == j && j < nt) {
                    const float v = __fmul_rn(D, ds[h]);
                    const int64_t o = (int64_t)(p0 + j) * a.I + h;
                    a.out[o] = bf16_rne(v);
                    if (a.gate_f32)
                        a.gate_f32[o] = v;
                }
            }
        }
    }
}

__global__ void debug_tail_kernel(const uint16_t *g, const uint16_t *u,
                                  int64_t n, uint16_t *res,
                                  const uint16_t *table, int mlx) {
    // (table: the page 52 tail's or the MLX tail's)
    grid_dependency_wait();
    for (int64_t j = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; j < n;
         j += (int64_t)gridDim.x * blockDim.x) {
        const uint16_t gT = g[j];
        uint16_t s, si;
        const uint16_t o = swiglu_tail_bits(table, gT, u[j], &s, &si);
        res[4 * j + 0] = s;
        res[4 * j + 1] = si;
        res[4 * j + 2] = o;
        // the sigmoid as the decode kernels form it for the page's tail:
        // in registers when the fast form is conclusive, else the table
        uint16_t sd = s;
        if (!mlx) {
            bool ok;
            sd = sigmoid_bf16_fast(bf16_f32(gT), &ok);
            if (!ok)
                sd = sigmoid_bf16_table(table, gT);
        }
        res[4 * j + 3] = sd;
    }
}

}  // namespace

cudaError_t launch_matvec(const GateUpArgs &a, cudaStream_t s) {
    if (matvec_latency_supported(a))
        return launch_matvec_latency(a, s);
    if (matvec_tma_supported(a))
        return launch_matvec_tma(a, s);
    const dim3 grid((unsigned)((a.I + kRowsPerBlock - 1) / kRowsPerBlock),
                    (unsigned)a.E);
    const dim3 block(kWarpsPerBlock * 32);
    if (a.down)
        return a.q8 ? launch_pdl(down_generic_kernel<true>, grid, block, 0, s,
                                 a)
                    : launch_pdl(down_generic_kernel<false>, grid, block, 0,
                                 s, a);
    // (the cp.async version's reduction depends on the call's size: not
    // used when the call must be batch-invariant; Q4 only)
    if (!a.invariant && !a.q8 && matvec_mma_supported(a))
        return launch_matvec_mma(a, s);
    return a.q8 ? launch_pdl(matvec_generic_kernel<true>, grid, block, 0, s, a)
                : launch_pdl(matvec_generic_kernel<false>, grid, block, 0, s,
                             a);
}

namespace {
// The bounded waits of the kernels on an mbarrier that nothing arrives on:
// thread 0 waits as the producers and consumers do (try_wait), thread 32 as
// the MMA issuer does (test_wait spin).  The first to run out raises
// Q4MOE_DEV_WAIT_TIMEOUT and the abort flag, which ends the other's wait.
__global__ void debug_wait_kernel(unsigned int *status, uint64_t limit_ns) {
    __shared__ uint64_t bar;
    __shared__ int abort_flag;
    grid_dependency_wait();
    if (threadIdx.x == 0) {
        sm100::mbar_init(&bar, 1);
        abort_flag = 0;
        sm100::fence_mbar_init();
    }
    __syncthreads();
    volatile int *abort = &abort_flag;
    if (threadIdx.x == 0)
        sm100::wait_phase(&bar, 0, abort, status, limit_ns);
    else if (threadIdx.x == 32)
        sm100::wait_spin(&bar, 0, abort, status, limit_ns);
    __syncthreads();
}
}  // namespace

cudaError_t launch_debug_wait(unsigned int *status, uint64_t limit_ns,
                              cudaStream_t s) {
    return launch_pdl(debug_wait_kernel, dim3(1), dim3(64), 0, s, status,
                      limit_ns);
}

cudaError_t launch_debug_tail(const uint16_t *g, const uint16_t *u, int64_t n,
                              uint16_t *res, const uint16_t *sigmoid,
                              bool mlx, cudaStream_t s) {
    if (n == 0)
        return cudaSuccess;
    const int blocks = (int)std::min<int64_t>((n + 255) / 256, 4096);
    return launch_pdl(debug_tail_kernel, dim3((unsigned)blocks), dim3(256), 0,
                      s, g, u, n, res,
                      mlx ? sigmoid + kSigmoidTable : sigmoid, mlx ? 1 : 0);
}

}  // namespace q4moe
