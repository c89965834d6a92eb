// q4moe_internal.cuh -- launch arguments and device helpers shared by the
// CUDA translation units of libq4moe (not part of the public ABI).
#pragma once

#include <cstdint>
#include <utility>
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>

#include "q4moe.h"

namespace q4moe {

// Everything a gate/up kernel needs, resolved and validated on the host.
// The down projection (down = 1) runs on the same kernels with the roles
// renamed: x is mid (bf16 [M][H], H = the projection's K, the MLP's
// intermediate size), row p reads x row p (token_of_row unused), I is its
// output rows (the MLP's hidden size), the gate and up sections both name
// the down words and scales, and the two halves of a tile are two blocks
// of output rows of the one matrix: out = bf16(sum * scale), no tail.
struct GateUpArgs {
    const uint16_t *x;           // bf16 [T][H]
    const uint8_t *base;         // slab of expert e at base + e * stride ...
    int64_t stride;
    const uint8_t *const *slab_ptrs;  // ... or at slab_ptrs[e] when non-null
    int64_t gate_w_off, up_w_off, gate_s_off, up_s_off;
    const int32_t *row_offsets;  // [E+1]
    const int32_t *token_of_row; // [M]
    int64_t M, H, I, T;          // T <= 0: token indices unchecked
    int32_t E;
    uint16_t *out;               // bf16 [M][I]
    float *gate_f32;             // optional [M][I]
    float *up_f32;               // optional [M][I]
    uint16_t *xg;                // optional workspace: bf16 [M][H], the
                                 // routed activations in grouped order
    unsigned int *status;        // device status word (Q4MOE_DEV_* bits)
    int32_t matvec_max_rows;     // experts with more rows go to the GEMM
    int32_t num_sms;
    int32_t matvec_tile;         // TMA matvec unit height (0: automatic)
    int32_t matvec_last;         // no GEMM launch follows the matvec's
    int32_t hold_next;           // 1: the single-expert latency kernel does
                                 // not release the next launch early (the
                                 // down stage of the expert MLP)
    const uint16_t *sigmoid;     // sigmoid tables: [2][65536] bf16, indexed
                                 // by the bf16 bits of gateT: the page 52
                                 // tail's, then the MLX tail's
    int32_t tail_mlx;            // 1: MLX's tail (trellis calls only)
    int32_t down;                // 1: the down projection (above)
    int32_t invariant;           // 1: batch-invariant matvec versions only
    int32_t q8;                  // 1: signed-byte weights (rows of H bytes)
    // trellis experts: block size, window bits, gate and up widths (the
    // gate/up word and scale offsets then name codes and f16 scales)
    int32_t tr_block, tr_window, tr_kg, tr_ku;
    int32_t tr_rows_per_warp;    // output rows one warp of the kernel takes
};

// Bytes of one weight row of K values.
__host__ __device__ __forceinline__ int64_t weight_row_bytes(
    const GateUpArgs &a, int64_t K) {
    return a.q8 ? K : K / 2;
}

// Host-side count of kernel launches (q4moe_launch_count).
void count_launches(int n);

// Programmatic dependent launch.  Every kernel of the library is launched
// with launch_pdl, so that its launch and set-up overlap the end of the
// previous kernel on the stream; each one calls grid_dependency_wait before
// it reads any input or writes any output (it returns once the previous
// kernel has completed and its memory is visible).  The next kernel may
// start launching as this one's blocks exit; only the matvec, when it is
// the call's last kernel, lets it start at once (grid_launch_dependents):
// measured, an early start slows a following GEMM, gather or grouping.
__device__ __forceinline__ void grid_dependency_wait() {
    asm volatile("griddepcontrol.wait;" ::: "memory");
}
__device__ __forceinline__ void grid_launch_dependents() {
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}

template <typename... KArgs, typename... Args>
cudaError_t launch_pdl(void (*kernel)(KArgs...), dim3 grid, dim3 block,
                       size_t smem, cudaStream_t s, Args &&...args) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = grid;
    cfg.blockDim = block;
    cfg.dynamicSmemBytes = smem;
    cfg.stream = s;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    const cudaError_t err =
        cudaLaunchKernelEx(&cfg, kernel, std::forward<Args>(args)...);
    count_launches(1);
    return err != cudaSuccess ? err : cudaGetLastError();
}

// Record `message` as the calling thread's last error; returns `code`.
int report_error(int code, const char *message);

cudaError_t launch_matvec(const GateUpArgs &a, cudaStream_t s);
bool matvec_mma_supported(const GateUpArgs &a);
cudaError_t launch_matvec_mma(const GateUpArgs &a, cudaStream_t s);
bool matvec_tma_supported(const GateUpArgs &a);
// One expert, at most 8 grouped rows (q4moe_matvec_lat.cu).
bool matvec_latency_supported(const GateUpArgs &a);
cudaError_t launch_matvec_latency(const GateUpArgs &a, cudaStream_t s);
cudaError_t launch_matvec_tma(const GateUpArgs &a, cudaStream_t s);
cudaError_t launch_gemm(const GateUpArgs &a, cudaStream_t s);
// The tcgen05 GEMM whose weights, dequantised tiles and token rows all move
// through TMA-fed rings (q4moe_gemm_tma.cu), on token rows already in
// grouped order (the workspace copy of x, or mid for the down projection).
bool gemm_tma_supported(const GateUpArgs &a);
cudaError_t launch_gemm_tma(const GateUpArgs &a, const uint16_t *rows,
                           cudaStream_t s);
cudaError_t launch_trellis_gate_up(const GateUpArgs &a, cudaStream_t s);
// GEMM tiles over the output rows of one expert's 256 grouped rows: 128
// intermediate rows (gate and up) per tile, or 256 output rows (two halves
// of 128) for the down projection.
__host__ __device__ __forceinline__ int gemm_row_tiles(const GateUpArgs &a) {
    return a.down ? (int)((a.I + 255) / 256) : (int)(a.I / 128);
}
bool gemm_supported(int64_t H, int64_t I, const GateUpArgs &a);
cudaError_t launch_group_rows(const int32_t *topk, int64_t pairs, int32_t k,
                              int32_t E, int32_t *row_offsets,
                              int32_t *token_of_row, int32_t *row_of_pair,
                              unsigned int *status, int num_sms,
                              cudaStream_t s);
cudaError_t launch_debug_wait(unsigned int *status, uint64_t limit_ns,
                              cudaStream_t s);
cudaError_t launch_debug_tail(const uint16_t *g, const uint16_t *u,
                              int64_t n, uint16_t *res,
                              const uint16_t *sigmoid, bool mlx,
                              cudaStream_t s);
// Entries of one sigmoid table; the MLX tail's table follows the page's.
constexpr int kSigmoidTable = 65536;

// ------------------------------------------------------------------------
// bf16 helpers.  Rounding: nearest, ties to even (page 54, codebook.ts,
// trellis_bf16), done by the hardware conversion (subnormals kept); every
// value reaching it is finite, but for the MLX sigmoid's exponential past
// FLT_MAX, an infinity, which converts to itself.
__device__ __forceinline__ uint16_t bf16_rne(float v) {
    return __bfloat16_as_ushort(__float2bfloat16_rn(v));
}

__device__ __forceinline__ float bf16_f32(uint32_t b16) {
    return __uint_as_float(b16 << 16);
}

// The same rounding done on the bit pattern with integer operations (the
// page's own formulation: add 0x7FFF plus the lowest kept bit, drop the low
// 16 bits), returning the rounded value as an f32 (bf16_round) or its bf16
// bits (bf16_bits).  Used on hot paths, where the integer unit is faster
// than the conversion unit.
__device__ __forceinline__ float bf16_round(float v) {
    const uint32_t u = __float_as_uint(v);
    return __uint_as_float((u + 0x7FFFu + ((u >> 16) & 1u)) & 0xFFFF0000u);
}

__device__ __forceinline__ uint16_t bf16_bits(float v) {
    const uint32_t u = __float_as_uint(v);
    return (uint16_t)((u + 0x7FFFu + ((u >> 16) & 1u)) >> 16);
}

// Two f32 values rounded to bf16 (to nearest even) by one packed
// conversion: lo in the low half, hi in the high half.
__device__ __forceinline__ uint32_t bf16x2_rn(float lo, float hi) {
    const __nv_bfloat162 r = __floats2bfloat162_rn(lo, hi);
    return *reinterpret_cast<const uint32_t *>(&r);
}

// The tail's two products, sil = bf16(gateT * sigT) and out =
// bf16(sil * upT), on packed pairs of bf16 (bit patterns).  Both operands
// of each product are bf16, so its exact value has at most 16 significant
// bits: from 2^-134 up it is an f32, and below 2^-134 it rounds to zero in
// bf16 whatever comes first.  The page's f32 multiply followed by rounding
// to bf16 is therefore a single rounding, the one the packed bf16 multiply
// (round to nearest even, subnormals kept) makes.
__device__ __forceinline__ uint32_t swiglu_tail_pair(uint32_t g2, uint32_t s2,
                                                     uint32_t u2) {
    const __nv_bfloat162 si =
        __hmul2_rn(*reinterpret_cast<const __nv_bfloat162 *>(&g2),
                   *reinterpret_cast<const __nv_bfloat162 *>(&s2));
    const __nv_bfloat162 o =
        __hmul2_rn(si, *reinterpret_cast<const __nv_bfloat162 *>(&u2));
    return *reinterpret_cast<const uint32_t *>(&o);
}

__device__ __forceinline__ float ex2_approx(float x) {
    float y;
    asm("ex2.approx.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}

__device__ __forceinline__ float rcp_approx(float x) {
    float y;
    asm("rcp.approx.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}

// bf16 sigmoid of a bf16 value g, in two parts so that callers can run the
// first on many values at once.  sigmoid_bf16_fast_f forms
// exp(-g) = 2^(-g log2 e) with the hardware ex2 approximation, carrying the
// rounding error of the argument: log2 e is split into a float head and
// tail, t = -g * head is rounded, and the exact remainder
// fma(-g, head, -t) - g * tail multiplies the result as 1 + r ln 2 (its
// square is below 2^-40).  Then sigmoid = rcp(1 + e).  For g > -16 its error
// against the page's f32 chain is a few f32 ulp (ex2 and rcp about 2 ulp
// each), so when it lies more than 16 ulp from a bf16 rounding midpoint both
// round to the same bf16 and *ok is set; otherwise the caller takes the
// table entry.  (sigmoidT depends on the 16-bit g only; the fast form's
// conclusive results and the table are tested against the oracle on all
// 65,536 inputs.)
__device__ __forceinline__ float sigmoid_bf16_fast_f(float g, bool *ok) {
    const float kHead = 1.44269502162933349609375f;  // float(log2 e)
    const float kTail = 1.925963033500011e-08f;      // log2 e - kHead
    const float kLn2 = 0.693147180559945309f;
    const float a = -fminf(g, 16.0f);  // sigmoidT is 1.0 for every g >= 16
    const float t = a * kHead;
    const float r = __fmaf_rn(a, kHead, -t) + a * kTail;
    const float p = ex2_approx(t);
    const float e = __fmaf_rn(p, r * kLn2, p);
    const float s = rcp_approx(1.0f + e);
    const int lo = (int)(__float_as_uint(s) & 0xFFFFu);
    *ok = (g > -16.0f) && (abs(lo - 0x8000) > 16);
    return bf16_round(s);
}

__device__ __forceinline__ uint16_t sigmoid_bf16_fast(float g, bool *ok) {
    return (uint16_t)(__float_as_uint(sigmoid_bf16_fast_f(g, ok)) >> 16);
}

// sigmoidT depends on the 16 bits of gateT only: the kernels read it from a
// table of all 65,536 values, constant data of the library image computed
// at build time from the page's f32 chain (tested against the oracle on
// every input).  The table is 128 KB and stays in L2.
__device__ __forceinline__ uint16_t sigmoid_bf16_table(const uint16_t *table,
                                                       uint16_t gT) {
    return __ldg(table + gT);
}

// gateT, upT -> out (bf16 bits).  sig and silu are also returned.  Both
// tails share the steps after the sigmoid; `table` selects the tail.
__device__ __forceinline__ uint16_t swiglu_tail_bits(const uint16_t *table,
                                                     uint16_t gT, uint16_t uT,
                                                     uint16_t *sigT,
                                                     uint16_t *siluT) {
    const float g = bf16_f32(gT);
    const uint16_t s = sigmoid_bf16_table(table, gT);
    const uint16_t si = bf16_rne(__fmul_rn(g, bf16_f32(s)));
    *sigT = s;
    *siluT = si;
    return bf16_rne(__fmul_rn(bf16_f32(si), bf16_f32(uT)));
}

// The same for one element whose latency matters more than its count (the
// matvec's few outputs per thread): the sigmoid computed in registers when
// the fast form is conclusive (it then equals the table entry: both are the
// correctly rounded chain), the table only otherwise.
__device__ __forceinline__ uint16_t swiglu_out(const uint16_t *table,
                                               float gate32, float up32) {
    const uint16_t gT = bf16_rne(gate32), uT = bf16_rne(up32);
    const float g = bf16_f32(gT);
    bool ok;
    uint16_t s = sigmoid_bf16_fast(g, &ok);
    if (!ok)
        s = sigmoid_bf16_table(table, gT);
    const uint16_t si = bf16_rne(__fmul_rn(g, bf16_f32(s)));
    return bf16_rne(__fmul_rn(bf16_f32(si), bf16_f32(uT)));
}

// Slab of expert e; null (and a status bit) for a misaligned table entry.
__device__ __forceinline__ const uint8_t *expert_slab(const GateUpArgs &a,
                                                      int e) {
    if (a.slab_ptrs == nullptr)
        return a.base + (int64_t)e * a.stride;
    const uint8_t *p = a.slab_ptrs[e];
    if (p == nullptr ||
        (reinterpret_cast<uintptr_t>(p) & (Q4MOE_SLAB_ALIGNMENT - 1)) != 0) {
        atomicOr(a.status, Q4MOE_DEV_BAD_SLAB_PTR);
        return nullptr;
    }
    return p;
}

// Stage row_offsets[0..E] in shared memory and check them (0 first, M last,
// never decreasing).  Every thread of the block must call it; returns false
// (and block 0 raises the status bit) when they are inconsistent.
__device__ __forceinline__ bool stage_row_offsets(const GateUpArgs &a,
                                                  int32_t *s_off) {
    __shared__ int s_bad;
    if (threadIdx.x == 0)
        s_bad = 0;
    __syncthreads();
    for (int e = threadIdx.x; e <= a.E; e += blockDim.x) {
        const int32_t v = a.row_offsets[e];
        s_off[e] = v;
        bool bad = (e == 0 && v != 0) || (e == a.E && v != a.M) || v < 0 ||
                   v > a.M;
        if (e > 0 && a.row_offsets[e - 1] > v)
            bad = true;
        if (bad)
            s_bad = 1;
    }
    __syncthreads();
    const bool ok = s_bad == 0;
    if (!ok && threadIdx.x == 0 && blockIdx.x == 0 && blockIdx.y == 0 &&
        blockIdx.z == 0)
        atomicOr(a.status, Q4MOE_DEV_BAD_ROW_OFFSETS);
    return ok;
}

// Experts with more rows than this go to the GEMM (the host's kernel
// choice; every kernel of the call reads the same value).  The staged row
// offsets are not needed: the choice is a row threshold.
__device__ __forceinline__ int32_t matvec_limit(const GateUpArgs &a,
                                                const int32_t *) {
    return a.matvec_max_rows;
}

// Token of grouped row p, or -1 (and a status bit) when out of range.
__device__ __forceinline__ int64_t row_token(const GateUpArgs &a, int64_t p) {
    const int32_t t = a.token_of_row[p];
    if (t < 0 || (a.T > 0 && t >= a.T)) {
        atomicOr(a.status, Q4MOE_DEV_BAD_TOKEN);
        return -1;
    }
    return t;
}

}  // namespace q4moe
