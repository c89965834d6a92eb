// q4moe_trellis.cu -- grouped gate/up + SwiGLU for trellis-coded (QTIP
// 1MAD) experts, with the row scale factored out of the sum.
//
// The arithmetic of the pages' factored trellis kernels ("@mlx-bun/
// inference 0.0.0-stage -> 1.0.0", page 57, trellis/gate-up-mma.ts and
// mixed-gate-up-factored.ts; the decode of page 54, trellis/codebook.ts):
//   state of weight t of a block = the L-bit window at bit (T-1-t)*k of the
//       block's T*k bits, wrapping (bit b is bit b%32 of word b/32);
//   y(state) = the byte sum of state*34038481 + 76625530 (mod 2^32) - 510;
//   G = sum_k y_k x_k in f32;  gate32 = G * (f32(scale) * RN32(1/147.8...));
// then the page 52 SwiGLU tail on gate32/up32.  Gate and up may be coded at
// different widths k.
//
// One warp owns an output row of one expert and up to 8 of its grouped rows
// at a time (every decoded weight serves all of them); lane l owns runs
// l, l+32, ... of 32 consecutive weights of a block, loads the k+1 words that
// hold their windows (as on the page, the words of a run end where the next
// run's start: the window of position j of the run starts at bit (31-j)*k of
// them) and decodes each weight once.  The code value y (-510..510) is
// formed in f32 without a conversion: y + 510 in the mantissa of 2^23 minus
// 2^23 + 510.  Decoding is integer arithmetic (about a dozen operations a
// weight): the kernel is bound by the integer pipe, not by HBM.
#include "q4moe_internal.cuh"

namespace q4moe {
namespace {

constexpr int kWarps = 4;
constexpr int kRowsPerWarp = 2;
constexpr int kRowsPerBlock = kWarps * kRowsPerWarp;
constexpr int kChunk = 8;
constexpr int kMaxBits = 8;

__device__ __forceinline__ float warp_sum(float v) {
#pragma unroll
    for (int d = 16; d > 0; d >>= 1)
        v += __shfl_xor_sync(0xffffffffu, v, d);
    return v;
}

// y(state) as f32 (exact).
__device__ __forceinline__ float trellis_y(uint32_t s) {
    const uint32_t x = s * 34038481u + 76625530u;
    const uint32_t p = (x & 0x00FF00FFu) + ((x >> 8) & 0x00FF00FFu);
    const uint32_t y510 = (p & 0xFFFFu) + (p >> 16);        // y + 510
    return __uint_as_float(0x4B000000u | y510) - 8389118.0f;
}

// The L-bit window at bit b of the words w[0..k] (b + L <= 32 * (k + 1)).
__device__ __forceinline__ uint32_t window(const uint32_t (&w)[kMaxBits + 1],
                                          int b, int L) {
    const int wi = b >> 5, off = b & 31;
    uint32_t v = w[wi] >> off;
    if (off + L > 32)
        v |= w[wi + 1] << (32 - off);
    return v & ((1u << L) - 1u);
}

// The k+1 words of a run: words w0 .. w0 + k of the block, wrapping.
__device__ __forceinline__ void load_run(const uint32_t *blk, int wpb, int w0,
                                         int k, uint32_t (&w)[kMaxBits + 1]) {
#pragma unroll
    for (int i = 0; i <= kMaxBits; ++i) {
        if (i <= k) {
            const int wi = w0 + i;
            w[i] = __ldg(blk + (wi >= wpb ? wi - wpb : wi));
        } else {
            w[i] = 0;
        }
    }
}

// KG, KU: the gate and up widths when known at compile time (the pages' 2,
// 3 and 4 bits: every window's word and shift become constants), else 0
// and the widths are read from the arguments.
template <int KG, int KU>
__global__ void __launch_bounds__(kWarps * 32)
trellis_gate_up_kernel(GateUpArgs a) {
    __shared__ int32_t s_off[Q4MOE_MAX_EXPERTS + 1];
    grid_dependency_wait();
    if (!stage_row_offsets(a, s_off))
        return;
    const int e = blockIdx.y;
    const int32_t r0 = s_off[e], r1 = s_off[e + 1];
    if (r1 == r0)
        return;
    const uint8_t *slab = expert_slab(a, e);
    if (slab == nullptr)
        return;
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const int Tb = a.tr_block, L = a.tr_window;
    const int kg = KG ? KG : a.tr_kg, ku = KU ? KU : a.tr_ku;
    const int gwpb = Tb * kg / 32, uwpb = Tb * ku / 32;
    const int runs_per_block = Tb / 32;
    const int nruns = (int)(a.H / 32);
    const int64_t grow_words = a.H / Tb * gwpb, urow_words = a.H / Tb * uwpb;
    const uint16_t *gs = reinterpret_cast<const uint16_t *>(slab + a.gate_s_off);
    const uint16_t *us = reinterpret_cast<const uint16_t *>(slab + a.up_s_off);
    const float rcp = __uint_as_float(0x3BDDB447u);   // RN32(1/147.800537109375)

    for (int rr = 0; rr < kRowsPerWarp; ++rr) {
        const int64_t i = (int64_t)blockIdx.x * kRowsPerBlock +
                          warp * kRowsPerWarp + rr;
        if (i >= a.I)
            break;
        const uint32_t *grow = reinterpret_cast<const uint32_t *>(
                                   slab + a.gate_w_off) + i * grow_words;
        const uint32_t *urow = reinterpret_cast<const uint32_t *>(
                                   slab + a.up_w_off) + i * urow_words;
        const float sg = __fmul_rn(__half2float(__ushort_as_half(gs[i])), rcp);
        const float su = __fmul_rn(__half2float(__ushort_as_half(us[i])), rcp);
        for (int32_t p0 = r0; p0 < r1; p0 += kChunk) {
            const int nt = min(kChunk, r1 - p0);
            int32_t tok[kChunk];
#pragma unroll
            for (int m = 0; m < kChunk; ++m)
                tok[m] = m < nt ? (int32_t)row_token(a, p0 + m) : -1;
            float ag[kChunk], au[kChunk];
#pragma unroll
            for (int m = 0; m < kChunk; ++m)
                ag[m] = au[m] = 0.0f;
            for (int run = lane; run < nruns; run += 32) {
                const int blk = run / runs_per_block;
                const int t0 = (run - blk * runs_per_block) * 32;
                uint32_t gw[kMaxBits + 1], uw[kMaxBits + 1];
                load_run(grow + (int64_t)blk * gwpb, gwpb,
                         (Tb - 32 - t0) * kg / 32, kg, gw);
                load_run(urow + (int64_t)blk * uwpb, uwpb,
                         (Tb - 32 - t0) * ku / 32, ku, uw);
                const int64_t c0 = (int64_t)blk * Tb + t0;
#pragma unroll
                for (int q = 0; q < 4; ++q) {
                    uint4 xv[kChunk];
#pragma unroll
                    for (int m = 0; m < kChunk; ++m)
                        xv[m] = tok[m] >= 0
                                    ? __ldg(reinterpret_cast<const uint4 *>(
                                                a.x + (int64_t)tok[m] * a.H +
                                                c0) + q)
                                    : make_uint4(0, 0, 0, 0);
#pragma unroll
                    for (int jj = 0; jj < 8; ++jj) {
                        const int j = q * 8 + jj;
                        const float yg = trellis_y(window(gw, (31 - j) * kg, L));
                        const float yu = trellis_y(window(uw, (31 - j) * ku, L));
#pragma unroll
                        for (int m = 0; m < kChunk; ++m) {
                            if (m >= nt)
                                continue;
                            const uint32_t h =
                                (&xv[m].x)[jj >> 1] >> (16 * (jj & 1));
                            const float xf = bf16_f32(h & 0xFFFFu);
                            ag[m] = __fmaf_rn(yg, xf, ag[m]);
                            au[m] = __fmaf_rn(yu, xf, au[m]);
                        }
                    }
                }
            }
#pragma unroll
            for (int m = 0; m < kChunk; ++m) {
                const float G = warp_sum(ag[m]);
                const float U = warp_sum(au[m]);
                if (lane == m && tok[m] >= 0) {
                    const float g32 = __fmul_rn(G, sg);
                    const float u32 = __fmul_rn(U, su);
                    const int64_t o = (int64_t)(p0 + m) * a.I + i;
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

template <int KG, int KU>
cudaError_t launch_widths(const GateUpArgs &a, cudaStream_t s) {
    const dim3 grid((unsigned)((a.I + kRowsPerBlock - 1) / kRowsPerBlock),
                    (unsigned)a.E);
    return launch_pdl(trellis_gate_up_kernel<KG, KU>, grid, dim3(kWarps * 32),
                      0, s, a);
}

template <int KG>
cudaError_t launch_up_width(const GateUpArgs &a, cudaStream_t s) {
    switch (a.tr_ku) {
    case 2: return launch_widths<KG, 2>(a, s);
    case 3: return launch_widths<KG, 3>(a, s);
    case 4: return launch_widths<KG, 4>(a, s);
    default: return launch_widths<0, 0>(a, s);
    }
}

}  // namespace

cudaError_t launch_trellis_gate_up(const GateUpArgs &a, cudaStream_t s) {
    switch (a.tr_kg) {
    case 2: return launch_up_width<2>(a, s);
    case 3: return launch_up_width<3>(a, s);
    case 4: return launch_up_width<4>(a, s);
    default: return launch_widths<0, 0>(a, s);
    }
}

}  // namespace q4moe
