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
// then the SwiGLU tail on gate32/up32: page 52's, or MLX's compiled SwiGLU
// in bf16 arithmetic, which the pages' mixed-width kernel ends with (the
// sigmoid from a table of all bf16 gate values).  Gate and up may be coded
// at different widths k.
//
// One warp owns an output row of one expert and up to 8 of its grouped rows
// at a time (every decoded weight serves all of them); lane l owns runs
// l, l+32, ... of 32 consecutive weights of a block, loads the k+1 words that
// hold their windows (as on the page, the words of a run end where the next
// run's start: the window of position j of the run starts at bit (31-j)*k of
// them) and decodes each weight once: a funnel shift and a mask for the
// state, a multiply-add for the hash, one dp4a for its byte sum placed in
// the mantissa of 2^23, one f32 subtraction for y (-510..510).  Decoding is
// integer arithmetic: the kernel is bound by the instruction issue rate,
// not by HBM.
#include "q4moe_internal.cuh"

namespace q4moe {
namespace {

constexpr int kWarps = 4;
constexpr int kMaxRowsPerWarp = 8;
constexpr int kChunk = 8;
constexpr int kMaxBits = 8;

__device__ __forceinline__ float warp_sum(float v) {
#pragma unroll
    for (int d = 16; d > 0; d >>= 1)
        v += __shfl_xor_sync(0xffffffffu, v, d);
    return v;
}

// y(state) as f32 (exact): the byte sum of x comes from one dp4a (bytes
// times 1, unsigned) whose accumulator 0x4B000000 places it in the
// mantissa of 2^23 (the sum is below 1021, so the exponent is untouched);
// subtracting 2^23 + 510 leaves y.
__device__ __forceinline__ float trellis_y(uint32_t s) {
    const uint32_t x = s * 34038481u + 76625530u;
    const uint32_t v = __dp4a(x, 0x01010101u, 0x4B000000u);
    return __uint_as_float(v) - 8389118.0f;
}

// The window at bit b of the words w[0..k], masked to L bits: one funnel
// shift of the two words it can touch (b < 32 * k, so word b/32 + 1 is
// always loaded).
__device__ __forceinline__ uint32_t window(const uint32_t (&w)[kMaxBits + 1],
                                          int b, uint32_t mask) {
    const int wi = b >> 5;
    return __funnelshift_r(w[wi], w[wi + 1], b & 31) & mask;
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

// This lane's part of the sums of one chunk of NT grouped rows (tok[m] the
// x row of chunk row m, or -1 for a row left out) over its runs of one
// output row: ag[m] = sum y_gate * x[m], au[m] likewise for up.
template <int KG, int KU, int NT>
__device__ __forceinline__ void chunk_sums(const GateUpArgs &a,
                                           const uint32_t *grow,
                                           const uint32_t *urow,
                                           const int32_t (&tok)[kChunk],
                                           uint32_t lmask, float (&ag)[kChunk],
                                           float (&au)[kChunk]) {
    const int lane = threadIdx.x & 31;
    const int Tb = a.tr_block;
    const int kg = KG ? KG : a.tr_kg, ku = KU ? KU : a.tr_ku;
    const int gwpb = Tb * kg / 32, uwpb = Tb * ku / 32;
    const int runs_per_block = Tb / 32;
    const int nruns = (int)(a.H / 32);
#pragma unroll
    for (int m = 0; m < kChunk; ++m)
        ag[m] = au[m] = 0.0f;
    for (int run = lane; run < nruns; run += 32) {
        const int blk = run / runs_per_block;
        const int t0 = (run - blk * runs_per_block) * 32;
        uint32_t gw[kMaxBits + 1], uw[kMaxBits + 1];
        load_run(grow + (int64_t)blk * gwpb, gwpb, (Tb - 32 - t0) * kg / 32,
                 kg, gw);
        load_run(urow + (int64_t)blk * uwpb, uwpb, (Tb - 32 - t0) * ku / 32,
                 ku, uw);
        const int64_t c0 = (int64_t)blk * Tb + t0;
#pragma unroll
        for (int q = 0; q < 4; ++q) {
            uint4 xv[NT];
#pragma unroll
            for (int m = 0; m < NT; ++m)
                xv[m] = tok[m] >= 0
                            ? __ldg(reinterpret_cast<const uint4 *>(
                                        a.x + (int64_t)tok[m] * a.H + c0) + q)
                            : make_uint4(0, 0, 0, 0);
#pragma unroll
            for (int jj = 0; jj < 8; ++jj) {
                const int j = q * 8 + jj;
                const float yg = trellis_y(window(gw, (31 - j) * kg, lmask));
                const float yu = trellis_y(window(uw, (31 - j) * ku, lmask));
#pragma unroll
                for (int m = 0; m < NT; ++m) {
                    const uint32_t h = (&xv[m].x)[jj >> 1];
                    const float xf = __uint_as_float(
                        (jj & 1) ? (h & 0xFFFF0000u) : (h << 16));
                    ag[m] = __fmaf_rn(yg, xf, ag[m]);
                    au[m] = __fmaf_rn(yu, xf, au[m]);
                }
            }
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
    const int Tb = a.tr_block;
    const uint32_t lmask = (1u << a.tr_window) - 1u;   // L <= 24
    const int kg = KG ? KG : a.tr_kg, ku = KU ? KU : a.tr_ku;
    const int64_t grow_words = a.H / Tb * (Tb * kg / 32);
    const int64_t urow_words = a.H / Tb * (Tb * ku / 32);
    const uint16_t *gs = reinterpret_cast<const uint16_t *>(slab + a.gate_s_off);
    const uint16_t *us = reinterpret_cast<const uint16_t *>(slab + a.up_s_off);
    const float rcp = __uint_as_float(0x3BDDB447u);   // RN32(1/147.800537109375)

    const int rpw = a.tr_rows_per_warp;
    for (int rr = 0; rr < rpw; ++rr) {
        const int64_t i = ((int64_t)blockIdx.x * kWarps + warp) * rpw + rr;
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
            // row counts 1, 2, 4, 8 (a chunk of 3 runs as 4 with a row left
            // out): fewer unrolled copies of the loop keep the instruction
            // cache warm (measured 6-15 % faster than one copy per count)
            if (nt == 1)
                chunk_sums<KG, KU, 1>(a, grow, urow, tok, lmask, ag, au);
            else if (nt == 2)
                chunk_sums<KG, KU, 2>(a, grow, urow, tok, lmask, ag, au);
            else if (nt <= 4)
                chunk_sums<KG, KU, 4>(a, grow, urow, tok, lmask, ag, au);
            else
                chunk_sums<KG, KU, 8>(a, grow, urow, tok, lmask, ag, au);
            // lane m keeps the sums of chunk row m; one copy of the tail
            // then serves every row (the kernel is sensitive to the size of
            // its unrolled code: eight copies of the tail cost 3 %)
            float Gm = 0.0f, Um = 0.0f;
            int32_t tm = -1;
#pragma unroll
            for (int m = 0; m < kChunk; ++m) {
                if (m >= nt)                     // warp-uniform
                    break;
                const float G = warp_sum(ag[m]);
                const float U = warp_sum(au[m]);
                if (lane == m) {
                    Gm = G;
                    Um = U;
                    tm = tok[m];
                }
            }
            if (lane < nt && tm >= 0) {
                const float g32 = __fmul_rn(Gm, sg);
                const float u32 = __fmul_rn(Um, su);
                const int64_t o = (int64_t)(p0 + lane) * a.I + i;
                uint16_t sT, siluT;
                a.out[o] = a.tail_mlx
                               ? swiglu_tail_bits(a.sigmoid + kSigmoidTable,
                                                  bf16_rne(g32),
                                                  bf16_rne(u32), &sT, &siluT)
                               : swiglu_out(a.sigmoid, g32, u32);
                if (a.gate_f32)
                    a.gate_f32[o] = g32;
                if (a.up_f32)
                    a.up_f32[o] = u32;
            }
        }
    }
}

// Rows per warp: the most (up to 8, amortising each block's set-up) that
// still leave two blocks per SM for the experts of the call.
template <int KG, int KU>
cudaError_t launch_widths(const GateUpArgs &a0, cudaStream_t s) {
    GateUpArgs a = a0;
    int rpw = kMaxRowsPerWarp;
    while (rpw > 1 && (a.I + kWarps * rpw - 1) / (kWarps * rpw) * a.E <
                          2ll * a.num_sms)
        rpw /= 2;
    a.tr_rows_per_warp = rpw;
    const dim3 grid((unsigned)((a.I + kWarps * rpw - 1) / (kWarps * rpw)),
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
