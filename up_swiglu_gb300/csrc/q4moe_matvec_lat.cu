// q4moe_matvec_lat.cu -- the fused gate/up + SwiGLU for one expert and at
// most 8 grouped rows (single-sequence decode), laid out for latency.
//
// Same arithmetic as the page's matvec (page 52, streamed-experts.ts,
// GATE_UP_SOURCE): per row i, gate and up sums over k of (nibble - 8, or
// the signed byte) * x in f32, row scale, bf16 gate/up, SwiGLU tail.
//
// A call this small is bound by its chain of latencies, not by bandwidth:
// 6.3 MB of weights (H=4096, I=1536) stream in under 1 us at the measured
// copy bandwidth.  Each CTA takes R = ceil(I / SMs) consecutive
// intermediate rows.  Before the dependency wait the CTA asks L2 to
// prefetch its weight rows (a prefetch only warms L2, the point of
// coherence, so it is safe whatever the previous kernel writes); the
// previous call releases this one as soon as its own CTAs hold their
// operands, so that prefetch overlaps the previous call's arithmetic.
// Right after the dependency wait one thread of each of 14 warps (15 for
// the down projection) issues the bulk copies (cp.async.bulk) of a gate
// row and the matching up row (one thread issuing them all took 0.26 us
// longer per call) while a thread of another warp reads the token indices
// and issues one copy per activation row, the row offsets are checked
// beside them, and the threads that finish the rows load their scales.
//
// The products go to the tensor core, mma.sync m16n8k16 (bf16 in, f32
// accumulate).  The CTA's 2R weight rows (gate rows, then up rows) form m16
// tiles of the A operand, the grouped rows being the first M columns of B,
// and the last 2R mod 16 rows n8 tiles of the B operand, the grouped rows
// being the first M rows of A; both forms take the activations in the same
// registers.  Every warp takes every 16th 32-wide K slice.  A thread's
// 32-bit (Q4) or 64-bit (Q8) weight load holds the 8 consecutive K of its
// slot group; the slots of A and B are filled in the same K order (for Q4
// the pairs {k, k+4}, which one mask-and-or per pair builds: a nibble n
// under the bf16 exponent of 128.0 reads 128 + n, and one bf16x2
// subtraction of 136 gives n - 8, exactly), so every product is exact.
// The 16 warps' partial sums meet in shared memory and are added in warp
// order, so a row's result depends on its own activations only and is the
// same on every run.
//
// The arithmetic is bound by the issue port of each SM sub-partition: the
// integer steps issue at half rate and an mma.sync m16n8k16 takes 8 issue
// cycles.
//
// Every wait is bounded; on time-out the CTA raises Q4MOE_DEV_WAIT_TIMEOUT
// and stores nothing.  Row offsets other than {0, M} raise
// Q4MOE_DEV_BAD_ROW_OFFSETS and nothing is stored; a token index out of
// range raises Q4MOE_DEV_BAD_TOKEN and its row is computed from zeros.
#include <algorithm>

#include "q4moe_internal.cuh"
#include "q4moe_sm100.cuh"

namespace q4moe {
namespace {

using namespace sm100;

constexpr int kLatWarps = 16;
constexpr int kLatThreads = kLatWarps * 32;
constexpr int kLatMaxRows = 8;               // grouped rows per call
constexpr int kLatMaxTileRows = 32;          // weight rows per CTA
constexpr int kLatMaxM16 = 2;                // m16 tiles: 2R <= 32 rows
constexpr int kLatMaxN8 = 2;                 // n8 tiles: 2R mod 16 < 16

// Shared-memory row pitches.  A weight row starts 16 (Q4) or 32 (Q8) bytes
// past a 128-byte multiple of the previous one, so the 8 rows of a tile
// that a warp reads at once fall in different banks; an activation row
// starts 64 bytes past one, for the same reason across grouped rows.
__host__ __device__ __forceinline__ int64_t lat_row_pitch(int64_t rb,
                                                          bool q8) {
    return (rb + 127) / 128 * 128 + (q8 ? 32 : 16);
}
__host__ __device__ __forceinline__ int64_t lat_x_pitch(int64_t H) {
    return (H * 2 + 127) / 128 * 128 + 64;
}
__host__ __device__ __forceinline__ int lat_tile_rows(int NR) {
    return (NR + 7) & ~7;
}

// Bulk copy of `bytes` (a multiple of 16, both addresses 16-byte aligned)
// from global to shared memory, completion reported to *bar as bytes.
__device__ __forceinline__ void bulk_g2s(uint32_t dst, const void *src,
                                         uint32_t bytes, uint64_t *bar) {
    asm volatile(
        "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes "
        "[%0], [%1], %2, [%3];" ::"r"(dst),
        "l"(src), "r"(bytes), "r"(smem_u32(bar))
        : "memory");
}

// The row offsets of a call's one expert must be {0, M}: *bad = whether
// they are not (block 0 raises the status bit).
__device__ __forceinline__ void check_single_offsets(const GateUpArgs &a,
                                                     int M, int *bad) {
    const int32_t off0 = __ldg(a.row_offsets), off1 = __ldg(a.row_offsets + 1);
    const bool b = off0 != 0 || off1 != M;
    *bad = b;
    if (b && blockIdx.x == 0)
        atomicOr(a.status, Q4MOE_DEV_BAD_ROW_OFFSETS);
}

__device__ __forceinline__ uint32_t sub_bf16x2(uint32_t a, uint32_t b) {
    uint32_t r;
    asm("sub.rn.bf16x2 %0, %1, %2;" : "=r"(r) : "r"(a), "r"(b));
    return r;
}

// Q4: the pairs {n_j - 8, n_{j+4} - 8} (j = 0..3) of one packed word.
__device__ __forceinline__ void nibble_pairs(uint32_t w, uint32_t (&b)[4]) {
#pragma unroll
    for (int j = 0; j < 4; ++j) {
        uint32_t v;
        asm("lop3.b32 %0, %1, 0x000F000F, 0x43004300, 0xEA;"
            : "=r"(v)
            : "r"(w >> (4 * j)));
        b[j] = sub_bf16x2(v, 0x43084308u);
    }
}

// Q8: the pairs {b0, b1}, {b2, b3} of a word of four signed bytes.  Under
// the bf16 exponent byte 0x43 the low seven bits m of a byte read 128 + m
// and its sign bit turns that into 256 + 2m; subtracting 128 + 128 * sign
// leaves the byte's value, exactly (8 significant bits at most).
__device__ __forceinline__ void byte_pairs(uint32_t w, uint32_t &lo,
                                           uint32_t &hi) {
    const uint32_t t0 = __byte_perm(w, 0x43434343u, 0x4140);
    const uint32_t t1 = __byte_perm(w, 0x43434343u, 0x4342);
    lo = sub_bf16x2(t0 & 0x437F437Fu, t0 & 0x43804380u);
    hi = sub_bf16x2(t1 & 0x437F437Fu, t1 & 0x43804380u);
}

// n8 form: A = grouped rows (rows 8..15 zero), B = 8 weight rows.
__device__ __forceinline__ void mma_n8(float (&c)[4], uint32_t a0,
                                       uint32_t a2, uint32_t b0,
                                       uint32_t b1) {
    asm volatile(
        "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 "
        "{%0,%1,%2,%3}, {%4,%6,%5,%6}, {%7,%8}, {%0,%1,%2,%3};"
        : "+f"(c[0]), "+f"(c[1]), "+f"(c[2]), "+f"(c[3])
        : "r"(a0), "r"(a2), "r"(0u), "r"(b0), "r"(b1));
}

// m16 form: A = 16 weight rows, B = grouped rows as columns.
__device__ __forceinline__ void mma_m16(float (&c)[4], uint32_t a0,
                                        uint32_t a1, uint32_t a2,
                                        uint32_t a3, uint32_t b0,
                                        uint32_t b1) {
    asm volatile(
        "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 "
        "{%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, {%0,%1,%2,%3};"
        : "+f"(c[0]), "+f"(c[1]), "+f"(c[2]), "+f"(c[3])
        : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}

// The four bf16 pairs of one weight row's word(s) for K slice c: pairs 0,
// 1 for the slice's first 16-wide step, 2, 3 for its second.
template <bool kQ8>
__device__ __forceinline__ void weight_pairs(const uint8_t *row, bool ok,
                                             int c, int t, uint32_t (&b)[4]) {
    if (kQ8) {
        uint2 w = make_uint2(0u, 0u);
        if (ok)
            w = *reinterpret_cast<const uint2 *>(row + (size_t)c * 32 + t * 8);
        byte_pairs(w.x, b[0], b[1]);
        byte_pairs(w.y, b[2], b[3]);
    } else {
        uint32_t w = 0x88888888u;                // zero weights
        if (ok)
            w = *reinterpret_cast<const uint32_t *>(row + (size_t)c * 16 +
                                                    t * 4);
        nibble_pairs(w, b);
    }
}

template <bool kQ8, bool kDown, int kM>
__global__ void __launch_bounds__(kLatThreads, 1)
matvec_latency_kernel(GateUpArgs a, int R) {
    extern __shared__ __align__(128) uint8_t smem[];
    // weights [kMats R][row pitch] (gate rows, then up rows; the down
    // projection's rows), activations bf16 [kM][x pitch] (rows of x, or of
    // mid), partial sums f32 [warps][tile rows][kM], barriers.  For the
    // down projection H is its K and I its output rows.
    constexpr int kMats = kDown ? 1 : 2;
    const int64_t rb = weight_row_bytes(a, a.H);
    const int64_t rp = lat_row_pitch(rb, kQ8), xp = lat_x_pitch(a.H);
    const int H = (int)a.H, M = (int)a.M;
    const int i0 = blockIdx.x * R;
    const int nr = min(R, (int)a.I - i0);
    const int NR = kMats * R, V = lat_tile_rows(NR);
    uint8_t *w_sm = smem;
    uint8_t *x_sm = smem + (size_t)NR * rp;
    float *part = reinterpret_cast<float *>(x_sm + (size_t)kM * xp);
    uint64_t *bars = reinterpret_cast<uint64_t *>(
        part + (size_t)kLatWarps * V * kM);
    __shared__ int s_tok[kLatMaxRows];
    __shared__ int s_bad, s_bad_tok;
    __shared__ int s_abort;

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    if (tid < kMats * nr) {
        // L2 prefetch of the CTA's weight rows (gate row tid / 2 or up row)
        const int64_t row = i0 + tid / kMats;
        prefetch_l2(a.base + (tid % kMats ? a.up_w_off : a.gate_w_off) +
                        row * rb,
                    (uint32_t)rb);
    }
    if (tid == 0) {
        mbar_init(&bars[0], 1);
        mbar_init(&bars[1], 1);
        s_abort = 0;
        fence_mbar_init();
    }
    __syncthreads();
    grid_dependency_wait();

    // gate/up: warp 15 checks the offsets beside the activation copies
    // (measured 0.7 % faster); the down projection, whose activation rows
    // need no token lookup, checks them after issuing those copies and
    // keeps warp 15 issuing weight rows (0.9 % faster)
    constexpr int kIssuers = kDown ? kLatWarps - 1 : kLatWarps - 2;
    if (lane == 0 && warp != 1 && warp <= kIssuers) {
        // the weight rows (they need nothing else): lane 0 of warp 0 and
        // of warps 2..kIssuers issues the rows r = k mod kIssuers (k = 0
        // for warp 0, warp - 1 for the others; a gate row and its up row
        // together), the first one expecting all the bytes (the barrier's
        // count of bytes may run ahead of it)
        const int k = warp == 0 ? 0 : warp - 1;
        if (k == 0)
            mbar_arrive_expect_tx(&bars[0], (uint32_t)(nr * kMats * rb));
        for (int r = k; r < nr; r += kIssuers) {
            const int64_t row = i0 + r;
            bulk_g2s(smem_u32(w_sm + (size_t)r * rp),
                     a.base + a.gate_w_off + row * rb, (uint32_t)rb,
                     &bars[0]);
            if (!kDown)
                bulk_g2s(smem_u32(w_sm + (size_t)(R + r) * rp),
                         a.base + a.up_w_off + row * rb, (uint32_t)rb,
                         &bars[0]);
        }
    } else if (!kDown && tid == (kLatWarps - 1) * 32) {
        // the row offsets of the one expert must be {0, M} (checked beside
        // the copies: only the stores wait for the answer)
        check_single_offsets(a, M, &s_bad);
    } else if (tid == 32) {
        // the token of each grouped row (the down projection reads mid row
        // p), then its activations
        uint32_t xbytes = 0;
        int tok[kLatMaxRows], bad_tok = 0;
#pragma unroll
        for (int p = 0; p < kM; ++p) {
            tok[p] = p >= M ? -1 : kDown ? p : (int)row_token(a, p);
            s_tok[p] = tok[p];
            if (tok[p] >= 0)
                xbytes += (uint32_t)H * 2;
            else if (p < M)
                bad_tok = 1;
        }
        s_bad_tok = bad_tok;
        mbar_arrive_expect_tx(&bars[1], xbytes);
#pragma unroll
        for (int p = 0; p < kM; ++p)
            if (tok[p] >= 0)
                bulk_g2s(smem_u32(x_sm + (size_t)p * xp),
                         a.x + (int64_t)tok[p] * H, (uint32_t)H * 2,
                         &bars[1]);
        if (kDown)
            check_single_offsets(a, M, &s_bad);
    }
    // the thread that finishes (row r, grouped row p) loads r's scales
    const bool fin = tid < nr * M;
    const int fr = fin ? tid % nr : 0, fp = fin ? tid / nr : 0;
    float sg = 0.0f, su = 0.0f;
    if (fin) {
        sg = __ldg(reinterpret_cast<const float *>(a.base + a.gate_s_off) +
                   i0 + fr);
        if (!kDown)
            su = __ldg(reinterpret_cast<const float *>(a.base + a.up_s_off) +
                       i0 + fr);
    }
    __syncthreads();                         // s_tok, s_bad, s_bad_tok
    if (s_bad_tok) {
        // a grouped row whose token index is out of range (status raised)
        // is computed from zeros, as in the other kernels
        for (int p = 0; p < M; ++p)
            if (s_tok[p] < 0)
                for (int k = tid; k < H; k += kLatThreads)
                    reinterpret_cast<uint16_t *>(x_sm + (size_t)p * xp)[k] = 0;
        __syncthreads();
    }
    if (!wait_phase(&bars[0], 0, &s_abort, a.status) ||
        !wait_phase(&bars[1], 0, &s_abort, a.status)) {
        // (a time-out: the copies in flight land before the CTA exits)
        if (tid == 0) {
            drain_phase(&bars[0], 0);
            drain_phase(&bars[1], 0);
        }
        return;
    }
    // The next launch may start now (its CTAs only prefetch before their
    // own dependency wait).  Released at the start of the kernel instead,
    // the next call's CTAs crowded these SMs and a chain of calls ran 2.3x
    // slower; released after the arithmetic, 14% slower than never.  The
    // expert MLP's down stage holds it (hold_next: measured faster there).
    if (a.matvec_last && !a.hold_next)
        grid_launch_dependents();

    // thread (g, t) of the warp: in an m16 tile weight rows g and g + 8
    // (A) and grouped rows 2t, 2t + 1 (columns of the result); in an n8
    // tile grouped row g (A) and weight rows 2t, 2t + 1 of the result.  The
    // activations of grouped row g, slots 2t and 2t + 8 of each 16-wide K
    // step, serve both forms.
    const int g = lane >> 2, t = lane & 3;
    const int T16 = NR / 16, T8 = (V - 16 * T16) / 8;
    // weight row v of the tiles holds data (the last CTA has nr < R)
    auto row_ok = [&](int v) {
        return v < NR && (kDown || v < R ? v < nr : v - R < nr);
    };
    const uint8_t *mrow[kLatMaxM16][2], *nrow[kLatMaxN8];
    bool mok[kLatMaxM16][2], nok[kLatMaxN8];
#pragma unroll
    for (int q = 0; q < kLatMaxM16; ++q)
#pragma unroll
        for (int h = 0; h < 2; ++h) {
            const int v = 16 * q + 8 * h + g;
            mok[q][h] = q < T16 && row_ok(v);
            mrow[q][h] = w_sm + (size_t)(mok[q][h] ? v : 0) * rp;
        }
#pragma unroll
    for (int j = 0; j < kLatMaxN8; ++j) {
        const int v = 16 * T16 + 8 * j + g;
        nok[j] = j < T8 && row_ok(v);
        nrow[j] = w_sm + (size_t)(nok[j] ? v : 0) * rp;
    }
    float am[kLatMaxM16][4], an[kLatMaxN8][4];
#pragma unroll
    for (int q = 0; q < kLatMaxM16; ++q)
        am[q][0] = am[q][1] = am[q][2] = am[q][3] = 0.0f;
#pragma unroll
    for (int j = 0; j < kLatMaxN8; ++j)
        an[j][0] = an[j][1] = an[j][2] = an[j][3] = 0.0f;
    const uint8_t *xrow = x_sm + (size_t)g * xp + (size_t)t * 16;
    const int slices = H / 32;
#pragma unroll 2
    for (int c = warp; c < slices; c += kLatWarps) {
        // activations K = 32c + 8t .. + 7 of grouped row g
        uint32_t xe0 = 0, xe2 = 0, xo0 = 0, xo2 = 0;
        if (g < M) {
            const uint4 v = *reinterpret_cast<const uint4 *>(xrow + (size_t)c * 64);
            if (kQ8) {
                xe0 = v.x; xe2 = v.y; xo0 = v.z; xo2 = v.w;
            } else {
                xe0 = __byte_perm(v.x, v.z, 0x5410);     // {x0, x4}
                xe2 = __byte_perm(v.x, v.z, 0x7632);     // {x1, x5}
                xo0 = __byte_perm(v.y, v.w, 0x5410);     // {x2, x6}
                xo2 = __byte_perm(v.y, v.w, 0x7632);     // {x3, x7}
            }
        }
#pragma unroll
        for (int q = 0; q < kLatMaxM16; ++q) {
            if (q >= T16)
                break;
            uint32_t lo[4], hi[4];
            weight_pairs<kQ8>(mrow[q][0], mok[q][0], c, t, lo);
            weight_pairs<kQ8>(mrow[q][1], mok[q][1], c, t, hi);
            mma_m16(am[q], lo[0], hi[0], lo[1], hi[1], xe0, xe2);
            mma_m16(am[q], lo[2], hi[2], lo[3], hi[3], xo0, xo2);
        }
#pragma unroll
        for (int j = 0; j < kLatMaxN8; ++j) {
            if (j >= T8)
                break;
            uint32_t b[4];
            weight_pairs<kQ8>(nrow[j], nok[j], c, t, b);
            mma_n8(an[j], xe0, xe2, b[0], b[1]);
            mma_n8(an[j], xo0, xo2, b[2], b[3]);
        }
    }
    // accumulators -> partials [warp][tile row][grouped row]
    float *pw = part + (size_t)warp * V * kM;
#pragma unroll
    for (int q = 0; q < kLatMaxM16; ++q) {
        if (q >= T16)
            break;
        const int v = 16 * q + g;
#pragma unroll
        for (int u = 0; u < 2; ++u)
            if (2 * t + u < M) {
                pw[(size_t)v * kM + 2 * t + u] = am[q][u];
                pw[(size_t)(v + 8) * kM + 2 * t + u] = am[q][2 + u];
            }
    }
    if (g < M) {
#pragma unroll
        for (int j = 0; j < kLatMaxN8; ++j) {
            if (j >= T8)
                break;
            const int v = 16 * T16 + 8 * j + 2 * t;
            pw[(size_t)v * kM + g] = an[j][0];
            pw[(size_t)(v + 1) * kM + g] = an[j][1];
        }
    }
    __syncthreads();
    if (!fin || s_bad)
        return;
    const int64_t o = (int64_t)fp * a.I + i0 + fr;
    float gs = part[(size_t)fr * kM + fp];
#pragma unroll
    for (int w = 1; w < kLatWarps; ++w)
        gs = __fadd_rn(gs, part[((size_t)w * V + fr) * kM + fp]);
    const float g32 = __fmul_rn(gs, sg);
    if (kDown) {
        // the down projection: scale, one rounding
        a.out[o] = bf16_rne(g32);
        if (a.gate_f32)
            a.gate_f32[o] = g32;
        return;
    }
    float us = part[(size_t)(R + fr) * kM + fp];
#pragma unroll
    for (int w = 1; w < kLatWarps; ++w)
        us = __fadd_rn(us, part[((size_t)w * V + R + fr) * kM + fp]);
    const float u32 = __fmul_rn(us, su);
    a.out[o] = swiglu_out(a.sigmoid, g32, u32);
    if (a.gate_f32)
        a.gate_f32[o] = g32;
    if (a.up_f32)
        a.up_f32[o] = u32;
}

size_t lat_smem(const GateUpArgs &a, int R, int kM) {
    const int64_t rb = weight_row_bytes(a, a.H);
    const int NR = (a.down ? 1 : 2) * R;
    return (size_t)NR * lat_row_pitch(rb, a.q8) +
           (size_t)kM * lat_x_pitch(a.H) +
           (size_t)kLatWarps * lat_tile_rows(NR) * kM * sizeof(float) +
           2 * sizeof(uint64_t);
}

int lat_bucket(int64_t M) { return M <= 1 ? 1 : M <= 2 ? 2 : M <= 4 ? 4 : 8; }

int lat_rows(const GateUpArgs &a) {
    return (int)((a.I + a.num_sms - 1) / a.num_sms);
}

template <bool kQ8, bool kDown, int kM>
cudaError_t launch_m(const GateUpArgs &a, cudaStream_t s) {
    const int R = lat_rows(a);
    const size_t smem = lat_smem(a, R, kM);
    cudaError_t err = cudaFuncSetAttribute(
        matvec_latency_kernel<kQ8, kDown, kM>,
        cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (err != cudaSuccess)
        return err;
    const unsigned grid = (unsigned)((a.I + R - 1) / R);
    return launch_pdl(matvec_latency_kernel<kQ8, kDown, kM>, dim3(grid),
                      dim3(kLatThreads), smem, s, a, R);
}

template <bool kQ8, bool kDown>
cudaError_t launch_q(const GateUpArgs &a, cudaStream_t s) {
    switch (lat_bucket(a.M)) {
    case 1: return launch_m<kQ8, kDown, 1>(a, s);
    case 2: return launch_m<kQ8, kDown, 2>(a, s);
    case 4: return launch_m<kQ8, kDown, 4>(a, s);
    default: return launch_m<kQ8, kDown, 8>(a, s);
    }
}

}  // namespace

// One expert, 1..8 grouped rows, gate/up or down, slabs at base (no
// pointer table), whole 16-byte weight rows and activation rows (16-byte
// aligned), K a multiple of 32, at most 32 weight rows per CTA (16 of each
// gate/up matrix), all of them in shared memory.
bool matvec_latency_supported(const GateUpArgs &a) {
    const int64_t rb = weight_row_bytes(a, a.H);
    if (a.E != 1 || a.M < 1 || a.M > kLatMaxRows || a.invariant ||
        a.slab_ptrs != nullptr || a.H % 32 != 0 || rb % 16 != 0 ||
        a.gate_w_off % 16 != 0 || a.up_w_off % 16 != 0 ||
        (reinterpret_cast<uintptr_t>(a.base) & 15) != 0 ||
        (reinterpret_cast<uintptr_t>(a.x) & 15) != 0)
        return false;
    const int R = lat_rows(a);
    return (a.down ? 1 : 2) * R <= kLatMaxTileRows &&
           lat_smem(a, R, lat_bucket(a.M)) <= 200 * 1024;
}

cudaError_t launch_matvec_latency(const GateUpArgs &a, cudaStream_t s) {
    if (a.down)
        return a.q8 ? launch_q<true, true>(a, s) : launch_q<false, true>(a, s);
    return a.q8 ? launch_q<true, false>(a, s) : launch_q<false, false>(a, s);
}

}  // namespace q4moe
