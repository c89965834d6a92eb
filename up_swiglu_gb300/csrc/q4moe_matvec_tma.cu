// q4moe_matvec_tma.cu -- the grouped matvec for experts with few rows
// (decode and verify), its weight stream moved by the tensor memory
// accelerator.
//
// Same arithmetic as the page's matvec (page 52, streamed-experts.ts,
// GATE_UP_SOURCE): per expert, row scale, bf16 gate/up, SwiGLU tail.  Each
// packed word is read from HBM once per call and serves all of the expert's
// grouped rows, 8 at a time (a chunk).
//
// Work unit = (expert, chunk of <= 8 grouped rows, tile of NB blocks of 16
// intermediate rows), over the whole K.  One CTA of 16 warps per SM takes a
// contiguous range of units.  Warp w takes block b = w / P of the tile and
// K part kp = w % P (P = 16 / NB) and multiplies with mma.sync m16n8k16
// (f32 accumulate): A rows 0-7 = gate rows g, rows 8-15 = up rows g of the
// same intermediate row, B = the chunk's 8 rows of x, so a thread's C
// fragment pairs gate and up of one output.
// A pipeline stage is 32 KB: for both gate and up, P/2 TMA boxes of 128
// bytes (256 K) x 16*NB rows, 128-byte swizzled, so a stage covers 128*P of
// K and every warp one 128-wide K step of it.  A ring of D stages keeps the
// stream in flight: one producer thread refills each slot once all consumer
// threads have released it (measured: issuing a stage's boxes from several
// lanes at once gains nothing).
// Weights are dequantised in registers to f16: masking a word (or the word
// shifted by 8) with 0x000F000F or 0x00F000F0 under the exponent of 1024.0
// gives 1024 + n or 1024 + 16 n for the pairs {n_j, n_j+4}; one f16x2 fma
// maps them to n - 8.  The chunk's activations are staged once in shared
// memory in the matching K order ((0,4,1,5,2,6,3,7) within each group of
// 8), bank-swizzled, and converted to f16 under a power-of-two scale that
// keeps every value exact; when no scale can (an exponent span over 32, a
// subnormal, values at the ends of the range) the chunk stays bf16 and the
// weights are dequantised to bf16 instead.  Thread (g, tq) of K half h
// reads 16-byte chunk 2*tq + h of its box rows, which keeps both operand
// loads free of bank conflicts.  When P > 1 the K parts of a block meet in
// shared memory in a fixed order (results are deterministic and a row's
// bits do not depend on the other rows of its chunk), each block's parts
// at their own named barrier; with two parts each finishes half of the
// block's rows (scales and tail), otherwise part 0 finishes all of them.
// Measured on the grouped decode, splitting the tail and replacing the
// barrier of all 16 warps by the block's own took 0.2125 to 0.2030 ms.
//
// The down projection (page 52, DOWN_SOURCE) runs on the same kernel
// (kDown): one matrix, a tile of 32*NB output rows whose two halves take the
// places of gate and up (the second box starts 16*NB rows further down the
// same tensor map), x = the grouped intermediate rows themselves, and the
// tail is the row scale and one bf16 rounding per output.
//
// Every mbarrier wait is bounded; on time-out the CTA raises
// Q4MOE_DEV_WAIT_TIMEOUT, waits for its copies in flight and exits.
#include <cuda.h>
#include <cudaTypedefs.h>

#include <algorithm>
#include <cstring>

#include "q4moe_internal.cuh"
#include "q4moe_sm100.cuh"

namespace q4moe {

PFN_cuTensorMapEncodeTiled_v12000 tensor_map_encoder();  // q4moe_gemm.cu

namespace {

using namespace sm100;

constexpr int kWarps = 16;                   // consumer warps
constexpr int kCThreads = kWarps * 32;
constexpr int kThreads = kCThreads + 32;     // + the producer warp
constexpr int kTok = 8;                      // grouped rows per chunk
// K values per 32-bit word, per box row (128 bytes) and per consumer warp
// and stage (half a box row), for packed nibbles (Q4) or bytes (Q8)
template <bool kQ8> struct Fmt {
    static constexpr int kPerWord = kQ8 ? 4 : 8;
    static constexpr int kBoxK = 32 * kPerWord;
    static constexpr int kStepK = kBoxK / 2;
};
constexpr uint32_t kStageBytes = 32768;
constexpr int kMaxStages = 4;

__device__ __forceinline__ int ceil_div(int a, int b) { return (a + b - 1) / b; }

struct Unit {
    int e, chunk, tile;
    int p0, nt;                              // first grouped row, rows
};

__device__ __forceinline__ int units_of(int n_e, int max_rows, int NT) {
    return (n_e > 0 && n_e <= max_rows) ? ceil_div(n_e, kTok) * NT : 0;
}

// Unit u (expert-major, then chunk, then tile).
__device__ __forceinline__ Unit unit_of(int u, const int32_t *off,
                                        const int32_t *pre, int E, int NT) {
    int lo = 0, hi = E;
    while (hi - lo > 1) {
        const int mid = (lo + hi) >> 1;
        if (pre[mid] <= u)
            lo = mid;
        else
            hi = mid;
    }
    Unit t;
    t.e = lo;
    const int local = u - pre[lo];
    t.chunk = local / NT;
    t.tile = local - t.chunk * NT;
    t.p0 = off[lo] + t.chunk * kTok;
    t.nt = min(kTok, off[lo + 1] - t.p0);
    return t;
}

// Physical 16-byte chunk of K chunk q (8 values) of staged row n.  The low
// three bits are XORed with (bits 3-4 of q, bit 0 of n), so that the eight
// threads of a shared-memory phase (two rows n, four tq whose chunks are 8
// apart) hit eight different bank groups.
__device__ __forceinline__ int xs_chunk(int q, int n) {
    return q ^ ((((q >> 3) & 3) << 1) | (n & 1));
}

// Q8: the same role for the activations of a byte-weight stage, whose
// threads read chunks 4 apart (tq); the XOR keeps the eight threads of a
// shared-memory phase on eight different bank groups.
__device__ __forceinline__ int xs_chunk_q8(int q, int n) {
    return q ^ ((((q >> 2) & 3) << 1) | (n & 1));
}

template <bool kQ8>
__device__ __forceinline__ int xs_phys(int q, int n) {
    return kQ8 ? xs_chunk_q8(q, n) : xs_chunk(q, n);
}

// 8 consecutive 16-bit values (uint4) -> K order (0,4,1,5,2,6,3,7).
__device__ __forceinline__ uint4 permute8(uint4 v) {
    return make_uint4(__byte_perm(v.x, v.z, 0x5410),
                      __byte_perm(v.x, v.z, 0x7632),
                      __byte_perm(v.y, v.w, 0x5410),
                      __byte_perm(v.y, v.w, 0x7632));
}

// The four pairs {n_j - 8, n_{j+4} - 8}, j = 0..3, of one packed word, as
// bf16x2 (nibble in the mantissa of 128.0, minus 136).
__device__ __forceinline__ void word_pairs_bf16(uint32_t w, uint32_t (&r)[4]) {
#pragma unroll
    for (int j = 0; j < 4; ++j) {
        const uint32_t v = ((w >> (4 * j)) & 0x000F000Fu) | 0x43004300u;
        __nv_bfloat162 b = *reinterpret_cast<const __nv_bfloat162 *>(&v);
        b = __hsub2(b, __halves2bfloat162(__ushort_as_bfloat16(0x4308),
                                          __ushort_as_bfloat16(0x4308)));
        r[j] = *reinterpret_cast<const uint32_t *>(&b);
    }
}

// (a & m) | o in one logic operation.
__device__ __forceinline__ uint32_t and_or(uint32_t a, uint32_t m, uint32_t o) {
    uint32_t r;
    asm("lop3.b32 %0, %1, %2, %3, 0xEA;" : "=r"(r) : "r"(a), "r"(m), "r"(o));
    return r;
}

__device__ __forceinline__ uint32_t fma_f16x2(uint32_t a, uint32_t b,
                                              uint32_t c) {
    uint32_t r;
    asm("fma.rn.f16x2 %0, %1, %2, %3;" : "=r"(r) : "r"(a), "r"(b), "r"(c));
    return r;
}

// The same four pairs as f16x2, in the same order.  f16 keeps ten mantissa
// bits, so both nibbles of a byte fit under the exponent of 1024.0: masking
// w (or w >> 8) with 0x000F000F gives 1024 + n, with 0x00F000F0 gives
// 1024 + 16 n; one f16x2 fma maps them to n - 8 (x 1 - 1032, and
// x 1/16 - 72).  Every value is a small integer, so each step is exact.
__device__ __forceinline__ void word_pairs_f16(uint32_t w, uint32_t (&r)[4]) {
    const uint32_t kMagic = 0x64006400u;           // 1024.0
    const uint32_t kOne = 0x3C003C00u, kLo = 0xE408E408u;    // 1, -1032
    const uint32_t kSixteenth = 0x2C002C00u, kHi = 0xD480D480u;  // 1/16, -72
    const uint32_t w8 = w >> 8;
    r[0] = fma_f16x2(and_or(w, 0x000F000Fu, kMagic), kOne, kLo);
    r[1] = fma_f16x2(and_or(w, 0x00F000F0u, kMagic), kSixteenth, kHi);
    r[2] = fma_f16x2(and_or(w8, 0x000F000Fu, kMagic), kOne, kLo);
    r[3] = fma_f16x2(and_or(w8, 0x00F000F0u, kMagic), kSixteenth, kHi);
}

template <bool kF16>
__device__ __forceinline__ void mma_16816(float (&c)[4], uint32_t a0,
                                          uint32_t a1, uint32_t a2,
                                          uint32_t a3, uint32_t b0,
                                          uint32_t b1) {
    if (kF16)
        asm volatile(
            "mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 "
            "{%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, {%0,%1,%2,%3};"
            : "+f"(c[0]), "+f"(c[1]), "+f"(c[2]), "+f"(c[3])
            : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
    else
        asm volatile(
            "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 "
            "{%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, {%0,%1,%2,%3};"
            : "+f"(c[0]), "+f"(c[1]), "+f"(c[2]), "+f"(c[3])
            : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}

// One K step: w[0..3] = 16 bytes of gate row g, up row g, gate row 8+g,
// up row 8+g; xb = the matching four 16-byte activation chunks (f16 or
// bf16, like the weights).
template <bool kF16>
__device__ __forceinline__ void step_mma(float (&acc)[2][4],
                                         const uint4 (&w)[4],
                                         const uint4 (&xb)[4]) {
    const uint32_t *wg0 = reinterpret_cast<const uint32_t *>(&w[0]);
    const uint32_t *wu0 = reinterpret_cast<const uint32_t *>(&w[1]);
    const uint32_t *wg1 = reinterpret_cast<const uint32_t *>(&w[2]);
    const uint32_t *wu1 = reinterpret_cast<const uint32_t *>(&w[3]);
#pragma unroll
    for (int wd = 0; wd < 4; ++wd) {
        uint32_t g0[4], u0[4], g1[4], u1[4];
        if (kF16) {
            word_pairs_f16(wg0[wd], g0);
            word_pairs_f16(wu0[wd], u0);
            word_pairs_f16(wg1[wd], g1);
            word_pairs_f16(wu1[wd], u1);
        } else {
            word_pairs_bf16(wg0[wd], g0);
            word_pairs_bf16(wu0[wd], u0);
            word_pairs_bf16(wg1[wd], g1);
            word_pairs_bf16(wu1[wd], u1);
        }
        const uint32_t *xw = reinterpret_cast<const uint32_t *>(&xb[wd]);
#pragma unroll
        for (int h = 0; h < 2; ++h) {
            mma_16816<kF16>(acc[0], g0[2 * h], u0[2 * h], g0[2 * h + 1],
                            u0[2 * h + 1], xw[2 * h], xw[2 * h + 1]);
            mma_16816<kF16>(acc[1], g1[2 * h], u1[2 * h], g1[2 * h + 1],
                            u1[2 * h + 1], xw[2 * h], xw[2 * h + 1]);
        }
    }
}

// The two pairs {b0, b1}, {b2, b3} of a word of four signed bytes, as f16x2
// (exact): with the sign bits flipped each byte is b + 128, placed under the
// exponent of 1024.0 it reads 1152 + b, and one fma subtracts 1152.
__device__ __forceinline__ void byte_pairs_f16(uint32_t w, uint32_t (&r)[2]) {
    const uint32_t t = w ^ 0x80808080u;
    const uint32_t kOne = 0x3C003C00u, kM1152 = 0xE480E480u;   // 1, -1152
    r[0] = fma_f16x2(__byte_perm(t, 0x64646464u, 0x5140), kOne, kM1152);
    r[1] = fma_f16x2(__byte_perm(t, 0x64646464u, 0x7362), kOne, kM1152);
}

// The same pairs as bf16x2, exact: under the bf16 exponent byte 0x43 the
// low seven bits m of a byte read 128 + m and its sign bit 128 or 256, and
// b = (128 + m) - (128 + 128 * sign) is exact in bf16 (at most 8 bits).
__device__ __forceinline__ void byte_pairs_bf16(uint32_t w, uint32_t (&r)[2]) {
#pragma unroll
    for (int j = 0; j < 2; ++j) {
        const uint32_t t = __byte_perm(w, 0x43434343u, j ? 0x4342 : 0x4140);
        const uint32_t m = t & 0x437F437Fu, c = t & 0x43804380u;
        const __nv_bfloat162 d =
            __hsub2(*reinterpret_cast<const __nv_bfloat162 *>(&m),
                    *reinterpret_cast<const __nv_bfloat162 *>(&c));
        r[j] = *reinterpret_cast<const uint32_t *>(&d);
    }
}

// One Q8 K step: w[0..3] = 16 bytes (16 K) of gate row g, up row g, gate
// row 8+g, up row 8+g; xb = the matching two 16-byte activation chunks
// (natural K order).  One mma per word and row pair.
template <bool kF16>
__device__ __forceinline__ void step_mma_q8(float (&acc)[2][4],
                                            const uint4 (&w)[4],
                                            const uint4 (&xb)[2]) {
    const uint32_t *wg0 = reinterpret_cast<const uint32_t *>(&w[0]);
    const uint32_t *wu0 = reinterpret_cast<const uint32_t *>(&w[1]);
    const uint32_t *wg1 = reinterpret_cast<const uint32_t *>(&w[2]);
    const uint32_t *wu1 = reinterpret_cast<const uint32_t *>(&w[3]);
    const uint32_t *xw = reinterpret_cast<const uint32_t *>(&xb[0]);
#pragma unroll
    for (int wd = 0; wd < 4; ++wd) {
        uint32_t g0[2], u0[2], g1[2], u1[2];
        if (kF16) {
            byte_pairs_f16(wg0[wd], g0);
            byte_pairs_f16(wu0[wd], u0);
            byte_pairs_f16(wg1[wd], g1);
            byte_pairs_f16(wu1[wd], u1);
        } else {
            byte_pairs_bf16(wg0[wd], g0);
            byte_pairs_bf16(wu0[wd], u0);
            byte_pairs_bf16(wg1[wd], g1);
            byte_pairs_bf16(wu1[wd], u1);
        }
        mma_16816<kF16>(acc[0], g0[0], u0[0], g0[1], u0[1], xw[2 * wd],
                        xw[2 * wd + 1]);
        mma_16816<kF16>(acc[1], g1[0], u1[0], g1[1], u1[1], xw[2 * wd],
                        xw[2 * wd + 1]);
    }
}

// bf16 pair -> f16 pair, both scaled by 2^s (s such that the result is a
// normal f32 below 2^16 for every nonzero half, checked by the caller):
// the exponent field is raised by s, then rounded to f16, exactly.
__device__ __forceinline__ uint32_t bf16x2_to_f16x2(uint32_t v, int s) {
    uint32_t lo = v << 16, hi = v & 0xFFFF0000u;
    if (lo & 0x7FFFFFFFu)
        lo += (uint32_t)s << 23;
    if (hi & 0x7FFFFFFFu)
        hi += (uint32_t)s << 23;
    __half2 h = __floats2half2_rn(__uint_as_float(lo), __uint_as_float(hi));
    return *reinterpret_cast<const uint32_t *>(&h);
}

// Exponent fields of the nonzero bf16 halves of v: running max, min, and a
// flag for subnormals.
__device__ __forceinline__ void exp_range(uint32_t v, int &emax, int &emin,
                                          int &sub) {
#pragma unroll
    for (int k = 0; k < 2; ++k) {
        const uint32_t h = (v >> (16 * k)) & 0xFFFFu;
        const int e = (int)((h >> 7) & 0xFFu);
        if (h & 0x7FFFu) {
            sub |= (e == 0);
            emax = max(emax, e);
            emin = min(emin, e);
        }
    }
}

// Bounded mbarrier wait: the common case (already complete) inline, the
// polling loop out of line.
__device__ __forceinline__ bool wait_full(uint64_t *bar, uint32_t parity,
                                          volatile int *abort,
                                          unsigned int *status) {
    return mbar_try_wait(bar, parity) ||
           wait_phase(bar, parity, abort, status);
}

// Barrier of the 16 consumer warps only (the producer keeps issuing).
__device__ __forceinline__ void consumer_sync() {
    asm volatile("bar.sync 1, %0;" ::"n"(kCThreads) : "memory");
}

// Barrier of the P K-part warps of block b: named barrier 2 + b (the
// consumer barrier itself when one block spans all of them).
template <int P>
__device__ __forceinline__ void group_sync(int b) {
    if (P == kWarps)
        consumer_sync();
    else
        asm volatile("bar.sync %0, %1;" ::"r"(2 + b), "n"(32 * P) : "memory");
}

// Unit u of a call with one expert: the rows follow from M alone.
__device__ __forceinline__ Unit unit_single(int u, int M, int NT) {
    Unit t;
    t.e = 0;
    t.chunk = u / NT;
    t.tile = u - t.chunk * NT;
    t.p0 = t.chunk * kTok;
    t.nt = min(kTok, M - t.p0);
    return t;
}

// Shared memory after the 1024-byte aligned ring: staged x, reduction
// buffer, barriers, per-warp exponent ranges, row offsets and unit prefix,
// abort flag, stage count.
__host__ __device__ __forceinline__ size_t red_bytes(int NB) {
    return (size_t)(kWarps - NB) * 32 * 2 * 16;
}

template <int NB, bool kDown, bool kQ8>
__global__ void __launch_bounds__(kThreads, 1)
matvec_tma_kernel(GateUpArgs a, const __grid_constant__ CUtensorMap tm_gate,
                  const __grid_constant__ CUtensorMap tm_up, int tok_cap,
                  int D) {
    constexpr int kPerWord = Fmt<kQ8>::kPerWord;
    constexpr int kBoxK = Fmt<kQ8>::kBoxK;
    constexpr int kStepK = Fmt<kQ8>::kStepK;
    constexpr int P = kWarps / NB;           // K parts per block
    constexpr int kBoxes = P / 2;            // boxes per matrix per stage
    constexpr int kRows = NB * 16;           // rows per box
    constexpr uint32_t kBoxBytes = kRows * 128;
    // output rows per tile, and the first row of the second ("up") half
    constexpr int kTileRows = kDown ? 2 * kRows : kRows;
    constexpr int kHiRow = kDown ? kRows : 0;
    static_assert(2 * kBoxes * kBoxBytes == kStageBytes, "stage size");

    extern __shared__ uint8_t smem_raw[];
    const uint32_t raw_u32 = smem_u32(smem_raw);
    uint8_t *ring = smem_raw + (((raw_u32 + 1023u) & ~1023u) - raw_u32);
    const int E = a.E;
    const int H = (int)a.H;
    uint8_t *xs = ring + (size_t)D * kStageBytes;
    float4 *red = reinterpret_cast<float4 *>(xs + (size_t)tok_cap * H * 2);
    uint64_t *full = reinterpret_cast<uint64_t *>(
        reinterpret_cast<uint8_t *>(red) + red_bytes(NB));
    uint64_t *empty = full + kMaxStages;
    int4 *s_erange = reinterpret_cast<int4 *>(empty + kMaxStages);
    int32_t *s_off = reinterpret_cast<int32_t *>(s_erange + kWarps);
    int32_t *s_pre = s_off + (E + 1);
    volatile int *abort_flag = reinterpret_cast<volatile int *>(s_pre + E + 1);
    int *s_issued = const_cast<int *>(abort_flag) + 1;

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int g = lane >> 2, tq = lane & 3;
    const int NT = ceil_div((int)a.I, kTileRows);  // tiles per chunk
    const int nst = ceil_div(H, P * kStepK); // stages per unit

    if (warp == kWarps && lane == 0) {
        for (int d = 0; d < D; ++d) {
            mbar_init(&full[d], 1);
            mbar_init(&empty[d], kCThreads);
        }
        *abort_flag = 0;
        *s_issued = 0;
        fence_mbar_init();
        tma_desc_prefetch(&tm_gate);
        tma_desc_prefetch(&tm_up);
    }
    __shared__ int s_single_bad;             // one expert: offsets != {0, M}
    __syncthreads();                         // barriers initialised
    if (a.matvec_last)
        grid_launch_dependents();
    grid_dependency_wait();

    int u0 = 0, u1 = 0;
    // One expert: the units, and each unit's rows, follow from M; thread 0
    // loads the two offsets now and checks them before the first store
    // (an inconsistent pair stores nothing), so no block-wide barrier or
    // dependent load stands between the dependency release and the work.
    int32_t off_lo = 0, off_hi = 0;
    if (E == 1) {
        const unsigned nunits = (unsigned)(ceil_div((int)a.M, kTok) * NT);
        const unsigned G = gridDim.x, bb = blockIdx.x, q = nunits / G,
                       r = nunits - q * G;
        u0 = (int)(bb * q + min(bb, r));
        u1 = u0 + (int)q + (bb < r ? 1 : 0);
        if (tid == 0) {
            off_lo = __ldg(a.row_offsets);
            off_hi = __ldg(a.row_offsets + 1);
        }
    } else if (stage_row_offsets(a, s_off)) {  // (synchronises the block)
        const int32_t mvmax = matvec_limit(a, s_off);
        if (warp == 0) {
            const int per = ceil_div(E, 32);
            const int e0 = lane * per;
            int sum = 0;
            for (int e = e0; e < min(E, e0 + per); ++e)
                sum += units_of(s_off[e + 1] - s_off[e], mvmax, NT);
            int incl = sum;
#pragma unroll
            for (int d = 1; d < 32; d <<= 1) {
                const int v = __shfl_up_sync(0xffffffffu, incl, d);
                if (lane >= d)
                    incl += v;
            }
            int run = incl - sum;
            for (int e = e0; e < min(E, e0 + per); ++e) {
                s_pre[e] = run;
                run += units_of(s_off[e + 1] - s_off[e], mvmax, NT);
            }
            if (lane == 31)
                s_pre[E] = incl;
        }
        __syncthreads();
        // balanced contiguous ranges: the first nunits % G CTAs take one
        // unit more
        const unsigned nunits = (unsigned)s_pre[E], G = gridDim.x;
        const unsigned b = blockIdx.x, q = nunits / G, r = nunits - q * G;
        u0 = (int)(b * q + min(b, r));
        u1 = u0 + (int)q + (b < r ? 1 : 0);
    }
    if (warp == kWarps) {
        // ---- producer: the CTA's stages in order, stage j into slot
        // j % D once every consumer thread has released stage j - D
        if (lane == 0) {
            int j = 0;
            bool ok = true;
            for (int u = u0; u < u1 && ok; ++u) {
                int e, tile;
                if (E == 1) {
                    e = 0;
                    tile = u % NT;
                } else {
                    const Unit t = unit_of(u, s_off, s_pre, E, NT);
                    e = t.e;
                    tile = t.tile;
                }
                const int row0 = tile * kTileRows;
                // the down projection's second half may lie past the last
                // row: not loaded (its stale slot is never stored)
                const bool hi = !kDown || row0 + kHiRow < (int)a.I;
                for (int st = 0; st < nst; ++st, ++j) {
                    const int slot = j % D;
                    if (j >= D && !wait_full(&empty[slot], (j / D - 1) & 1,
                                             abort_flag, a.status)) {
                        ok = false;
                        break;
                    }
                    const int k0 = st * P * kStepK;
                    const int nbox = min(kBoxes, ceil_div(H - k0, kBoxK));
                    mbar_arrive_expect_tx(&full[slot],
                                          (hi ? 2u : 1u) * nbox * kBoxBytes);
                    const uint32_t dst = smem_u32(ring) + slot * kStageBytes;
                    for (int bx = 0; bx < nbox; ++bx) {
                        const int c0 = (k0 + bx * kBoxK) / kPerWord;
                        tma_load_3d(dst + bx * kBoxBytes, &tm_gate, c0, row0,
                                    e, &full[slot]);
                        if (hi)
                            tma_load_3d(dst + (kBoxes + bx) * kBoxBytes,
                                        &tm_up, c0, row0 + kHiRow, e,
                                        &full[slot]);
                    }
                }
            }
            *s_issued = j;
        }
        __syncwarp();
    } else {
        // ---- consumers
        const int b = warp / P, kp = warp - b * P;
        const int bx = kp >> 1, h = kp & 1;
        const int xrow = min(g, tok_cap - 1);    // rows past the chunk read a
                                                 // stale row; never stored
        const int xsw = (tq << 1) | (xrow & 1);
        // the thread's activations: K from (2 tq + h) * kStepK / 4 within a
        // box row, in 16-byte chunks of the row staged at xrow
        const uint8_t *xbase = xs + (size_t)xrow * H * 2 +
                               (kQ8 ? (tq >> 1) : tq) * 128;
        const int wc = ((2 * tq + h) ^ g) << 4;  // swizzled chunk in a row
        const int r0 = b * 16 + g;
        int staged_e = -1, staged_chunk = -1;
        // rows i of the block this warp finishes: with two K parts each
        // takes one half, else part 0 takes both
        const bool own0 = kp == 0;
        const bool own1 = P == 2 ? kp == 1 : kp == 0;
        bool xf16 = false;
        float unscale = 1.0f;
        int j = 0;                               // stage counter
        bool ok = true;
        Unit t;
        t.e = -1;
        t.tile = NT;
        for (int u = u0; u < u1 && ok; ++u) {
            // several experts: the next tile of the same chunk without a
            // search (a single-block tile or one expert finds every unit
            // afresh: measured faster there)
            if (NB > 1 && E > 1 && t.e >= 0 && t.tile + 1 < NT)
                ++t.tile;
            else
                t = E == 1 ? unit_single(u, (int)a.M, NT)
                           : unit_of(u, s_off, s_pre, E, NT);
            const int rbase = t.tile * kTileRows + b * 16;  // block's 1st row
            const bool live = rbase < (int)a.I;
            const bool live_hi = kDown ? rbase + kHiRow < (int)a.I : live;
            const uint8_t *slab = a.base + (int64_t)t.e * a.stride;
            const float *gs_row = reinterpret_cast<const float *>(
                                      slab + a.gate_s_off) + rbase + g;
            const float *us_row = reinterpret_cast<const float *>(
                                      slab + a.up_s_off) + rbase + kHiRow + g;
            float sg[2] = {0.f, 0.f}, su[2] = {0.f, 0.f};
            if (live) {                          // in flight during the K loop
                if (own0)
                    sg[0] = gs_row[0];
                if (own1)
                    sg[1] = gs_row[8];
            }
            if (live_hi) {
                if (own0)
                    su[0] = us_row[0];
                if (own1)
                    su[1] = us_row[8];
            }
            if (t.e != staged_e || t.chunk != staged_chunk) {
                // stage the chunk's rows of x (K order (0,4,1,5,2,6,3,7) per 8,
                // swizzled) and find their exponent range
                consumer_sync();                 // all done with the old x
                const int qn = H / 8;
                int emax = 0, emin = 255, sub = 0;
                for (int idx = tid; idx < t.nt * qn; idx += kCThreads) {
                    const int n = idx / qn, q = idx - n * qn;
                    const int64_t tok =
                        kDown ? (int64_t)(t.p0 + n) : row_token(a, t.p0 + n);
                    uint4 v = make_uint4(0, 0, 0, 0);
                    if (tok >= 0)
                        v = __ldg(reinterpret_cast<const uint4 *>(a.x + tok * a.H) +
                                  q);
                    exp_range(v.x, emax, emin, sub);
                    exp_range(v.y, emax, emin, sub);
                    exp_range(v.z, emax, emin, sub);
                    exp_range(v.w, emax, emin, sub);
                    *reinterpret_cast<uint4 *>(xs + (size_t)n * H * 2 +
                                               xs_phys<kQ8>(q, n) * 16) =
                        kQ8 ? v : permute8(v);
                }
#pragma unroll
                for (int d = 16; d > 0; d >>= 1) {
                    emax = max(emax, __shfl_xor_sync(0xffffffffu, emax, d));
                    emin = min(emin, __shfl_xor_sync(0xffffffffu, emin, d));
                    sub |= __shfl_xor_sync(0xffffffffu, sub, d);
                }
                if (lane == 0)
                    s_erange[warp] = make_int4(emax, emin, sub, 0);
                consumer_sync();
                for (int w2 = 0; w2 < kWarps; ++w2) {
                    const int4 rr = s_erange[w2];
                    emax = max(emax, rr.x);
                    emin = min(emin, rr.y);
                    sub |= rr.z;
                }
                // f16 under the scale 2^s, s = 142 - emax, holds every nonzero
                // value exactly when all exponent fields lie within 32 of the
                // largest (values at most 2^15 * 1.99, lowest bit at least
                // 2^-24) and none is subnormal; else the chunk stays bf16.
                // All-zero rows: f16, s = 0.
                const int sc = emax == 0 ? 0 : 142 - emax;
                xf16 = !sub && (emax == 0 || (emax - emin <= 32 && sc >= -100 &&
                                              sc <= 100));
                unscale = xf16 ? __uint_as_float((uint32_t)(127 - sc) << 23)
                               : 1.0f;
                if (xf16) {
                    for (int idx = tid; idx < t.nt * qn; idx += kCThreads) {
                        const int n = idx / qn, q = idx - n * qn;
                        uint4 *p = reinterpret_cast<uint4 *>(
                            xs + (size_t)n * H * 2 + xs_phys<kQ8>(q, n) * 16);
                        const uint4 v = *p;
                        *p = make_uint4(bf16x2_to_f16x2(v.x, sc),
                                        bf16x2_to_f16x2(v.y, sc),
                                        bf16x2_to_f16x2(v.z, sc),
                                        bf16x2_to_f16x2(v.w, sc));
                    }
                }
                staged_e = t.e;
                staged_chunk = t.chunk;
                consumer_sync();
            }
            float acc[2][4];
#pragma unroll
            for (int i = 0; i < 2; ++i)
                acc[i][0] = acc[i][1] = acc[i][2] = acc[i][3] = 0.0f;

            // The unit's K stages.
            auto k_loop = [&]() -> bool {
                for (int st = 0; st < nst; ++st, ++j) {
                    const int slot = j % D;
                    if (!wait_full(&full[slot], (j / D) & 1, abort_flag,
                                   a.status))
                        return false;
                    const int kb = st * P * kStepK + bx * kBoxK;
                    if (live && kb < H) {
                        const uint8_t *wb =
                            ring + slot * kStageBytes + bx * kBoxBytes;
                        const uint8_t *ub = wb + kBoxes * kBoxBytes;
                        uint4 w[4];
                        w[0] = *reinterpret_cast<const uint4 *>(wb + r0 * 128 + wc);
                        w[1] = *reinterpret_cast<const uint4 *>(ub + r0 * 128 + wc);
                        w[2] = *reinterpret_cast<const uint4 *>(
                            wb + (r0 + 8) * 128 + wc);
                        w[3] = *reinterpret_cast<const uint4 *>(
                            ub + (r0 + 8) * 128 + wc);
                        const uint8_t *xk = xbase + kb * 2;
                        if (kQ8) {
                            uint4 xb[2];
#pragma unroll
                            for (int jj = 0; jj < 2; ++jj)
                                xb[jj] = *reinterpret_cast<const uint4 *>(
                                    xk + (((4 * (tq & 1) + 2 * h + jj) ^ xsw)
                                          << 4));
                            if (xf16)
                                step_mma_q8<true>(acc, w, xb);
                            else
                                step_mma_q8<false>(acc, w, xb);
                        } else {
                            uint4 xb[4];
#pragma unroll
                            for (int wd = 0; wd < 4; ++wd)
                                xb[wd] = *reinterpret_cast<const uint4 *>(
                                    xk + (((4 * h + wd) ^ xsw) << 4));
                            if (xf16)
                                step_mma<true>(acc, w, xb);
                            else
                                step_mma<false>(acc, w, xb);
                        }
                    }
                    mbar_arrive(&empty[slot]);   // this thread's reads are done
                }
                return true;
            };
            // once any warp has timed out every warp leaves before the next
            // barrier (a warp past its last wait would otherwise meet a
            // barrier the others never reach)
            ok = k_loop() && !*abort_flag;
            if (!ok)
                break;
            // the unit is complete: sum the K parts of each block in order
            // at their block's own barrier (one expert: the offsets' check
            // reaches every warp before the first store)
            if (E == 1 && tid == 0 && u == u0) {
                const bool bad = off_lo != 0 || off_hi != (int32_t)a.M;
                s_single_bad = bad;
                if (bad && blockIdx.x == 0)
                    atomicOr(a.status, Q4MOE_DEV_BAD_ROW_OFFSETS);
            }
            static_assert(P > 1, "every block has K parts to reduce");
            if (NB > 1 && E == 1 && u == u0)    // the blocks' barriers
                consumer_sync();                 // do not reach every warp
            if (P == 2) {
                // each part hands its partner the rows the partner
                // finishes (rows g for part 0, 8 + g for part 1) and forms
                // part 0 + part 1 of its own; the second barrier keeps the
                // next unit's writes off the buffer until both have read
                red[(b * 2 + kp) * 32 + lane] =
                    kp == 0 ? make_float4(acc[1][0], acc[1][1], acc[1][2],
                                          acc[1][3])
                            : make_float4(acc[0][0], acc[0][1], acc[0][2],
                                          acc[0][3]);
                group_sync<P>(b);
                const float4 v = red[(b * 2 + 1 - kp) * 32 + lane];
                if (kp == 0) {
                    acc[0][0] += v.x;
                    acc[0][1] += v.y;
                    acc[0][2] += v.z;
                    acc[0][3] += v.w;
                } else {
                    acc[1][0] = v.x + acc[1][0];
                    acc[1][1] = v.y + acc[1][1];
                    acc[1][2] = v.z + acc[1][2];
                    acc[1][3] = v.w + acc[1][3];
                }
                group_sync<P>(b);
            } else {
                if (kp != 0) {
                    const int ri = (b * (P - 1) + kp - 1) * 32 + lane;
                    red[ri * 2] = make_float4(acc[0][0], acc[0][1], acc[0][2],
                                              acc[0][3]);
                    red[ri * 2 + 1] = make_float4(acc[1][0], acc[1][1], acc[1][2],
                                                  acc[1][3]);
                }
                group_sync<P>(b);
                if (kp == 0) {
                    for (int w2 = 1; w2 < P; ++w2) {
                        const int ri = (b * (P - 1) + w2 - 1) * 32 + lane;
#pragma unroll
                        for (int i = 0; i < 2; ++i) {
                            const float4 v = red[ri * 2 + i];
                            acc[i][0] += v.x;
                            acc[i][1] += v.y;
                            acc[i][2] += v.z;
                            acc[i][3] += v.w;
                        }
                    }
                }
                group_sync<P>(b);
            }
            if ((own0 || own1) && live && !(E == 1 && s_single_bad)) {
#pragma unroll
                for (int i = 0; i < 2; ++i) {
                    if (!(i == 0 ? own0 : own1))
                        continue;
                    const int64_t row = (int64_t)rbase + 8 * i + g;
#pragma unroll
                    for (int jj = 0; jj < 2; ++jj) {
                        const int n = 2 * tq + jj;
                        if (n < t.nt) {
                            // undo the staging scale (a power of two: exact)
                            const float g32 = __fmul_rn(
                                __fmul_rn(acc[i][jj], unscale), sg[i]);
                            const float u32 = __fmul_rn(
                                __fmul_rn(acc[i][2 + jj], unscale), su[i]);
                            const int64_t o = (int64_t)(t.p0 + n) * a.I + row;
                            if (kDown) {
                                a.out[o] = bf16_rne(g32);
                                if (a.gate_f32)
                                    a.gate_f32[o] = g32;
                                if (live_hi) {
                                    a.out[o + kHiRow] = bf16_rne(u32);
                                    if (a.gate_f32)
                                        a.gate_f32[o + kHiRow] = u32;
                                }
                            } else {
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
        }
    }
    __syncthreads();
    // copies still in flight (only after a time-out): the last D issued
    if (tid == 0 && *abort_flag) {
        const int issued = *s_issued;
        for (int j = max(0, issued - D); j < issued; ++j)
            drain_phase(&full[j % D], (j / D) & 1);
    }
}

size_t tma_smem(const GateUpArgs &a, int NB, int D, int tok_cap) {
    return 1024 + (size_t)D * kStageBytes + (size_t)tok_cap * a.H * 2 +
           red_bytes(NB) + 2 * kMaxStages * sizeof(uint64_t) +
           kWarps * sizeof(int4) + sizeof(int32_t) * 2 * (size_t)(a.E + 1) +
           2 * sizeof(int);
}

constexpr size_t kSmemLimit = 227 * 1024 - 1024;  // room for static smem

// Weights of one section (gate or up) of every expert as a 3-D tensor of
// 32-bit words: {H/8 words, I rows, E experts}; boxes of 32 words (128
// bytes, the swizzle span) x `rows` rows of one expert.
cudaError_t encode_weight_map(const GateUpArgs &a, int64_t section_off,
                              int rows, CUtensorMap *map) {
    PFN_cuTensorMapEncodeTiled_v12000 enc = tensor_map_encoder();
    if (enc == nullptr)
        return cudaErrorNotSupported;
    const int64_t row_bytes = weight_row_bytes(a, a.H);
    const int64_t sec_bytes = (a.I * row_bytes + 15) / 16 * 16;
    const cuuint64_t dims[3] = {(cuuint64_t)(row_bytes / 4), (cuuint64_t)a.I,
                                (cuuint64_t)a.E};
    const cuuint64_t strides[2] = {
        (cuuint64_t)row_bytes,
        (cuuint64_t)(a.E > 1 ? a.stride : std::max<int64_t>(a.stride,
                                                            sec_bytes))};
    const cuuint32_t box[3] = {32, (cuuint32_t)rows, 1};
    const cuuint32_t estr[3] = {1, 1, 1};
    const CUresult r = enc(map, CU_TENSOR_MAP_DATA_TYPE_UINT32, 3,
                           const_cast<uint8_t *>(a.base + section_off), dims,
                           strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                           CU_TENSOR_MAP_SWIZZLE_128B,
                           CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                           CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS ? cudaSuccess : cudaErrorInvalidValue;
}

template <int NB, bool kDown, bool kQ8>
cudaError_t launch_nb(const GateUpArgs &a, int tok_cap, cudaStream_t s) {
    int D = kMaxStages;
    while (D > 2 && tma_smem(a, NB, D, tok_cap) > kSmemLimit)
        --D;
    const size_t smem = tma_smem(a, NB, D, tok_cap);
    CUtensorMap mg, mu;
    memset(&mg, 0, sizeof mg);
    memset(&mu, 0, sizeof mu);
    cudaError_t err = encode_weight_map(a, a.gate_w_off, NB * 16, &mg);
    if (err == cudaSuccess)
        err = encode_weight_map(a, a.up_w_off, NB * 16, &mu);
    if (err != cudaSuccess)
        return err;
    err = cudaFuncSetAttribute(matvec_tma_kernel<NB, kDown, kQ8>,
                               cudaFuncAttributeMaxDynamicSharedMemorySize,
                               (int)smem);
    if (err != cudaSuccess)
        return err;
    // a single expert's rows all above the matvec's limit: nothing to do
    if (a.E == 1 && a.M > a.matvec_max_rows)
        return cudaSuccess;
    return launch_pdl(matvec_tma_kernel<NB, kDown, kQ8>,
                      dim3((unsigned)a.num_sms), dim3(kThreads), smem, s, a,
                      mg, mu, tok_cap, D);
}

template <int NB>
cudaError_t launch_mode(const GateUpArgs &a, int tok_cap, cudaStream_t s) {
    if (a.q8)
        return a.down ? launch_nb<NB, true, true>(a, tok_cap, s)
                      : launch_nb<NB, false, true>(a, tok_cap, s);
    return a.down ? launch_nb<NB, true, false>(a, tok_cap, s)
                  : launch_nb<NB, false, false>(a, tok_cap, s);
}

}  // namespace

bool matvec_tma_supported(const GateUpArgs &a) {
    const int tok_cap = (int)std::min<int64_t>(kTok, a.M);
    const int box_k = a.q8 ? Fmt<true>::kBoxK : Fmt<false>::kBoxK;
    return a.slab_ptrs == nullptr && a.H % box_k == 0 && a.I % 16 == 0 &&
           a.gate_w_off % 16 == 0 && a.up_w_off % 16 == 0 &&
           (reinterpret_cast<uintptr_t>(a.base) & 15) == 0 &&
           a.H < (1ll << 31) && a.I < (1ll << 31) &&
           tensor_map_encoder() != nullptr &&
           tma_smem(a, 1, 2, tok_cap) <= kSmemLimit &&
           tma_smem(a, 8, 2, tok_cap) <= kSmemLimit;
}

// Tile height: the caller's, else the tallest (fewest K parts to reduce)
// that still gives at least four units per SM when each of the first
// min(E, M) experts holds one chunk.
cudaError_t launch_matvec_tma(const GateUpArgs &a, cudaStream_t s) {
    const int tok_cap = (int)std::min<int64_t>(kTok, a.M);
    switch (a.matvec_tile) {
    case 16: return launch_mode<1>(a, tok_cap, s);
    case 32: return launch_mode<2>(a, tok_cap, s);
    case 64: return launch_mode<4>(a, tok_cap, s);
    case 128: return launch_mode<8>(a, tok_cap, s);
    default: break;
    }
    const int64_t chunks = std::min<int64_t>(a.E, a.M);
    const int64_t rows16 = a.down ? 32 : 16;   // output rows per 16-row box
    const int64_t want = 4ll * a.num_sms;
    auto units = [&](int64_t nb) {
        return chunks * ((a.I + rows16 * nb - 1) / (rows16 * nb));
    };
    if (units(8) >= want)
        return launch_mode<8>(a, tok_cap, s);
    if (units(4) >= want)
        return launch_mode<4>(a, tok_cap, s);
    if (units(2) >= want)
        return launch_mode<2>(a, tok_cap, s);
    return launch_mode<1>(a, tok_cap, s);
}

}  // namespace q4moe
