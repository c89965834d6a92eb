// q4moe_gemm.cu -- grouped Q4 gate/up + SwiGLU on the tcgen05 tensor core,
// for experts with many rows (prefill).
//
// The pages give the fused gate/up/SwiGLU as a matvec (page 52,
// streamed-experts.ts, GATE_UP_SOURCE) and as an 8x8 simdgroup-matrix form
// for up to 8 rows (page 57, trellis/gate-up-mma.ts); this is the
// large-batch form of the same arithmetic for sm_103a:
//
//  tile   = 128 intermediate rows (i) of one expert x up to 256 of the
//           expert's grouped rows (tokens); both projections of the tile
//           share the token operand;
//  A      = the gate (and the up) weights of the tile's rows, dequantised
//           (nibble - 8, exact in bf16) into shared memory in the 128-byte
//           swizzled K-major layout, 64 K per pipeline stage;
//  B      = the tile's token rows of x in the same layout: with a
//           workspace, the rows are first copied once into grouped order
//           and each stage is at most five TMA boxes; without one,
//           they are gathered row by row with cp.async;
//  D      = two f32 accumulators in tensor memory (gate: columns 0..N-1,
//           up: columns 256..256+N-1), lane = intermediate row;
//  tail   = row scales, bf16 rounding and the SwiGLU chain, per element, as
//           in the matvec.
//
// Warp roles (512 threads, one CTA per SM, persistent over tiles):
//   0-7   epilogue (warp w reads TMEM lanes 32*(w%4)..; w/4 picks the
//         16-column chunks it handles)
//   8     TMEM allocation and the single thread that issues the MMAs
//   9-12  weight dequantisation (one A row of gate and of up per thread)
//   13-15 token rows: one thread issuing TMA boxes (workspace), or all
//         three warps gathering with cp.async, each thread's copies
//         counting as its arrival on the stage barrier when they land
// The down projection (page 52, DOWN_SOURCE) runs on the same kernel
// (kDown): a tile is 256 output rows of the one matrix, rows 0-127 in the
// "gate" accumulator and 128-255 in the "up" one (a half past the last row
// is dequantised as zeros and never stored); the token operand is mid
// itself, already in grouped order, read through TMA without a copy; the
// epilogue applies the row scale and rounds to bf16.
//
// Every wait on an mbarrier is bounded; on time-out the CTA raises
// Q4MOE_DEV_WAIT_TIMEOUT, drains its copies and MMAs, frees TMEM and exits.
#include <cuda.h>
#include <cudaTypedefs.h>

#include <algorithm>
#include <cstring>
#include <mutex>

#include "q4moe_internal.cuh"
#include "q4moe_sm100.cuh"

namespace q4moe {
namespace {

using namespace sm100;

constexpr int BM = 128;                      // intermediate rows per tile
constexpr int BK = 64;                       // K per stage
constexpr int NMAX = 256;                    // token rows per tile
// Two rings: the dequantised weights (A: gate and up tiles) refill within
// about one MMA stage, the token rows (B) come from HBM and need more
// stages in flight.
constexpr int A_STAGES = 3;
constexpr int B_STAGES = 3;

constexpr int A_BYTES = BM * BK * 2;         // 16 KB
constexpr int B_BYTES = NMAX * BK * 2;       // 32 KB
constexpr int A_STAGE_BYTES = 2 * A_BYTES;
constexpr int RING_BYTES = A_STAGES * A_STAGE_BYTES + B_STAGES * B_BYTES;
constexpr int kThreads = 512;
constexpr int kEpiWarps = 8;
constexpr int kMmaWarp = 8;
constexpr int kDeqWarp0 = 9;
constexpr int kDeqWarps = 4;
constexpr int kGatWarp0 = 13;
constexpr int kGatWarps = 3;
constexpr int kGatThreads = kGatWarps * 32;
constexpr int kGatItems = (NMAX * 8 + kGatThreads - 1) / kGatThreads;
constexpr int kPrefetch = 4;                 // k-blocks of weights in flight
constexpr uint32_t kTmemCols = 512;
constexpr uint32_t kUpCol = 256;
constexpr uint64_t kTimeoutNs = 4000000000ull;
// Tensor maps of the grouped activations with boxes of 256, 128, 64, 32
// and 16 rows: a tile of n rows (a multiple of 16) is at most five loads,
// one per set bit of n / 16 (each TMA instruction costs the single issuing
// thread on the order of a hundred cycles).
constexpr int kBoxLevels = 5;
struct XgMaps {
    CUtensorMap m[kBoxLevels];               // box rows 256 >> level
};

struct Ctl {
    uint64_t a_full[A_STAGES];
    uint64_t a_empty[A_STAGES];
    uint64_t b_full[B_STAGES];
    uint64_t b_empty[B_STAGES];
    uint64_t tmem_full;
    uint64_t tmem_empty;
    uint64_t drain;
    uint32_t tmem_base;
    int abort;
    int bad_offsets;
};

constexpr size_t smem_bytes(int E) {
    return 1024 + (size_t)RING_BYTES + sizeof(Ctl) +
           2 * sizeof(int32_t) * (size_t)(E + 1) + 16;
}

struct Tile {
    int e;          // expert
    int iblk;       // block of 128 intermediate rows
    int row0;       // first grouped row of the tile
    int nvalid;     // grouped rows in the tile
    int n;          // nvalid rounded up to 16 (the MMA's N)
};

__device__ __forceinline__ int ceil_div(int a, int b) { return (a + b - 1) / b; }

// Rows of expert e are split into ceil(n/256) chunks of equal size rounded
// up to 16.
__device__ __forceinline__ int chunk_rows(int n_e) {
    const int nch = ceil_div(n_e, NMAX);
    return ceil_div(ceil_div(n_e, nch), 16) * 16;
}

__device__ __forceinline__ Tile tile_of(int t, const int32_t *off,
                                        const int32_t *pre, int E, int IB) {
    int lo = 0, hi = E;
    while (hi - lo > 1) {
        const int mid = (lo + hi) >> 1;
        if (pre[mid] <= t)
            lo = mid;
        else
            hi = mid;
    }
    Tile ti;
    ti.e = lo;
    const int local = t - pre[lo];
    const int chunk = local / IB;
    ti.iblk = local - chunk * IB;
    const int n_e = off[lo + 1] - off[lo];
    const int cs = chunk_rows(n_e);
    ti.row0 = off[lo] + chunk * cs;
    ti.nvalid = min(cs, n_e - chunk * cs);
    ti.n = ceil_div(ti.nvalid, 16) * 16;
    return ti;
}

// One packed word (8 nibbles, K order) -> 8 bf16 (nibble - 8) in K order:
// each output pair (2j, 2j+1) is byte j of the word split into its two
// nibbles, placed in the low mantissa bits of 128.0 (0x4300) and then
// reduced by 136 (exact: the results are the integers -8..7).
__device__ __forceinline__ uint4 dequant_word(uint32_t w) {
    const uint32_t ws = w >> 4;
    uint32_t r[4];
#pragma unroll
    for (int j = 0; j < 4; ++j) {
        const uint32_t v =
            (__byte_perm(w, ws, (uint32_t)(j | ((4 + j) << 8))) &
             0x000F000Fu) | 0x43004300u;
        __nv_bfloat162 b = *reinterpret_cast<const __nv_bfloat162 *>(&v);
        const __nv_bfloat162 k136 =
            __halves2bfloat162(__ushort_as_bfloat16((unsigned short)0x4308),
                               __ushort_as_bfloat16((unsigned short)0x4308));
        b = __hsub2(b, k136);
        r[j] = *reinterpret_cast<const uint32_t *>(&b);
    }
    return make_uint4(r[0], r[1], r[2], r[3]);
}

// Two signed bytes, given as t = {b0, 0x43, b1, 0x43} (bytes, low first),
// -> bf16x2 {b0, b1}, exact: under the bf16 exponent byte 0x43 the low
// seven bits m of a byte read 128 + m, its sign bit reads 128 or 256, and
// b = (128 + m) - (128 + 128 * sign); the difference is an integer of at
// most 8 bits, so the bf16 subtraction is exact.
__device__ __forceinline__ uint32_t byte_pair_bf16(uint32_t t) {
    const uint32_t m = t & 0x437F437Fu, c = t & 0x43804380u;
    const __nv_bfloat162 r =
        __hsub2(*reinterpret_cast<const __nv_bfloat162 *>(&m),
                *reinterpret_cast<const __nv_bfloat162 *>(&c));
    return *reinterpret_cast<const uint32_t *>(&r);
}

// Two words of four signed bytes each (K order) -> 8 bf16, exact.
__device__ __forceinline__ uint4 dequant_bytes8(uint32_t w0, uint32_t w1) {
    return make_uint4(byte_pair_bf16(__byte_perm(w0, 0x43434343u, 0x4140)),
                      byte_pair_bf16(__byte_perm(w0, 0x43434343u, 0x4342)),
                      byte_pair_bf16(__byte_perm(w1, 0x43434343u, 0x4140)),
                      byte_pair_bf16(__byte_perm(w1, 0x43434343u, 0x4342)));
}

// Byte offset of 16-byte chunk c (0..7) of row r in a 128-byte-swizzled
// K-major tile.
__device__ __forceinline__ uint32_t sw128_offset(int r, int c) {
    return (uint32_t)((r >> 3) * 1024 + (r & 7) * 128 + ((c ^ (r & 7)) << 4));
}

// Copy the activations of each grouped row that the GEMM will read (rows of
// experts above the matvec's row limit) into the workspace, bf16 [M][H].
// The offsets are staged in shared memory (the expert of a row is a binary
// search there); one warp copies one row, each lane keeping four 16-byte
// loads in flight.  When the GEMM takes every expert the rows go rank by
// rank (rank r of every expert, then r + 1): an expert's rows are in token
// order, so a token's rows are copied close together and its activations
// are read from L2 after the first (prefill 0.810 -> 0.805 ms; with
// experts left to the matvec most rank slots are empty and the grouped
// order is kept: the verify width took 0.288 -> 0.308 ms rank by rank).
// kPairs writes each chunk of 8 activations in the order
// {0,4,1,5,2,6,3,7} (the Q4 gate/up form of q4moe_gemm_tma.cu, whose
// dequantised weights come in that order).
constexpr int kGatherThreads = 256;
template <bool kPairs, bool kByRank>
__global__ void __launch_bounds__(kGatherThreads)
gather_rows_kernel(GateUpArgs a) {
    extern __shared__ int32_t s_goff[];
    grid_dependency_wait();
    for (int e = threadIdx.x; e <= a.E; e += blockDim.x)
        s_goff[e] = a.row_offsets[e];
    __syncthreads();
    const int32_t mvmax = matvec_limit(a, s_goff);
    const int lane = threadIdx.x & 31;
    const int64_t chunks = a.H / 8;
    const int64_t wpb = blockDim.x / 32;
    const int64_t nwarps = (int64_t)gridDim.x * wpb;
    int32_t maxc = 0;                 // the largest expert's rows
    if (kByRank)
        for (int e = 0; e < a.E; ++e)
            maxc = max(maxc, s_goff[e + 1] - s_goff[e]);
    const int64_t n_idx = kByRank ? (int64_t)maxc * a.E : a.M;
    for (int64_t ii = blockIdx.x * wpb + (threadIdx.x >> 5); ii < n_idx;
         ii += nwarps) {
        int64_t p;
        int lo;                       // expert e with off[e] <= p < off[e+1]
        if (kByRank) {
            const int64_t r = ii / a.E;
            lo = (int)(ii - r * a.E);
            if (r >= s_goff[lo + 1] - s_goff[lo])
                continue;
            p = s_goff[lo] + r;
        } else {
            p = ii;
            lo = 0;
            int hi = a.E;
            while (hi - lo > 1) {
                const int mid = (lo + hi) >> 1;
                if (s_goff[mid] <= p)
                    lo = mid;
                else
                    hi = mid;
            }
        }
        if (s_goff[lo + 1] - s_goff[lo] <= mvmax)
            continue;
        int64_t t = 0;
        if (lane == 0)
            t = row_token(a, p);
        t = __shfl_sync(0xffffffffu, t, 0);
        uint4 *dst = reinterpret_cast<uint4 *>(a.xg + p * a.H);
        const uint4 *src = reinterpret_cast<const uint4 *>(a.x + t * a.H);
        for (int64_t c0 = lane; c0 < chunks; c0 += 128) {
            uint4 v[4];
#pragma unroll
            for (int u = 0; u < 4; ++u) {
                const int64_t c = c0 + 32 * u;
                v[u] = (t >= 0 && c < chunks) ? __ldg(src + c)
                                              : make_uint4(0, 0, 0, 0);
            }
#pragma unroll
            for (int u = 0; u < 4; ++u) {
                const int64_t c = c0 + 32 * u;
                if (kPairs) {           // {x0x1,x2x3,x4x5,x6x7} -> {x0x4,..}
                    const uint4 w = v[u];
                    v[u] = make_uint4(__byte_perm(w.x, w.z, 0x5410),
                                      __byte_perm(w.x, w.z, 0x7632),
                                      __byte_perm(w.y, w.w, 0x5410),
                                      __byte_perm(w.y, w.w, 0x7632));
                }
                if (c < chunks)
                    dst[c] = v[u];
            }
        }
    }
}

template <bool kTma, bool kDown, bool kQ8>
__global__ void __launch_bounds__(kThreads, 1)
gemm_tcgen05_kernel(GateUpArgs a, const __grid_constant__ XgMaps xg_maps) {
    static_assert(kTma || !kDown, "the down projection reads mid by TMA");
    extern __shared__ uint8_t smem_raw[];
    uint8_t *smem = reinterpret_cast<uint8_t *>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    uint8_t *stages = smem;
    Ctl *ctl = reinterpret_cast<Ctl *>(smem + (size_t)RING_BYTES);
    int32_t *s_off = reinterpret_cast<int32_t *>(ctl + 1);
    int32_t *s_pre = s_off + (a.E + 1);

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int E = a.E;
    const int IB = gemm_row_tiles(a);        // tiles over the output rows
    const int KB = (int)(a.H / BK);
    // first row of a tile's second half (down: 128 rows further)
    const int64_t hi_row = kDown ? BM : 0;
    const int64_t tile_rows = kDown ? 2 * BM : BM;

    if (tid == 0) {
        for (int s = 0; s < A_STAGES; ++s) {
            mbar_init(&ctl->a_full[s], kDeqWarps);
            mbar_init(&ctl->a_empty[s], 1);
        }
        for (int s = 0; s < B_STAGES; ++s) {
            mbar_init(&ctl->b_full[s], kTma ? 1 : kGatThreads);
            mbar_init(&ctl->b_empty[s], 1);
        }
        mbar_init(&ctl->tmem_full, 1);
        mbar_init(&ctl->tmem_empty, kEpiWarps);
        mbar_init(&ctl->drain, 1);
        ctl->abort = 0;
        ctl->bad_offsets = 0;
        fence_mbar_init();
    }
    if (warp == kMmaWarp) {
        tmem_alloc(&ctl->tmem_base, kTmemCols);
        tmem_relinquish();
    }
    grid_dependency_wait();
    // stage and check the row offsets
    for (int e = tid; e <= E; e += kThreads) {
        const int32_t v = a.row_offsets[e];
        s_off[e] = v;
        if ((e == 0 && v != 0) || (e == E && v != a.M) || v < 0 || v > a.M ||
            (e > 0 && a.row_offsets[e - 1] > v))
            ctl->bad_offsets = 1;
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const bool offsets_ok = ctl->bad_offsets == 0;
    const int32_t mvmax = matvec_limit(a, s_off);
    if (!offsets_ok && tid == 0 && blockIdx.x == 0)
        atomicOr(a.status, Q4MOE_DEV_BAD_ROW_OFFSETS);
    // tiles per expert (experts above the matvec's row limit), prefix sums
    if (warp == 0 && offsets_ok) {
        const int per = ceil_div(E, 32);
        const int e0 = lane * per;
        int sum = 0;
        for (int e = e0; e < min(E, e0 + per); ++e) {
            const int n_e = s_off[e + 1] - s_off[e];
            sum += (n_e > mvmax && n_e > 0)
                       ? IB * ceil_div(n_e, NMAX) : 0;
        }
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
            const int n_e = s_off[e + 1] - s_off[e];
            run += (n_e > mvmax && n_e > 0)
                       ? IB * ceil_div(n_e, NMAX) : 0;
        }
        if (lane == 31)
            s_pre[E] = incl;
    }
    __syncthreads();
    const int ntiles = offsets_ok ? s_pre[E] : 0;
    const uint32_t tmem = ctl->tmem_base;
    volatile int *abort = &ctl->abort;
    const uint32_t stage0 = smem_u32(stages);
    const uint32_t b_ring0 = stage0 + A_STAGES * A_STAGE_BYTES;

    if (kTma && warp >= kGatWarp0) {
        // ------------------------------------------- token rows via TMA
        if (warp == kGatWarp0 && lane == 0) {
            uint32_t g = 0;
            for (int t = blockIdx.x; t < ntiles && !*abort; t += gridDim.x) {
                const Tile ti = tile_of(t, s_off, s_pre, E, IB);

                bool ok = true;
                for (int kb = 0; kb < KB; ++kb, ++g) {
                    const uint32_t s = g % B_STAGES;
                    if (!wait_phase(&ctl->b_empty[s],
                                    ((g / B_STAGES) & 1) ^ 1, abort,
                                    a.status)) {
                        ok = false;
                        break;
                    }
                    mbar_arrive_expect_tx(&ctl->b_full[s],
                                          (uint32_t)ti.n * BK * 2);
                    const uint32_t bdst = b_ring0 + s * B_BYTES;
                    int off = 0;                 // rows issued so far
#pragma unroll
                    for (int lvl = 0; lvl < kBoxLevels; ++lvl) {
                        const int h = 256 >> lvl;
                        if (ti.n - off >= h) {
                            tma_load_2d(bdst + off * (BK * 2),
                                        &xg_maps.m[lvl], kb * BK,
                                        ti.row0 + off, &ctl->b_full[s]);
                            off += h;
                        }
                    }
                }
                if (!ok)
                    break;
            }
            // let the boxes still in flight land before the CTA exits
            for (uint32_t gg = g > B_STAGES ? g - B_STAGES : 0; gg < g; ++gg)
                drain_phase(&ctl->b_full[gg % B_STAGES], (gg / B_STAGES) & 1);
        }
    } else if (warp >= kGatWarp0) {
        // ---------------------------------------------------- token gather
        const int j = tid - kGatWarp0 * 32;
        const uint64_t keep = l2_policy_evict_last();
        uint32_t g = 0;
        for (int t = blockIdx.x; t < ntiles && !*abort; t += gridDim.x) {
            const Tile ti = tile_of(t, s_off, s_pre, E, IB);
            // per item: token row (>= 0), -1 zero fill, -2 nothing to copy
            int32_t tokm[kGatItems];
#pragma unroll
            for (int m = 0; m < kGatItems; ++m) {
                const int f = j + kGatThreads * m;
                const int n = f >> 3;
                tokm[m] = -2;
                if (n < ti.n) {
                    tokm[m] = -1;
                    if (n < ti.nvalid) {
                        const int64_t tok = row_token(a, ti.row0 + n);
                        if (tok >= 0)
                            tokm[m] = (int32_t)tok;
                    }
                }
            }
            bool ok = true;
            for (int kb = 0; kb < KB; ++kb, ++g) {
                const uint32_t s = g % B_STAGES;
                if (!wait_phase(&ctl->b_empty[s], ((g / B_STAGES) & 1) ^ 1,
                                abort, a.status)) {
                    ok = false;
                    break;
                }
                const uint32_t bdst = b_ring0 + s * B_BYTES;
#pragma unroll
                for (int m = 0; m < kGatItems; ++m) {
                    if (tokm[m] == -2)
                        continue;
                    const int f = j + kGatThreads * m;
                    const uint32_t dst = bdst + sw128_offset(f >> 3, f & 7);
                    if (tokm[m] >= 0)
                        cp_async_16_hint(dst,
                                         a.x + (int64_t)tokm[m] * a.H +
                                             (f & 7) * 8 + kb * BK,
                                         16, keep);
                    else
                        cp_async_16(dst, a.x, 0);
                }
                // counted as this thread's arrival once its copies landed
                cp_async_arrive_noinc(&ctl->b_full[s]);
            }
            if (!ok)
                break;
        }
        cp_async_wait<0>();
    } else if (warp >= kDeqWarp0) {
        // ------------------------------------------- weight dequantisation
        const int r = tid - kDeqWarp0 * 32;          // A row 0..127
        uint32_t g = 0;
        for (int t = blockIdx.x; t < ntiles && !*abort; t += gridDim.x) {
            const Tile ti = tile_of(t, s_off, s_pre, E, IB);
            const uint8_t *slab = expert_slab(a, ti.e);
            const int64_t row = (int64_t)ti.iblk * tile_rows + r;
            // the second half's row exists (always, for gate/up)
            const bool uok = slab && (!kDown || row + hi_row < a.I);
            // a k-block (64 K) of one row is kVecs 16-byte vectors: 32
            // bytes of nibbles (Q4) or 64 of signed bytes (Q8)
            constexpr int kVecs = kQ8 ? 4 : 2;
            constexpr int kDepth = kQ8 ? 2 : kPrefetch;  // k-blocks in flight
            const int64_t rb = weight_row_bytes(a, a.H);
            const uint4 *gp = slab ? reinterpret_cast<const uint4 *>(
                                         slab + a.gate_w_off + row * rb)
                                   : nullptr;
            const uint4 *up = uok ? reinterpret_cast<const uint4 *>(
                                        slab + a.up_w_off + (row + hi_row) * rb)
                                  : nullptr;
            uint4 ring[kDepth][2 * kVecs];
            // weight zero: nibble 8 (Q4) or byte 0 (Q8)
            const uint32_t z = kQ8 ? 0u : 0x88888888u;
            const uint4 kZero = make_uint4(z, z, z, z);
#pragma unroll
            for (int d = 0; d < kDepth; ++d) {
                const bool in = d < KB;
#pragma unroll
                for (int v = 0; v < kVecs; ++v) {
                    ring[d][v] = (in && slab) ? __ldg(gp + kVecs * d + v)
                                              : kZero;
                    ring[d][kVecs + v] = (in && uok)
                                             ? __ldg(up + kVecs * d + v)
                                             : kZero;
                }
            }
            bool ok = true;
            for (int kb0 = 0; kb0 < KB && ok; kb0 += kDepth) {
#pragma unroll
                for (int d = 0; d < kDepth; ++d) {
                    const int kb = kb0 + d;
                    if (kb >= KB)
                        break;
                    const uint32_t s = g % A_STAGES;
                    if (!wait_phase(&ctl->a_empty[s],
                                    ((g / A_STAGES) & 1) ^ 1, abort,
                                    a.status)) {
                        ok = false;
                        break;
                    }
                    uint8_t *ag = stages + (size_t)s * A_STAGE_BYTES;
                    uint8_t *au = ag + A_BYTES;
#pragma unroll
                    for (int c = 0; c < 8; ++c) {
                        // 16-byte chunk c of the row's 64 K: 8 values
                        const uint32_t *rg =
                            reinterpret_cast<const uint32_t *>(&ring[d][0]);
                        const uint32_t *ru =
                            reinterpret_cast<const uint32_t *>(&ring[d][kVecs]);
                        uint4 vg, vu;
                        if (kQ8) {
                            vg = dequant_bytes8(rg[2 * c], rg[2 * c + 1]);
                            vu = dequant_bytes8(ru[2 * c], ru[2 * c + 1]);
                        } else {
                            vg = dequant_word(rg[c]);
                            vu = dequant_word(ru[c]);
                        }
                        *reinterpret_cast<uint4 *>(ag + sw128_offset(r, c)) =
                            vg;
                        *reinterpret_cast<uint4 *>(au + sw128_offset(r, c)) =
                            vu;
                    }
                    const int kn = kb + kDepth;
                    if (kn < KB && slab) {
#pragma unroll
                        for (int v = 0; v < kVecs; ++v) {
                            ring[d][v] = __ldg(gp + kVecs * kn + v);
                            if (uok)
                                ring[d][kVecs + v] = __ldg(up + kVecs * kn + v);
                        }
                    }
                    fence_proxy_async_smem();
                    __syncwarp();
                    if (lane == 0)
                        mbar_arrive(&ctl->a_full[s]);
                    ++g;
                }
            }
            if (!ok)
                break;
        }
    } else if (warp == kMmaWarp) {
        // ------------------------------------------------------ MMA issue
        if (lane == 0) {
            uint32_t g = 0, it = 0;
            bool issued = false;
            for (int t = blockIdx.x; t < ntiles && !*abort;
                 t += gridDim.x, ++it) {
                const Tile ti = tile_of(t, s_off, s_pre, E, IB);
                const uint32_t idesc = idesc_bf16_m128((uint32_t)ti.n);
                if (!wait_phase(&ctl->tmem_empty, (it & 1) ^ 1, abort,
                                a.status))
                    break;
                tc_fence_after();
                bool ok = true;
                for (int kb = 0; kb < KB; ++kb, ++g) {
                    const uint32_t sa = g % A_STAGES, sb = g % B_STAGES;
                    if (!wait_phase(&ctl->b_full[sb], (g / B_STAGES) & 1,
                                    abort, a.status) ||
                        !wait_phase(&ctl->a_full[sa], (g / A_STAGES) & 1,
                                    abort, a.status)) {
                        ok = false;
                        break;
                    }
                    // token rows that arrived through cp.async (generic
                    // proxy) are ordered before the tensor core's reads
                    if (!kTma)
                        fence_proxy_async_smem();
                    tc_fence_after();
                    const uint32_t ag = stage0 + sa * A_STAGE_BYTES;
                    const uint32_t au = ag + A_BYTES;
                    const uint32_t bb = b_ring0 + sb * B_BYTES;
#pragma unroll
                    for (int ks = 0; ks < BK / 16; ++ks) {
                        const uint32_t acc = (kb > 0 || ks > 0) ? 1u : 0u;
                        const uint64_t bd = sw128_kmajor_desc(bb + ks * 32);
                        umma_bf16(tmem, sw128_kmajor_desc(ag + ks * 32), bd,
                                  idesc, acc);
                        umma_bf16(tmem + kUpCol,
                                  sw128_kmajor_desc(au + ks * 32), bd, idesc,
                                  acc);
                    }
                    umma_commit(&ctl->a_empty[sa]);
                    umma_commit(&ctl->b_empty[sb]);
                    issued = true;
                }
                if (!ok)
                    break;
                umma_commit(&ctl->tmem_full);
            }
            if (issued) {
                umma_commit(&ctl->drain);
                uint64_t t0 = globaltimer_ns();
                while (!mbar_try_wait(&ctl->drain, 0) &&
                       globaltimer_ns() - t0 < kTimeoutNs) {
                }
            }
        }
    } else {
        // ------------------------------------------------------- epilogue
        const int quad = warp & 3, half = warp >> 2;
        uint32_t it = 0;
        for (int t = blockIdx.x; t < ntiles && !*abort;
             t += gridDim.x, ++it) {
            const Tile ti = tile_of(t, s_off, s_pre, E, IB);
            if (!wait_phase(&ctl->tmem_full, it & 1, abort, a.status))
                break;
            tc_fence_after();
            const uint8_t *slab = expert_slab(a, ti.e);
            const int64_t i = (int64_t)ti.iblk * tile_rows + quad * 32 + lane;
            const bool hi_ok = !kDown || i + hi_row < a.I;
            float sg = 0.0f, su = 0.0f;
            if (slab) {
                sg = reinterpret_cast<const float *>(slab + a.gate_s_off)[i];
                if (hi_ok)
                    su = reinterpret_cast<const float *>(
                        slab + a.up_s_off)[i + hi_row];
            }
            const uint32_t tl = tmem + ((uint32_t)(quad * 32) << 16);
            for (int c0 = half * 16; c0 < ti.n; c0 += 32) {
                uint32_t gv[16], uv[16];
                tmem_ld16(tl + (uint32_t)c0, gv);
                tmem_ld16(tl + kUpCol + (uint32_t)c0, uv);
                tmem_ld_wait();
                if (!slab)
                    continue;
                if (kDown) {
                    // out = bf16(sum * scale) for both halves
                    const int64_t o0 = (int64_t)(ti.row0 + c0) * a.I + i;
#pragma unroll
                    for (int jj = 0; jj < 16; ++jj) {
                        const float lo = __fmul_rn(__uint_as_float(gv[jj]), sg);
                        const float hi = __fmul_rn(__uint_as_float(uv[jj]), su);
                        if (c0 + jj < ti.nvalid) {
                            const int64_t oi = o0 + (int64_t)jj * a.I;
                            a.out[oi] = bf16_bits(lo);
                            if (a.gate_f32)
                                a.gate_f32[oi] = lo;
                            if (hi_ok) {
                                a.out[oi + hi_row] = bf16_bits(hi);
                                if (a.gate_f32)
                                    a.gate_f32[oi + hi_row] = hi;
                            }
                        }
                    }
                    continue;
                }
                // all 16 columns branch-free (independent chains the
                // scheduler can interleave); sigmoids from the table
                float gT[16], uT[16], sT[16];
#pragma unroll
                for (int jj = 0; jj < 16; ++jj) {
                    const float g32 = __fmul_rn(__uint_as_float(gv[jj]), sg);
                    const float u32 = __fmul_rn(__uint_as_float(uv[jj]), su);
                    gv[jj] = __float_as_uint(g32);
                    uv[jj] = __float_as_uint(u32);
                    gT[jj] = bf16_round(g32);
                    uT[jj] = bf16_round(u32);
                    sT[jj] = bf16_f32(sigmoid_bf16_table(
                        a.sigmoid,
                        (uint16_t)(__float_as_uint(gT[jj]) >> 16)));
                }
                const int64_t o0 = (int64_t)(ti.row0 + c0) * a.I + i;
#pragma unroll
                for (int jj = 0; jj < 16; ++jj) {
                    const float si = bf16_round(__fmul_rn(gT[jj], sT[jj]));
                    const uint16_t o = bf16_bits(__fmul_rn(si, uT[jj]));
                    if (c0 + jj < ti.nvalid) {
                        const int64_t oi = o0 + (int64_t)jj * a.I;
                        a.out[oi] = o;
                        if (a.gate_f32)
                            a.gate_f32[oi] = __uint_as_float(gv[jj]);
                        if (a.up_f32)
                            a.up_f32[oi] = __uint_as_float(uv[jj]);
                    }
                }
            }
            tc_fence_before();
            __syncwarp();
            if (lane == 0)
                mbar_arrive(&ctl->tmem_empty);
        }
    }

    tc_fence_before();
    __syncthreads();
    if (warp == kMmaWarp) {
        __syncwarp();
        tc_fence_after();
        tmem_dealloc(tmem, kTmemCols);
    }
}

}  // namespace

// cuTensorMapEncodeTiled through the runtime's driver entry point (no
// link-time dependence on libcuda); null when the driver lacks it.
PFN_cuTensorMapEncodeTiled_v12000 tensor_map_encoder() {
    static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
    static std::once_flag once;
    std::call_once(once, [] {
        void *p = nullptr;
        cudaDriverEntryPointQueryResult q{};
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p,
                                             12000, cudaEnableDefault,
                                             &q) == cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
    });
    return fn;
}

bool gemm_supported(int64_t H, int64_t I, const GateUpArgs &a) {
    return H % BK == 0 && I % BM == 0 && a.gate_w_off % 16 == 0 &&
           a.up_w_off % 16 == 0 && a.E <= Q4MOE_MAX_EXPERTS;
}

namespace {

// Tensor maps of the grouped activations bf16 [M][H]: boxes of 64 columns
// (128 bytes, the swizzle span) x 256 >> level rows, 128-byte swizzle, rows
// past M read as zero.
cudaError_t encode_xg_maps(const GateUpArgs &a, const uint16_t *rows,
                           XgMaps *maps) {
    PFN_cuTensorMapEncodeTiled_v12000 enc = tensor_map_encoder();
    if (enc == nullptr)
        return cudaErrorNotSupported;
    const cuuint64_t dims[2] = {(cuuint64_t)a.H, (cuuint64_t)a.M};
    const cuuint64_t strides[1] = {(cuuint64_t)a.H * 2};
    const cuuint32_t estr[2] = {1, 1};
    for (int lvl = 0; lvl < kBoxLevels; ++lvl) {
        const cuuint32_t box[2] = {(cuuint32_t)BK, (cuuint32_t)(256 >> lvl)};
        const CUresult r = enc(&maps->m[lvl], CU_TENSOR_MAP_DATA_TYPE_BFLOAT16,
                               2, const_cast<uint16_t *>(rows), dims,
                               strides, box, estr,
                               CU_TENSOR_MAP_INTERLEAVE_NONE,
                               CU_TENSOR_MAP_SWIZZLE_128B,
                               CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                               CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
        if (r != CUDA_SUCCESS)
            return cudaErrorInvalidValue;
    }
    return cudaSuccess;
}

template <bool kTma, bool kDown, bool kQ8>
cudaError_t launch_gemm_fmt(const GateUpArgs &a, const XgMaps &maps,
                            cudaStream_t s) {
    const size_t smem = smem_bytes(a.E);
    cudaError_t err = cudaFuncSetAttribute(
        gemm_tcgen05_kernel<kTma, kDown, kQ8>,
        cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (err != cudaSuccess)
        return err;
    return launch_pdl(gemm_tcgen05_kernel<kTma, kDown, kQ8>,
                      dim3((unsigned)a.num_sms), dim3(kThreads), smem, s, a,
                      maps);
}

template <bool kTma, bool kDown>
cudaError_t launch_gemm_kernel(const GateUpArgs &a, const XgMaps &maps,
                               cudaStream_t s) {
    return a.q8 ? launch_gemm_fmt<kTma, kDown, true>(a, maps, s)
                : launch_gemm_fmt<kTma, kDown, false>(a, maps, s);
}

}  // namespace

cudaError_t launch_gemm(const GateUpArgs &a, cudaStream_t s) {
    const bool ts = gemm_tma_supported(a) && (a.down || a.xg != nullptr);
    if (ts && a.down)                // mid is grouped already: no copy
        return launch_gemm_tma(a, a.x, s);
    XgMaps maps;
    memset(&maps, 0, sizeof maps);
    if (a.down) {                    // mid is grouped already: no copy
        cudaError_t err = encode_xg_maps(a, a.x, &maps);
        if (err != cudaSuccess)
            return err;
        return launch_gemm_kernel<true, true>(a, maps, s);
    }
    if (a.xg == nullptr)
        return launch_gemm_kernel<false, false>(a, maps, s);
    cudaError_t err = encode_xg_maps(a, a.xg, &maps);
    if (err != cudaSuccess)
        return err;
    const int blocks = (int)std::min<int64_t>(
        (a.M + kGatherThreads / 32 - 1) / (kGatherThreads / 32),
        (int64_t)a.num_sms * 8);
    // the tensor-core GEMM's Q4 form reads its activations in paired
    // order; rank by rank when the GEMM takes every expert
    const bool pairs = ts && !a.q8, by_rank = a.matvec_max_rows == 0;
    void (*copy)(GateUpArgs) =
        pairs ? (by_rank ? gather_rows_kernel<true, true>
                         : gather_rows_kernel<true, false>)
              : (by_rank ? gather_rows_kernel<false, true>
                         : gather_rows_kernel<false, false>);
    if ((err = launch_pdl(copy,
                          dim3((unsigned)blocks), dim3(kGatherThreads),
                          sizeof(int32_t) * (size_t)(a.E + 1), s, a)) !=
        cudaSuccess)
        return err;
    if (ts)
        return launch_gemm_tma(a, a.xg, s);
    return launch_gemm_kernel<true, false>(a, maps, s);
}

}  // namespace q4moe
