// q4moe_gemm_tma.cu -- grouped Q4/Q8 gate/up + SwiGLU (and the down
// projection) on the tcgen05 tensor core, the token rows moved by TMA.
//
// The same arithmetic as the page's matvec (page 52, streamed-experts.ts,
// GATE_UP_SOURCE, and DOWN_SOURCE for the down projection), in the
// large-batch form for sm_103a:
//
//  tile   = 128 rows of each of the tile's two weight matrices (gate and
//           up of the same 128 intermediate rows; for the down projection
//           two blocks of 128 output rows of the one matrix) x up to 256 of
//           the expert's grouped rows;
//  A      = the tile's packed weights, each of 8 warps streaming its rows
//           (one row of one matrix per thread, a 64-K block by one 256-bit
//           load for nibbles, two for bytes) through a register ring four
//           64-K blocks deep (two for bytes), dequantised (nibble - 8 or the
//           signed byte, exact in bf16) into shared memory in the 128-byte
//           swizzled K-major layout, 64 K per stage, four stages;
//  B      = the tile's token rows (the grouped copy of x, or mid), 64 K per
//           stage in the same layout, at most five TMA boxes a stage, three
//           stages; for Q4 gate/up the copy holds each chunk of 8
//           activations in the paired order {0,4,1,5,2,6,3,7}, the order
//           in which A's cheapest dequantisation yields the weights;
//  D      = two f32 accumulators in tensor memory (gate: columns 0..N-1,
//           up: columns 256..256+N-1), lane = weight row;
//  tail   = row scales, bf16 rounding and the SwiGLU chain on packed pairs
//           of columns (one conversion rounds two values, two packed bf16
//           multiplies give two outputs; the bf16 sigmoid from the
//           library's constant table), or the down projection's scale and
//           rounding.
//
// Measured choices (prefill workload, traces of one CTA, steps in ms):
//  * the weights come 32 bytes per load instruction (ld.global.nc.v8):
//    Q4 0.895 -> 0.862, Q8 1.162 -> 0.998 against two 16-byte loads (half
//    the load instructions, and half the L1 lookups for rows that each
//    sit in their own line); and without allocating in L1, which then
//    keeps the sigmoid table: Q4 0.855 -> ~0.81, Q8 0.990 -> ~0.89 (with
//    16-byte loads the same hint had cost 0.93 -> 1.43);
//  * each dequantisation thread prefetches its row's line 2 blocks past
//    its register ring into L2: the ring's loads then wait on L2, not HBM
//    (0.977 -> 0.939 at 4 blocks with 16-byte loads; the bulk prefetch
//    instead, queued on the TMA unit, 1.37-1.59);
//  * the weights do not go through TMA: the SM's one TMA unit then also
//    serves the token rows, and with the HBM-cold weight boxes in its queue
//    the MMA thread waited ~800 cycles per stage for token rows (~100 with
//    the weights on ordinary loads);
//  * one thread issues every MMA and the tile's pace is its issue rate
//    (about 90 cycles per tcgen05.mma, 55 per commit, 300 per mbarrier
//    try_wait), so it waits by spinning on test_wait and each of its waits
//    covers a whole 64-K stage (8 MMAs).
//
// Warp roles (640 threads, one CTA per SM, persistent over tiles).  Warp
// w issues from SM sub-partition w % 4; the MMA thread shares its
// sub-partition with no dequantisation warp (measured: sharing one with two
// of them doubled the MMA thread's cost per stage):
//   0     TMEM allocation and the single thread that issues the MMAs
//   4     token-row producer (one thread issues the TMA boxes)
//   8     idle
//   1-3, 5-7, 9-10  dequantisation (the k-th of these warps takes rows
//         32*(k%4).. of matrix k/4, 0: gate, 1: up, one row per thread)
//   11    idle
//   12-19 epilogue: warp w reads TMEM lanes 32*(w%4).. (a warp reaches
//         only its own quarter of the lanes); (w-12)/4 picks the
//         8-column chunks it handles
//
// Every wait on an mbarrier is bounded; on time-out the CTA raises
// Q4MOE_DEV_WAIT_TIMEOUT, drains its copies and MMAs, frees TMEM and exits.
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

constexpr int BM = 128;                  // rows of each matrix per tile
constexpr int BK = 64;                   // K per A and B stage
constexpr int NMAX = 256;                // grouped rows per tile
constexpr int A_MAT = BM * BK * 2;       // 16 KB of bf16 per matrix
constexpr int A_STAGE = 2 * A_MAT;       // 32 KB
constexpr int AS = 4;                    // A stages
constexpr int B_BYTES = NMAX * BK * 2;   // 32 KB
constexpr int BS = 3;                    // token-row stages
constexpr int RING_BYTES = AS * A_STAGE + BS * B_BYTES;
constexpr int kThreads = 640;
constexpr int kMmaWarp = 0;
constexpr int kTokWarp = 4;
constexpr int kDeqWarps = 8;
constexpr int kEpiWarp0 = 12;
constexpr int kEpiWarps = 8;
constexpr uint32_t kTmemCols = 512;
constexpr uint32_t kUpCol = 256;
constexpr uint64_t kTimeoutNs = 4000000000ull;
constexpr int kBoxLevels = 5;            // token boxes of 256 >> level rows

// Index (0..7) of dequantisation warp w, or -1: the warps of sub-partitions
// 1-3 below the epilogue warps, but for 11.
__device__ __forceinline__ int deq_index(int w) {
    if (w >= 11 || (w & 3) == 0)
        return -1;
    return w - 1 - (w >> 2);
}

static_assert(A_STAGE % 1024 == 0 && B_BYTES % 1024 == 0,
              "stages must keep the 1024-byte alignment of the swizzle atoms");

struct XgMaps {
    CUtensorMap m[kBoxLevels];
};

struct Ctl {
    uint64_t a_full[AS];
    uint64_t a_empty[AS];
    uint64_t b_full[BS];
    uint64_t b_empty[BS];
    uint64_t tmem_full;
    uint64_t tmem_empty;
    uint64_t drain;
    uint32_t tmem_base;
    int abort;
    int bad_offsets;
    int b_issued;
};

constexpr size_t smem_bytes(int E) {
    return 1024 + (size_t)RING_BYTES + sizeof(Ctl) +
           2 * sizeof(int32_t) * (size_t)(E + 1) + 16;
}

struct Tile {
    int e, iblk, row0, nvalid, n;
};

__device__ __forceinline__ int ceil_div(int a, int b) { return (a + b - 1) / b; }

// Rows of expert e are split into ceil(n/256) chunks of equal size rounded
// up to 16.
__device__ __forceinline__ int chunk_rows(int n_e) {
    const int nch = ceil_div(n_e, NMAX);
    return ceil_div(ceil_div(n_e, nch), 16) * 16;
}

__device__ __forceinline__ int chunks_of(int n_e, int32_t mvmax) {
    return (n_e > mvmax && n_e > 0) ? ceil_div(n_e, NMAX) : 0;
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

// One packed word (8 nibbles, K order) -> 8 bf16 (nibble - 8) in the paired
// order {k, k+4}: output pair j holds nibbles j and j+4, which sit at bits
// 4j and 4j+16 of the word, so one shift and one mask-and-or place both
// under 128.0 (0x4300) before the subtraction of 136 — two operations per
// word fewer than the K order below.  The token rows' copy puts each chunk
// of 8 activations in the same order, so the products pair up as before.
__device__ __forceinline__ uint4 nibbles_bf16_pairs(uint32_t w) {
    const __nv_bfloat162 k136 =
        __halves2bfloat162(__ushort_as_bfloat16((unsigned short)0x4308),
                           __ushort_as_bfloat16((unsigned short)0x4308));
    uint32_t r[4];
#pragma unroll
    for (int j = 0; j < 4; ++j) {
        const uint32_t v = ((w >> (4 * j)) & 0x000F000Fu) | 0x43004300u;
        __nv_bfloat162 b = *reinterpret_cast<const __nv_bfloat162 *>(&v);
        b = __hsub2(b, k136);
        r[j] = *reinterpret_cast<const uint32_t *>(&b);
    }
    return make_uint4(r[0], r[1], r[2], r[3]);
}

// One packed word (8 nibbles, K order) -> 8 bf16 (nibble - 8) in K order:
// each output pair (2j, 2j+1) is byte j of the word split into its two
// nibbles, placed in the low mantissa bits of 128.0 (0x4300) and then
// reduced by 136 (exact: the results are the integers -8..7).
__device__ __forceinline__ uint4 nibbles_bf16(uint32_t w) {
    const uint32_t ws = w >> 4;
    const __nv_bfloat162 k136 =
        __halves2bfloat162(__ushort_as_bfloat16((unsigned short)0x4308),
                           __ushort_as_bfloat16((unsigned short)0x4308));
    uint32_t r[4];
#pragma unroll
    for (int j = 0; j < 4; ++j) {
        const uint32_t v =
            (__byte_perm(w, ws, (uint32_t)(j | ((4 + j) << 8))) &
             0x000F000Fu) | 0x43004300u;
        __nv_bfloat162 b = *reinterpret_cast<const __nv_bfloat162 *>(&v);
        b = __hsub2(b, k136);
        r[j] = *reinterpret_cast<const uint32_t *>(&b);
    }
    return make_uint4(r[0], r[1], r[2], r[3]);
}

// Two signed bytes given as t = {b0, 0x43, b1, 0x43} -> bf16x2 {b0, b1},
// exact: under the exponent byte 0x43 the low seven bits m read 128 + m and
// the sign bit 128 or 256; b = (128 + m) - (128 + 128 * sign).
__device__ __forceinline__ uint32_t byte_pair(uint32_t t) {
    const uint32_t m = t & 0x437F437Fu, c = t & 0x43804380u;
    const __nv_bfloat162 r =
        __hsub2(*reinterpret_cast<const __nv_bfloat162 *>(&m),
                *reinterpret_cast<const __nv_bfloat162 *>(&c));
    return *reinterpret_cast<const uint32_t *>(&r);
}

// Two words of four signed bytes each (K order) -> 8 bf16, exact.
__device__ __forceinline__ uint4 bytes_bf16(uint32_t w0, uint32_t w1) {
    return make_uint4(byte_pair(__byte_perm(w0, 0x43434343u, 0x4140)),
                      byte_pair(__byte_perm(w0, 0x43434343u, 0x4342)),
                      byte_pair(__byte_perm(w1, 0x43434343u, 0x4140)),
                      byte_pair(__byte_perm(w1, 0x43434343u, 0x4342)));
}

// 32 bytes of weights (two uint4) by one 256-bit load that leaves L1 to
// the epilogue's sigmoid table (each 32-byte sector is read once); p must
// be 32-byte aligned (gemm_tma_supported checks the sections; rows hold a
// whole number of 64-K blocks, a multiple of 32 bytes).
__device__ __forceinline__ void ldg_32(const uint4 *p, uint4 &lo, uint4 &hi) {
    asm("ld.global.nc.L1::no_allocate.v8.u32 "
        "{%0,%1,%2,%3,%4,%5,%6,%7}, [%8];"
        : "=r"(lo.x), "=r"(lo.y), "=r"(lo.z), "=r"(lo.w), "=r"(hi.x),
          "=r"(hi.y), "=r"(hi.z), "=r"(hi.w)
        : "l"(p));
}

// Byte offset of 16-byte chunk c (0..7) of row r in a 128-byte-swizzled
// K-major tile.
__device__ __forceinline__ uint32_t sw128_offset(int r, int c) {
    return (uint32_t)((r >> 3) * 1024 + (r & 7) * 128 + ((c ^ (r & 7)) << 4));
}

template <bool kDown, bool kQ8>
__global__ void __launch_bounds__(kThreads, 1)
gemm_tma_kernel(GateUpArgs a, const __grid_constant__ XgMaps xg_maps) {
    extern __shared__ uint8_t smem_raw[];
    uint8_t *smem = reinterpret_cast<uint8_t *>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    uint8_t *a_ring = smem;
    Ctl *ctl = reinterpret_cast<Ctl *>(smem + (size_t)RING_BYTES);
    int32_t *s_off = reinterpret_cast<int32_t *>(ctl + 1);
    int32_t *s_pre = s_off + (a.E + 1);

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int E = a.E;
    const int IB = gemm_row_tiles(a);        // tiles over the output rows
    const int KB = (int)(a.H / BK);          // A/B stages per tile
    const int64_t hi_row = kDown ? BM : 0;   // first row of the second matrix
    const int64_t tile_rows = kDown ? 2 * BM : BM;

    if (tid == 0) {
        for (int s = 0; s < AS; ++s) {
            mbar_init(&ctl->a_full[s], kDeqWarps);
            mbar_init(&ctl->a_empty[s], 1);
        }
        for (int s = 0; s < BS; ++s) {
            mbar_init(&ctl->b_full[s], 1);
            mbar_init(&ctl->b_empty[s], 1);
        }
        mbar_init(&ctl->tmem_full, 1);
        mbar_init(&ctl->tmem_empty, kEpiWarps);
        mbar_init(&ctl->drain, 1);
        ctl->abort = 0;
        ctl->bad_offsets = 0;
        ctl->b_issued = 0;
        fence_mbar_init();
        for (int l = 0; l < kBoxLevels; ++l)
            tma_desc_prefetch(&xg_maps.m[l]);
    }
    if (warp == kMmaWarp) {
        tmem_alloc(&ctl->tmem_base, kTmemCols);
        tmem_relinquish();
    }
    grid_dependency_wait();
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
        for (int e = e0; e < min(E, e0 + per); ++e)
            sum += IB * chunks_of(s_off[e + 1] - s_off[e], mvmax);
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
            run += IB * chunks_of(s_off[e + 1] - s_off[e], mvmax);
        }
        if (lane == 31)
            s_pre[E] = incl;
    }
    __syncthreads();
    const int ntiles = offsets_ok ? s_pre[E] : 0;
    const uint32_t tmem = ctl->tmem_base;
    volatile int *abort = &ctl->abort;
    const uint32_t a_ring0 = smem_u32(a_ring);
    const uint32_t b_ring0 = a_ring0 + AS * A_STAGE;

    if (warp == kTokWarp) {
        // ------------------------------------------- token rows via TMA
        if (lane == 0) {
            uint32_t g = 0;
            for (int t = blockIdx.x; t < ntiles && !*abort; t += gridDim.x) {
                const Tile ti = tile_of(t, s_off, s_pre, E, IB);
                bool ok = true;
                for (int kb = 0; kb < KB; ++kb, ++g) {
                    const uint32_t s = g % BS;
                    if (!wait_phase(&ctl->b_empty[s], ((g / BS) & 1) ^ 1,
                                    abort, a.status)) {
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
            ctl->b_issued = (int)g;
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
                if (!wait_spin(&ctl->tmem_empty, (it & 1) ^ 1, abort,
                               a.status))
                    break;
                tc_fence_after();
                bool ok = true;
                for (int kb = 0; kb < KB; ++kb, ++g) {
                    const uint32_t sa = g % AS, sb = g % BS;
                    if (!wait_spin(&ctl->b_full[sb], (g / BS) & 1, abort,
                                   a.status) ||
                        !wait_spin(&ctl->a_full[sa], (g / AS) & 1, abort,
                                   a.status)) {
                        ok = false;
                        break;
                    }
                    tc_fence_after();
                    const uint32_t ag = a_ring0 + sa * A_STAGE;
                    const uint32_t au = ag + A_MAT;
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
                const uint64_t t0 = globaltimer_ns();
                while (!mbar_try_wait(&ctl->drain, 0) &&
                       globaltimer_ns() - t0 < kTimeoutNs) {
                }
            }
        }
    } else if (deq_index(warp) >= 0) {
        // ------------------------------------------- weight dequantisation
        const int k = deq_index(warp);
        const int m = k >> 2;
        const int r = (k & 3) * 32 + lane;   // row in the tile
        // a 64-K block of one row: 32 bytes of nibbles or 64 of signed bytes,
        // kDepth blocks in flight
        constexpr int kVecs = kQ8 ? 4 : 2;
        constexpr int kDepth = kQ8 ? 2 : 4;
        constexpr int kBlocksPerLine = 128 / (kVecs * 16);
        // measured with 32-byte loads: 2 (Q4 0.8555 ms, Q8 0.991) against
        // 4 (0.8587, 0.996) and 8 (0.862, 1.010)
        constexpr int kPrefetch = 2;
        const int64_t rb = weight_row_bytes(a, a.H);
        const uint32_t z = kQ8 ? 0u : 0x88888888u;    // weight zero
        const uint4 kZero = make_uint4(z, z, z, z);
        static_assert(kDepth % 2 == 0 && AS % 2 == 0, "blocks go in pairs");
        uint32_t g = 0;
        bool ok = true;
        for (int t = blockIdx.x; t < ntiles && ok && !*abort;
             t += gridDim.x) {
            const Tile ti = tile_of(t, s_off, s_pre, E, IB);
            const int64_t row = (int64_t)ti.iblk * tile_rows + r +
                                (m ? hi_row : 0);
            // the down projection's second matrix may end before the tile
            const bool rok = !kDown || row < a.I;
            const uint4 *src = reinterpret_cast<const uint4 *>(
                a.base + (int64_t)ti.e * a.stride +
                (m ? a.up_w_off : a.gate_w_off) + row * rb);
            uint4 ring[kDepth][kVecs];
#pragma unroll
            for (int d = 0; d < kDepth; ++d) {
#pragma unroll
                for (int v = 0; v < kVecs; v += 2) {
                    if (rok && d < KB) {
                        ldg_32(src + kVecs * d + v, ring[d][v], ring[d][v + 1]);
                    } else {
                        ring[d][v] = kZero;
                        ring[d][v + 1] = kZero;
                    }
                }
            }
            // two 64-K blocks per round (one proxy fence for both)
            for (int kb0 = 0; kb0 < KB && ok; kb0 += kDepth) {
#pragma unroll
                for (int d = 0; d < kDepth; d += 2) {
                    const int kb = kb0 + d;
                    if (kb >= KB)
                        break;
                    const int nb = min(2, KB - kb);    // blocks this round
                    uint8_t *dst[2];
                    for (int q = 0; q < nb; ++q) {
                        const uint32_t sa = (g + q) % AS;
                        if (!wait_phase(&ctl->a_empty[sa],
                                        (((g + q) / AS) & 1) ^ 1, abort,
                                        a.status)) {
                            ok = false;
                            break;
                        }
                        dst[q] = a_ring + sa * A_STAGE + m * A_MAT;
                    }
                    if (!ok)
                        break;
#pragma unroll
                    for (int q = 0; q < 2; ++q) {
                        if (q >= nb)
                            break;
                        const uint32_t *wd =
                            reinterpret_cast<const uint32_t *>(&ring[d + q][0]);
#pragma unroll
                        for (int c = 0; c < 8; ++c) {
                            // 16-byte chunk c of the row's 64 K: 8 values
                            const uint4 v = kQ8 ? bytes_bf16(wd[2 * c],
                                                             wd[2 * c + 1])
                                                : kDown ? nibbles_bf16(wd[c])
                                                  : nibbles_bf16_pairs(wd[c]);
                            *reinterpret_cast<uint4 *>(dst[q] +
                                                       sw128_offset(r, c)) = v;
                        }
                        const int kn = kb + q + kDepth;
                        if (kn < KB && rok) {
#pragma unroll
                            for (int v = 0; v < kVecs; v += 2)
                                ldg_32(src + kVecs * kn + v, ring[d + q][v],
                                       ring[d + q][v + 1]);
                        }
                        // the row's 128-byte line kPrefetch blocks past
                        // the ring into L2, so the ring's loads find it
                        // there (a plain prefetch: the bulk form goes
                        // through the TMA unit the token rows need)
                        const int kp = kn + kPrefetch;
                        if (kp < KB && rok && (kp & (kBlocksPerLine - 1)) == 0)
                            prefetch_l2_line(src + kVecs * kp);
                    }
                    fence_proxy_async_smem();
                    __syncwarp();
                    if (lane == 0)
                        for (int q = 0; q < nb; ++q)
                            mbar_arrive(&ctl->a_full[(g + q) % AS]);
                    g += nb;
                }
            }
        }
    } else if (warp >= kEpiWarp0) {
        // ------------------------------------------------------- epilogue
        const int quad = warp & 3, half = (warp - kEpiWarp0) >> 2;
        uint32_t it = 0;
        for (int t = blockIdx.x; t < ntiles && !*abort;
             t += gridDim.x, ++it) {
            const Tile ti = tile_of(t, s_off, s_pre, E, IB);
            if (!wait_phase(&ctl->tmem_full, it & 1, abort, a.status))
                break;
            tc_fence_after();
            const uint8_t *slab = a.base + (int64_t)ti.e * a.stride;
            const int64_t i = (int64_t)ti.iblk * tile_rows + quad * 32 + lane;
            const bool hi_ok = !kDown || i + hi_row < a.I;
            const float sg = reinterpret_cast<const float *>(
                slab + a.gate_s_off)[i];
            const float su = hi_ok ? reinterpret_cast<const float *>(
                                         slab + a.up_s_off)[i + hi_row]
                                   : 0.0f;
            const uint32_t tl = tmem + ((uint32_t)(quad * 32) << 16);
            // 8-column chunks, alternating between the two warps of the
            // quarter; the loads of the next chunk are in flight while
            // this one is finished
            constexpr int kC = 8;
            uint32_t gv[kC], uv[kC];
            int c0 = half * kC;
            if (c0 < ti.n) {
                tmem_ld8(tl + (uint32_t)c0, gv);
                tmem_ld8(tl + kUpCol + (uint32_t)c0, uv);
            }
            tmem_ld_wait_regs(gv, uv);
            for (; c0 < ti.n; c0 += 2 * kC) {
                float g32[kC], u32[kC];
#pragma unroll
                for (int jj = 0; jj < kC; ++jj) {
                    g32[jj] = __fmul_rn(__uint_as_float(gv[jj]), sg);
                    u32[jj] = __fmul_rn(__uint_as_float(uv[jj]), su);
                }
                const int cn = c0 + 2 * kC;
                if (cn < ti.n) {
                    tmem_ld8(tl + (uint32_t)cn, gv);
                    tmem_ld8(tl + kUpCol + (uint32_t)cn, uv);
                }
                const int64_t o0 = (int64_t)(ti.row0 + c0) * a.I + i;
                if (kDown) {
                    // out = bf16(sum * scale) for both halves, rounded in
                    // packed pairs of columns
                    uint32_t lo[kC / 2], hi[kC / 2];
#pragma unroll
                    for (int jj = 0; jj < kC; jj += 2) {
                        lo[jj / 2] = bf16x2_rn(g32[jj], g32[jj + 1]);
                        hi[jj / 2] = bf16x2_rn(u32[jj], u32[jj + 1]);
                    }
#pragma unroll
                    for (int jj = 0; jj < kC; ++jj) {
                        if (c0 + jj < ti.nvalid) {
                            const int sh = (jj & 1) * 16;
                            const int64_t oi = o0 + (int64_t)jj * a.I;
                            a.out[oi] = (uint16_t)(lo[jj / 2] >> sh);
                            if (a.gate_f32)
                                a.gate_f32[oi] = g32[jj];
                            if (hi_ok) {
                                a.out[oi + hi_row] =
                                    (uint16_t)(hi[jj / 2] >> sh);
                                if (a.gate_f32)
                                    a.gate_f32[oi + hi_row] = u32[jj];
                            }
                        }
                    }
                } else {
                    // packed pairs of columns: gateT and upT by one
                    // conversion each, the sigmoids from the table, the
                    // two products by packed bf16 multiplies
                    uint32_t ob[kC / 2];
#pragma unroll
                    for (int jj = 0; jj < kC; jj += 2) {
                        const uint32_t g2 = bf16x2_rn(g32[jj], g32[jj + 1]);
                        const uint32_t s2 =
                            (uint32_t)sigmoid_bf16_table(a.sigmoid,
                                                         (uint16_t)g2) |
                            ((uint32_t)sigmoid_bf16_table(
                                 a.sigmoid, (uint16_t)(g2 >> 16))
                             << 16);
                        ob[jj / 2] = swiglu_tail_pair(
                            g2, s2, bf16x2_rn(u32[jj], u32[jj + 1]));
                    }
#pragma unroll
                    for (int jj = 0; jj < kC; ++jj) {
                        const uint16_t o =
                            (uint16_t)(ob[jj / 2] >> ((jj & 1) * 16));
                        if (c0 + jj < ti.nvalid) {
                            const int64_t oi = o0 + (int64_t)jj * a.I;
                            a.out[oi] = o;
                            if (a.gate_f32)
                                a.gate_f32[oi] = g32[jj];
                            if (a.up_f32)
                                a.up_f32[oi] = u32[jj];
                        }
                    }
                }
                tmem_ld_wait_regs(gv, uv);
            }
            tc_fence_before();
            __syncwarp();
            if (lane == 0)
                mbar_arrive(&ctl->tmem_empty);
        }
    }

    tc_fence_before();
    __syncthreads();
    // copies still in flight (only after a time-out): the last issued
    if (tid == 0 && *abort) {
        const int gb = ctl->b_issued;
        for (int g = max(0, gb - BS); g < gb; ++g)
            drain_phase(&ctl->b_full[g % BS], (g / BS) & 1);
    }
    __syncthreads();
    if (warp == kMmaWarp) {
        __syncwarp();
        tc_fence_after();
        tmem_dealloc(tmem, kTmemCols);
    }
}

// Tensor maps of the token rows bf16 [M][H] (the grouped copy of x, or
// mid): boxes of 64 columns (128 bytes) x 256 >> level rows, 128-byte
// swizzle, rows past M read as zero.
cudaError_t encode_token_maps(const GateUpArgs &a, const uint16_t *rows,
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

template <bool kDown, bool kQ8>
cudaError_t launch_fmt(const GateUpArgs &a, const uint16_t *rows,
                       cudaStream_t s) {
    XgMaps maps;
    memset(&maps, 0, sizeof maps);
    cudaError_t err = encode_token_maps(a, rows, &maps);
    if (err != cudaSuccess)
        return err;
    const size_t smem = smem_bytes(a.E);
    err = cudaFuncSetAttribute(gemm_tma_kernel<kDown, kQ8>,
                               cudaFuncAttributeMaxDynamicSharedMemorySize,
                               (int)smem);
    if (err != cudaSuccess)
        return err;
    return launch_pdl(gemm_tma_kernel<kDown, kQ8>, dim3((unsigned)a.num_sms),
                      dim3(kThreads), smem, s, a, maps);
}

}  // namespace

// This GEMM takes slabs at base + e * stride whose weight rows hold a whole
// number of 64-K stages, with 32-byte aligned weight sections (its weight
// loads are 32 bytes wide; the slab base and stride are multiples of
// Q4MOE_SLAB_ALIGNMENT).
bool gemm_tma_supported(const GateUpArgs &a) {
    static_assert(Q4MOE_SLAB_ALIGNMENT % 32 == 0, "32-byte weight loads");
    return a.slab_ptrs == nullptr && a.H % BK == 0 &&
           a.gate_w_off % 32 == 0 && a.up_w_off % 32 == 0 &&
           (reinterpret_cast<uintptr_t>(a.base) & 31) == 0 &&
           a.H < (1ll << 31) && a.I < (1ll << 31) &&
           smem_bytes(a.E) <= 227 * 1024 && tensor_map_encoder() != nullptr;
}

// Launch the kernel on token rows `rows` (bf16 [M][H] in grouped order).
cudaError_t launch_gemm_tma(const GateUpArgs &a, const uint16_t *rows,
                            cudaStream_t s) {
    if (a.down)
        return a.q8 ? launch_fmt<true, true>(a, rows, s)
                    : launch_fmt<true, false>(a, rows, s);
    return a.q8 ? launch_fmt<false, true>(a, rows, s)
                : launch_fmt<false, false>(a, rows, s);
}

}  // namespace q4moe
