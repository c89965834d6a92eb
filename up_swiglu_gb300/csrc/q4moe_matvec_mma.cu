// q4moe_matvec_mma.cu -- grouped Q4 gate/up + SwiGLU for experts with few
// rows (decode, speculative verify), on the warp-level tensor core path.
//
// Same arithmetic as the pages' GATE_UP_SOURCE (page 52, streamed-experts.ts):
// every packed word is read from HBM once per call and serves all of the
// expert's rows in the chunk (the shared-row idea of page 57's
// GATEUP_SHARED_M_SOURCE), the dot products accumulate in f32.
//
// Task = (expert, chunk of up to 8 grouped rows, block of 16 intermediate
// rows).  For one 128-wide K step a thread (group g = lane/4, quad member
// t = lane%4) holds 16 bytes (32 nibbles) of gate and up rows g and 8+g and
// issues sixteen mma.sync.m16n8k16 (bf16 in, f32 accumulate) with
//   A rows 0-7  = gate rows, A rows 8-15 = up rows of the same 8 i,
//   B columns   = the chunk's 8 grouped rows (tokens),
// so the C fragment of a thread already pairs gate and up of one i.
// Weights are dequantised straight into registers: word w gives the four
// bf16x2 {n_j, n_j+4} (j = 0..3) as (w >> 4j) & 0x000F000F placed in the
// mantissa of 128.0 and reduced by 136 (exact).  The K order inside each
// MMA follows that pairing; the activations are staged once per chunk in
// shared memory in the matching order ((0,4,1,5,2,6,3,7) within each group
// of 8) and bank-swizzled so that the B fragments load without conflicts.
// Each thread keeps the weights of its next K steps in flight through a
// shared-memory ring (cp.async) while it multiplies the current ones.  When
// warps split a task's K, their partial sums meet in shared memory in a fixed
// warp order; results are deterministic and a row's bits do not depend on
// the other rows of its chunk.
#include "q4moe_internal.cuh"

namespace q4moe {
namespace {

constexpr int kWarps = 16;
constexpr int kThreads = kWarps * 32;
constexpr int kRowsPerTask = 16;    // intermediate rows (two MMA row tiles)
constexpr int kTok = 8;             // grouped rows per chunk
constexpr int kStepK = 128;         // K per step (16 words per row)

struct Task {
    int e, chunk, blk;
    int p0, nt;                     // first grouped row, rows in the chunk
};

__device__ __forceinline__ int ceil_div(int a, int b) { return (a + b - 1) / b; }

__device__ __forceinline__ int groups_of(int n_e, int max_rows, int GB) {
    return (n_e > 0 && n_e <= max_rows) ? ceil_div(n_e, kTok) * GB : 0;
}

// Group t (in expert-major, chunk-major order) -> expert, chunk, group
// index within the chunk (returned in blk).
__device__ __forceinline__ Task group_of(int t, const int32_t *off,
                                         const int32_t *pre, int E, int GB) {
    int lo = 0, hi = E;
    while (hi - lo > 1) {
        const int mid = (lo + hi) >> 1;
        if (pre[mid] <= t)
            lo = mid;
        else
            hi = mid;
    }
    Task k;
    k.e = lo;
    const int local = t - pre[lo];
    k.chunk = local / GB;
    k.blk = local - k.chunk * GB;
    k.p0 = off[lo] + k.chunk * kTok;
    k.nt = min(kTok, off[lo + 1] - k.p0);
    return k;
}

// Physical 16-byte chunk of logical chunk q of token row n in the staged
// activations (bank swizzle for the B-fragment loads).
__device__ __forceinline__ int xs_chunk(int q, int n) {
    return (q & ~7) | ((q & 7) ^ ((q >> 3) & 1) ^ ((n & 1) << 1));
}

// 8 consecutive 16-bit values (uint4) -> K order (0,4,1,5,2,6,3,7).
__device__ __forceinline__ uint4 permute8(uint4 v) {
    return make_uint4(__byte_perm(v.x, v.z, 0x5410),
                      __byte_perm(v.x, v.z, 0x7632),
                      __byte_perm(v.y, v.w, 0x5410),
                      __byte_perm(v.y, v.w, 0x7632));
}

// The four pairs {n_j - 8, n_{j+4} - 8}, j = 0..3, of one packed word, as
// bf16x2 (nibble in the mantissa of 128.0, minus 136) ...
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

__device__ __forceinline__ void mma_16816(float (&c)[4], uint32_t a0,
                                          uint32_t a1, uint32_t a2,
                                          uint32_t a3, uint32_t b0,
                                          uint32_t b1) {
    asm volatile(
        "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 "
        "{%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, {%0,%1,%2,%3};"
        : "+f"(c[0]), "+f"(c[1]), "+f"(c[2]), "+f"(c[3])
        : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}

// One K step of one warp: w[0..3] = 16 bytes of gate row g, up row g,
// gate row 8+g, up row 8+g; xb = the four 16-byte activation chunks.
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
        word_pairs_bf16(wg0[wd], g0);
        word_pairs_bf16(wu0[wd], u0);
        word_pairs_bf16(wg1[wd], g1);
        word_pairs_bf16(wu1[wd], u1);
        const uint32_t *xw = reinterpret_cast<const uint32_t *>(&xb[wd]);
#pragma unroll
        for (int h = 0; h < 2; ++h) {
            mma_16816(acc[0], g0[2 * h], u0[2 * h], g0[2 * h + 1],
                      u0[2 * h + 1], xw[2 * h], xw[2 * h + 1]);
            mma_16816(acc[1], g1[2 * h], u1[2 * h], g1[2 * h + 1],
                      u1[2 * h + 1], xw[2 * h], xw[2 * h + 1]);
        }
    }
}

// cp.async of 16 bytes global -> shared (bypassing L1) and its waits.
__device__ __forceinline__ void cp16(uint32_t dst, const void *src) {
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(dst),
                 "l"(src)
                 : "memory");
}
__device__ __forceinline__ void cp_commit() {
    asm volatile("cp.async.commit_group;" ::: "memory");
}
template <int N>
__device__ __forceinline__ void cp_wait() {
    asm volatile("cp.async.wait_group %0;" ::"n"(N) : "memory");
}

// Work is handed out in groups: a group is 16/S consecutive blocks of 16
// intermediate rows of one (expert, chunk), one task per slot of S warps;
// the S warps of a slot split the task's K steps (warp kpart takes steps
// kpart, kpart+S, ...).  S = 1 streams whole rows per warp with no barrier
// inside a group; S = 16 spreads the few tasks of a tiny call over all
// warps.  Each thread copies its own weight bytes for the next R steps into
// a shared-memory ring with cp.async and reads back only those bytes, so its
// own cp.async.wait_group is all the synchronisation the ring needs.
template <int S, int R>
__global__ void __launch_bounds__(kThreads, 1)
matvec_mma_kernel(GateUpArgs a, int tok_cap) {
    constexpr int kSlots = kWarps / S;
    extern __shared__ __align__(128) uint8_t smem[];
    const int E = a.E;
    const int H = (int)a.H;
    // [kWarps][R][4][32] x 16 B weight ring, then the staged activations,
    // the reduction buffer (S > 1) and the row offsets
    uint8_t *ring = smem;
    uint8_t *xs = ring + (size_t)kWarps * R * 4 * 32 * 16;
    float4 *red = reinterpret_cast<float4 *>(xs + (size_t)tok_cap * H * 2);
    int32_t *s_off = reinterpret_cast<int32_t *>(
        red + (S > 1 ? kWarps * 32 * 2 : 0));
    int32_t *s_pre = s_off + (E + 1);

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int g = lane >> 2, tq = lane & 3;
    const int slot = warp / S, kpart = warp - slot * S;
    const int IBk = (int)(a.I / kRowsPerTask);
    const int GB = ceil_div(IBk, kSlots);          // groups per chunk
    const int steps = H / kStepK;                  // K steps in a row
    const int spw = ceil_div(steps, S);            // steps per warp per task
    if (a.matvec_last)
        grid_launch_dependents();
    grid_dependency_wait();

    if (!stage_row_offsets(a, s_off))
        return;
    const int32_t mvmax = matvec_limit(a, s_off);
    if (warp == 0) {
        const int per = ceil_div(E, 32);
        const int e0 = lane * per;
        int sum = 0;
        for (int e = e0; e < min(E, e0 + per); ++e)
            sum += groups_of(s_off[e + 1] - s_off[e], mvmax, GB);
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
            run += groups_of(s_off[e + 1] - s_off[e], mvmax, GB);
        }
        if (lane == 31)
            s_pre[E] = incl;
    }
    __syncthreads();
    const int ngroups = s_pre[E];
    const int gr_begin = (int)((int64_t)ngroups * blockIdx.x / gridDim.x);
    const int gr_end = (int)((int64_t)ngroups * (blockIdx.x + 1) / gridDim.x);
    if (gr_begin >= gr_end)
        return;
    const int ngr = gr_end - gr_begin;
    const int total = ngr * spw;                   // this warp's K steps

    auto task_at = [&](int gi) {
        Task k = group_of(gr_begin + gi, s_off, s_pre, E, GB);
        k.blk = k.blk * kSlots + slot;             // this slot's block
        return k;
    };

    // --- copy cursor: R steps ahead of the multiply
    const int64_t row_bytes = a.H / 2;
    int lgi = 0, lm = 0;
    const uint8_t *lg = nullptr, *lu = nullptr;    // gate / up rows of lane
    auto set_copy_task = [&](int gi) {
        const Task t = task_at(gi);
        const uint8_t *slab = expert_slab(a, t.e);
        lg = lu = nullptr;
        if (slab != nullptr && t.blk < IBk) {
            const int64_t off =
                ((int64_t)t.blk * kRowsPerTask + g) * row_bytes + tq * 16 +
                (int64_t)kpart * 64;
            lg = slab + a.gate_w_off + off;
            lu = slab + a.up_w_off + off;
        }
    };
    const uint32_t ring0 =
        static_cast<uint32_t>(__cvta_generic_to_shared(ring)) +
        (uint32_t)(warp * R * 4 * 32 + lane) * 16;
    auto copy_next = [&](int r) {                  // into ring slot r
        if (lgi < ngr) {
            if (lg != nullptr && kpart + S * lm < steps) {
                const int64_t o = (int64_t)lm * (S * 64);
                const uint32_t dst = ring0 + (uint32_t)(r * 4 * 32) * 16;
                cp16(dst, lg + o);
                cp16(dst + 32 * 16, lu + o);
                cp16(dst + 64 * 16, lg + o + 8 * row_bytes);
                cp16(dst + 96 * 16, lu + o + 8 * row_bytes);
            }
            if (++lm == spw) {
                lm = 0;
                if (++lgi < ngr)
                    set_copy_task(lgi);
            }
        }
        cp_commit();                               // one group per step
    };
    set_copy_task(0);
#pragma unroll
    for (int r = 0; r < R; ++r)
        copy_next(r);

    // byte offsets (within the staged activations) of this thread's four
    // B-fragment chunks at K step 0 (step kc adds kc * 256); rows past the
    // chunk read a stale in-bounds row whose output columns are not stored
    const int xrow = min(g, tok_cap - 1);
    int xoff[4];
#pragma unroll
    for (int q4 = 0; q4 < 4; ++q4)
        xoff[q4] = xrow * H * 2 +
                   ((tq >> 1) * 8 +
                    (((tq & 1) * 4 + q4) ^ (tq >> 1) ^ ((xrow & 1) << 1))) *
                       16;

    float acc[2][4];
    int staged_e = -1, staged_chunk = -1;
    Task k{};
    int gi = 0, m = 0;
    const uint4 *myring = reinterpret_cast<const uint4 *>(ring) +
                          (warp * R * 4 * 32 + lane);

    for (int j0 = 0; j0 < total; j0 += R) {
#pragma unroll
        for (int r = 0; r < R; ++r) {
            if (j0 + r >= total)
                break;
            if (m == 0) {
                k = task_at(gi);
                if (k.e != staged_e || k.chunk != staged_chunk) {
                    __syncthreads();      // everyone is done with the old x
                    const int qn = H / 8;
                    for (int idx = tid; idx < k.nt * qn; idx += kThreads) {
                        const int n = idx / qn, q = idx - n * qn;
                        const int64_t tok = row_token(a, k.p0 + n);
                        uint4 v = make_uint4(0, 0, 0, 0);
                        if (tok >= 0)
                            v = __ldg(reinterpret_cast<const uint4 *>(
                                          a.x + tok * a.H) + q);
                        *reinterpret_cast<uint4 *>(
                            xs + (int64_t)n * H * 2 + xs_chunk(q, n) * 16) =
                            permute8(v);
                    }
                    staged_e = k.e;
                    staged_chunk = k.chunk;
                    __syncthreads();
                }
#pragma unroll
                for (int i = 0; i < 2; ++i)
                    acc[i][0] = acc[i][1] = acc[i][2] = acc[i][3] = 0.0f;
            }
            cp_wait<R - 1>();             // this step's copies have landed
            const int kc = kpart + S * m;
            if (kc < steps && k.blk < IBk) {
                uint4 w[4], xb[4];
#pragma unroll
                for (int c = 0; c < 4; ++c)
                    w[c] = myring[(r * 4 + c) * 32];
                const uint8_t *xk = xs + kc * 256;
#pragma unroll
                for (int q4 = 0; q4 < 4; ++q4)
                    xb[q4] = *reinterpret_cast<const uint4 *>(xk + xoff[q4]);
                step_mma(acc, w, xb);
            }
            copy_next(r);
            if (m == spw - 1) {
                // the task is complete: sum over the slot's warps
                if (S > 1) {
                    red[(warp * 32 + lane) * 2] = make_float4(
                        acc[0][0], acc[0][1], acc[0][2], acc[0][3]);
                    red[(warp * 32 + lane) * 2 + 1] = make_float4(
                        acc[1][0], acc[1][1], acc[1][2], acc[1][3]);
                    __syncthreads();
                    if (kpart == 0) {
                        for (int w = 1; w < S; ++w) {
#pragma unroll
                            for (int i = 0; i < 2; ++i) {
                                const float4 v =
                                    red[((warp + w) * 32 + lane) * 2 + i];
                                acc[i][0] += v.x;
                                acc[i][1] += v.y;
                                acc[i][2] += v.z;
                                acc[i][3] += v.w;
                            }
                        }
                    }
                    __syncthreads();
                }
                const uint8_t *slab = expert_slab(a, k.e);
                if (kpart == 0 && k.blk < IBk && slab != nullptr) {
#pragma unroll
                    for (int i = 0; i < 2; ++i) {
                        const int64_t row =
                            (int64_t)k.blk * kRowsPerTask + 8 * i + g;
                        const float sg = reinterpret_cast<const float *>(
                            slab + a.gate_s_off)[row];
                        const float su = reinterpret_cast<const float *>(
                            slab + a.up_s_off)[row];
#pragma unroll
                        for (int jj = 0; jj < 2; ++jj) {
                            const int n = 2 * tq + jj;
                            if (n < k.nt) {
                                const float g32 = __fmul_rn(acc[i][jj], sg);
                                const float u32 =
                                    __fmul_rn(acc[i][2 + jj], su);
                                const int64_t o =
                                    (int64_t)(k.p0 + n) * a.I + row;
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
            if (++m == spw) {
                m = 0;
                ++gi;
            }
        }
    }
    cp_wait<0>();
}

template <int S, int R>
cudaError_t launch_split(const GateUpArgs &a, size_t smem, int tok_cap,
                         cudaStream_t s) {
    cudaError_t err = cudaFuncSetAttribute(
        matvec_mma_kernel<S, R>, cudaFuncAttributeMaxDynamicSharedMemorySize,
        (int)smem);
    if (err != cudaSuccess)
        return err;
    return launch_pdl(matvec_mma_kernel<S, R>, dim3((unsigned)a.num_sms),
                      dim3(kThreads), smem, s, a, tok_cap);
}

size_t matvec_smem(const GateUpArgs &a, int S, int R, int tok_cap) {
    return (size_t)kWarps * R * 4 * 32 * 16 + (size_t)tok_cap * a.H * 2 +
           (S > 1 ? sizeof(float4) * kWarps * 32 * 2 : 0) +
           sizeof(int32_t) * 2 * (size_t)(a.E + 1);
}

constexpr size_t kSmemLimit = 227 * 1024 - 1024;  // room for static smem

}  // namespace

bool matvec_mma_supported(const GateUpArgs &a) {
    const int tok_cap = (int)std::min<int64_t>(kTok, a.M);
    return a.H % kStepK == 0 && a.I % kRowsPerTask == 0 &&
           a.gate_w_off % 16 == 0 && a.up_w_off % 16 == 0 &&
           matvec_smem(a, 16, 2, tok_cap) <= kSmemLimit &&
           matvec_smem(a, 1, 2, tok_cap) <= kSmemLimit;
}

// Few grouped rows (a tiny call) -> split K over all 16 warps; otherwise
// whole tasks per warp.  The ring is 4 steps deep when shared memory
// allows, else 2.
cudaError_t launch_matvec_mma(const GateUpArgs &a, cudaStream_t s) {
    const int tok_cap = (int)std::min<int64_t>(kTok, a.M);
    if (a.M < 16) {
        if (matvec_smem(a, 16, 4, tok_cap) <= kSmemLimit)
            return launch_split<16, 4>(a, matvec_smem(a, 16, 4, tok_cap),
                                       tok_cap, s);
        return launch_split<16, 2>(a, matvec_smem(a, 16, 2, tok_cap),
                                   tok_cap, s);
    }
    if (matvec_smem(a, 1, 4, tok_cap) <= kSmemLimit)
        return launch_split<1, 4>(a, matvec_smem(a, 1, 4, tok_cap), tok_cap,
                                  s);
    return launch_split<1, 2>(a, matvec_smem(a, 1, 2, tok_cap), tok_cap, s);
}

}  // namespace q4moe
