/*
 * q4moe.h -- C ABI of the fused 4-bit MoE expert gate/up projection with
 * SwiGLU for one NVIDIA GB300 GPU (sm_103a), with the down projection that
 * completes the expert MLP, the signed 8-bit weight format of the same page
 * and trellis-coded (QTIP 1MAD) experts of pages 54 and 57
 * (q4moe_trellis_gate_up_swiglu, formula at its declaration).
 *
 * The operation follows "@mlx-bun/inference 0.0.0-stage -> 1.0.0", page 52,
 * src/kernels/glm52/streamed-experts.ts, GATE_UP_SOURCE (and the
 * Glm52CanonicalMetalExecutor around it), with the expert slot layout of
 * page 51, src/kernels/glm52/layout.ts, and the bf16 rounding of page 54,
 * src/kernels/trellis/codebook.ts, trellis_bf16.  For every grouped row p of
 * expert e, token t = token_to_expert_map[p], and output row i < I:
 *
 *   G  = sum_k (nib(gate_w[e][i][k/8], k%8) - 8) * x[t][k]      (f32 accumulate)
 *   U  = the same over up_w
 *   gateT = bf16(G * gate_s[e][i]),  upT = bf16(U * up_s[e][i])
 *   sigT  = bf16(1 / (1 + exp(-gateT)))       (f32 chain, no flush to zero)
 *   siluT = bf16(gateT * sigT)
 *   out[p][i] = bf16(siluT * upT)
 *
 * where nib(w, j) = (w >> 4j) & 0xF and bf16() rounds to nearest, ties to
 * even.  Summation order is not fixed by the pages: f32 gate/up agree with
 * an f64 accumulation to about 1e-5 relative; with integer activations in
 * [-8, 8] and power-of-two scales every sum is exact and the output is
 * bit-exact.
 *
 * The down projection of the same page (DOWN_SOURCE), which the page's
 * executor runs on the gate/up output mid of the same expert slot, completes
 * the expert MLP: for output row h < H,
 *
 *   out[p][h] = bf16(f32(sum_k (nib(down_w[e][h][k/8], k%8) - 8) * mid[p][k])
 *                    * down_s[e][h])
 *
 * (q4moe_down_proj; q4moe_expert_mlp runs both).
 *
 * Conventions for every entry point:
 *  - Return 0 (Q4MOE_OK) or a negative Q4MOE_ERR_* code; no C++ exception
 *    crosses the ABI.  q4moe_last_error() gives the calling thread's message
 *    for its last failure.
 *  - "device" pointers are CUDA device (or managed) memory of the current
 *    device; "host" pointers are ordinary host memory.  Every buffer is
 *    borrowed: the caller owns it and keeps it alive until the work queued
 *    on `stream` has completed.
 *  - GPU entry points are asynchronous on `stream`, allocate no memory and
 *    never synchronise the host (q4moe_device_status excepted).  The bf16
 *    sigmoid of every bf16 value (128 KB per tail) is constant data of the
 *    library image, so no call launches set-up work; the first call on a
 *    device only looks up the device addresses of that table and of the
 *    status word (host queries).
 *    Argument errors the host can see are returned before anything is
 *    launched.  Inconsistent data that only the
 *    GPU can see (row offsets, token indices, expert ids, slab pointers) sets
 *    a bit in the device status word (Q4MOE_DEV_*) and the affected rows are
 *    skipped; read it with q4moe_device_status().  Nothing traps the GPU.
 *  - Only sm_103 devices are accepted (Q4MOE_ERR_DEVICE otherwise).
 */
#ifndef Q4MOE_H_
#define Q4MOE_H_

#include <stdint.h>
#include <cuda_runtime_api.h>

#ifdef __cplusplus
extern "C" {
#endif

#define Q4MOE_ABI_VERSION 8

/* Slab base addresses and strides must be multiples of this (the pages use
 * 16 KiB, a multiple, for zero-copy residency slots; page 51 layout.ts). */
#define Q4MOE_SLAB_ALIGNMENT 4096

/* Most experts one call accepts (row offsets are staged on chip). */
#define Q4MOE_MAX_EXPERTS 1024

/* ---- status codes ------------------------------------------------------ */
#define Q4MOE_OK 0
#define Q4MOE_ERR_INVALID_ARG (-1) /* null pointer, bad size or dimension  */
#define Q4MOE_ERR_ALIGNMENT (-2)   /* slab base/stride/section misaligned  */
#define Q4MOE_ERR_RANGE (-3)       /* a slab section lies outside the slab */
#define Q4MOE_ERR_DEVICE (-4)      /* no usable sm_103 device              */
#define Q4MOE_ERR_CUDA (-5)        /* a CUDA runtime call or launch failed */
#define Q4MOE_ERR_DEVICE_DATA (-6) /* the device status word is nonzero    */

/* ---- device status bits (see q4moe_device_status) ----------------------- */
#define Q4MOE_DEV_BAD_ROW_OFFSETS 0x1u /* offsets not 0..M, or decreasing  */
#define Q4MOE_DEV_BAD_TOKEN 0x2u       /* token index outside [0, T)        */
#define Q4MOE_DEV_BAD_SLAB_PTR 0x4u    /* per-expert slab pointer misaligned */
#define Q4MOE_DEV_BAD_EXPERT_ID 0x8u   /* routed expert id outside [0, E)    */
#define Q4MOE_DEV_WAIT_TIMEOUT 0x10u   /* a bounded on-chip wait ran out     */

/* ---- weight formats (q4moe_layout_t.weight_format) --------------------- */
#define Q4MOE_FORMAT_Q4 0 /* packed nibbles, value = nibble - 8 (page 52, GATE_UP_SOURCE) */
#define Q4MOE_FORMAT_Q8 1 /* signed bytes, value = the byte (page 52, Q8_GATE_UP_SOURCE) */

/* ---- kernel selection (q4moe_options_t.kernel) -------------------------- */
#define Q4MOE_KERNEL_AUTO 0   /* by rows per expert                          */
#define Q4MOE_KERNEL_MATVEC 1 /* every expert on the streamed matvec         */
#define Q4MOE_KERNEL_GEMM 2   /* every nonempty expert on the tensor-core GEMM */
/* Every expert on the matvec with a fixed unit height (matvec_tile, 128 if
 * 0), never the GEMM or the cp.async matvec: each output's bits then depend
 * on its own row's inputs only, not on how many rows (or which) share the
 * call, so a row decoded alone and the same row in a verify batch agree bit
 * for bit (page 52's matvec has this property: one SIMD group per row and
 * sample).  Large groups stream each expert's weights once per 8 rows. */
#define Q4MOE_KERNEL_BATCH_INVARIANT 3

/*
 * SwiGLU tail (q4moe_options_t.tail), from the bf16 gateT and upT:
 *   PAGE (page 52, streamed-experts.ts, GATE_UP_SOURCE): sigT =
 *     bf16(1 / (1 + exp(-gateT))) in f32 (precise exp, IEEE add and divide),
 *     siluT = bf16(gateT * sigT), out = bf16(siluT * upT);
 *   MLX (page 57, mixed-gate-up-factored.ts: MLX's compiled SwiGLU "in T"),
 *     every step rounded to bf16: e = bf16(exp(|gateT|)), d = bf16(1 + e),
 *     y = bf16(1 / d), sigT = y if gateT < 0 else bf16(1 - y), then siluT
 *     and out as above.  Trellis calls only;
 *   AUTO: the pages' choice for the call (PAGE, except trellis calls whose
 *     gate and up widths differ, which take MLX).
 * Every value is exact against the definition (each operation correctly
 * rounded, no flush to zero).
 */
#define Q4MOE_TAIL_AUTO 0
#define Q4MOE_TAIL_PAGE 1
#define Q4MOE_TAIL_MLX 2

/*
 * Byte layout of one expert slab (page 51, layout.ts,
 * Glm52CanonicalMetalLayout).  Offsets are bytes from the start of the slab.
 *   gate_w_offset, up_w_offset: uint32 [I][H/8] row-major packed nibbles,
 *       4-byte aligned; element k of row i is nibble k%8 (bits 4*(k%8)) of
 *       word i*(H/8) + k/8.
 *   gate_s_offset, up_s_offset: f32 [I] row scales, 4-byte aligned.
 *   down_w_offset: uint32 [H][I/8] row-major packed nibbles (element k of
 *       output row h is nibble k%8 of word h*(I/8) + k/8), 4-byte aligned;
 *   down_s_offset: f32 [H] row scales, 4-byte aligned.  Both negative: the
 *       slab has no down sections (the gate/up calls never read them; the
 *       down calls then fail with Q4MOE_ERR_INVALID_ARG).
 *   weight_format Q4MOE_FORMAT_Q8 (page 52, Q8_GATE_UP_SOURCE and
 *       Q8_DOWN_SOURCE): the weight sections hold one signed byte per
 *       weight instead, int8 [I][H] (gate, up) and [H][I] (down), element k
 *       of a row at byte k; H and I must then be multiples of 4 (the page
 *       accepts any size; rows here start on 4-byte boundaries).  The tail,
 *       the scales and every rounding are the same as for Q4.
 * Each section must lie inside [0, slab_bytes) (page 51, validateRange).
 */
typedef struct q4moe_layout {
    int64_t hidden_size;       /* H: > 0, multiple of 8 (page 52, validateCall) */
    int64_t intermediate_size; /* I: > 0, multiple of 4 (of 8 for the down
                                  sections)                                     */
    int64_t slab_bytes;        /* bytes of one slab                             */
    int64_t gate_w_offset;
    int64_t up_w_offset;
    int64_t gate_s_offset;
    int64_t up_s_offset;
    int64_t down_w_offset;
    int64_t down_s_offset;
    int64_t weight_format;     /* Q4MOE_FORMAT_Q4 (0) or Q4MOE_FORMAT_Q8        */
} q4moe_layout_t;

/*
 * Where the expert slabs live.  Expert e's slab starts at
 *   slab_ptrs[e]                  if slab_ptrs != NULL (a device array of E
 *                                 device pointers, e.g. a residency cache's
 *                                 slots; each must be 4096-aligned, checked
 *                                 on the device), else
 *   base + e * slab_stride        (base 4096-aligned device pointer,
 *                                 slab_stride a multiple of 4096 and
 *                                 >= layout.slab_bytes).
 */
typedef struct q4moe_slabs {
    int32_t num_experts; /* E: 1 .. Q4MOE_MAX_EXPERTS */
    int32_t reserved0;   /* must be 0                 */
    const void *base;
    int64_t slab_stride;
    const void *const *slab_ptrs;
    q4moe_layout_t layout;
} q4moe_slabs_t;

/* Optional arguments of q4moe_gate_up_swiglu_ex (zero-initialise). */
typedef struct q4moe_options {
    int64_t num_tokens; /* T, rows of x; > 0 turns on the device check that
                           every token index is in [0, T)                  */
    float *gate_f32;    /* optional device f32 [M][I]: G * gate scale,
                           before rounding to bf16                         */
    float *up_f32;      /* optional device f32 [M][I]: U * up scale        */
    int32_t kernel;     /* Q4MOE_KERNEL_*                                  */
    int32_t matvec_tile; /* 0: chosen per call; else the height, in
                            intermediate rows, of the work unit of the
                            TMA-fed matvec (16, 32, 64 or 128; taller
                            units split K over fewer warps).  It changes
                            only the f32 summation order: every height
                            meets the same accuracy bound, and inputs
                            whose sums are exact give identical bits.
                            The other matvec versions ignore it.         */
    void *workspace;    /* optional device scratch of at least
                           q4moe_workspace_bytes(M, H) bytes, 256-byte
                           aligned, not overlapping any other argument.
                           With it the tensor-core GEMM reads the routed
                           activations once, grouped, through TMA (its
                           fast form also wants 32-byte aligned weight
                           sections; a layout with sections only 16-byte
                           aligned takes the row-by-row form); without it
                           the GEMM gathers them row by row.  Contents
                           are undefined after the call; calls that share a
                           workspace must be ordered on one stream.       */
    int64_t workspace_bytes; /* size of workspace                         */
    int32_t tail;       /* Q4MOE_TAIL_*: the SwiGLU tail (Q4 and Q8 calls
                           take AUTO or PAGE only)                         */
    int32_t reserved1;  /* must be 0                                       */
} q4moe_options_t;

/*
 * q4moe_gate_up_swiglu for callers that cannot allocate device memory (a
 * plugin inside a host engine that owns all GPU memory through its own pool,
 * code held to a fixed memory budget, a latency-critical loop that must not
 * risk the device synchronisation an allocation can bring).  The pages have
 * no counterpart: this is a library convenience.  Same arguments and result
 * as q4moe_gate_up_swiglu with a workspace, but the scratch is a fixed array
 * inside the library, Q4MOE_NOALLOC_SCRATCH_BYTES on every GPU that loads
 * it, held until the process exits; the call allocates nothing.
 *  - Limit: M * H * 2 bytes (q4moe_workspace_bytes) must not exceed
 *    Q4MOE_NOALLOC_SCRATCH_BYTES, else Q4MOE_ERR_INVALID_ARG with a message.
 *  - The first call on each device looks up the array's device address
 *    (cudaGetSymbolAddress) with that device current; make that first call
 *    before any stream capture.
 *  - Every call shares the one array and overwrites what it needs before
 *    reading it (nothing has to start at zero); calls that overlap on the
 *    GPU, on different streams, race on it.
 */
#define Q4MOE_NOALLOC_SCRATCH_BYTES (32u << 20)
int q4moe_gate_up_swiglu_noalloc(const void *x,
                                 const q4moe_slabs_t *expert_slabs,
                                 const int32_t *row_offsets_per_expert,
                                 const int32_t *token_to_expert_map,
                                 int64_t M, int64_t H, int64_t I, void *out,
                                 cudaStream_t stream);

/* Bytes of the optional workspace (q4moe_options_t.workspace) for M grouped
 * rows of hidden size H: the routed activations in grouped order, bf16
 * [M][H].  Host only; returns a negative code for negative arguments. */
int64_t q4moe_workspace_bytes(int64_t M, int64_t H);

/* ABI version of the loaded library (Q4MOE_ABI_VERSION). */
int q4moe_abi_version(void);

/* Message of the calling thread's last failed call ("" if none). The string
 * is owned by the library and valid until the thread's next call. */
const char *q4moe_last_error(void);

/*
 * Fill *layout with the canonical slab layout for (H, I): gate words at 0,
 * up words at I*H/2, gate scales at I*H, up scales at I*H + 4*I; when
 * I % 8 == 0 also down words at D = (I*H + 8*I) rounded up to 256 and down
 * scales at D + H*I/2 (else no down sections); slab size rounded up to
 * Q4MOE_SLAB_ALIGNMENT.  Host only.
 */
int q4moe_canonical_layout(int64_t H, int64_t I, q4moe_layout_t *layout);

/* The canonical layout for a weight format: Q4MOE_FORMAT_Q4 as above;
 * Q4MOE_FORMAT_Q8 with the same order and the weight sections twice as
 * large (gate bytes at 0, up at I*H, gate scales at 2*I*H, up scales at
 * 2*I*H + 4*I, down bytes at (2*I*H + 8*I) rounded up to 256, down scales
 * after them).  Host only. */
int q4moe_canonical_layout_format(int64_t H, int64_t I, int32_t format,
                                  q4moe_layout_t *layout);

/* Check a layout: dimensions (page 52, validateCall), section alignment and
 * ranges (page 51, validateRange).  Host only. */
int q4moe_validate_layout(const q4moe_layout_t *layout);

/*
 * Copy one expert's sections into a host slab buffer of layout->slab_bytes
 * bytes, zeroing the rest.  gate_w/up_w: host uint32 [I][H/8] (Q8 layouts:
 * the int8 [I][H] bytes, passed through the same pointer type); gate_s/up_s:
 * host f32 [I]; slab_host: host buffer.  Host only (copy the slab to the
 * device yourself).
 */
int q4moe_pack_slab(const q4moe_layout_t *layout, const uint32_t *gate_w,
                    const uint32_t *up_w, const float *gate_s,
                    const float *up_s, void *slab_host);

/*
 * Copy one expert's down sections into a host slab buffer already filled by
 * q4moe_pack_slab (nothing else is touched).  down_w: host uint32 [H][I/8]
 * (Q8: the int8 [H][I] bytes); down_s: host f32 [H].  Host only.
 */
int q4moe_pack_slab_down(const q4moe_layout_t *layout, const uint32_t *down_w,
                         const float *down_s, void *slab_host);

/*
 * Token -> expert grouping: a stable counting sort of the T*k routed
 * (token, slot) pairs by expert id.  The pages dispatch one expert slot at a
 * time with its rows as an [M, H] input (page 52, execute); this builds the
 * per-expert row lists for all experts at once.
 *   topk_ids      device int32 [T][k]: expert of slot j of token t.
 *   row_offsets   device int32 [E+1] out: expert e owns grouped rows
 *                 [row_offsets[e], row_offsets[e+1]); row_offsets[E] = T*k
 *                 minus the pairs with an id outside [0, E).
 *   token_of_row  device int32 [T*k] out: token of each grouped row, tokens
 *                 ascending within an expert.
 *   row_of_pair   device int32 [T*k] out: grouped row of pair t*k+j (-1 for
 *                 a bad id), for putting outputs back in token order.
 * An id outside [0, E) sets Q4MOE_DEV_BAD_EXPERT_ID and the pair is dropped.
 * T >= 0, 1 <= k, 1 <= E <= Q4MOE_MAX_EXPERTS, T*k < 2^31.
 */
int q4moe_group_rows(const int32_t *topk_ids, int64_t T, int32_t k,
                     int32_t E, int32_t *row_offsets, int32_t *token_of_row,
                     int32_t *row_of_pair, cudaStream_t stream);

/*
 * The fused gate/up + SwiGLU over grouped rows (the formula at the top).
 *   x                       device bf16 [T][H], row-major, row stride H.
 *   expert_slabs            host pointer, read during the call only.
 *   row_offsets_per_expert  device int32 [E+1], 0 = off[0] <= ... <= off[E] = M.
 *   token_to_expert_map     device int32 [M]: the row of x that grouped row
 *                           p reads (a "sorted per-expert row list"; the
 *                           name keeps the pages' wording).
 *   M                       grouped rows (>= 0; 0 is a no-op).
 *   H, I                    must equal the layout's.
 *   out                     device bf16 [M][I], grouped-row order, fully
 *                           written on success.
 * Kernel choice (Q4MOE_KERNEL_AUTO): with several experts and at least 4
 * grouped rows per expert on average (M >= 4 E), experts with more than 16
 * rows run on the tcgen05 tensor-core GEMM (tiles of 128 intermediate rows
 * x up to 256 grouped rows) and the others on the HBM-streaming matvec;
 * with fewer rows the matvec takes every expert and the GEMM is not
 * launched; from 128 rows per expert on average (M >= 128 E) the GEMM
 * takes every expert and the matvec is not launched.  One expert goes to
 * the GEMM when it has more than 48 rows and
 * makes at least one tile per SM, else to the matvec: with at most 8 rows
 * to a version laid out for latency (each SM a few rows, the K range split
 * over its warps; also for the down projection), which the batch-invariant
 * choice never uses.
 */
int q4moe_gate_up_swiglu(const void *x, const q4moe_slabs_t *expert_slabs,
                         const int32_t *row_offsets_per_expert,
                         const int32_t *token_to_expert_map, int64_t M,
                         int64_t H, int64_t I, void *out, cudaStream_t stream);

/* q4moe_gate_up_swiglu with options (opts may be NULL). */
int q4moe_gate_up_swiglu_ex(const void *x, const q4moe_slabs_t *expert_slabs,
                            const int32_t *row_offsets_per_expert,
                            const int32_t *token_to_expert_map, int64_t M,
                            int64_t H, int64_t I, void *out,
                            const q4moe_options_t *opts, cudaStream_t stream);

/*
 * The down projection over grouped rows (the second formula at the top;
 * page 52, streamed-experts.ts, DOWN_SOURCE).
 *   mid                     device bf16 [M][I], grouped-row order (the out of
 *                           the gate/up call), 16-byte aligned.
 *   expert_slabs            host pointer, read during the call only; its
 *                           layout must hold the down sections.
 *   row_offsets_per_expert  device int32 [E+1] as for the gate/up call.
 *   M                       grouped rows (>= 0; 0 is a no-op).
 *   H, I                    must equal the layout's; I % 8 == 0.
 *   out                     device bf16 [M][H], grouped-row order.
 *   opts                    may be NULL.  kernel and matvec_tile as for the
 *                           gate/up call (the matvec's unit then covers
 *                           twice matvec_tile output rows); gate_f32, if
 *                           set, receives f32 [M][H]: the sum times the
 *                           scale before rounding.  num_tokens, up_f32 and
 *                           workspace must be 0 / NULL (the rows of mid are
 *                           already grouped).
 * Kernel choice per expert as for gate/up, with experts above 32 rows (not
 * 16) on the GEMM when it is launched; the GEMM's tiles are 256 output
 * rows.  Summation order: as for gate/up (exact inputs give exact bits).
 */
int q4moe_down_proj(const void *mid, const q4moe_slabs_t *expert_slabs,
                    const int32_t *row_offsets_per_expert, int64_t M,
                    int64_t H, int64_t I, void *out,
                    const q4moe_options_t *opts, cudaStream_t stream);

/*
 * The whole routed expert MLP: q4moe_gate_up_swiglu_ex from x into mid,
 * then q4moe_down_proj from mid into out, queued on `stream` (the page's
 * executor, page 52, runs its gate/up kernel and then its down kernel on
 * the same slot).  Arguments as for those two calls; mid is caller-owned
 * device scratch bf16 [M][I], 16-byte aligned, not overlapping x or out,
 * and holds the gate/up output afterwards.  opts apply to the gate/up stage
 * as documented there (gate_f32/up_f32, num_tokens, workspace); kernel and
 * matvec_tile to both stages.
 */
int q4moe_expert_mlp(const void *x, const q4moe_slabs_t *expert_slabs,
                     const int32_t *row_offsets_per_expert,
                     const int32_t *token_to_expert_map, int64_t M, int64_t H,
                     int64_t I, void *mid, void *out,
                     const q4moe_options_t *opts, cudaStream_t stream);

/*
 * Trellis-coded experts (QTIP "1MAD" code; pages 57 and 54: trellis/
 * gate-up-mma.ts, mixed-gate-up-factored.ts, codebook.ts), gate and up
 * coded along the input (the pages' axis 1).  A row's H weights form H / T
 * blocks of T weights at k bits each: T * k / 32 uint32 words per block,
 * bit b of a block is bit b % 32 of word b / 32.  Weight t of a block has
 * the state s = the L bits at (T - 1 - t) * k of the block, taken modulo
 * T * k (wrapping), and the code value
 *   y(s) = (sum of the four bytes of s * 34038481 + 76625530 mod 2^32) - 510.
 * For grouped row p of expert e (token x[t]) and output row i:
 *   G = sum_k y_k * x[t][k]                      (f32 accumulate)
 *   gate32 = G * RN32(f32(gate_scale[i]) * RN32(1 / 147.800537109375))
 * (the row scale factored out of the sum, as on the pages), up likewise
 * with its own width, then the tail opts->tail selects: with
 * Q4MOE_TAIL_AUTO the pages' choice, the page 52 tail of Q4 when gate and
 * up share a width (page 57, gate-up-mma.ts) and MLX's compiled SwiGLU
 * (Q4MOE_TAIL_MLX) when they differ (page 57, mixed-gate-up-factored.ts).
 */
typedef struct q4moe_trellis_layout {
    int64_t hidden_size;       /* H: a multiple of block_size                 */
    int64_t intermediate_size; /* I > 0                                       */
    int32_t block_size;        /* T: weights per block, a multiple of 32 (the
                                  pages use 256)                              */
    int32_t window_bits;       /* L: state bits, 1..24, L <= T * k (pages: 12) */
    int32_t gate_bits;         /* k of gate, 1..8                             */
    int32_t up_bits;           /* k of up, 1..8 (may differ from gate's)      */
    int64_t slab_bytes;        /* bytes of one expert's slab                  */
    int64_t gate_codes_offset; /* uint32 [I][H/T * T*k/32], 4-byte aligned     */
    int64_t up_codes_offset;
    int64_t gate_scales_offset; /* f16 [I], 2-byte aligned                     */
    int64_t up_scales_offset;
} q4moe_trellis_layout_t;

/* Where trellis expert slabs live: as q4moe_slabs_t. */
typedef struct q4moe_trellis_slabs {
    int32_t num_experts; /* E: 1 .. Q4MOE_MAX_EXPERTS */
    int32_t reserved0;   /* must be 0                 */
    const void *base;
    int64_t slab_stride;
    const void *const *slab_ptrs;
    q4moe_trellis_layout_t layout;
} q4moe_trellis_slabs_t;

/* Canonical trellis slab: gate codes at 0, up codes, gate scales, up scales,
 * each section starting on a 256-byte boundary; size rounded up to
 * Q4MOE_SLAB_ALIGNMENT.  Host only. */
int q4moe_trellis_canonical_layout(int64_t H, int64_t I, int32_t block_size,
                                   int32_t window_bits, int32_t gate_bits,
                                   int32_t up_bits,
                                   q4moe_trellis_layout_t *layout);

/* Copy one expert's trellis sections into a host slab buffer (zeroing the
 * rest).  gate_codes/up_codes: host uint32 rows as described above;
 * gate_scales/up_scales: host f16 bit patterns [I].  Host only. */
int q4moe_trellis_pack_slab(const q4moe_trellis_layout_t *layout,
                            const uint32_t *gate_codes,
                            const uint32_t *up_codes,
                            const uint16_t *gate_scales,
                            const uint16_t *up_scales, void *slab_host);

/*
 * The fused trellis gate/up + SwiGLU over grouped rows (formula above).
 * Arguments as q4moe_gate_up_swiglu_ex: x device bf16 [T][H] (16-byte
 * aligned), row offsets and the token map on the device, out device bf16
 * [M][I].  opts may be NULL; num_tokens, gate_f32 and up_f32 as for Q4;
 * tail any Q4MOE_TAIL_*; kernel, matvec_tile and workspace must be 0.
 * One kernel (a warp per output row, each decoded weight serving up to 8
 * grouped rows); decoding is integer arithmetic, so the kernel is bound by
 * the integer pipe.
 */
int q4moe_trellis_gate_up_swiglu(const void *x,
                                 const q4moe_trellis_slabs_t *expert_slabs,
                                 const int32_t *row_offsets_per_expert,
                                 const int32_t *token_to_expert_map,
                                 int64_t M, int64_t H, int64_t I, void *out,
                                 const q4moe_options_t *opts,
                                 cudaStream_t stream);

/*
 * Wait for `stream`, then read the current device's status word into
 * *flags (Q4MOE_DEV_* bits accumulated since the last clear) and clear it
 * if `clear` is nonzero.  Returns Q4MOE_ERR_DEVICE_DATA when *flags != 0.
 * This is the one entry point that synchronises the host.
 */
int q4moe_device_status(cudaStream_t stream, uint32_t *flags, int clear);

/* Number of CUDA kernels this library has launched in this process (all
 * devices, all entry points); a host-side counter for benchmarks. */
int64_t q4moe_launch_count(void);

/*
 * Diagnostic: evaluate the device's SwiGLU tail alone.  For n elements,
 * from bf16 gate and up values (device uint16 [n] each) write the device
 * uint16 [n][4] results sigT, siluT, out (as the tensor-core GEMM forms
 * them, from the sigmoid table) and sigT as the decode kernels form it (in
 * registers when their fast form is conclusive, else from the table).
 * Used to test both forms of the tail exhaustively.
 */
int q4moe_debug_tail(const uint16_t *gate_bf16, const uint16_t *up_bf16,
                     int64_t n, uint16_t *res, cudaStream_t stream);

/* The same for the MLX tail (Q4MOE_TAIL_MLX), with the same arguments and
 * result layout (column 3 repeats sigT: every kernel takes the MLX sigmoid
 * from its table). */
int q4moe_debug_tail_mlx(const uint16_t *gate_bf16, const uint16_t *up_bf16,
                         int64_t n, uint16_t *res, cudaStream_t stream);

/*
 * Diagnostic: run the kernels' bounded on-chip waits (the try_wait form of
 * the producers and consumers and the spin of the MMA issuer) on an
 * mbarrier that nothing arrives on, with a limit of limit_ns (1e3 .. 1e9,
 * i.e. 1 us .. 1 s; the kernels themselves wait at most 4 s).  The kernel
 * gives up after the limit, raises Q4MOE_DEV_WAIT_TIMEOUT in the device
 * status word and returns; the device stays usable.  For testing the
 * time-out path.  No passage of the pages corresponds to it.
 */
int q4moe_debug_wait_timeout(int64_t limit_ns, cudaStream_t stream);

#ifdef __cplusplus
}
#endif
#endif /* Q4MOE_H_ */
