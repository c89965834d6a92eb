/*
 * q4moe_oracle.c -- plain, slow, CPU reference of the fused Q4 MoE expert
 * gate/up projection with SwiGLU.
 *
 * TEST INFRASTRUCTURE ONLY.  Nothing in the product path (the CUDA library
 * under up_swiglu_gb300/) includes, links or calls this file; only tests/,
 * __graft_entry__.smoke() and the cpu_baseline / reference legs of bench.py
 * load it.  It shares no code, header, table or constant with the CUDA path.
 *
 * Sources (all on the pages "@mlx-bun/inference 0.0.0-stage -> 1.0.0"):
 *  - page 52, src/kernels/glm52/streamed-experts.ts, GATE_UP_SOURCE: the
 *    per-row arithmetic (nibble p of packed word w is element 8w+p with value
 *    ((w >> 4p) & 0xF) - 8; f32 accumulation; times the f32 row scale; gate
 *    and up rounded to bf16; sigmoid, silu and the product each rounded to
 *    bf16);
 *  - page 54, src/kernels/trellis/codebook.ts, trellis_bf16: the f32 -> bf16
 *    rounding (round to nearest, ties to even, on the bit pattern);
 *  - page 52, DOWN_SOURCE: the down projection that follows gate/up in the
 *    same expert (the row of packed words belongs to output row h and runs
 *    over the intermediate index k; f32 accumulation; times the f32 row
 *    scale of h; rounded to bf16);
 *  - page 52, Q8_GATE_UP_SOURCE and Q8_DOWN_SOURCE: the same two
 *    operations on signed int8 weights (one byte per weight, row-major, the
 *    byte's two's-complement value, no zero point);
 *  - page 57 (trellis/gate-up-mma.ts, mixed-gate-up-factored.ts) and page
 *    54 (trellis/codebook.ts): the trellis (QTIP 1MAD) gate/up with the row
 *    scale factored out of the sum: code value y of state s is the byte sum
 *    of s * 34038481 + 76625530 (mod 2^32) minus 510, the state of weight t
 *    of a block is the L-bit window at bit (T - 1 - t) * k of the block's
 *    bits (wrapping), and gate = (sum_k y_k x_k) * (scale * (1/147.800537109375));
 *  - page 51, src/kernels/glm52/layout.ts: the per-expert section layout
 *    (the oracle takes the sections as separate arrays, so it never parses
 *    a slab).
 *
 * Readings taken where the pages leave a step open:
 *  - the dot product is accumulated in f64 (each product q*x is exact in
 *    f64, so the sum is the f64 rounding of the exact dot product, far
 *    tighter than any f32 order);
 *  - gate32 = (float)(G * (double)scale): one rounding to f32;
 *  - the sigmoid is the f32 chain of the page with every step correctly
 *    rounded and no flush to zero: e = RN32(exp(-g)) (+inf on overflow),
 *    d = RN32(1 + e), s = RN32(1 / d);  the add and the divide go through
 *    f64, which gives the correctly rounded f32 result (double has more than
 *    2*24+2 bits, so the double rounding is innocuous);
 *  - silu_mode 1 keeps the sigmoid in f32 (no bf16 rounding of s), the
 *    alternative reading of "bf16(silu(gate))"; mode 0 follows the page;
 *  - the second tail, MLX's compiled SwiGLU that the pages' mixed-width
 *    trellis kernel ends with (page 57, mixed-gate-up-factored.ts), works
 *    "in T" (bf16): every step is evaluated in f32, correctly rounded, and
 *    its result rounded to bf16 before the next step uses it; the sigmoid
 *    is 1 / (1 + exp(|g|)) for negative g and one minus that otherwise.
 *
 * Build: gcc -O2 -fopenmp -ffp-contract=off -shared -fPIC (no fast-math).
 */
#include <float.h>
#include <math.h>
#include <stdint.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

#if !defined(__STDC_IEC_559__) && !defined(__GCC_IEC_559)
#error "the oracle needs IEEE-754 float/double semantics (Annex F)"
#endif

/* ---- bf16 <-> f32 (page 54, codebook.ts, trellis_bf16) ------------------ */

/* Round an f32 to bf16, nearest with ties to even, on the bit pattern:
 * add 0x7FFF plus the lowest kept bit, keep the upper 16 bits.  Finite inputs
 * only (the pages' routine has no NaN case and none arises here). */
uint16_t q4o_bf16_rne(float v)
{
    uint32_t u;
    memcpy(&u, &v, sizeof u);
    u = u + 0x7FFFu + ((u >> 16) & 1u);
    return (uint16_t)(u >> 16);
}

float q4o_bf16_to_f32(uint16_t b)
{
    uint32_t u = (uint32_t)b << 16;
    float f;
    memcpy(&f, &u, sizeof f);
    return f;
}

/* q4o_bf16_rne over n values. */
void q4o_bf16_rne_array(int64_t n, const float *v, uint16_t *out)
{
    for (int64_t j = 0; j < n; ++j)
        out[j] = q4o_bf16_rne(v[j]);
}

/* ---- SwiGLU tail (page 52, streamed-experts.ts, GATE_UP_SOURCE tail) ---- */

/* res[0..4] = gateT, upT, sigmoidT, siluT, out  (bf16 bit patterns).
 * silu_mode 0: the page's chain (sigmoid rounded to bf16 before the product);
 * silu_mode 1: sigmoid kept in f32 (siluT = bf16(gateT * s32)). */
void q4o_tail(float gate32, float up32, int silu_mode, uint16_t res[5])
{
    const uint16_t gT = q4o_bf16_rne(gate32);
    const uint16_t uT = q4o_bf16_rne(up32);
    const float g = q4o_bf16_to_f32(gT);
    const float e32 = (float)exp(-(double)g);          /* +inf past FLT_MAX */
    const float d32 = (float)(1.0 + (double)e32);      /* RN32(1 + e)      */
    const float s32 = (float)(1.0 / (double)d32);      /* RN32(1 / d)      */
    const uint16_t sT = q4o_bf16_rne(s32);
    float silu32;
    if (silu_mode == 0)
        silu32 = g * q4o_bf16_to_f32(sT);               /* f32 multiply    */
    else
        silu32 = g * s32;
    const uint16_t siluT = q4o_bf16_rne(silu32);
    const float o32 = q4o_bf16_to_f32(siluT) * q4o_bf16_to_f32(uT);
    res[0] = gT;
    res[1] = uT;
    res[2] = sT;
    res[3] = siluT;
    res[4] = q4o_bf16_rne(o32);
}

/* The tail of the pages' mixed-width trellis kernel (page 57,
 * mixed-gate-up-factored.ts): MLX's compiled SwiGLU over the bf16 gate and
 * up, each step computed in f32 (correctly rounded) and rounded to bf16:
 *   eT = bf16(RN32(exp(|gateT|)))      (+inf once exp passes FLT_MAX)
 *   dT = bf16(RN32(1 + eT)),  yT = bf16(RN32(1 / dT))
 *   sigT = yT if gateT < 0 (false for -0), else bf16(1 - yT)
 *   siluT = bf16(gateT * sigT),  out = bf16(siluT * upT).
 * res[0..4] as q4o_tail: gateT, upT, sigT, siluT, out. */
void q4o_tail_mlx(float gate32, float up32, uint16_t res[5])
{
    const uint16_t gT = q4o_bf16_rne(gate32);
    const uint16_t uT = q4o_bf16_rne(up32);
    const float g = q4o_bf16_to_f32(gT);
    const float a = fabsf(g);
    const float e = q4o_bf16_to_f32(q4o_bf16_rne((float)exp((double)a)));
    const float d = q4o_bf16_to_f32(q4o_bf16_rne((float)(1.0 + (double)e)));
    const uint16_t yT = q4o_bf16_rne((float)(1.0 / (double)d));
    const uint16_t sT =
        g < 0.0f ? yT
                 : q4o_bf16_rne((float)(1.0 - (double)q4o_bf16_to_f32(yT)));
    const uint16_t siluT = q4o_bf16_rne(g * q4o_bf16_to_f32(sT));
    res[0] = gT;
    res[1] = uT;
    res[2] = sT;
    res[3] = siluT;
    res[4] = q4o_bf16_rne(q4o_bf16_to_f32(siluT) * q4o_bf16_to_f32(uT));
}

/* q4o_tail (tail 0, page 52) or q4o_tail_mlx (tail 1) of one element. */
static void q4o_tail_of(int tail, float gate32, float up32, uint16_t res[5])
{
    if (tail == 1)
        q4o_tail_mlx(gate32, up32, res);
    else
        q4o_tail(gate32, up32, 0, res);
}

/* q4o_tail_mlx over n elements: res is [n][5]. */
void q4o_tail_mlx_array(int64_t n, const float *gate32, const float *up32,
                        uint16_t *res)
{
    for (int64_t j = 0; j < n; ++j)
        q4o_tail_mlx(gate32[j], up32[j], res + 5 * j);
}

/* q4o_tail over n elements: res is [n][5] (gateT, upT, sigT, siluT, out). */
void q4o_tail_array(int64_t n, const float *gate32, const float *up32,
                    int silu_mode, uint16_t *res)
{
    for (int64_t j = 0; j < n; ++j)
        q4o_tail(gate32[j], up32[j], silu_mode, res + 5 * j);
}

/* ---- one dot product ---------------------------------------------------- */

/* G = sum_k (nib(w[k>>3], k&7) - 8) * x[k] over one packed row of H/8 words
 * (page 52, GATE_UP_SOURCE: word index = k / 8, place = k % 8, shift 4*place).
 * Also returns sum_k |(nib - 8) * x[k]|, the scale of the rounding error any
 * f32 summation order can make. */
static double q4o_dot(const uint32_t *wrow, const uint16_t *xrow, int64_t H,
                      double *absdot)
{
    double s = 0.0, a = 0.0;
    for (int64_t k = 0; k < H; ++k) {
        const uint32_t word = wrow[k >> 3];
        const int place = (int)(k & 7);
        const int q = (int)((word >> (4 * place)) & 0xFu) - 8;
        const double prod = (double)q * (double)q4o_bf16_to_f32(xrow[k]);
        s += prod;
        a += fabs(prod);
    }
    *absdot = a;
    return s;
}

/* The same over a row of H signed bytes (page 52, Q8_GATE_UP_SOURCE:
 * weight k is the int8 value of byte k of the row). */
static double q4o_dot_q8(const int8_t *wrow, const uint16_t *xrow, int64_t H,
                         double *absdot)
{
    double s = 0.0, a = 0.0;
    for (int64_t k = 0; k < H; ++k) {
        const double prod = (double)wrow[k] * (double)q4o_bf16_to_f32(xrow[k]);
        s += prod;
        a += fabs(prod);
    }
    *absdot = a;
    return s;
}

/* ---- argument checks shared by the entry points below ------------------- */

static int q4o_check(int64_t T, int64_t H, int64_t I, int32_t E,
                     const int32_t *row_offsets, const int32_t *token_of_row,
                     int64_t M)
{
    if (T < 0 || H <= 0 || I <= 0 || E <= 0 || M < 0 || (H % 8) != 0)
        return -1;
    if (row_offsets[0] != 0 || row_offsets[E] != M)
        return -2;
    for (int32_t e = 0; e < E; ++e)
        if (row_offsets[e + 1] < row_offsets[e])
            return -2;
    for (int64_t p = 0; p < M; ++p)
        if (token_of_row[p] < 0 || token_of_row[p] >= T)
            return -3;
    return 0;
}

static int32_t q4o_expert_of_row(const int32_t *row_offsets, int32_t E,
                                 int64_t p)
{
    for (int32_t e = 0; e < E; ++e)
        if (p >= row_offsets[e] && p < row_offsets[e + 1])
            return e;
    return -1;
}

/* One output element (grouped row p, intermediate row i).  Optional outputs
 * (any may be NULL): f32 gate/up before rounding, the f64 dot products and
 * their absolute-value sums. */
static void q4o_element(const uint16_t *x, int64_t H, int64_t I,
                        const uint32_t *gate_w, const uint32_t *up_w,
                        const float *gate_s, const float *up_s,
                        int32_t e, int64_t t, int64_t i, int silu_mode,
                        uint16_t *out, float *gate32, float *up32,
                        double *gdot, double *udot, double *gabs, double *uabs)
{
    const int64_t words = H / 8;
    const uint32_t *grow = gate_w + ((int64_t)e * I + i) * words;
    const uint32_t *urow = up_w + ((int64_t)e * I + i) * words;
    const uint16_t *xrow = x + t * H;
    double ga, ua;
    const double G = q4o_dot(grow, xrow, H, &ga);
    const double U = q4o_dot(urow, xrow, H, &ua);
    const float g32 = (float)(G * (double)gate_s[(int64_t)e * I + i]);
    const float u32 = (float)(U * (double)up_s[(int64_t)e * I + i]);
    uint16_t res[5];
    q4o_tail(g32, u32, silu_mode, res);
    *out = res[4];
    if (gate32) *gate32 = g32;
    if (up32) *up32 = u32;
    if (gdot) *gdot = G;
    if (udot) *udot = U;
    if (gabs) *gabs = ga;
    if (uabs) *uabs = ua;
}

/* ---- the whole grouped call ---------------------------------------------
 * x:            bf16 bits [T, H], row-major
 * gate_w/up_w:  uint32 [E, I, H/8]  (row i of expert e: H/8 packed words)
 * gate_s/up_s:  f32 [E, I]
 * row_offsets:  int32 [E+1], expert e owns grouped rows [off[e], off[e+1])
 * token_of_row: int32 [M], the row of x that grouped row p reads
 * out:          bf16 bits [M, I] in grouped-row order
 * Optional (NULL to skip): gate32/up32 f32 [M, I]; gdot/udot/gabs/uabs f64
 * [M, I].  Returns 0, or a negative code for inconsistent arguments. */
int q4o_gate_up_swiglu(const uint16_t *x, int64_t T, int64_t H, int64_t I,
                       int32_t E, const uint32_t *gate_w, const uint32_t *up_w,
                       const float *gate_s, const float *up_s,
                       const int32_t *row_offsets, const int32_t *token_of_row,
                       int64_t M, int silu_mode, uint16_t *out, float *gate32,
                       float *up32, double *gdot, double *udot, double *gabs,
                       double *uabs, int nthreads)
{
    const int rc = q4o_check(T, H, I, E, row_offsets, token_of_row, M);
    if (rc != 0)
        return rc;
#ifdef _OPENMP
    if (nthreads <= 0)
        nthreads = omp_get_max_threads();
#pragma omp parallel for schedule(dynamic, 8) num_threads(nthreads)
#endif
    for (int64_t pi = 0; pi < M * I; ++pi) {
        const int64_t p = pi / I, i = pi % I;
        const int32_t e = q4o_expert_of_row(row_offsets, E, p);
        q4o_element(x, H, I, gate_w, up_w, gate_s, up_s, e,
                    token_of_row[p], i, silu_mode, &out[pi],
                    gate32 ? &gate32[pi] : 0, up32 ? &up32[pi] : 0,
                    gdot ? &gdot[pi] : 0, udot ? &udot[pi] : 0,
                    gabs ? &gabs[pi] : 0, uabs ? &uabs[pi] : 0);
    }
    (void)nthreads;
    return 0;
}

/* The same arithmetic for n chosen elements (rows[j], cols[j]) only; the
 * outputs are indexed by j.  Used where the full problem is too large. */
int q4o_gate_up_swiglu_sampled(const uint16_t *x, int64_t T, int64_t H,
                               int64_t I, int32_t E, const uint32_t *gate_w,
                               const uint32_t *up_w, const float *gate_s,
                               const float *up_s, const int32_t *row_offsets,
                               const int32_t *token_of_row, int64_t M,
                               int silu_mode, int64_t n, const int64_t *rows,
                               const int64_t *cols, uint16_t *out,
                               float *gate32, float *up32, double *gabs,
                               double *uabs, int nthreads)
{
    const int rc = q4o_check(T, H, I, E, row_offsets, token_of_row, M);
    if (rc != 0)
        return rc;
    for (int64_t j = 0; j < n; ++j)
        if (rows[j] < 0 || rows[j] >= M || cols[j] < 0 || cols[j] >= I)
            return -4;
#ifdef _OPENMP
    if (nthreads <= 0)
        nthreads = omp_get_max_threads();
#pragma omp parallel for schedule(dynamic, 4) num_threads(nthreads)
#endif
    for (int64_t j = 0; j < n; ++j) {
        const int64_t p = rows[j], i = cols[j];
        const int32_t e = q4o_expert_of_row(row_offsets, E, p);
        q4o_element(x, H, I, gate_w, up_w, gate_s, up_s, e,
                    token_of_row[p], i, silu_mode, &out[j],
                    gate32 ? &gate32[j] : 0, up32 ? &up32[j] : 0, 0, 0,
                    gabs ? &gabs[j] : 0, uabs ? &uabs[j] : 0);
    }
    (void)nthreads;
    return 0;
}

/* ---- the down projection ------------------------------------------------
 * Page 52, streamed-experts.ts, DOWN_SOURCE, run after gate/up on the same
 * expert slot: grouped row p (of expert e) of the intermediate activations
 * mid, output row h:
 *   D = sum_k (nib(down_w[e][h][k/8], k%8) - 8) * mid[p][k]
 *   out[p][h] = bf16(f32(D * down_s[e][h]))
 * mid:         bf16 bits [M, I] in grouped-row order (the gate/up output)
 * down_w:      uint32 [E, H, I/8] (row h of expert e: I/8 packed words)
 * down_s:      f32 [E, H]
 * row_offsets: int32 [E+1]
 * out:         bf16 bits [M, H] in grouped-row order
 * Optional (NULL to skip): out32 f32 [M, H] (the value before the bf16
 * rounding), dabs f64 [M, H] (sum_k |w*mid|).  The sum is taken in f64
 * (exact products), rounded once to f32 with the scale, as for gate/up. */
static int q4o_down_check(int64_t M, int64_t I, int64_t H, int32_t E,
                          const int32_t *row_offsets)
{
    if (M < 0 || I <= 0 || H <= 0 || E <= 0 || (I % 8) != 0)
        return -1;
    if (row_offsets[0] != 0 || row_offsets[E] != M)
        return -2;
    for (int32_t e = 0; e < E; ++e)
        if (row_offsets[e + 1] < row_offsets[e])
            return -2;
    return 0;
}

static void q4o_down_element(const uint16_t *mid, int64_t I, int64_t H,
                             const uint32_t *down_w, const float *down_s,
                             int32_t e, int64_t p, int64_t h, uint16_t *out,
                             float *out32, double *dabs)
{
    const uint32_t *wrow = down_w + ((int64_t)e * H + h) * (I / 8);
    double a;
    const double D = q4o_dot(wrow, mid + p * I, I, &a);
    const float v = (float)(D * (double)down_s[(int64_t)e * H + h]);
    *out = q4o_bf16_rne(v);
    if (out32) *out32 = v;
    if (dabs) *dabs = a;
}

int q4o_down_proj(const uint16_t *mid, int64_t M, int64_t I, int64_t H,
                  int32_t E, const uint32_t *down_w, const float *down_s,
                  const int32_t *row_offsets, uint16_t *out, float *out32,
                  double *dabs, int nthreads)
{
    const int rc = q4o_down_check(M, I, H, E, row_offsets);
    if (rc != 0)
        return rc;
#ifdef _OPENMP
    if (nthreads <= 0)
        nthreads = omp_get_max_threads();
#pragma omp parallel for schedule(dynamic, 8) num_threads(nthreads)
#endif
    for (int64_t ph = 0; ph < M * H; ++ph) {
        const int64_t p = ph / H, h = ph % H;
        const int32_t e = q4o_expert_of_row(row_offsets, E, p);
        q4o_down_element(mid, I, H, down_w, down_s, e, p, h, &out[ph],
                         out32 ? &out32[ph] : 0, dabs ? &dabs[ph] : 0);
    }
    (void)nthreads;
    return 0;
}

/* The same for n chosen elements (rows[j], cols[j]); outputs indexed by j. */
int q4o_down_proj_sampled(const uint16_t *mid, int64_t M, int64_t I,
                          int64_t H, int32_t E, const uint32_t *down_w,
                          const float *down_s, const int32_t *row_offsets,
                          int64_t n, const int64_t *rows, const int64_t *cols,
                          uint16_t *out, float *out32, double *dabs,
                          int nthreads)
{
    const int rc = q4o_down_check(M, I, H, E, row_offsets);
    if (rc != 0)
        return rc;
    for (int64_t j = 0; j < n; ++j)
        if (rows[j] < 0 || rows[j] >= M || cols[j] < 0 || cols[j] >= H)
            return -4;
#ifdef _OPENMP
    if (nthreads <= 0)
        nthreads = omp_get_max_threads();
#pragma omp parallel for schedule(dynamic, 4) num_threads(nthreads)
#endif
    for (int64_t j = 0; j < n; ++j) {
        const int32_t e = q4o_expert_of_row(row_offsets, E, rows[j]);
        q4o_down_element(mid, I, H, down_w, down_s, e, rows[j], cols[j],
                         &out[j], out32 ? &out32[j] : 0, dabs ? &dabs[j] : 0);
    }
    (void)nthreads;
    return 0;
}

/* ---- token -> expert grouping -------------------------------------------
 * topk: int32 [T, k], the experts each token is routed to.  Produces the
 * per-expert row lists the gate/up call consumes: row_offsets [E+1]
 * (counts, exclusive prefix sum), token_of_row [T*k] (the token of each
 * grouped row) and row_of_pair [T*k] (the grouped row of pair t*k+j, for
 * putting outputs back in token order).  Rows of one expert keep the
 * token order (a stable counting sort).  Returns -1 on an expert id outside
 * [0, E). */
/* ---- Q8 (page 52, Q8_GATE_UP_SOURCE, Q8_DOWN_SOURCE) ---------------------
 * gate_w/up_w: int8 [E, I, H]; down_w: int8 [E, H, I]; everything else as
 * for Q4 (the tail and the roundings are the same). */
static void q4o_q8_element(const uint16_t *x, int64_t H, int64_t I,
                           const int8_t *gate_w, const int8_t *up_w,
                           const float *gate_s, const float *up_s, int32_t e,
                           int64_t t, int64_t i, int silu_mode, uint16_t *out,
                           float *gate32, float *up32, double *gabs,
                           double *uabs)
{
    const int8_t *grow = gate_w + ((int64_t)e * I + i) * H;
    const int8_t *urow = up_w + ((int64_t)e * I + i) * H;
    double ga, ua;
    const double G = q4o_dot_q8(grow, x + t * H, H, &ga);
    const double U = q4o_dot_q8(urow, x + t * H, H, &ua);
    const float g32 = (float)(G * (double)gate_s[(int64_t)e * I + i]);
    const float u32 = (float)(U * (double)up_s[(int64_t)e * I + i]);
    uint16_t res[5];
    q4o_tail(g32, u32, silu_mode, res);
    *out = res[4];
    if (gate32) *gate32 = g32;
    if (up32) *up32 = u32;
    if (gabs) *gabs = ga;
    if (uabs) *uabs = ua;
}

/* All M x I outputs, or (rows != NULL) the n elements (rows[j], cols[j]).
 * Same arguments and results as q4o_gate_up_swiglu(_sampled). */
int q4o_q8_gate_up_swiglu(const uint16_t *x, int64_t T, int64_t H, int64_t I,
                          int32_t E, const int8_t *gate_w, const int8_t *up_w,
                          const float *gate_s, const float *up_s,
                          const int32_t *row_offsets,
                          const int32_t *token_of_row, int64_t M,
                          int silu_mode, int64_t n, const int64_t *rows,
                          const int64_t *cols, uint16_t *out, float *gate32,
                          float *up32, double *gabs, double *uabs,
                          int nthreads)
{
    if (T < 0 || H <= 0 || I <= 0 || E <= 0 || M < 0)
        return -1;
    if (row_offsets[0] != 0 || row_offsets[E] != M)
        return -2;
    for (int32_t e = 0; e < E; ++e)
        if (row_offsets[e + 1] < row_offsets[e])
            return -2;
    for (int64_t p = 0; p < M; ++p)
        if (token_of_row[p] < 0 || token_of_row[p] >= T)
            return -3;
    if (rows == 0)
        n = M * I;
    else
        for (int64_t j = 0; j < n; ++j)
            if (rows[j] < 0 || rows[j] >= M || cols[j] < 0 || cols[j] >= I)
                return -4;
#ifdef _OPENMP
    if (nthreads <= 0)
        nthreads = omp_get_max_threads();
#pragma omp parallel for schedule(dynamic, 8) num_threads(nthreads)
#endif
    for (int64_t j = 0; j < n; ++j) {
        const int64_t p = rows ? rows[j] : j / I, i = rows ? cols[j] : j % I;
        const int32_t e = q4o_expert_of_row(row_offsets, E, p);
        q4o_q8_element(x, H, I, gate_w, up_w, gate_s, up_s, e,
                       token_of_row[p], i, silu_mode, &out[j],
                       gate32 ? &gate32[j] : 0, up32 ? &up32[j] : 0,
                       gabs ? &gabs[j] : 0, uabs ? &uabs[j] : 0);
    }
    (void)nthreads;
    return 0;
}

/* Q8 down projection: all M x H outputs, or the n elements (rows[j],
 * cols[j]) when rows != NULL. */
int q4o_q8_down_proj(const uint16_t *mid, int64_t M, int64_t I, int64_t H,
                     int32_t E, const int8_t *down_w, const float *down_s,
                     const int32_t *row_offsets, int64_t n,
                     const int64_t *rows, const int64_t *cols, uint16_t *out,
                     float *out32, double *dabs, int nthreads)
{
    if (M < 0 || I <= 0 || H <= 0 || E <= 0)
        return -1;
    if (row_offsets[0] != 0 || row_offsets[E] != M)
        return -2;
    for (int32_t e = 0; e < E; ++e)
        if (row_offsets[e + 1] < row_offsets[e])
            return -2;
    if (rows == 0)
        n = M * H;
    else
        for (int64_t j = 0; j < n; ++j)
            if (rows[j] < 0 || rows[j] >= M || cols[j] < 0 || cols[j] >= H)
                return -4;
#ifdef _OPENMP
    if (nthreads <= 0)
        nthreads = omp_get_max_threads();
#pragma omp parallel for schedule(dynamic, 8) num_threads(nthreads)
#endif
    for (int64_t j = 0; j < n; ++j) {
        const int64_t p = rows ? rows[j] : j / H, h = rows ? cols[j] : j % H;
        const int32_t e = q4o_expert_of_row(row_offsets, E, p);
        double a;
        const double D = q4o_dot_q8(down_w + ((int64_t)e * H + h) * I,
                                    mid + p * I, I, &a);
        const float v = (float)(D * (double)down_s[(int64_t)e * H + h]);
        out[j] = q4o_bf16_rne(v);
        if (out32) out32[j] = v;
        if (dabs) dabs[j] = a;
    }
    (void)nthreads;
    return 0;
}

/* ---- trellis (QTIP 1MAD) gate/up, factored row scale ---------------------
 * Codes of one row: H / Tb blocks of Tb * k / 32 words each (axis 1: coded
 * along the input); bit b of a block is bit b % 32 of word b / 32.  Scales
 * are f16 bit patterns, one per row. */

/* The L-bit state of weight t of a block of nbits = Tb * k bits: the bits
 * [p, p + L) with p = (Tb - 1 - t) * k, taken modulo nbits (page 54,
 * codebook.ts, trellis_state). */
static uint32_t q4o_trellis_state(const uint32_t *blk, int64_t nbits,
                                  int64_t t, int64_t Tb, int k, int L)
{
    const int64_t p = (Tb - 1 - t) * k;
    uint32_t s = 0;
    for (int j = 0; j < L; ++j) {
        const int64_t b = (p + j) % nbits;
        s |= ((blk[b >> 5] >> (b & 31)) & 1u) << j;
    }
    return s;
}

/* Code value of state s (page 54, codebook.ts, trellis_y): the sum of the
 * four bytes of s * 34038481 + 76625530 (mod 2^32), minus 510. */
int q4o_trellis_y(uint32_t s)
{
    const uint32_t x = s * 34038481u + 76625530u;
    return (int)(x & 255u) + (int)((x >> 8) & 255u) + (int)((x >> 16) & 255u) +
           (int)(x >> 24) - 510;
}

/* f16 bits -> f32 (exact). */
static float q4o_f16_to_f32(uint16_t h)
{
    const int sign = h >> 15, e = (h >> 10) & 31, m = h & 1023;
    double v;
    if (e == 0)
        v = ldexp((double)m, -24);
    else if (e == 31)
        v = m ? NAN : INFINITY;
    else
        v = ldexp((double)(1024 + m), e - 25);
    return (float)(sign ? -v : v);
}

/* The factored scale of a row: RN32(s * RN32(1 / 147.800537109375)) (page
 * 57, gate-up-mma.ts: float(scale) * TRELLIS_RCP). */
float q4o_trellis_scale(uint16_t s_f16)
{
    const float rcp = (float)(1.0 / 147.800537109375);
    return (float)((double)q4o_f16_to_f32(s_f16) * (double)rcp);
}

/* sum_k y_k x_k over one row (f64: exact), and sum_k |y_k x_k|. */
static double q4o_trellis_dot(const uint32_t *row, const uint16_t *xrow,
                              int64_t H, int64_t Tb, int k, int L,
                              double *absdot)
{
    const int64_t wpb = Tb * k / 32, nbits = Tb * k;
    double s = 0.0, a = 0.0;
    for (int64_t c = 0; c < H; ++c) {
        const int64_t blk = c / Tb, t = c % Tb;
        const int y = q4o_trellis_y(
            q4o_trellis_state(row + blk * wpb, nbits, t, Tb, k, L));
        const double prod = (double)y * (double)q4o_bf16_to_f32(xrow[c]);
        s += prod;
        a += fabs(prod);
    }
    *absdot = a;
    return s;
}

/* All M x I outputs, or (rows != NULL) the n elements (rows[j], cols[j]).
 * gate_codes: uint32 [E, I, H / Tb * Tb * kg / 32], up_codes likewise with
 * ku; gate_s/up_s: f16 bits [E, I].  Outputs as q4o_gate_up_swiglu
 * (gate32 = RN32(G * gate scale)); tail 0 ends with the page 52 tail (the
 * pages' equal-width kernels, gate-up-mma.ts), tail 1 with MLX's
 * (q4o_tail_mlx, the mixed-width kernel).  Needs H % Tb == 0,
 * Tb * k % 32 == 0, 1 <= L <= 24, L <= Tb * k. */
int q4o_trellis_gate_up_swiglu(const uint16_t *x, int64_t T, int64_t H,
                               int64_t I, int32_t E,
                               const uint32_t *gate_codes,
                               const uint32_t *up_codes,
                               const uint16_t *gate_s, const uint16_t *up_s,
                               int kg, int ku, int L, int64_t Tb,
                               const int32_t *row_offsets,
                               const int32_t *token_of_row, int64_t M,
                               int64_t n, const int64_t *rows,
                               const int64_t *cols, uint16_t *out,
                               float *gate32, float *up32, double *gabs,
                               double *uabs, int tail, int nthreads)
{
    if (tail != 0 && tail != 1)
        return -1;
    if (T < 0 || H <= 0 || I <= 0 || E <= 0 || M < 0 || Tb <= 0 ||
        H % Tb != 0 || kg < 1 || ku < 1 || kg > 8 || ku > 8 ||
        (Tb * kg) % 32 != 0 || (Tb * ku) % 32 != 0 || L < 1 || L > 24 ||
        L > Tb * kg || L > Tb * ku)
        return -1;
    if (row_offsets[0] != 0 || row_offsets[E] != M)
        return -2;
    for (int32_t e = 0; e < E; ++e)
        if (row_offsets[e + 1] < row_offsets[e])
            return -2;
    for (int64_t p = 0; p < M; ++p)
        if (token_of_row[p] < 0 || token_of_row[p] >= T)
            return -3;
    if (rows == 0)
        n = M * I;
    else
        for (int64_t j = 0; j < n; ++j)
            if (rows[j] < 0 || rows[j] >= M || cols[j] < 0 || cols[j] >= I)
                return -4;
    const int64_t gwords = H / Tb * (Tb * kg / 32);
    const int64_t uwords = H / Tb * (Tb * ku / 32);
#ifdef _OPENMP
    if (nthreads <= 0)
        nthreads = omp_get_max_threads();
#pragma omp parallel for schedule(dynamic, 4) num_threads(nthreads)
#endif
    for (int64_t j = 0; j < n; ++j) {
        const int64_t p = rows ? rows[j] : j / I, i = rows ? cols[j] : j % I;
        const int32_t e = q4o_expert_of_row(row_offsets, E, p);
        const uint16_t *xrow = x + (int64_t)token_of_row[p] * H;
        double ga, ua;
        const double G = q4o_trellis_dot(
            gate_codes + ((int64_t)e * I + i) * gwords, xrow, H, Tb, kg, L,
            &ga);
        const double U = q4o_trellis_dot(
            up_codes + ((int64_t)e * I + i) * uwords, xrow, H, Tb, ku, L,
            &ua);
        const float g32 = (float)(G * (double)q4o_trellis_scale(
                                          gate_s[(int64_t)e * I + i]));
        const float u32 = (float)(U * (double)q4o_trellis_scale(
                                          up_s[(int64_t)e * I + i]));
        uint16_t res[5];
        q4o_tail_of(tail, g32, u32, res);
        out[j] = res[4];
        if (gate32) gate32[j] = g32;
        if (up32) up32[j] = u32;
        if (gabs) gabs[j] = ga;
        if (uabs) uabs[j] = ua;
    }
    (void)nthreads;
    return 0;
}

/* The code values of one block (debug/pin helper): y[t] for t < Tb. */
int q4o_trellis_block_codes(const uint32_t *blk, int64_t Tb, int k, int L,
                            int32_t *y)
{
    if (Tb <= 0 || k < 1 || (Tb * k) % 32 != 0 || L < 1 || L > 24 ||
        L > Tb * k)
        return -1;
    for (int64_t t = 0; t < Tb; ++t)
        y[t] = q4o_trellis_y(q4o_trellis_state(blk, Tb * k, t, Tb, k, L));
    return 0;
}

/* The states of one block (pin helper). */
int q4o_trellis_block_states(const uint32_t *blk, int64_t Tb, int k, int L,
                             uint32_t *st)
{
    if (Tb <= 0 || k < 1 || (Tb * k) % 32 != 0 || L < 1 || L > 24 ||
        L > Tb * k)
        return -1;
    for (int64_t t = 0; t < Tb; ++t)
        st[t] = q4o_trellis_state(blk, Tb * k, t, Tb, k, L);
    return 0;
}

int q4o_group_rows(const int32_t *topk, int64_t T, int32_t k, int32_t E,
                   int32_t *row_offsets, int32_t *token_of_row,
                   int32_t *row_of_pair)
{
    if (T < 0 || k <= 0 || E <= 0)
        return -1;
    for (int32_t e = 0; e <= E; ++e)
        row_offsets[e] = 0;
    for (int64_t q = 0; q < T * k; ++q) {
        if (topk[q] < 0 || topk[q] >= E)
            return -1;
        row_offsets[topk[q] + 1] += 1;
    }
    for (int32_t e = 0; e < E; ++e)
        row_offsets[e + 1] += row_offsets[e];
    for (int32_t e = 0; e < E; ++e) {
        /* walk the pairs in order, so equal experts keep token order */
        int32_t next = row_offsets[e];
        for (int64_t q = 0; q < T * k; ++q) {
            if (topk[q] != e)
                continue;
            token_of_row[next] = (int32_t)(q / k);
            row_of_pair[q] = next;
            ++next;
        }
    }
    return 0;
}

int q4o_max_threads(void)
{
#ifdef _OPENMP
    return omp_get_max_threads();
#else
    return 1;
#endif
}
