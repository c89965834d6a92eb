// q4moe_api.cu -- the C ABI: argument validation, the device status word and
// kernel dispatch.  Validation rules follow the pages' host checks (page 52,
// streamed-experts.ts, validateCall; page 51, layout.ts, validateRange).
#include <algorithm>
#include <atomic>
#include <climits>
#include <cstdarg>
#include <cstdio>
#include <cstring>
#include <mutex>
#include <string>

#include "q4moe_internal.cuh"

namespace {

thread_local std::string t_last_error;

int fail(int code, const char *fmt, ...) {
    char buf[512];
    va_list ap;
    va_start(ap, fmt);
    vsnprintf(buf, sizeof buf, fmt, ap);
    va_end(ap);
    t_last_error = buf;
    return code;
}

int ok() {
    t_last_error.clear();
    return Q4MOE_OK;
}

int cuda_fail(cudaError_t err, const char *what) {
    return fail(Q4MOE_ERR_CUDA, "%s: %s (%d)", what, cudaGetErrorString(err),
                (int)err);
}

// Device status word: Q4MOE_DEV_* bits raised by kernels that meet
// inconsistent device-side data.  One per device (a __device__ variable
// exists once in every device context that loads the library).
__device__ unsigned int g_status_word;
// bf16 sigmoid of every bf16 gate value for each tail (page 52's, then
// MLX's): constant data of the library image, written at build time by the
// package's table generator (up_swiglu_gb300/build.py), so no call has to
// fill it
__device__ __align__(16) const uint16_t
    g_sigmoid_table[2 * q4moe::kSigmoidTable] = {
#include "q4moe_sigmoid_table.inc"
};

constexpr int kMaxDevices = 64;
struct DeviceInfo {
    bool ready = false;
    bool supported = false;
    int num_sms = 0;
    unsigned int *status = nullptr;
    const uint16_t *sigmoid = nullptr;
    char why[160] = {0};
};
DeviceInfo g_devices[kMaxDevices];
std::mutex g_devices_mutex;

// Per-device set-up, done on the first call that needs it with that device
// current: the compute capability check and the device addresses of the
// status word and the sigmoid tables (host queries only: nothing is
// launched and no stream is synchronised).
int device_info(DeviceInfo **out) {
    int dev = 0;
    cudaError_t err = cudaGetDevice(&dev);
    if (err != cudaSuccess)
        return cuda_fail(err, "cudaGetDevice");
    if (dev < 0 || dev >= kMaxDevices)
        return fail(Q4MOE_ERR_DEVICE, "device ordinal %d out of range", dev);
    std::lock_guard<std::mutex> lock(g_devices_mutex);
    DeviceInfo &d = g_devices[dev];
    if (!d.ready) {
        int major = 0, minor = 0, sms = 0;
        if ((err = cudaDeviceGetAttribute(
                 &major, cudaDevAttrComputeCapabilityMajor, dev)) !=
                cudaSuccess ||
            (err = cudaDeviceGetAttribute(
                 &minor, cudaDevAttrComputeCapabilityMinor, dev)) !=
                cudaSuccess ||
            (err = cudaDeviceGetAttribute(
                 &sms, cudaDevAttrMultiProcessorCount, dev)) != cudaSuccess)
            return cuda_fail(err, "cudaDeviceGetAttribute");
        d.num_sms = sms;
        d.supported = (major == 10 && minor == 3);
        if (!d.supported) {
            snprintf(d.why, sizeof d.why,
                     "device %d is sm_%d%d; this library is built for sm_103",
                     dev, major, minor);
        } else {
            void *p = nullptr;
            err = cudaGetSymbolAddress(&p, g_status_word);
            if (err != cudaSuccess)
                return cuda_fail(err, "cudaGetSymbolAddress(status word)");
            d.status = static_cast<unsigned int *>(p);
            if ((err = cudaGetSymbolAddress(&p, g_sigmoid_table)) !=
                cudaSuccess)
                return cuda_fail(err, "cudaGetSymbolAddress(sigmoid table)");
            d.sigmoid = static_cast<const uint16_t *>(p);
        }
        d.ready = true;
    }
    if (!d.supported)
        return fail(Q4MOE_ERR_DEVICE, "%s", d.why);
    *out = &d;
    return Q4MOE_OK;
}

bool aligned(const void *p, uintptr_t a) {
    return (reinterpret_cast<uintptr_t>(p) & (a - 1)) == 0;
}

bool overlap(const void *a, int64_t na, const void *b, int64_t nb) {
    const uintptr_t x = reinterpret_cast<uintptr_t>(a),
                    y = reinterpret_cast<uintptr_t>(b);
    return na > 0 && nb > 0 && x < y + (uintptr_t)nb && y < x + (uintptr_t)na;
}

int check_range(int64_t off, int64_t len, int64_t slab_bytes,
                const char *what) {
    if (off < 0)
        return fail(Q4MOE_ERR_RANGE, "%s offset must be non-negative", what);
    if (len < 0 || off > slab_bytes || len > slab_bytes - off)
        return fail(Q4MOE_ERR_RANGE, "%s exceed the expert slab", what);
    return Q4MOE_OK;
}

int validate_layout(const q4moe_layout_t *L) {
    if (L == nullptr)
        return fail(Q4MOE_ERR_INVALID_ARG, "layout is null");
    const int64_t H = L->hidden_size, I = L->intermediate_size;
    const bool q8 = L->weight_format == Q4MOE_FORMAT_Q8;
    if (L->weight_format != Q4MOE_FORMAT_Q4 && !q8)
        return fail(Q4MOE_ERR_INVALID_ARG, "unknown weight format %lld",
                    (long long)L->weight_format);
    if (H <= 0 || I <= 0)
        return fail(Q4MOE_ERR_INVALID_ARG,
                    "hidden and intermediate sizes must be positive");
    if (H % (q8 ? 4 : 8) != 0)
        return fail(Q4MOE_ERR_INVALID_ARG,
                    q8 ? "Q8 hidden size must be divisible by 4"
                       : "Q4 hidden size must be divisible by 8");
    if (I % 4 != 0)
        return fail(Q4MOE_ERR_INVALID_ARG,
                    "intermediate size must be divisible by 4");
    if (H > (INT64_C(1) << 24) || I > (INT64_C(1) << 24))
        return fail(Q4MOE_ERR_INVALID_ARG, "dimensions above 2^24");
    if (L->slab_bytes <= 0)
        return fail(Q4MOE_ERR_INVALID_ARG, "slab bytes must be positive");
    int rc;
    const int64_t wbytes = q8 ? I * H : I * (H / 2), sbytes = I * 4;
    if ((rc = check_range(L->gate_w_offset, wbytes, L->slab_bytes,
                          "gate weights")) ||
        (rc = check_range(L->up_w_offset, wbytes, L->slab_bytes,
                          "up weights")) ||
        (rc = check_range(L->gate_s_offset, sbytes, L->slab_bytes,
                          "gate scales")) ||
        (rc = check_range(L->up_s_offset, sbytes, L->slab_bytes,
                          "up scales")))
        return rc;
    if ((L->gate_w_offset | L->up_w_offset | L->gate_s_offset |
         L->up_s_offset) % 4 != 0)
        return fail(Q4MOE_ERR_ALIGNMENT,
                    "slab sections must start on 4-byte boundaries");
    // the down sections, when present (both offsets >= 0)
    if ((L->down_w_offset < 0) != (L->down_s_offset < 0))
        return fail(Q4MOE_ERR_INVALID_ARG,
                    "down weights and down scales must both be present or "
                    "both absent (negative offsets)");
    if (L->down_w_offset >= 0) {
        if (!q8 && I % 8 != 0)
            return fail(Q4MOE_ERR_INVALID_ARG,
                        "Q4 down sections need I divisible by 8");
        if ((rc = check_range(L->down_w_offset, q8 ? H * I : H * (I / 2),
                              L->slab_bytes,
                              "down weights")) ||
            (rc = check_range(L->down_s_offset, H * 4, L->slab_bytes,
                              "down scales")))
            return rc;
        if ((L->down_w_offset | L->down_s_offset) % 4 != 0)
            return fail(Q4MOE_ERR_ALIGNMENT,
                        "slab sections must start on 4-byte boundaries");
    }
    return Q4MOE_OK;
}

// Slab placement (base + e * stride or a pointer table), shared by the Q4/Q8
// and trellis slab descriptors.
int check_placement(int32_t num_experts, int32_t reserved0, const void *base,
                    int64_t stride, const void *const *ptrs,
                    int64_t slab_bytes) {
    if (num_experts <= 0 || num_experts > Q4MOE_MAX_EXPERTS)
        return fail(Q4MOE_ERR_INVALID_ARG, "num_experts must be in 1..%d",
                    Q4MOE_MAX_EXPERTS);
    if (reserved0 != 0)
        return fail(Q4MOE_ERR_INVALID_ARG, "reserved field must be 0");
    if (ptrs == nullptr) {
        if (base == nullptr)
            return fail(Q4MOE_ERR_INVALID_ARG,
                        "slab base is null and no pointer table given");
        if (!aligned(base, Q4MOE_SLAB_ALIGNMENT))
            return fail(Q4MOE_ERR_ALIGNMENT,
                        "slab base must be %d-byte aligned",
                        Q4MOE_SLAB_ALIGNMENT);
        if (stride % Q4MOE_SLAB_ALIGNMENT != 0 ||
            (num_experts > 1 && stride < slab_bytes) || stride < 0)
            return fail(Q4MOE_ERR_ALIGNMENT,
                        "slab stride must be a multiple of %d and at least "
                        "the slab size", Q4MOE_SLAB_ALIGNMENT);
    } else if (!aligned(ptrs, 8)) {
        return fail(Q4MOE_ERR_ALIGNMENT, "slab pointer table misaligned");
    }
    return Q4MOE_OK;
}

// Trellis layout: geometry and section ranges.
int validate_trellis_layout(const q4moe_trellis_layout_t *L) {
    if (L == nullptr)
        return fail(Q4MOE_ERR_INVALID_ARG, "layout is null");
    const int64_t H = L->hidden_size, I = L->intermediate_size;
    const int64_t T = L->block_size;
    if (H <= 0 || I <= 0 || T <= 0 || T % 32 != 0 || H % T != 0)
        return fail(Q4MOE_ERR_INVALID_ARG,
                    "need H, I > 0, block size a multiple of 32 dividing H");
    if (H > (INT64_C(1) << 24) || I > (INT64_C(1) << 24) || T > 65536)
        return fail(Q4MOE_ERR_INVALID_ARG, "dimensions too large");
    if (L->gate_bits < 1 || L->gate_bits > 8 || L->up_bits < 1 ||
        L->up_bits > 8)
        return fail(Q4MOE_ERR_INVALID_ARG, "code widths must be 1..8 bits");
    if (L->window_bits < 1 || L->window_bits > 24 ||
        L->window_bits > T * L->gate_bits || L->window_bits > T * L->up_bits)
        return fail(Q4MOE_ERR_INVALID_ARG, "window bits must be 1..24");
    if (L->slab_bytes <= 0)
        return fail(Q4MOE_ERR_INVALID_ARG, "slab bytes must be positive");
    int rc;
    if ((rc = check_range(L->gate_codes_offset, I * H * L->gate_bits / 8,
                          L->slab_bytes, "gate codes")) ||
        (rc = check_range(L->up_codes_offset, I * H * L->up_bits / 8,
                          L->slab_bytes, "up codes")) ||
        (rc = check_range(L->gate_scales_offset, I * 2, L->slab_bytes,
                          "gate scales")) ||
        (rc = check_range(L->up_scales_offset, I * 2, L->slab_bytes,
                          "up scales")))
        return rc;
    if ((L->gate_codes_offset | L->up_codes_offset) % 4 != 0 ||
        (L->gate_scales_offset | L->up_scales_offset) % 2 != 0)
        return fail(Q4MOE_ERR_ALIGNMENT,
                    "codes must start on 4-byte, scales on 2-byte boundaries");
    return Q4MOE_OK;
}

// Checks of the slab placement and the call's dimensions shared by every
// call that reads expert slabs.
int check_slabs(const q4moe_slabs_t *slabs, int64_t H, int64_t I,
                int64_t M) {
    if (slabs == nullptr)
        return fail(Q4MOE_ERR_INVALID_ARG, "expert_slabs is null");
    int rc = validate_layout(&slabs->layout);
    if (rc)
        return rc;
    const q4moe_layout_t &L = slabs->layout;
    if (H != L.hidden_size || I != L.intermediate_size)
        return fail(Q4MOE_ERR_INVALID_ARG,
                    "H, I (%lld, %lld) differ from the slab layout's "
                    "(%lld, %lld)", (long long)H, (long long)I,
                    (long long)L.hidden_size,
                    (long long)L.intermediate_size);
    if ((rc = check_placement(slabs->num_experts, slabs->reserved0,
                              slabs->base, slabs->slab_stride,
                              slabs->slab_ptrs, L.slab_bytes)))
        return rc;
    if (M < 0 || M > INT32_MAX)
        return fail(Q4MOE_ERR_INVALID_ARG, "M must be in 0..2^31-1");
    if (M > 0 && M * std::max(H, I) > (INT64_C(1) << 40))
        return fail(Q4MOE_ERR_INVALID_ARG, "output too large");
    return Q4MOE_OK;
}

int check_kernel_options(const q4moe_options_t &o, bool trellis = false) {
    if ((o.matvec_tile != 0 && o.matvec_tile != 16 && o.matvec_tile != 32 &&
         o.matvec_tile != 64 && o.matvec_tile != 128) ||
        o.kernel < Q4MOE_KERNEL_AUTO ||
        o.kernel > Q4MOE_KERNEL_BATCH_INVARIANT || o.num_tokens < 0 ||
        o.tail < Q4MOE_TAIL_AUTO || o.tail > Q4MOE_TAIL_MLX ||
        o.reserved1 != 0)
        return fail(Q4MOE_ERR_INVALID_ARG, "bad options");
    if (!trellis && o.tail == Q4MOE_TAIL_MLX)
        return fail(Q4MOE_ERR_INVALID_ARG,
                    "the MLX tail is built for trellis codes only");
    if (!aligned(o.gate_f32, 4) || !aligned(o.up_f32, 4))
        return fail(Q4MOE_ERR_ALIGNMENT, "debug outputs must be 4-byte "
                                         "aligned");
    return Q4MOE_OK;
}

// Checks of a down projection's own arguments (before anything launches).
int check_down(const q4moe_slabs_t *slabs, const void *mid, const void *out,
               const int32_t *row_offsets, int64_t M,
               const q4moe_options_t &o, bool own_options) {
    if (slabs->layout.down_w_offset < 0)
        return fail(Q4MOE_ERR_INVALID_ARG,
                    "the slab layout has no down sections");
    if (row_offsets == nullptr)
        return fail(Q4MOE_ERR_INVALID_ARG, "row_offsets_per_expert is null");
    if (M > 0 && (mid == nullptr || out == nullptr))
        return fail(Q4MOE_ERR_INVALID_ARG, "null pointer");
    if (!aligned(mid, 16))
        return fail(Q4MOE_ERR_ALIGNMENT, "mid must be 16-byte aligned");
    if (!aligned(out, 2))
        return fail(Q4MOE_ERR_ALIGNMENT, "out must be 2-byte aligned");
    if (own_options && (o.num_tokens != 0 || o.up_f32 != nullptr ||
                        o.workspace != nullptr || o.workspace_bytes != 0))
        return fail(Q4MOE_ERR_INVALID_ARG,
                    "the down projection takes no num_tokens, up_f32 or "
                    "workspace");
    return Q4MOE_OK;
}

std::atomic<int64_t> g_launches{0};

}  // namespace

namespace q4moe {
void count_launches(int n) { g_launches.fetch_add(n); }
int report_error(int code, const char *message) {
    return fail(code, "%s", message);
}
}  // namespace q4moe

namespace {

q4moe::GateUpArgs base_args(const q4moe_slabs_t *slabs, int64_t M,
                            const DeviceInfo *d, const q4moe_options_t &o) {
    q4moe::GateUpArgs a{};
    a.base = static_cast<const uint8_t *>(slabs->base);
    a.stride = slabs->slab_stride;
    a.slab_ptrs = reinterpret_cast<const uint8_t *const *>(slabs->slab_ptrs);
    a.M = M;
    a.E = slabs->num_experts;
    a.status = d->status;
    a.num_sms = d->num_sms;
    a.matvec_tile = o.matvec_tile;
    a.sigmoid = d->sigmoid;
    a.q8 = slabs->layout.weight_format == Q4MOE_FORMAT_Q8;
    return a;
}

// Kernel choice and launches of one projection (gate/up or down).
int dispatch(q4moe::GateUpArgs &a, const q4moe_options_t &o,
             const DeviceInfo *d, cudaStream_t stream) {
    const bool gemm_ok = q4moe::gemm_supported(a.H, a.I, a);
    int32_t matvec_max = INT32_MAX;
    if (o.kernel == Q4MOE_KERNEL_BATCH_INVARIANT) {
        // the matvec alone, one unit height for every call
        a.invariant = 1;
        if (a.matvec_tile == 0)
            a.matvec_tile = 128;
    } else if (o.kernel == Q4MOE_KERNEL_GEMM) {
        if (!gemm_ok)
            return fail(Q4MOE_ERR_INVALID_ARG,
                        a.down ? "the tensor-core GEMM needs I %% 64 == 0, "
                                 "H %% 128 == 0 and 16-byte aligned slab "
                                 "sections"
                               : "the tensor-core GEMM needs H %% 64 == 0, "
                                 "I %% 128 == 0 and 16-byte aligned slab "
                                 "sections");
        matvec_max = 0;
    } else if (o.kernel == Q4MOE_KERNEL_AUTO && gemm_ok) {
        // Several experts: when the call has at least 4 rows per expert on
        // average, experts above 16 rows (32 for the down projection) go
        // to the GEMM and the rest to the matvec (both launched; an
        // expert's count is known on the device only); with fewer rows the
        // matvec takes every expert (no GEMM launch).  Measured on the
        // verify workload (1024 rows over 160 experts, Zipf): gate/up 0.344
        // ms on the matvec alone, 0.294 ms with the experts above 16 rows
        // on the GEMM (12: 0.334, 24: 0.293, 32: 0.321); the down
        // projection 0.170 ms above 16, 0.162 above 32 (48: 0.179, 64:
        // 0.184); a GEMM launch that finds no expert costs ~3 % of the
        // grouped decode (256 rows over 128 experts).  From 128 rows per
        // expert on average the GEMM takes every expert and the matvec is
        // not launched: an expert of at most 16 rows is then rare even
        // under Zipf(1.1) routing over 160 experts, and the matvec launch
        // that finds none cost 3.5 us of the prefill step (0.896 ->
        // 0.893 ms).  One expert: the GEMM when its rows fill every SM
        // with tiles.
        const int64_t row_tiles = q4moe::gemm_row_tiles(a);
        const int64_t tiles = (a.M + 255) / 256 * row_tiles;
        if (a.E > 1 && a.M >= 128 * (int64_t)a.E) {
            matvec_max = 0;
        } else if (a.E > 1 && a.M >= 4 * (int64_t)a.E) {
            matvec_max = a.down ? 32 : 16;
        } else if (a.E == 1 && a.M > 48 && tiles >= d->num_sms) {
            matvec_max = 0;
        }
    }
    a.matvec_max_rows = matvec_max;

    cudaError_t err = cudaSuccess;
    a.matvec_last = matvec_max >= a.M;       // no GEMM launch after it
    if (matvec_max > 0 && (err = q4moe::launch_matvec(a, stream)) !=
                              cudaSuccess)
        return cuda_fail(err, "matvec launch");
    // every expert has at most M rows: no GEMM work when M <= matvec_max
    if (matvec_max < a.M && (err = q4moe::launch_gemm(a, stream)) !=
                                cudaSuccess)
        return cuda_fail(err, "gemm launch");
    return ok();
}

}  // namespace

extern "C" {

int64_t q4moe_launch_count(void) { return g_launches.load(); }

int q4moe_abi_version(void) { return Q4MOE_ABI_VERSION; }

const char *q4moe_last_error(void) { return t_last_error.c_str(); }

int64_t q4moe_workspace_bytes(int64_t M, int64_t H) {
    if (M < 0 || H < 0)
        return fail(Q4MOE_ERR_INVALID_ARG, "negative size");
    return (M * H * 2 + 255) / 256 * 256;
}

int q4moe_canonical_layout(int64_t H, int64_t I, q4moe_layout_t *layout) {
    return q4moe_canonical_layout_format(H, I, Q4MOE_FORMAT_Q4, layout);
}

int q4moe_canonical_layout_format(int64_t H, int64_t I, int32_t format,
                                  q4moe_layout_t *layout) {
    if (layout == nullptr)
        return fail(Q4MOE_ERR_INVALID_ARG, "layout is null");
    const bool q8 = format == Q4MOE_FORMAT_Q8;
    if (format != Q4MOE_FORMAT_Q4 && !q8)
        return fail(Q4MOE_ERR_INVALID_ARG, "unknown weight format %d",
                    (int)format);
    q4moe_layout_t L{};
    L.hidden_size = H;
    L.intermediate_size = I;
    L.weight_format = format;
    if (H <= 0 || I <= 0 || H % (q8 ? 4 : 8) != 0 || I % 4 != 0)
        return fail(Q4MOE_ERR_INVALID_ARG,
                    "need H > 0, H %% %d == 0, I > 0, I %% 4 == 0",
                    q8 ? 4 : 8);
    if (H > (INT64_C(1) << 24) || I > (INT64_C(1) << 24))
        return fail(Q4MOE_ERR_INVALID_ARG, "dimensions above 2^24");
    const int64_t wbytes = q8 ? I * H : I * (H / 2);
    L.gate_w_offset = 0;
    L.up_w_offset = wbytes;
    L.gate_s_offset = 2 * wbytes;
    L.up_s_offset = 2 * wbytes + 4 * I;
    int64_t used = 2 * wbytes + 8 * I;
    L.down_w_offset = L.down_s_offset = -1;
    if (q8 || I % 8 == 0) {
        L.down_w_offset = (used + 255) / 256 * 256;
        L.down_s_offset = L.down_w_offset + wbytes;
        used = L.down_s_offset + 4 * H;
    }
    L.slab_bytes = (used + Q4MOE_SLAB_ALIGNMENT - 1) /
                   Q4MOE_SLAB_ALIGNMENT * Q4MOE_SLAB_ALIGNMENT;
    *layout = L;
    return ok();
}

int q4moe_validate_layout(const q4moe_layout_t *layout) {
    const int rc = validate_layout(layout);
    return rc ? rc : ok();
}

int q4moe_pack_slab(const q4moe_layout_t *L, const uint32_t *gate_w,
                    const uint32_t *up_w, const float *gate_s,
                    const float *up_s, void *slab_host) {
    int rc = validate_layout(L);
    if (rc)
        return rc;
    if (!gate_w || !up_w || !gate_s || !up_s || !slab_host)
        return fail(Q4MOE_ERR_INVALID_ARG, "null pointer");
    const int64_t H = L->hidden_size, I = L->intermediate_size;
    const int64_t wbytes =
        L->weight_format == Q4MOE_FORMAT_Q8 ? I * H : I * (H / 2);
    uint8_t *s = static_cast<uint8_t *>(slab_host);
    memset(s, 0, (size_t)L->slab_bytes);
    memcpy(s + L->gate_w_offset, gate_w, (size_t)wbytes);
    memcpy(s + L->up_w_offset, up_w, (size_t)wbytes);
    memcpy(s + L->gate_s_offset, gate_s, (size_t)(I * 4));
    memcpy(s + L->up_s_offset, up_s, (size_t)(I * 4));
    return ok();
}

int q4moe_pack_slab_down(const q4moe_layout_t *L, const uint32_t *down_w,
                         const float *down_s, void *slab_host) {
    int rc = validate_layout(L);
    if (rc)
        return rc;
    if (L->down_w_offset < 0)
        return fail(Q4MOE_ERR_INVALID_ARG, "the layout has no down sections");
    if (!down_w || !down_s || !slab_host)
        return fail(Q4MOE_ERR_INVALID_ARG, "null pointer");
    const int64_t H = L->hidden_size, I = L->intermediate_size;
    uint8_t *s = static_cast<uint8_t *>(slab_host);
    memcpy(s + L->down_w_offset, down_w,
           (size_t)(L->weight_format == Q4MOE_FORMAT_Q8 ? H * I
                                                        : H * (I / 2)));
    memcpy(s + L->down_s_offset, down_s, (size_t)(H * 4));
    return ok();
}

int q4moe_trellis_canonical_layout(int64_t H, int64_t I, int32_t block_size,
                                   int32_t window_bits, int32_t gate_bits,
                                   int32_t up_bits,
                                   q4moe_trellis_layout_t *layout) {
    if (layout == nullptr)
        return fail(Q4MOE_ERR_INVALID_ARG, "layout is null");
    q4moe_trellis_layout_t L{};
    L.hidden_size = H;
    L.intermediate_size = I;
    L.block_size = block_size;
    L.window_bits = window_bits;
    L.gate_bits = gate_bits;
    L.up_bits = up_bits;
    L.slab_bytes = 1;
    // the geometry checks of validate_trellis_layout, before any size
    if (H <= 0 || I <= 0 || block_size <= 0 || block_size % 32 != 0 ||
        H % block_size != 0 || H > (INT64_C(1) << 24) ||
        I > (INT64_C(1) << 24) || gate_bits < 1 || gate_bits > 8 ||
        up_bits < 1 || up_bits > 8)
        return fail(Q4MOE_ERR_INVALID_ARG, "bad trellis geometry");
    auto up256 = [](int64_t v) { return (v + 255) / 256 * 256; };
    L.gate_codes_offset = 0;
    L.up_codes_offset = up256(I * H * gate_bits / 8);
    L.gate_scales_offset = up256(L.up_codes_offset + I * H * up_bits / 8);
    L.up_scales_offset = up256(L.gate_scales_offset + 2 * I);
    const int64_t used = L.up_scales_offset + 2 * I;
    L.slab_bytes = (used + Q4MOE_SLAB_ALIGNMENT - 1) / Q4MOE_SLAB_ALIGNMENT *
                   Q4MOE_SLAB_ALIGNMENT;
    const int rc = validate_trellis_layout(&L);
    if (rc)
        return rc;
    *layout = L;
    return ok();
}

int q4moe_trellis_pack_slab(const q4moe_trellis_layout_t *L,
                            const uint32_t *gate_codes,
                            const uint32_t *up_codes,
                            const uint16_t *gate_scales,
                            const uint16_t *up_scales, void *slab_host) {
    int rc = validate_trellis_layout(L);
    if (rc)
        return rc;
    if (!gate_codes || !up_codes || !gate_scales || !up_scales || !slab_host)
        return fail(Q4MOE_ERR_INVALID_ARG, "null pointer");
    const int64_t H = L->hidden_size, I = L->intermediate_size;
    uint8_t *s = static_cast<uint8_t *>(slab_host);
    memset(s, 0, (size_t)L->slab_bytes);
    memcpy(s + L->gate_codes_offset, gate_codes,
           (size_t)(I * H * L->gate_bits / 8));
    memcpy(s + L->up_codes_offset, up_codes, (size_t)(I * H * L->up_bits / 8));
    memcpy(s + L->gate_scales_offset, gate_scales, (size_t)(2 * I));
    memcpy(s + L->up_scales_offset, up_scales, (size_t)(2 * I));
    return ok();
}

int q4moe_trellis_gate_up_swiglu(const void *x,
                                 const q4moe_trellis_slabs_t *slabs,
                                 const int32_t *row_offsets,
                                 const int32_t *token_of_row, int64_t M,
                                 int64_t H, int64_t I, void *out,
                                 const q4moe_options_t *opts,
                                 cudaStream_t stream) {
    if (slabs == nullptr)
        return fail(Q4MOE_ERR_INVALID_ARG, "expert_slabs is null");
    int rc = validate_trellis_layout(&slabs->layout);
    if (rc)
        return rc;
    const q4moe_trellis_layout_t &L = slabs->layout;
    if (H != L.hidden_size || I != L.intermediate_size)
        return fail(Q4MOE_ERR_INVALID_ARG,
                    "H, I differ from the trellis layout's");
    if ((rc = check_placement(slabs->num_experts, slabs->reserved0,
                              slabs->base, slabs->slab_stride,
                              slabs->slab_ptrs, L.slab_bytes)))
        return rc;
    if (M < 0 || M > INT32_MAX || (M > 0 && M * I > (INT64_C(1) << 40)))
        return fail(Q4MOE_ERR_INVALID_ARG, "M out of range");
    if (row_offsets == nullptr)
        return fail(Q4MOE_ERR_INVALID_ARG, "row_offsets_per_expert is null");
    if (M > 0 && (x == nullptr || token_of_row == nullptr || out == nullptr))
        return fail(Q4MOE_ERR_INVALID_ARG, "null pointer");
    if (!aligned(x, 16))
        return fail(Q4MOE_ERR_ALIGNMENT, "x must be 16-byte aligned");
    if (!aligned(out, 2))
        return fail(Q4MOE_ERR_ALIGNMENT, "out must be 2-byte aligned");
    q4moe_options_t o{};
    if (opts != nullptr)
        o = *opts;
    if ((rc = check_kernel_options(o, true)))
        return rc;
    if (o.kernel != Q4MOE_KERNEL_AUTO || o.matvec_tile != 0 ||
        o.workspace != nullptr || o.workspace_bytes != 0)
        return fail(Q4MOE_ERR_INVALID_ARG,
                    "trellis calls take no kernel choice, tile or workspace");
    DeviceInfo *d = nullptr;
    rc = device_info(&d);
    if (rc)
        return rc;
    if (M == 0)
        return ok();
    q4moe::GateUpArgs a{};
    a.x = static_cast<const uint16_t *>(x);
    a.base = static_cast<const uint8_t *>(slabs->base);
    a.stride = slabs->slab_stride;
    a.slab_ptrs = reinterpret_cast<const uint8_t *const *>(slabs->slab_ptrs);
    a.gate_w_off = L.gate_codes_offset;
    a.up_w_off = L.up_codes_offset;
    a.gate_s_off = L.gate_scales_offset;
    a.up_s_off = L.up_scales_offset;
    a.row_offsets = row_offsets;
    a.token_of_row = token_of_row;
    a.M = M;
    a.H = H;
    a.I = I;
    a.T = o.num_tokens;
    a.E = slabs->num_experts;
    a.out = static_cast<uint16_t *>(out);
    a.gate_f32 = o.gate_f32;
    a.up_f32 = o.up_f32;
    a.status = d->status;
    a.num_sms = d->num_sms;
    a.sigmoid = d->sigmoid;
    a.tr_block = L.block_size;
    a.tr_window = L.window_bits;
    a.tr_kg = L.gate_bits;
    a.tr_ku = L.up_bits;
    // the pages' tail unless one is asked for: MLX's when the widths differ
    // (the mixed-width kernel), page 52's otherwise
    a.tail_mlx = o.tail == Q4MOE_TAIL_MLX ||
                 (o.tail == Q4MOE_TAIL_AUTO && L.gate_bits != L.up_bits);
    a.matvec_max_rows = INT32_MAX;
    const cudaError_t err = q4moe::launch_trellis_gate_up(a, stream);
    if (err != cudaSuccess)
        return cuda_fail(err, "trellis launch");
    return ok();
}

int q4moe_group_rows(const int32_t *topk_ids, int64_t T, int32_t k,
                     int32_t E, int32_t *row_offsets, int32_t *token_of_row,
                     int32_t *row_of_pair, cudaStream_t stream) {
    if (T < 0 || k <= 0 || E <= 0 || E > Q4MOE_MAX_EXPERTS)
        return fail(Q4MOE_ERR_INVALID_ARG,
                    "need T >= 0, k >= 1, 1 <= E <= %d", Q4MOE_MAX_EXPERTS);
    if (T > (int64_t)(INT32_MAX - 1024) / k)
        return fail(Q4MOE_ERR_INVALID_ARG, "T*k must stay below 2^31");
    if (row_offsets == nullptr || (T > 0 && (!topk_ids || !token_of_row ||
                                             !row_of_pair)))
        return fail(Q4MOE_ERR_INVALID_ARG, "null pointer");
    DeviceInfo *d = nullptr;
    int rc = device_info(&d);
    if (rc)
        return rc;
    cudaError_t err =
        q4moe::launch_group_rows(topk_ids, T * k, k, E, row_offsets,
                                 token_of_row, row_of_pair, d->status,
                                 d->num_sms, stream);
    if (err != cudaSuccess)
        return cuda_fail(err, "group_rows launch");
    return ok();
}

int q4moe_gate_up_swiglu_ex(const void *x, const q4moe_slabs_t *slabs,
                            const int32_t *row_offsets,
                            const int32_t *token_of_row, int64_t M, int64_t H,
                            int64_t I, void *out, const q4moe_options_t *opts,
                            cudaStream_t stream) {
    int rc = check_slabs(slabs, H, I, M);
    if (rc)
        return rc;
    if (row_offsets == nullptr)
        return fail(Q4MOE_ERR_INVALID_ARG, "row_offsets_per_expert is null");
    if (M > 0 && (x == nullptr || token_of_row == nullptr || out == nullptr))
        return fail(Q4MOE_ERR_INVALID_ARG, "null pointer");
    if (!aligned(x, 16))
        return fail(Q4MOE_ERR_ALIGNMENT, "x must be 16-byte aligned");
    if (!aligned(out, 2))
        return fail(Q4MOE_ERR_ALIGNMENT, "out must be 2-byte aligned");
    q4moe_options_t o{};
    if (opts != nullptr)
        o = *opts;
    if ((rc = check_kernel_options(o)))
        return rc;
    if (o.workspace != nullptr) {
        if (!aligned(o.workspace, 256))
            return fail(Q4MOE_ERR_ALIGNMENT,
                        "workspace must be 256-byte aligned");
        if (o.workspace_bytes < q4moe_workspace_bytes(M, H))
            return fail(Q4MOE_ERR_INVALID_ARG,
                        "workspace of %lld bytes is smaller than the %lld "
                        "this call needs", (long long)o.workspace_bytes,
                        (long long)q4moe_workspace_bytes(M, H));
    }

    DeviceInfo *d = nullptr;
    rc = device_info(&d);
    if (rc)
        return rc;
    if (M == 0)
        return ok();

    q4moe::GateUpArgs a = base_args(slabs, M, d, o);
    const q4moe_layout_t &L = slabs->layout;
    a.x = static_cast<const uint16_t *>(x);
    a.gate_w_off = L.gate_w_offset;
    a.up_w_off = L.up_w_offset;
    a.gate_s_off = L.gate_s_offset;
    a.up_s_off = L.up_s_offset;
    a.row_offsets = row_offsets;
    a.token_of_row = token_of_row;
    a.H = H;
    a.I = I;
    a.T = o.num_tokens;
    a.out = static_cast<uint16_t *>(out);
    a.gate_f32 = o.gate_f32;
    a.up_f32 = o.up_f32;
    a.xg = static_cast<uint16_t *>(o.workspace);
    return dispatch(a, o, d, stream);
}

namespace {

// The down projection; hold_next keeps the single-expert latency kernel
// from releasing the next launch early.  Measured on the single-expert
// decode (H=4096, I=1536, one row, graphs of 1000 calls): released early,
// a chain of down projections takes 3.59 us per call instead of 4.25, but
// an expert MLP (gate/up, then down, then the next gate/up) 10.24 instead
// of 9.24 us, the gate/up that follows losing more than the down gains.
int down_proj(const void *mid, const q4moe_slabs_t *slabs,
              const int32_t *row_offsets, int64_t M, int64_t H, int64_t I,
              void *out, const q4moe_options_t *opts, cudaStream_t stream,
              bool hold_next) {
    int rc = check_slabs(slabs, H, I, M);
    if (rc)
        return rc;
    q4moe_options_t o{};
    if (opts != nullptr)
        o = *opts;
    if ((rc = check_kernel_options(o)) ||
        (rc = check_down(slabs, mid, out, row_offsets, M, o, true)))
        return rc;
    DeviceInfo *d = nullptr;
    rc = device_info(&d);
    if (rc)
        return rc;
    if (M == 0)
        return ok();
    q4moe::GateUpArgs a = base_args(slabs, M, d, o);
    const q4moe_layout_t &L = slabs->layout;
    a.down = 1;
    a.x = static_cast<const uint16_t *>(mid);
    a.gate_w_off = a.up_w_off = L.down_w_offset;
    a.gate_s_off = a.up_s_off = L.down_s_offset;
    a.row_offsets = row_offsets;
    a.token_of_row = nullptr;
    a.H = I;                                 // the projection's K
    a.I = H;                                 // its output rows
    a.out = static_cast<uint16_t *>(out);
    a.gate_f32 = o.gate_f32;
    a.hold_next = hold_next;
    return dispatch(a, o, d, stream);
}

}  // namespace

int q4moe_down_proj(const void *mid, const q4moe_slabs_t *slabs,
                    const int32_t *row_offsets, int64_t M, int64_t H,
                    int64_t I, void *out, const q4moe_options_t *opts,
                    cudaStream_t stream) {
    return down_proj(mid, slabs, row_offsets, M, H, I, out, opts, stream,
                     false);
}

int q4moe_expert_mlp(const void *x, const q4moe_slabs_t *slabs,
                     const int32_t *row_offsets, const int32_t *token_of_row,
                     int64_t M, int64_t H, int64_t I, void *mid, void *out,
                     const q4moe_options_t *opts, cudaStream_t stream) {
    // every check of both stages before the first launch
    int rc = check_slabs(slabs, H, I, M);
    if (rc)
        return rc;
    q4moe_options_t o{};
    if (opts != nullptr)
        o = *opts;
    if ((rc = check_down(slabs, mid, out, row_offsets, M, o, false)))
        return rc;
    if (overlap(mid, M * I * 2, out, M * H * 2) ||
        overlap(mid, M * I * 2, x, M > 0 ? 1 : 0))
        return fail(Q4MOE_ERR_INVALID_ARG, "mid overlaps x or out");
    if ((rc = q4moe_gate_up_swiglu_ex(x, slabs, row_offsets, token_of_row, M,
                                      H, I, mid, &o, stream)))
        return rc;
    q4moe_options_t od{};
    od.kernel = o.kernel;
    od.matvec_tile = o.matvec_tile;
    return down_proj(mid, slabs, row_offsets, M, H, I, out, &od, stream,
                     true);
}

int q4moe_gate_up_swiglu(const void *x, const q4moe_slabs_t *slabs,
                         const int32_t *row_offsets,
                         const int32_t *token_of_row, int64_t M, int64_t H,
                         int64_t I, void *out, cudaStream_t stream) {
    return q4moe_gate_up_swiglu_ex(x, slabs, row_offsets, token_of_row, M, H,
                                   I, out, nullptr, stream);
}

int q4moe_device_status(cudaStream_t stream, uint32_t *flags, int clear) {
    if (flags == nullptr)
        return fail(Q4MOE_ERR_INVALID_ARG, "flags is null");
    DeviceInfo *d = nullptr;
    int rc = device_info(&d);
    if (rc)
        return rc;
    cudaError_t err = cudaStreamSynchronize(stream);
    if (err != cudaSuccess)
        return cuda_fail(err, "cudaStreamSynchronize");
    unsigned int v = 0;
    err = cudaMemcpy(&v, d->status, sizeof v, cudaMemcpyDeviceToHost);
    if (err != cudaSuccess)
        return cuda_fail(err, "reading the status word");
    if (clear) {
        const unsigned int zero = 0;
        err = cudaMemcpy(d->status, &zero, sizeof zero,
                         cudaMemcpyHostToDevice);
        if (err != cudaSuccess)
            return cuda_fail(err, "clearing the status word");
    }
    *flags = v;
    if (v != 0)
        return fail(Q4MOE_ERR_DEVICE_DATA, "device status 0x%x", v);
    return ok();
}

int q4moe_debug_tail(const uint16_t *gate_bf16, const uint16_t *up_bf16,
                     int64_t n, uint16_t *res, cudaStream_t stream) {
    if (n < 0 || (n > 0 && (!gate_bf16 || !up_bf16 || !res)))
        return fail(Q4MOE_ERR_INVALID_ARG, "bad arguments");
    DeviceInfo *d = nullptr;
    int rc = device_info(&d);
    if (rc)
        return rc;
    cudaError_t err = q4moe::launch_debug_tail(gate_bf16, up_bf16, n, res,
                                               d->sigmoid, false, stream);
    if (err != cudaSuccess)
        return cuda_fail(err, "debug tail launch");
    return ok();
}

int q4moe_debug_wait_timeout(int64_t limit_ns, cudaStream_t stream) {
    if (limit_ns < 1000 || limit_ns > 1000000000)
        return fail(Q4MOE_ERR_INVALID_ARG,
                    "limit_ns must be in 1e3 .. 1e9 (1 us .. 1 s)");
    DeviceInfo *d = nullptr;
    int rc = device_info(&d);
    if (rc)
        return rc;
    cudaError_t err =
        q4moe::launch_debug_wait(d->status, (uint64_t)limit_ns, stream);
    if (err != cudaSuccess)
        return cuda_fail(err, "debug wait launch");
    return ok();
}

int q4moe_debug_tail_mlx(const uint16_t *gate_bf16, const uint16_t *up_bf16,
                         int64_t n, uint16_t *res, cudaStream_t stream) {
    if (n < 0 || (n > 0 && (!gate_bf16 || !up_bf16 || !res)))
        return fail(Q4MOE_ERR_INVALID_ARG, "bad arguments");
    DeviceInfo *d = nullptr;
    int rc = device_info(&d);
    if (rc)
        return rc;
    cudaError_t err = q4moe::launch_debug_tail(gate_bf16, up_bf16, n, res,
                                               d->sigmoid, true, stream);
    if (err != cudaSuccess)
        return cuda_fail(err, "debug tail launch");
    return ok();
}

}  // extern "C"
