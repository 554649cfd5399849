// kda_api.cu -- the C ABI of libkda.so (declared in include/kda.h):
// argument validation, workspace sizing and launch sequencing on the
// caller's stream.  Nothing here allocates device memory or synchronises.
#include <cstdarg>
#include <cstdio>
#include <cstring>
#include <mutex>
#include <string>

#include "kda_internal.cuh"
#include "kda_tc.cuh"

namespace {

thread_local std::string g_last_error;

kda_status fail(kda_status code, const char* fmt, ...) {
    char buf[512];
    va_list ap;
    va_start(ap, fmt);
    vsnprintf(buf, sizeof(buf), fmt, ap);
    va_end(ap);
    g_last_error = buf;
    return code;
}

kda_status cuda_fail(cudaError_t e, const char* where) {
    return fail(KDA_ERR_CUDA, "%s: %s", where, cudaGetErrorString(e));
}

kda_status ok() {
    g_last_error.clear();
    return KDA_OK;
}

bool supported_d(int D) { return D == 16 || D == 32 || D == 64 || D == 128; }
bool valid_dtype(int dt) { return dt == KDA_BF16 || dt == KDA_FP32; }
size_t dsize(kda_dtype dt) { return dt == KDA_BF16 ? 2 : 4; }
bool aligned(const void* p, size_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }
size_t round_up(size_t x, size_t a) { return (x + a - 1) / a * a; }

bool overlap(const void* a, size_t na, const void* b, size_t nb) {
    if (!a || !b || na == 0 || nb == 0) return false;
    const uintptr_t x = reinterpret_cast<uintptr_t>(a), y = reinterpret_cast<uintptr_t>(b);
    return x < y + nb && y < x + na;
}

// Validates a host copy of cu_seqlens: cu[0] = 0, non-decreasing, cu[N] = T_total.
kda_status check_host_cu(const int32_t* cu, int N, int64_t T_total) {
    if (cu[0] != 0) return fail(KDA_ERR_INVALID_ARG, "cu_seqlens[0] = %d, expected 0", cu[0]);
    for (int n = 0; n < N; ++n)
        if (cu[n + 1] < cu[n])
            return fail(KDA_ERR_INVALID_ARG, "cu_seqlens decreases at %d (%d -> %d)", n, cu[n],
                        cu[n + 1]);
    if ((int64_t)cu[N] != T_total)
        return fail(KDA_ERR_INVALID_ARG, "cu_seqlens[N] = %d but T_total = %lld", cu[N],
                    (long long)T_total);
    return KDA_OK;
}

// Row stride and alignment rules for 16-byte vector access of token rows.
kda_status check_rows(const void* p, int64_t stride, int64_t min_stride, kda_dtype dt,
                      const char* name) {
    if (stride < min_stride)
        return fail(KDA_ERR_INVALID_ARG, "%s row stride %lld < %lld", name, (long long)stride,
                    (long long)min_stride);
    const int64_t vec = dt == KDA_BF16 ? 8 : 4;
    if (stride % vec)
        return fail(KDA_ERR_INVALID_ARG, "%s row stride %lld is not a multiple of %lld elements",
                    name, (long long)stride, (long long)vec);
    if (!aligned(p, 16)) return fail(KDA_ERR_INVALID_ARG, "%s is not 16-byte aligned", name);
    return KDA_OK;
}

struct PrefillPlan {
    int path;           // KDA_PATH_*
    bool tc;            // tensor-core path
    size_t ws_conv;     // bytes: convolved q|k|v rows, fp32 (SIMT path)
    size_t ws_o;        // bytes: o before the epilogue, fp32 (SIMT path)
    size_t ws_tc;       // bytes: tensor-core path scratch
    size_t total;
};

PrefillPlan plan_prefill(const kda_prefill_args& a) {
    PrefillPlan p{};
    const bool simt = (a.flags & KDA_FLAG_FORCE_SIMT) != 0;
    if (!simt && !(a.flags & KDA_FLAG_NO_RECURRENT) && kda::short_prefill_applies(a)) {
        p.path = KDA_PATH_RECURRENT;
        return p;
    }
    p.tc = !simt && kda::tc_prefill_applies(a);
    p.path = p.tc ? KDA_PATH_TENSOR_CORE : KDA_PATH_SIMT;
    const size_t T = (size_t)(a.T_total > 0 ? a.T_total : 0);
    const size_t HD = (size_t)a.H * a.D;
    if (p.tc) {
        p.ws_tc = round_up(kda::tc_prefill_workspace(a), 256);
    } else {
        p.ws_conv = round_up(T * 3 * HD * sizeof(float), 256);
        p.ws_o = round_up(T * HD * sizeof(float), 256);
    }
    p.total = p.ws_conv + p.ws_o + p.ws_tc;
    return p;
}

kda_status validate_prefill(const kda_prefill_args* a) {
    if (!a) return fail(KDA_ERR_INVALID_ARG, "args is NULL");
    if (a->N < 0 || a->H < 1 || a->T_total < 0)
        return fail(KDA_ERR_INVALID_ARG, "bad sizes N=%d H=%d T_total=%lld", a->N, a->H,
                    (long long)a->T_total);
    if (!supported_d(a->D)) return fail(KDA_ERR_UNSUPPORTED, "head width D=%d not in {16,32,64,128}", a->D);
    if (!kda::chunk_simt_supported(a->D, a->chunk))
        return fail(KDA_ERR_UNSUPPORTED, "chunk=%d not in {16,32,64}", a->chunk);
    if (!valid_dtype(a->io) || !valid_dtype(a->out_dtype))
        return fail(KDA_ERR_INVALID_ARG, "unknown dtype (io=%d out=%d)", (int)a->io, (int)a->out_dtype);
    if ((int64_t)a->H * a->D * 3 > (int64_t)1 << 30)
        return fail(KDA_ERR_UNSUPPORTED, "H*D too large");
    if (a->segments < 0 || a->segments > KDA_MAX_SEGMENTS)
        return fail(KDA_ERR_INVALID_ARG, "segments = %d not in [0, %d]", a->segments, KDA_MAX_SEGMENTS);
    if (a->N > 0 && !a->cu_seqlens) return fail(KDA_ERR_INVALID_ARG, "cu_seqlens is NULL");
    if (a->cu_seqlens_host) {
        kda_status st = check_host_cu(a->cu_seqlens_host, a->N, a->T_total);
        if (st) return st;
    } else if (a->N == 0 && a->T_total != 0) {
        return fail(KDA_ERR_INVALID_ARG, "N = 0 but T_total = %lld", (long long)a->T_total);
    }
    if (a->N == 0) return KDA_OK;
    if (!a->conv_w) return fail(KDA_ERR_INVALID_ARG, "conv_w is NULL");
    const int64_t HD = (int64_t)a->H * a->D;
    const size_t T = (size_t)a->T_total;
    if (a->T_total > 0) {
        if (!a->q || !a->k || !a->v || !a->g || !a->beta || !a->out)
            return fail(KDA_ERR_INVALID_ARG, "q, k, v, g, beta and out must be non-NULL");
        const int64_t xs = a->qkv_row_stride ? a->qkv_row_stride : HD;
        kda_status st;
        if ((st = check_rows(a->q, xs, HD, a->io, "q")) || (st = check_rows(a->k, xs, HD, a->io, "k")) ||
            (st = check_rows(a->v, xs, HD, a->io, "v")))
            return st;
        if (!aligned(a->g, 16) || !aligned(a->beta, 4) || !aligned(a->out, 16) ||
            (a->gate && !aligned(a->gate, 16)))
            return fail(KDA_ERR_INVALID_ARG, "g/out/gate must be 16-byte aligned, beta 4-byte");
        const size_t ob = T * HD * dsize(a->out_dtype);
        const size_t xb = (T - 1) * (size_t)xs * dsize(a->io) + HD * dsize(a->io);
        if (overlap(a->out, ob, a->q, xb) || overlap(a->out, ob, a->k, xb) ||
            overlap(a->out, ob, a->v, xb) || overlap(a->out, ob, a->g, T * HD * 4) ||
            overlap(a->out, ob, a->gate, a->gate ? T * HD * dsize(a->io) : 0))
            return fail(KDA_ERR_INVALID_ARG, "out overlaps an input");
    }
    const size_t sb = (size_t)a->N * HD * a->D * sizeof(float);
    if ((a->initial_state && !aligned(a->initial_state, 16)) ||
        (a->final_state && !aligned(a->final_state, 16)))
        return fail(KDA_ERR_INVALID_ARG, "initial_state/final_state must be 16-byte aligned");
    if (a->initial_state && a->final_state && a->initial_state != a->final_state &&
        overlap(a->initial_state, sb, a->final_state, sb))
        return fail(KDA_ERR_INVALID_ARG, "final_state partially overlaps initial_state");
    const size_t cb = (size_t)a->N * 3 * HD * 3 * dsize(a->io);
    if (overlap(a->conv_state_in, cb, a->conv_state_out, cb))
        return fail(KDA_ERR_INVALID_ARG, "conv_state_out overlaps conv_state_in");
    const PrefillPlan p = plan_prefill(*a);
    if (p.total > 0) {
        if (!a->workspace) return fail(KDA_ERR_WORKSPACE, "workspace is NULL (%zu bytes needed)", p.total);
        if (a->workspace_bytes < p.total)
            return fail(KDA_ERR_WORKSPACE, "workspace has %zu bytes, %zu needed", a->workspace_bytes, p.total);
        if (!aligned(a->workspace, 256)) return fail(KDA_ERR_WORKSPACE, "workspace is not 256-byte aligned");
    }
    return KDA_OK;
}

// Fixed scratch of kda_prefill_noalloc (see include/kda.h).  In host code
// this name is only a host-side stand-in: its device address comes from
// cudaGetSymbolAddress with the device current.
static __device__ __align__(256) unsigned char g_noalloc_scratch[KDA_NOALLOC_SCRATCH_BYTES];

// Device address of the fixed scratch on the current device.  Looked up on every call (a
// host-side lookup, no allocation), so the address is never stale: after cudaDeviceReset, or
// under another context on the same device, the lookup returns that context's copy.  The
// first lookup in a context also loads the library's device code there, which is why the
// first call on each device should come before any stream capture.
kda_status noalloc_scratch(void** out) {
    void* p = nullptr;
    const cudaError_t e = cudaGetSymbolAddress(&p, g_noalloc_scratch);
    if (e != cudaSuccess) return cuda_fail(e, "cudaGetSymbolAddress(fixed scratch)");
    if (!p) return fail(KDA_ERR_CUDA, "fixed scratch has no device address");
    *out = p;
    return KDA_OK;
}

std::once_flag g_dev_once[kda::kMaxDevices];
kda::DeviceInfo g_dev_info[kda::kMaxDevices];

}  // namespace

bool kda::current_device_info(kda::DeviceInfo* out) {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kda::kMaxDevices) return false;
    std::call_once(g_dev_once[dev], [dev] {
        kda::DeviceInfo d{0, 0, 0};
        cudaDeviceGetAttribute(&d.sm_count, cudaDevAttrMultiProcessorCount, dev);
        cudaDeviceGetAttribute(&d.cc_major, cudaDevAttrComputeCapabilityMajor, dev);
        cudaDeviceGetAttribute(&d.cc_minor, cudaDevAttrComputeCapabilityMinor, dev);
        g_dev_info[dev] = d;
    });
    *out = g_dev_info[dev];
    return out->sm_count > 0;
}

extern "C" {

const char* kda_status_string(int status) {
    switch (status) {
        case KDA_OK: return "ok";
        case KDA_ERR_INVALID_ARG: return "invalid argument";
        case KDA_ERR_UNSUPPORTED: return "unsupported shape or dtype";
        case KDA_ERR_WORKSPACE: return "workspace missing or too small";
        case KDA_ERR_CUDA: return "CUDA error";
        case KDA_ERR_TIMEOUT: return "device-side wait timed out";
        case KDA_ERR_DEVICE_ARG: return "inconsistent cu_seqlens on the device";
        default: return "unknown status";
    }
}

const char* kda_last_error(void) { return g_last_error.c_str(); }

int kda_version(void) { return 1 * 10000 + 4 * 100 + 1; }

kda_status kda_short_conv(const void* x, int64_t x_row_stride, const float* w,
                          const int32_t* cu_seqlens, const int32_t* cu_seqlens_host, int N,
                          int64_t T_total, int H, int D, const void* conv_state_in,
                          void* conv_state_out, void* y, int64_t y_row_stride, int l2norm_qk,
                          float eps_l2, kda_dtype io, int* d_status, kda_stream_t stream) {
    if (N < 0 || H < 1 || T_total < 0) return fail(KDA_ERR_INVALID_ARG, "bad sizes");
    if (!supported_d(D)) return fail(KDA_ERR_UNSUPPORTED, "head width D=%d not in {16,32,64,128}", D);
    if (!valid_dtype(io)) return fail(KDA_ERR_INVALID_ARG, "unknown dtype %d", (int)io);
    if (N > 0 && !cu_seqlens) return fail(KDA_ERR_INVALID_ARG, "cu_seqlens is NULL");
    if (cu_seqlens_host) {
        kda_status st = check_host_cu(cu_seqlens_host, N, T_total);
        if (st) return st;
    }
    if (N == 0) {
        if (T_total != 0) return fail(KDA_ERR_INVALID_ARG, "N = 0 but T_total != 0");
        return ok();
    }
    if (!w) return fail(KDA_ERR_INVALID_ARG, "w is NULL");
    const int64_t C3 = 3 * (int64_t)H * D;
    if (T_total > 0) {
        if (!x || !y) return fail(KDA_ERR_INVALID_ARG, "x and y must be non-NULL");
        kda_status st;
        if ((st = check_rows(x, x_row_stride, C3, io, "x")) || (st = check_rows(y, y_row_stride, C3, io, "y")))
            return st;
        const size_t xb = (size_t)((T_total - 1) * x_row_stride + C3) * dsize(io);
        const size_t yb = (size_t)((T_total - 1) * y_row_stride + C3) * dsize(io);
        if (overlap(x, xb, y, yb)) return fail(KDA_ERR_INVALID_ARG, "y overlaps x");
    }
    const size_t cb = (size_t)N * C3 * 3 * dsize(io);
    if (overlap(conv_state_in, cb, conv_state_out, cb))
        return fail(KDA_ERR_INVALID_ARG, "conv_state_out overlaps conv_state_in");
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    cudaError_t e;
    if (!cu_seqlens_host && (e = kda::launch_check_cu(cu_seqlens, N, T_total, d_status, s)))
        return cuda_fail(e, "check cu_seqlens");
    const int64_t HD = (int64_t)H * D;
    const kda::QKVParts parts{{x, static_cast<const char*>(x) + HD * dsize(io),
                               static_cast<const char*>(x) + 2 * HD * dsize(io)}};
    if ((e = kda::launch_short_conv(parts, x_row_stride, io, w, cu_seqlens, N, T_total, H, D,
                                    conv_state_in, y, y_row_stride, io, l2norm_qk, eps_l2, s)))
        return cuda_fail(e, "short conv");
    if (conv_state_out &&
        (e = kda::launch_conv_state_out(parts, x_row_stride, io, cu_seqlens, N, T_total, (int)C3,
                                        conv_state_in, conv_state_out, s)))
        return cuda_fail(e, "conv state");
    return ok();
}

kda_status kda_prefill_workspace_size(const kda_prefill_args* args, size_t* bytes) {
    if (!bytes) return fail(KDA_ERR_INVALID_ARG, "bytes is NULL");
    *bytes = 0;
    if (!args) return fail(KDA_ERR_INVALID_ARG, "args is NULL");
    if (!supported_d(args->D) || !kda::chunk_simt_supported(args->D, args->chunk))
        return fail(KDA_ERR_UNSUPPORTED, "unsupported D=%d / chunk=%d", args->D, args->chunk);
    if (args->T_total < 0 || args->H < 1 || args->N < 0) return fail(KDA_ERR_INVALID_ARG, "bad sizes");
    if (args->segments < 0 || args->segments > KDA_MAX_SEGMENTS)
        return fail(KDA_ERR_INVALID_ARG, "segments = %d not in [0, %d]", args->segments, KDA_MAX_SEGMENTS);
    *bytes = plan_prefill(*args).total;
    return ok();
}

kda_status kda_prefill_plan(const kda_prefill_args* args, int* path, int* segments) {
    if (!args || !path || !segments) return fail(KDA_ERR_INVALID_ARG, "NULL argument");
    *path = KDA_PATH_SIMT;
    *segments = 1;
    if (!supported_d(args->D) || !kda::chunk_simt_supported(args->D, args->chunk))
        return fail(KDA_ERR_UNSUPPORTED, "unsupported D=%d / chunk=%d", args->D, args->chunk);
    if (args->T_total < 0 || args->H < 1 || args->N < 0) return fail(KDA_ERR_INVALID_ARG, "bad sizes");
    if (args->segments < 0 || args->segments > KDA_MAX_SEGMENTS)
        return fail(KDA_ERR_INVALID_ARG, "segments = %d not in [0, %d]", args->segments, KDA_MAX_SEGMENTS);
    if (args->cu_seqlens_host && args->N > 0) {
        kda_status st = check_host_cu(args->cu_seqlens_host, args->N, args->T_total);
        if (st) return st;
    }
    const PrefillPlan p = plan_prefill(*args);
    *path = p.path;
    *segments = p.tc ? kda::tc_segments(*args) : 1;
    return ok();
}

kda_status kda_prefill(const kda_prefill_args* a, kda_stream_t stream) {
    kda_status st = validate_prefill(a);
    if (st) return st;
    if (a->N == 0) return ok();
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    const PrefillPlan p = plan_prefill(*a);
    const int64_t HD = (int64_t)a->H * a->D;
    const int64_t xs = a->qkv_row_stride ? a->qkv_row_stride : HD;
    const kda::QKVParts parts{{a->q, a->k, a->v}};
    cudaError_t e;
    if (!a->cu_seqlens_host &&
        (e = kda::launch_check_cu(a->cu_seqlens, a->N, a->T_total, a->d_status, s)))
        return cuda_fail(e, "check cu_seqlens");
    // the pipelined recurrent kernel rolls the conv state itself
    const bool short_tma = p.path == KDA_PATH_RECURRENT && kda::short_tma_applies(*a);
    if (a->conv_state_out && !short_tma &&
        (e = kda::launch_conv_state_out(parts, xs, a->io, a->cu_seqlens, a->N, a->T_total,
                                        (int)(3 * HD), a->conv_state_in, a->conv_state_out, s)))
        return cuda_fail(e, "conv state");
    if (p.path == KDA_PATH_RECURRENT) {
        if ((e = short_tma ? kda::launch_short_tma(*a, s) : kda::launch_short_prefill(*a, s)))
            return cuda_fail(e, "recurrent prefill");
        return ok();
    }
    if (p.tc) {
        if ((e = kda::launch_tc_prefill(*a, static_cast<char*>(a->workspace), s)))
            return cuda_fail(e, "tensor-core prefill");
        return ok();
    }
    float* ws_y = static_cast<float*>(a->workspace);
    float* ws_o = reinterpret_cast<float*>(static_cast<char*>(a->workspace) + p.ws_conv);
    if ((e = kda::launch_short_conv(parts, xs, a->io, a->conv_w, a->cu_seqlens, a->N, a->T_total,
                                    a->H, a->D, a->conv_state_in, ws_y, 3 * HD, KDA_FP32, 1,
                                    a->eps_l2, s)))
        return cuda_fail(e, "short conv");
    if ((e = kda::launch_chunk_simt(ws_y, a->g, a->beta, a->cu_seqlens, a->N, a->T_total, a->H,
                                    a->D, a->chunk, a->scale, a->initial_state, a->final_state,
                                    ws_o, s)))
        return cuda_fail(e, "chunk recurrence");
    if ((e = kda::launch_rms_gate(ws_o, a->T_total * a->H, a->D, a->gate, a->io, a->rms_w,
                                  a->eps_rms, a->out, a->out_dtype, s)))
        return cuda_fail(e, "epilogue");
    return ok();
}

kda_status kda_prefill_noalloc(const kda_prefill_args* args, kda_stream_t stream) {
    if (!args) return fail(KDA_ERR_INVALID_ARG, "args is NULL");
    kda_prefill_args a = *args;
    a.flags |= KDA_FLAG_FORCE_SIMT;  // the SIMT path is the one that stages data in scratch
    a.workspace = nullptr;
    a.workspace_bytes = 0;
    if (!supported_d(a.D) || !kda::chunk_simt_supported(a.D, a.chunk))
        return fail(KDA_ERR_UNSUPPORTED, "unsupported D=%d / chunk=%d", a.D, a.chunk);
    if (a.T_total < 0 || a.H < 1 || a.N < 0) return fail(KDA_ERR_INVALID_ARG, "bad sizes");
    const size_t need = plan_prefill(a).total;
    if (need > KDA_NOALLOC_SCRATCH_BYTES)
        return fail(KDA_ERR_WORKSPACE,
                    "kda_prefill_noalloc needs %zu bytes of scratch for T_total=%lld, H=%d, D=%d; "
                    "its fixed scratch holds %zu bytes (use kda_prefill with a workspace)",
                    need, (long long)a.T_total, a.H, a.D, (size_t)KDA_NOALLOC_SCRATCH_BYTES);
    if (need > 0) {
        void* p = nullptr;
        kda_status st = noalloc_scratch(&p);
        if (st) return st;
        a.workspace = p;
        a.workspace_bytes = KDA_NOALLOC_SCRATCH_BYTES;
    }
    return kda_prefill(&a, stream);
}

kda_status kda_gemm(const kda_gemm_args* g, kda_stream_t stream) {
    if (!g) return fail(KDA_ERR_INVALID_ARG, "args is NULL");
    if (g->M < 0 || g->N < 0 || g->K <= 0)
        return fail(KDA_ERR_INVALID_ARG, "bad sizes M=%d N=%d K=%d", g->M, g->N, g->K);
    if (g->K % 64) return fail(KDA_ERR_UNSUPPORTED, "K=%d is not a multiple of 64", g->K);
    if (!valid_dtype(g->c_dtype)) return fail(KDA_ERR_INVALID_ARG, "unknown dtype %d", (int)g->c_dtype);
    if (g->epilogue < KDA_EPI_NONE || g->epilogue > KDA_EPI_SIGMOID)
        return fail(KDA_ERR_INVALID_ARG, "unknown epilogue %d", g->epilogue);
    if (g->M == 0 || g->N == 0) return ok();
    if (!g->A || !g->W || !g->C) return fail(KDA_ERR_INVALID_ARG, "A, W and C must be non-NULL");
    if (g->lda < g->K || g->ldw < g->K || g->ldc < g->N)
        return fail(KDA_ERR_INVALID_ARG, "leading dimensions too small (lda=%lld ldw=%lld ldc=%lld)",
                    (long long)g->lda, (long long)g->ldw, (long long)g->ldc);
    if ((g->lda * 2) % 16 || (g->ldw * 2) % 16)
        return fail(KDA_ERR_INVALID_ARG, "lda and ldw must be multiples of 8 elements");
    if (!aligned(g->A, 16) || !aligned(g->W, 16) || !aligned(g->C, 16))
        return fail(KDA_ERR_INVALID_ARG, "A, W and C must be 16-byte aligned");
    const size_t ab = ((size_t)(g->M - 1) * g->lda + g->K) * 2, wb = ((size_t)(g->N - 1) * g->ldw + g->K) * 2;
    const size_t cb = ((size_t)(g->M - 1) * g->ldc + g->N) * dsize(g->c_dtype);
    if (overlap(g->C, cb, g->A, ab) || overlap(g->C, cb, g->W, wb))
        return fail(KDA_ERR_INVALID_ARG, "C overlaps A or W");
    if (!kda::gemm_supported_device()) return fail(KDA_ERR_UNSUPPORTED, "kda_gemm needs an sm_103 device");
    const cudaError_t e = kda::launch_gemm(*g, reinterpret_cast<cudaStream_t>(stream));
    if (e) return cuda_fail(e, "gemm");
    return ok();
}

// Validation of kda_backward (include/kda.h): sizes, dtypes, the host copy of cu_seqlens, every
// required pointer, alignment, and that no output overlaps another output or an input.
kda_status validate_backward(const kda_backward_args* b, kda::BackwardLayout* L) {
    if (!b) return fail(KDA_ERR_INVALID_ARG, "args is NULL");
    const kda_prefill_args& a = b->fwd;
    if (a.N < 0 || a.H < 1 || a.T_total < 0)
        return fail(KDA_ERR_INVALID_ARG, "bad sizes N=%d H=%d T_total=%lld", a.N, a.H, (long long)a.T_total);
    if (a.D != 128) return fail(KDA_ERR_UNSUPPORTED, "kda_backward needs D = 128 (got %d)", a.D);
    if (!valid_dtype(a.io) || !valid_dtype(a.out_dtype))
        return fail(KDA_ERR_INVALID_ARG, "unknown dtype (io=%d out=%d)", (int)a.io, (int)a.out_dtype);
    if ((int64_t)a.H * a.D * 3 > (int64_t)1 << 30 || (int64_t)a.N * a.H > 0x7fffffffLL)
        return fail(KDA_ERR_UNSUPPORTED, "H*D or N*H too large");
    if (!a.cu_seqlens_host) return fail(KDA_ERR_INVALID_ARG, "kda_backward needs cu_seqlens_host");
    if (a.N > 0 && !a.cu_seqlens) return fail(KDA_ERR_INVALID_ARG, "cu_seqlens is NULL");
    if (kda_status st = check_host_cu(a.cu_seqlens_host, a.N, a.T_total)) return st;
    *L = kda::backward_layout(*b);
    if (a.N == 0) return KDA_OK;
    if (!a.conv_w || !b->dconv_w) return fail(KDA_ERR_INVALID_ARG, "conv_w and dconv_w must be non-NULL");
    const int64_t HD = (int64_t)a.H * a.D;
    const size_t T = (size_t)a.T_total;
    const int64_t xs = a.qkv_row_stride ? a.qkv_row_stride : HD;
    const size_t rowf = T * HD * 4, sb = (size_t)a.N * HD * a.D * 4, cwb = (size_t)3 * HD * 16;
    const size_t csb = (size_t)a.N * 3 * HD * 3;
    size_t xb = 0;
    if (a.T_total > 0) {
        if (!a.q || !a.k || !a.v || !a.g || !a.beta || !b->dy || !b->dq || !b->dk || !b->dv || !b->dg ||
            !b->dbeta)
            return fail(KDA_ERR_INVALID_ARG, "q, k, v, g, beta, dy, dq, dk, dv, dg and dbeta must be non-NULL");
        kda_status st;
        if ((st = check_rows(a.q, xs, HD, a.io, "q")) || (st = check_rows(a.k, xs, HD, a.io, "k")) ||
            (st = check_rows(a.v, xs, HD, a.io, "v")))
            return st;
        xb = (T - 1) * (size_t)xs * dsize(a.io) + HD * dsize(a.io);
    }
    const void* a16[] = {a.g, a.gate, a.conv_w, a.initial_state, b->dy, b->d_final_state, b->dq, b->dk, b->dv,
                         b->dconv_w, b->dg, b->dgate, b->dinitial_state};
    for (const void* p : a16)
        if (p && !aligned(p, 16))
            return fail(KDA_ERR_INVALID_ARG, "g, gate, conv_w, the states, dy and the tensor gradients must be "
                                             "16-byte aligned");
    const void* a4[] = {a.beta, a.rms_w, b->dbeta, b->drms_w, b->dconv_state_in};
    for (const void* p : a4)
        if (p && !aligned(p, 4)) return fail(KDA_ERR_INVALID_ARG, "beta, rms_w and their gradients must be 4-byte aligned");
    struct Buf {
        const void* p;
        size_t n;
    };
    const Buf outs[] = {{b->dq, rowf}, {b->dk, rowf}, {b->dv, rowf}, {b->dconv_w, cwb}, {b->dg, rowf},
                        {b->dbeta, T * a.H * 4}, {b->dgate, rowf}, {b->drms_w, (size_t)a.D * 4},
                        {b->dinitial_state, sb}, {b->dconv_state_in, csb * 4}};
    const Buf ins[] = {{a.q, xb}, {a.k, xb}, {a.v, xb}, {a.g, rowf}, {a.beta, T * a.H * 4},
                       {a.gate, a.gate ? T * HD * dsize(a.io) : 0}, {a.conv_w, cwb},
                       {a.conv_state_in, csb * dsize(a.io)}, {a.rms_w, (size_t)a.D * 4}, {a.initial_state, sb},
                       {b->dy, T * HD * dsize(a.out_dtype)}, {b->d_final_state, sb},
                       {a.workspace, L->total}};
    const int no = sizeof(outs) / sizeof(outs[0]);
    for (int i = 0; i < no; ++i) {
        for (int j = i + 1; j < no; ++j)
            if (overlap(outs[i].p, outs[i].n, outs[j].p, outs[j].n))
                return fail(KDA_ERR_INVALID_ARG, "gradient outputs %d and %d overlap", i, j);
        for (const Buf& in : ins)
            if (overlap(outs[i].p, outs[i].n, in.p, in.n))
                return fail(KDA_ERR_INVALID_ARG, "gradient output %d overlaps an input or the workspace", i);
    }
    if (L->total > 0) {
        if (!a.workspace) return fail(KDA_ERR_WORKSPACE, "workspace is NULL (%zu bytes needed)", L->total);
        if (a.workspace_bytes < L->total)
            return fail(KDA_ERR_WORKSPACE, "workspace has %zu bytes, %zu needed", a.workspace_bytes, L->total);
        if (!aligned(a.workspace, 256)) return fail(KDA_ERR_WORKSPACE, "workspace is not 256-byte aligned");
    }
    return KDA_OK;
}

kda_status kda_backward_workspace_size(const kda_backward_args* b, size_t* bytes) {
    if (!bytes) return fail(KDA_ERR_INVALID_ARG, "bytes is NULL");
    *bytes = 0;
    if (!b) return fail(KDA_ERR_INVALID_ARG, "args is NULL");
    const kda_prefill_args& a = b->fwd;
    if (a.D != 128) return fail(KDA_ERR_UNSUPPORTED, "kda_backward needs D = 128 (got %d)", a.D);
    if (a.T_total < 0 || a.H < 1 || a.N < 0) return fail(KDA_ERR_INVALID_ARG, "bad sizes");
    if (!a.cu_seqlens_host) return fail(KDA_ERR_INVALID_ARG, "kda_backward needs cu_seqlens_host");
    if (kda_status st = check_host_cu(a.cu_seqlens_host, a.N, a.T_total)) return st;
    *bytes = kda::backward_layout(*b).total;
    return ok();
}

kda_status kda_backward(const kda_backward_args* b, kda_stream_t stream) {
    kda::BackwardLayout L{};
    if (kda_status st = validate_backward(b, &L)) return st;
    if (b->fwd.N == 0) return ok();
    const cudaError_t e = kda::launch_backward(*b, L, static_cast<char*>(b->fwd.workspace),
                                               reinterpret_cast<cudaStream_t>(stream));
    if (e) return cuda_fail(e, "backward");
    return ok();
}

kda_status kda_decode_step(const kda_decode_args* a, kda_stream_t stream) {
    if (!a) return fail(KDA_ERR_INVALID_ARG, "args is NULL");
    if (a->N < 0 || a->H < 1) return fail(KDA_ERR_INVALID_ARG, "bad sizes N=%d H=%d", a->N, a->H);
    if (!supported_d(a->D)) return fail(KDA_ERR_UNSUPPORTED, "head width D=%d not in {16,32,64,128}", a->D);
    if (!valid_dtype(a->io) || !valid_dtype(a->out_dtype)) return fail(KDA_ERR_INVALID_ARG, "unknown dtype");
    if ((int64_t)a->N * a->H > 0x7fffffffLL) return fail(KDA_ERR_UNSUPPORTED, "N*H too large");
    if (a->N == 0) return ok();
    if (!a->q || !a->k || !a->v || !a->g || !a->beta || !a->conv_w || !a->state || !a->conv_state || !a->out)
        return fail(KDA_ERR_INVALID_ARG, "q, k, v, g, beta, conv_w, state, conv_state and out must be non-NULL");
    const int64_t HD = (int64_t)a->H * a->D;
    const int64_t xs = a->qkv_row_stride ? a->qkv_row_stride : HD;
    if (xs < HD) return fail(KDA_ERR_INVALID_ARG, "qkv_row_stride %lld < H*D", (long long)xs);
    if (!aligned(a->state, 16)) return fail(KDA_ERR_INVALID_ARG, "state must be 16-byte aligned");
    const size_t sb = (size_t)a->N * HD * a->D * sizeof(float);
    const size_t ob = (size_t)a->N * HD * dsize(a->out_dtype);
    if (overlap(a->out, ob, a->state, sb)) return fail(KDA_ERR_INVALID_ARG, "out overlaps state");
    cudaError_t e = kda::launch_decode(*a, reinterpret_cast<cudaStream_t>(stream));
    if (e) return cuda_fail(e, "decode");
    return ok();
}

}  // extern "C"
