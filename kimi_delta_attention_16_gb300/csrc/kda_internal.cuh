// kda_internal.cuh -- device helpers and internal launch declarations shared
// by the libkda.so translation units.  Not part of the public ABI.
#pragma once

#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "../../include/kda.h"

namespace kda {

using bf16 = __nv_bfloat16;

// ------------------------------------------------------------------ math
// SiLU and sigmoid through the CUDA math library's expf (no hand-written
// approximations of library functions).
__device__ __forceinline__ float sigmoidf_(float x) { return 1.0f / (1.0f + expf(-x)); }
__device__ __forceinline__ float siluf_(float x) { return x / (1.0f + expf(-x)); }

// SiLU and sigmoid from one hardware tanh (one MUFU operation instead of an exponential
// and a reciprocal): sigmoid(x) = 1/2 + tanh(x/2)/2, silu(x) = x sigmoid(x).  tanh.approx
// has an absolute error of about 5e-4, so sigmoid is within ~2.5e-4 absolute and silu within
// ~2.5e-4 |x|: for the bf16-input paths only (their tolerance is 2e-3 after the L2 norm of q
// and k and the RMSNorm of o); the fp32 paths keep the IEEE functions above.
__device__ __forceinline__ float tanh_hw(float x) {
    float y;
    asm("tanh.approx.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}
__device__ __forceinline__ float silu_tanh(float x) {
    const float hx = 0.5f * x;
    return fmaf(hx, tanh_hw(hx), hx);
}
__device__ __forceinline__ float sigmoid_tanh(float x) { return fmaf(0.5f, tanh_hw(0.5f * x), 0.5f); }

// 2^x from the hardware base-2 exponential (ex2.approx, relative error ~2^-22); callers keep
// their log-decays in base 2 (g log2 e) so that e^g = 2^(g log2 e) needs no scaling here.
__device__ __forceinline__ float exp2_hw(float x) {
    float y;
    asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}
constexpr float kLog2e = 1.4426950408889634f;  // log2(e)

// ------------------------------------------------------------------ packed fp32 pairs
// Two fp32 values in one 64-bit register pair.  sm_100-class SMs execute fma/mul/add/sub
// on .f32x2 operands as one instruction per pair, each lane rounded exactly as the scalar
// instruction (round to nearest, no flush), which halves the issue slots of elementwise fp32
// arithmetic in the operand-building phases.
struct f2 {
    uint64_t v;
};
__device__ __forceinline__ f2 f2_of(float a, float b) {
    f2 r;
    asm("mov.b64 %0, {%1, %2};" : "=l"(r.v) : "f"(a), "f"(b));
    return r;
}
__device__ __forceinline__ f2 f2_dup(float a) { return f2_of(a, a); }
__device__ __forceinline__ float f2_lo(f2 x) { return __uint_as_float((uint32_t)x.v); }
__device__ __forceinline__ float f2_hi(f2 x) { return __uint_as_float((uint32_t)(x.v >> 32)); }
__device__ __forceinline__ f2 fma2(f2 a, f2 b, f2 c) {  // a * b + c
    f2 r;
    asm("fma.rn.f32x2 %0, %1, %2, %3;" : "=l"(r.v) : "l"(a.v), "l"(b.v), "l"(c.v));
    return r;
}
__device__ __forceinline__ f2 mul2(f2 a, f2 b) {
    f2 r;
    asm("mul.rn.f32x2 %0, %1, %2;" : "=l"(r.v) : "l"(a.v), "l"(b.v));
    return r;
}
__device__ __forceinline__ f2 add2(f2 a, f2 b) {
    f2 r;
    asm("add.rn.f32x2 %0, %1, %2;" : "=l"(r.v) : "l"(a.v), "l"(b.v));
    return r;
}
__device__ __forceinline__ f2 sub2(f2 a, f2 b) {
    f2 r;
    asm("sub.rn.f32x2 %0, %1, %2;" : "=l"(r.v) : "l"(a.v), "l"(b.v));
    return r;
}

// Activations and decay factors by input dtype: bf16 inputs take the one-MUFU tanh forms and
// the fast exponential (tolerance 2e-3), fp32 inputs the IEEE functions (tolerance 1e-5).
template <typename Tio> __device__ __forceinline__ float act_silu(float x) {
    if constexpr (sizeof(Tio) == 2) return silu_tanh(x); else return siluf_(x);
}
template <typename Tio> __device__ __forceinline__ float act_sigmoid(float x) {
    if constexpr (sizeof(Tio) == 2) return sigmoid_tanh(x); else return sigmoidf_(x);
}
template <typename Tio> __device__ __forceinline__ float decay_exp(float g) {
    if constexpr (sizeof(Tio) == 2) return __expf(g); else return expf(g);
}

// ------------------------------------------------------------------ scalar I/O
__device__ __forceinline__ float to_f(float x) { return x; }
__device__ __forceinline__ float to_f(bf16 x) { return __bfloat162float(x); }
template <typename T> __device__ __forceinline__ T from_f(float x);
template <> __device__ __forceinline__ float from_f<float>(float x) { return x; }
template <> __device__ __forceinline__ bf16 from_f<bf16>(float x) { return __float2bfloat16_rn(x); }

// ------------------------------------------------------------------ 8-wide vector I/O (16/32 B)
__device__ __forceinline__ void load8(const float* p, float v[8]) {
    const float4 a = reinterpret_cast<const float4*>(p)[0];
    const float4 b = reinterpret_cast<const float4*>(p)[1];
    v[0] = a.x; v[1] = a.y; v[2] = a.z; v[3] = a.w;
    v[4] = b.x; v[5] = b.y; v[6] = b.z; v[7] = b.w;
}
__device__ __forceinline__ void load8(const bf16* p, float v[8]) {
    const uint4 u = *reinterpret_cast<const uint4*>(p);
    const uint32_t w[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        v[2 * i] = __uint_as_float(w[i] << 16);
        v[2 * i + 1] = __uint_as_float(w[i] & 0xffff0000u);
    }
}
__device__ __forceinline__ void store8(float* p, const float v[8]) {
    reinterpret_cast<float4*>(p)[0] = make_float4(v[0], v[1], v[2], v[3]);
    reinterpret_cast<float4*>(p)[1] = make_float4(v[4], v[5], v[6], v[7]);
}
__device__ __forceinline__ uint32_t pack_bf16x2(float lo, float hi) {
    const __nv_bfloat162 t = __floats2bfloat162_rn(lo, hi);
    return *reinterpret_cast<const uint32_t*>(&t);
}
__device__ __forceinline__ void store8(bf16* p, const float v[8]) {
    uint4 u;
    u.x = pack_bf16x2(v[0], v[1]);
    u.y = pack_bf16x2(v[2], v[3]);
    u.z = pack_bf16x2(v[4], v[5]);
    u.w = pack_bf16x2(v[6], v[7]);
    *reinterpret_cast<uint4*>(p) = u;
}

// ------------------------------------------------------------------ sequences
// Clamped [start, end) of sequence n: every index stays inside [0, T_total)
// even when the device copy of cu_seqlens is inconsistent.
__device__ __forceinline__ void seq_range(const int32_t* cu, int n, int64_t T_total, int64_t& s,
                                          int64_t& e) {
    int64_t a = cu[n], b = cu[n + 1];
    a = a < 0 ? 0 : (a > T_total ? T_total : a);
    b = b < a ? a : (b > T_total ? T_total : b);
    s = a;
    e = b;
}

__device__ __forceinline__ void flag_status(int* d_status, int code) {
    if (d_status) atomicMax(d_status, code);
}

// Base pointers of the q, k and v parts of a token row (they may be offsets
// into one fused [T][3*H*D] buffer or three separate buffers sharing a row
// stride).
struct QKVParts {
    const void* p[3];
};

// ------------------------------------------------------------------ device attributes
// Highest device ordinal + 1 the library serves (its per-device caches are this long).
constexpr int kMaxDevices = 128;
struct DeviceInfo {
    int sm_count;  // streaming multiprocessors
    int cc_major;  // compute capability
    int cc_minor;
};
// Attributes of the current device, queried once per device (std::call_once, so concurrent
// first calls from several host threads are race-free) and cached for the process.  False
// when there is no current device or its ordinal is not below kMaxDevices.
bool current_device_info(DeviceInfo* out);

// ------------------------------------------------------------------ internal launchers
// Each returns cudaSuccess or the launch error; arguments are validated by the caller.

// cu_seqlens consistency check on the device (used when no host copy was given).
cudaError_t launch_check_cu(const int32_t* cu, int N, int64_t T_total, int* d_status,
                            cudaStream_t s);

// Conv + SiLU (+ L2 on channels < l2_limit).  x/y rows hold 3*H*D channels.
cudaError_t launch_short_conv(QKVParts x, int64_t xs, kda_dtype in_dt, const float* w,
                              const int32_t* cu, int N, int64_t T_total, int H, int D,
                              const void* cs_in, void* y, int64_t ys, kda_dtype out_dt,
                              int l2norm_qk, float eps, cudaStream_t s);

// Last three raw inputs of every sequence (rolling conv state for the next call).
cudaError_t launch_conv_state_out(QKVParts x, int64_t xs, kda_dtype dt, const int32_t* cu,
                                  int N, int64_t T_total, int n_ch, const void* cs_in,
                                  void* cs_out, cudaStream_t s);

// fp32 SIMT chunkwise recurrence: reads convolved q|k|v rows (fp32, stride 3*H*D),
// writes o before the epilogue (fp32 [T][H][D]) and the final state.
cudaError_t launch_chunk_simt(const float* qkv, const float* g, const float* beta,
                              const int32_t* cu, int N, int64_t T_total, int H, int D, int chunk,
                              float scale, const float* S0, float* S_fin, float* o_pre,
                              cudaStream_t s);
bool chunk_simt_supported(int D, int chunk);

// RMSNorm + sigmoid gate on fp32 o rows -> out.
cudaError_t launch_rms_gate(const float* o, int64_t rows, int D, const void* gate,
                            kda_dtype gate_dt, const float* rms_w, float eps, void* out,
                            kda_dtype out_dt, cudaStream_t s);

// Tensor-core projection GEMM with a fused epilogue (arguments validated by the caller).
bool gemm_supported_device();
cudaError_t launch_gemm(const kda_gemm_args& g, cudaStream_t s);

// Single-token decode step.
cudaError_t launch_decode(const kda_decode_args& a, cudaStream_t s);

// Recurrent prefill for batches whose sequences all have at most kShortMaxL
// tokens (D = 128; needs the host copy of cu_seqlens to decide).
constexpr int kShortMaxL = 8;
bool short_prefill_applies(const kda_prefill_args& a);
cudaError_t launch_short_prefill(const kda_prefill_args& a, cudaStream_t s);
// The pipelined TMA kernel of that path (16-byte aligned inputs, T_total > 0): it also writes
// conv_state_out itself, so no separate conv-state launch is needed when it applies.
bool short_tma_applies(const kda_prefill_args& a);
cudaError_t launch_short_tma(const kda_prefill_args& a, cudaStream_t s);

// Backward pass (D = 128): byte offsets of its workspace parts (each 256-byte aligned).
struct BackwardLayout {
    size_t x;        // [T][3][H][D] fp32: q^, k^ (after the L2 norm) and v (after the conv)
    size_t nrm;      // [T][H][2] fp32: the L2 denominators of q and k
    size_t o;        // [T][H][D] fp32: o before the epilogue, then its gradient
    size_t dx;       // [T][3][H][D] fp32: gradients of q^, k^, v, then of the conv outputs
    size_t e;        // [T][H][D] fp32: e_t = v_t - P_t^T k_t, then dk_write
    size_t w;        // [T][H][D] fp32: w_t = dS'_t^T k_t, then the write part of dg
    size_t sck;      // [slots][D][D] fp32: the state at the start of every segment
    size_t dsck;     // [slots][D][D] fp32: the state gradient at the end of every segment
    size_t segtot;   // [slots][D] fp32: dg sums per segment, then the carries
    size_t segown;   // [slots][D] fp32: the read part of each segment's dg sum
    size_t fin;      // [N][H][D] fp32: rowsum(dS_T . S_T)
    size_t prefix;   // [N + 1] int64: segments before each sequence
    size_t rec;      // [slots][kBwdSeg / kBwdChunk][kBwdRecFloats] fp32: the chunk records
    int64_t slots;   // checkpoint slots: H times the sum over sequences of ceil(len / kBwdSeg)
    int64_t max_seg; // the largest segment count of one sequence
    int64_t max_ch;  // the largest chunk count of one sequence
    size_t total;
};
constexpr int kBwdSeg = 64;  // tokens per checkpointed segment of the backward pass
constexpr int kBwdChunk = 16;  // tokens per chunk of the backward's sweeps
// floats of one chunk record: Kr, Qr, Kbar (16 x 128 each), M0, A0, T (16 x 16 each), C_last (128),
// beta (16)
constexpr int kBwdRecFloats = 3 * kBwdChunk * 128 + 3 * kBwdChunk * kBwdChunk + 128 + kBwdChunk;
BackwardLayout backward_layout(const kda_backward_args& b);  // needs fwd.cu_seqlens_host
cudaError_t launch_backward(const kda_backward_args& b, const BackwardLayout& L, char* ws, cudaStream_t s);

}  // namespace kda
