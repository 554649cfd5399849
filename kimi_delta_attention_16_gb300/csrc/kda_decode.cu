// kda_decode.cu -- one KDA decode step: a new token for each of N sequences,
// recurrent state and rolling conv state updated in place.
//
// Page "Animated Kimi K3 architecture diagram", section "LOCAL MEMORY: A
// FIXED MATRIX THAT PREDICTS, FORGETS, AND CORRECTS": DECAY S_bar =
// Diag(alpha_t) S_{t-1}, PROBE/CORRECT e_t = v_t - S_bar^T k_t, WRITE S_t =
// S_bar + beta_t k_t e_t^T; page "Kimi K3 / Architecture", KDA panel: read
// o_t = S_t^T q_t, head RMSNorm, sigmoid gate; short-conv panel: the
// autoregressive rolling state of the previous 3 values per channel.
//
// One CTA owns one (sequence, head).  Its D x D fp32 state slice is read
// once and written once with 16-byte accesses: thread (row group rg, column
// group cg) holds rows rg*RPT .. rg*RPT+RPT-1 of columns 4cg .. 4cg+3 in
// registers, and a warp covers whole 512-byte rows, so every access is
// coalesced.  The state loads are issued first and the conv prologue runs
// while they are in flight.  The two reductions over key rows (S_bar^T k and
// S^T q) go through shared memory.  The kernel is HBM-bound: the state's
// read + write is more than 95% of the bytes of a step.
#include "kda_internal.cuh"

namespace kda {

namespace {

template <int D>
struct DecodeShape {
    static constexpr int NT = (D * D / 4) < 256 ? (D * D / 4) : 256;  // threads
    static constexpr int TPR = D / 4;                                // threads per row
    static constexpr int RG = NT / TPR;                              // row groups
    static constexpr int RPT = D / RG;                               // rows per thread
    static_assert(RPT * RG == D && TPR <= 32, "decode shape");
};

template <int D, typename Tio, typename To>
__global__ void __launch_bounds__(DecodeShape<D>::NT)
k_decode(const Tio* __restrict__ q, const Tio* __restrict__ k, const Tio* __restrict__ v,
         int64_t xs, const Tio* __restrict__ gate, const float* __restrict__ g,
         const float* __restrict__ beta, const float* __restrict__ conv_w,
         const float* __restrict__ rms_w, float eps_l2, float eps_rms, float scale, int H,
         float* __restrict__ state, Tio* __restrict__ conv_state, To* __restrict__ out) {
    using Sh = DecodeShape<D>;
    constexpr int NT = Sh::NT, TPR = Sh::TPR, RG = Sh::RG, RPT = Sh::RPT;
    __shared__ float sx[3][D];        // convolved q, k, v of this head
    __shared__ float sred[RG][D];     // partial sums over row groups
    __shared__ float sinv[2];         // 1/|q|, 1/|k|

    const int nh = blockIdx.x;        // n * H + h
    const int n = nh / H, h = nh % H;
    const int tid = threadIdx.x;
    const int cg = tid % TPR, rg = tid / TPR;
    const int c0 = 4 * cg, r0 = rg * RPT;
    float* S = state + (int64_t)nh * D * D;

    // 1. stream the state slice in (16-byte loads, whole rows per warp)
    float4 s[RPT];
#pragma unroll
    for (int i = 0; i < RPT; ++i) s[i] = *reinterpret_cast<const float4*>(S + (r0 + i) * D + c0);

    // 2. conv + SiLU on the new token, rolling the conv state in place
    const int64_t HD = (int64_t)H * D;
    for (int idx = tid; idx < 3 * D; idx += NT) {
        const int part = idx / D, d = idx % D;
        const int64_t ch = part * HD + (int64_t)h * D + d;
        const Tio* src = part == 0 ? q : (part == 1 ? k : v);
        Tio* cs = conv_state + ((int64_t)n * 3 * HD + ch) * 3;
        const float x0 = to_f(cs[0]), x1 = to_f(cs[1]), x2 = to_f(cs[2]);
        const Tio xr = src[(int64_t)n * xs + (int64_t)h * D + d];
        const float x3 = to_f(xr);
        const float* w = conv_w + ch * 4;
        const float u = w[0] * x0 + w[1] * x1 + w[2] * x2 + w[3] * x3;
        cs[0] = cs[1];
        cs[1] = cs[2];
        cs[2] = xr;
        sx[part][d] = siluf_(u);
    }
    __syncthreads();

    // 3. L2 norms of q (warp 0) and k (warp 1 or, with one warp, the same warp)
    {
        const int warp = tid / 32, lane = tid % 32;
        constexpr int NW = NT / 32 > 0 ? NT / 32 : 1;
        for (int which = warp; which < 2; which += NW) {
            float ss = 0.f;
            for (int d = lane; d < D; d += 32) ss += sx[which][d] * sx[which][d];
#pragma unroll
            for (int off = 16; off > 0; off >>= 1) ss += __shfl_xor_sync(0xffffffffu, ss, off);
            if (lane == 0) sinv[which] = 1.0f / sqrtf(ss + eps_l2);
        }
    }
    __syncthreads();
    const float iq = sinv[0], ik = sinv[1];

    // 4. decay rows, probe: partial (S_bar^T k) over this thread's rows
    const float* gr = g + (int64_t)nh * D;
    float kr[RPT], qr[RPT];
    float4 p = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
    for (int i = 0; i < RPT; ++i) {
        const float a = expf(gr[r0 + i]);
        kr[i] = sx[1][r0 + i] * ik;
        qr[i] = sx[0][r0 + i] * iq;
        s[i].x *= a; s[i].y *= a; s[i].z *= a; s[i].w *= a;
        p.x = fmaf(kr[i], s[i].x, p.x); p.y = fmaf(kr[i], s[i].y, p.y);
        p.z = fmaf(kr[i], s[i].z, p.z); p.w = fmaf(kr[i], s[i].w, p.w);
    }
    *reinterpret_cast<float4*>(&sred[rg][c0]) = p;
    __syncthreads();

    // 5. correct: e = v - S_bar^T k; write: S = S_bar + beta k e^T; read: partial S^T q
    float4 e;
    {
        float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll 4
        for (int r = 0; r < RG; ++r) {
            const float4 t = *reinterpret_cast<const float4*>(&sred[r][c0]);
            acc.x += t.x; acc.y += t.y; acc.z += t.z; acc.w += t.w;
        }
        e.x = sx[2][c0 + 0] - acc.x; e.y = sx[2][c0 + 1] - acc.y;
        e.z = sx[2][c0 + 2] - acc.z; e.w = sx[2][c0 + 3] - acc.w;
    }
    const float b = beta[nh];
    float4 po = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
    for (int i = 0; i < RPT; ++i) {
        const float bk = b * kr[i];
        s[i].x = fmaf(bk, e.x, s[i].x); s[i].y = fmaf(bk, e.y, s[i].y);
        s[i].z = fmaf(bk, e.z, s[i].z); s[i].w = fmaf(bk, e.w, s[i].w);
        *reinterpret_cast<float4*>(S + (r0 + i) * D + c0) = s[i];
        po.x = fmaf(qr[i], s[i].x, po.x); po.y = fmaf(qr[i], s[i].y, po.y);
        po.z = fmaf(qr[i], s[i].z, po.z); po.w = fmaf(qr[i], s[i].w, po.w);
    }
    __syncthreads();  // everyone has read sred for e
    *reinterpret_cast<float4*>(&sred[rg][c0]) = po;
    __syncthreads();

    // 6. o = scale S^T q, head RMSNorm, sigmoid gate (row group 0 = first TPR threads of warp 0)
    if (rg == 0) {
        float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll 4
        for (int r = 0; r < RG; ++r) {
            const float4 t = *reinterpret_cast<const float4*>(&sred[r][c0]);
            acc.x += t.x; acc.y += t.y; acc.z += t.z; acc.w += t.w;
        }
        const float o[4] = {scale * acc.x, scale * acc.y, scale * acc.z, scale * acc.w};
        float ss = o[0] * o[0] + o[1] * o[1] + o[2] * o[2] + o[3] * o[3];
        constexpr unsigned kRowMask = TPR == 32 ? 0xffffffffu : ((1u << TPR) - 1u);
#pragma unroll
        for (int off = TPR / 2; off > 0; off >>= 1) ss += __shfl_xor_sync(kRowMask, ss, off);
        const float inv = 1.0f / sqrtf(ss / D + eps_rms);
        To* dst = out + (int64_t)nh * D + c0;
        const Tio* gt = gate ? gate + (int64_t)nh * D + c0 : nullptr;
#pragma unroll
        for (int m = 0; m < 4; ++m) {
            float y = o[m] * inv;
            if (rms_w) y *= rms_w[c0 + m];
            if (gt) y *= sigmoidf_(to_f(gt[m]));
            dst[m] = from_f<To>(y);
        }
    }
}

template <int D, typename Tio, typename To>
cudaError_t decode_launch(const kda_decode_args& a, cudaStream_t s) {
    const int64_t xs = a.qkv_row_stride ? a.qkv_row_stride : (int64_t)a.H * D;
    const unsigned blocks = (unsigned)((int64_t)a.N * a.H);
    if (blocks == 0) return cudaSuccess;
    k_decode<D, Tio, To><<<blocks, DecodeShape<D>::NT, 0, s>>>(
        (const Tio*)a.q, (const Tio*)a.k, (const Tio*)a.v, xs, (const Tio*)a.gate, a.g, a.beta,
        a.conv_w, a.rms_w, a.eps_l2, a.eps_rms, a.scale, a.H, a.state, (Tio*)a.conv_state,
        (To*)a.out);
    return cudaGetLastError();
}

template <int D>
cudaError_t decode_dt(const kda_decode_args& a, cudaStream_t s) {
    if (a.io == KDA_BF16 && a.out_dtype == KDA_BF16) return decode_launch<D, bf16, bf16>(a, s);
    if (a.io == KDA_BF16 && a.out_dtype == KDA_FP32) return decode_launch<D, bf16, float>(a, s);
    if (a.io == KDA_FP32 && a.out_dtype == KDA_FP32) return decode_launch<D, float, float>(a, s);
    if (a.io == KDA_FP32 && a.out_dtype == KDA_BF16) return decode_launch<D, float, bf16>(a, s);
    return cudaErrorInvalidValue;
}

}  // namespace

cudaError_t launch_decode(const kda_decode_args& a, cudaStream_t s) {
    switch (a.D) {
        case 16: return decode_dt<16>(a, s);
        case 32: return decode_dt<32>(a, s);
        case 64: return decode_dt<64>(a, s);
        case 128: return decode_dt<128>(a, s);
        default: return cudaErrorInvalidValue;
    }
}

}  // namespace kda
