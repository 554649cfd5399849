// kda_short.cu -- the recurrent path of kda_prefill for batches of short
// sequences (every sequence at most kShortMaxL tokens): multi-token decode
// and speculative verification, where a chunk of 64 would be mostly empty.
//
// Page "Animated Kimi K3 architecture diagram", section "LOCAL MEMORY: A
// FIXED MATRIX THAT PREDICTS, FORGETS, AND CORRECTS": per token, DECAY
// S_bar = Diag(alpha_t) S, PROBE/CORRECT e = v - S_bar^T k, WRITE
// S = S_bar + beta k e^T; page "Kimi K3 / Architecture": the short conv with
// its rolling window, the read o = S^T q, head RMSNorm and the sigmoid gate.
//
// This file holds the plain kernel of that path, for inputs the pipelined TMA
// kernel (kda_short_tma.cu) cannot take because they are not 16-byte aligned.
//
// Persistent CTAs (two per SM) walk contiguous head-major ranges of (sequence,
// head) units.  A unit's D x D fp32 state is read into registers once, takes
// the sequence's tokens one after another, and is written once; thread
// (row group rg = warp, column group cg = lane) holds rows 16 rg .. 16 rg + 15
// of columns 4 cg .. 4 cg + 3, so every state access is a coalesced 16-byte
// one.  Everything that does not depend on the state (conv + SiLU, L2 norms,
// decay factors) is done for all of the unit's tokens first; the token loop
// then needs one barrier per token, because the readout of token t - 1 and
// the decay and probe of token t share one pass over the state registers
// (S_{t-1}^T q_{t-1} before the decay, S_bar_t^T k_t after it) and their
// row-group partial sums are double-buffered.  While a unit computes, the next
// unit's state, rows and conv window are prefetched into L2.
#include "kda_internal.cuh"
#include "kda_tc_ptx.cuh"

namespace kda {

namespace {

constexpr int kD = 128;
constexpr int kShortThreads = 256;


__device__ __forceinline__ void prefetch_l2(const void* p) {
    asm volatile("prefetch.global.L2 [%0];" ::"l"(p) : "memory");
}

template <typename Tio, typename To>
__global__ void __launch_bounds__(kShortThreads, 2)
k_prefill_short(const Tio* __restrict__ q, const Tio* __restrict__ k, const Tio* __restrict__ v,
                int64_t xs, const Tio* __restrict__ gate, const float* __restrict__ g,
                const float* __restrict__ beta, const float* __restrict__ conv_w,
                const Tio* __restrict__ cs_in, const float* __restrict__ rms_w, float eps_l2,
                float eps_rms, float scale, int N, int H, const int32_t* __restrict__ cu,
                int64_t T_total, const float* S0, float* S_fin, To* __restrict__ out,
                int* d_status) {
    constexpr int L8 = kShortMaxL;
    // sbuf: raw q, k, v rows [L][3][128] while convolving, then the row-group partial sums
    // of the token loop: probe [2][8][128] and readout [2][8][128] (double-buffered by token)
    __shared__ __align__(16) float sbuf[4 * 8 * kD];
    __shared__ __align__(16) float sx[L8][3][kD];   // convolved q, k, v of every token
    __shared__ __align__(16) float salpha[L8][kD];  // e^g of every token
    __shared__ __align__(16) float sgate[L8][kD];
    __shared__ __align__(16) float sW[3 * kD * 4];  // conv taps of the current head
    __shared__ float sRms[kD];
    __shared__ float snorm[L8][2];                  // 1/|q|, 1/|k| per token
    __shared__ float sbeta[L8];
    __shared__ int s_head;
    float* sraw = sbuf;
    float* sredP = sbuf;
    float* sredO = sbuf + 2 * 8 * kD;

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int rg = warp, cg = lane;
    const int r0 = 16 * rg, c0 = 4 * cg;
    const int64_t HD = (int64_t)H * kD;
    const int units = N * H;
    const int per = (units + gridDim.x - 1) / gridDim.x;
    const int first = blockIdx.x * per;
    const int my_units = first < units ? (units - first < per ? units - first : per) : 0;
    auto unit_of = [&](int i, int& n, int& h) {  // head-major: j = h * N + n
        const int jj = first + i;
        h = jj / N;
        n = jj % N;
    };
    if (tid == 0) s_head = -1;
    for (int c = tid; c < kD; c += kShortThreads) sRms[c] = rms_w ? rms_w[c] : 1.f;
    __syncthreads();

    // L2 prefetch of everything unit i reads (state, conv window, token rows)
    auto prefetch_unit = [&](int i) {
        int n, h;
        unit_of(i, n, h);
        int64_t a, b;
        seq_range(cu, n, T_total, a, b);
        const int L = (int)((b - a) < L8 ? (b - a) : L8);
        const int u = n * H + h;
        if (S0) {
            const char* st = reinterpret_cast<const char*>(S0 + (int64_t)u * kD * kD);
            prefetch_l2(st + 128 * tid);
            prefetch_l2(st + 128 * (tid + kShortThreads));
        }
        // rows: per token q, k, v, gate (2 lines each for bf16, 4 for fp32) and g (4 lines)
        constexpr int kLines = kD * (int)sizeof(Tio) / 128;
        const int per_tok = 4 * kLines + 4;
        if (tid < L * per_tok) {
            const int tk = tid / per_tok, w = tid % per_tok;
            const int64_t t = a + tk;
            const char* p;
            if (w < 4 * kLines) {
                const int part = w / kLines, ln = w % kLines;
                const Tio* src = part == 0 ? q : part == 1 ? k : part == 2 ? v : gate;
                p = src ? reinterpret_cast<const char*>(src + (part < 3 ? t * xs : t * HD) + (int64_t)h * kD) + 128 * ln
                        : nullptr;
            } else {
                p = reinterpret_cast<const char*>(g + (t * H + h) * kD) + 128 * (w - 4 * kLines);
            }
            if (p) prefetch_l2(p);
        }
        if (cs_in && tid < 3 * 3 * kLines) {  // 3 parts x 128 channels x 3 values
            const int part = tid / (3 * kLines), ln = tid % (3 * kLines);
            prefetch_l2(reinterpret_cast<const char*>(cs_in + (((int64_t)n * 3 + part) * HD + (int64_t)h * kD) * 3) +
                        128 * ln);
        }
    };
    if (my_units > 0) prefetch_unit(0);

    for (int i = 0; i < my_units; ++i) {
        int n, h;
        unit_of(i, n, h);
        const int u = n * H + h;
        int64_t a, b;
        seq_range(cu, n, T_total, a, b);
        int L = (int)(b - a);
        if (L > L8) {  // the host routes only sequences of at most kShortMaxL tokens here
            if (tid == 0) flag_status(d_status, KDA_ERR_DEVICE_ARG);
            L = L8;
        }
        if (i + 1 < my_units) prefetch_unit(i + 1);
        if (h != s_head) {  // a new head: its conv taps (uniform branch; read after barrier A)
            for (int idx = tid; idx < 3 * kD * 4; idx += kShortThreads) {
                const int part = idx / (kD * 4), rem = idx % (kD * 4);
                sW[idx] = conv_w[(part * HD + (int64_t)h * kD) * 4 + rem];
            }
        }
        // ---- prologue: the unit's rows, decay factors and gates; its state into registers
        for (int idx = tid; idx < L * 3 * kD; idx += kShortThreads) {
            const int tau = idx / (3 * kD), ch = idx % (3 * kD), part = ch >> 7, d = ch & (kD - 1);
            const Tio* src = part == 0 ? q : (part == 1 ? k : v);
            sraw[idx] = to_f(src[(a + tau) * xs + (int64_t)h * kD + d]);
        }
        for (int idx = tid; idx < L * kD; idx += kShortThreads) {
            const int tau = idx >> 7, d = idx & (kD - 1);
            const int64_t row = ((a + tau) * H + h) * kD + d;
            salpha[tau][d] = decay_exp<Tio>(g[row]);
            sgate[tau][d] = gate ? to_f(gate[row]) : 0.f;
        }
        if (tid < L) sbeta[tid] = beta[(a + tid) * H + h];
        float4 s[16];
        {
            const float* src = S0 ? S0 + (int64_t)u * kD * kD : nullptr;
#pragma unroll
            for (int e = 0; e < 16; ++e)
                s[e] = src ? *reinterpret_cast<const float4*>(src + (r0 + e) * kD + c0) : make_float4(0.f, 0.f, 0.f, 0.f);
        }
        __syncthreads();  // A: raw rows, conv taps
        if (tid == 0) s_head = h;
        // conv + SiLU of every token (the window reaches into the rolling conv state)
        for (int idx = tid; idx < L * 3 * kD; idx += kShortThreads) {
            const int tau = idx / (3 * kD), ch = idx % (3 * kD), part = ch >> 7, d = ch & (kD - 1);
            const float4 w = *reinterpret_cast<const float4*>(&sW[ch * 4]);
            float x[4];
#pragma unroll
            for (int m = 0; m < 4; ++m) {
                const int rel = tau - 3 + m;
                x[m] = rel >= 0 ? sraw[rel * 3 * kD + ch]
                                : (cs_in ? to_f(cs_in[(((int64_t)n * 3 + part) * HD + (int64_t)h * kD + d) * 3 + 3 + rel]) : 0.f);
            }
            sx[tau][part][d] = act_silu<Tio>(w.x * x[0] + w.y * x[1] + w.z * x[2] + w.w * x[3]);
        }
        __syncthreads();  // B
        // L2 norms: warp w takes (token, q or k) pairs w, w + 8, ...
        for (int rr = warp; rr < 2 * L; rr += kShortThreads / 32) {
            const int tau = rr >> 1, which = rr & 1;
            float ss = 0.f;
#pragma unroll
            for (int d = lane; d < kD; d += 32) ss += sx[tau][which][d] * sx[tau][which][d];
#pragma unroll
            for (int off = 16; off > 0; off >>= 1) ss += __shfl_xor_sync(0xffffffffu, ss, off);
            if (lane == 0) snorm[tau][which] = 1.0f / sqrtf(ss + eps_l2);
        }
        __syncthreads();  // C: the partial-sum buffers (aliasing the raw rows) are free now

        // o of token tau (row group 0): sum of the readout partials, RMSNorm, gate, store
        auto emit = [&](int tau, int buf) {
            float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
            for (int rr = 0; rr < 8; ++rr) {
                const float4 tt = *reinterpret_cast<const float4*>(&sredO[(buf * 8 + rr) * kD + c0]);
                acc.x += tt.x; acc.y += tt.y; acc.z += tt.z; acc.w += tt.w;
            }
            const float o[4] = {acc.x, acc.y, acc.z, acc.w};
            float ss = o[0] * o[0] + o[1] * o[1] + o[2] * o[2] + o[3] * o[3];
#pragma unroll
            for (int off = 16; off > 0; off >>= 1) ss += __shfl_xor_sync(0xffffffffu, ss, off);
            const float inv = 1.0f / sqrtf(ss / kD + eps_rms);
            const int64_t row = ((a + tau) * H + h) * kD + c0;
#pragma unroll
            for (int m = 0; m < 4; ++m) {
                float y = o[m] * inv * sRms[c0 + m];
                if (gate) y *= act_sigmoid<Tio>(sgate[tau][c0 + m]);
                out[row + m] = from_f<To>(y);
            }
        };
        // ---- token loop, one barrier per token: the readout of token tau - 1 (its partials
        // over this thread's rows) shares a pass over the state with token tau's decay and probe
        for (int tau = 0; tau < L; ++tau) {
            const int buf = tau & 1;
            const float ik = snorm[tau][1];
            const float iqp = tau > 0 ? snorm[tau - 1][0] * scale : 0.f;
            float4 p = make_float4(0.f, 0.f, 0.f, 0.f), po = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
            for (int e = 0; e < 16; ++e) {
                if (tau > 0) {
                    const float qr = sx[tau - 1][0][r0 + e] * iqp;
                    po.x = fmaf(qr, s[e].x, po.x); po.y = fmaf(qr, s[e].y, po.y);
                    po.z = fmaf(qr, s[e].z, po.z); po.w = fmaf(qr, s[e].w, po.w);
                }
                const float al = salpha[tau][r0 + e];
                const float kr = sx[tau][1][r0 + e] * ik;
                s[e].x *= al; s[e].y *= al; s[e].z *= al; s[e].w *= al;
                p.x = fmaf(kr, s[e].x, p.x); p.y = fmaf(kr, s[e].y, p.y);
                p.z = fmaf(kr, s[e].z, p.z); p.w = fmaf(kr, s[e].w, p.w);
            }
            *reinterpret_cast<float4*>(&sredP[(buf * 8 + rg) * kD + c0]) = p;
            if (tau > 0) *reinterpret_cast<float4*>(&sredO[(buf * 8 + rg) * kD + c0]) = po;
            __syncthreads();
            // correct: e = v - S_bar^T k; write: S = S_bar + beta k e^T
            float4 ev = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
            for (int rr = 0; rr < 8; ++rr) {
                const float4 tt = *reinterpret_cast<const float4*>(&sredP[(buf * 8 + rr) * kD + c0]);
                ev.x += tt.x; ev.y += tt.y; ev.z += tt.z; ev.w += tt.w;
            }
            ev.x = sx[tau][2][c0] - ev.x; ev.y = sx[tau][2][c0 + 1] - ev.y;
            ev.z = sx[tau][2][c0 + 2] - ev.z; ev.w = sx[tau][2][c0 + 3] - ev.w;
            const float bb = sbeta[tau] * ik;
#pragma unroll
            for (int e = 0; e < 16; ++e) {
                const float bk = bb * sx[tau][1][r0 + e];
                s[e].x = fmaf(bk, ev.x, s[e].x); s[e].y = fmaf(bk, ev.y, s[e].y);
                s[e].z = fmaf(bk, ev.z, s[e].z); s[e].w = fmaf(bk, ev.w, s[e].w);
            }
            if (tau > 0 && rg == 0) emit(tau - 1, buf);
        }
        if (L > 0) {  // readout of the last token
            const int buf = L & 1;
            const float iq = snorm[L - 1][0] * scale;
            float4 po = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
            for (int e = 0; e < 16; ++e) {
                const float qr = sx[L - 1][0][r0 + e] * iq;
                po.x = fmaf(qr, s[e].x, po.x); po.y = fmaf(qr, s[e].y, po.y);
                po.z = fmaf(qr, s[e].z, po.z); po.w = fmaf(qr, s[e].w, po.w);
            }
            *reinterpret_cast<float4*>(&sredO[(buf * 8 + rg) * kD + c0]) = po;
            __syncthreads();
            if (rg == 0) emit(L - 1, buf);
        }
        if (S_fin) {
            float* dst = S_fin + (int64_t)u * kD * kD;
#pragma unroll
            for (int e = 0; e < 16; ++e) *reinterpret_cast<float4*>(dst + (r0 + e) * kD + c0) = s[e];
        }
        __syncthreads();  // D: every read of this unit's shared rows is done
    }
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

int device_sms() {
    DeviceInfo d;
    return current_device_info(&d) ? d.sm_count : 148;
}

template <typename Tio, typename To>
cudaError_t short_launch(const kda_prefill_args& a, cudaStream_t s) {
    const int units = a.N * a.H;
    const int sms = device_sms();
    const int blocks = units < 2 * sms ? units : 2 * sms;
    const int64_t xs = a.qkv_row_stride ? a.qkv_row_stride : (int64_t)a.H * kD;
    k_prefill_short<Tio, To><<<blocks, kShortThreads, 0, s>>>(
        (const Tio*)a.q, (const Tio*)a.k, (const Tio*)a.v, xs, (const Tio*)a.gate, a.g, a.beta, a.conv_w,
        (const Tio*)a.conv_state_in, a.rms_w, a.eps_l2, a.eps_rms, a.scale, a.N, a.H, a.cu_seqlens,
        a.T_total, a.initial_state, a.final_state, (To*)a.out, a.d_status);
    return cudaGetLastError();
}

}  // namespace

bool short_prefill_applies(const kda_prefill_args& a) {
    if (a.D != kD || !a.cu_seqlens_host || a.N < 1 || (int64_t)a.N * a.H > 0x7fffffffLL) return false;
    for (int n = 0; n < a.N; ++n)
        if (a.cu_seqlens_host[n + 1] - a.cu_seqlens_host[n] > kShortMaxL) return false;
    // 16-byte state rows (float4); everything else is read with scalar loads
    return (!a.initial_state || aligned16(a.initial_state)) && (!a.final_state || aligned16(a.final_state));
}

cudaError_t launch_short_prefill(const kda_prefill_args& a, cudaStream_t s) {
    if ((int64_t)a.N * a.H == 0) return cudaSuccess;
    if (a.io == KDA_BF16)
        return a.out_dtype == KDA_FP32 ? short_launch<bf16, float>(a, s) : short_launch<bf16, bf16>(a, s);
    return a.out_dtype == KDA_FP32 ? short_launch<float, float>(a, s) : short_launch<float, bf16>(a, s);
}

}  // namespace kda
