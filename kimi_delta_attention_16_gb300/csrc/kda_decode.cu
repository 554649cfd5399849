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
#include "kda_tc_ptx.cuh"

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
    // float4 accesses below: static shared arrays need an explicit 16-byte alignment
    __shared__ __align__(16) float sx[3][D];     // convolved q, k, v of this head
    __shared__ __align__(16) float sred[RG][D];  // partial sums over row groups
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


// ---------------------------------------------------------------------------------------
// Pipelined decode for D = 128: persistent CTAs (one per SM) walk units (sequence, head)
// with a 3-stage pipeline of 1D bulk copies (the TMA engine).  A unit's 64 KB state slice,
// its three conv-state segments, raw q/k/v, gate and log-decay arrive in shared memory
// two units ahead of the compute; the updated state and conv state leave with bulk
// stores, so HBM always has loads and stores in flight while the SM computes.
template <typename Tio>
struct DecodeStage {
    static constexpr uint32_t kState = 0;
    static constexpr uint32_t kConv = 65536;                               // [3][128][3]
    static constexpr uint32_t kConvPart = 128 * 3 * sizeof(Tio);
    static constexpr uint32_t kRaw = kConv + 3 * kConvPart;                // [3][128]
    static constexpr uint32_t kRawPart = 128 * sizeof(Tio);
    static constexpr uint32_t kGate = kRaw + 3 * kRawPart;                 // [128]
    static constexpr uint32_t kG = kGate + 128 * sizeof(Tio);              // [128] fp32
    static constexpr uint32_t kBytes = (kG + 512 + 127) / 128 * 128;
    static constexpr int kStages = 3;
    static constexpr uint32_t kSmem = kStages * kBytes + 128;
};

template <typename Tio, typename To>
__global__ void __launch_bounds__(256, 1)
k_decode_tma(const Tio* __restrict__ q, const Tio* __restrict__ k, const Tio* __restrict__ v, int64_t xs,
             const Tio* __restrict__ gate, const float* __restrict__ g, const float* __restrict__ beta,
             const float* __restrict__ conv_w, const float* __restrict__ rms_w, float eps_l2,
             float eps_rms, float scale, int H, int units, float* __restrict__ state,
             Tio* __restrict__ conv_state, To* __restrict__ out, int* d_status) {
    using St = DecodeStage<Tio>;
    constexpr int D = 128;
    extern __shared__ uint8_t smem_raw[];
    __shared__ uint64_t bars[St::kStages];
    __shared__ __align__(16) float sx[3][D];
    __shared__ __align__(16) float sred[8][D];  // float4 accesses: explicit 16-byte alignment
    __shared__ __align__(16) float sW[3 * D * 4];  // conv taps of the current head
    __shared__ float sRms[D];
    __shared__ float sbeta[St::kStages];
    __shared__ float sinv[2];
    __shared__ int s_head;
    const uint32_t raw_addr = tc::smem_u32(smem_raw);
    uint8_t* sm = smem_raw + (((raw_addr + 127u) & ~127u) - raw_addr);
    const uint32_t sbase = tc::smem_u32(sm);
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int64_t HD = (int64_t)H * D;
    // units in head-major order (j = h * N + n), one contiguous range per CTA, so a CTA meets
    // few distinct heads and keeps the current head's conv taps in shared memory
    const int per = (units + gridDim.x - 1) / gridDim.x;
    const int first = blockIdx.x * per;
    const int my_units = first < units ? (units - first < per ? units - first : per) : 0;
    const int Nseq = units / H;
    auto unit_of = [&](int i, int& n, int& h) {
        const int jj = first + i;
        h = jj / Nseq;
        n = jj % Nseq;
    };
    const uint32_t tx_bytes = 65536 + 3 * St::kConvPart + 3 * St::kRawPart + (gate ? St::kRawPart : 0) + 512;

    if (tid == 0) {
        for (int i = 0; i < St::kStages; ++i) tc::mbar_init(&bars[i], 1);
        tc::fence_mbar_init();
        s_head = -1;
    }
    for (int c = tid; c < D; c += 256) sRms[c] = rms_w ? rms_w[c] : 1.f;
    __syncthreads();

    auto issue = [&](int i) {  // bulk loads of this CTA's i-th unit
        const int b = i % St::kStages;
        int n, h;
        unit_of(i, n, h);
        const int u = n * H + h;
        const uint32_t st = sbase + b * St::kBytes;
        tc::mbar_expect_tx(&bars[b], tx_bytes);
        tc::bulk_load(st + St::kState, state + (int64_t)u * D * D, 65536, &bars[b]);
        const Tio* src[3] = {q, k, v};
#pragma unroll
        for (int p = 0; p < 3; ++p) {
            tc::bulk_load(st + St::kConv + p * St::kConvPart,
                          conv_state + (((int64_t)n * 3 + p) * HD + (int64_t)h * D) * 3, St::kConvPart, &bars[b]);
            tc::bulk_load(st + St::kRaw + p * St::kRawPart, src[p] + (int64_t)n * xs + (int64_t)h * D,
                          St::kRawPart, &bars[b]);
        }
        if (gate) tc::bulk_load(st + St::kGate, gate + (int64_t)u * D, St::kRawPart, &bars[b]);
        tc::bulk_load(st + St::kG, g + (int64_t)u * D, 512, &bars[b]);
    };
    if (tid == 0)
        for (int i = 0; i < St::kStages - 1 && i < my_units; ++i) issue(i);
    if (tid == 32)
        for (int i = 0; i < St::kStages - 1 && i < my_units; ++i) {
            int n, h;
            unit_of(i, n, h);
            sbeta[i % St::kStages] = beta[n * H + h];
        }

    const int cg = lane, rg = warp;  // 4 columns 4cg.., 16 rows 16rg..
    const int c0 = 4 * cg, r0 = 16 * rg;
    bool failed = false;
    for (int i = 0; i < my_units; ++i) {
        const int b = i % St::kStages;
        int n, h;
        unit_of(i, n, h);
        const int u = n * H + h;
        uint8_t* st = sm + b * St::kBytes;
        if (!__syncthreads_and(tc::mbar_wait(&bars[b], (i / St::kStages) & 1))) {
            failed = true;
            break;
        }
        if (h != s_head) {  // a new head: reload its conv taps (uniform branch)
            for (int idx = tid; idx < 3 * D * 4; idx += 256) {
                const int part = idx / (D * 4), rem = idx % (D * 4);
                sW[idx] = conv_w[(part * HD + (int64_t)h * D) * 4 + rem];
            }
            __syncthreads();
            if (tid == 0) s_head = h;
        }
        float* S = reinterpret_cast<float*>(st + St::kState);
        Tio* cs = reinterpret_cast<Tio*>(st + St::kConv);
        const Tio* xr = reinterpret_cast<const Tio*>(st + St::kRaw);
        // conv + SiLU on the new token; the rolled conv state stays in the stage for the store
        for (int idx = tid; idx < 3 * D; idx += 256) {
            const int part = idx >> 7, d = idx & (D - 1);
            Tio* c3 = cs + (part * D + d) * 3;
            const float x0 = to_f(c3[0]), x1 = to_f(c3[1]), x2 = to_f(c3[2]);
            const Tio xn = xr[part * D + d];
            const float4 w = *reinterpret_cast<const float4*>(&sW[(part * D + d) * 4]);
            const float uu = w.x * x0 + w.y * x1 + w.z * x2 + w.w * to_f(xn);
            c3[0] = c3[1];
            c3[1] = c3[2];
            c3[2] = xn;
            sx[part][d] = act_silu<Tio>(uu);
        }
        __syncthreads();
        if (warp < 2) {
            float ss = 0.f;
#pragma unroll
            for (int d = lane; d < D; d += 32) ss += sx[warp][d] * sx[warp][d];
#pragma unroll
            for (int off = 16; off > 0; off >>= 1) ss += __shfl_xor_sync(0xffffffffu, ss, off);
            if (lane == 0) sinv[warp] = 1.0f / sqrtf(ss + eps_l2);
        }
        __syncthreads();
        const float iq = sinv[0], ik = sinv[1];
        const float* gr = reinterpret_cast<const float*>(st + St::kG);
        float4 s[16];
        float kr[16], qr[16];
        float4 p = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
        for (int e = 0; e < 16; ++e) {
            s[e] = *reinterpret_cast<const float4*>(S + (r0 + e) * D + c0);
            const float a = decay_exp<Tio>(gr[r0 + e]);
            kr[e] = sx[1][r0 + e] * ik;
            qr[e] = sx[0][r0 + e] * iq;
            s[e].x *= a; s[e].y *= a; s[e].z *= a; s[e].w *= a;
            p.x = fmaf(kr[e], s[e].x, p.x); p.y = fmaf(kr[e], s[e].y, p.y);
            p.z = fmaf(kr[e], s[e].z, p.z); p.w = fmaf(kr[e], s[e].w, p.w);
        }
        *reinterpret_cast<float4*>(&sred[rg][c0]) = p;
        __syncthreads();
        float4 ev = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
        for (int rr = 0; rr < 8; ++rr) {
            const float4 t = *reinterpret_cast<const float4*>(&sred[rr][c0]);
            ev.x += t.x; ev.y += t.y; ev.z += t.z; ev.w += t.w;
        }
        ev.x = sx[2][c0] - ev.x; ev.y = sx[2][c0 + 1] - ev.y; ev.z = sx[2][c0 + 2] - ev.z; ev.w = sx[2][c0 + 3] - ev.w;
        const float bb = sbeta[b];
        float4 po = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
        for (int e = 0; e < 16; ++e) {
            const float bk = bb * kr[e];
            s[e].x = fmaf(bk, ev.x, s[e].x); s[e].y = fmaf(bk, ev.y, s[e].y);
            s[e].z = fmaf(bk, ev.z, s[e].z); s[e].w = fmaf(bk, ev.w, s[e].w);
            *reinterpret_cast<float4*>(S + (r0 + e) * D + c0) = s[e];
            po.x = fmaf(qr[e], s[e].x, po.x); po.y = fmaf(qr[e], s[e].y, po.y);
            po.z = fmaf(qr[e], s[e].z, po.z); po.w = fmaf(qr[e], s[e].w, po.w);
        }
        __syncthreads();  // everyone has read sred for e
        *reinterpret_cast<float4*>(&sred[rg][c0]) = po;
        tc::fence_async_smem();  // state and conv-state updates -> visible to the bulk store
        __syncthreads();
        if (tid == 0) {
            tc::bulk_store(state + (int64_t)u * D * D, sbase + b * St::kBytes + St::kState, 65536);
#pragma unroll
            for (int pp = 0; pp < 3; ++pp)
                tc::bulk_store(conv_state + (((int64_t)n * 3 + pp) * HD + (int64_t)h * D) * 3,
                               sbase + b * St::kBytes + St::kConv + pp * St::kConvPart, St::kConvPart);
            tc::bulk_commit();
            if (i + St::kStages - 1 < my_units) {
                tc::bulk_wait_read<1>();  // the store of the unit before this one has left its buffer
                issue(i + St::kStages - 1);
            }
        }
        if (tid == 32 && i + St::kStages - 1 < my_units) {  // beta two units ahead (read after later barriers)
            int n2, h2;
            unit_of(i + St::kStages - 1, n2, h2);
            sbeta[(i + St::kStages - 1) % St::kStages] = beta[n2 * H + h2];
        }
        if (rg == 0) {
            float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
            for (int rr = 0; rr < 8; ++rr) {
                const float4 t = *reinterpret_cast<const float4*>(&sred[rr][c0]);
                acc.x += t.x; acc.y += t.y; acc.z += t.z; acc.w += t.w;
            }
            const float o[4] = {scale * acc.x, scale * acc.y, scale * acc.z, scale * acc.w};
            float ss = o[0] * o[0] + o[1] * o[1] + o[2] * o[2] + o[3] * o[3];
#pragma unroll
            for (int off = 16; off > 0; off >>= 1) ss += __shfl_xor_sync(0xffffffffu, ss, off);
            const float inv = 1.0f / sqrtf(ss / D + eps_rms);
            const Tio* gt = gate ? reinterpret_cast<const Tio*>(st + St::kGate) + c0 : nullptr;
            To* dst = out + (int64_t)u * D + c0;
#pragma unroll
            for (int m = 0; m < 4; ++m) {
                float y = o[m] * inv;
                y *= sRms[c0 + m];
                if (gt) y *= act_sigmoid<Tio>(to_f(gt[m]));
                dst[m] = from_f<To>(y);
            }
        }
    }
    if (tid == 0) {
        tc::bulk_wait_all();
        if (failed) flag_status(d_status, KDA_ERR_TIMEOUT);
    }
    __syncthreads();
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

template <typename Tio, typename To>
cudaError_t decode_tma_launch(const kda_decode_args& a, cudaStream_t s) {
    using St = DecodeStage<Tio>;
    DeviceInfo dinfo;
    const int sms = current_device_info(&dinfo) ? dinfo.sm_count : 148;
    const int units = a.N * a.H;
    auto kern = k_decode_tma<Tio, To>;
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)St::kSmem);
    if (e != cudaSuccess) return e;
    const int64_t xs = a.qkv_row_stride ? a.qkv_row_stride : (int64_t)a.H * 128;
    kern<<<units < sms ? units : sms, 256, St::kSmem, s>>>(
        (const Tio*)a.q, (const Tio*)a.k, (const Tio*)a.v, xs, (const Tio*)a.gate, a.g, a.beta, a.conv_w,
        a.rms_w, a.eps_l2, a.eps_rms, a.scale, a.H, units, a.state, (Tio*)a.conv_state, (To*)a.out,
        a.d_status);
    return cudaGetLastError();
}

template <typename Tio>
bool decode_tma_ok(const kda_decode_args& a) {
    const int64_t xs = a.qkv_row_stride ? a.qkv_row_stride : (int64_t)a.H * 128;
    return a.D == 128 && (xs * (int64_t)sizeof(Tio)) % 16 == 0 && aligned16(a.q) && aligned16(a.k) &&
           aligned16(a.v) && aligned16(a.g) && aligned16(a.state) && aligned16(a.conv_state) &&
           aligned16(a.conv_w) &&
           (!a.gate || aligned16(a.gate)) && (int64_t)a.N * a.H < 0x7fffffffLL;
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
    if (D == 128 && a.io == KDA_BF16 && decode_tma_ok<bf16>(a))
        return a.out_dtype == KDA_FP32 ? decode_tma_launch<bf16, float>(a, s) : decode_tma_launch<bf16, bf16>(a, s);
    if (D == 128 && a.io == KDA_FP32 && decode_tma_ok<float>(a))
        return a.out_dtype == KDA_FP32 ? decode_tma_launch<float, float>(a, s) : decode_tma_launch<float, bf16>(a, s);
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
