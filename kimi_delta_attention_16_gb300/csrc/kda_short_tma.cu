// kda_short_tma.cu -- the recurrent path of kda_prefill for batches of short
// sequences (every sequence at most kShortMaxL tokens: multi-token decode and
// speculative verification) as a pipelined, memory-bound kernel.
//
// Page "Animated Kimi K3 architecture diagram", section "LOCAL MEMORY: A
// FIXED MATRIX THAT PREDICTS, FORGETS, AND CORRECTS": per token, DECAY
// S_bar = Diag(alpha_t) S, PROBE/CORRECT e = v - S_bar^T k, WRITE
// S = S_bar + beta k e^T; page "Kimi K3 / Architecture": the short conv with its
// rolling window of the last three raw values, the read o = S^T q, the head
// RMSNorm and the sigmoid output gate.
//
// A unit is one (sequence, head); its bytes are the 64 KB fp32 state in and
// out, the rolling conv window in and out and a few token rows, so the path is
// bound by HBM.  Persistent CTAs (one per SM, 256 threads) walk contiguous
// head-major ranges of units.  Each unit's state and conv window (1D bulk
// copies) and its token rows (one 2D tensor-map box of Lmax rows for each of
// q, k, v, gate and g) land in one of two shared-memory stages by the TMA
// engine, with mbarrier completion.  The state moves into registers at the
// start of the unit and its rows are converted into working arrays, so the
// stage is refilled with the unit after next while this one computes: two
// units' loads are in flight behind every unit's compute.  The state leaves
// from registers with coalesced stores.
//
// Thread (row group = warp, column group = lane) holds rows 16 w .. 16 w + 15
// of columns 4 l .. 4 l + 3.  One CTA barrier per token: the readout of token
// t - 1 (S_{t-1}^T q) and the decay and probe of token t (S_bar_t^T k) share
// one pass over the state registers and go through double-buffered row-group
// partials; warp (t - 1) mod 8 finishes token t - 1's output (RMSNorm, gate)
// after that barrier.
#include "kda_internal.cuh"
#include "kda_tc.cuh"
#include "kda_tc_ptx.cuh"

namespace kda {

namespace {

constexpr int kD = 128;
constexpr int kThreads = 256;
constexpr int kL8 = kShortMaxL;

__host__ __device__ constexpr uint32_t align128(uint32_t x) { return (x + 127u) & ~127u; }

// Byte offsets inside one stage for boxes of Lmax token rows.
template <typename Tio>
struct TmaStage {
    uint32_t conv, rows, part, g, bytes;
    __host__ __device__ explicit TmaStage(int Lmax) {
        conv = 65536;                                                     // [3][128][3] Tio
        rows = conv + align128(3 * kD * 3 * (uint32_t)sizeof(Tio));      // [4][Lmax][128] Tio: q, k, v, gate
        part = (uint32_t)Lmax * kD * (uint32_t)sizeof(Tio);
        g = rows + align128(4 * part);                                    // [Lmax][128] fp32
        bytes = g + align128((uint32_t)Lmax * kD * 4);
    }
};

// Tensor maps of the token rows: [T rows][H * 128 columns], boxes of 128 columns x Lmax rows.
struct ShortMaps {
    CUtensorMap q, k, v, gate, g;
};

__device__ __forceinline__ void tma_load_2d(uint32_t dst, const CUtensorMap* map, int x, int y, uint64_t* bar) {
    asm volatile(
        "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes [%0], [%1, {%2, %3}], [%4];" ::
            "r"(dst), "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y), "r"(tc::smem_u32(bar))
        : "memory");
}
// 4 bytes, of which the first src_bytes come from global memory and the rest are zero
__device__ __forceinline__ void cp_async4_zfill(uint32_t dst, const void* src, uint32_t src_bytes) {
    asm volatile("cp.async.ca.shared.global [%0], [%1], 4, %2;" ::"r"(dst), "l"(src), "r"(src_bytes) : "memory");
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }
__device__ __forceinline__ void cp_async_wait_all() { asm volatile("cp.async.wait_group 0;" ::: "memory"); }

__device__ __forceinline__ void fma4(float4& acc, float a, const float4& x) {
    acc.x = fmaf(a, x.x, acc.x);
    acc.y = fmaf(a, x.y, acc.y);
    acc.z = fmaf(a, x.z, acc.z);
    acc.w = fmaf(a, x.w, acc.w);
}

template <typename To>
__device__ __forceinline__ void store4(To* p, float a, float b, float c, float d);
template <>
__device__ __forceinline__ void store4<float>(float* p, float a, float b, float c, float d) {
    *reinterpret_cast<float4*>(p) = make_float4(a, b, c, d);
}
template <>
__device__ __forceinline__ void store4<bf16>(bf16* p, float a, float b, float c, float d) {
    *reinterpret_cast<uint2*>(p) = make_uint2(pack_bf16x2(a, b), pack_bf16x2(c, d));
}

template <typename Tio, typename To>
__global__ void __launch_bounds__(kThreads, 1)
k_short_tma(const __grid_constant__ ShortMaps maps, int Lmax, int has_gate, const Tio* __restrict__ cs_in,
            Tio* __restrict__ cs_out, const float* __restrict__ beta, const float* __restrict__ conv_w,
            const float* __restrict__ rms_w, float eps_l2, float eps_rms, float scale, int N, int H,
            const int32_t* __restrict__ cu, int64_t T_total, const float* S0, float* S_fin,
            To* __restrict__ out, int* d_status) {
    extern __shared__ uint8_t smem_raw[];
    __shared__ uint64_t bars[2];
    __shared__ __align__(16) float sx[kL8][3][kD];     // convolved q, k, v of every token
    __shared__ __align__(16) float salpha[kL8][kD];    // e^g of every token
    __shared__ __align__(16) float sgate[kL8][kD];     // sigmoid(gate) of every token (1 without a gate)
    __shared__ __align__(16) float sredP[2][8][kD];    // probe partials per row group, by token parity
    __shared__ __align__(16) float sredO[2][8][kD];    // readout partials per row group, by token parity
    __shared__ __align__(16) float sW[3 * kD * 4];     // conv taps of the current head
    __shared__ __align__(16) float sRms[kD];
    __shared__ float snorm[kL8][2];                    // 1/|q|, 1/|k| per token
    __shared__ float sbeta[2][kL8];                    // betas per unit parity

    const TmaStage<Tio> ST(Lmax);
    const uint32_t raw_addr = tc::smem_u32(smem_raw);
    uint8_t* sm = smem_raw + (((raw_addr + 127u) & ~127u) - raw_addr);
    const uint32_t sbase = tc::smem_u32(sm);
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int r0 = 16 * warp, c0 = 4 * lane;
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
    const uint32_t cs_bytes = 3u * kD * 3u * (uint32_t)sizeof(Tio);
    const uint32_t tx = (S0 ? 65536u : 0u) + (cs_in ? cs_bytes : 0u) + (has_gate ? 4u : 3u) * ST.part +
                        (uint32_t)Lmax * kD * 4u;

    if (tid == 0) {
        tc::mbar_init(&bars[0], 1);
        tc::mbar_init(&bars[1], 1);
        tc::fence_mbar_init();
    }
    for (int c = tid; c < kD; c += kThreads) sRms[c] = rms_w ? rms_w[c] : 1.f;
    __syncthreads();

    // Loads of this CTA's unit i into stage i & 1 (thread 0).  `pend` bit b: a fill of stage b
    // is in flight (its phase parity in bit 2 + b), for the exit path.
    uint32_t pend = 0;
    auto issue = [&](int i) {
        const int b = i & 1;
        int n, h;
        unit_of(i, n, h);
        int64_t a, e;
        seq_range(cu, n, T_total, a, e);
        const uint32_t st = sbase + (uint32_t)b * ST.bytes;
        tc::mbar_expect_tx(&bars[b], tx);
        if (S0) tc::bulk_load(st, S0 + ((int64_t)n * H + h) * kD * kD, 65536u, &bars[b]);
        if (cs_in)
            for (int p = 0; p < 3; ++p)
                tc::bulk_load(st + ST.conv + (uint32_t)p * (cs_bytes / 3u),
                              cs_in + (((int64_t)n * 3 + p) * HD + (int64_t)h * kD) * 3, cs_bytes / 3u, &bars[b]);
        const int x = h * kD, y = (int)a;
        tma_load_2d(st + ST.rows, &maps.q, x, y, &bars[b]);
        tma_load_2d(st + ST.rows + ST.part, &maps.k, x, y, &bars[b]);
        tma_load_2d(st + ST.rows + 2 * ST.part, &maps.v, x, y, &bars[b]);
        if (has_gate) tma_load_2d(st + ST.rows + 3 * ST.part, &maps.gate, x, y, &bars[b]);
        tma_load_2d(st + ST.g, &maps.g, x, y, &bars[b]);
        pend = (pend & ~(5u << b)) | ((1u | ((uint32_t)((i >> 1) & 1) << 2)) << b);
    };
    // betas of unit i -> sbeta[i & 1] (lanes 0..7 of warp 1, cp.async; zeros past the sequence)
    auto stage_beta = [&](int i) {
        int n, h;
        unit_of(i, n, h);
        int64_t a, e;
        seq_range(cu, n, T_total, a, e);
        const bool ok = lane < e - a;
        cp_async4_zfill(tc::smem_u32(&sbeta[i & 1][lane]), ok ? beta + (a + lane) * H + h : beta, ok ? 4u : 0u);
        cp_async_commit();
    };
    if (tid == 0) {
        if (my_units > 0) issue(0);
        if (my_units > 1) issue(1);
    }
    if (warp == 1 && lane < kL8 && my_units > 0) stage_beta(0);

    bool failed = false;
    int h_prev = -1;
    for (int i = 0; i < my_units; ++i) {
        const int b = i & 1;
        int n, h;
        unit_of(i, n, h);
        const int u = n * H + h;
        int64_t a, e;
        seq_range(cu, n, T_total, a, e);
        int L = (int)(e - a);
        if (L > Lmax) {  // the device cu_seqlens disagrees with the host copy that sized the boxes
            if (tid == 0) flag_status(d_status, KDA_ERR_DEVICE_ARG);
            L = Lmax;
        }
        // ---- A: this unit's stage has landed; conv taps of a new head
        bool ok = true;
        if (warp == 0) ok = tc::mbar_wait(&bars[b], (uint32_t)((i >> 1) & 1));
        if (tid == 0) pend &= ~(1u << b);
        if (warp == 1) cp_async_wait_all();
        if (h != h_prev)
            for (int idx = tid; idx < 3 * kD * 4; idx += kThreads) {
                const int part = idx / (kD * 4), rem = idx % (kD * 4);
                sW[idx] = conv_w[(part * HD + (int64_t)h * kD) * 4 + rem];
            }
        h_prev = h;
        if (__syncthreads_or(!ok)) {
            failed = true;
            break;
        }
        const uint8_t* st = sm + (uint32_t)b * ST.bytes;
        // the state into registers
        float4 s[16];
        {
            const float* Ss = reinterpret_cast<const float*>(st);
#pragma unroll
            for (int r = 0; r < 16; ++r)
                s[r] = S0 ? *reinterpret_cast<const float4*>(Ss + (r0 + r) * kD + c0) : make_float4(0.f, 0.f, 0.f, 0.f);
        }
        // conv + SiLU of every token, one channel per thread and step; the rolled window out
        for (int ch = tid; ch < 3 * kD; ch += kThreads) {
            const int part = ch >> 7, d = ch & (kD - 1);
            float p0 = 0.f, p1 = 0.f, p2 = 0.f;  // x[-3], x[-2], x[-1]
            if (cs_in) {
                const Tio* c3 = reinterpret_cast<const Tio*>(st + ST.conv) + ch * 3;
                p0 = to_f(c3[0]);
                p1 = to_f(c3[1]);
                p2 = to_f(c3[2]);
            }
            const Tio* rp = reinterpret_cast<const Tio*>(st + ST.rows + (uint32_t)part * ST.part) + d;
            const float4 w = *reinterpret_cast<const float4*>(&sW[ch * 4]);
            for (int t = 0; t < L; ++t) {
                const float x = to_f(rp[t * kD]);
                sx[t][part][d] = act_silu<Tio>(w.x * p0 + w.y * p1 + w.z * p2 + w.w * x);
                p0 = p1;
                p1 = p2;
                p2 = x;
            }
            if (cs_out) {  // last three raw values of the sequence (exact copies of Tio values)
                Tio* o3 = cs_out + (((int64_t)n * 3 + part) * HD + (int64_t)h * kD + d) * 3;
                o3[0] = from_f<Tio>(p0);
                o3[1] = from_f<Tio>(p1);
                o3[2] = from_f<Tio>(p2);
            }
        }
        {  // decay factors and gate sigmoids of every token
            const float* gs = reinterpret_cast<const float*>(st + ST.g);
            const Tio* gt = reinterpret_cast<const Tio*>(st + ST.rows + 3 * ST.part);
            for (int idx = tid; idx < L * kD; idx += kThreads) {
                const int t = idx >> 7, c = idx & (kD - 1);
                salpha[t][c] = decay_exp<Tio>(gs[idx]);
                sgate[t][c] = has_gate ? act_sigmoid<Tio>(to_f(gt[idx])) : 1.f;
            }
        }
        __syncthreads();  // B: stage b is read completely
        if (tid == 0 && i + 2 < my_units) issue(i + 2);
        if (warp == 1 && lane < kL8 && i + 1 < my_units) stage_beta(i + 1);
        // L2 norms of q and k, one vector per warp and step
        for (int vv = warp; vv < 2 * L; vv += kThreads / 32) {
            const int t = vv >> 1, which = vv & 1;
            const float4 x4 = *reinterpret_cast<const float4*>(&sx[t][which][c0]);
            float ss = x4.x * x4.x + x4.y * x4.y + x4.z * x4.z + x4.w * x4.w;
#pragma unroll
            for (int off = 16; off > 0; off >>= 1) ss += __shfl_xor_sync(0xffffffffu, ss, off);
            if (lane == 0) snorm[t][which] = 1.0f / sqrtf(ss + eps_l2);
        }
        __syncthreads();  // C

        // warp-level output of token t: o = scale S_t^T q / |q| from the readout partials, RMSNorm,
        // weight, gate, 4 columns per lane
        auto emit = [&](int t) {
            const float(*po)[kD] = sredO[t & 1];
            float4 o = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
            for (int w = 0; w < 8; ++w) {
                const float4 x = *reinterpret_cast<const float4*>(&po[w][c0]);
                o.x += x.x;
                o.y += x.y;
                o.z += x.z;
                o.w += x.w;
            }
            const float sq = snorm[t][0] * scale;
            o.x *= sq;
            o.y *= sq;
            o.z *= sq;
            o.w *= sq;
            float ss = o.x * o.x + o.y * o.y + o.z * o.z + o.w * o.w;
#pragma unroll
            for (int off = 16; off > 0; off >>= 1) ss += __shfl_xor_sync(0xffffffffu, ss, off);
            const float inv = 1.0f / sqrtf(ss * (1.0f / kD) + eps_rms);
            const float4 rw = *reinterpret_cast<const float4*>(&sRms[c0]);
            const float4 gg = *reinterpret_cast<const float4*>(&sgate[t][c0]);
            store4<To>(out + ((a + t) * H + h) * kD + c0, o.x * inv * rw.x * gg.x, o.y * inv * rw.y * gg.y,
                       o.z * inv * rw.z * gg.z, o.w * inv * rw.w * gg.w);
        };

        // ---- token loop: one barrier per token
        float kr[16];
        for (int t = 0; t < L; ++t) {
            const int buf = t & 1;
            float4 p = make_float4(0.f, 0.f, 0.f, 0.f), po = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
            for (int e4 = 0; e4 < 4; ++e4) {
                const float4 k4 = *reinterpret_cast<const float4*>(&sx[t][1][r0 + 4 * e4]);
                const float4 a4 = *reinterpret_cast<const float4*>(&salpha[t][r0 + 4 * e4]);
                const float kk[4] = {k4.x, k4.y, k4.z, k4.w}, aa[4] = {a4.x, a4.y, a4.z, a4.w};
                float qq[4] = {0.f, 0.f, 0.f, 0.f};
                if (t > 0) {
                    const float4 q4 = *reinterpret_cast<const float4*>(&sx[t - 1][0][r0 + 4 * e4]);
                    qq[0] = q4.x;
                    qq[1] = q4.y;
                    qq[2] = q4.z;
                    qq[3] = q4.w;
                }
#pragma unroll
                for (int m = 0; m < 4; ++m) {
                    float4& sv = s[4 * e4 + m];
                    fma4(po, qq[m], sv);  // readout of token t - 1, before this token's decay
                    sv.x *= aa[m];
                    sv.y *= aa[m];
                    sv.z *= aa[m];
                    sv.w *= aa[m];
                    fma4(p, kk[m], sv);
                    kr[4 * e4 + m] = kk[m];
                }
            }
            *reinterpret_cast<float4*>(&sredP[buf][warp][c0]) = p;
            if (t > 0) *reinterpret_cast<float4*>(&sredO[buf ^ 1][warp][c0]) = po;
            __syncthreads();
            // e = v - S_bar^T k / |k| for this thread's columns; the write takes beta e / |k|
            float4 pv = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
            for (int w = 0; w < 8; ++w) {
                const float4 x = *reinterpret_cast<const float4*>(&sredP[buf][w][c0]);
                pv.x += x.x;
                pv.y += x.y;
                pv.z += x.z;
                pv.w += x.w;
            }
            const float ik = snorm[t][1], bk = sbeta[b][t] * ik;
            const float4 v4 = *reinterpret_cast<const float4*>(&sx[t][2][c0]);
            const float4 ev = make_float4(bk * (v4.x - pv.x * ik), bk * (v4.y - pv.y * ik), bk * (v4.z - pv.z * ik),
                                          bk * (v4.w - pv.w * ik));
#pragma unroll
            for (int r = 0; r < 16; ++r) fma4(s[r], kr[r], ev);
            if (t > 0 && warp == ((t - 1) & 7)) emit(t - 1);
        }
        if (L > 0) {  // readout of the last token
            float4 po = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
            for (int e4 = 0; e4 < 4; ++e4) {
                const float4 q4 = *reinterpret_cast<const float4*>(&sx[L - 1][0][r0 + 4 * e4]);
                fma4(po, q4.x, s[4 * e4]);
                fma4(po, q4.y, s[4 * e4 + 1]);
                fma4(po, q4.z, s[4 * e4 + 2]);
                fma4(po, q4.w, s[4 * e4 + 3]);
            }
            *reinterpret_cast<float4*>(&sredO[(L - 1) & 1][warp][c0]) = po;
            __syncthreads();
            if (warp == ((L - 1) & 7)) emit(L - 1);
        }
        if (S_fin) {
            float* dst = S_fin + (int64_t)u * kD * kD;
#pragma unroll
            for (int r = 0; r < 16; ++r) *reinterpret_cast<float4*>(dst + (r0 + r) * kD + c0) = s[r];
        }
    }
    // fills still in flight (a wait above timed out): wait for them, bounded, before exiting
    if (tid == 0)
        for (int b = 0; b < 2; ++b)
            if ((pend >> b) & 1u) tc::mbar_wait(&bars[b], (pend >> (2 + b)) & 1u);
    cp_async_wait_all();
    if (failed && tid == 0) flag_status(d_status, KDA_ERR_TIMEOUT);
}

template <typename Tio>
uint32_t short_tma_smem(int Lmax) {
    return 2 * TmaStage<Tio>(Lmax).bytes + 128;
}

int max_len(const kda_prefill_args& a) {
    int m = 0;
    for (int n = 0; n < a.N; ++n) {
        const int L = a.cu_seqlens_host[n + 1] - a.cu_seqlens_host[n];
        m = L > m ? L : m;
    }
    return m;
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

template <typename Tio, typename To>
cudaError_t short_tma_launch(const kda_prefill_args& a, cudaStream_t s) {
    const int Lmax = max_len(a) > 0 ? max_len(a) : 1;
    const uint32_t smem = short_tma_smem<Tio>(Lmax);
    auto kern = k_short_tma<Tio, To>;
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
    const int64_t xs = a.qkv_row_stride ? a.qkv_row_stride : (int64_t)a.H * kD;
    const bool fp32 = a.io == KDA_FP32;
    const uint64_t cols = (uint64_t)a.H * kD, rows = (uint64_t)a.T_total, es = fp32 ? 4 : 2;
    ShortMaps maps;
    memset(&maps, 0, sizeof(maps));  // the gate map stays unused without a gate
    bool ok = encode_tensor_map_2d(&maps.q, a.q, fp32, cols, rows, (uint64_t)xs * es, kD, (uint32_t)Lmax, false) &&
              encode_tensor_map_2d(&maps.k, a.k, fp32, cols, rows, (uint64_t)xs * es, kD, (uint32_t)Lmax, false) &&
              encode_tensor_map_2d(&maps.v, a.v, fp32, cols, rows, (uint64_t)xs * es, kD, (uint32_t)Lmax, false) &&
              encode_tensor_map_2d(&maps.g, a.g, true, cols, rows, cols * 4, kD, (uint32_t)Lmax, false);
    if (ok && a.gate) ok = encode_tensor_map_2d(&maps.gate, a.gate, fp32, cols, rows, cols * es, kD, (uint32_t)Lmax, false);
    if (!ok) return cudaErrorInvalidValue;
    DeviceInfo d;
    const int sms = current_device_info(&d) ? d.sm_count : 148;
    const int units = a.N * a.H;
    kern<<<units < sms ? units : sms, kThreads, smem, s>>>(
        maps, Lmax, a.gate ? 1 : 0, (const Tio*)a.conv_state_in, (Tio*)a.conv_state_out, a.beta, a.conv_w, a.rms_w,
        a.eps_l2, a.eps_rms, a.scale, a.N, a.H, a.cu_seqlens, a.T_total, a.initial_state, a.final_state, (To*)a.out,
        a.d_status);
    return cudaGetLastError();
}

}  // namespace

bool short_tma_applies(const kda_prefill_args& a) {
    if (a.D != kD || a.T_total <= 0 || !a.cu_seqlens_host || a.N < 1) return false;
    const int64_t xs = a.qkv_row_stride ? a.qkv_row_stride : (int64_t)a.H * kD;
    const int64_t es = a.io == KDA_BF16 ? 2 : 4;
    if ((xs * es) % 16 || !aligned16(a.q) || !aligned16(a.k) || !aligned16(a.v) || !aligned16(a.g) ||
        (a.gate && !aligned16(a.gate)) || (a.conv_state_in && !aligned16(a.conv_state_in)) ||
        (a.initial_state && !aligned16(a.initial_state)) || (a.final_state && !aligned16(a.final_state)) ||
        (a.out && !aligned16(a.out)))
        return false;
    const int Lmax = max_len(a);
    if (Lmax > kShortMaxL) return false;
    const uint32_t smem = a.io == KDA_BF16 ? short_tma_smem<bf16>(Lmax > 0 ? Lmax : 1)
                                           : short_tma_smem<float>(Lmax > 0 ? Lmax : 1);
    return smem <= 232448u - 48u * 1024u;  // dynamic stages + the kernel's static arrays
}

cudaError_t launch_short_tma(const kda_prefill_args& a, cudaStream_t s) {
    if ((int64_t)a.N * a.H == 0) return cudaSuccess;
    if (a.io == KDA_BF16)
        return a.out_dtype == KDA_FP32 ? short_tma_launch<bf16, float>(a, s) : short_tma_launch<bf16, bf16>(a, s);
    return a.out_dtype == KDA_FP32 ? short_tma_launch<float, float>(a, s) : short_tma_launch<float, bf16>(a, s);
}

}  // namespace kda
