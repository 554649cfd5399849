// kda_backward.cu -- the backward pass of the KDA layer (training): reverse-mode
// derivatives of sum(dy . out) + sum(dS . final_state) with respect to every
// input of kda_prefill, D = 128, fp32 arithmetic (IEEE exp, SiLU, sigmoid).
//
// Page "Kimi K3 / Architecture", KDA panel (the layer: short conv + SiLU, L2
// norms of q and k, the recurrent state decayed, corrected and written per
// token, the readout S_t^T q_t, head RMSNorm and the sigmoid gate) and the
// page's training material (the model is trained, so the layer needs its
// derivatives); page "Animated Kimi K3 architecture diagram", LOCAL MEMORY
// section (the four moves, each an affine map of the state, whose adjoints run
// the same steps backwards).
//
// Per (sequence, head) unit, with P_t = Diag(alpha_t) S_{t-1}, e_t = v_t - P_t^T k_t,
// S_t = P_t + beta_t k_t e_t^T, o_t = scale S_t^T q_t:
//   prep      conv + SiLU + L2 norms: q^, k^, v (fp32) and |a_q|, |a_k|      (warp per token-head)
//   forward   the recurrence in column layout (each value column of S evolves on its own):
//             o_t, e_t, and S at the start of every kSeg-token segment          (4 CTAs per unit)
//   epilogue  y = n w sig(z), n = o r:  do = r dn - r^3 o (dn . o) / D, dgate, drms_w  (warp per row)
//   backward  the state gradient in column layout, tokens in reverse (each column of dS evolves
//             on its own): w_t = dS'^T k, dv = beta w, dbeta = w . e, e . do, and dS at the end
//             of every segment                                                  (4 CTAs per unit)
//   rows      per (unit, segment), all in parallel, row layout (with e, w and do known, each row
//             of S and of dS evolves on its own): dq, dk and dg (see k_bwd_rows)
//   carry     dg's sums over later segments and the final-state term
//   L2        da = (dx - x (x . dx)) / |a|, in place; dg += carry                 (warp per row)
//   conv      du = da sig(u) (1 + u (1 - sig(u))); dx, the taps' and the conv state's gradients
// No token's state is stored: the row kernels replay at most kSeg tokens from the checkpoints.
#include "kda_internal.cuh"

namespace kda {

namespace {

constexpr int kD = 128;
constexpr int kSeg = kBwdSeg;  // tokens per checkpointed segment

__device__ __forceinline__ float4 f4_fma(float a, float4 x, float4 y) {
    return make_float4(fmaf(a, x.x, y.x), fmaf(a, x.y, y.y), fmaf(a, x.z, y.z), fmaf(a, x.w, y.w));
}
__device__ __forceinline__ float4 f4_mul(float a, float4 x) { return make_float4(a * x.x, a * x.y, a * x.z, a * x.w); }
__device__ __forceinline__ float4 f4_add(float4 x, float4 y) { return make_float4(x.x + y.x, x.y + y.y, x.z + y.z, x.w + y.w); }
__device__ __forceinline__ float dot4(float4 x, float4 y) { return x.x * y.x + x.y * y.y + x.z * y.z + x.w * y.w; }
__device__ __forceinline__ float warp_sum(float v) {
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) v += __shfl_xor_sync(0xffffffffu, v, off);
    return v;
}
// Four consecutive inputs as floats (one 8-byte or 16-byte load).
__device__ __forceinline__ void load4(const bf16* p, float (&x)[4]) {
    const uint2 u = *reinterpret_cast<const uint2*>(p);
    x[0] = __uint_as_float(u.x << 16);
    x[1] = __uint_as_float(u.x & 0xffff0000u);
    x[2] = __uint_as_float(u.y << 16);
    x[3] = __uint_as_float(u.y & 0xffff0000u);
}
__device__ __forceinline__ void load4(const float* p, float (&x)[4]) {
    const float4 f = *reinterpret_cast<const float4*>(p);
    x[0] = f.x;
    x[1] = f.y;
    x[2] = f.z;
    x[3] = f.w;
}

// ------------------------------------------------------------------------------ prep
// One warp per (token, head): conv + SiLU of the q, k, v channels of the head (lane l: channels
// 4 l .. 4 l + 3), the L2 norms of q and k.  X: [T][3][H][D] fp32 (q^, k^, v), nrm: [T][H][2].
template <typename Tio>
__global__ void k_bwd_prep(const Tio* __restrict__ q, const Tio* __restrict__ k, const Tio* __restrict__ v,
                           int64_t xs, const float* __restrict__ conv_w, const Tio* __restrict__ cs_in,
                           const int32_t* __restrict__ cu, int N, int64_t T_total, int H, float eps_l2,
                           float* __restrict__ X, float* __restrict__ nrm) {
    const int64_t row = (int64_t)blockIdx.x * (blockDim.x / 32) + (threadIdx.x >> 5);
    const int lane = threadIdx.x & 31;
    if (row >= T_total * H) return;
    const int64_t t = row / H;
    const int h = (int)(row % H);
    // the sequence of token t (binary search over cu_seqlens)
    int lo = 0, hi = N;
    while (hi - lo > 1) {
        const int mid = (lo + hi) >> 1;
        if (cu[mid] <= t) lo = mid;
        else hi = mid;
    }
    const int n = lo;
    int64_t s0 = cu[n];
    s0 = s0 < 0 ? 0 : (s0 > t ? t : s0);  // keeps every index in bounds if cu is inconsistent
    const int64_t HD = (int64_t)H * kD;
    const Tio* src[3] = {q, k, v};
    float out[3][4];
    float ss[2] = {0.f, 0.f};
#pragma unroll
    for (int part = 0; part < 3; ++part) {
        // the raw inputs of the lane's 4 channels at t - 3 .. t: one vector load per token
        float x[4][4];  // [token j][channel m]
#pragma unroll
        for (int j = 0; j < 4; ++j) {
            const int64_t p = t - 3 + j;
            if (p >= s0) {
                load4(src[part] + p * xs + (int64_t)h * kD + 4 * lane, x[j]);
            } else {
#pragma unroll
                for (int m = 0; m < 4; ++m) {
                    const int64_t ch = (int64_t)part * HD + (int64_t)h * kD + 4 * lane + m;
                    x[j][m] = cs_in ? to_f(cs_in[((int64_t)n * 3 * HD + ch) * 3 + 3 + (p - s0)]) : 0.f;
                }
            }
        }
#pragma unroll
        for (int m = 0; m < 4; ++m) {
            const int64_t ch = (int64_t)part * HD + (int64_t)h * kD + 4 * lane + m;
            const float4 w = *reinterpret_cast<const float4*>(conv_w + ch * 4);
            const float u = w.x * x[0][m] + w.y * x[1][m] + w.z * x[2][m] + w.w * x[3][m];
            out[part][m] = u / (1.0f + expf(-u));
            if (part < 2) ss[part] += out[part][m] * out[part][m];
        }
    }
    const float nq = sqrtf(warp_sum(ss[0]) + eps_l2), nk = sqrtf(warp_sum(ss[1]) + eps_l2);
    float* xr = X + t * 3 * HD + (int64_t)h * kD + 4 * lane;
    *reinterpret_cast<float4*>(xr) = make_float4(out[0][0] / nq, out[0][1] / nq, out[0][2] / nq, out[0][3] / nq);
    *reinterpret_cast<float4*>(xr + HD) = make_float4(out[1][0] / nk, out[1][1] / nk, out[1][2] / nk, out[1][3] / nk);
    *reinterpret_cast<float4*>(xr + 2 * HD) = make_float4(out[2][0], out[2][1], out[2][2], out[2][3]);
    if (lane == 0) *reinterpret_cast<float2*>(nrm + row * 2) = make_float2(nq, nk);
}

// ------------------------------------------------------------------------------ staging helpers
// 16-byte and 4-byte asynchronous global -> shared copies (cp.async), one group per staged block.
__device__ __forceinline__ void cp16(void* dst, const void* src) {
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"((uint32_t)__cvta_generic_to_shared(dst)),
                 "l"(src)
                 : "memory");
}
__device__ __forceinline__ void cp4(void* dst, const void* src) {
    asm volatile("cp.async.ca.shared.global [%0], [%1], 4;" ::"r"((uint32_t)__cvta_generic_to_shared(dst)),
                 "l"(src)
                 : "memory");
}
__device__ __forceinline__ void cp_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }
template <int N>
__device__ __forceinline__ void cp_wait() {
    asm volatile("cp.async.wait_group %0;" ::"n"(N) : "memory");
}

// First checkpoint slot of unit (n, h): sequences in order, each holding H runs of its segment
// count (prefix[n] = segments of the sequences before n).  -1 when the unit's slots would end
// past `slots` (the host planned the layout from its copy of cu_seqlens; a device copy that
// disagrees must not send accesses out of the workspace).
__device__ __forceinline__ int64_t slot_base(const int64_t* prefix, int n, int H, int h, int64_t nseg,
                                             int64_t slots) {
    const int64_t base = prefix[n] * H + (int64_t)h * nseg;
    return (base >= 0 && base + nseg <= slots) ? base : -1;
}

// prefix[n] = sum over sequences m < n of ceil(len_m / kSeg), n = 0..N.  One block of 256.
__global__ void k_bwd_seg_prefix(const int32_t* __restrict__ cu, int N, int64_t T_total,
                                 int64_t* __restrict__ prefix) {
    __shared__ int64_t part[256];
    const int tid = threadIdx.x;
    const int per = (N + 255) / 256;
    const int a = tid * per < N ? tid * per : N, b = a + per < N ? a + per : N;
    int64_t sum = 0;
    for (int n = a; n < b; ++n) {
        int64_t s0, s1;
        seq_range(cu, n, T_total, s0, s1);
        sum += (s1 - s0 + kSeg - 1) / kSeg;
    }
    part[tid] = sum;
    __syncthreads();
    if (tid == 0) {
        int64_t run = 0;
        for (int i = 0; i < 256; ++i) {
            const int64_t x = part[i];
            part[i] = run;
            run += x;
        }
        prefix[N] = run;
    }
    __syncthreads();
    int64_t run = part[tid];
    for (int n = a; n < b; ++n) {
        prefix[n] = run;
        int64_t s0, s1;
        seq_range(cu, n, T_total, s0, s1);
        run += (s1 - s0 + kSeg - 1) / kSeg;
    }
}

// ------------------------------------------------------------------------------ column-layout sweeps
// One unit's state is split by value column over kColCtas CTAs of 4 warps (32 columns each).
// Lane l of warp w owns rows 8 r .. 8 r + 7 (r = l & 15) of the four columns
// c0 = 32 cq + 8 w + 4 (l >> 4) .. c0 + 3.  A
// per-column quantity of a token (e, o, w = dS^T k) is a sum over the rows of its column: the
// sixteen lanes of a column group.  Every (unit, column group) is an independent chain, and the
// CTAs of all units stay resident together (ten warps per SM at 96 units).  Each token is one pass over the state: the forward sweep
// finishes token t's update, accumulates o_t and the next token's S^T (alpha k) together; the
// backward sweep applies the later token's decay and correction, adds token t's readout gradient
// and accumulates w_t together.  No CTA barrier inside a token; tokens are staged kTB at a time
// (double-buffered cp.async), three barriers per block.
constexpr int kColCtas = 4;           // CTAs per unit
constexpr int kCols = kD / kColCtas;  // 32 columns per CTA
constexpr int kTB = 8;                // tokens per staged block
constexpr int kSlice = 12;            // floats between the 8-row slices of a staged 128-vector
constexpr int kPerm = 16 * kSlice;
__device__ __forceinline__ int perm_off(int row) { return (row >> 3) * kSlice + (row & 7); }

// One staged token: k^, exp(g), q^, exp(g) k^ (8-row slices 12 floats apart, so that the eight
// slices a quarter-warp reads at once fall in distinct banks), two slices of the CTA's columns, beta.
struct ColTok {
    float k[kPerm], a[kPerm], q[kPerm], ak[kPerm];
    float c0[kCols], c1[kCols];  // forward sweep: v; backward sweep: do and e
    float beta, pad[3];
};
constexpr int kColSmem = 2 * kTB * (int)sizeof(ColTok);

struct ColSrc {
    const float* p;  // element (token 0, head 0, channel 0)
    int64_t stride;  // elements between tokens
};

// Issues the copies of tokens [t0, t0 + nt) of head h into st[0 .. nt): the three row vectors
// (q^ and k^ from X, g into the alpha slot), `ncs` column slices (the CTA's columns), beta.
__device__ __forceinline__ void stage_cols(ColTok* st, int64_t t0, int nt, const float* X, const float* g,
                                           const float* beta, ColSrc s0, ColSrc s1, int ncs, int H, int h,
                                           int cq, int tid) {
    constexpr int kCC = kCols / 4;  // 16-byte chunks of one column slice
    const int64_t HD = (int64_t)H * kD;
    const int per = 96 + kCC * ncs + 1;
    for (int idx = tid; idx < nt * per; idx += 128) {
        const int tk = idx / per, j = idx - tk * per;
        const int64_t t = t0 + tk;
        ColTok& s = st[tk];
        if (j < 96) {
            const int part = j >> 5, jj = j & 31;
            const float* src = part == 0 ? X + t * 3 * HD + HD + (int64_t)h * kD
                             : part == 1 ? g + (t * H + h) * kD
                                         : X + t * 3 * HD + (int64_t)h * kD;
            float* dst = part == 0 ? s.k : part == 1 ? s.a : s.q;
            cp16(dst + (jj >> 1) * kSlice + (jj & 1) * 4, src + jj * 4);
        } else if (j < 96 + kCC * ncs) {
            const int jj = j - 96, which = jj / kCC, ch = jj - which * kCC;
            const ColSrc& cs = which == 0 ? s0 : s1;
            cp16((which == 0 ? s.c0 : s.c1) + ch * 4, cs.p + t * cs.stride + (int64_t)h * kD + cq * kCols + ch * 4);
        } else {
            cp4(&s.beta, beta + t * H + h);
        }
    }
}

// alpha = exp(g) in place and alpha k for the staged tokens (after the copies have landed and a
// barrier).
__device__ __forceinline__ void stage_exp_cols(ColTok* st, int nt, int tid) {
    for (int idx = tid; idx < nt * kD; idx += 128) {
        ColTok& s = st[idx >> 7];
        const int o = perm_off(idx & 127);
        const float a = expf(s.a[o]);
        s.a[o] = a;
        s.ak[o] = a * s.k[o];
    }
}

// The 8 rows of a lane's slice of a staged vector.
__device__ __forceinline__ void load_rows(const float* p, float (&x)[8]) {
    const float4 a = reinterpret_cast<const float4*>(p)[0], b = reinterpret_cast<const float4*>(p)[1];
    x[0] = a.x; x[1] = a.y; x[2] = a.z; x[3] = a.w;
    x[4] = b.x; x[5] = b.y; x[6] = b.z; x[7] = b.w;
}
// Four column sums over the sixteen lanes of a column group (lane bits 0..3), every lane gets all
// four.
__device__ __forceinline__ void sum16x4(float (&x)[4]) {
#pragma unroll
    for (int off = 1; off < 16; off <<= 1)
#pragma unroll
        for (int j = 0; j < 4; ++j) x[j] += __shfl_xor_sync(0xffffffffu, x[j], off);
}
// Four column sums over the sixteen lanes of a column group; afterwards lanes 4 j .. 4 j + 3 of the
// group (r = lane & 15) hold the total of value j.
__device__ __forceinline__ float sum16x4_split(float (&x)[4], int r) {
#pragma unroll
    for (int i = 0; i < 2; ++i) {
        const bool up = (r & 8) != 0;
        const float send = up ? x[i] : x[i + 2];
        x[i] = (up ? x[i + 2] : x[i]) + __shfl_xor_sync(0xffffffffu, send, 8);
    }
    {
        const bool up = (r & 4) != 0;
        const float send = up ? x[0] : x[1];
        x[0] = (up ? x[1] : x[0]) + __shfl_xor_sync(0xffffffffu, send, 4);
    }
    x[0] += __shfl_xor_sync(0xffffffffu, x[0], 2);
    return x[0] + __shfl_xor_sync(0xffffffffu, x[0], 1);
}
// The four values of sum16x4_split gathered on lane r = 0 of each column group.
__device__ __forceinline__ float4 gather4(float v, int lane) {
    const int base = lane & ~15;
    const float v1 = __shfl_sync(0xffffffffu, v, base + 4), v2 = __shfl_sync(0xffffffffu, v, base + 8),
                v3 = __shfl_sync(0xffffffffu, v, base + 12);
    return make_float4(v, v1, v2, v3);
}

// The state slice of a lane (rows 8 r .. 8 r + 7 of columns c0 .. c0 + 3) to / from a row-major
// D x D matrix.
__device__ __forceinline__ void load_slice(const float* M, int r, int c0, float (&s)[8][4]) {
#pragma unroll
    for (int m = 0; m < 8; ++m) {
        const float4 a = *reinterpret_cast<const float4*>(M + (8 * r + m) * kD + c0);
        s[m][0] = a.x;
        s[m][1] = a.y;
        s[m][2] = a.z;
        s[m][3] = a.w;
    }
}
__device__ __forceinline__ void store_slice(float* M, int r, int c0, const float (&s)[8][4]) {
#pragma unroll
    for (int m = 0; m < 8; ++m)
        *reinterpret_cast<float4*>(M + (8 * r + m) * kD + c0) = make_float4(s[m][0], s[m][1], s[m][2], s[m][3]);
}

// Forward sweep: the recurrence from the initial state; o_t and e_t of every token; the state at
// the start of every kSeg-token segment (Sck).  Grid: units x kColCtas CTAs of 128 threads.
__global__ void __launch_bounds__(128)
k_bwd_fwd_cols(const float* __restrict__ X, const float* __restrict__ g, const float* __restrict__ beta,
               const int32_t* __restrict__ cu, const int64_t* __restrict__ prefix, int64_t T_total, int H,
               float scale, const float* __restrict__ S0, float* __restrict__ O, float* __restrict__ E,
               float* __restrict__ Sck, int64_t slots, int* __restrict__ d_status) {
    extern __shared__ __align__(16) unsigned char smem_raw[];
    ColTok* buf = reinterpret_cast<ColTok*>(smem_raw);  // [2][kTB]
    const int u = blockIdx.x / kColCtas, cq = blockIdx.x % kColCtas, n = u / H, h = u % H;
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31, r = lane & 15;
    const int cl = warp * 8 + 4 * (lane >> 4), c0 = cq * kCols + cl;
    int64_t s0, s1;
    seq_range(cu, n, T_total, s0, s1);
    const int64_t nseg = (s1 - s0 + kSeg - 1) / kSeg;
    const int64_t sb = slot_base(prefix, n, H, h, nseg, slots);
    if (sb < 0) {
        if (tid == 0) flag_status(d_status, KDA_ERR_DEVICE_ARG);
        return;
    }
    const int64_t HD = (int64_t)H * kD;
    const ColSrc vs{X + 2 * HD, 3 * HD};
    float s[8][4];
    if (S0) {
        load_slice(S0 + (int64_t)u * kD * kD, r, c0, s);
    } else {
#pragma unroll
        for (int m = 0; m < 8; ++m)
#pragma unroll
            for (int c = 0; c < 4; ++c) s[m][c] = 0.f;
    }
    const int64_t nblk = (s1 - s0 + kTB - 1) / kTB;
    auto nt_of = [&](int64_t b) { return (int)(s1 - (s0 + b * kTB) < kTB ? s1 - (s0 + b * kTB) : kTB); };
    if (nblk > 0) stage_cols(buf, s0, nt_of(0), X, g, beta, vs, vs, 1, H, h, cq, tid);
    cp_commit();
    for (int64_t b = 0; b < nblk; ++b) {
        __syncthreads();  // block b - 1 is consumed: its buffer takes block b + 1
        if (b + 1 < nblk)
            stage_cols(buf + ((b + 1) & 1) * kTB, s0 + (b + 1) * kTB, nt_of(b + 1), X, g, beta, vs, vs, 1, H, h,
                       cq, tid);
        cp_commit();
        cp_wait<1>();
        __syncthreads();
        ColTok* st = buf + (b & 1) * kTB;
        const int nt = nt_of(b);
        stage_exp_cols(st, nt, tid);
        __syncthreads();
        float x[4];  // (P_t^T k_t) of the lane's columns: alpha_t k_t against S_{t-1}
        {
            float ak[8];
            load_rows(st[0].ak + r * kSlice, ak);
#pragma unroll
            for (int c = 0; c < 4; ++c) {
                float a0 = 0.f, a1 = 0.f;
#pragma unroll
                for (int m = 0; m < 8; m += 2) {
                    a0 = fmaf(ak[m], s[m][c], a0);
                    a1 = fmaf(ak[m + 1], s[m + 1][c], a1);
                }
                x[c] = a0 + a1;
            }
            sum16x4(x);
        }
        static_assert(kSeg % kTB == 0, "segments start at block starts");
        if ((b * kTB) % kSeg == 0) store_slice(Sck + (sb + b * kTB / kSeg) * kD * kD, r, c0, s);
        for (int tk = 0; tk < nt; ++tk) {
            const int64_t t = s0 + b * kTB + tk;
            const ColTok& T = st[tk];
            const ColTok& Nx = st[tk + 1 < nt ? tk + 1 : tk];
            const float4 v4 = *reinterpret_cast<const float4*>(T.c0 + cl);
            const float bt = T.beta;
            const float e[4] = {v4.x - x[0], v4.y - x[1], v4.z - x[2], v4.w - x[3]};
            const float be[4] = {bt * e[0], bt * e[1], bt * e[2], bt * e[3]};
            float a2[8], k2[8], q2[8], n2[8];
            load_rows(T.a + r * kSlice, a2);
            load_rows(T.k + r * kSlice, k2);
            load_rows(T.q + r * kSlice, q2);
            load_rows(Nx.ak + r * kSlice, n2);
            float o[2][4] = {{0.f, 0.f, 0.f, 0.f}, {0.f, 0.f, 0.f, 0.f}};
            float p[2][4] = {{0.f, 0.f, 0.f, 0.f}, {0.f, 0.f, 0.f, 0.f}};
#pragma unroll
            for (int m = 0; m < 8; ++m)
#pragma unroll
                for (int c = 0; c < 4; ++c) {
                    s[m][c] = fmaf(a2[m], s[m][c], k2[m] * be[c]);  // S_t = Diag(alpha) S_{t-1} + beta k e^T
                    o[m & 1][c] = fmaf(q2[m], s[m][c], o[m & 1][c]);
                    p[m & 1][c] = fmaf(n2[m], s[m][c], p[m & 1][c]);
                }
#pragma unroll
            for (int c = 0; c < 4; ++c) x[c] = p[0][c] + p[1][c];  // unused after a block's last token
            sum16x4(x);
            float y[4] = {o[0][0] + o[1][0], o[0][1] + o[1][1], o[0][2] + o[1][2], o[0][3] + o[1][3]};
            const float4 o4 = gather4(sum16x4_split(y, r), lane);
            if (r == 0) {
                *reinterpret_cast<float4*>(O + (t * H + h) * kD + c0) =
                    make_float4(scale * o4.x, scale * o4.y, scale * o4.z, scale * o4.w);
                *reinterpret_cast<float4*>(E + (t * H + h) * kD + c0) = make_float4(e[0], e[1], e[2], e[3]);
            }
        }
    }
}

// dS <- Diag(alpha) (dS - beta k w^T) with the factors of a staged token and nbw = -beta w of the
// lane's columns.
__device__ __forceinline__ void bwd_decay(float (&ds)[8][4], const float (&a2)[8], const float (&k2)[8],
                                          const float (&nbw)[4]) {
#pragma unroll
    for (int m = 0; m < 8; ++m)
#pragma unroll
        for (int c = 0; c < 4; ++c) ds[m][c] = a2[m] * fmaf(k2[m], nbw[c], ds[m][c]);
}

// One token of the backward sweep: dS' = [pending: Diag(alpha') (dS - beta' k' w'^T)] + scale q do^T
// with (alpha', k', -beta' w') of the later token, w = dS'^T k summed over the column group (all
// lanes get it); the stores and the dbeta / e.do partials of the token.
template <bool kPending>
__device__ __forceinline__ void bwd_token(float (&ds)[8][4], float (&nbw)[4], const ColTok& T, const ColTok& Pv,
                                          int r, int cl, int c0, int lane, float scale, int64_t t, int H, int h,
                                          float* W, float* dX, float* accb, float* acce) {
    const int64_t HD = (int64_t)H * kD;
    const float4 do4 = *reinterpret_cast<const float4*>(T.c0 + cl);
    const float4 e4 = *reinterpret_cast<const float4*>(T.c1 + cl);
    const float bt = T.beta;
    const float sd[4] = {scale * do4.x, scale * do4.y, scale * do4.z, scale * do4.w};
    float k2[8], q2[8];
    load_rows(T.k + r * kSlice, k2);
    load_rows(T.q + r * kSlice, q2);
    float wp[2][4] = {{0.f, 0.f, 0.f, 0.f}, {0.f, 0.f, 0.f, 0.f}};
    if constexpr (kPending) {
        float pa[8], pk[8];
        load_rows(Pv.a + r * kSlice, pa);
        load_rows(Pv.k + r * kSlice, pk);
#pragma unroll
        for (int m = 0; m < 8; ++m)
#pragma unroll
            for (int c = 0; c < 4; ++c) {
                const float d = pa[m] * fmaf(pk[m], nbw[c], ds[m][c]);
                ds[m][c] = fmaf(q2[m], sd[c], d);
                wp[m & 1][c] = fmaf(k2[m], ds[m][c], wp[m & 1][c]);
            }
    } else {
#pragma unroll
        for (int m = 0; m < 8; ++m)
#pragma unroll
            for (int c = 0; c < 4; ++c) {
                ds[m][c] = fmaf(q2[m], sd[c], ds[m][c]);
                wp[m & 1][c] = fmaf(k2[m], ds[m][c], wp[m & 1][c]);
            }
    }
    float w[4] = {wp[0][0] + wp[1][0], wp[0][1] + wp[1][1], wp[0][2] + wp[1][2], wp[0][3] + wp[1][3]};
    sum16x4(w);
#pragma unroll
    for (int c = 0; c < 4; ++c) nbw[c] = -bt * w[c];
    const bool lead = r == 0;
    if (lead) {
        *reinterpret_cast<float4*>(W + (t * H + h) * kD + c0) = make_float4(w[0], w[1], w[2], w[3]);
        *reinterpret_cast<float4*>(dX + t * 3 * HD + 2 * HD + (int64_t)h * kD + c0) =
            make_float4(bt * w[0], bt * w[1], bt * w[2], bt * w[3]);
    }
    float pb = lead ? w[0] * e4.x + w[1] * e4.y + w[2] * e4.z + w[3] * e4.w : 0.f;
    float pe = lead ? e4.x * do4.x + e4.y * do4.y + e4.z * do4.z + e4.w * do4.w : 0.f;
    pb += __shfl_xor_sync(0xffffffffu, pb, 16);
    pe += __shfl_xor_sync(0xffffffffu, pe, 16);
    if (lane == 0) {
        atomicAdd(accb, pb);
        atomicAdd(acce, pe);
    }
}

// Backward sweep of the state gradient, tokens in reverse: dS' = dS + scale q^ do^T,
// w = dS'^T k^, dv = beta w, then dS <- Diag(alpha) (dS' - beta k^ w^T) (applied in the next
// token's pass).  Writes w, dv, the sums dbeta = w . e and e . do of every token (atomics over the
// CTAs of a unit), the state gradient at the end of every segment (dSck: before that token's own
// terms) and at the start (dS0).  Blocks are the forward sweep's, taken last to first, so that
// every segment ends at the last token of a block.
__global__ void __launch_bounds__(128)
k_bwd_bwd_cols(const float* __restrict__ X, const float* __restrict__ g, const float* __restrict__ beta,
               const float* __restrict__ dO, const float* __restrict__ E, const int32_t* __restrict__ cu,
               const int64_t* __restrict__ prefix, int64_t T_total, int H, float scale,
               const float* __restrict__ dS_fin, float* __restrict__ W, float* __restrict__ dX,
               float* __restrict__ dbeta, float* __restrict__ edo, float* __restrict__ dSck,
               float* __restrict__ dS0, int64_t slots) {
    extern __shared__ __align__(16) unsigned char smem_raw[];
    ColTok* buf = reinterpret_cast<ColTok*>(smem_raw);  // [2][kTB]
    __shared__ float acc[2][2][kTB];                   // [block parity][dbeta, e.do][token]
    const int u = blockIdx.x / kColCtas, cq = blockIdx.x % kColCtas, n = u / H, h = u % H;
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31, r = lane & 15;
    const int cl = warp * 8 + 4 * (lane >> 4), c0 = cq * kCols + cl;
    if (tid < 4 * kTB) (&acc[0][0][0])[tid] = 0.f;
    int64_t s0, s1;
    seq_range(cu, n, T_total, s0, s1);
    const int64_t nseg = (s1 - s0 + kSeg - 1) / kSeg;
    const int64_t sb = slot_base(prefix, n, H, h, nseg, slots);
    if (sb < 0) return;  // flagged by the forward sweep
    const int64_t HD = (int64_t)H * kD;
    const ColSrc dos{dO, HD}, es{E, HD};
    float ds[8][4];
    if (dS_fin) {
        load_slice(dS_fin + (int64_t)u * kD * kD, r, c0, ds);
    } else {
#pragma unroll
        for (int m = 0; m < 8; ++m)
#pragma unroll
            for (int c = 0; c < 4; ++c) ds[m][c] = 0.f;
    }
    // step i takes block j = nblk - 1 - i: tokens [s0 + j kTB, min(s0 + (j + 1) kTB, s1))
    const int64_t nblk = (s1 - s0 + kTB - 1) / kTB;
    auto t0_of = [&](int64_t i) { return s0 + (nblk - 1 - i) * kTB; };
    auto nt_of = [&](int64_t i) { return (int)(s1 - t0_of(i) < kTB ? s1 - t0_of(i) : kTB); };
    if (nblk > 0) stage_cols(buf, t0_of(0), nt_of(0), X, g, beta, dos, es, 2, H, h, cq, tid);
    cp_commit();
    for (int64_t i = 0; i < nblk; ++i) {
        __syncthreads();
        if (i > 0 && tid < nt_of(i - 1)) {  // the sums of the previous step are complete
            const int p = (i - 1) & 1;
            const int64_t t = t0_of(i - 1) + tid;
            atomicAdd(dbeta + t * H + h, acc[p][0][tid]);
            atomicAdd(edo + t * H + h, acc[p][1][tid]);
            acc[p][0][tid] = 0.f;
            acc[p][1][tid] = 0.f;
        }
        if (i + 1 < nblk)
            stage_cols(buf + ((i + 1) & 1) * kTB, t0_of(i + 1), nt_of(i + 1), X, g, beta, dos, es, 2, H, h, cq,
                       tid);
        cp_commit();
        cp_wait<1>();
        __syncthreads();
        ColTok* st = buf + (i & 1) * kTB;
        const int nt = nt_of(i);
        const int64_t t0 = t0_of(i);
        stage_exp_cols(st, nt, tid);
        __syncthreads();
        // the block's last token ends a segment when the segment is full or the sequence ends there
        const int64_t tl = t0 + nt - 1;
        if ((tl - s0) % kSeg == kSeg - 1 || tl == s1 - 1) store_slice(dSck + (sb + (tl - s0) / kSeg) * kD * kD, r, c0, ds);
        float nbw[4];  // -beta w of the later token, whose decay is pending
        float* ab = &acc[i & 1][0][0];
        float* ae = &acc[i & 1][1][0];
        bwd_token<false>(ds, nbw, st[nt - 1], st[nt - 1], r, cl, c0, lane, scale, tl, H, h, W, dX, ab + nt - 1,
                         ae + nt - 1);
        for (int tk = nt - 2; tk >= 0; --tk)
            bwd_token<true>(ds, nbw, st[tk], st[tk + 1], r, cl, c0, lane, scale, t0 + tk, H, h, W, dX, ab + tk,
                            ae + tk);
        {  // the block's first token's decay, before its buffer is refilled
            float pa[8], pk[8];
            load_rows(st[0].a + r * kSlice, pa);
            load_rows(st[0].k + r * kSlice, pk);
            bwd_decay(ds, pa, pk, nbw);
        }
    }
    __syncthreads();
    if (nblk > 0 && tid < nt_of(nblk - 1)) {
        const int p = (nblk - 1) & 1;
        const int64_t t = t0_of(nblk - 1) + tid;
        atomicAdd(dbeta + t * H + h, acc[p][0][tid]);
        atomicAdd(edo + t * H + h, acc[p][1][tid]);
    }
    if (dS0) store_slice(dS0 + (int64_t)u * kD * kD, r, c0, ds);
}

// ------------------------------------------------------------------------------ row-layout segments
// One CTA of 256 threads per (unit, segment): thread (rg, cg) owns rows 8 rg .. 8 rg + 7 and columns
// 8 cg .. 8 cg + 7 (packed fp32 pairs); the row sums a token needs (S x, dS' e) go over the 16
// column groups of a half-warp.  With e, w and do known for every token, both sweeps are row-local:
//   forward from the segment's start state:  dq = scale (P do + beta k (e . do)),
//                                            dk_read = -beta P w,   P = Diag(alpha) S_{t-1};
//   backward from the segment's end gradient: dk_write = beta dS' e.
// dg follows from the decay entering only through e^{Gamma_t} (read keys and queries) and
// e^{-Gamma_t} (written keys), Gamma_t = sum_{s <= t} g_s:
//   dGamma_t = q^ dq + k^ dk_read - k^ dk_write,  dg_t = sum_{s >= t} dGamma_s + rowsum(dS_T . S_T);
// here the parts within the segment: dg <- -(sum of q dq + k dk_read over earlier tokens), the
// global rows of e and w (staged, so free) <- dk_write and the suffix sums of -k dk_write; per
// segment its sum of dGamma (segtot) and of the read part (segown); for the last segment of a
// sequence the final-state term (fin).  The sweeps only write global memory.
constexpr int kRowThreads = 256;
constexpr int kColVec = kD + 12;  // column vectors skewed by 4 floats every 32, so that the eight
                                  // column groups a quarter-warp reads fall in distinct banks
struct RowTok {
    float k[kD], a[kD], q[kD];
    float e[kColVec], d[kColVec], w[kColVec];
    float beta, edo, pad[2];
};
constexpr int kRowSmem = kSeg * (int)sizeof(RowTok);

// Sums 16 per-thread values over the 16 lanes of a half-warp (lane bits 0..3); afterwards lane
// cg holds the total of value cg.
__device__ __forceinline__ float reduce16_16(float (&v)[16], int cg) {
#pragma unroll
    for (int i = 0; i < 8; ++i) {
        const bool up = (cg & 8) != 0;
        const float send = up ? v[i] : v[i + 8];
        v[i] = (up ? v[i + 8] : v[i]) + __shfl_xor_sync(0xffffffffu, send, 8);
    }
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        const bool up = (cg & 4) != 0;
        const float send = up ? v[i] : v[i + 4];
        v[i] = (up ? v[i + 4] : v[i]) + __shfl_xor_sync(0xffffffffu, send, 4);
    }
#pragma unroll
    for (int i = 0; i < 2; ++i) {
        const bool up = (cg & 2) != 0;
        const float send = up ? v[i] : v[i + 2];
        v[i] = (up ? v[i + 2] : v[i]) + __shfl_xor_sync(0xffffffffu, send, 2);
    }
    const bool up = (cg & 1) != 0;
    const float send = up ? v[0] : v[1];
    return (up ? v[1] : v[0]) + __shfl_xor_sync(0xffffffffu, send, 1);
}
__device__ __forceinline__ void load8(const float* p, float (&x)[8]) {
    const float4 a = reinterpret_cast<const float4*>(p)[0], b = reinterpret_cast<const float4*>(p)[1];
    x[0] = a.x; x[1] = a.y; x[2] = a.z; x[3] = a.w;
    x[4] = b.x; x[5] = b.y; x[6] = b.z; x[7] = b.w;
}
__device__ __forceinline__ float pick8(const float (&x)[8], int a) {  // x[a] without local memory
    float r = x[0];
#pragma unroll
    for (int i = 1; i < 8; ++i) r = a == i ? x[i] : r;
    return r;
}
// Same for 8 values; afterwards lanes cg hold the total of value cg >> 1.
__device__ __forceinline__ float reduce8_16(float (&v)[8], int cg) {
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        const bool up = (cg & 8) != 0;
        const float send = up ? v[i] : v[i + 4];
        v[i] = (up ? v[i + 4] : v[i]) + __shfl_xor_sync(0xffffffffu, send, 8);
    }
#pragma unroll
    for (int i = 0; i < 2; ++i) {
        const bool up = (cg & 4) != 0;
        const float send = up ? v[i] : v[i + 2];
        v[i] = (up ? v[i + 2] : v[i]) + __shfl_xor_sync(0xffffffffu, send, 4);
    }
    {
        const bool up = (cg & 2) != 0;
        const float send = up ? v[0] : v[1];
        v[0] = (up ? v[1] : v[0]) + __shfl_xor_sync(0xffffffffu, send, 2);
    }
    return v[0] + __shfl_xor_sync(0xffffffffu, v[0], 1);
}

__device__ __forceinline__ void load8p(const float* p, f2 (&x)[4]) {  // 8 floats as 4 pairs
    const ulonglong2 a = reinterpret_cast<const ulonglong2*>(p)[0], b = reinterpret_cast<const ulonglong2*>(p)[1];
    x[0].v = a.x;
    x[1].v = a.y;
    x[2].v = b.x;
    x[3].v = b.y;
}
__device__ __forceinline__ float hsum(f2 x) { return f2_lo(x) + f2_hi(x); }

// Grid: units x max_seg CTAs (CTAs past a sequence's segment count return at once).
__global__ void __launch_bounds__(kRowThreads, 1)
k_bwd_rows(const float* __restrict__ X, const float* __restrict__ g, const float* __restrict__ beta,
           const float* __restrict__ dO, float* __restrict__ E, float* __restrict__ W,
           const float* __restrict__ edo, const int32_t* __restrict__ cu, const int64_t* __restrict__ prefix,
           int64_t T_total, int H, float scale, int max_seg, const float* __restrict__ Sck,
           const float* __restrict__ dSck, const float* __restrict__ dS_fin, float* __restrict__ dX,
           float* __restrict__ dg, float* __restrict__ segtot, float* __restrict__ segown, float* __restrict__ fin,
           int64_t slots) {
    extern __shared__ __align__(16) unsigned char smem_raw[];
    RowTok* st = reinterpret_cast<RowTok*>(smem_raw);  // [kSeg]
    const int u = blockIdx.x / max_seg, sg = blockIdx.x % max_seg, n = u / H, h = u % H;
    const int tid = threadIdx.x, rg = tid >> 4, cg = tid & 15;
    int64_t s0, s1;
    seq_range(cu, n, T_total, s0, s1);
    const int64_t nseg = (s1 - s0 + kSeg - 1) / kSeg;
    if (sg >= nseg) return;
    const int64_t sb = slot_base(prefix, n, H, h, nseg, slots);
    if (sb < 0) return;  // flagged by the forward sweep
    const int64_t HD = (int64_t)H * kD;
    const int64_t ta = s0 + (int64_t)sg * kSeg, tb = ta + kSeg < s1 ? ta + kSeg : s1;
    const int nt = (int)(tb - ta);
    // stage the segment: six 128-vectors (32 chunks each), beta and e . do per token
    for (int idx = tid; idx < nt * 194; idx += kRowThreads) {
        const int tk = idx / 194, j = idx - tk * 194;
        const int64_t t = ta + tk, th = t * H + h;
        RowTok& s = st[tk];
        if (j < 192) {
            const int part = j >> 5, jj = j & 31;
            const float* src = part == 0 ? X + t * 3 * HD + HD + (int64_t)h * kD
                             : part == 1 ? g + th * kD
                             : part == 2 ? X + t * 3 * HD + (int64_t)h * kD
                             : part == 3 ? E + th * kD
                             : part == 4 ? dO + th * kD
                                         : W + th * kD;
            float* dst = part == 0 ? s.k : part == 1 ? s.a : part == 2 ? s.q : part == 3 ? s.e : part == 4 ? s.d : s.w;
            cp16(dst + 4 * jj + (part >= 3 ? (jj >> 3) * 4 : 0), src + 4 * jj);
        } else {
            cp4(j == 192 ? &s.beta : &s.edo, (j == 192 ? beta : edo) + th);
        }
    }
    cp_commit();
    cp_wait<0>();
    __syncthreads();
    for (int idx = tid; idx < nt * kD; idx += kRowThreads) {
        float& x = st[idx >> 7].a[idx & 127];
        x = expf(x);
    }
    __syncthreads();
    const int r0 = 8 * rg, cs = 8 * cg + (cg >> 2) * 4;  // first row; column offset in a skewed vector
    const bool writer = (cg & 1) == 0;                  // lanes holding row r0 + (cg >> 1)
    const int ra = cg >> 1;
    // ---- forward: S from the segment's start state
    float pre = 0.f;  // writer lanes: sum over this segment's earlier tokens of q dq + k dk_read
    f2 s[8][4];
    {
        const float* src = Sck + (sb + sg) * kD * kD + 8 * cg;
#pragma unroll
        for (int a = 0; a < 8; ++a) load8p(src + (r0 + a) * kD, s[a]);
    }
    for (int tk = 0; tk < nt; ++tk) {
        const RowTok& T = st[tk];
        f2 e2[4], d2[4], w2[4];
        load8p(T.e + cs, e2);
        load8p(T.d + cs, d2);
        load8p(T.w + cs, w2);
        float kr[8], ar[8];
        load8(T.k + r0, kr);
        load8(T.a + r0, ar);
        float v[16];
#pragma unroll
        for (int a = 0; a < 8; ++a) {
            f2 x0 = mul2(s[a][0], d2[0]), x1 = mul2(s[a][0], w2[0]);
#pragma unroll
            for (int p = 1; p < 4; ++p) {
                x0 = fma2(s[a][p], d2[p], x0);
                x1 = fma2(s[a][p], w2[p], x1);
            }
            v[2 * a] = hsum(x0);
            v[2 * a + 1] = hsum(x1);
        }
        const float red = reduce16_16(v, cg);  // lane cg: value cg (row cg >> 1; S do if even, S w if odd)
        const float sw = __shfl_xor_sync(0xffffffffu, red, 1);
        const float bt = T.beta;
        {  // computed on every lane, stored by the writer lanes
            const int i = r0 + ra;
            const float al = pick8(ar, ra), ki = pick8(kr, ra);
            const float dq = scale * (al * red + bt * ki * T.edo);
            const float dkr = -bt * al * sw;
            const int64_t t = ta + tk;
            if (writer) {
                dX[t * 3 * HD + (int64_t)h * kD + i] = dq;
                dX[t * 3 * HD + HD + (int64_t)h * kD + i] = dkr;
                dg[(t * H + h) * kD + i] = -pre;  // minus the sum of dGamma_read over earlier tokens
            }
            pre += T.q[i] * dq + ki * dkr;
        }
#pragma unroll
        for (int a = 0; a < 8; ++a) {
            const f2 a2 = f2_dup(ar[a]), bk2 = f2_dup(bt * kr[a]);
#pragma unroll
            for (int p = 0; p < 4; ++p) s[a][p] = fma2(bk2, e2[p], mul2(a2, s[a][p]));
        }
    }
    if (tb == s1) {  // the sequence's final state: rowsum(dS_T . S_T)
        float f[8];
#pragma unroll
        for (int a = 0; a < 8; ++a) {
            float x = 0.f;
            if (dS_fin) {
                f2 d2[4];
                load8p(dS_fin + ((int64_t)u * kD + r0 + a) * kD + 8 * cg, d2);
                f2 y = mul2(d2[0], s[a][0]);
#pragma unroll
                for (int p = 1; p < 4; ++p) y = fma2(d2[p], s[a][p], y);
                x = hsum(y);
            }
            f[a] = x;
        }
        const float tot = reduce8_16(f, cg);
        if (writer) fin[(int64_t)u * kD + r0 + ra] = tot;
    }
    // ---- backward: dS from the segment's end gradient
    f2 (&ds)[8][4] = s;
    {
        const float* src = dSck + (sb + sg) * kD * kD + 8 * cg;
#pragma unroll
        for (int a = 0; a < 8; ++a) load8p(src + (r0 + a) * kD, ds[a]);
    }
    float run = 0.f;  // writer lanes: sum over this segment's tokens >= t of -k dk_write
    for (int tk = nt - 1; tk >= 0; --tk) {
        const RowTok& T = st[tk];
        f2 e2[4], d2[4], w2[4];
        load8p(T.e + cs, e2);
        load8p(T.d + cs, d2);
        load8p(T.w + cs, w2);
        float kr[8], ar[8], qr[8];
        load8(T.k + r0, kr);
        load8(T.a + r0, ar);
        load8(T.q + r0, qr);
        const float bt = T.beta;
        float y[8];
#pragma unroll
        for (int a = 0; a < 8; ++a) {
            const f2 sq2 = f2_dup(scale * qr[a]);
            ds[a][0] = fma2(sq2, d2[0], ds[a][0]);
            f2 x = mul2(ds[a][0], e2[0]);
#pragma unroll
            for (int p = 1; p < 4; ++p) {
                ds[a][p] = fma2(sq2, d2[p], ds[a][p]);
                x = fma2(ds[a][p], e2[p], x);
            }
            y[a] = hsum(x);
        }
        const float dse = reduce8_16(y, cg);  // (dS'_t e_t) of row cg >> 1
        {  // the token's e and w rows are staged, so their global rows take dk_write and the suffix
           // sums of -k dk_write (combined by the L2 kernel); stored by the writer lanes
            const int i = r0 + ra;
            const int64_t th = (ta + tk) * H + h;
            const float dkw = bt * dse;
            run -= pick8(kr, ra) * dkw;
            if (writer) {
                E[th * kD + i] = dkw;
                W[th * kD + i] = run;
            }
        }
#pragma unroll
        for (int a = 0; a < 8; ++a) {
            const f2 a2 = f2_dup(ar[a]), nbk2 = f2_dup(-bt * kr[a]);
#pragma unroll
            for (int p = 0; p < 4; ++p) ds[a][p] = mul2(a2, fma2(nbk2, w2[p], ds[a][p]));
        }
    }
    if (writer) {
        segtot[(sb + sg) * kD + r0 + ra] = pre + run;  // the segment's sum of dGamma
        segown[(sb + sg) * kD + r0 + ra] = pre;        // added to its own tokens (dg = -pre_t + run_t + ...)
    }
}

// dg carries: for each unit and channel, the segments from the last: the value to add to every
// token of segment sg is fin + the totals of the segments after it + its own read part (written
// over segtot).
__global__ void k_bwd_dg_carry(const int32_t* __restrict__ cu, const int64_t* __restrict__ prefix, int64_t T_total,
                               int H, const float* __restrict__ fin, float* __restrict__ segtot,
                               const float* __restrict__ segown, int64_t slots) {
    const int u = blockIdx.x, i = threadIdx.x, n = u / H, h = u % H;
    int64_t s0, s1;
    seq_range(cu, n, T_total, s0, s1);
    const int64_t nseg = (s1 - s0 + kSeg - 1) / kSeg;
    const int64_t sb = slot_base(prefix, n, H, h, nseg, slots);
    if (sb < 0 || nseg == 0) return;
    float carry = fin[(int64_t)u * kD + i];
    for (int64_t sg = nseg - 1; sg >= 0; --sg) {
        float* p = segtot + (sb + sg) * kD + i;
        const float x = *p;
        *p = carry + segown[(sb + sg) * kD + i];
        carry += x;
    }
}

// ------------------------------------------------------------------------------ epilogue backward
// One warp per (token, head) row: do (written over o), dgate, and the RMSNorm weight's gradient
// (block partials in shared memory, one atomic per channel and block).
template <typename Tg, typename Tdy>
__global__ void k_bwd_epilogue(float* __restrict__ O, const Tdy* __restrict__ dy, const Tg* __restrict__ gate,
                               const float* __restrict__ rms_w, float eps_rms, int64_t rows,
                               float* __restrict__ dgate, float* __restrict__ drms) {
    __shared__ float sdw[kD];
    for (int c = threadIdx.x; c < kD; c += blockDim.x) sdw[c] = 0.f;
    __syncthreads();
    const int lane = threadIdx.x & 31;
    const int64_t row = (int64_t)blockIdx.x * (blockDim.x / 32) + (threadIdx.x >> 5);
    if (row < rows) {
        const int c0 = 4 * lane;
        float* orow = O + row * kD + c0;
        const float4 o = *reinterpret_cast<const float4*>(orow);
        const float r = 1.0f / sqrtf(warp_sum(dot4(o, o)) * (1.0f / kD) + eps_rms);
        float dn[4], dw[4];
        const float ov[4] = {o.x, o.y, o.z, o.w};
        float dno = 0.f;
#pragma unroll
        for (int m = 0; m < 4; ++m) {
            const float w = rms_w ? rms_w[c0 + m] : 1.f;
            const float sg = gate ? 1.0f / (1.0f + expf(-to_f(gate[row * kD + c0 + m]))) : 1.f;
            const float d = to_f(dy[row * kD + c0 + m]);
            const float nv = ov[m] * r;
            if (dgate) dgate[row * kD + c0 + m] = gate ? d * nv * w * sg * (1.f - sg) : 0.f;
            dw[m] = d * nv * sg;
            dn[m] = d * w * sg;
            dno += dn[m] * ov[m];
        }
        dno = warp_sum(dno);
        const float r3 = r * r * r * dno * (1.0f / kD);
        *reinterpret_cast<float4*>(orow) =
            make_float4(r * dn[0] - r3 * ov[0], r * dn[1] - r3 * ov[1], r * dn[2] - r3 * ov[2], r * dn[3] - r3 * ov[3]);
        if (drms)
#pragma unroll
            for (int m = 0; m < 4; ++m) atomicAdd(&sdw[c0 + m], dw[m]);
    }
    __syncthreads();
    if (drms)
        for (int c = threadIdx.x; c < kD; c += blockDim.x) atomicAdd(&drms[c], sdw[c]);
}

// ------------------------------------------------------------------------------ L2 backward
// One warp per (token, head): dk^ = dk_read + dk_write (the latter in dkw); dq^ -> d a_q =
// (dq^ - q^ (q^ . dq^)) / |a_q|, same for k, in place; dg += the write part's suffix sum (dgw) and
// the carry of the token's segment.
__global__ void k_bwd_l2(const float* __restrict__ X, const float* __restrict__ nrm, const int32_t* __restrict__ cu,
                         const int64_t* __restrict__ prefix, int N, int64_t T_total, int H,
                         const float* __restrict__ segtot, const float* __restrict__ dkw,
                         const float* __restrict__ dgw, int64_t slots, float* __restrict__ dX,
                         float* __restrict__ dg) {
    const int64_t row = (int64_t)blockIdx.x * (blockDim.x / 32) + (threadIdx.x >> 5);
    const int lane = threadIdx.x & 31;
    if (row >= T_total * H) return;
    const int64_t t = row / H, HD = (int64_t)H * kD;
    const int h = (int)(row % H);
    const float2 nn = *reinterpret_cast<const float2*>(nrm + row * 2);
#pragma unroll
    for (int part = 0; part < 2; ++part) {
        const int64_t off = t * 3 * HD + part * HD + (int64_t)h * kD + 4 * lane;
        const float4 x = *reinterpret_cast<const float4*>(X + off);
        float4 d = *reinterpret_cast<const float4*>(dX + off);
        if (part == 1) d = f4_add(d, *reinterpret_cast<const float4*>(dkw + row * kD + 4 * lane));
        const float xd = warp_sum(dot4(x, d));
        const float inv = 1.0f / (part == 0 ? nn.x : nn.y);
        *reinterpret_cast<float4*>(dX + off) = make_float4((d.x - x.x * xd) * inv, (d.y - x.y * xd) * inv,
                                                           (d.z - x.z * xd) * inv, (d.w - x.w * xd) * inv);
    }
    int lo = 0, hi = N;
    while (hi - lo > 1) {
        const int mid = (lo + hi) >> 1;
        if (cu[mid] <= t) lo = mid;
        else hi = mid;
    }
    int64_t s0, s1;
    seq_range(cu, lo, T_total, s0, s1);
    if (t < s0 || t >= s1) return;
    const int64_t nseg = (s1 - s0 + kSeg - 1) / kSeg;
    const int64_t sb = slot_base(prefix, lo, H, h, nseg, slots);
    if (sb < 0) return;
    float4* p = reinterpret_cast<float4*>(dg + row * kD + 4 * lane);
    const float4 c = *reinterpret_cast<const float4*>(segtot + (sb + (t - s0) / kSeg) * kD + 4 * lane);
    const float4 w = *reinterpret_cast<const float4*>(dgw + row * kD + 4 * lane);
    *p = f4_add(f4_add(*p, c), w);
}

// ------------------------------------------------------------------------------ activation + conv backward
// One thread per (channel of 3 H D, tile of kConvTile tokens), tokens walked backwards: du =
// da silu'(u) (u recomputed from the raw inputs), dx_t = sum_j w_j du_{t+3-j}, the taps' gradient
// (one atomic per tap and thread), the conv state's gradient from the first three tokens' du of
// every sequence that starts in the tile.  The du of the three tokens after the tile (same
// sequence) are recomputed as a look-ahead.  Grid: cblocks channel blocks x tiles.
constexpr int kConvTile = 128;

template <typename Tio>
__global__ void k_bwd_conv(const Tio* __restrict__ q, const Tio* __restrict__ k, const Tio* __restrict__ v,
                           int64_t xs, const float* __restrict__ conv_w, const Tio* __restrict__ cs_in,
                           const int32_t* __restrict__ cu, int N, int64_t T_total, int H, int cblocks,
                           const float* __restrict__ dA, float* __restrict__ dq, float* __restrict__ dk,
                           float* __restrict__ dv, float* __restrict__ dconv_w, float* __restrict__ dcs) {
    const int64_t HD = (int64_t)H * kD;
    const int ch = (blockIdx.x % cblocks) * blockDim.x + threadIdx.x;
    const int64_t ta = (int64_t)(blockIdx.x / cblocks) * kConvTile;
    if (ch >= 3 * HD || ta >= T_total) return;
    const int64_t tb = ta + kConvTile < T_total ? ta + kConvTile : T_total;
    const int part = (int)(ch / HD);
    const int64_t hc = ch % HD;  // h * D + d
    const Tio* src = part == 0 ? q : part == 1 ? k : v;
    float* dst = part == 0 ? dq : part == 1 ? dk : dv;
    const float4 w = *reinterpret_cast<const float4*>(conv_w + (int64_t)ch * 4);
    // the sequence holding token tb - 1: the last n with cu[n] <= tb - 1
    int n = 0;
    {
        int lo = 0, hi = N;
        while (hi - lo > 1) {
            const int mid = (lo + hi) >> 1;
            if (cu[mid] <= tb - 1) lo = mid;
            else hi = mid;
        }
        n = lo;
    }
    int64_t s0, s1;
    seq_range(cu, n, T_total, s0, s1);
    auto raw = [&](int64_t p) -> float {  // raw input at position p; before s0: the conv state
        if (p >= s0) return to_f(src[p * xs + hc]);
        const int64_t j = 3 + (p - s0);
        return (cs_in && j >= 0) ? to_f(cs_in[((int64_t)n * 3 * HD + ch) * 3 + j]) : 0.f;
    };
    auto emit_state_grad = [&](float d0, float d1, float d2) {  // du_{s0}, du_{s0+1}, du_{s0+2}
        if (!dcs) return;
        float* dc = dcs + ((int64_t)n * 3 * HD + ch) * 3;
        dc[0] = w.x * d0;                       // x_{s0-3} feeds u_{s0} through tap 0
        dc[1] = w.y * d0 + w.x * d1;            // x_{s0-2}: u_{s0} (tap 1), u_{s0+1} (tap 0)
        dc[2] = w.z * d0 + w.y * d1 + w.x * d2; // x_{s0-1}: taps 2, 1, 0
    };
    float du1 = 0.f, du2 = 0.f, du3 = 0.f;  // du_{t+1}, du_{t+2}, du_{t+3}
    float gw0 = 0.f, gw1 = 0.f, gw2 = 0.f, gw3 = 0.f;
    float x0 = 0.f, x1 = 0.f, x2 = 0.f, x3 = 0.f;  // raw inputs at t - 3 .. t (a sliding window)
    // token t, given its oldest window input raw(t - 3) and its da (the window holds t - 2 .. t + 1)
    auto step = [&](int64_t t, float xnew, float da) {
        x3 = x2;
        x2 = x1;
        x1 = x0;
        x0 = xnew;
        const float uu = w.x * x0 + w.y * x1 + w.z * x2 + w.w * x3;
        const float sg = 1.0f / (1.0f + expf(-uu));
        const float du = da * sg * (1.0f + uu * (1.0f - sg));
        if (t < tb) {
            dst[t * HD + hc] = w.w * du + w.z * du1 + w.y * du2 + w.x * du3;
            gw0 += x0 * du;
            gw1 += x1 * du;
            gw2 += x2 * du;
            gw3 += x3 * du;
        }
        du3 = du2;
        du2 = du1;
        du1 = du;
    };
    const int64_t HD3 = 3 * HD;
    bool fresh = true;
    for (int64_t t = (tb + 3 < s1 ? tb + 3 : s1) - 1; t >= ta;) {
        if (t < s0) {  // crossed the start of sequence n (which lies inside the tile)
            emit_state_grad(du1, du2, du3);
            du1 = du2 = du3 = 0.f;
            while (n > 0) {
                --n;
                seq_range(cu, n, T_total, s0, s1);
                if (s0 <= t) break;
            }
            fresh = true;
        }
        if (fresh) {
            x0 = raw(t - 2);
            x1 = raw(t - 1);
            x2 = raw(t);
            fresh = false;
        }
        if (t - 6 >= s0 && t - 3 >= ta) {  // four tokens inside the sequence: their loads first
            const float r0 = to_f(src[(t - 3) * xs + hc]), r1 = to_f(src[(t - 4) * xs + hc]);
            const float r2 = to_f(src[(t - 5) * xs + hc]), r3 = to_f(src[(t - 6) * xs + hc]);
            const float d0 = dA[t * HD3 + ch], d1 = dA[(t - 1) * HD3 + ch];
            const float d2 = dA[(t - 2) * HD3 + ch], d3 = dA[(t - 3) * HD3 + ch];
            step(t, r0, d0);
            step(t - 1, r1, d1);
            step(t - 2, r2, d2);
            step(t - 3, r3, d3);
            t -= 4;
        } else {
            step(t, raw(t - 3), dA[t * HD3 + ch]);
            --t;
        }
    }
    if (s0 == ta) emit_state_grad(du1, du2, du3);  // sequence n starts at the tile's first token
    float* dw = dconv_w + (int64_t)ch * 4;
    atomicAdd(dw + 0, gw0);
    atomicAdd(dw + 1, gw1);
    atomicAdd(dw + 2, gw2);
    atomicAdd(dw + 3, gw3);
}

template <typename T>
const T* cptr(const void* p) { return static_cast<const T*>(p); }

template <typename Tio>
cudaError_t backward_launch(const kda_backward_args& b, const BackwardLayout& L, char* ws, cudaStream_t s) {
    const kda_prefill_args& a = b.fwd;
    const int64_t T = a.T_total, rows = T * a.H, units = (int64_t)a.N * a.H;
    const int64_t xs = a.qkv_row_stride ? a.qkv_row_stride : (int64_t)a.H * kD;
    float* X = reinterpret_cast<float*>(ws + L.x);
    float* nrm = reinterpret_cast<float*>(ws + L.nrm);
    float* O = reinterpret_cast<float*>(ws + L.o);
    float* dX = reinterpret_cast<float*>(ws + L.dx);
    float* E = reinterpret_cast<float*>(ws + L.e);
    float* W = reinterpret_cast<float*>(ws + L.w);
    float* edo = reinterpret_cast<float*>(ws + L.edo);
    float* Sck = reinterpret_cast<float*>(ws + L.sck);
    float* dSck = reinterpret_cast<float*>(ws + L.dsck);
    float* segtot = reinterpret_cast<float*>(ws + L.segtot);
    float* segown = reinterpret_cast<float*>(ws + L.segown);
    float* fin = reinterpret_cast<float*>(ws + L.fin);
    int64_t* prefix = reinterpret_cast<int64_t*>(ws + L.prefix);
    cudaError_t e;
    if ((e = cudaMemsetAsync(b.dconv_w, 0, sizeof(float) * 3 * a.H * kD * 4, s))) return e;
    if (b.drms_w && (e = cudaMemsetAsync(b.drms_w, 0, sizeof(float) * kD, s))) return e;
    if (b.dconv_state_in &&
        (e = cudaMemsetAsync(b.dconv_state_in, 0, sizeof(float) * a.N * 3 * a.H * kD * 3, s)))
        return e;
    if (rows > 0) {
        if ((e = cudaMemsetAsync(b.dbeta, 0, sizeof(float) * rows, s))) return e;
        if ((e = cudaMemsetAsync(edo, 0, sizeof(float) * rows, s))) return e;
    }
    k_bwd_seg_prefix<<<1, 256, 0, s>>>(a.cu_seqlens, a.N, T, prefix);
    if ((e = cudaGetLastError())) return e;
    const unsigned rb = (unsigned)((rows + 7) / 8);
    if (rows > 0) {
        k_bwd_prep<Tio><<<rb, 256, 0, s>>>(cptr<Tio>(a.q), cptr<Tio>(a.k), cptr<Tio>(a.v), xs, a.conv_w,
                                          cptr<Tio>(a.conv_state_in), a.cu_seqlens, a.N, T, a.H, a.eps_l2, X, nrm);
        if ((e = cudaGetLastError())) return e;
    }
    if ((e = cudaFuncSetAttribute(k_bwd_fwd_cols, cudaFuncAttributeMaxDynamicSharedMemorySize, kColSmem)) ||
        (e = cudaFuncSetAttribute(k_bwd_bwd_cols, cudaFuncAttributeMaxDynamicSharedMemorySize, kColSmem)) ||
        (e = cudaFuncSetAttribute(k_bwd_rows, cudaFuncAttributeMaxDynamicSharedMemorySize, kRowSmem)))
        return e;
    const unsigned cg = (unsigned)(units * kColCtas);
    k_bwd_fwd_cols<<<cg, 128, kColSmem, s>>>(X, a.g, a.beta, a.cu_seqlens, prefix, T, a.H, a.scale,
                                             a.initial_state, O, E, Sck, L.slots, a.d_status);
    if ((e = cudaGetLastError())) return e;
    if (rows > 0) {
        if (a.out_dtype == KDA_FP32)
            k_bwd_epilogue<Tio, float><<<rb, 256, 0, s>>>(O, cptr<float>(b.dy), cptr<Tio>(a.gate), a.rms_w, a.eps_rms,
                                                           rows, b.dgate, b.drms_w);
        else
            k_bwd_epilogue<Tio, bf16><<<rb, 256, 0, s>>>(O, cptr<bf16>(b.dy), cptr<Tio>(a.gate), a.rms_w, a.eps_rms,
                                                          rows, b.dgate, b.drms_w);
        if ((e = cudaGetLastError())) return e;
    }
    k_bwd_bwd_cols<<<cg, 128, kColSmem, s>>>(X, a.g, a.beta, O, E, a.cu_seqlens, prefix, T, a.H, a.scale,
                                             b.d_final_state, W, dX, b.dbeta, edo, dSck, b.dinitial_state,
                                             L.slots);
    if ((e = cudaGetLastError())) return e;
    if (rows == 0) return cudaSuccess;
    k_bwd_rows<<<(unsigned)(units * L.max_seg), kRowThreads, kRowSmem, s>>>(
        X, a.g, a.beta, O, E, W, edo, a.cu_seqlens, prefix, T, a.H, a.scale, (int)L.max_seg, Sck, dSck,
        b.d_final_state, dX, b.dg, segtot, segown, fin, L.slots);
    if ((e = cudaGetLastError())) return e;
    k_bwd_dg_carry<<<(unsigned)units, kD, 0, s>>>(a.cu_seqlens, prefix, T, a.H, fin, segtot, segown, L.slots);
    if ((e = cudaGetLastError())) return e;
    k_bwd_l2<<<rb, 256, 0, s>>>(X, nrm, a.cu_seqlens, prefix, a.N, T, a.H, segtot, E, W, L.slots, dX, b.dg);
    if ((e = cudaGetLastError())) return e;
    const int cblocks = (3 * a.H * kD + 255) / 256;
    const int64_t tiles = (T + kConvTile - 1) / kConvTile;
    k_bwd_conv<Tio><<<(unsigned)(cblocks * tiles), 256, 0, s>>>(
        cptr<Tio>(a.q), cptr<Tio>(a.k), cptr<Tio>(a.v), xs, a.conv_w, cptr<Tio>(a.conv_state_in), a.cu_seqlens,
        a.N, T, a.H, cblocks, dX, b.dq, b.dk, b.dv, b.dconv_w, b.dconv_state_in);
    return cudaGetLastError();
}

size_t al256(size_t x) { return (x + 255) / 256 * 256; }

}  // namespace

BackwardLayout backward_layout(const kda_backward_args& b) {
    const kda_prefill_args& a = b.fwd;
    BackwardLayout L{};
    const size_t T = (size_t)(a.T_total > 0 ? a.T_total : 0), H = (size_t)a.H, HD = H * kD;
    size_t segs = 0, max_seg = 0;
    if (a.cu_seqlens_host)
        for (int n = 0; n < a.N; ++n) {
            const size_t ns = (size_t)(a.cu_seqlens_host[n + 1] - a.cu_seqlens_host[n] + kSeg - 1) / kSeg;
            segs += ns;
            max_seg = ns > max_seg ? ns : max_seg;
        }
    const size_t N = (size_t)(a.N > 0 ? a.N : 0);
    size_t off = 0;
    auto take = [&](size_t bytes) {
        const size_t o = off;
        off += al256(bytes);
        return o;
    };
    L.x = take(T * 3 * HD * 4);
    L.nrm = take(T * H * 2 * 4);
    L.o = take(T * HD * 4);
    L.dx = take(T * 3 * HD * 4);
    L.e = take(T * HD * 4);
    L.w = take(T * HD * 4);
    L.edo = take(T * H * 4);
    L.slots = (int64_t)(segs * H);
    L.max_seg = (int64_t)max_seg;
    L.sck = take(segs * H * kD * kD * 4);
    L.dsck = take(segs * H * kD * kD * 4);
    L.segtot = take(segs * H * kD * 4);
    L.segown = take(segs * H * kD * 4);
    L.fin = take(N * H * kD * 4);
    L.prefix = take((N + 1) * 8);
    L.total = off;
    return L;
}

cudaError_t launch_backward(const kda_backward_args& b, const BackwardLayout& L, char* ws, cudaStream_t s) {
    if ((int64_t)b.fwd.N * b.fwd.H == 0) return cudaSuccess;
    return b.fwd.io == KDA_BF16 ? backward_launch<bf16>(b, L, ws, s) : backward_launch<float>(b, L, ws, s);
}

}  // namespace kda
