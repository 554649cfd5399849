// kda_backward.cu -- the backward pass of the KDA layer (training): reverse-mode
// derivatives of sum(dy . out) + sum(dS . final_state) with respect to every
// input of kda_prefill, D = 128, fp32 arithmetic.
//
// Page "Kimi K3 / Architecture", KDA panel (the layer: short conv + SiLU, L2
// norms of q and k, the recurrent state decayed, corrected and written per
// token, the readout S_t^T q_t, head RMSNorm and the sigmoid gate) and the
// page's training material (the model is trained, so the layer needs its
// derivatives); page "Animated Kimi K3 architecture diagram", LOCAL MEMORY
// section (the four moves, each an affine map of the state, whose adjoints run
// the same steps backwards).
//
// Steps, for each (sequence, head) unit (P = Diag(alpha_t) S_{t-1},
// e = v - P^T k, S_t = P + beta k e^T, o_t = scale S_t^T q):
//   prep       conv + SiLU + L2 norms: q^, k^, v (fp32) and |a_q|, |a_k|   (one warp per token-head)
//   replay     the forward recurrence token by token: o_t, and the state at the start of
//              every kSeg-token segment (checkpoints)                        (one CTA per unit)
//   epilogue   y = n w sig(z), n = o r:  do = r dn - r^3 o (dn . o) / D, dz, dw   (one warp per row)
//   recurrence segments in reverse; each replays its states from its checkpoint into a per-unit
//              scratch, then runs the tokens backwards carrying dS in registers:
//                dS += scale q do^T;  dq = scale S_t do;  w = dS^T k;  dv = beta w;
//                dbeta = w . e;  dk = beta (dS e - P w);  dP = dS - beta k w^T;
//                dg = rowsum(dP . P);  dS <- Diag(alpha) dP                (one CTA per unit)
//   L2         da = (dx - x (x . dx)) / |a|, in place                          (one warp per row)
//   conv       du = da sig(u) (1 + u (1 - sig(u))); dx_{t-3+j} += w_j du_t; dw_j += x_{t-3+j} du_t;
//              positions before the sequence give the conv state's gradient (one thread per
//              (sequence, channel), tokens walked backwards)
// The recurrence kernels hold the state as in the decode kernel: thread (warp w, lane l) owns rows
// 16 w .. 16 w + 15 of columns 4 l .. 4 l + 3; column sums over the rows go through per-warp
// partials in shared memory, row sums over the columns through warp shuffles.
#include "kda_internal.cuh"

namespace kda {

namespace {

constexpr int kD = 128;
constexpr int kSeg = kBwdSeg;  // tokens per checkpointed segment
constexpr int kRecThreads = 256;

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
// Sums 16 per-lane values over the 32 lanes of a warp; afterwards lane l holds the total of
// value (l >> 1) (lanes 2 i and 2 i + 1 both hold value i).
__device__ __forceinline__ float reduce16(float (&v)[16], int lane) {
#pragma unroll
    for (int i = 0; i < 8; ++i) {
        const bool up = (lane & 16) != 0;
        const float send = up ? v[i] : v[i + 8];
        v[i] = (up ? v[i + 8] : v[i]) + __shfl_xor_sync(0xffffffffu, send, 16);
    }
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        const bool up = (lane & 8) != 0;
        const float send = up ? v[i] : v[i + 4];
        v[i] = (up ? v[i + 4] : v[i]) + __shfl_xor_sync(0xffffffffu, send, 8);
    }
#pragma unroll
    for (int i = 0; i < 2; ++i) {
        const bool up = (lane & 4) != 0;
        const float send = up ? v[i] : v[i + 2];
        v[i] = (up ? v[i + 2] : v[i]) + __shfl_xor_sync(0xffffffffu, send, 4);
    }
    {
        const bool up = (lane & 2) != 0;
        const float send = up ? v[0] : v[1];
        v[0] = (up ? v[1] : v[0]) + __shfl_xor_sync(0xffffffffu, send, 2);
    }
    return v[0] + __shfl_xor_sync(0xffffffffu, v[0], 1);
}

// First checkpoint slot of unit (n, h): sequences in order, each holding H runs of its segment
// count.  -1 when the unit's slots would end past `slots` (the host planned the layout from its
// copy of cu_seqlens; a device copy that disagrees must not send writes out of the workspace).
__device__ __forceinline__ int64_t ckpt_base(const int32_t* cu, int n, int64_t T_total, int H, int h,
                                             int64_t slots) {
    int64_t b = 0;
    for (int m = 0; m < n; ++m) {
        int64_t a, e;
        seq_range(cu, m, T_total, a, e);
        b += (e - a + kSeg - 1) / kSeg;
    }
    int64_t a, e;
    seq_range(cu, n, T_total, a, e);
    const int64_t ns = (e - a + kSeg - 1) / kSeg;
    const int64_t base = b * H + (int64_t)h * ns;
    return base + ns <= slots ? base : -1;
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
#pragma unroll
        for (int m = 0; m < 4; ++m) {
            const int d = 4 * lane + m;
            const int64_t ch = (int64_t)part * HD + (int64_t)h * kD + d;
            const float4 w = *reinterpret_cast<const float4*>(conv_w + ch * 4);
            float x[4];
#pragma unroll
            for (int j = 0; j < 4; ++j) {
                const int64_t p = t - 3 + j;
                if (p >= s0) x[j] = to_f(src[part][p * xs + (int64_t)h * kD + d]);
                else x[j] = cs_in ? to_f(cs_in[((int64_t)n * 3 * HD + ch) * 3 + 3 + (p - s0)]) : 0.f;
            }
            const float u = w.x * x[0] + w.y * x[1] + w.z * x[2] + w.w * x[3];
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

// ------------------------------------------------------------------------------ recurrence pieces
// Per-token factors of one unit staged in shared memory: q^, k^, v, alpha, and (backward) do.
struct TokRows {
    float q[kD], k[kD], v[kD], a[kD];
};

// One forward step of the state held by this thread (rows r0 .. r0+15, columns c0 .. c0+3):
// s <- P + beta k e^T with P = Diag(alpha) s and e = v - P^T k.  red: [8][kD] partials.
// Two barriers of the CTA.  Leaves e (this thread's 4 columns) in *e_out.
__device__ __forceinline__ void fwd_step(float4 (&s)[16], const TokRows& tr, float beta, int r0, int c0, int warp,
                                         float (*red)[kD], float4* e_out) {
    float4 cp = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
    for (int i = 0; i < 16; ++i) {
        s[i] = f4_mul(tr.a[r0 + i], s[i]);
        cp = f4_fma(tr.k[r0 + i], s[i], cp);
    }
    *reinterpret_cast<float4*>(&red[warp][c0]) = cp;
    __syncthreads();
    float4 pk = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
    for (int w = 0; w < 8; ++w) pk = f4_add(pk, *reinterpret_cast<const float4*>(&red[w][c0]));
    const float4 vv = *reinterpret_cast<const float4*>(&tr.v[c0]);
    const float4 e = make_float4(vv.x - pk.x, vv.y - pk.y, vv.z - pk.z, vv.w - pk.w);
#pragma unroll
    for (int i = 0; i < 16; ++i) s[i] = f4_fma(beta * tr.k[r0 + i], e, s[i]);
    *e_out = e;
    __syncthreads();  // red is free again
}

// Stages token t's rows (threads 0..127: one channel each).
__device__ __forceinline__ void stage_rows(TokRows& tr, const float* X, const float* g, int64_t t, int H, int h,
                                           int tid) {
    if (tid < kD) {
        const int64_t HD = (int64_t)H * kD;
        const float* xr = X + t * 3 * HD + (int64_t)h * kD + tid;
        tr.q[tid] = xr[0];
        tr.k[tid] = xr[HD];
        tr.v[tid] = xr[2 * HD];
        tr.a[tid] = expf(g[(t * H + h) * kD + tid]);
    }
}

// ------------------------------------------------------------------------------ replay
// The forward recurrence of one unit per CTA: o_t (scale S_t^T q^) for every token into O, and
// the state at the start of every segment into the checkpoints.
__global__ void __launch_bounds__(kRecThreads, 1)
k_bwd_replay(const float* __restrict__ X, const float* __restrict__ g, const float* __restrict__ beta,
             const int32_t* __restrict__ cu, int64_t T_total, int H, float scale, const float* __restrict__ S0,
             float* __restrict__ O, float* __restrict__ ckpt, int64_t slots, int* __restrict__ d_status) {
    __shared__ __align__(16) TokRows tr;
    __shared__ __align__(16) float red[8][kD];
    const int u = blockIdx.x, n = u / H, h = u % H;
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int r0 = 16 * warp, c0 = 4 * lane;
    int64_t s0, s1;
    seq_range(cu, n, T_total, s0, s1);
    const int64_t cb = ckpt_base(cu, n, T_total, H, h, slots);
    if (cb < 0) {
        if (tid == 0) flag_status(d_status, KDA_ERR_DEVICE_ARG);
        return;
    }
    float4 s[16];
#pragma unroll
    for (int i = 0; i < 16; ++i)
        s[i] = S0 ? *reinterpret_cast<const float4*>(S0 + ((int64_t)u * kD + r0 + i) * kD + c0) : make_float4(0.f, 0.f, 0.f, 0.f);
    for (int64_t t = s0; t < s1; ++t) {
        if ((t - s0) % kSeg == 0) {
            float* dst = ckpt + (cb + (t - s0) / kSeg) * kD * kD;
#pragma unroll
            for (int i = 0; i < 16; ++i) *reinterpret_cast<float4*>(dst + (r0 + i) * kD + c0) = s[i];
        }
        stage_rows(tr, X, g, t, H, h, tid);
        __syncthreads();
        float4 e;
        fwd_step(s, tr, beta[t * H + h], r0, c0, warp, red, &e);
        // o = scale S_t^T q^: column sums over the rows
        float4 co = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
        for (int i = 0; i < 16; ++i) co = f4_fma(tr.q[r0 + i], s[i], co);
        *reinterpret_cast<float4*>(&red[warp][c0]) = co;
        __syncthreads();
        if (warp == 0) {
            float4 o = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
            for (int w = 0; w < 8; ++w) o = f4_add(o, *reinterpret_cast<const float4*>(&red[w][c0]));
            *reinterpret_cast<float4*>(O + (t * H + h) * kD + c0) = f4_mul(scale, o);
        }
        __syncthreads();  // red and tr are reused by the next token
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

// ------------------------------------------------------------------------------ recurrence backward
// One unit per CTA; segments in reverse.  For each: replay its states S_{t-1} into the unit's
// scratch (kSeg x D x D), then the tokens backwards.  dS is carried in registers.
// Outputs: dX [T][3][H][D] (dq^, dk^ and dv), dg, dbeta, dS0.
__global__ void __launch_bounds__(kRecThreads, 1)
k_bwd_recurrence(const float* __restrict__ X, const float* __restrict__ g, const float* __restrict__ beta,
                 const float* __restrict__ dO, const int32_t* __restrict__ cu, int64_t T_total, int H, float scale,
                 const float* __restrict__ ckpt, int64_t slots, float* __restrict__ scratch,
                 const float* __restrict__ dS_fin, float* __restrict__ dX, float* __restrict__ dg,
                 float* __restrict__ dbeta, float* __restrict__ dS0) {
    __shared__ __align__(16) TokRows tr;
    __shared__ __align__(16) float sdo[kD];
    __shared__ __align__(16) float red[8][kD];
    __shared__ __align__(16) float red2[8][kD];
    const int u = blockIdx.x, n = u / H, h = u % H;
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int r0 = 16 * warp, c0 = 4 * lane;
    const int64_t HD = (int64_t)H * kD;
    int64_t s0, s1;
    seq_range(cu, n, T_total, s0, s1);
    const int64_t cb = ckpt_base(cu, n, T_total, H, h, slots);
    if (cb < 0) return;  // flagged by the replay
    float* scr = scratch + (int64_t)u * kSeg * kD * kD;
    float4 ds[16];
#pragma unroll
    for (int i = 0; i < 16; ++i)
        ds[i] = dS_fin ? *reinterpret_cast<const float4*>(dS_fin + ((int64_t)u * kD + r0 + i) * kD + c0)
                       : make_float4(0.f, 0.f, 0.f, 0.f);
    const int64_t nseg = (s1 - s0 + kSeg - 1) / kSeg;
    for (int64_t sg = nseg - 1; sg >= 0; --sg) {
        const int64_t ta = s0 + sg * kSeg, tb = (ta + kSeg < s1) ? ta + kSeg : s1;
        // replay: S_{t-1} for t in [ta, tb) into the scratch
        {
            float4 s[16];
            const float* src = ckpt + (cb + sg) * kD * kD;
#pragma unroll
            for (int i = 0; i < 16; ++i) s[i] = *reinterpret_cast<const float4*>(src + (r0 + i) * kD + c0);
            for (int64_t t = ta; t < tb; ++t) {
                float* dst = scr + (t - ta) * kD * kD;
#pragma unroll
                for (int i = 0; i < 16; ++i) *reinterpret_cast<float4*>(dst + (r0 + i) * kD + c0) = s[i];
                if (t + 1 == tb) break;  // the last token's own update is not needed
                stage_rows(tr, X, g, t, H, h, tid);
                __syncthreads();
                float4 e;
                fwd_step(s, tr, beta[t * H + h], r0, c0, warp, red, &e);
            }
        }
        // the tokens backwards
        for (int64_t t = tb - 1; t >= ta; --t) {
            stage_rows(tr, X, g, t, H, h, tid);
            if (tid < kD) sdo[tid] = dO[(t * H + h) * kD + tid];
            __syncthreads();
            const float bt = beta[t * H + h];
            // P = Diag(alpha) S_{t-1};  dS += scale q do^T
            float4 p[16];
            const float* sp = scr + (t - ta) * kD * kD;
            const float4 dov = *reinterpret_cast<const float4*>(&sdo[c0]);
            float4 cp = make_float4(0.f, 0.f, 0.f, 0.f), cw = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
            for (int i = 0; i < 16; ++i) {
                p[i] = f4_mul(tr.a[r0 + i], *reinterpret_cast<const float4*>(sp + (r0 + i) * kD + c0));
                ds[i] = f4_fma(scale * tr.q[r0 + i], dov, ds[i]);
                cp = f4_fma(tr.k[r0 + i], p[i], cp);   // P^T k
                cw = f4_fma(tr.k[r0 + i], ds[i], cw);  // w = dS^T k
            }
            *reinterpret_cast<float4*>(&red[warp][c0]) = cp;
            *reinterpret_cast<float4*>(&red2[warp][c0]) = cw;
            __syncthreads();
            float4 pk = make_float4(0.f, 0.f, 0.f, 0.f), w = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
            for (int ww = 0; ww < 8; ++ww) {
                pk = f4_add(pk, *reinterpret_cast<const float4*>(&red[ww][c0]));
                w = f4_add(w, *reinterpret_cast<const float4*>(&red2[ww][c0]));
            }
            const float4 vv = *reinterpret_cast<const float4*>(&tr.v[c0]);
            const float4 e = make_float4(vv.x - pk.x, vv.y - pk.y, vv.z - pk.z, vv.w - pk.w);
            // dv = beta w (warp 0 writes), dbeta = w . e
            if (warp == 0) {
                *reinterpret_cast<float4*>(dX + t * 3 * HD + 2 * HD + (int64_t)h * kD + c0) = f4_mul(bt, w);
                const float db = warp_sum(dot4(w, e));
                if (lane == 0) dbeta[t * H + h] = db;
            }
            // row sums over the columns: dq = scale S_t do, dk = beta (dS e - P w), dg = rowsum(dP . P)
            float aq[16], ak[16], ag[16];
#pragma unroll
            for (int i = 0; i < 16; ++i) {
                const float kr = tr.k[r0 + i];
                const float4 st = f4_fma(bt * kr, e, p[i]);  // S_t
                aq[i] = dot4(st, dov);
                ak[i] = dot4(ds[i], e) - dot4(p[i], w);
                const float4 dp = f4_fma(-bt * kr, w, ds[i]);
                ag[i] = dot4(dp, p[i]);
                ds[i] = f4_mul(tr.a[r0 + i], dp);  // dS_{t-1}
            }
            const float sq = reduce16(aq, lane), sk = reduce16(ak, lane), sgv = reduce16(ag, lane);
            if ((lane & 1) == 0) {
                const int r = r0 + (lane >> 1);
                float* dxr = dX + t * 3 * HD + (int64_t)h * kD + r;
                dxr[0] = scale * sq;
                dxr[HD] = bt * sk;
                dg[(t * H + h) * kD + r] = sgv;
            }
            __syncthreads();  // tr, sdo, red, red2 are reused by the next token
        }
    }
    if (dS0)
#pragma unroll
        for (int i = 0; i < 16; ++i) *reinterpret_cast<float4*>(dS0 + ((int64_t)u * kD + r0 + i) * kD + c0) = ds[i];
}

// ------------------------------------------------------------------------------ L2 backward
// One warp per (token, head): dq^ -> d a_q = (dq^ - q^ (q^ . dq^)) / |a_q|, same for k, in place.
__global__ void k_bwd_l2(const float* __restrict__ X, const float* __restrict__ nrm, int64_t T_total, int H,
                         float* __restrict__ dX) {
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
        const float4 d = *reinterpret_cast<const float4*>(dX + off);
        const float xd = warp_sum(dot4(x, d));
        const float inv = 1.0f / (part == 0 ? nn.x : nn.y);
        *reinterpret_cast<float4*>(dX + off) = make_float4((d.x - x.x * xd) * inv, (d.y - x.y * xd) * inv,
                                                           (d.z - x.z * xd) * inv, (d.w - x.w * xd) * inv);
    }
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
    for (int64_t t = (tb + 3 < s1 ? tb + 3 : s1) - 1; t >= ta; --t) {
        if (t < s0) {  // crossed the start of sequence n (which lies inside the tile)
            emit_state_grad(du1, du2, du3);
            du1 = du2 = du3 = 0.f;
            while (n > 0) {
                --n;
                seq_range(cu, n, T_total, s0, s1);
                if (s0 <= t) break;
            }
        }
        const float x0 = raw(t - 3), x1 = raw(t - 2), x2 = raw(t - 1), x3 = raw(t);
        const float uu = w.x * x0 + w.y * x1 + w.z * x2 + w.w * x3;
        const float sg = 1.0f / (1.0f + expf(-uu));
        const float du = dA[t * 3 * HD + ch] * sg * (1.0f + uu * (1.0f - sg));
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
    float* ck = reinterpret_cast<float*>(ws + L.ckpt);
    float* scr = reinterpret_cast<float*>(ws + L.scratch);
    cudaError_t e;
    if ((e = cudaMemsetAsync(b.dconv_w, 0, sizeof(float) * 3 * a.H * kD * 4, s))) return e;
    if (b.drms_w && (e = cudaMemsetAsync(b.drms_w, 0, sizeof(float) * kD, s))) return e;
    if (rows > 0) {
        const unsigned rb = (unsigned)((rows + 7) / 8);
        k_bwd_prep<Tio><<<rb, 256, 0, s>>>(cptr<Tio>(a.q), cptr<Tio>(a.k), cptr<Tio>(a.v), xs, a.conv_w,
                                          cptr<Tio>(a.conv_state_in), a.cu_seqlens, a.N, T, a.H, a.eps_l2, X, nrm);
        if ((e = cudaGetLastError())) return e;
    }
    k_bwd_replay<<<(unsigned)units, kRecThreads, 0, s>>>(X, a.g, a.beta, a.cu_seqlens, T, a.H, a.scale,
                                                          a.initial_state, O, ck, L.slots, a.d_status);
    if ((e = cudaGetLastError())) return e;
    if (rows > 0) {
        const unsigned rb = (unsigned)((rows + 7) / 8);
        if (a.out_dtype == KDA_FP32)
            k_bwd_epilogue<Tio, float><<<rb, 256, 0, s>>>(O, cptr<float>(b.dy), cptr<Tio>(a.gate), a.rms_w, a.eps_rms,
                                                           rows, b.dgate, b.drms_w);
        else
            k_bwd_epilogue<Tio, bf16><<<rb, 256, 0, s>>>(O, cptr<bf16>(b.dy), cptr<Tio>(a.gate), a.rms_w, a.eps_rms,
                                                          rows, b.dgate, b.drms_w);
        if ((e = cudaGetLastError())) return e;
    }
    k_bwd_recurrence<<<(unsigned)units, kRecThreads, 0, s>>>(X, a.g, a.beta, O, a.cu_seqlens, T, a.H, a.scale, ck,
                                                              L.slots, scr, b.d_final_state, dX, b.dg, b.dbeta,
                                                              b.dinitial_state);
    if ((e = cudaGetLastError())) return e;
    if (rows > 0) {
        k_bwd_l2<<<(unsigned)((rows + 7) / 8), 256, 0, s>>>(X, nrm, T, a.H, dX);
        if ((e = cudaGetLastError())) return e;
    }
    if (b.dconv_state_in &&
        (e = cudaMemsetAsync(b.dconv_state_in, 0, sizeof(float) * a.N * 3 * a.H * kD * 3, s)))
        return e;
    if (rows == 0) return cudaSuccess;
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
    const size_t T = (size_t)(a.T_total > 0 ? a.T_total : 0), HD = (size_t)a.H * kD;
    size_t segs = 0;
    if (a.cu_seqlens_host)
        for (int n = 0; n < a.N; ++n) segs += (size_t)(a.cu_seqlens_host[n + 1] - a.cu_seqlens_host[n] + kSeg - 1) / kSeg;
    size_t off = 0;
    L.x = off;
    off += al256(T * 3 * HD * 4);
    L.nrm = off;
    off += al256(T * a.H * 2 * 4);
    L.o = off;
    off += al256(T * HD * 4);
    L.dx = off;
    off += al256(T * 3 * HD * 4);
    L.ckpt = off;
    L.slots = (int64_t)(segs * a.H);
    off += al256(segs * a.H * kD * kD * 4);
    L.scratch = off;
    off += al256((size_t)a.N * a.H * kSeg * kD * kD * 4);
    L.total = off;
    return L;
}

cudaError_t launch_backward(const kda_backward_args& b, const BackwardLayout& L, char* ws, cudaStream_t s) {
    if ((int64_t)b.fwd.N * b.fwd.H == 0) return cudaSuccess;
    return b.fwd.io == KDA_BF16 ? backward_launch<bf16>(b, L, ws, s) : backward_launch<float>(b, L, ws, s);
}

}  // namespace kda
