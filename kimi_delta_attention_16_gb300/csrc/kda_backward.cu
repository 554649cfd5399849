// kda_backward.cu -- the backward pass of the KDA layer (training): reverse-mode
// derivatives of sum(dy . out) + sum(dS . final_state) with respect to every
// input of kda_prefill, D = 128, fp32 arithmetic (IEEE exp, SiLU, sigmoid; the
// chunk products on the tensor cores as TF32 hi/lo splits, close to fp32).
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
//   records   per 16-token chunk, all in parallel: decayed keys and queries, the chunk's
//             triangular products and (I + A)^-1 (see "chunk form")          (CTA per chunk-head)
//   forward   the recurrence chunk by chunk: o_t, e_t, and S at the start of every
//             kSeg-token segment                                              (2 CTAs per unit)
//   epilogue  y = n w sig(z), n = o r:  do = r dn - r^3 o (dn . o) / D, dgate, drms_w  (warp per row)
//   backward  the state gradient chunk by chunk, last chunk first: w_t = dS'^T k, dv = beta w,
//             dbeta = w . e, and dS at the end of every segment               (2 CTAs per unit)
//   rows      per (unit, segment), all in parallel, chunk by chunk on tcgen05 with keys as TMEM
//             lanes (with e, w and do known): dq, dk and dg's pieces (see k_bwd_rows_tc)
//   carry     dg's sums over later segments and the final-state term
//   L2        da = (dx - x (x . dx)) / |a|, in place; dg += carry                 (warp per row)
//   conv      du = da sig(u) (1 + u (1 - sig(u))); dx, the taps' and the conv state's gradients
// No token's state is stored: the row kernels replay at most kSeg tokens from the checkpoints.
#include "kda_internal.cuh"
#include "kda_tc_ptx.cuh"

namespace kda {

namespace {

constexpr int kD = 128;
constexpr int kSeg = kBwdSeg;  // tokens per checkpointed segment

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

// ------------------------------------------------------------------------------ staging helpers
// 16-byte and 4-byte asynchronous global -> shared copies (cp.async), one group per staged block.
__device__ __forceinline__ void cp16(void* dst, const void* src) {
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"((uint32_t)__cvta_generic_to_shared(dst)),
                 "l"(src)
                 : "memory");
}
__device__ __forceinline__ void cp_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }
template <int N>
__device__ __forceinline__ void cp_wait() {
    asm volatile("cp.async.wait_group %0;" ::"n"(N) : "memory");
}

// ------------------------------------------------------------------------------ prep
// Conv + SiLU of the q, k, v channels of a head and the L2 norms of q and k, recomputed in fp32.
// X: [T][3][H][D] fp32 (q^, k^, v), nrm: [T][H][2].  One block of 8 warps per (64-token tile,
// head) first stages the tile's raw q, k, v rows t0 - 3 .. t0 + 63 in shared memory with one burst
// of cp.async (51 KB for bf16 inputs, all in flight at once; the C ABI's row rules put every row on
// a 16-byte boundary), then each warp takes every eighth token of the tile (lane l: channels
// 4 l .. 4 l + 3) and reads its windows there.
constexpr int kPrepTile = 64;
constexpr int kPrepRows = kPrepTile + 3;
template <typename Tio>
constexpr uint32_t prep_tile_smem() { return 3u * kPrepRows * kD * (uint32_t)sizeof(Tio); }

template <typename Tio>
__global__ void __launch_bounds__(256, 2)
k_bwd_prep_tile(const Tio* __restrict__ q, const Tio* __restrict__ k, const Tio* __restrict__ v,
                int64_t xs, const float* __restrict__ conv_w, const Tio* __restrict__ cs_in,
                const int32_t* __restrict__ cu, int N, int64_t T_total, int H, float eps_l2,
                float* __restrict__ X, float* __restrict__ nrm) {
    extern __shared__ __align__(16) uint8_t prep_sm[];
    Tio* raw = reinterpret_cast<Tio*>(prep_sm);  // [part][row r][D], row r = token t0 - 3 + r
    __shared__ __align__(16) float wt[3][4][kD];  // [part][tap][channel]
    __shared__ int s_n0;
    const int h = (int)(blockIdx.x % H);
    const int64_t t0 = (int64_t)(blockIdx.x / H) * kPrepTile;
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int64_t HD = (int64_t)H * kD;
    constexpr int kPieces = kD * (int)sizeof(Tio) / 16;  // 16-byte pieces per row
    constexpr int kElems = 16 / (int)sizeof(Tio);
    for (int i = tid; i < 3 * kPrepRows * kPieces; i += blockDim.x) {
        const int part = i / (kPrepRows * kPieces), rem = i - part * (kPrepRows * kPieces);
        const int r = rem / kPieces, c = rem - r * kPieces;
        const int64_t p = t0 - 3 + r;
        const Tio* sp = part == 0 ? q : (part == 1 ? k : v);
        if (p >= 0 && p < T_total)  // rows before 0 lie before every sequence start: replaced below
            cp16(raw + ((size_t)part * kPrepRows + r) * kD + c * kElems, sp + p * xs + (int64_t)h * kD + c * kElems);
    }
    cp_commit();
    for (int i = tid; i < 3 * kD; i += blockDim.x) {
        const int part = i / kD, ch = i - part * kD;
        const float4 w4 = *reinterpret_cast<const float4*>(conv_w + ((int64_t)part * HD + (int64_t)h * kD + ch) * 4);
        wt[part][0][ch] = w4.x;
        wt[part][1][ch] = w4.y;
        wt[part][2][ch] = w4.z;
        wt[part][3][ch] = w4.w;
    }
    if (tid == 0) {  // the sequence of the tile's first token (binary search over cu_seqlens)
        const int64_t tf = t0 < T_total ? t0 : T_total - 1;
        int lo = 0, hi = N;
        while (hi - lo > 1) {
            const int mid = (lo + hi) >> 1;
            if (cu[mid] <= tf) lo = mid;
            else hi = mid;
        }
        s_n0 = lo;
    }
    cp_wait<0>();
    __syncthreads();
    int n = s_n0;
    for (int j = warp; j < kPrepTile; j += 8) {
        const int64_t t = t0 + j;
        if (t >= T_total) break;
        while (n + 1 < N && cu[n + 1] <= t) ++n;  // the sequence of token t
        int64_t s0 = cu[n];
        s0 = s0 < 0 ? 0 : (s0 > t ? t : s0);  // keeps every index in bounds if cu is inconsistent
        const int64_t row = t * H + h;
        float out[3][4];
        float ss[2] = {0.f, 0.f};
#pragma unroll
        for (int part = 0; part < 3; ++part) {
            float x[4][4];  // [token t - 3 + m][channel]
#pragma unroll
            for (int m = 0; m < 4; ++m) {
                const int64_t p = t - 3 + m;
                if (p >= s0) {
                    load4(raw + ((size_t)part * kPrepRows + j + m) * kD + 4 * lane, x[m]);
                } else {
#pragma unroll
                    for (int c = 0; c < 4; ++c) {
                        const int64_t ch = (int64_t)part * HD + (int64_t)h * kD + 4 * lane + c;
                        x[m][c] = cs_in ? to_f(cs_in[((int64_t)n * 3 * HD + ch) * 3 + 3 + (p - s0)]) : 0.f;
                    }
                }
            }
            float w[4][4];  // [tap][channel]
#pragma unroll
            for (int tap = 0; tap < 4; ++tap) {
                const float4 w4 = *reinterpret_cast<const float4*>(&wt[part][tap][4 * lane]);
                w[tap][0] = w4.x;
                w[tap][1] = w4.y;
                w[tap][2] = w4.z;
                w[tap][3] = w4.w;
            }
#pragma unroll
            for (int c = 0; c < 4; ++c) {
                const float u = w[0][c] * x[0][c] + w[1][c] * x[1][c] + w[2][c] * x[2][c] + w[3][c] * x[3][c];
                out[part][c] = __fdividef(u, 1.0f + __expf(-u));  // (u -> -inf: u / inf = 0)
                if (part < 2) ss[part] += out[part][c] * out[part][c];
            }
        }
        const float nq = sqrtf(warp_sum(ss[0]) + eps_l2), nk = sqrtf(warp_sum(ss[1]) + eps_l2);
        const float rq = 1.0f / nq, rk = 1.0f / nk;
        float* xr = X + t * 3 * HD + (int64_t)h * kD + 4 * lane;
        *reinterpret_cast<float4*>(xr) = make_float4(out[0][0] * rq, out[0][1] * rq, out[0][2] * rq, out[0][3] * rq);
        *reinterpret_cast<float4*>(xr + HD) = make_float4(out[1][0] * rk, out[1][1] * rk, out[1][2] * rk, out[1][3] * rk);
        *reinterpret_cast<float4*>(xr + 2 * HD) = make_float4(out[2][0], out[2][1], out[2][2], out[2][3]);
        if (lane == 0) *reinterpret_cast<float2*>(nrm + row * 2) = make_float2(nq, nk);
    }
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

// ------------------------------------------------------------------------------ chunk form
// The forward sweep and the state-gradient sweep in chunks of kCk = 16 tokens.  A chunk's products
// run on the warp-level tensor cores (mma.sync m16n8k8 TF32): tiles of 16 tokens are below what
// tcgen05 takes.  Each operand x is split into hi = tf32(x) and lo = x - hi, and each product takes
// a_lo b_hi + a_hi b_lo + a_hi b_hi, close to fp32 accuracy.
// Per chunk, with G_t the running sum of the chunk's log decays up to token t (per key channel),
// C_t = exp(G_t), C'_t = exp(G_t - G_7) (anchored at the chunk's middle, so that no factor
// leaves e^{+-40} for g >= -5) and B = Diag(beta):
//   Kr_t = C_t k^_t,  Qr_t = C_t q^_t,  Kbar_t = k^_t C_last / C_t,
//   A0_ts = (C'_t k^_t) . (k^_s / C'_s) for s < t,  M0_ts = (C'_t q^_t) . (k^_s / C'_s) for s <= t,
//   T = (I + A0 B)^-1.
// Forward (the decay / probe / correct / write / read steps of the chunk's tokens, unrolled):
//   E = T (V - Kr S),  O = scale (Qr S + M0 B E),  S <- Diag(C_last) S + Kbar^T B E.
// State gradient, D the gradient of the state after the chunk (each token's adjoint unrolled):
//   Y = Kbar D + scale M0^T dO,  dV = T^T B Y,  W = Y - A0^T dV,
//   D <- Diag(C_last) D + Qr^T (scale dO) - Kr^T dV.
// Everything that does not involve the state (the factors, A0, M0, T) is formed for all chunks at
// once by k_bwd_chunk_prep into one record per (chunk, head); the two sweeps read the records.
constexpr int kCk = kBwdChunk;  // tokens per chunk
static_assert(kSeg % kCk == 0, "segments start at chunk starts");
constexpr int kChunksPerSeg = kSeg / kCk;
constexpr int kRecKr = 0, kRecQr = kCk * kD, kRecKb = 2 * kCk * kD, kRecM0 = 3 * kCk * kD,
              kRecA0 = kRecM0 + kCk * kCk, kRecT = kRecA0 + kCk * kCk, kRecCL = kRecT + kCk * kCk,
              kRecBeta = kRecCL + kD, kRec = kRecBeta + kCk;
static_assert(kRec == kBwdRecFloats && kRec % 4 == 0, "record layout");

__device__ __forceinline__ uint32_t tf32_of(float x) {
    uint32_t r;
    asm("cvt.rna.tf32.f32 %0, %1;" : "=r"(r) : "f"(x));
    return r;
}
// hi = tf32(x); lo = x - hi, passed as plain fp32 bits (the tensor core reads the leading 19 bits)
__device__ __forceinline__ void split_tf32(float x, uint32_t& hi, uint32_t& lo) {
    hi = tf32_of(x);
    lo = __float_as_uint(x - __uint_as_float(hi));
}
__device__ __forceinline__ void mma_tf32(float (&c)[4], const uint32_t (&a)[4], const uint32_t (&b)[2]) {
    asm volatile(
        "mma.sync.aligned.m16n8k8.row.col.f32.tf32.tf32.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
        "{%0,%1,%2,%3};"
        : "+f"(c[0]), "+f"(c[1]), "+f"(c[2]), "+f"(c[3])
        : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b[0]), "r"(b[1]));
}
struct Frag4 {
    uint32_t h[4], l[4];
};
struct Frag2 {
    uint32_t h[2], l[2];
};
// Accumulator fragments: lane (g = lane / 4, t = lane % 4) holds (row g, cols 2t, 2t + 1) in c[0], c[1]
// and (row g + 8, same cols) in c[2], c[3].  Such a fragment is an A operand unchanged when the k
// index within the tile is permuted (logical k = t <-> physical col 2 t, k = t + 4 <-> 2 t + 1);
// every B operand below is read with the same permutation.
__device__ __forceinline__ Frag4 afrag_acc(const float (&c)[4]) {
    Frag4 f;
    split_tf32(c[0], f.h[0], f.l[0]);
    split_tf32(c[2], f.h[1], f.l[1]);
    split_tf32(c[1], f.h[2], f.l[2]);
    split_tf32(c[3], f.h[3], f.l[3]);
    return f;
}
// B operand, n = row n0 + g of a row array, k = physical columns c0 + 2 t, c0 + 2 t + 1 (one float2).
__device__ __forceinline__ Frag2 bfrag_rows(const float* base, int stride, int n0, int c0, int g, int t) {
    const float2 x = *reinterpret_cast<const float2*>(base + (n0 + g) * stride + c0 + 2 * t);
    Frag2 f;
    split_tf32(x.x, f.h[0], f.l[0]);
    split_tf32(x.y, f.h[1], f.l[1]);
    return f;
}
// B operand, n = column n0 + g of a row array, k = physical rows r0 + 2 t, r0 + 2 t + 1.
__device__ __forceinline__ Frag2 bfrag_cols(const float* base, int stride, int r0, int n0, int g, int t) {
    Frag2 f;
    split_tf32(base[(r0 + 2 * t) * stride + n0 + g], f.h[0], f.l[0]);
    split_tf32(base[(r0 + 2 * t + 1) * stride + n0 + g], f.h[1], f.l[1]);
    return f;
}
// c += a b, split operands, the small terms first.
__device__ __forceinline__ void mma3(float (&c)[4], const Frag4& a, const Frag2& b) {
    mma_tf32(c, a.l, b.h);
    mma_tf32(c, a.h, b.l);
    mma_tf32(c, a.h, b.h);
}
// The same with the high product in `c` and the two corrections in `d` (two shorter chains).
__device__ __forceinline__ void mma3x(float (&c)[4], float (&d)[4], const Frag4& a, const Frag2& b) {
    mma_tf32(d, a.l, b.h);
    mma_tf32(c, a.h, b.h);
    mma_tf32(d, a.h, b.l);
}

// Record of chunk c of unit (n, h): slot-major, kChunksPerSeg records per checkpoint slot.
__device__ __forceinline__ int64_t rec_index(int64_t sb, int64_t c) { return sb * kChunksPerSeg + c; }

constexpr int kPs = kD + 4;  // row stride of the prep kernel's staged factor rows
// One CTA of 128 threads (thread = key channel) per (unit, chunk); grid units x max_chunks.
__global__ void __launch_bounds__(128)
k_bwd_chunk_prep(const float* __restrict__ X, const float* __restrict__ g, const float* __restrict__ beta,
                 const int32_t* __restrict__ cu, const int64_t* __restrict__ prefix, int64_t T_total, int H,
                 int max_ch, float* __restrict__ Rec, int64_t slots) {
    __shared__ __align__(16) float ka[kCk][kPs], qa[kCk][kPs], ki[kCk][kPs];
    __shared__ float a0[kCk][kCk + 1], bs[kCk];
    const int u = (int)(blockIdx.x / max_ch), c = (int)(blockIdx.x % max_ch), n = u / H, h = u % H;
    int64_t s0, s1;
    seq_range(cu, n, T_total, s0, s1);
    const int64_t nch = (s1 - s0 + kCk - 1) / kCk;
    if (c >= nch) return;
    const int64_t sb = slot_base(prefix, n, H, h, (s1 - s0 + kSeg - 1) / kSeg, slots);
    if (sb < 0) return;  // flagged by the forward sweep
    float* R = Rec + rec_index(sb, c) * kRec;
    const int i = threadIdx.x;
    const int64_t t0 = s0 + (int64_t)c * kCk, HD = (int64_t)H * kD;
    const int nt = (int)(s1 - t0 < kCk ? s1 - t0 : kCk);
    float qv[kCk], kv[kCk], G[kCk];
#pragma unroll
    for (int t = 0; t < kCk; ++t) {
        const bool live = t < nt;
        const int64_t tok = t0 + t;
        qv[t] = live ? X[tok * 3 * HD + (int64_t)h * kD + i] : 0.f;
        kv[t] = live ? X[tok * 3 * HD + HD + (int64_t)h * kD + i] : 0.f;
        G[t] = live ? g[(tok * H + h) * kD + i] : 0.f;
    }
    if (i < kCk) {
        const float b = i < nt ? beta[(t0 + i) * H + h] : 0.f;
        bs[i] = b;
        R[kRecBeta + i] = b;
    }
#pragma unroll
    for (int t = 1; t < kCk; ++t) G[t] += G[t - 1];
    const float gm = G[7], gl = G[kCk - 1];
#pragma unroll
    for (int t = 0; t < kCk; ++t) {
        const float ct = expf(G[t]), ca = expf(G[t] - gm);
        R[kRecKr + t * kD + i] = ct * kv[t];
        R[kRecQr + t * kD + i] = ct * qv[t];
        R[kRecKb + t * kD + i] = kv[t] * expf(gl - G[t]);
        ka[t][i] = ca * kv[t];
        qa[t][i] = ca * qv[t];
        ki[t][i] = kv[t] * expf(gm - G[t]);
    }
    R[kRecCL + i] = expf(gl);
    __syncthreads();
    {  // A0 (threads 0-63) and M0 (64-127): row t, columns s = sq + 4 m
        const int mat = i >> 6, t = (i >> 2) & 15, sq = i & 3;
        const float* xr = mat ? &qa[t][0] : &ka[t][0];
        float acc[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll 4
        for (int c4 = 0; c4 < kD; c4 += 4) {
            const float4 x = *reinterpret_cast<const float4*>(xr + c4);
#pragma unroll
            for (int m = 0; m < 4; ++m) {
                const float4 y = *reinterpret_cast<const float4*>(&ki[sq + 4 * m][c4]);
                acc[m] = fmaf(x.x, y.x, fmaf(x.y, y.y, fmaf(x.z, y.z, fmaf(x.w, y.w, acc[m]))));
            }
        }
#pragma unroll
        for (int m = 0; m < 4; ++m) {
            const int s = sq + 4 * m;
            const float val = (mat ? s <= t : s < t) ? acc[m] : 0.f;
            R[(mat ? kRecM0 : kRecA0) + t * kCk + s] = val;
            if (!mat) a0[t][s] = val;
        }
    }
    __syncthreads();
    if (i < 32) {  // T = (I + A0 B)^-1, right-looking substitution, lane = column j
        const int j = i & 15;
        float ac[kCk];
#pragma unroll
        for (int t = 0; t < kCk; ++t) ac[t] = 0.f;
#pragma unroll
        for (int s2 = 0; s2 < kCk; ++s2) {
            const float ts = (s2 == j ? 1.f : 0.f) - ac[s2];
            if (i < 16) R[kRecT + s2 * kCk + j] = ts;
            const float bts = bs[s2] * ts;
#pragma unroll
            for (int t = s2 + 1; t < kCk; ++t) ac[t] = fmaf(a0[t][s2], bts, ac[t]);
        }
    }
}

constexpr int kChCols = 64;  // value columns per CTA of the sweeps (4 warps x 16)
constexpr int kChCtas = kD / kChCols;
constexpr int kFs = kD + 8;  // rows read as float2 pairs at 8 g + 2 t: no bank conflicts
constexpr int kTs = kCk + 8; // 16-wide matrices read as float2 pairs
constexpr int kTc = kCk + 4; // 16-wide matrices read by column
constexpr int kChV = kChCols + 4;

struct FwdStage {
    float Kr[kCk][kFs], Qr[kCk][kFs];
    float Kb[kCk][kPs];
    float M0[kCk][kTs], T[kCk][kTs];
    float CL[kD], beta[kCk];
    float V[kCk][kChV];
};
constexpr int kFwdSmem = 2 * (int)sizeof(FwdStage);

// Issues the copies of one chunk's record and the CTA's v columns (nt rows, `vsrc` at the chunk's
// first token, rows vstride floats apart).
__device__ __forceinline__ void stage_fwd(FwdStage& st, const float* R, const float* vsrc, int64_t vstride, int nt,
                                          int tid) {
    for (int idx = tid; idx < kCk * (kD / 4); idx += 128) {
        const int r = idx >> 5, c4 = (idx & 31) * 4;
        cp16(&st.Kr[r][c4], R + kRecKr + r * kD + c4);
        cp16(&st.Qr[r][c4], R + kRecQr + r * kD + c4);
        cp16(&st.Kb[r][c4], R + kRecKb + r * kD + c4);
    }
    if (tid < 64) {
        const int r = tid >> 2, c4 = (tid & 3) * 4;
        cp16(&st.M0[r][c4], R + kRecM0 + r * kCk + c4);
        cp16(&st.T[r][c4], R + kRecT + r * kCk + c4);
    } else if (tid < 96) {
        cp16(&st.CL[(tid - 64) * 4], R + kRecCL + (tid - 64) * 4);
    } else if (tid < 100) {
        cp16(&st.beta[(tid - 96) * 4], R + kRecBeta + (tid - 96) * 4);
    }
    for (int idx = tid; idx < nt * (kChCols / 4); idx += 128) {
        const int r = idx >> 4, c4 = (idx & 15) * 4;
        cp16(&st.V[r][c4], vsrc + r * vstride + c4);
    }
}

// Forward sweep in chunks: the recurrence from the initial state; o_t (times scale) and e_t of every
// token; the state at the start of every kSeg-token segment (Sck).  One CTA of 4 warps per (unit,
// 64 value columns); warp w keeps S^T of its 16 columns cw .. cw + 15 as the accumulator fragments
// of 16 key tiles: s[n] = (col g, keys 8 n + 2 t, + 1), (col g + 8, same keys).
__global__ void __launch_bounds__(128, 2)
k_bwd_fwd_chunks(const float* __restrict__ X, const float* __restrict__ Rec, const int32_t* __restrict__ cu,
                 const int64_t* __restrict__ prefix, int64_t T_total, int H, float scale,
                 const float* __restrict__ S0, float* __restrict__ O, float* __restrict__ E,
                 float* __restrict__ Sck, int64_t slots, int* __restrict__ d_status) {
    extern __shared__ __align__(16) unsigned char smem_raw[];
    FwdStage* stg = reinterpret_cast<FwdStage*>(smem_raw);
    const int u = blockIdx.x / kChCtas, cq = blockIdx.x % kChCtas, n = u / H, h = u % H;
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31, gq = lane >> 2, tq = lane & 3;
    const int cl = 16 * warp, cw = cq * kChCols + cl;  // the warp's first column in the CTA / the head
    int64_t s0, s1;
    seq_range(cu, n, T_total, s0, s1);
    const int64_t sb = slot_base(prefix, n, H, h, (s1 - s0 + kSeg - 1) / kSeg, slots);
    if (sb < 0) {
        if (tid == 0) flag_status(d_status, KDA_ERR_DEVICE_ARG);
        return;
    }
    const int64_t HD = (int64_t)H * kD;
    float s[16][4];
    if (S0) {
        const float* S = S0 + (int64_t)u * kD * kD + cw + gq;
#pragma unroll
        for (int nt = 0; nt < 16; ++nt) {
            const int r = 8 * nt + 2 * tq;
            s[nt][0] = S[r * kD];
            s[nt][1] = S[(r + 1) * kD];
            s[nt][2] = S[r * kD + 8];
            s[nt][3] = S[(r + 1) * kD + 8];
        }
    } else {
#pragma unroll
        for (int nt = 0; nt < 16; ++nt) s[nt][0] = s[nt][1] = s[nt][2] = s[nt][3] = 0.f;
    }
    const int64_t nch = (s1 - s0 + kCk - 1) / kCk;
    auto nt_of = [&](int64_t c) { return (int)(s1 - (s0 + c * kCk) < kCk ? s1 - (s0 + c * kCk) : kCk); };
    const float* vb = X + 2 * HD + (int64_t)h * kD + cq * kChCols;
    if (nch > 0) stage_fwd(stg[0], Rec + rec_index(sb, 0) * kRec, vb + s0 * 3 * HD, 3 * HD, nt_of(0), tid);
    cp_commit();
    for (int64_t c = 0; c < nch; ++c) {
        const int nt = nt_of(c);
        const int64_t t0 = s0 + c * kCk;
        const FwdStage& st = stg[c & 1];
        if (c % kChunksPerSeg == 0) {  // the state at the start of a segment
            float* S = Sck + (sb + c / kChunksPerSeg) * kD * kD + cw + gq;
#pragma unroll
            for (int nt2 = 0; nt2 < 16; ++nt2) {
                const int r = 8 * nt2 + 2 * tq;
                S[r * kD] = s[nt2][0];
                S[(r + 1) * kD] = s[nt2][1];
                S[r * kD + 8] = s[nt2][2];
                S[(r + 1) * kD + 8] = s[nt2][3];
            }
        }
        cp_wait<0>();
        __syncthreads();  // chunk c has landed; chunk c - 1's buffer is free
        if (c + 1 < nch)
            stage_fwd(stg[(c + 1) & 1], Rec + rec_index(sb, c + 1) * kRec, vb + (t0 + kCk) * 3 * HD, 3 * HD,
                      nt_of(c + 1), tid);
        cp_commit();
        // R^T = S^T Kr^T, (Qr S)^T = S^T Qr^T; tokens as two n tiles
        float r[2][4], rc[2][4], p[2][4], pc[2][4];
#pragma unroll
        for (int j = 0; j < 2; ++j)
#pragma unroll
            for (int e = 0; e < 4; ++e) r[j][e] = rc[j][e] = p[j][e] = pc[j][e] = 0.f;
#pragma unroll
        for (int kk = 0; kk < 16; ++kk) {
            const Frag4 a = afrag_acc(s[kk]);
#pragma unroll
            for (int j = 0; j < 2; ++j) {
                mma3x(r[j], rc[j], a, bfrag_rows(&st.Kr[0][0], kFs, 8 * j, 8 * kk, gq, tq));
                mma3x(p[j], pc[j], a, bfrag_rows(&st.Qr[0][0], kFs, 8 * j, 8 * kk, gq, tq));
            }
        }
        // X = V - R; E = T X; Eb = B E
        float x[2][4];
#pragma unroll
        for (int j = 0; j < 2; ++j) {
            const int tk = 8 * j + 2 * tq;
            const bool l0 = tk < nt, l1 = tk + 1 < nt;
            x[j][0] = (l0 ? st.V[tk][cl + gq] : 0.f) - (r[j][0] + rc[j][0]);
            x[j][1] = (l1 ? st.V[tk + 1][cl + gq] : 0.f) - (r[j][1] + rc[j][1]);
            x[j][2] = (l0 ? st.V[tk][cl + gq + 8] : 0.f) - (r[j][2] + rc[j][2]);
            x[j][3] = (l1 ? st.V[tk + 1][cl + gq + 8] : 0.f) - (r[j][3] + rc[j][3]);
        }
        float e[2][4];
        {
            const Frag4 x0 = afrag_acc(x[0]), x1 = afrag_acc(x[1]);
#pragma unroll
            for (int q4 = 0; q4 < 4; ++q4) e[0][q4] = e[1][q4] = 0.f;
            mma3(e[0], x0, bfrag_rows(&st.T[0][0], kTs, 0, 0, gq, tq));
            mma3(e[1], x0, bfrag_rows(&st.T[0][0], kTs, 8, 0, gq, tq));
            mma3(e[1], x1, bfrag_rows(&st.T[0][0], kTs, 8, 8, gq, tq));
        }
        float eb[2][4];
#pragma unroll
        for (int j = 0; j < 2; ++j) {
            const float2 b2 = *reinterpret_cast<const float2*>(&st.beta[8 * j + 2 * tq]);
            eb[j][0] = b2.x * e[j][0];
            eb[j][1] = b2.y * e[j][1];
            eb[j][2] = b2.x * e[j][2];
            eb[j][3] = b2.y * e[j][3];
        }
        const Frag4 e0 = afrag_acc(eb[0]), e1 = afrag_acc(eb[1]);
        {  // O = scale (Qr S + M0 Eb)
            float o[2][4];
#pragma unroll
            for (int j = 0; j < 2; ++j)
#pragma unroll
                for (int q4 = 0; q4 < 4; ++q4) o[j][q4] = p[j][q4] + pc[j][q4];
            mma3(o[0], e0, bfrag_rows(&st.M0[0][0], kTs, 0, 0, gq, tq));
            mma3(o[1], e0, bfrag_rows(&st.M0[0][0], kTs, 8, 0, gq, tq));
            mma3(o[1], e1, bfrag_rows(&st.M0[0][0], kTs, 8, 8, gq, tq));
#pragma unroll
            for (int j = 0; j < 2; ++j) {
                const int tk = 8 * j + 2 * tq;
                if (tk < nt) {
                    const int64_t off = ((t0 + tk) * H + h) * kD + cw + gq;
                    O[off] = scale * o[j][0];
                    O[off + 8] = scale * o[j][2];
                    E[off] = e[j][0];
                    E[off + 8] = e[j][2];
                }
                if (tk + 1 < nt) {
                    const int64_t off = ((t0 + tk + 1) * H + h) * kD + cw + gq;
                    O[off] = scale * o[j][1];
                    O[off + 8] = scale * o[j][3];
                    E[off] = e[j][1];
                    E[off + 8] = e[j][3];
                }
            }
        }
        // S <- Diag(C_last) S + Kbar^T Eb
#pragma unroll
        for (int nt2 = 0; nt2 < 16; ++nt2) {
            const float2 c2 = *reinterpret_cast<const float2*>(&st.CL[8 * nt2 + 2 * tq]);
            s[nt2][0] *= c2.x;
            s[nt2][1] *= c2.y;
            s[nt2][2] *= c2.x;
            s[nt2][3] *= c2.y;
            mma3(s[nt2], e0, bfrag_cols(&st.Kb[0][0], kPs, 0, 8 * nt2, gq, tq));
            mma3(s[nt2], e1, bfrag_cols(&st.Kb[0][0], kPs, 8, 8 * nt2, gq, tq));
        }
    }
}

struct BwdStage {
    float Kb[kCk][kFs];
    float Qr[kCk][kPs], Kr[kCk][kPs];
    float M0[kCk][kTc], A0[kCk][kTc], T[kCk][kTc];
    float CL[kD], beta[kCk];
    float dO[kCk][kChV], E[kCk][kChV];
};
constexpr int kBwdSmem = 2 * (int)sizeof(BwdStage);

__device__ __forceinline__ void stage_bwd(BwdStage& st, const float* R, const float* dosrc, const float* esrc,
                                          int64_t stride, int nt, int tid) {
    for (int idx = tid; idx < kCk * (kD / 4); idx += 128) {
        const int r = idx >> 5, c4 = (idx & 31) * 4;
        cp16(&st.Kb[r][c4], R + kRecKb + r * kD + c4);
        cp16(&st.Qr[r][c4], R + kRecQr + r * kD + c4);
        cp16(&st.Kr[r][c4], R + kRecKr + r * kD + c4);
    }
    if (tid < 64) {
        const int r = tid >> 2, c4 = (tid & 3) * 4;
        cp16(&st.M0[r][c4], R + kRecM0 + r * kCk + c4);
        cp16(&st.A0[r][c4], R + kRecA0 + r * kCk + c4);
        cp16(&st.T[r][c4], R + kRecT + r * kCk + c4);
    } else if (tid < 96) {
        cp16(&st.CL[(tid - 64) * 4], R + kRecCL + (tid - 64) * 4);
    } else if (tid < 100) {
        cp16(&st.beta[(tid - 96) * 4], R + kRecBeta + (tid - 96) * 4);
    }
    for (int idx = tid; idx < nt * (kChCols / 4); idx += 128) {
        const int r = idx >> 4, c4 = (idx & 15) * 4;
        cp16(&st.dO[r][c4], dosrc + r * stride + c4);
        cp16(&st.E[r][c4], esrc + r * stride + c4);
    }
}

// State-gradient sweep in chunks, last chunk first: w_t = dS'^T k^_t, dv = beta w, the sum
// dbeta = w . e of every token (atomics over the CTAs of a unit), the state gradient at
// the end of every segment (dSck: before that token's own terms) and at the start (dS0).  Layout as
// in k_bwd_fwd_chunks, with D = dS in place of S.
__global__ void __launch_bounds__(128, 2)
k_bwd_bwd_chunks(const float* __restrict__ Rec, const float* __restrict__ dO, const float* __restrict__ E,
                 const int32_t* __restrict__ cu, const int64_t* __restrict__ prefix, int64_t T_total, int H,
                 float scale, const float* __restrict__ dS_fin, float* __restrict__ W, float* __restrict__ dX,
                 float* __restrict__ dbeta, float* __restrict__ dSck, float* __restrict__ dS0, int64_t slots) {
    extern __shared__ __align__(16) unsigned char smem_raw[];
    BwdStage* stg = reinterpret_cast<BwdStage*>(smem_raw);
    __shared__ float acc[2][kCk];  // [chunk parity][token]: dbeta
    const int u = blockIdx.x / kChCtas, cq = blockIdx.x % kChCtas, n = u / H, h = u % H;
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31, gq = lane >> 2, tq = lane & 3;
    const int cl = 16 * warp, cw = cq * kChCols + cl;
    if (tid < 2 * kCk) (&acc[0][0])[tid] = 0.f;
    int64_t s0, s1;
    seq_range(cu, n, T_total, s0, s1);
    const int64_t sb = slot_base(prefix, n, H, h, (s1 - s0 + kSeg - 1) / kSeg, slots);
    if (sb < 0) return;  // flagged by the forward sweep
    const int64_t HD = (int64_t)H * kD;
    float d[16][4];
    if (dS_fin) {
        const float* S = dS_fin + (int64_t)u * kD * kD + cw + gq;
#pragma unroll
        for (int nt = 0; nt < 16; ++nt) {
            const int r = 8 * nt + 2 * tq;
            d[nt][0] = S[r * kD];
            d[nt][1] = S[(r + 1) * kD];
            d[nt][2] = S[r * kD + 8];
            d[nt][3] = S[(r + 1) * kD + 8];
        }
    } else {
#pragma unroll
        for (int nt = 0; nt < 16; ++nt) d[nt][0] = d[nt][1] = d[nt][2] = d[nt][3] = 0.f;
    }
    const int64_t nch = (s1 - s0 + kCk - 1) / kCk;
    auto nt_of = [&](int64_t c) { return (int)(s1 - (s0 + c * kCk) < kCk ? s1 - (s0 + c * kCk) : kCk); };
    const int64_t coff = (int64_t)h * kD + cq * kChCols;
    auto stage = [&](int64_t c) {
        const int64_t t0 = s0 + c * kCk;
        stage_bwd(stg[c & 1], Rec + rec_index(sb, c) * kRec, dO + t0 * HD + coff, E + t0 * HD + coff, HD,
                  nt_of(c), tid);
    };
    if (nch > 0) stage(nch - 1);
    cp_commit();
    for (int64_t c = nch - 1; c >= 0; --c) {
        const int nt = nt_of(c);
        const int64_t t0 = s0 + c * kCk;
        const BwdStage& st = stg[c & 1];
        if (c % kChunksPerSeg == kChunksPerSeg - 1 || c == nch - 1) {  // the chunk ends a segment
            float* S = dSck + (sb + c / kChunksPerSeg) * kD * kD + cw + gq;
#pragma unroll
            for (int nt2 = 0; nt2 < 16; ++nt2) {
                const int r = 8 * nt2 + 2 * tq;
                S[r * kD] = d[nt2][0];
                S[(r + 1) * kD] = d[nt2][1];
                S[r * kD + 8] = d[nt2][2];
                S[(r + 1) * kD + 8] = d[nt2][3];
            }
        }
        cp_wait<0>();
        __syncthreads();  // chunk c has landed; chunk c + 1's buffer and sums are complete
        if (c + 1 < nch && tid < nt_of(c + 1)) {
            const int p = (int)((c + 1) & 1);
            const int64_t t = s0 + (c + 1) * kCk + tid;
            atomicAdd(dbeta + t * H + h, acc[p][tid]);
            acc[p][tid] = 0.f;
        }
        if (c > 0) stage(c - 1);
        cp_commit();
        // Y^T = D^T Kbar^T + scale dO^T M0 (tokens as two n tiles)
        float y[2][4], yc[2][4];
#pragma unroll
        for (int j = 0; j < 2; ++j)
#pragma unroll
            for (int e = 0; e < 4; ++e) y[j][e] = yc[j][e] = 0.f;
#pragma unroll
        for (int kk = 0; kk < 16; ++kk) {
            const Frag4 a = afrag_acc(d[kk]);
#pragma unroll
            for (int j = 0; j < 2; ++j) mma3x(y[j], yc[j], a, bfrag_rows(&st.Kb[0][0], kFs, 8 * j, 8 * kk, gq, tq));
        }
        Frag4 sdo[2];  // scale dO^T as A operands (k = tokens 8 kj ..), rows past the sequence zero
#pragma unroll
        for (int kj = 0; kj < 2; ++kj) {
            const int tk = 8 * kj + 2 * tq;
            const bool l0 = tk < nt, l1 = tk + 1 < nt;
            const float v[4] = {l0 ? scale * st.dO[tk][cl + gq] : 0.f, l1 ? scale * st.dO[tk + 1][cl + gq] : 0.f,
                                l0 ? scale * st.dO[tk][cl + gq + 8] : 0.f,
                                l1 ? scale * st.dO[tk + 1][cl + gq + 8] : 0.f};
            sdo[kj] = afrag_acc(v);
        }
#pragma unroll
        for (int j = 0; j < 2; ++j)
#pragma unroll
            for (int e = 0; e < 4; ++e) y[j][e] += yc[j][e];
        mma3(y[0], sdo[0], bfrag_cols(&st.M0[0][0], kTc, 0, 0, gq, tq));
        mma3(y[0], sdo[1], bfrag_cols(&st.M0[0][0], kTc, 8, 0, gq, tq));
        mma3(y[1], sdo[1], bfrag_cols(&st.M0[0][0], kTc, 8, 8, gq, tq));
        // dV^T = (B Y)^T T, W^T = Y^T - dV^T A0
        float dv[2][4], w[2][4];
        {
            float yb[2][4];
#pragma unroll
            for (int j = 0; j < 2; ++j) {
                const float2 b2 = *reinterpret_cast<const float2*>(&st.beta[8 * j + 2 * tq]);
                yb[j][0] = b2.x * y[j][0];
                yb[j][1] = b2.y * y[j][1];
                yb[j][2] = b2.x * y[j][2];
                yb[j][3] = b2.y * y[j][3];
            }
            const Frag4 y0 = afrag_acc(yb[0]), y1 = afrag_acc(yb[1]);
#pragma unroll
            for (int e = 0; e < 4; ++e) dv[0][e] = dv[1][e] = 0.f;
            mma3(dv[0], y0, bfrag_cols(&st.T[0][0], kTc, 0, 0, gq, tq));
            mma3(dv[0], y1, bfrag_cols(&st.T[0][0], kTc, 8, 0, gq, tq));
            mma3(dv[1], y1, bfrag_cols(&st.T[0][0], kTc, 8, 8, gq, tq));
        }
        Frag4 ndv[2];
#pragma unroll
        for (int j = 0; j < 2; ++j) {
            const float nv[4] = {-dv[j][0], -dv[j][1], -dv[j][2], -dv[j][3]};
            ndv[j] = afrag_acc(nv);
#pragma unroll
            for (int e = 0; e < 4; ++e) w[j][e] = y[j][e];
        }
        mma3(w[0], ndv[0], bfrag_cols(&st.A0[0][0], kTc, 0, 0, gq, tq));
        mma3(w[0], ndv[1], bfrag_cols(&st.A0[0][0], kTc, 8, 0, gq, tq));
        mma3(w[1], ndv[1], bfrag_cols(&st.A0[0][0], kTc, 8, 8, gq, tq));
        // stores and the per-token sums w . e over the warp's 16 columns
        {
            float pb[2][2];
#pragma unroll
            for (int j = 0; j < 2; ++j)
#pragma unroll
                for (int hlf = 0; hlf < 2; ++hlf) {
                    const int tk = 8 * j + 2 * tq + hlf;
                    pb[j][hlf] = 0.f;
                    if (tk < nt) {
                        const float e0 = st.E[tk][cl + gq], e1 = st.E[tk][cl + gq + 8];
                        const float w0 = w[j][hlf], w1 = w[j][2 + hlf];
                        pb[j][hlf] = w0 * e0 + w1 * e1;
                        const int64_t t = t0 + tk;
                        const int64_t off = (t * H + h) * kD + cw + gq;
                        W[off] = w0;
                        W[off + 8] = w1;
                        float* dv_row = dX + t * 3 * HD + 2 * HD + (int64_t)h * kD + cw + gq;
                        dv_row[0] = dv[j][hlf];
                        dv_row[8] = dv[j][2 + hlf];
                    }
                }
#pragma unroll
            for (int j = 0; j < 2; ++j)
#pragma unroll
                for (int hlf = 0; hlf < 2; ++hlf)
#pragma unroll
                    for (int off = 4; off < 32; off <<= 1) pb[j][hlf] += __shfl_xor_sync(0xffffffffu, pb[j][hlf], off);
            if (gq == 0) {
                const int p = (int)(c & 1);
#pragma unroll
                for (int j = 0; j < 2; ++j)
#pragma unroll
                    for (int hlf = 0; hlf < 2; ++hlf) {
                        const int tk = 8 * j + 2 * tq + hlf;
                        if (tk < nt) atomicAdd(&acc[p][tk], pb[j][hlf]);
                    }
            }
        }
        // D <- Diag(C_last) D + Qr^T (scale dO) - Kr^T dV
#pragma unroll
        for (int nt2 = 0; nt2 < 16; ++nt2) {
            const float2 c2 = *reinterpret_cast<const float2*>(&st.CL[8 * nt2 + 2 * tq]);
            d[nt2][0] *= c2.x;
            d[nt2][1] *= c2.y;
            d[nt2][2] *= c2.x;
            d[nt2][3] *= c2.y;
#pragma unroll
            for (int kj = 0; kj < 2; ++kj) {
                mma3(d[nt2], sdo[kj], bfrag_cols(&st.Qr[0][0], kPs, 8 * kj, 8 * nt2, gq, tq));
                mma3(d[nt2], ndv[kj], bfrag_cols(&st.Kr[0][0], kPs, 8 * kj, 8 * nt2, gq, tq));
            }
        }
    }
    __syncthreads();
    if (nch > 0 && tid < nt_of(0)) {
        const int64_t t = s0 + tid;
        atomicAdd(dbeta + t * H + h, acc[0][tid]);
    }
    if (dS0) {
        float* S = dS0 + (int64_t)u * kD * kD + cw + gq;
#pragma unroll
        for (int nt2 = 0; nt2 < 16; ++nt2) {
            const int r = 8 * nt2 + 2 * tq;
            S[r * kD] = d[nt2][0];
            S[(r + 1) * kD] = d[nt2][1];
            S[r * kD + 8] = d[nt2][2];
            S[(r + 1) * kD + 8] = d[nt2][3];
        }
    }
}

// ------------------------------------------------------------------------------ tcgen05 chunk sweeps
// The same chunk algebra with the products on the 5th-generation tensor cores (tcgen05.mma
// kind::tf32, accumulators in tensor memory).  One CTA of 4 warps per unit: thread j owns value
// column j, which is TMEM lane j.  M = 128 value columns; the state (S^T, lanes = columns,
// TMEM columns = keys) stays in TMEM as the accumulator of the update and, split into its TF32
// high part and remainder, as the A operand of the reads.  B operands are K-major tiles with the
// 128-byte swizzle (32 fp32 per row), built by the threads from the plain records one chunk ahead
// while the tensor core runs; both hi and lo parts (3 MMA terms per product, as above).
namespace tcs {
using namespace kda::tc;

__host__ __device__ constexpr uint32_t idesc_tf32(int M, int N) {
    return (1u << 4)                      // D: fp32
           | (2u << 7) | (2u << 10)       // A, B: tf32 (both K-major)
           | ((uint32_t)(N >> 3) << 17) | ((uint32_t)(M >> 4) << 24);
}
// D[tmem] (+)= A[tmem] * B[smem]^T, kind::tf32
__device__ __forceinline__ void mma_tf32_ts(uint32_t d, uint32_t a, uint64_t b, uint32_t id, uint32_t acc) {
    asm volatile(
        "{\n\t.reg .pred p;\n\tsetp.ne.b32 p, %4, 0;\n\t"
        "tcgen05.mma.cta_group::1.kind::tf32 [%0], [%1], %2, %3, p;\n\t}" ::"r"(d),
        "r"(a), "l"(b), "r"(id), "r"(acc)
        : "memory");
}
// Byte offset of fp32 elements (r, k .. k + 3), k % 4 == 0, in a K-major 128-byte-swizzled tile of
// `rows` rows: K-blocks of 32 elements, each rows x 128 bytes; within an 8-row atom the 16-byte
// chunk c of row r sits at chunk position c ^ (r % 8).
__device__ __forceinline__ uint32_t kmaj(int rows, int r, int k) {
    return (uint32_t)((k >> 5) * rows * 128 + r * 128 + ((((k & 31) >> 2) ^ (r & 7)) << 4));
}
// B descriptor for K-step ks (8 elements) of a K-major tile of `rows` rows.
__device__ __forceinline__ uint64_t bdesc(uint32_t base, int rows, int ks) {
    return desc_sw128(base + (uint32_t)((ks >> 2) * rows * 128 + (ks & 3) * 32), 16, 1024);
}
__device__ __forceinline__ float4 hi4(float4 x, float4& lo) {
    float4 h;
    h.x = __uint_as_float(tf32_of(x.x));
    h.y = __uint_as_float(tf32_of(x.y));
    h.z = __uint_as_float(tf32_of(x.z));
    h.w = __uint_as_float(tf32_of(x.w));
    lo = make_float4(x.x - h.x, x.y - h.y, x.z - h.z, x.w - h.w);
    return h;
}
__device__ __forceinline__ void sts128(unsigned char* base, uint32_t off, float4 v) {
    *reinterpret_cast<float4*>(base + off) = v;
}
// Waits on an MMA barrier: lane 0 of each warp polls (bounded), the warp follows.
__device__ __forceinline__ bool warp_wait(uint64_t* bar, uint32_t parity) {
    bool ok = true;
    if ((threadIdx.x & 31) == 0) ok = mbar_wait(bar, parity);
    ok = __shfl_sync(0xffffffffu, ok ? 1 : 0, 0) != 0;
    fence_after_sync();
    return ok;
}
// 32 consecutive TMEM columns of the thread's lane <-> registers.
__device__ __forceinline__ void tld32(uint32_t ta, float (&v)[32]) {
    uint32_t r[32];
    tmem_ld32(ta, r);
    tmem_ld_wait();
#pragma unroll
    for (int i = 0; i < 32; ++i) v[i] = __uint_as_float(r[i]);
}
__device__ __forceinline__ void tst32(uint32_t ta, const float (&v)[32]) {
    uint32_t a[16], b[16];
#pragma unroll
    for (int i = 0; i < 16; ++i) {
        a[i] = __float_as_uint(v[i]);
        b[i] = __float_as_uint(v[16 + i]);
    }
    tmem_st16(ta, a);
    tmem_st16(ta + 16, b);
}
__device__ __forceinline__ void tst16(uint32_t ta, const float (&v)[16]) {
    uint32_t a[16];
#pragma unroll
    for (int i = 0; i < 16; ++i) a[i] = __float_as_uint(v[i]);
    tmem_st16(ta, a);
}
}  // namespace tcs

// ------------------------------------------------------------------------------ tcgen05 row sweeps
// The row kernel's quantities in chunk form, per (unit, 64-token segment), with S_c the state at a
// chunk's start (from the segment's checkpoint, carried forward) and D the state gradient at its end
// (from the segment's checkpoint, carried backward); per token t of the chunk, with C, C', B as in
// the records and the chunk's Grams P = E dO^T, Q = E W^T (16 x 16):
//   dq_t   = scale (C_t (S_c do_t) + C'_t sum_{s<=t} beta_s P_st k^_s / C'_s),
//   dkr_t  = -beta_t (C_t (S_c w_t) + C'_t sum_{s<t} beta_s Q_st k^_s / C'_s),
//   dkw_t  = beta_t ((C_last / C_t) (D e_t) + (1 / C'_t) (sum_{tau>=t} scale P_t,tau C'_tau q^_tau
//                                                  - sum_{tau>t} beta_tau Q_t,tau C'_tau k^_tau)),
//   S_{c+1} = Diag(C_last) S_c + Kbar^T B E,   D <- Diag(C_last) D + Qr^T (scale dO) - Kr^T B W
// (each token's forward and adjoint steps unrolled; checked against the token loop in fp64 before
// it was written).  The products S_c [dO; W]^T (N = 32), D E^T (N = 16) and the two updates
// (N = 128) run on tcgen05 (kind::tf32, hi/lo terms); keys are TMEM lanes.  8 warps: warps w and
// w + 4 share lanes 32 (w % 4) ..; the per-token vector work is split between them.
// dg follows from the decay entering only through e^{Gamma_t} (read keys and queries) and
// e^{-Gamma_t} (written keys), Gamma_t = sum_{s <= t} g_s:
//   dGamma_t = q^ dq + k^ dk_read - k^ dk_write,  dg_t = sum_{s >= t} dGamma_s + rowsum(dS_T . S_T);
// here the parts within the segment: dg <- -(sum of q dq + k dk_read over earlier tokens), the global
// rows of e and w (staged, so free) <- dk_write and the suffix sums of -k dk_write; per segment its sum
// of dGamma (segtot) and of the read part (segown); for the last segment of a sequence the final-state
// term (fin).
constexpr int kRtThreads = 256;
constexpr int kRs = kD + 4;  // row stride of the staged E, dO, W rows (conflict-free Gram reads)
struct RtStage {
    float E[kCk][kRs], DO[kCk][kRs], W[kCk][kRs];
    float q[kCk][kD], k[kCk][kD], g[kCk][kD], R1[kCk][kD], R2[kCk][kD];
    float CL[kD], beta[kCk];
};
struct RowsTcSmem {
    unsigned char b1h[16384], b1l[16384];  // fwd: [dO; W] (32 x 128); bwd: E (16 x 128); K-major
    unsigned char b2h[16384], b2l[16384];  // fwd: (B E)^T (128 x 16); bwd: [scale dO; -B W]^T (128 x 32)
    RtStage st[2];
    float P[kChunksPerSeg][kCk][kCk], Q[kChunksPerSeg][kCk][kCk];
    float xch[kCk][kD];
    uint64_t barP, barU;
    uint32_t tbase;
    int fail;
};
constexpr int kRowsTcSmem = (int)sizeof(RowsTcSmem) + 1024;
static_assert(kRowsTcSmem <= 227 * 1024, "rows kernel shared memory");

// Issues the copies of one chunk: rows t0 .. t0 + nt - 1 of E, dO, W, q^, k^, g; two record rows
// (r1, r2 offsets in the record; r2 < 0: none), C_last and beta.  Run by 224 threads (q = 0 .. 223):
// q < 192 owns one (row kind, 16-byte column) and walks the rows; the last 32 the record rows.
__device__ __forceinline__ void rt_stage(RtStage& s, const float* X, const float* g, const float* E, const float* dO,
                                         const float* W, const float* R, int r1, int r2, int64_t t0, int nt, int H,
                                         int h, int q) {
    const int64_t HD = (int64_t)H * kD;
    const int c4 = (q & 31) * 4;
    if (q < 192) {
        const int part = q >> 5;
        const float* src;
        int64_t step;
        float* dst;
        int dstep;
        switch (part) {
            case 0: src = E + (t0 * H + h) * kD; step = HD; dst = &s.E[0][0]; dstep = kRs; break;
            case 1: src = dO + (t0 * H + h) * kD; step = HD; dst = &s.DO[0][0]; dstep = kRs; break;
            case 2: src = W + (t0 * H + h) * kD; step = HD; dst = &s.W[0][0]; dstep = kRs; break;
            case 3: src = X + t0 * 3 * HD + (int64_t)h * kD; step = 3 * HD; dst = &s.q[0][0]; dstep = kD; break;
            case 4: src = X + t0 * 3 * HD + HD + (int64_t)h * kD; step = 3 * HD; dst = &s.k[0][0]; dstep = kD; break;
            default: src = g + (t0 * H + h) * kD; step = HD; dst = &s.g[0][0]; dstep = kD; break;
        }
        src += c4;
        dst += c4;
        for (int row = 0; row < nt; ++row, src += step, dst += dstep) cp16(dst, src);
    } else {
#pragma unroll 4
        for (int row = 0; row < kCk; ++row) {
            cp16(&s.R1[row][c4], R + r1 + row * kD + c4);
            if (r2 >= 0) cp16(&s.R2[row][c4], R + r2 + row * kD + c4);
        }
        cp16(&s.CL[c4], R + kRecCL + c4);
        if (q < 196) cp16(&s.beta[4 * (q - 192)], R + kRecBeta + 4 * (q - 192));
    }
}

__global__ void __launch_bounds__(kRtThreads, 1)
k_bwd_rows_tc(const float* __restrict__ X, const float* __restrict__ g, const float* __restrict__ Rec,
              const float* __restrict__ dO, float* __restrict__ E, float* __restrict__ W,
              const int32_t* __restrict__ cu, const int64_t* __restrict__ prefix, int64_t T_total, int H,
              float scale, int max_seg, const float* __restrict__ Sck, const float* __restrict__ dSck,
              const float* __restrict__ dS_fin, float* __restrict__ dX, float* __restrict__ dg,
              float* __restrict__ segtot, float* __restrict__ segown, float* __restrict__ fin, int64_t slots,
              int* __restrict__ d_status) {
    using namespace tcs;
    extern __shared__ unsigned char smem_raw[];
    RowsTcSmem& sm = *reinterpret_cast<RowsTcSmem*>(smem_raw + ((1024 - (smem_u32(smem_raw) & 1023)) & 1023));
    const int u = blockIdx.x / max_seg, sg = blockIdx.x % max_seg, n = u / H, h = u % H;
    const int tid = threadIdx.x, warp = tid >> 5, role = warp >> 2, key = 32 * (warp & 3) + (tid & 31);
    int64_t s0, s1;
    seq_range(cu, n, T_total, s0, s1);
    const int64_t nseg = (s1 - s0 + kSeg - 1) / kSeg;
    if (sg >= nseg) return;
    const int64_t sb = slot_base(prefix, n, H, h, nseg, slots);
    if (sb < 0) return;  // flagged by the forward sweep
    const int64_t HD = (int64_t)H * kD;
    const int64_t ta = s0 + (int64_t)sg * kSeg, tb = ta + kSeg < s1 ? ta + kSeg : s1;
    const int ncs = (int)((tb - ta + kCk - 1) / kCk);
    auto nt_of = [&](int cc) { return (int)(tb - (ta + cc * kCk) < kCk ? tb - (ta + cc * kCk) : kCk); };
    if (tid == 0) {
        mbar_init(&sm.barP, 1);
        mbar_init(&sm.barU, 1);
        sm.fail = 0;
        fence_mbar_init();
    }
    if (warp == 0) tmem_alloc(&sm.tbase, 512);
    // stage k < ncs: forward chunk k (record row Kbar); k >= ncs: backward chunk 2 ncs - 1 - k (Qr, Kr)
    auto stage = [&](int k) {
        const bool fw = k < ncs;
        const int cc = fw ? k : 2 * ncs - 1 - k;
        const float* R = Rec + rec_index(sb, (int64_t)sg * kChunksPerSeg + cc) * kRec;
        if (tid >= 32)
            rt_stage(sm.st[k & 1], X, g, E, dO, W, R, fw ? kRecKb : kRecQr, fw ? -1 : kRecKr,
                     ta + (int64_t)cc * kCk, nt_of(cc), H, h, tid - 32);
    };
    stage(0);
    cp_commit();
    fence_before_sync();
    __syncthreads();
    fence_after_sync();
    const uint32_t tm = sm.tbase, tl = tm + ((uint32_t)(32 * (warp & 3)) << 16);
    const int cb = 64 * role;  // this thread's half of the state's 128 value columns in the TMEM passes
    {  // the segment's start state: lane = key, columns = value columns
        const float* Sg = Sck + ((sb + sg) * kD + key) * kD + cb;
#pragma unroll 1
        for (int c0 = 0; c0 < 64; c0 += 32) {
            float v[32];
#pragma unroll
            for (int i = 0; i < 32; i += 4) {
                const float4 x = *reinterpret_cast<const float4*>(Sg + c0 + i);
                v[i] = x.x;
                v[i + 1] = x.y;
                v[i + 2] = x.z;
                v[i + 3] = x.w;
            }
            tst32(tl + cb + c0, v);
        }
        tmem_st_wait();
    }
    const float4 z4 = make_float4(0.f, 0.f, 0.f, 0.f);
    float pre_q = 0.f, pre_k = 0.f, run = 0.f;  // role 0: the segment's running sums for its key
    // the state pass: high part and remainder of the state (A operand of the reads), then the decay
    auto state_pass = [&](const RtStage& s) {
        const float cl = s.CL[key];
#pragma unroll 1
        for (int c0 = 0; c0 < 64; c0 += 32) {
            float v[32], hv[32], lv[32];
            tld32(tl + cb + c0, v);
#pragma unroll
            for (int i = 0; i < 32; ++i) {
                hv[i] = __uint_as_float(tf32_of(v[i]));
                lv[i] = v[i] - hv[i];
                v[i] *= cl;
            }
            tst32(tl + 128 + cb + c0, hv);
            tst32(tl + 256 + cb + c0, lv);
            tst32(tl + cb + c0, v);
        }
    };
    auto sync_tc = [&]() {
        tmem_st_wait();
        fence_async_smem();
        fence_before_sync();
        __syncthreads();
        fence_after_sync();
    };
    // ---------------- forward: dq, dk_read, the read part of dg
#pragma unroll 1
    for (int cc = 0; cc < ncs; ++cc) {
        const int k = cc, nt = nt_of(cc);
        const int64_t t0 = ta + (int64_t)cc * kCk;
        const RtStage& s = sm.st[k & 1];
        if (cc > 0 && !sm.fail && !warp_wait(&sm.barU, (uint32_t)((k - 1) & 1))) sm.fail = 1;  // the state is complete
        cp_wait<0>();
        fence_before_sync();
        __syncthreads();
        fence_after_sync();
        // phase 1: the state's high part and remainder (then the decay); b1 = [dO; W] (rows 0-15 dO, 16-31 W)
        state_pass(s);
        for (int i4 = tid; i4 < 32 * 32; i4 += kRtThreads) {
            const int row = i4 >> 5, c4 = (i4 & 31) * 4, t = row & 15;
            const float4 x = t < nt ? *reinterpret_cast<const float4*>(row < 16 ? &s.DO[t][c4] : &s.W[t][c4]) : z4;
            float4 lo;
            const float4 hi = hi4(x, lo);
            const uint32_t off = kmaj(32, row, c4);
            sts128(sm.b1h, off, hi);
            sts128(sm.b1l, off, lo);
        }
        sync_tc();
        if (tid == 0 && !sm.fail) {  // [S do | S w]: A = S (high, low), B = [dO; W]
            const uint32_t id32 = idesc_tf32(128, 32), h1 = smem_u32(sm.b1h), l1 = smem_u32(sm.b1l);
#pragma unroll 1
            for (int ks = 0; ks < kD / 8; ++ks) {
                mma_tf32_ts(tm + 384, tm + 256 + 8 * ks, bdesc(h1, 32, ks), id32, ks > 0);
                mma_tf32_ts(tm + 384, tm + 128 + 8 * ks, bdesc(l1, 32, ks), id32, 1);
                mma_tf32_ts(tm + 384, tm + 128 + 8 * ks, bdesc(h1, 32, ks), id32, 1);
            }
            mma_commit(&sm.barP);
        }
        // phase 2, while the reads run (warp 0 issues them): warps 4-7 the Grams and the update's A
        // operand, warps 1-3 b2 = (B E)^T; then every warp but warp 0 the next chunk's copies
        if (role == 1) {
            const int w4 = warp - 4, gq = (tid & 31) >> 2, tq = tid & 3, nt8 = 8 * (w4 >> 1);
            const float(*Bm)[kRs] = (w4 & 1) ? s.W : s.DO;  // P = E dO^T (tasks 0, 2), Q = E W^T (1, 3)
            const bool ar0 = gq < nt, ar1 = gq + 8 < nt, bn = nt8 + gq < nt;
            float acc[4] = {0.f, 0.f, 0.f, 0.f}, accc[4] = {0.f, 0.f, 0.f, 0.f};  // high products, corrections
#pragma unroll 4
            for (int kc = 0; kc < kD; kc += 8) {
                const float2 x0 = ar0 ? *reinterpret_cast<const float2*>(&s.E[gq][kc + 2 * tq]) : make_float2(0.f, 0.f);
                const float2 x1 =
                    ar1 ? *reinterpret_cast<const float2*>(&s.E[gq + 8][kc + 2 * tq]) : make_float2(0.f, 0.f);
                const float2 y = bn ? *reinterpret_cast<const float2*>(&Bm[nt8 + gq][kc + 2 * tq]) : make_float2(0.f, 0.f);
                const float av[4] = {x0.x, x0.y, x1.x, x1.y};  // accumulator order: (g, 2t), (g, 2t+1), (g+8, ..)
                const Frag4 a = afrag_acc(av);
                Frag2 b;
                split_tf32(y.x, b.h[0], b.l[0]);
                split_tf32(y.y, b.h[1], b.l[1]);
                mma3x(acc, accc, a, b);
            }
            float(*G)[kCk] = (w4 & 1) ? sm.Q[cc] : sm.P[cc];
            G[gq][nt8 + 2 * tq] = acc[0] + accc[0];
            G[gq][nt8 + 2 * tq + 1] = acc[1] + accc[1];
            G[gq + 8][nt8 + 2 * tq] = acc[2] + accc[2];
            G[gq + 8][nt8 + 2 * tq + 1] = acc[3] + accc[3];
            float hv[16], lv[16];  // A of the update: Kbar^T (lane = key, 16 tokens)
#pragma unroll
            for (int t = 0; t < kCk; ++t) {
                const float x = s.R1[t][key];
                hv[t] = __uint_as_float(tf32_of(x));
                lv[t] = x - hv[t];
            }
            tst16(tl + 416, hv);
            tst16(tl + 448, lv);
        } else if (warp > 0) {
            for (int j = tid - 32; j < kD; j += 96) {  // row = value column j, K = token
#pragma unroll
                for (int m = 0; m < kCk; m += 4) {
                    float x[4];
#pragma unroll
                    for (int e = 0; e < 4; ++e) {
                        const int t = m + e;
                        x[e] = t < nt ? s.beta[t] * s.E[t][j] : 0.f;
                    }
                    float4 lo;
                    const float4 hi = hi4(make_float4(x[0], x[1], x[2], x[3]), lo);
                    const uint32_t off = kmaj(128, j, m);
                    sts128(sm.b2h, off, hi);
                    sts128(sm.b2l, off, lo);
                }
            }
        }
        if (k + 1 < 2 * ncs) stage(k + 1);
        cp_commit();
        // the key's decay factors over the chunk
        float C[kCk], Ca[kCk], Ki[kCk];
        {
            float G[kCk], acc = 0.f;
#pragma unroll
            for (int t = 0; t < kCk; ++t) {
                acc += t < nt ? s.g[t][key] : 0.f;
                G[t] = acc;
            }
#pragma unroll
            for (int t = 0; t < kCk; ++t) {
                C[t] = expf(G[t]);
                Ca[t] = expf(G[t] - G[7]);
                Ki[t] = (t < nt ? s.k[t][key] : 0.f) * expf(G[7] - G[t]);
            }
        }
        sync_tc();
        if (tid == 0 && !sm.fail) {  // S += Kbar^T (B E)
            const uint32_t id128 = idesc_tf32(128, 128), h2 = smem_u32(sm.b2h), l2 = smem_u32(sm.b2l);
#pragma unroll
            for (int ks = 0; ks < 2; ++ks) {
                mma_tf32_ts(tm, tm + 448 + 8 * ks, bdesc(h2, 128, ks), id128, 1);
                mma_tf32_ts(tm, tm + 416 + 8 * ks, bdesc(l2, 128, ks), id128, 1);
                mma_tf32_ts(tm, tm + 416 + 8 * ks, bdesc(h2, 128, ks), id128, 1);
            }
            mma_commit(&sm.barU);
        }
        if (!sm.fail && !warp_wait(&sm.barP, (uint32_t)(k & 1))) sm.fail = 1;
        float z[kCk];
        {
            uint32_t r[16];
            tmem_ld16(tl + 384 + 16 * role, r);
            tmem_ld_wait();
#pragma unroll
            for (int t = 0; t < kCk; ++t) z[t] = __uint_as_float(r[t]);
        }
        float cq[kCk], acc[kCk];
#pragma unroll
        for (int t = 0; t < kCk; ++t) acc[t] = 0.f;
        {  // right-looking over the Gram's rows: acc_t += beta_s (k^_s / C'_s) G_st (s <= t for dq, s < t for dk_read)
            const float(*G)[kCk] = role == 0 ? sm.P[cc] : sm.Q[cc];
#pragma unroll
            for (int s2 = 0; s2 < kCk; ++s2) {
                const float bk = s.beta[s2] * Ki[s2];
#pragma unroll
                for (int q4 = 0; q4 < kCk; q4 += 4) {
                    if (q4 + 3 < s2) continue;
                    const float4 p4 = *reinterpret_cast<const float4*>(&G[s2][q4]);
                    const float pv[4] = {p4.x, p4.y, p4.z, p4.w};
#pragma unroll
                    for (int e = 0; e < 4; ++e) {
                        const int t = q4 + e;
                        if (role == 0 ? t >= s2 : t > s2) acc[t] = fmaf(pv[e], bk, acc[t]);
                    }
                }
            }
        }
        float* dxr = dX + t0 * 3 * HD + role * HD + (int64_t)h * kD + key;  // dq (role 0) / dk_read rows
        if (role == 0) {  // dq
#pragma unroll
            for (int t = 0; t < kCk; ++t, dxr += 3 * HD) {
                const float dq = scale * (C[t] * z[t] + Ca[t] * acc[t]);
                cq[t] = t < nt ? s.q[t][key] * dq : 0.f;
                if (t < nt) *dxr = dq;
            }
        } else {  // dk_read
#pragma unroll
            for (int t = 0; t < kCk; ++t, dxr += 3 * HD) {
                const float dkr = -s.beta[t] * (C[t] * z[t] + Ca[t] * acc[t]);
                sm.xch[t][key] = t < nt ? s.k[t][key] * dkr : 0.f;
                if (t < nt) *dxr = dkr;
            }
        }
        __syncthreads();
        if (role == 0) {
            float* dgr = dg + (t0 * H + h) * kD + key;
#pragma unroll
            for (int t = 0; t < kCk; ++t, dgr += HD) {
                if (t < nt) *dgr = -(pre_q + pre_k);  // minus the earlier read part
                pre_q += cq[t];
                pre_k += sm.xch[t][key];
            }
        }
    }
    if (!sm.fail && !warp_wait(&sm.barU, (uint32_t)((ncs - 1) & 1))) sm.fail = 1;  // the segment's end state
    if (tb == s1) {  // the sequence's final state: rowsum(dS_T . S_T)
        float x = 0.f;
        if (dS_fin) {
            const float* Dr = dS_fin + ((int64_t)u * kD + key) * kD + cb;
#pragma unroll 1
            for (int c0 = 0; c0 < 64; c0 += 32) {
                float v[32];
                tld32(tl + cb + c0, v);
#pragma unroll
                for (int i = 0; i < 32; ++i) x = fmaf(Dr[c0 + i], v[i], x);
            }
        }
        if (role == 1) sm.xch[0][key] = x;
        __syncthreads();
        if (role == 0) fin[(int64_t)u * kD + key] = x + sm.xch[0][key];
    }
    fence_before_sync();
    __syncthreads();  // every read of the end state is done
    fence_after_sync();
    {  // the segment's end gradient replaces the state in TMEM
        const float* Dg = dSck + ((sb + sg) * kD + key) * kD + cb;
#pragma unroll 1
        for (int c0 = 0; c0 < 64; c0 += 32) {
            float v[32];
#pragma unroll
            for (int i = 0; i < 32; i += 4) {
                const float4 x = *reinterpret_cast<const float4*>(Dg + c0 + i);
                v[i] = x.x;
                v[i + 1] = x.y;
                v[i + 2] = x.z;
                v[i + 3] = x.w;
            }
            tst32(tl + cb + c0, v);
        }
        tmem_st_wait();
    }
    // ---------------- backward: dk_write and the write part of dg, chunks last to first
#pragma unroll 1
    for (int k = ncs; k < 2 * ncs; ++k) {
        const int cc = 2 * ncs - 1 - k, nt = nt_of(cc);
        const int64_t t0 = ta + (int64_t)cc * kCk;
        const RtStage& s = sm.st[k & 1];
        if (k > ncs && !sm.fail && !warp_wait(&sm.barU, (uint32_t)((k - 1) & 1))) sm.fail = 1;
        cp_wait<0>();
        fence_before_sync();
        __syncthreads();
        fence_after_sync();
        // phase 1: the gradient's high part and remainder (then the decay); b1 = E (16 rows)
        state_pass(s);
        for (int i4 = tid; i4 < 16 * 32; i4 += kRtThreads) {
            const int t = i4 >> 5, c4 = (i4 & 31) * 4;
            const float4 x = t < nt ? *reinterpret_cast<const float4*>(&s.E[t][c4]) : z4;
            float4 lo;
            const float4 hi = hi4(x, lo);
            const uint32_t off = kmaj(16, t, c4);
            sts128(sm.b1h, off, hi);
            sts128(sm.b1l, off, lo);
        }
        sync_tc();
        if (tid == 0 && !sm.fail) {  // D E^T: A = D (high, low), B = E
            const uint32_t id16 = idesc_tf32(128, 16), h1 = smem_u32(sm.b1h), l1 = smem_u32(sm.b1l);
#pragma unroll 1
            for (int ks = 0; ks < kD / 8; ++ks) {
                mma_tf32_ts(tm + 384, tm + 256 + 8 * ks, bdesc(h1, 16, ks), id16, ks > 0);
                mma_tf32_ts(tm + 384, tm + 128 + 8 * ks, bdesc(l1, 16, ks), id16, 1);
                mma_tf32_ts(tm + 384, tm + 128 + 8 * ks, bdesc(h1, 16, ks), id16, 1);
            }
            mma_commit(&sm.barP);
        }
        // phase 2, while D E^T runs: warps 4-7 the update's A operand [Qr | Kr]^T (lane = key,
        // 32 tokens), warps 1-3 b2 = [scale dO; -B W]^T (row = value column, K = 32); the next copies
        if (role == 1) {
#pragma unroll
            for (int half = 0; half < 2; ++half) {
                float hv[16], lv[16];
#pragma unroll
                for (int t = 0; t < kCk; ++t) {
                    const float x = half == 0 ? s.R1[t][key] : s.R2[t][key];
                    hv[t] = __uint_as_float(tf32_of(x));
                    lv[t] = x - hv[t];
                }
                tst16(tl + 416 + 16 * half, hv);
                tst16(tl + 448 + 16 * half, lv);
            }
        } else if (warp > 0) {
            for (int j = tid - 32; j < kD; j += 96) {
#pragma unroll
                for (int m = 0; m < 2 * kCk; m += 4) {
                    float x[4];
#pragma unroll
                    for (int e = 0; e < 4; ++e) {
                        const int kk = m + e, t = kk & 15;
                        x[e] = t >= nt ? 0.f : kk < kCk ? scale * s.DO[t][j] : -s.beta[t] * s.W[t][j];
                    }
                    float4 lo;
                    const float4 hi = hi4(make_float4(x[0], x[1], x[2], x[3]), lo);
                    const uint32_t off = kmaj(128, j, m);
                    sts128(sm.b2h, off, hi);
                    sts128(sm.b2l, off, lo);
                }
            }
        }
        if (k + 1 < 2 * ncs) stage(k + 1);
        cp_commit();
        float CLr[kCk], iCa[kCk], Xa[kCk];  // C_last / C_t, 1 / C'_t, C'_t x_t (x = q for role 0, k for role 1)
        {
            float G[kCk], acc = 0.f;
#pragma unroll
            for (int t = 0; t < kCk; ++t) {
                acc += t < nt ? s.g[t][key] : 0.f;
                G[t] = acc;
            }
#pragma unroll
            for (int t = 0; t < kCk; ++t) {
                CLr[t] = expf(G[kCk - 1] - G[t]);
                iCa[t] = expf(G[7] - G[t]);
                const float xv = t < nt ? (role == 0 ? s.q[t][key] : s.k[t][key]) : 0.f;
                Xa[t] = xv * expf(G[t] - G[7]);
            }
        }
        sync_tc();
        if (tid == 0 && !sm.fail) {  // D += [Qr | Kr]^T [scale dO; -B W]
            const uint32_t id128 = idesc_tf32(128, 128), h2 = smem_u32(sm.b2h), l2 = smem_u32(sm.b2l);
#pragma unroll
            for (int ks = 0; ks < 4; ++ks) {
                mma_tf32_ts(tm, tm + 448 + 8 * ks, bdesc(h2, 128, ks), id128, 1);
                mma_tf32_ts(tm, tm + 416 + 8 * ks, bdesc(l2, 128, ks), id128, 1);
                mma_tf32_ts(tm, tm + 416 + 8 * ks, bdesc(h2, 128, ks), id128, 1);
            }
            mma_commit(&sm.barU);
        }
        if (!sm.fail && !warp_wait(&sm.barP, (uint32_t)(k & 1))) sm.fail = 1;
        float x0[kCk];
        if (role == 0) {  // (C_last / C_t) (D e_t) + (1 / C'_t) scale sum_{tau >= t} P_t,tau C'_tau q^_tau
            uint32_t r[16];
            tmem_ld16(tl + 384, r);
            tmem_ld_wait();
#pragma unroll
            for (int t = 0; t < kCk; ++t) {
                float acc = 0.f;
#pragma unroll
                for (int q4 = 0; q4 < kCk; q4 += 4) {
                    if (q4 + 3 < t) continue;
                    const float4 p4 = *reinterpret_cast<const float4*>(&sm.P[cc][t][q4]);
                    const float pv[4] = {p4.x, p4.y, p4.z, p4.w};
#pragma unroll
                    for (int e = 0; e < 4; ++e)
                        if (q4 + e >= t) acc = fmaf(pv[e], Xa[q4 + e], acc);
                }
                x0[t] = CLr[t] * __uint_as_float(r[t]) + iCa[t] * scale * acc;
            }
        } else {  // -(1 / C'_t) sum_{tau > t} beta_tau Q_t,tau C'_tau k^_tau
#pragma unroll
            for (int t = 0; t < kCk; ++t) Xa[t] *= s.beta[t];
#pragma unroll
            for (int t = 0; t < kCk; ++t) {
                float acc = 0.f;
#pragma unroll
                for (int q4 = 0; q4 < kCk; q4 += 4) {
                    if (q4 + 3 <= t) continue;
                    const float4 p4 = *reinterpret_cast<const float4*>(&sm.Q[cc][t][q4]);
                    const float pv[4] = {p4.x, p4.y, p4.z, p4.w};
#pragma unroll
                    for (int e = 0; e < 4; ++e)
                        if (q4 + e > t) acc = fmaf(pv[e], Xa[q4 + e], acc);
                }
                sm.xch[t][key] = -iCa[t] * acc;
            }
        }
        __syncthreads();
        if (role == 0) {  // dk_write; its global E row and the suffix sum of -k dk_write in the W row
            const int64_t off0 = (t0 * H + h) * kD + key;
#pragma unroll
            for (int t = kCk - 1; t >= 0; --t) {
                if (t >= nt) continue;
                const float dkw = s.beta[t] * (x0[t] + sm.xch[t][key]);
                run -= s.k[t][key] * dkw;
                E[off0 + t * HD] = dkw;
                W[off0 + t * HD] = run;
            }
        }
    }
    if (!sm.fail && !warp_wait(&sm.barU, (uint32_t)((2 * ncs - 1) & 1))) sm.fail = 1;
    if (role == 0) {
        segtot[(sb + sg) * kD + key] = pre_q + pre_k + run;  // the segment's sum of dGamma
        segown[(sb + sg) * kD + key] = pre_q + pre_k;        // its read part
    }
    fence_before_sync();
    __syncthreads();
    if (sm.fail) {
        if (tid == 0) flag_status(d_status, KDA_ERR_TIMEOUT);
        __syncthreads();
    }
    fence_after_sync();
    if (warp == 0) {
        tmem_dealloc(tm, 512);
        tmem_relinquish();
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
constexpr int kEpiRows = 4;  // rows per warp
// Each warp takes kEpiRows consecutive (token, head) rows, all their loads issued first: do (written
// over o), dgate, and the RMSNorm weight's gradient (block partials in shared memory, one atomic per
// channel and block).
template <typename Tg, typename Tdy>
__global__ void k_bwd_epilogue(float* __restrict__ O, const Tdy* __restrict__ dy, const Tg* __restrict__ gate,
                               const float* __restrict__ rms_w, float eps_rms, int64_t rows,
                               float* __restrict__ dgate, float* __restrict__ drms) {
    __shared__ float sdw[kD];
    for (int c = threadIdx.x; c < kD; c += blockDim.x) sdw[c] = 0.f;
    __syncthreads();
    const int lane = threadIdx.x & 31, c0 = 4 * lane;
    // two consecutive rows per warp, every load of both issued before any arithmetic: o, dy, the
    // gate pre-activations, the RMSNorm weight
    const int64_t r0 = kEpiRows * ((int64_t)blockIdx.x * (blockDim.x / 32) + (threadIdx.x >> 5));
    float4 o[kEpiRows];
    float dyv[kEpiRows][4], gv[kEpiRows][4];
#pragma unroll
    for (int i = 0; i < kEpiRows; ++i) {
        const int64_t row = r0 + i;
        o[i] = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
        for (int m = 0; m < 4; ++m) dyv[i][m] = gv[i][m] = 0.f;
        if (row < rows) {
            o[i] = *reinterpret_cast<const float4*>(O + row * kD + c0);
            load4(dy + row * kD + c0, dyv[i]);
            if (gate) load4(gate + row * kD + c0, gv[i]);
        }
    }
    float4 wv = make_float4(1.f, 1.f, 1.f, 1.f);
    if (rms_w) wv = make_float4(rms_w[c0], rms_w[c0 + 1], rms_w[c0 + 2], rms_w[c0 + 3]);  // 4-byte aligned
    const float wm[4] = {wv.x, wv.y, wv.z, wv.w};
    float dw[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
    for (int i = 0; i < kEpiRows; ++i) {
        const int64_t row = r0 + i;
        if (row >= rows) break;  // warp-uniform
        const float r = 1.0f / sqrtf(warp_sum(dot4(o[i], o[i])) * (1.0f / kD) + eps_rms);
        float dn[4], dgv[4];
        const float ov[4] = {o[i].x, o[i].y, o[i].z, o[i].w};
        float dno = 0.f;
#pragma unroll
        for (int m = 0; m < 4; ++m) {
            const float sg = gate ? 1.0f / (1.0f + expf(-gv[i][m])) : 1.f;
            const float d = dyv[i][m];
            const float nv = ov[m] * r;
            dgv[m] = gate ? d * nv * wm[m] * sg * (1.f - sg) : 0.f;
            dw[m] += d * nv * sg;
            dn[m] = d * wm[m] * sg;
            dno += dn[m] * ov[m];
        }
        if (dgate) *reinterpret_cast<float4*>(dgate + row * kD + c0) = make_float4(dgv[0], dgv[1], dgv[2], dgv[3]);
        dno = warp_sum(dno);
        const float r3 = r * r * r * dno * (1.0f / kD);
        *reinterpret_cast<float4*>(O + row * kD + c0) =
            make_float4(r * dn[0] - r3 * ov[0], r * dn[1] - r3 * ov[1], r * dn[2] - r3 * ov[2], r * dn[3] - r3 * ov[3]);
    }
    if (drms)
#pragma unroll
        for (int m = 0; m < 4; ++m) atomicAdd(&sdw[c0 + m], dw[m]);
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
constexpr int kConvBatch = 8;  // tokens whose loads are issued together

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
        const float sg = __fdividef(1.0f, 1.0f + __expf(-uu));  // (uu -> -inf: 1 / inf = 0)
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
        if (t - (kConvBatch + 2) >= s0 && t - (kConvBatch - 1) >= ta) {
            // kConvBatch tokens inside the sequence: all their loads first
            float rr[kConvBatch], dd[kConvBatch];
#pragma unroll
            for (int i = 0; i < kConvBatch; ++i) {
                rr[i] = to_f(src[(t - 3 - i) * xs + hc]);
                dd[i] = dA[(t - i) * HD3 + ch];
            }
#pragma unroll
            for (int i = 0; i < kConvBatch; ++i) step(t - i, rr[i], dd[i]);
            t -= kConvBatch;
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
    }
    k_bwd_seg_prefix<<<1, 256, 0, s>>>(a.cu_seqlens, a.N, T, prefix);
    if ((e = cudaGetLastError())) return e;
    const unsigned rb = (unsigned)((rows + 7) / 8);
    if (rows > 0) {  // (rows start on 16-byte boundaries: the row rules of the C ABI)
        if ((e = cudaFuncSetAttribute(k_bwd_prep_tile<Tio>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                      (int)prep_tile_smem<Tio>())))
            return e;
        k_bwd_prep_tile<Tio><<<(unsigned)((T + kPrepTile - 1) / kPrepTile * a.H), 256, prep_tile_smem<Tio>(), s>>>(
            cptr<Tio>(a.q), cptr<Tio>(a.k), cptr<Tio>(a.v), xs, a.conv_w, cptr<Tio>(a.conv_state_in), a.cu_seqlens,
            a.N, T, a.H, a.eps_l2, X, nrm);
        if ((e = cudaGetLastError())) return e;
    }
    float* Rec = reinterpret_cast<float*>(ws + L.rec);
    if (rows > 0 && L.max_ch > 0) {
        k_bwd_chunk_prep<<<(unsigned)(units * L.max_ch), 128, 0, s>>>(X, a.g, a.beta, a.cu_seqlens, prefix, T, a.H,
                                                                       (int)L.max_ch, Rec, L.slots);
        if ((e = cudaGetLastError())) return e;
    }
    if ((e = cudaFuncSetAttribute(k_bwd_fwd_chunks, cudaFuncAttributeMaxDynamicSharedMemorySize, kFwdSmem)) ||
        (e = cudaFuncSetAttribute(k_bwd_bwd_chunks, cudaFuncAttributeMaxDynamicSharedMemorySize, kBwdSmem)))
        return e;
    k_bwd_fwd_chunks<<<(unsigned)(units * kChCtas), 128, kFwdSmem, s>>>(X, Rec, a.cu_seqlens, prefix, T, a.H, a.scale,
                                                                        a.initial_state, O, E, Sck, L.slots,
                                                                        a.d_status);
    if ((e = cudaGetLastError())) return e;
    if (rows > 0) {
        if (a.out_dtype == KDA_FP32)
            k_bwd_epilogue<Tio, float><<<(unsigned)((rows + 8 * kEpiRows - 1) / (8 * kEpiRows)), 256, 0, s>>>(O, cptr<float>(b.dy), cptr<Tio>(a.gate), a.rms_w, a.eps_rms,
                                                           rows, b.dgate, b.drms_w);
        else
            k_bwd_epilogue<Tio, bf16><<<(unsigned)((rows + 8 * kEpiRows - 1) / (8 * kEpiRows)), 256, 0, s>>>(O, cptr<bf16>(b.dy), cptr<Tio>(a.gate), a.rms_w, a.eps_rms,
                                                          rows, b.dgate, b.drms_w);
        if ((e = cudaGetLastError())) return e;
    }
    k_bwd_bwd_chunks<<<(unsigned)(units * kChCtas), 128, kBwdSmem, s>>>(Rec, O, E, a.cu_seqlens, prefix, T, a.H,
                                                                        a.scale, b.d_final_state, W, dX, b.dbeta,
                                                                        dSck, b.dinitial_state, L.slots);
    if ((e = cudaGetLastError())) return e;
    if (rows == 0) return cudaSuccess;
    if ((e = cudaFuncSetAttribute(k_bwd_rows_tc, cudaFuncAttributeMaxDynamicSharedMemorySize, kRowsTcSmem))) return e;
    k_bwd_rows_tc<<<(unsigned)(units * L.max_seg), kRtThreads, kRowsTcSmem, s>>>(
        X, a.g, Rec, O, E, W, a.cu_seqlens, prefix, T, a.H, a.scale, (int)L.max_seg, Sck, dSck, b.d_final_state, dX,
        b.dg, segtot, segown, fin, L.slots, a.d_status);
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
    size_t segs = 0, max_seg = 0, max_ch = 0;
    if (a.cu_seqlens_host)
        for (int n = 0; n < a.N; ++n) {
            const size_t ns = (size_t)(a.cu_seqlens_host[n + 1] - a.cu_seqlens_host[n] + kSeg - 1) / kSeg;
            segs += ns;
            max_seg = ns > max_seg ? ns : max_seg;
            const size_t nc = (size_t)(a.cu_seqlens_host[n + 1] - a.cu_seqlens_host[n] + kBwdChunk - 1) / kBwdChunk;
            max_ch = nc > max_ch ? nc : max_ch;
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
    L.slots = (int64_t)(segs * H);
    L.max_seg = (int64_t)max_seg;
    L.max_ch = (int64_t)max_ch;
    L.sck = take(segs * H * kD * kD * 4);
    L.dsck = take(segs * H * kD * kD * 4);
    L.segtot = take(segs * H * kD * 4);
    L.segown = take(segs * H * kD * 4);
    L.rec = take(segs * H * kBwdSeg / kBwdChunk * kBwdRecFloats * 4);
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
