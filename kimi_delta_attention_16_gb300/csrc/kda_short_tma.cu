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
// bound by HBM.  Persistent CTAs (one per SM) walk contiguous head-major
// ranges of units with two shared-memory stages.  A producer warp (one
// thread) fills stage i % 2 with unit i -- the state as four 2D tensor-map
// boxes of 32 columns with the 128-byte swizzle, the conv window by 1D bulk
// copies, the token rows as one box of Lmax rows for each of q, k, v, gate
// and g, the betas by plain loads -- and, once the compute warps have
// finished unit i - 2 there and written its state back into the stage, sends
// that state to final_state by four tensor-map stores before reusing the
// stage.  Neither the request issue nor the 64 KB store stalls a compute warp.
//
// Sixteen compute warps; warp w owns value columns 8 w .. 8 w + 7 and lane l
// owns the rows l, l + 32, l + 64, l + 96 of all eight, as packed fp32 pairs of
// adjacent columns.  A token's per-row factors (q, k, e^g) are then read by
// the 32 lanes of a warp from 32 consecutive floats (one shared-memory
// wavefront per 32 values, instead of the eight-lane broadcasts a
// column-per-lane layout needs), and the column sums over the key rows (the
// probe S_bar^T k and the readout S^T q) are one transposed reduction of the
// eight columns over the warp; no barrier is needed between tokens.  The
// state's shared-memory accesses (row r, column c at 16-byte chunk
// ((c mod 32) / 4) xor (r mod 8) of the swizzle) are conflict-free: the eight
// lanes of a quarter-warp read eight consecutive rows.  A unit's outputs are
// normalised (RMSNorm, weight, gate) during the next unit's conv, by the four
// warps that have no conv channel.
#include "kda_internal.cuh"
#include "kda_tc.cuh"
#include "kda_tc_ptx.cuh"

namespace kda {

namespace {

constexpr int kD = 128;
constexpr int kCompute = 512;             // sixteen compute warps
constexpr int kThreads = kCompute + 32;   // + the producer warp
constexpr int kL8 = kShortMaxL;
constexpr int kFs = kD;  // per-token stride (floats) of the factor arrays
// static shared memory of the kernel (sv, sgate[2], sW, sRms, snorm, sbeta, barriers)
constexpr uint32_t kStaticSmem = 4u * (3 * kL8 * kD + 3 * kD * 4 + kD + kL8 * 2 + 2 * kL8) + 32u;
// the warps that have no conv channel (3 * 128 channels over the first twelve warps); they
// normalise the previous unit's outputs while the others convolve
constexpr int kEmitWarp0 = 3 * kD / 32;
constexpr int kEmitWarps = kCompute / 32 - kEmitWarp0;

__host__ __device__ constexpr uint32_t align128(uint32_t x) { return (x + 127u) & ~127u; }

// Byte offsets inside one stage for boxes of Lmax token rows.  The state boxes use the
// 128-byte swizzle, so every stage starts on a 1024-byte boundary.
template <typename Tio>
struct TmaStage {
    uint32_t conv, rows, part, g, bytes;
    __host__ __device__ explicit TmaStage(int Lmax) {
        conv = 65536;                                                     // [3][128][3] Tio
        rows = conv + align128(3 * kD * 3 * (uint32_t)sizeof(Tio));      // [4][Lmax][128] Tio: q, k, v, gate
        part = (uint32_t)Lmax * kD * (uint32_t)sizeof(Tio);
        g = rows + align128(4 * part);                                    // [Lmax][128] fp32
        bytes = (g + (uint32_t)Lmax * kD * 4 + 1023u) & ~1023u;
    }
};

// Shared-memory byte offset of state element (row r, column c) in a stage: four boxes of
// 32 columns x 128 rows, 128-byte rows, 16-byte chunk j of row r at chunk j ^ (r % 8).
__device__ __forceinline__ uint32_t state_off(int r, int c) {
    return (uint32_t)((c >> 5) * 16384 + r * 128 + ((((c & 31) >> 2) ^ (r & 7)) << 4) + (c & 3) * 4);
}

// Tensor maps of the token rows: [T rows][H * 128 columns], boxes of 128 columns x Lmax rows.
struct ShortMaps {
    CUtensorMap q, k, v, gate, g;
    CUtensorMap s_in, s_out;  // states as [units * 128 rows][128 columns] fp32, boxes of 32 x 128
};

__device__ __forceinline__ void tma_load_2d(uint32_t dst, const CUtensorMap* map, int x, int y, uint64_t* bar) {
    asm volatile(
        "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes [%0], [%1, {%2, %3}], [%4];" ::
            "r"(dst), "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y), "r"(tc::smem_u32(bar))
        : "memory");
}
// shared -> global through a tensor map, tracked by the bulk groups of the issuing thread
__device__ __forceinline__ void tma_store_2d(const CUtensorMap* map, int x, int y, uint32_t src) {
    asm volatile("cp.async.bulk.tensor.2d.global.shared::cta.bulk_group [%0, {%1, %2}], [%3];" ::"l"(
                     reinterpret_cast<uint64_t>(map)),
                 "r"(x), "r"(y), "r"(src)
                 : "memory");
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

// named barrier 1 of the compute warps (the producer warp never joins it)
__device__ __forceinline__ void cbar() { asm volatile("bar.sync 1, %0;" ::"n"(kCompute) : "memory"); }
__device__ __forceinline__ bool cbar_or(bool v) {
    uint32_t r;
    asm volatile(
        "{\n\t.reg .pred p, q;\n\tsetp.ne.u32 p, %1, 0;\n\tbar.red.or.pred q, 1, %2, p;\n\tselp.u32 %0, 1, 0, q;\n\t}"
        : "=r"(r)
        : "r"(v ? 1u : 0u), "n"(kCompute)
        : "memory");
    return r != 0;
}
__device__ __forceinline__ void mbar_arrive(uint64_t* bar) {
    asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(tc::smem_u32(bar)) : "memory");
}
// Sums 8 per-lane values over the 32 lanes of a warp; afterwards lane l holds the total of value
// (l >> 2) & 7 (lanes 4 c .. 4 c + 3 hold value c).
__device__ __forceinline__ float reduce8_32(float (&v)[8], int lane) {
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        const bool up = (lane & 16) != 0;
        const float send = up ? v[i] : v[i + 4];
        v[i] = (up ? v[i + 4] : v[i]) + __shfl_xor_sync(0xffffffffu, send, 16);
    }
#pragma unroll
    for (int i = 0; i < 2; ++i) {
        const bool up = (lane & 8) != 0;
        const float send = up ? v[i] : v[i + 2];
        v[i] = (up ? v[i + 2] : v[i]) + __shfl_xor_sync(0xffffffffu, send, 8);
    }
    {
        const bool up = (lane & 4) != 0;
        const float send = up ? v[0] : v[1];
        v[0] = (up ? v[1] : v[0]) + __shfl_xor_sync(0xffffffffu, send, 4);
    }
    v[0] += __shfl_xor_sync(0xffffffffu, v[0], 2);
    return v[0] + __shfl_xor_sync(0xffffffffu, v[0], 1);
}

// Sums 16 per-lane values over the 32 lanes of a warp; afterwards lane l holds the total of value
// l >> 1.
__device__ __forceinline__ float reduce16_32(float (&v)[16], int lane) {
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

template <typename Tio, typename To>
__global__ void __launch_bounds__(kThreads, 1)
k_short_tma(const __grid_constant__ ShortMaps maps, int Lmax, int has_gate, int has_s0, int has_sfin,
            const Tio* __restrict__ cs_in, Tio* __restrict__ cs_out, const float* __restrict__ beta,
            const float* __restrict__ conv_w, const float* __restrict__ rms_w, float eps_l2, float eps_rms,
            float scale, int N, int H, const int32_t* __restrict__ cu, int64_t T_total, To* __restrict__ out,
            int* d_status) {
    extern __shared__ uint8_t smem_raw[];
    __shared__ uint64_t full[2], done[2];            // stage landed; compute warps done with it
    __shared__ __align__(16) float sv[kL8][kD];       // convolved v of every token
    __shared__ __align__(16) float sgate[2][kL8][kD]; // sigmoid(gate) of every token (1 without a gate), per unit parity
    __shared__ __align__(16) float sW[3 * kD * 4];    // conv taps of the current head
    __shared__ __align__(16) float sRms[kD];
    __shared__ float snorm[kL8][2];                   // 1/|q|, 1/|k| per token
    __shared__ float sbeta[2][kL8];                   // betas per stage

    const TmaStage<Tio> ST(Lmax);
    const uint32_t raw_addr = tc::smem_u32(smem_raw);
    uint8_t* sm = smem_raw + (((raw_addr + 1023u) & ~1023u) - raw_addr);
    const uint32_t sbase = tc::smem_u32(sm);
    // after the two stages: q, k and e^g ([Lmax][128]) of every token, then o before its
    // normalisation ([Lmax][128])
    float* fq = reinterpret_cast<float*>(sm + 2 * ST.bytes);
    float* fk = fq + Lmax * kFs;
    float* fa = fk + Lmax * kFs;
    float* so = fa + Lmax * kFs;
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
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

    if (tid == 0) {
        for (int b = 0; b < 2; ++b) {
            tc::mbar_init(&full[b], 1);
            tc::mbar_init(&done[b], kCompute);
        }
        tc::fence_mbar_init();
    }
    for (int c = tid; c < kD; c += kThreads) sRms[c] = rms_w ? rms_w[c] : 1.f;
    __syncthreads();

    if (warp == kCompute / 32) {
        // ------------------------------------------------------------ producer (one thread)
        if (lane != 0) return;
        const CUtensorMap* mp[7] = {&maps.q, &maps.k, &maps.v, &maps.g, &maps.gate, &maps.s_in, &maps.s_out};
        for (int m = 0; m < 7; ++m)
            if ((m != 4 || has_gate) && (m != 5 || has_s0) && (m != 6 || has_sfin))
                asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(mp[m])) : "memory");
        const uint32_t tx = (has_s0 ? 65536u : 0u) + (cs_in ? cs_bytes : 0u) + (has_gate ? 4u : 3u) * ST.part +
                            (uint32_t)Lmax * kD * 4u;
        uint32_t pend = 0;  // bit b: a fill of stage b in flight, its phase parity in bit 2 + b
        bool failed = false;
        // unit j is done with stage j % 2 and its state is back there: send it to final_state
        auto drain = [&](int j) -> bool {
            const int b = j & 1;
            if (!tc::mbar_wait(&done[b], (uint32_t)((j >> 1) & 1))) return false;
            if (has_sfin) {
                int n, h;
                unit_of(j, n, h);
                const int y = (n * H + h) * kD;
                for (int bx = 0; bx < 4; ++bx) tma_store_2d(&maps.s_out, 32 * bx, y, sbase + (uint32_t)b * ST.bytes + 16384u * bx);
                tc::bulk_commit();
                tc::bulk_wait_read<0>();  // the stage may be refilled once the stores have read it
            }
            return true;
        };
        for (int i = 0; i < my_units; ++i) {
            const int b = i & 1;
            if (i >= 2 && !drain(i - 2)) {
                failed = true;
                break;
            }
            int n, h;
            unit_of(i, n, h);
            int64_t a, e;
            seq_range(cu, n, T_total, a, e);
#pragma unroll
            for (int t = 0; t < kL8; ++t) sbeta[b][t] = t < e - a ? beta[(a + t) * H + h] : 0.f;
            const uint32_t st = sbase + (uint32_t)b * ST.bytes;
            tc::mbar_expect_tx(&full[b], tx);  // (its arrival also releases the betas above)
            if (has_s0)
                for (int bx = 0; bx < 4; ++bx) tma_load_2d(st + 16384u * bx, &maps.s_in, 32 * bx, (n * H + h) * kD, &full[b]);
            if (cs_in)
                for (int p = 0; p < 3; ++p)
                    tc::bulk_load(st + ST.conv + (uint32_t)p * (cs_bytes / 3u),
                                  cs_in + (((int64_t)n * 3 + p) * HD + (int64_t)h * kD) * 3, cs_bytes / 3u, &full[b]);
            const int x = h * kD, y = (int)a;
            tma_load_2d(st + ST.rows, &maps.q, x, y, &full[b]);
            tma_load_2d(st + ST.rows + ST.part, &maps.k, x, y, &full[b]);
            tma_load_2d(st + ST.rows + 2 * ST.part, &maps.v, x, y, &full[b]);
            if (has_gate) tma_load_2d(st + ST.rows + 3 * ST.part, &maps.gate, x, y, &full[b]);
            tma_load_2d(st + ST.g, &maps.g, x, y, &full[b]);
            pend = (pend & ~(5u << b)) | ((1u | ((uint32_t)((i >> 1) & 1) << 2)) << b);
        }
        if (!failed)
            for (int j = my_units > 2 ? my_units - 2 : 0; j < my_units; ++j)
                if (!drain(j)) {
                    failed = true;
                    break;
                }
        if (failed) {  // fills in flight: wait for them (bounded) before the shared memory goes away
            for (int b = 0; b < 2; ++b)
                if ((pend >> b) & 1u) tc::mbar_wait(&full[b], (pend >> (2 + b)) & 1u);
            flag_status(d_status, KDA_ERR_TIMEOUT);
        }
        tc::bulk_wait_all();
        return;
    }

    // ---------------------------------------------------------------- compute warps
    const int c0w = 8 * warp;  // the warp's first value column
    // output of a unit's tokens (warp w0 + t for token t, then every nw-th): o = scale S^T q / |q|
    // from the readout sums, RMSNorm, weight, gate
    auto emit_unit = [&](int64_t ja, int jh, int jL, int jb, int w0, int nw) {
        const int c0 = 4 * lane;
        for (int t = warp - w0; t < jL; t += nw) {
            const float sq = scale * snorm[t][0];
            float4 o = *reinterpret_cast<const float4*>(so + t * kD + c0);
            o.x *= sq;
            o.y *= sq;
            o.z *= sq;
            o.w *= sq;
            float ss = o.x * o.x + o.y * o.y + o.z * o.z + o.w * o.w;
#pragma unroll
            for (int off = 16; off > 0; off >>= 1) ss += __shfl_xor_sync(0xffffffffu, ss, off);
            const float inv = 1.0f / sqrtf(ss * (1.0f / kD) + eps_rms);
            const float4 rw = *reinterpret_cast<const float4*>(&sRms[c0]);
            const float4 gg = *reinterpret_cast<const float4*>(&sgate[jb][t][c0]);
            store4<To>(out + ((ja + t) * H + jh) * kD + c0, o.x * inv * rw.x * gg.x, o.y * inv * rw.y * gg.y,
                       o.z * inv * rw.z * gg.z, o.w * inv * rw.w * gg.w);
        }
    };
    int h_prev = -1;
    int64_t a_prev = 0;  // the previous unit (its outputs are emitted during this unit's conv)
    int L_prev = 0;
    bool failed = false;
    for (int i = 0; i < my_units; ++i) {
        const int b = i & 1;
        int n, h;
        unit_of(i, n, h);
        int64_t a, e;
        seq_range(cu, n, T_total, a, e);
        int L = (int)(e - a);
        if (L > Lmax) {  // the device cu_seqlens disagrees with the host copy that sized the boxes
            if (tid == 0) flag_status(d_status, KDA_ERR_DEVICE_ARG);
            L = Lmax;
        }
        // ---- A: this unit's stage has landed; conv taps of a new head
        bool ok = true;
        if (warp == 0) ok = tc::mbar_wait(&full[b], (uint32_t)((i >> 1) & 1));
        if (h != h_prev)
            for (int idx = tid; idx < 3 * kD * 4; idx += kCompute) {
                const int part = idx / (kD * 4), rem = idx % (kD * 4);
                sW[idx] = conv_w[(part * HD + (int64_t)h * kD) * 4 + rem];
            }
        const int hp = h_prev;
        h_prev = h;
        if (cbar_or(!ok)) {
            if (tid == 0) flag_status(d_status, KDA_ERR_TIMEOUT);
            failed = true;
            break;
        }
        uint8_t* st = sm + (uint32_t)b * ST.bytes;
        // conv + SiLU of every token, one channel per thread (warps 0-11); the rolled window out
        for (int ch = tid; ch < 3 * kD; ch += kCompute) {
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
            float* dst = part == 0 ? fq + d : part == 1 ? fk + d : &sv[0][d];
            const int dstride = part == 2 ? kD : kFs;
            float xr[kL8];  // every token's raw value first: one shared-memory round trip
#pragma unroll
            for (int t = 0; t < kL8; ++t) xr[t] = t < L ? to_f(rp[t * kD]) : 0.f;
#pragma unroll
            for (int t = 0; t < kL8; ++t)
                if (t < L) {
                    dst[t * dstride] = act_silu<Tio>(w.x * p0 + w.y * p1 + w.z * p2 + w.w * xr[t]);
                    p0 = p1;
                    p1 = p2;
                    p2 = xr[t];
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
            for (int idx = tid; idx < L * kD; idx += kCompute) {
                const int t = idx >> 7, c = idx & (kD - 1);
                fa[t * kFs + c] = decay_exp<Tio>(gs[idx]);
                sgate[b][t][c] = has_gate ? act_sigmoid<Tio>(to_f(gt[idx])) : 1.f;
            }
        }
        // the previous unit's outputs (its o, norms and gates are complete: every warp has passed
        // barrier A since; this unit writes o and the norms only after barrier B, and its gates
        // to the other parity)
        if (i > 0 && warp >= kEmitWarp0) emit_unit(a_prev, hp, L_prev, b ^ 1, kEmitWarp0, kEmitWarps);
        a_prev = a;
        L_prev = L;
        // the state into registers (after the conv, whose row loads it would otherwise queue
        // behind): s2[m][p] = columns c0w + 2 p, c0w + 2 p + 1 of row lane + 32 m
        f2 s2[4][4];
#pragma unroll
        for (int m = 0; m < 4; ++m) {
            const int r = lane + 32 * m;
#pragma unroll
            for (int hf = 0; hf < 2; ++hf) {
                float4 x = make_float4(0.f, 0.f, 0.f, 0.f);
                if (has_s0) x = *reinterpret_cast<const float4*>(st + state_off(r, c0w + 4 * hf));
                s2[m][2 * hf] = f2_of(x.x, x.y);
                s2[m][2 * hf + 1] = f2_of(x.z, x.w);
            }
        }
        cbar();  // B: the stage is read completely (the state stays there for the write-back)
        // L2 norms of q and k, one vector per warp
        if (warp < 2 * L) {
            const int t = warp >> 1;
            const float* src = (warp & 1 ? fk : fq) + t * kFs;  // lane: channels 4 lane .. 4 lane + 3
            const float4 x4 = *reinterpret_cast<const float4*>(src + 4 * lane);
            float ss = x4.x * x4.x + x4.y * x4.y + x4.z * x4.z + x4.w * x4.w;
#pragma unroll
            for (int off = 16; off > 0; off >>= 1) ss += __shfl_xor_sync(0xffffffffu, ss, off);
            if (lane == 0) snorm[t][warp & 1] = 1.0f / sqrtf(ss + eps_l2);
        }
        cbar();  // C

        // ---- tokens: no barrier between them.  The eight columns' sums over the warp go through one
        // transposed reduction per token, which carries token t's probe together with token
        // t - 1's readout (so the readout never adds a reduction of its own to the chain).
        f2 O[4] = {f2_dup(0.f), f2_dup(0.f), f2_dup(0.f), f2_dup(0.f)};  // readout of the previous token
        for (int t = 0; t < L; ++t) {
            const float* kt = fk + t * kFs + lane;
            const float* at = fa + t * kFs + lane;
            const float* qt = fq + t * kFs + lane;
            const float ik = snorm[t][1];
            f2 k2[4], P[4] = {f2_dup(0.f), f2_dup(0.f), f2_dup(0.f), f2_dup(0.f)};
#pragma unroll
            for (int m = 0; m < 4; ++m) {  // decay and probe
                k2[m] = f2_dup(kt[32 * m]);
                const f2 a2 = f2_dup(at[32 * m]);
#pragma unroll
                for (int p = 0; p < 4; ++p) {
                    s2[m][p] = mul2(a2, s2[m][p]);
                    P[p] = fma2(k2[m], s2[m][p], P[p]);
                }
            }
            float v16[16] = {f2_lo(P[0]), f2_hi(P[0]), f2_lo(P[1]), f2_hi(P[1]),
                             f2_lo(P[2]), f2_hi(P[2]), f2_lo(P[3]), f2_hi(P[3]),
                             f2_lo(O[0]), f2_hi(O[0]), f2_lo(O[1]), f2_hi(O[1]),
                             f2_lo(O[2]), f2_hi(O[2]), f2_lo(O[3]), f2_hi(O[3])};
            const float red = reduce16_32(v16, lane);  // lane l: value l >> 1
            if (t > 0 && lane >= 16 && (lane & 1) == 0) so[(t - 1) * kD + c0w + ((lane >> 1) - 8)] = red;
            // lanes 2c, 2c + 1 hold column c's probe: each lane forms the correction of the column
            // it holds (lanes 16-31 form unused values), then the eight are passed round
            const float el = sbeta[b][t] * ik * (sv[t][c0w + ((lane >> 1) & 7)] - ik * red);
            float e[8];
#pragma unroll
            for (int c = 0; c < 8; ++c) e[c] = __shfl_sync(0xffffffffu, el, 2 * c);
#pragma unroll
            for (int p = 0; p < 4; ++p) O[p] = f2_dup(0.f);
#pragma unroll
            for (int m = 0; m < 4; ++m) {  // write and readout
                const f2 q2 = f2_dup(qt[32 * m]);
#pragma unroll
                for (int p = 0; p < 4; ++p) {
                    s2[m][p] = fma2(k2[m], f2_of(e[2 * p], e[2 * p + 1]), s2[m][p]);
                    O[p] = fma2(q2, s2[m][p], O[p]);
                }
            }
        }
        if (L > 0) {  // the last token's readout
            float o8[8] = {f2_lo(O[0]), f2_hi(O[0]), f2_lo(O[1]), f2_hi(O[1]),
                           f2_lo(O[2]), f2_hi(O[2]), f2_lo(O[3]), f2_hi(O[3])};
            const float ot = reduce8_32(o8, lane);
            if ((lane & 3) == 0) so[(L - 1) * kD + c0w + ((lane >> 2) & 7)] = ot;
        }
        // the final state back into the stage for the producer's tensor-map stores; release it
        if (has_sfin) {
#pragma unroll
            for (int m = 0; m < 4; ++m) {
                const int r = lane + 32 * m;
#pragma unroll
                for (int hf = 0; hf < 2; ++hf)
                    *reinterpret_cast<float4*>(st + state_off(r, c0w + 4 * hf)) =
                        make_float4(f2_lo(s2[m][2 * hf]), f2_hi(s2[m][2 * hf]), f2_lo(s2[m][2 * hf + 1]),
                                    f2_hi(s2[m][2 * hf + 1]));
            }
            tc::fence_async_smem();
        }
        mbar_arrive(&done[b]);
    }
    if (my_units > 0 && !failed) {  // the last unit's outputs, once every token's o is complete
        cbar();
        emit_unit(a_prev, h_prev, L_prev, (my_units - 1) & 1, 0, kCompute / 32);
    }
}

// dynamic shared memory: two stages, the permuted q, k, e^g factors and o, alignment slack
template <typename Tio>
uint32_t short_tma_smem(int Lmax) {
    return 2 * TmaStage<Tio>(Lmax).bytes + (3u * kFs + kD) * (uint32_t)Lmax * 4u + 1024u;
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
    const uint64_t srows = (uint64_t)a.N * a.H * kD;  // states as [units * 128][128] fp32
    if (ok && a.initial_state) ok = encode_tensor_map_2d(&maps.s_in, a.initial_state, true, kD, srows, kD * 4, 32, kD, true);
    if (ok && a.final_state) ok = encode_tensor_map_2d(&maps.s_out, a.final_state, true, kD, srows, kD * 4, 32, kD, true);
    if (!ok) return cudaErrorInvalidValue;
    DeviceInfo d;
    const int sms = current_device_info(&d) ? d.sm_count : 148;
    const int units = a.N * a.H;
    kern<<<units < sms ? units : sms, kThreads, smem, s>>>(
        maps, Lmax, a.gate ? 1 : 0, a.initial_state ? 1 : 0, a.final_state ? 1 : 0, (const Tio*)a.conv_state_in,
        (Tio*)a.conv_state_out, a.beta, a.conv_w, a.rms_w, a.eps_l2, a.eps_rms, a.scale, a.N, a.H, a.cu_seqlens,
        a.T_total, (To*)a.out, a.d_status);
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
    return smem + kStaticSmem <= 232448u;  // dynamic + static within the per-block limit
}

cudaError_t launch_short_tma(const kda_prefill_args& a, cudaStream_t s) {
    if ((int64_t)a.N * a.H == 0) return cudaSuccess;
    if (a.io == KDA_BF16)
        return a.out_dtype == KDA_FP32 ? short_tma_launch<bf16, float>(a, s) : short_tma_launch<bf16, bf16>(a, s);
    return a.out_dtype == KDA_FP32 ? short_tma_launch<float, float>(a, s) : short_tma_launch<float, bf16>(a, s);
}

}  // namespace kda
