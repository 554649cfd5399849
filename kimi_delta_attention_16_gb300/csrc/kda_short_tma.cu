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
// ranges of units with three kinds of warps and two rings in shared memory:
//
//  - a producer warp (one thread) fills row slot i % 2 with unit i's token rows
//    (one box of Lmax rows for each of q, k, v, gate and g, the conv window by
//    1D bulk copies, the betas by plain loads) as soon as the prep warps have
//    read unit i - 2's rows there, and state slot i % 2 with its state (four 2D
//    tensor-map boxes of 32 columns with the 128-byte swizzle) once the compute
//    warps are through unit i - 2, whose final state it first sends out by
//    four tensor-map stores;
//  - four prep warps form everything of a unit that does not involve the state
//    (conv + SiLU, e^g, the gate sigmoids, the L2 norms, the betas) into the
//    factor buffers of the unit's parity, ahead of the compute warps, and
//    normalise a unit's outputs (RMSNorm, weight, gate) once its tokens are
//    through;
//  - sixteen compute warps run the token chain of each unit from its state
//    slot and write the final state back there; they never wait for one
//    another.
//
// Because the rows have a ring of their own, a unit's factors are ready long
// before its tokens run, and the state ring alone paces the unit.  Every
// hand-over is an mbarrier with a bounded wait.
//
// Compute warp w owns value columns 8 w .. 8 w + 7 and lane l owns the rows
// l, l + 32, l + 64, l + 96 of all eight, as packed fp32 pairs of adjacent
// columns.  A token's per-row factors (q, k, e^g) are then read by the 32
// lanes of a warp from 32 consecutive floats (one shared-memory wavefront per
// 32 values), and the column sums over the key rows (the probe S_bar^T k and
// the readout S^T q) are one transposed reduction of the eight columns over
// the warp; no barrier is needed between tokens.  The state's shared-memory
// accesses (row r, column c at 16-byte chunk ((c mod 32) / 4) xor (r mod 8) of
// the swizzle) are conflict-free: the eight lanes of a quarter-warp read eight
// consecutive rows.
#include "kda_internal.cuh"
#include "kda_tc.cuh"
#include "kda_tc_ptx.cuh"

namespace kda {

namespace {

constexpr int kD = 128;
constexpr int kCompute = 512;             // sixteen compute warps
constexpr int kPrep = 128;                // four prep warps
constexpr int kThreads = kCompute + kPrep + 32;  // + the producer warp
constexpr int kL8 = kShortMaxL;
constexpr int kFs = kD;  // per-token stride (floats) of the factor arrays
// static shared memory of the kernel (sv[2], sgate[2], sW, sRms, snorm[2], sbeta, sbf, spart,
// ten barriers)
constexpr uint32_t kStaticSmem =
    4u * (4 * kL8 * kD + 3 * kD * 4 + kD + 2 * kL8 * 2 + 2 * kL8 + 2 * kL8 + (kPrep / 32) * kL8 * 2) + 80u;
constexpr uint32_t kStateSlot = 65536;  // one state: four 2D boxes of 32 columns x 128 rows, fp32

__host__ __device__ constexpr uint32_t align128(uint32_t x) { return (x + 127u) & ~127u; }

// Byte offsets inside one slot of the row ring for boxes of Lmax token rows (the states have a
// ring of their own, two 64 KB slots with the 128-byte swizzle ahead of the row slots).
template <typename Tio>
struct RowSlot {
    uint32_t conv, rows, part, g, bytes;
    __host__ __device__ explicit RowSlot(int Lmax) {
        conv = 0;                                                         // [3][128][3] Tio
        rows = align128(3 * kD * 3 * (uint32_t)sizeof(Tio));             // [4][Lmax][128] Tio: q, k, v, gate
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

// named barrier 1 of the prep warps (no other warp joins it)
__device__ __forceinline__ void pbar() { asm volatile("bar.sync 1, %0;" ::"n"(kPrep) : "memory"); }
__device__ __forceinline__ bool pbar_or(bool v) {
    uint32_t r;
    asm volatile(
        "{\n\t.reg .pred p, q;\n\tsetp.ne.u32 p, %1, 0;\n\tbar.red.or.pred q, 1, %2, p;\n\tselp.u32 %0, 1, 0, q;\n\t}"
        : "=r"(r)
        : "r"(v ? 1u : 0u), "n"(kPrep)
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
    // state slot landed; compute warps done with a unit (its state slot and its factor buffers);
    // row slot landed; prep warps done reading a row slot; prep warps done forming a unit's factors
    __shared__ uint64_t sfull[2], done[2], rfull[2], rdone[2], ready[2];
    __shared__ __align__(16) float sv[2][kL8][kD];    // convolved v of every token, per unit parity
    __shared__ __align__(16) float sgate[2][kL8][kD]; // sigmoid(gate) of every token (1 without a gate)
    __shared__ __align__(16) float sW[3 * kD * 4];    // conv taps of the prep warps' current head
    __shared__ __align__(16) float sRms[kD];
    __shared__ float snorm[2][kL8][2];                // 1/|q|, 1/|k| per token
    __shared__ float sbeta[2][kL8];                   // betas per row slot (written by the producer)
    __shared__ float sbf[2][kL8];                     // betas per unit parity (copied by the prep warps)
    __shared__ float spart[kPrep / 32][kL8][2];       // per prep warp: partial sums of q^2, k^2

    const RowSlot<Tio> ST(Lmax);
    const uint32_t raw_addr = tc::smem_u32(smem_raw);
    uint8_t* sm = smem_raw + (((raw_addr + 1023u) & ~1023u) - raw_addr);
    const uint32_t sbase = tc::smem_u32(sm);
    // two state slots, two row slots, then per unit parity pb: q, k and e^g ([Lmax][kFs]) of every
    // token, then o before its normalisation ([Lmax][128])
    const uint32_t rbase = 2 * kStateSlot;  // first row slot
    float* const fbase = reinterpret_cast<float*>(sm + rbase + 2 * ST.bytes);
    auto fq = [&](int pb) { return fbase + (size_t)pb * 3 * Lmax * kFs; };
    auto fk = [&](int pb) { return fbase + ((size_t)pb * 3 + 1) * Lmax * kFs; };
    auto fa = [&](int pb) { return fbase + ((size_t)pb * 3 + 2) * Lmax * kFs; };
    auto so = [&](int pb) { return fbase + (size_t)6 * Lmax * kFs + (size_t)pb * Lmax * kD; };
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
    // unit i: (n, h), its first token a and its token count (at most Lmax: a device cu_seqlens
    // that disagrees with the host copy that sized the boxes is flagged by the prep warps)
    auto unit_rows = [&](int i, int& n, int& h, int64_t& a, bool flag) -> int {
        unit_of(i, n, h);
        int64_t e;
        seq_range(cu, n, T_total, a, e);
        int L = (int)(e - a);
        if (L > Lmax) {
            if (flag) flag_status(d_status, KDA_ERR_DEVICE_ARG);
            L = Lmax;
        }
        return L;
    };
    const uint32_t cs_bytes = 3u * kD * 3u * (uint32_t)sizeof(Tio);

    if (tid == 0) {
        for (int b = 0; b < 2; ++b) {
            tc::mbar_init(&sfull[b], 1);
            tc::mbar_init(&done[b], kCompute);
            tc::mbar_init(&rfull[b], 1);
            tc::mbar_init(&rdone[b], kPrep);
            tc::mbar_init(&ready[b], kPrep);
        }
        tc::fence_mbar_init();
    }
    for (int c = tid; c < kD; c += kThreads) sRms[c] = rms_w ? rms_w[c] : 1.f;
    __syncthreads();

    if (warp == (kCompute + kPrep) / 32) {
        // ------------------------------------------------------------ producer (one thread)
        // Unit i: its token rows into row slot i % 2 once the prep warps have read unit i - 2's
        // there, then its state into state slot i % 2 once the compute warps are through unit
        // i - 2, whose final state leaves first.  The rows of unit i + 1 are therefore issued as
        // soon as unit i - 2's tokens are done, well before the compute warps reach unit i + 1.
        if (lane != 0) return;
        const CUtensorMap* mp[7] = {&maps.q, &maps.k, &maps.v, &maps.g, &maps.gate, &maps.s_in, &maps.s_out};
        for (int m = 0; m < 7; ++m)
            if ((m != 4 || has_gate) && (m != 5 || has_s0) && (m != 6 || has_sfin))
                asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(mp[m])) : "memory");
        const uint32_t tx_rows = (cs_in ? cs_bytes : 0u) + (has_gate ? 4u : 3u) * ST.part + (uint32_t)Lmax * kD * 4u;
        const uint32_t tx_state = has_s0 ? kStateSlot : 0u;
        // bit b: a fill of state slot b in flight, its parity in bit 2 + b; bits 4 + r and 6 + r
        // the same for row slot r
        uint32_t pend = 0;
        bool failed = false;
        // unit j's tokens are through and its state is back in its slot: send it to final_state
        auto drain = [&](int j) -> bool {
            const int b = j & 1;
            if (!tc::mbar_wait(&done[b], (uint32_t)((j >> 1) & 1))) return false;
            if (has_sfin) {
                int n, h;
                unit_of(j, n, h);
                const int y = (n * H + h) * kD;
                for (int bx = 0; bx < 4; ++bx) tma_store_2d(&maps.s_out, 32 * bx, y, sbase + (uint32_t)b * kStateSlot + 16384u * bx);
                tc::bulk_commit();
                tc::bulk_wait_read<0>();  // the slot may be refilled once the stores have read it
            }
            return true;
        };
        for (int i = 0; i < my_units; ++i) {
            const int b = i & 1;
            int n, h;
            unit_of(i, n, h);
            int64_t a, e;
            seq_range(cu, n, T_total, a, e);
            // the rows (and betas) of unit i
            if (i >= 2 && !tc::mbar_wait(&rdone[b], (uint32_t)(((i - 2) >> 1) & 1))) {
                failed = true;
                break;
            }
#pragma unroll
            for (int t = 0; t < kL8; ++t) sbeta[b][t] = t < e - a ? beta[(a + t) * H + h] : 0.f;
            const uint32_t rs = sbase + rbase + (uint32_t)b * ST.bytes;
            tc::mbar_expect_tx(&rfull[b], tx_rows);  // (its arrival also releases the betas above)
            if (cs_in)
                for (int p = 0; p < 3; ++p)
                    tc::bulk_load(rs + ST.conv + (uint32_t)p * (cs_bytes / 3u),
                                  cs_in + (((int64_t)n * 3 + p) * HD + (int64_t)h * kD) * 3, cs_bytes / 3u, &rfull[b]);
            const int x = h * kD, y = (int)a;
            tma_load_2d(rs + ST.rows, &maps.q, x, y, &rfull[b]);
            tma_load_2d(rs + ST.rows + ST.part, &maps.k, x, y, &rfull[b]);
            tma_load_2d(rs + ST.rows + 2 * ST.part, &maps.v, x, y, &rfull[b]);
            if (has_gate) tma_load_2d(rs + ST.rows + 3 * ST.part, &maps.gate, x, y, &rfull[b]);
            tma_load_2d(rs + ST.g, &maps.g, x, y, &rfull[b]);
            pend = (pend & ~(0x50u << b)) | ((1u | ((uint32_t)((i >> 1) & 1) << 2)) << (4 + b));
            // the state of unit i
            if (i >= 2 && !drain(i - 2)) {
                failed = true;
                break;
            }
            tc::mbar_expect_tx(&sfull[b], tx_state);
            if (has_s0)
                for (int bx = 0; bx < 4; ++bx)
                    tma_load_2d(sbase + (uint32_t)b * kStateSlot + 16384u * bx, &maps.s_in, 32 * bx, (n * H + h) * kD, &sfull[b]);
            pend = (pend & ~(5u << b)) | ((1u | ((uint32_t)((i >> 1) & 1) << 2)) << b);
        }
        if (!failed)
            for (int j = my_units > 2 ? my_units - 2 : 0; j < my_units; ++j)
                if (!drain(j)) {
                    failed = true;
                    break;
                }
        if (failed) {  // fills in flight: wait for them (bounded) before the shared memory goes away
            for (int b = 0; b < 2; ++b) {
                if ((pend >> b) & 1u) tc::mbar_wait(&sfull[b], (pend >> (2 + b)) & 1u);
                if ((pend >> (4 + b)) & 1u) tc::mbar_wait(&rfull[b], (pend >> (6 + b)) & 1u);
            }
            flag_status(d_status, KDA_ERR_TIMEOUT);
        }
        tc::bulk_wait_all();
        return;
    }

    if (warp >= kCompute / 32) {
        // ------------------------------------------------------------ prep warps
        // Per unit j, ahead of the compute warps: conv + SiLU of the q, k, v channels (thread d:
        // channel d of each part), e^g and the gate sigmoids, the L2 norms and the betas, from
        // row slot j % 2 into the buffers of parity j & 1, then `rdone` (the row slot is free)
        // and `ready`.  Those buffers held unit j - 2: its outputs are normalised first, once
        // `done` shows that its tokens are through.
        const int ptid = tid - kCompute, pw = ptid >> 5, d = ptid;
        // outputs of unit j (warp pw for tokens pw, pw + 4): o = scale S^T q / |q| from the
        // readout sums, RMSNorm, weight, gate
        auto emit_unit = [&](int j) {
            int n, h;
            int64_t a;
            const int L = unit_rows(j, n, h, a, false), pb = j & 1, c0 = 4 * lane;
            for (int t = pw; t < L; t += kPrep / 32) {
                const float sq = scale * snorm[pb][t][0];
                float4 o = *reinterpret_cast<const float4*>(so(pb) + t * kD + c0);
                o.x *= sq;
                o.y *= sq;
                o.z *= sq;
                o.w *= sq;
                float ss = o.x * o.x + o.y * o.y + o.z * o.z + o.w * o.w;
#pragma unroll
                for (int off = 16; off > 0; off >>= 1) ss += __shfl_xor_sync(0xffffffffu, ss, off);
                const float inv = 1.0f / sqrtf(ss * (1.0f / kD) + eps_rms);
                const float4 rw = *reinterpret_cast<const float4*>(&sRms[c0]);
                const float4 gg = *reinterpret_cast<const float4*>(&sgate[pb][t][c0]);
                store4<To>(out + ((a + t) * H + h) * kD + c0, o.x * inv * rw.x * gg.x, o.y * inv * rw.y * gg.y,
                           o.z * inv * rw.z * gg.z, o.w * inv * rw.w * gg.w);
            }
        };
        int h_prev = -1;
        bool failed = false;
        for (int j = 0; j < my_units; ++j) {
            const int b = j & 1;
            int n, h;
            int64_t a;
            const int L = unit_rows(j, n, h, a, ptid == 0);
            if (j >= 2) {  // the buffers of parity b held unit j - 2: its tokens are through first
                const bool ok = ptid == 0 ? tc::mbar_wait(&done[b], (uint32_t)(((j - 2) >> 1) & 1)) : true;
                if (pbar_or(!ok)) {
                    failed = true;
                    break;
                }
                emit_unit(j - 2);
            }
            {  // the unit's rows have landed; conv taps of a new head
                const bool ok = ptid == 0 ? tc::mbar_wait(&rfull[b], (uint32_t)((j >> 1) & 1)) : true;
                if (h != h_prev)
                    for (int idx = ptid; idx < 3 * kD * 4; idx += kPrep) {
                        const int part = idx / (kD * 4), rem = idx % (kD * 4);
                        sW[idx] = conv_w[(part * HD + (int64_t)h * kD) * 4 + rem];
                    }
                h_prev = h;
                if (pbar_or(!ok)) {
                    failed = true;
                    break;
                }
            }
            const uint8_t* st = sm + rbase + (uint32_t)b * ST.bytes;
            if (ptid < kL8) sbf[b][ptid] = sbeta[b][ptid];  // (the row slot may be refilled before the tokens run)
            float sq2[kL8], sk2[kL8];  // squares of this channel's q and k per token
#pragma unroll
            for (int part = 0; part < 3; ++part) {  // conv + SiLU; the rolled window out
                const int ch = part * kD + d;
                float p0 = 0.f, p1 = 0.f, p2 = 0.f;  // x[-3], x[-2], x[-1]
                if (cs_in) {
                    const Tio* c3 = reinterpret_cast<const Tio*>(st + ST.conv) + ch * 3;
                    p0 = to_f(c3[0]);
                    p1 = to_f(c3[1]);
                    p2 = to_f(c3[2]);
                }
                const Tio* rp = reinterpret_cast<const Tio*>(st + ST.rows + (uint32_t)part * ST.part) + d;
                const float4 w = *reinterpret_cast<const float4*>(&sW[ch * 4]);
                float* dst = part == 0 ? fq(b) + d : part == 1 ? fk(b) + d : &sv[b][0][d];
                const int dstride = part == 2 ? kD : kFs;
                float xr[kL8];  // every token's raw value first: one shared-memory round trip
#pragma unroll
                for (int t = 0; t < kL8; ++t) xr[t] = t < L ? to_f(rp[t * kD]) : 0.f;
#pragma unroll
                for (int t = 0; t < kL8; ++t) {
                    float y = 0.f;
                    if (t < L) {
                        y = act_silu<Tio>(w.x * p0 + w.y * p1 + w.z * p2 + w.w * xr[t]);
                        dst[t * dstride] = y;
                        p0 = p1;
                        p1 = p2;
                        p2 = xr[t];
                    }
                    if (part == 0) sq2[t] = y * y;
                    if (part == 1) sk2[t] = y * y;
                }
                if (cs_out) {  // last three raw values of the sequence (exact copies of Tio values)
                    Tio* o3 = cs_out + (((int64_t)n * 3 + part) * HD + (int64_t)h * kD + d) * 3;
                    o3[0] = from_f<Tio>(p0);
                    o3[1] = from_f<Tio>(p1);
                    o3[2] = from_f<Tio>(p2);
                }
            }
            {  // decay factors and gate sigmoids of every token (channel d)
                const float* gs = reinterpret_cast<const float*>(st + ST.g);
                const Tio* gt = reinterpret_cast<const Tio*>(st + ST.rows + 3 * ST.part);
                for (int t = 0; t < L; ++t) {
                    fa(b)[t * kFs + d] = decay_exp<Tio>(gs[t * kD + d]);
                    sgate[b][t][d] = has_gate ? act_sigmoid<Tio>(to_f(gt[t * kD + d])) : 1.f;
                }
            }
            // L2 norms of q and k: sums over the warp, then over the four warps
#pragma unroll
            for (int t = 0; t < kL8; ++t) {
                if (t < L) {
                    float x = sq2[t], y = sk2[t];
#pragma unroll
                    for (int off = 16; off > 0; off >>= 1) {
                        x += __shfl_xor_sync(0xffffffffu, x, off);
                        y += __shfl_xor_sync(0xffffffffu, y, off);
                    }
                    if (lane == 0) {
                        spart[pw][t][0] = x;
                        spart[pw][t][1] = y;
                    }
                }
            }
            pbar();
            if (ptid < 2 * L) {
                const int t = ptid >> 1, qk = ptid & 1;
                float ssum = 0.f;
#pragma unroll
                for (int w4 = 0; w4 < kPrep / 32; ++w4) ssum += spart[w4][t][qk];
                snorm[b][t][qk] = 1.0f / sqrtf(ssum + eps_l2);
            }
            mbar_arrive(&rdone[b]);  // every read of the row slot is done
            mbar_arrive(&ready[b]);  // (releases every prep thread's writes of the unit's factors)
        }
        if (!failed)  // the last two units' outputs
            for (int j = my_units > 2 ? my_units - 2 : 0; j < my_units; ++j) {
                const bool ok = ptid == 0 ? tc::mbar_wait(&done[j & 1], (uint32_t)((j >> 1) & 1)) : true;
                if (pbar_or(!ok)) {
                    failed = true;
                    break;
                }
                emit_unit(j);
            }
        if (failed && ptid == 0) flag_status(d_status, KDA_ERR_TIMEOUT);
        return;
    }

    // ---------------------------------------------------------------- compute warps
    // Per unit i: the state from its slot into registers, the tokens, the readouts into o, the
    // final state back into the slot, then `done`.  The warps never wait for one another: each
    // owns its eight value columns, and lane 0 of each warp polls the barriers for it.
    const int c0w = 8 * warp;  // the warp's first value column
    for (int i = 0; i < my_units; ++i) {
        const int b = i & 1;
        int n, h;
        int64_t a;
        const int L = unit_rows(i, n, h, a, false);
        {
            bool ok = true;
            if (lane == 0)
                ok = tc::mbar_wait(&sfull[b], (uint32_t)((i >> 1) & 1)) && tc::mbar_wait(&ready[b], (uint32_t)((i >> 1) & 1));
            if (!__all_sync(0xffffffffu, ok)) {
                if (lane == 0) flag_status(d_status, KDA_ERR_TIMEOUT);
                break;
            }
            __syncwarp();
        }
        uint8_t* st = sm + (uint32_t)b * kStateSlot;
        // the state into registers: s2[m][p] = columns c0w + 2 p, c0w + 2 p + 1 of row lane + 32 m
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
        // ---- tokens: no barrier between them.  The eight columns' sums over the warp go through one
        // transposed reduction per token, which carries token t's probe together with token
        // t - 1's readout (so the readout never adds a reduction of its own to the chain).
        const float* fqb = fq(b);
        const float* fkb = fk(b);
        const float* fab = fa(b);
        float* sob = so(b);
        f2 O[4] = {f2_dup(0.f), f2_dup(0.f), f2_dup(0.f), f2_dup(0.f)};  // readout of the previous token
        for (int t = 0; t < L; ++t) {
            const float* kt = fkb + t * kFs + lane;
            const float* at = fab + t * kFs + lane;
            const float* qt = fqb + t * kFs + lane;
            const float ik = snorm[b][t][1];
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
            if (t > 0 && lane >= 16 && (lane & 1) == 0) sob[(t - 1) * kD + c0w + ((lane >> 1) - 8)] = red;
            // lanes 2c, 2c + 1 hold column c's probe: each lane forms the correction of the column
            // it holds (lanes 16-31 form unused values), then the eight are passed round
            const float el = sbf[b][t] * ik * (sv[b][t][c0w + ((lane >> 1) & 7)] - ik * red);
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
            if ((lane & 3) == 0) sob[(L - 1) * kD + c0w + ((lane >> 2) & 7)] = ot;
        }
        // the final state back into its slot for the producer's tensor-map stores; release the
        // slot and the unit's factor buffers
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
}

// dynamic shared memory: two state slots, two row slots, two sets (per unit parity) of the q, k,
// e^g factors and o, alignment slack
template <typename Tio>
uint32_t short_tma_smem(int Lmax) {
    return 2 * kStateSlot + 2 * RowSlot<Tio>(Lmax).bytes + 2 * (3u * kFs + kD) * (uint32_t)Lmax * 4u + 1024u;
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
