// kda_segscan.cu -- the two kernels that finish a segmented tensor-core
// prefill (D = 128): the in-order composition of the segments' affine state
// maps, and the output fix-up.
//
// Page "Kimi K3 / Architecture", KDA panel: the state is carried from chunk to
// chunk, and each step maps it as S -> (I - beta k k^T) Diag(e^g) S + beta k v^T,
// which is affine in S with a key-by-key linear part.  A run of steps is
// therefore affine too: segment s maps its start state S_s to
// S_{s+1} = M_s S_s + B_s, and each readout o_t = scale S_t^T q_t (and the
// intra-chunk terms that depend on S through v - S^T k) to o_t' + S_s^T f_t.
// The prefill kernel measures B_s and o_t' by running the segment from S = 0,
// and M_s and f_t by running it from S = I with v = 0.
#include "kda_tc.cuh"
#include "kda_tc_ptx.cuh"

namespace kda {

namespace {

constexpr int kD = 128;

__device__ __forceinline__ void cp_async16(uint32_t dst, const void* src) {
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(dst), "l"(src) : "memory");
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }
__device__ __forceinline__ void cp_async_wait_all() { asm volatile("cp.async.wait_group 0;" ::: "memory"); }

// ---------------------------------------------------------------- composition
// One block of 512 threads per unit walks its segments in order on the tensor cores
// (kind::f16, 3-term bf16 split, fp32 accumulate in TMEM):
//
//   S_{s+1}^T = S_s^T . M_s^T + B_s^T      A = S_s^T (TMEM, hi/lo), B = M_s (smem, hi/lo, K-major)
//
// Thread (lane j = 32 (warp % 4) + lane, quarter qt = warp / 4) owns rows c in
// [32 qt, 32 qt + 32) of column j of the states: it adds B_s[c][j] to its accumulator
// entries, stores S_{s+1}[c][j] (coalesced over j) and splits them back into the A operand
// for the next step.  M_s arrives as coalesced 32-byte pieces, four per thread.
constexpr int kCombThreads = 512;
constexpr uint32_t kCombOffBhi = 0;
constexpr uint32_t kCombOffBlo = 32768;
constexpr size_t kCombSmem = 65536 + 1024;  // + alignment slack
constexpr uint32_t kCombTmemCols = 256;     // S^T hi/lo [0,128), accumulator [128,256)

__device__ __forceinline__ void split2c(float a, float b, uint32_t& hi, uint32_t& lo) {
    hi = pack_bf16x2(a, b);
    const float ah = __uint_as_float(hi << 16), bh = __uint_as_float(hi & 0xffff0000u);
    lo = pack_bf16x2(a - ah, b - bh);
}

__global__ void __launch_bounds__(kCombThreads, 1)
k_seg_combine(SegPlan sp, float* __restrict__ S_fin, int* d_status) {
    using namespace tc;
    extern __shared__ uint8_t csm_raw[];
    __shared__ uint64_t bar;
    __shared__ uint32_t s_tbase;
    const uint32_t raw_addr = smem_u32(csm_raw);
    uint8_t* sm = csm_raw + (((raw_addr + 1023u) & ~1023u) - raw_addr);
    const uint32_t sbase = smem_u32(sm);
    const int u = blockIdx.x;
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int qd = warp & 3, qt = warp >> 2;
    const int j = 32 * qd + lane;
    const uint32_t lane_off = (uint32_t)(qd * 32) << 16;
    const int P = sp.P;
    const int64_t DD = (int64_t)kD * kD;
    const float* E = sp.end_state + (int64_t)u * P * DD;
    const float* M = sp.trans + (int64_t)u * P * DD;
    float* St = sp.start + (int64_t)u * P * DD;

    if (warp == 0) {
        tmem_alloc(&s_tbase, kCombTmemCols);
        tmem_relinquish();
    }
    if (tid == 0) {
        mbar_init(&bar, 1);
        fence_mbar_init();
    }
    fence_before_sync();
    __syncthreads();
    fence_after_sync();
    const uint32_t tb = s_tbase;
    const uint32_t idesc = idesc_bf16(128, 128, false, false);

    // rows [32 qt, 32 qt + 32) of column j -> A operand columns of that K range
    auto put_operand = [&](const float (&col)[32]) {
        uint32_t hi[16], lo[16];
#pragma unroll
        for (int i = 0; i < 16; ++i) split2c(col[2 * i], col[2 * i + 1], hi[i], lo[i]);
        tmem_st16(tb + lane_off + 16 * qt, hi);
        tmem_st16(tb + lane_off + 64 + 16 * qt, lo);
        tmem_st_wait();
    };
    {
        float col[32];
#pragma unroll
        for (int i = 0; i < 32; ++i) col[i] = E[(int64_t)(32 * qt + i) * kD + j];
#pragma unroll
        for (int i = 0; i < 32; ++i) St[DD + (int64_t)(32 * qt + i) * kD + j] = col[i];  // S_1
        put_operand(col);
    }
    bool failed = false;
    for (int s = 1; s < P; ++s) {
        // M_s -> B tile (K-major, 128-byte swizzle), hi and lo: piece (row c, k8) per thread
        {
            float4 a[4], b[4];
#pragma unroll
            for (int t = 0; t < 4; ++t) {
                const int idx = tid + t * kCombThreads, c = idx >> 4, k8 = idx & 15;
                const float* src = M + s * DD + (int64_t)c * kD + 8 * k8;
                a[t] = *reinterpret_cast<const float4*>(src);
                b[t] = *reinterpret_cast<const float4*>(src + 4);
            }
#pragma unroll
            for (int t = 0; t < 4; ++t) {
                const int idx = tid + t * kCombThreads, c = idx >> 4, k8 = idx & 15;
                uint4 hv, lv;
                split2c(a[t].x, a[t].y, hv.x, lv.x);
                split2c(a[t].z, a[t].w, hv.y, lv.y);
                split2c(b[t].x, b[t].y, hv.z, lv.z);
                split2c(b[t].z, b[t].w, hv.w, lv.w);
                *reinterpret_cast<uint4*>(sm + kCombOffBhi + kmajor_off(128, c, k8)) = hv;
                *reinterpret_cast<uint4*>(sm + kCombOffBlo + kmajor_off(128, c, k8)) = lv;
            }
        }
        fence_async_smem();
        fence_before_sync();
        __syncthreads();
        if (tid == 0) {
            fence_after_sync();
#pragma unroll
            for (int term = 0; term < 3; ++term) {
                const uint32_t acol = term == 1 ? 64 : 0;
                const uint32_t bt = sbase + (term == 2 ? kCombOffBlo : kCombOffBhi);
#pragma unroll
                for (int kk = 0; kk < 8; ++kk)
                    mma_ts(tb + 128, tb + acol + 8 * kk, desc_sw128(bt + (kk >> 2) * 128 * 128 + (kk & 3) * 32, 16, 1024),
                           idesc, (term | kk) != 0);
            }
            mma_commit(&bar);
        }
        // B_s entries of this thread, fetched while the tensor cores work
        float col[32];
        const float* Bs = E + s * DD;
#pragma unroll
        for (int i = 0; i < 32; ++i) col[i] = Bs[(int64_t)(32 * qt + i) * kD + j];
        failed = !__syncthreads_and(mbar_wait(&bar, (uint32_t)(s - 1) & 1u));
        if (failed) break;
        fence_after_sync();
        {
            uint32_t dv[32];
            tmem_ld32(tb + lane_off + 128 + 32 * qt, dv);
            tmem_ld_wait();
#pragma unroll
            for (int i = 0; i < 32; ++i) col[i] += __uint_as_float(dv[i]);
        }
        // S_{s+1}[c][j] for c in [32 qt, 32 qt + 32)
        float* dst = s + 1 < P ? St + (s + 1) * DD : (S_fin ? S_fin + (int64_t)u * DD : nullptr);
        if (dst)
#pragma unroll
            for (int i = 0; i < 32; ++i) dst[(int64_t)(32 * qt + i) * kD + j] = col[i];
        fence_before_sync();
        __syncthreads();  // every accumulator read and every read of the B tile is done
        fence_after_sync();
        if (s + 1 < P) put_operand(col);
    }
    if (failed && tid == 0) flag_status(d_status, KDA_ERR_TIMEOUT);
    fence_before_sync();
    __syncthreads();
    if (warp == 0) tmem_dealloc(tb, kCombTmemCols);
}

// ---------------------------------------------------------------- fix-up
// Block (pair, y): pair = u * (P - 1) + s - 1 names (unit, segment s >= 1); the
// block takes 64-token tiles y, y + gridDim.y, ... of that segment.  Per tile,
// on the tensor cores (kind::f16, fp32 accumulate in TMEM):
//
//   O^T[j][t] = sum_k S_s[k][j] F[t][k]      A = S_s^T (TMEM, hi/lo), B = F tile (smem, hi/lo)
//
// with the 3-term bf16 split hi.hi + lo.hi + hi.lo (about 2^-16 relative), then
// o = o' + O, y = o / sqrt(mean_j o^2 + eps) * w_j * sigmoid(gate).  Thread
// (lane j = 32 (warp % 4) + lane, half qt = warp / 4) finishes tokens
// [32 qt, 32 qt + 32) of value channel j, so the o', gate and y rows are
// read and written coalesced.  The next tile's F and gate rows are fetched
// with cp.async while the current one is multiplied and finished; two blocks
// share an SM (about 101 KB of shared memory and 256 TMEM columns each) and
// hide each other's load round-trips.
constexpr int kFixThreads = 256;
constexpr int kFixTile = 64;                  // tokens per tile (MMA N)
constexpr uint32_t kFixRawStride = 528;       // fp32 F rows, padded: conflict-free 16-byte reads
constexpr uint32_t kFixOffRaw = 0;
constexpr uint32_t kFixOffBhi = 34816;        // 64 x 528, rounded to 1024
constexpr uint32_t kFixOffBlo = kFixOffBhi + kFixTile * 256;
constexpr uint32_t kFixOffGate = kFixOffBlo + kFixTile * 256;  // 2 x [64 tokens][128] bf16
constexpr uint32_t kFixOffRed = kFixOffGate + 2 * kFixTile * 256;  // [4 quadrants][64 tokens] fp32
constexpr uint32_t kFixOffInv = kFixOffRed + 4 * kFixTile * 4;     // [64] fp32
constexpr size_t kFixSmem = kFixOffInv + kFixTile * 4 + 1024;  // + alignment slack
constexpr uint32_t kFixTmemCols = 256;        // S^T hi/lo [0,128), O^T [128,192)
static_assert(kFixTile * kFixRawStride <= kFixOffBhi, "F staging overlaps the operand tile");

__device__ __forceinline__ void split2(float a, float b, uint32_t& hi, uint32_t& lo) {
    hi = pack_bf16x2(a, b);
    const float ah = __uint_as_float(hi << 16), bh = __uint_as_float(hi & 0xffff0000u);
    lo = pack_bf16x2(a - ah, b - bh);
}

template <typename To>
__global__ void __launch_bounds__(kFixThreads, 2)
k_seg_fixup(SegPlan sp, const int32_t* __restrict__ cu, int64_t T_total, int H,
            const bf16* __restrict__ gate, const float* __restrict__ rms_w, float eps_rms,
            To* __restrict__ out, int* d_status) {
    using namespace tc;
    extern __shared__ uint8_t fsm_raw[];
    __shared__ uint64_t bar;
    __shared__ uint32_t s_tbase;
    const int Pm = sp.P - 1;
    const int u = blockIdx.x / Pm, s = blockIdx.x % Pm + 1;
    const int n = u / H, h = u % H;
    int64_t s0, s1;
    seq_range(cu, n, T_total, s0, s1);
    int64_t cb, ce;
    seg_chunk_range((s1 - s0 + 63) / 64, sp.P, sp.w, sp.wd, s, cb, ce);
    const int64_t ta = s0 + cb * 64;
    const int64_t tz = s0 + ce * 64 < s1 ? s0 + ce * 64 : s1;
    const int64_t ntiles = tz > ta ? (tz - ta + kFixTile - 1) / kFixTile : 0;
    if ((int64_t)blockIdx.y >= ntiles) return;

    const uint32_t raw_addr = smem_u32(fsm_raw);
    uint8_t* sm = fsm_raw + (((raw_addr + 1023u) & ~1023u) - raw_addr);
    const uint32_t sbase = smem_u32(sm);
    float* sRed = reinterpret_cast<float*>(sm + kFixOffRed);
    float* sInv = reinterpret_cast<float*>(sm + kFixOffInv);
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int qd = warp & 3, qt = warp >> 2;
    const int j = qd * 32 + lane;
    const uint32_t lane_off = (uint32_t)(qd * 32) << 16;

    if (warp == 0) {
        tmem_alloc(&s_tbase, kFixTmemCols);
        tmem_relinquish();
    }
    if (tid == 0) {
        mbar_init(&bar, 1);
        fence_mbar_init();
    }
    // F rows of a tile -> raw staging (fp32, padded rows) and its gate rows -> gate buffer
    // gbuf, one cp.async group
    auto stage = [&](int64_t tile, uint32_t gbuf) {
        const int64_t tb = ta + kFixTile * tile;
        for (int idx = tid; idx < kFixTile * 32; idx += kFixThreads) {
            const int row = idx >> 5, c4 = idx & 31;
            if (tb + row < tz)
                cp_async16(sbase + kFixOffRaw + row * kFixRawStride + 16 * c4,
                           sp.f_tr + ((tb + row) * H + h) * kD + 4 * c4);
        }
        if (gate)
            for (int idx = tid; idx < kFixTile * 16; idx += kFixThreads) {
                const int row = idx >> 4, c8 = idx & 15;
                if (tb + row < tz)
                    cp_async16(sbase + kFixOffGate + gbuf * (kFixTile * 256) + row * 256 + 16 * c8,
                               gate + ((tb + row) * H + h) * kD + 8 * c8);
            }
        cp_async_commit();
    };
    stage(blockIdx.y, 0);
    fence_before_sync();
    __syncthreads();
    fence_after_sync();
    const uint32_t tb = s_tbase;
    {
        // S_s^T operand: lane j holds column j of S_s, K = key channels [64 qt, 64 qt + 64)
        const float* St = sp.start + ((int64_t)u * sp.P + s) * kD * kD;
#pragma unroll
        for (int part = 2 * qt; part < 2 * qt + 2; ++part) {
            uint32_t hi[16], lo[16];
#pragma unroll
            for (int i = 0; i < 16; ++i)
                split2(St[(int64_t)(32 * part + 2 * i) * kD + j], St[(int64_t)(32 * part + 2 * i + 1) * kD + j], hi[i], lo[i]);
            tmem_st16(tb + lane_off + 16 * part, hi);
            tmem_st16(tb + lane_off + 64 + 16 * part, lo);
        }
        tmem_st_wait();
    }
    const float wj = rms_w ? rms_w[j] : 1.f;
    const uint32_t idesc = idesc_bf16(128, kFixTile, false, false);
    bool failed = false;
    uint32_t iter = 0;
    for (int64_t tile = blockIdx.y; tile < ntiles; tile += gridDim.y, ++iter) {
        const int64_t t0 = ta + kFixTile * tile;
        cp_async_wait_all();
        __syncthreads();  // raw F rows of this tile landed
        // raw fp32 -> hi/lo bf16, K-major 128-byte swizzle (rows past the segment are zero)
        for (int idx = tid; idx < kFixTile * 16; idx += kFixThreads) {
            const int row = idx >> 4, c8 = idx & 15;
            uint4 hv = make_uint4(0, 0, 0, 0), lv = make_uint4(0, 0, 0, 0);
            if (t0 + row < tz) {
                const float4 a = *reinterpret_cast<const float4*>(sm + kFixOffRaw + row * kFixRawStride + 32 * c8);
                const float4 b = *reinterpret_cast<const float4*>(sm + kFixOffRaw + row * kFixRawStride + 32 * c8 + 16);
                split2(a.x, a.y, hv.x, lv.x);
                split2(a.z, a.w, hv.y, lv.y);
                split2(b.x, b.y, hv.z, lv.z);
                split2(b.z, b.w, hv.w, lv.w);
            }
            *reinterpret_cast<uint4*>(sm + kFixOffBhi + kmajor_off(kFixTile, row, c8)) = hv;
            *reinterpret_cast<uint4*>(sm + kFixOffBlo + kmajor_off(kFixTile, row, c8)) = lv;
        }
        fence_async_smem();
        fence_before_sync();
        __syncthreads();  // operand tile complete; raw staging free
        if (tile + gridDim.y < ntiles) stage(tile + gridDim.y, (iter + 1) & 1u);
        if (tid == 0) {
            fence_after_sync();
#pragma unroll
            for (int term = 0; term < 3; ++term) {
                const uint32_t acol = term == 1 ? 64 : 0;
                const uint32_t bt = sbase + (term == 2 ? kFixOffBlo : kFixOffBhi);
#pragma unroll
                for (int kk = 0; kk < 8; ++kk)
                    mma_ts(tb + 128, tb + acol + 8 * kk,
                           desc_sw128(bt + (kk >> 2) * kFixTile * 128 + (kk & 3) * 32, 16, 1024), idesc,
                           (term | kk) != 0);
            }
            mma_commit(&bar);
        }
        // o' of this thread's 32 tokens, fetched while the tensor cores work
        const int64_t row0 = t0 + 32 * qt;                // first token of this thread
        const int nvalid = (int)(tz - row0 < 32 ? (tz - row0 < 0 ? 0 : tz - row0) : 32);
        const int64_t rstride = (int64_t)H * kD;          // elements between tokens
        const float* op = sp.o_loc + (row0 * H + h) * kD + j;
        float o[32];
#pragma unroll
        for (int e = 0; e < 32; ++e) o[e] = e < nvalid ? op[e * rstride] : 0.f;
        failed = !__syncthreads_and(mbar_wait(&bar, iter & 1u));
        if (failed) break;
        fence_after_sync();
#pragma unroll
        for (int half = 0; half < 2; ++half) {
            uint32_t dv[16];
            tmem_ld16(tb + lane_off + 128 + 32 * qt + 16 * half, dv);
            tmem_ld_wait();
#pragma unroll
            for (int e = 0; e < 16; ++e) o[16 * half + e] += __uint_as_float(dv[e]);
        }
        // sum over the warp's 32 channels of o^2, 16 tokens at a time: halve across lanes
        // 8, 4, 2, 1 apart, fold the two 16-lane halves (lane l then holds token l % 16 of
        // the group), then over the four quadrant warps through shared memory
        float tot = 0.f;
#pragma unroll
        for (int grp = 0; grp < 2; ++grp) {
            float sq[16];
#pragma unroll
            for (int e = 0; e < 16; ++e) sq[e] = o[16 * grp + e] * o[16 * grp + e];
#pragma unroll
            for (int sh = 8; sh >= 1; sh >>= 1) {
                const bool upper = (lane & sh) != 0;
#pragma unroll
                for (int i = 0; i < sh; ++i) {
                    const float send = upper ? sq[i] : sq[i + sh];
                    const float keep = upper ? sq[i + sh] : sq[i];
                    sq[i] = keep + __shfl_xor_sync(0xffffffffu, send, sh);
                }
            }
            sq[0] += __shfl_xor_sync(0xffffffffu, sq[0], 16);
            if ((lane >> 4) == grp) tot = sq[0];  // lane l keeps token 16 grp + l % 16 = l
        }
        sRed[qd * kFixTile + 32 * qt + lane] = tot;
        __syncthreads();
        if (tid < kFixTile)
            sInv[tid] = rsqrtf((sRed[tid] + sRed[kFixTile + tid] + sRed[2 * kFixTile + tid] +
                                sRed[3 * kFixTile + tid]) * (1.0f / kD) + eps_rms);
        __syncthreads();
        const bf16* gt = reinterpret_cast<const bf16*>(sm + kFixOffGate + (iter & 1u) * (kFixTile * 256)) +
                         32 * qt * kD + j;
        To* yp = out + (row0 * H + h) * kD + j;
#pragma unroll
        for (int e = 0; e < 32; ++e) {
            if (e < nvalid) {
                float y = o[e] * sInv[32 * qt + e] * wj;
                if (gate) y *= sigmoid_tanh(to_f(gt[e * kD]));
                yp[e * rstride] = from_f<To>(y);
            }
        }
        fence_before_sync();  // this tile's TMEM reads precede the next tile's MMAs (barrier above them)
    }
    cp_async_wait_all();
    if (failed && tid == 0) flag_status(d_status, KDA_ERR_TIMEOUT);
    fence_before_sync();
    __syncthreads();
    if (warp == 0) tmem_dealloc(tb, kFixTmemCols);
}

}  // namespace

cudaError_t launch_seg_combine(const SegPlan& sp, int units, float* S_fin, int* d_status, cudaStream_t s) {
    if (sp.P <= 1 || units <= 0) return cudaSuccess;
    cudaError_t e = cudaFuncSetAttribute(k_seg_combine, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         (int)kCombSmem);
    if (e != cudaSuccess) return e;
    k_seg_combine<<<(unsigned)units, kCombThreads, kCombSmem, s>>>(sp, S_fin, d_status);
    return cudaGetLastError();
}

cudaError_t launch_seg_fixup(const SegPlan& sp, const int32_t* cu, int N, int64_t T_total, int H,
                             const bf16* gate, const float* rms_w, float eps_rms, void* out,
                             kda_dtype out_dt, int sms, int* d_status, cudaStream_t s) {
    const int64_t pairs = (int64_t)N * H * (sp.P - 1);
    if (sp.P <= 1 || pairs <= 0 || T_total <= 0) return cudaSuccess;
    // two blocks per SM (shared memory, TMEM and registers allow no more); about four
    // blocks per SM over the pairs, so the last wave is short
    int64_t gy = (4 * (int64_t)sms + pairs - 1) / pairs;
    const int64_t max_tiles = (T_total + kFixTile - 1) / kFixTile;
    if (gy > max_tiles) gy = max_tiles;
    if (gy > 65535) gy = 65535;
    if (gy < 1) gy = 1;
    const dim3 grid((unsigned)pairs, (unsigned)gy);
    cudaError_t e;
    if (out_dt == KDA_FP32) {
        auto kern = k_seg_fixup<float>;
        if ((e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)kFixSmem)))
            return e;
        kern<<<grid, kFixThreads, kFixSmem, s>>>(sp, cu, T_total, H, gate, rms_w, eps_rms,
                                                 static_cast<float*>(out), d_status);
    } else {
        auto kern = k_seg_fixup<bf16>;
        if ((e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)kFixSmem)))
            return e;
        kern<<<grid, kFixThreads, kFixSmem, s>>>(sp, cu, T_total, H, gate, rms_w, eps_rms,
                                                 static_cast<bf16*>(out), d_status);
    }
    return cudaGetLastError();
}

}  // namespace kda
