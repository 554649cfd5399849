// kda_prefill_tc.cu -- fused KDA prefill on the Blackwell tensor cores
// (tcgen05, accumulators in tensor memory), D = 128, chunk C = 64, bf16 inputs.
//
// Page "Kimi K3 / Architecture", KDA panel: the chunkwise form, in which the
// state recurs from chunk to chunk and the tokens of a chunk are taken together
// as dense tensor-core tiles; page "Animated Kimi K3 architecture diagram": the
// state is carried across chunks.
//
// One CTA owns one (sequence, head) and walks its chunks in order; every
// stage of the layer runs inside it (conv + SiLU + L2, the chunk algebra,
// the state carry, RMSNorm + gate), so HBM sees only the layer's own inputs
// and outputs.  With a segmented plan (P > 1, few units) the grid holds
// 2P - 1 roles per unit: role 0 walks segment 0 from the initial state as
// above; role 2s - 1 walks segment s from a zero state and role 2s walks it
// with v = 0 from the identity.  Those two write scale * o in fp32 (no
// epilogue) and their end states; the combine and fix-up kernels finish.  Per chunk, with local token index r, G = cumulative log-decay,
// w = beta e (all per key channel c, value channel j):
//
//   G1  [M ; A]  = X1 . B1^T          intra-chunk q.k and beta k.k with decay  (N = 96)
//   G3  [P ; Q'] = S^T . [KG ; QG]^T  inter-chunk reads of the carried state  (N = 128)
//   T   = (I + A)^-1                  unit lower triangular, SIMT in shared memory
//   R   = beta (V - P)
//   G4  W^T = R^T . T^T                                                       (N = 64)
//   G5  O^T = Q'^T + W^T . M^T                                                (N = 64)
//   G6  dS^T = W^T . Kt                                                       (N = 128)
//   S  <- Diag(e^{G_last}) S + dS ;  y = RMSNorm(scale O) * w * sigmoid(gate)
//
// Decay factors e^{G_r - G_i} are split through anchors so that no factor
// overflows: within each 32-token half the anchor is the half's middle
// (factors <= e^{80} since the log-decay is bounded below by -5), and the
// block (second half x first half) uses anchor G_47 on the row side and
// e^{G_47 - G_i} <= 1 on the column side.  Factors that underflow do so only
// where the exact product is below e^{-7} of its operands... and it is the
// operand itself that vanishes, so the lost terms are negligible.
//
// Precision: every operand is split into bf16 hi + lo parts and products take
// hi.hi + lo.hi + hi.lo, so each contraction is accurate to about 2^-16
// relative; the state stays in fp32 registers.  T is split too: with full-strength
// writes (beta = 1) and no decay, correlated keys make W = T R cancel, and a bf16 T
// alone left about 1e-3 of error in the carried state.
//
// TMEM (512 columns of 128 lanes):
//   [  0,128)  S^T operand (hi 0-63, lo 64-127)  |  dS^T accumulator
//   [128,256)  X1 operand (hi, lo)               |  R^T operand (128-191), W accumulator (192-255)
//   [256,384)  P^T accumulator (256-319), then O^T (320-383)
//   [384,480)  [M;A] accumulator                 |  W^T operand (384-447)
#include <cuda.h>  // CUtensorMap (encoded through the runtime's driver entry point)
#include <cudaTypedefs.h>
#include <string.h>

#include "kda_tc.cuh"
#include "kda_tc_ptx.cuh"

namespace kda {

namespace {

using namespace tc;

constexpr int kD = 128;
constexpr int kC = 64;
constexpr int kThreads = 512;

// TMEM columns
constexpr uint32_t kColS = 0;
constexpr uint32_t kColX = 128;
constexpr uint32_t kColR = 128;
constexpr uint32_t kColW = 192;
constexpr uint32_t kColP = 256;
constexpr uint32_t kColO = 320;
constexpr uint32_t kColAM = 384;
constexpr uint32_t kColWop = 384;
constexpr uint32_t kTmemCols = 512;

// shared memory (bytes from a 1024-aligned base)
constexpr uint32_t kTileB1 = 96 * 256;   // 96 rows x 128 bf16, K-major
constexpr uint32_t kTileB3 = 128 * 256;  // 128 rows x 128 bf16, K-major
constexpr uint32_t kTileKT = 16384;      // 128 (N) x 64 (K) bf16, MN-major
constexpr uint32_t kKtLbo = 8192, kKtSbo = 1024;
constexpr uint32_t kOffB1hi = 0;
constexpr uint32_t kOffB1lo = kOffB1hi + kTileB1;
constexpr uint32_t kOffB3hi = kOffB1lo + kTileB1;
constexpr uint32_t kOffB3lo = kOffB3hi + kTileB3;
constexpr uint32_t kOffKThi = kOffB3lo + kTileB3;
constexpr uint32_t kOffKTlo = kOffKThi + kTileKT;
constexpr int kAs = 68;    // padded row stride of A (floats) in the triangular solve: float4 rows,
constexpr int kTs = 68;    // and of T: conflict-free when 8 lanes read 8 different rows
constexpr uint32_t kOffR1 = kOffKTlo + kTileKT;   // G fp32 (4 swizzled boxes)  |  A fp32 [64][kAs] + T fp32 [64][kTs]
constexpr uint32_t kR1Bytes = 64 * (kAs + kTs) * 4;
static_assert(kR1Bytes >= 4 * 8192, "G exceeds R1");
constexpr uint32_t kOffR2 = kOffR1 + kR1Bytes;     // T hi [64][64] | M hi | M lo | T lo (K-major, 8 KB each)
static_assert(kOffR2 % 1024 == 0, "R2 holds 128-byte-swizzled operand tiles");
constexpr int kKnS = 132;  // row stride (floats) of the normalized k rows parked in R2 during A3b
constexpr uint32_t kR2Bytes = 64 * kKnS * 4;       // 33792 >= 4 x 8 KB
constexpr uint32_t kOffTlo = 24576;                // T lo tile inside R2
static_assert(kOffTlo + 8192 <= kR2Bytes && kOffTlo % 1024 == 0, "T lo tile exceeds R2");
constexpr uint32_t kOffMisc = kOffR2 + kR2Bytes;
// Raw-row staging in operand regions while they are not operands, by 2D TMA boxes with the
// 128-byte swizzle (a box row is 128 bytes; its 16-byte chunk j sits at chunk j ^ (row & 7),
// so one-row-per-lane reads of the same columns are conflict-free):
//   B3 region, from G3's completion in chunk n-1 to A3a of chunk n: q and k rows t0-3 .. t0+63
//     (two 64-column boxes of 67 rows each, 9 KB apart)
//   B1 region, from G1's completion to the epilogue: v rows t0-3 .. t0+63 (same shape), gate
//     rows t0 .. t0+63 (two 64-column boxes of 64 rows, 8 KB apart)
//   R1, from E of chunk n-1 to the end of A3b of chunk n: g rows t0 .. t0+63 (four 32-column
//     fp32 boxes of 64 rows, 8 KB apart), scanned in place into G
//   K~ region, after G6: the y tile of the epilogue
constexpr int kRawRows = kC + 3;
constexpr uint32_t kRawBox = 9216;    // 67 rows x 128 bytes, rounded up to the 1024-byte swizzle period
constexpr uint32_t kGateBox = 8192;   // 64 rows x 128 bytes
constexpr uint32_t kGBox = 8192;      // 64 rows x 32 fp32
constexpr uint32_t kOffRawQ = kOffB3hi;
constexpr uint32_t kOffRawK = kOffB3hi + 2 * kRawBox;
constexpr uint32_t kOffRawV = kOffB1hi;
constexpr uint32_t kOffGateT = kOffB1hi + 2 * kRawBox;
constexpr uint32_t kOffYT = kOffKThi;              // [64][128] y tile (bf16 or fp32)
static_assert(kRawRows * 128 <= kRawBox, "raw box exceeds its slot");
static_assert(kOffRawK + 2 * kRawBox <= kOffKThi, "q/k staging exceeds the B3 region");
static_assert(kOffGateT + 2 * kGateBox <= kOffB3hi, "gate staging exceeds the B1 region");
static_assert(kOffYT + 64 * 128 * 4 <= kOffR1, "y tile exceeds the K~ region");
static_assert(kOffRawQ % 1024 == 0 && kOffRawK % 1024 == 0 && kOffRawV % 1024 == 0 && kOffGateT % 1024 == 0 &&
                  kOffR1 % 1024 == 0 && kRawBox % 1024 == 0,
              "swizzled TMA boxes start on 1024-byte boundaries");
// Byte offsets inside the staged boxes: bf16 element c of raw row rr (64-column boxes of
// box_bytes), and fp32 element c of g / G row rr (32-column boxes).
__device__ __forceinline__ uint32_t swz128(int rr, int chunk) {
    return (uint32_t)(rr * 128 + ((chunk ^ (rr & 7)) << 4));
}
__device__ __forceinline__ uint32_t raw_off(uint32_t box_bytes, int rr, int c) {
    return (uint32_t)(c >> 6) * box_bytes + swz128(rr, (c & 63) >> 3) + (uint32_t)(c & 7) * 2u;
}
__device__ __forceinline__ uint32_t g_off(int rr, int c) {
    return (uint32_t)(c >> 5) * kGBox + swz128(rr, (c & 31) >> 2) + (uint32_t)(c & 3) * 4u;
}

// Tensor maps of the staged inputs: [T rows][H * 128 columns], 128-byte swizzle, boxes as above.
struct TmaMaps {
    CUtensorMap q, k, v, gate, g;
};
__device__ __forceinline__ void prefetch_map(const CUtensorMap* map) {
    asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(map)) : "memory");
}
__device__ __forceinline__ void tma_load_2d(uint32_t dst, const CUtensorMap* map, int x, int y, uint64_t* bar) {
    asm volatile(
        "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes [%0], [%1, {%2, %3}], [%4];" ::
            "r"(dst), "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y), "r"(smem_u32(bar))
        : "memory");
}

// misc (floats)
constexpr int kMiscConvW = 0;                  // [3][128][4]
constexpr int kMiscConst = kMiscConvW + 1536;  // [9][128]
constexpr int kMiscBeta = kMiscConst + 9 * 128;
constexpr int kMiscSS = kMiscBeta + 64;        // [128 rows][4 quarters]
constexpr int kMiscRed = kMiscSS + 512;        // [64 tokens][4 quadrants]
constexpr int kMiscInv = kMiscRed + 256;       // [64] (spare)
constexpr int kMiscFloats = kMiscInv + 64;
constexpr uint32_t kSmemBytes = kOffMisc + kMiscFloats * 4 + 1024;  // + alignment slack
static_assert(kSmemBytes <= 232448 - 1024, "shared memory above the per-block limit");

// per-channel constants, rows of sConst
enum { cA0 = 0, cA1, cE0, cE1, cC2, cC3, cKt0, cKt1, cGam };


// 4 bytes, of which the first src_bytes come from global memory and the rest are zero
__device__ __forceinline__ void cp_async4_zfill(uint32_t dst, const void* src, uint32_t src_bytes) {
    asm volatile("cp.async.ca.shared.global [%0], [%1], 4, %2;" ::"r"(dst), "l"(src), "r"(src_bytes) : "memory");
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }
__device__ __forceinline__ void cp_async_wait_all() { asm volatile("cp.async.wait_group 0;" ::: "memory"); }

__device__ __forceinline__ void prefetch_line_l2(const void* p) {
    asm volatile("prefetch.global.L2 [%0];" ::"l"(p) : "memory");
}

// hi/lo bf16 split of a pair of floats, packed as bf16x2 words (first value in the low half)
__device__ __forceinline__ void split2p(f2 v, uint32_t& hi, uint32_t& lo) {
    hi = pack_bf16x2(f2_lo(v), f2_hi(v));
    const f2 r = sub2(v, f2_of(__uint_as_float(hi << 16), __uint_as_float(hi & 0xffff0000u)));
    lo = pack_bf16x2(f2_lo(r), f2_hi(r));
}
__device__ __forceinline__ void split2(float a, float b, uint32_t& hi, uint32_t& lo) { split2p(f2_of(a, b), hi, lo); }

// 8 floats -> hi and lo 16-byte chunks
__device__ __forceinline__ void split8(const float v[8], uint4& hi, uint4& lo) {
    split2(v[0], v[1], hi.x, lo.x);
    split2(v[2], v[3], hi.y, lo.y);
    split2(v[4], v[5], hi.z, lo.z);
    split2(v[6], v[7], hi.w, lo.w);
}
__device__ __forceinline__ void split8(const f2 v[4], uint4& hi, uint4& lo) {
    split2p(v[0], hi.x, lo.x);
    split2p(v[1], hi.y, lo.y);
    split2p(v[2], hi.z, lo.z);
    split2p(v[3], hi.w, lo.w);
}
// 8 consecutive floats of shared memory (16-byte aligned) as four pairs
__device__ __forceinline__ void ld_f2x4(const float* p, f2 (&d)[4]) {
    const float4 a = reinterpret_cast<const float4*>(p)[0];
    const float4 b = reinterpret_cast<const float4*>(p)[1];
    d[0] = f2_of(a.x, a.y);
    d[1] = f2_of(a.z, a.w);
    d[2] = f2_of(b.x, b.y);
    d[3] = f2_of(b.z, b.w);
}

// Waits for an MMA group's mbarrier and synchronises the CTA; true if the wait timed out.
// Only the polling warp (the one that issued the group) spins on the mbarrier: every warp
// spinning floods the shared-memory pipe the issuing thread needs.  The others sleep in the
// barrier, which also carries the outcome to every thread.
__device__ __forceinline__ bool wait_mma(uint64_t* bar, uint32_t parity, bool poller) {
    bool ok = true;
    if (poller) ok = mbar_wait(bar, parity);
    return __syncthreads_or(!ok) != 0;
}

// The triangular solve runs on warps 0..kSolveWarps-1 with their own named barrier (1);
// barrier 0 is __syncthreads.
constexpr int kSolveWarps = 6;
// Barrier of warps kSolveWarps..15 (named barrier 2), the warps that form R meanwhile.
__device__ __forceinline__ void d_sync() {
    asm volatile("bar.sync 2, %0;" ::"n"(kThreads - 32 * kSolveWarps) : "memory");
}
// Pair barriers of the operand phase (named barriers 4..11): in pair p = qt + 4 (qd & 1),
// k-row warp 4 qt + 2 + (qd & 1) arrives once its normalized k rows are in shared memory and
// q-row warp 4 qt + (qd & 1) waits for them.
__device__ __forceinline__ void pair_arrive(int p) { asm volatile("bar.arrive %0, 64;" ::"r"(4 + p) : "memory"); }
__device__ __forceinline__ void pair_sync(int p) { asm volatile("bar.sync %0, 64;" ::"r"(4 + p) : "memory"); }

// Barrier of the four warps 4 qt .. 4 qt + 3 of one token quarter (named barriers 12..15):
// the RMSNorm partial sums of the epilogue.
__device__ __forceinline__ void quarter_sync(int qt) { asm volatile("bar.sync %0, 128;" ::"r"(12 + qt) : "memory"); }

// Warps 8-15 (named barrier 1, which the solve uses in another phase): the log-decay scan
// that overlaps G5/G6.
__device__ __forceinline__ void scan_sync() { asm volatile("bar.sync 1, 256;" ::: "memory"); }
__device__ __forceinline__ void scan_arrive() { asm volatile("bar.arrive 1, 256;" ::: "memory"); }

// Barrier of warps 0-3 only (named barrier 3): the last two levels of the solve.
__device__ __forceinline__ void solver4_sync() { asm volatile("bar.sync 3, 128;" ::: "memory"); }
__device__ __forceinline__ void solver_sync() { asm volatile("bar.sync 1, %0;" ::"n"(32 * kSolveWarps) : "memory"); }

__device__ __forceinline__ void sts128(uint8_t* base, uint32_t off, const uint4& v) {
    *reinterpret_cast<uint4*>(base + off) = v;
}

template <typename To>
__global__ void __launch_bounds__(kThreads, 1)
k_tc_prefill(const bf16* __restrict__ q, const bf16* __restrict__ k, const bf16* __restrict__ v,
             int64_t xs, const float* __restrict__ conv_w, const bf16* __restrict__ cs_in,
             const float* __restrict__ g, const float* __restrict__ beta,
             const bf16* __restrict__ gate, const float* __restrict__ rms_w, float eps_l2,
             float eps_rms, float scale, const float* __restrict__ S0, float* __restrict__ S_fin,
             To* __restrict__ out, const int32_t* __restrict__ cu, int64_t T_total, int H,
             int* d_status, SegPlan sp, const __grid_constant__ TmaMaps maps, int flags) {
    extern __shared__ uint8_t smem_raw[];
    // G1 done, G3 done, G4 done, G5+G6 done; staged rows landed: g (next chunk), q/k (next
    // chunk), v/gate (this chunk)
    __shared__ uint64_t bars[7];
    __shared__ uint32_t s_tbase;
    __shared__ int s_dfail;  // set by warp 15 when it has waited for G3

    const uint32_t raw_addr = smem_u32(smem_raw);
    uint8_t* sm = smem_raw + (((raw_addr + 1023u) & ~1023u) - raw_addr);
    const uint32_t sbase = smem_u32(sm);
    // G element (row rr, channel c) in the swizzled g boxes of R1
    auto sGat = [&](int rr, int c) -> float& { return *reinterpret_cast<float*>(sm + kOffR1 + g_off(rr, c)); };
    float* sAf = reinterpret_cast<float*>(sm + kOffR1);                 // [64][kAs]
    float* sTf = reinterpret_cast<float*>(sm + kOffR1 + 64 * kAs * 4);  // [64][kTs]
    uint8_t* sTbf = sm + kOffR2;
    uint8_t* sMhi = sm + kOffR2 + 8192;
    uint8_t* sMlo = sm + kOffR2 + 16384;
    float* misc = reinterpret_cast<float*>(sm + kOffMisc);
    float* sConvW = misc + kMiscConvW;
    float* sConst = misc + kMiscConst;
    float* sBeta = misc + kMiscBeta;
    float* sSS = misc + kMiscSS;    // [128 rows][4 quarters]; also [4 quarters][128] column totals
    float* sRed = misc + kMiscRed;

    // Thread layout: 16 warps.  Warp w reaches TMEM lanes 32 (w % 4) .. + 31 (quadrant qd) and
    // owns quarter qt = w / 4 of the channels (64 rows x 128 channels tiles) or of the tokens.
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int qd = warp & 3, qt = warp >> 2;
    const int L = qd * 32 + lane;                 // this thread's TMEM lane
    const uint32_t lane_off = (uint32_t)(qd * 32) << 16;
    // role of this CTA (the grid holds units * (2P - 1) CTAs)
    const int units = (int)(gridDim.x / (2 * sp.P - 1));
    const int role = (int)(blockIdx.x / units), u = (int)(blockIdx.x % units);
    const int h = u % H, n = u / H;
    const int seg = (role + 1) >> 1;
    const bool zero_run = (role & 1) != 0;           // segment >= 1 from S = 0
    const bool ident_run = role > 0 && !zero_run;    // segment >= 1 from S = I with v = 0
    const bool raw_out = role > 0;                   // fp32 scale * o, no epilogue
    const bf16* __restrict__ gate_p = raw_out ? nullptr : gate;
    const int64_t HD = (int64_t)H * kD;
    int64_t s0, s1;
    seq_range(cu, n, T_total, s0, s1);
    int64_t cb, ce;  // this CTA's chunks [cb, ce) of the sequence
    seg_chunk_range((s1 - s0 + kC - 1) / kC, sp.P, sp.w, sp.wd, seg, cb, ce);

    if (warp == 0) {
        tmem_alloc(&s_tbase, kTmemCols);
        tmem_relinquish();
    }
    if (tid == 0) {
        for (int i = 0; i < 7; ++i) mbar_init(&bars[i], 1);
        fence_mbar_init();
        s_dfail = 0;
    }
    for (int idx = tid; idx < 3 * kD * 4; idx += kThreads) {  // [part][tap][channel]
        const int part = idx / (kD * 4), tap = (idx / kD) & 3, c = idx % kD;
        sConvW[idx] = conv_w[(part * HD + (int64_t)h * kD + c) * 4 + tap];
    }
    fence_before_sync();
    __syncthreads();
    fence_after_sync();
    const uint32_t tb = s_tbase;

    // ---- carried state: thread (lane j = L, quarter qt) keeps S[c][j] for c in [32qt, 32qt + 32)
    const int j = L;
    float Sreg[32];
    {
        const float* src = (role == 0 && S0) ? S0 + (((int64_t)n * H + h) * kD) * kD : nullptr;
#pragma unroll
        for (int i = 0; i < 32; ++i)
            Sreg[i] = src ? src[(int64_t)(32 * qt + i) * kD + j] : (ident_run && 32 * qt + i == j ? 1.f : 0.f);
    }
    auto store_state_operand = [&]() {  // S^T hi/lo -> TMEM columns [0,128)
        uint32_t hi[16], lo[16];
#pragma unroll
        for (int i = 0; i < 16; ++i) split2(Sreg[2 * i], Sreg[2 * i + 1], hi[i], lo[i]);
        tmem_st16(tb + lane_off + kColS + 16 * qt, hi);
        tmem_st16(tb + lane_off + kColS + 64 + 16 * qt, lo);
        tmem_st_wait();
    };
    store_state_operand();

    const uint32_t id_g1 = idesc_bf16(128, 96, false, false);
    const uint32_t id_g3 = idesc_bf16(128, 128, false, false);
    const uint32_t id_64 = idesc_bf16(128, 64, false, false);
    const uint32_t id_g6 = idesc_bf16(128, 128, false, true);
    bool failed = false;

    // Row staging by the TMA engine: one warp issues 1D bulk copies of whole rows (256 bytes of
    // bf16, 512 of fp32) and lane 0 arms the completion mbarrier for their bytes.  The rows of
    // chunk cj complete phase (cj - cb) of their barrier (bars[4] g, bars[5] q/k, bars[6]
    // v/gate), so every wait takes parity (cj - cb) & 1.  `pend` (uniform over the CTA) keeps,
    // per barrier i, bit 2i = a completion in flight and bit 2i+1 = its parity, for the exit path.
    uint32_t pend = 0;
    auto pend_set = [&](int i, int64_t cj) { pend |= (1u | ((uint32_t)((cj - cb) & 1) << 1)) << (2 * i); };
    auto pend_clear = [&](int i) { pend &= ~(3u << (2 * i)); };
    // q/k rows t0-3 .. t0+63 of chunk cj -> B3 region, four boxes from thread 32 wq (rows
    // outside the tensor read as zero; rows of a neighbouring sequence are never used)
    auto stage_qk = [&](int64_t cj, int wq) {
        if (cj == cb && (flags & KDA_FLAG_TEST_DROP_STAGING)) return;  // test only: never arrives
        if (tid == 32 * wq) {
            const int y = (int)(s0 + (int64_t)cj * kC - 3), x = h * kD;
            mbar_expect_tx(&bars[5], 4 * kRawRows * 128);
            tma_load_2d(sbase + kOffRawQ, &maps.q, x, y, &bars[5]);
            tma_load_2d(sbase + kOffRawQ + kRawBox, &maps.q, x + 64, y, &bars[5]);
            tma_load_2d(sbase + kOffRawK, &maps.k, x, y, &bars[5]);
            tma_load_2d(sbase + kOffRawK + kRawBox, &maps.k, x + 64, y, &bars[5]);
        }
        pend_set(1, cj);
    };
    // g rows of chunk cj -> R1, four boxes from thread 32 wq (bars[4]); its beta -> sBeta by
    // cp.async of threads 64 wq .. 64 wq + 63 (zeros past the sequence end).  Issued early, so
    // that the scan below finds the rows in shared memory.
    auto stage_G = [&](int64_t cj, int wq) {
        const int64_t tc0 = s0 + (int64_t)cj * kC;
        const int Lcj = (int)((s1 - tc0) < kC ? (s1 - tc0) : kC);
        if (tid == 32 * wq) {
            mbar_expect_tx(&bars[4], 4 * kGBox);
#pragma unroll
            for (int b4 = 0; b4 < 4; ++b4)
                tma_load_2d(sbase + kOffR1 + b4 * kGBox, &maps.g, h * kD + 32 * b4, (int)tc0, &bars[4]);
        }
        const int rb = tid - 64 * wq;
        if (rb >= 0 && rb < kC) {
            const bool ok = rb < Lcj;
            cp_async4_zfill(sbase + kOffMisc + (uint32_t)(kMiscBeta + rb) * 4u, ok ? beta + (tc0 + rb) * H + h : beta,
                            ok ? 4u : 0u);
        }
        cp_async_commit();
        pend_set(0, cj);
    };
    // Waits for stage_G(cj)'s rows (poller warp wq) and beta copies; false if the wait timed out.
    auto wait_G = [&](int64_t cj, int wq) -> bool {
        bool ok = true;
        if (warp == wq) ok = mbar_wait(&bars[4], (uint32_t)((cj - cb) & 1));
        pend_clear(0);
        cp_async_wait_all();
        return __syncthreads_or(!ok) == 0;
    };
    // G = cumsum(g log2 e) down each channel of the staged rows of chunk cj (four quarters of
    // 16 tokens; rows past the sequence end count as zero), in place; the caller has waited for
    // the rows.  One barrier inside.
    auto scan_G = [&](int64_t cj) {
        const int64_t tc0 = s0 + (int64_t)cj * kC;
        const int Lcj = (int)((s1 - tc0) < kC ? (s1 - tc0) : kC);
        const int c = tid & (kD - 1), hq = tid >> 7;
        float gv[16];
#pragma unroll
        for (int e = 0; e < 16; ++e) gv[e] = 16 * hq + e < Lcj ? sGat(16 * hq + e, c) * kLog2e : 0.f;  // base 2
        float acc = 0.f;
#pragma unroll
        for (int e = 0; e < 16; ++e) {
            acc += gv[e];
            gv[e] = acc;
        }
        sSS[hq * kD + c] = acc;  // quarter total per channel
        __syncthreads();
        float base = 0.f;
        for (int qq = 0; qq < hq; ++qq) base += sSS[qq * kD + c];
#pragma unroll
        for (int e = 0; e < 16; ++e) sGat(16 * hq + e, c) = gv[e] + base;
    };
    // The same scan on warps 8-15 alone, while thread 0 issues G5/G6: thread (channel c, half
    // h2) sums rows 32 h2 .. 32 h2 + 31; the first half passes its total on named barrier 1
    // (free in this phase of the chunk).
    auto scan_G_half = [&](int64_t cj) {
        const int64_t tc0 = s0 + (int64_t)cj * kC;
        const int Lcj = (int)((s1 - tc0) < kC ? (s1 - tc0) : kC);
        const int c = tid & (kD - 1), h2 = (tid >> 7) & 1, r0 = 32 * h2;
        float gv[32];
        float acc = 0.f;
#pragma unroll
        for (int e = 0; e < 32; ++e) {
            acc += r0 + e < Lcj ? sGat(r0 + e, c) * kLog2e : 0.f;  // base 2
            gv[e] = acc;
        }
        if (h2 == 0) {
            sSS[c] = acc;
            scan_arrive();
#pragma unroll
            for (int e = 0; e < 32; ++e) sGat(e, c) = gv[e];
        } else {
            scan_sync();
            const float base = sSS[c];
#pragma unroll
            for (int e = 0; e < 32; ++e) sGat(32 + e, c) = gv[e] + base;
        }
    };
    if (cb < ce) {
        if (tid == 0) {  // descriptors into the TMA unit's cache ahead of their first use
            prefetch_map(&maps.q);
            prefetch_map(&maps.k);
            prefetch_map(&maps.g);
            if (!ident_run) prefetch_map(&maps.v);
            if (gate_p) prefetch_map(&maps.gate);
        }
        stage_qk(cb, 2);
        stage_G(cb, 1);
        failed = !wait_G(cb, 1);
        if (!failed) scan_G(cb);
    }

    for (int64_t ci = cb; ci < ce && !failed; ++ci) {
        const int64_t t0 = s0 + ci * kC;
        const int Lc = (int)((s1 - t0) < kC ? (s1 - t0) : kC);
        const uint32_t par = (uint32_t)(ci - cb) & 1u;

        // ------------------------------------------------ A0: L2 prefetch of the next chunk's rows
        if (ci + 1 < ce) {
            // next chunk's rows into L2, one 128-byte line per thread and step
            const int64_t tn = t0 + kC;
            const int rr = tid & 63, which = tid >> 6;  // 8 line slots per row
            if (tn + rr < s1) {
                const int64_t row = tn + rr;
                const char* base;
                if (which < 2) base = reinterpret_cast<const char*>(q + row * xs + (int64_t)h * kD) + 128 * which;
                else if (which < 4) base = reinterpret_cast<const char*>(k + row * xs + (int64_t)h * kD) + 128 * (which - 2);
                else if (which < 6) base = ident_run ? nullptr : reinterpret_cast<const char*>(v + row * xs + (int64_t)h * kD) + 128 * (which - 4);
                else base = reinterpret_cast<const char*>(g + (row * H + h) * kD) + 256 * (which - 6);
                if (base) prefetch_line_l2(base);
                if (which >= 6) prefetch_line_l2(base + 128);
                if (gate_p && which < 2) prefetch_line_l2(reinterpret_cast<const char*>(gate_p + (row * H + h) * kD) + 128 * which);
            }
        }

        // q/k rows and G of this chunk were prepared during the previous chunk (or before the loop)
        {
            bool ok = true;
            if (warp == 0) ok = mbar_wait(&bars[5], par);
            pend_clear(1);
            failed = __syncthreads_or(!ok) != 0;
            if (failed) break;
        }

        // ------------------------------------------------ A2: per-channel anchors and factors
        if (tid < kD) {
            const int c = tid;
            const float a0 = sGat(15, c), a1 = sGat(47, c), g31 = sGat(31, c), gl = sGat(63, c);
            sConst[cA0 * kD + c] = a0;
            sConst[cA1 * kD + c] = a1;
            sConst[cE0 * kD + c] = exp2_hw(a0);
            sConst[cE1 * kD + c] = exp2_hw(a1);
            sConst[cC2 * kD + c] = exp2_hw(g31 - a0);
            sConst[cC3 * kD + c] = exp2_hw(a1 - g31);
            sConst[cKt0 * kD + c] = exp2_hw(gl - g31);
            sConst[cKt1 * kD + c] = exp2_hw(gl - a1);
            sConst[cGam * kD + c] = exp2_hw(gl);
        }

        // ------------------------------------------------ A3a: conv + SiLU of one q or k row (32 channels)
        const bool isq = L < 64;
        const int r = L & 63;
        const bool rvalid = r < Lc;
        const int c0 = 32 * qt;
        float x[32];
        {
            const int part = isq ? 0 : 1;
            const int64_t t = t0 + r;
            f2 ss2 = f2_dup(0.f);
#pragma unroll
            for (int g8 = 0; g8 < 4; ++g8) {
                const int cc = c0 + 8 * g8;
                float win[4][8];
#pragma unroll
                for (int m = 0; m < 4; ++m) {
                    const int64_t p = t - 3 + m;
                    if (!rvalid) {
#pragma unroll
                        for (int e = 0; e < 8; ++e) win[m][e] = 0.f;
                    } else if (p >= s0) {
                        load8(reinterpret_cast<const bf16*>(sm + (isq ? kOffRawQ : kOffRawK) +
                                                            raw_off(kRawBox, (int)(p - (t0 - 3)), cc)),
                              win[m]);
                    } else {
                        const int pos = (int)(p - s0);  // -3..-1
#pragma unroll
                        for (int e = 0; e < 8; ++e)
                            win[m][e] = cs_in ? to_f(cs_in[((int64_t)n * 3 * HD + part * HD + (int64_t)h * kD + cc + e) * 3 + 3 + pos]) : 0.f;
                    }
                }
                // channel pairs in packed fp32 (an invalid row has a zero window: silu(0) = 0)
                f2 u2[4];
#pragma unroll
                for (int m = 0; m < 4; ++m) {
                    const float4 wa = *reinterpret_cast<const float4*>(&sConvW[(part * 4 + m) * kD + cc]);
                    const float4 wb = *reinterpret_cast<const float4*>(&sConvW[(part * 4 + m) * kD + cc + 4]);
                    const f2 w2[4] = {f2_of(wa.x, wa.y), f2_of(wa.z, wa.w), f2_of(wb.x, wb.y), f2_of(wb.z, wb.w)};
#pragma unroll
                    for (int pp = 0; pp < 4; ++pp) {
                        const f2 xw = f2_of(win[m][2 * pp], win[m][2 * pp + 1]);
                        u2[pp] = m == 0 ? mul2(w2[pp], xw) : fma2(w2[pp], xw, u2[pp]);
                    }
                }
#pragma unroll
                for (int pp = 0; pp < 4; ++pp) {  // silu(u) = h + h tanh(h), h = u / 2
                    const f2 hx = mul2(u2[pp], f2_dup(0.5f));
                    const f2 sv = fma2(hx, f2_of(tanh_hw(f2_lo(hx)), tanh_hw(f2_hi(hx))), hx);
                    x[8 * g8 + 2 * pp] = f2_lo(sv);
                    x[8 * g8 + 2 * pp + 1] = f2_hi(sv);
                    ss2 = fma2(sv, sv, ss2);
                }
            }
            sSS[L * 4 + qt] = f2_lo(ss2) + f2_hi(ss2);
        }
        __syncthreads();

        // ------------------------------------------------ A3b: L2 norm, decay factors, operand tiles
        {
            const float4 ssv = *reinterpret_cast<const float4*>(&sSS[L * 4]);
            // rows past the sequence end are zero: give them a zero factor, not 0 * rsqrt(0 + eps)
            // (which is NaN when eps_l2 = 0 and would reach every token through the MMAs)
            const float inv = rvalid ? rsqrtf(ssv.x + ssv.y + ssv.z + ssv.w + eps_l2) : 0.f;
            const int hr = r >> 5;
            const float* cA = sConst + (hr ? cA1 : cA0) * kD;
            const float* cE = sConst + (hr ? cE1 : cE0) * kD;
            const float bt = sBeta[r];
            {  // normalize the row in place
                const f2 inv2 = f2_dup(inv);
#pragma unroll
                for (int i = 0; i < 16; ++i) {
                    const f2 y = mul2(f2_of(x[2 * i], x[2 * i + 1]), inv2);
                    x[2 * i] = f2_lo(y);
                    x[2 * i + 1] = f2_hi(y);
                }
            }
            // Load balance: the k rows also build B1 and K~, so their B3 rows (k e^{G_r}) are
            // built by the q-row warps of the same tokens, which hold the same decay factors:
            // the k-row warp leaves its normalized k in R2 (free until C) and arrives on the
            // pair's named barrier, the q-row warp waits on it.
            float* sKn = reinterpret_cast<float*>(sm + kOffR2);  // [64][kKnS] normalized k rows
            const int pair = qt + 4 * (qd & 1);  // quadrants 0 + 2 and 1 + 3, per channel quarter
            if (!isq) {
#pragma unroll
                for (int g8 = 0; g8 < 8; ++g8)
                    *reinterpret_cast<float4*>(&sKn[r * kKnS + c0 + 4 * g8]) =
                        make_float4(x[4 * g8], x[4 * g8 + 1], x[4 * g8 + 2], x[4 * g8 + 3]);
                pair_arrive(pair);
            } else {
                pair_sync(pair);
            }
            // X1 row: each 8-channel group goes to TMEM as soon as it is formed (columns
            // kColX + 16 qt + 4 g8 hi, + 64 lo), so the 64 KB of operand stores drain while the
            // other tiles are built instead of in front of the G1 issue.  Channel pairs in
            // packed fp32; log-decay sums in base 2.
#pragma unroll
            for (int g8 = 0; g8 < 4; ++g8) {
                const int cc = c0 + 8 * g8;
                f2 xv[4], dg[4], uu[4], EE[4];
                {
                    f2 gg[4], aa[4];
                    {  // G row r, columns cc .. cc + 7: two swizzled 16-byte chunks
                        const float4 g0 = *reinterpret_cast<const float4*>(sm + kOffR1 + g_off(r, cc));
                        const float4 g1 = *reinterpret_cast<const float4*>(sm + kOffR1 + g_off(r, cc + 4));
                        gg[0] = f2_of(g0.x, g0.y);
                        gg[1] = f2_of(g0.z, g0.w);
                        gg[2] = f2_of(g1.x, g1.y);
                        gg[3] = f2_of(g1.z, g1.w);
                    }
                    ld_f2x4(&cA[cc], aa);
                    ld_f2x4(&cE[cc], EE);
#pragma unroll
                    for (int pp = 0; pp < 4; ++pp) {
                        xv[pp] = f2_of(x[8 * g8 + 2 * pp], x[8 * g8 + 2 * pp + 1]);
                        dg[pp] = sub2(gg[pp], aa[pp]);  // G_r - G_anchor
                        uu[pp] = f2_of(exp2_hw(f2_lo(dg[pp])), exp2_hw(f2_hi(dg[pp])));
                    }
                }
                f2 t8[4];
                uint4 hi, lo;
                if (isq) {
                    // X1 row: q u ; QG row (B3 row 64 + r): q u E_h = q e^{G_r}
#pragma unroll
                    for (int pp = 0; pp < 4; ++pp) t8[pp] = mul2(xv[pp], uu[pp]);
                    split8(t8, hi, lo);
                    tmem_st4(tb + lane_off + kColX + 16 * qt + 4 * g8, hi);
                    tmem_st4(tb + lane_off + kColX + 64 + 16 * qt + 4 * g8, lo);
                    f2 ue[4];
#pragma unroll
                    for (int pp = 0; pp < 4; ++pp) {
                        ue[pp] = mul2(uu[pp], EE[pp]);
                        t8[pp] = mul2(xv[pp], ue[pp]);
                    }
                    split8(t8, hi, lo);
                    sts128(sm, kOffB3hi + kmajor_off(128, 64 + r, cc / 8), hi);
                    sts128(sm, kOffB3lo + kmajor_off(128, 64 + r, cc / 8), lo);
                    {
                        // KG row of k row r (B3 row r), for the k-row warp of the pair
                        f2 kn[4];
                        ld_f2x4(&sKn[r * kKnS + cc], kn);
#pragma unroll
                        for (int pp = 0; pp < 4; ++pp) t8[pp] = mul2(kn[pp], ue[pp]);
                        split8(t8, hi, lo);
                        sts128(sm, kOffB3hi + kmajor_off(128, r, cc / 8), hi);
                        sts128(sm, kOffB3lo + kmajor_off(128, r, cc / 8), lo);
                    }
                } else {
                    f2 kv[4];
                    const f2 bt2 = f2_dup(bt);
#pragma unroll
                    for (int pp = 0; pp < 4; ++pp) {
                        // X1 row: beta k u ; B1 row r: k v, v = e^{G_anchor - G_r}
                        t8[pp] = mul2(mul2(bt2, xv[pp]), uu[pp]);
                        kv[pp] = mul2(xv[pp], f2_of(exp2_hw(-f2_lo(dg[pp])), exp2_hw(-f2_hi(dg[pp]))));
                    }
                    split8(t8, hi, lo);
                    tmem_st4(tb + lane_off + kColX + 16 * qt + 4 * g8, hi);
                    tmem_st4(tb + lane_off + kColX + 64 + 16 * qt + 4 * g8, lo);
                    split8(kv, hi, lo);
                    sts128(sm, kOffB1hi + kmajor_off(96, r, cc / 8), hi);
                    sts128(sm, kOffB1lo + kmajor_off(96, r, cc / 8), lo);
                    // (B3 row r, k u E_h = k e^{G_r}, is built by the q-row warp of the pair)
                    f2 cst[4];
                    if (r < 32) {
                        // B1 row 64 + r: k e^{G_47 - G_r} = k v c2 c3 ; Kt row r: k v c2 e^{G_last - G_31}
                        f2 w8[4];
                        ld_f2x4(&sConst[cC2 * kD + cc], cst);
#pragma unroll
                        for (int pp = 0; pp < 4; ++pp) w8[pp] = mul2(kv[pp], cst[pp]);
                        ld_f2x4(&sConst[cC3 * kD + cc], cst);
#pragma unroll
                        for (int pp = 0; pp < 4; ++pp) t8[pp] = mul2(w8[pp], cst[pp]);
                        split8(t8, hi, lo);
                        sts128(sm, kOffB1hi + kmajor_off(96, 64 + r, cc / 8), hi);
                        sts128(sm, kOffB1lo + kmajor_off(96, 64 + r, cc / 8), lo);
                        ld_f2x4(&sConst[cKt0 * kD + cc], cst);
#pragma unroll
                        for (int pp = 0; pp < 4; ++pp) t8[pp] = mul2(w8[pp], cst[pp]);
                    } else {
                        // Kt row r: k v e^{G_last - G_47}
                        ld_f2x4(&sConst[cKt1 * kD + cc], cst);
#pragma unroll
                        for (int pp = 0; pp < 4; ++pp) t8[pp] = mul2(kv[pp], cst[pp]);
                    }
                    split8(t8, hi, lo);
                    sts128(sm, kOffKThi + mnmajor_off(kKtLbo, kKtSbo, cc / 8, r), hi);
                    sts128(sm, kOffKTlo + mnmajor_off(kKtLbo, kKtSbo, cc / 8, r), lo);
                }
            }
            tmem_st_wait();
        }
        fence_async_smem();
        fence_before_sync();
        __syncthreads();

        // ------------------------------------------------ B: issue G1 ([M;A])
        // (G3, the state reads, is issued later by warp 15, which the solve leaves idle: the
        // issuing thread waits while the tensor pipe accepts its MMAs, and G3 is needed only in D)
        if (tid == 0) {
            fence_after_sync();
            const uint32_t b1h = sbase + kOffB1hi, b1l = sbase + kOffB1lo;
#pragma unroll
            for (int term = 0; term < 3; ++term) {
                const uint32_t acol = kColX + (term == 1 ? 64 : 0);
                const uint32_t bt1 = term == 2 ? b1l : b1h;
#pragma unroll
                for (int kk = 0; kk < 8; ++kk)
                    mma_ts(tb + kColAM, tb + acol + 8 * kk,
                           desc_sw128(bt1 + (kk >> 2) * 96 * 128 + (kk & 3) * 32, 16, 1024), id_g1,
                           (term | kk) != 0);
            }
            mma_commit(&bars[0]);
        }

        // ------------------------------------------------ C: M and A from G1, T = (I + A)^-1
        failed = wait_mma(&bars[0], par, warp == 0);
        if (failed) break;
        fence_after_sync();
        // G1 is done with B1: v rows t0-3 .. t0+63 and gate rows t0 .. t0+63 there (boxes from
        // thread 32, bars[6]); the identity-start runs take neither
        const bool vg = !ident_run || gate_p;
        if (vg && tid == 32) {
            const int x = h * kD;
            mbar_expect_tx(&bars[6], (ident_run ? 0u : 2u * kRawRows * 128u) + (gate_p ? 2u * kGateBox : 0u));
            if (!ident_run) {
                tma_load_2d(sbase + kOffRawV, &maps.v, x, (int)(t0 - 3), &bars[6]);
                tma_load_2d(sbase + kOffRawV + kRawBox, &maps.v, x + 64, (int)(t0 - 3), &bars[6]);
            }
            if (gate_p) {
                tma_load_2d(sbase + kOffGateT, &maps.gate, x, (int)t0, &bars[6]);
                tma_load_2d(sbase + kOffGateT + kGateBox, &maps.gate, x + 64, (int)t0, &bars[6]);
            }
        }
        if (vg) pend_set(2, ci);
        {
            // thread: row r (q rows -> M, k rows -> A), columns i in [16qt, 16qt + 16).  The warp's rows
            // share one half hr, so the source block is warp-uniform: same half -> columns i,
            // row half 1 x column half 0 -> columns 64 + i (anchor G_47), otherwise zero.
            const int hr = r >> 5, hi_half = qt >> 1;
            float row[16];
            if (hi_half <= hr) {
                uint32_t dv[16];
                tmem_ld16(tb + lane_off + kColAM + (hi_half == hr ? 16 * qt : 64 + 16 * qt), dv);
                tmem_ld_wait();
#pragma unroll
                for (int e = 0; e < 16; ++e) {
                    const int i = 16 * qt + e;
                    const bool keep = isq ? (i <= r) : (i < r);
                    row[e] = keep ? __uint_as_float(dv[e]) : 0.f;
                }
            } else {
#pragma unroll
                for (int e = 0; e < 16; ++e) row[e] = 0.f;
            }
            if (isq) {
#pragma unroll
                for (int g8 = 0; g8 < 2; ++g8) {
                    uint4 hi, lo;
                    float t8[8];
#pragma unroll
                    for (int e = 0; e < 8; ++e) t8[e] = row[8 * g8 + e];
                    split8(t8, hi, lo);
                    sts128(sMhi, kmajor_off(64, r, 2 * qt + g8), hi);
                    sts128(sMlo, kmajor_off(64, r, 2 * qt + g8), lo);
                }
            } else {
#pragma unroll
                for (int e = 0; e < 16; e += 4)
                    *reinterpret_cast<float4*>(&sAf[r * kAs + 16 * qt + e]) = make_float4(row[e], row[e + 1], row[e + 2], row[e + 3]);
            }
        }
        {  // A and the M tiles are complete; the v / gate rows have landed
            bool ok = true;
            if (vg) {
                if (warp == 1) ok = mbar_wait(&bars[6], par);
                pend_clear(2);
            }
            fence_before_sync();
            failed = __syncthreads_or(!ok) != 0;
            if (failed) break;
        }
        // G3: [P ; Q'] = S^T . [KG ; QG]^T (state reads), from warp 15 while warps 0-5 solve
        if (tid == kThreads - 32) {
            fence_after_sync();
            const uint32_t b3h = sbase + kOffB3hi, b3l = sbase + kOffB3lo;
#pragma unroll
            for (int term = 0; term < 3; ++term) {
                const uint32_t acol = kColS + (term == 1 ? 64 : 0);
                const uint32_t bt3 = term == 2 ? b3l : b3h;
#pragma unroll
                for (int kk = 0; kk < 8; ++kk)
                    mma_ts(tb + kColP, tb + acol + 8 * kk,
                           desc_sw128(bt3 + (kk >> 2) * 128 * 128 + (kk & 3) * 32, 16, 1024), id_g3,
                           (term | kk) != 0);
            }
            mma_commit(&bars[1]);
        }
        // T: unit lower triangular inverse, on named barriers of its own while the other warps
        // form R (D) and warp 15 issues G3: warps 0-5 for the diagonal blocks and the first
        // block level (192 quads of outputs), warps 0-3 for the other two levels (128 and 64
        // quads) and the bf16 copy.  Diagonal 16x16 blocks: one warp per block, lane jj (lanes
        // 16..31 mirror 0..15) keeps column jj of the block in registers.
        float* sX = sSS;  // 3 slots of [16][16] X floats, 768 floats over sSS + sRed
        // Off-diagonal 16-blocks: X_IJ = sum_{K=J}^{I-1} A_IK T_KJ, then T_IJ = -T_II X_IJ.  A
        // thread makes one quad (row rr, columns 4 jq .. 4 jq + 3) of a block; A rows and T rows
        // come as float4 loads, the products in packed pairs on two chains (even / odd k).
        // x_quad adds A_IK T_KJ for K in [K0, K1) to (x01, x23).
        auto x_quad = [&](int I, int J, int K0, int K1, int rr, int jq, f2& x01, f2& x23) {
            f2 a01 = x01, a23 = x23, b01 = f2_dup(0.f), b23 = f2_dup(0.f);
            for (int K = K0; K < K1; ++K) {
#pragma unroll
                for (int m = 0; m < 4; ++m) {
                    const float4 a4 = *reinterpret_cast<const float4*>(&sAf[(16 * I + rr) * kAs + 16 * K + 4 * m]);
                    const float av[4] = {a4.x, a4.y, a4.z, a4.w};
#pragma unroll
                    for (int uu = 0; uu < 4; ++uu) {
                        const float4 t4 =
                            *reinterpret_cast<const float4*>(&sTf[(16 * K + 4 * m + uu) * kTs + 16 * J + 4 * jq]);
                        const f2 aa = f2_dup(av[uu]);
                        if (uu & 1) {
                            b01 = fma2(aa, f2_of(t4.x, t4.y), b01);
                            b23 = fma2(aa, f2_of(t4.z, t4.w), b23);
                        } else {
                            a01 = fma2(aa, f2_of(t4.x, t4.y), a01);
                            a23 = fma2(aa, f2_of(t4.z, t4.w), a23);
                        }
                    }
                }
            }
            x01 = add2(a01, b01);
            x23 = add2(a23, b23);
        };
        // The same for two block rows I1, I2 of one block column J: each T load feeds both.
        auto x_quad2 = [&](int I1, int I2, int J, int K0, int K1, int rr, int jq, f2& x01, f2& x23, f2& y01, f2& y23) {
            for (int K = K0; K < K1; ++K) {
#pragma unroll
                for (int m = 0; m < 4; ++m) {
                    const float4 a4 = *reinterpret_cast<const float4*>(&sAf[(16 * I1 + rr) * kAs + 16 * K + 4 * m]);
                    const float4 b4 = *reinterpret_cast<const float4*>(&sAf[(16 * I2 + rr) * kAs + 16 * K + 4 * m]);
                    const float av[4] = {a4.x, a4.y, a4.z, a4.w}, bv[4] = {b4.x, b4.y, b4.z, b4.w};
#pragma unroll
                    for (int uu = 0; uu < 4; ++uu) {
                        const float4 t4 =
                            *reinterpret_cast<const float4*>(&sTf[(16 * K + 4 * m + uu) * kTs + 16 * J + 4 * jq]);
                        const f2 t01 = f2_of(t4.x, t4.y), t23 = f2_of(t4.z, t4.w);
                        x01 = fma2(f2_dup(av[uu]), t01, x01);
                        x23 = fma2(f2_dup(av[uu]), t23, x23);
                        y01 = fma2(f2_dup(bv[uu]), t01, y01);
                        y23 = fma2(f2_dup(bv[uu]), t23, y23);
                    }
                }
            }
        };
        // X quads live in sX block slot `slot` ([16][16] floats)
        auto x_store = [&](int slot, int rr, int jq, f2 x01, f2 x23) {
            *reinterpret_cast<float4*>(&sX[(slot * 16 + rr) * 16 + 4 * jq]) =
                make_float4(f2_lo(x01), f2_hi(x01), f2_lo(x23), f2_hi(x23));
        };
        // T_IJ quad = -T_II X (X in slot J); T_II is lower triangular with exact zeros above
        auto t_quad = [&](int I, int J, int rr, int jq) {
            f2 a01 = f2_dup(0.f), a23 = f2_dup(0.f), b01 = f2_dup(0.f), b23 = f2_dup(0.f);
#pragma unroll
            for (int m = 0; m < 4; ++m) {
                const float4 t4 = *reinterpret_cast<const float4*>(&sTf[(16 * I + rr) * kTs + 16 * I + 4 * m]);
                const float tv[4] = {t4.x, t4.y, t4.z, t4.w};
#pragma unroll
                for (int uu = 0; uu < 4; ++uu) {
                    const float4 x4 = *reinterpret_cast<const float4*>(&sX[(J * 16 + 4 * m + uu) * 16 + 4 * jq]);
                    const f2 tt = f2_dup(tv[uu]);
                    if (uu & 1) {
                        b01 = fma2(tt, f2_of(x4.x, x4.y), b01);
                        b23 = fma2(tt, f2_of(x4.z, x4.w), b23);
                    } else {
                        a01 = fma2(tt, f2_of(x4.x, x4.y), a01);
                        a23 = fma2(tt, f2_of(x4.z, x4.w), a23);
                    }
                }
            }
            const f2 x01 = add2(a01, b01), x23 = add2(a23, b23);
            *reinterpret_cast<float4*>(&sTf[(16 * I + rr) * kTs + 16 * J + 4 * jq]) =
                make_float4(-f2_lo(x01), -f2_hi(x01), -f2_lo(x23), -f2_hi(x23));
        };
        const int q_rr = (tid >> 2) & 15, q_jq = tid & 3, q_blk = tid >> 6;
        if (warp < kSolveWarps) {
            if (warp < 4) {
                // Diagonal 16-block b0 as 2 x 2 blocks of 8: lanes (sub, c), sub = bit 3 of the
                // lane, invert the 8 x 8 diagonal block sub (lane c keeps column c; row rr
                // subtracts A_rr,ii t_ii for ii < rr on two chains); then the sub = 0 lanes form
                // T_10 = -T_11 (A_10 T_00) from shared memory.  Lanes 16-31 mirror 0-15.
                const int b0 = 16 * warp, sub = (lane >> 3) & 1, c8 = lane & 7, sb = b0 + 8 * sub;
                float t[8];
#pragma unroll
                for (int rr = 0; rr < 8; ++rr) {
                    float c0 = rr == c8 ? 1.f : 0.f, c1 = 0.f;
                    const float* arow = sAf + (sb + rr) * kAs + sb;
#pragma unroll
                    for (int q4 = 0; q4 < (rr + 3) / 4; ++q4) {
                        const float4 a4 = *reinterpret_cast<const float4*>(&arow[4 * q4]);
                        const float av[4] = {a4.x, a4.y, a4.z, a4.w};
#pragma unroll
                        for (int uu = 0; uu < 4; ++uu) {
                            const int ii = 4 * q4 + uu;
                            if (ii < rr) {
                                if (ii & 1) c1 -= av[uu] * t[ii];
                                else c0 -= av[uu] * t[ii];
                            }
                        }
                    }
                    t[rr] = c0 + c1;
                }
                if (lane < 16) {
#pragma unroll
                    for (int rr = 0; rr < 8; ++rr) {
                        sTf[(sb + rr) * kTs + sb + c8] = t[rr];
                        if (sub == 0) sTf[(b0 + rr) * kTs + b0 + 8 + c8] = 0.f;  // above the diagonal
                    }
                }
                __syncwarp();
                if (sub == 0) {
                    // X = A_10 T_00 (column c8 of T_00 is t), then T_10 = -T_11 X
                    float x[8];
#pragma unroll
                    for (int r8 = 0; r8 < 8; ++r8) {
                        const float* arow = sAf + (b0 + 8 + r8) * kAs + b0;
                        const float4 a0 = *reinterpret_cast<const float4*>(arow);
                        const float4 a1 = *reinterpret_cast<const float4*>(arow + 4);
                        x[r8] = a0.x * t[0] + a0.y * t[1] + a0.z * t[2] + a0.w * t[3] +
                                (a1.x * t[4] + a1.y * t[5] + a1.z * t[6] + a1.w * t[7]);
                    }
#pragma unroll
                    for (int r8 = 0; r8 < 8; ++r8) {
                        const float* trow = sTf + (b0 + 8 + r8) * kTs + b0 + 8;
                        const float4 u0 = *reinterpret_cast<const float4*>(trow);
                        const float4 u1 = *reinterpret_cast<const float4*>(trow + 4);
                        const float v = u0.x * x[0] + u0.y * x[1] + u0.z * x[2] + u0.w * x[3] +
                                        (u1.x * x[4] + u1.y * x[5] + u1.z * x[6] + u1.w * x[7]);
                        if (lane < 16) sTf[(b0 + 8 + r8) * kTs + b0 + c8] = -v;
                    }
                }
            }
            solver_sync();
            {  // level 1: T_10, T_21, T_32 (192 quads)
                f2 x01 = f2_dup(0.f), x23 = f2_dup(0.f);
                x_quad(q_blk + 1, q_blk, q_blk, q_blk + 1, q_rr, q_jq, x01, x23);
                x_store(q_blk, q_rr, q_jq, x01, x23);
            }
            solver_sync();
            t_quad(q_blk + 1, q_blk, q_rr, q_jq);
            solver_sync();
        }
        if (warp < 4) {
            {  // level 2: X_20 with A_30 T_00 + A_31 T_10 of X_30 (slot 2), sharing the T loads
               // (threads 0-63); X_31 (threads 64-127)
                f2 x01 = f2_dup(0.f), x23 = f2_dup(0.f);
                if (tid < 64) {
                    f2 y01 = f2_dup(0.f), y23 = f2_dup(0.f);
                    x_quad2(2, 3, 0, 0, 2, q_rr, q_jq, x01, x23, y01, y23);
                    x_store(2, q_rr, q_jq, y01, y23);
                } else {
                    x_quad(3, 1, 1, 3, q_rr, q_jq, x01, x23);
                }
                x_store(q_blk, q_rr, q_jq, x01, x23);
            }
            solver4_sync();
            t_quad(q_blk + 2, q_blk, q_rr, q_jq);
            solver4_sync();
            if (tid < 64) {  // level 3: X_30 = (slot 2) + A_32 T_20
                const float4 p4 = *reinterpret_cast<const float4*>(&sX[(2 * 16 + q_rr) * 16 + 4 * q_jq]);
                f2 x01 = f2_of(p4.x, p4.y), x23 = f2_of(p4.z, p4.w);
                x_quad(3, 0, 2, 3, q_rr, q_jq, x01, x23);
                x_store(0, q_rr, q_jq, x01, x23);
            }
            solver4_sync();
            if (tid < 64) t_quad(3, 0, q_rr, q_jq);
            solver4_sync();
            // T -> bf16 hi and lo, K-major [r][i]; blocks above the diagonal are zero
            for (int idx = tid; idx < 64 * 8; idx += 128) {
                const int rr = idx >> 3, k8 = idx & 7;
                const float4 u0 = *reinterpret_cast<const float4*>(&sTf[rr * kTs + 8 * k8]);
                const float4 u1 = *reinterpret_cast<const float4*>(&sTf[rr * kTs + 8 * k8 + 4]);
                const float tv[8] = {u0.x, u0.y, u0.z, u0.w, u1.x, u1.y, u1.z, u1.w};
                float t8[8];
#pragma unroll
                for (int e = 0; e < 8; ++e) t8[e] = 8 * k8 + e <= rr ? tv[e] : 0.f;
                uint4 hv, lv;
                split8(t8, hv, lv);
                sts128(sTbf, kmajor_off(64, rr, k8), hv);
                sts128(sTbf + kOffTlo, kmajor_off(64, rr, k8), lv);
            }
            fence_async_smem();
        }

        // ------------------------------------------------ D: v conv, R = beta (V - P), by warps 4-15
        // while warps 0-3 finish T: D needs P from G3, not T.  Warp 15 (G3's issuer) waits for G3
        // and a named barrier of warps 6-15 passes that on; warps 4 and 5 join after the first
        // solve level and wait for G3 themselves.  Each quadrant's 64 tokens are 8 half-blocks
        // of 8, shared by its three D warps as 3 + 3 + 2 (the late warps 4, 5 and G3's issuer 15
        // take two).
        bool dfail = false;
        if (warp >= 4) {
            if (warp >= kSolveWarps) {
                if (warp == kThreads / 32 - 1) {
                    const bool ok = mbar_wait(&bars[1], par);
                    if (lane == 0) s_dfail = ok ? 0 : 1;
                }
                d_sync();
                dfail = s_dfail != 0;
            } else {
                dfail = !mbar_wait(&bars[1], par);
            }
            fence_after_sync();
            if (!dfail) {
                const int rank = warp < kSolveWarps ? 2 : (warp - kSolveWarps) >> 2;
                const int hb0 = 3 * rank, nhb = rank < 2 ? 3 : 2;
                const f2 w0 = f2_dup(sConvW[8 * kD + j]), w1 = f2_dup(sConvW[9 * kD + j]),
                         w2 = f2_dup(sConvW[10 * kD + j]), w3 = f2_dup(sConvW[11 * kD + j]);
                auto vat = [&](int rr) -> float {  // staged v row rr (t0 - 3 + rr), channel j
                    return to_f(*reinterpret_cast<const bf16*>(sm + kOffRawV + raw_off(kRawBox, rr, j)));
                };
                auto raw = [&](int64_t p) -> float {
                    if (p >= s0) return vat((int)(p - (t0 - 3)));
                    const int pos = (int)(p - s0);
                    return cs_in ? to_f(cs_in[((int64_t)n * 3 * HD + 2 * HD + (int64_t)h * kD + j) * 3 + 3 + pos]) : 0.f;
                };
                for (int hb = hb0; hb < hb0 + nhb; ++hb) {
                    const int i0 = 8 * hb;  // tokens i in [i0, i0 + 8)
                    const int64_t tb0 = t0 + i0;
                    const bool vrows = i0 < Lc && !ident_run;  // the identity-start run takes v = 0
                    float p0 = vrows ? raw(tb0 - 3) : 0.f;
                    float p1 = vrows ? raw(tb0 - 2) : 0.f;
                    float p2 = vrows ? raw(tb0 - 1) : 0.f;
                    uint32_t pv[8];
                    tmem_ld8(tb + lane_off + kColP + i0, pv);
                    tmem_ld_wait();
                    uint4 rhi, rlo;
                    uint32_t* rh = &rhi.x;
                    uint32_t* rl = &rlo.x;
#pragma unroll
                    for (int e = 0; e < 8; e += 2) {
                        // tokens i, i + 1 as a packed pair: conv, silu, R = beta (v - P)
                        const int i = i0 + e;
                        const bool ok0 = i < Lc && !ident_run, ok1 = i + 1 < Lc && !ident_run;
                        const float x0 = ok0 ? vat(i + 3) : 0.f;
                        const float x1 = ok1 ? vat(i + 4) : 0.f;
                        f2 u = mul2(w0, f2_of(p0, p1));
                        u = fma2(w1, f2_of(p1, p2), u);
                        u = fma2(w2, f2_of(p2, x0), u);
                        u = fma2(w3, f2_of(x0, x1), u);
                        const f2 hx = mul2(u, f2_dup(0.5f));  // silu(u) = h + h tanh(h), h = u / 2
                        const f2 sv = fma2(hx, f2_of(tanh_hw(f2_lo(hx)), tanh_hw(f2_hi(hx))), hx);
                        const f2 vr = f2_of(ok0 ? f2_lo(sv) : 0.f, ok1 ? f2_hi(sv) : 0.f);
                        const float2 b2 = *reinterpret_cast<const float2*>(&sBeta[i]);
                        const f2 rv = mul2(f2_of(b2.x, b2.y),
                                           sub2(vr, f2_of(__uint_as_float(pv[e]), __uint_as_float(pv[e + 1]))));
                        split2p(rv, rh[e / 2], rl[e / 2]);
                        p0 = p2;
                        p1 = x0;
                        p2 = x1;
                    }
                    tmem_st4(tb + lane_off + kColR + 4 * hb, rhi);
                    tmem_st4(tb + lane_off + kColR + 32 + 4 * hb, rlo);
                }
                tmem_st_wait();
            }
        }
        fence_async_smem();  // generic accesses to R1 (A, T, G) ordered before E's bulk copies into it
        fence_before_sync();
        failed = __syncthreads_or(dfail) != 0;  // T (warps 0-3) and R (warps 4-15) complete
        if (failed) break;

        // ------------------------------------------------ E: G4  W^T = R^T T^T; next chunk's g, beta, q/k rows staged
        if (tid == 0) {
            fence_after_sync();
            const uint32_t tbf = sbase + kOffR2;
#pragma unroll
            for (int term = 0; term < 3; ++term) {  // R hi . T hi, R lo . T hi, R hi . T lo
                const uint32_t acol = kColR + (term == 1 ? 32 : 0);
                const uint32_t tt = tbf + (term == 2 ? kOffTlo : 0);
#pragma unroll
                for (int kk = 0; kk < 4; ++kk)
                    mma_ts(tb + kColW, tb + acol + 8 * kk, desc_sw128(tt + kk * 32, 16, 1024), id_64, (term | kk) != 0);
            }
            mma_commit(&bars[2]);
        }
        // next chunk: g rows and beta into R1 (the solve is done with A and T) and sBeta (D is
        // done with it), by warp 1 (warp 0 polls G4)
        if (ci + 1 < ce) stage_G(ci + 1, 1);
        failed = wait_mma(&bars[2], par, warp == 0);
        if (failed) break;
        fence_after_sync();

        // ------------------------------------------------ F: W^T -> hi/lo operand
        {
            uint32_t wv[16];
            tmem_ld16(tb + lane_off + kColW + 16 * qt, wv);
            tmem_ld_wait();
            uint32_t whi[8], wlo[8];
#pragma unroll
            for (int e = 0; e < 8; ++e)
                split2(__uint_as_float(wv[2 * e]), __uint_as_float(wv[2 * e + 1]), whi[e], wlo[e]);
            tmem_st8(tb + lane_off + kColWop + 8 * qt, whi);
            tmem_st8(tb + lane_off + kColWop + 32 + 8 * qt, wlo);
            tmem_st_wait();
        }
        fence_before_sync();
        __syncthreads();

        // ------------------------------------------------ G: G5 (O += W M^T), G6 (dS = W^T Kt)
        if (tid == 0) {
            fence_after_sync();
            const uint32_t mh = sbase + kOffR2 + 8192, ml = sbase + kOffR2 + 16384;
            const uint32_t kth = sbase + kOffKThi, ktl = sbase + kOffKTlo;
#pragma unroll
            for (int term = 0; term < 3; ++term) {
                const uint32_t acol = kColWop + (term == 1 ? 32 : 0);
                const uint32_t bm = term == 2 ? ml : mh;
#pragma unroll
                for (int kk = 0; kk < 4; ++kk)
                    mma_ts(tb + kColO, tb + acol + 8 * kk, desc_sw128(bm + kk * 32, 16, 1024), id_64, 1);
            }
#pragma unroll
            for (int term = 0; term < 3; ++term) {
                const uint32_t acol = kColWop + (term == 1 ? 32 : 0);
                const uint32_t bk = term == 2 ? ktl : kth;
#pragma unroll
                for (int kk = 0; kk < 4; ++kk)
                    mma_ts(tb + kColS, tb + acol + 8 * kk, desc_sw128(bk + kk * 2 * kKtSbo, kKtLbo, kKtSbo),
                           id_g6, (term | kk) != 0);
            }
            mma_commit(&bars[3]);
        }
        bool gok = true;
        if (ci + 1 < ce) {  // the next chunk's log-decay sums, on warps 8-15 while G5/G6 are issued
            if (warp >= 8) {
                if (warp == 8) gok = mbar_wait(&bars[4], (uint32_t)((ci + 1 - cb) & 1));
                scan_sync();  // the g rows have landed
                scan_G_half(ci + 1);
            }
            cp_async_wait_all();  // beta (threads 64-127)
        }
        {
            bool ok = true;
            if (warp == 0) ok = mbar_wait(&bars[3], par);
            failed = __syncthreads_or(!ok || !gok) != 0;
        }
        if (failed) break;  // (the exit path waits for the g rows again, bounded)
        if (ci + 1 < ce) pend_clear(0);
        fence_after_sync();

        // ------------------------------------------------ H: state update, output epilogue
        // the next chunk's q/k rows into B3 (G3 finished with it in D); they land while the
        // epilogue runs
        if (ci + 1 < ce) stage_qk(ci + 1, 3);
        {
            uint32_t dsv[32];
            tmem_ld32(tb + lane_off + kColS + 32 * qt, dsv);
            tmem_ld_wait();
#pragma unroll
            for (int e = 0; e < 32; e += 4) {  // S = Diag(gamma) S + dS, channel pairs packed
                const float4 gm = *reinterpret_cast<const float4*>(&sConst[cGam * kD + 32 * qt + e]);
                const f2 s01 = fma2(f2_of(gm.x, gm.y), f2_of(Sreg[e], Sreg[e + 1]),
                                    f2_of(__uint_as_float(dsv[e]), __uint_as_float(dsv[e + 1])));
                const f2 s23 = fma2(f2_of(gm.z, gm.w), f2_of(Sreg[e + 2], Sreg[e + 3]),
                                    f2_of(__uint_as_float(dsv[e + 2]), __uint_as_float(dsv[e + 3])));
                Sreg[e] = f2_lo(s01);
                Sreg[e + 1] = f2_hi(s01);
                Sreg[e + 2] = f2_lo(s23);
                Sreg[e + 3] = f2_hi(s23);
            }
            uint32_t ov[16];
            tmem_ld16(tb + lane_off + kColO + 16 * qt, ov);
            tmem_ld_wait();
            float o[16];
#pragma unroll
            for (int e = 0; e < 16; e += 2) {
                const f2 o2 = mul2(f2_dup(scale), f2_of(__uint_as_float(ov[e]), __uint_as_float(ov[e + 1])));
                o[e] = f2_lo(o2);
                o[e + 1] = f2_hi(o2);
            }
            if (raw_out) {
                float* ot = reinterpret_cast<float*>(sm + kOffYT);  // [64][128] fp32 o tile
#pragma unroll
                for (int e = 0; e < 16; ++e) ot[(16 * qt + e) * kD + j] = o[e];
            } else {
            // sum over the warp's 32 channels of o^2 for each of its 16 tokens:
            // halve across lanes 8, 4, 2, 1 apart, then fold the two 16-lane halves
            float sq[16];
#pragma unroll
            for (int e = 0; e < 16; e += 2) {
                const f2 o2 = f2_of(o[e], o[e + 1]);
                const f2 q2 = mul2(o2, o2);
                sq[e] = f2_lo(q2);
                sq[e + 1] = f2_hi(q2);
            }
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
            sq[0] += __shfl_xor_sync(0xffffffffu, sq[0], 16);  // lane l: token 16qt + (l & 15)
            // the four warps of token quarter qt (one per channel quadrant) exchange their
            // partial sums on a named barrier of their own; lane l < 16 of every warp then
            // forms 1 / rms of token 16 qt + l and the lanes pass it round by shuffles
            if (lane < 16) sRed[(16 * qt + lane) * 4 + qd] = sq[0];
            quarter_sync(qt);
            float inv_l;
            {
                const float4 r4 = *reinterpret_cast<const float4*>(&sRed[(16 * qt + (lane & 15)) * 4]);
                inv_l = rsqrtf((r4.x + r4.y + r4.z + r4.w) * (1.0f / kD) + eps_rms);
            }
            const float wj = rms_w ? rms_w[j] : 1.f;
            const uint8_t* gt = sm + kOffGateT;  // staged gate boxes
            To* yt = reinterpret_cast<To*>(sm + kOffYT);  // [64][128] y tile (K~ is free after G6)
#pragma unroll
            for (int e = 0; e < 16; e += 2) {  // tokens rr, rr + 1 packed
                const int rr = 16 * qt + e;
                const f2 iv = f2_of(__shfl_sync(0xffffffffu, inv_l, e), __shfl_sync(0xffffffffu, inv_l, e + 1));
                f2 y2 = mul2(mul2(f2_of(o[e], o[e + 1]), iv), f2_dup(wj));
                if (gate_p) {  // sigmoid(z) = 1/2 + tanh(z / 2) / 2
                    const f2 hz = mul2(f2_of(to_f(*reinterpret_cast<const bf16*>(gt + raw_off(kGateBox, rr, j))),
                                             to_f(*reinterpret_cast<const bf16*>(gt + raw_off(kGateBox, rr + 1, j)))),
                                       f2_dup(0.5f));
                    y2 = mul2(y2, fma2(f2_dup(0.5f), f2_of(tanh_hw(f2_lo(hz)), tanh_hw(f2_hi(hz))), f2_dup(0.5f)));
                }
                yt[rr * kD + j] = from_f<To>(f2_lo(y2));
                yt[(rr + 1) * kD + j] = from_f<To>(f2_hi(y2));
            }
            }
        }
        fence_before_sync();
        __syncthreads();  // every dS read is done before S^T overwrites those columns; y tile complete
        fence_after_sync();
        if (raw_out) {
            // fp32 o rows -> the zero-start or identity-start buffer, 16-byte coalesced stores
            float* dst = zero_run ? sp.o_loc : sp.f_tr;
            const uint4* ot = reinterpret_cast<const uint4*>(sm + kOffYT);
            for (int idx = tid; idx < Lc * 32; idx += kThreads) {
                const int rr = idx >> 5, vec = idx & 31;
                *reinterpret_cast<uint4*>(dst + ((t0 + rr) * H + h) * kD + 4 * vec) = ot[rr * 32 + vec];
            }
        } else {
            // y rows -> out, 16-byte coalesced stores
            constexpr int kVpr = kD * (int)sizeof(To) / 16;
            const uint4* yt = reinterpret_cast<const uint4*>(sm + kOffYT);
            for (int idx = tid; idx < Lc * kVpr; idx += kThreads) {
                const int rr = idx / kVpr, vec = idx % kVpr;
                *reinterpret_cast<uint4*>(out + ((t0 + rr) * H + h) * kD + vec * (16 / (int)sizeof(To))) =
                    yt[rr * kVpr + vec];
            }
        }
        store_state_operand();
        fence_before_sync();
        __syncthreads();
        fence_after_sync();
    }

    // row copies still in flight (a wait above timed out): wait for them, bounded, before the
    // shared memory is released
    if (tid == 0)
        for (int i = 0; i < 3; ++i)
            if ((pend >> (2 * i)) & 1u) mbar_wait(&bars[4 + i], (pend >> (2 * i + 1)) & 1u);
    cp_async_wait_all();
    if (failed) {
        if (tid == 0) flag_status(d_status, KDA_ERR_TIMEOUT);
    } else {
        float* dst = sp.P == 1 ? (S_fin ? S_fin + (((int64_t)n * H + h) * kD) * kD : nullptr)
                               : (ident_run ? sp.trans : sp.end_state) + (((int64_t)u * sp.P + seg) * kD) * kD;
        if (dst) {
#pragma unroll
            for (int i = 0; i < 32; ++i) dst[(int64_t)(32 * qt + i) * kD + j] = Sreg[i];
        }
    }
    fence_before_sync();
    __syncthreads();
    if (warp == 0) tmem_dealloc(tb, kTmemCols);
}

bool device_supports_tc() {
    DeviceInfo d;
    return current_device_info(&d) && d.cc_major == 10 && d.cc_minor == 3;
}

int device_sm_count() {
    DeviceInfo d;
    return current_device_info(&d) ? d.sm_count : 1;
}

// Cost model of the automatic segment choice, in units of one chunk step of one CTA
// (about 15 us measured on GB300, the same for every role):
//  - segment-0 CTAs occupy U SMs for its w / (w + P - 1) share of the chunks; the
//    2 U (P - 1) shorter CTAs of the later segments run on the other SMs in
//    w = ceil(2 U (P - 1) / (SMs - U)) waves, which the split balances;
//  - the fix-up streams 1,536 bytes per token-head of the later segments, measured at
//    about 39 ns per (unit, chunk), i.e. kFixupPerUnitChunk chunk steps, across the GPU;
//  - each extra launch and CTA start-up costs about kSegOverhead chunk steps.
constexpr double kFixupPerUnitChunk = 0.0027;
constexpr double kSegOverhead = 2.0;
// Fewest chunks per later segment the automatic choice allows.
constexpr double kMinSegChunks = 8.0;

// Workspace layout of a segmented launch (offsets in bytes, 256-aligned).
struct SegLayout {
    size_t end_state, trans, start, o_loc, f_tr, total;
};

size_t round256(size_t x) { return (x + 255) / 256 * 256; }

SegLayout seg_layout(const kda_prefill_args& a, int P) {
    SegLayout l{};
    if (P <= 1) return l;
    const size_t st = round256((size_t)a.N * a.H * P * kD * kD * sizeof(float));
    const size_t ob = round256((size_t)a.T_total * a.H * kD * sizeof(float));
    l.end_state = 0;
    l.trans = st;
    l.start = 2 * st;
    l.o_loc = 3 * st;
    l.f_tr = 3 * st + ob;
    l.total = 3 * st + 2 * ob;
    return l;
}

// cuTensorMapEncodeTiled from the driver, through the runtime (no link against libcuda)
PFN_cuTensorMapEncodeTiled_v12000 tensor_map_encoder() {
    static PFN_cuTensorMapEncodeTiled_v12000 fn = [] {
        void* p = nullptr;
        cudaDriverEntryPointQueryResult q{};
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) != cudaSuccess ||
            q != cudaDriverEntryPointSuccess)
            p = nullptr;
        return reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
    }();
    return fn;
}

// [rows][cols] row-major tensor of 2- or 4-byte elements with row pitch row_bytes, boxes of
// box_c x box_r elements, 128-byte swizzle, zeros outside the tensor.
bool encode_map(CUtensorMap* m, const void* base, bool fp32, uint64_t cols, uint64_t rows, uint64_t row_bytes,
                uint32_t box_c, uint32_t box_r) {
    return encode_tensor_map_2d(m, base, fp32, cols, rows, row_bytes, box_c, box_r, true);
}

template <typename To>
cudaError_t tc_launch(const kda_prefill_args& a, const SegPlan& sp, cudaStream_t s) {
    auto kern = k_tc_prefill<To>;
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)kSmemBytes);
    if (e != cudaSuccess) return e;
    const int64_t xs = a.qkv_row_stride ? a.qkv_row_stride : (int64_t)a.H * a.D;
    TmaMaps maps;
    memset(&maps, 0, sizeof(maps));  // maps of absent tensors are never used
    if (a.T_total > 0) {
        const uint64_t cols = (uint64_t)a.H * kD, rows = (uint64_t)a.T_total;
        bool ok = encode_map(&maps.q, a.q, false, cols, rows, (uint64_t)xs * 2, 64, kRawRows) &&
                  encode_map(&maps.k, a.k, false, cols, rows, (uint64_t)xs * 2, 64, kRawRows) &&
                  encode_map(&maps.v, a.v, false, cols, rows, (uint64_t)xs * 2, 64, kRawRows) &&
                  encode_map(&maps.g, a.g, true, cols, rows, cols * 4, 32, kC);
        if (ok && a.gate) ok = encode_map(&maps.gate, a.gate, false, cols, rows, cols * 2, 64, kC);
        if (!ok) return cudaErrorInvalidValue;
    }
    const unsigned grid = (unsigned)((int64_t)a.N * a.H * (2 * sp.P - 1));
    kern<<<grid, kThreads, kSmemBytes, s>>>(
        (const bf16*)a.q, (const bf16*)a.k, (const bf16*)a.v, xs, a.conv_w, (const bf16*)a.conv_state_in,
        a.g, a.beta, (const bf16*)a.gate, a.rms_w, a.eps_l2, a.eps_rms, a.scale, a.initial_state,
        a.final_state, (To*)a.out, a.cu_seqlens, a.T_total, a.H, a.d_status, sp, maps, a.flags);
    return cudaGetLastError();
}

}  // namespace

bool encode_tensor_map_2d(CUtensorMap* m, const void* base, bool fp32, uint64_t cols, uint64_t rows,
                          uint64_t row_bytes, uint32_t box_c, uint32_t box_r, bool swizzle128) {
    const PFN_cuTensorMapEncodeTiled_v12000 enc = tensor_map_encoder();
    if (!enc) return false;
    const cuuint64_t dims[2] = {cols, rows};
    const cuuint64_t strides[1] = {row_bytes};
    const cuuint32_t box[2] = {box_c, box_r};
    const cuuint32_t es[2] = {1, 1};
    return enc(m, fp32 ? CU_TENSOR_MAP_DATA_TYPE_FLOAT32 : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(base),
               dims, strides, box, es, CU_TENSOR_MAP_INTERLEAVE_NONE,
               swizzle128 ? CU_TENSOR_MAP_SWIZZLE_128B : CU_TENSOR_MAP_SWIZZLE_NONE,
               CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

bool tc_prefill_applies(const kda_prefill_args& a) {
    return a.D == kD && a.chunk == kC && a.io == KDA_BF16 && (int64_t)a.N * a.H <= 0x7fffffffLL &&
           device_supports_tc();
}

SegChoice tc_seg_choice(const kda_prefill_args& a) {
    if (a.segments > 0) return {a.segments < KDA_MAX_SEGMENTS ? a.segments : KDA_MAX_SEGMENTS, 1};
    const int64_t U = (int64_t)a.N * a.H;
    const int64_t S = device_sm_count();
    if (U <= 0 || a.T_total <= 0 || a.N <= 0 || U >= S) return {1, 1};
    const double C = (double)a.T_total / ((double)a.N * kC);  // mean chunks per sequence
    SegChoice best{1, 1};
    double best_cost = C;
    for (int P = 2; P <= KDA_MAX_SEGMENTS; ++P) {
        if (U * (2 * P - 1) > 0x7fffffffLL) break;
        const int64_t w = (2 * U * (P - 1) + (S - U) - 1) / (S - U);
        const double b = C / (double)(w + P - 1);  // chunks per later segment
        if (b < kMinSegChunks) continue;
        const double first = (double)w * b;
        const double cost = first + kFixupPerUnitChunk * (double)U * (C - first) + kSegOverhead;
        if (cost < best_cost) {
            best_cost = cost;
            best = {P, (int)w};
        }
    }
    return best;
}

int tc_segments(const kda_prefill_args& a) { return tc_seg_choice(a).P; }

size_t tc_prefill_workspace(const kda_prefill_args& a) { return seg_layout(a, tc_segments(a)).total; }

// Segment 0's share of the chunks, as w / wd: with the later segments' CTAs in w waves, it
// balances segment 0 against them.  Measured, a later segment's chunk step costs about 14/15 of
// segment 0's (its runs write raw readouts without the RMSNorm and gate epilogue; the identity-
// start run also skips the v conv) and each of its CTAs about 0.4 chunk steps of start-up, so for
// a sequence of the batch's mean chunk count nc the share is the c0 / nc that minimises
// max(c0, w (14/15 ceil((nc - c0) / (P - 1)) + 0.4)) near the balance point.  A forced P
// (w = 1) keeps equal segments.
static void seg_share(const kda_prefill_args& a, const SegChoice& sc, int& w, int& wd) {
    const int P = sc.P;
    w = 1;
    wd = P;
    if (P <= 1 || a.segments > 0 || a.N <= 0) return;
    const double mean = (double)a.T_total / ((double)a.N * kC);
    const int64_t nc = mean < 1.0 ? 1 : (int64_t)(mean + 0.5);
    if (nc > 0x3fffffffLL) {  // (keeps w / wd in int; the plain wave share there)
        w = sc.w;
        wd = sc.w + P - 1;
        return;
    }
    constexpr int64_t kLaterStep = 14, kStartUp = 6;  // fifteenths of a segment-0 chunk step
    const int64_t W = sc.w;
    const int64_t est = W * (kLaterStep * nc + kStartUp * (P - 1)) / (15 * (int64_t)(P - 1) + kLaterStep * W);
    int64_t c0 = est < nc ? est : nc, best = -1;
    for (int64_t c = est - 1; c <= est + 3; ++c) {
        if (c < 0 || c > nc) continue;
        const int64_t sl = (nc - c + P - 2) / (P - 1);
        const int64_t t0 = 15 * c, t1 = W * (kLaterStep * sl + kStartUp);
        const int64_t cost = t0 > t1 ? t0 : t1;
        if (best < 0 || cost < best) {
            best = cost;
            c0 = c;
        }
    }
    w = (int)c0;
    wd = (int)nc;
}

cudaError_t launch_tc_prefill(const kda_prefill_args& a, char* ws, cudaStream_t s) {
    const int64_t units = (int64_t)a.N * a.H;
    if (units == 0) return cudaSuccess;
    const SegChoice sc = tc_seg_choice(a);
    const int P = sc.P;
    SegPlan sp{};
    sp.P = P;
    seg_share(a, sc, sp.w, sp.wd);
    if (P > 1) {
        const SegLayout l = seg_layout(a, P);
        sp.end_state = reinterpret_cast<float*>(ws + l.end_state);
        sp.trans = reinterpret_cast<float*>(ws + l.trans);
        sp.start = reinterpret_cast<float*>(ws + l.start);
        sp.o_loc = reinterpret_cast<float*>(ws + l.o_loc);
        sp.f_tr = reinterpret_cast<float*>(ws + l.f_tr);
    }
    cudaError_t e = a.out_dtype == KDA_FP32 ? tc_launch<float>(a, sp, s) : tc_launch<bf16>(a, sp, s);
    if (e != cudaSuccess || P == 1) return e;
    if ((e = launch_seg_combine(sp, (int)units, a.final_state, a.d_status, s)) != cudaSuccess) return e;
    return launch_seg_fixup(sp, a.cu_seqlens, a.N, a.T_total, a.H, (const bf16*)a.gate, a.rms_w,
                            a.eps_rms, a.out, a.out_dtype, device_sm_count(), a.d_status, s);
}

}  // namespace kda
