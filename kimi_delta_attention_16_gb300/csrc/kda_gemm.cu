// kda_gemm.cu -- the projections around the KDA layer on the Blackwell tensor
// cores: C[M][N] = A[M][K] . W[N][K]^T (bf16 operands, fp32 accumulation in
// tensor memory) with the activation of its consumer fused into the epilogue.
//
// Page "Kimi K3 / Architecture", KDA panel: the normalized input x_t goes
// through linear projections to q, k, v and to alpha_t / beta_t (channel-wise
// retention and one write strength per head, the log-decay bounded below by
// -5); the head output y_t leaves through W_o.  The gated-MLA panel of the same
// page writes the output gate as sigmoid(W_g x_t), full rank, one value per
// output channel.  Epilogues:
//   KDA_EPI_NONE     C = acc                     (gate pre-activations, y W_o)
//   KDA_EPI_DECAY    C = -5 sigmoid(acc)         (log-decay g in (-5, 0), fp32)
//   KDA_EPI_SIGMOID  C = sigmoid(acc)            (write strength beta in (0, 1), fp32)
//
// Persistent CTAs, one per SM, walk 128 x 256 output tiles in bands of 16
// m-blocks: within a band the m-block runs fastest, then the n-block, so the
// tiles in flight together share W tiles and one 2048-row slice of A, and the
// L2 holds both (A is read from DRAM about once, W once per band).  Warp roles in a
// CTA of 256 threads: warp 0 lane 0 feeds a 4-stage ring of shared-memory
// stages (A 128 x 64 and W 256 x 64 bf16 boxes, 128-byte swizzle) by TMA;
// warp 1 lane 0 issues tcgen05.mma (M = 128, N = 256, K = 16) into one of two
// TMEM accumulators of 256 columns and commits each stage back to the
// producer; warps 4-7 read the finished accumulator (lane = row), apply the
// epilogue and store, while the next tile accumulates into the other buffer.
// Every mbarrier wait has a clock deadline: on expiry the CTA records
// KDA_ERR_TIMEOUT and winds down without a fault.
#include "kda_internal.cuh"
#include "kda_tc.cuh"
#include "kda_tc_ptx.cuh"

namespace kda {

namespace {

using namespace tc;

constexpr int kBM = 128, kBN = 256, kBK = 64, kStages = 4;
constexpr int kBandM = 16;  // m-blocks per band of the tile order
constexpr int kThreads = 256;
constexpr uint32_t kTileA = kBM * kBK * 2;  // 16 KB
constexpr uint32_t kTileB = kBN * kBK * 2;  // 32 KB
constexpr uint32_t kStageBytes = kTileA + kTileB;
constexpr uint32_t kSmemBytes = kStages * kStageBytes + 1024;  // + alignment slack
constexpr uint32_t kAccCols = kBN;                              // one fp32 accumulator
constexpr uint32_t kTmemCols = 2 * kAccCols;                    // double-buffered

struct GemmMaps {
    CUtensorMap a, w;
};

// Output tile t -> (m0, n0) in the banded order described above.
__device__ __forceinline__ void tile_origin(int t, int m_tiles, int n_tiles, int& m0, int& n0) {
    const int band = t / (kBandM * n_tiles), r = t % (kBandM * n_tiles);
    const int rows = m_tiles - band * kBandM < kBandM ? m_tiles - band * kBandM : kBandM;
    m0 = (band * kBandM + r % rows) * kBM;
    n0 = (r / rows) * kBN;
}

__device__ __forceinline__ void tma_load_2d(uint32_t dst, const CUtensorMap* map, int x, int y, uint64_t* bar) {
    asm volatile(
        "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes [%0], [%1, {%2, %3}], [%4];" ::
            "r"(dst), "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y), "r"(smem_u32(bar))
        : "memory");
}
__device__ __forceinline__ void mbar_arrive(uint64_t* bar) {
    asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_u32(bar)) : "memory");
}

template <int Epi>
__device__ __forceinline__ float epilogue_op(float x) {
    if (Epi == KDA_EPI_DECAY) return -5.0f / (1.0f + expf(-x));
    if (Epi == KDA_EPI_SIGMOID) return 1.0f / (1.0f + expf(-x));
    return x;
}

template <int Epi, typename To>
__global__ void __launch_bounds__(kThreads, 1)
k_gemm(const __grid_constant__ GemmMaps maps, int M, int N, int K, To* __restrict__ C, int64_t ldc,
       int* d_status) {
    extern __shared__ uint8_t smem_raw[];
    __shared__ uint64_t full[kStages], empty[kStages], acc_full[2], acc_empty[2];
    __shared__ uint32_t s_tbase;
    __shared__ int s_fail;
    const uint32_t raw_addr = smem_u32(smem_raw);
    uint8_t* sm = smem_raw + (((raw_addr + 1023u) & ~1023u) - raw_addr);
    const uint32_t sbase = smem_u32(sm);
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int m_tiles = (M + kBM - 1) / kBM, n_tiles = (N + kBN - 1) / kBN;
    const int tiles = m_tiles * n_tiles, kb_n = K / kBK;

    if (warp == 2) {
        tmem_alloc(&s_tbase, kTmemCols);
        tmem_relinquish();
    }
    if (tid == 0) {
        for (int s = 0; s < kStages; ++s) {
            mbar_init(&full[s], 1);
            mbar_init(&empty[s], 1);
        }
        for (int b = 0; b < 2; ++b) {
            mbar_init(&acc_full[b], 1);
            mbar_init(&acc_empty[b], 4 * 32);
        }
        fence_mbar_init();
        s_fail = 0;
    }
    fence_before_sync();
    __syncthreads();
    fence_after_sync();
    const uint32_t tb = s_tbase;
    bool failed = false;

    if (warp == 0 && lane == 0) {
        // ---- producer: stage ring, phase bit flips at every wrap
        asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(&maps.a)) : "memory");
        asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(&maps.w)) : "memory");
        int s = 0;
        uint32_t ph = 0, issued = 0;  // bit s of issued: stage s has had a fill; its last parity in bit 8 + s
        for (int t = blockIdx.x; t < tiles && !failed; t += gridDim.x) {
            int m0, n0;
            tile_origin(t, m_tiles, n_tiles, m0, n0);
            for (int kb = 0; kb < kb_n; ++kb) {
                if (!mbar_wait(&empty[s], ph ^ 1u)) {
                    failed = true;
                    break;
                }
                const uint32_t st = sbase + (uint32_t)s * kStageBytes;
                mbar_expect_tx(&full[s], kStageBytes);
                tma_load_2d(st, &maps.a, kb * kBK, m0, &full[s]);
                tma_load_2d(st + kTileA, &maps.w, kb * kBK, n0, &full[s]);
                issued = (issued & ~(0x101u << s)) | ((1u | (ph << 8)) << s);
                if (++s == kStages) {
                    s = 0;
                    ph ^= 1u;
                }
            }
        }
        if (failed) {
            s_fail = 1;
            // fills still in flight: wait for them (bounded) before the shared memory goes away
            for (int i = 0; i < kStages; ++i)
                if ((issued >> i) & 1u) mbar_wait(&full[i], (issued >> (8 + i)) & 1u);
        }
    } else if (warp == 1 && lane == 0) {
        // ---- MMA issuer
        const uint32_t idesc = idesc_bf16(kBM, kBN, false, false);
        int s = 0;
        uint32_t ph = 0;
        int it = 0;
        for (int t = blockIdx.x; t < tiles && !failed; t += gridDim.x, ++it) {
            const int b = it & 1;
            if (!mbar_wait(&acc_empty[b], (uint32_t)(((it >> 1) & 1) ^ 1))) {
                failed = true;
                break;
            }
            fence_after_sync();
            const uint32_t dcol = tb + (uint32_t)b * kAccCols;
            for (int kb = 0; kb < kb_n; ++kb) {
                if (!mbar_wait(&full[s], ph)) {
                    failed = true;
                    break;
                }
                fence_after_sync();
                const uint32_t st = sbase + (uint32_t)s * kStageBytes;
#pragma unroll
                for (int kk = 0; kk < kBK / 16; ++kk)
                    mma_ss(dcol, desc_sw128(st + kk * 32, 16, 1024), desc_sw128(st + kTileA + kk * 32, 16, 1024), idesc,
                           (kb | kk) != 0);
                mma_commit(&empty[s]);  // the stage is free once these MMAs have read it
                if (++s == kStages) {
                    s = 0;
                    ph ^= 1u;
                }
            }
            if (failed) break;
            mma_commit(&acc_full[b]);
        }
        if (failed) s_fail = 1;
    } else if (warp >= 4) {
        // ---- epilogue: warp 4 + q reads TMEM lanes 32 q .. 32 q + 31 (rows of the tile)
        const int q = warp & 3;
        const uint32_t lane_off = (uint32_t)(32 * q) << 16;
        int it = 0;
        for (int t = blockIdx.x; t < tiles; t += gridDim.x, ++it) {
            const int b = it & 1;
            bool ok = true;
            if (lane == 0) ok = mbar_wait(&acc_full[b], (uint32_t)((it >> 1) & 1));
            ok = __shfl_sync(0xffffffffu, ok ? 1 : 0, 0) != 0;
            if (!ok) {
                failed = true;
                break;
            }
            fence_after_sync();
            int m0, n0;
            tile_origin(t, m_tiles, n_tiles, m0, n0);
            const int row = m0 + 32 * q + lane;
            To* crow = C + (int64_t)row * ldc + n0;
#pragma unroll 1
            for (int j = 0; j < kBN / 32; ++j) {
                uint32_t v[32];
                tmem_ld32(tb + lane_off + (uint32_t)b * kAccCols + 32 * j, v);
                tmem_ld_wait();
                const int n = n0 + 32 * j;
                if (row < M && n < N) {
                    float f[32];
#pragma unroll
                    for (int e = 0; e < 32; ++e) f[e] = epilogue_op<Epi>(__uint_as_float(v[e]));
                    if (n + 32 <= N && (ldc * (int64_t)sizeof(To)) % 16 == 0) {
#pragma unroll
                        for (int e = 0; e < 32; e += 8) store8(crow + 32 * j + e, f + e);
                    } else {
#pragma unroll
                        for (int e = 0; e < 32; ++e)
                            if (n + e < N) crow[32 * j + e] = from_f<To>(f[e]);
                    }
                }
            }
            fence_before_sync();
            mbar_arrive(&acc_empty[b]);  // this thread is done with accumulator b
        }
        if (failed) s_fail = 1;
    }
    fence_before_sync();
    __syncthreads();
    if (s_fail && tid == 0) flag_status(d_status, KDA_ERR_TIMEOUT);
    if (warp == 2) tmem_dealloc(tb, kTmemCols);
}

template <int Epi, typename To>
cudaError_t gemm_launch(const kda_gemm_args& g, cudaStream_t s) {
    auto kern = k_gemm<Epi, To>;
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)kSmemBytes);
    if (e != cudaSuccess) return e;
    GemmMaps maps;
    if (!encode_tensor_map_2d(&maps.a, g.A, false, (uint64_t)g.K, (uint64_t)g.M, (uint64_t)g.lda * 2, kBK, kBM, true) ||
        !encode_tensor_map_2d(&maps.w, g.W, false, (uint64_t)g.K, (uint64_t)g.N, (uint64_t)g.ldw * 2, kBK, kBN, true))
        return cudaErrorInvalidValue;
    DeviceInfo d;
    const int sms = current_device_info(&d) ? d.sm_count : 148;
    const int tiles = ((g.M + kBM - 1) / kBM) * ((g.N + kBN - 1) / kBN);
    kern<<<tiles < sms ? tiles : sms, kThreads, kSmemBytes, s>>>(maps, g.M, g.N, g.K, (To*)g.C, g.ldc, g.d_status);
    return cudaGetLastError();
}

}  // namespace

bool gemm_supported_device() {
    DeviceInfo d;
    return current_device_info(&d) && d.cc_major == 10 && d.cc_minor == 3;
}

cudaError_t launch_gemm(const kda_gemm_args& g, cudaStream_t s) {
    if (g.M == 0 || g.N == 0) return cudaSuccess;
    const bool f32 = g.c_dtype == KDA_FP32;
    switch (g.epilogue) {
        case KDA_EPI_NONE: return f32 ? gemm_launch<KDA_EPI_NONE, float>(g, s) : gemm_launch<KDA_EPI_NONE, bf16>(g, s);
        case KDA_EPI_DECAY: return f32 ? gemm_launch<KDA_EPI_DECAY, float>(g, s) : gemm_launch<KDA_EPI_DECAY, bf16>(g, s);
        case KDA_EPI_SIGMOID:
            return f32 ? gemm_launch<KDA_EPI_SIGMOID, float>(g, s) : gemm_launch<KDA_EPI_SIGMOID, bf16>(g, s);
        default: return cudaErrorInvalidValue;
    }
}

}  // namespace kda
