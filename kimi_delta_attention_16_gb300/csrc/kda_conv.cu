// kda_conv.cu -- causal depthwise short convolution + SiLU (+ per-head L2 on
// q and k), and the rolling conv-state hand-off.
//
// Page "Kimi K3 / Architecture", panel "KDA short convolution . one channel c
// at token t": a width-4 causal window over x[t-3..t] of one channel, only
// time is mixed, left padding keeps the length, SiLU after the 4-tap sum,
// then q and k are L2-normalised and v is written as it is; the autoregressive rolling
// state keeps the previous 3 values of every channel.
//
// Layout: each row of x / y holds 3*H*D channels (q | k | v, channel =
// part*H*D + h*D + d).  One thread owns 8 consecutive channels (a 16-byte
// bf16 vector) and walks a run of TT consecutive tokens, keeping the last
// three raw values in registers, so every raw row is read once per run.
// The L2 norm of a head (D channels = D/8 lanes, aligned within a warp) is a
// shuffle reduction.  HBM-bound: one read of x, one write of y.
#include "kda_internal.cuh"

namespace kda {

namespace {

constexpr int kConvThreads = 256;
constexpr int kConvVec = 8;                              // channels per thread
constexpr int kConvChanPerBlock = kConvThreads * kConvVec;  // 2048
constexpr int kConvTokens = 32;                          // tokens per run

__global__ void k_check_cu(const int32_t* cu, int N, int64_t T_total, int* d_status) {
    const int n = blockIdx.x * blockDim.x + threadIdx.x;
    if (n > N) return;
    const int64_t c = cu[n];
    bool bad = c < 0 || c > T_total;
    if (n == 0) bad |= (c != 0);
    if (n == N) bad |= (c != T_total);
    if (n < N) bad |= (cu[n + 1] < c);
    if (bad) flag_status(d_status, KDA_ERR_DEVICE_ARG);
}

// Index of the sequence holding token t: largest n in [0, N) with cu[n] <= t.
__device__ __forceinline__ int find_seq(const int32_t* cu, int N, int64_t t) {
    int lo = 0, hi = N - 1;
    while (lo < hi) {
        const int mid = (lo + hi + 1) >> 1;
        if ((int64_t)cu[mid] <= t) lo = mid; else hi = mid - 1;
    }
    return lo;
}

template <typename Tin, typename Tout>
__global__ void __launch_bounds__(kConvThreads)
k_short_conv(QKVParts xp, int64_t xs, const float* __restrict__ w,
             const int32_t* __restrict__ cu, int N, int64_t T_total, int n_ch, int D,
             const Tin* __restrict__ cs_in, Tout* __restrict__ y, int64_t ys, int l2_limit,
             float eps) {
    const int ch0 = blockIdx.y * kConvChanPerBlock + threadIdx.x * kConvVec;
    const bool active = ch0 < n_ch;
    const int part_w = n_ch / 3;  // H*D channels per part, a multiple of 8
    const int part = active ? ch0 / part_w : 0;
    const void* base = part == 0 ? xp.p[0] : (part == 1 ? xp.p[1] : xp.p[2]);
    const Tin* __restrict__ x = static_cast<const Tin*>(base) + (ch0 - part * part_w);
    const int64_t t_begin = (int64_t)blockIdx.x * kConvTokens;
    int64_t t_end = t_begin + kConvTokens;
    if (t_end > T_total) t_end = T_total;
    const int lanes_per_head = D / kConvVec;  // 2..16, a power of two
    const bool do_l2 = ch0 < l2_limit;        // whole head groups share this

    float wt[kConvVec][4];
#pragma unroll
    for (int j = 0; j < kConvVec; ++j)
#pragma unroll
        for (int m = 0; m < 4; ++m) wt[j][m] = active ? w[(int64_t)(ch0 + j) * 4 + m] : 0.f;

    int n = find_seq(cu, N, t_begin);
    int64_t s, e;
    seq_range(cu, n, T_total, s, e);
    float win[3][kConvVec];  // raw x[t-3], x[t-2], x[t-1]
    bool need_window = true;

    for (int64_t t = t_begin; t < t_end; ++t) {
        while (t >= e && n < N - 1) {  // crossed into a later sequence
            ++n;
            seq_range(cu, n, T_total, s, e);
            need_window = true;
        }
        if (need_window) {
            const int64_t p = t - s;  // local position of t (may be < 0 if cu is inconsistent)
#pragma unroll
            for (int m = 0; m < 3; ++m) {
                const int64_t pos = p - 3 + m;
                if (!active) {
#pragma unroll
                    for (int j = 0; j < kConvVec; ++j) win[m][j] = 0.f;
                } else if (pos >= 0) {
                    load8(x + (s + pos) * xs, win[m]);
                } else {
#pragma unroll
                    for (int j = 0; j < kConvVec; ++j)
                        win[m][j] = (cs_in && pos >= -3)
                                        ? to_f(cs_in[((int64_t)n * n_ch + ch0 + j) * 3 + 3 + pos])
                                        : 0.f;
                }
            }
            need_window = false;
        }
        float xt[kConvVec], u[kConvVec];
        if (active) {
            load8(x + t * xs, xt);
        } else {
#pragma unroll
            for (int j = 0; j < kConvVec; ++j) xt[j] = 0.f;
        }
        float ss = 0.f;
#pragma unroll
        for (int j = 0; j < kConvVec; ++j) {
            const float a = wt[j][0] * win[0][j] + wt[j][1] * win[1][j] + wt[j][2] * win[2][j] +
                            wt[j][3] * xt[j];
            u[j] = siluf_(a);
            ss += u[j] * u[j];
            win[0][j] = win[1][j];
            win[1][j] = win[2][j];
            win[2][j] = xt[j];
        }
        // per-head sum of squares over lanes_per_head aligned lanes
        for (int off = 1; off < lanes_per_head; off <<= 1) ss += __shfl_xor_sync(0xffffffffu, ss, off);
        if (do_l2) {
            const float inv = 1.0f / sqrtf(ss + eps);
#pragma unroll
            for (int j = 0; j < kConvVec; ++j) u[j] *= inv;
        }
        if (active) store8(y + t * ys + ch0, u);
    }
}

template <typename T>
__global__ void k_conv_state_out(QKVParts xp, int64_t xs, const int32_t* __restrict__ cu,
                                 int N, int64_t T_total, int n_ch, const T* __restrict__ cs_in,
                                 T* __restrict__ cs_out) {
    const int64_t idx = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
    if (idx >= (int64_t)N * n_ch) return;
    const int n = (int)(idx / n_ch);
    const int ch = (int)(idx % n_ch);
    const int part_w = n_ch / 3;
    const int part = ch / part_w;
    const T* __restrict__ x =
        static_cast<const T*>(part == 0 ? xp.p[0] : (part == 1 ? xp.p[1] : xp.p[2]));
    const int c = ch - part * part_w;
    int64_t s, e;
    seq_range(cu, n, T_total, s, e);
    const int64_t L = e - s;
#pragma unroll
    for (int m = 0; m < 3; ++m) {
        const int64_t pos = L - 3 + m;
        T v;
        if (pos >= 0) v = x[(s + pos) * xs + c];
        else if (cs_in) v = cs_in[idx * 3 + 3 + pos];
        else v = from_f<T>(0.f);
        cs_out[idx * 3 + m] = v;
    }
}

}  // namespace

cudaError_t launch_check_cu(const int32_t* cu, int N, int64_t T_total, int* d_status,
                            cudaStream_t s) {
    if (!d_status) return cudaSuccess;
    const int threads = 256, blocks = (N + 1 + threads - 1) / threads;
    k_check_cu<<<blocks, threads, 0, s>>>(cu, N, T_total, d_status);
    return cudaGetLastError();
}

template <typename Tin, typename Tout>
static cudaError_t conv_impl(QKVParts x, int64_t xs, const float* w, const int32_t* cu, int N,
                             int64_t T_total, int H, int D, const void* cs_in, void* y, int64_t ys,
                             int l2norm_qk, float eps, cudaStream_t s) {
    const int n_ch = 3 * H * D;
    if (T_total == 0 || N == 0) return cudaSuccess;
    dim3 grid((unsigned)((T_total + kConvTokens - 1) / kConvTokens),
              (n_ch + kConvChanPerBlock - 1) / kConvChanPerBlock);
    k_short_conv<Tin, Tout><<<grid, kConvThreads, 0, s>>>(
        x, xs, w, cu, N, T_total, n_ch, D, static_cast<const Tin*>(cs_in),
        static_cast<Tout*>(y), ys, l2norm_qk ? 2 * H * D : 0, eps);
    return cudaGetLastError();
}

cudaError_t launch_short_conv(QKVParts x, int64_t xs, kda_dtype in_dt, const float* w,
                              const int32_t* cu, int N, int64_t T_total, int H, int D,
                              const void* cs_in, void* y, int64_t ys, kda_dtype out_dt,
                              int l2norm_qk, float eps, cudaStream_t s) {
    if (in_dt == KDA_BF16 && out_dt == KDA_BF16)
        return conv_impl<bf16, bf16>(x, xs, w, cu, N, T_total, H, D, cs_in, y, ys, l2norm_qk, eps, s);
    if (in_dt == KDA_BF16 && out_dt == KDA_FP32)
        return conv_impl<bf16, float>(x, xs, w, cu, N, T_total, H, D, cs_in, y, ys, l2norm_qk, eps, s);
    if (in_dt == KDA_FP32 && out_dt == KDA_FP32)
        return conv_impl<float, float>(x, xs, w, cu, N, T_total, H, D, cs_in, y, ys, l2norm_qk, eps, s);
    return cudaErrorInvalidValue;
}

cudaError_t launch_conv_state_out(QKVParts x, int64_t xs, kda_dtype dt, const int32_t* cu,
                                  int N, int64_t T_total, int n_ch, const void* cs_in,
                                  void* cs_out, cudaStream_t s) {
    const int64_t total = (int64_t)N * n_ch;
    if (total == 0) return cudaSuccess;
    const int threads = 256;
    const unsigned blocks = (unsigned)((total + threads - 1) / threads);
    if (dt == KDA_BF16)
        k_conv_state_out<bf16><<<blocks, threads, 0, s>>>(x, xs, cu, N,
                                                          T_total, n_ch,
                                                          static_cast<const bf16*>(cs_in),
                                                          static_cast<bf16*>(cs_out));
    else
        k_conv_state_out<float><<<blocks, threads, 0, s>>>(x, xs, cu, N,
                                                           T_total, n_ch,
                                                           static_cast<const float*>(cs_in),
                                                           static_cast<float*>(cs_out));
    return cudaGetLastError();
}

}  // namespace kda
