/*
 * kda.h -- C ABI of libkda.so: the Kimi Delta Attention (KDA) layer on one
 * GB300 (sm_103a).
 *
 * What the layer computes, per head of width D (page "Kimi K3 / Architecture",
 * panel "Kimi Delta Attention . one head at token t", and page "Animated Kimi
 * K3 architecture diagram", section "LOCAL MEMORY: A FIXED MATRIX THAT
 * PREDICTS, FORGETS, AND CORRECTS"):
 *
 *   short conv  u = sum_{j=0..3} w[j] x[t-3+j] per channel, then SiLU
 *   L2 norm     q <- q / sqrt(|q|^2 + eps_l2), same for k (v is not normalised)
 *   decay       S_bar = Diag(exp(g_t)) S_{t-1}           (g_t: log-decay per key channel)
 *   correct     e_t = v_t - S_bar^T k_t
 *   write       S_t = S_bar + beta_t k_t e_t^T          (beta_t: one scalar per token, head)
 *   read        o_t = scale * S_t^T q_t
 *   epilogue    y_t = o_t / sqrt(mean(o_t^2) + eps_rms) * w_rms * sigmoid(gate_t)
 *
 * The state S is a fixed D x D fp32 matrix per (sequence, head), row = key
 * channel, column = value channel.
 *
 * Conventions for every entry point:
 *  - Ownership: the caller owns every buffer.  The library allocates nothing
 *    on the device.  Its only device memory of its own is the fixed scratch
 *    array of kda_prefill_noalloc (below), and its only state between calls is
 *    a per-device cache of device attributes (SM count, compute capability).
 *  - Asynchrony: calls only enqueue work on `stream` (a cudaStream_t; NULL is
 *    the legacy default stream) and never synchronise.
 *  - Errors: invalid arguments return before anything is launched.  A launch
 *    failure returns KDA_ERR_CUDA.  Conditions found on the device (an
 *    inconsistent cu_seqlens) are written to the optional `d_status` word
 *    (a device int the caller zeroes) and the affected work is skipped; no
 *    kernel traps or asserts.
 *  - Value ranges: g is expected in [-5, 0] (the pages bound the log-decay
 *    below by -5) and beta in [0, 1].  They are not range-checked on the
 *    device.  Outside that range results may overflow to inf/NaN: on every
 *    path for g > 0 (growing state), and on the tensor-core path also for
 *    g < -5, whose split decay factors reach e^{16 |g|} (e^{96} > FLT_MAX at
 *    g = -6).  Both ends of the range, g = -5 and g = 0, are supported.
 *  - Shapes: D in {16, 32, 64, 128}; the tensor-core prefill path needs
 *    D = 128, chunk = 64 and bf16 inputs, everything else takes the fp32 SIMT
 *    path.
 */
#ifndef KDA_H
#define KDA_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* Same type as cudaStream_t, declared without the CUDA headers. */
typedef struct CUstream_st* kda_stream_t;

typedef enum {
    KDA_OK = 0,
    KDA_ERR_INVALID_ARG = 1, /* null pointer, bad size, misalignment, aliasing, bad cu_seqlens */
    KDA_ERR_UNSUPPORTED = 2, /* shape or dtype this library does not implement */
    KDA_ERR_WORKSPACE = 3,   /* workspace missing or smaller than kda_prefill_workspace_size */
    KDA_ERR_CUDA = 4,        /* a CUDA runtime call or launch failed */
    KDA_ERR_TIMEOUT = 5,     /* a bounded device-side wait gave up (reported via d_status) */
    KDA_ERR_DEVICE_ARG = 6   /* the device copy of cu_seqlens was inconsistent (via d_status) */
} kda_status;

typedef enum { KDA_BF16 = 0, KDA_FP32 = 1 } kda_dtype;

/* Static English text for a status code. */
const char* kda_status_string(int status);

/* Text describing the last error returned on the calling host thread. */
const char* kda_last_error(void);

/* Library version as major*10000 + minor*100 + patch. */
int kda_version(void);

/* ------------------------------------------------------------------------
 * kda_short_conv -- causal depthwise short convolution + SiLU (+ L2 on q, k).
 * Page "Kimi K3 / Architecture", panel "KDA short convolution . one channel
 * c at token t": window of width 4 over x[t-3..t] of one channel, only time
 * is mixed, left padding keeps the length, SiLU after the 4-tap sum; Q and K
 * are then L2-normalised per head, V is not.  Filter banks Wq, Wk, Wv; the
 * rolling state keeps the previous 3 raw values per channel ([B,36864,3] for
 * 96 heads of 128).
 *
 *   x         [T_total][row stride x_row_stride elements], channels q|k|v:
 *             channel = part*H*D + h*D + d (part 0=q, 1=k, 2=v); io dtype.
 *   w         [3*H*D][4] fp32; tap 3 multiplies x[t], tap 0 multiplies x[t-3].
 *   cu_seqlens device int32 [N+1]: cu[0]=0, non-decreasing, cu[N]=T_total.
 *             Sequences never see each other's tokens.
 *   cu_seqlens_host optional host copy; when given it is validated on the
 *             host (no device sync is ever needed).
 *   conv_state_in  [N][3*H*D][3] io dtype, oldest first, or NULL (zeros).
 *   conv_state_out [N][3*H*D][3] io dtype or NULL: the last 3 raw values of
 *             each sequence (taking conv_state_in into account for short
 *             sequences).  Must not overlap conv_state_in.
 *   y         [T_total][y_row_stride elements] io dtype; must not overlap x.
 *   l2norm_qk nonzero: L2-normalise the q and k parts per head with eps_l2.
 * Alignment: x, y 16-byte aligned; row strides multiples of 8 elements (bf16)
 * or 4 elements (fp32); D, H >= 1 with D in {16,32,64,128}.
 * ------------------------------------------------------------------------ */
kda_status kda_short_conv(const void* x, int64_t x_row_stride, const float* w,
                          const int32_t* cu_seqlens, const int32_t* cu_seqlens_host, int N,
                          int64_t T_total, int H, int D, const void* conv_state_in,
                          void* conv_state_out, void* y, int64_t y_row_stride, int l2norm_qk,
                          float eps_l2, kda_dtype io, int* d_status, kda_stream_t stream);

/* ------------------------------------------------------------------------
 * kda_prefill -- the whole layer over packed variable-length sequences.
 * Page "Kimi K3 / Architecture", KDA panel: the chunkwise form (the state
 * recurs from chunk to chunk, the tokens of a chunk are taken together as
 * dense tensor-core tiles); page "Animated Kimi K3 architecture diagram": the
 * state is carried across chunks.  Chunks of `chunk` tokens start at every
 * sequence start; the last chunk of a sequence may be partial.  The result
 * does not depend on `chunk` beyond rounding.
 * ------------------------------------------------------------------------ */
typedef struct {
    int N;                 /* sequences */
    int H;                 /* heads */
    int D;                 /* head width (dk = dv = D) */
    int chunk;             /* 16, 32 or 64 */
    int64_t T_total;       /* packed tokens */
    kda_dtype io;          /* dtype of q, k, v, gate and the conv states */
    kda_dtype out_dtype;   /* dtype of out */
    const int32_t* cu_seqlens;       /* device [N+1] */
    const int32_t* cu_seqlens_host;  /* host [N+1] or NULL (then only device-checked) */
    const void* q;         /* [T_total][qkv_row_stride] raw projections, before the conv */
    const void* k;         /* same layout as q */
    const void* v;         /* same layout as q */
    int64_t qkv_row_stride;/* elements between tokens of q/k/v; 0 means H*D */
    const float* conv_w;   /* [3][H*D][4] fp32 (q, k, v filter banks) */
    const void* conv_state_in;  /* [N][3*H*D][3] or NULL (zero left padding) */
    void* conv_state_out;       /* [N][3*H*D][3] or NULL; must not overlap conv_state_in */
    const float* g;        /* [T_total][H][D] fp32 log-decay, expected in [-5, 0] */
    const float* beta;     /* [T_total][H] fp32, expected in [0, 1] */
    const void* gate;      /* [T_total][H][D] pre-sigmoid output gate, io dtype, or NULL */
    const float* rms_w;    /* [D] fp32 RMSNorm weight, or NULL (ones) */
    float eps_l2;          /* typical 1e-6 */
    float eps_rms;         /* typical 1e-6 */
    float scale;           /* readout scale, typical 1.0 */
    const float* initial_state; /* [N][H][D][D] fp32 or NULL (zeros) */
    float* final_state;    /* [N][H][D][D] fp32 or NULL; may equal initial_state */
    void* out;             /* [T_total][H][D] out_dtype; must not overlap any input */
    void* workspace;       /* device scratch, 256-byte aligned, or NULL if size 0 */
    size_t workspace_bytes;
    int* d_status;         /* optional device int for device-side conditions */
    int flags;             /* KDA_FLAG_* */
    int segments;          /* tensor-core path: segments each sequence is cut into (below);
                              0 = chosen from N*H and the SM count, 1 = none, 2..16 forced */
} kda_prefill_args;

#define KDA_FLAG_FORCE_SIMT 1    /* take the fp32 SIMT path even where tensor cores apply */
#define KDA_FLAG_NO_RECURRENT 2  /* never take the recurrent short-sequence path (below) */
/* Test only: on the tensor-core path, the staging of each CTA's first q/k rows is never
 * issued, so the mbarrier wait for them runs out (after about 2 s of GPU clock); the kernel
 * then writes KDA_ERR_TIMEOUT to *d_status and returns without writing out or final_state.
 * Exercises the device-side timeout path without a fault or a hang; ignored by the other
 * paths. */
#define KDA_FLAG_TEST_DROP_STAGING 4

/* Paths of kda_prefill (reported by kda_prefill_plan):
 *  KDA_PATH_SIMT         fp32 SIMT chunkwise path (any D, chunk, dtype);
 *  KDA_PATH_TENSOR_CORE  tcgen05 chunkwise path (D = 128, chunk = 64, bf16 inputs);
 *  KDA_PATH_RECURRENT    token-by-token path for batches of short sequences:
 *                        D = 128, cu_seqlens_host given and every sequence at most
 *                        KDA_RECURRENT_MAX_LEN tokens (multi-token decode, speculative
 *                        verification); each (sequence, head) state is read and
 *                        written once, no workspace.  `chunk` does not matter there:
 *                        the result equals the chunkwise one up to rounding. */
#define KDA_PATH_SIMT 0
#define KDA_PATH_TENSOR_CORE 1
#define KDA_PATH_RECURRENT 2
#define KDA_RECURRENT_MAX_LEN 8

/* Segment-parallel scan (tensor-core path).  One (sequence, head) is a chain
 * of chunks, each depending on the state the previous one leaves.  When the
 * batch has too few (sequence, head) units to fill the GPU, each sequence's
 * chunks are cut into P contiguous segments of ceil(chunks / P) chunks.  Every
 * step of the recurrence maps the state affinely, S -> (I - beta k k^T)
 * Diag(e^g) S + beta k v^T, so a whole segment s maps its start state as
 * S_{s+1} = M_s S_s + B_s, and each of its outputs as o_t = o_t' + S_s^T f_t.
 * Segment 0 runs from the initial state as usual; every later segment runs
 * twice, in parallel with the others: from a zero state (its outputs o_t'
 * and B_s) and with v = 0 from the identity (f_t and M_s).  A second kernel
 * composes S_1 .. S_{P-1} and the final state in order, and a third adds
 * S_s^T f_t to o_t' and applies RMSNorm and the gate.  The results equal
 * the single-pass ones up to rounding.  Workspace: 3 P N H D^2 + 2 T_total H D
 * floats when P > 1, else none.  `segments` is ignored by the SIMT path. */
#define KDA_MAX_SEGMENTS 16

/* Bytes of workspace kda_prefill needs for these arguments (0 allowed). */
kda_status kda_prefill_workspace_size(const kda_prefill_args* args, size_t* bytes);

kda_status kda_prefill(const kda_prefill_args* args, kda_stream_t stream);

/* The plan kda_prefill takes for these arguments on the current device:
 * *path = one of KDA_PATH_*, and *segments = segments per sequence (1
 * except on the tensor-core path when segmenting applies).  Reads the sizes,
 * dtypes, flags, `segments`, the alignment of the state pointers and, when
 * given, cu_seqlens_host; no device pointer is dereferenced; launches nothing. */
kda_status kda_prefill_plan(const kda_prefill_args* args, int* path, int* segments);

/* ------------------------------------------------------------------------
 * kda_prefill_noalloc -- kda_prefill for callers that cannot allocate device
 * memory when they call it: a plugin inside a host application that owns
 * every device allocation and hands over only input and output buffers, a
 * service that reserved its whole memory budget at start-up, or a
 * latency-critical loop that cannot afford the device-wide synchronisation
 * of cudaMalloc/cudaFree.  The pages have no counterpart to this entry
 * point; it is a packaging convenience of this library.
 *
 * It runs the fp32 SIMT path (the path that stages data in scratch) with its
 * scratch taken from a fixed array of KDA_NOALLOC_SCRATCH_BYTES compiled
 * into the library.  Every GPU that loads the library holds that array
 * until the process exits.  args->workspace and args->workspace_bytes are
 * ignored; everything else means what it means for kda_prefill, and the
 * caller still provides every input and output buffer.  The call allocates
 * nothing: no cudaMalloc, no cudaFree, no allocating library routine.
 *
 * Limit: the SIMT path needs 16*T_total*H*D bytes of scratch (two 256-byte
 * aligned parts); a call needing more than KDA_NOALLOC_SCRATCH_BYTES returns
 * KDA_ERR_WORKSPACE before launching anything (use kda_prefill with a
 * workspace instead).
 *
 * Set-up: every call looks up the array's device address on the current
 * device (a host-side lookup that allocates nothing), so the address is
 * right after cudaDeviceReset or under another context too.  The first
 * lookup in a context also loads the library's device code there: make the
 * first call on each device before any stream capture begins.
 *
 * Sharing: all calls use the same array, which keeps the previous call's
 * contents.  Nothing in it needs to start at zero (every scratch byte a call
 * reads is written earlier in the same call).  Calls whose work overlaps on
 * the GPU (different streams, or host threads without ordering between
 * them) race on the array: order them on one stream.
 * ------------------------------------------------------------------------ */
#define KDA_NOALLOC_SCRATCH_BYTES ((size_t)64 << 20) /* 64 MiB per device */

kda_status kda_prefill_noalloc(const kda_prefill_args* args, kda_stream_t stream);

/* ------------------------------------------------------------------------
 * kda_decode_step -- one new token for each of N sequences, states updated
 * in place.  Page "Kimi K3 / Architecture", panel "KDA short convolution":
 * the rolling state keeps the previous 3 raw values of every channel; page
 * "Animated Kimi K3 architecture diagram": the four moves on one token.
 * ------------------------------------------------------------------------ */
typedef struct {
    int N, H, D;
    kda_dtype io;          /* dtype of q, k, v, gate and conv_state */
    kda_dtype out_dtype;   /* dtype of out */
    const void* q;         /* [N][qkv_row_stride] raw new token, before the conv */
    const void* k;
    const void* v;
    int64_t qkv_row_stride;/* 0 means H*D */
    const void* gate;      /* [N][H][D] or NULL */
    const float* g;        /* [N][H][D] */
    const float* beta;     /* [N][H] */
    const float* conv_w;   /* [3][H*D][4] */
    const float* rms_w;    /* [D] or NULL */
    float eps_l2, eps_rms, scale;
    float* state;          /* [N][H][D][D] fp32, read and written in place */
    void* conv_state;      /* [N][3*H*D][3] io dtype, rolled in place */
    void* out;             /* [N][H][D] out_dtype */
    int* d_status;
} kda_decode_args;

kda_status kda_decode_step(const kda_decode_args* args, kda_stream_t stream);

/* ------------------------------------------------------------------------
 * kda_gemm -- the projections around the layer on the tensor cores, with the
 * activation of their consumer fused into the epilogue:
 *
 *   C[M][N] = epilogue( A[M][K] . W[N][K]^T )
 *
 * Page "Kimi K3 / Architecture", KDA panel: the normalized input x_t goes through
 * linear projections to q, k, v and to alpha_t / beta_t (channel-wise
 * retention, one write strength per head, log-decay bounded below by -5); the
 * head output y_t leaves through W_o.  The gated-MLA panel of the same page writes
 * the output gate as sigmoid(W_g x_t), full rank, one value per output channel.
 * The pages give no activation for alpha and beta; this library reads "bounded
 * log-decay >= -5" as g = -5 sigmoid(z) and the write strength as beta =
 * sigmoid(z), so that g and beta land in the ranges kda_prefill expects.
 *
 *   KDA_EPI_NONE     C = acc              (e.g. gate pre-activations x W_g^T, or y W_o^T)
 *   KDA_EPI_DECAY    C = -5 sigmoid(acc)  (the log-decay g of kda_prefill, fp32)
 *   KDA_EPI_SIGMOID  C = sigmoid(acc)     (the write strength beta, fp32)
 *
 *   A  [M][lda] bf16 row-major (K contiguous); lda >= K, lda * 2 a multiple of 16 bytes.
 *   W  [N][ldw] bf16 row-major, the [out][in] layout of a linear layer's weight; ldw >= K,
 *      ldw * 2 a multiple of 16 bytes.
 *   C  [M][ldc] c_dtype (bf16 or fp32) row-major; ldc >= N; must not overlap A or W.
 *   K  a positive multiple of 64; M, N >= 0 (any value: ragged tiles are masked).
 * A, W and C 16-byte aligned.  Accumulation is fp32 on the tensor cores (tcgen05);
 * the result is rounded once to c_dtype.  Needs an sm_103 device (KDA_ERR_UNSUPPORTED
 * otherwise).  A wait that times out on the device is reported through d_status
 * (KDA_ERR_TIMEOUT).
 * ------------------------------------------------------------------------ */
typedef enum { KDA_EPI_NONE = 0, KDA_EPI_DECAY = 1, KDA_EPI_SIGMOID = 2 } kda_epilogue;

typedef struct {
    int M, N, K;
    const void* A;         /* [M][lda] bf16 */
    int64_t lda;
    const void* W;         /* [N][ldw] bf16 */
    int64_t ldw;
    void* C;               /* [M][ldc] c_dtype */
    int64_t ldc;
    kda_dtype c_dtype;
    int epilogue;          /* kda_epilogue */
    int* d_status;         /* optional device int for device-side conditions */
} kda_gemm_args;

kda_status kda_gemm(const kda_gemm_args* args, kda_stream_t stream);

/* ------------------------------------------------------------------------
 * kda_backward -- the gradients of the layer (training).  Page "Kimi K3 /
 * Architecture": the model is trained, so kda_prefill's layer needs its
 * reverse-mode derivatives; page "Animated Kimi K3 architecture diagram",
 * LOCAL MEMORY section: each token's four moves are an affine map of the
 * state, whose adjoint runs the same moves backwards.
 *
 * Given dy = dL/d out and dS_fin = dL/d final_state of one kda_prefill call,
 * it returns dL/d of every input of that call:
 *
 *   dq, dk, dv      [T_total][H][D] fp32 (raw projections, before the conv)
 *   dconv_w         [3][H*D][4] fp32 (summed over all tokens and sequences)
 *   dg              [T_total][H][D] fp32;  dbeta  [T_total][H] fp32
 *   dgate           [T_total][H][D] fp32, or NULL (not wanted; 0 when gate is NULL)
 *   drms_w          [D] fp32, or NULL (computed as for weights of ones when rms_w is NULL)
 *   dinitial_state  [N][H][D][D] fp32, or NULL
 *   dconv_state_in  [N][3*H*D][3] fp32, or NULL (the gradient of the left padding
 *                   when conv_state_in is NULL)
 *
 * The forward is recomputed, not saved: `fwd` holds the kda_prefill arguments
 * (N, H, T_total, io, cu_seqlens and its host copy, q, k, v, qkv_row_stride,
 * conv_w, conv_state_in, g, beta, gate, rms_w, eps_l2, eps_rms, scale,
 * initial_state); out_dtype there is the dtype of dy.  Its out, final_state,
 * conv_state_out, chunk, flags and segments are ignored; its workspace and
 * workspace_bytes are this call's scratch (kda_backward_workspace_size).
 * Supported: D = 128, io bf16 or fp32; arithmetic is fp32 (the decays e^g
 * and the gate sigmoid through the IEEE functions, the recomputed SiLU and its
 * derivative through the fast exponential and reciprocal, a few ulp; the
 * chunk products on the tensor cores as three TF32 terms of hi/lo splits,
 * close to fp32), so the result does not depend on the forward's path.
 *
 * Method: conv + SiLU + L2 norms recomputed per token; for every 16-token
 * chunk, all at once, the parts that do not involve the state (decayed keys
 * and queries, the chunk's triangular products and (I + A)^-1); the
 * recurrence replayed chunk by chunk, saving o_t, e_t = v_t - S_bar^T k_t and
 * the state at the start of every 64-token segment; the epilogue's derivative
 * per row; the state gradient run backwards chunk by chunk, saving
 * w_t = dS^T k_t and the gradient at the end of every segment; then every
 * segment in parallel, chunk by chunk from its two checkpoints (with e and w
 * known): dq, dk and the log-decay's gradient, which follows from g entering
 * only through the decayed read keys and queries and the un-decayed written
 * keys; last the L2 norm's, SiLU's and the conv's derivatives.  No per-token
 * state is stored.
 *
 * Needs cu_seqlens_host (the checkpoint layout is planned on the host).  The
 * outputs must not overlap each other or any input.  dconv_w and drms_w are
 * zeroed by the call and accumulated with atomics, so their last bits depend
 * on the order blocks finish.  Every pointer 16-byte aligned except beta,
 * dbeta (4-byte).
 * ------------------------------------------------------------------------ */
typedef struct {
    kda_prefill_args fwd;       /* the forward call (see above) + this call's workspace */
    const void* dy;             /* [T_total][H][D] fwd.out_dtype */
    const float* d_final_state; /* [N][H][D][D] fp32, or NULL (zero) */
    float* dq;
    float* dk;
    float* dv;
    float* dconv_w;
    float* dg;
    float* dbeta;
    float* dgate;
    float* drms_w;
    float* dinitial_state;
    float* dconv_state_in;
} kda_backward_args;

/* Bytes of workspace kda_backward needs (reads fwd.N, H, D, T_total and
 * fwd.cu_seqlens_host, which is required), each part rounded up to 256:
 *   36 T_total H D + 8 T_total H + 8 slots D^2 + 8 slots D
 *   + 16 slots (49 D + 784) + 4 N H D + 8 (N + 1),
 * slots = H times the sum over sequences of ceil(len / 64): 6.6 GB for one
 * sequence of 8192 tokens with 96 heads. */
kda_status kda_backward_workspace_size(const kda_backward_args* args, size_t* bytes);

kda_status kda_backward(const kda_backward_args* args, kda_stream_t stream);

#ifdef __cplusplus
}
#endif

#endif /* KDA_H */
