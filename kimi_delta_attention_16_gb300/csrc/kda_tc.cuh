// kda_tc.cuh -- entry points of the tensor-core (tcgen05) prefill path.
#pragma once

#include <cuda.h>  // CUtensorMap (encoded through the runtime's driver entry point, no libcuda link)

#include "kda_internal.cuh"

namespace kda {

// Encodes a 2D tiled tensor map over a row-major [rows][cols] tensor of bf16 (or fp32)
// elements with row pitch row_bytes: boxes of box_c x box_r elements, zeros outside the
// tensor, the 128-byte swizzle or none.  False when the driver entry point is missing or
// rejects the arguments (base not 16-byte aligned, pitch not a multiple of 16, ...).
bool encode_tensor_map_2d(CUtensorMap* m, const void* base, bool fp32, uint64_t cols, uint64_t rows,
                          uint64_t row_bytes, uint32_t box_c, uint32_t box_r, bool swizzle128);

// True when the tensor-core path takes these arguments (D = 128, chunk = 64,
// bf16 inputs) and this device supports it.
bool tc_prefill_applies(const kda_prefill_args& a);

// How the tensor-core path cuts each sequence: P segments (1 = none); segment 0
// holds the fraction w / (w + P - 1) of the chunks, the others share the rest
// equally.  args.segments forces P (with w = 1: equal segments); otherwise
// (P, w) minimise a cost model of the launch (see tc_seg_choice).
struct SegChoice {
    int P;
    int w;
};
SegChoice tc_seg_choice(const kda_prefill_args& a);
int tc_segments(const kda_prefill_args& a);

// Scratch bytes the tensor-core path needs.
size_t tc_prefill_workspace(const kda_prefill_args& a);

// Enqueues the tensor-core prefill; `ws` has tc_prefill_workspace(a) bytes.
cudaError_t launch_tc_prefill(const kda_prefill_args& a, char* ws, cudaStream_t s);

// ---------------------------------------------------------------- segment-parallel scan
// Buffers of one segmented launch (P > 1), all in the caller's workspace.  A
// unit u = n * H + h is one (sequence, head).
struct SegPlan {
    int P;             // segments per unit; 1 = one CTA walks each whole sequence
    int w, wd;         // segment 0 takes the first ceil(nc * w / wd) of a sequence's nc chunks
    float* end_state;  // [units][P][D][D]: segment 0's end state, then B_s (zero-start runs)
    float* trans;      // [units][P][D][D]: M_s, the end states of the identity-start runs
    float* start;      // [units][P][D][D]: S_s, the composed start state of segment s >= 1
    float* o_loc;      // [T][H][D]: scale * o of the zero-start runs (tokens of segments >= 1)
    float* f_tr;       // [T][H][D]: scale * o of the identity-start runs, v = 0
};

// Chunks [cb, ce) of segment s when a sequence of nc chunks is cut into P
// segments: segment 0 is the first ceil(nc * w / wd) chunks, the others split
// the rest into runs of ceil(rest / (P - 1)) (trailing segments may be short or
// empty).  w = 1, wd = P gives P segments of about nc / P.
__host__ __device__ __forceinline__ void seg_chunk_range(int64_t nc, int P, int w, int wd, int s, int64_t& cb,
                                                         int64_t& ce) {
    if (P <= 1) {
        cb = 0;
        ce = nc;
        return;
    }
    const int64_t den = wd;
    int64_t c0 = (nc * w + den - 1) / den;
    c0 = c0 < nc ? c0 : nc;
    if (s == 0) {
        cb = 0;
        ce = c0;
        return;
    }
    const int64_t sl = (nc - c0 + P - 2) / (P - 1);
    const int64_t b = c0 + (int64_t)(s - 1) * sl;
    cb = b < nc ? b : nc;
    ce = cb + sl < nc ? cb + sl : nc;
}

// Composes, per unit and in segment order, S_1 = end_state[0] and
// S_{s+1} = M_s S_s + B_s (tensor cores); writes S_1 .. S_{P-1} to sp.start and
// S_P to S_fin (when non-NULL, [N][H][D][D]).  A tensor-core wait that times out
// sets KDA_ERR_TIMEOUT in d_status.
cudaError_t launch_seg_combine(const SegPlan& sp, int units, float* S_fin, int* d_status, cudaStream_t s);

// For every token of segments s >= 1: o = o_loc + S_s^T f (tensor cores), then
// y = RMSNorm(o) * rms_w * sigmoid(gate) -> out (bf16 or fp32 rows [T][H][D]).
// A tensor-core wait that times out sets KDA_ERR_TIMEOUT in d_status.
cudaError_t launch_seg_fixup(const SegPlan& sp, const int32_t* cu, int N, int64_t T_total, int H,
                             const bf16* gate, const float* rms_w, float eps_rms, void* out,
                             kda_dtype out_dt, int sms, int* d_status, cudaStream_t s);

}  // namespace kda
