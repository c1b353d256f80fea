// ep_combine: the gate-weighted combine, the step after unpermute.
//
// EPLB tutorial, "EPLB 和 DeepEP 怎么协同？": results computed on the physical
// copies return to their logical owner; the owner adds up its top-k expert
// outputs weighted by the gate.  Here the local half of that, fused with the
// gather:
//     y[t][:] = bf16( sum over j = 0 .. k-1 of w[t][j] * grouped[dst_row[t*k+j]][:] )
// in float32, every product and every partial sum rounded on its own
// (__fmul_rn / __fadd_rn: no fused multiply-add), in ascending j from +0.0,
// a slot without a row adding nothing; the sum goes to bf16 by
// round-to-nearest-even and any NaN is stored as 0x7FC0.
//
// One warp per token: lane l handles the 16-byte vectors l, l+32, ... of the
// row; for every vector it first issues the loads of up to eight expert rows
// (evict-first: each grouped row is read once), then accumulates them in
// order.  Traffic per token: k rows read, one row written (plus dst_row and
// the weights).
#include "common.cuh"

namespace ultraep {
namespace {

constexpr int kCombThreads = 256;
constexpr int kBatch = 8;  // expert rows in flight per lane

__device__ __forceinline__ float bf16_low(uint32_t w) { return __uint_as_float(w << 16); }
__device__ __forceinline__ float bf16_high(uint32_t w) { return __uint_as_float(w & 0xFFFF0000u); }

// float32 -> bf16 bits: round to nearest, ties to even; NaN -> 0x7FC0
__device__ __forceinline__ uint32_t to_bf16(float f) {
    const uint32_t u = __float_as_uint(f);
    if ((u & 0x7F800000u) == 0x7F800000u && (u & 0x007FFFFFu) != 0u) return 0x7FC0u;
    const uint32_t upper = u >> 16, lower = u & 0xFFFFu;
    const bool up = lower > 0x8000u || (lower == 0x8000u && (upper & 1u));
    return upper + (up ? 1u : 0u);
}

__device__ __forceinline__ void accumulate(float (&acc)[8], float w, const uint4& v) {
    acc[0] = __fadd_rn(acc[0], __fmul_rn(w, bf16_low(v.x)));
    acc[1] = __fadd_rn(acc[1], __fmul_rn(w, bf16_high(v.x)));
    acc[2] = __fadd_rn(acc[2], __fmul_rn(w, bf16_low(v.y)));
    acc[3] = __fadd_rn(acc[3], __fmul_rn(w, bf16_high(v.y)));
    acc[4] = __fadd_rn(acc[4], __fmul_rn(w, bf16_low(v.z)));
    acc[5] = __fadd_rn(acc[5], __fmul_rn(w, bf16_high(v.z)));
    acc[6] = __fadd_rn(acc[6], __fmul_rn(w, bf16_low(v.w)));
    acc[7] = __fadd_rn(acc[7], __fmul_rn(w, bf16_high(v.w)));
}

__global__ void __launch_bounds__(kCombThreads)
combine_kernel(const uint4* __restrict__ grouped, int64_t n_tok, int64_t T, int k, int vpr,
               const int32_t* __restrict__ dst_row, const float* __restrict__ weights,
               uint4* __restrict__ y, int64_t N, int32_t* dev_status) {
    const int lane = threadIdx.x & 31;
    const int64_t w0 = ((int64_t)blockIdx.x * kCombThreads + threadIdx.x) >> 5;
    const int64_t nw = ((int64_t)gridDim.x * kCombThreads) >> 5;
    const int nch = (vpr + 31) / 32;
    bool range_err = false;
    for (int64_t tok = w0; tok < n_tok; tok += nw) {
        const int64_t inst = (tok < T) ? 0 : tok / T;
        // lanes j < k hold slot j's row and weight (k <= 32)
        int d = -1;
        float wt = 0.0f;
        if (lane < k) {
            d = __ldg(dst_row + tok * k + lane);
            wt = __ldg(weights + tok * k + lane);
            if (d >= N) {
                range_err = true;
                d = -1;
            }
        }
        const uint4* gbase = grouped + inst * N * vpr;
        uint4* yrow = y + tok * vpr;
        for (int c = 0; c < nch; ++c) {  // warp-uniform trip count
            const int x = c * 32 + lane;
            const bool act = x < vpr;
            float acc[8] = {0.0f, 0.0f, 0.0f, 0.0f, 0.0f, 0.0f, 0.0f, 0.0f};
            for (int j0 = 0; j0 < k; j0 += kBatch) {
                uint4 v[kBatch];
                int dv[kBatch];
                float wv[kBatch];
#pragma unroll
                for (int u = 0; u < kBatch; ++u) {
                    const int j = j0 + u;
                    dv[u] = __shfl_sync(kFull, d, j & 31);
                    wv[u] = __shfl_sync(kFull, wt, j & 31);
                    if (j >= k) dv[u] = -1;
                    v[u] = (act && dv[u] >= 0) ? __ldcs(gbase + (int64_t)dv[u] * vpr + x)
                                               : make_uint4(0u, 0u, 0u, 0u);
                }
#pragma unroll
                for (int u = 0; u < kBatch; ++u)
                    if (dv[u] >= 0) accumulate(acc, wv[u], v[u]);  // same for every lane
            }
            if (act) {
                uint4 o;
                o.x = to_bf16(acc[0]) | (to_bf16(acc[1]) << 16);
                o.y = to_bf16(acc[2]) | (to_bf16(acc[3]) << 16);
                o.z = to_bf16(acc[4]) | (to_bf16(acc[5]) << 16);
                o.w = to_bf16(acc[6]) | (to_bf16(acc[7]) << 16);
                __stcs(yrow + x, o);
            }
        }
    }
    if (__any_sync(kFull, range_err) && lane == 0) raise_flag(dev_status, EP_DEV_ROW_RANGE);
}

}  // namespace

cudaError_t launch_combine(const void* grouped, int64_t T, int32_t k, int32_t Hd, int32_t n_inst,
                           const int32_t* dst_row, const float* weights, void* y,
                           int32_t* dev_status, cudaStream_t s) {
    const int64_t n_tok = (int64_t)n_inst * T;
    if (n_tok == 0 || Hd == 0) return cudaSuccess;
    const int vpr = Hd * 2 / 16;
    const DeviceInfo di = device_info();
    int per_sm = 0;
    if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, combine_kernel, kCombThreads, 0) !=
            cudaSuccess || per_sm < 1)
        per_sm = 1;
    const int64_t warps_per_block = kCombThreads / 32;
    int64_t grid = (int64_t)di.sms * per_sm;
    if (grid > (n_tok + warps_per_block - 1) / warps_per_block)
        grid = (n_tok + warps_per_block - 1) / warps_per_block;
    combine_kernel<<<(unsigned)grid, kCombThreads, 0, s>>>(
        static_cast<const uint4*>(grouped), n_tok, T, k, vpr, dst_row, weights,
        static_cast<uint4*>(y), T * k, dev_status);
    return cudaGetLastError();
}

}  // namespace ultraep
