// ep_permute / ep_unpermute: bf16 row movement of dispatch and combine.
//
// EPLB tutorial, "EPLB 和 DeepEP 怎么协同？": dispatch sends every token to the
// physical copy of each of its top-k experts; combine gathers the results back
// to their logical owner.  Here both are the local (single-GPU) halves: row
// copies between token order and per-instance grouped order.
//
// permute is written as a scatter by token: a warp reads token t's row once
// (16-byte vector loads, evict-first) and stores it to the rows of its k
// slots (16-byte streaming stores).  Algorithmic traffic is therefore
// T rows read + T*k rows written; the gather form (one read per output row)
// would read every source row k times.
//
// unpermute is a gather: for each slot (t, j) the warp copies grouped row
// dst_row[t*k+j] into y[t][j]; y is written contiguously.
#include "common.cuh"

namespace ultraep {
namespace {

constexpr int kMoveThreads = 256;
constexpr int kUnroll = 4;  // 16-byte vectors per lane per step

__global__ void __launch_bounds__(kMoveThreads)
permute_kernel(const uint4* __restrict__ hidden, int64_t n_tok, int64_t T, int k, int vpr,
               const int32_t* __restrict__ dst_row, uint4* __restrict__ out, int64_t N,
               int32_t* dev_status) {
    const int lane = threadIdx.x & 31;
    const int64_t w0 = ((int64_t)blockIdx.x * kMoveThreads + threadIdx.x) >> 5;
    const int64_t nw = ((int64_t)gridDim.x * kMoveThreads) >> 5;
    bool range_err = false;
    for (int64_t tok = w0; tok < n_tok; tok += nw) {
        const int64_t inst = tok / T;
        int d = -1;
        if (lane < k) {
            d = __ldcs(dst_row + tok * k + lane);
            if (d >= N) {
                range_err = true;
                d = -1;
            }
        }
        const uint4* src = hidden + tok * vpr;
        uint4* obase = out + inst * N * vpr;
        for (int c0 = 0; c0 < vpr; c0 += 32 * kUnroll) {
            uint4 v[kUnroll];
#pragma unroll
            for (int u = 0; u < kUnroll; ++u) {
                const int x = c0 + u * 32 + lane;
                if (x < vpr) v[u] = __ldcs(src + x);
            }
            for (int j = 0; j < k; ++j) {
                const int dj = __shfl_sync(kFull, d, j);
                if (dj < 0) continue;
                uint4* o = obase + (int64_t)dj * vpr;
#pragma unroll
                for (int u = 0; u < kUnroll; ++u) {
                    const int x = c0 + u * 32 + lane;
                    if (x < vpr) __stcs(o + x, v[u]);
                }
            }
        }
    }
    if (__any_sync(kFull, range_err) && lane == 0) raise_flag(dev_status, EP_DEV_ROW_RANGE);
}

__global__ void __launch_bounds__(kMoveThreads)
unpermute_kernel(const uint4* __restrict__ grouped, int64_t n_tok, int64_t T, int k, int vpr,
                 const int32_t* __restrict__ dst_row, uint4* __restrict__ y, int64_t N,
                 int32_t* dev_status) {
    const int lane = threadIdx.x & 31;
    const int64_t w0 = ((int64_t)blockIdx.x * kMoveThreads + threadIdx.x) >> 5;
    const int64_t nw = ((int64_t)gridDim.x * kMoveThreads) >> 5;
    bool range_err = false;
    const uint4 zero = make_uint4(0u, 0u, 0u, 0u);
    for (int64_t tok = w0; tok < n_tok; tok += nw) {
        const int64_t inst = tok / T;
        int d = -1;
        if (lane < k) {
            d = __ldcs(dst_row + tok * k + lane);
            if (d >= N) {
                range_err = true;
                d = -1;
            }
        }
        const uint4* gbase = grouped + inst * N * vpr;
        uint4* ybase = y + tok * k * (int64_t)vpr;
        for (int j = 0; j < k; ++j) {
            const int dj = __shfl_sync(kFull, d, j);
            const uint4* srow = gbase + (int64_t)(dj < 0 ? 0 : dj) * vpr;
            uint4* yrow = ybase + (int64_t)j * vpr;
            for (int c0 = 0; c0 < vpr; c0 += 32 * kUnroll) {
                uint4 v[kUnroll];
#pragma unroll
                for (int u = 0; u < kUnroll; ++u) {
                    const int x = c0 + u * 32 + lane;
                    v[u] = (x < vpr && dj >= 0) ? __ldcs(srow + x) : zero;
                }
#pragma unroll
                for (int u = 0; u < kUnroll; ++u) {
                    const int x = c0 + u * 32 + lane;
                    if (x < vpr) __stcs(yrow + x, v[u]);
                }
            }
        }
    }
    if (__any_sync(kFull, range_err) && lane == 0) raise_flag(dev_status, EP_DEV_ROW_RANGE);
}

int grid_for(const void* kernel, int64_t n_tok) {
    const DeviceInfo di = device_info();
    int per_sm = 0;
    if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, kernel, kMoveThreads, 0) !=
            cudaSuccess || per_sm < 1)
        per_sm = 1;
    const int64_t full = (int64_t)di.sms * per_sm;
    const int64_t need = (n_tok + (kMoveThreads / 32) - 1) / (kMoveThreads / 32);
    return (int)(need < full ? need : full);
}

}  // namespace

cudaError_t launch_permute(const void* hidden, int64_t T, int32_t k, int32_t Hd, int32_t n_inst,
                           const int32_t* dst_row, void* out, int32_t* dev_status,
                           cudaStream_t s) {
    const int64_t n_tok = (int64_t)n_inst * T;
    if (n_tok == 0 || Hd == 0) return cudaSuccess;
    const int vpr = Hd * 2 / 16;
    const int grid = grid_for((const void*)permute_kernel, n_tok);
    permute_kernel<<<grid, kMoveThreads, 0, s>>>(static_cast<const uint4*>(hidden), n_tok, T, k,
                                                 vpr, dst_row, static_cast<uint4*>(out), T * k,
                                                 dev_status);
    return cudaGetLastError();
}

cudaError_t launch_unpermute(const void* grouped, int64_t T, int32_t k, int32_t Hd,
                             int32_t n_inst, const int32_t* dst_row, void* y,
                             int32_t* dev_status, cudaStream_t s) {
    const int64_t n_tok = (int64_t)n_inst * T;
    if (n_tok == 0 || Hd == 0) return cudaSuccess;
    const int vpr = Hd * 2 / 16;
    const int grid = grid_for((const void*)unpermute_kernel, n_tok);
    unpermute_kernel<<<grid, kMoveThreads, 0, s>>>(static_cast<const uint4*>(grouped), n_tok, T,
                                                   k, vpr, dst_row, static_cast<uint4*>(y),
                                                   T * k, dev_status);
    return cudaGetLastError();
}

}  // namespace ultraep
