// ep_permute / ep_unpermute: bf16 row movement of dispatch and combine.
//
// EPLB tutorial, "EPLB 和 DeepEP 怎么协同？": dispatch sends every token to the
// physical copy of each of its top-k experts; combine gathers the results back
// to their logical owner.  Here both are the local (single-GPU) halves: row
// copies between token order and per-instance grouped order.
//
// permute is written as a scatter by token: token t's row is read once and
// stored to the rows of its k slots.  Algorithmic traffic is therefore
// T rows read + T*k rows written; the gather form (one read per output row)
// would read every source row k times.  Rows of 1 KiB or more move with TMA
// bulk copies (permute_tma_kernel): every warp runs its own ring of
// shared-memory row buffers, its lane 0 issues one global->shared bulk copy
// per row (completion on an mbarrier) and k shared->global bulk copies out of
// the same buffer, so the copy engine, not the load/store units, moves the
// 8:1 write-heavy stream.  Shorter rows use a warp of 16-byte vector loads
// and streaming stores (permute_kernel).
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
        const int64_t inst = (tok < T) ? 0 : tok / T;
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
        const int64_t inst = (tok < T) ? 0 : tok / T;
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

// ---------------------------------------------------------------- TMA path
constexpr int kTmaWarps = 4;              // independent pipelines per block
constexpr int kStages = 6;                // row buffers per pipeline
constexpr int kSegMax = 8192;             // bytes per buffer (rows split above this)
constexpr int kTmaMinRow = 1024;          // shorter rows take the vector path
constexpr uint32_t kWaitLimit = 1u << 22; // mbarrier polls before giving up

__device__ __forceinline__ uint32_t smem_u32(const void* p) {
    return (uint32_t)__cvta_generic_to_shared(p);
}
__device__ __forceinline__ void mbar_init(uint64_t* bar, uint32_t count) {
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(bar)), "r"(count)
                 : "memory");
}
__device__ __forceinline__ void fence_mbar_init() {
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}
__device__ __forceinline__ void mbar_expect_tx(uint64_t* bar, uint32_t bytes) {
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_u32(bar)),
                 "r"(bytes)
                 : "memory");
}
__device__ __forceinline__ bool mbar_try_wait(uint64_t* bar, uint32_t parity) {
    uint32_t ok;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(ok)
        : "r"(smem_u32(bar)), "r"(parity)
        : "memory");
    return ok != 0;
}
// bounded wait on one phase of an mbarrier; false when the limit was reached
__device__ __forceinline__ bool mbar_wait(uint64_t* bar, uint32_t parity) {
    for (uint32_t n = 0; n < kWaitLimit; ++n)
        if (mbar_try_wait(bar, parity)) return true;
    return false;
}
__device__ __forceinline__ void bulk_g2s(void* sdst, const void* gsrc, uint32_t bytes,
                                         uint64_t* bar) {
    asm volatile(
        "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::
            "r"(smem_u32(sdst)),
        "l"(gsrc), "r"(bytes), "r"(smem_u32(bar))
        : "memory");
}
__device__ __forceinline__ void bulk_s2g(void* gdst, const void* ssrc, uint32_t bytes) {
    asm volatile("cp.async.bulk.global.shared::cta.bulk_group [%0], [%1], %2;" ::"l"(gdst),
                 "r"(smem_u32(ssrc)), "r"(bytes)
                 : "memory");
}
__device__ __forceinline__ void bulk_commit() {
    asm volatile("cp.async.bulk.commit_group;" ::: "memory");
}
// all but the newest committed group have finished reading shared memory
__device__ __forceinline__ void bulk_wait_read_all_but_one() {
    asm volatile("cp.async.bulk.wait_group.read 1;" ::: "memory");
}
__device__ __forceinline__ void bulk_wait_all() {
    asm volatile("cp.async.bulk.wait_group 0;" ::: "memory");
}

// One unit = one segment (<= kSegMax bytes) of one token's row.  Warp w of the
// grid handles units w, w + nw, w + 2nw, ...; unit i of the warp lives in
// buffer i % kStages, whose mbarrier completes phase (i / kStages) & 1.
__global__ void __launch_bounds__(kTmaWarps * 32, 1)
permute_tma_kernel(const char* __restrict__ hidden, int64_t n_tok, int64_t T, int k,
                   int rowbytes, int seg, int n_seg, const int32_t* __restrict__ dst_row,
                   char* __restrict__ out, int64_t N, int32_t* dev_status) {
    extern __shared__ __align__(128) unsigned char ring_all[];
    __shared__ __align__(8) uint64_t bars[kTmaWarps][kStages];
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    unsigned char* ring = ring_all + (size_t)warp * kStages * seg;
    uint64_t* bar = bars[warp];
    if (lane == 0) {
        for (int b = 0; b < kStages; ++b) mbar_init(&bar[b], 1);
        fence_mbar_init();
    }
    __syncwarp();

    const int64_t n_units = n_tok * n_seg;
    const int64_t gw = (int64_t)blockIdx.x * kTmaWarps + warp;
    const int64_t nw = (int64_t)gridDim.x * kTmaWarps;
    const int64_t my_n = gw < n_units ? (n_units - 1 - gw) / nw + 1 : 0;

    // unit -> (token, segment); one row segment is the common case
    auto split = [&](int64_t u, int64_t& tok, int& sg) {
        if (n_seg == 1) {
            tok = u;
            sg = 0;
        } else {
            tok = u / n_seg;
            sg = (int)(u - tok * n_seg);
        }
    };
    // lane 0: issue the load of the warp's unit i into its buffer
    auto issue_load = [&](int64_t i) {
        const int64_t u = gw + i * nw;
        int64_t tok;
        int sg;
        split(u, tok, sg);
        const uint32_t len = (uint32_t)min(seg, rowbytes - sg * seg);
        const int b = (int)(i % kStages);
        mbar_expect_tx(&bar[b], len);
        bulk_g2s(ring + (size_t)b * seg, hidden + tok * rowbytes + (int64_t)sg * seg, len, &bar[b]);
    };
    int64_t issued = 0;  // lane 0: loads issued so far (units 0 .. issued-1)
    if (lane == 0)
        for (; issued < my_n && issued < kStages; ++issued) issue_load(issued);

    bool range_err = false;
    int timed_out = 0;
    int64_t i = 0;
    for (; i < my_n; ++i) {
        const int64_t u = gw + i * nw;
        int64_t tok;
        int sg;
        split(u, tok, sg);
        const uint32_t len = (uint32_t)min(seg, rowbytes - sg * seg);
        const int b = (int)(i % kStages);
        int d = -1;
        if (lane < k) {
            d = __ldg(dst_row + tok * k + lane);
            if (d >= N) {
                range_err = true;
                d = -1;
            }
        }
        if (lane == 0) timed_out = mbar_wait(&bar[b], (uint32_t)((i / kStages) & 1)) ? 0 : 1;
        if (__shfl_sync(kFull, timed_out, 0)) break;
        const int64_t inst = (tok < T) ? 0 : tok / T;
        char* obase = out + (inst * N) * (int64_t)rowbytes + (int64_t)sg * seg;
        for (int j = 0; j < k; ++j) {
            const int dj = __shfl_sync(kFull, d, j);
            if (lane == 0 && dj >= 0) bulk_s2g(obase + (int64_t)dj * rowbytes, ring + (size_t)b * seg, len);
        }
        if (lane == 0) {
            bulk_commit();
            // the buffer of unit i-1 is refilled once its stores have read it
            if (i >= 1 && issued < my_n) {
                bulk_wait_read_all_but_one();
                issue_load(issued);
                ++issued;
            }
        }
        __syncwarp();
    }
    // After a timeout no further load is issued (the loop above stops before
    // its next issue_load); the loads already in flight are waited for, again
    // with a bound, before the block's shared memory is released.  If one of
    // them does not complete either, the block still exits and says so.
    int undrained = 0;
    if (lane == 0) {
        bulk_wait_all();
        for (int64_t x = i; x < issued; ++x)
            if (!mbar_wait(&bar[x % kStages], (uint32_t)((x / kStages) & 1))) undrained = 1;
    }
    const bool to = __shfl_sync(kFull, timed_out, 0) != 0;
    const bool ud = __shfl_sync(kFull, undrained, 0) != 0;
    const int flags = (__any_sync(kFull, range_err) ? EP_DEV_ROW_RANGE : 0) |
                      (to ? EP_DEV_COPY_TIMEOUT : 0) | (ud ? EP_DEV_COPY_UNDRAINED : 0);
    if (lane == 0 && flags) raise_flag(dev_status, flags);
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
    const int rowbytes = Hd * 2;
    if (rowbytes >= kTmaMinRow) {
        const int seg = rowbytes <= kSegMax ? rowbytes : kSegMax;
        const int n_seg = (rowbytes + seg - 1) / seg;
        const size_t smem = (size_t)kTmaWarps * kStages * seg;
        cudaError_t err = cudaFuncSetAttribute(permute_tma_kernel,
                                               cudaFuncAttributeMaxDynamicSharedMemorySize,
                                               (int)smem);
        if (err != cudaSuccess) return err;
        const int64_t units = n_tok * n_seg;
        const int64_t per_block = kTmaWarps;
        int64_t grid = device_info().sms;
        if (grid > (units + per_block - 1) / per_block) grid = (units + per_block - 1) / per_block;
        permute_tma_kernel<<<(unsigned)grid, kTmaWarps * 32, smem, s>>>(
            static_cast<const char*>(hidden), n_tok, T, k, rowbytes, seg, n_seg, dst_row,
            static_cast<char*>(out), T * k, dev_status);
        return cudaGetLastError();
    }
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
