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
// One warp per token, the row cut into chunks of 32 16-byte vectors (lane l
// handles vector l of a chunk).  An item is one chunk of up to eight of the
// token's expert rows; each lane copies its vectors of an item into shared
// memory with cp.async (16 bytes, no register held while in flight), four
// items deep, and accumulates the item that has landed.  Products and sums
// are the scalar __fmul_rn / __fadd_rn, which are never contracted into a
// fused multiply-add.  (The packed two-float mul.rn.f32x2 / add.rn.f32x2 were
// tried: ptxas fused them, -fmad=false notwithstanding, and the results
// differed on rounding ties.)  The bf16 conversion is the hardware
// round-to-nearest-even pair conversion, with a NaN result stored as 0x7FC0.  A lane reads only what its own copies wrote,
// so the pipeline needs no barrier.  Traffic per token: k rows read, one row
// written (plus dst_row and the weights).
#include "common.cuh"

namespace ultraep {
namespace {

constexpr int kCombWarps = 4;
constexpr int kCombThreads = kCombWarps * 32;
constexpr int kRowsPerItem = 8;
constexpr int kCombStages = 4;
constexpr size_t kCombSmem = (size_t)kCombWarps * kCombStages * kRowsPerItem * 32 * 16;

__device__ __forceinline__ uint32_t smem_addr(const void* p) {
    return (uint32_t)__cvta_generic_to_shared(p);
}
__device__ __forceinline__ void cp_async16(void* dst, const void* src) {
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(smem_addr(dst)), "l"(src)
                 : "memory");
}
__device__ __forceinline__ void cp_async_commit() {
    asm volatile("cp.async.commit_group;" ::: "memory");
}
// every group but the newest kCombStages - 2 has landed
__device__ __forceinline__ void cp_async_wait_item() {
    asm volatile("cp.async.wait_group %0;" ::"n"(kCombStages - 2) : "memory");
}

__device__ __forceinline__ float bf16_low(uint32_t w) { return __uint_as_float(w << 16); }
__device__ __forceinline__ float bf16_high(uint32_t w) { return __uint_as_float(w & 0xFFFF0000u); }

// acc[2h], acc[2h+1] += w * (the two bf16 of word v), each product and each
// sum rounded on its own
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

// two floats -> two bf16 (lo in the low half), round to nearest even; a NaN
// becomes 0x7FC0
__device__ __forceinline__ uint32_t to_bf16x2(float flo, float fhi) {
    const uint32_t lo = __float_as_uint(flo), hi = __float_as_uint(fhi);
    uint32_t r;
    asm("cvt.rn.bf16x2.f32 %0, %1, %2;" : "=r"(r) : "f"(fhi), "f"(flo));
    if ((lo & 0x7FFFFFFFu) > 0x7F800000u) r = (r & 0xFFFF0000u) | 0x7FC0u;
    if ((hi & 0x7FFFFFFFu) > 0x7F800000u) r = (r & 0x0000FFFFu) | 0x7FC00000u;
    return r;
}

__global__ void __launch_bounds__(kCombThreads)
combine_kernel(const uint4* __restrict__ grouped, int64_t n_tok, int64_t T, int k, int vpr,
               const int32_t* __restrict__ dst_row, const float* __restrict__ weights,
               uint4* __restrict__ y, int64_t N, int32_t* dev_status) {
    extern __shared__ __align__(16) uint4 cbuf[];
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    uint4* buf = cbuf + (size_t)warp * kCombStages * kRowsPerItem * 32;  // [stage][row][lane]
    const int64_t w0 = (int64_t)blockIdx.x * kCombWarps + warp;
    const int64_t nw = (int64_t)gridDim.x * kCombWarps;
    const int nch = (vpr + 31) / 32;
    const int nb = (k + kRowsPerItem - 1) / kRowsPerItem;  // row batches per chunk
    const int nit = nch * nb;                              // items per token
    bool range_err = false;
    for (int64_t tok = w0; tok < n_tok; tok += nw) {  // warp-uniform
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

        // copies of item it into stage it % kCombStages (always one commit,
        // so the group count per item is fixed)
        auto issue = [&](int it) {
            if (it < nit) {
                const int c = it / nb, b = it - c * nb;
                const int x = c * 32 + lane;
                uint4* st = buf + (size_t)(it % kCombStages) * kRowsPerItem * 32 + lane;
#pragma unroll
                for (int u = 0; u < kRowsPerItem; ++u) {
                    const int r = b * kRowsPerItem + u;
                    const int dr = __shfl_sync(kFull, d, r & 31);
                    if (r < k && dr >= 0 && x < vpr) cp_async16(st + u * 32, gbase + (int64_t)dr * vpr + x);
                }
            }
            cp_async_commit();
        };

#pragma unroll
        for (int it = 0; it < kCombStages - 1; ++it) issue(it);
        float acc[8];
        // this batch's rows: weights and which rows exist
        float wr[kRowsPerItem];
        unsigned has = 0u;
        for (int it = 0; it < nit; ++it) {  // warp-uniform
            issue(it + kCombStages - 1);
            cp_async_wait_item();
            const int c = it / nb, b = it - c * nb;
            const int x = c * 32 + lane;
            if (b == 0) {
#pragma unroll
                for (int h = 0; h < 8; ++h) acc[h] = 0.0f;
            }
            if (it < nb || nb > 1) {  // with k <= 8, once per token
                has = 0u;
#pragma unroll
                for (int u = 0; u < kRowsPerItem; ++u) {
                    const int r = b * kRowsPerItem + u;
                    const int dr = __shfl_sync(kFull, d, r & 31);
                    wr[u] = __shfl_sync(kFull, wt, r & 31);
                    has |= (r < k && dr >= 0) ? (1u << u) : 0u;
                }
            }
            if (x < vpr) {
                const uint4* st = buf + (size_t)(it % kCombStages) * kRowsPerItem * 32 + lane;
#pragma unroll
                for (int u = 0; u < kRowsPerItem; ++u) {
                    if ((has >> u) & 1u) {  // same for every lane
                        accumulate(acc, wr[u], st[u * 32]);
                    }
                }
                if (b == nb - 1) {
                    uint4 o;
                    o.x = to_bf16x2(acc[0], acc[1]);
                    o.y = to_bf16x2(acc[2], acc[3]);
                    o.z = to_bf16x2(acc[4], acc[5]);
                    o.w = to_bf16x2(acc[6], acc[7]);
                    __stcs(yrow + x, o);
                }
            }
        }
    }
    asm volatile("cp.async.wait_all;" ::: "memory");
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
    cudaError_t err = cudaFuncSetAttribute(combine_kernel,
                                           cudaFuncAttributeMaxDynamicSharedMemorySize,
                                           (int)kCombSmem);
    if (err != cudaSuccess) return err;
    int per_sm = 0;
    if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, combine_kernel, kCombThreads,
                                                      kCombSmem) != cudaSuccess ||
        per_sm < 1)
        per_sm = 1;
    int64_t grid = (int64_t)di.sms * per_sm;
    if (grid > (n_tok + kCombWarps - 1) / kCombWarps) grid = (n_tok + kCombWarps - 1) / kCombWarps;
    combine_kernel<<<(unsigned)grid, kCombThreads, kCombSmem, s>>>(
        static_cast<const uint4*>(grouped), n_tok, T, k, vpr, dst_row, weights,
        static_cast<uint4*>(y), T * k, dev_status);
    return cudaGetLastError();
}

}  // namespace ultraep
