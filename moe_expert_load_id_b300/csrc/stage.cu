// ep_stage: replica weight staging, the single-GPU half of weight distribution.
//
// UltraEP article (m.youleyou.com), "key design" section, forward-pass
// paragraph: after planning, the replicas' expert weights are distributed to
// the ranks hosting them; reserved-slot paragraph: the redundant slots are
// fixed buffers, reused across layers.  Here every spare slot x = r*S + s of
// every instance whose expert e = slot_expert[x] is valid (and, when the
// previous contents are given, differs from them) receives a copy of the
// expert's weights:  slot_w[x][:] = expert_w[e][:].
//
// A copy of whole rows: one warp per 64 KB chunk of a slot, 16-byte
// streaming loads and stores, eight in flight per lane.
#include "common.cuh"

namespace ultraep {
namespace {

constexpr int kStageThreads = 256;
constexpr int64_t kChunkVec = (64 * 1024) / 16;  // 16-byte vectors per chunk
constexpr int kInFlight = 8;

__global__ void __launch_bounds__(kStageThreads)
stage_kernel(const uint4* __restrict__ expert_w, int E, int64_t vpe, int nslot, int64_t cps,
             int64_t units, const int32_t* __restrict__ slot_expert,
             const int32_t* __restrict__ prev, uint4* __restrict__ slot_w, int32_t* dev_status) {
    const int lane = threadIdx.x & 31;
    const int64_t w0 = ((int64_t)blockIdx.x * kStageThreads + threadIdx.x) >> 5;
    const int64_t nw = ((int64_t)gridDim.x * kStageThreads) >> 5;
    bool bad = false;
    for (int64_t u = w0; u < units; u += nw) {
        const int64_t sc = u / cps;               // (instance, slot)
        const int64_t c = u - sc * cps;           // chunk of that slot
        const int64_t inst = sc / nslot;
        const int32_t e = slot_expert[sc];
        if (e == -1) continue;                    // empty slot
        if (e < -1 || e >= E) {                   // invalid id: flagged once per slot
            bad |= (c == 0);
            continue;
        }
        if (prev != nullptr && prev[sc] == e) continue;  // already holds e
        const int64_t v0 = c * kChunkVec;
        const int64_t n = min(kChunkVec, vpe - v0);
        const uint4* src = expert_w + ((int64_t)inst * E + e) * vpe + v0;
        uint4* dst = slot_w + sc * vpe + v0;
        for (int64_t i0 = 0; i0 < n; i0 += 32 * kInFlight) {
            uint4 v[kInFlight];
#pragma unroll
            for (int q = 0; q < kInFlight; ++q) {
                const int64_t i = i0 + q * 32 + lane;
                if (i < n) v[q] = __ldcs(src + i);
            }
#pragma unroll
            for (int q = 0; q < kInFlight; ++q) {
                const int64_t i = i0 + q * 32 + lane;
                if (i < n) __stcs(dst + i, v[q]);
            }
        }
    }
    if (bad && lane == 0) raise_flag(dev_status, EP_DEV_BAD_ID);
}

}  // namespace

cudaError_t launch_stage(const ep_domain_t& d, int32_t n_inst, const void* expert_w,
                         int64_t expert_bytes, const int32_t* slot_expert,
                         const int32_t* prev_slot_expert, void* slot_w, int32_t* dev_status,
                         cudaStream_t s) {
    const int nslot = d.R * d.S;
    const int64_t vpe = expert_bytes / 16;
    if (n_inst == 0 || nslot == 0 || vpe == 0) return cudaSuccess;
    const int64_t cps = (vpe + kChunkVec - 1) / kChunkVec;
    const int64_t units = (int64_t)n_inst * nslot * cps;
    const DeviceInfo di = device_info();
    int per_sm = 0;
    if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, stage_kernel, kStageThreads, 0) !=
            cudaSuccess || per_sm < 1)
        per_sm = 1;
    const int64_t warps_per_block = kStageThreads / 32;
    int64_t grid = (int64_t)di.sms * per_sm;
    if (grid > (units + warps_per_block - 1) / warps_per_block)
        grid = (units + warps_per_block - 1) / warps_per_block;
    stage_kernel<<<(unsigned)grid, kStageThreads, 0, s>>>(
        static_cast<const uint4*>(expert_w), d.E, vpe, nslot, cps, units, slot_expert,
        prev_slot_expert, static_cast<uint4*>(slot_w), dev_status);
    return cudaGetLastError();
}

}  // namespace ultraep
