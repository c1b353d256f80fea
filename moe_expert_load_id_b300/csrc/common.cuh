// Internal helpers shared by the sm_103a kernels of libultraep_b300.
#pragma once

#include <cstdint>
#include <cuda_runtime.h>

#include "ultraep.h"

namespace ultraep {

constexpr unsigned kFull = 0xffffffffu;

__device__ __forceinline__ unsigned lanemask_lt() {
    unsigned m;
    asm volatile("mov.u32 %0, %%lanemask_lt;" : "=r"(m));
    return m;
}

// Programmatic dependent launch.  pdl_wait blocks until the grid this one
// depends on has completed and its writes are visible; it returns at once
// when the kernel was launched without that dependency.  pdl_trigger lets a
// dependent grid start launching; it has no effect when none is waiting.
__device__ __forceinline__ void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
__device__ __forceinline__ void pdl_trigger() { asm volatile("griddepcontrol.launch_dependents;" ::: "memory"); }

// Set bits in the caller's device status word.
__device__ __forceinline__ void raise_flag(int32_t* dev_status, int32_t bits) {
    if (dev_status != nullptr) atomicOr(dev_status, bits);
}

// Source rank r of the simulated domain owns tokens [r*Tr, (r+1)*Tr), Tr = ceil(T/R).
__host__ __device__ __forceinline__ int64_t tokens_per_rank(int64_t T, int R) {
    return (T + R - 1) / R;
}

// ---------------------------------------------------------------- launchers
struct DeviceInfo {
    int sms;
    size_t smem_optin;
};
DeviceInfo device_info();

// count
int count_chunks_per_rank(const ep_domain_t& d, int64_t T, int32_t n_inst);
size_t count_workspace_bytes(const ep_domain_t& d, int64_t T, int32_t n_inst);
size_t count_ticket_bytes(int32_t n_inst);
// rows_only: write counts_src only (the planner of ep_balance sums the rows)
cudaError_t launch_count(const ep_domain_t& d, const int32_t* ids, int64_t T, int32_t n_inst,
                         int32_t* counts, int32_t* counts_src, int32_t* dev_status, void* ws,
                         cudaStream_t s, bool rows_only = false);
size_t count_noalloc_scratch_capacity();
cudaError_t launch_count_noalloc(const ep_domain_t& d, const int32_t* ids, int64_t T,
                                 int32_t n_inst, int32_t* counts, int32_t* counts_src,
                                 int32_t* dev_status, cudaStream_t s);

// plan
// counts_src non-null (ep_balance): every instance first sums counts_src over
// the source ranks into counts, then plans
cudaError_t launch_plan(const ep_domain_t& d, const int32_t* counts, int32_t n_inst,
                        int32_t max_iters, int32_t flags, int32_t* quota, int32_t* slot_expert, int32_t* rank_load,
                        int32_t* inst_ptr, int32_t* inst_id, int32_t* inst_cum, int32_t* n_iter,
                        int32_t* inst_status, cudaStream_t s, bool pdl = false,
                        const int32_t* counts_src = nullptr);

// reroute
cudaError_t launch_reroute(const ep_domain_t& d, const int32_t* ids, int64_t T, int32_t n_inst,
                           const int32_t* counts_src, const int32_t* quota,
                           const int32_t* inst_ptr, const int32_t* inst_id,
                           const int32_t* inst_cum, int32_t* dst_row, int32_t* src_slot,
                           int32_t* inst_offset, int32_t* dev_status, cudaStream_t s,
                           bool pdl = false);

// permute / unpermute
cudaError_t launch_permute(const void* hidden, int64_t T, int32_t k, int32_t Hd, int32_t n_inst,
                           const int32_t* dst_row, void* out, int32_t* dev_status,
                           cudaStream_t s);
cudaError_t launch_unpermute(const void* grouped, int64_t T, int32_t k, int32_t Hd,
                             int32_t n_inst, const int32_t* dst_row, void* y,
                             int32_t* dev_status, cudaStream_t s);

// combine
cudaError_t launch_combine(const void* grouped, int64_t T, int32_t k, int32_t Hd, int32_t n_inst,
                           const int32_t* dst_row, const float* weights, void* y,
                           int32_t* dev_status, cudaStream_t s);

// replica weight staging
cudaError_t launch_stage(const ep_domain_t& d, int32_t n_inst, const void* expert_w,
                         int64_t expert_bytes, const int32_t* slot_expert,
                         const int32_t* prev_slot_expert, void* slot_w, int32_t* dev_status,
                         cudaStream_t s);

}  // namespace ultraep
