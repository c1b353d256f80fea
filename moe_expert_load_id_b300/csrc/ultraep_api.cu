// C-ABI entry points of libultraep_b300: argument checks, then kernel launches.
// Every check here is host-side and happens before anything is enqueued.
#include <cstdint>
#include <mutex>

#include "common.cuh"

namespace ultraep {

DeviceInfo device_info() {
    static std::mutex mu;
    static DeviceInfo cache[64];
    static bool have[64] = {};
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return DeviceInfo{148, 227 * 1024};
    std::lock_guard<std::mutex> lock(mu);
    if (!have[dev]) {
        int sms = 148, optin = 227 * 1024;
        cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
        cudaDeviceGetAttribute(&optin, cudaDevAttrMaxSharedMemoryPerBlockOptin, dev);
        cache[dev] = DeviceInfo{sms, (size_t)optin};
        have[dev] = true;
    }
    return cache[dev];
}

namespace {

bool aligned(const void* p, uintptr_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }

bool domain_ok(const ep_domain_t* d) {
    if (d == nullptr) return false;
    if (d->R < 1 || d->R > EP_MAX_R) return false;
    if (d->E < 1 || d->E > EP_MAX_E || d->E % d->R != 0) return false;
    if (d->S < 0) return false;
    if (d->E / d->R + d->S > EP_MAX_INSTANCES_PER_RANK) return false;
    if (d->k < 1 || d->k > EP_MAX_K || d->k > d->E) return false;
    return true;
}

bool slots_ok(int64_t T, int32_t k) { return T >= 0 && T * (int64_t)k < (int64_t(1) << 31); }

// a required int32 array: non-null (when it holds elements) and 4-byte aligned
bool arr_ok(const void* p, bool nonempty) {
    if (!nonempty) return p == nullptr || aligned(p, 4);
    return p != nullptr && aligned(p, 4);
}

ep_status_t from_cuda(cudaError_t e) { return e == cudaSuccess ? EP_OK : EP_ERR_CUDA; }

bool rows_ok(int64_t T, int32_t k, int32_t Hd, int32_t n_inst) {
    if (n_inst < 0 || Hd < 0 || Hd % 8 != 0) return false;
    if (k < 1 || k > EP_MAX_K || !slots_ok(T, k)) return false;
    if (Hd > (1 << 29)) return false;  // row bytes (2*Hd) stay an int
    return true;
}

}  // namespace
}  // namespace ultraep

using namespace ultraep;

extern "C" {

size_t ep_count_workspace_bytes(const ep_domain_t* dom, int64_t T, int32_t n_inst) {
    if (!domain_ok(dom) || !slots_ok(T, dom->k) || n_inst < 0) return 0;
    return count_workspace_bytes(*dom, T, n_inst);
}

ep_status_t ep_count(const ep_domain_t* dom, const int32_t* topk_ids, int64_t T, int32_t n_inst,
                     int32_t* counts, int32_t* counts_src, int32_t* dev_status, void* workspace,
                     size_t workspace_bytes, void* stream) {
    if (!domain_ok(dom) || !slots_ok(T, dom->k) || n_inst < 0) return EP_ERR_INVAL;
    const bool any = n_inst > 0;
    if (!arr_ok(topk_ids, any && T > 0) || !arr_ok(counts, any) || !arr_ok(counts_src, any) ||
        !arr_ok(dev_status, false) || (any && !aligned(workspace, 16)))
        return EP_ERR_INVAL;
    if (!any) return EP_OK;
    if (workspace == nullptr || workspace_bytes < count_workspace_bytes(*dom, T, n_inst))
        return EP_ERR_WORKSPACE;
    return from_cuda(launch_count(*dom, topk_ids, T, n_inst, counts, counts_src, dev_status,
                                  workspace, static_cast<cudaStream_t>(stream)));
}

ep_status_t ep_count_noalloc(const ep_domain_t* dom, const int32_t* topk_ids, int64_t T,
                             int32_t n_inst, int32_t* counts, int32_t* counts_src,
                             int32_t* dev_status, void* stream) {
    if (!domain_ok(dom) || !slots_ok(T, dom->k) || n_inst < 0) return EP_ERR_INVAL;
    const bool any = n_inst > 0;
    if (!arr_ok(topk_ids, any && T > 0) || !arr_ok(counts, any) || !arr_ok(counts_src, any) ||
        !arr_ok(dev_status, false))
        return EP_ERR_INVAL;
    if (!any) return EP_OK;
    if (count_workspace_bytes(*dom, T, n_inst) > count_noalloc_scratch_capacity())
        return EP_ERR_WORKSPACE;
    return from_cuda(launch_count_noalloc(*dom, topk_ids, T, n_inst, counts, counts_src,
                                          dev_status, static_cast<cudaStream_t>(stream)));
}

ep_status_t ep_plan(const ep_domain_t* dom, const int32_t* counts, int32_t n_inst,
                    int32_t max_iters, int32_t* quota, int32_t* slot_expert, int32_t* rank_load, int32_t* inst_ptr,
                    int32_t* inst_id, int32_t* inst_cum, int32_t* n_iter, int32_t* inst_status,
                    void* stream) {
    if (!domain_ok(dom) || n_inst < 0) return EP_ERR_INVAL;
    const bool any = n_inst > 0;
    if (!arr_ok(counts, any) || !arr_ok(quota, any) || !arr_ok(slot_expert, any && dom->S > 0) ||
        !arr_ok(rank_load, any) || !arr_ok(inst_ptr, any) || !arr_ok(inst_id, any) ||
        !arr_ok(inst_cum, any) || !arr_ok(n_iter, any) || !arr_ok(inst_status, any))
        return EP_ERR_INVAL;
    if (!any) return EP_OK;
    if (max_iters <= 0) max_iters = EP_PLAN_MAX_ITERS;
    return from_cuda(launch_plan(*dom, counts, n_inst, max_iters, 0, quota, slot_expert, rank_load, inst_ptr,
                                 inst_id, inst_cum, n_iter, inst_status,
                                 static_cast<cudaStream_t>(stream)));
}

ep_status_t ep_plan_ex(const ep_domain_t* dom, const int32_t* counts, int32_t n_inst,
                       int32_t max_iters, int32_t flags, int32_t* quota, int32_t* slot_expert,
                       int32_t* rank_load, int32_t* inst_ptr, int32_t* inst_id,
                       int32_t* inst_cum, int32_t* n_iter, int32_t* inst_status, void* stream) {
    if (!domain_ok(dom) || n_inst < 0 || (flags & ~(EP_PLAN_SKIP | EP_PLAN_RELEASE)) != 0)
        return EP_ERR_INVAL;
    const bool any = n_inst > 0;
    if (!arr_ok(counts, any) || !arr_ok(quota, any) || !arr_ok(slot_expert, any && dom->S > 0) ||
        !arr_ok(rank_load, any) || !arr_ok(inst_ptr, any) || !arr_ok(inst_id, any) ||
        !arr_ok(inst_cum, any) || !arr_ok(n_iter, any) || !arr_ok(inst_status, any))
        return EP_ERR_INVAL;
    if (!any) return EP_OK;
    if (max_iters <= 0) max_iters = EP_PLAN_MAX_ITERS;
    return from_cuda(launch_plan(*dom, counts, n_inst, max_iters, flags, quota, slot_expert,
                                 rank_load, inst_ptr, inst_id, inst_cum, n_iter, inst_status,
                                 static_cast<cudaStream_t>(stream)));
}

ep_status_t ep_reroute(const ep_domain_t* dom, const int32_t* topk_ids, int64_t T, int32_t n_inst,
                       const int32_t* counts_src, const int32_t* quota, const int32_t* inst_ptr,
                       const int32_t* inst_id, const int32_t* inst_cum, int32_t* dst_row,
                       int32_t* src_slot, int32_t* inst_offset, int32_t* dev_status,
                       void* stream) {
    if (!domain_ok(dom) || !slots_ok(T, dom->k) || n_inst < 0) return EP_ERR_INVAL;
    const bool any = n_inst > 0;
    const bool slots = any && T > 0;
    if (!arr_ok(topk_ids, slots) || !arr_ok(counts_src, any) || !arr_ok(quota, any) ||
        !arr_ok(inst_ptr, any) || !arr_ok(inst_id, any) || !arr_ok(inst_cum, any) ||
        !arr_ok(dst_row, slots) || !arr_ok(src_slot, false) || !arr_ok(inst_offset, any) ||
        !arr_ok(dev_status, false))
        return EP_ERR_INVAL;
    if (!any) return EP_OK;
    return from_cuda(launch_reroute(*dom, topk_ids, T, n_inst, counts_src, quota, inst_ptr,
                                    inst_id, inst_cum, dst_row, src_slot, inst_offset,
                                    dev_status, static_cast<cudaStream_t>(stream)));
}

ep_status_t ep_balance(const ep_domain_t* dom, const int32_t* topk_ids, int64_t T,
                       int32_t n_inst, int32_t max_iters, const ep_balance_out_t* out,
                       int32_t* dev_status, void* workspace, size_t workspace_bytes,
                       void* stream) {
    if (out == nullptr || !domain_ok(dom) || !slots_ok(T, dom->k) || n_inst < 0)
        return EP_ERR_INVAL;
    const bool any = n_inst > 0;
    const bool slots = any && T > 0;
    if (!arr_ok(topk_ids, slots) || !arr_ok(out->counts, any) || !arr_ok(out->counts_src, any) ||
        !arr_ok(out->quota, any) || !arr_ok(out->slot_expert, any && dom->S > 0) ||
        !arr_ok(out->rank_load, any) || !arr_ok(out->inst_ptr, any) ||
        !arr_ok(out->inst_id, any) || !arr_ok(out->inst_cum, any) || !arr_ok(out->n_iter, any) ||
        !arr_ok(out->inst_status, any) || !arr_ok(out->dst_row, slots) ||
        !arr_ok(out->src_slot, false) || !arr_ok(out->inst_offset, any) ||
        !arr_ok(dev_status, false) || (any && !aligned(workspace, 16)))
        return EP_ERR_INVAL;
    if (!any) return EP_OK;
    if (workspace == nullptr || workspace_bytes < count_workspace_bytes(*dom, T, n_inst))
        return EP_ERR_WORKSPACE;
    if (max_iters <= 0) max_iters = EP_PLAN_MAX_ITERS;
    const cudaStream_t s = static_cast<cudaStream_t>(stream);
    // count writes the per-source-rank rows only; the planner sums them into
    // counts (one launch fewer synchronisation points on the critical path)
    cudaError_t err = launch_count(*dom, topk_ids, T, n_inst, out->counts, out->counts_src,
                                   dev_status, workspace, s, /*rows_only=*/true);
    if (err != cudaSuccess) return EP_ERR_CUDA;
    err = launch_plan(*dom, out->counts, n_inst, max_iters, 0, out->quota, out->slot_expert,
                      out->rank_load, out->inst_ptr, out->inst_id, out->inst_cum, out->n_iter,
                      out->inst_status, s, /*pdl=*/true, out->counts_src);
    if (err != cudaSuccess) return EP_ERR_CUDA;
    return from_cuda(launch_reroute(*dom, topk_ids, T, n_inst, out->counts_src, out->quota,
                                    out->inst_ptr, out->inst_id, out->inst_cum, out->dst_row,
                                    out->src_slot, out->inst_offset, dev_status, s,
                                    /*pdl=*/true));
}

ep_status_t ep_permute(const void* hidden, int64_t T, int32_t k, int32_t Hd, int32_t n_inst,
                       const int32_t* dst_row, void* out, int32_t* dev_status, void* stream) {
    if (!rows_ok(T, k, Hd, n_inst)) return EP_ERR_INVAL;
    const bool rows = n_inst > 0 && T > 0;
    if (rows && Hd > 0 && (hidden == nullptr || out == nullptr || !aligned(hidden, 16) ||
                           !aligned(out, 16)))
        return EP_ERR_INVAL;
    if (!arr_ok(dst_row, rows) || !arr_ok(dev_status, false)) return EP_ERR_INVAL;
    if (!rows) return EP_OK;
    return from_cuda(launch_permute(hidden, T, k, Hd, n_inst, dst_row, out, dev_status,
                                    static_cast<cudaStream_t>(stream)));
}

ep_status_t ep_unpermute(const void* grouped, int64_t T, int32_t k, int32_t Hd, int32_t n_inst,
                         const int32_t* dst_row, void* y, int32_t* dev_status, void* stream) {
    if (!rows_ok(T, k, Hd, n_inst)) return EP_ERR_INVAL;
    const bool rows = n_inst > 0 && T > 0;
    if (rows && Hd > 0 && (grouped == nullptr || y == nullptr || !aligned(grouped, 16) ||
                           !aligned(y, 16)))
        return EP_ERR_INVAL;
    if (!arr_ok(dst_row, rows) || !arr_ok(dev_status, false)) return EP_ERR_INVAL;
    if (!rows) return EP_OK;
    return from_cuda(launch_unpermute(grouped, T, k, Hd, n_inst, dst_row, y, dev_status,
                                      static_cast<cudaStream_t>(stream)));
}

ep_status_t ep_combine(const void* grouped, int64_t T, int32_t k, int32_t Hd, int32_t n_inst,
                       const int32_t* dst_row, const float* weights, void* y,
                       int32_t* dev_status, void* stream) {
    if (!rows_ok(T, k, Hd, n_inst)) return EP_ERR_INVAL;
    const bool rows = n_inst > 0 && T > 0;
    if (rows && Hd > 0 && (grouped == nullptr || y == nullptr || !aligned(grouped, 16) ||
                           !aligned(y, 16)))
        return EP_ERR_INVAL;
    if (!arr_ok(dst_row, rows) || !arr_ok(weights, rows) || !arr_ok(dev_status, false))
        return EP_ERR_INVAL;
    if (!rows) return EP_OK;
    return from_cuda(launch_combine(grouped, T, k, Hd, n_inst, dst_row, weights, y, dev_status,
                                    static_cast<cudaStream_t>(stream)));
}

ep_status_t ep_stage(const ep_domain_t* dom, int32_t n_inst, const void* expert_w,
                     int64_t expert_bytes, const int32_t* slot_expert,
                     const int32_t* prev_slot_expert, void* slot_w, int32_t* dev_status,
                     void* stream) {
    if (!domain_ok(dom) || n_inst < 0 || expert_bytes < 0 || expert_bytes % 16 != 0)
        return EP_ERR_INVAL;
    const bool any = n_inst > 0 && dom->S > 0 && expert_bytes > 0;
    if (any && (expert_w == nullptr || slot_w == nullptr || !aligned(expert_w, 16) ||
                !aligned(slot_w, 16)))
        return EP_ERR_INVAL;
    if (!arr_ok(slot_expert, any) || !arr_ok(prev_slot_expert, false) ||
        !arr_ok(dev_status, false))
        return EP_ERR_INVAL;
    if (!any) return EP_OK;
    return from_cuda(launch_stage(*dom, n_inst, expert_w, expert_bytes, slot_expert,
                                  prev_slot_expert, slot_w, dev_status,
                                  static_cast<cudaStream_t>(stream)));
}

const char* ep_status_str(ep_status_t s) {
    switch (s) {
        case EP_OK: return "EP_OK";
        case EP_ERR_INVAL: return "EP_ERR_INVAL: invalid argument";
        case EP_ERR_ITER_LIMIT: return "EP_ERR_ITER_LIMIT: plan hit its iteration cap";
        case EP_ERR_BAD_ID: return "EP_ERR_BAD_ID: expert id outside [0, E)";
        case EP_ERR_WORKSPACE: return "EP_ERR_WORKSPACE: workspace missing or too small";
        case EP_ERR_CUDA: return "EP_ERR_CUDA: a CUDA launch failed";
    }
    return "unknown ep_status_t";
}

}  // extern "C"
