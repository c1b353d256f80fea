// ep_plan: the coupled replica-placement + per-instance quota solve.
//
// UltraEP article (m.youleyou.com), "key design" section, control-plane
// paragraph: the solver fixes the load (quota) every expert instance receives,
// each exploration step either instantiates a new replica or shifts load, and
// it runs warp-parallel; reserved-slot paragraph: a fixed set of spare slots
// per rank, nothing allocated at run time.
//
// The pages do not give the rule; this kernel implements the fixed rule
// documented in ultraep.h (hot = argmax load, its largest instance, cold =
// least-loaded eligible rank, q = min(quota, floor(gap/2)), global stop), and
// the variants of ep_plan_ex.
//
// One warp per (layer, microbatch) instance.  The moves form one serial
// chain, so the design goal is the shortest dependent path per move.  The
// state is a shared-memory table per warp (plan_dev.cuh): the quota of every
// physical instance, the expert of every spare slot, per expert the 64-bit
// mask of ranks holding it, and the loads in registers (lane l: ranks l and
// l+32).  hot and cold are each one redux.sync over a packed key (load << 6 |
// rank index, the index flipped for the max so that the lowest rank wins
// ties); totals of 2^25 and more take a two-collective path (redux on the
// load, then a ballot for the lowest rank that attains it).  The flag-free
// rule runs plan_moves_table, the variants plan_moves_table_flags; the
// logical->physical CSR is built from the same tables after the loop.
#include <climits>

#include "common.cuh"
#include "plan_dev.cuh"

namespace ultraep {
namespace {

constexpr int kPlanWarps = 4;

template <bool kTwo, bool kFlags>
__global__ void __launch_bounds__(kPlanWarps * 32, 1)
plan_kernel(const int32_t* __restrict__ counts, int n_inst, int R, int E, int S, int max_iters,
            int flags,
            int32_t* __restrict__ quota_out, int32_t* __restrict__ slot_out,
            int32_t* __restrict__ load_out, int32_t* __restrict__ ptr_out,
            int32_t* __restrict__ id_out, int32_t* __restrict__ cum_out,
            int32_t* __restrict__ iter_out, int32_t* __restrict__ status_out,
            const int32_t* __restrict__ counts_src, int32_t* __restrict__ counts_out) {
    extern __shared__ __align__(16) unsigned char smem[];
    __shared__ int csr_warp_tot[kPlanWarps];
    // in ep_balance this grid is a programmatic dependent of ep_count: wait for
    // its counts, then let the dependent reroute start its plan-independent
    // work (for a plain launch both are no-ops)
    pdl_wait();
    pdl_trigger();
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int g = blockIdx.x * kPlanWarps + warp;
    const int H = E / R, W = H + S, P = R * W;
    const size_t wbytes = plan_warp_bytes(R, E, S);
    // the instance's counts: counts_src summed over the source ranks by the
    // whole block (ep_balance, whose count stops at the per-rank rows), or
    // the counts input
    const int32_t* cnt = counts + (int64_t)g * E;
    if (counts_src != nullptr) {
        int32_t* csum0 = reinterpret_cast<int32_t*>(smem + wbytes - align16((size_t)E * 4));
        const int g0 = blockIdx.x * kPlanWarps;
        const int nb = min(kPlanWarps, n_inst - g0);
        const float invE = 1.0f / (float)E;
        for (int x = threadIdx.x; x < kPlanWarps * E; x += kPlanWarps * 32) {
            const int w = small_div(x, invE);
            csum0[w * (wbytes / 4) + (x - w * E)] = 0;
        }
        __syncthreads();
        // thread (column, row group): column c, rows rg, rg + G, ...; sixteen
        // loads in flight per thread, so a 64 x 128 instance is one round trip
        // to L2 (where ep_count just left the rows).  With E a multiple of 4
        // and the rows 16-byte aligned a column is four experts (int4 loads).
        constexpr int kThr = kPlanWarps * 32;
        constexpr int kU = 16;
        if ((E & 3) == 0 && (reinterpret_cast<uintptr_t>(counts_src) & 15u) == 0) {
            const int Q = E >> 2;
            const int G = max(1, kThr / Q);
            const float invQG = 1.0f / (float)(Q * G), invQ = 1.0f / (float)Q;
            for (int x = threadIdx.x; x < nb * Q * G; x += kThr) {
                const int wi = small_div(x, invQG), rem = x - wi * Q * G;
                const int rg = small_div(rem, invQ), c = rem - rg * Q;
                const int4* cs =
                    reinterpret_cast<const int4*>(counts_src + (int64_t)(g0 + wi) * R * E) + c;
                int4 t = make_int4(0, 0, 0, 0);
                for (int r0 = rg; r0 < R; r0 += kU * G) {
                    int4 v[kU];
#pragma unroll
                    for (int u = 0; u < kU; ++u) {
                        const int rr = r0 + u * G;
                        v[u] = (rr < R) ? __ldg(cs + (int64_t)rr * Q) : make_int4(0, 0, 0, 0);
                    }
#pragma unroll
                    for (int u = 0; u < kU; ++u) {
                        t.x += v[u].x;
                        t.y += v[u].y;
                        t.z += v[u].z;
                        t.w += v[u].w;
                    }
                }
                int32_t* to = csum0 + wi * (wbytes / 4) + 4 * c;
                atomicAdd(to, t.x);
                atomicAdd(to + 1, t.y);
                atomicAdd(to + 2, t.z);
                atomicAdd(to + 3, t.w);
            }
        } else {
            const int G = max(1, kThr / E);
            for (int x = threadIdx.x; x < nb * E * G; x += kThr) {
                const int wi = x / (E * G), rem = x - wi * E * G;
                const int rg = rem / E, e = rem - rg * E;
                const int32_t* cs = counts_src + (int64_t)(g0 + wi) * R * E + e;
                int t = 0;
                for (int r0 = rg; r0 < R; r0 += kU * G) {
                    int v[kU];
#pragma unroll
                    for (int u = 0; u < kU; ++u) {
                        const int rr = r0 + u * G;
                        v[u] = (rr < R) ? __ldg(cs + (int64_t)rr * E) : 0;
                    }
#pragma unroll
                    for (int u = 0; u < kU; ++u) t += v[u];
                }
                atomicAdd(&csum0[wi * (wbytes / 4) + e], t);
            }
        }
        __syncthreads();
        if (g < n_inst) {
            const int32_t* mine = csum0 + warp * (wbytes / 4);
            for (int e = lane; e < E; e += 32) counts_out[(int64_t)g * E + e] = mine[e];
            cnt = mine;
        }
    }
    // each warp solves its instance (idle warps of the block skip to the barrier)
    const int g0 = blockIdx.x * kPlanWarps;
    const int nb = min(kPlanWarps, n_inst - g0);  // instances of this block
    auto tables = [&](int w, int32_t*& q, int32_t*& slot, uint64_t*& holder, int32_t*& pos,
                      int32_t*& val, int32_t*& Ls) {
        unsigned char* base = smem + (size_t)w * wbytes;
        q = reinterpret_cast<int32_t*>(base);
        slot = reinterpret_cast<int32_t*>(base + align16((size_t)P * 4));
        holder = reinterpret_cast<uint64_t*>(base + align16((size_t)P * 4) +
                                             align16((size_t)R * S * 4));
        pos = reinterpret_cast<int32_t*>(reinterpret_cast<unsigned char*>(holder) +
                                         align16((size_t)E * 8));
        val = pos + align16((size_t)(E + 1) * 4) / 4;
        Ls = val + align16((size_t)(E + R * S) * 4) / 4;  // [64] loads (variants)
    };
    if (g < n_inst) {
        // counts must be >= 0 with a total below 2^31; otherwise the instance is
        // rejected (EP_ERR_INVAL) and its outputs describe the home-only placement
        long long tot = 0;
        int status = plan_check_counts(cnt, E, lane, tot);
        int32_t *q, *slot, *pos, *val, *Ls;
        uint64_t* holder;
        tables(warp, q, slot, holder, pos, val, Ls);
        int iters = 0;
        plan_table_solve<kTwo, kFlags>(cnt, R, E, S, max_iters, flags, tot, q, slot, holder, Ls,
                                       lane, quota_out + (int64_t)g * P,
                                       slot_out + (int64_t)g * R * S, load_out + (int64_t)g * R,
                                       iters, status);
        if (lane == 0) {
            iter_out[g] = iters;
            status_out[g] = status;
        }
    }
    __syncthreads();
    // logical -> physical CSR of every instance of the block, by the whole block
    // (home first, then replicas by ascending rank = ascending p)
    for (int wi = 0; wi < nb; ++wi) {
        int32_t *q, *slot, *pos, *val, *Ls;
        uint64_t* holder;
        tables(wi, q, slot, holder, pos, val, Ls);
        const int gi = g0 + wi;
        plan_csr_block<kPlanWarps * 32>(q, slot, holder, R, E, S, pos, val, csr_warp_tot,
                                        ptr_out + (int64_t)gi * (E + 1),
                                        id_out + (int64_t)gi * (E + R * S),
                                        cum_out + (int64_t)gi * (E + R * S));
    }
}
template <bool kTwo, bool kFlags>
cudaError_t launch_plan_k(const ep_domain_t& d, const int32_t* counts, int32_t n_inst,
                          int32_t max_iters, int32_t flags, int32_t* quota, int32_t* slot_expert,
                          int32_t* rank_load, int32_t* inst_ptr, int32_t* inst_id,
                          int32_t* inst_cum, int32_t* n_iter, int32_t* inst_status,
                          cudaStream_t s, bool pdl, const int32_t* counts_src) {
    const size_t smem = kPlanWarps * plan_warp_bytes(d.R, d.E, d.S);
    if (smem > 48 * 1024) {
        cudaError_t err = cudaFuncSetAttribute(plan_kernel<kTwo, kFlags>,
                                               cudaFuncAttributeMaxDynamicSharedMemorySize,
                                               (int)smem);
        if (err != cudaSuccess) return err;
    }
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)((n_inst + kPlanWarps - 1) / kPlanWarps));
    cfg.blockDim = dim3(kPlanWarps * 32);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = s;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = pdl ? 1 : 0;
    return cudaLaunchKernelEx(&cfg, plan_kernel<kTwo, kFlags>, counts, (int)n_inst, (int)d.R,
                              (int)d.E, (int)d.S, (int)max_iters, (int)flags, quota, slot_expert,
                              rank_load, inst_ptr, inst_id, inst_cum, n_iter, inst_status,
                              counts_src, const_cast<int32_t*>(counts));
}

}  // namespace

cudaError_t launch_plan(const ep_domain_t& d, const int32_t* counts, int32_t n_inst,
                        int32_t max_iters, int32_t flags, int32_t* quota, int32_t* slot_expert,
                        int32_t* rank_load, int32_t* inst_ptr, int32_t* inst_id,
                        int32_t* inst_cum, int32_t* n_iter, int32_t* inst_status,
                        cudaStream_t s, bool pdl, const int32_t* counts_src) {
    if (n_inst == 0) return cudaSuccess;
    const bool two = d.R > 32;  // lane l also owns rank l + 32
    if (flags != 0)
        return two ? launch_plan_k<true, true>(d, counts, n_inst, max_iters, flags, quota,
                                               slot_expert, rank_load, inst_ptr, inst_id, inst_cum,
                                               n_iter, inst_status, s, pdl, counts_src)
                   : launch_plan_k<false, true>(d, counts, n_inst, max_iters, flags, quota,
                                                slot_expert, rank_load, inst_ptr, inst_id,
                                                inst_cum, n_iter, inst_status, s, pdl, counts_src);
    return two ? launch_plan_k<true, false>(d, counts, n_inst, max_iters, flags, quota,
                                            slot_expert, rank_load, inst_ptr, inst_id, inst_cum,
                                            n_iter, inst_status, s, pdl, counts_src)
               : launch_plan_k<false, false>(d, counts, n_inst, max_iters, flags, quota,
                                             slot_expert, rank_load, inst_ptr, inst_id, inst_cum,
                                             n_iter, inst_status, s, pdl, counts_src);
}

}  // namespace ultraep
