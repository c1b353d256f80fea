// ep_reroute: stable quota-prefix assignment of every (token, k) slot to a
// physical instance of its logical expert.
//
// UltraEP article (m.youleyou.com), "key design" section, forward-pass
// paragraph: reroute splits the tokens of one logical expert among its
// copies.  EPLB tutorial, "EPLB 和 DeepEP 怎么协同？": dispatch maps every top-k
// logical id to one physical copy.
//
// The within-expert rank of a slot is the number of earlier slots (smaller
// t*k+j) with the same expert.  With the slots of source rank r handled by one
// block, that rank is
//     (slots of e on source ranks < r)         from counts_src, an exclusive
//                                              prefix over r (no extra pass)
//   + (slots of e earlier in this rank)        running per-expert base
//   + (slots of e in earlier warps of a chunk) per-expert scan over warps
//   + (lanes below in the same 32-slot step)   popc(match.any group & lanemask_lt)
// A slot of rank x goes to the first instance of e's list whose inclusive
// cumulative quota exceeds x, at row  inst_offset[p] + x - (cum before p),
// i.e. x + delta[m] with delta precomputed per list entry.
//
// ids are read once from memory (kept in registers between the histogram and
// the assignment phase of a chunk); dst_row is written with coalesced
// streaming stores; the optional src_slot inverse is a scattered store.
#include <climits>

#include "common.cuh"

namespace ultraep {
namespace {

constexpr int kRrThreads = 512;
constexpr int kRrWarps = kRrThreads / 32;
constexpr int kItems = 8;  // 32-slot steps per warp per chunk
constexpr int kChunk = kRrThreads * kItems;

struct RrLayout {
    int P, M;  // instances, CSR capacity
    size_t bytes;
};

__host__ __device__ inline RrLayout rr_layout(int R, int E, int S) {
    RrLayout l;
    l.P = R * (E / R + S);
    l.M = E + R * S;
    // off[P+1] ptr[E+1] bcum[M] bdel[M] base[E] wcnt[kRrWarps][E]
    l.bytes = sizeof(int32_t) * ((size_t)(l.P + 1) + (E + 1) + 2 * (size_t)l.M + E +
                                 (size_t)kRrWarps * E);
    return l;
}

__global__ void __launch_bounds__(kRrThreads)
reroute_kernel(const int32_t* __restrict__ ids, int64_t T, int k, int R, int E, int S,
               const int32_t* __restrict__ counts_src, const int32_t* __restrict__ quota,
               const int32_t* __restrict__ inst_ptr, const int32_t* __restrict__ inst_id,
               const int32_t* __restrict__ inst_cum, int32_t* __restrict__ dst_row,
               int32_t* __restrict__ src_slot, int32_t* __restrict__ inst_offset,
               int32_t* dev_status) {
    extern __shared__ __align__(16) int32_t sm[];
    __shared__ int32_t warp_tot[kRrWarps];
    __shared__ int32_t flags;

    const RrLayout lay = rr_layout(R, E, S);
    const int P = lay.P, M = lay.M;
    int32_t* off = sm;              // [P+1] first row of each instance
    int32_t* ptr = off + (P + 1);   // [E+1] CSR row pointers (clamped)
    int32_t* bcum = ptr + (E + 1);  // [M]   inclusive cumulative quota
    int32_t* bdel = bcum + M;       // [M]   row - within-expert rank
    int32_t* base = bdel + M;       // [E]   running within-expert rank
    int32_t* wcnt = base + E;       // [kRrWarps][E]

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int inst = blockIdx.x / R, r = blockIdx.x % R;
    const int32_t* qg = quota + (int64_t)inst * P;
    if (tid == 0) flags = 0;

    // ---- inst_offset: exclusive prefix of quota over p (P <= 2048, 4 per thread)
    {
        constexpr int kIpt = 4;
        const int i0 = tid * kIpt;
        int v[kIpt];
        int local = 0;
#pragma unroll
        for (int u = 0; u < kIpt; ++u) {
            v[u] = (i0 + u < P) ? qg[i0 + u] : 0;
            local += v[u];
        }
        int x = local;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const int y = __shfl_up_sync(kFull, x, o);
            if (lane >= o) x += y;
        }
        if (lane == 31) warp_tot[warp] = x;
        __syncthreads();
        if (warp == 0) {
            int w = (lane < kRrWarps) ? warp_tot[lane] : 0;
#pragma unroll
            for (int o = 1; o < 32; o <<= 1) {
                const int y = __shfl_up_sync(kFull, w, o);
                if (lane >= o) w += y;
            }
            if (lane < kRrWarps) warp_tot[lane] = w;  // inclusive over warps
        }
        __syncthreads();
        int run = x - local + (warp > 0 ? warp_tot[warp - 1] : 0);
#pragma unroll
        for (int u = 0; u < kIpt; ++u) {
            if (i0 + u < P) off[i0 + u] = run;
            run += v[u];
        }
        if (tid == kRrThreads - 1) off[P] = warp_tot[kRrWarps - 1];
    }
    // ---- CSR pointers, per-expert base from earlier source ranks, zero warp counters
    const int32_t* pg = inst_ptr + (int64_t)inst * (E + 1);
    for (int e = tid; e <= E; e += kRrThreads) ptr[e] = min(max(pg[e], 0), M);
    for (int e = tid; e < E; e += kRrThreads) {
        int s = 0;
        const int32_t* cs = counts_src + (int64_t)inst * R * E + e;
        for (int rr = 0; rr < r; ++rr) s += cs[(int64_t)rr * E];
        base[e] = s;
    }
    for (int x = tid; x < kRrWarps * E; x += kRrThreads) wcnt[x] = 0;
    __syncthreads();
    {
        const int nM = ptr[E];
        const int32_t* ig = inst_id + (int64_t)inst * M;
        const int32_t* cg = inst_cum + (int64_t)inst * M;
        for (int m = tid; m < M; m += kRrThreads) {
            int cum = INT_MIN, del = 0;
            if (m < nM) {
                const int p = ig[m];
                if (p >= 0 && p < P) {
                    cum = cg[m];
                    del = off[p] - (cum - qg[p]);
                }
            }
            bcum[m] = cum;
            bdel[m] = del;
        }
    }
    if (r == 0) {
        int32_t* og = inst_offset + (int64_t)inst * (P + 1);
        for (int p = tid; p <= P; p += kRrThreads) og[p] = off[p];
    }
    __syncthreads();

    // ---- this block's slots: source rank r
    const int64_t Tr = tokens_per_rank(T, R);
    const int64_t N = T * k;
    const int64_t s0 = min(T, (int64_t)r * Tr) * k, s1 = min(T, (int64_t)(r + 1) * Tr) * k;
    const int32_t* idi = ids + (int64_t)inst * N;
    int32_t* dsti = dst_row + (int64_t)inst * N;
    int32_t* srci = src_slot ? src_slot + (int64_t)inst * N : nullptr;
    int32_t* wrow = wcnt + warp * E;
    const unsigned lt = lanemask_lt();
    int my_flags = 0;

    for (int64_t cs = s0; cs < s1; cs += kChunk) {
        const int64_t wb = cs + (int64_t)warp * 32 * kItems + lane;
        int ev[kItems];
        unsigned gm[kItems];
#pragma unroll
        for (int it = 0; it < kItems; ++it) {
            const int64_t i = wb + it * 32;
            ev[it] = (i < s1) ? __ldcs(idi + i) : -1;
        }
        // phase A: per-warp histogram of this chunk (warp-aggregated)
#pragma unroll
        for (int it = 0; it < kItems; ++it) {
            const int64_t i = wb + it * 32;
            const bool valid = ev[it] >= 0 && ev[it] < E;
            if (i < s1 && !valid) my_flags |= EP_DEV_BAD_ID;
            if (!valid) ev[it] = -1;
            gm[it] = __match_any_sync(kFull, ev[it]);
            if (valid && lane == __ffs(gm[it]) - 1) atomicAdd(&wrow[ev[it]], __popc(gm[it]));
        }
        __syncthreads();
        // phase B: per expert, exclusive scan over warps on top of the running base
        for (int e = tid; e < E; e += kRrThreads) {
            int run = base[e];
            for (int w = 0; w < kRrWarps; ++w) {
                const int c = wcnt[w * E + e];
                wcnt[w * E + e] = run;
                run += c;
            }
            base[e] = run;
        }
        __syncthreads();
        // phase C: within-expert rank -> instance -> row
#pragma unroll
        for (int it = 0; it < kItems; ++it) {
            const int64_t i = wb + it * 32;
            const int e = ev[it];
            const unsigned g = gm[it];
            const int b = (e >= 0) ? wrow[e] : 0;
            __syncwarp();
            if (e >= 0 && lane == __ffs(g) - 1) wrow[e] = b + __popc(g);
            __syncwarp();
            if (i < s1) {
                int d = -1;
                if (e >= 0) {
                    const int x = b + __popc(g & lt);
                    int m = ptr[e];
                    const int me = ptr[e + 1] - 1;
                    while (m < me && bcum[m] <= x) ++m;
                    if (m <= me && bcum[m] > x) {
                        d = x + bdel[m];
                        if (d < 0 || d >= N) d = -1;
                    }
                    if (d < 0) my_flags |= EP_DEV_QUOTA_OVERFLOW;
                }
                __stcs(dsti + i, d);
                if (srci != nullptr && d >= 0) srci[d] = (int32_t)i;
            }
        }
        for (int e = lane; e < E; e += 32) wrow[e] = 0;
        __syncwarp();
    }
    if (my_flags) atomicOr(&flags, my_flags);
    __syncthreads();
    if (tid == 0 && flags) raise_flag(dev_status, flags);
}

}  // namespace

cudaError_t launch_reroute(const ep_domain_t& d, const int32_t* ids, int64_t T, int32_t n_inst,
                           const int32_t* counts_src, const int32_t* quota,
                           const int32_t* inst_ptr, const int32_t* inst_id,
                           const int32_t* inst_cum, int32_t* dst_row, int32_t* src_slot,
                           int32_t* inst_offset, int32_t* dev_status, cudaStream_t s) {
    if (n_inst == 0) return cudaSuccess;
    const RrLayout lay = rr_layout(d.R, d.E, d.S);
    if (lay.bytes > 48 * 1024) {
        cudaError_t err = cudaFuncSetAttribute(reroute_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                               (int)lay.bytes);
        if (err != cudaSuccess) return err;
    }
    const int64_t blocks = (int64_t)n_inst * d.R;
    reroute_kernel<<<(unsigned)blocks, kRrThreads, lay.bytes, s>>>(
        ids, T, d.k, d.R, d.E, d.S, counts_src, quota, inst_ptr, inst_id, inst_cum, dst_row,
        src_slot, inst_offset, dev_status);
    return cudaGetLastError();
}

}  // namespace ultraep
