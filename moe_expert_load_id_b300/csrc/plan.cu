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
// least-loaded eligible rank, q = min(quota, floor(gap/2)), global stop).
//
// One warp per (layer, microbatch) instance.  The moves form one serial
// chain, so the design goal is the shortest dependent path per move.  Two
// move loops implement the rule: plan_moves_table on a shared-memory table
// (plan_dev.cuh) runs the flag-free rule, plan_moves on registers (below) the
// variants of ep_plan_ex.  The register loop:
//   - lane l owns ranks l and l+32 and keeps, in registers, each rank's load,
//     its instances (quota and expert, unrolled over a compile-time bound WB on
//     H+S) and its largest instance;
//   - hot and cold are each ONE redux.sync over a packed key
//     (load << 6 | rank index, the index flipped for the max so that the lowest
//     rank wins ties); instances whose loads could overflow the packing
//     (total >= 2^25) take a two-collective path (redux on the load, then a
//     ballot for the lowest rank that attains it);
//   - "rank c holds e" is a register compare in c's owner lane, so a move
//     touches no shared memory at all;
//   - every lane runs the same branch-free update on its own registers (a
//     no-op unless it owns hot or cold), so the warp never diverges.
// The register loop uses shared memory only after the loop, to build the
// logical->physical CSR table.
#include <climits>

#include "common.cuh"
#include "plan_dev.cuh"

namespace ultraep {
namespace {

constexpr int kPlanWarps = 4;
// the flag-free rule runs the shared-memory table loop from this register
// bound on (build-time tunable; the bounds are 2, 3, 4, 6, 8, 16, 32; 2: always)
#ifndef EP_PLAN_TABLE_MIN_WB
#define EP_PLAN_TABLE_MIN_WB 2
#endif
// Registers of one rank: quota and expert of local instance j (j < H: home of
// expert r*H + j; H <= j < W: spare slot j-H, expert -1 while empty).
template <int WB>
struct RankRegs {
    int q[WB];
    int x[WB];
    int load;      // -1: the rank does not exist
    unsigned occ;  // bit s: spare slot s holds an expert
    int bq;        // largest quota among its instances
    int bx;        // that instance: expert << 5 | j (lowest expert on ties)

    __device__ __forceinline__ void best(int W) {
        bq = -1;
        bx = INT_MAX;
#pragma unroll
        for (int j = 0; j < WB; ++j) {
            const int cx = (x[j] << 5) | j;
            const bool take = j < W && x[j] >= 0 && (q[j] > bq || (q[j] == bq && cx < bx));
            bq = take ? q[j] : bq;
            bx = take ? cx : bx;
        }
    }
    // the largest instance with quota >= 1 whose local index is not in excl
    // (the skip variant's next candidate); bq = -1 when there is none
    __device__ __forceinline__ void best_excl(int W, unsigned excl, int& cq, int& cxo) const {
        cq = -1;
        cxo = INT_MAX;
#pragma unroll
        for (int j = 0; j < WB; ++j) {
            const int cx = (x[j] << 5) | j;
            const bool ok = j < W && x[j] >= 0 && q[j] >= 1 && !((excl >> j) & 1u);
            const bool take = ok && (q[j] > cq || (q[j] == cq && cx < cxo));
            cq = take ? q[j] : cq;
            cxo = take ? cx : cxo;
        }
    }
    __device__ __forceinline__ bool holds(int e) const {
        bool h = false;
#pragma unroll
        for (int j = 0; j < WB; ++j) h |= (x[j] == e);
        return h;
    }
    __device__ __forceinline__ bool has_free(int S) const {
        return occ != ((S >= 32) ? ~0u : ((1u << S) - 1u));
    }
    // (the rank's load is updated by the move loop itself, ahead of these)
    // hot side: the owner lane (mine) removes mv from its instance j; with
    // release, a spare-slot instance left at quota 0 frees its slot
    __device__ __forceinline__ void take(int j, bool mine, int mv, int H, bool release) {
#pragma unroll
        for (int jj = 0; jj < WB; ++jj) {
            const bool from = mine && jj == j;
            q[jj] -= from ? mv : 0;
            const bool freed = release && from && jj >= H && q[jj] == 0;
            x[jj] = freed ? -1 : x[jj];
            occ &= freed ? ~(1u << (jj - H)) : ~0u;
        }
    }
    // cold side: the owner lane adds mv to its instance of e, filling the
    // lowest free spare slot when it does not hold e yet (without released
    // slots the filled ones are a prefix, so that is the count of filled
    // slots).  Only one instance grew, so the largest instance is updated in
    // place.
    template <bool kHoles>
    __device__ __forceinline__ void give(int e, bool held, bool mine, int H, int mv) {
        const int jn = held ? -1 : H + (kHoles ? __ffs(~occ) - 1 : __popc(occ));
        int nq = 0, nj = 0;
#pragma unroll
        for (int jj = 0; jj < WB; ++jj) {
            const bool to = mine && (held ? (x[jj] == e) : (jj == jn));
            x[jj] = to ? e : x[jj];
            q[jj] += to ? mv : 0;
            nq = to ? q[jj] : nq;
            nj = to ? jj : nj;
        }
        occ |= (mine && !held) ? (1u << (jn - H)) : 0u;
        const int cx = (e << 5) | nj;
        const bool better = mine && (nq > bq || (nq == bq && cx < bx));
        bq = better ? nq : bq;
        bx = better ? cx : bx;
    }
};

// One warp's move loop.  kPacked: hot and cold by one redux on a packed key.
// kTwo: R > 32, every lane owns a second rank (B).  Which half holds hot or
// cold is warp-uniform, so only that half's instance registers are updated.
// The loop is software-pipelined: as soon as the amount is known the two
// loads change and the next move's argmax is issued; the instance bookkeeping
// of the current move (take, give, largest instance) overlaps it.
// flags (warp-uniform; kFlags: compiled in at all, so that the base rule's
// loop carries none of it): EP_PLAN_SKIP -- when the hottest rank's largest
// instance cannot move, try its next instances, then the next-hottest ranks,
// and make the first move that can be made; EP_PLAN_RELEASE -- a spare-slot
// instance a move empties frees its slot.
template <int WB, bool kTwo, bool kPacked, bool kFlags>
__device__ __forceinline__ void plan_moves(RankRegs<WB>& A, RankRegs<WB>& B, int lane, int H,
                                           int S, int W, int R, int max_iters, int flags,
                                           int& iters, int& status) {
    const bool hasA = A.load >= 0, hasB = kTwo && B.load >= 0;
    const int ra = lane, rb = lane + 32;
    const bool skip = kFlags && (flags & EP_PLAN_SKIP) != 0;
    const bool release = kFlags && (flags & EP_PLAN_RELEASE) != 0;

    // candidate (hot, expert e with quota qsrc): the coldest eligible rank and
    // the amount; mv <= 0 when no move is possible
    auto evaluate = [&](int hot, int Lhot, int e, int qsrc, int& cold, bool& holdA,
                        bool& holdB) -> int {
        holdA = A.holds(e);
        holdB = kTwo && B.holds(e);
        const bool elA = hasA && ra != hot && (holdA || A.has_free(S));
        const bool elB = hasB && rb != hot && (holdB || B.has_free(S));
        int Lmin;
        if (kPacked) {
            const unsigned ca = elA ? ((unsigned)A.load << 6) | (unsigned)ra : 0xffffffffu;
            const unsigned cb = elB ? ((unsigned)B.load << 6) | (unsigned)rb : 0xffffffffu;
            const unsigned k = __reduce_min_sync(kFull, kTwo ? min(ca, cb) : ca);
            if (k == 0xffffffffu) return 0;  // no eligible rank
            cold = (int)(k & 63u);
            Lmin = (int)(k >> 6);
        } else {
            if (!__any_sync(kFull, elA || elB)) return 0;
            const int ca = elA ? A.load : INT_MAX;
            const int cb = elB ? B.load : INT_MAX;
            Lmin = __reduce_min_sync(kFull, kTwo ? min(ca, cb) : ca);
            const unsigned b0 = __ballot_sync(kFull, elA && ca == Lmin);
            const unsigned b1 = kTwo ? __ballot_sync(kFull, elB && cb == Lmin) : 0u;
            cold = b0 ? __ffs(b0) - 1 : 32 + __ffs(b1) - 1;
        }
        return min(qsrc, (Lhot - Lmin) >> 1);
    };

    int hot, Lmax;
    argmax_rank<kTwo, kPacked>(A.load, B.load, hasA, hasB, lane, hot, Lmax);
    while (true) {
        // 2. hot's largest-quota instance (lowest expert id on ties)
        bool hotB = kTwo && hot >= 32;
        int hl = hot & 31;
        int qmax = __shfl_sync(kFull, hotB ? B.bq : A.bq, hl);
        int bx = __shfl_sync(kFull, hotB ? B.bx : A.bx, hl);
        int e = bx >> 5, src_j = bx & 31;

        // 3-5. coldest eligible rank and the amount
        int cold = 0;
        bool holdA = false, holdB = false;
        int mv = evaluate(hot, Lmax, e, qmax, cold, holdA, holdB);
        if (mv <= 0) {
            if (!skip) break;  // the base rule's global stop
            // skip: hot's next instances, then the next-hottest ranks
            uint64_t rtried = 1ull << hot;
            unsigned itried = 1u << src_j;
            int ranks_tried = 1;
            while (mv <= 0) {
                int cq, cx;
                if (hotB) B.best_excl(W, itried, cq, cx); else A.best_excl(W, itried, cq, cx);
                cq = __shfl_sync(kFull, cq, hl);
                cx = __shfl_sync(kFull, cx, hl);
                if (cq >= 1) {
                    e = cx >> 5;
                    src_j = cx & 31;
                    itried |= 1u << src_j;
                    qmax = cq;
                    mv = evaluate(hot, Lmax, e, qmax, cold, holdA, holdB);
                    continue;
                }
                if (ranks_tried == R) break;  // every candidate tried
                // the hottest rank not tried yet (lowest index on ties)
                const bool tA = (rtried >> ra) & 1ull, tB = (rtried >> rb) & 1ull;
                argmax_rank<kTwo, kPacked>(tA ? -1 : A.load, tB ? -1 : B.load, hasA && !tA,
                                           hasB && !tB, lane, hot, Lmax);
                rtried |= 1ull << hot;
                ++ranks_tried;
                hotB = kTwo && hot >= 32;
                hl = hot & 31;
                itried = 0u;
            }
            if (mv <= 0) break;  // no candidate can move
        }
        // 6. safety cap
        if (iters == max_iters) {
            status = EP_ERR_ITER_LIMIT;
            break;
        }
        const bool coldB = kTwo && cold >= 32;
        const int cl = cold & 31;

        // 7. move.  Loads first, then the next move's argmax ...
        A.load += (ra == cold ? mv : 0) - (ra == hot ? mv : 0);
        if (kTwo) B.load += (rb == cold ? mv : 0) - (rb == hot ? mv : 0);
        int nhot, nLmax;
        argmax_rank<kTwo, kPacked>(A.load, B.load, hasA, hasB, lane, nhot, nLmax);
        // ... while hot's owner lane takes, cold's owner lane gives, and hot's
        // half refreshes its largest instance (only the half holding each of
        // them is touched)
        if (hotB) B.take(src_j, lane == hl, mv, H, release);
        else A.take(src_j, lane == hl, mv, H, release);
        if (coldB) B.template give<kFlags>(e, holdB, lane == cl, H, mv);
        else A.template give<kFlags>(e, holdA, lane == cl, H, mv);
        if (hotB) B.best(W); else A.best(W);
        hot = nhot;
        Lmax = nLmax;
        ++iters;
    }
}


template <int WB>
__device__ __forceinline__ void init_rank(RankRegs<WB>& X, int rk, int R, int H, int W,
                                          const int32_t* cnt) {
    const bool has = rk < R;
    unsigned sum = 0;
#pragma unroll
    for (int j = 0; j < WB; ++j) {
        const bool home = has && j < H;
        X.q[j] = home ? cnt[rk * H + j] : 0;
        X.x[j] = home ? rk * H + j : -1;
        sum += (unsigned)X.q[j];
    }
    X.load = has ? (int)sum : -1;
    X.occ = 0u;
    X.best(W);
}

template <int WB>
__device__ __forceinline__ void store_rank(const RankRegs<WB>& X, int rk, int R, int H, int S,
                                           int W, int32_t* q, int32_t* slot, uint64_t* holder,
                                           int32_t* qo, int32_t* so, int32_t* lo) {
    if (rk >= R) return;
#pragma unroll
    for (int j = 0; j < WB; ++j) {
        if (j < W) {
            q[rk * W + j] = X.q[j];
            qo[rk * W + j] = X.q[j];
        }
        if (j >= H && j < W) {
            slot[rk * S + (j - H)] = X.x[j];
            so[rk * S + (j - H)] = X.x[j];
            if (X.x[j] >= 0) atomicOr((unsigned long long*)&holder[X.x[j]], 1ull << rk);
        }
    }
    lo[rk] = X.load;
}

template <int WB, bool kTwo, bool kFlags>
__global__ void __launch_bounds__(kPlanWarps * 32, 1)
plan_kernel(const int32_t* __restrict__ counts, int n_inst, int R, int E, int S, int max_iters,
            int flags,
            int32_t* __restrict__ quota_out, int32_t* __restrict__ slot_out,
            int32_t* __restrict__ load_out, int32_t* __restrict__ ptr_out,
            int32_t* __restrict__ id_out, int32_t* __restrict__ cum_out,
            int32_t* __restrict__ iter_out, int32_t* __restrict__ status_out,
            const int32_t* __restrict__ counts_src, int32_t* __restrict__ counts_out) {
    extern __shared__ __align__(16) unsigned char smem[];
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
        for (int x = threadIdx.x; x < kPlanWarps * E; x += kPlanWarps * 32) {
            const int w = x / E;
            csum0[w * (wbytes / 4) + (x - w * E)] = 0;
        }
        __syncthreads();
        // thread (column, row group): column c of E, rows rg, rg + G, ...
        constexpr int kThr = kPlanWarps * 32;
        const int G = max(1, kThr / E);
        for (int x = threadIdx.x; x < nb * E * G; x += kThr) {
            const int wi = x / (E * G), rem = x - wi * E * G;
            const int rg = rem / E, e = rem - rg * E;
            const int32_t* cs = counts_src + (int64_t)(g0 + wi) * R * E + e;
            int t = 0;
            for (int r0 = rg; r0 < R; r0 += 8 * G) {
                int v[8];
#pragma unroll
                for (int u = 0; u < 8; ++u) {
                    const int rr = r0 + u * G;
                    v[u] = (rr < R) ? __ldg(cs + (int64_t)rr * E) : 0;
                }
#pragma unroll
                for (int u = 0; u < 8; ++u) t += v[u];
            }
            atomicAdd(&csum0[wi * (wbytes / 4) + e], t);
        }
        __syncthreads();
        if (g < n_inst) {
            const int32_t* mine = csum0 + warp * (wbytes / 4);
            for (int e = lane; e < E; e += 32) counts_out[(int64_t)g * E + e] = mine[e];
            cnt = mine;
        }
    }
    if (g >= n_inst) return;  // whole warp; no block-wide barrier follows

    // counts must be >= 0 with a total below 2^31; otherwise the instance is
    // rejected (EP_ERR_INVAL) and its outputs describe the home-only placement
    long long tot = 0;
    int status = plan_check_counts(cnt, E, lane, tot);

    unsigned char* base = smem + (size_t)warp * wbytes;
    int32_t* q = reinterpret_cast<int32_t*>(base);
    int32_t* slot = reinterpret_cast<int32_t*>(base + align16((size_t)P * 4));
    uint64_t* holder = reinterpret_cast<uint64_t*>(base + align16((size_t)P * 4) +
                                                   align16((size_t)R * S * 4));
    int32_t* csr_pos = reinterpret_cast<int32_t*>(reinterpret_cast<unsigned char*>(holder) +
                                                  align16((size_t)E * 8));
    int32_t* csr_val = csr_pos + align16((size_t)(E + 1) * 4) / 4;
    int32_t* qo = quota_out + (int64_t)g * P;
    int32_t* so = slot_out + (int64_t)g * R * S;
    int32_t* lo = load_out + (int64_t)g * R;
    int iters = 0;
    // the base rule runs on the shared-memory table (a move costs the same
    // whatever W: measured 0.38-0.39 us per move at W = 3 and 6, against 0.46
    // and 0.70 on registers); the variants run the register loop
    if constexpr (!kFlags && WB >= EP_PLAN_TABLE_MIN_WB) {
        // ---- the base rule on the shared-memory table
        plan_table_solve<kTwo>(cnt, R, E, S, max_iters, tot, q, slot, holder, lane, qo, so, lo,
                               iters, status);
    } else {
        // ---- registers: ranks lane (A) and lane+32 (B)
        RankRegs<WB> A, B;
        init_rank(A, lane, R, H, W, cnt);
        init_rank(B, lane + 32, R, H, W, cnt);
        if (status == EP_OK) {
            if (tot < kPackLimit)
                plan_moves<WB, kTwo, true, kFlags>(A, B, lane, H, S, W, R, max_iters, flags,
                                                   iters, status);
            else
                plan_moves<WB, kTwo, false, kFlags>(A, B, lane, H, S, W, R, max_iters, flags,
                                                    iters, status);
        }
        // outputs: quota, spare slots and loads straight from registers; the CSR
        // is built from a shared-memory copy
        for (int e = lane; e < E; e += 32) holder[e] = 1ull << (e / H);
        __syncwarp();
        store_rank(A, lane, R, H, S, W, q, slot, holder, qo, so, lo);
        store_rank(B, lane + 32, R, H, S, W, q, slot, holder, qo, so, lo);
    }
    __syncwarp();

    // logical -> physical CSR: home first, then replicas by ascending rank (= ascending p)
    plan_csr(q, slot, holder, R, E, S, lane, csr_pos, csr_val, ptr_out + (int64_t)g * (E + 1),
             id_out + (int64_t)g * (E + R * S), cum_out + (int64_t)g * (E + R * S));
    if (lane == 0) {
        iter_out[g] = iters;
        status_out[g] = status;
    }
}

template <int WB, bool kTwo, bool kFlags>
cudaError_t launch_plan_k(const ep_domain_t& d, const int32_t* counts, int32_t n_inst,
                           int32_t max_iters, int32_t flags, int32_t* quota, int32_t* slot_expert,
                           int32_t* rank_load, int32_t* inst_ptr, int32_t* inst_id,
                           int32_t* inst_cum, int32_t* n_iter, int32_t* inst_status,
                           cudaStream_t s, bool pdl, const int32_t* counts_src) {
    const size_t smem = kPlanWarps * plan_warp_bytes(d.R, d.E, d.S);
    if (smem > 48 * 1024) {
        cudaError_t err = cudaFuncSetAttribute(plan_kernel<WB, kTwo, kFlags>,
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
    return cudaLaunchKernelEx(&cfg, plan_kernel<WB, kTwo, kFlags>, counts, (int)n_inst, (int)d.R,
                              (int)d.E, (int)d.S, (int)max_iters, (int)flags, quota, slot_expert, rank_load,
                              inst_ptr, inst_id, inst_cum, n_iter, inst_status, counts_src,
                              const_cast<int32_t*>(counts));
}

// the flag-free base rule gets its own kernel
template <int WB, bool kTwo>
cudaError_t launch_plan_wb(const ep_domain_t& d, const int32_t* counts, int32_t n_inst,
                           int32_t max_iters, int32_t flags, int32_t* quota, int32_t* slot_expert,
                           int32_t* rank_load, int32_t* inst_ptr, int32_t* inst_id,
                           int32_t* inst_cum, int32_t* n_iter, int32_t* inst_status,
                           cudaStream_t s, bool pdl, const int32_t* counts_src) {
    if (flags != 0)
        return launch_plan_k<WB, kTwo, true>(d, counts, n_inst, max_iters, flags, quota,
                                             slot_expert, rank_load, inst_ptr, inst_id, inst_cum,
                                             n_iter, inst_status, s, pdl, counts_src);
    return launch_plan_k<WB, kTwo, false>(d, counts, n_inst, max_iters, flags, quota, slot_expert,
                                          rank_load, inst_ptr, inst_id, inst_cum, n_iter,
                                          inst_status, s, pdl, counts_src);
}

template <int WB>
cudaError_t launch_plan_r(const ep_domain_t& d, const int32_t* counts, int32_t n_inst,
                          int32_t max_iters, int32_t flags, int32_t* quota, int32_t* slot_expert,
                          int32_t* rank_load, int32_t* inst_ptr, int32_t* inst_id,
                          int32_t* inst_cum, int32_t* n_iter, int32_t* inst_status,
                          cudaStream_t s, bool pdl, const int32_t* counts_src) {
    if (d.R > 32)
        return launch_plan_wb<WB, true>(d, counts, n_inst, max_iters, flags, quota, slot_expert,
                                        rank_load, inst_ptr, inst_id, inst_cum, n_iter,
                                        inst_status, s, pdl, counts_src);
    return launch_plan_wb<WB, false>(d, counts, n_inst, max_iters, flags, quota, slot_expert,
                                     rank_load, inst_ptr, inst_id, inst_cum, n_iter,
                                     inst_status, s, pdl, counts_src);
}

}  // namespace

cudaError_t launch_plan(const ep_domain_t& d, const int32_t* counts, int32_t n_inst,
                        int32_t max_iters, int32_t flags, int32_t* quota, int32_t* slot_expert, int32_t* rank_load,
                        int32_t* inst_ptr, int32_t* inst_id, int32_t* inst_cum, int32_t* n_iter,
                        int32_t* inst_status, cudaStream_t s, bool pdl, const int32_t* counts_src) {
    if (n_inst == 0) return cudaSuccess;
    // register arrays sized to the instances per rank W = H + S (<= 32)
    const int W = d.E / d.R + d.S;
#define EP_PLAN_WB(wb)                                                                       \
    if (W <= wb)                                                                             \
        return launch_plan_r<wb>(d, counts, n_inst, max_iters, flags, quota, slot_expert, rank_load, \
                                 inst_ptr, inst_id, inst_cum, n_iter, inst_status, s, pdl, counts_src);
    EP_PLAN_WB(2)
    EP_PLAN_WB(3)
    EP_PLAN_WB(4)
    EP_PLAN_WB(6)
    EP_PLAN_WB(8)
    EP_PLAN_WB(16)
#undef EP_PLAN_WB
    return launch_plan_r<32>(d, counts, n_inst, max_iters, flags, quota, slot_expert, rank_load,
                             inst_ptr, inst_id, inst_cum, n_iter, inst_status, s, pdl, counts_src);
}

}  // namespace ultraep
