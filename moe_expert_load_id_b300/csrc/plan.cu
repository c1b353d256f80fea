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
// (see there) runs the flag-free rule, plan_moves on registers (below) the
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

namespace ultraep {
namespace {

constexpr int kPlanWarps = 4;
// the flag-free rule runs the shared-memory table loop from this register
// bound on (build-time tunable; the bounds are 2, 3, 4, 6, 8, 16, 32; 2: always)
#ifndef EP_PLAN_TABLE_MIN_WB
#define EP_PLAN_TABLE_MIN_WB 2
#endif
constexpr long long kPackLimit = 1ll << 25;  // total below this: loads fit a 6-bit-shifted key

__host__ __device__ inline size_t align16(size_t x) { return (x + 15) & ~size_t(15); }

__host__ __device__ inline size_t plan_warp_bytes(int R, int E, int S) {
    const int P = R * (E / R + S);
    return align16((size_t)P * 4) + align16((size_t)R * S * 4) + (size_t)E * 8;
}

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

// Hottest rank (lowest index on ties) and its load.
template <bool kTwo, bool kPacked>
__device__ __forceinline__ void argmax_rank(int la, int lb, bool hasA, bool hasB, int lane,
                                            int& hot, int& Lmax) {
    if (kPacked) {
        const unsigned ka = hasA ? ((unsigned)la << 6) | (unsigned)(63 - lane) : 0u;
        const unsigned kb = hasB ? ((unsigned)lb << 6) | (unsigned)(31 - lane) : 0u;
        const unsigned k = __reduce_max_sync(kFull, kTwo ? max(ka, kb) : ka);
        hot = 63 - (int)(k & 63u);
        Lmax = (int)(k >> 6);
    } else {
        Lmax = __reduce_max_sync(kFull, kTwo ? max(la, lb) : la);
        const unsigned b0 = __ballot_sync(kFull, la == Lmax);
        const unsigned b1 = kTwo ? __ballot_sync(kFull, lb == Lmax) : 0u;
        hot = b0 ? __ffs(b0) - 1 : 32 + __ffs(b1) - 1;
    }
}

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


// The base rule on a shared-memory table (the flag-free kernel): the warp's
// instance quotas q[P] (rank-major, W per rank), the experts of the spare
// slots slot[R*S] (-1: empty) and, per expert, the mask of ranks holding it;
// the loads stay in registers (lane l: ranks l and l+32).  Per move the hot
// rank's largest instance is one warp reduction over its W instances (lane j:
// instance j), eligibility is one 64-bit mask (holders of e | ranks with a
// free slot), and the bookkeeping is a few single-lane stores, so nothing in a
// move grows with the instances per rank.  Same rule, same ties, same outputs
// as plan_moves with no flags; the tables are exactly the epilogue's.
template <bool kTwo, bool kPacked>
__device__ __forceinline__ void plan_moves_table(int32_t* q, int32_t* slot, uint64_t* holder,
                                                 int& loadA, int& loadB, int lane, int H, int S,
                                                 int W, int R, int max_iters, int& iters,
                                                 int& status) {
    const bool hasA = loadA >= 0, hasB = kTwo && loadB >= 0;
    const int ra = lane, rb = lane + 32;
    const uint64_t exist = (R >= 64) ? ~0ull : ((1ull << R) - 1ull);
    uint64_t freem = S > 0 ? exist : 0ull;  // ranks with a free spare slot (warp-uniform)
    int hot, Lmax;
    argmax_rank<kTwo, kPacked>(loadA, loadB, hasA, hasB, lane, hot, Lmax);
    while (true) {
        // 2. hot's largest-quota instance, lowest expert on ties (lane j:
        // instance j; every rank has its H >= 1 home instances)
        int qj = -1;
        unsigned cxj = 0xffffffffu;
        if (lane < W) {  // the two loads are independent
            const int xj = lane < H ? hot * H + lane : slot[hot * S + (lane - H)];
            const int qv = q[hot * W + lane];
            if (xj >= 0) {
                qj = qv;
                cxj = ((unsigned)xj << 5) | (unsigned)lane;
            }
        }
        const int qmax = __reduce_max_sync(kFull, qj);
        const unsigned cx = __reduce_min_sync(kFull, qj == qmax ? cxj : 0xffffffffu);
        const int e = (int)(cx >> 5), src_j = (int)(cx & 31u);

        // 3-5. eligible ranks: the others that hold e or have a free slot;
        // the coldest of them (lowest rank on ties) and the amount
        const uint64_t hm = holder[e];
        const uint64_t el = (hm | freem) & exist & ~(1ull << hot);
        if (el == 0ull) break;  // no rank is eligible
        const bool elA = hasA && ((el >> ra) & 1ull);
        const bool elB = hasB && ((el >> rb) & 1ull);
        int cold, Lmin;
        if (kPacked) {
            const unsigned ca = elA ? ((unsigned)loadA << 6) | (unsigned)ra : 0xffffffffu;
            const unsigned cb = elB ? ((unsigned)loadB << 6) | (unsigned)rb : 0xffffffffu;
            const unsigned kk = __reduce_min_sync(kFull, kTwo ? min(ca, cb) : ca);
            cold = (int)(kk & 63u);
            Lmin = (int)(kk >> 6);
        } else {
            const int ca = elA ? loadA : INT_MAX;
            const int cb = elB ? loadB : INT_MAX;
            Lmin = __reduce_min_sync(kFull, kTwo ? min(ca, cb) : ca);
            const unsigned b0 = __ballot_sync(kFull, elA && ca == Lmin);
            const unsigned b1 = kTwo ? __ballot_sync(kFull, elB && cb == Lmin) : 0u;
            cold = b0 ? __ffs(b0) - 1 : 32 + __ffs(b1) - 1;
        }
        const int mv = min(qmax, (Lmax - Lmin) >> 1);
        if (mv <= 0) break;  // the global stop
        // 6. safety cap
        if (iters == max_iters) {
            status = EP_ERR_ITER_LIMIT;
            break;
        }
        // 7. move.  Loads first, then the next move's argmax ...
        loadA += (ra == cold ? mv : 0) - (ra == hot ? mv : 0);
        if (kTwo) loadB += (rb == cold ? mv : 0) - (rb == hot ? mv : 0);
        int nhot, nLmax;
        argmax_rank<kTwo, kPacked>(loadA, loadB, hasA, hasB, lane, nhot, nLmax);
        // ... and the tables: cold's instance of e is its home, a spare slot
        // already holding e, or its lowest free spare slot (filled now).  The
        // spare slots are read and voted on unconditionally (no branch), so
        // this overlaps the argmax above.
        const int sv = (lane < S) ? slot[cold * S + lane] : 0;
        const unsigned hit = __ballot_sync(kFull, lane < S && sv == e);
        const unsigned freeb = __ballot_sync(kFull, lane < S && sv < 0);  // cold's free slots
        const bool held = (hm >> cold) & 1ull;
        const int ej = e - cold * H;
        const bool home = (unsigned)ej < (unsigned)H;  // e is one of cold's home experts
        const unsigned pick = held ? hit : freeb;       // nonzero unless home: cold is eligible
        if (!home && pick == 0u) {                      // (never; keeps every index in range)
            status = EP_ERR_INVAL;
            break;
        }
        const int dj = home ? ej : H + __ffs(pick) - 1;
        // every read of this move was consumed by the warp's votes and
        // reductions above; the updates are fire-and-forget shared-memory
        // additions, no read-modify-write chain
        if (lane == 0) {
            atomicAdd(&q[hot * W + src_j], -mv);
            atomicAdd(&q[cold * W + dj], mv);
            if (!held) {
                slot[cold * S + (dj - H)] = e;
                holder[e] = hm | (1ull << cold);
            }
        }
        if (!held && (freeb & (freeb - 1u)) == 0u) freem &= ~(1ull << cold);  // its last free slot
        __syncwarp();  // the updates land before the next move reads the table
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
            int32_t* __restrict__ iter_out, int32_t* __restrict__ status_out) {
    extern __shared__ __align__(16) unsigned char smem[];
    // in ep_balance this grid is a programmatic dependent of ep_count: wait for
    // its counts, then let the dependent reroute start its plan-independent
    // work (for a plain launch both are no-ops)
    pdl_wait();
    pdl_trigger();
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int g = blockIdx.x * kPlanWarps + warp;
    if (g >= n_inst) return;  // whole warp; no block-wide barrier follows

    const int H = E / R, W = H + S, P = R * W;
    const int32_t* cnt = counts + (int64_t)g * E;

    // counts must be >= 0 with a total below 2^31; otherwise the instance is
    // rejected (EP_ERR_INVAL) and its outputs describe the home-only placement
    int status = EP_OK;
    long long tot = 0;
    {
        bool bad = false;
        for (int e = lane; e < E; e += 32) {
            bad |= cnt[e] < 0;
            tot += cnt[e];
        }
        bad = __any_sync(kFull, bad);
        for (int o = 16; o > 0; o >>= 1) tot += __shfl_xor_sync(kFull, tot, o);
        if (bad || tot > (long long)INT_MAX) status = EP_ERR_INVAL;
    }

    unsigned char* base = smem + (size_t)warp * plan_warp_bytes(R, E, S);
    int32_t* q = reinterpret_cast<int32_t*>(base);
    int32_t* slot = reinterpret_cast<int32_t*>(base + align16((size_t)P * 4));
    uint64_t* holder = reinterpret_cast<uint64_t*>(base + align16((size_t)P * 4) +
                                                   align16((size_t)R * S * 4));
    int32_t* qo = quota_out + (int64_t)g * P;
    int32_t* so = slot_out + (int64_t)g * R * S;
    int32_t* lo = load_out + (int64_t)g * R;
    int iters = 0;
    // the base rule runs on the shared-memory table (a move costs the same
    // whatever W: measured 0.38-0.39 us per move at W = 3 and 6, against 0.46
    // and 0.70 on registers); the variants run the register loop
    if constexpr (!kFlags && WB >= EP_PLAN_TABLE_MIN_WB) {
        // ---- the base rule on the shared-memory table
        for (int p = lane; p < P; p += 32) {
            const int r = p / W, j = p - r * W;
            q[p] = j < H ? cnt[r * H + j] : 0;
        }
        for (int x = lane; x < R * S; x += 32) slot[x] = -1;
        for (int e = lane; e < E; e += 32) holder[e] = 1ull << (e / H);
        int loadA = -1, loadB = -1;
        if (lane < R) {
            unsigned sum = 0;
            for (int j = 0; j < H; ++j) sum += (unsigned)cnt[lane * H + j];
            loadA = (int)sum;
        }
        if (kTwo && lane + 32 < R) {
            unsigned sum = 0;
            for (int j = 0; j < H; ++j) sum += (unsigned)cnt[(lane + 32) * H + j];
            loadB = (int)sum;
        }
        __syncwarp();
        if (status == EP_OK) {
            if (tot < kPackLimit)
                plan_moves_table<kTwo, true>(q, slot, holder, loadA, loadB, lane, H, S, W, R,
                                             max_iters, iters, status);
            else
                plan_moves_table<kTwo, false>(q, slot, holder, loadA, loadB, lane, H, S, W, R,
                                              max_iters, iters, status);
        }
        __syncwarp();
        for (int p = lane; p < P; p += 32) qo[p] = q[p];
        for (int x = lane; x < R * S; x += 32) so[x] = slot[x];
        if (lane < R) lo[lane] = loadA;
        if (kTwo && lane + 32 < R) lo[lane + 32] = loadB;
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
    int32_t* po = ptr_out + (int64_t)g * (E + 1);
    int32_t* io = id_out + (int64_t)g * (E + R * S);
    int32_t* co = cum_out + (int64_t)g * (E + R * S);
    int run = 0;
    for (int e0 = 0; e0 < E; e0 += 32) {
        const int e = e0 + lane;
        const uint64_t hm = (e < E) ? holder[e] : 0ull;
        const int n = __popcll(hm);
        int x = n;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const int y = __shfl_up_sync(kFull, x, o);
            if (lane >= o) x += y;
        }
        if (e < E) {
            int m = run + x - n;
            po[e] = m;
            const int home = e / H;
            const int hp = home * W + (e - home * H);
            int cum = q[hp];
            io[m] = hp;
            co[m] = cum;
            ++m;
            uint64_t rest = hm & ~(1ull << home);
            while (rest) {
                const int c = __ffsll((long long)rest) - 1;
                rest &= rest - 1;
                int j = 0;
                while (j < S && slot[c * S + j] != e) ++j;
                const int p = c * W + H + j;
                cum += q[p];
                io[m] = p;
                co[m] = cum;
                ++m;
            }
        }
        run += __shfl_sync(kFull, x, 31);
    }
    if (lane == 0) {
        po[E] = run;
        iter_out[g] = iters;
        status_out[g] = status;
    }
}

template <int WB, bool kTwo, bool kFlags>
cudaError_t launch_plan_k(const ep_domain_t& d, const int32_t* counts, int32_t n_inst,
                           int32_t max_iters, int32_t flags, int32_t* quota, int32_t* slot_expert,
                           int32_t* rank_load, int32_t* inst_ptr, int32_t* inst_id,
                           int32_t* inst_cum, int32_t* n_iter, int32_t* inst_status,
                           cudaStream_t s, bool pdl) {
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
                              inst_ptr, inst_id, inst_cum, n_iter, inst_status);
}

// the flag-free base rule gets its own kernel
template <int WB, bool kTwo>
cudaError_t launch_plan_wb(const ep_domain_t& d, const int32_t* counts, int32_t n_inst,
                           int32_t max_iters, int32_t flags, int32_t* quota, int32_t* slot_expert,
                           int32_t* rank_load, int32_t* inst_ptr, int32_t* inst_id,
                           int32_t* inst_cum, int32_t* n_iter, int32_t* inst_status,
                           cudaStream_t s, bool pdl) {
    if (flags != 0)
        return launch_plan_k<WB, kTwo, true>(d, counts, n_inst, max_iters, flags, quota,
                                             slot_expert, rank_load, inst_ptr, inst_id, inst_cum,
                                             n_iter, inst_status, s, pdl);
    return launch_plan_k<WB, kTwo, false>(d, counts, n_inst, max_iters, flags, quota, slot_expert,
                                          rank_load, inst_ptr, inst_id, inst_cum, n_iter,
                                          inst_status, s, pdl);
}

template <int WB>
cudaError_t launch_plan_r(const ep_domain_t& d, const int32_t* counts, int32_t n_inst,
                          int32_t max_iters, int32_t flags, int32_t* quota, int32_t* slot_expert,
                          int32_t* rank_load, int32_t* inst_ptr, int32_t* inst_id,
                          int32_t* inst_cum, int32_t* n_iter, int32_t* inst_status,
                          cudaStream_t s, bool pdl) {
    if (d.R > 32)
        return launch_plan_wb<WB, true>(d, counts, n_inst, max_iters, flags, quota, slot_expert,
                                        rank_load, inst_ptr, inst_id, inst_cum, n_iter,
                                        inst_status, s, pdl);
    return launch_plan_wb<WB, false>(d, counts, n_inst, max_iters, flags, quota, slot_expert,
                                     rank_load, inst_ptr, inst_id, inst_cum, n_iter,
                                     inst_status, s, pdl);
}

}  // namespace

cudaError_t launch_plan(const ep_domain_t& d, const int32_t* counts, int32_t n_inst,
                        int32_t max_iters, int32_t flags, int32_t* quota, int32_t* slot_expert, int32_t* rank_load,
                        int32_t* inst_ptr, int32_t* inst_id, int32_t* inst_cum, int32_t* n_iter,
                        int32_t* inst_status, cudaStream_t s, bool pdl) {
    if (n_inst == 0) return cudaSuccess;
    // register arrays sized to the instances per rank W = H + S (<= 32)
    const int W = d.E / d.R + d.S;
#define EP_PLAN_WB(wb)                                                                       \
    if (W <= wb)                                                                             \
        return launch_plan_r<wb>(d, counts, n_inst, max_iters, flags, quota, slot_expert, rank_load, \
                                 inst_ptr, inst_id, inst_cum, n_iter, inst_status, s, pdl);
    EP_PLAN_WB(2)
    EP_PLAN_WB(3)
    EP_PLAN_WB(4)
    EP_PLAN_WB(6)
    EP_PLAN_WB(8)
    EP_PLAN_WB(16)
#undef EP_PLAN_WB
    return launch_plan_r<32>(d, counts, n_inst, max_iters, flags, quota, slot_expert, rank_load,
                             inst_ptr, inst_id, inst_cum, n_iter, inst_status, s, pdl);
}

}  // namespace ultraep
