// Device code of the planner: the count checks, the shared-memory table move
// loops of the flag-free rule and of the rule variants, the register-cached
// loop of the skip variants (ranks of at most eight instances), and the
// logical->physical CSR epilogue.
//
// UltraEP article (m.youleyou.com), "key design" section, control-plane
// paragraph: the solver fixes the load (quota) every expert instance receives;
// each exploration step either instantiates a new replica or shifts load; it
// runs warp-parallel.  The rule itself (hot = argmax load, its largest
// instance, cold = least-loaded eligible rank, q = min(quota, floor(gap/2)),
// global stop) is the one documented in ultraep.h.
#pragma once

#include <climits>

#include "common.cuh"

namespace ultraep {

constexpr long long kPackLimit = 1ll << 25;  // total below this: loads fit a 6-bit-shifted key
constexpr long long kQPackLimit = 1ll << 21; // ... and quotas fit a 10-bit-shifted key

__host__ __device__ inline size_t align16(size_t x) { return (x + 15) & ~size_t(15); }

// floor(x / d) for 0 <= x < 2^21 and d >= 1, given inv_d = 1.0f / d (rounded
// to nearest, computed once by the caller).  (x + 1/2) / d lies at least
// 1 / (2d) away from every integer, and the two roundings in (x + 1/2) * inv_d
// change it by at most (x + 1/2) / d * 2^-22 < 1 / (2d), so truncation gives
// the exact quotient.  The planner's indices (instances, experts, slots) are
// far below 2^21; an integer division by a run-time value is a long
// instruction sequence, and these sit on the per-layer critical path.
__device__ __forceinline__ int small_div(int x, float inv_d) {
    return (int)(((float)x + 0.5f) * inv_d);
}

// One warp's shared memory: q[P], slot[R*S], holder[E] (the table), the CSR
// epilogue's scratch pos[E+1] and val[E+R*S], a copy of the loads Ls[64] (the
// rule variants), and the instance's counts[E] when the planner sums them
// itself (last).
__host__ __device__ inline size_t plan_warp_bytes(int R, int E, int S) {
    const int P = R * (E / R + S);
    return align16((size_t)P * 4) + align16((size_t)R * S * 4) + align16((size_t)E * 8) +
           align16((size_t)(E + 1) * 4) + align16((size_t)(E + R * S) * 4) + 64 * 4 +
           align16((size_t)E * 4);
}

// Hottest rank (lowest index on ties) and its load.
template <bool kTwo, bool kPacked>
__device__ __forceinline__ void argmax_rank(int la, int lb, bool hasA, bool hasB, int lane,
                                            int& hot, int& Lmax) {
    if (kPacked) {
        const unsigned ka = hasA ? ((unsigned)la << 6) | (unsigned)(63 - lane) : 0u;
        const unsigned kb = hasB ? ((unsigned)lb << 6) | (unsigned)(31 - lane) : 0u;
        const unsigned k = __reduce_max_sync(kFull, kTwo ? max(ka, kb) : ka);
        hot = (int)((k & 63u) ^ 63u);  // 63 - (k & 63)
        Lmax = (int)(k >> 6);
    } else {
        Lmax = __reduce_max_sync(kFull, kTwo ? max(la, lb) : la);
        const unsigned b0 = __ballot_sync(kFull, la == Lmax);
        const unsigned b1 = kTwo ? __ballot_sync(kFull, lb == Lmax) : 0u;
        hot = b0 ? __ffs(b0) - 1 : 32 + __ffs(b1) - 1;
    }
}

// The base rule on a shared-memory table (the flag-free kernel): the warp's
// instance quotas q[P] (rank-major, W per rank), the experts of the spare
// slots slot[R*S] (-1: empty) and, per expert, the mask of ranks holding it;
// the loads stay in registers (lane l: ranks l and l+32).  Per move the hot
// rank's largest instance is one warp reduction over its W instances (lane j:
// instance j), eligibility is one rank mask (holders of e | ranks with a free
// slot, each lane testing its own two bits), and the bookkeeping is a few
// single-lane stores, so nothing in a move grows with the instances per rank.
// The tables are exactly the epilogue's.
//
// Every quota and spare-slot entry of the table is read and written by one
// lane only: lane j owns local instance j of every rank (q[r*W + j] and, for
// j >= H, slot[r*S + j - H]); every lane writes the same value to a holder
// mask.  So each lane sees its own earlier writes in program order and a move
// needs no warp barrier before the next one reads the table: the bookkeeping
// of one move overlaps the search of the next.
//
// The moves form one dependent chain of warp reductions and shared-memory
// loads, issued in order by one warp, so every operation on it counts: rank
// masks are handled as two 32-bit halves (lane l tests bit l of each), and a
// rank holds e exactly when e is one of its home experts or one of its spare
// slots votes for e.
//
// kQPacked (total below 2^21): the hot rank's largest instance (lowest expert
// on ties) is one max-reduction over the key quota << 10 | 1023 - e; lanes
// without an instance offer 1024 - E, the key of expert E - 1 at quota 0,
// which can only win when every quota of the rank is 0 (then nothing moves).
template <bool kTwo, bool kPacked, bool kQPacked>
__device__ __forceinline__ void plan_moves_table(int32_t* q, int32_t* slot, uint64_t* holder,
                                                 int& loadA, int& loadB, int lane, int H, int S,
                                                 int W, int R, int E, int max_iters, int& iters,
                                                 int& status) {
    const bool hasA = loadA >= 0, hasB = kTwo && loadB >= 0;
    const int ra = lane, rb = lane + 32;
    // ranks with a free spare slot, as two halves (ranks 0-31, 32-63); a lane
    // only tests the bits of its own ranks, which exist
    unsigned freeLo = S > 0 ? ~0u : 0u, freeHi = freeLo;
    const bool owner = lane < W;            // lane j owns local instance j
    const bool spare = lane >= H && owner;  // ... a spare slot of every rank
    const unsigned lt = lanemask_lt();
    const unsigned noInst = (unsigned)(1024 - E);
    int hot, Lmax;
    argmax_rank<kTwo, kPacked>(loadA, loadB, hasA, hasB, lane, hot, Lmax);
    while (true) {
        // 2. hot's largest-quota instance, lowest expert on ties (lane j:
        // instance j; every rank has its H >= 1 home instances)
        int xj = -1, qv = 0;
        if (owner) {  // the two loads are independent
            xj = lane < H ? hot * H + lane : slot[hot * S + (lane - H)];
            qv = q[hot * W + lane];
        }
        int qmax, e;
        bool mine;  // this lane owns the instance that gives
        if (kQPacked) {
            const unsigned key = (xj >= 0) ? (((unsigned)qv << 10) | (unsigned)(1023 - xj)) : noInst;
            const unsigned kmax = __reduce_max_sync(kFull, key);
            qmax = (int)(kmax >> 10);
            e = 1023 - (int)(kmax & 1023u);
            mine = key == kmax;
        } else {
            const int qj = xj >= 0 ? qv : -1;
            const unsigned cxj = xj >= 0 ? (((unsigned)xj << 5) | (unsigned)lane) : 0xffffffffu;
            qmax = __reduce_max_sync(kFull, qj);
            const unsigned cx = __reduce_min_sync(kFull, qj == qmax ? cxj : 0xffffffffu);
            e = (int)(cx >> 5);
            mine = lane == (int)(cx & 31u);
        }

        // 3-5. eligible ranks: the others that hold e or have a free slot;
        // the coldest of them (lowest rank on ties) and the amount.  With no
        // eligible rank the reduction keeps its identity, which gives an
        // amount <= 0; the stop conditions and the cap are one branch.
        const uint64_t hm = holder[e];
        const unsigned mLo = (unsigned)hm | freeLo, mHi = (unsigned)(hm >> 32) | freeHi;
        const bool elA = hasA && ra != hot && ((mLo >> lane) & 1u);
        const bool elB = hasB && rb != hot && ((mHi >> lane) & 1u);
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
        // 6. stop: no rank eligible, or nothing to move (the global stop);
        // else the safety cap
        if (mv <= 0 || iters == max_iters) {
            if (mv > 0) status = EP_ERR_ITER_LIMIT;
            break;
        }
        // 7. move.  Loads first, then the next move's argmax ...
        loadA += (ra == cold ? mv : 0) - (ra == hot ? mv : 0);
        if (kTwo) loadB += (rb == cold ? mv : 0) - (rb == hot ? mv : 0);
        int nhot, nLmax;
        argmax_rank<kTwo, kPacked>(loadA, loadB, hasA, hasB, lane, nhot, nLmax);
        // ... and the tables: cold's instance of e is its home, a spare slot
        // already holding e, or its lowest free spare slot (filled now).  The
        // owner lanes read cold's spare slot and quota unconditionally and vote
        // on the slots; each lane then tests whether it is the instance (no
        // bit scan), so this overlaps the argmax above.
        const int sv = spare ? slot[cold * S + (lane - H)] : 0;
        const int qc = owner ? q[cold * W + lane] : 0;
        const unsigned hit = __ballot_sync(kFull, spare && sv == e);
        const unsigned freeb = __ballot_sync(kFull, spare && sv < 0);  // cold's free slots
        const int ej = e - cold * H;
        const bool home = (unsigned)ej < (unsigned)H;  // e is one of cold's home experts
        const bool held = home || hit != 0u;
        const unsigned pick = held ? hit : freeb;       // nonzero unless home: cold is eligible
        if (!home && pick == 0u) {                      // (never; keeps every index in range)
            status = EP_ERR_INVAL;
            break;
        }
        // this lane is cold's instance: e's home, else the lowest lane of pick
        const bool dst = home ? lane == ej : ((pick >> lane) & 1u) && (pick & lt) == 0u;
        // owner-lane updates, no read-modify-write across lanes
        if (mine) q[hot * W + lane] = qv - mv;
        if (dst) {
            q[cold * W + lane] = qc + mv;
            if (!held) slot[cold * S + (lane - H)] = e;
        }
        // cold now holds e (a no-op when it held it already); its last free
        // slot taken: it has none left
        const unsigned bit = 1u << (cold & 31);
        const bool lo = cold < 32;
        holder[e] = hm | ((uint64_t)(lo ? 0u : bit) << 32) | (lo ? bit : 0u);  // every lane
        const unsigned full = (!held && (freeb & (freeb - 1u)) == 0u) ? bit : 0u;
        freeLo &= lo ? ~full : ~0u;
        freeHi &= lo ? ~0u : ~full;
        hot = nhot;
        Lmax = nLmax;
        ++iters;
    }
}

// The rule variants of ep_plan_ex on the same shared-memory table.
//   EP_PLAN_SKIP: the move is the first (rank, instance) candidate that can
//   move, in the order ranks by load (highest first, lowest index on ties),
//   then a rank's instances with quota >= 1 by quota (largest first, lowest
//   expert on ties).  A candidate (c, e) can move exactly when some eligible
//   rank d != c (holding e, or with a free slot) has L[d] <= L[c] - 2: the
//   coldest eligible rank then gives q >= 1.  So every lane evaluates its own
//   ranks at once: each rank's mask of the ranks at least 2 below its load,
//   then each of the rank's instances against (holders of e | ranks with a
//   free slot); one reduction over the ranks that have a movable instance
//   picks the candidate.  A move costs the same however many candidates
//   cannot move.  The masks are built once (from a shared-memory copy of the
//   loads) and then kept: a move changes two loads, so every other rank
//   re-tests two bits, and the two ranks that moved take their masks from
//   two ballots each over the new loads.
//   EP_PLAN_RELEASE: a spare-slot instance a move leaves at quota 0 frees its
//   slot (its rank no longer holds the expert; the slot is free again).
// Without EP_PLAN_SKIP the candidate is the base rule's (the hottest rank's
// largest instance with quota >= 1) and the plan stops when it cannot move.
// Ls[64] is scratch for the loads; ranks >= R hold INT_MAX.
template <bool kTwo, bool kPacked>
__device__ __forceinline__ void plan_moves_table_flags(int32_t* q, int32_t* slot,
                                                       uint64_t* holder, int32_t* Ls,
                                                       int& loadA, int& loadB, int lane, int H,
                                                       int S, int W, int R, int max_iters,
                                                       int flags, int& iters, int& status) {
    const bool skip = (flags & EP_PLAN_SKIP) != 0;
    const bool release = (flags & EP_PLAN_RELEASE) != 0;
    const unsigned lt = lanemask_lt();
    const bool hasA = loadA >= 0, hasB = kTwo && loadB >= 0;
    const int ra = lane, rb = lane + 32;
    const uint64_t exist = (R >= 64) ? ~0ull : ((1ull << R) - 1ull);
    uint64_t freem = S > 0 ? exist : 0ull;  // ranks with a free spare slot (warp-uniform)
    Ls[ra] = hasA ? loadA : INT_MAX;
    Ls[rb] = hasB ? loadB : INT_MAX;
    __syncwarp();
    // my ranks' masks of the ranks at least 2 below them (a rank is never
    // below itself), as halves: ranks 0-31 and 32-63
    unsigned loA = 0u, hiA = 0u, loB = 0u, hiB = 0u;
    if (skip) {
        const int tA = loadA - 2, tB = loadB - 2;
#pragma unroll 4
        for (int d = 0; d < 32; d += 4) {
            const int4 v = *reinterpret_cast<const int4*>(Ls + d);
            const int4 w = *reinterpret_cast<const int4*>(Ls + 32 + d);
            loA |= ((unsigned)(v.x <= tA) | (unsigned)(v.y <= tA) << 1 |
                    (unsigned)(v.z <= tA) << 2 | (unsigned)(v.w <= tA) << 3) << d;
            hiA |= ((unsigned)(w.x <= tA) | (unsigned)(w.y <= tA) << 1 |
                    (unsigned)(w.z <= tA) << 2 | (unsigned)(w.w <= tA) << 3) << d;
            if (kTwo) {
                loB |= ((unsigned)(v.x <= tB) | (unsigned)(v.y <= tB) << 1 |
                        (unsigned)(v.z <= tB) << 2 | (unsigned)(v.w <= tB) << 3) << d;
                hiB |= ((unsigned)(w.x <= tB) | (unsigned)(w.y <= tB) << 1 |
                        (unsigned)(w.z <= tB) << 2 | (unsigned)(w.w <= tB) << 3) << d;
            }
        }
    }
    // the best instance (largest quota >= 1, lowest expert) of each of my two
    // ranks whose expert has an eligible rank in that rank's low mask; bq = -1
    // when there is none.  The two ranks' loads are issued together and the
    // tests are selects.
    auto best_movable2 = [&](uint64_t lowA, uint64_t lowB, int& bqA, int& beA, int& bjA,
                             int& bqB, int& beB, int& bjB) {
        bqA = bqB = -1;
        beA = beB = INT_MAX;
        bjA = bjB = 0;
        const bool tA = hasA && lowA != 0ull, tB = hasB && lowB != 0ull;
        if (!tA && !tB) return;
        for (int j = 0; j < W; ++j) {
            const bool home = j < H;
            const int exA = home ? ra * H + j : (tA ? slot[ra * S + (j - H)] : -1);
            const int exB = home ? rb * H + j : (tB ? slot[rb * S + (j - H)] : -1);
            const int qA = tA ? q[ra * W + j] : 0;
            const int qB = tB ? q[rb * W + j] : 0;
            const uint64_t hA = (tA && exA >= 0) ? holder[exA] : 0ull;
            const uint64_t hB = (tB && exB >= 0) ? holder[exB] : 0ull;
            const bool okA = tA && exA >= 0 && qA >= 1 && (qA > bqA || (qA == bqA && exA < beA)) &&
                             ((hA | freem) & lowA) != 0ull;
            const bool okB = tB && exB >= 0 && qB >= 1 && (qB > bqB || (qB == bqB && exB < beB)) &&
                             ((hB | freem) & lowB) != 0ull;
            bqA = okA ? qA : bqA;
            beA = okA ? exA : beA;
            bjA = okA ? j : bjA;
            bqB = okB ? qB : bqB;
            beB = okB ? exB : beB;
            bjB = okB ? j : bjB;
        }
    };
    while (true) {
        int c, Lc, e, qsrc, src_j;  // the candidate (warp-uniform)
        if (skip) {
            int bqA, beA, bjA, bqB, beB, bjB;
            best_movable2(((uint64_t)hiA << 32) | loA, kTwo ? ((uint64_t)hiB << 32) | loB : 0ull,
                          bqA, beA, bjA, bqB, beB, bjB);
            // the first rank in (load desc, index asc) order with a movable instance
            const bool mA = bqA >= 1, mB = kTwo && bqB >= 1;
            if (kPacked) {
                const unsigned ka = mA ? ((unsigned)loadA << 6) | (unsigned)(63 - ra) : 0u;
                const unsigned kb = mB ? ((unsigned)loadB << 6) | (unsigned)(31 - lane) : 0u;
                const unsigned k = __reduce_max_sync(kFull, kTwo ? max(ka, kb) : ka);
                if (k == 0u) break;  // no candidate can move
                c = 63 - (int)(k & 63u);
                Lc = (int)(k >> 6);
            } else {
                const int la = mA ? loadA : -1, lb = mB ? loadB : -1;
                Lc = __reduce_max_sync(kFull, kTwo ? max(la, lb) : la);
                if (Lc < 0) break;
                const unsigned b0 = __ballot_sync(kFull, mA && la == Lc);
                const unsigned b1 = kTwo ? __ballot_sync(kFull, mB && lb == Lc) : 0u;
                c = b0 ? __ffs(b0) - 1 : 32 + __ffs(b1) - 1;
            }
            const bool cB = c >= 32;
            const int cl = c & 31;
            qsrc = __shfl_sync(kFull, cB ? bqB : bqA, cl);
            e = __shfl_sync(kFull, cB ? beB : beA, cl);
            src_j = __shfl_sync(kFull, cB ? bjB : bjA, cl);
        } else {
            // the base candidate: the hottest rank's largest instance with quota >= 1
            argmax_rank<kTwo, kPacked>(loadA, loadB, hasA, hasB, lane, c, Lc);
            int qj = -1;
            unsigned cxj = 0xffffffffu;
            if (lane < W) {
                const int xj = lane < H ? c * H + lane : slot[c * S + (lane - H)];
                const int qv = q[c * W + lane];
                if (xj >= 0 && qv >= 1) {
                    qj = qv;
                    cxj = ((unsigned)xj << 5) | (unsigned)lane;
                }
            }
            qsrc = __reduce_max_sync(kFull, qj);
            if (qsrc < 1) break;
            const unsigned cx = __reduce_min_sync(kFull, qj == qsrc ? cxj : 0xffffffffu);
            e = (int)(cx >> 5);
            src_j = (int)(cx & 31u);
        }
        // the coldest eligible rank (lowest index on ties) and the amount
        const uint64_t hm = holder[e];
        const uint64_t el = (hm | freem) & exist & ~(1ull << c);
        if (el == 0ull) break;  // (base candidate only)
        const bool elA = hasA && (((unsigned)el >> lane) & 1u);
        const bool elB = hasB && (((unsigned)(el >> 32) >> lane) & 1u);
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
        // the table entries the move touches, read by their owner lanes (lane
        // j: instance j of a rank) while the move is decided
        const bool owner = lane < W, spare = owner && lane >= H;
        const int qs = owner ? q[c * W + lane] : 0;      // c's instances
        const int qc = owner ? q[cold * W + lane] : 0;   // cold's instances
        const int sv = spare ? slot[cold * S + (lane - H)] : 0;  // cold's spare slots
        const int mv = min(qsrc, (Lc - Lmin) >> 1);
        if (mv <= 0) break;  // (base candidate only: a skip candidate always moves)
        if (iters == max_iters) {
            status = EP_ERR_ITER_LIMIT;
            break;
        }
        // the move: loads, then cold's instance of e (its home, a spare slot
        // holding e, or its lowest free slot, filled now)
        loadA += (ra == cold ? mv : 0) - (ra == c ? mv : 0);
        if (kTwo) loadB += (rb == cold ? mv : 0) - (rb == c ? mv : 0);
        if (skip) {
            // the masks: c and cold from ballots over the new loads; every
            // other rank re-tests bits c and cold
            const int nLc = Lc - mv, nLd = Lmin + mv;
            const unsigned cLo = __ballot_sync(kFull, hasA && loadA <= nLc - 2);
            const unsigned cHi = kTwo ? __ballot_sync(kFull, hasB && loadB <= nLc - 2) : 0u;
            const unsigned dLo = __ballot_sync(kFull, hasA && loadA <= nLd - 2);
            const unsigned dHi = kTwo ? __ballot_sync(kFull, hasB && loadB <= nLd - 2) : 0u;
            const unsigned bc = 1u << (c & 31), bd = 1u << (cold & 31);
            const bool cLoHalf = c < 32, dLoHalf = cold < 32;
            auto retest = [&](int r, int L, unsigned& lo, unsigned& hi) {
                if (r == c) {
                    lo = cLo;
                    hi = cHi;
                } else if (r == cold) {
                    lo = dLo;
                    hi = dHi;
                } else {
                    const unsigned sc = nLc <= L - 2 ? bc : 0u, sd = nLd <= L - 2 ? bd : 0u;
                    if (cLoHalf) lo = (lo & ~bc) | sc;
                    else hi = (hi & ~bc) | sc;
                    if (dLoHalf) lo = (lo & ~bd) | sd;
                    else hi = (hi & ~bd) | sd;
                }
            };
            if (hasA) retest(ra, loadA, loA, hiA);
            if (hasB) retest(rb, loadB, loB, hiB);
        }
        // cold holds e as a home expert or in a spare slot (lane j votes for
        // instance j); else its lowest free slot takes e
        const unsigned hit = __ballot_sync(kFull, spare && sv == e);
        const unsigned freeb = __ballot_sync(kFull, spare && sv < 0);  // cold's free slots
        const int ej = e - cold * H;
        const bool home = (unsigned)ej < (unsigned)H;
        const bool held = home || hit != 0u;
        const unsigned pick = held ? hit : freeb;
        if (!home && pick == 0u) {  // (never; keeps every index in range)
            status = EP_ERR_INVAL;
            break;
        }
        // this lane is cold's instance: e's home, else the lowest lane of pick
        const bool dst = home ? lane == ej : ((pick >> lane) & 1u) && (pick & lt) == 0u;
        const bool freed = release && src_j >= H && qsrc == mv;  // the source replica emptied
        // owner-lane updates (c != cold, so no entry is written twice)
        if (lane == src_j) {
            q[c * W + lane] = qs - mv;
            if (freed) slot[c * S + (lane - H)] = -1;
        }
        if (dst) {
            q[cold * W + lane] = qc + mv;
            if (!held) slot[cold * S + (lane - H)] = e;
        }
        uint64_t h2 = held ? hm : (hm | (1ull << cold));
        if (freed) h2 &= ~(1ull << c);
        holder[e] = h2;  // every lane, the same value
        if (!held && (freeb & (freeb - 1u)) == 0u) freem &= ~(1ull << cold);  // its last free slot
        if (freed) freem |= 1ull << c;
        __syncwarp();  // the table, for every lane's next reads
        ++iters;
    }
}

// EP_PLAN_SKIP (with or without EP_PLAN_RELEASE) when a rank has kW <=
// kCachedW instances (W, a template parameter so that the loops over a
// rank's instances are exact): the same moves as plan_moves_table_flags, with each
// lane's own ranks' instances kept in registers: the expert of every
// instance (-1: a free spare slot), its quota and its expert's holder mask.
// A rank's best movable instance is then a pass over registers instead of
// dependent shared-memory reads (slot, quota, holder) on every move.  A move
// changes two quotas (on the lanes of c and of the receiving rank), maybe one
// spare slot on each of those ranks, and the holder mask of the moved expert,
// which every lane copies into each of its instances of that expert.  The
// shared-memory table is written back from the caches when the loop ends.
constexpr int kCachedW = 8;

template <int kN>
struct RankCache {
    int x[kN];       // expert of instance j (-1: a free spare slot)
    int q[kN];       // quota of instance j
    uint64_t h[kN];  // holder mask of that expert
};

template <bool kTwo, bool kPacked, int kW>
__device__ __forceinline__ void plan_moves_skip_cached(int32_t* q, int32_t* slot,
                                                       uint64_t* holder, int32_t* Ls,
                                                       int& loadA, int& loadB, int lane, int H,
                                                       int S, int R, int max_iters, int flags,
                                                       int& iters, int& status) {
    constexpr int W = kW;
    const bool release = (flags & EP_PLAN_RELEASE) != 0;
    const bool hasA = loadA >= 0, hasB = kTwo && loadB >= 0;
    const int ra = lane, rb = lane + 32;
    const uint64_t exist = (R >= 64) ? ~0ull : ((1ull << R) - 1ull);
    uint64_t freem = S > 0 ? exist : 0ull;  // ranks with a free spare slot (warp-uniform)
    // the caches of my ranks' instances
    RankCache<kW> A, B;
    auto fill = [&](RankCache<kW>& C, bool has, int r) {
#pragma unroll
        for (int j = 0; j < kW; ++j) {
            int x = -1, qq = 0;
            uint64_t hh = 0ull;
            if (has) {
                x = j < H ? r * H + j : slot[r * S + (j - H)];
                qq = q[r * W + j];
                hh = x >= 0 ? holder[x] : 0ull;
            }
            C.x[j] = x;
            C.q[j] = qq;
            C.h[j] = hh;
        }
    };
    fill(A, hasA, ra);
    if (kTwo) fill(B, hasB, rb);
    // my ranks' masks of the ranks at least 2 below them, as halves
    Ls[ra] = hasA ? loadA : INT_MAX;
    Ls[rb] = hasB ? loadB : INT_MAX;
    __syncwarp();
    unsigned loA = 0u, hiA = 0u, loB = 0u, hiB = 0u;
    {
        const int tA = loadA - 2, tB = loadB - 2;
#pragma unroll 4
        for (int d = 0; d < 32; d += 4) {
            const int4 v = *reinterpret_cast<const int4*>(Ls + d);
            const int4 w = *reinterpret_cast<const int4*>(Ls + 32 + d);
            loA |= ((unsigned)(v.x <= tA) | (unsigned)(v.y <= tA) << 1 |
                    (unsigned)(v.z <= tA) << 2 | (unsigned)(v.w <= tA) << 3) << d;
            hiA |= ((unsigned)(w.x <= tA) | (unsigned)(w.y <= tA) << 1 |
                    (unsigned)(w.z <= tA) << 2 | (unsigned)(w.w <= tA) << 3) << d;
            if (kTwo) {
                loB |= ((unsigned)(v.x <= tB) | (unsigned)(v.y <= tB) << 1 |
                        (unsigned)(v.z <= tB) << 2 | (unsigned)(v.w <= tB) << 3) << d;
                hiB |= ((unsigned)(w.x <= tB) | (unsigned)(w.y <= tB) << 1 |
                        (unsigned)(w.z <= tB) << 2 | (unsigned)(w.w <= tB) << 3) << d;
            }
        }
    }
    // a rank's best instance (largest quota >= 1, lowest expert) whose expert
    // has an eligible rank in the rank's low mask, as the key
    // quota << 32 | (2047 - expert) << 5 | j (0: none).  The instances are
    // tested independently and the keys meet in a max (experts are below
    // 2048 and distinct within a rank).  A quota >= 1 implies an expert (a
    // free slot has quota 0), and a lane without the rank caches free slots.
    auto best = [&](const RankCache<kW>& C, uint64_t low) -> uint64_t {
        uint64_t k = 0ull;
#pragma unroll
        for (int j = 0; j < kW; ++j) {
            const int x = C.x[j], qq = C.q[j];
            const bool ok = qq >= 1 && ((C.h[j] | freem) & low) != 0ull;
            const uint64_t kj = ok ? ((uint64_t)(unsigned)qq << 32) |
                                         ((unsigned)(2047 - x) << 5) | (unsigned)j
                                   : 0ull;
            k = kj > k ? kj : k;
        }
        return k;
    };
    while (true) {
        const uint64_t kA = best(A, ((uint64_t)hiA << 32) | loA);
        const uint64_t kB = kTwo ? best(B, ((uint64_t)hiB << 32) | loB) : 0ull;
        // the first rank in (load desc, index asc) order with a movable instance
        const bool mA = kA != 0ull, mB = kTwo && kB != 0ull;
        int c, Lc;
        if (kPacked) {
            const unsigned ka = mA ? ((unsigned)loadA << 6) | (unsigned)(63 - ra) : 0u;
            const unsigned kb = mB ? ((unsigned)loadB << 6) | (unsigned)(31 - lane) : 0u;
            const unsigned k = __reduce_max_sync(kFull, kTwo ? max(ka, kb) : ka);
            if (k == 0u) break;  // no candidate can move
            c = 63 - (int)(k & 63u);
            Lc = (int)(k >> 6);
        } else {
            const int la = mA ? loadA : -1, lb = mB ? loadB : -1;
            Lc = __reduce_max_sync(kFull, kTwo ? max(la, lb) : la);
            if (Lc < 0) break;
            const unsigned b0 = __ballot_sync(kFull, mA && la == Lc);
            const unsigned b1 = kTwo ? __ballot_sync(kFull, mB && lb == Lc) : 0u;
            c = b0 ? __ffs(b0) - 1 : 32 + __ffs(b1) - 1;
        }
        const bool cB = c >= 32;
        const int cl = c & 31;
        // c's best instance and its expert's holder mask, from c's lane
        const uint64_t kc = cB ? kB : kA;
        const int jc = (int)(kc & 31u);
        uint64_t bh = 0ull;
#pragma unroll
        for (int j = 0; j < kW; ++j) bh = j == jc ? (cB ? B.h[j] : A.h[j]) : bh;
        const int qsrc = (int)__shfl_sync(kFull, (unsigned)(kc >> 32), cl);
        const unsigned lo_key = __shfl_sync(kFull, (unsigned)kc, cl);
        const int e = 2047 - (int)(lo_key >> 5);
        const int src_j = (int)(lo_key & 31u);
        const uint64_t hm = ((uint64_t)__shfl_sync(kFull, (unsigned)(bh >> 32), cl) << 32) |
                            (uint64_t)__shfl_sync(kFull, (unsigned)bh, cl);
        // the coldest eligible rank (lowest index on ties)
        const uint64_t el = (hm | freem) & exist & ~(1ull << c);
        const bool elA = hasA && (((unsigned)el >> lane) & 1u);
        const bool elB = hasB && (((unsigned)(el >> 32) >> lane) & 1u);
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
        // the receiving rank's spare slots holding e, and its free ones (bit
        // j: instance j), from the lane that caches that rank
        unsigned hitA = 0u, freeA = 0u, hitB = 0u, freeB = 0u;
#pragma unroll
        for (int j = 0; j < kW; ++j) {
            if (j >= H) {
                hitA |= (A.x[j] == e ? 1u : 0u) << j;
                freeA |= (A.x[j] < 0 ? 1u : 0u) << j;
                if (kTwo) {
                    hitB |= (B.x[j] == e ? 1u : 0u) << j;
                    freeB |= (B.x[j] < 0 ? 1u : 0u) << j;
                }
            }
        }
        const bool dB = cold >= 32;
        const unsigned hf = __shfl_sync(kFull, dB ? (hitB | freeB << 16) : (hitA | freeA << 16),
                                        cold & 31);
        const unsigned hit = hf & 0xffffu, freeb = hf >> 16;
        const int mv = min(qsrc, (Lc - Lmin) >> 1);
        if (mv <= 0) break;  // (never: a movable candidate has a rank 2 below it)
        if (iters == max_iters) {
            status = EP_ERR_ITER_LIMIT;
            break;
        }
        // the move: loads, then the masks (c and cold from ballots over the new
        // loads; every other rank re-tests bits c and cold)
        loadA += (ra == cold ? mv : 0) - (ra == c ? mv : 0);
        if (kTwo) loadB += (rb == cold ? mv : 0) - (rb == c ? mv : 0);
        {
            const int nLc = Lc - mv, nLd = Lmin + mv;
            const unsigned cLo = __ballot_sync(kFull, hasA && loadA <= nLc - 2);
            const unsigned cHi = kTwo ? __ballot_sync(kFull, hasB && loadB <= nLc - 2) : 0u;
            const unsigned dLo = __ballot_sync(kFull, hasA && loadA <= nLd - 2);
            const unsigned dHi = kTwo ? __ballot_sync(kFull, hasB && loadB <= nLd - 2) : 0u;
            const unsigned bc = 1u << (c & 31), bd = 1u << (cold & 31);
            const bool cLoHalf = c < 32, dLoHalf = cold < 32;
            // (selects, no divergent branches: every lane takes the same path)
            const unsigned mcLo = cLoHalf ? bc : 0u, mcHi = cLoHalf ? 0u : bc;
            const unsigned mdLo = dLoHalf ? bd : 0u, mdHi = dLoHalf ? 0u : bd;
            auto retest = [&](int r, int L, unsigned& lo, unsigned& hi) {
                const bool sc = nLc <= L - 2, sd = nLd <= L - 2;
                const unsigned nlo = (lo & ~(mcLo | mdLo)) | (sc ? mcLo : 0u) | (sd ? mdLo : 0u);
                const unsigned nhi = (hi & ~(mcHi | mdHi)) | (sc ? mcHi : 0u) | (sd ? mdHi : 0u);
                lo = r == c ? cLo : (r == cold ? dLo : nlo);
                hi = r == c ? cHi : (r == cold ? dHi : nhi);
            };
            if (hasA) retest(ra, loadA, loA, hiA);
            if (hasB) retest(rb, loadB, loB, hiB);
        }
        // cold's instance of e: its home, a spare slot holding e, else its
        // lowest free slot
        const int ej = e - cold * H;
        const bool home = (unsigned)ej < (unsigned)H;
        const bool held = home || hit != 0u;
        const unsigned pick = held ? hit : freeb;
        if (!home && pick == 0u) {  // (never; keeps every index in range)
            status = EP_ERR_INVAL;
            break;
        }
        const int dst_j = home ? ej : __ffs(pick) - 1;
        const bool freed = release && src_j >= H && qsrc == mv;  // the source replica emptied
        uint64_t h2 = held ? hm : (hm | (1ull << cold));
        if (freed) h2 &= ~(1ull << c);
        // the caches (selects only): c's instance src_j and cold's instance
        // dst_j, then the holder mask of every cached instance of e
        auto apply = [&](RankCache<kW>& C, int r) {
            const int sj = r == c ? src_j : -1, dj = r == cold ? dst_j : -1;
#pragma unroll
            for (int j = 0; j < kW; ++j) {
                const bool js = j == sj, jd = j == dj;
                C.q[j] = js ? C.q[j] - mv : (jd ? C.q[j] + mv : C.q[j]);
                C.x[j] = (js && freed) ? -1 : ((jd && !held) ? e : C.x[j]);
                C.h[j] = C.x[j] == e ? h2 : C.h[j];  // (a free slot's is never read)
            }
        };
        apply(A, ra);
        if (kTwo) apply(B, rb);
        if (!held && (freeb & (freeb - 1u)) == 0u) freem &= ~(1ull << cold);  // its last free slot
        if (freed) freem |= 1ull << c;
        ++iters;
    }
    // the table from the caches: each lane its ranks' quotas and spare slots,
    // and the holder mask of each of their home experts (every expert has
    // one home rank, whose cache holds its current mask)
    auto write_back = [&](const RankCache<kW>& C, bool has, int r) {
        if (!has) return;
#pragma unroll
        for (int j = 0; j < kW; ++j) {
            q[r * W + j] = C.q[j];
            if (j >= H) slot[r * S + (j - H)] = C.x[j];
            else holder[C.x[j]] = C.h[j];
        }
    };
    write_back(A, hasA, ra);
    if (kTwo) write_back(B, hasB, rb);
    __syncwarp();
}

// The skip rule on the cached loop when W <= kCachedW; false: not handled.
template <bool kTwo, bool kPacked>
__device__ __forceinline__ bool plan_moves_skip_cached_w(int32_t* q, int32_t* slot,
                                                         uint64_t* holder, int32_t* Ls,
                                                         int& loadA, int& loadB, int lane, int H,
                                                         int S, int W, int R, int max_iters,
                                                         int flags, int& iters, int& status) {
#define EP_SKIP_CACHED_CASE(w)                                                                    \
    case w:                                                                                       \
        plan_moves_skip_cached<kTwo, kPacked, w>(q, slot, holder, Ls, loadA, loadB, lane, H, S, R, \
                                                 max_iters, flags, iters, status);                \
        return true;
    switch (W) {
        EP_SKIP_CACHED_CASE(1)
        EP_SKIP_CACHED_CASE(2)
        EP_SKIP_CACHED_CASE(3)
        EP_SKIP_CACHED_CASE(4)
        EP_SKIP_CACHED_CASE(5)
        EP_SKIP_CACHED_CASE(6)
        EP_SKIP_CACHED_CASE(7)
        EP_SKIP_CACHED_CASE(8)
        default:
            return false;
    }
#undef EP_SKIP_CACHED_CASE
}

// Counts must be >= 0 with a total below 2^31; otherwise the instance is
// rejected (EP_ERR_INVAL).  tot: the warp-uniform total.
__device__ __forceinline__ int plan_check_counts(const int32_t* cnt, int E, int lane,
                                                 long long& tot) {
    bool bad = false;
    tot = 0;
    for (int e = lane; e < E; e += 32) {
        const int v = cnt[e];
        bad |= v < 0;
        tot += v;
    }
    bad = __any_sync(kFull, bad);
    for (int o = 16; o > 0; o >>= 1) tot += __shfl_xor_sync(kFull, tot, o);
    return (bad || tot > (long long)INT_MAX) ? EP_ERR_INVAL : EP_OK;
}

// One instance on the shared-memory tables q[P], slot[R*S], holder[E]
// (plan_warp_bytes): the home placement from cnt, the move loop of the rule
// (kFlags: the variants of `flags`; only while status is EP_OK), then quota,
// spare slots and loads to qo / so / lo.  One warp; kTwo: R > 32.
template <bool kTwo, bool kFlags>
__device__ __forceinline__ void plan_table_solve(const int32_t* cnt, int R, int E, int S,
                                                 int max_iters, int flags, long long tot,
                                                 int32_t* q, int32_t* slot, uint64_t* holder,
                                                 int32_t* Ls, int lane, int32_t* qo, int32_t* so,
                                                 int32_t* lo, int& iters, int& status) {
    const int H = E / R, W = H + S, P = R * W;
    const float invW = 1.0f / (float)W, invH = 1.0f / (float)H;
    for (int p = lane; p < P; p += 32) {
        const int r = small_div(p, invW), j = p - r * W;
        q[p] = j < H ? cnt[r * H + j] : 0;
    }
    for (int x = lane; x < R * S; x += 32) slot[x] = -1;
    for (int e = lane; e < E; e += 32) holder[e] = 1ull << small_div(e, invH);
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
    if (kFlags) {
        bool done = false;
        if (status == EP_OK && (flags & EP_PLAN_SKIP) && W <= kCachedW)
            done = tot < kPackLimit
                       ? plan_moves_skip_cached_w<kTwo, true>(q, slot, holder, Ls, loadA, loadB,
                                                              lane, H, S, W, R, max_iters, flags,
                                                              iters, status)
                       : plan_moves_skip_cached_w<kTwo, false>(q, slot, holder, Ls, loadA, loadB,
                                                               lane, H, S, W, R, max_iters, flags,
                                                               iters, status);
        if (!done && status == EP_OK) {
            if (tot < kPackLimit)
                plan_moves_table_flags<kTwo, true>(q, slot, holder, Ls, loadA, loadB, lane, H, S,
                                                   W, R, max_iters, flags, iters, status);
            else
                plan_moves_table_flags<kTwo, false>(q, slot, holder, Ls, loadA, loadB, lane, H, S,
                                                    W, R, max_iters, flags, iters, status);
        }
    } else if (status == EP_OK) {
        if (tot < kQPackLimit)
            plan_moves_table<kTwo, true, true>(q, slot, holder, loadA, loadB, lane, H, S, W, R,
                                               E, max_iters, iters, status);
        else if (tot < kPackLimit)
            plan_moves_table<kTwo, true, false>(q, slot, holder, loadA, loadB, lane, H, S, W, R,
                                                E, max_iters, iters, status);
        else
            plan_moves_table<kTwo, false, false>(q, slot, holder, loadA, loadB, lane, H, S, W,
                                                 R, E, max_iters, iters, status);
    }
    __syncwarp();  // the table's entries, written by their owner lanes, for every lane
    for (int p = lane; p < P; p += 32) qo[p] = q[p];
    for (int x = lane; x < R * S; x += 32) so[x] = slot[x];
    if (lane < R) lo[lane] = loadA;
    if (kTwo && lane + 32 < R) lo[lane + 32] = loadB;
}

// Logical -> physical CSR from the tables: for each expert its home instance
// first, then its replicas by ascending rank (= ascending p), with inclusive
// cumulative quotas.  The whole block (kThreads threads) builds one instance's
// lists: a block scan over the holder counts gives the list offsets (writes
// po[0..E] and the home entries); every spare slot then finds its own place
// in its expert's list (1 + its expert's replicas on lower ranks); the
// running sums are one segmented block scan over all entries (a list starts
// at its home entry), so a hot expert's long list costs no more than a short
// one.  pos[E+1] and val[E+R*S] are shared-memory scratch (the offsets, and
// each entry's quota with bit 31 set on a list's first entry),
// wtot[kThreads/32] the scans' warp totals.  Called by every thread of the
// block; starts and ends with a block barrier's worth of ordering.
template <int kThreads>
__device__ __forceinline__ void plan_csr_block(const int32_t* q, const int32_t* slot,
                                               const uint64_t* holder, int R, int E, int S,
                                               int32_t* pos, int32_t* val, int* wtot,
                                               int32_t* po, int32_t* io, int32_t* co) {
    constexpr int kWarps = kThreads / 32;
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int H = E / R, W = H + S;
    const float invH = 1.0f / (float)H, invS = 1.0f / (float)max(S, 1);
    // thread t: experts [t*per, (t+1)*per)
    const int per = (E + kThreads - 1) / kThreads;
    const int e0 = min(E, tid * per), e1 = min(E, e0 + per);
    int n = 0;
    for (int e = e0; e < e1; ++e) n += __popcll(holder[e]);
    int x = n;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const int y = __shfl_up_sync(kFull, x, o);
        if (lane >= o) x += y;
    }
    if (lane == 31) wtot[warp] = x;
    __syncthreads();
    int below = 0, total = 0;
#pragma unroll
    for (int w = 0; w < kWarps; ++w) {
        const int t = wtot[w];
        below += (w < warp) ? t : 0;
        total += t;
    }
    int run = below + x - n;
    for (int e = e0; e < e1; ++e) {
        pos[e] = run;
        po[e] = run;
        const int home = small_div(e, invH);
        const int hp = home * W + (e - home * H);  // the home instance heads the list
        io[run] = hp;
        val[run] = q[hp] | INT_MIN;  // a list's first entry
        run += __popcll(holder[e]);
    }
    if (tid == 0) {
        pos[E] = total;
        po[E] = total;
    }
    __syncthreads();
    // replicas: slot (c, s) of expert e sits after e's home and e's replicas on ranks below c
    for (int xs = tid; xs < R * S; xs += kThreads) {
        const int e = slot[xs];
        if (e < 0) continue;
        const int c = small_div(xs, invS), sl = xs - c * S;
        const uint64_t lower = holder[e] & ~(1ull << small_div(e, invH)) & ((1ull << c) - 1ull);
        const int m = pos[e] + 1 + __popcll(lower);
        const int p = c * W + H + sl;
        io[m] = p;
        val[m] = q[p];
    }
    __syncthreads();
    // segmented inclusive scan of the entries: a value is (bit 31: a list
    // starts in it) | running sum, and seg(a, b) = b when b starts a list,
    // else a + b (the sums stay below 2^31).  Thread t takes a run of
    // consecutive entries: its own segmented sum, a warp scan and a scan of
    // the warp totals give the value entering its run.
    auto seg = [](unsigned a, unsigned b) -> unsigned { return (b >> 31) ? b : a + b; };
    const int Mu = pos[E];
    const int per2 = (Mu + kThreads - 1) / kThreads;
    const int m0 = min(Mu, tid * per2), m1 = min(Mu, m0 + per2);
    unsigned own = 0u;
    for (int m = m0; m < m1; ++m) own = seg(own, (unsigned)val[m]);
    unsigned sx = own;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const unsigned y = __shfl_up_sync(kFull, sx, o);
        if (lane >= o) sx = seg(y, sx);
    }
    unsigned ex = __shfl_up_sync(kFull, sx, 1);
    if (lane == 0) ex = 0u;
    if (lane == 31) wtot[warp] = (int)sx;
    __syncthreads();
    unsigned run2 = 0u;
#pragma unroll
    for (int w = 0; w < kWarps; ++w)
        if (w < warp) run2 = seg(run2, (unsigned)wtot[w]);
    run2 = seg(run2, ex);
    for (int m = m0; m < m1; ++m) {
        run2 = seg(run2, (unsigned)val[m]);
        co[m] = (int)(run2 & 0x7fffffffu);
    }
    __syncthreads();  // the scratch may be reused by the next call
}

}  // namespace ultraep
