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
//   + (lanes below in the same 32-slot step)   popc(group & lanemask_lt)
// The group of lanes holding the same id is found through a per-warp mask
// table in shared memory (each lane ORs in its bit; after a warp barrier the
// mask is the group); the group's leader advances the warp's running count.
//
// A slot of rank x goes to the first instance of e's list whose inclusive
// cumulative quota exceeds x, at row  inst_offset[p] + x - (cum before p),
// i.e. x + delta[m] with delta precomputed per list entry.  The per-warp
// scan also records, for every (warp, expert), the row of the warp's first
// rank and how many ranks its instance holds from there; a slot inside that
// range gets its row with one add, the rest (a warp's ranks crossing into the
// next replica) binary search the expert's list, which for a hot expert holds
// dozens of replicas.
//
// ids are read once from memory and kept, with their ranks, between the
// ranking and the row phase of a chunk: in registers in the 256-thread blocks
// of batched launches, in shared memory in the 1024-thread blocks of one-layer
// launches; dst_row is written with coalesced streaming stores; the optional
// src_slot inverse is a scattered store.
//
// Three kernels compute these rows and the launcher picks one by shape (see
// launch_reroute): the quad kernel for batched launches (two warps per source
// rank, one walking its first half forward and one its second half backward,
// two ranks per block, four slots per lane per step); the mask-table
// kernel above in 1024-thread blocks for one-layer launches, a source rank
// split over a thread-block cluster of two or four blocks when they fit; and
// the same kernel in 256-thread blocks for everything else.
//
// (A design with lane-private counters, each lane owning a contiguous run of
// slots, two shared-memory atomics per slot and one warp scan per expert
// pair, was slower in every configuration measured, also with a path free of
// per-slot tests for full aligned runs.)
#include <climits>
#include <type_traits>

#include <cooperative_groups.h>

#include "common.cuh"

namespace ultraep {
namespace {

namespace cg = cooperative_groups;

// 32-slot steps per warp per chunk (ids held in registers), blocks per SM of
// the many-block launches (build-time tunables)
#ifndef EP_REROUTE_ITEMS
#define EP_REROUTE_ITEMS 16
#endif
#ifndef EP_REROUTE_CLUSTER_PARTS
#define EP_REROUTE_CLUSTER_PARTS 1  // one-layer launches split a rank over a cluster (build-time tunable)
#endif
#ifndef EP_REROUTE_BLOCKS_PER_SM
#define EP_REROUTE_BLOCKS_PER_SM 4
#endif
constexpr int kItems = EP_REROUTE_ITEMS;
// Where a chunk's ids (and then their ranks) live: registers, or shared
// memory, which frees kItems registers per thread.  Measured: the one-layer
// launch (1024-thread blocks) 22.5 us with shared memory against 24.6, the
// batched launch (256-thread blocks) 407.5 us with registers against 411.7
// (five blocks per SM) to 421.9 (four).
#ifndef EP_REROUTE_EV_SMEM_NARROW
#define EP_REROUTE_EV_SMEM_NARROW 0  // build-time tunable: also for 256-thread blocks
#endif
template <int kThreads>
constexpr bool ev_in_smem() { return kThreads == 1024 || EP_REROUTE_EV_SMEM_NARROW; }

struct RrLayout {
    int P, M;        // instances, CSR capacity
    int Es, El;      // row strides of the per-warp int32 and uint16 tables
    size_t lim_off;  // byte offset of the uint16 table wlim
    size_t ev_off;   // byte offset of the ids of a chunk (when in shared memory)
    size_t bytes;
};

__host__ __device__ inline RrLayout rr_layout(int R, int E, int S, int warps, bool ev_smem,
                                              int items = kItems) {
    RrLayout l;
    l.P = R * (E / R + S);
    l.M = E + R * S;
    // Wide blocks: row strides one bank past a multiple of 32 words, so that
    // the entries of one expert in the 32 warps' rows (read together by the
    // scan over warps) fall in different banks.  Narrow blocks keep stride E
    // (measured ~1% faster batched).
    if (warps == 32) {
        l.Es = E | 1;
        l.El = (E + 2) & ~1;
        if ((l.El / 2) % 2 == 0) l.El += 2;
    } else {
        l.Es = l.El = E;
    }
    // int32: off[P+1] ptr[E+1] bcum[M] bdel[M] base[E] wx0[warps][Es] wdb[warps][Es]
    //        want[E] ctot[E]
    // uint16: wlim[warps][El]
    l.lim_off = sizeof(int32_t) * ((size_t)(l.P + 1) + (E + 1) + 2 * (size_t)l.M + E +
                                   2 * (size_t)warps * l.Es + 2 * (size_t)E);
    l.bytes = l.lim_off + sizeof(uint16_t) * (size_t)warps * l.El;
    l.ev_off = (l.bytes + 15) & ~(size_t)15;
    if (ev_smem) l.bytes = l.ev_off + sizeof(int32_t) * (size_t)items * warps * 32;
    return l;
}

// first index m in [lo, hi) with a[m] > x (hi when none)
__device__ __forceinline__ int upper_bound(const int32_t* a, int lo, int hi, int x) {
    int n = hi - lo;
    while (n > 0) {
        const int h = n >> 1;
        if (a[lo + h] <= x) {
            lo += h + 1;
            n -= h + 1;
        } else {
            n = h;
        }
    }
    return lo;
}

// The rank's counts in shared memory (nothing here depends on the plan):
//   base[E]   += slots of e on source ranks below r
//   want[E]   = counts_src[r][e] (not loaded when want is null); plan_tables
//             adds base[e] to it
// base must be zero, and a block barrier passed, before the call.  With E a
// multiple of 4 and the rows 16-byte aligned, thread (g, q) sums the int4
// column q (experts 4q .. 4q+3) over rows g, g+G, ... < r (G = threads /
// (E/4)), 2048 / threads loads in flight, at most 8 (every row of 64 ranks at
// E = 128 in one round for 256 threads and more); otherwise thread (g, e)
// sums column e the same way (G = threads / E).  The partial sums meet in
// base[] by atomics.
template <int kThreads>
__device__ __forceinline__ void rank_prefix(int R, int E, int inst, int r,
                                            const int32_t* __restrict__ counts_src,
                                            int32_t* base, int32_t* want) {
    constexpr int kU = 2048 / kThreads > 8 ? 8 : (2048 / kThreads > 1 ? 2048 / kThreads : 1);
    const int tid = threadIdx.x;
    const int32_t* own = counts_src + ((int64_t)inst * R + r) * E;
    if (want != nullptr)
        for (int e = tid; e < E; e += kThreads) want[e] = __ldg(own + e);
    const int32_t* cs = counts_src + (int64_t)inst * R * E;
    const int Q = E >> 2;
    if ((E & 3) == 0 && Q <= kThreads && (reinterpret_cast<uintptr_t>(cs) & 15u) == 0) {
        const int G = kThreads / Q;
        const int q = tid % Q, g = tid / Q;
        if (g < G) {
            int4 t = make_int4(0, 0, 0, 0);
            for (int r0 = g; r0 < r; r0 += kU * G) {
                int4 v[kU];
#pragma unroll
                for (int u = 0; u < kU; ++u) {
                    const int rr = r0 + u * G;
                    v[u] = (rr < r) ? __ldg(reinterpret_cast<const int4*>(cs + (int64_t)rr * E) + q)
                                    : make_int4(0, 0, 0, 0);
                }
#pragma unroll
                for (int u = 0; u < kU; ++u) {
                    t.x += v[u].x;
                    t.y += v[u].y;
                    t.z += v[u].z;
                    t.w += v[u].w;
                }
            }
            if (t.x != 0) atomicAdd(&base[4 * q], t.x);
            if (t.y != 0) atomicAdd(&base[4 * q + 1], t.y);
            if (t.z != 0) atomicAdd(&base[4 * q + 2], t.z);
            if (t.w != 0) atomicAdd(&base[4 * q + 3], t.w);
        }
    } else {
        const int G = (E <= kThreads) ? kThreads / E : 1;
        for (int x = tid; x < G * E; x += kThreads) {
            const int e = x % E, g = x / E;
            int t = 0;
            for (int r0 = g; r0 < r; r0 += kU * G) {
                int v[kU];
#pragma unroll
                for (int u = 0; u < kU; ++u) {
                    const int rr = r0 + u * G;
                    v[u] = (rr < r) ? cs[(int64_t)rr * E + e] : 0;
                }
#pragma unroll
                for (int u = 0; u < kU; ++u) t += v[u];
            }
            if (t != 0) atomicAdd(&base[e], t);
        }
    }
}

// Plan tables in shared memory:
//   off[P+1]  first row of each instance (exclusive prefix of quota over p)
//   ptr[E+1]  CSR row pointers of the instance lists, clamped to [0, M]
//   bcum[M]   inclusive cumulative quota of each list entry (INT_MIN if unused)
//   bdel[M]   row minus within-expert rank, for the ranks of that entry
//   want[E]   += base[e]: the running base after the block's last chunk when
//             counts_src describes these ids (when want is not null)
// rank_prefix must have run, and no block barrier is needed after it; the
// block of source rank 0 also writes inst_offset.  The caller puts a barrier
// between this and any read of the tables.
template <int kThreads>
__device__ __forceinline__ void plan_tables(int E, int P, int M, int inst, int r,
                                            const int32_t* __restrict__ quota,
                                            const int32_t* __restrict__ inst_ptr,
                                            const int32_t* __restrict__ inst_id,
                                            const int32_t* __restrict__ inst_cum,
                                            int32_t* __restrict__ inst_offset, int32_t* off,
                                            int32_t* ptr, int32_t* bcum, int32_t* bdel,
                                            int32_t* base, int32_t* want, int32_t* warp_tot,
                                            bool write_offsets = true) {
    constexpr int kWarps = kThreads / 32;
    constexpr int kIpt = (2048 + kThreads - 1) / kThreads;  // P <= 2048 quota per thread
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int32_t* qg = quota + (int64_t)inst * P;
    const int32_t* pg = inst_ptr + (int64_t)inst * (E + 1);
    const int32_t* ig = inst_id + (int64_t)inst * M;
    const int32_t* cg = inst_cum + (int64_t)inst * M;
    // every load of the plan's outputs is independent of the others, so the
    // prologue waits for memory once: the list entries are loaded whole and
    // the used length applied afterwards
    // the quotas: in registers (kIpt per thread) for wide blocks; narrow
    // blocks, whose kIpt registers would spill, stage them in off[] and scan
    // a contiguous run of them per thread
    constexpr bool kQReg = kIpt <= 4;
    int qv[kQReg ? kIpt : 1];
    if constexpr (kQReg) {
#pragma unroll
        for (int u = 0; u < kIpt; ++u) {
            const int p = tid * kIpt + u;
            qv[u] = (p < P) ? qg[p] : 0;
        }
    } else {
        for (int p = tid; p < P; p += kThreads) off[p] = qg[p];
    }
    const int nM = min(max(pg[E], 0), M);
    const int xn = max(E + 1, M);
    for (int x = tid; x < xn; x += kThreads) {
        const int pe = (x <= E) ? pg[x] : 0;
        const int pm = (x < M) ? ig[x] : -1;
        const int cm = (x < M) ? cg[x] : 0;
        if (x <= E) ptr[x] = min(max(pe, 0), M);
        if (x < M) {
            // cumulative quota, and for now the instance (-1 when unused or
            // out of range)
            const bool used = x < nM && pm >= 0 && pm < P;
            bcum[x] = used ? cm : INT_MIN;
            bdel[x] = used ? pm : -1;
        }
    }
    int qlocal = 0;
    int sb = 0, se = 0;  // (narrow blocks) this thread's run of quotas
    if constexpr (kQReg) {
#pragma unroll
        for (int u = 0; u < kIpt; ++u) qlocal += qv[u];
    } else {
        __syncthreads();
        const int seg = (P + kThreads - 1) / kThreads;
        sb = min(P, tid * seg);
        se = min(P, sb + seg);
        for (int p = sb; p < se; ++p) qlocal += off[p];
    }
    // inst_offset: exclusive prefix of quota over p
    int qx = qlocal;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const int y = __shfl_up_sync(kFull, qx, o);
        if (lane >= o) qx += y;
    }
    if (lane == 31) warp_tot[warp] = qx;
    __syncthreads();
    if (warp == 0) {
        int w = (lane < kWarps) ? warp_tot[lane] : 0;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const int y = __shfl_up_sync(kFull, w, o);
            if (lane >= o) w += y;
        }
        if (lane < kWarps) warp_tot[lane] = w;  // inclusive over warps
    }
    __syncthreads();
    {
        int run = qx - qlocal + (warp > 0 ? warp_tot[warp - 1] : 0);
        if constexpr (kQReg) {
#pragma unroll
            for (int u = 0; u < kIpt; ++u) {
                const int p = tid * kIpt + u;
                if (p < P) off[p] = run;
                run += qv[u];
            }
        } else {
            for (int p = sb; p < se; ++p) {  // (in place: each thread its own run)
                const int v = off[p];
                off[p] = run;
                run += v;
            }
        }
        if (tid == kThreads - 1) off[P] = warp_tot[kWarps - 1];
    }
    __syncthreads();
    // each thread adds the prefix to the want[] entries it loaded itself
    if (want != nullptr)
        for (int e = tid; e < E; e += kThreads) want[e] += base[e];
    // row minus within-expert rank of each entry: off[p] - (cum - quota[p]),
    // with quota[p] = off[p+1] - off[p] (each thread revisits its own entries)
    for (int m = tid; m < M; m += kThreads) {
        const int p = bdel[m];
        bdel[m] = (p >= 0) ? off[p] - (bcum[m] - (off[p + 1] - off[p])) : 0;
    }
    if (r == 0 && write_offsets) {
        int32_t* og = inst_offset + (int64_t)inst * (P + 1);
        for (int p = tid; p <= P; p += kThreads) og[p] = off[p];
    }
}

// One block per (instance, source rank); the rank's slots are processed in
// chunks of kThreads * kItems.  kThreads = 1024 when few blocks run (one
// instance: the whole rank is one chunk) and E <= 512; else 256, four blocks
// per SM (measured faster for batched calls than 512 x 2).
//
// kCl > 1 (one-layer launches): a thread-block cluster of kCl blocks shares
// one source rank, block c taking the c-th part of its slots as one chunk of
// kThreads * kIt.  After ranking its part (before the wait for the plan in
// ep_balance) every block publishes its per-expert totals; block c adds the
// totals of the blocks below it, read through distributed shared memory, to
// its starting ranks.  The rank's rows then take kCl SMs instead of one.
template <int kThreads, int kIt = kItems, int kCl = 1>
__global__ void __launch_bounds__(kThreads, kThreads == 256 ? EP_REROUTE_BLOCKS_PER_SM : 1024 / kThreads)
reroute_kernel(const int32_t* __restrict__ ids, int64_t T, int k, int R, int E, int S,
               const int32_t* __restrict__ counts_src, const int32_t* __restrict__ quota,
               const int32_t* __restrict__ inst_ptr, const int32_t* __restrict__ inst_id,
               const int32_t* __restrict__ inst_cum, int32_t* __restrict__ dst_row,
               int32_t* __restrict__ src_slot, int32_t* __restrict__ inst_offset,
               int32_t* dev_status, int early) {
    constexpr int kWarps = kThreads / 32;
    constexpr int kChunk = kThreads * kIt;
    extern __shared__ __align__(16) int32_t sm[];
    __shared__ int32_t warp_tot[kWarps];
    __shared__ int32_t flags;

    static_assert(kIt % 4 == 0, "phase C takes four steps at a time");
    constexpr bool kEvSmem = ev_in_smem<kThreads>();
    const RrLayout lay = rr_layout(R, E, S, kWarps, kEvSmem, kIt);
    const int P = lay.P, M = lay.M;
    int32_t* off = sm;              // [P+1] first row of each instance
    int32_t* ptr = off + (P + 1);   // [E+1] CSR row pointers (clamped)
    int32_t* bcum = ptr + (E + 1);  // [M]   inclusive cumulative quota
    int32_t* bdel = bcum + M;       // [M]   row - within-expert rank
    int32_t* base = bdel + M;       // [E]   within-expert rank of the chunk's first slot
    const int Es = lay.Es, El = lay.El;
    int32_t* wx0 = base + E;        // [kWarps][Es] per-warp counts, then each warp's first rank
    int32_t* wdb = wx0 + kWarps * Es;  // [kWarps][Es] row of that first rank
    int32_t* want = wdb + kWarps * Es;  // [E] expected base after the last chunk
    int32_t* ctot = want + E;           // [E] this block's per-expert totals (clusters)
    uint16_t* wlim = reinterpret_cast<uint16_t*>(reinterpret_cast<unsigned char*>(sm) + lay.lim_off);
                                    // [kWarps][El] ranks left in its instance (capped)

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int cl = (kCl > 1) ? (int)(blockIdx.x % kCl) : 0;  // rank in the cluster
    const int unit = (kCl > 1) ? (int)(blockIdx.x / kCl) : (int)blockIdx.x;
    const int inst = unit / R, r = unit % R;

    // ---- this block's slots (source rank r, part cl).  Out-of-range ids are
    // flagged at load time; slots past the end load as -1.
    // (32-bit division: T < 2^31 since T*k < 2^31)
    const int Tr = ((int)T + R - 1) / R;
    const int64_t N = T * k;
    const int64_t rs0 = min(T, (int64_t)r * Tr) * k, rs1 = min(T, (int64_t)(r + 1) * Tr) * k;
    const int64_t part = (rs1 - rs0 + kCl - 1) / kCl;
    const int64_t s0 = (kCl > 1) ? min(rs1, rs0 + cl * part) : rs0;
    const int64_t s1 = (kCl > 1) ? min(rs1, rs0 + (cl + 1) * part) : rs1;
    const int32_t* idi = ids + (int64_t)inst * N;
    int my_flags = 0;
    // item it of this thread: a register, or word it * kThreads + tid of the
    // chunk's shared array (consecutive threads, consecutive banks)
    int evr[kEvSmem ? 1 : kIt] = {};
    int* evs = reinterpret_cast<int*>(reinterpret_cast<unsigned char*>(sm) + lay.ev_off) + threadIdx.x;
    auto ev_get = [&](int it) -> int {
        if constexpr (kEvSmem) return evs[it * kThreads];
        else return evr[it];
    };
    auto ev_set = [&](int it, int v) {
        if constexpr (kEvSmem) evs[it * kThreads] = v;
        else evr[it] = v;
    };
    const int lbase = warp * 32 * kIt + lane;  // chunk-local index of item 0
    auto load_chunk = [&](int64_t cs) {
        const int nc = (int)min((int64_t)kChunk, s1 - cs);
        const int32_t* src = idi + cs;
#pragma unroll
        for (int it = 0; it < kIt; ++it) {
            const int li = lbase + it * 32;
            const int v = (li < nc) ? __ldcs(src + li) : -1;
            if (li < nc && (unsigned)v >= (unsigned)E) my_flags |= EP_DEV_BAD_ID;
            ev_set(it, v);
        }
    };
    // ---- shared tables that phase A needs: zero them first
    if (tid == 0) flags = 0;
    for (int x = tid; x < E + 2 * kWarps * Es; x += kThreads) base[x] = 0;  // base, wx0, wdb
    __syncthreads();

    int32_t* wrow = wx0 + warp * Es;
    const unsigned lt = lanemask_lt();
    // phase A: per-warp histogram and ranks inside the warp; ev becomes
    // e | rank << 10 (-1: no valid id).  The lanes holding the same id find
    // each other through the warp's mask row (the wdb row, idle until phase
    // B): each ORs its lane bit into mask[e]; after a warp barrier mask[e] is
    // the group.  Every lane of the group reads the warp's running count of e;
    // after a second barrier the group's lowest lane (leader) advances it and
    // clears mask[e] for the next step.
    auto phase_a = [&]() {
        uint32_t* mrow = reinterpret_cast<uint32_t*>(wdb) + warp * Es;
#pragma unroll
        for (int it = 0; it < kIt; ++it) {
            const int e = ev_get(it);
            const bool valid = (unsigned)e < (unsigned)E;
            if (valid) atomicOr(&mrow[e], 1u << lane);
            __syncwarp();
            // every lane of the group reads the group and the running count
            // itself (no shuffle from the leader), both loads at once
            const unsigned g = valid ? mrow[e] : 0u;
            const int old = valid ? wrow[e] : 0;
            const unsigned below = g & lt;
            __syncwarp();  // every read of mrow[e] and wrow[e] is done
            if (valid && below == 0u) {  // the group's lowest lane
                wrow[e] = old + __popc(g);
                mrow[e] = 0u;
            }
            __syncwarp();  // the clear lands before the next step's ORs
            ev_set(it, valid ? (e | ((old + __popc(below)) << 10)) : -1);
        }
    };
    // early (ep_balance): this grid is a programmatic dependent of ep_plan and
    // the ids were complete before ep_count started, so the first chunk's ids
    // are loaded and ranked before waiting for the plan.  Otherwise the wait
    // comes first (a plain launch returns from it at once).
    if (!early) pdl_wait();
    if (s0 < s1) {
        load_chunk(s0);
        phase_a();
    }
    // the rank's counts (ep_count's output, complete before the plan started)
    rank_prefix<kThreads>(R, E, inst, r, counts_src, base, want);
    int lower = 0;  // thread e: slots of e in the cluster's blocks below this one
    if constexpr (kCl > 1) {
        // the block's per-expert totals (its one chunk's per-warp counts),
        // read by the blocks above it through distributed shared memory
        // (E <= 512 < kThreads: thread e holds expert e)
        __syncthreads();
        for (int e = tid; e < E; e += kThreads) {
            int t = 0;
            for (int w = 0; w < kWarps; ++w) t += wx0[w * Es + e];
            ctot[e] = t;
        }
        cg::cluster_group cluster = cg::this_cluster();
        cluster.sync();
        if (tid < E)
            for (int c2 = 0; c2 < cl; ++c2) lower += cluster.map_shared_rank(ctot, c2)[tid];
        cluster.sync();  // every read of a block's totals is done before any block moves on
    }
    // phase B of the wide blocks, first half: for every (warp w, expert e) of
    // the chunk, the rank of the warp's first slot of e (base[e] + the slots of
    // e in warps below w).  The 32 lanes of a warp hold warps 0 .. 31 of one
    // expert: an exclusive scan across them.  It needs only counts, so the
    // first chunk's runs before the wait for the plan.
    auto scan_b = [&]() {
        constexpr int kEpp = kThreads / kWarps;  // experts per pass
        const int wv = tid % kWarps, ei = tid / kWarps;
        for (int eb = 0; eb < E; eb += kEpp) {  // same trip count in every lane
            const int e = eb + ei;
            const bool act = e < E;
            const int c = act ? wx0[wv * Es + e] : 0;
            const int b0 = act ? base[e] : 0;
            int incl = c;
#pragma unroll
            for (int o = 1; o < kWarps; o <<= 1) {
                const int y = __shfl_up_sync(kFull, incl, o, kWarps);
                if (wv >= o) incl += y;
            }
            const int x0 = b0 + incl - c;
            if (act) wx0[wv * Es + e] = x0;
            __syncwarp();  // every lane of the group has read base[e]
            if (act && wv == kWarps - 1) base[e] = x0 + c;
        }
    };
    // ... second half (the plan): the row of that rank and how many ranks its
    // instance holds from there, one independent search of e's list per lane
    auto search_b = [&]() {
        constexpr int kEpp = kThreads / kWarps;
        const int wv = tid % kWarps, ei = tid / kWarps;
        for (int eb = 0; eb < E; eb += kEpp) {
            const int e = eb + ei;
            if (e < E) {
                const int x0 = wx0[wv * Es + e];
                const int lo = ptr[e], end = ptr[e + 1];
                const int m = upper_bound(bcum, lo, end, x0);
                if (m < end) {
                    wdb[wv * Es + e] = x0 + bdel[m];
                    wlim[wv * El + e] = (uint16_t)min(bcum[m] - x0, 0xffff);
                } else {
                    wdb[wv * Es + e] = -1;
                    wlim[wv * El + e] = 0;
                }
            }
        }
    };
    constexpr bool kSplitB = kWarps == 32;
    if constexpr (kSplitB) {
        // want[] gets the prefix before base moves on; a block of a cluster
        // starts at the slots of the blocks below it
        __syncthreads();  // rank_prefix's adds and every warp's phase A
        if (want != nullptr)
            for (int e = tid; e < E; e += kThreads) want[e] += base[e];
        if constexpr (kCl > 1) {
            if (tid < E) base[tid] += lower;
        }
        __syncthreads();
        if (s0 < s1) scan_b();
    }
    if (early) pdl_wait();
    pdl_trigger();

    // ---- prologue: plan tables (want[] gets the rank's whole count, unless
    // done above); a block of a cluster starts at the slots of the blocks
    // below it
    plan_tables<kThreads>(E, P, M, inst, r, quota, inst_ptr, inst_id, inst_cum, inst_offset, off,
                          ptr, bcum, bdel, base, kSplitB ? nullptr : want, warp_tot, cl == 0);
    if constexpr (kCl > 1 && !kSplitB) {
        if (tid < E) base[tid] += lower;  // (thread e alone touches base[e] here)
    }
    // (the barrier before phase B orders the writes above before any read of
    // bcum / bdel)

    int32_t* dsti = dst_row + (int64_t)inst * N;
    int32_t* srci = src_slot ? src_slot + (int64_t)inst * N : nullptr;
    const int32_t* dbrow = wdb + warp * Es;
    const uint16_t* limrow = wlim + warp * El;
    for (int64_t cs = s0; cs < s1; cs += kChunk) {
        const int nc = (int)min((int64_t)kChunk, s1 - cs);
        if (cs != s0) {
            load_chunk(cs);
            phase_a();
        }
        __syncthreads();
        if constexpr (kWarps == 32) {
            // phase B (above): the scan over warps, then the search of each
            // (warp, expert) entry (measured 20.5 us per one-layer launch
            // against 22.5 for eight lanes per expert walking four warps each).
            // Narrow blocks, whose launches are issue-bound, keep the walk
            // below (four times fewer searches: 379 us against 393 on a
            // 94-layer batch).  The first chunk's scan ran before the plan.
            if (cs != s0) scan_b();
            search_b();  // (each thread reads back the entries it scanned)
        } else {
            // experts per phase-B pass: G consecutive threads share one expert's warps
            int G = 1;
            while (G * 2 <= kWarps && G * 2 * E <= kThreads) G *= 2;

            // phase-B bookkeeping of one (warp, expert): its first rank x0, the row of
            // that rank and how many ranks its instance still holds from there
            auto warp_entry = [&](int w, int e, int x0, int& m, int end) {
                while (m < end && bcum[m] <= x0) ++m;
                wx0[w * Es + e] = x0;
                if (m < end) {
                    wdb[w * Es + e] = x0 + bdel[m];
                    wlim[w * El + e] = (uint16_t)min(bcum[m] - x0, 0xffff);
                } else {
                    wdb[w * Es + e] = -1;
                    wlim[w * El + e] = 0;
                }
            };

            // phase B: per expert, exclusive scan over warps on top of base, and
            // each warp's entry (first rank, its row, ranks left in its instance)
            if (G == 1) {
                for (int e = tid; e < E; e += kThreads) {
                    int run = base[e];
                    const int end = ptr[e + 1];
                    int m = upper_bound(bcum, ptr[e], end, run);
                    for (int w = 0; w < kWarps; ++w) {
                        const int c = wx0[w * Es + e];
                        warp_entry(w, e, run, m, end);
                        run += c;
                    }
                    base[e] = run;
                }
            } else {
                const int e = tid / G, gi = tid % G;
                const bool act = e < E;
                const int per = kWarps / G;
                int loc = 0;
                const int b0 = act ? base[e] : 0;
                if (act)
                    for (int w = gi * per; w < (gi + 1) * per; ++w) loc += wx0[w * Es + e];
                int incl = loc;
                for (int o = 1; o < G; o <<= 1) {
                    const int y = __shfl_up_sync(kFull, incl, o, G);
                    if (gi >= o) incl += y;
                }
                __syncwarp();
                if (act) {
                    int run = b0 + incl - loc;
                    const int end = ptr[e + 1];
                    int m = upper_bound(bcum, ptr[e], end, run);
                    for (int w = gi * per; w < (gi + 1) * per; ++w) {
                        const int c = wx0[w * Es + e];
                        warp_entry(w, e, run, m, end);
                        run += c;
                    }
                    if (gi == G - 1) base[e] = run;
                }
            }
        }
        __syncthreads();
        // phase C: rank -> row.  Fast path: the rank is still inside the
        // instance of the warp's first rank; else binary search the list.
        // Full chunks skip the per-slot bounds test (warp-uniform branch).
        int32_t* dst = dsti + cs;
        auto phase_c = [&](auto full_tag) {
            constexpr bool kFullChunk = decltype(full_tag)::value;
            // four steps at a time: their rows first (no branch), then the rare
            // search for ranks past the instance of the warp's first rank
#pragma unroll
            for (int it0 = 0; it0 < kIt; it0 += 4) {
                int d[4];
                unsigned slow = 0u;
#pragma unroll
                for (int j = 0; j < 4; ++j) {
                    const int it = it0 + j;
                    const int li = lbase + it * 32;
                    const int v = (kFullChunk || li < nc) ? ev_get(it) : -1;
                    const bool has = v >= 0;
                    const int e = has ? (v & 1023) : 0;
                    const int rr = v >> 10;
                    d[j] = dbrow[e] + rr;
                    slow |= (has && rr >= (int)limrow[e]) ? (1u << j) : 0u;
                }
                if (slow) {
#pragma unroll
                    for (int j = 0; j < 4; ++j) {
                        if ((slow >> j) & 1u) {
                            const int v = ev_get(it0 + j);
                            const int e = v & 1023, rr = v >> 10;
                            const int x = wrow[e] + rr;
                            const int end = ptr[e + 1];
                            const int m = upper_bound(bcum, ptr[e], end, x);
                            d[j] = (m < end) ? x + bdel[m < M ? m : M - 1] : -1;
                        }
                    }
                }
#pragma unroll
                for (int j = 0; j < 4; ++j) {
                    const int it = it0 + j;
                    const int li = lbase + it * 32;
                    if (kFullChunk || li < nc) {
                        const bool has = ev_get(it) >= 0;
                        int dd = d[j];
                        if (has && (unsigned)dd >= (unsigned)N) {
                            dd = -1;
                            my_flags |= EP_DEV_QUOTA_OVERFLOW;
                        }
                        dd = has ? dd : -1;
                        __stcs(dst + li, dd);
                        if (srci != nullptr && dd >= 0) srci[dd] = (int32_t)(cs + li);
                    }
                }
            }
        };
        if (nc == kChunk) phase_c(std::true_type{});
        else phase_c(std::false_type{});
        __syncwarp();
        for (int e = lane; e < E; e += 32) {
            wrow[e] = 0;
            wdb[warp * Es + e] = 0;  // mask row of the next chunk's phase A
        }
        __syncwarp();
    }
    // every slot of the rank has been ranked: base[e] - (slots of e on earlier
    // ranks) is this rank's own count of e, which must equal counts_src[r][e]
    // (the within-expert ranks above started from the counts_src prefix); in
    // a cluster the block holding the rank's last part sees the whole count
    __syncthreads();
    if (cl == kCl - 1)
        for (int e = tid; e < E; e += kThreads)
            if (base[e] != want[e]) my_flags |= EP_DEV_COUNTS_MISMATCH;
    if (my_flags) atomicOr(&flags, my_flags);
    __syncthreads();
    if (tid == 0 && flags) raise_flag(dev_status, flags);
}

// ---------------------------------------------------------------- quad kernel
// Batched launches with k a multiple of 4 and 16-byte aligned ids and rows:
// two warps per (instance, source rank), consecutive source ranks of one
// instance per block.  A warp walks slots in steps of 128: lane l holds the
// 16-byte group of slots 4l .. 4l+3 of the step, four of one token's top-k
// ids, which a top-k gate makes distinct.  So a lane adds at most one bit to
// any expert's lane mask, and one OR per slot, one warp barrier and one
// 8-byte read per slot give every slot its place among the step's slots of
// its expert (the lanes below, or above, holding the same expert); one lane
// of the group then moves the expert's entry on.
//
// The two warps of a source rank split its steps and need nothing from each
// other.  The forward warp walks the first half in slot order from the
// prefix of counts_src over the earlier source ranks, the group's lowest lane
// advancing the expert's next rank.  The backward warp walks the second half
// in reverse from the prefix over the ranks up to and including this one: a
// slot's rank is the expert's top rank still free minus one minus the lanes
// above it in its group, and the group's highest lane lowers that top.  Each
// rank thus goes to the slot the stable order gives it.  Where the two walks
// meet, each expert's next forward rank must equal the lowest backward rank:
// that one compare per expert is the check of counts_src.
//
// Each expert has two entries in a warp's tables:
//   hot[e]  = {lane mask of the step, the row of e's next slot; backward, one
//              past it}
//   cold[e] = {the row just past e's current instance (backward: that
//              instance's first row), row - rank there}
// A slot's row is hot[e].row plus (forward) or minus one minus (backward) the
// lanes before it in its group.  Only a group that runs past its instance (a
// replica boundary, or the expert's quotas used up) takes the slow path: its
// slots search the expert's instance list and the group's last lane moves both
// entries on.  The top bit of hot[e].row marks the experts whose ranks on
// this source rank (by counts_src) reach a boundary at all; only their groups
// read cold[e] (rows are below 2^31, so the bit is free).
//
// Ids outside [0, E), and the slots past the end of a rank, use four spare
// entries E .. E+3 (one per position in the lane's group), whose rows are
// discarded.  A step in which some lane's four valid ids are not distinct (no
// top-k gate produces those) is ranked slot by slot instead: four sub-steps
// of 32 consecutive slots on the same tables.
// The SM's shared-memory pipe is the bound, so a block's time grows with the
// blocks sharing its SM, and the launch ends with the most loaded SM: two
// warps per source rank halve the unit of work, so the last wave of blocks
// is a smaller part of the launch.
#ifndef EP_REROUTE_QUAD_WARPS
#define EP_REROUTE_QUAD_WARPS 4  // build-time tunable (even)
#endif
constexpr int kQuadWarps = EP_REROUTE_QUAD_WARPS;
static_assert(kQuadWarps % 2 == 0, "two warps per source rank");
constexpr int kQuadRanks = kQuadWarps / 2;
constexpr int kQuadThreads = kQuadWarps * 32;
constexpr int kQuadAhead = 2;  // steps of ids loaded ahead of the one being ranked
constexpr unsigned kCross = 0x80000000u;  // hot[e].y: e's ranks here may cross a boundary
#ifndef EP_REROUTE_QUAD_MIN_RANKS
#define EP_REROUTE_QUAD_MIN_RANKS 296  // (instance, source rank) units from which the
                                        // quad kernel is used (build-time tunable)
#endif
#ifndef EP_REROUTE_QUAD_BLOCKS_PER_SM
#define EP_REROUTE_QUAD_BLOCKS_PER_SM 8  // build-time tunable
#endif

struct QuadLayout {
    int P, M;
    size_t pre_off;  // [kQuadRanks + 1][E] int32: prefix of counts_src for each rank
    size_t hot_off;  // [kQuadWarps][E + 4] uint2 {mask, next row}
    size_t cold_off; // [kQuadWarps][E + 4] int2 {instance bound row, row - rank}
    size_t bytes;
};

__host__ __device__ inline QuadLayout quad_layout(int R, int E, int S) {
    QuadLayout l;
    l.P = R * (E / R + S);
    l.M = E + R * S;
    // int32: off[P+1] ptr[E+1] bcum[M] bdel[M] base[E]
    l.pre_off = sizeof(int32_t) * ((size_t)(l.P + 1) + (E + 1) + 2 * (size_t)l.M + E);
    l.hot_off = (l.pre_off + sizeof(int32_t) * (size_t)(kQuadRanks + 1) * E + 15) & ~(size_t)15;
    l.cold_off = l.hot_off + sizeof(uint2) * (size_t)kQuadWarps * (E + 4);
    l.bytes = l.cold_off + sizeof(int2) * (size_t)kQuadWarps * (E + 4);
    return l;
}

__device__ __forceinline__ unsigned lanemask_gt() {
    unsigned m;
    asm volatile("mov.u32 %0, %%lanemask_gt;" : "=r"(m));
    return m;
}

__global__ void __launch_bounds__(kQuadThreads, EP_REROUTE_QUAD_BLOCKS_PER_SM)
reroute_quad_kernel(const int32_t* __restrict__ ids, int64_t T, int k, int R, int E, int S,
                    const int32_t* __restrict__ counts_src, const int32_t* __restrict__ quota,
                    const int32_t* __restrict__ inst_ptr, const int32_t* __restrict__ inst_id,
                    const int32_t* __restrict__ inst_cum, int32_t* __restrict__ dst_row,
                    int32_t* __restrict__ src_slot, int32_t* __restrict__ inst_offset,
                    int32_t* dev_status, int early) {
    extern __shared__ __align__(16) int32_t sm[];
    __shared__ int32_t warp_tot[kQuadWarps];
    __shared__ int32_t flags;
    const QuadLayout lay = quad_layout(R, E, S);
    const int P = lay.P, M = lay.M;
    int32_t* off = sm;              // [P+1]
    int32_t* ptr = off + (P + 1);   // [E+1]
    int32_t* bcum = ptr + (E + 1);  // [M]
    int32_t* bdel = bcum + M;       // [M]
    int32_t* base = bdel + M;       // [E] slots of e on source ranks below the block's first
    int32_t* pre = reinterpret_cast<int32_t*>(reinterpret_cast<unsigned char*>(sm) + lay.pre_off);
    uint2* hots = reinterpret_cast<uint2*>(reinterpret_cast<unsigned char*>(sm) + lay.hot_off);
    int2* colds = reinterpret_cast<int2*>(reinterpret_cast<unsigned char*>(sm) + lay.cold_off);

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int gpi = (R + kQuadRanks - 1) / kQuadRanks;  // blocks per instance
    const int inst = blockIdx.x / gpi;
    const int r0 = (blockIdx.x - inst * gpi) * kQuadRanks;
    const int j = warp >> 1;               // the warp's source rank within the block
    const bool back = (warp & 1) != 0;     // the backward walk of that rank
    const int r = r0 + j;
    const bool has_rank = r < R;
    const int nr = min(kQuadRanks, R - r0);  // ranks of this block

    // this warp's slots: source rank r (T*k < 2^31, so 32-bit offsets)
    const int Tr = ((int)T + R - 1) / R;
    const int64_t N = T * k;
    const int s0 = has_rank ? (int)min(T, (int64_t)r * Tr) * k : 0;
    const int s1 = has_rank ? (int)min(T, (int64_t)(r + 1) * Tr) * k : 0;
    const int L = s1 - s0;  // a multiple of 4
    const int nsteps = (L + 127) >> 7;
    const int half = (nsteps + 1) >> 1;  // steps [0, half) forward, [half, nsteps) backward
    const int nmine = back ? nsteps - half : half;
    const int32_t* idw = ids + (int64_t)inst * N + s0;
    int32_t* dsw = dst_row + (int64_t)inst * N + s0;
    int32_t* srci = src_slot ? src_slot + (int64_t)inst * N : nullptr;
    // the warp's i-th step, and its ids
    auto step_of = [&](int i) { return back ? nsteps - 1 - i : i; };
    auto load_step = [&](int i) -> int4 {
        const int sl = (step_of(i) << 7) + (lane << 2);
        return (i < nmine && sl < L) ? __ldcs(reinterpret_cast<const int4*>(idw + sl))
                                     : make_int4(-1, -1, -1, -1);
    };
    // the first steps' ids depend only on the call's input: in ep_balance they
    // are in flight while the planner finishes
    if (!early) pdl_wait();
    int4 buf[kQuadAhead];
#pragma unroll
    for (int a = 0; a < kQuadAhead; ++a) buf[a] = load_step(a);
    if (tid == 0) flags = 0;
    for (int e = tid; e < E; e += kQuadThreads) base[e] = 0;
    __syncthreads();
    // the counts (ep_count's output, complete before the plan started): the
    // slots of every expert on the ranks below the block's, and the block's
    // ranks' own rows
    rank_prefix<kQuadThreads>(R, E, inst, r0, counts_src, base, nullptr);
    {
        const int32_t* cs = counts_src + ((int64_t)inst * R + r0) * E;
        for (int x = tid; x < kQuadRanks * E; x += kQuadThreads) {
            const int w = x / E, e = x - w * E;
            pre[(w + 1) * E + e] = (w < nr) ? __ldg(cs + (int64_t)w * E + e) : 0;
        }
    }
    if (early) pdl_wait();
    pdl_trigger();

    // ---- prologue: plan tables, then each rank's prefix over source ranks
    plan_tables<kQuadThreads>(E, P, M, inst, r0, quota, inst_ptr, inst_id, inst_cum, inst_offset,
                              off, ptr, bcum, bdel, base, nullptr, warp_tot);
    __syncthreads();
    for (int e = tid; e < E; e += kQuadThreads) {
        int run = base[e];
        pre[e] = run;
#pragma unroll
        for (int w = 1; w <= kQuadRanks; ++w) {
            run += pre[w * E + e];
            pre[w * E + e] = run;
        }
    }
    __syncthreads();
    uint2* hot = hots + (size_t)warp * (E + 4);
    int2* cold = colds + (size_t)warp * (E + 4);
    int my_flags = 0;
    // backward: the entries for "the next rank to give is x - 1": the row one
    // past it and its instance's first row; with no such instance (x - 1 past
    // the quotas, or x <= 0) every later slot of e searches.  Returns the
    // instance's first rank (INT_MAX when none).
    auto back_entry = [&](int e, int x, unsigned& y, int2& c) -> int {
        const int b = ptr[e], end = ptr[e + 1];
        if (x > 0) {
            const int m = upper_bound(bcum, b, end, x - 1);
            if (m < end) {
                const int lo = (m > b) ? max(bcum[m - 1], 0) : 0;
                const int nd = bdel[m];
                y = (unsigned)(x + nd);
                c = make_int2(lo + nd, nd);
                return lo;
            }
        }
        y = (unsigned)x;
        c = make_int2(INT_MAX, 0);
        return INT_MAX;
    };
    if (has_rank) {
        // ---- the warp's tables: each expert's first row (its prefix mapped
        // through the plan) and the bound of that row's instance
        const int32_t* lo_pre = pre + j * E;
        const int32_t* hi_pre = pre + (j + 1) * E;
        for (int e = lane; e < E + 4; e += 32) {
            if (e < E) {
                const int lo = lo_pre[e], hi = hi_pre[e];
                if (!back) {
                    const int end = ptr[e + 1];
                    const int m = upper_bound(bcum, ptr[e], end, lo);
                    const int del = (m < end) ? bdel[m] : 0;  // quotas used up: every rank overflows
                    // the rank's ranks of e, by counts_src, all inside this
                    // instance: no group of e ever looks at cold[e]
                    const bool may_cross = m >= end || hi > bcum[m];
                    hot[e] = make_uint2(0u, (unsigned)(lo + del) | (may_cross ? kCross : 0u));
                    cold[e] = make_int2((m < end) ? bcum[m] + del : lo, del);
                } else {
                    unsigned y;
                    int2 c;
                    const int first = back_entry(e, hi, y, c);
                    hot[e] = make_uint2(0u, y | (first > lo ? kCross : 0u));
                    cold[e] = c;
                }
            } else {
                hot[e] = make_uint2(0u, 0u);
                cold[e] = make_int2(back ? INT_MIN : INT_MAX, 0);  // spare entries never cross
            }
        }
        __syncwarp();
        const unsigned bit = 1u << lane;
        uint32_t* hotw = reinterpret_cast<uint32_t*>(hot);
        // rank x of expert e past its entry: search e's instance list
        auto search = [&](int e, int x) -> int {
            if (x < 0) return -1;  // (backward, counts_src short of the ids)
            const int end = ptr[e + 1];
            const int m = upper_bound(bcum, ptr[e], end, x);
            if (m < end) return x + bdel[m];
            my_flags |= EP_DEV_QUOTA_OVERFLOW;
            return -1;
        };

        auto walk = [&](auto dir) {
            constexpr bool kB = decltype(dir)::value;
            // the lanes whose slots of a group come before this lane's
            const unsigned before = kB ? lanemask_gt() : lanemask_lt();
            // a group that ran past its instance: its last lane moves e's
            // entries to the instance of the next rank (rank = row - del)
            auto advance = [&](int e, int next_row, int del) {
                const int x = next_row - del;
                if constexpr (!kB) {
                    const int end = ptr[e + 1];
                    const int m = upper_bound(bcum, ptr[e], end, x);
                    const int nd = (m < end) ? bdel[m] : 0;
                    hot[e].y = (unsigned)(x + nd) | kCross;
                    cold[e] = make_int2((m < end) ? bcum[m] + nd : x, nd);
                } else {
                    unsigned y;
                    int2 c;
                    back_entry(e, x, y, c);
                    hot[e].y = y | kCross;
                    cold[e] = c;
                }
            };
            // row of the slot with `nb` lanes before it in a group whose
            // entry row is y, and the entry's next row after a group of n
            auto row_at = [](int y, int nb) { return kB ? y - 1 - nb : y + nb; };
            auto moved = [](int y, int n) { return kB ? y - n : y + n; };
            auto past = [](int row, int bound) { return kB ? row < bound : row >= bound; };
            auto done = [](int next, int bound) { return kB ? next <= bound : next >= bound; };
            // a step whose lanes hold a repeated id: four sub-steps of 32
            // consecutive slots, one slot per lane, in walk order
            auto step_by_slot = [&](int4 q, int st) {
#pragma unroll 1
                for (int aa = 0; aa < 4; ++aa) {
                    const int a = kB ? 3 - aa : aa;
                    const int srcl = (a << 3) + (lane >> 2), c = lane & 3;
                    const int qx = __shfl_sync(kFull, q.x, srcl), qy = __shfl_sync(kFull, q.y, srcl);
                    const int qz = __shfl_sync(kFull, q.z, srcl), qw = __shfl_sync(kFull, q.w, srcl);
                    const int id = c == 0 ? qx : c == 1 ? qy : c == 2 ? qz : qw;
                    const int sl = (st << 7) + (a << 5) + lane;
                    const bool v = (unsigned)id < (unsigned)E;
                    const int e = v ? id : E;
                    atomicOr(&hotw[2 * e], bit);
                    __syncwarp();
                    const uint2 h = hot[e];
                    const int2 cd = cold[e];
                    const unsigned bef = h.x & before;
                    const int y = (int)(h.y & ~kCross);
                    int row = row_at(y, __popc(bef));
                    const int nx = moved(y, __popc(h.x));
                    const bool last = bef == 0u;
                    __syncwarp();
                    if (last) hot[e] = make_uint2(0u, (unsigned)nx | (h.y & kCross));
                    if (v && past(row, cd.x)) row = search(e, row - cd.y);
                    __syncwarp();
                    if (last && v && done(nx, cd.x)) advance(e, nx, cd.y);
                    __syncwarp();
                    row = v ? row : -1;
                    if ((unsigned)row >= (unsigned)N && v && row >= 0) my_flags |= EP_DEV_QUOTA_OVERFLOW;
                    row = ((unsigned)row < (unsigned)N) ? row : -1;
                    if (sl < L) {
                        dsw[sl] = row;
                        if (srci != nullptr && row >= 0) srci[row] = s0 + sl;
                    }
                }
            };

            int ovf = 0, bad = 0;
#pragma unroll 1
            for (int i = 0; i < nmine; ++i) {
                const int st = kB ? nsteps - 1 - i : i;
                const int4 q = buf[0];
#pragma unroll
                for (int a = 0; a + 1 < kQuadAhead; ++a) buf[a] = buf[a + 1];
                buf[kQuadAhead - 1] = load_step(i + kQuadAhead);
                const int sl = (st << 7) + (lane << 2);
                // invalid ids and slots past the end: the spare entries E + a
                const bool v0 = (unsigned)q.x < (unsigned)E, v1 = (unsigned)q.y < (unsigned)E;
                const bool v2 = (unsigned)q.z < (unsigned)E, v3 = (unsigned)q.w < (unsigned)E;
                const int e0 = v0 ? q.x : E, e1 = v1 ? q.y : E + 1;
                const int e2 = v2 ? q.z : E + 2, e3 = v3 ? q.w : E + 3;
                bad |= (sl < L) && !(v0 && v1 && v2 && v3);
                const bool dup = (e0 == e1) || (e0 == e2) || (e0 == e3) || (e1 == e2) ||
                                 (e1 == e3) || (e2 == e3);
                if (__any_sync(kFull, dup)) {
                    step_by_slot(q, st);
                    continue;
                }
                atomicOr(&hotw[2 * e0], bit);
                atomicOr(&hotw[2 * e1], bit);
                atomicOr(&hotw[2 * e2], bit);
                atomicOr(&hotw[2 * e3], bit);
                __syncwarp();
                const uint2 h0 = hot[e0], h1 = hot[e1], h2 = hot[e2], h3 = hot[e3];
                const unsigned b0 = h0.x & before, b1 = h1.x & before;
                const unsigned b2 = h2.x & before, b3 = h3.x & before;
                const int y0 = (int)(h0.y & ~kCross), y1 = (int)(h1.y & ~kCross);
                const int y2 = (int)(h2.y & ~kCross), y3 = (int)(h3.y & ~kCross);
                int4 rows = make_int4(row_at(y0, __popc(b0)), row_at(y1, __popc(b1)),
                                      row_at(y2, __popc(b2)), row_at(y3, __popc(b3)));
                const int n0 = moved(y0, __popc(h0.x)), n1 = moved(y1, __popc(h1.x));
                const int n2 = moved(y2, __popc(h2.x)), n3 = moved(y3, __popc(h3.x));
                __syncwarp();
                if (b0 == 0u) hot[e0] = make_uint2(0u, (unsigned)n0 | (h0.y & kCross));
                if (b1 == 0u) hot[e1] = make_uint2(0u, (unsigned)n1 | (h1.y & kCross));
                if (b2 == 0u) hot[e2] = make_uint2(0u, (unsigned)n2 | (h2.y & kCross));
                if (b3 == 0u) hot[e3] = make_uint2(0u, (unsigned)n3 | (h3.y & kCross));
                // a group reaching the bound of its instance: its last lane
                // sees it (only experts whose ranks here may cross are checked)
                const bool x0 = b0 == 0u && (h0.y & kCross) && done(n0, cold[e0].x);
                const bool x1 = b1 == 0u && (h1.y & kCross) && done(n1, cold[e1].x);
                const bool x2 = b2 == 0u && (h2.y & kCross) && done(n2, cold[e2].x);
                const bool x3 = b3 == 0u && (h3.y & kCross) && done(n3, cold[e3].x);
                if (__any_sync(kFull, x0 || x1 || x2 || x3)) {
                    // every slot past its entry's bound searches; then the
                    // groups' last lanes move their entries on
                    const int2 c0 = cold[e0], c1 = cold[e1], c2 = cold[e2], c3 = cold[e3];
                    if (v0 && past(rows.x, c0.x)) rows.x = search(e0, rows.x - c0.y);
                    if (v1 && past(rows.y, c1.x)) rows.y = search(e1, rows.y - c1.y);
                    if (v2 && past(rows.z, c2.x)) rows.z = search(e2, rows.z - c2.y);
                    if (v3 && past(rows.w, c3.x)) rows.w = search(e3, rows.w - c3.y);
                    __syncwarp();
                    if (x0 && v0) advance(e0, n0, c0.y);
                    if (x1 && v1) advance(e1, n1, c1.y);
                    if (x2 && v2) advance(e2, n2, c2.y);
                    if (x3 && v3) advance(e3, n3, c3.y);
                }
                __syncwarp();
                rows.x = v0 ? rows.x : -1;
                rows.y = v1 ? rows.y : -1;
                rows.z = v2 ? rows.z : -1;
                rows.w = v3 ? rows.w : -1;
                ovf |= (rows.x >= (int)N) | (rows.y >= (int)N) | (rows.z >= (int)N) |
                       (rows.w >= (int)N);
                rows.x = ((unsigned)rows.x < (unsigned)N) ? rows.x : -1;
                rows.y = ((unsigned)rows.y < (unsigned)N) ? rows.y : -1;
                rows.z = ((unsigned)rows.z < (unsigned)N) ? rows.z : -1;
                rows.w = ((unsigned)rows.w < (unsigned)N) ? rows.w : -1;
                if (sl < L) {
                    __stcs(reinterpret_cast<int4*>(dsw + sl), rows);
                    if (srci != nullptr) {
                        const int g = s0 + sl;
                        if (rows.x >= 0) srci[rows.x] = g;
                        if (rows.y >= 0) srci[rows.y] = g + 1;
                        if (rows.z >= 0) srci[rows.z] = g + 2;
                        if (rows.w >= 0) srci[rows.w] = g + 3;
                    }
                }
            }
            if (ovf) my_flags |= EP_DEV_QUOTA_OVERFLOW;
            if (bad) my_flags |= EP_DEV_BAD_ID;
        };
        if (back)
            walk(std::true_type{});
        else
            walk(std::false_type{});
    }
    __syncthreads();
    // every slot of the rank is ranked: the forward walk's next rank of each
    // expert (row - del) must be the backward walk's lowest
    if (has_rank && !back) {
        const uint2* hb = hot + (E + 4);
        const int2* cb = cold + (E + 4);
        for (int e = lane; e < E; e += 32)
            if ((int)(hot[e].y & ~kCross) - cold[e].y != (int)(hb[e].y & ~kCross) - cb[e].y)
                my_flags |= EP_DEV_COUNTS_MISMATCH;
    }
    if (my_flags) atomicOr(&flags, my_flags);
    __syncthreads();
    if (tid == 0 && flags) raise_flag(dev_status, flags);
}

cudaError_t launch_reroute_quad(const ep_domain_t& d, const int32_t* ids, int64_t T,
                                int32_t n_inst, const int32_t* counts_src, const int32_t* quota,
                                const int32_t* inst_ptr, const int32_t* inst_id,
                                const int32_t* inst_cum, int32_t* dst_row, int32_t* src_slot,
                                int32_t* inst_offset, int32_t* dev_status, cudaStream_t s,
                                bool pdl) {
    const QuadLayout lay = quad_layout(d.R, d.E, d.S);
    if (lay.bytes > 48 * 1024) {
        cudaError_t err = cudaFuncSetAttribute(reroute_quad_kernel,
                                               cudaFuncAttributeMaxDynamicSharedMemorySize,
                                               (int)lay.bytes);
        if (err != cudaSuccess) return err;
    }
    const int gpi = (d.R + kQuadRanks - 1) / kQuadRanks;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)((int64_t)n_inst * gpi));
    cfg.blockDim = dim3(kQuadThreads);
    cfg.dynamicSmemBytes = lay.bytes;
    cfg.stream = s;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = pdl ? 1 : 0;
    return cudaLaunchKernelEx(&cfg, reroute_quad_kernel, ids, T, (int)d.k, (int)d.R, (int)d.E,
                              (int)d.S, counts_src, quota, inst_ptr, inst_id, inst_cum, dst_row,
                              src_slot, inst_offset, dev_status, pdl ? 1 : 0);
}

template <int kThreads, int kIt = kItems, int kCl = 1>
cudaError_t launch_reroute_t(const ep_domain_t& d, const int32_t* ids, int64_t T, int32_t n_inst,
                             const int32_t* counts_src, const int32_t* quota,
                             const int32_t* inst_ptr, const int32_t* inst_id,
                             const int32_t* inst_cum, int32_t* dst_row, int32_t* src_slot,
                             int32_t* inst_offset, int32_t* dev_status, cudaStream_t s,
                             bool pdl) {
    const RrLayout lay = rr_layout(d.R, d.E, d.S, kThreads / 32, ev_in_smem<kThreads>(), kIt);
    if (lay.bytes > 48 * 1024) {
        cudaError_t err = cudaFuncSetAttribute(reroute_kernel<kThreads, kIt, kCl>,
                                               cudaFuncAttributeMaxDynamicSharedMemorySize,
                                               (int)lay.bytes);
        if (err != cudaSuccess) return err;
    }
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)((int64_t)n_inst * d.R * kCl));
    cfg.blockDim = dim3(kThreads);
    cfg.dynamicSmemBytes = lay.bytes;
    cfg.stream = s;
    cudaLaunchAttribute attr[2];
    int na = 0;
    if (pdl) {
        attr[na].id = cudaLaunchAttributeProgrammaticStreamSerialization;
        attr[na].val.programmaticStreamSerializationAllowed = 1;
        ++na;
    }
    if (kCl > 1) {
        attr[na].id = cudaLaunchAttributeClusterDimension;
        attr[na].val.clusterDim.x = kCl;
        attr[na].val.clusterDim.y = 1;
        attr[na].val.clusterDim.z = 1;
        ++na;
    }
    cfg.attrs = attr;
    cfg.numAttrs = na;
    return cudaLaunchKernelEx(&cfg, reroute_kernel<kThreads, kIt, kCl>, ids, T, (int)d.k,
                              (int)d.R, (int)d.E, (int)d.S, counts_src, quota, inst_ptr, inst_id,
                              inst_cum, dst_row, src_slot, inst_offset, dev_status, pdl ? 1 : 0);
}

}  // namespace

cudaError_t launch_reroute(const ep_domain_t& d, const int32_t* ids, int64_t T, int32_t n_inst,
                           const int32_t* counts_src, const int32_t* quota,
                           const int32_t* inst_ptr, const int32_t* inst_id,
                           const int32_t* inst_cum, int32_t* dst_row, int32_t* src_slot,
                           int32_t* inst_offset, int32_t* dev_status, cudaStream_t s,
                           bool pdl) {
    if (n_inst == 0) return cudaSuccess;
    const int64_t blocks = (int64_t)n_inst * d.R;
    const DeviceInfo di = device_info();
    const int sms = di.sms;
    // k a multiple of 4 and 16-byte aligned ids: the quad kernel for batched
    // launches, when its tables fit in shared memory
    const bool quad_ok = d.k % 4 == 0 && (reinterpret_cast<uintptr_t>(ids) & 15u) == 0 &&
                         (reinterpret_cast<uintptr_t>(dst_row) & 15u) == 0 &&
                         quad_layout(d.R, d.E, d.S).bytes + 1024 <= di.smem_optin;
    if (quad_ok && blocks >= (int64_t)EP_REROUTE_QUAD_MIN_RANKS)
        return launch_reroute_quad(d, ids, T, n_inst, counts_src, quota, inst_ptr, inst_id,
                                   inst_cum, dst_row, src_slot, inst_offset, dev_status, s, pdl);
    // wide blocks only when their tables (and the chunk's ids) fit in shared memory
    const bool wide_fits =
        rr_layout(d.R, d.E, d.S, 1024 / 32, ev_in_smem<1024>()).bytes + 1024 <= di.smem_optin;
    if (blocks >= 2 * (int64_t)sms || d.E > 512 || !wide_fits)
        return launch_reroute_t<256>(d, ids, T, n_inst, counts_src, quota, inst_ptr, inst_id,
                                      inst_cum, dst_row, src_slot, inst_offset, dev_status, s, pdl);
    // one-layer launches: a cluster of 2 or 4 blocks per source rank, each
    // block one chunk of 8192 slots, when the rank has at most 32768 slots
    const int64_t rank_slots = tokens_per_rank(T, d.R) * d.k;
    constexpr int kPart = 1024 * 8;
    const bool parts_fit =
        rr_layout(d.R, d.E, d.S, 1024 / 32, ev_in_smem<1024>(), 8).bytes + 1024 <= di.smem_optin;
    // (1024-thread blocks hold an SM each: a cluster launch is used only when
    // all its blocks fit on the GPU at once)
    if (parts_fit && EP_REROUTE_CLUSTER_PARTS) {
        if (rank_slots > 2 * kPart && rank_slots <= 4 * kPart && blocks * 4 <= sms)
            return launch_reroute_t<1024, 8, 4>(d, ids, T, n_inst, counts_src, quota, inst_ptr,
                                                inst_id, inst_cum, dst_row, src_slot,
                                                inst_offset, dev_status, s, pdl);
        if (rank_slots > kPart && rank_slots <= 2 * kPart && blocks * 2 <= sms)
            return launch_reroute_t<1024, 8, 2>(d, ids, T, n_inst, counts_src, quota, inst_ptr,
                                                inst_id, inst_cum, dst_row, src_slot,
                                                inst_offset, dev_status, s, pdl);
        if (rank_slots > 2 * kPart && rank_slots <= 4 * kPart && blocks * 2 <= sms &&
            rr_layout(d.R, d.E, d.S, 1024 / 32, ev_in_smem<1024>(), 16).bytes + 1024 <= di.smem_optin)
            return launch_reroute_t<1024, 16, 2>(d, ids, T, n_inst, counts_src, quota, inst_ptr,
                                                 inst_id, inst_cum, dst_row, src_slot,
                                                 inst_offset, dev_status, s, pdl);
    }
    return launch_reroute_t<1024>(d, ids, T, n_inst, counts_src, quota, inst_ptr, inst_id,
                                   inst_cum, dst_row, src_slot, inst_offset, dev_status, s,
                                   pdl);
}

}  // namespace ultraep
