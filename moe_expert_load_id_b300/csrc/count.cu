// ep_count: exact per-expert load of the gate's top-k ids.
//
// UltraEP article (m.youleyou.com), "key design" section, forward-pass
// paragraph: the global load is obtained after gating and before planning.
//
// One block per (instance, source rank, chunk).  The block's histogram is a
// lane-column table hist[e][C] in shared memory: lane l adds its id e into
// column l % C, so at most 32/C updates of one warp instruction hit the same
// address, whatever the id distribution.  A hot expert therefore costs nothing extra; match.any-based
// aggregation, whose cost grows with the number of distinct ids in the warp,
// is not used.  ids are read with 16-byte streaming loads (scalar head and
// tail).
//
// The chunks of one source rank form a thread-block cluster: every block adds
// its totals into the first block's accumulator through distributed shared
// memory (atomics that need no reply), and after one cluster barrier the
// first block writes counts_src[r].  Source ranks of one
// instance meet in a last-block reduction (atomic ticket) that writes counts;
// its ticket lives in the caller's workspace and is reset by that block, so
// it is zero again after every call.
#include <mutex>

#include <cooperative_groups.h>

#include "common.cuh"

namespace ultraep {
namespace {

namespace cg = cooperative_groups;

// block size and 16-byte loads in flight per thread (build-time tunables).
// Four loads measured faster than two or three on all three 58 to 94-layer
// batches (0.77 / 0.88 / 0.88 of the HBM copy rate against 0.70 / 0.83 /
// 0.82 with two), though the 32 registers of eight blocks per SM spill a
// few bytes; budgeting registers for six or seven blocks per SM was slower.
#ifndef EP_COUNT_THREADS
#define EP_COUNT_THREADS 256
#endif
#ifndef EP_COUNT_VEC
#define EP_COUNT_VEC 4
#endif
constexpr int kCountThreads = EP_COUNT_THREADS;
constexpr int kVec = EP_COUNT_VEC;
// A launch whose blocks all fit on the GPU at once (one layer) is bound by
// load latency, not bandwidth: its blocks take four 16-byte loads per thread
// in flight (one round trip for a 16384-slot source rank in five chunks), at
// four blocks per SM.
constexpr int kVecWave = 4;
constexpr int kWaveBlocksPerSm = 4;
// Many-block launches: the blocks per SM the registers are budgeted for
#ifndef EP_COUNT_BATCH_MIN_BLOCKS
#define EP_COUNT_BATCH_MIN_BLOCKS (2048 / EP_COUNT_THREADS)  // build-time tunable
#endif
constexpr int kBatchMinBlocks = EP_COUNT_BATCH_MIN_BLOCKS;
#ifndef EP_COUNT_TARGET_BLOCKS
#define EP_COUNT_TARGET_BLOCKS (2 * 148)        // blocks a launch aims at (build-time tunable)
#endif
constexpr int kTargetBlocks = EP_COUNT_TARGET_BLOCKS;
constexpr int kMinChunk = kCountThreads * 4;    // at least one 16-byte load per thread
constexpr int kMaxChunksPerRank = 8;            // portable cluster size
#ifndef EP_COUNT_MIN_CHUNKS
#define EP_COUNT_MIN_CHUNKS 1                   // chunks per rank at least (build-time tunable)
#endif

// columns of the lane-column histogram: 16 (lanes l and l+16 share a column,
// at most a 2-way same-address collision) while E*16 ints fit 32 KB.  (32
// columns, whose table leaves room for three blocks per SM, measured slower.)
#ifndef EP_COUNT_COLS
#define EP_COUNT_COLS 16                        // lane columns at most (build-time tunable)
#endif
__host__ __device__ inline int count_cols(int E) {
    int C = EP_COUNT_COLS;
    while (C > 1 && E * C > 8192) C >>= 1;
    return C;
}

// the histogram table, reused by the last block's reduction as [G][E] partial
// sums (G * E = 4 * threads with int4 columns)
__host__ __device__ inline int count_hist_words(int E) {
    const int C = count_cols(E);
    return E * C > 4 * kCountThreads ? E * C : 4 * kCountThreads;
}

__host__ __device__ inline size_t count_smem_bytes(int E) {
    return sizeof(int32_t) * ((size_t)count_hist_words(E) + E);
}

// 16-byte id load: streaming (evict-first), or (EP_COUNT_LOAD_HINT = 1)
// through the non-coherent path with no L1 allocation and a 256-byte L2
// prefetch hint (a build-time tunable)
#ifndef EP_COUNT_LOAD_HINT
#define EP_COUNT_LOAD_HINT 0
#endif
__device__ __forceinline__ int4 load_ids(const int4* p) {
#if EP_COUNT_LOAD_HINT
    int4 v;
    asm volatile("ld.global.nc.L1::no_allocate.L2::256B.v4.s32 {%0, %1, %2, %3}, [%4];"
                 : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
                 : "l"(p));
    return v;
#else
    return __ldcs(p);
#endif
}

__device__ __forceinline__ void count_one(int v, int E, int32_t* hist, int C, int col, int& bad) {
    if ((unsigned)v < (unsigned)E) atomicAdd(&hist[v * C + col], 1);
    else bad = 1;
}

template <int kV, int kMinBlocks>
__global__ void __launch_bounds__(kCountThreads, kMinBlocks)
count_kernel(const int32_t* __restrict__ ids, int64_t T, int k, int R, int E, int cps,
             int32_t* __restrict__ counts, int32_t* __restrict__ counts_src,
             int32_t* dev_status, uint32_t* inst_ticket, int rows_only) {
    extern __shared__ __align__(16) int32_t sh[];
    __shared__ int bad;
    __shared__ int is_last;
    const int C = count_cols(E);
    int32_t* hist = sh;                          // [E][C], later scratch
    int32_t* blk = sh + count_hist_words(E);     // [E] rank total

    // A dependent planner (ep_balance) may launch now; it waits for this grid.
    pdl_trigger();
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    // block -> (instance, source rank, chunk); 32-bit divisions only (a 64-bit
    // division by a run-time value is a long software routine)
    const int b = (int)blockIdx.x;
    const int per_inst = R * cps;
    const int inst = b / per_inst;
    const int rc = b - inst * per_inst;
    const int r = rc / cps, c = rc - r * cps;  // c is also the block's rank in its cluster

    for (int x = tid; x < E * C; x += kCountThreads) hist[x] = 0;
    for (int x = tid; x < E; x += kCountThreads) blk[x] = 0;
    if (tid == 0) bad = 0;
    __syncthreads();
    // the first block's accumulator is zero before any block of the cluster
    // adds to it: arrive now, wait just before the adds
    cg::cluster_group cluster = cg::this_cluster();
    if (cps > 1) cluster.barrier_arrive();

    // this block's slots: chunk c of source rank r (T < 2^31 since T*k < 2^31)
    const int Ti = (int)T;
    const int Tr = (Ti + R - 1) / R;
    const int64_t t0 = min((int64_t)Ti, (int64_t)r * Tr), t1 = min((int64_t)Ti, (int64_t)(r + 1) * Tr);
    const int len = (int)((t1 - t0) * k);
    const int q = len / cps, rem = len - q * cps;
    const int64_t s0 = t0 * k + (int64_t)q * c + min(c, rem);
    const int64_t s1 = s0 + q + (c < rem ? 1 : 0);
    const int32_t* p0 = ids + (int64_t)inst * T * k + s0;
    const int64_t n = s1 - s0;
    // split into a scalar head up to the first 16-byte boundary, an int4 body
    // and a scalar tail
    const int64_t head = min(n, (int64_t)(((16u - ((uintptr_t)p0 & 15u)) & 15u) >> 2));
    const int64_t n4 = (n - head) >> 2;
    const int64_t tail0 = head + 4 * n4;
    const int4* body = reinterpret_cast<const int4*>(p0 + head);
    const int col = lane & (C - 1);
    int local_bad = 0;
    if (tid < head) count_one(__ldcs(p0 + tid), E, hist, C, col, local_bad);
    if (tid < n - tail0) count_one(__ldcs(p0 + tail0 + tid), E, hist, C, col, local_bad);
    // trip count is warp-uniform (v0 has no lane term)
    for (int64_t v0 = (int64_t)warp * 32 * kV; v0 < n4; v0 += (int64_t)kCountThreads * kV) {
        int4 w[kV];
#pragma unroll
        for (int u = 0; u < kV; ++u) {
            const int64_t vi = v0 + u * 32 + lane;
            w[u] = (vi < n4) ? load_ids(body + vi) : make_int4(0, 0, 0, 0);
        }
#pragma unroll
        for (int u = 0; u < kV; ++u) {
            if (v0 + u * 32 + lane < n4) {
                count_one(w[u].x, E, hist, C, col, local_bad);
                count_one(w[u].y, E, hist, C, col, local_bad);
                count_one(w[u].z, E, hist, C, col, local_bad);
                count_one(w[u].w, E, hist, C, col, local_bad);
            }
        }
    }
    if (local_bad) bad = 1;
    __syncthreads();

    // block total of expert e: thread e sums its C columns, starting at
    // column e % C (the rotation keeps one warp's reads 2-way per bank at
    // most), and adds it to the rank's total: the first block's accumulator,
    // through distributed shared memory in a cluster
    if (cps > 1) cluster.barrier_wait();
    int32_t* acc = (cps > 1 && c != 0) ? cluster.map_shared_rank(blk, 0) : blk;
    for (int e = tid; e < E; e += kCountThreads) {
        const int32_t* row = hist + e * C;
        int t = 0;
        for (int j = 0; j < C; ++j) t += row[(j + e) & (C - 1)];
        if (cps > 1) {
            if (t != 0) atomicAdd(acc + e, t);
        } else {
            blk[e] = t;
        }
    }
    if (tid == 0 && bad) raise_flag(dev_status, EP_DEV_BAD_ID);

    // one barrier: every block's adds are done (the cluster barrier orders
    // them before the first block's reads), then the first block writes the
    // rank's row
    const int64_t rank_row = ((int64_t)inst * R + r) * E;
    if (cps > 1) {
        cluster.sync();
        if (c != 0) return;
    } else {
        __syncthreads();
    }
    for (int e = tid; e < E; e += kCountThreads) counts_src[rank_row + e] = blk[e];

    // rows_only (ep_balance): the planner, which waits for this grid, sums the
    // rows itself, so the blocks stop here
    if (rows_only) return;
    // the last source rank of the instance folds counts_src into counts.  The
    // barrier orders the block's counts_src writes before thread 0's fence and
    // ticket (fences are cumulative), so one thread fences for the block; the
    // last block's thread 0 fences again before the block reads.
    __syncthreads();
    if (tid == 0) {
        __threadfence();
        is_last = (atomicAdd(&inst_ticket[inst], 1u) == (unsigned)(R - 1));
        if (is_last) __threadfence();
    }
    __syncthreads();
    if (!is_last) return;
    const int32_t* cs = counts_src + (int64_t)inst * R * E;
    constexpr int kU = 16;  // loads in flight per thread: 64 rows of E <= 256 in one round
    if ((E & 3) == 0 && (E >> 2) <= kCountThreads && (reinterpret_cast<uintptr_t>(cs) & 15u) == 0) {
        // thread (g, c) sums the int4 column c (experts 4c .. 4c+3) over rows
        // g, g+G, ... (G = threads / (E/4)); the partials meet in hist[G][E]
        const int Q = E >> 2;
        const int G = kCountThreads / Q;
        const int c = tid % Q, g = tid / Q;
        if (g < G) {
            const int4* col = reinterpret_cast<const int4*>(cs) + c;
            int4 t = make_int4(0, 0, 0, 0);
            for (int r0 = g; r0 < R; r0 += kU * G) {
                int4 v[kU];
#pragma unroll
                for (int u = 0; u < kU; ++u) {
                    const int rr = r0 + u * G;
                    v[u] = (rr < R) ? __ldcg(col + (int64_t)rr * Q) : make_int4(0, 0, 0, 0);
                }
#pragma unroll
                for (int u = 0; u < kU; ++u) {
                    t.x += v[u].x;
                    t.y += v[u].y;
                    t.z += v[u].z;
                    t.w += v[u].w;
                }
            }
            reinterpret_cast<int4*>(hist)[g * Q + c] = t;
        }
        __syncthreads();
        for (int e = tid; e < E; e += kCountThreads) {
            int sum = 0;
            for (int gg = 0; gg < G; ++gg) sum += hist[gg * E + e];
            counts[(int64_t)inst * E + e] = sum;
        }
    } else if (E <= kCountThreads) {
        // thread (g, e) sums rows g, g+G, ... of column e, G = threads / E
        const int G = kCountThreads / E;
        const int e = tid % E, g = tid / E;
        int t = 0;
        if (g < G) {
            for (int r0 = g; r0 < R; r0 += kU * G) {
                int v[kU];
#pragma unroll
                for (int u = 0; u < kU; ++u) {
                    const int rr = r0 + u * G;
                    v[u] = (rr < R) ? __ldcg(cs + (int64_t)rr * E + e) : 0;
                }
#pragma unroll
                for (int u = 0; u < kU; ++u) t += v[u];
            }
            hist[g * E + e] = t;
        }
        __syncthreads();
        if (tid < E) {
            int sum = 0;
            for (int gg = 0; gg < G; ++gg) sum += hist[gg * E + tid];
            counts[(int64_t)inst * E + tid] = sum;
        }
    } else {
        for (int e = tid; e < E; e += kCountThreads) {
            int t = 0;
            for (int r0 = 0; r0 < R; r0 += kU) {
                int v[kU];
#pragma unroll
                for (int u = 0; u < kU; ++u)
                    v[u] = (r0 + u < R) ? __ldcg(cs + (int64_t)(r0 + u) * E + e) : 0;
#pragma unroll
                for (int u = 0; u < kU; ++u) t += v[u];
            }
            counts[(int64_t)inst * E + e] = t;
        }
    }
    if (tid == 0) inst_ticket[inst] = 0u;
}

size_t align_up(size_t x, size_t a) { return (x + a - 1) / a * a; }

}  // namespace

// Chunks per source rank: enough blocks for two per SM, chunks of at least
// kMinChunk slots, and at most a portable cluster.
int count_chunks_per_rank(const ep_domain_t& d, int64_t T, int32_t n_inst) {
    const int64_t blocks = (int64_t)n_inst * d.R;
    if (blocks <= 0) return 1;
    int64_t cps = (kTargetBlocks + blocks - 1) / blocks;
    const int64_t slots_per_rank = tokens_per_rank(T, d.R) * d.k;
    int64_t cap = slots_per_rank / kMinChunk;
    if (cap < 1) cap = 1;
    if (cap > kMaxChunksPerRank) cap = kMaxChunksPerRank;
    if (cps < EP_COUNT_MIN_CHUNKS) cps = EP_COUNT_MIN_CHUNKS;
    if (cps > cap) cps = cap;
    if (cps < 1) cps = 1;
    return (int)cps;
}

// Workspace: [n_inst] instance tickets, which must start at zero.
size_t count_workspace_bytes(const ep_domain_t& d, int64_t T, int32_t n_inst) {
    (void)d;
    (void)T;
    return align_up((size_t)n_inst * sizeof(uint32_t), 256);
}

size_t count_ticket_bytes(int32_t n_inst) { return (size_t)n_inst * sizeof(uint32_t); }

cudaError_t launch_count(const ep_domain_t& d, const int32_t* ids, int64_t T, int32_t n_inst,
                         int32_t* counts, int32_t* counts_src, int32_t* dev_status, void* ws,
                         cudaStream_t s, bool rows_only) {
    if (n_inst == 0) return cudaSuccess;
    const int cps = count_chunks_per_rank(d, T, n_inst);
    uint32_t* inst_ticket = static_cast<uint32_t*>(ws);
    const size_t smem = count_smem_bytes(d.E);
    const int64_t blocks = (int64_t)n_inst * d.R * cps;
    // one wave (every block resident at once) with more than two 16-byte
    // loads per thread: the latency-bound variant (64 registers)
    const int64_t n4 = tokens_per_rank(T, d.R) * d.k / cps / 4;
    const bool wave = blocks <= (int64_t)device_info().sms * kWaveBlocksPerSm &&
                      n4 > (int64_t)kCountThreads * 2;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)blocks);
    cfg.blockDim = dim3(kCountThreads);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = s;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = (unsigned)cps;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cfg.attrs = attr;
    cfg.numAttrs = cps > 1 ? 1 : 0;
    if (wave)
        return cudaLaunchKernelEx(&cfg, count_kernel<kVecWave, kWaveBlocksPerSm>, ids, T, (int)d.k,
                                  (int)d.R, (int)d.E, cps, counts, counts_src, dev_status,
                                  inst_ticket, rows_only ? 1 : 0);
    return cudaLaunchKernelEx(&cfg, count_kernel<kVec, kBatchMinBlocks>, ids, T, (int)d.k,
                              (int)d.R, (int)d.E, cps, counts, counts_src, dev_status, inst_ticket,
                              rows_only ? 1 : 0);
}

}  // namespace ultraep

// ---------------------------------------------------------------------------
// ep_count without a caller workspace.
//
// Some callers cannot hand the library any device memory beyond the inputs and
// outputs: for example a plugin running inside an inference engine whose
// device memory is all owned by the engine's pool, or a hot path where the
// latency and implicit device synchronisation of cudaMalloc are not
// acceptable.  For them the workspace of ep_count lives in the fixed array
// below, which every GPU that loads this library keeps for the life of the
// process.
namespace ultraep {
namespace {

constexpr size_t kNoAllocScratchBytes = (size_t)EP_COUNT_NOALLOC_SCRATCH_BYTES;

// Host code sees only a stand-in for this array: the device address of each
// GPU's copy comes from cudaGetSymbolAddress, taken once per device.
static __device__ __align__(256) unsigned char g_count_scratch[kNoAllocScratchBytes];

struct ScratchAddress {
    std::mutex mu;
    void* ptr[64] = {};
};

cudaError_t scratch_address(void** out) {
    static ScratchAddress cache;
    int dev = 0;
    cudaError_t err = cudaGetDevice(&dev);
    if (err != cudaSuccess) return err;
    if (dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
    std::lock_guard<std::mutex> lock(cache.mu);
    if (cache.ptr[dev] == nullptr) {
        void* p = nullptr;
        err = cudaGetSymbolAddress(&p, g_count_scratch);
        if (err != cudaSuccess) return err;
        cache.ptr[dev] = p;
    }
    *out = cache.ptr[dev];
    return cudaSuccess;
}

}  // namespace

size_t count_noalloc_scratch_capacity() { return kNoAllocScratchBytes; }

cudaError_t launch_count_noalloc(const ep_domain_t& d, const int32_t* ids, int64_t T,
                                 int32_t n_inst, int32_t* counts, int32_t* counts_src,
                                 int32_t* dev_status, cudaStream_t s) {
    if (n_inst == 0) return cudaSuccess;
    void* scratch = nullptr;
    cudaError_t err = scratch_address(&scratch);
    if (err != cudaSuccess) return err;
    // The array keeps whatever the previous call left in it: the tickets that
    // must start at zero are cleared on the caller's stream before the launch.
    const size_t tickets = count_ticket_bytes(n_inst);
    err = cudaMemsetAsync(scratch, 0, tickets, s);
    if (err != cudaSuccess) return err;
    return launch_count(d, ids, T, n_inst, counts, counts_src, dev_status, scratch, s);
}

}  // namespace ultraep
