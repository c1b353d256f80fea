// ep_count: exact per-expert load of the gate's top-k ids.
//
// UltraEP article (m.youleyou.com), "key design" section, forward-pass
// paragraph: the global load is obtained after gating and before planning.
//
// One block per (instance, source rank, chunk).  Each warp keeps a private
// shared-memory histogram; the lanes of a warp that hold the same expert id
// are grouped with match.any and the group's lowest lane adds the group size
// (warp-aggregated update), so a hot expert costs one shared atomic per warp
// step instead of one per slot.  The block's histogram is the sum of its
// warps' rows.  Chunks of one source rank meet in a last-block reduction that
// writes counts_src[r]; source ranks of one instance meet in a second one that
// writes counts.  The tickets that find the last block live at the start of
// the caller's workspace and are reset by that block, so they are zero again
// after every call; the rest of the workspace holds the chunk partials.
#include <mutex>

#include "common.cuh"

namespace ultraep {
namespace {

constexpr int kCountThreads = 512;
constexpr int kCountWarps = kCountThreads / 32;
constexpr int kCountUnroll = 4;
constexpr int kTargetBlocks = 2 * 148;
constexpr int kMinSlotsPerChunk = 2048;
constexpr int kMaxChunksPerRank = 64;

__global__ void __launch_bounds__(kCountThreads)
count_kernel(const int32_t* __restrict__ ids, int64_t T, int k, int R, int E, int cps,
             int32_t* __restrict__ counts, int32_t* __restrict__ counts_src,
             int32_t* dev_status, uint32_t* inst_ticket, uint32_t* rank_ticket,
             int32_t* partial) {
    extern __shared__ int32_t hist[];  // [kCountWarps][E]
    __shared__ int bad;
    __shared__ int is_last;

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int64_t blk = blockIdx.x;
    const int per_inst = R * cps;
    const int inst = (int)(blk / per_inst);
    const int rc = (int)(blk % per_inst);
    const int r = rc / cps, c = rc % cps;

    for (int x = threadIdx.x; x < kCountWarps * E; x += kCountThreads) hist[x] = 0;
    if (threadIdx.x == 0) bad = 0;
    __syncthreads();

    // this block's slots: chunk c of source rank r
    const int64_t Tr = tokens_per_rank(T, R);
    const int64_t t0 = min(T, (int64_t)r * Tr), t1 = min(T, (int64_t)(r + 1) * Tr);
    const int64_t a = t0 * k, len = (t1 - t0) * k;
    const int64_t s0 = a + len * c / cps, s1 = a + len * (c + 1) / cps;
    const int32_t* src = ids + (int64_t)inst * T * k;
    int32_t* row = hist + warp * E;

    int local_bad = 0;
    for (int64_t i0 = s0 + (int64_t)warp * 32 * kCountUnroll; i0 < s1;
         i0 += (int64_t)kCountThreads * kCountUnroll) {
        int ev[kCountUnroll];
#pragma unroll
        for (int u = 0; u < kCountUnroll; ++u) {
            const int64_t i = i0 + u * 32 + lane;
            ev[u] = (i < s1) ? __ldg(src + i) : -1;
        }
#pragma unroll
        for (int u = 0; u < kCountUnroll; ++u) {
            const int64_t i = i0 + u * 32 + lane;
            const bool in = i < s1;
            const bool valid = in && ev[u] >= 0 && ev[u] < E;
            local_bad |= (in && !valid);
            const unsigned grp = __match_any_sync(kFull, valid ? ev[u] : -1);
            if (valid && lane == __ffs(grp) - 1) atomicAdd(&row[ev[u]], __popc(grp));
        }
    }
    if (local_bad) bad = 1;
    __syncthreads();

    const int64_t rank_row = ((int64_t)inst * R + r) * E;
    int32_t* out = (cps == 1) ? counts_src + rank_row : partial + (rank_row * cps + (int64_t)c * E);
    for (int e = threadIdx.x; e < E; e += kCountThreads) {
        int s = 0;
        for (int w = 0; w < kCountWarps; ++w) s += hist[w * E + e];
        out[e] = s;
    }
    if (threadIdx.x == 0 && bad) raise_flag(dev_status, EP_DEV_BAD_ID);

    if (cps > 1) {
        // the last chunk of source rank r folds the chunk partials into counts_src[r]
        __threadfence();
        __syncthreads();
        if (threadIdx.x == 0)
            is_last = (atomicAdd(&rank_ticket[(int64_t)inst * R + r], 1u) == (unsigned)(cps - 1));
        __syncthreads();
        if (!is_last) return;
        __threadfence();
        for (int e = threadIdx.x; e < E; e += kCountThreads) {
            int s = 0;
            for (int cc = 0; cc < cps; ++cc) s += __ldcg(partial + rank_row * cps + (int64_t)cc * E + e);
            counts_src[rank_row + e] = s;
        }
        if (threadIdx.x == 0) rank_ticket[(int64_t)inst * R + r] = 0u;
    }

    // the last source rank of the instance folds counts_src into counts
    __threadfence();
    __syncthreads();
    if (threadIdx.x == 0) is_last = (atomicAdd(&inst_ticket[inst], 1u) == (unsigned)(R - 1));
    __syncthreads();
    if (!is_last) return;
    __threadfence();
    for (int e = threadIdx.x; e < E; e += kCountThreads) {
        int s = 0;
        for (int rr = 0; rr < R; ++rr) s += __ldcg(counts_src + ((int64_t)inst * R + rr) * E + e);
        counts[(int64_t)inst * E + e] = s;
    }
    if (threadIdx.x == 0) inst_ticket[inst] = 0u;
}

size_t align_up(size_t x, size_t a) { return (x + a - 1) / a * a; }

}  // namespace

int count_chunks_per_rank(const ep_domain_t& d, int64_t T, int32_t n_inst) {
    const int64_t blocks = (int64_t)n_inst * d.R;
    if (blocks <= 0) return 1;
    int64_t cps = (kTargetBlocks + blocks - 1) / blocks;
    const int64_t slots_per_rank = tokens_per_rank(T, d.R) * d.k;
    int64_t cap = slots_per_rank / kMinSlotsPerChunk;
    if (cap < 1) cap = 1;
    if (cap > kMaxChunksPerRank) cap = kMaxChunksPerRank;
    if (cps > cap) cps = cap;
    if (cps < 1) cps = 1;
    return (int)cps;
}

// Workspace: [n_inst] instance tickets | [n_inst][R] rank tickets | partials
// [n_inst][R][cps][E] (only when cps > 1).  Tickets must start at zero.
size_t count_workspace_bytes(const ep_domain_t& d, int64_t T, int32_t n_inst) {
    const int cps = count_chunks_per_rank(d, T, n_inst);
    size_t ints = (size_t)n_inst + (size_t)n_inst * d.R;
    if (cps > 1) ints += (size_t)n_inst * d.R * cps * d.E;
    return align_up(ints * sizeof(int32_t), 256);
}

cudaError_t launch_count(const ep_domain_t& d, const int32_t* ids, int64_t T, int32_t n_inst,
                         int32_t* counts, int32_t* counts_src, int32_t* dev_status, void* ws,
                         cudaStream_t s) {
    if (n_inst == 0) return cudaSuccess;
    const int cps = count_chunks_per_rank(d, T, n_inst);
    uint32_t* inst_ticket = static_cast<uint32_t*>(ws);
    uint32_t* rank_ticket = inst_ticket + n_inst;
    int32_t* partial = reinterpret_cast<int32_t*>(rank_ticket + (size_t)n_inst * d.R);
    const size_t smem = (size_t)kCountWarps * d.E * sizeof(int32_t);
    if (smem > 48 * 1024) {
        cudaError_t err = cudaFuncSetAttribute(count_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                               (int)smem);
        if (err != cudaSuccess) return err;
    }
    const int64_t blocks = (int64_t)n_inst * d.R * cps;
    count_kernel<<<(unsigned)blocks, kCountThreads, smem, s>>>(ids, T, d.k, d.R, d.E, cps, counts,
                                                              counts_src, dev_status, inst_ticket,
                                                              rank_ticket, partial);
    return cudaGetLastError();
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
    const size_t tickets = (size_t)n_inst * (d.R + 1) * sizeof(uint32_t);
    err = cudaMemsetAsync(scratch, 0, tickets, s);
    if (err != cudaSuccess) return err;
    return launch_count(d, ids, T, n_inst, counts, counts_src, dev_status, scratch, s);
}

}  // namespace ultraep
