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
// One warp per (layer, microbatch) instance, all state on chip:
//   - rank loads in registers, lane l holds ranks l and l+32;
//   - quota[P], slot_expert[R*S] and a 64-bit holder mask per expert in the
//     warp's slice of shared memory;
//   - argmax / argmin over ranks: one redux.sync (__reduce_max/min_sync) on the
//     load, then a ballot for the lowest rank that attains it (no key packing,
//     so loads up to 2^31-1 are exact);
//   - eligibility is a 64-bit mask: (holders of e | ranks with a free slot)
//     minus the hot rank.
#include <climits>

#include "common.cuh"

namespace ultraep {
namespace {

constexpr int kPlanWarps = 4;

__host__ __device__ inline size_t align16(size_t x) { return (x + 15) & ~size_t(15); }

__host__ __device__ inline size_t plan_warp_bytes(int R, int E, int S) {
    const int P = R * (E / R + S);
    return align16((size_t)P * 4) + align16((size_t)R * S * 4) + (size_t)E * 8;
}

__global__ void __launch_bounds__(kPlanWarps * 32)
plan_kernel(const int32_t* __restrict__ counts, int n_inst, int R, int E, int S, int max_iters,
            int32_t* __restrict__ quota_out, int32_t* __restrict__ slot_out,
            int32_t* __restrict__ load_out, int32_t* __restrict__ ptr_out,
            int32_t* __restrict__ id_out, int32_t* __restrict__ cum_out,
            int32_t* __restrict__ iter_out, int32_t* __restrict__ status_out) {
    extern __shared__ __align__(16) unsigned char smem[];
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int g = blockIdx.x * kPlanWarps + warp;
    if (g >= n_inst) return;  // whole warp; no block-wide barrier follows

    const int H = E / R, W = H + S, P = R * W;
    unsigned char* base = smem + (size_t)warp * plan_warp_bytes(R, E, S);
    int32_t* q = reinterpret_cast<int32_t*>(base);
    int32_t* slot = reinterpret_cast<int32_t*>(base + align16((size_t)P * 4));
    uint64_t* holder = reinterpret_cast<uint64_t*>(base + align16((size_t)P * 4) +
                                                   align16((size_t)R * S * 4));
    const int32_t* cnt = counts + (int64_t)g * E;

    for (int p = lane; p < P; p += 32) q[p] = 0;
    for (int x = lane; x < R * S; x += 32) slot[x] = -1;
    __syncwarp();
    for (int e = lane; e < E; e += 32) {
        const int r = e / H;
        q[r * W + (e - r * H)] = cnt[e];
        holder[e] = 1ull << r;
    }
    __syncwarp();

    // loads of ranks lane and lane+32; -1 marks a rank that does not exist
    int L0 = -1, L1 = -1;
    if (lane < R) {
        int s = 0;
        for (int j = 0; j < H; ++j) s += q[lane * W + j];
        L0 = s;
    }
    if (lane + 32 < R) {
        int s = 0;
        for (int j = 0; j < H; ++j) s += q[(lane + 32) * W + j];
        L1 = s;
    }
    int used0 = 0, used1 = 0;  // filled spare slots of ranks lane, lane+32
    const uint64_t ranks = (R == 64) ? ~0ull : ((1ull << R) - 1);
    uint64_t free_mask = (S > 0) ? ranks : 0ull;  // ranks with a free spare slot
    int iters = 0, status = EP_OK;

    // counts must be >= 0 with a total below 2^31; otherwise the instance is
    // rejected (EP_ERR_INVAL) and its outputs describe the home-only placement
    {
        bool bad = false;
        long long tot = 0;
        for (int e = lane; e < E; e += 32) {
            bad |= cnt[e] < 0;
            tot += cnt[e];
        }
        bad = __any_sync(kFull, bad);
        for (int o = 16; o > 0; o >>= 1) tot += __shfl_xor_sync(kFull, tot, o);
        if (bad || tot > (long long)INT_MAX) status = EP_ERR_INVAL;
    }

    while (status == EP_OK) {
        // 1. hottest rank, lowest index on ties
        const int Lmax = __reduce_max_sync(kFull, max(L0, L1));
        const unsigned bh = __ballot_sync(kFull, L0 == Lmax);
        const int hot = bh ? __ffs(bh) - 1 : 32 + __ffs(__ballot_sync(kFull, L1 == Lmax)) - 1;

        // 2. hot's largest-quota instance, lowest expert id on ties (lane j = instance j)
        int ej = -1, qj = -1;
        if (lane < W) {
            ej = (lane < H) ? hot * H + lane : slot[hot * S + (lane - H)];
            if (ej >= 0) qj = q[hot * W + lane];
        }
        const int qmax = __reduce_max_sync(kFull, qj);
        const unsigned tie = __ballot_sync(kFull, qj == qmax);
        int src_lane;
        if (__popc(tie) == 1) {
            src_lane = __ffs(tie) - 1;
        } else {
            const bool in_tie = (tie >> lane) & 1u;
            const int emin = __reduce_min_sync(kFull, in_tie ? ej : INT_MAX);
            src_lane = __ffs(__ballot_sync(kFull, in_tie && ej == emin)) - 1;
        }
        const int e = __shfl_sync(kFull, ej, src_lane);

        // 3. eligible ranks: hold e or have a free slot, not the hot rank
        const uint64_t hm = holder[e];
        const uint64_t elig = (hm | free_mask) & ~(1ull << hot);
        if (elig == 0ull) break;  // slots ran out

        // 4. coldest eligible rank, lowest index on ties
        const int c0 = ((elig >> lane) & 1ull) ? L0 : INT_MAX;
        const int c1 = ((elig >> (lane + 32)) & 1ull) ? L1 : INT_MAX;
        const int Lmin = __reduce_min_sync(kFull, min(c0, c1));
        const unsigned bc = __ballot_sync(kFull, c0 == Lmin);
        const int cold = bc ? __ffs(bc) - 1 : 32 + __ffs(__ballot_sync(kFull, c1 == Lmin)) - 1;

        // 5. amount
        const int mv = min(qmax, (Lmax - Lmin) >> 1);
        if (mv <= 0) break;
        // 6. safety cap
        if (iters == max_iters) {
            status = EP_ERR_ITER_LIMIT;
            break;
        }

        // 7. cold's instance of e, filling its lowest free slot if it has none
        int p_dst;
        if ((hm >> cold) & 1ull) {
            if (cold == e / H) {
                p_dst = cold * W + (e - cold * H);
            } else {
                const unsigned bs = __ballot_sync(kFull, lane < S && slot[cold * S + lane] == e);
                p_dst = cold * W + H + __ffs(bs) - 1;
            }
        } else {
            const int uc = __shfl_sync(kFull, cold < 32 ? used0 : used1, cold & 31);
            p_dst = cold * W + H + uc;
            if (lane == 0) {
                slot[cold * S + uc] = e;
                holder[e] = hm | (1ull << cold);
            }
            if (lane == (cold & 31)) {
                if (cold < 32) ++used0; else ++used1;
            }
            if (uc + 1 == S) free_mask &= ~(1ull << cold);
        }
        if (lane == 0) {
            q[hot * W + src_lane] -= mv;
            q[p_dst] += mv;
        }
        if (lane == (hot & 31)) {
            if (hot < 32) L0 -= mv; else L1 -= mv;
        }
        if (lane == (cold & 31)) {
            if (cold < 32) L0 += mv; else L1 += mv;
        }
        ++iters;
        __syncwarp();
    }
    __syncwarp();

    // ---- outputs
    int32_t* qo = quota_out + (int64_t)g * P;
    for (int p = lane; p < P; p += 32) qo[p] = q[p];
    int32_t* so = slot_out + (int64_t)g * R * S;
    for (int x = lane; x < R * S; x += 32) so[x] = slot[x];
    if (lane < R) load_out[(int64_t)g * R + lane] = L0;
    if (lane + 32 < R) load_out[(int64_t)g * R + lane + 32] = L1;

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

}  // namespace

cudaError_t launch_plan(const ep_domain_t& d, const int32_t* counts, int32_t n_inst,
                        int32_t max_iters, int32_t* quota, int32_t* slot_expert, int32_t* rank_load,
                        int32_t* inst_ptr, int32_t* inst_id, int32_t* inst_cum, int32_t* n_iter,
                        int32_t* inst_status, cudaStream_t s) {
    if (n_inst == 0) return cudaSuccess;
    const size_t smem = kPlanWarps * plan_warp_bytes(d.R, d.E, d.S);
    if (smem > 48 * 1024) {
        cudaError_t err = cudaFuncSetAttribute(plan_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                               (int)smem);
        if (err != cudaSuccess) return err;
    }
    const unsigned blocks = (unsigned)((n_inst + kPlanWarps - 1) / kPlanWarps);
    plan_kernel<<<blocks, kPlanWarps * 32, smem, s>>>(counts, n_inst, d.R, d.E, d.S,
                                                       max_iters, quota, slot_expert,
                                                       rank_load, inst_ptr, inst_id, inst_cum,
                                                       n_iter, inst_status);
    return cudaGetLastError();
}

}  // namespace ultraep
