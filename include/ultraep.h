/*
 * ultraep.h -- C ABI of the UltraEP per-microbatch, per-layer balancing hot path
 * (hand-written CUDA for sm_103a, library libultraep_b300.so).
 *
 * The path, per (layer, microbatch) "instance":
 *     ep_count -> ep_plan -> ep_reroute -> ep_permute  [-> experts ->]  ep_unpermute
 *
 * Sources: UltraEP article (m.youleyou.com), section "key design"
 * (关键设计：让最优负载均衡走进生产); "UltraEP brings real-time MoE balancing to
 * Xiaohongshu's rack-scale inference stack", section "What UltraEP does";
 * EPLB tutorial, section "EPLB 和 DeepEP 怎么协同？" (dispatch / combine).
 *
 * Simulated EP domain (one GPU holds all of it): R ranks, E logical experts,
 * H = E/R home experts per rank, S spare ("redundant") slots per rank, top-k k.
 * Physical instances are numbered rank-major, P = R*(H+S):
 *     p = r*(H+S) + j;  j < H: home instance of expert r*H + j;
 *                       H <= j < H+S: spare slot j-H of rank r.
 * A token-slot is one (token t, choice j) pair, slot index i = t*k + j; one
 * slot is one unit of load.  Source rank of token t: t / ceil(T/R).
 *
 * Conventions shared by every entry point
 *  - Every pointer argument is a DEVICE pointer owned by the caller.  The
 *    library never allocates or frees memory and never synchronises with the
 *    host: every call only enqueues work on `stream` (a cudaStream_t; NULL is
 *    the legacy default stream) and returns.
 *  - Batching: n_inst independent instances are laid out back to back along the
 *    leading dimension of every array (e.g. topk_ids is [n_inst][T][k]).
 *  - Pointers must be 4-byte aligned (int32 arrays) and 16-byte aligned
 *    (bf16 row arrays); bf16 rows must be a multiple of 16 bytes (Hd % 8 == 0).
 *  - The return value reports only errors the host can see before launching:
 *    EP_ERR_INVAL (bad shape, null or misaligned pointer, limit exceeded),
 *    EP_ERR_WORKSPACE (workspace too small) and EP_ERR_CUDA (a launch failed).
 *    On any error nothing is enqueued (EP_ERR_CUDA: the launch that failed
 *    may have been partially enqueued).
 *  - Errors that depend on the data are reported on the device: `dev_status`
 *    (an int32 the caller zeroes; calls OR EP_DEV_* bits into it) and the
 *    per-instance `inst_status` of ep_plan.  Kernels never trap.
 *  - Limits: 1 <= R <= 64, E % R == 0, 1 <= E <= 1024, 0 <= S, H + S <= 32,
 *    1 <= k <= 32, k <= E, 0 <= T, T*k < 2^31, n_inst >= 0, and for the bf16
 *    row calls 0 <= Hd <= 2^29 (a row of at most 1 GiB).
 */
#ifndef ULTRAEP_H
#define ULTRAEP_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef struct {
    int32_t R; /* ranks */
    int32_t E; /* logical experts; H = E / R must be an integer */
    int32_t S; /* spare slots per rank */
    int32_t k; /* top-k */
} ep_domain_t;

typedef enum {
    EP_OK = 0,
    EP_ERR_INVAL = 1,
    EP_ERR_ITER_LIMIT = 2, /* per-instance status of ep_plan */
    EP_ERR_BAD_ID = 3,     /* reserved for callers mapping EP_DEV_BAD_ID */
    EP_ERR_WORKSPACE = 4,
    EP_ERR_CUDA = 5
} ep_status_t;

/* bits OR-ed into *dev_status by the kernels */
#define EP_DEV_BAD_ID 1         /* an expert id outside [0, E) was seen and skipped */
#define EP_DEV_QUOTA_OVERFLOW 2 /* a slot's within-expert rank exceeded its expert's quotas */
#define EP_DEV_ROW_RANGE 4      /* a dst_row entry was >= T*k; that row was skipped */
#define EP_DEV_COPY_TIMEOUT 8   /* a row copy did not complete within the kernel's wait
                                   limit; the call stopped early and its output is incomplete */
#define EP_DEV_COUNTS_MISMATCH 16 /* ep_reroute: counts_src does not hold the per-source-rank
                                     counts of these ids (e.g. another layer's); every row of
                                     that instance may be wrong */
#define EP_DEV_COPY_UNDRAINED 32  /* ep_permute, after EP_DEV_COPY_TIMEOUT: copies into shared
                                     memory were still pending when the block gave up waiting
                                     for them and exited; the whole launch's output, and any
                                     kernel sharing the GPU with it, is suspect */

#define EP_PLAN_MAX_ITERS (1 << 16)
#define EP_MAX_R 64
#define EP_MAX_E 1024
#define EP_MAX_K 32
#define EP_MAX_INSTANCES_PER_RANK 32

/* Bytes of workspace ep_count needs for this shape.  Returns 0 for invalid
 * arguments. */
size_t ep_count_workspace_bytes(const ep_domain_t *dom, int64_t T, int32_t n_inst);

/*
 * ep_count -- exact global load after the gate (UltraEP article, "key design",
 * forward-pass paragraph: the global load is obtained after gating, before
 * replication planning; rack-scale summary, "What UltraEP does": the actual
 * token load is read after the gate and before dispatch).
 *
 *   topk_ids   [n_inst][T][k] int32   the gate's top-k logical expert ids
 *   counts     [n_inst][E]    int32   out: counts[e] = #{slots with id e}
 *   counts_src [n_inst][R][E] int32   out: the same per source rank
 *                                     (tokens [r*ceil(T/R), (r+1)*ceil(T/R)))
 *   dev_status int32                  out: |= EP_DEV_BAD_ID if an id was
 *                                     outside [0, E) (it is skipped)
 *   workspace  ep_count_workspace_bytes() bytes, caller-owned, 16-byte
 *              aligned.  It holds one ticket per instance (its first 4*n_inst
 *              bytes), which finds the last block of the instance: the tickets
 *              must be zero before the first call, and every call resets them
 *              to zero on completion, so the workspace can be reused by later
 *              calls on the same stream without clearing.  Calls that share a
 *              workspace must not overlap on the GPU.
 */
ep_status_t ep_count(const ep_domain_t *dom, const int32_t *topk_ids, int64_t T, int32_t n_inst,
                     int32_t *counts, int32_t *counts_src, int32_t *dev_status,
                     void *workspace, size_t workspace_bytes, void *stream);

/*
 * ep_count_noalloc -- ep_count for callers that cannot allocate device memory.
 * The pages have no counterpart of this entry point.  It serves callers that
 * cannot hand the library a workspace: for example a plugin running inside an
 * inference engine whose device memory all belongs to the engine's pool, or a
 * hot path that cannot afford the latency and implicit device synchronisation
 * of cudaMalloc.  Arguments and results are those of ep_count without the
 * workspace, which here is a fixed array of EP_COUNT_NOALLOC_SCRATCH_BYTES
 * inside the library; every GPU that loads the library holds that array until
 * the process exits.
 *  - Returns EP_ERR_WORKSPACE, enqueueing nothing, when the shape needs more
 *    than that (ep_count_workspace_bytes(dom, T, n_inst) is larger).
 *  - The first call on a device, with that device current, looks up the
 *    array's device address (cudaGetSymbolAddress) and keeps it for the life
 *    of the process; make that first call before any stream capture.  After
 *    cudaDeviceReset on that device the kept address is stale: do not call
 *    ep_count_noalloc on a device after resetting it.
 *  - All calls on a device share the one array.  Each call clears the part
 *    that must start at zero (the tickets) on `stream` and then launches, so
 *    calls that overlap on the GPU (different streams or threads) race and
 *    give wrong counts: keep them ordered, e.g. on one stream.
 *  - Allocates nothing: it calls no cudaMalloc, cudaFree or allocating
 *    library routine.
 */
#define EP_COUNT_NOALLOC_SCRATCH_BYTES (64u << 10) /* tickets of up to 16384 instances per call */
ep_status_t ep_count_noalloc(const ep_domain_t *dom, const int32_t *topk_ids, int64_t T,
                             int32_t n_inst, int32_t *counts, int32_t *counts_src,
                             int32_t *dev_status, void *stream);

/*
 * ep_plan -- the coupled replica-placement + quota solve (UltraEP article,
 * "key design", control-plane paragraph: solve how much load each expert
 * instance finally receives, each step either instantiating a replica or
 * shifting load, warp-level parallel; reserved-slot paragraph: a fixed set of
 * spare slots per rank).  One warp solves each instance.
 *
 * The pages do not state the rule; this library fixes one deterministic rule:
 *   start: home instances carry their expert's count, spare slots are empty,
 *          L[r] = load of rank r;
 *   repeat: hot = argmax L (lowest r on ties); e = expert of hot's
 *     largest-quota instance (lowest expert id on ties); eligible = ranks
 *     c != hot that hold e or have a free spare slot (none: stop);
 *     cold = argmin L over eligible (lowest c on ties);
 *     q = min(that instance's quota, floor((L[hot] - L[cold]) / 2)) (0: stop);
 *     after max_iters moves, if another move is due: stop with
 *     EP_ERR_ITER_LIMIT, leaving the state as it is;
 *     move q to cold's instance of e, first filling cold's lowest free slot
 *     with e if cold does not hold e.  Slots are never released.
 *
 *   counts      [n_inst][E]       int32 in
 *   max_iters   cap on the moves of one instance; <= 0 means EP_PLAN_MAX_ITERS
 *   quota       [n_inst][P]       int32 out: load of every physical instance
 *   slot_expert [n_inst][R][S]    int32 out: expert in each spare slot, -1 empty
 *   rank_load   [n_inst][R]       int32 out
 *   inst_ptr    [n_inst][E+1]     int32 out: CSR row pointers of the
 *   inst_id     [n_inst][E+R*S]   int32 out:   logical -> physical table; for
 *   inst_cum    [n_inst][E+R*S]   int32 out:   expert e, entries inst_ptr[e] ..
 *               inst_ptr[e+1]-1 list its home instance first and then its
 *               replicas by ascending p, with inst_cum the inclusive running
 *               sum of their quotas.  Entries past inst_ptr[E] are not written.
 *   n_iter      [n_inst]          int32 out: moves made
 *   inst_status [n_inst]          int32 out: EP_OK, EP_ERR_ITER_LIMIT, or
 *               EP_ERR_INVAL when a count is negative or the counts sum to
 *               2^31 or more (no move is made; outputs show home placement)
 */
ep_status_t ep_plan(const ep_domain_t *dom, const int32_t *counts, int32_t n_inst,
                    int32_t max_iters, int32_t *quota, int32_t *slot_expert, int32_t *rank_load,
                    int32_t *inst_ptr, int32_t *inst_id, int32_t *inst_cum,
                    int32_t *n_iter, int32_t *inst_status, void *stream);

/*
 * ep_plan_ex -- ep_plan with variants of the rule (the pages leave the rule
 * open; these are the variants this library compares with it).  flags:
 *   EP_PLAN_SKIP: when the hottest rank's largest instance cannot move, try
 *     its next instances and then the next-hottest ranks (ranks by load,
 *     highest first; instances with quota >= 1 by quota, largest first; the
 *     base rule's ties) and make the first move that can be made; stop when
 *     none can.  The plan is the base plan followed by further moves, none of
 *     which raises the maximum load.
 *   EP_PLAN_RELEASE: a spare-slot instance that a move leaves at quota 0 frees
 *     its slot (slot_expert -1; the rank no longer holds the expert).
 * flags = 0 is ep_plan.  Other bits: EP_ERR_INVAL.  Arguments otherwise as
 * ep_plan.
 */
#define EP_PLAN_SKIP 1
#define EP_PLAN_RELEASE 2
ep_status_t ep_plan_ex(const ep_domain_t *dom, const int32_t *counts, int32_t n_inst,
                       int32_t max_iters, int32_t flags, int32_t *quota, int32_t *slot_expert,
                       int32_t *rank_load, int32_t *inst_ptr, int32_t *inst_id,
                       int32_t *inst_cum, int32_t *n_iter, int32_t *inst_status, void *stream);

/*
 * ep_reroute -- split every logical expert's slots among its instances
 * (UltraEP article, "key design", forward-pass paragraph: reroute divides the
 * tokens of one logical expert among its replicas; EPLB tutorial, dispatch:
 * every top-k logical id is mapped to one physical copy).
 *
 * Quota-prefix rule: the slots of expert e, in ascending slot index, get
 * within-expert ranks 0, 1, ...; a slot of rank r goes to the first entry of
 * e's instance list whose inst_cum exceeds r.  Rows are grouped by instance p
 * ascending and, inside an instance, by slot index ascending.
 *
 *   topk_ids    [n_inst][T][k]   int32 in
 *   counts_src  [n_inst][R][E]   int32 in: ep_count's per-source-rank counts
 *               of the SAME ids.  They stand in for a per-call workspace: the
 *               block of source rank r starts its ranks at the prefix of
 *               counts_src over ranks below r, so no second pass over the ids
 *               is needed.  After ranking its slots each block checks its own
 *               row against what it counted; a difference raises
 *               EP_DEV_COUNTS_MISMATCH, and then dst_row, src_slot and
 *               inst_offset of that instance must be treated as invalid.
 *   quota, inst_ptr, inst_id, inst_cum   in (from ep_plan)
 *   dst_row     [n_inst][T*k]    int32 out: row of each slot; -1 for a slot
 *                                with an invalid id or beyond its quotas
 *   src_slot    [n_inst][T*k]    int32 out (may be NULL): slot of each row;
 *                                entries past the last row are not written
 *   inst_offset [n_inst][P+1]    int32 out: first row of every instance
 *                                (exclusive prefix sum of quota)
 *   dev_status  int32            out: |= EP_DEV_BAD_ID, EP_DEV_QUOTA_OVERFLOW,
 *                                EP_DEV_COUNTS_MISMATCH
 */
ep_status_t ep_reroute(const ep_domain_t *dom, const int32_t *topk_ids, int64_t T, int32_t n_inst,
                       const int32_t *counts_src, const int32_t *quota, const int32_t *inst_ptr,
                       const int32_t *inst_id, const int32_t *inst_cum, int32_t *dst_row,
                       int32_t *src_slot, int32_t *inst_offset, int32_t *dev_status,
                       void *stream);

/*
 * ep_balance -- ep_count, ep_plan and ep_reroute in one call, for the
 * per-layer critical path (UltraEP article, "key design", forward-pass
 * paragraph: obtain the load, solve the plan, reroute, all on the GPU before
 * dispatch).  The three kernels are enqueued back to back on `stream` with
 * programmatic dependent launch: the planner launches while the count is
 * still running and waits on the device for its per-source-rank counts, which
 * it sums into counts itself (the count kernel stops at counts_src); the
 * reroute launches while the planner is still running, loads and ranks its
 * first chunk of ids and reads counts_src (neither depends on anything the
 * planner computes: the count grid completed before the planner let the
 * reroute launch) and only then waits for the plan.  Results are exactly
 * those of the three separate calls.
 *
 *   topk_ids, T, n_inst, max_iters, dev_status   as for ep_count / ep_plan
 *   workspace   as for ep_count (ep_count_workspace_bytes() bytes)
 *   out         the output arrays of the three calls (layouts as documented
 *               there); out->src_slot may be NULL
 * Errors: EP_ERR_INVAL / EP_ERR_WORKSPACE before anything is enqueued;
 * EP_ERR_CUDA if a launch failed (earlier launches of the call may have been
 * enqueued).
 */
typedef struct {
    int32_t *counts;      /* [n_inst][E]       */
    int32_t *counts_src;  /* [n_inst][R][E]    */
    int32_t *quota;       /* [n_inst][P]       */
    int32_t *slot_expert; /* [n_inst][R][S]    */
    int32_t *rank_load;   /* [n_inst][R]       */
    int32_t *inst_ptr;    /* [n_inst][E+1]     */
    int32_t *inst_id;     /* [n_inst][E+R*S]   */
    int32_t *inst_cum;    /* [n_inst][E+R*S]   */
    int32_t *n_iter;      /* [n_inst]          */
    int32_t *inst_status; /* [n_inst]          */
    int32_t *dst_row;     /* [n_inst][T*k]     */
    int32_t *src_slot;    /* [n_inst][T*k] or NULL */
    int32_t *inst_offset; /* [n_inst][P+1]     */
} ep_balance_out_t;

ep_status_t ep_balance(const ep_domain_t *dom, const int32_t *topk_ids, int64_t T,
                       int32_t n_inst, int32_t max_iters, const ep_balance_out_t *out,
                       int32_t *dev_status, void *workspace, size_t workspace_bytes,
                       void *stream);

/*
 * ep_permute -- the local half of dispatch (EPLB tutorial, "EPLB 和 DeepEP
 * 怎么协同？": every token is sent to the physical copy of each of its
 * top-k experts): out[dst_row[t*k+j]] = hidden[t] for every slot with a row.
 * Rows are copied bit for bit (bf16 payload never converted).
 *
 *   hidden  [n_inst][T][Hd]   bf16 in
 *   dst_row [n_inst][T*k]     int32 in (from ep_reroute); < 0: no row
 *   out     [n_inst][T*k][Hd] bf16 out; rows nobody maps to are not written
 *   dev_status int32          out: |= EP_DEV_ROW_RANGE for a dst_row >= T*k;
 *                             |= EP_DEV_COPY_TIMEOUT if a bulk row copy did not
 *                             complete within the kernel's bounded wait (the
 *                             output is then incomplete); |= EP_DEV_COPY_UNDRAINED
 *                             if, after that, copies were still pending when the
 *                             block exited
 *
 * Rows of 1 KiB or more move through shared memory with TMA bulk copies
 * (one global->shared copy per row, k shared->global copies); shorter rows
 * use 16-byte vector loads and stores.
 */
ep_status_t ep_permute(const void *hidden, int64_t T, int32_t k, int32_t Hd, int32_t n_inst,
                       const int32_t *dst_row, void *out, int32_t *dev_status, void *stream);

/*
 * ep_unpermute -- the local half of combine (EPLB tutorial, same section:
 * results on physical copies are gathered back to their logical owner), with
 * no gate weighting: y[t][j] = grouped[dst_row[t*k+j]]; a slot with no row
 * (dst_row < 0) gets a zero row.
 *
 *   grouped [n_inst][T*k][Hd] bf16 in
 *   dst_row [n_inst][T*k]     int32 in
 *   y       [n_inst][T][k][Hd] bf16 out
 *   dev_status int32          out: |= EP_DEV_ROW_RANGE for a dst_row >= T*k
 *                             (that output row is zeroed)
 */
ep_status_t ep_unpermute(const void *grouped, int64_t T, int32_t k, int32_t Hd, int32_t n_inst,
                         const int32_t *dst_row, void *y, int32_t *dev_status, void *stream);

/*
 * ep_combine -- the combine step with the gate weights, fused with the gather
 * of unpermute (EPLB tutorial, "EPLB 和 DeepEP 怎么协同？": results on the
 * physical copies return to their logical owner, which adds its top-k expert
 * outputs weighted by the gate):
 *     y[t][:] = bf16( sum over j = 0 .. k-1 of weights[t][j] * grouped[dst_row[t*k+j]][:] )
 * The pages give no arithmetic; this library fixes it: float32, every product
 * and every partial sum rounded on its own (no fused multiply-add), in
 * ascending j starting from +0.0; a slot with no row (dst_row < 0) adds
 * nothing; the sum is rounded to bf16 to nearest, ties to even; any NaN
 * result is stored as 0x7FC0.  The result is therefore deterministic and
 * bit-reproducible on any IEEE float32 machine.
 *
 *   grouped [n_inst][T*k][Hd] bf16 in (expert outputs in grouped row order)
 *   dst_row [n_inst][T*k]     int32 in (from ep_reroute)
 *   weights [n_inst][T][k]    float32 in (the gate's top-k weights)
 *   y       [n_inst][T][Hd]   bf16 out
 *   dev_status int32          out: |= EP_DEV_ROW_RANGE for a dst_row >= T*k
 *                             (that slot adds nothing)
 */
ep_status_t ep_combine(const void *grouped, int64_t T, int32_t k, int32_t Hd, int32_t n_inst,
                       const int32_t *dst_row, const float *weights, void *y,
                       int32_t *dev_status, void *stream);

/*
 * ep_stage -- replica weight staging, the single-GPU half of weight
 * distribution (UltraEP article, "key design", forward-pass paragraph: after
 * planning, the replicas' expert weights go to the ranks hosting them;
 * reserved-slot paragraph: the redundant slots are fixed buffers reused
 * across layers).  For every spare slot x = r*S + s of every instance:
 *     e = slot_expert[x]; e == -1: empty, nothing copied;
 *     e outside [-1, E): nothing copied, |= EP_DEV_BAD_ID;
 *     prev_slot_expert given and prev_slot_expert[x] == e: the slot already
 *         holds e, nothing copied (only new replicas move);
 *     else slot_w[x][:] = expert_w[e][:]   (expert_bytes bytes).
 *
 *   expert_w         [n_inst][E][expert_bytes] in (per-layer expert weights)
 *   expert_bytes     bytes of one expert's weights, a multiple of 16
 *   slot_expert      [n_inst][R][S] int32 in (from ep_plan)
 *   prev_slot_expert [n_inst][R][S] int32 in, may be NULL
 *   slot_w           [n_inst][R][S][expert_bytes] out (a cross-layer reused
 *                    buffer: n_inst = 1, staged again for every layer)
 * expert_w and slot_w must be 16-byte aligned.
 */
ep_status_t ep_stage(const ep_domain_t *dom, int32_t n_inst, const void *expert_w,
                     int64_t expert_bytes, const int32_t *slot_expert,
                     const int32_t *prev_slot_expert, void *slot_w, int32_t *dev_status,
                     void *stream);

/* Static string naming a status code. */
const char *ep_status_str(ep_status_t status);

#ifdef __cplusplus
}
#endif

#endif /* ULTRAEP_H */
