/*
 * ultraep_oracle.c -- the CPU oracle of the UltraEP balancing hot path.
 *
 * TEST INFRASTRUCTURE ONLY.  Nothing on the product path may call, link or
 * load this file: only the tests, the smoke check and the benchmark's CPU
 * baseline leg use it.  It shares no code, header, table or helper with the
 * CUDA library; it is a plain, slow, single-threaded restatement of what each
 * step computes, written so that it can be checked against its sources by eye.
 *
 * Sources (the web pages this method is described on):
 *   [A] UltraEP article (m.youleyou.com), section "关键设计：让最优负载均衡走进生产"
 *       (key design): the reserved-slot paragraph, the forward-pass paragraph
 *       (global load after the gate -> replication planning -> reroute) and the
 *       control-plane paragraph (solve the quota each expert instance receives;
 *       each exploration step may instantiate a replica or move load).
 *   [B] "UltraEP brings real-time MoE balancing to Xiaohongshu's rack-scale
 *       inference stack", section "What UltraEP does".
 *   [C] EPLB tutorial, section "EPLB 和 DeepEP 怎么协同？" (dispatch looks up the
 *       physical replica of each top-k logical id; combine gathers results back
 *       to their logical owner).
 *
 * The pages give no formula; where they are silent this file takes the
 * plainest reading, and every such reading is marked READING below.
 *
 * Steps 1-5 are integer-only.  The weighted combine at the end of the file
 * (the step after unpermute) is the one place with floating point: float32
 * products and sums, each rounded separately (the build disables FMA
 * contraction), then a round-to-nearest-even conversion to bf16.
 *
 * Domain: R ranks, E logical experts, H = E/R home experts per rank, S spare
 * (redundant) slots per rank, P = R*(H+S) physical instances numbered
 * rank-major: p = r*(H+S) + j.  For j < H, p is the home instance of expert
 * r*H + j (READING: contiguous home placement); for H <= j < H+S it is spare
 * slot j-H of rank r.
 */
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

#define ORACLE_OK 0
#define ORACLE_ITER_LIMIT 2

/* ------------------------------------------------------------------------ */
/* Step 1: exact per-expert load ("global load after the gate", [A] forward-
 * pass paragraph; [B] "reads the actual token load after the gate").
 *
 * counts[e]        = #{ slots i = t*k + j : ids[i] == e }
 * counts_src[r][e] = the same, restricted to tokens of source rank r, where
 *                    READING: rank r owns tokens [r*Tr, (r+1)*Tr), Tr = ceil(T/R).
 * One (token, k) slot is one unit of load (READING).  Ids outside [0, E) are
 * skipped; the return value is how many were skipped.                        */
int64_t oracle_count(const int32_t *ids, int64_t T, int32_t k, int32_t R, int32_t E,
                     int32_t *counts, int32_t *counts_src)
{
    int64_t Tr = (T + R - 1) / R;
    int64_t invalid = 0;
    for (int32_t e = 0; e < E; e++) counts[e] = 0;
    for (int64_t x = 0; x < (int64_t)R * E; x++) counts_src[x] = 0;
    for (int64_t t = 0; t < T; t++) {
        int64_t r = t / Tr;
        for (int32_t j = 0; j < k; j++) {
            int32_t e = ids[t * k + j];
            if (e < 0 || e >= E) { invalid++; continue; }
            counts[e] += 1;
            counts_src[r * E + e] += 1;
        }
    }
    return invalid;
}

/* ------------------------------------------------------------------------ */
/* Step 2: the coupled replica-placement + quota solve ([A] control-plane
 * paragraph: solve how much load each expert instance finally receives; one
 * exploration step either instantiates a new replica or shifts load; [A]
 * reserved-slot paragraph: a fixed set of spare slots per rank, no allocation).
 *
 * The pages do not give the rule.  This is the fixed deterministic reading:
 *   start: each home instance carries its expert's whole count, spare slots
 *          are empty, L[r] = sum of the quotas of the instances on rank r;
 *   repeat:
 *     1. hot  = argmax_r L[r]                      (ties: lowest r)
 *     2. on hot, the instance with the largest quota (ties: lowest expert id);
 *        call its expert e
 *     3. eligible = ranks c != hot that hold e (home or spare slot) or that
 *        still have a free spare slot; none -> stop (slots ran out)
 *     4. cold = argmin over eligible of L[c]       (ties: lowest c)
 *     5. q = min(quota of the hot instance, floor((L[hot] - L[cold]) / 2));
 *        q == 0 -> stop
 *     6. if max_iters moves were made already -> stop with ITER_LIMIT, state
 *        left as it is
 *     7. move q from the hot instance to cold's instance of e; if cold does
 *        not hold e, its lowest-index free slot receives e first (quota 0)
 *   READING: stopping is global (the rule never retries another instance or
 *   rank); slots are never released inside one plan; a replica whose quota
 *   falls to 0 still holds its expert.
 *
 * Outputs: quota[P], slot_expert[R*S] (-1 = empty), rank_load[R], and the
 * logical->physical table as CSR ([C]: per logical expert, its physical
 * copies): inst_ptr[E+1]; for expert e the entries inst_ptr[e] ..
 * inst_ptr[e+1]-1 list the home instance first, then the replicas in
 * ascending p (READING), with inst_cum the inclusive running sum of their
 * quotas.  Returns ORACLE_OK or ORACLE_ITER_LIMIT; *n_iter = moves made.     */
/* The logical -> physical table of a finished plan: for every expert, its
 * home instance first, then its replicas by ascending p, with the inclusive
 * running sum of their quotas (the order reroute's quota-prefix rule uses). */
static void build_instance_table(int32_t R, int32_t E, int32_t S, const int32_t *quota,
                                 const int32_t *slot_expert, int32_t *inst_ptr,
                                 int32_t *inst_id, int32_t *inst_cum)
{
    int32_t H = E / R, W = H + S, P = R * W;
    int32_t m = 0;
    for (int32_t e = 0; e < E; e++) {
        int32_t cum = 0;
        inst_ptr[e] = m;
        int32_t home_p = (e / H) * W + (e % H);
        cum += quota[home_p];
        inst_id[m] = home_p;
        inst_cum[m] = cum;
        m++;
        for (int32_t p = 0; p < P; p++) {
            int32_t j = p % W;
            if (j < H) continue;
            if (slot_expert[(p / W) * S + (j - H)] != e) continue;
            cum += quota[p];
            inst_id[m] = p;
            inst_cum[m] = cum;
            m++;
        }
    }
    inst_ptr[E] = m;
}

int oracle_plan(const int32_t *counts, int32_t R, int32_t E, int32_t S, int32_t max_iters,
                int32_t *quota, int32_t *slot_expert, int32_t *rank_load,
                int32_t *inst_ptr, int32_t *inst_id, int32_t *inst_cum, int32_t *n_iter)
{
    int32_t H = E / R;
    int32_t W = H + S;               /* instances per rank */
    int32_t P = R * W;
    int64_t *L = (int64_t *)calloc((size_t)R, sizeof(int64_t));
    int status = ORACLE_OK;
    int32_t moves = 0;

    for (int32_t p = 0; p < P; p++) quota[p] = 0;
    for (int32_t x = 0; x < R * S; x++) slot_expert[x] = -1;
    for (int32_t e = 0; e < E; e++) {
        int32_t home = e / H;
        quota[home * W + (e % H)] = counts[e];
        L[home] += counts[e];
    }

    for (;;) {
        /* 1. hottest rank, lowest index on ties */
        int32_t hot = 0;
        for (int32_t r = 1; r < R; r++)
            if (L[r] > L[hot]) hot = r;

        /* 2. its largest-quota instance, lowest expert id on ties */
        int32_t src_p = -1, src_e = -1;
        for (int32_t j = 0; j < W; j++) {
            int32_t p = hot * W + j;
            int32_t e = (j < H) ? hot * H + j : slot_expert[hot * S + (j - H)];
            if (e < 0) continue;
            if (src_p < 0 || quota[p] > quota[src_p] || (quota[p] == quota[src_p] && e < src_e)) {
                src_p = p;
                src_e = e;
            }
        }

        /* 3-4. coldest eligible rank, lowest index on ties */
        int32_t cold = -1;
        for (int32_t c = 0; c < R; c++) {
            if (c == hot) continue;
            int holds = (src_e / H == c);
            int has_free = 0;
            for (int32_t j = 0; j < S; j++) {
                if (slot_expert[c * S + j] == src_e) holds = 1;
                if (slot_expert[c * S + j] < 0) has_free = 1;
            }
            if (!(holds || has_free)) continue;
            if (cold < 0 || L[c] < L[cold]) cold = c;
        }
        if (cold < 0) break;                          /* slots ran out */

        /* 5. amount to move */
        int64_t half = (L[hot] - L[cold]) / 2;
        int64_t q = quota[src_p] < half ? quota[src_p] : half;
        if (q <= 0) break;

        /* 6. safety cap */
        if (moves == max_iters) { status = ORACLE_ITER_LIMIT; break; }

        /* 7. cold's instance of src_e, creating a replica if needed */
        int32_t dst_p = -1;
        if (src_e / H == cold) dst_p = cold * W + (src_e % H);
        for (int32_t j = 0; j < S && dst_p < 0; j++)
            if (slot_expert[cold * S + j] == src_e) dst_p = cold * W + H + j;
        for (int32_t j = 0; j < S && dst_p < 0; j++)
            if (slot_expert[cold * S + j] < 0) {
                slot_expert[cold * S + j] = src_e;
                dst_p = cold * W + H + j;
            }

        quota[src_p] -= (int32_t)q;
        quota[dst_p] += (int32_t)q;
        L[hot] -= q;
        L[cold] += q;
        moves++;
    }

    for (int32_t r = 0; r < R; r++) rank_load[r] = (int32_t)L[r];

    build_instance_table(R, E, S, quota, slot_expert, inst_ptr, inst_id, inst_cum);
    *n_iter = moves;
    free(L);
    return status;
}

/* ------------------------------------------------------------------------ */
/* Step 3: reroute ([A] forward-pass paragraph: reroute splits the tokens of
 * one logical expert among its copies; [C]: dispatch maps every top-k
 * logical id to one physical copy).
 *
 * Slots are visited in ascending i = t*k + j.  The slots of expert e, in that
 * order, get within-expert ranks 0, 1, 2, ...; a slot of rank r goes to the
 * first instance in e's list whose inclusive cumulative quota exceeds r
 * (quota prefix rule).  Rows are grouped by instance p ascending and, inside
 * an instance, by slot i ascending:
 *   inst_offset[p] = sum of quota[p'] for p' < p   (inst_offset[P] = total)
 *   dst_row[i]     = inst_offset[p] + (slots already placed in p)
 *   src_slot[row]  = the slot placed at that row.
 * Slots with an id outside [0, E), or beyond the quotas of their expert, get
 * dst_row = -1 and no row.                                                  */
void oracle_reroute(const int32_t *ids, int64_t T, int32_t k, int32_t R, int32_t E, int32_t S,
                    const int32_t *quota, const int32_t *inst_ptr, const int32_t *inst_id,
                    const int32_t *inst_cum, int32_t *dst_row, int32_t *src_slot,
                    int32_t *inst_offset)
{
    int32_t P = R * (E / R + S);
    int64_t N = T * k;
    int64_t *seen = (int64_t *)calloc((size_t)E, sizeof(int64_t));
    int64_t *fill = (int64_t *)calloc((size_t)P, sizeof(int64_t));

    inst_offset[0] = 0;
    for (int32_t p = 0; p < P; p++) inst_offset[p + 1] = inst_offset[p] + quota[p];

    for (int64_t i = 0; i < N; i++) {
        int32_t e = ids[i];
        dst_row[i] = -1;
        if (e < 0 || e >= E) continue;
        int64_t r = seen[e]++;
        int32_t p = -1;
        for (int32_t m = inst_ptr[e]; m < inst_ptr[e + 1]; m++)
            if (inst_cum[m] > r) { p = inst_id[m]; break; }
        if (p < 0) continue;
        int64_t row = inst_offset[p] + fill[p]++;
        dst_row[i] = (int32_t)row;
        src_slot[row] = (int32_t)i;
    }
    free(seen);
    free(fill);
}

/* ------------------------------------------------------------------------ */
/* Step 4: permute -- the local half of dispatch ([C]): each grouped row is the
 * hidden row of the token its slot came from,
 *   out[row][:] = hidden[src_slot[row] / k][:]   for row in [0, n_rows),
 * copied as raw 16-bit words (READING: bit copy, never through float, so
 * NaN payloads and -0 survive).                                             */
void oracle_permute(const uint16_t *hidden, int32_t k, int32_t Hd,
                    const int32_t *src_slot, int64_t n_rows, uint16_t *out)
{
    for (int64_t row = 0; row < n_rows; row++) {
        int64_t t = src_slot[row] / k;
        for (int32_t h = 0; h < Hd; h++)
            out[row * Hd + h] = hidden[t * Hd + h];
    }
}

/* ------------------------------------------------------------------------ */
/* Step 5: unpermute -- the local half of combine ([C]: results on physical
 * copies are gathered back to their logical owner), with no gate weighting:
 *   y[t][j][:] = grouped[dst_row[t*k + j]][:]
 * READING: a slot with no row (dst_row < 0) gets a zero row.                */
void oracle_unpermute(const uint16_t *grouped, int64_t T, int32_t k, int32_t Hd,
                      const int32_t *dst_row, uint16_t *y)
{
    for (int64_t i = 0; i < T * k; i++) {
        int64_t row = dst_row[i];
        for (int32_t h = 0; h < Hd; h++)
            y[i * Hd + h] = (row < 0) ? 0 : grouped[row * Hd + h];
    }
}

/* ------------------------------------------------------------------------ */
/* Weighted combine -- combine with the gate weights ([C]: results on the
 * physical copies return to their logical owner; the owner sums its top-k
 * expert outputs weighted by the gate):
 *   y[t][:] = bf16( sum over j = 0, 1, ..., k-1 of  w[t][j] * grouped[dst_row[t*k+j]][:] )
 * READING (the pages give no arithmetic):
 *   - float32 throughout; each product w*x is rounded to float32, then added
 *     to the running sum (rounded to float32), in ascending j, starting from
 *     +0.0;
 *   - a slot with no row (dst_row < 0) adds nothing;
 *   - the sum is rounded to bf16 to nearest, ties to even; any NaN result is
 *     stored as the quiet NaN 0x7FC0 (NaN payloads are not portable).       */
static float bf16_bits_to_f32(uint16_t b)
{
    uint32_t u = (uint32_t)b << 16;
    float f;
    memcpy(&f, &u, sizeof f);
    return f;
}

static uint16_t f32_to_bf16_bits(float f)
{
    uint32_t u;
    memcpy(&u, &f, sizeof u);
    if ((u & 0x7F800000u) == 0x7F800000u && (u & 0x007FFFFFu) != 0) return 0x7FC0u;
    /* keep the upper 16 bits; round on the lower 16: above half rounds up,
     * exactly half rounds to the even upper value */
    uint32_t upper = u >> 16, lower = u & 0xFFFFu;
    if (lower > 0x8000u || (lower == 0x8000u && (upper & 1u))) upper += 1u;
    return (uint16_t)upper;
}

void oracle_combine(const uint16_t *grouped, int64_t T, int32_t k, int32_t Hd,
                    const int32_t *dst_row, const float *w, uint16_t *y)
{
    for (int64_t t = 0; t < T; t++) {
        for (int32_t h = 0; h < Hd; h++) {
            float sum = 0.0f;
            for (int32_t j = 0; j < k; j++) {
                int64_t row = dst_row[t * k + j];
                if (row < 0) continue;
                float x = bf16_bits_to_f32(grouped[row * Hd + h]);
                float prod = w[t * k + j] * x;
                sum = sum + prod;
            }
            y[t * Hd + h] = f32_to_bf16_bits(sum);
        }
    }
}

/* ------------------------------------------------------------------------ */
/* Replica weight staging -- the single-GPU half of weight distribution ([A]
 * forward-pass paragraph: after planning, the replicas' expert weights are
 * distributed to the ranks that host them; reserved-slot paragraph: the
 * redundant slots are fixed buffers, reused across layers).  For every spare
 * slot x = r*S + s:
 *   e = slot_expert[x];  e == -1: empty, nothing copied;
 *   e outside [-1, E): invalid, nothing copied, counted in *n_bad;
 *   prev given and prev[x] == e: the slot already holds e, nothing copied;
 *   else slot_w[x][:] = expert_w[e][:]  (expert_bytes bytes), counted.
 * READING: "new replica" is a slot whose expert differs from what it held.  */
void oracle_stage(const uint8_t *expert_w, int32_t E, int64_t expert_bytes,
                  const int32_t *slot_expert, const int32_t *prev, int32_t R, int32_t S,
                  uint8_t *slot_w, int32_t *n_copied, int64_t *n_bad)
{
    *n_copied = 0;
    *n_bad = 0;
    for (int64_t x = 0; x < (int64_t)R * S; x++) {
        int32_t e = slot_expert[x];
        if (e == -1) continue;
        if (e < -1 || e >= E) { (*n_bad)++; continue; }
        if (prev != NULL && prev[x] == e) continue;
        memcpy(slot_w + x * expert_bytes, expert_w + (int64_t)e * expert_bytes, (size_t)expert_bytes);
        (*n_copied)++;
    }
}

/* ------------------------------------------------------------------------ */
/* Planner variants (variants of the step-2 rule; the pages leave the rule
 * open).  flags:
 *   ORACLE_PLAN_SKIP: the base rule stops as soon as the hottest rank's
 *   largest instance cannot move; this variant tries the candidates in order
 *   and makes the first move that is possible:
 *     hot candidates: ranks by load, highest first (lowest rank on ties);
 *     for each, its instances with quota >= 1 by quota, largest first (lowest
 *     expert id on ties);
 *     candidate (h, instance of e) is possible when some rank c != h holds e
 *     or has a free spare slot and, with cold the least-loaded such rank
 *     (lowest index on ties), q = min(quota, floor((L[h] - L[cold]) / 2)) >= 1.
 *   ORACLE_PLAN_RELEASE: a replica (spare-slot instance) whose quota a move
 *   takes to 0 is released: the slot becomes empty (-1) and its rank no longer
 *   holds the expert, so later moves may fill it.
 * Without SKIP only the first candidate is tried (the base rule's choice).
 * The move is the base rule's (cold's instance of e, its lowest free slot if
 * it does not hold e).  It stops when no candidate is possible, or with
 * ORACLE_ITER_LIMIT when max_iters moves were made and another is possible.
 * Every move lowers sum L^2 (q <= (L[h] - L[cold]) / 2), so it ends.  With
 * SKIP, while the base rule's candidate is possible both make the same move,
 * so the plan is the base plan followed by further moves, none of which raises
 * the maximum load (a move from h to cold leaves both below the old L[h]). */
#define ORACLE_PLAN_SKIP 1
#define ORACLE_PLAN_RELEASE 2
int oracle_plan_variant(const int32_t *counts, int32_t R, int32_t E, int32_t S,
                        int32_t max_iters, int32_t flags, int32_t *quota, int32_t *slot_expert,
                        int32_t *rank_load, int32_t *inst_ptr, int32_t *inst_id,
                        int32_t *inst_cum, int32_t *n_iter)
{
    int32_t H = E / R;
    int32_t W = H + S;
    int32_t P = R * W;
    int64_t *L = (int64_t *)calloc((size_t)R, sizeof(int64_t));
    char *rank_tried = (char *)calloc((size_t)R, 1);
    char *inst_tried = (char *)calloc((size_t)W, 1);
    int status = ORACLE_OK;
    int32_t moves = 0;

    for (int32_t p = 0; p < P; p++) quota[p] = 0;
    for (int32_t x = 0; x < R * S; x++) slot_expert[x] = -1;
    for (int32_t e = 0; e < E; e++) {
        quota[(e / H) * W + (e % H)] = counts[e];
        L[e / H] += counts[e];
    }

    for (;;) {
        int found = 0;
        int32_t hot = -1, src_p = -1, src_e = -1, cold = -1;
        int64_t q = 0;
        memset(rank_tried, 0, (size_t)R);
        int32_t n_ranks = (flags & ORACLE_PLAN_SKIP) ? R : 1;
        int32_t n_insts = (flags & ORACLE_PLAN_SKIP) ? W : 1;
        for (int32_t n = 0; n < n_ranks && !found; n++) {
            /* next hot candidate: highest load among ranks not tried yet */
            hot = -1;
            for (int32_t r = 0; r < R; r++)
                if (!rank_tried[r] && (hot < 0 || L[r] > L[hot])) hot = r;
            rank_tried[hot] = 1;
            memset(inst_tried, 0, (size_t)W);
            for (int32_t nj = 0; nj < n_insts && !found; nj++) {
                /* next instance of hot: largest quota >= 1 not tried yet */
                src_p = -1;
                src_e = -1;
                int32_t src_j = -1;
                for (int32_t j = 0; j < W; j++) {
                    int32_t p = hot * W + j;
                    int32_t e = (j < H) ? hot * H + j : slot_expert[hot * S + (j - H)];
                    if (e < 0 || inst_tried[j] || quota[p] < 1) continue;
                    if (src_p < 0 || quota[p] > quota[src_p] ||
                        (quota[p] == quota[src_p] && e < src_e)) {
                        src_p = p;
                        src_e = e;
                        src_j = j;
                    }
                }
                if (src_p < 0) break;                 /* hot has nothing left to try */
                inst_tried[src_j] = 1;
                /* coldest rank that holds src_e or has a free slot */
                cold = -1;
                for (int32_t c = 0; c < R; c++) {
                    if (c == hot) continue;
                    int holds = (src_e / H == c);
                    int has_free = 0;
                    for (int32_t j = 0; j < S; j++) {
                        if (slot_expert[c * S + j] == src_e) holds = 1;
                        if (slot_expert[c * S + j] < 0) has_free = 1;
                    }
                    if (!(holds || has_free)) continue;
                    if (cold < 0 || L[c] < L[cold]) cold = c;
                }
                if (cold < 0) continue;
                int64_t half = (L[hot] - L[cold]) / 2;
                q = quota[src_p] < half ? quota[src_p] : half;
                if (q >= 1) found = 1;
            }
        }
        if (!found) break;
        if (moves == max_iters) { status = ORACLE_ITER_LIMIT; break; }

        int32_t dst_p = -1;
        if (src_e / H == cold) dst_p = cold * W + (src_e % H);
        for (int32_t j = 0; j < S && dst_p < 0; j++)
            if (slot_expert[cold * S + j] == src_e) dst_p = cold * W + H + j;
        for (int32_t j = 0; j < S && dst_p < 0; j++)
            if (slot_expert[cold * S + j] < 0) {
                slot_expert[cold * S + j] = src_e;
                dst_p = cold * W + H + j;
            }
        quota[src_p] -= (int32_t)q;
        quota[dst_p] += (int32_t)q;
        L[hot] -= q;
        L[cold] += q;
        if ((flags & ORACLE_PLAN_RELEASE) && src_p % W >= H && quota[src_p] == 0)
            slot_expert[hot * S + (src_p % W - H)] = -1;
        moves++;
    }

    for (int32_t r = 0; r < R; r++) rank_load[r] = (int32_t)L[r];
    build_instance_table(R, E, S, quota, slot_expert, inst_ptr, inst_id, inst_cum);
    *n_iter = moves;
    free(L);
    free(rank_tried);
    free(inst_tried);
    return status;
}
