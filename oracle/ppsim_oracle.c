/*
 * ppsim_oracle.c -- plain, slow, CPU reference of the pipeline-schedule evaluator.
 *
 * TEST INFRASTRUCTURE ONLY.  This file is the oracle that the CUDA library is
 * checked against.  Only the tests, the smoke check and the benchmark's CPU
 * baseline may load it; the product path never does.  It shares no code,
 * header, table or constant with the CUDA library: every rule below is
 * restated from the pages' text, in the pages' order.
 *
 * Page short names used in citations:
 *   [1F1B]      "2. 1F1B"  (sgdbs.github.io, AI_Infra / 2.PipelineParallel / OneF1B)
 *   [GPipe->ZB] "Pipeline parallelism: from GPipe to 1F1B and Zero Bubble" (dlog.com.cn)
 *   [M040]      "Pipeline scheduling: GPipe, 1F1B, interleaving and overlap" (xuujii.github.io)
 *   [Megatron3] "Megatron-LM distributed training (3): pipeline parallel PP and 1F1B"
 *   [lpnh]      lpnh.cn news 2768528 (bubble formulas and 64xH100 table)
 *
 * What it computes, per schedule instance:
 *   1. the per-device op order from the schedule's rules (orc_order);
 *   2. every op's start/end tick with a discrete-event simulation on a global
 *      tick clock and a min-heap of events (orc_des), following the checker that
 *      [M040] §08 describes: each task waits for the previous task on its device
 *      and for the result it needs from the neighbouring stage;
 *   3. independently, the same times as a longest path over an explicit DAG in
 *      topological (Kahn) order (orc_longest_path) -- a cross-check of 2;
 *   4. makespan, busy/idle per device, the unreduced bubble pair and the peak
 *      count of held activations (ledger +1 at F, -1 at B);
 *   5. the validity checks [M040] §08 lists (no overlap on a device, every B
 *      has its F before it, gradients flow back, every device runs M*v F and
 *      M*v B).
 * Further schedules whose order depends on the costs, each simulated event by
 * event: Zero Bubble ZB1P / ZB2P (orc_zb_inst) and DualPipe's two routes
 * (orc_dp_inst); their readings are stated at their sections below.
 *
 * Readings taken where the pages are silent (each listed in the design notes):
 *   - GPipe backward order is last-in-first-out (D..A), from [M040] §02's table.
 *   - 1F1B stage k runs w = min(P-k, M) forwards, then (B, F) pairs taking the
 *     oldest B first, then the remaining B.  This is [1F1B] §2.3/§3.2's "P-k
 *     forwards" and equals [Megatron3]'s num_warmup = P-k-1 followed by the
 *     first steady F; both give F^w (B F)^(M-w) B^w.
 *   - Interleaved 1F1B: the op order is not printed on any page.  The oracle
 *     takes the Megatron interleaved order the pages point to ([1F1B] §6.1,
 *     [GPipe->ZB] Megatron section, [M040] §06): warmup 2(P-k-1)+(v-1)P
 *     forwards, then (F, B) pairs, then the remaining B; forward j maps to
 *     chunk (j mod Pv)/P and microbatch (j/(Pv))*P + j mod P, backward j to
 *     chunk v-1-(j mod Pv)/P with the same microbatch.  It needs M % P == 0
 *     ([M040] §06 divisibility note).
 *   - comm is a latency added on each cross-stage dependency edge; it occupies
 *     neither device.  comm[b] is the edge between virtual stages b and b+1.
 *   - All times are exact integers (int64 here).  An instance whose times do
 *     not fit in int32 is flagged ORC_ST_OVERFLOW; one with a negative cost or
 *     comm is flagged ORC_ST_NEG_COST.
 */
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#include <pthread.h>

#define ORC_GPIPE 0
#define ORC_1F1B 1
#define ORC_INTERLEAVED 2
#define ORC_GPIPE_FIFO 5

#define ORC_F 0
#define ORC_B 1

/* call-level return codes (numeric values follow the library's documented spec) */
#define ORC_OK 0
#define ORC_ERR_ARG 1
#define ORC_ERR_DIVISIBILITY 2
#define ORC_ERR_DEADLOCK 5
#define ORC_ERR_INVARIANT 6
#define ORC_ERR_NOMEM 7

/* per-instance status codes */
#define ORC_ST_OK 0
#define ORC_ST_NEG_COST 1
#define ORC_ST_OVERFLOW 2

#define ORC_INT32_MAX 2147483647LL

/* ORC_MUTANT plants one deliberate mistake (tests only: they compile mutant
 * copies to show that the pins catch plausible errors).  0 = the oracle. */
#ifndef ORC_MUTANT
#define ORC_MUTANT 0
#endif

/* ------------------------------------------------------------------------- */
/* 1. op order                                                               */
/* ------------------------------------------------------------------------- */

/* Fill the op order of device k: kind[j] (ORC_F / ORC_B), chunk[j], mb[j] for
 * j < 2*M*v.  Returns the op count, or a negative ORC_ERR_* code. */
int orc_order(int policy, int P, int M, int v, int k, int *kind, int *chunk, int *mb)
{
    int n = 0;
    if (P < 1 || M < 1 || v < 1 || k < 0 || k >= P) return -ORC_ERR_ARG;
    if (policy == ORC_GPIPE) {
        /* [M040] §02 table: all forwards A..D, then backwards D..A. */
        if (v != 1) return -ORC_ERR_ARG;
        for (int i = 0; i < M; ++i) { kind[n] = ORC_F; chunk[n] = 0; mb[n] = i; ++n; }
#if ORC_MUTANT == 3   /* mistake: first-in-first-out backward order */
        for (int i = 0; i < M; ++i) { kind[n] = ORC_B; chunk[n] = 0; mb[n] = i; ++n; }
#else
        for (int i = M - 1; i >= 0; --i) { kind[n] = ORC_B; chunk[n] = 0; mb[n] = i; ++n; }
#endif
        return n;
    }
    if (policy == ORC_GPIPE_FIFO) {
        /* the first-in-first-out variant of [M040] §02: backwards A..D */
        if (v != 1) return -ORC_ERR_ARG;
        for (int i = 0; i < M; ++i) { kind[n] = ORC_F; chunk[n] = 0; mb[n] = i; ++n; }
        for (int i = 0; i < M; ++i) { kind[n] = ORC_B; chunk[n] = 0; mb[n] = i; ++n; }
        return n;
    }
    if (policy == ORC_1F1B) {
        /* [1F1B] §2.3 / §3.2 table: warmup of P-k forwards, steady F-B pairs,
         * cooldown of the remaining B; the steady B is the oldest outstanding
         * microbatch ([Megatron3] "pop(0)").  Clamped to M when M < P-k. */
        if (v != 1) return -ORC_ERR_ARG;
        int w = P - k;
#if ORC_MUTANT == 2   /* mistake: Megatron's warmup count taken as the F count */
        w = P - k - 1;
#endif
        if (w > M) w = M;
        for (int i = 0; i < w; ++i) { kind[n] = ORC_F; chunk[n] = 0; mb[n] = i; ++n; }
        for (int q = 0; q < M - w; ++q) {
            kind[n] = ORC_B; chunk[n] = 0; mb[n] = q; ++n;
            kind[n] = ORC_F; chunk[n] = 0; mb[n] = w + q; ++n;
        }
        for (int i = M - w; i < M; ++i) { kind[n] = ORC_B; chunk[n] = 0; mb[n] = i; ++n; }
        return n;
    }
    if (policy == ORC_INTERLEAVED) {
        /* Device k holds virtual stages k, k+P, ... ([1F1B] §6.1; [M040] §06). */
        if (M % P != 0) return -ORC_ERR_DIVISIBILITY;
        int total = M * v;
        int w = 2 * (P - k - 1) + (v - 1) * P;
#if ORC_MUTANT == 13  /* mistake: one forward too many in the interleaved warmup */
        w += 1;
#endif
        if (w > total) w = total;
        int group = P * v;
        /* forward virtual index j */
#define FWD(j) do { int jj_ = (j); kind[n] = ORC_F; \
                    chunk[n] = (jj_ % group) / P; \
                    mb[n] = (jj_ / group) * P + jj_ % P; ++n; } while (0)
#define BWD(j) do { int jj_ = (j); kind[n] = ORC_B; \
                    chunk[n] = v - 1 - (jj_ % group) / P; \
                    mb[n] = (jj_ / group) * P + jj_ % P; ++n; } while (0)
        for (int j = 0; j < w; ++j) FWD(j);
        for (int i = 0; i < total - w; ++i) { FWD(w + i); BWD(i); }
        for (int i = total - w; i < total; ++i) BWD(i);
#undef FWD
#undef BWD
        return n;
    }
    return -ORC_ERR_ARG;
}

/* ------------------------------------------------------------------------- */
/* problem description shared by both evaluators                             */
/* ------------------------------------------------------------------------- */

typedef struct {
    int P, M, v, S, O;          /* devices, microbatches, chunks, virtual stages, ops per device */
    const int *kind, *chunk, *mb;   /* [P][O] op order */
    const int64_t *tf, *tb;     /* [S][M] costs of this instance */
    const int64_t *comm;        /* [S-1] edge latency (may be NULL: all 0) */
    const int64_t *comm_b;      /* [S-1] latency of backward edges, NULL: the same as comm */
} orc_inst;

static int64_t op_cost(const orc_inst *in, int dev, int j)
{
    int s = in->chunk[dev * in->O + j] * in->P + dev;
    int i = in->mb[dev * in->O + j];
    return in->kind[dev * in->O + j] == ORC_F ? in->tf[(int64_t)s * in->M + i]
                                              : in->tb[(int64_t)s * in->M + i];
}

static int64_t edge_comm(const orc_inst *in, int b)
{
    return in->comm ? in->comm[b] : 0;
}

/* Backward edges may have their own latency ([M040] §05: a forward boundary
 * carries the hidden activations, a backward one the activation gradients). */
static int64_t edge_comm_b(const orc_inst *in, int b)
{
#if ORC_MUTANT == 12  /* mistake: backward edges take the forward latency */
    return edge_comm(in, b);
#endif
    return in->comm_b ? in->comm_b[b] : edge_comm(in, b);
}

/* Locate every op (kind, s, i): pos[(kind*S + s)*M + i] = dev*O + j, or -1.
 * Returns 0, or ORC_ERR_INVARIANT if an op is missing, repeated or misplaced. */
static int build_pos(const orc_inst *in, int *pos)
{
    int S = in->S, M = in->M, P = in->P, O = in->O;
    for (int64_t x = 0; x < 2LL * S * M; ++x) pos[x] = -1;
    for (int d = 0; d < P; ++d) {
        for (int j = 0; j < O; ++j) {
            int kd = in->kind[d * O + j], c = in->chunk[d * O + j], i = in->mb[d * O + j];
            if ((kd != ORC_F && kd != ORC_B) || c < 0 || c >= in->v || i < 0 || i >= M)
                return ORC_ERR_INVARIANT;
            int s = c * P + d;
            int64_t key = ((int64_t)kd * S + s) * M + i;
            if (pos[key] != -1) return ORC_ERR_INVARIANT;   /* repeated op */
            pos[key] = d * O + j;
        }
    }
    for (int64_t x = 0; x < 2LL * S * M; ++x)
        if (pos[x] == -1) return ORC_ERR_INVARIANT;          /* missing op */
    return ORC_OK;
}

/* The dependencies of op (dev, j) from the pages' dependency model:
 *   F(s,i) needs F(s-1,i) (arrives comm[s-1] after it ends)  -- forward flows down;
 *   B(s,i) needs B(s+1,i) (arrives comm[s] after it ends)    -- gradient flows back;
 *   B(s,i) needs F(s,i) on its own device (no comm)           -- [GPipe->ZB] GPipe
 *   figure text: the backward needs the upper layer's B and the same layer's F;
 *   [M040] §01.  Writes up to 2 (op index, latency) pairs; returns the count. */
static int deps_of(const orc_inst *in, const int *pos, int dev, int j, int *dop, int64_t *dlat)
{
    int S = in->S, M = in->M, O = in->O;
    int kd = in->kind[dev * O + j], i = in->mb[dev * O + j];
    int s = in->chunk[dev * O + j] * in->P + dev;
    int nd = 0;
    if (kd == ORC_F) {
#if ORC_MUTANT == 1   /* mistake: forward edges carry no comm */
        if (s > 0) { dop[nd] = pos[((int64_t)ORC_F * S + (s - 1)) * M + i]; dlat[nd] = 0; ++nd; }
#else
        if (s > 0) { dop[nd] = pos[((int64_t)ORC_F * S + (s - 1)) * M + i]; dlat[nd] = edge_comm(in, s - 1); ++nd; }
#endif
    } else {
#if ORC_MUTANT != 4   /* mutant 4's mistake: B ignores the downstream gradient */
        if (s < S - 1) { dop[nd] = pos[((int64_t)ORC_B * S + (s + 1)) * M + i]; dlat[nd] = edge_comm_b(in, s); ++nd; }
#endif
        dop[nd] = pos[((int64_t)ORC_F * S + s) * M + i]; dlat[nd] = 0; ++nd;
    }
    return nd;
}

/* ------------------------------------------------------------------------- */
/* 2. discrete-event simulation                                              */
/* ------------------------------------------------------------------------- */

typedef struct { int64_t t; int64_t seq; int dev; int type; } orc_event;   /* type 0: op end, 1: wake */

typedef struct { orc_event *a; int64_t n, cap; } orc_heap;

static int ev_less(const orc_event *x, const orc_event *y)
{
    return x->t < y->t || (x->t == y->t && x->seq < y->seq);
}

static int heap_push(orc_heap *h, orc_event e)
{
    if (h->n == h->cap) {
        int64_t nc = h->cap ? 2 * h->cap : 64;
        orc_event *na = (orc_event *)realloc(h->a, (size_t)nc * sizeof(orc_event));
        if (!na) return ORC_ERR_NOMEM;
        h->a = na; h->cap = nc;
    }
    int64_t c = h->n++;
    h->a[c] = e;
    while (c > 0) {
        int64_t p = (c - 1) / 2;
        if (!ev_less(&h->a[c], &h->a[p])) break;
        orc_event t = h->a[c]; h->a[c] = h->a[p]; h->a[p] = t; c = p;
    }
    return ORC_OK;
}

static orc_event heap_pop(orc_heap *h)
{
    orc_event top = h->a[0];
    h->a[0] = h->a[--h->n];
    int64_t c = 0;
    for (;;) {
        int64_t l = 2 * c + 1, r = l + 1, m = c;
        if (l < h->n && ev_less(&h->a[l], &h->a[m])) m = l;
        if (r < h->n && ev_less(&h->a[r], &h->a[m])) m = r;
        if (m == c) break;
        orc_event t = h->a[c]; h->a[c] = h->a[m]; h->a[m] = t; c = m;
    }
    return top;
}

/* Simulate one instance.  start/end are [P][O].  Every device is free at tick
 * 0 and every microbatch input is ready at tick 0 ([1F1B] §5.2: stage 0 loads
 * microbatch i itself).  Ops are non-preemptive.  At each event time the
 * simulator first retires every event due at that time, then lets each idle
 * device start its next op if all its inputs have arrived; an input that is
 * done but still in flight schedules a wake-up at its arrival tick.
 * Returns ORC_OK or ORC_ERR_DEADLOCK (no event left while ops remain). */
int orc_des_inst(const orc_inst *in, const int *pos, int64_t *start, int64_t *end)
{
    int P = in->P, O = in->O;
    int total = P * O, finished = 0;
    int *cursor = (int *)calloc((size_t)P, sizeof(int));
    int *running = (int *)calloc((size_t)P, sizeof(int));
    unsigned char *done = (unsigned char *)calloc((size_t)total, 1);
    orc_heap h = {0, 0, 0};
    int64_t seq = 0, now = 0;
    int rc = ORC_OK;
    if (!cursor || !running || !done) { rc = ORC_ERR_NOMEM; goto out; }

    for (;;) {
        /* try to start an op on every idle device at time `now` */
        for (int d = 0; d < P; ++d) {
            if (running[d] || cursor[d] >= O) continue;
            int j = cursor[d];
            int dop[2]; int64_t dlat[2];
            int nd = deps_of(in, pos, d, j, dop, dlat);
            int ready = 1; int64_t arrive = 0;
            for (int x = 0; x < nd; ++x) {
                if (!done[dop[x]]) { ready = 0; break; }
                int64_t a = end[dop[x]] + dlat[x];
                if (a > arrive) arrive = a;
            }
            if (!ready) continue;               /* retried when the input's op ends */
            if (arrive > now) {                 /* input still on the wire */
                orc_event e = { arrive, seq++, d, 1 };
                if (heap_push(&h, e)) { rc = ORC_ERR_NOMEM; goto out; }
                continue;
            }
            int64_t c = op_cost(in, d, j);
            start[d * O + j] = now;
            end[d * O + j] = now + c;
            running[d] = 1;
            orc_event e = { now + c, seq++, d, 0 };
            if (heap_push(&h, e)) { rc = ORC_ERR_NOMEM; goto out; }
        }
        if (finished == total) break;
        if (h.n == 0) { rc = ORC_ERR_DEADLOCK; break; }
        /* advance the clock to the next event and retire everything due then */
        now = h.a[0].t;
        while (h.n > 0 && h.a[0].t == now) {
            orc_event e = heap_pop(&h);
            if (e.type == 0) {
                int d = e.dev;
                done[d * O + cursor[d]] = 1;
                cursor[d] += 1;
                running[d] = 0;
                finished += 1;
            }
        }
    }
out:
    free(cursor); free(running); free(done); free(h.a);
    return rc;
}

/* ------------------------------------------------------------------------- */
/* 3. independent cross-check: longest path over the explicit DAG            */
/* ------------------------------------------------------------------------- */

/* Build the DAG (device-order edges plus dependency edges weighted by comm),
 * order it with Kahn's algorithm and relax each node's start as the max over
 * its in-edges of (predecessor end + weight).  A node left unordered means a
 * cycle, i.e. the order deadlocks.  Returns ORC_OK or ORC_ERR_DEADLOCK. */
int orc_longest_path_inst(const orc_inst *in, const int *pos, int64_t *start, int64_t *end)
{
    int P = in->P, O = in->O, total = P * O;
    /* every node has at most 3 in-edges: previous op on its device + 2 deps */
    int *indeg = (int *)calloc((size_t)total, sizeof(int));
    int *succ = (int *)malloc((size_t)total * 3 * sizeof(int));
    int64_t *sw = (int64_t *)malloc((size_t)total * 3 * sizeof(int64_t));
    int *nsucc = (int *)calloc((size_t)total, sizeof(int));
    int *queue = (int *)malloc((size_t)total * sizeof(int));
    int rc = ORC_OK;
    if (!indeg || !succ || !sw || !nsucc || !queue) { rc = ORC_ERR_NOMEM; goto out; }
    for (int d = 0; d < P; ++d) {
        for (int j = 0; j < O; ++j) {
            int node = d * O + j;
            if (j > 0) {
                int pnode = node - 1;
                succ[pnode * 3 + nsucc[pnode]] = node; sw[pnode * 3 + nsucc[pnode]] = 0; nsucc[pnode]++;
                indeg[node]++;
            }
            int dop[2]; int64_t dlat[2];
            int nd = deps_of(in, pos, d, j, dop, dlat);
            for (int x = 0; x < nd; ++x) {
                int pnode = dop[x];
                if (nsucc[pnode] >= 3) { rc = ORC_ERR_INVARIANT; goto out; }
                succ[pnode * 3 + nsucc[pnode]] = node; sw[pnode * 3 + nsucc[pnode]] = dlat[x]; nsucc[pnode]++;
                indeg[node]++;
            }
        }
    }
    for (int x = 0; x < total; ++x) start[x] = 0;
    int qh = 0, qt = 0;
    for (int x = 0; x < total; ++x) if (indeg[x] == 0) queue[qt++] = x;
    while (qh < qt) {
        int u = queue[qh++];
        int d = u / O, j = u % O;
        end[u] = start[u] + op_cost(in, d, j);
        for (int e = 0; e < nsucc[u]; ++e) {
            int w = succ[u * 3 + e];
            int64_t cand = end[u] + sw[u * 3 + e];
            if (cand > start[w]) start[w] = cand;
            if (--indeg[w] == 0) queue[qt++] = w;
        }
    }
    if (qt != total) rc = ORC_ERR_DEADLOCK;
out:
    free(indeg); free(succ); free(sw); free(nsucc); free(queue);
    return rc;
}

/* ------------------------------------------------------------------------- */
/* 4./5. reductions and validity checks                                      */
/* ------------------------------------------------------------------------- */

/* The ledger of held activations ([1F1B] §4.1 table; [M040] §02/§03): +1 when
 * a forward finishes on the device, -1 when its backward releases it, counted
 * in op order; peak = running maximum.  Writes peak[P]. */
void orc_peak(int P, int O, const int *kind, int *peak)
{
    for (int d = 0; d < P; ++d) {
        int held = 0, pk = 0;
        for (int j = 0; j < O; ++j) {
#if ORC_MUTANT == 5   /* mistake: ledger releases on F and holds on B */
            held += kind[d * O + j] == ORC_F ? -1 : 1;
#else
            held += kind[d * O + j] == ORC_F ? 1 : -1;
#endif
            if (held > pk) pk = held;
        }
        peak[d] = pk;
    }
}

/* Validity checks of [M040] §08: no two ops overlap on a device; every B has
 * its F on the same device before it; every input arrives before the op that
 * uses it starts; each device runs exactly M*v F and M*v B.  Returns ORC_OK or
 * ORC_ERR_INVARIANT. */
static int check_inst(const orc_inst *in, const int *pos, const int64_t *start, const int64_t *end)
{
    int P = in->P, O = in->O;
    for (int d = 0; d < P; ++d) {
        int nf = 0, nb = 0;
        for (int j = 0; j < O; ++j) {
            int node = d * O + j;
            if (start[node] < 0 || end[node] != start[node] + op_cost(in, d, j)) return ORC_ERR_INVARIANT;
            if (j > 0 && start[node] < end[node - 1]) return ORC_ERR_INVARIANT;
            if (in->kind[node] == ORC_F) nf++; else nb++;
            int dop[2]; int64_t dlat[2];
            int nd = deps_of(in, pos, d, j, dop, dlat);
            for (int x = 0; x < nd; ++x)
                if (end[dop[x]] + dlat[x] > start[node]) return ORC_ERR_INVARIANT;
            if (in->kind[node] == ORC_B) {
                int fnode = dop[nd - 1];        /* F(s,i): same device, earlier */
                if (fnode / O != d || fnode % O >= j) return ORC_ERR_INVARIANT;
            }
        }
        if (nf != in->M * in->v || nb != in->M * in->v) return ORC_ERR_INVARIANT;
    }
    return ORC_OK;
}

/* ------------------------------------------------------------------------- */
/* single-instance entry point (int64 everything; used by tests)              */
/* ------------------------------------------------------------------------- */

/* Evaluate one instance with an explicit op order (kind/chunk/mb [P][O]).
 * method 0: discrete-event simulation; 1: longest path; 2: both, and compare.
 * Outputs: start/end [P][O], makespan, busy[P], idle[P], bub (num, den), peak[P].
 * Returns ORC_OK, ORC_ERR_DEADLOCK, ORC_ERR_INVARIANT or ORC_ERR_NOMEM. */
int orc_eval_explicit_fb(int P, int M, int v, const int *kind, const int *chunk, const int *mb,
                         const int64_t *tf, const int64_t *tb, const int64_t *comm, const int64_t *comm_b,
                         int method, int64_t *start, int64_t *end, int64_t *makespan, int64_t *busy,
                         int64_t *idle, int64_t *bub, int *peak);

int orc_eval_explicit(int P, int M, int v, const int *kind, const int *chunk, const int *mb,
                      const int64_t *tf, const int64_t *tb, const int64_t *comm, int method,
                      int64_t *start, int64_t *end, int64_t *makespan, int64_t *busy,
                      int64_t *idle, int64_t *bub, int *peak)
{
    return orc_eval_explicit_fb(P, M, v, kind, chunk, mb, tf, tb, comm, NULL, method, start, end, makespan,
                                busy, idle, bub, peak);
}

/* As orc_eval_explicit, with a separate latency comm_b [S-1] on the backward
 * edges (NULL: the same as comm). */
int orc_eval_explicit_fb(int P, int M, int v, const int *kind, const int *chunk, const int *mb,
                         const int64_t *tf, const int64_t *tb, const int64_t *comm, const int64_t *comm_b,
                         int method, int64_t *start, int64_t *end, int64_t *makespan, int64_t *busy,
                         int64_t *idle, int64_t *bub, int *peak)
{
    if (P < 1 || M < 1 || v < 1) return ORC_ERR_ARG;
    orc_inst in = { P, M, v, P * v, 2 * M * v, kind, chunk, mb, tf, tb, comm, comm_b };
    int total = P * in.O;
    int *pos = (int *)malloc((size_t)2 * in.S * M * sizeof(int));
    int64_t *s2 = (int64_t *)malloc((size_t)total * sizeof(int64_t));
    int64_t *e2 = (int64_t *)malloc((size_t)total * sizeof(int64_t));
    int rc;
    if (!pos || !s2 || !e2) { rc = ORC_ERR_NOMEM; goto out; }
    rc = build_pos(&in, pos);
    if (rc) goto out;
    if (method == 1) rc = orc_longest_path_inst(&in, pos, start, end);
    else rc = orc_des_inst(&in, pos, start, end);
    if (rc) goto out;
    if (method == 2) {
        rc = orc_longest_path_inst(&in, pos, s2, e2);
        if (rc) goto out;
        for (int x = 0; x < total; ++x)
            if (s2[x] != start[x] || e2[x] != end[x]) { rc = ORC_ERR_INVARIANT; goto out; }
    }
    rc = check_inst(&in, pos, start, end);
    if (rc) goto out;
    /* [M040] §04: window time, busy time per stage, bubble = idle / window;
     * [1F1B] §4.3: bubble ratio = total idle over P * total time. */
    int64_t mk = 0;
    for (int x = 0; x < total; ++x) if (end[x] > mk) mk = end[x];
    int64_t num = 0;
    for (int d = 0; d < P; ++d) {
        int64_t b = 0;
        for (int j = 0; j < in.O; ++j) b += op_cost(&in, d, j);
        busy[d] = b;
        idle[d] = mk - b;
        num += mk - b;
    }
    *makespan = mk;
    bub[0] = num;
    bub[1] = (int64_t)P * mk;
#if ORC_MUTANT == 6   /* mistake: bubble over ideal time instead of over the window */
    bub[1] = (int64_t)P * mk - num;
#endif
    orc_peak(P, in.O, kind, peak);
out:
    free(pos); free(s2); free(e2);
    return rc;
}

/* ------------------------------------------------------------------------- */
/* batch entry point (int32 inputs with strides, as the library takes them)   */
/* ------------------------------------------------------------------------- */

typedef struct {
    int policy, P, M, v;
    int64_t n;
    const int32_t *cost_f, *cost_b;
    int64_t cs_inst, cs_stage, cs_mb;
    const int32_t *comm, *comm_b;
    int64_t ms_inst, ms_bnd;
    int64_t *makespan, *idle, *bub_num, *bub_den;   /* idle [n][P] */
    int8_t *status;
    int64_t *op_start, *op_end;                      /* [n][P][O] or NULL */
    int method;
    const int *kind, *chunk, *mb;
    int64_t lo, hi;
    int rc;
} orc_batch_job;

static void *batch_worker(void *arg)
{
    orc_batch_job *jb = (orc_batch_job *)arg;
    int P = jb->P, M = jb->M, v = jb->v, S = P * v, O = 2 * M * v;
    int64_t *tf = (int64_t *)malloc((size_t)S * M * sizeof(int64_t));
    int64_t *tb = (int64_t *)malloc((size_t)S * M * sizeof(int64_t));
    int64_t *cm = (int64_t *)malloc((size_t)(S > 1 ? S - 1 : 1) * sizeof(int64_t));
    int64_t *cmb = (int64_t *)malloc((size_t)(S > 1 ? S - 1 : 1) * sizeof(int64_t));
    int64_t *st = (int64_t *)malloc((size_t)P * O * sizeof(int64_t));
    int64_t *en = (int64_t *)malloc((size_t)P * O * sizeof(int64_t));
    int64_t *busy = (int64_t *)malloc((size_t)P * sizeof(int64_t));
    int64_t *idle = (int64_t *)malloc((size_t)P * sizeof(int64_t));
    int *peak = (int *)malloc((size_t)P * sizeof(int));
    jb->rc = ORC_OK;
    if (!tf || !tb || !cm || !cmb || !st || !en || !busy || !idle || !peak) { jb->rc = ORC_ERR_NOMEM; goto out; }
    for (int64_t x = jb->lo; x < jb->hi; ++x) {
        int neg = 0;
        for (int s = 0; s < S; ++s)
            for (int i = 0; i < M; ++i) {
                int64_t off = x * jb->cs_inst + s * jb->cs_stage + i * jb->cs_mb;
                tf[s * M + i] = jb->cost_f[off];
                tb[s * M + i] = jb->cost_b[off];
                if (tf[s * M + i] < 0 || tb[s * M + i] < 0) neg = 1;
            }
        for (int b = 0; b < S - 1; ++b) {
            cm[b] = jb->comm ? jb->comm[x * jb->ms_inst + b * jb->ms_bnd] : 0;
            cmb[b] = jb->comm_b ? jb->comm_b[x * jb->ms_inst + b * jb->ms_bnd] : cm[b];
            if (cm[b] < 0 || cmb[b] < 0) neg = 1;
        }
        int64_t mk = 0, bub[2] = {0, 0};
        int rc = ORC_OK;
        if (!neg)
            rc = orc_eval_explicit_fb(P, M, v, jb->kind, jb->chunk, jb->mb, tf, tb, cm, cmb, jb->method,
                                      st, en, &mk, busy, idle, bub, peak);
        if (rc) { jb->rc = rc; goto out; }
        int8_t status = ORC_ST_OK;
        if (neg) status = ORC_ST_NEG_COST;
        else if (mk > ORC_INT32_MAX) status = ORC_ST_OVERFLOW;
        /* every time is <= makespan and every arrival is <= some start, so
         * makespan <= INT32_MAX means every intermediate fits in int32 */
        if (jb->status) jb->status[x] = status;
        jb->makespan[x] = neg ? 0 : mk;
        for (int d = 0; d < P; ++d) jb->idle[x * P + d] = neg ? 0 : idle[d];
        jb->bub_num[x] = bub[0];
        jb->bub_den[x] = bub[1];
        if (jb->op_start)
            for (int q = 0; q < P * O; ++q) {
                jb->op_start[x * P * O + q] = neg ? 0 : st[q];
                jb->op_end[x * P * O + q] = neg ? 0 : en[q];
            }
    }
out:
    free(tf); free(tb); free(cm); free(cmb); free(st); free(en); free(busy); free(idle); free(peak);
    return NULL;
}

/* Evaluate n instances of one policy/shape.  Costs are int32 [inst][stage][mb]
 * through element strides; comm is int32 [inst][boundary] through strides or
 * NULL (all zero).  Outputs are int64 (makespan[n], idle[n][P], bub_num[n],
 * bub_den[n]), int8 status[n], int32 peak[P], and optionally int64 op times
 * [n][P][O].  Instances are split statically over `nthreads` threads.
 * Returns ORC_OK or an ORC_ERR_* code. */
int orc_eval_batch_fb(int policy, int P, int M, int v, int64_t n,
                      const int32_t *cost_f, const int32_t *cost_b,
                      int64_t cs_inst, int64_t cs_stage, int64_t cs_mb,
                      const int32_t *comm, const int32_t *comm_b, int64_t ms_inst, int64_t ms_bnd,
                      int64_t *makespan, int64_t *idle, int64_t *bub_num, int64_t *bub_den,
                      int32_t *peak, int8_t *status, int64_t *op_start, int64_t *op_end,
                      int method, int nthreads);

int orc_eval_batch(int policy, int P, int M, int v, int64_t n,
                   const int32_t *cost_f, const int32_t *cost_b,
                   int64_t cs_inst, int64_t cs_stage, int64_t cs_mb,
                   const int32_t *comm, int64_t ms_inst, int64_t ms_bnd,
                   int64_t *makespan, int64_t *idle, int64_t *bub_num, int64_t *bub_den,
                   int32_t *peak, int8_t *status, int64_t *op_start, int64_t *op_end,
                   int method, int nthreads)
{
    return orc_eval_batch_fb(policy, P, M, v, n, cost_f, cost_b, cs_inst, cs_stage, cs_mb, comm, NULL, ms_inst,
                             ms_bnd, makespan, idle, bub_num, bub_den, peak, status, op_start, op_end, method,
                             nthreads);
}

/* As orc_eval_batch, with a separate latency comm_b on the backward edges
 * (same strides as comm; NULL: the same as comm). */
int orc_eval_batch_fb(int policy, int P, int M, int v, int64_t n,
                      const int32_t *cost_f, const int32_t *cost_b,
                      int64_t cs_inst, int64_t cs_stage, int64_t cs_mb,
                      const int32_t *comm, const int32_t *comm_b, int64_t ms_inst, int64_t ms_bnd,
                      int64_t *makespan, int64_t *idle, int64_t *bub_num, int64_t *bub_den,
                      int32_t *peak, int8_t *status, int64_t *op_start, int64_t *op_end,
                      int method, int nthreads)
{
    if (P < 1 || M < 1 || v < 1 || n < 0) return ORC_ERR_ARG;
    if (policy != ORC_INTERLEAVED && v != 1) return ORC_ERR_ARG;
    int O = 2 * M * v;
    int *kind = (int *)malloc((size_t)P * O * sizeof(int));
    int *chunk = (int *)malloc((size_t)P * O * sizeof(int));
    int *mbv = (int *)malloc((size_t)P * O * sizeof(int));
    int *pk = (int *)malloc((size_t)P * sizeof(int));
    int rc = ORC_OK;
    if (!kind || !chunk || !mbv || !pk) { rc = ORC_ERR_NOMEM; goto out; }
    for (int d = 0; d < P; ++d) {
        int got = orc_order(policy, P, M, v, d, kind + d * O, chunk + d * O, mbv + d * O);
        if (got < 0) { rc = -got; goto out; }
    }
    orc_peak(P, O, kind, pk);
    if (peak) for (int d = 0; d < P; ++d) peak[d] = pk[d];
    if (nthreads < 1) nthreads = 1;
    if (nthreads > 256) nthreads = 256;
    if ((int64_t)nthreads > n) nthreads = n > 0 ? (int)n : 1;
    orc_batch_job jobs[256];
    pthread_t th[256];
    for (int t = 0; t < nthreads; ++t) {
        orc_batch_job *jb = &jobs[t];
        jb->policy = policy; jb->P = P; jb->M = M; jb->v = v; jb->n = n;
        jb->cost_f = cost_f; jb->cost_b = cost_b;
        jb->cs_inst = cs_inst; jb->cs_stage = cs_stage; jb->cs_mb = cs_mb;
        jb->comm = comm; jb->comm_b = comm_b; jb->ms_inst = ms_inst; jb->ms_bnd = ms_bnd;
        jb->makespan = makespan; jb->idle = idle; jb->bub_num = bub_num; jb->bub_den = bub_den;
        jb->status = status; jb->op_start = op_start; jb->op_end = op_end;
        jb->method = method; jb->kind = kind; jb->chunk = chunk; jb->mb = mbv;
        jb->lo = n * t / nthreads; jb->hi = n * (t + 1) / nthreads;
        jb->rc = ORC_OK;
    }
    if (nthreads == 1) batch_worker(&jobs[0]);
    else {
        for (int t = 0; t < nthreads; ++t) pthread_create(&th[t], NULL, batch_worker, &jobs[t]);
        for (int t = 0; t < nthreads; ++t) pthread_join(th[t], NULL);
    }
    for (int t = 0; t < nthreads; ++t) if (jobs[t].rc) { rc = jobs[t].rc; break; }
out:
    free(kind); free(chunk); free(mbv); free(pk);
    return rc;
}

/* ------------------------------------------------------------------------- */
/* brute force over every valid order (tiny P, M)                             */
/* ------------------------------------------------------------------------- */

/* Enumerate, for every device, every order of F0..F(M-1), B0..B(M-1) in which
 * F_i precedes B_i (v = 1, unit costs, no comm), and run the simulator on every
 * combination.  Reports how many combinations deadlock or run, the minimum
 * makespan, how many orders reach it, and among those the minimum over orders
 * of the stage-0 peak and of the largest per-device peak.  This is the
 * exhaustive check behind [1F1B] §4.2 (no schedule that is not slower holds
 * fewer than P activations on stage 0) and §4.3 (total time 2(M+P-1)). */
int orc_bruteforce(int P, int M, int64_t *out /* [6] */)
{
    if (P < 1 || M < 1 || P > 4 || M > 4) return ORC_ERR_ARG;
    int O = 2 * M;
    {   /* refuse sizes whose enumeration would not finish quickly */
        double per = 1.0, comb = 1.0;
        for (int x = 2; x <= O; ++x) per *= x;
        for (int x = 0; x < M; ++x) per /= 2.0;
        for (int d = 0; d < P; ++d) comb *= per;
        if (comb > 2.0e7) return ORC_ERR_ARG;
    }
    /* list all single-device orders */
    int cap = 1;
    for (int x = 2; x <= O; ++x) cap *= x;          /* (2M)! upper bound */
    int *lists = (int *)malloc((size_t)cap * O * sizeof(int));   /* encoded op: kind*M + mb */
    int nl = 0;
    int perm[8];
    /* iterate over all permutations of 0..O-1 (op codes), keep the valid ones */
    for (int x = 0; x < O; ++x) perm[x] = x;
    for (;;) {
        int ok = 1;
        for (int i = 0; i < M && ok; ++i) {
            int pf = -1, pb = -1;
            for (int x = 0; x < O; ++x) { if (perm[x] == i) pf = x; if (perm[x] == M + i) pb = x; }
            if (pf > pb) ok = 0;
        }
        if (ok) { memcpy(lists + (size_t)nl * O, perm, (size_t)O * sizeof(int)); nl++; }
        /* next lexicographic permutation */
        int a = O - 2;
        while (a >= 0 && perm[a] > perm[a + 1]) a--;
        if (a < 0) break;
        int b = O - 1;
        while (perm[b] < perm[a]) b--;
        int t = perm[a]; perm[a] = perm[b]; perm[b] = t;
        for (int l = a + 1, r = O - 1; l < r; ++l, --r) { t = perm[l]; perm[l] = perm[r]; perm[r] = t; }
    }
    int *kind = (int *)malloc((size_t)P * O * sizeof(int));
    int *chunk = (int *)calloc((size_t)P * O, sizeof(int));
    int *mbv = (int *)malloc((size_t)P * O * sizeof(int));
    int64_t *tf = (int64_t *)malloc((size_t)P * M * sizeof(int64_t));
    int64_t *tb = (int64_t *)malloc((size_t)P * M * sizeof(int64_t));
    int64_t *cm = (int64_t *)calloc((size_t)P, sizeof(int64_t));
    int64_t *st = (int64_t *)malloc((size_t)P * O * sizeof(int64_t));
    int64_t *en = (int64_t *)malloc((size_t)P * O * sizeof(int64_t));
    int64_t busy[4], idle[4], bub[2], mk;
    int peak[4];
    for (int x = 0; x < P * M; ++x) { tf[x] = 1; tb[x] = 1; }
    int64_t nvalid = 0, ndead = 0, best = -1, nbest = 0, bestpk0 = -1, bestpkmax = -1;
    int idx[4] = {0, 0, 0, 0};
    for (;;) {
        for (int d = 0; d < P; ++d)
            for (int j = 0; j < O; ++j) {
                int code = lists[(size_t)idx[d] * O + j];
                kind[d * O + j] = code < M ? ORC_F : ORC_B;
                mbv[d * O + j] = code % M;
            }
        int rc = orc_eval_explicit(P, M, 1, kind, chunk, mbv, tf, tb, cm, 0, st, en, &mk, busy, idle, bub, peak);
        if (rc == ORC_ERR_DEADLOCK) ndead++;
        else if (rc == ORC_OK) {
            nvalid++;
            int pmax = 0;
            for (int d = 0; d < P; ++d) if (peak[d] > pmax) pmax = peak[d];
            if (best < 0 || mk < best) { best = mk; nbest = 0; bestpk0 = peak[0]; bestpkmax = pmax; }
            if (mk == best) {
                nbest++;
                if (peak[0] < bestpk0) bestpk0 = peak[0];
                if (pmax < bestpkmax) bestpkmax = pmax;
            }
        } else { free(lists); return rc; }
        int d = 0;
        while (d < P) { if (++idx[d] < nl) break; idx[d] = 0; d++; }
        if (d == P) break;
    }
    out[0] = nvalid; out[1] = ndead; out[2] = best; out[3] = nbest; out[4] = bestpk0; out[5] = bestpkmax;
    free(lists); free(kind); free(chunk); free(mbv); free(tf); free(tb); free(cm); free(st); free(en);
    return ORC_OK;
}

/* ------------------------------------------------------------------------- */
/* candidate partition search                                                 */
/* ------------------------------------------------------------------------- */

/* SplitMix64 (Steele, Lea & Flood, "Fast splittable pseudorandom number
 * generators", OOPSLA 2014; constants as in Vigna's public-domain
 * splitmix64.c): advance the state by the golden gamma, then mix. */
static uint64_t splitmix64_at(uint64_t state)
{
    uint64_t z = state + 0x9E3779B97F4A7C15ULL;
#if ORC_MUTANT == 7   /* mistake: one shift constant mistyped */
    z = (z ^ (z >> 31)) * 0xBF58476D1CE4E5B9ULL;
    z = (z ^ (z >> 27)) * 0x94D049BB133111EBULL;
    return z ^ (z >> 31);
#endif
    z = (z ^ (z >> 30)) * 0xBF58476D1CE4E5B9ULL;
    z = (z ^ (z >> 27)) * 0x94D049BB133111EBULL;
    return z ^ (z >> 31);
}

/* Binomial coefficient by Pascal's rule, exact in uint64 for n <= 1023, k <= 31
 * when it fits; returns UINT64_MAX on overflow. */
static uint64_t binom(int n, int k)
{
    if (k < 0 || n < 0 || k > n) return 0;
    if (k > n - k) k = n - k;
    uint64_t row[64];
    for (int j = 0; j <= k; ++j) row[j] = 0;
    row[0] = 1;
    for (int m = 1; m <= n; ++m) {
        int top = m < k ? m : k;
        for (int j = top; j >= 1; --j) {
            uint64_t s = row[j] + row[j - 1];
            if (s < row[j] || row[j] == UINT64_MAX || row[j - 1] == UINT64_MAX) s = UINT64_MAX;
            row[j] = s;
        }
    }
    return row[k];
}

/* Combinatorial number system (colex order): rank r in [0, C(N,K)) maps to
 * x_1 < ... < x_K in [0, N) with r = sum_i C(x_i, i); found greedily from i = K
 * down to 1 by taking the largest x with C(x, i) <= remaining rank. */
static void unrank_colex(uint64_t r, int N, int K, int *x)
{
    int hi = N - 1;
    for (int i = K; i >= 1; --i) {
        int c = hi;
        while (c >= i - 1 && binom(c, i) > r) c--;
#if ORC_MUTANT == 8   /* mistake: off-by-one in the greedy unranking */
        if (c > i - 1) c--;
#endif
        x[i - 1] = c;
        r -= binom(c, i);
        hi = c - 1;
    }
}

/* The split of colex rank r in [0, C(L-1, P-1)): the P-1 cut positions
 * x_1 < ... < x_{P-1} in [0, L-1) of rank r; stage t starts at layer x_t + 1
 * (stage 0 at layer 0).  Writes first[P+1], first[P] = L.  Ranks 0 .. C-1
 * enumerate every contiguous split once (the exhaustive search). */
void orc_rank_split(uint64_t r, int L, int P, int *first)
{
    int K = P - 1;
    int x[64];
    unrank_colex(r, L - 1, K, x);
    first[0] = 0;
    for (int t = 1; t <= K; ++t) first[t] = x[t - 1] + 1;
    first[P] = L;
}

/* Candidate c's contiguous split of L layers into P non-empty stages: draw
 * u = splitmix64(seed + c), rank = u mod C(L-1, P-1), unrank it to the P-1 cut
 * positions x_1 < ... < x_{P-1} in [0, L-1); stage t starts at layer
 * x_t + 1 (stage 0 at layer 0).  Writes first[P+1] (first layer of each stage,
 * first[P] = L).  This is the seeded candidate set standing in for the
 * profiling-based contiguous layer split ([GPipe->ZB] PipeDream/GPipe sections;
 * [M040] §05; [lpnh]: 80 layers into 8 stages). */
void orc_candidate_split(uint64_t seed, int64_t c, int L, int P, int *first)
{
    uint64_t total = binom(L - 1, P - 1);
    orc_rank_split((uint64_t)(splitmix64_at(seed + (uint64_t)c) % total), L, P, first);
}

typedef struct {
    const int32_t *ltf, *ltb; const int64_t *lact;
    int L, P, M, v; int32_t comm; int64_t cap; uint64_t seed;
    int64_t lo, hi;
    int32_t *all_mk;
    int64_t best_idx; int64_t best_mk;
    const int *kind, *chunk, *mb; const int *peak;
    int exhaustive;             /* candidate c is colex rank c instead of a seeded draw */
    int rc;
} orc_search_job;

static void *search_worker(void *arg)
{
    orc_search_job *jb = (orc_search_job *)arg;
    int P = jb->P, M = jb->M, v = jb->v, S = P * v, O = 2 * M * v;
    int first[65];
    int64_t *tf = (int64_t *)malloc((size_t)S * M * sizeof(int64_t));
    int64_t *tb = (int64_t *)malloc((size_t)S * M * sizeof(int64_t));
    int64_t *act = (int64_t *)malloc((size_t)S * sizeof(int64_t));
    int64_t *cm = (int64_t *)malloc((size_t)S * sizeof(int64_t));
    int64_t *st = (int64_t *)malloc((size_t)P * O * sizeof(int64_t));
    int64_t *en = (int64_t *)malloc((size_t)P * O * sizeof(int64_t));
    int64_t *busy = (int64_t *)malloc((size_t)P * sizeof(int64_t));
    int64_t *idle = (int64_t *)malloc((size_t)P * sizeof(int64_t));
    int *pk = (int *)malloc((size_t)P * sizeof(int));
    jb->best_idx = -1; jb->best_mk = -1; jb->rc = ORC_OK;
    for (int b = 0; b < S; ++b) cm[b] = jb->comm;
    for (int64_t c = jb->lo; c < jb->hi; ++c) {
        if (jb->exhaustive) orc_rank_split((uint64_t)c, jb->L, S, first);
        else orc_candidate_split(jb->seed, c, jb->L, S, first);
        for (int s = 0; s < S; ++s) {
            int64_t sf = 0, sb = 0, sa = 0;
            for (int l = first[s]; l < first[s + 1]; ++l) { sf += jb->ltf[l]; sb += jb->ltb[l]; sa += jb->lact[l]; }
            act[s] = sa;
            for (int i = 0; i < M; ++i) { tf[s * M + i] = sf; tb[s * M + i] = sb; }
        }
        /* peak bytes held on device d: the ledger of [1F1B] §4.1 weighted by
         * the bytes of the chunk each op belongs to (+ at F, - at B), at its
         * running maximum; with one chunk per device this is the peak count
         * times the stage's bytes */
        int rejected = 0;
        for (int d = 0; d < P && !rejected; ++d) {
            int64_t held = 0, top = 0;
            for (int j = 0; j < O; ++j) {
#if ORC_MUTANT == 18  /* mistake: every op weighted by the device's first chunk's bytes */
                int s = d;
#else
                int s = jb->chunk[d * O + j] * P + d;
#endif
                held += jb->kind[d * O + j] == ORC_F ? act[s] : -act[s];
                if (held > top) top = held;
            }
#if ORC_MUTANT == 16  /* mistake: a layout exactly at the cap is rejected */
            if (top >= jb->cap) rejected = 1;
#else
            if (top > jb->cap) rejected = 1;
#endif
        }
        int64_t mk = -1, bub[2];
        if (!rejected) {
            int rc = orc_eval_explicit(P, M, v, jb->kind, jb->chunk, jb->mb, tf, tb, cm, 0,
                                       st, en, &mk, busy, idle, bub, pk);
            if (rc) { jb->rc = rc; break; }
            if (mk > ORC_INT32_MAX) mk = -2;
        }
        if (jb->all_mk) jb->all_mk[c - jb->lo] = (int32_t)mk;
#if ORC_MUTANT == 17  /* mistake: a tie goes to the later candidate */
        if (mk >= 0 && (jb->best_idx < 0 || mk <= jb->best_mk)) { jb->best_mk = mk; jb->best_idx = c; }
#else
        if (mk >= 0 && (jb->best_idx < 0 || mk < jb->best_mk)) { jb->best_mk = mk; jb->best_idx = c; }
#endif
    }
    free(tf); free(tb); free(act); free(cm); free(st); free(en); free(busy); free(idle); free(pk);
    return NULL;
}

/* Score candidates c in [c_lo, c_hi) under 1F1B with M microbatches: stage k's
 * forward cost is the sum of its layers' forward costs, its backward cost the
 * sum of the layers' backward costs, comm the same on every boundary; a
 * candidate is rejected when some stage's peak held activations times its
 * activation bytes exceeds `cap`.  all_mk[c - c_lo] gets the makespan, -1 if
 * rejected, -2 if it overflows int32.  best = argmin (makespan, index) over the
 * range; best_idx = -1 when nothing is feasible.  first_best[P+1] gets the
 * winner's stage starts.  Returns ORC_OK or an ORC_ERR_* code. */
static int search_impl(const int32_t *layer_tf, const int32_t *layer_tb, const int64_t *layer_act,
                       int L, int P, int v, int M, int32_t comm, int64_t cap, uint64_t seed, int exhaustive,
                       int64_t c_lo, int64_t c_hi, int32_t *all_mk,
                       int64_t *best_idx, int64_t *best_mk, int *first_best, int nthreads)
{
    int S = P * v;
    if (P < 1 || v < 1 || S > 64 || L < S || M < 1 || c_lo < 0 || c_hi < c_lo) return ORC_ERR_ARG;
    if (v > 1 && M % P != 0) return ORC_ERR_DIVISIBILITY;
    if (binom(L - 1, S - 1) == UINT64_MAX) return ORC_ERR_ARG;
    if (exhaustive && (uint64_t)c_hi > binom(L - 1, S - 1)) return ORC_ERR_ARG;
    int O = 2 * M * v;
    int *kind = (int *)malloc((size_t)P * O * sizeof(int));
    int *chunk = (int *)malloc((size_t)P * O * sizeof(int));
    int *mbv = (int *)malloc((size_t)P * O * sizeof(int));
    int *pk = (int *)malloc((size_t)P * sizeof(int));
    for (int d = 0; d < P; ++d)
        orc_order(v > 1 ? ORC_INTERLEAVED : ORC_1F1B, P, M, v, d, kind + d * O, chunk + d * O, mbv + d * O);
    orc_peak(P, O, kind, pk);
    if (nthreads < 1) nthreads = 1;
    if (nthreads > 256) nthreads = 256;
    int64_t n = c_hi - c_lo;
    if (nthreads > n) nthreads = n > 0 ? (int)n : 1;
    orc_search_job jobs[256];
    pthread_t th[256];
    for (int t = 0; t < nthreads; ++t) {
        orc_search_job *jb = &jobs[t];
        jb->ltf = layer_tf; jb->ltb = layer_tb; jb->lact = layer_act;
        jb->L = L; jb->P = P; jb->M = M; jb->v = v; jb->comm = comm; jb->cap = cap; jb->seed = seed;
        jb->lo = c_lo + n * t / nthreads; jb->hi = c_lo + n * (t + 1) / nthreads;
        jb->all_mk = all_mk ? all_mk + (jb->lo - c_lo) : NULL;
        jb->kind = kind; jb->chunk = chunk; jb->mb = mbv; jb->peak = pk;
        jb->exhaustive = exhaustive;
    }
    if (nthreads == 1) search_worker(&jobs[0]);
    else {
        for (int t = 0; t < nthreads; ++t) pthread_create(&th[t], NULL, search_worker, &jobs[t]);
        for (int t = 0; t < nthreads; ++t) pthread_join(th[t], NULL);
    }
    int rc = ORC_OK;
    *best_idx = -1; *best_mk = -1;
    for (int t = 0; t < nthreads; ++t) {        /* ranges ascend, so first strict min wins ties */
        if (jobs[t].rc) { rc = jobs[t].rc; break; }
        if (jobs[t].best_idx >= 0 && (*best_idx < 0 || jobs[t].best_mk < *best_mk)) {
            *best_idx = jobs[t].best_idx; *best_mk = jobs[t].best_mk;
        }
    }
    if (first_best) {
        if (*best_idx < 0) for (int t = 0; t <= S; ++t) first_best[t] = -1;
        else if (exhaustive) orc_rank_split((uint64_t)*best_idx, L, S, first_best);
        else orc_candidate_split(seed, *best_idx, L, S, first_best);
    }
    free(kind); free(chunk); free(mbv); free(pk);
    return rc;
}

int orc_search(const int32_t *layer_tf, const int32_t *layer_tb, const int64_t *layer_act,
               int L, int P, int M, int32_t comm, int64_t cap, uint64_t seed,
               int64_t c_lo, int64_t c_hi, int32_t *all_mk,
               int64_t *best_idx, int64_t *best_mk, int *first_best, int nthreads)
{
    return search_impl(layer_tf, layer_tb, layer_act, L, P, 1, M, comm, cap, seed, 0, c_lo, c_hi, all_mk,
                       best_idx, best_mk, first_best, nthreads);
}

/* The search over interleaved layouts ([M040] §06: a device holds several
 * virtual stages; §05: split by measured cost and activation): each candidate
 * splits the L layers into S = P*v contiguous non-empty ranges (seeded draw of
 * a colex rank of C(L-1, S-1)); range s is virtual stage s, chunk s / P of
 * device s mod P.  Scored under interleaved 1F1B with M microbatches (M % P ==
 * 0); rejected when a device's peak held bytes (the chunk-weighted ledger)
 * exceeds `cap`.  first_best gets S+1 range starts. */
int orc_search_interleaved(const int32_t *layer_tf, const int32_t *layer_tb, const int64_t *layer_act,
                           int L, int P, int v, int M, int32_t comm, int64_t cap, uint64_t seed,
                           int64_t c_lo, int64_t c_hi, int32_t *all_mk,
                           int64_t *best_idx, int64_t *best_mk, int *first_best, int nthreads)
{
    return search_impl(layer_tf, layer_tb, layer_act, L, P, v, M, comm, cap, seed, 0, c_lo, c_hi, all_mk,
                       best_idx, best_mk, first_best, nthreads);
}

/* The exhaustive search ([lpnh]'s 80-layer split, every contiguous split):
 * as orc_search, but candidate c is the split of colex rank c, for ranks
 * [r_lo, r_hi) within [0, C(L-1, P-1)). */
int orc_search_ranks(const int32_t *layer_tf, const int32_t *layer_tb, const int64_t *layer_act,
                     int L, int P, int M, int32_t comm, int64_t cap,
                     int64_t r_lo, int64_t r_hi, int32_t *all_mk,
                     int64_t *best_idx, int64_t *best_mk, int *first_best, int nthreads)
{
    return search_impl(layer_tf, layer_tb, layer_act, L, P, 1, M, comm, cap, 0, 1, r_lo, r_hi, all_mk,
                       best_idx, best_mk, first_best, nthreads);
}

/* exposed for tests: C(n, k) and the raw generator, to pin them against
 * textbook values */
uint64_t orc_binom(int n, int k) { return binom(n, k); }
uint64_t orc_splitmix64(uint64_t state) { return splitmix64_at(state); }

/* ------------------------------------------------------------------------- */
/* Zero Bubble (ZB1P / ZB2P): the backward split into B and W                  */
/* ------------------------------------------------------------------------- */
/*
 * [GPipe->ZB] "Zero Bubble" and "ZB1P and ZB2P"; [1F1B] §6.2.  A microbatch's
 * backward splits into B (the input gradient, which the previous stage waits
 * for) and W (the weight gradient, needed only before the parameter update:
 * no cross-stage dependency).  W(s,i) runs on stage s's device after B(s,i).
 * The schedule keeps 1F1B's order of F and B and places W greedily: when the
 * next F or B cannot start because its input has not arrived, the device runs
 * a W that is ready instead; a device holds at most L microbatches whose F has
 * run and whose W has not, so an F that would exceed L waits for a W.
 *
 * Readings (the pages state the rules loosely; each is in the design notes):
 *   - F/B order: F^w (B F)^(M-w) B^w as in 1F1B, with w = min(P-k, M) for
 *     ZB1P and w = min(2(P-k), M) for ZB2P (more forwards in the warmup, about
 *     twice the activation budget).
 *   - L = P for ZB1P and 2P for ZB2P, on every device.
 *   - A device that becomes free at tick t decides:
 *       1. if its next F/B op X is an F and it holds L microbatches, it runs
 *          the oldest pending W;
 *       2. else if X's input has arrived by t, it runs X at t;
 *       3. else if a W is pending, it runs the oldest pending W at t;
 *       4. else it waits and runs X when X's input arrives.
 *     With no F/B op left it runs its pending W's, oldest first.
 *   - Pending W's run in the order of their B's.
 *   - Every F and B cost is at least 1 tick (a W may take 0).  Then whether
 *     an input has arrived by t depends on the costs alone, not on the order
 *     in which simultaneous decisions are taken: an F or B placed at t or
 *     later cannot end by t, and a W feeds no other device.  An instance with
 *     an F or B cost below 1 is flagged ORC_ST_ZERO_COST.
 *   - comm is the latency on F and B edges as in the other schedules; W has
 *     no cross-stage edge.
 *   - Held activations: +1 at F, -1 at W (a microbatch's saved data is
 *     released when its W is done); the peak is over the device's op order.
 * Op times are laid out [P][3][M]: device, kind (F, B, W), microbatch.
 */
#define ORC_ZB1P 3
#define ORC_ZB2P 4
#define ORC_W 2
#define ORC_ST_ZERO_COST 3

static int zb_warmup(int policy, int P, int M, int k)
{
    int w = policy == ORC_ZB2P ? 2 * (P - k) : P - k;
#if ORC_MUTANT == 10  /* mistake: ZB2P keeps 1F1B's warmup */
    w = P - k;
#endif
    return w < M ? w : M;
}

typedef struct {
    int P, M, L;
    const int64_t *tf, *tb, *tw, *comm;   /* costs [P][M], comm [P-1] or NULL */
    int *kind, *mb;                       /* F/B order [P][2M] */
    int *pos, *nf, *nb, *nw, *held, *state, *border;   /* border [P][M]: mb of the i-th B */
    int64_t *t_free;
    int64_t *start, *end;                 /* [P][3][M] */
    int64_t *busy;
    int *peak;
} zb_sim;

#define ZB_AT(z, k, kd, m) ((((k) * 3) + (kd)) * (z)->M + (m))

/* Arrival tick of the input of F/B op (kd, m) on device k: 0 without an input
 * edge, -1 while its producer is not placed. */
static int64_t zb_arrival(const zb_sim *z, int k, int kd, int m)
{
    if (kd == ORC_F) {
        if (k == 0) return 0;
        int64_t e = z->end[ZB_AT(z, k - 1, ORC_F, m)];
        return e < 0 ? -1 : e + (z->comm ? z->comm[k - 1] : 0);
    }
    /* B(k,m) also needs F(k,m), which precedes it on the same device */
    if (k == z->P - 1) return z->end[ZB_AT(z, k, ORC_F, m)];
    int64_t e = z->end[ZB_AT(z, k + 1, ORC_B, m)];
    return e < 0 ? -1 : e + (z->comm ? z->comm[k] : 0);
}

static void zb_place(zb_sim *z, int k, int kd, int m, int64_t s)
{
    int64_t c = kd == ORC_F ? z->tf[k * z->M + m] : (kd == ORC_B ? z->tb[k * z->M + m] : z->tw[k * z->M + m]);
    z->start[ZB_AT(z, k, kd, m)] = s;
    z->end[ZB_AT(z, k, kd, m)] = s + c;
    z->t_free[k] = s + c;
    z->busy[k] += c;
    if (kd == ORC_F) {
        z->nf[k]++;
        z->held[k]++;
        if (z->held[k] > z->peak[k]) z->peak[k] = z->held[k];
    } else if (kd == ORC_B) {
        z->border[k * z->M + z->nb[k]] = m;
        z->nb[k]++;
    } else {
        z->nw[k]++;
        z->held[k]--;
    }
    if (kd != ORC_W) z->pos[k]++;
}

static void zb_place_w(zb_sim *z, int k, int64_t s)
{
    zb_place(z, k, ORC_W, z->border[k * z->M + z->nw[k]], s);
}

/* A waiting device runs its next F/B op once the op's input is placed. */
static void zb_wake(zb_sim *z)
{
    int again = 1;
    while (again) {
        again = 0;
        for (int d = 0; d < z->P; ++d) {
            if (z->state[d] != 1) continue;
            int j = d * 2 * z->M + z->pos[d];
            int64_t arr = zb_arrival(z, d, z->kind[j], z->mb[j]);
            if (arr < 0) continue;
            z->state[d] = 0;
            zb_place(z, d, z->kind[j], z->mb[j], arr > z->t_free[d] ? arr : z->t_free[d]);
            again = 1;
        }
    }
}

/* Validity of a finished ZB schedule: per device no overlap and end = start +
 * cost; F/B in their order; every input arrived before use; W after its B;
 * at most L held. */
static int zb_check(const zb_sim *z)
{
    int P = z->P, M = z->M;
    for (int k = 0; k < P; ++k) {
        if (z->peak[k] > z->L) return ORC_ERR_INVARIANT;
        /* no overlap: sort this device's 3M ops by (start, end) (insertion
         * sort; a W of zero cost sorts before an op starting at its tick) */
        int n = 3 * M;
        int *ix = (int *)malloc((size_t)n * sizeof(int));
        if (!ix) return ORC_ERR_NOMEM;
        for (int q = 0; q < n; ++q) ix[q] = k * n + q;
        for (int a = 1; a < n; ++a) {
            int v = ix[a], b = a - 1;
            while (b >= 0 && (z->start[ix[b]] > z->start[v] ||
                              (z->start[ix[b]] == z->start[v] && z->end[ix[b]] > z->end[v]))) {
                ix[b + 1] = ix[b];
                --b;
            }
            ix[b + 1] = v;
        }
        int bad = 0;
        for (int a = 0; a + 1 < n; ++a)
            if (z->end[ix[a]] > z->start[ix[a + 1]]) bad = 1;
        free(ix);
        if (bad) return ORC_ERR_INVARIANT;
        for (int j = 0; j + 1 < 2 * M; ++j) {
            int a = k * 2 * M + j;
            if (z->start[ZB_AT(z, k, z->kind[a], z->mb[a])] > z->start[ZB_AT(z, k, z->kind[a + 1], z->mb[a + 1])])
                return ORC_ERR_INVARIANT;
        }
        for (int m = 0; m < M; ++m) {
            int64_t c[3] = { z->tf[k * M + m], z->tb[k * M + m], z->tw[k * M + m] };
            for (int kd = 0; kd < 3; ++kd)
                if (z->start[ZB_AT(z, k, kd, m)] < 0 || z->end[ZB_AT(z, k, kd, m)] != z->start[ZB_AT(z, k, kd, m)] + c[kd])
                    return ORC_ERR_INVARIANT;
            if (k > 0 && z->start[ZB_AT(z, k, ORC_F, m)] < z->end[ZB_AT(z, k - 1, ORC_F, m)] + (z->comm ? z->comm[k - 1] : 0))
                return ORC_ERR_INVARIANT;
            if (z->start[ZB_AT(z, k, ORC_B, m)] < z->end[ZB_AT(z, k, ORC_F, m)]) return ORC_ERR_INVARIANT;
            if (k < P - 1 && z->start[ZB_AT(z, k, ORC_B, m)] < z->end[ZB_AT(z, k + 1, ORC_B, m)] + (z->comm ? z->comm[k] : 0))
                return ORC_ERR_INVARIANT;
            if (z->start[ZB_AT(z, k, ORC_W, m)] < z->end[ZB_AT(z, k, ORC_B, m)]) return ORC_ERR_INVARIANT;
        }
    }
    return ORC_OK;
}

/* One ZB instance.  tf/tb [P][M] (every cost >= 1), tw [P][M] (>= 0), comm
 * [P-1] or NULL.  Outputs: start/end [P][3][M], makespan, busy[P], idle[P],
 * bub (num, den), peak[P].  Returns ORC_OK, ORC_ERR_ARG (policy, shape or a
 * cost out of range),
 * ORC_ERR_DEADLOCK, ORC_ERR_INVARIANT or ORC_ERR_NOMEM. */
int orc_zb_inst(int policy, int P, int M, const int64_t *tf, const int64_t *tb, const int64_t *tw,
                const int64_t *comm, int64_t *start, int64_t *end, int64_t *makespan,
                int64_t *busy, int64_t *idle, int64_t *bub, int *peak)
{
    if ((policy != ORC_ZB1P && policy != ORC_ZB2P) || P < 1 || M < 1) return ORC_ERR_ARG;
    for (int q = 0; q < P * M; ++q)
        if (tf[q] < 1 || tb[q] < 1 || tw[q] < 0) return ORC_ERR_ARG;
    zb_sim z;
    memset(&z, 0, sizeof(z));
    z.P = P; z.M = M; z.L = policy == ORC_ZB1P ? P : 2 * P;
    z.tf = tf; z.tb = tb; z.tw = tw; z.comm = comm;
    z.start = start; z.end = end; z.busy = busy; z.peak = peak;
    int O = 2 * M, rc = ORC_OK;
    z.kind = (int *)malloc((size_t)P * O * sizeof(int));
    z.mb = (int *)malloc((size_t)P * O * sizeof(int));
    z.border = (int *)malloc((size_t)P * M * sizeof(int));
    z.pos = (int *)calloc((size_t)P, sizeof(int));
    z.nf = (int *)calloc((size_t)P, sizeof(int));
    z.nb = (int *)calloc((size_t)P, sizeof(int));
    z.nw = (int *)calloc((size_t)P, sizeof(int));
    z.held = (int *)calloc((size_t)P, sizeof(int));
    z.state = (int *)calloc((size_t)P, sizeof(int));
    z.t_free = (int64_t *)calloc((size_t)P, sizeof(int64_t));
    if (!z.kind || !z.mb || !z.border || !z.pos || !z.nf || !z.nb || !z.nw || !z.held || !z.state || !z.t_free) {
        rc = ORC_ERR_NOMEM;
        goto out;
    }
    for (int k = 0; k < P; ++k) {
        int w = zb_warmup(policy, P, M, k), n = 0, *kd = z.kind + k * O, *mb = z.mb + k * O;
        for (int i = 0; i < w; ++i) { kd[n] = ORC_F; mb[n] = i; ++n; }
        for (int q = 0; q < M - w; ++q) {
            kd[n] = ORC_B; mb[n] = q; ++n;
            kd[n] = ORC_F; mb[n] = w + q; ++n;
        }
        for (int i = M - w; i < M; ++i) { kd[n] = ORC_B; mb[n] = i; ++n; }
        busy[k] = 0;
        peak[k] = 0;
    }
    for (int q = 0; q < 3 * P * M; ++q) { start[q] = -1; end[q] = -1; }

    for (;;) {
        /* the free device with the smallest tick decides (then the lowest index) */
        int k = -1, waiting = 0, left = 0;
        for (int d = 0; d < P; ++d) {
            if (z.state[d] == 2) continue;
            left = 1;
            if (z.state[d] == 1) { waiting = 1; continue; }
            if (k < 0 || z.t_free[d] < z.t_free[k]) k = d;
        }
        if (!left) break;
        if (k < 0) { rc = waiting ? ORC_ERR_DEADLOCK : ORC_ERR_INVARIANT; goto out; }
        int64_t t = z.t_free[k];
        int pend = z.nw[k] < z.nb[k];
        if (z.pos[k] == O) {
            if (pend) zb_place_w(&z, k, t);
            else z.state[k] = 2;
            continue;
        }
        int j = k * O + z.pos[k];
        int xk = z.kind[j], xm = z.mb[j];
#if ORC_MUTANT == 11  /* mistake: an F is admitted with L microbatches already held */
        if (xk == ORC_F && z.nf[k] - z.nw[k] > z.L) {
#else
        if (xk == ORC_F && z.nf[k] - z.nw[k] >= z.L) {
#endif
            if (!pend) { rc = ORC_ERR_INVARIANT; goto out; }
            zb_place_w(&z, k, t);
            continue;
        }
        int64_t arr = zb_arrival(&z, k, xk, xm);
#if ORC_MUTANT == 9   /* mistake: a pending W goes before a ready F/B */
        if (pend) zb_place_w(&z, k, t);
        else if (arr >= 0 && arr <= t) zb_place(&z, k, xk, xm, t);
#else
        if (arr >= 0 && arr <= t) zb_place(&z, k, xk, xm, t);
        else if (pend) zb_place_w(&z, k, t);
#endif
        else if (arr >= 0) zb_place(&z, k, xk, xm, arr);
        else z.state[k] = 1;
        zb_wake(&z);
    }
    rc = zb_check(&z);
    if (rc) goto out;
    {
        int64_t mk = 0, num = 0;
        for (int q = 0; q < 3 * P * M; ++q) if (end[q] > mk) mk = end[q];
        for (int k = 0; k < P; ++k) { idle[k] = mk - busy[k]; num += idle[k]; }
        *makespan = mk;
        bub[0] = num;
        bub[1] = (int64_t)P * mk;
    }
out:
    free(z.kind); free(z.mb); free(z.border); free(z.pos); free(z.nf); free(z.nb); free(z.nw);
    free(z.held); free(z.state); free(z.t_free);
    return rc;
}

typedef struct {
    int policy, P, M;
    const int32_t *cost_f, *cost_b, *cost_w;
    int64_t cs_inst, cs_stage, cs_mb;
    const int32_t *comm;
    int64_t ms_inst, ms_bnd;
    int64_t *makespan, *idle, *bub_num, *bub_den;
    int32_t *peak;                       /* [n][P] */
    int8_t *status;
    int64_t *op_start, *op_end;          /* [n][P][3][M] or NULL */
    int64_t lo, hi;
    int rc;
} orc_zb_job;

static void *zb_worker(void *arg)
{
    orc_zb_job *jb = (orc_zb_job *)arg;
    int P = jb->P, M = jb->M, n3 = 3 * P * M;
    int64_t *tf = (int64_t *)malloc((size_t)P * M * sizeof(int64_t));
    int64_t *tb = (int64_t *)malloc((size_t)P * M * sizeof(int64_t));
    int64_t *tw = (int64_t *)malloc((size_t)P * M * sizeof(int64_t));
    int64_t *cm = (int64_t *)malloc((size_t)(P > 1 ? P - 1 : 1) * sizeof(int64_t));
    int64_t *st = (int64_t *)malloc((size_t)n3 * sizeof(int64_t));
    int64_t *en = (int64_t *)malloc((size_t)n3 * sizeof(int64_t));
    int64_t *busy = (int64_t *)malloc((size_t)P * sizeof(int64_t));
    int64_t *idle = (int64_t *)malloc((size_t)P * sizeof(int64_t));
    int *peak = (int *)malloc((size_t)P * sizeof(int));
    jb->rc = ORC_OK;
    if (!tf || !tb || !tw || !cm || !st || !en || !busy || !idle || !peak) { jb->rc = ORC_ERR_NOMEM; goto out; }
    for (int64_t x = jb->lo; x < jb->hi; ++x) {
        int neg = 0, zero = 0;
        for (int s = 0; s < P; ++s)
            for (int i = 0; i < M; ++i) {
                int64_t off = x * jb->cs_inst + s * jb->cs_stage + i * jb->cs_mb;
                int q = s * M + i;
                tf[q] = jb->cost_f[off];
                tb[q] = jb->cost_b[off];
                tw[q] = jb->cost_w[off];
                if (tf[q] < 0 || tb[q] < 0 || tw[q] < 0) neg = 1;
                if (tf[q] < 1 || tb[q] < 1) zero = 1;
            }
        for (int b = 0; b < P - 1; ++b) {
            cm[b] = jb->comm ? jb->comm[x * jb->ms_inst + b * jb->ms_bnd] : 0;
            if (cm[b] < 0) neg = 1;
        }
        int64_t mk = 0, bub[2] = {0, 0};
        int8_t status = neg ? ORC_ST_NEG_COST : (zero ? ORC_ST_ZERO_COST : ORC_ST_OK);
        if (status == ORC_ST_OK) {
            int rc = orc_zb_inst(jb->policy, P, M, tf, tb, tw, cm, st, en, &mk, busy, idle, bub, peak);
            if (rc) { jb->rc = rc; goto out; }
            if (mk > ORC_INT32_MAX) status = ORC_ST_OVERFLOW;
        } else {
            for (int q = 0; q < n3; ++q) { st[q] = 0; en[q] = 0; }
            for (int d = 0; d < P; ++d) { idle[d] = 0; peak[d] = 0; }
        }
        if (jb->status) jb->status[x] = status;
        jb->makespan[x] = mk;
        for (int d = 0; d < P; ++d) {
            jb->idle[x * P + d] = idle[d];
            if (jb->peak) jb->peak[x * P + d] = peak[d];
        }
        jb->bub_num[x] = bub[0];
        jb->bub_den[x] = bub[1];
        if (jb->op_start)
            for (int q = 0; q < n3; ++q) {
                jb->op_start[x * n3 + q] = st[q];
                jb->op_end[x * n3 + q] = en[q];
            }
    }
out:
    free(tf); free(tb); free(tw); free(cm); free(st); free(en); free(busy); free(idle); free(peak);
    return NULL;
}

/* Evaluate n ZB instances.  Costs are int32 [inst][stage][mb] through element
 * strides (the same for F, B and W); comm int32 [inst][boundary] or NULL.
 * Outputs: int64 makespan[n], idle[n][P], bub_num[n], bub_den[n]; int32
 * peak[n][P] (may be NULL); int8 status[n]; optional int64 op times
 * [n][P][3][M].  Instances with a negative cost or comm (ORC_ST_NEG_COST) or an
 * F or B cost below 1 (ORC_ST_ZERO_COST) are not evaluated (outputs 0). */
int orc_zb_batch(int policy, int P, int M, int64_t n,
                 const int32_t *cost_f, const int32_t *cost_b, const int32_t *cost_w,
                 int64_t cs_inst, int64_t cs_stage, int64_t cs_mb,
                 const int32_t *comm, int64_t ms_inst, int64_t ms_bnd,
                 int64_t *makespan, int64_t *idle, int64_t *bub_num, int64_t *bub_den,
                 int32_t *peak, int8_t *status, int64_t *op_start, int64_t *op_end, int nthreads)
{
    if ((policy != ORC_ZB1P && policy != ORC_ZB2P) || P < 1 || M < 1 || n < 0) return ORC_ERR_ARG;
    if (nthreads < 1) nthreads = 1;
    if (nthreads > 256) nthreads = 256;
    if ((int64_t)nthreads > n) nthreads = n > 0 ? (int)n : 1;
    orc_zb_job jobs[256];
    pthread_t th[256];
    for (int t = 0; t < nthreads; ++t) {
        orc_zb_job *jb = &jobs[t];
        jb->policy = policy; jb->P = P; jb->M = M;
        jb->cost_f = cost_f; jb->cost_b = cost_b; jb->cost_w = cost_w;
        jb->cs_inst = cs_inst; jb->cs_stage = cs_stage; jb->cs_mb = cs_mb;
        jb->comm = comm; jb->ms_inst = ms_inst; jb->ms_bnd = ms_bnd;
        jb->makespan = makespan; jb->idle = idle; jb->bub_num = bub_num; jb->bub_den = bub_den;
        jb->peak = peak; jb->status = status; jb->op_start = op_start; jb->op_end = op_end;
        jb->lo = n * t / nthreads; jb->hi = n * (t + 1) / nthreads;
        jb->rc = ORC_OK;
    }
    if (nthreads == 1) zb_worker(&jobs[0]);
    else {
        for (int t = 0; t < nthreads; ++t) pthread_create(&th[t], NULL, zb_worker, &jobs[t]);
        for (int t = 0; t < nthreads; ++t) pthread_join(th[t], NULL);
    }
    for (int t = 0; t < nthreads; ++t) if (jobs[t].rc) return jobs[t].rc;
    return ORC_OK;
}

/* ------------------------------------------------------------------------- */
/* DualPipe: two routes through the same stages in opposite directions       */
/* ------------------------------------------------------------------------- */

/*
 * [GPipe->ZB] "DualPipe (DeepSeek-V3)": with P devices and the model cut into
 * P blocks of layers, one group of microbatches enters at device 0 and runs
 * blocks 0..P-1 on devices 0..P-1 (route A); the other group enters at device
 * P-1 and runs the same blocks in the same order on devices P-1..0 (route B).
 * So device d holds block d for route A and block P-1-d for route B (two
 * copies of the parameters), and a device that waits for one route's input
 * can run the other route's ready op.  The page leaves the merged order to the
 * original authors; the reading taken here:
 *   - route A carries microbatches 0..MA-1, route B microbatches MA..MA+MB-1;
 *   - on each route every stage keeps its 1F1B order ([1F1B] §2.3/§3.2):
 *     F^w (B F)^(Mr-w) B^w with w = min(P - s, Mr) at stage s of a route with
 *     Mr microbatches;
 *   - a device that is free at tick t runs an op whose input has arrived by t,
 *     taken from the front of either route's order; when both fronts are
 *     ready it takes a backward before a forward and, between two ops of the
 *     same kind, the route in which it is the earlier stage (route A when d <=
 *     P-1-d); when neither is ready it waits for the first arrival;
 *   - comm[l] is the latency of the link between devices l and l+1, the same
 *     for both routes and both directions; it occupies neither device;
 *   - costs are per (block s, microbatch g): F and B of microbatch g on block s
 *     take tf[s][g], tb[s][g] ticks wherever the block runs.  F and B costs
 *     are at least 1 tick, so whether an input "has arrived by t" depends on
 *     the costs alone and not on the order in which simultaneous decisions are
 *     taken;
 *   - the ledger counts held activations per device: +1 at each F, -1 at
 *     each B of either route.
 * Op times are stored by (block s, kind, microbatch g): index (s*2 + kind)*M + g.
 */
typedef struct {
    int P, MA, MB, M;
    const int64_t *tf, *tb, *comm;
    int64_t *start, *end;
    int nf[2][16], nb[2][16];
} dp_sim;

static int dp_stage(int P, int route, int d) { return route == 0 ? d : P - 1 - d; }

static int dp_link(int P, int route, int b)   /* link of the boundary between blocks b and b+1 */
{
#if ORC_MUTANT == 15  /* mistake: route B crosses the boundary on route A's link */
    (void)P; (void)route;
    return b;
#else
    return route == 0 ? b : P - 2 - b;
#endif
}

/* The front of route r's order on device d: 1 with *isF, *g (global
 * microbatch) and *s (block), or 0 when the route is done on d. */
static int dp_front(const dp_sim *z, int r, int d, int *isF, int *g, int *s)
{
    int Mr = r == 0 ? z->MA : z->MB, st = dp_stage(z->P, r, d);
    int w = z->P - st < Mr ? z->P - st : Mr;
    int nf = z->nf[r][d], nb = z->nb[r][d], q = nf + nb - w;
    if (nf + nb == 2 * Mr) return 0;
    *isF = q < 0 || (q < 2 * (Mr - w) && (q & 1));
    *g = (r == 0 ? 0 : z->MA) + (*isF ? nf : nb);
    *s = st;
    return 1;
}

/* Arrival tick of the input of op (route r, block s, kind, microbatch g), or
 * -1 while a producer is not placed. */
static int64_t dp_arrival(const dp_sim *z, int r, int s, int isF, int g)
{
    int P = z->P, M = z->M;
    if (isF) {
        if (s == 0) return 0;
        int64_t e = z->end[((s - 1) * 2 + ORC_F) * M + g];
        return e < 0 ? -1 : e + (z->comm ? z->comm[dp_link(P, r, s - 1)] : 0);
    }
    int64_t a = z->end[(s * 2 + ORC_F) * M + g];   /* its own forward, on the same device */
    if (a < 0) return -1;
    if (s < P - 1) {
        int64_t e = z->end[((s + 1) * 2 + ORC_B) * M + g];
        if (e < 0) return -1;
        e += z->comm ? z->comm[dp_link(P, r, s)] : 0;
        if (e > a) a = e;
    }
    return a;
}

static int dp_cmp_start(const void *x, const void *y)
{
    int64_t a = ((const int64_t *)x)[0], b = ((const int64_t *)y)[0];
    return a < b ? -1 : (a > b ? 1 : 0);
}

int orc_dp_inst(int P, int MA, int MB, const int64_t *tf, const int64_t *tb, const int64_t *comm,
                int64_t *start, int64_t *end, int64_t *makespan, int64_t *busy, int64_t *idle,
                int64_t *bub, int *peak)
{
    if (P < 1 || P > 16 || MA < 0 || MB < 0 || MA + MB < 1) return ORC_ERR_ARG;
    int M = MA + MB;
    for (int q = 0; q < P * M; ++q)
        if (tf[q] < 1 || tb[q] < 1) return ORC_ERR_ARG;
    dp_sim z;
    memset(&z, 0, sizeof(z));
    z.P = P; z.MA = MA; z.MB = MB; z.M = M;
    z.tf = tf; z.tb = tb; z.comm = comm; z.start = start; z.end = end;
    int64_t t_free[16];
    int held[16];
    for (int d = 0; d < P; ++d) { t_free[d] = 0; held[d] = 0; peak[d] = 0; busy[d] = 0; }
    for (int q = 0; q < 2 * P * M; ++q) { start[q] = -1; end[q] = -1; }
    int64_t T = 0;
    for (;;) {
        /* every device free by T takes the op the rules give it at T; what it
         * places ends after T, so no decision at T sees another one */
        for (int d = 0; d < P; ++d) {
            if (t_free[d] > T) continue;
            int best = -1, bF = 0, bg = 0, bs = 0;
            int pref = d <= P - 1 - d ? 0 : 1;
            for (int k = 0; k < 2; ++k) {
                int r = k == 0 ? pref : 1 - pref;   /* preferred route first */
                int isF, g, s;
                if (!dp_front(&z, r, d, &isF, &g, &s)) continue;
                int64_t a = dp_arrival(&z, r, s, isF, g);
                if (a < 0 || a > T) continue;
#if ORC_MUTANT == 14  /* mistake: a ready forward goes before a ready backward */
                if (best < 0 || (isF && !bF)) { best = r; bF = isF; bg = g; bs = s; }
#else
                if (best < 0 || (!isF && bF)) { best = r; bF = isF; bg = g; bs = s; }
#endif
            }
            if (best < 0) continue;
            int idx = (bs * 2 + (bF ? ORC_F : ORC_B)) * M + bg;
            int64_t c = bF ? tf[bs * M + bg] : tb[bs * M + bg];
            start[idx] = T;
            end[idx] = T + c;
            t_free[d] = T + c;
            busy[d] += c;
            if (bF) { z.nf[best][d]++; held[d]++; if (held[d] > peak[d]) peak[d] = held[d]; }
            else { z.nb[best][d]++; held[d]--; }
        }
        /* the next tick at which something can change: a device becomes free,
         * or an input a free device waits for arrives */
        int64_t next = -1;
        int left = 0;
        for (int d = 0; d < P; ++d) {
            int isF, g, s, any = 0;
            for (int r = 0; r < 2; ++r) {
                if (!dp_front(&z, r, d, &isF, &g, &s)) continue;
                any = 1;
                if (t_free[d] > T) continue;
                int64_t a = dp_arrival(&z, r, s, isF, g);
                if (a > T && (next < 0 || a < next)) next = a;
            }
            if (!any) continue;
            left = 1;
            if (t_free[d] > T && (next < 0 || t_free[d] < next)) next = t_free[d];
        }
        if (!left) break;
        if (next < 0) return ORC_ERR_DEADLOCK;
        T = next;
    }
    /* validity ([M040] §08): every op placed, no overlap on a device, every
     * input arrived before its op starts, every B after its F.  The overlap
     * check sorts each device's ops by start tick and compares neighbours. */
    {
        int64_t (*iv)[2] = (int64_t (*)[2])malloc((size_t)2 * M * sizeof(*iv));
        if (!iv) return ORC_ERR_NOMEM;
        for (int d = 0; d < P; ++d) {
            int n = 0;
            for (int r = 0; r < 2; ++r) {
                int s = dp_stage(P, r, d), g0 = r == 0 ? 0 : MA, g1 = r == 0 ? MA : M;
                for (int g = g0; g < g1; ++g)
                    for (int kd = 0; kd < 2; ++kd) {
                        iv[n][0] = start[(s * 2 + kd) * M + g];
                        iv[n][1] = end[(s * 2 + kd) * M + g];
                        ++n;
                    }
            }
            qsort(iv, (size_t)n, sizeof(*iv), dp_cmp_start);
            for (int q = 0; q < n; ++q) {
                if (iv[q][0] < 0 || iv[q][1] < iv[q][0] || (q > 0 && iv[q][0] < iv[q - 1][1])) {
                    free(iv);
                    return ORC_ERR_INVARIANT;
                }
            }
        }
        free(iv);
    }
    for (int r = 0; r < 2; ++r) {
        int g0 = r == 0 ? 0 : MA, g1 = r == 0 ? MA : M;
        for (int g = g0; g < g1; ++g)
            for (int s = 0; s < P; ++s) {
                int64_t fs = start[(s * 2 + ORC_F) * M + g], fe = end[(s * 2 + ORC_F) * M + g];
                int64_t bs = start[(s * 2 + ORC_B) * M + g];
                if (bs < fe) return ORC_ERR_INVARIANT;
                if (s > 0 && fs < end[((s - 1) * 2 + ORC_F) * M + g] + (comm ? comm[dp_link(P, r, s - 1)] : 0))
                    return ORC_ERR_INVARIANT;
                if (s < P - 1 && bs < end[((s + 1) * 2 + ORC_B) * M + g] + (comm ? comm[dp_link(P, r, s)] : 0))
                    return ORC_ERR_INVARIANT;
            }
    }
    int64_t mk = 0, num = 0;
    for (int q = 0; q < 2 * P * M; ++q) if (end[q] > mk) mk = end[q];
    for (int d = 0; d < P; ++d) { idle[d] = mk - busy[d]; num += idle[d]; }
    *makespan = mk;
    bub[0] = num;
    bub[1] = (int64_t)P * mk;
    return ORC_OK;
}

typedef struct {
    int P, MA, MB;
    const int32_t *cost_f, *cost_b;
    int64_t cs_inst, cs_stage, cs_mb;
    const int32_t *comm;
    int64_t ms_inst, ms_link;
    int64_t *makespan, *idle, *bub_num, *bub_den;
    int32_t *peak;                       /* [n][P] */
    int8_t *status;
    int64_t *op_start, *op_end;          /* [n][P][2][M] or NULL */
    int64_t lo, hi;
    int rc;
} orc_dp_job;

static void *dp_worker(void *arg)
{
    orc_dp_job *jb = (orc_dp_job *)arg;
    int P = jb->P, M = jb->MA + jb->MB, n2 = 2 * P * M;
    int64_t *tf = (int64_t *)malloc((size_t)P * M * sizeof(int64_t));
    int64_t *tb = (int64_t *)malloc((size_t)P * M * sizeof(int64_t));
    int64_t *cm = (int64_t *)malloc((size_t)(P > 1 ? P - 1 : 1) * sizeof(int64_t));
    int64_t *st = (int64_t *)malloc((size_t)n2 * sizeof(int64_t));
    int64_t *en = (int64_t *)malloc((size_t)n2 * sizeof(int64_t));
    int64_t busy[16], idle[16];
    int peak[16];
    jb->rc = ORC_OK;
    if (!tf || !tb || !cm || !st || !en) { jb->rc = ORC_ERR_NOMEM; goto out; }
    for (int64_t x = jb->lo; x < jb->hi; ++x) {
        int neg = 0, zero = 0;
        for (int s = 0; s < P; ++s)
            for (int g = 0; g < M; ++g) {
                int64_t off = x * jb->cs_inst + s * jb->cs_stage + g * jb->cs_mb;
                tf[s * M + g] = jb->cost_f[off];
                tb[s * M + g] = jb->cost_b[off];
                if (tf[s * M + g] < 0 || tb[s * M + g] < 0) neg = 1;
                if (tf[s * M + g] < 1 || tb[s * M + g] < 1) zero = 1;
            }
        for (int l = 0; l < P - 1; ++l) {
            cm[l] = jb->comm ? jb->comm[x * jb->ms_inst + l * jb->ms_link] : 0;
            if (cm[l] < 0) neg = 1;
        }
        int64_t mk = 0, bub[2] = {0, 0};
        int8_t status = neg ? ORC_ST_NEG_COST : (zero ? ORC_ST_ZERO_COST : ORC_ST_OK);
        if (status == ORC_ST_OK) {
            int rc = orc_dp_inst(P, jb->MA, jb->MB, tf, tb, cm, st, en, &mk, busy, idle, bub, peak);
            if (rc) { jb->rc = rc; goto out; }
            if (mk > ORC_INT32_MAX) status = ORC_ST_OVERFLOW;
        } else {
            for (int q = 0; q < n2; ++q) { st[q] = 0; en[q] = 0; }
            for (int d = 0; d < P; ++d) { idle[d] = 0; peak[d] = 0; }
        }
        if (jb->status) jb->status[x] = status;
        jb->makespan[x] = mk;
        for (int d = 0; d < P; ++d) {
            jb->idle[x * P + d] = idle[d];
            if (jb->peak) jb->peak[x * P + d] = peak[d];
        }
        jb->bub_num[x] = bub[0];
        jb->bub_den[x] = bub[1];
        if (jb->op_start)
            for (int q = 0; q < n2; ++q) {
                jb->op_start[x * n2 + q] = st[q];
                jb->op_end[x * n2 + q] = en[q];
            }
    }
out:
    free(tf); free(tb); free(cm); free(st); free(en);
    return NULL;
}

/* Evaluate n DualPipe instances (route A: microbatches 0..MA-1, route B:
 * MA..MA+MB-1).  Costs are int32 [inst][block][microbatch] through element
 * strides; comm int32 [inst][link] or NULL.  Outputs as orc_zb_batch, with
 * op times [n][P blocks][2 kinds][M]. */
int orc_dp_batch(int P, int MA, int MB, int64_t n,
                 const int32_t *cost_f, const int32_t *cost_b,
                 int64_t cs_inst, int64_t cs_stage, int64_t cs_mb,
                 const int32_t *comm, int64_t ms_inst, int64_t ms_link,
                 int64_t *makespan, int64_t *idle, int64_t *bub_num, int64_t *bub_den,
                 int32_t *peak, int8_t *status, int64_t *op_start, int64_t *op_end, int nthreads)
{
    if (P < 1 || P > 16 || MA < 0 || MB < 0 || MA + MB < 1 || n < 0) return ORC_ERR_ARG;
    if (nthreads < 1) nthreads = 1;
    if (nthreads > 256) nthreads = 256;
    if ((int64_t)nthreads > n) nthreads = n > 0 ? (int)n : 1;
    orc_dp_job jobs[256];
    pthread_t th[256];
    for (int t = 0; t < nthreads; ++t) {
        orc_dp_job *jb = &jobs[t];
        jb->P = P; jb->MA = MA; jb->MB = MB;
        jb->cost_f = cost_f; jb->cost_b = cost_b;
        jb->cs_inst = cs_inst; jb->cs_stage = cs_stage; jb->cs_mb = cs_mb;
        jb->comm = comm; jb->ms_inst = ms_inst; jb->ms_link = ms_link;
        jb->makespan = makespan; jb->idle = idle; jb->bub_num = bub_num; jb->bub_den = bub_den;
        jb->peak = peak; jb->status = status; jb->op_start = op_start; jb->op_end = op_end;
        jb->lo = n * t / nthreads; jb->hi = n * (t + 1) / nthreads;
        jb->rc = ORC_OK;
    }
    if (nthreads == 1) dp_worker(&jobs[0]);
    else {
        for (int t = 0; t < nthreads; ++t) pthread_create(&th[t], NULL, dp_worker, &jobs[t]);
        for (int t = 0; t < nthreads; ++t) pthread_join(th[t], NULL);
    }
    for (int t = 0; t < nthreads; ++t) if (jobs[t].rc) return jobs[t].rc;
    return ORC_OK;
}
