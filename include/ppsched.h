/*
 * ppsched.h -- C ABI of libppsched, a GB300 (sm_103a) batched evaluator of
 * pipeline-parallel training schedules: GPipe, synchronous 1F1B
 * (PipeDream-Flush), interleaved 1F1B and the Zero Bubble schedules ZB1P and
 * ZB2P.
 *
 * Sources, by page title and section (short names in brackets):
 *   [1F1B]      "2. 1F1B" (sgdbs.github.io, AI_Infra / 2.PipelineParallel / OneF1B)
 *   [GPipe->ZB] "Pipeline parallelism: from GPipe to 1F1B and Zero Bubble" (dlog.com.cn)
 *   [M040]      "Pipeline scheduling: GPipe, 1F1B, interleaving and compute-communication
 *               overlap" (xuujii.github.io, ai-infra-kb M040)
 *   [Megatron3] "Megatron-LM distributed training (3): pipeline parallelism PP and
 *               1F1B scheduling" (swordlidev.github.io)
 *   [lpnh]      lpnh.cn news 2768528 (GPipe / 1F1B / interleaved formulas, 80-layer model)
 *
 * The problem ([GPipe->ZB] Megatron section; [M040] §04; [lpnh]): P pipeline
 * stages (devices), M microbatches, v model chunks per device (interleaved
 * only; S = P*v virtual stages, device k holds virtual stages k, k+P, ...),
 * a forward cost t_f and backward cost t_b per (virtual stage, microbatch) and
 * a latency `comm` per stage boundary.  Dependencies ([GPipe->ZB] GPipe figure
 * text; [M040] §01, §08): F(s,i) needs F(s-1,i); B(s,i) needs B(s+1,i) and
 * F(s,i); a device runs one op at a time, in its schedule's order; a result
 * crossing boundary b (between virtual stages b and b+1) arrives comm[b] ticks
 * after its op ends.  Every op starts at the earliest tick its device is free
 * and its inputs have arrived (max-plus longest path).
 *
 * Conventions for every entry point:
 *   - Indices are 0-based.  O = 2*M*v ops per device; op position j indexes a
 *     device's order.
 *   - All times are int32 ticks; costs and comm must be >= 0.
 *   - Array arguments are caller-owned DEVICE memory unless stated otherwise.
 *   - Calls are asynchronous on `stream`.  pp_sched_eval and
 *     pp_sched_partition_search allocate nothing once the plan for their shape
 *     exists (pp_sched_plan, or the first call for that shape, builds it; that
 *     first call allocates device memory and synchronizes `stream`).
 *   - Return value: PP_OK or a PP_ERR_* code (argument errors are detected on the
 *     host before anything is launched).  Per-instance data problems are written
 *     to the optional `status` array instead.
 *   - One GPU: the library works on the calling thread's current device.
 */
#ifndef PPSCHED_H
#define PPSCHED_H

#include <stdint.h>
#include <cuda_runtime_api.h>

#ifdef __cplusplus
extern "C" {
#endif

#define PPSCHED_ABI_VERSION 1

/* Schedule policies.
 *  PP_GPIPE: every device runs F of microbatches 0..M-1, then B of M-1..0
 *    ([M040] §02 table: backwards from D to A).
 *  PP_1F1B: device k runs w = min(P-k, M) forwards, then M-w (B, F) pairs with
 *    the oldest outstanding B first, then the remaining w backwards ([1F1B] §2.3,
 *    §3.2 table; [Megatron3] "three phases": num_warmup = P-k-1 plus the first
 *    steady F is the same sequence).
 *  PP_INTERLEAVED_1F1B: v > 1 chunks per device; warmup 2(P-k-1)+(v-1)P forwards
 *    (capped at M*v), then (F, B) pairs, then the remaining B; forward j is chunk
 *    (j mod Pv)/P of microbatch (j/(Pv))*P + j mod P, backward j is chunk
 *    v-1-(j mod Pv)/P of the same microbatch.  Requires M % P == 0 ([M040] §06).
 *    The pages give the bubble, (P-1)/(vM+P-1) ([1F1B] §6.1), not the order; this
 *    order is the Megatron interleaved schedule they refer to.
 *  PP_GPIPE_FIFO: GPipe with the backwards in first-in-first-out order, B of
 *    microbatches 0..M-1 (the variant of [M040] §02's last-in-first-out table;
 *    the same makespan at uniform costs, other op times).
 *  PP_ZB1P, PP_ZB2P (Zero Bubble; only through pp_sched_eval_zb): the backward
 *    splits into B (input gradient) and W (weight gradient, no cross-stage
 *    edge); see pp_sched_eval_zb ([GPipe->ZB] "Zero Bubble", "ZB1P and ZB2P"). */
typedef enum {
    PP_GPIPE = 0,
    PP_1F1B = 1,
    PP_INTERLEAVED_1F1B = 2,
    PP_ZB1P = 3,
    PP_ZB2P = 4,
    PP_GPIPE_FIFO = 5
} pp_policy_t;

/* Return codes. */
#define PP_OK 0
#define PP_ERR_ARG 1           /* bad argument: P, M or v < 1, v != 1 for GPipe/1F1B,
                                  v < 2 for interleaved, NULL required pointer,
                                  n < 0, bad stride or alignment */
#define PP_ERR_DIVISIBILITY 2  /* interleaved with M % P != 0 */
#define PP_ERR_SIZE 3          /* shape beyond the limits below */
#define PP_ERR_CUDA 4          /* a CUDA runtime call failed */
#define PP_ERR_DEADLOCK 5      /* the generated order cannot run (internal check) */
#define PP_ERR_INTERNAL 6      /* an internal consistency check failed */

/* Per-instance status (int8) written by pp_sched_eval when `status` != NULL.
 * The other outputs of a flagged instance are unspecified. */
#define PP_ST_OK 0
#define PP_ST_NEG_COST 1       /* some cost or comm of the instance is negative */
#define PP_ST_OVERFLOW 2       /* some tick would exceed INT32_MAX (detected, not wrapped) */
#define PP_ST_ZERO_COST 3      /* Zero Bubble only: some F or B cost is below 1 tick */

/* Limits. */
#define PP_MAX_P 16            /* devices */
#define PP_MAX_S 64            /* virtual stages P*v */
#define PP_MAX_MV 32768        /* microbatches x chunks (ops per device = 2*M*v) */

/* Packed op, as returned by pp_sched_plan_ops: bit 31 = kind (0 = F, 1 = B),
 * bits 24..30 = chunk, bits 0..23 = microbatch. */
#define PP_OP_KIND(x) ((int)(((uint32_t)(x)) >> 31))
#define PP_OP_CHUNK(x) ((int)((((uint32_t)(x)) >> 24) & 0x7Fu))
#define PP_OP_MB(x) ((int)(((uint32_t)(x)) & 0xFFFFFFu))

/* Opaque plan: the schedule of one (policy, P, M, v), built on the GPU. */
typedef struct pp_plan pp_plan_t;

/* Build the plan for (policy, P, M, v) on the current device: the per-device op
 * order, each op's wavefront round (its start tick at unit cost, which is a
 * topological order of the dependency graph), the per-round op table the
 * evaluator walks, and the peak held-activation count per device ([1F1B] §4.1
 * ledger).  Allocates device memory and synchronizes `stream`.
 * *plan receives a library-owned object; free it with pp_sched_plan_destroy.
 * Errors: PP_ERR_ARG, PP_ERR_DIVISIBILITY, PP_ERR_SIZE, PP_ERR_DEADLOCK, PP_ERR_CUDA. */
int pp_sched_plan(pp_policy_t policy, int P, int M, int v, pp_plan_t **plan, cudaStream_t stream);

/* Plan facts: info[0] = rounds (unit-cost makespan), info[1] = ops per device,
 * info[2] = dependency value slots the generic evaluator needs, info[3] = 1 if the
 * register evaluator applies (GPipe, 1F1B), info[4] = P, info[5] = M, info[6] = v,
 * info[7] = policy.  `info` is host memory of 8 int32. */
int pp_sched_plan_info(const pp_plan_t *plan, int32_t *info);

/* Copy the plan to HOST memory: host_ops [P][2Mv] packed ops (see PP_OP_*),
 * host_peak [P] peak held activations per device, host_round [P][2Mv] each op's
 * wavefront round.  Any pointer may be NULL.  Synchronous. */
int pp_sched_plan_ops(const pp_plan_t *plan, uint32_t *host_ops, int32_t *host_peak, int32_t *host_round);

/* Free a plan (NULL is ignored).  The caller must not use it in flight. */
void pp_sched_plan_destroy(pp_plan_t *plan);

/* Evaluate n_instances schedule instances of one policy and shape.
 *
 * Inputs (device, int32):
 *   cost_f, cost_b: forward / backward cost of (instance x, virtual stage s,
 *     microbatch i) at element offset x*stride_inst + s*stride_stage + i*stride_mb.
 *     Strides may be 0 (broadcast).  The fast path wants stride_inst == 1 (the
 *     instance-minor layout [S][M][n], every load coalesced and 128-bit wide) with
 *     16-byte aligned bases and stride_stage, stride_mb multiples of 4; any other
 *     layout is accepted and gathered 4 bytes at a time.
 *   comm: latency of boundary b (virtual stages b and b+1) for instance x at
 *     x*comm_stride_inst + b*comm_stride_bnd, b < S-1; NULL means 0 everywhere.
 * Outputs (device; each may be NULL):
 *   makespan [n]          last end tick over all devices ([M040] §04 window time)
 *   idle [n][P]           makespan minus the device's summed op costs
 *   bub_num, bub_den [n]  exact bubble fraction = sum of idle / (P * makespan)
 *                         ([1F1B] §4.3; [M040] §04), unreduced; both 0 when the
 *                         makespan is 0
 *   peak [P]              peak held activations per device (cost-independent)
 *   op_start, op_end      each op's start / end tick at element offset
 *                         x*op_stride_inst + (k*O + j)*op_stride_op
 *   status [n]            PP_ST_* per instance
 * Errors: PP_ERR_ARG, PP_ERR_DIVISIBILITY, PP_ERR_SIZE, PP_ERR_CUDA, plus the plan
 * errors on a shape's first call. */
int pp_sched_eval(pp_policy_t policy, int P, int M, int v,
                  const int32_t *cost_f, const int32_t *cost_b,
                  int64_t stride_inst, int64_t stride_stage, int64_t stride_mb,
                  const int32_t *comm, int64_t comm_stride_inst, int64_t comm_stride_bnd,
                  int64_t n_instances,
                  int32_t *makespan, int32_t *idle, int64_t *bub_num, int64_t *bub_den,
                  int32_t *peak,
                  int32_t *op_start, int32_t *op_end, int64_t op_stride_inst, int64_t op_stride_op,
                  int8_t *status, cudaStream_t stream);

/* pp_sched_eval with a separate latency on the backward edges ([M040] §05: a
 * forward boundary carries the hidden activations, a backward boundary their
 * gradients).  comm_f[b] is added to F(b+1,i)'s input from F(b,i) and comm_b[b]
 * to B(b,i)'s input from B(b+1,i); both use comm_stride_inst and
 * comm_stride_bnd; either may be NULL (comm_b NULL: the same as comm_f, which
 * is pp_sched_eval).  With comm_b given, every policy runs on the generic
 * (lane) evaluator, which needs cost-row offsets below 2^30 elements
 * (PP_ERR_SIZE otherwise).  Everything else as pp_sched_eval. */
int pp_sched_eval_fb(pp_policy_t policy, int P, int M, int v,
                     const int32_t *cost_f, const int32_t *cost_b,
                     int64_t stride_inst, int64_t stride_stage, int64_t stride_mb,
                     const int32_t *comm_f, const int32_t *comm_b,
                     int64_t comm_stride_inst, int64_t comm_stride_bnd,
                     int64_t n_instances,
                     int32_t *makespan, int32_t *idle, int64_t *bub_num, int64_t *bub_den,
                     int32_t *peak,
                     int32_t *op_start, int32_t *op_end, int64_t op_stride_inst, int64_t op_stride_op,
                     int8_t *status, cudaStream_t stream);

/* pp_sched_eval from HOST memory: the entry for callers whose cost tables
 * are in host memory.  h_cost_f, h_cost_b are instance-minor [S][M][n] int32
 * (element (s, i, x) at (s*M + i)*n + x) and h_comm [S-1][n] or NULL, in host
 * memory (page-locked memory makes the copies asynchronous).  The call copies
 * the instances chunk by chunk into the caller's device workspace d_work
 * (256-byte aligned, work_bytes long; pp_sched_eval_host_workspace gives the
 * size that holds the whole batch in one chunk, and any smaller size down to
 * one chunk of 32 instances works), evaluates each chunk with pp_sched_eval
 * and copies the chunk's results into the HOST outputs h_makespan [n], h_idle
 * [n][P], h_bub_num [n], h_bub_den [n], h_peak [P], h_status [n] (each may be
 * NULL).  The host outputs are valid once `stream` completes.  When the
 * workspace holds two chunks of about n/4 instances (the size below does), the
 * chunks alternate between two workspace slots and the evaluation and result
 * copies of one chunk run on an auxiliary stream of the library while the
 * next chunk is copied in on `stream`; events join the auxiliary stream back
 * into `stream` before the call's work ends there.  The first such call on a
 * device creates that stream and its events (make it before any stream
 * capture); calls on one device enqueue one at a time.  With room for one
 * chunk only, chunks run one after another on `stream`.
 * Errors: as pp_sched_eval; PP_ERR_ARG for a misaligned workspace; PP_ERR_SIZE
 * when the workspace is smaller than a 32-instance chunk. */
int pp_sched_eval_host(pp_policy_t policy, int P, int M, int v,
                       const int32_t *h_cost_f, const int32_t *h_cost_b, const int32_t *h_comm,
                       int64_t n_instances, void *d_work, size_t work_bytes,
                       int32_t *h_makespan, int32_t *h_idle, int64_t *h_bub_num, int64_t *h_bub_den,
                       int32_t *h_peak, int8_t *h_status, cudaStream_t stream);

/* Device workspace bytes pp_sched_eval_host needs to take n_instances in one
 * chunk (0 for bad arguments). */
size_t pp_sched_eval_host_workspace(int P, int M, int v, int64_t n_instances);

/* Many evaluation problems, each with its own shape (policy, P, M, v), cost
 * tables and outputs, evaluated together.  This serves sweeps over schedule
 * shapes -- the bubble's dependence on P, M and v in [1F1B] §4.3 and §6.1 and
 * [M040] §04 -- where each shape has only a few instances: evaluated one call
 * at a time, each problem is a CTA or two walking hundreds of dependent rounds
 * and the GPU stays nearly idle.
 *
 * pp_problem_t holds the arguments of pp_sched_eval without per-op output;
 * every pointer is caller-owned device memory, as there.
 *
 * pp_sched_many_prepare checks every problem as pp_sched_eval would (the first
 * error found is returned and no handle is made), builds each shape's plan and
 * the kernel tables of its strides (allocating and synchronizing `stream`),
 * and records each problem in the handle:
 *   - GPipe, GPipe FIFO and 1F1B problems whose costs are the same for every
 *     microbatch (stride_mb == 0), and interleaved problems likewise, go to a
 *     fused kernel: one launch per kernel kind and table width (at most six)
 *     evaluates all of them, each problem's CTAs finding their problem in a
 *     job table the handle keeps in device memory;
 *   - every other problem (costs varying per microbatch, empty batches, shapes
 *     whose tables do not fit the fused kernels) is evaluated by pp_sched_eval
 *     inside pp_sched_many_eval.
 * The handle records the problems' pointers, not their data: between
 * evaluations the caller may rewrite the cost tables and read the outputs.
 *
 * pp_sched_many_eval enqueues the evaluation of every problem on `stream` (the
 * device must be the one the handle was prepared on); the results equal those
 * of pp_sched_eval on each problem.  The fused launches run side by side on
 * streams the library creates once per device (at the first evaluation with
 * more than one launch: make it before any stream capture), forked from
 * `stream` by an event and joined back into it, so the evaluation is ordered
 * on `stream` alone; evaluations on one device enqueue one at a time.  It
 * allocates no device memory; when every problem went to a fused kernel it
 * only launches kernels and records events, and can be captured in a CUDA
 * graph.  Evaluations of one handle that overlap on the GPU write the same
 * outputs; serialize them.
 *
 * pp_sched_many_info reports how many problems were fused, in how many
 * launches, and how many are evaluated one by one.
 *
 * The handle refers to the library's cached plans: call pp_sched_cache_clear
 * only after destroying every handle.  Free a handle with
 * pp_sched_many_destroy once its evaluations have completed.
 * Errors: as pp_sched_eval; PP_ERR_ARG for a null handle pointer, a negative
 * count or a null problem array with a positive count. */
typedef struct pp_problem {
    pp_policy_t policy;
    int P, M, v;
    const int32_t *cost_f, *cost_b;
    int64_t stride_inst, stride_stage, stride_mb;
    const int32_t *comm;
    int64_t comm_stride_inst, comm_stride_bnd;
    int64_t n_instances;
    int32_t *makespan, *idle;
    int64_t *bub_num, *bub_den;
    int32_t *peak;
    int8_t *status;
} pp_problem_t;

typedef struct pp_many pp_many_t;

int pp_sched_many_prepare(const pp_problem_t *problems, int n_problems, pp_many_t **many, cudaStream_t stream);
int pp_sched_many_eval(const pp_many_t *many, cudaStream_t stream);
int pp_sched_many_info(const pp_many_t *many, int *fused_problems, int *launches, int *other_problems);
void pp_sched_many_destroy(pp_many_t *many);

/* Score contiguous layer-to-stage partitions under 1F1B and return the best.
 * This is the profiling-based load balancing of [GPipe->ZB] (PipeDream and GPipe
 * sections: split layers into stages by measured cost) and [M040] §05, on the
 * [lpnh] workload (80 layers into 8 stages).
 *
 * Candidate c (c = cand_begin .. cand_begin+n_cand-1) is the split obtained by
 *   u = SplitMix64 output for state seed + c (Steele, Lea & Flood 2014),
 *   r = u mod C(L-1, P-1), and r unranked in colex order to cut positions
 *   x_1 < ... < x_{P-1} in [0, L-1); stage t starts at layer x_t + 1.
 * Stage k's forward cost is the sum of its layers' layer_tf, backward cost the
 * sum of layer_tb, activation bytes the sum of layer_act; every boundary has
 * latency `comm`.  A candidate is rejected when some stage's peak held
 * activations under 1F1B times its activation bytes exceeds act_cap.  The rest
 * are evaluated with M microbatches and the argmin (makespan, candidate index)
 * is returned.  When all_makespan is NULL, a candidate whose makespan provably
 * exceeds the best found so far is not evaluated: every 1F1B makespan is at
 * least max_k [sum_{j<k} (f_j + b_j) + 2k comm + M (f_k + b_k)] (stage k runs
 * its 2M ops one at a time after microbatch 0 crossed the stages before it,
 * and its last backward must cross them back); the result is the same.
 *
 * Inputs (device): layer_tf, layer_tb int32 [L]; layer_act int64 [L].
 * Outputs (device): best_idx int64 [1] (-1 if nothing is feasible),
 *   best_makespan int32 [1] (-1 then), best_cuts int32 [P-1] (first layer of
 *   stages 1..P-1; -1 then), all_makespan int32 [n_cand] or NULL (makespan, -1 if
 *   rejected by the cap, -2 if a tick would exceed INT32_MAX).
 * Limits: 1 <= P <= PP_MAX_P, P <= L <= 256, 0 <= n_cand < 2^32, M <= PP_MAX_MV,
 * and the number of splits C(L-1, P-1) below 2^64 - 1 (e.g. L <= 131 at P = 16);
 * PP_ERR_SIZE otherwise.
 * Errors: PP_ERR_ARG, PP_ERR_SIZE, PP_ERR_CUDA. */
int pp_sched_partition_search(const int32_t *layer_tf, const int32_t *layer_tb,
                              const int64_t *layer_act, int L, int P, int M, int32_t comm,
                              int64_t act_cap, uint64_t seed, int64_t cand_begin, int64_t n_cand,
                              int64_t *best_idx, int32_t *best_makespan, int32_t *best_cuts,
                              int32_t *all_makespan, cudaStream_t stream);

/* The exhaustive form of pp_sched_partition_search: scores the splits of colex
 * ranks rank_begin .. rank_begin + n_ranks - 1, every contiguous split of L
 * layers into P stages having one rank in [0, C(L-1, P-1)) (the cut positions
 * x_1 < ... < x_{P-1} of rank r satisfy r = sum_i C(x_i, i)).  Scoring, cap,
 * outputs and errors as pp_sched_partition_search, with best_rank in place of
 * best_idx (the winning rank; ties go to the lower rank; -1 if nothing is
 * feasible) and all_makespan indexed by rank - rank_begin.  A whole search is
 * rank_begin = 0, n_ranks = C(L-1, P-1) (2,898,753,715 for 80 layers into 8
 * stages); disjoint rank ranges reduce by (makespan, rank).
 * Ranks are int64, so where C(L-1, P-1) exceeds 2^63 only the ranks below 2^63
 * can be named.
 * Extra error: PP_ERR_ARG if rank_begin + n_ranks > C(L-1, P-1). */
int pp_sched_partition_search_ranks(const int32_t *layer_tf, const int32_t *layer_tb,
                                    const int64_t *layer_act, int L, int P, int M, int32_t comm,
                                    int64_t act_cap, int64_t rank_begin, int64_t n_ranks,
                                    int64_t *best_rank, int32_t *best_makespan, int32_t *best_cuts,
                                    int32_t *all_makespan, cudaStream_t stream);

/* The partition search over interleaved layouts ([M040] §06: a device holds
 * several virtual stages; §05: split by measured cost and activation).  Each
 * candidate c in [cand_begin, cand_begin + n_cand) cuts the L layers into
 * S = P*v contiguous non-empty ranges: u = SplitMix64(seed + c),
 * r = u mod C(L-1, S-1), unranked in colex order as pp_sched_partition_search
 * does with S-1 cuts; range s is virtual stage s (chunk s / P of device
 * s mod P).  A candidate is rejected when some device's held activation bytes
 * peak above act_cap (the [1F1B] §4.1 ledger over the interleaved order, +
 * the bytes of the op's range at F, - at B); the others are scored under
 * PP_INTERLEAVED_1F1B with M microbatches, every boundary with latency `comm`.
 * Outputs as pp_sched_partition_search; best_cuts has S-1 entries (first layer
 * of ranges 1..S-1).
 * Memory: the candidates are scored in chunks of up to 262,144 through a
 * scratch cost table the library allocates on a device's first call (about
 * 2 MB per virtual stage) and keeps; calls on one device share it, so calls
 * that overlap on the GPU must be serialized.  The first call for a shape also
 * builds its plan and a small table of its held-count vectors.  Only layouts
 * within the cap are evaluated, packed into the table; the call synchronizes
 * `stream` once per chunk to read how many there are.  When all_makespan is
 * NULL, a layout is not evaluated either when its makespan provably exceeds
 * the best of the chunks already scored (device d starts with microbatch 0's
 * forward of virtual stage d, ends with the backward of virtual stage d for
 * microbatch M-1 and runs its 2Mv ops one at a time); the result is the same.
 * Limits: v >= 2, P*v <= PP_MAX_S, M % P == 0, M*v <= PP_MAX_MV, S <= L <= 256,
 * n_cand < 2^32, and C(L-1, S-1) below 2^64 - 1 (e.g. L <= 84 at S = 64);
 * PP_ERR_SIZE otherwise.
 * Errors: PP_ERR_ARG, PP_ERR_DIVISIBILITY, PP_ERR_SIZE, PP_ERR_CUDA. */
int pp_sched_partition_search_interleaved(const int32_t *layer_tf, const int32_t *layer_tb,
                                          const int64_t *layer_act, int L, int P, int v, int M, int32_t comm,
                                          int64_t act_cap, uint64_t seed, int64_t cand_begin, int64_t n_cand,
                                          int64_t *best_idx, int32_t *best_makespan, int32_t *best_cuts,
                                          int32_t *all_makespan, cudaStream_t stream);

/* Evaluate n_instances DualPipe schedule instances: two routes through the
 * same P blocks of layers in opposite directions.  [GPipe->ZB] "DualPipe
 * (DeepSeek-V3)": microbatches 0..m_a-1 (route A) enter at device 0 and run
 * blocks 0..P-1 on devices 0..P-1; microbatches m_a..M-1 (route B) enter at
 * device P-1 and run the same blocks on devices P-1..0, so device d holds
 * block d of route A and block P-1-d of route B (two parameter copies).  The
 * page names the layout and its costs (peak p+1 activations, parameters x2)
 * but not the merged order; the library's reading:
 *   - at each of its stages a route keeps its 1F1B order F^w (B F)^(Mr-w) B^w,
 *     w = min(P - stage, Mr), Mr its microbatch count;
 *   - a device free at tick t runs an op at the front of either route whose
 *     input has arrived by t: a backward before a forward, and between two
 *     ops of one kind the route in which the device is the earlier stage
 *     (route A when d <= P-1-d); with neither input arrived it waits for the
 *     first arrival;
 *   - F and B costs must be at least 1 tick (else PP_ST_ZERO_COST).
 * The order depends on the costs, so there is no plan.
 *
 * Inputs (device, int32): cost_f, cost_b of (instance x, block s, microbatch
 *   g) at x*stride_inst + s*stride_stage + g*stride_mb (strides may be 0);
 *   comm of (instance x, link l), the latency between devices l and l+1 in
 *   both directions, at x*comm_stride_inst + l*comm_stride_link, NULL means 0.
 * Outputs (device; each may be NULL):
 *   makespan [n], idle [n][P], bub_num [n], bub_den [n]  as pp_sched_eval
 *   peak [n][P]      most activations held at once per device (+1 at F, -1 at B
 *                    of either route); it depends on the costs, hence per instance
 *   op_start, op_end op (block s, kind k (0 F, 1 B), microbatch g) of instance x
 *                    at x*op_stride_inst + ((s*2 + k)*M + g)*op_stride_op
 *   status [n]       PP_ST_* (negative cost or comm first, then a zero F/B
 *                    cost, then overflow)
 * Limits: 1 <= P <= PP_MAX_P, 1 <= M <= PP_MAX_MV, 0 <= m_a <= M.
 * The kernel runs in two exact phases (each lane on its own tick, then the
 * instances left unfinished on a common tick); the environment variable
 * PPSCHED_DP_PHASE1_STEPS, read at each call, sets the first phase's step cap
 * (default 8*M + 64).  The results do not depend on it; only the time does.
 * Errors: PP_ERR_ARG, PP_ERR_SIZE, PP_ERR_CUDA. */
int pp_sched_eval_dualpipe(int P, int M, int m_a, const int32_t *cost_f, const int32_t *cost_b,
                           int64_t stride_inst, int64_t stride_stage, int64_t stride_mb,
                           const int32_t *comm, int64_t comm_stride_inst, int64_t comm_stride_link,
                           int64_t n_instances, int32_t *makespan, int32_t *idle, int64_t *bub_num,
                           int64_t *bub_den, int32_t *peak, int32_t *op_start, int32_t *op_end,
                           int64_t op_stride_inst, int64_t op_stride_op, int8_t *status, cudaStream_t stream);

/* pp_sched_eval for GPipe and 1F1B that allocates no device memory.  (This
 * entry point has no counterpart on the pages; it exists for callers that
 * cannot let a library call cudaMalloc, e.g. code whose device memory belongs to
 * another allocator or that must not grow its device footprint while running.)
 *
 * Same arguments and results as pp_sched_eval with v = 1 and no per-op times.
 * The schedule tables are built in one array of 4 MiB that the library reserves
 * at file scope on every GPU that loads it and keeps until the process exits.
 *   - The first call on a device looks up that array's device address
 *     (cudaGetSymbolAddress); make that first call before any stream capture.
 *   - A call whose shape (policy, P, M) differs from the previous call's on the
 *     device rebuilds all tables in the array and synchronizes `stream` once
 *     (to read the plan's size).  A call with the previous shape but another
 *     stride pair (stride_stage, stride_mb) only enqueues the rebuild of the
 *     stride-dependent tables on `stream`, without a synchronization.  A call
 *     that repeats the previous shape and stride pair reuses the tables and
 *     just launches.
 *   - Every call shares the array: calls that overlap on the GPU (other streams,
 *     other threads) race; serialize them.  In particular a call on another
 *     stream must first wait for `stream` (an event), since a rebuild enqueued
 *     on `stream` may still be writing the tables it would read.
 *   - Shapes whose tables do not fit in the array return PP_ERR_SIZE;
 *     PP_INTERLEAVED_1F1B returns PP_ERR_ARG.
 * Inputs, outputs and strides: as pp_sched_eval.  Errors: as pp_sched_eval. */
int pp_sched_eval_noalloc(pp_policy_t policy, int P, int M,
                          const int32_t *cost_f, const int32_t *cost_b,
                          int64_t stride_inst, int64_t stride_stage, int64_t stride_mb,
                          const int32_t *comm, int64_t comm_stride_inst, int64_t comm_stride_bnd,
                          int64_t n_instances,
                          int32_t *makespan, int32_t *idle, int64_t *bub_num, int64_t *bub_den,
                          int32_t *peak, int8_t *status, cudaStream_t stream);

/* Human-readable name of a PP_ERR_* return code. */
const char *pp_sched_status_str(int code);

/* Free every cached plan of the calling process (all devices).  Not safe while
 * evaluations are in flight. */
void pp_sched_cache_clear(void);

/* The bounds-checked build.  (No counterpart on the pages: a debugging aid for
 * machines without a GPU memory checker.)  Compiled with -DPPS_CHECKED, the
 * kernels check every address they take from a run-time table or from the
 * call's sizes before using it: cost elements against what the strides reach,
 * value-slot and comm cells against the warp's rows in shared memory, slot
 * indices against the plan's slot count, split points against 0..L.  A failed
 * check skips the access (a load reads 0, a copy is zero-filled, a store is
 * dropped; the results are then wrong) and records the failure; nothing traps.
 * Returns 1 for a checked build, 0 otherwise.  *first_failure (may be NULL)
 * receives the first failure recorded since the previous call, 0 if none, and
 * the records are cleared: bit 63 set, the check site in bits 40..55 (1 cost
 * read, 2 slot read, 3 slot write, 4 comm cell, 5 slot index, 6 split point),
 * the low 40 bits of the offending offset below.  Synchronizes the device;
 * call it with no kernel of the library in flight. */
int pp_sched_debug_checks(uint64_t *first_failure);

/* Evaluate n_instances Zero Bubble schedule instances (policy PP_ZB1P or
 * PP_ZB2P, one stage per device).  [GPipe->ZB] "Zero Bubble" and "ZB1P and
 * ZB2P"; [1F1B] §6.2.  The backward of microbatch i on stage k splits into
 * B(k,i), which stage k-1 waits for, and W(k,i), which only needs B(k,i) on
 * the same device.  The op order depends on the costs, so there is no plan:
 *   - F and B keep 1F1B's order F^w (B F)^(M-w) B^w with w = min(P-k, M)
 *     (ZB1P) or min(2(P-k), M) (ZB2P: twice the warmup);
 *   - a device holds at most L = P (ZB1P) or 2P (ZB2P) microbatches whose F
 *     has run and whose W has not;
 *   - a device that becomes free at tick t runs, in this order of preference:
 *     the oldest pending W if its next F/B op is an F and it holds L; that
 *     F/B op if its input has arrived by t; the oldest pending W; else it
 *     waits for the F/B op's input.  With no F/B op left it runs its pending
 *     W's, oldest first.
 * These rules are stated loosely on the pages; the library takes this reading.
 * F and B costs must be at least 1 tick (W may be 0) so that "arrived by t"
 * depends on the costs alone; an instance with an F or B cost below 1 gets
 * PP_ST_ZERO_COST.
 *
 * Inputs (device, int32): cost_f, cost_b, cost_w of (instance x, stage k,
 *   microbatch i) at x*stride_inst + k*stride_stage + i*stride_mb (strides may
 *   be 0); comm [instance][boundary] through its strides, NULL means 0.
 * Outputs (device; each may be NULL):
 *   makespan [n], idle [n][P], bub_num [n], bub_den [n]  as pp_sched_eval
 *   peak [n][P]      most microbatches held at once per device (+1 at F, -1 at
 *                    W); it depends on the costs, hence per instance
 *   op_start, op_end each op's start / end tick at element offset
 *                    x*op_stride_inst + ((k*3 + kind)*M + i)*op_stride_op with
 *                    kind 0 = F, 1 = B, 2 = W
 *   status [n]       PP_ST_* (negative cost or comm first, then a zero F/B
 *                    cost, then overflow)
 * Limits: 1 <= P <= PP_MAX_P, 1 <= M <= PP_MAX_MV.
 * Errors: PP_ERR_ARG (policy, shape, NULL cost pointer with n > 0, negative
 * stride or n), PP_ERR_SIZE, PP_ERR_CUDA.  Allocates nothing; asynchronous. */
int pp_sched_eval_zb(pp_policy_t policy, int P, int M,
                     const int32_t *cost_f, const int32_t *cost_b, const int32_t *cost_w,
                     int64_t stride_inst, int64_t stride_stage, int64_t stride_mb,
                     const int32_t *comm, int64_t comm_stride_inst, int64_t comm_stride_bnd,
                     int64_t n_instances,
                     int32_t *makespan, int32_t *idle, int64_t *bub_num, int64_t *bub_den,
                     int32_t *peak,
                     int32_t *op_start, int32_t *op_end, int64_t op_stride_inst, int64_t op_stride_op,
                     int8_t *status, cudaStream_t stream);

#ifdef __cplusplus
}
#endif

#endif /* PPSCHED_H */
