// many.cu -- pp_sched_many_*: many evaluation problems, each with its own
// shape, costs and outputs, evaluated in a few launches.
//
// A single problem of a few instances is one CTA walking hundreds of
// dependent rounds: launched on its own it leaves the GPU idle.  Preparing a
// set of problems builds every problem's plan and kernel tables once, sorts
// the problems by the kernel that takes them (the microbatch-shared register
// evaluator for GPipe / 1F1B, the microbatch-shared lane evaluator for
// interleaved plans; one group per table width) and uploads one job record per
// problem.  An evaluation is then one launch per group, the groups side by
// side on streams of the library (forked from the caller's stream and joined
// back into it); each CTA finds its problem by binary search over the jobs'
// first CTAs.  Problems that no fused kernel takes get one pp_sched_eval each.
// A group's CTAs are as wide as its widest problem needs (up to the
// single-problem kernels' width), so problems of a few instances do not hold
// idle warps and their shared memory.
#include <algorithm>
#include <mutex>
#include <vector>

#include "eval_common.cuh"

struct pp_many {
    int device = 0;
    pps::ManyJob *d_jobs = nullptr;  // every group's jobs, group after group
    struct Group {
        int kind;       // 0: register evaluator, 1: lane evaluator
        int pmax;       // table width the group's kernel is compiled for
        int first;      // index of the group's first job in d_jobs
        int count;
        int warps;      // warps per CTA: what the widest job fills, capped
        int64_t ctas;   // CTAs of the fused launch
        size_t smem;    // dynamic shared memory per CTA (the largest job's)
    };
    std::vector<Group> groups;
    std::vector<pp_problem_t> rest;  // evaluated one by one
};

namespace pps {
namespace {

struct Pending {
    int kind, pmax;
    ManyJob job;
    int req;  // index of its table request
};

int prepare(const pp_problem_t *problems, int n_problems, pp_many *h, cudaStream_t stream) {
    // every shape's plan, the missing ones built in one batch
    std::vector<PlanShape> shapes(n_problems);
    for (int i = 0; i < n_problems; ++i)
        shapes[i] = PlanShape{(int)problems[i].policy, problems[i].P, problems[i].M, problems[i].v};
    std::vector<pp_plan *> plans(n_problems, nullptr);
    int rc = cached_plans(shapes.data(), n_problems, stream, plans.data());
    if (rc) return rc;
    // which fused kernel takes each problem, and the tables it needs
    std::vector<Pending> jobs;
    std::vector<TableReq> reqs;
    for (int i = 0; i < n_problems; ++i) {
        const pp_problem_t &p = problems[i];
        pp_plan *plan = plans[i];
        if (p.n_instances == 0) {
            h->rest.push_back(p);
            continue;
        }
        EvalArgs a = eval_args(plan, p.cost_f, p.cost_b, p.stride_inst, p.stride_stage, p.stride_mb, p.comm,
                               nullptr, p.comm_stride_inst, p.comm_stride_bnd, p.n_instances, p.makespan, p.idle,
                               p.bub_num, p.bub_den, p.peak, nullptr, nullptr, 0, 0, p.status);
        const int kind = reg_mbz_ok(plan, a) ? 0 : (lane_mbz_ok(plan, a) ? 1 : -1);
        if (kind < 0) {
            h->rest.push_back(p);
            continue;
        }
        jobs.push_back({kind, plan->pmax, {a, nullptr, 0, 0}, (int)reqs.size()});
        reqs.push_back({plan, a.s_stage, a.s_mb, kind, nullptr});
    }
    rc = build_tables(reqs.data(), (int)reqs.size(), stream);
    if (rc) return rc;
    for (Pending &j : jobs) {
        const pp_ktab *t = reqs[j.req].out;
        if (j.kind == 0) {
            j.job.a.ktab = t->d;
            j.job.a.ktab_words = t->words;
        } else {
            j.job.tab = t->d;
            if (lane_table_words(j.pmax, j.job.a.R, true, &j.job.nblocks) < 0) return PP_ERR_INTERNAL;
        }
    }
    // groups by kernel and table width; within a group the jobs with the most
    // rounds first, so that CTAs handed out last are short ones
    std::stable_sort(jobs.begin(), jobs.end(), [](const Pending &x, const Pending &y) {
        if (x.kind != y.kind) return x.kind < y.kind;
        if (x.pmax != y.pmax) return x.pmax < y.pmax;
        return x.job.a.R > y.job.a.R;
    });
    std::vector<ManyJob> flat;
    flat.reserve(jobs.size());
    for (size_t i = 0; i < jobs.size();) {
        pp_many::Group g{jobs[i].kind, jobs[i].pmax, (int)i, 0, 1, 0, 0};
        size_t end = i;
        int64_t widest = 1;
        for (; end < jobs.size() && jobs[end].kind == g.kind && jobs[end].pmax == g.pmax; ++end) {
            const EvalArgs &a = jobs[end].job.a;
            widest = std::max(widest, g.kind == 0 ? reg_mbz_warps(a) : lane_mbz_warps(g.pmax, a));
        }
        g.warps = (int)std::min<int64_t>(widest, g.kind == 0 ? kManyRegWarps : kManyLaneWarps);
        for (; i < end; ++i) {
            ManyJob j = jobs[i].job;
            j.block_begin = g.ctas;
            const EvalArgs &a = j.a;
            g.ctas += g.kind == 0 ? reg_mbz_ctas(a, g.warps) : lane_mbz_ctas(g.pmax, a, g.warps);
            g.smem = std::max(g.smem, g.kind == 0 ? reg_mbz_smem(g.pmax, a, g.warps)
                                                  : lane_mbz_smem(g.pmax, a, g.warps));
            flat.push_back(j);
            ++g.count;
        }
        if (g.ctas > 0x7FFFFFFF) return PP_ERR_SIZE;
        h->groups.push_back(g);
    }
    if (!flat.empty()) {
        PPS_CUDA_TRY(cudaMalloc(&h->d_jobs, flat.size() * sizeof(ManyJob)));
        PPS_CUDA_TRY(cudaMemcpyAsync(h->d_jobs, flat.data(), flat.size() * sizeof(ManyJob), cudaMemcpyHostToDevice,
                                     stream));
        PPS_CUDA_TRY(cudaStreamSynchronize(stream));
    }
    return PP_OK;
}

// Per device: streams that run the groups of one evaluation side by side
// (one group per stream), with the events that fork them from the caller's
// stream and join them back.  Evaluations on one device enqueue under a
// mutex, so each wait names its own evaluation's record.
constexpr int kMaxGroups = 6;  // 2 kernels x 3 table widths
struct Fork {
    bool ready = false;
    cudaStream_t s[kMaxGroups] = {};
    cudaEvent_t start = nullptr, done[kMaxGroups] = {};
};
std::mutex g_fork_mu;
Fork g_fork[64];

int fork_for_device(int dev, Fork **out) {
    if (dev < 0 || dev >= 64) return PP_ERR_INTERNAL;
    Fork &f = g_fork[dev];
    if (!f.ready) {
        for (int i = 0; i < kMaxGroups; ++i) {
            PPS_CUDA_TRY(cudaStreamCreateWithFlags(&f.s[i], cudaStreamNonBlocking));
            PPS_CUDA_TRY(cudaEventCreateWithFlags(&f.done[i], cudaEventDisableTiming));
        }
        PPS_CUDA_TRY(cudaEventCreateWithFlags(&f.start, cudaEventDisableTiming));
        f.ready = true;
    }
    *out = &f;
    return PP_OK;
}

int launch_group(const pp_many &m, const pp_many::Group &g, cudaStream_t st) {
    const ManyJob *d = m.d_jobs + g.first;
    return g.kind == 0 ? launch_reg_mbz_many(g.pmax, g.warps, d, g.count, g.ctas, g.smem, st)
                       : launch_lane_mbz_many(g.pmax, g.warps, d, g.count, g.ctas, g.smem, st);
}

// The fused launches: one group on `stream`, several side by side on the
// device's group streams, forked from and joined back into `stream`.
int launch_groups(const pp_many &m, cudaStream_t stream) {
    const int ng = (int)m.groups.size();
    if (ng == 0) return PP_OK;
    if (ng == 1) return launch_group(m, m.groups[0], stream);
    if (ng > kMaxGroups) return PP_ERR_INTERNAL;
    std::lock_guard<std::mutex> lk(g_fork_mu);
    Fork *f = nullptr;
    int rc = fork_for_device(m.device, &f);
    if (rc) return rc;
    PPS_CUDA_TRY(cudaEventRecord(f->start, stream));
    for (int i = 0; i < ng && !rc; ++i) {
        PPS_CUDA_TRY(cudaStreamWaitEvent(f->s[i], f->start, 0));
        rc = launch_group(m, m.groups[i], f->s[i]);
        PPS_CUDA_TRY(cudaEventRecord(f->done[i], f->s[i]));
    }
    // joined also after an error, so that nothing is left unordered
    for (int i = 0; i < ng; ++i) PPS_CUDA_TRY(cudaStreamWaitEvent(stream, f->done[i], 0));
    return rc;
}

}  // namespace
}  // namespace pps

extern "C" int pp_sched_many_prepare(const pp_problem_t *problems, int n_problems, pp_many_t **many,
                                     cudaStream_t stream) {
    using namespace pps;
    if (!many) return PP_ERR_ARG;
    *many = nullptr;
    if (n_problems < 0 || (n_problems > 0 && !problems)) return PP_ERR_ARG;
    // argument errors first, before any CUDA call
    for (int i = 0; i < n_problems; ++i) {
        const pp_problem_t &p = problems[i];
        const int rc = eval_check(p.policy, p.P, p.M, p.v, p.cost_f, p.cost_b, p.stride_inst, p.stride_stage,
                                  p.stride_mb, p.comm_stride_inst, p.comm_stride_bnd, p.n_instances);
        if (rc) return rc;
    }
    pp_many *h = new pp_many;
    const cudaError_t e = cudaGetDevice(&h->device);
    int rc = e == cudaSuccess ? PP_OK : cuda_status(e);
    if (!rc) rc = prepare(problems, n_problems, h, stream);
    if (rc) {
        pp_sched_many_destroy(h);
        return rc;
    }
    *many = h;
    return PP_OK;
}

extern "C" int pp_sched_many_eval(const pp_many_t *many, cudaStream_t stream) {
    using namespace pps;
    if (!many) return PP_ERR_ARG;
    int dev = 0;
    PPS_CUDA_TRY(cudaGetDevice(&dev));
    if (dev != many->device) return PP_ERR_ARG;
    const int rc = launch_groups(*many, stream);
    if (rc) return rc;
    for (const pp_problem_t &p : many->rest) {
        const int rc = pp_sched_eval(p.policy, p.P, p.M, p.v, p.cost_f, p.cost_b, p.stride_inst, p.stride_stage,
                                     p.stride_mb, p.comm, p.comm_stride_inst, p.comm_stride_bnd, p.n_instances,
                                     p.makespan, p.idle, p.bub_num, p.bub_den, p.peak, nullptr, nullptr, 0, 0,
                                     p.status, stream);
        if (rc) return rc;
    }
    return PP_OK;
}

extern "C" int pp_sched_many_info(const pp_many_t *many, int *fused_problems, int *launches, int *other_problems) {
    if (!many) return PP_ERR_ARG;
    int fused = 0;
    for (const pp_many::Group &g : many->groups) fused += g.count;
    if (fused_problems) *fused_problems = fused;
    if (launches) *launches = (int)many->groups.size();
    if (other_problems) *other_problems = (int)many->rest.size();
    return PP_OK;
}

extern "C" void pp_sched_many_destroy(pp_many_t *many) {
    if (!many) return;
    if (many->d_jobs) cudaFree(many->d_jobs);
    delete many;
}
