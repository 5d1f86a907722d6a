// host_entry.cu -- pp_sched_eval_host: the evaluation from HOST buffers.
//
// For callers whose cost tables live in host memory: the call copies a chunk
// of instances to a caller-provided device workspace (the instance-minor rows
// of the chunk, one 2D copy per table), evaluates it with pp_sched_eval and
// copies the chunk's results back to host memory.
//
// When the workspace holds two chunk slots, the batch is cut into about
// kPipeChunks chunks and the work runs on two streams: the caller's stream
// copies chunk i+1 in while an auxiliary stream of the library evaluates
// chunk i and copies its results out, so the evaluation and the result copies
// hide under the input copies (the host link is the bound).  Events order the
// slots' reuse, and the caller's stream finally waits for the auxiliary one,
// so the call is still ordered on `stream` alone.  With room for one slot only,
// chunks run one after another on `stream`.
#include <algorithm>
#include <mutex>
#include <vector>

#include "checks.cuh"
#include "internal.cuh"

namespace pps {
namespace {

constexpr size_t kAlign = 256;
// Chunks per batch in the two-slot pipeline: fewer leave more of the first
// copy and the last evaluation uncovered; more make the 2D copies' rows short
// (measured on the 65,536-instance 1F1B batch: 2, 4, 8, 16 chunks took 1.40,
// 1.36, 1.38, 1.45 ms per call against 1.40 ms in one chunk).
constexpr int64_t kPipeChunks = 4;

size_t align_up(size_t x) { return (x + kAlign - 1) / kAlign * kAlign; }

// Device row pitch of a chunk of c instances: a multiple of 32 instances, so
// the rows start on 128-byte boundaries and the vector loaders apply.
int64_t pitch_of(int64_t c) { return (c + 31) / 32 * 32; }

// Workspace bytes for a chunk of c instances.
size_t chunk_bytes(int64_t c, int S, int M, int P) {
    const int64_t cp = pitch_of(c);
    return align_up((size_t)S * M * cp * 4) * 2 + align_up((size_t)std::max(S - 1, 1) * cp * 4) +
           align_up((size_t)c * 4) + align_up((size_t)c * P * 4) + 2 * align_up((size_t)c * 8) + align_up((size_t)c) +
           align_up((size_t)P * 4);
}

// Largest chunk (a multiple of 32 instances, at most `cap`) of which `slots`
// fit in `work_bytes`; 0 if not even 32 instances fit.
int64_t fit_chunk(int64_t cap, int slots, size_t work_bytes, int S, int M, int P) {
    int64_t lo = 0, hi = cap;
    while (lo < hi) {
        const int64_t mid = (lo + hi + 1) / 2;
        if ((size_t)slots * chunk_bytes(mid, S, M, P) <= work_bytes) lo = mid;
        else hi = mid - 1;
    }
    return lo >= cap ? cap : lo / 32 * 32;
}

// One chunk's device buffers, carved from the workspace.
struct Slot {
    int32_t *df, *db, *dc, *dmk, *didle, *dpeak;
    int64_t *dbn, *dbd;
    int8_t *dst;
};

Slot carve(unsigned char *w, int64_t c, int S, int M, int P) {
    const int64_t cp = pitch_of(c);
    Slot sl;
    sl.df = reinterpret_cast<int32_t *>(w);
    w += align_up((size_t)S * M * cp * 4);
    sl.db = reinterpret_cast<int32_t *>(w);
    w += align_up((size_t)S * M * cp * 4);
    sl.dc = reinterpret_cast<int32_t *>(w);
    w += align_up((size_t)std::max(S - 1, 1) * cp * 4);
    sl.dmk = reinterpret_cast<int32_t *>(w);
    w += align_up((size_t)c * 4);
    sl.didle = reinterpret_cast<int32_t *>(w);
    w += align_up((size_t)c * P * 4);
    sl.dbn = reinterpret_cast<int64_t *>(w);
    w += align_up((size_t)c * 8);
    sl.dbd = reinterpret_cast<int64_t *>(w);
    w += align_up((size_t)c * 8);
    sl.dst = reinterpret_cast<int8_t *>(w);
    w += align_up((size_t)c);
    sl.dpeak = reinterpret_cast<int32_t *>(w);
    return sl;
}

// The host arguments of one call.
struct HostIO {
    pp_policy_t policy;
    int P, M, v, S;
    int64_t n;
    const int32_t *h_cost_f, *h_cost_b, *h_comm;
    int32_t *h_makespan, *h_idle, *h_peak;
    int64_t *h_bub_num, *h_bub_den;
    int8_t *h_status;
};

// Copies of chunk [c0, c0 + nc) into a slot of pitch cp, on `st`.
int copy_in(const HostIO &io, const Slot &sl, int64_t cp, int64_t c0, int64_t nc, cudaStream_t st) {
    const int64_t n = io.n;
    // rows of the chunk: [S*M][nc] out of [S*M][n] (instance-minor)
    PPS_CUDA_TRY(cudaMemcpy2DAsync(sl.df, cp * 4, io.h_cost_f + c0, n * 4, nc * 4, (size_t)io.S * io.M,
                                   cudaMemcpyHostToDevice, st));
    PPS_CUDA_TRY(cudaMemcpy2DAsync(sl.db, cp * 4, io.h_cost_b + c0, n * 4, nc * 4, (size_t)io.S * io.M,
                                   cudaMemcpyHostToDevice, st));
    if (io.h_comm && io.S > 1)
        PPS_CUDA_TRY(cudaMemcpy2DAsync(sl.dc, cp * 4, io.h_comm + c0, n * 4, nc * 4, (size_t)(io.S - 1),
                                       cudaMemcpyHostToDevice, st));
    return PP_OK;
}

// Evaluation of the chunk in a slot and the copies of its results, on `st`.
int eval_out(const HostIO &io, const Slot &sl, int64_t cp, int64_t c0, int64_t nc, cudaStream_t st) {
    const int P = io.P;
    const bool first = c0 == 0;
    int rc = pp_sched_eval(io.policy, P, io.M, io.v, sl.df, sl.db, 1, (int64_t)io.M * cp, cp,
                           io.h_comm ? sl.dc : nullptr, 1, cp, nc, io.h_makespan ? sl.dmk : nullptr,
                           io.h_idle ? sl.didle : nullptr, io.h_bub_num ? sl.dbn : nullptr,
                           io.h_bub_den ? sl.dbd : nullptr, (io.h_peak && first) ? sl.dpeak : nullptr, nullptr,
                           nullptr, 0, 0, io.h_status ? sl.dst : nullptr, st);
    if (rc) return rc;
    if (io.h_makespan)
        PPS_CUDA_TRY(cudaMemcpyAsync(io.h_makespan + c0, sl.dmk, nc * 4, cudaMemcpyDeviceToHost, st));
    if (io.h_idle)
        PPS_CUDA_TRY(cudaMemcpyAsync(io.h_idle + c0 * P, sl.didle, nc * P * 4, cudaMemcpyDeviceToHost, st));
    if (io.h_bub_num)
        PPS_CUDA_TRY(cudaMemcpyAsync(io.h_bub_num + c0, sl.dbn, nc * 8, cudaMemcpyDeviceToHost, st));
    if (io.h_bub_den)
        PPS_CUDA_TRY(cudaMemcpyAsync(io.h_bub_den + c0, sl.dbd, nc * 8, cudaMemcpyDeviceToHost, st));
    if (io.h_status) PPS_CUDA_TRY(cudaMemcpyAsync(io.h_status + c0, sl.dst, nc, cudaMemcpyDeviceToHost, st));
    if (io.h_peak && first)
        PPS_CUDA_TRY(cudaMemcpyAsync(io.h_peak, sl.dpeak, P * sizeof(int32_t), cudaMemcpyDeviceToHost, st));
    return PP_OK;
}

// Per device: the auxiliary stream and the events of the two-slot pipeline.
// Calls on one device enqueue under a mutex, so each wait names the record
// of its own call.
struct Pipe {
    bool ready = false;
    cudaStream_t aux = nullptr;
    cudaEvent_t start = nullptr, done = nullptr, in[2] = {}, freed[2] = {};
};
constexpr int kMaxDev = 64;
std::mutex g_pipe_mu;
Pipe g_pipe[kMaxDev];

int pipe_for_current_device(Pipe **out) {
    int dev = 0;
    PPS_CUDA_TRY(cudaGetDevice(&dev));
    if (dev < 0 || dev >= kMaxDev) return PP_ERR_INTERNAL;
    Pipe &p = g_pipe[dev];
    if (!p.ready) {
        PPS_CUDA_TRY(cudaStreamCreateWithFlags(&p.aux, cudaStreamNonBlocking));
        cudaEvent_t *evs[] = {&p.start, &p.done, &p.in[0], &p.in[1], &p.freed[0], &p.freed[1]};
        for (cudaEvent_t *e : evs) PPS_CUDA_TRY(cudaEventCreateWithFlags(e, cudaEventDisableTiming));
        p.ready = true;
    }
    *out = &p;
    return PP_OK;
}

// The two-slot pipeline over chunks of c instances (see the file comment).
int run_pipelined(const HostIO &io, unsigned char *w, int64_t c, cudaStream_t st) {
    std::lock_guard<std::mutex> lk(g_pipe_mu);
    Pipe *p = nullptr;
    int rc = pipe_for_current_device(&p);
    if (rc) return rc;
    const int64_t cp = pitch_of(c);
    const Slot slots[2] = {carve(w, c, io.S, io.M, io.P), carve(w + align_up(chunk_bytes(c, io.S, io.M, io.P)), c,
                                                                io.S, io.M, io.P)};
    // the auxiliary stream starts after the caller's earlier work
    PPS_CUDA_TRY(cudaEventRecord(p->start, st));
    PPS_CUDA_TRY(cudaStreamWaitEvent(p->aux, p->start, 0));
    int64_t i = 0;
    for (int64_t c0 = 0; c0 < io.n && !rc; c0 += c, ++i) {
        const int64_t nc = std::min(c, io.n - c0);
        const int k = (int)(i & 1);
        // the slot's previous chunk (i - 2) has been evaluated and copied out
        if (i >= 2) PPS_CUDA_TRY(cudaStreamWaitEvent(st, p->freed[k], 0));
        rc = copy_in(io, slots[k], cp, c0, nc, st);
        if (rc) break;
        PPS_CUDA_TRY(cudaEventRecord(p->in[k], st));
        PPS_CUDA_TRY(cudaStreamWaitEvent(p->aux, p->in[k], 0));
        rc = eval_out(io, slots[k], cp, c0, nc, p->aux);
        if (rc) break;
        PPS_CUDA_TRY(cudaEventRecord(p->freed[k], p->aux));
    }
    // the call ends on the caller's stream, also after an error
    PPS_CUDA_TRY(cudaEventRecord(p->done, p->aux));
    PPS_CUDA_TRY(cudaStreamWaitEvent(st, p->done, 0));
    return rc;
}

}  // namespace
}  // namespace pps

extern "C" int pp_sched_eval_host(pp_policy_t policy, int P, int M, int v, const int32_t *h_cost_f,
                                  const int32_t *h_cost_b, const int32_t *h_comm, int64_t n_instances,
                                  void *d_work, size_t work_bytes, int32_t *h_makespan, int32_t *h_idle,
                                  int64_t *h_bub_num, int64_t *h_bub_den, int32_t *h_peak, int8_t *h_status,
                                  cudaStream_t stream) {
    using namespace pps;
    int rc = check_shape((int)policy, P, M, v);
    if (rc) return rc;
    if (n_instances < 0) return PP_ERR_ARG;
    if (n_instances > 0 && (!h_cost_f || !h_cost_b || !d_work)) return PP_ERR_ARG;
    if ((reinterpret_cast<uintptr_t>(d_work) & (kAlign - 1)) != 0) return PP_ERR_ARG;
    const int S = P * v;
    const int64_t n = n_instances;
    if (n == 0) {
        if (h_peak) {
            // the peaks need the plan, not the costs
            if (work_bytes < align_up((size_t)P * 4) || !d_work) return PP_ERR_SIZE;
            int32_t *d_peak = static_cast<int32_t *>(d_work);
            rc = pp_sched_eval(policy, P, M, v, nullptr, nullptr, 0, 0, 0, nullptr, 0, 0, 0, nullptr, nullptr, nullptr,
                               nullptr, d_peak, nullptr, nullptr, 0, 0, nullptr, stream);
            if (rc) return rc;
            PPS_CUDA_TRY(cudaMemcpyAsync(h_peak, d_peak, P * sizeof(int32_t), cudaMemcpyDeviceToHost, stream));
        }
        return PP_OK;
    }
    const HostIO io{policy, P, M, v, S, n, h_cost_f, h_cost_b, h_comm, h_makespan, h_idle, h_peak,
                    h_bub_num, h_bub_den, h_status};
    unsigned char *w = static_cast<unsigned char *>(d_work);
    // two slots of about n / kPipeChunks instances, when the batch gives at
    // least two chunks and the workspace holds both slots
    const int64_t c2 = fit_chunk(pitch_of((n + kPipeChunks - 1) / kPipeChunks), 2, work_bytes, S, M, P);
    if (c2 > 0 && c2 < n) return run_pipelined(io, w, c2, stream);
    // one slot: the whole batch if it fits, else chunks one after another
    const int64_t c = chunk_bytes(n, S, M, P) <= work_bytes ? n : fit_chunk(n, 1, work_bytes, S, M, P);
    if (c == 0) return PP_ERR_SIZE;
    const Slot sl = carve(w, c, S, M, P);
    const int64_t cp = pitch_of(c);
    for (int64_t c0 = 0; c0 < n; c0 += c) {
        const int64_t nc = std::min(c, n - c0);
        rc = copy_in(io, sl, cp, c0, nc, stream);
        if (rc) return rc;
        rc = eval_out(io, sl, cp, c0, nc, stream);
        if (rc) return rc;
    }
    return PP_OK;
}

extern "C" size_t pp_sched_eval_host_workspace(int P, int M, int v, int64_t n_instances) {
    if (P < 1 || M < 1 || v < 1 || n_instances < 0) return 0;
    return pps::chunk_bytes(std::max<int64_t>(n_instances, 1), P * v, M, P);
}

// ---- the bounds-checked build's failure records ----

namespace pps {
namespace {
std::mutex g_check_mu;
std::vector<uint64_t (*)()> &check_readers() {
    static std::vector<uint64_t (*)()> readers;
    return readers;
}
}  // namespace

int register_check_reader(uint64_t (*reader)()) {
    std::lock_guard<std::mutex> lk(g_check_mu);
    check_readers().push_back(reader);
    return 0;
}
}  // namespace pps

extern "C" int pp_sched_debug_checks(uint64_t *first_failure) {
    uint64_t first = 0;
#ifdef PPS_CHECKED
    std::lock_guard<std::mutex> lk(pps::g_check_mu);
    for (uint64_t (*reader)() : pps::check_readers()) {
        const uint64_t w = reader();
        if (!first) first = w;
    }
    if (first_failure) *first_failure = first;
    return 1;
#else
    if (first_failure) *first_failure = first;
    return 0;
#endif
}
