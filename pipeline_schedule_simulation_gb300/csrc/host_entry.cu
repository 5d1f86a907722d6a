// host_entry.cu -- pp_sched_eval_host: the evaluation from HOST buffers.
//
// For callers whose cost tables live in host memory: the call copies a chunk
// of instances to a caller-provided device workspace (the instance-minor rows
// of the chunk, one 2D copy per table), evaluates it with pp_sched_eval and
// copies the chunk's results back to host memory, chunk after chunk, all on
// one stream.  The workspace bounds the device memory used; with one chunk the
// call is three copies, one evaluation and the result copies.
#include <algorithm>

#include "internal.cuh"

namespace pps {
namespace {

constexpr size_t kAlign = 256;

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
    // the largest chunk (a multiple of 32 instances, or the whole batch) that fits
    int64_t c = n;
    if (chunk_bytes(c, S, M, P) > work_bytes) {
        int64_t lo = 0, hi = n;
        while (lo < hi) {  // largest c with chunk_bytes(c) <= work_bytes
            const int64_t mid = (lo + hi + 1) / 2;
            if (chunk_bytes(mid, S, M, P) <= work_bytes) lo = mid;
            else hi = mid - 1;
        }
        c = lo / 32 * 32;
        if (c == 0) return PP_ERR_SIZE;
    }
    const int64_t cp = pitch_of(c);
    unsigned char *w = static_cast<unsigned char *>(d_work);
    int32_t *df = reinterpret_cast<int32_t *>(w);
    w += align_up((size_t)S * M * cp * 4);
    int32_t *db = reinterpret_cast<int32_t *>(w);
    w += align_up((size_t)S * M * cp * 4);
    int32_t *dc = reinterpret_cast<int32_t *>(w);
    w += align_up((size_t)std::max(S - 1, 1) * cp * 4);
    int32_t *dmk = reinterpret_cast<int32_t *>(w);
    w += align_up((size_t)c * 4);
    int32_t *didle = reinterpret_cast<int32_t *>(w);
    w += align_up((size_t)c * P * 4);
    int64_t *dbn = reinterpret_cast<int64_t *>(w);
    w += align_up((size_t)c * 8);
    int64_t *dbd = reinterpret_cast<int64_t *>(w);
    w += align_up((size_t)c * 8);
    int8_t *dst = reinterpret_cast<int8_t *>(w);
    w += align_up((size_t)c);
    int32_t *dpeak = reinterpret_cast<int32_t *>(w);

    for (int64_t c0 = 0; c0 < n; c0 += c) {
        const int64_t nc = std::min(c, n - c0);
        // rows of the chunk: [S*M][nc] out of [S*M][n] (instance-minor)
        PPS_CUDA_TRY(cudaMemcpy2DAsync(df, cp * 4, h_cost_f + c0, n * 4, nc * 4, (size_t)S * M,
                                       cudaMemcpyHostToDevice, stream));
        PPS_CUDA_TRY(cudaMemcpy2DAsync(db, cp * 4, h_cost_b + c0, n * 4, nc * 4, (size_t)S * M,
                                       cudaMemcpyHostToDevice, stream));
        if (h_comm && S > 1)
            PPS_CUDA_TRY(cudaMemcpy2DAsync(dc, cp * 4, h_comm + c0, n * 4, nc * 4, (size_t)(S - 1),
                                           cudaMemcpyHostToDevice, stream));
        rc = pp_sched_eval(policy, P, M, v, df, db, 1, (int64_t)M * cp, cp, h_comm ? dc : nullptr, 1, cp, nc,
                           h_makespan ? dmk : nullptr, h_idle ? didle : nullptr, h_bub_num ? dbn : nullptr,
                           h_bub_den ? dbd : nullptr, (h_peak && c0 == 0) ? dpeak : nullptr, nullptr, nullptr, 0, 0,
                           h_status ? dst : nullptr, stream);
        if (rc) return rc;
        if (h_makespan)
            PPS_CUDA_TRY(cudaMemcpyAsync(h_makespan + c0, dmk, nc * 4, cudaMemcpyDeviceToHost, stream));
        if (h_idle)
            PPS_CUDA_TRY(cudaMemcpyAsync(h_idle + c0 * P, didle, nc * P * 4, cudaMemcpyDeviceToHost, stream));
        if (h_bub_num)
            PPS_CUDA_TRY(cudaMemcpyAsync(h_bub_num + c0, dbn, nc * 8, cudaMemcpyDeviceToHost, stream));
        if (h_bub_den)
            PPS_CUDA_TRY(cudaMemcpyAsync(h_bub_den + c0, dbd, nc * 8, cudaMemcpyDeviceToHost, stream));
        if (h_status) PPS_CUDA_TRY(cudaMemcpyAsync(h_status + c0, dst, nc, cudaMemcpyDeviceToHost, stream));
        if (h_peak && c0 == 0)
            PPS_CUDA_TRY(cudaMemcpyAsync(h_peak, dpeak, P * sizeof(int32_t), cudaMemcpyDeviceToHost, stream));
    }
    return PP_OK;
}

extern "C" size_t pp_sched_eval_host_workspace(int P, int M, int v, int64_t n_instances) {
    if (P < 1 || M < 1 || v < 1 || n_instances < 0) return 0;
    return pps::chunk_bytes(std::max<int64_t>(n_instances, 1), P * v, M, P);
}
