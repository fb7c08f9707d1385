// host.cpp -- the host-only entry points (layout, accounting, waits, error
// names) and the helpers the launch wrappers share.
#include <chrono>
#include <cmath>
#include <cstring>
#include <mutex>
#include <thread>

#include "zero_internal.h"

namespace zero {

bool valid_hparams(const zero_hparams_t* hp)
{
    if (!hp || hp->step < 1) return false;
    const double v[5] = {hp->lr, hp->beta1, hp->beta2, hp->eps, hp->weight_decay};
    for (double x : v)
        if (!std::isfinite(x)) return false;
    return hp->lr >= 0 && hp->beta1 >= 0 && hp->beta1 < 1 && hp->beta2 >= 0 &&
           hp->beta2 < 1 && hp->eps > 0 && hp->weight_decay >= 0;
}

StepScalars make_scalars(const zero_hparams_t* hp, int32_t n_ranks)
{
    const double t = static_cast<double>(hp->step);
    StepScalars s;
    s.b1 = static_cast<float>(hp->beta1);
    s.b2 = static_cast<float>(hp->beta2);
    s.omb1 = static_cast<float>(1.0 - hp->beta1);
    s.omb2 = static_cast<float>(1.0 - hp->beta2);
    s.bc1 = static_cast<float>(1.0 - std::pow(hp->beta1, t));
    s.bc2 = static_cast<float>(1.0 - std::pow(hp->beta2, t));
    s.lr = static_cast<float>(hp->lr);
    s.eps = static_cast<float>(hp->eps);
    s.wd = static_cast<float>(hp->weight_decay);
    s.inv_n = static_cast<float>(1.0 / static_cast<double>(n_ranks));
    return s;
}

int cuda_status(cudaError_t e) { return e == cudaSuccess ? ZERO_OK : ZERO_ECUDA; }

namespace {
struct GeomEntry {
    int device;
    const void* kernel;
    int block;
    size_t smem;
    int blocks;
};
std::mutex g_geom_mu;
GeomEntry g_geom[256];
int g_geom_n = 0;
} // namespace

int persistent_blocks(const void* kernel, int block_threads, size_t dyn_smem)
{
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return -1;
    {
        std::lock_guard<std::mutex> lk(g_geom_mu);
        for (int i = 0; i < g_geom_n; ++i)
            if (g_geom[i].device == dev && g_geom[i].kernel == kernel &&
                g_geom[i].block == block_threads && g_geom[i].smem == dyn_smem)
                return g_geom[i].blocks;
    }
    int sms = 0, per_sm = 0;
    if (cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
        return -1;
    if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, kernel, block_threads,
                                                      dyn_smem) != cudaSuccess)
        return -1;
    if (per_sm < 1) per_sm = 1;
    const int blocks = sms * per_sm;
    std::lock_guard<std::mutex> lk(g_geom_mu);
    if (g_geom_n < 256) g_geom[g_geom_n++] = {dev, kernel, block_threads, dyn_smem, blocks};
    return blocks;
}

} // namespace zero

using namespace zero;

extern "C" int zero_layout(const int64_t* unit_sizes, int32_t n_units, int32_t n_ranks,
                           int32_t align_elems, zero_unit_t* out_units,
                           int64_t* out_total_padded)
{
    if (!unit_sizes || !out_units || !out_total_padded || n_units < 1 || n_ranks < 1 ||
        n_ranks > ZERO_MAX_RANKS || align_elems < 1 || align_elems % 8 != 0)
        return ZERO_EINVAL;
    const int64_t granule = static_cast<int64_t>(n_ranks) * align_elems;
    int64_t padded_so_far = 0, params_so_far = 0;
    for (int32_t u = 0; u < n_units; ++u) {
        const int64_t p = unit_sizes[u];
        if (p <= 0 || p > INT64_MAX / 4 - granule) return ZERO_EINVAL;
        const int64_t padded = ((p + granule - 1) / granule) * granule;
        zero_unit_t& U = out_units[u];
        U.n_params = p;
        U.n_padded = padded;
        U.shard_len = padded / n_ranks;
        U.offset = padded_so_far;
        U.shard_offset = padded_so_far / n_ranks;
        U.param_offset = params_so_far;
        U.pad = padded - p;
        padded_so_far += padded;
        params_so_far += p;
    }
    *out_total_padded = padded_so_far;
    return ZERO_OK;
}

extern "C" int zero_state_bytes(int64_t n_params, int32_t n_ranks, int32_t stage, int32_t K,
                                zero_bytes_t* out)
{
    if (!out || n_params <= 0 || n_ranks < 1 || stage < 0 || stage > 3 || K < 0)
        return ZERO_EINVAL;
    const double P = static_cast<double>(n_params);
    const double N = static_cast<double>(n_ranks);
    // Which of (optimizer state, gradients, weights) are divided by N.
    const bool shard_opt = stage >= 1, shard_grad = stage >= 2, shard_w = stage >= 3;
    zero_bytes_t b;
    b.weight_bytes = shard_w ? 2.0 * P / N : 2.0 * P;
    b.grad_bytes = shard_grad ? 2.0 * P / N : 2.0 * P;
    b.optim_bytes = shard_opt ? K * P / N : K * P;
    b.state_bytes = b.weight_bytes + b.grad_bytes + b.optim_bytes;
    // DDP's all-reduce is a reduce-scatter plus an all-gather (2P); ZeRO-1/2
    // keep that volume; ZeRO-3 adds the second (backward) all-gather (3P).
    b.comm_volume = (stage == 3 ? 3.0 : 2.0) * P;
    b.comm_sent_elems = b.comm_volume * (N - 1.0) / N;
    b.comm_sent_bytes = 2.0 * b.comm_sent_elems;
    b.hbm_bytes = (26.0 + 2.0 * N) * P + (stage == 3 ? 8.0 * P : 0.0);
    *out = b;
    return ZERO_OK;
}

extern "C" int zero_stream_wait(cudaStream_t stream, int64_t timeout_ms)
{
    if (timeout_ms < 0) return ZERO_EINVAL;
    const auto start = std::chrono::steady_clock::now();
    for (;;) {
        cudaError_t e = cudaStreamQuery(stream);
        if (e == cudaSuccess) return ZERO_OK;
        if (e != cudaErrorNotReady) return ZERO_ECUDA;
        const auto waited = std::chrono::duration_cast<std::chrono::milliseconds>(
            std::chrono::steady_clock::now() - start);
        if (waited.count() >= timeout_ms) return ZERO_ETIMEOUT;
        std::this_thread::sleep_for(std::chrono::microseconds(50));
    }
}

extern "C" const char* zero_strerror(int code)
{
    switch (code) {
    case ZERO_OK: return "ok";
    case ZERO_EINVAL: return "invalid argument";
    case ZERO_EALIGN: return "device pointer not 16-byte aligned";
    case ZERO_ECUDA: return "CUDA runtime error";
    case ZERO_ETIMEOUT: return "timed out waiting for the stream";
    default: return "unknown error";
    }
}
