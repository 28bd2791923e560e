// RoPE cos/sin table: built on the host in float64, stored on the device as
// float2 [max_positions][rotary_dim/2] = (mu cos(P w_j), mu sin(P w_j)).
//
// "RoPE, scaling, sliding window, attention sinks": the table of shape
// [max_position_embeddings, r] built once (section on RoPE), the YaRN frequency
// blend and mscale ("YaRN, precisely").  "#2961 rope: --rope-scaling dynamic":
// the table is rebuilt in place on host threads, bit for bit the single-thread
// build, so a captured CUDA graph keeps its pointer.
#include <algorithm>
#include <cmath>
#include <thread>
#include <vector>

#include "common.cuh"

struct sk_rope_table {
    sk_rope_config cfg;
    float2* d_table = nullptr;      // device, library-owned
    std::vector<float2> host;       // host copy of the table
};

namespace {

// Frequencies of the r/2 rotary pairs.  Plain RoPE: w_i = theta^(-2i/r).  YaRN
// (factor s > 1): the correction band [low, high] from the pair index at which a
// pair turns beta times in L0 tokens, d(beta) = r ln(L0 / (2 pi beta)) / (2 ln theta),
// low = max(floor d(beta_fast), 0), high = min(ceil d(beta_slow), r - 1); a linear
// ramp over the band (high nudged by 0.001 when equal to low); pairs below the band
// keep w_i, pairs above get w_i / s, the band interpolates linearly.
std::vector<double> pair_frequencies(const sk_rope_config& c, double factor) {
    const int half = c.rotary_dim / 2;
    std::vector<double> w(half);
    for (int i = 0; i < half; ++i)
        w[i] = 1.0 / std::pow(c.theta, (2.0 * i) / c.rotary_dim);
    if (factor <= 1.0) return w;
    const double two_pi = 6.283185307179586476925286766559;
    auto corr_dim = [&](double beta) {
        return c.rotary_dim * std::log(double(c.yarn_orig_ctx) / (beta * two_pi)) /
               (2.0 * std::log(c.theta));
    };
    double low = std::max(std::floor(corr_dim(c.beta_fast)), 0.0);
    double high = std::min(std::ceil(corr_dim(c.beta_slow)), double(c.rotary_dim - 1));
    if (low == high) high += 0.001;
    for (int i = 0; i < half; ++i) {
        double ramp = (double(i) - low) / (high - low);
        ramp = std::min(1.0, std::max(0.0, ramp));
        // weight of the interpolated frequency is the ramp, of the original 1 - ramp
        w[i] = (w[i] / factor) * ramp + w[i] * (1.0 - ramp);
    }
    return w;
}

double attention_mscale(double factor) {
    return factor <= 1.0 ? 1.0 : 0.1 * std::log(factor) + 1.0;
}

// Fill table rows [p_begin, p_end).  Each entry depends only on (P, j), so any split
// of the rows over threads gives the same bits.
void fill_rows(std::vector<float2>& out, const std::vector<double>& w, double mu, int64_t p_begin,
               int64_t p_end) {
    const int half = int(w.size());
    for (int64_t p = p_begin; p < p_end; ++p) {
        float2* row = out.data() + p * half;
        for (int j = 0; j < half; ++j) {
            const double a = double(p) * w[j];
            row[j] = make_float2(float(mu * std::cos(a)), float(mu * std::sin(a)));
        }
    }
}

void build_host_table(sk_rope_table* t) {
    const sk_rope_config& c = t->cfg;
    const std::vector<double> w = pair_frequencies(c, c.yarn_factor);
    const double mu = attention_mscale(c.yarn_factor);
    t->host.resize(size_t(c.max_positions) * (c.rotary_dim / 2));
    unsigned n_threads = std::max(1u, std::min(32u, std::thread::hardware_concurrency()));
    if (c.max_positions < 4096) n_threads = 1;
    std::vector<std::thread> pool;
    for (unsigned i = 0; i < n_threads; ++i) {
        const int64_t b = c.max_positions * i / n_threads;
        const int64_t e = c.max_positions * (i + 1) / n_threads;
        pool.emplace_back(fill_rows, std::ref(t->host), std::cref(w), mu, b, e);
    }
    for (auto& th : pool) th.join();
}

bool config_ok(const sk_rope_config& c) {
    if (c.head_dim != 64 && c.head_dim != 128) return false;
    if (c.rotary_dim < 16 || c.rotary_dim > c.head_dim || c.rotary_dim % 16 != 0) return false;
    if (!(c.theta > 1.0) || c.max_positions < 1) return false;
    if (c.yarn_factor > 1.0) {
        if (c.yarn_orig_ctx < 1 || !(c.beta_fast > 0.0) || !(c.beta_slow > 0.0)) return false;
    }
    return true;
}

sk_status upload(sk_rope_table* t, cudaStream_t stream) {
    const size_t bytes = t->host.size() * sizeof(float2);
    SK_CUDA_RET(cudaMemcpyAsync(t->d_table, t->host.data(), bytes, cudaMemcpyHostToDevice, stream));
    SK_CUDA_RET(cudaStreamSynchronize(stream));
    return SK_OK;
}

}  // namespace

extern "C" sk_status sk_rope_table_create(const sk_rope_config* cfg, void* stream,
                                          sk_rope_table** out) {
    SK_RET_IF(cfg == nullptr || out == nullptr, SK_ERR_ARG);
    *out = nullptr;
    SK_RET_IF(!config_ok(*cfg), SK_ERR_ARG);
    sk_rope_table* t = new sk_rope_table();
    t->cfg = *cfg;
    build_host_table(t);
    const size_t bytes = t->host.size() * sizeof(float2);
    if (cudaMalloc(&t->d_table, bytes) != cudaSuccess) {
        delete t;
        return SK_ERR_CUDA;
    }
    sk_status s = upload(t, static_cast<cudaStream_t>(stream));
    if (s != SK_OK) {
        cudaFree(t->d_table);
        delete t;
        return s;
    }
    *out = t;
    return SK_OK;
}

extern "C" sk_status sk_rope_table_rebuild(sk_rope_table* t, double new_yarn_factor, void* stream) {
    SK_RET_IF(t == nullptr, SK_ERR_ARG);
    sk_rope_config c = t->cfg;
    c.yarn_factor = new_yarn_factor;
    SK_RET_IF(!config_ok(c), SK_ERR_ARG);
    t->cfg = c;
    build_host_table(t);
    return upload(t, static_cast<cudaStream_t>(stream));
}

extern "C" void sk_rope_table_destroy(sk_rope_table* t) {
    if (t == nullptr) return;
    if (t->d_table != nullptr) cudaFree(t->d_table);
    delete t;
}

extern "C" sk_status sk_rope_table_info(const sk_rope_table* t, sk_rope_config* cfg_out,
                                        const void** device_cos_sin) {
    SK_RET_IF(t == nullptr, SK_ERR_ARG);
    if (cfg_out != nullptr) *cfg_out = t->cfg;
    if (device_cos_sin != nullptr) *device_cos_sin = t->d_table;
    return SK_OK;
}

// Accessors used by the kernels' entry points in other translation units.
namespace sk {
const float2* table_device(const sk_rope_table* t) { return t->d_table; }
const sk_rope_config& table_config(const sk_rope_table* t) { return t->cfg; }
}  // namespace sk
