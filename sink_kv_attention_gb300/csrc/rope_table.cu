// RoPE cos/sin table: built on the host in float64, stored on the device as
// float2 [max_positions][rotary_dim/2] = (mu cos(P w_j), mu sin(P w_j)).  Each entry
// comes from a block anchor and an offset by angle addition (see fill_rows).
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

// Positions are split into blocks of kBlock: P = P0 + k with P0 a multiple of kBlock.
// cos/sin(P w) come from the block's anchor cos/sin(P0 w) and the offset's
// cos/sin(k w) by the angle-addition formulas, in float64: two trigonometric calls
// per block and pair instead of two per entry.  Each entry is a fixed function of
// (P, j), so any split of the rows over threads gives the same bits.
constexpr int64_t kBlock = 64;

struct OffsetTrig {
    std::vector<double> c, s;  // [kBlock][half]: cos, sin of k w_j
};

OffsetTrig offset_trig(const std::vector<double>& w) {
    const int half = int(w.size());
    OffsetTrig t;
    t.c.resize(size_t(kBlock) * half);
    t.s.resize(size_t(kBlock) * half);
    for (int64_t k = 0; k < kBlock; ++k)
        for (int j = 0; j < half; ++j) {
            const double a = double(k) * w[j];
            t.c[k * half + j] = std::cos(a);
            t.s[k * half + j] = std::sin(a);
        }
    return t;
}

// Fill table rows [p_begin, p_end).
void fill_rows(float2* out, const std::vector<double>& w, const OffsetTrig& off, double mu, int64_t p_begin,
               int64_t p_end) {
    const int half = int(w.size());
    std::vector<double> ca(half), sa(half);
    for (int64_t p = p_begin; p < p_end; ++p) {
        const int64_t k = p % kBlock;
        if (p == p_begin || k == 0) {
            const double p0 = double(p - k);
            for (int j = 0; j < half; ++j) {
                const double a = p0 * w[j];
                ca[j] = std::cos(a);
                sa[j] = std::sin(a);
            }
        }
        const double* ck = off.c.data() + k * half;
        const double* sk = off.s.data() + k * half;
        float2* row = out + p * half;
        for (int j = 0; j < half; ++j) {
            const double c = ca[j] * ck[j] - sa[j] * sk[j];
            const double s = sa[j] * ck[j] + ca[j] * sk[j];
            row[j] = make_float2(float(mu * c), float(mu * s));
        }
    }
}

// Fill the whole table for `c` on n_threads host threads (0 = one per core, at most
// 32; small tables use one).
void fill_table(const sk_rope_config& c, unsigned n_threads, float2* out) {
    const std::vector<double> w = pair_frequencies(c, c.yarn_factor);
    const double mu = attention_mscale(c.yarn_factor);
    const OffsetTrig off = offset_trig(w);
    if (n_threads == 0) {
        n_threads = std::max(1u, std::min(32u, std::thread::hardware_concurrency()));
        if (c.max_positions < 4096) n_threads = 1;
    }
    n_threads = unsigned(std::min<int64_t>(n_threads, c.max_positions));
    if (n_threads <= 1) {
        fill_rows(out, w, off, mu, 0, c.max_positions);
        return;
    }
    std::vector<std::thread> pool;
    for (unsigned i = 0; i < n_threads; ++i) {
        const int64_t b = c.max_positions * i / n_threads;
        const int64_t e = c.max_positions * (i + 1) / n_threads;
        pool.emplace_back(fill_rows, out, std::cref(w), std::cref(off), mu, b, e);
    }
    for (auto& th : pool) th.join();
}

void build_host_table(sk_rope_table* t) {
    t->host.resize(size_t(t->cfg.max_positions) * (t->cfg.rotary_dim / 2));
    fill_table(t->cfg, 0, t->host.data());
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

extern "C" sk_status sk_rope_table_fill_host(const sk_rope_config* cfg, int32_t n_threads, float* out) {
    SK_RET_IF(cfg == nullptr || out == nullptr || n_threads < 0 || n_threads > 256, SK_ERR_ARG);
    SK_RET_IF(reinterpret_cast<uintptr_t>(out) & 7u, SK_ERR_ARG);
    SK_RET_IF(!config_ok(*cfg), SK_ERR_ARG);
    fill_table(*cfg, unsigned(n_threads), reinterpret_cast<float2*>(out));
    return SK_OK;
}

// Accessors used by the kernels' entry points in other translation units.
namespace sk {
const float2* table_device(const sk_rope_table* t) { return t->d_table; }
const sk_rope_config& table_config(const sk_rope_table* t) { return t->cfg; }
}  // namespace sk

// ---------------------------------------------------------------------------
// Dynamic YaRN: the factor follows the dialog's length.
//
// "#2961 rope: --rope-scaling dynamic", "What it does": the factor is 1 while the
// positions fit the trained context L0 and, past it, positions / L0 rounded up to a
// step and capped; when it changes, every cached key is turned from the old factor
// to the new one and the table is rebuilt in place, so captured CUDA graphs keep
// reading the same pointer.  Here the new factor's table is first built into a spare
// table, the keys are turned from the live table to the spare one (the rerotation
// kernel needs both), and the spare's contents are then copied over the live
// table's device buffer: the live pointer never changes and its contents are bitwise
// those of a fresh build at the new factor.
// ---------------------------------------------------------------------------

struct sk_rope_dynamic {
    sk_rope_table* live = nullptr;
    sk_rope_table* spare = nullptr;
    double step = 0.125;
    double cap = 1.0;
};

namespace {

double policy_factor(int64_t total, int64_t orig_ctx, double step, double cap) {
    if (total <= orig_ctx) return 1.0;
    const double f = std::ceil((double(total) / double(orig_ctx)) / step) * step;
    return std::min(f, cap);
}

bool policy_ok(int64_t total, int64_t orig_ctx, double step, double cap) {
    return total >= 0 && orig_ctx >= 1 && step > 0.0 && std::isfinite(step) && cap >= 1.0 && std::isfinite(cap);
}

double effective_factor(double f) { return f <= 1.0 ? 1.0 : f; }

}  // namespace

extern "C" sk_status sk_rope_dynamic_factor(int64_t total_positions, int64_t orig_ctx, double step, double cap,
                                            double* factor_out) {
    SK_RET_IF(factor_out == nullptr || !policy_ok(total_positions, orig_ctx, step, cap), SK_ERR_ARG);
    *factor_out = policy_factor(total_positions, orig_ctx, step, cap);
    return SK_OK;
}

extern "C" sk_status sk_rope_dynamic_create(const sk_rope_config* cfg, double step, double cap, void* stream,
                                            sk_rope_dynamic** out) {
    SK_RET_IF(cfg == nullptr || out == nullptr, SK_ERR_ARG);
    *out = nullptr;
    SK_RET_IF(cfg->yarn_orig_ctx < 1, SK_ERR_ARG);
    if (cap <= 0.0) cap = std::max(1.0, double(cfg->max_positions) / double(cfg->yarn_orig_ctx));
    SK_RET_IF(!policy_ok(0, cfg->yarn_orig_ctx, step, cap), SK_ERR_ARG);
    sk_rope_config c = *cfg;
    c.yarn_factor = effective_factor(c.yarn_factor);
    sk_rope_config scaled = c;  // the YaRN fields must be valid for any later factor
    scaled.yarn_factor = std::max(2.0, cap);
    SK_RET_IF(!config_ok(c) || !config_ok(scaled), SK_ERR_ARG);
    sk_rope_dynamic* d = new sk_rope_dynamic();
    d->step = step;
    d->cap = cap;
    sk_status s = sk_rope_table_create(&c, stream, &d->live);
    if (s == SK_OK) s = sk_rope_table_create(&c, stream, &d->spare);
    if (s != SK_OK) {
        sk_rope_table_destroy(d->live);
        sk_rope_table_destroy(d->spare);
        delete d;
        return s;
    }
    *out = d;
    return SK_OK;
}

extern "C" const sk_rope_table* sk_rope_dynamic_table(const sk_rope_dynamic* d) {
    return d == nullptr ? nullptr : d->live;
}

extern "C" double sk_rope_dynamic_current_factor(const sk_rope_dynamic* d) {
    return d == nullptr ? 0.0 : d->live->cfg.yarn_factor;
}

extern "C" sk_status sk_rope_dynamic_update(sk_rope_dynamic* d, int64_t total_positions,
                                            const sk_kv_layer* layers, int32_t n_layers, void* stream,
                                            double* factor_out, int32_t* switched_out) {
    SK_RET_IF(d == nullptr || total_positions < 0 || n_layers < 0, SK_ERR_ARG);
    SK_RET_IF(n_layers > 0 && layers == nullptr, SK_ERR_ARG);
    if (switched_out != nullptr) *switched_out = 0;
    sk_rope_table* live = d->live;
    sk_rope_table* spare = d->spare;
    SK_RET_IF(total_positions > live->cfg.max_positions, SK_ERR_POSITION_RANGE);
    const double f = policy_factor(total_positions, live->cfg.yarn_orig_ctx, d->step, d->cap);
    if (factor_out != nullptr) *factor_out = f;
    if (f == live->cfg.yarn_factor) return SK_OK;
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    // 1. the new factor's table, into the spare (host build, upload, stream synchronised)
    spare->cfg = live->cfg;
    spare->cfg.yarn_factor = f;
    build_host_table(spare);
    sk_status s = upload(spare, st);
    if (s != SK_OK) return s;
    // 2. turn every cached key from the live factor to the new one
    if (n_layers > 0) {
        s = sk_kv_rerotate(layers, n_layers, live, spare, stream);
        if (s != SK_OK) return s;
    }
    // 3. the live table takes the new contents in place
    const size_t bytes = spare->host.size() * sizeof(float2);
    SK_CUDA_RET(cudaMemcpyAsync(live->d_table, spare->d_table, bytes, cudaMemcpyDeviceToDevice, st));
    SK_CUDA_RET(cudaStreamSynchronize(st));
    std::swap(live->host, spare->host);
    live->cfg.yarn_factor = f;
    if (switched_out != nullptr) *switched_out = 1;
    return SK_OK;
}

extern "C" void sk_rope_dynamic_destroy(sk_rope_dynamic* d) {
    if (d == nullptr) return;
    sk_rope_table_destroy(d->live);
    sk_rope_table_destroy(d->spare);
    delete d;
}
