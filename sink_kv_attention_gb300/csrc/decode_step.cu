// The decode step with the token's RoPE + KV append folded into decode attention
// (sk_decode_step): the FUSED instantiations of the split and combine kernels in
// decode_kernels.cuh, their grid and workspace, and the entry point's checks.
//
// "Inference & 128K Long Context", 4.3-4.4: decode is bound by the KV bytes it streams;
// at batch 1 a step through a layer streams 16.8 MB in a few microseconds, and a
// separate append kernel (a few KB of work) costs a launch and a hand-off of about as
// much again.  Folded in, the step is two launches: the split kernel, which also writes
// the token, and the combine, which also advances the ring state.
#include "decode_kernels.cuh"

namespace sk {
namespace {

template <typename T, int D, int NREP>
struct StepLaunch {
    using C = DecodeCfg<T, D, NREP, false, false, true>;
    static constexpr int THREADS = C::THREADS;
    static constexpr size_t SMEM = C::SMEM;

    static int blocks_per_sm() {
        static PerDevice<int> cache;
        return cache.get(
            [] {
                int n = 0;
                if (cudaFuncSetAttribute(decode_split_kernel<T, D, NREP, false, false, true>,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize, int(SMEM)) != cudaSuccess ||
                    cudaOccupancyMaxActiveBlocksPerMultiprocessor(
                        &n, decode_split_kernel<T, D, NREP, false, false, true>, THREADS, SMEM) != cudaSuccess)
                    return 0;
                return n;
            },
            [](int n) { return n > 0; }, 0);
    }

    static int grid() { return std::max(1, blocks_per_sm()) * device_sm_count(); }

    // the partials (as sk_decode_attention's), then the split kernel's copy of the state
    static size_t partial_bytes(const sk_kv_layer& L) {
        return size_t(grid() + int64_t(L.batch) * L.n_kv_heads) * C::PARTIAL_FLOATS * sizeof(float);
    }
    static size_t workspace(const sk_kv_layer& L) { return partial_bytes(L) + size_t(L.batch) * 4 * sizeof(int64_t); }

    static cudaError_t run(DecodeParams p, const sk_kv_layer& L, cudaStream_t st) {
        if (blocks_per_sm() < 1) return cudaErrorInvalidConfiguration;
        static_assert((C::PARTIAL_FLOATS * sizeof(float)) % 8 == 0, "state copy alignment");
        // no more blocks than rows the cache can hold
        const int64_t rows = int64_t(L.batch) * L.n_kv_heads * L.capacity;
        p.n_blocks = int(std::max<int64_t>(1, std::min<int64_t>(grid(), rows)));
        p.snap = reinterpret_cast<int64_t*>(reinterpret_cast<uint8_t*>(p.ws) + partial_bytes(L));
        cudaError_t e = launch_pdl(decode_split_kernel<T, D, NREP, false, false, true>, dim3(p.n_blocks),
                                   dim3(THREADS), SMEM, st, p);
        if (e != cudaSuccess) return e;
        p.combine_wpu = combine_wpu(p.n_blocks, int64_t(L.batch) * L.n_kv_heads);
        const int64_t warps = int64_t(L.batch) * L.n_kv_heads * NREP * p.combine_wpu;
        return p.combine_wpu == 1 ? launch_pdl(decode_combine_kernel<T, D, NREP, true>,
                                               dim3(unsigned((warps + 7) / 8)), dim3(256), 0, st, p)
                                  : launch_pdl(decode_combine_group_kernel<T, D, NREP, true>,
                                               dim3(unsigned((warps + 7) / 8)), dim3(256), 0, st, p);
    }
};

template <typename T, int D>
bool dispatch_step(int nrep, bool want_ws, const sk_kv_layer& L, DecodeParams* p, cudaStream_t st, size_t* ws,
                   cudaError_t* e) {
    switch (nrep) {
#define SK_CASE(N)                                               \
    case N:                                                      \
        if (want_ws) *ws = StepLaunch<T, D, N>::workspace(L);    \
        else *e = StepLaunch<T, D, N>::run(*p, L, st);           \
        return true;
        SK_CASE(1)
        SK_CASE(2)
        SK_CASE(4)
#undef SK_CASE
        case 8:
            if constexpr (D == 64) {
                if (want_ws) *ws = StepLaunch<T, D, 8>::workspace(L);
                else *e = StepLaunch<T, D, 8>::run(*p, L, st);
                return true;
            }
            return false;
        default:
            return false;
    }
}

// Returns false for an unsupported (dtype, head_dim, n_rep) combination.
bool route_step(int io_dtype, const sk_kv_layer& L, int nrep, bool want_ws, DecodeParams* p, cudaStream_t st,
                size_t* ws, cudaError_t* e) {
    if (io_dtype == SK_BF16 && L.k_dtype == SK_BF16 && L.v_dtype == SK_BF16) {
        if (L.head_dim == 128) return dispatch_step<__nv_bfloat16, 128>(nrep, want_ws, L, p, st, ws, e);
        if (L.head_dim == 64) return dispatch_step<__nv_bfloat16, 64>(nrep, want_ws, L, p, st, ws, e);
    } else if (io_dtype == SK_F32 && L.k_dtype == SK_F32 && L.v_dtype == SK_F32) {
        if (L.head_dim == 128) return dispatch_step<float, 128>(nrep, want_ws, L, p, st, ws, e);
        if (L.head_dim == 64) return dispatch_step<float, 64>(nrep, want_ws, L, p, st, ws, e);
    }
    return false;
}

}  // namespace
}  // namespace sk

using namespace sk;

extern "C" size_t sk_decode_step_workspace_bytes(const sk_kv_layer* layer, int32_t n_q_heads) {
    if (check_layer(layer, n_q_heads) != SK_OK) return 0;
    size_t ws = 0;
    cudaError_t e = cudaSuccess;
    const int io = layer->k_dtype == SK_F32 ? SK_F32 : SK_BF16;
    if (!route_step(io, *layer, n_q_heads / layer->n_kv_heads, true, nullptr, nullptr, &ws, &e)) return 0;
    return ws;
}

extern "C" sk_status sk_decode_step(const sk_rope_table* table, const sk_kv_layer* layer, const void* q,
                                    int32_t n_q_heads, const void* k, const void* v, int32_t io_dtype,
                                    const float* sink_logits, void* out, void* workspace, size_t ws_bytes,
                                    void* stream) {
    sk_status s = check_layer(layer, n_q_heads);
    if (s != SK_OK) return s;
    const sk_kv_layer& L = *layer;
    SK_RET_IF(q == nullptr || k == nullptr || v == nullptr || out == nullptr || workspace == nullptr, SK_ERR_ARG);
    SK_RET_IF((reinterpret_cast<uintptr_t>(q) | reinterpret_cast<uintptr_t>(k) | reinterpret_cast<uintptr_t>(v) |
               reinterpret_cast<uintptr_t>(out) | reinterpret_cast<uintptr_t>(workspace)) &
                  15u,
              SK_ERR_ARG);
    SK_RET_IF(reinterpret_cast<uintptr_t>(sink_logits) & 3u, SK_ERR_ARG);
    if (L.kind == SK_LAYER_RING) SK_RET_IF(L.head == nullptr, SK_ERR_ARG);
    // Without a table the keys come rotated: no rotary dims and no position limit but
    // the counter's own (as sk_kv_append).
    const float2* tab = nullptr;
    int64_t max_pos = int64_t(1) << 62;
    int rotary_dim = 0, neox = 1;
    if (table != nullptr) {
        const sk_rope_config& c = table_config(table);
        SK_RET_IF(c.head_dim != L.head_dim, SK_ERR_ARG);
        tab = table_device(table);
        max_pos = c.max_positions;
        rotary_dim = c.rotary_dim;
        neox = c.neox != 0 ? 1 : 0;
    }
    const int nrep = n_q_heads / L.n_kv_heads;
    size_t need = 0;
    cudaError_t e = cudaSuccess;
    if (!route_step(io_dtype, L, nrep, true, nullptr, nullptr, &need, &e)) return SK_ERR_UNSUPPORTED;
    SK_RET_IF(ws_bytes < need, SK_ERR_ARG);
    DecodeParams p{};
    p.kc = L.k;
    p.vc = L.v;
    p.q = q;
    p.sink_logits = sink_logits;
    p.out = out;
    p.ws = static_cast<float*>(workspace);
    p.count = L.count;
    p.pos = L.pos;
    p.kscale = nullptr;
    p.err = L.err;
    p.cap = L.capacity;
    p.B = L.batch;
    p.Hkv = L.n_kv_heads;
    p.S = L.sinks;
    p.W = L.kind == SK_LAYER_RING ? L.window : 0;
    p.kind = L.kind;
    p.qscale = kLog2e / sqrtf(float(L.head_dim));
    p.k_new = k;
    p.v_new = v;
    p.table = tab;
    p.max_pos = max_pos;
    p.rotary_dim = rotary_dim;
    p.neox = neox;
    p.head = L.kind == SK_LAYER_RING ? L.head : nullptr;
    p.head_rw = L.head;
    p.count_rw = L.count;
    p.pos_rw = L.pos;
    route_step(io_dtype, L, nrep, false, &p, static_cast<cudaStream_t>(stream), nullptr, &e);
    return e == cudaSuccess ? SK_OK : SK_ERR_CUDA;
}
