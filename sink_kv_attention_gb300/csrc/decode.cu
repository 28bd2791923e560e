// Entry points of decode attention over contiguous and paged layers: argument checks,
// dispatch over (dtype, head_dim, n_rep) and the launches.  The kernels are in
// decode_kernels.cuh, shared with the decode step that folds the append in
// (decode_step.cu).
#include "decode_kernels.cuh"

namespace sk {
namespace {

template <typename T, int D, bool KQ = false>
bool dispatch(int nrep, bool want_ws, const sk_kv_layer& L, DecodeParams* p, cudaStream_t st, size_t* ws,
              cudaError_t* e) {
    switch (nrep) {
#define SK_CASE(N)                                                  \
    case N:                                                         \
        if (want_ws) *ws = DecodeLaunch<T, D, N, KQ>::workspace(L); \
        else *e = DecodeLaunch<T, D, N, KQ>::run(*p, L, st);        \
        return true;
        SK_CASE(1)
        SK_CASE(2)
        SK_CASE(4)
#undef SK_CASE
        case 8:
            if constexpr (D == 64) {
                if (want_ws) *ws = DecodeLaunch<T, D, 8>::workspace(L);
                else *e = DecodeLaunch<T, D, 8>::run(*p, L, st);
                return true;
            }
            return false;
        default:
            return false;
    }
}

// Returns false for an unsupported (dtype, head_dim, n_rep) combination.
bool route(int io_dtype, const sk_kv_layer& L, int nrep, bool want_ws, DecodeParams* p, cudaStream_t st,
           size_t* ws, cudaError_t* e) {
    if (io_dtype == SK_BF16 && L.k_dtype == SK_BF16 && L.v_dtype == SK_BF16) {
        if (L.head_dim == 128) return dispatch<__nv_bfloat16, 128>(nrep, want_ws, L, p, st, ws, e);
        if (L.head_dim == 64) return dispatch<__nv_bfloat16, 64>(nrep, want_ws, L, p, st, ws, e);
    } else if (io_dtype == SK_F32 && L.k_dtype == SK_F32 && L.v_dtype == SK_F32) {
        if (L.head_dim == 128) return dispatch<float, 128>(nrep, want_ws, L, p, st, ws, e);
        if (L.head_dim == 64) return dispatch<float, 64>(nrep, want_ws, L, p, st, ws, e);
    } else if (io_dtype == SK_BF16 && L.k_dtype == SK_I8 && L.v_dtype == SK_BF16) {
        if (L.head_dim == 128) return dispatch<__nv_bfloat16, 128, true>(nrep, want_ws, L, p, st, ws, e);
    }
    return false;
}

}  // namespace
}  // namespace sk

using namespace sk;

extern "C" size_t sk_decode_workspace_bytes(const sk_kv_layer* layer, int32_t n_q_heads) {
    if (check_layer(layer, n_q_heads) != SK_OK) return 0;
    size_t ws = 0;
    cudaError_t e = cudaSuccess;
    const int nrep = n_q_heads / layer->n_kv_heads;
    const int io = layer->k_dtype == SK_F32 ? SK_F32 : SK_BF16;
    if (!route(io, *layer, nrep, true, nullptr, nullptr, &ws, &e)) return 0;
    return ws;
}

extern "C" sk_status sk_decode_attention(const sk_kv_layer* layer, const void* q_rot, int32_t n_q_heads,
                                         int32_t io_dtype, const float* sink_logits, void* out,
                                         void* workspace, size_t ws_bytes, void* stream) {
    sk_status s = check_layer(layer, n_q_heads);
    if (s != SK_OK) return s;
    SK_RET_IF(q_rot == nullptr || out == nullptr || workspace == nullptr, SK_ERR_ARG);
    SK_RET_IF((reinterpret_cast<uintptr_t>(q_rot) | reinterpret_cast<uintptr_t>(workspace)) & 15u, SK_ERR_ARG);
    SK_RET_IF(reinterpret_cast<uintptr_t>(sink_logits) & 3u, SK_ERR_ARG);
    const sk_kv_layer& L = *layer;
    const int nrep = n_q_heads / L.n_kv_heads;
    size_t need = 0;
    cudaError_t e = cudaSuccess;
    if (!route(io_dtype, L, nrep, true, nullptr, nullptr, &need, &e)) return SK_ERR_UNSUPPORTED;
    SK_RET_IF(ws_bytes < need, SK_ERR_ARG);
    DecodeParams p{};
    p.kc = L.k;
    p.vc = L.v;
    p.q = q_rot;
    p.sink_logits = sink_logits;
    p.out = out;
    p.ws = static_cast<float*>(workspace);
    p.count = L.count;
    p.pos = L.pos;
    p.kscale = L.k_dtype == SK_I8 ? L.k_scale : nullptr;
    p.err = L.err;
    p.cap = L.capacity;
    p.B = L.batch;
    p.Hkv = L.n_kv_heads;
    p.S = L.sinks;
    p.kind = L.kind;
    p.qscale = kLog2e / sqrtf(float(L.head_dim));
    route(io_dtype, L, nrep, false, &p, static_cast<cudaStream_t>(stream), nullptr, &e);
    return e == cudaSuccess ? SK_OK : SK_ERR_CUDA;
}

// ---------------------------------------------------------------------------
// Decode attention over a paged layer.
// ---------------------------------------------------------------------------

namespace {

// The fields of a contiguous layer descriptor that route() and the workspace size read.
sk_kv_layer paged_as_layer(const sk_paged_layer& L) {
    sk_kv_layer v{};
    v.kind = kKindPaged;
    v.k_dtype = L.k_dtype;
    v.v_dtype = L.v_dtype;
    v.batch = L.batch;
    v.n_kv_heads = L.n_kv_heads;
    v.head_dim = L.head_dim;
    return v;
}

sk_status check_paged(const sk_paged_layer* layer, int32_t n_q_heads) {
    SK_RET_IF(layer == nullptr, SK_ERR_ARG);
    SK_RET_IF(paged_layer_check(*layer) != SK_OK, SK_ERR_ARG);
    SK_RET_IF(layer->batch > kMaxBatch, SK_ERR_UNSUPPORTED);
    SK_RET_IF(n_q_heads < 1 || n_q_heads % layer->n_kv_heads != 0, SK_ERR_ARG);
    return SK_OK;
}

}  // namespace

extern "C" size_t sk_paged_decode_workspace_bytes(const sk_paged_layer* layer, int32_t n_q_heads) {
    if (check_paged(layer, n_q_heads) != SK_OK) return 0;
    const sk_kv_layer L = paged_as_layer(*layer);
    size_t ws = 0;
    cudaError_t e = cudaSuccess;
    if (!route(L.k_dtype, L, n_q_heads / L.n_kv_heads, true, nullptr, nullptr, &ws, &e)) return 0;
    return ws;
}

extern "C" sk_status sk_paged_decode_attention(const sk_paged_layer* layer, const void* q_rot, int32_t n_q_heads,
                                               int32_t io_dtype, const float* sink_logits, void* out,
                                               void* workspace, size_t ws_bytes, void* stream) {
    sk_status s = check_paged(layer, n_q_heads);
    if (s != SK_OK) return s;
    SK_RET_IF(q_rot == nullptr || out == nullptr || workspace == nullptr, SK_ERR_ARG);
    SK_RET_IF((reinterpret_cast<uintptr_t>(q_rot) | reinterpret_cast<uintptr_t>(workspace)) & 15u, SK_ERR_ARG);
    SK_RET_IF(reinterpret_cast<uintptr_t>(sink_logits) & 3u, SK_ERR_ARG);
    const sk_paged_layer& PL = *layer;
    const sk_kv_layer L = paged_as_layer(PL);
    const int nrep = n_q_heads / L.n_kv_heads;
    size_t need = 0;
    cudaError_t e = cudaSuccess;
    if (!route(io_dtype, L, nrep, true, nullptr, nullptr, &need, &e)) return SK_ERR_UNSUPPORTED;
    SK_RET_IF(ws_bytes < need, SK_ERR_ARG);
    DecodeParams p{};
    p.kc = PL.k_pool;
    p.vc = PL.v_pool;
    p.q = q_rot;
    p.sink_logits = sink_logits;
    p.out = out;
    p.ws = static_cast<float*>(workspace);
    p.pos = PL.seq_lens;
    p.err = PL.err;
    p.B = PL.batch;
    p.Hkv = PL.n_kv_heads;
    p.S = PL.sinks;
    p.kind = kKindPaged;
    p.qscale = kLog2e / sqrtf(float(PL.head_dim));
    p.block_table = PL.block_table;
    p.sink_blocks = PL.sink_block_ids;
    p.pool_blocks = PL.n_blocks;
    p.bs = PL.block_size;
    p.bs_log2 = __builtin_ctz(unsigned(PL.block_size));
    p.max_blocks = PL.max_blocks;
    p.sink_len = PL.n_sink_blocks * PL.block_size;
    p.W = PL.window;
    route(io_dtype, L, nrep, false, &p, static_cast<cudaStream_t>(stream), nullptr, &e);
    return e == cudaSuccess ? SK_OK : SK_ERR_CUDA;
}

// ---------------------------------------------------------------------------
// Decode attention with the library's own fixed scratch (no allocation).
// ---------------------------------------------------------------------------

namespace {

// The scratch of sk_decode_attention_noalloc.  In host code this name is only a
// stand-in: its device address comes from cudaGetSymbolAddress, once per device.
static __device__ __align__(256) unsigned char g_noalloc_scratch[SK_DECODE_NOALLOC_SCRATCH_BYTES];

// Device address of g_noalloc_scratch on the current device, looked up on first use.
sk_status noalloc_scratch(void** out) {
    static std::mutex mu;
    static void* addr[64] = {};
    int dev = 0;
    SK_CUDA_RET(cudaGetDevice(&dev));
    SK_RET_IF(dev < 0 || dev >= 64, SK_ERR_UNSUPPORTED);
    std::lock_guard<std::mutex> lock(mu);
    if (addr[dev] == nullptr) {
        void* p = nullptr;
        SK_CUDA_RET(cudaGetSymbolAddress(&p, g_noalloc_scratch));
        SK_RET_IF(p == nullptr, SK_ERR_CUDA);
        addr[dev] = p;
    }
    *out = addr[dev];
    return SK_OK;
}

}  // namespace

extern "C" sk_status sk_decode_attention_noalloc(const sk_kv_layer* layer, const void* q_rot,
                                                 int32_t n_q_heads, int32_t io_dtype,
                                                 const float* sink_logits, void* out, void* stream) {
    sk_status s = check_layer(layer, n_q_heads);
    if (s != SK_OK) return s;
    SK_RET_IF(q_rot == nullptr || out == nullptr, SK_ERR_ARG);
    const int nrep = n_q_heads / layer->n_kv_heads;
    size_t need = 0;
    cudaError_t e = cudaSuccess;
    if (!route(io_dtype, *layer, nrep, true, nullptr, nullptr, &need, &e)) return SK_ERR_UNSUPPORTED;
    SK_RET_IF(need > SK_DECODE_NOALLOC_SCRATCH_BYTES, SK_ERR_CAPACITY);
    void* scratch = nullptr;
    s = noalloc_scratch(&scratch);
    if (s != SK_OK) return s;
    return sk_decode_attention(layer, q_rot, n_q_heads, io_dtype, sink_logits, out, scratch,
                               SK_DECODE_NOALLOC_SCRATCH_BYTES, stream);
}
