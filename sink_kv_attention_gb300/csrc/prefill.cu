// Prefill attention (causal + window + sinks) on the tensor cores.
#include "common.cuh"

extern "C" sk_status sk_prefill_attention(const void* q_rot, const void* k_rot, const void* v,
                                          int32_t batch, int32_t T, int32_t n_q_heads,
                                          int32_t n_kv_heads, int32_t head_dim, int64_t p0,
                                          int32_t sinks, int32_t window, void* out, void* stream) {
    (void)q_rot; (void)k_rot; (void)v; (void)batch; (void)T; (void)n_q_heads; (void)n_kv_heads;
    (void)head_dim; (void)p0; (void)sinks; (void)window; (void)out; (void)stream;
    return SK_ERR_UNSUPPORTED;
}
