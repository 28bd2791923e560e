// In-place rerotation of cached keys when the RoPE factor changes.
//
// "#2961 rope: --rope-scaling dynamic", "What it does": keys are cached after RoPE, so
// turning each pair of a key cached at factor A by a further angle p (w_B - w_A) and
// scaling it by mscale_B / mscale_A gives the key at factor B; int8 keys are
// dequantized, turned and requantized.  "Attention Sink 与 Streaming KV Cache": R_a R_b
// = R_{a+b}, so no raw key is needed.  The delta rotation comes from the two tables'
// entries at P: with (cA, sA) = mu_A (cos a, sin a) and (cB, sB) = mu_B (cos b, sin b),
//   (cB cA + sB sA) / mu_A^2 = (mu_B / mu_A) cos(b - a),
//   (sB cA - cB sA) / mu_A^2 = (mu_B / mu_A) sin(b - a).
//
// The same kernels turn the recent keys of ring layers by a uniform number of positions
// delta ("Attention Sink 与 Streaming KV Cache", "RoPE：absolute positions 与 local
// rerotation 是两种实现": a cache fed local positions moves its recent keys from p to
// p - 1 when the window slides; sink keys keep their positions).  The rotation is then
// the same for every row, R(delta w) with no mscale change, taken from one table: rows
// A = max(0, -delta) and B = max(0, delta) give exactly (cos, sin)(delta w) in the
// formulas above with mu_A = mu_B = mu.
//
// Layout of the work: one block covers a range of slots (and, when the slots alone
// give too few blocks, a stride of the sequences: blockIdx.y); each thread group owns
// one slot and walks every (layer, sequence, kv head) row at that slot, recomputing the
// delta only when the slot's position changes (never, for global layers).  The bf16
// path reads and writes only the rotary bytes of each row; the int8 path moves the
// whole row of codes plus its scale.
#include <algorithm>
#include <cmath>

#include "common.cuh"

namespace sk {
namespace {

constexpr int kThreads = 256;
constexpr int kMaxLayers = 128;

struct RerotLayer {
    void* k;
    float* scale;
    const int32_t* head;
    const int32_t* count;
    const int64_t* pos;
    uint32_t* err;
    int64_t cap;
    int kind, S, W;
};

struct RerotParams {
    RerotLayer layers[kMaxLayers];
    int n_layers;
    int B, Hkv, r;
    const float2* tA;
    const float2* tB;
    int64_t maxA, maxB;
    float inv_muA2;
    int shift;            // 1: uniform turn of the recent keys (sinks skipped)
    int64_t rowA, rowB;   // shift mode: the table rows whose entries give the turn
};

// Position held by `slot` of (layer, sequence b), or -1 when the slot is empty.
__device__ __forceinline__ int64_t slot_position(const RerotLayer& L, int b, int64_t slot) {
    if (slot >= L.cap) return -1;
    const int64_t pos = L.pos[b];
    if (L.kind == SK_LAYER_GLOBAL) return slot < pos ? slot : -1;
    if (slot < L.S) return slot < min(pos, int64_t(L.S)) ? slot : -1;
    const int64_t j = slot - L.S;
    const int count = L.count[b];
    if (j >= count) return -1;
    const int64_t W = L.W;
    const int64_t back = ((int64_t(L.head[b]) - 1 - j) % W + W) % W;  // steps behind the newest
    return pos - 1 - back;
}

// The slot's position for a factor change, or -1 to skip the slot.  In shift mode
// the sink slots are skipped and every other occupied slot gets key 0 (the turn does
// not depend on the position).
__device__ __forceinline__ int64_t rerot_key(const RerotParams& p, const RerotLayer& L, int b, int64_t slot) {
    const int64_t P = slot_position(L, b, slot);
    if (!p.shift) return P;
    return (P < 0 || slot < L.S) ? -1 : 0;
}

// Delta rotation (dc, ds) of NP consecutive pairs starting at j0, at position P (a
// factor change) or of the uniform turn (shift mode).
template <int NP>
__device__ __forceinline__ void delta_pairs(const RerotParams& p, int64_t P, int j0, float* dc,
                                            float* ds) {
    const int half = p.r / 2;
    const int64_t PA = p.shift ? p.rowA : P, PB = p.shift ? p.rowB : P;
    const float4* a4 = reinterpret_cast<const float4*>(p.tA + PA * half + j0);
    const float4* b4 = reinterpret_cast<const float4*>(p.tB + PB * half + j0);
#pragma unroll
    for (int i = 0; i < NP / 2; ++i) {
        const float4 a = __ldg(a4 + i), b = __ldg(b4 + i);
        dc[2 * i] = (b.x * a.x + b.y * a.y) * p.inv_muA2;
        ds[2 * i] = (b.y * a.x - b.x * a.y) * p.inv_muA2;
        dc[2 * i + 1] = (b.z * a.z + b.w * a.w) * p.inv_muA2;
        ds[2 * i + 1] = (b.w * a.z - b.z * a.w) * p.inv_muA2;
    }
}

// The same delta rotation as (cos, sin) pairs of consecutive rotary pairs: dc2[i] holds
// the cosines of pairs j0 + 2i and j0 + 2i + 1, ds2[i] their sines.
template <int N2>
__device__ __forceinline__ void delta_pairs2(const RerotParams& p, int64_t P, int j0, float2* dc2, float2* ds2) {
    const int half = p.r / 2;
    const int64_t PA = p.shift ? p.rowA : P, PB = p.shift ? p.rowB : P;
    const float4* a4 = reinterpret_cast<const float4*>(p.tA + PA * half + j0);
    const float4* b4 = reinterpret_cast<const float4*>(p.tB + PB * half + j0);
#pragma unroll
    for (int i = 0; i < N2; ++i) {
        const float4 a = __ldg(a4 + i), b = __ldg(b4 + i);
        dc2[i] = make_float2((b.x * a.x + b.y * a.y) * p.inv_muA2, (b.z * a.z + b.w * a.w) * p.inv_muA2);
        ds2[i] = make_float2((b.y * a.x - b.x * a.y) * p.inv_muA2, (b.w * a.z - b.z * a.w) * p.inv_muA2);
    }
}

// ---- bf16 keys: NeoX thread = 8 pairs (16 B of each half); GPT-J thread = 4 pairs ----
template <int D, bool NEOX>
__global__ void __launch_bounds__(kThreads) rerotate_bf16_kernel(RerotParams p) {
    constexpr int NP = NEOX ? 8 : 4;  // pairs per thread
    const int tpr = p.r / (2 * NP);   // threads per row
    const int spb = kThreads / tpr;   // slots per block
    const int t = threadIdx.x % tpr;
    const int local = threadIdx.x / tpr;
    if (local >= spb) return;
    const int64_t slot = int64_t(blockIdx.x) * spb + local;
    const int half = p.r / 2;
    const int j0 = t * NP;
    float dc[NP], ds[NP];
    int64_t lastP = -1;
    for (int l = 0; l < p.n_layers; ++l) {
        const RerotLayer& L = p.layers[l];
        for (int b = blockIdx.y; b < p.B; b += gridDim.y) {
            const int64_t P = rerot_key(p, L, b, slot);
            if (P < 0) continue;
            if (P >= p.maxA || P >= p.maxB) {
                set_error(L.err, SK_DEVERR_POSITION_RANGE);
                continue;
            }
            if (P != lastP) {
                delta_pairs<NP>(p, P, j0, dc, ds);
                lastP = P;
            }
            __nv_bfloat16* base = static_cast<__nv_bfloat16*>(L.k);
            for (int g0 = 0; g0 < p.Hkv; g0 += 4) {
                const int ng = min(4, p.Hkv - g0);
                uint4 x1[4], x2[4];
#pragma unroll
                for (int u = 0; u < 4; ++u) {
                    if (u < ng) {
                        const __nv_bfloat16* row =
                            base + ((int64_t(b) * p.Hkv + g0 + u) * L.cap + slot) * D;
                        if (NEOX) {
                            x1[u] = *reinterpret_cast<const uint4*>(row + j0);
                            x2[u] = *reinterpret_cast<const uint4*>(row + half + j0);
                        } else {
                            x1[u] = *reinterpret_cast<const uint4*>(row + 2 * j0);
                        }
                    }
                }
#pragma unroll
                for (int u = 0; u < 4; ++u) {
                    if (u >= ng) continue;
                    __nv_bfloat16* row = base + ((int64_t(b) * p.Hkv + g0 + u) * L.cap + slot) * D;
                    if (NEOX) {
                        float a[8], c[8];
                        ElemIO<__nv_bfloat16>::unpack(x1[u], a);
                        ElemIO<__nv_bfloat16>::unpack(x2[u], c);
                        float o1[8], o2[8];
#pragma unroll
                        for (int i = 0; i < 8; ++i) {
                            o1[i] = fmaf(-c[i], ds[i], a[i] * dc[i]);
                            o2[i] = fmaf(a[i], ds[i], c[i] * dc[i]);
                        }
                        *reinterpret_cast<uint4*>(row + j0) = ElemIO<__nv_bfloat16>::pack(o1);
                        *reinterpret_cast<uint4*>(row + half + j0) = ElemIO<__nv_bfloat16>::pack(o2);
                    } else {
                        float a[8], o[8];
                        ElemIO<__nv_bfloat16>::unpack(x1[u], a);
#pragma unroll
                        for (int i = 0; i < 4; ++i) {
                            o[2 * i] = fmaf(-a[2 * i + 1], ds[i], a[2 * i] * dc[i]);
                            o[2 * i + 1] = fmaf(a[2 * i], ds[i], a[2 * i + 1] * dc[i]);
                        }
                        *reinterpret_cast<uint4*>(row + 2 * j0) = ElemIO<__nv_bfloat16>::pack(o);
                    }
                }
            }
        }
    }
}

// ---- int8 keys + per-row fp32 scale: D/32 threads per row, 32 codes each ----
//
// The row is turned in code units: with x = code * s_old, the new codes are
// rint(x * 127 / max|x|) = rint(t * 127 / max|t|) for t = the turned codes, and the new
// scale is max|t| * s_old / 127.  Pairs of values go through packed fp32 arithmetic.

// 8 float pairs -> 16 codes rint(t * inv), ties to even (|t * inv| < 127.5 by construction).
__device__ __forceinline__ uint4 pairs_to_codes16(const float2* t, float inv) {
    const float2 inv2 = make_float2(inv, inv), magic = make_float2(12582912.0f, 12582912.0f);
    uint32_t r[16];
#pragma unroll
    for (int i = 0; i < 8; ++i) {
        // the product is rounded before the rounding add: no fused multiply-add
        const float2 y = __fadd2_rn(__fmul2_rn(t[i], inv2), magic);
        r[2 * i] = __float_as_uint(y.x);
        r[2 * i + 1] = __float_as_uint(y.y);
    }
    uint32_t w[4];
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        const uint32_t lo = __byte_perm(r[4 * i], r[4 * i + 1], 0x0040);
        const uint32_t hi = __byte_perm(r[4 * i + 2], r[4 * i + 3], 0x0040);
        w[i] = __byte_perm(lo, hi, 0x5410);
    }
    return make_uint4(w[0], w[1], w[2], w[3]);
}

constexpr int kRowsInFlight = 1;  // kv-head rows each thread loads before computing

template <int D, bool NEOX>
__global__ void __launch_bounds__(kThreads, 4) rerotate_i8_kernel(RerotParams p) {
    constexpr int TPR = D / 32;  // threads per row (aligned group of 2 or 4 lanes)
    constexpr int SPB = kThreads / TPR;
    const int t = threadIdx.x % TPR;
    const int64_t slot = int64_t(blockIdx.x) * SPB + threadIdx.x / TPR;
    const int half = p.r / 2;
    const bool rot = t < p.r / 32;
    // NeoX rotary thread t: codes [16t, 16t+16) and [half+16t, ...), pairs j0 = 16t.
    // GPT-J rotary thread t: codes [32t, 32t+32), pairs j0 = 16t.
    // Tail thread: codes [r + 32 (t - r/32), +32).
    const int j0 = 16 * t;
    const int off1 = rot ? (NEOX ? 16 * t : 32 * t) : p.r + 32 * (t - p.r / 32);
    const int off2 = rot ? (NEOX ? half + 16 * t : 32 * t + 16) : off1 + 16;
    // delta rotation of pairs j0 .. j0+15 as (cos, cos, sin, sin) of two consecutive
    // pairs, thread-minor in shared memory: keeping it in registers made the loop spill
    __shared__ float4 sdelta[8][kThreads];
    int64_t lastP = -1;
    for (int l = 0; l < p.n_layers; ++l) {
        const RerotLayer& L = p.layers[l];
        for (int b = blockIdx.y; b < p.B; b += gridDim.y) {
            // Lanes of one warp hold different slots, so validity differs between row
            // groups: every lane runs the loop and the shuffles, only valid rows touch memory.
            const int64_t P = rerot_key(p, L, b, slot);
            bool valid = P >= 0;
            if (valid && (P >= p.maxA || P >= p.maxB)) {
                set_error(L.err, SK_DEVERR_POSITION_RANGE);
                valid = false;
            }
            if (valid && rot && P != lastP) {
                float2 dc2[8], ds2[8];
                delta_pairs2<8>(p, P, j0, dc2, ds2);
#pragma unroll
                for (int i = 0; i < 8; ++i)
                    sdelta[i][threadIdx.x] = make_float4(dc2[i].x, dc2[i].y, ds2[i].x, ds2[i].y);
                lastP = P;
            }
            for (int g0 = 0; g0 < p.Hkv; g0 += kRowsInFlight) {
                const int ng = min(kRowsInFlight, p.Hkv - g0);
                uint4 u1[kRowsInFlight], u2[kRowsInFlight];
                float s_old[kRowsInFlight];
#pragma unroll
                for (int u = 0; u < kRowsInFlight; ++u) {  // issue the loads of the rows first
                    u1[u] = make_uint4(0, 0, 0, 0);
                    u2[u] = make_uint4(0, 0, 0, 0);
                    s_old[u] = 0.0f;
                    if (valid && u < ng) {
                        const int64_t crow = (int64_t(b) * p.Hkv + g0 + u) * L.cap + slot;
                        const int8_t* row = static_cast<const int8_t*>(L.k) + crow * D;
                        s_old[u] = L.scale[crow];
                        u1[u] = *reinterpret_cast<const uint4*>(row + off1);
                        u2[u] = *reinterpret_cast<const uint4*>(row + off2);
                    }
                }
#pragma unroll
                for (int u = 0; u < kRowsInFlight; ++u) {
                    if (u >= ng) break;  // uniform across the warp
                    const int64_t crow = (int64_t(b) * p.Hkv + g0 + u) * L.cap + slot;
                    int8_t* row = static_cast<int8_t*>(L.k) + crow * D;
                    float2 a[8], c[8];  // codes off1 .. +15 and off2 .. +15 as pairs
                    codes16_to_pairs(u1[u], a);
                    codes16_to_pairs(u2[u], c);
                    if (valid && rot) {
                        if (NEOX) {
                            // pair j: x1 = a, x2 = c -> (x1 dc - x2 ds, x2 dc + x1 ds)
#pragma unroll
                            for (int i = 0; i < 8; ++i) {
                                const float4 d = sdelta[i][threadIdx.x];
                                const float2 dc = make_float2(d.x, d.y), ds = make_float2(d.z, d.w);
                                const float2 x1 = a[i], x2 = c[i];
                                a[i] = __ffma2_rn(x1, dc, __fmul2_rn(make_float2(-x2.x, -x2.y), ds));
                                c[i] = __ffma2_rn(x2, dc, __fmul2_rn(x1, ds));
                            }
                        } else {
                            // interleaved pairs (2j, 2j+1) of codes [32t, 32t+32): regroup
                            float2 x1[8], x2[8];
#pragma unroll
                            for (int i = 0; i < 4; ++i) {
                                x1[i] = make_float2(a[2 * i].x, a[2 * i + 1].x);
                                x2[i] = make_float2(a[2 * i].y, a[2 * i + 1].y);
                                x1[4 + i] = make_float2(c[2 * i].x, c[2 * i + 1].x);
                                x2[4 + i] = make_float2(c[2 * i].y, c[2 * i + 1].y);
                            }
#pragma unroll
                            for (int i = 0; i < 8; ++i) {
                                const float4 d = sdelta[i][threadIdx.x];
                                const float2 dc = make_float2(d.x, d.y), ds = make_float2(d.z, d.w);
                                const float2 y1 = __ffma2_rn(x1[i], dc, __fmul2_rn(make_float2(-x2[i].x, -x2[i].y), ds));
                                const float2 y2 = __ffma2_rn(x2[i], dc, __fmul2_rn(x1[i], ds));
                                x1[i] = y1;
                                x2[i] = y2;
                            }
#pragma unroll
                            for (int i = 0; i < 4; ++i) {
                                a[2 * i] = make_float2(x1[i].x, x2[i].x);
                                a[2 * i + 1] = make_float2(x1[i].y, x2[i].y);
                                c[2 * i] = make_float2(x1[4 + i].x, x2[4 + i].x);
                                c[2 * i + 1] = make_float2(x1[4 + i].y, x2[4 + i].y);
                            }
                        }
                    }
                    float m0 = 0.0f, m1 = 0.0f;  // max |t| in code units, two chains
#pragma unroll
                    for (int i = 0; i < 8; ++i) {
                        m0 = fmaxf(m0, fmaxf(fabsf(a[i].x), fabsf(a[i].y)));
                        m1 = fmaxf(m1, fmaxf(fabsf(c[i].x), fabsf(c[i].y)));
                    }
                    float amax_c = fmaxf(m0, m1);
#pragma unroll
                    for (int o = TPR / 2; o > 0; o >>= 1)
                        amax_c = fmaxf(amax_c, __shfl_xor_sync(0xffffffffu, amax_c, o));
                    // new scale max|x| / 127 with x = t * s_old; codes rint(t * 127 / max|t|)
                    const float amax_x = amax_c * s_old[u];
                    const float s_new = amax_x == 0.0f ? 1.0f : __fdiv_rn(amax_x, 127.0f);
                    const float inv = amax_x == 0.0f ? 0.0f : __fdiv_rn(127.0f, amax_c);  // in code units
                    if (valid) {
                        *reinterpret_cast<uint4*>(row + off1) = pairs_to_codes16(a, inv);
                        *reinterpret_cast<uint4*>(row + off2) = pairs_to_codes16(c, inv);
                        if (t == 0) L.scale[crow] = s_new;
                    }
                }
            }
        }
    }
}

}  // namespace
}  // namespace sk

using namespace sk;

namespace {

// Checks the layers, fills p.layers / n_layers / B / Hkv / r and launches the kernel
// for the table config `c` (both tables share d_h, r, pairing and theta).
sk_status launch_rerotation(const sk_kv_layer* layers, int32_t n_layers, const sk_rope_config& c, bool rings_only,
                            RerotParams& p, cudaStream_t st) {
    SK_RET_IF(layers == nullptr || n_layers < 1 || n_layers > kMaxLayers, SK_ERR_ARG);
    const sk_kv_layer& L0 = layers[0];
    const int D = L0.head_dim;
    SK_RET_IF(D != c.head_dim, SK_ERR_ARG);
    SK_RET_IF(L0.k_dtype != SK_BF16 && L0.k_dtype != SK_I8, SK_ERR_UNSUPPORTED);
    SK_RET_IF(L0.k_dtype == SK_I8 && c.rotary_dim % 32 != 0, SK_ERR_UNSUPPORTED);
    p.n_layers = n_layers;
    p.B = L0.batch;
    p.Hkv = L0.n_kv_heads;
    p.r = c.rotary_dim;
    int64_t max_cap = 0;
    for (int l = 0; l < n_layers; ++l) {
        const sk_kv_layer& L = layers[l];
        SK_RET_IF(L.k == nullptr || L.pos == nullptr, SK_ERR_ARG);
        SK_RET_IF(L.batch != p.B || L.n_kv_heads != p.Hkv || L.head_dim != D ||
                      L.k_dtype != L0.k_dtype,
                  SK_ERR_ARG);
        SK_RET_IF(L.k_dtype == SK_I8 && L.k_scale == nullptr, SK_ERR_ARG);
        SK_RET_IF(reinterpret_cast<uintptr_t>(L.k) & 15u, SK_ERR_ARG);
        if (L.kind == SK_LAYER_RING) {
            SK_RET_IF(L.head == nullptr || L.count == nullptr || L.window < 1 || L.sinks < 0 ||
                          L.capacity != int64_t(L.sinks) + L.window,
                      SK_ERR_ARG);
        } else {
            SK_RET_IF(rings_only || L.kind != SK_LAYER_GLOBAL || L.capacity < 1, SK_ERR_ARG);
        }
        p.layers[l] = RerotLayer{L.k, L.k_scale, L.head, L.count, L.pos, L.err,
                                 L.capacity, L.kind, L.sinks, L.window};
        max_cap = std::max(max_cap, L.capacity);
    }
    const bool neox = c.neox != 0;
    const int spb = L0.k_dtype == SK_BF16 ? kThreads / (p.r / (neox ? 16 : 8)) : kThreads / (D / 32);
    const int64_t bx = (max_cap + spb - 1) / spb;
    // sequences split over blockIdx.y until there are about 16 blocks per SM
    const int64_t want = 16 * int64_t(device_sm_count());
    const int64_t by0 = std::min<int64_t>(p.B, std::max<int64_t>(1, (want + bx - 1) / bx));
    const int64_t per_block = (p.B + by0 - 1) / by0;  // sequences per block, the same for all
    const int by = int((p.B + per_block - 1) / per_block);
    const dim3 grid{unsigned(bx), unsigned(by), 1u};
    if (L0.k_dtype == SK_BF16) {
        if (D == 64)
            neox ? rerotate_bf16_kernel<64, true><<<grid, kThreads, 0, st>>>(p)
                 : rerotate_bf16_kernel<64, false><<<grid, kThreads, 0, st>>>(p);
        else
            neox ? rerotate_bf16_kernel<128, true><<<grid, kThreads, 0, st>>>(p)
                 : rerotate_bf16_kernel<128, false><<<grid, kThreads, 0, st>>>(p);
    } else {
        if (D == 64)
            neox ? rerotate_i8_kernel<64, true><<<grid, kThreads, 0, st>>>(p)
                 : rerotate_i8_kernel<64, false><<<grid, kThreads, 0, st>>>(p);
        else
            neox ? rerotate_i8_kernel<128, true><<<grid, kThreads, 0, st>>>(p)
                 : rerotate_i8_kernel<128, false><<<grid, kThreads, 0, st>>>(p);
    }
    return cudaGetLastError() == cudaSuccess ? SK_OK : SK_ERR_CUDA;
}

double mscale_of(const sk_rope_config& c) {
    return c.yarn_factor <= 1.0 ? 1.0 : 0.1 * std::log(c.yarn_factor) + 1.0;
}

}  // namespace

extern "C" sk_status sk_kv_rerotate(const sk_kv_layer* layers, int32_t n_layers,
                                    const sk_rope_table* from, const sk_rope_table* to,
                                    void* stream) {
    SK_RET_IF(layers == nullptr || from == nullptr || to == nullptr, SK_ERR_ARG);
    const sk_rope_config& ca = table_config(from);
    const sk_rope_config& cb = table_config(to);
    SK_RET_IF(ca.head_dim != cb.head_dim || ca.rotary_dim != cb.rotary_dim || ca.neox != cb.neox ||
                  ca.theta != cb.theta,
              SK_ERR_ARG);
    RerotParams p{};
    p.tA = table_device(from);
    p.tB = table_device(to);
    p.maxA = ca.max_positions;
    p.maxB = cb.max_positions;
    const double mu_a = mscale_of(ca);
    p.inv_muA2 = float(1.0 / (mu_a * mu_a));
    return launch_rerotation(layers, n_layers, ca, false, p, static_cast<cudaStream_t>(stream));
}

extern "C" sk_status sk_kv_shift_recent(const sk_kv_layer* layers, int32_t n_layers, const sk_rope_table* table,
                                        int32_t delta, void* stream) {
    SK_RET_IF(layers == nullptr || table == nullptr, SK_ERR_ARG);
    const sk_rope_config& c = table_config(table);
    const int64_t mag = delta < 0 ? -int64_t(delta) : int64_t(delta);
    SK_RET_IF(mag >= c.max_positions, SK_ERR_POSITION_RANGE);
    RerotParams p{};
    p.tA = p.tB = table_device(table);
    p.maxA = p.maxB = c.max_positions;
    const double mu = mscale_of(c);
    p.inv_muA2 = float(1.0 / (mu * mu));
    p.shift = 1;
    p.rowA = delta < 0 ? mag : 0;
    p.rowB = delta > 0 ? mag : 0;
    if (delta == 0) {  // nothing to turn; the arguments are still checked
        p.n_layers = 0;
        SK_RET_IF(n_layers < 1 || n_layers > kMaxLayers, SK_ERR_ARG);
        for (int l = 0; l < n_layers; ++l) SK_RET_IF(layers[l].kind != SK_LAYER_RING, SK_ERR_ARG);
        return SK_OK;
    }
    return launch_rerotation(layers, n_layers, c, true, p, static_cast<cudaStream_t>(stream));
}
