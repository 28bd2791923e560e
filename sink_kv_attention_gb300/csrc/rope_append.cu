// RoPE apply and fused RoPE + KV append (ring with pinned sinks, or global prefix).
//
// "RoPE, scaling, sliding window, attention sinks": the rotation listing
// (o1 = x1 cos - x2 sin, o2 = x2 cos + x1 sin), NeoX vs GPT-J pairing, partial rotary,
// table gather with no trigonometry at runtime, and one counter for angle and slot.
// "Inference & 128K Long Context", MixedKVCache: the ring's head/count rules and the
// global prefix; "Attention Sink 与 Streaming KV Cache": S pinned sink slots.
//
// Work layout: a row (one head of one token, head_dim elements) is handled by
// LPR = head_dim / (16 bytes / element size) lanes, each holding one 16-byte vector,
// so every load and store is a coalesced 16-byte access.  A NeoX pair (j, j + r/2)
// lives in two lanes of the same row; the partner's vector arrives by shuffle.
#include "rope_lane.cuh"

namespace sk {
namespace {

constexpr unsigned kFull = 0xffffffffu;
constexpr int kThreads = 256;
constexpr int kWarps = kThreads / 32;

// ---------------------------------------------------------------------------
// rope_apply: in-place rotation of x [n_tok][H][D].
// ---------------------------------------------------------------------------

struct ApplyParams {
    const float2* table;
    int64_t max_pos;
    int rotary_dim;
    void* x;
    int64_t n_tok;
    int H;
    const int64_t* positions;
    uint32_t* err;
};

constexpr int kApplyPasses = 4;  // row groups of a token each warp loads before rotating

// One warp per token (grid-stride): the token's position and this lane's (cos, sin)
// pairs are read once, then the token's H rows go through in passes of kApplyPasses
// row groups whose loads are all issued before the first rotation.
template <typename T, int D, bool NEOX>
__global__ void __launch_bounds__(kThreads) rope_apply_kernel(ApplyParams p) {
    using L = RowLayout<T, D>;
    constexpr int TCH = table_chunks<T, NEOX>();
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const int c = lane % L::LPR, rw = lane / L::LPR;
    const int half = p.rotary_dim / 2;
    int j0 = 0;
    const bool rot_lane = lane_pairs<T, D, NEOX>(p.rotary_dim, c, &j0);
    T* x = static_cast<T*>(p.x);
    for (int64_t tok = int64_t(blockIdx.x) * kWarps + warp; tok < p.n_tok; tok += int64_t(gridDim.x) * kWarps) {
        uint4* xt = reinterpret_cast<uint4*>(x + tok * p.H * D) + c;  // this lane's chunk of row 0
        const int64_t P = p.positions[tok];
        const bool ok = P >= 0 && P < p.max_pos;  // the same in every lane
        if (!ok) {
            if (lane == 0) set_error(p.err, SK_DEVERR_POSITION_RANGE);
            continue;
        }
        float4 cs[TCH];
        const float4* trow = reinterpret_cast<const float4*>(p.table + P * half + j0);
#pragma unroll
        for (int i = 0; i < TCH; ++i) cs[i] = rot_lane ? __ldg(trow + i) : make_float4(0.f, 0.f, 0.f, 0.f);
        for (int r0 = 0; r0 < p.H; r0 += kApplyPasses * L::RPW) {
            uint4 raw[kApplyPasses];
#pragma unroll
            for (int u = 0; u < kApplyPasses; ++u) {
                const int r = r0 + u * L::RPW + rw;
                raw[u] = r < p.H ? xt[r * (D / L::VEC)] : make_uint4(0, 0, 0, 0);
            }
#pragma unroll
            for (int u = 0; u < kApplyPasses; ++u) {
                const int r = r0 + u * L::RPW + rw;
                float f[L::VEC];
                ElemIO<T>::unpack(raw[u], f);
                rotate_lane<T, D, NEOX>(f, raw[u], cs, p.rotary_dim, c, lane, r < p.H);  // every lane shuffles
                if (r < p.H) xt[r * (D / L::VEC)] = ElemIO<T>::pack(f);
            }
        }
    }
}

// ---------------------------------------------------------------------------
// kv_append: rotate q (in place) and k (in place), write k and v into the cache.
// ---------------------------------------------------------------------------

struct AppendParams {
    const float2* table;
    int64_t max_pos;
    int rotary_dim;
    void* q;
    void* k;
    const void* v;
    int Hq, Hkv, T, B;
    void* kc;
    void* vc;
    float* kscale;
    int64_t cap;
    int S, W, kind;
    int32_t* head;
    int32_t* count;
    int64_t* pos;
    uint32_t* err;
    int fused_state;
    // paged layers (kind kKindPaged): pools in kc / vc, lengths in pos
    const int32_t* block_table;
    int max_blocks, bs, bs_log2;  // block_size = 1 << bs_log2
    int64_t n_blocks;
};


struct SeqState {
    int64_t pos;
    int head, count;
    bool ok;
    uint32_t err_bits;
};

__device__ __forceinline__ SeqState load_state(const AppendParams& p, int b) {
    SeqState s;
    s.pos = p.pos[b];
    s.head = p.kind == SK_LAYER_RING ? p.head[b] : 0;
    s.count = p.kind == SK_LAYER_RING ? p.count[b] : 0;
    s.err_bits = 0;
    if (s.pos < 0 || s.pos + p.T > p.max_pos) s.err_bits |= SK_DEVERR_POSITION_RANGE;
    if (p.kind == SK_LAYER_GLOBAL && s.pos + p.T > p.cap) s.err_bits |= SK_DEVERR_CAPACITY;
    if (p.kind == kKindPaged && s.pos + p.T > int64_t(p.max_blocks) * p.bs) s.err_bits |= SK_DEVERR_CAPACITY;
    s.ok = s.err_bits == 0;
    return s;
}

// Slot of chunk token t, or -1 when a long chunk drops it (ring rules in the header).
__device__ __forceinline__ int64_t token_slot(const AppendParams& p, const SeqState& s, int t) {
    const int64_t P = s.pos + t;
    if (p.kind == SK_LAYER_GLOBAL) return P;
    if (P < p.S) return P;
    const int64_t t0 = max(int64_t(0), min(int64_t(p.T), int64_t(p.S) - s.pos));
    const int64_t n = p.T - t0;
    const int64_t u = t - t0;
    if (n >= p.W) {
        if (u < n - p.W) return -1;
        return p.S + (u - (n - p.W));
    }
    return p.S + (s.head + u) % p.W;
}

// Cache row of kv head 0 for chunk token t and the row stride between kv heads; ok is
// false when the token is not stored (dropped by a long ring chunk, or a paged block id
// outside the pool, which also sets *bad_block).
struct CacheRow {
    int64_t base, hstride;
    bool ok;
};

template <bool PAGED>
__device__ __forceinline__ CacheRow cache_row(const AppendParams& p, const SeqState& s, int b, int t,
                                              bool* bad_block) {
    if constexpr (PAGED) {
        // "vLLM, from the inside out", PagedAttention: position P lives in request block
        // P / block_size at row P % block_size; the pool is [block][kv head][row][dim].
        const int64_t P = s.pos + t;
        const int32_t blk = p.block_table[int64_t(b) * p.max_blocks + (P >> p.bs_log2)];
        if (blk < 0 || blk >= p.n_blocks) {
            *bad_block = true;
            return CacheRow{0, 0, false};
        }
        return CacheRow{int64_t(blk) * p.Hkv * p.bs + (P & (p.bs - 1)), p.bs, true};
    } else {
        const int64_t slot = token_slot(p, s, t);
        return CacheRow{int64_t(b) * p.Hkv * p.cap + slot, p.cap, slot >= 0};
    }
}

__device__ __forceinline__ void advance_state(const AppendParams& p, const SeqState& s, int b) {
    if (!s.ok) {
        set_error(p.err, s.err_bits);
        return;
    }
    if (p.kind == SK_LAYER_RING) {
        const int64_t t0 = max(int64_t(0), min(int64_t(p.T), int64_t(p.S) - s.pos));
        const int64_t n = p.T - t0;
        if (n >= p.W) {
            p.head[b] = 0;
            p.count[b] = p.W;
        } else {
            p.head[b] = int((s.head + n) % p.W);
            p.count[b] = int(min(int64_t(p.W), s.count + n));
        }
    }
    p.pos[b] = s.pos + p.T;
}

template <typename KC> struct CacheStore;

template <> struct CacheStore<float> {
    template <int VEC>
    __device__ __forceinline__ static void store(void* base, int64_t elem, const float* f) {
        static_assert(VEC == 4, "f32 cache takes f32 rows");
        *reinterpret_cast<uint4*>(static_cast<float*>(base) + elem) = ElemIO<float>::pack(f);
    }
};

template <> struct CacheStore<__nv_bfloat16> {
    template <int VEC>
    __device__ __forceinline__ static void store(void* base, int64_t elem, const float* f) {
        static_assert(VEC == 8, "bf16 cache takes bf16 rows");
        *reinterpret_cast<uint4*>(static_cast<__nv_bfloat16*>(base) + elem) =
            ElemIO<__nv_bfloat16>::pack(f);
    }
};

constexpr int kAppendStages = 4;  // tokens in flight per block

// Shared memory of the append kernel: kAppendStages stages of one token's q, k and v
// rows (q first, then k, then v), plus the stage barriers.
template <typename IO> constexpr size_t append_stage_bytes(int hq, int hkv, int D) {
    return size_t(hq + 2 * hkv) * D * sizeof(IO);
}

// One block per (sequence, share of its tokens).  Lane 0 of the last warp streams each
// token's q, k and v rows (contiguous per tensor) into a kAppendStages-deep ring of
// shared-memory stages with 1-D bulk copies; the other warps rotate the rows out of
// shared memory (LPR lanes per row, 16-byte vectors, the NeoX partner vector by
// shuffle), write q and k back in place and k, v into the cache.
template <typename IO, typename KC, typename VC, int D, bool NEOX, bool PAGED>
__global__ void __launch_bounds__(kThreads + 32) kv_append_kernel(AppendParams p) {
    using L = RowLayout<IO, D>;
    constexpr int VEC = L::VEC;
    constexpr int TCH = table_chunks<IO, NEOX>();
    extern __shared__ __align__(128) uint8_t smem_raw[];
    const int b = blockIdx.y;
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const int c = lane % L::LPR, rw = lane / L::LPR;
    const int half = p.rotary_dim / 2;
    const int hq = p.q != nullptr ? p.Hq : 0;
    const int rows_per_tok = hq + 2 * p.Hkv;
    const size_t rows_bytes = size_t(rows_per_tok) * D * sizeof(IO);
    const size_t stage_bytes = rows_bytes + size_t(half) * sizeof(float2);  // rows, then the cos/sin row
    uint64_t* full_bar = reinterpret_cast<uint64_t*>(smem_raw + kAppendStages * stage_bytes);
    uint64_t* empty_bar = full_bar + kAppendStages;
    if (threadIdx.x == 0) {
        for (int st = 0; st < kAppendStages; ++st) {
            mbar_init(&full_bar[st], 1);
            mbar_init(&empty_bar[st], kWarps);
        }
        fence_barrier_init();
    }
    pdl_trigger();  // the attention after this kernel may launch and run its prologue
    if (warp == kWarps && lane == 0 && p.T == 1 && gridDim.x == 1) {
        // A one-token append (a decode step): warm L2 with the token's rows and, at the
        // position the state shows now, its cos/sin row, while earlier kernels finish.
        // Only a hint: the copies after the wait read whatever is final.
        const int64_t tok = int64_t(b);
        if (hq > 0) bulk_prefetch_l2(static_cast<const IO*>(p.q) + tok * p.Hq * D, uint32_t(hq * D * sizeof(IO)));
        bulk_prefetch_l2(static_cast<const IO*>(p.k) + tok * p.Hkv * D, uint32_t(p.Hkv * D * sizeof(IO)));
        bulk_prefetch_l2(static_cast<const IO*>(p.v) + tok * p.Hkv * D, uint32_t(p.Hkv * D * sizeof(IO)));
        const int64_t guess = p.pos[b];
        if (half > 0 && guess >= 0 && guess < p.max_pos)
            bulk_prefetch_l2(p.table + guess * half, uint32_t(half * sizeof(float2)));
    }
    pdl_wait();     // earlier kernels (the previous step's attention) are done
    __syncthreads();
    const SeqState s = load_state(p, b);
    const int n_tok = s.ok ? p.T : 0;
    bool timed_out = false;
    bool bad_block = false;

    IO* q = static_cast<IO*>(p.q);
    IO* k = static_cast<IO*>(p.k);
    const IO* v = static_cast<const IO*>(p.v);

    if (warp == kWarps) {
        // ------------------------------ producer ------------------------------
        if (lane == 0) {
            const uint64_t policy = l2_policy_evict_first();
            int st = 0;
            uint32_t phase = 0;
            for (int t = blockIdx.x; t < n_tok; t += gridDim.x) {
                if (!mbar_wait_bounded(&empty_bar[st], phase ^ 1)) timed_out = true;
                uint8_t* dst = smem_raw + st * stage_bytes;
                const int64_t tok = int64_t(b) * p.T + t;
                mbar_arrive_expect_tx(&full_bar[st], uint32_t(stage_bytes));
                if (hq > 0)
                    bulk_copy_g2s(dst, q + tok * p.Hq * D, uint32_t(hq * D * sizeof(IO)), &full_bar[st], policy);
                bulk_copy_g2s(dst + size_t(hq) * D * sizeof(IO), k + tok * p.Hkv * D,
                              uint32_t(p.Hkv * D * sizeof(IO)), &full_bar[st], policy);
                bulk_copy_g2s(dst + size_t(hq + p.Hkv) * D * sizeof(IO), v + tok * p.Hkv * D,
                              uint32_t(p.Hkv * D * sizeof(IO)), &full_bar[st], policy);
                if (half > 0)  // no table row when the keys come rotated
                    bulk_copy_g2s_nohint(dst + rows_bytes, p.table + (s.pos + t) * half, uint32_t(half * sizeof(float2)),
                                     &full_bar[st]);
                if (++st == kAppendStages) { st = 0; phase ^= 1; }
            }
            for (int i = 0; i < kAppendStages; ++i) {  // drain: no copy in flight at exit
                if (!mbar_wait_bounded(&empty_bar[st], phase ^ 1)) timed_out = true;
                if (++st == kAppendStages) { st = 0; phase ^= 1; }
            }
        }
    } else {
        // ------------------------------ consumers -----------------------------
        int j0 = 0;
        const bool rot_lane = lane_pairs<IO, D, NEOX>(p.rotary_dim, c, &j0);
        int st = 0;
        uint32_t phase = 0;
        for (int t = blockIdx.x; t < n_tok; t += gridDim.x) {
            const CacheRow crw = cache_row<PAGED>(p, s, b, t, &bad_block);
            const int64_t tok = int64_t(b) * p.T + t;
            // per-token bases; rows below add small per-row offsets only
            IO* qtok = q + tok * p.Hq * D;
            IO* ktok = k + tok * p.Hkv * D;
            if (!mbar_wait_bounded(&full_bar[st], phase)) timed_out = true;
            const uint8_t* stage = smem_raw + st * stage_bytes;
            // this lane's (cos, sin) pairs of position pos + t, copied in with the rows
            float4 cs[TCH];
            const float4* trow = reinterpret_cast<const float4*>(stage + rows_bytes) + j0 / 2;
            if constexpr (TCH == 4) {
                // The 8 lanes of a quarter warp read 64-byte-strided pieces of the row, which
                // fall on 2 of the 8 bank groups (4 wavefronts a load, in every quarter). Each
                // lane takes its 4 chunks starting at chunk m = (piece / 2) mod 4 instead, so a
                // load touches 8 distinct groups, and then undoes the rotation in registers
                // (measured: the prefill-chunk append 5010-5070 -> 5590-5640 GB/s).
                const int m = (j0 / 16) & 3;
                float4 t[4], u[4];
#pragma unroll
                for (int i = 0; i < 4; ++i) t[i] = rot_lane ? trow[(i + m) & 3] : make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
                for (int j = 0; j < 4; ++j) u[j] = (m & 1) ? t[(j + 3) & 3] : t[j];  // u[j] = chunk j + (m & 2)
#pragma unroll
                for (int j = 0; j < 4; ++j) cs[j] = (m & 2) ? u[(j + 2) & 3] : u[j];  // cs[j] = chunk j
            } else {
#pragma unroll
                for (int i = 0; i < TCH; ++i) cs[i] = rot_lane ? trow[i] : make_float4(0.f, 0.f, 0.f, 0.f);
            }
            for (int r0 = warp * L::RPW; r0 < rows_per_tok; r0 += kWarps * L::RPW) {
                const int r = r0 + rw;  // uniform trip count per warp; lanes past the token idle
                const bool live = r < rows_per_tok;
                const int which = r < hq ? 0 : (r < hq + p.Hkv ? 1 : 2);
                const int h = which == 0 ? r : (which == 1 ? r - hq : r - hq - p.Hkv);
                const uint4* srow = reinterpret_cast<const uint4*>(stage + size_t(r) * D * sizeof(IO));
                const uint4 raw = live ? srow[c] : make_uint4(0, 0, 0, 0);
                float f[VEC];
                ElemIO<IO>::unpack(raw, f);
                rotate_lane<IO, D, NEOX, true>(f, raw, cs, p.rotary_dim, c, lane, live && which < 2, srow);
                const uint4 out = ElemIO<IO>::pack(f);
                if (live && which == 0) reinterpret_cast<uint4*>(qtok + h * D)[c] = out;
                if (live && which == 1) reinterpret_cast<uint4*>(ktok + h * D)[c] = out;
                const int64_t crow = crw.base + int64_t(h) * crw.hstride;  // cache row index
                const bool store_kv = live && which != 0 && crw.ok;
                if constexpr (sizeof(KC) == 1) {
                    // int8 K: symmetric absmax over the row, codes rint(x * 127 / max|x|), ties to even.
                    float amax = 0.0f;
#pragma unroll
                    for (int i = 0; i < VEC; ++i) amax = fmaxf(amax, fabsf(f[i]));
#pragma unroll
                    for (int o = L::LPR / 2; o > 0; o >>= 1) amax = fmaxf(amax, __shfl_xor_sync(kFull, amax, o));
                    if (store_kv && which == 1) {
                        float scale, inv;
                        int8_row_scale(amax, &scale, &inv);
                        uint32_t w[VEC / 4];
#pragma unroll
                        for (int i = 0; i < VEC / 4; ++i) w[i] = float4_to_codes(f + 4 * i, inv);
                        int8_t* dst = static_cast<int8_t*>(p.kc) + crow * D + c * VEC;
                        if constexpr (VEC == 8)
                            *reinterpret_cast<uint2*>(dst) = make_uint2(w[0], w[1]);
                        else
                            *reinterpret_cast<uint32_t*>(dst) = w[0];
                        if (c == 0) p.kscale[crow] = scale;
                    }
                } else {
                    if (store_kv && which == 1)
                        reinterpret_cast<uint4*>(static_cast<KC*>(p.kc) + crow * D)[c] = out;
                }
                if (store_kv && which == 2) reinterpret_cast<uint4*>(static_cast<VC*>(p.vc) + crow * D)[c] = raw;
            }
            __syncwarp();
            if (lane == 0) mbar_arrive(&empty_bar[st]);
            if (++st == kAppendStages) { st = 0; phase ^= 1; }
        }
    }
    if (timed_out) set_error(p.err, SK_DEVERR_TIMEOUT);
    if (bad_block) set_error(p.err, SK_DEVERR_BLOCK_TABLE);
    if (p.fused_state) {
        __syncthreads();  // every thread has read the state before it changes
        if (threadIdx.x == 0) advance_state(p, s, b);
    }
}

__global__ void kv_append_state_kernel(AppendParams p) {
    const int b = blockIdx.x * blockDim.x + threadIdx.x;
    if (b >= p.B) return;
    const SeqState s = load_state(p, b);
    advance_state(p, s, b);
}

bool aligned16(const void* ptr) { return (reinterpret_cast<uintptr_t>(ptr) & 15u) == 0; }

template <typename T, int D, bool NEOX>
cudaError_t launch_apply(const ApplyParams& p, cudaStream_t st) {
    int64_t blocks = (p.n_tok + kWarps - 1) / kWarps;  // one warp per token
    blocks = std::min<int64_t>(blocks, int64_t(device_sm_count()) * 8);
    if (blocks < 1) blocks = 1;
    rope_apply_kernel<T, D, NEOX><<<unsigned(blocks), kThreads, 0, st>>>(p);
    return cudaGetLastError();
}

template <typename IO, typename KC, typename VC, int D, bool NEOX, bool PAGED>
cudaError_t launch_append(AppendParams p, cudaStream_t st) {
    const int hq = p.q != nullptr ? p.Hq : 0;
    const size_t smem = kAppendStages * (append_stage_bytes<IO>(hq, p.Hkv, D) + size_t(p.rotary_dim / 2) * 8) +
                        2 * kAppendStages * 8;
    if (smem > 200 * 1024) return cudaErrorInvalidValue;  // more heads than the stages can hold
    static PerDevice<cudaError_t> attr_cache;
    const cudaError_t attr = set_smem_limit_once(attr_cache, kv_append_kernel<IO, KC, VC, D, NEOX, PAGED>, 200 * 1024);
    if (attr != cudaSuccess) return attr;
    // blocks per sequence: one when a single block covers the tokens (it then also
    // advances the state), else enough blocks to fill the GPU
    int64_t gx = p.T <= kAppendStages ? 1 : std::min<int64_t>(p.T, std::max<int64_t>(1, 2 * device_sm_count() / p.B));
    p.fused_state = gx == 1 ? 1 : 0;
    dim3 grid(unsigned(gx), unsigned(p.B));
    cudaError_t e = launch_pdl(kv_append_kernel<IO, KC, VC, D, NEOX, PAGED>, grid, dim3(kThreads + 32), smem, st, p);
    if (e != cudaSuccess || p.fused_state) return e;
    kv_append_state_kernel<<<(p.B + 127) / 128, 128, 0, st>>>(p);
    return cudaGetLastError();
}

template <typename IO, typename KC, typename VC>
cudaError_t dispatch_append(const AppendParams& p, int D, bool neox, cudaStream_t st) {
    // paged layers get their own instantiation, so the ring/global kernel keeps its
    // register budget (two blocks per SM)
    if constexpr (sizeof(KC) != 1) {
        if (p.kind == kKindPaged) {
            if (D == 64)
                return neox ? launch_append<IO, KC, VC, 64, true, true>(p, st)
                            : launch_append<IO, KC, VC, 64, false, true>(p, st);
            return neox ? launch_append<IO, KC, VC, 128, true, true>(p, st)
                        : launch_append<IO, KC, VC, 128, false, true>(p, st);
        }
    }
    if (D == 64)
        return neox ? launch_append<IO, KC, VC, 64, true, false>(p, st)
                    : launch_append<IO, KC, VC, 64, false, false>(p, st);
    return neox ? launch_append<IO, KC, VC, 128, true, false>(p, st)
                : launch_append<IO, KC, VC, 128, false, false>(p, st);
}

}  // namespace
}  // namespace sk

using namespace sk;

extern "C" sk_status sk_rope_apply(const sk_rope_table* table, void* x, int32_t dtype, int64_t n_tok,
                                   int32_t n_heads, const int64_t* positions, uint32_t* err,
                                   void* stream) {
    SK_RET_IF(table == nullptr, SK_ERR_ARG);
    SK_RET_IF(n_tok < 0 || n_heads < 1, SK_ERR_ARG);
    SK_RET_IF(dtype != SK_BF16 && dtype != SK_F32, SK_ERR_UNSUPPORTED);
    if (n_tok == 0) return SK_OK;  // nothing is read: x and positions may be NULL
    SK_RET_IF(x == nullptr || positions == nullptr, SK_ERR_ARG);
    SK_RET_IF(!aligned16(x), SK_ERR_ARG);
    const sk_rope_config& c = table_config(table);
    ApplyParams p{table_device(table), c.max_positions, c.rotary_dim, x, n_tok, n_heads, positions, err};
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    cudaError_t e;
    const bool neox = c.neox != 0;
    if (dtype == SK_BF16) {
        if (c.head_dim == 64)
            e = neox ? launch_apply<__nv_bfloat16, 64, true>(p, st) : launch_apply<__nv_bfloat16, 64, false>(p, st);
        else
            e = neox ? launch_apply<__nv_bfloat16, 128, true>(p, st) : launch_apply<__nv_bfloat16, 128, false>(p, st);
    } else {
        if (c.head_dim == 64)
            e = neox ? launch_apply<float, 64, true>(p, st) : launch_apply<float, 64, false>(p, st);
        else
            e = neox ? launch_apply<float, 128, true>(p, st) : launch_apply<float, 128, false>(p, st);
    }
    return e == cudaSuccess ? SK_OK : SK_ERR_CUDA;
}

namespace {

sk_status run_append(const AppendParams& p, const sk_rope_config& c, int io_dtype, int k_dtype, int v_dtype,
                     int head_dim, cudaStream_t st) {
    const bool neox = c.neox != 0;
    cudaError_t e;
    if (io_dtype == SK_F32 && k_dtype == SK_F32 && v_dtype == SK_F32)
        e = dispatch_append<float, float, float>(p, head_dim, neox, st);
    else if (io_dtype == SK_BF16 && k_dtype == SK_BF16 && v_dtype == SK_BF16)
        e = dispatch_append<__nv_bfloat16, __nv_bfloat16, __nv_bfloat16>(p, head_dim, neox, st);
    else if (io_dtype == SK_BF16 && k_dtype == SK_I8 && v_dtype == SK_BF16 && p.kind != kKindPaged)
        e = dispatch_append<__nv_bfloat16, int8_t, __nv_bfloat16>(p, head_dim, neox, st);
    else
        return SK_ERR_UNSUPPORTED;
    return e == cudaSuccess ? SK_OK : SK_ERR_CUDA;
}

}  // namespace

extern "C" sk_status sk_kv_append(const sk_rope_table* table, const sk_kv_layer* layer, void* q,
                                  int32_t n_q_heads, void* k, const void* v, int32_t io_dtype,
                                  int32_t T, void* stream) {
    SK_RET_IF(layer == nullptr || T < 0, SK_ERR_ARG);
    SK_RET_IF(T > 0 && (k == nullptr || v == nullptr), SK_ERR_ARG);  // T = 0: k, v may be NULL
    SK_RET_IF(table == nullptr && q != nullptr, SK_ERR_ARG);  // nothing would rotate q
    const sk_kv_layer& L = *layer;
    // Without a table the keys come rotated: an identity "rotation" (no rotary dims)
    // and no position limit but the counter's own.
    sk_rope_config c{};
    if (table != nullptr) {
        c = table_config(table);
    } else {
        SK_RET_IF(L.head_dim != 64 && L.head_dim != 128, SK_ERR_UNSUPPORTED);
        c.head_dim = L.head_dim;
        c.rotary_dim = 0;
        c.neox = 1;
        c.max_positions = int64_t(1) << 62;
    }
    SK_RET_IF(L.k == nullptr || L.v == nullptr || L.pos == nullptr, SK_ERR_ARG);
    SK_RET_IF(L.batch < 1 || L.n_kv_heads < 1 || T < 0, SK_ERR_ARG);
    SK_RET_IF(L.head_dim != c.head_dim, SK_ERR_ARG);
    if (L.kind == SK_LAYER_RING) {
        SK_RET_IF(L.head == nullptr || L.count == nullptr, SK_ERR_ARG);
        SK_RET_IF(L.sinks < 0 || L.window < 1, SK_ERR_ARG);
        SK_RET_IF(L.capacity != int64_t(L.sinks) + L.window, SK_ERR_ARG);
    } else if (L.kind == SK_LAYER_GLOBAL) {
        SK_RET_IF(L.capacity < 1, SK_ERR_ARG);
    } else {
        return SK_ERR_ARG;
    }
    if (q != nullptr) SK_RET_IF(n_q_heads < 1 || n_q_heads % L.n_kv_heads != 0, SK_ERR_ARG);
    SK_RET_IF(!aligned16(k) || !aligned16(v) || !aligned16(L.k) || !aligned16(L.v), SK_ERR_ARG);  // NULL passes
    SK_RET_IF(q != nullptr && !aligned16(q), SK_ERR_ARG);
    if (L.k_dtype == SK_I8) SK_RET_IF(L.k_scale == nullptr, SK_ERR_ARG);
    if (T == 0) return SK_OK;

    AppendParams p{};
    p.table = table != nullptr ? table_device(table) : nullptr;
    p.max_pos = c.max_positions;
    p.rotary_dim = c.rotary_dim;
    p.q = q;
    p.k = k;
    p.v = v;
    p.Hq = n_q_heads;
    p.Hkv = L.n_kv_heads;
    p.T = T;
    p.B = L.batch;
    p.kc = L.k;
    p.vc = L.v;
    p.kscale = L.k_scale;
    p.cap = L.capacity;
    p.S = L.sinks;
    p.W = L.window;
    p.kind = L.kind;
    p.head = L.head;
    p.count = L.count;
    p.pos = L.pos;
    p.err = L.err;
    return run_append(p, c, io_dtype, L.k_dtype, L.v_dtype, L.head_dim, static_cast<cudaStream_t>(stream));
}

extern "C" sk_status sk_paged_append(const sk_rope_table* table, const sk_paged_layer* layer, void* q,
                                     int32_t n_q_heads, const void* k, const void* v, int32_t io_dtype,
                                     int32_t T, void* stream) {
    SK_RET_IF(table == nullptr || layer == nullptr || T < 0, SK_ERR_ARG);
    SK_RET_IF(T > 0 && (k == nullptr || v == nullptr), SK_ERR_ARG);  // T = 0: k, v may be NULL
    const sk_paged_layer& L = *layer;
    const sk_rope_config& c = table_config(table);
    SK_RET_IF(paged_layer_check(L) != SK_OK, SK_ERR_ARG);
    SK_RET_IF(L.head_dim != c.head_dim || T < 0, SK_ERR_ARG);
    if (q != nullptr) SK_RET_IF(n_q_heads < 1 || n_q_heads % L.n_kv_heads != 0 || !aligned16(q), SK_ERR_ARG);
    SK_RET_IF(!aligned16(k) || !aligned16(v), SK_ERR_ARG);
    if (T == 0) return SK_OK;
    AppendParams p{};
    p.table = table_device(table);
    p.max_pos = c.max_positions;
    p.rotary_dim = c.rotary_dim;
    p.q = q;
    p.k = const_cast<void*>(k);
    p.v = v;
    p.Hq = n_q_heads;
    p.Hkv = L.n_kv_heads;
    p.T = T;
    p.B = L.batch;
    p.kc = L.k_pool;
    p.vc = L.v_pool;
    p.kind = kKindPaged;
    p.pos = L.seq_lens;
    p.err = L.err;
    p.block_table = L.block_table;
    p.max_blocks = L.max_blocks;
    p.bs = L.block_size;
    p.bs_log2 = __builtin_ctz(unsigned(L.block_size));
    p.n_blocks = L.n_blocks;
    return run_append(p, c, io_dtype, L.k_dtype, L.v_dtype, L.head_dim, static_cast<cudaStream_t>(stream));
}
