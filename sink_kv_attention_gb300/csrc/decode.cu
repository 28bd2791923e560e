// Split-K (flash-decoding) GQA decode attention over the sink ∪ recent visible set.
//
// "Attention Sink 与 Streaming KV Cache", visible set V(P): in a ring layer after the
// query's own append the occupied slots [0, min(pos, S) + count) are exactly V(P), and
// attention is order-free, so no chronological gather is needed.  A global layer
// reads rows [0, pos).  "KV-Cache Engineering", 4.3-4.4 and 5.5: decode is bound by
// the KV bytes it streams, and the n_rep query heads of a GQA group share each K/V
// row, broadcast in registers instead of repeat_kv's copy.
//
// Kernel 1 (persistent): work item = (sequence b, kv head g, row chunk).  One producer
// lane streams K and V tiles of consecutive rows (contiguous in HBM) with 1-D bulk
// copies into a STAGES-deep shared-memory ring guarded by mbarriers.  Consumer warps
// take TILE rows per stage: 8-lane groups compute partial q.k dot products for
// 8/NREP rows x NREP heads, a butterfly reduce-scatter leaves one finished score per
// lane, online softmax in base 2, then P.V with each lane owning D/32 dims of all
// NREP heads.  Per item the warps' (m, l, acc) are merged in shared memory and one
// partial goes to the workspace.
// Kernel 2: per (b, q head) log-sum-exp combine of the partials.
#include <algorithm>

#include "common.cuh"

namespace sk {
namespace {

constexpr unsigned kFull = 0xffffffffu;
constexpr float kLog2e = 1.4426950408889634f;

struct DecodeParams {
    const void* kc;
    const void* vc;
    const void* q;
    void* out;
    float* ws;
    const int32_t* count;
    const int64_t* pos;
    uint32_t* err;
    int64_t cap;
    int B, Hkv, S, kind;
    int chunk;     // rows per work item (multiple of TILE)
    int n_parts;   // work items per (b, g)
    float qscale;  // log2(e) / sqrt(D)
};

__device__ __forceinline__ int64_t visible_rows(const DecodeParams& p, int b) {
    const int64_t pos = p.pos[b];
    if (p.kind == SK_LAYER_GLOBAL) return min(pos, p.cap);
    return min(pos, int64_t(p.S)) + int64_t(p.count[b]);
}

// Consumer warps per block: 8 unless two stages of K+V tiles would not fit.
template <typename T, int D, int NREP> constexpr int decode_warps() {
    constexpr int warp_stage_bytes = 2 * (4 * (8 / NREP)) * D * int(sizeof(T));
    return 2 * 8 * warp_stage_bytes <= 200 * 1024 ? 8 : (2 * 4 * warp_stage_bytes <= 200 * 1024 ? 4 : 2);
}

template <typename T, int D, int NREP> struct DecodeCfg {
    static constexpr int NWARPS = decode_warps<T, D, NREP>();
    static constexpr int VEC = ElemIO<T>::kPerVec;    // elements per 16-byte chunk
    static constexpr int CHUNKS = D / VEC;            // 16-byte chunks per row
    static constexpr int CPL = CHUNKS / 8;            // chunks per lane (QK)
    static constexpr int DPL = D / 8;                 // dims per lane (QK)
    static constexpr int RPG = 8 / NREP;              // rows per 8-lane group
    static constexpr int RPW = 4 * RPG;               // rows per warp per stage
    static constexpr int TILE = NWARPS * RPW;         // rows per stage
    static constexpr int DPV = D / 32;                // dims per lane (PV)
    static constexpr int ROW_BYTES = D * int(sizeof(T));
    static constexpr int STAGE_BYTES = 2 * TILE * ROW_BYTES;   // K tile then V tile
    static constexpr int STAGES_FIT = (200 * 1024) / STAGE_BYTES;
    static constexpr int STAGES = STAGES_FIT > 5 ? 5 : STAGES_FIT;
    static_assert(STAGES >= 2, "stage too large");
    static constexpr int MERGE_FLOATS = NWARPS * NREP * (D + 2);
    static constexpr int PS_FLOATS = NWARPS * (RPW * NREP + NREP);
    static constexpr size_t SMEM = size_t(STAGES) * STAGE_BYTES + size_t(MERGE_FLOATS) * 4 +
                                   size_t(PS_FLOATS) * 4 + 2 * STAGES * 8 + 16;
    static constexpr int THREADS = (NWARPS + 1) * 32;
    static constexpr int PARTIAL_FLOATS = NREP * (D + 2);
    static_assert(CPL >= 1 && DPV >= 1, "head_dim too small for this layout");
};

// Load `n` floats of this lane's PV slice of a row from shared memory.
template <typename T, int DPV>
__device__ __forceinline__ void load_pv_slice(const T* row, int lane, float* v) {
    if constexpr (sizeof(T) == 2) {
        if constexpr (DPV == 4) {
            const uint2 u = *reinterpret_cast<const uint2*>(row + lane * 4);
            float2 a = bf16x2_to_float2(u.x), b = bf16x2_to_float2(u.y);
            v[0] = a.x; v[1] = a.y; v[2] = b.x; v[3] = b.y;
        } else {
            const uint32_t u = *reinterpret_cast<const uint32_t*>(row + lane * 2);
            float2 a = bf16x2_to_float2(u);
            v[0] = a.x; v[1] = a.y;
        }
    } else {
        if constexpr (DPV == 4) {
            const float4 u = *reinterpret_cast<const float4*>(row + lane * 4);
            v[0] = u.x; v[1] = u.y; v[2] = u.z; v[3] = u.w;
        } else {
            const float2 u = *reinterpret_cast<const float2*>(row + lane * 2);
            v[0] = u.x; v[1] = u.y;
        }
    }
}

template <typename T, int D, int NREP>
__global__ void __launch_bounds__(DecodeCfg<T, D, NREP>::THREADS, 1)
    decode_split_kernel(DecodeParams p) {
    using C = DecodeCfg<T, D, NREP>;
    constexpr int NWARPS = C::NWARPS;
    constexpr int STAGES = C::STAGES;
    extern __shared__ __align__(128) uint8_t smem[];
    uint8_t* stages = smem;
    float* merge = reinterpret_cast<float*>(smem + size_t(STAGES) * C::STAGE_BYTES);
    float* ps_all = merge + C::MERGE_FLOATS;
    uint64_t* full_bar = reinterpret_cast<uint64_t*>(ps_all + C::PS_FLOATS);
    uint64_t* empty_bar = full_bar + STAGES;

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    if (threadIdx.x == 0) {
        for (int s = 0; s < STAGES; ++s) {
            mbar_init(&full_bar[s], 1);
            mbar_init(&empty_bar[s], NWARPS);
        }
        fence_barrier_init();
    }
    __syncthreads();

    const int64_t n_items = int64_t(p.B) * p.Hkv * p.n_parts;
    bool timed_out = false;

    if (warp == NWARPS) {
        // ------------------------------ producer ------------------------------
        if (lane == 0) {
            const uint64_t policy = l2_policy_evict_first();
            int stage = 0;
            uint32_t phase = 0;
            for (int64_t it = blockIdx.x; it < n_items; it += gridDim.x) {
                const int part = int(it % p.n_parts);
                const int64_t unit = it / p.n_parts;  // b * Hkv + g
                const int b = int(unit / p.Hkv);
                const int64_t L = visible_rows(p, b);
                const int64_t r0 = int64_t(part) * p.chunk;
                const int64_t r1 = min(L, r0 + p.chunk);
                const T* kbase = static_cast<const T*>(p.kc) + unit * p.cap * D;
                const T* vbase = static_cast<const T*>(p.vc) + unit * p.cap * D;
                for (int64_t row = r0; row < r1; row += C::TILE) {
                    const uint32_t n = uint32_t(min(int64_t(C::TILE), r1 - row));
                    if (!mbar_wait_bounded(&empty_bar[stage], phase ^ 1)) timed_out = true;
                    uint8_t* dst = stages + size_t(stage) * C::STAGE_BYTES;
                    mbar_arrive_expect_tx(&full_bar[stage], 2u * n * C::ROW_BYTES);
                    bulk_copy_g2s(dst, kbase + row * D, n * C::ROW_BYTES, &full_bar[stage], policy);
                    bulk_copy_g2s(dst + C::TILE * C::ROW_BYTES, vbase + row * D, n * C::ROW_BYTES,
                                  &full_bar[stage], policy);
                    if (++stage == STAGES) { stage = 0; phase ^= 1; }
                }
            }
            // Drain: wait until the consumers released every stage, so no copy is in
            // flight into shared memory when the block exits.
            for (int s = 0; s < STAGES; ++s) {
                if (!mbar_wait_bounded(&empty_bar[stage], phase ^ 1)) timed_out = true;
                if (++stage == STAGES) { stage = 0; phase ^= 1; }
            }
            if (timed_out) set_error(p.err, SK_DEVERR_TIMEOUT);
        }
        return;
    }

    // -------------------------------- consumers --------------------------------
    const int gi = lane >> 3, l8 = lane & 7;
    float* ps = ps_all + warp * (C::RPW * NREP + NREP);  // p[RPW][NREP] then alpha[NREP]
    // score owned by this lane after the reduce-scatter: row l8 / NREP of the group, head l8 % NREP
    const int my_j = l8 / NREP, my_h = l8 % NREP;
    const int my_row = gi * C::RPG + my_j;  // warp-local row of that score
    const T* qbase = static_cast<const T*>(p.q);
    int stage = 0;
    uint32_t phase = 0;

    for (int64_t it = blockIdx.x; it < n_items; it += gridDim.x) {
        const int part = int(it % p.n_parts);
        const int64_t unit = it / p.n_parts;
        const int b = int(unit / p.Hkv), g = int(unit % p.Hkv);
        const int64_t L = visible_rows(p, b);
        const int64_t r0 = int64_t(part) * p.chunk;
        const int64_t r1 = min(L, r0 + p.chunk);
        if (r1 <= r0) continue;

        // q slice of this lane, all NREP heads, pre-scaled by log2(e)/sqrt(D).
        float2 q2[NREP][C::DPL / 2];
#pragma unroll
        for (int h = 0; h < NREP; ++h) {
            const T* qrow = qbase + ((int64_t(b) * p.Hkv + g) * NREP + h) * D;
#pragma unroll
            for (int i = 0; i < C::CPL; ++i) {
                const uint4 raw = reinterpret_cast<const uint4*>(qrow)[l8 + 8 * i];
                float f[C::VEC];
                ElemIO<T>::unpack(raw, f);
#pragma unroll
                for (int e = 0; e < C::VEC / 2; ++e)
                    q2[h][i * C::VEC / 2 + e] =
                        make_float2(f[2 * e] * p.qscale, f[2 * e + 1] * p.qscale);
            }
        }

        float m_run = -INFINITY;  // running max of this lane's head (base-2 logits)
        float l_run = 0.0f;       // this lane's share of the running denominator
        float2 acc[NREP][C::DPV / 2];
#pragma unroll
        for (int h = 0; h < NREP; ++h)
#pragma unroll
            for (int d = 0; d < C::DPV / 2; ++d) acc[h][d] = make_float2(0.f, 0.f);

        for (int64_t row0 = r0; row0 < r1; row0 += C::TILE) {
            const int n = int(min(int64_t(C::TILE), r1 - row0));
            if (!mbar_wait_bounded(&full_bar[stage], phase)) timed_out = true;
            const T* ktile = reinterpret_cast<const T*>(stages + size_t(stage) * C::STAGE_BYTES);
            const T* vtile = ktile + C::TILE * D;
            const int wrow0 = warp * C::RPW;           // first tile row of this warp
            const int nw = max(0, min(C::RPW, n - wrow0));  // valid rows of this warp

            // ---- QK: partial dots of RPG rows x NREP heads over this lane's dims ----
            float part_s[8];
#pragma unroll
            for (int j = 0; j < C::RPG; ++j) {
                const int lr = gi * C::RPG + j;
                float2 kf[C::DPL / 2];
                if (lr < nw) {
                    const uint4* krow = reinterpret_cast<const uint4*>(ktile + (wrow0 + lr) * D);
#pragma unroll
                    for (int i = 0; i < C::CPL; ++i) {
                        const uint4 raw = krow[l8 + 8 * i];
                        float f[C::VEC];
                        ElemIO<T>::unpack(raw, f);
#pragma unroll
                        for (int e = 0; e < C::VEC / 2; ++e)
                            kf[i * C::VEC / 2 + e] = make_float2(f[2 * e], f[2 * e + 1]);
                    }
                } else {
#pragma unroll
                    for (int e = 0; e < C::DPL / 2; ++e) kf[e] = make_float2(0.f, 0.f);
                }
#pragma unroll
                for (int h = 0; h < NREP; ++h) {
                    float2 a = make_float2(0.f, 0.f);
#pragma unroll
                    for (int e = 0; e < C::DPL / 2; ++e) a = __ffma2_rn(q2[h][e], kf[e], a);
                    part_s[j * NREP + h] = a.x + a.y;
                }
            }
            // ---- butterfly reduce-scatter over the 8 lanes: lane l8 keeps value l8 ----
            {
                const bool b4 = (l8 & 4) != 0;
                float r4[4];
#pragma unroll
                for (int i = 0; i < 4; ++i) {
                    const float send = b4 ? part_s[i] : part_s[i + 4];
                    const float keep = b4 ? part_s[i + 4] : part_s[i];
                    r4[i] = keep + __shfl_xor_sync(kFull, send, 4);
                }
                const bool b2 = (l8 & 2) != 0;
                float r2[2];
#pragma unroll
                for (int i = 0; i < 2; ++i) {
                    const float send = b2 ? r4[i] : r4[i + 2];
                    const float keep = b2 ? r4[i + 2] : r4[i];
                    r2[i] = keep + __shfl_xor_sync(kFull, send, 2);
                }
                const bool b1 = (l8 & 1) != 0;
                const float send = b1 ? r2[0] : r2[1];
                const float keep = b1 ? r2[1] : r2[0];
                part_s[0] = keep + __shfl_xor_sync(kFull, send, 1);
            }
            const float s = my_row < nw ? part_s[0] : -INFINITY;

            // ---- online softmax (base 2) for this lane's head ----
            float tmax = s;
#pragma unroll
            for (int o = NREP; o < 32; o <<= 1) tmax = fmaxf(tmax, __shfl_xor_sync(kFull, tmax, o));
            const float m_new = fmaxf(m_run, tmax);
            const float m_use = m_new == -INFINITY ? 0.0f : m_new;
            const float alpha = exp2f(m_run - m_use);
            const float pr = exp2f(s - m_use);
            m_run = m_new;
            l_run = l_run * alpha + pr;
            ps[my_row * NREP + my_h] = pr;
            if (lane < NREP) ps[C::RPW * NREP + lane] = alpha;  // lane h holds head h
            __syncwarp();

            // ---- PV: acc[h] = acc[h] * alpha[h] + sum_rows p[row][h] v[row] ----
#pragma unroll
            for (int h = 0; h < NREP; ++h) {
                const float a = ps[C::RPW * NREP + h];
#pragma unroll
                for (int d = 0; d < C::DPV / 2; ++d) acc[h][d] = __fmul2_rn(acc[h][d], make_float2(a, a));
            }
            for (int r = 0; r < nw; ++r) {
                float vf[C::DPV];
                load_pv_slice<T, C::DPV>(vtile + (wrow0 + r) * D, lane, vf);
                float pw[NREP];
                if constexpr (NREP == 4) {
                    const float4 t = *reinterpret_cast<const float4*>(ps + r * 4);
                    pw[0] = t.x; pw[1] = t.y; pw[2] = t.z; pw[3] = t.w;
                } else {
#pragma unroll
                    for (int h = 0; h < NREP; ++h) pw[h] = ps[r * NREP + h];
                }
#pragma unroll
                for (int h = 0; h < NREP; ++h)
#pragma unroll
                    for (int d = 0; d < C::DPV / 2; ++d)
                        acc[h][d] = __ffma2_rn(make_float2(pw[h], pw[h]),
                                               make_float2(vf[2 * d], vf[2 * d + 1]), acc[h][d]);
            }
            __syncwarp();
            if (lane == 0) mbar_arrive(&empty_bar[stage]);
            if (++stage == STAGES) { stage = 0; phase ^= 1; }
        }

        // ---- merge the warps' partial states and write one partial ----
        float l_tot = l_run;
#pragma unroll
        for (int o = NREP; o < 32; o <<= 1) l_tot += __shfl_xor_sync(kFull, l_tot, o);
        float* mw = merge + warp * NREP * (D + 2);
        if (lane < NREP) {
            mw[lane] = m_run;          // lane h holds head h's max and total
            mw[NREP + lane] = l_tot;
        }
#pragma unroll
        for (int h = 0; h < NREP; ++h)
#pragma unroll
            for (int d = 0; d < C::DPV / 2; ++d) {
                mw[2 * NREP + h * D + lane * C::DPV + 2 * d] = acc[h][d].x;
                mw[2 * NREP + h * D + lane * C::DPV + 2 * d + 1] = acc[h][d].y;
            }
        asm volatile("bar.sync 1, %0;" ::"n"(NWARPS * 32) : "memory");
        float* out = p.ws + it * C::PARTIAL_FLOATS;
        for (int idx = threadIdx.x; idx < NREP * D; idx += NWARPS * 32) {
            const int h = idx / D, d = idx % D;
            float M = -INFINITY;
            for (int w = 0; w < NWARPS; ++w) M = fmaxf(M, merge[w * NREP * (D + 2) + h]);
            const float Mu = M == -INFINITY ? 0.0f : M;
            float a = 0.0f, lsum = 0.0f;
            for (int w = 0; w < NWARPS; ++w) {
                const float* mm = merge + w * NREP * (D + 2);
                const float f = exp2f(mm[h] - Mu);
                a += f * mm[2 * NREP + h * D + d];
                lsum += f * mm[NREP + h];
            }
            out[2 * NREP + h * D + d] = a;
            if (d == 0) {
                out[h] = M;
                out[NREP + h] = lsum;
            }
        }
        asm volatile("bar.sync 1, %0;" ::"n"(NWARPS * 32) : "memory");
    }
    if (timed_out) set_error(p.err, SK_DEVERR_TIMEOUT);
}

// One warp per (b, q head): log-sum-exp combine of the valid partials.
template <typename T, int D, int NREP>
__global__ void decode_combine_kernel(DecodeParams p) {
    constexpr int DPV = D / 32;
    constexpr int PF = NREP * (D + 2);
    const int warp_global = blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5);
    const int lane = threadIdx.x & 31;
    const int Hq = p.Hkv * NREP;
    if (warp_global >= p.B * Hq) return;
    const int b = warp_global / Hq, hq = warp_global % Hq;
    const int g = hq / NREP, h = hq % NREP;
    const int64_t L = visible_rows(p, b);
    const int n_valid = int(min(int64_t(p.n_parts), (L + p.chunk - 1) / p.chunk));
    const float* base = p.ws + ((int64_t(b) * p.Hkv + g) * p.n_parts) * PF;
    float M = -INFINITY;
    for (int i = 0; i < n_valid; ++i) M = fmaxf(M, base[i * PF + h]);
    const float Mu = M == -INFINITY ? 0.0f : M;
    float acc[DPV];
#pragma unroll
    for (int d = 0; d < DPV; ++d) acc[d] = 0.0f;
    float lsum = 0.0f;
    for (int i = 0; i < n_valid; ++i) {
        const float* pp = base + i * PF;
        const float f = exp2f(pp[h] - Mu);
        lsum += f * pp[NREP + h];
#pragma unroll
        for (int d = 0; d < DPV; ++d) acc[d] += f * pp[2 * NREP + h * D + lane * DPV + d];
    }
    const float inv = lsum > 0.0f ? 1.0f / lsum : 0.0f;
    T* o = static_cast<T*>(p.out) + (int64_t(b) * Hq + hq) * D + lane * DPV;
#pragma unroll
    for (int d = 0; d < DPV; ++d) {
        if constexpr (sizeof(T) == 2)
            o[d] = __float2bfloat16_rn(acc[d] * inv);
        else
            o[d] = acc[d] * inv;
    }
}

template <typename T, int D, int NREP>
struct DecodeLaunch {
    using C = DecodeCfg<T, D, NREP>;

    static int blocks_per_sm() {
        static int cached = -1;
        if (cached < 0) {
            int n = 0;
            if (cudaFuncSetAttribute(decode_split_kernel<T, D, NREP>,
                                     cudaFuncAttributeMaxDynamicSharedMemorySize,
                                     int(C::SMEM)) != cudaSuccess)
                return 0;
            if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(
                    &n, decode_split_kernel<T, D, NREP>, C::THREADS, C::SMEM) !=
                cudaSuccess)
                return 0;
            cached = n;
        }
        return cached;
    }

    // Rows per work item and items per (b, g): aim for ~24 items per resident block so
    // the static round-robin leaves little tail, with at least one tile per item.
    static void plan(const sk_kv_layer& L, int& chunk, int& n_parts) {
        const int64_t units = int64_t(L.batch) * L.n_kv_heads;
        const int64_t resident = int64_t(std::max(1, blocks_per_sm())) * device_sm_count();
        const int64_t max_parts = (L.capacity + C::TILE - 1) / C::TILE;
        int64_t parts = (24 * resident + units - 1) / units;
        parts = std::max<int64_t>(1, std::min(parts, max_parts));
        int64_t ch = (L.capacity + parts - 1) / parts;
        ch = (ch + C::TILE - 1) / C::TILE * C::TILE;
        chunk = int(ch);
        n_parts = int((L.capacity + ch - 1) / ch);
    }

    static size_t workspace(const sk_kv_layer& L) {
        int chunk, n_parts;
        plan(L, chunk, n_parts);
        return size_t(L.batch) * L.n_kv_heads * n_parts * C::PARTIAL_FLOATS * sizeof(float);
    }

    static cudaError_t run(DecodeParams p, const sk_kv_layer& L, cudaStream_t st) {
        const int bps = blocks_per_sm();
        if (bps < 1) return cudaErrorInvalidConfiguration;
        plan(L, p.chunk, p.n_parts);
        const int64_t n_items = int64_t(L.batch) * L.n_kv_heads * p.n_parts;
        const int64_t grid = std::min<int64_t>(n_items, int64_t(bps) * device_sm_count());
        decode_split_kernel<T, D, NREP>
            <<<unsigned(grid), C::THREADS, C::SMEM, st>>>(p);
        cudaError_t e = cudaGetLastError();
        if (e != cudaSuccess) return e;
        const int warps = L.batch * L.n_kv_heads * NREP;
        decode_combine_kernel<T, D, NREP><<<(warps + 7) / 8, 256, 0, st>>>(p);
        return cudaGetLastError();
    }
};

template <typename T, int D>
bool dispatch(int nrep, bool want_ws, const sk_kv_layer& L, DecodeParams* p, cudaStream_t st,
              size_t* ws, cudaError_t* e) {
    switch (nrep) {
#define SK_CASE(N)                                                              \
    case N:                                                                     \
        if (want_ws) *ws = DecodeLaunch<T, D, N>::workspace(L);                 \
        else *e = DecodeLaunch<T, D, N>::run(*p, L, st);                        \
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
bool route(int io_dtype, const sk_kv_layer& L, int nrep, bool want_ws, DecodeParams* p,
           cudaStream_t st, size_t* ws, cudaError_t* e) {
    if (io_dtype == SK_BF16 && L.k_dtype == SK_BF16 && L.v_dtype == SK_BF16) {
        if (L.head_dim == 128) return dispatch<__nv_bfloat16, 128>(nrep, want_ws, L, p, st, ws, e);
        if (L.head_dim == 64) return dispatch<__nv_bfloat16, 64>(nrep, want_ws, L, p, st, ws, e);
    } else if (io_dtype == SK_F32 && L.k_dtype == SK_F32 && L.v_dtype == SK_F32) {
        if (L.head_dim == 128) return dispatch<float, 128>(nrep, want_ws, L, p, st, ws, e);
        if (L.head_dim == 64) return dispatch<float, 64>(nrep, want_ws, L, p, st, ws, e);
    }
    return false;
}

sk_status check_layer(const sk_kv_layer* layer, int32_t n_q_heads) {
    SK_RET_IF(layer == nullptr, SK_ERR_ARG);
    const sk_kv_layer& L = *layer;
    SK_RET_IF(L.k == nullptr || L.v == nullptr || L.pos == nullptr, SK_ERR_ARG);
    SK_RET_IF(L.batch < 1 || L.n_kv_heads < 1 || L.capacity < 1, SK_ERR_ARG);
    SK_RET_IF(n_q_heads < 1 || n_q_heads % L.n_kv_heads != 0, SK_ERR_ARG);
    if (L.kind == SK_LAYER_RING) {
        SK_RET_IF(L.count == nullptr || L.sinks < 0 || L.window < 1, SK_ERR_ARG);
        SK_RET_IF(L.capacity != int64_t(L.sinks) + L.window, SK_ERR_ARG);
    } else {
        SK_RET_IF(L.kind != SK_LAYER_GLOBAL, SK_ERR_ARG);
    }
    SK_RET_IF((reinterpret_cast<uintptr_t>(L.k) | reinterpret_cast<uintptr_t>(L.v)) & 15u, SK_ERR_ARG);
    return SK_OK;
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

extern "C" sk_status sk_decode_attention(const sk_kv_layer* layer, const void* q_rot,
                                         int32_t n_q_heads, int32_t io_dtype, void* out,
                                         void* workspace, size_t ws_bytes, void* stream) {
    sk_status s = check_layer(layer, n_q_heads);
    if (s != SK_OK) return s;
    SK_RET_IF(q_rot == nullptr || out == nullptr || workspace == nullptr, SK_ERR_ARG);
    SK_RET_IF((reinterpret_cast<uintptr_t>(q_rot) | reinterpret_cast<uintptr_t>(workspace)) & 15u,
              SK_ERR_ARG);
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
    p.out = out;
    p.ws = static_cast<float*>(workspace);
    p.count = L.count;
    p.pos = L.pos;
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
