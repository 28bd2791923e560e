// Prefill attention of a prompt chunk over itself, causal + sliding window + sinks,
// on the tcgen05 tensor cores.
//
// Mask ("KV-Cache Engineering", 5.5, and "Attention Sink 与 Streaming KV Cache"):
// query t sees key k iff k <= t and (p0 + k < S or t - k < W); W <= 0 is a global
// layer (causal only).  "Inference & 128K Long Context", prefill vs decode: masking a
// dense score matrix does not cut FLOPs, so here only key tiles the mask leaves (at
// least partly) visible are visited: the sink tile(s) and the tiles of the window.  A
// sink tile below the window whose sinks fit in 16 keys is visited as a 16-key strip.
//
// One CTA = one (sequence, group of nh q heads sharing a kv head, block of qpb = 128 / nh
// queries): BM = 128 tile rows, row r = head r / qpb, query r % qpb.
//   warps 0-3  softmax: thread r owns query row r = TMEM lane r
//   warp 4     Q K^T issue (one lane)
//   warp 5     TMA loads of Q and K (one lane)
//   warp 6     TMA loads of V (one lane)
//   warp 7     P V issue (one lane)
// Per key tile i (BN = 64 keys):
//   S_i = Q K_i^T      tcgen05.mma M=128 N=64, into one of two TMEM S buffers
//   softmax_i          tcgen05.ld S_i, mask, online max/sum in base 2 with a lazy
//                      rescale of O (only when the row max grows by more than 2^8),
//                      P_i as bf16 pairs written back over S_i with tcgen05.st
//   O += P_i V_i       tcgen05.mma M=128 N=128 with A = P_i read from tensor memory
//                      and B = V_i as stored (MN-major: dims along the rows)
// QK of tile i+1 runs on the tensor cores while softmax of tile i runs, and softmax no
// longer waits for P.V of the previous tile (only a rare O rescale does); two CTAs per
// SM overlap one CTA's softmax with the other's MMAs.  Q K^T and P V are issued by two
// threads: an issuing thread blocks while the tensor pipe's queue is full, and with one
// thread P V_i waited behind the issue of Q K^T_{i+1} (measured: 1.629 -> 1.53 ms on the
// 32,768-token chunk).
// V tiles are loaded as they lie ([key][dim], like K) and serve P.V as an MN-major B
// operand, so V needs no transposed copy.
// An optional learned sink logit per query head (a denominator-only term) enters at
// the epilogue.
// Every wait is bounded; a timeout sets SK_DEVERR_TIMEOUT in the error word (see
// wait_or_flag for how the block then ends).
#include <cudaTypedefs.h>

#include <algorithm>
#include <mutex>

#include "tcgen05.cuh"

namespace sk {
namespace {

constexpr int BM = 128;
constexpr int BN = 64;
constexpr int HD = 128;
constexpr int kThreads = 8 * 32;
constexpr uint32_t kTmemCols = 256;  // S0 [0, 64), S1 [64, 128), O [128, 256)
constexpr float kRescaleThreshold = 8.0f;  // log2 units
constexpr int kSinkStrip = 16;
// Bounds of a learned sink logit ("Inference & 128K Long Context", "Sink clamp cache").
constexpr float kSinkLogitMin = -10.0f;
constexpr float kSinkLogitMax = 15.0f;

// shared-memory layout (bytes from a 1024-aligned base)
constexpr int SM_Q = 0;                       // Q dims 0-63 then 64-127: 2 x 16 KB
constexpr int SM_K = 32768;                   // 2 stages x (K lo 8 KB, K hi 8 KB)
constexpr int K_STAGE = 16384;
constexpr int SM_V = SM_K + 2 * K_STAGE;      // 2 stages x (V lo 8 KB, V hi 8 KB)
constexpr int V_STAGE = 16384;
constexpr int SM_BAR = SM_V + 2 * V_STAGE;
constexpr int N_BARS = 18;  // 17 used
constexpr int SM_TMEM = SM_BAR + N_BARS * 8;
constexpr int SM_BYTES = SM_TMEM + 16;
// Two CTAs per SM fit comfortably (2 x (SM_ALLOC + 1 KB reserved) < 228 KB), with
// room to align the base to 1024 bytes; the kernel checks and reports rather than
// overflow.
constexpr int SM_ALLOC = SM_BYTES + 1024;
static_assert(SM_ALLOC >= SM_BYTES + 896, "no room to align the shared-memory base");

// Queries and keys live in one index space.  Without a prior cache it is the chunk's:
// query t is key t, key j is visible to query t iff j <= t and (j < nsk or t - j < W).
// With one, keys [0, qoff) are the prior's (gathered into the workspace, padded with
// zero rows to qpad, a multiple of BN, so that no tile mixes prior and chunk keys) and
// key qpad + t is the chunk's key t, read in place.  Prior key j (j < qoff) is visible
// to query t iff j < nsk or t + qoff - j < W (all of them with W <= 0); padding is never
// visible; chunk key qpad + k is visible iff k <= t and (qpad + k < nskc or t - k < W).
struct PrefillParams {
    void* out;
    const float* sink_logits;  // [Hq] learned sinks or null
    uint32_t* err;
    int T, Hq, Hkv, B;
    int Tk, qoff, qpad;        // keys in the index space; prior keys; padded prior keys
    int nsk, W;                // leading sink keys (prior keys with a prior); window (<= 0: global)
    int nskc;                  // chunk sink keys end below this index (qpad + sinks - p0)
    int sink_end;              // index past the last sink key (the plan's sink tiles)
    int nqb;           // query blocks of qpb queries
    int nh, qpb;       // q heads packed per CTA (one GQA group's), queries per block: nh * qpb = BM
    float scale_log2;  // log2(e) / sqrt(head_dim)
    int stall_tile;    // -1; otherwise (self-test) P of this tile is never signalled ready
};

struct TilePlan {
    int n;          // tiles to visit
    int n_sink;     // leading sink tiles (below the window)
    int first_win;  // first window tile
};

__device__ __forceinline__ TilePlan plan_tiles(const PrefillParams& p, int q0) {
    TilePlan tp;
    const int q_last = min(q0 + p.qpb, p.T) - 1 + p.qpad;  // the last query's own key
    int win_lo = 0;                                          // the first query's oldest key
    if (p.W > 0) {
        const int prior_lo = q0 + p.qoff - p.W + 1;          // as a prior index
        win_lo = prior_lo < p.qoff ? max(0, prior_lo) : q0 + p.qpad - p.W + 1;
    }
    tp.first_win = win_lo / BN;
    const int last = q_last / BN;
    const int sink_keys = p.W > 0 ? min(p.Tk, p.sink_end) : 0;
    tp.n_sink = min(tp.first_win, (sink_keys + BN - 1) / BN);
    tp.n = tp.n_sink + (last - tp.first_win + 1);
    return tp;
}

__device__ __forceinline__ int key_tile(const TilePlan& tp, int i) {
    return i < tp.n_sink ? i : tp.first_win + (i - tp.n_sink);
}

// Every (query, key) of the tile visible to every query of the block?
__device__ __forceinline__ bool tile_full(const PrefillParams& p, int q0, int k0) {
    if (q0 + p.qpb > p.T) return false;
    const int t_last = q0 + p.qpb - 1;
    if (k0 < p.qpad) {  // prior keys (and padding)
        if (k0 + BN > p.qoff) return false;
        if (p.W <= 0) return true;
        return t_last + p.qoff - k0 < p.W || k0 + BN - 1 < p.nsk;
    }
    if (k0 + BN - 1 > q0 + p.qpad || k0 + BN > p.Tk) return false;
    if (p.W <= 0) return true;
    return t_last + p.qpad - k0 < p.W || k0 + BN - 1 < p.nskc;
}

// Visibility bounds of a boundary tile at key k0 for a query whose own key is qpad + tq:
// tile column j is visible iff j <= jmax and (j >= jwin or j < jsink).
__device__ __forceinline__ void tile_bounds(const PrefillParams& p, int tq, int k0, int& jmax, int& jwin,
                                            int& jsink) {
    if (k0 < p.qpad) {
        jmax = p.qoff - 1 - k0;  // padding never
        jwin = p.W > 0 ? tq + p.qoff - p.W + 1 - k0 : -(1 << 30);
        jsink = p.W > 0 ? p.nsk - k0 : -(1 << 30);
    } else {
        jmax = tq + p.qpad - k0;
        jwin = p.W > 0 ? tq + p.qpad - p.W + 1 - k0 : -(1 << 30);
        jsink = p.W > 0 ? p.nskc - k0 : -(1 << 30);
    }
}

// max of three floats in one instruction
__device__ __forceinline__ float fmax3(float a, float b, float c) {
    float d;
    asm("max.f32 %0, %1, %2, %3;" : "=f"(d) : "f"(a), "f"(b), "f"(c));
    return d;
}

// Bounded wait (about one second) that also gives up, after a few polls, once any role
// of the block has timed out (the abort flag in shared memory).  The fast path is the
// plain try_wait; the hot loops carry no extra exit tests, because each one measurably
// slowed the pipeline.  After a timeout the roles run out their loops without waiting
// (every wait fails within a few polls), so a stalled block ends within about a second
// of its first timeout rather than a second per remaining wait; its results are then
// undefined, every address stays inside its buffer, and the block drains the MMAs and
// copies it issued (bounded waits) before it frees its tensor memory.
__device__ __forceinline__ bool wait_or_flag(uint64_t* bar, uint32_t parity, bool& bad,
                                             volatile uint32_t* abort) {
    if (mbar_try_wait(bar, parity)) return true;
    const uint64_t t0 = global_timer_ns();
    while (true) {
#pragma unroll 1
        for (int i = 0; i < 32; ++i)
            if (mbar_try_wait(bar, parity)) return true;
        if (*abort != 0u || global_timer_ns() - t0 > 1000000000ull) break;
    }
    bad = true;
    *abort = 1u;
    return false;
}

__global__ void __launch_bounds__(kThreads, 2)
    prefill_attn_kernel(const __grid_constant__ CUtensorMap tmQ, const __grid_constant__ CUtensorMap tmK,
                        const __grid_constant__ CUtensorMap tmV, const __grid_constant__ CUtensorMap tmKc,
                        const __grid_constant__ CUtensorMap tmVc, PrefillParams p) {
    extern __shared__ __align__(128) uint8_t smem_raw[];
    const uint32_t raw_addr = smem_u32(smem_raw);
    const uint32_t pad = ((raw_addr + 1023u) & ~1023u) - raw_addr;
    if (pad + SM_BYTES > uint32_t(SM_ALLOC)) {  // uniform for the whole block
        if (threadIdx.x == 0) set_error(p.err, SK_DEVERR_TIMEOUT);
        return;
    }
    uint8_t* smem = smem_raw + pad;
    // Barriers come in pairs indexed by tile parity, so that no wait can see a phase
    // two tiles old (each wait below is at most one phase behind on its barrier).
    uint64_t* bars = reinterpret_cast<uint64_t*>(smem + SM_BAR);
    uint64_t* q_full = bars + 0;
    uint64_t* k_full = bars + 1;    // [2] K_i landed in K stage i & 1
    uint64_t* k_empty = bars + 3;   // [2] Q K_i^T done: K stage i & 1 free
    uint64_t* v_full = bars + 5;    // [2] V_i^T landed in V stage i & 1
    uint64_t* v_empty = bars + 7;   // [2] P_i V_i done: V stage i & 1 free
    uint64_t* s_full = bars + 9;    // [2] S_i = Q K_i^T in TMEM buffer i & 1
    uint64_t* p_full = bars + 11;   // [2] P_i (bf16) written over S_i
    uint64_t* pv_done = bars + 13;  // [2] O += P_i V_i done
    uint64_t* drain = bars + 15;    // [2] after a timeout: each issuing thread's MMAs done
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + SM_TMEM);
    volatile uint32_t* abort = reinterpret_cast<volatile uint32_t*>(smem + SM_TMEM + 4);

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    // block -> (query block, descending so the long blocks start first; head group;
    // sequence).  The nh heads of a group share a kv head, so each K / V tile serves
    // nh * qpb = BM rows: row r is head h0 + r / qpb, query q0 + r % qpb.
    const int n_hg = p.Hq / p.nh;
    const int b = blockIdx.x % p.B;
    const int h0 = ((blockIdx.x / p.B) % n_hg) * p.nh;
    const int qb = p.nqb - 1 - blockIdx.x / (p.B * n_hg);
    const int q0 = qb * p.qpb;
    const int g = h0 / (p.Hq / p.Hkv);
    const TilePlan tp = plan_tiles(p, q0);
    // a sink tile below the window whose sinks fit in kSinkStrip keys is visited as a
    // strip: Q K^T with N = kSinkStrip, P.V with K = kSinkStrip, kSinkStrip softmax columns
    const int n_strip = (tp.n_sink == 1 && p.nsk <= kSinkStrip) ? 1 : 0;

    if (threadIdx.x == 0) {
        mbar_init(q_full, 1);
        mbar_init(&drain[0], 1);
        mbar_init(&drain[1], 1);
        *abort = 0u;
        for (int s = 0; s < 2; ++s) {
            mbar_init(&k_full[s], 1);
            mbar_init(&k_empty[s], 1);
            mbar_init(&v_full[s], 1);
            mbar_init(&v_empty[s], 1);
            mbar_init(&s_full[s], 1);
            mbar_init(&p_full[s], 4);
            mbar_init(&pv_done[s], 1);
        }
        fence_barrier_init();
    }
    if (warp == 0) {
        tmem_alloc(tmem_slot, kTmemCols);
        tmem_relinquish();
    }
    tc_fence_before_sync();
    __syncthreads();
    tc_fence_after_sync();
    const uint32_t tmem = *tmem_slot;
    bool bad = false;

    if (warp == 5) {
        // ---------------------------- TMA loads: Q, K ----------------------------
        // K stage i & 1 is free once Q K_i^T is done, so K runs a tile ahead of V
        if (lane == 0) {
            mbar_arrive_expect_tx(q_full, 2 * BM * 128);
            for (int j = 0; j < p.nh; ++j) {
                tma_load_4d(smem + SM_Q + j * p.qpb * 128, &tmQ, 0, h0 + j, q0, b, q_full);
                tma_load_4d(smem + SM_Q + BM * 128 + j * p.qpb * 128, &tmQ, 64, h0 + j, q0, b, q_full);
            }
            for (int i = 0; i < tp.n; ++i) {
                const int s = i & 1;
                if (i >= 2) wait_or_flag(&k_empty[s], ((i >> 1) - 1) & 1, bad, abort);
                const int k0 = key_tile(tp, i) * BN;
                uint8_t* st = smem + SM_K + s * K_STAGE;
                mbar_arrive_expect_tx(&k_full[s], K_STAGE);
                // prior keys from the workspace, chunk keys in place
                const CUtensorMap* m = k0 < p.qpad ? &tmK : &tmKc;
                const int kr = k0 < p.qpad ? k0 : k0 - p.qpad;
                tma_load_4d(st, m, 0, g, kr, b, &k_full[s]);
                tma_load_4d(st + BN * 128, m, 64, g, kr, b, &k_full[s]);
            }
            if (bad) {  // the copies in flight land before the block leaves
                mbar_wait_bounded(q_full, 0);
                for (int i = max(0, tp.n - 2); i < tp.n; ++i) mbar_wait_bounded(&k_full[i & 1], (i >> 1) & 1);
            }
        }
    } else if (warp == 6) {
        // ----------------------------- TMA loads: V ------------------------------
        if (lane == 0) {
            for (int i = 0; i < tp.n; ++i) {
                const int s = i & 1;
                if (i >= 2) wait_or_flag(&v_empty[s], ((i >> 1) - 1) & 1, bad, abort);
                const int k0 = key_tile(tp, i) * BN;
                uint8_t* st = smem + SM_V + s * V_STAGE;
                mbar_arrive_expect_tx(&v_full[s], V_STAGE);
                const CUtensorMap* m = k0 < p.qpad ? &tmV : &tmVc;
                const int kr = k0 < p.qpad ? k0 : k0 - p.qpad;
                tma_load_4d(st, m, 0, g, kr, b, &v_full[s]);
                tma_load_4d(st + BN * 128, m, 64, g, kr, b, &v_full[s]);
            }
            if (bad)
                for (int i = max(0, tp.n - 2); i < tp.n; ++i) mbar_wait_bounded(&v_full[i & 1], (i >> 1) & 1);
        }
    } else if (warp == 4) {
        // ------------------------------- Q K^T issue -------------------------------
        if (lane == 0) {
            constexpr uint32_t idesc_qk = idesc_bf16_f32(BM, BN);
            constexpr uint32_t idesc_qk_strip = idesc_bf16_f32(BM, kSinkStrip);
            const uint32_t sq = smem_u32(smem + SM_Q);
            wait_or_flag(q_full, 0, bad, abort);
            tc_fence_after_sync();
            for (int i = 0; i < tp.n; ++i) {
                const int s = i & 1;
                wait_or_flag(&k_full[s], (i >> 1) & 1, bad, abort);
                // S buffer s last held P_{i-2}: its P.V must be done before QK_i overwrites it
                if (i >= 2) wait_or_flag(&pv_done[s], ((i >> 1) - 1) & 1, bad, abort);
                tc_fence_after_sync();
                const uint32_t sk = smem_u32(smem + SM_K + s * K_STAGE);
#pragma unroll
                for (int kk = 0; kk < HD / 16; ++kk) {
                    const uint32_t half = (kk >> 2);           // dims 0-63 or 64-127
                    const uint32_t off = (kk & 3) * 32;        // 16 dims = 32 bytes
                    const uint64_t da = desc_kmajor_sw128(sq + half * (BM * 128) + off);
                    const uint64_t db = desc_kmajor_sw128(sk + half * (BN * 128) + off);
                    umma_bf16(tmem + s * BN, da, db, i < n_strip ? idesc_qk_strip : idesc_qk, kk > 0 ? 1u : 0u);
                }
                umma_commit(&s_full[s]);
                umma_commit(&k_empty[s]);
            }
            if (bad) {  // this thread's MMAs done before the block frees tensor memory
                umma_commit(&drain[0]);
                mbar_wait_bounded(&drain[0], 0);
            }
        }
    } else if (warp == 7) {
        // -------------------------------- P V issue --------------------------------
        // A thread of its own: P.V of tile j goes as soon as P_j is written, not after the
        // next Q K^T's issue (each thread's commits track its own MMAs).
        if (lane == 0) {
            constexpr uint32_t idesc_pv = idesc_bf16_f32(BM, HD) | (1u << 16);  // B (V) MN-major
            for (int j = 0; j < tp.n; ++j) {
                const int s = j & 1;
                wait_or_flag(&p_full[s], (j >> 1) & 1, bad, abort);
                wait_or_flag(&v_full[s], (j >> 1) & 1, bad, abort);
                tc_fence_after_sync();
                const uint32_t sv = smem_u32(smem + SM_V + s * V_STAGE);
                if (j < n_strip) {
                    // the sink strip: its 16 keys, one K step (P_j in 8 TMEM columns)
                    const uint64_t db = desc_mnmajor_sw128(sv, BN * 128);
                    umma_bf16_tmem_a(tmem + 2 * BN, tmem + s * BN, db, idesc_pv, j > 0 ? 1u : 0u);
                } else {
#pragma unroll
                    for (int kk = 0; kk < BN / 16; ++kk) {
                        // A = P_j in TMEM: 16 keys = 8 columns of packed bf16 pairs; B = 16
                        // key rows of V (2 KB), dims 64-127 in the second 8 KB block
                        const uint64_t db = desc_mnmajor_sw128(sv + kk * 2048, BN * 128);
                        umma_bf16_tmem_a(tmem + 2 * BN, tmem + s * BN + kk * 8, db, idesc_pv,
                                         (j > 0 || kk > 0) ? 1u : 0u);
                    }
                }
                umma_commit(&pv_done[s]);
                umma_commit(&v_empty[s]);
            }
            if (bad) {
                umma_commit(&drain[1]);
                mbar_wait_bounded(&drain[1], 0);
            }
        }
    } else if (warp < 4) {
        // ------------------------------- softmax ---------------------------------
        const int r = threadIdx.x;           // 0..127: tile row and TMEM lane
        const int h = h0 + r / p.qpb;        // its q head
        const int t = q0 + r % p.qpb;        // its query
        const uint32_t lane_base = uint32_t(warp * 32) << 16;
        float m_run = -INFINITY, l_run = 0.0f;
        if (n_strip) {
            // tile 0, the sink strip: only sinks are visible (the window starts above it)
            wait_or_flag(&s_full[0], 0, bad, abort);
            tc_fence_after_sync();
            uint32_t raw[kSinkStrip];
            tmem_ld_32x16(tmem + lane_base, raw);
            tmem_ld_wait();
            float sc[kSinkStrip];
#pragma unroll
            for (int j = 0; j < kSinkStrip; ++j) sc[j] = j < p.nsk ? __uint_as_float(raw[j]) : -INFINITY;  // nsk <= qoff
            float mx = fmax3(sc[0], sc[1], sc[2]);
#pragma unroll
            for (int j = 3; j < kSinkStrip; j += 2) mx = fmax3(mx, sc[j], sc[j + 1 < kSinkStrip ? j + 1 : j]);
            m_run = mx * p.scale_log2;
            const float2 sc2 = make_float2(p.scale_log2, p.scale_log2);
            const float2 nm2 = make_float2(-m_run, -m_run);
            uint32_t pk[kSinkStrip / 2];
            float2 ls = make_float2(0.f, 0.f);
#pragma unroll
            for (int e = 0; e < kSinkStrip; e += 2) {
                const float2 x = __ffma2_rn(make_float2(sc[e], sc[e + 1]), sc2, nm2);
                const float p0 = fast_exp2_approx(x.x), p1 = fast_exp2_approx(x.y);
                ls = __fadd2_rn(ls, make_float2(p0, p1));
                pk[e >> 1] = float2_to_bf16x2(p0, p1);
            }
            tmem_st_32x8(tmem + lane_base, pk);
            l_run = ls.x + ls.y;
            tmem_st_wait();
            tc_fence_before_sync();
            __syncwarp();
            if (lane == 0) mbar_arrive(&p_full[0]);
        }
        for (int i = n_strip; i < tp.n; ++i) {
            const int s = i & 1;
            wait_or_flag(&s_full[s], (i >> 1) & 1, bad, abort);
            tc_fence_after_sync();
            uint32_t raw[64];
            tmem_ld_32x32(tmem + lane_base + s * BN, raw);
            tmem_ld_32x32(tmem + lane_base + s * BN + 32, raw + 32);
            tmem_ld_wait();

            const int k0 = key_tile(tp, i) * BN;
            const bool full = tile_full(p, q0, k0);
            float sc[64];
#pragma unroll
            for (int j = 0; j < 64; ++j) sc[j] = __uint_as_float(raw[j]);
            if (!full) {
                // key k0 + j visible iff j <= jmax and (j >= jwin or j < jsink): branch-free
                int jmax, jwin, jsink;
                tile_bounds(p, min(t, p.T - 1), k0, jmax, jwin, jsink);
#pragma unroll
                for (int j = 0; j < 64; ++j) {
                    const bool vis = (j <= jmax) && (j >= jwin || j < jsink);
                    sc[j] = vis ? sc[j] : -INFINITY;
                }
            }
            // row max of the raw scores with three-input max: 8 chains of 8 columns, then the chains
            float mx[8];
#pragma unroll
            for (int c = 0; c < 8; ++c) {
                float m = fmax3(sc[c], sc[c + 8], sc[c + 16]);
                m = fmax3(m, sc[c + 24], sc[c + 32]);
                m = fmax3(m, sc[c + 40], sc[c + 48]);
                mx[c] = fmaxf(m, sc[c + 56]);
            }
            const float m_tile =
                fmax3(fmax3(mx[0], mx[1], mx[2]), fmax3(mx[3], mx[4], mx[5]), fmaxf(mx[6], mx[7])) * p.scale_log2;
            // Lazy rescale: keep the running max unless the row max grows by more than
            // 2^8.  A row that has seen only masked keys (m_run = -inf) has O = 0 and
            // l = 0, so it adopts the new max without touching O.
            bool grow = i > 0 && m_tile > m_run + kRescaleThreshold && m_run != -INFINITY;
            if (m_run == -INFINITY) m_run = m_tile;
            if (__any_sync(0xffffffffu, grow)) {
                // O += P_{i-1} V_{i-1} must be done before O is rescaled
                wait_or_flag(&pv_done[(i - 1) & 1], ((i - 1) >> 1) & 1, bad, abort);
                tc_fence_after_sync();
                const float alpha = grow ? fast_exp2_approx(m_run - m_tile) : 1.0f;
#pragma unroll 1
                for (int c = 0; c < 4; ++c) {
                    uint32_t o[32];
                    tmem_ld_32x32(tmem + lane_base + 2 * BN + c * 32, o);
                    tmem_ld_wait();
#pragma unroll
                    for (int e = 0; e < 32; ++e) o[e] = __float_as_uint(__uint_as_float(o[e]) * alpha);
                    tmem_st_32x32(tmem + lane_base + 2 * BN + c * 32, o);
                }
                if (grow) {
                    l_run *= alpha;
                    m_run = m_tile;
                }
            }
            // p = 2^(s * scale - m): one packed FMA per pair, then the hardware exp2;
            // P (bf16 pairs) overwrites the first 32 columns of this tile's S buffer.
            const float m_ref = m_run == -INFINITY ? 0.0f : m_run;
            const float2 sc2 = make_float2(p.scale_log2, p.scale_log2);
            const float2 nm2 = make_float2(-m_ref, -m_ref);
            float2 ls[4] = {make_float2(0.f, 0.f), make_float2(0.f, 0.f), make_float2(0.f, 0.f),
                            make_float2(0.f, 0.f)};
            uint32_t pk[32];
#pragma unroll
            for (int e = 0; e < 64; e += 2) {
                const float2 x = __ffma2_rn(make_float2(sc[e], sc[e + 1]), sc2, nm2);
                const float p0 = fast_exp2_approx(x.x), p1 = fast_exp2_approx(x.y);
                ls[(e >> 1) & 3] = __fadd2_rn(ls[(e >> 1) & 3], make_float2(p0, p1));
                pk[e >> 1] = float2_to_bf16x2(p0, p1);
            }
            tmem_st_32x32(tmem + lane_base + s * BN, pk);
            const float2 l01 = __fadd2_rn(ls[0], ls[1]), l23 = __fadd2_rn(ls[2], ls[3]);
            const float2 l4 = __fadd2_rn(l01, l23);
            l_run += l4.x + l4.y;
            tmem_st_wait();
            tc_fence_before_sync();
            __syncwarp();
            if (lane == 0 && i != p.stall_tile) mbar_arrive(&p_full[s]);
        }
        // ---- epilogue: O / l -> bf16 rows ----
        wait_or_flag(&pv_done[(tp.n - 1) & 1], ((tp.n - 1) >> 1) & 1, bad, abort);
        tc_fence_after_sync();
        float inv = l_run > 0.0f ? 1.0f / l_run : 0.0f;
        if (p.sink_logits != nullptr) {
            // Learned sink: one more logit z in the denominator, no value row ("RoPE,
            // scaling, sliding window, attention sinks", "Hybrid models break the
            // uniform-spec assumption").  O and l are relative to m_run; bring both to
            // max(m_run, z) before adding 2^(z - max).
            const float z2 =
                fminf(fmaxf(p.sink_logits[h], kSinkLogitMin), kSinkLogitMax) * 1.4426950408889634f;
            const float m_ref = m_run == -INFINITY ? z2 : m_run;
            const float m_new = fmaxf(m_ref, z2);
            const float a = fast_exp2_approx(m_ref - m_new);
            inv = a / fmaf(l_run, a, fast_exp2_approx(z2 - m_new));
        }
        __nv_bfloat16* orow = static_cast<__nv_bfloat16*>(p.out) +
                              ((int64_t(b) * p.T + t) * p.Hq + h) * HD;
#pragma unroll
        for (int c = 0; c < 4; ++c) {
            uint32_t o[32];
            tmem_ld_32x32(tmem + lane_base + 2 * BN + c * 32, o);
            tmem_ld_wait();
            if (t < p.T) {
#pragma unroll
                for (int e = 0; e < 32; e += 8) {
                    const uint4 w = make_uint4(
                        float2_to_bf16x2(__uint_as_float(o[e]) * inv, __uint_as_float(o[e + 1]) * inv),
                        float2_to_bf16x2(__uint_as_float(o[e + 2]) * inv, __uint_as_float(o[e + 3]) * inv),
                        float2_to_bf16x2(__uint_as_float(o[e + 4]) * inv, __uint_as_float(o[e + 5]) * inv),
                        float2_to_bf16x2(__uint_as_float(o[e + 6]) * inv, __uint_as_float(o[e + 7]) * inv));
                    *reinterpret_cast<uint4*>(orow + c * 32 + e) = w;
                }
            }
        }
    }
    if (bad) set_error(p.err, SK_DEVERR_TIMEOUT);
    tc_fence_before_sync();
    __syncthreads();
    if (warp == 0) {
        tc_fence_after_sync();
        tmem_dealloc(tmem, kTmemCols);
    }
}

// The keys a chunk takes from a prior cache, in order: the first s0 positions (sink
// slots, or the prefix of a global layer), then the last cr positions before p0 (the
// newest cr entries of the ring in chronological order, or the global rows at those
// positions).  Key index j < s0 + cr of the gathered prior keys is prior row j.  A
// ring at position p0 holds ring_count = min(W, p0 - s0) entries; the chunk needs
// the newest cr <= ring_count of them.
struct PriorView {
    const __nv_bfloat16* k;  // [B][Hkv][cap][HD]
    const __nv_bfloat16* v;
    const int32_t* head;
    const int32_t* count;
    const int64_t* pos;
    int64_t cap, p0;
    int kind, S, W;  // the layer's kind, sinks and window
    int s0, cr, ring_count;
};

// Cache slot of prior row j of sequence b; always inside [0, cap), whatever the state.
__device__ __forceinline__ int64_t prior_slot(const PriorView& pv, int b, int j) {
    if (j < pv.s0) return j;
    const int r = j - pv.s0;
    if (pv.kind == SK_LAYER_GLOBAL) return pv.p0 - pv.cr + r;
    // ring: chronological entry cnt - cr + r of the cnt the ring holds
    const int cnt = min(max(pv.count[b], 0), pv.W);
    const int hd = ((pv.head[b] % pv.W) + pv.W) % pv.W;
    const int ci = min(max(cnt - pv.cr + r, 0), pv.W - 1);
    return pv.S + (cnt == pv.W ? (hd + ci) % pv.W : ci);
}

// The prior's keys and values kc, vc [B][qpad][Hkv][HD]: prior rows j < qoff in the
// order of the key index space (sinks, then recent positions oldest first), then zero
// rows up to qpad (never visible; zero so that no stale value meets a zero weight).  The
// chunk's own keys are not copied: the attention kernel reads them in place.  One thread
// per 16 bytes of a K row and the same 16 bytes of its V row.  The thread of (b, j = 0,
// g = 0, c = 0) checks that the prior's state matches the chunk's start (pos = p0; a ring
// holds ring_count recent entries).
__global__ void __launch_bounds__(256) gather_prior_kernel(PriorView pv, __nv_bfloat16* __restrict__ kc,
                                                           __nv_bfloat16* __restrict__ vc, int B, int qpad, int Hkv,
                                                           uint32_t* err) {
    constexpr int CH = HD / 8;  // 16-byte chunks per row
    const int qoff = pv.s0 + pv.cr;
    const int64_t total = int64_t(B) * qpad * Hkv * CH;
    for (int64_t i = int64_t(blockIdx.x) * blockDim.x + threadIdx.x; i < total;
         i += int64_t(gridDim.x) * blockDim.x) {
        const int c = int(i % CH);
        const int g = int((i / CH) % Hkv);
        const int64_t bj = i / (int64_t(CH) * Hkv);
        const int j = int(bj % qpad), b = int(bj / qpad);
        const int64_t dst = (bj * Hkv + g) * HD;
        if (j < qoff) {
            const int64_t row = ((int64_t(b) * Hkv + g) * pv.cap + prior_slot(pv, b, j)) * HD;
            if (j == 0 && g == 0 && c == 0) {
                const bool ok = pv.pos[b] == pv.p0 && (pv.kind == SK_LAYER_GLOBAL || pv.count[b] == pv.ring_count);
                if (!ok) set_error(err, SK_DEVERR_STATE);
            }
            reinterpret_cast<uint4*>(kc + dst)[c] = reinterpret_cast<const uint4*>(pv.k + row)[c];
            reinterpret_cast<uint4*>(vc + dst)[c] = reinterpret_cast<const uint4*>(pv.v + row)[c];
        } else {
            reinterpret_cast<uint4*>(kc + dst)[c] = make_uint4(0, 0, 0, 0);
            reinterpret_cast<uint4*>(vc + dst)[c] = make_uint4(0, 0, 0, 0);
        }
    }
}

PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
    static std::once_flag once;
    static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
    std::call_once(once, [] {
        void* ptr = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &ptr, 12000, cudaEnableDefault, &q) ==
                cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(ptr);
    });
    return fn;
}

bool make_map(CUtensorMap* m, const void* base, int rank, const cuuint64_t* dims, const cuuint64_t* strides,
              const cuuint32_t* box) {
    auto fn = encode_fn();
    if (fn == nullptr) return false;
    const cuuint32_t estr[4] = {1, 1, 1, 1};
    return fn(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, cuuint32_t(rank), const_cast<void*>(base), dims, strides, box,
              estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
              CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

}  // namespace
}  // namespace sk

using namespace sk;

namespace sk {
namespace {

// (s0, cr) of a chunk starting at p0: the sinks it sees, then the recent keys before
// p0 its first query still sees (W - 1 of them: a query's window includes itself);
// all of the prefix for a global attention (window <= 0).
void prior_split(int64_t p0, int32_t sinks, int32_t window, int64_t* s0, int64_t* cr) {
    if (window <= 0) {
        *s0 = 0;
        *cr = p0;
    } else {
        *s0 = std::min<int64_t>(sinks, p0);
        *cr = std::min<int64_t>(int64_t(window) - 1, p0 - *s0);
    }
}

}  // namespace
}  // namespace sk

extern "C" int64_t sk_prefill_prior_keys(int64_t p0, int32_t sinks, int32_t window) {
    if (p0 < 0 || sinks < 0) return -1;
    int64_t s0 = 0, cr = 0;
    prior_split(p0, sinks, window, &s0, &cr);
    return s0 + cr;
}

// Prior keys padded to a whole number of key tiles.
static int64_t padded_prior(int64_t prior_keys) { return (prior_keys + BN - 1) / BN * BN; }

extern "C" size_t sk_prefill_workspace_bytes(int32_t batch, int32_t T, int32_t n_kv_heads, int32_t head_dim,
                                             int64_t prior_keys) {
    if (batch < 1 || T < 0 || n_kv_heads < 1 || head_dim != HD || prior_keys < 0) return 0;
    const int64_t qpad = padded_prior(prior_keys);
    if (int64_t(T) + qpad > (int64_t(1) << 30)) return 0;
    // no scratch is used: a token size keeps 0 for "unsupported"
    if (prior_keys == 0 || T == 0) return 16;
    return 2 * size_t(batch) * qpad * n_kv_heads * HD * sizeof(__nv_bfloat16);  // the prior's keys and values
}

// sk_prefill_attention with a stall tile for the self-test (-1: none).
static sk_status prefill_launch(const void* q_rot, const void* k_rot, const void* v, int32_t batch, int32_t T,
                                int32_t n_q_heads, int32_t n_kv_heads, int32_t head_dim, int64_t p0, int32_t sinks,
                                int32_t window, const sk_kv_layer* prior, const float* sink_logits, void* out,
                                void* workspace, size_t ws_bytes, uint32_t* err, void* stream, int stall_tile) {
    SK_RET_IF(batch < 1 || T < 0 || n_q_heads < 1 || n_kv_heads < 1 || n_q_heads % n_kv_heads != 0, SK_ERR_ARG);
    // T = 0 reads and writes nothing: the chunk, output and workspace pointers may be NULL
    SK_RET_IF(T > 0 && (q_rot == nullptr || k_rot == nullptr || v == nullptr || out == nullptr ||
                        workspace == nullptr),
              SK_ERR_ARG);
    SK_RET_IF(p0 < 0 || sinks < 0, SK_ERR_ARG);
    SK_RET_IF(head_dim != HD, SK_ERR_UNSUPPORTED);
    const uintptr_t al = reinterpret_cast<uintptr_t>(q_rot) | reinterpret_cast<uintptr_t>(k_rot) |
                         reinterpret_cast<uintptr_t>(v) | reinterpret_cast<uintptr_t>(out) |
                         reinterpret_cast<uintptr_t>(workspace);
    SK_RET_IF(al & 15u, SK_ERR_ARG);
    SK_RET_IF(reinterpret_cast<uintptr_t>(sink_logits) & 3u, SK_ERR_ARG);
    PriorView pv{};
    int64_t qoff = 0;
    if (prior != nullptr) {
        const sk_kv_layer& L = *prior;
        SK_RET_IF(L.k == nullptr || L.v == nullptr || L.pos == nullptr, SK_ERR_ARG);
        SK_RET_IF(L.k_dtype != SK_BF16 || L.v_dtype != SK_BF16, SK_ERR_UNSUPPORTED);
        SK_RET_IF(L.batch != batch || L.n_kv_heads != n_kv_heads || L.head_dim != head_dim, SK_ERR_ARG);
        SK_RET_IF((reinterpret_cast<uintptr_t>(L.k) | reinterpret_cast<uintptr_t>(L.v)) & 15u, SK_ERR_ARG);
        int64_t s0 = 0, cr = 0;
        prior_split(p0, sinks, window, &s0, &cr);
        if (L.kind == SK_LAYER_RING) {
            // the ring must keep exactly the keys the chunk's mask admits
            SK_RET_IF(L.head == nullptr || L.count == nullptr, SK_ERR_ARG);
            SK_RET_IF(window <= 0 || L.sinks != sinks || L.window != window ||
                          L.capacity != int64_t(L.sinks) + L.window,
                      SK_ERR_ARG);
        } else {
            SK_RET_IF(L.kind != SK_LAYER_GLOBAL || L.capacity < 1, SK_ERR_ARG);
            SK_RET_IF(p0 > L.capacity, SK_ERR_CAPACITY);
        }
        qoff = s0 + cr;
        const int64_t ring_count = window > 0 ? std::min<int64_t>(window, p0 - s0) : 0;
        pv = PriorView{static_cast<const __nv_bfloat16*>(L.k), static_cast<const __nv_bfloat16*>(L.v), L.head,
                       L.count, L.pos, L.capacity, p0, L.kind, L.sinks, L.window, int(s0), int(cr),
                       int(ring_count)};
    }
    if (T == 0) return SK_OK;
    const int64_t qpad = padded_prior(qoff);
    const int64_t Tk64 = int64_t(T) + qpad;
    SK_RET_IF(Tk64 > (int64_t(1) << 30), SK_ERR_UNSUPPORTED);
    const size_t need = sk_prefill_workspace_bytes(batch, T, n_kv_heads, head_dim, qoff);
    SK_RET_IF(need == 0 || ws_bytes < need, SK_ERR_ARG);
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    const int Tk = int(Tk64);
    // the prior's keys and values (gathered, padded to qpad rows) in the workspace
    __nv_bfloat16* kc = static_cast<__nv_bfloat16*>(workspace);
    __nv_bfloat16* vc = kc + size_t(batch) * qpad * n_kv_heads * HD;

    // pack the q heads of a GQA group into one CTA (a power of two dividing n_rep, at
    // most 8): the K / V tiles are then loaded once for all of them
    const int nrep = n_q_heads / n_kv_heads;
    int nh = 1;
    while (nh < 8 && nrep % (2 * nh) == 0) nh *= 2;
    const int qpb = BM / nh;

    CUtensorMap mq, mk, mv, mkc, mvc;
    {
        const cuuint64_t dims[4] = {cuuint64_t(HD), cuuint64_t(n_q_heads), cuuint64_t(T), cuuint64_t(batch)};
        const cuuint64_t strides[3] = {cuuint64_t(HD) * 2, cuuint64_t(n_q_heads) * HD * 2,
                                       cuuint64_t(T) * n_q_heads * HD * 2};
        const cuuint32_t box[4] = {64, 1, cuuint32_t(qpb), 1};
        SK_RET_IF(!make_map(&mq, q_rot, 4, dims, strides, box), SK_ERR_CUDA);
    }
    const cuuint32_t kv_box[4] = {64, 1, BN, 1};
    {  // the chunk's keys and values, read in place
        const cuuint64_t dims[4] = {cuuint64_t(HD), cuuint64_t(n_kv_heads), cuuint64_t(T), cuuint64_t(batch)};
        const cuuint64_t strides[3] = {cuuint64_t(HD) * 2, cuuint64_t(n_kv_heads) * HD * 2,
                                       cuuint64_t(T) * n_kv_heads * HD * 2};
        SK_RET_IF(!make_map(&mkc, k_rot, 4, dims, strides, kv_box), SK_ERR_CUDA);
        SK_RET_IF(!make_map(&mvc, v, 4, dims, strides, kv_box), SK_ERR_CUDA);
    }
    if (qoff > 0) {  // the prior's, gathered
        const cuuint64_t dims[4] = {cuuint64_t(HD), cuuint64_t(n_kv_heads), cuuint64_t(qpad), cuuint64_t(batch)};
        const cuuint64_t strides[3] = {cuuint64_t(HD) * 2, cuuint64_t(n_kv_heads) * HD * 2,
                                       cuuint64_t(qpad) * n_kv_heads * HD * 2};
        SK_RET_IF(!make_map(&mk, kc, 4, dims, strides, kv_box), SK_ERR_CUDA);
        SK_RET_IF(!make_map(&mv, vc, 4, dims, strides, kv_box), SK_ERR_CUDA);
        const int64_t threads = int64_t(batch) * qpad * n_kv_heads * (HD / 8);
        const int64_t blocks = std::min<int64_t>((threads + 255) / 256, int64_t(device_sm_count()) * 16);
        gather_prior_kernel<<<unsigned(blocks), 256, 0, st>>>(pv, kc, vc, batch, int(qpad), n_kv_heads, err);
        SK_CUDA_RET(cudaGetLastError());
    } else {
        mk = mkc;  // no prior: every key tile is the chunk's
        mv = mvc;
    }

    static PerDevice<cudaError_t> attr;
    SK_CUDA_RET(set_smem_limit_once(attr, prefill_attn_kernel, SM_ALLOC));

    PrefillParams p{};
    p.out = out;
    p.sink_logits = sink_logits;
    p.err = err;
    p.T = T;
    p.Tk = Tk;
    p.qoff = int(qoff);
    p.qpad = int(qpad);
    // Sinks in the key index space.  Without a prior, chunk key k has position p0 + k:
    // keys below sinks - p0 are sinks.  With one, prior keys 0 .. min(sinks, p0) - 1 are
    // the positions below p0 that are sinks, and chunk keys (at qpad + k) whose position
    // p0 + k is below sinks are sinks too.
    const int64_t chunk_sinks = std::max<int64_t>(0, int64_t(sinks) - p0);
    if (window > 0) {
        p.nsk = int(qoff > 0 ? std::min<int64_t>(sinks, p0) : std::min<int64_t>(T, chunk_sinks));
        p.nskc = int(qpad + std::min<int64_t>(T, chunk_sinks));
        p.sink_end = int(chunk_sinks > 0 ? p.nskc : p.nsk);
    } else {
        p.nsk = p.nskc = p.sink_end = 0;
    }
    p.W = window;
    p.Hq = n_q_heads;
    p.Hkv = n_kv_heads;
    p.B = batch;
    p.nh = nh;
    p.qpb = qpb;
    p.nqb = (T + qpb - 1) / qpb;
    p.scale_log2 = 1.4426950408889634f / sqrtf(float(HD));
    p.stall_tile = stall_tile;
    const int64_t grid = int64_t(p.nqb) * (n_q_heads / nh) * batch;
    prefill_attn_kernel<<<unsigned(grid), kThreads, SM_ALLOC, st>>>(mq, mk, mv, mkc, mvc, p);
    SK_CUDA_RET(cudaGetLastError());
    return SK_OK;
}

extern "C" sk_status sk_prefill_attention(const void* q_rot, const void* k_rot, const void* v, int32_t batch,
                                          int32_t T, int32_t n_q_heads, int32_t n_kv_heads, int32_t head_dim,
                                          int64_t p0, int32_t sinks, int32_t window, const sk_kv_layer* prior,
                                          const float* sink_logits, void* out, void* workspace, size_t ws_bytes,
                                          uint32_t* err, void* stream) {
    return prefill_launch(q_rot, k_rot, v, batch, T, n_q_heads, n_kv_heads, head_dim, p0, sinks, window, prior,
                          sink_logits, out, workspace, ws_bytes, err, stream, -1);
}

extern "C" sk_status sk_selftest_prefill_stall(const void* q_rot, const void* k_rot, const void* v, int32_t batch,
                                               int32_t T, int32_t n_q_heads, int32_t n_kv_heads, int32_t head_dim,
                                               void* out, void* workspace, size_t ws_bytes, int32_t stall_tile,
                                               uint32_t* err, void* stream) {
    SK_RET_IF(err == nullptr || stall_tile < 0, SK_ERR_ARG);
    return prefill_launch(q_rot, k_rot, v, batch, T, n_q_heads, n_kv_heads, head_dim, 0, 0, 0, nullptr, nullptr,
                          out, workspace, ws_bytes, err, stream, stall_tile);
}
