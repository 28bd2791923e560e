// Split-K (flash-decoding) GQA decode attention over the sink ∪ recent visible set.
//
// "Attention Sink 与 Streaming KV Cache", visible set V(P): in a ring layer after the
// query's own append the occupied slots [0, min(pos, S) + count) are exactly V(P), and
// attention is order-free, so no chronological gather is needed.  A global layer
// reads rows [0, pos).  "KV-Cache Engineering", 4.3-4.4 and 5.5: decode is bound by
// the KV bytes it streams, and the n_rep query heads of a GQA group share each K/V
// row, broadcast in registers instead of repeat_kv's copy.
//
// Work split: the visible rows of all units (b, g) are laid end to end, R rows in
// all, and block c of P takes rows [ceil(cR/P), ceil((c+1)R/P)): every block gets the
// same number of rows whatever the lengths, and a unit cut between blocks yields one
// partial per block.  The partial of unit u from block c lives at workspace slot
// u + c: the blocks meeting unit u are consecutive and start at or after the last
// block of unit u - 1, so the slots never collide and (P + units) always suffice.
//
// Block: one producer lane streams K and V tiles (rows of one unit are contiguous in
// HBM) with 1-D bulk copies into a STAGES-deep shared-memory ring guarded by
// mbarriers.  Each consumer warp takes RPW rows of a tile: 8-lane groups compute
// partial q.k products for 8/NREP rows x NREP heads over 16 dims per lane; a
// butterfly reduce-scatter (3 shuffle rounds) leaves one finished score per lane --
// lanes visit rows and heads in an order permuted by their lane index so that every
// round adds the same register slots, with no selects; online softmax in base 2;
// then P.V with each lane owning D/32 dims of all NREP heads, the probabilities read
// back from shared memory as (p, p) pairs ready for packed fp32 FMAs.
// A second kernel combines each unit's partials by log-sum-exp; a learned sink logit
// (a per-head term in the softmax denominator) enters there.
//
// Instantiations: contiguous layers (ring or global) and paged layers (a block-table
// producer), each for bf16 or fp32 caches, and contiguous layers with int8 keys (128
// codes and one fp32 scale per K row, bf16 V): a lane decodes its 16 codes of a row
// exactly to fp32, and the reduced score is multiplied by the row's scale.  Before its
// PDL wait, a contiguous block asks L2 for the first rows of its share.
//
// FUSED kernels fold the token's RoPE + append into the step (contiguous bf16 or fp32
// layers).  The split kernel works on the rows visible after the append, computed from
// the state as it stands (the append's rules, below).  An extra warp per block (the
// token warp) rotates q of every unit the block meets, with the append's arithmetic,
// into a two-slot ring in shared memory that the consumers read instead of q in global
// memory; and the one block whose share holds a unit's new slot has it write the rotated
// key and the value there before the producer copies that tile.  No other block reads
// that slot, because the visible set after the append no longer holds the entry the
// token replaces.  The state itself is advanced by the combine kernel, from a copy the
// split kernel took, so that no block of either kernel reads a state another block is
// changing.
#pragma once

#include <algorithm>
#include <mutex>

#include "rope_lane.cuh"

namespace sk {
namespace {

constexpr unsigned kFull = 0xffffffffu;
constexpr float kLog2e = 1.4426950408889634f;
constexpr int kMaxBatch = 1024;
// Bounds of a learned sink logit ("Inference & 128K Long Context", "Sink clamp cache").
constexpr float kSinkLogitMin = -10.0f;
constexpr float kSinkLogitMax = 15.0f;

struct DecodeParams {
    const void* kc;
    const void* vc;
    const void* q;
    const float* sink_logits;  // [Hq] learned sinks or null
    void* out;
    float* ws;
    const int32_t* count;
    const int64_t* pos;
    const float* kscale;  // [B][Hkv][cap] per-row scales of an int8 K cache, else null
    uint32_t* err;
    int64_t cap;
    int B, Hkv, S, kind;
    int n_blocks;  // P: blocks of the split kernel
    int combine_wpu;  // warps per (b, q head) in the combine kernel
    float qscale;  // log2(e) / sqrt(D)
    // paged layers (kind kKindPaged): pools in kc / vc, request lengths in pos
    const int32_t* block_table;
    const int32_t* sink_blocks;
    int64_t pool_blocks;
    int bs, bs_log2, max_blocks, sink_len, W;  // block_size = 1 << bs_log2; W: window (paged, or a
                                               // ring in the FUSED kernels)
    // FUSED kernels: the token of this step and the state the combine advances
    const void* k_new;    // [B][Hkv][D] keys before rotation
    const void* v_new;    // [B][Hkv][D] values
    const float2* table;  // (cos, sin) rows [max_pos][rotary_dim / 2]; unused when rotary_dim is 0
    int64_t max_pos;
    int rotary_dim, neox;
    const int32_t* head;  // ring write index (null for a global layer)
    int32_t* head_rw;     // the same state, written by the combine kernel
    int32_t* count_rw;
    int64_t* pos_rw;
    int64_t* snap;        // [B][4]: pos, count, head as the split kernel read them
};

__device__ __forceinline__ int64_t visible_rows(const DecodeParams& p, int b) {
    const int64_t pos = p.pos[b];
    if (p.kind == kKindPaged) {
        // logical keys: the static sink tokens, then the request's own (none if empty)
        const int64_t L = pos > 0 ? pos + p.sink_len : 0;
        return (p.W <= 0 || L <= int64_t(p.S) + p.W) ? L : int64_t(p.S) + p.W;
    }
    if (p.kind == SK_LAYER_GLOBAL) return max(int64_t(0), min(pos, p.cap));
    return max(int64_t(0), min(pos, int64_t(p.S))) + int64_t(p.count[b]);
}

// One token appended to a contiguous layer, by the rules of the RoPE + KV append
// ("Inference & 128K Long Context", MixedKVCache; "Attention Sink 与 Streaming KV
// Cache": positions below S take the pinned sink slots): whether it is stored (the
// position inside the table, a global layer's capacity), its slot, and the state after
// it (the state as it was when it is not stored).  A ring slot outside the cache (a
// corrupt head) is refused with SK_DEVERR_STATE rather than written.
struct StepState {
    int64_t pos0;   // the token's position
    int64_t pos;    // the state after the step
    int head, count;
    int64_t slot;   // cache slot of the token (ok only)
    uint32_t err;
    bool ok;
};

__device__ __forceinline__ StepState step_state(const DecodeParams& p, int64_t pos, int head, int count) {
    StepState s{pos, pos, head, count, -1, 0u, false};
    if (pos < 0 || pos + 1 > p.max_pos) s.err |= SK_DEVERR_POSITION_RANGE;
    if (p.kind == SK_LAYER_GLOBAL && pos + 1 > p.cap) s.err |= SK_DEVERR_CAPACITY;
    if (s.err != 0) return s;
    if (p.kind == SK_LAYER_GLOBAL) {
        s.slot = pos;
    } else if (pos < p.S) {  // a sink slot; the ring's head and count stay (normalised)
        s.slot = pos;
        s.head = int(int64_t(head) % p.W);
        s.count = int(min(int64_t(p.W), int64_t(count)));
    } else if (p.W == 1) {
        s.slot = p.S;
        s.head = 0;
        s.count = 1;
    } else {  // the ring's write index, then one step on
        s.slot = p.S + int64_t(head) % p.W;
        s.head = int((int64_t(head) + 1) % p.W);
        s.count = int(min(int64_t(p.W), int64_t(count) + 1));
    }
    if (s.slot < 0 || s.slot >= p.cap) {
        s.err = SK_DEVERR_STATE;
        s.head = head;
        s.count = count;
        return s;
    }
    s.pos = pos + 1;
    s.ok = true;
    return s;
}

// Visible rows of a contiguous layer in the state s describes (as visible_rows).
__device__ __forceinline__ int64_t step_rows(const DecodeParams& p, const StepState& s) {
    if (p.kind == SK_LAYER_GLOBAL) return max(int64_t(0), min(s.pos, p.cap));
    return max(int64_t(0), min(s.pos, int64_t(p.S))) + int64_t(s.count);
}

__device__ __forceinline__ StepState live_step(const DecodeParams& p, int b) {
    return step_state(p, p.pos[b], p.head != nullptr ? p.head[b] : 0, p.count != nullptr ? p.count[b] : 0);
}

__device__ __forceinline__ StepState snap_step(const DecodeParams& p, int b) {
    const int64_t* sn = p.snap + 4 * int64_t(b);
    return step_state(p, sn[0], int(sn[2]), int(sn[1]));
}

// Where unit_prefix takes each sequence's row count from: the state (kRowsLive), the
// state after this step's token (kRowsStep), or the latter from the split kernel's copy
// of the state (kRowsSnap).
constexpr int kRowsLive = 0, kRowsStep = 1, kRowsSnap = 2;

template <int SRC>
__device__ __forceinline__ int64_t unit_rows(const DecodeParams& p, int b) {
    if constexpr (SRC == kRowsLive) return visible_rows(p, b);
    else if constexpr (SRC == kRowsStep) return step_rows(p, live_step(p, b));
    else return step_rows(p, snap_step(p, b));
}

// pre[b] = Hkv * sum_{b' < b} L_b'; pre[B] = R.  Computed by one warp into shared memory.
template <int SRC = kRowsLive>
__device__ __forceinline__ void unit_prefix(const DecodeParams& p, int64_t* pre, int lane) {
    int64_t carry = 0;
    for (int b0 = 0; b0 < p.B; b0 += 32) {
        const int b = b0 + lane;
        int64_t x = b < p.B ? int64_t(p.Hkv) * unit_rows<SRC>(p, b) : 0;
        // inclusive warp scan
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const int64_t y = __shfl_up_sync(kFull, x, o);
            if (lane >= o) x += y;
        }
        if (b < p.B) pre[b + 1] = carry + x;
        carry += __shfl_sync(kFull, x, 31);
    }
    if (lane == 0) pre[0] = 0;
}

__device__ __forceinline__ int64_t first_block_of(int64_t row, int64_t R, int P) {
    return (row * P) / R;
}

// Iterates the units (b, g) whose rows meet [lo, hi).
struct UnitWalk {
    const int64_t* pre;
    int B, Hkv;
    int b, g;
    __device__ __forceinline__ void seek(int64_t lo) {
        int l = 0, h = B;  // largest b with pre[b] <= lo < pre[b+1]
        while (h - l > 1) {
            const int m = (l + h) >> 1;
            if (pre[m] <= lo) l = m; else h = m;
        }
        b = l;
        const int64_t Lb = (pre[b + 1] - pre[b]) / Hkv;
        g = Lb > 0 ? int((lo - pre[b]) / Lb) : 0;
    }
    __device__ __forceinline__ int64_t len() const { return (pre[b + 1] - pre[b]) / Hkv; }
    __device__ __forceinline__ int64_t start() const { return pre[b] + int64_t(g) * len(); }
    __device__ __forceinline__ bool next() {
        if (++g == Hkv) {
            g = 0;
            do { ++b; } while (b < B && pre[b + 1] == pre[b]);
        }
        return b < B;
    }
};

// Tiles of a paged unit start where the key index is a multiple of the tile height (a
// power of two), so that a tile spans as few blocks as possible: each block piece costs
// two bulk copies, and small copies, not bytes, limit a gather of 16-token blocks.
// Returns the row residue (mod tile) at which this request's tiles start.
__device__ __forceinline__ int64_t tile_phase(const DecodeParams& p, int b, int tile) {
    const int64_t n_req = p.pos[b];
    const int64_t Lk = n_req > 0 ? n_req + p.sink_len : 0;
    if (!(p.W > 0 && Lk > int64_t(p.S) + p.W)) return 0;  // rows are keys
    return (int64_t(p.S) - (Lk - p.W)) & (tile - 1);       // row S holds key Lk - W
}

// End of the paged tile that starts at row0.
__device__ __forceinline__ int64_t tile_end(int64_t row0, int64_t r1, int64_t phase, int tile) {
    return min(r1, row0 + tile - ((row0 - phase) & (tile - 1)));
}

// Consumer warps per block: 8 unless two stages of K+V tiles would not fit.
template <typename T, int D, int NREP> constexpr int decode_warps() {
    constexpr int warp_stage_bytes = 2 * (4 * (8 / NREP)) * D * int(sizeof(T));
    return 2 * 8 * warp_stage_bytes <= 200 * 1024 ? 8 : (2 * 4 * warp_stage_bytes <= 200 * 1024 ? 4 : 2);
}

template <int N> constexpr int ilog2() { return N <= 1 ? 0 : 1 + ilog2<N / 2>(); }

// KQ: the K cache holds int8 codes (D bytes per row, one fp32 scale per row); V is T.
// PAGED: the block-table producer, whose tiles start at multiples of the tile height.
// FUSED: the decode step with the token's append folded in (one more warp, its barriers
// and a ring of QSLOTS rotated q rows of a unit in shared memory).
template <typename T, int D, int NREP, bool KQ = false, bool PAGED = false, bool FUSED = false> struct DecodeCfg {
    // Contiguous bf16 layers at n_rep 4 and d_h 128 (bf16 or int8 keys) run 12 consumer
    // warps, 3 per scheduler: the consumers' issue and latency bound these kernels
    // (measured against 8 warps: bf16 keys +2.4% on the windowed step with 3 stages,
    // int8 keys +13%).  Paged tiles keep a power-of-two height.
    static constexpr bool WIDE = !PAGED && NREP == 4 && D == 128 && sizeof(T) == 2;
    static constexpr int NWARPS = WIDE ? 12 : decode_warps<T, D, NREP>();
    static constexpr int LG = ilog2<NREP>();
    static constexpr int VEC = ElemIO<T>::kPerVec;    // elements per 16-byte chunk
    static constexpr int CPL = (D / VEC) / 8;         // chunks per lane (QK)
    static constexpr int DPL = D / 8;                 // dims per lane (QK)
    static constexpr int RPG = 8 / NREP;              // rows per 8-lane group
    static constexpr int RPW = 4 * RPG;               // rows per warp per stage
    static constexpr int TILE = NWARPS * RPW;         // rows per stage
    static_assert(!PAGED || (TILE & (TILE - 1)) == 0, "paged tile height must be a power of two");
    static constexpr int DPV = D / 32;                // dims per lane (PV)
    static constexpr int ROW_BYTES = D * int(sizeof(T));      // a V row (and a K row unless KQ)
    static constexpr int K_ROW_BYTES = KQ ? D : ROW_BYTES;
    static constexpr int STAGE_BYTES = TILE * (K_ROW_BYTES + ROW_BYTES);   // K tile then V tile
    static_assert(!KQ || (D == 128 && sizeof(T) == 2), "int8 keys: head_dim 128, bf16 queries and values");
    static constexpr int MERGE_FLOATS = NWARPS * NREP * (D + 2);
    static constexpr int PS_F2 = NWARPS * (RPW * NREP + NREP);  // (p, p) pairs + (alpha, alpha)
    static constexpr int QSLOTS = 2;
    static constexpr size_t QSLOT_BYTES = size_t(NREP) * D * sizeof(T);
    static constexpr size_t FUSED_BYTES = FUSED ? 64 + QSLOTS * QSLOT_BYTES : 0;  // barriers, then the q ring
    // as many stages (at most 5) as fit beside the rest in 227 KB, less 1 KB of slack
    static constexpr size_t OTHER_BYTES =
        size_t(MERGE_FLOATS) * 4 + size_t(PS_F2) * 8 + (kMaxBatch + 1) * 8 + 2 * 5 * 8 + FUSED_BYTES;
    static constexpr int STAGES_FIT = int((232448 - 1024 - OTHER_BYTES) / STAGE_BYTES);
    static constexpr int STAGES = STAGES_FIT > 5 ? 5 : STAGES_FIT;
    static_assert(STAGES >= 2, "stage too large");
    static constexpr size_t OFF_MERGE = size_t(STAGES) * STAGE_BYTES;
    static constexpr size_t OFF_PS = OFF_MERGE + size_t(MERGE_FLOATS) * 4;
    static constexpr size_t OFF_PRE = OFF_PS + size_t(PS_F2) * 8;
    static constexpr size_t OFF_BAR = OFF_PRE + size_t(kMaxBatch + 1) * 8;
    // FUSED: new_bar, q_full[QSLOTS], q_empty[QSLOTS] (at most 64 bytes), then the q ring
    static constexpr size_t OFF_FUSED = OFF_BAR + 2 * STAGES * 8;
    static constexpr size_t OFF_QSLOT = (OFF_FUSED + 64 + 15) / 16 * 16;
    static_assert(8 * (1 + 2 * QSLOTS) <= 64, "fused barriers");
    static constexpr size_t SMEM = FUSED ? OFF_QSLOT + QSLOTS * QSLOT_BYTES : OFF_BAR + 2 * STAGES * 8;
    static_assert(SMEM <= 232448, "shared memory");
    static constexpr int THREADS = (NWARPS + 1 + (FUSED ? 1 : 0)) * 32;
    static constexpr int PARTIAL_FLOATS = NREP * (D + 2);
    static_assert(CPL >= 1 && DPV >= 2, "head_dim too small for this layout");
    static_assert(OFF_PS % 16 == 0 && OFF_PRE % 16 == 0, "alignment");
};

// This lane's PV slice of a row (DPV dims starting at lane * DPV) as DPV/2 pairs.
template <typename T, int DPV>
__device__ __forceinline__ void load_pv_slice(const T* row, int lane, float2* v) {
    if constexpr (sizeof(T) == 2) {
        if constexpr (DPV == 4) {
            const uint2 u = *reinterpret_cast<const uint2*>(row + lane * 4);
            v[0] = bf16x2_to_float2(u.x);
            v[1] = bf16x2_to_float2(u.y);
        } else {
            v[0] = bf16x2_to_float2(*reinterpret_cast<const uint32_t*>(row + lane * 2));
        }
    } else {
        if constexpr (DPV == 4) {
            const float4 u = *reinterpret_cast<const float4*>(row + lane * 4);
            v[0] = make_float2(u.x, u.y);
            v[1] = make_float2(u.z, u.w);
        } else {
            v[0] = *reinterpret_cast<const float2*>(row + lane * 2);
        }
    }
}

// Producer of a paged layer: the whole warp.  The visible rows [row, row + n) of a
// tile map to at most two runs of logical keys (the leading sinks, then the window),
// each cut at block boundaries (static sink blocks hold whole blocks, so boundaries
// are multiples of block_size in logical key space); lane j copies run j, from the
// physical block its table entry names ("vLLM, from the inside out", PagedAttention:
// the kernel gathers keys and values block by block).  Lane 0 first waits for the
// stage and sets the expected bytes.
template <typename C, typename T, int D>
__device__ __forceinline__ void paged_producer(const DecodeParams& p, const int64_t* pre, int64_t lo, int64_t hi,
                                               uint8_t* stages, uint64_t* full_bar, uint64_t* empty_bar,
                                               int lane) {
    constexpr int STAGES = C::STAGES;
    const uint64_t policy = l2_policy_evict_first();
    const int64_t bs = p.bs;
    const int lg = p.bs_log2;  // block_size is a power of two: no divisions below
    const T* kpool = static_cast<const T*>(p.kc);
    const T* vpool = static_cast<const T*>(p.vc);
    bool timed_out = false, bad = false;
    int stage = 0;
    uint32_t phase = 0;
    UnitWalk w{pre, p.B, p.Hkv, 0, 0};
    w.seek(lo);
    do {
        const int64_t st = w.start();
        if (st >= hi) break;
        const int64_t r0 = max(lo, st) - st, r1 = min(hi, st + w.len()) - st;
        const int b = w.b, g = w.g;
        const int64_t n_req = p.pos[b];
        const int64_t Lk = n_req > 0 ? n_req + p.sink_len : 0;
        const bool split = p.W > 0 && Lk > int64_t(p.S) + p.W;  // sinks, then the last W keys
        const int64_t wstart = Lk - p.W;                          // first window key when split
        const int32_t* trow = p.block_table + int64_t(b) * p.max_blocks;
        // Lane l caches table entry cbase + l: the window's block ids are consecutive
        // entries, so one load serves several tiles and the copies are not held up by
        // a table read per tile.
        int64_t cbase = -64;
        int32_t cval = -1;
        int64_t nbase = -64;  // the next 32 entries, loaded ahead (nbase == cbase + 32 when valid)
        int32_t cnext = -1;
        const int64_t tph = tile_phase(p, b, C::TILE);
        // blocks in a full aligned tile (0: no fast path, blocks taller than a tile or more
        // blocks than lanes)
        const int64_t nb = (bs <= C::TILE && (C::TILE >> lg) <= 32) ? C::TILE >> lg : 0;
        for (int64_t row = r0, row_end; row < r1; row = row_end) {
            row_end = tile_end(row, r1, tph, C::TILE);
            const int64_t n = row_end - row;
            if (lane == 0) {
                if (!mbar_wait_bounded(&empty_bar[stage], phase ^ 1)) timed_out = true;
                mbar_arrive_expect_tx(&full_bar[stage], 2u * uint32_t(n) * C::ROW_BYTES);
            }
            __syncwarp();
            uint8_t* dst = stages + size_t(stage) * C::STAGE_BYTES;
            // Fast path: a full tile of window (or unsplit) keys starting on a block boundary
            // is exactly nb whole blocks, block j for lane j.
            const int64_t kfirst = (split && row >= p.S) ? wstart + (row - p.S) : row;
            if (nb > 0 && n == C::TILE && (!split || row >= p.S) && kfirst >= p.sink_len &&
                (kfirst & (bs - 1)) == 0) {
                const int64_t jb0 = (kfirst - p.sink_len) >> lg;
                if (jb0 < cbase || jb0 + nb > cbase + 32) {
                    if (nbase == cbase + 32 && jb0 >= nbase && jb0 + nb <= nbase + 32) {
                        cbase = nbase;
                        cval = cnext;
                    } else {
                        cbase = jb0;
                        cval = cbase + lane < p.max_blocks ? trow[cbase + lane] : -1;
                    }
                }
                if (jb0 + nb > cbase + 16 && nbase != cbase + 32) {  // load the next entries ahead
                    nbase = cbase + 32;
                    cnext = nbase + lane < p.max_blocks ? trow[nbase + lane] : -1;
                }
                const int32_t cached = __shfl_sync(kFull, cval, int(jb0 - cbase + lane) & 31);
                if (lane < nb) {
                    int64_t blk = cached;
                    if (blk < 0 || blk >= p.pool_blocks) {
                        bad = true;
                        blk = 0;  // stay inside the pool; the error word reports it
                    }
                    const int64_t src = (blk * p.Hkv + g) * bs * D;
                    const uint32_t bytes = uint32_t(bs) * C::ROW_BYTES;
                    const int64_t drow = int64_t(lane) << lg;
                    bulk_copy_g2s(dst + drow * C::ROW_BYTES, kpool + src, bytes, &full_bar[stage], policy);
                    bulk_copy_g2s(dst + (C::TILE + drow) * C::ROW_BYTES, vpool + src, bytes, &full_bar[stage],
                                  policy);
                }
                if (++stage == STAGES) { stage = 0; phase ^= 1; }
                continue;
            }
            // run piece 1: rows [row, e1), keys = rows; piece 2: rows [a2, row + n),
            // keys [k2a, k2b) = wstart + (rows - S)
            const int64_t e1 = split ? min(row + n, int64_t(p.S)) : row + n;
            const int64_t n1 = row < e1 ? ((e1 - 1) >> lg) - (row >> lg) + 1 : 0;
            const int64_t a2 = split ? max(row, int64_t(p.S)) : row + n;
            const int64_t k2a = wstart + (a2 - p.S), k2b = wstart + (row + n - p.S);
            const int64_t n2 = a2 < row + n ? ((k2b - 1) >> lg) - (k2a >> lg) + 1 : 0;
            for (int64_t j0 = 0; j0 < n1 + n2; j0 += 32) {  // uniform trip count
                const int64_t j = j0 + lane;
                const bool active = j < n1 + n2;
                int64_t key0 = 0, key1 = 0, drow = 0;
                if (active && j < n1) {
                    const int64_t blo = ((row >> lg) + j) << lg;
                    key0 = max(row, blo);
                    key1 = min(e1, blo + bs);
                    drow = key0 - row;
                } else if (active) {
                    const int64_t blo = ((k2a >> lg) + (j - n1)) << lg;
                    key0 = max(k2a, blo);
                    key1 = min(k2b, blo + bs);
                    drow = (a2 - row) + (key0 - k2a);
                }
                const bool in_table = active && key0 >= p.sink_len;
                const int64_t jb = in_table ? (key0 - p.sink_len) >> lg : 0;
                // refill the cache from this round's first table entry when its last one
                // is not cached (block ids past 2^32 are not cached, only read directly)
                const int64_t jmax = __reduce_max_sync(kFull, in_table ? uint32_t(jb) : 0u);
                if (__any_sync(kFull, in_table) && (jmax >= cbase + 32 || jmax < cbase)) {
                    cbase = __reduce_min_sync(kFull, in_table ? uint32_t(jb) : 0xffffffffu);
                    cval = cbase + lane < p.max_blocks ? trow[cbase + lane] : -1;
                }
                const int64_t ci = jb - cbase;
                const int32_t cached = __shfl_sync(kFull, cval, int(ci) & 31);
                if (!active) continue;
                int64_t blk;
                if (key0 < p.sink_len) blk = p.sink_blocks[key0 >> lg];
                else if (ci >= 0 && ci < 32) blk = cached;
                else blk = jb < p.max_blocks ? trow[jb] : -1;
                if (blk < 0 || blk >= p.pool_blocks) {
                    bad = true;
                    blk = 0;  // stay inside the pool; the error word reports it
                }
                const int64_t src = ((blk * p.Hkv + g) * bs + (key0 & (bs - 1))) * D;
                const uint32_t bytes = uint32_t(key1 - key0) * C::ROW_BYTES;
                bulk_copy_g2s(dst + drow * C::ROW_BYTES, kpool + src, bytes, &full_bar[stage], policy);
                bulk_copy_g2s(dst + (C::TILE + drow) * C::ROW_BYTES, vpool + src, bytes, &full_bar[stage], policy);
            }
            if (++stage == STAGES) { stage = 0; phase ^= 1; }
        }
    } while (w.next());
    if (lane == 0) {
        // drain: every issued stage has been released, so no copy is in flight at exit
        for (int s = 0; s < STAGES; ++s) {
            if (!mbar_wait_bounded(&empty_bar[stage], phase ^ 1)) timed_out = true;
            if (++stage == STAGES) { stage = 0; phase ^= 1; }
        }
        if (timed_out) set_error(p.err, SK_DEVERR_TIMEOUT);
    }
    if (bad) set_error(p.err, SK_DEVERR_BLOCK_TABLE);
}

// FUSED: chunk c of a row of T at `row` (a token's q or k row), rotated at position pos
// with the append's arithmetic and rounded to T as the append stores it (as loaded when
// rot is false).  The lane issues all its loads (its chunk, a NeoX partner chunk, its
// table pairs at indices clamped into the rotary part) before the arithmetic.
template <typename T, int D>
__device__ __forceinline__ uint4 rope_row_vec(const DecodeParams& p, const uint4* row, int c, int64_t pos, bool rot) {
    constexpr int VEC = ElemIO<T>::kPerVec;
    constexpr int LPR = D / VEC;
    uint4 raw = row[c];
    if (!rot) return raw;
    const int half = p.rotary_dim / 2;
    const float4* trow = reinterpret_cast<const float4*>(p.table + pos * half);
    float f[VEC];
    if (p.neox) {
        const int hc = half / VEC;  // vectors per half of the rotary part
        const int j0 = min(c < hc ? c : c - hc, hc - 1) * VEC;
        const uint4 pr = row[min(c < hc ? c + hc : c - hc, LPR - 1)];
        float4 cs[VEC / 2];
#pragma unroll
        for (int t = 0; t < VEC / 2; ++t) cs[t] = trow[j0 / 2 + t];
        if (c < 2 * hc) {
            ElemIO<T>::unpack(raw, f);
            rope_vec_neox<T>(f, pr, cs, c < hc);
            raw = ElemIO<T>::pack(f);
        }
    } else {
        const int nrc = p.rotary_dim / VEC;  // vectors of the rotary part
        const int j0 = min(c, nrc - 1) * (VEC / 2);
        float4 cs[VEC / 4];
#pragma unroll
        for (int t = 0; t < VEC / 4; ++t) cs[t] = trow[j0 / 2 + t];
        if (c < nrc) {
            ElemIO<T>::unpack(raw, f);
            rope_vec_gptj<T>(f, cs);
            raw = ElemIO<T>::pack(f);
        }
    }
    return raw;
}

// FUSED: the NREP q rows of unit (b, g), rotated as the append rotates them (not when
// the append would refuse the token), into `dst` in shared memory, in the layout of the
// q rows in global memory (one warp; a row takes D / (16 bytes / element) lanes).
template <typename T, int D, int NREP>
__device__ __forceinline__ void rotate_q_unit(const DecodeParams& p, int b, int g, const StepState& s, uint8_t* dst,
                                              int lane) {
    using L = RowLayout<T, D>;
    const int c = lane % L::LPR;
    const bool rot = s.ok && p.rotary_dim > 0;
    const T* qunit = static_cast<const T*>(p.q) + (int64_t(b) * p.Hkv + g) * NREP * D;
    for (int r = lane / L::LPR; r < NREP; r += 32 / L::LPR)
        reinterpret_cast<uint4*>(dst)[r * L::LPR + c] =
            rope_row_vec<T, D>(p, reinterpret_cast<const uint4*>(qunit + r * D), c, s.pos0, rot);
}

// FUSED: the block's first unit (b, g) in one round of loads: its NREP q rows, rotated
// as the append rotates them, into `qdst` in shared memory, and, when `write` is set,
// the token's key (rotated) and value into cache slot s.slot.  Row j of the batch is a
// q row for j < NREP, then the key, then the value; lane l takes chunk l % LPR of rows
// l / LPR, l / LPR + 32 / LPR, ...  Every lane issues all its loads (its chunks, NeoX
// partner chunks and, once, its table pairs: q and k share the token's position and
// the lane's chunk) before any arithmetic.
template <typename T, int D, int NREP>
__device__ __forceinline__ void first_unit_rows(const DecodeParams& p, int b, int g, const StepState& s, bool write,
                                                uint8_t* qdst, int lane) {
    using L = RowLayout<T, D>;
    constexpr int VEC = L::VEC;
    constexpr int RPP = 32 / L::LPR;                   // rows per pass of the warp
    constexpr int NP = (NREP + 2 + RPP - 1) / RPP;     // passes
    const int c = lane % L::LPR;
    const int nrows = NREP + (write ? 2 : 0);
    const bool rot = s.ok && p.rotary_dim > 0;
    const T* qunit = static_cast<const T*>(p.q) + (int64_t(b) * p.Hkv + g) * NREP * D;
    const int64_t src = (int64_t(b) * p.Hkv + g) * D;
    const T* krow = static_cast<const T*>(p.k_new) + src;
    const T* vrow = static_cast<const T*>(p.v_new) + src;
    auto row_of = [&](int j) -> const uint4* {
        return reinterpret_cast<const uint4*>(j < NREP ? qunit + j * D : (j == NREP ? krow : vrow));
    };
    const int half = p.rotary_dim / 2;
    const int hc = half / VEC, nrc = p.rotary_dim / VEC;
    const bool neox = p.neox != 0;
    const int pc = neox ? min(c < hc ? c + hc : c - hc, L::LPR - 1) : c;
    float4 cs[VEC / 2];
    if (rot) {
        const float4* trow = reinterpret_cast<const float4*>(p.table + s.pos0 * half);
        const int j0 = neox ? min(c < hc ? c : c - hc, hc - 1) * VEC : min(c, nrc - 1) * (VEC / 2);
#pragma unroll
        for (int t = 0; t < VEC / 2; ++t) cs[t] = (neox || t < VEC / 4) ? trow[j0 / 2 + t] : make_float4(0.f, 0.f, 0.f, 0.f);
    }
    uint4 raw[NP], pr[NP];
#pragma unroll
    for (int ps = 0; ps < NP; ++ps) {
        const int j = ps * RPP + lane / L::LPR;
        if (j < nrows) {
            const uint4* row = row_of(j);
            raw[ps] = row[c];
            pr[ps] = row[pc];
        }
    }
#pragma unroll
    for (int ps = 0; ps < NP; ++ps) {
        const int j = ps * RPP + lane / L::LPR;
        if (j >= nrows) continue;
        uint4 out = raw[ps];
        if (rot && j <= NREP) {  // q rows and the key
            float f[VEC];
            if (neox && c < 2 * hc) {
                ElemIO<T>::unpack(raw[ps], f);
                rope_vec_neox<T>(f, pr[ps], cs, c < hc);
                out = ElemIO<T>::pack(f);
            } else if (!neox && c < nrc) {
                ElemIO<T>::unpack(raw[ps], f);
                rope_vec_gptj<T>(f, cs);
                out = ElemIO<T>::pack(f);
            }
        }
        if (j < NREP) {
            reinterpret_cast<uint4*>(qdst)[j * L::LPR + c] = out;
        } else {
            T* cache = static_cast<T*>(const_cast<void*>(j == NREP ? p.kc : p.vc));
            reinterpret_cast<uint4*>(cache + ((int64_t(b) * p.Hkv + g) * p.cap + s.slot) * D)[c] = out;
        }
    }
}

// FUSED: the token's rows of unit (b, g) into cache slot s.slot: the key rotated at its
// position as the append rotates it, the value as given (one warp).
template <typename T, int D>
__device__ __forceinline__ void write_new_rows(const DecodeParams& p, int b, int g, const StepState& s, int lane) {
    using L = RowLayout<T, D>;
    const int c = lane % L::LPR;
    const int64_t src = (int64_t(b) * p.Hkv + g) * D;
    const int64_t dst = ((int64_t(b) * p.Hkv + g) * p.cap + s.slot) * D;
    for (int r = lane / L::LPR; r < 2; r += 32 / L::LPR) {
        if (r == 0) {
            const uint4* krow = reinterpret_cast<const uint4*>(static_cast<const T*>(p.k_new) + src);
            reinterpret_cast<uint4*>(static_cast<T*>(const_cast<void*>(p.kc)) + dst)[c] =
                rope_row_vec<T, D>(p, krow, c, s.pos0, p.rotary_dim > 0);
        } else {
            reinterpret_cast<uint4*>(static_cast<T*>(const_cast<void*>(p.vc)) + dst)[c] =
                reinterpret_cast<const uint4*>(static_cast<const T*>(p.v_new) + src)[c];
        }
    }
}

// FUSED: this block's share of the copy of the state (as it stands during the split
// kernel) that the combine kernel advances: block c writes sequences c, c + P, c + 2P, ...
// (one warp; every block of the grid writes its share, so each sequence once).
__device__ __forceinline__ void snapshot_share(const DecodeParams& p, int lane) {
    for (int b = blockIdx.x + lane * int(gridDim.x); b < p.B; b += 32 * int(gridDim.x)) {
        int64_t* sn = p.snap + 4 * int64_t(b);
        sn[0] = p.pos[b];
        sn[1] = p.count != nullptr ? p.count[b] : 0;
        sn[2] = p.head != nullptr ? p.head[b] : 0;
        sn[3] = 0;
    }
}

// Rows of K and V per block that the split kernel asks L2 to fetch before its PDL wait
// (128 KB per block at d_h = 128, bf16).  Measured on the 32 x 4096-row windowed step:
// 128 to 384 rows gave the same gain (about 5%); 768 and more gave less.
constexpr int kPrefetchRows = 256;

// L2 prefetch of the first kPrefetchRows K and V rows of this block's share, from a split
// computed on the current (possibly not yet final) state; rows clamped to the cache.
template <typename C, typename T, int D>
__device__ __forceinline__ void prefetch_share(const DecodeParams& p, const int64_t* pre) {
    const int P = gridDim.x, c = blockIdx.x;
    const int64_t R = pre[p.B];
    if (R <= 0) return;
    const int64_t lo = (int64_t(c) * R + P - 1) / P;
    const int64_t hi = min((int64_t(c + 1) * R + P - 1) / P, lo + kPrefetchRows);
    if (lo >= hi) return;
    UnitWalk w{pre, p.B, p.Hkv, 0, 0};
    w.seek(lo);
    do {
        const int64_t st = w.start();
        if (st >= hi) break;
        const int64_t r0 = max(lo, st) - st;
        const int64_t r1 = min(min(hi, st + w.len()) - st, p.cap);
        if (r1 > r0) {
            const int64_t unit = int64_t(w.b) * p.Hkv + w.g;
            bulk_prefetch_l2(static_cast<const uint8_t*>(p.kc) + (unit * p.cap + r0) * C::K_ROW_BYTES,
                             uint32_t(r1 - r0) * C::K_ROW_BYTES);
            bulk_prefetch_l2(static_cast<const T*>(p.vc) + (unit * p.cap + r0) * D,
                             uint32_t(r1 - r0) * C::ROW_BYTES);
        }
    } while (w.next());
}

// PAGED selects the block-table producer and key-aligned tiles.  The two layouts are
// separate instantiations: the contiguous kernel then carries none of the paged code
// (compiled into one kernel, the contiguous path measured 3-5% slower).  FUSED adds the
// warp that writes the step's token and rotates q: the consumers take their q rows from
// its ring in shared memory (rotating them in the consumer warps themselves cost 10-15%
// of the step: the rotation code alone, never executed, slowed the streaming loop).
template <typename T, int D, int NREP, bool PAGED, bool KQ, bool FUSED = false>
__global__ void __launch_bounds__(DecodeCfg<T, D, NREP, KQ, PAGED, FUSED>::THREADS, 1)
    decode_split_kernel(DecodeParams p) {
    using C = DecodeCfg<T, D, NREP, KQ, PAGED, FUSED>;
    static_assert(!FUSED || (!PAGED && !KQ), "the folded append is for contiguous bf16 or fp32 layers");
    constexpr int NWARPS = C::NWARPS;
    constexpr int STAGES = C::STAGES;
    constexpr int ROWS = FUSED ? kRowsStep : kRowsLive;
    extern __shared__ __align__(128) uint8_t smem[];
    uint8_t* stages = smem;
    float* merge = reinterpret_cast<float*>(smem + C::OFF_MERGE);
    float2* ps_all = reinterpret_cast<float2*>(smem + C::OFF_PS);
    int64_t* pre = reinterpret_cast<int64_t*>(smem + C::OFF_PRE);
    uint64_t* full_bar = reinterpret_cast<uint64_t*>(smem + C::OFF_BAR);
    uint64_t* empty_bar = full_bar + STAGES;
    // FUSED: the token's rows are in the cache; rotated q of a unit in q slot s
    uint64_t* new_bar = reinterpret_cast<uint64_t*>(smem + C::OFF_FUSED);
    uint64_t* q_full = new_bar + 1;
    uint64_t* q_empty = q_full + C::QSLOTS;
    uint8_t* qslots = smem + C::OFF_QSLOT;

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    pdl_trigger();  // the combine kernel may launch now; it waits for this grid to finish
    if (threadIdx.x == 0) {
        for (int s = 0; s < STAGES; ++s) {
            mbar_init(&full_bar[s], 1);
            mbar_init(&empty_bar[s], NWARPS);
        }
        if constexpr (FUSED) {
            mbar_init(new_bar, 1);
            for (int s = 0; s < C::QSLOTS; ++s) {
                mbar_init(&q_full[s], 1);
                mbar_init(&q_empty[s], NWARPS);
            }
        }
        fence_barrier_init();
    }
    if (!PAGED && warp == NWARPS && kPrefetchRows > 0) {
        // While the append before this kernel runs, the memory system is idle: warm L2
        // with the first rows of this block's share, split by the state as it reads now.
        // The append changes at most one row per unit and, on a full ring, no length, so
        // this is the final split in steady state; a stale guess only wastes the hint.
        // (Paged layers take no prefetch: per-block table reads made it a loss there.)
        unit_prefix<ROWS>(p, pre, lane);
        __syncwarp();
        if (lane == 0) prefetch_share<C, T, D>(p, pre);
        __syncwarp();
    }
    pdl_wait();  // the append before this kernel has written the state, q and the new rows
    __syncthreads();  // the producer has finished with the guessed split
    if (warp == 0) unit_prefix<ROWS>(p, pre, lane);
    __syncthreads();

    const int P = gridDim.x, c = blockIdx.x;
    const int64_t R = pre[p.B];
    const int64_t lo = (int64_t(c) * R + P - 1) / P;
    const int64_t hi = (int64_t(c + 1) * R + P - 1) / P;
    if (R == 0 || lo >= hi) {  // no rows here (the token warp still writes its share of the state copy)
        if constexpr (FUSED) {
            if (warp == NWARPS + 1) snapshot_share(p, lane);
        }
        return;
    }
    bool timed_out = false;

    if constexpr (PAGED) {
        if (warp == NWARPS) {
            paged_producer<C, T, D>(p, pre, lo, hi, stages, full_bar, empty_bar, lane);
            return;
        }
    }
    if constexpr (FUSED) {
        if (warp == NWARPS + 1) {
            // ------------------- the step's token, and q rotated -------------------
            // This block writes unit u's token when its share holds the token's slot (or,
            // for a slot past the visible rows, the unit's last row): exactly one block.
            // Order: the first unit's q rows together with its token rows (one round of
            // loads), the other units' token rows (releasing the producer), then q of
            // the other units, each into a ring slot the consumers have released: no
            // wait here depends on the producer's wait for the token rows.
            auto writes = [&](const UnitWalk& u, const StepState& s) {
                const int64_t jw = min(s.slot, u.len() - 1);
                const int64_t at = u.start() + jw;
                return s.ok && at >= lo && at < hi;
            };
            UnitWalk w{pre, p.B, p.Hkv, 0, 0};
            w.seek(lo);
            {
                const StepState s = live_step(p, w.b);
                first_unit_rows<T, D, NREP>(p, w.b, w.g, s, writes(w, s), qslots, lane);
                __syncwarp();
                if (lane == 0) mbar_arrive(&q_full[0]);
            }
            UnitWalk wt = w;
            while (wt.next() && wt.start() < hi) {
                const StepState s = live_step(p, wt.b);
                if (writes(wt, s)) write_new_rows<T, D>(p, wt.b, wt.g, s, lane);
            }
            // the bulk copies (async proxy) of this block read the token rows next
            asm volatile("fence.proxy.async.global;" ::: "memory");
            __syncwarp();
            if (lane == 0) mbar_arrive(new_bar);
            int k = 1;
            while (w.next() && w.start() < hi) {
                const int slot = k % C::QSLOTS;
                if (k >= C::QSLOTS) {
                    if (lane == 0 && !mbar_wait_bounded(&q_empty[slot], ((k / C::QSLOTS) - 1) & 1)) timed_out = true;
                    __syncwarp();
                }
                rotate_q_unit<T, D, NREP>(p, w.b, w.g, live_step(p, w.b), qslots + slot * C::QSLOT_BYTES, lane);
                __syncwarp();
                if (lane == 0) mbar_arrive(&q_full[slot]);
                ++k;
            }
            snapshot_share(p, lane);
            if (timed_out) set_error(p.err, SK_DEVERR_TIMEOUT);
            return;
        }
    }
    if (warp == NWARPS) {
        // ------------------------------ producer ------------------------------
        if (lane == 0) {
            const uint64_t policy = l2_policy_evict_first();
            int stage = 0;
            uint32_t phase = 0;
            bool token_written = !FUSED;
            UnitWalk w{pre, p.B, p.Hkv, 0, 0};
            w.seek(lo);
            do {
                const int64_t st = w.start();
                if (st >= hi) break;
                const int64_t r0 = max(lo, st) - st, r1 = min(hi, st + w.len()) - st;
                const int64_t unit = int64_t(w.b) * p.Hkv + w.g;
                int64_t slot_new = -1;  // FUSED: the row this block's writer warp fills
                if constexpr (FUSED) {
                    const StepState s = live_step(p, w.b);
                    if (s.ok) slot_new = s.slot;
                }
                const uint8_t* kbase = static_cast<const uint8_t*>(p.kc) + unit * p.cap * C::K_ROW_BYTES;
                const T* vbase = static_cast<const T*>(p.vc) + unit * p.cap * D;
                if constexpr (KQ) {  // warm L2 with the segment's row scales (16-byte aligned interior)
                    const uintptr_t a = (reinterpret_cast<uintptr_t>(p.kscale + unit * p.cap + r0) + 15) & ~uintptr_t(15);
                    const uintptr_t e = reinterpret_cast<uintptr_t>(p.kscale + unit * p.cap + r1) & ~uintptr_t(15);
                    if (e > a) bulk_prefetch_l2(reinterpret_cast<const void*>(a), uint32_t(e - a));
                }
                for (int64_t row = r0; row < r1; row += C::TILE) {
                    const uint32_t n = uint32_t(min(int64_t(C::TILE), r1 - row));
                    if (!token_written && slot_new >= row && slot_new < row + n) {
                        if (!mbar_wait_bounded(new_bar, 0)) timed_out = true;
                        token_written = true;
                    }
                    if (!mbar_wait_bounded(&empty_bar[stage], phase ^ 1)) timed_out = true;
                    uint8_t* dst = stages + size_t(stage) * C::STAGE_BYTES;
                    mbar_arrive_expect_tx(&full_bar[stage], n * uint32_t(C::K_ROW_BYTES + C::ROW_BYTES));
                    bulk_copy_g2s(dst, kbase + row * C::K_ROW_BYTES, n * C::K_ROW_BYTES, &full_bar[stage], policy);
                    bulk_copy_g2s(dst + C::TILE * C::K_ROW_BYTES, vbase + row * D, n * C::ROW_BYTES,
                                  &full_bar[stage], policy);
                    if (++stage == STAGES) { stage = 0; phase ^= 1; }
                }
            } while (w.next());
            // Drain: every issued stage has been released by the consumers, so no copy
            // is in flight into shared memory when the block exits.
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
    const int hperm = l8 & (NREP - 1);    // head order of this lane: hh ^ hperm
    const int rperm = l8 >> C::LG;        // row order of this lane: jj ^ rperm
    const int my_row = gi * C::RPG + rperm;   // score held after the reduce-scatter
    const int my_h = hperm;
    float2* ps = ps_all + warp * (C::RPW * NREP + NREP);  // (p,p)[RPW][NREP], then (alpha,alpha)[NREP]
    const T* qbase = static_cast<const T*>(p.q);
    int stage = 0;
    uint32_t phase = 0;
    int uk = 0;  // FUSED: units taken so far (the q ring's position)

    UnitWalk w{pre, p.B, p.Hkv, 0, 0};
    w.seek(lo);
    do {
        const int64_t st = w.start();
        if (st >= hi) break;
        const int64_t Lu = w.len();
        const int64_t r0 = max(lo, st) - st, r1 = min(hi, st + Lu) - st;
        const int b = w.b, g = w.g;
        const int64_t unit = int64_t(b) * p.Hkv + g;

        // q slice of this lane for the NREP heads in its permuted order, pre-scaled: the
        // dims of its K chunks (chunks l8 and l8 + 8 of 8 elements).  With int8 keys the
        // lane's dims are 16 l8 .. 16 l8 + 15 (one 16-code chunk), and q is held as int16
        // pairs with one scale per head: the dot product with the codes is then exact
        // integer arithmetic (dp2a), with no conversion of the codes.
        float2 q2[NREP][KQ ? 1 : C::DPL / 2];
        uint32_t q16[NREP][KQ ? 8 : 1];
        float qsc = p.qscale;  // int8 keys: the scale of this lane's head (slot 0) times qscale
        if constexpr (KQ) {
            float qf[NREP][16];
            float am[NREP];
#pragma unroll
            for (int hh = 0; hh < NREP; ++hh) {
                const T* qrow = qbase + (unit * NREP + (hh ^ hperm)) * D;
                am[hh] = 0.0f;
#pragma unroll
                for (int i = 0; i < 2; ++i) {
                    const uint4 raw = reinterpret_cast<const uint4*>(qrow)[2 * l8 + i];
                    ElemIO<T>::unpack(raw, qf[hh] + 8 * i);
                }
#pragma unroll
                for (int e = 0; e < 16; ++e) am[hh] = fmaxf(am[hh], fabsf(qf[hh][e]));
            }
            // max |q| of each head over its 128 dims: the 8 lanes of the group hold 16 dims
            // each; slot hh of the partner at xor distance x holds this lane's slot
            // hh ^ (x & (NREP - 1)) head
#pragma unroll
            for (int x = 1; x < 8; x <<= 1) {
                float t[NREP];
#pragma unroll
                for (int hh = 0; hh < NREP; ++hh) t[hh] = __shfl_xor_sync(kFull, am[hh ^ (x & (NREP - 1))], x);
#pragma unroll
                for (int hh = 0; hh < NREP; ++hh) am[hh] = fmaxf(am[hh], t[hh]);
            }
#pragma unroll
            for (int hh = 0; hh < NREP; ++hh) {
                const float inv = am[hh] > 0.0f ? 32767.0f / am[hh] : 0.0f;
#pragma unroll
                for (int e = 0; e < 8; ++e) {
                    const int lo = __float2int_rn(qf[hh][2 * e] * inv), hi = __float2int_rn(qf[hh][2 * e + 1] * inv);
                    q16[hh][e] = (uint32_t(lo) & 0xFFFFu) | (uint32_t(hi) << 16);
                }
            }
            qsc = (am[0] > 0.0f ? am[0] / 32767.0f : 0.0f) * p.qscale;
        } else {
            uint4 qv[NREP][C::CPL];
            if constexpr (FUSED) {
                // the unit's q rows, rotated by the token warp into the ring
                const int slot = uk % C::QSLOTS;
                if (!mbar_wait_bounded(&q_full[slot], (uk / C::QSLOTS) & 1)) timed_out = true;
                const uint4* qs = reinterpret_cast<const uint4*>(qslots + slot * C::QSLOT_BYTES);
#pragma unroll
                for (int hh = 0; hh < NREP; ++hh)
#pragma unroll
                    for (int i = 0; i < C::CPL; ++i) qv[hh][i] = qs[(hh ^ hperm) * (D / C::VEC) + l8 + 8 * i];
                __syncwarp();
                if (lane == 0) mbar_arrive(&q_empty[slot]);
                ++uk;
            } else {
#pragma unroll
                for (int hh = 0; hh < NREP; ++hh) {
                    const T* qrow = qbase + (unit * NREP + (hh ^ hperm)) * D;
#pragma unroll
                    for (int i = 0; i < C::CPL; ++i) qv[hh][i] = reinterpret_cast<const uint4*>(qrow)[l8 + 8 * i];
                }
            }
#pragma unroll
            for (int hh = 0; hh < NREP; ++hh) {
#pragma unroll
                for (int i = 0; i < C::CPL; ++i) {
                    float f[C::VEC];
                    ElemIO<T>::unpack(qv[hh][i], f);
#pragma unroll
                    for (int e = 0; e < C::VEC / 2; ++e)
                        q2[hh][i * C::VEC / 2 + e] = make_float2(f[2 * e] * p.qscale, f[2 * e + 1] * p.qscale);
                }
            }
        }

        float m_run = -INFINITY;  // running max of this lane's head (base-2 logits)
        float l_run = 0.0f;       // this lane's share of the running denominator
        float2 acc[NREP][C::DPV / 2];
#pragma unroll
        for (int h = 0; h < NREP; ++h)
#pragma unroll
            for (int d = 0; d < C::DPV / 2; ++d) acc[h][d] = make_float2(0.f, 0.f);

        // int8 keys: this lane's row scale, loaded one tile ahead of its use
        const float* srow = KQ ? p.kscale + unit * p.cap + warp * C::RPW + gi * C::RPG + rperm : nullptr;
        float ks_next = 1.0f;
        if constexpr (KQ) {
            if (r0 + warp * C::RPW + gi * C::RPG + rperm < r1) ks_next = __ldg(srow + r0);
        }
        const int64_t tph = PAGED ? tile_phase(p, b, C::TILE) : 0;
        int n = 0;
        for (int64_t row0 = r0; row0 < r1; row0 += PAGED ? n : C::TILE) {
            const int skip = PAGED ? int((row0 - tph) & (C::TILE - 1)) : 0;
            n = int(min(int64_t(C::TILE - skip), r1 - row0));
            if (!mbar_wait_bounded(&full_bar[stage], phase)) timed_out = true;
            const uint8_t* ktile = stages + size_t(stage) * C::STAGE_BYTES;
            const T* vtile = reinterpret_cast<const T*>(ktile + C::TILE * C::K_ROW_BYTES);
            const int wrow0 = warp * C::RPW;
            const int nw = max(0, min(C::RPW, n - wrow0));  // valid rows of this warp
            float kscale = 1.0f;  // int8 keys: the scale of this lane's row (used after the reduce)
            if constexpr (KQ) {
                kscale = ks_next;
                if (row0 + C::TILE + wrow0 + gi * C::RPG + rperm < r1) ks_next = __ldg(srow + row0 + C::TILE);
            }

            // ---- QK: slot jj*NREP + hh holds row (jj ^ rperm), head (hh ^ hperm) ----
            float part[8];
            if constexpr (KQ) {
                // int8 codes against int16 q: 8 dp2a per (row, head), exact int32 sums
                int ipart[8];
#pragma unroll
                for (int jj = 0; jj < C::RPG; ++jj) {
                    const int lr = gi * C::RPG + (jj ^ rperm);
                    const uint4 kw = lr < nw ? reinterpret_cast<const uint4*>(ktile + (wrow0 + lr) * C::K_ROW_BYTES)[l8]
                                             : make_uint4(0, 0, 0, 0);
                    const uint32_t w4[4] = {kw.x, kw.y, kw.z, kw.w};
#pragma unroll
                    for (int hh = 0; hh < NREP; ++hh) {
                        int a = 0;
#pragma unroll
                        for (int wi = 0; wi < 4; ++wi) {
                            a = __dp2a_lo(int(q16[hh][2 * wi]), int(w4[wi]), a);
                            a = __dp2a_hi(int(q16[hh][2 * wi + 1]), int(w4[wi]), a);
                        }
                        ipart[jj * NREP + hh] = a;
                    }
                }
#pragma unroll
                for (int i = 0; i < 4; ++i) ipart[i] += __shfl_xor_sync(kFull, ipart[i + 4], 4);
#pragma unroll
                for (int i = 0; i < 2; ++i) ipart[i] += __shfl_xor_sync(kFull, ipart[i + 2], 2);
                ipart[0] += __shfl_xor_sync(kFull, ipart[1], 1);
                part[0] = float(ipart[0]) * qsc;
            } else {
#pragma unroll
                for (int jj = 0; jj < C::RPG; ++jj) {
                    const int lr = gi * C::RPG + (jj ^ rperm);
                    float2 kf[C::DPL / 2];
                    if (lr < nw) {
                        const uint4* krow = reinterpret_cast<const uint4*>(ktile + (wrow0 + lr) * C::K_ROW_BYTES);
#pragma unroll
                        for (int i = 0; i < C::CPL; ++i) {
                            const uint4 raw = krow[l8 + 8 * i];
                            if constexpr (sizeof(T) == 2) {
                                kf[i * 4 + 0] = bf16x2_to_float2(raw.x);
                                kf[i * 4 + 1] = bf16x2_to_float2(raw.y);
                                kf[i * 4 + 2] = bf16x2_to_float2(raw.z);
                                kf[i * 4 + 3] = bf16x2_to_float2(raw.w);
                            } else {
                                kf[i * 2 + 0] = make_float2(__uint_as_float(raw.x), __uint_as_float(raw.y));
                                kf[i * 2 + 1] = make_float2(__uint_as_float(raw.z), __uint_as_float(raw.w));
                            }
                        }
                    } else {
#pragma unroll
                        for (int e = 0; e < C::DPL / 2; ++e) kf[e] = make_float2(0.f, 0.f);
                    }
#pragma unroll
                    for (int hh = 0; hh < NREP; ++hh) {
                        float2 a = __fmul2_rn(q2[hh][0], kf[0]);
#pragma unroll
                        for (int e = 1; e < C::DPL / 2; ++e) a = __ffma2_rn(q2[hh][e], kf[e], a);
                        part[jj * NREP + hh] = a.x + a.y;
                    }
                }
                // ---- butterfly reduce-scatter: slot i of lane L holds value i ^ L ----
#pragma unroll
                for (int i = 0; i < 4; ++i) part[i] += __shfl_xor_sync(kFull, part[i + 4], 4);
#pragma unroll
                for (int i = 0; i < 2; ++i) part[i] += __shfl_xor_sync(kFull, part[i + 2], 2);
                part[0] += __shfl_xor_sync(kFull, part[1], 1);
            }
            const float s = my_row < nw ? (KQ ? part[0] * kscale : part[0]) : -INFINITY;

            // ---- online softmax (base 2) for this lane's head ----
            float tmax = s;
#pragma unroll
            for (int o = NREP; o < 32; o <<= 1) tmax = fmaxf(tmax, __shfl_xor_sync(kFull, tmax, o));
            const float m_new = fmaxf(m_run, tmax);
            const float m_use = m_new == -INFINITY ? 0.0f : m_new;
            const float pr = fast_exp2_approx(s - m_use);
            // Lazy rescale (bf16 / fp32 keys, contiguous or paged, two-call path): the
            // accumulators are rescaled only in tiles where some head's running max grew
            // (warp-uniform); otherwise every head's factor would be exactly 1.  Measured:
            // windowed step +1.1%, paged +3.2%; int8 keys -0.4% and the decode step -0.4%,
            // which keep the rescale in every tile.
            constexpr bool kLazy = !KQ && !FUSED;
            const bool grew = kLazy ? __any_sync(kFull, m_new > m_run) : true;
            if (grew) {
                const float alpha = fast_exp2_approx(m_run - m_use);
                l_run = fmaf(l_run, alpha, pr);
                if (lane < NREP) ps[C::RPW * NREP + lane] = make_float2(alpha, alpha);  // lane h: head h
            } else {
                l_run += pr;
            }
            m_run = m_new;
            ps[my_row * NREP + my_h] = make_float2(pr, pr);
            __syncwarp();

            // ---- PV ----
            if (grew) {
#pragma unroll
                for (int h = 0; h < NREP; ++h) {
                    const float2 a2 = ps[C::RPW * NREP + h];
#pragma unroll
                    for (int d = 0; d < C::DPV / 2; ++d) acc[h][d] = __fmul2_rn(acc[h][d], a2);
                }
            }
            if (nw == C::RPW) {
#pragma unroll
                for (int r = 0; r < C::RPW; ++r) {
                    float2 vf[C::DPV / 2];
                    load_pv_slice<T, C::DPV>(vtile + (wrow0 + r) * D, lane, vf);
                    if constexpr (NREP >= 2 && !KQ && !PAGED) {
                        // the (p, p) pairs of two heads in one 16-byte load (measured: +2% on
                        // the contiguous bf16 step, -0.5 to -1% for paged layers and int8 keys)
#pragma unroll
                        for (int h = 0; h < NREP; h += 2) {
                            const float4 pp = *reinterpret_cast<const float4*>(&ps[r * NREP + h]);
#pragma unroll
                            for (int d = 0; d < C::DPV / 2; ++d) {
                                acc[h][d] = __ffma2_rn(make_float2(pp.x, pp.y), vf[d], acc[h][d]);
                                acc[h + 1][d] = __ffma2_rn(make_float2(pp.z, pp.w), vf[d], acc[h + 1][d]);
                            }
                        }
                    } else {
#pragma unroll
                        for (int h = 0; h < NREP; ++h) {
                            const float2 pp = ps[r * NREP + h];
#pragma unroll
                            for (int d = 0; d < C::DPV / 2; ++d) acc[h][d] = __ffma2_rn(pp, vf[d], acc[h][d]);
                        }
                    }
                }
            } else {
                for (int r = 0; r < nw; ++r) {
                    float2 vf[C::DPV / 2];
                    load_pv_slice<T, C::DPV>(vtile + (wrow0 + r) * D, lane, vf);
#pragma unroll
                    for (int h = 0; h < NREP; ++h) {
                        const float2 pp = ps[r * NREP + h];
#pragma unroll
                        for (int d = 0; d < C::DPV / 2; ++d) acc[h][d] = __ffma2_rn(pp, vf[d], acc[h][d]);
                    }
                }
            }
            __syncwarp();
            if (lane == 0) mbar_arrive(&empty_bar[stage]);
            if (++stage == STAGES) { stage = 0; phase ^= 1; }
        }

        // ---- merge the warps' states and write this block's partial of the unit ----
        float l_tot = l_run;
#pragma unroll
        for (int o = NREP; o < 32; o <<= 1) l_tot += __shfl_xor_sync(kFull, l_tot, o);
        float* mw = merge + warp * NREP * (D + 2);
        if (lane < NREP) {
            mw[lane] = m_run;  // lane h holds head h
            mw[NREP + lane] = l_tot;
        }
#pragma unroll
        for (int h = 0; h < NREP; ++h)
#pragma unroll
            for (int d = 0; d < C::DPV / 2; ++d)
                *reinterpret_cast<float2*>(mw + 2 * NREP + h * D + lane * C::DPV + 2 * d) = acc[h][d];
        asm volatile("bar.sync 1, %0;" ::"n"(NWARPS * 32) : "memory");
        const int64_t fb = first_block_of(st, R, P);
        float* outp = p.ws + (fb + unit + (c - fb)) * C::PARTIAL_FLOATS;
        for (int idx = threadIdx.x; idx < NREP * D; idx += NWARPS * 32) {
            const int h = idx / D, d = idx % D;
            float M = -INFINITY;
#pragma unroll
            for (int ww = 0; ww < NWARPS; ++ww) M = fmaxf(M, merge[ww * NREP * (D + 2) + h]);
            const float Mu = M == -INFINITY ? 0.0f : M;
            float a = 0.0f, lsum = 0.0f;
#pragma unroll
            for (int ww = 0; ww < NWARPS; ++ww) {
                const float* mm = merge + ww * NREP * (D + 2);
                const float f = fast_exp2_approx(mm[h] - Mu);
                a = fmaf(f, mm[2 * NREP + h * D + d], a);
                lsum = fmaf(f, mm[NREP + h], lsum);
            }
            outp[2 * NREP + h * D + d] = a;
            if (d == 0) {
                outp[h] = M;
                outp[NREP + h] = lsum;
            }
        }
        asm volatile("bar.sync 1, %0;" ::"n"(NWARPS * 32) : "memory");
    } while (w.next());
    if (timed_out) set_error(p.err, SK_DEVERR_TIMEOUT);
}

// FUSED: the step's state change for sequence b, after the split kernel (one thread per
// sequence; the split kernel's copy of the state decides, as in the split kernel).
__device__ __forceinline__ void advance_step(const DecodeParams& p, int b) {
    const StepState s = snap_step(p, b);
    if (!s.ok) {
        set_error(p.err, s.err);
        return;
    }
    if (p.kind == SK_LAYER_RING) {
        p.head_rw[b] = s.head;
        p.count_rw[b] = s.count;
    }
    p.pos_rw[b] = s.pos;
}

// Log-sum-exp combine of each unit's partials, one warp per (b, q head): the kernel for
// batches whose units meet one to three blocks each.  FUSED: rows after the step's
// token (before the wait from the state as it stands, a guess; after it from the split
// kernel's copy), and the warp of (b, q head 0) advances sequence b's state.
constexpr int kCombineFew = 3;  // partials a combine warp loads in one go

template <typename T, int D, int NREP, bool FUSED = false>
__global__ void __launch_bounds__(256) decode_combine_kernel(DecodeParams p) {
    constexpr int DPV = D / 32;
    constexpr int PF = NREP * (D + 2);
    // the row prefix from the state as read before the wait (a guess) and after it
    __shared__ int64_t pre[2][kMaxBatch + 1];
    const int lane = threadIdx.x & 31;
    pdl_trigger();
    // Before the wait the state is final unless the append ahead of the split kernel is
    // still running. The guess only picks the partials to load as soon as the wait
    // returns, alongside the state read after it, which decides whether they are used.
    if (threadIdx.x < 32) unit_prefix<FUSED ? kRowsStep : kRowsLive>(p, pre[0], lane);
    __syncthreads();
    const int warp_global = blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5);
    const int Hq = p.Hkv * NREP;
    const bool active = warp_global < p.B * Hq;
    const int b = active ? warp_global / Hq : 0, hq = active ? warp_global % Hq : 0;
    const int g = hq / NREP, h = hq % NREP;
    const int64_t unit = int64_t(b) * p.Hkv + g;
    const int P = p.n_blocks;
    // blocks fb..fb+n-1 own the unit's rows, except blocks whose row range is empty
    // (possible when R < P): those wrote nothing and are skipped.
    auto owns_rows = [&](int64_t c, int64_t R) { return (c * R + P - 1) / P < ((c + 1) * R + P - 1) / P; };
    float mv[kCombineFew], lv[kCombineFew], vv[kCombineFew][DPV];
    // every partial's max, sum and value slice of a unit cut between at most kCombineFew
    // blocks, at once (one round trip to L2); a block that wrote nothing gives max -inf
    auto load_few = [&](int64_t fb, int n, int64_t R) {
        const float* base = p.ws + (fb + unit) * PF;
#pragma unroll
        for (int i = 0; i < kCombineFew; ++i) {
            const bool own = i < n && owns_rows(fb + i, R);
            const float* pp = base + i * PF;
            mv[i] = own ? pp[h] : -INFINITY;
            lv[i] = own ? pp[NREP + h] : 0.0f;
#pragma unroll
            for (int d = 0; d < DPV; ++d) vv[i][d] = own ? pp[2 * NREP + h * D + lane * DPV + d] : 0.0f;
        }
    };
    // the guessed split of the unit; n0 = 0: nothing loaded early
    int64_t fb0 = 0, R0 = pre[0][p.B];
    int n0 = 0;
    {
        const int64_t s0 = pre[0][b], e0 = pre[0][b + 1];
        const int64_t L0 = (e0 - s0) / p.Hkv;
        if (active && R0 > 0 && L0 > 0 && s0 >= 0 && e0 <= R0) {
            const int64_t st0 = s0 + int64_t(g) * L0;
            fb0 = first_block_of(st0, R0, P);
            const int64_t lb0 = first_block_of(st0 + L0 - 1, R0, P);
            if (fb0 >= 0 && lb0 < P && lb0 - fb0 + 1 <= kCombineFew) n0 = int(lb0 - fb0 + 1);
        }
    }
    pdl_wait();  // the split kernel's partials are complete
    if (n0 > 0) load_few(fb0, n0, R0);
    if (threadIdx.x < 32) unit_prefix<FUSED ? kRowsSnap : kRowsLive>(p, pre[1], lane);
    if constexpr (FUSED) {
        if (active && hq == 0 && lane == 0) advance_step(p, b);
    }
    __syncthreads();
    if (!active) return;
    const int64_t R = pre[1][p.B];
    const int64_t Lb = (pre[1][b + 1] - pre[1][b]) / p.Hkv;
    T* o = static_cast<T*>(p.out) + (int64_t(b) * Hq + hq) * D + lane * DPV;
    if (Lb == 0) {
#pragma unroll
        for (int d = 0; d < DPV; ++d) o[d] = T(0.0f);
        return;
    }
    const int64_t st = pre[1][b] + int64_t(g) * Lb;
    const int64_t fb = first_block_of(st, R, P);
    const int64_t lb = first_block_of(st + Lb - 1, R, P);
    const int n = int(lb - fb + 1);
    // A learned sink is one more logit z (scaled-score units, clamped) in the
    // denominator with no value row ("RoPE, scaling, sliding window, attention sinks",
    // "Hybrid models break the uniform-spec assumption"); in base 2 it is z log2(e).
    const bool has_sink = p.sink_logits != nullptr;
    const float z2 = has_sink
                         ? fminf(fmaxf(p.sink_logits[hq], kSinkLogitMin), kSinkLogitMax) * kLog2e
                         : -INFINITY;
    float acc[DPV];
#pragma unroll
    for (int d = 0; d < DPV; ++d) acc[d] = 0.0f;
    float lsum;
    if (n <= kCombineFew) {
        // the same blocks under the same ownership rule: the early loads are the partials
        if (!(n0 == n && fb0 == fb && R0 == R)) load_few(fb, n, R);
        float M = z2;
#pragma unroll
        for (int i = 0; i < kCombineFew; ++i) M = fmaxf(M, mv[i]);
        const float Mu = M == -INFINITY ? 0.0f : M;
        lsum = has_sink ? fast_exp2_approx(z2 - Mu) : 0.0f;
#pragma unroll
        for (int i = 0; i < kCombineFew; ++i) {
            const float f = fast_exp2_approx(mv[i] - Mu);  // 0 for a block that wrote nothing
            lsum = fmaf(f, lv[i], lsum);
#pragma unroll
            for (int d = 0; d < DPV; ++d) acc[d] = fmaf(f, vv[i][d], acc[d]);
        }
    } else {
        // A unit cut between more blocks than usual (a long sequence among short ones):
        // the lanes take the partials 32 at a time for the max and the sum, then every
        // lane adds its dims of each partial, the weights broadcast by shuffle, several
        // partials' loads in flight at once.
        const float* base = p.ws + (fb + unit) * PF;
        float M = z2;
        for (int i0 = 0; i0 < n; i0 += 32) {
            const int i = i0 + lane;
            if (i < n && owns_rows(fb + i, R)) M = fmaxf(M, base[i * PF + h]);
        }
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) M = fmaxf(M, __shfl_xor_sync(kFull, M, o));
        const float Mu = M == -INFINITY ? 0.0f : M;
        float lpart = 0.0f;
        for (int i0 = 0; i0 < n; i0 += 32) {
            const int i = i0 + lane;
            // a block that owns none of the unit's rows wrote nothing here: weight 0,
            // and its (stale) slot is never read
            const bool own = i < n && owns_rows(fb + i, R);
            const float f = own ? fast_exp2_approx(base[i * PF + h] - Mu) : 0.0f;
            if (own) lpart = fmaf(f, base[i * PF + NREP + h], lpart);
            const int cnt = min(32, n - i0);
            constexpr int U = 4;
            for (int j0 = 0; j0 < cnt; j0 += U) {
                float fj[U], vj[U][DPV];
#pragma unroll
                for (int u = 0; u < U; ++u) {
                    fj[u] = __shfl_sync(kFull, f, (j0 + u) & 31);
                    const bool use = j0 + u < cnt && fj[u] != 0.0f;
                    const float* pp = base + (i0 + j0 + u) * PF + 2 * NREP + h * D + lane * DPV;
#pragma unroll
                    for (int d = 0; d < DPV; ++d) vj[u][d] = use ? pp[d] : 0.0f;
                    if (!use) fj[u] = 0.0f;
                }
#pragma unroll
                for (int u = 0; u < U; ++u)
#pragma unroll
                    for (int d = 0; d < DPV; ++d) acc[d] = fmaf(fj[u], vj[u][d], acc[d]);
            }
        }
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) lpart += __shfl_xor_sync(kFull, lpart, o);
        lsum = lpart + (has_sink ? fast_exp2_approx(z2 - Mu) : 0.0f);
    }
    const float inv = lsum > 0.0f ? 1.0f / lsum : 0.0f;
#pragma unroll
    for (int d = 0; d < DPV; ++d) {
        if constexpr (sizeof(T) == 2)
            o[d] = __float2bfloat16_rn(acc[d] * inv);
        else
            o[d] = acc[d] * inv;
    }
}

// KQ: int8 keys (contiguous layers only; paged layers hold bf16 or fp32 keys).

// Log-sum-exp combine for few, long units (a single sequence or a few): a group of
// p.combine_wpu warps (2, 4 or 8, all in one block) per (b, q head).  Warp `sub` of the group takes the partials
// [sub n / wpu, (sub + 1) n / wpu) of the n blocks that met the unit, kCombineBatch at a
// time, folding them into a running (max, sum, values); the group's warps then merge
// through shared memory.  The host picks wpu from the partials a unit meets on average,
// so that a warp's share is one batch: a single round trip to L2 after the wait (a
// single sequence of 8 kv heads meets about 20 blocks per unit).
constexpr int kCombineBatch = 4;  // partials a combine warp loads in one go

template <typename T, int D, int NREP, bool FUSED = false>
__global__ void __launch_bounds__(256) decode_combine_group_kernel(DecodeParams p) {
    constexpr int DPV = D / 32;
    constexpr int PF = NREP * (D + 2);
    constexpr int KB = kCombineBatch;
    // the row prefix from the state as read before the wait (a guess) and after it
    __shared__ int64_t pre[2][kMaxBatch + 1];
    __shared__ float mrg[8][2 + D];  // per warp: running max, sum and its lanes' values
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    pdl_trigger();
    // Before the wait the state is final unless the append ahead of the split kernel is
    // still running. The guess only picks the partials to load as soon as the wait
    // returns, alongside the state read after it, which decides whether they are used.
    if (threadIdx.x < 32) unit_prefix<FUSED ? kRowsStep : kRowsLive>(p, pre[0], lane);
    __syncthreads();
    const int wpu = p.combine_wpu;
    const int wg = blockIdx.x * 8 + warp;
    const int item = wg / wpu, sub = wg % wpu;
    const int Hq = p.Hkv * NREP;
    const bool active = item < p.B * Hq;
    const int b = active ? item / Hq : 0, hq = active ? item % Hq : 0;
    const int g = hq / NREP, h = hq % NREP;
    const int64_t unit = int64_t(b) * p.Hkv + g;
    const int P = p.n_blocks;
    // blocks fb..fb+n-1 meet the unit's rows, except blocks whose row range is empty
    // (possible when R < P): those wrote nothing and are skipped.
    auto owns_rows = [&](int64_t c, int64_t R) { return (c * R + P - 1) / P < ((c + 1) * R + P - 1) / P; };
    auto share = [&](int n, int* j0, int* j1) {
        *j0 = int(int64_t(sub) * n / wpu);
        *j1 = int(int64_t(sub + 1) * n / wpu);
    };
    float mv[KB], lv[KB], vv[KB][DPV];
    // max, sum and value slice of partials j0 .. j1-1 (at most KB) at once; a block
    // that wrote nothing gives max -inf and is never read
    auto load = [&](int64_t fb, int64_t R, int j0, int j1) {
        const float* base = p.ws + (fb + unit) * PF;
#pragma unroll
        for (int i = 0; i < KB; ++i) {
            const int j = j0 + i;
            const bool own = j < j1 && owns_rows(fb + j, R);
            const float* pp = base + j * PF;
            mv[i] = own ? pp[h] : -INFINITY;
            lv[i] = own ? pp[NREP + h] : 0.0f;
#pragma unroll
            for (int d = 0; d < DPV; ++d) vv[i][d] = own ? pp[2 * NREP + h * D + lane * DPV + d] : 0.0f;
        }
    };
    // the guessed split of the unit and this warp's first batch of it; n0 = 0: nothing
    // loaded early
    int64_t fb0 = 0, R0 = pre[0][p.B];
    int n0 = 0, g0 = 0, g1 = 0;
    {
        const int64_t s0 = pre[0][b], e0 = pre[0][b + 1];
        const int64_t L0 = (e0 - s0) / p.Hkv;
        if (active && R0 > 0 && L0 > 0 && s0 >= 0 && e0 <= R0) {
            const int64_t st0 = s0 + int64_t(g) * L0;
            fb0 = first_block_of(st0, R0, P);
            const int64_t lb0 = first_block_of(st0 + L0 - 1, R0, P);
            if (fb0 >= 0 && lb0 < P && lb0 >= fb0) n0 = int(lb0 - fb0 + 1);
        }
        if (n0 > 0) share(n0, &g0, &g1);
    }
    pdl_wait();  // the split kernel's partials are complete
    if (n0 > 0) load(fb0, R0, g0, min(g1, g0 + KB));
    if (threadIdx.x < 32) unit_prefix<FUSED ? kRowsSnap : kRowsLive>(p, pre[1], lane);
    if constexpr (FUSED) {
        if (active && hq == 0 && sub == 0 && lane == 0) advance_step(p, b);
    }
    __syncthreads();
    const int64_t R = pre[1][p.B];
    const int64_t Lb = active ? (pre[1][b + 1] - pre[1][b]) / p.Hkv : 0;
    float m_loc = -INFINITY, l_loc = 0.0f, acc[DPV];
#pragma unroll
    for (int d = 0; d < DPV; ++d) acc[d] = 0.0f;
    if (Lb > 0) {
        const int64_t st = pre[1][b] + int64_t(g) * Lb;
        const int64_t fb = first_block_of(st, R, P);
        const int n = int(first_block_of(st + Lb - 1, R, P) - fb + 1);
        int j0, j1;
        share(n, &j0, &j1);
        // the same blocks under the same ownership rule: the early loads are this batch
        const bool early = n0 == n && fb0 == fb && R0 == R;
        for (int jb = j0; jb < j1; jb += KB) {
            if (!(early && jb == j0)) load(fb, R, jb, min(j1, jb + KB));
            float Mb = m_loc;
#pragma unroll
            for (int i = 0; i < KB; ++i) Mb = fmaxf(Mb, mv[i]);
            const float Mu = Mb == -INFINITY ? 0.0f : Mb;
            const float alpha = fast_exp2_approx(m_loc - Mu);  // 0 while nothing is folded in
            l_loc *= alpha;
#pragma unroll
            for (int d = 0; d < DPV; ++d) acc[d] *= alpha;
#pragma unroll
            for (int i = 0; i < KB; ++i) {
                const float f = fast_exp2_approx(mv[i] - Mu);  // 0 for a block that wrote nothing
                l_loc = fmaf(f, lv[i], l_loc);
#pragma unroll
                for (int d = 0; d < DPV; ++d) acc[d] = fmaf(f, vv[i][d], acc[d]);
            }
            m_loc = Mb;
        }
    }
    // A learned sink is one more logit z (scaled-score units, clamped) in the
    // denominator with no value row ("RoPE, scaling, sliding window, attention sinks",
    // "Hybrid models break the uniform-spec assumption"); in base 2 it is z log2(e).
    const bool has_sink = p.sink_logits != nullptr;
    const float z2 = has_sink && active
                         ? fminf(fmaxf(p.sink_logits[hq], kSinkLogitMin), kSinkLogitMax) * kLog2e
                         : -INFINITY;
    float lsum;
    if (wpu > 1) {
        if (lane == 0) {
            mrg[warp][0] = m_loc;
            mrg[warp][1] = l_loc;
        }
#pragma unroll
        for (int d = 0; d < DPV; ++d) mrg[warp][2 + lane * DPV + d] = acc[d];
        __syncthreads();
        if (sub != 0 || !active) return;
        float M = z2;
        for (int s = 0; s < wpu; ++s) M = fmaxf(M, mrg[warp + s][0]);
        const float Mu = M == -INFINITY ? 0.0f : M;
        lsum = has_sink ? fast_exp2_approx(z2 - Mu) : 0.0f;
#pragma unroll
        for (int d = 0; d < DPV; ++d) acc[d] = 0.0f;
        for (int s = 0; s < wpu; ++s) {
            const float f = fast_exp2_approx(mrg[warp + s][0] - Mu);
            lsum = fmaf(f, mrg[warp + s][1], lsum);
#pragma unroll
            for (int d = 0; d < DPV; ++d) acc[d] = fmaf(f, mrg[warp + s][2 + lane * DPV + d], acc[d]);
        }
    } else {
        if (!active) return;
        const float M = fmaxf(z2, m_loc);
        const float Mu = M == -INFINITY ? 0.0f : M;
        const float f = fast_exp2_approx(m_loc - Mu);
        lsum = fmaf(f, l_loc, has_sink ? fast_exp2_approx(z2 - Mu) : 0.0f);
#pragma unroll
        for (int d = 0; d < DPV; ++d) acc[d] *= f;
    }
    T* o = static_cast<T*>(p.out) + (int64_t(b) * Hq + hq) * D + lane * DPV;
    const float inv = (Lb > 0 && lsum > 0.0f) ? 1.0f / lsum : 0.0f;
#pragma unroll
    for (int d = 0; d < DPV; ++d) {
        if constexpr (sizeof(T) == 2)
            o[d] = __float2bfloat16_rn(acc[d] * inv);
        else
            o[d] = acc[d] * inv;
    }
}

// Warps per (b, q head) of the combine: enough that a warp's share of the partials a
// unit meets on average (about P / units + 1) is one batch.
inline int combine_wpu(int P, int64_t units) {
    const int64_t avg = int64_t(P) / std::max<int64_t>(1, units) + 1;
    int w = 1;
    while (w < 8 && (avg + w - 1) / w > kCombineBatch) w <<= 1;
    return w;
}

// KQ: int8 keys (contiguous layers only; paged layers hold bf16 or fp32 keys).
template <typename T, int D, int NREP, bool KQ = false>
struct DecodeLaunch {
    using C = DecodeCfg<T, D, NREP, KQ, false>;   // contiguous layers
    using CP = DecodeCfg<T, D, NREP, KQ, true>;   // paged layers (never with int8 keys)

    // Every instantiation launched from here (contiguous, and paged unless KQ) gets its
    // shared-memory limit; the grid is sized from the smallest occupancy among them.
    static int blocks_per_sm() {
        static PerDevice<int> cache;
        return cache.get(
            [] {
                int n0 = 0, n1 = 0;
                if (cudaFuncSetAttribute(decode_split_kernel<T, D, NREP, false, KQ>,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize, int(C::SMEM)) != cudaSuccess ||
                    cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n0, decode_split_kernel<T, D, NREP, false, KQ>,
                                                                  C::THREADS, C::SMEM) != cudaSuccess)
                    return 0;
                if constexpr (KQ) {
                    return n0;
                } else {
                    if (cudaFuncSetAttribute(decode_split_kernel<T, D, NREP, true, false>,
                                             cudaFuncAttributeMaxDynamicSharedMemorySize,
                                             int(CP::SMEM)) != cudaSuccess ||
                        cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n1, decode_split_kernel<T, D, NREP, true, false>,
                                                                      CP::THREADS, CP::SMEM) != cudaSuccess)
                        return 0;
                    return std::min(n0, n1);
                }
            },
            [](int n) { return n > 0; }, 0);
    }

    static int grid() { return std::max(1, blocks_per_sm()) * device_sm_count(); }

    static size_t workspace(const sk_kv_layer& L) {
        return size_t(grid() + int64_t(L.batch) * L.n_kv_heads) * C::PARTIAL_FLOATS * sizeof(float);
    }

    static cudaError_t run(DecodeParams p, const sk_kv_layer& L, cudaStream_t st) {
        if (blocks_per_sm() < 1) return cudaErrorInvalidConfiguration;
        p.n_blocks = grid();
        if (p.kind != kKindPaged) {
            // no more blocks than rows the cache can hold: blocks without rows would only
            // add partials for the combine to skip
            const int64_t rows = int64_t(L.batch) * L.n_kv_heads * L.capacity;
            p.n_blocks = int(std::max<int64_t>(1, std::min<int64_t>(p.n_blocks, rows)));
        }
        cudaError_t e;
        if constexpr (KQ) {
            if (p.kind == kKindPaged) return cudaErrorInvalidValue;
            e = launch_pdl(decode_split_kernel<T, D, NREP, false, true>, dim3(p.n_blocks), dim3(C::THREADS), C::SMEM,
                           st, p);
        } else {
            e = p.kind == kKindPaged
                    ? launch_pdl(decode_split_kernel<T, D, NREP, true, false>, dim3(p.n_blocks), dim3(CP::THREADS),
                                 CP::SMEM, st, p)
                    : launch_pdl(decode_split_kernel<T, D, NREP, false, false>, dim3(p.n_blocks), dim3(C::THREADS),
                                 C::SMEM, st, p);
        }
        if (e != cudaSuccess) return e;
        p.combine_wpu = combine_wpu(p.n_blocks, int64_t(L.batch) * L.n_kv_heads);
        const int64_t warps = int64_t(L.batch) * L.n_kv_heads * NREP * p.combine_wpu;
        return p.combine_wpu == 1
                   ? launch_pdl(decode_combine_kernel<T, D, NREP>, dim3(unsigned((warps + 7) / 8)), dim3(256), 0, st,
                                p)
                   : launch_pdl(decode_combine_group_kernel<T, D, NREP>, dim3(unsigned((warps + 7) / 8)), dim3(256),
                                0, st, p);
    }
};

sk_status check_layer(const sk_kv_layer* layer, int32_t n_q_heads) {
    SK_RET_IF(layer == nullptr, SK_ERR_ARG);
    const sk_kv_layer& L = *layer;
    SK_RET_IF(L.k == nullptr || L.v == nullptr || L.pos == nullptr, SK_ERR_ARG);
    SK_RET_IF(L.batch < 1 || L.n_kv_heads < 1 || L.capacity < 1, SK_ERR_ARG);
    SK_RET_IF(L.batch > kMaxBatch, SK_ERR_UNSUPPORTED);
    SK_RET_IF(n_q_heads < 1 || n_q_heads % L.n_kv_heads != 0, SK_ERR_ARG);
    if (L.kind == SK_LAYER_RING) {
        SK_RET_IF(L.count == nullptr || L.sinks < 0 || L.window < 1, SK_ERR_ARG);
        SK_RET_IF(L.capacity != int64_t(L.sinks) + L.window, SK_ERR_ARG);
    } else {
        SK_RET_IF(L.kind != SK_LAYER_GLOBAL, SK_ERR_ARG);
    }
    SK_RET_IF((reinterpret_cast<uintptr_t>(L.k) | reinterpret_cast<uintptr_t>(L.v)) & 15u, SK_ERR_ARG);
    if (L.k_dtype == SK_I8)
        SK_RET_IF(L.k_scale == nullptr || (reinterpret_cast<uintptr_t>(L.k_scale) & 3u), SK_ERR_ARG);
    return SK_OK;
}

}  // namespace
}  // namespace sk
