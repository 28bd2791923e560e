// Per-lane rotary embedding of one 16-byte vector of a row, shared by the RoPE + KV
// append and by the decode step that folds the append into attention: both rotate a
// row with exactly this arithmetic, so the rotated rows they produce are bit-identical.
//
// "RoPE, scaling, sliding window, attention sinks": the rotation listing
// (o1 = x1 cos - x2 sin, o2 = x2 cos + x1 sin), NeoX vs GPT-J pairing, partial rotary,
// and the cos/sin table gather with no trigonometry at runtime.
#pragma once

#include "common.cuh"

namespace sk {
namespace {

template <typename T, int D> struct RowLayout {
    static constexpr int VEC = ElemIO<T>::kPerVec;  // elements per lane
    static constexpr int LPR = D / VEC;             // lanes per row: 8, 16 or 32
    static constexpr int RPW = 32 / LPR;            // rows per warp
};

// 16-byte chunks of (cos, sin) pairs a lane needs: NeoX lanes hold VEC pairs (one per
// element), GPT-J lanes VEC/2 pairs.
template <typename T, bool NEOX> constexpr int table_chunks() {
    return NEOX ? ElemIO<T>::kPerVec / 2 : ElemIO<T>::kPerVec / 4;
}

// First (cos, sin) pair index of lane c's elements, and whether the lane rotates.
template <typename T, int D, bool NEOX>
__device__ __forceinline__ bool lane_pairs(int rotary_dim, int c, int* j0) {
    constexpr int VEC = RowLayout<T, D>::VEC;
    if constexpr (NEOX) {
        const int hc = (rotary_dim / 2) / VEC;
        *j0 = (c < hc ? c : c - hc) * VEC;
        return c < 2 * hc;
    } else {
        *j0 = c * VEC / 2;
        return c * VEC < rotary_dim;
    }
}

// The rotation arithmetic of one 16-byte vector.  NeoX: the VEC elements f of a chunk
// in the first (first = true) or second half of the rotary part, with the partner
// vector pr from the other half and the (cos, sin) pairs of the chunk's VEC pairs in
// cs[0 .. VEC/2) (two pairs per float4).  GPT-J: adjacent pairs inside the vector, VEC/2
// pairs in cs[0 .. VEC/4).
template <typename T>
__device__ __forceinline__ void rope_vec_neox(float* f, const uint4& pr, const float4* cs, bool first) {
    constexpr int VEC = ElemIO<T>::kPerVec;
    float p[VEC];
    ElemIO<T>::unpack(pr, p);
    // first half: x1 c - x2 s; second half: x2 c + x1 s
    const float2 sg = first ? make_float2(-1.0f, -1.0f) : make_float2(1.0f, 1.0f);
#pragma unroll
    for (int i = 0; i < VEC / 2; ++i) {
        const float4 t = cs[i];  // (cos, sin) of the lane's pairs 2i, 2i+1
        const float2 fc = __fmul2_rn(make_float2(f[2 * i], f[2 * i + 1]), make_float2(t.x, t.z));
        const float2 ps = __fmul2_rn(make_float2(p[2 * i], p[2 * i + 1]), sg);
        const float2 o = __ffma2_rn(ps, make_float2(t.y, t.w), fc);
        f[2 * i] = o.x;
        f[2 * i + 1] = o.y;
    }
}

template <typename T>
__device__ __forceinline__ void rope_vec_gptj(float* f, const float4* cs) {
    constexpr int VEC = ElemIO<T>::kPerVec;
#pragma unroll
    for (int i = 0; i < VEC / 4; ++i) {
        const float4 t = cs[i];
        float x1 = f[4 * i], x2 = f[4 * i + 1];
        f[4 * i] = fmaf(-x2, t.y, x1 * t.x);
        f[4 * i + 1] = fmaf(x1, t.y, x2 * t.x);
        x1 = f[4 * i + 2];
        x2 = f[4 * i + 3];
        f[4 * i + 2] = fmaf(-x2, t.w, x1 * t.z);
        f[4 * i + 3] = fmaf(x1, t.w, x2 * t.z);
    }
}

// Rotate the VEC elements of this lane (c = lane index within its row), with the lane's
// (cos, sin) pairs at cs (global or shared memory).  A NeoX rotation needs the lane's
// partner vector in the other half of the rotary part: with ROW_IN_SMEM it is loaded
// from `row` (the row in shared memory), else every lane of the warp must call this (it
// shuffles).  `active` lanes update f.
template <typename T, int D, bool NEOX, bool ROW_IN_SMEM = false>
__device__ __forceinline__ void rotate_lane(float* f, const uint4& raw, const float4* cs, int rotary_dim, int c,
                                            int lane, bool active, const uint4* row = nullptr) {
    constexpr int VEC = RowLayout<T, D>::VEC;
    if constexpr (NEOX) {
        const int hc = (rotary_dim / 2) / VEC;  // vectors per half of the rotary part
        const bool rot = c < 2 * hc;
        const int partner_c = c < hc ? c + hc : c - hc;
        uint4 pr;
        if constexpr (ROW_IN_SMEM) {
            pr = active && rot ? row[partner_c] : raw;
        } else {
            const int src = lane - c + (rot ? partner_c : c);
            pr.x = __shfl_sync(0xffffffffu, raw.x, src);
            pr.y = __shfl_sync(0xffffffffu, raw.y, src);
            pr.z = __shfl_sync(0xffffffffu, raw.z, src);
            pr.w = __shfl_sync(0xffffffffu, raw.w, src);
        }
        if (active && rot) rope_vec_neox<T>(f, pr, cs, c < hc);
    } else {
        if (active && c * VEC < rotary_dim) rope_vec_gptj<T>(f, cs);
    }
}

}  // namespace
}  // namespace sk
