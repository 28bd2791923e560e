// Shared device helpers for libsinkkv: bf16 packing, mbarrier / bulk-copy PTX,
// bounded waits.  sm_103a only.
#pragma once

#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include <mutex>

#include "../../include/sinkkv.h"

#define SK_RET_IF(cond, status) \
    do {                        \
        if (cond) return (status); \
    } while (0)

#define SK_CUDA_RET(call)                          \
    do {                                           \
        cudaError_t e_ = (call);                   \
        if (e_ != cudaSuccess) return SK_ERR_CUDA; \
    } while (0)

namespace sk {

// ---------------------------------------------------------------------------
// Element types.
// ---------------------------------------------------------------------------

// Two bf16 in one 32-bit word -> two floats (bf16 is the high half of an fp32).
__device__ __forceinline__ float2 bf16x2_to_float2(uint32_t w) {
    return make_float2(__uint_as_float(w << 16), __uint_as_float(w & 0xffff0000u));
}

// Two floats -> two bf16 (round to nearest even) in one 32-bit word.
__device__ __forceinline__ uint32_t float2_to_bf16x2(float lo, float hi) {
    __nv_bfloat162 h = __floats2bfloat162_rn(lo, hi);
    return *reinterpret_cast<uint32_t*>(&h);
}

template <typename T> struct ElemIO;

template <> struct ElemIO<float> {
    static constexpr int kPerVec = 4;  // elements in 16 bytes
    __device__ __forceinline__ static void unpack(const uint4& u, float* f) {
        f[0] = __uint_as_float(u.x); f[1] = __uint_as_float(u.y);
        f[2] = __uint_as_float(u.z); f[3] = __uint_as_float(u.w);
    }
    __device__ __forceinline__ static uint4 pack(const float* f) {
        return make_uint4(__float_as_uint(f[0]), __float_as_uint(f[1]),
                          __float_as_uint(f[2]), __float_as_uint(f[3]));
    }
};

template <> struct ElemIO<__nv_bfloat16> {
    static constexpr int kPerVec = 8;
    __device__ __forceinline__ static void unpack(const uint4& u, float* f) {
        float2 a = bf16x2_to_float2(u.x), b = bf16x2_to_float2(u.y);
        float2 c = bf16x2_to_float2(u.z), d = bf16x2_to_float2(u.w);
        f[0] = a.x; f[1] = a.y; f[2] = b.x; f[3] = b.y;
        f[4] = c.x; f[5] = c.y; f[6] = d.x; f[7] = d.y;
    }
    __device__ __forceinline__ static uint4 pack(const float* f) {
        return make_uint4(float2_to_bf16x2(f[0], f[1]), float2_to_bf16x2(f[2], f[3]),
                          float2_to_bf16x2(f[4], f[5]), float2_to_bf16x2(f[6], f[7]));
    }
};

// ---------------------------------------------------------------------------
// int8 codes (symmetric, one fp32 scale per row).
// ---------------------------------------------------------------------------

// Codes of four values: rint(x * inv), rint half to even, for |x| <= max|x| of the row
// and inv = 127 / max|x| (so |x * inv| < 127.5 and the code lies in [-127, 127]).
// Adding 1.5 * 2^23 to a value of magnitude below 2^22 rounds it to the nearest
// integer (ties to even) and leaves that integer, two's complement, in the low byte.
__device__ __forceinline__ uint32_t float4_to_codes(const float* x, float inv) {
    uint32_t r[4];
#pragma unroll
    for (int e = 0; e < 4; ++e)  // the product is rounded first: no fused multiply-add here
        r[e] = __float_as_uint(__fadd_rn(__fmul_rn(x[e], inv), 12582912.0f));
    const uint32_t lo = __byte_perm(r[0], r[1], 0x0040);
    const uint32_t hi = __byte_perm(r[2], r[3], 0x0040);
    return __byte_perm(lo, hi, 0x5410);
}

// Row scale max|x| / 127 and its quantisation multiplier 127 / max|x| (IEEE fp32
// divisions, once per row); a zero row gets scale 1 and multiplier 0.
__device__ __forceinline__ void int8_row_scale(float amax, float* scale, float* inv) {
    if (amax == 0.0f) {
        *scale = 1.0f;
        *inv = 0.0f;
    } else {
        *scale = __fdiv_rn(amax, 127.0f);
        *inv = __fdiv_rn(127.0f, amax);
    }
}

// ---------------------------------------------------------------------------
// Shared-memory barriers and bulk copies (inline PTX).
// ---------------------------------------------------------------------------

__device__ __forceinline__ uint32_t smem_u32(const void* p) {
    return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ void mbar_init(uint64_t* bar, uint32_t count) {
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(bar)), "r"(count)
                 : "memory");
}

__device__ __forceinline__ void fence_barrier_init() {
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint64_t* bar, uint32_t bytes) {
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_u32(bar)),
                 "r"(bytes)
                 : "memory");
}

__device__ __forceinline__ void mbar_arrive(uint64_t* bar) {
    asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_u32(bar)) : "memory");
}

__device__ __forceinline__ bool mbar_try_wait(uint64_t* bar, uint32_t parity) {
    uint32_t ok;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}\n"
        : "=r"(ok)
        : "r"(smem_u32(bar)), "r"(parity)
        : "memory");
    return ok != 0;
}

__device__ __forceinline__ uint64_t global_timer_ns() {
    uint64_t t;
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
    return t;
}

// Wait for the phase of `bar` with the given parity.  Gives up after about one
// second and returns false; callers then record SK_DEVERR_TIMEOUT and carry on, so
// a kernel can never spin forever.
__device__ __forceinline__ bool mbar_wait_bounded(uint64_t* bar, uint32_t parity) {
    if (mbar_try_wait(bar, parity)) return true;
    const uint64_t t0 = global_timer_ns();
    while (true) {
#pragma unroll 1
        for (int i = 0; i < 32; ++i)
            if (mbar_try_wait(bar, parity)) return true;
        if (global_timer_ns() - t0 > 1000000000ull) return false;
    }
}

// L2 policy: data streamed once (evict first).
__device__ __forceinline__ uint64_t l2_policy_evict_first() {
    uint64_t p;
    asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(p));
    return p;
}

// One-dimensional bulk copy global -> shared, completion counted in bytes on `bar`.
// Both addresses 16-byte aligned, bytes a multiple of 16.
__device__ __forceinline__ void bulk_copy_g2s(void* smem_dst, const void* gmem_src, uint32_t bytes,
                                              uint64_t* bar, uint64_t policy) {
    asm volatile(
        "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes.L2::cache_hint "
        "[%0], [%1], %2, [%3], %4;" ::"r"(smem_u32(smem_dst)),
        "l"(gmem_src), "r"(bytes), "r"(smem_u32(bar)), "l"(policy)
        : "memory");
}

// Bulk prefetch of global memory into L2 (a hint: no completion, no data returned).
// Address 16-byte aligned, bytes a multiple of 16.
__device__ __forceinline__ void bulk_prefetch_l2(const void* gmem_src, uint32_t bytes) {
    asm volatile("cp.async.bulk.prefetch.L2.global [%0], %1;" ::"l"(gmem_src), "r"(bytes) : "memory");
}

// 16 int8 codes -> 8 exact float pairs (byte permute under 2^23, subtract 2^23 + 128).
__device__ __forceinline__ void codes16_to_pairs(const uint4& u, float2* f) {
    const uint32_t w[4] = {u.x ^ 0x80808080u, u.y ^ 0x80808080u, u.z ^ 0x80808080u, u.w ^ 0x80808080u};
    const float2 bias = make_float2(-8388736.0f, -8388736.0f);
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        f[2 * i] = __fadd2_rn(make_float2(__uint_as_float(__byte_perm(w[i], 0x4B000000u, 0x7540)),
                                          __uint_as_float(__byte_perm(w[i], 0x4B000000u, 0x7541))), bias);
        f[2 * i + 1] = __fadd2_rn(make_float2(__uint_as_float(__byte_perm(w[i], 0x4B000000u, 0x7542)),
                                              __uint_as_float(__byte_perm(w[i], 0x4B000000u, 0x7543))), bias);
    }
}

// 2^x with the hardware approximation (ex2.approx.ftz.f32): -inf -> +0.
__device__ __forceinline__ float fast_exp2_approx(float x) {
    float y;
    asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}

// Programmatic dependent launch: a kernel launched with launch_pdl may start while the
// previous kernel on the stream is still running.  pdl_wait() blocks until that kernel
// has completed and its writes are visible: call it before the first access to
// anything an earlier kernel writes.  pdl_trigger() lets the next kernel launch early.
// Both are no-ops for a kernel launched without the attribute.
__device__ __forceinline__ void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
__device__ __forceinline__ void pdl_trigger() { asm volatile("griddepcontrol.launch_dependents;" ::: "memory"); }

// The same copy without a cache hint (for small data that is read again, like table rows).
__device__ __forceinline__ void bulk_copy_g2s_nohint(void* smem_dst, const void* gmem_src, uint32_t bytes,
                                                     uint64_t* bar) {
    asm volatile(
        "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(
            smem_u32(smem_dst)),
        "l"(gmem_src), "r"(bytes), "r"(smem_u32(bar))
        : "memory");
}

__device__ __forceinline__ void set_error(uint32_t* err, uint32_t bits) {
    if (err != nullptr) atomicOr(err, bits);
}

}  // namespace sk

// Launch `kernel` with programmatic stream serialization allowed (see pdl_wait).
template <typename... KArgs, typename... Args>
cudaError_t launch_pdl(void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem, cudaStream_t st,
                       Args&&... args) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = grid;
    cfg.blockDim = block;
    cfg.dynamicSmemBytes = smem;
    cfg.stream = st;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, kernel, static_cast<Args&&>(args)...);
}

// Host helpers shared by the entry points.
namespace sk {
int device_sm_count();                                   // api.cu
const float2* table_device(const sk_rope_table* t);      // rope_table.cu
const sk_rope_config& table_config(const sk_rope_table* t);

// A value computed once for each device (the current one) and kept: kernel attributes
// and occupancy belong to a device, so a process that drives several GPUs sets them on
// each.  A result `keep` rejects is not kept, and the next call computes it again.
constexpr int kMaxDevices = 64;
template <typename V>
struct PerDevice {
    std::mutex mu;
    bool done[kMaxDevices] = {};
    V val[kMaxDevices] = {};
    template <typename Make, typename Keep>
    V get(Make make, Keep keep, V no_device) {
        int dev = 0;
        if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return no_device;
        std::lock_guard<std::mutex> lock(mu);
        if (!done[dev]) {
            val[dev] = make();
            done[dev] = keep(val[dev]);
        }
        return val[dev];
    }
};

// cudaFuncSetAttribute(kernel, MaxDynamicSharedMemorySize, bytes) once per device.
template <typename Kernel>
cudaError_t set_smem_limit_once(PerDevice<cudaError_t>& cache, Kernel kernel, int bytes) {
    return cache.get([&] { return cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes); },
                     [](cudaError_t e) { return e == cudaSuccess; }, cudaErrorInvalidDevice);
}
}

namespace sk {
// Kernel-side layer kind of a paged layer (sk_paged_layer); not an sk_layer_kind.
constexpr int kKindPaged = 2;

// Host check of a paged layer descriptor shared by the paged entry points.
inline sk_status paged_layer_check(const sk_paged_layer& L) {
    if (L.k_pool == nullptr || L.v_pool == nullptr || L.block_table == nullptr || L.seq_lens == nullptr)
        return SK_ERR_ARG;
    if (L.batch < 1 || L.n_kv_heads < 1 || L.max_blocks < 1 || L.n_blocks < 1) return SK_ERR_ARG;
    if (L.head_dim != 64 && L.head_dim != 128) return SK_ERR_ARG;
    if (L.block_size < 4 || L.block_size > 1024 || (L.block_size & (L.block_size - 1)) != 0) return SK_ERR_ARG;
    if (L.n_sink_blocks < 0 || (L.n_sink_blocks > 0 && L.sink_block_ids == nullptr)) return SK_ERR_ARG;
    if (int64_t(L.n_sink_blocks) * L.block_size > (int64_t(1) << 30)) return SK_ERR_ARG;
    if (L.sinks < 0 || L.k_dtype != L.v_dtype || (L.k_dtype != SK_BF16 && L.k_dtype != SK_F32)) return SK_ERR_ARG;
    if ((reinterpret_cast<uintptr_t>(L.k_pool) | reinterpret_cast<uintptr_t>(L.v_pool)) & 15u) return SK_ERR_ARG;
    return SK_OK;
}
}  // namespace sk
