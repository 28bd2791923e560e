// Miscellaneous C-ABI entry points and host helpers.
#include "common.cuh"

namespace sk {

// Streaming multiprocessors of the current device (152 on GB300), cached per device.
int device_sm_count() {
    static int cached[64] = {0};
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return 1;
    if (cached[dev] == 0) {
        int n = 0;
        if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || n < 1)
            n = 1;
        cached[dev] = n;
    }
    return cached[dev];
}

namespace {

// One thread waits, through the library's bounded wait, on an mbarrier that nothing
// will ever complete: the wait gives up after its limit and the error word says so.
__global__ void bounded_wait_probe_kernel(uint32_t* err) {
    __shared__ __align__(8) uint64_t bar;
    mbar_init(&bar, 1);
    fence_barrier_init();
    if (!mbar_wait_bounded(&bar, 0)) set_error(err, SK_DEVERR_TIMEOUT);
}

}  // namespace
}  // namespace sk

extern "C" sk_status sk_selftest_bounded_wait(uint32_t* err, void* stream) {
    SK_RET_IF(err == nullptr, SK_ERR_ARG);
    sk::bounded_wait_probe_kernel<<<1, 1, 0, static_cast<cudaStream_t>(stream)>>>(err);
    return cudaGetLastError() == cudaSuccess ? SK_OK : SK_ERR_CUDA;
}

extern "C" const char* sk_status_str(sk_status status) {
    switch (status) {
        case SK_OK: return "SK_OK";
        case SK_ERR_ARG: return "SK_ERR_ARG: invalid argument";
        case SK_ERR_CAPACITY: return "SK_ERR_CAPACITY: cache capacity exceeded";
        case SK_ERR_POSITION_RANGE: return "SK_ERR_POSITION_RANGE: position outside the RoPE table";
        case SK_ERR_UNSUPPORTED: return "SK_ERR_UNSUPPORTED: combination not implemented";
        case SK_ERR_CUDA: return "SK_ERR_CUDA: CUDA runtime error";
        default: return "unknown sk_status";
    }
}

extern "C" sk_status sk_sync_check(uint32_t* err, int32_t clear, void* stream, uint32_t* bits_out) {
    SK_RET_IF(err == nullptr, SK_ERR_ARG);
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    uint32_t bits = 0;
    SK_CUDA_RET(cudaMemcpyAsync(&bits, err, sizeof(bits), cudaMemcpyDeviceToHost, st));
    SK_CUDA_RET(cudaStreamSynchronize(st));
    if (clear && bits != 0) {
        SK_CUDA_RET(cudaMemsetAsync(err, 0, sizeof(uint32_t), st));
        SK_CUDA_RET(cudaStreamSynchronize(st));
    }
    if (bits_out != nullptr) *bits_out = bits;
    if (bits & SK_DEVERR_CAPACITY) return SK_ERR_CAPACITY;
    if (bits & SK_DEVERR_POSITION_RANGE) return SK_ERR_POSITION_RANGE;
    if (bits & (SK_DEVERR_BLOCK_TABLE | SK_DEVERR_STATE)) return SK_ERR_ARG;
    if (bits & SK_DEVERR_TIMEOUT) return SK_ERR_CUDA;
    return SK_OK;
}

extern "C" int32_t sk_version(void) { return 200; }
