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

}  // namespace sk

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

extern "C" int32_t sk_version(void) { return 200; }
