// abi.cu -- host-side pieces of the C ABI: status strings, device queries,
// and the offline int8 quantiser.
#include <math.h>
#include <stdlib.h>
#include <string.h>

#include <mutex>

#include "common.cuh"

namespace moe {

namespace {
std::mutex g_dev_mutex;
int g_sm_count[64];
int g_smem_optin[64];
}  // namespace

static void query_device(int dev) {
    std::lock_guard<std::mutex> lock(g_dev_mutex);
    if (dev < 0 || dev >= 64 || g_sm_count[dev] > 0) return;
    int v = 0;
    if (cudaDeviceGetAttribute(&v, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || v < 1)
        v = 1;
    int s = 0;
    if (cudaDeviceGetAttribute(&s, cudaDevAttrMaxSharedMemoryPerBlockOptin, dev) != cudaSuccess)
        s = 48 * 1024;
    g_smem_optin[dev] = s;
    g_sm_count[dev] = v;
}

int sm_count() {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return 1;
    query_device(dev);
    return (dev >= 0 && dev < 64) ? g_sm_count[dev] : 1;
}

int max_smem_optin() {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return 48 * 1024;
    query_device(dev);
    return (dev >= 0 && dev < 64) ? g_smem_optin[dev] : 48 * 1024;
}

bool pdl_enabled() {
    static const bool on = [] {
        const char *v = getenv("MOE_DISABLE_PDL");
        return !(v && v[0] == '1');
    }();
    return on;
}

}  // namespace moe

extern "C" const char *moe_status_string(int status) {
    switch (status) {
        case MOE_OK: return "MOE_OK: success";
        case MOE_ERR_INVALID_ARG: return "MOE_ERR_INVALID_ARG: invalid argument";
        case MOE_ERR_UNSUPPORTED: return "MOE_ERR_UNSUPPORTED: outside the supported limits";
        case MOE_ERR_ALIGNMENT:
            return "MOE_ERR_ALIGNMENT: pointer not 16-byte aligned or size not a multiple of 8";
        case MOE_ERR_WORKSPACE: return "MOE_ERR_WORKSPACE: workspace too small";
        case MOE_ERR_CUDA: return "MOE_ERR_CUDA: CUDA runtime or driver error";
        case MOE_ERR_DEVICE_CHECK: return "MOE_ERR_DEVICE_CHECK: device-side data check failed";
        case MOE_ERR_TIMEOUT: return "MOE_ERR_TIMEOUT: a bounded device-side wait ran out";
        default: return "unknown moe_status";
    }
}

extern "C" int moe_version(void) { return 100; }

static inline float bf16_to_float(uint16_t b) {
    const uint32_t u = static_cast<uint32_t>(b) << 16;
    float f;
    memcpy(&f, &u, sizeof f);
    return f;
}

extern "C" moe_status moe_quantize_w8(const uint16_t *w_host, int64_t rows, int64_t K,
                                      int8_t *q_host, float *scale_host) {
    if (!w_host || !q_host || !scale_host || rows < 0 || K < 1) return MOE_ERR_INVALID_ARG;
#pragma omp parallel for schedule(static)
    for (int64_t n = 0; n < rows; ++n) {
        const uint16_t *w = w_host + n * K;
        float amax = 0.0f;
        for (int64_t c = 0; c < K; ++c) amax = fmaxf(amax, fabsf(bf16_to_float(w[c])));
        const float scale = amax > 0.0f ? amax / 127.0f : 1.0f;
        scale_host[n] = scale;
        int8_t *q = q_host + n * K;
        for (int64_t c = 0; c < K; ++c) {
            float r = nearbyintf(bf16_to_float(w[c]) / scale);   // ties to even
            r = fminf(fmaxf(r, -127.0f), 127.0f);
            q[c] = static_cast<int8_t>(r);
        }
    }
    return MOE_OK;
}
