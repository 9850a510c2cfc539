// Library-wide state: error messages, the device status word, host helpers.
#include <cmath>
#include <cstdarg>
#include <cstdlib>
#include <cstdio>
#include <cstring>
#include <mutex>

#include "common.cuh"

namespace bsa {

static thread_local char g_msg[512] = "";

// One status word per device: kernels latch BSA_ERR_INDEX / BSA_ERR_TIMEOUT here.
__device__ int g_device_status = 0;

void set_error(const char* fmt, ...) {
    va_list ap;
    va_start(ap, fmt);
    vsnprintf(g_msg, sizeof(g_msg), fmt, ap);
    va_end(ap);
}

bsa_status fail(bsa_status code, const char* fmt, ...) {
    va_list ap;
    va_start(ap, fmt);
    vsnprintf(g_msg, sizeof(g_msg), fmt, ap);
    va_end(ap);
    return code;
}

bsa_status check_launch(const char* what) {
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return fail(BSA_ERR_CUDA, "%s: %s", what, cudaGetErrorString(e));
    return BSA_OK;
}

int* status_word() {
    static std::mutex mu;
    static int* addr[64] = {nullptr};
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return nullptr;
    std::lock_guard<std::mutex> lock(mu);
    if (!addr[dev]) {
        void* p = nullptr;
        if (cudaGetSymbolAddress(&p, g_device_status) != cudaSuccess) return nullptr;
        addr[dev] = static_cast<int*>(p);
    }
    return addr[dev];
}

__device__ unsigned g_sched[2 * kSchedSlots];

unsigned* sched_counter(cudaStream_t st) {
    static std::mutex mu;
    static unsigned* base[64] = {nullptr};
    static cudaStream_t owner[64][kSchedSlots];
    static int used[64] = {0};
    cudaStreamCaptureStatus cap = cudaStreamCaptureStatusNone;
    if (cudaStreamIsCapturing(st, &cap) != cudaSuccess) {
        cudaGetLastError();
        return nullptr;
    }
    if (cap != cudaStreamCaptureStatusNone) return nullptr;
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return nullptr;
    std::lock_guard<std::mutex> lock(mu);
    if (!base[dev]) {
        void* p = nullptr;
        if (cudaGetSymbolAddress(&p, g_sched) != cudaSuccess || !p) {
            cudaGetLastError();
            return nullptr;
        }
        base[dev] = static_cast<unsigned*>(p);
    }
    for (int i = 0; i < used[dev]; ++i)
        if (owner[dev][i] == st) return base[dev] + 2 * i;
    if (used[dev] == kSchedSlots) return nullptr;
    owner[dev][used[dev]] = st;
    return base[dev] + 2 * used[dev]++;
}

// BSA_FORCE_SIMT (set, and not "0") routes every attention stage to its
// CUDA-core kernel; the tests use it to compare the two kernel families.
bool force_simt() {
    const char* e = std::getenv("BSA_FORCE_SIMT");
    return e && e[0] && !(e[0] == '0' && e[1] == 0);
}

int test_stall_tile() {
    const char* e = std::getenv("BSA_TEST_STALL_TILE");
    if (!e || !e[0]) return -1;
    char* end = nullptr;
    const long v = std::strtol(e, &end, 10);
    return (end && *end == 0 && v >= 0 && v < 1000000) ? (int)v : -1;
}

}  // namespace bsa

extern "C" {

int bsa_version(void) { return 100; }

const char* bsa_last_error(void) { return bsa::g_msg; }

bsa_status bsa_device_status(void* stream) {
    cudaError_t e = cudaStreamSynchronize(bsa::as_stream(stream));
    if (e != cudaSuccess) return bsa::fail(BSA_ERR_CUDA, "stream sync: %s", cudaGetErrorString(e));
    int* w = bsa::status_word();
    if (!w) return bsa::fail(BSA_ERR_CUDA, "device status word unavailable");
    int v = 0;
    e = cudaMemcpyFromSymbol(&v, bsa::g_device_status, sizeof(int));
    if (e != cudaSuccess) return bsa::fail(BSA_ERR_CUDA, "status read: %s", cudaGetErrorString(e));
    int zero = 0;
    e = cudaMemcpyToSymbol(bsa::g_device_status, &zero, sizeof(int));
    if (e != cudaSuccess) return bsa::fail(BSA_ERR_CUDA, "status clear: %s", cudaGetErrorString(e));
    if (v != 0) bsa::set_error("device reported status %d", v);
    return static_cast<bsa_status>(v);
}

bsa_status bsa_get_device_status(void* stream) { return bsa_device_status(stream); }

const char* bsa_last_error_string(void) { return bsa_last_error(); }

int bsa_budget(int J, double sparsity) {
    if (J < 1 || !(sparsity >= 0.0 && sparsity <= 1.0)) return -1;
    double r = std::ceil((1.0 - sparsity) * (double)J - 1e-9);
    int R = (int)r;
    if (R > J) R = J;
    if (R < 1) R = 1;
    return R;
}

}  // extern "C"
