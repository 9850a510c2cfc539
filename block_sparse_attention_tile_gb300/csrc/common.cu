// Library-wide state: error messages, the device status word, host helpers.
#include <cmath>
#include <cstdarg>
#include <cstdio>
#include <cstring>
#include <mutex>

#include "common.cuh"

namespace bsa {

static thread_local char g_msg[512] = "";
static bool g_force_simt = false;

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

bool force_simt() { return g_force_simt; }

}  // namespace bsa

extern "C" {

int bsa_version(void) { return 100; }

const char* bsa_last_error(void) { return bsa::g_msg; }

void bsa_set_force_simt(int force) { bsa::g_force_simt = force != 0; }

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
