// Shared host/device helpers of the library's translation units.
#pragma once

#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include <cstdio>
#include <string>

#include "../../include/bsa.h"

namespace bsa {

// ---------------------------------------------------------------- host errors
void set_error(const char* fmt, ...);
bsa_status fail(bsa_status code, const char* fmt, ...);
bsa_status check_launch(const char* what);

// Device address of the device status word of the current device.
int* status_word();

// Whether the caller asked for the CUDA-core kernels only.
bool force_simt();

// Tests of the bounded waits only: BSA_TEST_STALL_TILE = n makes the next
// tensor-core token attention leave the K loads of each CTA's n-th tile
// unissued and limit every wait to 1 ms, so the waits run out, the kernel
// latches BSA_ERR_TIMEOUT and returns.  -1 (the default) when unset.
int test_stall_tile();

// Work counters of the persistent tensor-core kernels: a pair of unsigned
// (next item, CTAs done), both zero between launches, per (current device,
// stream) in static device memory.  Launches on one stream run one after
// another and the last CTA of each puts its pair back to zero.  Returns null
// (the kernel then takes every gridDim.x-th item, a static schedule) when
// all kSchedSlots pairs of the device are taken or when the stream is being
// captured into a CUDA graph: a graph may later be replayed while other work
// runs on the stream it was captured from, and must not share a pair with it.
constexpr int kSchedSlots = 64;
unsigned* sched_counter(cudaStream_t st);

inline cudaStream_t as_stream(void* s) { return reinterpret_cast<cudaStream_t>(s); }

#define BSA_REQUIRE(cond, ...)                                           \
    do {                                                                 \
        if (!(cond)) return ::bsa::fail(BSA_ERR_INVALID_ARG, __VA_ARGS__); \
    } while (0)

// ---------------------------------------------------------------- device helpers
__device__ __forceinline__ void raise_status(int* status, int code) {
    if (status) atomicCAS(status, 0, code);
}

__device__ __forceinline__ float to_f32(float x) { return x; }
__device__ __forceinline__ float to_f32(__nv_bfloat16 x) { return __bfloat162float(x); }

template <typename T> __device__ __forceinline__ T from_f32(float x);
template <> __device__ __forceinline__ float from_f32<float>(float x) { return x; }
template <> __device__ __forceinline__ __nv_bfloat16 from_f32<__nv_bfloat16>(float x) {
    return __float2bfloat16_rn(x);
}

__device__ __forceinline__ float warp_max(float v) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, o));
    return v;
}
__device__ __forceinline__ float warp_sum(float v) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
    return v;
}

constexpr float kLog2e = 1.4426950408889634f;
constexpr float kLn2 = 0.6931471805599453f;

}  // namespace bsa
