// Host-side launch helpers shared by the CUDA translation units.
#pragma once

#include <cuda_runtime.h>

#include <string>

#include "bfp_device.cuh"
#include "bfp_internal.h"

namespace bfp {

constexpr int64_t kDefaultWaitIters = int64_t(1) << 40;
constexpr uint64_t kDefaultWaitNanos = 2000000000ull;  // 2 s wall clock per wait

inline int cuda_fail(cudaError_t e, const char *what) {
    return fail(BFP_ECUDA, std::string(what) + ": " + cudaGetErrorString(e));
}

struct DeviceInfo {
    int device = -1;
    int sms = 0;
    int smem_optin = 0;
};

// SM count and opt-in shared memory of the current device.
int device_info(DeviceInfo *out);

inline dev::WaitCfg wait_cfg() {
    int64_t it = wait_limit();
    dev::WaitCfg w;
    if (it > 0) {
        w.iters = it;
        w.nanos = kDefaultWaitNanos;
    } else {
        w.iters = kDefaultWaitIters;
        w.nanos = kDefaultWaitNanos;
    }
    return w;
}

// cudaFuncSetAttribute(MaxDynamicSharedMemorySize) once per (kernel, device, size): the call costs
// microseconds of host time, which a one-row layer launch cannot afford every time.
int set_smem_attr(const void *kernel, int smem, const char *what);

// Workspace header: status word at byte 0 (16 bytes reserved).
constexpr size_t kWsHeader = 256;

__host__ __device__ inline size_t align_up(size_t v, size_t a) { return (v + a - 1) / a * a; }

}  // namespace bfp
