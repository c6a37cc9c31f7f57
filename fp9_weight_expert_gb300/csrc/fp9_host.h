// Host-side helpers for the C-ABI entry points: argument checks that run
// before anything touches CUDA, and cached device properties.
#pragma once

#include <cstdint>
#include <mutex>
#include <utility>

#include <cuda_runtime.h>

#include "fp9moe.h"

namespace fp9 {

inline bool aligned(const void* p, uintptr_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }

#define FP9_CHECK_ARG(cond, code) \
    do {                          \
        if (!(cond)) return (code); \
    } while (0)

#define FP9_CUDA_TRY(expr)                          \
    do {                                            \
        if ((expr) != cudaSuccess) {                \
            (void)cudaGetLastError();               \
            return FP9_ERR_CUDA;                    \
        }                                           \
    } while (0)

// Validates a bank's pointers, alignment and shape (no CUDA calls).
inline fp9_status check_bank(const fp9_ffn_bank& b, int64_t n, int64_t inter, int64_t hidden) {
    FP9_CHECK_ARG(b.n == n && b.inter == inter && b.hidden == hidden, FP9_ERR_SHAPE);
    const void* planes[6] = {b.gate_body, b.gate_sign, b.up_body, b.up_sign, b.down_body, b.down_sign};
    for (const void* p : planes) {
        FP9_CHECK_ARG(p != nullptr, FP9_ERR_INVALID_ARG);
        FP9_CHECK_ARG(aligned(p, 16), FP9_ERR_ALIGN);
    }
    return FP9_OK;
}

// Hidden-size rule of the fused kernels: a multiple of 128 (so that every
// row of the sign plane starts 16-byte aligned for the bulk copies) and at
// most FP9_MAX_HIDDEN (one 16-column chunk per consumer thread).
inline bool hidden_ok(int64_t h) { return h >= 128 && h <= FP9_MAX_HIDDEN && h % 128 == 0; }

// Launches `kernel` on `stream` as a programmatic dependent of the work
// queued before it: the launch may begin while the previous kernel is
// still running, and each kernel of this library executes
// griddepcontrol.wait before it reads anything an earlier launch wrote.
template <typename... KArgs, typename... Args>
cudaError_t launch_pdl(void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem, cudaStream_t stream,
                       Args&&... args) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = grid;
    cfg.blockDim = block;
    cfg.dynamicSmemBytes = smem;
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, kernel, std::forward<Args>(args)...);
}

// One-time set-up per device (kernel attributes): `run` calls `setup` the
// first time it is called with a given device current, under a mutex, so
// first calls from several host threads at once are safe. A set-up that
// fails is tried again on the next call.
struct DeviceOnce {
    std::mutex mu;
    bool done[64] = {};

    template <typename F>
    fp9_status run(F&& setup) {
        int dev = 0;
        if (cudaGetDevice(&dev) != cudaSuccess) {
            (void)cudaGetLastError();
            return FP9_ERR_CUDA;
        }
        if (dev < 0 || dev >= 64) return FP9_ERR_CUDA;
        std::lock_guard<std::mutex> lock(mu);
        if (!done[dev]) {
            const fp9_status st = setup();
            if (st != FP9_OK) return st;
            done[dev] = true;
        }
        return FP9_OK;
    }
};

// Number of SMs of the current device (-1 if it cannot be queried).
int32_t device_sm_count();

// Largest dynamic shared memory per block on the current device.
int32_t device_max_smem_optin();

}  // namespace fp9
