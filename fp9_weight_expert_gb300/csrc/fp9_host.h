// Host-side helpers for the C-ABI entry points: argument checks that run
// before anything touches CUDA, and cached device properties.
#pragma once

#include <cstdint>

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

// Number of SMs of the current device (-1 if it cannot be queried).
int32_t device_sm_count();

// Largest dynamic shared memory per block on the current device.
int32_t device_max_smem_optin();

}  // namespace fp9
