// gla_common.cuh — small helpers shared by the CUDA translation units of libgla.
//
// Nothing here computes any part of the method; it holds element conversions,
// the per-translation-unit device status word and host-side launch plumbing.
#pragma once

#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "gla.h"

namespace gla {

// ---- element types -------------------------------------------------------
__device__ __forceinline__ float to_f32(float x) { return x; }
__device__ __forceinline__ float to_f32(__nv_bfloat16 x) { return __bfloat162float(x); }

template <typename T> __device__ __forceinline__ T from_f32(float x);
template <> __device__ __forceinline__ float from_f32<float>(float x) { return x; }
template <> __device__ __forceinline__ __nv_bfloat16 from_f32<__nv_bfloat16>(float x) { return __float2bfloat16_rn(x); }

// Output gate factor (the gate g_t of the QKVG projection acts on the mixer output): kind 0 multiplies
// by SiLU(g) = g / (1 + e^-g), kind 1 by the sigmoid 1 / (1 + e^-g).  For g below about -87 the
// exponential overflows to +inf and the reciprocal to 0, which is the limit.
__device__ __forceinline__ float gate_factor(float g, int kind) {
    const float sig = __fdividef(1.f, 1.f + __expf(-g));
    return kind == 0 ? g * sig : sig;
}

// ---- chain bookkeeping ---------------------------------------------------
// A chain is one (sequence, head) pair.  Dense batches: sequence s covers rows
// s*T .. s*T+T-1.  Packed batches: rows cu[s] .. cu[s+1]-1.  Returns false (and
// lets the caller record GLA_ERR_DEVICE_ARG) when packed offsets are invalid.
struct SeqRange {
    int64_t start;
    int64_t len;
};

__device__ __forceinline__ bool seq_range(int s, int T, const int32_t *cu, SeqRange &r) {
    if (cu == nullptr) {
        r.start = (int64_t)s * T;
        r.len = T;
        return true;
    }
    const int32_t a = __ldg(cu + s), b = __ldg(cu + s + 1);
    if (a < 0 || b < a || b > T) {
        r.start = 0;
        r.len = 0;
        return false;
    }
    r.start = a;
    r.len = b - a;
    return true;
}

// ---- host helpers --------------------------------------------------------
inline bool aligned16(const void *p) { return p == nullptr || (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

// Per-device facts, queried once per device and cached (thread-safe).
struct DeviceInfo {
    int ok;           // 1 if the device is sm_103 (GB300 family)
    int sm_count;
    int max_smem_optin;
};
const DeviceInfo &device_info();

// Host-side count of kernel launches made by the library (gla_kernel_launches).
void count_launches(int n);

}  // namespace gla

// Each translation unit that launches kernels defines its own device status
// word with GLA_DEFINE_STATUS(name); gla_last_device_status() collects them.
#define GLA_DEFINE_STATUS(NAME)                                                            \
    static __device__ int g_status_##NAME;                                                 \
    static __device__ __forceinline__ void record_status(int code) {                       \
        atomicCAS(&g_status_##NAME, 0, code);                                              \
    }                                                                                      \
    namespace gla {                                                                        \
    int take_status_##NAME(cudaStream_t st) {                                              \
        int v = 0, zero = 0;                                                               \
        if (cudaMemcpyFromSymbolAsync(&v, g_status_##NAME, sizeof(int), 0,                 \
                                      cudaMemcpyDeviceToHost, st) != cudaSuccess)          \
            return GLA_ERR_LAUNCH;                                                         \
        if (cudaMemcpyToSymbolAsync(g_status_##NAME, &zero, sizeof(int), 0,                \
                                    cudaMemcpyHostToDevice, st) != cudaSuccess)            \
            return GLA_ERR_LAUNCH;                                                         \
        if (cudaStreamSynchronize(st) != cudaSuccess) return GLA_ERR_LAUNCH;               \
        return v;                                                                          \
    }                                                                                      \
    }
