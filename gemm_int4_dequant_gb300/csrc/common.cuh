// common.cuh -- small device/host helpers shared by the library's kernels.
#pragma once

#include <cuda.h>
#include <cudaTypedefs.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "w4.h"

namespace w4 {

// ---------------------------------------------------------------------------
// Host side
// ---------------------------------------------------------------------------

// Number of SMs of the current device (cached per device ordinal).
int sm_count();
// True if the current device is compute capability 10.3 (GB300).
bool device_is_sm103();

// cuTensorMapEncodeTiled, reached through the runtime's driver entry-point
// query (the library does not link the driver API); nullptr if unavailable.
PFN_cuTensorMapEncodeTiled_v12000 tensor_map_encoder();

inline bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

inline w4_status launch_status(cudaError_t e) { return e == cudaSuccess ? W4_OK : W4_ERR_CUDA; }

// Raise a kernel's dynamic shared-memory limit once per device (the call is
// not a stream operation, so it is kept out of the per-launch path and out of
// any stream capture after the first call).  `flags` is per-kernel storage
// with one slot per device ordinal; the slot records the largest size set.
template <typename Kernel>
inline cudaError_t ensure_smem_limit(Kernel k, int bytes, int (&flags)[64]) {
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if (dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
    if (flags[dev] >= bytes) return cudaSuccess;
    e = cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes);
    if (e == cudaSuccess) flags[dev] = bytes;
    return e;
}

// Threads given to each of a CTA's gn row groups when T threads split the
// groups' nb blocks (a thread takes every tpg-th block of its group, thread
// rounds go over the groups T / tpg at a time): T / gn, or one warp per
// group when that is not slower (a warp's lanes then read consecutive
// blocks of the same rows).  1 when there are more groups than threads.
__host__ __device__ inline int threads_per_group(int T, int64_t gn, int64_t nb) {
    if (gn >= T) return 1;
    const int even = static_cast<int>(T / gn);
    auto cost = [&](int tpg) {
        const int64_t per_round = T / tpg;
        return ((gn + per_round - 1) / per_round) * ((nb + tpg - 1) / tpg);
    };
    return (even < 32 && cost(32) <= cost(even)) ? 32 : even;
}

// ---------------------------------------------------------------------------
// Device side
// ---------------------------------------------------------------------------

// 16-byte streaming load of read-only data that is used exactly once: do not
// keep it in L1.
__device__ __forceinline__ uint4 ldg_stream_u4(const void* p) {
    uint4 v;
    asm volatile("ld.global.nc.L1::no_allocate.v4.u32 {%0,%1,%2,%3}, [%4];"
                 : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
                 : "l"(p));
    return v;
}

__device__ __forceinline__ uint32_t ldg_stream_u32(const void* p) {
    uint32_t v;
    asm volatile("ld.global.nc.L1::no_allocate.u32 %0, [%1];" : "=r"(v) : "l"(p));
    return v;
}

template <typename T>
__device__ __forceinline__ float to_f32(T v);
template <>
__device__ __forceinline__ float to_f32<float>(float v) { return v; }
template <>
__device__ __forceinline__ float to_f32<__nv_bfloat16>(__nv_bfloat16 v) { return __bfloat162float(v); }

template <typename T>
__device__ __forceinline__ T from_f32(float v);
template <>
__device__ __forceinline__ float from_f32<float>(float v) { return v; }
template <>
__device__ __forceinline__ __nv_bfloat16 from_f32<__nv_bfloat16>(float v) { return __float2bfloat16_rn(v); }

// bf16 bit pattern -> fp32 (bf16 is the top half of an fp32).
__device__ __forceinline__ float bf16_bits_to_f32(uint32_t bits16) { return __uint_as_float(bits16 << 16); }

}  // namespace w4
