// common.cuh -- small device helpers shared by the KDA kernels.
#pragma once
#include <cstdint>
#include <cuda_runtime.h>
#include <cuda_bf16.h>

namespace kda {

// Status codes mirrored from include/kda.h (device side).
constexpr int kStatusTimeout = -4;
constexpr int kStatusRange = -5;

// Device scratch of the prefill per (sequence, head): its hand-off ring of six
// 82944-byte blocks.
constexpr size_t kPrefillRingBytesPerPair = 6 * 82944;

// Segmented prefill: the int32 index arrays of its runs (segment bounds, start positions,
// roles, owning sequences; the call's own cu_seqlens and start positions), built on the host
// and handed to the setup kernel by value; the split sequences' segment ranges, handed to the
// chain kernel by value; and the role bits of a segment.
constexpr int kSegIdxMax = 512;
constexpr int kSegMaxChains = 32;
constexpr int kSegFirst = 1, kSegLast = 2, kSegMulti = 4;
struct SegChainBuf {
    int n;
    int32_t g0[kSegMaxChains];
    int32_t np[kSegMaxChains];
};
// Blocks per (segment, head) of the segmented prefill's transition bound (partial sums each).
constexpr int kSegBoundBlocks = 64;
struct SegIdxBuf {
    int n;
    int32_t v[kSegIdxMax];
};

// Bounded waits give up after this many nanoseconds (about one second).
constexpr unsigned long long kWaitLimitNs = 1000000000ull;

__device__ __forceinline__ float bf16_bits_to_f32(uint16_t b) {
    return __uint_as_float(static_cast<uint32_t>(b) << 16);
}

// Two packed bf16 values (low half = first element) -> two floats.
__device__ __forceinline__ float2 bf16x2_bits_to_f32(uint32_t w) {
    return make_float2(__uint_as_float(w << 16), __uint_as_float(w & 0xFFFF0000u));
}

__device__ __forceinline__ uint16_t f32_to_bf16_bits(float x) {
    return __bfloat16_as_ushort(__float2bfloat16_rn(x));
}

__device__ __forceinline__ uint32_t f32x2_to_bf16x2_bits(float lo, float hi) {
    __nv_bfloat162 h = __floats2bfloat162_rn(lo, hi);
    return *reinterpret_cast<uint32_t*>(&h);
}

// Two-lane fp32 arithmetic (one instruction, each lane rounded as its scalar form).
__device__ __forceinline__ float2 ffma2(float2 a, float2 b, float2 c) {
    uint64_t d;
    asm("fma.rn.f32x2 %0, %1, %2, %3;"
        : "=l"(d)
        : "l"(*reinterpret_cast<const uint64_t*>(&a)), "l"(*reinterpret_cast<const uint64_t*>(&b)),
          "l"(*reinterpret_cast<const uint64_t*>(&c)));
    return *reinterpret_cast<const float2*>(&d);
}
__device__ __forceinline__ float2 fmul2(float2 a, float2 b) {
    uint64_t d;
    asm("mul.rn.f32x2 %0, %1, %2;"
        : "=l"(d)
        : "l"(*reinterpret_cast<const uint64_t*>(&a)), "l"(*reinterpret_cast<const uint64_t*>(&b)));
    return *reinterpret_cast<const float2*>(&d);
}

// Raise a kernel's dynamic shared-memory limit on the current device, once per device
// (the attribute belongs to the device's copy of the kernel).  `done` holds one flag per
// device ordinal; setting the attribute twice is harmless, so no lock is needed.
constexpr int kMaxDevicesAttr = 64;
inline bool raise_smem_limit(const void* kernel, int bytes, bool (&done)[kMaxDevicesAttr]) {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevicesAttr) return false;
    if (!done[dev]) {
        if (cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes) != cudaSuccess)
            return false;
        done[dev] = true;
    }
    return true;
}

// Record a device-side failure (first writer wins).
__device__ __forceinline__ void set_status(int* status, int code) {
    if (status) atomicCAS(status, 0, code);
}

}  // namespace kda
