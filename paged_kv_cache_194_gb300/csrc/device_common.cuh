// Device helpers shared by the decode kernels: async copies, element
// conversions, warp reductions and the sequence-length clamp.
#pragma once

#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_fp8.h>

#include <cstdint>

#include "pkv_internal.h"

namespace pkv {

// 16-byte global->shared copy that bypasses L1; src_bytes = 0 zero-fills.
__device__ __forceinline__ void cp_async16(void* smem, const void* gmem, int src_bytes) {
    unsigned s = static_cast<unsigned>(__cvta_generic_to_shared(smem));
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;\n" ::"r"(s), "l"(gmem),
                 "r"(src_bytes)
                 : "memory");
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;\n" ::: "memory"); }
template <int N>
__device__ __forceinline__ void cp_async_wait() {
    asm volatile("cp.async.wait_group %0;\n" ::"n"(N) : "memory");
}

// bfloat16 is the upper half of a binary32 word.
__device__ __forceinline__ float bf16_lo(uint32_t w) { return __uint_as_float(w << 16); }
__device__ __forceinline__ float bf16_hi(uint32_t w) { return __uint_as_float(w & 0xFFFF0000u); }

__device__ __forceinline__ float2 e4m3x2_to_float2(uint16_t two) {
    __half2_raw hr = __nv_cvt_fp8x2_to_halfraw2(static_cast<__nv_fp8x2_storage_t>(two), __NV_E4M3);
    __half2 h;
    h = *reinterpret_cast<__half2*>(&hr);
    return __half22float2(h);
}

// Storage traits: elements per 16-byte chunk and chunk -> floats.
template <int DT>
struct KvTraits;

template <>
struct KvTraits<PKV_F32> {
    static constexpr int kBytes = 4;
    static constexpr int kPerChunk = 4;
    __device__ __forceinline__ static void to_float(const uint4& c, float* f) {
        f[0] = __uint_as_float(c.x);
        f[1] = __uint_as_float(c.y);
        f[2] = __uint_as_float(c.z);
        f[3] = __uint_as_float(c.w);
    }
};

template <>
struct KvTraits<PKV_BF16> {
    static constexpr int kBytes = 2;
    static constexpr int kPerChunk = 8;
    __device__ __forceinline__ static void to_float(const uint4& c, float* f) {
        const uint32_t w[4] = {c.x, c.y, c.z, c.w};
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            f[2 * i] = bf16_lo(w[i]);
            f[2 * i + 1] = bf16_hi(w[i]);
        }
    }
};

template <>
struct KvTraits<PKV_FP8_E4M3> {
    static constexpr int kBytes = 1;
    static constexpr int kPerChunk = 16;
    __device__ __forceinline__ static void to_float(const uint4& c, float* f) {
        const uint32_t w[4] = {c.x, c.y, c.z, c.w};
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            float2 a = e4m3x2_to_float2(static_cast<uint16_t>(w[i] & 0xFFFFu));
            float2 b = e4m3x2_to_float2(static_cast<uint16_t>(w[i] >> 16));
            f[4 * i] = a.x;
            f[4 * i + 1] = a.y;
            f[4 * i + 2] = b.x;
            f[4 * i + 3] = b.y;
        }
    }
};

__device__ __forceinline__ float warp_max(float v) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v = fmaxf(v, __shfl_xor_sync(0xFFFFFFFFu, v, o));
    return v;
}
__device__ __forceinline__ float warp_sum(float v) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xFFFFFFFFu, v, o);
    return v;
}

// Length a decode kernel uses for sequence b: the device value clamped to
// [0, max_len] (max_len <= max_blocks * block_size is checked on the host);
// out-of-range values are flagged once (by the caller passing report = true).
__device__ __forceinline__ int clamped_len(const DecodeArgs& a, int b, bool report) {
    int L = a.lens[b];
    const int cap = a.max_len;
    if (L < 0 || L > cap) {
        if (report && a.err) atomicOr(a.err, PKV_ERRBIT_SEQ_LEN);
        L = L < 0 ? 0 : cap;
    }
    return L;
}

// Tokens a launch may read for sequence b: the clamped length minus the
// positions after this launch's last query.
__device__ __forceinline__ int visible_len(const DecodeArgs& a, int b, bool report) {
    const int L = clamped_len(a, b, report) - a.len_trim;
    return L > 0 ? L : 0;
}

template <typename QT>
__device__ __forceinline__ float load_q(const QT* p);
template <>
__device__ __forceinline__ float load_q<float>(const float* p) { return *p; }
template <>
__device__ __forceinline__ float load_q<__nv_bfloat16>(const __nv_bfloat16* p) {
    return __bfloat162float(*p);
}

template <typename QT>
__device__ __forceinline__ QT to_out(float x);
template <>
__device__ __forceinline__ float to_out<float>(float x) { return x; }
template <>
__device__ __forceinline__ __nv_bfloat16 to_out<__nv_bfloat16>(float x) {
    return __float2bfloat16_rn(x);
}

}  // namespace pkv
