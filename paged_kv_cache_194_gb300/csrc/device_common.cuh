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

// Pool encoding of new K/V rows, shared by the append kernel and the fused
// append of the tensor-core attention kernel (so both write the same bytes).
// AppendChunk<pool, input>: kIn 16-byte input chunks -> one 16-byte chunk of
// pool elements; run() loads them from `src`, convert() takes them from
// registers.
__device__ __forceinline__ uint32_t pack_bf16x2_rn(float lo, float hi) {
    return static_cast<uint32_t>(__bfloat16_as_ushort(__float2bfloat16_rn(lo))) |
           (static_cast<uint32_t>(__bfloat16_as_ushort(__float2bfloat16_rn(hi))) << 16);
}

// 4 inputs -> 4 E4M3 codes: e4m3_rn_satfinite(fp32(x) * inv_scale).
__device__ __forceinline__ uint32_t quant4(float a, float b, float c, float d, float inv) {
    const __nv_fp8x2_storage_t lo =
        __nv_cvt_float2_to_fp8x2(make_float2(__fmul_rn(a, inv), __fmul_rn(b, inv)), __NV_SATFINITE, __NV_E4M3);
    const __nv_fp8x2_storage_t hi =
        __nv_cvt_float2_to_fp8x2(make_float2(__fmul_rn(c, inv), __fmul_rn(d, inv)), __NV_SATFINITE, __NV_E4M3);
    return static_cast<uint32_t>(lo) | (static_cast<uint32_t>(hi) << 16);
}

template <int PDT, int IDT>
struct AppendChunk;

template <>
struct AppendChunk<PKV_F32, PKV_F32> {  // 4 floats
    static constexpr int kIn = 1;
    __device__ static uint4 convert(const uint4* x, float) { return x[0]; }
};
template <>
struct AppendChunk<PKV_BF16, PKV_BF16> {  // 8 bf16
    static constexpr int kIn = 1;
    __device__ static uint4 convert(const uint4* x, float) { return x[0]; }
};
template <>
struct AppendChunk<PKV_BF16, PKV_F32> {  // 8 floats -> 8 bf16 (RN)
    static constexpr int kIn = 2;
    __device__ static uint4 convert(const uint4* x, float) {
        return make_uint4(pack_bf16x2_rn(__uint_as_float(x[0].x), __uint_as_float(x[0].y)),
                          pack_bf16x2_rn(__uint_as_float(x[0].z), __uint_as_float(x[0].w)),
                          pack_bf16x2_rn(__uint_as_float(x[1].x), __uint_as_float(x[1].y)),
                          pack_bf16x2_rn(__uint_as_float(x[1].z), __uint_as_float(x[1].w)));
    }
};
template <>
struct AppendChunk<PKV_FP8_E4M3, PKV_F32> {  // 16 floats -> 16 E4M3
    static constexpr int kIn = 4;
    __device__ static uint4 convert(const uint4* x, float inv) {
        uint32_t w[4];
#pragma unroll
        for (int i = 0; i < 4; ++i)
            w[i] = quant4(__uint_as_float(x[i].x), __uint_as_float(x[i].y), __uint_as_float(x[i].z),
                          __uint_as_float(x[i].w), inv);
        return make_uint4(w[0], w[1], w[2], w[3]);
    }
};
template <>
struct AppendChunk<PKV_FP8_E4M3, PKV_BF16> {  // 16 bf16 -> 16 E4M3
    static constexpr int kIn = 2;
    __device__ static uint4 convert(const uint4* x, float inv) {
        const uint32_t in[8] = {x[0].x, x[0].y, x[0].z, x[0].w, x[1].x, x[1].y, x[1].z, x[1].w};
        uint32_t w[4];
#pragma unroll
        for (int i = 0; i < 4; ++i)
            w[i] = quant4(bf16_lo(in[2 * i]), bf16_hi(in[2 * i]), bf16_lo(in[2 * i + 1]),
                          bf16_hi(in[2 * i + 1]), inv);
        return make_uint4(w[0], w[1], w[2], w[3]);
    }
};

// Load the kIn input chunks at src and convert them.
template <int PDT, int IDT>
__device__ __forceinline__ uint4 append_chunk(const uint8_t* src, float inv) {
    uint4 x[AppendChunk<PDT, IDT>::kIn];
#pragma unroll
    for (int i = 0; i < AppendChunk<PDT, IDT>::kIn; ++i) x[i] = reinterpret_cast<const uint4*>(src)[i];
    return AppendChunk<PDT, IDT>::convert(x, inv);
}

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
