// storage.cuh -- how the kernels read and write the element types a, b and h
// may be stored in.  Arithmetic and every carried value stay fp32: a stored
// element is widened exactly on load, and each fp32 result is rounded once, to
// nearest with ties to even, on store.
#pragma once

#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <stdint.h>

#include "kernels.cuh"

namespace linrec {

template <int DT> struct Storage;

template <> struct Storage<kDtypeF32> {
    using raw = float;
    static constexpr int bytes = 4;
    static __device__ __forceinline__ float get(float x) { return x; }
    static __device__ __forceinline__ float put(float x) { return x; }
};

// bfloat16: the upper 16 bits of the binary32 word of the same value.
template <> struct Storage<kDtypeBF16> {
    using raw = unsigned short;
    static constexpr int bytes = 2;
    static __device__ __forceinline__ float get(unsigned short w) { return __uint_as_float((unsigned int)w << 16); }
    static __device__ __forceinline__ unsigned short put(float x) {
        return __bfloat16_as_ushort(__float2bfloat16_rn(x));
    }
    // Two elements in one 32-bit word (the one at the lower address in the low half):
    // widened exactly, or rounded once each into one word (one instruction per pair).
    static __device__ __forceinline__ float2 get2(uint32_t w) {
        return make_float2(__uint_as_float(w << 16), __uint_as_float(w & 0xffff0000u));
    }
    static __device__ __forceinline__ uint32_t put2(float x, float y) {
        const __nv_bfloat162 v = __floats2bfloat162_rn(x, y);   // x in the low half
        uint32_t w;
        memcpy(&w, &v, sizeof(w));
        return w;
    }
};

// IEEE 754 binary16.
template <> struct Storage<kDtypeF16> {
    using raw = unsigned short;
    static constexpr int bytes = 2;
    static __device__ __forceinline__ float get(unsigned short w) { return __half2float(__ushort_as_half(w)); }
    static __device__ __forceinline__ unsigned short put(float x) { return __half_as_ushort(__float2half_rn(x)); }
    // two elements in one 32-bit word, as for bfloat16
    static __device__ __forceinline__ float2 get2(uint32_t w) {
        __half2 h2;
        static_assert(sizeof(h2) == sizeof(w), "half2 is one word");
        memcpy(&h2, &w, sizeof(w));
        return __half22float2(h2);
    }
    static __device__ __forceinline__ uint32_t put2(float x, float y) {
        const __half2 v = __floats2half2_rn(x, y);               // x in the low half
        uint32_t w;
        memcpy(&w, &v, sizeof(w));
        return w;
    }
};

}  // namespace linrec
