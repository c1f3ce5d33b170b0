// storage.cuh -- how the kernels read and write the element types a, b and h
// may be stored in.  Arithmetic and every carried value stay fp32: a stored
// element is widened exactly on load, and each fp32 result is rounded once, to
// nearest with ties to even, on store.
#pragma once

#include <cuda_bf16.h>
#include <cuda_fp16.h>

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
};

// IEEE 754 binary16.
template <> struct Storage<kDtypeF16> {
    using raw = unsigned short;
    static constexpr int bytes = 2;
    static __device__ __forceinline__ float get(unsigned short w) { return __half2float(__ushort_as_half(w)); }
    static __device__ __forceinline__ unsigned short put(float x) { return __half_as_ushort(__float2half_rn(x)); }
};

}  // namespace linrec
