// checked.cuh -- the index-checked build.  Compiled with -DLINREC_DEBUG, every
// plain global load and store of the kernels first tests that the bytes it
// touches lie inside the array they belong to; an access outside is skipped (a
// load then yields zeros) and recorded: a count and the byte offset of the first
// one, per translation unit, read and cleared by linrec_debug_bad_accesses().
// TMA box copies need no test: the copy engine clips them to the tensor.  In the
// normal build inside() is the constant true and every test compiles away.
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

namespace linrec {

#ifdef LINREC_DEBUG
namespace {
__device__ unsigned long long g_bad_count;   // accesses skipped in this translation unit
__device__ long long g_bad_first = -1;       // byte offset of the first one from its array's start
__device__ long long g_out_cap;              // tests: > 0 makes every output array end at this byte
}  // namespace

// Whether the `width` bytes at p lie inside the n_elems elements at base (an output
// array is cut at g_out_cap bytes when that is set).
template <typename P, typename Q>
__device__ __forceinline__ bool inside(const P *p, const Q *base, long long n_elems, bool output = false,
                                       long long width = (long long)sizeof(P)) {
    long long bytes = n_elems * (long long)sizeof(Q);
    if (output && g_out_cap > 0 && bytes > g_out_cap) bytes = g_out_cap;
    const long long off = (long long)(reinterpret_cast<const char *>(p) - reinterpret_cast<const char *>(base));
    if (off >= 0 && off + width <= bytes) return true;
    if (atomicAdd(&g_bad_count, 1ull) == 0ull) g_bad_first = off;
    return false;
}

// Host side, one per translation unit with kernels: read and clear its record and set
// the output cap (0 removes it).  Synchronises the device.
#define LINREC_CHECKED_REPORT(NAME)                                                               \
    cudaError_t NAME(unsigned long long *count, long long *first, long long out_cap) {            \
        const unsigned long long zero = 0ull;                                                     \
        const long long none = -1;                                                                \
        cudaError_t e = cudaMemcpyFromSymbol(count, g_bad_count, sizeof(*count));                 \
        if (e == cudaSuccess) e = cudaMemcpyFromSymbol(first, g_bad_first, sizeof(*first));       \
        if (e == cudaSuccess) e = cudaMemcpyToSymbol(g_bad_count, &zero, sizeof(zero));           \
        if (e == cudaSuccess) e = cudaMemcpyToSymbol(g_bad_first, &none, sizeof(none));           \
        if (e == cudaSuccess) e = cudaMemcpyToSymbol(g_out_cap, &out_cap, sizeof(out_cap));       \
        return e;                                                                                 \
    }
#else
template <typename P, typename Q>
__device__ __forceinline__ constexpr bool inside(const P *, const Q *, long long, bool = false,
                                                 long long = 0) {
    return true;
}
#define LINREC_CHECKED_REPORT(NAME)                                                               \
    cudaError_t NAME(unsigned long long *count, long long *first, long long) {                    \
        *count = 0ull;                                                                            \
        *first = -1;                                                                              \
        return cudaSuccess;                                                                       \
    }
#endif

}  // namespace linrec
