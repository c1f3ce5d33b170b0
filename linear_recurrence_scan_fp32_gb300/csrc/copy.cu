// copy.cu -- dst = src with 16-byte vector loads and stores, grid-stride.
// Not part of the scan: it measures, in the same process, the copy bandwidth
// that bounds any kernel that reads and writes each byte once.
#include "kernels.cuh"

namespace linrec {

namespace {

__global__ void __launch_bounds__(256)
copy_vec4_kernel(const float4 *__restrict__ src, float4 *__restrict__ dst, long long n4) {
    const long long stride = (long long)gridDim.x * blockDim.x;
    for (long long i = (long long)blockIdx.x * blockDim.x + threadIdx.x; i < n4; i += stride)
        __stcs(dst + i, __ldcs(src + i));
}

__global__ void __launch_bounds__(256)
copy_scalar_kernel(const float *__restrict__ src, float *__restrict__ dst, long long n) {
    const long long stride = (long long)gridDim.x * blockDim.x;
    for (long long i = (long long)blockIdx.x * blockDim.x + threadIdx.x; i < n; i += stride)
        dst[i] = src[i];
}

}  // namespace

cudaError_t launch_copy(const float *src, float *dst, int64_t n, int sm_count, cudaStream_t stream) {
    const bool vec = ((reinterpret_cast<uintptr_t>(src) | reinterpret_cast<uintptr_t>(dst)) & 15u) == 0;
    const long long blocks = (long long)sm_count * 8;
    if (vec) {
        const long long n4 = n / 4;
        if (n4 > 0)
            copy_vec4_kernel<<<(unsigned)blocks, 256, 0, stream>>>(
                reinterpret_cast<const float4 *>(src), reinterpret_cast<float4 *>(dst), n4);
        if (n - n4 * 4 > 0)
            copy_scalar_kernel<<<1, 32, 0, stream>>>(src + n4 * 4, dst + n4 * 4, n - n4 * 4);
    } else {
        copy_scalar_kernel<<<(unsigned)blocks, 256, 0, stream>>>(src, dst, n);
    }
    return cudaGetLastError();
}

}  // namespace linrec
