// regcarry16.cu -- the register-carry path on 16-bit storage (bfloat16 and
// IEEE binary16).
//
// The same walk as the fp32 register path: one thread owns V adjacent channels
// of one batch index and carries their h through t = 0 .. L-1 in fp32
// registers, with the loads of the next P steps in flight.  V 16-bit elements
// move as one word of 2V bytes (V = 8: one 16-byte load of a and of b per
// step).  Each element is widened on load and each h rounded once on store
// (storage.cuh).  It is the path for pointers not 16-byte aligned and for
// D % 8 != 0, which the chunked path's copies cannot take.
#include "checked.cuh"
#include "kernels.cuh"
#include "storage.cuh"

namespace linrec {

namespace {

template <int V> struct Word;   // V 16-bit elements in one load
template <> struct Word<1> { using type = unsigned short; };
template <> struct Word<2> { using type = unsigned int; };
template <> struct Word<4> { using type = uint2; };
template <> struct Word<8> { using type = uint4; };

template <int V>
__device__ __forceinline__ typename Word<V>::type ld_word(const typename Word<V>::type *p) { return __ldcs(p); }
template <int V>
__device__ __forceinline__ void st_word(typename Word<V>::type *p, typename Word<V>::type w) { __stcs(p, w); }

// A thread's V elements of one step: widened, and h rounded back.
template <int DT, int V>
__device__ __forceinline__ void widen(const typename Word<V>::type &w, float (&x)[V]) {
    if constexpr (V == 1) {
        x[0] = Storage<DT>::get(w);
    } else {
        uint32_t u[V / 2];
        memcpy(u, &w, sizeof(u));
#pragma unroll
        for (int i = 0; i < V / 2; ++i) {
            const float2 f = Storage<DT>::get2(u[i]);
            x[2 * i] = f.x;
            x[2 * i + 1] = f.y;
        }
    }
}
template <int DT, int V>
__device__ __forceinline__ typename Word<V>::type narrow(const float (&x)[V]) {
    typename Word<V>::type w;
    if constexpr (V == 1) {
        w = Storage<DT>::put(x[0]);
    } else {
        uint32_t u[V / 2];
#pragma unroll
        for (int i = 0; i < V / 2; ++i) u[i] = Storage<DT>::put2(x[2 * i], x[2 * i + 1]);
        memcpy(&w, u, sizeof(u));
    }
    return w;
}

template <int DT, int V, int P>
__global__ void __launch_bounds__(256)
regcarry16_kernel(const unsigned short *__restrict__ a, const unsigned short *__restrict__ b,
                  unsigned short *__restrict__ h, const long long L, const long long D,
                  const long long groups_per_batch, const long long n_groups, const float *h_init, float *h_last)
{
    using W = typename Word<V>::type;
    const long long g = (long long)blockIdx.x * blockDim.x + threadIdx.x;
    if (g >= n_groups) return;
    const long long bi = g / groups_per_batch;
    const long long dch = (g - bi * groups_per_batch) * V;   // first channel of this thread
    const long long off = bi * L * D + dch;
    const W *pa = reinterpret_cast<const W *>(a + off);
    const W *pb = reinterpret_cast<const W *>(b + off);
    W *ph = reinterpret_cast<W *>(h + off);
    const long long stride = D / V;           // one time step, in words
    // extents for the index-checked build: elements of a, b, h, and of h_init / h_last
    const long long n_all = (n_groups / groups_per_batch) * L * D;
    const long long n_state = (n_groups / groups_per_batch) * D;
    auto ld = [&](const W *p, const unsigned short *base) -> W {
#ifdef LINREC_DEBUG
        if (!inside(p, base, n_all)) {
            W w;
            memset(&w, 0, sizeof(W));
            return w;
        }
#endif
        return ld_word<V>(p);
    };

    W ra[P], rb[P];
#pragma unroll
    for (int j = 0; j < P; ++j) {
        if (j < L) {
            ra[j] = ld(pa + j * stride, a);
            rb[j] = ld(pb + j * stride, b);
        }
    }
    float hv[V];
#pragma unroll
    for (int v = 0; v < V; ++v)
        hv[v] = (h_init && inside(h_init + bi * D + dch + v, h_init, n_state)) ? h_init[bi * D + dch + v] : 0.0f;
    if (!h_init) memset(&ra[0], 0, sizeof(W));   // h_{-1} = 0 and a_0 is never used: its word := +0
    for (long long t0 = 0; t0 < L; t0 += P) {
#pragma unroll
        for (int j = 0; j < P; ++j) {
            const long long t = t0 + j;
            if (t < L) {
                float xa[V], xb[V];
                widen<DT, V>(ra[j], xa);
                widen<DT, V>(rb[j], xb);
#pragma unroll
                for (int v = 0; v < V; ++v) hv[v] = fmaf(xa[v], hv[v], xb[v]);
                if (inside(ph + t * stride, h, n_all, true)) st_word<V>(ph + t * stride, narrow<DT, V>(hv));
                const long long tn = t + P;
                if (tn < L) {
                    ra[j] = ld(pa + tn * stride, a);
                    rb[j] = ld(pb + tn * stride, b);
                }
            }
        }
    }
    if (h_last) {
#pragma unroll
        for (int v = 0; v < V; ++v)
            if (inside(h_last + bi * D + dch + v, h_last, n_state, true)) h_last[bi * D + dch + v] = hv[v];
    }
}

template <int DT, int V, int P>
cudaError_t launch_one(int threads, const void *a, const void *b, void *h, int64_t B, int64_t L, int64_t D,
                       const float *h_init, float *h_last, cudaStream_t stream) {
    const long long gpb = D / V;
    const long long n = B * gpb;
    const long long blocks = (n + threads - 1) / threads;
    regcarry16_kernel<DT, V, P><<<(unsigned)blocks, threads, 0, stream>>>(
        static_cast<const unsigned short *>(a), static_cast<const unsigned short *>(b),
        static_cast<unsigned short *>(h), L, D, gpb, n, h_init, h_last);
    return cudaGetLastError();
}

template <int DT>
cudaError_t launch_dt(int vec, int prefetch, int threads, const void *a, const void *b, void *h, int64_t B,
                      int64_t L, int64_t D, const float *h_init, float *h_last, cudaStream_t stream) {
#define LINREC_R16(V, P)                                                                          \
    if (vec == V && prefetch == P) return launch_one<DT, V, P>(threads, a, b, h, B, L, D, h_init, h_last, stream);
    LINREC_R16(8, 4) LINREC_R16(8, 8) LINREC_R16(8, 16)
    LINREC_R16(4, 4) LINREC_R16(4, 8) LINREC_R16(4, 16)
    LINREC_R16(2, 4) LINREC_R16(2, 8) LINREC_R16(2, 16)
    LINREC_R16(1, 4) LINREC_R16(1, 8) LINREC_R16(1, 16)
#undef LINREC_R16
    return cudaErrorInvalidValue;
}

}  // namespace

bool regcarry16_supported(int vec, int prefetch) {
    return (vec == 1 || vec == 2 || vec == 4 || vec == 8) && (prefetch == 4 || prefetch == 8 || prefetch == 16);
}

cudaError_t launch_regcarry16(int dtype, int vec, int prefetch, int threads, const void *a, const void *b, void *h,
                              int64_t B, int64_t L, int64_t D, const float *h_init, float *h_last,
                              cudaStream_t stream) {
    if (dtype == kDtypeBF16)
        return launch_dt<kDtypeBF16>(vec, prefetch, threads, a, b, h, B, L, D, h_init, h_last, stream);
    if (dtype == kDtypeF16)
        return launch_dt<kDtypeF16>(vec, prefetch, threads, a, b, h, B, L, D, h_init, h_last, stream);
    return cudaErrorInvalidValue;
}

LINREC_CHECKED_REPORT(checked_report_regcarry16)

}  // namespace linrec
