// regcarry.cu -- the register-carry path of the linear-recurrence scan.
//
// h_0 = b_0, h_t = a_t*h_{t-1} + b_t per channel (POPCORNBENCH "Kimi-K2.6 l1_p9",
// problem statement).  One thread owns V adjacent channels of one batch index
// (V = 4: one 16-byte load of a and of b per step; a warp covers 32*V
// consecutive floats of a row, so every access is coalesced along D) and walks
// t = 0 .. L-1 with h in registers.  Only the FMA chain is serial: the loads of
// a_t, b_t do not depend on h, so the loads of the next P steps are kept in
// flight in a register ring, which is what keeps HBM busy when the number of
// channels alone does not.
#include "checked.cuh"
#include "kernels.cuh"

namespace linrec {

namespace {

template <int V> struct VecT;
template <> struct VecT<1> { using type = float; };
template <> struct VecT<2> { using type = float2; };
template <> struct VecT<4> { using type = float4; };

__device__ __forceinline__ float ld_stream(const float *p) { return __ldcs(p); }
__device__ __forceinline__ float2 ld_stream(const float2 *p) { return __ldcs(p); }
__device__ __forceinline__ float4 ld_stream(const float4 *p) { return __ldcs(p); }
__device__ __forceinline__ void st_stream(float *p, float v) { __stcs(p, v); }
__device__ __forceinline__ void st_stream(float2 *p, float2 v) { __stcs(p, v); }
__device__ __forceinline__ void st_stream(float4 *p, float4 v) { __stcs(p, v); }

__device__ __forceinline__ float step(float a, float h, float b) { return fmaf(a, h, b); }
__device__ __forceinline__ float2 step(float2 a, float2 h, float2 b) {
    return make_float2(fmaf(a.x, h.x, b.x), fmaf(a.y, h.y, b.y));
}
__device__ __forceinline__ float4 step(float4 a, float4 h, float4 b) {
    return make_float4(fmaf(a.x, h.x, b.x), fmaf(a.y, h.y, b.y), fmaf(a.z, h.z, b.z), fmaf(a.w, h.w, b.w));
}
__device__ __forceinline__ void zero(float &v) { v = 0.0f; }
__device__ __forceinline__ void zero(float2 &v) { v = make_float2(0.0f, 0.0f); }
__device__ __forceinline__ void zero(float4 &v) { v = make_float4(0.0f, 0.0f, 0.0f, 0.0f); }

template <int V, int P>
__global__ void __launch_bounds__(256)
regcarry_kernel(const float *__restrict__ a, const float *__restrict__ b, float *__restrict__ h,
                const long long L, const long long D, const long long groups_per_batch,
                const long long n_groups, const float *h_init, float *h_last)
{
    using vec = typename VecT<V>::type;
    const long long g = (long long)blockIdx.x * blockDim.x + threadIdx.x;
    if (g >= n_groups) return;
    const long long bi = g / groups_per_batch;
    const long long dch = (g - bi * groups_per_batch) * V;   // first channel of this thread
    const long long off = bi * L * D + dch;
    const vec *pa = reinterpret_cast<const vec *>(a + off);
    const vec *pb = reinterpret_cast<const vec *>(b + off);
    vec *ph = reinterpret_cast<vec *>(h + off);
    const long long stride = D / V;           // one time step, in vectors
    // extents for the index-checked build: elements of a, b, h, and of h_init / h_last
    const long long n_all = (n_groups / groups_per_batch) * L * D;
    const long long n_state = (n_groups / groups_per_batch) * D;
    auto ld = [&](const vec *p, const float *base) -> vec {
#ifdef LINREC_DEBUG
        if (!inside(p, base, n_all)) {
            vec v;
            zero(v);
            return v;
        }
#endif
        return ld_stream(p);
    };

    vec ra[P], rb[P];
#pragma unroll
    for (int j = 0; j < P; ++j) {
        if (j < L) {
            ra[j] = ld(pa + j * stride, a);
            rb[j] = ld(pb + j * stride, b);
        }
    }
    vec hv;
    zero(hv);
    if (h_init) {                             // continue from the given state: a_0 is used
        float *hvs = reinterpret_cast<float *>(&hv);
#pragma unroll
        for (int v = 0; v < V; ++v) {
            const float *src = h_init + bi * D + dch + v;
            hvs[v] = inside(src, h_init, n_state) ? *src : 0.0f;
        }
    } else {
        zero(ra[0]);                          // h_{-1} = 0 and a_0 is never used
    }
    for (long long t0 = 0; t0 < L; t0 += P) {
#pragma unroll
        for (int j = 0; j < P; ++j) {
            const long long t = t0 + j;
            if (t < L) {
                hv = step(ra[j], hv, rb[j]);
                if (inside(ph + t * stride, h, n_all, true)) st_stream(ph + t * stride, hv);
                const long long tn = t + P;
                if (tn < L) {
                    ra[j] = ld(pa + tn * stride, a);
                    rb[j] = ld(pb + tn * stride, b);
                }
            }
        }
    }
    if (h_last) {
        const float *hvs = reinterpret_cast<const float *>(&hv);
#pragma unroll
        for (int v = 0; v < V; ++v) {
            float *dst = h_last + bi * D + dch + v;
            if (inside(dst, h_last, n_state, true)) *dst = hvs[v];
        }
    }
}

template <int V, int P>
cudaError_t launch_one(int threads, const float *a, const float *b, float *h, int64_t B, int64_t L,
                       int64_t D, const float *h_init, float *h_last, cudaStream_t stream) {
    const long long gpb = D / V;
    const long long n = B * gpb;
    const long long blocks = (n + threads - 1) / threads;
    regcarry_kernel<V, P><<<(unsigned)blocks, threads, 0, stream>>>(a, b, h, L, D, gpb, n, h_init, h_last);
    return cudaGetLastError();
}

template <typename T, int V> __device__ __forceinline__ float &lane_of(T &v, int i) {
    return reinterpret_cast<float *>(&v)[i];
}

// Segmented form, for few channels and long sequences: thread (seg, g) owns channel
// group g over the steps [seg * seg_len, (seg + 1) * seg_len).  Two launches.
//  reduce: compose the segment's maps into (A, B) per channel -> aggA / aggB [seg][channel];
//  apply:  fold the maps of segments 0 .. seg-1 over the state before the sequence (h_init
//          or 0), in order, into the h entering the segment; replay the segment from it.
// The first step's slope is dropped without a carried-in state, as in the one-pass kernel.
template <int V, int P, bool APPLY>
__global__ void __launch_bounds__(256)
regcarry_seg_kernel(const float *__restrict__ a, const float *__restrict__ b, float *__restrict__ h,
                    const long long L, const long long D, const long long groups_per_batch,
                    const long long n_groups, const long long seg_len, const long long nseg,
                    const float *h_init, float *h_last, float *__restrict__ aggA, float *__restrict__ aggB)
{
    using vec = typename VecT<V>::type;
    const long long tid = (long long)blockIdx.x * blockDim.x + threadIdx.x;
    if (tid >= n_groups * nseg) return;
    const long long seg = tid / n_groups;     // consecutive threads: consecutive channel groups
    const long long g = tid - seg * n_groups;
    const long long bi = g / groups_per_batch;
    const long long dch = (g - bi * groups_per_batch) * V;
    const long long n_ch = n_groups * V;      // channels, B * D
    const long long ch0 = bi * D + dch;       // this thread's first channel, as an index of (B, D)
    const long long t_begin = seg * seg_len;
    const long long t_end = (t_begin + seg_len < L) ? t_begin + seg_len : L;
    const long long off = bi * L * D + dch;
    const vec *pa = reinterpret_cast<const vec *>(a + off);
    const vec *pb = reinterpret_cast<const vec *>(b + off);
    vec *ph = reinterpret_cast<vec *>(h + off);
    const long long stride = D / V;
    // extents for the index-checked build
    const long long n_all = (n_groups / groups_per_batch) * L * D;
    const long long n_state = n_ch, n_agg = nseg * n_ch;
    auto ld = [&](const vec *p, const float *base) -> vec {
#ifdef LINREC_DEBUG
        if (!inside(p, base, n_all)) {
            vec v;
            zero(v);
            return v;
        }
#endif
        return ld_stream(p);
    };

    vec ra[P], rb[P];
#pragma unroll
    for (int j = 0; j < P; ++j) {
        if (t_begin + j < t_end) {
            ra[j] = ld(pa + (t_begin + j) * stride, a);
            rb[j] = ld(pb + (t_begin + j) * stride, b);
        }
    }
    if (seg == 0 && !h_init) zero(ra[0]);     // h_{-1} = 0 and a_0 is never used

    vec hv, Av;                                // apply: running h; reduce: (Av, hv) is the composed map
    zero(hv);
#pragma unroll
    for (int v = 0; v < V; ++v) lane_of<vec, V>(Av, v) = 1.0f;
    if (APPLY) {
        // the h entering the segment: the state before the sequence, then every earlier segment's map
#pragma unroll
        for (int v = 0; v < V; ++v) {
            float c = (h_init && inside(h_init + ch0 + v, h_init, n_state)) ? h_init[ch0 + v] : 0.0f;
            for (long long j = 0; j < seg; ++j) {
                const long long w = j * n_ch + ch0 + v;
                if (inside(aggA + w, aggA, n_agg) && inside(aggB + w, aggB, n_agg)) c = fmaf(aggA[w], c, aggB[w]);
            }
            lane_of<vec, V>(hv, v) = c;
        }
    }
    for (long long t0 = t_begin; t0 < t_end; t0 += P) {
#pragma unroll
        for (int j = 0; j < P; ++j) {
            const long long t = t0 + j;
            if (t < t_end) {
                hv = step(ra[j], hv, rb[j]);
                if (APPLY) {
                    if (inside(ph + t * stride, h, n_all, true)) st_stream(ph + t * stride, hv);
                } else {
#pragma unroll
                    for (int v = 0; v < V; ++v) lane_of<vec, V>(Av, v) *= lane_of<vec, V>(ra[j], v);
                }
                const long long tn = t + P;
                if (tn < t_end) {
                    ra[j] = ld(pa + tn * stride, a);
                    rb[j] = ld(pb + tn * stride, b);
                }
            }
        }
    }
    if (!APPLY) {
#pragma unroll
        for (int v = 0; v < V; ++v) {
            const long long w = seg * n_ch + ch0 + v;
            if (inside(aggA + w, aggA, n_agg)) aggA[w] = lane_of<vec, V>(Av, v);
            if (inside(aggB + w, aggB, n_agg)) aggB[w] = lane_of<vec, V>(hv, v);
        }
    } else if (h_last && t_end == L) {
#pragma unroll
        for (int v = 0; v < V; ++v)
            if (inside(h_last + ch0 + v, h_last, n_state, true)) h_last[ch0 + v] = lane_of<vec, V>(hv, v);
    }
}

template <int V>
cudaError_t launch_seg_one(int threads, const float *a, const float *b, float *h, int64_t B, int64_t L, int64_t D,
                           int64_t nseg, const float *h_init, float *h_last, float *aggA, float *aggB,
                           cudaStream_t stream) {
    const long long gpb = D / V;
    const long long n = B * gpb;
    const long long seg_len = (L + nseg - 1) / nseg;
    const long long blocks = (n * nseg + threads - 1) / threads;
    regcarry_seg_kernel<V, 8, false><<<(unsigned)blocks, threads, 0, stream>>>(a, b, h, L, D, gpb, n, seg_len, nseg,
                                                                                h_init, h_last, aggA, aggB);
    cudaError_t err = cudaGetLastError();
    if (err != cudaSuccess) return err;
    regcarry_seg_kernel<V, 8, true><<<(unsigned)blocks, threads, 0, stream>>>(a, b, h, L, D, gpb, n, seg_len, nseg,
                                                                               h_init, h_last, aggA, aggB);
    return cudaGetLastError();
}

// Gradient, right to left: c_t = a_{t+1} c_{t+1} + g_t; db_t = c_t; da_t = c_t h_{t-1}.
// The ring holds (g_t, a_{t+1}, h_{t-1}) for the next P steps down.
template <int V, int P>
__global__ void __launch_bounds__(256)
regcarry_backward_kernel(const float *__restrict__ a, const float *__restrict__ h, const float *__restrict__ g,
                         float *__restrict__ da, float *__restrict__ db, const long long L, const long long D,
                         const long long groups_per_batch, const long long n_groups, const float *h_init,
                         const float *dh_last, float *dh_init)
{
    using vec = typename VecT<V>::type;
    const long long gi = (long long)blockIdx.x * blockDim.x + threadIdx.x;
    if (gi >= n_groups) return;
    const long long bi = gi / groups_per_batch;
    const long long dch = (gi - bi * groups_per_batch) * V;
    const long long off = bi * L * D + dch;
    const vec *pa = reinterpret_cast<const vec *>(a + off);
    const vec *ph = reinterpret_cast<const vec *>(h + off);
    const vec *pg = reinterpret_cast<const vec *>(g + off);
    vec *pda = reinterpret_cast<vec *>(da + off);
    vec *pdb = reinterpret_cast<vec *>(db + off);
    const long long stride = D / V;
    const bool want_da = da != nullptr;
    vec one, zv;
    zero(zv);
#pragma unroll
    for (int v = 0; v < V; ++v) lane_of<vec, V>(one, v) = 1.0f;

    // extents for the index-checked build: elements of a, h, g, da, db, and of the (B, D) states
    const long long n_all = (n_groups / groups_per_batch) * L * D;
    const long long n_state = (n_groups / groups_per_batch) * D;
    auto ld = [&](const vec *p, const float *base) { return inside(p, base, n_all) ? ld_stream(p) : zv; };
    auto load = [&](long long t, vec &rg, vec &ra, vec &rh) {
        rg = ld(pg + t * stride, g);
        ra = (t + 1 < L) ? ld(pa + (t + 1) * stride, a) : one;   // the carry enters row L-1 whole
        rh = (want_da && t >= 1) ? ld(ph + (t - 1) * stride, h) : zv;
    };
    vec rg[P], ra[P], rh[P];
#pragma unroll
    for (int j = 0; j < P; ++j)
        if (L - 1 - j >= 0) load(L - 1 - j, rg[j], ra[j], rh[j]);
    vec cv;
    zero(cv);
    if (dh_last) {
#pragma unroll
        for (int v = 0; v < V; ++v) {
            const float *src = dh_last + bi * D + dch + v;
            lane_of<vec, V>(cv, v) = inside(src, dh_last, n_state) ? *src : 0.0f;
        }
    }
    for (long long t0 = 0; t0 < L; t0 += P) {
#pragma unroll
        for (int j = 0; j < P; ++j) {
            const long long t = L - 1 - (t0 + j);
            if (t >= 0) {
                cv = step(ra[j], cv, rg[j]);
                if (inside(pdb + t * stride, db, n_all, true)) st_stream(pdb + t * stride, cv);
                if (want_da) {
                    vec hp = rh[j];
                    if (t == 0) {
#pragma unroll
                        for (int v = 0; v < V; ++v) {
                            const float *src = h_init + bi * D + dch + v;
                            lane_of<vec, V>(hp, v) = (h_init && inside(src, h_init, n_state)) ? *src : 0.0f;
                        }
                    }
                    vec out;
#pragma unroll
                    for (int v = 0; v < V; ++v) lane_of<vec, V>(out, v) = lane_of<vec, V>(cv, v) * lane_of<vec, V>(hp, v);
                    if (inside(pda + t * stride, da, n_all, true)) st_stream(pda + t * stride, out);
                }
                if (t == 0 && dh_init) {
#pragma unroll
                    for (int v = 0; v < V; ++v) {
                        float *dst = dh_init + bi * D + dch + v;
                        if (inside(dst, dh_init, n_state, true) && inside(a + off + v, a, n_all))
                            *dst = a[off + v] * lane_of<vec, V>(cv, v);
                    }
                }
                const long long tn = t - P;
                if (tn >= 0) load(tn, rg[j], ra[j], rh[j]);
            }
        }
    }
}

template <int V>
cudaError_t launch_back_one(int threads, const float *a, const float *h, const float *g, float *da, float *db,
                            int64_t B, int64_t L, int64_t D, const float *h_init, const float *dh_last,
                            float *dh_init, cudaStream_t stream) {
    const long long gpb = D / V;
    const long long n = B * gpb;
    const long long blocks = (n + threads - 1) / threads;
    regcarry_backward_kernel<V, 8><<<(unsigned)blocks, threads, 0, stream>>>(a, h, g, da, db, L, D, gpb, n, h_init,
                                                                             dh_last, dh_init);
    return cudaGetLastError();
}

}  // namespace

cudaError_t launch_regcarry_backward(int vec, int threads, const float *a, const float *h, const float *g, float *da,
                                     float *db, int64_t B, int64_t L, int64_t D, const float *h_init,
                                     const float *dh_last, float *dh_init, cudaStream_t stream) {
    if (vec == 4) return launch_back_one<4>(threads, a, h, g, da, db, B, L, D, h_init, dh_last, dh_init, stream);
    if (vec == 2) return launch_back_one<2>(threads, a, h, g, da, db, B, L, D, h_init, dh_last, dh_init, stream);
    if (vec == 1) return launch_back_one<1>(threads, a, h, g, da, db, B, L, D, h_init, dh_last, dh_init, stream);
    return cudaErrorInvalidValue;
}

cudaError_t launch_regcarry_segmented(int vec, int threads, const float *a, const float *b, float *h, int64_t B,
                                      int64_t L, int64_t D, int64_t nseg, const float *h_init, float *h_last,
                                      float *aggA, float *aggB, cudaStream_t stream) {
    if (nseg < 1) return cudaErrorInvalidValue;
    if (vec == 4) return launch_seg_one<4>(threads, a, b, h, B, L, D, nseg, h_init, h_last, aggA, aggB, stream);
    if (vec == 2) return launch_seg_one<2>(threads, a, b, h, B, L, D, nseg, h_init, h_last, aggA, aggB, stream);
    if (vec == 1) return launch_seg_one<1>(threads, a, b, h, B, L, D, nseg, h_init, h_last, aggA, aggB, stream);
    return cudaErrorInvalidValue;
}

bool regcarry_supported(int vec, int prefetch) {
    return (vec == 1 || vec == 2 || vec == 4) && (prefetch == 4 || prefetch == 8 || prefetch == 16);
}

cudaError_t launch_regcarry(int vec, int prefetch, int threads, const float *a, const float *b, float *h,
                            int64_t B, int64_t L, int64_t D, const float *h_init, float *h_last,
                            cudaStream_t stream) {
#define LINREC_RC(V, P) \
    if (vec == V && prefetch == P) return launch_one<V, P>(threads, a, b, h, B, L, D, h_init, h_last, stream);
    LINREC_RC(4, 4) LINREC_RC(4, 8) LINREC_RC(4, 16)
    LINREC_RC(2, 4) LINREC_RC(2, 8) LINREC_RC(2, 16)
    LINREC_RC(1, 4) LINREC_RC(1, 8) LINREC_RC(1, 16)
#undef LINREC_RC
    return cudaErrorInvalidValue;
}

LINREC_CHECKED_REPORT(checked_report_regcarry)

}  // namespace linrec
