// rows.cu -- the scan on (B, D, L) tensors: time innermost, so channel (i, d)
// is the contiguous row i*D + d of length L.  "Kimi-K2.6 l1_p9" (its transpose
// discussion) names this layout as the one in which a warp reads a channel's
// steps contiguously; here it is a layout callers may hold their data in, not
// an intermediate copy.
//
// A row's first step has no predecessor: its map x -> a_0*x + b_0 becomes the
// constant map (0, a_0*h_init + b_0), or (0, b_0) without a state.  So the
// recurrence run straight through row after row restarts by itself at every
// row, and a warp can scan several consecutive rows as one stream.
//
// One warp owns a unit: k consecutive whole rows (one pass), or one segment of
// a row (two passes, for few long rows).  It walks the unit's elements in
// chunks of 32*V: lane l holds elements l*V .. l*V+V-1 of the chunk, loaded as
// one vector of V stored elements per array, so each array moves as one
// contiguous warp access.  Per chunk a lane composes its V maps (later map on
// the left, "Kimi-K2.6 l1_p9", derivation of the associative operator), a
// 5-step shuffle scan gives every lane the composition of the lanes before it,
// each lane replays its V steps from the carried h and stores them, and lane
// 31's last h is the carry into the next chunk.  The loads of the next P
// chunks are in flight in a register ring meanwhile, across row boundaries.
//
// Two passes: a reduce launch writes each segment's composed map, the
// library's (B, L, D) scan turns the maps, laid out (1, segments, rows), into
// every segment's last h, and an apply launch rescans every segment from the h
// before it.
#include "checked.cuh"
#include "kernels.cuh"
#include "ptx.cuh"
#include "storage.cuh"

namespace linrec {

namespace {

constexpr unsigned kAll = 0xffffffffu;

// 32 bytes per lane: two 16-byte accesses, so the shuffle scan of each chunk is
// shared by twice the elements.
struct alignas(16) Vec32 { uint4 lo, hi; };

template <int BYTES> struct RawVec;
template <> struct RawVec<32> { using type = Vec32; };
template <> struct RawVec<16> { using type = uint4; };
template <> struct RawVec<8> { using type = uint2; };
template <> struct RawVec<4> { using type = unsigned int; };
template <> struct RawVec<2> { using type = unsigned short; };

// Streaming (evict-first) vector load and store of one lane's V elements.
template <typename W>
__device__ __forceinline__ W ldcs_vec(const W *p) { return __ldcs(p); }
template <>
__device__ __forceinline__ Vec32 ldcs_vec<Vec32>(const Vec32 *p) {
    const uint4 *q = reinterpret_cast<const uint4 *>(p);
    return Vec32{__ldcs(q), __ldcs(q + 1)};
}
template <typename W>
__device__ __forceinline__ void stcs_vec(W *p, const W &w) { __stcs(p, w); }
template <>
__device__ __forceinline__ void stcs_vec<Vec32>(Vec32 *p, const Vec32 &w) {
    uint4 *q = reinterpret_cast<uint4 *>(p);
    __stcs(q, w.lo);
    __stcs(q + 1, w.hi);
}

template <int DT, int V, typename W>
__device__ __forceinline__ void unpack(const W &w, float (&x)[V]) {
    using E = typename Storage<DT>::raw;
    const E *e = reinterpret_cast<const E *>(&w);
#pragma unroll
    for (int v = 0; v < V; ++v) x[v] = Storage<DT>::get(e[v]);
}

template <int DT, int V, typename W>
__device__ __forceinline__ W pack(const float (&x)[V]) {
    using E = typename Storage<DT>::raw;
    W w;
    E *e = reinterpret_cast<E *>(&w);
#pragma unroll
    for (int v = 0; v < V; ++v) e[v] = Storage<DT>::put(x[v]);
    return w;
}

template <int DT, int V, int P>
__global__ void __launch_bounds__(256)
rows_scan_kernel(const typename Storage<DT>::raw *__restrict__ a, const typename Storage<DT>::raw *__restrict__ b,
                 typename Storage<DT>::raw *__restrict__ h, const long long R, const long long L,
                 const long long seg_len, const long long nseg, const long long rows_per_unit, const int mode,
                 const float *h_init, float *h_last, float *__restrict__ aggA, float *__restrict__ aggB,
                 const float *__restrict__ aggH, float *__restrict__ aggX)
{
    using E = typename Storage<DT>::raw;
    using W = typename RawVec<V * (int)sizeof(E)>::type;
    constexpr int CH = 32 * V;                // elements per chunk
    pdl_wait();   // launched as a programmatic dependent: nothing before it is touched yet
    const long long u = ((long long)blockIdx.x * blockDim.x + threadIdx.x) >> 5;
    const int lane = threadIdx.x & 31;
    const long long units = nseg > 1 ? R * nseg : (R + rows_per_unit - 1) / rows_per_unit;
    if (u >= units) return;                   // u is the same for the whole warp
    // the unit: elements [e0, e1) of the flattened (R, L) array, starting in row r0 at step t0
    long long r0, g = 0, e0, e1, t0;
    if (nseg > 1) {
        r0 = u / nseg;
        g = u - r0 * nseg;
        t0 = g * seg_len;
        e0 = r0 * L + t0;
        e1 = r0 * L + ((t0 + seg_len < L) ? t0 + seg_len : L);
    } else {
        r0 = u * rows_per_unit;
        const long long r1 = (r0 + rows_per_unit < R) ? r0 + rows_per_unit : R;
        t0 = 0;
        e0 = r0 * L;
        e1 = r1 * L;
    }
    const bool reduce = mode == kRowsReduce, apply = mode == kRowsApply;
    // where this lane's first element of the current chunk is: row `row`, step `t`
    long long row = r0, t = t0 + lane * V;
    if (t >= L) { row += t / L; t %= L; }
    // extents for the index-checked build: elements of a, b, h; of the per-row states; of the
    // per-segment arrays
    const long long n_all = R * L, n_seg = nseg * R;
    // the h entering the unit: irrelevant when it starts a row (the first map is constant)
    float carry = (apply && g > 0 && inside(aggH + (g - 1) * R + r0, aggH, n_seg)) ? aggH[(g - 1) * R + r0] : 0.0f;
    float runA = 1.0f, runB = 0.0f;           // reduce: the segment's composed map so far

    const E *pa = a + e0;
    const E *pb = b + e0;
    E *ph = h + e0;
    const long long n = e1 - e0;              // a multiple of V (L % V == 0)
    auto ld = [&](const E *p, const E *base) -> W {
#ifdef LINREC_DEBUG
        if (!inside(reinterpret_cast<const W *>(p), base, n_all)) {
            W w;
            memset(&w, 0, sizeof(W));
            return w;
        }
#endif
        return ldcs_vec<W>(reinterpret_cast<const W *>(p));
    };
    W ra[P], rb[P];
#pragma unroll
    for (int j = 0; j < P; ++j) {
        const long long off = (long long)j * CH + lane * V;
        if (off < n) {
            ra[j] = ld(pa + off, a);
            rb[j] = ld(pb + off, b);
        }
    }
    for (long long c0 = 0; c0 < n; c0 += (long long)P * CH) {
#pragma unroll
        for (int j = 0; j < P; ++j) {
            const long long c = c0 + (long long)j * CH;
            if (c >= n) break;                // the same for the whole warp
            const long long off = c + lane * V;
            const bool valid = off < n;       // then all V elements are, and they share a row
            float xa[V], xb[V];
            if (valid) {
                unpack<DT, V>(ra[j], xa);
                unpack<DT, V>(rb[j], xb);
            } else {
#pragma unroll
                for (int v = 0; v < V; ++v) { xa[v] = 1.0f; xb[v] = 0.0f; }   // the identity map
            }
            const long long nxt = off + (long long)P * CH;
            if (nxt < n) {
                ra[j] = ld(pa + nxt, a);
                rb[j] = ld(pb + nxt, b);
            }
            if (valid && t == 0) {            // a row's first step: the constant map
                if (h_init) {
                    // two passes: the apply launch reads the state the reduce launch kept,
                    // since h_last may be the same buffer as h_init
                    const float s0 = apply ? (inside(aggX + row, aggX, R) ? aggX[row] : 0.0f)
                                           : (inside(h_init + row, h_init, R) ? h_init[row] : 0.0f);
                    if (reduce && inside(aggX + row, aggX, R)) aggX[row] = s0;
                    xb[0] = fmaf(xa[0], s0, xb[0]);
                }
                xa[0] = 0.0f;
            }

            float A = 1.0f, Bv = 0.0f;
#pragma unroll
            for (int v = 0; v < V; ++v) {
                Bv = fmaf(xa[v], Bv, xb[v]);
                A = xa[v] * A;
            }
            // inclusive scan over the lanes: lane l ends with lanes 0..l composed
#pragma unroll
            for (int o = 1; o < 32; o <<= 1) {
                const float uA = __shfl_up_sync(kAll, A, o);
                const float uB = __shfl_up_sync(kAll, Bv, o);
                if (lane >= o) {              // (later) o (earlier)
                    Bv = fmaf(A, uB, Bv);
                    A = A * uA;
                }
            }
            if (reduce) {
                const float tA = __shfl_sync(kAll, A, 31), tB = __shfl_sync(kAll, Bv, 31);
                runB = fmaf(tA, runB, tB);
                runA = tA * runA;
            } else {
                float eA = __shfl_up_sync(kAll, A, 1), eB = __shfl_up_sync(kAll, Bv, 1);
                if (lane == 0) { eA = 1.0f; eB = 0.0f; }
                float hv = fmaf(eA, carry, eB);
                float out[V];
#pragma unroll
                for (int v = 0; v < V; ++v) {
                    hv = fmaf(xa[v], hv, xb[v]);
                    out[v] = hv;
                }
                if (valid) {
                    if (inside(reinterpret_cast<W *>(ph + off), h, n_all, true))
                        stcs_vec<W>(reinterpret_cast<W *>(ph + off), pack<DT, V, W>(out));
                    if (h_last && t + V == L && inside(h_last + row, h_last, R, true)) h_last[row] = hv;
                }
                carry = __shfl_sync(kAll, hv, 31);   // h at the chunk's end (a partial chunk ends the unit)
            }
            t += CH;                          // the lane's element in the next chunk
            if (t >= L) {
                if (L >= CH) { t -= L; ++row; }
                else { row += t / L; t %= L; }
            }
        }
    }
    if (reduce && lane == 0) {
        // the first segment starts its row, so its map is constant: the scan of these
        // maps from 0 gives every segment's last h
        if (inside(aggA + g * R + r0, aggA, n_seg)) aggA[g * R + r0] = runA;
        if (inside(aggB + g * R + r0, aggB, n_seg)) aggB[g * R + r0] = runB;
    }
    pdl_release();   // this warp's unit is done: the next launch may be scheduled
}

template <int DT, int V, int P>
cudaError_t launch_one(const RowsLaunch &p, cudaStream_t stream) {
    using E = typename Storage<DT>::raw;
    const long long units = p.nseg > 1 ? p.R * p.nseg : (p.R + p.rows_per_unit - 1) / p.rows_per_unit;
    const long long blocks = (units * 32 + kRowsThreads - 1) / kRowsThreads;
    const E *a = static_cast<const E *>(p.a), *b = static_cast<const E *>(p.b);
    E *h = static_cast<E *>(p.h);
    long long R = p.R, L = p.L, seg_len = p.seg_len, nseg = p.nseg, rpu = p.rows_per_unit;
    int mode = p.mode;
    const float *h_init = p.h_init, *aggH = p.aggH;
    float *h_last = p.h_last, *aggA = p.aggA, *aggB = p.aggB, *aggX = p.aggX;
    void *args[] = {&a, &b, &h, &R, &L, &seg_len, &nseg, &rpu, &mode, &h_init, &h_last, &aggA, &aggB, &aggH, &aggX};
    return launch_dependent(reinterpret_cast<const void *>(&rows_scan_kernel<DT, V, P>), dim3((unsigned)blocks),
                            dim3(kRowsThreads), 0, stream, args);
}

template <int DT, int P>
cudaError_t launch_dt(const RowsLaunch &p, cudaStream_t stream) {
    constexpr int EB = (int)sizeof(typename Storage<DT>::raw);
    switch (p.vec * EB) {
        case 32: return launch_one<DT, 32 / EB, P>(p, stream);
        case 16: return launch_one<DT, 16 / EB, P>(p, stream);
        case 8: return launch_one<DT, 8 / EB, P>(p, stream);
        case 4: return launch_one<DT, 4 / EB, P>(p, stream);
        case 2:
            if constexpr (EB == 2) return launch_one<DT, 1, P>(p, stream);
            else return cudaErrorInvalidValue;
    }
    return cudaErrorInvalidValue;
}

}  // namespace

bool rows_supported(int dtype, int vec, int prefetch) {
    const int eb = elem_bytes_of(dtype);
    return vec >= 1 && (vec & (vec - 1)) == 0 && vec * eb <= 32 && (prefetch == 2 || prefetch == 4);
}

cudaError_t launch_rows(const RowsLaunch &p, cudaStream_t stream) {
    if (!rows_supported(p.dtype, p.vec, p.prefetch)) return cudaErrorInvalidValue;
    if (p.rows_per_unit < 1 || p.nseg < 1 || (p.nseg > 1 && p.rows_per_unit != 1)) return cudaErrorInvalidValue;
    if (p.R == 0 || p.L == 0) return cudaSuccess;
    if (p.dtype == kDtypeF32) return p.prefetch == 4 ? launch_dt<kDtypeF32, 4>(p, stream)
                                                     : launch_dt<kDtypeF32, 2>(p, stream);
    if (p.dtype == kDtypeBF16) return p.prefetch == 4 ? launch_dt<kDtypeBF16, 4>(p, stream)
                                                      : launch_dt<kDtypeBF16, 2>(p, stream);
    if (p.dtype == kDtypeF16) return p.prefetch == 4 ? launch_dt<kDtypeF16, 4>(p, stream)
                                                     : launch_dt<kDtypeF16, 2>(p, stream);
    return cudaErrorInvalidValue;
}

LINREC_CHECKED_REPORT(checked_report_rows)

}  // namespace linrec
