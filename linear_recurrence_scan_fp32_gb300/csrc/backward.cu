// backward.cu -- the gradient of the linear-recurrence scan, TMA-staged.
//
// Forward: h_t = a_t*h_{t-1} + b_t (POPCORNBENCH "Kimi-K2.6 l1_p9", problem
// statement), h_{-1} = h_init or 0.  For a loss with dL/dh = g the chain rule
// gives, with c_t = dL/dh_t in total,
//
//     c_{L-1} = g_{L-1} + dh_last,     c_t = g_t + a_{t+1} * c_{t+1},
//     db_t = c_t,    da_t = c_t * h_{t-1},    dh_init = a_0 * c_0,
//
// the same first-order recurrence run right to left, with the slope taken one
// step later (a_{t+1}).  So the kernel is the forward chunked kernel on the
// reversed sequence: chunk qr = 0 is the last time chunk, a thread walks its
// rows from the bottom of the tile up, and the carry entering a chunk (the
// running c) comes from the chunk after it in time, in register (slice-owner
// mode), by the shared decoupled look-back, or (two-pass mode, for few long
// slices) from a scan of the tiles' maps: a reduce launch writes every tile's
// map, the library's forward scan composes them in reversed chunk order, and
// an apply launch gives each tile the running c of the chunk after it.  Per tile the ring holds three
// boxes: g (rows t0 .. t0+TT-1), a one row later (a_{t+1}) and h one row
// earlier (h_{t-1}; only when da is wanted).  Out-of-range rows arrive as
// zeros; rows past L-1 are given the identity map (slope 1, value 0) so the
// carry entering the last row passes through them unchanged.
#include "kernels.cuh"
#include "lookback.cuh"
#include "ptx.cuh"

namespace linrec {

namespace {

constexpr uint32_t kTmaPolls = 1u << 22;

struct TileCoord {
    long long id;                       // tile id (>= n_tiles: no tile)
    int qr;                             // time chunk counted from the end
    int bi;                             // batch index
    int d0;                             // first channel
    int pad;
};

template <int TD, int TT, int S, int ST>
struct __align__(128) BackSmem {
    float g[ST][TT * TD];
    float a[ST][TT * TD];               // row r holds a_{t0 + r + 1}
    float h[ST][TT * TD];               // row r holds h_{t0 + r - 1}
    float segA[S][TD + 32 / S], segB[S][TD + 32 / S];   // padded: the transposed reads hit 32 banks
    float carry[TD];
    uint64_t full[ST];
    TileCoord tile[ST];
    uint32_t tag;
};

// FM >= 0 compiles the one carry mode FM (`mode` must equal it; -1 takes it at run time), and
// launch_backward takes such a copy where there is one.  Without the other modes' code the slice-
// owner copies need 80-92 registers against 103-130, and resident CTAs per SM stay the same
// (shared memory or the launch bounds hold them).  Measured on GB300, us per call, general ->
// slice-owner copy: (32, 4096, 256) 103.3 -> 101.7, (56, 4096, 256) 182.7 -> 177.8, (64, 512,
// 1024) 102.6 -> 100.8, (64, 2048, 1024) 388.7 -> 385.6; (16, 4096, 256), (1, 32768, 4096) and
// (8, 4096, 4096) unchanged.
template <int TD, int TT, int S, int ST, int FM = -1>
__global__ void __launch_bounds__(TD * S, (TD * S >= 512) ? 1 : 2)
chunked_backward_kernel(const __grid_constant__ CUtensorMap map_g,
                        const __grid_constant__ CUtensorMap map_a,
                        const __grid_constant__ CUtensorMap map_h,
                        const float *__restrict__ a_glob, float *__restrict__ da, float *__restrict__ db,
                        const long long L, const long long D,
                        const long long slices_per_batch, const long long n_slices,
                        const long long chunks, const long long n_tiles,
                        const int mode,              // kModeOwn, kModeLookback, kModeReduce or kModeApply
                        Control *__restrict__ ctrl, unsigned long long *__restrict__ words,
                        unsigned int *__restrict__ status, const long long spin_limit,
                        const long long silent_tile, const float *h_init, const float *dh_last,
                        float *dh_init)
{
    constexpr int K = TT / S;
    constexpr int R = (S >= 4) ? 16 / S : 4;
    constexpr uint32_t kBox = TT * TD * sizeof(float);
    static_assert(TT % S == 0 && TD % 32 == 0 && (32 % S) == 0 && S >= 2 && ST >= 2, "tile shape");
    using Smem = BackSmem<TD, TT, S, ST>;
    extern __shared__ __align__(128) unsigned char smem_raw[];
    Smem &sm = *reinterpret_cast<Smem *>(smem_raw);

    const bool own = FM >= 0 ? FM == kModeOwn : mode == kModeOwn;
    const bool lookback = FM >= 0 ? FM == kModeLookback : mode == kModeLookback;
    const bool reduce = FM >= 0 ? FM == kModeReduce : mode == kModeReduce;
    const bool apply = FM >= 0 ? FM == kModeApply : mode == kModeApply;
    const bool want_da = da != nullptr;
    const bool load_h = want_da && !reduce;   // the reduce launch needs the maps only: g and a
    const uint32_t stage_bytes = (load_h ? 3u : 2u) * kBox;
    // two-pass mode: per-tile maps and the scanned running c, indexed [tile id][channel], and
    // each slice's c entering the last chunk, indexed [slice][channel]
    float *const tileA = reinterpret_cast<float *>(words);
    float *const tileB = tileA + n_tiles * TD;
    const float *const tileH = tileB + n_tiles * TD;
    float *const tileX = tileB + 2 * n_tiles * TD;
    pdl_wait();   // launched as a programmatic dependent: nothing before it is touched yet
    const int tid = threadIdx.x;
    const int c = tid % TD;
    const int s = tid / TD;
    const int cc = tid / S;
    const int ss = tid % S;
    const int gbase = (tid & 31) & ~(S - 1);

    unsigned long long *const wAggA = words;
    unsigned long long *const wAggB = words + n_tiles * TD;
    unsigned long long *const wInc = words + 2 * n_tiles * TD;
    // extents for the index-checked build: elements of a, h, g, da, db, and of the (B, D) states
    const long long n_all = (n_slices / slices_per_batch) * L * D;
    const long long n_state = (n_slices / slices_per_batch) * D;

    auto issue = [&](int st, long long id, long long qr, long long slice) {
        const long long bi = slice / slices_per_batch;
        const int d0 = (int)((slice - bi * slices_per_batch) * TD);
        const int t0 = (int)((chunks - 1 - qr) * TT);
        sm.tile[st] = TileCoord{id, (int)qr, (int)bi, d0, 0};
        mbar_arrive_expect_tx(&sm.full[st], stage_bytes);
        tma_load_3d(sm.g[st], &map_g, &sm.full[st], d0, t0, (int)bi);
        tma_load_3d(sm.a[st], &map_a, &sm.full[st], d0, t0 + 1, (int)bi);
        if (load_h) tma_load_3d(sm.h[st], &map_h, &sm.full[st], d0, t0 - 1, (int)bi);
    };
    auto finish = [&](int st) { sm.tile[st] = TileCoord{n_tiles, 0, 0, 0, 0}; };
    long long own_slice = blockIdx.x, own_q = 0, own_m = 0;
    auto next_tile = [&](long long &qr, long long &slice) -> long long {
        if (reduce || apply) {                // independent tiles, static round-robin
            const long long k = blockIdx.x + (own_m++) * (long long)gridDim.x;
            if (k >= n_tiles) return n_tiles;
            const long long id = apply ? n_tiles - 1 - k : k;
            qr = id / n_slices;
            slice = id - qr * n_slices;
            return id;
        }
        if (own) {
            if (own_slice >= n_slices) return n_tiles;
            qr = own_q;
            slice = own_slice;
            if (++own_q == chunks) { own_q = 0; own_slice += gridDim.x; }
            return qr * n_slices + slice;
        }
        const long long id = (long long)atomicAdd(&ctrl->tile_counter, 1ull);
        if (id >= n_tiles) return n_tiles;
        qr = id / n_slices;
        slice = id - qr * n_slices;
        return id;
    };

    const bool misaligned = (smem_u32(smem_raw) & 127u) != 0;
    if (tid == 0) {
        long long first = n_tiles;
        if (misaligned) {
            atomicOr(status, kStatusTmaTimeout);
            if (lookback) atomicExch(&ctrl->abort, 1u);
        } else {
            for (int st = 0; st < ST; ++st) mbar_init(&sm.full[st], 1);
            mbar_fence_init();
            tmap_prefetch(&map_g);
            tmap_prefetch(&map_a);
            if (load_h) tmap_prefetch(&map_h);
            if (lookback) {
                sm.tag = tag_of(ld_relaxed_u32(&ctrl->epoch));
            }
            long long qr = 0, slice = 0;
            first = next_tile(qr, slice);
            if (first < n_tiles) issue(0, first, qr, slice);
        }
        if (first >= n_tiles) finish(0);
    }
    __syncthreads();

    const uint32_t tag = lookback ? sm.tag : 0u;
    uint32_t phases = 0;
    long long next_fill = 1;
    bool ended = sm.tile[0].id >= n_tiles;
    long long ahead = -1, ahead_q = 0, ahead_slice = 0;
    uint32_t abort_seen = 0;
    float run = 0.0f;

    for (long long k = 0;; ++k) {
        const int st = (int)(k % ST);
        const TileCoord tc = sm.tile[st];
        const long long id = tc.id;
        if (id >= n_tiles) break;

        if (!mbar_wait_bounded(&sm.full[st], (phases >> st) & 1u, kTmaPolls)) {
            atomicOr(status, kStatusTmaTimeout);
            if (lookback) atomicExch(&ctrl->abort, 1u);
        }
        phases ^= 1u << st;

        if (tid == 0) {
            if (!ended && abort_seen != 0) {
                ended = true;
                finish((int)(next_fill % ST));
            }
            while (!ended && next_fill < k + ST) {
                const int s2 = (int)(next_fill % ST);
                long long nq = ahead_q, nslice = ahead_slice;
                const long long nid = ahead >= 0 ? ahead : next_tile(nq, nslice);
                ahead = -1;
                if (nid >= n_tiles) {
                    ended = true;
                    finish(s2);
                } else {
                    issue(s2, nid, nq, nslice);
                }
                ++next_fill;
            }
            if (lookback) {
                if (!ended && ahead < 0) ahead = next_tile(ahead_q, ahead_slice);
                abort_seen = ld_relaxed_u32(&ctrl->abort);
            }
        }

        const long long qr = tc.qr, bi = tc.bi, d0 = tc.d0;
        const long long t0 = (chunks - 1 - qr) * TT;
        const int rtop = TT - 1 - s * K;      // this thread's first (latest) row; it walks up K rows

        // ---- compose this thread's K steps, latest first ----------------------------
        float al[K], gg[K];
#pragma unroll
        for (int j = 0; j < K; ++j) {
            const int r = rtop - j;
            gg[j] = sm.g[st][r * TD + c];
            // slope a_{t+1}; rows at or past L-1 get 1 so the carry reaches row L-1 whole
            al[j] = (t0 + r >= L - 1) ? 1.0f : sm.a[st][r * TD + c];
        }
        float A = 1.0f, Bv = 0.0f;
#pragma unroll
        for (int j = 0; j < K; ++j) {
            Bv = fmaf(al[j], Bv, gg[j]);
            A = al[j] * A;
        }
        sm.segA[s][c] = A;
        sm.segB[s][c] = Bv;
        __syncthreads();

        // ---- shuffle scan over the S segment pairs of each channel -------------------
        float xA = sm.segA[ss][cc], xB = sm.segB[ss][cc];
#pragma unroll
        for (int off = 1; off < S; off <<= 1) {
            const float uA = __shfl_up_sync(kFull, xA, off, S);
            const float uB = __shfl_up_sync(kFull, xB, off, S);
            if (ss >= off) {
                xB = fmaf(xA, uB, xB);
                xA = xA * uA;
            }
        }
        float eA = __shfl_up_sync(kFull, xA, 1, S);
        float eB = __shfl_up_sync(kFull, xB, 1, S);
        if (ss == 0) { eA = 1.0f; eB = 0.0f; }
        sm.segA[ss][cc] = eA;
        sm.segB[ss][cc] = eB;
        const float tA = __shfl_sync(kFull, xA, S - 1, S);
        const float tB = __shfl_sync(kFull, xB, S - 1, S);

        // ---- the running c entering the tile from later in time ----------------------
        const float c_after = (dh_last && d0 + cc < D && inside(dh_last + bi * D + d0 + cc, dh_last, n_state))
                                  ? dh_last[bi * D + d0 + cc]
                                  : 0.0f;
        if (own) {
            if (ss == 0) {
                const float carry = (qr == 0) ? c_after : run;
                run = fmaf(tA, carry, tB);
                sm.carry[cc] = carry;
            }
        } else if (reduce) {
            // the tile's map; the last chunk's absorbs dh_last, so the scan of these maps
            // from 0 (in reversed chunk order) is the chain of running c values
            if (ss == 0) {
                if (inside(tileA + id * TD + cc, tileA, n_tiles * TD)) tileA[id * TD + cc] = (qr == 0) ? 0.0f : tA;
                if (inside(tileB + id * TD + cc, tileB, n_tiles * TD))
                    tileB[id * TD + cc] = (qr == 0) ? fmaf(tA, c_after, tB) : tB;
                // kept for the apply launch: dh_init may be the same buffer as dh_last, and the
                // apply launch writes it while other tiles still need the incoming state
                if (qr == 0 && inside(tileX + id * TD + cc, tileX, n_slices * TD)) tileX[id * TD + cc] = c_after;
            }
        } else if (apply) {
            if (ss == 0)
                sm.carry[cc] = (qr == 0) ? (inside(tileX + id * TD + cc, tileX, n_slices * TD) ? tileX[id * TD + cc] : 0.0f)
                                         : (inside(tileH + (id - n_slices) * TD + cc, tileH, n_tiles * TD)
                                                ? tileH[(id - n_slices) * TD + cc]
                                                : 0.0f);
        } else {
            const bool publish = (qr + 1 < chunks) && (id != silent_tile);
            float carry = c_after;
            if (qr > 0)
                carry = lookback_carry<S, R>(id, n_slices, TD, cc, ss, gbase, tag, publish, tA, tB, c_after,
                                             wAggA, wAggB, wInc, n_tiles * TD, ctrl, status, spin_limit);
            if (ss == 0) {
                if (publish && inside(wInc + id * TD + cc, wInc, n_tiles * TD))
                    st_relaxed_u64(&wInc[id * TD + cc], pack_word(tag, fmaf(tA, carry, tB)));
                sm.carry[cc] = carry;
            }
        }
        __syncthreads();

        // ---- replay from the carried value; db = c, da = c * h_{t-1} ------------------
        float cv = fmaf(sm.segA[s][c], sm.carry[c], sm.segB[s][c]);
        const long long d = d0 + c;
        if (!reduce && d < D) {
            const long long trow = t0 + rtop;             // latest row of this thread
            float *pdb = db + (bi * L + trow) * D + d;
            float *pda = want_da ? da + (bi * L + trow) * D + d : nullptr;
#pragma unroll
            for (int j = 0; j < K; ++j) {
                cv = fmaf(al[j], cv, gg[j]);
                const long long t = trow - j;
                if (t < L) {
                    if (inside(pdb - (long long)j * D, db, n_all, true)) pdb[-(long long)j * D] = cv;
                    if (want_da) {
                        const float hp = (t == 0) ? ((h_init && inside(h_init + bi * D + d, h_init, n_state))
                                                         ? h_init[bi * D + d]
                                                         : 0.0f)
                                                  : sm.h[st][(rtop - j) * TD + c];
                        if (inside(pda - (long long)j * D, da, n_all, true)) pda[-(long long)j * D] = cv * hp;
                    }
                    if (t == 0 && dh_init && inside(dh_init + bi * D + d, dh_init, n_state, true) &&
                        inside(a_glob + bi * L * D + d, a_glob, n_all))
                        dh_init[bi * D + d] = a_glob[bi * L * D + d] * cv;
                }
            }
        }
        __syncthreads();
    }

    pdl_release();   // this CTA's tiles are done: the next launch may be scheduled

    if (lookback) {
        __syncthreads();
        if (tid == 0) {
            __threadfence();
            const unsigned int prev = atomicAdd(&ctrl->done, 1u);
            if (prev == gridDim.x - 1) {
                __threadfence();
                atomicExch(&ctrl->tile_counter, 0ull);
                atomicExch(&ctrl->done, 0u);
                atomicExch(&ctrl->abort, 0u);
                atomicExch(&ctrl->epoch, next_epoch(ld_relaxed_u32(&ctrl->epoch)));
                __threadfence();
            }
        }
    }
}

template <int TD, int TT, int S, int ST>
constexpr ChunkedVariant make_variant() {
    return ChunkedVariant{TD, TT, S, ST, TD * S, sizeof(BackSmem<TD, TT, S, ST>)};
}

#define LINREC_BACKWARD_VARIANTS(X) \
    X(32, 128, 8, 2)                \
    X(32, 64, 4, 3)                 \
    X(32, 64, 4, 4)                 \
    X(64, 64, 4, 2)                 \
    X(64, 128, 8, 2)                \
    X(128, 64, 4, 2)                \
    X(256, 32, 2, 2)

#define LINREC_V_ENTRY(TD, TT, S, ST) make_variant<TD, TT, S, ST>(),
const ChunkedVariant kVariants[] = {LINREC_BACKWARD_VARIANTS(LINREC_V_ENTRY)};
#undef LINREC_V_ENTRY

const void *kernel_of(const ChunkedVariant *v) {
#define LINREC_K_ENTRY(TD, TT, S, ST)                                                        \
    if (v->tile_d == TD && v->tile_t == TT && v->segments == S && v->stages == ST)           \
        return reinterpret_cast<const void *>(&chunked_backward_kernel<TD, TT, S, ST>);
    LINREC_BACKWARD_VARIANTS(LINREC_K_ENTRY)
#undef LINREC_K_ENTRY
    return nullptr;
}

}  // namespace

const ChunkedVariant *backward_variants(int *count) {
    *count = (int)(sizeof(kVariants) / sizeof(kVariants[0]));
    return kVariants;
}

cudaError_t backward_ctas_per_sm(const ChunkedVariant *v, int *ctas) {
    const void *fn = kernel_of(v);
    if (!fn) return cudaErrorInvalidValue;
    cudaError_t err = cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)v->smem_bytes);
    if (err != cudaSuccess) return err;
    return cudaOccupancyMaxActiveBlocksPerMultiprocessor(ctas, fn, v->threads, v->smem_bytes);
}

// The copy of a variant's kernel compiled for carry mode `mode` alone: every tile in slice-owner
// mode; the tiles of the two-pass and look-back modes ({32, 128} and {64, 128}) in those too.
static const void *fixed_backward_kernel(const ChunkedVariant *v, int mode) {
#define LINREC_OB_ENTRY(TD, TT, S, ST)                                                              \
    if (mode == kModeOwn && v->tile_d == TD && v->tile_t == TT && v->segments == S && v->stages == ST) \
        return reinterpret_cast<const void *>(&chunked_backward_kernel<TD, TT, S, ST, kModeOwn>);
    LINREC_BACKWARD_VARIANTS(LINREC_OB_ENTRY)
#undef LINREC_OB_ENTRY
#define LINREC_OB_CHAINED(TD, TT, S, ST)                                                            \
    if (v->tile_d == TD && v->tile_t == TT && v->segments == S && v->stages == ST) {                \
        if (mode == kModeLookback)                                                                  \
            return reinterpret_cast<const void *>(&chunked_backward_kernel<TD, TT, S, ST, kModeLookback>); \
        if (mode == kModeReduce)                                                                    \
            return reinterpret_cast<const void *>(&chunked_backward_kernel<TD, TT, S, ST, kModeReduce>);   \
        if (mode == kModeApply)                                                                     \
            return reinterpret_cast<const void *>(&chunked_backward_kernel<TD, TT, S, ST, kModeApply>);    \
    }
    LINREC_OB_CHAINED(32, 128, 8, 2)
    LINREC_OB_CHAINED(64, 128, 8, 2)
#undef LINREC_OB_CHAINED
    return nullptr;
}

cudaError_t launch_backward(const BackwardLaunch &p, cudaStream_t stream) {
    const void *fn = fixed_backward_kernel(p.variant, p.mode);
    if (!fn) fn = kernel_of(p.variant);
    if (!fn) return cudaErrorInvalidValue;
    cudaError_t err = cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                           (int)p.variant->smem_bytes);
    if (err != cudaSuccess) return err;
    long long L = p.L, D = p.D, spb = p.slices_per_batch, ns = p.n_slices, ch = p.chunks, nt = p.n_tiles;
    long long spin = p.spin_limit, silent = p.silent_tile;
    int mode = p.mode;
    const float *a = p.a;
    float *da = p.da, *db = p.db;
    Control *ctrl = p.ctrl;
    unsigned long long *words = p.words;
    unsigned int *status = p.status;
    const float *h_init = p.h_init, *dh_last = p.dh_last;
    float *dh_init = p.dh_init;
    void *args[] = {(void *)&p.map_g, (void *)&p.map_a, (void *)&p.map_h, &a, &da, &db, &L, &D, &spb, &ns, &ch,
                    &nt, &mode, &ctrl, &words, &status, &spin, &silent, &h_init, &dh_last, &dh_init};
    return launch_dependent(fn, dim3((unsigned)p.grid), dim3((unsigned)p.variant->threads), p.variant->smem_bytes,
                            stream, args);
}

LINREC_CHECKED_REPORT(checked_report_backward)

}  // namespace linrec
