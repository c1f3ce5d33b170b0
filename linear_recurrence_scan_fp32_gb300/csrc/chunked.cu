// chunked.cu -- the TMA-staged, look-back path of the linear-recurrence scan.
//
// h_0 = b_0, h_t = a_t*h_{t-1} + b_t per channel (POPCORNBENCH "Kimi-K2.6 l1_p9",
// problem statement).  The (B, L, D) problem is cut into tiles of TT time steps
// x TD channels of one batch index.  Tile id = chunk * n_slices + slice, so
// tile ids advance in time for all channel slices together, and the tile
// before tile i in the same slice is tile i - n_slices.
//
// Per tile, inside one CTA of TD * S threads:
//  1. TMA copies the a and b boxes (TT x TD fp32 each) into a shared-memory
//     ring of ST stages; one mbarrier per stage counts the bytes.
//  2. Thread (channel c, segment s) composes its K = TT/S consecutive affine
//     maps x -> a*x + b into one pair (A, B), later map on the left:
//     (a2,b2) o (a1,b1) = (a2*a1, a2*b1 + b2) ("Kimi-K2.6 l1_p9", derivation of
//     the associative operator).  Its a, b values stay in registers.
//  3. A warp-shuffle scan over the S segment pairs of each channel gives every
//     segment its exclusive prefix and the tile its aggregate.
//  4. Decoupled look-back (one thread per channel): publish the tile aggregate,
//     walk back over earlier tiles of the same slice, composing aggregates
//     until an inclusive value is found, publish this tile's inclusive value.
//     Only the running value h crosses tile boundaries ("Kimi-K2.6 l1_p9",
//     the running_h carry): h_out = A_prefix * h_in + B_prefix.
//  5. Every thread replays its K steps from the carried value and stores h.
//
// Tile ids come from an atomic counter, so every predecessor of a tile was
// handed to a CTA that is running or done: the look-back cannot wait on a tile
// that is not yet scheduled.  Every wait is bounded; on expiry the kernel
// records an error bit in the status word and carries on with NaN.
#include "kernels.cuh"
#include "ptx.cuh"

namespace linrec {

namespace {

constexpr uint32_t kTmaPolls = 1u << 22;   // ~1 s of polls with back-off

template <int TD, int TT, int S, int ST>
struct __align__(128) ChunkSmem {
    float a[ST][TT * TD];
    float b[ST][TT * TD];
    float segA[S][TD], segB[S][TD];     // per-segment aggregates
    float preA[S][TD], preB[S][TD];     // exclusive prefix of each segment
    float tileA[TD], tileB[TD], carry[TD];
    uint64_t full[ST];                  // one mbarrier per ring stage
    long long tile_id[ST];              // tile loaded into each stage (>= n_tiles: none)
    uint32_t tag;                       // look-back tag of this launch
    uint32_t ended;                     // the tile counter ran out (thread 0 only)
};

__device__ __forceinline__ void decode_tile(long long id, long long n_slices, long long slices_per_batch,
                                            long long &q, long long &bi, long long &d0, int td) {
    q = id / n_slices;
    const long long p = id - q * n_slices;
    bi = p / slices_per_batch;
    d0 = (p - bi * slices_per_batch) * td;
}

template <int TD, int TT, int S, int ST>
__global__ void __launch_bounds__(TD * S, 1)
chunked_scan_kernel(const __grid_constant__ CUtensorMap map_a,
                    const __grid_constant__ CUtensorMap map_b,
                    float *__restrict__ h,
                    const long long L, const long long D,
                    const long long slices_per_batch, const long long n_slices,
                    const long long chunks, const long long n_tiles,
                    Control *__restrict__ ctrl, unsigned long long *__restrict__ words,
                    unsigned int *__restrict__ status,
                    const long long spin_limit, const long long silent_tile)
{
    constexpr int K = TT / S;                 // time steps per thread
    constexpr uint32_t kStageBytes = 2u * TT * TD * sizeof(float);
    static_assert(TT % S == 0 && TD % 32 == 0 && (32 % S) == 0 && ST >= 2, "tile shape");
    using Smem = ChunkSmem<TD, TT, S, ST>;
    extern __shared__ __align__(128) unsigned char smem_raw[];
    Smem &sm = *reinterpret_cast<Smem *>(smem_raw);

    const int tid = threadIdx.x;
    const int c = tid % TD;                   // channel within the tile
    const int s = tid / TD;                   // segment within the tile

    unsigned long long *const wAggA = words;
    unsigned long long *const wAggB = words + n_tiles * TD;
    unsigned long long *const wInc = words + 2 * n_tiles * TD;

    auto issue = [&](int st, long long id) {
        long long q, bi, d0;
        decode_tile(id, n_slices, slices_per_batch, q, bi, d0, TD);
        mbar_arrive_expect_tx(&sm.full[st], kStageBytes);
        tma_load_3d(sm.a[st], &map_a, &sm.full[st], (int)d0, (int)(q * TT), (int)bi);
        tma_load_3d(sm.b[st], &map_b, &sm.full[st], (int)d0, (int)(q * TT), (int)bi);
    };
    auto grab = [&]() -> long long {
        return (long long)atomicAdd(&ctrl->tile_counter, 1ull);
    };

    // TMA writes whole boxes at 128-byte aligned shared addresses; the layout
    // guarantees it when the dynamic window is aligned, so check that once.
    const bool misaligned = (smem_u32(smem_raw) & 127u) != 0;
    if (misaligned) {
        if (tid == 0) {
            atomicOr(status, kStatusTmaTimeout);
            atomicExch(&ctrl->abort, 1u);
        }
    }
    if (tid == 0 && !misaligned) {
        for (int st = 0; st < ST; ++st) mbar_init(&sm.full[st], 1);
        mbar_fence_init();
        tmap_prefetch(&map_a);
        tmap_prefetch(&map_b);
        uint32_t tag = ld_relaxed_u32(&ctrl->epoch) + 1u;
        sm.tag = tag == 0 ? 1u : tag;
        uint32_t ended = 0;
        for (int st = 0; st < ST; ++st) {
            long long id = n_tiles;
            if (!ended) {
                id = grab();
                if (id >= n_tiles) { ended = 1; id = n_tiles; }
            }
            sm.tile_id[st] = id;
            if (id < n_tiles) issue(st, id);
        }
        sm.ended = ended;
    }
    if (misaligned && tid == 0) {
        for (int st = 0; st < ST; ++st) sm.tile_id[st] = n_tiles;
    }
    __syncthreads();

    const uint32_t tag = sm.tag;
    uint32_t phases = 0;                      // bit st: parity of the next completion of stage st

    for (long long k = 0;; ++k) {
        const int st = (int)(k % ST);
        const long long id = sm.tile_id[st];
        if (id >= n_tiles) break;

        if (!mbar_wait_bounded(&sm.full[st], (phases >> st) & 1u, kTmaPolls)) {
            atomicOr(status, kStatusTmaTimeout);
            atomicExch(&ctrl->abort, 1u);
        }
        phases ^= 1u << st;

        long long q, bi, d0;
        decode_tile(id, n_slices, slices_per_batch, q, bi, d0, TD);
        const long long t0 = q * TT;
        const int r0 = s * K;
        const long long rem = L - (t0 + r0);
        const int nv = rem <= 0 ? 0 : (rem >= K ? K : (int)rem);   // valid steps of this thread
        const bool seq_start = (q == 0 && s == 0);                  // holds t = 0 of its channel

        // ---- 2. compose this thread's K steps -----------------------------
        const float *ta = sm.a[st] + r0 * TD + c;
        const float *tb = sm.b[st] + r0 * TD + c;
        float ra[K], rb[K];
#pragma unroll
        for (int j = 0; j < K; ++j) {
            ra[j] = ta[j * TD];
            rb[j] = tb[j * TD];
        }
        if (seq_start) ra[0] = 0.0f;          // h_{-1} = 0: the first slope never matters
        float A = 1.0f, Bv = 0.0f;
#pragma unroll
        for (int j = 0; j < K; ++j) {
            if (j < nv) {
                Bv = fmaf(ra[j], Bv, rb[j]);
                A = ra[j] * A;
            }
        }

        // ---- 3. shuffle scan over the S segments of each channel --------------
        float tA, tB;                          // tile aggregate (valid in threads tid < TD)
        if constexpr (S > 1) {
            sm.segA[s][c] = A;
            sm.segB[s][c] = Bv;
            __syncthreads();
            const int cc = tid / S, ss = tid % S;   // transposed role: lanes walk the segments
            float xA = sm.segA[ss][cc], xB = sm.segB[ss][cc];
#pragma unroll
            for (int off = 1; off < S; off <<= 1) {
                const float uA = __shfl_up_sync(0xffffffffu, xA, off, S);
                const float uB = __shfl_up_sync(0xffffffffu, xB, off, S);
                if (ss >= off) {               // (later) o (earlier)
                    xB = fmaf(xA, uB, xB);
                    xA = xA * uA;
                }
            }
            float eA = __shfl_up_sync(0xffffffffu, xA, 1, S);
            float eB = __shfl_up_sync(0xffffffffu, xB, 1, S);
            if (ss == 0) { eA = 1.0f; eB = 0.0f; }
            sm.preA[ss][cc] = eA;
            sm.preB[ss][cc] = eB;
            if (ss == S - 1) { sm.tileA[cc] = xA; sm.tileB[cc] = xB; }
            __syncthreads();
            tA = sm.tileA[c];
            tB = sm.tileB[c];
        } else {
            tA = A;
            tB = Bv;
        }

        // ---- 4. decoupled look-back, one thread per channel --------------------
        if (tid < TD) {
            const bool publish = (q + 1 < chunks) && (id != silent_tile);
            const long long me = id * TD + c;
            float carry;
            if (q == 0) {
                carry = 0.0f;
            } else {
                long long j = id - n_slices;
                const unsigned long long w = ld_relaxed_u64(&wInc[j * TD + c]);
                if (word_tag(w) == tag) {
                    carry = word_val(w);
                } else {
                    if (publish) {
                        st_relaxed_u64(&wAggA[me], pack_word(tag, tA));
                        st_relaxed_u64(&wAggB[me], pack_word(tag, tB));
                    }
                    float accA = 1.0f, accB = 0.0f;   // composition of tiles j+1 .. id-1
                    long long polls = 0;
                    unsigned int nap = 32;
                    for (;;) {
                        const unsigned long long wi = ld_relaxed_u64(&wInc[j * TD + c]);
                        if (word_tag(wi) == tag) {
                            carry = fmaf(accA, word_val(wi), accB);
                            break;
                        }
                        const unsigned long long wa = ld_relaxed_u64(&wAggA[j * TD + c]);
                        const unsigned long long wb = ld_relaxed_u64(&wAggB[j * TD + c]);
                        if (word_tag(wa) == tag && word_tag(wb) == tag) {
                            accB = fmaf(accA, word_val(wb), accB);   // acc o aggregate(j)
                            accA = accA * word_val(wa);
                            j -= n_slices;
                            if (j < 0) { carry = accB; break; }      // h before the first chunk is 0
                            polls = 0;
                            nap = 32;
                            continue;
                        }
                        if (++polls > spin_limit ||
                            ((polls & 63) == 0 && ld_relaxed_u32(&ctrl->abort) != 0)) {
                            atomicOr(status, kStatusLookbackTimeout);
                            carry = __uint_as_float(0x7fc00000u);  // NaN marks the lost carry
                            break;
                        }
                        __nanosleep(nap);
                        if (nap < 1024) nap <<= 1;
                    }
                }
            }
            if (publish) st_relaxed_u64(&wInc[me], pack_word(tag, fmaf(tA, carry, tB)));
            sm.carry[c] = carry;
        }
        __syncthreads();

        // ---- 5. replay the steps from the carried value, store h ----------------
        const float carry = sm.carry[c];
        float hc;
        if constexpr (S > 1) hc = fmaf(sm.preA[s][c], carry, sm.preB[s][c]);
        else hc = carry;
        const bool dvalid = (d0 + c) < D;
        float *hp = h + ((bi * L + t0 + r0) * D + d0 + c);
#pragma unroll
        for (int j = 0; j < K; ++j) {
            if (j < nv) {
                hc = fmaf(ra[j], hc, rb[j]);
                if (dvalid) hp[(long long)j * D] = hc;
            }
        }
        __syncthreads();                      // stage st and the scratch arrays are free again

        if (tid == 0) {
            long long nid = n_tiles;
            if (!sm.ended && ld_relaxed_u32(&ctrl->abort) != 0) sm.ended = 1;
            if (!sm.ended) {
                nid = grab();
                if (nid >= n_tiles) { sm.ended = 1; nid = n_tiles; }
            }
            sm.tile_id[st] = nid;
            if (nid < n_tiles) issue(st, nid);
        }
    }

    // The last CTA to finish resets the counters and advances the epoch for the next launch.
    __syncthreads();
    if (tid == 0) {
        __threadfence();
        const unsigned int prev = atomicAdd(&ctrl->done, 1u);
        if (prev == gridDim.x - 1) {
            __threadfence();
            atomicExch(&ctrl->tile_counter, 0ull);
            atomicExch(&ctrl->done, 0u);
            atomicExch(&ctrl->abort, 0u);
            atomicAdd(&ctrl->epoch, 1u);
            __threadfence();
        }
    }
}

template <int TD, int TT, int S, int ST>
constexpr ChunkedVariant make_variant() {
    return ChunkedVariant{TD, TT, S, ST, TD * S, sizeof(ChunkSmem<TD, TT, S, ST>)};
}

#define LINREC_CHUNKED_VARIANTS(X) \
    X(128, 64, 4, 2)               \
    X(128, 64, 4, 3)               \
    X(128, 32, 2, 3)               \
    X(256, 32, 2, 2)               \
    X(64, 128, 8, 2)               \
    X(64, 64, 4, 2)                \
    X(64, 64, 4, 3)                \
    X(32, 128, 8, 2)               \
    X(32, 64, 4, 3)

#define LINREC_V_ENTRY(TD, TT, S, ST) make_variant<TD, TT, S, ST>(),
const ChunkedVariant kVariants[] = {LINREC_CHUNKED_VARIANTS(LINREC_V_ENTRY)};
#undef LINREC_V_ENTRY

const void *kernel_of(const ChunkedVariant *v) {
#define LINREC_K_ENTRY(TD, TT, S, ST)                                                        \
    if (v->tile_d == TD && v->tile_t == TT && v->segments == S && v->stages == ST)           \
        return reinterpret_cast<const void *>(&chunked_scan_kernel<TD, TT, S, ST>);
    LINREC_CHUNKED_VARIANTS(LINREC_K_ENTRY)
#undef LINREC_K_ENTRY
    return nullptr;
}

}  // namespace

const ChunkedVariant *chunked_variants(int *count) {
    *count = (int)(sizeof(kVariants) / sizeof(kVariants[0]));
    return kVariants;
}

cudaError_t chunked_ctas_per_sm(const ChunkedVariant *v, int *ctas) {
    const void *fn = kernel_of(v);
    if (!fn) return cudaErrorInvalidValue;
    cudaError_t err = cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)v->smem_bytes);
    if (err != cudaSuccess) return err;
    return cudaOccupancyMaxActiveBlocksPerMultiprocessor(ctas, fn, v->threads, v->smem_bytes);
}

cudaError_t launch_chunked(const ChunkedLaunch &p, cudaStream_t stream) {
    const void *fn = kernel_of(p.variant);
    if (!fn) return cudaErrorInvalidValue;
    cudaError_t err = cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                           (int)p.variant->smem_bytes);
    if (err != cudaSuccess) return err;
    long long L = p.L, D = p.D, spb = p.slices_per_batch, ns = p.n_slices, ch = p.chunks, nt = p.n_tiles;
    long long spin = p.spin_limit, silent = p.silent_tile;
    float *h = p.h;
    Control *ctrl = p.ctrl;
    unsigned long long *words = p.words;
    unsigned int *status = p.status;
    void *args[] = {(void *)&p.map_a, (void *)&p.map_b, &h, &L, &D, &spb, &ns, &ch, &nt,
                    &ctrl, &words, &status, &spin, &silent};
    return cudaLaunchKernel(fn, dim3((unsigned)p.grid), dim3((unsigned)p.variant->threads), args,
                            p.variant->smem_bytes, stream);
}

}  // namespace linrec
