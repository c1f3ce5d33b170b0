// chunked_kernel.cuh -- the TMA-staged chunked path of the linear-recurrence scan:
// the kernel template, instantiated for fp32 storage in chunked.cu and for
// 16-bit storage in chunked16.cu.
//
// h_0 = b_0, h_t = a_t*h_{t-1} + b_t per channel (POPCORNBENCH "Kimi-K2.6 l1_p9",
// problem statement).  The (B, L, D) problem is cut into tiles of TT time steps
// x TD channels of one batch index.  A slice is the TD channels of one batch
// index over all L; its tiles are its time chunks q = 0 .. chunks-1, and tile
// id = q * n_slices + slice.
//
// Per tile, inside one CTA of TD/CPT * S threads (CPT = channels per thread, 1, or
// 2 for 16-bit storage; the results do not depend on it):
//  1. TMA copies the a and b boxes (TT x TD stored elements each) into a
//     shared-memory ring of ST stages; one mbarrier per stage counts the bytes.
//     A stage is refilled as soon as every thread has its tile in registers
//     (after the tile's first barrier), so up to ST + 1 tiles are in flight.
//     Elements are widened to fp32 as threads read them (storage.cuh); all
//     arithmetic and every carry is fp32, and h is rounded once when stored.
//  2. Thread (channel group c, segment s) composes, for each of its channels, its
//     K = TT/S consecutive affine maps x -> a*x + b into one pair (A, B), later
//     map on the left:
//     (a2,b2) o (a1,b1) = (a2*a1, a2*b1 + b2) ("Kimi-K2.6 l1_p9", derivation of
//     the associative operator).  Its a, b values stay in registers.
//  3. A warp-shuffle scan over the S segment pairs of each channel gives every
//     segment its exclusive prefix and the tile its aggregate (A_q, B_q).
//  4. The carry: the h value entering the tile.  Only this running value
//     crosses tile boundaries ("Kimi-K2.6 l1_p9", the running_h carry).  It is
//     defined as the chain H_q = A_q * H_{q-1} + B_q over the slice's tiles
//     (H before the first chunk = 0), which both modes below evaluate with the
//     same fma sequence, so they return the same bits.
//       slice-owner mode: a CTA owns whole slices (static round-robin) and
//         walks their chunks in order; the carry stays in a register.
//       look-back mode (few slices, long L): tiles of a slice run on different
//         CTAs; each publishes its aggregate, walks back over earlier tiles of
//         its slice to the nearest inclusive value (S lanes per channel, a
//         window of S*R tiles per round trip), replays the chain forward from
//         it and publishes its own inclusive value.
//       two-pass mode (few slices, long L; three launches): a reduce launch
//         writes every tile's aggregate, the library scans those aggregates
//         (a problem 1/TT the size, with these same kernels), and an apply
//         launch gives each tile the inclusive value of the tile before it.
//         Tiles are independent in both launches; the apply launch visits
//         them in reverse order so the inputs the reduce launch read last
//         are still in L2.
//       blocks mode (few slices, long L; one launch, a separate instantiation,
//         BM = true): a block is G consecutive tiles of a slice, taken in order
//         from a counter.  The CTA composes the block's tiles into one map
//         (reduce pass, nothing stored), gets the h entering the block by the
//         same decoupled look-back over block maps, then takes the same G
//         tiles again (apply pass: re-read, mostly from L2) and finishes them
//         as slice-owner mode does.  HBM traffic lies between the 12 bytes
//         (fp32) per element of one pass and the 20 of two-pass, by how much
//         of the re-read L2 still holds.
//  5. Every thread replays its K steps from h_in = A_prefix * carry + B_prefix
//     and stores h.
//
// In look-back mode tile ids come from an atomic counter, taken in the order
// CTAs start on them, so every predecessor of a tile was handed to a CTA that
// is running or done.  Every wait is bounded; on expiry the kernel records an
// error bit in the status word and carries on with NaN.
#pragma once

#include "checked.cuh"
#include "kernels.cuh"
#include "lookback.cuh"
#include "ptx.cuh"
#include "storage.cuh"

namespace linrec {

namespace {

constexpr uint32_t kTmaPolls = 1u << 22;   // ~1 s of polls with back-off

// Where a ring stage's tile sits: decoded once by the thread that loads it.
struct TileCoord {
    long long id;                       // tile id (>= n_tiles: no tile, the CTA is done)
    int q;                              // time chunk
    int bi;                             // batch index
    int d0;                             // first channel
    int flags;                          // blocks mode: kApplyPass | kFirstOfPass | kLastOfPass
};
constexpr int kApplyPass = 1, kFirstOfPass = 2, kLastOfPass = 4;

// A thread's K steps of a and b for its CPT adjacent channels, held in registers
// from the compose to the replay; a(j, i) and b(j, i) are step j of channel i.
// fp32 storage keeps floats.  16-bit storage keeps the stored words and widens each
// one (exactly) where it is used: with one channel per thread two steps share a
// 32-bit register; with two channels a register holds both channels of a step, as
// shared memory does, so one 32-bit load fetches it.  Either way a 16-bit tile of
// twice the elements costs the registers of an fp32 tile.
template <int DT, int K, int CPT,
          int KIND = (Storage<DT>::bytes == 4 || (CPT == 1 && K % 2 != 0)) ? 0 : (CPT == 1 ? 1 : 2)>
struct TileRegs;

template <int DT, int K>
struct TileRegs<DT, K, 1, 0> {
    float a_[K], b_[K];
    template <typename E>
    __device__ __forceinline__ void load(const E *ta, const E *tb, int stride) {
#pragma unroll
        for (int j = 0; j < K; ++j) {
            a_[j] = Storage<DT>::get(ta[j * stride]);
            b_[j] = Storage<DT>::get(tb[j * stride]);
        }
    }
    __device__ __forceinline__ float a(int j, int) const { return a_[j]; }
    __device__ __forceinline__ float b(int j, int) const { return b_[j]; }
    __device__ __forceinline__ void zero_a0() { a_[0] = 0.0f; }
};

__device__ __forceinline__ unsigned short half_of(uint32_t w, int hi) {
    return (unsigned short)(hi ? (w >> 16) : (w & 0xffffu));
}

template <int DT, int K>
struct TileRegs<DT, K, 1, 1> {
    uint32_t a_[K / 2], b_[K / 2];            // step 2i in the low half, step 2i + 1 in the high half
    template <typename E>
    __device__ __forceinline__ void load(const E *ta, const E *tb, int stride) {
#pragma unroll
        for (int i = 0; i < K / 2; ++i) {
            a_[i] = (uint32_t)ta[2 * i * stride] | ((uint32_t)ta[(2 * i + 1) * stride] << 16);
            b_[i] = (uint32_t)tb[2 * i * stride] | ((uint32_t)tb[(2 * i + 1) * stride] << 16);
        }
    }
    __device__ __forceinline__ float a(int j, int) const { return Storage<DT>::get(half_of(a_[j >> 1], j & 1)); }
    __device__ __forceinline__ float b(int j, int) const { return Storage<DT>::get(half_of(b_[j >> 1], j & 1)); }
    __device__ __forceinline__ void zero_a0() { a_[0] &= 0xffff0000u; }   // the word 0 is +0 in both formats
};

template <int DT, int K>
struct TileRegs<DT, K, 2, 2> {
    uint32_t a_[K], b_[K];                    // step j: the first channel in the low half
    template <typename E>
    __device__ __forceinline__ void load(const E *ta, const E *tb, int stride) {
#pragma unroll
        for (int j = 0; j < K; ++j) {
            a_[j] = *reinterpret_cast<const uint32_t *>(ta + j * stride);
            b_[j] = *reinterpret_cast<const uint32_t *>(tb + j * stride);
        }
    }
    __device__ __forceinline__ float a(int j, int i) const { return Storage<DT>::get(half_of(a_[j], i)); }
    __device__ __forceinline__ float b(int j, int i) const { return Storage<DT>::get(half_of(b_[j], i)); }
    __device__ __forceinline__ void zero_a0() { a_[0] = 0u; }
};

// A thread's CPT adjacent floats of a shared row (8-byte aligned for CPT = 2).
template <int CPT>
__device__ __forceinline__ void st_group(float *p, const float (&v)[CPT]) {
    if constexpr (CPT == 1) *p = v[0];
    else *reinterpret_cast<float2 *>(p) = make_float2(v[0], v[1]);
}
template <int CPT>
__device__ __forceinline__ void ld_group(const float *p, float (&v)[CPT]) {
    if constexpr (CPT == 1) {
        v[0] = *p;
    } else {
        const float2 x = *reinterpret_cast<const float2 *>(p);
        v[0] = x.x;
        v[1] = x.y;
    }
}
// h of a thread's CPT adjacent channels at one step, rounded once each.
template <int DT, int CPT>
__device__ __forceinline__ void st_h(typename Storage<DT>::raw *p, const float (&v)[CPT]) {
    if constexpr (CPT == 1) *p = Storage<DT>::put(v[0]);
    else *reinterpret_cast<uint32_t *>(p) = Storage<DT>::put2(v[0], v[1]);
}

template <typename E, int TD, int TT, int S, int ST>
struct __align__(128) ChunkSmem {
    E a[ST][TT * TD];                   // stored elements, as the boxes arrive
    E b[ST][TT * TD];
    // Per-segment pairs, then their exclusive prefixes, and the h entering the tile:
    // two copies, used by alternate tiles (see the barriers in the tile loop).  A row
    // holds TD + 32/S floats: a warp of the transposed role reads 32/S channels x S
    // segments, which the padding spreads over all 32 banks.
    float segA[2][S][TD + 32 / S], segB[2][S][TD + 32 / S];
    float carry[2][TD];
    uint64_t full[ST];                  // one mbarrier per ring stage
    TileCoord tile[ST];                 // tile loaded into each stage
    uint32_t tag;                       // look-back tag of this launch
};

// FM >= 0 compiles the one carry mode FM (kModeOwn, kModeLookback, kModeReduce or kModeApply;
// `mode` must equal it): none of the other modes' code is in the kernel, which then needs fewer
// registers and instructions.  FM = -1 takes the mode at run time.
template <int DT, int TD, int TT, int S, int ST, int CPT, bool BM = false, int FM = -1>
__global__ void __launch_bounds__(TD / CPT * S, (TD / CPT * S >= 512) ? 1 : 2)
chunked_scan_kernel(const __grid_constant__ CUtensorMap map_a,
                    const __grid_constant__ CUtensorMap map_b,
                    typename Storage<DT>::raw *__restrict__ h,
                    const long long L, const long long D,
                    const long long slices_per_batch, const long long n_slices,
                    const long long chunks, const long long n_tiles,
                    const int mode,              // kModeLookback, kModeOwn, kModeReduce, kModeApply;
                                                 // kModeBlocks (BM instantiations only)
                    const int group,             // blocks mode: tiles per block (G)
                    Control *__restrict__ ctrl, unsigned long long *__restrict__ words,
                    unsigned int *__restrict__ status,
                    const long long spin_limit, const long long silent_tile,
                    const float *h_init, float *h_last)
{
    constexpr int K = TT / S;                 // time steps per thread
    constexpr int R = (S >= 4) ? 16 / S : 4;  // look-back: predecessors per lane
    using E = typename Storage<DT>::raw;      // stored element type
    constexpr uint32_t kStageBytes = 2u * TT * TD * sizeof(E);
    const bool own = FM >= 0 ? FM == kModeOwn : mode == kModeOwn;
    const bool lookback = FM >= 0 ? FM == kModeLookback : mode == kModeLookback;
    const bool reduce = FM >= 0 ? FM == kModeReduce : mode == kModeReduce;
    const bool apply = FM >= 0 ? FM == kModeApply : mode == kModeApply;
    const bool blocks = FM < 0 && BM && mode == kModeBlocks;
    // speculative mode (copies compiled for it alone): `group` segments of each sequence, seen as
    // batch rows bi = b * group + segment of a (B * group, L / group, D) view of the same memory
    const bool spec = FM == kModeSpec;        // segments scanned from 0, their maps published
    const bool repair = FM == kModeRepair;    // the tiles left unstored, from the true carry
    const bool chained = lookback || blocks;  // tiles or blocks joined by the look-back words
    // blocks mode: blocks per slice, and all blocks (block id = block index * n_slices + slice)
    const long long bps = BM ? (chunks + group - 1) / group : 0;
    const long long n_blocks = bps * n_slices;
    // two-pass mode: per-tile aggregates and the scanned inclusive values, indexed [tile id][channel],
    // and each channel's starting state, indexed [slice][channel]
    float *const tileA = reinterpret_cast<float *>(words);
    float *const tileB = tileA + n_tiles * TD;
    const float *const tileH = tileB + n_tiles * TD;
    float *const tileX = tileB + 2 * n_tiles * TD;
    constexpr int TC = TD / CPT;              // channel groups of a tile
    static_assert(TT % S == 0 && TD % 32 == 0 && (32 % S) == 0 && S >= 2 && ST >= 2, "tile shape");
    // two channels per thread: 16-bit storage, shared rows of an even number of floats
    static_assert(CPT == 1 || (CPT == 2 && Storage<DT>::bytes == 2 && (32 / S) % 2 == 0), "channels per thread");
    using Smem = ChunkSmem<E, TD, TT, S, ST>;
    extern __shared__ __align__(128) unsigned char smem_raw[];
    Smem &sm = *reinterpret_cast<Smem *>(smem_raw);

    pdl_wait();   // launched as a programmatic dependent: nothing before it is touched yet

    const int tid = threadIdx.x;
    const int c = tid % TC;                   // channel group: channels CPT*c .. CPT*c + CPT-1 of the tile
    const int s = tid / TC;                   // segment within the tile
    const int cc = tid / S;                   // transposed role: channels cc, cc + TC, ... (one per
    const int ss = tid % S;                   // group), and the segment / look-back window lane
    const int gbase = (tid & 31) & ~(S - 1);  // first lane of this channel's group in the warp

    // look-back words, [unit][channel]: units are tiles, or blocks in blocks mode
    const long long n_units = blocks ? n_blocks : n_tiles;
    // extents for the index-checked build: elements of h, and of h_init / h_last
    const long long n_h = (n_slices / slices_per_batch) * L * D;
    const long long n_state = (n_slices / slices_per_batch) * D / ((spec || repair) ? group : 1);
    // speculative mode: each slice's map over its segment, [slice][channel] pairs (A, B)
    float *const segmap = reinterpret_cast<float *>(words);
    const long long n_segmap = 2 * n_slices * TD;
    unsigned long long *const wAggA = words;
    unsigned long long *const wAggB = words + n_units * TD;
    unsigned long long *const wInc = words + 2 * n_units * TD;

    // (thread 0) record stage st's tile and start its two box copies.
    auto issue = [&](int st, long long id, long long q, long long slice, int flags) {
        const long long bi = slice / slices_per_batch;
        const int d0 = (int)((slice - bi * slices_per_batch) * TD);
        sm.tile[st] = TileCoord{id, (int)q, (int)bi, d0, flags};
        mbar_arrive_expect_tx(&sm.full[st], kStageBytes);
        tma_load_3d(sm.a[st], &map_a, &sm.full[st], d0, (int)(q * TT), (int)bi);
        tma_load_3d(sm.b[st], &map_b, &sm.full[st], d0, (int)(q * TT), (int)bi);
    };
    auto finish = [&](int st) { sm.tile[st] = TileCoord{n_tiles, 0, 0, 0, 0}; };
    // (thread 0) the CTA's next tile.  Slice-owner mode: slices blockIdx.x,
    // blockIdx.x + gridDim.x, ... each walked from chunk 0 to chunks-1, tracked
    // in (own_slice, own_q).  Look-back mode: the next id from the tile counter.
    long long own_slice = blockIdx.x, own_q = 0, own_m = 0;
    long long stop_slice = -1;                // (speculative, repair; every thread) the slice whose slope
                                              // product has reached 0: from there on it stays decided
    // (thread 0, blocks mode) the block being walked, its pass, the next tile of the pass, its tiles
    long long bm_blk = -1;
    int bm_pass = 0, bm_g = 0, bm_cnt = 0;
    auto next_tile = [&](long long &q, long long &slice, int &flags) -> long long {
        flags = 0;
        if constexpr (BM) {
            if (blocks) {
                // a block's G tiles twice (reduce pass, then apply pass), then the next block
                if (bm_blk < 0 || (bm_pass == 1 && bm_g == bm_cnt)) {
                    const long long b = (long long)atomicAdd(&ctrl->tile_counter, 1ull);
                    if (b >= n_blocks) return n_tiles;
                    bm_blk = b;
                    bm_pass = 0;
                    bm_g = 0;
                    const long long left = chunks - (b / n_slices) * group;
                    bm_cnt = left < group ? (int)left : group;
                } else if (bm_g == bm_cnt) {
                    bm_pass = 1;
                    bm_g = 0;
                }
                const long long bq = bm_blk / n_slices;
                slice = bm_blk - bq * n_slices;
                q = bq * group + bm_g;
                flags = (bm_pass ? kApplyPass : 0) | (bm_g == 0 ? kFirstOfPass : 0) |
                        (bm_g == bm_cnt - 1 ? kLastOfPass : 0);
                ++bm_g;
                return q * n_slices + slice;
            }
        }
        if (reduce || apply) {                // independent tiles, static round-robin
            const long long k = blockIdx.x + (own_m++) * (long long)gridDim.x;
            if (k >= n_tiles) return n_tiles;
            const long long id = apply ? n_tiles - 1 - k : k;
            q = id / n_slices;
            slice = id - q * n_slices;
            return id;
        }
        if (own || spec || repair) {
            for (;;) {
                if (own_slice >= n_slices) return n_tiles;
                // repair: no first segment (the speculative launch stored it), and nothing of a
                // slice after its slopes' product reached 0 (the speculative launch stored the rest)
                if (repair && (((own_slice / slices_per_batch) % group) == 0 ||
                               (own_q > 0 && own_slice == stop_slice))) {
                    own_q = 0;
                    own_slice += gridDim.x;
                    continue;
                }
                q = own_q;
                slice = own_slice;
                if (repair && own_q == 0) flags |= kFirstOfPass;
                if (++own_q == chunks) { own_q = 0; own_slice += gridDim.x; }
                return q * n_slices + slice;
            }
        }
        const long long id = (long long)atomicAdd(&ctrl->tile_counter, 1ull);
        if (id >= n_tiles) return n_tiles;
        q = id / n_slices;
        slice = id - q * n_slices;
        return id;
    };

    // TMA writes whole boxes at 128-byte aligned shared addresses; the layout
    // guarantees it when the dynamic window is aligned, so check that once.
    const bool misaligned = (smem_u32(smem_raw) & 127u) != 0;
    if (tid == 0) {
        long long first = n_tiles;
        if (misaligned) {
            atomicOr(status, kStatusTmaTimeout);
            if (chained) atomicExch(&ctrl->abort, 1u);
        } else {
            for (int st = 0; st < ST; ++st) mbar_init(&sm.full[st], 1);
            mbar_fence_init();
            tmap_prefetch(&map_a);
            tmap_prefetch(&map_b);
            if (chained) {
                sm.tag = tag_of(ld_relaxed_u32(&ctrl->epoch));
            }
            // One tile at launch: in look-back mode tiles are then taken in the order
            // CTAs start on them, so a tile's predecessors are never parked in another
            // CTA's ring behind later work.
            long long q = 0, slice = 0;
            int flags = 0;
            first = next_tile(q, slice, flags);
            if (first < n_tiles) issue(0, first, q, slice, flags);
        }
        if (first >= n_tiles) finish(0);
    }
    __syncthreads();

    const uint32_t tag = chained ? sm.tag : 0u;
    uint32_t phases = 0;                      // bit st: parity of the next completion of stage st
    long long next_fill = 1;                  // (thread 0) next ring slot to fill
    bool ended = sm.tile[0].id >= n_tiles;    // (thread 0) no more tiles to take
    long long ahead = -1, ahead_q = 0, ahead_slice = 0;   // (thread 0, look-back) tile taken early
    uint32_t abort_seen = 0;                  // (thread 0, look-back) abort word, read one iteration early
    float run[CPT];                           // (slice-owner, ss == 0) inclusive values of the last tile
    float bA[CPT], bB[CPT];                   // (blocks mode, reduce pass) the block's map so far
    float runA[CPT];                          // (speculative, repair; ss == 0) slope product of the segment
                                              // through the current tile
#pragma unroll
    for (int i = 0; i < CPT; ++i) { run[i] = 0.0f; bA[i] = 1.0f; bB[i] = 0.0f; runA[i] = 1.0f; }

    // (thread 0) fill ring slots up to (not including) slot `limit`; slot n goes to stage n % ST.
    // In look-back mode the next tile id is taken one fill ahead, so the atomic's
    // round trip overlaps a tile's work instead of delaying the next copy.
    auto refill = [&](long long limit) {
        if (!ended && abort_seen != 0) {
            ended = true;
            finish((int)(next_fill % ST));
        }
        while (!ended && next_fill < limit) {
            const int s2 = (int)(next_fill % ST);
            long long nq = ahead_q, nslice = ahead_slice;
            int nflags = 0;
            const long long nid = ahead >= 0 ? ahead : next_tile(nq, nslice, nflags);
            ahead = -1;
            if (nid >= n_tiles) {
                ended = true;
                finish(s2);
            } else {
                issue(s2, nid, nq, nslice, nflags);
            }
            ++next_fill;
        }
        if (lookback) {
            int unused = 0;
            if (!ended && ahead < 0) ahead = next_tile(ahead_q, ahead_slice, unused);
        }
        if (chained) abort_seen = ld_relaxed_u32(&ctrl->abort);
    };

    for (long long k = 0;; ++k) {
        const int st = (int)(k % ST);
        const TileCoord tc = sm.tile[st];
        const long long id = tc.id;
        if (id >= n_tiles) break;

        // The first iteration fills the rest of the ring before it waits (the abort
        // word is still unread, so no slot is closed here while others read this
        // stage's TileCoord).  After that every stage is refilled as soon as its
        // tile has been read, below.
        if (tid == 0 && k == 0) refill(ST);

        if (!mbar_wait_bounded(&sm.full[st], (phases >> st) & 1u, kTmaPolls)) {
            atomicOr(status, kStatusTmaTimeout);
            if (chained) atomicExch(&ctrl->abort, 1u);
        }
        phases ^= 1u << st;

        const long long q = tc.q, bi = tc.bi, d0 = tc.d0;
        const long long t0 = q * TT;
        const int r0 = s * K;
        const long long rem = L - (t0 + r0);
        const int nv = rem <= 0 ? 0 : (rem >= K ? K : (int)rem);   // valid steps of this thread
        const bool seq_start = (q == 0 && s == 0);                  // holds t = 0 of its channel
        // the batch row of h_init / h_last (speculative mode: the sequence, not its segment)
        const long long sbi = (spec || repair) ? bi / group : bi;
        // repair: a tile loaded ahead of its slice's stop stores nothing (the speculative launch did)
        const bool skip = repair && (id - q * n_slices) == stop_slice;
        bool live = false;                  // (speculative, repair; ss == 0) a slope product not yet 0

        // ---- 2. compose this thread's K steps -----------------------------------
        const E *ta = sm.a[st] + r0 * TD + CPT * c;
        const E *tb = sm.b[st] + r0 * TD + CPT * c;
        TileRegs<DT, K, CPT> r;
        r.load(ta, tb, TD);
        // h_{-1} = 0: the first slope never matters (speculative mode: only at the real start; a
        // later segment starts from 0 but its first slope belongs to the segment's map)
        if (seq_start && !h_init && ((!spec && !repair) || (bi % group) == 0)) r.zero_a0();
        float A[CPT], Bv[CPT];
#pragma unroll
        for (int i = 0; i < CPT; ++i) { A[i] = 1.0f; Bv[i] = 0.0f; }
#pragma unroll
        for (int j = 0; j < K; ++j) {
            if (j < nv) {
#pragma unroll
                for (int i = 0; i < CPT; ++i) {
                    Bv[i] = fmaf(r.a(j, i), Bv[i], r.b(j, i));
                    A[i] = r.a(j, i) * A[i];
                }
            }
        }
        float (&segA)[S][TD + 32 / S] = sm.segA[k & 1];
        float (&segB)[S][TD + 32 / S] = sm.segB[k & 1];
        float (&carry_in)[TD] = sm.carry[k & 1];
        st_group<CPT>(&segA[s][CPT * c], A);
        st_group<CPT>(&segB[s][CPT * c], Bv);
        __syncthreads();
        // Every thread now holds this tile's a and b in registers: stage st is free,
        // so its next tile (slot k + ST) starts copying while this one is finished.
        if (tid == 0) refill(k + ST + 1);

        // ---- 3. shuffle scan over the S segment pairs of each channel -----------
        float tA[CPT], tB[CPT];                 // the tile's aggregate of each channel
#pragma unroll
        for (int i = 0; i < CPT; ++i) {
            const int ch = cc + i * TC;
            float xA = segA[ss][ch], xB = segB[ss][ch];
#pragma unroll
            for (int off = 1; off < S; off <<= 1) {
                const float uA = __shfl_up_sync(kFull, xA, off, S);
                const float uB = __shfl_up_sync(kFull, xB, off, S);
                if (ss >= off) {              // (later) o (earlier)
                    xB = fmaf(xA, uB, xB);
                    xA = xA * uA;
                }
            }
            float eA = __shfl_up_sync(kFull, xA, 1, S);
            float eB = __shfl_up_sync(kFull, xB, 1, S);
            if (ss == 0) { eA = 1.0f; eB = 0.0f; }
            segA[ss][ch] = eA;                // same slot this thread read: no other reader
            segB[ss][ch] = eB;
            tA[i] = __shfl_sync(kFull, xA, S - 1, S);
            tB[i] = __shfl_sync(kFull, xB, S - 1, S);
        }

        // ---- 4. the carry entering the tile ---------------------------------------
#pragma unroll
        for (int i = 0; i < CPT; ++i) {
            const int ch = cc + i * TC;
            // h before the first chunk: the carried-in state, or 0.
            const float h_before = (h_init && d0 + ch < D && inside(h_init + sbi * D + d0 + ch, h_init, n_state))
                                       ? h_init[sbi * D + d0 + ch]
                                       : 0.0f;
            if (spec) {
                // a segment's chain from 0 (the first segment's from the carried-in state); at its
                // end the segment's map (slope product, h) goes out, the first segment's with slope 0.
                // A tile is exact, and stored, once the slope product before it is 0.
                if (ss == 0) {
                    const bool first_seg = (bi % group) == 0;
                    const float carry = (q == 0) ? (first_seg ? h_before : 0.0f) : run[i];
                    run[i] = fmaf(tA[i], carry, tB[i]);
                    live = live || q == 0 || runA[i] != 0.0f;
                    runA[i] = (q == 0) ? tA[i] : tA[i] * runA[i];
                    carry_in[ch] = carry;
                    if (q + 1 == chunks) {
                        const long long at = ((id - q * n_slices) * TD + ch) * 2;
                        if (inside(segmap + at, segmap, n_segmap, false, 8)) {
                            segmap[at] = first_seg ? 0.0f : runA[i];
                            segmap[at + 1] = run[i];
                        }
                    }
                }
            } else if (repair) {
                // the tiles the speculative launch left unstored, from the true h entering the
                // segment, up to the first tile after which the slope product is 0 in every channel
                // and the carry finite (0 * NaN is NaN: a NaN carried in reaches every later h, so
                // the tiles the speculative launch stored are then written again)
                float hin = 0.0f;
                if (tc.flags & kFirstOfPass) {   // the same for the whole CTA
                    // the maps of segments 0 .. g-1 of this sequence and channel slice, in order
                    // (later on the left); lane ss composes its part of them, kSpecParts loads
                    // in flight a round, and the shuffle scan joins the parts.  The first map's
                    // slope is 0, so the offset is that h.
                    const long long slice = id - q * n_slices;
                    const long long g = bi % group;
                    const long long base = slice - g * slices_per_batch;   // the first segment's slice
                    const int part = (int)((g + S - 1) / S);
                    float xA = 1.0f, xB = 0.0f;
                    for (int j0 = 0; j0 < part; j0 += kSpecParts) {
                        float mA[kSpecParts], mB[kSpecParts];
#pragma unroll
                        for (int j = 0; j < kSpecParts; ++j) {
                            const long long sj = (long long)ss * part + j0 + j;
                            const long long at = ((base + sj * slices_per_batch) * TD + ch) * 2;
                            const bool ok = j0 + j < part && sj < g && inside(segmap + at, segmap, n_segmap, false, 8);
                            mA[j] = ok ? segmap[at] : 1.0f;
                            mB[j] = ok ? segmap[at + 1] : 0.0f;
                        }
#pragma unroll
                        for (int j = 0; j < kSpecParts; ++j) {
                            xB = fmaf(mA[j], xB, mB[j]);
                            xA = mA[j] * xA;
                        }
                    }
#pragma unroll
                    for (int off = 1; off < S; off <<= 1) {
                        const float uA = __shfl_up_sync(kFull, xA, off, S);
                        const float uB = __shfl_up_sync(kFull, xB, off, S);
                        if (ss >= off) {
                            xB = fmaf(xA, uB, xB);
                            xA = xA * uA;
                        }
                    }
                    hin = __shfl_sync(kFull, xB, S - 1, S);
                }
                if (ss == 0) {
                    const float carry = (q == 0) ? hin : run[i];
                    run[i] = fmaf(tA[i], carry, tB[i]);
                    runA[i] = (q == 0) ? tA[i] : tA[i] * runA[i];
                    live = live || runA[i] != 0.0f || !isfinite(run[i]);
                    carry_in[ch] = carry;
                }
            } else if (own) {
                if (ss == 0) {
                    const float carry = (q == 0) ? h_before : run[i];
                    run[i] = fmaf(tA[i], carry, tB[i]);
                    carry_in[ch] = carry;
                }
            } else if (reduce) {
                // the tile's map; the first chunk's absorbs the carried-in state, so the scan of
                // these maps from 0 is the chain of inclusive values
                if (ss == 0) {
                    if (inside(tileA + id * TD + ch, tileA, n_tiles * TD)) tileA[id * TD + ch] = (q == 0) ? 0.0f : tA[i];
                    if (inside(tileB + id * TD + ch, tileB, n_tiles * TD))
                        tileB[id * TD + ch] = (q == 0) ? fmaf(tA[i], h_before, tB[i]) : tB[i];
                    // kept for the apply launch: h_last may be the same buffer as h_init, and the
                    // apply launch writes it while other tiles still need the starting state
                    if (q == 0 && inside(tileX + id * TD + ch, tileX, n_slices * TD)) tileX[id * TD + ch] = h_before;
                }
            } else if (apply) {
                if (ss == 0)
                    carry_in[ch] = (q == 0) ? (inside(tileX + id * TD + ch, tileX, n_slices * TD) ? tileX[id * TD + ch] : 0.0f)
                                            : (inside(tileH + (id - n_slices) * TD + ch, tileH, n_tiles * TD)
                                                   ? tileH[(id - n_slices) * TD + ch]
                                                   : 0.0f);
            } else if (blocks) {
                if (tc.flags & kApplyPass) {
                    // as slice-owner mode, from the h entering the block (left in run by the reduce pass)
                    if (ss == 0) {
                        const float carry = run[i];
                        run[i] = fmaf(tA[i], carry, tB[i]);
                        carry_in[ch] = carry;
                    }
                } else {
                    // the block's map, later tile on the left; every lane of the group holds it
                    if (tc.flags & kFirstOfPass) {
                        bA[i] = tA[i];
                        bB[i] = tB[i];
                    } else {
                        bB[i] = fmaf(tA[i], bB[i], tB[i]);
                        bA[i] = tA[i] * bA[i];
                    }
                    if (tc.flags & kLastOfPass) {   // uniform over the CTA: the look-back's ballots
                        const long long bq = q / group;
                        const long long bid = bq * n_slices + bi * slices_per_batch + d0 / TD;
                        const bool publish = (bq + 1 < bps) && (bid != silent_tile);
                        float carry = h_before;
                        if (bq > 0)
                            carry = lookback_carry<S, R>(bid, n_slices, TD, ch, ss, gbase, tag, publish, bA[i],
                                                         bB[i], h_before, wAggA, wAggB, wInc, n_units * TD, ctrl,
                                                         status, spin_limit);
                        if (ss == 0) {
                            if (publish && inside(wInc + bid * TD + ch, wInc, n_units * TD))
                                st_relaxed_u64(&wInc[bid * TD + ch], pack_word(tag, fmaf(bA[i], carry, bB[i])));
                            run[i] = carry;
                        }
                    }
                }
            } else {
                const bool publish = (q + 1 < chunks) && (id != silent_tile);
                float carry = h_before;
                if (q > 0)
                    carry = lookback_carry<S, R>(id, n_slices, TD, ch, ss, gbase, tag, publish, tA[i], tB[i],
                                                 h_before, wAggA, wAggB, wInc, n_units * TD, ctrl, status,
                                                 spin_limit);
                if (ss == 0) {
                    if (publish && inside(wInc + id * TD + ch, wInc, n_units * TD))
                        st_relaxed_u64(&wInc[id * TD + ch], pack_word(tag, fmaf(tA[i], carry, tB[i])));
                    carry_in[ch] = carry;
                }
            }
        }
        // Once the slope product is exactly 0 in every channel of the slice, the true carry no
        // longer reaches h: the rest of the segment's speculative h is exact.  The two launches
        // take the same products of the same tiles, so they draw the line at the same tile, and
        // neither goes back on it (a later non-finite slope would turn the product's 0 into NaN).
        bool defer = false;                     // (speculative) the tile is left to the repair launch
        if (spec) {
            const long long sl = id - q * n_slices;
            if (!__syncthreads_or(live)) stop_slice = sl;
            defer = stop_slice != sl && (bi % group) != 0;
        } else if (repair) {
            if (!__syncthreads_or(live)) stop_slice = id - q * n_slices;
        } else {
            __syncthreads();
        }

        // ---- 5. replay the steps from the carried value, store h -----------------
        float hc[CPT], pA[CPT], pB[CPT];
        ld_group<CPT>(&segA[s][CPT * c], pA);
        ld_group<CPT>(&segB[s][CPT * c], pB);
        ld_group<CPT>(&carry_in[CPT * c], hc);
#pragma unroll
        for (int i = 0; i < CPT; ++i) hc[i] = fmaf(pA[i], hc[i], pB[i]);
        // (D is even when CPT = 2, so a group is inside D or wholly past it)
        const bool stores = !reduce && !(blocks && !(tc.flags & kApplyPass)) && !skip && !defer;
        if (stores && (d0 + CPT * c) < D) {
            E *hp = h + ((bi * L + t0 + r0) * D + d0 + CPT * c);
            if (nv == K) {
#pragma unroll
                for (int j = 0; j < K; ++j) {
#pragma unroll
                    for (int i = 0; i < CPT; ++i) hc[i] = fmaf(r.a(j, i), hc[i], r.b(j, i));
                    if (inside(hp + (long long)j * D, h, n_h, true, CPT * (long long)sizeof(E)))
                        st_h<DT, CPT>(hp + (long long)j * D, hc);
                }
            } else {
#pragma unroll
                for (int j = 0; j < K; ++j) {
                    if (j < nv) {
#pragma unroll
                        for (int i = 0; i < CPT; ++i) hc[i] = fmaf(r.a(j, i), hc[i], r.b(j, i));
                        if (inside(hp + (long long)j * D, h, n_h, true, CPT * (long long)sizeof(E)))
                            st_h<DT, CPT>(hp + (long long)j * D, hc);
                    }
                }
            }
            // the thread holding t = L-1 hands the state out (speculative mode: of the last segment)
            if (h_last && nv > 0 && t0 + r0 + nv == L && (!(spec || repair) || (bi % group) == group - 1)) {
#pragma unroll
                for (int i = 0; i < CPT; ++i)
                    if (inside(h_last + sbi * D + d0 + CPT * c + i, h_last, n_state, true))
                        h_last[sbi * D + d0 + CPT * c + i] = hc[i];
            }
        }
        // No barrier here.  Stage st was last read before this tile's first
        // barrier, after which thread 0 refilled it; its TileCoord was read into
        // registers at the top of the iteration.  The next tile writes the other
        // copy of segA / segB / carry; the one after it writes this copy again
        // only after two more barriers, which every thread reaches after
        // finishing this tile.
    }

    // This CTA's tiles are done: the launch that follows may be scheduled (it waits
    // for this whole grid before it touches memory).  Not earlier: its CTAs would take
    // slots while this grid still runs (measured 3 % slower on (32, 4096, 256)).
    pdl_release();

    // Look-back and blocks modes: the last CTA to finish resets the counters and
    // advances the epoch for the next launch on this workspace.
    if (chained) {
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

template <int DT, int TD, int TT, int S, int ST, int CPT, bool BM = false>
constexpr ChunkedVariant make_variant() {
    return ChunkedVariant{TD, TT, S, ST, TD / CPT * S, sizeof(ChunkSmem<typename Storage<DT>::raw, TD, TT, S, ST>),
                          (int)sizeof(typename Storage<DT>::raw), CPT, BM ? 1 : 0};
}

}  // namespace

}  // namespace linrec
