// chain.cu -- chain mode of the chunked path, for few long channel slices: one
// launch that reads a and b and writes h once (12 bytes per fp32 element).
//
// The carry of tile q of a slice is H_{q-1}, where H_q = A_q * H_{q-1} + B_q is the
// chain of the slice's tile maps (A_q, B_q) from H_{-1} = the carried-in state or 0
// ("Kimi-K2.6 l1_p9", the running_h carry: only the running h crosses a chunk).
// Slice-owner mode walks that chain in one CTA; here it is split by role:
//
//  - Worker CTAs take tiles round-robin, in order, and keep one tile ahead:
//    iteration k composes tile k as soon as its boxes land (step 2 and 3 of the
//    chunked kernel: per-thread maps, then the shuffle scan over segments) and
//    publishes its map (A, B) at once; then it takes the carry of tile k-1, whose
//    map went out one iteration earlier, replays tile k-1 from it and stores h.
//    The ring stage of tile k is held from its compose until its a and b are moved
//    into registers for the next iteration's replay, so the ring has one more
//    stage than the slice-owner kernel's.
//  - Resolver CTAs (the first n_res of the grid) walk the chain, which is
//    independent per channel.  A group of warps serves some channels of one
//    slice: while loader warps read the published maps of the next window of
//    tiles, one warp folds the usable prefix of the current window into H in
//    tile order (lane = channel) and publishes every H_q as it makes it.
//
// Both roles evaluate H_q = fma(A_q, H_{q-1}, B_q) in tile order, as slice-owner
// mode does, so the results are the same bits.  The launch is cooperative: a
// worker waits for a resolver, so every CTA must be resident at once.  All words
// carry the launch's epoch tag and validate themselves; every wait is bounded and,
// when it runs out, records a status bit, sets the abort word and yields NaN.
#include "chunked_kernel.cuh"

namespace linrec {

namespace {

constexpr int kChainLoads = 8;   // loads (of 32 lanes) a resolver loader issues per window
constexpr int kChainStrideMax = 8;   // the largest stride of published H values
// The stride the resolver publishes H at: every 8th chunk (measured on GB300 against every
// chunk: (1, 1048576, 64) 717 -> 569 us; the maps a worker folds itself cost little).
constexpr int kChainStride = 8;

// What a resolver CTA keeps in shared memory (it overlays the workers' ring): two
// windows of maps per group of warps, [buffer][tile * channels of the group + channel].
template <int NW>
struct ChainResolverSmem {
    float rA[2][NW * kChainLoads * 32], rB[2][NW * kChainLoads * 32];
    int first_bad[2][NW];                               // per loader: first unusable tile of its part
    int stop[2][NW];                                    // per group: give up before that round
};

// One step of a thread's CPT adjacent channels from a shared row, widened to fp32.
template <int DT, int CPT>
__device__ __forceinline__ void step_from_smem(const typename Storage<DT>::raw *p, float (&v)[CPT]) {
    if constexpr (CPT == 1) {
        v[0] = Storage<DT>::get(p[0]);
    } else {
        const uint32_t w = *reinterpret_cast<const uint32_t *>(p);
        v[0] = Storage<DT>::get(half_of(w, 0));
        v[1] = Storage<DT>::get(half_of(w, 1));
    }
}

template <int DT, int TD, int TT, int S, int ST, int CPT>
__global__ void __launch_bounds__(TD / CPT * S, (TD / CPT * S >= 512) ? 1 : 2)
chain_scan_kernel(const __grid_constant__ CUtensorMap map_a,
                  const __grid_constant__ CUtensorMap map_b,
                  typename Storage<DT>::raw *__restrict__ h,
                  const long long L, const long long D,
                  const long long slices_per_batch, const long long n_slices,
                  const long long chunks, const long long n_tiles,
                  const int n_res,                 // resolver CTAs (blockIdx.x < n_res)
                  const int gpc,                   // channel groups per resolver CTA (a power of two <= warps)
                  const int cpg,                   // channels per group (4, 8, 16 or 32)
                  const int stride,                // H is published for chunks q with q % stride == stride-1
                  Control *__restrict__ ctrl, unsigned long long *__restrict__ words,
                  unsigned int *__restrict__ status,
                  const long long spin_limit, const long long silent_tile,
                  const float *h_init, float *h_last)
{
    constexpr int K = TT / S;                 // time steps per thread
    constexpr int TC = TD / CPT;              // channel groups of a tile
    constexpr int NT = TC * S;                // threads
    constexpr int NW = NT / 32;               // warps
    using E = typename Storage<DT>::raw;
    constexpr uint32_t kStageBytes = 2u * TT * TD * sizeof(E);
    static_assert(TD == 32, "a resolver lane serves one channel of a 32-channel slice");
    static_assert(TT % S == 0 && (32 % S) == 0 && S >= 2 && ST >= 3 && NT % 32 == 0, "tile shape");
    static_assert(CPT == 1 || (CPT == 2 && Storage<DT>::bytes == 2 && (32 / S) % 2 == 0), "channels per thread");
    using Smem = ChunkSmem<E, TD, TT, S, ST>;
    using RSmem = ChainResolverSmem<NW>;
    static_assert(sizeof(RSmem) <= sizeof(Smem), "the resolver's arrays fit the ring");
    extern __shared__ __align__(128) unsigned char smem_raw[];
    __shared__ uint32_t s_tag;

    pdl_wait();   // launched as a programmatic dependent: nothing before it is touched yet

    const int tid = threadIdx.x;
    if (tid == 0) s_tag = tag_of(ld_relaxed_u32(&ctrl->epoch));
    __syncthreads();
    const uint32_t tag = s_tag;
    // [tile][channel] pairs of tagged words (A, B), then [tile][channel] tagged H
    unsigned long long *const wAgg = words;
    unsigned long long *const wInc = words + 2 * n_tiles * TD;
    const long long n_state = (n_slices / slices_per_batch) * D;
    const float kNaN = __uint_as_float(0x7fc00000u);

    if ((int)blockIdx.x < n_res) {
        // ================================ resolver ================================
        // A group of nwg warps walks the chains of cpg channels of one slice (each channel's
        // chain is independent; splitting a slice's channels over groups on several CTAs
        // spreads the reads of the maps and the writes of H over several SMs).  Loader warps
        // (all but the first; the only warp when nwg = 1) read the next window of maps into
        // one buffer while the chain warp folds the current window from the other, lane =
        // channel, and publishes each H as it makes it.  A window's usable part is its prefix
        // of tiles whose words all carry this launch's tag.
        RSmem &rs = *reinterpret_cast<RSmem *>(smem_raw);
        const int lane = tid & 31, warp = tid >> 5;
        const int nwg = NW / gpc;              // warps per group
        const int gl = warp / nwg, wg = warp - gl * nwg;
        const int groups_per_slice = TD / cpg;
        const long long grp = (long long)blockIdx.x * gpc + gl;
        if (grp < n_slices * groups_per_slice) {
            const long long slice = grp / groups_per_slice;
            const int c0 = (int)(grp - slice * groups_per_slice) * cpg;   // the group's first channel
            const long long bi = slice / slices_per_batch;
            const long long d0 = (slice - bi * slices_per_batch) * TD;
            const int P = 32 / cpg;                // tiles per load instruction
            const int lc = lane % cpg, lo = lane / cpg;
            const int loaders = nwg > 1 ? nwg - 1 : 1;
            const bool loads = nwg == 1 || wg >= 1;
            const bool chains = wg == 0;
            const int li = nwg > 1 ? wg - 1 : 0;   // this loader's part of the window
            const int per = kChainLoads * P;       // tiles per loader
            const int win = loaders * per;         // tiles per window
            const int base = gl * nwg * kChainLoads * 32;   // the group's part of each buffer
            const long long need = chunks - 1;     // H_0 .. H_{chunks-2}: the last tile has no successor
            const int bar = 1 + gl, bar_threads = 32 * nwg;
            float H = 0.0f;
            if (lane < cpg && h_init && d0 + c0 + lane < D && inside(h_init + bi * D + d0 + c0 + lane, h_init, n_state))
                H = h_init[bi * D + d0 + c0 + lane];
            unsigned long long wa[kChainLoads], wb[kChainLoads];
            // (loaders) read this warp's part of the window starting at chunk qs
            auto issue = [&](long long qs) {
#pragma unroll
                for (int i = 0; i < kChainLoads; ++i) {
                    wa[i] = wb[i] = 0ull;
                    const long long q = qs + li * per + i * P + lo;
                    const long long at = ((q * n_slices + slice) * TD + c0 + lc) * 2;
                    if (q < need && inside(wAgg + at, wAgg, 2 * n_tiles * TD, false, 16))
                        ld_relaxed_v2_u64(wAgg + at, wa[i], wb[i]);
                }
            };
            // (loaders) the values into buffer b, and the first unusable tile of this part
            auto commit = [&](int b) {
                int bad = win;
#pragma unroll
                for (int i = kChainLoads - 1; i >= 0; --i) {
                    const int t = li * per + i * P + lo;
                    if (word_tag(wa[i]) != tag || word_tag(wb[i]) != tag) bad = t;
                    rs.rA[b][base + t * cpg + lc] = word_val(wa[i]);
                    rs.rB[b][base + t * cpg + lc] = word_val(wb[i]);
                }
                bad = __reduce_min_sync(kFull, bad);
                if (lane == 0) rs.first_bad[b][gl * nwg + li] = bad;
            };
            if (loads) {
                issue(0);
                commit(0);
            }
            if (tid == 32 * gl * nwg) rs.stop[0][gl] = 0;
            bar_sync_group(bar, bar_threads);
            long long q = 0, idle = 0;
            unsigned int nap = 64;
            for (int r = 0; q < need; ++r) {
                const int b = r & 1;
                if (rs.stop[b][gl]) break;      // decided by the chain warp last round
                int used = win;
                for (int w = 0; w < loaders; ++w) used = min(used, rs.first_bad[b][gl * nwg + w]);
                const long long qn = q + used;  // start of the next window
                if (loads && qn < need) issue(qn);
                if (chains) {
                    // fold the window's usable prefix into H in tile order, publishing each H_q
                    for (int j0 = 0; j0 < used; j0 += 16) {
                        float va[16], vb[16];
#pragma unroll
                        for (int e = 0; e < 16; ++e) {
                            const int t = (j0 + e < used ? j0 + e : j0) * cpg + (lane < cpg ? lane : 0);
                            va[e] = rs.rA[b][base + t];
                            vb[e] = rs.rB[b][base + t];
                        }
#pragma unroll
                        for (int e = 0; e < 16; ++e) {
                            if (j0 + e < used && lane < cpg) {
                                H = fmaf(va[e], H, vb[e]);
                                const long long qe = q + j0 + e;
                                const long long at = (qe * n_slices + slice) * TD + c0 + lane;
                                if ((qe & (stride - 1)) == stride - 1 && inside(wInc + at, wInc, n_tiles * TD))
                                    st_relaxed_u64(wInc + at, pack_word(tag, H));
                            }
                        }
                    }
                    if (lane == 0) {
                        int stop = 0;
                        if (used == 0 &&
                            (idle + 1 > spin_limit || ((idle & 15) == 15 && ld_relaxed_u32(&ctrl->abort) != 0))) {
                            stop = 1;
                            atomicOr(status, kStatusLookbackTimeout);
                            atomicExch(&ctrl->abort, 1u);
                        }
                        rs.stop[b ^ 1][gl] = stop;
                    }
                }
                if (loads && qn < need) commit(b ^ 1);
                if (used == 0) {
                    ++idle;
                    __nanosleep(nap);
                    if (nap < 1024) nap <<= 1;
                } else {
                    idle = 0;
                    nap = 64;
                }
                bar_sync_group(bar, bar_threads);
                q = qn;
            }
        }
    } else {
        // ================================= worker =================================
        // Tiles go round-robin: worker w takes tile ids w, w + n_workers, ... in order (all
        // CTAs are resident, so every tile a resolver waits for is being worked on).
        Smem &sm = *reinterpret_cast<Smem *>(smem_raw);
        const int c = tid % TC;                   // channel group: channels CPT*c .. CPT*c + CPT-1
        const int s = tid / TC;                   // segment within the tile
        const int cc = tid / S;                   // transposed role: channels cc, cc + TC, ...
        const int ss = tid % S;                   // and the segment
        const long long n_h = (n_slices / slices_per_batch) * L * D;
        const long long wk = (long long)blockIdx.x - n_res, n_workers = (long long)gridDim.x - n_res;

        auto issue = [&](int st, long long id) {
            const long long q = id / n_slices;
            const long long slice = id - q * n_slices;
            const long long bi = slice / slices_per_batch;
            const int d0 = (int)((slice - bi * slices_per_batch) * TD);
            sm.tile[st] = TileCoord{id, (int)q, (int)bi, d0, 0};
            mbar_arrive_expect_tx(&sm.full[st], kStageBytes);
            tma_load_3d(sm.a[st], &map_a, &sm.full[st], d0, (int)(q * TT), (int)bi);
            tma_load_3d(sm.b[st], &map_b, &sm.full[st], d0, (int)(q * TT), (int)bi);
        };
        auto finish = [&](int st) { sm.tile[st] = TileCoord{n_tiles, 0, 0, 0, 0}; };

        const bool misaligned = (smem_u32(smem_raw) & 127u) != 0;
        if (tid == 0) {
            if (misaligned) {
                atomicOr(status, kStatusTmaTimeout);
                atomicExch(&ctrl->abort, 1u);
                finish(0);
            } else {
                for (int st = 0; st < ST; ++st) mbar_init(&sm.full[st], 1);
                mbar_fence_init();
                tmap_prefetch(&map_a);
                tmap_prefetch(&map_b);
                if (wk < n_tiles) issue(0, wk);
                else finish(0);
            }
        }
        __syncthreads();

        uint32_t phases = 0;                      // bit st: parity of the next completion of stage st
        long long next_fill = 1;                  // (thread 0) next ring slot to fill
        bool ended = sm.tile[0].id >= n_tiles;    // (thread 0) no more tiles
        uint32_t abort_seen = 0;                  // (thread 0) abort word, read one fill early
        // (thread 0) fill ring slots up to (not including) `limit`; slot n is tile wk + n * n_workers
        // and goes to stage n % ST
        auto refill = [&](long long limit) {
            if (!ended && abort_seen != 0) {
                ended = true;
                finish((int)(next_fill % ST));
            }
            while (!ended && next_fill < limit) {
                const int s2 = (int)(next_fill % ST);
                const long long nid = wk + next_fill * n_workers;
                if (nid >= n_tiles) {
                    ended = true;
                    finish(s2);
                } else {
                    issue(s2, nid);
                }
                ++next_fill;
            }
            abort_seen = ld_relaxed_u32(&ctrl->abort);
        };
        // (threads 0 .. TD-1, lane = channel) the published H of tile `pred`, first read `v`
        // (issued before the compose), then polled with a bound
        auto carry_of = [&](long long pred, int ch, unsigned long long v) -> float {
            const unsigned long long *w = wInc + pred * TD + ch;
            long long n = 0;
            unsigned int nap = 32;
            for (;;) {
                if (word_tag(v) == tag) return word_val(v);
                if (++n > spin_limit || ((n & 63) == 0 && ld_relaxed_u32(&ctrl->abort) != 0)) {
                    atomicOr(status, kStatusLookbackTimeout);
                    atomicExch(&ctrl->abort, 1u);
                    return kNaN;
                }
                __nanosleep(nap);
                if (nap < 256) nap <<= 1;
                v = inside(w, wInc, n_tiles * TD) ? ld_relaxed_u64(w) : 0ull;
            }
        };

        // (threads 0 .. TD-1) a published map (A, B), first read (wa, wb), polled with a bound;
        // on expiry both words become NaN
        auto map_of = [&](const unsigned long long *w, unsigned long long &wa, unsigned long long &wb) {
            long long n = 0;
            unsigned int nap = 32;
            while (word_tag(wa) != tag || word_tag(wb) != tag) {
                if (++n > spin_limit || ((n & 63) == 0 && ld_relaxed_u32(&ctrl->abort) != 0)) {
                    atomicOr(status, kStatusLookbackTimeout);
                    atomicExch(&ctrl->abort, 1u);
                    wa = wb = pack_word(tag, kNaN);
                    return;
                }
                __nanosleep(nap);
                if (nap < 256) nap <<= 1;
                if (inside(w, wAgg, 2 * n_tiles * TD, false, 16)) ld_relaxed_v2_u64(w, wa, wb);
            }
        };

        TileRegs<DT, K, CPT> r;                   // the previous tile's a and b, for its replay
        TileCoord pc{n_tiles, 0, 0, 0, 0};        // the previous tile
        bool have_prev = false;
        for (long long k = 0;; ++k) {
            const int st = (int)(k % ST);
            const int kb = (int)(k & 1), pb = kb ^ 1;
            const TileCoord tc = sm.tile[st];
            const bool cur = tc.id < n_tiles;
            if (!cur && !have_prev) break;
            // The first iteration fills the rest of the ring before it waits.
            if (tid == 0 && k == 0) refill(ST);
            // The carry of tile k-1 is H_{q-1} (q its chunk).  The resolver publishes H only for
            // chunks p with p % stride == stride-1; the words this tile needs, the last such H at
            // or before q-1 and the maps of the r chunks after it, are read now, so the reads'
            // latency passes during tile k's compose.
            unsigned long long pre = 0ull, fa[kChainStrideMax - 1], fb[kChainStrideMax - 1];
            int fold = 0;                                 // r: maps to fold onto that H
            long long qh = -1;                            // the chunk of that H (-1: none, the state)
            const long long pslice = pc.id - (long long)pc.q * n_slices;
            if (have_prev && tid < TD && pc.q > 0) {
                const long long qp = pc.q - 1;
                fold = (int)((qp + 1) & (stride - 1));
                qh = qp - fold;
                if (qh >= 0) {
                    const unsigned long long *w = wInc + (qh * n_slices + pslice) * TD + tid;
                    pre = inside(w, wInc, n_tiles * TD) ? ld_relaxed_u64(w) : 0ull;
                }
#pragma unroll
                for (int i = 0; i < kChainStrideMax - 1; ++i) {
                    fa[i] = fb[i] = 0ull;
                    const unsigned long long *w = wAgg + (((qh + 1 + i) * n_slices + pslice) * TD + tid) * 2;
                    if (i < fold && inside(w, wAgg, 2 * n_tiles * TD, false, 16)) ld_relaxed_v2_u64(w, fa[i], fb[i]);
                }
            }

            // ---- compose tile k from shared memory (its stage stays held) ----------
            const int r0 = s * K;
            if (cur) {
                if (!mbar_wait_bounded(&sm.full[st], (phases >> st) & 1u, kTmaPolls)) {
                    atomicOr(status, kStatusTmaTimeout);
                    atomicExch(&ctrl->abort, 1u);
                }
                phases ^= 1u << st;
                const long long rem = L - ((long long)tc.q * TT + r0);
                const int nv = rem <= 0 ? 0 : (rem >= K ? K : (int)rem);
                const bool zero_a0 = tc.q == 0 && s == 0 && !h_init;   // h_{-1} = 0: a_0 never matters
                const E *ta = sm.a[st] + r0 * TD + CPT * c;
                const E *tb = sm.b[st] + r0 * TD + CPT * c;
                float A[CPT], Bv[CPT];
#pragma unroll
                for (int i = 0; i < CPT; ++i) { A[i] = 1.0f; Bv[i] = 0.0f; }
#pragma unroll
                for (int j = 0; j < K; ++j) {
                    if (j < nv) {
                        float av[CPT], bv[CPT];
                        step_from_smem<DT, CPT>(ta + j * TD, av);
                        step_from_smem<DT, CPT>(tb + j * TD, bv);
                        if (j == 0 && zero_a0) {
#pragma unroll
                            for (int i = 0; i < CPT; ++i) av[i] = 0.0f;
                        }
#pragma unroll
                        for (int i = 0; i < CPT; ++i) {
                            Bv[i] = fmaf(av[i], Bv[i], bv[i]);
                            A[i] = av[i] * A[i];
                        }
                    }
                }
                st_group<CPT>(&sm.segA[kb][s][CPT * c], A);
                st_group<CPT>(&sm.segB[kb][s][CPT * c], Bv);
            }
            __syncthreads();
            // Every thread has finished iteration k-1, which moved tile k-1's a and b into
            // registers: its stage (slot k-1) takes slot k-1+ST.
            if (tid == 0 && k >= 1) refill(k + ST);

            // ---- tile k: shuffle scan over its segments; publish its map ----------------
            if (cur) {
                float (&segA)[S][TD + 32 / S] = sm.segA[kb];
                float (&segB)[S][TD + 32 / S] = sm.segB[kb];
#pragma unroll
                for (int i = 0; i < CPT; ++i) {
                    const int ch = cc + i * TC;
                    float xA = segA[ss][ch], xB = segB[ss][ch];
#pragma unroll
                    for (int off = 1; off < S; off <<= 1) {
                        const float uA = __shfl_up_sync(kFull, xA, off, S);
                        const float uB = __shfl_up_sync(kFull, xB, off, S);
                        if (ss >= off) {          // (later) o (earlier)
                            xB = fmaf(xA, uB, xB);
                            xA = xA * uA;
                        }
                    }
                    float eA = __shfl_up_sync(kFull, xA, 1, S);
                    float eB = __shfl_up_sync(kFull, xB, 1, S);
                    if (ss == 0) { eA = 1.0f; eB = 0.0f; }
                    segA[ss][ch] = eA;
                    segB[ss][ch] = eB;
                    const float tA = __shfl_sync(kFull, xA, S - 1, S);
                    const float tB = __shfl_sync(kFull, xB, S - 1, S);
                    // the resolver needs every map but the slice's last
                    if (ss == 0 && tc.q + 1 < chunks && tc.id != silent_tile) {
                        unsigned long long *w = wAgg + (tc.id * TD + ch) * 2;
                        if (inside(w, wAgg, 2 * n_tiles * TD, false, 16))
                            st_relaxed_v2_u64(w, pack_word(tag, tA), pack_word(tag, tB));
                    }
                }
            }
            // ---- the carry entering tile k-1 ---------------------------------------------
            if (have_prev && tid < TD) {
                const int ch = tid;
                float carry;
                const long long at = (long long)pc.bi * D + pc.d0 + ch;
                const float h_before = (h_init && pc.d0 + ch < D && inside(h_init + at, h_init, n_state)) ? h_init[at] : 0.0f;
                if (pc.q == 0) {
                    carry = h_before;
                } else {
                    carry = qh >= 0 ? carry_of(qh * n_slices + pslice, ch, pre) : h_before;
#pragma unroll
                    for (int i = 0; i < kChainStrideMax - 1; ++i) {
                        if (i < fold) {
                            const unsigned long long *w = wAgg + (((qh + 1 + i) * n_slices + pslice) * TD + ch) * 2;
                            map_of(w, fa[i], fb[i]);
                            carry = fmaf(word_val(fa[i]), carry, word_val(fb[i]));
                        }
                    }
                }
                sm.carry[pb][ch] = carry;
            }
            __syncthreads();

            // ---- replay tile k-1 from its carry, store h ----------------------------------
            if (have_prev) {
                const long long q = pc.q, bi = pc.bi, d0 = pc.d0;
                const long long t0 = q * TT;
                const long long rem = L - (t0 + r0);
                const int nv = rem <= 0 ? 0 : (rem >= K ? K : (int)rem);
                float hc[CPT], pA[CPT], pB[CPT];
                ld_group<CPT>(&sm.segA[pb][s][CPT * c], pA);
                ld_group<CPT>(&sm.segB[pb][s][CPT * c], pB);
                ld_group<CPT>(&sm.carry[pb][CPT * c], hc);
#pragma unroll
                for (int i = 0; i < CPT; ++i) hc[i] = fmaf(pA[i], hc[i], pB[i]);
                if ((d0 + CPT * c) < D) {
                    E *hp = h + ((bi * L + t0 + r0) * D + d0 + CPT * c);
#pragma unroll
                    for (int j = 0; j < K; ++j) {
                        if (j < nv) {
#pragma unroll
                            for (int i = 0; i < CPT; ++i) hc[i] = fmaf(r.a(j, i), hc[i], r.b(j, i));
                            if (inside(hp + (long long)j * D, h, n_h, true, CPT * (long long)sizeof(E)))
                                st_h<DT, CPT>(hp + (long long)j * D, hc);
                        }
                    }
                    // the thread holding t = L-1 hands the state out
                    if (h_last && nv > 0 && t0 + r0 + nv == L) {
#pragma unroll
                        for (int i = 0; i < CPT; ++i)
                            if (inside(h_last + bi * D + d0 + CPT * c + i, h_last, n_state, true))
                                h_last[bi * D + d0 + CPT * c + i] = hc[i];
                    }
                }
            }
            if (!cur) break;                      // slot k was the end: nothing after it was filled
            // ---- tile k's a and b into registers for the next iteration; its stage is free after
            // the next iteration's first barrier --------------------------------------------------
            r.load(sm.a[st] + r0 * TD + CPT * c, sm.b[st] + r0 * TD + CPT * c, TD);
            if (tc.q == 0 && s == 0 && !h_init) r.zero_a0();
            pc = tc;
            have_prev = true;
        }
    }

    // This CTA's work is done: the launch that follows may be scheduled (it waits for
    // this whole grid before it touches memory).
    pdl_release();
    // The last CTA to finish resets the counters and moves the epoch on for the next launch.
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

#define LINREC_CHAIN_F32_VARIANTS(X) X(32, 128, 8, 3, 1) X(32, 256, 16, 3, 1)
#define LINREC_CHAIN_16_VARIANTS(X) X(32, 256, 8, 3, 2)

template <int DT, int TD, int TT, int S, int ST, int CPT>
constexpr ChunkedVariant make_chain_variant() {
    ChunkedVariant v = make_variant<DT, TD, TT, S, ST, CPT>();
    v.chain = 1;
    return v;
}

#define LINREC_CV_F32(TD, TT, S, ST, CPT) make_chain_variant<kDtypeF32, TD, TT, S, ST, CPT>(),
#define LINREC_CV_16(TD, TT, S, ST, CPT) make_chain_variant<kDtypeBF16, TD, TT, S, ST, CPT>(),
const ChunkedVariant kChainF32[] = {LINREC_CHAIN_F32_VARIANTS(LINREC_CV_F32)};
const ChunkedVariant kChain16[] = {LINREC_CHAIN_16_VARIANTS(LINREC_CV_16)};
#undef LINREC_CV_F32
#undef LINREC_CV_16

}  // namespace

const ChunkedVariant *chain_variants(int dtype, int *count) {
    if (dtype == kDtypeF32) {
        *count = (int)(sizeof(kChainF32) / sizeof(kChainF32[0]));
        return kChainF32;
    }
    *count = (int)(sizeof(kChain16) / sizeof(kChain16[0]));
    return kChain16;
}

const void *chain_kernel(const ChunkedVariant *v, int dtype) {
    if (!v->chain) return nullptr;
#define LINREC_CK(DT, TD, TT, S, ST, CPT)                                                                  \
    if (dtype == DT && v->tile_d == TD && v->tile_t == TT && v->segments == S && v->stages == ST &&      \
        v->cpt == CPT)                                                                                     \
        return reinterpret_cast<const void *>(&chain_scan_kernel<DT, TD, TT, S, ST, CPT>);
#define LINREC_CK_F32(TD, TT, S, ST, CPT) LINREC_CK(kDtypeF32, TD, TT, S, ST, CPT)
#define LINREC_CK_BF16(TD, TT, S, ST, CPT) LINREC_CK(kDtypeBF16, TD, TT, S, ST, CPT)
#define LINREC_CK_F16(TD, TT, S, ST, CPT) LINREC_CK(kDtypeF16, TD, TT, S, ST, CPT)
    LINREC_CHAIN_F32_VARIANTS(LINREC_CK_F32)
    LINREC_CHAIN_16_VARIANTS(LINREC_CK_BF16)
    LINREC_CHAIN_16_VARIANTS(LINREC_CK_F16)
#undef LINREC_CK_F32
#undef LINREC_CK_BF16
#undef LINREC_CK_F16
#undef LINREC_CK
    return nullptr;
}

// How the resolver work is laid out: every slice's TD channel chains are split into
// groups of cpg channels (fewer channels per group when there are few slices, so that
// the reads of the maps and the writes of H spread over more SMs); about kMaxResolvers
// CTAs, each serving gpc groups (a power of two, at most one group per warp).  Returns
// the resolver CTAs, more than kMaxResolvers only when the slices outnumber the warps
// of that many CTAs (the plan then refuses chain mode).
int chain_layout(int64_t n_slices, int warps, int *cpg_out, int *gpc_out) {
    constexpr int kMaxResolvers = kChainMaxResolvers;
    const int cpg = n_slices <= 1 ? 4 : n_slices <= 4 ? 8 : n_slices <= 8 ? 16 : 32;
    const int64_t groups = n_slices * (32 / cpg);
    int gpc = 1;
    while (gpc < warps && (groups + gpc - 1) / gpc > kMaxResolvers) gpc *= 2;
    *cpg_out = cpg;
    *gpc_out = gpc;
    return (int)((groups + gpc - 1) / gpc);
}

cudaError_t launch_chain(const ChunkedLaunch &p, cudaStream_t stream) {
    const ChunkedVariant *v = p.variant;
    const void *fn = chain_kernel(v, p.dtype);
    if (!fn || p.mode != kModeChain) return cudaErrorInvalidValue;
    int cpg = 0, gpc = 0;
    const int n_res = chain_layout(p.n_slices, v->threads / 32, &cpg, &gpc);
    if (p.grid <= n_res) return cudaErrorInvalidValue;   // no worker
    cudaError_t err = cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)v->smem_bytes);
    if (err != cudaSuccess) return err;
    long long L = p.L, D = p.D, spb = p.slices_per_batch, ns = p.n_slices, ch = p.chunks, nt = p.n_tiles;
    long long spin = p.spin_limit, silent = p.silent_tile;
    int nres = n_res, stride = kChainStride;
    void *h = p.h;
    Control *ctrl = p.ctrl;
    unsigned long long *words = p.words;
    unsigned int *status = p.status;
    const float *h_init = p.h_init;
    float *h_last = p.h_last;
    void *args[] = {(void *)&p.map_a, (void *)&p.map_b, &h, &L, &D, &spb, &ns, &ch, &nt, &nres, &gpc, &cpg, &stride,
                    &ctrl, &words, &status, &spin, &silent, &h_init, &h_last};
    // Cooperative: workers wait on resolvers, so every CTA must be resident together.
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)p.grid);
    cfg.blockDim = dim3((unsigned)v->threads);
    cfg.dynamicSmemBytes = v->smem_bytes;
    cfg.stream = stream;
    cudaLaunchAttribute attr[2];
    attr[0].id = cudaLaunchAttributeCooperative;
    attr[0].val.cooperative = 1;
    attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[1].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 2;
    err = cudaLaunchKernelExC(&cfg, fn, args);
    if (err == cudaSuccess) return err;
    // without the programmatic dependence, should the runtime refuse the pair
    cudaGetLastError();
    cfg.numAttrs = 1;
    return cudaLaunchKernelExC(&cfg, fn, args);
}

LINREC_CHECKED_REPORT(checked_report_chain)

}  // namespace linrec
