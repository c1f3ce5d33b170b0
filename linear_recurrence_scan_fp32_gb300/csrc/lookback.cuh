// lookback.cuh -- the decoupled look-back shared by the forward and backward
// chunked kernels: the carry entering a tile, from tagged words published by
// the earlier tiles of its slice.
#pragma once

#include "checked.cuh"
#include "kernels.cuh"
#include "ptx.cuh"

namespace linrec {

constexpr unsigned kFull = 0xffffffffu;

// Look-back mode: the h value entering tile `id` for channel cc, computed by
// groups of S lanes per channel.  Lane ss watches R predecessors: window
// position p = r*S + ss is tile id - (1 + p) * n_slices, so one round trip
// covers W = S*R earlier tiles of the slice.  Each round reads the inclusive
// words of the window first and the aggregate words only of the positions
// between this tile and the nearest inclusive value.  The group walks back
// over windows that hold aggregates only, then replays the chain forward
// from the inclusive value it found, re-reading the aggregates it passed.
template <int S, int R>
__device__ __forceinline__ float lookback_carry(
    const long long id, const long long n_slices, const int TD, const int cc, const int ss, const int gbase,
    const uint32_t tag, const bool publish_agg, const float tA, const float tB, const float h_before,
    unsigned long long *__restrict__ wAggA, unsigned long long *__restrict__ wAggB,
    const unsigned long long *__restrict__ wInc, const long long n_words, Control *__restrict__ ctrl,
    unsigned int *__restrict__ status, const long long spin_limit)
{
    // (n_words: the words of each of the three arrays; a word outside reads as untagged)
    auto word = [&](const unsigned long long *arr, long long i) -> unsigned long long {
        return inside(arr + i, arr, n_words) ? ld_relaxed_u64(arr + i) : 0ull;
    };
    constexpr int W = S * R;
    static_assert(W <= 32, "window fits a 32-bit mask");
    constexpr unsigned GM = (S == 32) ? kFull : ((1u << S) - 1u);
    const long long me = id * TD + cc;
    // Successors may need this tile's aggregate before its carry is known.
    if (publish_agg && ss == 0 && inside(wAggA + me, wAggA, n_words) && inside(wAggB + me, wAggB, n_words)) {
        st_relaxed_u64(&wAggA[me], pack_word(tag, tA));
        st_relaxed_u64(&wAggB[me], pack_word(tag, tB));
    }
    long long base = id - n_slices;           // tile at window position 0: the predecessor
    int skipped = 0;                          // windows holding aggregates only
    int pstar = -1;                           // window position of the nearest inclusive value
    bool failed = false;
    float vA[R], vB[R], vH[R];                // what this lane read for its R tiles
    bool have[R];                             // aggregate of that tile already read
#pragma unroll
    for (int r = 0; r < R; ++r) { vA[r] = 1.0f; vB[r] = 0.0f; vH[r] = 0.0f; have[r] = false; }
    long long idle = 0;
    unsigned int nap = 32;
    for (;;) {
        const bool active = pstar < 0 && !failed;
        // inclusive words of the window
        unsigned inc_g = 0;
#pragma unroll
        for (int r = 0; r < R; ++r) {
            bool inc = false;
            if (active) {
                const long long j = base - (long long)(r * S + ss) * n_slices;
                if (j < 0) {
                    inc = true;
                    vH[r] = h_before;         // before the first chunk: the carried-in state
                } else {
                    const unsigned long long wi = word(wInc, j * TD + cc);
                    inc = word_tag(wi) == tag;
                    vH[r] = word_val(wi);
                }
            }
            inc_g |= ((__ballot_sync(kFull, active && inc) >> gbase) & GM) << (r * S);
        }
        const int pc = inc_g ? __ffs(inc_g) - 1 : W;   // nearest inclusive position (W: none)
        // aggregate words of the positions before it
        unsigned none_g = 0;
#pragma unroll
        for (int r = 0; r < R; ++r) {
            const int p = r * S + ss;
            bool missing = false;
            if (active && p < pc && !have[r]) {
                const long long j = base - (long long)p * n_slices;
                const unsigned long long wa = word(wAggA, j * TD + cc);
                const unsigned long long wb = word(wAggB, j * TD + cc);
                if (word_tag(wa) == tag && word_tag(wb) == tag) {
                    vA[r] = word_val(wa);
                    vB[r] = word_val(wb);
                    have[r] = true;
                } else {
                    missing = true;
                }
            }
            none_g |= ((__ballot_sync(kFull, missing) >> gbase) & GM) << (r * S);
        }
        bool progressed = false;
        if (active) {
            if (none_g == 0) {
                if (pc < W) {
                    pstar = pc;
                } else {
                    ++skipped;
                    base -= (long long)W * n_slices;
#pragma unroll
                    for (int r = 0; r < R; ++r) have[r] = false;
                }
                progressed = true;
            }
            if (progressed) {
                idle = 0;
            } else if (++idle > spin_limit || ((idle & 63) == 0 && ld_relaxed_u32(&ctrl->abort) != 0)) {
                failed = true;
                if (ss == 0) atomicOr(status, kStatusLookbackTimeout);
            }
        }
        if (__all_sync(kFull, pstar >= 0 || failed)) break;
        if (__any_sync(kFull, progressed)) {
            nap = 32;
        } else {
            __nanosleep(nap);
            if (nap < 1024) nap <<= 1;
        }
    }

    // Replay the chain forward from the inclusive value: the rest of its window,
    // then every skipped window, the one nearest to this tile last.
    const int pf = pstar < 0 ? 0 : pstar;
    float mine_h = vH[0];
#pragma unroll
    for (int r = 1; r < R; ++r)
        if (pf / S == r) mine_h = vH[r];
    float H = __shfl_sync(kFull, mine_h, pf % S, S);
#pragma unroll
    for (int p = W - 1; p >= 0; --p) {
        const float ap = __shfl_sync(kFull, vA[p / S], p % S, S);
        const float bp = __shfl_sync(kFull, vB[p / S], p % S, S);
        if (p < pstar) H = fmaf(ap, H, bp);
    }
    const int most = __reduce_max_sync(kFull, failed ? 0 : skipped);
    for (int w = most - 1; w >= 0; --w) {
        const bool mine = !failed && w < skipped;
        if (mine) {
#pragma unroll
            for (int r = 0; r < R; ++r) {
                const long long j = id - n_slices - ((long long)w * W + r * S + ss) * n_slices;
                vA[r] = word_val(word(wAggA, j * TD + cc));
                vB[r] = word_val(word(wAggB, j * TD + cc));
            }
        }
#pragma unroll
        for (int p = W - 1; p >= 0; --p) {
            const float ap = __shfl_sync(kFull, vA[p / S], p % S, S);
            const float bp = __shfl_sync(kFull, vB[p / S], p % S, S);
            if (mine) H = fmaf(ap, H, bp);
        }
    }
    return failed ? __uint_as_float(0x7fc00000u) : H;   // NaN marks a lost carry
}

}  // namespace linrec
