// linrec_api.cu -- the C ABI of liblinrec (declared in include/linrec.h):
// argument checks, the size-based dispatcher, the per-stream look-back
// workspace, tensor-map encoding and the launches.  Host code only.
#include <cuda.h>
#include <cuda_runtime.h>

#include <atomic>
#include <map>
#include <memory>
#include <mutex>
#include <tuple>
#include <utility>

#include "kernels.cuh"
#include "linrec.h"

using namespace linrec;

namespace {

constexpr int kVersion = 200;               // 0.2.0
constexpr int64_t kDefaultSpinLimit = 1 << 20;
constexpr int kRegcarryThreads = 256;
// forward scans: the register path from this many 16-byte threads per SM on
constexpr int64_t kRegcarryMinThreadsPerSm = 96;
// Few slices: the two-pass mode from this many time chunks of 128 steps on.
constexpr int64_t kTwoPassMinChunks = 64;
// Two-pass levels: a call's own problem (level 0) and the scan of its tile maps (level 1) may take
// two-pass mode; the scan of those maps' maps (level 2) may not.  Measured on GB300 (us per call,
// the level-1 scan in look-back -> two-pass mode): (1, 1048576, 64) 204.0 -> 200.1, whose level-1
// problem (1, 8192, 64) has 64 chunks; the rest of the long shapes measured had fewer (unchanged).
constexpr int kTwoPassLevels = 2;
// Speculative mode: the shortest segment, the most segments, and the shortest segment for the
// dispatcher's choice.  The repair launch recomputes each segment's tiles up to the first after
// which the slope product is exactly 0 in fp32; the rest the speculative launch stored.  Bytes
// per element: 12 + 8 * (that share of the segment), 20 where the slopes never decay.  With
// a ~ U[0.9, 1) the product reaches 0 after about 2000 steps: 16 tiles of a 64-tile segment.
// Measured on GB300, us per call against two-pass or chain mode, a ~ U[0.9, 1) / a = 1:
// (1, 1048576, 64) 148.8 / 215.7 vs 200.5; (1, 4194304, 32) 270 / 428 vs 398; (4, 65536, 256)
// 147 / 209 vs chain 183; with 4096-step segments 9-12 % faster / 6-12 % slower ((1, 1048576, 32),
// (8, 65536, 64)); with 1024-step segments slower either way ((1, 131072, 64) 29.2 vs 26.9).
constexpr int64_t kSpecMinSteps = 1024;
constexpr int64_t kSpecMaxSegments = 1024;
constexpr int kSpecCtasPerSm = 2;
constexpr int64_t kSpecDefaultSteps = 8192;
// fp32 forward scans that would take the two-pass mode, and that the speculative mode does not
// take, take chain mode instead from this many 32-channel slices on, with 256-step tiles from kChainLongSteps steps on (half the
// tiles for the resolvers to fold), 128-step tiles below.  Measured on GB300 (us per call,
// two-pass -> chain): (2, 131072, 128) 112 -> 106, (3, 131072, 128) 160 -> 145, (6, 65536,
// 128) 158 -> 138, (4, 65536, 256) 209 -> 183, (3, 32768, 1024) 306 -> 262, (1, 32768, 512)
// 61.7 -> 55.8, (16, 8192, 128) 59.8 -> 53.6 (128-step tiles; 55.1 with 256); with fewer
// slices chain mode loses ((1, 524288, 128) 211 -> 228, (1, 1048576, 64) 212 -> 328), and in
// 16-bit storage it loses at every slice count measured.
constexpr int64_t kChainMinSlices = 8;
constexpr int64_t kChainLongSteps = 32768;
// Wide slices (see plan_impl): from this many time steps, on a grid of at least this
// share of the SMs.
constexpr int64_t kWideMinSteps = 256;
// Segmented register path: bytes of loads in flight to aim for per SM, the shortest
// segment, the most segments.
constexpr int64_t kSegBytesPerSm = 48 * 1024;
constexpr int64_t kSegMinSteps = 64;
constexpr int64_t kSegMax = 256;
// fp32 forward slice-owner mode from this share of the SM count in slices.
constexpr int kOwnMinSlicesPct = 84;
// ... and at any slice count when a slice has at most this many chunks of 128 steps: the
// look-back mode's tile counter and end-of-launch atomics cost more than walking so few
// chunks in order.  Measured on GB300 (us per call, CUDA graph of back-to-back calls,
// look-back -> slice-owner): (1, 128, 32) 5.7 -> 2.2, (4, 256, 32) 6.2 -> 3.5, (32 slices,
// 512 steps) 6.9 -> 6.2, (64 slices, 512) 7.4 -> 6.3, (127 slices, 512) 10.0 -> 6.3; at 6
// chunks look-back wins below about 100 slices ((64 slices, 768) 8.4 against 8.9).
constexpr int64_t kOwnShortChunks = 4;
constexpr int kWideMinGridPct = 84;
constexpr int64_t kWide64MinSteps = 4096;
// Blocks mode: default time steps per block (tiles per block = this / tile_t).
constexpr int64_t kBlockSteps = 1024;
constexpr size_t kWorkspaceHead = 256;      // Control block, padded
// (B, D, L) layout: rows alone give each SM this many warps -> one pass, each warp
// scanning consecutive rows until it holds about kRowsStreamElems[16-bit] elements,
// while at least kRowsStreamWarps warps per SM remain (measured on GB300: the many
// short rows of the (256, 4096, 128) shape want 16 rows per warp in fp32, 64 in
// 16-bit storage); otherwise two passes over segments of at least
// kRowsMinSegChunks chunks, about kRowsTargetWarps warps per SM in all.
constexpr int64_t kRowsMinWarps = 16;
constexpr int64_t kRowsStreamWarps = 32;
constexpr int64_t kRowsStreamElems = 2048;
constexpr int64_t kRowsStreamElems16 = 8192;
constexpr int64_t kRowsTargetWarps = 32;
constexpr int64_t kRowsMinSegChunks = 8;

// Device facts: written once under g_mu before the pointer is handed out; the resident-CTA
// counts are filled in as variants are first used, by any thread (atomics, 0 = not queried).
struct DeviceInfo {
    bool ready = false;
    bool supported = false;
    int sm_count = 0;
    std::atomic<int> ctas_per_sm[3][64];       // per storage type and chunked variant
    std::atomic<int> back_ctas_per_sm[64];     // per backward variant
    std::atomic<int> chain_ctas_per_sm[3][8];  // per storage type and chain variant
    DeviceInfo() {
        for (auto &row : ctas_per_sm)
            for (auto &x : row) x.store(0, std::memory_order_relaxed);
        for (auto &x : back_ctas_per_sm) x.store(0, std::memory_order_relaxed);
        for (auto &row : chain_ctas_per_sm)
            for (auto &x : row) x.store(0, std::memory_order_relaxed);
    }
};

// Locking: g_mu guards the two maps below and is held only to look an entry up.  A call
// then holds its stream's own mutex for the rest of its work (plan, workspace, tensor maps,
// launches): calls on different streams run concurrently; calls on one stream, which run in
// order on the GPU anyway, take turns, so one never frees a workspace another is about to
// launch with.
std::mutex g_mu;
std::map<int, DeviceInfo> g_devices;

struct Slot {
    unsigned char *base = nullptr;
    size_t bytes = 0;
    bool captured = false;   // used by a call captured into a CUDA graph: never freed
};
// What a workspace slot holds.  A look-back slot holds the Control block and
// tagged words only (zero when allocated), so a word whose tag matches the
// current epoch was written by this launch; the two-pass mode's plain float
// arrays live in slots of their own, where no tag is ever looked for.
enum SlotKind { kSlotTagged = 0, kSlotArrays = 1 };
// The library's state for one (device, stream): its workspace slots keyed by (level, kind);
// level 1 is the two-pass mode's scan of its aggregates.
struct StreamState {
    std::mutex mu;                           // held by a call on this stream for its whole work
    std::map<std::pair<int, int>, Slot> slots;
};
std::map<std::pair<int, uintptr_t>, std::unique_ptr<StreamState>> g_streams;

// The state of (dev, stream), created on first use (takes g_mu briefly).
StreamState *stream_state(int dev, cudaStream_t stream) {
    std::lock_guard<std::mutex> lock(g_mu);
    std::unique_ptr<StreamState> &p = g_streams[std::make_pair(dev, reinterpret_cast<uintptr_t>(stream))];
    if (!p) p.reset(new StreamState);
    return p.get();
}

// The state of (dev, stream) if the library has used that stream, else NULL.
StreamState *find_stream_state(int dev, cudaStream_t stream) {
    std::lock_guard<std::mutex> lock(g_mu);
    auto it = g_streams.find(std::make_pair(dev, reinterpret_cast<uintptr_t>(stream)));
    return it == g_streams.end() ? nullptr : it->second.get();
}

typedef CUresult (*EncodeTiledFn)(CUtensorMap *, CUtensorMapDataType, cuuint32_t, void *, const cuuint64_t *,
                                  const cuuint64_t *, const cuuint32_t *, const cuuint32_t *, CUtensorMapInterleave,
                                  CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);
EncodeTiledFn g_encode = nullptr;

// [x, x + xbytes) and [y, y + ybytes) share a byte.
bool overlaps(const void *x, int64_t xbytes, const void *y, int64_t ybytes) {
    const uintptr_t a0 = reinterpret_cast<uintptr_t>(x), b0 = reinterpret_cast<uintptr_t>(y);
    return a0 < b0 + (uintptr_t)ybytes && b0 < a0 + (uintptr_t)xbytes;
}
bool overlaps(const void *x, const void *y, int64_t bytes) { return overlaps(x, bytes, y, bytes); }

int align_of(const void *a, const void *b, const void *h) {
    const uintptr_t u = reinterpret_cast<uintptr_t>(a) | reinterpret_cast<uintptr_t>(b) |
                        reinterpret_cast<uintptr_t>(h);
    if ((u & 15u) == 0) return 16;
    if ((u & 7u) == 0) return 8;
    if ((u & 3u) == 0) return 4;
    return 2;
}

// Sizes: non-negative, and B*L*D*16 bytes representable.
linrec_status_t check_sizes(int64_t B, int64_t L, int64_t D, int64_t *n_out) {
    if (B < 0 || L < 0 || D < 0) return LINREC_ERR_INVALID_VALUE;
    *n_out = 0;
    if (B == 0 || L == 0 || D == 0) return LINREC_OK;
    const int64_t lim = INT64_MAX / 16;
    if (L > lim / D) return LINREC_ERR_INVALID_VALUE;
    const int64_t ld = L * D;
    if (B > lim / ld) return LINREC_ERR_INVALID_VALUE;
    *n_out = B * ld;
    return LINREC_OK;
}

const ChunkedVariant *variants_of(bool backward, int dtype, int *n) {
    if (backward) return backward_variants(n);
    return dtype == kDtypeF32 ? chunked_variants(n) : chunked_variants_16(n);
}

const ChunkedVariant *find_variant(int tile_d, int tile_t, int stages, int cpt, int segments, int *index,
                                   bool backward, int dtype, bool blocks = false) {
    int n = 0;
    const ChunkedVariant *v = variants_of(backward, dtype, &n);
    for (int i = 0; i < n; ++i) {
        if (v[i].tile_d == tile_d && v[i].tile_t == tile_t && (stages == 0 || v[i].stages == stages) &&
            (cpt == 0 || v[i].cpt == cpt) && (segments == 0 || v[i].segments == segments) &&
            (v[i].blocks != 0) == blocks) {
            if (index) *index = i;
            return &v[i];
        }
    }
    return nullptr;
}

// Default chunked tile.  Slice-owner mode: narrow 32-channel slices (more
// slices to spread over the SMs) with a 3-deep ring.  Look-back mode: the
// widest slice D fills, so fewer tiles take part in each carry chain.  16-bit
// storage (measured on GB300): 128-step tiles while slices are scarce, 64-step
// tiles with a 6-deep ring once every SM has several slices and in two-pass
// mode, {32, 128, 4} for look-back.
// 16-bit storage: tiles of 256 steps, the bytes of an fp32 tile of 128 (each thread
// holds its 32 steps packed two to a register); measured on GB300 against 128-step
// tiles: 4885 vs 3621 GB/s on (32, 4096, 256), 6269 vs 4343 on (64, 2048, 1024).
// Sequences shorter than 256 steps take 64-step tiles with a 6-deep ring.
int tile_t_16(int64_t L) { return L >= 256 ? 256 : 64; }

// 16-bit storage, the {32, 256, 2} tile: how many adjacent channels a thread owns
// and how many segments share a channel's 256 steps.  Two channels per thread take
// one 32-bit shared-memory load and one packed store per step for both.  Measured
// on GB300 (bfloat16, us per call, one / two channels per thread):
//  - slice-owner, sm_count < slices <= 3 * sm_count: 128 threads (2 channels,
//    8 segments), three CTAs per SM, one wave: (32, 4096, 256) 38.4 -> 36.6,
//    (57, 4096, 256) 71.8 -> 60.0, (8, 8192, 1024) 72.2 -> 68.7;
//  - slice-owner otherwise: 256 threads (2 channels, 16 segments), no slower at any
//    shape and 1-3 % faster at most: (64, 2048, 1024) 124.7 -> 122.7; the 128-thread
//    CTAs leave a slow tail there ((76, 4096, 256) 73.7 -> 83.7);
//  - two-pass: 128 threads, (1, 1048576, 64) 126.2 -> 116.2;
//  - look-back: one channel per thread (35.0 against 36.7 on (4, 16384, 256)).
void default_groups_16(int64_t slices, int sm_count, bool own, bool twopass, int *cpt, int *segments) {
    if (own) {
        const bool one_wave = slices > sm_count && slices <= 3 * (int64_t)sm_count;
        *cpt = 2;
        *segments = one_wave ? 8 : 16;
    } else if (twopass) {
        *cpt = 2;
        *segments = 8;
    } else {
        *cpt = 1;
        *segments = 8;
    }
}

// Wide slices (fp32, L >= kWideMinSteps, the dispatcher's own tile): the widest of 256
// or 128 channels whose slice count splits evenly over at least kWideMinGridPct % of the
// SMs, one CTA of 512 threads per SM; returns that width (0: none) and the grid.  Every
// CTA then owns the same number of slices, and each box row is 1 or 0.5 KB of
// contiguous memory.  Measured on GB300 (us per call, the previous choice -> this one):
// (64, 2048, 1024) 260 (register path) -> 229 ({128, 64}, 128 CTAs x 4 slices), (128,
// 1024, 1024) 249 -> 232 ({256, 32}, 128 x 4), (8, 4096, 4096) 261 -> 234 ({256, 32}, 128
// x 1), (32, 1024, 4096) 247 -> 229, (256, 1024, 256) 133 -> 118, (32, 512, 4096) 125 ->
// 117, (64, 256, 2048) 65 -> 61.  Without an even split the wide tiles lose ((64, 512,
// 4096): 1024 slices on 152 CTAs, 265 against 246 on the register path).  The gradient
// kernel likewise: (64, 2048, 1024) 419 -> 395 ({128, 64} x 4), (128, 1024, 1024) 448 -> 391.
// A tile wider than D is never taken: its boxes would be mostly padding ((128, 1024, 64)
// took {256, 32} at 43 us).  Forward scans of at least kWide64MinSteps steps also take
// 64-channel slices ({64, 128}, 512 threads, one CTA per SM) by the same rule, measured on
// GB300 against the 32-channel default (us per call): (32, 4096, 256) 62.4 -> 61.3, (8, 8192,
// 1024) 125.7 -> 117.4, (19, 4096, 512) 78.8 -> 75.2, (38, 4096, 256) 80.8 -> 75.9, (4, 8192,
// 2048) 127.1 -> 117.7, (2, 32768, 4096) 522 -> 470; shorter sequences lose ((76, 2048, 256)
// 73.8 -> 75.4, (32, 2048, 256) 31.7 -> 32.8) and so does the gradient ((32, 4096, 256) 101.9
// -> 103.5).
int wide_slices(int64_t B, int64_t L, int64_t D, int sm_count, bool backward, int64_t *grid) {
    if (L < kWideMinSteps) return 0;
    for (int td : {256, 128, 64}) {
        if (td > D || (td == 64 && (backward || L < kWide64MinSteps))) continue;
        const int64_t slices = B * ((D + td - 1) / td);
        const int64_t k = (slices + sm_count - 1) / sm_count;        // slices per CTA
        if (slices % k == 0 && (slices / k) * 100 >= (int64_t)kWideMinGridPct * sm_count) {
            *grid = slices / k;
            return td;
        }
    }
    return 0;
}

void default_tile(int64_t B, int64_t L, int64_t D, int sm_count, bool own, bool twopass, bool backward, int dtype,
                  int *tile_d, int *tile_t, int *stages) {
    if (dtype != kDtypeF32) {
        *tile_d = 32;
        *tile_t = tile_t_16(L);
        *stages = *tile_t == 256 ? 2 : 6;
        return;
    }
    own = own || twopass;
    if (backward) {   // three boxes per stage
        if (own) { *tile_d = 32; *tile_t = 128; *stages = 2; return; }
        if (D >= 64) { *tile_d = 64; *tile_t = 128; *stages = 2; }
        else { *tile_d = 32; *tile_t = 128; *stages = 2; }
        return;
    }
    // fp32 slice-owner and two-pass modes: a 2-deep ring.  Each stage is refilled
    // as soon as its tile is in registers, so up to three tiles are in flight per
    // CTA; on GB300 a 3-deep ring (four in flight) measured 9-11 % slower at every
    // shape (lower DRAM efficiency, not too few bytes in flight).
    if (own && !twopass && !backward) {
        // Slices just past one round of the {32, 128} CTAs (two per SM): smaller CTAs (128
        // threads, 64-step tiles) that take them all in one round.  Measured on GB300 (us per
        // call, {32, 128, 2} -> this): 320 slices (40, 4096, 256) 102 -> 87 and (10, 4096, 1024)
        // 102 -> 86 with a 4-deep ring; 352 slices (44, 8192, 256) 201 -> 174 (4-deep); 384
        // slices (48, 4096, 256) 103 -> 94, (12, 4096, 1024) 103 -> 92, (24, 4096, 512)
        // 103 -> 93 with a 3-deep ring (the 4-deep one there: 107, 103, 105).  From 448
        // slices on the spread {32, 128} grid stays ahead.
        const int64_t slices = B * ((D + 31) / 32), c1 = 2 * (int64_t)sm_count;
        *tile_d = 32;
        if (slices > c1 && slices * 100 <= c1 * 120) { *tile_t = 64; *stages = 4; return; }
        if (slices * 100 > c1 * 120 && slices * 100 <= c1 * 133) { *tile_t = 64; *stages = 3; return; }
        *tile_t = 128;
        *stages = 2;
        return;
    }
    if (own) { *tile_d = 32; *tile_t = 128; *stages = 2; return; }
    if (D >= 64) { *tile_d = 64; *tile_t = 128; *stages = 2; }
    else { *tile_d = 32; *tile_t = 128; *stages = 3; }
}

// Chain mode (chain.cu): its own tile (the first compiled chain variant of the storage type,
// or the one opt names), every resident CTA launched: resolver CTAs first, one group of warps
// per slice, then workers; the look-back words of every tile (three per channel).
linrec_status_t plan_chain(int64_t B, int64_t L, int64_t D, int sm_count, int ctas_per_sm,
                           const linrec_options_t *opt, linrec_plan_t *plan, int *variant_index, int dtype) {
    int n = 0;
    const ChunkedVariant *vars = chain_variants(dtype, &n);
    const ChunkedVariant *v = nullptr;
    // fp32: 256-step tiles for long sequences, 128-step ones below (the 16-bit variant has 256)
    const int want_t = opt->tile_t ? opt->tile_t : (dtype == kDtypeF32 ? (L >= kChainLongSteps ? 256 : 128) : 0);
    for (int i = 0; i < n && !v; ++i) {
        const ChunkedVariant &c = vars[i];
        if ((opt->tile_d == 0 || opt->tile_d == c.tile_d) && (want_t == 0 || want_t == c.tile_t) &&
            (opt->stages == 0 || opt->stages == c.stages) && (opt->segments == 0 || opt->segments == c.segments) &&
            (opt->vec == 0 || opt->vec == c.cpt)) {
            v = &c;
            if (variant_index) *variant_index = i;
        }
    }
    if (!v) return LINREC_ERR_INVALID_VALUE;
    plan->chain = 1;
    plan->vec = v->cpt;
    plan->tile_d = v->tile_d;
    plan->tile_t = v->tile_t;
    plan->segments = v->segments;
    plan->stages = v->stages;
    plan->threads = v->threads;
    plan->smem_bytes = v->smem_bytes;
    const int64_t slices = B * ((D + v->tile_d - 1) / v->tile_d);
    plan->chunks = (L + v->tile_t - 1) / v->tile_t;
    plan->n_tiles = slices * plan->chunks;
    int per_sm = ctas_per_sm;
    if (per_sm <= 0) {
        per_sm = (int)((227 * 1024) / (v->smem_bytes + 1024));
        if (per_sm < 1) per_sm = 1;
    }
    if (opt->ctas_per_sm > 0 && opt->ctas_per_sm < per_sm) per_sm = opt->ctas_per_sm;
    int cpg = 0, gpc = 0;
    const int64_t n_res = chain_layout(slices, v->threads / 32, &cpg, &gpc);
    // chain mode is for few slices: each resolver group serves one slice's channels, at most one
    // group per warp of at most kChainMaxResolvers CTAs
    if (n_res > kChainMaxResolvers) return LINREC_ERR_INVALID_VALUE;
    int64_t grid = (int64_t)sm_count * per_sm;
    if (grid > n_res + plan->n_tiles) grid = n_res + plan->n_tiles;
    if (grid <= n_res) return LINREC_ERR_INVALID_VALUE;   // no room for a worker beside the resolvers
    plan->grid = grid;
    plan->workspace_bytes = kWorkspaceHead + (size_t)3 * (size_t)plan->n_tiles * (size_t)v->tile_d * 8u;
    return LINREC_OK;
}

// Speculative mode (chunk_mode 6): the {32, 128, 2-stage} tile, whose fixed copies hold the two
// modes (a 3-stage ring measured 4-11 % slower: (1, 1048576, 64) 148.4 -> 154.8 us); G segments
// per sequence (opt->group, else the largest divisor of L with at least kSpecMinSteps steps per
// segment, at most kSpecMaxSegments, and slices within one round of kSpecCtasPerSm CTAs per SM:
// the repair copy's registers hold it to two, and a fixed figure gives the same G with or without
// the occupancy query); one CTA per slice of the (B * G, L / G, D) view in both launches; the
// segments' maps as plain floats (two per channel and slice).
linrec_status_t plan_speculative(int64_t B, int64_t L, int64_t D, int sm_count, int ctas_per_sm,
                                 const linrec_options_t *opt, linrec_plan_t *plan, int *variant_index) {
    int n = 0;
    const ChunkedVariant *vars = chunked_variants(&n);
    const ChunkedVariant *v = nullptr;
    for (int i = 0; i < n && !v; ++i) {
        const ChunkedVariant &c = vars[i];
        if (c.tile_d == 32 && c.tile_t == 128 && c.segments == 8 && c.stages == 2 && !c.blocks && !c.chain &&
            (opt->tile_d == 0 || opt->tile_d == 32) && (opt->tile_t == 0 || opt->tile_t == 128) &&
            (opt->stages == 0 || opt->stages == 2) && (opt->segments == 0 || opt->segments == 8) &&
            (opt->vec == 0 || opt->vec == 1)) {
            v = &c;
            if (variant_index) *variant_index = i;
        }
    }
    if (!v) return LINREC_ERR_INVALID_VALUE;
    int per_sm = ctas_per_sm;
    if (per_sm <= 0) {
        per_sm = (int)((227 * 1024) / (v->smem_bytes + 1024));
        if (per_sm < 1) per_sm = 1;
    }
    if (opt->ctas_per_sm > 0 && opt->ctas_per_sm < per_sm) per_sm = opt->ctas_per_sm;
    const int64_t spb = (D + v->tile_d - 1) / v->tile_d;
    const int64_t round = (int64_t)sm_count * per_sm;
    int64_t G = 0;
    if (opt->group > 0) {
        G = opt->group;
        if (L % G != 0 || L / G < kSpecMinSteps || G > kSpecMaxSegments) return LINREC_ERR_INVALID_VALUE;
    } else {
        const int64_t per_sm_g = per_sm < kSpecCtasPerSm ? per_sm : kSpecCtasPerSm;
        int64_t most = (int64_t)sm_count * per_sm_g / (B * spb);
        if (most > kSpecMaxSegments) most = kSpecMaxSegments;
        for (int64_t g = most; g >= 2 && G == 0; --g)
            if (L % g == 0 && L / g >= kSpecMinSteps) G = g;
    }
    if (G < 2) return LINREC_ERR_INVALID_VALUE;
    plan->speculative = (int)G;
    plan->vec = 1;
    plan->tile_d = v->tile_d;
    plan->tile_t = v->tile_t;
    plan->segments = v->segments;
    plan->stages = v->stages;
    plan->threads = v->threads;
    plan->smem_bytes = v->smem_bytes;
    const int64_t slices = B * G * spb;
    plan->chunks = (L / G + v->tile_t - 1) / v->tile_t;
    plan->n_tiles = slices * plan->chunks;
    plan->grid = slices < round ? slices : round;
    plan->workspace_bytes = kWorkspaceHead + (size_t)2 * (size_t)slices * (size_t)v->tile_d * 4u;
    return LINREC_OK;
}

linrec_status_t plan_impl(int64_t B, int64_t L, int64_t D, int sm_count, int align_bytes, int ctas_per_sm,
                          const linrec_options_t *opt, linrec_plan_t *plan, int *variant_index,
                          bool backward = false, bool allow_twopass = true, int dtype = kDtypeF32) {
    linrec_options_t none = {};
    if (!opt) opt = &none;
    if (!plan || sm_count <= 0) return LINREC_ERR_INVALID_VALUE;
    int64_t n = 0;
    linrec_status_t st = check_sizes(B, L, D, &n);
    if (st != LINREC_OK) return st;
    *plan = linrec_plan_t{};
    if (n == 0) return LINREC_OK;

    const int eb = elem_bytes_of(dtype);
    if (backward && dtype != kDtypeF32) return LINREC_ERR_INVALID_VALUE;
    const bool tma_ok = align_bytes >= 16 && (D * eb) % 16 == 0 && D <= INT32_MAX && B <= INT32_MAX &&
                        L <= (int64_t)INT32_MAX - 1024;
    // 1. Wide slices, ahead of everything else (see wide_slices).
    int64_t wide_grid = 0;
    const int wide_td = (dtype == kDtypeF32 && opt->chunk_mode == 0 && opt->tile_d == 0 && opt->tile_t == 0 &&
                         (opt->path == LINREC_PATH_AUTO || opt->path == LINREC_PATH_CHUNKED) && tma_ok)
                            ? wide_slices(B, L, D, sm_count, backward, &wide_grid)
                            : 0;
    // 2. The register path when the channels alone keep enough loads in flight: a
    // forward scan with at least kRegcarryMinThreadsPerSm threads of 16 bytes of
    // channels per SM.  Measured on GB300, fp32: (256, 128, 4096) 6922 vs 6007 GB/s
    // for the chunked kernel; at 32768 channels it loses (4361 vs 5722 on (8, 4096,
    // 4096)).  16-bit storage: only below 256 steps, where the chunked kernel cannot use
    // its 256-step tiles ((256, 128, 4096) bfloat16 6391 vs 4638; (64, 512, 4096) 6309
    // vs 6574 for the chunked kernel).
    // 3. Otherwise the TMA-staged chunked kernel whenever its copies are legal; the
    // register path also takes misaligned pointers and rows that are not a multiple of
    // 16 bytes.
    int path = opt->path;
    if (path == LINREC_PATH_AUTO) {
        const int lanes = 16 / eb;            // channels in 16 bytes
        const bool many = !backward && D % lanes == 0 && align_bytes >= 16 &&
                          (dtype == kDtypeF32 || L < 256) &&
                          B * (D / lanes) >= kRegcarryMinThreadsPerSm * (int64_t)sm_count;
        path = (tma_ok && (!many || wide_td)) ? LINREC_PATH_CHUNKED : LINREC_PATH_REGCARRY;
    }
    plan->path = path;

    if (path == LINREC_PATH_REGCARRY) {
        // widest vector of channels (16 bytes at most) that the alignment and D allow
        const int maxv = 16 / eb;
        int vec = opt->vec;
        if (vec == 0) {
            vec = maxv;
            while (vec > 1 && (D % vec != 0 || align_bytes < eb * vec)) vec /= 2;
        }
        if (vec <= 0 || D % vec != 0 || align_bytes < eb * vec) return LINREC_ERR_INVALID_VALUE;
        // steps loaded ahead: 16 when threads are scarce (under 160 per SM) or L is short,
        // otherwise 8 (measured: (64, 1024, 4096) 6747 GB/s with 8, 6511 with 16)
        const int64_t per_sm = B * (D / vec) / sm_count;
        int prefetch = opt->prefetch ? opt->prefetch
                                     : (vec != maxv || per_sm < 160 || L <= 512) ? 16 : 8;
        const bool ok = dtype == kDtypeF32 ? regcarry_supported(vec, prefetch) : regcarry16_supported(vec, prefetch);
        if (!ok) return LINREC_ERR_INVALID_VALUE;
        plan->vec = vec;
        plan->prefetch = prefetch;
        const int64_t groups = B * (D / vec);
        // Few channel groups (fp32 forward; odd D and misaligned pointers land here): cut the
        // time axis into segments, a reduce launch and an apply launch with 8 steps in flight,
        // enough segments for about kSegBytesPerSm bytes of loads in flight per SM, each at
        // least kSegMinSteps long, at most kSegMax (the apply launch folds the earlier maps one
        // by one).  20 bytes per element instead of 12, but the channels alone would leave the
        // GPU idle: (7, 3000, 777) 1593 us in one pass.
        int64_t nseg = 1;
        if (dtype == kDtypeF32 && !backward && allow_twopass && opt->chunk_mode != 1 &&
            groups < kRegcarryMinThreadsPerSm * (int64_t)sm_count) {
            const int64_t want = kSegBytesPerSm * (int64_t)sm_count / (8 * 8 * vec);   // threads
            nseg = (want + groups - 1) / groups;
            if (nseg > L / kSegMinSteps) nseg = L / kSegMinSteps;
            if (nseg > kSegMax) nseg = kSegMax;
            if (nseg < 2) nseg = 1;
        }
        if (nseg > 1) {
            plan->twopass = 1;
            plan->segments = (int)nseg;
            plan->threads = kRegcarryThreads;
            plan->grid = (groups * nseg + kRegcarryThreads - 1) / kRegcarryThreads;
            plan->workspace_bytes = (size_t)2 * (size_t)nseg * (size_t)(B * D) * 4u;
            return LINREC_OK;
        }
        // Narrower blocks when there are few channel groups, so the grid still
        // covers every SM (at least two blocks per SM where the groups allow).
        int threads = kRegcarryThreads;
        while (threads > 32 && (groups + threads - 1) / threads < 2 * (int64_t)sm_count) threads /= 2;
        plan->threads = threads;
        plan->grid = (groups + threads - 1) / threads;
        return LINREC_OK;
    }
    if (path != LINREC_PATH_CHUNKED || !tma_ok) return LINREC_ERR_INVALID_VALUE;

    // Slice-owner mode when the channel slices alone give every SM work.
    // Otherwise each slice's chunks are spread over CTAs: joined by look-back
    // when the chains are short, or, for long chains (whose look-back would be
    // bound by how fast inclusive values travel down the chain), by the
    // two-pass mode: reduce, scan the aggregates, apply.
    if (opt->chunk_mode < 0 || opt->chunk_mode > 6) return LINREC_ERR_INVALID_VALUE;
    if (opt->chunk_mode == 3 && !allow_twopass) return LINREC_ERR_INVALID_VALUE;
    if ((opt->chunk_mode == 4 || opt->chunk_mode == 5) && backward) return LINREC_ERR_INVALID_VALUE;
    if (opt->group < 0 || (opt->group > 0 && opt->chunk_mode != 4 && opt->chunk_mode != 6))
        return LINREC_ERR_INVALID_VALUE;
    if (opt->chunk_mode == 5 && !wide_td)
        return plan_chain(B, L, D, sm_count, ctas_per_sm, opt, plan, variant_index, dtype);
    if (opt->chunk_mode == 6) {
        if (dtype != kDtypeF32 || backward) return LINREC_ERR_INVALID_VALUE;
        return plan_speculative(B, L, D, sm_count, ctas_per_sm, opt, plan, variant_index);
    }
    bool own = false, twopass = false, blk = false;
    if (wide_td) {
        own = true;
    } else if (opt->chunk_mode == 0) {
        const int td = opt->tile_d ? opt->tile_d : 32;
        // fp32 forward: slice-owner from kOwnMinSlicesPct % of the SM count on (128 slices of
        // 32 channels on 152 SMs: (16, 4096, 256) 57 -> 44 us, (1, 32768, 4096) 406 -> 333
        // against the look-back and two-pass modes); otherwise from one slice per SM
        const int64_t need = (dtype == kDtypeF32 && !backward) ? ((int64_t)sm_count * kOwnMinSlicesPct + 99) / 100
                                                               : (int64_t)sm_count;
        own = B * ((D + td - 1) / td) >= need;
        const int tt = opt->tile_t ? opt->tile_t : (dtype == kDtypeF32 ? 128 : tile_t_16(L));
        if (dtype == kDtypeF32 && !backward && (L + tt - 1) / tt <= kOwnShortChunks) own = true;
        twopass = !own && allow_twopass && (L + tt - 1) / tt >= kTwoPassMinChunks;
        const bool plain = dtype == kDtypeF32 && !backward && opt->tile_d == 0 && opt->tile_t == 0 &&
                           opt->stages == 0 && opt->segments == 0 && opt->vec == 0;
        if (twopass && plain) {
            // few long chains: speculative mode where its segments are long
            linrec_plan_t sp = *plan;
            int svi = -1;
            if (plan_speculative(B, L, D, sm_count, ctas_per_sm, opt, &sp, &svi) == LINREC_OK &&
                L / sp.speculative >= kSpecDefaultSteps) {
                *plan = sp;
                if (variant_index) *variant_index = svi;
                return LINREC_OK;
            }
        }
        if (twopass && plain && B * ((D + 31) / 32) >= kChainMinSlices)
            return plan_chain(B, L, D, sm_count, ctas_per_sm, opt, plan, variant_index, dtype);
    } else {
        own = opt->chunk_mode == 1;
        twopass = opt->chunk_mode == 3;
        blk = opt->chunk_mode == 4;
    }
    int tile_d = opt->tile_d, tile_t = opt->tile_t, stages = opt->stages;
    if (wide_td) {
        tile_d = wide_td;
        tile_t = 8192 / wide_td;              // 32 KB per box: {256, 32} or {128, 64}
        if (stages == 0) stages = 2;
    } else if (tile_d == 0 || tile_t == 0) {
        int dd, dt, ds;
        default_tile(B, L, D, sm_count, own, twopass || blk, backward, dtype, &dd, &dt, &ds);
        // blocks mode in 16-bit storage: the 256-step tile (the one compiled for it) at any L
        if (blk && dtype != kDtypeF32) { dt = 256; ds = 2; }
        if (tile_d == 0) tile_d = dd;
        if (tile_t == 0) tile_t = dt;
        if (stages == 0) stages = ds;
    }
    // vec on the chunked path: channels per thread (0 = the first variant of the tile)
    int cpt = opt->vec;
    int segs = opt->segments;
    if (cpt == 0 && segs == 0 && dtype != kDtypeF32 && !backward && tile_d == 32 && tile_t == 256 &&
        (stages == 0 || stages == 2))
        default_groups_16(B * ((D + 31) / 32), sm_count, own, twopass || blk, &cpt, &segs);
    const ChunkedVariant *v = find_variant(tile_d, tile_t, stages, cpt, segs, variant_index, backward, dtype, blk);
    if (!v && opt->stages == 0)
        v = find_variant(tile_d, tile_t, 0, cpt, segs, variant_index, backward, dtype, blk);
    if (!v) return LINREC_ERR_INVALID_VALUE;
    plan->lookback = (own || twopass || blk) ? 0 : 1;
    plan->twopass = twopass ? 1 : 0;
    // blocks mode: tiles per block, kBlockSteps time steps by default
    plan->blocks = blk ? (opt->group > 0 ? opt->group : (int)((kBlockSteps + v->tile_t - 1) / v->tile_t)) : 0;
    plan->vec = v->cpt;
    plan->tile_d = v->tile_d;
    plan->tile_t = v->tile_t;
    plan->segments = v->segments;
    plan->stages = v->stages;
    plan->threads = v->threads;
    plan->smem_bytes = v->smem_bytes;
    const int64_t spb = (D + v->tile_d - 1) / v->tile_d;
    plan->chunks = (L + v->tile_t - 1) / v->tile_t;
    plan->n_tiles = B * spb * plan->chunks;
    int per_sm = ctas_per_sm;
    if (per_sm <= 0) {
        per_sm = (int)((227 * 1024) / (v->smem_bytes + 1024));
        if (per_sm < 1) per_sm = 1;
    }
    if (opt->ctas_per_sm > 0 && opt->ctas_per_sm < per_sm) per_sm = opt->ctas_per_sm;
    int64_t grid = (int64_t)sm_count * per_sm;
    const int64_t n_blocks = blk ? B * spb * ((plan->chunks + plan->blocks - 1) / plan->blocks) : 0;
    const int64_t units = own ? B * spb : blk ? n_blocks : plan->n_tiles;   // slices, blocks or tiles
    if (grid > units) grid = units;
    if (wide_td && grid > wide_grid) {
        grid = wide_grid;                     // the even split chosen above
    } else if (own && dtype == kDtypeF32) {
        // Slices go round-robin, so every CTA works on the same time rows of adjacent slices
        // at once (whole contiguous rows for the DRAM).  The busiest CTA owns ceil(slices /
        // grid) of them.  When fewer than half the CTAs have a slice in that last round, the
        // few still running cannot keep the DRAM busy: then take the fewest CTAs that keep
        // the same maximum, so every CTA owns (nearly) as many slices and all finish together.
        // Measured on GB300 (us per call): (8, 4096, 4096) 284 -> 262, (16, 2048, 2048) 140 ->
        // 127, (48, 4096, 256) 119 -> 103, (40, 4096, 512) 173 -> 156; the gradient (8, 4096,
        // 4096) 436 -> 395, (48, 4096, 256) 192 -> 171; with a fuller last round
        // it loses ((64, 2048, 1024) 272 -> 280), and so it does in 16-bit storage, where the
        // CTAs' issue rate rather than the DRAM bounds the kernel ((8, 4096, 4096) 126 -> 140).
        const int64_t waves = (units + grid - 1) / grid;
        const int64_t last = units - (waves - 1) * grid;
        if (waves > 1 && 2 * last < grid) grid = (units + waves - 1) / waves;
    }
    plan->grid = grid;
    plan->workspace_bytes = kWorkspaceHead;
    if (twopass) plan->workspace_bytes += ((size_t)3 * (size_t)plan->n_tiles + (size_t)(B * spb)) *
                                          (size_t)v->tile_d * 4u;
    else if (blk) plan->workspace_bytes += (size_t)3 * (size_t)n_blocks * (size_t)v->tile_d * 8u;
    else if (!own) plan->workspace_bytes += (size_t)3 * (size_t)plan->n_tiles * (size_t)v->tile_d * 8u;
    return LINREC_OK;
}

// Device facts, queried once per device (takes g_mu briefly).
DeviceInfo *device_info(int dev) {
    std::lock_guard<std::mutex> lock(g_mu);
    DeviceInfo &di = g_devices[dev];
    if (!di.ready) {
        int major = 0, minor = 0, sms = 0;
        if (cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev) != cudaSuccess ||
            cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev) != cudaSuccess ||
            cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) {
            cudaGetLastError();
            return nullptr;
        }
        di.supported = (major == 10 && minor == 3);
        di.sm_count = sms;
        di.ready = true;
    }
    return &di;
}

bool get_encoder() {
    static std::once_flag once;
    std::call_once(once, [] {
        void *fn = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000, cudaEnableDefault, &q) ==
                cudaSuccess && q == cudaDriverEntryPointSuccess && fn)
            g_encode = reinterpret_cast<EncodeTiledFn>(fn);
        cudaGetLastError();
    });
    return g_encode != nullptr;
}

// The resident CTAs per SM cached in `slot`, queried with `query` the first time.
template <typename Q>
int cached_ctas(std::atomic<int> &slot, Q query) {
    int c = slot.load(std::memory_order_relaxed);
    if (c > 0) return c;
    if (query(&c) != cudaSuccess || c <= 0) {
        cudaGetLastError();
        return 0;
    }
    slot.store(c, std::memory_order_relaxed);
    return c;
}

bool encode_map(CUtensorMap *map, const void *base, int64_t B, int64_t L, int64_t D, int tile_d, int tile_t,
                int dtype = kDtypeF32) {
    const cuuint64_t eb = (cuuint64_t)elem_bytes_of(dtype);
    const cuuint64_t dims[3] = {(cuuint64_t)D, (cuuint64_t)L, (cuuint64_t)B};
    const cuuint64_t strides[2] = {(cuuint64_t)D * eb, (cuuint64_t)L * (cuuint64_t)D * eb};
    const cuuint32_t box[3] = {(cuuint32_t)tile_d, (cuuint32_t)tile_t, 1u};
    const cuuint32_t estr[3] = {1u, 1u, 1u};
    const CUtensorMapDataType type = dtype == kDtypeBF16  ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16
                                     : dtype == kDtypeF16 ? CU_TENSOR_MAP_DATA_TYPE_FLOAT16
                                                          : CU_TENSOR_MAP_DATA_TYPE_FLOAT32;
    return g_encode(map, type, 3, const_cast<void *>(base), dims, strides, box, estr,
                    CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                    CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// The workspace of (dev, stream, level, kind), grown in stream order and zeroed
// when (re)allocated.  Caller holds the stream's mutex.
Slot *workspace(int dev, cudaStream_t stream, size_t need, int level = 0, SlotKind kind = kSlotTagged) {
    Slot &s = stream_state(dev, stream)->slots[std::make_pair(level, (int)kind)];
    // While the stream is being captured into a CUDA graph nothing is allocated (the
    // graph would own the memory); a slot a captured call uses stays allocated for good,
    // since the graph keeps its address.
    cudaStreamCaptureStatus cap = cudaStreamCaptureStatusNone;
    if (cudaStreamIsCapturing(stream, &cap) != cudaSuccess) {
        cudaGetLastError();
        return nullptr;
    }
    if (cap != cudaStreamCaptureStatusNone) {
        if (s.bytes < need) return nullptr;
        s.captured = true;
        return &s;
    }
    if (s.bytes >= need) return &s;
    size_t bytes = (need + (1u << 20) - 1) & ~(size_t)((1u << 20) - 1);
    void *p = nullptr;
    if (cudaMallocAsync(&p, bytes, stream) != cudaSuccess) {
        cudaGetLastError();
        return nullptr;
    }
    if (cudaMemsetAsync(p, 0, bytes, stream) != cudaSuccess) {
        cudaGetLastError();
        cudaFreeAsync(p, stream);
        return nullptr;
    }
    if (s.base && !s.captured) cudaFreeAsync(s.base, stream);
    s.base = static_cast<unsigned char *>(p);
    s.bytes = bytes;
    s.captured = false;
    return &s;
}

// Chain mode: every resident CTA of its variant (from the occupancy API), one cooperative launch.
linrec_status_t scan_chain_locked(DeviceInfo *di, int dev, const void *a, const void *b, void *h, int64_t B,
                                  int64_t L, int64_t D, int dtype, cudaStream_t stream, const linrec_options_t *opt,
                                  int level, linrec_plan_t plan, int vi) {
    int nvar = 0;
    const ChunkedVariant *vars = chain_variants(dtype, &nvar);
    if (vi < 0 || vi >= nvar || vi >= 8 || dtype < 0 || dtype > 2) return LINREC_ERR_INVALID_VALUE;
    const int per_sm = cached_ctas(di->chain_ctas_per_sm[dtype][vi],
                                   [&](int *c) { return chunked_ctas_per_sm(&vars[vi], c, dtype); });
    if (per_sm <= 0) return LINREC_ERR_LAUNCH;
    linrec_status_t st = plan_chain(B, L, D, di->sm_count, per_sm, opt, &plan, &vi, dtype);
    if (st != LINREC_OK) return st;
    if (!get_encoder()) return LINREC_ERR_LAUNCH;
    ChunkedLaunch p;
    p.variant = &vars[vi];
    p.dtype = dtype;
    if (!encode_map(&p.map_a, a, B, L, D, plan.tile_d, plan.tile_t, dtype) ||
        !encode_map(&p.map_b, b, B, L, D, plan.tile_d, plan.tile_t, dtype))
        return LINREC_ERR_LAUNCH;
    Slot *ws = workspace(dev, stream, plan.workspace_bytes, level);
    if (!ws) return LINREC_ERR_WORKSPACE;
    p.h = h;
    p.L = L;
    p.D = D;
    p.slices_per_batch = (D + plan.tile_d - 1) / plan.tile_d;
    p.n_slices = B * p.slices_per_batch;
    p.chunks = plan.chunks;
    p.n_tiles = plan.n_tiles;
    p.grid = plan.grid;
    p.mode = kModeChain;
    p.ctrl = reinterpret_cast<Control *>(ws->base);
    p.words = reinterpret_cast<unsigned long long *>(ws->base + kWorkspaceHead);
    p.status = opt->d_status ? opt->d_status : &p.ctrl->status;
    p.spin_limit = opt->spin_limit > 0 ? opt->spin_limit : kDefaultSpinLimit;
    p.silent_tile = opt->test_silent_tile > 0 ? opt->test_silent_tile - 1 : -1;
    p.h_init = opt->h_init;
    p.h_last = opt->h_last;
    if (launch_chunked(p, stream) != cudaSuccess) {
        cudaGetLastError();
        return LINREC_ERR_LAUNCH;
    }
    return LINREC_OK;
}

// Speculative mode: the (B * G, L / G, D) view of a, b and h, the speculative launch, then the
// repair launch.
linrec_status_t scan_spec_locked(DeviceInfo *di, int dev, const void *a, const void *b, void *h, int64_t B,
                                 int64_t L, int64_t D, cudaStream_t stream, const linrec_options_t *opt, int level,
                                 linrec_plan_t plan, int vi) {
    int nvar = 0;
    const ChunkedVariant *vars = chunked_variants(&nvar);
    if (vi < 0 || vi >= nvar || vi >= 64) return LINREC_ERR_INVALID_VALUE;
    const int per_sm = cached_ctas(di->ctas_per_sm[kDtypeF32][vi],
                                   [&](int *c) { return chunked_ctas_per_sm(&vars[vi], c, kDtypeF32); });
    if (per_sm <= 0) return LINREC_ERR_LAUNCH;
    linrec_status_t st = plan_speculative(B, L, D, di->sm_count, per_sm, opt, &plan, &vi);
    if (st != LINREC_OK) return st;
    if (!get_encoder()) return LINREC_ERR_LAUNCH;
    const int64_t G = plan.speculative, Bv = B * G, Lv = L / G;
    ChunkedLaunch p;
    p.variant = &vars[vi];
    p.dtype = kDtypeF32;
    if (!encode_map(&p.map_a, a, Bv, Lv, D, plan.tile_d, plan.tile_t) ||
        !encode_map(&p.map_b, b, Bv, Lv, D, plan.tile_d, plan.tile_t))
        return LINREC_ERR_LAUNCH;
    Slot *ws = workspace(dev, stream, kWorkspaceHead, level);
    if (!ws) return LINREC_ERR_WORKSPACE;
    Slot *arrays = workspace(dev, stream, plan.workspace_bytes - kWorkspaceHead, level, kSlotArrays);
    if (!arrays) return LINREC_ERR_WORKSPACE;
    p.h = h;
    p.L = Lv;
    p.D = D;
    p.slices_per_batch = (D + plan.tile_d - 1) / plan.tile_d;
    p.n_slices = Bv * p.slices_per_batch;
    p.chunks = plan.chunks;
    p.n_tiles = plan.n_tiles;
    p.grid = plan.grid;
    p.mode = kModeSpec;
    p.group = (int)G;
    p.ctrl = reinterpret_cast<Control *>(ws->base);
    p.words = reinterpret_cast<unsigned long long *>(arrays->base);
    p.status = opt->d_status ? opt->d_status : &p.ctrl->status;
    p.spin_limit = opt->spin_limit > 0 ? opt->spin_limit : kDefaultSpinLimit;
    p.silent_tile = -1;
    p.h_init = opt->h_init;
    p.h_last = opt->h_last;
    if (launch_chunked(p, stream) != cudaSuccess) {
        cudaGetLastError();
        return LINREC_ERR_LAUNCH;
    }
    p.mode = kModeRepair;
    if (launch_chunked(p, stream) != cudaSuccess) {
        cudaGetLastError();
        return LINREC_ERR_LAUNCH;
    }
    return LINREC_OK;
}

// The forward scan, arguments checked, the stream's mutex held.  `level` is 0 for a caller's
// problem and 1 for the two-pass mode's scan of its tile aggregates (always fp32).
linrec_status_t scan_locked(DeviceInfo *di, int dev, const void *a, const void *b, void *h, int64_t B,
                            int64_t L, int64_t D, int dtype, cudaStream_t stream, const linrec_options_t *opt,
                            int level) {
    const float *h_init = opt->h_init;
    float *h_last = opt->h_last;
    const int align = align_of(a, b, h);
    linrec_plan_t plan;
    int vi = -1;
    linrec_status_t st = plan_impl(B, L, D, di->sm_count, align, 0, opt, &plan, &vi, false, level < kTwoPassLevels,
                                   dtype);
    if (st != LINREC_OK) return st;

    if (plan.path == LINREC_PATH_REGCARRY && plan.twopass) {
        // segmented: the per-segment maps in an array slot of this stream
        Slot *arrays = workspace(dev, stream, plan.workspace_bytes, level, kSlotArrays);
        if (!arrays) return LINREC_ERR_WORKSPACE;
        float *aggA = reinterpret_cast<float *>(arrays->base);
        float *aggB = aggA + (int64_t)plan.segments * B * D;
        cudaError_t err = launch_regcarry_segmented(plan.vec, plan.threads, static_cast<const float *>(a),
                                                    static_cast<const float *>(b), static_cast<float *>(h), B, L, D,
                                                    plan.segments, h_init, h_last, aggA, aggB, stream);
        return err == cudaSuccess ? LINREC_OK : LINREC_ERR_LAUNCH;
    }
    if (plan.path == LINREC_PATH_REGCARRY) {
        cudaError_t err =
            dtype == kDtypeF32
                ? launch_regcarry(plan.vec, plan.prefetch, plan.threads, static_cast<const float *>(a),
                                  static_cast<const float *>(b), static_cast<float *>(h), B, L, D, h_init, h_last,
                                  stream)
                : launch_regcarry16(dtype, plan.vec, plan.prefetch, plan.threads, a, b, h, B, L, D, h_init, h_last,
                                    stream);
        return err == cudaSuccess ? LINREC_OK : LINREC_ERR_LAUNCH;
    }

    if (plan.chain) return scan_chain_locked(di, dev, a, b, h, B, L, D, dtype, stream, opt, level, plan, vi);
    if (plan.speculative) return scan_spec_locked(di, dev, a, b, h, B, L, D, stream, opt, level, plan, vi);

    // chunked: resident CTAs per SM from the occupancy API, then the real plan
    int nvar = 0;
    const ChunkedVariant *variants = variants_of(false, dtype, &nvar);
    if (vi < 0 || vi >= 64 || dtype < 0 || dtype > 2) return LINREC_ERR_INVALID_VALUE;
    const int per_sm = cached_ctas(di->ctas_per_sm[dtype][vi],
                                   [&](int *c) { return chunked_ctas_per_sm(&variants[vi], c, dtype); });
    if (per_sm <= 0) return LINREC_ERR_LAUNCH;
    st = plan_impl(B, L, D, di->sm_count, align, per_sm, opt, &plan, &vi, false, level < kTwoPassLevels,
                   dtype);
    if (st != LINREC_OK) return st;
    if (!get_encoder()) return LINREC_ERR_LAUNCH;

    ChunkedLaunch p;
    p.variant = &variants[vi];
    p.dtype = dtype;
    if (!encode_map(&p.map_a, a, B, L, D, plan.tile_d, plan.tile_t, dtype) ||
        !encode_map(&p.map_b, b, B, L, D, plan.tile_d, plan.tile_t, dtype))
        return LINREC_ERR_LAUNCH;
    // two-pass: the Control block in the tagged slot (for the status word), the
    // per-tile arrays in an array slot
    Slot *ws = workspace(dev, stream, plan.twopass ? kWorkspaceHead : plan.workspace_bytes, level);
    if (!ws) return LINREC_ERR_WORKSPACE;
    Slot *arrays = nullptr;
    if (plan.twopass) {
        arrays = workspace(dev, stream, plan.workspace_bytes - kWorkspaceHead, level, kSlotArrays);
        if (!arrays) return LINREC_ERR_WORKSPACE;
    }
    p.h = h;
    p.L = L;
    p.D = D;
    p.slices_per_batch = (D + plan.tile_d - 1) / plan.tile_d;
    p.n_slices = B * p.slices_per_batch;
    p.chunks = plan.chunks;
    p.n_tiles = plan.n_tiles;
    p.grid = plan.grid;
    p.mode = plan.twopass ? kModeReduce : plan.blocks ? kModeBlocks : plan.lookback ? kModeLookback : kModeOwn;
    p.group = plan.blocks;
    p.ctrl = reinterpret_cast<Control *>(ws->base);
    p.words = reinterpret_cast<unsigned long long *>(arrays ? arrays->base : ws->base + kWorkspaceHead);
    p.status = opt->d_status ? opt->d_status : &p.ctrl->status;
    p.spin_limit = opt->spin_limit > 0 ? opt->spin_limit : kDefaultSpinLimit;
    p.silent_tile = opt->test_silent_tile > 0 ? opt->test_silent_tile - 1 : -1;
    p.h_init = h_init;
    p.h_last = h_last;
    cudaError_t err = launch_chunked(p, stream);
    if (err != cudaSuccess) {
        cudaGetLastError();
        return LINREC_ERR_LAUNCH;
    }
    if (!plan.twopass) return LINREC_OK;

    // Two-pass mode: the per-tile maps form a (1, chunks, n_slices * tile_d) problem, row-major
    // by tile id; its scan gives every tile's inclusive value.  Then the apply launch.
    float *tileA = reinterpret_cast<float *>(p.words);
    float *tileB = tileA + p.n_tiles * plan.tile_d;
    float *tileH = tileB + p.n_tiles * plan.tile_d;
    linrec_options_t inner = {};
    inner.d_status = p.status;
    inner.spin_limit = opt->spin_limit;
    st = scan_locked(di, dev, tileA, tileB, tileH, 1, p.chunks, p.n_slices * plan.tile_d, kDtypeF32, stream, &inner,
                     level + 1);
    if (st != LINREC_OK) return st;
    p.mode = kModeApply;
    p.grid = plan.grid;
    err = launch_chunked(p, stream);
    if (err != cudaSuccess) {
        cudaGetLastError();
        return LINREC_ERR_LAUNCH;
    }
    return LINREC_OK;
}

// The (B, D, L) dispatcher: vector width, one pass or two, segment length.
linrec_status_t plan_bdl_impl(int64_t B, int64_t D, int64_t L, int dtype, int sm_count, int align_bytes,
                              const linrec_options_t *opt, linrec_plan_t *plan, int64_t *seg_len_out) {
    linrec_options_t none = {};
    if (!opt) opt = &none;
    if (!plan || sm_count <= 0 || dtype < 0 || dtype > 2) return LINREC_ERR_INVALID_VALUE;
    int64_t n = 0;
    linrec_status_t st = check_sizes(B, L, D, &n);
    if (st != LINREC_OK) return st;
    *plan = linrec_plan_t{};
    plan->path = LINREC_PATH_ROWS;
    if (opt->path != LINREC_PATH_AUTO && opt->path != LINREC_PATH_ROWS) return LINREC_ERR_INVALID_VALUE;
    if (opt->chunk_mode != 0 && opt->chunk_mode != 1 && opt->chunk_mode != 3) return LINREC_ERR_INVALID_VALUE;
    if (n == 0) return LINREC_OK;
    const int eb = elem_bytes_of(dtype);
    // Widest lane vector that L and the pointers allow: 16 bytes for fp32, 32 (two
    // 16-byte accesses) for 16-bit storage, whose chunks would otherwise spend more
    // issue slots on the shuffle scan than on the elements (measured on GB300:
    // (32, 256, 4096) bfloat16 at 6071 GB/s against 5520 with 16-byte lanes).
    int vec = opt->vec;
    if (vec == 0) {
        vec = (eb == 2 ? 32 : 16) / eb;
        while (vec > 1 && (L % vec != 0 || align_bytes < (eb * vec < 16 ? eb * vec : 16))) vec /= 2;
    }
    // 32-byte vectors are two 16-byte accesses: 16-byte alignment suffices
    if (vec <= 0 || (vec & (vec - 1)) != 0 || vec * eb > 32 || L % vec != 0 ||
        align_bytes < (eb * vec < 16 ? eb * vec : 16))
        return LINREC_ERR_INVALID_VALUE;
    const int64_t R = B * D;
    const int64_t ch = 32 * (int64_t)vec;
    if (opt->rows_per_warp < 0 || (opt->rows_per_warp > 0 && opt->chunk_mode == 3)) return LINREC_ERR_INVALID_VALUE;
    bool twopass = opt->chunk_mode == 3;
    if (opt->chunk_mode == 0)
        twopass = opt->rows_per_warp == 0 && R < kRowsMinWarps * sm_count && L >= 2 * kRowsMinSegChunks * ch;
    int64_t seg_len = L, nseg = 1;
    if (twopass) {
        const int64_t want = (kRowsTargetWarps * sm_count + R - 1) / R;   // segments per row
        int64_t len = (L + want - 1) / want;
        len = (len + ch - 1) / ch * ch;
        if (len < kRowsMinSegChunks * ch) len = kRowsMinSegChunks * ch;
        seg_len = len;
        nseg = (L + seg_len - 1) / seg_len;
        if (nseg < 2 && opt->chunk_mode == 0) {
            twopass = false;
            seg_len = L;
            nseg = 1;
        }
    }
    int64_t k = 1;                            // rows per warp (one pass)
    if (!twopass) {
        if (opt->rows_per_warp > 0) {
            k = opt->rows_per_warp;
        } else {
            k = (eb == 4 ? kRowsStreamElems : kRowsStreamElems16) / L;
            const int64_t cap = R / (kRowsStreamWarps * sm_count);
            if (k > cap) k = cap;
        }
        if (k < 1) k = 1;
        if (k > R) k = R;
    }
    // loads in flight: 2 chunks (measured best on every shape with the default vectors)
    const int prefetch = opt->prefetch ? opt->prefetch : 2;
    if (!rows_supported(dtype, vec, prefetch)) return LINREC_ERR_INVALID_VALUE;
    const int64_t units = twopass ? R * nseg : (R + k - 1) / k;
    plan->vec = vec;
    plan->prefetch = prefetch;
    plan->tile_t = seg_len > INT32_MAX ? INT32_MAX : (int)seg_len;
    plan->tile_d = k > INT32_MAX ? INT32_MAX : (int)k;
    plan->chunks = nseg;
    plan->twopass = twopass ? 1 : 0;
    plan->threads = kRowsThreads;
    plan->n_tiles = units;
    plan->grid = (units * 32 + kRowsThreads - 1) / kRowsThreads;
    plan->workspace_bytes = twopass ? kWorkspaceHead + (size_t)(3 * nseg * R + R) * 4u : 0;
    if (seg_len_out) *seg_len_out = seg_len;
    return LINREC_OK;
}

// The (B, D, L) scan, arguments checked, the stream's mutex held.
linrec_status_t scan_bdl_locked(DeviceInfo *di, int dev, const void *a, const void *b, void *h, int64_t B,
                                int64_t D, int64_t L, int dtype, cudaStream_t stream, const linrec_options_t *opt) {
    linrec_plan_t plan;
    int64_t seg_len = 0;
    linrec_status_t st = plan_bdl_impl(B, D, L, dtype, di->sm_count, align_of(a, b, h), opt, &plan, &seg_len);
    if (st != LINREC_OK) return st;
    RowsLaunch p;
    p.dtype = dtype;
    p.vec = plan.vec;
    p.prefetch = plan.prefetch;
    p.a = a;
    p.b = b;
    p.h = h;
    p.R = B * D;
    p.L = L;
    p.seg_len = seg_len;
    p.nseg = plan.chunks;
    p.rows_per_unit = plan.twopass ? 1 : plan.tile_d;
    p.h_init = opt->h_init;
    p.h_last = opt->h_last;
    if (!plan.twopass) {
        p.mode = kRowsFull;
        if (launch_rows(p, stream) != cudaSuccess) {
            cudaGetLastError();
            return LINREC_ERR_LAUNCH;
        }
        return LINREC_OK;
    }
    // Two passes: the segments' maps, laid out (1, segments, rows), scanned by the (B, L, D) path.
    Slot *ws = workspace(dev, stream, kWorkspaceHead, 0);            // control block: status word
    if (!ws) return LINREC_ERR_WORKSPACE;
    const size_t cells = (size_t)(p.nseg * p.R);
    Slot *arr = workspace(dev, stream, (3 * cells + (size_t)p.R) * 4u, 0, kSlotArrays);
    if (!arr) return LINREC_ERR_WORKSPACE;
    float *aggA = reinterpret_cast<float *>(arr->base);
    float *aggB = aggA + cells;
    float *aggH = aggB + cells;
    p.aggA = aggA;
    p.aggB = aggB;
    p.aggH = aggH;
    p.aggX = aggH + cells;
    p.mode = kRowsReduce;
    if (launch_rows(p, stream) != cudaSuccess) {
        cudaGetLastError();
        return LINREC_ERR_LAUNCH;
    }
    linrec_options_t inner = {};
    inner.d_status = opt->d_status ? opt->d_status : &reinterpret_cast<Control *>(ws->base)->status;
    inner.spin_limit = opt->spin_limit;
    st = scan_locked(di, dev, aggA, aggB, aggH, 1, p.nseg, p.R, kDtypeF32, stream, &inner, 1);
    if (st != LINREC_OK) return st;
    p.mode = kRowsApply;
    if (launch_rows(p, stream) != cudaSuccess) {
        cudaGetLastError();
        return LINREC_ERR_LAUNCH;
    }
    return LINREC_OK;
}

}  // namespace

extern "C" {

const char *linrec_status_string(linrec_status_t s) {
    switch (s) {
        case LINREC_OK: return "LINREC_OK";
        case LINREC_ERR_INVALID_VALUE: return "LINREC_ERR_INVALID_VALUE: bad size, NULL pointer or option";
        case LINREC_ERR_ALIAS: return "LINREC_ERR_ALIAS: h overlaps a or b";
        case LINREC_ERR_UNSUPPORTED_DEVICE: return "LINREC_ERR_UNSUPPORTED_DEVICE: needs compute capability 10.3";
        case LINREC_ERR_LAUNCH: return "LINREC_ERR_LAUNCH: a CUDA call failed while enqueueing";
        case LINREC_ERR_WORKSPACE: return "LINREC_ERR_WORKSPACE: look-back workspace allocation failed";
        case LINREC_ERR_LOOKBACK_TIMEOUT: return "LINREC_ERR_LOOKBACK_TIMEOUT: a tile gave up on its predecessor";
        case LINREC_ERR_TMA_TIMEOUT: return "LINREC_ERR_TMA_TIMEOUT: a bulk copy did not complete in time";
    }
    return "unknown linrec status";
}

int linrec_version(void) { return kVersion; }

int linrec_debug_checks(void) {
#ifdef LINREC_DEBUG
    return 1;
#else
    return 0;
#endif
}

linrec_status_t linrec_debug_bad_accesses(uint64_t *count, int64_t *first_offset, int64_t output_cap_bytes) {
    if (!count || !first_offset || output_cap_bytes < 0) return LINREC_ERR_INVALID_VALUE;
    using Report = cudaError_t (*)(unsigned long long *, long long *, long long);
    const Report reports[] = {checked_report_chunked,  checked_report_chunked16, checked_report_backward,
                              checked_report_regcarry, checked_report_regcarry16, checked_report_rows,
                              checked_report_chain,    checked_report_fixed,     checked_report_fixed16};
    unsigned long long total = 0;
    long long first = -1;
    for (Report r : reports) {
        unsigned long long c = 0;
        long long f = -1;
        if (r(&c, &f, (long long)output_cap_bytes) != cudaSuccess) {
            cudaGetLastError();
            return LINREC_ERR_LAUNCH;
        }
        total += c;
        if (first < 0 && c > 0) first = f;
    }
    *count = total;
    *first_offset = first;
    return LINREC_OK;
}

linrec_status_t linrec_plan_f32(int64_t B, int64_t L, int64_t D, int sm_count, int align_bytes, int ctas_per_sm,
                                const linrec_options_t *opt, linrec_plan_t *plan) {
    return plan_impl(B, L, D, sm_count, align_bytes, ctas_per_sm, opt, plan, nullptr);
}

size_t linrec_workspace_bytes(int64_t B, int64_t L, int64_t D) {
    int dev = 0, sms = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) !=
                                                  cudaSuccess || sms <= 0) {
        cudaGetLastError();
        return 0;
    }
    // the plan of a default call (the grid does not change the workspace)
    linrec_plan_t plan;
    if (plan_impl(B, L, D, sms, 16, 0, nullptr, &plan, nullptr) != LINREC_OK || plan.path != LINREC_PATH_CHUNKED)
        return 0;
    size_t total = plan.workspace_bytes;
    // each two-pass level scans its tile maps, a (1, chunks, slices * tile_d) problem with a
    // workspace of its own, which may itself take two-pass mode while level < kTwoPassLevels
    int64_t b = B, d = D;
    for (int level = 1; plan.twopass && plan.path == LINREC_PATH_CHUNKED; ++level) {
        const int64_t width = b * ((d + plan.tile_d - 1) / plan.tile_d) * plan.tile_d;
        linrec_plan_t inner;
        if (plan_impl(1, plan.chunks, width, sms, 16, 0, nullptr, &inner, nullptr, false, level < kTwoPassLevels) !=
            LINREC_OK)
            break;
        total += inner.workspace_bytes;
        b = 1;
        d = width;
        plan = inner;
    }
    return total;
}

}  // extern "C"

namespace {

// The forward entry points: argument checks, then the scan.  B, L, D are the
// batch, time and channel sizes in either layout; bdl selects the time-innermost
// (B, D, L) layout, otherwise the tensors are (B, L, D).
linrec_status_t scan_entry(int dtype, bool bdl, const void *a, const void *b, void *h, int64_t B, int64_t L,
                           int64_t D, void *stream_ptr, const linrec_options_t *opt) {
    linrec_options_t none = {};
    if (!opt) opt = &none;
    int64_t n = 0;
    linrec_status_t st = check_sizes(B, L, D, &n);
    if (st != LINREC_OK) return st;
    if (n == 0) return LINREC_OK;
    if (!a || !b || !h) return LINREC_ERR_INVALID_VALUE;
    const int64_t nb = n * elem_bytes_of(dtype);
    if (overlaps(h, a, nb) || overlaps(h, b, nb)) return LINREC_ERR_ALIAS;
    const float *h_init = opt->h_init;
    float *h_last = opt->h_last;
    const int64_t nstate = B * D * 4;
    if (h_init && (overlaps(h_init, nstate, h, nb) ||
                   (h_last && h_last != h_init && overlaps(h_init, h_last, nstate))))
        return LINREC_ERR_ALIAS;
    if (h_last && (overlaps(h_last, nstate, a, nb) || overlaps(h_last, nstate, b, nb) ||
                   overlaps(h_last, nstate, h, nb)))
        return LINREC_ERR_ALIAS;
    cudaStream_t stream = static_cast<cudaStream_t>(stream_ptr);

    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) {
        cudaGetLastError();
        return LINREC_ERR_LAUNCH;
    }
    DeviceInfo *di = device_info(dev);
    if (!di) return LINREC_ERR_LAUNCH;
    if (!di->supported) return LINREC_ERR_UNSUPPORTED_DEVICE;
    std::lock_guard<std::mutex> lock(stream_state(dev, stream)->mu);

    if (bdl) return scan_bdl_locked(di, dev, a, b, h, B, D, L, dtype, stream, opt);
    return scan_locked(di, dev, a, b, h, B, L, D, dtype, stream, opt, 0);
}

}  // namespace

extern "C" {

linrec_status_t linrec_scan_f32_ex(const float *a, const float *b, float *h, int64_t B, int64_t L, int64_t D,
                                   void *stream, const linrec_options_t *opt) {
    return scan_entry(kDtypeF32, false, a, b, h, B, L, D, stream, opt);
}

linrec_status_t linrec_scan_bf16_ex(const uint16_t *a, const uint16_t *b, uint16_t *h, int64_t B, int64_t L,
                                    int64_t D, void *stream, const linrec_options_t *opt) {
    return scan_entry(kDtypeBF16, false, a, b, h, B, L, D, stream, opt);
}

linrec_status_t linrec_scan_f16_ex(const uint16_t *a, const uint16_t *b, uint16_t *h, int64_t B, int64_t L,
                                   int64_t D, void *stream, const linrec_options_t *opt) {
    return scan_entry(kDtypeF16, false, a, b, h, B, L, D, stream, opt);
}

linrec_status_t linrec_scan_bf16(const uint16_t *a, const uint16_t *b, uint16_t *h, int64_t B, int64_t L,
                                 int64_t D, void *stream) {
    return scan_entry(kDtypeBF16, false, a, b, h, B, L, D, stream, nullptr);
}

linrec_status_t linrec_scan_f16(const uint16_t *a, const uint16_t *b, uint16_t *h, int64_t B, int64_t L, int64_t D,
                                void *stream) {
    return scan_entry(kDtypeF16, false, a, b, h, B, L, D, stream, nullptr);
}

linrec_status_t linrec_plan_16(int64_t B, int64_t L, int64_t D, int sm_count, int align_bytes, int ctas_per_sm,
                               const linrec_options_t *opt, linrec_plan_t *plan) {
    return plan_impl(B, L, D, sm_count, align_bytes, ctas_per_sm, opt, plan, nullptr, false, true, kDtypeBF16);
}

linrec_status_t linrec_scan_f32_bdl(const float *a, const float *b, float *h, int64_t B, int64_t D, int64_t L,
                                    void *stream) {
    return scan_entry(kDtypeF32, true, a, b, h, B, L, D, stream, nullptr);
}

linrec_status_t linrec_scan_f32_bdl_ex(const float *a, const float *b, float *h, int64_t B, int64_t D, int64_t L,
                                       void *stream, const linrec_options_t *opt) {
    return scan_entry(kDtypeF32, true, a, b, h, B, L, D, stream, opt);
}

linrec_status_t linrec_scan_bf16_bdl_ex(const uint16_t *a, const uint16_t *b, uint16_t *h, int64_t B, int64_t D,
                                        int64_t L, void *stream, const linrec_options_t *opt) {
    return scan_entry(kDtypeBF16, true, a, b, h, B, L, D, stream, opt);
}

linrec_status_t linrec_scan_f16_bdl_ex(const uint16_t *a, const uint16_t *b, uint16_t *h, int64_t B, int64_t D,
                                       int64_t L, void *stream, const linrec_options_t *opt) {
    return scan_entry(kDtypeF16, true, a, b, h, B, L, D, stream, opt);
}

linrec_status_t linrec_plan_bdl(int64_t B, int64_t D, int64_t L, int elem_bytes, int sm_count, int align_bytes,
                                const linrec_options_t *opt, linrec_plan_t *plan) {
    if (elem_bytes != 4 && elem_bytes != 2) return LINREC_ERR_INVALID_VALUE;
    return plan_bdl_impl(B, D, L, elem_bytes == 4 ? kDtypeF32 : kDtypeBF16, sm_count, align_bytes, opt, plan,
                         nullptr);
}

linrec_status_t linrec_scan_f32(const float *a, const float *b, float *h, int64_t B, int64_t L, int64_t D,
                                void *stream) {
    return linrec_scan_f32_ex(a, b, h, B, L, D, stream, nullptr);
}

linrec_status_t linrec_plan_f32_backward(int64_t B, int64_t L, int64_t D, int sm_count, int align_bytes,
                                         int ctas_per_sm, const linrec_options_t *opt, linrec_plan_t *plan) {
    return plan_impl(B, L, D, sm_count, align_bytes, ctas_per_sm, opt, plan, nullptr, true);
}

linrec_status_t linrec_scan_f32_backward_ex(const float *a, const float *h, const float *g, float *da, float *db,
                                            int64_t B, int64_t L, int64_t D, const float *h_init,
                                            const float *dh_last, float *dh_init, void *stream_ptr,
                                            const linrec_options_t *opt) {
    linrec_options_t none = {};
    if (!opt) opt = &none;
    int64_t n = 0;
    linrec_status_t st = check_sizes(B, L, D, &n);
    if (st != LINREC_OK) return st;
    if (n == 0) return LINREC_OK;
    if (!a || !g || !db || (da && !h)) return LINREC_ERR_INVALID_VALUE;
    const int64_t nb = n * 4, sb = B * D * 4;
    // outputs against inputs and each other; db may be g itself
    struct R { const void *p; int64_t bytes; };
    const R ins[] = {{a, nb}, {da ? h : nullptr, nb}, {g, nb}, {h_init, sb}, {dh_last, sb}};
    const R outs[] = {{da, nb}, {db, nb}, {dh_init, sb}};
    for (int i = 0; i < 3; ++i) {
        if (!outs[i].p) continue;
        for (int j = 0; j < 5; ++j) {
            if (!ins[j].p) continue;
            if (i == 1 && j == 2 && db == g) continue;
            if (overlaps(outs[i].p, outs[i].bytes, ins[j].p, ins[j].bytes)) return LINREC_ERR_ALIAS;
        }
        for (int j = i + 1; j < 3; ++j)
            if (outs[j].p && overlaps(outs[i].p, outs[i].bytes, outs[j].p, outs[j].bytes)) return LINREC_ERR_ALIAS;
    }
    cudaStream_t stream = static_cast<cudaStream_t>(stream_ptr);
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) {
        cudaGetLastError();
        return LINREC_ERR_LAUNCH;
    }
    DeviceInfo *di = device_info(dev);
    if (!di) return LINREC_ERR_LAUNCH;
    if (!di->supported) return LINREC_ERR_UNSUPPORTED_DEVICE;
    std::lock_guard<std::mutex> lock(stream_state(dev, stream)->mu);

    const uintptr_t u = reinterpret_cast<uintptr_t>(a) | reinterpret_cast<uintptr_t>(g) |
                        reinterpret_cast<uintptr_t>(db) | (da ? reinterpret_cast<uintptr_t>(da) |
                                                                reinterpret_cast<uintptr_t>(h) : 0u);
    const int align = (u & 15u) == 0 ? 16 : (u & 7u) == 0 ? 8 : 4;
    linrec_plan_t plan;
    int vi = -1;
    st = plan_impl(B, L, D, di->sm_count, align, 0, opt, &plan, &vi, true);
    if (st != LINREC_OK) return st;
    if (plan.path == LINREC_PATH_REGCARRY) {
        cudaError_t err = launch_regcarry_backward(plan.vec, plan.threads, a, h, g, da, db, B, L, D, h_init, dh_last,
                                                   dh_init, stream);
        return err == cudaSuccess ? LINREC_OK : LINREC_ERR_LAUNCH;
    }
    int nvar = 0;
    const ChunkedVariant *variants = backward_variants(&nvar);
    if (vi < 0 || vi >= 64) return LINREC_ERR_INVALID_VALUE;
    const int per_sm = cached_ctas(di->back_ctas_per_sm[vi],
                                   [&](int *c) { return backward_ctas_per_sm(&variants[vi], c); });
    if (per_sm <= 0) return LINREC_ERR_LAUNCH;
    st = plan_impl(B, L, D, di->sm_count, align, per_sm, opt, &plan, &vi, true);
    if (st != LINREC_OK) return st;
    if (!get_encoder()) return LINREC_ERR_LAUNCH;
    BackwardLaunch p;
    p.variant = &variants[vi];
    if (!encode_map(&p.map_g, g, B, L, D, plan.tile_d, plan.tile_t) ||
        !encode_map(&p.map_a, a, B, L, D, plan.tile_d, plan.tile_t) ||
        !encode_map(&p.map_h, da ? h : a, B, L, D, plan.tile_d, plan.tile_t))
        return LINREC_ERR_LAUNCH;
    // two-pass: the Control block in the tagged slot, the per-tile arrays in an array slot
    Slot *ws = workspace(dev, stream, plan.twopass ? kWorkspaceHead : plan.workspace_bytes);
    if (!ws) return LINREC_ERR_WORKSPACE;
    Slot *arrays = nullptr;
    if (plan.twopass) {
        arrays = workspace(dev, stream, plan.workspace_bytes - kWorkspaceHead, 0, kSlotArrays);
        if (!arrays) return LINREC_ERR_WORKSPACE;
    }
    p.a = a;
    p.da = da;
    p.db = db;
    p.L = L;
    p.D = D;
    p.slices_per_batch = (D + plan.tile_d - 1) / plan.tile_d;
    p.n_slices = B * p.slices_per_batch;
    p.chunks = plan.chunks;
    p.n_tiles = plan.n_tiles;
    p.grid = plan.grid;
    p.mode = plan.twopass ? kModeReduce : plan.lookback ? kModeLookback : kModeOwn;
    p.ctrl = reinterpret_cast<Control *>(ws->base);
    p.words = reinterpret_cast<unsigned long long *>(arrays ? arrays->base : ws->base + kWorkspaceHead);
    p.status = opt->d_status ? opt->d_status : &p.ctrl->status;
    p.spin_limit = opt->spin_limit > 0 ? opt->spin_limit : kDefaultSpinLimit;
    p.silent_tile = opt->test_silent_tile > 0 ? opt->test_silent_tile - 1 : -1;
    p.h_init = h_init;
    p.dh_last = dh_last;
    p.dh_init = dh_init;
    cudaError_t err = launch_backward(p, stream);
    if (err != cudaSuccess) {
        cudaGetLastError();
        return LINREC_ERR_LAUNCH;
    }
    if (!plan.twopass) return LINREC_OK;

    // Two-pass mode: the tiles' maps, in reversed chunk order, form a (1, chunks,
    // n_slices * tile_d) problem whose forward scan gives every tile's running c.
    float *tileA = reinterpret_cast<float *>(p.words);
    float *tileB = tileA + p.n_tiles * plan.tile_d;
    float *tileH = tileB + p.n_tiles * plan.tile_d;
    linrec_options_t inner = {};
    inner.d_status = p.status;
    inner.spin_limit = opt->spin_limit;
    st = scan_locked(di, dev, tileA, tileB, tileH, 1, p.chunks, p.n_slices * plan.tile_d, kDtypeF32, stream, &inner,
                     1);
    if (st != LINREC_OK) return st;
    p.mode = kModeApply;
    err = launch_backward(p, stream);
    if (err != cudaSuccess) {
        cudaGetLastError();
        return LINREC_ERR_LAUNCH;
    }
    return LINREC_OK;
}

linrec_status_t linrec_scan_f32_backward(const float *a, const float *h, const float *g, float *da, float *db,
                                         int64_t B, int64_t L, int64_t D, const float *h_init,
                                         const float *dh_last, float *dh_init, void *stream) {
    return linrec_scan_f32_backward_ex(a, h, g, da, db, B, L, D, h_init, dh_last, dh_init, stream, nullptr);
}

linrec_status_t linrec_scan_f32_carry(const float *a, const float *b, float *h, int64_t B, int64_t L, int64_t D,
                                      const float *h_init, float *h_last, void *stream) {
    linrec_options_t opt = {};
    opt.h_init = h_init;
    opt.h_last = h_last;
    return linrec_scan_f32_ex(a, b, h, B, L, D, stream, &opt);
}

linrec_status_t linrec_stream_status(void *stream_ptr) {
    cudaStream_t stream = static_cast<cudaStream_t>(stream_ptr);
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) {
        cudaGetLastError();
        return LINREC_ERR_LAUNCH;
    }
    unsigned char *base = nullptr;
    if (StreamState *ss = find_stream_state(dev, stream)) {
        std::lock_guard<std::mutex> lock(ss->mu);
        auto it = ss->slots.find(std::make_pair(0, (int)kSlotTagged));
        if (it != ss->slots.end()) base = it->second.base;
    }
    unsigned int word = 0;
    if (base) {
        Control *ctrl = reinterpret_cast<Control *>(base);
        if (cudaMemcpyAsync(&word, &ctrl->status, sizeof(word), cudaMemcpyDeviceToHost, stream) != cudaSuccess ||
            cudaStreamSynchronize(stream) != cudaSuccess) {
            cudaGetLastError();
            return LINREC_ERR_LAUNCH;
        }
        if (word != 0 && (cudaMemsetAsync(&ctrl->status, 0, sizeof(word), stream) != cudaSuccess ||
                          cudaStreamSynchronize(stream) != cudaSuccess)) {
            cudaGetLastError();
            return LINREC_ERR_LAUNCH;
        }
    }
    // failures of linrec_scan_f32_noalloc calls made without a status word of their own
    unsigned int fixed = 0;
    if (noalloc_take_status(dev, stream, &fixed) != cudaSuccess) {
        cudaGetLastError();
        return LINREC_ERR_LAUNCH;
    }
    word |= fixed;
    if (word == 0) return LINREC_OK;
    if (word & kStatusLookbackTimeout) return LINREC_ERR_LOOKBACK_TIMEOUT;
    if (word & kStatusTmaTimeout) return LINREC_ERR_TMA_TIMEOUT;
    return LINREC_ERR_LAUNCH;
}

linrec_status_t linrec_debug_set_epoch(void *stream_ptr, int fixed_array, uint32_t epoch) {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) {
        cudaGetLastError();
        return LINREC_ERR_LAUNCH;
    }
    if (fixed_array) {
        if (noalloc_set_epoch(dev, epoch) != cudaSuccess) {
            cudaGetLastError();
            return LINREC_ERR_WORKSPACE;
        }
        return LINREC_OK;
    }
    unsigned char *base = nullptr;
    if (StreamState *ss = find_stream_state(dev, static_cast<cudaStream_t>(stream_ptr))) {
        std::lock_guard<std::mutex> lock(ss->mu);
        auto it = ss->slots.find(std::make_pair(0, (int)kSlotTagged));
        if (it != ss->slots.end()) base = it->second.base;
    }
    if (!base) return LINREC_ERR_WORKSPACE;
    cudaStream_t stream = static_cast<cudaStream_t>(stream_ptr);
    Control *ctrl = reinterpret_cast<Control *>(base);
    if (cudaMemcpyAsync(&ctrl->epoch, &epoch, sizeof(epoch), cudaMemcpyHostToDevice, stream) != cudaSuccess ||
        cudaStreamSynchronize(stream) != cudaSuccess) {
        cudaGetLastError();
        return LINREC_ERR_LAUNCH;
    }
    return LINREC_OK;
}

linrec_status_t linrec_copy_f32(const float *src, float *dst, int64_t n, void *stream) {
    if (n < 0) return LINREC_ERR_INVALID_VALUE;
    if (n == 0) return LINREC_OK;
    if (!src || !dst) return LINREC_ERR_INVALID_VALUE;
    if (n > INT64_MAX / 8) return LINREC_ERR_INVALID_VALUE;
    if (overlaps(src, dst, n * 4)) return LINREC_ERR_ALIAS;
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) {
        cudaGetLastError();
        return LINREC_ERR_LAUNCH;
    }
    int sms = 0;
    {
        DeviceInfo *di = device_info(dev);
        if (!di) return LINREC_ERR_LAUNCH;
        if (!di->supported) return LINREC_ERR_UNSUPPORTED_DEVICE;
        sms = di->sm_count;
    }
    return launch_copy(src, dst, n, sms, static_cast<cudaStream_t>(stream)) == cudaSuccess ? LINREC_OK
                                                                                            : LINREC_ERR_LAUNCH;
}

}  // extern "C"
