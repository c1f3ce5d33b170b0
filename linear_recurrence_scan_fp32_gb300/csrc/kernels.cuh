// kernels.cuh -- interface between the host API (linrec_api.cu) and the
// kernel translation units.  Internal to liblinrec; not installed.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <stddef.h>
#include <stdint.h>

namespace linrec {

// Per-(device, stream) control block at the head of the look-back workspace.
// Zeroed once when allocated; afterwards the last CTA of every chunked launch
// resets the tile counter, the done counter and the abort word and advances
// the epoch, so no memset is needed between calls.
struct alignas(64) Control {
    unsigned long long tile_counter;  // next tile id to hand out (dynamic, in order)
    unsigned int done;                // CTAs of the current launch that have finished
    unsigned int epoch;               // launches completed on this workspace
    unsigned int status;              // OR of (1 << linrec_status_t) device-side failures
    unsigned int abort;               // set when a bulk copy timed out: stop taking tiles
    unsigned int pad[10];
};
static_assert(sizeof(Control) == 64, "control block layout");

constexpr unsigned int kStatusLookbackTimeout = 1u << 6;  // 1 << LINREC_ERR_LOOKBACK_TIMEOUT
constexpr unsigned int kStatusTmaTimeout = 1u << 7;       // 1 << LINREC_ERR_TMA_TIMEOUT

// How a, b and h are stored (the linrec_dtype_t values).  Arithmetic and
// carries are fp32 for all three.
constexpr int kDtypeF32 = 0;
constexpr int kDtypeBF16 = 1;
constexpr int kDtypeF16 = 2;
constexpr int elem_bytes_of(int dtype) { return dtype == kDtypeF32 ? 4 : 2; }

// Launch `fn` as a programmatic dependent of the work before it on `stream` (the
// kernel calls pdl_wait() before touching global memory): back-to-back calls then
// overlap one launch's start with the previous one's drain.
inline cudaError_t launch_dependent(const void *fn, dim3 grid, dim3 block, size_t smem, cudaStream_t stream,
                                    void **args) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = grid;
    cfg.blockDim = block;
    cfg.dynamicSmemBytes = smem;
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelExC(&cfg, fn, args);
}

// ---- register-carry path ---------------------------------------------------
// One thread walks `vec` adjacent channels through all L steps, with the loads
// of the next `prefetch` steps in flight in registers.
// h_init (B x D, may be NULL): state each sequence continues from (a_0 is then
// used); h_last (B x D, may be NULL): receives h[:, L-1, :].
bool regcarry_supported(int vec, int prefetch);
cudaError_t launch_regcarry(int vec, int prefetch, int threads, const float *a, const float *b,
                            float *h, int64_t B, int64_t L, int64_t D, const float *h_init, float *h_last,
                            cudaStream_t stream);
// The segmented form for few channels: the time axis cut into nseg segments, a reduce
// launch writing each segment's map to aggA / aggB ([segment][B * D] floats each) and an
// apply launch that folds the earlier segments' maps into each segment's carry.
cudaError_t launch_regcarry_segmented(int vec, int threads, const float *a, const float *b, float *h, int64_t B,
                                      int64_t L, int64_t D, int64_t nseg, const float *h_init, float *h_last,
                                      float *aggA, float *aggB, cudaStream_t stream);
// The same on 16-bit storage (dtype kDtypeBF16 or kDtypeF16): `vec` in {1, 2, 4, 8}
// elements per thread; h_init and h_last stay fp32.
bool regcarry16_supported(int vec, int prefetch);
cudaError_t launch_regcarry16(int dtype, int vec, int prefetch, int threads, const void *a, const void *b,
                              void *h, int64_t B, int64_t L, int64_t D, const float *h_init, float *h_last,
                              cudaStream_t stream);

// ---- chunked path ----------------------------------------------------------
// A tile is (tile_t time steps) x (tile_d channels) of one batch index, staged in
// shared memory by TMA.  `segments` threads share each channel's tile_t steps.
struct ChunkedVariant {
    int tile_d, tile_t, segments, stages;
    int threads;         // tile_d / cpt * segments
    size_t smem_bytes;   // dynamic shared memory per CTA
    int elem_bytes = 4;  // stored element size: 4 (fp32) or 2 (bfloat16 and binary16)
    int cpt = 1;         // adjacent channels per thread: 1, or 2 (16-bit storage)
    int blocks = 0;      // 1: compiled for blocks mode (and only used there)
    int chain = 0;       // 1: the chain-mode kernel (chain.cu), used only there
};
// The compiled variants (tile_d, tile_t, segments, stages combinations): fp32
// storage, and 16-bit storage (each shape compiled for bfloat16 and binary16).
const ChunkedVariant *chunked_variants(int *count);
const ChunkedVariant *chunked_variants_16(int *count);
// The kernel of a 16-bit variant for dtype kDtypeBF16 or kDtypeF16 (NULL if none).
const void *chunked16_kernel(const ChunkedVariant *v, int dtype);

// How the chunked forward kernel gets each tile's carry.
constexpr int kModeLookback = 0;   // tiles of a slice on different CTAs, decoupled look-back
constexpr int kModeOwn = 1;        // a CTA owns whole slices, carry in a register
constexpr int kModeReduce = 2;     // two-pass, first launch: write every tile's aggregate
constexpr int kModeApply = 3;      // two-pass, last launch: carry from the scanned aggregates
constexpr int kModeBlocks = 4;     // one launch: blocks of G tiles, reduce, look-back over blocks,
                                   // apply from L2 (variants with blocks = 1 only)
constexpr int kModeChain = 5;      // one cooperative launch: workers compose a tile ahead and publish its
                                   // map, resolver CTAs walk each slice's chain of maps (chain.cu)
// Speculative mode, two launches over a (B * G, L / G, D) view of the problem (G segments per
// sequence, `group` = G), compiled only into copies fixed to one of them (chunked_fixed.cu):
constexpr int kModeSpec = 6;       // each segment scanned from 0 (the first from the carried-in state),
                                   // its map (slope product, h) published: [slice][channel] pairs
constexpr int kModeRepair = 7;     // each later segment's start corrected with its true carry until
                                   // the slope product reaches exactly 0
constexpr int kSpecParts = 16;     // repair: earlier segments' maps a lane loads at once

struct ChunkedLaunch {
    const ChunkedVariant *variant;
    int dtype = kDtypeF32;       // storage of a, b and h
    CUtensorMap map_a, map_b;    // 3-D {D, L, B} maps of the stored type, box {tile_d, tile_t, 1}
    void *h;
    int64_t L, D;
    int64_t slices_per_batch;    // ceil(D / tile_d)
    int64_t n_slices;            // B * slices_per_batch
    int64_t chunks;              // ceil(L / tile_t)
    int64_t n_tiles;             // n_slices * chunks
    int64_t grid;
    int mode;                    // kModeLookback, kModeOwn, kModeReduce, kModeApply, kModeBlocks
    int group = 0;               // blocks mode: tiles per block
    Control *ctrl;
    unsigned long long *words;   // look-back mode: 3 * n_tiles * tile_d words; blocks mode: 3 * blocks *
                                 // tile_d words; two-pass modes: the per-tile A, B and scanned H arrays
                                 // (3 * n_tiles * tile_d floats)
    unsigned int *status;        // where device-side failures are recorded
    int64_t spin_limit;
    int64_t silent_tile;         // tile id that publishes nothing (tests), or -1
    const float *h_init = nullptr;   // (B x D) state to continue from, or NULL
    float *h_last = nullptr;         // (B x D) last state out, or NULL
};
// Number of CTAs of this variant that fit on one SM (occupancy API).
cudaError_t chunked_ctas_per_sm(const ChunkedVariant *v, int *ctas, int dtype = kDtypeF32);
// The copy of a variant's kernel compiled for carry mode `mode` alone (chunked_fixed.cu for fp32,
// chunked16_fixed.cu for 16-bit storage), which launch_chunked takes in place of the general
// kernel; NULL where there is none.
const void *fixed_kernel_f32(const ChunkedVariant *v, int mode);
const void *fixed_kernel_16(const ChunkedVariant *v, int dtype, int mode);
cudaError_t launch_chunked(const ChunkedLaunch &args, cudaStream_t stream);

// Chain mode (chain.cu): its compiled variants per storage type (the 16-bit ones serve
// bfloat16 and binary16 alike), the kernel of one, the layout of the resolver CTAs
// (returns their number; channels per group and groups per CTA out), and the launch
// (mode kModeChain; grid = resolver CTAs + workers, all resident at once).
const ChunkedVariant *chain_variants(int dtype, int *count);
const void *chain_kernel(const ChunkedVariant *v, int dtype);
int chain_layout(int64_t n_slices, int warps, int *cpg, int *gpc);
constexpr int kChainMaxResolvers = 16;   // resolver CTAs at most (slices beyond them: no chain mode)
cudaError_t launch_chain(const ChunkedLaunch &args, cudaStream_t stream);

// ---- backward (gradient) kernels -----------------------------------------------
// c_t = g_t + a_{t+1} c_{t+1} (c_{L-1} = g_{L-1} + dh_last), db = c,
// da_t = c_t h_{t-1} (h_{-1} = h_init or 0), dh_init = a_0 c_0.
struct BackwardLaunch {
    const ChunkedVariant *variant;
    CUtensorMap map_g, map_a, map_h;   // 3-D {D, L, B} maps of g, a and h (h unused without da)
    const float *a;                    // for a_0 in dh_init
    float *da = nullptr, *db = nullptr;
    int64_t L, D, slices_per_batch, n_slices, chunks, n_tiles, grid;
    int mode;                          // kModeOwn, kModeLookback, kModeReduce, kModeApply
    Control *ctrl;
    unsigned long long *words;
    unsigned int *status;
    int64_t spin_limit;
    int64_t silent_tile;
    const float *h_init = nullptr, *dh_last = nullptr;
    float *dh_init = nullptr;
};
const ChunkedVariant *backward_variants(int *count);
cudaError_t backward_ctas_per_sm(const ChunkedVariant *v, int *ctas);
cudaError_t launch_backward(const BackwardLaunch &args, cudaStream_t stream);
cudaError_t launch_regcarry_backward(int vec, int threads, const float *a, const float *h, const float *g, float *da,
                                     float *db, int64_t B, int64_t L, int64_t D, const float *h_init,
                                     const float *dh_last, float *dh_init, cudaStream_t stream);

// ---- (B, D, L) layout: one warp per row segment ------------------------------
constexpr int kRowsThreads = 256;
constexpr int kRowsFull = 0;     // whole rows, carry from h_init (or 0), write h
constexpr int kRowsReduce = 1;   // two-pass, first launch: each segment's composed map to aggA / aggB
constexpr int kRowsApply = 2;    // two-pass, last launch: rescan each segment from the h before it

struct RowsLaunch {
    int dtype = kDtypeF32;
    int vec = 4;                 // stored elements per lane per chunk (one vector load)
    int prefetch = 4;            // chunks whose loads are in flight ahead (2 or 4)
    const void *a = nullptr, *b = nullptr;
    void *h = nullptr;
    int64_t R = 0, L = 0;        // rows (B * D) and their length
    int64_t seg_len = 0, nseg = 1;   // segment length (a multiple of 32 * vec) and segments per row
    int64_t rows_per_unit = 1;       // one pass: consecutive whole rows per warp (1 when nseg > 1)
    int mode = kRowsFull;
    const float *h_init = nullptr;   // (R) state each row continues from, or NULL
    float *h_last = nullptr;         // (R) last state out, or NULL
    float *aggA = nullptr, *aggB = nullptr;   // two-pass: [segment][row] composed maps
    const float *aggH = nullptr;              // two-pass: [segment][row] last h of each segment
    float *aggX = nullptr;                    // two-pass with h_init: (R) copy of the state for the apply launch
};
bool rows_supported(int dtype, int vec, int prefetch);
cudaError_t launch_rows(const RowsLaunch &args, cudaStream_t stream);

// ---- index-checked build -------------------------------------------------------
// Per translation unit with kernels: read and clear the count of accesses skipped by
// the checks of checked.cuh and the byte offset of the first; set the output cap
// (tests).  In the normal build they report nothing.
cudaError_t checked_report_chunked(unsigned long long *count, long long *first, long long out_cap);
cudaError_t checked_report_chunked16(unsigned long long *count, long long *first, long long out_cap);
cudaError_t checked_report_backward(unsigned long long *count, long long *first, long long out_cap);
cudaError_t checked_report_regcarry(unsigned long long *count, long long *first, long long out_cap);
cudaError_t checked_report_regcarry16(unsigned long long *count, long long *first, long long out_cap);
cudaError_t checked_report_rows(unsigned long long *count, long long *first, long long out_cap);
cudaError_t checked_report_chain(unsigned long long *count, long long *first, long long out_cap);
cudaError_t checked_report_fixed(unsigned long long *count, long long *first, long long out_cap);
cudaError_t checked_report_fixed16(unsigned long long *count, long long *first, long long out_cap);

// ---- the fixed array of linrec_scan_f32_noalloc (noalloc.cu) ---------------------
// Its status word on device dev, read on `stream` and cleared (0 if unused); and, for
// tests, its epoch word.
cudaError_t noalloc_take_status(int dev, cudaStream_t stream, unsigned int *word);
cudaError_t noalloc_set_epoch(int dev, unsigned int epoch);

// ---- copy-ceiling kernel ---------------------------------------------------
cudaError_t launch_copy(const float *src, float *dst, int64_t n, int sm_count, cudaStream_t stream);

}  // namespace linrec
