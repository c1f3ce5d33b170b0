/*
 * linrec.h -- C ABI of liblinrec, a GB300 (sm_103a) first-order linear-recurrence scan.
 *
 * The operation (POPCORNBENCH trace "Kimi-K2.6 l1_p9", problem statement; the
 * same statement opens "FW-GLM-5-1 l1_p9"): for fp32 tensors a, b, h of shape
 * (B, L, D), row-major with D contiguous (element (i,t,d) at i*L*D + t*D + d),
 * every channel (i, d) is an independent sequence
 *
 *     h[i,0,d] = b[i,0,d]
 *     h[i,t,d] = a[i,t,d] * h[i,t-1,d] + b[i,t,d]        0 < t < L.
 *
 * a[i,0,d] is never used.  The kernels evaluate it as a scan of the affine maps
 * x -> a_t*x + b_t under composition, later map on the left:
 * (a2,b2) o (a1,b1) = (a2*a1, a2*b1 + b2) ("Kimi-K2.6 l1_p9", derivation of the
 * associative operator), with only the running value h carried from one time
 * chunk to the next (same page, the running_h carry).
 *
 * Conventions for every entry point below:
 *  - Pointers a, b, h are device memory of the CURRENT CUDA device, owned by
 *    the caller; the library never frees or retains them.  a and b are read,
 *    h is written (B*L*D floats).  h must not overlap a or b (no in-place).
 *    a and b may be the same buffer.
 *  - Any alignment is accepted.  16-byte aligned a, b, h and D % 4 == 0 let
 *    the fastest kernels run; other inputs take a scalar-load variant.
 *  - stream is a cudaStream_t passed as void* (NULL = the legacy default
 *    stream).  Work is enqueued asynchronously on it: the returned status
 *    covers argument checks and the launch; a kernel's own failure surfaces at
 *    the caller's next synchronisation, or through linrec_stream_status().
 *  - B*L*D == 0 returns LINREC_OK with no launch (pointers may then be NULL).
 *  - Results are deterministic: a given build, device, shape and path returns
 *    the same bits on every call.
 *  - Thread-safe: calls from several host threads may run concurrently.  Calls
 *    on one stream run in order; each stream gets its own look-back workspace,
 *    so calls on different streams may overlap on the GPU.
 *  - The kernels are launched as programmatic dependents: a call's kernel may
 *    be scheduled while the previous work on the stream drains, but it touches
 *    no memory before that work has completed, so stream order holds as for a
 *    plain launch.
 *  - CUDA graphs: every device-pointer entry point (not linrec_scan_f32_host,
 *    not linrec_stream_status, which synchronises) may be called on a stream
 *    that is being captured.  The library allocates nothing during capture:
 *    the call uses the workspace the library already holds for that stream,
 *    so first make the same call (or one of the same shape and mode) once on
 *    that stream outside capture; otherwise the call returns
 *    LINREC_ERR_WORKSPACE and enqueues nothing.  A captured workspace is never
 *    freed (later, larger calls on the stream get a new one).  Replays of the
 *    graph use the capturing stream's workspace wherever they are launched, so
 *    a replay must not overlap other work that uses it: an uncaptured call on
 *    the capturing stream, or a replay of another graph captured on it.
 */
#ifndef LINREC_H_
#define LINREC_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
    LINREC_OK = 0,
    LINREC_ERR_INVALID_VALUE = 1,      /* negative size, NULL with a non-zero size, size overflow */
    LINREC_ERR_ALIAS = 2,              /* h overlaps a or b */
    LINREC_ERR_UNSUPPORTED_DEVICE = 3, /* the current device is not compute capability 10.3 */
    LINREC_ERR_LAUNCH = 4,             /* a CUDA call failed while enqueueing the work */
    LINREC_ERR_WORKSPACE = 5,          /* the look-back workspace could not be allocated (or the
                                          stream is capturing and holds too little: see below) */
    LINREC_ERR_LOOKBACK_TIMEOUT = 6,   /* a kernel gave up waiting on a predecessor tile */
    LINREC_ERR_TMA_TIMEOUT = 7         /* a kernel gave up waiting on a bulk copy */
} linrec_status_t;

typedef enum {
    LINREC_PATH_AUTO = 0,      /* the dispatcher chooses */
    LINREC_PATH_REGCARRY = 1,  /* one thread per 1/2/4 adjacent channels, loads prefetched in registers */
    LINREC_PATH_CHUNKED = 2,   /* TMA-staged (time x channel) tiles, shuffle scan, decoupled look-back */
    LINREC_PATH_ROWS = 3       /* (B, D, L) layout: a warp per row segment, shuffle scan along the row */
} linrec_path_t;

/*
 * linrec_scan_f32 -- h = scan(a, b) as defined above.  See the conventions.
 * Returns LINREC_OK, or an error code without launching anything.
 */
linrec_status_t linrec_scan_f32(const float *a, const float *b, float *h,
                                int64_t B, int64_t L, int64_t D, void *stream);

/*
 * Options for linrec_scan_f32_ex and linrec_plan_f32.  Zero-initialise, then
 * set what you need; a zero field means "the dispatcher's choice".
 */
typedef struct {
    int path;            /* linrec_path_t */
    int vec;             /* regcarry: channels per thread, 1, 2 or 4 (16-bit storage: 1, 2, 4 or 8);
                            chunked: adjacent channels per thread, 1, or 2 for 16-bit storage (one
                            32-bit shared-memory load and one packed store per step for both) */
    int prefetch;        /* regcarry: time steps loaded ahead, 4, 8 or 16 */
    int tile_t;          /* chunked: time steps per tile */
    int tile_d;          /* chunked: channels per tile */
    int stages;          /* chunked: tiles in flight per CTA (shared-memory ring depth) */
    int ctas_per_sm;     /* chunked: cap on resident CTAs per SM (0 = as many as fit) */
    int chunk_mode;      /* chunked: 1 = each CTA owns whole channel slices and carries h from
                            chunk to chunk itself; 2 = chunks of a slice spread over CTAs, joined
                            by the decoupled look-back; 3 = two passes: a launch writes every
                            chunk's aggregate, the aggregates are scanned, a launch applies them
                            (the gradient runs them in reversed chunk order); 4 = blocks (forward
                            only): one launch; a CTA composes a block of `group` consecutive
                            chunks of a slice, joins the blocks of the slice by the decoupled
                            look-back, then re-reads the block (from L2) and writes h; 5 = chain
                            (forward only): one launch that reads and writes every element once;
                            worker CTAs compose each chunk as it lands and publish its aggregate
                            before they finish the chunk before it, while resolver CTAs fold each
                            slice's aggregates in chunk order into the running h entering every
                            chunk (the same values, bit for bit, as mode 1); it takes at most 128
                            slices of 32 channels (B * ceil(D/32); 64 in 16-bit storage), more
                            return LINREC_ERR_INVALID_VALUE; 6 = speculative (fp32 forward only):
                            two launches; each sequence is cut into G equal segments (G divides
                            L, L/G >= 1024; `group`, else the dispatcher's), every segment is
                            scanned from 0 (the first from the carried-in state) and publishes
                            its map, and a chunk is stored once the product of the slopes from
                            the segment's start to it is exactly 0 in fp32 in all 32 channels of
                            its slice (the true carry then no longer reaches h); the second
                            launch takes each later segment's true carry from the maps before it
                            and writes the chunks left unstored.  12 bytes moved per element
                            plus 8 for each element before that point: 20, as for mode 3, where
                            the slopes never decay; 0 = the dispatcher's choice */
    unsigned int *d_status; /* device word (may be NULL): the kernel ORs 1 << linrec_status_t
                               into it on a device-side failure; otherwise the stream's own word
                               is used (read it with linrec_stream_status) */
    const float *h_init; /* (B, D) state each sequence continues from, or NULL (see linrec_scan_f32_carry) */
    float *h_last;       /* (B, D) receives h[:, L-1, :], or NULL */
    int64_t spin_limit;  /* chunked: polls of a predecessor before giving up (0 = default, ~1 s) */
    int64_t test_silent_tile; /* chunked, tests only: 0 = off; k > 0 makes tile id k-1
                                 publish nothing, so its successor's look-back times out */
    int rows_per_warp;   /* (B, D, L) layout, one pass: consecutive rows each warp scans as one
                            stream (0 = the dispatcher's choice) */
    int segments;        /* chunked: segments a tile's time steps are split into, one thread
                            each per channel group (0 = the dispatcher's choice for its default
                            16-bit tile, else the first compiled variant of the tile) */
    int group;           /* chunk_mode 4: chunks per block (0 = 1024 time steps' worth);
                            chunk_mode 6: segments per sequence (0 = the dispatcher's choice);
                            any other chunk_mode takes 0 only */
} linrec_options_t;

/*
 * linrec_scan_f32_carry -- the scan continued from a state, for scanning a long
 * sequence in segments or streaming it.  The running value h is the only
 * thing that crosses a chunk boundary ("Kimi-K2.6 l1_p9", the running_h
 * carry); this entry point takes it in and hands it out:
 *
 *     h[i,t,d] = a[i,t,d] * h[i,t-1,d] + b[i,t,d]   for every t >= 0,
 *     h[i,-1,d] = h_init[i*D + d]                    (so a[i,0,d] is used)
 *     h_last[i*D + d] = h[i,L-1,d].
 *
 * h_init == NULL gives linrec_scan_f32's definition (h_0 = b_0, a_0 unused);
 * h_last == NULL skips the last state.  h_init and h_last are (B, D) fp32
 * device arrays, row-major, any 4-byte alignment.  h_last may be the same
 * buffer as h_init (the state is updated in place: every channel reads its
 * h_init before any h_last is written); any other overlap between h_init,
 * h_last, a, b and h returns LINREC_ERR_ALIAS.  Scanning [0, L1) and then
 * [L1, L) continued from the first call's h_last gives the same values as
 * one call over [0, L) up to rounding (the tiles differ).
 */
linrec_status_t linrec_scan_f32_carry(const float *a, const float *b, float *h,
                                      int64_t B, int64_t L, int64_t D,
                                      const float *h_init, float *h_last, void *stream);

/*
 * linrec_scan_f32_backward -- the gradient of linrec_scan_f32_carry, for
 * training.  The pages do not write it down; it follows from the definition
 * above ("Kimi-K2.6 l1_p9", problem statement) by the chain rule.  With
 * g = dL/dh (B, L, D) and c_t = dL/dh_t in total:
 *
 *     c_{L-1} = g_{L-1} + dh_last,    c_t = g_t + a_{t+1} * c_{t+1},
 *     db_t = c_t,    da_t = c_t * h_{t-1},    dh_init = a_0 * c_0,
 *
 * with h_{-1} = h_init (or 0 when h_init is NULL: a_0 was unused, da_0 = 0).
 * It is the same recurrence run right to left with the slope one step later,
 * on the same machinery: slice-owner, look-back or (few long slices) two-pass
 * mode, the last moving 28 bytes per element with da instead of 20 but
 * waiting on no chain.  Pointers are device memory of the current device:
 *   a, g        (B, L, D) in;  h (B, L, D) in: the forward output (needed
 *               only for da; may be NULL when da is NULL);
 *   da          (B, L, D) out or NULL (then h is not read: 12 bytes moved
 *               per element instead of 20);  db (B, L, D) out;
 *   h_init      (B, D) in or NULL: the forward's starting state;
 *   dh_last     (B, D) in or NULL: gradient arriving at h[:, L-1, :] from
 *               outside the scan (e.g. from a later segment's dh_init);
 *   dh_init     (B, D) out or NULL: gradient of the starting state, to pass
 *               to the earlier segment's dh_last when a long sequence was
 *               scanned in segments.
 * db may be the same buffer as g (updated in place); no other output may
 * overlap an input or another output (LINREC_ERR_ALIAS).  Other conventions
 * as for linrec_scan_f32.
 */
linrec_status_t linrec_scan_f32_backward(const float *a, const float *h, const float *g,
                                         float *da, float *db, int64_t B, int64_t L, int64_t D,
                                         const float *h_init, const float *dh_last, float *dh_init,
                                         void *stream);

/* linrec_scan_f32_backward with explicit options (path, chunk mode, tile, status word). */
linrec_status_t linrec_scan_f32_backward_ex(const float *a, const float *h, const float *g,
                                            float *da, float *db, int64_t B, int64_t L, int64_t D,
                                            const float *h_init, const float *dh_last, float *dh_init,
                                            void *stream, const linrec_options_t *opt);

/*
 * linrec_scan_f32_host -- the scan on HOST buffers a, b (read) and h (written),
 * row-major (B, L, D) like the device entry points.
 *  - When a, b and h are all page-locked host memory the device can address
 *    (cudaHostAlloc, cudaHostRegister), every byte of each, the kernels read
 *    and write them in place over the host link: no copies, no device memory.
 *    A buffer only partly page-locked (say a registered prefix of a larger
 *    block) is moved by the copy pipeline below instead.
 *  - Otherwise the library moves the data itself: the problem is cut into
 *    pieces of about 48 MB (whole sequences of a few batch indices, or, for
 *    long sequences, runs of time steps chained through the carry of
 *    linrec_scan_f32_carry), and the copy to the device, the scan and the
 *    copy back of successive pieces overlap on three internal streams
 *    through a ring of three device slots, allocated on first use and kept
 *    per device.
 * Either way the work starts after what is already queued on `stream` and
 * `stream` waits for its end: synchronise `stream` before reading h, and keep
 * a, b, h alive until then.  h must not overlap a or b (LINREC_ERR_ALIAS).
 * Pipelined calls are serialised per device by the library.
 */
linrec_status_t linrec_scan_f32_host(const float *a, const float *b, float *h,
                                     int64_t B, int64_t L, int64_t D, void *stream);

/* linrec_scan_f32 with explicit options (forced path, tile shape, status word, carry).  One
   options struct stands where a minimal form would take (int path, unsigned int *d_status):
   it carries both, plus the chunk mode, tile, carried state and test hooks, and NULL means
   every default. */
linrec_status_t linrec_scan_f32_ex(const float *a, const float *b, float *h,
                                   int64_t B, int64_t L, int64_t D, void *stream,
                                   const linrec_options_t *opt);

/* What a call would launch: filled by linrec_plan_f32 without touching a GPU. */
typedef struct {
    int path;              /* LINREC_PATH_REGCARRY or LINREC_PATH_CHUNKED */
    int vec, prefetch;     /* regcarry parameters */
    int tile_t, tile_d, segments, stages; /* chunked parameters */
    int lookback;          /* chunked: 1 = look-back mode */
    int twopass;           /* chunked: 1 = two-pass mode (reduce, scan of aggregates, apply);
                              lookback = twopass = 0: slice-owner mode */
    int threads;           /* threads per CTA */
    int64_t grid;          /* CTAs launched */
    int64_t n_tiles;       /* chunked: tiles of tile_t x tile_d */
    int64_t chunks;        /* chunked: time chunks per channel slice */
    size_t smem_bytes;     /* dynamic shared memory per CTA */
    size_t workspace_bytes;/* chunked: control block + look-back words for this call */
    int blocks;            /* chunked: blocks mode, chunks per block (0 = another mode) */
    int chain;             /* chunked: 1 = chain mode (one cooperative launch: worker CTAs publish
                              each chunk's aggregate a chunk ahead, resolver CTAs walk each slice's
                              chain of aggregates; grid = resolvers + workers) */
    int speculative;       /* chunked: speculative mode, segments per sequence (0 = another mode);
                              chunks and n_tiles count the segments as sequences of L/segments */
} linrec_plan_t;

/*
 * linrec_plan_f32 -- run the dispatcher for a device with sm_count SMs.
 * align_bytes: the largest of 16, 8, 4 that divides the addresses of a, b
 * and h (4 for plain fp32 pointers).  ctas_per_sm: resident CTAs per SM that
 * the chunked kernel gets on the device (0 = estimate from shared memory).
 * Pure host logic; no CUDA call.  Returns LINREC_ERR_INVALID_VALUE for bad
 * sizes or for options that name a path or variant these inputs cannot take.
 */
linrec_status_t linrec_plan_f32(int64_t B, int64_t L, int64_t D, int sm_count, int align_bytes,
                                int ctas_per_sm, const linrec_options_t *opt, linrec_plan_t *plan);

/* The same for linrec_scan_f32_backward (its own tile table). */
linrec_status_t linrec_plan_f32_backward(int64_t B, int64_t L, int64_t D, int sm_count, int align_bytes,
                                         int ctas_per_sm, const linrec_options_t *opt, linrec_plan_t *plan);

/*
 * 16-bit storage.  linrec_scan_bf16 and linrec_scan_f16 run the same scan with
 * a, b and h stored as bfloat16 words (sign 1, exponent 8, fraction 7 bits) or
 * IEEE 754 binary16 words (sign 1, exponent 5, fraction 10 bits), passed as
 * uint16_t arrays of B*L*D elements in the same (B, L, D) layout.  The pages
 * store everything in fp32; the scan is bound by the bytes it moves, and
 * 16-bit storage moves half of them.
 *  - Every element is widened exactly to fp32; all arithmetic and every
 *    carried value are fp32, on the same kernels and in the same order as
 *    linrec_scan_f32; each h is that fp32 result rounded once to the nearest
 *    16-bit value, ties to even (binary16 overflows to infinity from 65520 on).
 *    So |h - exact| <= u*|exact| + (1 + u)*e32, with u = 2^-8 (bfloat16) or
 *    2^-11 (binary16) and e32 the error of the fp32 scan.
 *  - Options as for linrec_scan_f32_ex.  h_init and h_last, when given, are
 *    fp32 (B, D) arrays: the state carried between calls keeps full precision.
 *  - 16-byte aligned a, b, h with D % 8 == 0 take the chunked kernel; other
 *    inputs (any 2-byte alignment) take the register path.
 * Other conventions as for linrec_scan_f32.
 */
linrec_status_t linrec_scan_bf16(const uint16_t *a, const uint16_t *b, uint16_t *h,
                                 int64_t B, int64_t L, int64_t D, void *stream);
linrec_status_t linrec_scan_f16(const uint16_t *a, const uint16_t *b, uint16_t *h,
                                int64_t B, int64_t L, int64_t D, void *stream);
linrec_status_t linrec_scan_bf16_ex(const uint16_t *a, const uint16_t *b, uint16_t *h,
                                    int64_t B, int64_t L, int64_t D, void *stream,
                                    const linrec_options_t *opt);
linrec_status_t linrec_scan_f16_ex(const uint16_t *a, const uint16_t *b, uint16_t *h,
                                   int64_t B, int64_t L, int64_t D, void *stream,
                                   const linrec_options_t *opt);

/* The dispatcher's decision for 16-bit storage (bfloat16 and binary16 alike);
   align_bytes may also be 2.  Otherwise as linrec_plan_f32. */
linrec_status_t linrec_plan_16(int64_t B, int64_t L, int64_t D, int sm_count, int align_bytes,
                               int ctas_per_sm, const linrec_options_t *opt, linrec_plan_t *plan);

/*
 * (B, D, L) layout.  linrec_scan_f32_bdl runs the same recurrence on tensors
 * whose TIME axis is innermost: element (i, d, t) at i*D*L + d*L + t, so every
 * channel (i, d) is one contiguous row of L values (row i*D + d):
 *
 *     h[i,d,0] = b[i,d,0],    h[i,d,t] = a[i,d,t] * h[i,d,t-1] + b[i,d,t].
 *
 * "Kimi-K2.6 l1_p9" weighs this layout (its transpose discussion) as the one
 * in which a warp reads a channel's steps contiguously; callers that hold their
 * data this way need no transpose.  Note the argument order B, D, L.
 *  - Many rows: one pass, a warp per row, L read in 32*V-step chunks with a
 *    shuffle scan and the carry in a register.  Few long rows: two passes over
 *    row segments (each segment's map, the scan of those maps by the (B, L, D)
 *    kernels, each segment rescanned from its carry): 20 bytes per fp32
 *    element instead of 12.
 *  - Vector width V (stored elements per lane per chunk): by default the widest
 *    that divides L and that the pointers' alignment allows, up to 16 bytes for
 *    fp32 and 32 bytes (two 16-byte accesses) for 16-bit storage; any alignment
 *    of the element type works.
 *  - The _ex forms take the options: h_init / h_last ((B, D) fp32, row i*D + d,
 *    as for linrec_scan_f32_carry), d_status, vec (1, 2, 4, 8 for fp32; 1, 2,
 *    4, 8, 16 for 16-bit storage; at most 32 bytes, needing min(16, bytes)-byte
 *    alignment), prefetch (2 or 4 chunks), chunk_mode (0 auto, 1 one pass,
 *    3 two passes); path must be 0 or LINREC_PATH_ROWS.
 * Other conventions as for linrec_scan_f32 (and, for the 16-bit forms, as for
 * linrec_scan_bf16 / linrec_scan_f16).
 */
linrec_status_t linrec_scan_f32_bdl(const float *a, const float *b, float *h,
                                    int64_t B, int64_t D, int64_t L, void *stream);
linrec_status_t linrec_scan_f32_bdl_ex(const float *a, const float *b, float *h,
                                       int64_t B, int64_t D, int64_t L, void *stream,
                                       const linrec_options_t *opt);
linrec_status_t linrec_scan_bf16_bdl_ex(const uint16_t *a, const uint16_t *b, uint16_t *h,
                                        int64_t B, int64_t D, int64_t L, void *stream,
                                        const linrec_options_t *opt);
linrec_status_t linrec_scan_f16_bdl_ex(const uint16_t *a, const uint16_t *b, uint16_t *h,
                                       int64_t B, int64_t D, int64_t L, void *stream,
                                       const linrec_options_t *opt);

/* The dispatcher's decision for the (B, D, L) layout with elem_bytes-byte storage
   (4: fp32, 2: bfloat16 or binary16).  path = LINREC_PATH_ROWS; vec, prefetch;
   one pass: tile_d = consecutive rows per warp; two passes: tile_t = the
   segment length, chunks = segments per row; n_tiles = warps (units of work);
   twopass; workspace_bytes = the two-pass arrays. */
linrec_status_t linrec_plan_bdl(int64_t B, int64_t D, int64_t L, int elem_bytes, int sm_count,
                                int align_bytes, const linrec_options_t *opt, linrec_plan_t *plan);

/*
 * linrec_stream_status -- synchronise `stream`, then return and clear the
 * device-side status of the library's work on it: LINREC_OK, or the first of
 * LINREC_ERR_LOOKBACK_TIMEOUT / LINREC_ERR_TMA_TIMEOUT that a kernel recorded.
 * It also reports and clears the failures of linrec_scan_f32_noalloc calls on
 * the current device that were made with d_status == NULL (their fixed array
 * keeps one status word for all streams).  A stream the library has not used
 * reports LINREC_OK.
 */
linrec_status_t linrec_stream_status(void *stream);

/*
 * linrec_copy_f32 -- dst[i] = src[i], i < n, on the current device.  A plain
 * 16-byte vector copy kernel used as the in-run copy-bandwidth ceiling next to
 * the scan (no part of the scan itself).  Same pointer rules as the scan.
 */
linrec_status_t linrec_copy_f32(const float *src, float *dst, int64_t n, void *stream);

/*
 * linrec_scan_f32_noalloc -- the chunked look-back scan for callers that must
 * not allocate device memory.  The pages this library follows have no
 * counterpart to it.  Callers it is for: code that enqueues work while a CUDA
 * graph is being captured or from a real-time loop, where an allocation can
 * stall on a device-wide synchronisation; plug-ins whose host application owns
 * all device memory through its own allocator and forbids other allocations;
 * services that must keep a fixed, known memory footprint.
 *
 * Same operation, pointer and size rules as linrec_scan_f32, and also:
 *  - a, b and h must be 16-byte aligned and D % 4 == 0 (the chunked kernel's
 *    tensor copies need it); otherwise LINREC_ERR_INVALID_VALUE.
 *  - The scratch is one fixed array of LINREC_NOALLOC_SCRATCH_BYTES (16 MiB)
 *    compiled into the library; every GPU that loads the library holds it
 *    until the process exits.  Shapes with at least as many 32-channel
 *    slices (B * ceil(D/32)) as the GPU has SMs need only its 256-byte
 *    control block.  Fewer, longer slices use the look-back words, about
 *    24 * B * D * L / 128 bytes: (1, 1048576, 64) fits, (1, 2^24, 64) does
 *    not.  A problem that needs more returns LINREC_ERR_WORKSPACE without
 *    launching anything.
 *  - It calls no allocation routine: no cudaMalloc, cudaMallocAsync or
 *    cudaFree, and nothing that calls them.
 *  - The first call on each device looks up the array's device address and
 *    the kernel's occupancy (once per device); make that first call before
 *    any stream capture.
 *  - Every call uses the same array, which keeps what the last call left.
 *    The array's tile counters are zero when the library loads and the last
 *    block of every launch resets them (a launch whose waits ran out
 *    included), so a call enqueues nothing but its kernel; each call tags its
 *    look-back words with a per-call epoch that the launch advances, so words
 *    left by earlier calls are never mistaken for its own.  Calls that
 *    overlap on the GPU (on different streams, or graph launches in flight
 *    together) race on the array and return wrong results: run them one
 *    after another.
 *  - d_status (may be NULL): a device word the kernel ORs
 *    1 << LINREC_ERR_LOOKBACK_TIMEOUT or 1 << LINREC_ERR_TMA_TIMEOUT into if
 *    a bounded wait runs out; the output then holds NaN where the carry was
 *    lost.  With d_status == NULL the failure goes to a status word in the
 *    array instead, which linrec_stream_status reports and clears (on any
 *    stream of the device; synchronise the streams those calls ran on first).
 */
#define LINREC_NOALLOC_SCRATCH_BYTES (16u * 1024u * 1024u)
linrec_status_t linrec_scan_f32_noalloc(const float *a, const float *b, float *h,
                                        int64_t B, int64_t L, int64_t D, void *stream,
                                        unsigned int *d_status);

/* Human-readable name of a status code (static storage). */
const char *linrec_status_string(linrec_status_t status);

/*
 * linrec_workspace_bytes -- device memory that a linrec_scan_f32 call on
 * (B, L, D) with 16-byte-aligned pointers holds on the current device: the
 * control block and look-back words, plus, in two-pass mode, the tile maps
 * and the workspace of their scan.  The library allocates it on the call's
 * stream at the first call that needs it, rounding each allocation up to a
 * MiB, and keeps it for later calls on that stream (see CUDA graphs above).
 * Returns 0 for the register path, an empty or invalid shape, or when no CUDA
 * device is usable.
 */
size_t linrec_workspace_bytes(int64_t B, int64_t L, int64_t D);

/*
 * The index-checked build (compiled with -DLINREC_DEBUG, e.g. by the package's
 * _build.build(checked=True) into liblinrec_checked.so).  Every plain global
 * load and store of the scan kernels first tests that it lies inside its array;
 * one outside is skipped (a load yields zeros) and counted.  TMA copies are
 * clipped to the tensor by the hardware and need no test.  It serves as the
 * memory checker of this library where no external one can run.
 *
 * linrec_debug_checks: 1 in the index-checked build, 0 otherwise.
 * linrec_debug_bad_accesses: synchronises the current device, then returns
 *   and clears the number of accesses skipped since the last call and the byte
 *   offset of the first one from the start of its array (-1 if none); and sets
 *   output_cap_bytes: > 0 makes every output array (h, da, db, the states
 *   handed out) end at that many bytes, so that a test can watch the checks skip
 *   stores without any real out-of-bounds access; 0 removes the cap.  The
 *   normal build reports 0 and -1 and ignores the cap.
 */
int linrec_debug_checks(void);
linrec_status_t linrec_debug_bad_accesses(uint64_t *count, int64_t *first_offset, int64_t output_cap_bytes);

/*
 * linrec_debug_range_covers -- 1 if the bytes [p, p + bytes) lie inside the address
 * range [range_start, range_start + range_size), else 0 (also for bytes == 0).  Pure
 * host logic, exported so that tests can check it: linrec_scan_f32_host reads and
 * writes host buffers in place only when the driver's range of each buffer's first
 * byte covers the whole buffer (and its last byte is mapped at the matching device
 * address); any buffer only partly page-locked goes through the copy pipeline.
 */
int linrec_debug_range_covers(uintptr_t range_start, size_t range_size, uintptr_t p, size_t bytes);

/*
 * linrec_debug_set_epoch -- tests only: write `epoch` into the epoch word of the
 * look-back workspace the library holds for `stream` on the current device
 * (fixed_array == 0; LINREC_ERR_WORKSPACE if it holds none yet), or of the fixed
 * array of linrec_scan_f32_noalloc (fixed_array != 0).  Synchronous.  A launch
 * tags its words with a tag derived from the epoch and moves the epoch on; this
 * lets a test start just below the point where the epoch word wraps around.
 */
linrec_status_t linrec_debug_set_epoch(void *stream, int fixed_array, uint32_t epoch);

/* Library version as major*10000 + minor*100 + patch. */
int linrec_version(void);

#ifdef __cplusplus
}
#endif

#endif /* LINREC_H_ */
