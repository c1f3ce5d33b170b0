// chunked.cu -- the chunked path on fp32 storage: its compiled tile variants,
// and the occupancy query and launch shared by every storage type.  The kernel
// itself is in chunked_kernel.cuh.
#include "chunked_kernel.cuh"

namespace linrec {

namespace {

#define LINREC_CHUNKED_VARIANTS(X) \
    X(128, 64, 4, 2)               \
    X(128, 64, 4, 3)               \
    X(128, 32, 2, 3)               \
    X(256, 32, 2, 2)               \
    X(64, 128, 8, 2)               \
    X(64, 64, 4, 2)                \
    X(64, 64, 4, 3)                \
    X(32, 128, 8, 2)               \
    X(32, 128, 8, 3)               \
    X(32, 64, 4, 3)                \
    X(32, 64, 4, 4)                \
    X(32, 32, 2, 6)
// compiled again for blocks mode
#define LINREC_CHUNKED_BLOCK_VARIANTS(X) \
    X(32, 128, 8, 2)                     \
    X(64, 128, 8, 2)

#define LINREC_V_ENTRY(TD, TT, S, ST) make_variant<kDtypeF32, TD, TT, S, ST, 1>(),
#define LINREC_VB_ENTRY(TD, TT, S, ST) make_variant<kDtypeF32, TD, TT, S, ST, 1, true>(),
const ChunkedVariant kVariants[] = {LINREC_CHUNKED_VARIANTS(LINREC_V_ENTRY)
                                        LINREC_CHUNKED_BLOCK_VARIANTS(LINREC_VB_ENTRY)};
#undef LINREC_V_ENTRY
#undef LINREC_VB_ENTRY

const void *kernel_of(const ChunkedVariant *v, int dtype) {
    if (v->chain) return chain_kernel(v, dtype);
    if (dtype != kDtypeF32) return chunked16_kernel(v, dtype);
    if (v->elem_bytes != 4) return nullptr;
#define LINREC_K_ENTRY(TD, TT, S, ST)                                                                \
    if (v->tile_d == TD && v->tile_t == TT && v->segments == S && v->stages == ST && v->cpt == 1 &&  \
        !v->blocks)                                                                                  \
        return reinterpret_cast<const void *>(&chunked_scan_kernel<kDtypeF32, TD, TT, S, ST, 1>);
    LINREC_CHUNKED_VARIANTS(LINREC_K_ENTRY)
#undef LINREC_K_ENTRY
#define LINREC_KB_ENTRY(TD, TT, S, ST)                                                               \
    if (v->tile_d == TD && v->tile_t == TT && v->segments == S && v->stages == ST && v->cpt == 1 &&  \
        v->blocks)                                                                                   \
        return reinterpret_cast<const void *>(&chunked_scan_kernel<kDtypeF32, TD, TT, S, ST, 1, true>);
    LINREC_CHUNKED_BLOCK_VARIANTS(LINREC_KB_ENTRY)
#undef LINREC_KB_ENTRY
    return nullptr;
}

}  // namespace

const ChunkedVariant *chunked_variants(int *count) {
    *count = (int)(sizeof(kVariants) / sizeof(kVariants[0]));
    return kVariants;
}

cudaError_t chunked_ctas_per_sm(const ChunkedVariant *v, int *ctas, int dtype) {
    const void *fn = kernel_of(v, dtype);
    if (!fn) return cudaErrorInvalidValue;
    cudaError_t err = cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)v->smem_bytes);
    if (err != cudaSuccess) return err;
    return cudaOccupancyMaxActiveBlocksPerMultiprocessor(ctas, fn, v->threads, v->smem_bytes);
}

cudaError_t launch_chunked(const ChunkedLaunch &p, cudaStream_t stream) {
    if (p.mode == kModeChain || p.variant->chain) return launch_chain(p, stream);
    const void *fn = p.dtype == kDtypeF32 ? fixed_kernel_f32(p.variant, p.mode)
                                          : fixed_kernel_16(p.variant, p.dtype, p.mode);
    // the speculative modes are compiled into their fixed copies only
    if (!fn && (p.mode == kModeSpec || p.mode == kModeRepair)) return cudaErrorInvalidValue;
    if (!fn) fn = kernel_of(p.variant, p.dtype);
    if (!fn) return cudaErrorInvalidValue;
    cudaError_t err = cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                           (int)p.variant->smem_bytes);
    if (err != cudaSuccess) return err;
    long long L = p.L, D = p.D, spb = p.slices_per_batch, ns = p.n_slices, ch = p.chunks, nt = p.n_tiles;
    long long spin = p.spin_limit, silent = p.silent_tile;
    int mode = p.mode, group = p.group;
    if ((mode == kModeBlocks) != (p.variant->blocks != 0) || (mode == kModeBlocks && group <= 0))
        return cudaErrorInvalidValue;
    void *h = p.h;
    Control *ctrl = p.ctrl;
    unsigned long long *words = p.words;
    unsigned int *status = p.status;
    const float *h_init = p.h_init;
    float *h_last = p.h_last;
    void *args[] = {(void *)&p.map_a, (void *)&p.map_b, &h, &L, &D, &spb, &ns, &ch, &nt, &mode,
                    &group, &ctrl, &words, &status, &spin, &silent, &h_init, &h_last};
    return launch_dependent(fn, dim3((unsigned)p.grid), dim3((unsigned)p.variant->threads), p.variant->smem_bytes,
                            stream, args);
}

LINREC_CHECKED_REPORT(checked_report_chunked)

}  // namespace linrec
