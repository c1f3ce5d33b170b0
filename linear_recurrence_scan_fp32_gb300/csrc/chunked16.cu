// chunked16.cu -- the chunked path on 16-bit storage (bfloat16 and IEEE
// binary16): the tile variants compiled for it.  A 16-bit box is half the bytes
// of an fp32 box of the same shape, so these variants keep more stages in
// flight to hold the same bytes per SM.  The kernel is in chunked_kernel.cuh.
#include "chunked_kernel.cuh"

namespace linrec {

namespace {

#define LINREC_CHUNKED16_VARIANTS(X) \
    X(32, 128, 8, 3, 1)              \
    X(32, 128, 8, 4, 1)              \
    X(32, 128, 8, 6, 1)              \
    X(64, 128, 8, 2, 1)              \
    X(64, 128, 8, 3, 1)              \
    X(64, 64, 4, 4, 1)               \
    X(32, 64, 4, 6, 1)               \
    X(128, 64, 4, 3, 1)              \
    X(32, 256, 8, 2, 1)              \
    X(32, 256, 8, 3, 1)              \
    X(32, 256, 16, 2, 2)             \
    X(32, 256, 8, 2, 2)              \
    X(32, 64, 8, 6, 2)
// compiled again for blocks mode
#define LINREC_CHUNKED16_BLOCK_VARIANTS(X) \
    X(32, 256, 8, 2, 2)

#define LINREC_V_ENTRY(TD, TT, S, ST, CPT) make_variant<kDtypeBF16, TD, TT, S, ST, CPT>(),
#define LINREC_VB_ENTRY(TD, TT, S, ST, CPT) make_variant<kDtypeBF16, TD, TT, S, ST, CPT, true>(),
const ChunkedVariant kVariants16[] = {LINREC_CHUNKED16_VARIANTS(LINREC_V_ENTRY)
                                          LINREC_CHUNKED16_BLOCK_VARIANTS(LINREC_VB_ENTRY)};
#undef LINREC_V_ENTRY
#undef LINREC_VB_ENTRY

// both 16-bit kinds share each variant's shared-memory layout
#define LINREC_SAME_SIZE(TD, TT, S, ST, CPT)                                                     \
    static_assert(sizeof(ChunkSmem<Storage<kDtypeBF16>::raw, TD, TT, S, ST>) ==                  \
                  sizeof(ChunkSmem<Storage<kDtypeF16>::raw, TD, TT, S, ST>), "16-bit layouts");
LINREC_CHUNKED16_VARIANTS(LINREC_SAME_SIZE)
#undef LINREC_SAME_SIZE

}  // namespace

const ChunkedVariant *chunked_variants_16(int *count) {
    *count = (int)(sizeof(kVariants16) / sizeof(kVariants16[0]));
    return kVariants16;
}

const void *chunked16_kernel(const ChunkedVariant *v, int dtype) {
    if (v->elem_bytes != 2) return nullptr;
#define LINREC_K_ENTRY(TD, TT, S, ST, CPT, BM)                                                          \
    if (v->tile_d == TD && v->tile_t == TT && v->segments == S && v->stages == ST && v->cpt == CPT &&     \
        (v->blocks != 0) == BM) {                                                                        \
        if (dtype == kDtypeBF16)                                                                         \
            return reinterpret_cast<const void *>(&chunked_scan_kernel<kDtypeBF16, TD, TT, S, ST, CPT, BM>); \
        if (dtype == kDtypeF16)                                                                          \
            return reinterpret_cast<const void *>(&chunked_scan_kernel<kDtypeF16, TD, TT, S, ST, CPT, BM>);  \
        return nullptr;                                                                                  \
    }
#define LINREC_K_PLAIN(TD, TT, S, ST, CPT) LINREC_K_ENTRY(TD, TT, S, ST, CPT, false)
#define LINREC_K_BLOCKS(TD, TT, S, ST, CPT) LINREC_K_ENTRY(TD, TT, S, ST, CPT, true)
    LINREC_CHUNKED16_VARIANTS(LINREC_K_PLAIN)
    LINREC_CHUNKED16_BLOCK_VARIANTS(LINREC_K_BLOCKS)
#undef LINREC_K_PLAIN
#undef LINREC_K_BLOCKS
#undef LINREC_K_ENTRY
    return nullptr;
}

LINREC_CHECKED_REPORT(checked_report_chunked16)

}  // namespace linrec
