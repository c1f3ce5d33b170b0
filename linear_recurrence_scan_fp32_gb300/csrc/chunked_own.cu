// chunked_own.cu -- slice-owner-only copies of two chunked tiles (chunked_kernel.cuh with
// OWN = true), launched instead of the general kernel of the same tile when a call runs in
// slice-owner mode.  With none of the look-back, two-pass and blocks code in them they need
// fewer registers (fp32 {32, 128}: 90 against 108; 16-bit {32, 256}, two channels per thread:
// 124 against 159) and fewer instructions, and resident CTAs per SM stay the same (the fp32
// tile is held to two by its registers and its launch bounds, the 16-bit one to three by
// shared memory).  Measured on GB300, us per call, general -> slice-owner-only:
//   (32, 4096, 256) bfloat16 35.8 -> 32.5, binary16 34.3 -> 32.3;
//   (16, 4096, 256) fp32 44.3 -> 36.3, (1, 32768, 4096) fp32 334 -> 276;
//   other shapes on these tiles within 1 % ((56, 4096, 256) fp32 106.8 -> 107.7).
// The other tiles keep their general kernel: there the copy measured slower ((64, 2048, 1024)
// fp32 on {256, 32} 232 -> 252; the {32, 64} tiles of 1.2 to 1.33 rounds 87 -> 96, their
// lower register count letting a third CTA onto some SMs).
#include "chunked_kernel.cuh"

namespace linrec {

namespace {

#define LINREC_OWN_F32_VARIANTS(X) X(32, 128, 8, 2)
#define LINREC_OWN_16_VARIANTS(X) X(32, 256, 8, 2, 2)

}  // namespace

const void *own_kernel(const ChunkedVariant *v, int dtype) {
    if (v->blocks || v->chain) return nullptr;
#define LINREC_OWN_F32(TD, TT, S, ST)                                                                    \
    if (dtype == kDtypeF32 && v->elem_bytes == 4 && v->cpt == 1 && v->tile_d == TD && v->tile_t == TT && \
        v->segments == S && v->stages == ST)                                                             \
        return reinterpret_cast<const void *>(&chunked_scan_kernel<kDtypeF32, TD, TT, S, ST, 1, false, true>);
    LINREC_OWN_F32_VARIANTS(LINREC_OWN_F32)
#undef LINREC_OWN_F32
#define LINREC_OWN_16(TD, TT, S, ST, CPT)                                                                \
    if (v->elem_bytes == 2 && v->cpt == CPT && v->tile_d == TD && v->tile_t == TT && v->segments == S &&   \
        v->stages == ST) {                                                                               \
        if (dtype == kDtypeBF16)                                                                         \
            return reinterpret_cast<const void *>(&chunked_scan_kernel<kDtypeBF16, TD, TT, S, ST, CPT, false, true>); \
        if (dtype == kDtypeF16)                                                                          \
            return reinterpret_cast<const void *>(&chunked_scan_kernel<kDtypeF16, TD, TT, S, ST, CPT, false, true>);  \
    }
    LINREC_OWN_16_VARIANTS(LINREC_OWN_16)
#undef LINREC_OWN_16
    return nullptr;
}

LINREC_CHECKED_REPORT(checked_report_own)

}  // namespace linrec
