// chunked16_fixed.cu -- copies of a 16-bit chunked tile (bfloat16 and binary16), each compiled
// for one carry mode (chunked_kernel.cuh, FM >= 0), which launch_chunked takes in place of the
// general kernel of the same tile when a call runs in that mode.  Without the other modes' code
// they need fewer registers and instructions (slice-owner 124, look-back 142, reduce 54, apply
// 126, against 159); resident CTAs per SM do not drop (shared memory holds them to three).
// Measured on GB300, us per call, general -> fixed-mode copy, {32, 256} with two channels per
// thread:
//   slice-owner: (32, 4096, 256) bfloat16 35.8 -> 32.5, binary16 34.3 -> 32.3; other shapes
//     within 1 %;
//   two-pass: (1, 1048576, 64) bfloat16 116.5 -> 109.9, (1, 131072, 64) 20.6 -> 18.1.
// The other 16-bit tiles keep the general kernel ({32, 256} with 16 segments measured slower in
// slice-owner mode: (64, 2048, 1024) bfloat16 122.9 -> 139.8).
#include "chunked_kernel.cuh"

namespace linrec {

// {tile_d, tile_t, segments, stages, channels per thread}
#define LINREC_FIXED_16(X) X(32, 256, 8, 2, 2)

const void *fixed_kernel_16(const ChunkedVariant *v, int dtype, int mode) {
    if (v->blocks || v->chain || v->elem_bytes != 2) return nullptr;
#define LINREC_FX(TD, TT, S, ST, CPT, M)                                                                     \
    if (mode == M)                                                                                           \
        return dtype == kDtypeBF16                                                                           \
                   ? reinterpret_cast<const void *>(&chunked_scan_kernel<kDtypeBF16, TD, TT, S, ST, CPT, false, M>) \
                   : reinterpret_cast<const void *>(&chunked_scan_kernel<kDtypeF16, TD, TT, S, ST, CPT, false, M>);
#define LINREC_FX_ALL(TD, TT, S, ST, CPT)                                                                    \
    if (v->tile_d == TD && v->tile_t == TT && v->segments == S && v->stages == ST && v->cpt == CPT &&        \
        (dtype == kDtypeBF16 || dtype == kDtypeF16)) {                                                       \
        LINREC_FX(TD, TT, S, ST, CPT, kModeOwn) LINREC_FX(TD, TT, S, ST, CPT, kModeLookback)                 \
        LINREC_FX(TD, TT, S, ST, CPT, kModeReduce) LINREC_FX(TD, TT, S, ST, CPT, kModeApply)                 \
    }
    LINREC_FIXED_16(LINREC_FX_ALL)
#undef LINREC_FX_ALL
#undef LINREC_FX
    return nullptr;
}

LINREC_CHECKED_REPORT(checked_report_fixed16)

}  // namespace linrec
