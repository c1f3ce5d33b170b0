// chunked_fixed.cu -- copies of fp32 chunked tiles, each compiled for one carry mode
// (chunked_kernel.cuh, FM >= 0), which launch_chunked takes in place of the general kernel of
// the same tile when a call runs in that mode.  Without the other modes' code they need fewer
// registers and instructions ({32, 128}: slice-owner 90, look-back 96, reduce 56, apply 92,
// against 108); resident CTAs per SM do not drop (launch bounds, shared memory or the registers
// of the general kernel still set them).  Measured on GB300, us per call, general -> copy:
//   slice-owner, {32, 128}: (16, 4096, 256) 44.3 -> 36.3, (1, 32768, 4096) 334 -> 276; other
//     shapes within 1 % ((56, 4096, 256) 106.8 -> 107.7);
//   two-pass (reduce and apply {32, 128}, the scan of the tile maps in look-back {64, 128} or
//     {32, 128}): (1, 1048576, 64) 211.1 -> 204.3, (1, 131072, 64) 32.7 -> 27.0;
//   look-back: (1, 4096, 64) 9.9 -> 9.2, (2, 4096, 256) 12.1 -> 11.4, (8, 2048, 256) 16.3 -> 15.5.
// The other tiles keep the general kernel: on them the slice-owner copy measured slower
// ((64, 2048, 1024) on {256, 32} 232 -> 252; the {32, 64} tiles of 1.2 to 1.33 rounds 87 -> 96,
// their lower register count letting a third CTA onto some SMs).
#include "chunked_kernel.cuh"

namespace linrec {

// {tile_d, tile_t, segments, stages}: the fp32 tiles with copies in slice-owner, look-back,
// reduce and apply modes (the second list: look-back, reduce and apply only; the third: the two
// speculative modes, which exist in these copies alone)
#define LINREC_FIXED_F32_ALL(X) X(32, 128, 8, 2)
#define LINREC_FIXED_F32_CHAINED(X) X(32, 128, 8, 3) X(64, 128, 8, 2)
#define LINREC_FIXED_F32_SPEC(X) X(32, 128, 8, 2)

const void *fixed_kernel_f32(const ChunkedVariant *v, int mode) {
    if (v->blocks || v->chain || v->elem_bytes != 4 || v->cpt != 1) return nullptr;
#define LINREC_FX(TD, TT, S, ST, M)                                                                          \
    if (mode == M) return reinterpret_cast<const void *>(&chunked_scan_kernel<kDtypeF32, TD, TT, S, ST, 1, false, M>);
#define LINREC_FX_ALL(TD, TT, S, ST)                                                                         \
    if (v->tile_d == TD && v->tile_t == TT && v->segments == S && v->stages == ST) {                         \
        LINREC_FX(TD, TT, S, ST, kModeOwn) LINREC_FX(TD, TT, S, ST, kModeLookback)                           \
        LINREC_FX(TD, TT, S, ST, kModeReduce) LINREC_FX(TD, TT, S, ST, kModeApply)                           \
    }
#define LINREC_FX_CHAINED(TD, TT, S, ST)                                                                     \
    if (v->tile_d == TD && v->tile_t == TT && v->segments == S && v->stages == ST) {                         \
        LINREC_FX(TD, TT, S, ST, kModeLookback) LINREC_FX(TD, TT, S, ST, kModeReduce)                        \
        LINREC_FX(TD, TT, S, ST, kModeApply)                                                                 \
    }
#define LINREC_FX_SPEC(TD, TT, S, ST)                                                                        \
    if (v->tile_d == TD && v->tile_t == TT && v->segments == S && v->stages == ST) {                         \
        LINREC_FX(TD, TT, S, ST, kModeSpec) LINREC_FX(TD, TT, S, ST, kModeRepair)                            \
    }
    LINREC_FIXED_F32_ALL(LINREC_FX_ALL)
    LINREC_FIXED_F32_CHAINED(LINREC_FX_CHAINED)
    LINREC_FIXED_F32_SPEC(LINREC_FX_SPEC)
#undef LINREC_FX_ALL
#undef LINREC_FX_CHAINED
#undef LINREC_FX_SPEC
#undef LINREC_FX
    return nullptr;
}

LINREC_CHECKED_REPORT(checked_report_fixed)

}  // namespace linrec
