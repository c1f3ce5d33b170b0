// noalloc.cu -- linrec_scan_f32_noalloc: the chunked look-back scan with its
// scratch in a fixed array compiled into the library, for callers that may
// not allocate device memory (see include/linrec.h for who they are).
//
// Nothing here allocates: no cudaMalloc / cudaMallocAsync / cudaFree, and no
// library routine that does.  The array below is a static __device__ object:
// each device that loads the library holds it until the process exits.
#include <cuda.h>
#include <cuda_runtime.h>

#include <mutex>

#include "kernels.cuh"
#include "linrec.h"

using namespace linrec;

namespace {

// [Control block, padded to 256 bytes][look-back words].  Zero at load time.
static __device__ __align__(256) unsigned char g_noalloc_scratch[LINREC_NOALLOC_SCRATCH_BYTES];

constexpr size_t kHead = 256;
constexpr int kMaxDevices = 64;
constexpr int64_t kSpinLimit = 1 << 20;

struct DeviceSetup {
    bool ready = false;
    bool supported = false;
    int sm_count = 0;
    unsigned char *scratch = nullptr;   // device address of g_noalloc_scratch on this device
    int ctas_per_sm[64] = {};
};

std::mutex g_mu;
DeviceSetup g_setup[kMaxDevices];

typedef CUresult (*EncodeTiledFn)(CUtensorMap *, CUtensorMapDataType, cuuint32_t, void *, const cuuint64_t *,
                                  const cuuint64_t *, const cuuint32_t *, const cuuint32_t *, CUtensorMapInterleave,
                                  CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);
EncodeTiledFn g_encode = nullptr;

// Once per device, with that device current: its facts and the array's device address.
// In host code g_noalloc_scratch names a host-side stand-in, never the device memory.
bool setup_device(int dev, DeviceSetup *&out) {
    DeviceSetup &s = g_setup[dev];
    if (!s.ready) {
        int major = 0, minor = 0, sms = 0;
        if (cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev) != cudaSuccess ||
            cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev) != cudaSuccess ||
            cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) {
            cudaGetLastError();
            return false;
        }
        s.supported = (major == 10 && minor == 3);
        s.sm_count = sms;
        if (s.supported) {
            void *ptr = nullptr;
            if (cudaGetSymbolAddress(&ptr, g_noalloc_scratch) != cudaSuccess || ptr == nullptr) {
                cudaGetLastError();
                return false;
            }
            s.scratch = static_cast<unsigned char *>(ptr);
        }
        s.ready = true;
    }
    out = &s;
    return true;
}

bool encode(CUtensorMap *map, const float *base, int64_t B, int64_t L, int64_t D, int tile_d, int tile_t) {
    const cuuint64_t dims[3] = {(cuuint64_t)D, (cuuint64_t)L, (cuuint64_t)B};
    const cuuint64_t strides[2] = {(cuuint64_t)D * 4u, (cuuint64_t)L * (cuuint64_t)D * 4u};
    const cuuint32_t box[3] = {(cuuint32_t)tile_d, (cuuint32_t)tile_t, 1u};
    const cuuint32_t estr[3] = {1u, 1u, 1u};
    return g_encode(map, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 3, const_cast<float *>(base), dims, strides, box, estr,
                    CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                    CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

bool overlap(const void *x, const void *y, int64_t bytes) {
    const uintptr_t a0 = reinterpret_cast<uintptr_t>(x), b0 = reinterpret_cast<uintptr_t>(y);
    return a0 < b0 + (uintptr_t)bytes && b0 < a0 + (uintptr_t)bytes;
}

}  // namespace

namespace linrec {

// The array's status word on device `dev` (set by noalloc calls made without a status
// word of their own), read on `stream` and cleared when set; 0 if the device has not run
// such a call.  Called by linrec_stream_status.
cudaError_t noalloc_take_status(int dev, cudaStream_t stream, unsigned int *word) {
    *word = 0;
    if (dev < 0 || dev >= kMaxDevices) return cudaSuccess;
    unsigned int *status = nullptr;
    {
        std::lock_guard<std::mutex> lock(g_mu);
        if (!g_setup[dev].ready || !g_setup[dev].scratch) return cudaSuccess;
        status = &reinterpret_cast<Control *>(g_setup[dev].scratch)->status;
    }
    cudaError_t e = cudaMemcpyAsync(word, status, sizeof(*word), cudaMemcpyDeviceToHost, stream);
    if (e == cudaSuccess) e = cudaStreamSynchronize(stream);
    if (e == cudaSuccess && *word != 0) {
        e = cudaMemsetAsync(status, 0, sizeof(*word), stream);
        if (e == cudaSuccess) e = cudaStreamSynchronize(stream);
    }
    return e;
}

// Tests: the array's epoch word on device `dev` (set up first), written synchronously.
cudaError_t noalloc_set_epoch(int dev, unsigned int epoch) {
    DeviceSetup *ds = nullptr;
    {
        std::lock_guard<std::mutex> lock(g_mu);
        if (dev < 0 || dev >= kMaxDevices || !setup_device(dev, ds) || !ds->scratch) return cudaErrorInvalidValue;
    }
    Control *ctrl = reinterpret_cast<Control *>(ds->scratch);
    return cudaMemcpy(&ctrl->epoch, &epoch, sizeof(epoch), cudaMemcpyHostToDevice);
}

}  // namespace linrec

extern "C" linrec_status_t linrec_scan_f32_noalloc(const float *a, const float *b, float *h, int64_t B, int64_t L,
                                                   int64_t D, void *stream_ptr, unsigned int *d_status) {
    if (B < 0 || L < 0 || D < 0) return LINREC_ERR_INVALID_VALUE;
    if (B == 0 || L == 0 || D == 0) return LINREC_OK;
    const int64_t lim = INT64_MAX / 16;
    if (L > lim / D || B > lim / (L * D)) return LINREC_ERR_INVALID_VALUE;
    const int64_t n = B * L * D;
    if (!a || !b || !h) return LINREC_ERR_INVALID_VALUE;
    if (overlap(h, a, n * 4) || overlap(h, b, n * 4)) return LINREC_ERR_ALIAS;
    const uintptr_t al = reinterpret_cast<uintptr_t>(a) | reinterpret_cast<uintptr_t>(b) |
                         reinterpret_cast<uintptr_t>(h);
    if ((al & 15u) != 0 || D % 4 != 0) return LINREC_ERR_INVALID_VALUE;
    cudaStream_t stream = static_cast<cudaStream_t>(stream_ptr);

    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) {
        cudaGetLastError();
        return LINREC_ERR_LAUNCH;
    }
    if (dev < 0 || dev >= kMaxDevices) return LINREC_ERR_LAUNCH;
    std::lock_guard<std::mutex> lock(g_mu);
    DeviceSetup *ds = nullptr;
    if (!setup_device(dev, ds)) return LINREC_ERR_LAUNCH;
    if (!ds->supported) return LINREC_ERR_UNSUPPORTED_DEVICE;

    // The dispatcher's chunked tile for this shape, then the resident CTAs of that variant.
    linrec_options_t opt = {};
    opt.path = LINREC_PATH_CHUNKED;
    // one launch on the fixed array: slice-owner or look-back mode, never the two-pass mode
    {
        linrec_plan_t probe;
        if (linrec_plan_f32(B, L, D, ds->sm_count, 16, 0, &opt, &probe) == LINREC_OK &&
            (probe.twopass || probe.blocks || probe.chain || probe.speculative))
            opt.chunk_mode = 2;
    }
    linrec_plan_t plan;
    linrec_status_t st = linrec_plan_f32(B, L, D, ds->sm_count, 16, 0, &opt, &plan);
    if (st != LINREC_OK) return st;
    if (plan.workspace_bytes > LINREC_NOALLOC_SCRATCH_BYTES) return LINREC_ERR_WORKSPACE;
    int nvar = 0;
    const ChunkedVariant *vars = chunked_variants(&nvar);
    int vi = -1;
    for (int i = 0; i < nvar && i < 64; ++i)
        if (vars[i].tile_d == plan.tile_d && vars[i].tile_t == plan.tile_t && vars[i].stages == plan.stages &&
            !vars[i].blocks)
            vi = i;
    if (vi < 0) return LINREC_ERR_INVALID_VALUE;
    if (ds->ctas_per_sm[vi] == 0) {
        int c = 0;
        if (chunked_ctas_per_sm(&vars[vi], &c) != cudaSuccess || c <= 0) {
            cudaGetLastError();
            return LINREC_ERR_LAUNCH;
        }
        ds->ctas_per_sm[vi] = c;
    }
    st = linrec_plan_f32(B, L, D, ds->sm_count, 16, ds->ctas_per_sm[vi], &opt, &plan);
    if (st != LINREC_OK) return st;

    if (!g_encode) {
        void *fn = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000, cudaEnableDefault, &q) !=
                cudaSuccess || q != cudaDriverEntryPointSuccess || !fn) {
            cudaGetLastError();
            return LINREC_ERR_LAUNCH;
        }
        g_encode = reinterpret_cast<EncodeTiledFn>(fn);
    }
    ChunkedLaunch p;
    p.variant = &vars[vi];
    if (!encode(&p.map_a, a, B, L, D, plan.tile_d, plan.tile_t) ||
        !encode(&p.map_b, b, B, L, D, plan.tile_d, plan.tile_t))
        return LINREC_ERR_LAUNCH;

    // The tile counter, the done count and the abort word start at zero (the array is zero
    // when the library loads) and the last CTA of every launch resets them, a launch whose
    // waits ran out included; the epoch word it advances tells this call's look-back words
    // from those earlier calls left in the array.  So nothing is cleared here, and nothing
    // comes between this launch and the work before it on the stream.
    Control *ctrl = reinterpret_cast<Control *>(ds->scratch);
    p.h = h;
    p.L = L;
    p.D = D;
    p.slices_per_batch = (D + plan.tile_d - 1) / plan.tile_d;
    p.n_slices = B * p.slices_per_batch;
    p.chunks = plan.chunks;
    p.n_tiles = plan.n_tiles;
    p.grid = plan.grid;
    p.mode = plan.lookback ? kModeLookback : kModeOwn;
    p.ctrl = ctrl;
    p.words = reinterpret_cast<unsigned long long *>(ds->scratch + kHead);
    p.status = d_status ? d_status : &ctrl->status;
    p.spin_limit = kSpinLimit;
    p.silent_tile = -1;
    if (launch_chunked(p, stream) != cudaSuccess) {
        cudaGetLastError();
        return LINREC_ERR_LAUNCH;
    }
    return LINREC_OK;
}
