// host_pipeline.cu -- linrec_scan_f32_host: the scan on host buffers, with the
// host-to-device copies, the kernels and the device-to-host copies of
// successive pieces overlapped.
//
// The problem is cut into pieces of nb batch indices x nl time steps (about
// kPieceBytes of a + b + h each).  Pieces of one batch group that follow each
// other in time are chained through the carry (linrec_scan_f32_carry's h_last
// of one piece is h_init of the next), so a single long sequence pipelines as
// well as a large batch.  Three device slots rotate over three internal
// streams:
//
//     copy-in stream:   wait slot free -> a, b piece to device  -> event in
//     compute stream:   wait in        -> scan (carry in/out)    -> event done
//     copy-out stream:  wait done      -> h piece to host        -> event free
//
// The caller's stream is joined at both ends: the pieces start after the work
// already queued on it, and it waits for the last copy-out.  Pieces are 2-D
// copies (rows = batch indices, pitch = L*D floats), so any piece of the
// row-major (B, L, D) host arrays moves as one cudaMemcpy2DAsync.
//
// When all three buffers are page-locked (or registered) host memory the GPU
// can address, the copies are skipped: the kernels read a, b and write h in
// host memory directly over the host link (measured on GB300: ~300 GB/s of
// scan traffic against ~250 GB/s for the copy pipeline, both close to the
// link's ~210 GB/s host-to-device read rate, and no device memory is used).
#include <cuda.h>
#include <cuda_runtime.h>

#include <mutex>

#include "linrec.h"

namespace {

typedef CUresult (*PointerAttrFn)(void *, CUpointer_attribute, CUdeviceptr);

// The driver's record of the address range p belongs to (its start and size), where the
// driver keeps one for this kind of memory; false when it does not say.
bool range_of(const void *p, uintptr_t *start, size_t *size) {
    static PointerAttrFn fn = nullptr;
    static std::once_flag once;
    std::call_once(once, [] {
        void *f = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuPointerGetAttribute", &f, 12000, cudaEnableDefault, &q) ==
                cudaSuccess && q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<PointerAttrFn>(f);
        cudaGetLastError();
    });
    if (!fn) return false;
    CUdeviceptr s0 = 0;
    size_t n = 0;
    const CUdeviceptr at = static_cast<CUdeviceptr>(reinterpret_cast<uintptr_t>(p));
    if (fn(&s0, CU_POINTER_ATTRIBUTE_RANGE_START_ADDR, at) != CUDA_SUCCESS ||
        fn(&n, CU_POINTER_ATTRIBUTE_RANGE_SIZE, at) != CUDA_SUCCESS)
        return false;
    *start = static_cast<uintptr_t>(s0);
    *size = n;
    return true;
}

// Whether the device can address every byte of [p, p + bytes) through page-locked host
// memory, and the device address of p.  A buffer only partly page-locked (a registration
// of a prefix of a larger block, a pointer into a pinned block shorter than the buffer)
// must take the copy pipeline: a kernel reading the rest would touch unmapped addresses.
// So the first and the last byte must both be page-locked host memory, mapped at device
// addresses the same distance apart, and, where the driver reports the range the first
// byte belongs to, that range must hold the last byte too.
bool mapped_whole(const void *p, size_t bytes, const void **dev) {
    const char *q = static_cast<const char *>(p);
    cudaPointerAttributes first, last;
    if (cudaPointerGetAttributes(&first, q) != cudaSuccess || cudaPointerGetAttributes(&last, q + bytes - 1) != cudaSuccess) {
        cudaGetLastError();
        return false;
    }
    if (first.type != cudaMemoryTypeHost || last.type != cudaMemoryTypeHost || !first.devicePointer ||
        !last.devicePointer)
        return false;
    if (static_cast<const char *>(last.devicePointer) != static_cast<const char *>(first.devicePointer) + (bytes - 1))
        return false;
    uintptr_t start = 0;
    size_t size = 0;
    if (range_of(p, &start, &size) && !linrec_debug_range_covers(start, size, reinterpret_cast<uintptr_t>(p), bytes))
        return false;
    *dev = first.devicePointer;
    return true;
}

constexpr int kSlots = 3;
constexpr int64_t kPieceBytes = 48ll << 20;   // a + b + h per piece

struct Pipe {
    bool ready = false;
    cudaStream_t in = nullptr, comp = nullptr, out = nullptr;
    cudaEvent_t ev_in[kSlots] = {}, ev_done[kSlots] = {}, ev_free[kSlots] = {}, ev_start = nullptr;
    float *buf = nullptr;          // kSlots x (a, b, h) of slot_elems floats each
    float *state = nullptr;        // carry between pieces of one batch group: nb x D
    int64_t slot_elems = 0, state_elems = 0;
};

std::mutex g_pipe_mu;
Pipe g_pipes[64];

bool make_pipe(Pipe &p) {
    if (p.ready) return true;
    if (cudaStreamCreateWithFlags(&p.in, cudaStreamNonBlocking) != cudaSuccess ||
        cudaStreamCreateWithFlags(&p.comp, cudaStreamNonBlocking) != cudaSuccess ||
        cudaStreamCreateWithFlags(&p.out, cudaStreamNonBlocking) != cudaSuccess ||
        cudaEventCreateWithFlags(&p.ev_start, cudaEventDisableTiming) != cudaSuccess)
        return false;
    for (int i = 0; i < kSlots; ++i) {
        if (cudaEventCreateWithFlags(&p.ev_in[i], cudaEventDisableTiming) != cudaSuccess ||
            cudaEventCreateWithFlags(&p.ev_done[i], cudaEventDisableTiming) != cudaSuccess ||
            cudaEventCreateWithFlags(&p.ev_free[i], cudaEventDisableTiming) != cudaSuccess)
            return false;
    }
    p.ready = true;
    return true;
}

// Device buffers for pieces of `elems` floats and a state of `state_elems`, grown in
// stream order on the copy-in stream (it is the first to touch a slot).
bool reserve(Pipe &p, int64_t elems, int64_t state_elems) {
    if (p.slot_elems < elems) {
        // the buffers may still be in use by queued pieces: free them after all three streams
        if (p.buf) {
            if (cudaStreamSynchronize(p.in) != cudaSuccess || cudaStreamSynchronize(p.comp) != cudaSuccess ||
                cudaStreamSynchronize(p.out) != cudaSuccess)
                return false;
            cudaFreeAsync(p.buf, p.in);
            p.buf = nullptr;
        }
        void *ptr = nullptr;
        if (cudaMallocAsync(&ptr, (size_t)elems * 3 * kSlots * sizeof(float), p.in) != cudaSuccess) return false;
        p.buf = static_cast<float *>(ptr);
        p.slot_elems = elems;
    }
    if (p.state_elems < state_elems) {
        if (p.state) {
            if (cudaStreamSynchronize(p.comp) != cudaSuccess) return false;
            cudaFreeAsync(p.state, p.comp);
            p.state = nullptr;
        }
        void *ptr = nullptr;
        if (cudaMallocAsync(&ptr, (size_t)state_elems * sizeof(float), p.comp) != cudaSuccess) return false;
        p.state = static_cast<float *>(ptr);
        p.state_elems = state_elems;
    }
    // the compute and copy-out streams must see the allocations made on the copy-in stream
    cudaEvent_t e = p.ev_start;
    if (cudaEventRecord(e, p.in) != cudaSuccess || cudaStreamWaitEvent(p.comp, e, 0) != cudaSuccess ||
        cudaStreamWaitEvent(p.out, e, 0) != cudaSuccess)
        return false;
    return true;
}

}  // namespace

extern "C" linrec_status_t linrec_scan_f32_host(const float *a, const float *b, float *h, int64_t B, int64_t L,
                                                int64_t D, void *stream_ptr) {
    if (B < 0 || L < 0 || D < 0) return LINREC_ERR_INVALID_VALUE;
    if (B == 0 || L == 0 || D == 0) return LINREC_OK;
    const int64_t lim = INT64_MAX / 16;
    if (L > lim / D || B > lim / (L * D)) return LINREC_ERR_INVALID_VALUE;
    if (!a || !b || !h) return LINREC_ERR_INVALID_VALUE;
    const int64_t n = B * L * D;
    const uintptr_t h0 = reinterpret_cast<uintptr_t>(h), hb = (uintptr_t)(n * 4);
    for (const void *in : {static_cast<const void *>(a), static_cast<const void *>(b)}) {
        const uintptr_t x = reinterpret_cast<uintptr_t>(in);
        if (x < h0 + hb && h0 < x + hb) return LINREC_ERR_ALIAS;
    }
    cudaStream_t user = static_cast<cudaStream_t>(stream_ptr);
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) {
        cudaGetLastError();
        return LINREC_ERR_LAUNCH;
    }

    // Page-locked host memory the device can address, every byte of it: scan it in place.
    const void *dptr[3] = {nullptr, nullptr, nullptr};
    bool direct = true;
    const void *hptr[3] = {a, b, h};
    for (int i = 0; i < 3 && direct; ++i) direct = mapped_whole(hptr[i], (size_t)n * sizeof(float), &dptr[i]);
    if (direct)
        return linrec_scan_f32(static_cast<const float *>(dptr[0]), static_cast<const float *>(dptr[1]),
                               static_cast<float *>(const_cast<void *>(dptr[2])), B, L, D, stream_ptr);

    // piece shape: whole sequences of nb batch indices, or nl steps of one batch index
    const int64_t per_step = D * 12;                     // bytes of a + b + h per time step
    int64_t nb, nl;
    if (L * per_step >= kPieceBytes) {
        nb = 1;
        nl = kPieceBytes / per_step;
        if (nl < 1) nl = 1;
    } else {
        nl = L;
        nb = kPieceBytes / (L * per_step);
        if (nb < 1) nb = 1;
        if (nb > B) nb = B;
    }
    const bool chained = nl < L;

    std::lock_guard<std::mutex> lock(g_pipe_mu);
    Pipe &p = g_pipes[dev];
    if (!make_pipe(p)) {
        cudaGetLastError();
        return LINREC_ERR_LAUNCH;
    }
    if (!reserve(p, nb * nl * D, nb * D)) {
        cudaGetLastError();
        return LINREC_ERR_WORKSPACE;
    }
    // start after the caller's queued work
    if (cudaEventRecord(p.ev_start, user) != cudaSuccess || cudaStreamWaitEvent(p.in, p.ev_start, 0) != cudaSuccess) {
        cudaGetLastError();
        return LINREC_ERR_LAUNCH;
    }

    const size_t pitch = (size_t)L * D * sizeof(float);
    int64_t k = 0;
    linrec_status_t st = LINREC_OK;
    for (int64_t b0 = 0; b0 < B && st == LINREC_OK; b0 += nb) {
        const int64_t pb = (B - b0 < nb) ? B - b0 : nb;
        for (int64_t l0 = 0; l0 < L; l0 += nl, ++k) {
            const int64_t pl = (L - l0 < nl) ? L - l0 : nl;
            const int slot = (int)(k % kSlots);
            float *da = p.buf + (size_t)slot * 3 * p.slot_elems;
            float *db = da + p.slot_elems;
            float *dh = db + p.slot_elems;
            const size_t width = (size_t)pl * D * sizeof(float);
            const size_t off = (size_t)(b0 * L + l0) * D;
            cudaError_t err = cudaSuccess;
            if (k >= kSlots) err = cudaStreamWaitEvent(p.in, p.ev_free[slot], 0);
            if (err == cudaSuccess) err = cudaMemcpy2DAsync(da, width, a + off, pitch, width, pb,
                                                            cudaMemcpyHostToDevice, p.in);
            if (err == cudaSuccess) err = cudaMemcpy2DAsync(db, width, b + off, pitch, width, pb,
                                                            cudaMemcpyHostToDevice, p.in);
            if (err == cudaSuccess) err = cudaEventRecord(p.ev_in[slot], p.in);
            if (err == cudaSuccess) err = cudaStreamWaitEvent(p.comp, p.ev_in[slot], 0);
            if (err != cudaSuccess) {
                cudaGetLastError();
                st = LINREC_ERR_LAUNCH;
                break;
            }
            st = linrec_scan_f32_carry(da, db, dh, pb, pl, D, (chained && l0 > 0) ? p.state : nullptr,
                                       chained ? p.state : nullptr, p.comp);
            if (st != LINREC_OK) break;
            err = cudaEventRecord(p.ev_done[slot], p.comp);
            if (err == cudaSuccess) err = cudaStreamWaitEvent(p.out, p.ev_done[slot], 0);
            if (err == cudaSuccess) err = cudaMemcpy2DAsync(h + off, pitch, dh, width, width, pb,
                                                            cudaMemcpyDeviceToHost, p.out);
            if (err == cudaSuccess) err = cudaEventRecord(p.ev_free[slot], p.out);
            if (err != cudaSuccess) {
                cudaGetLastError();
                st = LINREC_ERR_LAUNCH;
                break;
            }
        }
    }
    // the caller's stream waits for the last copy-out (also on failure, for what was queued)
    cudaEvent_t last = p.ev_free[(k + kSlots - 1) % kSlots];
    if (k > 0 && (cudaStreamWaitEvent(user, last, 0) != cudaSuccess)) {
        cudaGetLastError();
        if (st == LINREC_OK) st = LINREC_ERR_LAUNCH;
    }
    return st;
}

extern "C" int linrec_debug_range_covers(uintptr_t range_start, size_t range_size, uintptr_t p, size_t bytes) {
    // [p, p + bytes) inside [range_start, range_start + range_size), without overflow
    if (bytes == 0 || p < range_start) return 0;
    const uintptr_t off = p - range_start;
    return off <= range_size && bytes <= range_size - off ? 1 : 0;
}
