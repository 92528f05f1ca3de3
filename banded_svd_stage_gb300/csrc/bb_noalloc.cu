// bb_reduce_noalloc: the reduction without any device allocation.
//
// Some callers cannot allocate device memory at the point where they need the
// reduction: their device memory is owned by another allocator or a fixed
// pool that hands out no extra buffers, or they run where cudaMalloc /
// cudaFree are not acceptable (cudaFree synchronizes the whole device, and
// either call can stall or fail under a memory budget).  bb_create allocates
// the per-sweep progress counters and the status word, so those callers
// cannot use bb_reduce.  This entry point takes that scratch from a fixed
// array in the library's own device image instead; the caller passes only
// the band and the outputs.
#include <cuda_runtime.h>

#include <mutex>
#include <string>

#include "../../include/bb.h"
#include "bb_internal.h"

namespace {

// Scratch of the persistent scheduler: entries [0, n) are the per-sweep
// progress counters of the pass being run, entry kNoAllocMaxN the device
// status word.  Every device that loads the library holds this array (256
// KiB + 256 B) until the process exits.
constexpr int64_t kNoAllocMaxN = 65536;
constexpr int kStatusIndex = (int)kNoAllocMaxN;
static __device__ __align__(256) int g_noalloc_scratch[kNoAllocMaxN + 64];

struct DeviceSlot {
    bool ready = false;
    int* scratch = nullptr;  // device address of g_noalloc_scratch on this device
    int num_sms = 0;
    int clock_khz = 0;
};

constexpr int kMaxDevices = 64;
std::mutex g_mu;
DeviceSlot g_slots[kMaxDevices];

bb_status fail(bb_status st, const std::string& msg) {
    bb::set_last_error(msg.c_str());
    return st;
}

// Once per device, with that device current: the device address of the
// scratch array (host code only knows a host-side stand-in for its name).
bb_status device_slot(DeviceSlot** out) {
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return fail(BB_ERR_CUDA, std::string("cudaGetDevice: ") + cudaGetErrorString(e));
    if (dev < 0 || dev >= kMaxDevices) return fail(BB_ERR_INVALID_ARG, "device ordinal too large");
    std::lock_guard<std::mutex> lock(g_mu);
    DeviceSlot& s = g_slots[dev];
    if (!s.ready) {
        void* ptr = nullptr;
        e = cudaGetSymbolAddress(&ptr, g_noalloc_scratch);
        if (e != cudaSuccess || ptr == nullptr)
            return fail(BB_ERR_CUDA, std::string("cudaGetSymbolAddress(scratch): ") + cudaGetErrorString(e));
        e = cudaDeviceGetAttribute(&s.num_sms, cudaDevAttrMultiProcessorCount, dev);
        if (e == cudaSuccess) e = cudaDeviceGetAttribute(&s.clock_khz, cudaDevAttrClockRate, dev);
        if (e != cudaSuccess) return fail(BB_ERR_CUDA, std::string("device attributes: ") + cudaGetErrorString(e));
        if (s.clock_khz <= 0) s.clock_khz = 2000000;
        s.scratch = static_cast<int*>(ptr);
        s.ready = true;
    }
    *out = &s;
    return BB_OK;
}

bool on_device(const void* p) {
    cudaPointerAttributes a;
    if (cudaPointerGetAttributes(&a, p) != cudaSuccess) {
        cudaGetLastError();
        return false;
    }
    return a.type == cudaMemoryTypeDevice || a.type == cudaMemoryTypeManaged;
}

template <typename T>
bb_status run_all(T* band, int64_t n, int64_t bw, int64_t ldab, int64_t tw, T* d, T* e,
                  const DeviceSlot& slot, cudaStream_t s) {
    int* progress = slot.scratch;
    int* status = slot.scratch + kStatusIndex;
    const int ku = (int)(bw + tw);
    // the status word keeps the previous call's value: clear it first
    cudaError_t err = cudaMemsetAsync(status, 0, sizeof(int), s);
    if (err == cudaSuccess) err = bb::run_zero_fill<T>(band, n, ldab, (int)tw, ku, s);
    int64_t b = bw;
    while (err == cudaSuccess && b > 1) {
        const int64_t t = std::min<int64_t>(tw, b - 1);
        bb::PassArgs P;
        P.n = n;
        P.ldab = ldab;
        P.b = (int)b;
        P.t = (int)t;
        P.bp = (int)(b - t);
        P.ku = ku;
        P.nsweeps = (int)std::max<int64_t>(0, n - (b - t) - 1);
        P.lag = bb::pass_lag_cycle((int)b, (int)t);
        P.lagh = bb::pass_lag_half((int)b, (int)t);
        P.stall_sweep = -1;
        P.wait_budget = 4000ULL * (unsigned long long)slot.clock_khz;  // 4 s
        bb::LaunchCfg cfg;
        cfg.tpb = bb::auto_tpb((int)b, (int)t);
        cfg.max_ctas = 0;
        cfg.num_sms = slot.num_sms;
        // run_pass clears the progress counters of the pass before launching
        err = bb::run_pass<T>(band, P, 0, cfg, progress, status, s, nullptr);
        b -= t;
    }
    if (err == cudaSuccess) err = bb::run_extract<T>(band, n, ldab, ku, d, e, s);
    if (err != cudaSuccess) {
        // Work of earlier passes may still run on the shared scratch: drain the
        // stream before the caller's lock is released, so that the next call
        // does not clear the counters and the status word under it.
        (void)cudaStreamSynchronize(s);
        (void)cudaGetLastError();
        return fail(BB_ERR_CUDA, std::string("launch: ") + cudaGetErrorString(err));
    }
    int st = 0;
    err = cudaMemcpyAsync(&st, status, sizeof(int), cudaMemcpyDeviceToHost, s);
    const cudaError_t sync_err = cudaStreamSynchronize(s);  // always drained before the lock is released
    if (err == cudaSuccess) err = sync_err;
    if (err != cudaSuccess) return fail(BB_ERR_CUDA, std::string("completion: ") + cudaGetErrorString(err));
    if (st != 0) return fail((bb_status)st, "device-side progress wait timed out");
    return BB_OK;
}

}  // namespace

extern "C" bb_status bb_reduce_noalloc(void* band_ptr, int64_t n, int64_t bw, int64_t ldab,
                                       int64_t tw, bb_dtype dtype, void* d_out, void* e_out,
                                       bb_stream_t stream) {
    if (dtype != BB_F32 && dtype != BB_F64) return fail(BB_ERR_DTYPE, "unknown dtype");
    if (n < 1 || bw < 0 || bw >= n) return fail(BB_ERR_INVALID_ARG, "need n >= 1 and 0 <= bw < n");
    if (n > kNoAllocMaxN)
        return fail(BB_ERR_INVALID_ARG, "bb_reduce_noalloc: n exceeds the fixed scratch of 65536 sweeps; "
                                        "use bb_create/bb_reduce for larger matrices");
    if (tw < 1 || tw > std::max<int64_t>(1, bw - 1)) return fail(BB_ERR_INVALID_ARG, "need 1 <= tw <= max(1, bw - 1)");
    if (tw > 64) return fail(BB_ERR_INVALID_ARG, "tw > 64 is not supported");
    if (ldab < bw + 2 * tw + 1) return fail(BB_ERR_LDAB, "ldab < bw + 2*tw + 1");
    {
        const size_t es = dtype == BB_F64 ? 8 : 4;
        const int w1 = (int)tw + 1;
        const int wm = w1 <= 8 ? 8 : w1 <= 9 ? 9 : w1 <= 16 ? 16 : w1 <= 17 ? 17 : w1 <= 32 ? 32 : w1 <= 33 ? 33 : 65;
        const size_t smem = es * ((size_t)wm + 2 + (size_t)(2 * (bw + tw) + 1) * (wm | 1));
        if (smem > 227 * 1024) return fail(BB_ERR_INVALID_ARG, "bandwidth too large for the shared-memory tile");
    }
    if (!band_ptr || !d_out || (n > 1 && !e_out)) return fail(BB_ERR_INVALID_ARG, "null band, d or e pointer");
    if (!on_device(band_ptr) || !on_device(d_out) || (n > 1 && !on_device(e_out)))
        return fail(BB_ERR_INVALID_ARG, "band, d and e must be device pointers");
    DeviceSlot* slot = nullptr;
    bb_status st = device_slot(&slot);
    if (st != BB_OK) return st;
    std::lock_guard<std::mutex> lock(g_mu);  // one call at a time per process uses the scratch
    cudaStream_t s = (cudaStream_t)stream;
    if (dtype == BB_F32)
        return run_all<float>((float*)band_ptr, n, bw, ldab, tw, (float*)d_out, (float*)e_out, *slot, s);
    return run_all<double>((double*)band_ptr, n, bw, ldab, tw, (double*)d_out, (double*)e_out, *slot, s);
}
