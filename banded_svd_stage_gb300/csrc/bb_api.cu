// C-ABI layer of libbb.so: argument checks, the pass planner, workspace
// ownership and the launch sequence of one reduction.  See include/bb.h.
#include <cuda_runtime.h>

#include <algorithm>
#include <cstdio>
#include <cstring>
#include <new>
#include <string>
#include <vector>

#include "../../include/bb.h"
#include "bb_half.h"
#include "bb_internal.h"
#include "bb_sym.h"
#include "bb_vectors.h"

namespace {

thread_local std::string g_last_error;

bb_status fail(bb_status st, const std::string& msg) {
    g_last_error = msg;
    return st;
}

bb_status cuda_fail(cudaError_t e, const char* what) {
    return fail(BB_ERR_CUDA, std::string(what) + ": " + cudaGetErrorString(e));
}

struct PassPlan {
    int b, t;
};

// Largest order (and so bandwidth) any entry point accepts.
constexpr int64_t kMaxOrder = (int64_t)1 << 30;

// The plan: b = bw; while b > 1: t = min(tw, b - 1); pass (b, t); b -= t.
// Every pass but the last removes tw and the last ends at 1, so pass i is
// b = bw - i tw, t = min(tw, b - 1), and there are ceil((bw - 1) / tw).
int64_t count_passes(int64_t bw, int64_t tw) {
    if (bw <= 1 || bw > kMaxOrder || tw < 1) return 0;
    return (bw - 1 + tw - 1) / tw;
}
PassPlan pass_at(int64_t bw, int64_t tw, int64_t i) {
    const int64_t b = bw - i * tw;
    return {(int)b, (int)std::min(tw, b - 1)};
}
// The whole plan, for callers whose bandwidth is already bounded by the
// shared-memory check of its widest pass (at most a few thousand passes).
std::vector<PassPlan> plan_passes(int64_t bw, int64_t tw) {
    std::vector<PassPlan> out;
    const int64_t np = count_passes(bw, tw);
    out.reserve((size_t)np);
    for (int64_t i = 0; i < np; ++i) out.push_back(pass_at(bw, tw, i));
    return out;
}

// Shared memory of the flag kernel's tile for pass (b, t): the widest pass,
// the first, decides whether a reduction fits.
size_t flag_tile_bytes(int64_t b, int64_t t, size_t elem) {
    const int64_t w = t + 1;
    const int64_t wm = w <= 8 ? 8 : w <= 9 ? 9 : w <= 16 ? 16 : w <= 17 ? 17 : w <= 32 ? 32 : w <= 33 ? 33 : 65;
    return elem * ((size_t)wm + 2 + (size_t)(2 * (b + t) + 1) * (size_t)(wm | 1));
}

int64_t steps_of_sweep(int64_t n, int b, int t, int64_t r) {
    int64_t last = n - 2 - r - (b - t);
    return last < 0 ? 0 : last / b + 1;
}

size_t elem_size(bb_dtype d) { return d == BB_F64 ? 8 : d == BB_F16 ? 2 : 4; }

bool is_device_pointer(const void* p) {
    cudaPointerAttributes a;
    if (cudaPointerGetAttributes(&a, p) != cudaSuccess) {
        cudaGetLastError();
        return false;
    }
    return a.type == cudaMemoryTypeDevice || a.type == cudaMemoryTypeManaged;
}

}  // namespace

struct bb_handle {
    int64_t n = 0, bw = 0;
    bb_dtype dtype = BB_F32;
    int device = 0, num_sms = 0, clock_khz = 0;
    int* d_progress = nullptr;  // n int32 per-sweep progress counters
    int* d_status = nullptr;    // device status word
    // parameters
    int scheduler = 0, tpb = 0, max_ctas = 0, stall_sweep = -1, timing = 0, group_size = 0;
    int64_t wait_ms = 4000, pass_lo = 0, pass_hi = 1 << 30;
    // staging buffers of bb_reduce_host
    void* s_band = nullptr;
    size_t s_band_bytes = 0;
    void* s_de = nullptr;
    // working copy of the band with a 16-byte aligned column stride (group
    // kernel on a caller layout its bulk copies cannot address)
    void* work = nullptr;
    size_t work_bytes = 0;
    // scheduler 4: per-cycle launches of each pass captured once in a CUDA
    // graph (on a stream of the handle) and replayed on the caller's stream
    struct PassGraph {
        const void* band = nullptr;
        int64_t ldab = 0, n = 0;
        int b = 0, t = 0, tpb = 0;
        int64_t launches = 0;
        cudaGraphExec_t exec = nullptr;
    };
    std::vector<PassGraph> graphs;  // by pass index
    cudaStream_t capture_stream = nullptr;
    // reflector record of the last whole reduction (BB_PARAM_RECORD)
    int record = 0;
    void* rec_v = nullptr;
    void* rec_tau = nullptr;
    long long* rec_prefix = nullptr;  // per pass, steps of the sweeps before r
    size_t rec_v_bytes = 0, rec_tau_bytes = 0, rec_prefix_bytes = 0;
    std::vector<long long> rec_prefix_host;
    bool rec_valid = false;
    int64_t rec_tw = 0;
    // statistics of the last reduction
    int64_t last_launches = 0;
    std::vector<cudaEvent_t> ev;  // 2 per pass
    int64_t last_passes = 0;
    std::vector<int> pass_kernel, pass_group;  // per pass of the last reduction
};

extern "C" {

const char* bb_last_error(void) { return g_last_error.c_str(); }

int64_t bb_required_ldab(int64_t bw, int64_t tw) { return bw + 2 * tw + 1; }

int64_t bb_num_passes(int64_t bw, int64_t tw) { return count_passes(bw, tw); }

bb_status bb_pass_info(int64_t bw, int64_t tw, int64_t i, int64_t* b, int64_t* t) {
    if (i < 0 || i >= count_passes(bw, tw) || !b || !t)
        return fail(BB_ERR_INVALID_ARG, "bb_pass_info: pass index out of range");
    const PassPlan ps = pass_at(bw, tw, i);
    *b = ps.b;
    *t = ps.t;
    return BB_OK;
}

// The group-kernel plan queries of bb_group_plan (sym = false: the
// bidiagonal chase; elem_bytes 2 = binary16 columns) and bb_sym_group_plan
// (sym = true, elem_bytes 4 or 8).
static bb_status group_plan_query(const char* who, bool sym, int64_t n, int64_t bw, int64_t tw, int64_t elem_bytes,
                                  int64_t pass, int64_t group_size, int64_t* g, int64_t* nslot, int64_t* ahead,
                                  int64_t* lds) {
    const bool elem_ok = (elem_bytes == 4 || elem_bytes == 8 || (!sym && elem_bytes == 2));
    if (n < 1 || n >= bb::kGroupMaxN || bw < 0 || bw >= n || tw < 1 || tw > std::max<int64_t>(1, bw - 1) ||
        pass < 0 || pass >= count_passes(bw, tw) || !g || !nslot || !ahead || !lds || !elem_ok || group_size < 0)
        return fail(BB_ERR_INVALID_ARG, std::string(who) + ": argument out of range");
    try {
        const PassPlan ps = pass_at(bw, tw, pass);
        bb::PassArgs P{};
        P.n = n;
        P.b = ps.b;
        P.t = ps.t;
        P.bp = P.b - P.t;
        P.nsweeps = (int)std::max<int64_t>(0, n - P.bp - 1);
        bb::GroupArgs ga{};
        bool ok;
        if (sym) {  // lower band storage, one two-sided step per tick
            P.ku = 0;
            P.lag = bb::sym_pass_lag(P.b, P.t);
            P.lagh = P.lag;
            const int wmax = bb::sym_group_wmax(P.t + 1);
            ok = P.nsweeps > 0 && wmax > 0 &&
                 bb::plan_group(P, wmax, (size_t)elem_bytes, (int)group_size, &ga, bb::ChaseKind::kSym);
        } else {
            P.ku = (int)(bw + tw);
            P.lagh = bb::pass_lag_half(P.b, P.t);
            if (elem_bytes == 2)  // binary16 storage, float arithmetic
                ok = bb::half_choose_group(P, 3, (int)group_size, &ga);
            else
                ok = P.nsweeps > 0 &&
                     bb::plan_group(P, bb::wmax_bucket(P.t + 1), (size_t)elem_bytes, (int)group_size, &ga);
        }
        *g = ok ? ga.g : 0;
        *nslot = ok ? ga.nslot : 0;
        *ahead = ok ? ga.ahead : 0;
        *lds = ok ? ga.lds : 0;
        return BB_OK;
    } catch (const std::bad_alloc&) {
        return fail(BB_ERR_NOMEM, std::string(who) + ": host allocation failed");
    } catch (...) {
        return fail(BB_ERR_INTERNAL, std::string(who) + ": unexpected host exception");
    }
}

bb_status bb_group_plan(int64_t n, int64_t bw, int64_t tw, int64_t elem_bytes, int64_t pass, int64_t group_size,
                        int64_t* g, int64_t* nslot, int64_t* ahead, int64_t* lds) {
    return group_plan_query("bb_group_plan", false, n, bw, tw, elem_bytes, pass, group_size, g, nslot, ahead, lds);
}

bb_status bb_sym_group_plan(int64_t n, int64_t bw, int64_t tw, int64_t elem_bytes, int64_t pass,
                            int64_t group_size, int64_t* g, int64_t* nslot, int64_t* ahead, int64_t* lds) {
    return group_plan_query("bb_sym_group_plan", true, n, bw, tw, elem_bytes, pass, group_size, g, nslot, ahead,
                            lds);
}

double bb_model_bytes(int64_t n, int64_t bw, int64_t tw, int64_t elem_bytes, int64_t pass) {
    double total = 0;
    const int64_t np = count_passes(bw, tw);
    for (int64_t pi = 0; pi < np; ++pi) {
        if (pass >= 0 && pi != pass) continue;
        const PassPlan ps = pass_at(bw, tw, pi);
        const int b = ps.b, t = ps.t;
        for (int64_t r = 0; r + (b - t) + 1 <= n - 1; ++r) {
            const int64_t K = steps_of_sweep(n, b, t, r);
            for (int64_t k = 0; k < K; ++k) {
                const int64_t c = r + (b - t) + k * b;
                const int64_t p = (k == 0) ? r : c - b;
                const int64_t ce = std::min(c + t, n - 1);
                const int64_t cend = std::min(ce + b, n - 1);
                const int64_t w = ce - c + 1;
                total += 2.0 * elem_bytes * (double)((ce - p + 1) * w + w * (cend - c + 1));
            }
        }
    }
    return total;
}

int64_t bb_model_steps(int64_t n, int64_t bw, int64_t tw, int64_t pass) {
    int64_t total = 0;
    const int64_t np = count_passes(bw, tw);
    for (int64_t pi = 0; pi < np; ++pi) {
        if (pass >= 0 && pi != pass) continue;
        const PassPlan ps = pass_at(bw, tw, pi);
        const int b = ps.b, t = ps.t;
        for (int64_t r = 0; r + (b - t) + 1 <= n - 1; ++r) total += steps_of_sweep(n, b, t, r);
    }
    return total;
}

bb_handle* bb_create(int64_t n, int64_t bw, bb_dtype dtype) {
    if (dtype != BB_F32 && dtype != BB_F64 && dtype != BB_F16) {
        fail(BB_ERR_DTYPE, "bb_create: unknown dtype");
        return nullptr;
    }
    if (n < 1 || n > kMaxOrder || bw < 0 || bw >= n) {
        fail(BB_ERR_INVALID_ARG, "bb_create: need n >= 1 and 0 <= bw < n");
        return nullptr;
    }
    bb_handle* h = new (std::nothrow) bb_handle();
    if (!h) {
        fail(BB_ERR_NOMEM, "bb_create: host allocation failed");
        return nullptr;
    }
    h->n = n;
    h->bw = bw;
    h->dtype = dtype;
    cudaError_t e = cudaGetDevice(&h->device);
    if (e == cudaSuccess) e = cudaDeviceGetAttribute(&h->num_sms, cudaDevAttrMultiProcessorCount, h->device);
    if (e == cudaSuccess) e = cudaDeviceGetAttribute(&h->clock_khz, cudaDevAttrClockRate, h->device);
    if (e == cudaSuccess) e = cudaMalloc(&h->d_progress, sizeof(int) * (size_t)n);
    if (e == cudaSuccess) e = cudaMalloc(&h->d_status, sizeof(int));
    if (e == cudaSuccess) e = cudaMemset(h->d_status, 0, sizeof(int));
    if (e != cudaSuccess) {
        cuda_fail(e, "bb_create");
        bb_destroy(h);
        return nullptr;
    }
    if (h->clock_khz <= 0) h->clock_khz = 2000000;
    return h;
}

void bb_destroy(bb_handle* h) {
    if (!h) return;
    if (h->d_progress) cudaFree(h->d_progress);
    if (h->d_status) cudaFree(h->d_status);
    if (h->s_band) cudaFree(h->s_band);
    if (h->s_de) cudaFree(h->s_de);
    if (h->rec_v) cudaFree(h->rec_v);
    if (h->rec_tau) cudaFree(h->rec_tau);
    if (h->rec_prefix) cudaFree(h->rec_prefix);
    if (h->work) cudaFree(h->work);
    for (auto& pg : h->graphs)
        if (pg.exec) cudaGraphExecDestroy(pg.exec);
    if (h->capture_stream) cudaStreamDestroy(h->capture_stream);
    for (auto ev : h->ev) cudaEventDestroy(ev);
    delete h;
}

bb_status bb_set_param(bb_handle* h, int param, int64_t value) {
    if (!h) return fail(BB_ERR_INVALID_ARG, "bb_set_param: null handle");
    switch (param) {
        case BB_PARAM_SCHEDULER:
            if (value < 0 || value > 4) return fail(BB_ERR_INVALID_ARG, "scheduler must be 0, 1, 2, 3 or 4");
            h->scheduler = (int)value;
            return BB_OK;
        case BB_PARAM_TPB:
            if (value != 0 && (value < 32 || value > 1024 || value % 32 != 0))
                return fail(BB_ERR_INVALID_ARG, "tpb must be 0 or a multiple of 32 in [32, 1024]");
            h->tpb = (int)value;
            return BB_OK;
        case BB_PARAM_MAX_CTAS:
            if (value < 0 || value > (1 << 20)) return fail(BB_ERR_INVALID_ARG, "max_ctas out of range");
            h->max_ctas = (int)value;
            return BB_OK;
        case BB_PARAM_WAIT_BUDGET_MS:
            if (value < 1 || value > 600000) return fail(BB_ERR_INVALID_ARG, "wait budget out of range");
            h->wait_ms = value;
            return BB_OK;
        case BB_PARAM_PASS_LO:
            if (value < 0) return fail(BB_ERR_INVALID_ARG, "pass_lo < 0");
            h->pass_lo = value;
            return BB_OK;
        case BB_PARAM_PASS_HI:
            if (value < 0) return fail(BB_ERR_INVALID_ARG, "pass_hi < 0");
            h->pass_hi = value;
            return BB_OK;
        case BB_PARAM_STALL_SWEEP:
            if (value < -1 || value >= h->n) return fail(BB_ERR_INVALID_ARG, "stall sweep out of range");
            h->stall_sweep = (int)value;
            return BB_OK;
        case BB_PARAM_TIMING:
            h->timing = value ? 1 : 0;
            return BB_OK;
        case BB_PARAM_GROUP_SIZE:
            if (value < 0 || value > 32) return fail(BB_ERR_INVALID_ARG, "group size must be in [0, 32]");
            h->group_size = (int)value;
            return BB_OK;
        case BB_PARAM_RECORD:
            h->record = value ? 1 : 0;
            return BB_OK;
        default:
            return fail(BB_ERR_INVALID_ARG, "unknown parameter");
    }
}

int64_t bb_get_param(const bb_handle* h, int param) {
    if (!h) return -1;
    switch (param) {
        case BB_PARAM_SCHEDULER: return h->scheduler;
        case BB_PARAM_TPB: return h->tpb;
        case BB_PARAM_MAX_CTAS: return h->max_ctas;
        case BB_PARAM_WAIT_BUDGET_MS: return h->wait_ms;
        case BB_PARAM_PASS_LO: return h->pass_lo;
        case BB_PARAM_PASS_HI: return h->pass_hi;
        case BB_PARAM_STALL_SWEEP: return h->stall_sweep;
        case BB_PARAM_TIMING: return h->timing;
        case BB_PARAM_GROUP_SIZE: return h->group_size;
        case BB_PARAM_RECORD: return h->record;
        default: return -1;
    }
}

int64_t bb_last_launches(const bb_handle* h) { return h ? h->last_launches : -1; }

int64_t bb_last_pass_kernel(const bb_handle* h, int64_t i) {
    if (!h || i < 0 || i >= (int64_t)h->pass_kernel.size()) return -1;
    return h->pass_kernel[i];
}
int64_t bb_last_pass_group(const bb_handle* h, int64_t i) {
    if (!h || i < 0 || i >= (int64_t)h->pass_group.size()) return -1;
    return h->pass_group[i];
}
int64_t bb_last_num_passes(const bb_handle* h) { return h ? h->last_passes : -1; }

bb_status bb_last_pass_ms(bb_handle* h, int64_t i, double* ms) {
    if (!h || !ms) return fail(BB_ERR_INVALID_ARG, "bb_last_pass_ms: null argument");
    if (!h->timing || i < 0 || i >= h->last_passes || (size_t)(2 * i + 1) >= h->ev.size())
        return fail(BB_ERR_INVALID_ARG, "bb_last_pass_ms: no timing for this pass");
    float f = 0;
    cudaError_t e = cudaEventElapsedTime(&f, h->ev[2 * i], h->ev[2 * i + 1]);
    if (e != cudaSuccess) return cuda_fail(e, "bb_last_pass_ms");
    *ms = f;
    return BB_OK;
}

bb_status bb_status_sync(bb_handle* h, bb_stream_t stream) {
    if (!h) return fail(BB_ERR_INVALID_ARG, "bb_status_sync: null handle");
    cudaStream_t s = (cudaStream_t)stream;
    int st = 0;
    cudaError_t e = cudaMemcpyAsync(&st, h->d_status, sizeof(int), cudaMemcpyDeviceToHost, s);
    if (e == cudaSuccess) e = cudaStreamSynchronize(s);
    if (e != cudaSuccess) return cuda_fail(e, "bb_status_sync");
    if (st != 0) {
        e = cudaMemsetAsync(h->d_status, 0, sizeof(int), s);
        if (e == cudaSuccess) e = cudaStreamSynchronize(s);
        if (e != cudaSuccess) return cuda_fail(e, "bb_status_sync: clearing status");
        return fail((bb_status)st, st == BB_ERR_TIMEOUT ? "device-side progress wait timed out"
                                   : st == BB_ERR_INTERNAL ? "device-side consistency check failed"
                                                           : "device reported an error");
    }
    return BB_OK;
}

}  // extern "C"

static bb_status check_reduce_args(bb_handle* h, int64_t ldab, int64_t tw) {
    if (!h) return fail(BB_ERR_INVALID_ARG, "null handle");
    const int64_t tw_max = std::max<int64_t>(1, h->bw - 1);
    if (tw < 1 || tw > tw_max) return fail(BB_ERR_INVALID_ARG, "need 1 <= tw <= max(1, bw - 1)");
    if (tw + 1 > bb::kMaxW) return fail(BB_ERR_INVALID_ARG, "tw > 64 is not supported");
    if (ldab < bb_required_ldab(h->bw, tw)) return fail(BB_ERR_LDAB, "ldab < bw + 2*tw + 1");
    if ((double)ldab * (double)h->n > 9.0e18 / 8) return fail(BB_ERR_INVALID_ARG, "band too large");
    // shared memory of the widest pass (the first): tile of (b + t + 1)
    // columns; later passes have a smaller b and no larger t (the binary16
    // path keeps no tile)
    if (h->dtype != BB_F16 && count_passes(h->bw, tw) > 0 &&
        flag_tile_bytes(h->bw, std::min<int64_t>(tw, h->bw - 1), elem_size(h->dtype)) > 227 * 1024)
        return fail(BB_ERR_INVALID_ARG, "bandwidth too large for the shared-memory tile");
    return BB_OK;
}

// Scheduler 4: the per-cycle launches of pass pi, captured into a CUDA graph
// the first time (and again whenever the band, ldab or the pass changes),
// then replayed on stream s with one graph launch.  Capture runs on a stream
// of the handle, since the caller's stream may be the legacy default stream.
template <typename T>
static cudaError_t run_pass_graph(bb_handle* h, int64_t pi, T* band, int64_t ldab, const bb::PassArgs& P,
                                  const bb::LaunchCfg& cfg, cudaStream_t s, bb::LaunchStats* st) {
    cudaError_t err;
    if ((int64_t)h->graphs.size() <= pi) h->graphs.resize((size_t)pi + 1);
    bb_handle::PassGraph& pg = h->graphs[(size_t)pi];
    const bool hit = pg.exec && pg.band == band && pg.ldab == ldab && pg.n == P.n && pg.b == P.b &&
                     pg.t == P.t && pg.tpb == cfg.tpb;
    if (!hit) {
        if (pg.exec) {
            cudaGraphExecDestroy(pg.exec);
            pg.exec = nullptr;
        }
        if (!h->capture_stream) {
            err = cudaStreamCreateWithFlags(&h->capture_stream, cudaStreamNonBlocking);
            if (err != cudaSuccess) return err;
        }
        bb::LaunchStats cs;
        err = cudaStreamBeginCapture(h->capture_stream, cudaStreamCaptureModeRelaxed);
        if (err != cudaSuccess) return err;
        cudaError_t lerr = bb::run_pass<T>(band, P, 1, cfg, h->d_progress, h->d_status, h->capture_stream, &cs);
        cudaGraph_t graph = nullptr;
        err = cudaStreamEndCapture(h->capture_stream, &graph);
        if (lerr != cudaSuccess || err != cudaSuccess) {
            if (graph) cudaGraphDestroy(graph);
            return lerr != cudaSuccess ? lerr : err;
        }
        err = cudaGraphInstantiate(&pg.exec, graph, 0);
        cudaGraphDestroy(graph);
        if (err != cudaSuccess) {
            pg.exec = nullptr;
            return err;
        }
        pg.band = band;
        pg.ldab = ldab;
        pg.n = P.n;
        pg.b = P.b;
        pg.t = P.t;
        pg.tpb = cfg.tpb;
        pg.launches = cs.launches;
    }
    err = cudaGraphLaunch(pg.exec, s);
    if (st) {
        st->launches += pg.launches;  // kernels the graph runs
        st->kernel = 4;
    }
    return err;
}

template <typename T>
static bb_status reduce_impl(bb_handle* h, T* band, int64_t ldab, int64_t tw, T* d, T* e,
                             cudaStream_t s) {
    const int64_t n = h->n;
    const int ku = (int)(h->bw + tw);
    cudaError_t err;
    h->last_launches = 0;
    h->last_passes = 0;
    h->pass_kernel.clear();
    h->pass_group.clear();
    auto plan = plan_passes(h->bw, tw);
    const int64_t lo = std::max<int64_t>(0, h->pass_lo);
    const int64_t hi = std::min<int64_t>((int64_t)plan.size(), h->pass_hi);
    // reflector record: whole reductions only, on the flag kernel
    h->rec_valid = false;
    const bool rec = h->record && lo == 0 && hi == (int64_t)plan.size();
    const int sched = rec ? 2 : h->scheduler;
    std::vector<long long> rec_base(plan.size(), 0);
    std::vector<size_t> rec_prefix_off(plan.size(), 0);
    if (rec) {
        h->rec_prefix_host.clear();
        long long total = 0;
        for (size_t pi = 0; pi < plan.size(); ++pi) {
            const int b = plan[pi].b, t = plan[pi].t;
            rec_base[pi] = 2 * total;
            rec_prefix_off[pi] = h->rec_prefix_host.size();
            long long acc = 0;
            for (int64_t r = 0; r < n; ++r) {
                h->rec_prefix_host.push_back(acc);
                acc += steps_of_sweep(n, b, t, r);
            }
            total += acc;
        }
        const size_t es = sizeof(T);
        const size_t vb = es * (size_t)(2 * total) * (size_t)(tw + 1), tb = es * (size_t)(2 * total);
        const size_t pb = sizeof(long long) * h->rec_prefix_host.size();
        auto grow = [&](void** ptr, size_t* have, size_t need) -> cudaError_t {
            if (*have >= need && *ptr) return cudaSuccess;
            if (*ptr) cudaFree(*ptr);
            *ptr = nullptr;
            *have = 0;
            cudaError_t e2 = cudaMalloc(ptr, std::max<size_t>(need, 16));
            if (e2 == cudaSuccess) *have = need;
            return e2;
        };
        err = grow(&h->rec_v, &h->rec_v_bytes, vb);
        if (err == cudaSuccess) err = grow(&h->rec_tau, &h->rec_tau_bytes, tb);
        if (err == cudaSuccess) err = grow((void**)&h->rec_prefix, &h->rec_prefix_bytes, pb);
        if (err != cudaSuccess) return fail(BB_ERR_NOMEM, "reflector record allocation failed");
        err = cudaMemcpyAsync(h->rec_prefix, h->rec_prefix_host.data(), pb, cudaMemcpyHostToDevice, s);
        if (err != cudaSuccess) return cuda_fail(err, "reflector record prefix copy");
    }
    auto pass_args = [&](int64_t pi, int64_t ld) {
        const int b = plan[pi].b, t = plan[pi].t;
        bb::PassArgs P;
        P.n = n;
        P.ldab = ld;
        P.b = b;
        P.t = t;
        P.bp = b - t;
        P.ku = ku;
        P.nsweeps = (int)std::max<int64_t>(0, n - (b - t) - 1);
        P.lag = bb::pass_lag_cycle(b, t);
        P.lagh = bb::pass_lag_half(b, t);
        P.stall_sweep = h->stall_sweep;
        P.wait_budget = (unsigned long long)h->wait_ms * (unsigned long long)h->clock_khz;
        if (rec) {
            P.rec_v = h->rec_v;
            P.rec_tau = h->rec_tau;
            P.rec_prefix = h->rec_prefix + rec_prefix_off[pi];
            P.rec_base = rec_base[pi];
            P.rec_stride = (int)tw + 1;
        }
        return P;
    };
    // The group kernel moves whole columns with bulk copies, which need a
    // 16-byte aligned column stride: on any other layout the reduction runs
    // on an aligned working copy (one strided copy in, one out).
    T* wb = band;
    int64_t ldw = ldab;
    bool any_group = false;
    for (int64_t pi = lo; pi < hi; ++pi)
        any_group = any_group || bb::choose_group(pass_args(pi, ldab), sched, h->group_size, sizeof(T), nullptr);
    if (any_group && !bb::group_layout_ok(band, ldab, sizeof(T))) {
        const int64_t q = 16 / (int64_t)sizeof(T);
        ldw = (ldab + q - 1) / q * q;
        const size_t bytes = sizeof(T) * (size_t)ldw * (size_t)n;
        if (h->work_bytes < bytes) {
            if (h->work) cudaFree(h->work);
            h->work = nullptr;
            h->work_bytes = 0;
            err = cudaMalloc(&h->work, bytes);
            if (err != cudaSuccess) return fail(BB_ERR_NOMEM, "working band allocation failed");
            h->work_bytes = bytes;
        }
        wb = (T*)h->work;
        err = cudaMemcpy2DAsync(wb, sizeof(T) * ldw, band, sizeof(T) * ldab, sizeof(T) * ldab, (size_t)n,
                                cudaMemcpyDeviceToDevice, s);
        if (err != cudaSuccess) return cuda_fail(err, "copy to the working band");
    }
    if (lo == 0) {
        err = bb::run_zero_fill<T>(wb, n, ldw, (int)tw, ku, s);
        if (err != cudaSuccess) return cuda_fail(err, "zero fill launch");
        h->last_launches += 1;
    }
    if (h->timing) {
        size_t need = 2 * (size_t)std::max<int64_t>(0, hi - lo);
        while (h->ev.size() < need) {
            cudaEvent_t ev;
            err = cudaEventCreate(&ev);
            if (err != cudaSuccess) return cuda_fail(err, "cudaEventCreate");
            h->ev.push_back(ev);
        }
    }
    for (int64_t pi = lo; pi < hi; ++pi) {
        const bb::PassArgs P = pass_args(pi, ldw);
        bb::LaunchCfg cfg;
        cfg.tpb = h->tpb ? h->tpb : bb::auto_tpb(P.b, P.t);
        cfg.max_ctas = h->max_ctas;
        cfg.num_sms = h->num_sms;
        cfg.group_size = h->group_size;
        bb::LaunchStats st;
        if (h->timing) cudaEventRecord(h->ev[2 * (pi - lo)], s);
        if (sched == 4) {
            err = run_pass_graph<T>(h, pi, wb, ldw, P, cfg, s, &st);
        } else {
            err = bb::run_pass<T>(wb, P, sched, cfg, h->d_progress, h->d_status, s, &st);
        }
        if (h->timing) cudaEventRecord(h->ev[2 * (pi - lo) + 1], s);
        h->last_launches += st.launches;
        if (err != cudaSuccess) return cuda_fail(err, "pass launch");
        h->last_passes += 1;
        h->pass_kernel.push_back(st.kernel);
        h->pass_group.push_back(st.group);
    }
    err = bb::run_extract<T>(wb, n, ldw, ku, d, e, s);
    if (err != cudaSuccess) return cuda_fail(err, "extract launch");
    h->last_launches += 1;
    if (wb != band) {
        err = cudaMemcpy2DAsync(band, sizeof(T) * ldab, wb, sizeof(T) * ldw, sizeof(T) * ldab, (size_t)n,
                                cudaMemcpyDeviceToDevice, s);
        if (err != cudaSuccess) return cuda_fail(err, "copy back from the working band");
    }
    if (rec) {
        h->rec_valid = true;
        h->rec_tw = tw;
    }
    return BB_OK;
}

// Binary16 storage (float arithmetic), per pass the group kernel with
// binary16 columns (where the scheduler rule of bb_reduce picks it) or the
// binary16 flag kernel (bb_half.cu).  The pass range, timing, grid cap, wait
// budget, group size and fault injection apply.
static bb_status half_reduce(bb_handle* h, void* band, int64_t ldab, int64_t tw, void* d, void* e,
                             cudaStream_t s) {
    const int64_t n = h->n;
    const int ku = (int)(h->bw + tw);
    cudaError_t err;
    h->last_launches = 0;
    h->last_passes = 0;
    h->pass_kernel.clear();
    h->pass_group.clear();
    h->rec_valid = false;
    const int64_t np = count_passes(h->bw, tw);
    const int64_t lo = std::max<int64_t>(0, h->pass_lo);
    const int64_t hi = std::min<int64_t>(np, h->pass_hi);
    const int sched = h->scheduler;
    auto pass_args = [&](int64_t pi, int64_t ld) {
        const PassPlan ps = pass_at(h->bw, tw, pi);
        bb::PassArgs P;
        P.n = n;
        P.ldab = ld;
        P.b = ps.b;
        P.t = ps.t;
        P.bp = ps.b - ps.t;
        P.ku = ku;
        P.nsweeps = (int)std::max<int64_t>(0, n - P.bp - 1);
        P.lag = bb::pass_lag_cycle(P.b, P.t);
        P.lagh = bb::pass_lag_half(P.b, P.t);
        P.stall_sweep = h->stall_sweep;
        P.wait_budget = (unsigned long long)h->wait_ms * (unsigned long long)h->clock_khz;
        return P;
    };
    // The group kernel moves whole columns with bulk copies, which need a
    // 16-byte aligned column stride: on any other layout the reduction runs
    // on an aligned working copy (one strided copy in, one out).
    void* wb = band;
    int64_t ldw = ldab;
    bool any_group = false;
    for (int64_t pi = lo; pi < hi; ++pi)
        any_group = any_group || bb::half_choose_group(pass_args(pi, ldab), sched, h->group_size, nullptr);
    const size_t elem = 2;
    if (any_group && !bb::group_layout_ok(band, ldab, elem)) {
        const int64_t q = 16 / (int64_t)elem;
        ldw = (ldab + q - 1) / q * q;
        const size_t bytes = elem * (size_t)ldw * (size_t)n;
        if (h->work_bytes < bytes) {
            if (h->work) cudaFree(h->work);
            h->work = nullptr;
            h->work_bytes = 0;
            err = cudaMalloc(&h->work, bytes);
            if (err != cudaSuccess) return fail(BB_ERR_NOMEM, "working band allocation failed");
            h->work_bytes = bytes;
        }
        wb = h->work;
        err = cudaMemcpy2DAsync(wb, elem * ldw, band, elem * ldab, elem * ldab, (size_t)n, cudaMemcpyDeviceToDevice,
                                s);
        if (err != cudaSuccess) return cuda_fail(err, "copy to the working band");
    }
    if (lo == 0) {
        err = bb::run_half_zero_fill(wb, n, ldw, (int)tw, ku, h->num_sms, s);
        if (err != cudaSuccess) return cuda_fail(err, "zero fill launch");
        h->last_launches += 1;
    }
    if (h->timing) {
        const size_t need = 2 * (size_t)std::max<int64_t>(0, hi - lo);
        while (h->ev.size() < need) {
            cudaEvent_t ev;
            err = cudaEventCreate(&ev);
            if (err != cudaSuccess) return cuda_fail(err, "cudaEventCreate");
            h->ev.push_back(ev);
        }
    }
    bb::HalfLaunch L;
    L.num_sms = h->num_sms;
    L.max_ctas = h->max_ctas;
    L.scheduler = sched;
    L.group_size = h->group_size;
    L.progress = h->d_progress;
    L.status = h->d_status;
    for (int64_t pi = lo; pi < hi; ++pi) {
        const bb::PassArgs P = pass_args(pi, ldw);
        bb::GroupArgs ga{};
        const bool grp = bb::group_layout_ok(wb, ldw, elem) && bb::half_choose_group(P, sched, h->group_size, &ga);
        if (h->timing) cudaEventRecord(h->ev[2 * (pi - lo)], s);
        err = bb::run_half_pass(wb, P, L, grp ? &ga : nullptr, s);
        if (h->timing) cudaEventRecord(h->ev[2 * (pi - lo) + 1], s);
        if (err != cudaSuccess) return cuda_fail(err, "pass launch");
        h->last_launches += (P.nsweeps > 0) ? 1 : 0;
        h->last_passes += 1;
        h->pass_kernel.push_back(grp ? 3 : 5);
        h->pass_group.push_back(grp ? ga.g : 0);
    }
    err = bb::run_half_extract(wb, n, ldw, ku, d, e, h->num_sms, s);
    if (err != cudaSuccess) return cuda_fail(err, "extract launch");
    h->last_launches += 1;
    if (wb != band) {
        err = cudaMemcpy2DAsync(band, elem * ldab, wb, elem * ldw, elem * ldab, (size_t)n, cudaMemcpyDeviceToDevice,
                                s);
        if (err != cudaSuccess) return cuda_fail(err, "copy back from the working band");
    }
    return BB_OK;
}

extern "C" {

static bb_status reduce_checked(bb_handle* h, void* band_ptr, int64_t ldab, int64_t tw, void* d_out,
                                void* e_out, bb_stream_t stream) {
    bb_status st = check_reduce_args(h, ldab, tw);
    if (st != BB_OK) return st;
    if (!band_ptr || !d_out || (h->n > 1 && !e_out))
        return fail(BB_ERR_INVALID_ARG, "null band, d or e pointer");
    if (!is_device_pointer(band_ptr) || !is_device_pointer(d_out) ||
        (h->n > 1 && !is_device_pointer(e_out)))
        return fail(BB_ERR_INVALID_ARG, "band, d and e must be device pointers");
    cudaStream_t s = (cudaStream_t)stream;
    if (h->dtype == BB_F16) return half_reduce(h, band_ptr, ldab, tw, d_out, e_out, s);
    if (h->dtype == BB_F32)
        return reduce_impl<float>(h, (float*)band_ptr, ldab, tw, (float*)d_out, (float*)e_out, s);
    return reduce_impl<double>(h, (double*)band_ptr, ldab, tw, (double*)d_out, (double*)e_out, s);
}

// No C++ exception crosses the C ABI: host allocation failures (the handle's
// per-pass bookkeeping) come back as BB_ERR_NOMEM.
bb_status bb_reduce(bb_handle* h, void* band_ptr, int64_t ldab, int64_t tw, void* d_out,
                    void* e_out, bb_stream_t stream) {
    try {
        return reduce_checked(h, band_ptr, ldab, tw, d_out, e_out, stream);
    } catch (const std::bad_alloc&) {
        return fail(BB_ERR_NOMEM, "bb_reduce: host allocation failed");
    } catch (...) {
        return fail(BB_ERR_INTERNAL, "bb_reduce: unexpected host exception");
    }
}

int64_t bb_sym_required_ldab(int64_t bw, int64_t tw) { return bw + tw + 1; }

static bb_status sym_checked(bb_handle* h, void* band_ptr, int64_t ldab, int64_t tw, void* d_out, void* e_out,
                             bb_stream_t stream) {
    if (!h) return fail(BB_ERR_INVALID_ARG, "null handle");
    if (h->dtype == BB_F16) return fail(BB_ERR_DTYPE, "bb_sym_reduce: binary16 storage is not supported");
    const int64_t tw_max = std::max<int64_t>(1, h->bw - 1);
    if (tw < 1 || tw > tw_max) return fail(BB_ERR_INVALID_ARG, "need 1 <= tw <= max(1, bw - 1)");
    if (tw > 64) return fail(BB_ERR_INVALID_ARG, "tw > 64 is not supported");
    if (ldab < bb_sym_required_ldab(h->bw, tw)) return fail(BB_ERR_LDAB, "ldab < bw + tw + 1");
    if ((double)ldab * (double)h->n > 9.0e18 / 8) return fail(BB_ERR_INVALID_ARG, "band too large");
    if (!band_ptr || !d_out || (h->n > 1 && !e_out)) return fail(BB_ERR_INVALID_ARG, "null band, d or e pointer");
    if (!is_device_pointer(band_ptr) || !is_device_pointer(d_out) || (h->n > 1 && !is_device_pointer(e_out)))
        return fail(BB_ERR_INVALID_ARG, "band, d and e must be device pointers");
    bb::SymLaunch L;
    L.num_sms = h->num_sms;
    L.max_ctas = h->max_ctas;
    L.stall_sweep = h->stall_sweep;
    L.wait_budget = (unsigned long long)h->wait_ms * (unsigned long long)h->clock_khz;
    L.progress = h->d_progress;
    L.status = h->d_status;
    L.scheduler = h->scheduler;
    L.group_size = h->group_size;
    long long nl = 0;
    bb::SymPassStats st;
    cudaError_t err;
    const size_t elem = (h->dtype == BB_F32) ? 4 : 8;
    const cudaStream_t s = (cudaStream_t)stream;
    // The group kernel moves whole columns with bulk copies, which need a
    // 16-byte aligned column stride: on any other layout the reduction runs
    // on an aligned working copy (one strided copy in, one out).
    void* wb = band_ptr;
    int64_t ldw = ldab;
    if (bb::sym_any_group(h->n, (int)h->bw, (int)tw, L, elem) && !bb::group_layout_ok(band_ptr, ldab, elem)) {
        const int64_t q = 16 / (int64_t)elem;
        ldw = (ldab + q - 1) / q * q;
        const size_t bytes = elem * (size_t)ldw * (size_t)h->n;
        if (h->work_bytes < bytes) {
            if (h->work) cudaFree(h->work);
            h->work = nullptr;
            h->work_bytes = 0;
            err = cudaMalloc(&h->work, bytes);
            if (err != cudaSuccess) return fail(BB_ERR_NOMEM, "working band allocation failed");
            h->work_bytes = bytes;
        }
        wb = h->work;
        err = cudaMemcpy2DAsync(wb, elem * ldw, band_ptr, elem * ldab, elem * ldab, (size_t)h->n,
                                cudaMemcpyDeviceToDevice, s);
        if (err != cudaSuccess) return cuda_fail(err, "copy to the working band");
    }
    if (h->dtype == BB_F32)
        err = bb::run_sym<float>((float*)wb, h->n, ldw, (int)h->bw, (int)tw, (float*)d_out, (float*)e_out, L, s,
                                 &nl, &st);
    else
        err = bb::run_sym<double>((double*)wb, h->n, ldw, (int)h->bw, (int)tw, (double*)d_out, (double*)e_out, L,
                                  s, &nl, &st);
    if (err == cudaSuccess && wb != band_ptr)
        err = cudaMemcpy2DAsync(band_ptr, elem * ldab, wb, elem * ldw, elem * ldab, (size_t)h->n,
                                cudaMemcpyDeviceToDevice, s);
    h->last_launches = nl;
    h->last_passes = (int64_t)st.kernel.size();
    h->pass_kernel = st.kernel;
    h->pass_group = st.group;
    if (err != cudaSuccess) return cuda_fail(err, "bb_sym_reduce launch");
    return BB_OK;
}

bb_status bb_sym_reduce(bb_handle* h, void* band_ptr, int64_t ldab, int64_t tw, void* d_out, void* e_out,
                        bb_stream_t stream) {
    try {
        return sym_checked(h, band_ptr, ldab, tw, d_out, e_out, stream);
    } catch (const std::bad_alloc&) {
        return fail(BB_ERR_NOMEM, "bb_sym_reduce: host allocation failed");
    } catch (...) {
        return fail(BB_ERR_INTERNAL, "bb_sym_reduce: unexpected host exception");
    }
}

bb_status bb_back_transform(bb_handle* h, void* U, int64_t ldu, void* V, int64_t ldv, bb_stream_t stream) {
    if (!h) return fail(BB_ERR_INVALID_ARG, "null handle");
    if (!h->rec_valid)
        return fail(BB_ERR_INVALID_ARG, "bb_back_transform: no recorded reduction (set BB_PARAM_RECORD first)");
    if ((U && ldu < h->n) || (V && ldv < h->n)) return fail(BB_ERR_INVALID_ARG, "ldu and ldv must be >= n");
    if ((U && !is_device_pointer(U)) || (V && !is_device_pointer(V)))
        return fail(BB_ERR_INVALID_ARG, "U and V must be device pointers");
    long long nl = 0;
    cudaError_t err;
    const int stride = (int)h->rec_tw + 1;
    if (h->dtype == BB_F32)
        err = bb::run_back_transform<float>(h->n, (int)h->bw, (int)h->rec_tw, (const float*)h->rec_v,
                                            (const float*)h->rec_tau, stride, (float*)U, ldu, (float*)V, ldv,
                                            h->num_sms, (cudaStream_t)stream, &nl);
    else
        err = bb::run_back_transform<double>(h->n, (int)h->bw, (int)h->rec_tw, (const double*)h->rec_v,
                                             (const double*)h->rec_tau, stride, (double*)U, ldu, (double*)V, ldv,
                                             h->num_sms, (cudaStream_t)stream, &nl);
    h->last_launches = nl;
    if (err != cudaSuccess) return cuda_fail(err, "bb_back_transform launch");
    return BB_OK;
}

bb_status bb_reduce_host(bb_handle* h, const void* band_host, int64_t ldab, int64_t tw,
                         void* d_host, void* e_host, bb_stream_t stream) {
    bb_status st = check_reduce_args(h, ldab, tw);
    if (st != BB_OK) return st;
    if (!band_host || !d_host || (h->n > 1 && !e_host))
        return fail(BB_ERR_INVALID_ARG, "null band, d or e pointer");
    const size_t es = elem_size(h->dtype);
    const size_t band_bytes = es * (size_t)ldab * (size_t)h->n;
    cudaError_t err;
    if (h->s_band_bytes < band_bytes) {
        if (h->s_band) cudaFree(h->s_band);
        h->s_band = nullptr;
        h->s_band_bytes = 0;
        err = cudaMalloc(&h->s_band, band_bytes);
        if (err != cudaSuccess) return fail(BB_ERR_NOMEM, "staging band allocation failed");
        h->s_band_bytes = band_bytes;
    }
    if (!h->s_de) {
        err = cudaMalloc(&h->s_de, es * (size_t)(2 * h->n));
        if (err != cudaSuccess) return fail(BB_ERR_NOMEM, "staging d/e allocation failed");
    }
    cudaStream_t s = (cudaStream_t)stream;
    err = cudaMemcpyAsync(h->s_band, band_host, band_bytes, cudaMemcpyHostToDevice, s);
    if (err != cudaSuccess) return cuda_fail(err, "band copy to device");
    char* dd = (char*)h->s_de;
    char* ee = dd + es * (size_t)h->n;
    st = bb_reduce(h, h->s_band, ldab, tw, dd, ee, stream);
    if (st != BB_OK) return st;
    err = cudaMemcpyAsync(d_host, dd, es * (size_t)h->n, cudaMemcpyDeviceToHost, s);
    if (err == cudaSuccess && h->n > 1)
        err = cudaMemcpyAsync(e_host, ee, es * (size_t)(h->n - 1), cudaMemcpyDeviceToHost, s);
    if (err != cudaSuccess) return cuda_fail(err, "d/e copy to host");
    return bb_status_sync(h, stream);
}

}  // extern "C"

namespace bb {
void set_last_error(const char* msg) { g_last_error = msg ? msg : ""; }
}  // namespace bb
