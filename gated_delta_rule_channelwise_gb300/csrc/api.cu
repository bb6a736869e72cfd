// C ABI entry points of libcgdr: host-side argument checks and dispatch.
// The operation and the argument conventions are documented in cgdr.h.
#include <atomic>
#include <mutex>

#include "cgdr_internal.cuh"
#include "cgdr_debug.h"

namespace {

bool dim_ok(int d) { return d == 32 || d == 64 || d == 128; }

bool aligned(const void *p, size_t n) { return (reinterpret_cast<uintptr_t>(p) % n) == 0; }

bool strides_ok(int64_t s0, int64_t s1, int64_t s2, int64_t mult) {
    return s0 >= 0 && s1 >= 0 && s2 >= 0 && s0 % mult == 0 && s1 % mult == 0 && s2 % mult == 0;
}

cgdr_status check(const cgdr_args *a, bool prefill) {
    if (!a) return CGDR_ERR_INVALID_ARG;
    if (a->B < 0 || a->T < 0 || a->Hk <= 0 || a->Hv <= 0) return CGDR_ERR_INVALID_ARG;
    if (a->Hv % a->Hk != 0) return CGDR_ERR_INVALID_ARG;
    if (!prefill && a->T != 1) return CGDR_ERR_INVALID_ARG;
    if (!dim_ok(a->dk) || !dim_ok(a->dv)) return CGDR_ERR_UNSUPPORTED;
    if (a->dtype != CGDR_F32 && a->dtype != CGDR_BF16) return CGDR_ERR_UNSUPPORTED;
    if (a->o_dtype != CGDR_F32 && a->o_dtype != CGDR_BF16) return CGDR_ERR_UNSUPPORTED;
    if (a->gate != CGDR_GATE_CHANNEL && a->gate != CGDR_GATE_GDN) return CGDR_ERR_UNSUPPORTED;
    if (prefill && !(a->chunk == 0 || a->chunk == 16 || a->chunk == 32 || a->chunk == 64))
        return CGDR_ERR_UNSUPPORTED;
    if (prefill && (a->prefill_path < CGDR_PREFILL_AUTO || a->prefill_path > CGDR_PREFILL_COOP))
        return CGDR_ERR_INVALID_ARG;
    if (a->B == 0 || a->T == 0) return CGDR_OK;  // nothing to do: no pointer is touched
    if (!aligned(a->status, 4)) return CGDR_ERR_ALIGNMENT;

    if (!a->q || !a->k || !a->v || !a->state || !a->o) return CGDR_ERR_INVALID_ARG;
    if (a->gate == CGDR_GATE_CHANNEL && (!a->g || !a->beta)) return CGDR_ERR_INVALID_ARG;
    if (a->gate == CGDR_GATE_GDN && (!a->a || !a->b || !a->A_log || !a->dt_bias))
        return CGDR_ERR_INVALID_ARG;

    const size_t esz = a->dtype == CGDR_BF16 ? 2 : 4;
    const int64_t vec = (int64_t)(16 / esz);
    const int64_t ovec = a->o_dtype == CGDR_BF16 ? 8 : 4;
    // decode ignores the token strides
    const int64_t q_st = prefill ? a->q_st : 0, k_st = prefill ? a->k_st : 0;
    const int64_t v_st = prefill ? a->v_st : 0, o_st = prefill ? a->o_st : 0;
    const int64_t g_st = prefill ? a->g_st : 0, be_st = prefill ? a->beta_st : 0;
    const int64_t a_st = prefill ? a->a_st : 0, b_st = prefill ? a->b_st : 0;
    if (!aligned(a->q, 16) || !aligned(a->k, 16) || !aligned(a->v, 16) || !aligned(a->o, 16) ||
        !aligned(a->state, 16))
        return CGDR_ERR_ALIGNMENT;
    if (!strides_ok(a->q_sb, q_st, a->q_sh, vec) || !strides_ok(a->k_sb, k_st, a->k_sh, vec) ||
        !strides_ok(a->v_sb, v_st, a->v_sh, vec) || !strides_ok(a->o_sb, o_st, a->o_sh, ovec))
        return CGDR_ERR_ALIGNMENT;
    if (a->gate == CGDR_GATE_CHANNEL) {
        if (!aligned(a->g, 16) || !strides_ok(a->g_sb, g_st, a->g_sh, 4)) return CGDR_ERR_ALIGNMENT;
        if (!aligned(a->beta, 4) || !strides_ok(a->beta_sb, be_st, a->beta_sh, 1)) return CGDR_ERR_ALIGNMENT;
    } else {
        if (!aligned(a->a, esz) || !aligned(a->b, esz) || !aligned(a->A_log, 4) || !aligned(a->dt_bias, 4))
            return CGDR_ERR_ALIGNMENT;
        if (!strides_ok(a->a_sb, a_st, a->a_sh, 1) || !strides_ok(a->b_sb, b_st, a->b_sh, 1))
            return CGDR_ERR_ALIGNMENT;
    }
    return CGDR_OK;
}

}  // namespace

namespace cgdr {

PFN_cuTensorMapEncodeTiled_v12000 tensor_map_encoder() {
    static std::once_flag once;
    static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
    std::call_once(once, [] {
        void *f = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &f, 12000, cudaEnableDefault, &q) ==
                cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(f);
    });
    return fn;
}

namespace {
int64_t footprint(const void *p, int64_t B, int64_t T, int64_t H, int64_t d, int64_t sb, int64_t st, int64_t sh) {
    if (p == nullptr || B <= 0 || T <= 0 || H <= 0) return 0;
    return (B - 1) * sb + (T - 1) * st + (H - 1) * sh + d;
}
}  // namespace

// Debug builds: elements taken off o's footprint for the current thread's call (the test entry
// point of cgdr_debug.h sets it around one call; thread-local, so other threads are unaffected).
thread_local int64_t t_debug_o_shrink = 0;

Extents extents_of(const cgdr_args &a, bool prefill, size_t ws_bytes) {
    const int64_t T = prefill ? a.T : 1;
    Extents e;
    e.q = footprint(a.q, a.B, T, a.Hk, a.dk, a.q_sb, a.q_st, a.q_sh);
    e.k = footprint(a.k, a.B, T, a.Hk, a.dk, a.k_sb, a.k_st, a.k_sh);
    e.v = footprint(a.v, a.B, T, a.Hv, a.dv, a.v_sb, a.v_st, a.v_sh);
    e.o = footprint(a.o, a.B, T, a.Hv, a.dv, a.o_sb, a.o_st, a.o_sh);
    const bool chan = a.gate == CGDR_GATE_CHANNEL;
    e.g = chan ? footprint(a.g, a.B, T, a.Hv, a.dk, a.g_sb, a.g_st, a.g_sh) : 0;
    e.beta = chan ? footprint(a.beta, a.B, T, a.Hv, 1, a.beta_sb, a.beta_st, a.beta_sh) : 0;
    e.a = chan ? 0 : footprint(a.a, a.B, T, a.Hv, 1, a.a_sb, a.a_st, a.a_sh);
    e.b = chan ? 0 : footprint(a.b, a.B, T, a.Hv, 1, a.b_sb, a.b_st, a.b_sh);
    e.A_log = chan || a.A_log == nullptr ? 0 : a.Hv;
    e.dt_bias = chan || a.dt_bias == nullptr ? 0 : a.Hv;
    e.state = a.state == nullptr ? 0 : (int64_t)a.B * a.Hv * a.dk * a.dv;
    e.ws = (int64_t)ws_bytes;
    e.o -= t_debug_o_shrink;
    return e;
}

int current_device() {
    int dev = -1;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return -1;
    return dev;
}

int device_sms() {
    static std::atomic<int> cache[kMaxDevices];
    const int dev = current_device();
    if (dev < 0) return 0;
    int sms = cache[dev].load(std::memory_order_relaxed);
    if (sms == 0) {
        if (cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || sms <= 0) {
            cudaGetLastError();
            return 0;
        }
        cache[dev].store(sms, std::memory_order_relaxed);
    }
    return sms;
}

bool smem_limit_once(SmemOnce &once, const void *fn, int bytes) {
    const int dev = current_device();
    if (dev < 0) return false;
    const uint64_t bit = 1ull << dev;
    if (once.mask.load(std::memory_order_acquire) & bit) return true;
    // idempotent: two threads racing here both set the same attribute
    if (cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes) != cudaSuccess) return false;
    once.mask.fetch_or(bit, std::memory_order_acq_rel);
    return true;
}

int prefill_path(const cgdr_args &a, bool allow_cluster) {
    const int choice = a.prefill_path;
    const bool few = a.T >= 1 && a.T <= kRecurrentMaxT;
    if (few && (choice == CGDR_PREFILL_AUTO || choice == CGDR_PREFILL_RECURRENT)) return CGDR_PREFILL_RECURRENT;
    if (choice == CGDR_PREFILL_SIMT || !prefill_tc05_supported(a)) return CGDR_PREFILL_SIMT;
    int path = choice == CGDR_PREFILL_RECURRENT ? CGDR_PREFILL_AUTO : choice;
    const int64_t units = (int64_t)a.B * a.Hv;
    if (path == CGDR_PREFILL_COOP && prefill_coop_grid() <= units) path = CGDR_PREFILL_AUTO;
    if (path == CGDR_PREFILL_AUTO) {
        // Whichever needs the least time, from cycles per chunk of one head measured on GB300
        // (clock64 phase stamps, T = 4000): one CTA per head 23 K, resident one per SM; a
        // four-CTA cluster 6.3 K (its three preparers need 18.9 K per chunk each), 36 clusters
        // resident; the cooperative grid max(5.3 K for the state CTA, 18.9 K x heads /
        // preparers), all heads at once.
        const int cap = prefill_cluster_capacity();
        const int sms = device_sms();
        const int grid = prefill_coop_grid();
        int64_t best = sms > 0 ? (units + sms - 1) / sms * 230 : 0;                 // per head (x 100 cycles)
        path = CGDR_PREFILL_PER_HEAD;
        if (cap > 0 && (units + cap - 1) / cap * 63 < best) {
            best = (units + cap - 1) / cap * 63;
            path = CGDR_PREFILL_CLUSTER;
        }
        if (grid > units) {
            const int64_t prep = (189 * units + (grid - units) - 1) / (grid - units);
            const int64_t coop = prep > 53 ? prep : 53;
            if (coop < best) path = CGDR_PREFILL_COOP;
        }
    }
    if ((path == CGDR_PREFILL_CLUSTER || path == CGDR_PREFILL_COOP) && !allow_cluster) path = CGDR_PREFILL_PER_HEAD;
    return path;
}

size_t prefill_workspace_for(const cgdr_args &a, int path) {
    if (path == CGDR_PREFILL_CLUSTER) return prefill_cluster_workspace(a);
    if (path == CGDR_PREFILL_COOP) return prefill_coop_workspace(a);
    if (path == CGDR_PREFILL_PER_HEAD) return prefill_tc05_workspace(a);
    return 0;
}

cgdr_status prefill_dispatch(const cgdr_args &a, int path, void *ws, size_t ws_bytes, cudaStream_t s) {
    if (path == CGDR_PREFILL_RECURRENT) return launch_recurrent(a, s);
    if (path == CGDR_PREFILL_SIMT) return launch_prefill_simt(a, s);
    const size_t need = prefill_workspace_for(a, path);
    if (ws == nullptr || ws_bytes < need || (reinterpret_cast<uintptr_t>(ws) % 16) != 0) return CGDR_ERR_WORKSPACE;
    const cgdr_status st = path == CGDR_PREFILL_CLUSTER ? launch_prefill_cluster(a, ws, ws_bytes, s)
                           : path == CGDR_PREFILL_COOP  ? launch_prefill_coop(a, ws, ws_bytes, s)
                                                        : launch_prefill_tc05(a, ws, ws_bytes, s);
    // the driver's tensor-map encoder refused a tensor that the host check accepted: CUDA-core kernel
    return st == CGDR_ERR_ALIGNMENT ? launch_prefill_simt(a, s) : st;
}

}  // namespace cgdr

extern "C" {

int cgdr_abi_version(void) { return CGDR_ABI_VERSION; }

const char *cgdr_status_string(int s) {
    switch (s) {
        case CGDR_OK: return "CGDR_OK";
        case CGDR_ERR_INVALID_ARG: return "CGDR_ERR_INVALID_ARG: null pointer, bad size, Hv % Hk != 0 or T != 1 for decode";
        case CGDR_ERR_UNSUPPORTED: return "CGDR_ERR_UNSUPPORTED: dk/dv/chunk/dtype/gate outside the supported set";
        case CGDR_ERR_ALIGNMENT: return "CGDR_ERR_ALIGNMENT: misaligned pointer or stride";
        case CGDR_ERR_WORKSPACE: return "CGDR_ERR_WORKSPACE: workspace too small";
        case CGDR_ERR_CUDA: return "CGDR_ERR_CUDA: a CUDA call or kernel launch failed";
        case CGDR_ERR_TIMEOUT: return "CGDR_ERR_TIMEOUT: a bounded device wait gave up";
        case CGDR_ERR_BOUNDS: return "CGDR_ERR_BOUNDS: a debug build's device index check failed";
        case CGDR_ERR_RANGE: return "CGDR_ERR_RANGE: an fp16 tensor-core operand left the fp16 range";
        default: return "unknown cgdr status";
    }
}

cgdr_status cgdr_validate(const cgdr_args *a, int for_prefill) { return check(a, for_prefill != 0); }

cgdr_status cgdr_decode(const cgdr_args *a, void *stream) {
    cgdr_status st = check(a, false);
    if (st != CGDR_OK || a->B == 0) return st;
    return cgdr::launch_decode(*a, static_cast<cudaStream_t>(stream));
}

size_t cgdr_prefill_workspace_size(const cgdr_args *a) {
    if (check(a, true) != CGDR_OK || a->B == 0 || a->T == 0) return 0;
    return cgdr::prefill_workspace_for(*a, cgdr::prefill_path(*a, true));
}

int cgdr_prefill_path_for(const cgdr_args *a) {
    if (check(a, true) != CGDR_OK || a->B == 0 || a->T == 0) return CGDR_PREFILL_AUTO;
    return cgdr::prefill_path(*a, true);
}

cgdr_status cgdr_prefill(const cgdr_args *a, void *ws, size_t ws_bytes, void *stream) {
    cgdr_status st = check(a, true);
    if (st != CGDR_OK || a->B == 0 || a->T == 0) return st;
    return cgdr::prefill_dispatch(*a, cgdr::prefill_path(*a, true), ws, ws_bytes, static_cast<cudaStream_t>(stream));
}

cgdr_status cgdr_debug_decode_shrunk_o(const cgdr_args *a, int64_t o_shrink, void *stream) {
#ifdef CGDR_DEBUG_CHECKS
    cgdr::t_debug_o_shrink = o_shrink;
    const cgdr_status st = cgdr_decode(a, stream);
    cgdr::t_debug_o_shrink = 0;
    return st;
#else
    (void)a; (void)o_shrink; (void)stream;
    return CGDR_ERR_UNSUPPORTED;
#endif
}

cgdr_status cgdr_workspace_status(const void *ws, void *stream) {
    if (ws == nullptr) return CGDR_ERR_INVALID_ARG;
    int word = 0;
    if (cudaMemcpyAsync(&word, ws, sizeof(int), cudaMemcpyDeviceToHost, static_cast<cudaStream_t>(stream)) !=
            cudaSuccess ||
        cudaStreamSynchronize(static_cast<cudaStream_t>(stream)) != cudaSuccess)
        return CGDR_ERR_CUDA;
    return word == 0 ? CGDR_OK : static_cast<cgdr_status>(word);
}

}  // extern "C"
