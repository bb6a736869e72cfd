// Internal declarations and device helpers shared by the libcgdr kernels.
#pragma once

#include <atomic>

#include <cuda_runtime.h>
#include <cudaTypedefs.h>
#include <cuda_bf16.h>
#include <stdint.h>

#include "cgdr.h"

namespace cgdr {

// ---------------------------------------------------------------- host side
constexpr int kMaxDevices = 64;
// The calling thread's current device, or -1 (also for an index past kMaxDevices).
int current_device();
// SM count of the current device, queried once per device; 0 if unknown.
int device_sms();
// Per-kernel record of the devices whose dynamic shared-memory limit has been raised.
struct SmemOnce {
    std::atomic<uint64_t> mask{0};
};
// Raises `fn`'s dynamic shared-memory limit to `bytes` once per device; false on failure.
bool smem_limit_once(SmemOnce &once, const void *fn, int bytes);
// Polls of a bounded device wait on a kernel's own data (args.wait_polls, 0 = default; a
// negative value also asks for the injected first wait, see inject_of).
constexpr uint32_t kDefaultPolls = 1u << 20;
inline uint32_t polls_of(const cgdr_args &a) {
    return a.wait_polls > 0 ? (uint32_t)a.wait_polls : (a.wait_polls < 0 ? (uint32_t)(-(int64_t)a.wait_polls) : kDefaultPolls);
}
// Test hook: the first main-loop wait of every block waits on a barrier nothing completes.
inline int inject_of(const cgdr_args &a) { return a.wait_polls < 0 ? 1 : 0; }

// Element counts of each tensor's footprint ((B-1) sb + (T-1) st + (H-1) sh + d for a strided
// [B,T,H,d] view; 0 for an absent tensor) and the workspace bytes.  Kernels built with
// CGDR_DEBUG_CHECKS test every global access against them.
struct Extents {
    int64_t q, k, v, g, beta, a, b, o, state, A_log, dt_bias, ws;
};
Extents extents_of(const cgdr_args &a, bool prefill, size_t ws_bytes);

cgdr_status launch_decode(const cgdr_args &a, cudaStream_t s);
// Prefill with 1 <= T <= kRecurrentMaxT: the decode kernel stepping through the tokens.
constexpr int kRecurrentMaxT = 8;
cgdr_status launch_recurrent(const cgdr_args &a, cudaStream_t s);
cgdr_status launch_prefill_simt(const cgdr_args &a, cudaStream_t s);
bool prefill_tc05_supported(const cgdr_args &a);
size_t prefill_tc05_workspace(const cgdr_args &a);
cgdr_status launch_prefill_tc05(const cgdr_args &a, void *ws, size_t ws_bytes, cudaStream_t s);
int prefill_cluster_capacity();
size_t prefill_cluster_workspace(const cgdr_args &a);
int prefill_coop_grid();
size_t prefill_coop_workspace(const cgdr_args &a);
cgdr_status launch_prefill_coop(const cgdr_args &a, void *ws, size_t ws_bytes, cudaStream_t s);
// The prefill kernel for `a` given a.prefill_path (CGDR_PREFILL_PER_HEAD, _CLUSTER, _COOP, _SIMT
// or _RECURRENT); allow_cluster = false maps the kernels with a hand-off ring (cluster,
// cooperative) to the per-head one.
int prefill_path(const cgdr_args &a, bool allow_cluster);
size_t prefill_workspace_for(const cgdr_args &a, int path);
// Runs the kernel `path` (as prefill_path returned it) with the given workspace.
cgdr_status prefill_dispatch(const cgdr_args &a, int path, void *ws, size_t ws_bytes, cudaStream_t s);
cgdr_status launch_prefill_cluster(const cgdr_args &a, void *ws, size_t ws_bytes, cudaStream_t s);

// The driver's tiled tensor-map encoder, looked up once through the runtime (nullptr if
// the driver does not provide it).
PFN_cuTensorMapEncodeTiled_v12000 tensor_map_encoder();

inline float eps_of(const cgdr_args &a) { return a.eps < 0.f ? 1e-6f : a.eps; }
inline float qscale_of(const cgdr_args &a) {
    return a.q_scale > 0.f ? a.q_scale : 1.0f / sqrtf((float)a.dk);
}
inline int chunk_of(const cgdr_args &a) { return a.chunk == 0 ? 64 : a.chunk; }

// ---------------------------------------------------------------- device side
// Debug builds (CGDR_DEBUG_CHECKS): `off` must lie in [0, n); a failed check stores
// CGDR_ERR_BOUNDS in the given status words (either may be null) and the caller skips the
// access.  Release builds: always true, no code.
__device__ __forceinline__ bool in_bounds(int64_t off, int64_t n, int *st0, int *st1) {
#ifdef CGDR_DEBUG_CHECKS
    if (off >= 0 && off < n) return true;
    if (st0 != nullptr) atomicExch(st0, (int)CGDR_ERR_BOUNDS);
    if (st1 != nullptr) atomicExch(st1, (int)CGDR_ERR_BOUNDS);
    return false;
#else
    (void)off; (void)n; (void)st0; (void)st1;
    return true;
#endif
}
// Both ends of an access of `count` elements starting at `off`.
__device__ __forceinline__ bool range_in_bounds(int64_t off, int64_t count, int64_t n, int *st0, int *st1) {
    return in_bounds(off, n, st0, st1) && in_bounds(off + count - 1, n, st0, st1);
}

template <typename T> struct Cvt;
template <> struct Cvt<float> {
    static __device__ __forceinline__ float to_f(float x) { return x; }
    static __device__ __forceinline__ float from_f(float x) { return x; }
};
template <> struct Cvt<__nv_bfloat16> {
    static __device__ __forceinline__ float to_f(__nv_bfloat16 x) { return __bfloat162float(x); }
    static __device__ __forceinline__ __nv_bfloat16 from_f(float x) { return __float2bfloat16_rn(x); }
};

__device__ __forceinline__ float warp_sum(float x) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) x += __shfl_xor_sync(0xffffffffu, x, o);
    return x;
}

// softplus with the usual threshold: x above 20 is returned unchanged.
__device__ __forceinline__ float softplus_f(float x) { return x > 20.f ? x : log1pf(expf(x)); }
__device__ __forceinline__ float sigmoid_f(float x) { return 1.f / (1.f + expf(-x)); }

// Scalar GatedDeltaNet gate: g = -exp(A_log) * softplus(a + dt_bias).
__device__ __forceinline__ float gdn_gate(float A_log, float a, float dt_bias) {
    return -expf(A_log) * softplus_f(a + dt_bias);
}

__device__ __forceinline__ uint32_t smem_u32(const void *p) {
    return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

// Asynchronous global -> shared copies (16 or 4 bytes); a false `valid` zero-fills
// the destination without reading the source.
__device__ __forceinline__ void cp_async16(uint32_t dst, const void *src, bool valid) {
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;" ::"r"(dst), "l"(src), "r"(valid ? 16 : 0) : "memory");
}
__device__ __forceinline__ void cp_async4(uint32_t dst, const void *src, bool valid) {
    asm volatile("cp.async.ca.shared.global [%0], [%1], 4, %2;" ::"r"(dst), "l"(src), "r"(valid ? 4 : 0) : "memory");
}
// L2 eviction-priority policies (createpolicy) for cache-hinted copies: data read once
// (evict first) and data written now to be read back soon (evict last).
__device__ __forceinline__ uint64_t l2_evict_first() {
    uint64_t pol;
    asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(pol));
    return pol;
}
__device__ __forceinline__ uint64_t l2_evict_last() {
    uint64_t pol;
    asm volatile("createpolicy.fractional.L2::evict_last.b64 %0, 1.0;" : "=l"(pol));
    return pol;
}
// cp_async16 with an L2 policy for the source line.
__device__ __forceinline__ void cp_async16_hint(uint32_t dst, const void *src, bool valid, uint64_t pol) {
    asm volatile("cp.async.cg.shared.global.L2::cache_hint [%0], [%1], 16, %2, %3;" ::"r"(dst), "l"(src),
                 "r"(valid ? 16 : 0), "l"(pol) : "memory");
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }
__device__ __forceinline__ void cp_async_wait_all() { asm volatile("cp.async.wait_all;" ::: "memory"); }

__device__ __forceinline__ uint32_t pack_bf16x2(float lo, float hi) {
    __nv_bfloat162 v = __floats2bfloat162_rn(lo, hi);
    return *reinterpret_cast<uint32_t *>(&v);
}

// ldmatrix: four 8x8 b16 matrices; lane l supplies the row address of
// matrix l/8, row l%8.  Register j receives matrix j.
__device__ __forceinline__ void ldsm_x4(uint32_t &r0, uint32_t &r1, uint32_t &r2, uint32_t &r3,
                                        uint32_t addr) {
    asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0,%1,%2,%3}, [%4];\n"
                 : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3) : "r"(addr));
}
__device__ __forceinline__ void ldsm_x4_t(uint32_t &r0, uint32_t &r1, uint32_t &r2, uint32_t &r3,
                                          uint32_t addr) {
    asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0,%1,%2,%3}, [%4];\n"
                 : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3) : "r"(addr));
}

// D = A(16x16, row) * B(16x8, col) + D, bf16 inputs, fp32 accumulate.
__device__ __forceinline__ void mma_bf16(float (&d)[4], const uint32_t (&a)[4], uint32_t b0, uint32_t b1) {
    asm volatile(
        "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
        "{%0,%1,%2,%3};\n"
        : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
        : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}

}  // namespace cgdr
