// Chunked prefill on a four-CTA thread-block cluster per (batch, v-head),
// for launches with too few heads to fill the GPU one CTA per head.
//
// The chunkwise WY/UT form of "Add parallel chunked prefill for channelwise
// gated delta rule" (executorch PR #21061, Summary) splits into work that
// needs the state (the carry S <- e^gC S + Kend^T U with U = U~ - W S, and the
// output O = Qg S + P U) and work that does not (decay prefix, operand tiles,
// causal terms, the triangular transform Tb).  Only the first is serial along
// T.  So:
//   rank 0 (the chain)     keeps S^T in tensor memory and, per chunk, forms
//                          W = Tb Kg and U~ = Tb V, then the state-dependent
//                          contractions, and writes o;
//   ranks 1..3 (preparers) take chunks round robin (chunk c on rank
//                          1 + c % 3) and run the state-free phases.
// Hand-off through L2: a preparer sends the tiles it has built in shared
// memory -- Qg, Kg^T, V^T, Tb, e^gC (inbox A image) and Kend^T, P (inbox B
// image), fp16 tiles -- with bulk stores into one of its three slots of a ring in the
// workspace, each piece at its place in rank 0's shared-memory tile layout,
// and arrives on rank 0's ready barrier for that slot; rank 0 pulls each
// image into its inbox with one bulk load as soon as the inbox is free, and
// arrives on the preparer's slot-free barrier once both loads have landed.
// (Bulk copies through L2 move data about five times faster than copies
// between the CTAs' shared memories, and run beside the threads' work.)  One
// barrier per slot on each side keeps every barrier at most one phase ahead
// of its waiter.  Every wait is bounded; a wait that gives up records
// CGDR_ERR_TIMEOUT and every CTA leaves its loop, frees tensor memory and
// meets the others at the final cluster barrier.
#include <atomic>
#include <mutex>

#include "prefill_tc05_chunk.cuh"

namespace cgdr {
namespace {

using namespace tc05c;

constexpr int CLUSTER = 4, NPREP = CLUSTER - 1, NSLOTP = 3, NSLOT = NSLOTP * NPREP;   // NSLOTP slots per preparer

// one hand-off slot (bytes): the inbox A image, then the inbox B image
constexpr int SL_QG = 0;                         // Qg   [64 x 128] fp16 tile
constexpr int SL_KG = 16384;                     // Kg^T [128 x 64] fp16 tile
constexpr int SL_VT = 32768;                     // V^T  [128 x 64] fp16 tile
constexpr int SL_TB = 49152;                     // Tb   [64 x 64] fp16 tile
constexpr int SL_DEC = 57344;                    // e^gC [128] fp32
constexpr uint32_t A_BYTES = 57344 + 512;
constexpr int SL_KP = (int)A_BYTES;              // [Kend^T ; P] [192 x 64] fp16 tile (rows 0..127 Kend^T, 128..191 P)
constexpr uint32_t B_BYTES = 24576;
constexpr size_t SLOT_BYTES = A_BYTES + B_BYTES;
constexpr size_t WS_HEADER = 256;                // status word, then the slots
static_assert(SLOT_BYTES % 16 == 0 && SL_KP % 16 == 0, "bulk copies need 16-byte alignment");

// rank 0 shared memory map (bytes from the 1024-aligned base)
// Inbox A: Qg lands in rows 0..63 of the [Qg; -W] tile (one bulk load per 64-column block, so
// that S^T [Qg; -W]^T is a single N = 128 product), the rest of the image after that tile.
constexpr int CH_QW = 0;                         // [Qg ; -W] [128 x 128] fp16 tile (rows 64..127: -W, built here)
constexpr int CH_A_REST = 32768;                 // the image from SL_KG on
constexpr int CH_KG = CH_A_REST + SL_KG - SL_KG, CH_VT = CH_A_REST + SL_VT - SL_KG, CH_TB = CH_A_REST + SL_TB - SL_KG;
constexpr int CH_DEC = CH_A_REST + SL_DEC - SL_KG;
constexpr uint32_t A_REST_BYTES = A_BYTES - SL_KG;
constexpr int CH_UR = 74752;                     // U^T [128 x 64] fp16 tile
constexpr int CH_IN_B = CH_UR + 16384;           // inbox B: the slot's last B_BYTES
constexpr int CH_KP = CH_IN_B;
constexpr int CH_MISC = CH_IN_B + 24576;
constexpr int CH_MBAR = CH_MISC, CH_FULL_A = CH_MISC + 8, CH_FULL_B = CH_MISC + 16, CH_TMEM = CH_MISC + 24;
constexpr int CH_READY = CH_MISC + 32;           // NSLOT barriers, one per slot
constexpr int CH_OST = CH_MISC + 1024;           // o of one chunk [64 tokens][128] in o's dtype (TMA store source)
constexpr int CH_END = CH_OST + 32768;
static_assert(CH_READY + 8 * NSLOT <= CH_OST, "misc words overlap");
static_assert(SL_KG == 16384 && CH_A_REST + (int)A_REST_BYTES <= CH_UR, "inbox A overlaps");
static_assert(CH_QW % 1024 == 0 && CH_UR % 1024 == 0 && CH_IN_B % 1024 == 0 && CH_KG % 1024 == 0 &&
              CH_VT % 1024 == 0 && CH_TB % 1024 == 0, "tiles must be 1024-aligned");
constexpr int CL_SMEM_BYTES = (CH_END > M_END ? CH_END : M_END) + 1024;
static_assert(CL_SMEM_BYTES <= 232448, "shared memory over the per-block limit");
// rank 0 tensor memory columns: S^T, then O^T, then U^T, so that [O^T | U^T] and
// [S^T | O^T] are each one accumulator of a single MMA; W^T and the fp16 copy of S^T after them
constexpr uint32_t T_S = 0, T_O = 128, T_U = 192, T_W = 256, T_S16 = 320;

// ---------------------------------------------------------------- cluster and bulk-copy primitives
__device__ __forceinline__ uint32_t cluster_ctarank() {
    uint32_t r;
    asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
    return r;
}
// The shared::cluster address of the same offset in CTA `rank` of this cluster.
__device__ __forceinline__ uint32_t mapa_rank(uint32_t addr, uint32_t rank) {
    uint32_t r;
    asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(r) : "r"(addr), "r"(rank));
    return r;
}
__device__ __forceinline__ void cluster_barrier() {
    asm volatile("barrier.cluster.arrive.release.aligned;\nbarrier.cluster.wait.acquire.aligned;" ::: "memory");
}
// Non-blocking test, with cluster-scope acquire, of the phase with the given parity.
__device__ __forceinline__ bool cl_test(uint32_t mbar, uint32_t parity) {
    uint32_t done;
    asm volatile(
        "{\n.reg .pred p;\nmbarrier.test_wait.parity.acquire.cluster.shared::cta.b64 p, [%1], %2;\n"
        "selp.u32 %0, 1, 0, p;\n}\n"
        : "=r"(done) : "r"(mbar), "r"(parity) : "memory");
    return done != 0;
}
// Bounded wait (`polls` polls), with cluster-scope acquire, for the phase of a local barrier
// with the given parity.
__device__ __forceinline__ bool cl_wait(uint32_t mbar, uint32_t parity, uint32_t polls) {
    for (uint32_t it = 0; it < polls; ++it) {
        uint32_t done;
        asm volatile(
            "{\n.reg .pred p;\nmbarrier.try_wait.parity.acquire.cluster.shared::cta.b64 p, [%1], %2;\n"
            "selp.u32 %0, 1, 0, p;\n}\n"
            : "=r"(done) : "r"(mbar), "r"(parity) : "memory");
        if (done) return true;
    }
    return false;
}
__device__ __forceinline__ void arrive_expect_tx(uint32_t mbar, uint32_t bytes) {
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(mbar), "r"(bytes) : "memory");
}
__device__ __forceinline__ void remote_arrive(uint32_t mbar_cluster) {
    asm volatile("mbarrier.arrive.release.cluster.shared::cluster.b64 _, [%0];" ::"r"(mbar_cluster) : "memory");
}
// Arrive without release: for a signal that orders nothing of this thread's own memory
// operations (a release would first wait for its outstanding global stores).
__device__ __forceinline__ void remote_arrive_relaxed(uint32_t mbar_cluster) {
    asm volatile("mbarrier.arrive.relaxed.cluster.shared::cluster.b64 _, [%0];" ::"r"(mbar_cluster) : "memory");
}
// Order this thread's generic-proxy global accesses with later bulk copies (async proxy).
__device__ __forceinline__ void fence_global_to_async() { asm volatile("fence.proxy.async.global;" ::: "memory"); }
// Bulk copy of `bytes` from this CTA's shared memory to global memory; bulk_commit closes
// a group of them.  wait_read<N>: at most N most recent groups still reading shared memory;
// bulk_store_wait: every group's writes complete.
// The ring is read back within microseconds: keep its lines (evict last) against the
// streamed inputs.
__device__ __forceinline__ void bulk_store(void *dst, uint32_t src, uint32_t bytes) {
    asm volatile("cp.async.bulk.global.shared::cta.bulk_group.L2::cache_hint [%0], [%1], %2, %3;"
                 ::"l"(dst), "r"(src), "r"(bytes), "l"(l2_evict_last()) : "memory");
}
// bulk_store into the workspace, skipped (debug build) when it would leave the workspace
__device__ __forceinline__ void ring_store(const Tc05Params &p, char *dst, uint32_t src, uint32_t bytes) {
    const int64_t off = (int64_t)(dst - reinterpret_cast<const char *>(p.err));
    if (range_in_bounds(off, bytes, p.ext.ws, p.err, p.status)) bulk_store(dst, src, bytes);
}
__device__ __forceinline__ void bulk_commit() { asm volatile("cp.async.bulk.commit_group;" ::: "memory"); }
// TMA tensor store of the box at (0, token t0, head, batch) of map tm from this CTA's shared memory.
__device__ __forceinline__ void tma_store_tile(const CUtensorMap *tm, uint32_t src, int t0, int head, int b) {
    asm volatile("cp.async.bulk.tensor.4d.global.shared::cta.tile.bulk_group [%0, {%1, %2, %3, %4}], [%5];"
                 ::"l"(reinterpret_cast<uint64_t>(tm)), "r"(0), "r"(t0), "r"(head), "r"(b), "r"(src) : "memory");
}
template <int N>
__device__ __forceinline__ void bulk_wait_read() { asm volatile("cp.async.bulk.wait_group.read %0;" ::"n"(N) : "memory"); }
__device__ __forceinline__ void bulk_store_wait() { asm volatile("cp.async.bulk.wait_group 0;" ::: "memory"); }
// Bulk copy of `bytes` from global memory into this CTA's shared memory, completion on `mbar`.
// (A ring slot is read once: its lines may go first.)
__device__ __forceinline__ void bulk_load(uint32_t dst, const void *src, uint32_t bytes, uint32_t mbar) {
    asm volatile(
        "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes.L2::cache_hint [%0], [%1], %2, [%3], %4;"
        ::"r"(dst), "l"(src), "r"(bytes), "r"(mbar), "l"(l2_evict_first()) : "memory");
}

__device__ __forceinline__ uint32_t owner_of(int c) { return 1u + (uint32_t)(c % NPREP); }
// Slot of chunk c among the head's NSLOT: NSLOTP per preparer, in turn over its chunks.
__device__ __forceinline__ int slot_of(int c) { return NSLOTP * (c % NPREP) + (c / NPREP) % NSLOTP; }
// Parity of the phase, on a per-slot barrier, that belongs to chunk c.
__device__ __forceinline__ uint32_t slot_parity(int c) { return (uint32_t)((c / NPREP / NSLOTP) & 1); }

// Global-memory flags of the cooperative kernel (one int each, gpu scope).
__device__ __forceinline__ int ld_acquire_gpu(const int *f) {
    int v;
    asm volatile("ld.acquire.gpu.global.b32 %0, [%1];" : "=r"(v) : "l"(f) : "memory");
    return v;
}
__device__ __forceinline__ void st_release_gpu(int *f, int v) {
    asm volatile("st.release.gpu.global.b32 [%0], %1;" ::"l"(f), "r"(v) : "memory");
}
__device__ __forceinline__ void st_relaxed_gpu(int *f, int v) {
    asm volatile("st.relaxed.gpu.global.b32 [%0], %1;" ::"l"(f), "r"(v) : "memory");
}

// The hand-off between the CTAs that prepare a head's chunks and the CTA that carries its
// state: where chunk c's slot is, and how "chunk c is in its slot" (preparer -> state CTA,
// after the slot's bulk stores completed) and "chunk c's slot may be rewritten" (state CTA ->
// preparer, after both of its bulk loads landed) are signalled.  Every wait is bounded.
template <bool kCoop>
struct Link;

// Four-CTA cluster: NSLOTP slots per preparer, one mbarrier per slot on each side, arrives
// across the cluster's shared memories.
template <>
struct Link<false> {
    unsigned char *slots;                          // the head's NSLOT slots
    __device__ unsigned char *slot(int c) const { return slots + slot_of(c) * SLOT_BYTES; }
    // state CTA, thread 0
    __device__ bool ready_test(uint32_t sbase, int c) const {
        return cl_test(sbase + CH_READY + 8 * slot_of(c), slot_parity(c));
    }
    __device__ bool ready_wait(uint32_t sbase, int c, uint32_t polls) const {
        return cl_wait(sbase + CH_READY + 8 * slot_of(c), slot_parity(c), polls);
    }
    // Nothing of this thread's own memory operations to order, so no release.
    __device__ void release(uint32_t sbase, int c) const {
        remote_arrive_relaxed(mapa_rank(sbase + M_SLOTFREE + 8 * ((c / NPREP) % NSLOTP), owner_of(c)));
    }
    // preparer, thread kIO: chunk c is this preparer's own chunk kown
    __device__ bool free_wait(uint32_t sbase, int, int kown, uint32_t polls) const {
        return kown < NSLOTP ||
               cl_wait(sbase + M_SLOTFREE + 8 * (kown % NSLOTP), (uint32_t)((kown / NSLOTP - 1) & 1), polls);
    }
    __device__ void announce(uint32_t sbase, int c) const {
        bulk_store_wait();
        remote_arrive(mapa_rank(sbase + CH_READY + 8 * slot_of(c), 0));
    }
};

// Cooperative grid: NSLOT_COOP slots per head, chunk c in slot c % NSLOT_COOP, and per slot two
// sequence numbers in the workspace: ready = 1 + the last chunk stored there, freed = 1 + the
// last chunk read out of it.
constexpr int NSLOT_COOP = 8;
template <>
struct Link<true> {
    unsigned char *slots;                          // the head's NSLOT_COOP slots
    int *ready, *freed;                            // the head's flags, NSLOT_COOP each
    __device__ unsigned char *slot(int c) const { return slots + (c % NSLOT_COOP) * SLOT_BYTES; }
    __device__ bool ready_test(uint32_t, int c) const { return ld_acquire_gpu(ready + c % NSLOT_COOP) > c; }
    __device__ bool ready_wait(uint32_t, int c, uint32_t polls) const {
        for (uint32_t it = 0; it < polls; ++it)
            if (ready_test(0u, c)) return true;
        return false;
    }
    // (both bulk loads of chunk c completed before; the preparer acquires this flag)
    __device__ void release(uint32_t, int c) const { st_relaxed_gpu(freed + c % NSLOT_COOP, c + 1); }
    __device__ bool free_wait(uint32_t, int c, int, uint32_t polls) const {
        if (c < NSLOT_COOP) return true;
        for (uint32_t it = 0; it < polls; ++it)
            if (ld_acquire_gpu(freed + c % NSLOT_COOP) > c - NSLOT_COOP) {
                fence_global_to_async();             // the slot's next writes are bulk (async-proxy) stores
                return true;
            }
        return false;
    }
    __device__ void announce(uint32_t, int c) const {
        bulk_store_wait();
        fence_global_to_async();
        st_release_gpu(ready + c % NSLOT_COOP, c + 1);
    }
};

// ---------------------------------------------------------------- rank 0: the state carry
constexpr int kOIO = 32;                         // rank 0: issues and waits for the TMA stores of o
// ia, ib count the bulk loads issued on full_A, full_B (thread 0), so that a
// failure can wait for the one that may still be landing.
// Per chunk c, with W^T(c) and U~^T(c) already in tensor memory:
//   S^T copied to fp16 (S16) and decayed; -W(c) into the [Qg; -W] tile; [O^T | U^T] +=
//   S16 [Qg; -W]^T (o of chunk c - 1 is stored meanwhile); U^T copied to an fp16 tile;
//   [S^T | O^T] += U^T [Kend^T; P]^T, and right behind it on the tensor core W^T(c + 1),
//   U~^T(c + 1) from the next inbox A.
template <bool kCoop>
__device__ __forceinline__ bool run_chain(const Tc05Params &p, const Head &hd, char *sm, uint32_t tmem, MmaBar &mb,
                                          int n, const Link<kCoop> &lk, int &ia, int &ib) {
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int wq = warp & 3, wc = warp >> 2;
    const uint32_t sbase = smem_u32(sm);
    const uint32_t lane_off = (uint32_t)(32 * wq) << 16;
    const int trow = 32 * wq + lane;
    const int64_t sbase_e = ((int64_t)hd.b * p.Hv + hd.h) * DK * DV;   // the head's state tile (elements)
    float *state = p.state + sbase_e;
    const int64_t obase = hd.b * p.o_sb + hd.h * p.o_sh;
    const float *dec = f32p(sm, CH_DEC);            // e^gC of the chunk in inbox A
    // (debug build) a ring access outside the workspace is skipped; its barrier phase still completes
    auto ws_off = [&](int c) { return (int64_t)(lk.slot(c) - reinterpret_cast<const unsigned char *>(p.err)); };
    auto load_a = [&](int c) {
        ++ia;
        const int64_t off = ws_off(c) + SL_QG;
        if (range_in_bounds(off, A_BYTES, p.ext.ws, p.err, p.status)) {
            const unsigned char *src = lk.slot(c);
            arrive_expect_tx(sbase + CH_FULL_A, A_BYTES);
#pragma unroll
            for (int kb = 0; kb < 2; ++kb)               // Qg: 64-row blocks into rows 0..63 of [Qg; -W]
                bulk_load(sbase + CH_QW + kb * 16384, src + SL_QG + kb * 8192, 8192, sbase + CH_FULL_A);
            bulk_load(sbase + CH_A_REST, src + SL_KG, A_REST_BYTES, sbase + CH_FULL_A);
        } else {
            asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(sbase + CH_FULL_A) : "memory");
        }
    };
    auto load_b = [&](int c) {
        ++ib;
        const int64_t off = ws_off(c) + SL_KP;
        if (range_in_bounds(off, B_BYTES, p.ext.ws, p.err, p.status)) {
            arrive_expect_tx(sbase + CH_FULL_B, B_BYTES);
            bulk_load(sbase + CH_IN_B, lk.slot(c) + SL_KP, B_BYTES, sbase + CH_FULL_B);
        } else {
            asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(sbase + CH_FULL_B) : "memory");
        }
    };
    // (thread 0) W^T = Kg^T Tb^T and U~^T = V^T Tb^T of the chunk in inbox A (fp16 operands)
    auto issue_wu = [&]() {
        gemm16<64, 64>(tmem + T_W, sbase + CH_KG, sbase + CH_TB, false);
        gemm16<64, 64>(tmem + T_U, sbase + CH_VT, sbase + CH_TB, false);
    };
    // o of chunk cp (this thread's 16 tokens of column trow) into the staging tile, fenced for the
    // TMA store that thread kOIO issues after the next barrier; without an o map, thread stores
    auto stage_o = [&](const float (&ov)[16]) {
        if (p.o_f32) {
            float *t = f32p(sm, CH_OST);
#pragma unroll
            for (int k = 0; k < 16; ++k) t[(16 * wc + k) * DV + trow] = ov[k];
        } else {
            __nv_bfloat16 *t = reinterpret_cast<__nv_bfloat16 *>(sm + CH_OST);
#pragma unroll
            for (int k = 0; k < 16; k += 2) {                  // tokens in pairs: one conversion each
                const __nv_bfloat162 h = __floats2bfloat162_rn(ov[k], ov[k + 1]);
                t[(16 * wc + k) * DV + trow] = __low2bfloat16(h);
                t[(16 * wc + k + 1) * DV + trow] = __high2bfloat16(h);
            }
        }
        fence_smem_to_async();
    };
    auto store_prev_o = [&](const float (&ov)[16], int cp) {
        const int t0 = cp * C, nv = min(16, p.T - t0 - 16 * wc);
        const int64_t off0 = obase + (int64_t)(t0 + 16 * wc) * p.o_st + trow;
        if (p.o_f32) {
            float *op = static_cast<float *>(p.o) + off0;
#pragma unroll
            for (int k = 0; k < 16; ++k)
                if (k < nv && in_bounds(off0 + k * p.o_st, p.ext.o, p.err, p.status)) op[k * p.o_st] = ov[k];
        } else {
            __nv_bfloat16 *op = static_cast<__nv_bfloat16 *>(p.o) + off0;
#pragma unroll
            for (int k = 0; k < 16; ++k)
                if (k < nv && in_bounds(off0 + k * p.o_st, p.ext.o, p.err, p.status)) op[k * p.o_st] = __float2bfloat16_rn(ov[k]);
        }
    };

    // state -> T_S = S^T: row j = trow, columns i in [32 wc, 32 wc + 32)
    {
        float v[32];
#pragma unroll
        for (int c = 0; c < 32; ++c) {
            const int64_t e = (int64_t)(32 * wc + c) * DV + trow;
            v[c] = in_bounds(sbase_e + e, p.ext.state, p.err, p.status) ? state[e] : 0.f;
        }
        tmem_st32(tmem + lane_off + T_S + 32 * wc, v);
    }
    if (n > 0) {
        int okw = 1;
        if (tid == 0) {
            okw = lk.ready_wait(sbase, 0, p.polls);
            if (okw) {
                fence_global_to_async();
                load_a(0);
                load_b(0);
                okw = cl_wait(sbase + CH_FULL_A, 0u, p.polls);
            }
            if (okw) issue_wu();
            commit(mb.mbar);
        }
        if (!mma_wait(mb)) return false;
        if (__syncthreads_or(!okw)) return false;
    }
    float oprev[16];                       // O^T columns 16 wc .. + 15 of a chunk, lane trow
    for (int c = 0; c < n; ++c) {
        // ---------------------------------------------------------- [O^T | U^T] += S16 [Qg; -W]^T
        {
            // S16 <- S^T as fp16 pairs; S^T <- S^T Diag(e^gC) (the carry accumulates onto it)
            float amax = s16_and_decay(tmem + lane_off + T_S, tmem + lane_off + T_S16, 32 * wc, dec);
            float w16[16];
            tmem_ld16(tmem + lane_off + T_W + 16 * wc, w16);                 // -W [r][i] into rows 64..127
#pragma unroll
            for (int j = 0; j < 16; j += 2) st_h_rows(sm, CH_QW, 128, 64 + 16 * wc + j, trow, -w16[j], -w16[j + 1], amax);
            if (amax > kF16Max) record_range(p.err, p.status);
        }
        if (c > 0) tmem_ld16(tmem + lane_off + T_O + 16 * wc, oprev);       // o of chunk c - 1
        if (p.o_tma && tid == kOIO) bulk_wait_read<0>();                     // the staging tile is free
        {
            float z[16];
#pragma unroll
            for (int m = 0; m < 16; ++m) z[m] = 0.f;
            tmem_st16(tmem + lane_off + T_O + 16 * wc, z);                   // O^T starts at 0
        }
        fence_smem_to_async();
        fence_before_sync();
        __syncthreads();
        if (tid == 0) {
            fence_after_sync();
            gemm16_ts<128, 128>(tmem + T_O, tmem + T_S16, sbase + CH_QW, true);
            commit(mb.mbar);
        }
        if (c > 0) {
            if (p.o_tma) stage_o(oprev);
            else store_prev_o(oprev, c - 1);
        }
        if (!mma_wait(mb)) return false;
        if (p.o_tma && c > 0 && tid == kOIO) {
            tma_store_tile(&p.tm.o, sbase + CH_OST, (c - 1) * C, hd.h, hd.b);
            bulk_commit();
        }
        // inbox A is free (its tiles and e^gC were read): pull the next image now if it is there
        bool next_a = false;
        if (tid == 0 && c + 1 < n && lk.ready_test(sbase, c + 1)) {
            fence_global_to_async();
            load_a(c + 1);
            next_a = true;
        }
        {
            float u[16], amax = 0.f;
            tmem_ld16(tmem + lane_off + T_U + 16 * wc, u);
#pragma unroll
            for (int k = 0; k < 16; k += 4)                                   // U^T [j][s], fp16
                st_h4(sm, CH_UR, 128, trow, 16 * wc + k, u[k], u[k + 1], u[k + 2], u[k + 3], amax);
            if (amax > kF16Max) record_range(p.err, p.status);
        }
        fence_smem_to_async();
        fence_before_sync();
        // ---------------------------------------------------------- inbox B: [Kend^T; P]
        {
            const bool done = tid != 0 || cl_wait(sbase + CH_FULL_B, (uint32_t)(c & 1), p.polls);
            if (__syncthreads_or(!done)) return false;
        }
        int okw = 1;
        if (tid == 0) {
            // [S^T | O^T] += U^T [Kend^T; P]^T
            fence_after_sync();
            gemm16<192, 64>(tmem + T_S, sbase + CH_UR, sbase + CH_KP, true);
            // both images of chunk c have landed (their bulk loads completed, which this
            // thread observed): its slot may be rewritten
            lk.release(sbase, c);
            if (c + 1 < n) {
                // the next chunk's W^T, U~^T queue behind it on the tensor core
                if (!next_a) {
                    okw = lk.ready_wait(sbase, c + 1, p.polls);
                    if (okw) {
                        fence_global_to_async();
                        load_a(c + 1);
                    }
                }
                if (okw) okw = cl_wait(sbase + CH_FULL_A, (uint32_t)((c + 1) & 1), p.polls);
                if (okw) issue_wu();
            }
            commit(mb.mbar);
        }
        {
            // the products' wait, whose barrier also carries thread 0's hand-off outcome
            bool done = true;
            if (tid == 0) done = mbar_wait(mb.mbar, mb.phase, mb.polls) && okw;
            mb.phase ^= 1u;
            if (__syncthreads_or(!done)) return false;
            fence_after_sync();
        }
        if (tid == 0 && c + 1 < n) load_b(c + 1);                          // inbox B was read
    }
    if (n > 0) {                                                             // last chunk's o
        tmem_ld16(tmem + lane_off + T_O + 16 * wc, oprev);
        if (p.o_tma) {
            if (tid == kOIO) bulk_wait_read<0>();
            __syncthreads();
            stage_o(oprev);
            __syncthreads();
            if (tid == kOIO) {
                tma_store_tile(&p.tm.o, sbase + CH_OST, (n - 1) * C, hd.h, hd.b);
                bulk_commit();
            }
        } else {
            store_prev_o(oprev, n - 1);
        }
    }
    if (p.o_tma && tid == kOIO) bulk_store_wait();                        // every o store complete
    float v[32];
    tmem_ld32(tmem + lane_off + T_S + 32 * wc, v);
#pragma unroll
    for (int c = 0; c < 32; ++c) {
        const int64_t e = (int64_t)(32 * wc + c) * DV + trow;
        if (in_bounds(sbase_e + e, p.ext.state, p.err, p.status)) state[e] = v[c];
    }
    return true;
}

// ---------------------------------------------------------------- preparers: state-free phases
// A preparer takes its jobs (head, chunk) in order.  Every output leaves by bulk store from the
// shared-memory tile it was built in, as soon as the tile is complete; the staging of the next
// job's rows follows once the tiles have been read.  Thread 0 issues the tensor-core work and
// the TMA staging; thread kIO (a warp with no part in the triangular solve's serial steps)
// issues the bulk stores, waits for their reads, and announces job k > 0 after the operand phase
// of job k + 1 (or after the loop), when its stores have long completed (job 0 at once).
constexpr int kIO = 448;

template <bool kCoop>
struct Job {
    Head hd;
    int c;                                       // chunk
    int kown;                                    // the job's index among this preparer's jobs
    Link<kCoop> lk;
};

// jobs(k, job): job k of this preparer, false past the last.
template <bool kCoop, class Jobs>
__device__ __forceinline__ bool run_prep(const Tc05Params &p, char *sm, uint32_t tmem, MmaBar &mb, StageTrack &st,
                                         Jobs jobs) {
    const int tid = threadIdx.x;
    const uint32_t sbase = smem_u32(sm);
    volatile int *slot_ok = reinterpret_cast<volatile int *>(sm + M_FLAG);
    Job<kCoop> cur, nxt, prev;
    if (!jobs(0, cur)) return true;
    st.stage<STG_V | STG_K | STG_ONCE>(p, cur.hd, sbase, cur.c * C);
    st.stage<STG_Q | STG_G | STG_ONCE | STG_LAST>(p, cur.hd, sbase, cur.c * C);
    ChunkRegs cr;
    bool pending = false;                        // (thread kIO) prev has not been announced yet
    for (int k = 0;; ++k) {
        const bool more = jobs(k + 1, nxt);
        const int t0 = cur.c * C, L = min(C, p.T - t0);
        char *slot = reinterpret_cast<char *>(cur.lk.slot(cur.c));
        if (!st.wait(sbase, p.polls, p.inject && k == 0)) return false;
        // operand tiles; prefetch the next job's g rows into L2 (they are staged last)
        prep_chunk<false, true>(p, cur.hd, sm, t0, L, more ? nxt.hd : cur.hd, more ? nxt.c * C : p.T, sm + R_B, 64, cr);
        if (tid == kIO) {
            if (pending) prev.lk.announce(sbase, prev.c);
            // the slot's previous chunk has been pulled by the state CTA
            const int okw = cur.lk.free_wait(sbase, cur.c, cur.kown, p.polls);
            if (okw) {
                // Qg, Kg^T, e^gC
                ring_store(p, slot + SL_QG, sbase + R_B, 16384);
                ring_store(p, slot + SL_KG, sbase + R_C, 16384);
                ring_store(p, slot + SL_DEC, sbase + M_DEC, 512);
                bulk_commit();
            }
            *slot_ok = okw;                                              // read after the next barrier
        }
        if (!causal_terms<true>(sm, tmem, mb, cr, sm + R_F, 64, 0)) return false;
        if (*slot_ok == 0) return false;
        if (tid == kIO) {
            // P (64-row tile) into rows 128..191 of [Kend^T; P]; V^T
            ring_store(p, slot + SL_KP + 16384, sbase + R_F, 8192);
            ring_store(p, slot + SL_VT, sbase + RC_VT, 16384);
            bulk_commit();
        }
        solve_tb<true>(sm, cr);                                           // and Kend^T into A1_KE
        if (cr.amax > kF16Max) record_range(p.err, p.status);
        if (tid == kIO) {
            ring_store(p, slot + SL_TB, sbase + R_G, 8192);
            ring_store(p, slot + SL_KP, sbase + A1_KE, 16384);             // Kend^T: rows 0..127 of [Kend^T; P]
            bulk_commit();
            bulk_wait_read<0>();                                           // R_B, R_C, R_F, R_G, A1_KE read
            // the first job is announced at once (its state CTA has nothing else to work on);
            // later ones after the next job's operand phase, when their stores have long completed
            pending = k > 0;
            if (k == 0) cur.lk.announce(sbase, cur.c);
        }
        __syncthreads();
        prev = cur;
        if (!more) break;
        st.stage<STG_Q | STG_V | STG_K | STG_G | STG_ONCE | STG_LAST>(p, nxt.hd, sbase, nxt.c * C);
        cur = nxt;
    }
    if (tid == kIO && pending) prev.lk.announce(sbase, prev.c);           // the last job
    return true;
}

// After a wait gave up (thread 0): record it, give the tensor core and the last bulk load on
// each inbox (at most one can be outstanding) a bounded chance to finish.
__device__ __forceinline__ void drain_after_failure(const Tc05Params &p, uint32_t sbase, MmaBar &mb, bool chain,
                                                    int ia, int ib, StageTrack &st) {
    record_timeout(p);
    mbar_wait(mb.mbar, mb.phase ^ 1u, kSpin);
    if (ia > 0) cl_wait(sbase + CH_FULL_A, (uint32_t)((ia - 1) & 1), kSpin);
    if (ib > 0) cl_wait(sbase + CH_FULL_B, (uint32_t)((ib - 1) & 1), kSpin);
    if (!chain) st.drain(sbase);
}

__global__ void __cluster_dims__(CLUSTER, 1, 1) __launch_bounds__(NT, 1)
    prefill_cluster_kernel(const __grid_constant__ Tc05Params p) {
    extern __shared__ __align__(1024) char smem_raw[];
    char *sm = smem_raw + ((1024 - (smem_u32(smem_raw) & 1023)) & 1023);
    const uint32_t sbase = smem_u32(sm);
    const int rank = (int)cluster_ctarank();
    const bool chain = rank == 0;
    const Head hd = head_of(p, blockIdx.y, blockIdx.x / CLUSTER);
    const Link<false> lk{p.slots + ((size_t)hd.b * p.Hv + hd.h) * NSLOT * SLOT_BYTES};
    const int tid = threadIdx.x, warp = tid >> 5;
    const int n = (p.T + C - 1) / C;
    uint32_t *tslot = reinterpret_cast<uint32_t *>(sm + (chain ? CH_TMEM : M_TMEM));
    MmaBar mb{sbase + (chain ? CH_MBAR : M_MBAR), 0u, p.polls};
    if (tid == 0) {
        mbar_init(mb.mbar, 1);
        if (chain) {
            mbar_init(sbase + CH_FULL_A, 1);
            mbar_init(sbase + CH_FULL_B, 1);
            for (int i = 0; i < NSLOT; ++i) mbar_init(sbase + CH_READY + 8 * i, 1);
        } else {
            for (int i = 0; i < NSLOTP; ++i) mbar_init(sbase + M_SLOTFREE + 8 * i, 1);
            mbar_init(sbase + M_STAGE, 1);
            mbar_init(sbase + M_DEAD, 1);
        }
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    }
    if (warp == 0) tmem_alloc(smem_u32(tslot), T_COLS);
    fence_before_sync();
    __syncthreads();
    fence_after_sync();
    const uint32_t tmem = *tslot;
    cluster_barrier();                         // every CTA's barriers exist before any remote use

    int ia = 0, ib = 0;
    StageTrack st;
    bool ok;
    if (chain) {
        ok = run_chain<false>(p, hd, sm, tmem, mb, n, lk, ia, ib);
    } else {
        // own chunk k: chunk rank - 1 + 3 k of this head
        ok = run_prep<false>(p, sm, tmem, mb, st, [&](int k, Job<false> &j) {
            j.c = rank - 1 + NPREP * k;
            j.kown = k;
            j.hd = hd;
            j.lk = lk;
            return j.c < n;
        });
    }
    if (!ok && tid == 0) drain_after_failure(p, sbase, mb, chain, ia, ib, st);
    if (tid == (chain ? kOIO : kIO)) bulk_store_wait();   // no bulk store may still read this CTA's shared memory
    cp_async_wait_all();
    fence_before_sync();
    __syncthreads();
    if (warp == 0) tmem_dealloc(tmem, T_COLS);
    cluster_barrier();                         // no CTA leaves while another may still address it
}

// The same work as a cooperative grid with one CTA per SM: CTA u < B * Hv carries the state of
// (batch, v-head) u, every other CTA prepares chunks for all heads, job j = (chunk j / (B Hv),
// unit j % (B Hv)) on preparer j % (number of preparers).  All CTAs are resident together (a
// cooperative launch), so the flag waits between them always make progress.
__global__ void __launch_bounds__(NT, 1) prefill_coop_kernel(const __grid_constant__ Tc05Params p) {
    extern __shared__ __align__(1024) char smem_raw[];
    char *sm = smem_raw + ((1024 - (smem_u32(smem_raw) & 1023)) & 1023);
    const uint32_t sbase = smem_u32(sm);
    const int units = p.B * p.Hv;
    const bool chain = (int)blockIdx.x < units;
    const int tid = threadIdx.x, warp = tid >> 5;
    const int n = (p.T + C - 1) / C;
    auto link_of = [&](int u) {
        return Link<true>{p.slots + (size_t)u * NSLOT_COOP * SLOT_BYTES, p.flags + 2 * NSLOT_COOP * u,
                          p.flags + 2 * NSLOT_COOP * u + NSLOT_COOP};
    };
    uint32_t *tslot = reinterpret_cast<uint32_t *>(sm + (chain ? CH_TMEM : M_TMEM));
    MmaBar mb{sbase + (chain ? CH_MBAR : M_MBAR), 0u, p.polls};
    if (tid == 0) {
        mbar_init(mb.mbar, 1);
        if (chain) {
            mbar_init(sbase + CH_FULL_A, 1);
            mbar_init(sbase + CH_FULL_B, 1);
        } else {
            mbar_init(sbase + M_STAGE, 1);
            mbar_init(sbase + M_DEAD, 1);
        }
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    }
    if (warp == 0) tmem_alloc(smem_u32(tslot), T_COLS);
    fence_before_sync();
    __syncthreads();
    fence_after_sync();
    const uint32_t tmem = *tslot;

    int ia = 0, ib = 0;
    StageTrack st;
    bool ok;
    if (chain) {
        const int u = (int)blockIdx.x;
        ok = run_chain<true>(p, head_of(p, u / p.Hv, u % p.Hv), sm, tmem, mb, n, link_of(u), ia, ib);
    } else {
        const int pid = (int)blockIdx.x - units, nprep = (int)gridDim.x - units;
        const int64_t jobs_total = (int64_t)units * n;
        ok = run_prep<true>(p, sm, tmem, mb, st, [&](int k, Job<true> &j) {
            const int64_t jj = pid + (int64_t)nprep * k;
            if (jj >= jobs_total) return false;
            const int u = (int)(jj % units);
            j.c = (int)(jj / units);
            j.kown = k;
            j.hd = head_of(p, u / p.Hv, u % p.Hv);
            j.lk = link_of(u);
            return true;
        });
    }
    if (!ok && tid == 0) drain_after_failure(p, sbase, mb, chain, ia, ib, st);
    if (tid == (chain ? kOIO : kIO)) bulk_store_wait();
    cp_async_wait_all();
    fence_before_sync();
    __syncthreads();
    if (warp == 0) tmem_dealloc(tmem, T_COLS);
}

std::mutex g_cluster_mutex;
int g_cluster_fit[kMaxDevices];                         // per device: clusters resident at once, + 1 (0 = not queried)
int g_coop_grid[kMaxDevices];                           // per device: CTAs of a cooperative grid, + 1 (0 = not queried)

size_t coop_flag_bytes(const cgdr_args &a) { return ((size_t)a.B * a.Hv * 2 * NSLOT_COOP * sizeof(int) + 255) / 256 * 256; }

}  // namespace

// Number of four-CTA clusters of this kernel the current device runs at once (0 if none fit).
int prefill_cluster_capacity() {
    const int dev = current_device();
    if (dev < 0) return 0;
    std::lock_guard<std::mutex> lock(g_cluster_mutex);
    if (g_cluster_fit[dev] == 0) {
        int fit = 0;
        if (cudaFuncSetAttribute(prefill_cluster_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 CL_SMEM_BYTES) == cudaSuccess) {
            cudaLaunchConfig_t cfg = {};
            cfg.gridDim = dim3(CLUSTER, 1, 1);
            cfg.blockDim = dim3(NT, 1, 1);
            cfg.dynamicSmemBytes = CL_SMEM_BYTES;
            if (cudaOccupancyMaxActiveClusters(&fit, prefill_cluster_kernel, &cfg) != cudaSuccess) fit = 0;
        }
        cudaGetLastError();
        g_cluster_fit[dev] = fit + 1;
    }
    return g_cluster_fit[dev] - 1;
}

// CTAs of a cooperative grid of the cooperative kernel on the current device (every CTA resident
// at once; 0 if the device cannot launch it).
int prefill_coop_grid() {
    const int dev = current_device();
    if (dev < 0) return 0;
    std::lock_guard<std::mutex> lock(g_cluster_mutex);
    if (g_coop_grid[dev] == 0) {
        int grid = 0, coop = 0, per_sm = 0, sms = 0;
        if (cudaDeviceGetAttribute(&coop, cudaDevAttrCooperativeLaunch, dev) == cudaSuccess && coop &&
            cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) == cudaSuccess &&
            cudaFuncSetAttribute(prefill_coop_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, CL_SMEM_BYTES) ==
                cudaSuccess &&
            cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, prefill_coop_kernel, NT, CL_SMEM_BYTES) == cudaSuccess)
            grid = per_sm * sms;
        cudaGetLastError();
        g_coop_grid[dev] = grid + 1;
    }
    return g_coop_grid[dev] - 1;
}

size_t prefill_coop_workspace(const cgdr_args &a) {
    return WS_HEADER + coop_flag_bytes(a) + (size_t)a.B * a.Hv * NSLOT_COOP * SLOT_BYTES;
}

cgdr_status launch_prefill_coop(const cgdr_args &a, void *ws, size_t ws_bytes, cudaStream_t s) {
    const int grid = prefill_coop_grid();
    if (grid <= a.B * a.Hv) return CGDR_ERR_UNSUPPORTED;
    Tc05Params p;
    if (!make_params(a, ws, ws_bytes, p)) return CGDR_ERR_ALIGNMENT;
    p.flags = reinterpret_cast<int *>(static_cast<unsigned char *>(ws) + WS_HEADER);
    p.slots = static_cast<unsigned char *>(ws) + WS_HEADER + coop_flag_bytes(a);
    // the status word and every sequence number start at 0
    if (cudaMemsetAsync(ws, 0, WS_HEADER + coop_flag_bytes(a), s) != cudaSuccess) return CGDR_ERR_CUDA;
    void *args[] = {&p};
    if (cudaLaunchCooperativeKernel(reinterpret_cast<const void *>(prefill_coop_kernel), dim3(grid), dim3(NT), args,
                                    CL_SMEM_BYTES, s) != cudaSuccess) {
        cudaGetLastError();
        return CGDR_ERR_CUDA;
    }
    return CGDR_OK;
}

size_t prefill_cluster_workspace(const cgdr_args &a) {
    return WS_HEADER + (size_t)a.B * a.Hv * NSLOT * SLOT_BYTES;
}

cgdr_status launch_prefill_cluster(const cgdr_args &a, void *ws, size_t ws_bytes, cudaStream_t s) {
    Tc05Params p;
    if (!make_params(a, ws, ws_bytes, p)) return CGDR_ERR_ALIGNMENT;
    p.slots = static_cast<unsigned char *>(ws) + WS_HEADER;
    static SmemOnce smem_once;
    if (cudaMemsetAsync(ws, 0, sizeof(int), s) != cudaSuccess) return CGDR_ERR_CUDA;
    if (!smem_limit_once(smem_once, reinterpret_cast<const void *>(prefill_cluster_kernel), CL_SMEM_BYTES))
        return CGDR_ERR_CUDA;
    dim3 grid(CLUSTER * a.Hv, a.B);
    prefill_cluster_kernel<<<grid, NT, CL_SMEM_BYTES, s>>>(p);
    return cudaGetLastError() == cudaSuccess ? CGDR_OK : CGDR_ERR_CUDA;
}

}  // namespace cgdr
