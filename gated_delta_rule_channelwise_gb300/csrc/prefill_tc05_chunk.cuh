// Per-chunk phases of the tcgen05 chunked prefill (TF32 operands, fp32
// accumulators in tensor memory), dk = dv = 128, chunk 64, 512 threads.
//
// The chunkwise WY/UT form of "Add parallel chunked prefill for channelwise
// gated delta rule" (executorch PR #21061, Summary).  These are the steps of
// one chunk that do not touch the recurrent state: the per-channel log-decay
// prefix, the decay-scaled operand tiles, the causal query/key terms A and P
// and the beta-folded triangular transform Tb = (I + A)^-1 Diag(beta).  The
// one-CTA-per-head kernel runs them in line with its state carry; the cluster
// kernel runs them on the producer CTAs.  A ragged last chunk runs through the
// same code (rows past the end are identity tokens: q = k = v = 0, g = 0,
// beta = 0).
//
// Every contraction has one of the 128-wide dimensions as its rows (M = 128):
//   D1 [A;P]^T-free form:  [beta kn e^(g-gm) ; qn e^(g-gm)] . (kn e^(gm-g))^T   (128 x 64, K = dk)
//   D2 = W^T   = (kn e^g)^T . Tb^T          (dk x C,  K = C)
//   D3 = U^T   = V^T . Tb^T - S^T . W^T     (dv x C,  K = C then dk)
//   D4 = O^T   = S^T . (qn e^g)^T + U^T . P^T   (dv x C)
//   D0 = S^T  <- S^T Diag(e^gC) + U^T . Kend,   Kend = kn e^(gC - g)   (dv x dk, K = C)
// gm is the log-decay prefix at the chunk's middle row: with it both factors
// of e^(g_r - g_s) stay finite while 32 tokens of log-decay stay within 80 in
// magnitude on every channel.  A chunk outside that range forms A and P on
// the CUDA cores from exponentials of differences instead (exact for any
// decay).
//
// Operand precision.  D1's anchored factors span up to e^80, so D1 takes TF32 tiles.  W, U~ and
// the U^T products take fp16 tiles, which round like TF32 (10 mantissa bits) for values below
// 65504 in magnitude, move half the bytes and run at twice the rate.  The state products
// S^T [Qg; -W]^T read S^T as TF32 straight from the fp32 state in the per-head kernel; the
// cluster kernel's state CTA, whose chain is the serial part, keeps an fp16 copy of S^T in
// tensor memory and runs them in fp16 too (Qg in fp16, prep_chunk<.., true>).  Every fp16
// value is checked against the fp16 range; a chunk that would overflow it records
// CGDR_ERR_RANGE.
#pragma once

#include <cuda.h>
#include <cuda_fp16.h>

#include "cgdr_internal.cuh"
#include "tc05.cuh"

namespace cgdr {
namespace tc05c {

using namespace tc05;

constexpr int C = 64, DK = 128, DV = 128, NT = 512;
constexpr float kRange = 80.f;           // max |gamma_r - gamma_mid| for the tensor-core causal terms
constexpr uint32_t kSpin = kDefaultPolls;   // bounded mbarrier wait (polls) of the drains after a failure

// shared memory map of a CTA that prepares chunks (bytes from a 1024-aligned base)
constexpr int R_A1 = 0;                  // 64 KB: X1 | A32 + scratch, Kend^T (fp16), X fp32 | U^T (fp16) ; wide: q~, k~
constexpr int R_A2 = 65536;              // 32 KB: X2 (kn e^(gm-g)), the source of Kend ; wide: gamma
constexpr int R_B = 98304;               // 32 KB: Qg = qn e^g [64 x 128] (TF32, or fp16 for the cluster kernel)
constexpr int R_C = 131072;              // 32 KB: Kg^T [128 x 64], V^T [128 x 64] | -W [64 x 128] (fp16)
constexpr int R_F = 163840;              // 16 KB: P  [64 x 64] (fp16)
constexpr int R_G = 180224;              // 16 KB: Tb [64 x 64] (fp16)
constexpr int R_MISC = 196608;
// misc (fp32 unless noted)
constexpr int M_RQ = R_MISC, M_RK = M_RQ + 256, M_BETA = M_RK + 256, M_GS = M_BETA + 256;
constexpr int M_H0 = M_GS + 256, M_GM = M_H0 + 2048, M_GC = M_GM + 512, M_DEC = M_GC + 512;
constexpr int M_MBAR = M_DEC + 512, M_TMEM = M_MBAR + 8, M_SLOTFREE = M_TMEM + 8;   // 4 barriers
constexpr int M_STAGE = M_SLOTFREE + 32;  // staging barrier: the TMA tiles of the next chunk's rows
constexpr int M_FLAG = M_STAGE + 8;       // int flag passed between threads across a barrier
constexpr int M_DEAD = M_FLAG + 8;        // a barrier nothing arrives on (target of the injected failure)
constexpr int M_END = M_DEAD + 8;
constexpr int PREP_SMEM_BYTES = M_END + 1024;            // + alignment slack
constexpr int LDA = 68;                  // fp32 A rows (padded, 16-byte aligned)
constexpr int LDZ = 20;                  // fp32 rows of the ten 16 x 16 Z blocks of the solve (padded)
constexpr int A1_A32 = R_A1, A1_Z = R_A1 + 64 * LDA * 4, A1_KE = R_A1 + 32768;   // Kend^T built during the solve
constexpr int RC_VT = R_C + 16384;       // V^T beside Kg^T
constexpr int A1_XS = R_A1 + 49152;     // fp32 X = (I + A)^-1 during the solve (16 KB)
static_assert(A1_Z + 10 * 16 * LDZ * 4 <= A1_KE && A1_KE + 16384 <= A1_XS && A1_XS + 16384 <= R_A2, "A1 overflow");
// Staged raw inputs of a chunk (TMA tiles; beta by cp.async), loaded while an earlier chunk finishes:
// q rows -> F, k rows -> G (bf16 [64][128]); g rows -> A2 (fp32 [64][128]);
// v rows -> B (bf16 [64][128]); beta -> B + 16 KB (fp32 [64]).
constexpr int ST_Q = R_F, ST_K = R_G, ST_G = R_A2, ST_V = R_B, ST_BETA = R_B + 16384;
static_assert(PREP_SMEM_BYTES <= 232448, "shared memory over the per-block limit");

// tensor memory columns
constexpr uint32_t T_D0 = 0, T_D1 = 128, T_D2 = 192, T_D3 = 256, T_D4 = 320, T_COLS = 512;

// TMA tensor maps of the inputs and of o: 4-D (channel, token, head, batch) with the caller's
// strides, box = 128 channels x 64 tokens; input rows past T read as zeros, o rows past T are
// not written.
struct Tc05Maps {
    CUtensorMap q, k, v, g, o;
};

struct Tc05Params {
    Tc05Maps tm;                         // first: 64-byte aligned
    int B, T, Hk, Hv, l2norm, gate, o_f32;
    float q_scale, eps;
    const __nv_bfloat16 *q, *k, *v;
    int64_t q_sb, q_st, q_sh, k_sb, k_st, k_sh, v_sb, v_st, v_sh;
    const float *g, *beta;
    int64_t g_sb, g_st, g_sh, beta_sb, beta_st, beta_sh;
    const __nv_bfloat16 *ga, *gb;
    int64_t a_sb, a_st, a_sh, b_sb, b_st, b_sh;
    const float *A_log, *dt_bias;
    float *state;
    void *o;
    int64_t o_sb, o_st, o_sh;
    int *err;                            // device word set to CGDR_ERR_TIMEOUT if a wait gives up
    int *status;                         // the caller's optional status word (the same code)
    uint32_t polls;                      // polls of the main-loop waits (drains use kSpin)
    int inject;                          // test hook: the first staging wait targets M_DEAD
    Extents ext;                         // footprints for the index checks of a debug build
    unsigned char *slots;                // cluster kernels: hand-off ring in the workspace (unused per head)
    int *flags;                          // cooperative kernel: the ring's sequence numbers
    int o_tma;                           // tm.o describes o (else o is written by thread stores)
};

// Records a wait that gave up (one thread per CTA).
__device__ __forceinline__ void record_timeout(const Tc05Params &p) {
    atomicExch(p.err, (int)CGDR_ERR_TIMEOUT);
    if (p.status != nullptr) atomicExch(p.status, (int)CGDR_ERR_TIMEOUT);
}

bool make_params(const cgdr_args &a, void *ws, size_t ws_bytes, Tc05Params &p);   // false if a tensor map cannot be encoded
// Whether every input's strides can be described by a tensor map (host arithmetic only).
bool maps_describable(const cgdr_args &a);
// Fills the tensor maps of `a` through the driver's encoder; false if it cannot (then the
// tensor-core kernels do not run).
bool make_maps(const cgdr_args &a, Tc05Maps &tm);

__device__ __forceinline__ float *f32p(char *base, int off) { return reinterpret_cast<float *>(base + off); }
__device__ __forceinline__ void st_tile(char *base, int region, int R, int r, int k, float x) {
    *reinterpret_cast<float *>(base + region + sw_off(R, r, k)) = tf32r(x);
}
// Four consecutive K elements (k0 % 4 == 0) of row r: one 16-byte chunk of the swizzled tile.
__device__ __forceinline__ void st_tile4(char *base, int region, int R, int r, int k0, float a, float b, float c,
                                         float d) {
    *reinterpret_cast<float4 *>(base + region + sw_off(R, r, k0)) = make_float4(tf32r(a), tf32r(b), tf32r(c), tf32r(d));
}
// Unrounded store: the tensor core reads the value as TF32 by dropping the low mantissa bits
// (the Qg operand, whose truncation leaves the result unchanged to the printed digits in
// emulation).
__device__ __forceinline__ void st_raw(char *base, int region, int R, int r, int k, float x) {
    *reinterpret_cast<float *>(base + region + sw_off(R, r, k)) = x;
}
__device__ __forceinline__ float ld_tile(const char *base, int region, int R, int r, int k) {
    return *reinterpret_cast<const float *>(base + region + sw_off(R, r, k));
}
// Four consecutive K elements (k0 % 4 == 0) of row r of an fp16 tile, rounded to nearest: one
// 8-byte store.  amax keeps the largest magnitude stored, for the range check.
__device__ __forceinline__ uint32_t h2_bits(__half2 h) {
    uint32_t u;
    memcpy(&u, &h, 4);
    return u;
}
__device__ __forceinline__ void st_h4(char *base, int region, int R, int r, int k0, float a, float b, float c,
                                      float d, float &amax) {
    amax = fmaxf(amax, fmaxf(fmaxf(fabsf(a), fabsf(b)), fmaxf(fabsf(c), fabsf(d))));
    *reinterpret_cast<uint2 *>(base + region + sw_off16(R, r, k0)) =
        make_uint2(h2_bits(__floats2half2_rn(a, b)), h2_bits(__floats2half2_rn(c, d)));
}
__device__ __forceinline__ void st_h(char *base, int region, int R, int r, int k, float x, float &amax) {
    amax = fmaxf(amax, fabsf(x));
    *reinterpret_cast<__half *>(base + region + sw_off16(R, r, k)) = __float2half_rn(x);
}
// Elements (r, k) = a and (r + 1, k) = b of an fp16 tile, converted together (one paired
// conversion instead of two).
__device__ __forceinline__ void st_h_rows(char *base, int region, int R, int r, int k, float a, float b,
                                          float &amax) {
    amax = fmaxf(amax, fmaxf(fabsf(a), fabsf(b)));
    const __half2 h = __floats2half2_rn(a, b);
    *reinterpret_cast<__half *>(base + region + sw_off16(R, r, k)) = __low2half(h);
    *reinterpret_cast<__half *>(base + region + sw_off16(R, r + 1, k)) = __high2half(h);
}
// One pass over this thread's 32 columns [i0, i0 + 32) of S^T in tensor memory (lane quarter
// at lane_off): the fp16 copy into columns s16 + i0 / 2 .. (the A operand of the state
// products), then S^T <- S^T Diag(dec) in place.  Two 16-column halves keep few registers live.
// Returns the largest magnitude seen (for the fp16 range check).
__device__ __forceinline__ float s16_and_decay(uint32_t t_s, uint32_t s16, int i0, const float *dec) {
    float amax = 0.f;
#pragma unroll 1
    for (int half = 0; half < 2; ++half) {
        const int j0 = i0 + 16 * half;
        float sv[16], h[8];
        tmem_ld16(t_s + j0, sv);
#pragma unroll
        for (int k = 0; k < 8; ++k) {
            amax = fmaxf(amax, fmaxf(fabsf(sv[2 * k]), fabsf(sv[2 * k + 1])));
            h[k] = __uint_as_float(h2_bits(__floats2half2_rn(sv[2 * k], sv[2 * k + 1])));
        }
        tmem_st8(s16 + j0 / 2, h);
#pragma unroll
        for (int k = 0; k < 16; ++k) sv[k] *= dec[j0 + k];
        tmem_st16(t_s + j0, sv);
    }
    return amax;
}
// Largest magnitude an fp16 operand may take (the largest finite fp16).
constexpr float kF16Max = 65504.f;
// Records an fp16 operand out of range (one thread per CTA, or any thread: idempotent).
__device__ __forceinline__ void record_range(int *err, int *status) {
    atomicExch(err, (int)CGDR_ERR_RANGE);
    if (status != nullptr) atomicExch(status, (int)CGDR_ERR_RANGE);
}

// This CTA's (batch, v-head) and the bases of its input rows.
struct Head {
    int b, h;
    const __nv_bfloat16 *qb, *kb, *vb;
    const float *gbase;
};

__device__ __forceinline__ Head head_of(const Tc05Params &p, int b, int h) {
    const int hk = h / (p.Hv / p.Hk);
    Head hd;
    hd.b = b;
    hd.h = h;
    hd.qb = p.q + b * p.q_sb + hk * p.q_sh;
    hd.kb = p.k + b * p.k_sb + hk * p.k_sh;
    hd.vb = p.v + b * p.v_sb + h * p.v_sh;
    hd.gbase = p.g + b * p.g_sb + h * p.g_sh;
    return hd;
}

// TMA load of one 128 x 64 tile (channels x tokens at token tn) of a 4-D tensor map into
// shared memory, completion counted in bytes on mbar; L2 evict-first or default.
__device__ __forceinline__ void tma_tile(uint32_t dst, const CUtensorMap *tm, int tn, int head, int b, uint32_t mbar,
                                         bool once, uint64_t pol) {
    if (once)
        asm volatile(
            "cp.async.bulk.tensor.4d.shared::cluster.global.tile.mbarrier::complete_tx::bytes.L2::cache_hint "
            "[%0], [%1, {%2, %3, %4, %5}], [%6], %7;"
            ::"r"(dst), "l"(reinterpret_cast<uint64_t>(tm)), "r"(0), "r"(tn), "r"(head), "r"(b), "r"(mbar), "l"(pol)
            : "memory");
    else
        asm volatile(
            "cp.async.bulk.tensor.4d.shared::cluster.global.tile.mbarrier::complete_tx::bytes "
            "[%0], [%1, {%2, %3, %4, %5}], [%6];"
            ::"r"(dst), "l"(reinterpret_cast<uint64_t>(tm)), "r"(0), "r"(tn), "r"(head), "r"(b), "r"(mbar)
            : "memory");
}
// L2 prefetch of the same tile.
__device__ __forceinline__ void tma_prefetch(const CUtensorMap *tm, int tn, int head, int b) {
    asm volatile("cp.async.bulk.prefetch.tensor.4d.L2.global.tile [%0, {%1, %2, %3, %4}];"
                 ::"l"(reinterpret_cast<uint64_t>(tm)), "r"(0), "r"(tn), "r"(head), "r"(b) : "memory");
}

// Staging of the raw rows of the chunk starting at token tn: q, k, v (bf16 [64][128]) and g
// (fp32 [64][128]) by TMA tiles on the staging barrier M_STAGE (thread 0: expect the bytes,
// issue the tiles, and with STG_LAST arrive, which closes the chunk's phase); beta by
// cp.async (one commit group per call, empty unless STG_V).  Rows past T arrive as zeros.
// STG_ONCE marks the rows evict-first in L2 (each is read once; for a kernel that keeps
// other data resident in L2 beside the streamed inputs).
enum : int { STG_Q = 1, STG_K = 2, STG_V = 4, STG_G = 8, STG_ONCE = 16, STG_LAST = 32 };
template <int PARTS>
__device__ __forceinline__ void stage_rows(const Tc05Params &p, const Head &hd, uint32_t sbase, int tn) {
    const int tid = threadIdx.x;
    if (tid == 0) {
        const bool once = (PARTS & STG_ONCE) != 0;
        const uint64_t pol = once ? l2_evict_first() : 0;
        const bool g_on = (PARTS & STG_G) && p.gate == CGDR_GATE_CHANNEL;
        const uint32_t bytes = ((PARTS & STG_Q) ? 16384u : 0u) + ((PARTS & STG_K) ? 16384u : 0u) +
                               ((PARTS & STG_V) ? 16384u : 0u) + (g_on ? 32768u : 0u);
        const uint32_t mbar = sbase + M_STAGE;
        if (bytes) asm volatile("mbarrier.expect_tx.relaxed.cta.shared::cta.b64 [%0], %1;" ::"r"(mbar), "r"(bytes) : "memory");
        const int hk = hd.h / (p.Hv / p.Hk);
        if (PARTS & STG_V) tma_tile(sbase + ST_V, &p.tm.v, tn, hd.h, hd.b, mbar, once, pol);
        if (PARTS & STG_K) tma_tile(sbase + ST_K, &p.tm.k, tn, hk, hd.b, mbar, once, pol);
        if (PARTS & STG_Q) tma_tile(sbase + ST_Q, &p.tm.q, tn, hk, hd.b, mbar, once, pol);
        if (g_on) tma_tile(sbase + ST_G, &p.tm.g, tn, hd.h, hd.b, mbar, once, pol);
        if (PARTS & STG_LAST) asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(mbar) : "memory");
    }
    if ((PARTS & STG_V) && p.gate == CGDR_GATE_CHANNEL && tid < C) {
        const int Ln = min(C, p.T - tn);
        const bool ok_row = tid < Ln;
        const int64_t t = tn + (ok_row ? tid : 0);
        const int64_t e = hd.b * p.beta_sb + t * p.beta_st + hd.h * p.beta_sh;
        cp_async4(sbase + ST_BETA + 4 * tid, p.beta + e, ok_row && in_bounds(e, p.ext.beta, p.err, p.status));
    }
    cp_async_commit();
}

// Phases of the staging barrier: closed by an STG_LAST call, waited for, and whether one
// has been opened by a call without STG_LAST and not yet closed.  The values are the same
// in every thread of the CTA.
struct StageTrack {
    uint32_t issued = 0, waited = 0;
    bool half = false;

    template <int PARTS>
    __device__ __forceinline__ void stage(const Tc05Params &p, const Head &hd, uint32_t sbase, int tn);
    // Waits for the staged rows of the next chunk (the oldest closed phase and this
    // thread's beta copies); every thread calls it.  False if the wait gave up in any
    // thread: the phase then still counts as not waited for, so that drain() waits for it.
    // Thread 0 polls the barrier; the other warps sleep at the CTA barrier that carries the
    // outcome (the tiles' writes, acquired by thread 0, are ordered before every thread's reads
    // by that barrier).
    __device__ __forceinline__ bool wait(uint32_t sbase, uint32_t polls, bool dead = false) {
        bool done = true;
        if (threadIdx.x == 0)
            done = dead ? mbar_wait(sbase + M_DEAD, 0u, polls) : mbar_wait(sbase + M_STAGE, waited & 1u, polls);
        cp_async_wait_all();
        const bool ok = __syncthreads_or(!done) == 0;
        if (ok) ++waited;
        return ok;
    }
    // After a failure (thread 0): closes an open phase, then waits (full limit) for the one
    // phase that can still be outstanding -- at most one is, closed or open -- so that no
    // tile is still landing in this CTA's shared memory when it leaves.
    __device__ __forceinline__ void drain(uint32_t sbase) {
        if (half) asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(sbase + M_STAGE) : "memory");
        if (half || issued > waited) mbar_wait(sbase + M_STAGE, waited & 1u, kSpin);
    }
};

template <int PARTS>
__device__ __forceinline__ void StageTrack::stage(const Tc05Params &p, const Head &hd, uint32_t sbase, int tn) {
    stage_rows<PARTS>(p, hd, sbase, tn);
    if (PARTS & STG_LAST) {
        ++issued;
        half = false;
    } else {
        half = true;
    }
}

// The CTA's tensor-core completion barrier, the parity it waits for next and the polls of
// that wait.
struct MmaBar {
    uint32_t mbar;
    uint32_t phase;
    uint32_t polls;
};

// Waits (bounded) for the committed MMAs: thread 0 polls, the other warps sleep at the CTA
// barrier that carries the outcome, then every thread fences its later tensor-memory accesses
// after it.  False if the wait gave up.  The phase advances either way, so after a failure
// the outstanding commit is phase ^ 1.
__device__ __forceinline__ bool mma_wait(MmaBar &mb) {
    bool done = true;
    if (threadIdx.x == 0) done = mbar_wait(mb.mbar, mb.phase, mb.polls);
    mb.phase ^= 1u;
    const bool bad = __syncthreads_or(!done) != 0;
    fence_after_sync();
    return !bad;
}

// Per-thread values that live across the phases of one chunk: thread (channel
// ci = tid % 128, row quarter cq = tid / 128).
struct ChunkRegs {
    float lam[16];                       // log-decay prefix of channel ci at rows 16 cq .. 16 cq + 15
    float vreg[16];                      // v column ci at those rows
    float gm, gcv;                       // prefix at the anchor row 32 and at the chunk's end
    bool wide;                           // the chunk's decay range is beyond kRange
    float amax;                          // largest magnitude this thread stored into an fp16 tile
};

// Row norms, beta, the log-decay prefix and the decay-scaled operand tiles of
// the chunk at t0 (L valid rows) from its staged raw rows; also prefetches the
// rows of head hd_pf at t_pf into L2.  The Qg tile goes to rows 0..63 of the qg_rows-row tile
// at qg (shared or global memory, same tile image).  Ends with the operand
// tiles fenced for the tensor core.
// kPrefetchQKV = false prefetches only the g rows (for callers that stage q, k, v early);
// kQgF16: Qg as an fp16 tile (else TF32).
template <bool kPrefetchQKV, bool kQgF16>
__device__ __forceinline__ void prep_chunk(const Tc05Params &p, const Head &hd, char *sm, int t0, int L,
                                           const Head &hd_pf, int t_pf, char *qg, int qg_rows, ChunkRegs &cr) {
    const int tid = threadIdx.x;
    const int ci = tid & 127, cq = tid >> 7;
    float *sRq = f32p(sm, M_RQ), *sRk = f32p(sm, M_RK), *sBeta = f32p(sm, M_BETA), *sGs = f32p(sm, M_GS);
    float *sQt = f32p(sm, M_H0), *sGm = f32p(sm, M_GM), *sGc = f32p(sm, M_GC), *sDec = f32p(sm, M_DEC);
    if (t_pf < p.T && tid == 0) {
        // L2 prefetch of the rows at t_pf, one TMA prefetch per tile
        const int hk = hd_pf.h / (p.Hv / p.Hk);
        if (kPrefetchQKV) {
            tma_prefetch(&p.tm.q, t_pf, hk, hd_pf.b);
            tma_prefetch(&p.tm.k, t_pf, hk, hd_pf.b);
            tma_prefetch(&p.tm.v, t_pf, hd_pf.h, hd_pf.b);
        }
        if (p.gate == CGDR_GATE_CHANNEL) tma_prefetch(&p.tm.g, t_pf, hd_pf.h, hd_pf.b);
    }
    // row norms from the staged raw q/k rows: four threads per row (q rows on warps 0-7, k rows
    // on warps 8-15), each summing 32 channels from four 16-byte pieces taken in a row-rotated
    // order (so a warp's loads spread over all banks), then two shuffle steps
    {
        const int rn = tid >> 2, part = tid & 3, row = rn & 63;
        const char *src = sm + (rn < 64 ? ST_Q : ST_K) + row * 256 + part * 64;
        float ss = 0.f;
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            const uint4 w = *reinterpret_cast<const uint4 *>(src + 16 * ((i + rn) & 3));
            const uint32_t wv[4] = {w.x, w.y, w.z, w.w};
#pragma unroll
            for (int e = 0; e < 4; ++e) {
                const float2 f = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162 *>(&wv[e]));
                ss = fmaf(f.x, f.x, ss);
                ss = fmaf(f.y, f.y, ss);
            }
        }
        ss += __shfl_xor_sync(0xffffffffu, ss, 1);
        ss += __shfl_xor_sync(0xffffffffu, ss, 2);
        if (part == 0) {
            if (rn < 64) sRq[row] = (p.l2norm ? rsqrtf(ss + p.eps) : 1.f) * p.q_scale;
            else sRk[row] = p.l2norm ? rsqrtf(ss + p.eps) : 1.f;
        }
    }
    if (tid < C) {
        const int r = tid;
        float be = 0.f, gs = 0.f;
        if (r < L) {
            const int64_t t = t0 + r;
            if (p.gate == CGDR_GATE_CHANNEL) {
                be = f32p(sm, ST_BETA)[r];
            } else {
                const int64_t ea = hd.b * p.a_sb + t * p.a_st + hd.h * p.a_sh, eb = hd.b * p.b_sb + t * p.b_st + hd.h * p.b_sh;
                const bool ok = in_bounds(ea, p.ext.a, p.err, p.status) && in_bounds(eb, p.ext.b, p.err, p.status) &&
                                in_bounds(hd.h, p.ext.A_log, p.err, p.status) && in_bounds(hd.h, p.ext.dt_bias, p.err, p.status);
                if (ok) {
                    be = sigmoid_f(__bfloat162float(p.gb[eb]));
                    gs = gdn_gate(p.A_log[hd.h], __bfloat162float(p.ga[ea]), p.dt_bias[hd.h]);
                }
            }
        }
        sBeta[r] = be;
        sGs[r] = gs;
    }
    // per-channel log-decay prefix: thread (channel ci, rows 16 cq .. +15), first within its
    // quarter; a per-channel gate needs only the staged g rows, so that runs before the barrier
    auto quarter_prefix = [&](bool scalar_gate) {
        float run = 0.f;
#pragma unroll
        for (int jj = 0; jj < 16; ++jj) {
            const int r = 16 * cq + jj;
            float gv = 0.f;
            if (r < L) gv = scalar_gate ? sGs[r] : f32p(sm, ST_G)[r * DK + ci];
            run += gv;
            cr.lam[jj] = run;
        }
        sQt[cq * DK + ci] = run;
    };
    if (p.gate == CGDR_GATE_CHANNEL) quarter_prefix(false);
    __syncthreads();
    if (p.gate != CGDR_GATE_CHANNEL) {
        quarter_prefix(true);
        __syncthreads();
    }
    {
        // every thread forms its quarter's offset, the anchor (row 32) and the chunk total
        // from the four quarter totals of its channel
        const float q0 = sQt[ci], q1 = sQt[DK + ci], q2 = sQt[2 * DK + ci], q3 = sQt[3 * DK + ci];
        const float q01 = q0 + q1, q012 = q01 + q2;
        const float off = cq == 0 ? 0.f : (cq == 1 ? q0 : (cq == 2 ? q01 : q012));
#pragma unroll
        for (int jj = 0; jj < 16; ++jj) cr.lam[jj] += off;
        const float g32 = 32 < L ? (p.gate == CGDR_GATE_CHANNEL ? f32p(sm, ST_G)[32 * DK + ci] : sGs[32]) : 0.f;
        cr.gm = g32 + q01;                   // gamma at row 32 (the anchor)
        cr.gcv = q3 + q012;                  // gamma at the end of the chunk
        if (cq == 0) {
            sGm[ci] = cr.gm;
            sGc[ci] = cr.gcv;
        }
    }
    const float gm = cr.gm;
    cr.amax = 0.f;
    // v column ci for this thread's 16 rows (staged), read before B is reused for Qg
    {
        const __nv_bfloat16 *vs = reinterpret_cast<const __nv_bfloat16 *>(sm + ST_V);
#pragma unroll
        for (int jj = 0; jj < 16; ++jj) cr.vreg[jj] = __bfloat162float(vs[(16 * cq + jj) * DK + ci]);
    }
    bool wide_local = false;
#pragma unroll
    for (int jj = 0; jj < 16; ++jj) wide_local |= fabsf(cr.lam[jj] - gm) > kRange;
    const bool wide = __syncthreads_or(wide_local) != 0;
    cr.wide = wide;
    // decay-scaled operands
    {
        // e^gm when it is a normal fp32 number (gm > -80): then e^g = e^gm e^(g - gm) without a third exp
        const float emv = gm > -80.f ? __expf(gm) : 0.f;
        const __nv_bfloat16 *qs = reinterpret_cast<const __nv_bfloat16 *>(sm + ST_Q);
        const __nv_bfloat16 *ks = reinterpret_cast<const __nv_bfloat16 *>(sm + ST_K);
        float kg4[4], rk4[4], rq4[4], be4[4], qprev = 0.f;
        // the whole warp takes e^g = e^gm e^(g - gm) (a uniform branch: no second exponential)
        const bool fastw = __all_sync(0xffffffffu, !wide && emv > 0.f);
#pragma unroll
        for (int jj = 0; jj < 16; ++jj) {
            const int r = 16 * cq + jj;
            if ((jj & 3) == 0) {                 // per-row factors of the next four rows: one 16-byte load each
                const float4 a = *reinterpret_cast<const float4 *>(sRk + r);
                const float4 b2 = *reinterpret_cast<const float4 *>(sRq + r);
                const float4 c2 = *reinterpret_cast<const float4 *>(sBeta + r);
                rk4[0] = a.x; rk4[1] = a.y; rk4[2] = a.z; rk4[3] = a.w;
                rq4[0] = b2.x; rq4[1] = b2.y; rq4[2] = b2.z; rq4[3] = b2.w;
                be4[0] = c2.x; be4[1] = c2.y; be4[2] = c2.z; be4[3] = c2.w;
            }
            const float kt = __bfloat162float(ks[r * DK + ci]) * rk4[jj & 3];
            const float qt = __bfloat162float(qs[r * DK + ci]) * rq4[jj & 3];
            float eg, e1 = 0.f;
            if (!wide) e1 = __expf(cr.lam[jj] - gm);
            if (fastw) eg = emv * e1;
            else eg = (!wide && emv > 0.f) ? emv * e1 : __expf(cr.lam[jj]);
            if (kQgF16) {                                           // Qg [r][i], rows in pairs
                if (jj & 1) st_h_rows(qg, 0, qg_rows, r - 1, ci, qprev, qt * eg, cr.amax);
                else qprev = qt * eg;
            } else {
                st_raw(qg, 0, qg_rows, r, ci, qt * eg);             // (taken as TF32 by truncation)
            }
            kg4[jj & 3] = kt * eg;
            if ((jj & 3) == 3) st_h4(sm, R_C, 128, ci, r - 3, kg4[0], kg4[1], kg4[2], kg4[3], cr.amax);   // Kg^T [i][s]
            if (!wide) {
                const float e2 = __expf(gm - cr.lam[jj]);
                st_tile(sm, R_A1, 128, r, ci, be4[jj & 3] * kt * e1);   // X1 rows 0..63
                st_tile(sm, R_A1, 128, 64 + r, ci, qt * e1);         // X1 rows 64..127
                st_tile(sm, R_A2, 64, r, ci, kt * e2);               // X2
            } else {
                f32p(sm, R_A1)[r * DK + ci] = qt;
                f32p(sm, R_A1 + 32768)[r * DK + ci] = kt;
                f32p(sm, R_A2)[r * DK + ci] = cr.lam[jj];
            }
        }
    }
    if (tid < DK) sDec[tid] = expf(sGc[tid]);
    fence_smem_to_async();
    fence_before_sync();
    __syncthreads();
}

// The causal terms: A (fp32, strictly lower, beta-folded) into A1_A32, P (lower
// with diagonal) into rows pt_row0 .. pt_row0 + 63 of the pt_rows-row tile at pt
// (shared or global memory), the Kend source into R_A2 for a wide chunk, and
// V^T into RC_VT.  False if a tensor-core wait gave up.
// kBulkOut: P and V^T leave by bulk copy, so fence them for the async proxy.
template <bool kBulkOut>
__device__ __forceinline__ bool causal_terms(char *sm, uint32_t tmem, MmaBar &mb, ChunkRegs &cr, char *pt,
                                             int pt_rows, int pt_row0) {
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int wq = warp & 3, wc = warp >> 2;
    const int ci = tid & 127, cq = tid >> 7;
    const uint32_t sbase = smem_u32(sm);
    const uint32_t lane_off = (uint32_t)(32 * wq) << 16;
    const int trow = 32 * wq + lane;
    float *sA = f32p(sm, A1_A32), *sBeta = f32p(sm, M_BETA);
    // V^T [j][s] into R_C's second half (exact in fp16 for bf16 values of magnitude 2^-14 .. 65504)
    auto store_vt = [&]() {
#pragma unroll
        for (int jj = 0; jj < 16; jj += 4)
            st_h4(sm, RC_VT, 128, ci, 16 * cq + jj, cr.vreg[jj], cr.vreg[jj + 1], cr.vreg[jj + 2], cr.vreg[jj + 3], cr.amax);
    };
    if (!cr.wide) {
        if (tid == 0) {
            fence_after_sync();
            gemm<64, 128>(tmem + T_D1, sbase + R_A1, sbase + R_A2, false);
            commit(mb.mbar);
        }
        store_vt();                          // while the product runs (it reads A1 and A2 only)
        if (!mma_wait(mb)) return false;
        float v[16];
        tmem_ld16(tmem + lane_off + T_D1 + 16 * wc, v);
        if (trow < 64) {
#pragma unroll
            for (int c = 0; c < 16; ++c) {
                const int s = 16 * wc + c;
                sA[trow * LDA + s] = s < trow ? v[c] : 0.f;
            }
        } else {
            const int r = trow - 64;
#pragma unroll
            for (int c = 0; c < 16; c += 4) {
                const int s = 16 * wc + c;
                st_h4(pt, 0, pt_rows, pt_row0 + r, s, s <= r ? v[c] : 0.f, s + 1 <= r ? v[c + 1] : 0.f,
                      s + 2 <= r ? v[c + 2] : 0.f, s + 3 <= r ? v[c + 3] : 0.f, cr.amax);
            }
        }
    } else {
        // exact form for a chunk with a wide decay range: exponentials of differences
        const float *qt = f32p(sm, R_A1), *kt = f32p(sm, R_A1 + 32768), *gg = f32p(sm, R_A2);
        float ra[8], rp[8];
#pragma unroll
        for (int e = 0; e < 8; ++e) {
            const int idx = tid + NT * e, r = idx >> 6, s = idx & 63;
            float sa = 0.f, sp = 0.f;
            if (s <= r) {
#pragma unroll 1
                for (int i = 0; i < DK; ++i) {
                    const float d = expf(gg[r * DK + i] - gg[s * DK + i]);
                    const float ksd = kt[s * DK + i] * d;
                    sa = fmaf(kt[r * DK + i], ksd, sa);
                    sp = fmaf(qt[r * DK + i], ksd, sp);
                }
            }
            ra[e] = s < r ? sBeta[r] * sa : 0.f;
            rp[e] = sp;
        }
        // Kend source in A2 (overwrites gamma once every thread is past the sums)
        float ksrc[16];
#pragma unroll
        for (int jj = 0; jj < 16; ++jj) {
            const int r = 16 * cq + jj;
            ksrc[jj] = kt[r * DK + ci] * expf(cr.gcv - cr.lam[jj]);
        }
        __syncthreads();
#pragma unroll
        for (int jj = 0; jj < 16; ++jj) st_tile(sm, R_A2, 64, 16 * cq + jj, ci, ksrc[jj]);
#pragma unroll
        for (int e = 0; e < 8; ++e) {
            const int idx = tid + NT * e, r = idx >> 6, s = idx & 63;
            sA[r * LDA + s] = ra[e];
            st_h(pt, 0, pt_rows, pt_row0 + r, s, rp[e], cr.amax);
        }
        store_vt();
    }
    if (kBulkOut) fence_smem_to_async();
    __syncthreads();
    return true;
}

// Kend^T [i][s] = X2 [s][i] e^(gC - gm) into A1_KE as an fp16 tile, by all threads: thread
// (channel ci, rows 16 cq .. + 15).  A wide chunk's X2 region holds the Kend source itself.
__device__ __forceinline__ void build_kend(char *sm, ChunkRegs &cr) {
    const int tid = threadIdx.x, ci = tid & 127, cq = tid >> 7;
    const float sc = cr.wide ? 1.f : __expf(cr.gcv - cr.gm);
#pragma unroll
    for (int jj = 0; jj < 16; jj += 4) {
        const int s0 = 16 * cq + jj;
        st_h4(sm, A1_KE, 128, ci, s0, ld_tile(sm, R_A2, 64, s0, ci) * sc, ld_tile(sm, R_A2, 64, s0 + 1, ci) * sc,
              ld_tile(sm, R_A2, 64, s0 + 2, ci) * sc, ld_tile(sm, R_A2, 64, s0 + 3, ci) * sc, cr.amax);
    }
}

// Element (r, c) of the 64 x 64 fp32 X = (I + A)^-1 held in A1_XS during the solve: rows of 64
// floats with the 16-byte chunks XOR-swizzled by r % 8, so that a float4 of eight different
// rows hits eight different bank groups.
__device__ __forceinline__ int xs_off(int r, int c) { return r * 64 + ((((c >> 2) ^ (r & 7))) << 2) + (c & 3); }

// Operands of the 16 x 16 block products of the solve: the float4 at (r, c), c a multiple of 4,
// of a block of X (A1_XS), of A (A1_A32) or of one of the Z blocks (A1_Z).
struct XsBlk {
    const float *p;
    int r0, c0;
    __device__ __forceinline__ float4 operator()(int r, int c) const {
        return *reinterpret_cast<const float4 *>(p + xs_off(r0 + r, c0 + c));
    }
};
struct ABlk {
    const float *p;
    int r0, c0;
    __device__ __forceinline__ float4 operator()(int r, int c) const {
        return *reinterpret_cast<const float4 *>(p + (r0 + r) * LDA + c0 + c);
    }
};
struct ZBlk {
    const float *p;
    int blk;
    __device__ __forceinline__ float4 operator()(int r, int c) const {
        return *reinterpret_cast<const float4 *>(p + (blk * 16 + r) * LDZ + c);
    }
};

// acc += L R for 16 x 16 blocks, one warp per block: the lane owns rows rp and rp + 8
// (rp = lane % 8) and columns c4 .. c4 + 3 (c4 = 4 (lane / 8)).  Each quarter-warp reads one
// float4 of R per step (one address per four lanes) and eight rows of L in distinct bank groups.
template <class L, class R>
__device__ __forceinline__ void blk_mma(float (&acc)[2][4], const L &lf, const R &rt, int rp, int c4) {
#pragma unroll
    for (int k4 = 0; k4 < 16; k4 += 4) {
        const float4 l0 = lf(rp, k4), l1 = lf(rp + 8, k4);
        const float lv[2][4] = {{l0.x, l0.y, l0.z, l0.w}, {l1.x, l1.y, l1.z, l1.w}};
#pragma unroll
        for (int kk = 0; kk < 4; ++kk) {
            const float4 b = rt(k4 + kk, c4);
#pragma unroll
            for (int i = 0; i < 2; ++i) {
                acc[i][0] = fmaf(lv[i][kk], b.x, acc[i][0]);
                acc[i][1] = fmaf(lv[i][kk], b.y, acc[i][1]);
                acc[i][2] = fmaf(lv[i][kk], b.z, acc[i][2]);
                acc[i][3] = fmaf(lv[i][kk], b.w, acc[i][3]);
            }
        }
    }
}

// Tb = (I + A)^-1 Diag(beta) into R_G as an fp16 tile, by 16 x 16 blocks (and with kKend, while
// 64 threads run the diagonal substitution, Kend^T = (kn e^(gC - g))^T into A1_KE as an fp16
// tile; see build_kend).  With X_RR = (I + A_RR)^-1 and Z_Rm = X_RR A_Rm, block row R of
// (I + A) X = I gives X_RS = -sum_{m=S}^{R-1} Z_Rm X_mS for R > S.  After the diagonal blocks
// (forward substitution, one thread per column), three block-product phases, one warp per
// 16 x 16 product:
//   Z_Rm for the six pairs m < R (and the zero blocks above the diagonal of Tb);
//   X_10, X_21, X_32 from the diagonal blocks, and Z'_30 = Z_30 - Z_32 Z_20, Z'_31 = Z_31 - Z_32 Z_21;
//   X_20, X_31, and X_30 = -(Z'_30 X_00 + Z'_31 X_10) (X_20 substituted into the row-3 sum),
//   the two products of each block on two warps.
// Every block of Tb is stored (scaled by beta, in fp16) by the warp that forms it; X stays in
// fp32 in A1_XS for the later phases.  Ends with Tb fenced for the tensor core.
template <bool kKend>
__device__ __forceinline__ void solve_tb(char *sm, ChunkRegs &cr) {
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    float &amax = cr.amax;
    const float *sA = f32p(sm, A1_A32), *sBeta = f32p(sm, M_BETA);
    float *sZ = f32p(sm, A1_Z), *sXs = f32p(sm, A1_XS);
    if (kKend && tid >= 64 && tid < 448) {
        // Kend^T [i][s] = X2 [s][i] e^(gC_i - gm_i) (a wide chunk's X2 region holds the Kend
        // source itself): thread (channel i, row quads q0, q0 + 3, ...)
        const int i = (tid - 64) & 127, q0 = (tid - 64) >> 7;
        const float sc = cr.wide ? 1.f : __expf(f32p(sm, M_GC)[i] - f32p(sm, M_GM)[i]);
        for (int q = q0; q < 16; q += 3) {
            const int s0 = 4 * q;
            st_h4(sm, A1_KE, 128, i, s0, ld_tile(sm, R_A2, 64, s0, i) * sc, ld_tile(sm, R_A2, 64, s0 + 1, i) * sc,
                  ld_tile(sm, R_A2, 64, s0 + 2, i) * sc, ld_tile(sm, R_A2, 64, s0 + 3, i) * sc, amax);
        }
    }
    if (tid < 64) {
        // X_RR column jc (zero above the diagonal, as the recurrence gives), and Tb's diagonal block
        const int Rb = tid >> 4, jc = tid & 15;
        float x[16];
#pragma unroll
        for (int r = 0; r < 16; ++r) {
            float acc = r == jc ? 1.f : 0.f;
#pragma unroll
            for (int s2 = 0; s2 < r; ++s2) acc = fmaf(-sA[(16 * Rb + r) * LDA + 16 * Rb + s2], x[s2], acc);
            x[r] = acc;
        }
        const float bj = sBeta[16 * Rb + jc];
#pragma unroll
        for (int r = 0; r < 16; ++r) {
            sXs[xs_off(16 * Rb + r, 16 * Rb + jc)] = x[r];
            st_h(sm, R_G, 64, 16 * Rb + r, 16 * Rb + jc, x[r] * bj, amax);
        }
    }
    __syncthreads();
    const int rp = lane & 7, c4 = 4 * (lane >> 3);
    float acc[2][4];
    auto zero = [&]() {
#pragma unroll
        for (int i = 0; i < 2; ++i)
#pragma unroll
            for (int j = 0; j < 4; ++j) acc[i][j] = 0.f;
    };
    auto put_z = [&](int blk, float sg) {
#pragma unroll
        for (int i = 0; i < 2; ++i)
            *reinterpret_cast<float4 *>(sZ + (blk * 16 + rp + 8 * i) * LDZ + c4) =
                make_float4(sg * acc[i][0], sg * acc[i][1], sg * acc[i][2], sg * acc[i][3]);
    };
    auto put_x = [&](int Rb, int Sb) {                 // X_RS = -acc, kept for the next phase
#pragma unroll
        for (int i = 0; i < 2; ++i)
            *reinterpret_cast<float4 *>(sXs + xs_off(16 * Rb + rp + 8 * i, 16 * Sb + c4)) =
                make_float4(-acc[i][0], -acc[i][1], -acc[i][2], -acc[i][3]);
    };
    auto put_tb = [&](int Rb, int Sb) {                // Tb_RS = -acc Diag(beta_S)
        const float4 be = *reinterpret_cast<const float4 *>(sBeta + 16 * Sb + c4);
#pragma unroll
        for (int i = 0; i < 2; ++i)
            st_h4(sm, R_G, 64, 16 * Rb + rp + 8 * i, 16 * Sb + c4, -acc[i][0] * be.x, -acc[i][1] * be.y,
                  -acc[i][2] * be.z, -acc[i][3] * be.w, amax);
    };
    auto neg_z = [&](int blk) {                        // acc = -Z_blk
#pragma unroll
        for (int i = 0; i < 2; ++i) {
            const float4 z = ZBlk{sZ, blk}(rp + 8 * i, c4);
            acc[i][0] = -z.x; acc[i][1] = -z.y; acc[i][2] = -z.z; acc[i][3] = -z.w;
        }
    };
    // Z block index of pair (R, m): R (R - 1) / 2 + m; block 6 holds Z'_31, blocks 7..9 the
    // second products of the last phase
    if (warp < 6) {
        const int Rb = warp == 0 ? 1 : (warp < 3 ? 2 : 3), mb = warp - Rb * (Rb - 1) / 2;
        zero();
        blk_mma(acc, XsBlk{sXs, 16 * Rb, 16 * Rb}, ABlk{sA, 16 * Rb, 16 * mb}, rp, c4);
        put_z(warp, 1.f);
    } else if (warp < 12) {
        // block (R, S), R < S, of Tb is zero: lane = (row, 8-column half), one 16-byte store
        const int u = warp - 6, Rb = u < 3 ? 0 : (u < 5 ? 1 : 2), Sb = u < 3 ? u + 1 : (u < 5 ? u - 1 : 3);
        *reinterpret_cast<uint4 *>(sm + R_G + sw_off16(64, 16 * Rb + (lane >> 1), 16 * Sb + 8 * (lane & 1))) =
            make_uint4(0u, 0u, 0u, 0u);
    }
    __syncthreads();
    if (warp < 3) {                                    // X_{d+1,d} = -Z_{d+1,d} X_dd
        const int d = warp, zb = d == 0 ? 0 : (d == 1 ? 2 : 5);
        zero();
        blk_mma(acc, ZBlk{sZ, zb}, XsBlk{sXs, 16 * d, 16 * d}, rp, c4);
        if (d < 2) put_x(d + 1, d);
        put_tb(d + 1, d);
    } else if (warp < 5) {                             // Z'_30 (in place of Z_30), Z'_31 (block 6)
        const int m = warp - 3;
        neg_z(3 + m);
        blk_mma(acc, ZBlk{sZ, 5}, ZBlk{sZ, 1 + m}, rp, c4);
        put_z(m == 0 ? 3 : 6, -1.f);
    }
    __syncthreads();
    if (warp < 6) {
        // X_20 = -(Z_20 X_00 + Z_21 X_10), X_31 = -(Z_31 X_11 + Z_32 X_21), X_30 = -(Z'_30 X_00 + Z'_31 X_10):
        // block j = warp % 3; warp j forms the first product, warp j + 3 the second and hands it over
        const int j = warp % 3, second = warp >= 3;
        const int Rb = j == 1 ? 3 : 2 + (j == 2), Sb = j == 1 ? 1 : 0;
        const int zb = second ? (j == 0 ? 2 : (j == 1 ? 5 : 6)) : (j == 0 ? 1 : (j == 1 ? 4 : 3));
        zero();
        blk_mma(acc, ZBlk{sZ, zb}, XsBlk{sXs, 16 * Sb + 16 * second, 16 * Sb}, rp, c4);
        if (second) {
            put_z(7 + j, 1.f);
            if (j == 0) named_bar_arrive<1, 64>();
            else if (j == 1) named_bar_arrive<2, 64>();
            else named_bar_arrive<3, 64>();
        } else {
            if (j == 0) named_bar_sync<1, 64>();
            else if (j == 1) named_bar_sync<2, 64>();
            else named_bar_sync<3, 64>();
#pragma unroll
            for (int i = 0; i < 2; ++i) {
                const float4 z = ZBlk{sZ, 7 + j}(rp + 8 * i, c4);
                acc[i][0] += z.x; acc[i][1] += z.y; acc[i][2] += z.z; acc[i][3] += z.w;
            }
            put_tb(Rb, Sb);
        }
    }
    fence_smem_to_async();
    fence_before_sync();
    __syncthreads();
}

// Columns [16 wc, 16 wc + 16) of O^T (chunk at t0, L valid tokens) from TMEM to o.
__device__ __forceinline__ void store_o(const Tc05Params &p, int64_t obase, uint32_t taddr, int t0, int L) {
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int wq = warp & 3, wc = warp >> 2;
    const int trow = 32 * wq + lane;
    float v[16];
    tmem_ld16(taddr + ((uint32_t)(32 * wq) << 16) + 16 * wc, v);
    const int64_t off0 = obase + (int64_t)(t0 + 16 * wc) * p.o_st + trow;
    const int nv = min(16, L - 16 * wc);
    if (p.o_f32) {
        float *op = static_cast<float *>(p.o) + off0;
#pragma unroll
        for (int c = 0; c < 16; ++c)
            if (c < nv && in_bounds(off0 + c * p.o_st, p.ext.o, p.err, p.status)) op[c * p.o_st] = v[c];
    } else {
        __nv_bfloat16 *op = static_cast<__nv_bfloat16 *>(p.o) + off0;
#pragma unroll
        for (int c = 0; c < 16; c += 2) {                      // tokens in pairs: one conversion each
            const __nv_bfloat162 h = __floats2bfloat162_rn(v[c], v[c + 1]);
            if (c < nv && in_bounds(off0 + c * p.o_st, p.ext.o, p.err, p.status)) op[c * p.o_st] = __low2bfloat16(h);
            if (c + 1 < nv && in_bounds(off0 + (c + 1) * p.o_st, p.ext.o, p.err, p.status))
                op[(c + 1) * p.o_st] = __high2bfloat16(h);
        }
    }
}

}  // namespace tc05c
}  // namespace cgdr
