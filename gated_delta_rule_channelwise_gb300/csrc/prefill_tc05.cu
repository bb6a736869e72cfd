// Chunked prefill on the fifth-generation tensor cores (tcgen05, TF32
// operands, fp32 accumulators in tensor memory), dk = dv = 128, chunk 64.
//
// The chunkwise WY/UT form of "Add parallel chunked prefill for channelwise
// gated delta rule" (executorch PR #21061, Summary): per chunk the
// per-channel log-decay prefix, the causal query/key terms, the beta-folded
// triangular transform, the WY pseudo-keys and pseudo-values and the state
// carry; a ragged last chunk runs through the same code (rows past the end
// are identity tokens: q = k = v = 0, g = 0, beta = 0).
//
// One CTA owns one (batch, v-head) and walks its chunks in order; the state
// lives in tensor memory as S^T [dv x dk] for the whole sequence.  Every
// contraction is written so that its rows are one of the 128-wide dimensions
// (M = 128, the natural tcgen05 shape):
//   D1 [A;P]^T-free form:  [beta kn e^(g-gm) ; qn e^(g-gm)] . (kn e^(gm-g))^T   (128 x 64, K = dk)
//   D2 = W^T   = (kn e^g)^T . Tb^T          (dk x C,  K = C)  Tb = (I + A)^-1 Diag(beta)
//   D3 = U^T   = V^T . Tb^T - S^T . W^T     (dv x C,  K = C then dk)
//   D4 = O^T   = S^T . (qn e^g)^T + U^T . P^T   (dv x C)
//   D0 = S^T  <- S^T Diag(e^gC) + U^T . Kend,   Kend = kn e^(gC - g)   (dv x dk, K = C)
// gm is the log-decay prefix at the chunk's middle row: with it both factors
// of e^(g_r - g_s) stay finite while 32 tokens of log-decay stay within 80 in
// magnitude on every channel.  A chunk outside that range forms A and P on
// the CUDA cores from exponentials of differences instead (exact for any
// decay).  TF32 operands (rounded to nearest) with fp32 accumulation keep the
// error near 1e-2 of the output RMS or below; the state is carried in fp32.
#include <mutex>

#include "cgdr_internal.cuh"
#include "tc05.cuh"

namespace cgdr {
namespace {

using namespace tc05;

constexpr int C = 64, DK = 128, DV = 128, NT = 512;
constexpr float kRange = 80.f;           // max |gamma_r - gamma_mid| for the tensor-core causal terms
constexpr uint32_t kSpin = 1u << 20;     // bounded mbarrier wait (iterations)

// shared memory map (bytes from a 1024-aligned base)
constexpr int R_A1 = 0;                  // 64 KB: X1 | A32 + scratch, V^T | S^T copy | U^T ; wide: q~, k~
constexpr int R_A2 = 65536;              // 32 KB: X2 (kn e^(gm-g)), the source of Kend ; wide: gamma
constexpr int R_B = 98304;               // 32 KB: Qg = qn e^g            [64 x 128]
constexpr int R_C = 131072;              // 32 KB: Kg^T [128 x 64] | -W [64 x 128] | Kend^T [128 x 64]
constexpr int R_F = 163840;              // 16 KB: P  [64 x 64]
constexpr int R_G = 180224;              // 16 KB: Xs fp32 [64][64] | Tb [64 x 64]
constexpr int R_MISC = 196608;
// misc (fp32 unless noted)
constexpr int M_RQ = R_MISC, M_RK = M_RQ + 256, M_BETA = M_RK + 256, M_GS = M_BETA + 256;
constexpr int M_H0 = M_GS + 256, M_GM = M_H0 + 2048, M_GC = M_GM + 512, M_DEC = M_GC + 512;
constexpr int M_MBAR = M_DEC + 512, M_TMEM = M_MBAR + 8, M_END = M_TMEM + 8;
constexpr int SMEM_BYTES = M_END + 1024;                 // + alignment slack
constexpr int LDA = 65;                  // fp32 A rows (padded)
constexpr int A1_A32 = R_A1, A1_Z = R_A1 + 64 * LDA * 4, A1_VT = R_A1 + 32768;
static_assert(A1_Z + 6 * 256 * 4 <= A1_VT, "A1 overflow");
// Staged raw inputs of a chunk (written by cp.async during the previous chunk's last MMAs):
// q rows -> F, k rows -> G (bf16 [64][128]); g rows -> A2 (fp32 [64][128]);
// v rows -> B (bf16 [64][128]); beta -> B + 16 KB (fp32 [64]).
constexpr int ST_Q = R_F, ST_K = R_G, ST_G = R_A2, ST_V = R_B, ST_BETA = R_B + 16384;
static_assert(SMEM_BYTES <= 232448, "shared memory over the per-block limit");

// tensor memory columns
constexpr uint32_t T_D0 = 0, T_D1 = 128, T_D2 = 192, T_D3 = 256, T_D4 = 320, T_COLS = 512;

struct Tc05Params {
    int T, Hk, Hv, l2norm, gate, o_f32;
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
};

__device__ __forceinline__ float *f32p(char *base, int off) { return reinterpret_cast<float *>(base + off); }
__device__ __forceinline__ void st_tile(char *base, int region, int R, int r, int k, float x) {
    *reinterpret_cast<float *>(base + region + sw_off(R, r, k)) = tf32r(x);
}
// Four consecutive K elements (k0 % 4 == 0) of row r: one 16-byte chunk of the swizzled tile.
__device__ __forceinline__ void st_tile4(char *base, int region, int R, int r, int k0, float a, float b, float c,
                                         float d) {
    *reinterpret_cast<float4 *>(base + region + sw_off(R, r, k0)) = make_float4(tf32r(a), tf32r(b), tf32r(c), tf32r(d));
}
__device__ __forceinline__ float ld_tile(const char *base, int region, int R, int r, int k) {
    return *reinterpret_cast<const float *>(base + region + sw_off(R, r, k));
}

__global__ void __launch_bounds__(NT, 1) prefill_tc05_kernel(const Tc05Params p) {
    extern __shared__ __align__(1024) char smem_raw[];
    char *sm = smem_raw + ((1024 - (smem_u32(smem_raw) & 1023)) & 1023);
    const uint32_t sbase = smem_u32(sm);
    float *sRq = f32p(sm, M_RQ), *sRk = f32p(sm, M_RK), *sBeta = f32p(sm, M_BETA), *sGs = f32p(sm, M_GS);
    float *sQt = f32p(sm, M_H0), *sGm = f32p(sm, M_GM), *sGc = f32p(sm, M_GC), *sDec = f32p(sm, M_DEC);
    float *sA = f32p(sm, A1_A32), *sZ = f32p(sm, A1_Z), *sXs = f32p(sm, R_G);
    const uint32_t mbar = sbase + M_MBAR;
    uint32_t *tslot = reinterpret_cast<uint32_t *>(sm + M_TMEM);

    const int h = blockIdx.x, b = blockIdx.y;
    const int hk = h / (p.Hv / p.Hk);
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int wq = warp & 3, wc = warp >> 2;                 // TMEM lane quarter, column quarter
    const int ci = tid & 127, cq = tid >> 7;                 // channel (or column), row quarter (16 rows)
    const __nv_bfloat16 *qb = p.q + b * p.q_sb + hk * p.q_sh;
    const __nv_bfloat16 *kb = p.k + b * p.k_sb + hk * p.k_sh;
    const __nv_bfloat16 *vb = p.v + b * p.v_sb + h * p.v_sh;
    const float *gbase = p.g + b * p.g_sb + h * p.g_sh;
    float *state = p.state + ((size_t)b * p.Hv + h) * DK * DV;
    const int64_t obase = b * p.o_sb + h * p.o_sh;

    if (tid == 0) {
        mbar_init(mbar, 1);
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    }
    if (warp == 0) tmem_alloc(smem_u32(tslot), T_COLS);
    fence_before_sync();
    __syncthreads();
    fence_after_sync();
    const uint32_t tmem = *tslot;
    const uint32_t lane_off = (uint32_t)(32 * wq) << 16;
    const int trow = 32 * wq + lane;                         // this thread's TMEM lane / tile row

    // state -> D0 = S^T: row j = trow, columns i in [32 wc, 32 wc + 32)
    {
        float v[32];
#pragma unroll
        for (int c = 0; c < 32; ++c) v[c] = state[(size_t)(32 * wc + c) * DV + trow];
        tmem_st32(tmem + lane_off + T_D0 + 32 * wc, v);
    }
    // cp.async staging of a chunk's raw rows: part 0 = v, beta, k; part 1 = q, g.
    auto stage = [&](int part, int tn) {
        const int Ln = min(C, p.T - tn);
        if (part == 0) {
            for (int idx = tid; idx < C * 16; idx += NT) {
                const int r = idx >> 4, c16 = idx & 15;
                const bool ok_row = r < Ln;
                const int64_t t = tn + (ok_row ? r : 0);
                cp_async16(sbase + ST_V + r * 256 + c16 * 16, vb + t * p.v_st + 8 * c16, ok_row);
                cp_async16(sbase + ST_K + r * 256 + c16 * 16, kb + t * p.k_st + 8 * c16, ok_row);
            }
            if (p.gate == CGDR_GATE_CHANNEL && tid < C) {
                const bool ok_row = tid < Ln;
                const int64_t t = tn + (ok_row ? tid : 0);
                cp_async4(sbase + ST_BETA + 4 * tid, p.beta + b * p.beta_sb + t * p.beta_st + h * p.beta_sh, ok_row);
            }
        } else {
            for (int idx = tid; idx < C * 16; idx += NT) {
                const int r = idx >> 4, c16 = idx & 15;
                const bool ok_row = r < Ln;
                const int64_t t = tn + (ok_row ? r : 0);
                cp_async16(sbase + ST_Q + r * 256 + c16 * 16, qb + t * p.q_st + 8 * c16, ok_row);
            }
            if (p.gate == CGDR_GATE_CHANNEL) {
                for (int idx = tid; idx < C * 32; idx += NT) {
                    const int r = idx >> 5, c16 = idx & 31;
                    const bool ok_row = r < Ln;
                    const int64_t t = tn + (ok_row ? r : 0);
                    cp_async16(sbase + ST_G + r * 512 + c16 * 16, gbase + t * p.g_st + 4 * c16, ok_row);
                }
            }
        }
        cp_async_commit();
    };
    if (p.T > 0) {
        stage(0, 0);
        stage(1, 0);
    }
    fence_before_sync();
    __syncthreads();

    uint32_t phase = 0;
    bool ok = true;
    auto mma_wait = [&]() -> bool {
        bool done = mbar_wait(mbar, phase, kSpin);
        phase ^= 1u;
        const bool bad = __syncthreads_or(!done) != 0;
        fence_after_sync();
        return !bad;
    };

    for (int t0 = 0; t0 < p.T && ok; t0 += C) {
        const int L = min(C, p.T - t0);
        cp_async_wait_all();
        __syncthreads();
        // ------------------------------------------------------------ P1
        // prefetch the next chunk's rows into L2
        if (t0 + C < p.T) {
            for (int idx = tid; idx < C * 16; idx += NT) {
                const int r = idx >> 4, part = idx & 15;
                const int64_t t = t0 + C + r;
                if (t >= p.T || part >= 10) continue;
                const void *ptr;
                if (part < 2) ptr = qb + t * p.q_st + 64 * part;
                else if (part < 4) ptr = kb + t * p.k_st + 64 * (part - 2);
                else if (part < 6) ptr = vb + t * p.v_st + 64 * (part - 4);
                else ptr = p.gate == CGDR_GATE_CHANNEL ? (const void *)(gbase + t * p.g_st + 32 * (part - 6)) : nullptr;
                if (ptr) asm volatile("prefetch.global.L2 [%0];" ::"l"(ptr));
            }
        }
        // row norms (a warp per 4 rows) from the staged raw q/k rows
        {
            uint2 qr[4], kr[4];
#pragma unroll
            for (int jj = 0; jj < 4; ++jj) {
                const int r = 4 * warp + jj;
                qr[jj] = *reinterpret_cast<const uint2 *>(sm + ST_Q + r * 256 + 8 * lane);
                kr[jj] = *reinterpret_cast<const uint2 *>(sm + ST_K + r * 256 + 8 * lane);
            }
            float ss[8];
#pragma unroll
            for (int jj = 0; jj < 4; ++jj) {
                const float2 q0 = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162 *>(&qr[jj].x));
                const float2 q1 = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162 *>(&qr[jj].y));
                const float2 k0 = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162 *>(&kr[jj].x));
                const float2 k1 = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162 *>(&kr[jj].y));
                ss[2 * jj] = q0.x * q0.x + q0.y * q0.y + q1.x * q1.x + q1.y * q1.y;
                ss[2 * jj + 1] = k0.x * k0.x + k0.y * k0.y + k1.x * k1.x + k1.y * k1.y;
            }
#pragma unroll
            for (int o = 16; o > 0; o >>= 1) {
#pragma unroll
                for (int e = 0; e < 8; ++e) ss[e] += __shfl_xor_sync(0xffffffffu, ss[e], o);
            }
            if (lane < 4) {
                const int r = 4 * warp + lane;
                float sq = ss[0], sk = ss[1];
#pragma unroll
                for (int jj = 1; jj < 4; ++jj)
                    if (lane == jj) { sq = ss[2 * jj]; sk = ss[2 * jj + 1]; }
                sRq[r] = (p.l2norm ? rsqrtf(sq + p.eps) : 1.f) * p.q_scale;
                sRk[r] = p.l2norm ? rsqrtf(sk + p.eps) : 1.f;
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
                    be = sigmoid_f(__bfloat162float(p.gb[b * p.b_sb + t * p.b_st + h * p.b_sh]));
                    gs = gdn_gate(p.A_log[h], __bfloat162float(p.ga[b * p.a_sb + t * p.a_st + h * p.a_sh]), p.dt_bias[h]);
                }
            }
            sBeta[r] = be;
            sGs[r] = gs;
        }
        __syncthreads();
        // per-channel log-decay prefix: thread (channel ci, rows 16 cq .. +15)
        float lam[16];
        {
            float run = 0.f;
#pragma unroll
            for (int jj = 0; jj < 16; ++jj) {
                const int r = 16 * cq + jj;
                float gv = 0.f;
                if (r < L) gv = p.gate == CGDR_GATE_CHANNEL ? f32p(sm, ST_G)[r * DK + ci] : sGs[r];
                run += gv;
                lam[jj] = run;
            }
            sQt[cq * DK + ci] = run;
        }
        __syncthreads();
        {
            float off = 0.f;
            for (int qq = 0; qq < cq; ++qq) off += sQt[qq * DK + ci];
#pragma unroll
            for (int jj = 0; jj < 16; ++jj) lam[jj] += off;
            if (cq == 2) sGm[ci] = lam[0];       // gamma at row 32 (the anchor)
            if (cq == 3) sGc[ci] = lam[15];      // gamma at the end of the chunk
        }
        __syncthreads();
        const float gm = sGm[ci], gcv = sGc[ci];
        // v column ci for this thread's 16 rows (staged), read before B is reused for Qg
        float vreg[16];
        {
            const __nv_bfloat16 *vs = reinterpret_cast<const __nv_bfloat16 *>(sm + ST_V);
#pragma unroll
            for (int jj = 0; jj < 16; ++jj) vreg[jj] = __bfloat162float(vs[(16 * cq + jj) * DK + ci]);
        }
        bool wide_local = false;
#pragma unroll
        for (int jj = 0; jj < 16; ++jj) wide_local |= fabsf(lam[jj] - gm) > kRange;
        const bool wide = __syncthreads_or(wide_local) != 0;
        // decay-scaled operands
        {
            // e^gm when it is a normal fp32 number (gm > -80): then e^g = e^gm e^(g - gm) without a third exp
            const float emv = gm > -80.f ? __expf(gm) : 0.f;
            const __nv_bfloat16 *qs = reinterpret_cast<const __nv_bfloat16 *>(sm + R_F);
            const __nv_bfloat16 *ks = reinterpret_cast<const __nv_bfloat16 *>(sm + R_G);
            float kg4[4];
#pragma unroll
            for (int jj = 0; jj < 16; ++jj) {
                const int r = 16 * cq + jj;
                const float kt = __bfloat162float(ks[r * DK + ci]) * sRk[r];
                const float qt = __bfloat162float(qs[r * DK + ci]) * sRq[r];
                float eg, e1 = 0.f;
                if (!wide) e1 = __expf(lam[jj] - gm);
                eg = (!wide && emv > 0.f) ? emv * e1 : __expf(lam[jj]);
                st_tile(sm, R_B, 64, r, ci, qt * eg);             // Qg [r][i]
                kg4[jj & 3] = kt * eg;
                if ((jj & 3) == 3) st_tile4(sm, R_C, 128, ci, r - 3, kg4[0], kg4[1], kg4[2], kg4[3]);   // Kg^T [i][s]
                if (!wide) {
                    const float e2 = __expf(gm - lam[jj]);
                    st_tile(sm, R_A1, 128, r, ci, sBeta[r] * kt * e1);   // X1 rows 0..63
                    st_tile(sm, R_A1, 128, 64 + r, ci, qt * e1);         // X1 rows 64..127
                    st_tile(sm, R_A2, 64, r, ci, kt * e2);               // X2
                } else {
                    f32p(sm, R_A1)[r * DK + ci] = qt;
                    f32p(sm, R_A1 + 32768)[r * DK + ci] = kt;
                    f32p(sm, R_A2)[r * DK + ci] = lam[jj];
                }
            }
        }
        if (tid < DK) sDec[tid] = expf(sGc[tid]);
        fence_smem_to_async();
        fence_before_sync();
        __syncthreads();
        // ------------------------------------------------------------ causal terms A, P
        if (!wide) {
            if (tid == 0) {
                fence_after_sync();
                gemm<64, 128>(tmem + T_D1, sbase + R_A1, sbase + R_A2, false);
                commit(mbar);
            }
            if (!(ok = mma_wait())) break;
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
                    st_tile4(sm, R_F, 64, r, s, s <= r ? v[c] : 0.f, s + 1 <= r ? v[c + 1] : 0.f,
                             s + 2 <= r ? v[c + 2] : 0.f, s + 3 <= r ? v[c + 3] : 0.f);
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
                ksrc[jj] = kt[r * DK + ci] * expf(gcv - lam[jj]);
            }
            __syncthreads();
#pragma unroll
            for (int jj = 0; jj < 16; ++jj) st_tile(sm, R_A2, 64, 16 * cq + jj, ci, ksrc[jj]);
#pragma unroll
            for (int e = 0; e < 8; ++e) {
                const int idx = tid + NT * e, r = idx >> 6, s = idx & 63;
                sA[r * LDA + s] = ra[e];
                st_tile(sm, R_F, 64, r, s, rp[e]);
            }
        }
        // V^T [j][s] (exact: bf16 values are TF32 values)
#pragma unroll
        for (int jj = 0; jj < 16; jj += 4)
            *reinterpret_cast<float4 *>(sm + A1_VT + sw_off(128, ci, 16 * cq + jj)) =
                make_float4(vreg[jj], vreg[jj + 1], vreg[jj + 2], vreg[jj + 3]);
        __syncthreads();
        // ------------------------------------------------------------ Tb = (I + A)^-1 Diag(beta)
        if (tid < 64) {
            const int Rb = tid >> 4, jc = tid & 15;
            float x[16];
#pragma unroll
            for (int r = 0; r < 16; ++r) {
                float acc = r == jc ? 1.f : 0.f;
#pragma unroll
                for (int s2 = 0; s2 < r; ++s2) acc = fmaf(-sA[(16 * Rb + r) * LDA + 16 * Rb + s2], x[s2], acc);
                x[r] = acc;
            }
#pragma unroll
            for (int r = 0; r < 16; ++r) sXs[(16 * Rb + r) * 64 + 16 * Rb + jc] = x[r];
        }
        __syncthreads();
        // Z_Rm = X_RR A_Rm for the six block pairs m < R (pair index R(R-1)/2 + m)
        for (int idx = tid; idx < 6 * 256; idx += NT) {
            const int pi = idx >> 8, rho = (idx >> 4) & 15, c = idx & 15;
            const int Rb = pi == 0 ? 1 : (pi < 3 ? 2 : 3), mb = pi - Rb * (Rb - 1) / 2;
            float a4[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
            for (int u = 0; u < 16; ++u)
                a4[u & 3] = fmaf(sXs[(16 * Rb + rho) * 64 + 16 * Rb + u], sA[(16 * Rb + u) * LDA + 16 * mb + c], a4[u & 3]);
            sZ[idx] = (a4[0] + a4[1]) + (a4[2] + a4[3]);
        }
        __syncthreads();
        // X_RS = -sum_{m=S}^{R-1} Z_Rm X_mS, one block diagonal at a time
#pragma unroll 1
        for (int d = 1; d < 4; ++d) {
            const int nblk = 4 - d;
            for (int idx = tid; idx < nblk * 256; idx += NT) {
                const int blk = idx >> 8, Rb = d + blk, Sb = Rb - d, rho = (idx >> 4) & 15, c = idx & 15;
                float a4[4] = {0.f, 0.f, 0.f, 0.f};
                for (int mm = Sb; mm < Rb; ++mm) {
                    const float *z = sZ + (Rb * (Rb - 1) / 2 + mm) * 256 + rho * 16;
                    const float *xs = sXs + (16 * mm) * 64 + 16 * Sb + c;
#pragma unroll
                    for (int u = 0; u < 16; ++u) a4[u & 3] = fmaf(z[u], xs[u * 64], a4[u & 3]);
                }
                sXs[(16 * Rb + rho) * 64 + 16 * Sb + c] = -((a4[0] + a4[1]) + (a4[2] + a4[3]));
            }
            __syncthreads();
        }
        {
            // thread t converts elements [4t, 4t+4) and [2048 + 4t, 2048 + 4t + 4): 16-byte reads, no conflicts
            float4 tv[2];
#pragma unroll
            for (int e = 0; e < 2; ++e) {
                const int idx = 2048 * e + 4 * tid, r = idx >> 6, s2 = idx & 63;
                const float4 x = *reinterpret_cast<const float4 *>(sXs + idx);
                tv[e] = make_float4(s2 <= r ? x.x * sBeta[s2] : 0.f, s2 + 1 <= r ? x.y * sBeta[s2 + 1] : 0.f,
                                    s2 + 2 <= r ? x.z * sBeta[s2 + 2] : 0.f, s2 + 3 <= r ? x.w * sBeta[s2 + 3] : 0.f);
            }
            __syncthreads();
#pragma unroll
            for (int e = 0; e < 2; ++e) {
                const int idx = 2048 * e + 4 * tid, r = idx >> 6, s2 = idx & 63;
                st_tile4(sm, R_G, 64, r, s2, tv[e].x, tv[e].y, tv[e].z, tv[e].w);
            }
        }
        fence_smem_to_async();
        fence_before_sync();
        __syncthreads();
        // ------------------------------------------------------------ W^T, U~^T
        if (tid == 0) {
            fence_after_sync();
            gemm<64, 64>(tmem + T_D2, sbase + R_C, sbase + R_G, false);    // W^T  = Kg^T Tb^T
            gemm<64, 64>(tmem + T_D3, sbase + A1_VT, sbase + R_G, false);  // U~^T = V^T Tb^T
            commit(mbar);
        }
        if (!(ok = mma_wait())) break;
        // -W [r][i] from D2; S^T copy [j][i] from D0, then D0 <- D0 Diag(e^gC)
        {
            float w16[16];
            tmem_ld16(tmem + lane_off + T_D2 + 16 * wc, w16);
#pragma unroll
            for (int c = 0; c < 16; ++c) st_tile(sm, R_C, 64, 16 * wc + c, trow, -w16[c]);
            float v[32];
            const int i0 = 32 * wc;
            tmem_ld32(tmem + lane_off + T_D0 + i0, v);
#pragma unroll
            for (int c = 0; c < 32; c += 4) st_tile4(sm, R_A1, 128, trow, i0 + c, v[c], v[c + 1], v[c + 2], v[c + 3]);
#pragma unroll
            for (int c = 0; c < 32; ++c) v[c] *= sDec[i0 + c];
            tmem_st32(tmem + lane_off + T_D0 + i0, v);
        }
        fence_smem_to_async();
        fence_before_sync();
        __syncthreads();
        // ------------------------------------------------------------ U^T, O^T (state part)
        if (tid == 0) {
            fence_after_sync();
            gemm<64, 128>(tmem + T_D3, sbase + R_A1, sbase + R_C, true);   // U^T += S^T (-W)^T
            gemm<64, 128>(tmem + T_D4, sbase + R_A1, sbase + R_B, false);  // O^T  = S^T Qg^T
            commit(mbar);
        }
        if (!(ok = mma_wait())) break;
        if (t0 + C < p.T) stage(0, t0 + C);          // B and G are free: next chunk's v, beta, k
        {
            float v[16];
            tmem_ld16(tmem + lane_off + T_D3 + 16 * wc, v);
#pragma unroll
            for (int c = 0; c < 16; c += 4)                                                  // U^T [j][s]
                st_tile4(sm, R_A1, 128, trow, 16 * wc + c, v[c], v[c + 1], v[c + 2], v[c + 3]);
            const float sc = wide ? 1.f : __expf(gcv - gm);
#pragma unroll
            for (int jj = 0; jj < 16; jj += 4) {                                             // Kend^T [i][s]
                const int s0 = 16 * cq + jj;
                st_tile4(sm, R_C, 128, ci, s0, ld_tile(sm, R_A2, 64, s0, ci) * sc, ld_tile(sm, R_A2, 64, s0 + 1, ci) * sc,
                         ld_tile(sm, R_A2, 64, s0 + 2, ci) * sc, ld_tile(sm, R_A2, 64, s0 + 3, ci) * sc);
            }
        }
        fence_smem_to_async();
        fence_before_sync();
        __syncthreads();
        // ------------------------------------------------------------ O^T += U^T P^T ; S^T += U^T Kend
        if (tid == 0) {
            fence_after_sync();
            gemm<64, 64>(tmem + T_D4, sbase + R_A1, sbase + R_F, true);
            gemm<128, 64>(tmem + T_D0, sbase + R_A1, sbase + R_C, true);
            commit(mbar);
        }
        if (!(ok = mma_wait())) break;
        if (t0 + C < p.T) stage(1, t0 + C);          // F and A2 are free: next chunk's q, g
        {
            float v[16];
            tmem_ld16(tmem + lane_off + T_D4 + 16 * wc, v);
            const int64_t off0 = obase + (int64_t)(t0 + 16 * wc) * p.o_st + trow;
            const int nv = min(16, L - 16 * wc);
            if (p.o_f32) {
                float *op = static_cast<float *>(p.o) + off0;
#pragma unroll
                for (int c = 0; c < 16; ++c)
                    if (c < nv) op[c * p.o_st] = v[c];
            } else {
                __nv_bfloat16 *op = static_cast<__nv_bfloat16 *>(p.o) + off0;
#pragma unroll
                for (int c = 0; c < 16; ++c)
                    if (c < nv) op[c * p.o_st] = __float2bfloat16_rn(v[c]);
            }
        }
        fence_before_sync();
        __syncthreads();
    }

    if (ok) {
        float v[32];
        tmem_ld32(tmem + lane_off + T_D0 + 32 * wc, v);
#pragma unroll
        for (int c = 0; c < 32; ++c) state[(size_t)(32 * wc + c) * DV + trow] = v[c];
    } else {
        // a wait gave up: record it, give the tensor core a bounded chance to finish, release TMEM
        if (tid == 0) {
            atomicExch(p.err, (int)CGDR_ERR_TIMEOUT);
            mbar_wait(mbar, phase ^ 1u, kSpin);
        }
    }
    fence_before_sync();
    __syncthreads();
    if (warp == 0) tmem_dealloc(tmem, T_COLS);
}

}  // namespace

bool prefill_tc05_supported(const cgdr_args &a) {
    return a.dtype == CGDR_BF16 && a.dk == 128 && a.dv == 128 && chunk_of(a) == 64;
}

size_t prefill_tc05_workspace(const cgdr_args &) { return 256; }

cgdr_status launch_prefill_tc05(const cgdr_args &a, void *ws, cudaStream_t s) {
    Tc05Params p;
    p.T = a.T; p.Hk = a.Hk; p.Hv = a.Hv; p.l2norm = a.l2norm_qk != 0; p.gate = a.gate;
    p.o_f32 = a.o_dtype == CGDR_F32;
    p.q_scale = qscale_of(a); p.eps = eps_of(a);
    p.q = static_cast<const __nv_bfloat16 *>(a.q);
    p.k = static_cast<const __nv_bfloat16 *>(a.k);
    p.v = static_cast<const __nv_bfloat16 *>(a.v);
    p.q_sb = a.q_sb; p.q_st = a.q_st; p.q_sh = a.q_sh;
    p.k_sb = a.k_sb; p.k_st = a.k_st; p.k_sh = a.k_sh;
    p.v_sb = a.v_sb; p.v_st = a.v_st; p.v_sh = a.v_sh;
    p.g = a.g; p.beta = a.beta;
    p.g_sb = a.g_sb; p.g_st = a.g_st; p.g_sh = a.g_sh;
    p.beta_sb = a.beta_sb; p.beta_st = a.beta_st; p.beta_sh = a.beta_sh;
    p.ga = static_cast<const __nv_bfloat16 *>(a.a);
    p.gb = static_cast<const __nv_bfloat16 *>(a.b);
    p.a_sb = a.a_sb; p.a_st = a.a_st; p.a_sh = a.a_sh;
    p.b_sb = a.b_sb; p.b_st = a.b_st; p.b_sh = a.b_sh;
    p.A_log = a.A_log; p.dt_bias = a.dt_bias;
    p.state = a.state; p.o = a.o;
    p.o_sb = a.o_sb; p.o_st = a.o_st; p.o_sh = a.o_sh;
    p.err = static_cast<int *>(ws);
    if (cudaMemsetAsync(ws, 0, sizeof(int), s) != cudaSuccess) return CGDR_ERR_CUDA;
    if (cudaFuncSetAttribute(prefill_tc05_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, SMEM_BYTES) !=
        cudaSuccess)
        return CGDR_ERR_CUDA;
    dim3 grid(a.Hv, a.B);
    prefill_tc05_kernel<<<grid, NT, SMEM_BYTES, s>>>(p);
    return cudaGetLastError() == cudaSuccess ? CGDR_OK : CGDR_ERR_CUDA;
}

}  // namespace cgdr

// ---------------------------------------------------------------------------
// Allocation-free prefill: the scratch is this file's static device array.
namespace cgdr {
namespace {

__device__ __align__(256) unsigned char g_noalloc_scratch[CGDR_NOALLOC_SCRATCH_BYTES];

constexpr int kMaxDevices = 64;
std::mutex g_noalloc_mutex;
void *g_noalloc_ptr[kMaxDevices] = {};

// Address of this device's copy of the static scratch; looked up once per
// device, with that device current (the caller's current device).
cgdr_status noalloc_scratch(int dev, void **out) {
    if (dev < 0 || dev >= kMaxDevices) return CGDR_ERR_CUDA;
    std::lock_guard<std::mutex> lock(g_noalloc_mutex);
    if (g_noalloc_ptr[dev] == nullptr) {
        void *p = nullptr;
        if (cudaGetSymbolAddress(&p, g_noalloc_scratch) != cudaSuccess || p == nullptr) return CGDR_ERR_CUDA;
        g_noalloc_ptr[dev] = p;
    }
    *out = g_noalloc_ptr[dev];
    return CGDR_OK;
}

}  // namespace
}  // namespace cgdr

extern "C" cgdr_status cgdr_prefill_noalloc(const cgdr_args *a, void *stream) {
    const cgdr_status st = cgdr_validate(a, 1);
    if (st != CGDR_OK || a->B == 0 || a->T == 0) return st;
    const size_t need = cgdr_prefill_workspace_size(a);
    if (need > CGDR_NOALLOC_SCRATCH_BYTES) return CGDR_ERR_WORKSPACE;
    if (need == 0) return cgdr_prefill(a, nullptr, 0, stream);
    int dev = -1;
    if (cudaGetDevice(&dev) != cudaSuccess) return CGDR_ERR_CUDA;
    void *scratch = nullptr;
    const cgdr_status s2 = cgdr::noalloc_scratch(dev, &scratch);
    if (s2 != CGDR_OK) return s2;
    return cgdr_prefill(a, scratch, CGDR_NOALLOC_SCRATCH_BYTES, stream);
}
