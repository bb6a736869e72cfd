// Chunked prefill with the per-chunk contractions on the tensor cores
// (bf16 operands, fp32 accumulation), dk = 128, chunk C = 64.
//
// The chunkwise WY/UT form of "Add parallel chunked prefill for channelwise
// gated delta rule" (executorch PR #21061, Summary).  One CTA owns one
// (batch, v-head, WS-column slab of dv) and walks the chunks of its sequence
// in order; the state slab S [dk x WS] stays in fp32 registers (as mma
// accumulators) across chunks, so the only serial dependence is along T.
// Per chunk (rows >= L of a ragged last chunk are identity tokens: q = k =
// v = 0, g = 0, beta = 0, so the same code serves the tail):
//
//   1  row norms of q and k, beta
//   2  per-channel log-decay prefix inside each 16-row block, decay-scaled
//      bf16 operands (below), Vb = beta * V
//   3  A = strictly-lower(beta_r kn_r . kn_s e^(gamma_r - gamma_s)) and
//      P = lower(qn_r . kn_s e^(gamma_r - gamma_s)) on the tensor cores
//   4  Tinv = (I + A)^-1: 16x16 diagonal blocks by forward substitution,
//      off-diagonal blocks by block back-substitution (fp32)
//   5  -W = -Tinv (beta kn e^gamma)   and   U~ = Tinv Vb   (tensor cores)
//   6  U = U~ - W S;  O = (qn e^gamma) S + P U;  S = e^gamma_C S + Kend^T U
//      with Kend = kn e^(gamma_C - gamma)          (tensor cores)
//
// Anchoring.  e^(gamma_r - gamma_s) cannot be formed as e^gamma_r e^-gamma_s:
// with strong decay e^-gamma_s overflows fp32/bf16 within one chunk.  Each
// 16-row block R has the anchor a_R = its first row.  For block rows R and
// column blocks S <= R,
//     e^(gamma_r - gamma_s) = E_r * D(R,S) * F_s,
//     E_r = e^(gamma_r - gamma_aR) <= 1,   D(R,S) = e^(gamma_aR - gamma_aS) <= 1,
//     F_s = e^(gamma_aS - gamma_s)  >= 1  (at most the decay of 15 tokens).
// E goes into the row operand; F * D(R,.) into one column operand per block
// row (MR_R, 16(R+1) rows).  Every factor is finite as long as 15 tokens of
// log-decay stay above -80 per channel.
#include "cgdr_internal.cuh"

namespace cgdr {
namespace {

constexpr int C = 64, DK = 128, NT = 256;
constexpr int LDK = DK + 8;  // padded bf16 row strides: conflict-free ldmatrix
constexpr int LDC = C + 8;
constexpr int LDA = C + 1;   // fp32 [64][65]

template <int WS>
struct Lay {
    static constexpr int LDW = WS + 8;
    static constexpr int NPW = WS / 16;        // n8 tiles per warp in U and O
    static constexpr int NS = WS / 8;          // n8 tiles per warp in S
    // region Y, stages 2-3
    static constexpr int KL = 0;
    static constexpr int QL = KL + 64 * LDK * 2;
    static constexpr int MR = QL + 64 * LDK * 2;
    static constexpr int Y_END = MR + 160 * LDK * 2;
    // region Y, stages 4-6
    static constexpr int A32 = 0;
    static constexpr int TI32 = A32 + 64 * LDA * 4;
    static constexpr int TB = TI32 + 64 * LDA * 4;
    static constexpr int WN = TB + 64 * LDC * 2;
    static constexpr int SCR = WN + 64 * LDK * 2;
    static_assert(SCR + 3 * 256 * 4 <= Y_END, "region Y overflow");
    // persistent buffers
    static constexpr int KG = Y_END;
    static constexpr int QG = KG + 64 * LDK * 2;
    static constexpr int KE = QG + 64 * LDK * 2;
    static constexpr int PP = KE + 64 * LDK * 2;
    static constexpr int VB = PP + 64 * LDC * 2;
    static constexpr int SB = VB + 64 * LDW * 2;
    static constexpr int UU = SB + 2 * DK * LDW * 2;
    static constexpr int F32 = UU + 64 * LDW * 2;
    // fp32 misc: rq[64] rk[64] beta[64] gs[64] lam[4][128] g0[4][128] decay[128]
    static constexpr int RQ = F32, RK = RQ + 256, BETA = RK + 256, GS = BETA + 256;
    static constexpr int LAM = GS + 256, G0 = LAM + 2048, DEC = G0 + 2048;
    static constexpr int BYTES = DEC + 512;
};

struct TcParams {
    int T, Hk, Hv, dv, l2norm, gate;
    float q_scale, eps;
    const __nv_bfloat16 *q, *k, *v;
    int64_t q_sb, q_st, q_sh, k_sb, k_st, k_sh, v_sb, v_st, v_sh;
    const float *g, *beta;
    int64_t g_sb, g_st, g_sh, beta_sb, beta_st, beta_sh;
    const __nv_bfloat16 *ga, *gb;
    int64_t a_sb, a_st, a_sh, b_sb, b_st, b_sh;
    const float *A_log, *dt_bias;
    float *state;
    __nv_bfloat16 *o;
    int64_t o_sb, o_st, o_sh;
};

__device__ __forceinline__ void st_bf16x2(char *base, int off_elems, float lo, float hi) {
    *reinterpret_cast<uint32_t *>(base + off_elems * 2) = pack_bf16x2(lo, hi);
}

template <int WS>
__global__ void __launch_bounds__(NT, 1) prefill_tc_kernel(const TcParams p) {
    using Y = Lay<WS>;
    constexpr int LDW = Y::LDW, NPW = Y::NPW, NS = Y::NS;
    extern __shared__ __align__(128) char sm[];
    float *sRq = reinterpret_cast<float *>(sm + Y::RQ);
    float *sRk = reinterpret_cast<float *>(sm + Y::RK);
    float *sBeta = reinterpret_cast<float *>(sm + Y::BETA);
    float *sGs = reinterpret_cast<float *>(sm + Y::GS);
    float *sLam = reinterpret_cast<float *>(sm + Y::LAM);
    float *sG0 = reinterpret_cast<float *>(sm + Y::G0);
    float *sDec = reinterpret_cast<float *>(sm + Y::DEC);
    float *sA = reinterpret_cast<float *>(sm + Y::A32);
    float *sTi = reinterpret_cast<float *>(sm + Y::TI32);
    float *sScr = reinterpret_cast<float *>(sm + Y::SCR);
    __nv_bfloat16 *sTb = reinterpret_cast<__nv_bfloat16 *>(sm + Y::TB);
    const uint32_t uKL = smem_u32(sm + Y::KL), uQL = smem_u32(sm + Y::QL), uMR = smem_u32(sm + Y::MR);
    const uint32_t uTB = smem_u32(sm + Y::TB), uWN = smem_u32(sm + Y::WN);
    const uint32_t uKG = smem_u32(sm + Y::KG), uQG = smem_u32(sm + Y::QG), uKE = smem_u32(sm + Y::KE);
    const uint32_t uPP = smem_u32(sm + Y::PP), uVB = smem_u32(sm + Y::VB), uSB = smem_u32(sm + Y::SB);
    const uint32_t uUU = smem_u32(sm + Y::UU);

    const int slab = blockIdx.x, h = blockIdx.y, b = blockIdx.z;
    const int hk = h / (p.Hv / p.Hk);
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int gq = lane >> 2, tq = lane & 3;   // mma fragment row / column-pair
    const int col0 = slab * WS;
    float *state = p.state + ((size_t)b * p.Hv + h) * DK * p.dv + col0;
    const __nv_bfloat16 *qb = p.q + b * p.q_sb + hk * p.q_sh;
    const __nv_bfloat16 *kb = p.k + b * p.k_sb + hk * p.k_sh;
    const __nv_bfloat16 *vb = p.v + b * p.v_sb + h * p.v_sh + col0;
    __nv_bfloat16 *ob = p.o + b * p.o_sb + h * p.o_sh + col0;

    // State slab: warp w owns rows 16w..16w+15 (all WS columns) as fp32 accumulators.
    float accS[NS][4];
#pragma unroll
    for (int n = 0; n < NS; ++n) {
        const int i0 = 16 * warp + gq, c = 8 * n + 2 * tq;
        const float2 x0 = *reinterpret_cast<const float2 *>(state + (size_t)i0 * p.dv + c);
        const float2 x1 = *reinterpret_cast<const float2 *>(state + (size_t)(i0 + 8) * p.dv + c);
        accS[n][0] = x0.x; accS[n][1] = x0.y; accS[n][2] = x1.x; accS[n][3] = x1.y;
        st_bf16x2(sm + Y::SB, i0 * LDW + c, x0.x, x0.y);
        st_bf16x2(sm + Y::SB, (i0 + 8) * LDW + c, x1.x, x1.y);
    }
    int cur = 0;

    for (int t0 = 0; t0 < p.T; t0 += C) {
        const int L = min(C, p.T - t0);
        // ------------------------------------------------ 1: norms, beta, scalar gate
#pragma unroll 2
        for (int j = 0; j < 8; ++j) {
            const int r = warp * 8 + j;
            float sq = 0.f, sk = 0.f;
            if (r < L) {
                const int64_t t = t0 + r;
                const uint2 qr = *reinterpret_cast<const uint2 *>(qb + t * p.q_st + 4 * lane);
                const uint2 kr = *reinterpret_cast<const uint2 *>(kb + t * p.k_st + 4 * lane);
                const float2 q0 = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162 *>(&qr.x));
                const float2 q1 = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162 *>(&qr.y));
                const float2 k0 = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162 *>(&kr.x));
                const float2 k1 = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162 *>(&kr.y));
                sq = q0.x * q0.x + q0.y * q0.y + q1.x * q1.x + q1.y * q1.y;
                sk = k0.x * k0.x + k0.y * k0.y + k1.x * k1.x + k1.y * k1.y;
            }
            sq = warp_sum(sq);
            sk = warp_sum(sk);
            if (lane == 0) {
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
                    be = p.beta[b * p.beta_sb + t * p.beta_st + h * p.beta_sh];
                } else {
                    be = sigmoid_f(__bfloat162float(p.gb[b * p.b_sb + t * p.b_st + h * p.b_sh]));
                    gs = gdn_gate(p.A_log[h], __bfloat162float(p.ga[b * p.a_sb + t * p.a_st + h * p.a_sh]),
                                  p.dt_bias[h]);
                }
            }
            sBeta[r] = be;
            sGs[r] = gs;
        }
        __syncthreads();
        // ------------------------------------------------ 2a: in-block log-decay prefix
        // thread: block R = tid / 64 (rows 16R..16R+15), channels 2cp, 2cp+1
        const int R = tid >> 6, cp = tid & 63, ch = 2 * cp;
        float lam0[16], lam1[16];
        {
            float run0 = 0.f, run1 = 0.f;
#pragma unroll
            for (int j = 0; j < 16; ++j) {
                const int r = 16 * R + j;
                float2 gv = make_float2(0.f, 0.f);
                if (r < L) {
                    if (p.gate == CGDR_GATE_CHANNEL)
                        gv = *reinterpret_cast<const float2 *>(p.g + b * p.g_sb + (int64_t)(t0 + r) * p.g_st +
                                                               h * p.g_sh + ch);
                    else
                        gv = make_float2(sGs[r], sGs[r]);
                }
                run0 += gv.x; run1 += gv.y;
                lam0[j] = run0; lam1[j] = run1;
            }
            sLam[R * DK + ch] = run0; sLam[R * DK + ch + 1] = run1;
            sG0[R * DK + ch] = lam0[0]; sG0[R * DK + ch + 1] = lam1[0];
        }
        __syncthreads();
        // ------------------------------------------------ 2b: decay-scaled bf16 operands
        {
            float gamA[2][4], gamC[2];
#pragma unroll
            for (int c = 0; c < 2; ++c) {
                float run = 0.f;
#pragma unroll
                for (int Rp = 0; Rp < 4; ++Rp) {
                    gamA[c][Rp] = run + sG0[Rp * DK + ch + c];   // gamma at anchor row of block Rp
                    run += sLam[Rp * DK + ch + c];
                }
                gamC[c] = run;
            }
            float expA[2], expCA[2], D[2][4];
#pragma unroll
            for (int c = 0; c < 2; ++c) {
                float ga = 0.f;
#pragma unroll
                for (int Rp = 0; Rp < 4; ++Rp) if (Rp == R) ga = gamA[c][Rp];
                expA[c] = expf(ga);
                expCA[c] = expf(gamC[c] - ga);
#pragma unroll
                for (int Rp = 0; Rp < 4; ++Rp) D[c][Rp] = Rp > R ? expf(gamA[c][Rp] - ga) : 1.f;
            }
            if (R == 0) { sDec[ch] = expf(gamC[0]); sDec[ch + 1] = expf(gamC[1]); }
#pragma unroll
            for (int j = 0; j < 16; ++j) {
                const int r = 16 * R + j;
                float2 kf = make_float2(0.f, 0.f), qf = make_float2(0.f, 0.f);
                if (r < L) {
                    const int64_t t = t0 + r;
                    kf = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162 *>(kb + t * p.k_st + ch));
                    qf = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162 *>(qb + t * p.q_st + ch));
                }
                const float rk = sRk[r], rq = sRq[r], be = sBeta[r];
                const float k0 = kf.x * rk, k1 = kf.y * rk, q0 = qf.x * rq, q1 = qf.y * rq;
                const float e0 = __expf(lam0[j] - lam0[0]), e1 = __expf(lam1[j] - lam1[0]);
                const float f0 = __expf(fminf(lam0[0] - lam0[j], 80.f));
                const float f1 = __expf(fminf(lam1[0] - lam1[j], 80.f));
                st_bf16x2(sm + Y::KL, r * LDK + ch, k0 * e0 * be, k1 * e1 * be);
                st_bf16x2(sm + Y::QL, r * LDK + ch, q0 * e0, q1 * e1);
#pragma unroll
                for (int Rp = 0; Rp < 4; ++Rp) {
                    if (Rp >= R) {
                        const int base = 8 * Rp * (Rp + 1);     // first row of MR_Rp
                        st_bf16x2(sm + Y::MR, (base + r) * LDK + ch, k0 * f0 * D[0][Rp], k1 * f1 * D[1][Rp]);
                    }
                }
                st_bf16x2(sm + Y::KG, r * LDK + ch, k0 * be * e0 * expA[0], k1 * be * e1 * expA[1]);
                st_bf16x2(sm + Y::QG, r * LDK + ch, q0 * e0 * expA[0], q1 * e1 * expA[1]);
                st_bf16x2(sm + Y::KE, r * LDK + ch, k0 * f0 * expCA[0], k1 * f1 * expCA[1]);
            }
        }
        // Vb = beta * V slab
        for (int idx = tid; idx < C * (WS / 8); idx += NT) {
            const int r = idx / (WS / 8), seg = idx % (WS / 8);
            uint4 raw = make_uint4(0u, 0u, 0u, 0u);
            if (r < L) raw = *reinterpret_cast<const uint4 *>(vb + (int64_t)(t0 + r) * p.v_st + 8 * seg);
            const float be = sBeta[r];
            uint32_t w[4] = {raw.x, raw.y, raw.z, raw.w};
#pragma unroll
            for (int u = 0; u < 4; ++u) {
                const float2 f = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162 *>(&w[u]));
                w[u] = pack_bf16x2(f.x * be, f.y * be);
            }
            *reinterpret_cast<uint4 *>(sm + Y::VB + (r * LDW + 8 * seg) * 2) = make_uint4(w[0], w[1], w[2], w[3]);
        }
        __syncthreads();
        // ------------------------------------------------ 3: A and P (tensor cores)
        float res[5][4];
        {
            const int X = warp >> 2, q4 = warp & 3;
            const uint32_t uL = X == 0 ? uKL : uQL;
            uint32_t af[8][4];
            int curR = -1;
#pragma unroll
            for (int e = 0; e < 5; ++e) {
                const int f = 5 * q4 + e;
                const int Rr = f < 2 ? 0 : (f < 6 ? 1 : (f < 12 ? 2 : 3));
                const int jt = f - (Rr == 0 ? 0 : (Rr == 1 ? 2 : (Rr == 2 ? 6 : 12)));
                if (Rr != curR) {
                    curR = Rr;
#pragma unroll
                    for (int ks = 0; ks < 8; ++ks)
                        ldsm_x4(af[ks][0], af[ks][1], af[ks][2], af[ks][3],
                                uL + ((16 * Rr + (lane & 15)) * LDK + 16 * ks + (lane >> 4) * 8) * 2);
                }
                float acc[4] = {0.f, 0.f, 0.f, 0.f};
                const int base = 8 * Rr * (Rr + 1);
#pragma unroll
                for (int ks = 0; ks < 8; ks += 2) {
                    uint32_t b0, b1, b2, b3;
                    ldsm_x4(b0, b1, b2, b3, uMR + ((base + 8 * jt + (lane & 7)) * LDK + 16 * ks + (lane >> 3) * 8) * 2);
                    mma_bf16(acc, af[ks], b0, b1);
                    mma_bf16(acc, af[ks + 1], b2, b3);
                }
#pragma unroll
                for (int u = 0; u < 4; ++u) res[e][u] = acc[u];
            }
        }
        __syncthreads();   // every read of KL/QL/MR is done: region Y is reused below
        {
            const int X = warp >> 2, q4 = warp & 3;
#pragma unroll
            for (int e = 0; e < 5; ++e) {
                const int f = 5 * q4 + e;
                const int Rr = f < 2 ? 0 : (f < 6 ? 1 : (f < 12 ? 2 : 3));
                const int jt = f - (Rr == 0 ? 0 : (Rr == 1 ? 2 : (Rr == 2 ? 6 : 12)));
                const int r0 = 16 * Rr + gq, s0 = 8 * jt + 2 * tq;
#pragma unroll
                for (int hh = 0; hh < 2; ++hh) {
                    const int r = r0 + 8 * hh;
                    const float v0 = res[e][2 * hh], v1 = res[e][2 * hh + 1];
                    if (X == 0) {
                        sA[r * LDA + s0] = s0 < r ? v0 : 0.f;
                        sA[r * LDA + s0 + 1] = s0 + 1 < r ? v1 : 0.f;
                    } else {
                        st_bf16x2(sm + Y::PP, r * LDC + s0, s0 <= r ? v0 : 0.f, s0 + 1 <= r ? v1 : 0.f);
                    }
                }
            }
        }
        __syncthreads();
        // ------------------------------------------------ 4: Tinv = (I + A)^-1
        if (tid < 64) {
            const int Rb = tid >> 4, jc = tid & 15;
            float x[16];
#pragma unroll
            for (int r = 0; r < 16; ++r) {
                float acc = r == jc ? 1.f : 0.f;
#pragma unroll
                for (int s = 0; s < r; ++s) acc = fmaf(-sA[(16 * Rb + r) * LDA + 16 * Rb + s], x[s], acc);
                x[r] = acc;
            }
#pragma unroll
            for (int r = 0; r < 16; ++r) {
                sTi[(16 * Rb + r) * LDA + 16 * Rb + jc] = x[r];
                sTb[(16 * Rb + r) * LDC + 16 * Rb + jc] = __float2bfloat16_rn(x[r]);
            }
        }
        __syncthreads();
#pragma unroll 1
        for (int d = 1; d < 4; ++d) {
            const int nblk = 4 - d;
            for (int idx = tid; idx < nblk * 256; idx += NT) {
                const int blk = idx >> 8, Rb = d + blk, Sb = Rb - d, rho = (idx >> 4) & 15, c = idx & 15;
                float acc = 0.f;
                for (int m = Sb; m < Rb; ++m) {
#pragma unroll
                    for (int u = 0; u < 16; ++u)
                        acc = fmaf(sA[(16 * Rb + rho) * LDA + 16 * m + u], sTi[(16 * m + u) * LDA + 16 * Sb + c], acc);
                }
                sScr[blk * 256 + rho * 16 + c] = acc;
            }
            __syncthreads();
            for (int idx = tid; idx < nblk * 256; idx += NT) {
                const int blk = idx >> 8, Rb = d + blk, Sb = Rb - d, rho = (idx >> 4) & 15, c = idx & 15;
                float acc = 0.f;
#pragma unroll
                for (int u = 0; u < 16; ++u)
                    acc = fmaf(sTi[(16 * Rb + rho) * LDA + 16 * Rb + u], sScr[blk * 256 + u * 16 + c], acc);
                sTi[(16 * Rb + rho) * LDA + 16 * Sb + c] = -acc;
                sTb[(16 * Rb + rho) * LDC + 16 * Sb + c] = __float2bfloat16_rn(-acc);
            }
            __syncthreads();
        }
        // ------------------------------------------------ 5: -W = -Tinv Kg,  U~ = Tinv Vb
        {
#pragma unroll 1
            for (int Rr = 0; Rr < 4; ++Rr) {
                float a0[4] = {0.f, 0.f, 0.f, 0.f}, a1[4] = {0.f, 0.f, 0.f, 0.f};
                for (int ks = 0; ks <= Rr; ++ks) {
                    uint32_t af[4], b0, b1, b2, b3;
                    ldsm_x4(af[0], af[1], af[2], af[3], uTB + ((16 * Rr + (lane & 15)) * LDC + 16 * ks + (lane >> 4) * 8) * 2);
                    ldsm_x4_t(b0, b1, b2, b3,
                              uKG + ((16 * ks + (lane & 7) + ((lane >> 3) & 1) * 8) * LDK + 16 * warp + (lane >> 4) * 8) * 2);
                    mma_bf16(a0, af, b0, b1);
                    mma_bf16(a1, af, b2, b3);
                }
                const int r = 16 * Rr + gq, c = 16 * warp + 2 * tq;
                st_bf16x2(sm + Y::WN, r * LDK + c, -a0[0], -a0[1]);
                st_bf16x2(sm + Y::WN, (r + 8) * LDK + c, -a0[2], -a0[3]);
                st_bf16x2(sm + Y::WN, r * LDK + c + 8, -a1[0], -a1[1]);
                st_bf16x2(sm + Y::WN, (r + 8) * LDK + c + 8, -a1[2], -a1[3]);
            }
        }
        const int mu = warp >> 1, nb = (warp & 1) * NPW;   // this warp's U/O tiles
        float accU[NPW][4];
#pragma unroll
        for (int n = 0; n < NPW; ++n) accU[n][0] = accU[n][1] = accU[n][2] = accU[n][3] = 0.f;
        for (int ks = 0; ks <= mu; ++ks) {
            uint32_t af[4];
            ldsm_x4(af[0], af[1], af[2], af[3], uTB + ((16 * mu + (lane & 15)) * LDC + 16 * ks + (lane >> 4) * 8) * 2);
#pragma unroll
            for (int np = 0; np < NPW / 2; ++np) {
                uint32_t b0, b1, b2, b3;
                ldsm_x4_t(b0, b1, b2, b3,
                          uVB + ((16 * ks + (lane & 7) + ((lane >> 3) & 1) * 8) * LDW + (nb + 2 * np) * 8 + (lane >> 4) * 8) * 2);
                mma_bf16(accU[2 * np], af, b0, b1);
                mma_bf16(accU[2 * np + 1], af, b2, b3);
            }
        }
        __syncthreads();
        // ------------------------------------------------ 6a: U = U~ - W S
        const uint32_t uS = uSB + cur * DK * LDW * 2;
#pragma unroll
        for (int ks = 0; ks < DK / 16; ++ks) {
            uint32_t af[4];
            ldsm_x4(af[0], af[1], af[2], af[3], uWN + ((16 * mu + (lane & 15)) * LDK + 16 * ks + (lane >> 4) * 8) * 2);
#pragma unroll
            for (int np = 0; np < NPW / 2; ++np) {
                uint32_t b0, b1, b2, b3;
                ldsm_x4_t(b0, b1, b2, b3,
                          uS + ((16 * ks + (lane & 7) + ((lane >> 3) & 1) * 8) * LDW + (nb + 2 * np) * 8 + (lane >> 4) * 8) * 2);
                mma_bf16(accU[2 * np], af, b0, b1);
                mma_bf16(accU[2 * np + 1], af, b2, b3);
            }
        }
#pragma unroll
        for (int n = 0; n < NPW; ++n) {
            const int r = 16 * mu + gq, c = (nb + n) * 8 + 2 * tq;
            st_bf16x2(sm + Y::UU, r * LDW + c, accU[n][0], accU[n][1]);
            st_bf16x2(sm + Y::UU, (r + 8) * LDW + c, accU[n][2], accU[n][3]);
        }
        __syncthreads();
        // ------------------------------------------------ 6b: O = Qg S + P U
        {
            float accO[NPW][4];
#pragma unroll
            for (int n = 0; n < NPW; ++n) accO[n][0] = accO[n][1] = accO[n][2] = accO[n][3] = 0.f;
#pragma unroll
            for (int ks = 0; ks < DK / 16; ++ks) {
                uint32_t af[4];
                ldsm_x4(af[0], af[1], af[2], af[3], uQG + ((16 * mu + (lane & 15)) * LDK + 16 * ks + (lane >> 4) * 8) * 2);
#pragma unroll
                for (int np = 0; np < NPW / 2; ++np) {
                    uint32_t b0, b1, b2, b3;
                    ldsm_x4_t(b0, b1, b2, b3,
                              uS + ((16 * ks + (lane & 7) + ((lane >> 3) & 1) * 8) * LDW + (nb + 2 * np) * 8 + (lane >> 4) * 8) * 2);
                    mma_bf16(accO[2 * np], af, b0, b1);
                    mma_bf16(accO[2 * np + 1], af, b2, b3);
                }
            }
            for (int ks = 0; ks <= mu; ++ks) {
                uint32_t af[4];
                ldsm_x4(af[0], af[1], af[2], af[3], uPP + ((16 * mu + (lane & 15)) * LDC + 16 * ks + (lane >> 4) * 8) * 2);
#pragma unroll
                for (int np = 0; np < NPW / 2; ++np) {
                    uint32_t b0, b1, b2, b3;
                    ldsm_x4_t(b0, b1, b2, b3,
                              uUU + ((16 * ks + (lane & 7) + ((lane >> 3) & 1) * 8) * LDW + (nb + 2 * np) * 8 + (lane >> 4) * 8) * 2);
                    mma_bf16(accO[2 * np], af, b0, b1);
                    mma_bf16(accO[2 * np + 1], af, b2, b3);
                }
            }
#pragma unroll
            for (int n = 0; n < NPW; ++n) {
                const int r = 16 * mu + gq, c = (nb + n) * 8 + 2 * tq;
                if (r < L)
                    *reinterpret_cast<uint32_t *>(ob + (int64_t)(t0 + r) * p.o_st + c) = pack_bf16x2(accO[n][0], accO[n][1]);
                if (r + 8 < L)
                    *reinterpret_cast<uint32_t *>(ob + (int64_t)(t0 + r + 8) * p.o_st + c) = pack_bf16x2(accO[n][2], accO[n][3]);
            }
        }
        // ------------------------------------------------ 6c: S = e^gamma_C S + Kend^T U
        {
            const float d0 = sDec[16 * warp + gq], d1 = sDec[16 * warp + gq + 8];
#pragma unroll
            for (int n = 0; n < NS; ++n) {
                accS[n][0] *= d0; accS[n][1] *= d0; accS[n][2] *= d1; accS[n][3] *= d1;
            }
#pragma unroll
            for (int ks = 0; ks < C / 16; ++ks) {
                uint32_t af[4];
                const int mi = lane >> 3;
                ldsm_x4_t(af[0], af[1], af[2], af[3],
                          uKE + ((16 * ks + (lane & 7) + (mi >> 1) * 8) * LDK + 16 * warp + (mi & 1) * 8) * 2);
#pragma unroll
                for (int np = 0; np < NS / 2; ++np) {
                    uint32_t b0, b1, b2, b3;
                    ldsm_x4_t(b0, b1, b2, b3,
                              uUU + ((16 * ks + (lane & 7) + ((lane >> 3) & 1) * 8) * LDW + 16 * np + (lane >> 4) * 8) * 2);
                    mma_bf16(accS[2 * np], af, b0, b1);
                    mma_bf16(accS[2 * np + 1], af, b2, b3);
                }
            }
            const int nxt = cur ^ 1;
            char *sNext = sm + Y::SB + nxt * DK * LDW * 2;
#pragma unroll
            for (int n = 0; n < NS; ++n) {
                const int i0 = 16 * warp + gq, c = 8 * n + 2 * tq;
                st_bf16x2(sNext, i0 * LDW + c, accS[n][0], accS[n][1]);
                st_bf16x2(sNext, (i0 + 8) * LDW + c, accS[n][2], accS[n][3]);
            }
            cur = nxt;
        }
        __syncthreads();
    }
#pragma unroll
    for (int n = 0; n < NS; ++n) {
        const int i0 = 16 * warp + gq, c = 8 * n + 2 * tq;
        *reinterpret_cast<float2 *>(state + (size_t)i0 * p.dv + c) = make_float2(accS[n][0], accS[n][1]);
        *reinterpret_cast<float2 *>(state + (size_t)(i0 + 8) * p.dv + c) = make_float2(accS[n][2], accS[n][3]);
    }
}

template <int WS>
cgdr_status launch_ws(const TcParams &p, int B, cudaStream_t s) {
    const int smem = Lay<WS>::BYTES;
    if (cudaFuncSetAttribute(prefill_tc_kernel<WS>, cudaFuncAttributeMaxDynamicSharedMemorySize, smem) != cudaSuccess)
        return CGDR_ERR_CUDA;
    dim3 grid(p.dv / WS, p.Hv, B);
    prefill_tc_kernel<WS><<<grid, NT, smem, s>>>(p);
    return cudaGetLastError() == cudaSuccess ? CGDR_OK : CGDR_ERR_CUDA;
}

}  // namespace

bool prefill_tc_supported(const cgdr_args &a) {
    return a.dtype == CGDR_BF16 && a.dk == 128 && chunk_of(a) == 64 && (a.dv % 32) == 0;
}

size_t prefill_tc_workspace(const cgdr_args &) { return 0; }

cgdr_status launch_prefill_tc(const cgdr_args &a, void *, size_t, cudaStream_t s) {
    TcParams p;
    p.T = a.T; p.Hk = a.Hk; p.Hv = a.Hv; p.dv = a.dv; p.l2norm = a.l2norm_qk != 0; p.gate = a.gate;
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
    p.state = a.state;
    p.o = static_cast<__nv_bfloat16 *>(a.o);
    p.o_sb = a.o_sb; p.o_st = a.o_st; p.o_sh = a.o_sh;
    int dev = 0, sms = 148;
    if (cudaGetDevice(&dev) == cudaSuccess) cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    // Narrow slabs give more CTAs when there are few (batch, head) chains; wide
    // slabs avoid repeating the per-chunk preparation when there are many.
    const long ctas32 = (long)a.B * a.Hv * (a.dv / 32);
    if (a.dv % 64 != 0 || ctas32 <= 2L * sms) return launch_ws<32>(p, a.B, s);
    return launch_ws<64>(p, a.B, s);
}

}  // namespace cgdr
