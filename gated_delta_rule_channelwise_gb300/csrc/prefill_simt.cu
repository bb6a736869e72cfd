// Chunked prefill on the CUDA cores, fp32 throughout.
//
// The chunkwise WY/UT form of "Add parallel chunked prefill for channelwise
// gated delta rule" (executorch PR #21061, Summary), written for clarity
// rather than speed: it serves fp32 inputs (where bf16 tensor-core operands
// would miss the fp32 tolerance) and shapes the tensor-core kernel does not
// cover.  One CTA owns one (batch, v-head, 32-column slab of dv); columns of
// the state are independent given q, k, g and beta, so slabs never exchange
// data.  Per chunk of C tokens (rows >= L of a ragged last chunk are
// identity tokens: q = k = v = 0, g = 0, beta = 0):
//   gamma_r = sum_{s<=r} g_s                       log-decay prefix per channel
//   A_rs = beta_r sum_i k_ri k_si e^(gamma_ri - gamma_si)   s < r
//   P_rs =        sum_i q_ri k_si e^(gamma_ri - gamma_si)   s <= r
//   Tm   = (I + A)^-1 Diag(beta)                   forward substitution
//   W    = Tm (K e^gamma),   U = Tm V - W S        WY pseudo-keys / -values
//   O    = (Q e^gamma) S + P U
//   S    = e^gamma_C S + (K e^(gamma_C - gamma))^T U
// Pairwise decays are exponentials of differences, so nothing overflows.
#include "cgdr_internal.cuh"

namespace cgdr {
namespace {

constexpr int SIMT_WS = 32;     // dv columns per CTA
constexpr int SIMT_NT = 256;

struct PrefillParams {
    int T, Hk, Hv, dv, l2norm, gate, o_f32;
    float q_scale, eps;
    const void *q, *k, *v;
    int64_t q_sb, q_st, q_sh, k_sb, k_st, k_sh, v_sb, v_st, v_sh;
    const float *g, *beta;
    int64_t g_sb, g_st, g_sh, beta_sb, beta_st, beta_sh;
    const void *ga, *gb;
    int64_t a_sb, a_st, a_sh, b_sb, b_st, b_sh;
    const float *A_log, *dt_bias;
    float *state;
    void *o;
    int64_t o_sb, o_st, o_sh;
    int *status;                 // the caller's optional status word (debug-build index checks)
    Extents ext;                 // footprints for the index checks of a debug build
};

template <int DK, int C>
struct SimtSmem {
    static constexpr int CD = C * DK, CC = C * (C + 1), CW = C * SIMT_WS;
    static constexpr int floats = 4 * CD + 3 * CC + 2 * CW + DK * SIMT_WS + 3 * C + DK;
    static constexpr size_t bytes = sizeof(float) * floats;
};

template <int DK, int C, typename T>
__global__ void __launch_bounds__(SIMT_NT) prefill_simt_kernel(const PrefillParams p) {
    using SM = SimtSmem<DK, C>;
    constexpr int LC = C + 1;
    constexpr int WS = SIMT_WS;
    extern __shared__ float smem[];
    float *sQ = smem;                 // q normalised, later q e^gamma
    float *sK = sQ + SM::CD;          // k normalised, later k e^(gamma_C - gamma)
    float *sG = sK + SM::CD;          // gamma, later W
    float *sKg = sG + SM::CD;         // k e^gamma
    float *sA = sKg + SM::CD;
    float *sP = sA + SM::CC;
    float *sT = sP + SM::CC;
    float *sV = sT + SM::CC;          // v slab, later U
    float *sO = sV + SM::CW;          // U~ (pseudo-values)
    float *sS = sO + SM::CW;          // state slab [DK][WS]
    float *sBeta = sS + DK * WS;
    float *sRq = sBeta + C;
    float *sRk = sRq + C;
    float *sDecay = sRk + C;

    const int slab = blockIdx.x, h = blockIdx.y, b = blockIdx.z;
    const int hk = h / (p.Hv / p.Hk);
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int col0 = slab * WS;
    const int64_t sbase_e = ((int64_t)b * p.Hv + h) * DK * p.dv;
    float *state = p.state + sbase_e;
    int *const st0 = p.status;

    for (int idx = tid; idx < DK * WS; idx += SIMT_NT) {
        const int i = idx / WS, j = idx % WS;
        const int64_t e = (int64_t)i * p.dv + col0 + j;
        sS[idx] = in_bounds(sbase_e + e, p.ext.state, st0, nullptr) ? state[e] : 0.f;
    }

    const int64_t qo = b * p.q_sb + hk * p.q_sh, ko = b * p.k_sb + hk * p.k_sh, vo = b * p.v_sb + h * p.v_sh + col0;
    const T *qb = static_cast<const T *>(p.q) + qo;
    const T *kb = static_cast<const T *>(p.k) + ko;
    const T *vb = static_cast<const T *>(p.v) + vo;
    const int64_t obase = b * p.o_sb + h * p.o_sh + col0;

    for (int t0 = 0; t0 < p.T; t0 += C) {
        const int L = min(C, p.T - t0);
        __syncthreads();
        // ---- load the chunk (identity tokens past the end)
        for (int idx = tid; idx < C * DK; idx += SIMT_NT) {
            const int r = idx / DK, i = idx % DK;
            float qv = 0.f, kv = 0.f, gv = 0.f;
            if (r < L) {
                const int64_t t = t0 + r;
                if (in_bounds(qo + t * p.q_st + i, p.ext.q, st0, nullptr)) qv = Cvt<T>::to_f(qb[t * p.q_st + i]);
                if (in_bounds(ko + t * p.k_st + i, p.ext.k, st0, nullptr)) kv = Cvt<T>::to_f(kb[t * p.k_st + i]);
                if (p.gate == CGDR_GATE_CHANNEL) {
                    const int64_t e = b * p.g_sb + t * p.g_st + h * p.g_sh + i;
                    if (in_bounds(e, p.ext.g, st0, nullptr)) gv = p.g[e];
                } else {
                    const int64_t e = b * p.a_sb + t * p.a_st + h * p.a_sh;
                    if (in_bounds(e, p.ext.a, st0, nullptr) && in_bounds(h, p.ext.A_log, st0, nullptr) &&
                        in_bounds(h, p.ext.dt_bias, st0, nullptr))
                        gv = gdn_gate(p.A_log[h], Cvt<T>::to_f(static_cast<const T *>(p.ga)[e]), p.dt_bias[h]);
                }
            }
            sQ[idx] = qv; sK[idx] = kv; sG[idx] = gv;
        }
        for (int idx = tid; idx < C * WS; idx += SIMT_NT) {
            const int r = idx / WS, j = idx % WS;
            const int64_t e = (int64_t)(t0 + r) * p.v_st + j;
            sV[idx] = r < L && in_bounds(vo + e, p.ext.v, st0, nullptr) ? Cvt<T>::to_f(vb[e]) : 0.f;
        }
        for (int r = tid; r < C; r += SIMT_NT) {
            float be = 0.f;
            if (r < L) {
                const int64_t t = t0 + r;
                if (p.gate == CGDR_GATE_CHANNEL) {
                    const int64_t e = b * p.beta_sb + t * p.beta_st + h * p.beta_sh;
                    if (in_bounds(e, p.ext.beta, st0, nullptr)) be = p.beta[e];
                } else {
                    const int64_t e = b * p.b_sb + t * p.b_st + h * p.b_sh;
                    if (in_bounds(e, p.ext.b, st0, nullptr))
                        be = sigmoid_f(Cvt<T>::to_f(static_cast<const T *>(p.gb)[e]));
                }
            }
            sBeta[r] = be;
        }
        __syncthreads();
        // ---- row norms (a warp per row) and the log-decay prefix (a thread per channel)
        for (int r = warp; r < C; r += SIMT_NT / 32) {
            float sq = 0.f, sk = 0.f;
            for (int i = lane; i < DK; i += 32) {
                sq += sQ[r * DK + i] * sQ[r * DK + i];
                sk += sK[r * DK + i] * sK[r * DK + i];
            }
            sq = warp_sum(sq);
            sk = warp_sum(sk);
            if (lane == 0) {
                sRq[r] = (p.l2norm ? rsqrtf(sq + p.eps) : 1.f) * p.q_scale;
                sRk[r] = p.l2norm ? rsqrtf(sk + p.eps) : 1.f;
            }
        }
        for (int i = tid; i < DK; i += SIMT_NT) {
            float acc = 0.f;
            for (int r = 0; r < C; ++r) { acc += sG[r * DK + i]; sG[r * DK + i] = acc; }
        }
        __syncthreads();
        for (int idx = tid; idx < C * DK; idx += SIMT_NT) {
            const int r = idx / DK;
            sQ[idx] *= sRq[r];
            sK[idx] *= sRk[r];
        }
        __syncthreads();
        // ---- causal terms A (strictly lower, beta-scaled rows) and P (lower)
        for (int idx = tid; idx < C * C; idx += SIMT_NT) {
            const int r = idx / C, s = idx % C;
            float sa = 0.f, sp = 0.f;
            if (s <= r) {
                for (int i = 0; i < DK; ++i) {
                    const float d = expf(sG[r * DK + i] - sG[s * DK + i]);
                    const float ks = sK[s * DK + i] * d;
                    sa = fmaf(sK[r * DK + i], ks, sa);
                    sp = fmaf(sQ[r * DK + i], ks, sp);
                }
            }
            sA[r * LC + s] = s < r ? sBeta[r] * sa : 0.f;
            sP[r * LC + s] = sp;
        }
        __syncthreads();
        // ---- decay-scaled operands
        for (int idx = tid; idx < C * DK; idx += SIMT_NT) {
            const int i = idx % DK;
            const float gr = sG[idx], gc = sG[(C - 1) * DK + i];
            const float kv = sK[idx];
            sKg[idx] = kv * expf(gr);
            sQ[idx] *= expf(gr);
            sK[idx] = kv * expf(gc - gr);
        }
        for (int i = tid; i < DK; i += SIMT_NT) sDecay[i] = expf(sG[(C - 1) * DK + i]);
        // ---- Tm = (I + A)^-1 Diag(beta), one row at a time
        for (int r = 0; r < C; ++r) {
            for (int j = tid; j < C; j += SIMT_NT) {
                float acc = 0.f;
                if (j <= r) {
                    acc = j == r ? sBeta[r] : 0.f;
                    for (int s = j; s < r; ++s) acc -= sA[r * LC + s] * sT[s * LC + j];
                }
                sT[r * LC + j] = acc;
            }
            __syncthreads();
        }
        // ---- W = Tm (K e^gamma) into sG;  U~ = Tm V into sO
        for (int idx = tid; idx < C * DK; idx += SIMT_NT) {
            const int r = idx / DK, i = idx % DK;
            float acc = 0.f;
            for (int s = 0; s <= r; ++s) acc = fmaf(sT[r * LC + s], sKg[s * DK + i], acc);
            sG[idx] = acc;
        }
        for (int idx = tid; idx < C * WS; idx += SIMT_NT) {
            const int r = idx / WS, j = idx % WS;
            float acc = 0.f;
            for (int s = 0; s <= r; ++s) acc = fmaf(sT[r * LC + s], sV[s * WS + j], acc);
            sO[idx] = acc;
        }
        __syncthreads();
        // ---- U = U~ - W S  (into sV)
        for (int idx = tid; idx < C * WS; idx += SIMT_NT) {
            const int r = idx / WS, j = idx % WS;
            float acc = sO[idx];
            for (int i = 0; i < DK; ++i) acc = fmaf(-sG[r * DK + i], sS[i * WS + j], acc);
            sV[idx] = acc;
        }
        __syncthreads();
        // ---- O = (Q e^gamma) S + P U
        for (int idx = tid; idx < C * WS; idx += SIMT_NT) {
            const int r = idx / WS, j = idx % WS;
            if (r >= L) continue;
            float acc = 0.f;
            for (int i = 0; i < DK; ++i) acc = fmaf(sQ[r * DK + i], sS[i * WS + j], acc);
            for (int s = 0; s <= r; ++s) acc = fmaf(sP[r * LC + s], sV[s * WS + j], acc);
            const int64_t off = obase + (int64_t)(t0 + r) * p.o_st + j;
            if (!in_bounds(off, p.ext.o, st0, nullptr)) continue;
            if (p.o_f32)
                static_cast<float *>(p.o)[off] = acc;
            else
                static_cast<__nv_bfloat16 *>(p.o)[off] = __float2bfloat16_rn(acc);
        }
        __syncthreads();
        // ---- S = e^gamma_C S + (K e^(gamma_C - gamma))^T U
        for (int idx = tid; idx < DK * WS; idx += SIMT_NT) {
            const int i = idx / WS, j = idx % WS;
            float acc = sDecay[i] * sS[idx];
            for (int r = 0; r < C; ++r) acc = fmaf(sK[r * DK + i], sV[r * WS + j], acc);
            sS[idx] = acc;
        }
    }
    __syncthreads();
    for (int idx = tid; idx < DK * WS; idx += SIMT_NT) {
        const int i = idx / WS, j = idx % WS;
        const int64_t e = (int64_t)i * p.dv + col0 + j;
        if (in_bounds(sbase_e + e, p.ext.state, st0, nullptr)) state[e] = sS[idx];
    }
}

template <int DK, int C, typename T>
cgdr_status launch_t(const PrefillParams &p, int B, cudaStream_t s) {
    static SmemOnce smem_once;
    const size_t smem = SimtSmem<DK, C>::bytes;
    if (!smem_limit_once(smem_once, reinterpret_cast<const void *>(prefill_simt_kernel<DK, C, T>), (int)smem))
        return CGDR_ERR_CUDA;
    dim3 grid(p.dv / SIMT_WS, p.Hv, B);
    prefill_simt_kernel<DK, C, T><<<grid, SIMT_NT, smem, s>>>(p);
    return cudaGetLastError() == cudaSuccess ? CGDR_OK : CGDR_ERR_CUDA;
}

template <typename T>
cgdr_status launch_dtype(const PrefillParams &p, int B, int dk, int C, cudaStream_t s) {
#define CGDR_SIMT_CASE(K, CC) \
    if (dk == K && C == CC) return launch_t<K, CC, T>(p, B, s);
    CGDR_SIMT_CASE(32, 16) CGDR_SIMT_CASE(32, 32) CGDR_SIMT_CASE(32, 64)
    CGDR_SIMT_CASE(64, 16) CGDR_SIMT_CASE(64, 32) CGDR_SIMT_CASE(64, 64)
    CGDR_SIMT_CASE(128, 16) CGDR_SIMT_CASE(128, 32) CGDR_SIMT_CASE(128, 64)
#undef CGDR_SIMT_CASE
    return CGDR_ERR_UNSUPPORTED;
}

}  // namespace

cgdr_status launch_prefill_simt(const cgdr_args &a, cudaStream_t s) {
    PrefillParams p;
    p.T = a.T; p.Hk = a.Hk; p.Hv = a.Hv; p.dv = a.dv; p.l2norm = a.l2norm_qk != 0; p.gate = a.gate;
    p.o_f32 = a.o_dtype == CGDR_F32;
    p.q_scale = qscale_of(a); p.eps = eps_of(a);
    p.q = a.q; p.k = a.k; p.v = a.v;
    p.q_sb = a.q_sb; p.q_st = a.q_st; p.q_sh = a.q_sh;
    p.k_sb = a.k_sb; p.k_st = a.k_st; p.k_sh = a.k_sh;
    p.v_sb = a.v_sb; p.v_st = a.v_st; p.v_sh = a.v_sh;
    p.g = a.g; p.beta = a.beta;
    p.g_sb = a.g_sb; p.g_st = a.g_st; p.g_sh = a.g_sh;
    p.beta_sb = a.beta_sb; p.beta_st = a.beta_st; p.beta_sh = a.beta_sh;
    p.ga = a.a; p.gb = a.b;
    p.a_sb = a.a_sb; p.a_st = a.a_st; p.a_sh = a.a_sh;
    p.b_sb = a.b_sb; p.b_st = a.b_st; p.b_sh = a.b_sh;
    p.A_log = a.A_log; p.dt_bias = a.dt_bias;
    p.state = a.state; p.o = a.o; p.o_sb = a.o_sb; p.o_st = a.o_st; p.o_sh = a.o_sh;
    p.status = a.status;
    p.ext = extents_of(a, true, 0);
    const int C = chunk_of(a);
    if (a.dtype == CGDR_BF16) return launch_dtype<__nv_bfloat16>(p, a.B, a.dk, C, s);
    return launch_dtype<float>(p, a.B, a.dk, C, s);
}

}  // namespace cgdr
