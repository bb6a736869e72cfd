// Decode (T = 1): each (batch, v-head) state tile is read once, updated in
// registers and written once.
//
// "Add fused GatedDeltaNet decode Triton kernel" (executorch PR #18865) fuses
// the Q/K/V split, the q/k L2 norm, the head repeat, the gating and the state
// update into one kernel; "Two-pass optimization for channelwise gated delta
// rule kernel" (executorch PR #21020) brings the state traversals per token
// down to two.  Here the split is pointer arithmetic (strides into the packed
// row), and the two traversals are register sweeps over a tile that is read
// from HBM once and written once:
//   sweep 1:  vh = S^T (alpha * kn)            (decay folded into the key)
//   sweep 2:  S  = alpha * S + kn u^T,  u = beta (v - vh);  o += S^T qn
// The same kernel steps through up to eight tokens per call (prefill with a
// small T: the token recurrence itself, the route "T == 1 keeps the token
// recurrence" of "Add parallel chunked prefill for channelwise gated delta
// rule" (Summary) extended to a few tokens): the tile stays in registers from
// token to token and is still read once and written once.
// Layout: a warp instruction covers RW consecutive rows of the dk x dv tile
// with 16-byte (float4) loads, so every access is a full 128-byte line.  The
// reduction over dk runs in registers, then across the row-lanes of a warp
// with shuffles, then across warps through a small shared array.
#include "cgdr_internal.cuh"

namespace cgdr {
namespace {

struct DecodeParams {
    int Hk, Hv, l2norm, gate, o_f32;
    int ntok;                                         // tokens per call (1 for decode, up to kRecurrentMaxT)
    float q_scale, eps;
    const void *q, *k, *v;
    int64_t q_sb, q_sh, q_st, k_sb, k_sh, k_st, v_sb, v_sh, v_st;
    const float *g, *beta;
    int64_t g_sb, g_sh, g_st, beta_sb, beta_sh, beta_st;
    const void *ga, *gb;
    int64_t a_sb, a_sh, a_st, b_sb, b_sh, b_st;
    const float *A_log, *dt_bias;
    float *state;
    void *o;
    int64_t o_sb, o_sh, o_st;
    int *status;                                      // optional: CGDR_ERR_TIMEOUT if a wait gave up
    uint32_t polls;                                   // polls of the main-loop tile waits
    int inject;                                       // test hook: the first tile wait targets a dead barrier
    Extents ext;                                      // footprints for the index checks of a debug build
};

template <int DK, int DV>
struct DecodeShape {
    static constexpr int CL = DV / 4;                 // lanes across one row (float4 each)
    static constexpr int RW = 32 / CL;                // rows per warp instruction
    static constexpr int NT_RAW = DK * DV / 64;       // 16 float4 per thread
    static constexpr int NT = NT_RAW < 32 ? 32 : (NT_RAW > 256 ? 256 : NT_RAW);
    static constexpr int NW = NT / 32;
    static constexpr int RPT = DK / (NW * RW);        // rows per thread
    static_assert(RPT * NW * RW == DK, "tile does not split evenly");
};

__device__ __forceinline__ void st_stream(float *p, float4 v) { __stcs(reinterpret_cast<float4 *>(p), v); }

template <typename T>
__device__ __forceinline__ float4 load4(const T *p);
template <>
__device__ __forceinline__ float4 load4<float>(const float *p) { return *reinterpret_cast<const float4 *>(p); }
template <>
__device__ __forceinline__ float4 load4<__nv_bfloat16>(const __nv_bfloat16 *p) {
    uint2 raw = *reinterpret_cast<const uint2 *>(p);
    __nv_bfloat162 lo = *reinterpret_cast<__nv_bfloat162 *>(&raw.x);
    __nv_bfloat162 hi = *reinterpret_cast<__nv_bfloat162 *>(&raw.y);
    float2 a = __bfloat1622float2(lo), b = __bfloat1622float2(hi);
    return make_float4(a.x, a.y, b.x, b.y);
}

template <typename T>
__device__ __forceinline__ void store4(T *p, float4 v);
template <>
__device__ __forceinline__ void store4<float>(float *p, float4 v) { *reinterpret_cast<float4 *>(p) = v; }
template <>
__device__ __forceinline__ void store4<__nv_bfloat16>(__nv_bfloat16 *p, float4 v) {
    uint2 raw;
    raw.x = pack_bf16x2(v.x, v.y);
    raw.y = pack_bf16x2(v.z, v.w);
    *reinterpret_cast<uint2 *>(p) = raw;
}

// Persistent form: one CTA per SM walks its (batch, head) units; state tiles
// stream through a ring of NS shared-memory stages filled by TMA bulk copies
// (cp.async.bulk, completion on an mbarrier), the small per-unit rows (q, k,
// v, g) by cp.async, so the next tiles are already in flight while the
// current one is updated and written back with 16-byte streaming stores.
template <int DK, int DV, typename T, int NTOK>
struct PipeShape {
    static constexpr int NS = NTOK == 1 ? 3 : 2;
    static constexpr int TILE = DK * DV * 4;
    static constexpr int ROWQ = ((DK * (int)sizeof(T) + 15) / 16) * 16;
    static constexpr int ROWV = ((DV * (int)sizeof(T) + 15) / 16) * 16;
    static constexpr int ROWG = DK * 4;
    static constexpr int SMALL1 = 2 * ROWQ + ROWV + ROWG;      // one token's q, k, v, g rows
    static constexpr int SMALL = NTOK * SMALL1;
    static constexpr int STAGE = ((TILE + SMALL + 127) / 128) * 128;
    static constexpr int BYTES = NS * STAGE + 64 + 128;   // stages, mbarriers (NS + 1 <= 8), alignment slack
};

__device__ __forceinline__ void bulk_g2s(uint32_t dst, const void *src, uint32_t bytes, uint32_t mbar) {
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(mbar), "r"(bytes) : "memory");
    asm volatile("cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];"
                 ::"r"(dst), "l"(src), "r"(bytes), "r"(mbar) : "memory");
}
__device__ __forceinline__ bool mbar_wait_parity(uint32_t mbar, uint32_t parity, uint32_t max_iters) {
    for (uint32_t it = 0; it < max_iters; ++it) {
        uint32_t done;
        asm volatile("{\n.reg .pred p;\nmbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\nselp.u32 %0, 1, 0, p;\n}\n"
                     : "=r"(done) : "r"(mbar), "r"(parity) : "memory");
        if (done) return true;
    }
    return false;
}
template <int N>
__device__ __forceinline__ void cp_async_wait_groups() { asm volatile("cp.async.wait_group %0;" ::"n"(N) : "memory"); }

template <int DK, int DV, typename T, int NTOK>
__global__ void __launch_bounds__(DecodeShape<DK, DV>::NT, 1) decode_kernel(const DecodeParams p, int units) {
    using Sh = DecodeShape<DK, DV>;
    using Ps = PipeShape<DK, DV, T, NTOK>;
    constexpr int CL = Sh::CL, RW = Sh::RW, NW = Sh::NW, RPT = Sh::RPT, NT = Sh::NT, NS = Ps::NS;
    static_assert(NTOK <= NT, "one thread per token holds its scalars");
    const int ntok = NTOK == 1 ? 1 : p.ntok;
    constexpr uint32_t kSpin = kDefaultPolls;         // drain waits always use the full limit
    extern __shared__ __align__(128) char dsm_raw[];
    char *dsm = dsm_raw + ((128 - (smem_u32(dsm_raw) & 127)) & 127);
    const uint32_t sb = smem_u32(dsm);
    const uint32_t mbar0 = sb + NS * Ps::STAGE;
    __shared__ float s_kn[DK], s_qn[DK], s_alpha[DK];
    __shared__ float4 s_red[NW][CL];
    __shared__ float s_beta;

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int c = lane % CL, r = lane / CL;
    const int G = gridDim.x;

    // mbar0 + 8 * NS: a barrier nothing ever arrives on (the target of the injected failure)
    if (tid == 0) {
        for (int st = 0; st <= NS; ++st) asm volatile("mbarrier.init.shared::cta.b64 [%0], 1;" ::"r"(mbar0 + 8 * st));
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    }
    __syncthreads();

    // Issue the copies of unit u into stage st (every thread commits one cp.async group).
    auto issue = [&](int u, int st) {
        if (u < units) {
            const int b = u / p.Hv, h = u % p.Hv, hk = h / (p.Hv / p.Hk);
            const uint32_t base = sb + st * Ps::STAGE;
            if (tid == 0) {
                if (range_in_bounds((int64_t)u * DK * DV, DK * DV, p.ext.state, p.status, nullptr))
                    bulk_g2s(base, p.state + (size_t)u * DK * DV, Ps::TILE, mbar0 + 8 * st);
                else   // (debug build) a tile outside the state: no copy, the stage's phase still completes
                    asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(mbar0 + 8 * st) : "memory");
            }
            constexpr int nq = Ps::ROWQ / 16, nv = Ps::ROWV / 16, ng = Ps::ROWG / 16;
            constexpr int eq = 16 / (int)sizeof(T);                  // elements per 16-byte piece (q, k, v)
            const int per = 2 * nq + nv + (p.gate == CGDR_GATE_CHANNEL ? ng : 0);   // 16-byte pieces per token
            for (int x = tid; x < ntok * per; x += NT) {
                const int t = x / per, y = x - t * per;
                const uint32_t sm0 = base + Ps::TILE + t * Ps::SMALL1;
                if (y < nq) {
                    const int64_t e = b * p.q_sb + t * p.q_st + hk * p.q_sh + eq * y;
                    cp_async16(sm0 + 16 * y, static_cast<const T *>(p.q) + e,
                               range_in_bounds(e, eq, p.ext.q, p.status, nullptr));
                } else if (y < 2 * nq) {
                    const int64_t e = b * p.k_sb + t * p.k_st + hk * p.k_sh + eq * (y - nq);
                    cp_async16(sm0 + Ps::ROWQ + 16 * (y - nq), static_cast<const T *>(p.k) + e,
                               range_in_bounds(e, eq, p.ext.k, p.status, nullptr));
                } else if (y < 2 * nq + nv) {
                    const int64_t e = b * p.v_sb + t * p.v_st + h * p.v_sh + eq * (y - 2 * nq);
                    cp_async16(sm0 + 2 * Ps::ROWQ + 16 * (y - 2 * nq), static_cast<const T *>(p.v) + e,
                               range_in_bounds(e, eq, p.ext.v, p.status, nullptr));
                } else {
                    const int64_t e = b * p.g_sb + t * p.g_st + h * p.g_sh + 4 * (y - 2 * nq - nv);
                    cp_async16(sm0 + 2 * Ps::ROWQ + Ps::ROWV + 16 * (y - 2 * nq - nv), p.g + e,
                               range_in_bounds(e, 4, p.ext.g, p.status, nullptr));
                }
            }
        }
        cp_async_commit();
    };
    // Per-unit scalars (beta, or a and b of the scalar gate), kept two units ahead in registers:
    // thread t holds those of token t.
    auto scalars = [&](int u) -> float2 {
        float2 x = make_float2(0.f, 0.f);
        if (tid < ntok && u < units) {
            const int b = u / p.Hv, h = u % p.Hv, t = tid;
            if (p.gate == CGDR_GATE_CHANNEL) {
                const int64_t e = b * p.beta_sb + t * p.beta_st + h * p.beta_sh;
                if (in_bounds(e, p.ext.beta, p.status, nullptr)) x.x = p.beta[e];
            } else {
                const int64_t ea = b * p.a_sb + t * p.a_st + h * p.a_sh, eb = b * p.b_sb + t * p.b_st + h * p.b_sh;
                if (in_bounds(ea, p.ext.a, p.status, nullptr)) x.x = Cvt<T>::to_f(static_cast<const T *>(p.ga)[ea]);
                if (in_bounds(eb, p.ext.b, p.status, nullptr)) x.y = Cvt<T>::to_f(static_cast<const T *>(p.gb)[eb]);
            }
        }
        return x;
    };

    const int u0 = blockIdx.x;
    for (int st = 0; st < NS - 1; ++st) issue(u0 + st * G, st);
    float2 sc0 = scalars(u0), sc1 = scalars(u0 + G);
    bool failed = false;
    int kf = 0;                                       // iteration whose tile wait gave up

    for (int k = 0;; ++k) {
        const int u = u0 + k * G;
        if (u >= units) break;
        const int st = k % NS;
        issue(u0 + (k + NS - 1) * G, (k + NS - 1) % NS);
        const float2 sc = sc0;
        sc0 = sc1;
        sc1 = scalars(u0 + (k + 2) * G);

        // thread 0 polls the tile's barrier; the other warps sleep at the barrier below, which
        // carries the outcome and orders the tile's bytes before their reads
        const bool dead = p.inject && k == 0;
        const bool got = tid != 0 || mbar_wait_parity(dead ? mbar0 + 8 * NS : mbar0 + 8 * st,
                                                      dead ? 0u : (uint32_t)((k / NS) & 1), p.polls);
        cp_async_wait_groups<NS - 1>();
        const int b = u / p.Hv, h = u % p.Hv;
        if (__syncthreads_or(!got)) {
            failed = true;
            kf = k;
            break;
        }
        const char *stage = dsm + st * Ps::STAGE;
        const float *S = reinterpret_cast<const float *>(stage);

        float4 s[RPT];
#pragma unroll
        for (int ii = 0; ii < RPT; ++ii) {
            const int row = (warp * RPT + ii) * RW + r;
            s[ii] = *reinterpret_cast<const float4 *>(S + row * DV + 4 * c);
        }
        float *Sg = p.state + (size_t)u * DK * DV;
        for (int t = 0; t < ntok; ++t) {
            const char *rows = stage + Ps::TILE + t * Ps::SMALL1;
            const T *sq = reinterpret_cast<const T *>(rows);
            const T *sk = reinterpret_cast<const T *>(rows + Ps::ROWQ);
            const T *sv = reinterpret_cast<const T *>(rows + 2 * Ps::ROWQ);
            const float *sg = reinterpret_cast<const float *>(rows + 2 * Ps::ROWQ + Ps::ROWV);
            const float4 vv = load4<T>(sv + 4 * c);
            // q/k L2 norm (a warp each), decay alpha, beta
            for (int which = warp; which < 2; which += NW) {
                const T *x = which == 0 ? sq : sk;
                float vals[DK / 32];
                float ss = 0.f;
#pragma unroll
                for (int j = 0; j < DK / 32; ++j) {
                    vals[j] = Cvt<T>::to_f(x[lane + 32 * j]);
                    ss += vals[j] * vals[j];
                }
                ss = warp_sum(ss);
                float scale = p.l2norm ? rsqrtf(ss + p.eps) : 1.f;
                if (which == 0) scale *= p.q_scale;
                float *dst = which == 0 ? s_qn : s_kn;
#pragma unroll
                for (int j = 0; j < DK / 32; ++j) dst[lane + 32 * j] = vals[j] * scale;
            }
            if (p.gate == CGDR_GATE_CHANNEL) {
                for (int i = tid; i < DK; i += NT) s_alpha[i] = expf(sg[i]);
                if (tid == t) s_beta = sc.x;
            } else {
                if (tid == t) {
                    const bool hin = in_bounds(h, p.ext.A_log, p.status, nullptr) && in_bounds(h, p.ext.dt_bias, p.status, nullptr);
                    s_alpha[0] = expf(gdn_gate(hin ? p.A_log[h] : 0.f, sc.x, hin ? p.dt_bias[h] : 0.f));
                    s_beta = sigmoid_f(sc.y);
                }
                __syncthreads();
                const float al = s_alpha[0];
                __syncthreads();
                for (int i = tid; i < DK; i += NT) s_alpha[i] = al;
            }
            __syncthreads();

            // sweep 1: vh = S^T (alpha * kn)
            float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
            for (int ii = 0; ii < RPT; ++ii) {
                const int row = (warp * RPT + ii) * RW + r;
                const float ak = s_alpha[row] * s_kn[row];
                acc.x = fmaf(ak, s[ii].x, acc.x);
                acc.y = fmaf(ak, s[ii].y, acc.y);
                acc.z = fmaf(ak, s[ii].z, acc.z);
                acc.w = fmaf(ak, s[ii].w, acc.w);
            }
#pragma unroll
            for (int off = CL; off < 32; off <<= 1) {
                acc.x += __shfl_xor_sync(0xffffffffu, acc.x, off);
                acc.y += __shfl_xor_sync(0xffffffffu, acc.y, off);
                acc.z += __shfl_xor_sync(0xffffffffu, acc.z, off);
                acc.w += __shfl_xor_sync(0xffffffffu, acc.w, off);
            }
            if (r == 0) s_red[warp][c] = acc;
            __syncthreads();
            float4 vh = s_red[0][c];
#pragma unroll
            for (int w = 1; w < NW; ++w) {
                const float4 tt = s_red[w][c];
                vh.x += tt.x; vh.y += tt.y; vh.z += tt.z; vh.w += tt.w;
            }
            const float beta = s_beta;
            const float4 uu = make_float4(beta * (vv.x - vh.x), beta * (vv.y - vh.y), beta * (vv.z - vh.z),
                                          beta * (vv.w - vh.w));
            __syncthreads();  // s_red is reused below

            // sweep 2: decay + rank-one write, o accumulated; the tile is stored once, after the last token
            const bool last = t == ntok - 1;
            float4 o = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
            for (int ii = 0; ii < RPT; ++ii) {
                const int row = (warp * RPT + ii) * RW + r;
                const float al = s_alpha[row], kn = s_kn[row], qn = s_qn[row];
                float4 x = s[ii];
                x.x = fmaf(al, x.x, kn * uu.x);
                x.y = fmaf(al, x.y, kn * uu.y);
                x.z = fmaf(al, x.z, kn * uu.z);
                x.w = fmaf(al, x.w, kn * uu.w);
                o.x = fmaf(qn, x.x, o.x);
                o.y = fmaf(qn, x.y, o.y);
                o.z = fmaf(qn, x.z, o.z);
                o.w = fmaf(qn, x.w, o.w);
                s[ii] = x;
                if (last && range_in_bounds((int64_t)u * DK * DV + row * DV + 4 * c, 4, p.ext.state, p.status, nullptr))
                    st_stream(Sg + (size_t)row * DV + 4 * c, x);
            }
#pragma unroll
            for (int off = CL; off < 32; off <<= 1) {
                o.x += __shfl_xor_sync(0xffffffffu, o.x, off);
                o.y += __shfl_xor_sync(0xffffffffu, o.y, off);
                o.z += __shfl_xor_sync(0xffffffffu, o.z, off);
                o.w += __shfl_xor_sync(0xffffffffu, o.w, off);
            }
            if (r == 0) s_red[warp][c] = o;
            __syncthreads();
            if (warp == 0 && r == 0) {
                float4 tt = s_red[0][c];
#pragma unroll
                for (int w = 1; w < NW; ++w) {
                    const float4 y = s_red[w][c];
                    tt.x += y.x; tt.y += y.y; tt.z += y.z; tt.w += y.w;
                }
                const int64_t off = b * p.o_sb + t * p.o_st + h * p.o_sh + 4 * c;
                if (range_in_bounds(off, 4, p.ext.o, p.status, nullptr)) {
                    if (p.o_f32) store4<float>(static_cast<float *>(p.o) + off, tt);
                    else store4<__nv_bfloat16>(static_cast<__nv_bfloat16 *>(p.o) + off, tt);
                }
            }
            __syncthreads();  // the token's rows, the norms and s_red are free again
        }
    }

    if (failed) {
        // A tile did not arrive in time at iteration kf: mark this CTA's outputs from there on with
        // NaN and report it, then wait for every tile copy still in flight (iterations kf ..
        // kf + NS - 1 were issued, each into stage j % NS as that stage's use j / NS) before the
        // CTA's shared memory is released.
        if (tid == 0 && p.status != nullptr) atomicExch(p.status, (int)CGDR_ERR_TIMEOUT);
        for (int k = kf;; ++k) {
            const int u = u0 + k * G;
            if (u >= units) break;
            const int b = u / p.Hv, h = u % p.Hv;
            for (int j = tid; j < ntok * DV; j += NT) {
                const int64_t off = b * p.o_sb + (j / DV) * p.o_st + h * p.o_sh + j % DV;
                if (!in_bounds(off, p.ext.o, p.status, nullptr)) continue;
                if (p.o_f32) static_cast<float *>(p.o)[off] = __int_as_float(0x7fc00000);
                else static_cast<__nv_bfloat16 *>(p.o)[off] = __float2bfloat16_rn(__int_as_float(0x7fc00000));
            }
        }
        if (tid == 0)
            for (int j = kf; j < kf + NS; ++j)
                if (u0 + j * G < units) mbar_wait_parity(mbar0 + 8 * (j % NS), (uint32_t)((j / NS) & 1), kSpin);
    }
    asm volatile("cp.async.wait_all;" ::: "memory");
}

template <int DK, int DV, typename T, int NTOK>
cgdr_status launch_t(const DecodeParams &p, int units, cudaStream_t s) {
    using Sh = DecodeShape<DK, DV>;
    using Ps = PipeShape<DK, DV, T, NTOK>;
    static SmemOnce smem_once;
    const int sms = device_sms();
    if (sms <= 0) return CGDR_ERR_CUDA;
    // units per CTA as even as the SM count allows
    const int per = (units + sms - 1) / sms;
    const int grid = (units + per - 1) / per;
    if (!smem_limit_once(smem_once, reinterpret_cast<const void *>(decode_kernel<DK, DV, T, NTOK>), Ps::BYTES))
        return CGDR_ERR_CUDA;
    decode_kernel<DK, DV, T, NTOK><<<grid, Sh::NT, Ps::BYTES, s>>>(p, units);
    return cudaGetLastError() == cudaSuccess ? CGDR_OK : CGDR_ERR_CUDA;
}

template <typename T, int NTOK>
cgdr_status launch_dtype(const DecodeParams &p, int dk, int dv, int units, cudaStream_t s) {
#define CGDR_DEC_CASE(K, V) \
    if (dk == K && dv == V) return launch_t<K, V, T, NTOK>(p, units, s);
    CGDR_DEC_CASE(32, 32) CGDR_DEC_CASE(32, 64) CGDR_DEC_CASE(32, 128)
    CGDR_DEC_CASE(64, 32) CGDR_DEC_CASE(64, 64) CGDR_DEC_CASE(64, 128)
    CGDR_DEC_CASE(128, 32) CGDR_DEC_CASE(128, 64) CGDR_DEC_CASE(128, 128)
#undef CGDR_DEC_CASE
    return CGDR_ERR_UNSUPPORTED;
}

DecodeParams params_of(const cgdr_args &a, int ntok) {
    DecodeParams p;
    p.Hk = a.Hk; p.Hv = a.Hv; p.l2norm = a.l2norm_qk != 0; p.gate = a.gate; p.o_f32 = a.o_dtype == CGDR_F32;
    p.ntok = ntok;
    p.q_scale = qscale_of(a); p.eps = eps_of(a);
    p.q = a.q; p.k = a.k; p.v = a.v;
    p.q_sb = a.q_sb; p.q_sh = a.q_sh; p.k_sb = a.k_sb; p.k_sh = a.k_sh; p.v_sb = a.v_sb; p.v_sh = a.v_sh;
    p.g = a.g; p.beta = a.beta;
    p.g_sb = a.g_sb; p.g_sh = a.g_sh; p.beta_sb = a.beta_sb; p.beta_sh = a.beta_sh;
    p.ga = a.a; p.gb = a.b;
    p.a_sb = a.a_sb; p.a_sh = a.a_sh; p.b_sb = a.b_sb; p.b_sh = a.b_sh;
    p.A_log = a.A_log; p.dt_bias = a.dt_bias;
    p.state = a.state; p.o = a.o; p.o_sb = a.o_sb; p.o_sh = a.o_sh;
    p.status = a.status; p.polls = polls_of(a); p.inject = inject_of(a);
    p.ext = extents_of(a, ntok > 1, 0);
    // token strides: a single token never steps them (decode ignores them)
    const bool one = ntok == 1;
    p.q_st = one ? 0 : a.q_st; p.k_st = one ? 0 : a.k_st; p.v_st = one ? 0 : a.v_st; p.g_st = one ? 0 : a.g_st;
    p.beta_st = one ? 0 : a.beta_st; p.a_st = one ? 0 : a.a_st; p.b_st = one ? 0 : a.b_st;
    p.o_st = one ? 0 : a.o_st;
    return p;
}

}  // namespace

cgdr_status launch_decode(const cgdr_args &a, cudaStream_t s) {
    const DecodeParams p = params_of(a, 1);
    const int units = a.B * a.Hv;
    if (a.dtype == CGDR_BF16) return launch_dtype<__nv_bfloat16, 1>(p, a.dk, a.dv, units, s);
    return launch_dtype<float, 1>(p, a.dk, a.dv, units, s);
}

cgdr_status launch_recurrent(const cgdr_args &a, cudaStream_t s) {
    if (a.T < 1 || a.T > kRecurrentMaxT) return CGDR_ERR_UNSUPPORTED;
    const DecodeParams p = params_of(a, a.T);
    const int units = a.B * a.Hv;
    if (a.dtype == CGDR_BF16) return launch_dtype<__nv_bfloat16, kRecurrentMaxT>(p, a.dk, a.dv, units, s);
    return launch_dtype<float, kRecurrentMaxT>(p, a.dk, a.dv, units, s);
}

}  // namespace cgdr
