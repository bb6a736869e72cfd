// Decode (T = 1): one CTA per (batch, v-head) state tile, held in registers.
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
// Layout: a warp instruction covers RW consecutive rows of the dk x dv tile
// with 16-byte (float4) loads, so every access is a full 128-byte line.  The
// reduction over dk runs in registers, then across the row-lanes of a warp
// with shuffles, then across warps through a small shared array.
#include "cgdr_internal.cuh"

namespace cgdr {
namespace {

struct DecodeParams {
    int Hk, Hv, l2norm, gate, o_f32;
    float q_scale, eps;
    const void *q, *k, *v;
    int64_t q_sb, q_sh, k_sb, k_sh, v_sb, v_sh;
    const float *g, *beta;
    int64_t g_sb, g_sh, beta_sb, beta_sh;
    const void *ga, *gb;
    int64_t a_sb, a_sh, b_sb, b_sh;
    const float *A_log, *dt_bias;
    float *state;
    void *o;
    int64_t o_sb, o_sh;
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

__device__ __forceinline__ float4 ld_stream(const float *p) { return __ldcs(reinterpret_cast<const float4 *>(p)); }
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

template <int DK, int DV, typename T>
__global__ void __launch_bounds__(DecodeShape<DK, DV>::NT, 2) decode_kernel(const DecodeParams p) {
    using Sh = DecodeShape<DK, DV>;
    constexpr int CL = Sh::CL, RW = Sh::RW, NW = Sh::NW, RPT = Sh::RPT;
    __shared__ float s_kn[DK], s_qn[DK], s_alpha[DK];
    __shared__ float4 s_red[NW][CL];
    __shared__ float s_beta;

    const int bh = blockIdx.x;
    const int b = bh / p.Hv, h = bh % p.Hv;
    const int hk = h / (p.Hv / p.Hk);
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int c = lane % CL, r = lane / CL;
    float *S = p.state + (size_t)bh * DK * DV;

    // 1. Issue every state load first so the whole tile is in flight while
    //    the norms and the gate are computed.
    float4 s[RPT];
#pragma unroll
    for (int ii = 0; ii < RPT; ++ii) {
        const int row = (warp * RPT + ii) * RW + r;
        s[ii] = ld_stream(S + (size_t)row * DV + 4 * c);
    }

    // 2. q/k L2 norm (a warp each), per-channel decay alpha and beta.
    const T *q = static_cast<const T *>(p.q) + b * p.q_sb + hk * p.q_sh;
    const T *k = static_cast<const T *>(p.k) + b * p.k_sb + hk * p.k_sh;
    for (int which = warp; which < 2; which += NW) {
        const T *x = which == 0 ? q : k;
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
        const float *g = p.g + b * p.g_sb + h * p.g_sh;
        for (int i = threadIdx.x; i < DK; i += blockDim.x) s_alpha[i] = expf(g[i]);
        if (threadIdx.x == 0) s_beta = p.beta[b * p.beta_sb + h * p.beta_sh];
    } else {
        const float av = Cvt<T>::to_f(static_cast<const T *>(p.ga)[b * p.a_sb + h * p.a_sh]);
        const float alpha = expf(gdn_gate(p.A_log[h], av, p.dt_bias[h]));
        for (int i = threadIdx.x; i < DK; i += blockDim.x) s_alpha[i] = alpha;
        if (threadIdx.x == 0)
            s_beta = sigmoid_f(Cvt<T>::to_f(static_cast<const T *>(p.gb)[b * p.b_sb + h * p.b_sh]));
    }
    __syncthreads();

    // 3. Sweep 1: vh = S^T (alpha * kn) over this thread's rows.
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
        const float4 t = s_red[w][c];
        vh.x += t.x; vh.y += t.y; vh.z += t.z; vh.w += t.w;
    }
    const float4 vv = load4<T>(static_cast<const T *>(p.v) + b * p.v_sb + h * p.v_sh + 4 * c);
    const float beta = s_beta;
    const float4 u = make_float4(beta * (vv.x - vh.x), beta * (vv.y - vh.y), beta * (vv.z - vh.z),
                                 beta * (vv.w - vh.w));
    __syncthreads();  // s_red is reused below

    // 4. Sweep 2: decay + rank-one write, accumulate o, store the tile once.
    float4 o = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
    for (int ii = 0; ii < RPT; ++ii) {
        const int row = (warp * RPT + ii) * RW + r;
        const float al = s_alpha[row], kn = s_kn[row], qn = s_qn[row];
        float4 x = s[ii];
        x.x = fmaf(al, x.x, kn * u.x);
        x.y = fmaf(al, x.y, kn * u.y);
        x.z = fmaf(al, x.z, kn * u.z);
        x.w = fmaf(al, x.w, kn * u.w);
        o.x = fmaf(qn, x.x, o.x);
        o.y = fmaf(qn, x.y, o.y);
        o.z = fmaf(qn, x.z, o.z);
        o.w = fmaf(qn, x.w, o.w);
        st_stream(S + (size_t)row * DV + 4 * c, x);
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
        float4 t = s_red[0][c];
#pragma unroll
        for (int w = 1; w < NW; ++w) {
            const float4 y = s_red[w][c];
            t.x += y.x; t.y += y.y; t.z += y.z; t.w += y.w;
        }
        const int64_t off = b * p.o_sb + h * p.o_sh + 4 * c;
        if (p.o_f32)
            store4<float>(static_cast<float *>(p.o) + off, t);
        else
            store4<__nv_bfloat16>(static_cast<__nv_bfloat16 *>(p.o) + off, t);
    }
}

template <int DK, int DV, typename T>
cgdr_status launch_t(const DecodeParams &p, int units, cudaStream_t s) {
    using Sh = DecodeShape<DK, DV>;
    decode_kernel<DK, DV, T><<<units, Sh::NT, 0, s>>>(p);
    return cudaGetLastError() == cudaSuccess ? CGDR_OK : CGDR_ERR_CUDA;
}

template <typename T>
cgdr_status launch_dtype(const DecodeParams &p, int dk, int dv, int units, cudaStream_t s) {
#define CGDR_DEC_CASE(K, V) \
    if (dk == K && dv == V) return launch_t<K, V, T>(p, units, s);
    CGDR_DEC_CASE(32, 32) CGDR_DEC_CASE(32, 64) CGDR_DEC_CASE(32, 128)
    CGDR_DEC_CASE(64, 32) CGDR_DEC_CASE(64, 64) CGDR_DEC_CASE(64, 128)
    CGDR_DEC_CASE(128, 32) CGDR_DEC_CASE(128, 64) CGDR_DEC_CASE(128, 128)
#undef CGDR_DEC_CASE
    return CGDR_ERR_UNSUPPORTED;
}

}  // namespace

cgdr_status launch_decode(const cgdr_args &a, cudaStream_t s) {
    DecodeParams p;
    p.Hk = a.Hk; p.Hv = a.Hv; p.l2norm = a.l2norm_qk != 0; p.gate = a.gate; p.o_f32 = a.o_dtype == CGDR_F32;
    p.q_scale = qscale_of(a); p.eps = eps_of(a);
    p.q = a.q; p.k = a.k; p.v = a.v;
    p.q_sb = a.q_sb; p.q_sh = a.q_sh; p.k_sb = a.k_sb; p.k_sh = a.k_sh; p.v_sb = a.v_sb; p.v_sh = a.v_sh;
    p.g = a.g; p.beta = a.beta;
    p.g_sb = a.g_sb; p.g_sh = a.g_sh; p.beta_sb = a.beta_sb; p.beta_sh = a.beta_sh;
    p.ga = a.a; p.gb = a.b;
    p.a_sb = a.a_sb; p.a_sh = a.a_sh; p.b_sb = a.b_sb; p.b_sh = a.b_sh;
    p.A_log = a.A_log; p.dt_bias = a.dt_bias;
    p.state = a.state; p.o = a.o; p.o_sb = a.o_sb; p.o_sh = a.o_sh;
    const int units = a.B * a.Hv;
    if (a.dtype == CGDR_BF16) return launch_dtype<__nv_bfloat16>(p, a.dk, a.dv, units, s);
    return launch_dtype<float>(p, a.dk, a.dv, units, s);
}

}  // namespace cgdr
