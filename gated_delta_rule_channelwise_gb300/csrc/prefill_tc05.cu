// Chunked prefill on the fifth-generation tensor cores (tcgen05, TF32 and fp16
// operands, fp32 accumulators in tensor memory), dk = dv = 128, chunk 64:
// one CTA per (batch, v-head) walks its chunks in order, with the state in
// tensor memory as S^T [dv x dk] for the whole sequence.
//
// The chunkwise WY/UT form of "Add parallel chunked prefill for channelwise
// gated delta rule" (executorch PR #21061, Summary); the per-chunk phases
// that do not touch the state (decay prefix, operand tiles, causal terms,
// triangular transform) are in prefill_tc05_chunk.cuh and shared with the
// cluster kernel.  TF32 and fp16 operands (rounded to nearest; the same 10
// mantissa bits) with fp32 accumulation keep the error near 1e-2 of the output
// RMS or below; the state is carried in fp32.
#include <mutex>

#include "prefill_tc05_chunk.cuh"

namespace cgdr {
namespace {

using namespace tc05c;

static_assert(PREP_SMEM_BYTES <= 232448, "shared memory over the per-block limit");

__global__ void __launch_bounds__(NT, 1) prefill_tc05_kernel(const __grid_constant__ Tc05Params p) {
    extern __shared__ __align__(1024) char smem_raw[];
    char *sm = smem_raw + ((1024 - (smem_u32(smem_raw) & 1023)) & 1023);
    const uint32_t sbase = smem_u32(sm);
    const float *sDec = f32p(sm, M_DEC);
    uint32_t *tslot = reinterpret_cast<uint32_t *>(sm + M_TMEM);

    const Head hd = head_of(p, blockIdx.y, blockIdx.x);
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int wq = warp & 3, wc = warp >> 2;                 // TMEM lane quarter, column quarter
    const int64_t sbase_e = ((int64_t)hd.b * p.Hv + hd.h) * DK * DV;   // the head's state tile (elements)
    float *state = p.state + sbase_e;
    const int64_t obase = hd.b * p.o_sb + hd.h * p.o_sh;

    MmaBar mb{sbase + M_MBAR, 0u, p.polls};
    if (tid == 0) {
        mbar_init(mb.mbar, 1);
        mbar_init(sbase + M_STAGE, 1);
        mbar_init(sbase + M_DEAD, 1);
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
        for (int c = 0; c < 32; ++c) {
            const int64_t e = (int64_t)(32 * wc + c) * DV + trow;
            v[c] = in_bounds(sbase_e + e, p.ext.state, p.err, p.status) ? state[e] : 0.f;
        }
        tmem_st32(tmem + lane_off + T_D0 + 32 * wc, v);
    }
    StageTrack st;
    if (p.T > 0) {
        st.stage<STG_V | STG_K>(p, hd, sbase, 0);
        st.stage<STG_Q | STG_G | STG_LAST>(p, hd, sbase, 0);
    }
    fence_before_sync();
    __syncthreads();

    bool ok = true;
    ChunkRegs cr;
    for (int t0 = 0; t0 < p.T && ok; t0 += C) {
        const int L = min(C, p.T - t0);
        if (!(ok = st.wait(sbase, p.polls, p.inject && t0 == 0))) break;
        prep_chunk<true, false>(p, hd, sm, t0, L, hd, t0 + C, sm + R_B, 64, cr);
        if (!(ok = causal_terms<false>(sm, tmem, mb, cr, sm + R_F, 64, 0))) break;
        solve_tb<false>(sm, cr);
        // ------------------------------------------------------------ W^T, U~^T (fp16 operands)
        if (tid == 0) {
            fence_after_sync();
            gemm16<64, 64>(tmem + T_D2, sbase + R_C, sbase + R_G, false);    // W^T  = Kg^T Tb^T
            gemm16<64, 64>(tmem + T_D3, sbase + RC_VT, sbase + R_G, false);  // U~^T = V^T Tb^T
            commit(mb.mbar);
        }
        if (!(ok = mma_wait(mb))) break;
        // -W [r][i] from D2
        {
            float w16[16];
            tmem_ld16(tmem + lane_off + T_D2 + 16 * wc, w16);
#pragma unroll
            for (int c = 0; c < 16; ++c) st_tile(sm, R_C, 64, 16 * wc + c, trow, -w16[c]);
        }
        fence_smem_to_async();
        fence_before_sync();
        __syncthreads();
        // ------------------------------------------------------------ U^T, O^T (state part)
        if (tid == 0) {
            // S^T is read straight from tensor memory (taken as TF32)
            fence_after_sync();
            gemm_ts<64, 128>(tmem + T_D3, tmem + T_D0, sbase + R_C, true);    // U^T += S^T (-W)^T
            gemm_ts<64, 128>(tmem + T_D4, tmem + T_D0, sbase + R_B, false);   // O^T  = S^T Qg^T
            commit(mb.mbar);
        }
        if (!(ok = mma_wait(mb))) break;
        if (t0 + C < p.T) st.stage<STG_V | STG_K>(p, hd, sbase, t0 + C);   // B and G are free
        {
            // D0 <- D0 Diag(e^gC), now that the products above have read it
            float sv[32];
            const int i0 = 32 * wc;
            tmem_ld32(tmem + lane_off + T_D0 + i0, sv);
#pragma unroll
            for (int c = 0; c < 32; ++c) sv[c] *= sDec[i0 + c];
            tmem_st32(tmem + lane_off + T_D0 + i0, sv);
        }
        build_kend(sm, cr);                                                                  // Kend^T
        {
            float v[16];
            tmem_ld16(tmem + lane_off + T_D3 + 16 * wc, v);
#pragma unroll
            for (int c = 0; c < 16; c += 4)                                                  // U^T [j][s]
                st_h4(sm, R_A1, 128, trow, 16 * wc + c, v[c], v[c + 1], v[c + 2], v[c + 3], cr.amax);
            if (cr.amax > kF16Max) record_range(p.err, p.status);
        }
        fence_smem_to_async();
        fence_before_sync();
        __syncthreads();
        // ------------------------------------------------------------ O^T += U^T P^T ; S^T += U^T Kend
        if (tid == 0) {
            fence_after_sync();
            gemm16<64, 64>(tmem + T_D4, sbase + R_A1, sbase + R_F, true);
            gemm16<128, 64>(tmem + T_D0, sbase + R_A1, sbase + A1_KE, true);
            commit(mb.mbar);
        }
        if (t0 + C < p.T) st.stage<STG_G>(p, hd, sbase, t0 + C);           // A2 is free (Kend^T was read out of it)
        if (!(ok = mma_wait(mb))) break;
        if (t0 + C < p.T) st.stage<STG_Q | STG_LAST>(p, hd, sbase, t0 + C);   // F is free
        store_o(p, obase, tmem + T_D4, t0, L);
        fence_before_sync();
        __syncthreads();
    }

    if (ok) {
        float v[32];
        tmem_ld32(tmem + lane_off + T_D0 + 32 * wc, v);
#pragma unroll
        for (int c = 0; c < 32; ++c) {
            const int64_t e = (int64_t)(32 * wc + c) * DV + trow;
            if (in_bounds(sbase_e + e, p.ext.state, p.err, p.status)) state[e] = v[c];
        }
    } else {
        // a wait gave up: record it, give the tensor core a bounded chance to finish, release TMEM
        if (tid == 0) {
            record_timeout(p);
            mbar_wait(mb.mbar, mb.phase ^ 1u, kSpin);
            st.drain(sbase);
        }
    }
    cp_async_wait_all();
    fence_before_sync();
    __syncthreads();
    if (warp == 0) tmem_dealloc(tmem, T_COLS);
}

}  // namespace

bool prefill_tc05_supported(const cgdr_args &a) {
    return a.dtype == CGDR_BF16 && a.dk == 128 && a.dv == 128 && chunk_of(a) == 64 && tc05c::maps_describable(a);
}

size_t prefill_tc05_workspace(const cgdr_args &) { return 256; }

namespace tc05c {

namespace {

// Byte strides of a 4-D map with dims (channel, token, head, batch) and element strides
// (st, sh, sb); false if a tensor map cannot take them (each a positive multiple of 16 bytes
// below 2^40).
bool map_strides(size_t esz, const cuuint64_t dims[4], int64_t st, int64_t sh, int64_t sb, cuuint64_t strides[3]) {
    const int64_t given[3] = {st, sh, sb};
    for (int i = 0; i < 3; ++i) {
        // a dimension of extent 1 is never stepped: give it the dense stride whatever the caller passed
        const cuuint64_t dense = i == 0 ? dims[0] * esz : strides[i - 1] * dims[i];
        if (dims[i + 1] == 1) {
            strides[i] = dense;
        } else {
            if (given[i] <= 0) return false;
            strides[i] = (cuuint64_t)given[i] * esz;
        }
        if (strides[i] % 16 != 0 || strides[i] >= (1ull << 40)) return false;
    }
    return true;
}

bool encode4(CUtensorMap &m, CUtensorMapDataType type, size_t esz, const void *base, int dch, int T, int H, int B,
             int64_t st, int64_t sh, int64_t sb) {
    const cuuint64_t dims[4] = {(cuuint64_t)dch, (cuuint64_t)T, (cuuint64_t)H, (cuuint64_t)B};
    cuuint64_t strides[3];
    if (!map_strides(esz, dims, st, sh, sb, strides)) return false;
    const cuuint32_t box[4] = {(cuuint32_t)dch, (cuuint32_t)C, 1, 1};
    const cuuint32_t estr[4] = {1, 1, 1, 1};
    return tensor_map_encoder()(&m, type, 4, const_cast<void *>(base), dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                    CU_TENSOR_MAP_SWIZZLE_NONE, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                    CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}
bool describable(size_t esz, int dch, const cgdr_args &a, int H, int64_t st, int64_t sh, int64_t sb) {
    const cuuint64_t dims[4] = {(cuuint64_t)dch, (cuuint64_t)a.T, (cuuint64_t)H, (cuuint64_t)a.B};
    cuuint64_t strides[3];
    return map_strides(esz, dims, st, sh, sb, strides);
}
}  // namespace

bool maps_describable(const cgdr_args &a) {
    if (a.T <= 0 || a.B <= 0) return true;                  // nothing to launch
    return describable(2, a.dk, a, a.Hk, a.q_st, a.q_sh, a.q_sb) && describable(2, a.dk, a, a.Hk, a.k_st, a.k_sh, a.k_sb) &&
           describable(2, a.dv, a, a.Hv, a.v_st, a.v_sh, a.v_sb) &&
           (a.gate != CGDR_GATE_CHANNEL || describable(4, a.dk, a, a.Hv, a.g_st, a.g_sh, a.g_sb));
}

bool make_maps(const cgdr_args &a, Tc05Maps &tm) {
    if (tensor_map_encoder() == nullptr || a.T <= 0 || a.B <= 0) return false;
    const auto bf = CU_TENSOR_MAP_DATA_TYPE_BFLOAT16;
    bool ok = encode4(tm.q, bf, 2, a.q, a.dk, a.T, a.Hk, a.B, a.q_st, a.q_sh, a.q_sb) &&
              encode4(tm.k, bf, 2, a.k, a.dk, a.T, a.Hk, a.B, a.k_st, a.k_sh, a.k_sb) &&
              encode4(tm.v, bf, 2, a.v, a.dv, a.T, a.Hv, a.B, a.v_st, a.v_sh, a.v_sb);
    if (ok && a.gate == CGDR_GATE_CHANNEL)
        ok = encode4(tm.g, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 4, a.g, a.dk, a.T, a.Hv, a.B, a.g_st, a.g_sh, a.g_sb);
    return ok;
}

bool make_params(const cgdr_args &a, void *ws, size_t ws_bytes, Tc05Params &p) {
    if (!make_maps(a, p.tm)) return false;
    p.B = a.B; p.T = a.T; p.Hk = a.Hk; p.Hv = a.Hv; p.l2norm = a.l2norm_qk != 0; p.gate = a.gate;
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
    p.status = a.status;
    p.polls = polls_of(a);
    p.inject = inject_of(a);
    p.ext = extents_of(a, true, ws_bytes);
    p.slots = nullptr;
    p.flags = nullptr;
    // o by TMA tensor stores where a map can describe it (a 16-byte aligned base and strides)
    p.o_tma = describable(p.o_f32 ? 4 : 2, a.dv, a, a.Hv, a.o_st, a.o_sh, a.o_sb) &&
              encode4(p.tm.o, p.o_f32 ? CU_TENSOR_MAP_DATA_TYPE_FLOAT32 : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16,
                      p.o_f32 ? 4 : 2, a.o, a.dv, a.T, a.Hv, a.B, a.o_st, a.o_sh, a.o_sb);
    return true;
}
}  // namespace tc05c

cgdr_status launch_prefill_tc05(const cgdr_args &a, void *ws, size_t ws_bytes, cudaStream_t s) {
    static SmemOnce smem_once;
    tc05c::Tc05Params p;
    if (!tc05c::make_params(a, ws, ws_bytes, p)) return CGDR_ERR_ALIGNMENT;
    if (cudaMemsetAsync(ws, 0, sizeof(int), s) != cudaSuccess) return CGDR_ERR_CUDA;
    if (!smem_limit_once(smem_once, reinterpret_cast<const void *>(prefill_tc05_kernel), tc05c::PREP_SMEM_BYTES))
        return CGDR_ERR_CUDA;
    dim3 grid(a.Hv, a.B);
    prefill_tc05_kernel<<<grid, tc05c::NT, tc05c::PREP_SMEM_BYTES, s>>>(p);
    return cudaGetLastError() == cudaSuccess ? CGDR_OK : CGDR_ERR_CUDA;
}

}  // namespace cgdr

// ---------------------------------------------------------------------------
// Allocation-free prefill: the scratch is this file's static device array.
namespace cgdr {
namespace {

__device__ __align__(256) unsigned char g_noalloc_scratch[CGDR_NOALLOC_SCRATCH_BYTES];

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
    // the cluster kernel's hand-off ring does not fit the static scratch: per-head kernel instead;
    // the kernel is chosen once and that choice is what runs
    const int path = cgdr::prefill_path(*a, false);
    const size_t need = cgdr::prefill_workspace_for(*a, path);
    if (need > CGDR_NOALLOC_SCRATCH_BYTES) return CGDR_ERR_WORKSPACE;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    if (need == 0) return cgdr::prefill_dispatch(*a, path, nullptr, 0, s);
    int dev = -1;
    if (cudaGetDevice(&dev) != cudaSuccess) return CGDR_ERR_CUDA;
    void *scratch = nullptr;
    const cgdr_status s2 = cgdr::noalloc_scratch(dev, &scratch);
    if (s2 != CGDR_OK) return s2;
    return cgdr::prefill_dispatch(*a, path, scratch, CGDR_NOALLOC_SCRATCH_BYTES, s);
}
