// Chunked prefill on a four-CTA thread-block cluster per (batch, v-head),
// for launches with too few heads to fill the GPU one CTA per head.
//
// The chunkwise WY/UT form of "Add parallel chunked prefill for channelwise
// gated delta rule" (executorch PR #21061, Summary) splits into work that
// needs the state (the carry S <- e^gC S + Kend^T U with U = U~ - W S, and the
// output O = Qg S + P U) and work that does not (decay prefix, operand tiles,
// causal terms, the triangular transform, W and U~).  Only the first is
// serial along T.  So:
//   rank 0 (the chain)   keeps S^T in tensor memory and, per chunk, runs the
//                        four state-dependent contractions and writes o;
//   ranks 1..3 (preparers) take chunks round robin (chunk c on rank
//                        1 + c % 3), run the state-free phases and push
//                        -W, Qg, U~^T, e^gC (inbox A) and P, Kend^T (inbox B)
//                        into rank 0's shared memory with bulk copies over
//                        the cluster (distributed shared memory).
// Handshake per chunk c: rank 0's full_A / full_B barriers count the bytes
// of c's pushes (armed with expect_tx before the preparer may push); once
// rank 0's contractions have read inbox A (B) of chunk c it arrives on
// free_A (free_B) of the preparer of chunk c + 1.  Every wait is bounded;
// a wait that gives up records CGDR_ERR_TIMEOUT and every CTA leaves its
// loop, drains its copies, frees tensor memory and meets the others at the
// final cluster barrier.
#include <atomic>
#include <mutex>

#include "prefill_tc05_chunk.cuh"

namespace cgdr {
namespace {

using namespace tc05c;

constexpr int CLUSTER = 4, NPREP = CLUSTER - 1;

// rank 0 shared memory map (bytes from the 1024-aligned base)
constexpr int CH_IN_A = 0;
constexpr int CH_W = CH_IN_A;                    // -W    [64 x 128] tile
constexpr int CH_QG = CH_IN_A + 32768;           // Qg    [64 x 128] tile
constexpr int CH_UT = CH_IN_A + 65536;           // U~^T  [128 x 64] fp32 in tile order (not rounded)
constexpr int CH_DEC = CH_IN_A + 98304;          // e^gC  [128] fp32
constexpr uint32_t A_BYTES = 98304 + 512;
constexpr int CH_SC = 99328;                     // S^T copy [128 x 128] tile, then U^T [128 x 64]
constexpr int CH_IN_B = CH_SC + 65536;
constexpr int CH_P = CH_IN_B;                    // P      [64 x 64] tile
constexpr int CH_KE = CH_IN_B + 16384;           // Kend^T [128 x 64] tile
constexpr uint32_t B_BYTES = 16384 + 32768;
constexpr int CH_MISC = CH_IN_B + 49152;
constexpr int CH_MBAR = CH_MISC, CH_FULL_A = CH_MISC + 8, CH_FULL_B = CH_MISC + 16, CH_TMEM = CH_MISC + 24;
constexpr int CH_END = CH_MISC + 32;
static_assert(CH_SC % 1024 == 0 && CH_IN_B % 1024 == 0 && CH_KE % 1024 == 0, "tiles must be 1024-aligned");
constexpr int CL_SMEM_BYTES = (CH_END > M_END ? CH_END : M_END) + 1024;
static_assert(CL_SMEM_BYTES <= 232448, "shared memory over the per-block limit");

// ---------------------------------------------------------------- cluster primitives
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
// Bounded wait, with cluster-scope acquire, for the phase of a local barrier with the given parity.
__device__ __forceinline__ bool cl_wait(uint32_t mbar, uint32_t parity) {
    for (uint32_t it = 0; it < kSpin; ++it) {
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
// Bulk copy of `bytes` from this CTA's shared memory into another CTA's, completion
// counted in bytes on the destination CTA's barrier.
__device__ __forceinline__ void push(uint32_t dst_cluster, uint32_t src, uint32_t bytes, uint32_t mbar_cluster) {
    asm volatile(
        "cp.async.bulk.shared::cluster.shared::cta.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];"
        ::"r"(dst_cluster), "r"(src), "r"(bytes), "r"(mbar_cluster) : "memory");
}
__device__ __forceinline__ void push_commit() { asm volatile("cp.async.bulk.commit_group;" ::: "memory"); }
__device__ __forceinline__ void push_wait_read() { asm volatile("cp.async.bulk.wait_group.read 0;" ::: "memory"); }
__device__ __forceinline__ void push_wait_done() { asm volatile("cp.async.bulk.wait_group 0;" ::: "memory"); }

__device__ __forceinline__ uint32_t owner_of(int c) { return 1u + (uint32_t)(c % NPREP); }

// ---------------------------------------------------------------- rank 0: the state carry
__device__ __forceinline__ bool run_chain(const Tc05Params &p, const Head &hd, char *sm, uint32_t tmem, MmaBar &mb,
                                          int n) {
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int wq = warp & 3, wc = warp >> 2;
    const uint32_t sbase = smem_u32(sm);
    const uint32_t lane_off = (uint32_t)(32 * wq) << 16;
    const int trow = 32 * wq + lane;
    float *state = p.state + ((size_t)hd.b * p.Hv + hd.h) * DK * DV;
    const int64_t obase = hd.b * p.o_sb + hd.h * p.o_sh;
    const float *dec = f32p(sm, CH_DEC);

    // state -> D0 = S^T: row j = trow, columns i in [32 wc, 32 wc + 32)
    {
        float v[32];
#pragma unroll
        for (int c = 0; c < 32; ++c) v[c] = state[(size_t)(32 * wc + c) * DV + trow];
        tmem_st32(tmem + lane_off + T_D0 + 32 * wc, v);
    }
    for (int c = 0; c < n; ++c) {
        const uint32_t d4 = (c & 1) ? T_D4B : T_D4;
        // ---------------------------------------------------------- inbox A: -W, Qg, U~^T, e^gC
        {
            const bool done = cl_wait(sbase + CH_FULL_A, (uint32_t)(c & 1));
            if (__syncthreads_or(!done)) return false;
        }
        if (tid == 0 && c + 1 < n) arrive_expect_tx(sbase + CH_FULL_A, A_BYTES);
        {
            float u[16];
#pragma unroll
            for (int m = 0; m < 4; ++m) {
                const float4 x = *reinterpret_cast<const float4 *>(sm + CH_UT + sw_off(128, trow, 16 * wc + 4 * m));
                u[4 * m] = x.x; u[4 * m + 1] = x.y; u[4 * m + 2] = x.z; u[4 * m + 3] = x.w;
            }
            tmem_st16(tmem + lane_off + T_D3 + 16 * wc, u);                  // D3 = U~^T
            float v[32];
            const int i0 = 32 * wc;
            tmem_ld32(tmem + lane_off + T_D0 + i0, v);                       // S^T copy, then D0 <- D0 Diag(e^gC)
#pragma unroll
            for (int k = 0; k < 32; k += 4) st_tile4(sm, CH_SC, 128, trow, i0 + k, v[k], v[k + 1], v[k + 2], v[k + 3]);
#pragma unroll
            for (int k = 0; k < 32; ++k) v[k] *= dec[i0 + k];
            tmem_st32(tmem + lane_off + T_D0 + i0, v);
        }
        fence_smem_to_async();
        fence_before_sync();
        __syncthreads();
        if (tid == 0) {
            fence_after_sync();
            gemm<64, 128>(tmem + T_D3, sbase + CH_SC, sbase + CH_W, true);    // U^T = U~^T + S^T (-W)^T
            gemm<64, 128>(tmem + d4, sbase + CH_SC, sbase + CH_QG, false);    // O^T = S^T Qg^T
            commit(mb.mbar);
        }
        if (c > 0) store_o(p, obase, tmem + ((c & 1) ? T_D4 : T_D4B), (c - 1) * C, C);   // previous chunk's o
        if (!mma_wait(mb)) return false;
        if (tid == 0 && c + 1 < n) remote_arrive(mapa_rank(sbase + M_FREE_A, owner_of(c + 1)));
        {
            float v[16];
            tmem_ld16(tmem + lane_off + T_D3 + 16 * wc, v);
#pragma unroll
            for (int k = 0; k < 16; k += 4)                                   // U^T [j][s]
                st_tile4(sm, CH_SC, 128, trow, 16 * wc + k, v[k], v[k + 1], v[k + 2], v[k + 3]);
        }
        fence_smem_to_async();
        fence_before_sync();
        // ---------------------------------------------------------- inbox B: P, Kend^T
        {
            const bool done = cl_wait(sbase + CH_FULL_B, (uint32_t)(c & 1));
            if (__syncthreads_or(!done)) return false;
        }
        if (tid == 0) {
            if (c + 1 < n) arrive_expect_tx(sbase + CH_FULL_B, B_BYTES);
            fence_after_sync();
            gemm<64, 64>(tmem + d4, sbase + CH_SC, sbase + CH_P, true);       // O^T += U^T P^T
            gemm<128, 64>(tmem + T_D0, sbase + CH_SC, sbase + CH_KE, true);   // S^T += U^T Kend
            commit(mb.mbar);
        }
        if (!mma_wait(mb)) return false;
        if (tid == 0 && c + 1 < n) remote_arrive(mapa_rank(sbase + M_FREE_B, owner_of(c + 1)));
    }
    if (n > 0) store_o(p, obase, tmem + (((n - 1) & 1) ? T_D4B : T_D4), (n - 1) * C, p.T - (n - 1) * C);
    float v[32];
    tmem_ld32(tmem + lane_off + T_D0 + 32 * wc, v);
#pragma unroll
    for (int c = 0; c < 32; ++c) state[(size_t)(32 * wc + c) * DV + trow] = v[c];
    return true;
}

// ---------------------------------------------------------------- ranks 1..3: state-free phases
__device__ __forceinline__ bool run_prep(const Tc05Params &p, const Head &hd, char *sm, uint32_t tmem, MmaBar &mb,
                                         int n, int rank) {
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int wq = warp & 3, wc = warp >> 2;
    const int ci = tid & 127, cq = tid >> 7;
    const uint32_t sbase = smem_u32(sm);
    const uint32_t lane_off = (uint32_t)(32 * wq) << 16;
    const int trow = 32 * wq + lane;
    const int c_first = rank - 1;
    if (c_first < n) {
        stage_rows<STG_V | STG_K>(p, hd, sbase, c_first * C);
        stage_rows<STG_Q | STG_G>(p, hd, sbase, c_first * C);
    }
    int nfree = 0;
    ChunkRegs cr;
    for (int c = c_first; c < n; c += NPREP) {
        const int t0 = c * C, L = min(C, p.T - t0), tn = t0 + NPREP * C;
        cp_async_wait_all();
        __syncthreads();
        prep_chunk(p, hd, sm, t0, L, tn, cr);
        if (!causal_terms(sm, tmem, mb, cr)) return false;
        solve_tb(sm);
        if (tid == 0) {
            fence_after_sync();
            gemm<64, 64>(tmem + T_D2, sbase + R_C, sbase + R_G, false);    // W^T  = Kg^T Tb^T
            gemm<64, 64>(tmem + T_D3, sbase + A1_VT, sbase + R_G, false);  // U~^T = V^T Tb^T
            commit(mb.mbar);
        }
        if (!mma_wait(mb)) return false;
        if (tn < p.T) stage_rows<STG_K>(p, hd, sbase, tn);                 // G is free
        {
            float w16[16];
            tmem_ld16(tmem + lane_off + T_D2 + 16 * wc, w16);
#pragma unroll
            for (int k = 0; k < 16; ++k) st_tile(sm, R_C, 64, 16 * wc + k, trow, -w16[k]);   // -W [r][i]
            float u16[16];
            tmem_ld16(tmem + lane_off + T_D3 + 16 * wc, u16);
#pragma unroll
            for (int k = 0; k < 16; k += 4)                                   // U~^T [j][s], full fp32
                *reinterpret_cast<float4 *>(sm + A1_VT + sw_off(128, trow, 16 * wc + k)) =
                    make_float4(u16[k], u16[k + 1], u16[k + 2], u16[k + 3]);
            const float sc = cr.wide ? 1.f : __expf(cr.gcv - cr.gm);
#pragma unroll
            for (int jj = 0; jj < 16; jj += 4) {                              // Kend^T [i][s]
                const int s0 = 16 * cq + jj;
                st_tile4(sm, R_A1, 128, ci, s0, ld_tile(sm, R_A2, 64, s0, ci) * sc,
                         ld_tile(sm, R_A2, 64, s0 + 1, ci) * sc, ld_tile(sm, R_A2, 64, s0 + 2, ci) * sc,
                         ld_tile(sm, R_A2, 64, s0 + 3, ci) * sc);
            }
        }
        fence_smem_to_async();
        __syncthreads();
        if (tn < p.T) stage_rows<STG_G>(p, hd, sbase, tn);                 // A2 is free
        int pushed = 1;
        if (tid == 0) {
            const uint32_t fullA = mapa_rank(sbase + CH_FULL_A, 0), fullB = mapa_rank(sbase + CH_FULL_B, 0);
            bool okw = c == 0 || cl_wait(sbase + M_FREE_A, (uint32_t)(nfree & 1));
            if (okw) {
                push(mapa_rank(sbase + CH_W, 0), sbase + R_C, 32768, fullA);
                push(mapa_rank(sbase + CH_QG, 0), sbase + R_B, 32768, fullA);
                push(mapa_rank(sbase + CH_UT, 0), sbase + A1_VT, 32768, fullA);
                push(mapa_rank(sbase + CH_DEC, 0), sbase + M_DEC, 512, fullA);
            }
            okw = okw && (c == 0 || cl_wait(sbase + M_FREE_B, (uint32_t)(nfree & 1)));
            if (okw) {
                push(mapa_rank(sbase + CH_P, 0), sbase + R_F, 16384, fullB);
                push(mapa_rank(sbase + CH_KE, 0), sbase + R_A1, 32768, fullB);
            }
            push_commit();
            push_wait_read();
            pushed = okw ? 1 : 0;
        }
        if (c > 0) ++nfree;
        if (__syncthreads_or(!pushed)) return false;
        if (tn < p.T) stage_rows<STG_Q | STG_V>(p, hd, sbase, tn);         // F and B are free
    }
    return true;
}

__global__ void __cluster_dims__(CLUSTER, 1, 1) __launch_bounds__(NT, 1) prefill_cluster_kernel(const Tc05Params p) {
    extern __shared__ __align__(1024) char smem_raw[];
    char *sm = smem_raw + ((1024 - (smem_u32(smem_raw) & 1023)) & 1023);
    const uint32_t sbase = smem_u32(sm);
    const int rank = (int)cluster_ctarank();
    const bool chain = rank == 0;
    const Head hd = head_of(p, blockIdx.y, blockIdx.x / CLUSTER);
    const int tid = threadIdx.x, warp = tid >> 5;
    const int n = (p.T + C - 1) / C;
    uint32_t *tslot = reinterpret_cast<uint32_t *>(sm + (chain ? CH_TMEM : M_TMEM));
    MmaBar mb{sbase + (chain ? CH_MBAR : M_MBAR), 0u};
    if (tid == 0) {
        mbar_init(mb.mbar, 1);
        if (chain) {
            mbar_init(sbase + CH_FULL_A, 1);
            mbar_init(sbase + CH_FULL_B, 1);
        } else {
            mbar_init(sbase + M_FREE_A, 1);
            mbar_init(sbase + M_FREE_B, 1);
        }
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
        if (chain && n > 0) {
            arrive_expect_tx(sbase + CH_FULL_A, A_BYTES);
            arrive_expect_tx(sbase + CH_FULL_B, B_BYTES);
        }
    }
    if (warp == 0) tmem_alloc(smem_u32(tslot), T_COLS);
    fence_before_sync();
    __syncthreads();
    fence_after_sync();
    const uint32_t tmem = *tslot;
    cluster_barrier();                         // every CTA's barriers exist before any remote use

    const bool ok = chain ? run_chain(p, hd, sm, tmem, mb, n) : run_prep(p, hd, sm, tmem, mb, n, rank);
    if (!ok && tid == 0) {
        // a wait gave up: record it and give the tensor core a bounded chance to finish
        atomicExch(p.err, (int)CGDR_ERR_TIMEOUT);
        mbar_wait(mb.mbar, mb.phase ^ 1u, kSpin);
    }
    if (!chain && tid == 0) push_wait_done();  // every copy into rank 0 has landed
    fence_before_sync();
    __syncthreads();
    if (warp == 0) tmem_dealloc(tmem, T_COLS);
    cluster_barrier();                         // no CTA leaves while another may still address it
}

std::mutex g_cluster_mutex;
int g_cluster_fit[64];                         // per device: clusters resident at once, + 1 (0 = not queried)

}  // namespace

// Number of four-CTA clusters of this kernel the current device runs at once (0 if none fit).
int prefill_cluster_capacity() {
    int dev = -1;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return 0;
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

cgdr_status launch_prefill_cluster(const cgdr_args &a, void *ws, cudaStream_t s) {
    const Tc05Params p = make_params(a, ws);
    if (cudaMemsetAsync(ws, 0, sizeof(int), s) != cudaSuccess) return CGDR_ERR_CUDA;
    if (cudaFuncSetAttribute(prefill_cluster_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, CL_SMEM_BYTES) !=
        cudaSuccess)
        return CGDR_ERR_CUDA;
    dim3 grid(CLUSTER * a.Hv, a.B);
    prefill_cluster_kernel<<<grid, NT, CL_SMEM_BYTES, s>>>(p);
    return cudaGetLastError() == cudaSuccess ? CGDR_OK : CGDR_ERR_CUDA;
}

}  // namespace cgdr
