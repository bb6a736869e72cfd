// Blackwell (sm_100 family) fifth-generation tensor core helpers: tcgen05.mma
// with operands in shared memory and the accumulator in tensor memory (TMEM).
//
// TF32 operand tiles are fp32 values rounded to TF32, stored K-major with the
// 128-byte swizzle: a tile of R rows and K columns is split into K/32 blocks
// of 32 fp32 (128 bytes per row); each block is R x 128 bytes, contiguous,
// 1024-byte aligned; inside a row the sixteen-byte chunk c sits at chunk
// position c ^ (row % 8).  One MMA instruction consumes K = 8 (32 bytes), so
// the k-th step starts 32 bytes into the row of its 128-byte block.
#pragma once

#include <stdint.h>

namespace cgdr {
namespace tc05 {

// x rounded to TF32 (10 explicit mantissa bits), to nearest with ties away from zero: half a
// TF32 ulp is added to the magnitude bits, then the 13 low bits are dropped -- the result of
// cvt.rna.tf32.f32 for every finite x, in two integer instructions instead of a conversion
// (the prefill kernels measured 1-3 % faster with it, bit-identical).
__device__ __forceinline__ float tf32r(float x) {
    return __uint_as_float((__float_as_uint(x) + 0x1000u) & 0xFFFFE000u);
}

// Byte offset of element (r, k) in a K-major 128B-swizzled fp32 tile with R rows.
__host__ __device__ __forceinline__ uint32_t sw_off(int R, int r, int k) {
    const int kb = k >> 5, c = (k & 31) >> 2;
    return (uint32_t)(kb * R * 128 + r * 128 + ((c ^ (r & 7)) << 4) + ((k & 3) << 2));
}

// Shared-memory matrix descriptor: start address, SBO = 1024 B (8 rows of
// 128 B), descriptor version 1, 128-byte swizzle.
__device__ __forceinline__ uint64_t smem_desc(uint32_t addr) {
    uint64_t d = (uint64_t)((addr >> 4) & 0x3FFF);
    d |= (uint64_t)1 << 16;
    d |= (uint64_t)(1024 >> 4) << 32;
    d |= (uint64_t)1 << 46;
    d |= (uint64_t)2 << 61;
    return d;
}

// Instruction descriptor: D fp32, A and B TF32, both K-major, M = 128.
__host__ __device__ constexpr uint32_t idesc_tf32(int N) {
    return (1u << 4) | (2u << 7) | (2u << 10) | ((uint32_t)(N >> 3) << 17) | ((uint32_t)(128 >> 4) << 24);
}

__device__ __forceinline__ void mma_tf32(uint32_t d_tmem, uint64_t a, uint64_t b, uint32_t idesc, uint32_t acc) {
    asm volatile(
        "{\n.reg .pred p;\nsetp.ne.u32 p, %4, 0;\n"
        "tcgen05.mma.cta_group::1.kind::tf32 [%0], %1, %2, %3, p;\n}\n"
        ::"r"(d_tmem), "l"(a), "l"(b), "r"(idesc), "r"(acc));
}

// D[128 x N] (+)= A[128 x K] * B[N x K]^T; A and B are K-major swizzled tiles
// with 128 and N rows.  Issued by one thread.  The descriptors are built once: a byte offset
// o (a multiple of 16) moves a descriptor's start-address field by o / 16, and shared
// addresses stay below 2^18, so the field never carries into the next one.
template <int N, int K>
__device__ __forceinline__ void gemm(uint32_t d_tmem, uint32_t a_smem, uint32_t b_smem, bool accumulate) {
    constexpr uint32_t idesc = idesc_tf32(N);
    const uint64_t ad = smem_desc(a_smem), bd = smem_desc(b_smem);
#pragma unroll
    for (int ks = 0; ks < K / 8; ++ks) {
        constexpr int kAStep = 128 * 128 / 16, kBStep = N * 128 / 16;
        const uint64_t a = ad + (uint64_t)((ks >> 2) * kAStep + (ks & 3) * 2);
        const uint64_t b = bd + (uint64_t)((ks >> 2) * kBStep + (ks & 3) * 2);
        mma_tf32(d_tmem, a, b, idesc, (accumulate || ks > 0) ? 1u : 0u);
    }
}

// The same with A read from tensor memory: A[m][k] = TMEM[lane m][column a_tmem + k],
// fp32 values taken as TF32 (the low 13 mantissa bits are ignored).
__device__ __forceinline__ void mma_tf32_ts(uint32_t d_tmem, uint32_t a_tmem, uint64_t b, uint32_t idesc, uint32_t acc) {
    asm volatile(
        "{\n.reg .pred p;\nsetp.ne.u32 p, %4, 0;\n"
        "tcgen05.mma.cta_group::1.kind::tf32 [%0], [%1], %2, %3, p;\n}\n"
        ::"r"(d_tmem), "r"(a_tmem), "l"(b), "r"(idesc), "r"(acc));
}

template <int N, int K>
__device__ __forceinline__ void gemm_ts(uint32_t d_tmem, uint32_t a_tmem, uint32_t b_smem, bool accumulate) {
    constexpr uint32_t idesc = idesc_tf32(N);
    const uint64_t bd = smem_desc(b_smem);
#pragma unroll
    for (int ks = 0; ks < K / 8; ++ks) {
        const uint64_t b = bd + (uint64_t)((ks >> 2) * (N * 128 / 16) + (ks & 3) * 2);
        mma_tf32_ts(d_tmem, a_tmem + 8 * ks, b, idesc, (accumulate || ks > 0) ? 1u : 0u);
    }
}

// fp16 operand tiles.  fp16 carries the same 10 explicit mantissa bits as TF32, so for values
// well inside its range (|x| < 65504) it rounds no worse than TF32 in absolute terms, at half
// the bytes and twice the tensor-core rate.  Same K-major 128-byte swizzle: a block holds 64
// halves per row, and one instruction consumes K = 16 (32 bytes), so the descriptor steps are
// those of the TF32 tiles.
__host__ __device__ __forceinline__ uint32_t sw_off16(int R, int r, int k) {
    const int kb = k >> 6, c = (k & 63) >> 3;
    return (uint32_t)(kb * R * 128 + r * 128 + ((c ^ (r & 7)) << 4) + ((k & 7) << 1));
}

// Instruction descriptor: D fp32, A and B fp16 (both K-major), M = 128.
__host__ __device__ constexpr uint32_t idesc_f16(int N) {
    return (1u << 4) | ((uint32_t)(N >> 3) << 17) | ((uint32_t)(128 >> 4) << 24);
}

__device__ __forceinline__ void mma_f16(uint32_t d_tmem, uint64_t a, uint64_t b, uint32_t idesc, uint32_t acc) {
    asm volatile(
        "{\n.reg .pred p;\nsetp.ne.u32 p, %4, 0;\n"
        "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n}\n"
        ::"r"(d_tmem), "l"(a), "l"(b), "r"(idesc), "r"(acc));
}

// D[128 x N] (+)= A[128 x K] * B[N x K]^T with fp16 tiles (128 and N rows).
template <int N, int K>
__device__ __forceinline__ void gemm16(uint32_t d_tmem, uint32_t a_smem, uint32_t b_smem, bool accumulate) {
    constexpr uint32_t idesc = idesc_f16(N);
    const uint64_t ad = smem_desc(a_smem), bd = smem_desc(b_smem);
#pragma unroll
    for (int ks = 0; ks < K / 16; ++ks) {
        constexpr int kAStep = 128 * 128 / 16, kBStep = N * 128 / 16;
        const uint64_t a = ad + (uint64_t)((ks >> 2) * kAStep + (ks & 3) * 2);
        const uint64_t b = bd + (uint64_t)((ks >> 2) * kBStep + (ks & 3) * 2);
        mma_f16(d_tmem, a, b, idesc, (accumulate || ks > 0) ? 1u : 0u);
    }
}

// The same with A read from tensor memory: A[m][k] = the fp16 pair in TMEM[lane m][column
// a_tmem + k / 2] (element k in the low half for even k), K = 16 per instruction (8 columns).
__device__ __forceinline__ void mma_f16_ts(uint32_t d_tmem, uint32_t a_tmem, uint64_t b, uint32_t idesc, uint32_t acc) {
    asm volatile(
        "{\n.reg .pred p;\nsetp.ne.u32 p, %4, 0;\n"
        "tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], %2, %3, p;\n}\n"
        ::"r"(d_tmem), "r"(a_tmem), "l"(b), "r"(idesc), "r"(acc));
}

template <int N, int K>
__device__ __forceinline__ void gemm16_ts(uint32_t d_tmem, uint32_t a_tmem, uint32_t b_smem, bool accumulate) {
    constexpr uint32_t idesc = idesc_f16(N);
    const uint64_t bd = smem_desc(b_smem);
#pragma unroll
    for (int ks = 0; ks < K / 16; ++ks) {
        const uint64_t b = bd + (uint64_t)((ks >> 2) * (N * 128 / 16) + (ks & 3) * 2);
        mma_f16_ts(d_tmem, a_tmem + 8 * ks, b, idesc, (accumulate || ks > 0) ? 1u : 0u);
    }
}

__device__ __forceinline__ void commit(uint32_t mbar) {
    asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(mbar));
}

__device__ __forceinline__ void mbar_init(uint32_t mbar, uint32_t count) {
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(mbar), "r"(count));
}

__device__ __forceinline__ bool mbar_try_wait(uint32_t mbar, uint32_t parity) {
    uint32_t done;
    asm volatile(
        "{\n.reg .pred p;\nmbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\nselp.u32 %0, 1, 0, p;\n}\n"
        : "=r"(done) : "r"(mbar), "r"(parity) : "memory");
    return done != 0;
}

// Bounded wait for the phase with the given parity; returns false on timeout.
__device__ __forceinline__ bool mbar_wait(uint32_t mbar, uint32_t parity, uint32_t max_iters) {
    for (uint32_t it = 0; it < max_iters; ++it)
        if (mbar_try_wait(mbar, parity)) return true;
    return false;
}

__device__ __forceinline__ void fence_before_sync() { asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory"); }
// Named barrier kId (1 .. 15; 0 is the one __syncthreads uses) over kN threads (a multiple of 32):
// the arriving warps go on, the syncing ones wait until all n have arrived, and see the shared
// memory the arriving ones wrote before arriving.
template <int kId, int kN>
__device__ __forceinline__ void named_bar_arrive() { asm volatile("bar.arrive %0, %1;" ::"n"(kId), "n"(kN) : "memory"); }
template <int kId, int kN>
__device__ __forceinline__ void named_bar_sync() { asm volatile("bar.sync %0, %1;" ::"n"(kId), "n"(kN) : "memory"); }
__device__ __forceinline__ void fence_after_sync() { asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory"); }
// Make this thread's generic-proxy shared-memory writes visible to the tensor core.
__device__ __forceinline__ void fence_smem_to_async() { asm volatile("fence.proxy.async.shared::cta;" ::: "memory"); }

__device__ __forceinline__ void tmem_alloc(uint32_t dst_smem, uint32_t ncols) {
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(dst_smem), "r"(ncols));
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;");
}
__device__ __forceinline__ void tmem_dealloc(uint32_t taddr, uint32_t ncols) {
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(ncols));
}

// 32 consecutive fp32 columns of this thread's TMEM lane (warp-wide).
__device__ __forceinline__ void tmem_ld32(uint32_t taddr, float (&v)[32]) {
    uint32_t r[32];
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x32.b32 "
        "{%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,"
        "%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31}, [%32];\n"
        : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]),
          "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15]),
          "=r"(r[16]), "=r"(r[17]), "=r"(r[18]), "=r"(r[19]), "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]),
          "=r"(r[24]), "=r"(r[25]), "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]), "=r"(r[31])
        : "r"(taddr));
    asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
#pragma unroll
    for (int i = 0; i < 32; ++i) v[i] = __uint_as_float(r[i]);
}

// 16 consecutive fp32 columns of this thread's TMEM lane (warp-wide).
__device__ __forceinline__ void tmem_ld16(uint32_t taddr, float (&v)[16]) {
    uint32_t r[16];
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x16.b32 "
        "{%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15}, [%16];\n"
        : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]),
          "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15])
        : "r"(taddr));
    asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
#pragma unroll
    for (int i = 0; i < 16; ++i) v[i] = __uint_as_float(r[i]);
}

// 16 consecutive fp32 columns of this thread's TMEM lane (warp-wide store).
__device__ __forceinline__ void tmem_st16(uint32_t taddr, const float (&v)[16]) {
    asm volatile(
        "tcgen05.st.sync.aligned.32x32b.x16.b32 [%0], "
        "{%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16};\n"
        ::"r"(taddr),
          "r"(__float_as_uint(v[0])), "r"(__float_as_uint(v[1])), "r"(__float_as_uint(v[2])), "r"(__float_as_uint(v[3])),
          "r"(__float_as_uint(v[4])), "r"(__float_as_uint(v[5])), "r"(__float_as_uint(v[6])), "r"(__float_as_uint(v[7])),
          "r"(__float_as_uint(v[8])), "r"(__float_as_uint(v[9])), "r"(__float_as_uint(v[10])), "r"(__float_as_uint(v[11])),
          "r"(__float_as_uint(v[12])), "r"(__float_as_uint(v[13])), "r"(__float_as_uint(v[14])), "r"(__float_as_uint(v[15])));
    asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory");
}

// 8 consecutive 32-bit columns of this thread's TMEM lane (warp-wide store).
__device__ __forceinline__ void tmem_st8(uint32_t taddr, const float (&v)[8]) {
    asm volatile(
        "tcgen05.st.sync.aligned.32x32b.x8.b32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8};\n"
        ::"r"(taddr),
          "r"(__float_as_uint(v[0])), "r"(__float_as_uint(v[1])), "r"(__float_as_uint(v[2])), "r"(__float_as_uint(v[3])),
          "r"(__float_as_uint(v[4])), "r"(__float_as_uint(v[5])), "r"(__float_as_uint(v[6])), "r"(__float_as_uint(v[7])));
    asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory");
}

__device__ __forceinline__ void tmem_st32(uint32_t taddr, const float (&v)[32]) {
    asm volatile(
        "tcgen05.st.sync.aligned.32x32b.x32.b32 [%0], "
        "{%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16,"
        "%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31,%32};\n"
        ::"r"(taddr),
          "r"(__float_as_uint(v[0])), "r"(__float_as_uint(v[1])), "r"(__float_as_uint(v[2])), "r"(__float_as_uint(v[3])),
          "r"(__float_as_uint(v[4])), "r"(__float_as_uint(v[5])), "r"(__float_as_uint(v[6])), "r"(__float_as_uint(v[7])),
          "r"(__float_as_uint(v[8])), "r"(__float_as_uint(v[9])), "r"(__float_as_uint(v[10])), "r"(__float_as_uint(v[11])),
          "r"(__float_as_uint(v[12])), "r"(__float_as_uint(v[13])), "r"(__float_as_uint(v[14])), "r"(__float_as_uint(v[15])),
          "r"(__float_as_uint(v[16])), "r"(__float_as_uint(v[17])), "r"(__float_as_uint(v[18])), "r"(__float_as_uint(v[19])),
          "r"(__float_as_uint(v[20])), "r"(__float_as_uint(v[21])), "r"(__float_as_uint(v[22])), "r"(__float_as_uint(v[23])),
          "r"(__float_as_uint(v[24])), "r"(__float_as_uint(v[25])), "r"(__float_as_uint(v[26])), "r"(__float_as_uint(v[27])),
          "r"(__float_as_uint(v[28])), "r"(__float_as_uint(v[29])), "r"(__float_as_uint(v[30])), "r"(__float_as_uint(v[31])));
    asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory");
}

}  // namespace tc05
}  // namespace cgdr
