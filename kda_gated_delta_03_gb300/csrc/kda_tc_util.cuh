// Device and host helpers shared by the tcgen05 prefill kernels (fused and two-phase).
#pragma once

#include <cuda.h>
#include <cudaTypedefs.h>

#include <cstring>
#include <mutex>

#include "kda_internal.cuh"

namespace kda {
namespace {

constexpr int C = 64;
constexpr int DK = 128;
constexpr int NT = 256;
constexpr long long kWaitLimit = 4000000000LL;   // clock cycles (about 2 s)

// ---- shared memory map (bytes) ----
constexpr int F_LD = 132;                        // floats per A/P factor row
constexpr int AT_LD = 68;                        // floats per row of the 64x64 solve tiles
// raw tiles, written by TMA: k, q as two 128B-swizzled boxes of 64 rows x 64 bf16, alpha (then g) as
// four 128B-swizzled boxes of 64 rows x 32 fp32, then the v slice dense (64 rows x NV bf16)
constexpr int OFF_K = 0;
constexpr int OFF_Q = 16384;
constexpr int OFF_G = 32768;
constexpr int OFF_V = 65536;
constexpr int align1k(int x) { return (x + 1023) / 1024 * 1024; }

// tcgen05 A/P operands (offsets from region X): R_b at the running row offset 16*b*(b+1)/2 rows, each
// row 512 B of TF32 in K-major canonical layout; [Lk_b; Lq_b] (32 rows) after all R_b.
__host__ __device__ constexpr int g1_r_off(int b) { return 8192 * (b * (b + 1) / 2); }
constexpr int G1_L_OFF = 81920;
constexpr int G1_BYTES = G1_L_OFF + 4 * 16384;

// ---- small PTX helpers ----
__device__ __forceinline__ uint32_t saddr(const void* p) { return (uint32_t)__cvta_generic_to_shared(p); }

// Byte offset of element (row, k) of a K-major TF32 operand with K columns:
// core matrices of 8 rows x 16 B, K-adjacent ones 128 B apart, 8-row groups K*32 B apart.
__device__ __forceinline__ uint32_t op_off(int row, int k, int K) {
    return (uint32_t)((row >> 3) * (K * 32) + (k >> 2) * 128 + (row & 7) * 16 + (k & 3) * 4);
}

// Byte offsets inside the raw tiles (128-byte swizzle: 16-byte chunk c of row r sits at chunk c ^ (r & 7)).
__device__ __forceinline__ int g_off(int r, int i) {      // fp32 [64][128] as four 32-column boxes
    return ((i >> 5) << 13) + (r << 7) + ((((i & 31) >> 2) ^ (r & 7)) << 4) + ((i & 3) << 2);
}
__device__ __forceinline__ int kq_off(int r, int i) {     // bf16 [64][128] as two 64-column boxes
    return ((i >> 6) << 13) + (r << 7) + ((((i & 63) >> 3) ^ (r & 7)) << 4) + ((i & 7) << 1);
}

// Byte offset of element (row, k) of a K-major bf16 operand with K columns (core matrices of 8 rows x
// 8 elements; 8-row groups K*16 B apart).
__device__ __forceinline__ uint32_t op_off_h(int row, int k, int K) {
    return (uint32_t)((row >> 3) * (K * 16) + (k >> 3) * 128 + (row & 7) * 16 + (k & 7) * 2);
}

// Shared-memory matrix descriptor: K-major, no swizzle, K-adjacent core matrices 128 B apart,
// 8-row groups `sbo` bytes apart.
__device__ __forceinline__ uint64_t desc_sbo(uint32_t addr, uint32_t sbo) {
    return (uint64_t)((addr >> 4) & 0x3FFFu) | ((uint64_t)(128u >> 4) << 16) | ((uint64_t)((sbo >> 4) & 0x3FFFu) << 32) |
           (1ull << 46);
}
__device__ __forceinline__ uint64_t op_desc(uint32_t addr, int K) { return desc_sbo(addr, (uint32_t)K * 32u); }
// The same for a 16-bit operand (op_off_h layout: 8-row groups K*16 B apart).
__device__ __forceinline__ uint64_t op_desc_h(uint32_t addr, int K) { return desc_sbo(addr, (uint32_t)K * 16u); }

// K-major TF32 operand with 128-byte swizzle: atoms of 8 rows x 128 B (32 elements of K) on 1 KiB
// boundaries, 16-byte chunk c of atom row r stored at chunk c ^ r; row-groups 1 KiB apart, K-atoms
// N * 128 B apart.  A warp writing one row, K = 32 consecutive lanes, hits 32 distinct banks.
__device__ __forceinline__ uint32_t sw128_off(int row, int k, int N) {
    return (uint32_t)((k >> 5) * (N * 128) + (row >> 3) * 1024 + (row & 7) * 128 + ((((k & 31) >> 2) ^ (row & 7)) << 4) +
                      (k & 3) * 4);
}
// The same layout for 16-bit elements: an atom row holds 64 elements of K.
__device__ __forceinline__ uint32_t sw128_off_h(int row, int k, int N) {
    return (uint32_t)((k >> 6) * (N * 128) + (row >> 3) * 1024 + (row & 7) * 128 + ((((k & 63) >> 3) ^ (row & 7)) << 4) +
                      (k & 7) * 2);
}
// Descriptor of one 32-byte K-step of such an operand (8 TF32 or 16 fp16 elements): `addr` = base +
// K-atom offset + offset within the atom row.
__device__ __forceinline__ uint64_t desc_sw128(uint32_t addr) {
    return (uint64_t)((addr >> 4) & 0x3FFFu) | (1ull << 16) | ((uint64_t)(1024u >> 4) << 32) | (1ull << 46) |
           (2ull << 61);
}

// One lane of a converged warp (for issuing tcgen05 work from a warp that stays converged).
__device__ __forceinline__ bool elect_one() {
    uint32_t pred = 0;
    asm volatile("{\n.reg .pred p;\nelect.sync _|p, 0xffffffff;\nselp.u32 %0, 1, 0, p;\n}\n" : "=r"(pred));
    return pred != 0;
}

__host__ __device__ constexpr uint32_t idesc_bf16(int M, int N) {
    return (1u << 4) | (1u << 7) | (1u << 10) | ((uint32_t)(N >> 3) << 17) | ((uint32_t)(M >> 4) << 24);
}

__host__ __device__ constexpr uint32_t idesc_f16(int M, int N) {      // fp16 A and B, fp32 accumulator
    return (1u << 4) | ((uint32_t)(N >> 3) << 17) | ((uint32_t)(M >> 4) << 24);
}

__host__ __device__ constexpr uint32_t idesc_tf32(int M, int N) {
    return (1u << 4) | (2u << 7) | (2u << 10) | ((uint32_t)(N >> 3) << 17) | ((uint32_t)(M >> 4) << 24);
}

// One tcgen05.mma; the descriptors of successive k-steps differ only in the start-address field, so
// callers advance them by adding (bytes >> 4).
__device__ __forceinline__ void umma_tf32_1(uint32_t d_tmem, uint64_t a, uint64_t b, uint32_t idesc, uint32_t acc) {
    asm volatile(
        "{\n.reg .pred p;\nsetp.ne.b32 p, %4, 0;\n"
        "tcgen05.mma.cta_group::1.kind::tf32 [%0], %1, %2, %3, p;\n}\n" ::"r"(d_tmem),
        "l"(a), "l"(b), "r"(idesc), "r"(acc));
}
__device__ __forceinline__ void umma_bf16_1(uint32_t d_tmem, uint64_t a, uint64_t b, uint32_t idesc, uint32_t acc) {
    asm volatile(
        "{\n.reg .pred p;\nsetp.ne.b32 p, %4, 0;\n"
        "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n}\n" ::"r"(d_tmem),
        "l"(a), "l"(b), "r"(idesc), "r"(acc));
}
// kind::f16 with fp16 operands: the same instruction, the types are the instruction descriptor's.
__device__ __forceinline__ void umma_f16_1(uint32_t d_tmem, uint64_t a, uint64_t b, uint32_t idesc, uint32_t acc) {
    umma_bf16_1(d_tmem, a, b, idesc, acc);
}

// D (+)= A B^T with A [M x K] and B [N x K] K-major TF32 operands in shared memory (8 elements per step).
template <int K>
__device__ __forceinline__ void umma_tf32(uint32_t d_tmem, uint32_t a_addr, uint32_t b_addr, uint32_t idesc,
                                          bool accumulate) {
    const uint64_t a = op_desc(a_addr, K), b = op_desc(b_addr, K);
#pragma unroll
    for (int ks = 0; ks < K / 8; ++ks)
        umma_tf32_1(d_tmem, a + (uint64_t)(ks * 16), b + (uint64_t)(ks * 16), idesc, (accumulate || ks > 0) ? 1u : 0u);
}

// D (+)= A B^T with bf16 K-major operands (16 elements per step).
template <int K>
__device__ __forceinline__ void umma_bf16(uint32_t d_tmem, uint32_t a_addr, uint32_t b_addr, uint32_t idesc,
                                          bool accumulate) {
    const uint64_t a = desc_sbo(a_addr, (uint32_t)K * 16u), b = desc_sbo(b_addr, (uint32_t)K * 16u);
#pragma unroll
    for (int ks = 0; ks < K / 16; ++ks)
        umma_bf16_1(d_tmem, a + (uint64_t)(ks * 16), b + (uint64_t)(ks * 16), idesc, (accumulate || ks > 0) ? 1u : 0u);
}

__device__ __forceinline__ void umma_commit(uint32_t mbar) {
    asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(mbar)
                 : "memory");
}

__device__ __forceinline__ bool mbar_wait(uint32_t mbar, uint32_t parity, long long limit = kWaitLimit) {
    const long long t0 = clock64();
    while (true) {
        uint32_t done;
        asm volatile(
            "{\n.reg .pred p;\nmbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\nselp.u32 %0, 1, 0, p;\n}\n"
            : "=r"(done)
            : "r"(mbar), "r"(parity)
            : "memory");
        if (done) return true;
        if (clock64() - t0 > limit) return false;
    }
}

#ifdef KDA_TEST_HOOKS
// Test builds only (-DKDA_TEST_HOOKS): when PrefillParams::test_stall is set, a kernel waits on a barrier
// that nothing completes, with its first copies already in flight, so that the bounded wait gives up
// (after about 1 ms) and the kernel's abandon path runs: KDA_DEVERR_TIMEOUT, its copies drained, TMEM
// freed.  `never` is an mbarrier initialised with one pending arrival that no thread ever makes.
constexpr long long kTestStallLimit = 2000000LL;
__device__ __forceinline__ bool test_stall_wait(uint32_t never) { return mbar_wait(never, 0u, kTestStallLimit); }
#endif

__device__ __forceinline__ void fence_async_smem() { asm volatile("fence.proxy.async.shared::cta;" ::: "memory"); }
__device__ __forceinline__ void tc_fence_before() { asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory"); }
__device__ __forceinline__ void tc_fence_after() { asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory"); }

// 32 consecutive 32-bit TMEM columns of this thread's lane (warp w reads lanes 32w..32w+31).
__device__ __forceinline__ void tmem_ld32(uint32_t taddr, float* v) {
    uint32_t r[32];
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x32.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,"
        "%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31}, [%32];\n"
        "tcgen05.wait::ld.sync.aligned;\n"
        : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]),
          "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15]),
          "=r"(r[16]), "=r"(r[17]), "=r"(r[18]), "=r"(r[19]), "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]),
          "=r"(r[24]), "=r"(r[25]), "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]), "=r"(r[31])
        : "r"(taddr)
        : "memory");
#pragma unroll
    for (int i = 0; i < 32; ++i) v[i] = __uint_as_float(r[i]);
}

// Store 32 consecutive 32-bit TMEM columns of this thread's lane (warp w writes lanes 32(w%4)..+31); no wait:
// tmem_wait_st() completes a thread's stores before a barrier that orders them before tensor-core reads.
__device__ __forceinline__ void tmem_st32(uint32_t taddr, const float* v) {
    asm volatile(
        "tcgen05.st.sync.aligned.32x32b.x32.b32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16,"
        "%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31,%32};\n"
        :: "r"(taddr), "r"(__float_as_uint(v[0])), "r"(__float_as_uint(v[1])), "r"(__float_as_uint(v[2])),
          "r"(__float_as_uint(v[3])), "r"(__float_as_uint(v[4])), "r"(__float_as_uint(v[5])), "r"(__float_as_uint(v[6])),
          "r"(__float_as_uint(v[7])), "r"(__float_as_uint(v[8])), "r"(__float_as_uint(v[9])), "r"(__float_as_uint(v[10])),
          "r"(__float_as_uint(v[11])), "r"(__float_as_uint(v[12])), "r"(__float_as_uint(v[13])), "r"(__float_as_uint(v[14])),
          "r"(__float_as_uint(v[15])), "r"(__float_as_uint(v[16])), "r"(__float_as_uint(v[17])), "r"(__float_as_uint(v[18])),
          "r"(__float_as_uint(v[19])), "r"(__float_as_uint(v[20])), "r"(__float_as_uint(v[21])), "r"(__float_as_uint(v[22])),
          "r"(__float_as_uint(v[23])), "r"(__float_as_uint(v[24])), "r"(__float_as_uint(v[25])), "r"(__float_as_uint(v[26])),
          "r"(__float_as_uint(v[27])), "r"(__float_as_uint(v[28])), "r"(__float_as_uint(v[29])), "r"(__float_as_uint(v[30])),
          "r"(__float_as_uint(v[31]))
        : "memory");
}
// Store 16 consecutive 32-bit TMEM columns of this thread's lane (no wait).
__device__ __forceinline__ void tmem_st16(uint32_t taddr, const float* v) {
    asm volatile(
        "tcgen05.st.sync.aligned.32x32b.x16.b32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16};\n"
        :: "r"(taddr), "r"(__float_as_uint(v[0])), "r"(__float_as_uint(v[1])), "r"(__float_as_uint(v[2])),
          "r"(__float_as_uint(v[3])), "r"(__float_as_uint(v[4])), "r"(__float_as_uint(v[5])), "r"(__float_as_uint(v[6])),
          "r"(__float_as_uint(v[7])), "r"(__float_as_uint(v[8])), "r"(__float_as_uint(v[9])), "r"(__float_as_uint(v[10])),
          "r"(__float_as_uint(v[11])), "r"(__float_as_uint(v[12])), "r"(__float_as_uint(v[13])), "r"(__float_as_uint(v[14])),
          "r"(__float_as_uint(v[15]))
        : "memory");
}
__device__ __forceinline__ void tmem_wait_st() { asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory"); }

// Store 64 columns of 16 TMEM lanes (16x256b shape, eight 8-column blocks; no wait): lane (g, t) = (lane / 4,
// lane % 4) of the warp supplies v[4 j + 2 h + c] for TMEM lane g + 8 h (from the address's lane) and column
// 8 j + 2 t + c.  An M = 64 accumulator keeps its rows in lanes 0..15 of each quadrant, so all 32 threads
// carry rows the tensor core uses.
__device__ __forceinline__ void tmem_st16x256b_x8(uint32_t taddr, const float* v) {
    asm volatile(
        "tcgen05.st.sync.aligned.16x256b.x8.b32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16,"
        "%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31,%32};\n"
        :: "r"(taddr), "r"(__float_as_uint(v[0])), "r"(__float_as_uint(v[1])), "r"(__float_as_uint(v[2])),
          "r"(__float_as_uint(v[3])), "r"(__float_as_uint(v[4])), "r"(__float_as_uint(v[5])), "r"(__float_as_uint(v[6])),
          "r"(__float_as_uint(v[7])), "r"(__float_as_uint(v[8])), "r"(__float_as_uint(v[9])), "r"(__float_as_uint(v[10])),
          "r"(__float_as_uint(v[11])), "r"(__float_as_uint(v[12])), "r"(__float_as_uint(v[13])), "r"(__float_as_uint(v[14])),
          "r"(__float_as_uint(v[15])), "r"(__float_as_uint(v[16])), "r"(__float_as_uint(v[17])), "r"(__float_as_uint(v[18])),
          "r"(__float_as_uint(v[19])), "r"(__float_as_uint(v[20])), "r"(__float_as_uint(v[21])), "r"(__float_as_uint(v[22])),
          "r"(__float_as_uint(v[23])), "r"(__float_as_uint(v[24])), "r"(__float_as_uint(v[25])), "r"(__float_as_uint(v[26])),
          "r"(__float_as_uint(v[27])), "r"(__float_as_uint(v[28])), "r"(__float_as_uint(v[29])), "r"(__float_as_uint(v[30])),
          "r"(__float_as_uint(v[31]))
        : "memory");
}

// 16 consecutive 32-bit TMEM columns of this thread's lane.
__device__ __forceinline__ void tmem_ld16(uint32_t taddr, float* v) {
    uint32_t r[16];
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x16.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15}, [%16];\n"
        "tcgen05.wait::ld.sync.aligned;\n"
        : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]),
          "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15])
        : "r"(taddr)
        : "memory");
#pragma unroll
    for (int i = 0; i < 16; ++i) v[i] = __uint_as_float(r[i]);
}

// Hardware base-2 exponential and logarithm (PTX ex2.approx / lg2.approx, relative error ~2^-22,
// denormal results flushed to zero: an underflowed decay factor is an exact zero here).
__device__ __forceinline__ float ex2f(float x) {
    float y;
    asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}
__device__ __forceinline__ float lg2f(float x) {
    float y;
    asm("lg2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}

// 8 consecutive 32-bit TMEM columns of this thread's lane.
__device__ __forceinline__ void tmem_ld8(uint32_t taddr, float* v) {
    uint32_t r[8];
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x8.b32 {%0,%1,%2,%3,%4,%5,%6,%7}, [%8];\n"
        "tcgen05.wait::ld.sync.aligned;\n"
        : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7])
        : "r"(taddr)
        : "memory");
#pragma unroll
    for (int i = 0; i < 8; ++i) v[i] = __uint_as_float(r[i]);
}

template <int N>
__device__ __forceinline__ void tmem_ld(uint32_t taddr, float* v) {
    if constexpr (N == 8) {
        tmem_ld8(taddr, v);
    } else if constexpr (N == 16) {
        tmem_ld16(taddr, v);
    } else {
        static_assert(N == 32, "8, 16 or 32 columns");
        tmem_ld32(taddr, v);
    }
}

__device__ __forceinline__ uint32_t pack_bf16x2(float lo, float hi) {
    const __nv_bfloat162 h = __floats2bfloat162_rn(lo, hi);
    return *reinterpret_cast<const uint32_t*>(&h);
}

__device__ __forceinline__ uint32_t to_tf32(float x) {
    uint32_t r;
    asm("cvt.rna.tf32.f32 %0, %1;" : "=r"(r) : "f"(x));
    return r;
}

__device__ __forceinline__ void mma_16x8x8(float (&d)[4], uint32_t a0, uint32_t a1, uint32_t a2, uint32_t a3,
                                           uint32_t b0, uint32_t b1) {
    asm volatile(
        "mma.sync.aligned.m16n8k8.row.col.f32.tf32.tf32.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
        "{%0,%1,%2,%3};\n"
        : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
        : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}

__device__ __forceinline__ float tf32r(float x) { return __uint_as_float(to_tf32(x)); }

// Four 8x8 b16 matrices = four 8-row x 4-column fp32 tiles; lane l supplies the row address of tile l/8.
__device__ __forceinline__ void ldsm_x4(uint32_t addr, uint32_t (&r)[4]) {
    asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0,%1,%2,%3}, [%4];\n"
                 : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3])
                 : "r"(addr));
}

__device__ __forceinline__ void mbar_expect_tx(uint32_t mbar, uint32_t bytes) {
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(mbar), "r"(bytes) : "memory");
}

// TMA tile load of box (x, y, z) of a 3-D tensor map into shared memory, completing on an mbarrier.
__device__ __forceinline__ void tma_load_3d(uint32_t dst, const CUtensorMap* map, int x, int y, int z, uint32_t mbar) {
    asm volatile(
        "cp.async.bulk.tensor.3d.shared::cluster.global.tile.mbarrier::complete_tx::bytes [%0], [%1, {%2, %3, %4}], [%5];\n"
        ::"r"(dst), "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y), "r"(z), "r"(mbar)
        : "memory");
}

__device__ __forceinline__ void cp_async4(uint32_t dst, const void* src, bool valid) {
    asm volatile("cp.async.ca.shared.global [%0], [%1], 4, %2;\n" ::"r"(dst), "l"(src), "r"(valid ? 4 : 0)
                 : "memory");
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;\n" ::: "memory"); }
__device__ __forceinline__ void cp_async_wait_all() { asm volatile("cp.async.wait_group 0;\n" ::: "memory"); }

__device__ __forceinline__ float bf(const __nv_bfloat16* p) { return __bfloat162float(*p); }

// Tensor maps of the raw inputs: k, q [T, H, 128] bf16 (64-column boxes), alpha [T, H, 128] fp32
// (32-column boxes), v [T, H, d_v] bf16 (32-column box); each box is 64 tokens of one head.
struct TcMaps {
    CUtensorMap k, q, a, v;
};

PFN_cuTensorMapEncodeTiled_v12000 tensor_map_encoder() {
    static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
    static std::once_flag once;
    std::call_once(once, [] {
        void* ptr = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &ptr, 12000, cudaEnableDefault, &q) ==
                cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(ptr);
    });
    return fn;
}

// 3-D map over [T][H][cols] with a box of (box_cols, 1 head, 64 tokens).
bool encode_rows(PFN_cuTensorMapEncodeTiled_v12000 enc, CUtensorMap* m, CUtensorMapDataType dt, const void* base,
                 int esize, int cols, int H, int T, int box_cols, CUtensorMapSwizzle sw) {
    const cuuint64_t dims[3] = {(cuuint64_t)cols, (cuuint64_t)H, (cuuint64_t)T};
    const cuuint64_t strides[2] = {(cuuint64_t)cols * esize, (cuuint64_t)cols * esize * H};
    const cuuint32_t box[3] = {(cuuint32_t)box_cols, 1u, (cuuint32_t)C};
    const cuuint32_t estr[3] = {1u, 1u, 1u};
    return enc(m, dt, 3, const_cast<void*>(base), dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, sw,
               CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

}  // namespace
}  // namespace kda
