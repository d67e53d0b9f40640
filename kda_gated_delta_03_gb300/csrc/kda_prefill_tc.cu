// Chunkwise KDA prefill on the 5th-generation tensor cores: bf16 q/k/v, d_k = d_v = 128.
//
// Same chunkwise algebra as the CUDA-core kernel ("Kimi K3, explained", section
// "Training in chunks": WY form inside a chunk, only the state carried across
// chunks).  Per head, chunk of C = 64 tokens starting from state S (d_k x d_v),
// g = running sum of log2 alpha (per key channel), Gamma = 2^g:
//
//   A_rs = beta_r sum_i k_ri k_si 2^(g_ri - g_si)  (s < r),  P_rs likewise with q_r (s <= r)
//   T'   = (I + A)^-1 Diag(beta)                                 (blocked UT solve)
//   [W | Utilde] = T' [Gamma . K | V]                             tcgen05, M=64 N=160 K=64
//   X = W S,  O = (Gamma . Q) S                                   tcgen05, M=64 N=32 K=128
//   U = Utilde - X;  O += P U                                     tcgen05, M=64 N=32 K=64
//   S <- Diag(Gamma_C) S + Khat^T U                               tcgen05, M=128 N=32 K=64
//
// A and P are computed per 16-row block b with the decay split at the block's
// middle row (reference g_ref(b) = g at row 16b+7): k_ri 2^(g_ri - g_ref) times
// k_si 2^(g_ref - g_si).  Each block has its own reference, so these 16-row
// products run as warp-level m16n8k8 TF32 MMAs; every larger product runs on
// tcgen05 with float32 operands read as TF32 from shared memory (K-major, no
// swizzle: 8-row x 16-byte core matrices) and float32 accumulators in TMEM.
// Derived operands stay TF32/FP32 (only q, k, v are bf16), and the state is
// kept in float32 registers, one key row per pair of threads.
//
// One CTA = (sequence, head, 32 value columns); 256 threads (two threads per
// TMEM lane, splitting the columns); thread 0 issues the tcgen05 MMAs.  The next chunk's inputs are fetched with cp.async while
// the current chunk runs its state-dependent GEMMs.  Every wait on an MMA
// completion is bounded; on timeout the CTA records KDA_DEVERR_TIMEOUT, frees
// its TMEM and stops.

#include "kda_internal.cuh"

namespace kda {
namespace {

constexpr int C = 64;
constexpr int DK = 128;
constexpr int NV = 32;
constexpr int NT = 256;
constexpr long long kWaitLimit = 4000000000LL;   // clock cycles (about 2 s)

// ---- shared memory map (bytes) ----
constexpr int KQ_LD = 136;                       // bf16 per raw k / q row (272 B)
constexpr int G_LD = 132;                        // floats per log-decay row
constexpr int F_LD = 132;                        // floats per A/P factor row
constexpr int AT_LD = 68;                        // floats per row of the 64x64 solve tiles
constexpr int OFF_K = 0;
constexpr int OFF_Q = OFF_K + C * KQ_LD * 2;     // 17408
constexpr int OFF_G = OFF_Q + C * KQ_LD * 2;     // 34816
constexpr int OFF_BETA = OFF_G + C * G_LD * 4;   // 68608
constexpr int OFF_V = OFF_BETA + 256;            // 68864
constexpr int OFF_X = OFF_V + C * NV * 2;        // 72960  region X, 64 KiB
constexpr int OFF_Y = OFF_X + 65536;             // 138496 region Y, 56 KiB
constexpr int OFF_P = OFF_Y + 57344;             // 195840 P operand
constexpr int OFF_S = OFF_P + 16384;             // 212224 S^T operand
constexpr int OFF_MISC = OFF_S + 16384;          // 228608
constexpr int SMEM_BYTES = OFF_MISC + 64 + DK * 4;
// region X: G1 factors -> solve tiles -> W, Gamma.Q operands
constexpr int X_R = 0, X_LK = C * F_LD * 4, X_LQ = X_LK + 16 * F_LD * 4;
constexpr int X_A = 0, X_T = C * AT_LD * 4, X_SCR = 2 * C * AT_LD * 4;
constexpr int X_W = 0, X_QT = 32768;
// region Y: T' and [Gamma.K | V]^T operands -> Khat^T and U^T operands
constexpr int Y_T = 0, Y_KV = 16384;
constexpr int Y_KH = 0, Y_U = 32768;
// misc
constexpr int M_MBAR = 0, M_TMEM = 8, M_ABORT = 12, M_GAMC = 64;
// TMEM columns
constexpr uint32_t TM_WU = 0, TM_X = 160, TM_O = 192, TM_S = 224, TM_COLS = 256;

static_assert(X_LQ + 16 * F_LD * 4 <= 65536 && X_SCR + 3 * 256 * 4 <= 65536, "region X");
static_assert(SMEM_BYTES <= 232448, "shared memory");

// ---- small PTX helpers ----
__device__ __forceinline__ uint32_t saddr(const void* p) { return (uint32_t)__cvta_generic_to_shared(p); }

// Byte offset of element (row, k) of a K-major TF32 operand with K columns:
// core matrices of 8 rows x 16 B, K-adjacent ones 128 B apart, 8-row groups K*32 B apart.
__device__ __forceinline__ uint32_t op_off(int row, int k, int K) {
    return (uint32_t)((row >> 3) * (K * 32) + (k >> 2) * 128 + (row & 7) * 16 + (k & 3) * 4);
}

__device__ __forceinline__ uint64_t op_desc(uint32_t addr, int K) {
    return (uint64_t)((addr >> 4) & 0x3FFFu) | ((uint64_t)(128u >> 4) << 16) |
           ((uint64_t)(((uint32_t)K * 32u >> 4) & 0x3FFFu) << 32) | (1ull << 46);
}

__host__ __device__ constexpr uint32_t idesc_tf32(int M, int N) {
    return (1u << 4) | (2u << 7) | (2u << 10) | ((uint32_t)(N >> 3) << 17) | ((uint32_t)(M >> 4) << 24);
}

// D (+)= A B^T with A [M x K] and B [N x K] K-major TF32 operands in shared memory.
__device__ __forceinline__ void umma_tf32(uint32_t d_tmem, uint32_t a_addr, uint32_t b_addr, int K, uint32_t idesc,
                                          bool accumulate) {
    for (int ks = 0; ks < K / 8; ++ks) {
        const uint64_t a = op_desc(a_addr + ks * 256, K), b = op_desc(b_addr + ks * 256, K);
        const uint32_t acc = (accumulate || ks > 0) ? 1u : 0u;
        asm volatile(
            "{\n.reg .pred p;\nsetp.ne.b32 p, %4, 0;\n"
            "tcgen05.mma.cta_group::1.kind::tf32 [%0], %1, %2, %3, p;\n}\n" ::"r"(d_tmem),
            "l"(a), "l"(b), "r"(idesc), "r"(acc));
    }
}

__device__ __forceinline__ void umma_commit(uint32_t mbar) {
    asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(mbar)
                 : "memory");
}

__device__ __forceinline__ bool mbar_wait(uint32_t mbar, uint32_t parity) {
    const long long t0 = clock64();
    while (true) {
        uint32_t done;
        asm volatile(
            "{\n.reg .pred p;\nmbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\nselp.u32 %0, 1, 0, p;\n}\n"
            : "=r"(done)
            : "r"(mbar), "r"(parity)
            : "memory");
        if (done) return true;
        if (clock64() - t0 > kWaitLimit) return false;
    }
}

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

__device__ __forceinline__ void cp_async16(uint32_t dst, const void* src, bool valid) {
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;\n" ::"r"(dst), "l"(src), "r"(valid ? 16 : 0)
                 : "memory");
}
__device__ __forceinline__ void cp_async4(uint32_t dst, const void* src, bool valid) {
    asm volatile("cp.async.ca.shared.global [%0], [%1], 4, %2;\n" ::"r"(dst), "l"(src), "r"(valid ? 4 : 0)
                 : "memory");
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;\n" ::: "memory"); }
__device__ __forceinline__ void cp_async_wait_all() { asm volatile("cp.async.wait_group 0;\n" ::: "memory"); }

__device__ __forceinline__ float bf(const __nv_bfloat16* p) { return __bfloat162float(*p); }

struct Tile {
    const __nv_bfloat16* k;
    const __nv_bfloat16* q;
    const __nv_bfloat16* v;
    const float* alpha;
    const float* beta;
    int H;
    int h;
    int j0;
    int dv;
};

// Fetch the raw inputs of the chunk starting at token t0 (L valid rows; the rest zero-filled).
__device__ __forceinline__ void issue_chunk_loads(unsigned char* sm, const Tile& g, int32_t t0, int L, int tid) {
    for (int e = tid; e < C * 16; e += NT) {
        const int r = e >> 4, c = e & 15;
        const bool ok = r < L;
        const int64_t row = ok ? ((int64_t)(t0 + r) * g.H + g.h) : 0;
        cp_async16(saddr(sm + OFF_K + r * KQ_LD * 2 + c * 16), g.k + row * DK + c * 8, ok);
        cp_async16(saddr(sm + OFF_Q + r * KQ_LD * 2 + c * 16), g.q + row * DK + c * 8, ok);
    }
    for (int e = tid; e < C * 32; e += NT) {
        const int r = e >> 5, c = e & 31;
        const bool ok = r < L;
        const int64_t row = ok ? ((int64_t)(t0 + r) * g.H + g.h) : 0;
        cp_async16(saddr(sm + OFF_G + (r * G_LD + c * 4) * 4), g.alpha + row * DK + c * 4, ok);
    }
    for (int e = tid; e < C * 4; e += NT) {
        const int r = e >> 2, c = e & 3;
        const bool ok = r < L;
        const int64_t row = ok ? ((int64_t)(t0 + r) * g.H + g.h) : 0;
        cp_async16(saddr(sm + OFF_V + r * NV * 2 + c * 16), g.v + row * g.dv + g.j0 + c * 8, ok);
    }
    for (int r = tid; r < C; r += NT) {
        const bool ok = r < L;
        const int64_t row = ok ? ((int64_t)(t0 + r) * g.H + g.h) : 0;
        cp_async4(saddr(sm + OFF_BETA + r * 4), g.beta + row, ok);
    }
    cp_async_commit();
}

__global__ void __launch_bounds__(NT, 1) kda_prefill_tc_kernel(PrefillParams p) {
    extern __shared__ __align__(1024) unsigned char sm[];
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int gid = lane >> 2, tig = lane & 3;
    const int quad = warp & 3;             // TMEM lane quadrant this warp may access
    const int half = warp >> 2;            // which 16 of the 32 value columns this thread takes in epilogues
    const int ch = tid & (DK - 1);         // key channel of the per-channel stages
    const int rh = tid >> 7;               // row half of the per-channel stages

    // ---- work item ----
    const int item = blockIdx.x;
    const int slice = item % p.slices;
    const int rest = item / p.slices;
    const int h = rest % p.H;
    const int rank = rest / p.H;
    const int n = p.order ? p.order[rank] : rank;
    const int j0 = slice * NV;
    const int32_t t_begin = p.cu_seqlens[n];
    const int32_t t_end = p.cu_seqlens[n + 1];
    if (t_begin < 0 || t_end < t_begin || t_end > p.total_tokens || (n == 0 && t_begin != 0) ||
        (n == p.num_seqs - 1 && t_end != p.total_tokens)) {
        if (tid == 0) atomicOr(p.err, KDA_DEVERR_CU_SEQLENS);
        return;
    }
    const int H = p.H;
    Tile g{static_cast<const __nv_bfloat16*>(p.k), static_cast<const __nv_bfloat16*>(p.q),
           static_cast<const __nv_bfloat16*>(p.v), p.alpha, p.beta, H, h, j0, p.dv};
    __nv_bfloat16* go = static_cast<__nv_bfloat16*>(p.o);

    __nv_bfloat16* kraw = reinterpret_cast<__nv_bfloat16*>(sm + OFF_K);
    __nv_bfloat16* qraw = reinterpret_cast<__nv_bfloat16*>(sm + OFF_Q);
    __nv_bfloat16* vraw = reinterpret_cast<__nv_bfloat16*>(sm + OFF_V);
    float* G = reinterpret_cast<float*>(sm + OFF_G);
    float* sbeta = reinterpret_cast<float*>(sm + OFF_BETA);
    float* sgam = reinterpret_cast<float*>(sm + OFF_MISC + M_GAMC);
    unsigned char* X = sm + OFF_X;
    unsigned char* Y = sm + OFF_Y;
    unsigned char* opP = sm + OFF_P;
    volatile int* s_abort = reinterpret_cast<volatile int*>(sm + OFF_MISC + M_ABORT);
    uint32_t* s_tmem = reinterpret_cast<uint32_t*>(sm + OFF_MISC + M_TMEM);
    const uint32_t mbar = saddr(sm + OFF_MISC + M_MBAR);

    // ---- set-up: barrier, TMEM, first loads ----
    if (tid == 0) {
        asm volatile("mbarrier.init.shared::cta.b64 [%0], 1;" ::"r"(mbar) : "memory");
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
        *s_abort = 0;
    }
    if (warp == 0) {
        asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(saddr(s_tmem)),
                     "r"(TM_COLS)
                     : "memory");
        asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
    }
    if (t_begin < t_end) issue_chunk_loads(sm, g, t_begin, min(C, t_end - t_begin), tid);

    // state: key row srow, value columns 16*half .. 16*half+15 of this slice, float32 in registers
    const int srow = 32 * quad + lane;
    const int64_t state_off = (((int64_t)n * H + h) * DK + srow) * (int64_t)p.dv + j0 + 16 * half;
    float S[16];
#pragma unroll
    for (int j = 0; j < 16; j += 4) {
        float4 v4 = p.state_in ? *reinterpret_cast<const float4*>(p.state_in + state_off + j)
                               : make_float4(0.f, 0.f, 0.f, 0.f);
        S[j] = v4.x; S[j + 1] = v4.y; S[j + 2] = v4.z; S[j + 3] = v4.w;
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *s_tmem;
    const uint32_t tlane = (uint32_t)(quad * 32) << 16;   // this warp's TMEM lane quadrant
    uint32_t phase = 0;
    bool aborted = false;

    auto write_state_operand = [&]() {
#pragma unroll
        for (int j = 0; j < 16; ++j)
            *reinterpret_cast<float*>(sm + OFF_S + op_off(16 * half + j, srow, DK)) = S[j];
    };
    auto wait_mma = [&]() -> bool {
        if (!mbar_wait(mbar, phase)) {
            atomicOr(p.err, KDA_DEVERR_TIMEOUT);
            *s_abort = 1;
        }
        phase ^= 1u;
        __syncthreads();
        if (*s_abort) return false;
        tc_fence_after();
        return true;
    };
    write_state_operand();

    for (int32_t t0 = t_begin; t0 < t_end && !aborted; t0 += C) {
        const int L = min(C, t_end - t0);
        cp_async_wait_all();
        __syncthreads();

        // ---- 1. g = running sum of clamped log2 alpha per key channel: each thread scans 32 rows,
        //         then the upper half adds the lower half's total ----
        {
            float la[32];
#pragma unroll
            for (int x = 0; x < 32; ++x) la[x] = G[(32 * rh + x) * G_LD + ch];
            float acc = 0.f;
#pragma unroll
            for (int x = 0; x < 32; ++x) {
                acc += (32 * rh + x < L) ? fmaxf(lg2f(la[x]), kLog2AlphaMin) : 0.f;
                la[x] = acc;
            }
#pragma unroll
            for (int x = 0; x < 32; ++x) G[(32 * rh + x) * G_LD + ch] = la[x];
            __syncthreads();
            if (rh == 1) {
                const float base = G[31 * G_LD + ch];
#pragma unroll
                for (int x = 0; x < 32; ++x) G[(32 + x) * G_LD + ch] = la[x] + base;
                sgam[ch] = ex2f(la[31] + base);
            }
        }
        __syncthreads();

        // ---- 2. A and P by 16-row blocks (warp-level TF32 MMA, two accumulator chains each) ----
        float* R = reinterpret_cast<float*>(X + X_R);
        float* Lk = reinterpret_cast<float*>(X + X_LK);
        float* Lq = reinterpret_cast<float*>(X + X_LQ);
        float res[6][4];
#pragma unroll
        for (int b = 0; b < 4; ++b) {
            {   // factors of block b: thread (channel, row half)
                const float ref = G[(16 * b + 7) * G_LD + ch];
                if (b > 0) {
                    const float f = ex2f(ref - G[(16 * b - 9) * G_LD + ch]);
                    for (int s = rh; s < 16 * b; s += 2) R[s * F_LD + ch] *= f;
                }
#pragma unroll
                for (int x = 0; x < 8; ++x) {
                    const int rr = 8 * rh + x, r = 16 * b + rr;
                    const float gr = G[r * G_LD + ch];
                    const float kv = bf(kraw + r * KQ_LD + ch);
                    R[r * F_LD + ch] = kv * ex2f(ref - gr);
                    const float f = ex2f(gr - ref);
                    Lk[rr * F_LD + ch] = kv * f;
                    Lq[rr * F_LD + ch] = bf(qraw + r * KQ_LD + ch) * f;
                }
            }
            __syncthreads();
            const int base = b == 0 ? 0 : (b == 1 ? 1 : (b == 2 ? 2 : 4));
#pragma unroll
            for (int m = 0; m < 2; ++m) {
                const int cidx = warp + 8 * m;             // (which, n-tile) combination
                if (m <= (b >= 2 ? 1 : 0) && cidx < 4 * (b + 1)) {
                    const int ntiles = 2 * (b + 1);
                    const float* Lf = cidx < ntiles ? Lk : Lq;
                    const int nt = cidx < ntiles ? cidx : cidx - ntiles;
                    float d0[4] = {0.f, 0.f, 0.f, 0.f}, d1[4] = {0.f, 0.f, 0.f, 0.f};
                    const float* la0 = Lf + gid * F_LD + tig;
                    const float* la1 = Lf + (gid + 8) * F_LD + tig;
                    const float* rb = R + (8 * nt + gid) * F_LD + tig;
#pragma unroll 4
                    for (int kk = 0; kk < DK / 8; kk += 2) {
                        const int k0 = kk * 8, k1 = k0 + 8;
                        mma_16x8x8(d0, to_tf32(la0[k0]), to_tf32(la1[k0]), to_tf32(la0[k0 + 4]), to_tf32(la1[k0 + 4]),
                                   to_tf32(rb[k0]), to_tf32(rb[k0 + 4]));
                        mma_16x8x8(d1, to_tf32(la0[k1]), to_tf32(la1[k1]), to_tf32(la0[k1 + 4]), to_tf32(la1[k1 + 4]),
                                   to_tf32(rb[k1]), to_tf32(rb[k1 + 4]));
                    }
#pragma unroll
                    for (int e = 0; e < 4; ++e) res[base + m][e] = d0[e] + d1[e];
                }
            }
            __syncthreads();
        }
        // scatter: A (fp32, for the solve) and P (TF32 operand)
        float* Ab = reinterpret_cast<float*>(X + X_A);
        float* Tb = reinterpret_cast<float*>(X + X_T);
        float* scr = reinterpret_cast<float*>(X + X_SCR);
#pragma unroll
        for (int b = 0; b < 4; ++b) {
            const int base = b == 0 ? 0 : (b == 1 ? 1 : (b == 2 ? 2 : 4));
#pragma unroll
            for (int m = 0; m < 2; ++m) {
                const int cidx = warp + 8 * m;
                if (m <= (b >= 2 ? 1 : 0) && cidx < 4 * (b + 1)) {
                    const int ntiles = 2 * (b + 1);
                    const bool isk = cidx < ntiles;
                    const int nt = isk ? cidx : cidx - ntiles;
#pragma unroll
                    for (int e = 0; e < 4; ++e) {
                        const int r = 16 * b + gid + ((e & 2) ? 8 : 0);
                        const int s = 8 * nt + 2 * tig + (e & 1);
                        const float d = res[base + m][e];
                        if (isk)
                            Ab[r * AT_LD + s] = s < r ? sbeta[r] * d : 0.f;
                        else
                            *reinterpret_cast<float*>(opP + op_off(r, s, C)) = s <= r ? d : 0.f;
                    }
                }
            }
        }
        for (int e = tid; e < C * C; e += NT) {        // P beyond each row block's columns is zero
            const int r = e >> 6, s = e & 63;
            if (s >= 16 * ((r >> 4) + 1)) *reinterpret_cast<float*>(opP + op_off(r, s, C)) = 0.f;
        }
        __syncthreads();

        // ---- 3. T = (I + A)^-1 by 16x16 blocks ----
        if (tid < 64) {
            const int b = tid >> 4, c = tid & 15;
            float tc[16];
#pragma unroll
            for (int r = 0; r < 16; ++r) tc[r] = (r == c) ? 1.f : 0.f;
#pragma unroll
            for (int r = 1; r < 16; ++r) {
                float acc = 0.f;
#pragma unroll
                for (int m = 0; m < r; ++m) acc = fmaf(Ab[(16 * b + r) * AT_LD + 16 * b + m], tc[m], acc);
                if (r > c) tc[r] = -acc;
            }
#pragma unroll
            for (int r = 0; r < 16; ++r) Tb[(16 * b + r) * AT_LD + 16 * b + c] = tc[r];
        }
        __syncthreads();
        // off-diagonal blocks, by distance d = b - c
#pragma unroll
        for (int d = 1; d < 4; ++d) {
            const int nblk = 4 - d;
            for (int e = tid; e < nblk * 256; e += NT) {   // Z = sum_{c<=m<b} A_bm T_mc
                const int c = e >> 8, row = (e >> 4) & 15, col = e & 15;
                const int b = c + d;
                float acc0 = 0.f, acc1 = 0.f;
                for (int mb = c; mb < b; ++mb) {
#pragma unroll
                    for (int x = 0; x < 16; x += 2) {
                        acc0 = fmaf(Ab[(16 * b + row) * AT_LD + 16 * mb + x], Tb[(16 * mb + x) * AT_LD + 16 * c + col], acc0);
                        acc1 = fmaf(Ab[(16 * b + row) * AT_LD + 16 * mb + x + 1],
                                    Tb[(16 * mb + x + 1) * AT_LD + 16 * c + col], acc1);
                    }
                }
                scr[e] = acc0 + acc1;
            }
            __syncthreads();
            for (int e = tid; e < nblk * 256; e += NT) {   // T_bc = -T_bb Z
                const int c = e >> 8, row = (e >> 4) & 15, col = e & 15;
                const int b = c + d;
                float acc0 = 0.f, acc1 = 0.f;
#pragma unroll
                for (int x = 0; x < 16; x += 2) {
                    acc0 = fmaf(Tb[(16 * b + row) * AT_LD + 16 * b + x], scr[(c << 8) + (x << 4) + col], acc0);
                    acc1 = fmaf(Tb[(16 * b + row) * AT_LD + 16 * b + x + 1], scr[(c << 8) + ((x + 1) << 4) + col], acc1);
                }
                Tb[(16 * b + row) * AT_LD + 16 * c + col] = -(acc0 + acc1);
            }
            __syncthreads();
        }
        // T' = T Diag(beta) -> operand (M=64 rows r, K=64 cols m)
        for (int e = tid; e < C * 16; e += NT) {
            const int r = ((e >> 7) << 3) | (e & 7), q4 = (e >> 3) & 15;
            const int m0 = 4 * q4;
            float4 v;
            v.x = m0 + 0 <= r ? Tb[r * AT_LD + m0 + 0] * sbeta[m0 + 0] : 0.f;
            v.y = m0 + 1 <= r ? Tb[r * AT_LD + m0 + 1] * sbeta[m0 + 1] : 0.f;
            v.z = m0 + 2 <= r ? Tb[r * AT_LD + m0 + 2] * sbeta[m0 + 2] : 0.f;
            v.w = m0 + 3 <= r ? Tb[r * AT_LD + m0 + 3] * sbeta[m0 + 3] : 0.f;
            *reinterpret_cast<float4*>(Y + Y_T + op_off(r, m0, C)) = v;
        }
        // [Gamma.K | V]^T -> operand (N=160 rows, K=64 time)
        for (int e = tid; e < 160 * 16; e += NT) {
            const int nrow = ((e >> 7) << 3) | (e & 7), q4 = (e >> 3) & 15;
            const int m0 = 4 * q4;
            float4 v;
            if (nrow < DK) {
                const int i = nrow;
                v.x = ex2f(G[(m0 + 0) * G_LD + i]) * bf(kraw + (m0 + 0) * KQ_LD + i);
                v.y = ex2f(G[(m0 + 1) * G_LD + i]) * bf(kraw + (m0 + 1) * KQ_LD + i);
                v.z = ex2f(G[(m0 + 2) * G_LD + i]) * bf(kraw + (m0 + 2) * KQ_LD + i);
                v.w = ex2f(G[(m0 + 3) * G_LD + i]) * bf(kraw + (m0 + 3) * KQ_LD + i);
            } else {
                const int j = nrow - DK;
                v.x = bf(vraw + (m0 + 0) * NV + j);
                v.y = bf(vraw + (m0 + 1) * NV + j);
                v.z = bf(vraw + (m0 + 2) * NV + j);
                v.w = bf(vraw + (m0 + 3) * NV + j);
            }
            *reinterpret_cast<float4*>(Y + Y_KV + op_off(nrow, m0, C)) = v;
        }
        fence_async_smem();
        __syncthreads();

        // ---- 4. [W | Utilde] = T' [Gamma.K | V]  (M=64, N=160, K=64) ----
        if (tid == 0) {
            tc_fence_after();
            umma_tf32(tmem + TM_WU, saddr(Y + Y_T), saddr(Y + Y_KV), C, idesc_tf32(64, 160), false);
            umma_commit(mbar);
        }
        if (!wait_mma()) { aborted = true; break; }

        // ---- 5. operands of the state-dependent GEMMs ----
        float Ut[16];
        const int myrow = 16 * quad + lane;                // M=64 accumulator row of this lane (lane < 16)
        {
            float v[32];
#pragma unroll
            for (int cb = 0; cb < 2; ++cb) {
                const int c0 = 64 * half + 32 * cb;
                tmem_ld32(tmem + tlane + TM_WU + c0, v);
                if (lane < 16) {
#pragma unroll
                    for (int x = 0; x < 32; x += 4)
                        *reinterpret_cast<float4*>(X + X_W + op_off(myrow, c0 + x, DK)) =
                            make_float4(v[x], v[x + 1], v[x + 2], v[x + 3]);
                }
            }
            tmem_ld16(tmem + tlane + TM_WU + DK + 16 * half, Ut);
        }
        for (int e = tid; e < C * 32; e += NT) {            // Gamma . Q  (M=64, K=128)
            const int r = ((e >> 8) << 3) | (e & 7), q4 = (e >> 3) & 31;
            const int i0 = 4 * q4;
            const float4 gg = *reinterpret_cast<const float4*>(G + r * G_LD + i0);
            float4 v;
            v.x = ex2f(gg.x) * bf(qraw + r * KQ_LD + i0 + 0);
            v.y = ex2f(gg.y) * bf(qraw + r * KQ_LD + i0 + 1);
            v.z = ex2f(gg.z) * bf(qraw + r * KQ_LD + i0 + 2);
            v.w = ex2f(gg.w) * bf(qraw + r * KQ_LD + i0 + 3);
            *reinterpret_cast<float4*>(X + X_QT + op_off(r, i0, DK)) = v;
        }
        for (int e = tid; e < DK * 16; e += NT) {           // Khat^T  (M=128 rows i, K=64 time)
            const int i = ((e >> 7) << 3) | (e & 7), q4 = (e >> 3) & 15;
            const int s0 = 4 * q4;
            const float gl = G[(C - 1) * G_LD + i];
            float4 v;
            v.x = ex2f(gl - G[(s0 + 0) * G_LD + i]) * bf(kraw + (s0 + 0) * KQ_LD + i);
            v.y = ex2f(gl - G[(s0 + 1) * G_LD + i]) * bf(kraw + (s0 + 1) * KQ_LD + i);
            v.z = ex2f(gl - G[(s0 + 2) * G_LD + i]) * bf(kraw + (s0 + 2) * KQ_LD + i);
            v.w = ex2f(gl - G[(s0 + 3) * G_LD + i]) * bf(kraw + (s0 + 3) * KQ_LD + i);
            *reinterpret_cast<float4*>(Y + Y_KH + op_off(i, s0, C)) = v;
        }
        fence_async_smem();
        tc_fence_before();
        __syncthreads();
        // the raw tiles are free: fetch the next chunk while the state GEMMs run
        if (t0 + C < t_end) issue_chunk_loads(sm, g, t0 + C, min(C, t_end - t0 - C), tid);

        // ---- 6. X = W S, O = (Gamma.Q) S ----
        if (tid == 0) {
            tc_fence_after();
            umma_tf32(tmem + TM_X, saddr(X + X_W), saddr(sm + OFF_S), DK, idesc_tf32(64, NV), false);
            umma_tf32(tmem + TM_O, saddr(X + X_QT), saddr(sm + OFF_S), DK, idesc_tf32(64, NV), false);
            umma_commit(mbar);
        }
        if (!wait_mma()) { aborted = true; break; }

        // ---- 7. U = Utilde - X  ->  U^T operand (N=32 rows j, K=64 time) ----
        {
            float xv[16];
            tmem_ld16(tmem + tlane + TM_X + 16 * half, xv);
            if (lane < 16) {
#pragma unroll
                for (int j = 0; j < 16; ++j)
                    *reinterpret_cast<float*>(Y + Y_U + op_off(16 * half + j, myrow, C)) = Ut[j] - xv[j];
            }
        }
        fence_async_smem();
        tc_fence_before();
        __syncthreads();

        // ---- 8. O += P U,  D = Khat^T U ----
        if (tid == 0) {
            tc_fence_after();
            umma_tf32(tmem + TM_O, saddr(opP), saddr(Y + Y_U), C, idesc_tf32(64, NV), true);
            umma_tf32(tmem + TM_S, saddr(Y + Y_KH), saddr(Y + Y_U), C, idesc_tf32(128, NV), false);
            umma_commit(mbar);
        }
        if (!wait_mma()) { aborted = true; break; }

        // ---- 9. outputs and the carried state ----
        {
            float ov[16];
            tmem_ld16(tmem + tlane + TM_O + 16 * half, ov);
            if (lane < 16 && myrow < L) {
                __nv_bfloat16* dst = go + ((int64_t)(t0 + myrow) * H + h) * p.dv + j0 + 16 * half;
#pragma unroll
                for (int x = 0; x < 16; x += 8) {
                    __align__(16) __nv_bfloat16 pk[8];
#pragma unroll
                    for (int y = 0; y < 8; ++y) pk[y] = __float2bfloat16_rn(p.scale * ov[x + y]);
                    *reinterpret_cast<uint4*>(dst + x) = *reinterpret_cast<const uint4*>(pk);
                }
            }
            float dsv[16];
            tmem_ld16(tmem + tlane + TM_S + 16 * half, dsv);
            const float gamC = sgam[srow];
#pragma unroll
            for (int j = 0; j < 16; ++j) S[j] = fmaf(gamC, S[j], dsv[j]);
            write_state_operand();
        }
        fence_async_smem();
        tc_fence_before();
        __syncthreads();
    }

    // ---- state out, TMEM release ----
    if (!aborted) {
#pragma unroll
        for (int j = 0; j < 16; j += 4)
            *reinterpret_cast<float4*>(p.state_out + state_off + j) = make_float4(S[j], S[j + 1], S[j + 2], S[j + 3]);
    }
    cp_async_wait_all();
    tc_fence_before();
    __syncthreads();
    if (warp == 0) {
        tc_fence_after();
        asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem), "r"(TM_COLS) : "memory");
    }
}

}  // namespace

bool prefill_tc_supported(const PrefillParams& p, kda_dtype dt) {
    return dt == KDA_DTYPE_BF16 && p.dk == DK && p.dv == DK;
}

int prefill_tc_slices(int dv) { return dv / NV; }

cudaError_t launch_prefill_tc(const PrefillParams& p, cudaStream_t s) {
    cudaError_t e = cudaFuncSetAttribute(kda_prefill_tc_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, SMEM_BYTES);
    if (e != cudaSuccess) return e;
    const int64_t blocks = (int64_t)p.num_seqs * p.H * p.slices;
    if (blocks <= 0) return cudaSuccess;
    if (blocks > 2147483647LL) return cudaErrorInvalidValue;
    kda_prefill_tc_kernel<<<(unsigned)blocks, NT, SMEM_BYTES, s>>>(p);
    return cudaGetLastError();
}

}  // namespace kda
