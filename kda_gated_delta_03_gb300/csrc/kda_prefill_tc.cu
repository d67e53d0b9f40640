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
// TMEM lane, splitting the columns); thread 0 issues the tcgen05 MMAs.  The next chunk's rows are fetched with bulk copies (one per row,
// completing on an mbarrier) while the current chunk runs its state-dependent GEMMs.  Every wait on an MMA
// completion is bounded; on timeout the CTA records KDA_DEVERR_TIMEOUT, frees
// its TMEM and stops.

#include "kda_tc_util.cuh"

namespace kda {
namespace {

// region X: G1 factors -> solve tiles -> bf16 W and Gamma.Q operands
constexpr int X_R = 0, X_LK = C * F_LD * 4, X_LQ = X_LK + 16 * F_LD * 4;
constexpr int X_A = 0, X_T = C * AT_LD * 4, X_SCR = 2 * C * AT_LD * 4;
constexpr int X_W = 0, X_QT = 16384;
constexpr int X_BYTES = 51200;
// region Y: T' and [Gamma.K | V]^T operands -> Khat^T and U^T operands
constexpr int Y_T = 0, Y_KV = 16384;
constexpr int Y_KH = 0, Y_U = 32768;
// misc
constexpr int M_MBAR = 0, M_TMEM = 8, M_ABORT = 12, M_LBAR = 16, M_GAMC = 64;

// Everything that depends on the number NV of value columns a CTA carries (32 or 64).
template <int NV>
struct Cfg {
    static constexpr int CPT = NV / 2;                                   // columns per thread in epilogues
    static constexpr int OFF_BETA = OFF_V + C * NV * 2;
    static constexpr int OFF_ASC = OFF_BETA + 256;                      // per-head alpha of the chunk's rows
    static constexpr int OFF_S = align1k(OFF_ASC + 256);                // S^T operand (bf16, NV x 128)
    static constexpr int OFF_MISC = OFF_S + NV * DK * 2;
    static constexpr int OFF_X = align1k(OFF_MISC + 64 + DK * 4);
    static constexpr int Y_BYTES = (16384 + (DK + NV) * 256) > (32768 + NV * 256) ? (16384 + (DK + NV) * 256)
                                                                                 : (32768 + NV * 256);
    static constexpr int OFF_Y = OFF_X + X_BYTES;
    static constexpr int OFF_P = OFF_Y + Y_BYTES;                        // P operand (TF32, 64 x 64)
    // With 32 value columns the A/P products run on tcgen05: their TF32 operands (per row block b,
    // R_b with 16(b+1) rows and [Lk_b; Lq_b] with 32 rows) span X, Y and P while they are live.
    static constexpr bool TC_AP = (NV == 32);
    static constexpr int SMEM_BYTES =
        (TC_AP && OFF_X + G1_BYTES > OFF_P + 16384) ? OFF_X + G1_BYTES : OFF_P + 16384;
    static constexpr uint32_t TX_BYTES = 2 * 16384 + 32768 + C * NV * 2; // bytes one chunk's TMA loads deliver
    // TMEM columns: [W | Utilde] (M=64), X and O (M=64), the state update (M=128)
    static constexpr uint32_t TM_WU = 0, TM_X = DK + NV, TM_O = TM_X + NV, TM_S = TM_O + NV;
    static constexpr uint32_t TM_COLS = (TM_S + NV) <= 256 ? 256 : 512;
    static_assert(SMEM_BYTES <= 232448, "shared memory");
    static_assert(OFF_V % 1024 == 0 && OFF_X % 1024 == 0, "alignment");
};

static_assert(X_LQ + 16 * F_LD * 4 <= X_BYTES && X_SCR + 3 * 256 * 4 <= X_BYTES && X_QT + 16384 <= X_BYTES, "region X");

struct Tile {
    const float* beta;
    const float* alpha;   // per-head alpha (KDA_ALPHA_PER_HEAD), else unused
    int alpha_mode;
    int H;
    int h;
    int j0;
};

// Fetch the raw rows of the chunk starting at token t0: one thread issues the 9 TMA box loads
// (completing on `lbar`); beta (strided by H) goes through 4-byte cp.async with zero fill.  Rows at
// or past the sequence end are zeroed by the consumer.
template <int NV>
__device__ __forceinline__ void issue_chunk_loads(unsigned char* sm, const TcMaps& m, const Tile& g, int32_t t0,
                                                  int L, int tid, uint32_t lbar) {
    const bool per_channel = g.alpha_mode == KDA_ALPHA_PER_CHANNEL;
    if (tid == 32) {
        mbar_expect_tx(lbar, Cfg<NV>::TX_BYTES - (per_channel ? 0u : 32768u));
        tma_load_3d(saddr(sm + OFF_K), &m.k, 0, g.h, t0, lbar);
        tma_load_3d(saddr(sm + OFF_K + 8192), &m.k, 64, g.h, t0, lbar);
        tma_load_3d(saddr(sm + OFF_Q), &m.q, 0, g.h, t0, lbar);
        tma_load_3d(saddr(sm + OFF_Q + 8192), &m.q, 64, g.h, t0, lbar);
        if (per_channel) {
#pragma unroll
            for (int b = 0; b < 4; ++b) tma_load_3d(saddr(sm + OFF_G + b * 8192), &m.a, 32 * b, g.h, t0, lbar);
        }
        tma_load_3d(saddr(sm + OFF_V), &m.v, g.j0, g.h, t0, lbar);
    }
    for (int r = tid; r < C; r += NT) {
        const bool ok = r < L;
        const int64_t row = ok ? ((int64_t)(t0 + r) * g.H + g.h) : 0;
        cp_async4(saddr(sm + Cfg<NV>::OFF_BETA + r * 4), g.beta + row, ok);
        if (g.alpha_mode == KDA_ALPHA_PER_HEAD) cp_async4(saddr(sm + Cfg<NV>::OFF_ASC + r * 4), g.alpha + row, ok);
    }
    cp_async_commit();
}

template <int NV>
__global__ void __launch_bounds__(NT, 1) kda_prefill_tc_kernel(PrefillParams p, const __grid_constant__ TcMaps maps) {
    using CF = Cfg<NV>;
    constexpr int CPT = CF::CPT;
    constexpr int OFF_BETA = CF::OFF_BETA, OFF_X = CF::OFF_X, OFF_Y = CF::OFF_Y, OFF_P = CF::OFF_P,
                  OFF_S = CF::OFF_S, OFF_MISC = CF::OFF_MISC;
    constexpr uint32_t TM_WU = CF::TM_WU, TM_X = CF::TM_X, TM_O = CF::TM_O, TM_S = CF::TM_S, TM_COLS = CF::TM_COLS;
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
    if (tid == 0 && h == 0 && slice == 0 && snapshot_offsets_bad(p, n, t_end - t_begin))
        atomicOr(p.err, KDA_DEVERR_SNAPSHOTS);
    const int H = p.H;
    Tile g{p.beta, p.alpha, p.alpha_mode, H, h, j0};
    __nv_bfloat16* go = static_cast<__nv_bfloat16*>(p.o);

    __nv_bfloat16* vraw = reinterpret_cast<__nv_bfloat16*>(sm + OFF_V);
    auto Gat = [&](int r, int i) -> float& { return *reinterpret_cast<float*>(sm + OFF_G + g_off(r, i)); };
    auto kat = [&](int r, int i) { return bf(reinterpret_cast<const __nv_bfloat16*>(sm + OFF_K + kq_off(r, i))); };
    auto qat = [&](int r, int i) { return bf(reinterpret_cast<const __nv_bfloat16*>(sm + OFF_Q + kq_off(r, i))); };
    float* sbeta = reinterpret_cast<float*>(sm + OFF_BETA);
    float* sgam = reinterpret_cast<float*>(sm + OFF_MISC + M_GAMC);
    unsigned char* X = sm + OFF_X;
    unsigned char* Y = sm + OFF_Y;
    unsigned char* opP = sm + OFF_P;
    volatile int* s_abort = reinterpret_cast<volatile int*>(sm + OFF_MISC + M_ABORT);
    uint32_t* s_tmem = reinterpret_cast<uint32_t*>(sm + OFF_MISC + M_TMEM);
    const uint32_t mbar = saddr(sm + OFF_MISC + M_MBAR);
    const uint32_t lbar = saddr(sm + OFF_MISC + M_LBAR);

    if (saddr(sm) & 1023u) {                          // the swizzled tiles need a 1 KiB-aligned base
        if (tid == 0) atomicOr(p.err, KDA_DEVERR_TIMEOUT);
        return;
    }

    // ---- set-up: barrier, TMEM, first loads ----
    if (tid == 0) {
        asm volatile("mbarrier.init.shared::cta.b64 [%0], 1;" ::"r"(mbar) : "memory");
        asm volatile("mbarrier.init.shared::cta.b64 [%0], 1;" ::"r"(lbar) : "memory");
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
        *s_abort = 0;
    }
    if (warp == 0) {
        asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(saddr(s_tmem)),
                     "r"(TM_COLS)
                     : "memory");
        asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
    }

    // state: key row srow, value columns CPT*half .. CPT*half+CPT-1 of this slice, float32 in registers
    const int srow = 32 * quad + lane;
    const int64_t state_off = (((int64_t)n * H + h) * DK + srow) * (int64_t)p.dv + j0 + CPT * half;
    float S[CPT];
#pragma unroll
    for (int j = 0; j < CPT; j += 4) {
        float4 v4 = p.state_in ? *reinterpret_cast<const float4*>(p.state_in + state_off + j)
                               : make_float4(0.f, 0.f, 0.f, 0.f);
        S[j] = v4.x; S[j + 1] = v4.y; S[j + 2] = v4.z; S[j + 3] = v4.w;
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *s_tmem;
    const uint32_t tlane = (uint32_t)(quad * 32) << 16;   // this warp's TMEM lane quadrant
    uint32_t phase = 0, lphase = 0;
    bool aborted = false;
    bool loads_pending = false;
    if (t_begin < t_end) {
        issue_chunk_loads<NV>(sm, maps, g, t_begin, min(C, t_end - t_begin), tid, lbar);
        loads_pending = true;
    }
#ifdef KDA_TEST_HOOKS
    if (p.test_stall) {                              // the first copies are in flight: give up a wait now
        if (tid == 0) {
            asm volatile("mbarrier.init.shared::cta.b64 [%0], 1;" ::"r"(saddr(sm + OFF_MISC + 24)) : "memory");
            asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
        }
        __syncthreads();
        if (!test_stall_wait(saddr(sm + OFF_MISC + 24))) {
            atomicOr(p.err, KDA_DEVERR_TIMEOUT);
            *s_abort = 1;
        }
        __syncthreads();
    }
#endif

    auto write_state_operand = [&]() {           // S^T as a bf16 operand; even lanes store key pairs
#pragma unroll
        for (int j = 0; j < CPT; ++j) {
            const float partner = __shfl_xor_sync(0xffffffffu, S[j], 1);
            if (!(lane & 1))
                *reinterpret_cast<uint32_t*>(sm + OFF_S + op_off_h(CPT * half + j, srow, DK)) = pack_bf16x2(S[j], partner);
        }
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
    for (int e = tid; e < C * C; e += NT) {             // P beyond each row block's columns is always zero
        const int r = e >> 6, s = e & 63;
        if (s >= 16 * ((r >> 4) + 1)) *reinterpret_cast<float*>(opP + op_off(r, s, C)) = 0.f;
    }

    for (int32_t t0 = t_begin; t0 < t_end && !aborted; t0 += C) {
        const int L = min(C, t_end - t0);
        cp_async_wait_all();
        if (!mbar_wait(lbar, lphase)) {
            atomicOr(p.err, KDA_DEVERR_TIMEOUT);
            *s_abort = 1;
        }
        lphase ^= 1u;
        loads_pending = false;
        __syncthreads();
        if (*s_abort) { aborted = true; break; }
        if (L < C) {                                    // zero the rows past the sequence end
            for (int e = tid; e < (C - L) * 16; e += NT) {
                const int r = L + (e >> 4), c = e & 15;      // 16-byte chunk c of row r (two boxes of 8)
                const int off = ((c >> 3) << 13) + (r << 7) + ((c & 7) << 4);
                *reinterpret_cast<uint4*>(sm + OFF_K + off) = make_uint4(0, 0, 0, 0);
                *reinterpret_cast<uint4*>(sm + OFF_Q + off) = make_uint4(0, 0, 0, 0);
                if (c < NV / 8) *reinterpret_cast<uint4*>(sm + OFF_V + r * NV * 2 + c * 16) = make_uint4(0, 0, 0, 0);
            }
            __syncthreads();
        }

        // ---- 1. g = running sum of clamped log2 alpha per key channel: each thread scans 32 rows,
        //         then the upper half adds the lower half's total ----
        {
            float la[32];
            const float* sasc = reinterpret_cast<const float*>(sm + CF::OFF_ASC);
#pragma unroll
            for (int x = 0; x < 32; ++x)
                la[x] = p.alpha_mode == KDA_ALPHA_PER_CHANNEL ? Gat(32 * rh + x, ch)
                        : p.alpha_mode == KDA_ALPHA_PER_HEAD  ? sasc[32 * rh + x]
                                                              : 1.f;
            float acc = 0.f;
#pragma unroll
            for (int x = 0; x < 32; ++x) {
                acc += (32 * rh + x < L) ? fmaxf(lg2f(la[x]), kLog2AlphaMin) : 0.f;
                la[x] = acc;
            }
#pragma unroll
            for (int x = 0; x < 32; ++x) Gat(32 * rh + x, ch) = la[x];
            __syncthreads();
            if (rh == 1) {
                const float base = Gat(31, ch);
#pragma unroll
                for (int x = 0; x < 32; ++x) Gat(32 + x, ch) = la[x] + base;
                sgam[ch] = ex2f(la[31] + base);
            }
        }
        __syncthreads();

        // ---- 2. A and P by 16-row blocks ----
        float* Ab = reinterpret_cast<float*>(X + X_A);
        float* Tb = reinterpret_cast<float*>(X + X_T);
        float* scr = reinterpret_cast<float*>(X + X_SCR);
        if constexpr (CF::TC_AP) {
            // Factors in one pass: thread (channel quad cq, row j within each 8-row group) keeps its rows'
            // k_s 2^(ref_b - g_s) across blocks (rescaled by 2^(ref_b - ref_{b-1}), never re-exponentiated)
            // and writes R_b (rows < 16(b+1)) and [Lk_b; Lq_b] as TF32 operands.
            const int cq = 4 * warp + (lane >> 3), j = lane & 7, i0 = 4 * cq;
            float4 rv[8];
            float4 refp = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
            for (int b = 0; b < 4; ++b) {
                const float4 ref = *reinterpret_cast<const float4*>(sm + OFF_G + g_off(16 * b + 7, i0));
                if (b > 0) {
                    const float4 f = make_float4(ex2f(ref.x - refp.x), ex2f(ref.y - refp.y), ex2f(ref.z - refp.z),
                                                 ex2f(ref.w - refp.w));
#pragma unroll
                    for (int gi = 0; gi < 2 * b; ++gi)
                        rv[gi] = make_float4(rv[gi].x * f.x, rv[gi].y * f.y, rv[gi].z * f.z, rv[gi].w * f.w);
                }
                refp = ref;
#pragma unroll
                for (int u = 0; u < 2; ++u) {                 // the two new rows of this thread in block b
                    const int gi = 2 * b + u, fr = 8 * gi + j;
                    const float4 gg = *reinterpret_cast<const float4*>(sm + OFF_G + g_off(fr, i0));
                    const uint2 kk = *reinterpret_cast<const uint2*>(sm + OFF_K + kq_off(fr, i0));
                    const uint2 qq = *reinterpret_cast<const uint2*>(sm + OFF_Q + kq_off(fr, i0));
                    const __nv_bfloat162* k2 = reinterpret_cast<const __nv_bfloat162*>(&kk);
                    const __nv_bfloat162* q2 = reinterpret_cast<const __nv_bfloat162*>(&qq);
                    const float kx = __low2float(k2[0]), ky = __high2float(k2[0]), kz = __low2float(k2[1]),
                                kw = __high2float(k2[1]);
                    rv[gi] = make_float4(kx * ex2f(ref.x - gg.x), ky * ex2f(ref.y - gg.y), kz * ex2f(ref.z - gg.z),
                                         kw * ex2f(ref.w - gg.w));
                    const float fx = ex2f(gg.x - ref.x), fy = ex2f(gg.y - ref.y), fz = ex2f(gg.z - ref.z),
                                fw = ex2f(gg.w - ref.w);
                    unsigned char* lb = X + G1_L_OFF + b * 16384;
                    *reinterpret_cast<float4*>(lb + op_off(8 * u + j, i0, DK)) =
                        make_float4(tf32r(kx * fx), tf32r(ky * fy), tf32r(kz * fz), tf32r(kw * fw));
                    *reinterpret_cast<float4*>(lb + op_off(16 + 8 * u + j, i0, DK)) =
                        make_float4(tf32r(__low2float(q2[0]) * fx), tf32r(__high2float(q2[0]) * fy),
                                    tf32r(__low2float(q2[1]) * fz), tf32r(__high2float(q2[1]) * fw));
                }
                unsigned char* rb = X + g1_r_off(b);
#pragma unroll
                for (int gi = 0; gi < 2 * (b + 1); ++gi)
                    *reinterpret_cast<float4*>(rb + op_off(8 * gi + j, i0, DK)) =
                        make_float4(tf32r(rv[gi].x), tf32r(rv[gi].y), tf32r(rv[gi].z), tf32r(rv[gi].w));
            }
            fence_async_smem();
            tc_fence_before();
            __syncthreads();
            // D_b = R_b [Lk_b; Lq_b]^T (M=64 rows s, N=32, K=128), the four blocks interleaved by k-step
            if (tid == 0) {
                tc_fence_after();
                constexpr uint32_t id = idesc_tf32(64, 32);
                uint64_t ad[4], bdsc[4];
#pragma unroll
                for (int b = 0; b < 4; ++b) {
                    ad[b] = op_desc(saddr(X + g1_r_off(b)), DK);
                    bdsc[b] = op_desc(saddr(X + G1_L_OFF + b * 16384), DK);
                }
#pragma unroll
                for (int ks = 0; ks < DK / 8; ++ks) {
#pragma unroll
                    for (int b = 0; b < 4; ++b)
                        umma_tf32_1(tmem + TM_WU + 32 * b, ad[b] + (uint64_t)(ks * 16), bdsc[b] + (uint64_t)(ks * 16), id,
                                    ks > 0 ? 1u : 0u);
                }
                umma_commit(mbar);
            }
            if (!wait_mma()) { aborted = true; break; }
            // scatter: A (fp32, for the solve) and P (TF32 operand); lane row s = 16*quad + lane
            {
                const int sr = 16 * quad + lane;
                float v[32];
#pragma unroll
                for (int bb = 0; bb < 2; ++bb) {
                    const int b = 2 * half + bb;
                    tmem_ld32(tmem + tlane + TM_WU + 32 * b, v);
                    if (lane < 16) {
#pragma unroll
                        for (int c = 0; c < 16; ++c) {
                            const int r = 16 * b + c;
                            Ab[r * AT_LD + sr] = sr < r ? sbeta[r] * v[c] : 0.f;
                            *reinterpret_cast<float*>(opP + op_off(r, sr, C)) = sr <= r ? v[16 + c] : 0.f;
                        }
                    }
                }
            }
            tc_fence_before();
            __syncthreads();
        } else {
        float* R = reinterpret_cast<float*>(X + X_R);
        float* Lk = reinterpret_cast<float*>(X + X_LK);
        float* Lq = reinterpret_cast<float*>(X + X_LQ);
        float res[6][4];
#pragma unroll
        for (int b = 0; b < 4; ++b) {
            {   // factors of block b: thread (channel, row half); all loads first, then math, then stores
                const float ref = Gat(16 * b + 7, ch);
                float gr[8], kv[8], qv[8];
#pragma unroll
                for (int x = 0; x < 8; ++x) {
                    const int r = 16 * b + 8 * rh + x;
                    gr[x] = Gat(r, ch);
                    kv[x] = kat(r, ch);
                    qv[x] = qat(r, ch);
                }
                if (b > 0) {
                    const float f = ex2f(ref - Gat(16 * b - 9, ch));
                    float old[24];
#pragma unroll
                    for (int x = 0; x < 8 * b; ++x) old[x] = R[(rh + 2 * x) * F_LD + ch];
#pragma unroll
                    for (int x = 0; x < 8 * b; ++x) R[(rh + 2 * x) * F_LD + ch] = tf32r(old[x] * f);
                }
#pragma unroll
                for (int x = 0; x < 8; ++x) {
                    const int rr = 8 * rh + x, r = 16 * b + rr;
                    const float f = ex2f(gr[x] - ref);
                    R[r * F_LD + ch] = tf32r(kv[x] * ex2f(ref - gr[x]));
                    Lk[rr * F_LD + ch] = tf32r(kv[x] * f);
                    Lq[rr * F_LD + ch] = tf32r(qv[x] * f);
                }
            }
            __syncthreads();
            const int base = b == 0 ? 0 : (b == 1 ? 1 : (b == 2 ? 2 : 4));
            const int ntiles = 2 * (b + 1);
            const bool has0 = warp < 4 * (b + 1);                 // combination (which, n-tile) = warp
            const bool has1 = b >= 2 && warp + 8 < 4 * (b + 1);    // second combination = warp + 8
            if (has0) {
                auto addrs = [&](int cidx, uint32_t& a_addr, uint32_t& b_addr) {
                    const float* Lf = cidx < ntiles ? Lk : Lq;
                    const int nt = cidx < ntiles ? cidx : cidx - ntiles;
                    a_addr = saddr(Lf + ((lane & 7) + ((lane >> 3) & 1) * 8) * F_LD + (lane >> 4) * 4);
                    b_addr = saddr(R + (8 * nt + (lane & 7)) * F_LD + (lane >> 3) * 4);
                };
                uint32_t a0a, b0a, a1a = 0, b1a = 0;
                addrs(warp, a0a, b0a);
                if (has1) addrs(warp + 8, a1a, b1a);
                float d[4][4] = {}, e4[4][4] = {};
#pragma unroll
                for (int kk = 0; kk < DK / 8; kk += 4) {            // 4 k-steps, 4 independent chains
                    const uint32_t off = kk * 32;                     // 8 fp32 per k-step
                    uint32_t fa[4][4], fb0[4], fb1[4];
#pragma unroll
                    for (int t = 0; t < 4; ++t) ldsm_x4(a0a + off + 32 * t, fa[t]);
                    ldsm_x4(b0a + off, fb0);
                    ldsm_x4(b0a + off + 64, fb1);
                    mma_16x8x8(d[0], fa[0][0], fa[0][1], fa[0][2], fa[0][3], fb0[0], fb0[1]);
                    mma_16x8x8(d[1], fa[1][0], fa[1][1], fa[1][2], fa[1][3], fb0[2], fb0[3]);
                    mma_16x8x8(d[2], fa[2][0], fa[2][1], fa[2][2], fa[2][3], fb1[0], fb1[1]);
                    mma_16x8x8(d[3], fa[3][0], fa[3][1], fa[3][2], fa[3][3], fb1[2], fb1[3]);
                    if (has1) {
#pragma unroll
                        for (int t = 0; t < 4; ++t) ldsm_x4(a1a + off + 32 * t, fa[t]);
                        ldsm_x4(b1a + off, fb0);
                        ldsm_x4(b1a + off + 64, fb1);
                        mma_16x8x8(e4[0], fa[0][0], fa[0][1], fa[0][2], fa[0][3], fb0[0], fb0[1]);
                        mma_16x8x8(e4[1], fa[1][0], fa[1][1], fa[1][2], fa[1][3], fb0[2], fb0[3]);
                        mma_16x8x8(e4[2], fa[2][0], fa[2][1], fa[2][2], fa[2][3], fb1[0], fb1[1]);
                        mma_16x8x8(e4[3], fa[3][0], fa[3][1], fa[3][2], fa[3][3], fb1[2], fb1[3]);
                    }
                }
#pragma unroll
                for (int e = 0; e < 4; ++e) {
                    res[base][e] = (d[0][e] + d[1][e]) + (d[2][e] + d[3][e]);
                    if (b >= 2) res[base + 1][e] = (e4[0][e] + e4[1][e]) + (e4[2][e] + e4[3][e]);
                }
            }
            __syncthreads();
        }
        // scatter: A (fp32, for the solve) and P (TF32 operand)
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
        __syncthreads();

        }

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
        // off-diagonal blocks, by distance d = b - c:  Z = sum_{c<=m<b} A_bm T_mc,  T_bc = -T_bb Z.
        // One warp per (block, 8-column tile), warp-level TF32 MMA; Z is staged per warp to become the
        // B operand of the second product.
        {
            float* zs = scr + warp * 128;
#pragma unroll
            for (int d = 1; d < 4; ++d) {
                if (warp < 2 * (4 - d)) {
                    const int c = warp >> 1, b = c + d, col0 = 16 * c + 8 * (warp & 1);
                    const int arow = (lane & 7) + ((lane >> 3) & 1) * 8, acol = (lane >> 4) * 4;
                    float z[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
                    for (int t = 0; t < d; ++t) {
                        const int m = c + t;
#pragma unroll
                        for (int ks = 0; ks < 2; ++ks) {
                            uint32_t a[4];
                            ldsm_x4(saddr(Ab + (16 * b + arow) * AT_LD + 16 * m + 8 * ks + acol), a);
                            const uint32_t b0 = __float_as_uint(Tb[(16 * m + 8 * ks + tig) * AT_LD + col0 + gid]);
                            const uint32_t b1 = __float_as_uint(Tb[(16 * m + 8 * ks + tig + 4) * AT_LD + col0 + gid]);
                            mma_16x8x8(z, a[0], a[1], a[2], a[3], b0, b1);
                        }
                    }
                    zs[gid * 8 + 2 * tig] = z[0];
                    zs[gid * 8 + 2 * tig + 1] = z[1];
                    zs[(gid + 8) * 8 + 2 * tig] = z[2];
                    zs[(gid + 8) * 8 + 2 * tig + 1] = z[3];
                    __syncwarp();
                    float tv[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
                    for (int ks = 0; ks < 2; ++ks) {
                        uint32_t a[4];
                        ldsm_x4(saddr(Tb + (16 * b + arow) * AT_LD + 16 * b + 8 * ks + acol), a);
                        const uint32_t b0 = __float_as_uint(zs[(8 * ks + tig) * 8 + gid]);
                        const uint32_t b1 = __float_as_uint(zs[(8 * ks + tig + 4) * 8 + gid]);
                        mma_16x8x8(tv, a[0], a[1], a[2], a[3], b0, b1);
                    }
                    Tb[(16 * b + gid) * AT_LD + col0 + 2 * tig] = -tv[0];
                    Tb[(16 * b + gid) * AT_LD + col0 + 2 * tig + 1] = -tv[1];
                    Tb[(16 * b + gid + 8) * AT_LD + col0 + 2 * tig] = -tv[2];
                    Tb[(16 * b + gid + 8) * AT_LD + col0 + 2 * tig + 1] = -tv[3];
                    __syncwarp();
                }
                __syncthreads();
            }
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
        // [Gamma.K | V]^T -> operand (N=160 rows, K=64 time); lanes run over channels
        for (int e = tid; e < DK * 16; e += 2 * NT) {       // two items per iteration
            const int i = e & (DK - 1), m0 = 4 * (e >> 7), m1 = m0 + 4 * (NT >> 7);
            float gg[8], kk8[8];
#pragma unroll
            for (int x = 0; x < 4; ++x) {
                gg[x] = Gat(m0 + x, i); kk8[x] = kat(m0 + x, i);
                gg[4 + x] = Gat(m1 + x, i); kk8[4 + x] = kat(m1 + x, i);
            }
            *reinterpret_cast<float4*>(Y + Y_KV + op_off(i, m0, C)) =
                make_float4(ex2f(gg[0]) * kk8[0], ex2f(gg[1]) * kk8[1], ex2f(gg[2]) * kk8[2], ex2f(gg[3]) * kk8[3]);
            *reinterpret_cast<float4*>(Y + Y_KV + op_off(i, m1, C)) =
                make_float4(ex2f(gg[4]) * kk8[4], ex2f(gg[5]) * kk8[5], ex2f(gg[6]) * kk8[6], ex2f(gg[7]) * kk8[7]);
        }
        for (int e = tid; e < NV * 16; e += NT) {
            const int j = e & (NV - 1), m0 = 4 * (e / NV);
            *reinterpret_cast<float4*>(Y + Y_KV + op_off(DK + j, m0, C)) =
                make_float4(bf(vraw + (m0 + 0) * NV + j), bf(vraw + (m0 + 1) * NV + j), bf(vraw + (m0 + 2) * NV + j),
                            bf(vraw + (m0 + 3) * NV + j));
        }
        fence_async_smem();
        __syncthreads();

        // ---- 4. [W | Utilde] = T' [Gamma.K | V]  (M=64, N=160, K=64) ----
        if (tid == 0) {
            tc_fence_after();
            umma_tf32<C>(tmem + TM_WU, saddr(Y + Y_T), saddr(Y + Y_KV), idesc_tf32(64, DK + NV), false);
            umma_commit(mbar);
        }
        if (!wait_mma()) { aborted = true; break; }

        // ---- 5. operands of the state-dependent GEMMs ----
        const int myrow = 16 * quad + lane;                // M=64 accumulator row of this lane (lane < 16)
        {
            float v[32];
#pragma unroll
            for (int cb = 0; cb < 2; ++cb) {
                const int c0 = 64 * half + 32 * cb;
                tmem_ld32(tmem + tlane + TM_WU + c0, v);
                if (lane < 16) {
#pragma unroll
                    for (int x = 0; x < 32; x += 8)
                        *reinterpret_cast<uint4*>(X + X_W + op_off_h(myrow, c0 + x, DK)) =
                            make_uint4(pack_bf16x2(v[x], v[x + 1]), pack_bf16x2(v[x + 2], v[x + 3]),
                                       pack_bf16x2(v[x + 4], v[x + 5]), pack_bf16x2(v[x + 6], v[x + 7]));
                }
            }
        }
        for (int e = tid; e < C * 16; e += NT) {            // Gamma . Q as bf16 (M=64, K=128), 8 channels per item
            const int r = ((e >> 7) << 3) | (e & 7), i0 = 8 * ((e >> 3) & 15);
            const float4 ga = *reinterpret_cast<const float4*>(sm + OFF_G + g_off(r, i0));
            const float4 gb = *reinterpret_cast<const float4*>(sm + OFF_G + g_off(r, i0 + 4));
            const uint4 qq = *reinterpret_cast<const uint4*>(sm + OFF_Q + kq_off(r, i0));
            const __nv_bfloat162* q2 = reinterpret_cast<const __nv_bfloat162*>(&qq);
            *reinterpret_cast<uint4*>(X + X_QT + op_off_h(r, i0, DK)) =
                make_uint4(pack_bf16x2(ex2f(ga.x) * __low2float(q2[0]), ex2f(ga.y) * __high2float(q2[0])),
                           pack_bf16x2(ex2f(ga.z) * __low2float(q2[1]), ex2f(ga.w) * __high2float(q2[1])),
                           pack_bf16x2(ex2f(gb.x) * __low2float(q2[2]), ex2f(gb.y) * __high2float(q2[2])),
                           pack_bf16x2(ex2f(gb.z) * __low2float(q2[3]), ex2f(gb.w) * __high2float(q2[3])));
        }
        for (int e = tid; e < DK * 16; e += 2 * NT) {       // Khat^T  (M=128 rows i, K=64 time), two items
            const int i = e & (DK - 1), s0 = 4 * (e >> 7), s1 = s0 + 4 * (NT >> 7);
            const float gl = Gat(C - 1, i);
            float gg[8], kk8[8];
#pragma unroll
            for (int x = 0; x < 4; ++x) {
                gg[x] = Gat(s0 + x, i); kk8[x] = kat(s0 + x, i);
                gg[4 + x] = Gat(s1 + x, i); kk8[4 + x] = kat(s1 + x, i);
            }
            *reinterpret_cast<float4*>(Y + Y_KH + op_off(i, s0, C)) =
                make_float4(ex2f(gl - gg[0]) * kk8[0], ex2f(gl - gg[1]) * kk8[1], ex2f(gl - gg[2]) * kk8[2],
                            ex2f(gl - gg[3]) * kk8[3]);
            *reinterpret_cast<float4*>(Y + Y_KH + op_off(i, s1, C)) =
                make_float4(ex2f(gl - gg[4]) * kk8[4], ex2f(gl - gg[5]) * kk8[5], ex2f(gl - gg[6]) * kk8[6],
                            ex2f(gl - gg[7]) * kk8[7]);
        }
        fence_async_smem();
        tc_fence_before();
        __syncthreads();
        // the raw tiles are free: fetch the next chunk while the state GEMMs run
        if (t0 + C < t_end) {
            issue_chunk_loads<NV>(sm, maps, g, t0 + C, min(C, t_end - t0 - C), tid, lbar);
            loads_pending = true;
        }

        // ---- 6. X = W S, O = (Gamma.Q) S ----
        if (tid == 0) {
            tc_fence_after();
            umma_bf16<DK>(tmem + TM_X, saddr(X + X_W), saddr(sm + OFF_S), idesc_bf16(64, NV), false);
            umma_bf16<DK>(tmem + TM_O, saddr(X + X_QT), saddr(sm + OFF_S), idesc_bf16(64, NV), false);
            umma_commit(mbar);
        }
        if (!wait_mma()) { aborted = true; break; }

        // ---- 7. U = Utilde - X  ->  U^T operand (N=32 rows j, K=64 time) ----
        {
            float ut[CPT], xv[CPT];
            tmem_ld<CPT>(tmem + tlane + TM_WU + DK + CPT * half, ut);     // Utilde stays in TMEM until here
            tmem_ld<CPT>(tmem + tlane + TM_X + CPT * half, xv);
            if (lane < 16) {
#pragma unroll
                for (int j = 0; j < CPT; ++j)
                    *reinterpret_cast<float*>(Y + Y_U + op_off(CPT * half + j, myrow, C)) = ut[j] - xv[j];
            }
        }
        fence_async_smem();
        tc_fence_before();
        __syncthreads();

        // ---- 8. O += P U,  D = Khat^T U ----
        if (tid == 0) {
            tc_fence_after();
            umma_tf32<C>(tmem + TM_O, saddr(opP), saddr(Y + Y_U), idesc_tf32(64, NV), true);
            umma_tf32<C>(tmem + TM_S, saddr(Y + Y_KH), saddr(Y + Y_U), idesc_tf32(128, NV), false);
            umma_commit(mbar);
        }
        if (!wait_mma()) { aborted = true; break; }

        // ---- 9. outputs and the carried state ----
        {
            float ov[CPT];
            tmem_ld<CPT>(tmem + tlane + TM_O + CPT * half, ov);
            if (lane < 16 && myrow < L) {
                __nv_bfloat16* dst = go + ((int64_t)(t0 + myrow) * H + h) * p.dv + j0 + CPT * half;
#pragma unroll
                for (int x = 0; x < CPT; x += 8) {
                    __align__(16) __nv_bfloat16 pk[8];
#pragma unroll
                    for (int y = 0; y < 8; ++y) pk[y] = __float2bfloat16_rn(p.scale * ov[x + y]);
                    *reinterpret_cast<uint4*>(dst + x) = *reinterpret_cast<const uint4*>(pk);
                }
            }
            float dsv[CPT];
            tmem_ld<CPT>(tmem + tlane + TM_S + CPT * half, dsv);
            const float gamC = sgam[srow];
#pragma unroll
            for (int j = 0; j < CPT; ++j) S[j] = fmaf(gamC, S[j], dsv[j]);
            write_state_operand();
            if (p.snap_every > 0) {                  // the state after this chunk, if a snapshot is due
                const int64_t slot = snapshot_slot(p, n, t0 + L - t_begin, t_end - t_begin);
                if (slot >= 0) {
                    float* dst = p.snapshots + ((slot * H + h) * DK + srow) * (int64_t)p.dv + j0 + CPT * half;
#pragma unroll
                    for (int j = 0; j < CPT; j += 4)
                        *reinterpret_cast<float4*>(dst + j) = make_float4(S[j], S[j + 1], S[j + 2], S[j + 3]);
                }
            }
        }
        fence_async_smem();
        tc_fence_before();
        __syncthreads();
    }

    // ---- state out, TMEM release ----
    if (!aborted) {
#pragma unroll
        for (int j = 0; j < CPT; j += 4)
            *reinterpret_cast<float4*>(p.state_out + state_off + j) = make_float4(S[j], S[j + 1], S[j + 2], S[j + 3]);
    }
    cp_async_wait_all();
    if (loads_pending) mbar_wait(lbar, lphase);         // bounded: never leave copies in flight
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

int prefill_tc_slices(int32_t num_seqs, int32_t H, int32_t dv) {
    // 64 value columns per CTA when there are enough (sequence, head) units to fill the GPU, otherwise 32
    return (int64_t)num_seqs * H >= 148 ? dv / 64 : dv / 32;
}

template <int NV>
cudaError_t launch_tc(const PrefillParams& p, cudaStream_t s) {
    TcMaps maps;
    std::memset(&maps, 0, sizeof maps);
    if (p.total_tokens > 0) {                        // with no tokens no CTA loads anything
        auto enc = tensor_map_encoder();
        if (!enc) return cudaErrorNotSupported;
        const int T = p.total_tokens;
        if (!encode_rows(enc, &maps.k, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, p.k, 2, DK, p.H, T, 64,
                         CU_TENSOR_MAP_SWIZZLE_128B) ||
            !encode_rows(enc, &maps.q, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, p.q, 2, DK, p.H, T, 64,
                         CU_TENSOR_MAP_SWIZZLE_128B) ||
            (p.alpha_mode == KDA_ALPHA_PER_CHANNEL &&
             !encode_rows(enc, &maps.a, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, p.alpha, 4, DK, p.H, T, 32,
                          CU_TENSOR_MAP_SWIZZLE_128B)) ||
            !encode_rows(enc, &maps.v, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, p.v, 2, p.dv, p.H, T, NV,
                         CU_TENSOR_MAP_SWIZZLE_NONE))
            return cudaErrorInvalidValue;
    }
    constexpr int SMEM_BYTES = Cfg<NV>::SMEM_BYTES;
    cudaError_t e = cudaFuncSetAttribute(kda_prefill_tc_kernel<NV>, cudaFuncAttributeMaxDynamicSharedMemorySize, SMEM_BYTES);
    if (e != cudaSuccess) return e;
    const int64_t blocks = (int64_t)p.num_seqs * p.H * p.slices;
    if (blocks <= 0) return cudaSuccess;
    if (blocks > 2147483647LL) return cudaErrorInvalidValue;
    kda_prefill_tc_kernel<NV><<<(unsigned)blocks, NT, SMEM_BYTES, s>>>(p, maps);
    return cudaGetLastError();
}

cudaError_t launch_prefill_tc(const PrefillParams& p, cudaStream_t s) {
    const int nv = p.dv / p.slices;
    if (nv == 64) return launch_tc<64>(p, s);
    if (nv == 32) return launch_tc<32>(p, s);
    return cudaErrorInvalidValue;
}

}  // namespace kda
