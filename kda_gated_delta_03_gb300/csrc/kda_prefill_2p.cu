// Two-phase chunkwise prefill for a single long sequence: bf16 q/k/v, d_k = d_v = 128.
//
// The chunk algebra is that of the single-kernel path ("Kimi K3, explained", section "Training in
// chunks": WY form inside a chunk, only the state carried across chunks).  With U = Utilde - W S the
// chunk's output and state update are affine in the chunk-start state S:
//
//   O     = (Gamma.Q) S + P U            = Q' S + P Utilde,         Q' = Gamma.Q - P W
//   S_new = Diag(Gamma_C) S + Khat^T U   = Diag(Gamma_C) S + B - M S,  M = Khat^T W,  B = Khat^T Utilde
//
// Phase 1 computes, for every (head, chunk) of a window in parallel, everything that does not depend
// on S -- g, A and P, T' = (I + A)^-1 Diag(beta), [W | Utilde], and from them Q', M, B and P Utilde --
// and stores it as a record in the workspace, Q' and M already in the byte layout of a tensor-core
// operand.  Phase 2 walks the chunks in order, one CTA per (head, 32 value columns), bulk-loading each
// record one chunk ahead; per chunk it issues a single batch of tensor-core products,
//
//   [Q'; M_top] S  and  M S              tcgen05 kind::tf32, M=128, N=32, K=128
//
// followed by the fp32 update S <- Gamma_C . S + B - M S and o = scale (Q' S + P Utilde).  Folding W
// into M and Q' doubles phase 1's work on W but leaves one round trip through the tensor core on the
// sequential path instead of two, and no U tile to build between them.
//
// Long sequences are processed in windows of chunks so that the workspace stays bounded; the state
// passes between windows through state_out.  Every wait is bounded (KDA_DEVERR_TIMEOUT on expiry).

#include "kda_tc_util.cuh"

namespace kda {
namespace {

// ---- one (head, chunk) record in the workspace ----
constexpr int REC_QM = 0;          // [Q'; M]: 192 x 128 TF32 K-major operand (96 KiB)
constexpr int REC_B = 98304;       // B = Khat^T Utilde: fp32 [32 column quads][128 rows][4] (64 KiB)
constexpr int REC_O = 163840;      // P Utilde: fp32 [32 column quads][64 rows][4] (32 KiB)
constexpr int REC_G = 196608;      // Gamma_C: fp32 [128]
constexpr int REC_BYTES = 197120;
constexpr int QM_BYTES = (C + DK) * DK * 4;
constexpr int SNV = 32;            // value columns per chain CTA
constexpr int SLICES = DK / SNV;
constexpr size_t kWindowBudget = size_t(512) << 20;   // workspace bytes the records of one window may use
static_assert(QM_BYTES == REC_B && REC_B + DK * DK * 4 == REC_O && REC_O + C * DK * 4 == REC_G, "record layout");

// ---- phase 1 shared memory ----
constexpr int P_OFF_V = OFF_V;                     // v tile, dense 64 x 128 bf16
constexpr int P_OFF_BETA = OFF_V + C * DK * 2;     // 81920
constexpr int P_OFF_MISC = P_OFF_BETA + 256;
constexpr int P_OFF_S = align1k(P_OFF_MISC + 64 + DK * 4);   // scratch, 144 KiB
// scratch sub-regions (offsets from P_OFF_S)
constexpr int PS_A = 0, PS_T = C * AT_LD * 4, PS_SCR = 2 * C * AT_LD * 4;   // solve tiles
constexpr int PS_OPT = 38912, PS_KV = PS_OPT + 16384;                     // T' and [Gamma.K | V]^T (N = 256)
constexpr int PS_P = 122880;                                               // P operand
constexpr int PS_WU = 0, PS_KH = 65536;                                    // fold operands, after [W | Utilde]
constexpr int P_SMEM = P_OFF_S + G1_BYTES;
static_assert(PS_KV + (DK + DK) * 256 <= PS_P && PS_P + 16384 <= G1_BYTES, "phase-1 scratch");
static_assert(PS_KH + DK * C * 4 <= PS_P, "phase-1 fold operands");
static_assert(P_SMEM <= 232448, "phase-1 shared memory");

// ---- phase 2 shared memory ----
constexpr int C_OFF_S = 2 * QM_BYTES;              // S^T operand: TF32 32 x 128, 128-byte swizzle
constexpr int C_OFF_MISC = C_OFF_S + SNV * DK * 4;
constexpr int C_SMEM = C_OFF_MISC + 64;
static_assert(C_OFF_S % 1024 == 0 && C_SMEM <= 232448, "phase-2 shared memory");

struct PrepMaps {
    CUtensorMap k, q, a, v;   // v with a 128-column box
};

__device__ __forceinline__ void bulk_g2s(uint32_t dst, const void* src, uint32_t bytes, uint32_t mbar) {
    asm volatile("cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];\n" ::"r"(dst),
                 "l"(src), "r"(bytes), "r"(mbar)
                 : "memory");
}

__device__ __forceinline__ bool valid_single_sequence(const PrefillParams& p) {
    return p.num_seqs == 1 && p.cu_seqlens[0] == 0 && p.cu_seqlens[1] == p.total_tokens;
}

// ============================================================================================
// Phase 1: one CTA per (head, chunk) of the window [c_begin, c_begin + n_chunks).
// ============================================================================================
__global__ void __launch_bounds__(NT, 1)
    kda_prefill_prep_kernel(PrefillParams p, const __grid_constant__ PrepMaps maps, unsigned char* records,
                            int c_begin) {
    extern __shared__ __align__(1024) unsigned char sm[];
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int gid = lane >> 2, tig = lane & 3;
    const int quad = warp & 3, half = warp >> 2;
    const int ch = tid & (DK - 1), rh = tid >> 7;
    const int H = p.H;
    const int h = blockIdx.x % H, cw = blockIdx.x / H;
    const int32_t t0 = (int32_t)(c_begin + cw) * C;
    if (!valid_single_sequence(p)) {
        if (tid == 0) atomicOr(p.err, KDA_DEVERR_CU_SEQLENS);
        return;
    }
    if (t0 >= p.total_tokens) return;
    if (saddr(sm) & 1023u) {
        if (tid == 0) atomicOr(p.err, KDA_DEVERR_TIMEOUT);
        return;
    }
    const int L = min(C, p.total_tokens - t0);
    unsigned char* rec = records + (size_t)(cw * H + h) * REC_BYTES;

    const __nv_bfloat16* vraw = reinterpret_cast<const __nv_bfloat16*>(sm + P_OFF_V);
    float* sbeta = reinterpret_cast<float*>(sm + P_OFF_BETA);
    float* sgam = reinterpret_cast<float*>(sm + P_OFF_MISC + 64);
    unsigned char* X = sm + P_OFF_S;
    volatile int* s_abort = reinterpret_cast<volatile int*>(sm + P_OFF_MISC + 12);
    uint32_t* s_tmem = reinterpret_cast<uint32_t*>(sm + P_OFF_MISC + 8);
    const uint32_t mbar = saddr(sm + P_OFF_MISC), lbar = saddr(sm + P_OFF_MISC + 16);
    auto Gat = [&](int r, int i) -> float& { return *reinterpret_cast<float*>(sm + OFF_G + g_off(r, i)); };
    auto kat = [&](int r, int i) { return bf(reinterpret_cast<const __nv_bfloat16*>(sm + OFF_K + kq_off(r, i))); };

    if (tid == 0) {
        asm volatile("mbarrier.init.shared::cta.b64 [%0], 1;" ::"r"(mbar) : "memory");
        asm volatile("mbarrier.init.shared::cta.b64 [%0], 1;" ::"r"(lbar) : "memory");
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
        *s_abort = 0;
    }
    if (warp == 0) {
        asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(saddr(s_tmem)), "r"(512)
                     : "memory");
        asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *s_tmem;
    const uint32_t tlane = (uint32_t)(quad * 32) << 16;
    uint32_t phase = 0;
    bool ok = true;

    // ---- raw tiles by TMA (v with one 128-column box), beta by plain loads ----
    if (tid == 32) {
        mbar_expect_tx(lbar, 2 * 16384 + 32768 + C * DK * 2);
        tma_load_3d(saddr(sm + OFF_K), &maps.k, 0, h, t0, lbar);
        tma_load_3d(saddr(sm + OFF_K + 8192), &maps.k, 64, h, t0, lbar);
        tma_load_3d(saddr(sm + OFF_Q), &maps.q, 0, h, t0, lbar);
        tma_load_3d(saddr(sm + OFF_Q + 8192), &maps.q, 64, h, t0, lbar);
#pragma unroll
        for (int b = 0; b < 4; ++b) tma_load_3d(saddr(sm + OFF_G + b * 8192), &maps.a, 32 * b, h, t0, lbar);
        tma_load_3d(saddr(sm + P_OFF_V), &maps.v, 0, h, t0, lbar);
    }
    if (tid < C) sbeta[tid] = tid < L ? p.beta[(int64_t)(t0 + tid) * H + h] : 0.f;
    if (!mbar_wait(lbar, 0)) {
        atomicOr(p.err, KDA_DEVERR_TIMEOUT);
        *s_abort = 1;
    }
    __syncthreads();
    if (*s_abort) ok = false;
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
    do {
        if (!ok) break;
        if (L < C) {                                    // rows past the sequence end read as zero
            for (int e = tid; e < (C - L) * 16; e += NT) {
                const int r = L + (e >> 4), c = e & 15;
                const int off = ((c >> 3) << 13) + (r << 7) + ((c & 7) << 4);
                *reinterpret_cast<uint4*>(sm + OFF_K + off) = make_uint4(0, 0, 0, 0);
                *reinterpret_cast<uint4*>(sm + OFF_Q + off) = make_uint4(0, 0, 0, 0);
                *reinterpret_cast<uint4*>(sm + P_OFF_V + r * DK * 2 + c * 16) = make_uint4(0, 0, 0, 0);
            }
            __syncthreads();
        }

        // ---- 1. g = running sum of clamped log2 alpha per key channel ----
        {
            float la[32];
#pragma unroll
            for (int x = 0; x < 32; ++x) la[x] = Gat(32 * rh + x, ch);
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

        // ---- 2. A and P: per 16-row block b, R_b [Lk_b; Lq_b]^T on tcgen05 (M=64, N=32, K=128) ----
        float* Ab = reinterpret_cast<float*>(X + PS_A);
        float* Tb = reinterpret_cast<float*>(X + PS_T);
        float* scr = reinterpret_cast<float*>(X + PS_SCR);
        unsigned char* opP = X + PS_P;
        {
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
                for (int u = 0; u < 2; ++u) {
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
        }
        fence_async_smem();
        tc_fence_before();
        __syncthreads();
        if (warp == 0 && elect_one()) {
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
                    umma_tf32_1(tmem + 32 * b, ad[b] + (uint64_t)(ks * 16), bdsc[b] + (uint64_t)(ks * 16), id,
                                ks > 0 ? 1u : 0u);
            }
            umma_commit(mbar);
        }
        if (!wait_mma()) { ok = false; break; }
        {                                               // scatter: A (fp32) and P (TF32 operand)
            const int sr = 16 * quad + lane;
            float v[32];
#pragma unroll
            for (int bb = 0; bb < 2; ++bb) {
                const int b = 2 * half + bb;
                tmem_ld32(tmem + tlane + 32 * b, v);
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
        // T' = T Diag(beta) -> operand (M=64, K=64)
        for (int e = tid; e < C * 16; e += NT) {
            const int r = ((e >> 7) << 3) | (e & 7), m0 = 4 * ((e >> 3) & 15);
            float4 v;
            v.x = m0 + 0 <= r ? Tb[r * AT_LD + m0 + 0] * sbeta[m0 + 0] : 0.f;
            v.y = m0 + 1 <= r ? Tb[r * AT_LD + m0 + 1] * sbeta[m0 + 1] : 0.f;
            v.z = m0 + 2 <= r ? Tb[r * AT_LD + m0 + 2] * sbeta[m0 + 2] : 0.f;
            v.w = m0 + 3 <= r ? Tb[r * AT_LD + m0 + 3] * sbeta[m0 + 3] : 0.f;
            *reinterpret_cast<float4*>(X + PS_OPT + op_off(r, m0, C)) = v;
        }
        // [Gamma.K | V]^T -> operand (N=256 rows, K=64 time)
        for (int e = tid; e < DK * 16; e += NT) {
            const int i = e & (DK - 1), m0 = 4 * (e >> 7);
            float gg[4], kk4[4];
#pragma unroll
            for (int x = 0; x < 4; ++x) { gg[x] = Gat(m0 + x, i); kk4[x] = kat(m0 + x, i); }
            *reinterpret_cast<float4*>(X + PS_KV + op_off(i, m0, C)) =
                make_float4(ex2f(gg[0]) * kk4[0], ex2f(gg[1]) * kk4[1], ex2f(gg[2]) * kk4[2], ex2f(gg[3]) * kk4[3]);
            *reinterpret_cast<float4*>(X + PS_KV + op_off(DK + i, m0, C)) =
                make_float4(bf(vraw + (m0 + 0) * DK + i), bf(vraw + (m0 + 1) * DK + i), bf(vraw + (m0 + 2) * DK + i),
                            bf(vraw + (m0 + 3) * DK + i));
        }
        fence_async_smem();
        tc_fence_before();
        __syncthreads();

        // ---- 4. [W | Utilde] = T' [Gamma.K | V]  (M=64, N=256, K=64) ----
        if (warp == 0 && elect_one()) {
            tc_fence_after();
            umma_tf32<C>(tmem, saddr(X + PS_OPT), saddr(X + PS_KV), idesc_tf32(64, 2 * DK), false);
            umma_commit(mbar);
        }
        if (!wait_mma()) { ok = false; break; }

        // ---- 5. fold operands: [W | Utilde]^T (N=256, K=64, 128-byte swizzle) and Khat^T (M=128, K=64) ----
        unsigned char* opWU = X + PS_WU;
        unsigned char* opKH = X + PS_KH;
        {
            const int sr = 16 * quad + lane;                     // time row of this lane (lanes < 16)
            float v[32];
#pragma unroll
            for (int cb = 0; cb < 4; ++cb) {
                const int c0 = 128 * half + 32 * cb;
                tmem_ld32(tmem + tlane + c0, v);
                if (lane < 16) {
#pragma unroll
                    for (int x = 0; x < 32; ++x)
                        *reinterpret_cast<float*>(opWU + sw128_off(c0 + x, sr, 2 * DK)) = tf32r(v[x]);
                }
            }
        }
        for (int e = tid; e < DK * 16; e += NT) {
            const int i = e & (DK - 1), s0 = 4 * (e >> 7);
            const float gl = Gat(C - 1, i);
            float gg[4], kk4[4];
#pragma unroll
            for (int x = 0; x < 4; ++x) { gg[x] = Gat(s0 + x, i); kk4[x] = kat(s0 + x, i); }
            *reinterpret_cast<float4*>(opKH + op_off(i, s0, C)) =
                make_float4(tf32r(ex2f(gl - gg[0]) * kk4[0]), tf32r(ex2f(gl - gg[1]) * kk4[1]),
                            tf32r(ex2f(gl - gg[2]) * kk4[2]), tf32r(ex2f(gl - gg[3]) * kk4[3]));
        }
        fence_async_smem();
        tc_fence_before();
        __syncthreads();

        // ---- 6. [M | B] = Khat^T [W | Utilde] (M=128) and [PW | P Utilde] = P [W | Utilde] (M=64); N=256, K=64 ----
        if (warp == 0) {
            if (elect_one()) {
                tc_fence_after();
                const uint64_t ak = op_desc(saddr(opKH), C), ap = op_desc(saddr(opP), C);
                const uint32_t wb = saddr(opWU);
#pragma unroll
                for (int ks = 0; ks < C / 8; ++ks) {
                    const uint64_t bd = desc_sw128(wb + (ks >> 2) * (2 * DK * 128) + (ks & 3) * 32);
                    umma_tf32_1(tmem, ak + (uint64_t)(ks * 16), bd, idesc_tf32(128, 2 * DK), ks > 0 ? 1u : 0u);
                    umma_tf32_1(tmem + 2 * DK, ap + (uint64_t)(ks * 16), bd, idesc_tf32(64, 2 * DK), ks > 0 ? 1u : 0u);
                }
                umma_commit(mbar);
            }
            __syncwarp();
        }
        if (!wait_mma()) { ok = false; break; }

        // ---- 7. the record, from TMEM straight to global memory ----
        {
            const int i = 32 * quad + lane;                      // M=128 accumulator row
            const int r = 16 * quad + lane;                      // M=64 accumulator row (lanes < 16)
            float v[32];
#pragma unroll
            for (int cb = 0; cb < 2; ++cb) {                     // M = Khat^T W -> rows 64.. of [Q'; M]
                const int c0 = 64 * half + 32 * cb;
                tmem_ld32(tmem + tlane + c0, v);
#pragma unroll
                for (int x = 0; x < 32; x += 4)
                    *reinterpret_cast<float4*>(rec + REC_QM + op_off(C + i, c0 + x, DK)) =
                        make_float4(tf32r(v[x]), tf32r(v[x + 1]), tf32r(v[x + 2]), tf32r(v[x + 3]));
            }
#pragma unroll
            for (int cb = 0; cb < 2; ++cb) {                     // B = Khat^T Utilde
                const int c0 = 64 * half + 32 * cb;
                tmem_ld32(tmem + tlane + DK + c0, v);
#pragma unroll
                for (int x = 0; x < 32; x += 4)
                    *reinterpret_cast<float4*>(rec + REC_B + (((c0 + x) >> 2) * DK + i) * 16) =
                        make_float4(v[x], v[x + 1], v[x + 2], v[x + 3]);
            }
#pragma unroll
            for (int cb = 0; cb < 2; ++cb) {                     // Q' = Gamma.Q - P W -> rows 0..63 of [Q'; M]
                const int c0 = 64 * half + 32 * cb;
                tmem_ld32(tmem + tlane + 2 * DK + c0, v);
                if (lane < 16) {
#pragma unroll
                    for (int x = 0; x < 32; x += 4) {
                        const float4 gg = *reinterpret_cast<const float4*>(sm + OFF_G + g_off(r, c0 + x));
                        const uint2 qq = *reinterpret_cast<const uint2*>(sm + OFF_Q + kq_off(r, c0 + x));
                        const __nv_bfloat162* q2 = reinterpret_cast<const __nv_bfloat162*>(&qq);
                        *reinterpret_cast<float4*>(rec + REC_QM + op_off(r, c0 + x, DK)) =
                            make_float4(tf32r(ex2f(gg.x) * __low2float(q2[0]) - v[x]),
                                        tf32r(ex2f(gg.y) * __high2float(q2[0]) - v[x + 1]),
                                        tf32r(ex2f(gg.z) * __low2float(q2[1]) - v[x + 2]),
                                        tf32r(ex2f(gg.w) * __high2float(q2[1]) - v[x + 3]));
                    }
                }
            }
#pragma unroll
            for (int cb = 0; cb < 2; ++cb) {                     // P Utilde
                const int c0 = 64 * half + 32 * cb;
                tmem_ld32(tmem + tlane + 3 * DK + c0, v);
                if (lane < 16) {
#pragma unroll
                    for (int x = 0; x < 32; x += 4)
                        *reinterpret_cast<float4*>(rec + REC_O + (((c0 + x) >> 2) * C + r) * 16) =
                            make_float4(v[x], v[x + 1], v[x + 2], v[x + 3]);
                }
            }
            if (tid < DK) reinterpret_cast<float*>(rec + REC_G)[tid] = sgam[tid];
        }
    } while (false);

    tc_fence_before();
    __syncthreads();
    if (warp == 0) {
        tc_fence_after();
        asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem), "r"(512) : "memory");
    }
}

// ============================================================================================
// Phase 2: one CTA per (head, 32 value columns), chunks [c_begin, c_begin + n_chunks) in order.
// ============================================================================================
__global__ void __launch_bounds__(NT, 1)
    kda_prefill_chain_kernel(PrefillParams p, const unsigned char* records, int c_begin, int n_chunks,
                             const float* state_in) {
    extern __shared__ __align__(1024) unsigned char sm[];
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int quad = warp & 3, half = warp >> 2;
    constexpr int CPT = SNV / 2;                      // value columns per thread
    const int H = p.H;
    const int h = blockIdx.x / SLICES, slice = blockIdx.x % SLICES, j0 = slice * SNV;
    if (!valid_single_sequence(p)) {
        if (tid == 0) atomicOr(p.err, KDA_DEVERR_CU_SEQLENS);
        return;
    }
    if (saddr(sm) & 1023u) {
        if (tid == 0) atomicOr(p.err, KDA_DEVERR_TIMEOUT);
        return;
    }
    const int32_t T = p.total_tokens;
    __nv_bfloat16* go = static_cast<__nv_bfloat16*>(p.o);
    volatile int* s_abort = reinterpret_cast<volatile int*>(sm + C_OFF_MISC + 12);
    uint32_t* s_tmem = reinterpret_cast<uint32_t*>(sm + C_OFF_MISC + 8);
    const uint32_t mbar = saddr(sm + C_OFF_MISC);
    const uint32_t lbar0 = saddr(sm + C_OFF_MISC + 16), lbar1 = saddr(sm + C_OFF_MISC + 24);
    unsigned char* sop = sm + C_OFF_S;
    constexpr uint32_t TM_O = 0, TM_S = 32;           // [Q'; M_top] S and M S accumulators

    if (tid == 0) {
        asm volatile("mbarrier.init.shared::cta.b64 [%0], 1;" ::"r"(mbar) : "memory");
        asm volatile("mbarrier.init.shared::cta.b64 [%0], 1;" ::"r"(lbar0) : "memory");
        asm volatile("mbarrier.init.shared::cta.b64 [%0], 1;" ::"r"(lbar1) : "memory");
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
        *s_abort = 0;
    }
    if (warp == 0) {
        asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(saddr(s_tmem)), "r"(64)
                     : "memory");
        asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
    }
    const int srow = 32 * quad + lane;                // state row (key channel) of this thread
    const int jc = j0 + CPT * half;                   // first value column of this thread
    const int64_t state_off = (((int64_t)h) * DK + srow) * (int64_t)p.dv + jc;
    float S[CPT];
#pragma unroll
    for (int j = 0; j < CPT; j += 4) {
        const float4 v4 = state_in ? *reinterpret_cast<const float4*>(state_in + state_off + j)
                                   : make_float4(0.f, 0.f, 0.f, 0.f);
        S[j] = v4.x; S[j + 1] = v4.y; S[j + 2] = v4.z; S[j + 3] = v4.w;
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *s_tmem;
    const uint32_t tlane = (uint32_t)(quad * 32) << 16;
    uint32_t phase = 0, lph = 0;      // lph bit b: parity of buffer b's next load;  pend bit b: a load in flight
    uint32_t pend = 0;
    bool aborted = false;

    auto issue = [&](int ci) {                        // bulk-load [Q'; M] of chunk ci into buffer ci & 1
        if (tid == 32) {
            const int b = ci & 1;
            const unsigned char* rec = records + (size_t)(ci * H + h) * REC_BYTES;
            const uint32_t lb = b ? lbar1 : lbar0;
            mbar_expect_tx(lb, QM_BYTES);
            bulk_g2s(saddr(sm + b * QM_BYTES), rec + REC_QM, QM_BYTES, lb);
        }
        pend |= 1u << (ci & 1);
    };
    auto write_state_operand = [&]() {                // S^T as a TF32 operand: row = value column, K = srow
#pragma unroll
        for (int j = 0; j < CPT; ++j)
            *reinterpret_cast<float*>(sop + sw128_off(CPT * half + j, srow, SNV)) = tf32r(S[j]);
    };
    write_state_operand();
    if (n_chunks > 0) issue(0);
    if (n_chunks > 1) issue(1);
    fence_async_smem();
    __syncthreads();

    for (int ci = 0; ci < n_chunks && !aborted; ++ci) {
        const int b = ci & 1;
        const uint32_t abuf = saddr(sm + b * QM_BYTES);
        const unsigned char* rec = records + (size_t)(ci * H + h) * REC_BYTES;
        const int32_t t0 = (c_begin + ci) * C;
        const int L = min(C, T - t0);
        if (!mbar_wait(b ? lbar1 : lbar0, (lph >> b) & 1u)) {
            atomicOr(p.err, KDA_DEVERR_TIMEOUT);
            *s_abort = 1;
        }
        lph ^= 1u << b;
        pend &= ~(1u << b);
        __syncthreads();
        if (*s_abort) { aborted = true; break; }

        // [Q'; M_top] S and M S: 2 x 16 TF32 steps, one commit
        if (warp == 0) {
            if (elect_one()) {
                tc_fence_after();
                constexpr uint32_t id = idesc_tf32(128, SNV);
                const uint64_t a_o = op_desc(abuf, DK), a_s = op_desc(abuf + C * DK * 4, DK);
                const uint32_t sb = saddr(sop);
#pragma unroll
                for (int ks = 0; ks < DK / 8; ++ks) {
                    const uint64_t bd = desc_sw128(sb + (ks >> 2) * (SNV * 128) + (ks & 3) * 32);
                    umma_tf32_1(tmem + TM_O, a_o + (uint64_t)(ks * 16), bd, id, ks > 0 ? 1u : 0u);
                    umma_tf32_1(tmem + TM_S, a_s + (uint64_t)(ks * 16), bd, id, ks > 0 ? 1u : 0u);
                }
                umma_commit(mbar);
            }
            __syncwarp();
        }
        // the chunk's B, P Utilde and Gamma_C, loaded while the products run
        float4 bq[CPT / 4], oq[CPT / 4];
#pragma unroll
        for (int m = 0; m < CPT / 4; ++m)
            bq[m] = __ldg(reinterpret_cast<const float4*>(rec + REC_B + (((jc + 4 * m) >> 2) * DK + srow) * 16));
        if (quad < 2) {
#pragma unroll
            for (int m = 0; m < CPT / 4; ++m)
                oq[m] = __ldg(reinterpret_cast<const float4*>(rec + REC_O + (((jc + 4 * m) >> 2) * C + srow) * 16));
        }
        const float gamC = __ldg(reinterpret_cast<const float*>(rec + REC_G) + srow);
        if (!mbar_wait(mbar, phase)) {
            atomicOr(p.err, KDA_DEVERR_TIMEOUT);
            *s_abort = 1;
        }
        phase ^= 1u;
        __syncthreads();
        if (*s_abort) { aborted = true; break; }
        tc_fence_after();
        {
            float d[CPT];
            tmem_ld16(tmem + tlane + TM_S + CPT * half, d);
#pragma unroll
            for (int m = 0; m < CPT / 4; ++m) {
                S[4 * m + 0] = fmaf(gamC, S[4 * m + 0], bq[m].x - d[4 * m + 0]);
                S[4 * m + 1] = fmaf(gamC, S[4 * m + 1], bq[m].y - d[4 * m + 1]);
                S[4 * m + 2] = fmaf(gamC, S[4 * m + 2], bq[m].z - d[4 * m + 2]);
                S[4 * m + 3] = fmaf(gamC, S[4 * m + 3], bq[m].w - d[4 * m + 3]);
            }
            write_state_operand();
            if (quad < 2) {                           // output rows 0..63 live in lanes 0..63
                tmem_ld16(tmem + tlane + TM_O + CPT * half, d);
                if (srow < L) {
                    __nv_bfloat16* dst = go + ((int64_t)(t0 + srow) * H + h) * p.dv + jc;
#pragma unroll
                    for (int x = 0; x < CPT; x += 8) {
                        const float4 o0 = oq[x / 4], o1 = oq[x / 4 + 1];
                        *reinterpret_cast<uint4*>(dst + x) =
                            make_uint4(pack_bf16x2(p.scale * (d[x] + o0.x), p.scale * (d[x + 1] + o0.y)),
                                       pack_bf16x2(p.scale * (d[x + 2] + o0.z), p.scale * (d[x + 3] + o0.w)),
                                       pack_bf16x2(p.scale * (d[x + 4] + o1.x), p.scale * (d[x + 5] + o1.y)),
                                       pack_bf16x2(p.scale * (d[x + 6] + o1.z), p.scale * (d[x + 7] + o1.w)));
                    }
                }
            }
        }
        fence_async_smem();
        tc_fence_before();
        __syncthreads();
        if (ci + 2 < n_chunks) issue(ci + 2);          // this buffer is free again
    }

    if (!aborted) {
#pragma unroll
        for (int j = 0; j < CPT; j += 4)
            *reinterpret_cast<float4*>(p.state_out + state_off + j) = make_float4(S[j], S[j + 1], S[j + 2], S[j + 3]);
    }
    if (pend & 1u) mbar_wait(lbar0, lph & 1u);         // bounded: never leave copies in flight
    if (pend & 2u) mbar_wait(lbar1, (lph >> 1) & 1u);
    tc_fence_before();
    __syncthreads();
    if (warp == 0) {
        tc_fence_after();
        asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem), "r"(64) : "memory");
    }
}

int64_t window_chunks(int32_t H) {
    const int64_t w = (int64_t)(kWindowBudget / ((size_t)H * REC_BYTES));
    return w < 1 ? 1 : w;
}

}  // namespace

bool prefill_2p_supported(int32_t num_seqs, int64_t total_tokens, int32_t H, int32_t d_k, int32_t d_v,
                          kda_dtype dt) {
    return num_seqs == 1 && total_tokens > 0 && dt == KDA_DTYPE_BF16 && d_k == DK && d_v == DK && H > 0;
}

size_t prefill_2p_min_workspace(int32_t H) { return (size_t)H * REC_BYTES; }

size_t prefill_2p_workspace(int64_t total_tokens, int32_t H) {
    const int64_t chunks = (total_tokens + C - 1) / C;
    const int64_t w = chunks < window_chunks(H) ? chunks : window_chunks(H);
    return (size_t)w * H * REC_BYTES;
}

cudaError_t launch_prefill_2p(const PrefillParams& p, void* workspace, size_t workspace_bytes, cudaStream_t s) {
    auto enc = tensor_map_encoder();
    if (!enc) return cudaErrorNotSupported;
    PrepMaps maps;
    std::memset(&maps, 0, sizeof maps);
    const int T = p.total_tokens;
    if (!encode_rows(enc, &maps.k, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, p.k, 2, DK, p.H, T, 64, CU_TENSOR_MAP_SWIZZLE_128B) ||
        !encode_rows(enc, &maps.q, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, p.q, 2, DK, p.H, T, 64, CU_TENSOR_MAP_SWIZZLE_128B) ||
        !encode_rows(enc, &maps.a, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, p.alpha, 4, DK, p.H, T, 32,
                     CU_TENSOR_MAP_SWIZZLE_128B) ||
        !encode_rows(enc, &maps.v, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, p.v, 2, p.dv, p.H, T, DK, CU_TENSOR_MAP_SWIZZLE_NONE))
        return cudaErrorInvalidValue;
    cudaError_t e = cudaFuncSetAttribute(kda_prefill_prep_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, P_SMEM);
    if (e != cudaSuccess) return e;
    e = cudaFuncSetAttribute(kda_prefill_chain_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, C_SMEM);
    if (e != cudaSuccess) return e;
    unsigned char* rec = static_cast<unsigned char*>(workspace);
    const int64_t chunks = (T + C - 1) / C;
    int64_t wmax = (int64_t)(workspace_bytes / prefill_2p_min_workspace(p.H));   // records the workspace holds
    if (wmax > window_chunks(p.H)) wmax = window_chunks(p.H);
    if (wmax < 1) return cudaErrorInvalidValue;
    for (int64_t c0 = 0; c0 < chunks; c0 += wmax) {
        const int64_t n = chunks - c0 < wmax ? chunks - c0 : wmax;
        kda_prefill_prep_kernel<<<(unsigned)(n * p.H), NT, P_SMEM, s>>>(p, maps, rec, (int)c0);
        if ((e = cudaGetLastError()) != cudaSuccess) return e;
        kda_prefill_chain_kernel<<<(unsigned)(p.H * SLICES), NT, C_SMEM, s>>>(p, rec, (int)c0, (int)n,
                                                                               c0 == 0 ? p.state_in : p.state_out);
        if ((e = cudaGetLastError()) != cudaSuccess) return e;
    }
    return cudaSuccess;
}

}  // namespace kda
