// Backward pass 3 at d = 128 in matrix form: one unit per (sequence, chunk, head), every gradient of the
// chunk from a fixed sequence of products, with no per-token state.
//
// "Kimi K3, explained" (section "Training in chunks") writes a chunk of L tokens as products of small
// matrices once its start state S_0 is known: with g_r the running sum of ln alpha over the chunk,
// Gamma = exp(g), E_rsi = exp(g_ri - g_si) (s <= r),
//
//   Bt_rs = sum_i k_ri k_si E_rsi (s < r),  P_rs = sum_i q_ri k_si E_rsi (s <= r),  T = (I + Diag(beta) Bt)^-1
//   W = T Diag(beta) (Gamma . K),  U = T Diag(beta) V - W S_0,  Khat = (Gamma_L / Gamma) . K
//   O = (Gamma . Q) S_0 + P U,  S_1 = Diag(Gamma_L) S_0 + Khat^T U.
//
// Reverse mode through those products, given dO = scale * grad_o and the gradient dS_1 of the end state
// (pass 2), is again a sequence of products:
//
//   dU = P^T dO + Khat dS_1,  dP = (dO U^T) on s <= r,  dQs = dO S_0^T,  dKhat = U dS_1^T,  dW = -dU S_0^T
//   dT = dW (beta . Gamma . K)^T + dU (beta . V)^T,  dA = -(T^T dT T^T) on s < r,  dBt = Diag(beta) dA
//   dq = sum_s dP_rs k_s E_rs + Gamma . dQs,  dv = beta . (T^T dU)
//   dk = sum_r dP_rs q_r E_rs + sum_s dBt_rs k_s E_rs + sum_r dBt_rs k_r E_rs + beta Gamma . (T^T dW)
//        + (Gamma_L / Gamma) . dKhat
//   dbeta_r = sum_s dA_rs Bt_rs + sum_i (Gamma k)_ri (T^T dW)_ri + sum_i v_ri (T^T dU)_ri
//   dg = q . (first dq term) - k . (first dk term) + k . (second) - k . (third) + q Gamma . dQs
//        + beta Gamma k . (T^T dW) - k (Gamma_L / Gamma) . dKhat,
//        and on the chunk's last row also sum_s (dKhat . Khat)_s + Gamma_L . rowsum(dS_1 . S_0)
//   d ln alpha_s = sum_{r >= s} dg_r,  dalpha = d ln alpha / alpha.
//
// The decayed sums over E are taken per block of 16 rows with a reference row inside the block (the
// forward's own device): E_rsi = 2^(G_ri - G_ref) 2^(G_ref - G_si) with G = running sum of log2 alpha
// (clamped at -15 per token, as in the forward), so that no factor exceeds 2^120 and every product is a
// plain dot product of scaled operands.  For bf16 inputs the products run on mma.sync m16n8k8 TF32 (fp32
// accumulate): the plain ones and Bt, P with single TF32 operands, the decayed sums that feed the decay
// gradient with split (hi + lo) TF32; for fp32 inputs every product is fp32 FFMA.  The chunk's 64 x 128
// matrices live in a per-CTA scratch (L2), its 64 x 64 matrices, k and G in shared memory.  Rows past
// the end of a partial chunk read as zero with beta = 0 and alpha = 1, which leaves the valid rows'
// results unchanged.

#include <type_traits>

#include "kda_internal.cuh"

namespace kda {
namespace {

constexpr int MC = 64;                 // chunk rows
constexpr int MD = 128;                // head dimension (key = value)
constexpr int MNT = 256;
constexpr int LD64 = 68;               // floats per row of a shared 64 x 64 matrix
constexpr int LDY = 132;               // floats per row of a shared scaled operand (float4 reads, no conflicts)
constexpr int MAT = MC * MD;           // floats per scratch matrix

// shared memory (floats)
constexpr int F_P = 0;                             // P
constexpr int F_T = F_P + MC * LD64;               // T
constexpr int F_BT = F_T + MC * LD64;              // Bt
constexpr int F_DP = F_BT + MC * LD64;             // dP  } dP, dA, Y and the staging area are contiguous: the
constexpr int F_DA = F_DP + MC * LD64;             // dA  } products before dP (or dA) is written run their
constexpr int F_Y = F_DA + MC * LD64;              //     } cp.async ring over them, with more stages in flight
                                                   // scaled operands [64][LDY]; dT and X [64][LD64] each
constexpr int F_STG = F_Y + 2 * MC * LD64;         // product staging: A [16][LD64], B [16][LDY]; also 2 x [16][LDY]
constexpr int F_VEC = F_STG + 2 * 16 * LDY;        // beta [64], G_C [128], row sums [128], column sums [2][128], [64]
constexpr int F_K = F_VEC + 64 + 128 + 128 + 256 + 64;        // k [64][128]
constexpr int F_G = F_K + MC * MD;                 // G [64][128]
constexpr int MAT_SMEM_FLOATS = F_G + MC * MD;
static_assert(2 * MC * LD64 >= MC * LDY, "scaled operand area");

// scratch matrices (each [64][128] fp32, row-major) per CTA; a later matrix takes the slot of one whose
// last reader has run (dO -> T^T dW, beta Gamma K -> dq_p, beta V -> dk_r, W -> dQs, U -> dk_p,
// Khat -> dKhat, dU -> dk_s, dW -> T^T dU), so that the scratch of all CTAs stays within L2
enum : int { XQ = 0, XV, XDO, XKTB, XVB, XW, XU, XKH, XDU, XDW, X_COUNT,
             XTDW = XDO, XRQ = XKTB, XRK = XVB, XDQS = XW, XCP = XU, XDKH = XKH, XCK = XDU, XTDU = XDW };
static_assert((size_t)X_COUNT * MAT * 4 <= kBwdMatScratchBytes, "per-CTA scratch");

// 2^x by the hardware approximation (ex2.approx.ftz: relative error about 2^-22, results below 2^-126
// flushed to zero, which only drops decay factors far below every other term)
__device__ __forceinline__ float ex2a(float x) {
    float y;
    asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}
__device__ __forceinline__ float ldf(const float* p) { return *p; }
// 16 bytes of a token row as floats
__device__ __forceinline__ void ld16f(const float* p, float* o) {
    const float4 v = __ldg(reinterpret_cast<const float4*>(p));
    o[0] = v.x; o[1] = v.y; o[2] = v.z; o[3] = v.w;
}
__device__ __forceinline__ void ld16f(const __nv_bfloat16* p, float* o) {
    const uint4 v = __ldg(reinterpret_cast<const uint4*>(p));
    const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
    for (int c = 0; c < 4; ++c) {
        o[2 * c] = __uint_as_float(w[c] << 16);
        o[2 * c + 1] = __uint_as_float(w[c] & 0xFFFF0000u);
    }
}
__device__ __forceinline__ void st4(float* p, const float* v, float s = 1.f) {
    *reinterpret_cast<float4*>(p) = make_float4(s * v[0], s * v[1], s * v[2], s * v[3]);
}

__device__ __forceinline__ uint32_t tf32_bits(float x) {
    uint32_t r;
    asm("cvt.rna.tf32.f32 %0, %1;" : "=r"(r) : "f"(x));
    return r;
}
__device__ __forceinline__ void mma_tf32(float* d, const uint32_t* a, uint32_t b0, uint32_t b1) {
    asm volatile("mma.sync.aligned.m16n8k8.row.col.f32.tf32.tf32.f32 {%0, %1, %2, %3}, {%4, %5, %6, %7}, {%8, %9}, "
                 "{%0, %1, %2, %3};\n"
                 : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
                 : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}

// One m16n8 tile over `ksteps` steps of k = 8: d += A B with A(m, k) = fa(m, k), B(k, n) = fb(k, n) given as
// TF32 bits (m < 16, n < 8 relative to the tile).
template <class FA, class FB>
__device__ __forceinline__ void tile_mma(float (&d)[4], int ksteps, FA fa, FB fb) {
    const int lane = threadIdx.x & 31, g = lane >> 2, t = lane & 3;
#pragma unroll 2
    for (int ks = 0; ks < ksteps; ++ks) {
        const int k0 = 8 * ks;
        const uint32_t a[4] = {fa(g, k0 + t), fa(g + 8, k0 + t), fa(g, k0 + t + 4), fa(g + 8, k0 + t + 4)};
        mma_tf32(d, a, fb(k0 + t, g), fb(k0 + t + 4, g));
    }
}
__device__ __forceinline__ float tf32r(float x) { return __uint_as_float(tf32_bits(x)); }
// MA x NB m16n8 tiles (A fragments shared along a row of tiles, B along a column) with fp32 operands
// split as x = hi + lo (both TF32) and d += A_hi B_hi + A_hi B_lo + A_lo B_hi: about fp32 accuracy.
// The decayed sums that feed the decay gradient need it: its terms cancel, and
// single TF32 operands there leave a relative error of about 3e-2 in dalpha (a float64 emulation of
// this arithmetic on the prefill workload), against 3e-4 split.
// The tiles' MMAs interleave, so that no warp waits on one accumulator's chain.
template <int MA, int NB, class FA, class FB>
__device__ __forceinline__ void tiles_mma3(float (&d)[MA][NB][4], int ksteps, FA fa, FB fb) {
    const int lane = threadIdx.x & 31, g = lane >> 2, t = lane & 3;
    auto split = [](float x, uint32_t& hi, uint32_t& lo) {
        hi = tf32_bits(x);
        lo = tf32_bits(x - __uint_as_float(hi));
    };
#pragma unroll 1
    for (int ks = 0; ks < ksteps; ++ks) {
        const int k0 = 8 * ks;
        uint32_t ah[MA][4], al[MA][4], bh[NB][2], bl[NB][2];
#pragma unroll
        for (int ma = 0; ma < MA; ++ma) {
            split(fa(ma, g, k0 + t), ah[ma][0], al[ma][0]);
            split(fa(ma, g + 8, k0 + t), ah[ma][1], al[ma][1]);
            split(fa(ma, g, k0 + t + 4), ah[ma][2], al[ma][2]);
            split(fa(ma, g + 8, k0 + t + 4), ah[ma][3], al[ma][3]);
        }
#pragma unroll
        for (int nb = 0; nb < NB; ++nb) {
            split(fb(nb, k0 + t, g), bh[nb][0], bl[nb][0]);
            split(fb(nb, k0 + t + 4, g), bh[nb][1], bl[nb][1]);
        }
#pragma unroll
        for (int ma = 0; ma < MA; ++ma)
#pragma unroll
            for (int nb = 0; nb < NB; ++nb) mma_tf32(d[ma][nb], al[ma], bh[nb][0], bh[nb][1]);
#pragma unroll
        for (int ma = 0; ma < MA; ++ma)
#pragma unroll
            for (int nb = 0; nb < NB; ++nb) mma_tf32(d[ma][nb], ah[ma], bl[nb][0], bl[nb][1]);
#pragma unroll
        for (int ma = 0; ma < MA; ++ma)
#pragma unroll
            for (int nb = 0; nb < NB; ++nb) mma_tf32(d[ma][nb], ah[ma], bh[nb][0], bh[nb][1]);
    }
}
// The same for MA products that share no operand, d[ma] += A_ma B_ma (B fragments per ma), in one k-loop so
// that their MMA chains interleave.
template <int MA, int NB, class FA, class FB>
__device__ __forceinline__ void tiles_mma3_sep(float (&d)[MA][NB][4], int ksteps, FA fa, FB fb) {
    const int lane = threadIdx.x & 31, g = lane >> 2, t = lane & 3;
    auto split = [](float x, uint32_t& hi, uint32_t& lo) {
        hi = tf32_bits(x);
        lo = tf32_bits(x - __uint_as_float(hi));
    };
#pragma unroll 1
    for (int ks = 0; ks < ksteps; ++ks) {
        const int k0 = 8 * ks;
        uint32_t ah[MA][4], al[MA][4], bh[MA][NB][2], bl[MA][NB][2];
#pragma unroll
        for (int ma = 0; ma < MA; ++ma) {
            split(fa(ma, g, k0 + t), ah[ma][0], al[ma][0]);
            split(fa(ma, g + 8, k0 + t), ah[ma][1], al[ma][1]);
            split(fa(ma, g, k0 + t + 4), ah[ma][2], al[ma][2]);
            split(fa(ma, g + 8, k0 + t + 4), ah[ma][3], al[ma][3]);
#pragma unroll
            for (int nb = 0; nb < NB; ++nb) {
                split(fb(ma, nb, k0 + t, g), bh[ma][nb][0], bl[ma][nb][0]);
                split(fb(ma, nb, k0 + t + 4, g), bh[ma][nb][1], bl[ma][nb][1]);
            }
        }
#pragma unroll
        for (int ma = 0; ma < MA; ++ma)
#pragma unroll
            for (int nb = 0; nb < NB; ++nb) mma_tf32(d[ma][nb], al[ma], bh[ma][nb][0], bh[ma][nb][1]);
#pragma unroll
        for (int ma = 0; ma < MA; ++ma)
#pragma unroll
            for (int nb = 0; nb < NB; ++nb) mma_tf32(d[ma][nb], ah[ma], bl[ma][nb][0], bl[ma][nb][1]);
#pragma unroll
        for (int ma = 0; ma < MA; ++ma)
#pragma unroll
            for (int nb = 0; nb < NB; ++nb) mma_tf32(d[ma][nb], ah[ma], bh[ma][nb][0], bh[ma][nb][1]);
    }
}
// outputs written once: streaming stores, so that they do not push the scratch out of L2
__device__ __forceinline__ void st_out(float* p, int64_t i, float x) { __stcs(p + i, x); }
__device__ __forceinline__ void st_out(__nv_bfloat16* p, int64_t i, float x) { __stcs(p + i, __float2bfloat16_rn(x)); }

// Output element acc[i][j] of a 64 x NN product sits at (mrow(i), mcol(j)).  CUDA-core path (TC false):
// thread (tr, tc) = (tid / 16, tid % 16) owns rows 4 tr + i and columns 4 tc + (j & 3) + 64 (j >> 2) (NN =
// 128) or 4 tc + j (NN = 64).  Tensor-core path: warp w owns rows 32 (w & 1) .. + 31 and columns NN/4 (w >> 1)
// .. + NN/4 - 1 as 2 x (NN / 32) m16n8 tiles; lane (g, t) = (lane / 4, lane % 4) holds rows g, g + 8 and
// columns 2 t, 2 t + 1 of each tile (i = 2 m-tile + row half, j = 2 n-tile + column).
template <bool TC>
__device__ __forceinline__ int mrow(int i) {
    const int tid = threadIdx.x;
    if constexpr (TC) return 32 * ((tid >> 5) & 1) + 16 * (i >> 1) + ((tid & 31) >> 2) + 8 * (i & 1);
    else return 4 * (tid >> 4) + i;
}
template <int NN, bool TC>
__device__ __forceinline__ int mcol(int j) {
    const int tid = threadIdx.x;
    if constexpr (TC) return (NN / 4) * (tid >> 6) + 8 * (j >> 1) + 2 * (tid & 3) + (j & 1);
    else return NN == 128 ? 4 * (tid & 15) + (j & 3) + 64 * (j >> 2) : 4 * (tid & 15) + j;
}

// The CUDA-core product (fp32 inputs): acc[i][j] += sum_{k < KK} A(mrow(i), k) B(k, mcol(j)) for this
// thread's part of a 64 x NN product in fp32 FFMA, with A(m, k) = A[m am + k ak] and B(k, n) = B[k bk +
// n bn] (global or shared).  16 k at a time are staged through shared memory, the next 16 fetched into
// registers while the current ones are used.
constexpr int LDA = 72;                               // staged A row (k-major): conflict-free fragment loads
static_assert(16 * LDA + 16 * (128 + 8) <= 2 * 16 * LDY, "staging area");
static_assert(3 * (64 * 20 + 128 * 20) <= 2 * MC * LD64 + 2 * 16 * LDY, "product ring (scaled-operand and staging areas)");
static_assert(5 * (64 * 20 + 128 * 20) <= 4 * MC * LD64 + 2 * 16 * LDY, "five-stage ring from dP on");
static_assert(4 * (64 * 20 + 128 * 20) <= 3 * MC * LD64 + 2 * 16 * LDY, "four-stage ring from dA on");
template <int NN, int KK>
__device__ __forceinline__ void mm(const float* A, int am, int ak, const float* B, int bk, int bn, float* stage,
                                   float (&acc)[4][NN / 16]) {
    constexpr int NJ = NN / 16;
    constexpr int LB = NN + 8;
    float* sa = stage;                                 // [16][LDA]: sa[k][m]
    float* sb = stage + 16 * LDA;                      // [16][LB]:  sb[k][n]
    const int tid = threadIdx.x, tr = tid >> 4, tc = tid & 15;
    float ra[4], rb[NJ];
    auto fetch = [&](int k0) {
#pragma unroll
        for (int e = 0; e < 4; ++e) {
            const int idx = tid + MNT * e;
            const int m = ak == 1 ? idx >> 4 : idx & 63, k = ak == 1 ? idx & 15 : idx >> 6;
            ra[e] = ldf(A + m * am + (k0 + k) * ak);
        }
#pragma unroll
        for (int e = 0; e < NJ; ++e) {
            const int idx = tid + MNT * e;
            const int n = bn == 1 ? idx % NN : idx >> 4, k = bn == 1 ? idx / NN : idx & 15;
            rb[e] = ldf(B + (k0 + k) * bk + n * bn);
        }
    };
    auto put = [&]() {
#pragma unroll
        for (int e = 0; e < 4; ++e) {
            const int idx = tid + MNT * e;
            const int m = ak == 1 ? idx >> 4 : idx & 63, k = ak == 1 ? idx & 15 : idx >> 6;
            sa[k * LDA + m] = ra[e];
        }
#pragma unroll
        for (int e = 0; e < NJ; ++e) {
            const int idx = tid + MNT * e;
            const int n = bn == 1 ? idx % NN : idx >> 4, k = bn == 1 ? idx / NN : idx & 15;
            sb[k * LB + n] = rb[e];
        }
    };
    fetch(0);
#pragma unroll 1
    for (int k0 = 0; k0 < KK; k0 += 16) {
        __syncthreads();                               // the previous chunk's readers are done
        put();
        __syncthreads();
        if (k0 + 16 < KK) fetch(k0 + 16);
        {
#pragma unroll 4
            for (int k = 0; k < 16; ++k) {
                const float4 a = *reinterpret_cast<const float4*>(sa + k * LDA + 4 * tr);
                float b[NJ];
                const float4 b0 = *reinterpret_cast<const float4*>(sb + k * LB + 4 * tc);
                b[0] = b0.x; b[1] = b0.y; b[2] = b0.z; b[3] = b0.w;
                if constexpr (NJ == 8) {
                    const float4 b1 = *reinterpret_cast<const float4*>(sb + k * LB + 64 + 4 * tc);
                    b[4] = b1.x; b[5] = b1.y; b[6] = b1.z; b[7] = b1.w;
                }
                const float av[4] = {a.x, a.y, a.z, a.w};
#pragma unroll
                for (int i = 0; i < 4; ++i)
#pragma unroll
                    for (int j = 0; j < NJ; ++j) acc[i][j] = fmaf(av[i], b[j], acc[i][j]);
            }
        }
    }
    __syncthreads();                                   // the staging area is free again
}

__device__ __forceinline__ void cp_async16(float* dst, const float* src) {
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16;\n" ::"r"((uint32_t)__cvta_generic_to_shared(dst)), "l"(src)
                 : "memory");
}
__device__ __forceinline__ void cp_async_commit_group() { asm volatile("cp.async.commit_group;\n" ::: "memory"); }
template <int N>
__device__ __forceinline__ void cp_async_wait_group() { asm volatile("cp.async.wait_group %0;\n" ::"n"(N) : "memory"); }

// The tensor-core product: acc[i][j] += sum_{k < KK} A(mrow(i), k) B(k, mcol(j)) on mma.sync m16n8k8 TF32
// (fp32 accumulate), with A(m, k) = AT ? A[k lda + m] : A[m lda + k] and B(k, n) = BT ? B[n ldb + k] :
// B[k ldb + n].  An operand in shared memory (AS, BS) is read in place; one in global memory streams
// through a ring of three 16-k stages by 16-byte cp.async, two stages ahead of the one in use, each
// stored so that the fragment loads are free of bank conflicts (k-contiguous rows of 20 floats, or
// k-major rows of 72 / NN + 8).  Operands are rounded to TF32 (nearest) as their fragments are loaded.
constexpr int RING_STAGE = 64 * 20 + 128 * 20;     // floats per stage: A 64 x 20, B up to 128 x 20
template <int NN, int KK, bool AS, bool AT, bool BS, bool BT, int NRS>
__device__ __forceinline__ void mm_tc(const float* A, int lda, const float* B, int ldb, float* ring,
                                      float (&acc)[4][NN / 16]) {
    constexpr int NST = KK / 16;
    static_assert(NRS >= 3 && NRS <= 5, "ring stages");
    constexpr int LAR = 20, LAT = 72, LBR = NN + 8, LBT = 20;
    const int tid = threadIdx.x, lane = tid & 31, w = tid >> 5, g = lane >> 2, t = lane & 3;
    const int m0 = 32 * (w & 1), n0 = (NN / 4) * (w >> 1);
    auto issue = [&](int st) {
        float* sa = ring + (st % NRS) * RING_STAGE;
        float* sb = sa + 64 * 20;
        const int k0 = 16 * st;
        if constexpr (!AS) {
            if constexpr (!AT) {
                const int m = tid >> 2, kq = (tid & 3) * 4;
                cp_async16(sa + m * LAR + kq, A + m * lda + k0 + kq);
            } else {
                const int k = tid >> 4, mq = (tid & 15) * 4;
                cp_async16(sa + k * LAT + mq, A + (k0 + k) * lda + mq);
            }
        }
        if constexpr (!BS) {
#pragma unroll
            for (int e = 0; e < NN / 64; ++e) {
                const int idx = tid + MNT * e;
                if constexpr (!BT) {
                    const int k = idx / (NN / 4), nq = (idx % (NN / 4)) * 4;
                    cp_async16(sb + k * LBR + nq, B + (k0 + k) * ldb + nq);
                } else {
                    const int n = idx >> 2, kq = (idx & 3) * 4;
                    cp_async16(sb + n * LBT + kq, B + n * ldb + k0 + kq);
                }
            }
        }
        cp_async_commit_group();
    };
#pragma unroll
    for (int j = 0; j < NRS - 1; ++j)
        if (j < NST) issue(j);
#pragma unroll 1
    for (int st = 0; st < NST; ++st) {
        const int ahead = min(NST - 1 - st, NRS - 2);  // stages committed after st
        if (ahead >= 3) cp_async_wait_group<3>();
        else if (ahead == 2) cp_async_wait_group<2>();
        else if (ahead == 1) cp_async_wait_group<1>();
        else cp_async_wait_group<0>();
        __syncthreads();                               // stage st landed for every thread; stage st - 1 is read
        if (st + NRS - 1 < NST) issue(st + NRS - 1);   // into the slot of stage st - 1
        const float* sa = ring + (st % NRS) * RING_STAGE;
        const float* sb = sa + 64 * 20;
        const int k0 = 16 * st;
        auto fa = [&](int m, int kl) -> float {        // kl: k within the stage
            if constexpr (AS) return AT ? A[(k0 + kl) * lda + m] : A[m * lda + k0 + kl];
            else return AT ? sa[kl * LAT + m] : sa[m * LAR + kl];
        };
        auto fb = [&](int kl, int n) -> float {
            if constexpr (BS) return BT ? B[n * ldb + k0 + kl] : B[(k0 + kl) * ldb + n];
            else return BT ? sb[n * LBT + kl] : sb[kl * LBR + n];
        };
#pragma unroll
        for (int kk = 0; kk < 16; kk += 8) {
            uint32_t a[2][4];
#pragma unroll
            for (int mt = 0; mt < 2; ++mt) {
                const int m = m0 + 16 * mt + g;
                a[mt][0] = tf32_bits(fa(m, kk + t));
                a[mt][1] = tf32_bits(fa(m + 8, kk + t));
                a[mt][2] = tf32_bits(fa(m, kk + t + 4));
                a[mt][3] = tf32_bits(fa(m + 8, kk + t + 4));
            }
#pragma unroll
            for (int nt = 0; nt < NN / 32; ++nt) {
                const int n = n0 + 8 * nt + g;
                const uint32_t b0 = tf32_bits(fb(kk + t, n)), b1 = tf32_bits(fb(kk + t + 4, n));
#pragma unroll
                for (int mt = 0; mt < 2; ++mt) {
                    float d[4] = {acc[2 * mt][2 * nt], acc[2 * mt][2 * nt + 1], acc[2 * mt + 1][2 * nt],
                                  acc[2 * mt + 1][2 * nt + 1]};
                    mma_tf32(d, a[mt], b0, b1);
                    acc[2 * mt][2 * nt] = d[0];
                    acc[2 * mt][2 * nt + 1] = d[1];
                    acc[2 * mt + 1][2 * nt] = d[2];
                    acc[2 * mt + 1][2 * nt + 1] = d[3];
                }
            }
        }
    }
    __syncthreads();                                   // the ring is free again
}

// One product of the chunk: on the tensor cores (TC) or in fp32 on the CUDA cores.
template <bool TC, int NN, int KK, bool AS, bool AT, bool BS, bool BT, int NRS = 3>
__device__ __forceinline__ void prod(const float* A, int lda, const float* B, int ldb, float* ring, float* stage,
                                     float (&acc)[4][NN / 16]) {
    if constexpr (TC) mm_tc<NN, KK, AS, AT, BS, BT, NRS>(A, lda, B, ldb, ring, acc);
    else mm<NN, KK>(A, AT ? 1 : lda, AT ? lda : 1, B, BT ? 1 : ldb, BT ? ldb : 1, stage, acc);
}

// the 128-column layout of the elementwise and decayed passes: thread tid % 16 owns columns
// 4 (tid % 16) + (j & 3) + 64 (j >> 2)
__device__ __forceinline__ int col8(int j) {
    const int tc = threadIdx.x & 15;
    return 4 * tc + (j & 3) + 64 * (j >> 2);
}
template <int NN>
__device__ __forceinline__ void zero(float (&acc)[4][NN / 16]) {
#pragma unroll
    for (int i = 0; i < 4; ++i)
#pragma unroll
        for (int j = 0; j < NN / 16; ++j) acc[i][j] = 0.f;
}
// store a 64 x 128 product (times s) into a scratch matrix
template <bool TC>
__device__ __forceinline__ void put128(float* X, const float (&acc)[4][8], float s = 1.f) {
#pragma unroll
    for (int i = 0; i < 4; ++i)
#pragma unroll
        for (int j = 0; j < 8; ++j) X[mrow<TC>(i) * MD + mcol<128, TC>(j)] = s * acc[i][j];
}

template <typename TIn>
__global__ void __launch_bounds__(MNT, 1) kda_bwd_chunk_mat_kernel(BwdParams p) {
    extern __shared__ __align__(16) float fsm[];
    float* sP = fsm + F_P;
    float* sT = fsm + F_T;
    float* sDP = fsm + F_DP;
    float* sDA = fsm + F_DA;
    float* sBT = fsm + F_BT;
    float* sY = fsm + F_Y;
    float* stg = fsm + F_STG;
    float* ring5 = fsm + F_DP;                         // product rings while dP (ring5) or dA (ring4) is free
    float* ring4 = fsm + F_DA;
    float* sbeta = fsm + F_VEC;
    float* sgc = sbeta + 64;                           // G of the chunk's last row, per key channel
    float* srow = sgc + 128;                           // sum_j dS_1[i][j] S_0[i][j], per key channel i
    float* scol = srow + 128;                          // [2][128] column partial sums
    float* sdb = scol + 256;                           // [64] sum_s dA_rs Bt_rs
    float* sK = fsm + F_K;
    float* sG = fsm + F_G;
    const float* G = sG;

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31, tr = tid >> 4, tc = tid & 15;
    // bf16 inputs: the plain products on TF32 tensor cores; fp32 inputs: on the CUDA cores in fp32
    constexpr bool TC = std::is_same<TIn, __nv_bfloat16>::value;
    auto cv = [](float x) { return TC ? tf32r(x) : x; };      // operands of the tensor-core products
    const int H = p.H;
    const TIn* gq = static_cast<const TIn*>(p.q);
    const TIn* gk = static_cast<const TIn*>(p.k);
    const TIn* gv = static_cast<const TIn*>(p.v);
    const TIn* gdo = static_cast<const TIn*>(p.d_o);
    TIn* gdq = static_cast<TIn*>(p.d_q);
    TIn* gdk = static_cast<TIn*>(p.d_k);
    TIn* gdv = static_cast<TIn*>(p.d_v);
    float* X = p.scratch + (int64_t)blockIdx.x * (int64_t)(kBwdMatScratchBytes / 4);
    auto M = [&](int x) { return X + x * MAT; };

    const int units = p.chunk_offsets[p.num_seqs] * H;
    for (int unit = blockIdx.x; unit < units; unit += gridDim.x) {
        const int h = unit % H, ci = unit / H;
        int n = 0;
        {                                             // the sequence of chunk unit ci: choff[n] <= ci < choff[n + 1]
            int hi = p.num_seqs;
            while (hi - n > 1) {
                const int mid = (n + hi) >> 1;
                if (p.chunk_offsets[mid] <= ci) n = mid; else hi = mid;
            }
        }
        const int c = ci - p.chunk_offsets[n];
        const int32_t tb = p.cu_seqlens[n], te = p.cu_seqlens[n + 1];
        if (tb < 0 || te < tb || te > p.total_tokens) {
            if (tid == 0) atomicOr(p.err, KDA_DEVERR_CU_SEQLENS);
            continue;
        }
        const int64_t sidx = ((int64_t)n * H + h) * MD * MD;
        const int nch = (te - tb + kChunk - 1) / kChunk;
        const int32_t t0 = tb + c * kChunk;
        const int L = min(kChunk, te - t0);
        // S_0: the initial state or the snapshot after chunk c - 1; dS_1: grad_state_out or from pass 2
        const float* S0 = c == 0 ? (p.state_in ? p.state_in + sidx : nullptr)
                                 : p.snapshots + ((int64_t)(p.snap_offsets[n] + c - 1) * H + h) * MD * MD;
        const float* dS1 = c == nch - 1 ? (p.d_state_out ? p.d_state_out + sidx : nullptr)
                                        : p.dstate_b + ((int64_t)(p.snap_offsets[n] + c) * H + h) * MD * MD;

        // ---- inputs: k (shared), q, v, dO = scale grad_o (scratch), log2 alpha (shared), beta ----
        {
            constexpr int EV = 16 / (int)sizeof(TIn);
#pragma unroll
            for (int jj = 0; jj < MAT / EV / MNT; ++jj) {
                const int e0 = (tid + MNT * jj) * EV, r = e0 >> 7;
                const int64_t g0 = ((int64_t)(t0 + r) * H + h) * MD + (e0 & 127);
                float kv[EV], qv[EV], vv[EV], dv[EV], av[EV];
                if (r < L) {
                    ld16f(gk + g0, kv);
                    ld16f(gq + g0, qv);
                    ld16f(gv + g0, vv);
                    ld16f(gdo + g0, dv);
#pragma unroll
                    for (int x = 0; x < EV; x += 4) ld16f(p.alpha + g0 + x, av + x);
#pragma unroll
                    for (int x = 0; x < EV; ++x) av[x] = fmaxf(__log2f(av[x]), kLog2AlphaMin);
                } else {
#pragma unroll
                    for (int x = 0; x < EV; ++x) kv[x] = qv[x] = vv[x] = dv[x] = av[x] = 0.f;
                }
#pragma unroll
                for (int x = 0; x < EV; x += 4) {
                    st4(sK + e0 + x, kv + x);
                    st4(M(XQ) + e0 + x, qv + x);
                    st4(M(XV) + e0 + x, vv + x);
                    st4(M(XDO) + e0 + x, dv + x, p.scale);
                    st4(sG + e0 + x, av + x);
                }
            }
        }
        if (tid < MC) sbeta[tid] = tid < L ? p.beta[(int64_t)(t0 + tid) * H + h] : 0.f;
        {                                              // sum_j dS_1[i][j] S_0[i][j]: two threads per key row
            const int i = tid >> 1, j0 = (tid & 1) * 64;
            float sr = 0.f;
            if (S0 && dS1) {
#pragma unroll
                for (int j = 0; j < 64; j += 4) {
                    const float4 a4 = __ldg(reinterpret_cast<const float4*>(dS1 + i * MD + j0 + j));
                    const float4 b4 = __ldg(reinterpret_cast<const float4*>(S0 + i * MD + j0 + j));
                    sr = fmaf(a4.x, b4.x, fmaf(a4.y, b4.y, fmaf(a4.z, b4.z, fmaf(a4.w, b4.w, sr))));
                }
            }
            sr += __shfl_xor_sync(0xffffffffu, sr, 1);
            if ((tid & 1) == 0) srow[i] = sr;
        }
        __syncthreads();
        {                                              // G = running sum over rows, two threads per key channel
            const int i = tid & 127, half = tid >> 7;
            float run = 0.f, v[32];
#pragma unroll
            for (int rr = 0; rr < 32; ++rr) {
                run += sG[(32 * half + rr) * MD + i];
                v[rr] = run;
            }
            if (half == 0) scol[i] = run;
            __syncthreads();
            const float off = half ? scol[i] : 0.f;
#pragma unroll
            for (int rr = 0; rr < 32; ++rr) sG[(32 * half + rr) * MD + i] = v[rr] + off;
            if (half) sgc[i] = v[31] + off;
        }
        __syncthreads();

        // ---- Bt and P, one block of 16 rows at a time (reference row 16 b + 7) ----
        for (int b = 0; b < 4; ++b) {
            const int ref = 16 * b + 7, ns = 16 * (b + 1);
            float* sKB = stg;                          // [16][LDY]: k_r 2^(G_r - G_ref) for the block's rows
            float* sQB = stg + 16 * LDY;               // [16][LDY]: q_r 2^(G_r - G_ref)
            for (int e = tid; e < ns * MD; e += MNT) {
                const int s = e >> 7, i = e & 127;
                sY[s * LDY + i] = cv(sK[e] * ex2a(G[ref * MD + i] - G[e]));
            }
            {
                float qv[16 * MD / MNT];
#pragma unroll
                for (int u = 0; u < 16 * MD / MNT; ++u) qv[u] = M(XQ)[16 * b * MD + tid + MNT * u];
#pragma unroll
                for (int u = 0; u < 16 * MD / MNT; ++u) {
                    const int e = tid + MNT * u, r = e >> 7, i = e & 127, x = 16 * b * MD + e;
                    const float f = ex2a(G[x] - G[ref * MD + i]);
                    sKB[r * LDY + i] = cv(sK[x] * f);
                    sQB[r * LDY + i] = cv(qv[u] * f);
                }
            }
            __syncthreads();
            if constexpr (TC) {
                // [KB; QB] (32 x 128) times Y^T (128 x ns): m-tile 0 gives Bt, m-tile 1 gives P
                const int ntn = ns / 8, g = lane >> 2, t = lane & 3;
                for (int tau = warp; tau < 2 * ntn; tau += 8) {
                    const int mt = tau / ntn, nt = tau - mt * ntn;
                    const float* Ab = stg + mt * 16 * LDY;
                    float d[4] = {0.f, 0.f, 0.f, 0.f};
                    tile_mma(d, MD / 8, [&](int m, int k) { return __float_as_uint(Ab[m * LDY + k]); },
                             [&](int k, int n) { return __float_as_uint(sY[(8 * nt + n) * LDY + k]); });
#pragma unroll
                    for (int q = 0; q < 4; ++q) {
                        const int r = 16 * b + g + 8 * (q >> 1), sc = 8 * nt + 2 * t + (q & 1);
                        if (mt == 0) sBT[r * LD64 + sc] = sc < r ? d[q] : 0.f;
                        else sP[r * LD64 + sc] = sc <= r ? d[q] : 0.f;
                    }
                }
                for (int e = tid; e < 16 * (MC - ns); e += MNT) {     // the block's rows right of column ns
                    const int r = 16 * b + e / (MC - ns), sc = ns + e % (MC - ns);
                    sBT[r * LD64 + sc] = 0.f;
                    sP[r * LD64 + sc] = 0.f;
                }
                __syncthreads();
                continue;
            }
            const int o = tr, r = 16 * b + o;
            float dk4[4] = {0.f, 0.f, 0.f, 0.f}, dq4[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll 4
            for (int i = 0; i < MD; i += 4) {
                const float4 kb = *reinterpret_cast<const float4*>(sKB + o * LDY + i);
                const float4 qb = *reinterpret_cast<const float4*>(sQB + o * LDY + i);
#pragma unroll
                for (int j = 0; j < 4; ++j) {
                    const int s = tc + 16 * j;
                    if (s < ns) {
                        const float4 y = *reinterpret_cast<const float4*>(sY + s * LDY + i);
                        dk4[j] = fmaf(kb.x, y.x, fmaf(kb.y, y.y, fmaf(kb.z, y.z, fmaf(kb.w, y.w, dk4[j]))));
                        dq4[j] = fmaf(qb.x, y.x, fmaf(qb.y, y.y, fmaf(qb.z, y.z, fmaf(qb.w, y.w, dq4[j]))));
                    }
                }
            }
#pragma unroll
            for (int j = 0; j < 4; ++j) {
                const int s = tc + 16 * j;
                sBT[r * LD64 + s] = s < r ? dk4[j] : 0.f;
                sP[r * LD64 + s] = s <= r ? dq4[j] : 0.f;
            }
            __syncthreads();
        }

        // ---- T = (I + A)^-1, A = Diag(beta) Bt, by 16 x 16 blocks: each diagonal block by forward substitution
        //      (a thread per column), then T_bc = -T_bb sum_{m = c}^{b - 1} A_bm T_mc in order of b - c ----
        for (int e = tid; e < MC * MC; e += MNT) sT[(e >> 6) * LD64 + (e & 63)] = 0.f;
        __syncthreads();
        if (tid < MC) {                                // a thread per column c of diagonal block b
            const int b = tid >> 4, c = tid & 15;
            // right-looking: once t[m] is known it enters every later row's sum (the same FMAs in the same
            // order per sum as row by row, with a dependent path of one FMA per row)
            float t[16], z[16];
#pragma unroll
            for (int r = 0; r < 16; ++r) z[r] = 0.f;
#pragma unroll
            for (int m = 0; m < 16; ++m) {
                t[m] = m == c ? 1.f : (m > c ? -sbeta[16 * b + m] * z[m] : 0.f);
#pragma unroll
                for (int r = m + 1; r < 16; ++r) z[r] = fmaf(sBT[(16 * b + r) * LD64 + 16 * b + m], t[m], z[r]);
            }
#pragma unroll
            for (int r = 0; r < 16; ++r) sT[(16 * b + r) * LD64 + 16 * b + c] = t[r];
        }
        __syncthreads();
        {
            float* sZ = sY;                            // [64][LD64]
            for (int d = 1; d < 4; ++d) {
                for (int e = tid; e < (4 - d) * 256; e += MNT) {
                    const int c = e >> 8, b = c + d, r = 16 * b + ((e >> 4) & 15), col = 16 * c + (e & 15);
                    float z = 0.f;
                    for (int m = 16 * c; m < 16 * b; ++m) z = fmaf(sBT[r * LD64 + m], sT[m * LD64 + col], z);
                    sZ[r * LD64 + col] = sbeta[r] * z;
                }
                __syncthreads();
                for (int e = tid; e < (4 - d) * 256; e += MNT) {
                    const int c = e >> 8, b = c + d, r = 16 * b + ((e >> 4) & 15), col = 16 * c + (e & 15);
                    float t = 0.f;
                    for (int m = 16 * b; m <= r; ++m) t = fmaf(sT[r * LD64 + m], sZ[m * LD64 + col], t);
                    sT[r * LD64 + col] = -t;
                }
                __syncthreads();
            }
        }
        // beta Gamma K, beta V and Khat = 2^(G_C - G) K
#pragma unroll 1
        for (int e0 = tid; e0 < MAT; e0 += 8 * MNT) {
            float vv[8];
#pragma unroll
            for (int u = 0; u < 8; ++u) vv[u] = M(XV)[e0 + MNT * u];
#pragma unroll
            for (int u = 0; u < 8; ++u) {
                const int e = e0 + MNT * u, r = e >> 7, i = e & 127;
                const float kk = sK[e], g = G[e];
                M(XKTB)[e] = sbeta[r] * kk * ex2a(g);
                M(XVB)[e] = sbeta[r] * vv[u];
                M(XKH)[e] = kk * ex2a(sgc[i] - g);
            }
        }
        __syncthreads();

        float acc[4][8];
        // W = T (beta Gamma K);  Utilde = T (beta V);  U = Utilde - W S_0
        zero<128>(acc);
        prod<TC, 128, 64, true, false, false, false, 5>(sT, LD64, M(XKTB), MD, ring5, stg, acc);
        put128<TC>(M(XW), acc);
        zero<128>(acc);
        prod<TC, 128, 64, true, false, false, false, 5>(sT, LD64, M(XVB), MD, ring5, stg, acc);
        __syncthreads();                               // W is written
        if (S0) {
            float ws[4][8];
            zero<128>(ws);
            prod<TC, 128, 128, false, false, false, false, 5>(M(XW), MD, S0, MD, ring5, stg, ws);
#pragma unroll
            for (int i = 0; i < 4; ++i)
#pragma unroll
                for (int j = 0; j < 8; ++j) acc[i][j] -= ws[i][j];
        }
        put128<TC>(M(XU), acc);
        __syncthreads();
        // dU = P^T dO + Khat dS_1
        zero<128>(acc);
        prod<TC, 128, 64, true, true, false, false, 5>(sP, LD64, M(XDO), MD, ring5, stg, acc);
        if (dS1) prod<TC, 128, 128, false, false, false, false, 5>(M(XKH), MD, dS1, MD, ring5, stg, acc);
        put128<TC>(M(XDU), acc);
        // dP = dO U^T on s <= r
        {
            float a64[4][4];
            zero<64>(a64);
            prod<TC, 64, 128, false, false, false, true, 5>(M(XDO), MD, M(XU), MD, ring5, stg, a64);
#pragma unroll
            for (int i = 0; i < 4; ++i)
#pragma unroll
                for (int j = 0; j < 4; ++j) {
                    const int r = mrow<TC>(i), s = mcol<64, TC>(j);
                    sDP[r * LD64 + s] = s <= r ? a64[i][j] : 0.f;
                }
        }
        __syncthreads();
        // dQs = dO S_0^T;  dKhat = U dS_1^T;  dW = -dU S_0^T
        zero<128>(acc);
        if (S0) prod<TC, 128, 128, false, false, false, true, 4>(M(XDO), MD, S0, MD, ring4, stg, acc);
        put128<TC>(M(XDQS), acc);
        zero<128>(acc);
        if (dS1) prod<TC, 128, 128, false, false, false, true, 4>(M(XU), MD, dS1, MD, ring4, stg, acc);
        put128<TC>(M(XDKH), acc);
        zero<128>(acc);
        if (S0) prod<TC, 128, 128, false, false, false, true, 4>(M(XDU), MD, S0, MD, ring4, stg, acc);
        put128<TC>(M(XDW), acc, -1.f);
        __syncthreads();
        // dT = dW (beta Gamma K)^T + dU (beta V)^T, kept on a > b (the only part T^T dT T^T reads below
        // the diagonal); X = dT T^T; dA = -(T^T X) on s < r
        float* sDT = sP;                               // P is not read after dU
        float* sX = sDA;                               // dA is written once X has been read
        {
            float a64[4][4];
            zero<64>(a64);
            prod<TC, 64, 128, false, false, false, true, 4>(M(XDW), MD, M(XKTB), MD, ring4, stg, a64);
            prod<TC, 64, 128, false, false, false, true, 4>(M(XDU), MD, M(XVB), MD, ring4, stg, a64);
#pragma unroll
            for (int i = 0; i < 4; ++i)
#pragma unroll
                for (int j = 0; j < 4; ++j) {
                    const int r = mrow<TC>(i), s = mcol<64, TC>(j);
                    sDT[r * LD64 + s] = s < r ? a64[i][j] : 0.f;
                }
            __syncthreads();
            zero<64>(a64);
            prod<TC, 64, 64, true, false, true, true>(sDT, LD64, sT, LD64, sY, stg, a64);
#pragma unroll
            for (int i = 0; i < 4; ++i)
#pragma unroll
                for (int j = 0; j < 4; ++j) sX[mrow<TC>(i) * LD64 + mcol<64, TC>(j)] = a64[i][j];
            __syncthreads();
            zero<64>(a64);
            prod<TC, 64, 64, true, true, true, false>(sT, LD64, sX, LD64, sY, stg, a64);
#pragma unroll
            for (int i = 0; i < 4; ++i)
#pragma unroll
                for (int j = 0; j < 4; ++j) {
                    const int r = mrow<TC>(i), s = mcol<64, TC>(j);
                    sDA[r * LD64 + s] = s < r ? -a64[i][j] : 0.f;
                }
        }
        // T^T dW, T^T dU
        zero<128>(acc);
        prod<TC, 128, 64, true, true, false, false>(sT, LD64, M(XDW), MD, sY, stg, acc);
        put128<TC>(M(XTDW), acc);
        zero<128>(acc);
        prod<TC, 128, 64, true, true, false, false>(sT, LD64, M(XDU), MD, sY, stg, acc);
        put128<TC>(M(XTDU), acc);
        __syncthreads();
        // sum_s dA_rs Bt_rs per row, then dA -> dBt = Diag(beta) dA
        for (int r = warp; r < MC; r += 8) {
            float s = sDA[r * LD64 + lane] * sBT[r * LD64 + lane] + sDA[r * LD64 + 32 + lane] * sBT[r * LD64 + 32 + lane];
#pragma unroll
            for (int o = 16; o > 0; o >>= 1) s += __shfl_xor_sync(0xffffffffu, s, o);
            if (lane == 0) sdb[r] = s;
        }
        __syncthreads();
        for (int e = tid; e < MC * MC; e += MNT) sDA[(e >> 6) * LD64 + (e & 63)] *= sbeta[e >> 6];
        __syncthreads();

        // ---- row-side decayed sums for block b: sum_{s} X_rs k_s E_rs = 2^(G_r - G_ref) sum_s X_rs Y_s ----
        for (int b = 0; b < 4; ++b) {
            const int ref = 16 * b + 7, ns = 16 * (b + 1);
            for (int e = tid; e < ns * MD; e += MNT) {
                const int s = e >> 7, i = e & 127;
                sY[s * LDY + i] = sK[e] * ex2a(G[ref * MD + i] - G[e]);
            }
            __syncthreads();
            if constexpr (TC) {
                // [dP; dBt] rows of the block (32 x ns) times Y (ns x 128), split TF32: m-tile 0 gives dq_p,
                // m-tile 1 dk_r
                // (warp w: column tiles w and w + 8 of both)
                const int g = lane >> 2, t = lane & 3;
                float d[2][2][4] = {};
                tiles_mma3<2, 2>(d, ns / 8,
                                 [&](int ma, int m, int k) { return (ma == 0 ? sDP : sDA)[(16 * b + m) * LD64 + k]; },
                                 [&](int nb, int k, int n) { return sY[k * LDY + 8 * (warp + 8 * nb) + n]; });
#pragma unroll
                for (int ma = 0; ma < 2; ++ma) {
                    float* out = M(ma == 0 ? XRQ : XRK);
#pragma unroll
                    for (int nb = 0; nb < 2; ++nb)
#pragma unroll
                        for (int q = 0; q < 4; ++q) {
                            const int r = 16 * b + g + 8 * (q >> 1), i = 8 * (warp + 8 * nb) + 2 * t + (q & 1);
                            out[r * MD + i] = ex2a(G[r * MD + i] - G[ref * MD + i]) * d[ma][nb][q];
                        }
                }
                __syncthreads();
                continue;
            }
            const int r = 16 * b + tr;
            float aq[8], ak[8];
#pragma unroll
            for (int j = 0; j < 8; ++j) aq[j] = ak[j] = 0.f;
            for (int s = 0; s < ns; ++s) {
                const float xp = sDP[r * LD64 + s], xa = sDA[r * LD64 + s];
                const float4 y0 = *reinterpret_cast<const float4*>(sY + s * LDY + 4 * tc);
                const float4 y1 = *reinterpret_cast<const float4*>(sY + s * LDY + 64 + 4 * tc);
                const float yv[8] = {y0.x, y0.y, y0.z, y0.w, y1.x, y1.y, y1.z, y1.w};
#pragma unroll
                for (int j = 0; j < 8; ++j) {
                    aq[j] = fmaf(xp, yv[j], aq[j]);
                    ak[j] = fmaf(xa, yv[j], ak[j]);
                }
            }
#pragma unroll
            for (int j = 0; j < 8; ++j) {
                const int i = col8(j);
                const float f = ex2a(G[r * MD + i] - G[ref * MD + i]);
                M(XRQ)[r * MD + i] = f * aq[j];
                M(XRK)[r * MD + i] = f * ak[j];
            }
            __syncthreads();
        }
        // ---- column-side decayed sums for block b of s: sum_{r >= s} X_rs y_r E_rs
        //      = 2^(G_ref - G_s) sum_r X_rs (y_r 2^(G_r - G_ref)), y = q with X = dP, y = k with X = dBt ----
        if constexpr (TC) {
            // both passes of block b share the factors 2^(G_r - G_ref) and 2^(G_ref - G_s): one build writes
            // Y_q (q rows, in sY) and Y_k (k rows, in the P and T area, free since the products), then the two
            // split-TF32 products, X^T (16 x (64 - r0), the block's columns s) times Y ((64 - r0) x 128)
            float* sYk = sP;                           // [64][LDY] over P and T
            const int g = lane >> 2, t = lane & 3;
            for (int b = 0; b < 4; ++b) {
                const int ref = 16 * b + 7, r0 = 16 * b;
#pragma unroll 1
                for (int e0 = r0 * MD + tid; e0 < MAT; e0 += 8 * MNT) {
                    float yv[8];
#pragma unroll
                    for (int u = 0; u < 8; ++u) yv[u] = M(XQ)[e0 + MNT * u];
#pragma unroll
                    for (int u = 0; u < 8; ++u) {
                        const int e = e0 + MNT * u, r = e >> 7, i = e & 127;
                        const float f = ex2a(G[e] - G[ref * MD + i]);
                        sY[(r - r0) * LDY + i] = yv[u] * f;
                        sYk[(r - r0) * LDY + i] = sK[e] * f;
                    }
                }
                __syncthreads();
                float dd[2][2][4] = {};                    // [0]: X = dP, Y = Y_q; [1]: X = dBt, Y = Y_k
                tiles_mma3_sep<2, 2>(dd, (MC - r0) / 8,
                                     [&](int ma, int m, int k) { return (ma ? sDA : sDP)[(r0 + k) * LD64 + r0 + m]; },
                                     [&](int ma, int nb, int k, int n) {
                                         return (ma ? sYk : sY)[k * LDY + 8 * (warp + 8 * nb) + n];
                                     });
#pragma unroll
                for (int nb = 0; nb < 2; ++nb)
#pragma unroll
                    for (int q = 0; q < 4; ++q) {
                        const int sr = r0 + g + 8 * (q >> 1), i = 8 * (warp + 8 * nb) + 2 * t + (q & 1);
                        const float f = ex2a(G[ref * MD + i] - G[sr * MD + i]);
                        M(XCP)[sr * MD + i] = f * dd[0][nb][q];
                        M(XCK)[sr * MD + i] = f * dd[1][nb][q];
                    }
                __syncthreads();
            }
        } else {
            for (int b = 0; b < 4; ++b) {
                const int ref = 16 * b + 7, r0 = 16 * b;
                for (int pass = 0; pass < 2; ++pass) {
                    const float* src = pass == 0 ? M(XQ) : sK;
                    const float* xs = pass == 0 ? sDP : sDA;
#pragma unroll 1
                    for (int e0 = r0 * MD + tid; e0 < MAT; e0 += 8 * MNT) {      // (64 - r0) x 128 = 2048 multiples
                        float yv[8];
#pragma unroll
                        for (int u = 0; u < 8; ++u) yv[u] = src[e0 + MNT * u];
#pragma unroll
                        for (int u = 0; u < 8; ++u) {
                            const int e = e0 + MNT * u, r = e >> 7, i = e & 127;
                            sY[(r - r0) * LDY + i] = yv[u] * ex2a(G[e] - G[ref * MD + i]);
                        }
                    }
                    __syncthreads();
                    const int s = r0 + tr;
                    float a8[8];
#pragma unroll
                    for (int j = 0; j < 8; ++j) a8[j] = 0.f;
                    for (int r = r0; r < MC; ++r) {
                        const float x = xs[r * LD64 + s];
                        const float4 y0 = *reinterpret_cast<const float4*>(sY + (r - r0) * LDY + 4 * tc);
                        const float4 y1 = *reinterpret_cast<const float4*>(sY + (r - r0) * LDY + 64 + 4 * tc);
                        const float yv[8] = {y0.x, y0.y, y0.z, y0.w, y1.x, y1.y, y1.z, y1.w};
#pragma unroll
                        for (int j = 0; j < 8; ++j) a8[j] = fmaf(x, yv[j], a8[j]);
                    }
                    float* out = M(pass == 0 ? XCP : XCK);
#pragma unroll
                    for (int j = 0; j < 8; ++j) {
                        const int i = col8(j);
                        out[s * MD + i] = ex2a(G[ref * MD + i] - G[s * MD + i]) * a8[j];
                    }
                    __syncthreads();
                }
            }
        }
        // ---- dq, dk, dv; dg into shared memory (the P and T area, free since the column-side sums); the
        //      rest of dbeta (row sums of Gamma k . T^T dW + v . T^T dU) and the column sums of dKhat . Khat
        //      on the way.  Element x = tid + 256 u keeps the key channel i = tid % 128; 8 elements at a
        //      time, their loads issued before any store ----
        float* sDG = sP;                               // [64][128]
        float colp = 0.f;
#pragma unroll 1
        for (int x0 = tid; x0 < MAT; x0 += 8 * MNT) {
            float rq[8], rk[8], cp[8], ck[8], dqs[8], tdw[8], dkh[8], tdu[8], qv[8], vv[8];
#pragma unroll
            for (int u = 0; u < 8; ++u) {
                const int x = x0 + MNT * u;
                rq[u] = M(XRQ)[x]; rk[u] = M(XRK)[x]; cp[u] = M(XCP)[x]; ck[u] = M(XCK)[x];
                dqs[u] = M(XDQS)[x]; tdw[u] = M(XTDW)[x]; dkh[u] = M(XDKH)[x]; tdu[u] = M(XTDU)[x];
                qv[u] = M(XQ)[x]; vv[u] = M(XV)[x];
            }
#pragma unroll
            for (int u = 0; u < 8; ++u) {
                const int x = x0 + MNT * u, r = x >> 7, i = x & 127;
                const float gam = ex2a(G[x]), kh = ex2a(sgc[i] - G[x]);
                const float kv = sK[x], be = sbeta[r];
                const float d = qv[u] * rq[u] - kv * cp[u] + kv * rk[u] - kv * ck[u] + dqs[u] * qv[u] * gam +
                                be * tdw[u] * kv * gam - dkh[u] * kv * kh;
                colp = fmaf(dkh[u], kv * kh, colp);
                sY[r * LDY + i] = fmaf(kv * gam, tdw[u], vv[u] * tdu[u]);     // summed by rows below
                sDG[x] = r < L ? d : 0.f;
                if (r < L) {
                    const int64_t o = ((int64_t)(t0 + r) * H + h) * MD + i;
                    st_out(gdq, o, rq[u] + dqs[u] * gam);
                    st_out(gdk, o, cp[u] + rk[u] + ck[u] + be * tdw[u] * gam + dkh[u] * kh);
                    st_out(gdv, o, be * tdu[u]);
                }
            }
        }
        scol[(tid >> 7) * 128 + (tid & 127)] = colp;
        __syncthreads();
        {                                              // row sums of the dbeta terms: four threads per row
            const int r = tid >> 2, q4 = tid & 3;
            float db = 0.f;
#pragma unroll
            for (int j = 0; j < 32; j += 4) {
                const float4 v4 = *reinterpret_cast<const float4*>(sY + r * LDY + 32 * q4 + j);
                db += (v4.x + v4.y) + (v4.z + v4.w);
            }
            db += __shfl_xor_sync(0xffffffffu, db, 1);
            db += __shfl_xor_sync(0xffffffffu, db, 2);
            if (q4 == 0 && r < L) p.d_beta[(int64_t)(t0 + r) * H + h] = sdb[r] + db;
        }
        // ---- d ln alpha = running sum of dg from the last row up; dalpha = d ln alpha / alpha ----
        {
            const int i = tid & 127, half = tid >> 7;
            // the last row's own term: sum_s dKhat . Khat + Gamma_L . rowsum(dS_1 . S_0)
            const float extra = scol[i] + scol[128 + i] + ex2a(sgc[i]) * srow[i];
            float dg[32], al[32], tot = 0.f;
#pragma unroll
            for (int rr = 0; rr < 32; ++rr) {
                const int r = 32 * half + rr;
                dg[rr] = sDG[r * MD + i] + (r == L - 1 ? extra : 0.f);
                al[rr] = r < L ? __ldg(p.alpha + ((int64_t)(t0 + r) * H + h) * MD + i) : 1.f;
                tot += dg[rr];
            }
            __syncthreads();                           // every thread has read the column sums
            if (half == 1) scol[i] = tot;
            __syncthreads();
            float run = half == 0 ? scol[i] : 0.f;
#pragma unroll
            for (int rr = 31; rr >= 0; --rr) {
                const int r = 32 * half + rr;
                run += dg[rr];
                if (r < L) st_out(p.d_alpha, ((int64_t)(t0 + r) * H + h) * MD + i, run / al[rr]);
            }
        }
        __syncthreads();                               // the scratch and shared matrices are free
    }
}

}  // namespace

cudaError_t launch_bwd_chunk_mat(const BwdParams& p, kda_dtype dt, int grid, cudaStream_t s) {
    constexpr int smem = MAT_SMEM_FLOATS * 4;
    cudaError_t e;
    if (dt == KDA_DTYPE_BF16) {
        if ((e = cudaFuncSetAttribute(kda_bwd_chunk_mat_kernel<__nv_bfloat16>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                      smem)) != cudaSuccess)
            return e;
        kda_bwd_chunk_mat_kernel<__nv_bfloat16><<<grid, MNT, smem, s>>>(p);
    } else {
        if ((e = cudaFuncSetAttribute(kda_bwd_chunk_mat_kernel<float>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                      smem)) != cudaSuccess)
            return e;
        kda_bwd_chunk_mat_kernel<float><<<grid, MNT, smem, s>>>(p);
    }
    return cudaGetLastError();
}

}  // namespace kda
