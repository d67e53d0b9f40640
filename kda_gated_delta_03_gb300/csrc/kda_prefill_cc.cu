// Chunkwise KDA prefill on CUDA cores, float32 arithmetic throughout.
//
// This is the precise path (float32 inputs, and every head size this build
// supports).  It follows the chunkwise form of the recurrence ("Kimi K3,
// explained", section "Training in chunks": WY representation inside a chunk,
// only the state carried between chunks).  Per head, chunk of C = 64 tokens
// r = 0..L-1 starting from state S (d_k x d_v):
//
//   g_r   = sum_{s<=r} log2 alpha_s                    (per key channel)
//   A_rs  = beta_r sum_i k_ri k_si 2^(g_ri - g_si)      s <  r
//   P_rs  =        sum_i q_ri k_si 2^(g_ri - g_si)      s <= r
//   [W | Utilde] = (I + A)^-1 Diag(beta) [2^g . K | V]  (forward substitution)
//   U     = Utilde - W S
//   O     = (2^g . Q) S + P U,          o = scale * O
//   S     = Diag(2^g_L) S + Khat^T U,   Khat_s = 2^(g_L - g_s) . k_s
//
// The decay products 2^(g_ri - g_si) are factorised per 16-row block b with a
// reference g_ref(b) = g at row 16b+7: k_ri 2^(g_ri - g_ref) times
// k_si 2^(g_ref - g_si).  With log2 alpha clamped at -15 per token both factors
// stay inside float32 range (|exponent| <= 8 * 15 within the block, and <= 0
// for earlier columns), so no per-element exponential is needed.
//
// Work item: (sequence, head, d_v slice of NV columns).  Value columns of the
// state are independent, so slices only repeat the key-only work.

#include "kda_internal.cuh"

namespace kda {
namespace {

constexpr int C = kChunk;
constexpr int NT = 256;

template <int DK, int NV>
struct CcSmem {
    static constexpr int LDR = DK + 1;           // odd stride: column access across lanes
    static constexpr int LDX = DK + NV;
    static constexpr int XFLOATS = (C * LDX > C * LDR) ? C * LDX : C * LDR;
    float K[C * DK];      // k, later Khat
    float Q[C * DK];      // q, later Gamma . q
    float G[C * DK];      // cumulative log2 decay
    float X[XFLOATS];     // R factors (A/P stage), then [W | Utilde], then [W | U]
    float A[C * C];
    float P[C * C];
    float S[DK * NV];     // state slice
    float Lk[16 * DK];    // row factors of the current row block
    float Lq[16 * DK];
    float beta[C];
    float ref[DK];
    float ref_prev[DK];
    float gamL[DK];
};

template <int DK, int NV, typename TIn>
__global__ void __launch_bounds__(NT, 1) kda_prefill_cc_kernel(PrefillParams p) {
    extern __shared__ __align__(16) unsigned char smem_raw[];
    using Sm = CcSmem<DK, NV>;
    Sm& sm = *reinterpret_cast<Sm*>(smem_raw);
    constexpr int LDR = Sm::LDR;
    constexpr int LDX = Sm::LDX;
    const int tid = threadIdx.x;

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
    const bool bad = t_begin < 0 || t_end < t_begin || t_end > p.total_tokens || (n == 0 && t_begin != 0) ||
                     (n == p.num_seqs - 1 && t_end != p.total_tokens);
    if (bad) {
        if (tid == 0) atomicOr(p.err, KDA_DEVERR_CU_SEQLENS);
        return;
    }
    if (tid == 0 && h == 0 && slice == 0 && snapshot_offsets_bad(p, n, t_end - t_begin))
        atomicOr(p.err, KDA_DEVERR_SNAPSHOTS);
    const int H = p.H;
    const TIn* gq = static_cast<const TIn*>(p.q);
    const TIn* gk = static_cast<const TIn*>(p.k);
    const TIn* gv = static_cast<const TIn*>(p.v);
    TIn* go = static_cast<TIn*>(p.o);
    const int64_t state_off = ((int64_t)n * H + h) * DK * (int64_t)p.dv;

    // ---- state in ----
    for (int e = tid; e < DK * NV; e += NT) {
        const int i = e / NV, j = e % NV;
        sm.S[e] = p.state_in ? p.state_in[state_off + (int64_t)i * p.dv + j0 + j] : 0.f;
    }

    for (int32_t t0 = t_begin; t0 < t_end; t0 += C) {
        const int L = min(C, t_end - t0);
        __syncthreads();

        // ---- stage 0: load k, q (padded rows are zero), beta ----
        for (int e = tid; e < C * DK; e += NT) {
            const int r = e / DK, i = e % DK;
            const int64_t gi = ((int64_t)(t0 + r) * H + h) * DK + i;
            sm.K[e] = r < L ? load_as_float(gk, gi) : 0.f;
            sm.Q[e] = r < L ? load_as_float(gq, gi) : 0.f;
        }
        for (int e = tid; e < C * DK; e += NT) {
            const int r = e / DK, i = e % DK;
            sm.G[e] = r < L ? fmaxf(log2f(alpha_at(p.alpha, p.alpha_mode, (int64_t)(t0 + r) * H + h, DK, i)),
                                    kLog2AlphaMin)
                            : 0.f;
        }
        for (int r = tid; r < C; r += NT) sm.beta[r] = r < L ? p.beta[(int64_t)(t0 + r) * H + h] : 0.f;
        __syncthreads();

        // ---- stage 1: cumulative log2 decay per channel (in place) ----
        if (tid < DK) {
            float g = 0.f;
            for (int r = 0; r < C; ++r) {
                g += sm.G[r * DK + tid];
                sm.G[r * DK + tid] = g;
            }
        }
        __syncthreads();

        // ---- stage 2: A and P, one 16-row block at a time ----
        for (int b = 0; b * 16 < L; ++b) {
            const int ncol = 16 * (b + 1);
            for (int i = tid; i < DK; i += NT) {
                sm.ref_prev[i] = b ? sm.ref[i] : 0.f;
                sm.ref[i] = sm.G[(16 * b + 7) * DK + i];
            }
            __syncthreads();
            // R rows: new block s in [16b, 16b+16), rescale of earlier rows
            for (int e = tid; e < ncol * DK; e += NT) {
                const int s = e / DK, i = e % DK;
                if (s >= 16 * b)
                    sm.X[s * LDR + i] = sm.K[s * DK + i] * exp2f(sm.ref[i] - sm.G[s * DK + i]);
                else
                    sm.X[s * LDR + i] *= exp2f(sm.ref[i] - sm.ref_prev[i]);
            }
            for (int e = tid; e < 16 * DK; e += NT) {
                const int rr = e / DK, i = e % DK;
                const int r = 16 * b + rr;
                const float f = exp2f(sm.G[r * DK + i] - sm.ref[i]);
                sm.Lk[e] = sm.K[r * DK + i] * f;
                sm.Lq[e] = sm.Q[r * DK + i] * f;
            }
            __syncthreads();
            for (int e = tid; e < 16 * ncol; e += NT) {
                const int rr = e / ncol, s = e % ncol;
                const int r = 16 * b + rr;
                float a = 0.f, pq = 0.f;
                if (s <= r) {
                    const float* lk = sm.Lk + rr * DK;
                    const float* lq = sm.Lq + rr * DK;
                    const float* rs = sm.X + s * LDR;
#pragma unroll 8
                    for (int i = 0; i < DK; ++i) {
                        a = fmaf(lk[i], rs[i], a);
                        pq = fmaf(lq[i], rs[i], pq);
                    }
                }
                sm.A[r * C + s] = s < r ? sm.beta[r] * a : 0.f;
                sm.P[r * C + s] = pq;
            }
            __syncthreads();
        }

        // ---- stage 3: [W | Utilde] = (I + A)^-1 Diag(beta) [2^g . K | V] ----
        for (int e = tid; e < C * LDX; e += NT) {
            const int r = e / LDX, c = e % LDX;
            float x = 0.f;
            if (r < L) {
                if (c < DK)
                    x = sm.beta[r] * exp2f(sm.G[r * DK + c]) * sm.K[r * DK + c];
                else
                    x = sm.beta[r] * load_as_float(gv, ((int64_t)(t0 + r) * H + h) * p.dv + j0 + (c - DK));
            }
            sm.X[r * LDX + c] = x;
        }
        __syncthreads();
        for (int c = tid; c < LDX; c += NT) {          // each column is an independent triangular solve
            for (int r = 1; r < L; ++r) {
                float acc0 = sm.X[r * LDX + c], acc1 = 0.f;
                const float* arow = sm.A + r * C;
                int s = 0;
                for (; s + 1 < r; s += 2) {
                    acc0 = fmaf(-arow[s], sm.X[s * LDX + c], acc0);
                    acc1 = fmaf(-arow[s + 1], sm.X[(s + 1) * LDX + c], acc1);
                }
                if (s < r) acc0 = fmaf(-arow[s], sm.X[s * LDX + c], acc0);
                sm.X[r * LDX + c] = acc0 + acc1;
            }
        }
        // ---- stage 4: Khat, Gamma . Q, Gamma_L (in place) ----
        for (int e = tid; e < C * DK; e += NT) {
            const int r = e / DK, i = e % DK;
            const float g = sm.G[r * DK + i];
            const float gl = sm.G[(C - 1) * DK + i];
            sm.K[e] *= exp2f(gl - g);
            sm.Q[e] *= exp2f(g);
        }
        for (int i = tid; i < DK; i += NT) sm.gamL[i] = exp2f(sm.G[(C - 1) * DK + i]);
        __syncthreads();

        // ---- stage 5: U = Utilde - W S (in place of Utilde) ----
        for (int e = tid; e < C * NV; e += NT) {
            const int r = e / NV, j = e % NV;
            const float* w = sm.X + r * LDX;
            float acc0 = 0.f, acc1 = 0.f;
#pragma unroll 4
            for (int i = 0; i < DK; i += 2) {
                acc0 = fmaf(w[i], sm.S[i * NV + j], acc0);
                acc1 = fmaf(w[i + 1], sm.S[(i + 1) * NV + j], acc1);
            }
            sm.X[r * LDX + DK + j] -= acc0 + acc1;
        }
        __syncthreads();

        // ---- stage 6: O = (Gamma . Q) S + P U  ->  o ----
        for (int e = tid; e < C * NV; e += NT) {
            const int r = e / NV, j = e % NV;
            if (r >= L) continue;
            const float* qt = sm.Q + r * DK;
            float acc0 = 0.f, acc1 = 0.f;
#pragma unroll 4
            for (int i = 0; i < DK; i += 2) {
                acc0 = fmaf(qt[i], sm.S[i * NV + j], acc0);
                acc1 = fmaf(qt[i + 1], sm.S[(i + 1) * NV + j], acc1);
            }
            const float* prow = sm.P + r * C;
            for (int s = 0; s <= r; ++s) acc0 = fmaf(prow[s], sm.X[s * LDX + DK + j], acc0);
            store_from_float(go, ((int64_t)(t0 + r) * H + h) * p.dv + j0 + j, p.scale * (acc0 + acc1));
        }

        // ---- stage 7: S = Diag(Gamma_L) S + Khat^T U ----
        constexpr int PER = (DK * NV + NT - 1) / NT;
        float snew[PER];
#pragma unroll
        for (int m = 0; m < PER; ++m) {
            const int e = tid + m * NT;
            if (e < DK * NV) {
                const int i = e / NV, j = e % NV;
                float acc = sm.gamL[i] * sm.S[e];
                for (int s = 0; s < L; ++s) acc = fmaf(sm.K[s * DK + i], sm.X[s * LDX + DK + j], acc);
                snew[m] = acc;
            }
        }
        __syncthreads();
#pragma unroll
        for (int m = 0; m < PER; ++m) {
            const int e = tid + m * NT;
            if (e < DK * NV) sm.S[e] = snew[m];
        }
        if (p.snap_every > 0) {                      // the state after this chunk, if a snapshot is due
            const int64_t slot = snapshot_slot(p, n, t0 + L - t_begin, t_end - t_begin);
            if (slot >= 0) {
                float* dst = p.snapshots + (slot * H + h) * DK * (int64_t)p.dv + j0;
#pragma unroll
                for (int m = 0; m < PER; ++m) {
                    const int e = tid + m * NT;
                    if (e < DK * NV) dst[(int64_t)(e / NV) * p.dv + e % NV] = snew[m];
                }
            }
        }
    }
    __syncthreads();

    // ---- state out ----
    for (int e = tid; e < DK * NV; e += NT) {
        const int i = e / NV, j = e % NV;
        p.state_out[state_off + (int64_t)i * p.dv + j0 + j] = sm.S[e];
    }
}

template <int DK, int NV, typename TIn>
cudaError_t launch_cc(const PrefillParams& p, cudaStream_t s) {
    const size_t smem = sizeof(CcSmem<DK, NV>);
    auto kern = kda_prefill_cc_kernel<DK, NV, TIn>;
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
    const int64_t blocks = (int64_t)p.num_seqs * p.H * p.slices;
    if (blocks <= 0) return cudaSuccess;
    if (blocks > 2147483647LL) return cudaErrorInvalidValue;
    kern<<<(unsigned)blocks, NT, smem, s>>>(p);
    return cudaGetLastError();
}

template <typename TIn>
cudaError_t launch_cc_t(const PrefillParams& p, cudaStream_t s) {
    switch (p.dk) {
        case 16: return launch_cc<16, 16, TIn>(p, s);
        case 64: return launch_cc<64, 32, TIn>(p, s);
        case 128: return launch_cc<128, 32, TIn>(p, s);
        default: return cudaErrorInvalidValue;
    }
}

}  // namespace

int prefill_cc_slices(int dv) { return dv <= 32 ? 1 : dv / 32; }

cudaError_t launch_prefill_cc(const PrefillParams& p, kda_dtype dt, cudaStream_t s) {
    return dt == KDA_DTYPE_BF16 ? launch_cc_t<__nv_bfloat16>(p, s) : launch_cc_t<float>(p, s);
}

__global__ void kda_order_kernel(const int32_t* cu, int32_t n, int32_t* order) {
    const int i = blockIdx.x * blockDim.x + threadIdx.x;
    if (i >= n) return;
    if (n > 4096) {                 // quadratic ranking only for moderate batch counts
        order[i] = i;
        return;
    }
    const int64_t li = (int64_t)cu[i + 1] - cu[i];
    int rank = 0;
    for (int j = 0; j < n; ++j) {
        const int64_t lj = (int64_t)cu[j + 1] - cu[j];
        rank += (lj > li) || (lj == li && j < i);
    }
    order[rank] = i;
}

cudaError_t launch_order(const int32_t* cu_seqlens, int32_t num_seqs, int32_t* order, cudaStream_t s) {
    const int threads = 128;
    const int blocks = (num_seqs + threads - 1) / threads;
    kda_order_kernel<<<blocks, threads, 0, s>>>(cu_seqlens, num_seqs, order);
    return cudaGetLastError();
}

}  // namespace kda
