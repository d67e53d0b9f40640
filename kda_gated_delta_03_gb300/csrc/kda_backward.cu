// Backward pass of the KDA prefill (reverse mode of the recurrence), chunk-parallel.
//
// Forward per head and token ("Kimi K3, explained", section "The math"; S is d_k x d_v, key channel
// i = row, value channel j = column):
//   S' = Diag(alpha_t) S_{t-1},  x = S'^T k_t,  S_t = S' + beta_t k_t (v_t - x)^T,  o_t = scale S_t^T q_t
// Backward, from the last token back, with G the gradient of S_t (later tokens included), u = v_t - x:
//   G += scale q_t do_t^T
//   dq_t = scale S_t do_t;  dbeta_t = k_t^T G u;  du = beta_t G^T k_t;  dv_t = du;  dx = -du
//   dk_t = beta_t G u + S' dx;  G' = G + k_t dx^T;  dalpha_t[i] = sum_j G'[i][j] S_{t-1}[i][j]
//   G <- Diag(alpha_t) G'                                       (the gradient of S_{t-1})
//
// Three passes after the snapshot offsets:
//   1. forward recompute: the library's own prefill writes the state at every 64-token boundary;
//   2. the state-gradient chain (kda_bwd_dstate_kernel): G alone, carried back token by token,
//      G <- Diag(alpha_t) (I - beta_t k_t k_t^T) (G + scale q_t do_t^T), which needs no forward state
//      and splits by value column; it writes G at every 64-token boundary and the gradient of the
//      initial state (for one bf16 d = 128 sequence whose recompute ran as one window, the chain goes
//      chunk by chunk from the recompute's records instead: kda_bwd_dstate_records_kernel);
//   3. the chunk pass: one unit per (sequence, chunk, head), independent of the others given the
//      chunk's start state (a snapshot) and the gradient of its end state (from pass 2).  At d = 128 it
//      runs in matrix form (kda_bwd_chunk_mat_kernel, kda_backward_mat.cu); at d = 16 and 64
//      kda_prefill_bwd_kernel replays the chunk's tokens into a per-CTA scratch (63 states) and walks
//      them back with the per-token rules above.  A thread holds 8 key rows x 4 value columns of S, of G
//      and of S_{t-1}; sums over key rows go through shared memory, sums over value columns through warp
//      shuffles (the LPR threads of a row group are consecutive lanes).

#include "kda_internal.cuh"

namespace kda {
namespace {

// Snapshot offsets of the forward recompute, off[n] = sum over m < n of floor(len_m / 64), and chunk
// offsets, choff[n] = sum over m < n of ceil(len_m / 64) (the chunk units of pass 3).  The workspace
// holds floor(T / 64) boundary slots, enough for any cu_seqlens with 0 <= cu[0] <= ... <= cu[N] <= T;
// any other cu_seqlens sets the error bit and zeroes both arrays, so that nothing is written past the
// slots (the recompute then writes no snapshot, and the chunk pass has no units).
__global__ void kda_bwd_offsets_kernel(const int32_t* cu, int32_t N, int32_t T, int32_t* off, int32_t* choff,
                                       unsigned* err) {
    if (blockIdx.x == 0 && threadIdx.x == 0) {
        bool ok = cu[0] >= 0 && cu[N] <= T;
        for (int n = 0; n < N && ok; ++n) ok = cu[n + 1] >= cu[n];
        int32_t acc = 0, cacc = 0;
        off[0] = 0;
        choff[0] = 0;
        for (int n = 0; n < N; ++n) {
            const int32_t len = ok ? cu[n + 1] - cu[n] : 0;
            acc += len / kChunk;
            cacc += (len + kChunk - 1) / kChunk;
            off[n + 1] = acc;
            choff[n + 1] = cacc;
        }
        if (!ok) atomicOr(err, KDA_DEVERR_CU_SEQLENS);
    }
}

template <int D, int NT>
struct BwdCfg {
    static constexpr int LPR = D / 4;          // float4 column groups per row (= lanes sharing a row group)
    static constexpr int RPP = NT / LPR;       // row groups
    static constexpr int PASSES = D / RPP;     // rows per thread
    static_assert(NT % LPR == 0 && D % RPP == 0 && LPR <= 32 && 32 % LPR == 0, "bad backward tiling");
};

// Reduce-scatter over the consecutive lanes of a row group (xor offsets O, O/2, .., 1): each lane brings
// V partial sums; while the count is even a level halves it (a lane keeps the half its offset bit
// selects and adds its partner's copy of that half), after that a level adds all of them.  Afterwards
// v[0 .. rs_count - 1] of the lane at position c are complete sums of the values rs_base(c) ..
// rs_base(c) + rs_count - 1, replicated over the lanes that differ only in the bits rs_mask().
template <int O, int V>
__device__ __forceinline__ void rs_step(float* v, int c) {
    if constexpr (O >= 1) {
        if constexpr (V % 2 == 0) {
            constexpr int HV = V / 2;
            const bool up = (c & O) != 0;
#pragma unroll
            for (int i = 0; i < HV; ++i) {
                const float send = up ? v[i] : v[HV + i];
                const float keep = up ? v[HV + i] : v[i];
                v[i] = keep + __shfl_xor_sync(0xffffffffu, send, O);
            }
            rs_step<O / 2, HV>(v, c);
        } else {
#pragma unroll
            for (int i = 0; i < V; ++i) v[i] += __shfl_xor_sync(0xffffffffu, v[i], O);
            rs_step<O / 2, V>(v, c);
        }
    }
}
template <int O, int V>
__device__ __forceinline__ int rs_base(int c) {
    if constexpr (O >= 1) {
        if constexpr (V % 2 == 0) return ((c & O) ? V / 2 : 0) + rs_base<O / 2, V / 2>(c);
        else return rs_base<O / 2, V>(c);
    } else {
        return 0;
    }
}
template <int O, int V>
__host__ __device__ constexpr int rs_mask() {
    if constexpr (O >= 1) {
        if constexpr (V % 2 == 0) return rs_mask<O / 2, V / 2>();
        else return O | rs_mask<O / 2, V>();
    } else {
        return 0;
    }
}

__device__ __forceinline__ void cp16(void* dst, const void* src) {
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16;\n" ::"r"((uint32_t)__cvta_generic_to_shared(dst)),
                 "l"(src)
                 : "memory");
}
__device__ __forceinline__ void cp4(void* dst, const void* src) {
    asm volatile("cp.async.ca.shared.global [%0], [%1], 4;\n" ::"r"((uint32_t)__cvta_generic_to_shared(dst)),
                 "l"(src)
                 : "memory");
}
__device__ __forceinline__ void cp_commit() { asm volatile("cp.async.commit_group;\n" ::: "memory"); }
template <int N>
__device__ __forceinline__ void cp_wait() { asm volatile("cp.async.wait_group %0;\n" ::"n"(N) : "memory"); }

// ---- pass 2: the state-gradient chain ----
// One CTA per (sequence, head, slice of SW value columns); lane j of every warp holds column j of the
// slice, warp w key rows RPW w .. RPW w + RPW - 1.  (Eight warps of 16 rows at d = 128 were slower: the
// chain is bound by its per-token barrier and reduction latency, which more warps lengthen.)  The token vectors stream through a ring of NBUF
// slots, NBUF - 1 tokens ahead.
template <int D>
struct DsCfg {
    static constexpr int SW = D < 32 ? D : 32;      // value columns per CTA
    static constexpr int RPW = D < 32 ? D : 32;     // key rows per warp
    static constexpr int NW = D / RPW;              // warps
    static constexpr int NT = 32 * NW;
    static constexpr int SLICES = D / SW;
    static constexpr int NBUF = 8;
};

template <int D, int SW, typename TIn>
struct DsTok {
    TIn q[D], k[D];
    float a[D];
    TIn g[SW];                                      // the slice of the output gradient
    float beta[4];
};

// eight consecutive elements as float
__device__ __forceinline__ void ld8(const float* p, float* o) {
    const float4 a = reinterpret_cast<const float4*>(p)[0], b = reinterpret_cast<const float4*>(p)[1];
    o[0] = a.x; o[1] = a.y; o[2] = a.z; o[3] = a.w; o[4] = b.x; o[5] = b.y; o[6] = b.z; o[7] = b.w;
}
__device__ __forceinline__ void ld8(const __nv_bfloat16* p, float* o) {
    const uint4 w = *reinterpret_cast<const uint4*>(p);
    const uint32_t u[4] = {w.x, w.y, w.z, w.w};
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        o[2 * i] = __uint_as_float(u[i] << 16);
        o[2 * i + 1] = __uint_as_float(u[i] & 0xFFFF0000u);
    }
}

template <int D, typename TIn>
__global__ void __launch_bounds__(DsCfg<D>::NT) kda_bwd_dstate_kernel(BwdParams p) {
    using CF = DsCfg<D>;
    constexpr int SW = CF::SW, RPW = CF::RPW, NW = CF::NW, NT = CF::NT, NBUF = CF::NBUF;
    constexpr int EV = 16 / sizeof(TIn);
    __shared__ __align__(16) DsTok<D, SW, TIn> ring[NBUF];
    __shared__ float red[NW][SW];

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int H = p.H;
    const int slice = blockIdx.x % CF::SLICES, nh = blockIdx.x / CF::SLICES;
    const int h = nh % H, n = nh / H;
    const int32_t tb = p.cu_seqlens[n], te = p.cu_seqlens[n + 1];
    if (tb < 0 || te < tb || te > p.total_tokens) {
        if (tid == 0) atomicOr(p.err, KDA_DEVERR_CU_SEQLENS);
        return;
    }
    const TIn* gq = static_cast<const TIn*>(p.q);
    const TIn* gk = static_cast<const TIn*>(p.k);
    const TIn* gdo = static_cast<const TIn*>(p.d_o);
    const bool col = lane < SW;
    const int j = slice * SW + (col ? lane : 0);
    const int r0 = warp * RPW;
    const int64_t sidx = ((int64_t)n * H + h) * D * D;
    float G[RPW];
#pragma unroll
    for (int x = 0; x < RPW; ++x)
        G[x] = (p.d_state_out && col) ? p.d_state_out[sidx + (int64_t)(r0 + x) * D + j] : 0.f;

    const int len = te - tb;
    auto fetch = [&](int slot, int32_t t) {
        const int64_t row = (int64_t)t * H + h;
        DsTok<D, SW, TIn>& s = ring[slot];
        for (int e = tid; e < D / EV; e += NT) {
            cp16(s.q + e * EV, gq + row * D + e * EV);
            cp16(s.k + e * EV, gk + row * D + e * EV);
        }
        for (int e = tid; e < D / 4; e += NT) cp16(s.a + e * 4, p.alpha + row * D + e * 4);
        for (int e = tid; e < SW / EV; e += NT) cp16(s.g + e * EV, gdo + row * D + slice * SW + e * EV);
        if (tid == 0) cp4(s.beta, p.beta + row);
    };
#pragma unroll 1
    for (int i = 0; i < NBUF - 1; ++i) {
        if (i < len) fetch(i, te - 1 - i);
        cp_commit();
    }
#pragma unroll 1
    for (int i = 0; i < len; ++i) {
        const int32_t t = te - 1 - i;
        cp_wait<NBUF - 2>();
        __syncthreads();                            // token i landed; every thread is past token i - 1
        if (i + NBUF - 1 < len) fetch((i + NBUF - 1) % NBUF, te - NBUF - i);
        cp_commit();
        const DsTok<D, SW, TIn>& s = ring[i % NBUF];
        const float dov = col ? p.scale * to_float(s.g[lane]) : 0.f;
        float pp[4] = {0.f, 0.f, 0.f, 0.f};           // four independent partial sums
        float kv[RPW];                                // k of this warp's rows, kept for the update
#pragma unroll
        for (int x0 = 0; x0 < RPW; x0 += 8) {
            float qv[8];
            ld8(s.q + r0 + x0, qv);
            ld8(s.k + r0 + x0, kv + x0);
#pragma unroll
            for (int x = 0; x < 8; ++x) {
                G[x0 + x] = fmaf(qv[x], dov, G[x0 + x]);
                pp[x & 3] = fmaf(G[x0 + x], kv[x0 + x], pp[x & 3]);
            }
        }
        const float part = (pp[0] + pp[1]) + (pp[2] + pp[3]);
        float w = part;
        if constexpr (NW > 1) {
            if (col) red[warp][lane] = part;
            __syncthreads();
            w = 0.f;
#pragma unroll
            for (int x = 0; x < NW; ++x) w += red[x][col ? lane : 0];
        }
        const float bw = s.beta[0] * w;
#pragma unroll
        for (int x0 = 0; x0 < RPW; x0 += 8) {
            float av[8];
            ld8(s.a + r0 + x0, av);
#pragma unroll
            for (int x = 0; x < 8; ++x) G[x0 + x] = av[x] * fmaf(-kv[x0 + x], bw, G[x0 + x]);
        }
        // after token tb + 64 c (c >= 1), G is the gradient of the state after chunk c - 1
        const int32_t rel = t - tb;
        if (rel > 0 && (rel % kChunk) == 0 && col) {
            float* dst = p.dstate_b + ((int64_t)(p.snap_offsets[n] + rel / kChunk - 1) * H + h) * D * D + j;
#pragma unroll
            for (int x = 0; x < RPW; ++x) dst[(int64_t)(r0 + x) * D] = G[x];
        }
    }
    if (p.d_state_in && col) {
#pragma unroll
        for (int x = 0; x < RPW; ++x) p.d_state_in[sidx + (int64_t)(r0 + x) * D + j] = G[x];
    }
    cp_wait<0>();
}

// Per-token vectors of the chunk, double-buffered in shared memory and fetched one token ahead.
template <int D, typename TIn>
struct TokVec {
    TIn q[D], k[D], v[D], g[D];   // g: the output gradient
    float a[D];
    float beta[4];
};

template <int D, int NT, typename TIn>
__global__ void __launch_bounds__(NT, 1) kda_prefill_bwd_kernel(BwdParams p) {
    using CF = BwdCfg<D, NT>;
    constexpr int LPR = CF::LPR, RPP = CF::RPP, PASSES = CF::PASSES;
    constexpr int EV = 16 / sizeof(TIn);              // elements of TIn per 16-byte copy
    extern __shared__ __align__(16) unsigned char dsm[];
    float* prevbuf = reinterpret_cast<float*>(dsm);   // [2][D * D]: S_{t-1} of the next backward step
    TokVec<D, TIn>* tv = reinterpret_cast<TokVec<D, TIn>*>(dsm + 2 * D * D * 4);
    __shared__ float su[D], sdx[D];
    __shared__ float red0[RPP][D], red1[RPP][D];
    __shared__ float sdb[RPP];

    const int tid = threadIdx.x;
    const int cg = tid % LPR, rg = tid / LPR;
    const int H = p.H;
    const TIn* gq = static_cast<const TIn*>(p.q);
    const TIn* gk = static_cast<const TIn*>(p.k);
    const TIn* gv = static_cast<const TIn*>(p.v);
    const TIn* gdo = static_cast<const TIn*>(p.d_o);
    TIn* gdq = static_cast<TIn*>(p.d_q);
    TIn* gdk = static_cast<TIn*>(p.d_k);
    TIn* gdv = static_cast<TIn*>(p.d_v);
    float* scratch = p.scratch + (int64_t)blockIdx.x * (kChunk - 1) * D * D;
    auto row_of = [&](int m) { return rg + RPP * m; };
    auto ld_state = [&](const float* base, float4* s) {
#pragma unroll
        for (int m = 0; m < PASSES; ++m) s[m] = *reinterpret_cast<const float4*>(base + (int64_t)row_of(m) * D + 4 * cg);
    };
    auto st_state = [&](float* base, const float4* s) {
#pragma unroll
        for (int m = 0; m < PASSES; ++m) *reinterpret_cast<float4*>(base + (int64_t)row_of(m) * D + 4 * cg) = s[m];
    };
    // asynchronous fetches: the vectors of token `row` into buffer b (q and g only when `full`), and a
    // state (each thread its own elements) into prevbuf b
    auto fetch_vec = [&](int b, int64_t row, bool full) {
        TokVec<D, TIn>& t = tv[b];
        for (int e = tid; e < D / EV; e += NT) {
            cp16(t.k + e * EV, gk + row * D + e * EV);
            cp16(t.v + e * EV, gv + row * D + e * EV);
            if (full) {
                cp16(t.q + e * EV, gq + row * D + e * EV);
                cp16(t.g + e * EV, gdo + row * D + e * EV);
            }
        }
        for (int e = tid; e < D / 4; e += NT) cp16(t.a + e * 4, p.alpha + row * D + e * 4);
        if (tid == 0) cp4(t.beta, p.beta + row);
    };
    auto fetch_state = [&](int b, const float* base) {
        float* dst = prevbuf + b * D * D;
#pragma unroll
        for (int m = 0; m < PASSES; ++m) {
            const int64_t off = (int64_t)row_of(m) * D + 4 * cg;
            if (base) cp16(dst + off, base + off);
            else *reinterpret_cast<float4*>(dst + off) = make_float4(0.f, 0.f, 0.f, 0.f);
        }
    };
    auto own_state = [&](int b, float4* s) {          // this thread's elements of prevbuf b
        const float* src = prevbuf + b * D * D;
#pragma unroll
        for (int m = 0; m < PASSES; ++m) s[m] = *reinterpret_cast<const float4*>(src + (int64_t)row_of(m) * D + 4 * cg);
    };
    auto f = [](TIn x) { return to_float(x); };

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
        const int64_t sidx = ((int64_t)n * H + h) * D * D;
        const int nch = (te - tb + kChunk - 1) / kChunk;
        // the gradient of the chunk's end state: grad_state_out for the last chunk, else from pass 2
        float4 g[PASSES];
        const float* gend = c == nch - 1 ? (p.d_state_out ? p.d_state_out + sidx : nullptr)
                                         : p.dstate_b + ((int64_t)(p.snap_offsets[n] + c) * H + h) * D * D;
        if (gend) ld_state(gend, g);
        else
#pragma unroll
            for (int m = 0; m < PASSES; ++m) g[m] = make_float4(0.f, 0.f, 0.f, 0.f);
        {
            const int32_t t0 = tb + c * kChunk;
            const int L = min(kChunk, te - t0);
            // the chunk's start state: the initial state, or the snapshot after chunk c - 1
            const float* start = c == 0 ? (p.state_in ? p.state_in + sidx : nullptr)
                                        : p.snapshots + ((int64_t)(p.snap_offsets[n] + c - 1) * H + h) * D * D;
            float4 s[PASSES];
            if (start) ld_state(start, s);
            else
#pragma unroll
                for (int m = 0; m < PASSES; ++m) s[m] = make_float4(0.f, 0.f, 0.f, 0.f);

            // ---- forward replay of the chunk; states after tokens 0 .. L-2 go to the scratch ----
            __syncthreads();                          // the vector buffers are free
            fetch_vec(0, (int64_t)t0 * H + h, false);
            cp_commit();
            for (int i = 0; i < L; ++i) {
                const int b = i & 1;
                cp_wait<0>();
                __syncthreads();                      // buffer b landed; every thread is past step i - 1 (buffer b ^ 1)
                if (i + 1 < L) fetch_vec(b ^ 1, (int64_t)(t0 + i + 1) * H + h, false);
                cp_commit();
                const TokVec<D, TIn>& t = tv[b];
                float4 px = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
                for (int m = 0; m < PASSES; ++m) {
                    const int r = row_of(m);
                    const float w = t.a[r] * f(t.k[r]);
                    px.x = fmaf(w, s[m].x, px.x); px.y = fmaf(w, s[m].y, px.y);
                    px.z = fmaf(w, s[m].z, px.z); px.w = fmaf(w, s[m].w, px.w);
                }
                reinterpret_cast<float4*>(red0[rg])[cg] = px;
                __syncthreads();
                for (int j = tid; j < D; j += NT) {
                    float x = 0.f;
#pragma unroll
                    for (int r = 0; r < RPP; ++r) x += red0[r][j];
                    su[j] = t.beta[0] * (f(t.v[j]) - x);   // beta (v - x)
                }
                __syncthreads();
                const float4 bu = reinterpret_cast<const float4*>(su)[cg];
#pragma unroll
                for (int m = 0; m < PASSES; ++m) {
                    const int r = row_of(m);
                    const float a = t.a[r], kk = f(t.k[r]);
                    s[m].x = fmaf(kk, bu.x, a * s[m].x); s[m].y = fmaf(kk, bu.y, a * s[m].y);
                    s[m].z = fmaf(kk, bu.z, a * s[m].z); s[m].w = fmaf(kk, bu.w, a * s[m].w);
                }
                if (i < L - 1) st_state(scratch + (int64_t)i * D * D, s);
            }
            __threadfence_block();                    // this thread's scratch stores before its own re-reads
            __syncthreads();

            // ---- backward over the chunk; s holds S_t; the step's S_{t-1} and vectors were fetched ahead ----
            fetch_vec(0, (int64_t)(t0 + L - 1) * H + h, true);
            fetch_state(0, L >= 2 ? scratch + (int64_t)(L - 2) * D * D : start);
            cp_commit();
            for (int i = L - 1, b = 0; i >= 0; --i, b ^= 1) {
                const int64_t row = (int64_t)(t0 + i) * H + h;
                if (i >= 1) {                         // the next step's vectors and S_{t-2}
                    fetch_vec(b ^ 1, row - H, true);
                    fetch_state(b ^ 1, i >= 2 ? scratch + (int64_t)(i - 2) * D * D : start);
                }
                cp_commit();
                cp_wait<1>();
                __syncthreads();
                const TokVec<D, TIn>& t = tv[b];
                float4 prev[PASSES];
                own_state(b, prev);
                const float beta = t.beta[0];
                const float4 dov = make_float4(f(t.g[4 * cg]), f(t.g[4 * cg + 1]), f(t.g[4 * cg + 2]), f(t.g[4 * cg + 3]));
                // G += scale q do^T; dq = scale S_t do; column partials of x = S'^T k and G^T k
                float4 px = make_float4(0.f, 0.f, 0.f, 0.f), pg = px;
                float dqv[PASSES];
#pragma unroll
                for (int m = 0; m < PASSES; ++m) {
                    const int r = row_of(m);
                    const float sqr = p.scale * f(t.q[r]);
                    g[m].x = fmaf(sqr, dov.x, g[m].x); g[m].y = fmaf(sqr, dov.y, g[m].y);
                    g[m].z = fmaf(sqr, dov.z, g[m].z); g[m].w = fmaf(sqr, dov.w, g[m].w);
                    dqv[m] = s[m].x * dov.x + s[m].y * dov.y + s[m].z * dov.z + s[m].w * dov.w;
                    const float kk = f(t.k[r]), ak = t.a[r] * kk;
                    px.x = fmaf(ak, prev[m].x, px.x); px.y = fmaf(ak, prev[m].y, px.y);
                    px.z = fmaf(ak, prev[m].z, px.z); px.w = fmaf(ak, prev[m].w, px.w);
                    pg.x = fmaf(kk, g[m].x, pg.x); pg.y = fmaf(kk, g[m].y, pg.y);
                    pg.z = fmaf(kk, g[m].z, pg.z); pg.w = fmaf(kk, g[m].w, pg.w);
                }
                rs_step<LPR / 2, PASSES>(dqv, cg);
                if ((cg & rs_mask<LPR / 2, PASSES>()) == 0)
                    store_from_float(gdq, row * D + row_of(rs_base<LPR / 2, PASSES>(cg)), p.scale * dqv[0]);
                reinterpret_cast<float4*>(red0[rg])[cg] = px;
                reinterpret_cast<float4*>(red1[rg])[cg] = pg;
                __syncthreads();
                for (int j = tid; j < D; j += NT) {
                    float x = 0.f, gk = 0.f;
#pragma unroll
                    for (int r = 0; r < RPP; ++r) { x += red0[r][j]; gk += red1[r][j]; }
                    const float du = beta * gk;
                    su[j] = f(t.v[j]) - x;            // u
                    sdx[j] = -du;                     // dx
                    store_from_float(gdv, row * D + j, du);
                }
                __syncthreads();
                const float4 u4 = reinterpret_cast<const float4*>(su)[cg];
                const float4 dx4 = reinterpret_cast<const float4*>(sdx)[cg];
                // per row: gu = (G u)_r, sdxr = (S' dx)_r, da = sum_j G'_rj S_{t-1,rj}, interleaved as
                // tv[3 m + 0 .. 2] so that the reduce-scatter leaves all three of one row on one lane
                float tv[3 * PASSES];
#pragma unroll
                for (int m = 0; m < PASSES; ++m) {
                    const int r = row_of(m);
                    const float a = t.a[r], kk = f(t.k[r]);
                    tv[3 * m] = g[m].x * u4.x + g[m].y * u4.y + g[m].z * u4.z + g[m].w * u4.w;
                    tv[3 * m + 1] = a * (prev[m].x * dx4.x + prev[m].y * dx4.y + prev[m].z * dx4.z + prev[m].w * dx4.w);
                    // G' = G + k dx^T; dalpha = row sums of G' (.) S_{t-1}; G <- Diag(alpha) G'
                    float4 gp;
                    gp.x = fmaf(kk, dx4.x, g[m].x); gp.y = fmaf(kk, dx4.y, g[m].y);
                    gp.z = fmaf(kk, dx4.z, g[m].z); gp.w = fmaf(kk, dx4.w, g[m].w);
                    tv[3 * m + 2] = gp.x * prev[m].x + gp.y * prev[m].y + gp.z * prev[m].z + gp.w * prev[m].w;
                    g[m] = make_float4(a * gp.x, a * gp.y, a * gp.z, a * gp.w);
                    s[m] = prev[m];
                }
                rs_step<LPR / 2, 3 * PASSES>(tv, cg);
                constexpr int TMASK = rs_mask<LPR / 2, 3 * PASSES>();
                const int rr = row_of(rs_base<LPR / 2, 3 * PASSES>(cg) / 3);
                float dbp = f(t.k[rr]) * tv[0];               // k_r (G u)_r, summed over this row group's rows
#pragma unroll
                for (int o = LPR / 2; o > TMASK; o >>= 1) dbp += __shfl_xor_sync(0xffffffffu, dbp, o);
                if ((cg & TMASK) == 0) {
                    store_from_float(gdk, row * D + rr, beta * tv[0] + tv[1]);
                    p.d_alpha[row * D + rr] = tv[2];
                }
                if (cg == 0) sdb[rg] = dbp;
                __syncthreads();
                if (tid == 0) {
                    float db = 0.f;
                    for (int r = 0; r < RPP; ++r) db += sdb[r];
                    p.d_beta[row] = db;
                }
            }
        }
        __syncthreads();
    }
    cp_wait<0>();
}

template <int D, int NT, typename TIn>
constexpr int bwd_smem() { return 2 * D * D * 4 + 2 * (int)sizeof(TokVec<D, TIn>); }

template <int D, int NT, typename TIn>
cudaError_t launch_bwd_d(const BwdParams& p, int grid, cudaStream_t s) {
    constexpr int smem = bwd_smem<D, NT, TIn>();
    cudaError_t e = cudaFuncSetAttribute(kda_prefill_bwd_kernel<D, NT, TIn>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         smem);
    if (e != cudaSuccess) return e;
    kda_prefill_bwd_kernel<D, NT, TIn><<<grid, NT, smem, s>>>(p);
    return cudaGetLastError();
}

template <int D, typename TIn>
cudaError_t launch_dstate_d(const BwdParams& p, cudaStream_t s) {
    const int64_t grid = (int64_t)p.num_seqs * p.H * DsCfg<D>::SLICES;
    if (grid <= 0) return cudaSuccess;
    kda_bwd_dstate_kernel<D, TIn><<<(unsigned)grid, DsCfg<D>::NT, 0, s>>>(p);
    return cudaGetLastError();
}

template <typename TIn>
cudaError_t launch_bwd_t(const BwdParams& p, kda_dtype dt, int grid, cudaStream_t s) {
    cudaError_t e = cudaErrorInvalidValue;
    if (p.records) e = launch_bwd_dstate_records(p, dt, p.records, s);   // chunk by chunk from the records
    else switch (p.dk) {
        case 128: e = launch_dstate_d<128, TIn>(p, s); break;
        case 64: e = launch_dstate_d<64, TIn>(p, s); break;
        case 16: e = launch_dstate_d<16, TIn>(p, s); break;
        default: break;
    }
    if (e != cudaSuccess) return e;
    switch (p.dk) {
        case 128: return launch_bwd_chunk_mat(p, dt, grid, s);
        case 64: return launch_bwd_d<64, 256, TIn>(p, grid, s);
        case 16: return launch_bwd_d<16, 32, TIn>(p, grid, s);
        default: return cudaErrorInvalidValue;
    }
}

}  // namespace

cudaError_t launch_bwd_offsets(const int32_t* cu, int32_t N, int32_t T, int32_t* off, int32_t* choff, unsigned* err,
                               cudaStream_t s) {
    kda_bwd_offsets_kernel<<<1, 32, 0, s>>>(cu, N, T, off, choff, err);
    return cudaGetLastError();
}

cudaError_t launch_prefill_bwd(const BwdParams& p, kda_dtype dt, int grid, cudaStream_t s) {
    return dt == KDA_DTYPE_BF16 ? launch_bwd_t<__nv_bfloat16>(p, dt, grid, s) : launch_bwd_t<float>(p, dt, grid, s);
}

}  // namespace kda
