// Fused KDA decode step: one pass over each resident d x d float32 state.
//
// For one token of one head ("Kimi K3, explained", section "How Kimi Delta
// Attention works, step by step": decay, erase, write, read), with the state
// S[i][j] (i = key channel, j = value channel):
//
//   x_j = sum_i alpha_i k_i S_ij           (what the decayed state returns for k)
//   y_j = sum_i alpha_i q_i S_ij           (the query read of the decayed state)
//   delta_j = beta (v_j - x_j)             (the delta-rule correction)
//   S_ij <- alpha_i S_ij + k_i delta_j     (decay + erase + write, in place)
//   o_j = scale (y_j + (q . k) delta_j)    (= scale * S_new^T q)
//
// The state is read from HBM once and written once, as float32 or (kda_decode_step_bf16_state) as
// bf16 (at d = 128 by the streaming kernel of kda_decode_bf16s.cu).  Each CTA owns one (sequence, head) state: a warp reads whole rows with 128-bit
// streaming loads, so every thread holds D*D/NT values in registers across the
// two reductions over the key channels (partial sums in registers, then across
// row groups through shared memory), and writes the updated rows back with
// streaming stores.

#include "kda_internal.cuh"

namespace kda {
namespace {

// float32 state
template <int D, int NT, typename TIn>
__global__ void __launch_bounds__(NT, (D == 128 ? 2 : 4)) kda_decode_kernel(DecodeParams p) {
    constexpr int LPR = D / 4;          // float4 column groups per row
    constexpr int RPP = NT / LPR;       // rows per pass
    constexpr int PASSES = D / RPP;     // passes over the rows
    static_assert(NT % LPR == 0 && D % RPP == 0, "bad decode tiling");

    __shared__ float sq[D], sk[D], sa[D], sdelta[D];
    __shared__ float sx[RPP][D], sy[RPP][D];
    __shared__ float s_qk;

    const int tid = threadIdx.x;
    const int bh = blockIdx.x;
    const int b = bh / p.H;
    const int h = bh - b * p.H;
    const int slot = p.state_idx ? p.state_idx[b] : b;
    if (slot < 0 || slot >= p.num_slots) {
        if (tid == 0) atomicOr(p.err, KDA_DEVERR_STATE_IDX);
        return;
    }
    float* S = static_cast<float*>(p.state) + ((int64_t)slot * p.H + h) * (int64_t)(D * D);
    const int cg = tid % LPR;
    const int rg = tid / LPR;

    // 1. issue every state load of this thread before anything else
    float4 s[PASSES];
#pragma unroll
    for (int m = 0; m < PASSES; ++m)
        s[m] = __ldcs(reinterpret_cast<const float4*>(S + (int64_t)(rg + RPP * m) * D) + cg);

    // 2. stage q, k, alpha of this (sequence, head)
    const int64_t row = (int64_t)b * p.H + h;
    const TIn* q = static_cast<const TIn*>(p.q);
    const TIn* k = static_cast<const TIn*>(p.k);
    for (int i = tid; i < D; i += NT) {
        sq[i] = load_as_float(q, row * D + i);
        sk[i] = load_as_float(k, row * D + i);
        sa[i] = alpha_at(p.alpha, p.alpha_mode, row, D, i);
    }
    __syncthreads();

    // 3. partial reductions over this thread's rows
    float4 px = make_float4(0.f, 0.f, 0.f, 0.f), py = px;
#pragma unroll
    for (int m = 0; m < PASSES; ++m) {
        const int r = rg + RPP * m;
        const float ak = sa[r] * sk[r], aq = sa[r] * sq[r];
        px.x = fmaf(ak, s[m].x, px.x); px.y = fmaf(ak, s[m].y, px.y);
        px.z = fmaf(ak, s[m].z, px.z); px.w = fmaf(ak, s[m].w, px.w);
        py.x = fmaf(aq, s[m].x, py.x); py.y = fmaf(aq, s[m].y, py.y);
        py.z = fmaf(aq, s[m].z, py.z); py.w = fmaf(aq, s[m].w, py.w);
    }
    reinterpret_cast<float4*>(sx[rg])[cg] = px;
    reinterpret_cast<float4*>(sy[rg])[cg] = py;
    if (tid < 32) {
        float acc = 0.f;
        for (int i = tid; i < D; i += 32) acc = fmaf(sq[i], sk[i], acc);
#pragma unroll
        for (int off = 16; off > 0; off >>= 1) acc += __shfl_xor_sync(0xffffffffu, acc, off);
        if (tid == 0) s_qk = acc;
    }
    __syncthreads();

    // 4. finish the reductions per value channel: delta and the output
    const float beta = p.beta[row];
    const TIn* v = static_cast<const TIn*>(p.v);
    TIn* o = static_cast<TIn*>(p.o);
    for (int j = tid; j < D; j += NT) {
        float x = 0.f, y = 0.f;
#pragma unroll
        for (int g = 0; g < RPP; ++g) { x += sx[g][j]; y += sy[g][j]; }
        const float delta = beta * (load_as_float(v, row * D + j) - x);
        sdelta[j] = delta;
        store_from_float(o, row * D + j, p.scale * fmaf(s_qk, delta, y));
    }
    __syncthreads();

    // 5. decay + erase + write, streamed back in place
    const float4 d4 = reinterpret_cast<const float4*>(sdelta)[cg];
#pragma unroll
    for (int m = 0; m < PASSES; ++m) {
        const int r = rg + RPP * m;
        const float a = sa[r], kk = sk[r];
        float4 n;
        n.x = fmaf(kk, d4.x, a * s[m].x);
        n.y = fmaf(kk, d4.y, a * s[m].y);
        n.z = fmaf(kk, d4.z, a * s[m].z);
        n.w = fmaf(kk, d4.w, a * s[m].w);
        __stcs(reinterpret_cast<float4*>(S + (int64_t)r * D) + cg, n);
    }
}

// float32 state at d = 128, split by value columns: the step is independent per value column j (only
// q . k is shared, and each CTA recomputes it), so two CTAs of 256 threads each take 64 columns of one
// state; four CTAs per SM keep more loads and stores in flight than two whole-state CTAs.
template <int D, int CW, int NT, typename TIn>
__global__ void __launch_bounds__(NT, 4) kda_decode_cols_kernel(DecodeParams p) {
    constexpr int LPR = CW / 4;         // float4 column groups per row of the slice
    constexpr int RPP = NT / LPR;       // rows per pass
    constexpr int PASSES = D / RPP;
    constexpr int SPLIT = D / CW;
    static_assert(NT % LPR == 0 && D % RPP == 0 && D % CW == 0, "bad decode tiling");

    __shared__ float sq[D], sk[D], sa[D], sdelta[CW];
    __shared__ float sx[RPP][CW], sy[RPP][CW];
    __shared__ float s_qk;

    const int tid = threadIdx.x;
    const int bh = blockIdx.x / SPLIT, c0 = (blockIdx.x % SPLIT) * CW;
    const int b = bh / p.H;
    const int h = bh - b * p.H;
    const int slot = p.state_idx ? p.state_idx[b] : b;
    if (slot < 0 || slot >= p.num_slots) {
        if (tid == 0) atomicOr(p.err, KDA_DEVERR_STATE_IDX);
        return;
    }
    float* S = static_cast<float*>(p.state) + ((int64_t)slot * p.H + h) * (int64_t)(D * D) + c0;
    const int cg = tid % LPR;
    const int rg = tid / LPR;

    float4 s[PASSES];
#pragma unroll
    for (int m = 0; m < PASSES; ++m)
        s[m] = __ldcs(reinterpret_cast<const float4*>(S + (int64_t)(rg + RPP * m) * D) + cg);

    const int64_t row = (int64_t)b * p.H + h;
    const TIn* q = static_cast<const TIn*>(p.q);
    const TIn* k = static_cast<const TIn*>(p.k);
    for (int i = tid; i < D; i += NT) {
        sq[i] = load_as_float(q, row * D + i);
        sk[i] = load_as_float(k, row * D + i);
        sa[i] = alpha_at(p.alpha, p.alpha_mode, row, D, i);
    }
    __syncthreads();

    float4 px = make_float4(0.f, 0.f, 0.f, 0.f), py = px;
#pragma unroll
    for (int m = 0; m < PASSES; ++m) {
        const int r = rg + RPP * m;
        const float ak = sa[r] * sk[r], aq = sa[r] * sq[r];
        px.x = fmaf(ak, s[m].x, px.x); px.y = fmaf(ak, s[m].y, px.y);
        px.z = fmaf(ak, s[m].z, px.z); px.w = fmaf(ak, s[m].w, px.w);
        py.x = fmaf(aq, s[m].x, py.x); py.y = fmaf(aq, s[m].y, py.y);
        py.z = fmaf(aq, s[m].z, py.z); py.w = fmaf(aq, s[m].w, py.w);
    }
    reinterpret_cast<float4*>(sx[rg])[cg] = px;
    reinterpret_cast<float4*>(sy[rg])[cg] = py;
    if (tid < 32) {
        float acc = 0.f;
        for (int i = tid; i < D; i += 32) acc = fmaf(sq[i], sk[i], acc);
#pragma unroll
        for (int off = 16; off > 0; off >>= 1) acc += __shfl_xor_sync(0xffffffffu, acc, off);
        if (tid == 0) s_qk = acc;
    }
    __syncthreads();

    const float beta = p.beta[row];
    const TIn* v = static_cast<const TIn*>(p.v);
    TIn* o = static_cast<TIn*>(p.o);
    for (int j = tid; j < CW; j += NT) {
        float x = 0.f, y = 0.f;
#pragma unroll
        for (int g = 0; g < RPP; ++g) { x += sx[g][j]; y += sy[g][j]; }
        const float delta = beta * (load_as_float(v, row * D + c0 + j) - x);
        sdelta[j] = delta;
        store_from_float(o, row * D + c0 + j, p.scale * fmaf(s_qk, delta, y));
    }
    __syncthreads();

    const float4 d4 = reinterpret_cast<const float4*>(sdelta)[cg];
#pragma unroll
    for (int m = 0; m < PASSES; ++m) {
        const int r = rg + RPP * m;
        const float a = sa[r], kk = sk[r];
        float4 n;
        n.x = fmaf(kk, d4.x, a * s[m].x);
        n.y = fmaf(kk, d4.y, a * s[m].y);
        n.z = fmaf(kk, d4.z, a * s[m].z);
        n.w = fmaf(kk, d4.w, a * s[m].w);
        __stcs(reinterpret_cast<float4*>(S + (int64_t)r * D) + cg, n);
    }
}

// bf16 state at d = 16 and 64: the same step through a storage adapter.
// State storage: float, or bf16 (read as bf16, updated in fp32, rounded to nearest-even on the way back).
// One 16-byte access holds VEC state elements of a row.
template <typename TS> struct StateIO;
template <> struct StateIO<float> {
    static constexpr int VEC = 4;
    __device__ static void load(const float* p, float* v) {
        const float4 t = __ldcs(reinterpret_cast<const float4*>(p));
        v[0] = t.x; v[1] = t.y; v[2] = t.z; v[3] = t.w;
    }
    __device__ static void store(float* p, const float* v) {
        __stcs(reinterpret_cast<float4*>(p), make_float4(v[0], v[1], v[2], v[3]));
    }
};
template <> struct StateIO<__nv_bfloat16> {
    static constexpr int VEC = 8;
    __device__ static void load(const __nv_bfloat16* p, float* v) {
        const uint4 t = __ldcs(reinterpret_cast<const uint4*>(p));
        const __nv_bfloat162* h = reinterpret_cast<const __nv_bfloat162*>(&t);
#pragma unroll
        for (int i = 0; i < 4; ++i) { v[2 * i] = __low2float(h[i]); v[2 * i + 1] = __high2float(h[i]); }
    }
    __device__ static void store(__nv_bfloat16* p, const float* v) {
        uint4 t;
        __nv_bfloat162* h = reinterpret_cast<__nv_bfloat162*>(&t);
#pragma unroll
        for (int i = 0; i < 4; ++i) h[i] = __floats2bfloat162_rn(v[2 * i], v[2 * i + 1]);
        __stcs(reinterpret_cast<uint4*>(p), t);
    }
};

template <int D, int NT, typename TIn, typename TS>
__global__ void __launch_bounds__(NT, (D == 128 ? 2 : 4)) kda_decode_gen_kernel(DecodeParams p) {
    constexpr int VEC = StateIO<TS>::VEC;
    constexpr int LPR = D / VEC;        // 16-byte column groups per row
    constexpr int RPP = NT / LPR;       // rows per pass
    constexpr int PASSES = D / RPP;     // passes over the rows
    static_assert(NT % LPR == 0 && D % RPP == 0, "bad decode tiling");

    __shared__ float sq[D], sk[D], sa[D], sdelta[D];
    __shared__ float sx[RPP][D], sy[RPP][D];
    __shared__ float s_qk;

    const int tid = threadIdx.x;
    const int bh = blockIdx.x;
    const int b = bh / p.H;
    const int h = bh - b * p.H;
    const int slot = p.state_idx ? p.state_idx[b] : b;
    if (slot < 0 || slot >= p.num_slots) {
        if (tid == 0) atomicOr(p.err, KDA_DEVERR_STATE_IDX);
        return;
    }
    TS* S = static_cast<TS*>(p.state) + ((int64_t)slot * p.H + h) * (int64_t)(D * D);
    const int cg = tid % LPR;
    const int rg = tid / LPR;

    // 1. issue every state load of this thread before anything else
    float s[PASSES][VEC];
#pragma unroll
    for (int m = 0; m < PASSES; ++m) StateIO<TS>::load(S + (int64_t)(rg + RPP * m) * D + cg * VEC, s[m]);

    // 2. stage q, k, alpha of this (sequence, head)
    const int64_t row = (int64_t)b * p.H + h;
    const TIn* q = static_cast<const TIn*>(p.q);
    const TIn* k = static_cast<const TIn*>(p.k);
    for (int i = tid; i < D; i += NT) {
        sq[i] = load_as_float(q, row * D + i);
        sk[i] = load_as_float(k, row * D + i);
        sa[i] = alpha_at(p.alpha, p.alpha_mode, row, D, i);
    }
    __syncthreads();

    // 3. partial reductions over this thread's rows
    float px[VEC], py[VEC];
#pragma unroll
    for (int c = 0; c < VEC; ++c) px[c] = py[c] = 0.f;
#pragma unroll
    for (int m = 0; m < PASSES; ++m) {
        const int r = rg + RPP * m;
        const float ak = sa[r] * sk[r], aq = sa[r] * sq[r];
#pragma unroll
        for (int c = 0; c < VEC; ++c) {
            px[c] = fmaf(ak, s[m][c], px[c]);
            py[c] = fmaf(aq, s[m][c], py[c]);
        }
    }
#pragma unroll
    for (int c = 0; c < VEC; c += 4) {
        reinterpret_cast<float4*>(sx[rg] + cg * VEC)[c / 4] = make_float4(px[c], px[c + 1], px[c + 2], px[c + 3]);
        reinterpret_cast<float4*>(sy[rg] + cg * VEC)[c / 4] = make_float4(py[c], py[c + 1], py[c + 2], py[c + 3]);
    }
    if (tid < 32) {
        float acc = 0.f;
        for (int i = tid; i < D; i += 32) acc = fmaf(sq[i], sk[i], acc);
#pragma unroll
        for (int off = 16; off > 0; off >>= 1) acc += __shfl_xor_sync(0xffffffffu, acc, off);
        if (tid == 0) s_qk = acc;
    }
    __syncthreads();

    // 4. finish the reductions per value channel: delta and the output
    const float beta = p.beta[row];
    const TIn* v = static_cast<const TIn*>(p.v);
    TIn* o = static_cast<TIn*>(p.o);
    for (int j = tid; j < D; j += NT) {
        float x = 0.f, y = 0.f;
#pragma unroll
        for (int g = 0; g < RPP; ++g) { x += sx[g][j]; y += sy[g][j]; }
        const float delta = beta * (load_as_float(v, row * D + j) - x);
        sdelta[j] = delta;
        store_from_float(o, row * D + j, p.scale * fmaf(s_qk, delta, y));
    }
    __syncthreads();

    // 5. decay + erase + write, streamed back in place
    float dl[VEC];
#pragma unroll
    for (int c = 0; c < VEC; ++c) dl[c] = sdelta[cg * VEC + c];
#pragma unroll
    for (int m = 0; m < PASSES; ++m) {
        const int r = rg + RPP * m;
        const float a = sa[r], kk = sk[r];
        float n[VEC];
#pragma unroll
        for (int c = 0; c < VEC; ++c) n[c] = fmaf(kk, dl[c], a * s[m][c]);
        StateIO<TS>::store(S + (int64_t)r * D + cg * VEC, n);
    }
}

template <typename TIn, typename TS>
cudaError_t launch_decode_t(const DecodeParams& p, cudaStream_t s) {
    const unsigned grid = (unsigned)((int64_t)p.B * p.H);
    switch (p.d) {
        case 128:
            if (p.state_bf16) return cudaErrorInvalidValue;   // streamed by launch_decode_bf16s_stream
            kda_decode_cols_kernel<128, 64, 256, TIn><<<2 * grid, 256, 0, s>>>(p);
            break;
        case 64:
            if (p.state_bf16) kda_decode_gen_kernel<64, 64, TIn, TS><<<grid, 64, 0, s>>>(p);
            else kda_decode_kernel<64, 64, TIn><<<grid, 64, 0, s>>>(p);
            break;
        case 16:
            if (p.state_bf16) kda_decode_gen_kernel<16, 32, TIn, TS><<<grid, 32, 0, s>>>(p);
            else kda_decode_kernel<16, 32, TIn><<<grid, 32, 0, s>>>(p);
            break;
        default: return cudaErrorInvalidValue;
    }
    return cudaGetLastError();
}

}  // namespace

cudaError_t launch_decode(const DecodeParams& p, kda_dtype dt, cudaStream_t s) {
    if (p.state_bf16 && p.d == 128) return launch_decode_bf16s_stream(p, dt, s);
    if (p.state_bf16)
        return dt == KDA_DTYPE_BF16 ? launch_decode_t<__nv_bfloat16, __nv_bfloat16>(p, s)
                                    : launch_decode_t<float, __nv_bfloat16>(p, s);
    return dt == KDA_DTYPE_BF16 ? launch_decode_t<__nv_bfloat16, float>(p, s) : launch_decode_t<float, float>(p, s);
}

}  // namespace kda
