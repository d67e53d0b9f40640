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
// The state is read from HBM once and written once.  Each CTA owns one
// (sequence, head) state: a warp reads whole 512-byte rows with 128-bit
// streaming loads, so every thread holds D*D/NT floats in registers across the
// two reductions over the key channels (partial sums in registers, then across
// row groups through shared memory), and writes the updated rows back with
// streaming stores.

#include "kda_internal.cuh"

namespace kda {
namespace {

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
    float* S = p.state + ((int64_t)slot * p.H + h) * (int64_t)(D * D);
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
        sa[i] = p.alpha[row * D + i];
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

template <typename TIn>
cudaError_t launch_decode_t(const DecodeParams& p, cudaStream_t s) {
    const unsigned grid = (unsigned)((int64_t)p.B * p.H);
    switch (p.d) {
        case 128: kda_decode_kernel<128, 256, TIn><<<grid, 256, 0, s>>>(p); break;
        case 64: kda_decode_kernel<64, 64, TIn><<<grid, 64, 0, s>>>(p); break;
        case 16: kda_decode_kernel<16, 32, TIn><<<grid, 32, 0, s>>>(p); break;
        default: return cudaErrorInvalidValue;
    }
    return cudaGetLastError();
}

}  // namespace

cudaError_t launch_decode(const DecodeParams& p, kda_dtype dt, cudaStream_t s) {
    return dt == KDA_DTYPE_BF16 ? launch_decode_t<__nv_bfloat16>(p, s) : launch_decode_t<float>(p, s);
}

}  // namespace kda
