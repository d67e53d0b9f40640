// Fused KDA decode step on a bf16-stored state at d = 128, as a persistent streaming kernel.
//
// The arithmetic is the decode step of "Kimi K3, explained" (section "How Kimi Delta Attention works,
// step by step": decay, erase, write, read) on the state S[i][j] (i = key channel, j = value channel):
//
//   x_j = sum_i alpha_i k_i S_ij,  y_j = sum_i alpha_i q_i S_ij,  delta_j = beta (v_j - x_j)
//   S_ij <- alpha_i S_ij + k_i delta_j,  o_j = scale (y_j + (q . k) delta_j)
//
// computed in fp32 from the stored bf16 values and rounded to bf16 once when written back.  A bf16
// state is 32 KiB, so a CTA that loads one state, reduces, then writes it leaves the memory system idle
// through its reductions.  Here two CTAs per SM each loop over their share of the (sequence, head)
// states and keep the next two of them in flight: one thread copies each state (one 32 KiB bulk copy)
// and its token's q, k, v and alpha into a three-stage shared-memory ring, completing on the stage's
// mbarrier, while the CTA works on the current stage.  Updated rows go straight from registers to
// global memory with streaming stores.

#include "kda_tc_util.cuh"

namespace kda {
namespace {

constexpr int SD = 128;                              // key = value dimension
constexpr int SNT = 256;                             // threads: 16 row groups x 16 column groups of 8
constexpr int SSTAGES = 3;
constexpr int ST_BYTES = SD * SD * 2;                // one bf16 state
constexpr int ST_VEC = SD * 4;                       // room for one fp32 vector of SD
constexpr int ST_Q = ST_BYTES, ST_K = ST_Q + ST_VEC, ST_V = ST_K + ST_VEC, ST_A = ST_V + ST_VEC;
constexpr int STAGE_BYTES = ST_A + ST_VEC;
constexpr int OFF_RED = SSTAGES * STAGE_BYTES;       // fp32 partial sums x, y: [8 warps][SD] each
constexpr int OFF_DELTA = OFF_RED + 2 * 8 * SD * 4;  // fp32 delta [SD]
constexpr int OFF_MISC = OFF_DELTA + SD * 4;         // 3 mbarriers, 3 stage slots, 4 q.k partials
constexpr int DS_SMEM = OFF_MISC + 64;
static_assert(STAGE_BYTES % 16 == 0 && OFF_MISC % 8 == 0, "bulk copies need 16-byte offsets");
static_assert(2 * (DS_SMEM + 1024) <= 233472, "two CTAs per SM");

__device__ __forceinline__ void ds_bulk_g2s(uint32_t dst, const void* src, uint32_t bytes, uint32_t mbar) {
    asm volatile("cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];\n" ::"r"(dst),
                 "l"(src), "r"(bytes), "r"(mbar)
                 : "memory");
}
__device__ __forceinline__ void ds_arrive(uint32_t mbar) {
    asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(mbar) : "memory");
}
__device__ __forceinline__ float ds_lo(uint32_t w) { return __uint_as_float(w << 16); }
__device__ __forceinline__ float ds_hi(uint32_t w) { return __uint_as_float(w & 0xFFFF0000u); }
__device__ __forceinline__ float ds_in(const float* p, int i) { return p[i]; }
__device__ __forceinline__ float ds_in(const __nv_bfloat16* p, int i) { return __bfloat162float(p[i]); }

template <typename TIn>
__global__ void __launch_bounds__(SNT, 2) kda_decode_bf16s_stream_kernel(DecodeParams p) {
    extern __shared__ __align__(16) unsigned char sm[];
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int cg = tid & 15, rg = tid >> 4;           // columns 8 cg .. 8 cg + 7; rows rg + 16 m
    const int64_t n_states = (int64_t)p.B * p.H;
    const int n_local = n_states > blockIdx.x ? (int)((n_states - 1 - blockIdx.x) / gridDim.x) + 1 : 0;
    float* sx = reinterpret_cast<float*>(sm + OFF_RED);
    float* sy = sx + 8 * SD;
    float* sdelta = reinterpret_cast<float*>(sm + OFF_DELTA);
    int* sslot = reinterpret_cast<int*>(sm + OFF_MISC + 24);
    float* sqk = reinterpret_cast<float*>(sm + OFF_MISC + 40);
    const uint32_t full = saddr(sm + OFF_MISC);
    const bool per_channel = p.alpha_mode == KDA_ALPHA_PER_CHANNEL;
    const TIn* gq = static_cast<const TIn*>(p.q);
    const TIn* gk = static_cast<const TIn*>(p.k);
    const TIn* gv = static_cast<const TIn*>(p.v);
    TIn* go = static_cast<TIn*>(p.o);
    __nv_bfloat16* gs = static_cast<__nv_bfloat16*>(p.state);

    if (tid == 0) {
        for (int s = 0; s < SSTAGES; ++s)
            asm volatile("mbarrier.init.shared::cta.b64 [%0], 1;" ::"r"(full + 8 * s) : "memory");
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    }
    __syncthreads();

    // thread 0: state i of this CTA (with its token's q, k, v, alpha) into stage i mod SSTAGES; its slot
    // was read one issue earlier, so that the copy is never held up by that load
    auto slot_of = [&](int i) -> int {
        const int b = (int)((blockIdx.x + (int64_t)i * gridDim.x) / p.H);
        return p.state_idx ? __ldg(p.state_idx + b) : b;
    };
    auto issue = [&](int i, int slot) {
        const int64_t st = blockIdx.x + (int64_t)i * gridDim.x;
        const int s = i % SSTAGES;
        const uint32_t bar = full + 8 * s;
        if (slot < 0 || slot >= p.num_slots) {
            atomicOr(p.err, KDA_DEVERR_STATE_IDX);
            sslot[s] = -1;
            ds_arrive(bar);                               // completes the phase with nothing copied
            return;
        }
        sslot[s] = slot;
        const uint32_t dst = saddr(sm + s * STAGE_BYTES);
        constexpr uint32_t vb = SD * sizeof(TIn);
        asm volatile("fence.proxy.async.shared::cta;" ::: "memory");   // the stage's earlier reads come first
        mbar_expect_tx(bar, ST_BYTES + 3 * vb + (per_channel ? SD * 4 : 0));
        ds_bulk_g2s(dst, gs + ((int64_t)slot * p.H + (int)(st % p.H)) * (SD * SD), ST_BYTES, bar);
        ds_bulk_g2s(dst + ST_Q, gq + st * SD, vb, bar);
        ds_bulk_g2s(dst + ST_K, gk + st * SD, vb, bar);
        ds_bulk_g2s(dst + ST_V, gv + st * SD, vb, bar);
        if (per_channel) ds_bulk_g2s(dst + ST_A, p.alpha + st * SD, SD * 4, bar);
    };
    int issued = 0, slot_next = 0;
    if (tid == 0) {
        for (; issued < SSTAGES - 1 && issued < n_local; ++issued) issue(issued, slot_of(issued));
        if (issued < n_local) slot_next = slot_of(issued);
    }
    // beta (and a per-head alpha) of the current state, read one state ahead
    float beta_next = 0.f, ahead_next = 1.f;
    if (n_local > 0) {
        if (tid < SD) beta_next = p.beta[blockIdx.x];
        if (!per_channel) ahead_next = alpha_at(p.alpha, p.alpha_mode, blockIdx.x, SD, 0);
    }

    int i = 0;
    for (; i < n_local; ++i) {
        if (tid == 0 && issued < n_local) {                      // into the stage read by state i - 1
            issue(issued, slot_next);
            if (++issued < n_local) slot_next = slot_of(issued);
        }
        const int64_t st = blockIdx.x + (int64_t)i * gridDim.x;
        const int s = i % SSTAGES;
        const float beta = beta_next, ahead = ahead_next;
        if (i + 1 < n_local) {
            if (tid < SD) beta_next = p.beta[st + gridDim.x];
            if (!per_channel) ahead_next = alpha_at(p.alpha, p.alpha_mode, st + gridDim.x, SD, 0);
        }
        bool ok = mbar_wait(full + 8 * s, (uint32_t)(i / SSTAGES) & 1u);
        const int slot = sslot[s];
        const unsigned char* sb = sm + s * STAGE_BYTES;
        const TIn* sq = reinterpret_cast<const TIn*>(sb + ST_Q);
        const TIn* sk = reinterpret_cast<const TIn*>(sb + ST_K);
        const float* sa = reinterpret_cast<const float*>(sb + ST_A);

        uint4 w[8];
        float ka[8], aa[8];
        if (ok && slot >= 0) {
            float px[8], py[8];
#pragma unroll
            for (int c = 0; c < 8; ++c) px[c] = py[c] = 0.f;
#pragma unroll
            for (int m = 0; m < 8; ++m) {
                const int r = rg + 16 * m;
                w[m] = *reinterpret_cast<const uint4*>(sb + r * (SD * 2) + cg * 16);
                const float a = per_channel ? sa[r] : ahead, kr = ds_in(sk, r);
                ka[m] = kr;
                aa[m] = a;
                const float ak = a * kr, aq = a * ds_in(sq, r);
                const uint32_t u[4] = {w[m].x, w[m].y, w[m].z, w[m].w};
#pragma unroll
                for (int c = 0; c < 4; ++c) {
                    const float lo = ds_lo(u[c]), hi = ds_hi(u[c]);
                    px[2 * c] = fmaf(ak, lo, px[2 * c]);
                    px[2 * c + 1] = fmaf(ak, hi, px[2 * c + 1]);
                    py[2 * c] = fmaf(aq, lo, py[2 * c]);
                    py[2 * c + 1] = fmaf(aq, hi, py[2 * c + 1]);
                }
            }
#pragma unroll
            for (int c = 0; c < 8; ++c) {                 // lanes l and l + 16: the same columns, rows 16 apart
                px[c] += __shfl_xor_sync(0xffffffffu, px[c], 16);
                py[c] += __shfl_xor_sync(0xffffffffu, py[c], 16);
            }
            if (lane < 16) {
                float4* dx = reinterpret_cast<float4*>(sx + warp * SD + cg * 8);
                float4* dy = reinterpret_cast<float4*>(sy + warp * SD + cg * 8);
                dx[0] = make_float4(px[0], px[1], px[2], px[3]);
                dx[1] = make_float4(px[4], px[5], px[6], px[7]);
                dy[0] = make_float4(py[0], py[1], py[2], py[3]);
                dy[1] = make_float4(py[4], py[5], py[6], py[7]);
            }
            if (warp < 4) {
                float qk = ds_in(sq, tid) * ds_in(sk, tid);
#pragma unroll
                for (int off = 16; off > 0; off >>= 1) qk += __shfl_xor_sync(0xffffffffu, qk, off);
                if (lane == 0) sqk[warp] = qk;
            }
        }
        if (!__syncthreads_and(ok)) break;
        if (slot >= 0 && tid < SD) {
            float x = 0.f, y = 0.f;
#pragma unroll
            for (int g = 0; g < 8; ++g) {
                x += sx[g * SD + tid];
                y += sy[g * SD + tid];
            }
            const float qk = (sqk[0] + sqk[1]) + (sqk[2] + sqk[3]);
            const float delta = beta * (ds_in(reinterpret_cast<const TIn*>(sb + ST_V), tid) - x);
            sdelta[tid] = delta;
            store_from_float(go, st * SD + tid, p.scale * fmaf(qk, delta, y));
        }
        __syncthreads();
        if (slot >= 0) {
            float dl[8];
#pragma unroll
            for (int c = 0; c < 8; ++c) dl[c] = sdelta[cg * 8 + c];
            __nv_bfloat16* S = gs + ((int64_t)slot * p.H + (int)(st % p.H)) * (SD * SD);
#pragma unroll
            for (int m = 0; m < 8; ++m) {
                const int r = rg + 16 * m;
                const uint32_t u[4] = {w[m].x, w[m].y, w[m].z, w[m].w};
                uint32_t n[4];
#pragma unroll
                for (int c = 0; c < 4; ++c) {
                    const __nv_bfloat162 t = __floats2bfloat162_rn(fmaf(ka[m], dl[2 * c], aa[m] * ds_lo(u[c])),
                                                                   fmaf(ka[m], dl[2 * c + 1], aa[m] * ds_hi(u[c])));
                    n[c] = *reinterpret_cast<const uint32_t*>(&t);
                }
                __stcs(reinterpret_cast<uint4*>(S + r * SD) + cg, make_uint4(n[0], n[1], n[2], n[3]));
            }
        }
    }
    if (i < n_local && tid == 0) {
        // a stage wait ran out: record it and let every copy still in flight land before the CTA exits
        atomicOr(p.err, KDA_DEVERR_TIMEOUT);
        for (int j = i; j < issued; ++j) mbar_wait(full + 8 * (j % SSTAGES), (uint32_t)(j / SSTAGES) & 1u);
    }
}

}  // namespace

cudaError_t launch_decode_bf16s_stream(const DecodeParams& p, kda_dtype dt, cudaStream_t s) {
    int dev = 0, sms = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if ((e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev)) != cudaSuccess) return e;
    const int64_t n_states = (int64_t)p.B * p.H;
    const unsigned grid = (unsigned)(n_states < 2 * sms ? n_states : 2 * sms);
    if (grid == 0) return cudaSuccess;
    if (dt == KDA_DTYPE_BF16) {
        if ((e = cudaFuncSetAttribute(kda_decode_bf16s_stream_kernel<__nv_bfloat16>,
                                      cudaFuncAttributeMaxDynamicSharedMemorySize, DS_SMEM)) != cudaSuccess)
            return e;
        kda_decode_bf16s_stream_kernel<__nv_bfloat16><<<grid, SNT, DS_SMEM, s>>>(p);
    } else {
        if ((e = cudaFuncSetAttribute(kda_decode_bf16s_stream_kernel<float>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                      DS_SMEM)) != cudaSuccess)
            return e;
        kda_decode_bf16s_stream_kernel<float><<<grid, SNT, DS_SMEM, s>>>(p);
    }
    return cudaGetLastError();
}

}  // namespace kda
