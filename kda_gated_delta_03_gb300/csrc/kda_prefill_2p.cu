// Two-phase chunkwise prefill: bf16 q/k/v, d_k = d_v = 128, one sequence or several.
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
// operand.  Phase 2 walks the chunks in order, one CTA per (head, NV value columns: 32, or 16 for one
// sequence with few heads), bulk-loading each record one chunk ahead; per chunk it issues a single batch
// of tensor-core products,
//
//   M S (M=128)  and  Q' S (M=64)       tcgen05 kind::f16 (fp16 record and state operands), N=NV, K=128
//
// followed by the fp32 update S <- Gamma_C . S + B - M S and o = scale (Q' S + P Utilde).  Folding W
// into M and Q' doubles phase 1's work on W but leaves one round trip through the tensor core on the
// sequential path instead of two, and no U tile to build between them.
//
// Long sequences are processed in windows of chunks so that the workspace stays bounded; the state
// passes between windows through state_out.  Several sequences number their chunks one after the other
// (chunk offsets computed on the device from cu_seqlens), phase 1 runs over every chunk of the window
// whatever its sequence, and phase 2 runs one CTA per (sequence, head, slice), longest sequences first.
// Every wait is bounded (KDA_DEVERR_TIMEOUT on expiry).

#include "kda_tc_util.cuh"

namespace kda {
namespace {

// ---- one (head, chunk) record in the workspace ----
constexpr int REC_QM = 0;          // [Q'; M]: 192 x 128 fp16 K-major operand (48 KiB)
constexpr int REC_B = 49152;       // B = Khat^T Utilde: fp16 [32 column quads][128 rows][4] (32 KiB)
constexpr int REC_O = 81920;       // P Utilde: fp16 [32 column quads][64 rows][4] (16 KiB)
constexpr int REC_G = 98304;       // Gamma_C: fp32 [128]
constexpr int REC_E = 98816;       // e_c: int32, B and P Utilde are stored divided by 2^e_c
constexpr int REC_BYTES = 99072;   // padded to 256 bytes, so that every record's stores and loads stay sector-aligned
constexpr int QM_BYTES = (C + DK) * DK * 2;
// Q', M, B, P Utilde and the chain's state operand are fp16: the same 10-bit significand as TF32, in half
// the bytes, for values within fp16's range, which the kernels check (KDA_DEVERR_RANGE)
constexpr float kF16Max = 65504.f;
// Magnitudes are kept inside that range by powers of two.  A chunk whose largest |v| is at least 2^6 stores
// its value-side products (Utilde, B, P Utilde) divided by 2^e_c, e_c = the exponent of that largest |v|.
// The chain carries its state divided by 2^E: E is chosen before each chunk's state operand is written,
// as the larger of the chunk's e_c and the exponent of the largest |state| at the previous chunk (all
// state warps' maxima, exchanged in shared memory off the sequential path), so that neither large values
// nor large states leave fp16's range, and a state that shrinks again returns to a small E.  Key-side
// products (Q', M, T') stay O(1) for unit-norm keys and are still checked.  Powers of two are exact: with
// every |v| and |state| below 2^6 nothing is scaled.
constexpr uint32_t kScaleFromBf16 = 0x4280u;   // bf16 bits of 2^6
constexpr int kScaleFromExp = 6;

// 2^n as a float for n in [-126, 127] (exact)
__device__ __forceinline__ float exp2i(int n) { return __int_as_float((n + 127) << 23); }
// the scale exponent of a magnitude given as bf16 bits (0 below 2^8, at most 126)
__device__ __forceinline__ int scale_exp_bf16(uint32_t mag_bits) {
    return mag_bits >= kScaleFromBf16 ? min((int)((mag_bits >> 7) & 0xFFu) - 127, 126) : 0;
}
// the same for a magnitude given as fp32 bits
__device__ __forceinline__ int scale_exp_f32(uint32_t mag_bits) {
    return mag_bits >= (kScaleFromBf16 << 16) ? min((int)((mag_bits >> 23) & 0xFFu) - 127, 126) : 0;
}
// the same for a magnitude given as fp32 bits of the value divided by 2^E
__device__ __forceinline__ int scale_exp_f32_at(uint32_t mag_bits, int E) {
    if (mag_bits < 0x00800000u) return 0;          // zero or denormal: far below 2^6 for any E <= 126
    const int e = (int)((mag_bits >> 23) & 0xFFu) - 127 + E;
    return e >= kScaleFromExp ? min(e, 126) : 0;
}
constexpr int SNV = 32;            // value columns per chain CTA
constexpr int kPrefetchAhead = 4;  // chunks between the chain's L2 prefetch of a record's B and its use
constexpr int SLICES = DK / SNV;
constexpr size_t kBufBudget = size_t(128) << 20;      // record bytes per buffer of the overlapped schedule
                                                      // (about 170 chunks at H = 8: short enough that the
                                                      // first window's phase 1, which nothing overlaps, is
                                                      // short; long enough to amortise the launches)
constexpr size_t kOneWindowBudget = size_t(1) << 30;  // record bytes of the recommended workspace, one sequence
constexpr size_t kMultiWindowBudget = size_t(16) << 30;  // the same for several sequences: with one window every
                                                         // chain CTA has chunks (with 1 GiB windows most CTAs of
                                                         // each window's chain found none and exited: varlen_64
                                                         // took 14.5 instead of 13.5 ms)
static_assert(QM_BYTES == REC_B && REC_B + DK * DK * 2 == REC_O && REC_O + C * DK * 2 == REC_G, "record layout");
static_assert(REC_B % 16 == 0 && REC_O % 16 == 0 && REC_G % 16 == 0 && (REC_BYTES - REC_G) % 16 == 0 &&
                  REC_BYTES % 256 == 0 && (SNV / 4) * C * 8 % 16 == 0,
              "bulk copies and L2 prefetches of record pieces: 16-byte aligned, multiples of 16 bytes");

// ---- phase 1 shared memory ----
constexpr int P_OFF_V = OFF_V;                     // v tile, dense 64 x 128 bf16
constexpr int P_OFF_BETA = OFF_V + C * DK * 2;     // 81920
constexpr int P_OFF_MISC = P_OFF_BETA + 256;
constexpr int P_OFF_ASC = P_OFF_MISC + 64 + DK * 4;         // per-head alpha of the unit's rows (256 B)
constexpr int P_OFF_VMX = P_OFF_ASC + 256;                  // per-warp largest |v| of the unit (8 x u32)
constexpr int P_OFF_S = align1k(P_OFF_VMX + 32);            // scratch, 144 KiB
// scratch sub-regions (offsets from P_OFF_S)
constexpr int PS_A = 0, PS_T = C * AT_LD * 4, PS_SCR = 2 * C * AT_LD * 4;   // solve tiles
constexpr int PS_OPT = 38912, PS_KV = PS_OPT + 16384;                     // T' and [Gamma.K | V]^T (N = 256)
constexpr int PS_P = 122880;                                               // P operand
constexpr int PS_WU = 0, PS_KH = 65536;                                    // fold operands, after [W | Utilde]
constexpr int ONE_L_OFF = C * DK * 4;                                     // one-reference A/P: R, then L
constexpr float kOneRefMax = 125.f;                                        // log2 of the largest factor
constexpr int P_OFF_CS = P_OFF_S + G1_BYTES;               // several sequences: chunk offsets and cu_seqlens
constexpr int CS_MAX = 128;                                 // (N + 1 <= CS_MAX entries each) cached for the lookups
constexpr int P_SMEM = P_OFF_CS + 2 * CS_MAX * 4;
static_assert(PS_KV + (DK + DK) * 256 <= PS_P && PS_P + 16384 <= G1_BYTES, "phase-1 scratch");
static_assert(PS_KH + DK * C * 4 <= PS_P, "phase-1 fold operands");
static_assert(P_SMEM <= 232448, "phase-1 shared memory");

// ---- phase 2 shared memory and threads ----
constexpr int SOP_BYTES = SNV * DK * 2;            // S^T operand: fp16 NV x 128 (NV <= 32), 128-byte swizzle
constexpr int C_OFF_S = 2 * QM_BYTES;              // two record buffers, then two S^T operands
constexpr int C_OFF_MISC = C_OFF_S + 2 * SOP_BYTES;
// misc: 0 lbar[2], 16 dbar[2], 32 obar[2], 48 sbar, 64 ofree[2], 96 TMEM address, 100 abort flag,
// 104 test barrier, 128 per-warp largest |state_in| (8 x u32), 160 ebar[4], 192 E of chunk c (ring of 4),
// 208 per-warp largest |S_c| / 2^E at the operand of chunk c (2 x 8 x u32)
constexpr int CM_SMX0 = 128, CM_EBAR = 160, CM_ERING = 192, CM_SLOT = 208;
constexpr int C_SMEM = C_OFF_MISC + 272;
constexpr int C_NT = NT + 6 * 32;                  // 8 state warps, the MMA-issue warp, the record-loader warp,
                                                   // 4 output warps (one per TMEM lane quadrant)
static_assert(C_OFF_S % 1024 == 0 && C_SMEM <= 232448, "phase-2 shared memory");

struct PrepMaps {
    CUtensorMap k, q, a, v;   // v with a 128-column box
};

__device__ __forceinline__ void bulk_g2s(uint32_t dst, const void* src, uint32_t bytes, uint32_t mbar) {
    asm volatile("cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];\n" ::"r"(dst),
                 "l"(src), "r"(bytes), "r"(mbar)
                 : "memory");
}

// an L2 prefetch of global bytes (16-byte aligned, a multiple of 16 bytes); nothing to wait for
__device__ __forceinline__ void prefetch_l2(const void* src, uint32_t bytes) {
    asm volatile("cp.async.bulk.prefetch.L2.global [%0], %1;" ::"l"(src), "r"(bytes) : "memory");
}

// mbar_wait for a waiter off the critical path: it sleeps between polls, leaving issue slots to the warps
// that share its scheduler (bounded like mbar_wait)
__device__ __forceinline__ bool mbar_wait_lazy(uint32_t mbar, uint32_t parity) {
    const long long t0 = clock64();
    while (true) {
        uint32_t done;
        asm volatile("{\n.reg .pred p;\nmbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\nselp.u32 %0, 1, 0, p;\n}\n"
                     : "=r"(done)
                     : "r"(mbar), "r"(parity)
                     : "memory");
        if (done) return true;
        if (clock64() - t0 > kWaitLimit) return false;
        __nanosleep(200);
    }
}

// fp32 -> TF32 for the A/P factors: rounded to nearest with ties away from zero by adding half a TF32 ulp
// to the magnitude bits and dropping the low 13, on the integer ALUs.  The factor build is bound by the
// special-function pipe (two exponentials per element), which the conversion instruction also uses: this
// form took 1.5% off phase 1 (and was slower than that instruction where nothing else loads the pipe).
// Finite inputs round exactly as that instruction does; a NaN may come out as another NaN or as -0, but a
// NaN in k or q reaches the outputs anyway through the other operands built from them.
__device__ __forceinline__ float tf32_rna(float x) {
    return __uint_as_float((__float_as_uint(x) + 0x1000u) & 0xFFFFE000u);
}

__device__ __forceinline__ void mbar_arrive(uint32_t mbar) {
    asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(mbar) : "memory");
}

__device__ __forceinline__ uint32_t pack_half2(float a, float b) {
    const __half2 h = __floats2half2_rn(a, b);
    return *reinterpret_cast<const uint32_t*>(&h);
}

__device__ __forceinline__ float4 half4_to_float4(uint2 w) {
    const float2 a = __half22float2(*reinterpret_cast<const __half2*>(&w.x));
    const float2 b = __half22float2(*reinterpret_cast<const __half2*>(&w.y));
    return make_float4(a.x, a.y, b.x, b.y);
}

__device__ __forceinline__ bool valid_single_sequence(const PrefillParams& p) {
    return p.num_seqs == 1 && p.cu_seqlens[0] == 0 && p.cu_seqlens[1] == p.total_tokens;
}

// Chunks of all sequences are numbered sequence by sequence: sequence n owns chunks [choff[n], choff[n+1])
// (choff from kda_chunk_offsets_kernel; nullptr for one sequence, whose chunks are simply t / 64).
// The sequence that owns chunk gc (the last n with choff[n] <= gc, which skips empty sequences).
__device__ __forceinline__ int chunk_seq(const int32_t* choff, int32_t N, int64_t gc) {
    int lo = 0, hi = N;
    while (hi - lo > 1) {
        const int mid = (lo + hi) >> 1;
        if (choff[mid] <= gc) lo = mid; else hi = mid;
    }
    return lo;
}
// First token of chunk gc and the end token of its sequence.
__device__ __forceinline__ void chunk_span(const PrefillParams& p, const int32_t* choff, int64_t gc, int32_t& t0,
                                           int32_t& t_end, const int32_t* cu = nullptr) {
    if (!choff) {
        t0 = (int32_t)(gc * C);
        t_end = p.total_tokens;
        return;
    }
    if (!cu) cu = p.cu_seqlens;
    const int n = chunk_seq(choff, p.num_seqs, gc);
    t0 = cu[n] + (int32_t)(gc - choff[n]) * C;
    t_end = cu[n + 1];
}

// Chunk offsets of the sequences (chunks of 64 tokens, the last one partial) and the check of cu_seqlens;
// with an inconsistent cu_seqlens every sequence counts as empty (nothing is computed, KDA_DEVERR_CU_SEQLENS).
__global__ void kda_chunk_offsets_kernel(const int32_t* cu, int32_t N, int32_t T, int32_t* choff, unsigned* err) {
    if (blockIdx.x != 0 || threadIdx.x != 0) return;
    bool ok = cu[0] == 0 && cu[N] == T;
    for (int n = 0; n < N && ok; ++n) ok = cu[n + 1] >= cu[n];
    int32_t acc = 0;
    choff[0] = 0;
    for (int n = 0; n < N; ++n) {
        acc += ok ? (cu[n + 1] - cu[n] + C - 1) / C : 0;
        choff[n + 1] = acc;
    }
    if (!ok) atomicOr(err, KDA_DEVERR_CU_SEQLENS);
}

// ============================================================================================
// Phase 1: persistent CTAs over the units (chunk-major: unit = window chunk * H + head) of the window
// starting at chunk c_begin.  The raw tiles of a CTA's next unit are loaded while it stores the
// current unit's record.
// ============================================================================================
// MULTI: several sequences (chunk offsets in choff); otherwise one sequence, whose chunk arithmetic is then
// compiled without the lookups.
template <bool MULTI>
__global__ void __launch_bounds__(NT, 1)
    kda_prefill_prep_kernel(PrefillParams p, const __grid_constant__ PrepMaps maps, unsigned char* records,
                            int c_begin, int n_units, const int32_t* choff_arg) {
    // the chain kernel after this one may be scheduled at once: its CTAs take SMs as this kernel's leave
    // (neither fits beside the other) and wait for its completion before reading a record
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
    const int32_t* choff = MULTI ? choff_arg : nullptr;
    const int32_t* cu = nullptr;                     // cu_seqlens for the chunk lookups (global unless cached)
    extern __shared__ __align__(1024) unsigned char sm[];
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int gid = lane >> 2, tig = lane & 3;
    const int quad = warp & 3, half = warp >> 2;
    const int ch = tid & (DK - 1), rh = tid >> 7;
    const int H = p.H;
    if (!choff && !valid_single_sequence(p)) {
        if (tid == 0) atomicOr(p.err, KDA_DEVERR_CU_SEQLENS);
        return;
    }
    if (saddr(sm) & 1023u) {
        if (tid == 0) atomicOr(p.err, KDA_DEVERR_TIMEOUT);
        return;
    }
    {                                                // units that exist: chunks [c_begin, all chunks) x heads
        const int64_t nc = choff ? (int64_t)choff[p.num_seqs] : ((int64_t)p.total_tokens + C - 1) / C;
        const int64_t have = (nc - c_begin) * H;
        if (have < n_units) n_units = have < 0 ? 0 : (int)have;
    }

    const __nv_bfloat16* vraw = reinterpret_cast<const __nv_bfloat16*>(sm + P_OFF_V);
    float* sbeta = reinterpret_cast<float*>(sm + P_OFF_BETA);
    float* sgam = reinterpret_cast<float*>(sm + P_OFF_MISC + 64);
    float* sasc = reinterpret_cast<float*>(sm + P_OFF_ASC);  // per-head alpha of the unit's token rows
    unsigned char* X = sm + P_OFF_S;
    volatile int* s_abort = reinterpret_cast<volatile int*>(sm + P_OFF_MISC + 12);
    uint32_t* s_tmem = reinterpret_cast<uint32_t*>(sm + P_OFF_MISC + 8);
    // lbar: the q and alpha tiles; vkbar: the v and k tiles, which are fetched earlier (v once step 3 has
    // read this unit's v, k once step 5 has read its k)
    const uint32_t mbar = saddr(sm + P_OFF_MISC), lbar = saddr(sm + P_OFF_MISC + 16);
    const uint32_t vkbar = saddr(sm + P_OFF_MISC + 24);
    auto Gat = [&](int r, int i) -> float& { return *reinterpret_cast<float*>(sm + OFF_G + g_off(r, i)); };
    auto kat = [&](int r, int i) { return bf(reinterpret_cast<const __nv_bfloat16*>(sm + OFF_K + kq_off(r, i))); };

    if (tid == 0) {
        asm volatile("mbarrier.init.shared::cta.b64 [%0], 1;" ::"r"(mbar) : "memory");
        asm volatile("mbarrier.init.shared::cta.b64 [%0], 1;" ::"r"(lbar) : "memory");
        asm volatile("mbarrier.init.shared::cta.b64 [%0], 1;" ::"r"(vkbar) : "memory");
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
        *s_abort = 0;
    }
    if (MULTI && p.num_seqs + 1 <= CS_MAX) {         // the lookups of every unit read shared memory
        int32_t* cs = reinterpret_cast<int32_t*>(sm + P_OFF_CS);
        for (int e = tid; e <= p.num_seqs; e += NT) {
            cs[e] = choff_arg[e];
            cs[CS_MAX + e] = p.cu_seqlens[e];
        }
        choff = cs;
        cu = cs + CS_MAX;
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
    // TMEM columns: [M | B] of step 6 at 0..255 and [P W | P Utilde] at 256..511; the A/P and [W | Utilde]^T
    // products of steps 2 and 4 use 256..383, so that a unit's M, B and P Utilde can stay in TMEM and drain
    // to its record while the next unit runs its steps 1-5
    constexpr uint32_t TM_W = 2 * DK;
    const int mi = 32 * quad + lane;                         // M=128 accumulator row of this thread
    const int mr = 16 * quad + lane;                         // M=64 accumulator row (lanes < 16)
    unsigned char* rec_prev = nullptr;                       // record whose M, B, P Utilde are still in TMEM
    uint32_t phase = 0;

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
    // several sequences: the span of this CTA's next unit, found once per unit (with its beta) and kept in
    // shared memory for that unit's tile fetches and its own start
    int32_t* s_span = reinterpret_cast<int32_t*>(sm + P_OFF_MISC + 48);
    int span_unit = -1;                               // the unit s_span holds (block-uniform)
    // raw tiles of unit u by TMA (v with one 128-column box), in three groups
    auto unit_rows = [&](int u, int& hu, int32_t& tu) {
        hu = u % H;
        if (MULTI && u == span_unit) {
            tu = s_span[0];
        } else {
            int32_t te;
            chunk_span(p, choff, (int64_t)c_begin + u / H, tu, te, cu);
        }
    };
    auto issue_v = [&](int u) {                      // arms vkbar for v and k together
        if (tid == 32) {
            int hu; int32_t tu;
            unit_rows(u, hu, tu);
            mbar_expect_tx(vkbar, 16384 + C * DK * 2);
            tma_load_3d(saddr(sm + P_OFF_V), &maps.v, 0, hu, tu, vkbar);
        }
    };
    auto issue_k = [&](int u) {
        if (tid == 32) {
            int hu; int32_t tu;
            unit_rows(u, hu, tu);
            tma_load_3d(saddr(sm + OFF_K), &maps.k, 0, hu, tu, vkbar);
            tma_load_3d(saddr(sm + OFF_K + 8192), &maps.k, 64, hu, tu, vkbar);
        }
    };
    auto issue_qa = [&](int u) {
        if (tid == 32) {
            int hu; int32_t tu;
            unit_rows(u, hu, tu);
            const bool per_channel = p.alpha_mode == KDA_ALPHA_PER_CHANNEL;
            mbar_expect_tx(lbar, 16384 + (per_channel ? 32768 : 0));
            tma_load_3d(saddr(sm + OFF_Q), &maps.q, 0, hu, tu, lbar);
            tma_load_3d(saddr(sm + OFF_Q + 8192), &maps.q, 64, hu, tu, lbar);
            if (per_channel) {
#pragma unroll
                for (int b = 0; b < 4; ++b)
                    tma_load_3d(saddr(sm + OFF_G + b * 8192), &maps.a, 32 * b, hu, tu, lbar);
            }
        }
    };
    // piece 0-1: M (columns 0..127, TF32 rows 64.. of [Q'; M]); 2-3: B (128..255, fp32); 4: P Utilde
    // (384..511, lanes of rows 0..63).  Warp-collective; every thread calls it.
    bool big = false;                                        // a value outside fp16's range was seen
    auto drain = [&](int piece) {
        if (!rec_prev) return;
        __syncwarp();                                        // converged after an elected-lane MMA issue
        tc_fence_after();
        float v[32];
        if (piece < 4) {
            const int c0 = 64 * half + 32 * (piece & 1);
            tmem_ld32(tmem + tlane + (piece >= 2 ? DK : 0) + c0, v);
            if (piece < 2) {
#pragma unroll
                for (int x = 0; x < 32; x += 8) {                // one 16-byte core-matrix row per store
                    big |= fmaxf(fmaxf(fmaxf(fabsf(v[x]), fabsf(v[x + 1])), fmaxf(fabsf(v[x + 2]), fabsf(v[x + 3]))),
                                 fmaxf(fmaxf(fabsf(v[x + 4]), fabsf(v[x + 5])), fmaxf(fabsf(v[x + 6]), fabsf(v[x + 7])))) > kF16Max;
                    *reinterpret_cast<uint4*>(rec_prev + REC_QM + op_off_h(C + mi, c0 + x, DK)) =
                        make_uint4(pack_half2(v[x], v[x + 1]), pack_half2(v[x + 2], v[x + 3]),
                                   pack_half2(v[x + 4], v[x + 5]), pack_half2(v[x + 6], v[x + 7]));
                }
            } else {
#pragma unroll
                for (int x = 0; x < 32; x += 4) {
                    big |= fmaxf(fmaxf(fabsf(v[x]), fabsf(v[x + 1])), fmaxf(fabsf(v[x + 2]), fabsf(v[x + 3]))) > kF16Max;
                    *reinterpret_cast<uint2*>(rec_prev + REC_B + (((c0 + x) >> 2) * DK + mi) * 8) =
                        make_uint2(pack_half2(v[x], v[x + 1]), pack_half2(v[x + 2], v[x + 3]));
                }
            }
        } else {
#pragma unroll
            for (int cb = 0; cb < 2; ++cb) {
                const int c0 = 64 * half + 32 * cb;
                tmem_ld32(tmem + tlane + 3 * DK + c0, v);
                if (lane < 16) {
#pragma unroll
                    for (int x = 0; x < 32; x += 4) {
                        big |= fmaxf(fmaxf(fabsf(v[x]), fabsf(v[x + 1])), fmaxf(fabsf(v[x + 2]), fabsf(v[x + 3]))) > kF16Max;
                        *reinterpret_cast<uint2*>(rec_prev + REC_O + (((c0 + x) >> 2) * C + mr) * 8) =
                            make_uint2(pack_half2(v[x], v[x + 1]), pack_half2(v[x + 2], v[x + 3]));
                    }
                }
            }
        }
        tc_fence_before();
    };
    uint32_t lph = 0, vkph = 0;
    bool load_pending = (int)blockIdx.x < n_units;   // q and alpha of the next unit in flight
    bool vk_pending = load_pending;                   // v (and k) of the next unit in flight
    bool k_issued = load_pending;
    // beta (and a per-head alpha) of this thread's token row: a unit's values go to shared memory at the end
    // of the previous unit, from registers loaded at that unit's start, so no load latency is waited on
    float beta_next = 0.f, alpha_next = 1.f;
    const bool per_head = p.alpha_mode == KDA_ALPHA_PER_HEAD;
    if (load_pending) {
        issue_v(blockIdx.x);
        issue_k(blockIdx.x);
        issue_qa(blockIdx.x);
        int32_t tn, tn_end;
        chunk_span(p, choff, (int64_t)c_begin + (int)blockIdx.x / H, tn, tn_end, cu);
        if (tid < C) {
            const int64_t row = (int64_t)(tn + tid) * H + (int)blockIdx.x % H;
            const bool in = tn + tid < tn_end;
            sbeta[tid] = in ? p.beta[row] : 0.f;
            sasc[tid] = per_head && in ? p.alpha[row] : 1.f;
        }
    }
#ifdef KDA_TEST_HOOKS
    if (p.test_stall) {                              // the first copies are in flight: give up a wait now
        if (tid == 0) {
            asm volatile("mbarrier.init.shared::cta.b64 [%0], 1;" ::"r"(saddr(sm + P_OFF_MISC + 32)) : "memory");
            asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
        }
        __syncthreads();
        if (!test_stall_wait(saddr(sm + P_OFF_MISC + 32))) {
            atomicOr(p.err, KDA_DEVERR_TIMEOUT);
            *s_abort = 1;
        }
        __syncthreads();
    }
#endif

    for (int u = blockIdx.x; u < n_units; u += gridDim.x) {
        int32_t t0, t_end;                              // the chunk's first token and its sequence's end
        if (MULTI && u == span_unit) {
            t0 = s_span[0];
            t_end = s_span[1];
        } else {
            chunk_span(p, choff, (int64_t)c_begin + u / H, t0, t_end, cu);
        }
        const int L = min(C, t_end - t0);
        unsigned char* rec = records + (size_t)u * REC_BYTES;
        const int un = u + (int)gridDim.x;                       // this CTA's next unit
        if (!mbar_wait(vkbar, vkph) || !mbar_wait(lbar, lph)) {
            atomicOr(p.err, KDA_DEVERR_TIMEOUT);
            *s_abort = 1;
        }
        lph ^= 1u;
        vkph ^= 1u;
        load_pending = vk_pending = false;
        tc_fence_before();
        __syncthreads();
        if (*s_abort) break;
        if (tid < C && un < n_units) {                  // the next unit's beta (and alpha), used at this unit's end
            int32_t tn, tn_end;
            chunk_span(p, choff, (int64_t)c_begin + un / H, tn, tn_end, cu);
            const int64_t row = (int64_t)(tn + tid) * H + un % H;
            beta_next = tn + tid < tn_end ? p.beta[row] : 0.f;
            alpha_next = per_head && tn + tid < tn_end ? p.alpha[row] : 1.f;
            if (MULTI && tid == 0) {
                s_span[0] = tn;
                s_span[1] = tn_end;
            }
        }
        // s_span is read (tile fetches of unit un, the start of the next iteration) only after this unit's
        // next barrier
        if (MULTI) span_unit = un < n_units ? un : -1;
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

        // ---- 1. g = running sum of clamped log2 alpha per key channel; the largest |v| of the chunk ----
        bool one_ref;
        {
            const uint4* vv = reinterpret_cast<const uint4*>(sm + P_OFF_V) + tid;   // 16 B per thread per step
            uint32_t vm = 0u;                           // largest bf16 magnitude bits of this thread's 32 values
#pragma unroll
            for (int x = 0; x < 4; ++x) {               // two bf16 magnitudes per 32-bit word, maxima per half
                const uint4 w = vv[x * NT];
                vm = __vmaxu2(vm, __vmaxu2(__vmaxu2(w.x & 0x7FFF7FFFu, w.y & 0x7FFF7FFFu),
                                           __vmaxu2(w.z & 0x7FFF7FFFu, w.w & 0x7FFF7FFFu)));
            }
            vm = __reduce_max_sync(0xffffffffu, max(vm >> 16, vm & 0xFFFFu));
            if (lane == 0) reinterpret_cast<uint32_t*>(sm + P_OFF_VMX)[warp] = vm;
        }
        {
            float la[32];
#pragma unroll
            for (int x = 0; x < 32; ++x)
                la[x] = p.alpha_mode == KDA_ALPHA_PER_CHANNEL ? Gat(32 * rh + x, ch) : sasc[32 * rh + x];
            float acc = 0.f;
#pragma unroll
            for (int x = 0; x < 32; ++x) {
                acc += (32 * rh + x < L) ? fmaxf(lg2f(la[x]), kLog2AlphaMin) : 0.f;
                la[x] = acc;
            }
#pragma unroll
            for (int x = 0; x < 32; ++x) Gat(32 * rh + x, ch) = la[x];
            __syncthreads();
            // one decay reference for the whole chunk (row 31) keeps every factor of step 2 inside float range
            // when each channel decays by at most 2^kOneRefMax over rows 0..31 and over rows 31..63
            float span = la[0] - la[31];                // g_0 - g_31 (rows 0..31 of this channel)
            if (rh == 1) {
                const float base = Gat(31, ch);
#pragma unroll
                for (int x = 0; x < 32; ++x) Gat(32 + x, ch) = la[x] + base;
                sgam[ch] = ex2f(la[31] + base);
                span = -la[31];                         // g_31 - g_63
            }
            one_ref = !__syncthreads_or(span > kOneRefMax);
        }
        int ec;                                         // this chunk's value scale exponent
        {
            const uint4 m0 = *reinterpret_cast<const uint4*>(sm + P_OFF_VMX);
            const uint4 m1 = *reinterpret_cast<const uint4*>(sm + P_OFF_VMX + 16);
            ec = scale_exp_bf16(max(max(max(m0.x, m0.y), max(m0.z, m0.w)), max(max(m1.x, m1.y), max(m1.z, m1.w))));
        }
        const float vscale = exp2i(-ec);

        // ---- 2. A and P on tcgen05: with one reference (the decay allows it) one product of 16 instructions,
        //         otherwise one per 16-row block with its own reference ----
        float* Ab = reinterpret_cast<float*>(X + PS_A);
        float* Tb = reinterpret_cast<float*>(X + PS_T);
        float* scr = reinterpret_cast<float*>(X + PS_SCR);
        unsigned char* opP = X + PS_P;
        if (one_ref) {
            // L = [2^(g - g_31) . K; 2^(g - g_31) . Q] (M=128 rows r') and R = 2^(g_31 - g) . K (N=64 rows s), TF32,
            // K=128 channels: D[r'][s] = the A-part (rows r' < 64) and the P-part (rows r' >= 64) of the chunk
            const int cq = 4 * warp + (lane >> 3), j = lane & 7, i0 = 4 * cq;
            const float4 ref = *reinterpret_cast<const float4*>(sm + OFF_G + g_off(31, i0));
#pragma unroll
            for (int gi = 0; gi < 8; ++gi) {
                const int fr = 8 * gi + j;
                const float4 gg = *reinterpret_cast<const float4*>(sm + OFF_G + g_off(fr, i0));
                const uint2 kk = *reinterpret_cast<const uint2*>(sm + OFF_K + kq_off(fr, i0));
                const uint2 qq = *reinterpret_cast<const uint2*>(sm + OFF_Q + kq_off(fr, i0));
                const __nv_bfloat162* k2 = reinterpret_cast<const __nv_bfloat162*>(&kk);
                const __nv_bfloat162* q2 = reinterpret_cast<const __nv_bfloat162*>(&qq);
                const float kx = __low2float(k2[0]), ky = __high2float(k2[0]), kz = __low2float(k2[1]),
                            kw = __high2float(k2[1]);
                const float fx = ex2f(gg.x - ref.x), fy = ex2f(gg.y - ref.y), fz = ex2f(gg.z - ref.z),
                            fw = ex2f(gg.w - ref.w);
                *reinterpret_cast<float4*>(X + op_off(fr, i0, DK)) =
                    make_float4(tf32_rna(kx * ex2f(ref.x - gg.x)), tf32_rna(ky * ex2f(ref.y - gg.y)),
                                tf32_rna(kz * ex2f(ref.z - gg.z)), tf32_rna(kw * ex2f(ref.w - gg.w)));
                *reinterpret_cast<float4*>(X + ONE_L_OFF + op_off(fr, i0, DK)) =
                    make_float4(tf32_rna(kx * fx), tf32_rna(ky * fy), tf32_rna(kz * fz), tf32_rna(kw * fw));
                *reinterpret_cast<float4*>(X + ONE_L_OFF + op_off(C + fr, i0, DK)) =
                    make_float4(tf32_rna(__low2float(q2[0]) * fx), tf32_rna(__high2float(q2[0]) * fy),
                                tf32_rna(__low2float(q2[1]) * fz), tf32_rna(__high2float(q2[1]) * fw));
            }
            fence_async_smem();
            tc_fence_before();
            __syncthreads();
            if (warp == 0 && elect_one()) {
                tc_fence_after();
                constexpr uint32_t id = idesc_tf32(128, C);
                const uint64_t ad = op_desc(saddr(X + ONE_L_OFF), DK), bd = op_desc(saddr(X), DK);
#pragma unroll
                for (int ks = 0; ks < DK / 8; ++ks)
                    umma_tf32_1(tmem + TM_W, ad + (uint64_t)(ks * 16), bd + (uint64_t)(ks * 16), id, ks > 0 ? 1u : 0u);
                umma_commit(mbar);
            }
        } else {
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
                        make_float4(tf32_rna(kx * fx), tf32_rna(ky * fy), tf32_rna(kz * fz), tf32_rna(kw * fw));
                    *reinterpret_cast<float4*>(lb + op_off(16 + 8 * u + j, i0, DK)) =
                        make_float4(tf32_rna(__low2float(q2[0]) * fx), tf32_rna(__high2float(q2[0]) * fy),
                                    tf32_rna(__low2float(q2[1]) * fz), tf32_rna(__high2float(q2[1]) * fw));
                }
                unsigned char* rb = X + g1_r_off(b);
#pragma unroll
                for (int gi = 0; gi < 2 * (b + 1); ++gi)
                    *reinterpret_cast<float4*>(rb + op_off(8 * gi + j, i0, DK)) =
                        make_float4(tf32_rna(rv[gi].x), tf32_rna(rv[gi].y), tf32_rna(rv[gi].z), tf32_rna(rv[gi].w));
            }
            fence_async_smem();
            tc_fence_before();
            __syncthreads();
            if (warp == 0 && elect_one()) {             // per 16-row block b: R_b [Lk_b; Lq_b]^T, M=64, N=32
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
                        umma_tf32_1(tmem + TM_W + 32 * b, ad[b] + (uint64_t)(ks * 16), bdsc[b] + (uint64_t)(ks * 16),
                                    id, ks > 0 ? 1u : 0u);
                }
                umma_commit(mbar);
            }
        }
        drain(0);                                       // while the products run
        drain(1);
        if (!wait_mma()) break;
        if (one_ref) {                                  // scatter: row r' of D, columns s = 32 half .. + 31
            float v[32];
            tmem_ld32(tmem + tlane + TM_W + 32 * half, v);
            const int s0 = 32 * half;
            if (quad < 2) {                             // A (fp32, strictly lower, beta-scaled), row r
                const int r = 32 * quad + lane;
                const float br = sbeta[r];
#pragma unroll
                for (int x = 0; x < 32; x += 4)
                    *reinterpret_cast<float4*>(Ab + r * AT_LD + s0 + x) =
                        make_float4(s0 + x < r ? br * v[x] : 0.f, s0 + x + 1 < r ? br * v[x + 1] : 0.f,
                                    s0 + x + 2 < r ? br * v[x + 2] : 0.f, s0 + x + 3 < r ? br * v[x + 3] : 0.f);
            } else {                                    // P (fp16 operand, lower with the diagonal), row r
                const int r = 32 * quad + lane - C;
#pragma unroll
                for (int x = 0; x < 32; x += 8)
                    *reinterpret_cast<uint4*>(opP + op_off_h(r, s0 + x, C)) = make_uint4(
                        pack_half2(s0 + x <= r ? v[x] : 0.f, s0 + x + 1 <= r ? v[x + 1] : 0.f),
                        pack_half2(s0 + x + 2 <= r ? v[x + 2] : 0.f, s0 + x + 3 <= r ? v[x + 3] : 0.f),
                        pack_half2(s0 + x + 4 <= r ? v[x + 4] : 0.f, s0 + x + 5 <= r ? v[x + 5] : 0.f),
                        pack_half2(s0 + x + 6 <= r ? v[x + 6] : 0.f, s0 + x + 7 <= r ? v[x + 7] : 0.f));
            }
        } else {                                        // scatter: A (fp32) and P (fp16 operand)
            const int sr = 16 * quad + lane;
            float v[32];
#pragma unroll
            for (int bb = 0; bb < 2; ++bb) {
                const int b = 2 * half + bb;
                tmem_ld32(tmem + tlane + TM_W + 32 * b, v);
                if (lane < 16) {
#pragma unroll
                    for (int c = 0; c < 16; ++c) {
                        const int r = 16 * b + c;
                        Ab[r * AT_LD + sr] = sr < r ? sbeta[r] * v[c] : 0.f;
                        *reinterpret_cast<__half*>(opP + op_off_h(r, sr, C)) = __float2half_rn(sr <= r ? v[16 + c] : 0.f);
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
        // T' = T Diag(beta) -> fp16 operand (M=64, K=64); the operands of steps 4 and 6 are fp16 (the same
        // 10-bit significand as TF32; their values are O(1) for unit-norm keys, and v and T' are checked)
        for (int e = tid; e < C * 8; e += NT) {                    // row r, columns m0 .. m0 + 7 per thread
            const int r = (e & 7) | (((e >> 6) & 7) << 3), m0 = 8 * ((e >> 3) & 7);
            const float4 t0 = *reinterpret_cast<const float4*>(Tb + r * AT_LD + m0);
            const float4 t1 = *reinterpret_cast<const float4*>(Tb + r * AT_LD + m0 + 4);
            const float4 b0 = *reinterpret_cast<const float4*>(sbeta + m0);
            const float4 b1 = *reinterpret_cast<const float4*>(sbeta + m0 + 4);
            float v[8] = {t0.x * b0.x, t0.y * b0.y, t0.z * b0.z, t0.w * b0.w, t1.x * b1.x, t1.y * b1.y, t1.z * b1.z, t1.w * b1.w};
#pragma unroll
            for (int x = 0; x < 8; ++x) v[x] = m0 + x <= r ? v[x] : 0.f;
            big |= fmaxf(fmaxf(fmaxf(fabsf(v[0]), fabsf(v[1])), fmaxf(fabsf(v[2]), fabsf(v[3]))),
                         fmaxf(fmaxf(fabsf(v[4]), fabsf(v[5])), fmaxf(fabsf(v[6]), fabsf(v[7])))) > kF16Max;
            *reinterpret_cast<uint4*>(X + PS_OPT + op_off_h(r, m0, C)) =
                make_uint4(pack_half2(v[0], v[1]), pack_half2(v[2], v[3]), pack_half2(v[4], v[5]), pack_half2(v[6], v[7]));
        }
        // [Gamma.K | V]^T -> fp16 operand (N=256 rows, K=64 time), v scaled by 2^-e_c
        // 8 time rows of channel i per thread, one 16-byte core-matrix row per store: a warp's four 8-row
        // groups lie 1 KiB apart (the same banks), so 8-byte stores took as many wavefronts for half the bytes
        for (int e = tid; e < DK * 8; e += NT) {
            const int i = e & (DK - 1), m0 = 8 * (e >> 7);
            float gk[8], vv[8];
#pragma unroll
            for (int x = 0; x < 8; ++x) {
                gk[x] = ex2f(Gat(m0 + x, i)) * kat(m0 + x, i);
                vv[x] = vscale * bf(vraw + (m0 + x) * DK + i);
            }
            *reinterpret_cast<uint4*>(X + PS_KV + op_off_h(i, m0, C)) =
                make_uint4(pack_half2(gk[0], gk[1]), pack_half2(gk[2], gk[3]), pack_half2(gk[4], gk[5]),
                           pack_half2(gk[6], gk[7]));
            big |= fmaxf(fmaxf(fmaxf(fabsf(vv[0]), fabsf(vv[1])), fmaxf(fabsf(vv[2]), fabsf(vv[3]))),
                         fmaxf(fmaxf(fabsf(vv[4]), fabsf(vv[5])), fmaxf(fabsf(vv[6]), fabsf(vv[7])))) > kF16Max;
            *reinterpret_cast<uint4*>(X + PS_KV + op_off_h(DK + i, m0, C)) =
                make_uint4(pack_half2(vv[0], vv[1]), pack_half2(vv[2], vv[3]), pack_half2(vv[4], vv[5]),
                           pack_half2(vv[6], vv[7]));
        }
        fence_async_smem();
        tc_fence_before();
        __syncthreads();
        if (un < n_units) {                                      // this unit's v is read: fetch the next v
            issue_v(un);
            vk_pending = true;
            k_issued = false;
        }

        // ---- 4. [W | Utilde]^T = [Gamma.K | V]^T T'^T  (two M=128 halves, N=64, K=64) ----
        if (warp == 0 && elect_one()) {
            tc_fence_after();
            constexpr uint32_t id = idesc_f16(128, C);
            const uint64_t aw = op_desc_h(saddr(X + PS_KV), C), au = op_desc_h(saddr(X + PS_KV + DK * C * 2), C);
            const uint64_t bt = op_desc_h(saddr(X + PS_OPT), C);
#pragma unroll
            for (int ks = 0; ks < C / 16; ++ks) {
                umma_f16_1(tmem + TM_W, aw + (uint64_t)(ks * 16), bt + (uint64_t)(ks * 16), id, ks > 0 ? 1u : 0u);
                umma_f16_1(tmem + TM_W + C, au + (uint64_t)(ks * 16), bt + (uint64_t)(ks * 16), id, ks > 0 ? 1u : 0u);
            }
            umma_commit(mbar);
        }
        drain(2);                                       // while the products run
        drain(3);
        if (!wait_mma()) break;

        // ---- 5. fold operands: [W | Utilde]^T (N=256, K=64) and Khat^T (M=128, K=64) ----
        unsigned char* opWU = X + PS_WU;
        unsigned char* opKH = X + PS_KH;
        {
            const int n = DK * half + 32 * quad + lane;          // row of [W | Utilde]^T held by this lane
            float v[32];
#pragma unroll
            for (int cb = 0; cb < 2; ++cb) {
                tmem_ld32(tmem + tlane + TM_W + C * half + 32 * cb, v);
#pragma unroll
                for (int x = 0; x < 32; x += 8) {
                    big |= fmaxf(fmaxf(fmaxf(fabsf(v[x]), fabsf(v[x + 1])), fmaxf(fabsf(v[x + 2]), fabsf(v[x + 3]))),
                                 fmaxf(fmaxf(fabsf(v[x + 4]), fabsf(v[x + 5])), fmaxf(fabsf(v[x + 6]), fabsf(v[x + 7])))) > kF16Max;
                    *reinterpret_cast<uint4*>(opWU + op_off_h(n, 32 * cb + x, C)) =
                        make_uint4(pack_half2(v[x], v[x + 1]), pack_half2(v[x + 2], v[x + 3]),
                                   pack_half2(v[x + 4], v[x + 5]), pack_half2(v[x + 6], v[x + 7]));
                }
            }
        }
        for (int e = tid; e < DK * 8; e += NT) {                  // 8 time rows of channel i per thread
            const int i = e & (DK - 1), s0 = 8 * (e >> 7);
            const float gl = Gat(C - 1, i);
            float kh[8];
#pragma unroll
            for (int x = 0; x < 8; ++x) kh[x] = ex2f(gl - Gat(s0 + x, i)) * kat(s0 + x, i);
            *reinterpret_cast<uint4*>(opKH + op_off_h(i, s0, C)) =
                make_uint4(pack_half2(kh[0], kh[1]), pack_half2(kh[2], kh[3]), pack_half2(kh[4], kh[5]),
                           pack_half2(kh[6], kh[7]));
        }
        drain(4);                                       // the last piece, before step 6 writes its columns
        rec_prev = nullptr;
        {
            // -Gamma.Q into the PW half of step 6's M=64 accumulator (row r at lane r % 16 of quadrant r / 16,
            // columns 2 DK + c) and zeros into its P Utilde half, so that step 6 accumulates PW - Gamma.Q = -Q'
            // and q and alpha are free from here on; each warp writes the 64 columns of its own quadrant that
            // it has just read the [W | Utilde]^T accumulator from, lane (g, t) rows 16 quad + g (+ 8) and
            // column pairs 8 j + 2 t (16x256b shape: every lane carries rows the products use)
            float v[32];
#pragma unroll
            for (int j = 0; j < 8; ++j)
#pragma unroll
                for (int h = 0; h < 2; ++h) {
                    const int r = 16 * quad + gid + 8 * h, c = 64 * half + 8 * j + 2 * tig;
                    const float2 gg = *reinterpret_cast<const float2*>(sm + OFF_G + g_off(r, c));
                    const __nv_bfloat162 q2 = *reinterpret_cast<const __nv_bfloat162*>(sm + OFF_Q + kq_off(r, c));
                    v[4 * j + 2 * h] = -ex2f(gg.x) * __low2float(q2);
                    v[4 * j + 2 * h + 1] = -ex2f(gg.y) * __high2float(q2);
                }
            tmem_st16x256b_x8(tmem + tlane + 2 * DK + 64 * half, v);
#pragma unroll
            for (int x = 0; x < 32; ++x) v[x] = 0.f;
            tmem_st16x256b_x8(tmem + tlane + 3 * DK + 64 * half, v);
            tmem_wait_st();
        }
        fence_async_smem();
        tc_fence_before();
        __syncthreads();
        if (un < n_units) {                  // this unit's k, q and alpha are read: fetch the next unit's tiles
            issue_k(un);
            k_issued = true;
            issue_qa(un);
            load_pending = true;
        }

        // ---- 6. [M | B] = Khat^T [W | Utilde] (M=128) and [PW | P Utilde] = P [W | Utilde] (M=64); N=256, K=64 ----
        if (warp == 0) {
            if (elect_one()) {
                tc_fence_after();
                const uint64_t ak = op_desc_h(saddr(opKH), C), ap = op_desc_h(saddr(opP), C);
                const uint64_t bw = op_desc_h(saddr(opWU), C);
#pragma unroll
                for (int ks = 0; ks < C / 16; ++ks) {
                    const uint64_t bd = bw + (uint64_t)(ks * 16);
                    umma_f16_1(tmem, ak + (uint64_t)(ks * 16), bd, idesc_f16(128, 2 * DK), ks > 0 ? 1u : 0u);
                    umma_f16_1(tmem + 2 * DK, ap + (uint64_t)(ks * 16), bd, idesc_f16(64, 2 * DK), 1u);
                }
                umma_commit(mbar);
            }
            __syncwarp();
        }
        if (!wait_mma()) break;

        // ---- 7. the record: Q' and Gamma_C now; M, B and P Utilde stay in TMEM and drain during the next unit ----
        float v[32];
#pragma unroll
        for (int cb = 0; cb < 2; ++cb) {                         // Q' = Gamma.Q - P W -> rows 0..63 of [Q'; M]
            // (the accumulator holds P W - Gamma.Q)
            const int c0 = 64 * half + 32 * cb;
            tmem_ld32(tmem + tlane + 2 * DK + c0, v);
            if (lane < 16) {
#pragma unroll
                for (int x = 0; x < 32; x += 8) {                // one 16-byte core-matrix row per store
                    big |= fmaxf(fmaxf(fmaxf(fabsf(v[x]), fabsf(v[x + 1])), fmaxf(fabsf(v[x + 2]), fabsf(v[x + 3]))),
                                 fmaxf(fmaxf(fabsf(v[x + 4]), fabsf(v[x + 5])), fmaxf(fabsf(v[x + 6]), fabsf(v[x + 7])))) > kF16Max;
                    *reinterpret_cast<uint4*>(rec + REC_QM + op_off_h(mr, c0 + x, DK)) =
                        make_uint4(pack_half2(-v[x], -v[x + 1]), pack_half2(-v[x + 2], -v[x + 3]),
                                   pack_half2(-v[x + 4], -v[x + 5]), pack_half2(-v[x + 6], -v[x + 7]));
                }
            }
        }
        if (tid < DK) reinterpret_cast<float*>(rec + REC_G)[tid] = sgam[tid];
        if (tid == 0) *reinterpret_cast<int*>(rec + REC_E) = ec;
        rec_prev = rec;
        fence_async_smem();
        tc_fence_before();
        __syncthreads();
        if (un < n_units && tid < C) {                           // beta was read in steps 2-3, alpha in step 1
            sbeta[tid] = beta_next;
            sasc[tid] = alpha_next;
        }
    }

    // the last unit's M, B and P Utilde (not after an abort: the products may not have completed)
    if (!*s_abort)
        for (int piece = 0; piece < 5; ++piece) drain(piece);
    // bounded: never leave copies in flight (after an abort between the v and k fetches the k tiles are
    // fetched too, so that vkbar's phase can complete)
    if (big) atomicOr(p.err, KDA_DEVERR_RANGE);
    if (vk_pending && !k_issued) issue_k(blockIdx.x);
    if (vk_pending) mbar_wait(vkbar, vkph);
    if (load_pending) mbar_wait(lbar, lph);
    tc_fence_before();
    __syncthreads();
    if (warp == 0) {
        tc_fence_after();
        asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem), "r"(512) : "memory");
    }
}

// ============================================================================================
// Phase 2: one CTA per (sequence, head, NV value columns); it walks that sequence's chunks inside the window
// [c_begin, c_begin + n_chunks) in order, from state_in where the sequence starts in the window and from
// the state carried in state_out otherwise, and leaves its state in state_out.  With several sequences
// (choff set) blockIdx enumerates (order[i], head, slice), longest sequences first; a CTA whose sequence
// has no chunk in the window exits at once (a zero-length sequence copies state_in to state_out in the
// first window).
//
// Warps 0-7 hold the state (thread = one key channel, NV/2 value columns) and run the fp32 update;
// warp 8 issues the products, warp 9 the record loads; warps 10-13 run the output epilogue (the output
// product is M=64, whose row 16 q + i sits at lane i of TMEM lane quadrant q, and warp w reaches quadrant
// w mod 4).  Per chunk c:
//   warp 8:      wait record c, sbar ("S_c written") and ofree (output of c-2 read); issue M S_c -> dbar,
//                then Q' S_c -> obar (issued while the state warps update S)
//   warp 9:      wait obar, load record c+2 into the freed buffer; prefetch B and P Utilde of c+4 into L2
//   warps 0-7:   wait dbar; S_{c+1} = Gamma_C S_c + B - M S_c; write the S^T operand of c+1; arrive on sbar
//   warps 10-13: wait obar and the end of chunk c's state update (state warp 0 publishes E of c+1);
//                o = scale (Q' S_c + P Utilde) for rows 0..63; arrive on ofree
// so the output products and epilogue of one chunk overlap the state products of the next, and the
// state warps' proxy fence never waits on output traffic.  The S^T operand and the output accumulator
// are double-buffered; M S uses one accumulator (it is read before the arrival on sbar).  Every barrier
// can run at most one phase ahead of each of its waiters.
// ============================================================================================
template <bool MULTI, int NV>
__global__ void __launch_bounds__(C_NT, 1)
    kda_prefill_chain_kernel(PrefillParams p, const unsigned char* records, int c_begin, int n_window,
                             const int32_t* choff_arg, const int32_t* order) {
    const int32_t* choff = MULTI ? choff_arg : nullptr;
    extern __shared__ __align__(1024) unsigned char sm[];
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int quad = warp & 3, half = (warp >> 2) & 1;
    static_assert(NV == 16 || NV == 32, "16 or 32 value columns per CTA");
    constexpr int CPT = NV / 2;                       // value columns per state thread
    constexpr int NSL = DK / NV;                      // slices of a head
    const int H = p.H;
    const int seq_i = blockIdx.x / (H * NSL), hs = blockIdx.x % (H * NSL);
    const int h = hs / NSL, slice = hs % NSL, j0 = slice * NV;
    if (!choff && !valid_single_sequence(p)) {
        if (tid == 0) atomicOr(p.err, KDA_DEVERR_CU_SEQLENS);
        return;
    }
    // this CTA's sequence, its tokens [s0, s0 + T) and its chunks inside the window [g0, g0 + n_chunks)
    const int n = choff ? (order ? order[seq_i] : seq_i) : 0;
    const int32_t s0 = choff ? p.cu_seqlens[n] : 0;
    const int32_t T = choff ? (choff[n + 1] > choff[n] ? p.cu_seqlens[n + 1] - s0 : 0) : p.total_tokens;
    const int64_t cseq = choff ? choff[n] : 0, cseq_end = choff ? choff[n + 1] : ((int64_t)T + C - 1) / C;
    const int64_t g0 = cseq > c_begin ? cseq : c_begin;
    const int64_t g1 = cseq_end < (int64_t)c_begin + n_window ? cseq_end : (int64_t)c_begin + n_window;
    const int n_chunks = g1 > g0 ? (int)(g1 - g0) : 0;
    const int64_t state_base = ((int64_t)n * H + h) * DK * (int64_t)p.dv;   // this (sequence, head)'s state
    if (g0 == cseq && h == 0 && slice == 0 && tid == 0 && (n_chunks > 0 || c_begin == 0) &&
        snapshot_offsets_bad(p, n, T))
        atomicOr(p.err, KDA_DEVERR_SNAPSHOTS);
    if (n_chunks == 0) {
        if (cseq == cseq_end && c_begin == 0 && tid < 256) {      // an empty sequence: state_out = state_in
            for (int e = tid; e < DK * NV / 4; e += 256) {
                const int64_t at = state_base + (int64_t)(e / (NV / 4)) * p.dv + j0 + 4 * (e % (NV / 4));
                const float4 v4 = p.state_in ? *reinterpret_cast<const float4*>(p.state_in + at)
                                             : make_float4(0.f, 0.f, 0.f, 0.f);
                *reinterpret_cast<float4*>(p.state_out + at) = v4;
            }
        }
        return;
    }
    // the state this window starts from: state_in where the sequence starts here, else the carried state
    const float* state_in = g0 == cseq ? p.state_in : p.state_out;
    if (saddr(sm) & 1023u) {
        if (tid == 0) atomicOr(p.err, KDA_DEVERR_TIMEOUT);
        return;
    }
    __nv_bfloat16* go = static_cast<__nv_bfloat16*>(p.o);
    unsigned char* misc = sm + C_OFF_MISC;
    volatile int* s_abort = reinterpret_cast<volatile int*>(misc + 100);
    uint32_t* s_tmem = reinterpret_cast<uint32_t*>(misc + 96);
    const uint32_t lbar = saddr(misc), dbar = saddr(misc + 16), obar = saddr(misc + 32), sbar = saddr(misc + 48);
    const uint32_t ofree = saddr(misc + 64);
    // ebar[c & 3]: E of chunk c's state operand is in E_ring[c & 3] (one arrival, by state warp 0)
    const uint32_t ebar = saddr(misc + CM_EBAR);
    volatile int* e_ring = reinterpret_cast<volatile int*>(misc + CM_ERING);
    uint32_t* smax = reinterpret_cast<uint32_t*>(misc + CM_SLOT);   // read only after an mbarrier acquire
    constexpr uint32_t TM_S = 0, TM_O = 32;           // M S accumulator; two Q' S accumulators

    if (tid == 0) {
        for (int b = 0; b < 2; ++b) {
            asm volatile("mbarrier.init.shared::cta.b64 [%0], 1;" ::"r"(lbar + 8 * b) : "memory");
            asm volatile("mbarrier.init.shared::cta.b64 [%0], 1;" ::"r"(dbar + 8 * b) : "memory");
            asm volatile("mbarrier.init.shared::cta.b64 [%0], 1;" ::"r"(obar + 8 * b) : "memory");
        }
        asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(sbar), "r"(NT) : "memory");
        for (int b = 0; b < 2; ++b)
            asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(ofree + 8 * b), "r"(128) : "memory");
        for (int b = 0; b < 4; ++b)
            asm volatile("mbarrier.init.shared::cta.b64 [%0], 1;" ::"r"(ebar + 8 * b) : "memory");
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
        *s_abort = 0;
    }
    if (warp == 0) {
        asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(saddr(s_tmem)), "r"(128)
                     : "memory");
        asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
    }
    // the state scale exponent E_0 of this slice's state_in (the state warps' rows, read once here)
    uint32_t* s_smx = reinterpret_cast<uint32_t*>(misc + CM_SMX0);
    if (warp < 8) {
        uint32_t m = 0u;
        if (state_in) {
            const float* src = state_in + state_base + (int64_t)(32 * quad + lane) * p.dv + j0 + CPT * half;
#pragma unroll
            for (int j = 0; j < CPT; j += 4) {
                const float4 v4 = *reinterpret_cast<const float4*>(src + j);
                m = max(m, max(max(__float_as_uint(fabsf(v4.x)), __float_as_uint(fabsf(v4.y))),
                               max(__float_as_uint(fabsf(v4.z)), __float_as_uint(fabsf(v4.w)))));
            }
        }
        m = __reduce_max_sync(0xffffffffu, m);
        if (lane == 0) s_smx[warp] = m;
    }
    // launched as phase 1's programmatic dependent (one stream): everything above reads only what was
    // written before phase 1 started; the records are read below, once phase 1 has completed
    asm volatile("griddepcontrol.wait;" ::: "memory");
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *s_tmem;
    int E0;                                           // every thread: the state is carried divided by 2^E
    {
        uint32_t m = 0u;
#pragma unroll
        for (int w = 0; w < 8; ++w) m = max(m, s_smx[w]);
        E0 = scale_exp_f32(m);
    }
    if (tid == 0) {                                   // chunk 0's state operand is at scale E_0
        e_ring[0] = E0;
        mbar_arrive(ebar);
    }
    auto fail = [&]() {
        atomicOr(p.err, KDA_DEVERR_TIMEOUT);
        *s_abort = 1;
    };
#ifdef KDA_TEST_HOOKS
    if (p.test_stall) {                              // give up a wait before the roles start
        if (tid == 0) {
            asm volatile("mbarrier.init.shared::cta.b64 [%0], 1;" ::"r"(saddr(misc + 104)) : "memory");
            asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
        }
        __syncthreads();
        if (!test_stall_wait(saddr(misc + 104))) fail();
        __syncthreads();
    }
#endif

    const uint32_t sop0 = saddr(sm + C_OFF_S);
    if (warp == 8) {
        // ---------------- products: M S_c (sequential path), then Q' S_c ----------------
        const uint64_t a_s0 = op_desc_h(saddr(sm) + C * DK * 2, DK), a_o0 = op_desc_h(saddr(sm), DK);
        const uint64_t b_s0 = desc_sw128(sop0);
        int issued = 0;                               // chunks whose products were issued
        for (int ci = 0; ci < n_chunks; ++ci) {
            const int b = ci & 1;
            const uint32_t par = (uint32_t)(ci >> 1) & 1u;
            if (!mbar_wait(lbar + 8 * b, par)) fail();
            if (!mbar_wait(sbar, (uint32_t)ci & 1u)) fail();
            // the output accumulator of chunk ci was last read by the output warps for chunk ci - 2
            if (ci >= 2 && !mbar_wait(ofree + 8 * b, par ^ 1u)) fail();
            if (*s_abort) break;
            tc_fence_after();
            if (elect_one()) {
                const uint64_t bs = b_s0 + (uint64_t)((b * SOP_BYTES) >> 4);
                const uint64_t as = a_s0 + (uint64_t)((b * QM_BYTES) >> 4), ao = a_o0 + (uint64_t)((b * QM_BYTES) >> 4);
#pragma unroll
                for (int ks = 0; ks < DK / 16; ++ks)           // 16 fp16 = 32 bytes of K per step
                    umma_f16_1(tmem + TM_S, as + (uint64_t)(ks * 16),
                               bs + (uint64_t)(((ks >> 2) * (NV * 128) + (ks & 3) * 32) >> 4), idesc_f16(128, NV),
                               ks > 0 ? 1u : 0u);
                umma_commit(dbar + 8 * b);
#pragma unroll
                for (int ks = 0; ks < DK / 16; ++ks)
                    umma_f16_1(tmem + TM_O + NV * b, ao + (uint64_t)(ks * 16),
                               bs + (uint64_t)(((ks >> 2) * (NV * 128) + (ks & 3) * 32) >> 4), idesc_f16(64, NV),
                               ks > 0 ? 1u : 0u);
                umma_commit(obar + 8 * b);
            }
            __syncwarp();
            issued = ci + 1;
        }
        // never leave products in flight
        if (issued > 0) mbar_wait(obar + 8 * ((issued - 1) & 1), (uint32_t)((issued - 1) >> 1) & 1u);
    } else if (warp == 9) {
        // ---------------- record loads: [Q'; M] of chunk c + 2 once the products of c are done ----------------
        auto load = [&](int ci) {                     // [Q'; M] of chunk ci into buffer ci & 1
            if (lane == 0) {
                const uint32_t lb = lbar + 8 * (ci & 1);
                mbar_expect_tx(lb, QM_BYTES);
                bulk_g2s(saddr(sm + (ci & 1) * QM_BYTES), records + (size_t)((g0 - c_begin + ci) * H + h) * REC_BYTES + REC_QM,
                         QM_BYTES, lb);
            }
        };
        // this slice's B and P Utilde and the chunk's Gamma_C, pulled into L2 kPrefetchAhead chunks before the
        // state and output warps read them (the records were written long before and are no longer in L2;
        // a load from DRAM one chunk ahead was still in flight at the state update)
        auto prefetch = [&](int ci) {
            if (lane == 0 && ci < n_chunks) {
                const unsigned char* rec = records + (size_t)((g0 - c_begin + ci) * H + h) * REC_BYTES;
                prefetch_l2(rec + REC_B + (size_t)(j0 >> 2) * DK * 8, (NV / 4) * DK * 8);
                prefetch_l2(rec + REC_O + (size_t)(j0 >> 2) * C * 8, (NV / 4) * C * 8);
                prefetch_l2(rec + REC_G, REC_BYTES - REC_G);
            }
        };
        for (int c = 1; c < kPrefetchAhead; ++c) prefetch(c);
        if (n_chunks > 0) load(0);
        if (n_chunks > 1) load(1);
        int loaded = n_chunks < 2 ? n_chunks : 2;
        for (int ci = 0; ci + 2 < n_chunks; ++ci) {
            if (*s_abort) break;
            if (!mbar_wait_lazy(obar + 8 * (ci & 1), (uint32_t)(ci >> 1) & 1u)) { fail(); break; }
            load(ci + 2);
            prefetch(ci + kPrefetchAhead);
            loaded = ci + 3;
        }
        // never leave copies in flight: every issued load completes (bounded waits)
        for (int ci = loaded - 2 < 0 ? 0 : loaded - 2; ci < loaded; ++ci)
            mbar_wait(lbar + 8 * (ci & 1), (uint32_t)(ci >> 1) & 1u);
    } else if (warp >= 10) {
        // ---------------- output warps: rows 0..63 of chunk c (M=64: row 16 q + i at lane i of quadrant q) ----------------
        const int orow = 16 * quad + (lane & 15);
        const uint32_t tlane = (uint32_t)(32 * quad) << 16;
        uint2 oq[NV / 4];                              // raw fp16, converted where used
        int eo = 0;                                    // the chunk's value scale exponent
        auto fetch_o = [&](int ci) {                  // the chunk's P Utilde for this row and slice
            const unsigned char* rec = records + (size_t)((g0 - c_begin + ci) * H + h) * REC_BYTES;
#pragma unroll
            for (int m = 0; m < NV / 4; ++m)
                oq[m] = lane < 16 ? __ldg(reinterpret_cast<const uint2*>(rec + REC_O + (((j0 + 4 * m) >> 2) * C + orow) * 8))
                                  : make_uint2(0u, 0u);
            eo = __ldg(reinterpret_cast<const int*>(rec + REC_E));
        };
        if (n_chunks > 0) fetch_o(0);
        for (int ci = 0; ci < n_chunks; ++ci) {
            const int b = ci & 1;
            if (*s_abort) break;
            if (!mbar_wait(obar + 8 * b, (uint32_t)(ci >> 1) & 1u)) { fail(); break; }
            if (!mbar_wait(ebar + 8 * (ci & 3), (uint32_t)(ci >> 2) & 1u)) { fail(); break; }
            // start the epilogue once state warp 0 has finished this chunk's update (it publishes the next
            // chunk's E), so that it runs under the next round trip through the tensor core instead of
            // taking issue slots from the update
            if (ci + 1 < n_chunks && !mbar_wait(ebar + 8 * ((ci + 1) & 3), (uint32_t)((ci + 1) >> 2) & 1u)) { fail(); break; }
            const int E = e_ring[ci & 3];               // the scale of the chunk's state operand
            tc_fence_after();
            float d[NV];
            tmem_ld<NV>(tmem + tlane + TM_O + NV * b, d);
            tc_fence_before();
            mbar_arrive(ofree + 8 * b);
            const int32_t t0 = (int32_t)(g0 - cseq + ci) * C;   // within the sequence
            if (lane < 16 && orow < min(C, T - t0)) {
                __nv_bfloat16* dst = go + ((int64_t)(s0 + t0 + orow) * H + h) * p.dv + j0;
                const float fd = exp2i(E), fo = exp2i(eo);      // 1 unless values or the state are large
#pragma unroll
                for (int x = 0; x < NV; x += 8) {
                    const float4 o0 = half4_to_float4(oq[x / 4]), o1 = half4_to_float4(oq[x / 4 + 1]);
                    *reinterpret_cast<uint4*>(dst + x) = make_uint4(
                        pack_bf16x2(p.scale * (fd * d[x] + fo * o0.x), p.scale * (fd * d[x + 1] + fo * o0.y)),
                        pack_bf16x2(p.scale * (fd * d[x + 2] + fo * o0.z), p.scale * (fd * d[x + 3] + fo * o0.w)),
                        pack_bf16x2(p.scale * (fd * d[x + 4] + fo * o1.x), p.scale * (fd * d[x + 5] + fo * o1.y)),
                        pack_bf16x2(p.scale * (fd * d[x + 6] + fo * o1.z), p.scale * (fd * d[x + 7] + fo * o1.w)));
                }
            }
            if (ci + 1 < n_chunks) fetch_o(ci + 1);
        }
    } else if (warp < 8) {
        // ---------------- state warps ----------------
        const uint32_t tlane = (uint32_t)(quad * 32) << 16;
        const int srow = 32 * quad + lane;            // state row (key channel)
        const int jc = j0 + CPT * half;               // first value column of this thread
        const int64_t state_off = state_base + (int64_t)srow * p.dv + jc;
        float S[CPT];                                 // the state divided by 2^E
        int E = E0;
        {
            const float f = exp2i(-E0);
#pragma unroll
            for (int j = 0; j < CPT; j += 4) {
                const float4 v4 = state_in ? *reinterpret_cast<const float4*>(state_in + state_off + j)
                                           : make_float4(0.f, 0.f, 0.f, 0.f);
                S[j] = f * v4.x; S[j + 1] = f * v4.y; S[j + 2] = f * v4.z; S[j + 3] = f * v4.w;
            }
        }
        bool big = false;                             // a state value outside fp16's range was seen
        // S^T of chunk c: row = value column, K = srow, fp16; and this warp's largest |S| (m, this thread's,
        // computed where S is) for the choice of the next scale
        auto write_state_operand = [&](int c, float m) {
            unsigned char* sop = sm + C_OFF_S + (c & 1) * SOP_BYTES;
            const uint32_t mw = __reduce_max_sync(0xffffffffu, __float_as_uint(m));   // its latency under the stores
#pragma unroll
            for (int j = 0; j < CPT; ++j)
                *reinterpret_cast<__half*>(sop + sw128_off_h(CPT * half + j, srow, NV)) = __float2half_rn(S[j]);
            big |= m > kF16Max;
            if (lane == 0) smax[(c & 1) * 8 + warp] = mw;
            fence_async_smem();
            tc_fence_before();
            mbar_arrive(sbar);
        };
        auto absmax = [&]() {                         // a tree, not a chain of dependent maxima
            float m[CPT / 2];
#pragma unroll
            for (int j = 0; j < CPT / 2; ++j) m[j] = fmaxf(fabsf(S[2 * j]), fabsf(S[2 * j + 1]));
#pragma unroll
            for (int w = CPT / 4; w >= 1; w >>= 1)
#pragma unroll
                for (int j = 0; j < w; ++j) m[j] = fmaxf(m[j], m[j + w]);
            return m[0];
        };
        // the chunk's B, Gamma_C and value scale, fetched one chunk ahead, after the proxy fence (which would
        // wait on them)
        uint2 bq[CPT / 4];                             // raw fp16: converted where used
        float gamC = 0.f;
        int eb = 0;                                    // the chunk's value scale exponent
        auto fetch_b = [&](int ci) {
            const unsigned char* rec = records + (size_t)((g0 - c_begin + ci) * H + h) * REC_BYTES;
#pragma unroll
            for (int m = 0; m < CPT / 4; ++m)
                bq[m] = __ldg(reinterpret_cast<const uint2*>(rec + REC_B + (((jc + 4 * m) >> 2) * DK + srow) * 8));
            gamC = __ldg(reinterpret_cast<const float*>(rec + REC_G) + srow);
            eb = __ldg(reinterpret_cast<const int*>(rec + REC_E));
        };
        write_state_operand(0, absmax());
        if (n_chunks > 0) fetch_b(0);
        // the next snapshot point after the window start (never reached when there are no snapshots)
        int32_t snap_next = p.snap_every > 0 ? ((int32_t)(g0 - cseq) * C / p.snap_every + 1) * p.snap_every : -1;
        bool ok = true;
        for (int ci = 0; ci < n_chunks; ++ci) {
            const int b = ci & 1;
            const uint32_t par = (uint32_t)(ci >> 1) & 1u;
            if (*s_abort) { ok = false; break; }
            // every state warp's largest |S_c| (written before its arrival on sbar for chunk c; that phase is
            // complete, so this wait returns at once and orders the reads after those writes)
            if (!mbar_wait(sbar, (uint32_t)ci & 1u)) { fail(); ok = false; break; }
            const uint4 m0 = reinterpret_cast<const uint4*>(const_cast<const uint32_t*>(smax))[2 * b];
            const uint4 m1 = reinterpret_cast<const uint4*>(const_cast<const uint32_t*>(smax))[2 * b + 1];
            const uint32_t ms = max(max(max(m0.x, m0.y), max(m0.z, m0.w)), max(max(m1.x, m1.y), max(m1.z, m1.w)));
            const int e_state = scale_exp_f32_at(ms, E);
            if (!mbar_wait(dbar + 8 * b, par)) { fail(); ok = false; break; }
            tc_fence_after();
            float d[CPT];
            tmem_ld<CPT>(tmem + tlane + TM_S + CPT * half, d);
            if (eb == E) {                             // the record's B is at the state's scale (always when nothing is scaled)
#pragma unroll
                for (int m = 0; m < CPT / 4; ++m) {
                    const float4 b4 = half4_to_float4(bq[m]);
                    S[4 * m + 0] = fmaf(gamC, S[4 * m + 0], b4.x - d[4 * m + 0]);
                    S[4 * m + 1] = fmaf(gamC, S[4 * m + 1], b4.y - d[4 * m + 1]);
                    S[4 * m + 2] = fmaf(gamC, S[4 * m + 2], b4.z - d[4 * m + 2]);
                    S[4 * m + 3] = fmaf(gamC, S[4 * m + 3], b4.w - d[4 * m + 3]);
                }
            } else {                                   // B is stored divided by 2^eb; S carried divided by 2^E
                const float sb = exp2i(eb - E);
#pragma unroll
                for (int m = 0; m < CPT / 4; ++m) {
                    const float4 b4 = half4_to_float4(bq[m]);
                    S[4 * m + 0] = fmaf(gamC, S[4 * m + 0], fmaf(sb, b4.x, -d[4 * m + 0]));
                    S[4 * m + 1] = fmaf(gamC, S[4 * m + 1], fmaf(sb, b4.y, -d[4 * m + 1]));
                    S[4 * m + 2] = fmaf(gamC, S[4 * m + 2], fmaf(sb, b4.z, -d[4 * m + 2]));
                    S[4 * m + 3] = fmaf(gamC, S[4 * m + 3], fmaf(sb, b4.w, -d[4 * m + 3]));
                }
            }
            // the scale of S_{c+1}: that of the chunk's values or of the state before it, whichever is larger
            const int E_next = max(eb, e_state);
            if (E_next != E) {
                const float r = exp2i(E - E_next);
#pragma unroll
                for (int j = 0; j < CPT; ++j) S[j] *= r;
                E = E_next;
            }
            const int32_t t_done = min(T, (int32_t)(g0 - cseq + ci + 1) * C);   // tokens of the sequence now in S
            if (ci + 1 < n_chunks) {
                // the operand buffer of S_{c+1} was last read by the products of chunk c-1; they were issued
                // before chunk c's state products, whose commit (dbar, waited above) tracks every earlier
                // tensor-core operation of the issuing thread, so they are complete
                write_state_operand(ci + 1, absmax());
                if (tid == 0) {                        // the output warps' copy of E for chunk c+1
                    e_ring[(ci + 1) & 3] = E;
                    mbar_arrive(ebar + 8 * ((ci + 1) & 3));
                }
                fetch_b(ci + 1);
            }
            // a snapshot of the state after this chunk, if due (off the sequential path: after the operand
            // of the next chunk is out; the check is a compare against the next snapshot point)
            if (t_done == snap_next) {
                const int64_t slot = snapshot_slot(p, n, t_done, T);
                if (slot >= 0) {
                    float* dst = p.snapshots + ((slot * H + h) * DK + srow) * (int64_t)p.dv + jc;
                    const float f = exp2i(E);
#pragma unroll
                    for (int x = 0; x < CPT; x += 4)
                        *reinterpret_cast<float4*>(dst + x) = make_float4(f * S[x], f * S[x + 1], f * S[x + 2], f * S[x + 3]);
                }
                snap_next += p.snap_every;
            }
        }
        if (ok && !*s_abort) {
            const float f = exp2i(E);
#pragma unroll
            for (int j = 0; j < CPT; j += 4)
                *reinterpret_cast<float4*>(p.state_out + state_off + j) =
                    make_float4(f * S[j], f * S[j + 1], f * S[j + 2], f * S[j + 3]);
        }
        if (big) atomicOr(p.err, KDA_DEVERR_RANGE);
    }
    tc_fence_before();
    __syncthreads();
    if (warp == 0) {
        tc_fence_after();
        asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem), "r"(128) : "memory");
    }
}

// ============================================================================================
// Backward pass, state-gradient chain from the records of a one-window forward recompute.  The chunk's
// map from its start state to its end state is S -> Diag(Gamma_C) S + B - M S and its output O = Q' S +
// P Utilde, so the gradient of its start state is
//     dS_start = Diag(Gamma_C) dS_end - M^T dS_end + Q'^T dO          (dO = scale * grad_o of the chunk)
// ("Kimi K3, explained", section "Training in chunks": the state alone passes between chunks, here in
// reverse).  One CTA per (head, 32 value columns) walks the chunks from the last to the first; warp w
// owns rows 16 w .. 16 w + 15 of the gradient, in fp32 mma accumulators across chunks, and each chunk is
// one product [-M^T | Q'^T] (16 x 192 per warp) x [dS; dO] (192 x 32) of warp-level m16n8k16 fp16 MMAs:
// M and Q' come fp16 from the record, dS and dO are rounded to fp16 for the operand only (the same
// 10-bit significand as the forward's TF32/fp16 operands).  The next chunk's record and grad_o rows are
// fetched while the current one is used.
// ============================================================================================
constexpr int BR_NT = 256;
constexpr int BR_LD = SNV + 8;                                    // fp16 per operand row (80 B: no bank conflicts)
constexpr int BR_OFF_DS = 2 * (QM_BYTES + 512);                   // two record buffers ([Q'; M] and Gamma_C)
constexpr int BR_OFF_DO = BR_OFF_DS + 2 * DK * BR_LD * 2;         // two -dS operands (128 x 32 fp16)
constexpr int BR_SMEM = BR_OFF_DO + 2 * C * BR_LD * 2;            // two dO operands (64 x 32 fp16)

__device__ __forceinline__ void br_cp16(void* dst, const void* src) {
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16;\n" ::"r"(saddr(dst)), "l"(src) : "memory");
}
__device__ __forceinline__ void ldsm_x4_t(uint32_t addr, uint32_t (&r)[4]) {
    asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0,%1,%2,%3}, [%4];\n"
                 : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3])
                 : "r"(addr));
}
__device__ __forceinline__ void mma_f16_16x8x16(float (&d)[4], const uint32_t (&a)[4], uint32_t b0, uint32_t b1) {
    asm volatile(
        "mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
        "{%0,%1,%2,%3};\n"
        : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
        : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}

template <typename TIn>
__global__ void __launch_bounds__(BR_NT, 1) kda_bwd_dstate_records_kernel(BwdParams p, const unsigned char* records) {
    extern __shared__ __align__(1024) unsigned char sm[];
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int gid = lane >> 2, tig = lane & 3;
    const int H = p.H, h = blockIdx.x / SLICES, j0 = (blockIdx.x % SLICES) * SNV;
    const int32_t T = p.total_tokens;
    if (p.num_seqs != 1 || p.cu_seqlens[0] != 0 || p.cu_seqlens[1] != T) {
        if (tid == 0) atomicOr(p.err, KDA_DEVERR_CU_SEQLENS);
        return;
    }
    const int nch = (T + C - 1) / C;
    const int a0 = 16 * warp;                                     // this warp's gradient rows
    const TIn* gdo = static_cast<const TIn*>(p.d_o);
    auto rec_buf = [&](int b) { return sm + b * (QM_BYTES + 512); };
    __half* dsh = reinterpret_cast<__half*>(sm + BR_OFF_DS);      // [2][128][BR_LD]: -dS, fp16
    __half* doh = reinterpret_cast<__half*>(sm + BR_OFF_DO);      // [2][64][BR_LD]: dO, fp16
    bool big = false;
    // the chunk's [Q'; M] and Gamma_C into buffer b (cp.async), and its grad_o rows into registers: they
    // are stored (scaled, fp16, zero past the sequence end) only after the current chunk's products
    constexpr int DOPT = C * SNV / 2 / BR_NT;                     // column pairs of grad_o per thread
    float dov[DOPT][2];
    auto fetch = [&](int c, int b) {
        const unsigned char* rec = records + ((size_t)c * H + h) * REC_BYTES;
        unsigned char* dst = rec_buf(b);
        for (int e = tid; e < QM_BYTES / 16; e += BR_NT) br_cp16(dst + e * 16, rec + REC_QM + e * 16);
        if (tid < 32) br_cp16(dst + QM_BYTES + tid * 16, rec + REC_G + tid * 16);
        asm volatile("cp.async.commit_group;\n" ::: "memory");
        const int32_t t0 = c * C;
#pragma unroll
        for (int x = 0; x < DOPT; ++x) {
            const int e = tid + x * BR_NT, r = e / (SNV / 2), jj = 2 * (e % (SNV / 2));
            const int64_t at = ((int64_t)(t0 + r) * H + h) * DK + j0 + jj;
            dov[x][0] = t0 + r < T ? load_as_float(gdo, at) : 0.f;
            dov[x][1] = t0 + r < T ? load_as_float(gdo, at + 1) : 0.f;
        }
    };
    auto store_do = [&](int b) {
#pragma unroll
        for (int x = 0; x < DOPT; ++x) {
            const int e = tid + x * BR_NT, r = e / (SNV / 2), jj = 2 * (e % (SNV / 2));
            const float x0 = p.scale * dov[x][0], x1 = p.scale * dov[x][1];
            big |= fmaxf(fabsf(x0), fabsf(x1)) > kF16Max;
            *reinterpret_cast<__half2*>(doh + (b * C + r) * BR_LD + jj) = __floats2half2_rn(x0, x1);
        }
    };
    // accumulator fragment of n-tile nt: rows a0 + gid (+ 8), columns 8 nt + 2 tig (+ 1)
    float acc[4][4];
#pragma unroll
    for (int nt = 0; nt < 4; ++nt)
#pragma unroll
        for (int e = 0; e < 4; ++e) {
            const int a = a0 + gid + 8 * (e >> 1), jj = 8 * nt + 2 * tig + (e & 1);
            acc[nt][e] = p.d_state_out ? p.d_state_out[((int64_t)h * DK + a) * DK + j0 + jj] : 0.f;
        }
    auto put_operand = [&](int b) {                               // -dS in fp16, for the next chunk's product
#pragma unroll
        for (int nt = 0; nt < 4; ++nt)
#pragma unroll
            for (int hr = 0; hr < 2; ++hr) {
                const int a = a0 + gid + 8 * hr, jj = 8 * nt + 2 * tig;
                big |= fmaxf(fabsf(acc[nt][2 * hr]), fabsf(acc[nt][2 * hr + 1])) > kF16Max;
                *reinterpret_cast<__half2*>(dsh + (b * DK + a) * BR_LD + jj) =
                    __floats2half2_rn(-acc[nt][2 * hr], -acc[nt][2 * hr + 1]);
            }
    };
    put_operand(0);
    if (nch > 0) {
        fetch(nch - 1, 0);
        store_do(0);
    }
    int cur = 0;
    for (int c = nch - 1; c >= 0; --c) {
        const int b = (nch - 1 - c) & 1;
        if (c > 0) fetch(c - 1, b ^ 1);
        else asm volatile("cp.async.commit_group;\n" ::: "memory");
        asm volatile("cp.async.wait_group 1;\n" ::: "memory");
        __syncthreads();                                   // chunk c's record and dO, and the -dS operand, are in place
        const unsigned char* qm = rec_buf(b);
        const float* gam = reinterpret_cast<const float*>(qm + QM_BYTES);
        const float g_lo = gam[a0 + gid], g_hi = gam[a0 + gid + 8];
#pragma unroll
        for (int nt = 0; nt < 4; ++nt) {
            acc[nt][0] *= g_lo; acc[nt][1] *= g_lo; acc[nt][2] *= g_hi; acc[nt][3] *= g_hi;
        }
        // A fragment (rows a0.., k0.. of -M^T or Q'^T): ldmatrix.trans of the stored M (rows k, 8 consecutive
        // a per 16 bytes) or Q' (rows r); lanes 8m..8m+7 address the rows of tile m = (k0 + 8 (m >> 1),
        // a0 + 8 (m & 1)), which come out in the fragment's register order.  B fragments (k0.., 8 nt..) of
        // the row-major -dS / dO operands: tiles (k0, 8 nt), (k0 + 8, 8 nt) for two n-tiles per ldmatrix.
        const __half* ds = dsh + cur * DK * BR_LD;
        const __half* dO = doh + b * C * BR_LD;
#pragma unroll
        for (int ks = 0; ks < (DK + C) / 16; ++ks) {
            const bool mpart = ks < DK / 16;
            const int k0 = mpart ? 16 * ks : 16 * (ks - DK / 16);
            uint32_t af[4], b01[4], b23[4];
            ldsm_x4_t(saddr(qm + op_off_h((mpart ? C : 0) + k0 + (lane & 7) + 8 * (lane >> 4),
                                          a0 + 8 * ((lane >> 3) & 1), DK)), af);
            const __half* brow = (mpart ? ds : dO) + (k0 + (lane & 7) + 8 * ((lane >> 3) & 1)) * BR_LD + 8 * (lane >> 4);
            ldsm_x4_t(saddr(brow), b01);                   // n-tiles 0 and 1
            ldsm_x4_t(saddr(brow + 16), b23);              // n-tiles 2 and 3
            mma_f16_16x8x16(acc[0], af, b01[0], b01[1]);
            mma_f16_16x8x16(acc[1], af, b01[2], b01[3]);
            mma_f16_16x8x16(acc[2], af, b23[0], b23[1]);
            mma_f16_16x8x16(acc[3], af, b23[2], b23[3]);
        }
        put_operand(cur ^ 1);
        if (c > 0) store_do(b ^ 1);                        // chunk c - 1's grad_o, loaded during the products
        // the gradient of the state after chunk c - 1 (the snapshot slot of that boundary)
        if (c > 0) {
            float* dst = p.dstate_b + (((int64_t)(p.snap_offsets[0] + c - 1) * H + h) * DK) * DK + j0;
#pragma unroll
            for (int nt = 0; nt < 4; ++nt)
#pragma unroll
                for (int hr = 0; hr < 2; ++hr)
                    *reinterpret_cast<float2*>(dst + (int64_t)(a0 + gid + 8 * hr) * DK + 8 * nt + 2 * tig) =
                        make_float2(acc[nt][2 * hr], acc[nt][2 * hr + 1]);
        }
        cur ^= 1;
        __syncthreads();                                   // buffers b and the old operand are free
    }
    if (p.d_state_in) {
#pragma unroll
        for (int nt = 0; nt < 4; ++nt)
#pragma unroll
            for (int hr = 0; hr < 2; ++hr)
                *reinterpret_cast<float2*>(p.d_state_in + ((int64_t)h * DK + a0 + gid + 8 * hr) * DK + j0 + 8 * nt + 2 * tig) =
                    make_float2(acc[nt][2 * hr], acc[nt][2 * hr + 1]);
    }
    if (big) atomicOr(p.err, KDA_DEVERR_RANGE);
    asm volatile("cp.async.wait_group 0;\n" ::: "memory");
}

int64_t buffer_chunks(int32_t H) {                   // chunks of records one overlap buffer holds
    const int64_t w = (int64_t)(kBufBudget / ((size_t)H * REC_BYTES));
    return w < 1 ? 1 : w;
}

// Side stream and events of the overlapped schedule, created once per device and kept for the life of
// the process.
struct SideStream {
    cudaStream_t stream = nullptr;
    cudaEvent_t fork = nullptr, prep_done[2] = {nullptr, nullptr}, chain_done[2] = {nullptr, nullptr};
};
constexpr int kMaxDevices = 64;
std::mutex g_side_mutex;
SideStream g_side[kMaxDevices];
std::mutex g_enqueue_mutex[kMaxDevices];

cudaError_t side_stream(int dev, SideStream** out) {
    if (dev < 0 || dev >= kMaxDevices) return cudaErrorInvalidDevice;
    std::lock_guard<std::mutex> lock(g_side_mutex);
    SideStream& ss = g_side[dev];
    if (!ss.stream) {
        SideStream t;
        cudaError_t e = cudaStreamCreateWithFlags(&t.stream, cudaStreamNonBlocking);
        if (e != cudaSuccess) return e;
        cudaEvent_t* evs[5] = {&t.fork, &t.prep_done[0], &t.prep_done[1], &t.chain_done[0], &t.chain_done[1]};
        for (cudaEvent_t* ev : evs)
            if ((e = cudaEventCreateWithFlags(ev, cudaEventDisableTiming)) != cudaSuccess) return e;
        ss = t;
    }
    *out = &ss;
    return cudaSuccess;
}

}  // namespace

bool prefill_2p_supported(int32_t num_seqs, int64_t total_tokens, int32_t H, int32_t d_k, int32_t d_v,
                          kda_dtype dt) {
    return num_seqs >= 1 && total_tokens > 0 && dt == KDA_DTYPE_BF16 && d_k == DK && d_v == DK && H > 0;
}

// Workspace of the two-phase path: with several sequences, their chunk offsets (N + 1 int32) and their
// longest-first order (N int32), each 256-byte aligned; then the records of one window (or of two).
static size_t align256(size_t x) { return (x + 255) / 256 * 256; }
size_t prefill_2p_header(int32_t num_seqs) {
    return num_seqs > 1 ? align256(4 * ((size_t)num_seqs + 1)) + align256(4 * (size_t)num_seqs) : 0;
}
int64_t prefill_2p_max_chunks(int32_t num_seqs, int64_t total_tokens) {   // chunks of all sequences, at most
    return num_seqs > 1 ? total_tokens / C + num_seqs : (total_tokens + C - 1) / C;
}

size_t prefill_2p_min_workspace(int32_t num_seqs, int32_t H) {
    return prefill_2p_header(num_seqs) + (size_t)H * REC_BYTES;
}

size_t prefill_2p_workspace(int32_t num_seqs, int64_t total_tokens, int32_t H, size_t record_budget) {
    const int64_t chunks = prefill_2p_max_chunks(num_seqs, total_tokens);
    if (record_budget == 0) record_budget = num_seqs > 1 ? kMultiWindowBudget : kOneWindowBudget;
    int64_t cap = (int64_t)(record_budget / ((size_t)H * REC_BYTES));
    if (num_seqs == 1 && cap < 2 * buffer_chunks(H)) cap = 2 * buffer_chunks(H);
    return prefill_2p_header(num_seqs) + (size_t)(chunks < cap ? chunks : cap) * H * REC_BYTES;
}

// Value columns per chain CTA: 16 for one sequence whose 16-column chain still leaves half the SMs to phase 1
// (few heads: there the chain's per-chunk latency sets the time, and half the columns halve the state warps'
// update and operand write), otherwise 32.
static int chain_columns(int32_t num_seqs, int32_t H, int sms) {
    return num_seqs == 1 && 2 * H * (DK / 16) <= sms ? 16 : 32;
}

WindowPlan prefill_2p_plan(int32_t num_seqs, int64_t chunks, int32_t H, size_t workspace_bytes, int sms) {
    const size_t hdr = prefill_2p_header(num_seqs);
    const int64_t cap = workspace_bytes > hdr ? (int64_t)((workspace_bytes - hdr) / ((size_t)H * REC_BYTES)) : 0;
    const int64_t one = buffer_chunks(H);
    const bool overlap_ok = num_seqs == 1 && 2 * H * SLICES <= sms;   // the chain leaves half the SMs to phase 1
    WindowPlan w;
    if (overlap_ok && chunks > one && cap >= 2) {
        // one sequence, few heads: phase 1 of the next window runs beside the chain of this one, on double
        // buffers
        w.window = cap / 2 < one ? cap / 2 : one; w.buffers = 2;
    } else {
        // otherwise the windows run back to back, as few as fit
        w.window = chunks < cap ? chunks : cap; w.buffers = 1;
    }
    if (w.window < 1) w.window = 1;
    return w;
}

// Phase 1 of window w+1 runs on a side stream while phase 2 of window w runs on the caller's stream,
// with the records double-buffered, when the chain leaves SMs free (few heads); otherwise the windows
// run back to back on the caller's stream.  Ordering is by events only, and every side-stream launch is
// joined back into the caller's stream before the call returns.
cudaError_t launch_prefill_2p(const PrefillParams& p, void* workspace, size_t workspace_bytes, cudaStream_t s) {
    auto enc = tensor_map_encoder();
    if (!enc) return cudaErrorNotSupported;
    PrepMaps maps;
    std::memset(&maps, 0, sizeof maps);
    const int T = p.total_tokens;
    if (!encode_rows(enc, &maps.k, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, p.k, 2, DK, p.H, T, 64, CU_TENSOR_MAP_SWIZZLE_128B) ||
        !encode_rows(enc, &maps.q, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, p.q, 2, DK, p.H, T, 64, CU_TENSOR_MAP_SWIZZLE_128B) ||
        (p.alpha_mode == KDA_ALPHA_PER_CHANNEL &&
         !encode_rows(enc, &maps.a, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, p.alpha, 4, DK, p.H, T, 32,
                      CU_TENSOR_MAP_SWIZZLE_128B)) ||
        !encode_rows(enc, &maps.v, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, p.v, 2, p.dv, p.H, T, DK, CU_TENSOR_MAP_SWIZZLE_NONE))
        return cudaErrorInvalidValue;
    const bool multi = p.num_seqs > 1;
    cudaError_t e = cudaFuncSetAttribute(multi ? kda_prefill_prep_kernel<true> : kda_prefill_prep_kernel<false>,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize, P_SMEM);
    if (e != cudaSuccess) return e;
    int dev = 0, sms = 0;
    if ((e = cudaGetDevice(&dev)) != cudaSuccess) return e;
    if ((e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev)) != cudaSuccess) return e;
    const int nv = chain_columns(p.num_seqs, p.H, sms);
    e = cudaFuncSetAttribute(multi ? kda_prefill_chain_kernel<true, 32>
                                   : (nv == 16 ? kda_prefill_chain_kernel<false, 16> : kda_prefill_chain_kernel<false, 32>),
                             cudaFuncAttributeMaxDynamicSharedMemorySize, C_SMEM);
    if (e != cudaSuccess) return e;
    const int N = p.num_seqs;
    const size_t hdr = prefill_2p_header(N);
    const int64_t chunks = prefill_2p_max_chunks(N, T);
    const WindowPlan plan = prefill_2p_plan(N, chunks, p.H, workspace_bytes, sms);
    const size_t buf_bytes = (size_t)plan.window * p.H * REC_BYTES;
    if (hdr + buf_bytes * plan.buffers > workspace_bytes) return cudaErrorInvalidValue;
    // several sequences: their chunk offsets and their longest-first order head the workspace
    int32_t* choff = nullptr;
    int32_t* order = nullptr;
    if (N > 1) {
        choff = static_cast<int32_t*>(workspace);
        order = reinterpret_cast<int32_t*>(static_cast<unsigned char*>(workspace) + align256(4 * ((size_t)N + 1)));
        kda_chunk_offsets_kernel<<<1, 32, 0, s>>>(p.cu_seqlens, N, T, choff, p.err);
        if ((e = cudaGetLastError()) != cudaSuccess) return e;
        if ((e = launch_order(p.cu_seqlens, N, order, s)) != cudaSuccess) return e;
    }
    const int chain_ctas = N * p.H * (DK / nv);
    SideStream* ss = nullptr;
    std::unique_lock<std::mutex> enqueue;             // concurrent callers must not interleave event records
    if (plan.buffers == 2) {
        if ((e = side_stream(dev, &ss)) != cudaSuccess) return e;
        enqueue = std::unique_lock<std::mutex>(g_enqueue_mutex[dev]);
        if ((e = cudaEventRecord(ss->fork, s)) != cudaSuccess) return e;
        if ((e = cudaStreamWaitEvent(ss->stream, ss->fork, 0)) != cudaSuccess) return e;
    }
    int w = 0;
    for (int64_t c0 = 0; c0 < chunks; c0 += plan.window, ++w) {
        const int64_t n = chunks - c0 < plan.window ? chunks - c0 : plan.window;
        const int units = (int)(n * p.H);
        const int buf = w % plan.buffers;
        unsigned char* rec = static_cast<unsigned char*>(workspace) + hdr + buf * buf_bytes;
        cudaStream_t ps = ss ? ss->stream : s;
        // phase 1 shares the GPU with the previous window's chain when overlapped
        int grid = (ss && w > 0) ? sms - chain_ctas : sms;
        if (grid > units) grid = units;
        if (ss && w >= 2 && (e = cudaStreamWaitEvent(ps, ss->chain_done[buf], 0)) != cudaSuccess) return e;
        if (multi)
            kda_prefill_prep_kernel<true><<<(unsigned)grid, NT, P_SMEM, ps>>>(p, maps, rec, (int)c0, units, choff);
        else
            kda_prefill_prep_kernel<false><<<(unsigned)grid, NT, P_SMEM, ps>>>(p, maps, rec, (int)c0, units, nullptr);
        if ((e = cudaGetLastError()) != cudaSuccess) return e;
        if (ss) {
            if ((e = cudaEventRecord(ss->prep_done[buf], ps)) != cudaSuccess) return e;
            if ((e = cudaStreamWaitEvent(s, ss->prep_done[buf], 0)) != cudaSuccess) return e;
        }
        // on one stream the chain is phase 1's programmatic dependent: its launch and prologue overlap phase
        // 1's last units (it waits for phase 1's completion before its first record read)
        cudaLaunchConfig_t cfg = {};
        cfg.gridDim = dim3((unsigned)chain_ctas);
        cfg.blockDim = dim3(C_NT);
        cfg.dynamicSmemBytes = C_SMEM;
        cfg.stream = s;
        cudaLaunchAttribute attr[1];
        attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
        attr[0].val.programmaticStreamSerializationAllowed = 1;
        cfg.attrs = attr;
        cfg.numAttrs = ss ? 0 : 1;
        const unsigned char* crec = rec;
        const int cb = (int)c0, cn = (int)n;
        if (multi)
            e = cudaLaunchKernelEx(&cfg, kda_prefill_chain_kernel<true, 32>, p, crec, cb, cn,
                                   static_cast<const int32_t*>(choff), static_cast<const int32_t*>(order));
        else if (nv == 16)
            e = cudaLaunchKernelEx(&cfg, kda_prefill_chain_kernel<false, 16>, p, crec, cb, cn,
                                   static_cast<const int32_t*>(nullptr), static_cast<const int32_t*>(nullptr));
        else
            e = cudaLaunchKernelEx(&cfg, kda_prefill_chain_kernel<false, 32>, p, crec, cb, cn,
                                   static_cast<const int32_t*>(nullptr), static_cast<const int32_t*>(nullptr));
        if (e != cudaSuccess) return e;
        if ((e = cudaGetLastError()) != cudaSuccess) return e;
        if (ss && (e = cudaEventRecord(ss->chain_done[buf], s)) != cudaSuccess) return e;
    }
    return cudaSuccess;
}

cudaError_t launch_bwd_dstate_records(const BwdParams& p, kda_dtype dt, const unsigned char* records, cudaStream_t s) {
    const unsigned grid = (unsigned)(p.H * SLICES);
    cudaError_t e;
    if (dt == KDA_DTYPE_BF16) {
        e = cudaFuncSetAttribute(kda_bwd_dstate_records_kernel<__nv_bfloat16>,
                                 cudaFuncAttributeMaxDynamicSharedMemorySize, BR_SMEM);
        if (e != cudaSuccess) return e;
        kda_bwd_dstate_records_kernel<__nv_bfloat16><<<grid, BR_NT, BR_SMEM, s>>>(p, records);
    } else {
        e = cudaFuncSetAttribute(kda_bwd_dstate_records_kernel<float>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 BR_SMEM);
        if (e != cudaSuccess) return e;
        kda_bwd_dstate_records_kernel<float><<<grid, BR_NT, BR_SMEM, s>>>(p, records);
    }
    return cudaGetLastError();
}

}  // namespace kda
