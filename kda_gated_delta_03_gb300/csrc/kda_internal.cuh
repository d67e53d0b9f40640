// Internal interfaces between the C-ABI host code (kda_api.cu) and the kernels.
#pragma once

#include <cuda_runtime.h>
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cstdint>

#include "kda.h"

namespace kda {

constexpr int kChunk = 64;             // tokens per chunk of the chunkwise prefill
constexpr float kLog2AlphaMin = -15.f; // clamp of log2(alpha) per token

// Everything a prefill kernel needs, already validated on the host.
struct PrefillParams {
    const void* q;
    const void* k;
    const void* v;
    const float* beta;
    const float* alpha;
    const int32_t* cu_seqlens;   // [num_seqs + 1], device
    const int32_t* order;        // [num_seqs] sequences longest first (device), or nullptr
    int32_t num_seqs;
    int32_t total_tokens;
    int32_t H;
    int32_t dk;
    int32_t dv;
    int32_t slices;              // d_v slices per (sequence, head)
    float scale;
    const float* state_in;       // may be nullptr
    float* state_out;
    void* o;
    unsigned* err;               // device error word
    int32_t alpha_mode;          // KDA_ALPHA_PER_CHANNEL [T,H,dk], KDA_ALPHA_PER_HEAD [T,H], KDA_ALPHA_NONE
    // optional state snapshots: the state after every snap_every tokens of each sequence
    int32_t snap_every;          // tokens (a multiple of kChunk), 0 = none
    float* snapshots;            // [snap_offsets[num_seqs], H, dk, dv]
    const int32_t* snap_offsets; // device [num_seqs + 1]
#ifdef KDA_TEST_HOOKS
    int32_t test_stall;          // test builds only: make the tcgen05 prefill kernels' bounded waits give up
#endif
};

struct DecodeParams {
    const void* q;
    const void* k;
    const void* v;
    const float* beta;
    const float* alpha;
    void* state;                 // float, or bf16 when state_bf16
    bool state_bf16;
    int32_t alpha_mode;          // as in PrefillParams
    const int32_t* state_idx;    // may be nullptr
    int32_t num_slots;
    void* o;
    int32_t B;
    int32_t H;
    int32_t d;
    float scale;
    unsigned* err;
};

// Everything the backward kernel needs (per-channel alpha), already validated on the host.
struct BwdParams {
    const void* q;
    const void* k;
    const void* v;
    const float* beta;
    const float* alpha;
    const int32_t* cu_seqlens;
    int32_t num_seqs;
    int32_t total_tokens;
    int32_t H;
    int32_t dk;
    int32_t dv;
    float scale;
    const float* state_in;       // may be nullptr
    const void* d_o;
    const float* d_state_out;    // may be nullptr
    void* d_q;
    void* d_k;
    void* d_v;
    float* d_beta;
    float* d_alpha;
    float* d_state_in;           // may be nullptr
    const float* snapshots;      // forward state after every 64 tokens of each sequence
    const int32_t* snap_offsets; // [num_seqs + 1]: first snapshot slot of each sequence
    const int32_t* chunk_offsets;// [num_seqs + 1]: first chunk unit of each sequence
    float* dstate_b;             // gradient of the state after every 64 tokens (snapshot slots)
    float* scratch;              // per CTA: 63 states of the chunk being walked back
    const unsigned char* records;// the one-window forward recompute's per-chunk records, or nullptr
    unsigned* err;
};
constexpr int kBwdMaxCtas = 160;   // chunk-pass CTAs (one per SM)
// Pass 3 at d = 128 in matrix form (kda_backward_mat.cu), one CTA per SM, each with this much scratch
// (ten 64 x 128 fp32 matrices; the token walk at d = 16, 64 takes 63 states per CTA instead).
constexpr size_t kBwdMatScratchBytes = (size_t)10 * 64 * 128 * 4;
cudaError_t launch_bwd_chunk_mat(const BwdParams& p, kda_dtype dt, int grid, cudaStream_t s);

// Launchers (return the launch error, if any).
cudaError_t launch_decode(const DecodeParams& p, kda_dtype dt, cudaStream_t s);
// The bf16-stored state at d = 128 (kda_decode_bf16s.cu): a persistent kernel streaming the states.
cudaError_t launch_decode_bf16s_stream(const DecodeParams& p, kda_dtype dt, cudaStream_t s);
cudaError_t launch_prefill_cc(const PrefillParams& p, kda_dtype dt, cudaStream_t s);
cudaError_t launch_prefill_tc(const PrefillParams& p, cudaStream_t s);
bool prefill_tc_supported(const PrefillParams& p, kda_dtype dt);
int prefill_tc_slices(int32_t num_seqs, int32_t H, int32_t dv);
// Two-phase prefill (bf16, d_k = d_v = 128): per-chunk records in the workspace, then the state chain.
bool prefill_2p_supported(int32_t num_seqs, int64_t total_tokens, int32_t H, int32_t d_k, int32_t d_v,
                          kda_dtype dt);
// recommended bytes; record_budget caps the records (0: 1 GiB for one sequence, 16 GiB for several)
size_t prefill_2p_workspace(int32_t num_seqs, int64_t total_tokens, int32_t H, size_t record_budget = 0);
struct WindowPlan {
    int64_t window;   // chunks per window
    int buffers;      // 2: phase 1 of the next window overlaps phase 2 of this one (side stream)
};
int64_t prefill_2p_max_chunks(int32_t num_seqs, int64_t total_tokens);
WindowPlan prefill_2p_plan(int32_t num_seqs, int64_t chunks, int32_t H, size_t workspace_bytes, int sms);
size_t prefill_2p_min_workspace(int32_t num_seqs, int32_t H);   // bytes for one chunk per window
cudaError_t launch_prefill_2p(const PrefillParams& p, void* workspace, size_t workspace_bytes, cudaStream_t s);
cudaError_t launch_order(const int32_t* cu_seqlens, int32_t num_seqs, int32_t* order, cudaStream_t s);
cudaError_t launch_bwd_offsets(const int32_t* cu, int32_t N, int32_t T, int32_t* off, int32_t* choff, unsigned* err,
                               cudaStream_t s);
cudaError_t launch_prefill_bwd(const BwdParams& p, kda_dtype dt, int grid, cudaStream_t s);
cudaError_t launch_bwd_dstate_records(const BwdParams& p, kda_dtype dt, const unsigned char* records, cudaStream_t s);

// Number of CUDA-core prefill d_v slices for a head size.
int prefill_cc_slices(int dv);

// Whether snap_offsets fails to give sequence n (length len) floor(len / snap_every) slots.
__device__ __forceinline__ bool snapshot_offsets_bad(const PrefillParams& p, int n, int32_t len) {
    if (p.snap_every <= 0) return false;
    const int32_t base = p.snap_offsets[n], cnt = p.snap_offsets[n + 1] - base;
    return base < 0 || cnt != len / p.snap_every;
}

// Snapshot slot of the state after token t_rel (counted from the start of sequence n, whose length is
// len), -1 if that point takes none, -2 if snap_offsets is inconsistent for sequence n (nothing is
// written; snapshot_offsets_bad reports it).
__device__ __forceinline__ int64_t snapshot_slot(const PrefillParams& p, int n, int32_t t_rel, int32_t len) {
    if (p.snap_every <= 0 || t_rel <= 0 || t_rel % p.snap_every != 0) return -1;
    const int32_t base = p.snap_offsets[n], cnt = p.snap_offsets[n + 1] - base;
    if (base < 0 || cnt != len / p.snap_every) return -2;
    return (int64_t)base + t_rel / p.snap_every - 1;
}

// The decay of key channel i at token-head row `row` (= t * H + h) under the given alpha layout.
__device__ __forceinline__ float alpha_at(const float* alpha, int mode, int64_t row, int dk, int i) {
    return mode == KDA_ALPHA_PER_CHANNEL ? alpha[row * dk + i] : mode == KDA_ALPHA_PER_HEAD ? alpha[row] : 1.f;
}

__device__ __forceinline__ float to_float(float x) { return x; }
__device__ __forceinline__ float to_float(__nv_bfloat16 x) { return __bfloat162float(x); }

__device__ __forceinline__ float load_as_float(const float* p, int64_t i) { return p[i]; }
__device__ __forceinline__ float load_as_float(const __nv_bfloat16* p, int64_t i) {
    return __bfloat162float(p[i]);
}
__device__ __forceinline__ void store_from_float(float* p, int64_t i, float x) { p[i] = x; }
__device__ __forceinline__ void store_from_float(__nv_bfloat16* p, int64_t i, float x) {
    p[i] = __float2bfloat16_rn(x);
}

}  // namespace kda
