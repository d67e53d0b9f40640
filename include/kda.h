/*
 * kda.h -- C ABI of libkda, a single-GPU (sm_103a) implementation of the Kimi
 * Delta Attention (KDA) operator.
 *
 * The operator ("Kimi K3, explained", section "The math", and section "How
 * Kimi Delta Attention works, step by step"): per head a fixed state S is
 * decayed channel by channel, the delta rule erases what S returns for the key
 * and writes the new value, and the query reads the result.  The page writes S
 * as d_v x d_k with o_t = S_t q_t; this library stores the transpose,
 * S[d_k][d_v] (d_v contiguous), so that
 *
 *     S_t = (I - beta_t k_t k_t^T) Diag(alpha_t) S_{t-1} + beta_t k_t v_t^T
 *     o_t = scale * S_t^T q_t
 *
 * which is the same operator.  alpha_t in (0,1]^{d_k} is the per-channel decay
 * (one value per key channel, which is what KDA adds over Gated DeltaNet),
 * beta_t in [0,1] the write strength.  q and k are expected L2-normalised by the
 * caller; the library does not renormalise.
 *
 * Conventions for every entry point:
 *  - All tensor pointers are DEVICE pointers to contiguous row-major arrays,
 *    owned by the caller.  The library never allocates, frees or retains them,
 *    and keeps no state between calls except one 32-bit error word per device
 *    (a static device variable, see kda_get_device_error).
 *  - Work is enqueued asynchronously on `stream` (a cudaStream_t; NULL = the
 *    legacy default stream) on the current device.  Arguments are validated on
 *    the host before anything is launched; a validation failure launches
 *    nothing and returns the status.  Conditions only visible on the device
 *    (inconsistent cu_seqlens contents, out-of-range state slots) make the
 *    kernels skip the affected work and set bits of the device error word.
 *  - Alignment: q, k, v, o, alpha, states 16 bytes; beta, cu_seqlens,
 *    state_idx 4 bytes; workspace 256 bytes.
 *  - dtype (kda_dtype) applies to q, k, v and o.  beta, alpha and the states
 *    are always float32.
 *  - Supported sizes: d_k == d_v in {16, 64, 128}.  Other sizes return
 *    KDA_ERR_UNSUPPORTED.
 *  - Numerics: log2(alpha) is clamped below at -15 per token (alpha >= 2^-15
 *    ~= 3.1e-5 per token and channel); smaller alphas, including alpha = 0,
 *    decay as if alpha were 2^-15.  Intermediates are float32 (bf16 tensor-core
 *    operands only for the raw bf16 q, k, v).
 */
#ifndef KDA_H
#define KDA_H

#include <stddef.h>
#include <stdint.h>

#if defined(__GNUC__)
#define KDA_API __attribute__((visibility("default")))
#else
#define KDA_API
#endif

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
    KDA_OK = 0,
    KDA_ERR_INVALID_ARG = 1,  /* null/misaligned pointer, negative size, bad scale        */
    KDA_ERR_UNSUPPORTED = 2,  /* head size or dtype this build has no kernel for           */
    KDA_ERR_WORKSPACE = 3,    /* workspace missing or smaller than the required size       */
    KDA_ERR_CUDA = 4,         /* a CUDA runtime call or launch failed                      */
    KDA_ERR_DEVICE = 5,       /* kda_get_device_error found device-detected errors         */
    KDA_ERR_TOO_LARGE = 6     /* problem exceeds the fixed scratch of kda_prefill_noalloc  */
} kda_status;

typedef enum { KDA_DTYPE_F32 = 0, KDA_DTYPE_BF16 = 1 } kda_dtype;

/*
 * Layout of alpha (the forget gate).  "Kimi K3, explained", section "The math":
 * with every alpha equal to 1 the update is DeltaNet's delta rule, with one
 * alpha per head it is Gated DeltaNet, and KDA gives every key channel its own.
 */
typedef enum {
    KDA_ALPHA_PER_CHANNEL = 0,  /* KDA: alpha [tokens, H, d_k] float32, 16-byte aligned       */
    KDA_ALPHA_PER_HEAD = 1,     /* Gated DeltaNet: alpha [tokens, H] float32, 4-byte aligned */
    KDA_ALPHA_NONE = 2          /* DeltaNet: no decay; alpha is not read and may be NULL     */
} kda_alpha_mode;

/* Bits of the device error word. */
#define KDA_DEVERR_CU_SEQLENS 0x1u  /* cu_seqlens not monotone / cu[0] != 0 / cu[N] != total  */
#define KDA_DEVERR_STATE_IDX 0x2u   /* decode state_idx entry outside [0, num_slots)          */
#define KDA_DEVERR_TIMEOUT 0x4u     /* a bounded wait inside a kernel gave up (work abandoned) */
#define KDA_DEVERR_SNAPSHOTS 0x8u   /* snapshot_offsets disagree with the sequence lengths       */
#define KDA_DEVERR_RANGE 0x10u      /* one-sequence bf16 d=128 prefill: a key-side chunk product
                                       (Q', M, T' below) beyond fp16's range (|x| > 65504), which
                                       needs keys far from unit norm; results invalid */

/*
 * Bytes of device workspace kda_prefill needs for this problem (0 is a valid
 * answer).  Pure host function; never fails (returns 0 for invalid sizes).
 *  - bf16 with d_k = d_v = 128 (the two-phase path): the per-chunk records
 *    (99,072 bytes per chunk and head; up to 1 GiB of them for one sequence,
 *    up to 16 GiB for several, so that all chunks of a batch of sequences fit
 *    one window), preceded, for several sequences, by their chunk offsets and
 *    their longest-first order (4 (N + 1) and 4 N bytes, each rounded up to
 *    256).  kda_prefill also accepts less, down to one chunk's records after
 *    those offsets; it then walks the chunks in more windows, with identical
 *    results.
 *  - Other several-sequence calls: the longest-first schedule, 4 bytes per
 *    sequence.
 */
KDA_API size_t kda_prefill_workspace_size(int32_t num_seqs, int64_t total_tokens, int32_t H, int32_t d_k,
                                  int32_t d_v, kda_dtype dt);

/*
 * Number of kernel launches a kda_prefill call with these arguments makes on the
 * current device (diagnostics: launch budgets, profiler capture ranges), or -1
 * for arguments kda_prefill would reject on the host.  The two-phase path makes
 * two launches per window of chunks (plus two for the chunk offsets and the
 * order of several sequences), and its window count depends on
 * workspace_bytes and on the device's SM count.  Calls cudaGetDevice and
 * cudaDeviceGetAttribute; enqueues nothing.
 */
KDA_API int64_t kda_prefill_launch_count(int32_t num_seqs, int64_t total_tokens, int32_t H, int32_t d_k,
                                         int32_t d_v, kda_dtype dt, size_t workspace_bytes);

/*
 * Chunkwise-parallel prefill over packed variable-length sequences, with state
 * in and state out ("Kimi K3, explained", section "Training in chunks": the
 * sequence is split into chunks, the per-token decay-and-erase products inside
 * a chunk are rewritten in WY form so most of the work becomes matrix
 * products, and only the state is carried from chunk to chunk).  Results equal
 * the token-by-token recurrence above up to rounding.  Append-prefill (the
 * agentic workload of the hex-index review, where new context continues a long
 * history) is this call with state_in set to an earlier call's state_out.
 *
 *   q, k        [total_tokens, H, d_k]  dtype dt
 *   v           [total_tokens, H, d_v]  dtype dt
 *   beta        [total_tokens, H]       float32, write strength in [0,1]
 *   alpha       [total_tokens, H, d_k]  float32, per-channel decay in (0,1]
 *   cu_seqlens  [num_seqs + 1]          int32 device array, cu[0] = 0,
 *               non-decreasing, cu[num_seqs] = total_tokens; sequence n owns
 *               tokens [cu[n], cu[n+1]).  Zero-length sequences are allowed:
 *               their state_out is their state_in (or zero).
 *   state_in    [num_seqs, H, d_k, d_v] float32, or NULL for zero states
 *   state_out   [num_seqs, H, d_k, d_v] float32 (may equal state_in, in place)
 *   o           [total_tokens, H, d_v]  dtype dt, o_t = scale * S_t^T q_t
 *   workspace   device scratch of at least kda_prefill_workspace_size(...)
 *               bytes (may be NULL when that size is 0); contents need not be
 *               initialised and are clobbered.
 * Returns KDA_OK once the work is enqueued.  Bad cu_seqlens contents are
 * reported through the device error word (KDA_DEVERR_CU_SEQLENS); the
 * sequences they affect are skipped.
 */
KDA_API kda_status kda_prefill(const void* q, const void* k, const void* v, const float* beta,
                       const float* alpha, const int32_t* cu_seqlens, int32_t num_seqs,
                       int64_t total_tokens, int32_t H, int32_t d_k, int32_t d_v, kda_dtype dt,
                       float scale, const float* state_in, float* state_out, void* o,
                       void* workspace, size_t workspace_bytes, void* stream);

/*
 * Options of kda_prefill_ex.  Zero-initialise and set what is used.
 *
 * alpha_mode selects the layout of `alpha` (kda_alpha_mode): per key channel
 * (KDA, the default), one value per token and head (Gated DeltaNet: 4 bytes per
 * token-head instead of 4 * d_k), or none (DeltaNet).
 *
 * State snapshots ("Kimi K3 changed the memory math for agentic AI forever",
 * section "But KDA State Is Not Additive": the recurrent state depends on the
 * whole prefix, so restartable checkpoints and prefix reuse keep copies of it
 * at fixed token intervals): with snapshot_every > 0, the state of sequence n after its
 * first (m + 1) * snapshot_every tokens is written to
 * snapshots[snapshot_offsets[n] + m] for m = 0 .. floor(len_n /
 * snapshot_every) - 1 (a snapshot at len_n equals that sequence's
 * state_out).
 *
 * single_kernel (nonzero): bf16 sequences with d_k = d_v = 128 run the
 * single-kernel tensor-core path (TF32 / bf16 operands, one CTA per sequence,
 * head and value slice; the workspace then needs only the longest-first order
 * of several sequences) instead of the two-phase path, whose per-chunk records
 * and state operand are fp16.  The
 * two-phase path keeps values and states of any magnitude inside fp16's range
 * with exact power-of-two scales (per chunk for v, per chunk and slice for the
 * state); only key-side products far outside O(1), which need keys far from
 * unit norm, set KDA_DEVERR_RANGE, and this option is then the way out.  Results
 * agree to the same tolerance; the two-phase path is faster.
 *   snapshot_every    tokens between snapshots: 0, or a positive multiple of 64
 *   snapshots         [snapshot_offsets[num_seqs], H, d_k, d_v] float32 device
 *                     buffer, 16-byte aligned
 *   snapshot_offsets  [num_seqs + 1] int32 device array, non-decreasing, with
 *                     snapshot_offsets[n + 1] - snapshot_offsets[n] =
 *                     floor(len_n / snapshot_every); a sequence whose count
 *                     disagrees gets no snapshots and sets
 *                     KDA_DEVERR_SNAPSHOTS.
 */
typedef struct kda_prefill_options {
    int32_t snapshot_every;
    float* snapshots;
    const int32_t* snapshot_offsets;
    int32_t alpha_mode;             /* kda_alpha_mode; 0 = KDA_ALPHA_PER_CHANNEL */
    int32_t single_kernel;          /* nonzero: see below */
} kda_prefill_options;

/*
 * kda_prefill with options (NULL options = kda_prefill).  Snapshots add only
 * their own writes (64 KiB per snapshot and head at d = 128); outputs and
 * state_out are those of kda_prefill.
 */
KDA_API kda_status kda_prefill_ex(const void* q, const void* k, const void* v, const float* beta,
                          const float* alpha, const int32_t* cu_seqlens, int32_t num_seqs,
                          int64_t total_tokens, int32_t H, int32_t d_k, int32_t d_v, kda_dtype dt,
                          float scale, const float* state_in, float* state_out, void* o,
                          void* workspace, size_t workspace_bytes, void* stream,
                          const kda_prefill_options* options);

/*
 * Backward pass of kda_prefill (per-channel alpha): given the gradients grad_o
 * of the outputs and grad_state_out of the final states (NULL = zero),
 * computes the gradients of q, k, v, beta, alpha and state_in for the loss
 * sum(o * grad_o) + sum(state_out * grad_state_out).  It is the reverse mode of
 * the token recurrence ("Kimi K3, explained", section "The math"), in three
 * passes: a forward recompute that stores the state at every 64-token
 * boundary; a reverse chain that carries only the state gradient and stores it
 * at the same boundaries (for one bf16 d=128 sequence whose recompute fits one
 * window of records, chunk by chunk from those records: dS_start =
 * Diag(Gamma_C) dS_end - M^T dS_end + Q'^T dO; otherwise token by token); and a
 * chunk-parallel pass that, per (sequence, 64-token chunk, head), takes every
 * gradient of the chunk from its start state and its end-state gradient: at
 * d = 128 in matrix form, the chunk's products of "Training in chunks" run in
 * reverse (on TF32 tensor cores for bf16 inputs, in fp32 for fp32 inputs), at
 * d = 16 and 64 by replaying the chunk and walking it back token by token.
 * Arguments are kda_prefill's, plus:
 *   grad_o          [total_tokens, H, d_v] dtype dt
 *   grad_state_out  [num_seqs, H, d_k, d_v] float32, or NULL
 *   grad_q, grad_k  [total_tokens, H, d_k] dtype dt;  grad_v [total_tokens, H, d_v]
 *   grad_beta       [total_tokens, H] float32;  grad_alpha [total_tokens, H, d_k]
 *   grad_state_in   [num_seqs, H, d_k, d_v] float32, or NULL (not computed)
 *   workspace       at least kda_prefill_backward_workspace_size(...) bytes
 * The decay clamp of the forward (log2 alpha >= -15 per token) is not
 * differentiated: the d = 16 and 64 walk uses alpha as given, the d = 128
 * chunk form the clamped decays inside a chunk (as the forward does), and
 * both give the gradient of alpha itself.
 */
KDA_API size_t kda_prefill_backward_workspace_size(int32_t num_seqs, int64_t total_tokens, int32_t H,
                                           int32_t d_k, int32_t d_v, kda_dtype dt);
KDA_API kda_status kda_prefill_backward(const void* q, const void* k, const void* v, const float* beta,
                                const float* alpha, const int32_t* cu_seqlens, int32_t num_seqs,
                                int64_t total_tokens, int32_t H, int32_t d_k, int32_t d_v, kda_dtype dt,
                                float scale, const float* state_in, const void* grad_o,
                                const float* grad_state_out, void* grad_q, void* grad_k, void* grad_v,
                                float* grad_beta, float* grad_alpha, float* grad_state_in, void* workspace,
                                size_t workspace_bytes, void* stream);

/*
 * One fused decode step for B sequences, each with H resident states
 * ("Kimi K3, explained", section "How Kimi Delta Attention works, step by
 * step", and the question on constant-cost decode: one fixed-size state update
 * and read per generated token, independent of context length).  Each state is
 * read once, decayed, delta-corrected, written back in place, and queried.
 *
 *   q, k        [B, H, d_k]  dtype dt;  v [B, H, d_v] dtype dt
 *   beta        [B, H] float32;  alpha [B, H, d_k] float32
 *   state       [num_slots, H, d_k, d_v] float32 pool, updated in place
 *   state_idx   [B] int32 device array: row b uses slot state_idx[b]; NULL
 *               means slot b (then num_slots >= B).  Slots must be distinct
 *               within one call.  Out-of-range entries skip the row and set
 *               KDA_DEVERR_STATE_IDX.
 *   o           [B, H, d_v] dtype dt
 */
KDA_API kda_status kda_decode_step(const void* q, const void* k, const void* v, const float* beta,
                           const float* alpha, float* state, const int32_t* state_idx,
                           int32_t num_slots, void* o, int32_t B, int32_t H, int32_t d_k,
                           int32_t d_v, kda_dtype dt, float scale, void* stream);

/*
 * kda_decode_step on a state pool stored in bf16 ([num_slots, H, d_k, d_v]
 * bf16, updated in place): each state is read as bf16, updated in float32 and
 * written back rounded to nearest-even bf16.  The pages size the recurrent
 * state at 2 bytes per element ("Kimi K3 changed the memory math for agentic
 * AI forever", section "Linear Attention's Promise"), which halves the decode
 * step's state traffic.  Every other argument, result and error is kda_decode_step's.  The
 * state carries bf16 rounding from step to step, so results agree with the
 * float32-state step only to bf16 precision.
 */
KDA_API kda_status kda_decode_step_bf16_state(const void* q, const void* k, const void* v, const float* beta,
                                      const float* alpha, void* state, const int32_t* state_idx,
                                      int32_t num_slots, void* o, int32_t B, int32_t H, int32_t d_k,
                                      int32_t d_v, kda_dtype dt, float scale, void* stream);

/*
 * Options of kda_decode_step_ex.  Zero-initialise and set what is used.
 *   alpha_mode   kda_alpha_mode: layout of alpha ([B, H, d_k], [B, H], or not read)
 *   state_dtype  KDA_DTYPE_F32 (default) or KDA_DTYPE_BF16 (the pool is bf16, as
 *                kda_decode_step_bf16_state)
 */
typedef struct kda_decode_options {
    int32_t alpha_mode;
    int32_t state_dtype;
} kda_decode_options;

/* kda_decode_step with options (NULL options = kda_decode_step); `state` is float32 or bf16. */
KDA_API kda_status kda_decode_step_ex(const void* q, const void* k, const void* v, const float* beta,
                              const float* alpha, void* state, const int32_t* state_idx, int32_t num_slots,
                              void* o, int32_t B, int32_t H, int32_t d_k, int32_t d_v, kda_dtype dt,
                              float scale, void* stream, const kda_decode_options* options);

/*
 * kda_prefill without a workspace argument, for callers that cannot allocate
 * device memory.  (The pages have no counterpart; this is an interface
 * convenience.)  Typical callers: a serving process whose memory manager has
 * reserved the GPU's memory up front and hands out no scratch buffers, or a
 * host program that reaches this library only through the C ABI and has no
 * device allocator of its own.  Arguments, results and errors are those of
 * kda_prefill, except:
 *  - bf16 d = 128 runs the single-kernel chunkwise path (kda_prefill's
 *    two-phase path needs its workspace for per-chunk records), as
 *    kda_prefill_ex with single_kernel set; results agree with kda_prefill
 *    within rounding.
 *  - The scratch kda_prefill takes as `workspace` for several sequences (their
 *    longest-first order) lives in a fixed static device array of
 *    KDA_NOALLOC_MAX_SEQS int32 entries (64 KiB), which every GPU that loads
 *    libkda holds until the process exits.  num_seqs > KDA_NOALLOC_MAX_SEQS
 *    returns KDA_ERR_TOO_LARGE before anything is launched.
 *  - The function allocates and frees nothing.  The first call on a device
 *    looks up the array's device address (cudaGetSymbolAddress, with that
 *    device current) and caches it; make that first call on each device before
 *    any stream capture.
 *  - Every call shares the one array, which keeps the last call's contents;
 *    each call rewrites every entry it reads, so nothing needs clearing.  Calls
 *    whose work overlaps on the GPU (for example on two unordered streams)
 *    race on the array and must be serialised by the caller.
 */
#define KDA_NOALLOC_MAX_SEQS 16384
KDA_API kda_status kda_prefill_noalloc(const void* q, const void* k, const void* v, const float* beta,
                                       const float* alpha, const int32_t* cu_seqlens, int32_t num_seqs,
                                       int64_t total_tokens, int32_t H, int32_t d_k, int32_t d_v,
                                       kda_dtype dt, float scale, const float* state_in,
                                       float* state_out, void* o, void* stream);

/*
 * kda_prefill with q, k, v, beta, alpha, cu_seqlens, state_in, state_out and o
 * in HOST memory (same shapes and dtypes as kda_prefill; alpha per key
 * channel).  The inputs cross to the device segment by segment on an internal
 * copy stream while earlier segments compute on `stream`, and each segment's o
 * (and its sequences' final states) cross back on a second internal stream as
 * soon as they are ready, so the transfers and the compute overlap.  One
 * sequence is cut at multiples of 64 tokens with its state carried between
 * segments (the same chunks as one kda_prefill call, so the same results);
 * several sequences are grouped at sequence boundaries.
 *
 *   cu_seqlens       host [num_seqs + 1]: cu[0] = 0, non-decreasing,
 *                    cu[num_seqs] = total_tokens (checked here, on the host)
 *   state_in         host [num_seqs, H, d_k, d_v] float32, or NULL (zeros)
 *   state_out, o     host outputs, written when `stream` completes
 *   device_buffer    device memory of at least
 *                    kda_prefill_host_buffer_size(...) bytes, 256-byte aligned,
 *                    caller-owned: device copies of inputs and outputs and
 *                    the prefill's workspace.  Reuse it only on `stream`.
 *
 * Asynchronous on `stream`: every host buffer must stay valid and unchanged
 * until `stream` completes.  Pinned (page-locked) host memory is needed for
 * the copies to overlap; pageable memory works but serialises them.  Returns
 * KDA_ERR_INVALID_ARG / KDA_ERR_UNSUPPORTED / KDA_ERR_WORKSPACE before any
 * copy or launch, KDA_ERR_CUDA if a CUDA call fails.  As for kda_prefill, the
 * "Kimi K3, explained" section "The math" defines what is computed.
 */
KDA_API size_t kda_prefill_host_buffer_size(int32_t num_seqs, int64_t total_tokens, int32_t H, int32_t d_k,
                                            int32_t d_v, kda_dtype dt);
KDA_API kda_status kda_prefill_host(const void* q, const void* k, const void* v, const float* beta,
                                    const float* alpha, const int32_t* cu_seqlens, int32_t num_seqs,
                                    int64_t total_tokens, int32_t H, int32_t d_k, int32_t d_v, kda_dtype dt,
                                    float scale, const float* state_in, float* state_out, void* o,
                                    void* device_buffer, size_t device_buffer_bytes, void* stream);

/*
 * Synchronises `stream`, then reads and clears the current device's error
 * word.  *bits (may be NULL) receives the KDA_DEVERR_* bits that were set.
 * Returns KDA_OK if none were set, KDA_ERR_DEVICE if some were, KDA_ERR_CUDA if
 * a CUDA call failed.
 */
KDA_API kda_status kda_get_device_error(void* stream, uint32_t* bits);

/* Static, human-readable name of a status code. */
KDA_API const char* kda_status_string(kda_status s);

#ifdef __cplusplus
}
#endif

#endif /* KDA_H */
