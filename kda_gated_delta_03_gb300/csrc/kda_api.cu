// C ABI of libkda: host-side validation, scheduling and dispatch.
//
// Every entry point validates its arguments completely on the host before it
// touches the CUDA runtime, so a rejected call launches nothing.  The only
// state the library keeps is one 32-bit error word per device (a file-scope
// __device__ variable), which kernels set when they detect inconsistent
// device-side inputs and kda_get_device_error reads back and clears.

#include <cmath>
#include <cstring>
#include <mutex>

#include "kda_internal.cuh"

namespace {

__device__ unsigned g_kda_device_error = 0u;

constexpr int kMaxDevices = 64;
std::mutex g_err_mutex;
unsigned* g_err_addr[kMaxDevices] = {};

kda_status error_word(unsigned** out) {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return KDA_ERR_CUDA;
    std::lock_guard<std::mutex> lock(g_err_mutex);
    if (!g_err_addr[dev]) {
        void* p = nullptr;
        if (cudaGetSymbolAddress(&p, g_kda_device_error) != cudaSuccess) return KDA_ERR_CUDA;
        g_err_addr[dev] = static_cast<unsigned*>(p);
    }
    *out = g_err_addr[dev];
    return KDA_OK;
}

bool aligned(const void* p, size_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }

bool supported_head(int32_t dk, int32_t dv) { return dk == dv && (dk == 16 || dk == 64 || dk == 128); }

size_t align_up(size_t x, size_t a) { return (x + a - 1) / a * a; }

// alpha's pointer requirements under its layout (DeltaNet reads none).
bool alpha_ok(const float* alpha, int32_t mode) {
    if (mode == KDA_ALPHA_NONE) return true;
    if (mode == KDA_ALPHA_PER_HEAD) return alpha && aligned(alpha, 4);
    return mode == KDA_ALPHA_PER_CHANNEL && alpha && aligned(alpha, 16);
}

// Scratch of kda_prefill_noalloc: the longest-first sequence order, in a fixed
// static device array so that the entry point never allocates.  Host code must
// not pass the array's name to a kernel (on the host it is only a stand-in);
// the device address is looked up once per device and cached.
static __device__ __align__(256) int32_t g_kda_noalloc_order[KDA_NOALLOC_MAX_SEQS];
std::mutex g_noalloc_mutex;
int32_t* g_noalloc_addr[kMaxDevices] = {};

kda_status noalloc_scratch(int32_t** out) {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return KDA_ERR_CUDA;
    std::lock_guard<std::mutex> lock(g_noalloc_mutex);
    if (!g_noalloc_addr[dev]) {
        int32_t* ptr = nullptr;
        if (cudaGetSymbolAddress((void**)&ptr, g_kda_noalloc_order) != cudaSuccess || !ptr) return KDA_ERR_CUDA;
        g_noalloc_addr[dev] = ptr;
    }
    *out = g_noalloc_addr[dev];
    return KDA_OK;
}

#ifdef KDA_TEST_HOOKS
int32_t g_test_stall = 0;   // test builds only: set by kda_test_stall_prefill
#endif

}  // namespace

#ifdef KDA_TEST_HOOKS
// Test builds only (-DKDA_TEST_HOOKS; not in kda.h): while `on` is nonzero, the tcgen05 prefill kernels of
// later kda_prefill calls give up a bounded wait on purpose, so that a test can check the give-up path.
extern "C" KDA_API void kda_test_stall_prefill(int32_t on) { g_test_stall = on; }
#endif

extern "C" {

const char* kda_status_string(kda_status s) {
    switch (s) {
        case KDA_OK: return "KDA_OK";
        case KDA_ERR_INVALID_ARG: return "KDA_ERR_INVALID_ARG";
        case KDA_ERR_UNSUPPORTED: return "KDA_ERR_UNSUPPORTED";
        case KDA_ERR_WORKSPACE: return "KDA_ERR_WORKSPACE";
        case KDA_ERR_CUDA: return "KDA_ERR_CUDA";
        case KDA_ERR_DEVICE: return "KDA_ERR_DEVICE";
        case KDA_ERR_TOO_LARGE: return "KDA_ERR_TOO_LARGE";
    }
    return "KDA_ERR_UNKNOWN";
}

size_t kda_prefill_workspace_size(int32_t num_seqs, int64_t total_tokens, int32_t H, int32_t d_k,
                                  int32_t d_v, kda_dtype dt) {
    if (kda::prefill_2p_supported(num_seqs, total_tokens, H, d_k, d_v, dt))   // per-chunk records
        return align_up(kda::prefill_2p_workspace(num_seqs, total_tokens, H), 256);
    if (num_seqs <= 1) return 0;
    // longest-first schedule of the sequences
    return align_up(sizeof(int32_t) * (size_t)num_seqs, 256);
}

int64_t kda_prefill_launch_count(int32_t num_seqs, int64_t total_tokens, int32_t H, int32_t d_k, int32_t d_v,
                                 kda_dtype dt, size_t workspace_bytes) {
    if (num_seqs < 0 || total_tokens < 0 || total_tokens > INT32_MAX || H <= 0 || d_k <= 0 || d_v <= 0) return -1;
    if ((dt != KDA_DTYPE_F32 && dt != KDA_DTYPE_BF16) || !supported_head(d_k, d_v)) return -1;
    if (num_seqs == 0) return total_tokens == 0 ? 0 : -1;
    if (kda::prefill_2p_supported(num_seqs, total_tokens, H, d_k, d_v, dt)) {
        if (workspace_bytes < kda::prefill_2p_min_workspace(num_seqs, H)) return -1;
        int dev = 0, sms = 0;
        if (cudaGetDevice(&dev) != cudaSuccess ||
            cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
            return -1;
        const int64_t chunks = kda::prefill_2p_max_chunks(num_seqs, total_tokens);
        const kda::WindowPlan plan = kda::prefill_2p_plan(num_seqs, chunks, H, workspace_bytes, sms);
        // several sequences: chunk offsets and longest-first order first
        return (num_seqs > 1 ? 2 : 0) + 2 * ((chunks + plan.window - 1) / plan.window);
    }
    return num_seqs > 1 ? 2 : 1;                      // longest-first order, then the chunkwise kernel
}

kda_status kda_prefill(const void* q, const void* k, const void* v, const float* beta,
                       const float* alpha, const int32_t* cu_seqlens, int32_t num_seqs,
                       int64_t total_tokens, int32_t H, int32_t d_k, int32_t d_v, kda_dtype dt,
                       float scale, const float* state_in, float* state_out, void* o,
                       void* workspace, size_t workspace_bytes, void* stream) {
    return kda_prefill_ex(q, k, v, beta, alpha, cu_seqlens, num_seqs, total_tokens, H, d_k, d_v, dt, scale, state_in,
                          state_out, o, workspace, workspace_bytes, stream, nullptr);
}

kda_status kda_prefill_ex(const void* q, const void* k, const void* v, const float* beta,
                          const float* alpha, const int32_t* cu_seqlens, int32_t num_seqs,
                          int64_t total_tokens, int32_t H, int32_t d_k, int32_t d_v, kda_dtype dt,
                          float scale, const float* state_in, float* state_out, void* o,
                          void* workspace, size_t workspace_bytes, void* stream,
                          const kda_prefill_options* options) {
    // ---- host-side validation (no CUDA call before this block ends) ----
    const int32_t snap_every = options ? options->snapshot_every : 0;
    if (snap_every < 0 || snap_every % kda::kChunk != 0) return KDA_ERR_INVALID_ARG;
    if (snap_every > 0 && (!options->snapshots || !options->snapshot_offsets || !aligned(options->snapshots, 16) ||
                           !aligned(options->snapshot_offsets, 4)))
        return KDA_ERR_INVALID_ARG;
    if (num_seqs < 0 || total_tokens < 0 || total_tokens > INT32_MAX || H <= 0 || d_k <= 0 ||
        d_v <= 0 || !std::isfinite(scale))
        return KDA_ERR_INVALID_ARG;
    if (dt != KDA_DTYPE_F32 && dt != KDA_DTYPE_BF16) return KDA_ERR_INVALID_ARG;
    if (!supported_head(d_k, d_v)) return KDA_ERR_UNSUPPORTED;
    if (num_seqs == 0) return total_tokens == 0 ? KDA_OK : KDA_ERR_INVALID_ARG;
    if (!cu_seqlens || !state_out || !aligned(cu_seqlens, 4) || !aligned(state_out, 16))
        return KDA_ERR_INVALID_ARG;
    if (state_in && !aligned(state_in, 16)) return KDA_ERR_INVALID_ARG;
    const int32_t alpha_mode = options ? options->alpha_mode : KDA_ALPHA_PER_CHANNEL;
    if (alpha_mode != KDA_ALPHA_PER_CHANNEL && alpha_mode != KDA_ALPHA_PER_HEAD && alpha_mode != KDA_ALPHA_NONE)
        return KDA_ERR_INVALID_ARG;
    if (total_tokens > 0) {
        if (!q || !k || !v || !beta || !o || !alpha_ok(alpha, alpha_mode)) return KDA_ERR_INVALID_ARG;
        if (!aligned(q, 16) || !aligned(k, 16) || !aligned(v, 16) || !aligned(o, 16) || !aligned(beta, 4))
            return KDA_ERR_INVALID_ARG;
    }
    const bool two_phase = kda::prefill_2p_supported(num_seqs, total_tokens, H, d_k, d_v, dt) &&
                           !(options && options->single_kernel);
    // the two-phase path takes any workspace down to one chunk's records and uses more windows
    const size_t need = two_phase ? kda::prefill_2p_min_workspace(num_seqs, H)
                          : num_seqs > 1 ? align_up(sizeof(int32_t) * (size_t)num_seqs, 256)   // longest-first order
                                         : 0;
    if (need > 0 && (!workspace || workspace_bytes < need || !aligned(workspace, 256)))
        return KDA_ERR_WORKSPACE;

    // ---- launch ----
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    unsigned* err = nullptr;
    if (error_word(&err) != KDA_OK) return KDA_ERR_CUDA;

    kda::PrefillParams p{};
    p.q = q; p.k = k; p.v = v; p.beta = beta; p.alpha = alpha;
    p.cu_seqlens = cu_seqlens;
    p.order = nullptr;
    p.num_seqs = num_seqs;
    p.total_tokens = static_cast<int32_t>(total_tokens);
    p.H = H; p.dk = d_k; p.dv = d_v;
    p.scale = scale;
    p.state_in = state_in; p.state_out = state_out; p.o = o;
    p.err = err;
    p.alpha_mode = alpha_mode;
#ifdef KDA_TEST_HOOKS
    p.test_stall = g_test_stall;
#endif
    p.snap_every = snap_every;
    p.snapshots = snap_every > 0 ? options->snapshots : nullptr;
    p.snap_offsets = snap_every > 0 ? options->snapshot_offsets : nullptr;
    if (two_phase) {
        p.slices = 1;
        if (kda::launch_prefill_2p(p, workspace, workspace_bytes, s) != cudaSuccess) return KDA_ERR_CUDA;
        return KDA_OK;
    }
    if (need > 0) {
        int32_t* order = static_cast<int32_t*>(workspace);
        if (kda::launch_order(cu_seqlens, num_seqs, order, s) != cudaSuccess) return KDA_ERR_CUDA;
        p.order = order;
    }
    if (kda::prefill_tc_supported(p, dt)) {
        p.slices = kda::prefill_tc_slices(num_seqs, H, d_v);
        if (kda::launch_prefill_tc(p, s) != cudaSuccess) return KDA_ERR_CUDA;
    } else {
        p.slices = kda::prefill_cc_slices(d_v);
        if (kda::launch_prefill_cc(p, dt, s) != cudaSuccess) return KDA_ERR_CUDA;
    }
    return KDA_OK;
}

}  // extern "C"

namespace {

kda_status decode_impl(const void* q, const void* k, const void* v, const float* beta, const float* alpha,
                       void* state, bool state_bf16, int32_t alpha_mode, const int32_t* state_idx, int32_t num_slots,
                       void* o, int32_t B, int32_t H, int32_t d_k, int32_t d_v, kda_dtype dt, float scale,
                       void* stream) {
    if (B < 0 || H <= 0 || d_k <= 0 || d_v <= 0 || num_slots < 0 || !std::isfinite(scale))
        return KDA_ERR_INVALID_ARG;
    if (dt != KDA_DTYPE_F32 && dt != KDA_DTYPE_BF16) return KDA_ERR_INVALID_ARG;
    if (alpha_mode != KDA_ALPHA_PER_CHANNEL && alpha_mode != KDA_ALPHA_PER_HEAD && alpha_mode != KDA_ALPHA_NONE)
        return KDA_ERR_INVALID_ARG;
    if (!supported_head(d_k, d_v)) return KDA_ERR_UNSUPPORTED;
    if (B == 0) return KDA_OK;
    if (!q || !k || !v || !beta || !alpha_ok(alpha, alpha_mode) || !state || !o) return KDA_ERR_INVALID_ARG;
    if (!aligned(q, 16) || !aligned(k, 16) || !aligned(v, 16) || !aligned(o, 16) || !aligned(beta, 4) ||
        !aligned(state, 16))
        return KDA_ERR_INVALID_ARG;
    if (state_idx ? !aligned(state_idx, 4) : num_slots < B) return KDA_ERR_INVALID_ARG;

    cudaStream_t s = static_cast<cudaStream_t>(stream);
    unsigned* err = nullptr;
    if (error_word(&err) != KDA_OK) return KDA_ERR_CUDA;
    kda::DecodeParams p{};
    p.q = q; p.k = k; p.v = v; p.beta = beta; p.alpha = alpha;
    p.state = state; p.state_bf16 = state_bf16; p.alpha_mode = alpha_mode;
    p.state_idx = state_idx; p.num_slots = num_slots;
    p.o = o; p.B = B; p.H = H; p.d = d_k; p.scale = scale; p.err = err;
    if (kda::launch_decode(p, dt, s) != cudaSuccess) return KDA_ERR_CUDA;
    return KDA_OK;
}

}  // namespace

extern "C" {

kda_status kda_decode_step(const void* q, const void* k, const void* v, const float* beta,
                           const float* alpha, float* state, const int32_t* state_idx,
                           int32_t num_slots, void* o, int32_t B, int32_t H, int32_t d_k,
                           int32_t d_v, kda_dtype dt, float scale, void* stream) {
    return decode_impl(q, k, v, beta, alpha, state, false, KDA_ALPHA_PER_CHANNEL, state_idx, num_slots, o, B, H,
                       d_k, d_v, dt, scale, stream);
}

kda_status kda_decode_step_bf16_state(const void* q, const void* k, const void* v, const float* beta,
                                      const float* alpha, void* state, const int32_t* state_idx,
                                      int32_t num_slots, void* o, int32_t B, int32_t H, int32_t d_k,
                                      int32_t d_v, kda_dtype dt, float scale, void* stream) {
    return decode_impl(q, k, v, beta, alpha, state, true, KDA_ALPHA_PER_CHANNEL, state_idx, num_slots, o, B, H,
                       d_k, d_v, dt, scale, stream);
}

kda_status kda_decode_step_ex(const void* q, const void* k, const void* v, const float* beta, const float* alpha,
                              void* state, const int32_t* state_idx, int32_t num_slots, void* o, int32_t B,
                              int32_t H, int32_t d_k, int32_t d_v, kda_dtype dt, float scale, void* stream,
                              const kda_decode_options* options) {
    const int32_t sdt = options ? options->state_dtype : KDA_DTYPE_F32;
    if (sdt != KDA_DTYPE_F32 && sdt != KDA_DTYPE_BF16) return KDA_ERR_INVALID_ARG;
    return decode_impl(q, k, v, beta, alpha, state, sdt == KDA_DTYPE_BF16,
                       options ? options->alpha_mode : KDA_ALPHA_PER_CHANNEL, state_idx, num_slots, o, B, H, d_k,
                       d_v, dt, scale, stream);
}

kda_status kda_prefill_noalloc(const void* q, const void* k, const void* v, const float* beta,
                               const float* alpha, const int32_t* cu_seqlens, int32_t num_seqs,
                               int64_t total_tokens, int32_t H, int32_t d_k, int32_t d_v, kda_dtype dt,
                               float scale, const float* state_in, float* state_out, void* o, void* stream) {
    // ---- host-side validation, as kda_prefill, plus the fixed scratch limit ----
    if (num_seqs < 0 || total_tokens < 0 || total_tokens > INT32_MAX || H <= 0 || d_k <= 0 ||
        d_v <= 0 || !std::isfinite(scale))
        return KDA_ERR_INVALID_ARG;
    if (dt != KDA_DTYPE_F32 && dt != KDA_DTYPE_BF16) return KDA_ERR_INVALID_ARG;
    if (!supported_head(d_k, d_v)) return KDA_ERR_UNSUPPORTED;
    if (num_seqs > KDA_NOALLOC_MAX_SEQS) return KDA_ERR_TOO_LARGE;
    if (num_seqs == 0) return total_tokens == 0 ? KDA_OK : KDA_ERR_INVALID_ARG;
    if (!cu_seqlens || !state_out || !aligned(cu_seqlens, 4) || !aligned(state_out, 16))
        return KDA_ERR_INVALID_ARG;
    if (state_in && !aligned(state_in, 16)) return KDA_ERR_INVALID_ARG;
    if (total_tokens > 0) {
        if (!q || !k || !v || !beta || !alpha || !o) return KDA_ERR_INVALID_ARG;
        if (!aligned(q, 16) || !aligned(k, 16) || !aligned(v, 16) || !aligned(o, 16) ||
            !aligned(alpha, 16) || !aligned(beta, 4))
            return KDA_ERR_INVALID_ARG;
    }

    // ---- launch, with the static scratch in place of a workspace ----
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    unsigned* err = nullptr;
    if (error_word(&err) != KDA_OK) return KDA_ERR_CUDA;
    kda::PrefillParams p{};
    p.q = q; p.k = k; p.v = v; p.beta = beta; p.alpha = alpha;
    p.cu_seqlens = cu_seqlens;
    p.order = nullptr;
    p.num_seqs = num_seqs;
    p.total_tokens = static_cast<int32_t>(total_tokens);
    p.H = H; p.dk = d_k; p.dv = d_v;
    p.scale = scale;
    p.state_in = state_in; p.state_out = state_out; p.o = o;
    p.err = err;
    p.alpha_mode = KDA_ALPHA_PER_CHANNEL;
    if (num_seqs > 1) {
        int32_t* order = nullptr;
        if (noalloc_scratch(&order) != KDA_OK) return KDA_ERR_CUDA;
        if (kda::launch_order(cu_seqlens, num_seqs, order, s) != cudaSuccess) return KDA_ERR_CUDA;
        p.order = order;
    }
    if (kda::prefill_tc_supported(p, dt)) {
        p.slices = kda::prefill_tc_slices(num_seqs, H, d_v);
        if (kda::launch_prefill_tc(p, s) != cudaSuccess) return KDA_ERR_CUDA;
    } else {
        p.slices = kda::prefill_cc_slices(d_v);
        if (kda::launch_prefill_cc(p, dt, s) != cudaSuccess) return KDA_ERR_CUDA;
    }
    return KDA_OK;
}

namespace {
// Workspace of the backward pass: [snapshot and chunk offsets | snapshots | state gradients at the same
// boundaries | o and state_out of the recompute | the recompute's own workspace | per-CTA chunk states]
struct BwdLayout {
    size_t off, snaps, gb, o, st, fwd, scratch, total;
};
// chunk units of the chunk pass, at most: every sequence adds at most one partial chunk
int64_t bwd_max_units(int32_t N, int64_t T, int32_t H) { return (T / kda::kChunk + N) * H; }
BwdLayout bwd_layout(int32_t N, int64_t T, int32_t H, int32_t d, kda_dtype dt) {
    BwdLayout L{};
    const size_t dd = (size_t)d * d * 4, esize = dt == KDA_DTYPE_BF16 ? 2 : 4;
    const int64_t units = bwd_max_units(N, T, H);
    const size_t ctas = (size_t)(units < kda::kBwdMaxCtas ? units : kda::kBwdMaxCtas);
    size_t at = 0;
    L.off = at; at = align_up(at + (size_t)(N + 1) * 8, 256);
    L.snaps = at; at = align_up(at + (size_t)(T / kda::kChunk) * H * dd, 256);
    L.gb = at; at = align_up(at + (size_t)(T / kda::kChunk) * H * dd, 256);
    L.o = at; at = align_up(at + (size_t)T * H * d * esize, 256);
    L.st = at; at = align_up(at + (size_t)N * H * dd, 256);
    // the forward recompute: one sequence may take the two-phase path (records), several the single-kernel
    // path (the longest-first order only)
    L.fwd = at;
    at = align_up(at + (N == 1 ? kda_prefill_workspace_size(1, T, H, d, d, dt) : align_up(4 * (size_t)N, 256)), 256);
    // per-CTA scratch of the chunk pass: the matrix form's matrices at d = 128, the token walk's states else
    L.scratch = at; at = align_up(at + ctas * (d == 128 ? kda::kBwdMatScratchBytes : (kda::kChunk - 1) * dd), 256);
    L.total = at;
    return L;
}
}  // namespace

size_t kda_prefill_backward_workspace_size(int32_t num_seqs, int64_t total_tokens, int32_t H, int32_t d_k,
                                           int32_t d_v, kda_dtype dt) {
    if (num_seqs <= 0 || total_tokens < 0 || H <= 0 || !supported_head(d_k, d_v)) return 0;
    return bwd_layout(num_seqs, total_tokens, H, d_k, dt).total;
}

kda_status kda_prefill_backward(const void* q, const void* k, const void* v, const float* beta, const float* alpha,
                                const int32_t* cu_seqlens, int32_t num_seqs, int64_t total_tokens, int32_t H,
                                int32_t d_k, int32_t d_v, kda_dtype dt, float scale, const float* state_in,
                                const void* grad_o, const float* grad_state_out, void* grad_q, void* grad_k,
                                void* grad_v, float* grad_beta, float* grad_alpha, float* grad_state_in, void* workspace,
                                size_t workspace_bytes, void* stream) {
    // ---- host-side validation ----
    if (num_seqs < 0 || total_tokens < 0 || total_tokens > INT32_MAX || H <= 0 || d_k <= 0 || d_v <= 0 ||
        !std::isfinite(scale))
        return KDA_ERR_INVALID_ARG;
    if (dt != KDA_DTYPE_F32 && dt != KDA_DTYPE_BF16) return KDA_ERR_INVALID_ARG;
    if (!supported_head(d_k, d_v)) return KDA_ERR_UNSUPPORTED;
    if (num_seqs == 0) return total_tokens == 0 ? KDA_OK : KDA_ERR_INVALID_ARG;
    if (!cu_seqlens || !aligned(cu_seqlens, 4)) return KDA_ERR_INVALID_ARG;
    if ((state_in && !aligned(state_in, 16)) || (grad_state_out && !aligned(grad_state_out, 16)) ||
        (grad_state_in && !aligned(grad_state_in, 16)))
        return KDA_ERR_INVALID_ARG;
    if (total_tokens > 0) {
        if (!q || !k || !v || !beta || !alpha || !grad_o || !grad_q || !grad_k || !grad_v || !grad_beta ||
            !grad_alpha)
            return KDA_ERR_INVALID_ARG;
        if (!aligned(q, 16) || !aligned(k, 16) || !aligned(v, 16) || !aligned(alpha, 16) || !aligned(beta, 4) ||
            !aligned(grad_o, 16) || !aligned(grad_q, 16) || !aligned(grad_k, 16) || !aligned(grad_v, 16) ||
            !aligned(grad_beta, 4) || !aligned(grad_alpha, 16))
            return KDA_ERR_INVALID_ARG;
    }
    const BwdLayout L = bwd_layout(num_seqs, total_tokens, H, d_k, dt);
    if (!workspace || workspace_bytes < L.total || !aligned(workspace, 256)) return KDA_ERR_WORKSPACE;

    // ---- forward recompute with a snapshot at every chunk boundary, then the walk back ----
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    unsigned* err = nullptr;
    if (error_word(&err) != KDA_OK) return KDA_ERR_CUDA;
    unsigned char* ws = static_cast<unsigned char*>(workspace);
    int32_t* off = reinterpret_cast<int32_t*>(ws + L.off);
    int32_t* choff = off + (num_seqs + 1);
    float* snaps = reinterpret_cast<float*>(ws + L.snaps);
    if (kda::launch_bwd_offsets(cu_seqlens, num_seqs, static_cast<int32_t>(total_tokens), off, choff, err, s) !=
        cudaSuccess)
        return KDA_ERR_CUDA;
    kda_prefill_options opts{};
    opts.snapshot_every = kda::kChunk;
    opts.snapshots = snaps;
    opts.snapshot_offsets = off;
    opts.single_kernel = num_seqs > 1 ? 1 : 0;        // several sequences: the single-kernel recompute
    const kda_status fs = kda_prefill_ex(q, k, v, beta, alpha, cu_seqlens, num_seqs, total_tokens, H, d_k, d_v, dt,
                                         scale, state_in, reinterpret_cast<float*>(ws + L.st), ws + L.o, ws + L.fwd,
                                         L.scratch - L.fwd, stream, &opts);
    if (fs != KDA_OK) return fs;
    if (total_tokens == 0 && !grad_state_in) return KDA_OK;
    kda::BwdParams p{};
    p.q = q; p.k = k; p.v = v; p.beta = beta; p.alpha = alpha; p.cu_seqlens = cu_seqlens;
    p.num_seqs = num_seqs; p.total_tokens = static_cast<int32_t>(total_tokens); p.H = H; p.dk = d_k; p.dv = d_v;
    p.scale = scale; p.state_in = state_in; p.d_o = grad_o; p.d_state_out = grad_state_out;
    p.d_q = grad_q; p.d_k = grad_k; p.d_v = grad_v; p.d_beta = grad_beta; p.d_alpha = grad_alpha;
    p.d_state_in = grad_state_in;
    p.snapshots = snaps; p.snap_offsets = off; p.chunk_offsets = choff;
    p.dstate_b = reinterpret_cast<float*>(ws + L.gb);
    p.scratch = reinterpret_cast<float*>(ws + L.scratch);
    p.err = err;
    int dev = 0, sms = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
        return KDA_ERR_CUDA;
    // one bf16 d=128 sequence whose forward recompute ran as one window: every chunk's record (Q', M,
    // Gamma_C) is still in the workspace, and the state-gradient chain walks chunks instead of tokens
    if (num_seqs == 1 && kda::prefill_2p_supported(num_seqs, total_tokens, H, d_k, d_v, dt) && total_tokens > 0) {
        const int64_t chunks = (total_tokens + kda::kChunk - 1) / kda::kChunk;
        const kda::WindowPlan plan = kda::prefill_2p_plan(1, chunks, H, L.scratch - L.fwd, sms);
        if (plan.window >= chunks) p.records = ws + L.fwd;
    }
    const int64_t units = bwd_max_units(num_seqs, total_tokens, H);
    int grid = (int)(units < kda::kBwdMaxCtas ? units : kda::kBwdMaxCtas);
    if (grid > sms) grid = sms;
    if (grid < 1) grid = 1;
    if (kda::launch_prefill_bwd(p, dt, grid, s) != cudaSuccess) return KDA_ERR_CUDA;
    return KDA_OK;
}

kda_status kda_get_device_error(void* stream, uint32_t* bits) {
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    unsigned* err = nullptr;
    if (error_word(&err) != KDA_OK) return KDA_ERR_CUDA;
    unsigned host = 0;
    if (cudaStreamSynchronize(s) != cudaSuccess) return KDA_ERR_CUDA;
    if (cudaMemcpy(&host, err, sizeof host, cudaMemcpyDeviceToHost) != cudaSuccess) return KDA_ERR_CUDA;
    if (host != 0u && cudaMemset(err, 0, sizeof host) != cudaSuccess) return KDA_ERR_CUDA;
    if (bits) *bits = host;
    return host ? KDA_ERR_DEVICE : KDA_OK;
}

}  // extern "C"
