// kda_prefill_host: the prefill with inputs and outputs in host memory.
//
// The transfers and the compute are pipelined over segments of the packed token array: the inputs of
// segment i+1 cross to the device on a copy stream while segment i computes on the caller's stream,
// and each segment's outputs cross back on a second copy stream as soon as its prefill is done.  A
// single sequence is cut at multiples of 64 tokens and its state carried from one segment to the next
// (the chunks are exactly those of one call, so the results are identical); several sequences are
// grouped at sequence boundaries.  The host link moves about 200 GB/s each way, so for bf16 d=128
// the copies take longer than the compute and the pipeline hides all but the last segment's compute.

#include <algorithm>
#include <cmath>
#include <mutex>

#include "kda_internal.cuh"

namespace {

constexpr int kMaxDevices = 64;
constexpr int kMaxSegments = 16;
constexpr int64_t kSegmentTokens = 1024;     // target tokens per segment

struct HostPipe {
    bool ready = false;
    cudaStream_t h2d = nullptr, d2h = nullptr;
    cudaEvent_t fork = nullptr, out_done = nullptr;
    cudaEvent_t in_done[kMaxSegments] = {}, seg_done[kMaxSegments] = {};
};
HostPipe g_pipe[kMaxDevices];
std::mutex g_pipe_mutex[kMaxDevices];        // held while a call enqueues: event records must not interleave

cudaError_t host_pipe(int dev, HostPipe** out) {
    HostPipe& hp = g_pipe[dev];
    if (!hp.ready) {
        cudaError_t e;
        if ((e = cudaStreamCreateWithFlags(&hp.h2d, cudaStreamNonBlocking)) != cudaSuccess) return e;
        if ((e = cudaStreamCreateWithFlags(&hp.d2h, cudaStreamNonBlocking)) != cudaSuccess) return e;
        if ((e = cudaEventCreateWithFlags(&hp.fork, cudaEventDisableTiming)) != cudaSuccess) return e;
        if ((e = cudaEventCreateWithFlags(&hp.out_done, cudaEventDisableTiming)) != cudaSuccess) return e;
        for (int i = 0; i < kMaxSegments; ++i) {
            if ((e = cudaEventCreateWithFlags(&hp.in_done[i], cudaEventDisableTiming)) != cudaSuccess) return e;
            if ((e = cudaEventCreateWithFlags(&hp.seg_done[i], cudaEventDisableTiming)) != cudaSuccess) return e;
        }
        hp.ready = true;
    }
    *out = &hp;
    return cudaSuccess;
}

struct Segment {
    int64_t t0, t1;      // token rows [t0, t1)
    int32_t n0, n1;      // sequences [n0, n1); for one cut sequence both segments hold sequence 0
};

// One sequence: equal cuts at multiples of 64 tokens, about kSegmentTokens each.
int64_t single_sequence_cut(int64_t T) {
    int64_t want = (T + kSegmentTokens - 1) / kSegmentTokens;
    if (want > kMaxSegments) want = kMaxSegments;
    if (want < 1) want = 1;
    const int64_t per = (T + want - 1) / want;
    return (per + kda::kChunk - 1) / kda::kChunk * kda::kChunk;
}

int plan_segments(const int32_t* cu, int32_t N, int64_t T, Segment* seg) {
    if (T == 0) {
        seg[0] = {0, 0, 0, N};
        return 1;
    }
    int S = 0;
    if (N == 1) {
        const int64_t per = single_sequence_cut(T);
        for (int64_t a = 0; a < T; a += per) seg[S++] = {a, std::min(T, a + per), 0, 1};
        return S;
    }
    const int64_t per = std::max<int64_t>(kSegmentTokens, (T + kMaxSegments - 1) / kMaxSegments);
    for (int32_t n0 = 0; n0 < N;) {
        int32_t n1 = n0 + 1;
        while (n1 < N && (int64_t)cu[n1 + 1] - cu[n0] <= per) ++n1;
        if (S == kMaxSegments - 1) n1 = N;                 // the last segment takes the rest
        seg[S++] = {cu[n0], cu[n1], n0, n1};
        n0 = n1;
    }
    return S;
}

// The cu_seqlens of every segment, rebased to the segment's first token, from the full array on the
// device (one sequence cut into segments: [0, length of the segment]).
struct SegCu {
    int32_t count, cut;
    int32_t at[kMaxSegments], n0[kMaxSegments], n1[kMaxSegments], t0[kMaxSegments], t1[kMaxSegments];
};
__global__ void kda_segment_cu_kernel(const int32_t* cu, SegCu sc, int32_t* out) {
    for (int i = 0; i < sc.count; ++i) {
        if (sc.cut) {
            if (threadIdx.x == 0) {
                out[sc.at[i]] = 0;
                out[sc.at[i] + 1] = sc.t1[i] - sc.t0[i];
            }
        } else {
            for (int j = threadIdx.x; j <= sc.n1[i] - sc.n0[i]; j += blockDim.x)
                out[sc.at[i] + j] = cu[sc.n0[i] + j] - sc.t0[i];
        }
    }
}

// Device buffer: [q | k | v | beta | alpha | o | state_in | state_out | cu_seqlens, then every segment's |
// workspace]
struct HostLayout {
    size_t q, k, v, beta, alpha, o, s_in, s_out, cu, ws, ws_bytes, total;
};
size_t a256(size_t x) { return (x + 255) / 256 * 256; }
HostLayout host_layout(int32_t N, int64_t T, int32_t H, int32_t dk, int32_t dv, kda_dtype dt) {
    HostLayout L{};
    const size_t es = dt == KDA_DTYPE_BF16 ? 2 : 4;
    const size_t rows = (size_t)T * H, states = (size_t)N * H * dk * dv * 4;
    size_t at = 0;
    L.q = at; at = a256(at + rows * dk * es);
    L.k = at; at = a256(at + rows * dk * es);
    L.v = at; at = a256(at + rows * dv * es);
    L.beta = at; at = a256(at + rows * 4);
    L.alpha = at; at = a256(at + rows * dk * 4);
    L.o = at; at = a256(at + rows * dv * es);
    L.s_in = at; at = a256(at + states);
    L.s_out = at; at = a256(at + states);
    L.cu = at; at = a256(at + (size_t)(2 * N + 2 * kMaxSegments + 2) * 4);
    // a segment holds at most N sequences and T tokens; one sequence is cut into segments of at most
    // single_sequence_cut(T) tokens, and a group of several may hold a single sequence (whose path, for
    // bf16 d=128, needs the per-chunk records)
    // (for several sequences the records are held to the one-sequence budget of 1 GiB: a segment is short,
    // and more windows only lengthen the walk, not the results)
    const size_t ws_multi = kda::prefill_2p_supported(N, T, H, dk, dv, dt)
                                ? a256(kda::prefill_2p_workspace(N, T, H, size_t(1) << 30))
                                : kda_prefill_workspace_size(N, T, H, dk, dv, dt);
    L.ws_bytes = N == 1 ? kda_prefill_workspace_size(1, std::min<int64_t>(T, single_sequence_cut(T)), H, dk, dv, dt)
                        : std::max(ws_multi, kda_prefill_workspace_size(1, T, H, dk, dv, dt));
    L.ws = at; at = a256(at + L.ws_bytes);
    L.total = at;
    return L;
}

bool supported(int32_t dk, int32_t dv) { return dk == dv && (dk == 16 || dk == 64 || dk == 128); }

}  // namespace

size_t kda_prefill_host_buffer_size(int32_t num_seqs, int64_t total_tokens, int32_t H, int32_t d_k, int32_t d_v,
                                    kda_dtype dt) {
    if (num_seqs <= 0 || total_tokens < 0 || total_tokens > INT32_MAX || H <= 0 || !supported(d_k, d_v) ||
        (dt != KDA_DTYPE_F32 && dt != KDA_DTYPE_BF16))
        return 0;
    return host_layout(num_seqs, total_tokens, H, d_k, d_v, dt).total;
}

kda_status kda_prefill_host(const void* q, const void* k, const void* v, const float* beta, const float* alpha,
                            const int32_t* cu_seqlens, int32_t num_seqs, int64_t total_tokens, int32_t H,
                            int32_t d_k, int32_t d_v, kda_dtype dt, float scale, const float* state_in,
                            float* state_out, void* o, void* device_buffer, size_t device_buffer_bytes, void* stream) {
    // ---- host-side validation (cu_seqlens is in host memory, so it is checked here in full) ----
    if (num_seqs <= 0 || total_tokens < 0 || total_tokens > INT32_MAX || H <= 0 || d_k <= 0 || d_v <= 0)
        return KDA_ERR_INVALID_ARG;
    if (dt != KDA_DTYPE_F32 && dt != KDA_DTYPE_BF16) return KDA_ERR_INVALID_ARG;
    if (!std::isfinite(scale)) return KDA_ERR_INVALID_ARG;
    if (!supported(d_k, d_v)) return KDA_ERR_UNSUPPORTED;
    if (!cu_seqlens || !state_out) return KDA_ERR_INVALID_ARG;
    if (total_tokens > 0 && (!q || !k || !v || !beta || !alpha || !o)) return KDA_ERR_INVALID_ARG;
    if (cu_seqlens[0] != 0 || cu_seqlens[num_seqs] != total_tokens) return KDA_ERR_INVALID_ARG;
    for (int32_t n = 0; n < num_seqs; ++n)
        if (cu_seqlens[n + 1] < cu_seqlens[n]) return KDA_ERR_INVALID_ARG;
    const HostLayout L = host_layout(num_seqs, total_tokens, H, d_k, d_v, dt);
    if (!device_buffer || device_buffer_bytes < L.total || (reinterpret_cast<uintptr_t>(device_buffer) & 255u))
        return KDA_ERR_WORKSPACE;

    Segment seg[kMaxSegments];
    const int S = plan_segments(cu_seqlens, num_seqs, total_tokens, seg);
    const bool cut = num_seqs == 1;                          // one sequence, state carried between segments
    SegCu sc{};
    sc.count = S;
    sc.cut = cut ? 1 : 0;
    for (int i = 0, at = num_seqs + 1; i < S; ++i) {       // the segment arrays follow the full copy
        sc.at[i] = at;
        sc.n0[i] = seg[i].n0; sc.n1[i] = seg[i].n1;
        sc.t0[i] = (int32_t)seg[i].t0; sc.t1[i] = (int32_t)seg[i].t1;
        at += cut ? 2 : seg[i].n1 - seg[i].n0 + 1;
    }

    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return KDA_ERR_CUDA;
    std::lock_guard<std::mutex> lock(g_pipe_mutex[dev]);
    HostPipe* hp = nullptr;
    if (host_pipe(dev, &hp) != cudaSuccess) return KDA_ERR_CUDA;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    unsigned char* db = static_cast<unsigned char*>(device_buffer);
    const size_t es = dt == KDA_DTYPE_BF16 ? 2 : 4;
    const size_t st = (size_t)H * d_k * d_v * 4;
    auto ok = [](cudaError_t e) { return e == cudaSuccess; };

    // the copy streams start after the work already queued on the caller's stream
    if (!ok(cudaEventRecord(hp->fork, s)) || !ok(cudaStreamWaitEvent(hp->h2d, hp->fork, 0)) ||
        !ok(cudaStreamWaitEvent(hp->d2h, hp->fork, 0)))
        return KDA_ERR_CUDA;
    // once the copy streams are forked, every return joins them back into the caller's stream, so that no
    // copy that reads or writes the caller's host buffers outlives the call unordered (also on an error)
    auto join = [&](kda_status st_) -> kda_status {
        bool joined = ok(cudaEventRecord(hp->fork, hp->h2d)) && ok(cudaStreamWaitEvent(hp->d2h, hp->fork, 0)) &&
                      ok(cudaEventRecord(hp->out_done, hp->d2h)) && ok(cudaStreamWaitEvent(s, hp->out_done, 0));
        return st_ != KDA_OK ? st_ : (joined ? KDA_OK : KDA_ERR_CUDA);
    };
    int32_t* cu_dev = reinterpret_cast<int32_t*>(db + L.cu);
    if (!ok(cudaMemcpyAsync(cu_dev, cu_seqlens, (size_t)(num_seqs + 1) * 4, cudaMemcpyHostToDevice, hp->h2d)))
        return join(KDA_ERR_CUDA);
    kda_segment_cu_kernel<<<1, 128, 0, hp->h2d>>>(cu_dev, sc, cu_dev);
    if (!ok(cudaGetLastError())) return join(KDA_ERR_CUDA);
    // inputs, segment by segment
    for (int i = 0; i < S; ++i) {
        const size_t r0 = (size_t)seg[i].t0 * H, nr = (size_t)(seg[i].t1 - seg[i].t0) * H;
        if (nr > 0) {
            const char* src[5] = {static_cast<const char*>(q), static_cast<const char*>(k), static_cast<const char*>(v),
                                  reinterpret_cast<const char*>(beta), reinterpret_cast<const char*>(alpha)};
            const size_t off[5] = {L.q, L.k, L.v, L.beta, L.alpha};
            const size_t width[5] = {d_k * es, d_k * es, d_v * es, 4, (size_t)d_k * 4};
            for (int a = 0; a < 5; ++a)
                if (!ok(cudaMemcpyAsync(db + off[a] + r0 * width[a], src[a] + r0 * width[a], nr * width[a],
                                        cudaMemcpyHostToDevice, hp->h2d)))
                    return join(KDA_ERR_CUDA);
        }
        if (state_in && (!cut || i == 0)) {
            const size_t b0 = (size_t)seg[i].n0 * st, nb = (size_t)(seg[i].n1 - seg[i].n0) * st;
            if (!ok(cudaMemcpyAsync(db + L.s_in + b0, reinterpret_cast<const char*>(state_in) + b0, nb,
                                    cudaMemcpyHostToDevice, hp->h2d)))
                return join(KDA_ERR_CUDA);
        }
        if (!ok(cudaEventRecord(hp->in_done[i], hp->h2d))) return join(KDA_ERR_CUDA);
    }
    // compute on the caller's stream, outputs back on the second copy stream
    for (int i = 0; i < S; ++i) {
        const size_t r0 = (size_t)seg[i].t0 * H, nr = (size_t)(seg[i].t1 - seg[i].t0) * H;
        const int32_t segN = seg[i].n1 - seg[i].n0;
        const float* sin = nullptr;
        if (cut) sin = i == 0 ? (state_in ? reinterpret_cast<const float*>(db + L.s_in) : nullptr)
                              : reinterpret_cast<const float*>(db + L.s_out);
        else if (state_in) sin = reinterpret_cast<const float*>(db + L.s_in + (size_t)seg[i].n0 * st);
        float* sout = reinterpret_cast<float*>(db + L.s_out + (size_t)seg[i].n0 * st);
        if (!ok(cudaStreamWaitEvent(s, hp->in_done[i], 0))) return join(KDA_ERR_CUDA);
        const kda_status ks = kda_prefill_ex(db + L.q + r0 * d_k * es, db + L.k + r0 * d_k * es,
                                             db + L.v + r0 * d_v * es, reinterpret_cast<const float*>(db + L.beta) + r0,
                                             reinterpret_cast<const float*>(db + L.alpha) + r0 * d_k, cu_dev + sc.at[i],
                                             segN, seg[i].t1 - seg[i].t0, H, d_k, d_v, dt, scale, sin, sout,
                                             db + L.o + r0 * d_v * es, db + L.ws, L.ws_bytes, s, nullptr);
        if (ks != KDA_OK) return join(ks);
        if (!ok(cudaEventRecord(hp->seg_done[i], s)) || !ok(cudaStreamWaitEvent(hp->d2h, hp->seg_done[i], 0)))
            return join(KDA_ERR_CUDA);
        if (nr > 0 && !ok(cudaMemcpyAsync(static_cast<char*>(o) + r0 * d_v * es, db + L.o + r0 * d_v * es,
                                          nr * d_v * es, cudaMemcpyDeviceToHost, hp->d2h)))
            return join(KDA_ERR_CUDA);
        if (!cut || i == S - 1) {
            const size_t b0 = (size_t)seg[i].n0 * st, nb = (size_t)(seg[i].n1 - seg[i].n0) * st;
            if (!ok(cudaMemcpyAsync(reinterpret_cast<char*>(state_out) + b0, db + L.s_out + b0, nb,
                                    cudaMemcpyDeviceToHost, hp->d2h)))
                return join(KDA_ERR_CUDA);
        }
    }
    // the caller's stream completes only after the last copy back
    return join(KDA_OK);
}
