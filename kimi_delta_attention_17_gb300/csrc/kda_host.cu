// Host-buffer entry points: the prefill and a run of decode steps whose inputs
// and outputs live in host memory. The work is cut into windows (prefill: whole
// 64-token chunks of each sequence; decode: one step); window w + 1's inputs
// are copied in on one copy stream and window w - 1's outputs copied out on
// another while window w computes on the caller's stream. All device memory is
// the caller's workspace; nothing here allocates device memory.
#include <string.h>

#include <algorithm>
#include <vector>

#include "kda_internal.cuh"

namespace kda {
namespace {

// Most sequence pieces in one prefill window: bounds the per-window state
// buffers (each piece carries H * dk * dv fp32 in and out).
constexpr int kHostMaxPieces = 16;
constexpr size_t kAlign = 256;

struct Piece {
    int seq;        // sequence index
    long long off;  // first token of the piece within its sequence
    int len;        // tokens
};
struct Window {
    long long tok0;  // first packed token
    long long ntok;
    int p0, np;      // pieces [p0, p0 + np)
};

// Splits the sequences (lengths len[n], packed back to back) into windows of at
// most `W` tokens and kHostMaxPieces pieces. A sequence is cut only at a
// multiple of 64 tokens from its start, so every chunk is the chunk of the
// uncut call. Zero-length sequences produce no piece.
void plan(const std::vector<long long> &len, long long W, std::vector<Piece> &pieces,
          std::vector<Window> &wins) {
    long long tok = 0;
    Window cur{0, 0, 0, 0};
    auto close = [&]() {
        if (cur.np > 0) wins.push_back(cur);
        cur = Window{tok, 0, (int)pieces.size(), 0};
    };
    for (int n = 0; n < (int)len.size(); ++n) {
        long long o = 0;
        while (o < len[n]) {
            if (cur.np == kHostMaxPieces || cur.ntok == W) close();
            long long take = std::min(len[n] - o, W - cur.ntok);
            if (take < len[n] - o) take = take / kChunk * kChunk;  // a cut: whole chunks
            if (take == 0) {
                close();
                continue;
            }
            pieces.push_back(Piece{n, o, (int)take});
            cur.ntok += take;
            ++cur.np;
            o += take;
            tok += take;
        }
    }
    close();
}

// Window-local packed offsets, passed by value to a one-thread kernel (no host
// staging buffer is needed for them).
struct Offsets {
    int n;
    int v[kHostMaxPieces + 1];
};
__global__ void set_offsets(int *dst, Offsets o) {
    for (int i = 0; i <= o.n; ++i) dst[i] = o.v[i];
}

// Byte sizes of the per-token tensors of one window of W tokens.
struct Sizes {
    size_t q, v, g, beta, out, state;
};
Sizes sizes(long long W, int H, int dk, int dv, kda_dtype dtype, int decay) {
    const size_t e = dtype == KDA_DTYPE_BF16 ? 2 : 4;
    const size_t gper = decay == KDA_DECAY_CHANNEL ? (size_t)dk * 4 : decay == KDA_DECAY_SCALAR ? 4 : 0;
    return Sizes{(size_t)W * H * dk * e, (size_t)W * H * dv * e, (size_t)W * H * gper,
                 (size_t)W * H * 4, (size_t)W * H * dv * e, (size_t)H * dk * dv * 4};
}

// Workspace carve-up of the prefill: two window buffers (inputs, outputs,
// offsets, piece states in and out), then the inner prefill's workspace.
struct HostWs {
    char *q[2], *k[2], *v[2], *g[2], *beta[2], *out[2];
    int *offs[2];
    float *init[2], *fin[2];
    char *inner;
    size_t inner_bytes, total;
};
HostWs carve(char *base, long long W, int H, int dk, int dv, kda_dtype dtype, int decay) {
    const Sizes s = sizes(W, H, dk, dv, dtype, decay);
    HostWs w{};
    size_t off = 0;
    auto take = [&](size_t bytes) {
        char *p = base ? base + off : nullptr;
        off += align_up(bytes, kAlign);
        return p;
    };
    for (int b = 0; b < 2; ++b) {
        w.q[b] = take(s.q);
        w.k[b] = take(s.q);
        w.v[b] = take(s.v);
        w.g[b] = take(s.g);
        w.beta[b] = take(s.beta);
        w.out[b] = take(s.out);
        w.offs[b] = reinterpret_cast<int *>(take((kHostMaxPieces + 1) * sizeof(int)));
        w.init[b] = reinterpret_cast<float *>(take(kHostMaxPieces * s.state));
        w.fin[b] = reinterpret_cast<float *>(take(kHostMaxPieces * s.state));
    }
    // The inner calls carry 1 .. kHostMaxPieces sequences; a single sequence is
    // sized as a one-sequence batch, which can need the segment buffers.
    w.inner_bytes = std::max(kda_chunk_fwd_workspace_size(1, (int)W, H, dk, dv, kHostMaxPieces, dtype),
                             kda_chunk_fwd_workspace_size(1, (int)W, H, dk, dv, 1, dtype));
    w.inner = take(w.inner_bytes);
    w.total = off;
    return w;
}

// Copy streams and events of one host-buffer call, created for the call and
// released at its end (destroying a stream or event with work pending is
// allowed: its resources are freed once the work completes).
struct Pipe {
    cudaStream_t in = nullptr, out = nullptr;
    cudaEvent_t start = nullptr, loaded[2] = {}, computed[2] = {}, drained[2] = {}, done = nullptr;
    bool ok = true;
    Pipe() {
        ok = cudaStreamCreateWithFlags(&in, cudaStreamNonBlocking) == cudaSuccess &&
             cudaStreamCreateWithFlags(&out, cudaStreamNonBlocking) == cudaSuccess &&
             cudaEventCreateWithFlags(&start, cudaEventDisableTiming) == cudaSuccess &&
             cudaEventCreateWithFlags(&done, cudaEventDisableTiming) == cudaSuccess;
        for (int b = 0; b < 2 && ok; ++b)
            ok = cudaEventCreateWithFlags(&loaded[b], cudaEventDisableTiming) == cudaSuccess &&
                 cudaEventCreateWithFlags(&computed[b], cudaEventDisableTiming) == cudaSuccess &&
                 cudaEventCreateWithFlags(&drained[b], cudaEventDisableTiming) == cudaSuccess;
    }
    ~Pipe() {
        for (int b = 0; b < 2; ++b) {
            if (loaded[b]) cudaEventDestroy(loaded[b]);
            if (computed[b]) cudaEventDestroy(computed[b]);
            if (drained[b]) cudaEventDestroy(drained[b]);
        }
        if (start) cudaEventDestroy(start);
        if (done) cudaEventDestroy(done);
        if (in) cudaStreamDestroy(in);
        if (out) cudaStreamDestroy(out);
    }
};

bool aligned16h(const void *p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

}  // namespace
}  // namespace kda

using namespace kda;

extern "C" size_t kda_chunk_fwd_host_workspace_size(int H, int dk, int dv, kda_dtype dtype,
                                                    const kda_options *options,
                                                    int window_tokens) {
    if (H <= 0 || window_tokens <= 0 || window_tokens % kChunk != 0) return 0;
    if (!(dk == dv && (dk == 64 || dk == 128))) return 0;
    if (dtype != KDA_DTYPE_F32 && dtype != KDA_DTYPE_BF16) return 0;
    const int decay = options ? (int)options->decay : (int)KDA_DECAY_CHANNEL;
    if (decay != KDA_DECAY_CHANNEL && decay != KDA_DECAY_SCALAR && decay != KDA_DECAY_NONE) return 0;
    return carve(nullptr, window_tokens, H, dk, dv, dtype, decay).total;
}

extern "C" kda_status kda_chunk_fwd_host(const void *q, const void *k, const void *v,
                                         const float *g, const float *beta, float scale,
                                         const float *init_state, const int32_t *cu_seqlens,
                                         void *out, float *final_state, int B, int T, int H,
                                         int dk, int dv, int num_seqs, kda_dtype dtype,
                                         const kda_options *options, int window_tokens,
                                         void *workspace, size_t workspace_bytes,
                                         cudaStream_t stream) {
    // The arguments of the device call (host pointers are checked the same way,
    // cu_seqlens is a host array here and is read now).
    const kda_status chk = chunk_fwd_check(q, k, v, g, beta, scale, init_state, nullptr, out,
                                           final_state, B, T, H, dk, dv, B, dtype, options);
    if (cu_seqlens ? (B != 1 || num_seqs <= 0) : num_seqs != B) return KDA_ERR_INVALID_ARGUMENT;
    if (chk != KDA_OK) return chk;
    if (options && options->segments < 0) return KDA_ERR_INVALID_ARGUMENT;
    const int decay = options ? (int)options->decay : (int)KDA_DECAY_CHANNEL;
    const size_t need = kda_chunk_fwd_host_workspace_size(H, dk, dv, dtype, options, window_tokens);
    if (need == 0) return KDA_ERR_INVALID_ARGUMENT;
    if (!workspace || workspace_bytes < need ||
        (reinterpret_cast<uintptr_t>(workspace) & (kAlign - 1)) != 0)
        return KDA_ERR_WORKSPACE;

    const long long tokens = (long long)B * T;
    std::vector<long long> len(num_seqs, T);
    if (cu_seqlens) {
        if (cu_seqlens[0] != 0 || cu_seqlens[num_seqs] != tokens) return KDA_ERR_INVALID_ARGUMENT;
        for (int n = 0; n < num_seqs; ++n) {
            if (cu_seqlens[n + 1] < cu_seqlens[n]) return KDA_ERR_INVALID_ARGUMENT;
            len[n] = cu_seqlens[n + 1] - cu_seqlens[n];
        }
    }
    std::vector<Piece> pieces;
    std::vector<Window> wins;
    plan(len, window_tokens, pieces, wins);

    const HostWs ws = carve(static_cast<char *>(workspace), window_tokens, H, dk, dv, dtype, decay);
    const Sizes s = sizes(1, H, dk, dv, dtype, decay);  // per token (and one state)
    const char *hq = static_cast<const char *>(q), *hk = static_cast<const char *>(k);
    const char *hv = static_cast<const char *>(v), *hg = reinterpret_cast<const char *>(g);
    const char *hb = reinterpret_cast<const char *>(beta);
    char *ho = static_cast<char *>(out);
    kda_options opt = options ? *options : kda_options{KDA_DECAY_CHANNEL, KDA_GATE_LOG, 0.f, 0, 0};
    opt.segments = 1;  // windows are packed calls; the serial chain keeps results bit-identical

    // Zero-length sequences: the final state is the initial one (or zeros),
    // written now on the host.
    if (final_state)
        for (int n = 0; n < num_seqs; ++n)
            if (len[n] == 0) {
                float *dst = final_state + (size_t)n * H * dk * dv;
                if (init_state && init_state != final_state)
                    memcpy(dst, init_state + (size_t)n * H * dk * dv, s.state);
                else if (!init_state)
                    memset(dst, 0, s.state);
            }
    if (wins.empty()) return KDA_OK;

    Pipe pp;
    if (!pp.ok) return KDA_ERR_CUDA;
    auto ck = [](cudaError_t e) { return e == cudaSuccess; };
    bool ok = ck(cudaEventRecord(pp.start, stream)) && ck(cudaStreamWaitEvent(pp.in, pp.start, 0)) &&
              ck(cudaStreamWaitEvent(pp.out, pp.start, 0));
    for (size_t w = 0; w < wins.size() && ok; ++w) {
        const Window &wi = wins[w];
        const int b = (int)(w & 1);
        // ---- copies in (window w's inputs; new sequences' initial states)
        if (w >= 2) ok = ok && ck(cudaStreamWaitEvent(pp.in, pp.computed[b], 0));
        const long long t0 = wi.tok0;
        ok = ok && ck(cudaMemcpyAsync(ws.q[b], hq + t0 * s.q, wi.ntok * s.q, cudaMemcpyHostToDevice, pp.in)) &&
             ck(cudaMemcpyAsync(ws.k[b], hk + t0 * s.q, wi.ntok * s.q, cudaMemcpyHostToDevice, pp.in)) &&
             ck(cudaMemcpyAsync(ws.v[b], hv + t0 * s.v, wi.ntok * s.v, cudaMemcpyHostToDevice, pp.in)) &&
             ck(cudaMemcpyAsync(ws.beta[b], hb + t0 * s.beta, wi.ntok * s.beta, cudaMemcpyHostToDevice, pp.in));
        if (s.g) ok = ok && ck(cudaMemcpyAsync(ws.g[b], hg + t0 * s.g, wi.ntok * s.g, cudaMemcpyHostToDevice, pp.in));
        for (int p = 0; p < wi.np && ok; ++p) {
            const Piece &pc = pieces[wi.p0 + p];
            float *dst = ws.init[b] + (size_t)p * H * dk * dv;
            if (pc.off == 0 && init_state)
                ok = ck(cudaMemcpyAsync(dst, init_state + (size_t)pc.seq * H * dk * dv, s.state,
                                        cudaMemcpyHostToDevice, pp.in));
        }
        ok = ok && ck(cudaEventRecord(pp.loaded[b], pp.in));
        // ---- compute on the caller's stream
        ok = ok && ck(cudaStreamWaitEvent(stream, pp.loaded[b], 0));
        if (w >= 2) ok = ok && ck(cudaStreamWaitEvent(stream, pp.drained[b], 0));
        Offsets offs{};
        offs.n = wi.np;
        for (int p = 0; p < wi.np; ++p) offs.v[p + 1] = offs.v[p] + pieces[wi.p0 + p].len;
        if (ok) {
            set_offsets<<<1, 1, 0, stream>>>(ws.offs[b], offs);
            ok = ck(cudaGetLastError());
        }
        for (int p = 0; p < wi.np && ok; ++p) {
            const Piece &pc = pieces[wi.p0 + p];
            float *dst = ws.init[b] + (size_t)p * H * dk * dv;
            if (pc.off > 0)  // continues the previous window's last piece
                ok = ck(cudaMemcpyAsync(dst, ws.fin[b ^ 1] + (size_t)(wins[w - 1].np - 1) * H * dk * dv,
                                        s.state, cudaMemcpyDeviceToDevice, stream));
            else if (!init_state)
                ok = ck(cudaMemsetAsync(dst, 0, s.state, stream));
        }
        if (ok) {
            const kda_status st = kda_chunk_fwd_opt(
                ws.q[b], ws.k[b], ws.v[b], s.g ? reinterpret_cast<const float *>(ws.g[b]) : nullptr,
                reinterpret_cast<const float *>(ws.beta[b]), scale, ws.init[b], ws.offs[b], ws.out[b],
                ws.fin[b], 1, (int)wi.ntok, H, dk, dv, wi.np, dtype, &opt, ws.inner, ws.inner_bytes,
                stream, nullptr);
            if (st != KDA_OK) return st;
        }
        ok = ok && ck(cudaEventRecord(pp.computed[b], stream));
        // ---- copies out (outputs; final states of sequences that end here)
        ok = ok && ck(cudaStreamWaitEvent(pp.out, pp.computed[b], 0)) &&
             ck(cudaMemcpyAsync(ho + t0 * s.out, ws.out[b], wi.ntok * s.out, cudaMemcpyDeviceToHost, pp.out));
        for (int p = 0; p < wi.np && ok && final_state; ++p) {
            const Piece &pc = pieces[wi.p0 + p];
            if (pc.off + pc.len == len[pc.seq])
                ok = ck(cudaMemcpyAsync(final_state + (size_t)pc.seq * H * dk * dv,
                                        ws.fin[b] + (size_t)p * H * dk * dv, s.state,
                                        cudaMemcpyDeviceToHost, pp.out));
        }
        ok = ok && ck(cudaEventRecord(pp.drained[b], pp.out));
    }
    // The caller's stream reaches the end of the call once every copy is done.
    ok = ok && ck(cudaEventRecord(pp.done, pp.out)) && ck(cudaStreamWaitEvent(stream, pp.done, 0));
    return ok ? KDA_OK : KDA_ERR_CUDA;
}

extern "C" size_t kda_decode_host_workspace_size(int N, int H, int dk, int dv, kda_dtype dtype,
                                                 const kda_options *options) {
    if (N <= 0 || H <= 0 || !(dk == dv && (dk == 64 || dk == 128))) return 0;
    if (dtype != KDA_DTYPE_F32 && dtype != KDA_DTYPE_BF16) return 0;
    const int decay = options ? (int)options->decay : (int)KDA_DECAY_CHANNEL;
    const Sizes s = sizes(N, H, dk, dv, dtype, decay);
    return 2 * (2 * align_up(s.q, kAlign) + align_up(s.v, kAlign) + align_up(s.g, kAlign) +
                align_up(s.beta, kAlign) + align_up(s.out, kAlign));
}

extern "C" kda_status kda_decode_host(const void *q, const void *k, const void *v, const float *g,
                                      const float *beta, float scale, float *state, void *out,
                                      int steps, int N, int H, int dk, int dv, kda_dtype dtype,
                                      const kda_options *options, void *workspace,
                                      size_t workspace_bytes, cudaStream_t stream) {
    if (steps < 0 || N <= 0 || H <= 0) return KDA_ERR_INVALID_ARGUMENT;
    if (steps == 0) return KDA_OK;
    if (!q || !k || !v || !beta || !state || !out) return KDA_ERR_INVALID_ARGUMENT;
    if (!aligned16h(q) || !aligned16h(k) || !aligned16h(v) || !aligned16h(out) || !aligned16h(state))
        return KDA_ERR_INVALID_ARGUMENT;
    const size_t need = kda_decode_host_workspace_size(N, H, dk, dv, dtype, options);
    if (need == 0) return (dk == dv && (dk == 64 || dk == 128)) ? KDA_ERR_INVALID_ARGUMENT : KDA_ERR_UNSUPPORTED;
    if (!workspace || workspace_bytes < need ||
        (reinterpret_cast<uintptr_t>(workspace) & (kAlign - 1)) != 0)
        return KDA_ERR_WORKSPACE;
    const int decay = options ? (int)options->decay : (int)KDA_DECAY_CHANNEL;
    if (decay != KDA_DECAY_NONE && !g) return KDA_ERR_INVALID_ARGUMENT;
    const Sizes s = sizes(N, H, dk, dv, dtype, decay);  // one step
    char *base = static_cast<char *>(workspace);
    char *bq[2], *bk[2], *bv[2], *bg[2], *bb[2], *bo[2];
    size_t off = 0;
    auto take = [&](size_t bytes) {
        char *p = base + off;
        off += align_up(bytes, kAlign);
        return p;
    };
    for (int b = 0; b < 2; ++b) {
        bq[b] = take(s.q);
        bk[b] = take(s.q);
        bv[b] = take(s.v);
        bg[b] = take(s.g);
        bb[b] = take(s.beta);
        bo[b] = take(s.out);
    }
    const char *hq = static_cast<const char *>(q), *hk = static_cast<const char *>(k);
    const char *hv = static_cast<const char *>(v), *hg = reinterpret_cast<const char *>(g);
    const char *hb = reinterpret_cast<const char *>(beta);
    char *ho = static_cast<char *>(out);
    Pipe pp;
    if (!pp.ok) return KDA_ERR_CUDA;
    auto ck = [](cudaError_t e) { return e == cudaSuccess; };
    bool ok = ck(cudaEventRecord(pp.start, stream)) && ck(cudaStreamWaitEvent(pp.in, pp.start, 0)) &&
              ck(cudaStreamWaitEvent(pp.out, pp.start, 0));
    for (int t = 0; t < steps && ok; ++t) {
        const int b = t & 1;
        if (t >= 2) ok = ck(cudaStreamWaitEvent(pp.in, pp.computed[b], 0));
        ok = ok && ck(cudaMemcpyAsync(bq[b], hq + (size_t)t * s.q, s.q, cudaMemcpyHostToDevice, pp.in)) &&
             ck(cudaMemcpyAsync(bk[b], hk + (size_t)t * s.q, s.q, cudaMemcpyHostToDevice, pp.in)) &&
             ck(cudaMemcpyAsync(bv[b], hv + (size_t)t * s.v, s.v, cudaMemcpyHostToDevice, pp.in)) &&
             ck(cudaMemcpyAsync(bb[b], hb + (size_t)t * s.beta, s.beta, cudaMemcpyHostToDevice, pp.in));
        if (s.g) ok = ok && ck(cudaMemcpyAsync(bg[b], hg + (size_t)t * s.g, s.g, cudaMemcpyHostToDevice, pp.in));
        ok = ok && ck(cudaEventRecord(pp.loaded[b], pp.in)) && ck(cudaStreamWaitEvent(stream, pp.loaded[b], 0));
        if (t >= 2) ok = ok && ck(cudaStreamWaitEvent(stream, pp.drained[b], 0));
        if (ok) {
            const kda_status st = kda_decode_step_opt(bq[b], bk[b], bv[b],
                                                      s.g ? reinterpret_cast<const float *>(bg[b]) : nullptr,
                                                      reinterpret_cast<const float *>(bb[b]), scale, state,
                                                      bo[b], N, H, dk, dv, dtype, options, stream);
            if (st != KDA_OK) return st;
        }
        ok = ok && ck(cudaEventRecord(pp.computed[b], stream)) && ck(cudaStreamWaitEvent(pp.out, pp.computed[b], 0)) &&
             ck(cudaMemcpyAsync(ho + (size_t)t * s.out, bo[b], s.out, cudaMemcpyDeviceToHost, pp.out)) &&
             ck(cudaEventRecord(pp.drained[b], pp.out));
    }
    ok = ok && ck(cudaEventRecord(pp.done, pp.out)) && ck(cudaStreamWaitEvent(stream, pp.done, 0));
    return ok ? KDA_OK : KDA_ERR_CUDA;
}
