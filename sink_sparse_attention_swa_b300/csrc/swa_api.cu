// swa_api.cu -- the extern "C" entry points of libswa (declared in swa.h):
// argument validation, workspace handling and dispatch to the launchers.
#include <cmath>
#include <cstdint>
#include <cstring>
#include <mutex>
#include <thread>
#include <vector>

#include "swa_internal.h"

namespace {

using namespace swa;

constexpr int kVersion = 100;  // 0.1.0

bool aligned16(const void *p) { return p != nullptr && (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

bool scale_ok(float s) { return std::isfinite(s) && s > 0.f; }

// Common shape checks; returns SWA_OK, SWA_ERR_INVALID_ARG or SWA_ERR_UNSUPPORTED.
int check_heads(int B, int H, int Hkv, int d, int w, int g)
{
    if (B < 1 || H < 1 || Hkv < 1 || w < 1 || g < 0) return SWA_ERR_INVALID_ARG;
    if (H % Hkv != 0) return SWA_ERR_INVALID_ARG;
    if (static_cast<long long>(w) + g > INT32_MAX) return SWA_ERR_INVALID_ARG;
    if (d != 64 && d != 128) return SWA_ERR_UNSUPPORTED;
    return SWA_OK;
}

// The library-owned decode workspace of swa_decode: one buffer per (device,
// stream), so calls on different streams never share partials.  The per-thread
// default stream has one handle for every thread, so that handle is keyed by
// the calling thread too.  A buffer that is outgrown is retired, not freed: a
// kernel enqueued earlier may still read it, and a CUDA graph captured earlier
// may still name it.  Retired buffers are kept until the process exits (the
// sizes grow at least twofold, so they add up to less than the live one).
struct StreamWorkspace {
    cudaStream_t stream;
    std::thread::id thread;
    void *ptr;
    size_t bytes;
};
struct DeviceWorkspaces {
    std::vector<StreamWorkspace> live;
    std::vector<void *> retired;
};
std::mutex g_ws_mu;
DeviceWorkspaces g_ws[kMaxDevices];

// Returns a workspace of at least `need` bytes for (current device, stream),
// growing it if needed; nullptr with *rc set on failure.  Called with g_ws_mu
// held.
void *stream_workspace(cudaStream_t stream, size_t need, int *rc)
{
    const int dev = current_device();
    if (dev < 0) {
        *rc = SWA_ERR_CUDA;
        return nullptr;
    }
    const std::thread::id tid =
        stream == cudaStreamPerThread ? std::this_thread::get_id() : std::thread::id();
    DeviceWorkspaces &D = g_ws[dev];
    StreamWorkspace *W = nullptr;
    for (auto &e : D.live)
        if (e.stream == stream && e.thread == tid) W = &e;
    if (W == nullptr) {
        D.live.push_back(StreamWorkspace{stream, tid, nullptr, 0});
        W = &D.live.back();
    }
    if (W->bytes < need) {
        const size_t grow = need > 2 * W->bytes ? need : 2 * W->bytes;
        void *p = nullptr;
        if (cudaMalloc(&p, grow) != cudaSuccess) {
            // clear the runtime's last-error state, so that the next launch's
            // error check does not report this failure as its own
            (void)cudaGetLastError();
            *rc = SWA_ERR_ALLOC;
            return nullptr;
        }
        if (W->ptr != nullptr) D.retired.push_back(W->ptr);
        W->ptr = p;
        W->bytes = grow;
    }
    return W->ptr;
}

}  // namespace

extern "C" {

int swa_prefill_sink_logit(const void *Q, const void *K, const void *V, void *O, float *lse,
                           const float *sink_logit, int B, int H, int Hkv, int n, int d, int w,
                           int g, float scale, swa_dtype dtype, swa_stream_t stream)
{
    int rc = check_heads(B, H, Hkv, d, w, g);
    if (rc != SWA_OK) return rc;
    if (n < 1 || n > INT32_MAX - 256 || !scale_ok(scale)) return SWA_ERR_INVALID_ARG;
    if (!aligned16(Q) || !aligned16(K) || !aligned16(V) || !aligned16(O)) return SWA_ERR_INVALID_ARG;
    if (lse != nullptr && (reinterpret_cast<uintptr_t>(lse) & 3u)) return SWA_ERR_INVALID_ARG;
    if (sink_logit != nullptr && (reinterpret_cast<uintptr_t>(sink_logit) & 3u))
        return SWA_ERR_INVALID_ARG;
    if (static_cast<long long>(B) * H * ((n + 127) / 128) > INT32_MAX) return SWA_ERR_INVALID_ARG;
    cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
    if (dtype == SWA_BF16)
        return launch_prefill_bf16(Q, K, V, O, lse, sink_logit, B, H, Hkv, n, n, d, w, g, scale,
                                   nullptr, 1, 0, st);
    if (dtype == SWA_F32)
        return launch_prefill_f32(Q, K, V, O, lse, sink_logit, B, H, Hkv, n, n, d, w, g, scale,
                                  nullptr, 1, 0, st);
    return SWA_ERR_INVALID_ARG;
}

}  // extern "C"

namespace {
// swa_prefill_pattern, with an optional tile-walk log for the bf16 kernels.
int prefill_pattern_impl(const void *Q, const void *K, const void *V, void *O, float *lse,
                         const float *sink_logit, int B, int H, int Hkv, int n, int d,
                         swa_pattern pattern, int w, int g, int r, float scale, swa_dtype dtype,
                         swa_stream_t stream, int32_t *walk)
{
    if (pattern == SWA_PATTERN_WINDOW && walk == nullptr)
        return swa_prefill_sink_logit(Q, K, V, O, lse, sink_logit, B, H, Hkv, n, d, w, g, scale,
                                      dtype, stream);
    if (pattern != SWA_PATTERN_WINDOW && pattern != SWA_PATTERN_DILATED &&
        pattern != SWA_PATTERN_STRIDED && pattern != SWA_PATTERN_LANDMARK)
        return SWA_ERR_INVALID_ARG;
    if (r < 1 || n < 1 || n > INT32_MAX - 256) return SWA_ERR_INVALID_ARG;
    if (pattern == SWA_PATTERN_STRIDED) w = n;  // no limit on the number of strides back
    int rc = check_heads(B, H, Hkv, d, w, g);
    if (rc != SWA_OK) return rc;
    // residue classes carry no sink columns (a sink below g belongs to one class only)
    if ((pattern == SWA_PATTERN_DILATED || pattern == SWA_PATTERN_STRIDED) && g != 0)
        return SWA_ERR_UNSUPPORTED;
    if (!scale_ok(scale)) return SWA_ERR_INVALID_ARG;
    if (!aligned16(Q) || !aligned16(K) || !aligned16(V) || !aligned16(O)) return SWA_ERR_INVALID_ARG;
    if (lse != nullptr && (reinterpret_cast<uintptr_t>(lse) & 3u)) return SWA_ERR_INVALID_ARG;
    if (sink_logit != nullptr && (reinterpret_cast<uintptr_t>(sink_logit) & 3u))
        return SWA_ERR_INVALID_ARG;
    int R = 1, rl = 0, wk = w;
    if (pattern == SWA_PATTERN_LANDMARK) {
        rl = r;
    } else if (pattern != SWA_PATTERN_WINDOW) {
        R = r < n ? r : n;  // strides past the sequence: each class is one row
        const int rows = (n + R - 1) / R;
        if (pattern == SWA_PATTERN_STRIDED || wk > rows) wk = rows;
    }
    const long long n_hi = (n + R - 1) / R;
    // work items (tensor-core kernels) and CTAs (fp32 kernel) stay below 2^31
    if (static_cast<long long>(B) * H * (((n_hi + 127) / 128) * R) > INT32_MAX ||
        ((n_hi + 63) / 64) * R > INT32_MAX)
        return SWA_ERR_INVALID_ARG;
    cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
    if (dtype == SWA_BF16)
        return launch_prefill_bf16(Q, K, V, O, lse, sink_logit, B, H, Hkv, n, n, d, wk, g, scale,
                                   nullptr, R, rl, st, walk);
    if (walk != nullptr) return SWA_ERR_UNSUPPORTED;  // the log is of the tensor-core kernels
    if (dtype == SWA_F32)
        return launch_prefill_f32(Q, K, V, O, lse, sink_logit, B, H, Hkv, n, n, d, wk, g, scale,
                                  nullptr, R, rl, st);
    return SWA_ERR_INVALID_ARG;
}

}  // namespace

extern "C" {

int swa_prefill_pattern(const void *Q, const void *K, const void *V, void *O, float *lse,
                        const float *sink_logit, int B, int H, int Hkv, int n, int d,
                        swa_pattern pattern, int w, int g, int r, float scale, swa_dtype dtype,
                        swa_stream_t stream)
{
    return prefill_pattern_impl(Q, K, V, O, lse, sink_logit, B, H, Hkv, n, d, pattern, w, g, r,
                                scale, dtype, stream, nullptr);
}

int swa_debug_prefill_walk(const void *Q, const void *K, const void *V, void *O, int B, int H,
                           int Hkv, int n, int d, swa_pattern pattern, int w, int g, int r,
                           float scale, int32_t *log, int64_t log_entries, swa_stream_t stream)
{
    if (log == nullptr || (reinterpret_cast<uintptr_t>(log) & 15u) || log_entries < 0)
        return SWA_ERR_INVALID_ARG;
    cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
    // header: the entry count (zero), then the capacity as a 64-bit count
    const int64_t header[4] = {0, log_entries, 0, 0};
    if (cudaMemcpyAsync(log, header, sizeof(header), cudaMemcpyHostToDevice, st) != cudaSuccess ||
        cudaStreamSynchronize(st) != cudaSuccess)
        return SWA_ERR_CUDA;
    return prefill_pattern_impl(Q, K, V, O, nullptr, nullptr, B, H, Hkv, n, d, pattern, w, g, r,
                                scale, SWA_BF16, stream, log);
}

int swa_debug_prefill_cta_pairs(const void *Q, const void *K, const void *V, void *O, float *lse,
                                int B, int H, int Hkv, int n, int d, int w, int g, float scale,
                                swa_stream_t stream)
{
    int rc = check_heads(B, H, Hkv, d, w, g);
    if (rc != SWA_OK) return rc;
    if (n < 1 || n > INT32_MAX - 256 || !scale_ok(scale)) return SWA_ERR_INVALID_ARG;
    if (!aligned16(Q) || !aligned16(K) || !aligned16(V) || !aligned16(O)) return SWA_ERR_INVALID_ARG;
    if (lse != nullptr && (reinterpret_cast<uintptr_t>(lse) & 3u)) return SWA_ERR_INVALID_ARG;
    if (static_cast<long long>(B) * H * ((n + 127) / 128) > INT32_MAX) return SWA_ERR_INVALID_ARG;
    return launch_prefill_bf16(Q, K, V, O, lse, nullptr, B, H, Hkv, n, n, d, w, g, scale, nullptr,
                               1, 0, reinterpret_cast<cudaStream_t>(stream), nullptr, true);
}

size_t swa_prefill_chunk_workspace_bytes(int B, int Hkv, int T, int d, int w, int g,
                                         swa_dtype dtype)
{
    if (check_heads(B, Hkv, Hkv, d, w, g) != SWA_OK || T < 1) return 0;
    if (dtype != SWA_BF16 && dtype != SWA_F32) return 0;
    const size_t elem = dtype == SWA_BF16 ? 2 : 4;
    return 2 * static_cast<size_t>(B) * Hkv * static_cast<size_t>(chunk_rows_max(w, g, T)) * d *
           elem;
}

int swa_prefill_chunk(const void *Q, const void *k_new, const void *v_new, void *Kcache,
                      void *Vcache, const int32_t *pos0, void *O, float *lse,
                      const float *sink_logit, int B, int H, int Hkv, int T, int d, int w, int g,
                      float scale, int append, swa_dtype dtype, void *workspace,
                      size_t workspace_bytes, swa_stream_t stream)
{
    int rc = check_heads(B, H, Hkv, d, w, g);
    if (rc != SWA_OK) return rc;
    if (T < 1 || T > INT32_MAX - 256 || !scale_ok(scale)) return SWA_ERR_INVALID_ARG;
    if (dtype != SWA_BF16 && dtype != SWA_F32) return SWA_ERR_INVALID_ARG;
    if (!aligned16(Q) || !aligned16(k_new) || !aligned16(v_new) || !aligned16(Kcache) ||
        !aligned16(Vcache) || !aligned16(O) || pos0 == nullptr ||
        (reinterpret_cast<uintptr_t>(pos0) & 3u))
        return SWA_ERR_INVALID_ARG;
    if (lse != nullptr && (reinterpret_cast<uintptr_t>(lse) & 3u)) return SWA_ERR_INVALID_ARG;
    if (sink_logit != nullptr && (reinterpret_cast<uintptr_t>(sink_logit) & 3u))
        return SWA_ERR_INVALID_ARG;
    const long long rows = chunk_rows_max(w, g, T);
    if (rows > INT32_MAX - 256) return SWA_ERR_INVALID_ARG;
    if (static_cast<long long>(B) * H * ((T + 127) / 128) > INT32_MAX) return SWA_ERR_INVALID_ARG;
    const size_t need = swa_prefill_chunk_workspace_bytes(B, Hkv, T, d, w, g, dtype);
    if (workspace == nullptr || workspace_bytes < need || !aligned16(workspace))
        return SWA_ERR_WORKSPACE;
    cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
    uint8_t *Kx = static_cast<uint8_t *>(workspace);
    uint8_t *Vx = Kx + need / 2;
    rc = launch_chunk_gather(Kx, Vx, Kcache, Vcache, k_new, v_new, pos0, B, Hkv, T, d, w, g, dtype,
                             st);
    if (rc != SWA_OK) return rc;
    if (append) {  // the key lists are already copied out, so the ring may be overwritten
        rc = launch_cache_append(Kcache, Vcache, k_new, v_new, pos0, T, B, Hkv, d, w, g, dtype, st);
        if (rc != SWA_OK) return rc;
    }
    if (dtype == SWA_BF16)
        return launch_prefill_bf16(Q, Kx, Vx, O, lse, sink_logit, B, H, Hkv, T,
                                   static_cast<int>(rows), d, w, g, scale, pos0, 1, 0, st);
    return launch_prefill_f32(Q, Kx, Vx, O, lse, sink_logit, B, H, Hkv, T, static_cast<int>(rows),
                              d, w, g, scale, pos0, 1, 0, st);
}

int swa_prefill_ex(const void *Q, const void *K, const void *V, void *O, float *lse, int B, int H,
                   int Hkv, int n, int d, int w, int g, float scale, swa_dtype dtype,
                   swa_stream_t stream)
{
    return swa_prefill_sink_logit(Q, K, V, O, lse, nullptr, B, H, Hkv, n, d, w, g, scale, dtype,
                                  stream);
}

int swa_prefill(const void *Q, const void *K, const void *V, void *O, int B, int H, int Hkv, int n,
                int d, int w, int g, float scale, swa_stream_t stream)
{
    return swa_prefill_ex(Q, K, V, O, nullptr, B, H, Hkv, n, d, w, g, scale, SWA_BF16, stream);
}

size_t swa_decode_workspace_bytes(int B, int H, int Hkv, int d, int w, int g, int num_splits)
{
    if (check_heads(B, H, Hkv, d, w, g) != SWA_OK || num_splits < 0 || num_splits > 1024) return 0;
    return decode_workspace_bytes(B, H, Hkv, d, decode_ctas(B, H, Hkv, w, g, num_splits));
}

int swa_decode_sink_logit(const void *q, const void *Kcache, const void *Vcache,
                          const int32_t *pos, const float *sink_logit, int B, int H, int Hkv,
                          int d, int w, int g, float scale, void *O, float *lse, swa_dtype dtype,
                          int num_splits, void *workspace, size_t workspace_bytes,
                          swa_stream_t stream)
{
    int rc = check_heads(B, H, Hkv, d, w, g);
    if (rc != SWA_OK) return rc;
    if (dtype != SWA_BF16 && dtype != SWA_F32) return SWA_ERR_INVALID_ARG;
    if (!scale_ok(scale) || num_splits < 0 || num_splits > 1024) return SWA_ERR_INVALID_ARG;
    if (!aligned16(q) || !aligned16(Kcache) || !aligned16(Vcache) || !aligned16(O) ||
        pos == nullptr || (reinterpret_cast<uintptr_t>(pos) & 3u))
        return SWA_ERR_INVALID_ARG;
    if (lse != nullptr && (reinterpret_cast<uintptr_t>(lse) & 3u)) return SWA_ERR_INVALID_ARG;
    if (sink_logit != nullptr && (reinterpret_cast<uintptr_t>(sink_logit) & 3u))
        return SWA_ERR_INVALID_ARG;
    const int ctas = decode_ctas(B, H, Hkv, w, g, num_splits);
    const size_t need = decode_workspace_bytes(B, H, Hkv, d, ctas);
    if (workspace == nullptr || workspace_bytes < need || !aligned16(workspace))
        return SWA_ERR_WORKSPACE;
    return launch_decode(q, Kcache, Vcache, pos, sink_logit, B, H, Hkv, d, w, g, scale, O, lse,
                         dtype, ctas, workspace, reinterpret_cast<cudaStream_t>(stream));
}

int swa_decode_ex(const void *q, const void *Kcache, const void *Vcache, const int32_t *pos, int B,
                  int H, int Hkv, int d, int w, int g, float scale, void *O, float *lse,
                  swa_dtype dtype, int num_splits, void *workspace, size_t workspace_bytes,
                  swa_stream_t stream)
{
    return swa_decode_sink_logit(q, Kcache, Vcache, pos, nullptr, B, H, Hkv, d, w, g, scale, O, lse,
                                 dtype, num_splits, workspace, workspace_bytes, stream);
}

int swa_decode(const void *q, const void *Kcache, const void *Vcache, const int32_t *pos, int B,
               int H, int Hkv, int d, int w, int g, float scale, void *O, swa_stream_t stream)
{
    int rc = check_heads(B, H, Hkv, d, w, g);
    if (rc != SWA_OK) return rc;
    const size_t need = decode_workspace_bytes(B, H, Hkv, d, decode_ctas(B, H, Hkv, w, g, 0));
    cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
    // the lock is held until both kernels are enqueued, so the table is never
    // changed under a call that is still choosing its buffer
    std::lock_guard<std::mutex> lk(g_ws_mu);
    void *ws = stream_workspace(st, need, &rc);
    if (ws == nullptr) return rc;
    return swa_decode_ex(q, Kcache, Vcache, pos, B, H, Hkv, d, w, g, scale, O, nullptr, SWA_BF16, 0,
                         ws, need, stream);
}

int swa_cache_append(void *Kcache, void *Vcache, const void *k_new, const void *v_new,
                     const int32_t *pos0, int T, int B, int Hkv, int d, int w, int g,
                     swa_dtype dtype, swa_stream_t stream)
{
    int rc = check_heads(B, Hkv, Hkv, d, w, g);
    if (rc != SWA_OK) return rc;
    if (T < 0 || (dtype != SWA_BF16 && dtype != SWA_F32)) return SWA_ERR_INVALID_ARG;
    if (T == 0) return SWA_OK;
    if (!aligned16(Kcache) || !aligned16(Vcache) || !aligned16(k_new) || !aligned16(v_new) ||
        pos0 == nullptr || (reinterpret_cast<uintptr_t>(pos0) & 3u))
        return SWA_ERR_INVALID_ARG;
    return launch_cache_append(Kcache, Vcache, k_new, v_new, pos0, T, B, Hkv, d, w, g, dtype,
                               reinterpret_cast<cudaStream_t>(stream));
}

int64_t swa_count_pairs(int64_t n, int64_t w, int64_t g)
{
    if (n < 0 || w < 1 || g < 0) return -1;
    // window part: row i reads min(i+1, w) keys
    int64_t total = (n <= w) ? n * (n + 1) / 2 : w * (w + 1) / 2 + (n - w) * w;
    // sinks below the window start: row i >= w gains min(g, i-w+1)
    const int64_t m = n - w;
    if (m > 0) total += (m <= g) ? m * (m + 1) / 2 : g * (g + 1) / 2 + (m - g) * g;
    return total;
}

int swa_enumerate_tiles(int64_t n, int64_t w, int64_t g, int BM, int BN, int32_t *cls, size_t cap)
{
    if (n < 1 || n > INT32_MAX / 2 || w < 1 || g < 0 || BM < 1 || BN < 1 || cls == nullptr)
        return SWA_ERR_INVALID_ARG;
    const int64_t nq = (n + BM - 1) / BM, nk = (n + BN - 1) / BN;
    if (static_cast<uint64_t>(nq) * static_cast<uint64_t>(nk) > cap) return SWA_ERR_INVALID_ARG;
    const int wi = static_cast<int>(w < INT32_MAX / 2 ? w : INT32_MAX / 2);
    const int gi = static_cast<int>(g < INT32_MAX / 2 ? g : INT32_MAX / 2);
    std::memset(cls, 0, sizeof(int32_t) * static_cast<size_t>(nq * nk));
    for (int qt = 0; qt < nq; ++qt) {
        const TileRange tr = tile_range(qt, static_cast<int>(n), wi, gi, BM, BN);
        for (int j = 0; j < tr.count; ++j) {
            const int kt = tile_kt(tr, j);
            cls[static_cast<size_t>(qt) * nk + kt] = tile_full(tr, kt, wi, gi, BN) ? 2 : 1;
        }
    }
    return SWA_OK;
}

int swa_enumerate_landmark_tiles(int64_t n, int64_t w, int64_t g, int64_t r, int BM, int BN,
                                 int32_t *cls, size_t cap)
{
    if (n < 1 || n > INT32_MAX / 2 || w < 1 || g < 0 || r < 1 || BM < 1 || BN < 1 ||
        cls == nullptr)
        return SWA_ERR_INVALID_ARG;
    const int64_t nl = (n + r - 1) / r;  // landmarks 0, r, 2r, ...
    const int64_t nq = (n + BM - 1) / BM, nk = (nl + BN - 1) / BN;
    if (static_cast<uint64_t>(nq) * static_cast<uint64_t>(nk) > cap) return SWA_ERR_INVALID_ARG;
    const int wi = static_cast<int>(w < INT32_MAX / 2 ? w : INT32_MAX / 2);
    const int gi = static_cast<int>(g < INT32_MAX / 2 ? g : INT32_MAX / 2);
    const int ri = static_cast<int>(r < INT32_MAX / 2 ? r : INT32_MAX / 2);
    std::memset(cls, 0, sizeof(int32_t) * static_cast<size_t>(nq * nk));
    for (int qt = 0; qt < nq; ++qt) {
        TileRange tr = tile_range(qt, static_cast<int>(n), wi, gi, BM, BN);
        tr.count = 0;
        add_landmarks(tr, wi, gi, ri, BN);
        for (int j = 0; j < tr.nl; ++j) {
            const int lt = tr.lt0 + j;
            cls[static_cast<size_t>(qt) * nk + lt] = land_full(tr, lt, wi, gi, ri, BN) ? 2 : 1;
        }
    }
    return SWA_OK;
}

int swa_chunk_key_positions(int64_t pos0, int w, int g, int T, int64_t *position, size_t cap,
                            int32_t *query_offset)
{
    if (pos0 < 0 || pos0 > INT32_MAX - static_cast<int64_t>(T) || w < 1 || g < 0 || T < 1 ||
        position == nullptr || query_offset == nullptr ||
        static_cast<long long>(w) + g > INT32_MAX)
        return SWA_ERR_INVALID_ARG;
    const long long rows = chunk_rows_max(w, g, T);
    // the row count is the return value, so it must stay below the error codes' range
    if (rows > INT32_MAX || static_cast<unsigned long long>(rows) > cap) return SWA_ERR_INVALID_ARG;
    const int ps = static_cast<int>(pos0);
    const int S = chunk_sinks(ps, g), W0 = chunk_w0(ps, w, g), pad = chunk_pad(ps, w, g);
    const long long L = static_cast<long long>(chunk_keys(ps, w, g, T));
    for (long long r = 0; r < rows; ++r) {
        int64_t v = -1;  // padding, or past the list
        if (r < L) {
            if (r < S)
                v = r;
            else if (r >= S + pad)
                v = W0 + (r - S - pad);
        }
        position[r] = v;
    }
    *query_offset = chunk_offset(ps, w, g);
    return static_cast<int>(rows);
}

int swa_cache_slot(int64_t p, int w, int g, int32_t *ring_slot, int32_t *sink_slot)
{
    if (p < 0 || w < 1 || g < 0 || static_cast<long long>(w) + g > INT32_MAX ||
        ring_slot == nullptr || sink_slot == nullptr)
        return SWA_ERR_INVALID_ARG;
    *ring_slot = static_cast<int32_t>(p % w);
    *sink_slot = (p < g) ? static_cast<int32_t>(w + p) : -1;
    return SWA_OK;
}

int swa_debug_inject_stall(int kind, int64_t wait_ns)
{
    if (kind != 0 && kind != SWA_STALL_PREFILL && kind != SWA_STALL_DECODE) return SWA_ERR_INVALID_ARG;
    return set_injected_stall(kind, wait_ns);
}

int swa_debug_shrink_bounds(void)
{
#ifdef SWA_DEBUG
    return set_injected_stall(INJECT_SHRINK_BOUNDS, 0);
#else
    return SWA_ERR_UNSUPPORTED;  // a product build has no checks to shrink
#endif
}

int swa_get_device_status(swa_stream_t stream)
{
    return read_and_clear_status(reinterpret_cast<cudaStream_t>(stream));
}

const char *swa_status_string(int status)
{
    switch (status) {
    case SWA_OK: return "SWA_OK";
    case SWA_ERR_INVALID_ARG: return "SWA_ERR_INVALID_ARG";
    case SWA_ERR_UNSUPPORTED: return "SWA_ERR_UNSUPPORTED";
    case SWA_ERR_CUDA: return "SWA_ERR_CUDA";
    case SWA_ERR_DEVICE_TIMEOUT: return "SWA_ERR_DEVICE_TIMEOUT";
    case SWA_ERR_ALLOC: return "SWA_ERR_ALLOC";
    case SWA_ERR_WORKSPACE: return "SWA_ERR_WORKSPACE";
    case SWA_ERR_DEVICE_BOUNDS: return "SWA_ERR_DEVICE_BOUNDS";
    default: return "SWA_ERR_UNKNOWN";
    }
}

int swa_version(void) { return kVersion; }

int swa_selftest_umma(const void *A, const void *Bk, const void *Bn, float *D1, float *D2,
                      swa_stream_t stream)
{
    if (!aligned16(A) || !aligned16(Bk) || !aligned16(Bn) || !aligned16(D1) || !aligned16(D2))
        return SWA_ERR_INVALID_ARG;
    return launch_selftest_umma(A, Bk, Bn, D1, D2, reinterpret_cast<cudaStream_t>(stream));
}

}  // extern "C"
