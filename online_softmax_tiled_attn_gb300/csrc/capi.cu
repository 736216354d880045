// capi.cu -- the extern "C" boundary of libosmattn.so (declared in include/osm_attn.h).
//
// Every argument is checked here, on the host, before anything is launched; a rejected call
// launches nothing and touches no buffer.
#include <cuda_runtime.h>

#include <cmath>
#include <cstdint>
#include <mutex>

#include "osm_internal.h"

namespace {

bool aligned(const void* p, uintptr_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }

// [a, a + a_bytes) and [b, b + b_bytes) share at least one byte.
bool overlaps(const void* a, uint64_t a_bytes, const void* b, uint64_t b_bytes) {
    const uintptr_t x = reinterpret_cast<uintptr_t>(a), y = reinterpret_cast<uintptr_t>(b);
    return x < y + b_bytes && y < x + a_bytes;
}

// a * b without signed overflow, for non-negative operands; false when it would overflow.
bool mul_ok(int64_t a, int64_t b, int64_t* out) {
    if (a != 0 && b > INT64_MAX / a) return false;
    *out = a * b;
    return true;
}

// The checks and dispatch shared by the split-key and grouped-head entry points: Q, O
// [B, H, Nq, d], K, V [B, H_kv, Nk, d], LSE [B, H, Nq], optional kv_lens [B] (device),
// n_splits key ranges (1: one pass, no workspace; > 1: partial states in ws_O, ws_LSE).
int attention_call(const void* Q, const void* K, const void* V, void* O, float* LSE, int64_t B,
                   int64_t H, int64_t H_kv, int64_t Nq, int64_t Nk, int64_t d, float scale,
                   int causal, const int32_t* kv_lens, int64_t n_splits, float* ws_O,
                   float* ws_LSE, void* stream, const uint32_t* mask = nullptr,
                   int64_t mask_bs = 0, int64_t mask_hs = 0, uint32_t* tile_map = nullptr,
                   int64_t tile_map_words = 0) {
    if (B < 0 || H < 0 || H_kv < 0 || Nq < 0 || Nk < 0 || d < 0) return FA_ERR_INVALID_ARG;
    if (H > 0 && (H_kv < 1 || H % H_kv != 0)) return FA_ERR_INVALID_ARG;
    int64_t bh, rows, q_elems, bh_kv, kv_rows, kv_elems;
    if (!mul_ok(B, H, &bh) || !mul_ok(bh, Nq, &rows) || !mul_ok(rows, d, &q_elems) ||
        !mul_ok(B, H_kv, &bh_kv) || !mul_ok(bh_kv, Nk, &kv_rows) ||
        !mul_ok(kv_rows, d, &kv_elems) || q_elems > INT64_MAX / 4 || kv_elems > INT64_MAX / 4)
        return FA_ERR_INVALID_ARG;
    if (rows == 0) return FA_OK;
    if (d != 64 && d != 128) return FA_ERR_UNSUPPORTED;
    if (!O || !aligned(O, 16) || (LSE && !aligned(LSE, 4))) return FA_ERR_INVALID_ARG;
    if (!std::isfinite(scale) || !(scale > 0.f)) return FA_ERR_INVALID_ARG;
    const uint64_t q_bytes = static_cast<uint64_t>(q_elems) * 2;
    const uint64_t lse_bytes = static_cast<uint64_t>(rows) * 4;
    if (LSE && overlaps(LSE, lse_bytes, O, q_bytes)) return FA_ERR_INVALID_ARG;
    const cudaStream_t st = static_cast<cudaStream_t>(stream);
    if (Nk == 0)  // no key at all: every row is empty (O = 0, LSE = -inf)
        return osm::fa_fwd_splitkv_launch(nullptr, nullptr, nullptr, O, LSE,
                                          osm::AttnShape{bh, 1, 1, Nq, 0, d, nullptr, 0}, scale,
                                          causal != 0, 0, nullptr, nullptr, st);
    if (!Q || !K || !V) return FA_ERR_INVALID_ARG;
    if (!aligned(Q, 16) || !aligned(K, 16) || !aligned(V, 16)) return FA_ERR_INVALID_ARG;
    if (n_splits < 1 || n_splits > 256) return FA_ERR_INVALID_ARG;
    const uint64_t kv_bytes = static_cast<uint64_t>(kv_elems) * 2;
    if (overlaps(O, q_bytes, Q, q_bytes) || overlaps(O, q_bytes, K, kv_bytes) ||
        overlaps(O, q_bytes, V, kv_bytes))
        return FA_ERR_INVALID_ARG;
    if (LSE && (overlaps(LSE, lse_bytes, Q, q_bytes) || overlaps(LSE, lse_bytes, K, kv_bytes) ||
                overlaps(LSE, lse_bytes, V, kv_bytes)))
        return FA_ERR_INVALID_ARG;
    if (mask) {
        // Rows of 4 * ceil(Nk / 128) words, 16-byte aligned: the strides are whole 16-byte
        // groups, and the furthest row must not reach an output.
        const int64_t words = 4 * ((Nk + 127) / 128);
        if (!aligned(mask, 16) || mask_bs < 0 || mask_hs < 0 || mask_bs % 4 != 0 ||
            mask_hs % 4 != 0)
            return FA_ERR_INVALID_ARG;
        int64_t ext, t1, t2, t3;
        if (!mul_ok(B - 1, mask_bs, &t1) || !mul_ok(H - 1, mask_hs, &t2) ||
            !mul_ok(Nq, words, &t3) || t1 > INT64_MAX / 8 || t2 > INT64_MAX / 8 ||
            t3 > INT64_MAX / 8)
            return FA_ERR_INVALID_ARG;
        ext = (t1 + t2 + t3) * 4;
        if (overlaps(mask, static_cast<uint64_t>(ext), O, q_bytes) ||
            (LSE && overlaps(mask, static_cast<uint64_t>(ext), LSE, lse_bytes)))
            return FA_ERR_INVALID_ARG;
        if (tile_map) {
            // written by the pre-pass, then read by the attention: apart from every input
            // and output
            const int64_t need = osm::mask_tile_map_words(B, H, Nq, Nk, mask_bs, mask_hs);
            if (!aligned(tile_map, 4) || need < 0 || tile_map_words < need ||
                need > INT64_MAX / 8)
                return FA_ERR_INVALID_ARG;
            const uint64_t tm_bytes = static_cast<uint64_t>(need) * 4;
            const void* other[6] = {Q, K, V, O, LSE, mask};
            const uint64_t other_bytes[6] = {q_bytes, kv_bytes, kv_bytes, q_bytes,
                                             LSE ? lse_bytes : 0, static_cast<uint64_t>(ext)};
            for (int i = 0; i < 6; ++i)
                if (overlaps(tile_map, tm_bytes, other[i], other_bytes[i]))
                    return FA_ERR_INVALID_ARG;
        }
    } else if (tile_map) {
        return FA_ERR_INVALID_ARG;
    }
    const uint64_t len_bytes = static_cast<uint64_t>(B) * 4;
    if (kv_lens && (!aligned(kv_lens, 4) || overlaps(kv_lens, len_bytes, O, q_bytes) ||
                    (LSE && overlaps(kv_lens, len_bytes, LSE, lse_bytes))))
        return FA_ERR_INVALID_ARG;
    if (n_splits > 1) {
        int64_t wo, wl;
        if (!mul_ok(q_elems, n_splits, &wo) || !mul_ok(rows, n_splits, &wl) || wo > INT64_MAX / 4)
            return FA_ERR_INVALID_ARG;
        if (!ws_O || !ws_LSE || !aligned(ws_O, 16) || !aligned(ws_LSE, 4))
            return FA_ERR_INVALID_ARG;
        const uint64_t wo_bytes = static_cast<uint64_t>(wo) * 4;
        const uint64_t wl_bytes = static_cast<uint64_t>(wl) * 4;
        const void* ins[4] = {Q, K, V, kv_lens};
        const uint64_t in_bytes[4] = {q_bytes, kv_bytes, kv_bytes, kv_lens ? len_bytes : 0};
        for (int i = 0; i < 4; ++i)
            if (overlaps(ws_O, wo_bytes, ins[i], in_bytes[i]) ||
                overlaps(ws_LSE, wl_bytes, ins[i], in_bytes[i]))
                return FA_ERR_INVALID_ARG;
        if (overlaps(ws_O, wo_bytes, O, q_bytes) || overlaps(ws_LSE, wl_bytes, O, q_bytes) ||
            overlaps(ws_O, wo_bytes, ws_LSE, wl_bytes) ||
            (LSE && (overlaps(ws_O, wo_bytes, LSE, lse_bytes) ||
                     overlaps(ws_LSE, wl_bytes, LSE, lse_bytes))))
            return FA_ERR_INVALID_ARG;
    }
    return osm::fa_fwd_splitkv_launch(
        Q, K, V, O, LSE,
        osm::AttnShape{B, H, H_kv, Nq, Nk, d, kv_lens, 0, mask, mask_bs, mask_hs, tile_map},
        scale, causal != 0, n_splits, ws_O, ws_LSE, st);
}

}  // namespace

namespace {

// fa_fwd_host's copy streams and events, one set per device, made on first use and kept for
// the life of the process; calls enqueue under one lock, so that the events of one call are
// not re-recorded by another before its waits are enqueued.
constexpr int kHostPipeMaxChunks = 64;
constexpr int kHostPipeMaxDevices = 64;
struct HostPipe {
    bool ready = false;
    // One stream each way.  (A host-to-device stream per input, Q, K and V, made the copies of
    // B2 H32 N8192 d128 slower, not faster: 723 against 914 TFLOP/s end to end.)
    cudaStream_t h2d = nullptr, d2h = nullptr;
    cudaEvent_t start = nullptr, done = nullptr;
    cudaEvent_t in[kHostPipeMaxChunks] = {}, out[kHostPipeMaxChunks] = {};
};
std::mutex g_host_pipe_mu;
HostPipe g_host_pipes[kHostPipeMaxDevices];

// The current device's pipe (made if needed), or nullptr.  Caller holds g_host_pipe_mu.
HostPipe* host_pipe() {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kHostPipeMaxDevices)
        return nullptr;
    HostPipe& p = g_host_pipes[dev];
    if (p.ready) return &p;
    bool ok = cudaStreamCreateWithFlags(&p.h2d, cudaStreamNonBlocking) == cudaSuccess &&
              cudaStreamCreateWithFlags(&p.d2h, cudaStreamNonBlocking) == cudaSuccess &&
              cudaEventCreateWithFlags(&p.start, cudaEventDisableTiming) == cudaSuccess &&
              cudaEventCreateWithFlags(&p.done, cudaEventDisableTiming) == cudaSuccess;
    for (int c = 0; ok && c < kHostPipeMaxChunks; ++c)
        ok = cudaEventCreateWithFlags(&p.in[c], cudaEventDisableTiming) == cudaSuccess &&
             cudaEventCreateWithFlags(&p.out[c], cudaEventDisableTiming) == cudaSuccess;
    if (!ok) return nullptr;  // what was made stays for the next attempt to reuse
    p.ready = true;
    return &p;
}

}  // namespace

extern "C" {

int fa_fwd_gqa_plan(int64_t B, int64_t H, int64_t H_kv, int64_t Nq, int64_t Nk, int64_t d,
                    int64_t n_splits, int64_t* splits_out, int64_t* ws_o_floats,
                    int64_t* ws_lse_floats) {
    if (!splits_out || !ws_o_floats || !ws_lse_floats) return FA_ERR_INVALID_ARG;
    if (B < 0 || H < 0 || H_kv < 0 || Nq < 0 || Nk < 0 || d < 0 || n_splits < 0 ||
        n_splits > 256)
        return FA_ERR_INVALID_ARG;
    if (H > 0 && (H_kv < 1 || H % H_kv != 0)) return FA_ERR_INVALID_ARG;
    int64_t bh, rows, elems, bh_kv;
    if (!mul_ok(B, H, &bh) || !mul_ok(bh, Nq, &rows) || !mul_ok(rows, d, &elems) ||
        !mul_ok(B, H_kv, &bh_kv))
        return FA_ERR_INVALID_ARG;
    if (d != 64 && d != 128) return FA_ERR_UNSUPPORTED;
    // The kernel runs the query heads of a key/value head as one packed row block.
    const int64_t packed_rows = H_kv > 0 && H > 0 ? (H / H_kv) * Nq : Nq;
    const int64_t splits = osm::splitkv_choose_splits(bh_kv, packed_rows, Nk, n_splits);
    int64_t o = 0, l = 0;
    if (splits > 1 && (!mul_ok(elems, splits, &o) || !mul_ok(rows, splits, &l)))
        return FA_ERR_INVALID_ARG;
    *splits_out = splits;
    *ws_o_floats = splits > 1 ? o : 0;
    *ws_lse_floats = splits > 1 ? l : 0;
    return FA_OK;
}

int fa_fwd(const void* Q, const void* K, const void* V, void* O, float* LSE, int64_t B,
           int64_t H, int64_t N, int64_t d, float scale, int causal, void* stream) {
    if (B < 0 || H < 0 || N < 0 || d < 0) return FA_ERR_INVALID_ARG;
    int64_t bh, rows, elems;
    if (!mul_ok(B, H, &bh) || !mul_ok(bh, N, &rows) || !mul_ok(rows, d, &elems) ||
        elems > INT64_MAX / 2)
        return FA_ERR_INVALID_ARG;
    if (rows == 0) return FA_OK;
    if (d != 64 && d != 128) return FA_ERR_UNSUPPORTED;
    if (!Q || !K || !V || !O) return FA_ERR_INVALID_ARG;
    if (!aligned(Q, 16) || !aligned(K, 16) || !aligned(V, 16) || !aligned(O, 16))
        return FA_ERR_INVALID_ARG;
    if (LSE && !aligned(LSE, 4)) return FA_ERR_INVALID_ARG;
    if (!std::isfinite(scale) || !(scale > 0.f)) return FA_ERR_INVALID_ARG;
    const uint64_t bytes = static_cast<uint64_t>(elems) * 2;      // each of Q, K, V, O
    const uint64_t lse_bytes = static_cast<uint64_t>(rows) * 4;   // LSE
    if (overlaps(O, bytes, Q, bytes) || overlaps(O, bytes, K, bytes) ||
        overlaps(O, bytes, V, bytes))
        return FA_ERR_INVALID_ARG;
    if (LSE && (overlaps(LSE, lse_bytes, O, bytes) || overlaps(LSE, lse_bytes, Q, bytes) ||
                overlaps(LSE, lse_bytes, K, bytes) || overlaps(LSE, lse_bytes, V, bytes)))
        return FA_ERR_INVALID_ARG;
    return osm::fa_fwd_launch(Q, K, V, O, LSE, bh, N, d, scale, causal != 0,
                              static_cast<cudaStream_t>(stream));
}

int fa_fwd_host(const void* Q_host, const void* K_host, const void* V_host, void* O_host,
                float* LSE_host, void* Q_dev, void* K_dev, void* V_dev, void* O_dev,
                float* LSE_dev, int64_t B, int64_t H, int64_t N, int64_t d, float scale,
                int causal, int64_t n_chunks, void* stream) {
    if (B < 0 || H < 0 || N < 0 || d < 0 || n_chunks < 0 || n_chunks > kHostPipeMaxChunks)
        return FA_ERR_INVALID_ARG;
    int64_t bh, rows, elems;
    if (!mul_ok(B, H, &bh) || !mul_ok(bh, N, &rows) || !mul_ok(rows, d, &elems) ||
        elems > INT64_MAX / 2)
        return FA_ERR_INVALID_ARG;
    if (rows == 0) return FA_OK;
    if (d != 64 && d != 128) return FA_ERR_UNSUPPORTED;
    if (!Q_host || !K_host || !V_host || !O_host) return FA_ERR_INVALID_ARG;
    if ((LSE_host == nullptr) != (LSE_dev == nullptr)) return FA_ERR_INVALID_ARG;
    if (!Q_dev || !K_dev || !V_dev || !O_dev) return FA_ERR_INVALID_ARG;
    if (!aligned(Q_dev, 16) || !aligned(K_dev, 16) || !aligned(V_dev, 16) ||
        !aligned(O_dev, 16) || (LSE_dev && !aligned(LSE_dev, 4)))
        return FA_ERR_INVALID_ARG;
    if (!std::isfinite(scale) || !(scale > 0.f)) return FA_ERR_INVALID_ARG;
    const uint64_t bytes = static_cast<uint64_t>(elems) * 2;     // each of Q, K, V, O
    const uint64_t lse_bytes = static_cast<uint64_t>(rows) * 4;  // LSE
    const void* dev[4] = {Q_dev, K_dev, V_dev, O_dev};
    for (int i = 0; i < 4; ++i) {
        for (int j = i + 1; j < 4; ++j)
            if (overlaps(dev[i], bytes, dev[j], bytes)) return FA_ERR_INVALID_ARG;
        if (LSE_dev && overlaps(LSE_dev, lse_bytes, dev[i], bytes)) return FA_ERR_INVALID_ARG;
    }
    // Groups of whole heads, never more than the heads.  By default one group per 12 MB of
    // inputs, 1 to 16 groups: measured on GB300, B2 H32 N8192 d128 (403 MB) ran best at 8-16
    // groups and B4 H16 N2048 d64 (50 MB) at 4; smaller groups pay launch and copy latency.
    int64_t n = n_chunks;
    if (n == 0) {
        const uint64_t in_bytes = 3 * bytes;
        n = static_cast<int64_t>(in_bytes / (12ull << 20));
        n = n < 1 ? 1 : (n > 16 ? 16 : n);
    }
    if (n > bh) n = bh;
    const cudaStream_t st = static_cast<cudaStream_t>(stream);
    std::lock_guard<std::mutex> lock(g_host_pipe_mu);
    HostPipe* P = host_pipe();
    if (!P) return FA_ERR_CUDA;
    const uint64_t head_bytes = static_cast<uint64_t>(N) * static_cast<uint64_t>(d) * 2;
    const uint64_t head_lse = static_cast<uint64_t>(N) * 4;
    auto ok = [](cudaError_t e) { return e == cudaSuccess; };
    if (!ok(cudaEventRecord(P->start, st)) || !ok(cudaStreamWaitEvent(P->h2d, P->start, 0)) ||
        !ok(cudaStreamWaitEvent(P->d2h, P->start, 0)))
        return FA_ERR_CUDA;
    int rc = FA_OK;
    for (int64_t c = 0; c < n && rc == FA_OK; ++c) {
        const int64_t h0 = bh * c / n, h1 = bh * (c + 1) / n;  // heads [h0, h1)
        const uint64_t off = static_cast<uint64_t>(h0) * head_bytes;
        const uint64_t len = static_cast<uint64_t>(h1 - h0) * head_bytes;
        auto at = [&](const void* base, uint64_t o) {
            return static_cast<const char*>(base) + o;
        };
        auto atw = [&](void* base, uint64_t o) { return static_cast<char*>(base) + o; };
        if (!ok(cudaMemcpyAsync(atw(Q_dev, off), at(Q_host, off), len, cudaMemcpyHostToDevice,
                                P->h2d)) ||
            !ok(cudaMemcpyAsync(atw(K_dev, off), at(K_host, off), len, cudaMemcpyHostToDevice,
                                P->h2d)) ||
            !ok(cudaMemcpyAsync(atw(V_dev, off), at(V_host, off), len, cudaMemcpyHostToDevice,
                                P->h2d)) ||
            !ok(cudaEventRecord(P->in[c], P->h2d)) || !ok(cudaStreamWaitEvent(st, P->in[c], 0))) {
            rc = FA_ERR_CUDA;
            break;
        }
        float* lse_c = LSE_dev ? LSE_dev + h0 * N : nullptr;
        rc = osm::fa_fwd_launch(at(Q_dev, off), at(K_dev, off), at(V_dev, off), atw(O_dev, off),
                                lse_c, h1 - h0, N, d, scale, causal != 0, st);
        if (rc != FA_OK) break;
        if (!ok(cudaEventRecord(P->out[c], st)) || !ok(cudaStreamWaitEvent(P->d2h, P->out[c], 0)) ||
            !ok(cudaMemcpyAsync(atw(O_host, off), at(O_dev, off), len, cudaMemcpyDeviceToHost,
                                P->d2h)) ||
            (LSE_host && !ok(cudaMemcpyAsync(LSE_host + h0 * N, lse_c,
                                             static_cast<uint64_t>(h1 - h0) * head_lse,
                                             cudaMemcpyDeviceToHost, P->d2h)))) {
            rc = FA_ERR_CUDA;
            break;
        }
    }
    // Whatever was enqueued, `stream` waits for both copy streams before its later work.
    const bool joined = ok(cudaEventRecord(P->done, P->d2h)) &&
                        ok(cudaStreamWaitEvent(st, P->done, 0)) &&
                        ok(cudaEventRecord(P->done, P->h2d)) &&
                        ok(cudaStreamWaitEvent(st, P->done, 0));
    if (rc == FA_OK && !joined) rc = FA_ERR_CUDA;
    return rc;
}

int fa_fwd_splitkv_plan(int64_t B, int64_t H, int64_t Nq, int64_t Nk, int64_t d,
                        int64_t n_splits, int64_t* splits_out, int64_t* ws_o_floats,
                        int64_t* ws_lse_floats) {
    if (!splits_out || !ws_o_floats || !ws_lse_floats) return FA_ERR_INVALID_ARG;
    if (B < 0 || H < 0 || Nq < 0 || Nk < 0 || d < 0 || n_splits < 0 || n_splits > 256)
        return FA_ERR_INVALID_ARG;
    int64_t bh, rows, elems;
    if (!mul_ok(B, H, &bh) || !mul_ok(bh, Nq, &rows) || !mul_ok(rows, d, &elems))
        return FA_ERR_INVALID_ARG;
    if (d != 64 && d != 128) return FA_ERR_UNSUPPORTED;
    const int64_t splits = osm::splitkv_choose_splits(bh, Nq, Nk, n_splits);
    int64_t o = 0, l = 0;
    if (splits > 1 && (!mul_ok(elems, splits, &o) || !mul_ok(rows, splits, &l)))
        return FA_ERR_INVALID_ARG;
    *splits_out = splits;
    *ws_o_floats = splits > 1 ? o : 0;
    *ws_lse_floats = splits > 1 ? l : 0;
    return FA_OK;
}

int fa_fwd_splitkv(const void* Q, const void* K, const void* V, void* O, float* LSE, int64_t B,
                   int64_t H, int64_t Nq, int64_t Nk, int64_t d, float scale, int causal,
                   int64_t n_splits, float* ws_O, float* ws_LSE, void* stream) {
    return attention_call(Q, K, V, O, LSE, B, H, H, Nq, Nk, d, scale, causal, nullptr, n_splits,
                          ws_O, ws_LSE, stream);
}

int fa_fwd_gqa(const void* Q, const void* K, const void* V, void* O, float* LSE, int64_t B,
               int64_t H, int64_t H_kv, int64_t Nq, int64_t Nk, int64_t d, float scale,
               int causal, const int32_t* kv_lens, int64_t n_splits, float* ws_O, float* ws_LSE,
               void* stream) {
    return attention_call(Q, K, V, O, LSE, B, H, H_kv, Nq, Nk, d, scale, causal, kv_lens,
                          n_splits, ws_O, ws_LSE, stream);
}

int fa_fwd_mask(const void* Q, const void* K, const void* V, void* O, float* LSE, int64_t B,
                int64_t H, int64_t Nq, int64_t Nk, int64_t d, float scale, int causal,
                const uint32_t* mask, int64_t mask_b_stride, int64_t mask_h_stride,
                uint32_t* tile_map, int64_t tile_map_words, void* stream) {
    if (!mask) return FA_ERR_INVALID_ARG;
    return attention_call(Q, K, V, O, LSE, B, H, H, Nq, Nk, d, scale, causal, nullptr, 1,
                          nullptr, nullptr, stream, mask, mask_b_stride, mask_h_stride,
                          tile_map, tile_map_words);
}

int fa_fwd_gqa_mask(const void* Q, const void* K, const void* V, void* O, float* LSE,
                    int64_t B, int64_t H, int64_t H_kv, int64_t Nq, int64_t Nk, int64_t d,
                    float scale, int causal, const int32_t* kv_lens, const uint32_t* mask,
                    int64_t mask_b_stride, int64_t mask_h_stride, uint32_t* tile_map,
                    int64_t tile_map_words, int64_t n_splits, float* ws_O, float* ws_LSE,
                    void* stream) {
    if (!mask) return FA_ERR_INVALID_ARG;
    return attention_call(Q, K, V, O, LSE, B, H, H_kv, Nq, Nk, d, scale, causal, kv_lens,
                          n_splits, ws_O, ws_LSE, stream, mask, mask_b_stride, mask_h_stride,
                          tile_map, tile_map_words);
}

int fa_fwd_gqa_mask_plan(int64_t B, int64_t H, int64_t H_kv, int64_t Nq, int64_t Nk, int64_t d,
                         int64_t mask_b_stride, int64_t mask_h_stride, int64_t n_splits,
                         int64_t* splits_out, int64_t* ws_o_floats, int64_t* ws_lse_floats,
                         int64_t* tile_map_words) {
    if (!splits_out || !ws_o_floats || !ws_lse_floats || !tile_map_words)
        return FA_ERR_INVALID_ARG;
    if (B < 0 || H < 0 || H_kv < 0 || Nq < 0 || Nk < 0 || d < 0 || n_splits < 0 ||
        n_splits > 256 || mask_b_stride < 0 || mask_h_stride < 0 || Nq > (1LL << 30) ||
        Nk > (1LL << 30) || B > (1LL << 30) || H > (1LL << 30))
        return FA_ERR_INVALID_ARG;
    if (H > 0 && (H_kv < 1 || H % H_kv != 0)) return FA_ERR_INVALID_ARG;
    int64_t bh, rows, elems;
    if (!mul_ok(B, H, &bh) || !mul_ok(bh, Nq, &rows) || !mul_ok(rows, d, &elems))
        return FA_ERR_INVALID_ARG;
    if (d != 64 && d != 128) return FA_ERR_UNSUPPORTED;
    const int64_t words = osm::mask_tile_map_words(B, H, Nq, Nk, mask_b_stride, mask_h_stride);
    if (words < 0) return FA_ERR_INVALID_ARG;
    // With a mask the query heads run as their own row blocks (no packing by key/value head).
    const int64_t splits = osm::splitkv_choose_splits(bh, Nq, Nk, n_splits);
    int64_t o = 0, l = 0;
    if (splits > 1 && (!mul_ok(elems, splits, &o) || !mul_ok(rows, splits, &l)))
        return FA_ERR_INVALID_ARG;
    *splits_out = splits;
    *ws_o_floats = splits > 1 ? o : 0;
    *ws_lse_floats = splits > 1 ? l : 0;
    *tile_map_words = words;
    return FA_OK;
}

int fa_fwd_mask_plan(int64_t B, int64_t H, int64_t Nq, int64_t Nk, int64_t mask_b_stride,
                     int64_t mask_h_stride, int64_t* tile_map_words) {
    if (!tile_map_words || B < 0 || H < 0 || Nq < 0 || Nk < 0 || mask_b_stride < 0 ||
        mask_h_stride < 0 || Nq > (1LL << 30) || Nk > (1LL << 30) || B > (1LL << 30) ||
        H > (1LL << 30))
        return FA_ERR_INVALID_ARG;
    int64_t words = osm::mask_tile_map_words(B, H, Nq, Nk, mask_b_stride, mask_h_stride);
    if (words < 0) return FA_ERR_INVALID_ARG;
    *tile_map_words = words;
    return FA_OK;
}

int fa_bwd_gqa(const void* Q, const void* K, const void* V, const void* O, const void* dO,
               const float* LSE, void* dQ, void* dK, void* dV, float* ws_D, int64_t B, int64_t H,
               int64_t H_kv, int64_t N, int64_t d, float scale, int causal,
               const int32_t* kv_lens, void* stream) {
    if (B < 0 || H < 0 || H_kv < 0 || N < 0 || d < 0) return FA_ERR_INVALID_ARG;
    if (H > 0 && (H_kv < 1 || H % H_kv != 0)) return FA_ERR_INVALID_ARG;
    int64_t bh, rows, elems, bh_kv, kv_elems;
    if (!mul_ok(B, H, &bh) || !mul_ok(bh, N, &rows) || !mul_ok(rows, d, &elems) ||
        elems > INT64_MAX / 4 || !mul_ok(B, H_kv, &bh_kv) || !mul_ok(bh_kv, N, &kv_elems) ||
        !mul_ok(kv_elems, d, &kv_elems))
        return FA_ERR_INVALID_ARG;
    if (rows == 0) return FA_OK;
    if (d != 64 && d != 128) return FA_ERR_UNSUPPORTED;
    if (!std::isfinite(scale) || !(scale > 0.f)) return FA_ERR_INVALID_ARG;
    // inputs Q, K, V, O, dO, LSE (+ kv_lens); outputs dQ, dK, dV and the workspace D
    const void* ins[7] = {Q, K, V, O, dO, LSE, kv_lens};
    const void* outs[4] = {dQ, dK, dV, ws_D};
    const uint64_t q_bytes = static_cast<uint64_t>(elems) * 2;     // a bf16 [B, H, N, d] tensor
    const uint64_t kv_bytes = static_cast<uint64_t>(kv_elems) * 2;  // a bf16 [B, H_kv, N, d]
    const uint64_t r_bytes = static_cast<uint64_t>(rows) * 4;      // one fp32 value per row
    const uint64_t in_bytes[7] = {q_bytes, kv_bytes, kv_bytes, q_bytes, q_bytes, r_bytes,
                                  kv_lens ? static_cast<uint64_t>(B) * 4 : 0};
    const uint64_t out_bytes[4] = {q_bytes, kv_bytes, kv_bytes, r_bytes};
    for (int i = 0; i < 6; ++i)
        if (!ins[i] || !aligned(ins[i], i < 5 ? 16 : 4)) return FA_ERR_INVALID_ARG;
    if (kv_lens && !aligned(kv_lens, 4)) return FA_ERR_INVALID_ARG;
    for (int i = 0; i < 4; ++i)
        if (!outs[i] || !aligned(outs[i], i < 3 ? 16 : 4)) return FA_ERR_INVALID_ARG;
    for (int i = 0; i < 4; ++i) {
        for (int j = 0; j < 7; ++j)
            if (overlaps(outs[i], out_bytes[i], ins[j], in_bytes[j])) return FA_ERR_INVALID_ARG;
        for (int j = i + 1; j < 4; ++j)
            if (overlaps(outs[i], out_bytes[i], outs[j], out_bytes[j])) return FA_ERR_INVALID_ARG;
    }
    return osm::fa_bwd_launch(Q, K, V, O, dO, LSE, dQ, dK, dV, ws_D, B, H, H_kv, N, d, kv_lens,
                              scale, causal != 0, static_cast<cudaStream_t>(stream));
}

int fa_bwd(const void* Q, const void* K, const void* V, const void* O, const void* dO,
           const float* LSE, void* dQ, void* dK, void* dV, float* ws_D, int64_t B, int64_t H,
           int64_t N, int64_t d, float scale, int causal, void* stream) {
    return fa_bwd_gqa(Q, K, V, O, dO, LSE, dQ, dK, dV, ws_D, B, H, H, N, d, scale, causal,
                      nullptr, stream);
}

int osm_softmax_topk(const float* x, int64_t rows, int64_t cols, int64_t k, float* values,
                     int32_t* indices, float* lse, void* stream) {
    if (rows < 0 || cols < 0 || k < 1) return FA_ERR_INVALID_ARG;
    if (rows == 0) return FA_OK;
    if (k > cols) return FA_ERR_INVALID_ARG;
    if (k > 1024) return FA_ERR_UNSUPPORTED;
    int64_t elems, outs;
    if (!mul_ok(rows, cols, &elems) || !mul_ok(rows, k, &outs) || elems > INT64_MAX / 4)
        return FA_ERR_INVALID_ARG;
    if (!x || !values || !indices) return FA_ERR_INVALID_ARG;
    if (!aligned(x, 4) || !aligned(values, 4) || !aligned(indices, 4) || (lse && !aligned(lse, 4)))
        return FA_ERR_INVALID_ARG;
    const uint64_t x_bytes = static_cast<uint64_t>(elems) * 4;
    const uint64_t o_bytes = static_cast<uint64_t>(outs) * 4;
    const uint64_t l_bytes = static_cast<uint64_t>(rows) * 4;
    if (overlaps(values, o_bytes, x, x_bytes) || overlaps(indices, o_bytes, x, x_bytes) ||
        overlaps(values, o_bytes, indices, o_bytes))
        return FA_ERR_INVALID_ARG;
    if (lse && (overlaps(lse, l_bytes, x, x_bytes) || overlaps(lse, l_bytes, values, o_bytes) ||
                overlaps(lse, l_bytes, indices, o_bytes)))
        return FA_ERR_INVALID_ARG;
    return osm::osm_softmax_topk_launch(x, rows, cols, k, values, indices, lse,
                                        static_cast<cudaStream_t>(stream));
}

int osm_softmax(const float* x, float* y, int64_t rows, int64_t cols, float* lse,
                void* stream) {
    if (rows < 0 || cols < 0) return FA_ERR_INVALID_ARG;
    int64_t elems;
    if (!mul_ok(rows, cols, &elems) || elems > INT64_MAX / 4) return FA_ERR_INVALID_ARG;
    if (elems == 0) return FA_OK;  // nothing to read or write (lse is not written)
    if (!x || !y) return FA_ERR_INVALID_ARG;
    if (!aligned(x, 4) || !aligned(y, 4) || (lse && !aligned(lse, 4))) return FA_ERR_INVALID_ARG;
    const uint64_t xy_bytes = static_cast<uint64_t>(elems) * 4;
    if (x != y && overlaps(x, xy_bytes, y, xy_bytes)) return FA_ERR_INVALID_ARG;
    if (lse && (overlaps(lse, static_cast<uint64_t>(rows) * 4, x, xy_bytes) ||
                overlaps(lse, static_cast<uint64_t>(rows) * 4, y, xy_bytes)))
        return FA_ERR_INVALID_ARG;
    return osm::osm_softmax_launch(x, y, rows, cols, lse, static_cast<cudaStream_t>(stream));
}

const char* fa_status_string(int status) {
    switch (status) {
        case FA_OK: return "FA_OK";
        case FA_ERR_INVALID_ARG: return "FA_ERR_INVALID_ARG: invalid argument";
        case FA_ERR_UNSUPPORTED: return "FA_ERR_UNSUPPORTED: valid but not supported by this build";
        case FA_ERR_CUDA: return "FA_ERR_CUDA: a CUDA call failed";
        case FA_ERR_TIMEOUT: return "FA_ERR_TIMEOUT: a kernel gave up a bounded wait";
        case FA_ERR_SCRATCH_LIMIT:
            return "FA_ERR_SCRATCH_LIMIT: the partial states do not fit in the fixed scratch array";
        default: return "unknown fa_status";
    }
}

int osm_attn_device_status(void* stream, int* status) {
    if (!status) return FA_ERR_INVALID_ARG;
    int raw = 0;
    const int rc = osm::fa_read_device_status(static_cast<cudaStream_t>(stream), &raw);
    if (rc != FA_OK) return rc;
    *status = raw & 0xff;
    return FA_OK;
}

int osm_attn_selftest_wait(int64_t timeout_us, void* stream) {
    return osm::selftest_wait_launch(timeout_us, static_cast<cudaStream_t>(stream));
}

int osm_attn_abi_version(void) { return OSM_ATTN_ABI_VERSION; }

}  // extern "C"

namespace osm {
unsigned long long fa_wait_timeout_ns() { return 2000000000ull; }  // 2 s
}  // namespace osm
