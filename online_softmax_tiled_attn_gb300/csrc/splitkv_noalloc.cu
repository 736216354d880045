// splitkv_noalloc.cu -- fa_fwd_splitkv_noalloc: the split-key attention without allocation.
//
// Some callers cannot allocate device memory while they run a step: an inference engine that
// calls attention from a plugin or custom-operator hook, where the host framework owns every
// device buffer and forbids allocation inside that hook, or a latency-critical decode loop that
// must not pay for an allocator call or risk an out-of-memory failure in the middle of a step.
// fa_fwd_splitkv needs a workspace for the per-range partial states; this entry point takes it
// from a fixed array in device memory instead, so the caller passes only inputs and outputs.
#include <cuda_runtime.h>

#include <mutex>

#include "osm_internal.h"

namespace {

// Scratch for the partial outputs and log-sum-exps of the split-key path: 4 Mi floats
// (16 MiB).  Every GPU that loads the library holds it until the process exits.  All calls on
// a device share it and it keeps the last call's contents.
constexpr int64_t kScratchFloats = int64_t(4) << 20;
static __device__ __align__(256) float g_splitkv_scratch[kScratchFloats];

constexpr int kMaxDevices = 64;
std::mutex g_scratch_mu;
float* g_scratch_addr[kMaxDevices] = {};

// Device address of the scratch array on the current device.  Resolved on the first call made
// with that device current (cudaGetSymbolAddress), then cached.
int scratch_address(float** out) {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return FA_ERR_CUDA;
    if (dev < 0 || dev >= kMaxDevices) return FA_ERR_UNSUPPORTED;
    std::lock_guard<std::mutex> lock(g_scratch_mu);
    if (g_scratch_addr[dev] == nullptr) {
        void* p = nullptr;
        if (cudaGetSymbolAddress(&p, g_splitkv_scratch) != cudaSuccess || p == nullptr)
            return FA_ERR_CUDA;
        g_scratch_addr[dev] = static_cast<float*>(p);
    }
    *out = g_scratch_addr[dev];
    return FA_OK;
}

}  // namespace

extern "C" OSM_ATTN_API int fa_fwd_splitkv_noalloc(const void* Q, const void* K, const void* V,
                                                   void* O, float* LSE, int64_t B, int64_t H,
                                                   int64_t Nq, int64_t Nk, int64_t d,
                                                   float scale, int causal, int64_t n_splits,
                                                   void* stream) {
    if (B < 0 || H < 0 || Nq < 0 || Nk < 0 || d < 0 || n_splits < 0 || n_splits > 256)
        return FA_ERR_INVALID_ARG;
    if (B > (int64_t(1) << 31) || H > (int64_t(1) << 31) || Nq > (int64_t(1) << 31))
        return FA_ERR_INVALID_ARG;
    const int64_t bh = B * H;
    if (bh != 0 && Nq > INT64_MAX / bh) return FA_ERR_INVALID_ARG;
    const int64_t rows = bh * Nq;
    if (rows == 0) return FA_OK;
    if (d != 64 && d != 128) return FA_ERR_UNSUPPORTED;
    if (Nk == 0)  // every row is empty; no partial state is needed
        return fa_fwd_splitkv(Q, K, V, O, LSE, B, H, Nq, Nk, d, scale, causal, 0, nullptr, nullptr,
                              stream);
    const int64_t splits = osm::splitkv_choose_splits(bh, Nq, Nk, n_splits);
    if (splits <= 1)
        return fa_fwd_splitkv(Q, K, V, O, LSE, B, H, Nq, Nk, d, scale, causal, 1, nullptr, nullptr,
                              stream);
    // Partial outputs [splits, rows, d] followed by partial log-sum-exps [splits, rows].
    if (rows > kScratchFloats / (splits * (d + 1))) return FA_ERR_SCRATCH_LIMIT;
    float* base = nullptr;
    const int st = scratch_address(&base);
    if (st != FA_OK) return st;
    // Every (range, row) entry the combine reads is written by the attention kernel of the same
    // call (empty ranges write their empty state), so nothing has to be cleared beforehand.
    return fa_fwd_splitkv(Q, K, V, O, LSE, B, H, Nq, Nk, d, scale, causal, splits, base,
                          base + splits * rows * d, stream);
}
