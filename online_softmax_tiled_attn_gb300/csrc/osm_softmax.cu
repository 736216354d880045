// osm_softmax.cu -- single-pass (online-normalizer) row softmax for sm_103a.
//
// The method: "How FlashAttention avoids storing the giant score table" (spicyshark.co,
// Online softmax lesson), sections "The idea" and "The implementation": the running maximum m
// and the running sum l = sum exp(x - m), rescaled by exp(m_old - m_new) when the maximum
// grows, give both statistics in one read of the row; two partial states of disjoint parts of a
// row merge by taking the larger max and rescaling each side's l by exp(its max - the larger
// max) (the two-worker merge at the end of "From softmax to attention"); the shares are
// y_j = exp(x_j - m) / l.
//
// GB300 mapping (HBM-bound: 4 bytes read + 4 bytes written per element):
//   * a row is split across the lanes of a warp (rows up to 1024 columns) or the 256 threads
//     of a CTA (rows up to 16384 columns); each thread loads its part with 16-byte loads into
//     registers, forms its own (m, l), and the partial states are merged with warp shuffles
//     (and shared memory across warps) by the two-worker merge;
//   * y is written from the registers: the row is read from HBM exactly once;
//   * longer rows stream: each thread runs the online update block by block over its part,
//     the states are merged, and a second read of the row writes y (two reads, one write);
//   * persistent grid: a multiple of the SM count, rows handed out round-robin.
// Exponentials are ex2 of (x - m) * log2(e): x - m is formed first so that the largest shares
// keep full relative accuracy.
#include <cuda_runtime.h>

#include <climits>
#include <cmath>
#include <mutex>

#include "osm_internal.h"

namespace osm {
namespace {

constexpr float kLog2e = 1.4426950408889634f;
constexpr int kCtaThreads = 256;

__device__ __forceinline__ float ex2a(float x) {
    float y;
    asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}

struct Stat {
    float m;  // largest value seen
    float l;  // sum of exp(x - m) over the values seen
};

// The two-worker merge of two partial states.
__device__ __forceinline__ Stat merge(Stat a, Stat b) {
    const float m = fmaxf(a.m, b.m);
    if (m == -INFINITY) return Stat{-INFINITY, 0.f};
    return Stat{m, a.l * ex2a((a.m - m) * kLog2e) + b.l * ex2a((b.m - m) * kLog2e)};
}

__device__ __forceinline__ Stat warp_merge(Stat s) {
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) {
        Stat o;
        o.m = __shfl_xor_sync(0xffffffffu, s.m, off);
        o.l = __shfl_xor_sync(0xffffffffu, s.l, off);
        s = merge(s, o);
    }
    return s;
}

// State of the values a thread holds (one block of the online recurrence).
template <int NE>
__device__ __forceinline__ Stat local_stat(const float (&v)[NE]) {
    float mx = -INFINITY;
#pragma unroll
    for (int e = 0; e < NE; ++e) mx = fmaxf(mx, v[e]);
    const float mu = (mx == -INFINITY) ? 0.f : mx;  // nothing finite: adds nothing
    float l = 0.f;
#pragma unroll
    for (int e = 0; e < NE; ++e) l += ex2a((v[e] - mu) * kLog2e);
    return Stat{mx, l};
}

// Loads the NE values of thread `t` (of `nthr` threads sharing the row) into registers;
// positions past the row read -inf.  VEC: 16-byte loads of float4 groups.
template <int NE, bool VEC>
__device__ __forceinline__ void load_part(const float* row, int cols, int t,
                                          int nthr, float (&v)[NE]) {
    if constexpr (VEC) {
        const float4* r4 = reinterpret_cast<const float4*>(row);
        const int nc4 = cols >> 2;
#pragma unroll
        for (int k = 0; k < NE / 4; ++k) {
            const int i = t + k * nthr;
            float4 q = make_float4(-INFINITY, -INFINITY, -INFINITY, -INFINITY);
            if (i < nc4) q = __ldcs(r4 + i);
            v[4 * k] = q.x;
            v[4 * k + 1] = q.y;
            v[4 * k + 2] = q.z;
            v[4 * k + 3] = q.w;
        }
    } else {
#pragma unroll
        for (int k = 0; k < NE; ++k) {
            const int i = t + k * nthr;
            v[k] = i < cols ? __ldcs(row + i) : -INFINITY;
        }
    }
}

template <int NE, bool VEC>
__device__ __forceinline__ void store_part(float* row, int cols, int t, int nthr,
                                           const float (&v)[NE], float m, float inv_l) {
    const float mu = (m == -INFINITY) ? 0.f : m;
    if constexpr (VEC) {
        float4* r4 = reinterpret_cast<float4*>(row);
        const int nc4 = cols >> 2;
#pragma unroll
        for (int k = 0; k < NE / 4; ++k) {
            const int i = t + k * nthr;
            if (i < nc4) {
                float4 q;
                q.x = ex2a((v[4 * k] - mu) * kLog2e) * inv_l;
                q.y = ex2a((v[4 * k + 1] - mu) * kLog2e) * inv_l;
                q.z = ex2a((v[4 * k + 2] - mu) * kLog2e) * inv_l;
                q.w = ex2a((v[4 * k + 3] - mu) * kLog2e) * inv_l;
                __stcs(r4 + i, q);
            }
        }
    } else {
#pragma unroll
        for (int k = 0; k < NE; ++k) {
            const int i = t + k * nthr;
            if (i < cols) __stcs(row + i, ex2a((v[k] - mu) * kLog2e) * inv_l);
        }
    }
}

__device__ __forceinline__ void finish(Stat s, float* lse, long long r, float& inv_l) {
    inv_l = s.l > 0.f ? 1.f / s.l : 0.f;
    if (lse) lse[r] = s.m + logf(s.l);
}

// One warp per row.
template <int NE, bool VEC>
__global__ void __launch_bounds__(kCtaThreads)
    softmax_warp_rows(const float* x, float* y, float* __restrict__ lse,
                      long long rows, int cols) {
    const int lane = threadIdx.x & 31;
    const long long wpc = kCtaThreads / 32;
    for (long long r = blockIdx.x * wpc + (threadIdx.x >> 5); r < rows; r += gridDim.x * wpc) {
        float v[NE];
        load_part<NE, VEC>(x + r * cols, cols, lane, 32, v);
        const Stat s = warp_merge(local_stat<NE>(v));
        float inv_l;
        finish(s, lane == 0 ? lse : nullptr, r, inv_l);
        store_part<NE, VEC>(y + r * cols, cols, lane, 32, v, s.m, inv_l);
    }
}

// CTA-wide merge; `sm` holds two buffers of one Stat per warp (alternating by row parity, so
// one __syncthreads per row suffices).
__device__ __forceinline__ Stat cta_merge(Stat s, Stat (*sm)[kCtaThreads / 32], int buf) {
    s = warp_merge(s);
    if ((threadIdx.x & 31) == 0) sm[buf][threadIdx.x >> 5] = s;
    __syncthreads();
    Stat t = sm[buf][0];
#pragma unroll
    for (int w = 1; w < kCtaThreads / 32; ++w) t = merge(t, sm[buf][w]);
    return t;
}

// One CTA per row, the row kept in registers.
template <int NE, bool VEC>
__global__ void __launch_bounds__(kCtaThreads)
    softmax_cta_rows(const float* x, float* y, float* __restrict__ lse,
                     long long rows, int cols) {
    __shared__ Stat sm[2][kCtaThreads / 32];
    int buf = 0;
    for (long long r = blockIdx.x; r < rows; r += gridDim.x, buf ^= 1) {
        float v[NE];
        load_part<NE, VEC>(x + r * cols, cols, threadIdx.x, kCtaThreads, v);
        const Stat s = cta_merge(local_stat<NE>(v), sm, buf);
        float inv_l;
        finish(s, threadIdx.x == 0 ? lse : nullptr, r, inv_l);
        store_part<NE, VEC>(y + r * cols, cols, threadIdx.x, kCtaThreads, v, s.m, inv_l);
    }
}

// One CTA per row, rows too long for registers: online update over 16-byte (or 4-byte) blocks,
// merge, then a second read to write y.
template <bool VEC>
__global__ void __launch_bounds__(kCtaThreads)
    softmax_cta_stream(const float* x, float* y, float* __restrict__ lse,
                       long long rows, int cols) {
    __shared__ Stat sm[2][kCtaThreads / 32];
    int buf = 0;
    for (long long r = blockIdx.x; r < rows; r += gridDim.x, buf ^= 1) {
        const float* xr = x + r * cols;
        float* yr = y + r * cols;
        Stat s{-INFINITY, 0.f};
        constexpr int W = VEC ? 4 : 1;
        const int nblk = VEC ? (cols >> 2) : cols;
        for (int i = threadIdx.x; i < nblk; i += kCtaThreads) {
            float v[W];
            if constexpr (VEC) {
                const float4 q = __ldcs(reinterpret_cast<const float4*>(xr) + i);
                v[0] = q.x; v[1] = q.y; v[2] = q.z; v[3] = q.w;
            } else {
                v[0] = __ldcs(xr + i);
            }
            s = merge(s, local_stat<W>(v));
        }
        s = cta_merge(s, sm, buf);
        float inv_l;
        finish(s, threadIdx.x == 0 ? lse : nullptr, r, inv_l);
        const float mu = (s.m == -INFINITY) ? 0.f : s.m;
        for (int i = threadIdx.x; i < nblk; i += kCtaThreads) {
            if constexpr (VEC) {
                const float4 q = __ldcs(reinterpret_cast<const float4*>(xr) + i);
                float4 o;
                o.x = ex2a((q.x - mu) * kLog2e) * inv_l;
                o.y = ex2a((q.y - mu) * kLog2e) * inv_l;
                o.z = ex2a((q.z - mu) * kLog2e) * inv_l;
                o.w = ex2a((q.w - mu) * kLog2e) * inv_l;
                __stcs(reinterpret_cast<float4*>(yr) + i, o);
            } else {
                __stcs(yr + i, ex2a((__ldcs(xr + i) - mu) * kLog2e) * inv_l);
            }
        }
    }
}

int sm_count() {
    static int n = 0;
    static std::once_flag once;
    std::call_once(once, [] {
        int dev = 0;
        if (cudaGetDevice(&dev) != cudaSuccess ||
            cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
            n = 0;
    });
    return n;
}

template <typename Kern>
int launch_persistent(Kern kern, long long work_items, const float* x, float* y, float* lse,
                      long long rows, int cols, cudaStream_t stream) {
    const int sms = sm_count();
    if (sms <= 0) return FA_ERR_CUDA;
    int per_sm = 0;
    if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, kern, kCtaThreads, 0) !=
            cudaSuccess ||
        per_sm <= 0)
        return FA_ERR_CUDA;
    long long grid = static_cast<long long>(sms) * per_sm;
    if (grid > work_items) grid = work_items;
    if (grid < 1) grid = 1;
    kern<<<static_cast<unsigned>(grid), kCtaThreads, 0, stream>>>(x, y, lse, rows, cols);
    return cudaGetLastError() == cudaSuccess ? FA_OK : FA_ERR_CUDA;
}

template <bool VEC>
int dispatch(const float* x, float* y, float* lse, long long rows, int cols,
             cudaStream_t stream) {
    const long long warps_rows = (rows + 7) / 8;  // 8 rows (warps) per CTA
    if (cols <= 32 * 4)
        return launch_persistent(softmax_warp_rows<4, VEC>, warps_rows, x, y, lse, rows, cols, stream);
    if (cols <= 32 * 8)
        return launch_persistent(softmax_warp_rows<8, VEC>, warps_rows, x, y, lse, rows, cols, stream);
    if (cols <= 32 * 16)
        return launch_persistent(softmax_warp_rows<16, VEC>, warps_rows, x, y, lse, rows, cols, stream);
    if (cols <= 32 * 32)
        return launch_persistent(softmax_warp_rows<32, VEC>, warps_rows, x, y, lse, rows, cols, stream);
    if (cols <= kCtaThreads * 8)
        return launch_persistent(softmax_cta_rows<8, VEC>, rows, x, y, lse, rows, cols, stream);
    if (cols <= kCtaThreads * 16)
        return launch_persistent(softmax_cta_rows<16, VEC>, rows, x, y, lse, rows, cols, stream);
    if (cols <= kCtaThreads * 32)
        return launch_persistent(softmax_cta_rows<32, VEC>, rows, x, y, lse, rows, cols, stream);
    if (cols <= kCtaThreads * 64)
        return launch_persistent(softmax_cta_rows<64, VEC>, rows, x, y, lse, rows, cols, stream);
    return launch_persistent(softmax_cta_stream<VEC>, rows, x, y, lse, rows, cols, stream);
}

}  // namespace

int osm_softmax_launch(const float* x, float* y, int64_t rows, int64_t cols, float* lse,
                       cudaStream_t stream) {
    if (cols > INT_MAX) return FA_ERR_UNSUPPORTED;
    const bool vec = (cols % 4 == 0) && (reinterpret_cast<uintptr_t>(x) % 16 == 0) &&
                     (reinterpret_cast<uintptr_t>(y) % 16 == 0);
    return vec ? dispatch<true>(x, y, lse, rows, static_cast<int>(cols), stream)
               : dispatch<false>(x, y, lse, rows, static_cast<int>(cols), stream);
}

}  // namespace osm
