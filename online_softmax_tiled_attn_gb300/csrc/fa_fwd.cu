// fa_fwd.cu -- exact attention forward, tile by tile with the online softmax, for sm_103a.
//
// The method: "How FlashAttention avoids storing the giant score table" (spicyshark.co,
// Online softmax lesson), section "From softmax to attention" (per key block: scores, new
// running max, alpha = exp(m - m_new), p = exp(s - m_new), l = l*alpha + sum p,
// acc = acc*alpha + p V, divide by l after the last block) and "The implementation" (a block
// that leaves the max at -inf adds nothing); "kbwen.com FlashAttention", sections "Two
// blocks" and "More than two blocks" (query blocks in the outer loop, key blocks inside,
// each query row with its own max, sum and partial output).
//
// GB300 mapping of one CTA = one tile of 128 query rows of one (b, h):
//   warp 4 (one lane)  TMA: Q tile once, then K and V tiles of 128 keys into a 2-stage ring
//                      (128-byte swizzled, zero fill past N).
//   warp 5 (one lane)  tcgen05.mma: S = Q K^T into TMEM columns [0, 128), then
//                      O += P V into TMEM columns [128, 128 + d); fp32 accumulators.
//                      S(j+1) is issued as soon as the softmax warps have S(j) in registers,
//                      so the tensor core computes the next scores while they work.
//   warps 0-3          the online softmax, one query row per thread (TMEM lane = row):
//                      tcgen05.ld of the S row, mask, running max, ex2 of the scaled and
//                      shifted scores, running sum, P rounded to bf16 into shared memory for
//                      the second MMA, rescale of the O row in TMEM by alpha when the max
//                      moved, and at the end O / l (bf16) and LSE = m + ln l (fp32).
// The exponentials are base 2 with scale*log2(e) folded into one FFMA (the lesson's note on
// base-2 exponentials in "Where this is used in practice"); LSE is converted back to natural
// log.  Causal: key tiles above the diagonal are never visited; only the diagonal tile and a
// ragged last tile are masked element by element.
//
// Every mbarrier wait is bounded (%globaltimer deadline).  A wait that gives up records
// FA_ERR_TIMEOUT in a device status word; the CTA then drains its own TMA loads and MMAs,
// frees its TMEM and exits.
#include <cuda_runtime.h>

#include <cmath>
#include <mutex>

#include "osm_internal.h"
#include "ptx_sm103.cuh"

namespace osm {

__device__ int g_fa_device_status = 0;

namespace {

constexpr int kBM = 128;       // query rows per tile: one TMEM lane per row
constexpr int kBN = 128;       // keys per key/value tile
constexpr int kStages = 2;     // K/V ring depth
constexpr int kThreads = 192;  // warps 0-3 softmax, 4 TMA, 5 MMA
constexpr uint32_t kTmemCols = 256;
constexpr uint32_t kTmemS = 0;    // S columns [0, 128)
constexpr uint32_t kTmemO = 128;  // O columns [128, 128 + d)
constexpr int kHalfBytes = 128 * 128;  // one 64-column half of a 128-row bf16 tile
constexpr uint64_t kDrainNs = 1000000000ull;  // drain waits: at least 1 s

struct Bars {
    uint64_t q_full;
    uint64_t k_full[kStages];
    uint64_t v_full[kStages];
    uint64_t kv_empty[kStages];
    uint64_t s_full;
    uint64_t s_free;
    uint64_t p_full;
    uint64_t pv_done;
    uint64_t mma_done;
    uint32_t tmem_base;
};

template <int D>
struct Layout {
    static constexpr int kHalves = D / 64;
    static constexpr int kTileBytes = kHalves * kHalfBytes;  // 128 rows x D bf16
    static constexpr int kQ = 0;
    static constexpr int kK = kQ + kTileBytes;
    static constexpr int kV = kK + kStages * kTileBytes;
    static constexpr int kP = kV + kStages * kTileBytes;  // 128 x 128 bf16 = 2 halves
    static constexpr int kBars = kP + 2 * kHalfBytes;
    static constexpr int kBytes = kBars + static_cast<int>(sizeof(Bars));
    static constexpr int kDynSmem = kBytes + 1024;  // slack for 1024-byte alignment
};

// All 32 lanes wait on the same phase; the outcome is made warp-uniform so that the
// .sync.aligned tcgen05 instructions that follow are never reached by a partial warp.
__device__ __forceinline__ bool warp_wait(uint64_t* bar, uint32_t parity, uint64_t timeout_ns) {
    const bool ok = mbar_wait(bar, parity, timeout_ns);
    return __all_sync(0xffffffffu, ok);
}

__device__ __forceinline__ void record_timeout(int where) {
    atomicCAS(&g_fa_device_status, 0, FA_ERR_TIMEOUT | (where << 8));
}

template <int D, bool CAUSAL>
__global__ void __launch_bounds__(kThreads, 1)
    fa_fwd_kernel(const __grid_constant__ CUtensorMap tmQ, const __grid_constant__ CUtensorMap tmK,
                  const __grid_constant__ CUtensorMap tmV, __nv_bfloat16* __restrict__ O,
                  float* __restrict__ LSE, int N, int BH, int n_qtiles, float scale_log2,
                  unsigned long long timeout_ns) {
    using L = Layout<D>;
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
    Bars* bars = reinterpret_cast<Bars*>(smem + L::kBars);
    const uint32_t sQ = smem_u32(smem + L::kQ);
    const uint32_t sK = smem_u32(smem + L::kK);
    const uint32_t sV = smem_u32(smem + L::kV);
    const uint32_t sP = smem_u32(smem + L::kP);

    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;

    // Work item: causal runs the longest rows (highest query tiles) first.
    int q_tile, bh;
    if (CAUSAL) {
        q_tile = n_qtiles - 1 - static_cast<int>(blockIdx.x) / BH;
        bh = static_cast<int>(blockIdx.x) % BH;
    } else {
        q_tile = static_cast<int>(blockIdx.x) % n_qtiles;
        bh = static_cast<int>(blockIdx.x) / n_qtiles;
    }
    const int n_kv_all = (N + kBN - 1) / kBN;
    const int n_kv = CAUSAL ? min(n_kv_all, q_tile + 1) : n_kv_all;

    if (threadIdx.x == 0) {
        mbar_init(&bars->q_full, 1);
        for (int s = 0; s < kStages; ++s) {
            mbar_init(&bars->k_full[s], 1);
            mbar_init(&bars->v_full[s], 1);
            mbar_init(&bars->kv_empty[s], 1);
        }
        mbar_init(&bars->s_full, 1);
        mbar_init(&bars->s_free, 128);
        mbar_init(&bars->p_full, 128);
        mbar_init(&bars->pv_done, 1);
        mbar_init(&bars->mma_done, 1);
        fence_mbar_init();
    }
    if (warp == 5) {
        tmem_alloc(&bars->tmem_base, kTmemCols);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = bars->tmem_base;

    if (warp == 4) {
        // ---------------------------------------------------------------- TMA producer
        if (lane == 0) {
            tma_prefetch_desc(&tmQ);
            tma_prefetch_desc(&tmK);
            tma_prefetch_desc(&tmV);
            constexpr uint32_t kTx = L::kTileBytes;
            mbar_arrive_expect_tx(&bars->q_full, kTx);
            for (int h = 0; h < L::kHalves; ++h)
                tma_load_3d(smem + L::kQ + h * kHalfBytes, &tmQ, &bars->q_full, h * 64,
                            q_tile * kBM, bh);
            int issued = 0;
            for (int j = 0; j < n_kv; ++j) {
                const int s = j % kStages;
                if (j >= kStages &&
                    !mbar_wait(&bars->kv_empty[s], ((j / kStages) - 1) & 1, timeout_ns)) {
                    record_timeout(1);
                    break;
                }
                mbar_arrive_expect_tx(&bars->k_full[s], kTx);
                for (int h = 0; h < L::kHalves; ++h)
                    tma_load_3d(smem + L::kK + s * L::kTileBytes + h * kHalfBytes, &tmK,
                                &bars->k_full[s], h * 64, j * kBN, bh);
                mbar_arrive_expect_tx(&bars->v_full[s], kTx);
                for (int h = 0; h < L::kHalves; ++h)
                    tma_load_3d(smem + L::kV + s * L::kTileBytes + h * kHalfBytes, &tmV,
                                &bars->v_full[s], h * 64, j * kBN, bh);
                issued = j + 1;
            }
            // Drain: every load this thread issued has landed before the CTA may exit.
            // (Each stage's last load is the last phase of its barriers, so the wait ends.)
            const uint64_t drain_ns = timeout_ns > kDrainNs ? timeout_ns : kDrainNs;
            mbar_wait(&bars->q_full, 0, drain_ns);
            for (int s = 0; s < kStages && s < issued; ++s) {
                const int jl = s + ((issued - 1 - s) / kStages) * kStages;
                mbar_wait(&bars->k_full[s], (jl / kStages) & 1, drain_ns);
                mbar_wait(&bars->v_full[s], (jl / kStages) & 1, drain_ns);
            }
        }
    } else if (warp == 5) {
        // ---------------------------------------------------------------- MMA issuer
        if (lane == 0) {
            constexpr uint32_t idS = idesc_bf16_f32(kBM, kBN, 0);
            constexpr uint32_t idO = idesc_bf16_f32(kBM, D, 1);
            bool ok = mbar_wait(&bars->q_full, 0, timeout_ns);
            if (!ok) record_timeout(2);
            auto issue_s = [&](int j) -> bool {
                const int s = j % kStages;
                if (!mbar_wait(&bars->k_full[s], (j / kStages) & 1, timeout_ns)) return false;
                tc_fence_after();
                const uint32_t kb = sK + s * L::kTileBytes;
#pragma unroll
                for (int kk = 0; kk < D / 16; ++kk) {
                    const uint32_t off = (kk >> 2) * kHalfBytes + (kk & 3) * 32;
                    umma_ss(tmem + kTmemS, smem_desc_sw128(sQ + off, 16, 1024),
                            smem_desc_sw128(kb + off, 16, 1024), idS, kk > 0 ? 1u : 0u);
                }
                umma_commit(&bars->s_full);
                return true;
            };
            if (ok && !issue_s(0)) {
                record_timeout(3);
                ok = false;
            }
            for (int j = 0; ok && j < n_kv; ++j) {
                if (j + 1 < n_kv) {
                    if (!mbar_wait(&bars->s_free, j & 1, timeout_ns) || !issue_s(j + 1)) {
                        record_timeout(4);
                        break;
                    }
                }
                const int s = j % kStages;
                if (!mbar_wait(&bars->v_full[s], (j / kStages) & 1, timeout_ns) ||
                    !mbar_wait(&bars->p_full, j & 1, timeout_ns)) {
                    record_timeout(5);
                    break;
                }
                tc_fence_after();
                const uint32_t vb = sV + s * L::kTileBytes;
#pragma unroll
                for (int kk = 0; kk < kBN / 16; ++kk) {
                    const uint32_t poff = (kk >> 2) * kHalfBytes + (kk & 3) * 32;
                    umma_ss(tmem + kTmemO, smem_desc_sw128(sP + poff, 16, 1024),
                            smem_desc_sw128(vb + kk * 2048, kHalfBytes, 1024), idO,
                            (j > 0 || kk > 0) ? 1u : 0u);
                }
                umma_commit(&bars->pv_done);
                umma_commit(&bars->kv_empty[s]);
            }
            // Drain: no MMA may still write TMEM when it is freed.
            umma_commit(&bars->mma_done);
            mbar_wait(&bars->mma_done, 0, timeout_ns > kDrainNs ? timeout_ns : kDrainNs);
        }
        __syncwarp();
    } else {
        // ---------------------------------------------------------------- softmax warps
        const int r = threadIdx.x;  // row in the tile == TMEM lane
        const uint32_t lane_addr = static_cast<uint32_t>(warp * 32) << 16;
        const uint32_t tS = tmem + lane_addr + kTmemS;
        const uint32_t tO = tmem + lane_addr + kTmemO;
        const int q_row = q_tile * kBM + r;
        const int key_limit = CAUSAL ? min(N - 1, q_row) : N - 1;  // last allowed key
        float m = -INFINITY;  // running max of scale*log2(e)*s
        float l = 0.f;        // running sum of 2^(t - m)
        bool ok = true;
        for (int j = 0; j < n_kv; ++j) {
            if (!warp_wait(&bars->s_full, j & 1, timeout_ns)) {
                record_timeout(6);
                ok = false;
                break;
            }
            tc_fence_after();
            uint32_t sr[128];
            tmem_ld128_sync(tS, sr);
            tc_fence_before();
            mbar_arrive(&bars->s_free);  // S is in registers: the next S may overwrite it

            const int kv0 = j * kBN;
            if (kv0 + kBN - 1 > key_limit) {
#pragma unroll
                for (int e = 0; e < 128; ++e)
                    if (kv0 + e > key_limit) sr[e] = __float_as_uint(-INFINITY);
            }
            float mx8[8];
#pragma unroll
            for (int u = 0; u < 8; ++u) mx8[u] = __uint_as_float(sr[u]);
#pragma unroll
            for (int e = 8; e < 128; ++e) mx8[e & 7] = fmaxf(mx8[e & 7], __uint_as_float(sr[e]));
            const float mx = fmaxf(fmaxf(fmaxf(mx8[0], mx8[1]), fmaxf(mx8[2], mx8[3])),
                                   fmaxf(fmaxf(mx8[4], mx8[5]), fmaxf(mx8[6], mx8[7])));
            const float m_new = fmaxf(m, mx * scale_log2);
            // A row with nothing allowed yet keeps m = -inf; shift by 0 so no -inf - -inf.
            const float m_use = (m_new == -INFINITY) ? 0.f : m_new;
            const float alpha = ex2_approx(m - m_use);
            float rs8[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
            uint32_t p[64];
#pragma unroll
            for (int e = 0; e < 128; e += 2) {
                const float a = ex2_approx(fmaf(__uint_as_float(sr[e]), scale_log2, -m_use));
                const float b = ex2_approx(fmaf(__uint_as_float(sr[e + 1]), scale_log2, -m_use));
                rs8[(e >> 1) & 7] += a + b;
                p[e >> 1] = pack_bf16x2(a, b);
            }
            const float rs = ((rs8[0] + rs8[1]) + (rs8[2] + rs8[3])) +
                             ((rs8[4] + rs8[5]) + (rs8[6] + rs8[7]));
            l = l * alpha + rs;
            m = m_new;

            if (j > 0) {
                // The previous P V must be done: it reads P from shared memory and writes O.
                if (!warp_wait(&bars->pv_done, (j - 1) & 1, timeout_ns)) {
                    record_timeout(7);
                    ok = false;
                    break;
                }
                tc_fence_after();
                if (__any_sync(0xffffffffu, alpha != 1.f)) {
#pragma unroll
                    for (int c = 0; c < D / 32; ++c) {
                        uint32_t o[32];
                        tmem_ld32_sync(tO + c * 32, o);
#pragma unroll
                        for (int e = 0; e < 32; ++e)
                            o[e] = __float_as_uint(__uint_as_float(o[e]) * alpha);
                        tmem_st32_sync(tO + c * 32, o);
                    }
                }
            }
            // P row r -> K-major, 128-byte swizzled operand tile (two 64-key halves).
#pragma unroll
            for (int c = 0; c < 16; ++c) {
                const uint32_t addr = sP + (c >> 3) * kHalfBytes + r * 128 +
                                      ((static_cast<uint32_t>(c & 7) ^ (r & 7)) << 4);
                st_shared_v4(addr, p[4 * c], p[4 * c + 1], p[4 * c + 2], p[4 * c + 3]);
            }
            fence_proxy_async_smem();
            tc_fence_before();
            mbar_arrive(&bars->p_full);
        }
        if (ok && !warp_wait(&bars->pv_done, (n_kv - 1) & 1, timeout_ns)) {
            record_timeout(8);
            ok = false;
        }
        tc_fence_after();
        if (ok) {
            // Epilogue: O = acc / l in bf16, LSE = (m + log2 l) * ln 2.
            const float inv_l = l > 0.f ? 1.f / l : 0.f;
            const bool store = q_row < N;
            __nv_bfloat16* orow = O + (static_cast<size_t>(bh) * N + q_row) * D;
#pragma unroll
            for (int c = 0; c < D / 32; ++c) {
                uint32_t o[32];
                tmem_ld32_sync(tO + c * 32, o);
                uint32_t pk[16];
#pragma unroll
                for (int e = 0; e < 16; ++e)
                    pk[e] = pack_bf16x2(__uint_as_float(o[2 * e]) * inv_l,
                                        __uint_as_float(o[2 * e + 1]) * inv_l);
                if (store) {
                    uint4* dst = reinterpret_cast<uint4*>(orow + c * 32);
#pragma unroll
                    for (int v = 0; v < 4; ++v)
                        dst[v] = make_uint4(pk[4 * v], pk[4 * v + 1], pk[4 * v + 2], pk[4 * v + 3]);
                }
            }
            if (store && LSE != nullptr)
                LSE[static_cast<size_t>(bh) * N + q_row] = (m + __log2f(l)) * 0.69314718055994531f;
        }
    }

    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    if (warp == 5) tmem_dealloc(tmem, kTmemCols);
}

template <int D, bool CAUSAL>
int launch_one(const CUtensorMap& tq, const CUtensorMap& tk, const CUtensorMap& tv, void* O,
               float* LSE, int N, int BH, float scale, cudaStream_t stream) {
    using L = Layout<D>;
    static std::once_flag once;
    static cudaError_t attr_err = cudaSuccess;
    std::call_once(once, [] {
        attr_err = cudaFuncSetAttribute(fa_fwd_kernel<D, CAUSAL>,
                                        cudaFuncAttributeMaxDynamicSharedMemorySize, L::kDynSmem);
    });
    if (attr_err != cudaSuccess) return FA_ERR_CUDA;
    const int n_qtiles = (N + kBM - 1) / kBM;
    const long long ctas = static_cast<long long>(n_qtiles) * BH;
    if (ctas > 0x7fffffffLL) return FA_ERR_UNSUPPORTED;
    const float scale_log2 = scale * 1.4426950408889634f;
    fa_fwd_kernel<D, CAUSAL><<<static_cast<unsigned>(ctas), kThreads, L::kDynSmem, stream>>>(
        tq, tk, tv, static_cast<__nv_bfloat16*>(O), LSE, N, BH, n_qtiles, scale_log2,
        fa_wait_timeout_ns());
    return cudaGetLastError() == cudaSuccess ? FA_OK : FA_ERR_CUDA;
}

}  // namespace

int fa_fwd_launch(const void* Q, const void* K, const void* V, void* O, float* LSE, int64_t BH,
                  int64_t N, int64_t d, float scale, bool causal, cudaStream_t stream) {
    if (N > (1LL << 30) || BH > (1LL << 30)) return FA_ERR_UNSUPPORTED;
    CUtensorMap tq, tk, tv;
    int st = make_bhnd_tensor_map(&tq, Q, BH, N, d);
    if (st == FA_OK) st = make_bhnd_tensor_map(&tk, K, BH, N, d);
    if (st == FA_OK) st = make_bhnd_tensor_map(&tv, V, BH, N, d);
    if (st != FA_OK) return st;
    const int n = static_cast<int>(N), bh = static_cast<int>(BH);
    if (d == 64)
        return causal ? launch_one<64, true>(tq, tk, tv, O, LSE, n, bh, scale, stream)
                      : launch_one<64, false>(tq, tk, tv, O, LSE, n, bh, scale, stream);
    if (d == 128)
        return causal ? launch_one<128, true>(tq, tk, tv, O, LSE, n, bh, scale, stream)
                      : launch_one<128, false>(tq, tk, tv, O, LSE, n, bh, scale, stream);
    return FA_ERR_UNSUPPORTED;
}

int fa_read_device_status(cudaStream_t stream, int* status) {
    if (cudaStreamSynchronize(stream) != cudaSuccess) return FA_ERR_CUDA;
    int v = 0;
    if (cudaMemcpyFromSymbol(&v, g_fa_device_status, sizeof(int)) != cudaSuccess)
        return FA_ERR_CUDA;
    const int zero = 0;
    if (cudaMemcpyToSymbol(g_fa_device_status, &zero, sizeof(int)) != cudaSuccess)
        return FA_ERR_CUDA;
    *status = v;
    return FA_OK;
}

}  // namespace osm
