// fa_fwd.cu -- exact attention forward, tile by tile with the online softmax, for sm_103a.
//
// The method: "How FlashAttention avoids storing the giant score table" (spicyshark.co,
// Online softmax lesson), section "From softmax to attention" (per key block: scores, new
// running max, alpha = exp(m - m_new), p = exp(s - m_new), l = l*alpha + sum p,
// acc = acc*alpha + p V, divide by l after the last block) and "The implementation" (a block
// that leaves the max at -inf adds nothing); "kbwen.com FlashAttention", sections "Two
// blocks" and "More than two blocks" (query blocks in the outer loop, key blocks inside,
// each query row with its own max, sum and partial output).  The shift used inside the
// exponentials may be any common constant per row ("The fix: subtract the maximum": the
// factor cancels), which is what allows the lazy rescale below.
//
// GB300 mapping.  One CTA owns two 128-row query tiles (t = 0, 1) of one (b, h); both walk the
// same 128-key K/V tiles, so each K/V tile is staged once for 256 query rows.
//   warps 0-3   softmax of tile 0, warps 4-7 softmax of tile 1: one query row per thread, the
//               row's TMEM lane.  tcgen05.ld of the S row (128 fp32), mask, row max, ex2 of
//               the scaled and shifted scores (scale*log2(e) folded into one FFMA), row sum,
//               P rounded to bf16 and written back into TMEM over the upper half of S.
//               At the end: O / l to bf16 and LSE = (m + log2 l) * ln 2.
//   warps 8-11  correction: when a row's reference max moved, scale that row of the O
//               accumulator in TMEM by alpha before the next P V is issued.
//   warp 12     tcgen05.mma (one thread): S_t = Q_t K^T (A and B from shared memory), then
//               O_t += P_t V (A = P_t from TMEM, B = V from shared memory); fp32 accumulators.
//               The two tiles alternate, so the tensor core works on one tile while the
//               other tile's softmax runs.
//   warp 13     TMA: Q_0, Q_1 once, K and V tiles into 2-stage rings (128-byte swizzle,
//               zero fill past N).
// TMEM (512 columns): S_0 [0,128), S_1 [128,256), O_0 [256, 256+d), O_1 [256+d, 256+2d);
// P_t occupies columns [64,128) of S_t (two bf16 per column).
// Lazy rescale: a row keeps its reference max m until a tile's max exceeds it by more than
// 8 (log2 units); the exponentials then stay <= 2^8, far inside fp32/bf16 range, and O only
// needs rescaling when the reference moves.
// Causal: key tiles above the diagonal are never visited; only diagonal and ragged tiles are
// masked element by element.
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
constexpr int kThreads = 512;  // 16 warps, see the role table above
constexpr uint32_t kTmemCols = 512;
constexpr int kHalfBytes = 128 * 128;         // one 64-column half of a 128-row bf16 tile
constexpr uint64_t kDrainNs = 1000000000ull;  // drain waits: at least 1 s
constexpr float kRescaleThreshold = 8.0f;     // log2 units

struct Bars {
    uint64_t q_full[2];
    uint64_t k_full[2], k_empty[2];
    uint64_t v_full[2], v_empty[2];
    uint64_t s_full[2];       // S_t computed (tcgen05.commit)
    uint64_t p_full[2];       // P_t written to TMEM (128 softmax threads)
    uint64_t pv_done[2];      // O_t += P_t V finished (tcgen05.commit)
    uint64_t alpha_ready[2];  // per-row rescale factors published (128 softmax threads)
    uint64_t o_ready[2];      // O_t rescaled, ready for the next P V (128 correction threads)
    uint64_t mma_done;
    uint32_t tmem_base;
    float alpha[2][kBM];
};

template <int D>
struct Layout {
    static constexpr int kHalves = D / 64;
    static constexpr int kTileBytes = kHalves * kHalfBytes;  // 128 rows x D bf16
    static constexpr int kQ = 0;                             // 2 tiles
    static constexpr int kK = kQ + 2 * kTileBytes;           // 2 stages
    static constexpr int kV = kK + 2 * kTileBytes;           // 2 stages
    static constexpr int kBars = kV + 2 * kTileBytes;
    static constexpr int kBytes = kBars + static_cast<int>(sizeof(Bars));
    static constexpr int kDynSmem = kBytes + 1024;  // slack for 1024-byte alignment
    static constexpr uint32_t kTmemO = 256;         // O_0 at 256, O_1 at 256 + D
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
                  float* __restrict__ LSE, int N, int BH, int n_pairs, float scale_log2,
                  unsigned long long timeout_ns) {
    using L = Layout<D>;
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
    Bars* bars = reinterpret_cast<Bars*>(smem + L::kBars);
    const uint32_t sQ = smem_u32(smem + L::kQ);
    const uint32_t sK = smem_u32(smem + L::kK);
    const uint32_t sV = smem_u32(smem + L::kV);

    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;

    // Work item: a pair of query tiles.  Causal runs the longest rows first.
    int pair, bh;
    if (CAUSAL) {
        pair = n_pairs - 1 - static_cast<int>(blockIdx.x) / BH;
        bh = static_cast<int>(blockIdx.x) % BH;
    } else {
        pair = static_cast<int>(blockIdx.x) % n_pairs;
        bh = static_cast<int>(blockIdx.x) / n_pairs;
    }
    const int n_kv_all = (N + kBN - 1) / kBN;
    int n_kv[2];
#pragma unroll
    for (int t = 0; t < 2; ++t) {
        const int qt = 2 * pair + t;
        if (qt * kBM >= N)
            n_kv[t] = 0;  // a tile entirely past N: nothing to compute or store
        else
            n_kv[t] = CAUSAL ? min(n_kv_all, qt + 1) : n_kv_all;
    }
    const int J = max(n_kv[0], n_kv[1]);

    if (threadIdx.x == 0) {
        for (int t = 0; t < 2; ++t) {
            mbar_init(&bars->q_full[t], 1);
            mbar_init(&bars->k_full[t], 1);
            mbar_init(&bars->k_empty[t], 1);
            mbar_init(&bars->v_full[t], 1);
            mbar_init(&bars->v_empty[t], 1);
            mbar_init(&bars->s_full[t], 1);
            mbar_init(&bars->p_full[t], 128);
            mbar_init(&bars->pv_done[t], 1);
            mbar_init(&bars->alpha_ready[t], 128);
            mbar_init(&bars->o_ready[t], 128);
        }
        mbar_init(&bars->mma_done, 1);
        fence_mbar_init();
    }
    if (warp == 12) {
        tmem_alloc(&bars->tmem_base, kTmemCols);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = bars->tmem_base;

    if (warp >= 12) {
        setmaxnreg_dec<56>();
        if (warp == 13 && lane == 0) {
            // ---------------------------------------------------------------- TMA producer
            tma_prefetch_desc(&tmQ);
            tma_prefetch_desc(&tmK);
            tma_prefetch_desc(&tmV);
            constexpr uint32_t kTx = L::kTileBytes;
            for (int t = 0; t < 2; ++t) {
                mbar_arrive_expect_tx(&bars->q_full[t], kTx);
                for (int h = 0; h < L::kHalves; ++h)
                    tma_load_3d(smem + L::kQ + t * L::kTileBytes + h * kHalfBytes, &tmQ,
                                &bars->q_full[t], h * 64, (2 * pair + t) * kBM, bh);
            }
            int k_issued = 0, v_issued = 0;
            for (int j = 0; j < J; ++j) {
                const int s = j & 1;
                const uint32_t ph = ((j >> 1) - 1) & 1;
                if (j >= 2 && !mbar_wait(&bars->k_empty[s], ph, timeout_ns)) {
                    record_timeout(1);
                    break;
                }
                mbar_arrive_expect_tx(&bars->k_full[s], kTx);
                for (int h = 0; h < L::kHalves; ++h)
                    tma_load_3d(smem + L::kK + s * L::kTileBytes + h * kHalfBytes, &tmK,
                                &bars->k_full[s], h * 64, j * kBN, bh);
                k_issued = j + 1;
                if (j >= 2 && !mbar_wait(&bars->v_empty[s], ph, timeout_ns)) {
                    record_timeout(2);
                    break;
                }
                mbar_arrive_expect_tx(&bars->v_full[s], kTx);
                for (int h = 0; h < L::kHalves; ++h)
                    tma_load_3d(smem + L::kV + s * L::kTileBytes + h * kHalfBytes, &tmV,
                                &bars->v_full[s], h * 64, j * kBN, bh);
                v_issued = j + 1;
            }
            // Drain: every load this thread issued has landed before the CTA may exit.  The
            // last load into a stage is the last phase of that stage's barrier, so it ends.
            const uint64_t drain_ns = timeout_ns > kDrainNs ? timeout_ns : kDrainNs;
            mbar_wait(&bars->q_full[0], 0, drain_ns);
            mbar_wait(&bars->q_full[1], 0, drain_ns);
            for (int s = 0; s < 2; ++s) {
                if (s < k_issued) {
                    const int jl = s + ((k_issued - 1 - s) >> 1) * 2;
                    mbar_wait(&bars->k_full[s], (jl >> 1) & 1, drain_ns);
                }
                if (s < v_issued) {
                    const int jl = s + ((v_issued - 1 - s) >> 1) * 2;
                    mbar_wait(&bars->v_full[s], (jl >> 1) & 1, drain_ns);
                }
            }
        } else if (warp == 12 && lane == 0) {
            // ---------------------------------------------------------------- MMA issuer
            constexpr uint32_t idS = idesc_bf16_f32(kBM, kBN, 0);
            constexpr uint32_t idO = idesc_bf16_f32(kBM, D, 1);
            auto issue_s = [&](int t, int j) {
                const uint32_t qb = sQ + t * L::kTileBytes;
                const uint32_t kb = sK + (j & 1) * L::kTileBytes;
#pragma unroll
                for (int kk = 0; kk < D / 16; ++kk) {
                    const uint32_t off = (kk >> 2) * kHalfBytes + (kk & 3) * 32;
                    umma_ss(tmem + t * 128, smem_desc_sw128(qb + off, 16, 1024),
                            smem_desc_sw128(kb + off, 16, 1024), idS, kk > 0 ? 1u : 0u);
                }
                umma_commit(&bars->s_full[t]);
            };
            auto issue_pv = [&](int t, int j) {
                const uint32_t vb = sV + (j & 1) * L::kTileBytes;
                const uint32_t p_tmem = tmem + t * 128 + 64;
#pragma unroll
                for (int kk = 0; kk < kBN / 16; ++kk)
                    umma_ts(tmem + L::kTmemO + t * D, p_tmem + kk * 8,
                            smem_desc_sw128(vb + kk * 2048, kHalfBytes, 1024), idO,
                            (j > 0 || kk > 0) ? 1u : 0u);
                umma_commit(&bars->pv_done[t]);
            };
            bool ok = J > 0;
            if (ok) {
                ok = mbar_wait(&bars->q_full[0], 0, timeout_ns) &&
                     mbar_wait(&bars->q_full[1], 0, timeout_ns) &&
                     mbar_wait(&bars->k_full[0], 0, timeout_ns);
                if (!ok) record_timeout(3);
            }
            if (ok) {
                tc_fence_after();
                for (int t = 0; t < 2; ++t)
                    if (n_kv[t] > 0) issue_s(t, 0);
                umma_commit(&bars->k_empty[0]);
            }
            for (int j = 0; ok && j < J; ++j) {
                const int s = j & 1;
                if (!mbar_wait(&bars->v_full[s], (j >> 1) & 1, timeout_ns)) {
                    record_timeout(4);
                    break;
                }
                bool k_next = false;  // K_{j+1} seen landed
                for (int t = 0; ok && t < 2; ++t) {
                    if (j >= n_kv[t]) continue;
                    if (!mbar_wait(&bars->p_full[t], j & 1, timeout_ns) ||
                        !mbar_wait(&bars->o_ready[t], j & 1, timeout_ns)) {
                        record_timeout(5);
                        ok = false;
                        break;
                    }
                    tc_fence_after();
                    issue_pv(t, j);
                    if (j + 1 < n_kv[t]) {
                        // S_t(j+1) overwrites the columns P_t(j) is read from: wait for P V.
                        if ((!k_next && !mbar_wait(&bars->k_full[(j + 1) & 1], ((j + 1) >> 1) & 1,
                                                   timeout_ns)) ||
                            !mbar_wait(&bars->pv_done[t], j & 1, timeout_ns)) {
                            record_timeout(6);
                            ok = false;
                            break;
                        }
                        k_next = true;
                        tc_fence_after();
                        issue_s(t, j + 1);
                    }
                }
                if (!ok) break;
                umma_commit(&bars->v_empty[s]);
                if (j + 1 < J) umma_commit(&bars->k_empty[(j + 1) & 1]);
            }
            // Drain: no MMA may still write TMEM when it is freed.
            umma_commit(&bars->mma_done);
            mbar_wait(&bars->mma_done, 0, timeout_ns > kDrainNs ? timeout_ns : kDrainNs);
        }
        __syncwarp();
    } else if (warp >= 8) {
        // -------------------------------------------------------------------- correction
        setmaxnreg_dec<72>();
        const int r = threadIdx.x - 256;  // row == TMEM lane (warp % 4 selects the lane quarter)
        const uint32_t lane_addr = static_cast<uint32_t>((warp & 3) * 32) << 16;
        bool ok = true;
        for (int j = 0; ok && j < J; ++j) {
            for (int t = 0; t < 2; ++t) {
                if (j >= n_kv[t]) continue;
                if (!warp_wait(&bars->alpha_ready[t], j & 1, timeout_ns)) {
                    record_timeout(7);
                    ok = false;
                    break;
                }
                if (j > 0) {
                    if (!warp_wait(&bars->pv_done[t], (j - 1) & 1, timeout_ns)) {
                        record_timeout(8);
                        ok = false;
                        break;
                    }
                    tc_fence_after();
                    const float a = bars->alpha[t][r];
                    if (__any_sync(0xffffffffu, a != 1.f)) {
                        const uint32_t tO = tmem + lane_addr + L::kTmemO + t * D;
#pragma unroll
                        for (int c = 0; c < D / 32; ++c) {
                            uint32_t o[32];
                            tmem_ld32_sync(tO + c * 32, o);
#pragma unroll
                            for (int e = 0; e < 32; ++e)
                                o[e] = __float_as_uint(__uint_as_float(o[e]) * a);
                            tmem_st32_sync(tO + c * 32, o);
                        }
                    }
                }
                tc_fence_before();
                mbar_arrive(&bars->o_ready[t]);
            }
        }
    } else {
        // -------------------------------------------------------------------- softmax
        setmaxnreg_inc<192>();
        const int t = warp >> 2;               // query tile of this warpgroup
        const int r = threadIdx.x & 127;        // row in the tile == TMEM lane
        const uint32_t lane_addr = static_cast<uint32_t>((warp & 3) * 32) << 16;
        const uint32_t tS = tmem + lane_addr + t * 128;
        const uint32_t tP = tS + 64;
        const uint32_t tO = tmem + lane_addr + L::kTmemO + t * D;
        const int q_row = (2 * pair + t) * kBM + r;
        const int key_limit = CAUSAL ? min(N - 1, q_row) : N - 1;  // last allowed key
        const int nkv = n_kv[t];
        float m = -INFINITY;  // reference max of scale*log2(e)*s for this row
        float l = 0.f;        // running sum of 2^(scale*log2(e)*s - m)
        bool ok = true;
        for (int j = 0; j < nkv; ++j) {
            if (!warp_wait(&bars->s_full[t], j & 1, timeout_ns)) {
                record_timeout(9);
                ok = false;
                break;
            }
            tc_fence_after();
            uint32_t sr[128];
            tmem_ld128_sync(tS, sr);

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
                                   fmaxf(fmaxf(mx8[4], mx8[5]), fmaxf(mx8[6], mx8[7]))) *
                             scale_log2;
            // Move the reference only when this tile's max exceeds it by more than the
            // threshold (always on the first finite tile: m = -inf gives +inf > threshold).
            const float m_new = (mx - m > kRescaleThreshold) ? mx : m;
            const float alpha = (m_new == m) ? 1.f : ex2_approx(m - m_new);
            bars->alpha[t][r] = alpha;
            mbar_arrive(&bars->alpha_ready[t]);
            // Nothing allowed yet (m_new = -inf): shift by 0 so every term is exp(-inf) = 0.
            const float m_use = (m_new == -INFINITY) ? 0.f : m_new;
            float rs8[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
            uint32_t p[64];
#pragma unroll
            for (int e = 0; e < 128; e += 2) {
                const float a = ex2_approx(fmaf(__uint_as_float(sr[e]), scale_log2, -m_use));
                const float b = ex2_approx(fmaf(__uint_as_float(sr[e + 1]), scale_log2, -m_use));
                rs8[(e >> 1) & 7] += a + b;
                p[e >> 1] = pack_bf16x2(a, b);
            }
            tmem_st64_sync(tP, p);
            tc_fence_before();
            mbar_arrive(&bars->p_full[t]);
            const float rs = ((rs8[0] + rs8[1]) + (rs8[2] + rs8[3])) +
                             ((rs8[4] + rs8[5]) + (rs8[6] + rs8[7]));
            l = l * alpha + rs;
            m = m_new;
        }
        if (ok && nkv > 0) {
            if (!warp_wait(&bars->pv_done[t], (nkv - 1) & 1, timeout_ns)) {
                record_timeout(10);
                ok = false;
            }
        }
        tc_fence_after();
        if (ok && nkv > 0) {
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
    if (warp == 12) tmem_dealloc(tmem, kTmemCols);
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
    const int n_pairs = (n_qtiles + 1) / 2;
    const long long ctas = static_cast<long long>(n_pairs) * BH;
    if (ctas > 0x7fffffffLL) return FA_ERR_UNSUPPORTED;
    const float scale_log2 = scale * 1.4426950408889634f;
    fa_fwd_kernel<D, CAUSAL><<<static_cast<unsigned>(ctas), kThreads, L::kDynSmem, stream>>>(
        tq, tk, tv, static_cast<__nv_bfloat16*>(O), LSE, N, BH, n_pairs, scale_log2,
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
