// fa_bwd.cu -- gradients of the exact attention (the backward pass), for sm_103a.
//
// The method: the pages say training recomputes the scores in the backward pass instead of
// storing them ("FlashAttention" (paweldubiel.com notes), "Mechanism and details"; "How
// FlashAttention avoids storing the giant score table" (spicyshark.co, Online softmax lesson),
// "Where this is used in practice").  With the forward's log-sum-exp the shares of a key tile
// are recomputed as P = exp(scale S - LSE) without any running max, and the derivative of the
// definition gives, for the output gradient dO,
//     dV_j = sum_i P_ij dO_i,  dP_ij = dO_i . V_j,  D_i = dO_i . O_i,  dS_ij = P_ij (dP_ij - D_i),
//     dQ_i = scale sum_j dS_ij K_j,  dK_j = scale sum_i dS_ij Q_i.
//
// GB300 mapping.  One CTA (4 warps) per (head, 128-key tile) walks the query tiles that see
// its keys.  Every product runs on the tensor cores (tcgen05.mma, fp32 accumulators in TMEM),
// issued by one thread:
//   S^T  = K Q^T    (keys x queries)      A = K, B = Q      shared memory
//   dP^T = V dO^T   (keys x queries)      A = V, B = dO     shared memory
//   dV  += P^T dO   (keys x d)            A = P^T (TMEM, bf16), B = dO
//   dK  += dS^T Q   (keys x d)            A = dS^T (TMEM, bf16), B = Q
//   dQ_i = dS K     (queries x d)         A = dS (shared memory, written by the threads), B = K
// Thread r owns key row r (its TMEM lane) for P and dS and query row r for dQ_i, whose fp32
// partial sums are added to a workspace with vector reductions (each query tile receives one
// from every key tile); a last kernel scales it by `scale` into bf16 dQ.  D is computed first
// by its own kernel.  The steps of a query tile run one after the other (load, two products,
// shares, three products, dQ out): this kernel is written for clarity, not yet overlapped.
// TMEM (512 columns): S^T [0,128), whose 32-column groups, once read, take P^T and dS^T of the
// same queries (P^T in the first 16 columns of a group, dS^T in the last 16); dP^T [128,256)
// then dQ_i [128, 128 + d); dV [256, 256 + d); dK [256 + d, 256 + 2d).
//
// Every wait is bounded; a wait that gives up records FA_ERR_TIMEOUT and the CTA stops after
// draining its own loads and products.
#include <cuda_runtime.h>

#include <cmath>
#include <mutex>

#include "osm_internal.h"
#include "ptx_sm103.cuh"

namespace osm {
namespace {

constexpr int kTile = 128;
constexpr int kThreads = 128;
constexpr int kHalf = 128 * 128;  // bytes of one 64-column half of a 128-row bf16 tile
constexpr uint64_t kDrainNs = 1000000000ull;

template <int D>
struct BwdCfg {
    static constexpr int kTileBytes = (D / 64) * kHalf;
    static constexpr int kK = 0;
    static constexpr int kV = kK + kTileBytes;
    static constexpr int kQ = kV + kTileBytes;
    static constexpr int kG = kQ + kTileBytes;   // dO
    static constexpr int kS = kG + kTileBytes;   // dS^T, 128 keys x 128 queries bf16
    static constexpr int kLse = kS + 2 * kHalf;  // 128 floats
    static constexpr int kDd = kLse + 512;       // 128 floats
    static constexpr int kBar = kDd + 512;       // mbarriers
    static constexpr int kBytes = kBar + 64;
    // Every CTA holds all 512 TMEM columns: the request is kept above half of the SM's shared
    // memory so that two CTAs never share an SM (the second would wait in its allocation).
    static constexpr int kDynSmem = kBytes + 1024 > 116 * 1024 ? kBytes + 1024 : 116 * 1024;
    static constexpr uint32_t kTmemS = 0, kTmemDP = 128;
    static constexpr uint32_t kTmemDQ = 128, kTmemDV = 256, kTmemDK = 256 + D;
    static_assert(kTmemDK + D <= 512, "TMEM budget");
    static_assert(kDynSmem <= 227 * 1024, "shared memory budget");
};

struct BwdParams {
    float* ws_dQ;       // [BH, N, D] fp32, zeroed by the first kernel
    const float* LSE;   // [BH, N]
    const float* Dv;    // [BH, N]
    __nv_bfloat16* dK;  // [BH, N, D]
    __nv_bfloat16* dV;
    int N, n_tiles;
    float scale, scale_log2;
    unsigned long long timeout_ns;
    int* status;  // the library's device status word
};

__device__ __forceinline__ void red_add_v4(float* p, float a, float b, float c, float d) {
    asm volatile("red.global.add.v4.f32 [%0], {%1, %2, %3, %4};" ::"l"(p), "f"(a), "f"(b),
                 "f"(c), "f"(d)
                 : "memory");
}

// D_i = dO_i . O_i for every row (fp32 from the bf16 rows), and the dQ workspace set to zero.
// One warp per row.
template <int D>
__global__ void __launch_bounds__(256) bwd_prep_kernel(const __nv_bfloat16* __restrict__ O,
                                                       const __nv_bfloat16* __restrict__ dO,
                                                       float* __restrict__ Dv,
                                                       float* __restrict__ ws_dQ,
                                                       long long rows) {
    constexpr int E = D / 32;
    const int lane = threadIdx.x & 31;
    for (long long r = (static_cast<long long>(blockIdx.x) * blockDim.x + threadIdx.x) >> 5;
         r < rows; r += (static_cast<long long>(gridDim.x) * blockDim.x) >> 5) {
        float acc = 0.f;
#pragma unroll
        for (int e = 0; e < E; ++e) {
            const size_t k = static_cast<size_t>(r) * D + lane * E + e;
            acc += __bfloat162float(O[k]) * __bfloat162float(dO[k]);
            ws_dQ[k] = 0.f;
        }
#pragma unroll
        for (int off = 16; off > 0; off >>= 1) acc += __shfl_xor_sync(0xffffffffu, acc, off);
        if (lane == 0) Dv[r] = acc;
    }
}

// dQ = scale * workspace, to bf16.
__global__ void __launch_bounds__(256) bwd_dq_kernel(const float* __restrict__ ws,
                                                     __nv_bfloat16* __restrict__ dQ, float scale,
                                                     long long n) {
    for (long long i = static_cast<long long>(blockIdx.x) * blockDim.x + threadIdx.x; i < n;
         i += static_cast<long long>(gridDim.x) * blockDim.x)
        dQ[i] = __float2bfloat16_rn(ws[i] * scale);
}

template <int D, bool CAUSAL>
__global__ void __launch_bounds__(kThreads, 1)
    bwd_kernel(const __grid_constant__ CUtensorMap tmQ, const __grid_constant__ CUtensorMap tmK,
               const __grid_constant__ CUtensorMap tmV, const __grid_constant__ CUtensorMap tmG,
               const BwdParams prm) {
    using C = BwdCfg<D>;
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
    uint64_t* bar_kv = reinterpret_cast<uint64_t*>(smem + C::kBar);
    uint64_t* bar_qg = bar_kv + 1;
    uint64_t* bar_mma = bar_kv + 2;
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(bar_kv + 3);
    float* lse_s = reinterpret_cast<float*>(smem + C::kLse);
    float* d_s = reinterpret_cast<float*>(smem + C::kDd);
    const int tid = threadIdx.x, warp = tid >> 5;
    const int bh = blockIdx.x / prm.n_tiles, jt = blockIdx.x % prm.n_tiles;
    const int N = prm.N;
    const unsigned long long tmo = prm.timeout_ns;

    if (tid == 0) {
        mbar_init(bar_kv, 1);
        mbar_init(bar_qg, 1);
        mbar_init(bar_mma, 1);
        fence_mbar_init();
    }
    if (warp == 0) {
        tmem_alloc(tmem_slot, 512);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tmem_slot;
    const uint32_t lane_addr = static_cast<uint32_t>(warp * 32) << 16;

    if (tid == 0) {
        mbar_arrive_expect_tx(bar_kv, 2 * C::kTileBytes);
        for (int h = 0; h < D / 64; ++h) {
            tma_load_3d(smem + C::kK + h * kHalf, &tmK, bar_kv, h * 64, jt * kTile, bh);
            tma_load_3d(smem + C::kV + h * kHalf, &tmV, bar_kv, h * 64, jt * kTile, bh);
        }
    }
    bool ok = mbar_wait(bar_kv, 0, tmo);
    ok = __syncthreads_and(ok);
    if (!ok && tid == 0) atomicCAS(prm.status, 0, FA_ERR_TIMEOUT | (20 << 8));

    const uint32_t sK = smem_u32(smem + C::kK), sV = smem_u32(smem + C::kV);
    const uint32_t sQ = smem_u32(smem + C::kQ), sG = smem_u32(smem + C::kG);
    const uint32_t sS = smem_u32(smem + C::kS);
    const int key = jt * kTile + tid;  // this thread's key row
    const int i_begin = CAUSAL ? jt : 0;
    const int n_q = (N + kTile - 1) / kTile;
    int phase = 0, mphase = 0;
    int issued_loads = 0;
    bool mma_pending = false;  // products issued whose completion has not been waited for
    bool first = true;

    for (int it = i_begin; ok && it < n_q; ++it) {
        // ---- load Q_i, dO_i (TMA) and LSE_i, D_i (plain loads) ----------------------------
        if (tid == 0) {
            mbar_arrive_expect_tx(bar_qg, 2 * C::kTileBytes);
            for (int h = 0; h < D / 64; ++h) {
                tma_load_3d(smem + C::kQ + h * kHalf, &tmQ, bar_qg, h * 64, it * kTile, bh);
                tma_load_3d(smem + C::kG + h * kHalf, &tmG, bar_qg, h * 64, it * kTile, bh);
            }
        }
        ++issued_loads;
        {
            const int q = it * kTile + tid;
            const size_t row = static_cast<size_t>(bh) * N + q;
            lse_s[tid] = q < N ? prm.LSE[row] : INFINITY;  // past the end: share 0
            d_s[tid] = q < N ? prm.Dv[row] : 0.f;
        }
        ok = mbar_wait(bar_qg, phase, tmo);
        ok = __syncthreads_and(ok);
        if (!ok) {
            if (tid == 0) atomicCAS(prm.status, 0, FA_ERR_TIMEOUT | (21 << 8));
            break;
        }
        phase ^= 1;

        // ---- S^T = K Q^T and dP^T = V dO^T ---------------------------------------------------
        if (tid == 0) {
            tc_fence_after();
            constexpr uint32_t id = idesc_bf16_f32_ab(kTile, kTile, 0, 0);
            for (int kk = 0; kk < D / 16; ++kk) {
                const uint32_t off = (kk >> 2) * kHalf + (kk & 3) * 32;
                umma_ss(tmem + C::kTmemS, smem_desc_sw128(sK + off, 16, 1024),
                        smem_desc_sw128(sQ + off, 16, 1024), id, kk > 0 ? 1u : 0u);
            }
            for (int kk = 0; kk < D / 16; ++kk) {
                const uint32_t off = (kk >> 2) * kHalf + (kk & 3) * 32;
                umma_ss(tmem + C::kTmemDP, smem_desc_sw128(sV + off, 16, 1024),
                        smem_desc_sw128(sG + off, 16, 1024), id, kk > 0 ? 1u : 0u);
            }
            umma_commit(bar_mma);
        }
        mma_pending = true;
        ok = mbar_wait(bar_mma, mphase, tmo);
        ok = __syncthreads_and(ok);
        if (!ok) {
            if (tid == 0) atomicCAS(prm.status, 0, FA_ERR_TIMEOUT | (22 << 8));
            break;
        }
        mphase ^= 1;
        mma_pending = false;
        tc_fence_after();

        // ---- P^T = exp(scale S^T - LSE), dS^T = P^T (dP^T - D) ------------------------------
        {
            const bool key_ok = key < N;
#pragma unroll 1
            for (int c = 0; c < 4; ++c) {  // 32 query columns at a time
                uint32_t sv[32], gv[32], pw[16], dsw[16];
                tmem_ld32_sync(tmem + lane_addr + C::kTmemS + c * 32, sv);
                tmem_ld32_sync(tmem + lane_addr + C::kTmemDP + c * 32, gv);
#pragma unroll
                for (int e = 0; e < 32; e += 2) {
                    float p2[2], d2[2];
#pragma unroll
                    for (int u = 0; u < 2; ++u) {
                        const int col = c * 32 + e + u;
                        const int q = it * kTile + col;
                        const bool allowed = key_ok && (!CAUSAL || key <= q);
                        const float p =
                            allowed ? ex2_approx(__uint_as_float(sv[e + u]) * prm.scale_log2 -
                                                 lse_s[col] * 1.4426950408889634f)
                                    : 0.f;
                        p2[u] = p;
                        d2[u] = p * (__uint_as_float(gv[e + u]) - d_s[col]);
                    }
                    pw[e / 2] = pack_bf16x2(p2[0], p2[1]);
                    dsw[e / 2] = pack_bf16x2(d2[0], d2[1]);
                }
                // P^T and dS^T of these 32 query columns (16 bf16 pairs each) go into the 32
                // columns of S^T just read: P^T at [32c, 32c + 16), dS^T at [32c + 16, 32c + 32).
                tmem_st16_sync(tmem + lane_addr + C::kTmemS + c * 32, pw);
                tmem_st16_sync(tmem + lane_addr + C::kTmemS + c * 32 + 16, dsw);
                // dS^T row `tid` into shared memory, 128-byte swizzled as a TMA tile would be:
                // half c / 2, 16-byte chunks (c % 2) * 4 .. + 4 of the row.
#pragma unroll
                for (int u = 0; u < 4; ++u) {
                    const int ch = (c & 1) * 4 + u;
                    st_shared_v4(sS + (c >> 1) * kHalf + tid * 128 + ((ch ^ (tid & 7)) << 4),
                                 dsw[4 * u], dsw[4 * u + 1], dsw[4 * u + 2], dsw[4 * u + 3]);
                }
            }
        }
        fence_proxy_async_smem();  // the tensor core reads dS^T through the async proxy
        tc_fence_before();
        __syncthreads();

        // ---- dV += P^T dO, dK += dS^T Q, dQ_i = dS K ---------------------------------------
        if (tid == 0) {
            tc_fence_after();
            constexpr uint32_t idT = idesc_bf16_f32_ab(kTile, D, 0, 1);
            constexpr uint32_t idQ = idesc_bf16_f32_ab(kTile, D, 1, 1);
            for (int kk = 0; kk < kTile / 16; ++kk) {
                // A_k: queries 16k..16k+15 of P^T / dS^T (8 columns; see the layout above);
                // B_k: query rows 16k..16k+15 of dO / Q, MN-major (d contiguous)
                const uint32_t a = C::kTmemS + (kk >> 1) * 32 + (kk & 1) * 8;
                umma_ts(tmem + C::kTmemDV, tmem + a, smem_desc_sw128(sG + kk * 2048, kHalf, 1024),
                        idT, (!first || kk > 0) ? 1u : 0u);
                umma_ts(tmem + C::kTmemDK, tmem + a + 16,
                        smem_desc_sw128(sQ + kk * 2048, kHalf, 1024), idT,
                        (!first || kk > 0) ? 1u : 0u);
            }
            for (int kk = 0; kk < kTile / 16; ++kk)
                // A_k: key rows 16k..16k+15 of dS^T (queries contiguous), B_k: of K
                umma_ss(tmem + C::kTmemDQ, smem_desc_sw128(sS + kk * 2048, kHalf, 1024),
                        smem_desc_sw128(sK + kk * 2048, kHalf, 1024), idQ, kk > 0 ? 1u : 0u);
            umma_commit(bar_mma);
        }
        first = false;
        mma_pending = true;
        ok = mbar_wait(bar_mma, mphase, tmo);
        ok = __syncthreads_and(ok);
        if (!ok) {
            if (tid == 0) atomicCAS(prm.status, 0, FA_ERR_TIMEOUT | (23 << 8));
            break;
        }
        mphase ^= 1;
        mma_pending = false;
        tc_fence_after();

        // ---- dQ_i partial sums into the workspace -----------------------------------------
        {
            const int q = it * kTile + tid;  // TMEM lane = query row for this product
            float* dst = prm.ws_dQ + (static_cast<size_t>(bh) * N + q) * D;
#pragma unroll
            for (int c = 0; c < D / 32; ++c) {
                uint32_t v[32];
                tmem_ld32_sync(tmem + lane_addr + C::kTmemDQ + c * 32, v);
                if (q < N) {
#pragma unroll
                    for (int e = 0; e < 32; e += 4)
                        red_add_v4(dst + c * 32 + e, __uint_as_float(v[e]),
                                   __uint_as_float(v[e + 1]), __uint_as_float(v[e + 2]),
                                   __uint_as_float(v[e + 3]));
                }
            }
        }
        tc_fence_before();
        __syncthreads();
    }

    if (ok) {
        // ---- dV and scale * dK of this key tile ----------------------------------------------
        // The TMEM loads are warp-wide (.sync.aligned): every lane issues them, and only the
        // stores are limited to the keys that exist.
        tc_fence_after();
        const size_t row = static_cast<size_t>(bh) * N + (key < N ? key : 0);
#pragma unroll
        for (int c = 0; c < D / 32; ++c) {
            uint32_t v[32], k[32];
            tmem_ld32_sync(tmem + lane_addr + C::kTmemDV + c * 32, v);
            tmem_ld32_sync(tmem + lane_addr + C::kTmemDK + c * 32, k);
            if (key < N) {
                uint4* dv = reinterpret_cast<uint4*>(prm.dV + row * D + c * 32);
                uint4* dk = reinterpret_cast<uint4*>(prm.dK + row * D + c * 32);
#pragma unroll
                for (int w = 0; w < 4; ++w) {
                    dv[w] = make_uint4(
                        pack_bf16x2(__uint_as_float(v[8 * w]), __uint_as_float(v[8 * w + 1])),
                        pack_bf16x2(__uint_as_float(v[8 * w + 2]), __uint_as_float(v[8 * w + 3])),
                        pack_bf16x2(__uint_as_float(v[8 * w + 4]), __uint_as_float(v[8 * w + 5])),
                        pack_bf16x2(__uint_as_float(v[8 * w + 6]), __uint_as_float(v[8 * w + 7])));
                    const float s = prm.scale;
                    dk[w] = make_uint4(pack_bf16x2(__uint_as_float(k[8 * w]) * s,
                                                   __uint_as_float(k[8 * w + 1]) * s),
                                       pack_bf16x2(__uint_as_float(k[8 * w + 2]) * s,
                                                   __uint_as_float(k[8 * w + 3]) * s),
                                       pack_bf16x2(__uint_as_float(k[8 * w + 4]) * s,
                                                   __uint_as_float(k[8 * w + 5]) * s),
                                       pack_bf16x2(__uint_as_float(k[8 * w + 6]) * s,
                                                   __uint_as_float(k[8 * w + 7]) * s));
                }
            }
        }
    } else if (tid == 0) {
        // Drain: the loads and products this CTA started finish before it exits.
        const uint64_t drain = tmo > kDrainNs ? tmo : kDrainNs;
        mbar_wait(bar_kv, 0, drain);
        if (issued_loads > 0) mbar_wait(bar_qg, (issued_loads - 1) & 1, drain);
        if (mma_pending) mbar_wait(bar_mma, mphase, drain);
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    if (warp == 0) tmem_dealloc(tmem, 512);
}

int bwd_sm_count() {
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

template <int D, bool CAUSAL>
int launch_bwd(const CUtensorMap& tq, const CUtensorMap& tk, const CUtensorMap& tv,
               const CUtensorMap& tg, const BwdParams& prm, long long BH, cudaStream_t stream) {
    using C = BwdCfg<D>;
    static std::once_flag once;
    static cudaError_t attr = cudaSuccess;
    std::call_once(once, [] {
        attr = cudaFuncSetAttribute(bwd_kernel<D, CAUSAL>,
                                    cudaFuncAttributeMaxDynamicSharedMemorySize, C::kDynSmem);
    });
    if (attr != cudaSuccess) return FA_ERR_CUDA;
    const long long ctas = BH * prm.n_tiles;
    if (ctas > 0x7fffffffLL) return FA_ERR_UNSUPPORTED;
    bwd_kernel<D, CAUSAL>
        <<<static_cast<unsigned>(ctas), kThreads, C::kDynSmem, stream>>>(tq, tk, tv, tg, prm);
    return cudaGetLastError() == cudaSuccess ? FA_OK : FA_ERR_CUDA;
}

}  // namespace

int fa_bwd_launch(const void* Q, const void* K, const void* V, const void* O, const void* dO,
                  const float* LSE, void* dQ, void* dK, void* dV, float* ws_dQ, float* ws_D,
                  int64_t BH, int64_t N, int64_t d, float scale, bool causal,
                  cudaStream_t stream) {
    if (N > (1LL << 30) || BH > (1LL << 30)) return FA_ERR_UNSUPPORTED;
    const long long rows = BH * N;
    const long long sms = bwd_sm_count() > 0 ? bwd_sm_count() : 148;
    long long grid = (rows + 7) / 8;
    if (grid > sms * 16) grid = sms * 16;
    if (d == 64)
        bwd_prep_kernel<64><<<static_cast<unsigned>(grid), 256, 0, stream>>>(
            static_cast<const __nv_bfloat16*>(O), static_cast<const __nv_bfloat16*>(dO), ws_D,
            ws_dQ, rows);
    else
        bwd_prep_kernel<128><<<static_cast<unsigned>(grid), 256, 0, stream>>>(
            static_cast<const __nv_bfloat16*>(O), static_cast<const __nv_bfloat16*>(dO), ws_D,
            ws_dQ, rows);
    if (cudaGetLastError() != cudaSuccess) return FA_ERR_CUDA;

    CUtensorMap tq, tk, tv, tg;
    int st = make_bhnd_tensor_map(&tq, Q, BH, N, d);
    if (st == FA_OK) st = make_bhnd_tensor_map(&tk, K, BH, N, d);
    if (st == FA_OK) st = make_bhnd_tensor_map(&tv, V, BH, N, d);
    if (st == FA_OK) st = make_bhnd_tensor_map(&tg, dO, BH, N, d);
    if (st != FA_OK) return st;
    BwdParams prm{};
    prm.ws_dQ = ws_dQ;
    prm.LSE = LSE;
    prm.Dv = ws_D;
    prm.dK = static_cast<__nv_bfloat16*>(dK);
    prm.dV = static_cast<__nv_bfloat16*>(dV);
    prm.N = static_cast<int>(N);
    prm.n_tiles = static_cast<int>((N + kTile - 1) / kTile);
    prm.scale = scale;
    prm.scale_log2 = scale * 1.4426950408889634f;
    prm.timeout_ns = fa_wait_timeout_ns();
    prm.status = device_status_word();
    if (!prm.status) return FA_ERR_CUDA;
    if (d == 64)
        st = causal ? launch_bwd<64, true>(tq, tk, tv, tg, prm, BH, stream)
                    : launch_bwd<64, false>(tq, tk, tv, tg, prm, BH, stream);
    else
        st = causal ? launch_bwd<128, true>(tq, tk, tv, tg, prm, BH, stream)
                    : launch_bwd<128, false>(tq, tk, tv, tg, prm, BH, stream);
    if (st != FA_OK) return st;

    const long long n = rows * d;
    long long g2 = (n + 255) / 256;
    if (g2 > sms * 32) g2 = sms * 32;
    bwd_dq_kernel<<<static_cast<unsigned>(g2), 256, 0, stream>>>(
        ws_dQ, static_cast<__nv_bfloat16*>(dQ), scale, n);
    return cudaGetLastError() == cudaSuccess ? FA_OK : FA_ERR_CUDA;
}

}  // namespace osm
