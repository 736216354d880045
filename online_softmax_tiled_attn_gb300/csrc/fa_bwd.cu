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
// GB300 mapping: three launches on the caller's stream.
//   1. bwd_prep_kernel: D_i = dO_i . O_i (fp32, one warp per row).
//   2. bwd_kv_kernel: one CTA per (head, 128-key tile) walks the query tiles that see its
//      keys and accumulates dK and dV of its keys in TMEM (keys = TMEM lanes).
//   3. bwd_q_kernel: one CTA per (head, 128-query tile) walks the key tiles its queries see,
//      recomputes S and dP and accumulates dQ in TMEM (queries = TMEM lanes).
// Computing dQ by its own pass costs two more products per tile pair than adding per-key-tile
// partial sums of dQ into memory, but on this part the L2 reductions that the partial sums
// need (64 KB per tile pair) run slower than the products they would save, and the pass
// leaves every gradient deterministic: each is summed in a fixed order.
//
// Both tile kernels put their roles on separate warps so that loads, tensor-core products and
// element-wise work overlap:
//   warp 16      TMA loads (the CTA's own tile once, the walked tiles into a two-stage ring).
//   warp 17      one thread issues every tcgen05.mma (bf16 operands, fp32 accumulators).
//   warps 0-15   the element-wise work, thread = TMEM lane (row), four warps per 32 lanes
//                with 16 of each 64 columns each (enough warps to hide the TMEM load and
//                store latencies); a tile's first half of the walked rows is handed to the
//                tensor cores before the second half is computed.  They also write the CTA's
//                gradients at the end.
// Every wait is bounded; a wait that gives up records FA_ERR_TIMEOUT and its role stops; the
// CTA drains its own loads and products before it frees TMEM and exits.
#include <cuda_runtime.h>

#include <cmath>
#include <mutex>

#include "osm_internal.h"
#include "ptx_sm103.cuh"

namespace osm {
namespace {

constexpr int kTile = 128;
constexpr int kHalf = 128 * 128;  // bytes of one 64-column half of a 128-row bf16 tile
constexpr int kSoftWarps = 16;    // warps 0-15
constexpr int kTmaWarp = 16;
constexpr int kMmaWarp = 17;
// The MMA warp runs its loop as a whole, converged warp and one elected lane issues each
// product and commit: the operands are then warp-uniform values, and one warp issues short
// products at the tensor core's pace (a loop run by lane 0 alone issues one per ~49-75 clocks).
constexpr bool kWarpIssue = true;
constexpr int kThreads = 18 * 32;
constexpr uint64_t kDrainNs = 1000000000ull;
constexpr float kLog2e = 1.4426950408889634f;

// Every CTA holds all 512 TMEM columns: the shared-memory request is kept above half of the
// SM's so that two CTAs never share an SM (the second would wait in its allocation).
constexpr int dyn_smem(int bytes) { return bytes + 1024 > 116 * 1024 ? bytes + 1024 : 116 * 1024; }

struct BwdParams {
    const float* LSE;   // [B H, N]
    const float* Dv;    // [B H, N], written by bwd_prep_kernel
    __nv_bfloat16* dQ;  // [B H, N, D]
    __nv_bfloat16* dK;  // [B H_kv, N, D]
    __nv_bfloat16* dV;
    int N, n_tiles;
    int H, H_kv;        // query heads and key/value heads per sequence (H_kv divides H)
    int BH, BH_kv;      // B H and B H_kv
    int head_group_q;   // query heads per L2-sized group of the dQ grid
    int head_group_kv;  // key/value heads per L2-sized group of the dK, dV grid
    const int32_t* kv_lens;  // [B] valid keys per sequence, or nullptr (all N)
    float scale, scale_log2;
    unsigned long long timeout_ns;
    int* status;  // the library's device status word
};

// Keys of sequence b that take part: kv_lens[b] clamped to [0, N], or N.
__device__ __forceinline__ int seq_keys(const BwdParams& prm, int b) {
    return prm.kv_lens ? min(max(prm.kv_lens[b], 0), prm.N) : prm.N;
}

__device__ __forceinline__ void record_timeout(int* status, int where) {
    atomicCAS(status, 0, FA_ERR_TIMEOUT | (where << 8));
}

// The grid walks groups of heads whose walked tiles fit in L2 together; inside a group the
// tile index is outer and the head inner, so that the CTAs in flight read different heads'
// tiles and, with a causal mask, the tiles with the most work start first.  Returns the head
// and the tile position (0 = first to start) of this CTA.
__device__ __forceinline__ void grid_place(int n_heads, int head_group, int n_tiles, int& bh,
                                           int& pos) {
    const int per_group = head_group * n_tiles;
    const int g = blockIdx.x / per_group, idx = blockIdx.x % per_group;
    const int heads = min(head_group, n_heads - g * head_group);
    bh = g * head_group + idx % heads;
    pos = idx / heads;
}

// Eight (d = 128) or four (d = 64) K16 steps of an SS product over K-major 128-byte swizzled
// tiles stored as 64-column halves.
template <int D>
__device__ __forceinline__ void mma_ss_kmajor(uint32_t d_tmem, uint32_t sA, uint32_t sB,
                                              uint32_t idesc) {
    issue_ss_x4<kWarpIssue>(d_tmem, smem_desc_sw128(sA, 16, 1024),
                            smem_desc_sw128(sB, 16, 1024), idesc, 0u);
    if constexpr (D == 128)
        issue_ss_x4<kWarpIssue>(d_tmem, smem_desc_sw128(sA + kHalf, 16, 1024),
                                smem_desc_sw128(sB + kHalf, 16, 1024), idesc, 1u);
}

// Rows [64 half, 64 half + 64) of the walked dimension of a TS product whose A operand (bf16
// pairs, in TMEM) starts every 16-column group (the layout the element-wise warps write: the
// 16 walked rows of K16 step k at columns 16 k .. 16 k + 7); B is the MN-major tile at sB.
__device__ __forceinline__ void mma_ts_half(uint32_t d_tmem, uint32_t a_tmem, uint32_t sB,
                                            int half, uint32_t idesc, uint32_t accumulate) {
    issue_ts_x4_stride16<kWarpIssue>(d_tmem, a_tmem + half * 64,
                                     smem_desc_sw128(sB + half * 4 * 2048, kHalf, 1024), idesc,
                                     accumulate);
}

// Writes N fp32 values (times sc) of one row as bf16.
template <int N>
__device__ __forceinline__ void store_row(__nv_bfloat16* dst, const uint32_t (&v)[N], float sc) {
    uint4* o = reinterpret_cast<uint4*>(dst);
#pragma unroll
    for (int w = 0; w < N / 8; ++w)
        o[w] = make_uint4(
            pack_bf16x2(__uint_as_float(v[8 * w]) * sc, __uint_as_float(v[8 * w + 1]) * sc),
            pack_bf16x2(__uint_as_float(v[8 * w + 2]) * sc, __uint_as_float(v[8 * w + 3]) * sc),
            pack_bf16x2(__uint_as_float(v[8 * w + 4]) * sc, __uint_as_float(v[8 * w + 5]) * sc),
            pack_bf16x2(__uint_as_float(v[8 * w + 6]) * sc, __uint_as_float(v[8 * w + 7]) * sc));
}

// D_i = dO_i . O_i for every row (fp32 from the bf16 rows).  One warp per row.
template <int D>
__global__ void __launch_bounds__(256) bwd_prep_kernel(const __nv_bfloat16* __restrict__ O,
                                                       const __nv_bfloat16* __restrict__ dO,
                                                       float* __restrict__ Dv, long long rows) {
    constexpr int E = D / 32;
    const int lane = threadIdx.x & 31;
    for (long long r = (static_cast<long long>(blockIdx.x) * blockDim.x + threadIdx.x) >> 5;
         r < rows; r += (static_cast<long long>(gridDim.x) * blockDim.x) >> 5) {
        float acc = 0.f;
#pragma unroll
        for (int e = 0; e < E; ++e) {
            const size_t k = static_cast<size_t>(r) * D + lane * E + e;
            acc += __bfloat162float(O[k]) * __bfloat162float(dO[k]);
        }
#pragma unroll
        for (int off = 16; off > 0; off >>= 1) acc += __shfl_xor_sync(0xffffffffu, acc, off);
        if (lane == 0) Dv[r] = acc;
    }
}

// ============================================================================================
// dK, dV: one CTA per (head, key tile)
// ============================================================================================
// TMEM (512 columns): two buffers of 128 columns (keys x queries), one per query tile in
// flight, and the accumulators dV [256, 256 + d), dK [256 + d, 256 + 2d).  The buffer of query
// tile t holds in turn:
//   S^T = K Q_t^T        B = Q_t (shared memory, K-major)
//   dP^T = V dO_t^T      B = dO_t, written over S^T once the element-wise warps have read it
//                        (they keep the shares P^T in registers meanwhile)
//   P^T, dS^T (bf16)     written over dP^T by the element-wise warps: each 16-column group,
//                        read by the warp that owns it, takes P^T in its first 8 columns and
//                        dS^T in its last 8
//   dV += P^T dO_t, dK += dS^T Q_t     A in TMEM, B = dO_t, Q_t MN-major
// For d = 64 K and V, the A operands of S^T and dP^T, are copied once into TMEM too (the last
// 64 columns): those products then read only B from shared memory (an N = 128 product with
// both operands in shared memory needs the port's whole 128 bytes a clock), and their shared
// memory serves a three-stage Q, dO ring.  For d = 128 TMEM has no room for them: they stay in
// shared memory with a two-stage ring.
template <int D>
struct KvCfg {
    static constexpr int kTileBytes = (D / 64) * kHalf;
    static constexpr bool kKvInTmem = D == 64;
    static constexpr int kStages = kKvInTmem ? 3 : 2;
    static constexpr int kK = 0;                             // K, V (d = 128)
    static constexpr int kV = kK + kTileBytes;
    static constexpr int kQ = kKvInTmem ? 0 : kV + kTileBytes;  // Q, kStages stages
    static constexpr int kG = kQ + kStages * kTileBytes;     // dO, kStages stages
    static constexpr int kLD = kG + kStages * kTileBytes;    // per query pair: -LSE log2e, -D
    static constexpr int kBar = kLD + 1024;
    static constexpr int kBytes = kBar + 256;
    static constexpr int kDynSmem = dyn_smem(kBytes);
    // d = 64: K and V arrive in the last stage (its Q and dO halves) and are copied to TMEM
    // before the stage's first Q, dO load.
    static constexpr int kKLoad = kKvInTmem ? kQ + (kStages - 1) * kTileBytes : kK;
    static constexpr int kVLoad = kKvInTmem ? kG + (kStages - 1) * kTileBytes : kV;
    static constexpr uint32_t kTmemBuf = 0, kTmemDV = 256, kTmemDK = 256 + D;
    static constexpr uint32_t kTmemK = kTmemDK + D, kTmemV = kTmemK + D / 2;
    static_assert(kKvInTmem ? kTmemV + D / 2 <= 512 : kTmemDK + D <= 512, "TMEM budget");
    static_assert(kDynSmem <= 227 * 1024, "shared memory budget");
};

enum KvBar {
    kKvBarKV = 0,       // K, V landed
    kKvBarKVCopied = 1, // K, V copied to TMEM: their shared memory may be reused (d = 64)
    kKvBarFull = 2,     // [3] Q_t, dO_t landed in a stage
    kKvBarEmpty = 5,    // [3] a stage's products are done
    kKvBarSFull = 8,    // [2] S^T in TMEM buffer b
    kKvBarSFree = 10,   // [2] the dV, dK products have read buffer b
    kKvBarRead = 12,    // S^T read (one arrival per element-wise warp)
    kKvBarDpFull = 13,  // dP^T in the buffer
    kKvBarPds = 14,     // [2] P^T, dS^T of query half h written (one arrival per warp)
    kKvBarAcc = 16,     // the last dV, dK products done
    kKvBarDrain = 17,   // the issuing thread's products done, on the way out after a timeout
    kKvNumBars = 18
};

// The shares of 16 queries (columns c0 .. c0 + 15 of the buffer at t_buf) for this thread's
// key row: P = exp2(S scale log2e - LSE log2e).  `lo`: first allowed query column of the row
// (0 unless the tile needs masking; 128 masks the row).
template <bool MASK>
__device__ __forceinline__ void kv_shares(uint32_t t_buf, const float4* ld, int c0, int lo,
                                          float scale_log2, float (&p)[16]) {
    uint32_t sv[16];
    tmem_ld16_sync(t_buf + c0, sv);
    const float2 sl2 = make_float2(scale_log2, scale_log2);
#pragma unroll
    for (int e = 0; e < 8; ++e) {
        const float4 L = ld[c0 / 2 + e];  // columns c0 + 2e, +1: -LSE log2e, -D
        const float2 a = ffma2(make_float2(__uint_as_float(sv[2 * e]), __uint_as_float(sv[2 * e + 1])),
                               sl2, make_float2(L.x, L.y));
        p[2 * e] = ex2_approx(a.x);
        p[2 * e + 1] = ex2_approx(a.y);
        if (MASK) {
            if (c0 + 2 * e < lo) p[2 * e] = 0.f;
            if (c0 + 2 * e + 1 < lo) p[2 * e + 1] = 0.f;
        }
    }
}

// dS = P (dP - D) of the same 16 queries from the dP^T columns, then P^T and dS^T (bf16 pairs)
// written over those columns: P^T in the first 8, dS^T in the last 8.
__device__ __forceinline__ void kv_grads(uint32_t t_buf, const float4* ld, int c0,
                                         const float (&p)[16]) {
    uint32_t gv[16];
    tmem_ld16_sync(t_buf + c0, gv);
    uint32_t pw[8], dw[8];
#pragma unroll
    for (int e = 0; e < 8; ++e) {
        const float4 L = ld[c0 / 2 + e];
        const float2 g = fadd2(make_float2(__uint_as_float(gv[2 * e]), __uint_as_float(gv[2 * e + 1])),
                               make_float2(L.z, L.w));
        const float2 ds = fmul2(make_float2(p[2 * e], p[2 * e + 1]), g);
        pw[e] = pack_bf16x2(p[2 * e], p[2 * e + 1]);
        dw[e] = pack_bf16x2(ds.x, ds.y);
    }
    tmem_st8x2_sync(t_buf + c0, pw, t_buf + c0 + 8, dw);
}

// A TS product over d: A (bf16 pairs, d / 2 TMEM columns at a_tmem) times the K-major,
// 128-byte swizzled tile at sB (64-column halves), overwriting D.
template <int D>
__device__ __forceinline__ void mma_ts_kmajor(uint32_t d_tmem, uint32_t a_tmem, uint32_t sB,
                                              uint32_t idesc) {
#pragma unroll
    for (int h = 0; h < D / 64; ++h)
        issue_ts_x4<kWarpIssue>(d_tmem, a_tmem + h * 32,
                                smem_desc_sw128(sB + h * kHalf, 16, 1024), 32 / 16, idesc,
                                h > 0 ? 1u : 0u);
}

template <int D, bool CAUSAL>
__global__ void __launch_bounds__(kThreads, 1)
    bwd_kv_kernel(const __grid_constant__ CUtensorMap tmQ, const __grid_constant__ CUtensorMap tmK,
                  const __grid_constant__ CUtensorMap tmV, const __grid_constant__ CUtensorMap tmG,
                  const BwdParams prm) {
    using C = KvCfg<D>;
    constexpr int NS = C::kStages;
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
    uint64_t* bars = reinterpret_cast<uint64_t*>(smem + C::kBar);
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(bars + kKvNumBars);
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    // Key tile 0 sees the most query tiles under a causal mask: it starts first.  bhk: the
    // key/value head; its query heads are bh_q0 .. bh_q0 + group - 1, whose query tiles are
    // walked one head after another (the key and value gradients of a shared head sum over
    // its query heads).  Keys at or past the sequence's length take no part.
    int bhk, jt;
    grid_place(prm.BH_kv, prm.head_group_kv, prm.n_tiles, bhk, jt);
    const int N = prm.N;
    const int group = prm.H / prm.H_kv;
    const int b_seq = bhk / prm.H_kv;
    const int bh_q0 = b_seq * prm.H + (bhk - b_seq * prm.H_kv) * group;
    const int len = seq_keys(prm, b_seq);
    const int i0 = CAUSAL ? jt : 0;
    const int n_it1 = prm.n_tiles - i0;  // query tiles walked per query head
    // A key tile with no key below the length walks nothing; its gradients are 0.
    const int n_it = jt * kTile < len ? group * n_it1 : 0;
    const unsigned long long tmo = prm.timeout_ns;

    if (threadIdx.x == 0) {
        mbar_init(&bars[kKvBarKV], 1);
        mbar_init(&bars[kKvBarKVCopied], 1);
        for (int s = 0; s < NS; ++s) {
            mbar_init(&bars[kKvBarFull + s], 1);
            mbar_init(&bars[kKvBarEmpty + s], 1);
        }
        for (int s = 0; s < 2; ++s) {
            mbar_init(&bars[kKvBarSFull + s], 1);
            mbar_init(&bars[kKvBarSFree + s], 1);
            mbar_init(&bars[kKvBarPds + s], kSoftWarps);
        }
        mbar_init(&bars[kKvBarRead], kSoftWarps);
        mbar_init(&bars[kKvBarDpFull], 1);
        mbar_init(&bars[kKvBarAcc], 1);
        mbar_init(&bars[kKvBarDrain], 1);
        fence_mbar_init();
    }
    if (warp == kMmaWarp) {
        tmem_alloc(tmem_slot, 512);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tmem_slot;

    if (warp == kTmaWarp) {
        if (lane == 0 && n_it > 0) {
            // ---- loads ----------------------------------------------------------------------
            mbar_arrive_expect_tx(&bars[kKvBarKV], 2 * C::kTileBytes);
            for (int h = 0; h < D / 64; ++h) {
                tma_load_3d(smem + C::kKLoad + h * kHalf, &tmK, &bars[kKvBarKV], h * 64,
                            jt * kTile, bhk);
                tma_load_3d(smem + C::kVLoad + h * kHalf, &tmV, &bars[kKvBarKV], h * 64,
                            jt * kTile, bhk);
            }
            int issued = 0;
            int hq = bh_q0, it = i0;  // query head and query tile of walked tile t
            for (int t = 0; t < n_it; ++t, it = it + 1 < prm.n_tiles ? it + 1 : (++hq, i0)) {
                const int s = t % NS, u = t / NS;  // stage, its use count
                bool waited = true;
                if (u >= 1)
                    waited = mbar_wait(&bars[kKvBarEmpty + s], (u - 1) & 1, tmo, true);
                else if (C::kKvInTmem && s == NS - 1)  // K, V sit in the last stage until copied
                    waited = mbar_wait(&bars[kKvBarKVCopied], 0, tmo, true);
                if (!waited) {
                    record_timeout(prm.status, 20);
                    break;
                }
                uint8_t* q = smem + C::kQ + s * C::kTileBytes;
                uint8_t* g = smem + C::kG + s * C::kTileBytes;
                const int row = it * kTile;
                mbar_arrive_expect_tx(&bars[kKvBarFull + s], 2 * C::kTileBytes);
                for (int h = 0; h < D / 64; ++h) {
                    tma_load_3d(q + h * kHalf, &tmQ, &bars[kKvBarFull + s], h * 64, row, hq);
                    tma_load_3d(g + h * kHalf, &tmG, &bars[kKvBarFull + s], h * 64, row, hq);
                }
                ++issued;
            }
            // Whatever happened elsewhere, the copies this thread started land before exit.
            const uint64_t drain = tmo > kDrainNs ? tmo : kDrainNs;
            mbar_wait(&bars[kKvBarKV], 0, drain, true);
            if (issued > 0)
                mbar_wait(&bars[kKvBarFull + (issued - 1) % NS], ((issued - 1) / NS) & 1, drain,
                          true);
        }
    } else if (warp == kMmaWarp) {
        if ((kWarpIssue || lane == 0) && n_it > 0) {  // a converged warp, or lane 0
            auto iwait = [&](uint64_t* bar, uint32_t parity) {
                return issuer_wait<kWarpIssue>(bar, parity, tmo);
            };
            // ---- tensor-core products -------------------------------------------------------
            // Order per query tile t (buffer b = t % 2): dP^T once S^T is read, S^T of tile
            // t + 1 into the other buffer (once tile t - 1's dV, dK are done with it), then
            // dV, dK of each query half once its P^T, dS^T are written.  (A scheduler that
            // issued whichever product was ready, testing the barriers without blocking, ran
            // slower: its polling took issue slots from the element-wise warps.)
            constexpr uint32_t idS = idesc_bf16_f32_ab(kTile, kTile, 0, 0);
            constexpr uint32_t idT = idesc_bf16_f32_ab(kTile, D, 0, 1);
            const uint32_t tK = tmem + C::kTmemK, tV = tmem + C::kTmemV;
            const uint32_t sK = smem_u32(smem + C::kK), sV = smem_u32(smem + C::kV);
            bool ok = iwait(&bars[kKvBarKV], 0);
            int where = 21;
            if (ok && C::kKvInTmem) {
                tc_fence_after();
                const uint32_t sKs = smem_u32(smem + C::kKLoad), sVs = smem_u32(smem + C::kVLoad);
#pragma unroll
                for (int kk = 0; kk < D / 16; ++kk) {
                    const uint32_t off = (kk >> 2) * kHalf + (kk & 3) * 32;
                    issue_tmem_cp<kWarpIssue>(tK + kk * 8, smem_desc_sw128(sKs + off, 16, 1024));
                    issue_tmem_cp<kWarpIssue>(tV + kk * 8, smem_desc_sw128(sVs + off, 16, 1024));
                }
                issue_commit<kWarpIssue>(&bars[kKvBarKVCopied]);
            }
            if (ok) ok = iwait(&bars[kKvBarFull], 0);
            if (ok) {
                tc_fence_after();
                const uint32_t sQ0 = smem_u32(smem + C::kQ);
                if constexpr (C::kKvInTmem)
                    mma_ts_kmajor<D>(tmem + C::kTmemBuf, tK, sQ0, idS);
                else
                    mma_ss_kmajor<D>(tmem + C::kTmemBuf, sK, sQ0, idS);
                issue_commit<kWarpIssue>(&bars[kKvBarSFull]);
            }
            for (int t = 0; ok && t < n_it; ++t) {
                const int b = t & 1, s = t % NS, s1 = (t + 1) % NS;
                const uint32_t buf = tmem + C::kTmemBuf + b * 128;
                const uint32_t sQ = smem_u32(smem + C::kQ + s * C::kTileBytes);
                const uint32_t sG = smem_u32(smem + C::kG + s * C::kTileBytes);
                where = 22;
                if (!(ok = iwait(&bars[kKvBarRead], t & 1))) break;
                tc_fence_after();
                if constexpr (C::kKvInTmem)
                    mma_ts_kmajor<D>(buf, tV, sG, idS);
                else
                    mma_ss_kmajor<D>(buf, sV, sG, idS);
                issue_commit<kWarpIssue>(&bars[kKvBarDpFull]);
                if (t + 1 < n_it) {
                    where = 24;
                    if (!(ok = iwait(&bars[kKvBarFull + s1], ((t + 1) / NS) & 1))) break;
                    where = 25;
                    if (t >= 1 && !(ok = iwait(&bars[kKvBarSFree + (b ^ 1)], ((t - 1) >> 1) & 1)))
                        break;
                    tc_fence_after();
                    const uint32_t nbuf = tmem + C::kTmemBuf + (b ^ 1) * 128;
                    const uint32_t sQ1 = smem_u32(smem + C::kQ + s1 * C::kTileBytes);
                    if constexpr (C::kKvInTmem)
                        mma_ts_kmajor<D>(nbuf, tK, sQ1, idS);
                    else
                        mma_ss_kmajor<D>(nbuf, sK, sQ1, idS);
                    issue_commit<kWarpIssue>(&bars[kKvBarSFull + (b ^ 1)]);
                }
#pragma unroll
                for (int h = 0; h < 2; ++h) {
                    where = 26 + h;
                    if (!(ok = iwait(&bars[kKvBarPds + h], t & 1))) break;
                    tc_fence_after();
                    const uint32_t acc = (t > 0 || h > 0) ? 1u : 0u;
                    mma_ts_half(tmem + C::kTmemDV, buf, sG, h, idT, acc);
                    mma_ts_half(tmem + C::kTmemDK, buf + 8, sQ, h, idT, acc);
                }
                if (!ok) break;
                issue_commit<kWarpIssue>(&bars[kKvBarSFree + b]);
                issue_commit<kWarpIssue>(&bars[kKvBarEmpty + s]);
            }
            if (ok) {
                issue_commit<kWarpIssue>(&bars[kKvBarAcc]);
            } else {
                record_timeout(prm.status, where);
                // The products already issued finish before TMEM is freed.
                issue_commit<kWarpIssue>(&bars[kKvBarDrain]);
                issuer_wait<kWarpIssue>(&bars[kKvBarDrain], 0, tmo > kDrainNs ? tmo : kDrainNs,
                                        true);
            }
        }
    } else {
        // ---- P^T and dS^T (warps 0-15) ------------------------------------------------------
        const int q4 = warp & 3, sub = warp >> 2;
        const int r = q4 * 32 + lane;  // key row within the tile = TMEM lane
        const int key = jt * kTile + r;
        const uint32_t t_row = tmem + (static_cast<uint32_t>(q4 * 32) << 16);
        float* ld_s = reinterpret_cast<float*>(smem + C::kLD);
        const float4* ld4 = reinterpret_cast<const float4*>(smem + C::kLD);
        // Thread st (0..255) stages one value per query tile: -LSE log2e of column st (st < 128)
        // or -D of column st - 128; a column past N gets -inf and 0 (its shares are 0).
        const int st = warp * 32 + lane;
        const bool stager = st < 256;
        const int col = st & 127;
        const int slot = (col >> 1) * 4 + (col & 1) + (st >= 128 ? 2 : 0);
        // Walked tiles run over query tiles i0 .. n_tiles - 1 of query head bh_q0, then of the
        // next query head of the group, and so on.
        auto stage_value = [&](int hq, int it) -> float {
            const int q = it * kTile + col;
            if (q >= N) return st < 128 ? -INFINITY : 0.f;
            const size_t row = static_cast<size_t>(hq) * N + q;
            return st < 128 ? -prm.LSE[row] * kLog2e : -prm.Dv[row];
        };
        // Key rows at or past the sequence's length (or past N: a ragged last key tile) and, on
        // the diagonal tile of a causal mask, the queries before the key are masked: first
        // allowed column of this row.
        const bool ragged_keys = (jt + 1) * kTile > len;
        const int lo_row = key < len ? 0 : kTile;
        if (stager && n_it > 0) ld_s[slot] = stage_value(bh_q0, i0);
        named_bar_sync(1, kSoftWarps * 32);
        bool ok = true;
        int hq = bh_q0, it = i0;  // query head and query tile of walked tile t
        for (int t = 0; t < n_it; ++t, it = it + 1 < prm.n_tiles ? it + 1 : (++hq, i0)) {
            const int b = t & 1;
            const bool wrap = it + 1 == prm.n_tiles;
            const uint32_t t_buf = t_row + C::kTmemBuf + b * 128;
            const float next = stager && t + 1 < n_it
                                   ? stage_value(wrap ? hq + 1 : hq, wrap ? i0 : it + 1)
                                   : 0.f;
            bool good = mbar_wait(&bars[kKvBarSFull + b], (t >> 1) & 1, tmo);
            if (good) {
                tc_fence_after();
                const bool diag = CAUSAL && it == jt;
                const int lo = diag ? (key < len ? r : kTile) : lo_row;
                float p[2][16];
                // shares of both query halves (this warp's 16 columns of each); the S^T
                // columns are then handed over to dP^T
#pragma unroll
                for (int h = 0; h < 2; ++h) {
                    const int c0 = h * 64 + sub * 16;
                    if (diag || ragged_keys)
                        kv_shares<true>(t_buf, ld4, c0, lo, prm.scale_log2, p[h]);
                    else
                        kv_shares<false>(t_buf, ld4, c0, 0, prm.scale_log2, p[h]);
                }
                tc_fence_before();
                __syncwarp();
                if (lane == 0) mbar_arrive(&bars[kKvBarRead]);
                good = mbar_wait(&bars[kKvBarDpFull], t & 1, tmo);
                if (good) {
                    tc_fence_after();
#pragma unroll
                    for (int h = 0; h < 2; ++h) {
                        kv_grads(t_buf, ld4, h * 64 + sub * 16, p[h]);
                        tc_fence_before();
                        __syncwarp();
                        if (lane == 0) mbar_arrive(&bars[kKvBarPds + h]);
                    }
                }
            }
            if (!good && lane == 0) record_timeout(prm.status, 28);
            // All element-wise warps agree before the staged values are replaced.
            if (!named_bar_and(1, kSoftWarps * 32, good)) {
                ok = false;
                break;
            }
            if (stager) ld_s[slot] = next;
            named_bar_sync(1, kSoftWarps * 32);
        }
        if (ok) {
            // ---- dV (warps 0-7) and scale * dK (warps 8-15), half of the columns per warp ----
            const bool is_v = sub < 2;
            const int c0 = (sub & 1) * (D / 2);
            const uint32_t src = t_row + (is_v ? C::kTmemDV : C::kTmemDK) + c0;
            __nv_bfloat16* out = (is_v ? prm.dV : prm.dK) +
                                 (static_cast<size_t>(bhk) * N + (key < N ? key : 0)) * D + c0;
            const float sc = is_v ? 1.f : prm.scale;
            if (n_it == 0) {
                // no key of the tile below the length: its gradients are 0
                uint32_t v[32];
#pragma unroll
                for (int e = 0; e < 32; ++e) v[e] = 0u;
#pragma unroll
                for (int c = 0; c < D / 64; ++c)
                    if (key < N) store_row<32>(out + c * 32, v, 1.f);
            } else if (!mbar_wait(&bars[kKvBarAcc], 0, tmo)) {
                if (lane == 0) record_timeout(prm.status, 29);
            } else {
                tc_fence_after();
                // The TMEM loads are warp-wide (.sync.aligned): every lane issues them, and
                // only the stores are limited to the keys that exist.
#pragma unroll
                for (int c = 0; c < D / 64; ++c) {
                    uint32_t v[32];
                    tmem_ld32_sync(src + c * 32, v);
                    if (key < N) store_row<32>(out + c * 32, v, sc);
                }
            }
        }
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    if (warp == kMmaWarp) tmem_dealloc(tmem, 512);
}

// ============================================================================================
// dQ: one CTA per (head, query tile)
// ============================================================================================
// TMEM (512 columns): S [0,128) and [128,256) (two buffers, queries x keys), whose 16-column
// groups, once read by the warp that owns them, take dS of the same 16 keys in their first 8
// columns (bf16 pairs); dP [256,384); dQ [384, 384 + d).
//   S   = Q K_j^T      A = Q, B = K_j       shared memory, K-major
//   dP  = dO V_j^T     A = dO, B = V_j      shared memory, K-major
//   dQ += dS K_j       A = dS in TMEM, B = K_j MN-major
// K_j is read by the first and the last product of a key tile, V_j only by dP: K gets three
// ring stages and V two, each released as soon as its last reader is done, so that the load of
// a tile has about a tile's time to land.
template <int D>
struct QCfg {
    static constexpr int kTileBytes = (D / 64) * kHalf;
    static constexpr int kKStages = 3, kVStages = 2;
    static constexpr int kQ = 0;
    static constexpr int kG = kQ + kTileBytes;                // dO
    static constexpr int kK = kG + kTileBytes;                // kKStages stages
    static constexpr int kV = kK + kKStages * kTileBytes;     // kVStages stages
    static constexpr int kBar = kV + kVStages * kTileBytes;
    static constexpr int kBytes = kBar + 256;
    static constexpr int kDynSmem = dyn_smem(kBytes);
    static constexpr uint32_t kTmemS = 0, kTmemDP = 256, kTmemDQ = 384;
    static_assert(kTmemDQ + D <= 512, "TMEM budget");
    static_assert(kDynSmem <= 227 * 1024, "shared memory budget");
};

enum QBar {
    kQBarQG = 0,       // Q, dO landed
    kQBarKFull = 1,    // [3] K_j landed in a stage
    kQBarKEmpty = 4,   // [3] the products reading a K stage are done
    kQBarVFull = 7,    // [2] V_j landed in a stage
    kQBarVEmpty = 9,   // [2] dP has read a V stage
    kQBarSFull = 11,   // [2] S in TMEM buffer b
    kQBarSFree = 13,   // [2] dQ products done with the dS in buffer b
    kQBarDpFull = 15,  // dP in TMEM
    kQBarP0 = 16,      // dS of keys 0-63 written (one arrival per element-wise warp)
    kQBarP1 = 17,      // ... of keys 64-127 (and all of S, dP read)
    kQBarAcc = 18,     // the last dQ products done
    kQBarDrain = 19,
    kQNumBars = 20
};

// dS of 16 keys (part `part` of the 32-key chunk c) of the current key tile for this thread's
// query row, written over the first 8 of the same 16 S columns (bf16 pairs).
// nlse2 = -LSE log2e and nD = -D of the row; `hi`: last allowed key column of this row (127
// unless the tile needs masking).
template <bool MASK>
__device__ __forceinline__ void q_part(uint32_t t_s, uint32_t t_dp, int c, int part, float nlse2,
                                       float nD, int hi, float scale_log2) {
    const int c0 = c * 32 + part * 16;  // first key column
    uint32_t sv[16], gv[16];
    tmem_ld16x2_sync(t_s + c0, t_dp + c0, sv, gv);
    uint32_t dw[8];
    const float2 sl2 = make_float2(scale_log2, scale_log2);
    const float2 nl = make_float2(nlse2, nlse2), nd = make_float2(nD, nD);
#pragma unroll
    for (int e = 0; e < 8; ++e) {
        const float2 a = ffma2(make_float2(__uint_as_float(sv[2 * e]), __uint_as_float(sv[2 * e + 1])),
                               sl2, nl);
        float p0 = ex2_approx(a.x), p1 = ex2_approx(a.y);
        if (MASK) {
            const int col = c0 + 2 * e;
            p0 = col <= hi ? p0 : 0.f;
            p1 = col + 1 <= hi ? p1 : 0.f;
        }
        const float2 g = fadd2(make_float2(__uint_as_float(gv[2 * e]), __uint_as_float(gv[2 * e + 1])), nd);
        const float2 ds = fmul2(make_float2(p0, p1), g);
        dw[e] = pack_bf16x2(ds.x, ds.y);
    }
    tmem_st8_sync(t_s + c0, dw);
}

template <int D, bool CAUSAL>
__global__ void __launch_bounds__(kThreads, 1)
    bwd_q_kernel(const __grid_constant__ CUtensorMap tmQ, const __grid_constant__ CUtensorMap tmK,
                 const __grid_constant__ CUtensorMap tmV, const __grid_constant__ CUtensorMap tmG,
                 const BwdParams prm) {
    using C = QCfg<D>;
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
    uint64_t* bars = reinterpret_cast<uint64_t*>(smem + C::kBar);
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(bars + kQNumBars);
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    // The last query tile sees the most key tiles under a causal mask: it starts first.  bh:
    // the query head; bhk: the key/value head it reads.  Only key tiles holding a key below the
    // sequence's length are walked; with none, dQ is 0.
    int bh, pos;
    grid_place(prm.BH, prm.head_group_q, prm.n_tiles, bh, pos);
    const int qt = prm.n_tiles - 1 - pos;
    const int N = prm.N;
    const int b_seq = bh / prm.H;
    const int bhk = b_seq * prm.H_kv + (bh - b_seq * prm.H) / (prm.H / prm.H_kv);
    const int len = seq_keys(prm, b_seq);
    const int n_j = min(CAUSAL ? qt + 1 : prm.n_tiles, (len + kTile - 1) / kTile);
    const unsigned long long tmo = prm.timeout_ns;

    if (threadIdx.x == 0) {
        mbar_init(&bars[kQBarQG], 1);
        for (int s = 0; s < C::kKStages; ++s) {
            mbar_init(&bars[kQBarKFull + s], 1);
            mbar_init(&bars[kQBarKEmpty + s], 1);
        }
        for (int s = 0; s < 2; ++s) {
            mbar_init(&bars[kQBarVFull + s], 1);
            mbar_init(&bars[kQBarVEmpty + s], 1);
            mbar_init(&bars[kQBarSFull + s], 1);
            mbar_init(&bars[kQBarSFree + s], 1);
        }
        mbar_init(&bars[kQBarDpFull], 1);
        mbar_init(&bars[kQBarP0], kSoftWarps);
        mbar_init(&bars[kQBarP1], kSoftWarps);
        mbar_init(&bars[kQBarAcc], 1);
        mbar_init(&bars[kQBarDrain], 1);
        fence_mbar_init();
    }
    if (warp == kMmaWarp) {
        tmem_alloc(tmem_slot, 512);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tmem_slot;

    if (warp == kTmaWarp) {
        if (lane == 0 && n_j > 0) {
            // ---- loads ----------------------------------------------------------------------
            mbar_arrive_expect_tx(&bars[kQBarQG], 2 * C::kTileBytes);
            for (int h = 0; h < D / 64; ++h) {
                tma_load_3d(smem + C::kQ + h * kHalf, &tmQ, &bars[kQBarQG], h * 64, qt * kTile,
                            bh);
                tma_load_3d(smem + C::kG + h * kHalf, &tmG, &bars[kQBarQG], h * 64, qt * kTile,
                            bh);
            }
            int k_issued = 0, v_issued = 0;
            for (int j = 0; j < n_j; ++j) {
                const int ks = j % C::kKStages, ku = j / C::kKStages;  // stage, its use count
                if (ku >= 1 && !mbar_wait(&bars[kQBarKEmpty + ks], (ku - 1) & 1, tmo, true)) {
                    record_timeout(prm.status, 30);
                    break;
                }
                uint8_t* k = smem + C::kK + ks * C::kTileBytes;
                mbar_arrive_expect_tx(&bars[kQBarKFull + ks], C::kTileBytes);
                for (int h = 0; h < D / 64; ++h)
                    tma_load_3d(k + h * kHalf, &tmK, &bars[kQBarKFull + ks], h * 64, j * kTile,
                                bhk);
                ++k_issued;
                const int vs = j & 1;
                if (j >= 2 && !mbar_wait(&bars[kQBarVEmpty + vs], ((j >> 1) - 1) & 1, tmo, true)) {
                    record_timeout(prm.status, 30);
                    break;
                }
                uint8_t* v = smem + C::kV + vs * C::kTileBytes;
                mbar_arrive_expect_tx(&bars[kQBarVFull + vs], C::kTileBytes);
                for (int h = 0; h < D / 64; ++h)
                    tma_load_3d(v + h * kHalf, &tmV, &bars[kQBarVFull + vs], h * 64, j * kTile,
                                bhk);
                ++v_issued;
            }
            const uint64_t drain = tmo > kDrainNs ? tmo : kDrainNs;
            mbar_wait(&bars[kQBarQG], 0, drain, true);
            if (k_issued > 0) {
                const int j = k_issued - 1;
                mbar_wait(&bars[kQBarKFull + j % C::kKStages], (j / C::kKStages) & 1, drain, true);
            }
            if (v_issued > 0) {
                const int j = v_issued - 1;
                mbar_wait(&bars[kQBarVFull + (j & 1)], (j >> 1) & 1, drain, true);
            }
        }
    } else if (warp == kMmaWarp) {
        if ((kWarpIssue || lane == 0) && n_j > 0) {  // a converged warp, or lane 0
            auto iwait = [&](uint64_t* bar, uint32_t parity) {
                return issuer_wait<kWarpIssue>(bar, parity, tmo);
            };
            // ---- tensor-core products -------------------------------------------------------
            // Order per key tile j: S of tile j + 1 into the other buffer (while the
            // element-wise warps work on tile j), dQ of the first half of tile j's keys, of the
            // second half, then dP of tile j + 1 (its columns were read with the hand-over).
            const uint32_t sQ = smem_u32(smem + C::kQ), sG = smem_u32(smem + C::kG);
            constexpr uint32_t idS = idesc_bf16_f32_ab(kTile, kTile, 0, 0);
            constexpr uint32_t idT = idesc_bf16_f32_ab(kTile, D, 0, 1);
            int where = 31;
            bool ok = iwait(&bars[kQBarQG], 0) && iwait(&bars[kQBarKFull], 0) &&
                      iwait(&bars[kQBarVFull], 0);
            if (ok) {
                tc_fence_after();
                mma_ss_kmajor<D>(tmem + C::kTmemS, sQ, smem_u32(smem + C::kK), idS);
                issue_commit<kWarpIssue>(&bars[kQBarSFull]);
                mma_ss_kmajor<D>(tmem + C::kTmemDP, sG, smem_u32(smem + C::kV), idS);
                issue_commit<kWarpIssue>(&bars[kQBarDpFull]);
                issue_commit<kWarpIssue>(&bars[kQBarVEmpty]);
            }
            for (int j = 0; ok && j < n_j; ++j) {
                const int s = j & 1, s1 = (j + 1) & 1;
                const int ks = j % C::kKStages, ks1 = (j + 1) % C::kKStages;
                if (j + 1 < n_j) {
                    where = 32;
                    if (!(ok = iwait(&bars[kQBarKFull + ks1], ((j + 1) / C::kKStages) & 1)))
                        break;
                    where = 33;
                    if (j >= 1 && !(ok = iwait(&bars[kQBarSFree + s1], ((j - 1) >> 1) & 1)))
                        break;
                    tc_fence_after();
                    mma_ss_kmajor<D>(tmem + C::kTmemS + s1 * 128, sQ,
                                     smem_u32(smem + C::kK + ks1 * C::kTileBytes), idS);
                    issue_commit<kWarpIssue>(&bars[kQBarSFull + s1]);
                }
                const uint32_t sKj = smem_u32(smem + C::kK + ks * C::kTileBytes);
#pragma unroll
                for (int half = 0; half < 2; ++half) {
                    where = 34 + half;
                    if (!(ok = iwait(&bars[kQBarP0 + half], j & 1))) break;
                    tc_fence_after();
                    mma_ts_half(tmem + C::kTmemDQ, tmem + C::kTmemS + s * 128, sKj, half, idT,
                                (j > 0 || half > 0) ? 1u : 0u);
                }
                if (!ok) break;
                issue_commit<kWarpIssue>(&bars[kQBarSFree + s]);
                issue_commit<kWarpIssue>(&bars[kQBarKEmpty + ks]);
                if (j + 1 < n_j) {
                    where = 36;
                    if (!(ok = iwait(&bars[kQBarVFull + s1], ((j + 1) >> 1) & 1))) break;
                    tc_fence_after();
                    mma_ss_kmajor<D>(tmem + C::kTmemDP, sG,
                                     smem_u32(smem + C::kV + s1 * C::kTileBytes), idS);
                    issue_commit<kWarpIssue>(&bars[kQBarDpFull]);
                    issue_commit<kWarpIssue>(&bars[kQBarVEmpty + s1]);
                }
            }
            if (ok) {
                issue_commit<kWarpIssue>(&bars[kQBarAcc]);
            } else {
                record_timeout(prm.status, where);
                issue_commit<kWarpIssue>(&bars[kQBarDrain]);
                issuer_wait<kWarpIssue>(&bars[kQBarDrain], 0, tmo > kDrainNs ? tmo : kDrainNs,
                                        true);
            }
        }
    } else {
        // ---- dS (warps 0-15) -----------------------------------------------------------------
        const int q4 = warp & 3, sub = warp >> 2;
        const int r = q4 * 32 + lane;  // query row within the tile = TMEM lane
        const int q = qt * kTile + r;
        const uint32_t t_row = tmem + (static_cast<uint32_t>(q4 * 32) << 16);
        // A row past N has shares 0 (-LSE log2e = -inf) and is never written.
        const size_t row = static_cast<size_t>(bh) * N + (q < N ? q : 0);
        const float nlse2 = q < N ? -prm.LSE[row] * kLog2e : -INFINITY;
        const float nD = q < N ? -prm.Dv[row] : 0.f;
        bool ok = true;
        for (int j = 0; j < n_j; ++j) {
            const int s = j & 1;
            bool good = mbar_wait(&bars[kQBarSFull + s], (j >> 1) & 1, tmo) &&
                        mbar_wait(&bars[kQBarDpFull], j & 1, tmo);
            if (!good) {
                if (lane == 0) record_timeout(prm.status, 37);
                ok = false;
                break;
            }
            tc_fence_after();
            // Masks: keys after the query on the diagonal tile of a causal mask, and keys at or
            // past the sequence's length (or past N: the ragged last key tile): last allowed
            // key column of this row.
            const bool diag = CAUSAL && j == qt;
            const bool ragged_keys = (j + 1) * kTile > len;
            int hi = kTile - 1;
            if (diag) hi = r;
            if (ragged_keys && len - 1 - j * kTile < hi) hi = len - 1 - j * kTile;
            const uint32_t t_s = t_row + C::kTmemS + s * 128, t_dp = t_row + C::kTmemDP;
#pragma unroll 1
            for (int k = 0; k < 2; ++k) {
                const int c = 2 * k + (sub >> 1);  // keys 0-63 first, then 64-127
                if (diag || ragged_keys)
                    q_part<true>(t_s, t_dp, c, sub & 1, nlse2, nD, hi, prm.scale_log2);
                else
                    q_part<false>(t_s, t_dp, c, sub & 1, nlse2, nD, kTile - 1, prm.scale_log2);
                tc_fence_before();
                __syncwarp();
                if (lane == 0) mbar_arrive(&bars[kQBarP0 + k]);
            }
        }
        if (ok) {
            // ---- scale * dQ of this query tile (a quarter of the columns per warp) ------------
            constexpr int kZCols = D / 4;
            if (n_j == 0) {
                // no key below the length: dQ is 0
                uint32_t v[kZCols];
#pragma unroll
                for (int e = 0; e < kZCols; ++e) v[e] = 0u;
                if (q < N) store_row<kZCols>(prm.dQ + row * D + sub * kZCols, v, 1.f);
            } else if (!mbar_wait(&bars[kQBarAcc], 0, tmo)) {
                if (lane == 0) record_timeout(prm.status, 38);
            } else {
                tc_fence_after();
                constexpr int kCols = D / 4;
                const uint32_t src = t_row + C::kTmemDQ + sub * kCols;
                __nv_bfloat16* out = prm.dQ + row * D + sub * kCols;
                uint32_t v[kCols];
                if constexpr (kCols == 32) {
                    tmem_ld32_sync(src, v);
                } else {
                    tmem_ld16_sync(src, v);
                }
                if (q < N) store_row<kCols>(out, v, prm.scale);
            }
        }
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    if (warp == kMmaWarp) tmem_dealloc(tmem, 512);
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
int launch_tiles(const CUtensorMap& tq, const CUtensorMap& tk, const CUtensorMap& tv,
                 const CUtensorMap& tg, const BwdParams& prm, cudaStream_t stream) {
    static std::once_flag once;
    static cudaError_t attr = cudaSuccess;
    std::call_once(once, [] {
        attr = cudaFuncSetAttribute(bwd_kv_kernel<D, CAUSAL>,
                                    cudaFuncAttributeMaxDynamicSharedMemorySize,
                                    KvCfg<D>::kDynSmem);
        if (attr == cudaSuccess)
            attr = cudaFuncSetAttribute(bwd_q_kernel<D, CAUSAL>,
                                        cudaFuncAttributeMaxDynamicSharedMemorySize,
                                        QCfg<D>::kDynSmem);
    });
    if (attr != cudaSuccess) return FA_ERR_CUDA;
    const long long kv_ctas = static_cast<long long>(prm.BH_kv) * prm.n_tiles;
    const long long q_ctas = static_cast<long long>(prm.BH) * prm.n_tiles;
    if (q_ctas > 0x7fffffffLL) return FA_ERR_UNSUPPORTED;
    bwd_kv_kernel<D, CAUSAL>
        <<<static_cast<unsigned>(kv_ctas), kThreads, KvCfg<D>::kDynSmem, stream>>>(tq, tk, tv, tg,
                                                                                  prm);
    if (cudaGetLastError() != cudaSuccess) return FA_ERR_CUDA;
    bwd_q_kernel<D, CAUSAL><<<static_cast<unsigned>(q_ctas), kThreads, QCfg<D>::kDynSmem, stream>>>(
        tq, tk, tv, tg, prm);
    return cudaGetLastError() == cudaSuccess ? FA_OK : FA_ERR_CUDA;
}

}  // namespace

int fa_bwd_launch(const void* Q, const void* K, const void* V, const void* O, const void* dO,
                  const float* LSE, void* dQ, void* dK, void* dV, float* ws_D, int64_t B,
                  int64_t H, int64_t H_kv, int64_t N, int64_t d, const int32_t* kv_lens,
                  float scale, bool causal, cudaStream_t stream) {
    const int64_t BH = B * H, BH_kv = B * H_kv;
    if (N > (1LL << 30) || BH > (1LL << 30) || H_kv < 1 || H % H_kv != 0)
        return FA_ERR_UNSUPPORTED;
    const long long rows = BH * N;
    const long long sms = bwd_sm_count() > 0 ? bwd_sm_count() : 148;
    long long grid = (rows + 7) / 8;
    if (grid > sms * 16) grid = sms * 16;
    if (d == 64)
        bwd_prep_kernel<64><<<static_cast<unsigned>(grid), 256, 0, stream>>>(
            static_cast<const __nv_bfloat16*>(O), static_cast<const __nv_bfloat16*>(dO), ws_D,
            rows);
    else
        bwd_prep_kernel<128><<<static_cast<unsigned>(grid), 256, 0, stream>>>(
            static_cast<const __nv_bfloat16*>(O), static_cast<const __nv_bfloat16*>(dO), ws_D,
            rows);
    if (cudaGetLastError() != cudaSuccess) return FA_ERR_CUDA;

    CUtensorMap tq, tk, tv, tg;
    int st = make_bhnd_tensor_map(&tq, Q, BH, N, d);
    if (st == FA_OK) st = make_bhnd_tensor_map(&tk, K, BH_kv, N, d);
    if (st == FA_OK) st = make_bhnd_tensor_map(&tv, V, BH_kv, N, d);
    if (st == FA_OK) st = make_bhnd_tensor_map(&tg, dO, BH, N, d);
    if (st != FA_OK) return st;
    BwdParams prm{};
    prm.LSE = LSE;
    prm.Dv = ws_D;
    prm.dQ = static_cast<__nv_bfloat16*>(dQ);
    prm.dK = static_cast<__nv_bfloat16*>(dK);
    prm.dV = static_cast<__nv_bfloat16*>(dV);
    prm.N = static_cast<int>(N);
    prm.n_tiles = static_cast<int>((N + kTile - 1) / kTile);
    prm.H = static_cast<int>(H);
    prm.H_kv = static_cast<int>(H_kv);
    prm.BH = static_cast<int>(BH);
    prm.BH_kv = static_cast<int>(BH_kv);
    prm.kv_lens = kv_lens;
    // Heads per group of each grid.  If the tiles that the heads' CTAs walk (two bf16 [N, d]
    // tensors per head: Q and dO of a key/value head's query heads for dK, dV; K and V, shared
    // by the query heads of a group, for dQ) fit in 64 MB, half of L2, one group.  Otherwise,
    // with a causal mask, groups that fit (inside a group the longest tiles start first, which
    // keeps the tail short); without one, a head (a key/value head's query heads for dQ) at a
    // time (measured fastest: the CTAs in flight share two or three heads).
    const long long share = H / H_kv, budget = 64LL << 20;
    auto head_group = [&](long long heads, long long head_bytes, long long one_at_a_time) {
        long long g = heads;
        if (head_bytes * heads > budget) g = causal ? budget / head_bytes : one_at_a_time;
        return static_cast<int>(g < 1 ? 1 : (g > heads ? heads : g));
    };
    prm.head_group_kv = head_group(BH_kv, 4LL * N * d * share, 1);
    prm.head_group_q = head_group(BH, (4LL * N * d + share - 1) / share, share);
    prm.scale = scale;
    prm.scale_log2 = scale * kLog2e;
    prm.timeout_ns = fa_wait_timeout_ns();
    prm.status = device_status_word();
    if (!prm.status) return FA_ERR_CUDA;
    if (d == 64)
        return causal ? launch_tiles<64, true>(tq, tk, tv, tg, prm, stream)
                      : launch_tiles<64, false>(tq, tk, tv, tg, prm, stream);
    return causal ? launch_tiles<128, true>(tq, tk, tv, tg, prm, stream)
                  : launch_tiles<128, false>(tq, tk, tv, tg, prm, stream);
}

}  // namespace osm
