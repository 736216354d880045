// fa_fwd.cu -- exact attention forward, tile by tile with the online softmax, for sm_103a.
//
// The method: "How FlashAttention avoids storing the giant score table" (spicyshark.co,
// Online softmax lesson), section "From softmax to attention" (per key block: scores, new
// running max, alpha = exp(m - m_new), p = exp(s - m_new), l = l*alpha + sum p,
// acc = acc*alpha + p V, divide by l after the last block), "The implementation" (a block that
// leaves the max at -inf adds nothing) and the two-worker merge at the end of "From softmax to
// attention"; "kbwen.com FlashAttention", sections "Two blocks" and "More than two blocks"
// (query blocks in the outer loop, key blocks inside, each query row with its own max, sum
// and partial output).  The shift used inside the exponentials may be any common constant per
// row ("The fix: subtract the maximum": the factor cancels), which allows the lazy rescale.
//
// GB300 mapping.  A persistent CTA per SM works through a list of work items, each a 128-row
// query tile of one (b, h) against a range of its key tiles (128 keys each); the pipelines run
// on from one item into the next.  Both products run on the tensor cores:
//   S = Q K^T   d = 128: A = Q in TMEM (tcgen05.cp from shared memory); d = 64: A = Q in
//               shared memory; B = K tile (shared memory, K-major)
//   O += P V    A = P (TMEM), B = V tile (shared memory, MN-major)
// TMEM (512 columns): S0 [0,128), S1 [128,256), then kP P buffers of 64 columns, kOAcc O
// accumulators of d columns and kQ Q buffers of d/2 columns: d = 128 one of each (512
// columns), d = 64 two P buffers and two O accumulators (one per softmax group) and no Q.
// bf16 operands hold two values per 32-bit column.  S of key tile J goes to S(J & 1), P of
// tile J to P(J % kP).
//   warps 0-3, 4-7  two softmax warpgroups that take the key tiles in turn (group g the tiles
//                   J with J & 1 == g), one query row per thread (its TMEM lane), whole rows:
//                   tcgen05.ld of the 128 scores, mask, row max, lazy reference max, ex2 of
//                   the scaled and shifted scores (scale*log2(e) folded into one FFMA), the
//                   group's own running sum, P rounded to bf16 into a P buffer.  While one
//                   group computes the exponentials of tile J the other already works on tile
//                   J+1.  d = 128: the groups share one O accumulator; the row's reference max
//                   is handed on from the previous tile through shared memory (a producer /
//                   consumer named barrier, the only link between the groups), and when it
//                   moves (rare: only beyond 2^8) the group scales O in TMEM by alpha before
//                   its P V.  d = 64: each group keeps its own reference max and O
//                   accumulator, and the epilogue merges the two.  At the end of an item each
//                   group leaves its (m, l) for the epilogue.
//   warps 8, 9      tcgen05.mma: warp 8 (d = 128: after copying each item's Q into TMEM)
//                   issues S(J+2) as soon as S(J) has been read (two tiles ahead of the
//                   softmax), warp 9 issues O += P(J) V(J) as soon as P(J) is stored.  One
//                   thread cannot issue M128 N128 K16 MMAs much faster than the tensor core
//                   runs them, so two independent issuers keep it fed; at d = 128 each runs
//                   as a converged warp with one elected lane issuing.  fp32 accumulators.
//   warps 10, 11    TMA: the K ring (warp 10: d = 128 each item's Q tile, then its K tiles;
//                   d = 64 the K tiles, and Q into two shared-memory buffers of its own) and
//                   the V ring (warp 11); 128-byte swizzle, zero fill past the end of the
//                   sequence.
//                   With an explicit mask the V producer also brings each tile's mask bits
//                   (16 bytes for each of the 128 query rows) and the tile's index into the V
//                   slot, where the softmax reads them after the slot's barrier.
//   warps 12-15     epilogue: the two groups' (m, l) combined with the two-worker merge, O read
//                   from TMEM once the item's last P V is done (the next item's first P V
//                   waits for that read), O / l to bf16 into a 16 KB staging buffer in shared
//                   memory, 64 columns at a time, each half written out by one TMA store; and
//                   LSE = (m + log2 l) * ln 2.
// Causal: key tiles above the diagonal are never visited; only diagonal and ragged tiles are
// masked element by element.  With an explicit mask's tile map, key tiles holding no allowed
// key for the query tile are not visited either.
//
// Every mbarrier wait is bounded (%globaltimer deadline).  A wait that gives up records
// FA_ERR_TIMEOUT in a device status word; the CTA then drains its own TMA loads and MMAs,
// frees its TMEM and exits.  The named barriers between the softmax groups are passed the same
// number of times by every thread also after a timeout, so they cannot hang.
#include <cuda_runtime.h>

#include <cmath>
#include <mutex>
#include <type_traits>

#include "osm_internal.h"
#include "ptx_sm103.cuh"

namespace osm {

__device__ int g_fa_device_status = 0;

namespace {

constexpr int kBM = 128;        // query rows per tile: one TMEM lane per row
constexpr int kBN = 128;        // keys per key/value tile
constexpr int kThreads = 512;   // 16 warps, see the role table above
constexpr int kMmaWarp = 8;     // issues S = Q K^T (and owns the TMEM allocation)
constexpr int kMmaPvWarp = 9;   // issues O += P V
constexpr int kTmaWarp = 10;    // Q and K loads
constexpr int kTmaVWarp = 11;   // V loads
constexpr int kEpiWarp0 = 12;   // warps 12-15: epilogue
constexpr uint32_t kTmemCols = 512;
constexpr int kHalfBytes = 128 * 128;         // one 64-column half of a 128-row bf16 tile
constexpr uint64_t kDrainNs = 1000000000ull;  // drain waits: at least 1 s
constexpr float kRescaleThreshold = 8.0f;     // log2 units
// When the reference max moves, it moves to the tile's max plus this headroom (log2 units), so
// that a row whose max keeps climbing (large logits) moves it rarely: only once the max has
// climbed by the headroom plus the threshold.  Every share stays <= 2^threshold as before; the
// shares of the row max start at 2^-headroom, far above the bottom of the fp32 / bf16 range.
constexpr float kRescaleHeadroom = 24.0f;
constexpr uint32_t kBarHandOff = 1;  // named barriers 1, 2: reference max of tile J -> J+1
constexpr uint32_t kBarTeardown = 3; // named barrier 3: TMEM no longer used (warps 0-9, 12-15)
constexpr uint32_t kTeardownThreads = 448;
constexpr uint32_t kBarEpi = 4;      // named barrier 4: the epilogue's four warps
constexpr int kMaxStages = 8;
constexpr int kFinSlots = 4;         // final (m, l) of the last items, see fin_full

// Counters.  A CTA works through its work items (query tile, head, key range) in order and
// numbers everything it streams across items: the key tiles J (S buffer J & 1, P buffer
// J % kP, V ring slot J % stages), the K-ring entries (each non-empty item's Q tile followed by
// its K tiles), the items it and the non-empty items qi (Q buffer qi % kQ).  Barrier phases
// follow from these counters, so the pipelines run on from one item into the next.
struct Bars {
    uint64_t k_full[kMaxStages], k_empty[kMaxStages];  // K ring (Q tiles and K tiles)
    uint64_t v_full[kMaxStages], v_empty[kMaxStages];  // V ring
    uint64_t s_full[2];   // S buffer b holds S of a tile J with J & 1 == b (tcgen05.commit)
    uint64_t s_free[2];   // S buffer b read into registers by its group (4 warps)
    uint64_t p_full[2];   // P buffer b stored, O rescaled if needed (4 warps)
    // O += P(J) V finished (tcgen05.commit) -> pv_done[J & 3].  A parity wait tells a phase
    // from the one two completions later only if the waiter is never that far behind: every
    // wait on these is for a P V at most one tile older than one the waiter has already seen
    // complete and at least one tile older than any that can complete, so four barriers make
    // each wait exact (see pv_wait).
    uint64_t pv_done[4];
    uint64_t q_free[2];   // the last S of item qi has read Q buffer qi % kQ (tcgen05.commit)
    uint64_t q_full[2];   // d = 64: item qi's Q tile has landed in shared-memory buffer qi & 1
    uint64_t o_full;      // every P V of a non-empty item finished (tcgen05.commit)
    uint64_t o_free;      // O of a non-empty item read by the epilogue (4 warps)
    // Both softmax groups have written their final (m, l) of item k into fin[k % kFinSlots]
    // (8 warps); the epilogue has read them (4 warps) and the slot may take item k + kFinSlots.
    uint64_t fin_full[kFinSlots];
    uint64_t fin_free[kFinSlots];
    uint64_t mma_done;
    uint64_t mma_pv_done;
    uint32_t tmem_base;
    float mref[2][kBM];                // reference max of tile J for tile J+1: [J & 1][row]
    float fin[kFinSlots][2][2][kBM];   // [item slot][group][m, l][row]
    // MASK: the key tile in V ring slot s, written by the V producer before its arrival on
    // v_full[s] (ordered by that barrier for the softmax, which reads it after the wait).
    int v_kt[kMaxStages];
};

template <int D, bool M = false>  // M: the kernel reads an explicit mask
struct Cfg {
    // d = 64: the two softmax groups are independent workers.  Each keeps its own running max,
    // running sum and O accumulator over the key tiles it takes, and the epilogue combines the
    // two partial states with the two-worker merge; no reference max passes between them.
    // Two accumulators need 64 more TMEM columns, so the Q tile stays in shared memory and S
    // is an SS product.  (d = 128 has no room for a second accumulator.)
    static constexpr bool kIndep = D == 64;
    static constexpr int kHalves = D / 64;
    static constexpr int kTileBytes = kHalves * kHalfBytes;  // 128 rows x D bf16
    // K ring and V ring depth (d = 64 with a mask: 4, for the mask bits' slots)
    static constexpr int kStages = D == 128 ? 3 : (M ? 4 : 5);
    static constexpr int kK = 0;
    static constexpr int kV = kK + kStages * kTileBytes;
    static constexpr int kQs = kV + kStages * kTileBytes;     // kIndep: two Q tile buffers
    static constexpr int kMsk = kQs + (kIndep ? 2 * kTileBytes : 0);  // MASK: mask bits
    static constexpr int kMskBytes = kBM * 16;              // 128 query rows x 16 bytes
    static constexpr int kBars = kMsk + (M ? kStages * kMskBytes : 0);
    // The epilogue's staging buffer: 64 columns of the O tile (128 rows x 128 bytes, the
    // 128-byte swizzle of the tensor map) on their way to a TMA store.
    static constexpr int kOst = (kBars + static_cast<int>(sizeof(Bars)) + 1023) & ~1023;
    static constexpr int kOstBytes = kHalfBytes;
    static constexpr int kBytes = kOst + kOstBytes;
    // Registers per thread after the role split: the softmax groups hold a row of 128 scores
    // (at d = 64 they need more than 200); the epilogue writes O into the staging buffer as it
    // reads it.  Measured at d = 128: 200 for the softmax and 72 for an epilogue that held
    // half a row while the first half's store drained was 1-3 % slower on the dense case.
    static constexpr int kSoftRegs = 208;
    static constexpr int kEpiRegs = 56;
    static_assert(2 * 128 * kSoftRegs + 128 * 40 + 128 * kEpiRegs <= 65536, "register split");
    static constexpr int kDynSmem = kBytes + 1024;  // slack for 1024-byte alignment
    // Waits that let the waiting thread sleep until the phase completes instead of polling:
    // polling takes issue slots from the warps sharing the SMSP.  And the MMA issuers either
    // run as whole, converged warps with one elected lane issuing (kWarpIssue), or as lane 0
    // alone.  Measured per head dimension on GB300: at d = 128 converged issue with sleeping
    // waits is 2-4 % faster; at d = 64 (SS products for S, bound by shared memory) lane-0
    // issue with polling waits is 4 % faster (sleeping issuer waits there: -1 to -2 %).  The
    // softmax's sleeping waits: causal d = 128 +1.4 %.
    static constexpr bool kWarpIssue = D == 128;
    static constexpr bool kSleepMma = D == 128;
    static constexpr bool kSleepSoftmax = true;
    static constexpr int kP = kIndep ? 2 : 1;       // P buffers (kIndep: one per group)
    static constexpr int kQ = kIndep ? 0 : 1;       // Q buffers in TMEM
    static constexpr int kOAcc = kIndep ? 2 : 1;    // O accumulators (kIndep: one per group)
    static constexpr uint32_t kTmemS = 0;           // S0, S1: 128 columns each
    static constexpr uint32_t kTmemP = 256;         // P buffers: 64 columns each
    static constexpr uint32_t kTmemO = kTmemP + 64 * kP;    // O accumulators: D columns each
    static constexpr uint32_t kTmemQ = kTmemO + kOAcc * D;  // Q buffers: D/2 columns each
    static_assert(kTmemQ + kQ * (D / 2) <= kTmemCols, "TMEM budget");
    static_assert(kDynSmem <= 227 * 1024, "shared memory budget");
    static_assert(kStages <= kMaxStages, "ring depth");
};

// All 32 lanes wait on the same phase; the outcome is made warp-uniform so that the
// .sync.aligned tcgen05 instructions that follow are never reached by a partial warp.
__device__ __forceinline__ bool warp_wait(uint64_t* bar, uint32_t parity, uint64_t timeout_ns,
                                          bool suspend = false) {
    const bool ok = mbar_wait(bar, parity, timeout_ns, suspend);
    return __all_sync(0xffffffffu, ok);
}

// One arrival per warp, after every lane's prior tcgen05 accesses are ordered before it.
__device__ __forceinline__ void warp_arrive_tc(uint64_t* bar) {
    tc_fence_before();
    __syncwarp();
    if ((threadIdx.x & 31) == 0) mbar_arrive(bar);
}

// Wait until O += P(k) V has finished.  Callers guarantee that P(k-4) V has finished and that
// P(k+4) V cannot have, so the parity of completion k >> 2 of barrier k & 3 is unambiguous.
__device__ __forceinline__ bool pv_wait(Bars* bars, int k, uint64_t timeout_ns,
                                        bool sleep = false) {
    return warp_wait(&bars->pv_done[k & 3], (k >> 2) & 1, timeout_ns, sleep);
}

__device__ __forceinline__ void record_timeout(int where) {
    atomicCAS(&g_fa_device_status, 0, FA_ERR_TIMEOUT | (where << 8));
}

__device__ __forceinline__ void named_bar_arrive(uint32_t id, uint32_t count) {
    asm volatile("bar.arrive %0, %1;" ::"r"(id), "r"(count) : "memory");
}

// Launch parameters.  The key range of one head is cut into n_splits contiguous ranges of
// tiles_per_split key tiles; with n_splits == 1 (SPLIT == false) a work item covers every key
// and writes the final O (bf16) and LSE, otherwise it writes its range's normalised partial
// output (fp32) and log-sum-exp to the workspace for the combine kernel.
struct FaKernelParams {
    __nv_bfloat16* O;  // [BH, Nq, D] bf16 (SPLIT == false)
    float* LSE;        // [BH, Nq] or nullptr (SPLIT == false)
    float* ws_O;       // [n_splits, BH, Nq, D] fp32 (SPLIT == true)
    float* ws_LSE;     // [n_splits, BH, Nq] (SPLIT == true)
    int Nq, Nk, BH, n_qtiles, n_splits, tiles_per_split, n_items;
    int head_group;  // causal: heads whose items are interleaved (their K, V share the L2)
    int H, H_kv;     // query heads and key/value heads per sequence (BH = sequences x H)
    // Query positions per original head.  Nq == q_pos, except when the query heads that share
    // a key/value head are packed into one row block (Nq = group x q_pos): row r of a block is
    // then position r % q_pos of query head r / q_pos.
    int q_pos;
    const int32_t* kv_lens;  // [BH / H] valid keys per sequence, or nullptr (all Nk valid)
    // Explicit mask (uint32 words, one bit per key, 1 = allowed), or nullptr: the row of query
    // head bh = b H + h, position i, starts at mask + b mask_bs + h mask_hs + i mask_words, and
    // each key tile's 128 bits are one 16-byte group of it.
    const uint32_t* mask;
    long long mask_bs, mask_hs;
    int mask_words;
    float scale_log2;
    unsigned long long timeout_ns;
};

// The host's launch state: the kernel's parameters, and the mask's tile map, which reaches the
// kernel (MASK == 2) with the mask's tensor map instead.
struct FaParams : FaKernelParams {
    // Optional tile map of the mask (MASK == 2), or nullptr: bit kt % 32 of word kt / 32 of
    // the row at tile_map + (inst * n_qtiles + q_tile) * tmap_words is 0 when no key of key
    // tile kt is allowed for any query of the query tile; such tiles are skipped.  inst is the
    // mask's instance: b and h of the query head where the mask strides are nonzero.
    const uint32_t* tile_map;
    int tmap_words;
};

// One work item: a 128-row query tile of query head bh (over all sequences) against key tiles
// [kt0, kt0 + n_kv) of key/value head kvh, which holds kv_len valid keys.
struct Item {
    int q_tile, bh, split, kt0, n_kv, kvh, kv_len;
    // MASK with a tile map that leaves some tile out: the item visits only the allowed tiles
    // of [kt0, kt_end), n_kv of them; tm is the query tile's row of the map, and tm_bits holds
    // the allowed tiles of its word tm_word not visited yet.  Otherwise (tm == nullptr) tiles
    // kt0 .. kt0 + n_kv - 1.
    const uint32_t* tm;
    int kt_end, tm_word;
    uint32_t tm_bits;
};

// Word wi of an item's tile-map row, without the tiles outside [kt0, kt_end).
__device__ __forceinline__ uint32_t map_word(const Item& w, int wi) {
    uint32_t bits = w.tm[wi];
    if (wi == (w.kt0 >> 5)) bits &= ~0u << (w.kt0 & 31);
    if (wi == ((w.kt_end - 1) >> 5) && (w.kt_end & 31)) bits &= ~(~0u << (w.kt_end & 31));
    return bits;
}

// Work item idx of the launch.  Non-causal items go head by head, so the CTAs running at one
// time share the K and V of a few heads.  Causal items go in groups of head_group heads (as
// many as keep their K and V in L2 together), and within a group the longest rows (highest
// query tiles) first, so that the CTAs' shares even out.
template <bool CAUSAL, bool TMAP = false>
__device__ __forceinline__ Item decode_item(int idx, const FaKernelParams& prm,
                                            const uint32_t* tile_map = nullptr,
                                            int tmap_words = 0) {
    Item w;
    if (CAUSAL) {
        const int per_head = prm.n_qtiles * prm.n_splits;
        const int group = idx / (prm.head_group * per_head);
        const int h0 = group * prm.head_group;
        const int hg = min(prm.head_group, prm.BH - h0);  // heads in this group
        const int r = idx - h0 * per_head;
        const int k = r / (hg * prm.n_splits);  // rank of the query tile, longest rows first
        const int packed = (prm.q_pos % kBM == 0 && prm.Nq % prm.q_pos == 0)
                               ? prm.Nq / prm.q_pos : 1;  // query heads per row block
        if (packed > 1) {
            // packed query heads: the tiles at the same position of the block's heads in turn
            const int per = prm.q_pos / kBM;  // tiles per query head
            w.q_tile = (k % packed) * per + (per - 1 - k / packed);
        } else {
            w.q_tile = prm.n_qtiles - 1 - k;
        }
        w.bh = h0 + (r % (hg * prm.n_splits)) / prm.n_splits;
        w.split = r % prm.n_splits;
    } else {
        w.split = idx % prm.n_splits;
        w.q_tile = (idx / prm.n_splits) % prm.n_qtiles;
        w.bh = idx / (prm.n_splits * prm.n_qtiles);
    }
    // Grouped heads: query head h of sequence b reads key/value head h / (H / H_kv) of it.
    const int b = w.bh / prm.H;
    w.kvh = b * prm.H_kv + (w.bh - b * prm.H) / (prm.H / prm.H_kv);
    w.kv_len = prm.Nk;
    if (prm.kv_lens != nullptr) w.kv_len = min(max(prm.kv_lens[b], 0), prm.Nk);
    // Causal: the queries are the last Nq of the Nk positions, so query row q sees keys
    // j <= q + Nk - Nq; key tiles wholly past the query tile's last row, or past the
    // sequence's own keys, are skipped.
    const int n_kv_all = (w.kv_len + kBN - 1) / kBN;
    w.kt0 = w.split * prm.tiles_per_split;
    int kt1 = min(n_kv_all, w.kt0 + prm.tiles_per_split);
    if (CAUSAL) {
        // the largest query position among the tile's rows
        const int r0 = w.q_tile * kBM, r1 = min(r0 + kBM, prm.Nq) - 1;
        const int pos_max = (r0 / prm.q_pos != r1 / prm.q_pos) ? prm.q_pos - 1 : r1 % prm.q_pos;
        const long long last_key = static_cast<long long>(pos_max) + (prm.Nk - prm.q_pos);
        kt1 = min(static_cast<long long>(kt1), last_key < 0 ? 0 : last_key / kBN + 1);
    }
    w.n_kv = max(0, kt1 - w.kt0);
    w.tm = nullptr;
    if (TMAP) {
        w.kt_end = w.kt0 + w.n_kv;
        w.tm_word = -1;
        w.tm_bits = 0u;
    }
    if (TMAP && tile_map != nullptr && w.n_kv > 0) {
        const int b = w.bh / prm.H, h = w.bh - (w.bh / prm.H) * prm.H;
        const int inst = (prm.mask_bs != 0 ? b : 0) * (prm.mask_hs != 0 ? prm.H : 1) +
                         (prm.mask_hs != 0 ? h : 0);
        w.tm = tile_map + (static_cast<long long>(inst) * prm.n_qtiles + w.q_tile) * tmap_words;
        int n = 0;
        for (int wi = w.kt0 >> 5; wi <= (w.kt_end - 1) >> 5; ++wi) {
            const uint32_t bits = map_word(w, wi);
            if (wi == (w.kt0 >> 5)) {
                w.tm_word = wi;
                w.tm_bits = bits;
            }
            n += __popc(bits);
        }
        if (n == w.n_kv) w.tm = nullptr;  // every tile allowed: visit them in a row
        w.n_kv = n;
    }
    return w;
}

// The key tiles an item visits, in order: next() hands out the next one.  With a tile map
// (tm != nullptr) the allowed tiles are taken one by one from the word in hand, and the map is
// read again only when that word is used up (kt_end means none is left; callers visit exactly
// n_kv tiles); otherwise the tiles follow one another from kt0.
struct TileCursor {
    const uint32_t* tm;
    int kt, kt_end, word;  // kt: the tile handed out last
    uint32_t bits;         // allowed tiles of word `word` not handed out yet

    __device__ __forceinline__ explicit TileCursor(const Item& w)
        : tm(w.tm), kt(w.kt0 - 1), kt_end(w.kt_end), word(w.tm_word), bits(w.tm_bits) {}

    __device__ __forceinline__ int next() {
        if (tm == nullptr) return ++kt;
        while (bits == 0u) {
            if (++word > ((kt_end - 1) >> 5)) return kt = kt_end;
            bits = tm[word];  // a word past the first: only the end of the range cuts it
            if (word == ((kt_end - 1) >> 5) && (kt_end & 31)) bits &= ~(~0u << (kt_end & 31));
        }
        kt = (word << 5) + __ffs(bits) - 1;
        bits &= bits - 1u;
        return kt;
    }
};

// This CTA's work items in order, then -1.  The items are dealt out group by group (causal:
// the head groups of decode_item, each with its longest rows first; otherwise one group of
// all items), in rounds of gridDim.x, alternately forwards and backwards: CTA c takes item c
// of a forward round and item gridDim.x - 1 - c of a backward one, so that the long items of
// one round and the short ones of the next even out.  Round r of group g runs forwards when
// r + g is even, so that a group's last, partial round starts where the previous group's
// left off.  (Counting each item as its key tiles plus three for its boundary, one sequence
// over all groups, whose partial rounds fall on the same CTAs, leaves the busiest CTA of the
// causal B2 H32 N8192 launch 3.1 % above the mean, and this order 0.4 %; measured, the launch
// ran 0.2-0.8 % faster.)
struct ItemSeq {
    int P, c, n_items, gsz;  // CTAs, this CTA, items, items per group
    int k = 0;               // items handed out so far (one group: all of them)
    int g = 0, g0 = 0;       // group and its first item
    int r = 0, cnt = 0;      // next round of the group, this CTA's items in the group
    __device__ __forceinline__ ItemSeq(int n, int group_items)
        : P(static_cast<int>(gridDim.x)), c(static_cast<int>(blockIdx.x)), n_items(n),
          gsz(group_items > 0 && group_items < n ? group_items : n) {
        if (gsz < n_items) start_group();
    }
    __device__ __forceinline__ void start_group() {
        const int G = min(gsz, n_items - g0);
        const int R = G / P, m = G - R * P;
        cnt = R;
        if (m > 0 && (((R + g) & 1) == 0 ? c < m : c >= P - m)) ++cnt;
        r = 0;
    }
    __device__ __forceinline__ int next() {
        if (gsz >= n_items) {  // one group: round k, forwards when k is even
            const int idx = k * P + ((k & 1) ? P - 1 - c : c);
            ++k;
            return idx < n_items ? idx : -1;
        }
        while (g0 < n_items && r >= cnt) {
            g0 += gsz;
            ++g;
            if (g0 < n_items) start_group();
        }
        if (g0 >= n_items) return -1;
        const int p = (((r + g) & 1) == 0) ? c : P - 1 - c;
        const int idx = g0 + r * P + p;
        ++r;
        return idx;
    }
};

// Items per group of ItemSeq: causal launches interleave the items of head_group heads.
template <bool CAUSAL>
__device__ __forceinline__ int item_group(const FaKernelParams& prm) {
    return CAUSAL ? prm.head_group * prm.n_qtiles * prm.n_splits : prm.n_items;
}

// Waits until every phase a producer thread started on a ring has completed: the last entry
// put into each slot is the last phase of that slot's barrier, so each of these waits ends.
__device__ __forceinline__ void drain_ring(uint64_t* full, int stages, int issued,
                                           uint64_t timeout_ns) {
    const uint64_t drain_ns = timeout_ns > kDrainNs ? timeout_ns : kDrainNs;
    for (int s = 0; s < stages && s < issued; ++s) {
        const int last = s + ((issued - 1 - s) / stages) * stages;
        mbar_wait(&full[s], (last / stages) & 1, drain_ns);
    }
}

// The mask's tensor map and tile map, a kernel parameter only where a mask is read.
struct MaskArgs {
    CUtensorMap map;
    const uint32_t* tile_map;  // MASK == 2: the tile map (FaParams::tile_map)
    int tmap_words;
};
struct NoMaskMap {};
template <int MASK>
using MaskMap = typename std::conditional<(MASK != 0), MaskArgs, NoMaskMap>::type;

template <int MASK>
__device__ __forceinline__ const uint32_t* tile_map_of(const MaskMap<MASK>& m) {
    if constexpr (MASK == 2) return m.tile_map;
    else return nullptr;
}
template <int MASK>
__device__ __forceinline__ int tmap_words_of(const MaskMap<MASK>& m) {
    if constexpr (MASK == 2) return m.tmap_words;
    else return 0;
}

// MASK: 1 = an explicit mask is read (prm.mask), 2 = the same with the mask's tile map
// (prm.tile_map); separate instantiations, so that the unmasked kernels' code is unchanged.
template <int D, bool CAUSAL, bool SPLIT, int MASK = 0>
__global__ void __launch_bounds__(kThreads, 1)
    fa_fwd_kernel(const __grid_constant__ CUtensorMap tmQ, const __grid_constant__ CUtensorMap tmK,
                  const __grid_constant__ CUtensorMap tmV, const __grid_constant__ MaskMap<MASK> tmM,
                  const __grid_constant__ CUtensorMap tmO, const FaKernelParams prm) {
    using C = Cfg<D, (MASK != 0)>;
    constexpr int S_ = C::kStages;
    const int Nq = prm.Nq, Nk = prm.Nk;
    const unsigned long long timeout_ns = prm.timeout_ns;
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
    Bars* bars = reinterpret_cast<Bars*>(smem + C::kBars);
    const uint32_t sK = smem_u32(smem + C::kK);
    const uint32_t sV = smem_u32(smem + C::kV);
    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;

    if (threadIdx.x == 0) {
        for (int s = 0; s < S_; ++s) {
            mbar_init(&bars->k_full[s], 1);
            mbar_init(&bars->k_empty[s], 1);
            mbar_init(&bars->v_full[s], 1);
            mbar_init(&bars->v_empty[s], 1);
        }
        for (int b = 0; b < 2; ++b) {
            mbar_init(&bars->s_full[b], 1);
            mbar_init(&bars->s_free[b], 4);
            mbar_init(&bars->p_full[b], 4);
            mbar_init(&bars->q_free[b], 1);
            mbar_init(&bars->q_full[b], 1);
        }
        for (int b = 0; b < 4; ++b) mbar_init(&bars->pv_done[b], 1);
        for (int b = 0; b < kFinSlots; ++b) {
            mbar_init(&bars->fin_full[b], 8);
            mbar_init(&bars->fin_free[b], 4);
        }
        mbar_init(&bars->o_full, 1);
        mbar_init(&bars->o_free, 4);
        mbar_init(&bars->mma_done, 1);
        mbar_init(&bars->mma_pv_done, 1);
        fence_mbar_init();
    }
    if (warp == kMmaWarp) {
        tmem_alloc(&bars->tmem_base, kTmemCols);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = bars->tmem_base;

    // Registers: a softmax thread holds a whole row of 128 scores, the other warps little:
    // 2 x 128 x kSoftRegs + 128 x 40 + 128 x kEpiRegs is the 512 x 128 launched.  Each role branch sets its
    // own limit and never rejoins the others; the TMEM is freed by warp 8 after a named
    // barrier that the softmax groups, warp 9 and the epilogue arrive at when done with it.
    if (warp >= kEpiWarp0) {
        setmaxnreg_dec<C::kEpiRegs>();
        // ------------------------------------------------------------------ epilogue
        // Per item: the two groups' (m, l) merged with the two-worker merge, O / l read from
        // TMEM once every P V of the item is done, then O (bf16, or the fp32 partial for the
        // split-key path) and LSE = (m + log2 l) * ln 2 written out; row r of the tile is TMEM
        // lane r, one per thread.  An item whose key range is empty (split-key ranges past the
        // diagonal or past Nk) never ran P V: it writes O = 0 and LSE = -inf.
        const int r = threadIdx.x & 127;
        const uint32_t tO = tmem + (static_cast<uint32_t>((warp & 3) * 32) << 16) + C::kTmemO;
        bool ok = true;
        int qi = 0;
        ItemSeq items0(prm.n_items, item_group<CAUSAL>(prm));
        for (int k = 0;; ++k) {
            const int idx = items0.next();
            if (idx < 0) break;
            const Item w = decode_item<CAUSAL, MASK == 2>(idx, prm, tile_map_of<MASK>(tmM), tmap_words_of<MASK>(tmM));
            const int slot = k % kFinSlots;
            const bool have = w.n_kv > 0;
            // The groups' (m, l) of the item, and O once its last P V is done.  The four warps
            // agree on the outcome of their waits before they go on, so that a wait given up
            // in one of them never leaves the others at the staging barrier.
            bool good = warp_wait(&bars->fin_full[slot], (k / kFinSlots) & 1, timeout_ns, true);
            if (!good) record_timeout(12);
            if (good && have) {
                good = warp_wait(&bars->o_full, qi & 1, timeout_ns, true);
                if (!good) record_timeout(13);
            }
            if (!named_bar_and(kBarEpi, 128, good)) {
                ok = false;
                break;
            }
            if (have) tc_fence_after();
            const float m0 = bars->fin[slot][0][0][r], l0 = bars->fin[slot][0][1][r];
            const float m1 = bars->fin[slot][1][0][r], l1 = bars->fin[slot][1][1][r];
            __syncwarp();
            if (lane == 0) mbar_arrive(&bars->fin_free[slot]);
            const float M = fmaxf(m0, m1);
            // The two groups' states relative to M.  A group with nothing (m = -inf: no tile
            // of the item, or no allowed key in its tiles) weighs 0.
            const float w0 = m0 == -INFINITY ? 0.f : ex2_approx(m0 - M);
            const float w1 = m1 == -INFINITY ? 0.f : ex2_approx(m1 - M);
            const float lt = l0 * w0 + l1 * w1;
            const int q_row = w.q_tile * kBM + r;
            const bool store = q_row < Nq;
            const float inv_l = lt > 0.f ? 1.f / lt : 0.f;
            const size_t row = static_cast<size_t>(w.bh) * Nq + q_row;
            const size_t ws_row = static_cast<size_t>(w.split) * prm.BH * Nq + row;
            if constexpr (SPLIT) {
                // fp32 partials, stored as they are read: 32 columns of the shared accumulator
                // per step, or 16 of each group's (d = 64), within the register budget; the
                // next item's first P V waits for the last step.
                constexpr int CW = C::kIndep ? 16 : 32;
#pragma unroll 1
                for (int c = 0; c < D / CW; ++c) {
                    float o[CW];
                    if (!have) {
#pragma unroll
                        for (int e = 0; e < CW; ++e) o[e] = 0.f;
                    } else if constexpr (C::kIndep) {
                        uint32_t a[16], b[16];
                        tmem_ld16x2_sync(tO + c * 16, tO + D + c * 16, a, b);
                        // A group that weighs 0 may hold another item's sums: never read.
#pragma unroll
                        for (int e = 0; e < 16; ++e)
                            o[e] = (w0 != 0.f ? __uint_as_float(a[e]) * w0 : 0.f) +
                                   (w1 != 0.f ? __uint_as_float(b[e]) * w1 : 0.f);
                    } else {
                        uint32_t a[32];
                        tmem_ld32_sync(tO + c * 32, a);
#pragma unroll
                        for (int e = 0; e < 32; ++e) o[e] = __uint_as_float(a[e]);
                    }
                    if (have && c == D / CW - 1) warp_arrive_tc(&bars->o_free);
                    if (!store) continue;
                    float4* dst = reinterpret_cast<float4*>(prm.ws_O + ws_row * D + c * CW);
#pragma unroll
                    for (int v = 0; v < CW / 4; ++v)
                        dst[v] = make_float4(o[4 * v] * inv_l, o[4 * v + 1] * inv_l,
                                             o[4 * v + 2] * inv_l, o[4 * v + 3] * inv_l);
                }
            } else {
                // O / l in bf16 through the staging buffer (128 rows x 64 columns, the
                // 128-byte swizzle of the tensor map), one TMA store of the 128 x 64 box per
                // half (rows past Nq are not written): one bulk store instead of a 16-byte
                // store per row and column group, which crowded the softmax's shared-memory
                // and TMEM traffic.  Each half goes into the buffer as it is read, once the
                // buffer's previous store has read it; after the last read the next item's
                // first P V may overwrite O.
                uint8_t* ost = smem + C::kOst;
                uint8_t* rowp = ost + r * 128;
                auto chunk = [&](int j) -> uint4* {  // 16-byte chunk j (columns 8j..8j+7)
                    return reinterpret_cast<uint4*>(rowp + ((j ^ (r & 7)) << 4));
                };
                if (threadIdx.x == kEpiWarp0 * 32) bulk_wait_group_read<0>();
                named_bar_sync(kBarEpi, 128);
                if constexpr (C::kIndep) {
                    // The two groups' accumulators, 8 columns of each per step.
#pragma unroll
                    for (int j = 0; j < 8; ++j) {
                        uint32_t q4[4] = {0u, 0u, 0u, 0u};  // bf16 +0 pairs
                        if (have) {
                            uint32_t a[8], b[8];
                            tmem_ld8x2_sync(tO + j * 8, tO + D + j * 8, a, b);
                            // A group that weighs 0 may hold another item's sums: never read.
#pragma unroll
                            for (int e = 0; e < 4; ++e) {
                                const float x0 =
                                    (w0 != 0.f ? __uint_as_float(a[2 * e]) * w0 : 0.f) +
                                    (w1 != 0.f ? __uint_as_float(b[2 * e]) * w1 : 0.f);
                                const float x1 =
                                    (w0 != 0.f ? __uint_as_float(a[2 * e + 1]) * w0 : 0.f) +
                                    (w1 != 0.f ? __uint_as_float(b[2 * e + 1]) * w1 : 0.f);
                                q4[e] = pack_bf16x2(x0 * inv_l, x1 * inv_l);
                            }
                        }
                        *chunk(j) = make_uint4(q4[0], q4[1], q4[2], q4[3]);
                    }
                    if (have) warp_arrive_tc(&bars->o_free);
                } else {
#pragma unroll
                    for (int c = 0; c < 4; ++c) {
                        uint32_t q8[8] = {0u, 0u, 0u, 0u, 0u, 0u, 0u, 0u};
                        if (have) {
                            uint32_t a[16];
                            tmem_ld16_sync(tO + c * 16, a);
#pragma unroll
                            for (int e = 0; e < 8; ++e)
                                q8[e] = pack_bf16x2(__uint_as_float(a[2 * e]) * inv_l,
                                                    __uint_as_float(a[2 * e + 1]) * inv_l);
                        }
                        *chunk(2 * c) = make_uint4(q8[0], q8[1], q8[2], q8[3]);
                        *chunk(2 * c + 1) = make_uint4(q8[4], q8[5], q8[6], q8[7]);
                    }
                }
                fence_proxy_async_smem();
                named_bar_sync(kBarEpi, 128);
                if (threadIdx.x == kEpiWarp0 * 32) {
                    tma_store_3d(&tmO, ost, 0, w.q_tile * kBM, w.bh);
                    bulk_commit_group();
                }
                if constexpr (C::kHalves == 2) {
                    // half 1 into the buffer once half 0's store has read it
                    if (threadIdx.x == kEpiWarp0 * 32) bulk_wait_group_read<0>();
                    named_bar_sync(kBarEpi, 128);
#pragma unroll
                    for (int c = 0; c < 4; ++c) {
                        uint32_t q8[8] = {0u, 0u, 0u, 0u, 0u, 0u, 0u, 0u};
                        if (have) {
                            uint32_t a[16];
                            tmem_ld16_sync(tO + 64 + c * 16, a);
#pragma unroll
                            for (int e = 0; e < 8; ++e)
                                q8[e] = pack_bf16x2(__uint_as_float(a[2 * e]) * inv_l,
                                                    __uint_as_float(a[2 * e + 1]) * inv_l);
                        }
                        *chunk(2 * c) = make_uint4(q8[0], q8[1], q8[2], q8[3]);
                        *chunk(2 * c + 1) = make_uint4(q8[4], q8[5], q8[6], q8[7]);
                    }
                    if (have) warp_arrive_tc(&bars->o_free);
                    fence_proxy_async_smem();
                    named_bar_sync(kBarEpi, 128);
                    if (threadIdx.x == kEpiWarp0 * 32) {
                        tma_store_3d(&tmO, ost, 64, w.q_tile * kBM, w.bh);
                        bulk_commit_group();
                    }
                }
            }
            if (store) {
                const float lse = have ? (M + __log2f(lt)) * 0.69314718055994531f : -INFINITY;
                if (SPLIT)
                    prm.ws_LSE[ws_row] = lse;
                else if (prm.LSE != nullptr)
                    prm.LSE[row] = lse;
            }
            qi += have ? 1 : 0;
        }
        (void)ok;
        // The TMA stores of O have read the staging buffer and written O before the CTA ends.
        if (!SPLIT && threadIdx.x == kEpiWarp0 * 32) bulk_wait_group<0>();
        tc_fence_before();
        named_bar_arrive(kBarTeardown, kTeardownThreads);
    } else if (warp >= kMmaWarp) {
        setmaxnreg_dec<40>();
        // The MMA issuers' waits (see Cfg::kWarpIssue and Cfg::kSleepMma).
        auto iwait = [&](uint64_t* bar, uint32_t parity) {
            return issuer_wait<C::kWarpIssue>(bar, parity, timeout_ns, C::kSleepMma);
        };
        constexpr bool W = C::kWarpIssue;
        if (warp == kTmaWarp) {
            // ------------------------------------------------------ TMA: Q and K tiles, K ring
            if (lane == 0) {
                tma_prefetch_desc(&tmQ);
                tma_prefetch_desc(&tmK);
                tma_prefetch_desc(&tmV);
                if constexpr (MASK != 0) tma_prefetch_desc(&tmM.map);
                constexpr uint32_t kTx = C::kTileBytes;
                if constexpr (C::kIndep) {
                    // Each non-empty item's Q tile into shared-memory buffer qi & 1, once the
                    // last S of item qi - 2 has read that buffer; its K tiles into the K ring.
                    int e = 0, qi = 0;
                    bool ok = true;
                    ItemSeq items1(prm.n_items, item_group<CAUSAL>(prm));
                    for (int k = 0; ok; ++k) {
                        const int idx = items1.next();
                        if (idx < 0) break;
                        const Item w = decode_item<CAUSAL, MASK == 2>(idx, prm, tile_map_of<MASK>(tmM), tmap_words_of<MASK>(tmM));
                        if (w.n_kv == 0) continue;
                        const int qb = qi & 1;
                        if (qi >= 2 && !mbar_wait(&bars->q_free[qb], ((qi >> 1) - 1) & 1,
                                                  timeout_ns, true)) {
                            record_timeout(1);
                            break;
                        }
                        mbar_arrive_expect_tx(&bars->q_full[qb], kTx);
                        tma_load_3d(smem + C::kQs + qb * C::kTileBytes, &tmQ, &bars->q_full[qb], 0,
                                    w.q_tile * kBM, w.bh);
                        ++qi;
                        TileCursor tiles(w);
                        for (int t = 0; t < w.n_kv; ++t, ++e) {
                            const int kt = tiles.next();
                            const int s = e % S_;
                            if (e >= S_ && !mbar_wait(&bars->k_empty[s], ((e / S_) - 1) & 1,
                                                      timeout_ns, true)) {
                                record_timeout(1);
                                ok = false;
                                break;
                            }
                            mbar_arrive_expect_tx(&bars->k_full[s], kTx);
                            tma_load_3d(smem + C::kK + s * C::kTileBytes, &tmK, &bars->k_full[s],
                                        0, kt * kBN, w.kvh);
                        }
                    }
                    drain_ring(bars->k_full, S_, e, timeout_ns);
                    drain_ring(bars->q_full, 2, qi, timeout_ns);
                } else {
                    int e = 0;  // K-ring entries issued
                    bool ok = true;
                    ItemSeq items2(prm.n_items, item_group<CAUSAL>(prm));
                    for (int k = 0; ok; ++k) {
                        const int idx = items2.next();
                        if (idx < 0) break;
                        const Item w = decode_item<CAUSAL, MASK == 2>(idx, prm, tile_map_of<MASK>(tmM), tmap_words_of<MASK>(tmM));
                        // t = -1: the item's Q tile, then its key tiles (key tile kt).
                        TileCursor tiles(w);
                        int kt = tiles.next();
                        for (int t = w.n_kv > 0 ? -1 : 0; t < w.n_kv; ++t, ++e) {
                            const int s = e % S_;
                            if (e >= S_ && !mbar_wait(&bars->k_empty[s], ((e / S_) - 1) & 1,
                                                      timeout_ns, true)) {
                                record_timeout(1);
                                ok = false;
                                break;
                            }
                            mbar_arrive_expect_tx(&bars->k_full[s], kTx);
                            const CUtensorMap* map = t < 0 ? &tmQ : &tmK;
                            const int row =
                                t < 0 ? w.q_tile * kBM : (MASK == 2 ? kt : w.kt0 + t) * kBN;
                            const int head = t < 0 ? w.bh : w.kvh;
                            for (int h = 0; h < C::kHalves; ++h)
                                tma_load_3d(smem + C::kK + s * C::kTileBytes + h * kHalfBytes, map,
                                            &bars->k_full[s], h * 64, row, head);
                            if (t >= 0) kt = MASK == 2 ? tiles.next() : kt + 1;
                        }
                    }
                    drain_ring(bars->k_full, S_, e, timeout_ns);
                }
            }
        } else if (warp == kTmaVWarp) {
            // ------------------------------------------------------ TMA: V tiles, V ring
            if (lane == 0) {
                constexpr uint32_t kTx = C::kTileBytes;
                int J = 0;  // V tiles issued
                bool ok = true;
                ItemSeq items3(prm.n_items, item_group<CAUSAL>(prm));
                for (int k = 0; ok; ++k) {
                    const int idx = items3.next();
                    if (idx < 0) break;
                    const Item w = decode_item<CAUSAL, MASK == 2>(idx, prm, tile_map_of<MASK>(tmM), tmap_words_of<MASK>(tmM));
                    TileCursor tiles(w);
                    int kt = MASK == 2 ? tiles.next() : w.kt0;
                    for (int t = 0; t < w.n_kv;
                         ++t, ++J, kt = MASK == 2 ? tiles.next() : kt + 1) {
                        const int s = J % S_;
                        if (J >= S_ &&
                            !mbar_wait(&bars->v_empty[s], ((J / S_) - 1) & 1, timeout_ns, true)) {
                            record_timeout(2);
                            ok = false;
                            break;
                        }
                        if (MASK) bars->v_kt[s] = kt;
                        mbar_arrive_expect_tx(&bars->v_full[s],
                                              MASK ? kTx + C::kMskBytes : kTx);
                        for (int h = 0; h < C::kHalves; ++h)
                            tma_load_3d(smem + C::kV + s * C::kTileBytes + h * kHalfBytes, &tmV,
                                        &bars->v_full[s], h * 64,
                                        (MASK == 2 ? kt : w.kt0 + t) * kBN, w.kvh);
                        if constexpr (MASK != 0) {
                            // The tile's mask bits for the 128 query rows ride with V: the
                            // slot is freed only after P V, when the softmax has used them.
                            const int b = w.bh / prm.H, h = w.bh - b * prm.H;
                            tma_load_4d(smem + C::kMsk + s * C::kMskBytes, &tmM.map,
                                        &bars->v_full[s], 4 * kt, w.q_tile * kBM,
                                        prm.mask_hs != 0 ? h : 0, prm.mask_bs != 0 ? b : 0);
                        }
                    }
                }
                drain_ring(bars->v_full, S_, J, timeout_ns);
            }
        } else if (warp == kMmaWarp) {
            // ------------------------------------------------------ MMA: S = Q K^T
            if (C::kWarpIssue || lane == 0) {  // a converged warp, or lane 0
                constexpr uint32_t idS = idesc_bf16_f32(kBM, kBN, 0);
                if constexpr (C::kIndep) {
                    // SS products: A = the item's Q tile in shared-memory buffer qi & 1, B = the
                    // K tile, both K-major and 128-byte swizzled; four K16 steps (d = 64).
                    int e = 0, J = 0, qi = 0;
                    bool ok = true;
                    ItemSeq items4(prm.n_items, item_group<CAUSAL>(prm));
                    for (int k = 0; ok; ++k) {
                        const int idx = items4.next();
                        if (idx < 0) break;
                        const Item w = decode_item<CAUSAL, MASK == 2>(idx, prm, tile_map_of<MASK>(tmM), tmap_words_of<MASK>(tmM));
                        if (w.n_kv == 0) continue;
                        const int qb = qi & 1;
                        if (!iwait(&bars->q_full[qb], (qi >> 1) & 1)) {
                            record_timeout(3);
                            break;
                        }
                        const uint64_t qdesc =
                            smem_desc_sw128(smem_u32(smem + C::kQs + qb * C::kTileBytes), 16, 1024);
                        for (int t = 0; t < w.n_kv; ++t, ++J, ++e) {
                            // S(J) overwrites S(J-2): its group must have read it.
                            const int s = e % S_;
                            const int b = J & 1;
                            if ((J >= 2 && !iwait(&bars->s_free[b], ((J >> 1) - 1) & 1)) ||
                                !iwait(&bars->k_full[s], (e / S_) & 1)) {
                                record_timeout(5);
                                ok = false;
                                break;
                            }
                            tc_fence_after();
                            issue_ss_x4<W>(tmem + C::kTmemS + b * 128, qdesc,
                                           smem_desc_sw128(sK + s * C::kTileBytes, 16, 1024),
                                           idS, 0u);
                            issue_commit<W>(&bars->s_full[b]);
                            issue_commit<W>(&bars->k_empty[s]);
                        }
                        if (ok) issue_commit<W>(&bars->q_free[qb]);
                        ++qi;
                    }
                } else {
                    int e = 0, J = 0, qi = 0;
                    bool ok = true;
                    ItemSeq items5(prm.n_items, item_group<CAUSAL>(prm));
                    for (int k = 0; ok; ++k) {
                        const int idx = items5.next();
                        if (idx < 0) break;
                        const Item w = decode_item<CAUSAL, MASK == 2>(idx, prm, tile_map_of<MASK>(tmM), tmap_words_of<MASK>(tmM));
                        if (w.n_kv == 0) continue;
                        // The item's Q tile: K ring -> Q buffer qb in TMEM (tcgen05.cp, ordered
                        // before the MMAs below), once the S of item qi - kQ, the buffer's
                        // previous reader, has finished.
                        const int qb = qi % C::kQ;
                        const uint32_t tQ = tmem + C::kTmemQ + qb * (D / 2);
                        int s = e % S_;
                        if ((qi >= C::kQ &&
                             !iwait(&bars->q_free[qb], ((qi - C::kQ) / C::kQ) & 1)) ||
                            !iwait(&bars->k_full[s], (e / S_) & 1)) {
                            record_timeout(3);
                            ok = false;
                            break;
                        }
                        tc_fence_after();
                        {
                            const uint32_t qs = sK + s * C::kTileBytes;
#pragma unroll
                            for (int kk = 0; kk < D / 16; ++kk)
                                issue_tmem_cp<W>(tQ + kk * 8,
                                                 smem_desc_sw128(qs + (kk >> 2) * kHalfBytes +
                                                                     (kk & 3) * 32,
                                                                 16, 1024));
                        }
                        issue_commit<W>(&bars->k_empty[s]);
                        ++e;
                        for (int t = 0; t < w.n_kv; ++t, ++J, ++e) {
                            // S(J) overwrites S(J-2): its group must have read it.
                            s = e % S_;
                            const int b = J & 1;
                            if ((J >= 2 && !iwait(&bars->s_free[b], ((J >> 1) - 1) & 1)) ||
                                !iwait(&bars->k_full[s], (e / S_) & 1)) {
                                record_timeout(5);
                                ok = false;
                                break;
                            }
                            tc_fence_after();
                            // B_k: the K tile's 16-element slice k (32 bytes apart within each
                            // 64-column half of the K-major, 128-byte swizzled tile).
                            const uint32_t kb = sK + s * C::kTileBytes;
#pragma unroll
                            for (int h = 0; h < C::kHalves; ++h)
                                issue_ts_x4<W>(tmem + C::kTmemS + b * 128, tQ + h * 32,
                                               smem_desc_sw128(kb + h * kHalfBytes, 16, 1024),
                                               32 / 16, idS, h > 0 ? 1u : 0u);
                            issue_commit<W>(&bars->s_full[b]);
                            issue_commit<W>(&bars->k_empty[s]);
                        }
                        if (ok) issue_commit<W>(&bars->q_free[qb]);
                        ++qi;
                    }
                }
                // Drain: no MMA of this thread may still write TMEM when it is freed.
                issue_commit<W>(&bars->mma_done);
                issuer_wait<W>(&bars->mma_done, 0,
                                           timeout_ns > kDrainNs ? timeout_ns : kDrainNs, false);
            }
            __syncwarp();
            named_bar_sync(kBarTeardown, kTeardownThreads);
            tc_fence_after();
            tmem_dealloc(tmem, kTmemCols);
        } else if (warp == kMmaPvWarp) {
            // ------------------------------------------------------ MMA: O += P V
            if (C::kWarpIssue || lane == 0) {  // a converged warp, or lane 0
                constexpr uint32_t idO = idesc_bf16_f32(kBM, D, 1);
                int J = 0, qi = 0;
                int vs = 0, vph = 0;  // V ring slot of tile J and its phase
                int pb = 0, pph = 0;  // P buffer of tile J and its phase
                bool ok = true;
                ItemSeq items6(prm.n_items, item_group<CAUSAL>(prm));
                for (int k = 0; ok; ++k) {
                    const int idx = items6.next();
                    if (idx < 0) break;
                    const Item w = decode_item<CAUSAL, MASK == 2>(idx, prm, tile_map_of<MASK>(tmM), tmap_words_of<MASK>(tmM));
                    if (w.n_kv == 0) continue;
                    // The first P V of an item overwrites O: the epilogue must have read the
                    // previous item's.
                    if (qi >= 1 &&
                        !iwait(&bars->o_free, (qi - 1) & 1)) {
                        record_timeout(11);
                        ok = false;
                        break;
                    }
                    for (int t = 0; t < w.n_kv; ++t, ++J) {
                        // P is what the tile usually waits for; V has landed long before.
                        if (!iwait(&bars->p_full[pb], pph) ||
                            !iwait(&bars->v_full[vs], vph)) {
                            record_timeout(6);
                            ok = false;
                            break;
                        }
                        tc_fence_after();
                        // B_k: rows 16k..16k+15 of the V tile (MN-major), 2048 bytes apart.
                        // With one accumulator per group (d = 64), tile J goes into the
                        // accumulator of group J & 1, and each group's first tile of the item
                        // (t = 0 or 1) overwrites it.
                        const uint32_t acc_o = C::kIndep ? C::kTmemO + (J & 1) * D : C::kTmemO;
                        const bool first = C::kIndep ? t < 2 : t == 0;
                        issue_ts_x8<W>(tmem + acc_o, tmem + C::kTmemP + pb * 64,
                                       smem_desc_sw128(sV + vs * C::kTileBytes, kHalfBytes, 1024),
                                       2048 / 16, idO, first ? 0u : 1u);
                        issue_commit<W>(&bars->pv_done[J & 3]);
                        issue_commit<W>(&bars->v_empty[vs]);
                        if (++vs == S_) { vs = 0; vph ^= 1; }
                        if (++pb == C::kP) { pb = 0; pph ^= 1; }
                    }
                    // every P V of the item, for the epilogue
                    if (ok) issue_commit<W>(&bars->o_full);
                    ++qi;
                }
                issue_commit<W>(&bars->mma_pv_done);
                issuer_wait<W>(&bars->mma_pv_done, 0,
                                           timeout_ns > kDrainNs ? timeout_ns : kDrainNs, false);
            }
            __syncwarp();
            tc_fence_before();
            named_bar_arrive(kBarTeardown, kTeardownThreads);
        }
    } else {
        setmaxnreg_inc<C::kSoftRegs>();
        // -------------------------------------------------------------------- softmax
        const int g = warp >> 2;          // this group takes the key tiles J with J & 1 == g
        const int r = threadIdx.x & 127;  // row in the tile == TMEM lane
        const uint32_t lane_addr = static_cast<uint32_t>((warp & 3) * 32) << 16;
        const uint32_t tS = tmem + lane_addr + C::kTmemS + g * 128;
        // This group's O accumulator (d = 64: one per group; d = 128: the shared one).
        const uint32_t tO = tmem + lane_addr + C::kTmemO + (C::kIndep ? g * D : 0);
        const float scale_log2 = prm.scale_log2;
        // Key tiles of this CTA over all its items: the hand-off of the reference max runs
        // through all of them (a tile that starts an item ignores what it receives), so that
        // every tile J >= 1 passes its consumer barrier and the groups stay in step.
        int J_total = 0;
        ItemSeq items7(prm.n_items, item_group<CAUSAL>(prm));
        for (int k = 0;; ++k) {
            const int idx = items7.next();
            if (idx < 0) break;
            J_total += decode_item<CAUSAL, MASK == 2>(idx, prm, tile_map_of<MASK>(tmM), tmap_words_of<MASK>(tmM)).n_kv;
        }
        bool ok = true;
        int J0 = 0;  // first key tile of the item
        ItemSeq items8(prm.n_items, item_group<CAUSAL>(prm));
        for (int k = 0;; ++k) {
            const int idx = items8.next();
            if (idx < 0) break;
            int n, kt0, key_limit;
            {
                const Item w = decode_item<CAUSAL, MASK == 2>(idx, prm, tile_map_of<MASK>(tmM), tmap_words_of<MASK>(tmM));
                n = w.n_kv;
                kt0 = w.kt0;
                const int q_row = w.q_tile * kBM + r;
                const int pos = q_row % prm.q_pos;  // position of the row's query
                key_limit = CAUSAL ? min(w.kv_len - 1, pos + (Nk - prm.q_pos)) : w.kv_len - 1;
            }
            float m_last = -INFINITY;  // reference max this group used last (scaled, log2)
            float l = 0.f;             // this group's sum of 2^(t - m_last) over its tiles
            // Hand-off barrier passes of this group, in order: for each of its tiles J, a
            // consumer pass (bar.sync) when J >= 1 and a producer pass (bar.arrive) when
            // J + 1 < J_total.  A group that stops early because a wait gave up makes up the
            // missing passes after the loop.
            int J = J0 + ((J0 & 1) != g ? 1 : 0);
            int stage = 0;  // 0: before tile J's consumer pass, 1: before its producer pass
            for (; ok && J < J0 + n; J += 2, stage = 0) {
                const int t = J - J0;  // tile within the item
                if (!warp_wait(&bars->s_full[g], (J >> 1) & 1, timeout_ns, C::kSleepSoftmax)) {
                    record_timeout(8);
                    ok = false;
                    break;
                }
                tc_fence_after();
                uint32_t sr[128];
                tmem_ld128_sync(tS, sr);
                warp_arrive_tc(&bars->s_free[g]);  // S(J) is in registers: S(J+2) may go there
                // MASK: the key tile of visit J and the row's 128 bits of it came with V(J)
                // into V slot J % S_ (the visits of a tile map step over empty tiles; rows
                // past Nq read zero fill); otherwise visit t is tile kt0 + t.
                int kv0 = (kt0 + t) * kBN;
                uint4 mw;
                if constexpr (MASK != 0) {
                    const int vs = J % S_;
                    if (!warp_wait(&bars->v_full[vs], (J / S_) & 1, timeout_ns)) {
                        record_timeout(17);
                        ok = false;
                        break;
                    }
                    kv0 = bars->v_kt[vs] * kBN;
                    mw = reinterpret_cast<const uint4*>(smem + C::kMsk + vs * C::kMskBytes)[r];
                }
                if constexpr (MASK != 0) {
                    // The explicit mask: a key whose bit is 0 takes no part (score -inf).  The
                    // key limit (causal, key lengths, the end of the keys) is folded into the
                    // words first, so that one masking pass serves both (a second unrolled pass
                    // over the row cost these kernels instruction-fetch stalls).  Words of all
                    // ones (the usual case for structured masks) cost one test.
                    uint32_t words[4] = {mw.x, mw.y, mw.z, mw.w};
                    const int lim = key_limit - kv0;  // the limit allows keys e <= lim
#pragma unroll
                    for (int c = 0; c < 4; ++c) {
                        const int lc = lim - 32 * c;
                        words[c] &= lc >= 31 ? 0xffffffffu
                                             : (lc < 0 ? 0u : (0xffffffffu >> (31 - lc)));
                    }
#pragma unroll
                    for (int c = 0; c < 4; ++c) {
                        if (words[c] == 0xffffffffu) continue;
#pragma unroll
                        for (int e = 0; e < 32; ++e)
                            if (!((words[c] >> e) & 1u)) sr[c * 32 + e] = __float_as_uint(-INFINITY);
                    }
                } else if (kv0 + kBN - 1 > key_limit) {
#pragma unroll
                    for (int e = 0; e < 128; ++e)
                        if (kv0 + e > key_limit) sr[e] = __float_as_uint(-INFINITY);
                }
                // Row max with two-input max.f32: on this GPU the three-input form issues far
                // more slowly and holds back the exponentials that follow.
                float m16[16];
#pragma unroll
                for (int u = 0; u < 16; ++u) m16[u] = __uint_as_float(sr[u]);
#pragma unroll
                for (int e = 16; e < 128; ++e)
                    m16[e & 15] = fmaxf(m16[e & 15], __uint_as_float(sr[e]));
#pragma unroll
                for (int w = 8; w >= 1; w >>= 1)
#pragma unroll
                    for (int u = 0; u < w; ++u) m16[u] = fmaxf(m16[u], m16[u + w]);
                const float mx = m16[0] * scale_log2;
                // Reference max after tile J-1 (the other group's), handed over per row; the
                // first tile of an item starts from -inf.  Independent groups (d = 64) keep
                // their own reference instead.
                float m_prev = -INFINITY;
                if constexpr (C::kIndep) {
                    m_prev = m_last;
                } else if (J >= 1) {
                    named_bar_sync(kBarHandOff + ((J - 1) & 1), 256);
                    if (t >= 1) m_prev = bars->mref[(J - 1) & 1][r];
                }
                stage = 1;
                // Move the reference only when this tile's max exceeds it by more than the
                // threshold (always on the first finite tile: -inf gives +inf > threshold),
                // and then past the tile's max by the headroom.
                const float m_new =
                    (mx - m_prev > kRescaleThreshold) ? mx + kRescaleHeadroom : m_prev;
                if (!C::kIndep && J + 1 < J_total) {
                    bars->mref[J & 1][r] = m_new;
                    named_bar_arrive(kBarHandOff + (J & 1), 256);
                }
                stage = 2;
                // O (after P(J-1) V) is relative to m_prev; this group's l to m_last.
                const float alpha_o = (m_new == m_prev) ? 1.f : ex2_approx(m_prev - m_new);
                const float alpha_l = (m_new == m_last) ? 1.f : ex2_approx(m_last - m_new);
                // Nothing allowed yet (m_new = -inf): shift by 0 so every term is exp(-inf) = 0.
                const float m_use = (m_new == -INFINITY) ? 0.f : m_new;
                uint32_t p[64];
                float2 rs = make_float2(0.f, 0.f), rs2 = make_float2(0.f, 0.f);
                const float2 c2 = make_float2(scale_log2, scale_log2);
                const float2 nm2 = make_float2(-m_use, -m_use);
#pragma unroll
                for (int e = 0; e < 128; e += 4) {
                    float2 t0 = ffma2(
                        make_float2(__uint_as_float(sr[e]), __uint_as_float(sr[e + 1])), c2, nm2);
                    float2 t1 = ffma2(
                        make_float2(__uint_as_float(sr[e + 2]), __uint_as_float(sr[e + 3])), c2,
                        nm2);
                    t0.x = ex2_approx(t0.x);
                    t0.y = ex2_approx(t0.y);
                    t1.x = ex2_approx(t1.x);
                    t1.y = ex2_approx(t1.y);
                    rs = fadd2(rs, t0);
                    rs2 = fadd2(rs2, t1);
                    p[e >> 1] = pack_bf16x2(t0.x, t0.y);
                    p[(e >> 1) + 1] = pack_bf16x2(t1.x, t1.y);
                }
                l = l * alpha_l + ((rs.x + rs.y) + (rs2.x + rs2.y));
                m_last = m_new;
                // P buffer pb was last read by P(J - kP) V.
                const int pb = J % C::kP;
                if (J >= C::kP && !pv_wait(bars, J - C::kP, timeout_ns, C::kSleepSoftmax)) {
                    record_timeout(9);
                    ok = false;
                    break;
                }
                // The reference moved: O must be rescaled after the last P V into it and
                // before P(J) V: P(J-1) V for the shared accumulator; with one accumulator per
                // group, P(J-2) V (waited for above), except on the group's first tile of the
                // item, whose P V overwrites it.
                if (t >= (C::kIndep ? 2 : 1) && __any_sync(0xffffffffu, alpha_o != 1.f)) {
                    if (!C::kIndep && !pv_wait(bars, J - 1, timeout_ns, C::kSleepSoftmax)) {
                        record_timeout(14);
                        ok = false;
                        break;
                    }
                    tc_fence_after();
#pragma unroll
                    for (int c = 0; c < D / 32; ++c) {
                        uint32_t o[32];
                        tmem_ld32_sync(tO + c * 32, o);
#pragma unroll
                        for (int e = 0; e < 32; ++e)
                            o[e] = __float_as_uint(__uint_as_float(o[e]) * alpha_o);
                        tmem_st32_sync(tO + c * 32, o);
                    }
                }
                tc_fence_after();
                tmem_st64_sync(tmem + lane_addr + C::kTmemP + pb * 64, p);
                warp_arrive_tc(&bars->p_full[pb]);
            }
            // Make up the hand-off passes a stop left out, in the same order.
            for (; !C::kIndep && J < J0 + n; J += 2, stage = 0) {
                if (stage == 0 && J >= 1) named_bar_sync(kBarHandOff + ((J - 1) & 1), 256);
                if (stage <= 1 && J + 1 < J_total)
                    named_bar_arrive(kBarHandOff + (J & 1), 256);
            }
            // This group's (m, l) of the item for the epilogue, once it has read the slot's
            // previous item.
            const int slot = k % kFinSlots;
            if (ok && k >= kFinSlots &&
                !warp_wait(&bars->fin_free[slot], ((k / kFinSlots) - 1) & 1, timeout_ns)) {
                record_timeout(16);
                ok = false;
            }
            bars->fin[slot][g][0][r] = m_last;
            bars->fin[slot][g][1][r] = l;
            __syncwarp();
            if (lane == 0) mbar_arrive(&bars->fin_full[slot]);
            J0 += n;
        }
        tc_fence_before();
        named_bar_arrive(kBarTeardown, kTeardownThreads);
    }
}

// Combine of the split-key partial states: for each row, the partial outputs O_s (normalised
// by their own sums) and log-sum-exps LSE_s are merged with the lesson's two-worker merge in
// log form: M = max_s LSE_s, w_s = exp(LSE_s - M), O = sum_s w_s O_s / sum_s w_s,
// LSE = M + ln sum_s w_s.  Empty ranges have LSE_s = -inf and weigh nothing; a row with no
// allowed key at all gets O = 0 and LSE = -inf.  One warp per row, D/32 values per lane.
template <int D>
__global__ void __launch_bounds__(256)
    splitkv_combine_kernel(const float* __restrict__ ws_O, const float* __restrict__ ws_LSE,
                           __nv_bfloat16* __restrict__ O, float* __restrict__ LSE, long long rows,
                           int n_splits) {
    constexpr int E = D / 32;  // values per lane
    const int lane = threadIdx.x & 31;
    for (long long r = (static_cast<long long>(blockIdx.x) * blockDim.x + threadIdx.x) >> 5;
         r < rows; r += (static_cast<long long>(gridDim.x) * blockDim.x) >> 5) {
        float M = -INFINITY;
        for (int s = lane; s < n_splits; s += 32) M = fmaxf(M, ws_LSE[s * rows + r]);
#pragma unroll
        for (int off = 16; off > 0; off >>= 1) M = fmaxf(M, __shfl_xor_sync(0xffffffffu, M, off));
        float acc[E];
#pragma unroll
        for (int e = 0; e < E; ++e) acc[e] = 0.f;
        float wsum = 0.f;
        if (M != -INFINITY) {
            for (int s = 0; s < n_splits; ++s) {
                const float ls = ws_LSE[s * rows + r];
                const float w = ex2_approx((ls - M) * 1.4426950408889634f);  // ls = -inf -> 0
                wsum += w;
                const float* src = ws_O + (static_cast<size_t>(s) * rows + r) * D + lane * E;
                if (E == 4) {
                    const float4 v = *reinterpret_cast<const float4*>(src);
                    acc[0] += w * v.x;
                    acc[1] += w * v.y;
                    acc[2] += w * v.z;
                    acc[E > 3 ? 3 : 0] += w * v.w;
                } else {
                    const float2 v = *reinterpret_cast<const float2*>(src);
                    acc[0] += w * v.x;
                    acc[E > 1 ? 1 : 0] += w * v.y;
                }
            }
        }
        const float inv = wsum > 0.f ? 1.f / wsum : 0.f;
        __nv_bfloat16* dst = O + static_cast<size_t>(r) * D + lane * E;
        if (E == 4) {
            uint2 pk;
            pk.x = pack_bf16x2(acc[0] * inv, acc[1 % E] * inv);
            pk.y = pack_bf16x2(acc[2 % E] * inv, acc[3 % E] * inv);
            *reinterpret_cast<uint2*>(dst) = pk;
        } else {
            *reinterpret_cast<uint32_t*>(dst) = pack_bf16x2(acc[0] * inv, acc[1 % E] * inv);
        }
        if (lane == 0 && LSE != nullptr)
            LSE[r] = (M == -INFINITY) ? -INFINITY : M + logf(wsum);
    }
}

int device_sm_count() {
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

template <int MASK>
MaskMap<MASK> mask_map(const CUtensorMap& tm, const FaParams& p) {
    if constexpr (MASK != 0) return MaskArgs{tm, MASK == 2 ? p.tile_map : nullptr, p.tmap_words};
    else return NoMaskMap{};
}

template <int D, bool CAUSAL, bool SPLIT, int MASK = 0>
int launch_kernel(const CUtensorMap& tq, const CUtensorMap& tk, const CUtensorMap& tv,
                  const CUtensorMap& tm,
                  const FaParams& prm, cudaStream_t stream) {
    using C = Cfg<D, (MASK != 0)>;
    static std::once_flag once;
    static cudaError_t attr_err = cudaSuccess;
    std::call_once(once, [] {
        attr_err = cudaFuncSetAttribute(fa_fwd_kernel<D, CAUSAL, SPLIT, MASK>,
                                        cudaFuncAttributeMaxDynamicSharedMemorySize, C::kDynSmem);
    });
    if (attr_err != cudaSuccess) return FA_ERR_CUDA;
    const long long items = static_cast<long long>(prm.n_qtiles) * prm.BH * prm.n_splits;
    if (items > 0x7fffffffLL) return FA_ERR_UNSUPPORTED;
    if (items == 0) return FA_OK;
    // Persistent: one CTA per SM (the shared memory and TMEM allow no more), each taking every
    // gridDim.x-th work item.
    FaParams p = prm;
    p.n_items = static_cast<int>(items);
    {
        // Causal: when the K and V of all heads (2 x Nk x D bf16 each per head) would not stay
        // in the L2 together, interleave only as many heads as fit in 64 MB, about half of it.
        const long long kv_bytes = 4LL * prm.Nk * D;
        const long long share = prm.H / prm.H_kv;  // query heads reading one K/V head
        long long g = prm.BH;
        if (kv_bytes > 0 && kv_bytes * (prm.BH / share) > (128LL << 20))
            g = ((64LL << 20) / kv_bytes) * share;
        p.head_group = static_cast<int>(g < 1 ? 1 : (g > prm.BH ? prm.BH : g));
    }
    // The output's tensor map (bf16 [BH, Nq, D], as Q's); the split-key kernels write fp32
    // partials with plain stores and take Q's map in its place.
    CUtensorMap to = tq;
    if (!SPLIT) {
        const int st = make_bhnd_tensor_map(&to, prm.O, prm.BH, prm.Nq, D);
        if (st != FA_OK) return st;
    }
    const int sms = device_sm_count();
    const long long ctas = (sms > 0 && items > sms) ? sms : items;
    fa_fwd_kernel<D, CAUSAL, SPLIT, MASK>
        <<<static_cast<unsigned>(ctas), kThreads, C::kDynSmem, stream>>>(
            tq, tk, tv, mask_map<MASK>(tm, p), to, static_cast<const FaKernelParams&>(p));
    return cudaGetLastError() == cudaSuccess ? FA_OK : FA_ERR_CUDA;
}

// The tile map of an explicit mask.  Block `blk` = inst * n_qtiles + qt covers query tile qt of
// mask instance inst (b = inst / inst_h, h = inst % inst_h); bit kt of its row is set when some
// query row of the tile allows some key of key tile kt.  For each word of the row (32 key
// tiles), lane l of warp w ORs the 16-byte group of key tile 32 * word + l down rows w, w + 4,
// ... of the tile (a warp reads 512 consecutive bytes of a row), the warps' votes meet in
// shared memory; bits past Nk in the last key tile are not keys and are dropped.
__global__ void __launch_bounds__(128)
    mask_tile_map_kernel(const uint32_t* __restrict__ mask, long long mask_bs, long long mask_hs,
                         int inst_h, int Nq, int Nk, int mask_words, int n_qtiles, int n_kt,
                         int tmap_words, long long n_blocks, uint32_t* __restrict__ out) {
    __shared__ uint32_t votes[4];
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    for (long long blk = blockIdx.x; blk < n_blocks; blk += gridDim.x) {
        const int qt = static_cast<int>(blk % n_qtiles);
        const long long inst = blk / n_qtiles;
        const uint32_t* base = mask + (inst / inst_h) * mask_bs + (inst % inst_h) * mask_hs;
        const int r0 = qt * kBM, r1 = min(r0 + kBM, Nq);
        uint32_t* row_out = out + blk * tmap_words;
        for (int wi = 0; wi < tmap_words; ++wi) {
            const int kt = 32 * wi + lane;
            bool any = false;
            if (kt < n_kt) {
                uint4 acc = make_uint4(0u, 0u, 0u, 0u);
#pragma unroll 8
                for (int r = r0 + warp; r < r1; r += 4) {
                    const uint4 v = reinterpret_cast<const uint4*>(
                        base + static_cast<long long>(r) * mask_words)[kt];
                    acc.x |= v.x;
                    acc.y |= v.y;
                    acc.z |= v.z;
                    acc.w |= v.w;
                }
                const int valid = Nk - kt * kBN;  // keys of this tile below Nk
                if (valid < kBN) {
                    uint32_t w[4] = {acc.x, acc.y, acc.z, acc.w};
#pragma unroll
                    for (int c = 0; c < 4; ++c) {
                        const int vb = valid - 32 * c;
                        if (vb <= 0) w[c] = 0u;
                        else if (vb < 32) w[c] &= ~(~0u << vb);
                    }
                    acc = make_uint4(w[0], w[1], w[2], w[3]);
                }
                any = (acc.x | acc.y | acc.z | acc.w) != 0u;
            }
            const unsigned bal = __ballot_sync(0xffffffffu, any);
            if (lane == 0) votes[warp] = bal;
            __syncthreads();
            if (threadIdx.x == 0) row_out[wi] = votes[0] | votes[1] | votes[2] | votes[3];
            __syncthreads();
        }
    }
}

template <bool SPLIT>
int launch_dispatch(int64_t d, bool causal, const CUtensorMap& tq, const CUtensorMap& tk,
                    const CUtensorMap& tv, const CUtensorMap& tm, const FaParams& prm,
                    cudaStream_t stream) {
    if (prm.mask) {  // explicit masks: one pass or split keys, with or without a tile map
        const bool map = prm.tile_map != nullptr;
        if (d == 64) {
            if (map)
                return causal ? launch_kernel<64, true, SPLIT, 2>(tq, tk, tv, tm, prm, stream)
                              : launch_kernel<64, false, SPLIT, 2>(tq, tk, tv, tm, prm, stream);
            return causal ? launch_kernel<64, true, SPLIT, 1>(tq, tk, tv, tm, prm, stream)
                          : launch_kernel<64, false, SPLIT, 1>(tq, tk, tv, tm, prm, stream);
        }
        if (d == 128) {
            if (map)
                return causal ? launch_kernel<128, true, SPLIT, 2>(tq, tk, tv, tm, prm, stream)
                              : launch_kernel<128, false, SPLIT, 2>(tq, tk, tv, tm, prm, stream);
            return causal ? launch_kernel<128, true, SPLIT, 1>(tq, tk, tv, tm, prm, stream)
                          : launch_kernel<128, false, SPLIT, 1>(tq, tk, tv, tm, prm, stream);
        }
        return FA_ERR_UNSUPPORTED;
    }
    if (d == 64)
        return causal ? launch_kernel<64, true, SPLIT>(tq, tk, tv, tm, prm, stream)
                      : launch_kernel<64, false, SPLIT>(tq, tk, tv, tm, prm, stream);
    if (d == 128)
        return causal ? launch_kernel<128, true, SPLIT>(tq, tk, tv, tm, prm, stream)
                      : launch_kernel<128, false, SPLIT>(tq, tk, tv, tm, prm, stream);
    return FA_ERR_UNSUPPORTED;
}

int make_maps(const void* Q, const void* K, const void* V, const AttnShape& sh, CUtensorMap* tq,
              CUtensorMap* tk, CUtensorMap* tv) {
    int st = make_bhnd_tensor_map(tq, Q, sh.B * sh.H, sh.Nq, sh.d);
    if (st == FA_OK) st = make_bhnd_tensor_map(tk, K, sh.B * sh.H_kv, sh.Nk, sh.d);
    if (st == FA_OK) st = make_bhnd_tensor_map(tv, V, sh.B * sh.H_kv, sh.Nk, sh.d);
    return st;
}

bool shape_fits(const AttnShape& sh) {
    return sh.Nq <= (1LL << 30) && sh.Nk <= (1LL << 30) && sh.B * sh.H <= (1LL << 30) &&
           sh.H_kv >= 1 && sh.H % sh.H_kv == 0;
}

FaParams base_params(const AttnShape& sh, float scale) {
    FaParams prm{};
    prm.Nq = static_cast<int>(sh.Nq);
    prm.Nk = static_cast<int>(sh.Nk);
    prm.BH = static_cast<int>(sh.B * sh.H);
    prm.H = static_cast<int>(sh.H);
    prm.H_kv = static_cast<int>(sh.H_kv);
    prm.kv_lens = sh.kv_lens;
    prm.mask = sh.mask;
    prm.mask_bs = sh.mask_bs;
    prm.mask_hs = sh.mask_hs;
    prm.mask_words = static_cast<int>(4 * ((sh.Nk + kBN - 1) / kBN));
    prm.q_pos = static_cast<int>(sh.q_pos > 0 ? sh.q_pos : sh.Nq);
    prm.n_qtiles = static_cast<int>((sh.Nq + kBM - 1) / kBM);
    prm.tile_map = sh.tile_map;
    prm.tmap_words = static_cast<int>(((sh.Nk + kBN - 1) / kBN + 31) / 32);
    prm.scale_log2 = scale * 1.4426950408889634f;
    prm.timeout_ns = fa_wait_timeout_ns();
    return prm;
}

// Fills the tile map of sh.mask into sh.tile_map (stream-ordered before the attention).
int launch_mask_tile_map(const AttnShape& sh, cudaStream_t stream) {
    const int n_qtiles = static_cast<int>((sh.Nq + kBM - 1) / kBM);
    const int n_kt = static_cast<int>((sh.Nk + kBN - 1) / kBN);
    const long long inst_b = sh.mask_bs != 0 ? sh.B : 1, inst_h = sh.mask_hs != 0 ? sh.H : 1;
    const long long n_blocks = inst_b * inst_h * n_qtiles;
    if (n_blocks <= 0 || n_kt <= 0) return FA_OK;
    const long long grid = n_blocks < 65535LL * 16 ? n_blocks : 65535LL * 16;
    mask_tile_map_kernel<<<static_cast<unsigned>(grid), 128, 0, stream>>>(
        sh.mask, sh.mask_bs, sh.mask_hs, static_cast<int>(inst_h), static_cast<int>(sh.Nq),
        static_cast<int>(sh.Nk), static_cast<int>(4 * n_kt), n_qtiles, n_kt, (n_kt + 31) / 32,
        n_blocks, sh.tile_map);
    return cudaGetLastError() == cudaSuccess ? FA_OK : FA_ERR_CUDA;
}

// An explicit mask's tensor map, and its tile map filled by the pre-pass on `stream` when the
// caller gave a buffer for it (otherwise prm.tile_map is cleared: no tile is skipped).
int setup_mask(const AttnShape& sh, FaParams* prm, CUtensorMap* tm, cudaStream_t stream) {
    if (!sh.mask) {
        prm->tile_map = nullptr;
        return FA_OK;
    }
    const int64_t n_kt = (sh.Nk + kBN - 1) / kBN;
    int rc = make_mask_tensor_map(tm, sh.mask, 4 * n_kt, sh.Nq, sh.mask_hs != 0 ? sh.H : 1,
                                  sh.mask_bs != 0 ? sh.B : 1, sh.mask_hs, sh.mask_bs);
    if (rc != FA_OK) return rc;
    if (sh.tile_map) {
        rc = launch_mask_tile_map(sh, stream);
        if (rc != FA_OK) return rc;
    } else {
        prm->tile_map = nullptr;
    }
    return FA_OK;
}

}  // namespace

AttnShape pack_query_heads(const AttnShape& sh) {
    if (sh.H_kv <= 0 || sh.H_kv >= sh.H || sh.q_pos > 0 || sh.mask) return sh;
    return AttnShape{sh.B, sh.H_kv, sh.H_kv, (sh.H / sh.H_kv) * sh.Nq, sh.Nk, sh.d, sh.kv_lens,
                     sh.Nq};
}

int fa_fwd_launch(const void* Q, const void* K, const void* V, void* O, float* LSE, int64_t BH,
                  int64_t N, int64_t d, float scale, bool causal, cudaStream_t stream) {
    return fa_fwd_shape_launch(Q, K, V, O, LSE, AttnShape{BH, 1, 1, N, N, d, nullptr, 0}, scale,
                               causal, stream);
}

int fa_fwd_shape_launch(const void* Q, const void* K, const void* V, void* O, float* LSE,
                        const AttnShape& shape, float scale, bool causal, cudaStream_t stream) {
    const AttnShape sh = pack_query_heads(shape);
    if (!shape_fits(sh)) return FA_ERR_UNSUPPORTED;
    CUtensorMap tq, tk, tv;
    const int st = make_maps(Q, K, V, sh, &tq, &tk, &tv);
    if (st != FA_OK) return st;
    FaParams prm = base_params(sh, scale);
    CUtensorMap tm{};
    const int mrc = setup_mask(sh, &prm, &tm, stream);
    if (mrc != FA_OK) return mrc;
    prm.O = static_cast<__nv_bfloat16*>(O);
    prm.LSE = LSE;
    prm.n_splits = 1;
    prm.tiles_per_split = static_cast<int>((sh.Nk + kBN - 1) / kBN);
    return launch_dispatch<false>(sh.d, causal, tq, tk, tv, tm, prm, stream);
}

int64_t mask_tile_map_words(int64_t B, int64_t H, int64_t Nq, int64_t Nk, int64_t mask_bs,
                            int64_t mask_hs) {
    const int64_t n_qtiles = (Nq + kBM - 1) / kBM, n_kt = (Nk + kBN - 1) / kBN;
    int64_t a, b, c;
    if (__builtin_mul_overflow(mask_bs != 0 ? B : 1, mask_hs != 0 ? H : 1, &a) ||
        __builtin_mul_overflow(a, n_qtiles, &b) || __builtin_mul_overflow(b, (n_kt + 31) / 32, &c))
        return -1;
    return c;
}

int64_t splitkv_choose_splits(int64_t BH, int64_t Nq, int64_t Nk, int64_t requested) {
    const int64_t n_kv_all = (Nk + kBN - 1) / kBN;
    if (n_kv_all <= 0) return 0;
    int64_t splits = requested;
    if (splits <= 0) {
        // Enough CTAs for about eight waves, so the key ranges of a few heads spread over
        // every SM; the combine that follows is cheap next to the attention.
        const int64_t base = ((Nq + kBM - 1) / kBM) * BH;
        const int64_t sms = device_sm_count() > 0 ? device_sm_count() : 148;
        splits = base > 0 ? (8 * sms + base - 1) / base : 1;
        if (splits > 64) splits = 64;
    }
    if (splits > n_kv_all) splits = n_kv_all;
    if (splits < 1) splits = 1;
    // Every split gets the same number of key tiles; drop the ranges left empty by rounding.
    const int64_t tps = (n_kv_all + splits - 1) / splits;
    return (n_kv_all + tps - 1) / tps;
}

int fa_fwd_splitkv_launch(const void* Q, const void* K, const void* V, void* O, float* LSE,
                          const AttnShape& shape, float scale, bool causal, int64_t n_splits,
                          float* ws_O, float* ws_LSE, cudaStream_t stream) {
    const AttnShape sh = pack_query_heads(shape);
    if (!shape_fits(sh)) return FA_ERR_UNSUPPORTED;
    const long long rows = static_cast<long long>(sh.B * sh.H) * sh.Nq;
    if (n_splits > 1) {
        CUtensorMap tq, tk, tv;
        const int st = make_maps(Q, K, V, sh, &tq, &tk, &tv);
        if (st != FA_OK) return st;
        const int64_t n_kv_all = (sh.Nk + kBN - 1) / kBN;
        FaParams prm = base_params(sh, scale);
        prm.ws_O = ws_O;
        prm.ws_LSE = ws_LSE;
        prm.n_splits = static_cast<int>(n_splits);
        prm.tiles_per_split = static_cast<int>((n_kv_all + n_splits - 1) / n_splits);
        CUtensorMap tm{};
        const int mrc = setup_mask(sh, &prm, &tm, stream);
        if (mrc != FA_OK) return mrc;
        const int rc = launch_dispatch<true>(sh.d, causal, tq, tk, tv, tm, prm, stream);
        if (rc != FA_OK) return rc;
    } else if (n_splits == 1) {
        return fa_fwd_shape_launch(Q, K, V, O, LSE, sh, scale, causal, stream);
    }
    // n_splits > 1: merge the partial states; n_splits == 0 (no key at all): O = 0, LSE = -inf.
    const long long warps = rows;
    long long grid = (warps + 7) / 8;
    if (grid > 65535LL * 64) grid = 65535LL * 64;
    if (grid < 1) return FA_OK;
    const int ns = static_cast<int>(n_splits > 1 ? n_splits : 0);
    if (sh.d == 64)
        splitkv_combine_kernel<64><<<static_cast<unsigned>(grid), 256, 0, stream>>>(
            ws_O, ws_LSE, static_cast<__nv_bfloat16*>(O), LSE, rows, ns);
    else
        splitkv_combine_kernel<128><<<static_cast<unsigned>(grid), 256, 0, stream>>>(
            ws_O, ws_LSE, static_cast<__nv_bfloat16*>(O), LSE, rows, ns);
    return cudaGetLastError() == cudaSuccess ? FA_OK : FA_ERR_CUDA;
}

namespace {
// Waits on an mbarrier that nothing ever completes, with the same bounded wait the attention
// kernel uses, and records the timeout in the device status word.  Exercises the error path
// without touching TMA, TMEM or the tensor cores.
__global__ void __launch_bounds__(32, 1) selftest_wait_kernel(unsigned long long timeout_ns) {
    __shared__ uint64_t bar;
    if (threadIdx.x == 0) {
        mbar_init(&bar, 1);
        fence_mbar_init();
    }
    __syncwarp();
    if (!warp_wait(&bar, 0, timeout_ns) && threadIdx.x == 0) record_timeout(15);
}
}  // namespace

int selftest_wait_launch(long long timeout_us, cudaStream_t stream) {
    if (timeout_us < 1 || timeout_us > 10000000) return FA_ERR_INVALID_ARG;
    const unsigned long long timeout_ns = static_cast<unsigned long long>(timeout_us) * 1000ull;
    selftest_wait_kernel<<<1, 32, 0, stream>>>(timeout_ns);
    return cudaGetLastError() == cudaSuccess ? FA_OK : FA_ERR_CUDA;
}

int* device_status_word() {
    static int* addr = nullptr;
    static std::once_flag once;
    std::call_once(once, [] {
        void* p = nullptr;
        if (cudaGetSymbolAddress(&p, g_fa_device_status) == cudaSuccess)
            addr = static_cast<int*>(p);
    });
    return addr;
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
