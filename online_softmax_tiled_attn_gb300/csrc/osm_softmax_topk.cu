// osm_softmax_topk.cu -- softmax with top-k selection in one read of each row, for sm_103a.
//
// The method: "How FlashAttention avoids storing the giant score table" (spicyshark.co,
// Online softmax lesson), section "Where this is used in practice": the online normaliser also
// serves softmax fused with top-k selection (only the k largest scores are kept).  While a
// thread streams its part of a row it keeps the running (m, l) of "The idea" and the k best
// (value, column) pairs it has seen; the threads' partial states are then combined, (m, l) by
// the two-worker merge of "From softmax to attention" and the top-k lists by repeatedly taking
// the best head among the lists.  The outputs are the k columns with the largest x (ties: the
// smaller column first), their shares y = exp(x - m) / l, and lse = m + ln l.
//
// GB300 mapping (HBM-bound: 4 bytes read per element, nothing written per element).  Rows with
// 16-byte access and k >= 2 take the staged kernels further down (rows brought into shared
// memory by bulk copies); the register kernels described here serve k = 1 and rows that are
// not 16-byte aligned:
//   * rows up to 4096 columns: one warp per row; longer rows: the 8 warps of a CTA share a row
//     and their lists meet in shared memory;
//   * 16-byte loads when the row allows them;
//   * k >= 2, two passes over the row, the second from L2: the first keeps the running (m, l)
//     of each thread's part, whose running maximum comes with it; the k-th largest of the
//     threads' maxima (over a warp; the largest such value over the warps of a CTA) is a floor
//     under the row's k-th largest value, since k distinct entries reach it.  The second pass
//     offers only the values at or above max(floor, the list's bar) to the list, so that almost
//     every value costs a load and one comparison.  (One pass that offered every value to the
//     list ran at 2.1 and 1.5 TB/s for the two bench workloads: while the list's bar is still
//     low, most values of the first steps enter it; one pass that compared against a floor
//     taken after its first step ran at 3.0 and 1.7 TB/s, with fewer loads in flight than a
//     pure first pass; fewer rows in flight, or chunks, so that the second pass surely hits
//     L2, ran slower than the full grid.)
//   * the k best so far live across the lanes of a warp, one per lane; a value is compared
//     with the k-th best (the bar, the same in every lane), and the few that beat it are
//     inserted with a ballot and a shuffle.  (Per-thread sorted lists, which most values of a
//     short per-thread stream enter, measured 0.2-1 TB/s for k = 8..32.)
//   * k = 1: one pass, a best per lane;
//   * persistent grid, rows handed out round-robin.
#include <cuda_runtime.h>

#include <climits>
#include <cmath>
#include <mutex>

#include "osm_internal.h"
#include "ptx_sm103.cuh"

namespace osm {
namespace {

constexpr float kLog2e = 1.4426950408889634f;
constexpr int kThreads = 256;
constexpr int kWarps = kThreads / 32;

__device__ __forceinline__ float ex2a(float x) {
    float y;
    asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}

// (x, j) ranks before (y, i): larger value first, then the smaller column.
__device__ __forceinline__ bool before(float x, int j, float y, int i) {
    return x > y || (x == y && j < i);
}

struct Stat {
    float m, l;
};

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

// One block of the online recurrence: the values v[0..n) enter the state.
template <int N>
__device__ __forceinline__ void update(Stat& s, const float (&v)[N]) {
    float mx = v[0];
#pragma unroll
    for (int e = 1; e < N; ++e) mx = fmaxf(mx, v[e]);
    const float m = fmaxf(s.m, mx);
    if (m == -INFINITY) return;  // nothing finite yet: adds nothing
    float l = s.m == -INFINITY ? 0.f : s.l * ex2a((s.m - m) * kLog2e);
#pragma unroll
    for (int e = 0; e < N; ++e) l += ex2a((v[e] - m) * kLog2e);
    s = Stat{m, l};
}

// The warp's k best (value, column) pairs so far, one per lane, best in lane 0; lanes >= k hold
// nothing (-inf, INT_MAX).  The k-th best (lane k - 1) is the bar a new value must beat, so
// once the bar has risen almost every value costs one comparison.
struct WarpTop {
    float v = -INFINITY;
    int c = INT_MAX;
    float bar_v = -INFINITY;  // the k-th best so far, the same in every lane
    int bar_c = INT_MAX;

    // Inserts (x, j), which ranks before the bar, at its place; the entries after it move down
    // one lane and the k-th drops out.
    __device__ __forceinline__ void insert(float x, int j, int k) {
        const int lane = threadIdx.x & 31;
        const unsigned ahead = __ballot_sync(0xffffffffu, lane < k && before(v, c, x, j));
        const int pos = __popc(ahead);  // entries that stay ahead of (x, j)
        const float uv = __shfl_up_sync(0xffffffffu, v, 1);
        const int uc = __shfl_up_sync(0xffffffffu, c, 1);
        if (lane < k) {
            if (lane > pos) {
                v = uv;
                c = uc;
            } else if (lane == pos) {
                v = x;
                c = j;
            }
        }
        bar_v = __shfl_sync(0xffffffffu, v, k - 1);
        bar_c = __shfl_sync(0xffffffffu, c, k - 1);
    }
    __device__ __forceinline__ void finish() {}

    // Every lane offers n values (x[e], col[e]); one vote tells whether any lane holds a value
    // that beats the bar, and those lanes' values are then inserted one at a time, each
    // re-checked against the bar as it rises.
    template <int N>
    __device__ __forceinline__ void offer(const float (&x)[N], const int (&col)[N], int k) {
        bool mine = false;
#pragma unroll
        for (int e = 0; e < N; ++e) mine |= before(x[e], col[e], bar_v, bar_c);
        unsigned lanes = __ballot_sync(0xffffffffu, mine);
        while (lanes) {
            const int src = __ffs(lanes) - 1;
            lanes &= lanes - 1;
#pragma unroll
            for (int e = 0; e < N; ++e) {
                const float xv = __shfl_sync(0xffffffffu, x[e], src);
                const int xc = __shfl_sync(0xffffffffu, col[e], src);
                if (before(xv, xc, bar_v, bar_c)) insert(xv, xc, k);
            }
        }
    }
};

// k = 1: each lane keeps its own best (no vote per step); finish() leaves the warp's best in
// lane 0 and nothing in the other lanes, as WarpTop holds it.
struct LaneBest {
    float v = -INFINITY;
    int c = INT_MAX;

    template <int N>
    __device__ __forceinline__ void offer(const float (&x)[N], const int (&col)[N], int) {
#pragma unroll
        for (int e = 0; e < N; ++e)
            if (before(x[e], col[e], v, c)) {
                v = x[e];
                c = col[e];
            }
    }
    __device__ __forceinline__ void finish() {
#pragma unroll
        for (int off = 16; off > 0; off >>= 1) {
            const float ov = __shfl_xor_sync(0xffffffffu, v, off);
            const int oc = __shfl_xor_sync(0xffffffffu, c, off);
            if (before(ov, oc, v, c)) {
                v = ov;
                c = oc;
            }
        }
        if ((threadIdx.x & 31) != 0) {
            v = -INFINITY;
            c = INT_MAX;
        }
    }
};

// Streams the row part of thread t (of nthr threads sharing the row) into its state and the
// warp's list.  All 32 lanes of a warp run the same iterations (the list lives across lanes).
template <bool VEC, class Top>
__device__ __forceinline__ void scan(const float* row, int cols, int t, int nthr, int k,
                                     Stat& st, Top& top) {
    const int lane = threadIdx.x & 31;
    const int lane0 = t - lane;  // the warp's first thread
    if constexpr (VEC) {
        // Four 16-byte loads in flight per thread before any of them is used.
        constexpr int kAhead = 4;
        const float4* r4 = reinterpret_cast<const float4*>(row);
        const int n4 = cols >> 2;
        for (int u0 = lane0; u0 < n4; u0 += kAhead * nthr) {
            float4 q[kAhead];
#pragma unroll
            for (int a = 0; a < kAhead; ++a) {
                const int u = u0 + a * nthr + lane;
                q[a] = u < n4 ? __ldcs(r4 + u)
                              : make_float4(-INFINITY, -INFINITY, -INFINITY, -INFINITY);
            }
#pragma unroll
            for (int a = 0; a < kAhead; ++a) {
                const int u = u0 + a * nthr + lane;
                const float v[4] = {q[a].x, q[a].y, q[a].z, q[a].w};
                const bool in = u < n4;
                if (in) update(st, v);
                // past the row: (-inf, INT_MAX) never beats the bar
                const int col[4] = {in ? 4 * u : INT_MAX, in ? 4 * u + 1 : INT_MAX,
                                    in ? 4 * u + 2 : INT_MAX, in ? 4 * u + 3 : INT_MAX};
                top.offer(v, col, k);
            }
        }
    } else {
        // Four 4-byte loads per thread per step, columns nthr apart.
        for (int j0 = lane0; j0 < cols; j0 += 4 * nthr) {
            float v[4];
            int col[4];
#pragma unroll
            for (int a = 0; a < 4; ++a) {
                const int j = j0 + a * nthr + lane;
                const bool in = j < cols;
                v[a] = in ? __ldcs(row + j) : -INFINITY;
                col[a] = in ? j : INT_MAX;
            }
            update(st, v);  // -inf past the row adds nothing
            top.offer(v, col, k);
        }
    }
}

// The 32 lanes' values sorted across the warp in descending order (bitonic network): lane i
// gets the (i+1)-th largest.
__device__ __forceinline__ float warp_sorted_desc(float x) {
    const int lane = threadIdx.x & 31;
#pragma unroll
    for (int size = 2; size <= 32; size <<= 1) {
#pragma unroll
        for (int stride = size >> 1; stride > 0; stride >>= 1) {
            const float o = __shfl_xor_sync(0xffffffffu, x, stride);
            const bool desc = (lane & size) == 0 || size == 32;
            const bool lower = (lane & stride) == 0;
            x = (lower == desc) ? fmaxf(x, o) : fminf(x, o);
        }
    }
    return x;
}

// The k-th largest of the 32 lanes' values (the same in every lane).
__device__ __forceinline__ float warp_kth_largest(float x, int k) {
    return __shfl_sync(0xffffffffu, warp_sorted_desc(x), k - 1);
}

// k >= 2, pass 1 over units [lo, hi) of a row (a unit is a float4 in the vector form, a
// float otherwise; thread t of nthr takes units lo + t, lo + t + nthr, ...): the online state,
// whose running maximum st.m comes with it.  The loads keep the data in L2 for pass 2.
template <bool VEC>
__device__ __forceinline__ void stats_pass(const float* row, int lo, int hi, int t, int nthr,
                                           Stat& st) {
    constexpr int kAhead = 4;
    for (int u0 = lo + t; u0 < hi; u0 += kAhead * nthr) {
        if constexpr (VEC) {
            const float4* r4 = reinterpret_cast<const float4*>(row);
            float4 q[kAhead];
#pragma unroll
            for (int a = 0; a < kAhead; ++a) {
                const int u = u0 + a * nthr;
                q[a] = u < hi ? __ldcg(r4 + u)
                              : make_float4(-INFINITY, -INFINITY, -INFINITY, -INFINITY);
            }
#pragma unroll
            for (int a = 0; a < kAhead; ++a) {
                const float v[4] = {q[a].x, q[a].y, q[a].z, q[a].w};
                update(st, v);  // -inf past the range adds nothing
            }
        } else {
            float v[kAhead];
#pragma unroll
            for (int a = 0; a < kAhead; ++a) {
                const int j = u0 + a * nthr;
                v[a] = j < hi ? __ldcg(row + j) : -INFINITY;
            }
            update(st, v);
        }
    }
}

// k >= 2, pass 2 over the same units: the values at or above `floor` are offered to the warp's
// list.  All 32 lanes of a warp run the same iterations (the list lives across lanes).
template <bool VEC>
__device__ __forceinline__ void select_pass(const float* row, int lo, int hi, int t, int nthr,
                                            int k, float floor, WarpTop& top) {
    constexpr int kAhead = 4;
    const int lane = threadIdx.x & 31;
    for (int u0 = lo + t - lane; u0 < hi; u0 += kAhead * nthr) {
        if constexpr (VEC) {
            const float4* r4 = reinterpret_cast<const float4*>(row);
            float4 q[kAhead];
#pragma unroll
            for (int a = 0; a < kAhead; ++a) {
                const int u = u0 + a * nthr + lane;
                q[a] = u < hi ? __ldcs(r4 + u)
                              : make_float4(-INFINITY, -INFINITY, -INFINITY, -INFINITY);
            }
#pragma unroll
            for (int a = 0; a < kAhead; ++a) {
                const int u = u0 + a * nthr + lane;
                const float thr = fmaxf(floor, top.bar_v);
                const bool cand = u < hi && (q[a].x >= thr || q[a].y >= thr || q[a].z >= thr ||
                                             q[a].w >= thr);
                if (__ballot_sync(0xffffffffu, cand)) {
                    // a lane without a candidate offers nothing: (-inf, INT_MAX) never enters
                    const float v[4] = {cand ? q[a].x : -INFINITY, cand ? q[a].y : -INFINITY,
                                        cand ? q[a].z : -INFINITY, cand ? q[a].w : -INFINITY};
                    const int col[4] = {cand ? 4 * u : INT_MAX, cand ? 4 * u + 1 : INT_MAX,
                                        cand ? 4 * u + 2 : INT_MAX, cand ? 4 * u + 3 : INT_MAX};
                    top.offer(v, col, k);
                }
            }
        } else {
            float v[kAhead];
            int col[kAhead];
            const float thr = fmaxf(floor, top.bar_v);
            bool cand = false;
#pragma unroll
            for (int a = 0; a < kAhead; ++a) {
                const int j = u0 + a * nthr + lane;
                const bool in = j < hi;
                v[a] = in ? __ldcs(row + j) : -INFINITY;
                col[a] = in ? j : INT_MAX;
                cand |= in && v[a] >= thr;
            }
            if (__ballot_sync(0xffffffffu, cand)) top.offer(v, col, k);
        }
    }
}

template <class Top>
constexpr bool kFiltered = false;
template <>
constexpr bool kFiltered<WarpTop> = true;

// Lane t < k writes the t-th best with its share.
template <class Top>
__device__ __forceinline__ void write_top(const Top& top, int k, Stat s, float* vals, int* idx) {
    const int lane = threadIdx.x & 31;
    const float mu = s.m == -INFINITY ? 0.f : s.m;
    const float inv_l = s.l > 0.f ? 1.f / s.l : 0.f;
    if (lane < k) {
        vals[lane] = ex2a((top.v - mu) * kLog2e) * inv_l;
        idx[lane] = top.c;
    }
}

// ---------------------------------------------------------------------------------------------
// Rows of up to 4096 columns with 16-byte access, k >= 2: rows staged in shared memory.
// Each warp owns one or more row buffers; its lane 0 brings rows into them with bulk copies
// (cp.async.bulk), and a buffer takes its next row as soon as the warp has swept it, so the
// copy runs while the warp finishes the row (the row is read from HBM once, and no register
// holds it across a wait).  From shared memory the warp sweeps the row twice:
//   1. the lane maxima, sorted across the warp: the largest is the row max m, the k-th largest
//      the floor (k distinct entries reach it, so every entry of the top k does too);
//   2. each lane's sum of exp(x - m), and the compaction of the float4 groups that can still
//      bring an entry into the top k (largest entry at or above the floor and not below the
//      list's k-th entry, the bar) into a small candidate buffer, one vote per group.
//      Whenever it holds 32 entries or more, 32 of them are sorted across the warp (a bitonic
//      network) and merged into the warp's list of the best 32 so far (the better of entry i
//      and entry 31 - i of the two sorted lists, then a bitonic merge), and the bar rises.
//      (Entry-by-entry compaction, eight votes per step, cost half again as many
//      instructions per row.)
// The lane sums add up to l by a warp sum; lse = m + ln l.
constexpr int kStagedMaxCols = 4096;
constexpr int kStagedWarps = 4;       // warps per CTA
constexpr int kStagedMaxRing = 4;     // row buffers per warp
constexpr int kCoarseCap = 136;       // 7 groups left over + one step's 128 groups
constexpr int kFineCap = 64;          // 31 entries left over + one batch's 32
constexpr int kCandBytes = kCoarseCap * 4 + kFineCap * 8;  // per warp
constexpr unsigned long long kStagedDrainNs = 1000000000ull;

__device__ __forceinline__ float max4(const float4& q) {
    return fmaxf(fmaxf(q.x, q.y), fmaxf(q.z, q.w));
}

// Compare-exchange with the lane `stride` away: this lane keeps the better of the two entries
// if keep_better, else the worse (the order of `before`; all entries are distinct except the
// padding (-inf, INT_MAX)).
__device__ __forceinline__ void cmpx(float& v, int& c, int stride, bool keep_better) {
    const float ov = __shfl_xor_sync(0xffffffffu, v, stride);
    const int oc = __shfl_xor_sync(0xffffffffu, c, stride);
    if (before(ov, oc, v, c) == keep_better) {
        v = ov;
        c = oc;
    }
}

// Sorts one entry per lane across the warp, best in lane 0 (bitonic network).
__device__ __forceinline__ void warp_sort_desc(float& v, int& c) {
    const int lane = threadIdx.x & 31;
#pragma unroll
    for (int size = 2; size <= 32; size <<= 1) {
#pragma unroll
        for (int stride = size >> 1; stride > 0; stride >>= 1) {
            const bool desc = (lane & size) == 0 || size == 32;
            const bool lower = (lane & stride) == 0;
            cmpx(v, c, stride, lower == desc);
        }
    }
}

// (lv, lc): the warp's list of the best 32 so far, sorted, best in lane 0.  (xv, xc): one new
// entry per lane.  Leaves the best 32 of both in (lv, lc), sorted.
__device__ __forceinline__ void merge_batch(float& lv, int& lc, float xv, int xc) {
    const int lane = threadIdx.x & 31;
    warp_sort_desc(xv, xc);
    // the new entries in ascending order against the list's descending: the better of each
    // pair are the best 32 of the union, as a bitonic sequence
    const float rv = __shfl_sync(0xffffffffu, xv, 31 - lane);
    const int rc = __shfl_sync(0xffffffffu, xc, 31 - lane);
    if (before(rv, rc, lv, lc)) {
        lv = rv;
        lc = rc;
    }
#pragma unroll
    for (int stride = 16; stride > 0; stride >>= 1) cmpx(lv, lc, stride, (lane & stride) == 0);
}

// Lane 0 only: the bulk copy of row r into buffer `buf`, completing on `bar`.
__device__ __forceinline__ void staged_issue(float4* buf, const float* x, long long r, int cols,
                                             uint64_t* bar) {
    const uint32_t bytes = static_cast<uint32_t>(cols) * 4u;
    mbar_arrive_expect_tx(bar, bytes);
    bulk_load(buf, x + r * cols, bytes, bar);
}

// The warp's selection state while it sweeps a row: its list of the best 32 so far (one entry
// per lane, sorted), the bar (the list's k-th entry), the floor, and two candidate buffers.
// The coarse one holds float4 groups of the row (by index: the row is still in shared memory)
// whose largest entry can still reach the top k; their entries are then tested one by one, and
// the few that pass go to the fine buffer, which is merged into the list 32 at a time.
struct Sweep {
    int* cu;    // [kCoarseCap] groups (float4 index in the row)
    float* fv;  // [kFineCap] entries: value
    int* fc;    //             and column
    float floor;
    float lv = -INFINITY, bar_v = -INFINITY;
    int lc = INT_MAX, bar_c = INT_MAX;
    int n = 0, nf = 0;  // entries of the two buffers (the same in every lane)
    int col0 = 0;       // column of the staged segment's first entry
    float2 acc[4] = {{0.f, 0.f}, {0.f, 0.f}, {0.f, 0.f}, {0.f, 0.f}};  // lane sums, 4 chains
};

// Tests the coarse buffer's groups, 8 at a time (32 entries, one per lane), entry by entry
// against the floor and the bar; the entries that pass go to the fine buffer, which is merged
// into the list whenever it holds 32.  Without `all`, only whole batches of 8 groups are taken
// and the rest moves to the front; with `all`, every group is taken.
__device__ __forceinline__ void sweep_flush(const float* __restrict__ rowf, Sweep& S, int k,
                                            bool all) {
    const int lane = threadIdx.x & 31;
    const unsigned lt = (1u << lane) - 1u;
    __syncwarp();
    const int lim = all ? S.n : (S.n & ~7);
    int base = 0;
    for (; base < lim; base += 8) {
        const int g = base + (lane >> 2);
        float v = -INFINITY;
        int c = INT_MAX;
        if (g < S.n) {
            const int cr = 4 * S.cu[g] + (lane & 3);  // within the segment
            v = rowf[cr];
            c = S.col0 + cr;
        }
        const bool keep = g < S.n && v >= S.floor && before(v, c, S.bar_v, S.bar_c);
        const unsigned bal = __ballot_sync(0xffffffffu, keep);
        if (keep) {
            const int pos = S.nf + __popc(bal & lt);
            S.fv[pos] = v;
            S.fc[pos] = c;
        }
        S.nf += __popc(bal);
        if (S.nf >= 32) {
            __syncwarp();
            merge_batch(S.lv, S.lc, S.fv[lane], S.fc[lane]);
            const int rem = S.nf - 32;
            float tv = 0.f;
            int tc = 0;
            if (lane < rem) {
                tv = S.fv[32 + lane];
                tc = S.fc[32 + lane];
            }
            __syncwarp();
            if (lane < rem) {
                S.fv[lane] = tv;
                S.fc[lane] = tc;
            }
            __syncwarp();
            S.nf = rem;
            S.bar_v = __shfl_sync(0xffffffffu, S.lv, k - 1);
            S.bar_c = __shfl_sync(0xffffffffu, S.lc, k - 1);
        }
    }
    const int rem = all ? 0 : S.n - base;  // fewer than 8 groups
    int tu = 0;
    if (lane < rem) tu = S.cu[base + lane];
    __syncwarp();
    if (lane < rem) S.cu[lane] = tu;
    __syncwarp();
    S.n = rem;
}

// One step of the second sweep: four float4 per lane from u0 (bounds-checked if CHECK).  The
// lane sums take exp2((x - m) * log2e): x - m first, so that the largest terms keep full
// relative accuracy whatever the size of m.
template <bool CHECK>
__device__ __forceinline__ void sweep_step(const float4* __restrict__ s4, int n4, int u0,
                                           float2 c2, float2 nmu, Sweep& S, int k) {
    const int lane = threadIdx.x & 31;
    float4 q[4];
#pragma unroll
    for (int a = 0; a < 4; ++a) {
        const int u = u0 + 32 * a + lane;
        q[a] = (!CHECK || u < n4) ? s4[u]
                                  : make_float4(-INFINITY, -INFINITY, -INFINITY, -INFINITY);
    }
#pragma unroll
    for (int a = 0; a < 4; ++a) {
        const float2 t0 = fmul2(fadd2(make_float2(q[a].x, q[a].y), nmu), c2);
        const float2 t1 = fmul2(fadd2(make_float2(q[a].z, q[a].w), nmu), c2);
        S.acc[(2 * a) & 3] = fadd2(S.acc[(2 * a) & 3], make_float2(ex2a(t0.x), ex2a(t0.y)));
        S.acc[(2 * a + 1) & 3] =
            fadd2(S.acc[(2 * a + 1) & 3], make_float2(ex2a(t1.x), ex2a(t1.y)));
    }
    const float thr = fmaxf(S.floor, S.bar_v);
    float m4[4];
    bool p[4];
#pragma unroll
    for (int a = 0; a < 4; ++a) {
        m4[a] = max4(q[a]);
        p[a] = (!CHECK || u0 + 32 * a + lane < n4) && m4[a] >= thr;
    }
    if (__any_sync(0xffffffffu, p[0] || p[1] || p[2] || p[3])) {
        const unsigned lt = (1u << lane) - 1u;
#pragma unroll
        for (int a = 0; a < 4; ++a) {
            const int u = u0 + 32 * a + lane;
            // a group whose largest entry only equals the bar can beat it only with a smaller
            // column (ties at the floor, below any bar, all enter)
            const bool in = p[a] && (m4[a] > thr || thr > S.bar_v || S.col0 + 4 * u < S.bar_c);
            const unsigned bal = __ballot_sync(0xffffffffu, in);
            if (in) S.cu[S.n + __popc(bal & lt)] = u;
            S.n += __popc(bal);
        }
        if (S.n >= 8) sweep_flush(reinterpret_cast<const float*>(s4), S, k, false);
    }
}

// One staged segment of a row (n4 float4 in shared memory) enters the warp's state: sweep 1
// (the lane maxima, sorted across the warp: the segment's max, and its floor, which raises
// the running floor), the running max m, with the lane sums rescaled by exp(m_old - m_new)
// when it grows (the online recurrence of "The idea"), then sweep 2.  The segment's coarse
// candidates are all tested before it returns, so that its buffer can take the next copy.
__device__ __forceinline__ void sweep_segment(const float4* __restrict__ s4, int n4, int k,
                                              Sweep& S, float& m) {
    const int lane = threadIdx.x & 31;
    float ma = -INFINITY, mb = -INFINITY, mc = -INFINITY, md = -INFINITY;
    int u = lane;
    for (; u + 96 < n4; u += 128) {
        ma = fmaxf(ma, max4(s4[u]));
        mb = fmaxf(mb, max4(s4[u + 32]));
        mc = fmaxf(mc, max4(s4[u + 64]));
        md = fmaxf(md, max4(s4[u + 96]));
    }
    for (; u < n4; u += 32) ma = fmaxf(ma, max4(s4[u]));
    // Two values per lane, the maxima of disjoint groups (distinct entries): the k-th largest
    // of the 64 is a floor (k distinct entries reach it), and a tighter one than the k-th
    // largest of the 32 lane maxima.  With A and B the two sets sorted across the warp, it is
    // the largest of A[k-1], B[k-1] and min(A[i], B[k-2-i]) for i < k - 1.
    const float sa = warp_sorted_desc(fmaxf(ma, mb));
    const float sb = warp_sorted_desc(fmaxf(mc, md));
    const float sb_pair = __shfl_sync(0xffffffffu, sb, (k - 2 - lane) & 31);
    float kth = lane < k - 1 ? fminf(sa, sb_pair) : -INFINITY;
    if (lane == k - 1) kth = fmaxf(sa, sb);
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) kth = fmaxf(kth, __shfl_xor_sync(0xffffffffu, kth, off));
    S.floor = fmaxf(S.floor, kth);
    const float m_new = fmaxf(m, fmaxf(__shfl_sync(0xffffffffu, sa, 0), __shfl_sync(0xffffffffu, sb, 0)));
    if (m != -INFINITY && m_new != m) {  // the same in every lane
        const float f = ex2a((m - m_new) * kLog2e);
#pragma unroll
        for (int a = 0; a < 4; ++a) S.acc[a] = fmul2(S.acc[a], make_float2(f, f));
    }
    m = m_new;
    // Sweep 2: every lane runs the same steps (the list lives across lanes).
    const float mu = m == -INFINITY ? 0.f : m;  // nothing finite yet: every term exp(-inf) = 0
    const float2 c2 = make_float2(kLog2e, kLog2e);
    const float2 nmu = make_float2(-mu, -mu);
    int u0 = 0;
    for (; u0 + 128 <= n4; u0 += 128) sweep_step<false>(s4, n4, u0, c2, nmu, S, k);
    if (u0 < n4) sweep_step<true>(s4, n4, u0, c2, nmu, S, k);
    if (S.n > 0) sweep_flush(reinterpret_cast<const float*>(s4), S, k, true);
}

// The list after the last segment: the fine buffer's rest merged in.
__device__ __forceinline__ void sweep_finish(Sweep& S) {
    const int lane = threadIdx.x & 31;
    if (S.nf > 0) {
        __syncwarp();
        const bool has = lane < S.nf;
        merge_batch(S.lv, S.lc, has ? S.fv[lane] : -INFINITY, has ? S.fc[lane] : INT_MAX);
        S.nf = 0;
    }
}

// The warp's sum of exp(x - m) over everything it swept (the same in every lane).
__device__ __forceinline__ float sweep_sum(const Sweep& S) {
    float l = (S.acc[0].x + S.acc[0].y) + (S.acc[1].x + S.acc[1].y) +
              ((S.acc[2].x + S.acc[2].y) + (S.acc[3].x + S.acc[3].y));
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) l += __shfl_xor_sync(0xffffffffu, l, off);
    return l;
}

// The candidate buffers of a warp in its kCandBytes of shared memory.
__device__ __forceinline__ void sweep_bind(Sweep& S, uint8_t* cand) {
    S.cu = reinterpret_cast<int*>(cand);
    S.fv = reinterpret_cast<float*>(cand + kCoarseCap * 4);
    S.fc = reinterpret_cast<int*>(cand + kCoarseCap * 4 + kFineCap * 4);
}

// The staged kernel.  Warp w of CTA c takes rows c * kStagedWarps + w, then that plus the
// number of warps in the grid, and so on; `ring` buffers of `pitch4` float4 per warp, then a
// candidate buffer per warp.  Every wait is bounded: a warp that gives up records
// FA_ERR_TIMEOUT in *status, waits (bounded) for the copies it still has in flight and leaves.
__global__ void __launch_bounds__(kStagedWarps * 32)
    topk_staged_rows(const float* __restrict__ x, long long rows, int cols, int k,
                     float* __restrict__ vals, int* __restrict__ idx, float* __restrict__ lse,
                     int ring, int pitch4, int* status, unsigned long long timeout_ns) {
    extern __shared__ __align__(128) float4 staged_smem[];
    __shared__ uint64_t bars[kStagedWarps][kStagedMaxRing];
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const long long row_f4 = static_cast<long long>(ring) * pitch4;  // per warp
    float4* buf = staged_smem + warp * row_f4;
    uint8_t* cand = reinterpret_cast<uint8_t*>(staged_smem + kStagedWarps * row_f4) +
                    warp * kCandBytes;
    uint64_t* bar = bars[warp];
    const long long tw = static_cast<long long>(gridDim.x) * kStagedWarps;
    const long long r0 = static_cast<long long>(blockIdx.x) * kStagedWarps + warp;
    const int n4 = cols >> 2;
    if (lane == 0) {
        for (int b = 0; b < ring; ++b) mbar_init(&bar[b], 1);
        fence_mbar_init();
        for (int b = 0; b < ring; ++b)
            if (r0 + b * tw < rows) staged_issue(buf + b * pitch4, x, r0 + b * tw, cols, &bar[b]);
    }
    __syncwarp();
    int i = 0;
    for (long long r = r0; r < rows; r += tw, ++i) {
        const int b = i % ring;
        if (!__all_sync(0xffffffffu, mbar_wait(&bar[b], (i / ring) & 1, timeout_ns))) {
            if (lane == 0) {
                atomicCAS(status, 0, FA_ERR_TIMEOUT | (40 << 8));
                const unsigned long long drain =
                    timeout_ns > kStagedDrainNs ? timeout_ns : kStagedDrainNs;
                for (int j = i; j < i + ring && r0 + j * tw < rows; ++j)
                    mbar_wait(&bar[j % ring], (j / ring) & 1, drain);
            }
            return;
        }
        Sweep S;
        sweep_bind(S, cand);
        S.floor = -INFINITY;
        float m = -INFINITY;
        sweep_segment(buf + b * pitch4, n4, k, S, m);
        // Every lane has read buffer b: it may take row r + ring * tw.  The generic-proxy
        // reads are ordered before the bulk copy's writes by the fence.
        __syncwarp();
        if (lane == 0 && r + ring * tw < rows) {
            fence_proxy_async_smem();
            staged_issue(buf + b * pitch4, x, r + ring * tw, cols, &bar[b]);
        }
        sweep_finish(S);
        const float l = sweep_sum(S);
        const float mu = m == -INFINITY ? 0.f : m;
        if (lse && lane == 0) lse[r] = m + logf(l);
        if (lane < k) {
            vals[r * k + lane] = ex2a((S.lv - mu) * kLog2e) * (l > 0.f ? 1.f / l : 0.f);
            idx[r * k + lane] = S.lc;
        }
    }
}

// Rows longer than kStagedMaxCols (16-byte access, k >= 2): each row is cut into segments of
// kSegCols columns, staged like the short rows, and the W warps of a CTA share a row: warp w
// takes segments w, w + W, ... and carries its running floor, bar, list and (m, l) across
// them.  At the end of the row the warps' states meet in shared memory: warp 0 merges the
// lists (merge_batch) and the (m, l) pairs (the two-worker merge) and writes the row.  A CTA
// takes rows blockIdx.x, blockIdx.x + gridDim.x, ...  W is chosen per launch so that the rows
// fill the SMs in as few segment times as possible.
constexpr int kSegCols = 4096;
constexpr int kLongMaxWarps = 8;

__global__ void __launch_bounds__(kLongMaxWarps * 32)
    topk_staged_long(const float* __restrict__ x, long long rows, int cols, int k,
                     float* __restrict__ vals, int* __restrict__ idx, float* __restrict__ lse,
                     int ring, int* status, unsigned long long timeout_ns) {
    extern __shared__ __align__(128) float4 long_smem[];
    __shared__ uint64_t bars[kLongMaxWarps][kStagedMaxRing];
    __shared__ float xv[2][kLongMaxWarps][32];  // [row parity][warp][list entry]
    __shared__ int xc[2][kLongMaxWarps][32];
    __shared__ float xm[2][kLongMaxWarps], xl[2][kLongMaxWarps];
    constexpr int kSeg4 = kSegCols / 4;
    const int W = blockDim.x >> 5;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    float4* buf = long_smem + static_cast<long long>(warp) * ring * kSeg4;
    uint8_t* cand = reinterpret_cast<uint8_t*>(long_smem + static_cast<long long>(W) * ring * kSeg4) +
                    warp * kCandBytes;
    uint64_t* bar = bars[warp];
    const int nseg = (cols + kSegCols - 1) / kSegCols;
    const int spw = (nseg + W - 1) / W;  // segment slots of a warp per row (some past nseg)
    const long long my_rows =
        rows > blockIdx.x ? (rows - 1 - blockIdx.x) / gridDim.x + 1 : 0;
    const long long n_items = my_rows * spw;
    // Lane 0 issues the copies: item i is segment warp + (i % spw) W of the CTA's row i / spw
    // (no copy past the last segment); copy number c goes to buffer c % ring.
    long long next_item = 0;
    int issued = 0;
    auto issue_upto = [&](int limit) {
        while (issued < limit && next_item < n_items) {
            const int sg = warp + static_cast<int>(next_item % spw) * W;
            if (sg < nseg) {
                const long long row = blockIdx.x + (next_item / spw) * gridDim.x;
                const int c0 = sg * kSegCols;
                const uint32_t bytes = static_cast<uint32_t>(min(kSegCols, cols - c0)) * 4u;
                const int b = issued % ring;
                mbar_arrive_expect_tx(&bar[b], bytes);
                bulk_load(buf + b * kSeg4, x + row * cols + c0, bytes, &bar[b]);
                ++issued;
            }
            ++next_item;
        }
    };
    if (lane == 0) {
        for (int b = 0; b < ring; ++b) mbar_init(&bar[b], 1);
        fence_mbar_init();
        issue_upto(ring);
    }
    __syncwarp();
    int consumed = 0;   // copies this warp has waited for
    bool dead = false;  // a wait gave up: no more waits or copies, but every barrier is kept
    for (long long ri = 0; ri < my_rows; ++ri) {
        const long long r = blockIdx.x + ri * gridDim.x;
        const int par = static_cast<int>(ri & 1);
        Sweep S;
        sweep_bind(S, cand);
        S.floor = -INFINITY;
        float m = -INFINITY;
        for (int j = 0; j < spw && !dead; ++j) {
            const int sg = warp + j * W;
            if (sg >= nseg) break;
            const int b = consumed % ring;
            if (!__all_sync(0xffffffffu,
                            mbar_wait(&bar[b], (consumed / ring) & 1, timeout_ns))) {
                if (lane == 0) atomicCAS(status, 0, FA_ERR_TIMEOUT | (41 << 8));
                dead = true;
                break;
            }
            S.col0 = sg * kSegCols;
            sweep_segment(buf + b * kSeg4, (min(kSegCols, cols - sg * kSegCols)) >> 2, k, S, m);
            ++consumed;
            // every lane has read the buffer: it may take the next copy
            __syncwarp();
            if (lane == 0) {
                fence_proxy_async_smem();
                issue_upto(consumed + ring);
            }
        }
        sweep_finish(S);
        const float l = sweep_sum(S);
        xv[par][warp][lane] = S.lv;
        xc[par][warp][lane] = S.lc;
        if (lane == 0) {
            xm[par][warp] = m;
            xl[par][warp] = l;
        }
        // The slots of this parity were last read for row ri - 2, before warp 0 arrived here
        // for row ri - 1, so one barrier per row keeps writers and the reader apart.
        named_bar_sync(1, blockDim.x);
        if (warp == 0) {
            float M = -INFINITY;
            for (int w = 0; w < W; ++w) M = fmaxf(M, xm[par][w]);
            float L = 0.f;
            for (int w = 0; w < W; ++w)
                if (xm[par][w] != -INFINITY) L += xl[par][w] * ex2a((xm[par][w] - M) * kLog2e);
            float lv = S.lv;
            int lc = S.lc;
            for (int w = 1; w < W; ++w) merge_batch(lv, lc, xv[par][w][lane], xc[par][w][lane]);
            const float mu = M == -INFINITY ? 0.f : M;
            if (lse && lane == 0) lse[r] = M + logf(L);
            if (lane < k) {
                vals[r * k + lane] = ex2a((lv - mu) * kLog2e) * (L > 0.f ? 1.f / L : 0.f);
                idx[r * k + lane] = lc;
            }
        }
    }
    // Copies still in flight (only after a wait gave up) end before the CTA leaves.
    if (lane == 0) {
        const unsigned long long drain = timeout_ns > kStagedDrainNs ? timeout_ns : kStagedDrainNs;
        for (int c = consumed; c < issued; ++c) mbar_wait(&bar[c % ring], (c / ring) & 1, drain);
    }
}

template <bool VEC, class Top>
__global__ void __launch_bounds__(kThreads) topk_warp_rows(const float* __restrict__ x,
                                                           long long rows, int cols, int k,
                                                           float* __restrict__ vals,
                                                           int* __restrict__ idx,
                                                           float* __restrict__ lse) {
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    for (long long r = static_cast<long long>(blockIdx.x) * kWarps + warp; r < rows;
         r += static_cast<long long>(gridDim.x) * kWarps) {
        Stat st{-INFINITY, 0.f};
        Top top;
        if constexpr (kFiltered<Top>) {
            const int n = VEC ? cols >> 2 : cols;
            stats_pass<VEC>(x + r * cols, 0, n, lane, 32, st);
            select_pass<VEC>(x + r * cols, 0, n, lane, 32, k, warp_kth_largest(st.m, k), top);
        } else {
            scan<VEC>(x + r * cols, cols, lane, 32, k, st, top);
        }
        top.finish();
        st = warp_merge(st);
        if (lse && lane == 0) lse[r] = st.m + logf(st.l);
        write_top(top, k, st, vals + r * k, idx + r * k);
    }
}

template <bool VEC, class Top>
__global__ void __launch_bounds__(kThreads) topk_cta_rows(const float* __restrict__ x,
                                                          long long rows, int cols, int k,
                                                          float* __restrict__ vals,
                                                          int* __restrict__ idx,
                                                          float* __restrict__ lse) {
    __shared__ float cv[kWarps][32];
    __shared__ int cc[kWarps][32];
    __shared__ Stat cs[kWarps];
    __shared__ float cf[kWarps];
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    for (long long r = blockIdx.x; r < rows; r += gridDim.x) {
        Stat st{-INFINITY, 0.f};
        Top top;
        if constexpr (kFiltered<Top>) {
            const int n = VEC ? cols >> 2 : cols;
            stats_pass<VEC>(x + r * cols, 0, n, threadIdx.x, kThreads, st);
            // each warp's floor holds for the whole row; the largest is the tightest
            const float f = warp_kth_largest(st.m, k);
            if (lane == 0) cf[warp] = f;
            __syncthreads();
            float floor = cf[0];
#pragma unroll
            for (int w = 1; w < kWarps; ++w) floor = fmaxf(floor, cf[w]);
            select_pass<VEC>(x + r * cols, 0, n, threadIdx.x, kThreads, k, floor, top);
        } else {
            scan<VEC>(x + r * cols, cols, threadIdx.x, kThreads, k, st, top);
        }
        top.finish();
        st = warp_merge(st);
        cv[warp][lane] = top.v;
        cc[warp][lane] = top.c;
        if (lane == 0) cs[warp] = st;
        __syncthreads();
        if (warp == 0) {
            Stat s = lane < kWarps ? cs[lane] : Stat{-INFINITY, 0.f};
            s = warp_merge(s);
            if (lse && lane == 0) lse[r] = s.m + logf(s.l);
            // The other warps' lists enter warp 0's list, one warp's list per step.
            for (int w = 1; w < kWarps; ++w) {
                const float v[1] = {cv[w][lane]};
                const int col[1] = {cc[w][lane]};
                top.offer(v, col, k);
            }
            top.finish();
            write_top(top, k, s, vals + r * k, idx + r * k);
        }
        __syncthreads();  // the shared lists are refilled for the next row
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

// The staged kernel: CTAs of four warps, each warp with one to kStagedMaxRing row buffers, as
// many CTAs per SM as fit.
int launch_staged(const float* x, long long rows, int cols, int k, float* vals, int* idx,
                  float* lse, cudaStream_t stream) {
    constexpr int kSmemCap = 100 * 1024;  // above any request below
    static cudaError_t attr = cudaSuccess;
    static std::once_flag once;
    std::call_once(once, [] {
        attr = cudaFuncSetAttribute(topk_staged_rows, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                    kSmemCap);
    });
    if (attr != cudaSuccess) return FA_ERR_CUDA;
    int* status = device_status_word();
    if (!status) return FA_ERR_CUDA;
    const int pitch4 = ((cols >> 2) + 7) & ~7;  // float4 per buffer: 128-byte multiples
    const int buf_bytes = pitch4 * 16;
    // Row buffers: as many (up to kStagedMaxRing) as leave room for four CTAs (16 warps) per SM
    // in 228 KB; at least one (the longest rows: three CTAs).
    int ring = (228 * 1024 / 16 - kCandBytes - 512) / buf_bytes;
    ring = ring < 1 ? 1 : (ring > kStagedMaxRing ? kStagedMaxRing : ring);
    const int smem = kStagedWarps * (ring * buf_bytes + kCandBytes);
    int per_sm = 0;
    if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, topk_staged_rows,
                                                      kStagedWarps * 32, smem) != cudaSuccess)
        return FA_ERR_CUDA;
    if (per_sm < 1) per_sm = 1;
    const long long sms = sm_count() > 0 ? sm_count() : 148;
    long long grid = (rows + kStagedWarps - 1) / kStagedWarps;
    if (grid > sms * per_sm) grid = sms * per_sm;
    topk_staged_rows<<<static_cast<unsigned>(grid), kStagedWarps * 32, smem, stream>>>(
        x, rows, cols, k, vals, idx, lse, ring, pitch4, status, fa_wait_timeout_ns());
    return cudaGetLastError() == cudaSuccess ? FA_OK : FA_ERR_CUDA;
}

// The long-row kernel: one segment buffer per warp; the CTA width W (1 to kLongMaxWarps) with
// the fewest segment times, ceil(rows / resident CTAs) x ceil(segments / W), the narrowest on
// ties.
int launch_long(const float* x, long long rows, int cols, int k, float* vals, int* idx,
                float* lse, cudaStream_t stream) {
    constexpr int kRing = 1;
    constexpr int kWarpBytes = kRing * kSegCols * 4 + kCandBytes;
    static cudaError_t attr = cudaSuccess;
    static std::once_flag once;
    std::call_once(once, [] {
        attr = cudaFuncSetAttribute(topk_staged_long, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                    kLongMaxWarps * kWarpBytes);
    });
    if (attr != cudaSuccess) return FA_ERR_CUDA;
    int* status = device_status_word();
    if (!status) return FA_ERR_CUDA;
    const long long sms = sm_count() > 0 ? sm_count() : 148;
    const long long nseg = (cols + kSegCols - 1) / kSegCols;
    int best_w = 1;
    long long best_cost = -1, best_grid = 1;
    for (int w = 1; w <= kLongMaxWarps; ++w) {
        int per_sm = 0;
        if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, topk_staged_long, w * 32,
                                                          w * kWarpBytes) != cudaSuccess)
            return FA_ERR_CUDA;
        if (per_sm < 1) continue;
        const long long slots = sms * per_sm;
        const long long cost = ((rows + slots - 1) / slots) * ((nseg + w - 1) / w);
        if (best_cost < 0 || cost < best_cost) {
            best_cost = cost;
            best_w = w;
            best_grid = rows < slots ? rows : slots;
        }
    }
    if (best_cost < 0) return FA_ERR_CUDA;
    topk_staged_long<<<static_cast<unsigned>(best_grid), best_w * 32, best_w * kWarpBytes,
                       stream>>>(x, rows, cols, k, vals, idx, lse, kRing, status,
                                 fa_wait_timeout_ns());
    return cudaGetLastError() == cudaSuccess ? FA_OK : FA_ERR_CUDA;
}

template <class Top>
int launch(const float* x, long long rows, int cols, int k, float* vals, int* idx, float* lse,
           cudaStream_t stream) {
    const bool vec = (cols % 4 == 0) && (reinterpret_cast<uintptr_t>(x) % 16 == 0);
    const long long sms = sm_count() > 0 ? sm_count() : 148;
    // k >= 2 with 16-byte access: the staged kernels (the register kernels' vector forms for
    // k >= 2 are not built).
    if constexpr (kFiltered<Top>) {
        if (vec)
            return cols <= kStagedMaxCols
                       ? launch_staged(x, rows, cols, k, vals, idx, lse, stream)
                       : launch_long(x, rows, cols, k, vals, idx, lse, stream);
    }
    if (cols <= 4096) {
        long long grid = (rows + kWarps - 1) / kWarps;
        if (grid > sms * 8) grid = sms * 8;
        if constexpr (!kFiltered<Top>) {
            if (vec) {
                topk_warp_rows<true, Top><<<static_cast<unsigned>(grid), kThreads, 0, stream>>>(
                    x, rows, cols, k, vals, idx, lse);
                return cudaGetLastError() == cudaSuccess ? FA_OK : FA_ERR_CUDA;
            }
        }
        topk_warp_rows<false, Top><<<static_cast<unsigned>(grid), kThreads, 0, stream>>>(
            x, rows, cols, k, vals, idx, lse);
    } else {
        long long grid = rows;
        if (grid > sms * 8) grid = sms * 8;
        if constexpr (!kFiltered<Top>) {
            if (vec) {
                topk_cta_rows<true, Top><<<static_cast<unsigned>(grid), kThreads, 0, stream>>>(
                    x, rows, cols, k, vals, idx, lse);
                return cudaGetLastError() == cudaSuccess ? FA_OK : FA_ERR_CUDA;
            }
        }
        topk_cta_rows<false, Top><<<static_cast<unsigned>(grid), kThreads, 0, stream>>>(
            x, rows, cols, k, vals, idx, lse);
    }
    return cudaGetLastError() == cudaSuccess ? FA_OK : FA_ERR_CUDA;
}

// --------------------------------------------------------------------------------------------
// k > 32: a floor, candidates in shared memory, one CTA per row
// --------------------------------------------------------------------------------------------
// For k beyond the warp-wide list, a CTA of T threads (256 or 512) takes a row:
//   * each thread carries its online (m, l) of "The idea" and the Q largest values it has seen
//     (Q = 1, 2 or 4, the fewest with T * Q >= 2k).  Any thread whose Q-th largest is at least
//     F has Q entries of the row at or above F; so the ceil(k / Q)-th largest of the threads'
//     Q-th largest values is a floor F under the k-th largest value of the row (a bitonic
//     network over the CTA's T values picks it), and so is the smallest over the warps of a
//     warp's c-th largest lane value when the warps' c add up to ceil(k / Q);
//   * the row's first 64 T columns are read twice: once for (m, l) and the Q largest, which
//     give the first F, and once more (from L2) to append every entry at or above F to a
//     candidate buffer in shared memory (a warp reserves its slots with one atomic);
//   * the rest of the row is read once: every value is offered against the thread's F, then
//     enters (m, l) and the Q largest, and each warp renews its F from the published warp
//     floors as it goes.  F only rises, so an entry at or above a later floor was at or above
//     the floor it was offered against: the buffer holds every entry seen so far at or above
//     any floor in use, the whole top k with the ties at the k-th value.  Entries below the
//     floor are dropped when the buffer is half full.
// At the end of the row the (m, l) pairs meet by the two-worker merge, the final F (from all of
// the row's values, at or above every floor used before) drops the rest, the buffer is sorted
// (larger value first, then the smaller column) and its first k entries are the row's top k.
// A row that overflowed the buffer is read once more against the final F.
// Rows where more than 16 T entries reach the final floor (many ties at it, or fewer than k
// finite values) take the exact route instead: radix selection of the k-th largest on an
// order-preserving 32-bit key, eight bits per pass over the row, then a pass in column order
// that keeps the entries above it and the first of the entries equal to it.
constexpr int kSelMaxK = 1024;
// A CTA of T threads keeps 16 T candidate entries (value, column) in shared memory.
template <int T>
struct SelCfg {
    static constexpr int kWarps = T / 32;
    static constexpr int kCap = 16 * T;
    static constexpr int kSmem = kCap * 8;
};

// Larger value -> larger key, equal values (-0 and +0 included) -> equal keys; NaN is outside
// the contract.
__device__ __forceinline__ uint32_t order_key(float v) {
    uint32_t b = __float_as_uint(v);
    if (b == 0x80000000u) b = 0u;  // -0 ranks as +0: the tie rule decides between them
    return (b & 0x80000000u) ? ~b : (b | 0x80000000u);
}

// The digit of the k-th largest among the counts hist[0..255] (from the top), and how many of
// the entries to count from it are still to be taken: on entry `need` entries are wanted, on
// return need - (count of the larger digits).  Thread 0 only.
__device__ __forceinline__ int pick_digit(const unsigned* hist, unsigned& need) {
    unsigned acc = 0;
    for (int dgt = 255; dgt >= 0; --dgt) {
        if (acc + hist[dgt] >= need) {
            need -= acc;
            return dgt;
        }
        acc += hist[dgt];
    }
    return 0;  // not reached: the counts of a pass sum to at least `need`
}

// Bitonic sort of n (a power of two, up to SelCfg<T>::kCap) pairs in shared memory, best first
// (larger value, then the smaller column).  Every thread of the CTA calls it.
template <int T>
__device__ __forceinline__ void sort_pairs(float* sv, int* si, int n) {
    const int t = threadIdx.x;
    for (int size = 2; size <= n; size <<= 1) {
        for (int stride = size >> 1; stride > 0; stride >>= 1) {
            for (int i = t; i < n; i += T) {
                const int j = i ^ stride;
                if (j > i) {
                    const bool up = (i & size) == 0;  // this block ascends in rank
                    if (before(sv[j], si[j], sv[i], si[i]) == up) {
                        const float tv = sv[i];
                        sv[i] = sv[j];
                        sv[j] = tv;
                        const int ti = si[i];
                        si[i] = si[j];
                        si[j] = ti;
                    }
                }
            }
            __syncthreads();
        }
    }
}

// Exclusive prefix sum over the CTA of one count per thread; *total gets the sum.  Uses
// scratch[SelCfg<T>::kWarps]; every thread calls it.
template <int T>
__device__ __forceinline__ unsigned cta_exclusive_scan(unsigned v, unsigned* scratch,
                                                       unsigned* total) {
    const int lane = threadIdx.x & 31, wid = threadIdx.x >> 5;
    unsigned inc = v;
#pragma unroll
    for (int off = 1; off < 32; off <<= 1) {
        const unsigned o = __shfl_up_sync(0xffffffffu, inc, off);
        if (lane >= off) inc += o;
    }
    if (lane == 31) scratch[wid] = inc;
    __syncthreads();
    unsigned base = 0, all = 0;
#pragma unroll
    for (int w = 0; w < SelCfg<T>::kWarps; ++w) {
        const unsigned c = scratch[w];
        base += w < wid ? c : 0u;
        all += c;
    }
    *total = all;
    __syncthreads();  // scratch is free again
    return base + inc - v;
}

// Keeps the first n buffer entries at or above f (in some order); returns their count.
template <int T>
__device__ __forceinline__ unsigned drop_below(float* sv, int* si, unsigned n, float f,
                                               unsigned* scratch) {
    constexpr int kPer = SelCfg<T>::kCap / T;
    const int t = threadIdx.x;
    float v[kPer];
    int c[kPer];
    unsigned keep = 0;
#pragma unroll
    for (int e = 0; e < kPer; ++e) {
        const unsigned i = static_cast<unsigned>(e * T + t);
        v[e] = i < n ? sv[i] : -INFINITY;
        c[e] = i < n ? si[i] : 0;
        keep += (i < n && v[e] >= f) ? 1u : 0u;
    }
    unsigned total;
    unsigned pos = cta_exclusive_scan<T>(keep, scratch, &total);  // all reads done (barrier)
#pragma unroll
    for (int e = 0; e < kPer; ++e) {
        const unsigned i = static_cast<unsigned>(e * T + t);
        if (i < n && v[e] >= f) {
            sv[pos] = v[e];
            si[pos] = c[e];
            ++pos;
        }
    }
    __syncthreads();
    return total;
}

template <int T>
struct SelShared {
    float xv[2][T];  // exchange buffers of cta_sort_desc
    int xc[2][T];
    float floor;
    unsigned hist[256];
    unsigned scratch[SelCfg<T>::kWarps];
    unsigned warp_ties[SelCfg<T>::kWarps];
    float red_m[SelCfg<T>::kWarps], red_l[SelCfg<T>::kWarps];
    float wfloor[SelCfg<T>::kWarps];  // each warp's last published floor
    unsigned count, prefix, need, ties;
    int overflow;
};

// Bitonic sort of one (value, column) pair per thread over the CTA, best first: thread i ends
// with the (i+1)-th best pair.  Partners less than a warp apart trade by shuffles; the others
// through two alternating shared buffers, one barrier per such step.
template <int T>
__device__ __forceinline__ void cta_sort_desc(float& v, int& c, SelShared<T>& sh) {
    const int i = threadIdx.x;
    int buf = 0;
    for (int size = 2; size <= T; size <<= 1) {
        for (int stride = size >> 1; stride > 0; stride >>= 1) {
            float ov;
            int oc;
            if (stride >= 32) {
                sh.xv[buf][i] = v;
                sh.xc[buf][i] = c;
                __syncthreads();
                ov = sh.xv[buf][i ^ stride];
                oc = sh.xc[buf][i ^ stride];
                buf ^= 1;
            } else {
                ov = __shfl_xor_sync(0xffffffffu, v, stride);
                oc = __shfl_xor_sync(0xffffffffu, c, stride);
            }
            // a block with (i & size) == 0 ends best first: its lower half keeps the better
            const bool keep_better = ((i & stride) == 0) == ((i & size) == 0);
            if (keep_better ? before(ov, oc, v, c) : before(v, c, ov, oc)) {
                v = ov;
                c = oc;
            }
        }
    }
}

// The exact route: the k entries of the row (in some order) into sv/si, by radix selection.
template <int T>
__device__ void select_exact(const float* __restrict__ xr, int cols, int k, float* sv, int* si,
                             SelShared<T>& sh) {
    const int t = threadIdx.x, lane = t & 31, wid = t >> 5;
    if (t == 0) {
        sh.prefix = 0u;
        sh.need = static_cast<unsigned>(k);
    }
    for (int shift = 24; shift >= 0; shift -= 8) {
        for (int i = t; i < 256; i += T) sh.hist[i] = 0u;
        __syncthreads();
        const unsigned prefix = sh.prefix;
        for (int c = t; c < cols; c += T) {
            const uint32_t key = order_key(xr[c]);
            if (shift == 24 || (key >> (shift + 8)) == prefix)
                atomicAdd(&sh.hist[(key >> shift) & 0xffu], 1u);
        }
        __syncthreads();
        if (t == 0) {
            unsigned need = sh.need;
            sh.prefix = (prefix << 8) | static_cast<unsigned>(pick_digit(sh.hist, need));
            sh.need = need;
        }
        __syncthreads();
    }
    // sh.prefix is the k-th largest key: every entry above it is kept, and the first sh.need
    // (by column) of the entries equal to it.
    const uint32_t kth = sh.prefix;
    const unsigned ties_wanted = sh.need;
    if (t == 0) {
        sh.count = 0u;
        sh.ties = 0u;
    }
    __syncthreads();
    for (int c0 = 0; c0 < cols; c0 += T) {
        const int c = c0 + t;
        const float v = c < cols ? xr[c] : 0.f;
        const uint32_t key = c < cols ? order_key(v) : 0u;
        if (c < cols && key > kth) {
            const unsigned slot = atomicAdd(&sh.count, 1u);
            sv[slot] = v;
            si[slot] = c;
        }
        const bool tie = c < cols && key == kth;
        const unsigned b = __ballot_sync(0xffffffffu, tie);
        if (lane == 0) sh.warp_ties[wid] = __popc(b);
        __syncthreads();
        unsigned before_me = sh.ties;  // ties in the chunks before this one
        for (int w = 0; w < wid; ++w) before_me += sh.warp_ties[w];
        before_me += __popc(b & ((1u << lane) - 1u));
        if (tie && before_me < ties_wanted) {
            const unsigned slot = atomicAdd(&sh.count, 1u);
            sv[slot] = v;
            si[slot] = c;
        }
        __syncthreads();
        if (t == 0) {
            unsigned all = 0;
            for (int w = 0; w < SelCfg<T>::kWarps; ++w) all += sh.warp_ties[w];
            sh.ties += all;
        }
        __syncthreads();
    }
}

template <int Q>
__device__ __forceinline__ void keep_largest(float (&b)[Q], float v) {
    if (v > b[Q - 1]) {
#pragma unroll
        for (int i = Q - 1; i > 0; --i) b[i] = v > b[i - 1] ? b[i - 1] : fmaxf(b[i], v);
        b[0] = fmaxf(b[0], v);
    }
}

// A step of the sweep over a row: each thread takes kN values (four float4 in the vector form,
// four floats otherwise).  The first kHead steps of a row (64 T columns) take two passes (the
// second from L2), which set the first floor; a warp renews its floor every kRefresh later
// steps (16384 columns), and every kCheck steps (128 T columns) the CTA meets to drop buffer
// entries below the floor once the buffer is half full.  Measured on 512 rows of 131072
// columns: renewing every 8192 columns made k = 100 and k = 33 1.5 and 2.6 % slower (the warp
// sort's cost), every 32768 made k = 1024 (512 threads) 21 % slower (the buffer overflowed).
template <int T, bool VEC>
struct SelStep {
    static constexpr int kN = VEC ? 16 : 4;
    static constexpr int kCols = kN * T;
    static constexpr int kHead = 64 * T / kCols;
    static constexpr int kRefresh = 16384 / kCols;
    static constexpr int kCheck = 128 * T / kCols;
};

// Thread t's values of the step that starts at column `base` (a multiple of 4 in the vector
// form); columns at or past c1 read as -inf.
template <int T, bool VEC>
__device__ __forceinline__ void load_step(const float* __restrict__ xr, int base, int c1,
                                          float (&v)[SelStep<T, VEC>::kN]) {
    const int t = threadIdx.x;
    if constexpr (VEC) {
        const float4* r4 = reinterpret_cast<const float4*>(xr);
        const int u1 = c1 >> 2;
#pragma unroll
        for (int a = 0; a < SelStep<T, VEC>::kN / 4; ++a) {
            const int u = (base >> 2) + a * T + t;
            const float4 q = u < u1 ? __ldg(r4 + u)
                                    : make_float4(-INFINITY, -INFINITY, -INFINITY, -INFINITY);
            v[4 * a] = q.x;
            v[4 * a + 1] = q.y;
            v[4 * a + 2] = q.z;
            v[4 * a + 3] = q.w;
        }
    } else {
#pragma unroll
        for (int a = 0; a < 4; ++a) {
            const int j = base + a * T + t;
            v[a] = j < c1 ? __ldg(xr + j) : -INFINITY;
        }
    }
}

// The column of value e of thread t's share of the step at `base`.
template <int T, bool VEC>
__device__ __forceinline__ int step_col(int base, int e) {
    if constexpr (VEC) return 4 * ((base >> 2) + (e >> 2) * T + static_cast<int>(threadIdx.x)) + (e & 3);
    return base + e * T + static_cast<int>(threadIdx.x);
}

// The largest of a step's values (a tree of pairwise maxima).
template <int N>
__device__ __forceinline__ float step_max(const float (&v)[N]) {
    float w[N / 2];
#pragma unroll
    for (int e = 0; e < N / 2; ++e) w[e] = fmaxf(v[2 * e], v[2 * e + 1]);
#pragma unroll
    for (int n = N / 2; n > 1; n >>= 1) {
#pragma unroll
        for (int e = 0; e < n / 2; ++e) w[e] = fmaxf(w[2 * e], w[2 * e + 1]);
    }
    return w[0];
}

// A step's values (largest mx) enter (m, l) and the thread's Q largest.  exp(x - m) in packed
// pairs, x - m first, then the scale; l is rescaled by exp(m_old - m_new) only when the running
// max grows (from -inf: the old l, 0, stays 0).
template <int Q, int N>
__device__ __forceinline__ void take_step(Stat& s, float (&best)[Q], const float (&v)[N],
                                          float mx) {
    const float m = fmaxf(s.m, mx);
    if (m != -INFINITY) {  // else nothing finite yet: adds nothing
        float l = s.l;
        if (m != s.m) l *= ex2a((s.m - m) * kLog2e);
        const float2 nm = make_float2(-m, -m), c2 = make_float2(kLog2e, kLog2e);
        float2 acc = make_float2(0.f, 0.f);
#pragma unroll
        for (int e = 0; e < N; e += 2) {
            const float2 d = fmul2(fadd2(make_float2(v[e], v[e + 1]), nm), c2);
            acc = fadd2(acc, make_float2(ex2a(d.x), ex2a(d.y)));
        }
        s = Stat{m, l + (acc.x + acc.y)};
    }
    if constexpr (Q == 1) {
        best[0] = fmaxf(best[0], mx);
    } else if (mx > best[Q - 1]) {
#pragma unroll
        for (int e = 0; e < N; ++e) keep_largest(best, v[e]);
    }
}

// The values of a step (columns below c1) at or above f enter the buffer, four at a time: a
// vote on the four's largest value, then a ballot per value and one atomic per warp for the
// slots.  Entries past SelCfg<T>::kCap are not stored and mark the row overflowed.
template <int T, bool VEC>
__device__ __forceinline__ void offer_step(const float (&v)[SelStep<T, VEC>::kN], int base,
                                           int c1, float f, float* sv, int* si,
                                           SelShared<T>& sh) {
    const unsigned lt = (1u << (threadIdx.x & 31)) - 1u;
#pragma unroll
    for (int g = 0; g < SelStep<T, VEC>::kN; g += 4) {
        const float gm = fmaxf(fmaxf(v[g], v[g + 1]), fmaxf(v[g + 2], v[g + 3]));
        if (!__any_sync(0xffffffffu, gm >= f)) continue;
        bool p[4];
        unsigned bal[4];
        unsigned total = 0;
#pragma unroll
        for (int e = 0; e < 4; ++e) {
            p[e] = step_col<T, VEC>(base, g + e) < c1 && v[g + e] >= f;
            bal[e] = __ballot_sync(0xffffffffu, p[e]);
            total += __popc(bal[e]);
        }
        unsigned slot = 0;
        if ((threadIdx.x & 31) == 0) slot = atomicAdd(&sh.count, total);
        slot = __shfl_sync(0xffffffffu, slot, 0);
#pragma unroll
        for (int e = 0; e < 4; ++e) {
            if (p[e]) {
                const unsigned pos = slot + __popc(bal[e] & lt);
                if (pos < SelCfg<T>::kCap) {
                    sv[pos] = v[g + e];
                    si[pos] = step_col<T, VEC>(base, g + e);
                } else {
                    sh.overflow = 1;
                }
            }
            slot += __popc(bal[e]);
        }
    }
}

// The ceil(k / Q)-th largest of the threads' Q-th largest values: a floor under the k-th
// largest value of the row (every thread gets it; the CTA meets).
template <int T>
__device__ __forceinline__ float cta_floor(float bar, int r_bar, SelShared<T>& sh) {
    int bc = static_cast<int>(threadIdx.x);
    cta_sort_desc<T>(bar, bc, sh);
    if (static_cast<int>(threadIdx.x) == r_bar - 1) sh.floor = bar;
    __syncthreads();
    return sh.floor;
}

template <int T, int Q, bool VEC>
__global__ void __launch_bounds__(T, 1024 / T)
    topk_select_rows(const float* __restrict__ x, long long rows, int cols, int k,
                     float* __restrict__ vals, int32_t* __restrict__ idx,
                     float* __restrict__ lse) {
    using S = SelStep<T, VEC>;
    constexpr int N = S::kN;
    constexpr int W = SelCfg<T>::kWarps;
    extern __shared__ __align__(16) unsigned char sel_smem[];
    float* sv = reinterpret_cast<float*>(sel_smem);
    int* si = reinterpret_cast<int*>(sel_smem + SelCfg<T>::kCap * 4);
    __shared__ SelShared<T> sh;
    volatile float* wfloor = sh.wfloor;
    const int t = threadIdx.x, lane = t & 31, wid = t >> 5;
    const int r_bar = (k + Q - 1) / Q;     // the floor is the r_bar-th largest thread bar
    const int c_w = (r_bar + W - 1) / W;   // a warp's floor: the c_w-th largest of its lane bars
    for (long long row = blockIdx.x; row < rows; row += gridDim.x) {
        const float* xr = x + row * cols;
        if (t == 0) {
            sh.count = 0u;
            sh.overflow = 0;
        }
        if (lane == 0) wfloor[wid] = -INFINITY;
        Stat st{-INFINITY, 0.f};
        float best[Q];
#pragma unroll
        for (int i = 0; i < Q; ++i) best[i] = -INFINITY;
        __syncthreads();
        // ---- the head: (m, l) and the Q largest of each thread, the floor F, then the head's
        // entries at or above F (its second read hits L2) ----
        const int h = min(cols, S::kHead * S::kCols);
        for (int base = 0; base < h; base += S::kCols) {
            float v[N];
            load_step<T, VEC>(xr, base, h, v);
            take_step(st, best, v, step_max(v));
        }
        // the first step after the head is on its way during the floor and the head's offers
        float vn[N];
        if (h < cols) load_step<T, VEC>(xr, h, cols, vn);
        float F = cta_floor<T>(best[Q - 1], r_bar, sh);
        for (int base = 0; base < h; base += S::kCols) {
            float v[N];
            load_step<T, VEC>(xr, base, h, v);
            offer_step<T, VEC>(v, base, h, F, sv, si, sh);
        }
        // ---- the rest of the row in one pass, the next step's loads in flight while a step is
        // worked: each step is offered against the floor (only when its largest value reaches
        // it), then enters (m, l) and the bars.  A warp's floor (its c_w-th largest lane bar:
        // c_w Q of its entries reach it) is published in shared memory; the smallest published
        // value is a floor for the row, since the W warps together have W c_w Q >= k entries
        // at or above it.  Bars only rise, so a stale value is a floor too, and no barrier is
        // needed. ----
        int step = 0;
        for (int base = h; base < cols; base += S::kCols) {
            float v[N];
#pragma unroll
            for (int e = 0; e < N; ++e) v[e] = vn[e];
            if (base < cols - S::kCols) load_step<T, VEC>(xr, base + S::kCols, cols, vn);
            const float mx = step_max(v);
            if (__any_sync(0xffffffffu, mx >= F)) offer_step<T, VEC>(v, base, cols, F, sv, si, sh);
            take_step(st, best, v, mx);
            ++step;
            if (step % S::kRefresh == 0) {
                const float wf = warp_kth_largest(best[Q - 1], c_w);
                if (lane == 0) wfloor[wid] = wf;
                __syncwarp();
                float f = lane < W ? wfloor[lane] : INFINITY;
#pragma unroll
                for (int off = 16; off > 0; off >>= 1)
                    f = fminf(f, __shfl_xor_sync(0xffffffffu, f, off));
                F = fmaxf(F, f);
            }
            // the trip count is the same in every thread, so every thread meets here
            if (step % S::kCheck == 0 &&
                __syncthreads_or(*reinterpret_cast<volatile unsigned*>(&sh.count) >
                                 SelCfg<T>::kCap / 2)) {
                const unsigned n_now = sh.count;
                if (n_now <= SelCfg<T>::kCap) {
                    // every thread's F is at most the final floor below
                    const unsigned kept = drop_below<T>(sv, si, n_now, F, sh.scratch);
                    if (t == 0) sh.count = kept;
                }
                __syncthreads();
            }
        }
        __syncthreads();  // every entry is in
        // ---- the final floor, from every value's bars: at or above every floor used above,
        // so the buffer holds every entry of the row at or above it ----
        F = cta_floor<T>(best[Q - 1], r_bar, sh);
        if (sh.overflow) {
            // more than the buffer reached the running floors: once more over the row against
            // the final floor
            __syncthreads();  // every thread has read the flag
            if (t == 0) {
                sh.count = 0u;
                sh.overflow = 0;
            }
            __syncthreads();
            for (int base = 0; base < cols; base += S::kCols) {
                float v[N];
                load_step<T, VEC>(xr, base, cols, v);
                offer_step<T, VEC>(v, base, cols, F, sv, si, sh);
            }
            __syncthreads();
        }
        // ---- (m, l) of the row ----
        st = warp_merge(st);
        if (lane == 0) {
            sh.red_m[wid] = st.m;
            sh.red_l[wid] = st.l;
        }
        __syncthreads();
        Stat a{sh.red_m[0], sh.red_l[0]};
        for (int w = 1; w < SelCfg<T>::kWarps; ++w) a = merge(a, Stat{sh.red_m[w], sh.red_l[w]});
        const float m = a.m, l = a.l;
        // ---- the top k: from the buffer, else by the exact route ----
        int n;
        if (sh.overflow) {
            __syncthreads();  // every thread has read the flag
            select_exact(xr, cols, k, sv, si, sh);
            n = k;
        } else {
            const unsigned total = sh.count;
            __syncthreads();  // every thread has read the count
            n = static_cast<int>(drop_below<T>(sv, si, total, F, sh.scratch));
        }
        // ---- outputs: the shares exp(x - m) / l, the columns, lse = m + ln l ----
        const float inv_l = l > 0.f ? 1.f / l : 0.f;
        if (n <= T) {
            float v = t < n ? sv[t] : -INFINITY;
            int c = t < n ? si[t] : INT_MAX;
            cta_sort_desc<T>(v, c, sh);
            if (t < k) {
                vals[row * k + t] = (m == -INFINITY) ? 0.f : ex2a((v - m) * kLog2e) * inv_l;
                idx[row * k + t] = c;
            }
        } else {
            int np = 1;
            while (np < n) np <<= 1;
            for (int i = n + t; i < np; i += T) {
                sv[i] = -INFINITY;
                si[i] = INT_MAX;
            }
            __syncthreads();
            sort_pairs<T>(sv, si, np);
            for (int i = t; i < k; i += T) {
                const float v = sv[i];
                vals[row * k + i] = (m == -INFINITY) ? 0.f : ex2a((v - m) * kLog2e) * inv_l;
                idx[row * k + i] = si[i];
            }
        }
        if (t == 0 && lse != nullptr) lse[row] = (m == -INFINITY) ? -INFINITY : m + logf(l);
        __syncthreads();
    }
}

template <int T, int Q, bool VEC>
int launch_select_q(const float* x, int64_t rows, int cols, int k, float* vals,
                    int32_t* idx, float* lse, cudaStream_t stream) {
    static int blocks_per_sm = 0;
    static cudaError_t attr = cudaSuccess;
    static std::once_flag once;
    std::call_once(once, [] {
        attr = cudaFuncSetAttribute(topk_select_rows<T, Q, VEC>,
                                    cudaFuncAttributeMaxDynamicSharedMemorySize, SelCfg<T>::kSmem);
        if (attr == cudaSuccess &&
            cudaOccupancyMaxActiveBlocksPerMultiprocessor(&blocks_per_sm, topk_select_rows<T, Q, VEC>,
                                                          T, SelCfg<T>::kSmem) != cudaSuccess)
            blocks_per_sm = 1;
    });
    if (attr != cudaSuccess) return FA_ERR_CUDA;
    const long long sms = sm_count() > 0 ? sm_count() : 148;
    long long grid = sms * (blocks_per_sm > 0 ? blocks_per_sm : 1);
    if (grid > rows) grid = rows;
    topk_select_rows<T, Q, VEC><<<static_cast<unsigned>(grid), T, SelCfg<T>::kSmem, stream>>>(
        x, rows, cols, k, vals, idx, lse);
    return cudaGetLastError() == cudaSuccess ? FA_OK : FA_ERR_CUDA;
}

// The CTA width by k: 256 threads (four CTAs per SM, whose latency-bound steps overlap) up to
// k = 256, 512 threads (two per SM, a floor from more threads' values and a buffer of 8192)
// beyond.  Measured on 512 rows of 131072 columns with the earlier form that read every row
// twice: k = 100 took 0.142 ms with 512 threads and 0.120 with 256; k = 1024 took 0.268 with
// 512 threads and 0.362 with 256 (Q = 8, 4096 entries); k = 33 took 0.113 with 256 threads and
// 0.149 with 128 (eight CTAs per SM).
constexpr int kSelSmallK = 256;

template <int T, int Q>
int launch_select_vec(bool vec, const float* x, int64_t rows, int cols, int k, float* vals,
                      int32_t* idx, float* lse, cudaStream_t stream) {
    return vec ? launch_select_q<T, Q, true>(x, rows, cols, k, vals, idx, lse, stream)
               : launch_select_q<T, Q, false>(x, rows, cols, k, vals, idx, lse, stream);
}

int launch_select(const float* x, int64_t rows, int cols, int k, float* vals, int32_t* idx,
                  float* lse, cudaStream_t stream) {
    const bool vec = (cols % 4 == 0) && (reinterpret_cast<uintptr_t>(x) % 16 == 0);
    // Q per thread: the fewest with T * Q >= 2k.
    if (k <= kSelSmallK) {
        if (2 * k <= 256) return launch_select_vec<256, 1>(vec, x, rows, cols, k, vals, idx, lse, stream);
        return launch_select_vec<256, 2>(vec, x, rows, cols, k, vals, idx, lse, stream);
    }
    if (2 * k <= 512) return launch_select_vec<512, 1>(vec, x, rows, cols, k, vals, idx, lse, stream);
    if (2 * k <= 1024) return launch_select_vec<512, 2>(vec, x, rows, cols, k, vals, idx, lse, stream);
    return launch_select_vec<512, 4>(vec, x, rows, cols, k, vals, idx, lse, stream);
}

}  // namespace

int osm_softmax_topk_launch(const float* x, int64_t rows, int64_t cols, int64_t k, float* vals,
                            int32_t* idx, float* lse, cudaStream_t stream) {
    if (cols > INT_MAX / 2 || rows > (1LL << 40)) return FA_ERR_UNSUPPORTED;
    if (k < 1 || k > kSelMaxK) return FA_ERR_UNSUPPORTED;
    const int c = static_cast<int>(cols), kk = static_cast<int>(k);
    if (k == 1) return launch<LaneBest>(x, rows, c, kk, vals, idx, lse, stream);
    if (k > 32) return launch_select(x, rows, c, kk, vals, idx, lse, stream);
    return launch<WarpTop>(x, rows, c, kk, vals, idx, lse, stream);
}

}  // namespace osm
