// device_plan.cuh -- the device plan of paged decode (PKV_DECODE_DEVICE_PLAN):
// every CTA of phase 1 plans from the device's context lengths itself, so that
// a call captured into a CUDA graph with capacity bounds launches phase 1 over
// the actual work only, with no planning kernel in front of it.
//
// Plan: the rule of the host planner (api.cu, auto_partition) applied to the
// actual longest context max_n and total sum_n -- P starts at P0 (or max_n
// rounded up to a page, if shorter) and halves while HR_rule * ceil(sum_n / P)
// (the description's KV heads x row tiles) is below six items per SM, down to
// four pages -- then raised, if needed, to ceil(max_n / NS_cap) rounded up to
// a page so that no sequence has more splits than the workspace holds.
// Items: sequence b has ns_b = max(1, ceil(n_b / P)) splits (one item writes
// the zero rows of an empty context) for each of its HR (grid KV head, row
// tile) pairs -- a grid KV head is a pair of KV heads when the CTAs take two
// -- in the order (b, split, KV head, row tile): the host plan's items without
// its empty splits, each sequence's split-major (a split's KV heads read the
// same pages close together, and decoding an item divides by HR, not by the
// sequence's split count; the order changes no result).  The CTAs of the
// fixed grid take items blockIdx.x, blockIdx.x + gridDim.x, ...
//
// Every warp of a CTA plans for itself (the same result in each), so that no
// broadcast and no block barrier stand between the lengths and the first
// page load.  The planning is on the critical path of every CTA's start, in
// SMs whose other CTAs are streaming, so it is kept short: the first 256
// lengths are read once, 8 consecutive ones per lane, and the item is found
// with one warp scan of the lanes' item counts and a search among one lane's
// 8 sequences; sequences past the first 256, and a CTA's later items, are
// walked 32 at a time from memory.
//
// The plan depends only on the context lengths and the problem, which the
// layers of one decode step share.  So the planning call also records it for
// them: the first item of each split writes {sequence, split, context} to
// entry k / HR of a table in the workspace (item k; a split's HR items are
// consecutive) and the one holding the last split writes the split count.  A
// call flagged PKV_DECODE_PLAN_READY reads its items from there -- one load
// of the header and of its first entry in flight together, in place of the
// planning chain -- after checking every value against the bounds.
#pragma once

#include "decode_common.cuh"

namespace pkv {

// Error bit of a call that reuses a plan (PKV_DECODE_PLAN_READY) and finds
// none of this problem in the workspace: the affected rows are unspecified.
constexpr uint32_t kErrStalePlan = 2u;

struct PlanRule {
    int P_fixed;     // > 0: this partition (caller option)
    int num_splits;  // > 0 (without P_fixed): split the longest context this many ways
    int P0;          // planner start: 512 tokens per column tile and KV head of the CTA
    int need;        // ceil(6 per SM / HR_rule): the rule's work-item target per (KV head, row tile)
                     // pair the rule counts (the description's)
    int NS_cap;      // split count of the bounds (the workspace's)
    int sum32;       // B * n_cap < 2^31: the total context fits a 32-bit warp reduction
};

// ceil(a / b) rounded up to a page, for the rule's rare paths.  Not inlined:
// inlined, the division was evaluated even when its branch was not taken,
// which puts its latency on every CTA's start.
static __device__ __noinline__ int plan_pages_cdiv(int a, int b) {
    const int q = a > 0 ? (a - 1) / b + 1 : 0;   // no overflow near INT_MAX
    return (q + kPageTokens - 1) / kPageTokens * kPageTokens;
}

// The partition for the actual longest (mx) and total (sum) context.  The
// halving test in 32-bit-friendly form: HR * ceil(sum / P) >= target  <=>
// ceil(sum / P) >= need = ceil(target / HR)  <=>  sum > (need - 1) * P.
__device__ __forceinline__ int device_plan_partition_rule(const PlanRule& r, int mx, long long sum) {
    constexpr int BS = kPageTokens;
    auto round_up = [](int a) { return a > 0 ? ((a - 1) / BS + 1) * BS : 0; };   // BS: a shift
    const int maxn = mx > 0 ? mx : 1;
    int P;
    if (r.P_fixed > 0) {
        P = r.P_fixed;
    } else if (r.num_splits > 0) {
        P = plan_pages_cdiv(maxn, r.num_splits);
    } else {
        P = round_up(maxn < r.P0 ? maxn : r.P0);
        const int min_p = 4 * BS;
        const long long s1 = sum > 0 ? sum : 1;
        const long long need1 = r.need - 1;
        while (P > min_p) {
            if (s1 > need1 * P) break;   // enough work items
            int np = round_up(P / 2);
            if (np < min_p) np = min_p;
            if (np >= P) break;
            P = np;
        }
    }
    // No more splits than the workspace holds: P >= ceil(mx / NS_cap) rounded
    // up to a page, which for P a multiple of the page is P * NS_cap >= mx.
    if ((long long)P * r.NS_cap < mx) P = plan_pages_cdiv(mx, r.NS_cap);
    return P;
}

// Sequences 8 l .. 8 l + 7 go to lane l: the first kPlanRegSeqs * 32 clamped
// context lengths stay in each warp's registers (0 past the last sequence).
constexpr int kPlanRegSeqs = 8;
constexpr int kPlanRegB = 32 * kPlanRegSeqs;

struct PlanRegs {
    int n[kPlanRegSeqs];
};

// Longest and total context (each clamped to [0, n_cap]) over B sequences;
// every lane of the warp gets both, and pr its lane's first lengths.
__device__ __forceinline__ void warp_context_stats(const int32_t* ctx, int B, int n_cap, bool sum32, int lane,
                                                   PlanRegs& pr, int* mx, long long* sum) {
    const int b0 = kPlanRegSeqs * lane;
    if ((reinterpret_cast<uintptr_t>(ctx) & 15) == 0 && b0 + kPlanRegSeqs <= B) {
        const int4 v0 = *reinterpret_cast<const int4*>(ctx + b0);
        const int4 v1 = *reinterpret_cast<const int4*>(ctx + b0 + 4);
        pr.n[0] = v0.x, pr.n[1] = v0.y, pr.n[2] = v0.z, pr.n[3] = v0.w;
        pr.n[4] = v1.x, pr.n[5] = v1.y, pr.n[6] = v1.z, pr.n[7] = v1.w;
    } else {
#pragma unroll
        for (int u = 0; u < kPlanRegSeqs; ++u) pr.n[u] = b0 + u < B ? ctx[b0 + u] : 0;
    }
    int m = 0;
    long long s = 0;
#pragma unroll
    for (int u = 0; u < kPlanRegSeqs; ++u) {
        pr.n[u] = clampi(pr.n[u], 0, n_cap);
        m = max(m, pr.n[u]);
        s += pr.n[u];
    }
    constexpr int U = 8;   // further sequences: U loads in flight per lane
    for (int base = kPlanRegB; base < B; base += 32 * U) {
        int v[U];
#pragma unroll
        for (int u = 0; u < U; ++u) {
            const int b = base + 32 * u + lane;
            v[u] = b < B ? ctx[b] : 0;
        }
#pragma unroll
        for (int u = 0; u < U; ++u) {
            const int n = clampi(v[u], 0, n_cap);
            m = max(m, n);
            s += n;
        }
    }
    m = __reduce_max_sync(0xffffffffu, m);
    if (sum32) {   // no lane's or warp's total can overflow 32 bits
        s = __reduce_add_sync(0xffffffffu, (unsigned)s);
    } else {
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) s += __shfl_xor_sync(0xffffffffu, s, o);
    }
    *mx = m;
    *sum = s;
}

// Divisions of the walk: by the partition P (splits of a context) and by HR
// (items of a split), each a shift when a power of two (the usual case).
__device__ __forceinline__ int log2_if_pow2(int x) { return (x & (x - 1)) == 0 ? 31 - __clz(x) : -1; }

struct PlanDiv {
    int P, psh;    // psh = log2 P, or -1
    int HR, hsh;   // hsh = log2 HR, or -1
    __device__ __forceinline__ PlanDiv(int P_, int HR_) {
        P = P_;
        psh = log2_if_pow2(P_);
        HR = HR_;
        hsh = log2_if_pow2(HR_);
    }
    // Items of a context of n tokens: max(1, ceil(n / P)) splits (an empty
    // context has one, which writes its zero rows) times HR.  POW2: psh >= 0.
    // (The shift and the division stay in separate code: a select between
    // them had the division evaluated every time, ~1000 cycles for 8 lengths.)
    template <bool POW2>
    __device__ __forceinline__ int items(int n) const {
        const int m = max(n, 1) - 1;
        return ((POW2 ? (m >> psh) : m / P) + 1) * HR;
    }
    __device__ __forceinline__ int split_of(int j) const { return hsh >= 0 ? j >> hsh : j / HR; }
};

// Sequences [0, b0) hold items [0, base); b0 is a multiple of 32.  A CTA's
// items only grow, so its cursor only moves forward.
struct PlanCursor {
    int b0;
    long long base;
};

// Item k among the first kPlanRegB sequences, from the registers (warp-wide,
// every lane gets the result): sequence *b, item *j within it and its clamped
// context *n_b.  Sets *total to the plan's item count when every sequence is
// among them (else -1), and the cursor to the 32-sequence chunk of the item
// (or past the registers' sequences when k lies beyond them).  Returns false
// when k is not among them.
__device__ __forceinline__ bool warp_plan_first_item(const PlanRegs& pr, int B, const PlanDiv& dv, long long k,
                                                     PlanCursor& cur, int lane, int* b, int* j, int* n_b,
                                                     long long* total) {
    int c[kPlanRegSeqs], t = 0;
    if (dv.psh >= 0) {
#pragma unroll
        for (int u = 0; u < kPlanRegSeqs; ++u) c[u] = kPlanRegSeqs * lane + u < B ? dv.items<true>(pr.n[u]) : 0;
    } else {
#pragma unroll
        for (int u = 0; u < kPlanRegSeqs; ++u) c[u] = kPlanRegSeqs * lane + u < B ? dv.items<false>(pr.n[u]) : 0;
    }
#pragma unroll
    for (int u = 0; u < kPlanRegSeqs; ++u) t += c[u];
    int incl = t;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const int v = __shfl_up_sync(0xffffffffu, incl, o);
        if (lane >= o) incl += v;
    }
    const int all = __shfl_sync(0xffffffffu, incl, 31);
    *total = B <= kPlanRegB ? all : -1;
    if (k >= all) {
        cur.b0 = kPlanRegB;
        cur.base = all;
        return false;
    }
    const int src = __ffs(__ballot_sync(0xffffffffu, k < incl)) - 1;
    // In lane src: the sequence u holding item rem of the lane is the number of
    // the lane's running item sums at or below rem (selects, no branches).
    const int rem = (int)(k - (incl - t));   // meaningful in lane src
    int pre = 0, before = 0, u_hit = 0, nn = pr.n[0];
#pragma unroll
    for (int u = 0; u < kPlanRegSeqs; ++u) {
        pre += c[u];
        const bool past = pre <= rem;
        before = past ? pre : before;
        u_hit += past ? 1 : 0;
        if (u + 1 < kPlanRegSeqs) nn = past ? pr.n[u + 1] : nn;
    }
    const int bb = kPlanRegSeqs * lane + u_hit, jj = rem - before;
    *b = __shfl_sync(0xffffffffu, bb, src);
    *j = __shfl_sync(0xffffffffu, jj, src);
    *n_b = __shfl_sync(0xffffffffu, nn, src);
    // chunk of 32 sequences holding *b starts at lane 4 q's sequences
    const int q = *b >> 5;
    cur.b0 = 32 * q;
    cur.base = __shfl_sync(0xffffffffu, incl - t, (32 / kPlanRegSeqs) * q);
    return true;
}

// Item k of the plan at or after the cursor, walking the lengths in memory 32
// sequences at a time (warp-wide, every lane gets the result); false when k
// is past the last item.
__device__ __forceinline__ bool warp_plan_item(const int32_t* ctx, int B, int n_cap, const PlanDiv& dv, long long k,
                                               PlanCursor& cur, int lane, int* b, int* j, int* n_b) {
    for (; cur.b0 < B; cur.b0 += 32) {
        const int bb = cur.b0 + lane;
        int n = 0, cnt = 0;
        if (bb < B) {
            n = clampi(ctx[bb], 0, n_cap);
            cnt = dv.psh >= 0 ? dv.items<true>(n) : dv.items<false>(n);
        }
        int incl = cnt;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const int v = __shfl_up_sync(0xffffffffu, incl, o);
            if (lane >= o) incl += v;
        }
        const int chunk_items = __shfl_sync(0xffffffffu, incl, 31);
        if (k < cur.base + chunk_items) {
            const unsigned hit = __ballot_sync(0xffffffffu, k < cur.base + incl);
            const int src = __ffs(hit) - 1;
            const int excl = __shfl_sync(0xffffffffu, incl - cnt, src);
            *b = cur.b0 + src;
            *j = (int)(k - cur.base - excl);
            *n_b = __shfl_sync(0xffffffffu, n, src);
            return true;
        }
        cur.base += chunk_items;
    }
    return false;
}

}  // namespace pkv
