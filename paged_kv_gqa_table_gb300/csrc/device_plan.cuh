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
// -- in the order (b, KV head, row tile, split), split fastest: the grid order
// of the host plan without its empty splits.  The CTAs of the fixed grid take
// items blockIdx.x, blockIdx.x + gridDim.x, ...; each walks the sequences
// forward, 32 at a time, to find its next item.
#pragma once

#include "decode_common.cuh"

namespace pkv {

struct PlanRule {
    int P_fixed;     // > 0: this partition (caller option)
    int num_splits;  // > 0 (without P_fixed): split the longest context this many ways
    int P0;          // planner start: 512 tokens per column tile and KV head of the CTA
    int HR_rule;     // (KV head, row tile) pairs the rule counts: the description's
    int num_sms;     // the rule's work-item target is 6 per SM
    int NS_cap;      // split count of the bounds (the workspace's)
};

// The partition for the actual longest (mx) and total (sum) context.  The
// halving test in 32-bit-friendly form: HR * ceil(sum / P) >= target  <=>
// ceil(sum / P) >= need = ceil(target / HR)  <=>  sum > (need - 1) * P.
__device__ __forceinline__ int device_plan_partition_rule(const PlanRule& r, int mx, long long sum) {
    constexpr int BS = kPageTokens;
    auto cdiv = [](int a, int b) { return a > 0 ? (a - 1) / b + 1 : 0; };   // no overflow near INT_MAX
    auto round_up = [&](int a) { return cdiv(a, BS) * BS; };
    const int maxn = mx > 0 ? mx : 1;
    int P;
    if (r.P_fixed > 0) {
        P = r.P_fixed;
    } else if (r.num_splits > 0) {
        P = round_up(cdiv(maxn, r.num_splits));
    } else {
        P = round_up(maxn < r.P0 ? maxn : r.P0);
        const int min_p = 4 * BS, HR = r.HR_rule;
        const long long target = 6LL * r.num_sms;
        const long long need = (target + HR - 1) / HR;
        const long long s1 = sum > 0 ? sum : 1;
        while (P > min_p) {
            if (s1 > (need - 1) * (long long)P) break;   // enough work items
            int np = round_up(P / 2);
            if (np < min_p) np = min_p;
            if (np >= P) break;
            P = np;
        }
    }
    const int fit = round_up(cdiv(mx, r.NS_cap));   // splits within NS_cap
    return P < fit ? fit : P;
}

// Longest and total context (each clamped to [0, n_cap]) over B sequences;
// every lane of the warp gets both.
__device__ __forceinline__ void warp_context_stats(const int32_t* ctx, int B, int n_cap, int lane, int* mx,
                                                   long long* sum) {
    int m = 0;
    long long s = 0;
    constexpr int U = 8;   // loads in flight per lane: one memory round trip per 256 sequences
    for (int base = 0; base < B; base += 32 * U) {
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
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
        m = max(m, __shfl_xor_sync(0xffffffffu, m, o));
        s += __shfl_xor_sync(0xffffffffu, s, o);
    }
    *mx = m;
    *sum = s;
}

// Sequences [b0, b0 + 32 * k) hold items [0, base); a CTA's items only grow.
struct PlanCursor {
    int b0;
    long long base;
};

// Item k of the plan (warp-wide, every lane gets the result): sequence *b,
// item *j within it, its clamped context *n_b and split count *nsb; false
// when k is past the last item.
__device__ __forceinline__ bool warp_plan_item(const int32_t* ctx, int B, int n_cap, int P, int HR, long long k,
                                               PlanCursor& cur, int lane, int* b, int* j, int* n_b, int* nsb) {
    for (; cur.b0 < B; cur.b0 += 32) {
        const int bb = cur.b0 + lane;
        int n = 0, cnt = 0;
        if (bb < B) {
            n = clampi(ctx[bb], 0, n_cap);
            cnt = max(1, n > 0 ? (n - 1) / P + 1 : 0) * HR;
        }
        int incl = cnt;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const int v = __shfl_up_sync(0xffffffffu, incl, o);
            if (lane >= o) incl += v;
        }
        const int total = __shfl_sync(0xffffffffu, incl, 31);
        if (k < cur.base + total) {
            const unsigned hit = __ballot_sync(0xffffffffu, k < cur.base + incl);
            const int src = __ffs(hit) - 1;
            const int excl = __shfl_sync(0xffffffffu, incl - cnt, src);
            *b = cur.b0 + src;
            *j = (int)(k - cur.base - excl);
            *n_b = __shfl_sync(0xffffffffu, n, src);
            *nsb = __shfl_sync(0xffffffffu, cnt, src) / HR;
            return true;
        }
        cur.base += total;
    }
    return false;
}

}  // namespace pkv
