// schedule.cu -- the device plan of paged decode: one CTA turns the device's
// context lengths into the split plan and a list of non-empty work items, so
// that a call captured into a CUDA graph with capacity bounds launches phase 1
// over the actual work only.
//
// Plan: the rule of the host planner (api.cu, auto_partition) applied to the
// actual longest context max_n and total sum_n -- P starts at P0 (or max_n
// rounded up to a page, if shorter) and halves while HR_rule * ceil(sum_n / P)
// (the description's KV heads x row tiles) is below six items per SM, down to
// four pages -- then raised, if needed, to
// ceil(max_n / NS_cap) rounded up to a page so that no sequence has more splits
// than the workspace holds.  Items: sequence b has ns_b = max(1, ceil(n_b / P))
// splits (one item writes the zero rows of an empty context) for each of its
// Hkv * RT (grid KV head, row tile) pairs -- a grid KV head is a pair of KV
// heads when the CTAs take two -- listed as (b, kvh | rt << 16, s, n_b)
// with s fastest: the grid order of the host plan without its empty splits
// (n_b rides along so that a CTA needs one load to start its item).
#include "internal.h"

namespace pkv {

__global__ void __launch_bounds__(1024) decode_schedule_kernel(const SchedParams p) {
    // Lets phase 1, queued behind this kernel, start its prologue (it waits for the list).
    asm volatile("griddepcontrol.launch_dependents;");
    constexpr int CH = 1024;   // sequences per chunk: one per thread
    __shared__ int s_max[32];
    __shared__ long long s_sum[32];
    __shared__ int s_P, s_total;
    __shared__ int s_cnt[CH], s_off[CH], s_n[CH], s_warp[32];
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5, nw = blockDim.x >> 5;

    // 1. longest and total context, clamped as the decode kernels clamp them
    //    (the first chunk's lengths stay in shared memory for step 2)
    int mx = 0;
    long long sum = 0;
    for (int b = tid; b < p.B; b += blockDim.x) {
        const int n = clampi(p.ctx[b], 0, p.n_cap);
        if (b < CH) s_n[b] = n;
        mx = max(mx, n);
        sum += n;
    }
    for (int o = 16; o > 0; o >>= 1) {
        mx = max(mx, __shfl_xor_sync(0xffffffffu, mx, o));
        sum += __shfl_xor_sync(0xffffffffu, sum, o);
    }
    if (lane == 0) {
        s_max[warp] = mx;
        s_sum[warp] = sum;
    }
    __syncthreads();
    if (warp == 0) {
        mx = lane < nw ? s_max[lane] : 0;
        sum = lane < nw ? s_sum[lane] : 0;
        for (int o = 16; o > 0; o >>= 1) {
            mx = max(mx, __shfl_xor_sync(0xffffffffu, mx, o));
            sum += __shfl_xor_sync(0xffffffffu, sum, o);
        }
        if (lane == 0) {
            // The rule in 32-bit arithmetic (64-bit integer division is slow
            // here): HR * ceil(sum / P) >= target  <=>
            // ceil(sum / P) >= need = ceil(target / HR)  <=>  sum > (need - 1) * P.
            const int BS = p.BS;
            auto cdiv = [](int a, int b) { return a > 0 ? (a - 1) / b + 1 : 0; };   // no overflow near INT_MAX
            auto round_up = [&](int a) { return cdiv(a, BS) * BS; };
            const int maxn = mx > 0 ? mx : 1;
            int P;
            if (p.P_fixed > 0) {
                P = p.P_fixed;
            } else if (p.num_splits > 0) {
                P = round_up(cdiv(maxn, p.num_splits));
            } else {
                P = round_up(maxn < p.P0 ? maxn : p.P0);
                const int min_p = 4 * BS, HR = p.HR_rule;
                const long long target = 6LL * p.num_sms;
                const long long need = (target + HR - 1) / HR;   // once
                const long long s1 = sum > 0 ? sum : 1;
                while (P > min_p) {
                    if (s1 > (need - 1) * (long long)P) break;   // enough work items
                    int np = round_up(P / 2);
                    if (np < min_p) np = min_p;
                    if (np >= P) break;
                    P = np;
                }
            }
            const int fit = round_up(cdiv(mx, p.NS_cap));   // splits within NS_cap
            if (P < fit) P = fit;
            s_P = P;
            p.hdr[0] = P;
            p.hdr[1] = mx > 0 ? cdiv(mx, P) : 1;
        }
    }
    __syncthreads();
    const int P = s_P;
    const int HR = p.Hkv * p.RT;

    // 2. items per sequence, scanned CH sequences at a time; each warp then
    //    writes the items of every nw-th sequence of the chunk
    int base = 0;
    for (int c0 = 0; c0 < p.B; c0 += CH) {
        const int b = c0 + tid;
        int n = 0, cnt = 0;
        if (b < p.B) {
            n = c0 == 0 ? s_n[tid] : clampi(p.ctx[b], 0, p.n_cap);
            cnt = max(1, n > 0 ? (n - 1) / P + 1 : 0) * HR;
        }
        int incl = cnt;   // inclusive scan within the warp
        for (int o = 1; o < 32; o <<= 1) {
            const int v = __shfl_up_sync(0xffffffffu, incl, o);
            if (lane >= o) incl += v;
        }
        if (lane == 31) s_warp[warp] = incl;
        __syncthreads();
        if (warp == 0) {   // exclusive scan of the warp totals
            const int v = lane < nw ? s_warp[lane] : 0;
            int w_incl = v;
            for (int o = 1; o < 32; o <<= 1) {
                const int u = __shfl_up_sync(0xffffffffu, w_incl, o);
                if (lane >= o) w_incl += u;
            }
            if (lane < nw) s_warp[lane] = w_incl - v;
            if (lane == 31) s_total = w_incl;
        }
        __syncthreads();
        s_cnt[tid] = cnt;
        s_off[tid] = base + s_warp[warp] + incl - cnt;
        s_n[tid] = n;
        __syncthreads();
        const int m = min(CH, p.B - c0);
        for (int k = warp; k < m; k += nw) {
            const int items = s_cnt[k], off = s_off[k], nsb = items / HR, nk = s_n[k];
            for (int j = lane; j < items; j += 32) {
                const int kr = j / nsb;
                p.list[off + j] = make_int4(c0 + k, (kr / p.RT) | ((kr % p.RT) << 16), j - kr * nsb, nk);
            }
        }
        base += s_total;
        __syncthreads();
    }
    if (tid == 0) p.hdr[2] = base;
}

cudaError_t launch_schedule(const SchedParams& p, cudaStream_t stream) {
    decode_schedule_kernel<<<1, 1024, 0, stream>>>(p);
    return cudaGetLastError();
}

}  // namespace pkv
