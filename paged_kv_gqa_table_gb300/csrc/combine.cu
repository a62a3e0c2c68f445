// combine.cu -- phase 2 of paged decode attention (cross-split log-sum-exp
// combine) and the optional block-table validator.
//
// Combine ("koas-w.github.io flash-decode post", _flash_decode_combine_kernel;
// "paged_attention_v2_triton.py", _reduce_partitions_kernel):
//   M = max_s m_s,  f_s = e^{m_s - M},  out = sum_s f_s acc_s / sum_s f_s l_s.
// Rows are (sequence b, query token i, head h), i < q_len; a row whose causal
// window n - q_len + i + 1 is empty (n == 0 for one token) is zero.
#include "internal.h"

namespace pkv {

// Context length of row r's sequence (clamped) and whether its query token's
// causal window is empty.
__device__ __forceinline__ int row_context(const CombineParams& p, long long r, bool* empty) {
    const long long bi = r / p.Hq;   // b * q_len + i
    int n = p.ctx[bi / p.q_len];
    n = n < 0 ? 0 : (n > p.n_cap ? p.n_cap : n);
    *empty = n - p.q_len + (int)(bi % p.q_len) + 1 <= 0;
    return n;
}

// One warp per row (sequence, query token, head); lane l owns elements [l*D/32, (l+1)*D/32).
// Splits are merged a chunk at a time (32 / (D/32) splits): the chunk's m, l
// and acc rows are all loaded before any is used, so a chunk costs one memory
// round trip,
// and the chunks fold into a running (M, L, acc) by log-sum-exp rescaling.
// Launched as a programmatic dependent of phase 1: the prologue (context
// length) runs while phase 1 finishes; griddepcontrol.wait precedes every
// read of the partials.
template <typename T, int D>
__global__ void __launch_bounds__(256) combine_kernel(const CombineParams p) {
    constexpr int EPL = D / 32;   // elements per lane
    constexpr int CH = 32 / EPL;  // splits per chunk: 32 floats of acc in flight per lane
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const long long bh = (long long)blockIdx.x * 8 + warp;
    const bool live = bh < (long long)p.B * p.q_len * p.Hq;
    int n = 0;
    bool empty = true;
    if (live) n = row_context(p, bh, &empty);
    asm volatile("griddepcontrol.wait;" ::: "memory");
    if (!live) return;
    T* o = reinterpret_cast<T*>(p.out) + bh * D + lane * EPL;
    if (empty) {
        if (p.skip_single) return;   // phase 1 wrote the zero row
#pragma unroll
        for (int e = 0; e < EPL; ++e) o[e] = from_float<T>(0.f);
        return;
    }
    // Under the device plan the partition is read from the header phase 1
    // wrote (checked: the header may be another problem's), and the first
    // chunk's partials are loaded together with it, clamped to the row's
    // ns_stride splits of the workspace and masked once the split count is
    // known; under the host plan the split count comes first.
    int ns = -1;
    if (!p.sched_hdr) {
        ns = (int)min(((long long)n + p.P - 1) / p.P, (long long)p.ns_stride);
        if (p.skip_single && ns <= 1) return;   // phase 1 wrote this row directly
    }
    const float* pm = p.part_m + bh * p.ns_stride;
    const float* pl = p.part_l + bh * p.ns_stride;
    const float* pa = p.part_acc + bh * p.ns_stride * D + lane * EPL;
    constexpr float kLog2e = 1.4426950408889634f;
    float M = -INFINITY, L = 0.f, acc[EPL];
#pragma unroll
    for (int e = 0; e < EPL; ++e) acc[e] = 0.f;
    for (int c0 = 0;; c0 += CH) {
        // Unconditional loads (index clamped to the last split) so that all
        // of the chunk's loads are in flight together; padding is masked.
        const int lim = ns >= 0 ? ns : p.ns_stride;
        float m[CH], l[CH], a[CH][EPL];
#pragma unroll
        for (int j = 0; j < CH; ++j) {
            const int sj = min(c0 + j, lim - 1);
            m[j] = __ldg(pm + sj);
            l[j] = __ldg(pl + sj);
#pragma unroll
            for (int e = 0; e < EPL; e += 2) {
                const float2 v = __ldg(reinterpret_cast<const float2*>(pa + (size_t)sj * D + e));
                a[j][e] = v.x;
                a[j][e + 1] = v.y;
            }
        }
        if (ns < 0) {
            const int P = device_plan_partition(p.sched_hdr[0]);
            ns = (int)min(((long long)n + P - 1) / P, (long long)p.ns_stride);
            if (p.skip_single && ns <= 1) return;   // phase 1 wrote this row directly
        }
        // Splits past the row's last are padding: weight 0 and values 0 (a
        // speculatively loaded one may hold anything).
#pragma unroll
        for (int j = 0; j < CH; ++j)
            if (c0 + j >= ns) {
                m[j] = -INFINITY;
                l[j] = 0.f;
#pragma unroll
                for (int e = 0; e < EPL; ++e) a[j][e] = 0.f;
            }
        float Mc = M;
#pragma unroll
        for (int j = 0; j < CH; ++j) Mc = fmaxf(Mc, m[j]);
        const float r = ex2((M - Mc) * kLog2e);   // rescale of the running sums (0 at the start)
        L *= r;
#pragma unroll
        for (int e = 0; e < EPL; ++e) acc[e] *= r;
#pragma unroll
        for (int j = 0; j < CH; ++j) {
            const float f = ex2((m[j] - Mc) * kLog2e);   // a sentinel or padding (-inf) gives 0
            L += f * l[j];
#pragma unroll
            for (int e = 0; e < EPL; ++e) acc[e] += f * a[j][e];
        }
        M = Mc;
        if (c0 + CH >= ns) break;
    }
    const float inv = 1.f / L;
#pragma unroll
    for (int e = 0; e < EPL; e += 2) {
        const uint32_t packed = Mma<T>::pack(acc[e] * inv, acc[e + 1] * inv);
        *reinterpret_cast<uint32_t*>(o + e) = packed;
    }
}

// Rows with many splits (long contexts): one CTA of 8 warps per row; warp w
// folds chunks w, w+8, ... of splits, so the chunks' memory round
// trips overlap across warps; the warps' running (M, L, acc) are then merged
// through shared memory.
template <typename T, int D>
__global__ void __launch_bounds__(256) combine_wide_kernel(const CombineParams p) {
    constexpr int EPL = D / 32, CH = 32 / EPL, NW = 8;
    __shared__ float s_acc[NW][D];
    __shared__ float s_m[NW], s_l[NW];
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const long long bh = blockIdx.x;
    bool empty = true;
    const int n = row_context(p, bh, &empty);
    asm volatile("griddepcontrol.wait;" ::: "memory");
    const int P = p.sched_hdr ? device_plan_partition(p.sched_hdr[0]) : p.P;
    const int ns = (int)min(((long long)n + P - 1) / P, (long long)p.ns_stride);
    if (p.skip_single && ns <= 1) return;
    T* o = reinterpret_cast<T*>(p.out) + bh * D;
    if (empty) {
        for (int d = threadIdx.x; d < D; d += blockDim.x) o[d] = from_float<T>(0.f);
        return;
    }
    const float* pm = p.part_m + bh * p.ns_stride;
    const float* pl = p.part_l + bh * p.ns_stride;
    const float* pa = p.part_acc + bh * p.ns_stride * D + lane * EPL;
    constexpr float kLog2e = 1.4426950408889634f;
    float M = -INFINITY, L = 0.f, acc[EPL];
#pragma unroll
    for (int e = 0; e < EPL; ++e) acc[e] = 0.f;
    for (int c0 = warp * CH; c0 < ns; c0 += NW * CH) {
        // Unconditional loads (index clamped to the last split) so that all
        // of the chunk's loads are in flight together; padding gets m = -inf.
        float m[CH], l[CH], a[CH][EPL];
#pragma unroll
        for (int j = 0; j < CH; ++j) {
            const int sj = min(c0 + j, ns - 1);
            m[j] = __ldg(pm + sj);
            l[j] = __ldg(pl + sj);
#pragma unroll
            for (int e = 0; e < EPL; e += 2) {
                const float2 v = __ldg(reinterpret_cast<const float2*>(pa + (size_t)sj * D + e));
                a[j][e] = v.x;
                a[j][e + 1] = v.y;
            }
        }
#pragma unroll
        for (int j = 0; j < CH; ++j)
            if (c0 + j >= ns) m[j] = -INFINITY;
        float Mc = M;
#pragma unroll
        for (int j = 0; j < CH; ++j) Mc = fmaxf(Mc, m[j]);
        const float r = ex2((M - Mc) * kLog2e);
        L *= r;
#pragma unroll
        for (int e = 0; e < EPL; ++e) acc[e] *= r;
#pragma unroll
        for (int j = 0; j < CH; ++j) {
            const float f = ex2((m[j] - Mc) * kLog2e);
            L += f * l[j];
#pragma unroll
            for (int e = 0; e < EPL; ++e) acc[e] += f * a[j][e];
        }
        M = Mc;
    }
#pragma unroll
    for (int e = 0; e < EPL; ++e) s_acc[warp][lane * EPL + e] = acc[e];
    if (lane == 0) {
        s_m[warp] = M;
        s_l[warp] = L;
    }
    __syncthreads();
    float Mt = -INFINITY;
#pragma unroll
    for (int w = 0; w < NW; ++w) Mt = fmaxf(Mt, s_m[w]);
    float f[NW], Lt = 0.f;
#pragma unroll
    for (int w = 0; w < NW; ++w) {
        f[w] = ex2((s_m[w] - Mt) * kLog2e);   // 0 for a warp that had no chunk
        Lt += f[w] * s_l[w];
    }
    const float inv = 1.f / Lt;
    for (int d = threadIdx.x; d < D; d += blockDim.x) {
        float v = 0.f;
#pragma unroll
        for (int w = 0; w < NW; ++w) v += f[w] * s_acc[w][d];
        o[d] = from_float<T>(v * inv);
    }
}

// Plans with more splits than this use one CTA per row instead of one warp.
constexpr int kWideCombineSplits = 32;

template <typename T, int D>
cudaError_t launch_combine_t(const CombineParams& p, cudaLaunchConfig_t& cfg) {
    const long long rows = (long long)p.B * p.q_len * p.Hq;
    if (p.ns_stride > kWideCombineSplits) {
        cfg.gridDim = dim3((unsigned)rows);
        return cudaLaunchKernelEx(&cfg, combine_wide_kernel<T, D>, p);
    }
    cfg.gridDim = dim3((unsigned)((rows + 7) / 8));
    return cudaLaunchKernelEx(&cfg, combine_kernel<T, D>, p);
}

cudaError_t launch_combine(int dtype, int D, const CombineParams& p, cudaStream_t stream, bool after_phase1) {
    if ((long long)p.B * p.q_len * p.Hq == 0) return cudaSuccess;
    cudaLaunchConfig_t cfg = {};
    cfg.blockDim = dim3(256);
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = after_phase1 ? 1 : 0;
    const bool bf = dtype == 1;
    switch (D) {
        case 64: return bf ? launch_combine_t<__nv_bfloat16, 64>(p, cfg) : launch_combine_t<__half, 64>(p, cfg);
        case 128: return bf ? launch_combine_t<__nv_bfloat16, 128>(p, cfg) : launch_combine_t<__half, 128>(p, cfg);
        case 256: return bf ? launch_combine_t<__nv_bfloat16, 256>(p, cfg) : launch_combine_t<__half, 256>(p, cfg);
        default: return cudaErrorInvalidValue;
    }
}

// ---------------------------------------------------------------- validator
// One CTA per sequence.  Bit 0: context length out of range; bit 1: a live
// block-table entry outside [0, num_blocks).
__global__ void __launch_bounds__(128) validate_table_kernel(const int32_t* table, const int32_t* ctx, int MBPS,
                                                              int BS, int NB, int max_ctx, uint32_t* err) {
    const int b = blockIdx.x;
    int n = ctx[b];
    const long long cap = (long long)MBPS * BS;
    if (n < 0 || n > max_ctx || (long long)n > cap) {
        if (threadIdx.x == 0) atomicOr(err, 1u);
        n = n < 0 ? 0 : (int)((long long)n > cap ? cap : n);
    }
    const int pages = (n + BS - 1) / BS;
    bool bad = false;
    for (int j = threadIdx.x; j < pages; j += blockDim.x) {
        const int id = table[(size_t)b * MBPS + j];
        bad |= (id < 0 || id >= NB);
    }
    if (__syncthreads_or(bad) && threadIdx.x == 0) atomicOr(err, 2u);
}

cudaError_t launch_validate(const int32_t* table, const int32_t* ctx, int B, int MBPS, int BS, int NB, int max_ctx,
                            uint32_t* err, cudaStream_t stream) {
    if (B == 0) return cudaSuccess;
    validate_table_kernel<<<B, 128, 0, stream>>>(table, ctx, MBPS, BS, NB, max_ctx, err);
    return cudaGetLastError();
}

}  // namespace pkv
