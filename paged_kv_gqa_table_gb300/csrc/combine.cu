// combine.cu -- phase 2 of paged decode attention (cross-split log-sum-exp
// combine) and the optional block-table validator.
//
// Combine ("koas-w.github.io flash-decode post", _flash_decode_combine_kernel;
// "paged_attention_v2_triton.py", _reduce_partitions_kernel):
//   M = max_s m_s,  f_s = e^{m_s - M},  out = sum_s f_s acc_s / sum_s f_s l_s.
// One CTA of 8 warps per (sequence, query head): warp w takes splits
// s = w, w+8, ...; each lane owns D/32 consecutive elements of acc (vector
// loads), so a warp reads one split's row as one coalesced request.
#include "internal.h"

namespace pkv {

template <typename T, int D>
__global__ void __launch_bounds__(256) combine_kernel(const CombineParams p) {
    constexpr int NW = 8;
    constexpr int EPL = D / 32;   // elements per lane
    __shared__ float s_red[NW][D];
    __shared__ float s_l[NW];
    __shared__ float s_m[NW];

    const int bh = blockIdx.x;
    const int b = bh / p.Hq;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    int n = p.ctx[b];
    n = n < 0 ? 0 : (n > p.n_cap ? p.n_cap : n);
    const int ns = (n + p.P - 1) / p.P;
    if (p.skip_single && ns <= 1) return;   // phase 1 wrote this row directly
    T* o = reinterpret_cast<T*>(p.out) + (size_t)bh * D;
    if (n == 0) {
        for (int d = threadIdx.x; d < D; d += blockDim.x) o[d] = from_float<T>(0.f);
        return;
    }
    const float* pm = p.part_m + (size_t)bh * p.ns_stride;
    const float* pl = p.part_l + (size_t)bh * p.ns_stride;
    const float* pa = p.part_acc + (size_t)bh * p.ns_stride * D;

    float mx = -INFINITY;
    for (int s = threadIdx.x; s < ns; s += blockDim.x) mx = fmaxf(mx, pm[s]);
#pragma unroll
    for (int k = 16; k > 0; k >>= 1) mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, k));
    if (lane == 0) s_m[warp] = mx;
    __syncthreads();
    float M = s_m[0];
#pragma unroll
    for (int w = 1; w < NW; ++w) M = fmaxf(M, s_m[w]);

    constexpr float kLog2e = 1.4426950408889634f;
    float a[EPL];
#pragma unroll
    for (int e = 0; e < EPL; ++e) a[e] = 0.f;
    float L = 0.f;
#pragma unroll 4
    for (int s = warp; s < ns; s += NW) {
        const float f = ex2((pm[s] - M) * kLog2e);   // a sentinel (-inf) gives 0
        L += f * pl[s];
        const float* row = pa + (size_t)s * D + lane * EPL;
#pragma unroll
        for (int e = 0; e < EPL; e += 4) {
            const float4 v = *reinterpret_cast<const float4*>(row + e);
            a[e] += f * v.x;
            a[e + 1] += f * v.y;
            a[e + 2] += f * v.z;
            a[e + 3] += f * v.w;
        }
    }
#pragma unroll
    for (int e = 0; e < EPL; ++e) s_red[warp][lane * EPL + e] = a[e];
    if (lane == 0) s_l[warp] = L;
    __syncthreads();
    float Lt = 0.f;
#pragma unroll
    for (int w = 0; w < NW; ++w) Lt += s_l[w];
    const float inv = 1.f / Lt;
    for (int d = threadIdx.x; d < D; d += blockDim.x) {
        float v = 0.f;
#pragma unroll
        for (int w = 0; w < NW; ++w) v += s_red[w][d];
        o[d] = from_float<T>(v * inv);
    }
}

// D = 64 leaves two elements per lane; the float4 loop above needs four.
template <typename T>
__global__ void __launch_bounds__(256) combine_kernel_d64(const CombineParams p) {
    constexpr int D = 64, NW = 8;
    __shared__ float s_red[NW][D];
    __shared__ float s_l[NW];
    __shared__ float s_m[NW];
    const int bh = blockIdx.x;
    const int b = bh / p.Hq;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    int n = p.ctx[b];
    n = n < 0 ? 0 : (n > p.n_cap ? p.n_cap : n);
    const int ns = (n + p.P - 1) / p.P;
    if (p.skip_single && ns <= 1) return;
    T* o = reinterpret_cast<T*>(p.out) + (size_t)bh * D;
    if (n == 0) {
        for (int d = threadIdx.x; d < D; d += blockDim.x) o[d] = from_float<T>(0.f);
        return;
    }
    const float* pm = p.part_m + (size_t)bh * p.ns_stride;
    const float* pl = p.part_l + (size_t)bh * p.ns_stride;
    const float* pa = p.part_acc + (size_t)bh * p.ns_stride * D;
    float mx = -INFINITY;
    for (int s = threadIdx.x; s < ns; s += blockDim.x) mx = fmaxf(mx, pm[s]);
#pragma unroll
    for (int k = 16; k > 0; k >>= 1) mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, k));
    if (lane == 0) s_m[warp] = mx;
    __syncthreads();
    float M = s_m[0];
#pragma unroll
    for (int w = 1; w < NW; ++w) M = fmaxf(M, s_m[w]);
    constexpr float kLog2e = 1.4426950408889634f;
    float a0 = 0.f, a1 = 0.f, L = 0.f;
#pragma unroll 4
    for (int s = warp; s < ns; s += NW) {
        const float f = ex2((pm[s] - M) * kLog2e);
        L += f * pl[s];
        const float2 v = *reinterpret_cast<const float2*>(pa + (size_t)s * D + lane * 2);
        a0 += f * v.x;
        a1 += f * v.y;
    }
    s_red[warp][lane * 2] = a0;
    s_red[warp][lane * 2 + 1] = a1;
    if (lane == 0) s_l[warp] = L;
    __syncthreads();
    float Lt = 0.f;
#pragma unroll
    for (int w = 0; w < NW; ++w) Lt += s_l[w];
    const float inv = 1.f / Lt;
    for (int d = threadIdx.x; d < D; d += blockDim.x) {
        float v = 0.f;
#pragma unroll
        for (int w = 0; w < NW; ++w) v += s_red[w][d];
        o[d] = from_float<T>(v * inv);
    }
}

cudaError_t launch_combine(int dtype, int D, const CombineParams& p, cudaStream_t stream) {
    const unsigned grid = (unsigned)((long long)p.B * p.Hq);
    if (grid == 0) return cudaSuccess;
    const bool bf = dtype == 1;
    switch (D) {
        case 64:
            if (bf)
                combine_kernel_d64<__nv_bfloat16><<<grid, 256, 0, stream>>>(p);
            else
                combine_kernel_d64<__half><<<grid, 256, 0, stream>>>(p);
            break;
        case 128:
            if (bf)
                combine_kernel<__nv_bfloat16, 128><<<grid, 256, 0, stream>>>(p);
            else
                combine_kernel<__half, 128><<<grid, 256, 0, stream>>>(p);
            break;
        case 256:
            if (bf)
                combine_kernel<__nv_bfloat16, 256><<<grid, 256, 0, stream>>>(p);
            else
                combine_kernel<__half, 256><<<grid, 256, 0, stream>>>(p);
            break;
        default:
            return cudaErrorInvalidValue;
    }
    return cudaGetLastError();
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
