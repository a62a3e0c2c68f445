// decode.cuh -- phase 1 of paged GQA decode attention on sm_103a.
//
// One CTA per (sequence b, KV head, split s).  Split s covers tokens
// [s*P, min((s+1)*P, n)) of the sequence (fixed partitions as in
// "paged_attention_v2_triton.py", _partition_attn_kernel; page-granular
// splits as in the flash-decode post's _flash_decode_partial_kernel).
//
// Roles: warp NWC is the producer: it reads the split's block-table entries
// (32 per coalesced load, one chunk ahead) and, per page, issues TMA tensor
// loads of that page's K and V slices for this KV head into a STAGES-deep
// shared-memory ring (full/empty mbarriers).  Each page is loaded ONCE for the
// whole GQA group.  Warps 0..NWC-1 consume pages round-robin, each keeping its
// own online-softmax state for all G query heads of the group:
//
//   S^T[t][h] = K[t][:] . Q[h][:]          mma.sync m16n8k16, tokens = M (16 per
//                                           page), padded heads = N (8 per tile)
//   m' = max(m, max_t S), alpha = 2^(m-m'), P = 2^(S-m'), l' = alpha*l + sum P
//   O^T[d][h] = alpha*O^T[d][h] + V^T[d][t] P^T[t][h]   (P^T from movmatrix)
//
// Scores are kept in log2 units (scale*log2 e folded into one multiply).  The
// warps' states are merged through shared memory at the end; the CTA writes
// either the final normalised row (the sequence has a single split) or the
// unnormalised fp32 partial (acc, m, l) of its split, m in natural-log units
// (the partial-buffer convention of the flash-decode post).
//
// Shared-memory layouts of one page slice (BS = 16 tokens):
//   NHD : TMA boxes of 64 elements x BS rows, 128-byte swizzle, so that the
//         eight 16-byte rows an ldmatrix phase reads fall in distinct banks.
//   VLLM: the slice copied verbatim: K [D/8][BS][8] (already conflict-free
//         for ldmatrix), V [D][BS] (two-way conflicts at most).
#pragma once

#include "ptx.cuh"

namespace pkv {

enum { kLayoutNHD = 0, kLayoutVLLM = 1 };

struct DecodeParams {
    const void* q;           // [B][Hq][D]
    const int32_t* table;    // [B][MBPS]
    const int32_t* ctx;      // [B]
    void* out;               // [B][Hq][D]
    float* part_acc;         // [B][Hq][ns_stride][D]
    float* part_m;           // [B][Hq][ns_stride]
    float* part_l;           // [B][Hq][ns_stride]
    uint32_t* err;           // device error word or nullptr
    int B, Hq, Hkv, G, MBPS, NB;
    int P;                   // tokens per split (multiple of BS)
    int NS;                  // splits in the grid
    int ns_stride;           // split extent of the partial arrays
    int n_cap;               // context lengths are clamped to [0, n_cap]
    float scale_log2;        // scale * log2(e)
    int partials_only;       // 1: always write partials (+ sentinels), never out
};

template <int D>
struct DecodeTile {
    static constexpr int BS = 16;
    static constexpr int NWC = 4;                                   // consumer warps
    static constexpr int SLICE = BS * D * 2;                        // bytes of one page slice
    static constexpr int STAGES = D == 64 ? 12 : (D == 128 ? 8 : 4);
    static constexpr int RED_STRIDE = D + 4;                        // floats per reduction row
    static constexpr int smem_bytes(int nt) {
        return 1024 + STAGES * 2 * SLICE + STAGES * 2 * 8 + 2 * NWC * nt * 8 * 4 + 16;
    }
};

__device__ __forceinline__ int clampi(int v, int lo, int hi) { return v < lo ? lo : (v > hi ? hi : v); }

// Byte offset of 16-byte chunk c (c < D/8) of token row t in an NHD slice
// written by 64-element TMA boxes with 128-byte swizzle.
template <int BS>
__device__ __forceinline__ uint32_t nhd_off(int t, int c) {
    return (uint32_t)((c >> 3) * (BS * 128) + t * 128 + (((c & 7) ^ (t & 7)) << 4));
}

template <typename T, int LAYOUT, int D, int NT>
__global__ void __launch_bounds__((DecodeTile<D>::NWC + 1) * 32)
    decode_phase1_kernel(const DecodeParams p, const __grid_constant__ CUtensorMap tmk,
                         const __grid_constant__ CUtensorMap tmv) {
    using Tile = DecodeTile<D>;
    constexpr int BS = Tile::BS, NWC = Tile::NWC, SLICE = Tile::SLICE, STAGES = Tile::STAGES;
    constexpr int KT = D / 16;   // k-steps of Q.K^T and d-tiles of P.V
    constexpr int HP = NT * 8;   // padded heads
    constexpr int RS = Tile::RED_STRIDE;
    static_assert(NWC * HP * RS * 4 <= STAGES * 2 * SLICE, "reduction buffer must fit in the ring");

    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    uint8_t* ring = smem;
    uint64_t* full = reinterpret_cast<uint64_t*>(smem + STAGES * 2 * SLICE);
    uint64_t* empty = full + STAGES;
    float* st_m = reinterpret_cast<float*>(empty + STAGES);
    float* st_l = st_m + NWC * HP;
    volatile int* abort_flag = reinterpret_cast<volatile int*>(st_l + NWC * HP);   // set on a wait timeout

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    int item = blockIdx.x;
    const int s = item % p.NS;
    item /= p.NS;
    const int kvh = item % p.Hkv;
    const int b = item / p.Hkv;
    const int h0 = kvh * p.G;

    const int n = clampi(p.ctx[b], 0, p.n_cap);
    const int ns_b = (n + p.P - 1) / p.P;
    const int t0 = s * p.P;
    const int t1 = min(t0 + p.P, n);

    if (t0 >= t1) {
        // Split past the context.  Partials mode writes the (-inf, 0, 0)
        // sentinel; an empty context (n == 0) writes a zero output row.
        if (p.partials_only) {
            for (int i = threadIdx.x; i < p.G * D; i += blockDim.x) {
                const size_t row = ((size_t)b * p.Hq + h0 + i / D) * p.ns_stride + s;
                p.part_acc[row * D + i % D] = 0.f;
                if (i % D == 0) {
                    p.part_m[row] = -INFINITY;
                    p.part_l[row] = 0.f;
                }
            }
        } else if (n == 0 && s == 0) {
            T* o = reinterpret_cast<T*>(p.out) + ((size_t)b * p.Hq + h0) * D;
            for (int i = threadIdx.x; i < p.G * D; i += blockDim.x) o[i] = from_float<T>(0.f);
        }
        return;
    }

    if (threadIdx.x == 0) {
        for (int i = 0; i < STAGES; ++i) {
            mbar_init(&full[i], 1);
            mbar_init(&empty[i], 1);
        }
        fence_barrier_init();
        *abort_flag = 0;
    }
    __syncthreads();

    const int pg0 = t0 / BS;                        // first page of the split (sequence-relative)
    const int npg = (t1 + BS - 1) / BS - pg0;       // pages in the split
    const int32_t* trow = p.table + (size_t)b * p.MBPS + pg0;

    if (warp == NWC) {
        // ------------------------------------------------------------ producer
        const uint64_t pol = policy_evict_first();
        if (lane == 0) {
            prefetch_tensormap(&tmk);
            prefetch_tensormap(&tmv);
        }
        int id_cur = lane < npg ? trow[lane] : 0;
        int id_nxt = 32 + lane < npg ? trow[32 + lane] : 0;
        bool ok = true;
        int issued = 0;
        for (int i = 0; i < npg; ++i) {
            const int stg = i % STAGES;
            if (i >= STAGES) {
                const bool got = mbar_wait(&empty[stg], ((i / STAGES) - 1) & 1);
                if (!__all_sync(0xffffffffu, got && *abort_flag == 0)) {
                    ok = false;
                    *abort_flag = 1;
                    break;
                }
            }
            int phys = __shfl_sync(0xffffffffu, id_cur, i & 31);
            phys = (phys < 0 || phys >= p.NB) ? 0 : phys;   // bad entries never leave the pool
            if (lane == 0) {
                uint8_t* kd = ring + stg * 2 * SLICE;
                uint8_t* vd = kd + SLICE;
                const int z = phys * p.Hkv + kvh;
                mbar_arrive_expect_tx(&full[stg], 2 * SLICE);
                if (LAYOUT == kLayoutNHD) {
#pragma unroll
                    for (int j = 0; j < D / 64; ++j) {
                        tma_load_3d(kd + j * BS * 128, &tmk, &full[stg], j * 64, 0, z, pol);
                        tma_load_3d(vd + j * BS * 128, &tmv, &full[stg], j * 64, 0, z, pol);
                    }
                } else {
                    tma_load_3d(kd, &tmk, &full[stg], 0, 0, z, pol);
                    tma_load_3d(vd, &tmv, &full[stg], 0, 0, z, pol);
                }
            }
            issued = i + 1;
            if ((i & 31) == 31) {
                id_cur = id_nxt;
                const int j = i + 33 + lane;
                id_nxt = j < npg ? trow[j] : 0;
            }
        }
        // Never leave with copies in flight into this CTA's shared memory.
        for (int i = max(0, issued - STAGES); i < issued; ++i)
            if (!mbar_wait(&full[i % STAGES], (i / STAGES) & 1)) ok = false;
        if (!ok && lane == 0 && p.err) atomicOr(p.err, kErrTimeout);
        return;
    }

    // ---------------------------------------------------------------- consumers
    uint32_t qf[NT][KT][2];
    {
        const T* qb = reinterpret_cast<const T*>(p.q) + ((size_t)b * p.Hq + h0) * D;
#pragma unroll
        for (int nt = 0; nt < NT; ++nt) {
            const int hh = nt * 8 + (lane >> 2);
#pragma unroll
            for (int kk = 0; kk < KT; ++kk) {
                if (hh < p.G) {
                    const uint32_t* qr = reinterpret_cast<const uint32_t*>(qb + hh * D + kk * 16 + 2 * (lane & 3));
                    qf[nt][kk][0] = qr[0];
                    qf[nt][kk][1] = qr[4];
                } else {
                    qf[nt][kk][0] = 0u;
                    qf[nt][kk][1] = 0u;
                }
            }
        }
    }

    float acc[KT][NT][4];
    float mrun[NT][2], lrun[NT][2];
#pragma unroll
    for (int dt = 0; dt < KT; ++dt)
#pragma unroll
        for (int nt = 0; nt < NT; ++nt)
#pragma unroll
            for (int e = 0; e < 4; ++e) acc[dt][nt][e] = 0.f;
#pragma unroll
    for (int nt = 0; nt < NT; ++nt) {
        mrun[nt][0] = mrun[nt][1] = -INFINITY;
        lrun[nt][0] = lrun[nt][1] = 0.f;
    }

    const int last_pg = (n - 1) / BS;
    const int mi = lane >> 3, r8 = lane & 7;   // ldmatrix: matrix index and row within it
    bool ok = true;

    for (int i = warp; i < npg; i += NWC) {
        const int stg = i % STAGES;
        const bool got = mbar_wait(&full[stg], (i / STAGES) & 1);
        if (!__all_sync(0xffffffffu, got && *abort_flag == 0)) {
            ok = false;
            *abort_flag = 1;
            break;
        }
        uint8_t* ks = ring + stg * 2 * SLICE;
        uint8_t* vs = ks + SLICE;
        const uint32_t ks_a = smem_u32(ks), vs_a = smem_u32(vs);
        const int valid = (pg0 + i == last_pg) ? n - last_pg * BS : BS;

        // S^T = K . Q^T  (16 tokens x 8 heads per n-tile)
        float sc[NT][4];
#pragma unroll
        for (int nt = 0; nt < NT; ++nt) sc[nt][0] = sc[nt][1] = sc[nt][2] = sc[nt][3] = 0.f;
#pragma unroll
        for (int kk = 0; kk < KT; ++kk) {
            uint32_t a[4];
            const int t = r8 + ((mi & 1) << 3);
            const int c = kk * 2 + (mi >> 1);
            if (LAYOUT == kLayoutNHD)
                ldsm_x4(ks_a + nhd_off<BS>(t, c), a);
            else
                ldsm_x4(ks_a + (uint32_t)(c * BS * 16 + t * 16), a);
#pragma unroll
            for (int nt = 0; nt < NT; ++nt) Mma<T>::run(sc[nt], a, qf[nt][kk][0], qf[nt][kk][1]);
        }

        // scale to log2 units, mask tokens past the context (select, so a NaN
        // in an unread slot cannot leak), online-softmax update
        const int tr = lane >> 2;
#pragma unroll
        for (int nt = 0; nt < NT; ++nt) {
#pragma unroll
            for (int e = 0; e < 4; ++e) {
                const int t = tr + ((e >> 1) << 3);
                sc[nt][e] = t < valid ? sc[nt][e] * p.scale_log2 : -INFINITY;
            }
#pragma unroll
            for (int j = 0; j < 2; ++j) {
                float mx = fmaxf(sc[nt][j], sc[nt][j + 2]);
                mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 4));
                mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 8));
                mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 16));
                const float mnew = fmaxf(mrun[nt][j], mx);
                const float alpha = ex2(mrun[nt][j] - mnew);
                mrun[nt][j] = mnew;
                sc[nt][j] = ex2(sc[nt][j] - mnew);
                sc[nt][j + 2] = ex2(sc[nt][j + 2] - mnew);
                lrun[nt][j] = lrun[nt][j] * alpha + (sc[nt][j] + sc[nt][j + 2]);
#pragma unroll
                for (int dt = 0; dt < KT; ++dt) {
                    acc[dt][nt][j] *= alpha;
                    acc[dt][nt][j + 2] *= alpha;
                }
            }
        }

        // P^T as the B operand: transpose the two 8x8 (token x head) halves.
        uint32_t pb[NT][2];
#pragma unroll
        for (int nt = 0; nt < NT; ++nt) {
            pb[nt][0] = movmatrix_trans(Mma<T>::pack(sc[nt][0], sc[nt][1]));
            pb[nt][1] = movmatrix_trans(Mma<T>::pack(sc[nt][2], sc[nt][3]));
        }

        // Zero the V rows past the context on the sequence's last page so
        // that P = 0 times whatever they hold stays 0.
        if (valid < BS) {
            if (LAYOUT == kLayoutNHD) {
                const int chunks = (BS - valid) * (D / 8);
                for (int c = lane; c < chunks; c += 32) {
                    const int t = valid + c / (D / 8);
                    const int rem = c % (D / 8);
                    *reinterpret_cast<uint4*>(vs + (rem >> 3) * (BS * 128) + t * 128 + ((rem & 7) << 4)) =
                        make_uint4(0u, 0u, 0u, 0u);
                }
            } else {
                for (int d = lane; d < D; d += 32)
                    for (int t = valid; t < BS; ++t) reinterpret_cast<uint16_t*>(vs)[d * BS + t] = 0;
            }
            fence_proxy_async_smem();
            __syncwarp();
        }

        // O^T += V^T . P^T
#pragma unroll
        for (int dt = 0; dt < KT; ++dt) {
            uint32_t a[4];
            if (LAYOUT == kLayoutNHD) {
                const int t = r8 + ((mi >> 1) << 3);
                const int c = dt * 2 + (mi & 1);
                ldsm_x4_trans(vs_a + nhd_off<BS>(t, c), a);
            } else {
                const int d = dt * 16 + r8 + ((mi & 1) << 3);
                const int jc = mi >> 1;
                ldsm_x4(vs_a + (uint32_t)(d * BS * 2 + jc * 16), a);
            }
#pragma unroll
            for (int nt = 0; nt < NT; ++nt) Mma<T>::run(acc[dt][nt], a, pb[nt][0], pb[nt][1]);
        }
        __syncwarp();
        if (lane == 0) mbar_arrive(&empty[stg]);
    }
    if (!ok && lane == 0 && p.err) atomicOr(p.err, kErrTimeout);

    // ------------------------------------------------- merge the warps' states
#pragma unroll
    for (int nt = 0; nt < NT; ++nt)
#pragma unroll
        for (int j = 0; j < 2; ++j) {
            float l = lrun[nt][j];
            l += __shfl_xor_sync(0xffffffffu, l, 4);
            l += __shfl_xor_sync(0xffffffffu, l, 8);
            l += __shfl_xor_sync(0xffffffffu, l, 16);
            lrun[nt][j] = l;
        }
    if (lane < 4) {
#pragma unroll
        for (int nt = 0; nt < NT; ++nt)
#pragma unroll
            for (int j = 0; j < 2; ++j) {
                st_m[warp * HP + nt * 8 + 2 * lane + j] = mrun[nt][j];
                st_l[warp * HP + nt * 8 + 2 * lane + j] = lrun[nt][j];
            }
    }
    named_bar_sync(1, NWC * 32);   // every consumer is past its last page

    float* red = reinterpret_cast<float*>(ring);
#pragma unroll
    for (int nt = 0; nt < NT; ++nt)
#pragma unroll
        for (int j = 0; j < 2; ++j) {
            const int h = nt * 8 + 2 * (lane & 3) + j;
            float M = -INFINITY;
#pragma unroll
            for (int w = 0; w < NWC; ++w) M = fmaxf(M, st_m[w * HP + h]);
            const float f = ex2(mrun[nt][j] - M);   // 0 for a warp that saw no page
            float* row = red + (warp * HP + h) * RS + (lane >> 2);
#pragma unroll
            for (int dt = 0; dt < KT; ++dt) {
                row[dt * 16] = acc[dt][nt][j] * f;
                row[dt * 16 + 8] = acc[dt][nt][j + 2] * f;
            }
        }
    named_bar_sync(1, NWC * 32);

    const bool direct = !p.partials_only && ns_b == 1;
    for (int idx = threadIdx.x; idx < p.G * (D / 4); idx += NWC * 32) {
        const int h = idx / (D / 4);
        const int d = (idx % (D / 4)) * 4;
        float M = -INFINITY;
#pragma unroll
        for (int w = 0; w < NWC; ++w) M = fmaxf(M, st_m[w * HP + h]);
        float L = 0.f;
        float4 sum = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
        for (int w = 0; w < NWC; ++w) {
            L += st_l[w * HP + h] * ex2(st_m[w * HP + h] - M);
            const float4 v = *reinterpret_cast<const float4*>(red + (w * HP + h) * RS + d);
            sum.x += v.x;
            sum.y += v.y;
            sum.z += v.z;
            sum.w += v.w;
        }
        const size_t bh = (size_t)b * p.Hq + h0 + h;
        if (direct) {
            const float inv = 1.f / L;
            T o4[4] = {from_float<T>(sum.x * inv), from_float<T>(sum.y * inv), from_float<T>(sum.z * inv),
                       from_float<T>(sum.w * inv)};
            *reinterpret_cast<uint2*>(reinterpret_cast<T*>(p.out) + bh * D + d) = *reinterpret_cast<uint2*>(o4);
        } else {
            const size_t row = bh * p.ns_stride + s;
            *reinterpret_cast<float4*>(p.part_acc + row * D + d) = sum;
            if (d == 0) {
                p.part_m[row] = M * 0.69314718055994531f;   // log2 units -> natural-log units
                p.part_l[row] = L;
            }
        }
    }
}

// Host-side launcher for one instantiation.
template <typename T, int LAYOUT, int D, int NT>
cudaError_t launch_decode_phase1(const DecodeParams& p, const CUtensorMap& tmk, const CUtensorMap& tmv,
                                 cudaStream_t stream) {
    using Tile = DecodeTile<D>;
    auto kern = decode_phase1_kernel<T, LAYOUT, D, NT>;
    const int smem = Tile::smem_bytes(NT);
    static bool attr_set[64] = {};
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if (dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
    if (!attr_set[dev]) {
        e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
        if (e != cudaSuccess) return e;
        attr_set[dev] = true;
    }
    const long long grid = (long long)p.B * p.Hkv * p.NS;
    kern<<<(unsigned)grid, (Tile::NWC + 1) * 32, smem, stream>>>(p, tmk, tmv);
    return cudaGetLastError();
}

}  // namespace pkv
