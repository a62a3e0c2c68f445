// mla.cu -- MLA paged causal prefill on sm_103a tensor cores (tcgen05 + TMEM).
//
// Problem (kernelindex.com "flashinfer gemini-2.5-pro triton xvhq2i",
// mla_paged_prefill_causal_h16_ckv512_kpe64_ps1, sections 2-4): for query
// token t of sequence b and head h,
//   logit_j = sm_scale * (q_nope[t][h] . ckv[page_j] + q_pe[t][h] . kpe[page_j]),
//   visible keys j <= prefix + (t - qo_indptr[b]), prefix = kv_len - q_len,
//   out[t][h] = softmax(logit) . ckv,   lse[t][h] = log2 sum_j exp(logit_j).
//
// The page computes this in two passes (an LSE pass, then a pass that
// recomputes every logit); here it is one online-softmax pass on the tensor
// cores, with the 16 heads of 8 query tokens stacked into one 128-row tile
// that shares each gathered key row.
//
// CTA = (sequence, 8-token row tile, half of the 512 output columns).  TMEM
// (512 columns x 128 lanes, fp32) holds two S tiles of 128 keys (double
// buffer) and the CTA's 256 output columns, which is why the output is split
// across two CTAs that each recompute S.  Shared memory holds the whole Q
// tile (9 chunks of 128 rows x 64 bf16 = 144 KB), a 3-stage ring of 16 KB
// key chunks (128 gathered rows x 64 bf16) and the bf16 P tile (32 KB), all
// in the 128-byte-swizzled layout the UMMA descriptors describe.  A ckv chunk
// serves as the K-major B operand of S = Q.K^T and, re-described MN-major,
// as the B operand V of O = P.V.
//
// Warps: 0 = producer (cp.async gathers rows through kv_indices, zero-filling
// rows past the visible range); 1 = TMEM allocator and single-thread MMA
// issuer; 2..5 = softmax (one thread per row / TMEM lane): online max/sum in
// log2 units, lazy O rescaling (only when the running max grows by more than
// 8, i.e. a factor 256), P written as bf16, final O / l and the base-2 LSE.
#include "internal.h"
#include "tcgen05.cuh"

namespace pkv {

namespace mla {
constexpr int kHeads = 16, kDc = 512, kDr = 64;
constexpr int kTok = 8;                 // query tokens per row tile
constexpr int kRows = kTok * kHeads;    // 128 TMEM lanes
constexpr int kKeys = 128;              // keys per block
constexpr int kChunk = kRows * 64 * 2;  // 16 KB: 128 rows x 64 bf16
constexpr int kQChunks = 9;             // 8 x ckv + 1 x kpe
constexpr int kVChunks = 4;             // 256 output columns / 64
constexpr int kStages = 3;
constexpr int kThreads = 192;
constexpr int kBars = 2 * kStages + 8;
constexpr int kSmemBytes = 1024 + (kQChunks + kStages + 2) * kChunk + kBars * 8 + 2 * kKeys * 4 + 16;
constexpr float kLazyRescale = 8.f;     // log2 units
}  // namespace mla


__global__ void __launch_bounds__(mla::kThreads, 1) mla_prefill_kernel(const MlaParams p) {
    using namespace mla;
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    uint8_t* sQ = smem;
    uint8_t* sRing = sQ + kQChunks * kChunk;
    uint8_t* sP = sRing + kStages * kChunk;
    uint64_t* bars = reinterpret_cast<uint64_t*>(sP + 2 * kChunk);
    uint64_t* ring_full = bars;
    uint64_t* ring_empty = bars + kStages;
    uint64_t* q_full = bars + 2 * kStages;
    uint64_t* s_full = q_full + 1;     // [2]
    uint64_t* s_free = s_full + 2;     // [2]
    uint64_t* p_full = s_free + 2;
    uint64_t* p_free = p_full + 1;
    uint64_t* mma_done = p_free + 1;
    int32_t* s_pages = reinterpret_cast<int32_t*>(bars + kBars);   // [2][kKeys]
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(s_pages + 2 * kKeys);
    volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int half = blockIdx.x & 1;
    const int tile = blockIdx.x >> 1;

    // Row tile -> (sequence, first token).  Within a sequence the tiles are
    // visited last-token-first so the tiles with the most keys start first.
    int b = -1, i0 = 0;
    for (int bb = 0, acc = 0; bb < p.batch; ++bb) {
        const int nt = (p.qo_indptr[bb + 1] - p.qo_indptr[bb] + kTok - 1) / kTok;
        if (tile < acc + nt) {
            b = bb;
            i0 = (nt - 1 - (tile - acc)) * kTok;
            break;
        }
        acc += nt;
    }
    if (b < 0) return;
    const int q0 = p.qo_indptr[b], q_len = p.qo_indptr[b + 1] - q0;
    const int kv0 = p.kv_indptr[b], kv_len = p.kv_indptr[b + 1] - kv0;
    const int prefix = kv_len - q_len;
    const int ntok = min(kTok, q_len - i0);
    // keys any row of the tile may see (none when the pool is empty)
    const int n_keys = p.num_pages > 0 ? max(0, min(kv_len, prefix + i0 + ntok)) : 0;
    const int J = (n_keys + kKeys - 1) / kKeys;

    if (J == 0) {   // no visible key (empty KV): out = 0, lse = -inf
        for (int i = threadIdx.x; i < ntok * kHeads * 32; i += blockDim.x) {
            const int r = i / 32, c = i % 32;
            const size_t t = (size_t)(q0 + i0 + r / kHeads);
            reinterpret_cast<uint4*>(p.out + (t * kHeads + r % kHeads) * kDc + half * 256)[c] =
                make_uint4(0u, 0u, 0u, 0u);
            if (half == 0 && c == 0) p.lse[t * kHeads + r % kHeads] = -INFINITY;
        }
        return;
    }

    if (threadIdx.x == 0) {
        for (int i = 0; i < kStages; ++i) {
            mbar_init(&ring_full[i], 32);
            mbar_init(&ring_empty[i], 1);
        }
        mbar_init(q_full, 32);
        for (int i = 0; i < 2; ++i) {
            mbar_init(&s_full[i], 1);
            mbar_init(&s_free[i], 128);
        }
        mbar_init(p_full, 128);
        mbar_init(p_free, 1);
        mbar_init(mma_done, 1);
        fence_barrier_init();
        *abort_flag = 0;
    }
    if (warp == 1) {
        tmem_alloc(tmem_slot, 512);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tmem_slot;

    if (warp == 0) {
        // ------------------------------------------------------------ producer
        const __nv_bfloat16* qn_base = p.q_nope + (size_t)(q0 + i0) * kHeads * kDc;
        const __nv_bfloat16* qp_base = p.q_pe + (size_t)(q0 + i0) * kHeads * kDr;
        for (int idx = lane; idx < kRows * kQChunks * 8; idx += 32) {
            const int r = idx / (kQChunks * 8), rem = idx % (kQChunks * 8);
            const int c = rem >> 3, piece = rem & 7;
            const bool ok = r / kHeads < ntok;
            const __nv_bfloat16* src = c < 8 ? qn_base + (size_t)r * kDc + c * 64 + piece * 8
                                             : qp_base + (size_t)r * kDr + piece * 8;
            cp_async16(smem_u32(sQ + c * kChunk + r * 128 + ((piece ^ (r & 7)) << 4)), ok ? src : p.q_nope,
                       ok ? 16u : 0u);
        }
        cp_async_commit();
        cp_async_wait<0>();
        fence_proxy_async_smem();
        mbar_arrive(q_full);

        bool ok = true;
        int k = 0;   // running chunk index (same order as the MMA issuer consumes them)
        auto retire = [&](int kk) {
            fence_proxy_async_smem();
            mbar_arrive(&ring_full[kk % kStages]);
        };
        auto load_chunk = [&](int jb, int c) -> bool {
            const int stage = k % kStages;
            if (k >= kStages) {
                const bool got = mbar_wait(&ring_empty[stage], ((k / kStages) - 1) & 1);
                if (!__all_sync(0xffffffffu, got && *abort_flag == 0)) return false;
            }
            const int32_t* pages = s_pages + (jb & 1) * kKeys;
            uint8_t* dst = sRing + stage * kChunk;
            for (int idx = lane; idx < kKeys * 8; idx += 32) {
                const int row = idx >> 3, piece = idx & 7;
                const bool live = jb * kKeys + row < n_keys;
                const int page = pages[row];
                const __nv_bfloat16* src = c < 8 ? p.ckv + (size_t)page * kDc + c * 64 + piece * 8
                                                 : p.kpe + (size_t)page * kDr + piece * 8;
                cp_async16(smem_u32(dst + row * 128 + ((piece ^ (row & 7)) << 4)), live ? src : p.ckv,
                           live ? 16u : 0u);
            }
            cp_async_commit();
            if (k >= kStages - 1) {
                cp_async_wait<kStages - 1>();
                retire(k - (kStages - 1));
            }
            ++k;
            return true;
        };
        for (int step = 0; step <= J && ok; ++step) {
            if (step < J) {
                // page ids of key block `step` (clamped into the pool)
                __syncwarp();
                for (int row = lane; row < kKeys; row += 32) {
                    const int key = step * kKeys + row;
                    int pg = key < n_keys ? p.kv_indices[kv0 + key] : 0;
                    pg = (pg < 0 || pg >= p.num_pages) ? 0 : pg;
                    s_pages[(step & 1) * kKeys + row] = pg;
                }
                __syncwarp();
                for (int c = 0; c < kQChunks && ok; ++c) ok = load_chunk(step, c);
            }
            if (step >= 1)
                for (int v = 0; v < kVChunks && ok; ++v) ok = load_chunk(step - 1, half * kVChunks + v);
        }
        cp_async_wait<0>();
        if (ok)
            for (int kk = max(0, k - (kStages - 1)); kk < k; ++kk) retire(kk);
        else
            *abort_flag = 1;
    } else if (warp == 1) {
        // ----------------------------------------------------------- MMA issuer
        if (lane == 0) {
            const uint32_t idesc_qk = umma_idesc_bf16_f32(kRows, kKeys, false);
            const uint32_t idesc_pv = umma_idesc_bf16_f32(kRows, 64, true);
            const uint32_t q_addr = smem_u32(sQ), ring_addr = smem_u32(sRing), p_addr = smem_u32(sP);
            bool ok = mbar_wait(q_full, 0);
            tc_fence_after();
            int k = 0;
            for (int step = 0; step <= J && ok; ++step) {
                if (step < J) {
                    const int sb = step & 1;
                    if (step >= 2) {
                        ok = mbar_wait(&s_free[sb], ((step >> 1) - 1) & 1) && *abort_flag == 0;
                        tc_fence_after();
                    }
                    for (int c = 0; c < kQChunks && ok; ++c, ++k) {
                        const int stage = k % kStages;
                        ok = mbar_wait(&ring_full[stage], (k / kStages) & 1) && *abort_flag == 0;
                        tc_fence_after();
                        if (!ok) break;
#pragma unroll
                        for (int kk = 0; kk < 4; ++kk)
                            umma_bf16(tmem + sb * kKeys,
                                      umma_desc_sw128(q_addr + c * kChunk + kk * 32, 16, 1024),
                                      umma_desc_sw128(ring_addr + stage * kChunk + kk * 32, 16, 1024), idesc_qk,
                                      (c | kk) != 0);
                        umma_commit(&ring_empty[stage]);
                    }
                    if (ok) umma_commit(&s_full[sb]);
                }
                if (step >= 1 && ok) {
                    const int jb = step - 1;
                    ok = mbar_wait(p_full, jb & 1) && *abort_flag == 0;
                    tc_fence_after();
                    for (int v = 0; v < kVChunks && ok; ++v, ++k) {
                        const int stage = k % kStages;
                        ok = mbar_wait(&ring_full[stage], (k / kStages) & 1) && *abort_flag == 0;
                        tc_fence_after();
                        if (!ok) break;
#pragma unroll
                        for (int kk = 0; kk < kKeys / 16; ++kk)
                            umma_bf16(tmem + 2 * kKeys + v * 64,
                                      umma_desc_sw128(p_addr + (kk >> 2) * kChunk + (kk & 3) * 32, 16, 1024),
                                      umma_desc_sw128(ring_addr + stage * kChunk + kk * 2048, kChunk, 1024),
                                      idesc_pv, jb > 0 || kk > 0);
                        umma_commit(&ring_empty[stage]);
                    }
                    if (ok) umma_commit(p_free);
                }
            }
            if (!ok) *abort_flag = 1;
            // never release TMEM with MMAs in flight
            umma_commit(mma_done);
            mbar_wait(mma_done, 0);
        }
        __syncwarp();
    } else {
        // ------------------------------------------------------------- softmax
        const int quad = warp & 3;
        const int row = quad * 32 + lane;
        const int tok = i0 + row / kHeads;
        const int lim = prefix + tok;   // last visible key of this row
        const uint32_t t_row = tmem + ((uint32_t)(quad * 32) << 16);
        float m = -INFINITY, l = 0.f;
        bool ok = true;
        for (int j = 0; j < J; ++j) {
            const int sb = j & 1;
            const bool got = mbar_wait(&s_full[sb], (j >> 1) & 1);
            if (!__all_sync(0xffffffffu, got && *abort_flag == 0)) {
                ok = false;
                break;
            }
            tc_fence_after();
            float s[kKeys];
#pragma unroll
            for (int c = 0; c < kKeys / 32; ++c) {
                float v[32];
                tmem_ld32(t_row + sb * kKeys + c * 32, v);
                tmem_wait_ld();
#pragma unroll
                for (int i = 0; i < 32; ++i) s[c * 32 + i] = v[i];
            }
            tc_fence_before();
            mbar_arrive(&s_free[sb]);

            float mx = -INFINITY;
#pragma unroll
            for (int c = 0; c < kKeys; ++c) {
                const int key = j * kKeys + c;
                s[c] = (key <= lim && key < n_keys) ? s[c] * p.scale_log2 : -INFINITY;
                mx = fmaxf(mx, s[c]);
            }
            const float m_new = fmaxf(m, mx);
            float m_use = m, alpha = 1.f;
            if (m == -INFINITY || m_new > m + kLazyRescale) {
                m_use = m_new == -INFINITY ? 0.f : m_new;
                alpha = ex2(m - m_use);
            }
            float ls = 0.f;
#pragma unroll
            for (int c = 0; c < kKeys; ++c) {
                s[c] = ex2(s[c] - m_use);
                ls += s[c];
            }
            l = l * alpha + ls;
            m = m_use;

            if (j >= 1) {
                // P(j-1) has been consumed and O holds it: rescale O, reuse P.
                const bool got2 = mbar_wait(p_free, (j - 1) & 1);
                if (!__all_sync(0xffffffffu, got2 && *abort_flag == 0)) {
                    ok = false;
                    break;
                }
                tc_fence_after();
                if (__any_sync(0xffffffffu, alpha != 1.f)) {
#pragma unroll 1
                    for (int c = 0; c < 256 / 32; ++c) {
                        float o[32];
                        tmem_ld32(t_row + 2 * kKeys + c * 32, o);
                        tmem_wait_ld();
#pragma unroll
                        for (int i = 0; i < 32; ++i) o[i] *= alpha;
                        tmem_st32(t_row + 2 * kKeys + c * 32, o);
                    }
                    tmem_wait_st();
                }
            }
#pragma unroll
            for (int pc = 0; pc < kKeys / 8; ++pc) {
                uint4 v;
                v.x = Mma<__nv_bfloat16>::pack(s[pc * 8 + 0], s[pc * 8 + 1]);
                v.y = Mma<__nv_bfloat16>::pack(s[pc * 8 + 2], s[pc * 8 + 3]);
                v.z = Mma<__nv_bfloat16>::pack(s[pc * 8 + 4], s[pc * 8 + 5]);
                v.w = Mma<__nv_bfloat16>::pack(s[pc * 8 + 6], s[pc * 8 + 7]);
                const int khalf = pc >> 3, piece = pc & 7;
                *reinterpret_cast<uint4*>(sP + khalf * kChunk + row * 128 + ((piece ^ (row & 7)) << 4)) = v;
            }
            fence_proxy_async_smem();
            tc_fence_before();
            mbar_arrive(p_full);
        }
        if (ok) {
            const bool got = mbar_wait(p_free, (J - 1) & 1);
            ok = __all_sync(0xffffffffu, got && *abort_flag == 0);
            tc_fence_after();
        }
        if (ok) {
            const bool live = row / kHeads < ntok;
            const size_t t = (size_t)(q0 + tok);
            const int h = row % kHeads;
            const float inv = l > 0.f ? 1.f / l : 0.f;
            __nv_bfloat16* orow = p.out + (t * kHeads + h) * kDc + half * 256;
#pragma unroll 1
            for (int c = 0; c < 256 / 32; ++c) {
                float o[32];
                tmem_ld32(t_row + 2 * kKeys + c * 32, o);
                tmem_wait_ld();
                if (live) {
#pragma unroll
                    for (int q4 = 0; q4 < 4; ++q4) {
                        uint4 v;
                        v.x = Mma<__nv_bfloat16>::pack(o[q4 * 8 + 0] * inv, o[q4 * 8 + 1] * inv);
                        v.y = Mma<__nv_bfloat16>::pack(o[q4 * 8 + 2] * inv, o[q4 * 8 + 3] * inv);
                        v.z = Mma<__nv_bfloat16>::pack(o[q4 * 8 + 4] * inv, o[q4 * 8 + 5] * inv);
                        v.w = Mma<__nv_bfloat16>::pack(o[q4 * 8 + 6] * inv, o[q4 * 8 + 7] * inv);
                        reinterpret_cast<uint4*>(orow + c * 32)[q4] = v;
                    }
                }
            }
            if (live && half == 0) p.lse[t * kHeads + h] = l > 0.f ? m + log2f(l) : -INFINITY;
        } else {
            *abort_flag = 1;
        }
    }

    tc_fence_before();
    __syncthreads();
    if (warp == 1) {
        tc_fence_after();
        tmem_dealloc(tmem, 512);
    }
}

cudaError_t launch_mla_prefill(const MlaParams& p, cudaStream_t stream) {
    static bool attr_set[64] = {};
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if (dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
    if (!attr_set[dev]) {
        e = cudaFuncSetAttribute(mla_prefill_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, mla::kSmemBytes);
        if (e != cudaSuccess) return e;
        attr_set[dev] = true;
    }
    const long long tiles = (long long)(p.total_q + mla::kTok - 1) / mla::kTok + p.batch;
    if (tiles <= 0) return cudaSuccess;
    mla_prefill_kernel<<<(unsigned)(2 * tiles), mla::kThreads, mla::kSmemBytes, stream>>>(p);
    return cudaGetLastError();
}

}  // namespace pkv
