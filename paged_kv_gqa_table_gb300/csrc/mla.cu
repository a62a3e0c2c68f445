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
// (512 columns x 128 lanes, fp32) holds the CTA's 256 output columns O, one
// S tile of 128 keys and two bf16 P tiles (the A operand of O += P.V, read
// from TMEM), which is why the output is split across two CTAs that each
// recompute S.  Shared memory holds the whole Q tile (9 chunks of 128 rows x
// 64 bf16 = 144 KB, one 2-D TMA box each) and a 5-stage ring of 16 KB
// chunks, all in the 128-byte-swizzled layout the UMMA descriptors describe.
// Per block of 128 keys the ring carries 9 K chunks (128 keys x 64 columns,
// the K-major B operand of S = Q.K^T, N = 128) and 4 V chunks (32 keys x the
// CTA's 256 output columns as four 64-column blocks 4 KB apart, the MN-major
// B operand of O += P.V, N = 256).  Both are cut from the same staged ckv
// rows.
//
// Page size 1 makes every key its own page.  Gathering 128-byte row pieces
// per tile (up to ~100 tiles read each key) keeps too few bytes in flight
// per TMA operation, so mla_stage_kernel first copies each referenced row
// (ckv | kpe, 1152 bytes) once into a workspace, sequence by sequence, each
// sequence padded with zero rows to a multiple of 128 rows; the attention
// kernel then loads 128 consecutive staged rows per 16 KB box.  A box never
// leaves its sequence's staged rows, as the page's kernel never loads a key
// outside [kv_pages_start, kv_pages_end): rows of a box past the tile's
// keys are the sequence's own later keys or zero rows, masked in the
// softmax, so another sequence's cache rows cannot reach this output.
//
// Warps: 0 = producer (one thread issues the Q boxes and then, after the
// staging grid has completed, the key boxes); 1 = TMEM allocator and
// single-thread MMA issuer;
// 2..5 = softmax (one thread per row / TMEM lane): online max/sum in log2
// units, lazy O rescaling (only when the running max grows by more than 8,
// i.e. a factor 256), P stored to TMEM as bf16, final O / l and the base-2
// LSE.
#include <algorithm>

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
constexpr int kVChunks = 4;             // 128 keys / 32 keys per V chunk
constexpr int kStages = 5;
constexpr int kThreads = 192;
constexpr int kBars = 2 * kStages + 8;
constexpr int kSmemBytes = 1024 + (kQChunks + kStages) * kChunk + kBars * 8 + 16;
constexpr uint32_t kColS = 256, kColP = 384;   // TMEM columns: O [0,256), S [256,384), P x2 [384,512)
constexpr float kLazyRescale = 8.f;     // log2 units
}  // namespace mla


// Staged rows of sequence b: its kv_len keys rounded up to kMlaSeqAlign rows.
__device__ __forceinline__ int mla_padded_len(const MlaParams& p, int b) {
    const int kv_len = max(0, p.kv_indptr[b + 1] - p.kv_indptr[b]);
    return (kv_len + kMlaSeqAlign - 1) / kMlaSeqAlign * kMlaSeqAlign;
}

// Sequence b's keys are staged at rows [off_b, off_b + kv_len_b), off_b the
// sum of the earlier sequences' padded lengths: staged[off_b + j] =
// ckv[kv_indices[kv_indptr[b] + j]] | kpe[...], then zero rows up to the next
// multiple of kMlaSeqAlign, so a 128-row box of one sequence never reaches the
// next sequence's keys.  Keys whose kv_indices entry lies past nnz are staged
// as zero rows (and reported); rows past stage_rows are not written (their
// boxes read the tensor map's zero fill).  One warp per row; each warp walks
// the sequences forward as its rows advance.
__global__ void __launch_bounds__(256) mla_stage_kernel(const MlaParams p) {
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
    if (blockIdx.x == 0 && threadIdx.x == 0 && p.kv_indptr[p.batch] > p.nnz) atomicOr(p.err, 2u);
    const int lane = threadIdx.x & 31;
    const long long warps = (long long)gridDim.x * (blockDim.x >> 5);
    const uint4 zero = make_uint4(0u, 0u, 0u, 0u);
    int b = 0;
    long long off = 0;   // first staged row of sequence b
    int pad = p.batch > 0 ? mla_padded_len(p, 0) : 0;
    for (long long r = (long long)blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5); r < p.stage_rows;
         r += warps) {
        while (b < p.batch && r >= off + pad) {
            off += pad;
            if (++b < p.batch) pad = mla_padded_len(p, b);
        }
        if (b >= p.batch) break;
        const int j = (int)(r - off);
        const int kv0 = p.kv_indptr[b];
        const int kv_len = p.kv_indptr[b + 1] - kv0;
        uint4* dst = reinterpret_cast<uint4*>(p.stage + (size_t)r * kMlaStageRowBytes);
        uint4 a = zero, c = zero, d = zero;
        if (j < kv_len && kv0 + j >= 0 && kv0 + j < p.nnz) {
            int pg = p.kv_indices[kv0 + j];
            pg = (pg < 0 || pg >= p.num_pages) ? 0 : pg;
            const uint4* ck = reinterpret_cast<const uint4*>(p.ckv + (size_t)pg * mla::kDc);
            const uint4* kp = reinterpret_cast<const uint4*>(p.kpe + (size_t)pg * mla::kDr);
            a = __ldg(ck + lane);
            c = __ldg(ck + 32 + lane);
            if (lane < 8) d = __ldg(kp + lane);
        }
        dst[lane] = a;
        dst[32 + lane] = c;
        if (lane < 8) dst[64 + lane] = d;
    }
}

__global__ void __launch_bounds__(mla::kThreads, 1)
    mla_prefill_kernel(const MlaParams p, const __grid_constant__ CUtensorMap tm_qn,
                       const __grid_constant__ CUtensorMap tm_qp, const __grid_constant__ CUtensorMap tm_kv,
                       const __grid_constant__ CUtensorMap tm_v) {
    using namespace mla;
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    uint8_t* sQ = smem;
    uint8_t* sRing = sQ + kQChunks * kChunk;
    uint64_t* bars = reinterpret_cast<uint64_t*>(sRing + kStages * kChunk);
    uint64_t* ring_full = bars;
    uint64_t* ring_empty = bars + kStages;
    uint64_t* q_full = bars + 2 * kStages;
    uint64_t* s_full = q_full + 1;
    uint64_t* s_free = s_full + 1;
    uint64_t* p_full = s_free + 1;     // [2]
    uint64_t* p_free = p_full + 2;     // [2]
    uint64_t* mma_done = p_free + 2;
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(bars + kBars);
    volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int half = blockIdx.x & 1;
    const int tile = blockIdx.x >> 1;

    // Row tile -> (sequence, first token).  Within a sequence the tiles are
    // visited last-token-first so the tiles with the most keys start first.
    // kv0 = the sequence's first staged row (the padded offsets of the earlier
    // sequences).
    int b = -1, i0 = 0, kv0 = 0;
    for (int bb = 0, acc = 0; bb < p.batch; ++bb) {
        const int nt = (p.qo_indptr[bb + 1] - p.qo_indptr[bb] + kTok - 1) / kTok;
        if (tile < acc + nt) {
            b = bb;
            i0 = (nt - 1 - (tile - acc)) * kTok;
            break;
        }
        acc += nt;
        kv0 += mla_padded_len(p, bb);
    }
    if (b < 0) return;
    const int q0 = p.qo_indptr[b], q_len = p.qo_indptr[b + 1] - q0;
    const int kv_len = p.kv_indptr[b + 1] - p.kv_indptr[b];
    const int prefix = kv_len - q_len;
    const int ntok = min(kTok, q_len - i0);
    // keys any row of the tile may see (none when the pool or the staging area is empty)
    const int n_keys = (p.num_pages > 0 && p.stage_rows > 0) ? max(0, min(kv_len, prefix + i0 + ntok)) : 0;
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
            mbar_init(&ring_full[i], 1);
            mbar_init(&ring_empty[i], 1);
        }
        mbar_init(q_full, 1);
        mbar_init(s_full, 1);
        mbar_init(s_free, 128);
        for (int i = 0; i < 2; ++i) {
            mbar_init(&p_full[i], 128);
            mbar_init(&p_free[i], 1);
        }
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
        if (lane == 0) {
            prefetch_tensormap(&tm_kv);
            const int y = (q0 + i0) * kHeads;   // rows past the tensor are zero-filled
            mbar_arrive_expect_tx(q_full, kQChunks * kChunk);
            for (int c = 0; c < kQChunks - 1; ++c) tma_load_2d(sQ + c * kChunk, &tm_qn, q_full, c * 64, y);
            tma_load_2d(sQ + (kQChunks - 1) * kChunk, &tm_qp, q_full, 0, y);
            // the staged keys are written by the preceding grid
            asm volatile("griddepcontrol.wait;" ::: "memory");
            bool ok = true;
            int k = 0;   // running chunk index (same order as the MMA issuer consumes them)
            // v < 0: K chunk (128 keys of block jb, columns [x, x + 64));
            // v >= 0: V chunk v (keys 32v .. 32v + 31 of block jb, the CTA's 256 columns)
            auto load_chunk = [&](int jb, int x, int v) -> bool {
                const int stage = k % kStages;
                if (k >= kStages && !(mbar_wait(&ring_empty[stage], ((k / kStages) - 1) & 1) && *abort_flag == 0))
                    return false;
                uint8_t* dst = sRing + stage * kChunk;
                mbar_arrive_expect_tx(&ring_full[stage], kChunk);
                if (v < 0) {
                    tma_load_2d(dst, &tm_kv, &ring_full[stage], x, kv0 + jb * kKeys);
                } else {
#pragma unroll
                    for (int n = 0; n < 4; ++n)
                        tma_load_2d(dst + n * 4096, &tm_v, &ring_full[stage], (half * 4 + n) * 64,
                                    kv0 + jb * kKeys + v * 32);
                }
                ++k;
                return true;
            };
            for (int step = 0; step <= J && ok; ++step) {
                if (step < J)
                    for (int c = 0; c < kQChunks && ok; ++c) ok = load_chunk(step, c * 64, -1);
                if (step >= 1)
                    for (int v = 0; v < kVChunks && ok; ++v) ok = load_chunk(step - 1, 0, v);
            }
            if (!ok) {
                *abort_flag = 1;
                atomicOr(p.err, kErrTimeout);
            }
            // Never leave with copies in flight: wait for the last fill of
            // every stage and for Q (immediate unless the pipeline aborted).
            for (int kk = max(0, k - kStages); kk < k; ++kk) mbar_wait(&ring_full[kk % kStages], (kk / kStages) & 1);
            mbar_wait(q_full, 0);
        }
        __syncwarp();
    } else if (warp == 1) {
        // ----------------------------------------------------------- MMA issuer
        if (lane == 0) {
            const uint32_t idesc_qk = umma_idesc_bf16_f32(kRows, kKeys, false);
            const uint32_t idesc_pv = umma_idesc_bf16_f32(kRows, 256, true);
            const uint32_t q_addr = smem_u32(sQ), ring_addr = smem_u32(sRing);
            bool ok = mbar_wait(q_full, 0);
            tc_fence_after();
            int k = 0;
            for (int step = 0; step <= J && ok; ++step) {
                if (step < J) {
                    if (step >= 1) {   // softmax has read S(step - 1)
                        ok = mbar_wait(s_free, (step - 1) & 1) && *abort_flag == 0;
                        tc_fence_after();
                    }
                    for (int c = 0; c < kQChunks && ok; ++c, ++k) {
                        // TMA data only: no tcgen05 fence, and no abort-flag load on this
                        // path (the issue thread's extra latency stalls the tensor pipe; a
                        // stalled pipeline ends in a timed-out wait anyway)
                        const int stage = k % kStages;
                        ok = mbar_wait(&ring_full[stage], (k / kStages) & 1);
                        if (!ok) break;
#pragma unroll
                        for (int kk = 0; kk < 4; ++kk)
                            umma_bf16(tmem + kColS, umma_desc_sw128(q_addr + c * kChunk + kk * 32, 16, 1024),
                                      umma_desc_sw128(ring_addr + stage * kChunk + kk * 32, 16, 1024), idesc_qk,
                                      (c | kk) != 0);
                        umma_commit(&ring_empty[stage]);
                    }
                    if (ok) umma_commit(s_full);
                }
                if (step >= 1 && ok) {
                    const int jb = step - 1, pb = jb & 1;
                    ok = mbar_wait(&p_full[pb], (jb >> 1) & 1) && *abort_flag == 0;
                    tc_fence_after();
                    for (int v = 0; v < kVChunks && ok; ++v, ++k) {
                        const int stage = k % kStages;
                        ok = mbar_wait(&ring_full[stage], (k / kStages) & 1);
                        if (!ok) break;
                        // keys 32v + 16kk .. +15: P columns (32v + 16kk) / 2; B = 16 key rows
                        // of the four 64-column blocks (MN-major: blocks 4 KB apart, 8-row
                        // groups 1 KB apart)
#pragma unroll
                        for (int kk = 0; kk < 2; ++kk)
                            umma_bf16_tmem_a(tmem, tmem + kColP + pb * 64 + v * 16 + kk * 8,
                                             umma_desc_sw128(ring_addr + stage * kChunk + kk * 2048, 4096, 1024),
                                             idesc_pv, (jb | v | kk) != 0);
                        umma_commit(&ring_empty[stage]);
                    }
                    if (ok) umma_commit(&p_free[pb]);
                }
            }
            if (!ok) {
                *abort_flag = 1;
                atomicOr(p.err, kErrTimeout);
            }
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
            const bool got = mbar_wait(s_full, j & 1);
            if (!__all_sync(0xffffffffu, got && *abort_flag == 0)) {
                ok = false;
                break;
            }
            tc_fence_after();
            float s[kKeys];
#pragma unroll
            for (int c = 0; c < kKeys / 32; ++c) {
                float v[32];
                tmem_ld32(t_row + kColS + c * 32, v);
                tmem_wait_ld();
#pragma unroll
                for (int i = 0; i < 32; ++i) s[c * 32 + i] = v[i];
            }
            tc_fence_before();
            mbar_arrive(s_free);

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

            const int pb = j & 1;
            bool got2 = true;
            if (j >= 1 && __any_sync(0xffffffffu, alpha != 1.f)) {
                // O holds P(j-1).V: wait for it, then rescale this warp's rows.
                got2 = mbar_wait(&p_free[pb ^ 1], ((j - 1) >> 1) & 1);
                if (__all_sync(0xffffffffu, got2 && *abort_flag == 0)) {
                    tc_fence_after();
#pragma unroll 1
                    for (int c = 0; c < 256 / 32; ++c) {
                        float o[32];
                        tmem_ld32(t_row + c * 32, o);
                        tmem_wait_ld();
#pragma unroll
                        for (int i = 0; i < 32; ++i) o[i] *= alpha;
                        tmem_st32(t_row + c * 32, o);
                    }
                    tmem_wait_st();
                }
            } else if (j >= 2) {
                // P buffer pb was last read by P(j-2).V
                got2 = mbar_wait(&p_free[pb], ((j - 2) >> 1) & 1);
                tc_fence_after();
            }
            if (!__all_sync(0xffffffffu, got2 && *abort_flag == 0)) {
                ok = false;
                break;
            }
#pragma unroll
            for (int h2 = 0; h2 < 2; ++h2) {
                uint32_t pk[32];
#pragma unroll
                for (int i = 0; i < 32; ++i)
                    pk[i] = Mma<__nv_bfloat16>::pack(s[h2 * 64 + 2 * i], s[h2 * 64 + 2 * i + 1]);
                tmem_st32(t_row + kColP + pb * 64 + h2 * 32, pk);
            }
            tmem_wait_st();
            tc_fence_before();
            mbar_arrive(&p_full[pb]);
        }
        if (ok) {
            const bool got = mbar_wait(&p_free[(J - 1) & 1], ((J - 1) >> 1) & 1);
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
                tmem_ld32(t_row + c * 32, o);
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
            if (lane == 0) atomicOr(p.err, kErrTimeout);
        }
    }

    tc_fence_before();
    __syncthreads();
    if (warp == 1) {
        tc_fence_after();
        tmem_dealloc(tmem, 512);
    }
}

cudaError_t launch_mla_prefill(const MlaParams& p, const MlaMaps& maps, cudaStream_t stream) {
    static std::atomic<bool> attr_set[kMaxDevices];
    static std::mutex attr_mu;
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    e = once_per_device(attr_set, attr_mu, dev, [] {
        return cudaFuncSetAttribute(mla_prefill_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                    mla::kSmemBytes);
    });
    if (e != cudaSuccess) return e;
    const long long tiles = (long long)(p.total_q + mla::kTok - 1) / mla::kTok + p.batch;
    if (tiles <= 0) return cudaSuccess;
    const bool staged = p.num_pages > 0 && p.stage_rows > 0;
    if (staged) {
        // one warp per staged row, capped at 16 waves of 8-warp CTAs per SM
        int sms = 0;
        e = device_sm_count(dev, &sms);
        if (e != cudaSuccess) return e;
        const long long want = ((long long)p.stage_rows + 7) / 8;
        mla_stage_kernel<<<(unsigned)std::min<long long>(want, (long long)sms * 8 * 16), 256, 0, stream>>>(p);
        e = cudaGetLastError();
        if (e != cudaSuccess) return e;
    }
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)(2 * tiles));
    cfg.blockDim = dim3(mla::kThreads);
    cfg.dynamicSmemBytes = mla::kSmemBytes;
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = staged ? 1 : 0;
    return cudaLaunchKernelEx(&cfg, mla_prefill_kernel, p, maps.q_nope, maps.q_pe, maps.kv, maps.v);
}

}  // namespace pkv
