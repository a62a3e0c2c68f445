// decode.cuh -- phase 1 of paged GQA decode attention on sm_103a.
//
// One CTA per (sequence b, KV head, row tile, split s); for FP8 caches with
// few query rows per KV head, per pair of adjacent KV heads (kLayoutNHD8x2).
// Split s covers tokens [s*P, min((s+1)*P, n)) of the sequence (fixed
// partitions as in "paged_attention_v2_triton.py", _partition_attn_kernel;
// page-granular splits as in the flash-decode post's
// _flash_decode_partial_kernel).  The
// query rows of (b, KV head) -- q_len tokens x G heads -- are the mma N
// columns, 8 * NT per CTA; more rows than that take several row tiles.
//
// Roles: warp NWC is the producer: it reads the split's block-table entries
// (32 per coalesced load, one chunk ahead) and, per page, issues TMA tensor
// loads of that page's K and V slices for this KV head into a STAGES-deep
// shared-memory ring (full/empty mbarriers).  Each page is loaded ONCE for the
// CTA's query rows.  Warps 0..NWC-1 consume pages round-robin, each keeping its
// own online-softmax state for all of them:
//
//   S^T[t][h] = K[t][:] . Q[h][:]          mma.sync m16n8k16, tokens = M (16 per
//                                           page), query rows = N (8 per tile)
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

#include <climits>
#include <type_traits>

#include "decode_common.cuh"
#include "device_plan.cuh"
#include "once.h"

namespace pkv {

struct DecodeParams {
    const void* q;           // [B][q_len][Hq][D]
    const int32_t* table;    // [B][MBPS]
    const int32_t* ctx;      // [B]
    void* out;               // [B][q_len][Hq][D]
    float* part_acc;         // [B][q_len][Hq][ns_stride][D]
    float* part_m;           // [B][q_len][Hq][ns_stride]
    float* part_l;           // [B][q_len][Hq][ns_stride]
    uint32_t* err;           // device error word or nullptr
    int B, Hq, Hkv, G, MBPS, NB;   // Hkv, G: the grid's KV heads and query heads per grid KV head
    int Hc, Gc;              // the cache's KV heads and query heads per cache KV head (Hkv = Hc / 2,
                             // G = 2 Gc for kLayoutNHD8x2, else Hc = Hkv, Gc = G)
    int q_len;               // query tokens per sequence (the last q_len positions)
    int R;                   // query rows per (sequence, KV head): G * q_len
    int RT;                  // row tiles: ceil(R / (8 * NT))
    int P;                   // tokens per split (multiple of BS)
    int NS;                  // splits in the grid
    int ns_stride;           // split extent of the partial arrays
    int n_cap;               // context lengths are clamped to [0, n_cap]
    float scale_log2;        // scale * log2(e) (times k_scale for FP8 caches)
    float v_scale;           // multiplies the output / partial acc (FP8 caches; 1 otherwise)
    const float* alibi;      // [Hq] ALiBi slopes (natural-log units) or nullptr
    int partials_only;       // 1: always write partials (+ sentinels), never out
    // Device plan (plan_hdr != nullptr): every CTA plans from ctx with `rule`
    // and takes the non-empty items blockIdx.x, blockIdx.x + gridDim.x, ...;
    // CTA 0 writes {P, splits of the longest context} to plan_hdr[0..1] for the
    // combine, and the plan's splits go to plan_tab (plan_hdr[2] of them) for
    // the calls that reuse it (plan_ready).
    int* plan_hdr;
    int4* plan_tab;          // [B * rule.NS_cap] {sequence, split, clamped context, 0} in item order
    int plan_ready;          // 1: take the items from plan_hdr / plan_tab instead of planning
    PlanRule rule;
    uint32_t stress_ns;      // producer pause after each page's copies (pkv_set_stress_delay), 0: none
    uint32_t stress_consumer_ns;   // consumer warp pause after each page, 0: none
};

template <int D, int LAYOUT>
struct DecodeTile {
    static constexpr int BS = kPageTokens;
    static constexpr int KVB = (LAYOUT == kLayoutNHD8 || LAYOUT == kLayoutNHD8x2) ? 1 : 2;   // bytes per element
    static constexpr int HEADS = LAYOUT == kLayoutNHD8x2 ? 2 : 1;   // KV heads per CTA
    // Consumer warps and ring stages.  The CTAs of a launch are short (a split),
    // and each spends its start-up (context length, table, first page) with its
    // ring empty, so more CTAs per SM with the same bytes in flight per SM keep
    // the SM streaming: at D = 128 three consumers with 6 stages (16-bit, 48 KB)
    // or 9 stages (FP8, 36 KB) give four or five CTAs per SM instead of three.
    // FP8 pages at D = 256 keep twice the 16-bit stages (the same bytes).  Head
    // pairs (8 KB stages) keep the 16-bit depth: 6 stages, four CTAs per SM.
    static constexpr int NWC = D == 128 ? 3 : 4;
    static constexpr int SLICE = BS * D * KVB * HEADS;              // bytes of one page's K (or V) in a stage
    static constexpr int STAGES =
        HEADS == 2 ? 6 : (D == 64 ? 12 : (D == 128 ? (KVB == 1 ? 9 : 6) : (KVB == 1 ? 8 : 4)));
    // FP8 pages with D = 64 are expanded to fp16 in a per-consumer-warp K/V
    // slice pair; D >= 128 goes straight from the ring into mma fragments.
    static constexpr int STAGING = (KVB == 1 && D < 128) ? NWC * 2 * BS * D * 2 : 0;
    static constexpr int RED_STRIDE = D + 4;                        // floats per reduction row
    // Two column tiles at D = 128 keep the CTA's Q fragments in shared memory
    // (one 16-row tile) instead of 32 registers per thread, so that four CTAs
    // fit on an SM (the kernel is then compiled for 4 blocks per SM).
    __host__ __device__ static constexpr bool q_shared(int nt) { return nt == 2 && D == 128; }
    // CTAs per SM the shared-Q kernels (D = 128) are compiled for (their register budget)
    static constexpr int QS_MIN_BLOCKS = 4;
    __host__ __device__ static constexpr int qtile_bytes(int nt) { return q_shared(nt) ? 16 * D * 2 : 0; }
    __host__ __device__ static constexpr int smem_bytes(int nt) {
        return 1024 + STAGES * 2 * SLICE + STAGING + qtile_bytes(nt) + STAGES * 2 * 8 + 2 * NWC * nt * 8 * 4 + 16;
    }
};

// GEN: the general kernel (several query tokens per sequence, ALiBi), compiled
// separately so that the one-token kernel without bias keeps its registers.
// SCHED (with GEN): the CTA takes the device plan's items in turn instead of
// its one grid-order item, planning them (kSchedPlan) or reading them from the
// plan an earlier call left (kSchedReuse); each compiled separately, since the
// item loops cost registers and the kernel with shared Q tiles is at its limit.
// STRESS: compiled with the pauses of pkv_set_stress_delay (race testing); the
// ordinary instantiations have none, so the test facility costs them nothing.
constexpr int kSchedGrid = 0, kSchedPlan = 1, kSchedReuse = 2;

template <typename T, int LAYOUT, int D, int NT, bool GEN, int SCHED, bool STRESS>
__device__ __forceinline__ void decode_phase1_body(const DecodeParams& p, const CUtensorMap& tmk,
                                                   const CUtensorMap& tmv) {
    static_assert(GEN || SCHED == kSchedGrid, "the device plan runs the general kernel");
    using Tile = DecodeTile<D, LAYOUT>;
    constexpr bool KV8 = LAYOUT == kLayoutNHD8 || LAYOUT == kLayoutNHD8x2;
    constexpr int HEADS = Tile::HEADS;
    constexpr bool DIRECT8 = KV8 && D >= 128;   // page_step_fp8, no staging
    using MT = typename std::conditional<KV8, __half, T>::type;   // tensor-core operand type
    constexpr int BS = Tile::BS, NWC = Tile::NWC, SLICE = Tile::SLICE, STAGES = Tile::STAGES;
    constexpr int KT = D / 16;   // k-steps of Q.K^T and d-tiles of P.V
    constexpr int HP = NT * 8;   // padded heads
    constexpr int RS = Tile::RED_STRIDE;
    static_assert(NWC * HP * RS * 4 <= STAGES * 2 * SLICE + Tile::STAGING,
                  "reduction buffer must fit in the ring (and staging)");
    // Pages go to consumer warps round-robin: with STAGES a multiple of NWC a
    // warp only re-waits on stages it consumed itself, so a parity wait can
    // never be satisfied by the previous lap's phase.
    static_assert(STAGES % NWC == 0, "ring depth must be a multiple of the consumer warps");

    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    uint8_t* ring = smem;
    uint8_t* staging = smem + STAGES * 2 * SLICE;   // FP8 only: [NWC][K, V][BS][D] fp16
    constexpr bool QS = Tile::q_shared(NT);
    uint8_t* qtile = staging + Tile::STAGING;       // QS: the CTA's Q fragments, 16 rows of D
    uint64_t* full = reinterpret_cast<uint64_t*>(qtile + Tile::qtile_bytes(NT));
    uint64_t* empty = full + STAGES;
    float* st_m = reinterpret_cast<float*>(empty + STAGES);
    float* st_l = st_m + NWC * HP;
    volatile int* abort_flag = reinterpret_cast<volatile int*>(st_l + NWC * HP);   // set on a wait timeout

    // Lets the combine kernel queued behind this one start its prologue as
    // soon as every CTA of this grid is running (it waits for our results).
    asm volatile("griddepcontrol.launch_dependents;");
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    bool inited = false;   // the ring's barriers have been initialised (uniform)

    // One work item: split s of row tile rt of KV head kvh of sequence b, with
    // P-token partitions (n_known: its clamped context length, or -1 to load
    // it).  Every thread of the CTA runs it.
    auto run_item = [&](const int b, const int kvh, const int rt, const int s, const int P, const int n_known) {
        const QCols qc{b, kvh * p.G, rt * HP, p.R, p.G, p.q_len, p.Hq};
        const int ncols = min(HP, p.R - qc.col0);   // live columns of this CTA

        const int n = n_known >= 0 ? n_known : clampi(p.ctx[b], 0, p.n_cap);
        const int ns_b = (n + P - 1) / P;
        const int t0 = s * P;
        const int t1 = min(t0 + P, n);

        if (t0 >= t1) {
            // Split past the context.  Partials mode writes the (-inf, 0, 0)
            // sentinel; an empty context (n == 0) writes zero output rows.
            if (p.partials_only) {
                for (int i = threadIdx.x; i < ncols * D; i += blockDim.x) {
                    const size_t row = qc.row(i / D) * p.ns_stride + s;
                    p.part_acc[row * D + i % D] = 0.f;
                    if (i % D == 0) {
                        p.part_m[row] = -INFINITY;
                        p.part_l[row] = 0.f;
                    }
                }
            } else if (n == 0 && s == 0) {
                for (int i = threadIdx.x; i < ncols * D; i += blockDim.x)
                    reinterpret_cast<T*>(p.out)[qc.row(i / D) * D + i % D] = from_float<T>(0.f);
            }
            return;
        }

        if (threadIdx.x == 0) {
            for (int i = 0; i < STAGES; ++i) {
                if (inited) {   // a later item of this CTA: every phase of the previous one is complete
                    mbar_inval(&full[i]);
                    mbar_inval(&empty[i]);
                }
                mbar_init(&full[i], 1);
                mbar_init(&empty[i], 1);
            }
            fence_barrier_init();
            *abort_flag = 0;
        }
        __syncthreads();
        inited = true;

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
                    issue_page_loads<LAYOUT, D>(kd, kd + SLICE, &tmk, &tmv, &full[stg], phys * p.Hc + HEADS * kvh,
                                                pol);
                }
                if (STRESS && p.stress_ns) __nanosleep(p.stress_ns);
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
        float scale_log2 = p.scale_log2;
        if constexpr (DIRECT8) {
            const int qe = fp8_q_frags<T, D, NT>(qf, reinterpret_cast<const T*>(p.q), qc, lane);
            scale_log2 *= exp2f((float)qe);
        } else {
            load_q_frags<T, D, NT>(qf, reinterpret_cast<const T*>(p.q), qc, lane);
        }
        if constexpr (KV8 && !DIRECT8 && std::is_same<T, __nv_bfloat16>::value) {
            // bf16 queries meet fp16 keys: convert them, scaled by 2^-e when
            // |q| > 2^15 so that they stay inside the fp16 range (e is the same
            // in every warp: each holds the whole group's Q); 2^e goes into the
            // score scale.
            uint32_t mx = 0;
#pragma unroll
            for (int nt = 0; nt < NT; ++nt)
#pragma unroll
                for (int kk = 0; kk < KT; ++kk)
#pragma unroll
                    for (int j = 0; j < 2; ++j)
                        mx = max(mx, max((qf[nt][kk][j] << 16) & 0x7FFFFFFFu, qf[nt][kk][j] & 0x7FFF0000u));
            mx = __reduce_max_sync(0xffffffffu, mx);
            const int ex = (int)((mx >> 23) & 0xFF) - 127;   // floor(log2 max|q|) for normal values
            const int e = min(max(ex - 14, 0), 120);
            const float down = exp2f((float)-e);
            scale_log2 *= exp2f((float)e);
#pragma unroll
            for (int nt = 0; nt < NT; ++nt)
#pragma unroll
                for (int kk = 0; kk < KT; ++kk)
#pragma unroll
                    for (int j = 0; j < 2; ++j) {
                        const uint32_t w = qf[nt][kk][j];
                        const __half2 h = __floats2half2_rn(__uint_as_float(w << 16) * down,
                                                            __uint_as_float(w & 0xFFFF0000u) * down);
                        qf[nt][kk][j] = *reinterpret_cast<const uint32_t*>(&h);
                    }
        }
        if constexpr (QS) {   // one copy for the CTA; the page steps reload it per k-step
            if (warp == 0) store_q_frags<D>(qtile, qf, lane);
            named_bar_sync(1, NWC * 32);
        }
        const uint32_t qs_a = smem_u32(qtile);
        WarpState<D, NT> ws;
        ws.reset();
        ColTerms<NT> ct;
        if constexpr (HEADS == 2) {   // the pair's columns: Gc query heads of each KV head per query token
#pragma unroll
            for (int j = 0; j < 2; ++j) ct.second[0][j] = (qc.col0 + 2 * (lane & 3) + j) % p.G >= p.Gc;
        }
        if constexpr (GEN) {
#pragma unroll
            for (int nt = 0; nt < NT; ++nt)
#pragma unroll
                for (int j = 0; j < 2; ++j) {
                    const int c = nt * 8 + 2 * (lane & 3) + j;
                    const bool live = qc.live(c);
                    const int gc = qc.col0 + c;
                    ct.shift[nt][j] = live ? p.q_len - 1 - gc / p.G : 0;
                    ct.slope[nt][j] =
                        (live && p.alibi) ? __ldg(p.alibi + qc.h0 + gc % p.G) * 1.4426950408889634f : 0.f;
                }
        }

        const int last_pg = (n - 1) / BS;
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
            const int valid = (pg0 + i == last_pg) ? n - last_pg * BS : BS;
            ct.pos0 = (pg0 + i) * BS - (n - 1);
            if constexpr (DIRECT8) {
                page_step_fp8<D, NT, GEN, QS, HEADS>(ks, ks + SLICE, valid, scale_log2, qf, ws, lane, ct, qs_a);
                __syncwarp();
                if (lane == 0) mbar_arrive(&empty[stg]);
            } else if constexpr (KV8) {
                // expand into this warp's fp16 slices; the ring stage is free again at once
                uint8_t* sk = staging + warp * 2 * (BS * D * 2);
                expand_fp8_slice<D>(ks, sk, lane);
                expand_fp8_slice<D>(ks + SLICE, sk + BS * D * 2, lane);
                __syncwarp();
                if (lane == 0) mbar_arrive(&empty[stg]);
                page_step<MT, kLayoutNHD, D, NT, GEN>(sk, sk + BS * D * 2, valid, scale_log2, qf, ws, lane, ct);
                __syncwarp();
            } else {
                page_step<T, LAYOUT, D, NT, GEN, QS>(ks, ks + SLICE, valid, scale_log2, qf, ws, lane, ct, qs_a);
                __syncwarp();
                if (lane == 0) mbar_arrive(&empty[stg]);
            }
            if (STRESS && p.stress_consumer_ns) __nanosleep(p.stress_consumer_ns);
        }
        if (!ok && lane == 0 && p.err) atomicOr(p.err, kErrTimeout);

        // ------------------------------------------------- merge the warps' states
        ws.finish_l();
        if (lane < 4) {
#pragma unroll
            for (int nt = 0; nt < NT; ++nt)
#pragma unroll
                for (int j = 0; j < 2; ++j) {
                    st_m[warp * HP + nt * 8 + 2 * lane + j] = ws.m[nt][j];
                    st_l[warp * HP + nt * 8 + 2 * lane + j] = ws.l[nt][j];
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
                if (M == -INFINITY) M = 0.f;   // a column that saw no visible token: every f is 0
                const float f = ex2(ws.m[nt][j] - M);   // 0 for a warp that saw no page
                if constexpr (DIRECT8) {   // mma rows g, g+8 of d-tile dt hold d = 16dt + 2g, 16dt + 2g + 1
                    float* row = red + (warp * HP + h) * RS + 2 * (lane >> 2);
#pragma unroll
                    for (int dt = 0; dt < KT; ++dt) {
                        row[dt * 16] = ws.acc[dt][nt][j] * f;
                        row[dt * 16 + 1] = ws.acc[dt][nt][j + 2] * f;
                    }
                } else {
                    float* row = red + (warp * HP + h) * RS + (lane >> 2);
#pragma unroll
                    for (int dt = 0; dt < KT; ++dt) {
                        row[dt * 16] = ws.acc[dt][nt][j] * f;
                        row[dt * 16 + 8] = ws.acc[dt][nt][j + 2] * f;
                    }
                }
            }
        named_bar_sync(1, NWC * 32);

        const bool direct = !p.partials_only && ns_b == 1;
        for (int idx = threadIdx.x; idx < ncols * (D / 4); idx += NWC * 32) {
            const int h = idx / (D / 4);
            const int d = (idx % (D / 4)) * 4;
            float M = -INFINITY;
#pragma unroll
            for (int w = 0; w < NWC; ++w) M = fmaxf(M, st_m[w * HP + h]);
            const float Mref = M == -INFINITY ? 0.f : M;   // no visible token: L = 0, sum = 0
            float L = 0.f;
            float4 sum = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
            for (int w = 0; w < NWC; ++w) {
                L += st_l[w * HP + h] * ex2(st_m[w * HP + h] - Mref);
                const float4 v = *reinterpret_cast<const float4*>(red + (w * HP + h) * RS + d);
                sum.x += v.x;
                sum.y += v.y;
                sum.z += v.z;
                sum.w += v.w;
            }
            sum.x *= p.v_scale;
            sum.y *= p.v_scale;
            sum.z *= p.v_scale;
            sum.w *= p.v_scale;
            const size_t bh = qc.row(h);
            if (direct) {
                const float inv = L > 0.f ? 1.f / L : 0.f;   // an empty causal window gives a zero row
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
    };   // run_item

    if constexpr (SCHED == kSchedGrid) {   // grid order: this CTA's one item
        int item = blockIdx.x;
        const int s = item % p.NS;
        item /= p.NS;
        int rt = 0;
        if (p.RT > 1) {   // several row tiles (keeps the division off the one-tile critical path)
            rt = item % p.RT;
            item /= p.RT;
        }
        run_item(item / p.Hkv, item % p.Hkv, rt, s, p.P, -1);
        return;
    }
    const int HR = p.Hkv * p.RT;
    if constexpr (SCHED == kSchedReuse) {
        // The plan an earlier call of the same problem and context lengths
        // left in the workspace: the partition and split count from the
        // header, and item k's sequence, split and context from entry k / HR
        // of the table (a split's HR items are consecutive).  The first entry
        // is requested before the header arrives.  Every value is checked
        // before use -- P a positive multiple of the page, as every plan's;
        // an entry's sequence, split and context inside the bounds, its first
        // key below its context, and (s + 1) P + n within int, so that no
        // key or page index of run_item overflows -- so a workspace without
        // this problem's plan costs wrong rows and error bit 1, never an
        // access outside the arguments.
        const int tab_len = p.B * p.rule.NS_cap;
        const int hsh = log2_if_pow2(HR);
        const int g0 = hsh >= 0 ? (int)(blockIdx.x >> hsh) : (int)blockIdx.x / HR;
        int4 e = g0 < tab_len ? __ldg(p.plan_tab + g0) : make_int4(-1, 0, 0, 0);
        const int P = p.plan_hdr[0], G = p.plan_hdr[2];
        if (P < kPageTokens || (P & (kPageTokens - 1)) != 0 || G < p.B || G > tab_len) {
            if (blockIdx.x == 0 && threadIdx.x == 0 && p.err) atomicOr(p.err, kErrStalePlan);
            return;
        }
        // Items: G * HR <= B * NS_cap * HR < 2^31 (the host bounds the plan's
        // items), so k + gridDim.x stays below 2^32.
        const unsigned total = (unsigned)G * (unsigned)HR;
        if (threadIdx.x == 0) *abort_flag = 0;
        for (unsigned k = blockIdx.x; k < total; k += gridDim.x) {
            const int g = (int)(hsh >= 0 ? k >> hsh : k / (unsigned)HR);   // < G <= tab_len
            if (k != blockIdx.x) e = __ldg(p.plan_tab + g);
            const int b = e.x, sp = e.y, n = e.z;
            if (b < 0 || b >= p.B || sp < 0 || sp >= p.rule.NS_cap || n < 0 || n > p.n_cap ||
                (long long)sp * P >= (long long)max(n, 1) || (long long)(sp + 1) * P + n > INT_MAX) {
                if (threadIdx.x == 0 && p.err) atomicOr(p.err, kErrStalePlan);
                continue;   // uniform in the CTA: every thread read the same entry
            }
            const int kr = (int)k - g * HR;
            run_item(b, p.RT == 1 ? kr : kr / p.RT, p.RT == 1 ? 0 : kr % p.RT, sp, P, n);
            if (k + gridDim.x >= total) return;   // no further item: free the SM's slot at once
            fence_proxy_async_smem();
            __syncthreads();
            if (*abort_flag) break;
        }
        return;
    } else {
        // Device plan (device_plan.cuh): every warp plans from the context lengths
        // and finds this CTA's items one by one (the same in each warp, so no
        // broadcast and no barrier precede the first item); CTA 0 publishes the
        // partition for the combine kernel, and the first item of each split
        // records the split in the table for the calls that reuse the plan.
        PlanCursor cur{0, 0};
        int P = 0, b = 0, j = 0, n = 0;
        bool found = false, only = false;
        {
            PlanRegs pr;
            int mx = 0;
            long long sum = 0, total = -1;
            warp_context_stats(p.ctx, p.B, p.n_cap, p.rule.sum32 != 0, lane, pr, &mx, &sum);
            P = device_plan_partition_rule(p.rule, mx, sum);
            if (blockIdx.x == 0 && threadIdx.x == 0) {
                p.plan_hdr[0] = P;
                p.plan_hdr[1] = mx > 0 ? (mx - 1) / P + 1 : 1;
            }
            const PlanDiv dv(P, HR);
            found = warp_plan_first_item(pr, p.B, dv, blockIdx.x, cur, lane, &b, &j, &n, &total);
            if (!found) found = warp_plan_item(p.ctx, p.B, p.n_cap, dv, blockIdx.x, cur, lane, &b, &j, &n);
            only = total >= 0 && (long long)blockIdx.x + gridDim.x >= total;   // no second item
        }
        const PlanDiv dv(P, HR);
        // Read after each item's closing barrier; an empty item does not set it.
        if (threadIdx.x == 0) *abort_flag = 0;
        for (long long k = blockIdx.x;; k += gridDim.x) {
            if (k != blockIdx.x) found = warp_plan_item(p.ctx, p.B, p.n_cap, dv, k, cur, lane, &b, &j, &n);
            if (!found) break;
            const int s = dv.split_of(j);   // item j of a sequence: split s, then (grid KV head, row tile) kr
            const int kr = j - s * HR;
            if (kr == 0 && threadIdx.x == 0) {   // split k / HR of the plan (< B * NS_cap: P bounds the splits)
                const int g = dv.split_of((int)k);
                p.plan_tab[g] = make_int4(b, s, n, 0);
                if (b == p.B - 1 && (long long)(s + 1) * P >= n) p.plan_hdr[2] = g + 1;   // the last split
            }
            run_item(b, p.RT == 1 ? kr : kr / p.RT, p.RT == 1 ? 0 : kr % p.RT, s, P, n);
            if (only) return;           // leave at once, freeing the SM's slot for the next CTA
            fence_proxy_async_smem();   // this item's generic writes to the ring before the next item's copies
            __syncthreads();            // every role is done with the ring, the barriers and the Q tile
            if (*abort_flag) break;     // a wait timed out (already reported): take no further item
        }
    }
}

template <typename T, int LAYOUT, int D, int NT, bool GEN, int SCHED, bool STRESS>
__global__ void __launch_bounds__((DecodeTile<D, LAYOUT>::NWC + 1) * 32)
    decode_phase1_kernel(const DecodeParams p, const __grid_constant__ CUtensorMap tmk,
                         const __grid_constant__ CUtensorMap tmv) {
    decode_phase1_body<T, LAYOUT, D, NT, GEN, SCHED, STRESS>(p, tmk, tmv);
}

// The same for the shared-Q tiles, compiled for four CTAs per SM.
template <typename T, int LAYOUT, int D, int NT, bool GEN, int SCHED, bool STRESS>
__global__ void __launch_bounds__((DecodeTile<D, LAYOUT>::NWC + 1) * 32, DecodeTile<D, LAYOUT>::QS_MIN_BLOCKS)
    decode_phase1_kernel_qs(const DecodeParams p, const __grid_constant__ CUtensorMap tmk,
                            const __grid_constant__ CUtensorMap tmv) {
    decode_phase1_body<T, LAYOUT, D, NT, GEN, SCHED, STRESS>(p, tmk, tmv);
}

// Host-side launcher for one instantiation (one-token without bias, general,
// or general over the device plan's items; STRESS: with the race-testing pauses).
template <typename T, int LAYOUT, int D, int NT, bool GEN, int SCHED, bool STRESS>
cudaError_t launch_decode_phase1_variant(const DecodeParams& p, long long grid, const CUtensorMap& tmk,
                                         const CUtensorMap& tmv, cudaStream_t stream) {
    using Tile = DecodeTile<D, LAYOUT>;
    auto kern = [] {   // only the entry this instantiation uses is compiled
        if constexpr (Tile::q_shared(NT))
            return decode_phase1_kernel_qs<T, LAYOUT, D, NT, GEN, SCHED, STRESS>;
        else
            return decode_phase1_kernel<T, LAYOUT, D, NT, GEN, SCHED, STRESS>;
    }();
    const int smem = Tile::smem_bytes(NT);
    static std::atomic<bool> attr_set[kMaxDevices];
    static std::mutex attr_mu;
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    e = once_per_device(attr_set, attr_mu, dev, [&] {
        return cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
    });
    if (e != cudaSuccess) return e;
    kern<<<(unsigned)grid, (Tile::NWC + 1) * 32, smem, stream>>>(p, tmk, tmv);
    return cudaGetLastError();
}

template <typename T, int LAYOUT, int D, int NT, bool STRESS>
cudaError_t launch_decode_phase1_kind(const DecodeParams& p, long long grid, const CUtensorMap& tmk,
                                      const CUtensorMap& tmv, cudaStream_t stream) {
    // A reused plan under the race-testing pauses is planned again: the same
    // items, and no third stress instantiation.
    if (p.plan_hdr && p.plan_ready && !STRESS)
        return launch_decode_phase1_variant<T, LAYOUT, D, NT, true, kSchedReuse, STRESS>(p, grid, tmk, tmv, stream);
    if (p.plan_hdr)
        return launch_decode_phase1_variant<T, LAYOUT, D, NT, true, kSchedPlan, STRESS>(p, grid, tmk, tmv, stream);
    if (p.alibi || p.q_len > 1)
        return launch_decode_phase1_variant<T, LAYOUT, D, NT, true, kSchedGrid, STRESS>(p, grid, tmk, tmv, stream);
    return launch_decode_phase1_variant<T, LAYOUT, D, NT, false, kSchedGrid, STRESS>(p, grid, tmk, tmv, stream);
}

template <typename T, int LAYOUT, int D, int NT>
cudaError_t launch_decode_phase1(const DecodeParams& p, long long grid, const CUtensorMap& tmk,
                                 const CUtensorMap& tmv, cudaStream_t stream) {
    if (p.stress_ns || p.stress_consumer_ns)
        return launch_decode_phase1_kind<T, LAYOUT, D, NT, true>(p, grid, tmk, tmv, stream);
    return launch_decode_phase1_kind<T, LAYOUT, D, NT, false>(p, grid, tmk, tmv, stream);
}

// Head pairs (kLayoutNHD8x2, D = 128, one column tile); under the device plan
// the device plan lists the items per KV-head pair.
template <typename T>
cudaError_t launch_decode_phase1_pairs(const DecodeParams& p, long long grid, const CUtensorMap& tmk,
                                       const CUtensorMap& tmv, cudaStream_t stream) {
    return launch_decode_phase1<T, kLayoutNHD8x2, 128, 1>(p, grid, tmk, tmv, stream);
}

}  // namespace pkv
