// decode_common.cuh -- the per-page arithmetic of paged GQA decode phase 1
// (decode.cuh): query-column maps, the page steps for 16-bit and FP8 pages,
// and the TMA page loads.
//
// One consumer warp handles one 16-token page of one KV head for all the
// query rows of its CTA (heads of the group x query tokens, padded to NT tiles
// of 8):
//   S^T[t][h] = K[t][:] . Q[h][:]           mma.sync m16n8k16, tokens = M, query rows = N
//   m' = max(m, max_t S), alpha = 2^(m - m'), P = 2^(S - m'), l' = alpha l + sum_t P
//   O^T[d][h] = alpha O^T[d][h] + V^T[d][t] P^T[t][h]   (P^T via movmatrix)
// ("paged_attention_v2_triton.py", _partition_attn_kernel docstring steps 1-4;
// flash-decode post, _flash_decode_partial_kernel loop body.)  Scores are in
// log2 units: scale_log2 = scale * log2(e).
#pragma once

#include <type_traits>

#include "ptx.cuh"

namespace pkv {

// kLayoutNHD8: the NHD layout with FP8 E4M3 elements (K = k_scale * fp8,
// V = v_scale * fp8), fp16 tensor-core arithmetic: at D = 64 its pages are
// expanded to fp16 in shared memory and take the kLayoutNHD path; at D >= 128
// they go from the ring straight into mma fragments (page_step_fp8).
// kLayoutNHD8x2: the same cache with one CTA per pair of adjacent KV heads
// (D = 128, at most 4 query rows per KV head, so that both heads' rows fill
// one 8-column tile): the two heads' slices of a page are contiguous in the
// NHD layout, so one ring stage takes both with one 4 KB box for K and one for
// V instead of two 2 KB stages.
enum { kLayoutNHD = 0, kLayoutVLLM = 1, kLayoutNHD8 = 2, kLayoutNHD8x2 = 3 };
constexpr int kPageTokens = 16;

__device__ __forceinline__ int clampi(int v, int lo, int hi) { return v < lo ? lo : (v > hi ? hi : v); }

// Partition of a device plan read back from a workspace header, kept a page
// multiple in [one page, 2^30]: a valid plan is unchanged (its partition is a
// page multiple of at least four pages), and a header another problem left
// behind cannot make a split count or a token index overflow.
__device__ __forceinline__ int device_plan_partition(int P) {
    return clampi(P, kPageTokens, 1 << 30) / kPageTokens * kPageTokens;
}

// Byte offset of 16-byte chunk c (c < D/8) of token row t in an NHD slice
// written by 64-element TMA boxes with 128-byte swizzle.
template <int BS>
__device__ __forceinline__ uint32_t nhd_off(int t, int c) {
    return (uint32_t)((c >> 3) * (BS * 128) + t * 128 + (((c & 7) ^ (t & 7)) << 4));
}

// The query columns of one CTA (the mma N dimension).  A (sequence b, KV
// head) pair has R = G * q_len query rows: query token i (0 <= i < q_len) of
// every head of the group.  Column c of the CTA is row gc = col0 + c, i.e.
// token i = gc / G of head h0 + gc % G; columns at or past R are padding (zero
// queries, never written).  row() is the row index of q, out and the partials,
// all [B][q_len][Hq][...].
struct QCols {
    int b, h0, col0, R, G, q_len, Hq;
    __device__ __forceinline__ bool live(int c) const { return col0 + c < R; }
    __device__ __forceinline__ int token(int c) const { return (col0 + c) / G; }
    __device__ __forceinline__ size_t row(int c) const {
        const int gc = col0 + c;
        if (q_len == 1) return (size_t)b * Hq + h0 + gc;   // no division on the one-token path
        return ((size_t)b * q_len + gc / G) * Hq + h0 + gc % G;
    }
};

// Q^T fragments (mma B operand) of columns [nt*8, nt*8+8); padding columns are zero.
template <typename T, int D, int NT>
__device__ __forceinline__ void load_q_frags(uint32_t (&qf)[NT][D / 16][2], const T* q, const QCols& qc, int lane) {
#pragma unroll
    for (int nt = 0; nt < NT; ++nt) {
        const int c = nt * 8 + (lane >> 2);
        const bool live = qc.live(c);
        const T* qb = q + (live ? qc.row(c) : 0) * D;
#pragma unroll
        for (int kk = 0; kk < D / 16; ++kk) {
            if (live) {
                const uint32_t* qr = reinterpret_cast<const uint32_t*>(qb + kk * 16 + 2 * (lane & 3));
                qf[nt][kk][0] = qr[0];
                qf[nt][kk][1] = qr[4];
            } else {
                qf[nt][kk][0] = 0u;
                qf[nt][kk][1] = 0u;
            }
        }
    }
}

template <int D, int NT>
struct WarpState {
    float acc[D / 16][NT][4];   // O^T fragments: (d = dt*16 + lane/4 (+8), h = nt*8 + 2*(lane&3) + j)
    float m[NT][2];             // running max per head column (log2 units), uniform across lane/4
    float l[NT][2];             // running sum, per lane (reduced across lane/4 at the end)

    __device__ __forceinline__ void reset() {
#pragma unroll
        for (int dt = 0; dt < D / 16; ++dt)
#pragma unroll
            for (int nt = 0; nt < NT; ++nt)
#pragma unroll
                for (int e = 0; e < 4; ++e) acc[dt][nt][e] = 0.f;
#pragma unroll
        for (int nt = 0; nt < NT; ++nt) {
            m[nt][0] = m[nt][1] = -INFINITY;
            l[nt][0] = l[nt][1] = 0.f;
        }
    }

    // Completes l: sums the per-lane partial sums over the 8 token rows.
    __device__ __forceinline__ void finish_l() {
#pragma unroll
        for (int nt = 0; nt < NT; ++nt)
#pragma unroll
            for (int j = 0; j < 2; ++j) {
                float v = l[nt][j];
                v += __shfl_xor_sync(0xffffffffu, v, 4);
                v += __shfl_xor_sync(0xffffffffu, v, 8);
                v += __shfl_xor_sync(0xffffffffu, v, 16);
                l[nt][j] = v;
            }
    }
};

// Per-column terms of the general kernel (GEN), for the lane's accumulator
// columns nt*8 + 2*(lane&3) + j:
//   shift: q_len - 1 - i for query token i, which sits at pos_i = n - 1 - shift
//          (bottom-right rule); page token t is at t_abs = page start + t, and
//          rel = t_abs - pos_i = pos0 + t + shift with pos0 the page's first
//          position minus (n - 1).  The key is visible iff rel <= 0;
//   slope: its head's ALiBi slope in log2 units (0 without ALiBi): bias slope * rel.
// second (kLayoutNHD8x2, any kernel): the column's query head belongs to the
// second KV head of the CTA's pair.
template <int NT>
struct ColTerms {
    float slope[NT][2];
    int shift[NT][2];
    int pos0;
    bool second[NT][2];
};

// Folds one page (K slice ks, V slice vs in shared memory) into the warp's
// state; `valid` = tokens of the page inside the context (1..16).  Tokens past
// it are masked by select, and their V rows are zeroed first, so whatever the
// unread slots hold (NaN included) cannot reach the result.  With GEN, tokens
// past a column's causal window are masked by select as well (their V rows lie
// inside the context, so P = 0 multiplies finite cache values), and a column
// that has seen no visible token keeps m = -inf with alpha = P = 0.
// Q^T fragments of k-step kk for both column tiles (NT = 2) from the CTA's
// shared copy (qs_a: its shared address; rows of D 16-bit values, 16-byte
// chunks XOR-swizzled by row & 7, holding each lane's fragments as stored by
// store_q_frags).
template <int D>
__device__ __forceinline__ void load_q_smem(uint32_t qs_a, int kk, int lane, uint32_t (&b)[4]) {
    const int mi = lane >> 3, r8 = lane & 7;
    const int row = ((mi >> 1) << 3) + r8;
    ldsm_x4(qs_a + (uint32_t)(row * D * 2 + (((2 * kk + (mi & 1)) ^ r8) << 4)), b);
}
template <int D>
__device__ __forceinline__ void store_q_frags(uint8_t* qs, const uint32_t (&qf)[2][D / 16][2], int lane) {
#pragma unroll
    for (int nt = 0; nt < 2; ++nt) {
        const int row = nt * 8 + (lane >> 2);
#pragma unroll
        for (int kk = 0; kk < D / 16; ++kk)
#pragma unroll
            for (int j = 0; j < 2; ++j)
                *reinterpret_cast<uint32_t*>(qs + row * D * 2 + (((2 * kk + j) ^ (row & 7)) << 4) + 4 * (lane & 3)) =
                    qf[nt][kk][j];
    }
}

template <typename T, int LAYOUT, int D, int NT, bool GEN, bool QS = false>
__device__ __forceinline__ void page_step(uint8_t* ks, uint8_t* vs, int valid, float scale_log2,
                                          const uint32_t (&qf)[NT][D / 16][2], WarpState<D, NT>& st, int lane,
                                          const ColTerms<NT>& ct, uint32_t qs_a = 0) {
    constexpr int BS = kPageTokens, KT = D / 16;
    const int mi = lane >> 3, r8 = lane & 7;   // ldmatrix: matrix index and row within it
    const uint32_t ks_a = smem_u32(ks), vs_a = smem_u32(vs);

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
        if constexpr (QS) {
            static_assert(NT == 2, "the shared Q copy holds two column tiles");
            uint32_t b[4];
            load_q_smem<D>(qs_a, kk, lane, b);
            Mma<T>::run(sc[0], a, b[0], b[1]);
            Mma<T>::run(sc[1], a, b[2], b[3]);
        } else {
#pragma unroll
            for (int nt = 0; nt < NT; ++nt) Mma<T>::run(sc[nt], a, qf[nt][kk][0], qf[nt][kk][1]);
        }
    }

    // scale to log2 units, mask, online-softmax update
    const int tr = lane >> 2;
#pragma unroll
    for (int nt = 0; nt < NT; ++nt) {
#pragma unroll
        for (int e = 0; e < 4; ++e) {
            const int t = tr + ((e >> 1) << 3);
            float v = sc[nt][e] * scale_log2;
            if constexpr (GEN) {
                const int rel = ct.pos0 + t + ct.shift[nt][e & 1];   // key position - query position
                v = fmaf(ct.slope[nt][e & 1], (float)rel, v);
                sc[nt][e] = rel <= 0 ? v : -INFINITY;   // also masks every token past the context
            } else {
                sc[nt][e] = t < valid ? v : -INFINITY;
            }
        }
#pragma unroll
        for (int j = 0; j < 2; ++j) {
            float mx = fmaxf(sc[nt][j], sc[nt][j + 2]);
            mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 4));
            mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 8));
            mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 16));
            const float mnew = fmaxf(st.m[nt][j], mx);
            const float mref = (GEN && mnew == -INFINITY) ? 0.f : mnew;   // nothing visible yet
            const float alpha = ex2(st.m[nt][j] - mref);
            st.m[nt][j] = mnew;
            sc[nt][j] = ex2(sc[nt][j] - mref);
            sc[nt][j + 2] = ex2(sc[nt][j + 2] - mref);
            st.l[nt][j] = st.l[nt][j] * alpha + (sc[nt][j] + sc[nt][j + 2]);
#pragma unroll
            for (int dt = 0; dt < KT; ++dt) {
                st.acc[dt][nt][j] *= alpha;
                st.acc[dt][nt][j + 2] *= alpha;
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

    // Zero the V rows past the context so that P = 0 times whatever they hold stays 0.
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
        for (int nt = 0; nt < NT; ++nt) Mma<T>::run(st.acc[dt][nt], a, pb[nt][0], pb[nt][1]);
    }
}

// Two FP8 E4M3 values (low byte first) to two fp16 values, exactly (every
// E4M3 value is an fp16 value).
__device__ __forceinline__ uint32_t e4m3x2_to_f16x2(uint16_t v) {
    uint32_t r;
    asm("cvt.rn.f16x2.e4m3x2 %0, %1;" : "=r"(r) : "h"(v));
    return r;
}

// Expands one FP8 page slice ([BS][D] bytes, row-major, as TMA copied it)
// into the fp16 NHD slice layout page_step reads (nhd_off: 64-element blocks,
// 128-byte swizzle).  One warp; each lane converts 8 bytes at a time.
template <int D>
__device__ __forceinline__ void expand_fp8_slice(const uint8_t* src, uint8_t* dst, int lane) {
    constexpr int BS = kPageTokens, CH = D / 8;   // 16-byte fp16 chunks per row
#pragma unroll
    for (int idx = lane; idx < BS * CH; idx += 32) {
        const int t = idx / CH, c = idx % CH;
        const uint2 w = *reinterpret_cast<const uint2*>(src + t * D + c * 8);
        uint4 o;
        o.x = e4m3x2_to_f16x2((uint16_t)(w.x & 0xFFFFu));
        o.y = e4m3x2_to_f16x2((uint16_t)(w.x >> 16));
        o.z = e4m3x2_to_f16x2((uint16_t)(w.y & 0xFFFFu));
        o.w = e4m3x2_to_f16x2((uint16_t)(w.y >> 16));
        *reinterpret_cast<uint4*>(dst + nhd_off<BS>(t, c)) = o;
    }
}

// ---- FP8 pages straight into fp16 mma fragments (D >= 128) ------------------
//
// The slices arrive as 128-byte-wide TMA boxes with 128-byte swizzle: token row
// t of 128-column block j, 16-byte chunk c (16 elements) at
// j*BS*128 + t*128 + ((c ^ (t & 7)) << 4).  An ldmatrix.x4 (b16 view) of
// chunks (c, c+1), rows 0-7 and 8-15 gives lane (g = lane/4, q = lane%4) the
// bytes 4q..4q+3 of its row in each chunk.
//
// S^T = K.Q^T: the four bytes of one chunk feed one m16n8k16 with the
// k-index permuted -- mma k = 2q+j <-> d = 16c+4q+j and k = 2q+8+j <->
// d = 16c+4q+2+j -- so the Q (B) fragments are loaded with the same
// permutation (fp8_q_frags) and the dot products are unchanged.
// O^T += V^T.P^T: ldmatrix.x4.trans gives lane (g, q) the bytes
// V[2q][2g], V[2q][2g+1], V[2q+1][2g], V[2q+1][2g+1] of a chunk; one byte
// permute splits them into rows d = 2g and 2g+1 for tokens (2q, 2q+1), i.e.
// mma rows g and g+8 hold d = 16c+2g and 16c+2g+1: the output rows are
// permuted, and the merge writes them back in order.

__device__ __forceinline__ uint32_t fp8_off(int t, int c) {   // chunk c (16 B) of row t
    return (uint32_t)((c >> 3) * (kPageTokens * 128) + t * 128 + (((c & 7) ^ (t & 7)) << 4));
}

// Q fragments in the permuted k order above: qf[nt][kk][0] = (q[16kk+4q], q[16kk+4q+1]),
// qf[nt][kk][1] = (q[16kk+4q+2], q[16kk+4q+3]) of column nt*8 + g, as fp16 pairs.
// bf16 queries are scaled by 2^-e (returned) when |q| > 2^15 to fit fp16; e is
// a warp-wide maximum, the same in every warp of the CTA.
template <typename T, int D, int NT>
__device__ __forceinline__ int fp8_q_frags(uint32_t (&qf)[NT][D / 16][2], const T* qv, const QCols& qc, int lane) {
    const int g = lane >> 2, q = lane & 3;
    uint2 raw[NT][D / 16];
#pragma unroll
    for (int nt = 0; nt < NT; ++nt) {
        const int c = nt * 8 + g;
        const bool live = qc.live(c);
        const T* qb = qv + (live ? qc.row(c) : 0) * D;
#pragma unroll
        for (int kk = 0; kk < D / 16; ++kk)
            raw[nt][kk] = live ? *reinterpret_cast<const uint2*>(qb + kk * 16 + 4 * q) : make_uint2(0u, 0u);
    }
    if constexpr (std::is_same<T, __half>::value) {
#pragma unroll
        for (int nt = 0; nt < NT; ++nt)
#pragma unroll
            for (int kk = 0; kk < D / 16; ++kk) {
                qf[nt][kk][0] = raw[nt][kk].x;
                qf[nt][kk][1] = raw[nt][kk].y;
            }
        return 0;
    } else {
        uint32_t mx = 0;
#pragma unroll
        for (int nt = 0; nt < NT; ++nt)
#pragma unroll
            for (int kk = 0; kk < D / 16; ++kk) {
                const uint32_t w0 = raw[nt][kk].x, w1 = raw[nt][kk].y;
                mx = max(mx, max((w0 << 16) & 0x7FFFFFFFu, w0 & 0x7FFF0000u));
                mx = max(mx, max((w1 << 16) & 0x7FFFFFFFu, w1 & 0x7FFF0000u));
            }
        mx = __reduce_max_sync(0xffffffffu, mx);
        const int e = min(max((int)((mx >> 23) & 0xFF) - 127 - 14, 0), 120);
        const float down = exp2f((float)-e);
        auto cv = [&](uint32_t w) {
            const __half2 h = __floats2half2_rn(__uint_as_float(w << 16) * down, __uint_as_float(w & 0xFFFF0000u) * down);
            return *reinterpret_cast<const uint32_t*>(&h);
        };
#pragma unroll
        for (int nt = 0; nt < NT; ++nt)
#pragma unroll
            for (int kk = 0; kk < D / 16; ++kk) {
                qf[nt][kk][0] = cv(raw[nt][kk].x);
                qf[nt][kk][1] = cv(raw[nt][kk].y);
            }
        return e;
    }
}

// A-operand fragment of one 16-byte FP8 chunk pair of a K slice (ldmatrix
// registers rr[0..1]: tokens t and t + 8), as fp16 pairs.
__device__ __forceinline__ void fp8_k_frag(const uint32_t* rr, uint32_t (&a)[4]) {
    a[0] = e4m3x2_to_f16x2((uint16_t)(rr[0] & 0xFFFFu));
    a[1] = e4m3x2_to_f16x2((uint16_t)(rr[1] & 0xFFFFu));
    a[2] = e4m3x2_to_f16x2((uint16_t)(rr[0] >> 16));
    a[3] = e4m3x2_to_f16x2((uint16_t)(rr[1] >> 16));
}
// The same for a transposed V chunk pair (k = token order restored by a byte permute).
__device__ __forceinline__ void fp8_v_frag(const uint32_t* rr, uint32_t (&a)[4]) {
    const uint32_t lo = __byte_perm(rr[0], 0u, 0x3120), hi = __byte_perm(rr[1], 0u, 0x3120);
    a[0] = e4m3x2_to_f16x2((uint16_t)(lo & 0xFFFFu));
    a[1] = e4m3x2_to_f16x2((uint16_t)(lo >> 16));
    a[2] = e4m3x2_to_f16x2((uint16_t)(hi & 0xFFFFu));
    a[3] = e4m3x2_to_f16x2((uint16_t)(hi >> 16));
}

// One FP8 page (swizzled K and V slices in the ring) into the warp's state, as
// page_step; fp16 tensor-core arithmetic.  V rows past `valid` are zeroed in
// the ring stage first (the caller fences before the stage is refilled).
// HEADS = 2 (kLayoutNHD8x2): ks and vs hold two KV heads' slices, BS * D bytes
// apart, and the column tile holds both heads' query rows (ct.second marks the
// second head's).  Each column takes its scores from its own head's keys, and
// P goes into each head's P.V product with the other head's columns zeroed,
// so a column sees exactly the arithmetic of the one-head kernel.
template <int D, int NT, bool GEN, bool QS = false, int HEADS = 1>
__device__ __forceinline__ void page_step_fp8(uint8_t* ks, uint8_t* vs, int valid, float scale_log2,
                                              const uint32_t (&qf)[NT][D / 16][2], WarpState<D, NT>& st, int lane,
                                              const ColTerms<NT>& ct, uint32_t qs_a = 0) {
    static_assert(HEADS == 1 || (HEADS == 2 && NT == 1 && !QS && D == 128), "head pairs: one column tile, D = 128");
    constexpr int BS = kPageTokens, KT = D / 16, HOFF = BS * D;   // HOFF: bytes between the heads' slices
    const int mi = lane >> 3, r8 = lane & 7;
    const int t_l = r8 + ((mi & 1) << 3), c_l = mi >> 1;   // this lane's ldmatrix row and chunk offset
    const uint32_t ks_a = smem_u32(ks), vs_a = smem_u32(vs);

    float sc[NT][4], sc2[4] = {0.f, 0.f, 0.f, 0.f};   // sc2: the second head's scores
#pragma unroll
    for (int nt = 0; nt < NT; ++nt) sc[nt][0] = sc[nt][1] = sc[nt][2] = sc[nt][3] = 0.f;
#pragma unroll
    for (int c2 = 0; c2 < KT / 2; ++c2) {
        uint32_t r[4], r2[4];
        ldsm_x4(ks_a + fp8_off(t_l, 2 * c2 + c_l), r);
        if constexpr (HEADS == 2) ldsm_x4(ks_a + HOFF + fp8_off(t_l, 2 * c2 + c_l), r2);
#pragma unroll
        for (int h = 0; h < 2; ++h) {   // chunk 2*c2 + h: k-step kk
            uint32_t a[4];
            fp8_k_frag(r + 2 * h, a);
            if constexpr (HEADS == 2) {
                uint32_t a2[4];
                fp8_k_frag(r2 + 2 * h, a2);
                Mma<__half>::run(sc[0], a, qf[0][2 * c2 + h][0], qf[0][2 * c2 + h][1]);
                Mma<__half>::run(sc2, a2, qf[0][2 * c2 + h][0], qf[0][2 * c2 + h][1]);
            } else if constexpr (QS) {
                static_assert(NT == 2, "the shared Q copy holds two column tiles");
                uint32_t b[4];
                load_q_smem<D>(qs_a, 2 * c2 + h, lane, b);
                Mma<__half>::run(sc[0], a, b[0], b[1]);
                Mma<__half>::run(sc[1], a, b[2], b[3]);
            } else {
#pragma unroll
                for (int nt = 0; nt < NT; ++nt)
                    Mma<__half>::run(sc[nt], a, qf[nt][2 * c2 + h][0], qf[nt][2 * c2 + h][1]);
            }
        }
    }
    if constexpr (HEADS == 2) {
#pragma unroll
        for (int e = 0; e < 4; ++e)
            if (ct.second[0][e & 1]) sc[0][e] = sc2[e];
    }

    // scale to log2 units, mask, online-softmax update (as page_step)
    const int tr = lane >> 2;
#pragma unroll
    for (int nt = 0; nt < NT; ++nt) {
#pragma unroll
        for (int e = 0; e < 4; ++e) {
            const int t = tr + ((e >> 1) << 3);
            float v = sc[nt][e] * scale_log2;
            if constexpr (GEN) {
                const int rel = ct.pos0 + t + ct.shift[nt][e & 1];   // key position - query position
                v = fmaf(ct.slope[nt][e & 1], (float)rel, v);
                sc[nt][e] = rel <= 0 ? v : -INFINITY;   // also masks every token past the context
            } else {
                sc[nt][e] = t < valid ? v : -INFINITY;
            }
        }
#pragma unroll
        for (int j = 0; j < 2; ++j) {
            float mx = fmaxf(sc[nt][j], sc[nt][j + 2]);
            mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 4));
            mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 8));
            mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 16));
            const float mnew = fmaxf(st.m[nt][j], mx);
            const float mref = (GEN && mnew == -INFINITY) ? 0.f : mnew;   // nothing visible yet
            const float alpha = ex2(st.m[nt][j] - mref);
            st.m[nt][j] = mnew;
            sc[nt][j] = ex2(sc[nt][j] - mref);
            sc[nt][j + 2] = ex2(sc[nt][j + 2] - mref);
            st.l[nt][j] = st.l[nt][j] * alpha + (sc[nt][j] + sc[nt][j + 2]);
#pragma unroll
            for (int dt = 0; dt < KT; ++dt) {
                st.acc[dt][nt][j] *= alpha;
                st.acc[dt][nt][j + 2] *= alpha;
            }
        }
    }
    uint32_t pb[NT][2], pb2[2];   // pb2: the second head's P (HEADS = 2; then pb holds the first's)
    if constexpr (HEADS == 2) {
        float p1[4], p2[4];
#pragma unroll
        for (int e = 0; e < 4; ++e) {
            p1[e] = ct.second[0][e & 1] ? 0.f : sc[0][e];
            p2[e] = ct.second[0][e & 1] ? sc[0][e] : 0.f;
        }
        pb[0][0] = movmatrix_trans(Mma<__half>::pack(p1[0], p1[1]));
        pb[0][1] = movmatrix_trans(Mma<__half>::pack(p1[2], p1[3]));
        pb2[0] = movmatrix_trans(Mma<__half>::pack(p2[0], p2[1]));
        pb2[1] = movmatrix_trans(Mma<__half>::pack(p2[2], p2[3]));
    } else {
#pragma unroll
        for (int nt = 0; nt < NT; ++nt) {
            pb[nt][0] = movmatrix_trans(Mma<__half>::pack(sc[nt][0], sc[nt][1]));
            pb[nt][1] = movmatrix_trans(Mma<__half>::pack(sc[nt][2], sc[nt][3]));
        }
    }

    if (valid < BS) {   // zero whole V rows past the context (layout-agnostic within a row)
        constexpr int ROWB = 128 / 16;   // 16-byte pieces per 128-byte row
        const int per_head = (BS - valid) * ROWB * (D / 128);
        for (int i = lane; i < HEADS * per_head; i += 32) {
            const int hh = i / per_head, k = i % per_head;
            const int blk = k / ((BS - valid) * ROWB), rem = k % ((BS - valid) * ROWB);
            uint8_t* row = vs + hh * HOFF + blk * (BS * 128) + (valid + rem / ROWB) * 128;
            *reinterpret_cast<uint4*>(row + (rem % ROWB) * 16) = make_uint4(0u, 0u, 0u, 0u);
        }
        fence_proxy_async_smem();
        __syncwarp();
    }

#pragma unroll
    for (int c2 = 0; c2 < KT / 2; ++c2) {
        uint32_t r[4], r2[4];
        ldsm_x4_trans(vs_a + fp8_off(t_l, 2 * c2 + c_l), r);
        if constexpr (HEADS == 2) ldsm_x4_trans(vs_a + HOFF + fp8_off(t_l, 2 * c2 + c_l), r2);
#pragma unroll
        for (int h = 0; h < 2; ++h) {   // chunk 2*c2 + h: output rows dt = 2*c2 + h
            uint32_t a[4];
            fp8_v_frag(r + 2 * h, a);
#pragma unroll
            for (int nt = 0; nt < NT; ++nt) Mma<__half>::run(st.acc[2 * c2 + h][nt], a, pb[nt][0], pb[nt][1]);
            if constexpr (HEADS == 2) {
                uint32_t a2[4];
                fp8_v_frag(r2 + 2 * h, a2);
                Mma<__half>::run(st.acc[2 * c2 + h][0], a2, pb2[0], pb2[1]);
            }
        }
    }
}

// Issues the TMA loads of one page slice pair (K and V of one KV head, or of
// two adjacent ones for kLayoutNHD8x2) into a ring stage, completing on `bar`.
template <int LAYOUT, int D>
__device__ __forceinline__ void issue_page_loads(uint8_t* kd, uint8_t* vd, const CUtensorMap* tmk,
                                                 const CUtensorMap* tmv, uint64_t* bar, int slice, uint64_t pol) {
    constexpr int BS = kPageTokens;
    if (LAYOUT == kLayoutNHD8x2) {   // `slice` is the pair's first: one {128, BS, 2} box each (D = 128)
        mbar_arrive_expect_tx(bar, 4 * BS * D);
        tma_load_3d(kd, tmk, bar, 0, 0, slice, pol);
        tma_load_3d(vd, tmv, bar, 0, 0, slice, pol);
        return;
    }
    if (LAYOUT == kLayoutNHD8) {
        mbar_arrive_expect_tx(bar, 2 * BS * D);
        if (D >= 128) {   // 128-byte-wide swizzled boxes (page_step_fp8)
#pragma unroll
            for (int j = 0; j < D / 128; ++j) {
                tma_load_3d(kd + j * BS * 128, tmk, bar, j * 128, 0, slice, pol);
                tma_load_3d(vd + j * BS * 128, tmv, bar, j * 128, 0, slice, pol);
            }
        } else {          // one unswizzled {D, BS} byte box (expanded by expand_fp8_slice)
            tma_load_3d(kd, tmk, bar, 0, 0, slice, pol);
            tma_load_3d(vd, tmv, bar, 0, 0, slice, pol);
        }
        return;
    }
    mbar_arrive_expect_tx(bar, 2 * BS * D * 2);
    if (LAYOUT == kLayoutNHD) {
#pragma unroll
        for (int j = 0; j < D / 64; ++j) {
            tma_load_3d(kd + j * BS * 128, tmk, bar, j * 64, 0, slice, pol);
            tma_load_3d(vd + j * BS * 128, tmv, bar, j * 64, 0, slice, pol);
        }
    } else {
        tma_load_3d(kd, tmk, bar, 0, 0, slice, pol);
        tma_load_3d(vd, tmv, bar, 0, 0, slice, pol);
    }
}

}  // namespace pkv
