// mla.cu -- MLA paged causal prefill on sm_103a tensor cores (tcgen05 + TMEM),
// one CTA pair (cta_group::2) per tile.
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
// cores, with the 16 heads of 16 query tokens stacked into one 256-row tile
// that shares each gathered key row.
//
// Cluster = a CTA pair = (sequence, 16-token row tile, half of the 512 output
// columns).  CTA r of the pair holds rows 128r .. 128r + 127 (tokens 8r ..
// 8r + 7 of the tile): its Q rows in shared memory (9 chunks of 128 rows x 64
// bf16 = 144 KB, one 2-D TMA box each) and, in its TMEM (512 columns), those
// rows' 256 output columns O and two fp32 S buffers of 128 keys; a block's
// bf16 P is written over its scores (the TMEM A operand of O += P.V), so the
// tensor core computes the next block's scores into the other buffer while
// the softmax warps work.  One thread of CTA 0 issues every MMA for both
// (M = 256): B operands are split between the CTAs, so each SM loads half of
// every key block -- per 128 keys, 9 K sub-chunks of 64 keys x 64 columns
// (its half of the N = 128 keys of S = Q.K^T) and 4 V sub-chunks of 32 keys x
// 128 output columns (its half of the N = 256 columns of O += P.V), 8 KB each,
// two per 16 KB slot of a 5-slot ring, in the 128-byte-swizzled layout of the
// UMMA descriptors.  A one-SM tile would read all of every chunk; the pair
// halves the L2-to-SM bytes per MMA.  O in TMEM (256 of the 512 columns) is
// why the two halves of the output are separate tasks.
//
// S once per tile (replay, when the caller bounds kv_len): only the first
// half's tasks run here; each exports its key blocks' bf16 P (chunk-major,
// 8 keys of all 128 rows per 2 KB, so that the softmax warps' stores are
// coalesced), the factor O was rescaled by before each block, one flag per
// softmax warp (did any row rescale) and the final row sums.
// mla_replay_kernel, the next grid, computes the other half from them with
// the same arithmetic, so S = Q.K^T runs once per tile; without the bound
// each half computes S itself (1.53x the algorithmic tensor work).
//
// Page size 1 makes every key its own page.  Gathering 128-byte row pieces
// per tile (up to ~100 tiles read each key) keeps too few bytes in flight
// per TMA operation, so mla_stage_kernel first copies each referenced row
// (ckv | kpe, 1152 bytes) once into a workspace, sequence by sequence, each
// sequence padded with zero rows to a multiple of 128 rows; the attention
// kernel then loads consecutive staged rows per box.  A box never leaves its
// sequence's staged rows, as the page's kernel never loads a key outside
// [kv_pages_start, kv_pages_end): rows of a box past the tile's keys are the
// sequence's own later keys or zero rows, masked in the softmax, so another
// sequence's cache rows cannot reach this output.
//
// Synchronisation.  Both CTAs' TMA copies of a chunk complete on CTA 0's
// `full` barrier (cta_group::2 loads; CTA 0's producer expects the bytes of
// both), which CTA 0's MMA thread waits on.  Its commits arrive on the
// barriers of both CTAs (multicast): `empty` (a ring slot is free),
// `s_full` (scores of a block in an S buffer), `pv_buf` (O += P.V of a block
// done), `mma_done`.  The softmax warps of both CTAs arrive on CTA 0's
// `p_full` (P written over the scores), one elected lane per warp.
//
// Warps: 0 = producer (one thread issues the Q boxes and the key boxes, the
// latter after the staging grid has completed); 1 = TMEM allocation, then
// CTA 0's MMA issuer; 2..9 = softmax, two warps per TMEM lane quadrant, each
// taking 64 of a block's 128 keys for its 32 rows: online max/sum in log2
// units, lazy O rescaling (only when the running max grows by more than 8,
// i.e. a factor 256), P stored to TMEM as bf16, final O / l and the base-2
// LSE.  Every wait is bounded; both CTAs meet at a cluster barrier before the
// TMEM is freed.
#include <algorithm>

#include "internal.h"
#include "tcgen05.cuh"

namespace pkv {

namespace mla {
constexpr int kHeads = 16, kDc = 512, kDr = 64;
constexpr int kTok = 8;                   // query tokens per CTA
constexpr int kPairTok = 2 * kTok;        // query tokens per CTA pair (row tile)
constexpr int kRows = kTok * kHeads;      // 128 TMEM lanes per CTA
constexpr int kKeys = 128;                // keys per block: N of S over the pair
constexpr int kHalfKeys = kKeys / 2;      // keys of a block each CTA loads for S
constexpr int kQChunk = kRows * 64 * 2;   // 16 KB: 128 rows x 64 bf16
constexpr int kQChunks = 9;               // 8 x ckv + 1 x kpe
constexpr int kSub = 8192;                // K sub-chunk: 64 keys x 64 bf16; V sub-chunk: 32 keys x 128 bf16
constexpr int kSlot = 2 * kSub;           // ring slot: two sub-chunks
constexpr int kKSlots = 5;                // per block: K columns 0-127, ..., 384-511, then kpe 512-575 alone
constexpr int kVSlots = 2;                // per block: keys 0-63, 64-127 of this CTA's 128 output columns
constexpr int kStages = 5;
constexpr int kSoftmaxWarps = 8;          // two per TMEM lane quadrant, each 64 of a block's 128 keys
constexpr int kThreads = 64 + 32 * kSoftmaxWarps;
constexpr int kBars = 2 * kStages + kQChunks + 20;
constexpr int kRedBytes = 2 * kRows * 4;   // row max / row sum exchange: [key half][row]
constexpr int kSmemBytes = 1024 + kQChunks * kQChunk + kStages * kSlot + kRedBytes + kBars * 8 + 32;
static_assert(kSmemBytes <= 232448, "shared memory per CTA");
// TMEM columns: O [0,256), S buffers [256,384) and [384,512); block j's scores go
// to buffer j % 2, and its bf16 P is written over them in place (key half h at
// columns 64h .. 64h + 31 of the buffer, where that half's scores were).
constexpr uint32_t kColS = 256;
constexpr float kLazyRescale = 8.f;       // log2 units
constexpr uint16_t kBothCtas = 3;         // multicast mask of the pair
}  // namespace mla


// Staged rows of sequence b: its kv_len keys rounded up to kMlaSeqAlign rows.
__device__ __forceinline__ int mla_padded_len(const MlaParams& p, int b) {
    const int kv_len = max(0, p.kv_indptr[b + 1] - p.kv_indptr[b]);
    return (kv_len + kMlaSeqAlign - 1) / kMlaSeqAlign * kMlaSeqAlign;
}

// Key blocks (128 keys) that the rows of 16-token tile t of sequence b may
// see: the tile's last token sees prefix + its index + 1 keys (none without a
// pool or staged keys).
__device__ __forceinline__ int mla_tile_blocks(const MlaParams& p, int b, int t) {
    const int q_len = p.qo_indptr[b + 1] - p.qo_indptr[b];
    const int kv_len = p.kv_indptr[b + 1] - p.kv_indptr[b];
    const int i0 = t * mla::kPairTok;
    const int n_keys = (p.num_pages > 0 && p.stage_rows > 0)
                           ? max(0, min(kv_len, kv_len - q_len + i0 + min(mla::kPairTok, q_len - i0)))
                           : 0;
    return (n_keys + mla::kKeys - 1) / mla::kKeys;
}

// Exclusive scan of one int per thread over a 256-thread block; returns the
// thread's prefix and sets *total.  Uses `sbuf` (8 ints).
__device__ __forceinline__ int block_scan_256(int v, int* sbuf, int* total) {
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    int x = v;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const int y = __shfl_up_sync(0xffffffffu, x, o);
        if (lane >= o) x += y;
    }
    if (lane == 31) sbuf[warp] = x;
    __syncthreads();
    int wsum = 0, all = 0;
#pragma unroll
    for (int w = 0; w < 8; ++w) {
        const int t = sbuf[w];
        if (w < warp) wsum += t;
        all += t;
    }
    __syncthreads();
    *total = all;
    return wsum + x - v;
}

// The task list (one block of 256 threads): every (16-token row tile, output
// half) pair of the batch, tiles with the most key blocks first (a counting
// sort on the block count), so that the persistent CTA pairs, which take the
// list in turns, start the longest tiles first.  Also the first row tile and
// the first staged row of every sequence.
constexpr int kTaskBins = 2048;   // block counts at or above kTaskBins - 1 share the last bin
__device__ void mla_build_tasks(const MlaParams& p) {
    __shared__ int bins[kTaskBins];
    __shared__ int sbuf[8];
    const int tid = threadIdx.x;
    // per-sequence first tile and first staged row (scans over the batch, 256 at a time)
    int tile_carry = 0, row_carry = 0;
    for (int base = 0; base < p.batch; base += 256) {
        const int b = base + tid;
        const int nt = b < p.batch ? max(0, (p.qo_indptr[b + 1] - p.qo_indptr[b] + mla::kPairTok - 1) / mla::kPairTok) : 0;
        const int rows = b < p.batch ? mla_padded_len(p, b) : 0;
        int t_total = 0, r_total = 0;
        const int t_ex = block_scan_256(nt, sbuf, &t_total);
        const int r_ex = block_scan_256(rows, sbuf, &r_total);
        if (b < p.batch) {
            p.seq_tile[b] = tile_carry + t_ex;
            p.seq_row[b] = row_carry + r_ex;
        }
        tile_carry += t_total;
        row_carry += r_total;
    }
    const int T = tile_carry;   // row tiles of the batch
    if (tid == 0) p.seq_tile[p.batch] = T;
    for (int i = tid; i < kTaskBins; i += 256) bins[i] = 0;
    __syncthreads();   // seq_tile / seq_row written (global, same block) and bins cleared
    // tile t -> (sequence, tile of the sequence): the last sequence whose first tile is <= t
    auto seq_of = [&](int t) {
        int lo = 0, hi = p.batch - 1;
        while (lo < hi) {
            const int mid = (lo + hi + 1) >> 1;
            if (p.seq_tile[mid] <= t) lo = mid;
            else hi = mid - 1;
        }
        return lo;
    };
    for (int t = tid; t < T; t += 256) {
        const int b = seq_of(t);
        atomicAdd(&bins[min(mla_tile_blocks(p, b, t - p.seq_tile[b]), kTaskBins - 1)], 1);
    }
    __syncthreads();
    // bin starts in decreasing block count: thread tid owns bins kTaskBins - 8 tid - 1 .. - 8
    int own[8], sum = 0;
#pragma unroll
    for (int i = 0; i < 8; ++i) {
        own[i] = bins[kTaskBins - 1 - (8 * tid + i)];
        sum += own[i];
    }
    int total = 0;
    int start = block_scan_256(sum, sbuf, &total);
#pragma unroll
    for (int i = 0; i < 8; ++i) {
        bins[kTaskBins - 1 - (8 * tid + i)] = start;
        start += own[i];
    }
    __syncthreads();
    // bin 0 starts after every tile with keys
    const int keyed = bins[0];
    __syncthreads();   // every thread read bins[0] before the positions are taken
    // Without replay: list position i holds both output halves of its tile,
    // entries 2i and 2i + 1.  With replay: entry i holds the first half of the
    // i-th tile with keys, the second half is entry L + i of the replay list
    // (L = keyed + 2 * tiles without keys); tiles without keys keep both
    // halves, entries keyed + 2 j and + 1.
    const int L = p.replay ? T + (T - keyed) : 0;
    if (tid == 0) {
        p.task_count[1] = p.replay ? keyed : min(2 * keyed, p.max_tasks);
        p.task_count[2] = 0;   // next task with keys to hand out
        p.task_count[3] = 0;   // next replay task to hand out
        p.task_count[4] = p.replay ? max(0, min(keyed, p.max_tasks - L)) : 0;
        p.task_count[5] = L;
    }
    for (int t = tid; t < T; t += 256) {
        const int b = seq_of(t);
        const int tt = t - p.seq_tile[b];
        const int J = mla_tile_blocks(p, b, tt);
        const int pos = atomicAdd(&bins[min(J, kTaskBins - 1)], 1);
        const int4 e = make_int4(b, tt * mla::kPairTok, p.seq_row[b], J);
        const int4 e1 = make_int4(e.x, e.y, e.z, e.w | (1 << 30));
        if (!p.replay) {
            if (2 * pos + 1 < p.max_tasks) {
                p.tasks[2 * pos] = e;
                p.tasks[2 * pos + 1] = e1;
            }
        } else if (J > 0) {   // L + pos < 2 T <= max_tasks
            if (L + pos < p.max_tasks) {
                p.tasks[pos] = e;
                p.tasks[L + pos] = e1;
            }
        } else if (pos + (pos - keyed) + 1 < p.max_tasks) {
            p.tasks[keyed + 2 * (pos - keyed)] = e;
            p.tasks[keyed + 2 * (pos - keyed) + 1] = e1;
        }
    }
    if (tid == 0) p.task_count[0] = min(p.replay ? L : 2 * T, p.max_tasks);
    if (!p.replay) return;
    // export blocks: the listed tiles' key blocks in list order
    __syncthreads();   // the task entries are written (global, same block)
    int carry = 0;
    for (int base = 0; base < keyed; base += 256) {
        const int i = base + tid;
        const int J = i < keyed ? (p.tasks[i].w & 0x3FFFFFFF) : 0;
        int total = 0;
        const int ex = block_scan_256(J, sbuf, &total);
        if (i < keyed) p.exp_base[i] = carry + ex;
        carry += total;
    }
    if (tid == 0 && carry > p.exp_cap) atomicOr(p.err, 4u);   // a kv_len above max_kv_len
}

// Block 0 builds the task list; every block stages key rows: sequence b's keys
// at rows [off_b, off_b + kv_len_b), off_b the sum of the earlier sequences'
// padded lengths: staged[off_b + j] = ckv[kv_indices[kv_indptr[b] + j]] |
// kpe[...], then zero rows up to the next multiple of kMlaSeqAlign, so a
// 128-row box of one sequence never reaches the next sequence's keys.  Keys
// whose kv_indices entry lies past nnz are staged as zero rows (and
// reported); rows past stage_rows are not written (their boxes read the
// tensor map's zero fill).  One warp per row; each warp walks the sequences
// forward as its rows advance.
__global__ void __launch_bounds__(256) mla_stage_kernel(const MlaParams p) {
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
    if (blockIdx.x == 0) {
        if (threadIdx.x == 0 && p.kv_indptr[p.batch] > p.nnz) atomicOr(p.err, 2u);
        mla_build_tasks(p);
    }
    if (p.num_pages <= 0) return;
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

// One value swapped between the two softmax warps of a TMEM quadrant through
// shared memory: xa completes when both wrote, xb when both read (its wait
// comes before the next write).  x counts the swaps done (the phase).  False
// if a wait timed out.
__device__ __forceinline__ bool mla_swap(uint64_t* xa, uint64_t* xb, int& x, float* mine_slot,
                                         const float* peer_slot, float mine, float& theirs) {
    if (x >= 1 && !mbar_wait(xb, (x - 1) & 1)) return false;   // the partner read the last value
    *mine_slot = mine;
    mbar_arrive(xa);
    if (!mbar_wait(xa, x & 1)) return false;
    theirs = *peer_slot;
    mbar_arrive(xb);
    ++x;
    return true;
}

// One task of the list, as every role of both CTAs of a pair decodes it.
struct MlaTask {
    int q0, q_len, kv0, prefix, tok0, ntok, n_keys, J, half;
};

__device__ __forceinline__ MlaTask mla_task(const MlaParams& p, int idx, uint32_t rank) {
    const int4 e = p.tasks[idx];
    MlaTask t;
    const int b = e.x, i0 = e.y;
    t.kv0 = e.z;
    t.J = e.w & 0x3FFFFFFF;
    t.half = (e.w >> 30) & 1;
    t.q0 = p.qo_indptr[b];
    t.q_len = p.qo_indptr[b + 1] - t.q0;
    const int kv_len = p.kv_indptr[b + 1] - p.kv_indptr[b];
    t.prefix = kv_len - t.q_len;
    const int ntok_pair = min(mla::kPairTok, t.q_len - i0);
    t.tok0 = i0 + (int)rank * mla::kTok;
    t.ntok = max(0, min(mla::kTok, t.q_len - t.tok0));
    t.n_keys = (p.num_pages > 0 && p.stage_rows > 0) ? max(0, min(kv_len, t.prefix + i0 + ntok_pair)) : 0;
    return t;
}

// STRESS: compiled with the pauses of pkv_set_stress_delay (race testing); the
// ordinary instantiation has none, so the test facility costs it nothing.
template <bool STRESS>
__global__ void __cluster_dims__(2, 1, 1) __launch_bounds__(mla::kThreads, 1)
    mla_prefill_kernel(const MlaParams p, const __grid_constant__ CUtensorMap tm_qn,
                       const __grid_constant__ CUtensorMap tm_qp, const __grid_constant__ CUtensorMap tm_k,
                       const __grid_constant__ CUtensorMap tm_v) {
    using namespace mla;
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    uint8_t* sQ = smem;
    uint8_t* sRing = sQ + kQChunks * kQChunk;
    float* red = reinterpret_cast<float*>(sRing + kStages * kSlot);   // [2][kRows]
    uint64_t* bars = reinterpret_cast<uint64_t*>(reinterpret_cast<uint8_t*>(red) + kRedBytes);
    uint64_t* full = bars;                     // [kStages] CTA 0: both CTAs' copies of a slot landed
    uint64_t* empty = bars + kStages;          // [kStages] the MMAs read the slot (both CTAs)
    uint64_t* q_full = bars + 2 * kStages;     // [kQChunks] CTA 0: both CTAs' Q chunk landed (per task)
    uint64_t* q_free = q_full + kQChunks;      // the task's last S MMAs done: Q may be replaced (both)
    uint64_t* s_full = q_free + 1;             // [2] per S buffer: the scores are in TMEM (both CTAs)
    uint64_t* p_full = s_full + 2;             // [2] per S buffer, CTA 0: both CTAs wrote P over them
    uint64_t* mma_done = p_full + 2;
    uint64_t* xa = mma_done + 1;               // [4] per TMEM quadrant: both softmax warps wrote `red`
    uint64_t* xb = xa + 4;                     // [4] per TMEM quadrant: both read the partner's value
    uint64_t* task_bar = xb + 4;               // [4] a task index handed out is in task_slot (both CTAs)
    // [2] per S buffer: O += P.V of its latest block done (both CTAs).  One
    // barrier per buffer, not one for all blocks: every wait on it then has
    // exactly one such MMA outstanding, so the phase parity names it.  (With a
    // single barrier, a softmax warp at the end of a task could find the P.V
    // of its last two blocks both pending -- the last block's S completes
    // before they are issued -- and a parity wait for the last one passed.)
    uint64_t* pv_buf = task_bar + 4;
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(bars + kBars);
    volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);
    int* task_slot = reinterpret_cast<int*>(tmem_slot + 2);   // [4]

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const uint32_t rank = cluster_ctarank();   // 0 issues the MMAs
    const int pair = blockIdx.x >> 1, pairs = gridDim.x >> 1;

    if (threadIdx.x == 0) {
        for (int i = 0; i < kStages; ++i) {
            mbar_init(&full[i], 1);
            mbar_init(&empty[i], 1);
        }
        for (int i = 0; i < kQChunks; ++i) mbar_init(&q_full[i], 1);
        mbar_init(q_free, 1);
        for (int i = 0; i < 2; ++i) {
            mbar_init(&s_full[i], 1);
            mbar_init(&p_full[i], 2 * kSoftmaxWarps);   // every softmax warp of both CTAs
        }
        mbar_init(mma_done, 1);
        for (int i = 0; i < 2; ++i) mbar_init(&pv_buf[i], 1);
        for (int i = 0; i < 4; ++i) {
            mbar_init(&xa[i], 64);
            mbar_init(&xb[i], 64);
            mbar_init(&task_bar[i], 1);
        }
        fence_barrier_init();
        *abort_flag = 0;
    }
    if (warp == 1) {
        tmem_alloc_pair(tmem_slot, 512);
        tmem_relinquish_pair();
    }
    // the task list and the staged keys are written by the preceding grid
    asm volatile("griddepcontrol.wait;" ::: "memory");
    // the replay grid may start its set-up once every CTA of this one runs (it
    // waits for this grid's completion before reading the export)
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
    const int n_tasks = p.task_count[0], n_keyed = p.task_count[1];
    tc_fence_before();
    cluster_sync();   // both CTAs: barriers initialised, TMEM allocated
    tc_fence_after();
    const uint32_t tmem = *tmem_slot;
    // Tasks with keys are handed out one at a time, in list order (longest
    // first), by CTA 0's producer thread, which takes the next one from a
    // counter in the workspace when it starts on it and passes its index to
    // every role of both CTAs through task_slot / task_bar (4 entries, used in
    // turn: task r in entry r % 4; index -1 ends the list).  An entry is
    // reused only after every role has moved past the task it held: the
    // producer starts task r + 4 after it has loaded every ring slot of task
    // r + 3, which the MMA thread frees only while working on task r + 2 or
    // later, and each of those needs the softmax warps' P of that task.
    auto hand_out = [&](int r) -> int {
        int idx = atomicAdd(&p.task_count[2], 1);
        if (idx >= n_keyed) idx = -1;
        task_slot[r & 3] = idx;
        st_shared_cluster(mapa_shared(smem_u32(&task_slot[r & 3]), 1), idx);
        mbar_arrive(&task_bar[r & 3]);
        mbar_arrive_release_cluster(mapa_shared(smem_u32(&task_bar[r & 3]), 1));
        return idx;
    };
    // -2: the wait timed out
    auto next_task = [&](int r) -> int {
        if (!mbar_wait_acq_cluster(&task_bar[r & 3], (r >> 2) & 1)) return -2;
        return *reinterpret_cast<volatile int*>(&task_slot[r & 3]);
    };

    if (warp == 0) {
        // ------------------------------------------------------------ producer
        // Both CTAs load their halves; the copies complete on CTA 0's barriers,
        // whose expected byte counts (set by CTA 0 alone) cover both halves.
        // Per key block: 5 K slots (columns 64c .. 64c + 127 of this CTA's 64
        // keys, c = 0, 2, 4, 6; then the kpe columns 512 .. 575 alone) and 2 V
        // slots (this CTA's 128 output columns of keys 0-63, then 64-127), in
        // the MMA thread's order: per task K(0), then K(j + 1) and V(j) for
        // each block j.  A task's Q comes chunk by chunk, each just ahead of
        // the first K slot that needs it, once the previous task's last S
        // MMAs have released the Q buffer.
        if (lane == 0) {
            prefetch_tensormap(&tm_k);
            prefetch_tensormap(&tm_v);
            const bool lead = rank == 0;
            bool ok = true;
            int k = 0, stage = 0, n = 0;   // ring slots, ring index, tasks with keys
            uint32_t phase = 0;
            auto load_slot = [&](int row, int c, int v, int half) -> bool {
                if (k >= kStages && !(mbar_wait(&empty[stage], phase ^ 1) && *abort_flag == 0)) return false;
                uint8_t* dst = sRing + stage * kSlot;
                const uint32_t bar = mapa_shared(smem_u32(&full[stage]), 0);
                if (v < 0) {
                    const int subs = c < 4 ? 2 : 1;
                    if (lead) mbar_arrive_expect_tx(&full[stage], 2 * subs * kSub);
                    for (int s2 = 0; s2 < subs; ++s2)
                        tma_load_2d_pair(dst + s2 * kSub, &tm_k, bar, (2 * c + s2) * 64, row + (int)rank * kHalfKeys);
                } else {
                    if (lead) mbar_arrive_expect_tx(&full[stage], 2 * kSlot);
#pragma unroll
                    for (int w = 0; w < 2; ++w)
#pragma unroll
                        for (int nn = 0; nn < 2; ++nn)
                            tma_load_2d_pair(dst + w * kSub + nn * 4096, &tm_v, bar,
                                             half * 256 + (int)rank * 128 + nn * 64, row + v * 64 + w * 32);
                }
                if (STRESS && p.stress_ns) __nanosleep(p.stress_ns);
                ++k;
                if (++stage == kStages) {
                    stage = 0;
                    phase ^= 1;
                }
                return true;
            };
            for (int r = 0; ok; ++r) {
                const int idx = lead ? hand_out(r) : next_task(r);
                if (idx < 0) {
                    ok = idx == -1;
                    break;
                }
                const MlaTask t = mla_task(p, idx, rank);
                const int y = (t.q0 + t.tok0) * kHeads;   // rows past the tensor are zero-filled
                auto load_q = [&](int c) {
                    if (lead) mbar_arrive_expect_tx(&q_full[c], 2 * kQChunk);
                    const uint32_t bar = mapa_shared(smem_u32(&q_full[c]), 0);
                    if (c < kQChunks - 1)
                        tma_load_2d_pair(sQ + c * kQChunk, &tm_qn, bar, c * 64, y);
                    else
                        tma_load_2d_pair(sQ + c * kQChunk, &tm_qp, bar, 0, y);
                    if (STRESS && p.stress_ns) __nanosleep(p.stress_ns);
                };
                // the previous task's S MMAs are done with Q
                if (n >= 1 && !(mbar_wait(q_free, (n - 1) & 1) && *abort_flag == 0)) {
                    ok = false;
                    break;
                }
                for (int c = 0; c < kKSlots && ok; ++c) {   // K(0), with Q
                    load_q(2 * c);
                    if (c < 4) load_q(2 * c + 1);
                    ok = load_slot(t.kv0, c, -1, t.half);
                }
                for (int jb = 0; jb < t.J && ok; ++jb) {
                    if (jb + 1 < t.J)
                        for (int c = 0; c < kKSlots && ok; ++c) ok = load_slot(t.kv0 + (jb + 1) * kKeys, c, -1, t.half);
                    for (int v = 0; v < kVSlots && ok; ++v) ok = load_slot(t.kv0 + jb * kKeys, 0, v, t.half);
                }
                ++n;
            }
            if (!ok) {
                *abort_flag = 1;
                atomicOr(p.err, kErrTimeout);
            }
            // CTA 0: never leave with copies in flight into either CTA's shared
            // memory: wait for the last fill of every slot and of Q (immediate
            // unless the pipeline aborted).  CTA 1 cannot observe its copies;
            // it stays resident until CTA 0 is past this point (cluster barrier
            // below).
            if (lead) {
                for (int kk = max(0, k - kStages); kk < k; ++kk)
                    mbar_wait(&full[kk % kStages], (kk / kStages) & 1);
                if (n >= 1)
                    for (int c = 0; c < kQChunks; ++c) mbar_wait(&q_full[c], (n - 1) & 1);
            }
        }
        __syncwarp();
    } else if (warp == 1 && rank == 1) {
        // CTA 0's last commit also arrives here: no MMA of the pair still reads
        // this CTA's shared memory or writes its TMEM after it.
        if (lane == 0) mbar_wait(mma_done, 0);
        __syncwarp();
    } else if (warp == 1) {
        // ------------------------------------------------ CTA 0: the MMA issuer
        // Per task: S(0); then for each block j: S(j + 1) into the other S
        // buffer (the tensor core works on it while the softmax warps turn
        // S(j) into P(j)), then O += P(j).V(j).  S buffers alternate over the
        // blocks of all tasks (G counts them).  S(j + 2) reuses P(j)'s columns
        // only once O += P(j).V(j) has completed (pv_buf); a task's first
        // O += P.V overwrites O, which the
        // softmax warps have read out by then (they write that block's P
        // after their epilogue).  Kept lean: the thread waits ~70 cycles per
        // issued MMA for the pipe anyway, so descriptors are formed once and
        // advanced by adding the address step (16 bytes per unit; every
        // operand address stays below 256 KB, so the 14-bit field never
        // carries), and the ring index and phase are counters.
        if (lane == 0) {
            const uint32_t idesc_qk = umma_idesc_bf16_f32(2 * kRows, kKeys, false);
            const uint32_t idesc_pv = umma_idesc_bf16_f32(2 * kRows, 256, true);
            const uint64_t dq = umma_desc_sw128(smem_u32(sQ), 16, 1024);
            const uint64_t dk = umma_desc_sw128(smem_u32(sRing), 16, 1024);
            const uint64_t dv = umma_desc_sw128(smem_u32(sRing), 4096, 1024);
            bool ok = true;
            int stage = 0, n = 0, G = 0;   // ring index, tasks with keys, blocks issued before this task
            uint32_t phase = 0;
            auto next = [&]() {
                if (++stage == kStages) {
                    stage = 0;
                    phase ^= 1;
                }
            };
            // S(block g)[256 rows][128 keys] = Q . K^T into buffer g % 2: A rows from each
            // CTA's Q chunk, B keys 64 from each CTA's sub-chunk (K-major, 8-row groups
            // 1 KB apart); 4 MMAs of 16 columns per sub-chunk
            auto issue_s = [&](int g, bool first, bool last) -> bool {
                const uint32_t d = tmem + kColS + (g & 1) * 128;
                // The buffer holds P(g - 2), the TMEM operand of O += P(g - 2).V:
                // that MMA completes before these overwrite it.
                if (g >= 2) {
                    if (!mbar_wait(&pv_buf[g & 1], ((g - 2) >> 1) & 1)) return false;
                    tc_fence_after();
                }
                for (int c = 0; c < kKSlots; ++c) {
                    if (first) {   // Q arrives chunk by chunk with the task's first block
                        if (!mbar_wait(&q_full[2 * c], n & 1) || (c < 4 && !mbar_wait(&q_full[2 * c + 1], n & 1)))
                            return false;
                        tc_fence_after();
                    }
                    // TMA data only: no tcgen05 fence
                    if (!mbar_wait(&full[stage], phase)) return false;
                    const uint64_t a0 = dq + (uint64_t)((2 * c * kQChunk) >> 4);
                    const uint64_t b0 = dk + (uint64_t)((stage * kSlot) >> 4);
#pragma unroll
                    for (int s2 = 0; s2 < 2; ++s2) {
                        if (s2 == 1 && c == kKSlots - 1) break;   // the kpe slot holds one sub-chunk
#pragma unroll
                        for (int kk = 0; kk < 4; ++kk)
                            umma_bf16_pair(d, a0 + (uint64_t)((s2 * kQChunk + kk * 32) >> 4),
                                           b0 + (uint64_t)((s2 * kSub + kk * 32) >> 4), idesc_qk, (c | s2 | kk) != 0);
                    }
                    umma_commit_pair_mc(&empty[stage], kBothCtas);
                    next();
                    if (STRESS && p.stress_consumer_ns) __nanosleep(p.stress_consumer_ns);
                }
                umma_commit_pair_mc(&s_full[g & 1], kBothCtas);
                if (last) umma_commit_pair_mc(q_free, kBothCtas);   // Q no longer read
                return true;
            };
            // O += P(g).V(g): keys 64v + 32w + 16kk .. +15 are P columns 64v + 16w + 8kk of
            // buffer g % 2; B = 16 key rows of the 256 output columns, 128 from each CTA's
            // sub-chunk w (MN-major: two 64-column blocks 4 KB apart, 8-row groups 1 KB apart)
            auto issue_pv = [&](int g, bool first) -> bool {
                if (!(mbar_wait(&p_full[g & 1], (g >> 1) & 1) && *abort_flag == 0)) return false;
                tc_fence_after();
                const uint32_t a_p = tmem + kColS + (g & 1) * 128;
                for (int v = 0; v < kVSlots; ++v) {
                    if (!mbar_wait(&full[stage], phase)) return false;
                    const uint64_t b0 = dv + (uint64_t)((stage * kSlot) >> 4);
#pragma unroll
                    for (int w = 0; w < 2; ++w)
#pragma unroll
                        for (int kk = 0; kk < 2; ++kk)
                            umma_bf16_tmem_a_pair(tmem, a_p + v * 64 + w * 16 + kk * 8,
                                                  b0 + (uint64_t)((w * kSub + kk * 2048) >> 4), idesc_pv,
                                                  !first || (v | w | kk) != 0);
                    umma_commit_pair_mc(&empty[stage], kBothCtas);
                    next();
                    if (STRESS && p.stress_consumer_ns) __nanosleep(p.stress_consumer_ns);
                }
                umma_commit_pair_mc(&pv_buf[g & 1], kBothCtas);
                return true;
            };
            for (int r = 0; ok; ++r) {
                const int idx = next_task(r);
                if (idx < 0) {
                    ok = idx == -1;
                    break;
                }
                const int J = p.tasks[idx].w & 0x3FFFFFFF;
                ok = issue_s(G, true, J == 1);
                for (int j = 0; j < J && ok; ++j) {
                    if (j + 1 < J) ok = issue_s(G + j + 1, false, j + 2 == J);
                    ok = ok && issue_pv(G + j, j == 0);
                }
                G += J;
                ++n;
            }
            if (!ok) {
                *abort_flag = 1;
                atomicOr(p.err, kErrTimeout);
            }
            // never free TMEM with MMAs in flight (the commit reaches both CTAs)
            umma_commit_pair_mc(mma_done, kBothCtas);
            mbar_wait(mma_done, 0);
        }
        __syncwarp();
    } else {
        // ------------------------------------------------------------- softmax
        // Two warps per TMEM lane quadrant (a warp reaches only the lanes
        // 32 * (warp % 4) ..): warp group kh = 0 takes keys 0-63 of every
        // block, kh = 1 keys 64-127.  A warp reads its 64 scores, then the
        // two warps of a quadrant swap their row maxima through shared memory
        // (mbarriers xa: both wrote, xb: both read; every wait bounded), so
        // both apply the same running maximum and lazy-rescale decision.  Each
        // keeps a partial row sum, rescales and writes 128 of the 256 output
        // columns; the sums are merged at the end of a task the same way.
        const int quad = warp & 3;
        const int kh = (warp - 2) >> 2;   // key half of the block
        const int row = quad * 32 + lane;
        const uint32_t t_row = tmem + ((uint32_t)(quad * 32) << 16);
        const float sc = p.scale_log2;
        float* my_red = red + kh * kRows + row;
        const float* peer_red = red + (kh ^ 1) * kRows + row;
        int x = 0;       // swaps done (phase of xa / xb)
        int G = 0;       // blocks of the earlier tasks
        bool ok = true;
        // tasks without a visible key (empty KV), listed last: out = 0, lse = -inf
        for (int idx = n_keyed + pair; idx < n_tasks; idx += pairs) {
            const MlaTask t = mla_task(p, idx, rank);
            const int tok = t.tok0 + row / kHeads;
            const size_t tq = (size_t)(t.q0 + tok);
            const int h = row % kHeads;
            if (row / kHeads < t.ntok) {
                uint4* orow = reinterpret_cast<uint4*>(p.out + (tq * kHeads + h) * kDc + t.half * 256 + kh * 128);
                for (int c = 0; c < 16; ++c) orow[c] = make_uint4(0u, 0u, 0u, 0u);
                if (t.half == 0 && kh == 0) p.lse[tq * kHeads + h] = -INFINITY;
            }
        }
        for (int r = 0; ok; ++r) {
            int idx = 0;
            if (lane == 0) idx = next_task(r);
            idx = __shfl_sync(0xffffffffu, idx, 0);   // warp-uniform
            if (idx < 0) {
                ok = idx == -1;
                break;
            }
            const MlaTask t = mla_task(p, idx, rank);
            const int tok = t.tok0 + row / kHeads;
            const bool live = row / kHeads < t.ntok;
            const size_t tq = (size_t)(t.q0 + tok);
            const int h = row % kHeads;
            __nv_bfloat16* orow = p.out + (tq * kHeads + h) * kDc + t.half * 256 + kh * 128;
            const int lim = t.prefix + tok;   // last visible key of this row
            // keys <= this are visible to every row of this CTA: blocks below it need no mask
            const int unmasked_below = min(t.prefix + t.tok0, t.n_keys - 1);
            // replay: the first half's tasks export their blocks for the second
            const int xb0 = (p.replay && t.half == 0) ? p.exp_base[idx] : 0;
            const bool xp = p.replay && t.half == 0 && xb0 + t.J <= p.exp_cap;
            float m = -INFINITY, l = 0.f;
            for (int j = 0; j < t.J; ++j) {
                const int g = G + j;
                const bool got = mbar_wait(&s_full[g & 1], (g >> 1) & 1);
                if (!__all_sync(0xffffffffu, got && *abort_flag == 0)) {
                    ok = false;
                    break;
                }
                tc_fence_after();
                const uint32_t t_s = t_row + kColS + (g & 1) * 128 + kh * 64;   // this warp's scores, then P
                float s[kKeys / 2];   // this warp's 64 keys
                {
                    float v0[32], v1[32];
                    tmem_ld32(t_s, v0);
                    tmem_ld32(t_s + 32, v1);
                    tmem_wait_ld();
#pragma unroll
                    for (int i = 0; i < 32; ++i) {
                        s[i] = v0[i];
                        s[32 + i] = v1[i];
                    }
                }

                // scale to log2 units, mask, row maximum (8 independent chains)
                float mx8[8];
#pragma unroll
                for (int i = 0; i < 8; ++i) mx8[i] = -INFINITY;
                const int key0 = j * kKeys + kh * 64;
                if (j * kKeys + kKeys - 1 <= unmasked_below) {
#pragma unroll
                    for (int c = 0; c < kKeys / 2; ++c) {
                        s[c] *= sc;
                        mx8[c & 7] = fmaxf(mx8[c & 7], s[c]);
                    }
                } else {
#pragma unroll
                    for (int c = 0; c < kKeys / 2; ++c) {
                        const int key = key0 + c;
                        s[c] = (key <= lim && key < t.n_keys) ? s[c] * sc : -INFINITY;
                        mx8[c & 7] = fmaxf(mx8[c & 7], s[c]);
                    }
                }
                float mx = fmaxf(fmaxf(fmaxf(mx8[0], mx8[1]), fmaxf(mx8[2], mx8[3])),
                                 fmaxf(fmaxf(mx8[4], mx8[5]), fmaxf(mx8[6], mx8[7])));
                float mx_peer = -INFINITY;
                if (!__all_sync(0xffffffffu, mla_swap(&xa[quad], &xb[quad], x, my_red, peer_red, mx, mx_peer))) {
                    ok = false;
                    break;
                }
                mx = fmaxf(mx, mx_peer);
                const float m_new = fmaxf(m, mx);
                float m_use = m, alpha = 1.f;
                if (m == -INFINITY || m_new > m + kLazyRescale) {
                    m_use = m_new == -INFINITY ? 0.f : m_new;
                    alpha = ex2(m - m_use);
                }
                float ls8[8];
#pragma unroll
                for (int i = 0; i < 8; ++i) ls8[i] = 0.f;
#pragma unroll
                for (int c = 0; c < kKeys / 2; ++c) {
                    s[c] = ex2(s[c] - m_use);
                    ls8[c & 7] += s[c];
                }
                const float ls = ((ls8[0] + ls8[1]) + (ls8[2] + ls8[3])) + ((ls8[4] + ls8[5]) + (ls8[6] + ls8[7]));
                l = l * alpha + ls;
                m = m_use;

                bool got2 = true;
                if (j >= 1 && __any_sync(0xffffffffu, alpha != 1.f)) {
                    // O holds P(j-1).V: wait for it, then rescale this warp's rows (its 128 columns).
                    got2 = mbar_wait(&pv_buf[(g - 1) & 1], ((g - 1) >> 1) & 1);
                    if (__all_sync(0xffffffffu, got2 && *abort_flag == 0)) {
                        tc_fence_after();
#pragma unroll 1
                        for (int c = 0; c < 128 / 32; ++c) {
                            float o[32];
                            tmem_ld32(t_row + kh * 128 + c * 32, o);
                            tmem_wait_ld();
#pragma unroll
                            for (int i = 0; i < 32; ++i) o[i] *= alpha;
                            tmem_st32(t_row + kh * 128 + c * 32, o);
                        }
                        tmem_wait_st();
                    }
                }
                if (!__all_sync(0xffffffffu, got2 && *abort_flag == 0)) {
                    ok = false;
                    break;
                }
                uint32_t pk[32];
#pragma unroll
                for (int i = 0; i < 32; ++i) pk[i] = Mma<__nv_bfloat16>::pack(s[2 * i], s[2 * i + 1]);
                tmem_st32(t_s, pk);   // over this warp's own scores, already read
                tmem_wait_st();
                tc_fence_before();
                __syncwarp();
                if (lane == 0) mbar_arrive_remote(mapa_shared(smem_u32(&p_full[g & 1]), 0));
                if (xp) {
                    // The export, after p_full so that O += P.V need not wait for it: P
                    // (keys 2i, 2i + 1 in word i) chunk-major, 16 bytes (8 keys) of each
                    // row, row after row, so that each store of the warp writes 512
                    // contiguous bytes; the factor O was rescaled by; the flag.
                    const size_t eb = (size_t)(xb0 + j) * 2 + rank;
                    uint4* dst = reinterpret_cast<uint4*>(p.exp_p + (eb * 2 + kh) * (kRows * 64)) + row;
#pragma unroll
                    for (int q = 0; q < 8; ++q)
                        dst[q * kRows] = make_uint4(pk[4 * q], pk[4 * q + 1], pk[4 * q + 2], pk[4 * q + 3]);
                    if (kh == 0) p.exp_alpha[eb * kRows + row] = alpha;
                    const bool any = __any_sync(0xffffffffu, j >= 1 && alpha != 1.f);
                    if (lane == 0) p.exp_flag[eb * 8 + (warp - 2)] = any ? 1 : 0;
                }
                if (STRESS && p.stress_consumer_ns) __nanosleep(p.stress_consumer_ns);
            }
            if (!ok) break;
            G += t.J;
            // O complete after the task's last O += P.V
            // The S of the task's last block completing says nothing of the
            // O += P.V of its last two blocks: wait for both.
            bool done = t.J < 2 || mbar_wait(&pv_buf[(G - 2) & 1], ((G - 2) >> 1) & 1);
            done = done && mbar_wait(&pv_buf[(G - 1) & 1], ((G - 1) >> 1) & 1);
            ok = __all_sync(0xffffffffu, done && *abort_flag == 0);
            tc_fence_after();
            // the quadrant's two partial row sums (a partner that left early never
            // arrives; the bounded wait then ends with no output written)
            float l_peer = 0.f;
            ok = __all_sync(0xffffffffu, ok && mla_swap(&xa[quad], &xb[quad], x, my_red, peer_red, l, l_peer));
            if (!ok) break;
            l += l_peer;
            if (xp && kh == 0) p.exp_l[((size_t)idx * 2 + rank) * kRows + row] = l;
            const float inv = l > 0.f ? 1.f / l : 0.f;
#pragma unroll 1
            for (int c = 0; c < 128 / 32; ++c) {
                float o[32];
                tmem_ld32(t_row + kh * 128 + c * 32, o);
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
            if (live && t.half == 0 && kh == 0) p.lse[tq * kHeads + h] = l > 0.f ? m + log2f(l) : -INFINITY;
            tc_fence_before();   // O read out before this warp's next P store lets O be overwritten
        }
        if (!ok) {
            *abort_flag = 1;
            if (lane == 0) atomicOr(p.err, kErrTimeout);
        }
    }

    // Both CTAs: every role is done with the pair's barriers, shared memory
    // and TMEM before either CTA frees its TMEM or exits.
    tc_fence_before();
    cluster_sync();
    tc_fence_after();
    if (warp == 1) tmem_dealloc_pair(tmem, 512);
}

namespace mla {
constexpr int kRStages = 12;              // replay ring: P chunks and V slots, 16 KB each
constexpr int kRBars = 2 * kRStages + 10;
constexpr int kRSmemBytes = 1024 + kRStages * kSlot + kRBars * 8 + 32;
static_assert(kRSmemBytes <= 232448, "shared memory per CTA");
}  // namespace mla

// The second output half of every row tile with keys, from what the first
// half's tasks exported (replay): per key block j, O += P(j).V(j) with the
// exported bf16 P(j) as the shared-memory A operand (copied as exported:
// K-major without swizzle, 8 keys of every row per 2 KB, so that the
// exporting warps' stores are coalesced), and before a block for which the first half
// rescaled its O, the same rescale of this O by the exported factors; at the
// end O / l with the exported row sums.  The arithmetic is the first half
// task's, so the result equals computing S again for this half.
//
// Same pairs as the prefill kernel: CTA r holds rows 128r .. 128r + 127 of
// the tile, their 256 output columns O in TMEM, and loads its 128 rows of
// each P chunk (keys 64c .. 64c + 63 of a block) and 128 of the 256 output
// columns of V; CTA 0's one thread issues the MMAs (M = 256, N = 256).
// Ring order per block: P chunk 0, V keys 0-63, P chunk 1, V keys 64-127.
// A rescale is a hand-off: the MMA thread lets every MMA issued so far
// complete (drain), asks the scale warps of both CTAs (resc_req), and waits
// for all of them (resc_done) before the block's MMAs.  Each request is
// answered before the next, and each task's O is read out (o_free) before
// the next task's first MMA overwrites it, so every wait has one phase
// outstanding.
template <bool STRESS>
__global__ void __cluster_dims__(2, 1, 1) __launch_bounds__(mla::kThreads, 1)
    mla_replay_kernel(const MlaParams p, const __grid_constant__ CUtensorMap tm_p,
                      const __grid_constant__ CUtensorMap tm_v) {
    using namespace mla;
    extern __shared__ uint8_t smem_raw[];
    uint8_t* sRing = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    uint64_t* bars = reinterpret_cast<uint64_t*>(sRing + kRStages * kSlot);
    uint64_t* full = bars;                     // [kRStages] CTA 0: both CTAs' copies of a slot landed
    uint64_t* empty = bars + kRStages;         // [kRStages] the MMAs read the slot (both CTAs)
    uint64_t* resc_req = empty + kRStages;     // O may be rescaled (both CTAs)
    uint64_t* resc_done = resc_req + 1;        // CTA 0: every scale warp of both CTAs rescaled
    uint64_t* o_ready = resc_done + 1;         // the task's MMAs are done (both CTAs)
    uint64_t* o_free = o_ready + 1;            // CTA 0: every warp of both CTAs read O out
    uint64_t* drain = o_free + 1;              // CTA 0: the MMAs issued so far are done
    uint64_t* mma_done = drain + 1;            // both CTAs: the last MMA is done
    uint64_t* task_bar = mma_done + 1;         // [4] a task index handed out is in task_slot (both CTAs)
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(bars + kRBars);
    volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);
    int* task_slot = reinterpret_cast<int*>(tmem_slot + 2);   // [4]

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const uint32_t rank = cluster_ctarank();   // 0 issues the MMAs

    if (threadIdx.x == 0) {
        for (int i = 0; i < kRStages; ++i) {
            mbar_init(&full[i], 1);
            mbar_init(&empty[i], 1);
        }
        mbar_init(resc_req, 1);
        mbar_init(resc_done, 2 * kSoftmaxWarps);
        mbar_init(o_ready, 1);
        mbar_init(o_free, 2 * kSoftmaxWarps);
        mbar_init(drain, 1);
        mbar_init(mma_done, 1);
        for (int i = 0; i < 4; ++i) mbar_init(&task_bar[i], 1);
        fence_barrier_init();
        *abort_flag = 0;
    }
    if (warp == 1) {
        tmem_alloc_pair(tmem_slot, 256);
        tmem_relinquish_pair();
    }
    // the lists and the export are written by the preceding grids
    asm volatile("griddepcontrol.wait;" ::: "memory");
    const int n_rep = p.task_count[4], L = p.task_count[5];
    tc_fence_before();
    cluster_sync();
    tc_fence_after();
    const uint32_t tmem = *tmem_slot;
    // replay tasks handed out one at a time by CTA 0's producer (as in the prefill kernel)
    auto hand_out = [&](int r) -> int {
        int pos = atomicAdd(&p.task_count[3], 1);
        if (pos >= n_rep) pos = -1;
        task_slot[r & 3] = pos;
        st_shared_cluster(mapa_shared(smem_u32(&task_slot[r & 3]), 1), pos);
        mbar_arrive(&task_bar[r & 3]);
        mbar_arrive_release_cluster(mapa_shared(smem_u32(&task_bar[r & 3]), 1));
        return pos;
    };
    auto next_task = [&](int r) -> int {
        if (!mbar_wait_acq_cluster(&task_bar[r & 3], (r >> 2) & 1)) return -2;
        return *reinterpret_cast<volatile int*>(&task_slot[r & 3]);
    };
    // some row of the pair was rescaled before export block xb (16 flag bytes)
    auto flags_of = [&](int xb) -> uint4 { return *reinterpret_cast<const uint4*>(p.exp_flag + (size_t)xb * 16); };
    auto any_flag = [](uint4 f) { return (f.x | f.y | f.z | f.w) != 0u; };

    if (warp == 0) {
        // ------------------------------------------------------------ producer
        if (lane == 0) {
            prefetch_tensormap(&tm_p);
            prefetch_tensormap(&tm_v);
            const bool lead = rank == 0;
            bool ok = true;
            int k = 0, stage = 0;   // ring slots, ring index
            uint32_t phase = 0;
            // P chunk c of export block xb (this CTA's 128 rows), or V keys
            // row + 64c .. + 63 (this CTA's 128 of the second half's columns)
            auto load = [&](int xb, int row, int c, bool is_p) -> bool {
                if (k >= kRStages && !(mbar_wait(&empty[stage], phase ^ 1) && *abort_flag == 0)) return false;
                uint8_t* dst = sRing + stage * kSlot;
                const uint32_t bar = mapa_shared(smem_u32(&full[stage]), 0);
                if (lead) mbar_arrive_expect_tx(&full[stage], 2 * kSlot);
                if (is_p) {
                    tma_load_2d_pair(dst, &tm_p, bar, 0, ((xb * 2 + (int)rank) * 2 + c) * kRows);
                } else {
#pragma unroll
                    for (int w = 0; w < 2; ++w)
#pragma unroll
                        for (int nn = 0; nn < 2; ++nn)
                            tma_load_2d_pair(dst + w * kSub + nn * 4096, &tm_v, bar, 256 + (int)rank * 128 + nn * 64,
                                             row + c * 64 + w * 32);
                }
                if (STRESS && p.stress_ns) __nanosleep(p.stress_ns);
                ++k;
                if (++stage == kRStages) {
                    stage = 0;
                    phase ^= 1;
                }
                return true;
            };
            for (int r = 0; ok; ++r) {
                const int pos = lead ? hand_out(r) : next_task(r);
                if (pos < 0) {
                    ok = pos == -1;
                    break;
                }
                const int4 e = p.tasks[L + pos];
                const int J = e.w & 0x3FFFFFFF, xb0 = p.exp_base[pos];
                for (int j = 0; j < J && ok; ++j)
                    for (int c = 0; c < 2 && ok; ++c) {
                        ok = load(xb0 + j, 0, c, true);
                        ok = ok && load(0, e.z + j * kKeys, c, false);
                    }
            }
            if (!ok) {
                *abort_flag = 1;
                atomicOr(p.err, kErrTimeout);
            }
            // CTA 0: no copy into either CTA's shared memory still in flight
            if (lead)
                for (int kk = max(0, k - kRStages); kk < k; ++kk) mbar_wait(&full[kk % kRStages], (kk / kRStages) & 1);
        }
        __syncwarp();
    } else if (warp == 1 && rank == 1) {
        if (lane == 0) mbar_wait(mma_done, 0);
        __syncwarp();
    } else if (warp == 1) {
        // ------------------------------------------------ CTA 0: the MMA issuer
        if (lane == 0) {
            const uint32_t idesc = umma_idesc_bf16_f32(2 * kRows, 256, true);
            // P: K-major without swizzle, as exported: 8 keys (16 bytes) of 128 rows per 2 KB,
            // 8-row core matrices 128 bytes apart
            const uint64_t da = umma_desc_noswizzle(smem_u32(sRing), 2048, 128);
            const uint64_t dv = umma_desc_sw128(smem_u32(sRing), 4096, 1024);   // V: MN-major, as in the prefill kernel
            bool ok = true;
            int stage = 0, n = 0, nreq = 0;   // ring index, tasks done, rescales (= drains) requested
            uint32_t phase = 0;
            auto next = [&]() {
                if (++stage == kRStages) {
                    stage = 0;
                    phase ^= 1;
                }
            };
            for (int r = 0; ok; ++r) {
                const int pos = next_task(r);
                if (pos < 0) {
                    ok = pos == -1;
                    break;
                }
                const int4 e = p.tasks[L + pos];
                const int J = e.w & 0x3FFFFFFF, xb0 = p.exp_base[pos];
                const bool fits = xb0 + J <= p.exp_cap;
                // the previous task's O is read out before this task's first MMA overwrites it
                if (n >= 1) {
                    if (!(mbar_wait_acq_cluster(o_free, (n - 1) & 1) && *abort_flag == 0)) {
                        ok = false;
                        break;
                    }
                    tc_fence_after();
                }
                uint4 fl = make_uint4(0u, 0u, 0u, 0u);   // flags of block j, loaded a block ahead
                if (fits && J > 1) fl = flags_of(xb0 + 1);
                for (int j = 0; j < J && ok; ++j) {
                    uint4 f = make_uint4(0u, 0u, 0u, 0u);
                    if (j >= 1) {
                        f = fl;
                        if (fits && j + 1 < J) fl = flags_of(xb0 + j + 1);
                    }
                    if (j >= 1 && any_flag(f)) {
                        umma_commit_pair_mc(drain, 1);   // O += P(j - 1).V and all before it
                        ok = mbar_wait(drain, nreq & 1);
                        tc_fence_after();
                        mbar_arrive(resc_req);
                        mbar_arrive_release_cluster(mapa_shared(smem_u32(resc_req), 1));
                        ok = ok && mbar_wait_acq_cluster(resc_done, nreq & 1) && *abort_flag == 0;
                        ++nreq;
                        tc_fence_after();
                        if (!ok) break;
                    }
                    for (int c = 0; c < 2 && ok; ++c) {
                        if (!mbar_wait(&full[stage], phase)) {
                            ok = false;
                            break;
                        }
                        const int sp = stage;
                        const uint64_t a0 = da + (uint64_t)((stage * kSlot) >> 4);
                        next();
                        if (!mbar_wait(&full[stage], phase)) {
                            ok = false;
                            break;
                        }
                        const uint64_t b0 = dv + (uint64_t)((stage * kSlot) >> 4);
                        // keys 16i .. 16i + 15 of the chunk: A key groups 2i, 2i + 1 (4 KB per
                        // 16 keys), B rows of V sub-chunk i / 2 (2 KB per 16 keys)
#pragma unroll
                        for (int i = 0; i < 4; ++i)
                            umma_bf16_pair(tmem, a0 + (uint64_t)((i * 4096) >> 4),
                                           b0 + (uint64_t)((((i >> 1) * kSub) + (i & 1) * 2048) >> 4), idesc,
                                           (j | c | i) != 0);
                        umma_commit_pair_mc(&empty[sp], kBothCtas);
                        umma_commit_pair_mc(&empty[stage], kBothCtas);
                        next();
                        if (STRESS && p.stress_consumer_ns) __nanosleep(p.stress_consumer_ns);
                    }
                }
                if (!ok) break;
                umma_commit_pair_mc(o_ready, kBothCtas);
                ++n;
            }
            if (!ok) {
                *abort_flag = 1;
                atomicOr(p.err, kErrTimeout);
            }
            umma_commit_pair_mc(mma_done, kBothCtas);
            mbar_wait(mma_done, 0);
        }
        __syncwarp();
    } else {
        // ---------------------------------------------- rescale and epilogue
        // Warp (quad, kh) as in the prefill kernel: rows quad * 32 + lane, O
        // columns 128 kh .. 128 kh + 127 of this half.
        const int quad = warp & 3;
        const int kh = (warp - 2) >> 2;
        const int row = quad * 32 + lane;
        const uint32_t t_row = tmem + ((uint32_t)(quad * 32) << 16);
        int n = 0, nreq = 0;
        bool ok = true;
        for (int r = 0; ok; ++r) {
            int pos = 0;
            if (lane == 0) pos = next_task(r);
            pos = __shfl_sync(0xffffffffu, pos, 0);
            if (pos < 0) {
                ok = pos == -1;
                break;
            }
            const MlaTask t = mla_task(p, L + pos, rank);
            const int xb0 = p.exp_base[pos];
            const bool fits = xb0 + t.J <= p.exp_cap;
            const float l = fits ? p.exp_l[((size_t)pos * 2 + rank) * kRows + row] : 0.f;
            for (int j = 1; j < t.J && fits; ++j) {
                if (!any_flag(flags_of(xb0 + j))) continue;
                const bool got = mbar_wait_acq_cluster(resc_req, nreq & 1);
                ++nreq;
                if (!__all_sync(0xffffffffu, got && *abort_flag == 0)) {
                    ok = false;
                    break;
                }
                tc_fence_after();
                const size_t eb = (size_t)(xb0 + j) * 2 + rank;
                if (p.exp_flag[eb * 8 + (warp - 2)]) {   // this warp's rows: as the first half did
                    const float alpha = p.exp_alpha[eb * kRows + row];
#pragma unroll 1
                    for (int c = 0; c < 128 / 32; ++c) {
                        float o[32];
                        tmem_ld32(t_row + kh * 128 + c * 32, o);
                        tmem_wait_ld();
#pragma unroll
                        for (int i = 0; i < 32; ++i) o[i] *= alpha;
                        tmem_st32(t_row + kh * 128 + c * 32, o);
                    }
                    tmem_wait_st();
                }
                tc_fence_before();
                __syncwarp();
                if (lane == 0) mbar_arrive_remote(mapa_shared(smem_u32(resc_done), 0));
            }
            if (!ok) break;
            ok = __all_sync(0xffffffffu, mbar_wait(o_ready, n & 1) && *abort_flag == 0);
            if (!ok) break;
            tc_fence_after();
            const int tok = t.tok0 + row / kHeads;
            const bool live = row / kHeads < t.ntok;
            const size_t tq = (size_t)(t.q0 + tok);
            __nv_bfloat16* orow = p.out + (tq * kHeads + row % kHeads) * kDc + 256 + kh * 128;
            const float inv = l > 0.f ? 1.f / l : 0.f;
#pragma unroll 1
            for (int c = 0; c < 128 / 32; ++c) {
                float o[32];
                tmem_ld32(t_row + kh * 128 + c * 32, o);
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
            tc_fence_before();   // O read out before the next task's first MMA overwrites it
            __syncwarp();
            if (lane == 0) mbar_arrive_remote(mapa_shared(smem_u32(o_free), 0));
            ++n;
        }
        if (!ok) {
            *abort_flag = 1;
            if (lane == 0) atomicOr(p.err, kErrTimeout);
        }
    }

    tc_fence_before();
    cluster_sync();
    tc_fence_after();
    if (warp == 1) tmem_dealloc_pair(tmem, 256);
}

cudaError_t launch_mla_prefill(const MlaParams& p, const MlaMaps& maps, cudaStream_t stream) {
    static std::atomic<bool> attr_set[kMaxDevices];
    static std::mutex attr_mu;
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    e = once_per_device(attr_set, attr_mu, dev, [] {
        cudaError_t r = cudaFuncSetAttribute(mla_prefill_kernel<false>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                             mla::kSmemBytes);
        if (r == cudaSuccess)
            r = cudaFuncSetAttribute(mla_prefill_kernel<true>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                     mla::kSmemBytes);
        if (r == cudaSuccess)
            r = cudaFuncSetAttribute(mla_replay_kernel<false>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                     mla::kRSmemBytes);
        if (r == cudaSuccess)
            r = cudaFuncSetAttribute(mla_replay_kernel<true>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                     mla::kRSmemBytes);
        return r;
    });
    if (e != cudaSuccess) return e;
    if (p.max_tasks <= 0) return cudaSuccess;
    int sms = 0;
    e = device_sm_count(dev, &sms);
    if (e != cudaSuccess) return e;
    // task list (block 0) and staged keys: one warp per staged row, capped at
    // 16 waves of 8-warp CTAs per SM
    const long long want = std::max<long long>(1, ((long long)p.stage_rows + 7) / 8);
    mla_stage_kernel<<<(unsigned)std::min<long long>(want, (long long)sms * 8 * 16), 256, 0, stream>>>(p);
    e = cudaGetLastError();
    if (e != cudaSuccess) return e;
    // persistent CTA pairs, one per two SMs (never more than the tasks)
    const long long pairs = std::min<long long>(p.max_tasks, std::max(1, sms / 2));
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)(2 * pairs));
    cfg.blockDim = dim3(mla::kThreads);
    cfg.dynamicSmemBytes = mla::kSmemBytes;
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    const bool stress = p.stress_ns || p.stress_consumer_ns;
    e = stress ? cudaLaunchKernelEx(&cfg, mla_prefill_kernel<true>, p, maps.q_nope, maps.q_pe, maps.kv, maps.v)
               : cudaLaunchKernelEx(&cfg, mla_prefill_kernel<false>, p, maps.q_nope, maps.q_pe, maps.kv, maps.v);
    if (e != cudaSuccess || !p.replay) return e;
    // the second output half from the export: the same persistent pairs, a
    // programmatic dependent of the prefill grid (set-up overlaps its tail)
    cfg.dynamicSmemBytes = mla::kRSmemBytes;
    return stress ? cudaLaunchKernelEx(&cfg, mla_replay_kernel<true>, p, maps.p_exp, maps.v)
                  : cudaLaunchKernelEx(&cfg, mla_replay_kernel<false>, p, maps.p_exp, maps.v);
}

}  // namespace pkv
