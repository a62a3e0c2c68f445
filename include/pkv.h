/*
 * pkv.h -- C ABI of libpkv: paged-KV-cache attention for LLM decode on GB300
 * (sm_103a), and its MLA paged causal prefill variant.
 *
 * Conventions shared by every entry point:
 *  - Pointers named as tensors are DEVICE pointers owned by the caller; the
 *    library never allocates, frees, copies to the host or synchronises.
 *    Shapes are passed explicitly; every tensor is dense and row-major in the
 *    layout written beside it.
 *  - Work is enqueued on `stream` (a cudaStream_t; NULL = legacy default
 *    stream) and the call returns without waiting for it.
 *  - Every call returns a pkv_status.  Argument errors are found on the host
 *    before anything is launched; nothing on the device traps or asserts.
 *  - 16-bit floating-point data is fp16 or bf16 (pkv_dtype); arithmetic is
 *    fp32 with fp32 softmax statistics.
 *
 * Sources, cited by page title and function:
 *  [V2]  "paged_attention_v2_triton.py -- CCCL-derived Triton PagedAttention V2"
 *        (paged_attention_v2_triton launcher, _partition_attn_kernel,
 *        _reduce_partitions_kernel).
 *  [FD]  koas-w.github.io flash-decode post (paged_decode_attention,
 *        Decode_Paged_GQAAttention_Kernel, _flash_decode_partial_kernel,
 *        _flash_decode_combine_kernel).
 *  [MLA] kernelindex.com "flashinfer gemini-2.5-pro triton xvhq2i"
 *        (mla_paged_prefill_causal_h16_ckv512_kpe64_ps1: run / _forward and
 *        the kernel's sections 2-4).
 *
 * Several query tokens per sequence (speculative / multi-token decode,
 * pkv_decode_desc.q_len > 1) follow [MLA]'s bottom-right causal rule
 * (section "3. Pass 1") on the decode cache layouts: the q_len tokens are the
 * last q_len positions of the context, and token i attends keys up to its
 * own position.
 */
#ifndef PKV_H_
#define PKV_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef struct CUstream_st* pkv_stream_t;  /* same type as cudaStream_t */

/* The library is built with hidden symbol visibility and exports only the
 * functions below (so two copies of it in one process share no state). */
#if defined(__GNUC__)
#define PKV_API __attribute__((visibility("default")))
#else
#define PKV_API
#endif

typedef enum {
    PKV_OK = 0,
    PKV_INVALID_ARG = 1,          /* null pointer, bad shape, misaligned pointer, bad enum */
    PKV_UNSUPPORTED = 2,          /* valid but not compiled: head_dim, block size, layout with FP8 */
    PKV_WORKSPACE_TOO_SMALL = 3,  /* workspace_bytes below the size query's answer */
    PKV_CUDA_ERROR = 4,           /* a CUDA runtime call or a launch failed */
    PKV_BAD_BLOCK_TABLE = 5       /* reported by pkv_validate_block_table only */
} pkv_status;

typedef enum {
    PKV_F16 = 0,
    PKV_BF16 = 1,
    /* OCP FP8 E4M3 ("e4m3fn"), for KV caches only (pkv_decode_desc.kv_dtype):
     * cached value = scale * fp8, with the per-tensor k_scale / v_scale.  [V2]'s
     * launcher carries kv_cache_dtype, k_scale and v_scale but ignores them;
     * this is the plain reading of those arguments. */
    PKV_FP8_E4M3 = 2
} pkv_dtype;

/* pkv_decode_desc.kv_dtype: the caches hold elements of `dtype` (fp16 / bf16). */
#define PKV_KV_AS_Q 0

typedef enum {
    /* k_cache and v_cache both [num_blocks][Hkv][block_size][D] ([FD]
     * Decode_Paged_GQAAttention_Kernel argument list). */
    PKV_LAYOUT_NHD = 0,
    /* vLLM layout ([V2] _partition_attn_kernel argument list):
     * key_cache [num_blocks][Hkv][D/x][block_size][x] with x = 16 bytes / element
     * size (x_pack = 8 for fp16/bf16), value_cache [num_blocks][Hkv][D][block_size]. */
    PKV_LAYOUT_VLLM = 1
} pkv_layout;

/* Problem description of one decode step (q_len query tokens per sequence). */
typedef struct {
    int B;                   /* sequences in the batch */
    int Hq;                  /* query heads; Hq % Hkv == 0, group G = Hq / Hkv */
    int Hkv;                 /* KV heads; query head h reads KV head h / G */
    int D;                   /* head dim: 64, 128 or 256 */
    int block_size;          /* tokens per page: 16 */
    int max_blocks_per_seq;  /* columns of block_table */
    int num_blocks;          /* pages in the pool */
    int max_context_len;     /* host-known upper bound on context_lens[] (plans the grid) */
    long long sum_context_len; /* host-known sum of context_lens[], or an upper bound on it (sizes the grid) */
    int dtype;               /* pkv_dtype of q, caches and out */
    int layout;              /* pkv_layout */
    int x_pack;              /* VLLM layout only: must be 8 */
    int kv_dtype;            /* PKV_KV_AS_Q, or PKV_FP8_E4M3 (NHD layout; q and out stay `dtype`) */
    float k_scale;           /* FP8 caches: K = k_scale * fp8 (finite, > 0); ignored otherwise */
    float v_scale;           /* FP8 caches: V = v_scale * fp8 (finite, > 0); ignored otherwise */
    /* Query tokens per sequence, >= 1 (1 = plain decode).  q and out are
     * [B][q_len][Hq][D]; context_lens[b] = n counts the q_len new tokens, whose
     * K and V are already in the cache.  Query token i sits at position
     * n - q_len + i and attends keys t <= n - q_len + i; where that window is
     * empty (n < q_len - i) its rows are zero. */
    int q_len;
} pkv_decode_desc;

/* pkv_decode_opts.flags bits (see pkv_paged_decode_attention): plan on the
 * device; with it, reuse the plan an earlier call left in the workspace. */
#define PKV_DECODE_DEVICE_PLAN 1
#define PKV_DECODE_PLAN_READY 2

/* Optional knobs; pass NULL for the defaults (all zero). */
typedef struct {
    int partition_tokens;    /* tokens per split, a multiple of block_size; 0 = planner */
    int num_splits;          /* used when partition_tokens == 0: split the longest context this many ways */
    int flags;               /* 0, PKV_DECODE_DEVICE_PLAN, or that | PKV_DECODE_PLAN_READY; other bits are invalid */
    /* Optional cudaEvent_t handles recorded on `stream` right before and right
     * after the phase-1 kernel, so a caller can time that kernel alone inside a
     * full call.  NULL = not recorded. */
    void* phase1_event_start;
    void* phase1_event_stop;
    /* Optional ALiBi slopes, device fp32 [Hq] (4-byte aligned): the score of
     * key position t for a query at position pos (n - 1 for one token per
     * sequence) gains alibi_slopes[h] * (t - pos) before the softmax (ALiBi's
     * linear bias, zero at the query's own position; [V2]'s launcher takes
     * alibi_slopes and ignores them).  NULL = no bias. */
    const float* alibi_slopes;
} pkv_decode_opts;

/* Text of a status code (static storage). */
PKV_API const char* pkv_status_string(int status);

/* ABI version of this header: 9 (8 kept no split table for PKV_DECODE_PLAN_READY; 7 had no pkv_mla_desc.max_kv_len; 6 no pkv_set_stress_delay; 5 no pkv_static_scratch_error and staged
 * MLA keys unpadded; 4 no plan reuse; 3 no device plan; 2 no q_len; 1 no kv_dtype / k_scale / v_scale). */
PKV_API int pkv_version(void);

/*
 * Split planner (host only, deterministic integer arithmetic).  Splits every
 * sequence into partitions of *partition_tokens tokens (a multiple of
 * block_size): split s covers tokens [s*P, min((s+1)*P, n)) ([V2] fixed
 * 512-token partitions; [FD] page-granular splits).  *num_splits =
 * ceil(max_context_len / P) (at least 1) is the grid extent along splits.
 * num_sms <= 0 queries the current device.  The default picks P = 512 tokens
 * per column tile of a CTA and per KV head it holds -- 1024 when a CTA holds
 * 16 query rows, or when an FP8 cache at D = 128 with an even Hkv has at most
 * 4 query rows (G * q_len) per KV head, so that a CTA takes a pair of KV
 * heads; else 512 -- or the longest context, if shorter, halved while the
 * estimated number of (sequence, KV head, row tile, split) work items stays
 * below 6 * num_sms, down to 4 * block_size.  Row tiles: the G * q_len query rows of a
 * (sequence, KV head) pair are covered 16 at a time (8 for D = 256 or for at
 * most 8 rows).
 */
PKV_API int pkv_plan_splits(const pkv_decode_desc* desc, const pkv_decode_opts* opts, int num_sms,
                    int* num_splits, int* partition_tokens);

/*
 * Bytes of scratch memory pkv_paged_decode_attention needs for this problem
 * and these options (256-byte header, then fp32 split partials m, l
 * [B][q_len][Hq][NS] and acc [B][q_len][Hq][NS][D] when the plan has more
 * than one split; with PKV_DECODE_DEVICE_PLAN, NS is the split count of the
 * bounds and a split table of B * NS 16-byte entries follows; each of the
 * four arrays starts on a 256-byte boundary).
 * num_sms as for pkv_plan_splits.  The workspace must be 256-byte aligned.
 * Word 0 of the header collects device-side error bits (bit 0: a pipeline
 * wait timed out; bit 1: a call with PKV_DECODE_PLAN_READY found no valid
 * plan of its problem in the workspace, and rows it could not place are
 * unspecified); zero it once after allocating.
 */
PKV_API int pkv_decode_workspace_size(const pkv_decode_desc* desc, const pkv_decode_opts* opts, int num_sms,
                              size_t* bytes);

/*
 * Paged GQA decode attention ([FD] paged_decode_attention; [V2]
 * paged_attention_v2_triton):
 *   out[b][i][h][:] = sum_t softmax_t(scale * q[b][i][h] . K_t) V_t,
 *   t < context_lens[b] - q_len + i + 1   (t < context_lens[b] for q_len = 1),
 * with K_t, V_t the slot t % block_size of page block_table[b][t / block_size]
 * of KV head h / G.  An empty window (context_lens[b] == 0 for q_len = 1)
 * gives a zero row.  K and V inside the context must be finite: with
 * q_len > 1 a masked key's V row still meets a zero weight.
 *   q, out        [B][q_len][Hq][D] of dtype (4-byte aligned; out 8-byte aligned)
 *   k/v_cache     per layout (16-byte aligned); may be NULL when num_blocks == 0
 *   block_table   int32 [B][max_blocks_per_seq] (may be NULL when max_blocks_per_seq
 *                 == 0); entries past a sequence's last
 *                 page are never used (-1 is the customary filler).  A live entry
 *                 outside [0, num_blocks) is a caller error: it is clamped to a
 *                 valid page (no out-of-bounds access, result unspecified);
 *                 pkv_validate_block_table reports it.
 *   context_lens  int32 [B]; values are clamped to
 *                 [0, min(max_context_len, max_blocks_per_seq * block_size)].
 * Phase 1 runs one CTA per (sequence, KV head, row tile, split) of the
 * pkv_plan_splits plan, loading each page once for all the query rows of a
 * row tile (the whole group when G * q_len <= 16, or <= 8 for D = 256); sequences with more than
 * one split are merged by a log-sum-exp combine kernel launched as a
 * programmatic dependent of phase 1.  Calls sharing one workspace must be
 * ordered on the GPU (one stream).
 *
 * flags & PKV_DECODE_DEVICE_PLAN: the split plan is made on the device from
 * context_lens: every CTA of phase 1 applies the planner rule of
 * pkv_plan_splits to the actual longest and total context (with the
 * partition raised where needed so that the splits fit the bounds' split
 * count) and finds its own non-empty work items; max_context_len and
 * sum_context_len are then only capacity bounds that size the workspace.
 * Phase 1 runs a fixed grid of min(bound items, 24 per SM) CTAs that take
 * the items in order, so a call captured into a CUDA graph with loose bounds
 * launches no CTA per empty split, and no planning kernel runs before it.
 * pkv_decode_partials does not take this flag.
 *
 * A device-planned call also leaves its plan in the workspace: the partition,
 * the split count and a table with the sequence, split and context length of
 * every split of the plan.
 *
 * flags & PKV_DECODE_PLAN_READY (with PKV_DECODE_DEVICE_PLAN): states that the
 * last device-planned call on this workspace had the same desc, partition
 * options and context_lens values and completed without error bits (the
 * layers of one decode step), and that no other call used the workspace
 * since.  Phase 1 then takes its items from that plan instead of planning;
 * the workspace keeps it for further such calls.  Every value read from the
 * workspace is checked against the bounds first: if the statement is false,
 * the result is unspecified and error bit 1 may be set, but no memory
 * outside the arguments is accessed.
 */
PKV_API int pkv_paged_decode_attention(const pkv_decode_desc* desc, const pkv_decode_opts* opts,
                               const void* q, const void* k_cache, const void* v_cache,
                               const int32_t* block_table, const int32_t* context_lens,
                               float scale, void* out,
                               void* workspace, size_t workspace_bytes, pkv_stream_t stream);

/*
 * Phase 1 alone, for layered testing ([FD] _flash_decode_partial_kernel):
 * writes, for every sequence b, query token i, query head h and split
 * s < *num_splits_out, the unnormalised fp32 partial of the tokens of split s
 * inside query i's causal window, in natural-log units:
 *   part_m[b][i][h][s] = max_t s_t,  part_l[b][i][h][s] = sum_t exp(s_t - m),
 *   part_acc[b][i][h][s][:] = sum_t exp(s_t - m) V_t,
 * and the sentinel (-inf, 0, 0) where that range is empty.  The arrays are
 * [B][q_len][Hq][num_splits_capacity] (and [...][D]); the call fails with
 * PKV_WORKSPACE_TOO_SMALL if the plan needs more splits than the capacity.
 */
PKV_API int pkv_decode_partials(const pkv_decode_desc* desc, const pkv_decode_opts* opts,
                        const void* q, const void* k_cache, const void* v_cache,
                        const int32_t* block_table, const int32_t* context_lens, float scale,
                        float* part_acc, float* part_m, float* part_l, int num_splits_capacity,
                        int* partition_tokens_out, int* num_splits_out, pkv_stream_t stream);

/*
 * Phase 2 alone ([FD] _flash_decode_combine_kernel; [V2]
 * _reduce_partitions_kernel): for every (b, i, h) with n = context_lens[b]
 * (clamped as above), NS_b = ceil(n / partition_tokens) splits are merged:
 *   M = max_s m_s,  out = sum_s e^{m_s - M} acc_s / sum_s e^{m_s - M} l_s,
 * and an empty causal window (n == 0 for q_len = 1) gives zeros.  Partials
 * are laid out as pkv_decode_partials writes them with num_splits columns.
 */
PKV_API int pkv_combine(const pkv_decode_desc* desc, int partition_tokens, int num_splits,
                const int32_t* context_lens, const float* part_acc, const float* part_m,
                const float* part_l, void* out, pkv_stream_t stream);

/*
 * Optional device-side validator of the paged indexing (never traps).  ORs
 * into *err_word (device, 4 bytes, caller-zeroed):
 *   bit 0  some context_lens[b] < 0, > max_context_len or > max_blocks_per_seq * block_size
 *   bit 1  some live block_table entry (block index < ceil(n / block_size)) is
 *          outside [0, num_blocks)
 * Entries past a sequence's live range are not inspected.
 */
PKV_API int pkv_validate_block_table(const pkv_decode_desc* desc, const int32_t* block_table,
                             const int32_t* context_lens, uint32_t* err_word, pkv_stream_t stream);

/* Problem description of one MLA paged prefill call (page size 1, bf16). */
typedef struct {
    int total_q;    /* query tokens over the batch: rows of q_nope, q_pe, out, lse */
    int num_heads;  /* query heads: 16 */
    int d_ckv;      /* latent (ckv) width, also the output width: 512 */
    int d_kpe;      /* rope (kpe) width: 64 */
    int batch;      /* sequences; qo_indptr and kv_indptr hold batch + 1 entries */
    int num_pages;  /* rows of ckv_cache and kpe_cache */
    int nnz;        /* kv_indptr[batch] (entries of kv_indices), or an upper bound of it */
    int max_kv_len; /* an upper bound of every sequence's kv_len, or 0 (none given).  With a
                     * bound, S = Q.K^T is computed once per 16-token row tile: the tasks of the
                     * first 256 output columns export each key block's softmax weights P
                     * (bf16) and rescale factors, and a second kernel computes the other 256
                     * columns from them (bit-identical to computing S again); the workspace
                     * grows accordingly (pkv_mla_workspace_size).  Without one, each half of
                     * the output columns computes S itself. */
} pkv_mla_desc;

/*
 * Bytes of scratch memory pkv_mla_paged_prefill needs: a 256-byte header;
 * the work list of 16-byte entries, one per (16-token row tile, half of the
 * output columns), 2 * (ceil(total_q / 16) + batch) of them; two ints per
 * sequence (plus one); then nnz + 128 * batch staged key rows of 1152 bytes
 * (ckv 512 + kpe 64 bf16; every sequence's keys start on a multiple of 128
 * rows, the rows in between are zero; no rows when nnz == 0); each part
 * rounded up to 256 bytes.  With max_kv_len > 0, also, for up to
 * E = (ceil(total_q / 16) + batch) * ceil(max_kv_len / 128) exported key
 * blocks, 66,576 bytes each (P 65,536, rescale factors 1,024, flags 16), and
 * 1 KB of row sums plus 4 bytes per row tile.  The workspace must be 256-byte
 * aligned.  Word 0 of the header collects device-side error bits (bit 0: a
 * pipeline wait timed out; bit 1: kv_indptr[batch] > nnz, so keys past nnz
 * were not staged and the result is unspecified; bit 2: some kv_len exceeds
 * max_kv_len, the export did not fit and the second half of the output
 * columns is unspecified); zero it once after allocating.
 */
PKV_API int pkv_mla_workspace_size(const pkv_mla_desc* desc, size_t* bytes);

/*
 * MLA paged causal prefill ([MLA] run / _forward and the kernel's sections
 * 2-4).  For sequence b (query tokens qo_indptr[b] .. qo_indptr[b+1]-1, cached
 * rows kv_indices[kv_indptr[b] .. kv_indptr[b+1]-1], prefix = kv_len - q_len)
 * and query token i of it, head h:
 *   logit_j = sm_scale * (q_nope[t][h] . ckv[page_j] + q_pe[t][h] . kpe[page_j])
 *   for the visible keys j <= prefix + i (bottom-right causal),
 *   out[t][h][:] = sum_j softmax(logit)_j ckv[page_j][:],
 *   lse[t][h]    = log2 sum_j exp(logit_j)            (base 2).
 * A sequence with kv_len == 0 gives out = 0 and lse = -inf.
 *   q_nope   bf16 [total_q][16][512]     q_pe       bf16 [total_q][16][64]
 *   ckv_cache bf16 [num_pages][1][512]   kpe_cache  bf16 [num_pages][1][64]
 *   qo_indptr, kv_indptr int32 [batch+1] (starting at 0), kv_indices int32 [nnz]
 *   out      bf16 [total_q][16][512]     lse        fp32 [total_q][16]
 * Tensors 16-byte aligned (lse 4-byte).  kv_len < q_len is a caller error
 * (rows with no visible key get out = 0, lse = -inf); page ids outside
 * [0, num_pages) are clamped to page 0 (no out-of-bounds access, result
 * unspecified).  A sequence's own cached rows must be finite: a row one of
 * its queries does not see still enters the tensor-core products with weight
 * 0.  No other sequence's rows enter them ([MLA] loads a sequence's keys
 * only, section "3. Pass 1"): a non-finite row in one sequence leaves the
 * other sequences' outputs unchanged.
 * The q -> sequence map of [MLA]'s host loop is computed on the device from
 * qo_indptr.
 * Two kernels run: the first copies every referenced key row, sequence by
 * sequence, into the workspace (one gather per call instead of one per query
 * tile) and lists the work, longest row tiles first; the second, launched as
 * its programmatic dependent, runs one pair of CTAs per two SMs that take the
 * listed tiles in turns and stream the staged rows with tensor-memory-access
 * boxes.  workspace / workspace_bytes as pkv_mla_workspace_size describes;
 * calls sharing one workspace must be ordered on the GPU (one stream).
 */
PKV_API int pkv_mla_paged_prefill(const pkv_mla_desc* desc, const void* q_nope, const void* q_pe,
                          const void* ckv_cache, const void* kpe_cache, const int32_t* qo_indptr,
                          const int32_t* kv_indptr, const int32_t* kv_indices, float sm_scale,
                          void* out, float* lse, void* workspace, size_t workspace_bytes,
                          pkv_stream_t stream);

/*
 * pkv_paged_decode_attention_static -- the same decode step as
 * pkv_paged_decode_attention, for callers that cannot allocate device memory.
 * The pages have no counterpart of this entry point.
 *
 * Who needs it: code that runs where allocating is not allowed or not safe --
 * a plugin whose enqueue hook is handed a stream but no allocator, an engine
 * that carves all device memory out of a fixed pool at start-up, or a
 * latency-critical loop where cudaMalloc could synchronise the device.
 *
 * The step's scratch (error word, split partials and, with the device plan,
 * the plan's header words and split table) lives in one
 * file-scope device array of PKV_STATIC_SCRATCH_BYTES (32 MiB), which
 * every GPU that loads libpkv reserves until the process exits.  This call
 * allocates nothing: no cudaMalloc, cudaFree or allocating library routine.
 * Once every argument has passed the regular entry point's checks, it clears
 * the array's 4-byte error word (word 0 of the header) with cudaMemsetAsync
 * on `stream` and runs the regular entry point on the array; the rest of the
 * array (a device plan's header words and split table included) keeps the
 * previous call's contents.  pkv_static_scratch_error reads the error word.
 *  - A problem whose workspace (pkv_decode_workspace_size) exceeds the array
 *    is refused with PKV_WORKSPACE_TOO_SMALL before anything is launched.
 *  - PKV_DECODE_PLAN_READY is refused (PKV_INVALID_ARG) unless the previous
 *    successful call of this entry point on the device was device-planned
 *    (PKV_DECODE_DEVICE_PLAN) with the same desc and partition options, as
 *    the flag states.
 *  - The first call on a device looks up the array's device address (with
 *    that device current); make that first call before any stream capture.
 *  - Every call on a device shares the one array and it keeps the last call's
 *    contents: calls whose work overlaps on the GPU (different streams, no
 *    ordering between them) race on it and produce garbage.  Order them on
 *    one stream, or use the workspace entry point.
 * Arguments, layouts and errors are otherwise those of
 * pkv_paged_decode_attention.
 */
#define PKV_STATIC_SCRATCH_BYTES ((size_t)32 << 20)
PKV_API int pkv_paged_decode_attention_static(const pkv_decode_desc* desc, const pkv_decode_opts* opts,
                                      const void* q, const void* k_cache, const void* v_cache,
                                      const int32_t* block_table, const int32_t* context_lens,
                                      float scale, void* out, pkv_stream_t stream);

/*
 * Copies the static array's error word (the device-side error bits of the
 * last pkv_paged_decode_attention_static call on the current device; bit 0:
 * a pipeline wait timed out and the output is unspecified) into *dst, with
 * cudaMemcpyAsync on `stream`, ordered after the work already on it.  dst is
 * 4 bytes of device or host memory (pinned host memory keeps the copy
 * asynchronous).  Allocates nothing.
 */
PKV_API int pkv_static_scratch_error(uint32_t* dst, pkv_stream_t stream);

/*
 * Timing perturbation for race testing.  From the next call on, in every
 * kernel launched by this library, the copy producers -- decode phase 1's page
 * loads, the MLA prefill's Q and key loads -- pause producer_delay_ns
 * nanoseconds after each copy they issue, and the consumers -- decode phase
 * 1's consumer warps after each page, the MLA prefill's MMA thread after each
 * ring slot and its softmax warps after each key block -- pause
 * consumer_delay_ns (0, the default, turns either off).  The results must not
 * change: the kernels order every role after what it reads by barriers, never
 * by timing, and a parity test run under a delay checks that (a parity wait on
 * a barrier two phases behind the expected one passes at once; a slow role is
 * what shows such a wait).  Calls become slower; nothing else changes.
 * Process-wide and thread-safe; calls already enqueued keep the values they
 * were launched with.
 * Returns PKV_OK, or PKV_INVALID_ARG if either delay is above 1,000,000 ns.
 */
PKV_API int pkv_set_stress_delay(uint32_t producer_delay_ns, uint32_t consumer_delay_ns);

#ifdef __cplusplus
}
#endif

#endif /* PKV_H_ */
