// api.cu -- the C ABI of libpkv (declared in include/pkv.h): argument
// validation, the split planner, TMA descriptor set-up and kernel dispatch.
// Host code only; nothing here touches device memory directly.
#include <algorithm>
#include <atomic>
#include <climits>
#include <cmath>
#include <cudaTypedefs.h>
#include <cstring>
#include <mutex>

#include "internal.h"
#include "pkv.h"
#include "trace.h"

using namespace pkv;

namespace {

constexpr int kBS = 16;          // compiled page size
constexpr int kHeaderBytes = 256;

// pkv_set_stress_delay: producer / consumer pauses, read by every launch.
std::atomic<uint32_t> g_stress_ns{0}, g_stress_consumer_ns{0};

long long ceil_div(long long a, long long b) { return (a + b - 1) / b; }
long long round_up(long long a, long long b) { return ceil_div(a, b) * b; }
size_t align256(size_t x) { return (x + 255) & ~size_t(255); }
bool aligned(const void* p, size_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }

int check_desc(const pkv_decode_desc* d) {
    if (!d) return PKV_INVALID_ARG;
    if (d->B < 0 || d->Hq <= 0 || d->Hkv <= 0 || d->D <= 0 || d->block_size <= 0 || d->max_blocks_per_seq < 0 ||
        d->num_blocks < 0 || d->max_context_len < 0 || d->sum_context_len < 0 || d->q_len <= 0)
        return PKV_INVALID_ARG;
    if (d->Hq % d->Hkv != 0) return PKV_INVALID_ARG;
    if (d->dtype != PKV_F16 && d->dtype != PKV_BF16) return PKV_INVALID_ARG;
    if (d->layout != PKV_LAYOUT_NHD && d->layout != PKV_LAYOUT_VLLM) return PKV_INVALID_ARG;
    if (d->layout == PKV_LAYOUT_VLLM && d->x_pack != 8) return PKV_INVALID_ARG;
    if (d->kv_dtype != PKV_KV_AS_Q && d->kv_dtype != PKV_FP8_E4M3) return PKV_INVALID_ARG;
    if (d->kv_dtype == PKV_FP8_E4M3) {
        if (!(std::isfinite(d->k_scale) && d->k_scale > 0.f && std::isfinite(d->v_scale) && d->v_scale > 0.f))
            return PKV_INVALID_ARG;
        if (d->layout != PKV_LAYOUT_NHD) return PKV_UNSUPPORTED;
    }
    if ((long long)d->max_context_len > (long long)d->max_blocks_per_seq * d->block_size) return PKV_INVALID_ARG;
    if (d->max_context_len > 0 && d->num_blocks == 0) return PKV_INVALID_ARG;
    if (d->D != 64 && d->D != 128 && d->D != 256) return PKV_UNSUPPORTED;
    if (d->block_size != kBS) return PKV_UNSUPPORTED;
    if ((long long)d->num_blocks * d->Hkv > INT_MAX) return PKV_UNSUPPORTED;
    if ((long long)d->q_len * d->Hq > INT_MAX || (long long)d->B * d->q_len * d->Hq > INT_MAX)
        return PKV_UNSUPPORTED;
    return PKV_OK;
}

// Query-column tiling of phase 1: a (sequence, KV head) pair has R = G * q_len
// query rows; a CTA holds 8 * nt of them as mma columns (nt = 2 when more than
// 8 rows and D <= 128, else 1: D = 256 keeps its accumulators to one tile) and
// rt = ceil(R / (8 * nt)) CTAs cover them.
struct ColumnTiles {
    int nt, rt, R;
};
ColumnTiles column_tiles(const pkv_decode_desc* d) {
    const long long R = (long long)(d->Hq / d->Hkv) * d->q_len;   // <= q_len * Hq <= INT_MAX
    const int nt = (R > 8 && d->D <= 128) ? 2 : 1;
    return ColumnTiles{nt, (int)ceil_div(R, 8LL * nt), (int)R};
}

int current_sm_count(int* out) {
    return current_device_sm_count(out) == cudaSuccess ? PKV_OK : PKV_CUDA_ERROR;
}

// FP8 caches at D = 128 whose query rows per KV head (G * q_len) fill at most
// half a column tile run one CTA per pair of adjacent KV heads: both heads'
// page slices are contiguous, so each ring stage moves 4 KB boxes instead of
// 2 KB ones, with the same tensor-core work per byte.
bool head_pairs(const pkv_decode_desc* d) {
    return d->kv_dtype == PKV_FP8_E4M3 && d->D == 128 && d->Hkv % 2 == 0 &&
           2LL * (d->Hq / d->Hkv) * d->q_len <= 8;
}

// Base partition: 512 tokens per column tile of the CTA and per KV head it
// holds (512, or 1024 for two column tiles or a pair of KV heads: a CTA's
// fixed costs -- loading Q, merging its warps' columns, writing the partials
// -- grow with its columns, and fewer splits shorten the combine).
long long base_partition(const pkv_decode_desc* d) {
    return 512LL * column_tiles(d).nt * (head_pairs(d) ? 2 : 1);
}

// Default partition: the base partition, or the longest context rounded up to
// a page, if shorter; halved while the estimated number of non-empty work
// items Hkv * row_tiles * ceil(sum_n / P) stays below six per SM, down to
// four pages.  The device plan applies the same rule to the actual lengths.
long long auto_partition(const pkv_decode_desc* d, int num_sms) {
    const long long BS = d->block_size;
    const long long maxn = d->max_context_len > 0 ? d->max_context_len : 1;
    const long long P0 = base_partition(d);
    long long P = round_up(maxn < P0 ? maxn : P0, BS);
    const long long min_p = 4 * BS;
    const long long target = 6LL * num_sms;
    const long long sum = d->sum_context_len > 0 ? d->sum_context_len : 1;
    while (P > min_p) {
        const long long units = (long long)d->Hkv * column_tiles(d).rt * ceil_div(sum, P);
        if (units >= target) break;
        long long np = round_up(P / 2, BS);
        if (np < min_p) np = min_p;
        if (np >= P) break;
        P = np;
    }
    return P;
}

int plan(const pkv_decode_desc* d, const pkv_decode_opts* o, int num_sms, int* ns, int* P) {
    int st = check_desc(d);
    if (st) return st;
    if (o && (o->flags & ~(PKV_DECODE_DEVICE_PLAN | PKV_DECODE_PLAN_READY)) != 0) return PKV_INVALID_ARG;
    if (o && (o->flags & PKV_DECODE_PLAN_READY) && !(o->flags & PKV_DECODE_DEVICE_PLAN)) return PKV_INVALID_ARG;
    if (num_sms <= 0) {
        st = current_sm_count(&num_sms);
        if (st) return st;
    }
    long long p;
    if (o && o->partition_tokens > 0) {
        p = o->partition_tokens;
        if (p % d->block_size != 0) return PKV_INVALID_ARG;
    } else if (o && o->num_splits > 0) {
        const long long maxn = d->max_context_len > 0 ? d->max_context_len : 1;
        p = round_up(ceil_div(maxn, o->num_splits), d->block_size);
    } else if (o && (o->partition_tokens < 0 || o->num_splits < 0)) {
        return PKV_INVALID_ARG;
    } else {
        p = auto_partition(d, num_sms);
    }
    long long n_splits = ceil_div(d->max_context_len, p);
    if (n_splits < 1) n_splits = 1;
    if (p > INT_MAX || n_splits > INT_MAX || (long long)d->B * d->Hkv * column_tiles(d).rt * n_splits > INT_MAX)
        return PKV_UNSUPPORTED;
    *P = (int)p;
    *ns = (int)n_splits;
    return PKV_OK;
}

size_t partial_bytes(const pkv_decode_desc* d, int ns) {
    const size_t rows = (size_t)d->B * d->q_len * d->Hq * ns;
    return 2 * align256(rows * 4) + align256(rows * d->D * 4);
}

bool device_plan(const pkv_decode_opts* o) { return o && (o->flags & PKV_DECODE_DEVICE_PLAN); }

// Work items of the bounds' plan: (sequence, KV head, row tile, split) slots.
long long plan_items(const pkv_decode_desc* d, int ns) {
    return (long long)d->B * d->Hkv * column_tiles(d).rt * ns;
}

// The device plan's split table: a 16-byte entry per (sequence, split) of the bounds.
size_t plan_table_bytes(const pkv_decode_desc* d, int ns) { return align256((size_t)d->B * ns * 16); }

// Workspace: 256-byte header | split partials (more than one split) | the
// device plan's split table (with PKV_DECODE_DEVICE_PLAN).
size_t required_workspace(const pkv_decode_desc* d, const pkv_decode_opts* o, int ns) {
    return kHeaderBytes + (ns > 1 ? partial_bytes(d, ns) : 0) + (device_plan(o) ? plan_table_bytes(d, ns) : 0);
}

// Header words of the device plan: {P, splits of the longest context, splits
// of the plan (the table's entries)}.
constexpr int kSchedHeaderWord = 4;
// Phase-1 CTAs of the device plan: enough to fill the GPU many times over;
// more items than this are taken in turns.
constexpr int kDevicePlanCtasPerSm = 24;

// cuTensorMapEncodeTiled through the runtime's driver entry point (no -lcuda).
PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
    static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
    static std::once_flag once;
    std::call_once(once, [] {
        void* p = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) ==
                cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
    });
    return fn;
}

// Page slice of one KV head as a 3-D tensor {inner, rows, num_blocks * Hkv}.
//   NHD : {D, BS, NB*Hkv}, box {64, BS, 1}, 128-byte swizzle.
//   VLLM: the contiguous D*BS-element slice viewed as {256, D*BS/256, NB*Hkv},
//         box {256, D*BS/256, 1}, no swizzle.
int encode_cache_map(CUtensorMap* map, const void* base, const pkv_decode_desc* d, int heads) {
    auto fn = encode_fn();
    if (!fn) return PKV_CUDA_ERROR;
    const cuuint64_t slices = (cuuint64_t)d->num_blocks * d->Hkv;
    cuuint64_t dims[3], strides[2];
    cuuint32_t box[3], estr[3] = {1, 1, 1};
    CUtensorMapSwizzle swz;
    CUtensorMapDataType type = CU_TENSOR_MAP_DATA_TYPE_UINT16;
    if (d->kv_dtype == PKV_FP8_E4M3) {
        // {D, BS, NB*Hkv} bytes, one {D, BS} box per page slice (per two
        // adjacent slices, {D, BS, 2}, for head pairs)
        type = CU_TENSOR_MAP_DATA_TYPE_UINT8;
        dims[0] = d->D;
        dims[1] = d->block_size;
        dims[2] = slices;
        strides[0] = (cuuint64_t)d->D;
        strides[1] = (cuuint64_t)d->D * d->block_size;
        // D >= 128: 128-byte-wide boxes with 128-byte swizzle (read straight into mma
        // fragments); D = 64: one unswizzled {64, BS} box (expanded in shared memory)
        box[0] = d->D >= 128 ? 128 : d->D;
        box[1] = d->block_size;
        box[2] = (cuuint32_t)heads;
        swz = d->D >= 128 ? CU_TENSOR_MAP_SWIZZLE_128B : CU_TENSOR_MAP_SWIZZLE_NONE;
    } else if (d->layout == PKV_LAYOUT_NHD) {
        dims[0] = d->D;
        dims[1] = d->block_size;
        dims[2] = slices;
        strides[0] = (cuuint64_t)d->D * 2;
        strides[1] = (cuuint64_t)d->D * d->block_size * 2;
        box[0] = 64;
        box[1] = d->block_size;
        box[2] = 1;
        swz = CU_TENSOR_MAP_SWIZZLE_128B;
    } else {
        const cuuint64_t e = (cuuint64_t)d->D * d->block_size;
        dims[0] = 256;
        dims[1] = e / 256;
        dims[2] = slices;
        strides[0] = 512;
        strides[1] = e * 2;
        box[0] = 256;
        box[1] = (cuuint32_t)(e / 256);
        box[2] = 1;
        swz = CU_TENSOR_MAP_SWIZZLE_NONE;
    }
    CUresult r = fn(map, type, 3, const_cast<void*>(base), dims, strides, box, estr,
                    CU_TENSOR_MAP_INTERLEAVE_NONE, swz, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                    CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS ? PKV_OK : PKV_INVALID_ARG;
}

// Row-major 2-D bf16 tensor {cols, rows} with a {box_cols, box_rows} box and
// 128-byte swizzle (box_cols * 2 <= 128), or none (the box copied as it is).
int encode_rows_map(CUtensorMap* map, const void* base, cuuint64_t cols, cuuint64_t rows, cuuint32_t box_cols,
                    cuuint32_t box_rows, bool swizzle = true) {
    auto fn = encode_fn();
    if (!fn) return PKV_CUDA_ERROR;
    cuuint64_t dims[2] = {cols, rows}, strides[1] = {cols * 2};
    cuuint32_t box[2] = {box_cols, box_rows}, estr[2] = {1, 1};
    CUresult r = fn(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(base), dims, strides, box, estr,
                    CU_TENSOR_MAP_INTERLEAVE_NONE, swizzle ? CU_TENSOR_MAP_SWIZZLE_128B : CU_TENSOR_MAP_SWIZZLE_NONE,
                    CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                    CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS ? PKV_OK : PKV_INVALID_ARG;
}

// Launches phase 1 over the grid (sequence, KV head, row tile, split), or
// over `grid` CTAs that take the device plan's listed items.
cudaError_t dispatch_phase1(const pkv_decode_desc* d, const DecodeParams& p, const CUtensorMap& k,
                            const CUtensorMap& v, cudaStream_t s, long long grid = 0) {
    const int nt = column_tiles(d).nt;
    if (grid <= 0) grid = (long long)p.B * p.Hkv * p.RT * p.NS;
    const bool bf = d->dtype == PKV_BF16;
    if (d->kv_dtype == PKV_FP8_E4M3)
        return bf ? launch_decode_nhd8_bf16(d->D, nt, p, grid, k, v, s)
                  : launch_decode_nhd8_f16(d->D, nt, p, grid, k, v, s);
    if (d->layout == PKV_LAYOUT_NHD)
        return bf ? launch_decode_nhd_bf16(d->D, nt, p, grid, k, v, s)
                  : launch_decode_nhd_f16(d->D, nt, p, grid, k, v, s);
    return bf ? launch_decode_vllm_bf16(d->D, nt, p, grid, k, v, s)
              : launch_decode_vllm_f16(d->D, nt, p, grid, k, v, s);
}

// An empty pool (num_blocks == 0, so every context is empty) may come with null
// caches, and a table without columns with a null table: neither is ever read.
int check_tensors(const pkv_decode_desc* d, const void* q, const void* k, const void* v, const int32_t* table,
                  const int32_t* ctx) {
    if (!q || !ctx) return PKV_INVALID_ARG;
    if ((!k || !v) && d->num_blocks > 0) return PKV_INVALID_ARG;
    if (!table && d->max_blocks_per_seq > 0) return PKV_INVALID_ARG;
    if (!aligned(q, 4) || !aligned(k, 16) || !aligned(v, 16) || !aligned(table, 4) || !aligned(ctx, 4))
        return PKV_INVALID_ARG;
    return PKV_OK;
}

// Common set-up of phase 1: parameters and the two tensor maps (pairs: one
// CTA per pair of KV heads, see head_pairs).
int prepare_phase1(const pkv_decode_desc* d, int P, int NS, const void* q, const void* k, const void* v,
                   const int32_t* table, const int32_t* ctx, float scale, bool pairs, DecodeParams* p,
                   CUtensorMap* mk, CUtensorMap* mv) {
    *p = DecodeParams{};
    p->q = q;
    p->table = table;
    p->ctx = ctx;
    p->B = d->B;
    p->Hq = d->Hq;
    p->Hkv = d->Hkv;
    p->G = d->Hq / d->Hkv;
    const ColumnTiles ct = column_tiles(d);
    p->q_len = d->q_len;
    p->R = ct.R;
    p->RT = ct.rt;
    p->Hc = p->Hkv;
    p->Gc = p->G;
    if (pairs) {
        p->Hkv = d->Hkv / 2;
        p->G = 2 * p->Gc;
        p->R = p->G * d->q_len;   // <= 8: one column tile
        p->RT = 1;
    }
    p->MBPS = d->max_blocks_per_seq;
    p->NB = d->num_blocks;
    p->P = P;
    p->NS = NS;
    p->ns_stride = NS;
    p->n_cap = d->max_context_len;
    const bool fp8 = d->kv_dtype == PKV_FP8_E4M3;
    p->scale_log2 = (float)((double)scale * (fp8 ? (double)d->k_scale : 1.0) * 1.4426950408889634);
    p->stress_ns = g_stress_ns.load(std::memory_order_relaxed);
    p->stress_consumer_ns = g_stress_consumer_ns.load(std::memory_order_relaxed);
    p->v_scale = fp8 ? d->v_scale : 1.f;
    if (d->max_context_len == 0) return PKV_OK;   // maps unused: every split is empty
    int st = encode_cache_map(mk, k, d, pairs ? 2 : 1);
    if (st) return st;
    return encode_cache_map(mv, v, d, pairs ? 2 : 1);
}

void record(void* ev, cudaStream_t s) {
    if (ev) cudaEventRecord(reinterpret_cast<cudaEvent_t>(ev), s);
}

}  // namespace

extern "C" {

const char* pkv_status_string(int status) {
    switch (status) {
        case PKV_OK: return "ok";
        case PKV_INVALID_ARG: return "invalid argument";
        case PKV_UNSUPPORTED: return "unsupported configuration";
        case PKV_WORKSPACE_TOO_SMALL: return "workspace too small";
        case PKV_CUDA_ERROR: return "CUDA error";
        case PKV_BAD_BLOCK_TABLE: return "bad block table";
        default: return "unknown status";
    }
}

int pkv_version(void) { return 9; }

int pkv_set_stress_delay(uint32_t producer_delay_ns, uint32_t consumer_delay_ns) {
    if (producer_delay_ns > 1000000u || consumer_delay_ns > 1000000u) return PKV_INVALID_ARG;
    g_stress_ns.store(producer_delay_ns, std::memory_order_relaxed);
    g_stress_consumer_ns.store(consumer_delay_ns, std::memory_order_relaxed);
    return PKV_OK;
}

int pkv_plan_splits(const pkv_decode_desc* desc, const pkv_decode_opts* opts, int num_sms, int* num_splits,
                    int* partition_tokens) {
    if (!num_splits || !partition_tokens) return PKV_INVALID_ARG;
    return plan(desc, opts, num_sms, num_splits, partition_tokens);
}

int pkv_decode_workspace_size(const pkv_decode_desc* desc, const pkv_decode_opts* opts, int num_sms, size_t* bytes) {
    if (!bytes) return PKV_INVALID_ARG;
    int ns = 0, P = 0;
    int st = plan(desc, opts, num_sms, &ns, &P);
    if (st) return st;
    *bytes = required_workspace(desc, opts, ns);
    return PKV_OK;
}

int pkv_paged_decode_attention(const pkv_decode_desc* desc, const pkv_decode_opts* opts, const void* q,
                               const void* k_cache, const void* v_cache, const int32_t* block_table,
                               const int32_t* context_lens, float scale, void* out, void* workspace,
                               size_t workspace_bytes, pkv_stream_t stream) {
    return pkv::paged_decode_impl(desc, opts, q, k_cache, v_cache, block_table, context_lens, scale, out, workspace,
                                  workspace_bytes, stream, false);
}

}  // extern "C"

// The decode step behind both decode entry points.  Every argument is checked
// before anything is enqueued; with clear_err_word the workspace's error word
// is then zeroed on `stream` ahead of the kernels.
int pkv::paged_decode_impl(const pkv_decode_desc* desc, const pkv_decode_opts* opts, const void* q,
                           const void* k_cache, const void* v_cache, const int32_t* block_table,
                           const int32_t* context_lens, float scale, void* out, void* workspace,
                           size_t workspace_bytes, pkv_stream_t stream, bool clear_err_word) {
    int st = check_desc(desc);
    if (st) return st;
    if (desc->B == 0) return PKV_OK;
    st = check_tensors(desc, q, k_cache, v_cache, block_table, context_lens);
    if (st) return st;
    if (!out || !aligned(out, 8) || !workspace || !aligned(workspace, 256) || !std::isfinite(scale))
        return PKV_INVALID_ARG;
    if (opts && opts->alibi_slopes && !aligned(opts->alibi_slopes, 4)) return PKV_INVALID_ARG;
    int ns = 0, P = 0;
    st = plan(desc, opts, 0, &ns, &P);
    if (st) return st;
    if (workspace_bytes < required_workspace(desc, opts, ns)) return PKV_WORKSPACE_TOO_SMALL;

    DecodeParams p;
    CUtensorMap mk{}, mv{};
    st = prepare_phase1(desc, P, ns, q, k_cache, v_cache, block_table, context_lens, scale, head_pairs(desc), &p,
                        &mk, &mv);
    if (st) return st;
    if (opts) p.alibi = opts->alibi_slopes;
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    uint8_t* ws = static_cast<uint8_t*>(workspace);
    if (clear_err_word && cudaMemsetAsync(ws, 0, sizeof(uint32_t), s) != cudaSuccess) return PKV_CUDA_ERROR;
    p.out = out;
    p.err = reinterpret_cast<uint32_t*>(ws);
    uint8_t* parts = ws + kHeaderBytes;
    const size_t rows = (size_t)desc->B * desc->q_len * desc->Hq * ns;
    p.part_m = reinterpret_cast<float*>(parts);
    p.part_l = reinterpret_cast<float*>(parts + align256(rows * 4));
    p.part_acc = reinterpret_cast<float*>(parts + 2 * align256(rows * 4));

    if (desc->max_context_len == 0) {
        // Every context is empty: the combine kernel writes the zero rows.
        CombineParams c{context_lens, nullptr, nullptr, nullptr, out, desc->B, desc->Hq, P, ns, 0, 0, desc->q_len,
                        nullptr};
        TraceRange r("pkv::decode.combine");
        return launch_combine(desc->dtype, desc->D, c, s, false) == cudaSuccess ? PKV_OK : PKV_CUDA_ERROR;
    }
    long long grid = 0;
    if (device_plan(opts)) {
        // Phase 1 plans from the device's context lengths (every CTA of a fixed
        // grid, device_plan.cuh) and takes the non-empty items in turns.
        if (desc->Hkv > 0xFFFF || column_tiles(desc).rt > 0x7FFF) return PKV_UNSUPPORTED;
        int sms = 0;
        st = current_sm_count(&sms);
        if (st) return st;
        const ColumnTiles ct = column_tiles(desc);
        // The rule counts the description's KV heads, as the host planner does;
        // items are per grid KV head (a pair under head pairs).
        p.plan_hdr = reinterpret_cast<int*>(ws) + kSchedHeaderWord;
        p.plan_tab = reinterpret_cast<int4*>(parts + (ns > 1 ? partial_bytes(desc, ns) : 0));
        p.plan_ready = (opts->flags & PKV_DECODE_PLAN_READY) ? 1 : 0;
        const int hr_rule = desc->Hkv * ct.rt;
        p.rule = PlanRule{opts->partition_tokens > 0 ? P : 0, opts->partition_tokens > 0 ? 0 : opts->num_splits,
                          (int)base_partition(desc), (6 * sms + hr_rule - 1) / hr_rule, ns,
                          (long long)desc->B * p.n_cap < (1LL << 31) ? 1 : 0};
        grid = std::min(plan_items(desc, ns), (long long)kDevicePlanCtasPerSm * sms);
    }
    record(opts ? opts->phase1_event_start : nullptr, s);
    {
        TraceRange r("pkv::decode.phase1");
        if (dispatch_phase1(desc, p, mk, mv, s, grid) != cudaSuccess) return PKV_CUDA_ERROR;
    }
    record(opts ? opts->phase1_event_stop : nullptr, s);
    if (ns > 1) {
        // Programmatic dependent of phase 1 (unless an event sits between them).
        TraceRange r("pkv::decode.combine");
        CombineParams c{context_lens, p.part_acc, p.part_m, p.part_l, out, desc->B, desc->Hq, P, ns, p.n_cap, 1,
                        desc->q_len, p.plan_hdr};
        if (launch_combine(desc->dtype, desc->D, c, s, !(opts && opts->phase1_event_stop)) != cudaSuccess)
            return PKV_CUDA_ERROR;
    }
    return PKV_OK;
}

extern "C" {

int pkv_decode_partials(const pkv_decode_desc* desc, const pkv_decode_opts* opts, const void* q, const void* k_cache,
                        const void* v_cache, const int32_t* block_table, const int32_t* context_lens, float scale,
                        float* part_acc, float* part_m, float* part_l, int num_splits_capacity,
                        int* partition_tokens_out, int* num_splits_out, pkv_stream_t stream) {
    int st = check_desc(desc);
    if (st) return st;
    if (device_plan(opts)) return PKV_UNSUPPORTED;   // partials are laid out by the host plan
    if (desc->B > 0) {
        st = check_tensors(desc, q, k_cache, v_cache, block_table, context_lens);
        if (st) return st;
        if (!part_acc || !part_m || !part_l || !aligned(part_acc, 16) || !std::isfinite(scale))
            return PKV_INVALID_ARG;
        if (opts && opts->alibi_slopes && !aligned(opts->alibi_slopes, 4)) return PKV_INVALID_ARG;
    }
    int ns = 0, P = 0;
    st = plan(desc, opts, 0, &ns, &P);
    if (st) return st;
    if (partition_tokens_out) *partition_tokens_out = P;
    if (num_splits_out) *num_splits_out = ns;
    if (ns > num_splits_capacity) return PKV_WORKSPACE_TOO_SMALL;
    if (desc->B == 0) return PKV_OK;
    DecodeParams p;
    CUtensorMap mk, mv;
    st = prepare_phase1(desc, P, ns, q, k_cache, v_cache, block_table, context_lens, scale, head_pairs(desc), &p,
                        &mk, &mv);
    if (st) return st;
    if (opts) p.alibi = opts->alibi_slopes;
    p.partials_only = 1;
    p.ns_stride = num_splits_capacity;
    p.part_acc = part_acc;
    p.part_m = part_m;
    p.part_l = part_l;
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    if (desc->max_context_len == 0) {
        // Maps were not encoded; every split is empty, so the kernel only
        // writes sentinels and never dereferences them.
        mk = CUtensorMap{};
        mv = CUtensorMap{};
    }
    record(opts ? opts->phase1_event_start : nullptr, s);
    {
        TraceRange r("pkv::decode.phase1");
        if (dispatch_phase1(desc, p, mk, mv, s) != cudaSuccess) return PKV_CUDA_ERROR;
    }
    record(opts ? opts->phase1_event_stop : nullptr, s);
    return PKV_OK;
}

int pkv_combine(const pkv_decode_desc* desc, int partition_tokens, int num_splits, const int32_t* context_lens,
                const float* part_acc, const float* part_m, const float* part_l, void* out, pkv_stream_t stream) {
    int st = check_desc(desc);
    if (st) return st;
    if (partition_tokens <= 0 || partition_tokens % desc->block_size != 0 || num_splits <= 0) return PKV_INVALID_ARG;
    if (ceil_div(desc->max_context_len, partition_tokens) > num_splits) return PKV_INVALID_ARG;
    if (desc->B == 0) return PKV_OK;
    if (!context_lens || !part_acc || !part_m || !part_l || !out || !aligned(part_acc, 16)) return PKV_INVALID_ARG;
    CombineParams c{context_lens, part_acc, part_m, part_l, out, desc->B, desc->Hq, partition_tokens, num_splits,
                    desc->max_context_len, 0, desc->q_len, nullptr};
    TraceRange r("pkv::decode.combine");
    return launch_combine(desc->dtype, desc->D, c, reinterpret_cast<cudaStream_t>(stream), false) == cudaSuccess
               ? PKV_OK
               : PKV_CUDA_ERROR;
}

int pkv_validate_block_table(const pkv_decode_desc* desc, const int32_t* block_table, const int32_t* context_lens,
                             uint32_t* err_word, pkv_stream_t stream) {
    int st = check_desc(desc);
    if (st) return st;
    if (desc->B == 0) return PKV_OK;
    if (!block_table || !context_lens || !err_word) return PKV_INVALID_ARG;
    return launch_validate(block_table, context_lens, desc->B, desc->max_blocks_per_seq, desc->block_size,
                           desc->num_blocks, desc->max_context_len, err_word,
                           reinterpret_cast<cudaStream_t>(stream)) == cudaSuccess
               ? PKV_OK
               : PKV_CUDA_ERROR;
}

// Staged key rows: every key once, each sequence padded to a multiple of
// kMlaSeqAlign rows (at most kMlaSeqAlign - 1 zero rows per sequence).
static long long mla_stage_rows(const pkv_mla_desc& d) {
    return d.nnz > 0 ? (long long)d.nnz + (long long)kMlaSeqAlign * d.batch : 0;
}

// Tasks of the persistent prefill kernel: (16-token row tile, output half)
// pairs, at most 2 * (ceil(total_q / 16) + batch).
static long long mla_max_tasks(const pkv_mla_desc& d) {
    return 2 * (((long long)d.total_q + 15) / 16 + d.batch);
}

// Exported key blocks with a max_kv_len bound: every row tile sees at most
// ceil(max_kv_len / 128) blocks.
static long long mla_export_blocks(const pkv_mla_desc& d) {
    return d.max_kv_len > 0 ? mla_max_tasks(d) / 2 * (((long long)d.max_kv_len + 127) / 128) : 0;
}

static int check_mla_desc(const pkv_mla_desc* desc) {
    if (!desc) return PKV_INVALID_ARG;
    const pkv_mla_desc& d = *desc;
    if (d.total_q < 0 || d.batch < 0 || d.num_pages < 0 || d.nnz < 0 || d.num_heads <= 0 || d.d_ckv <= 0 ||
        d.d_kpe <= 0)
        return PKV_INVALID_ARG;
    if (d.total_q > 0 && d.batch == 0) return PKV_INVALID_ARG;
    if (d.num_heads != 16 || d.d_ckv != 512 || d.d_kpe != 64) return PKV_UNSUPPORTED;
    if ((long long)d.total_q * d.num_heads * d.d_ckv > (long long)1 << 40) return PKV_UNSUPPORTED;
    if (d.max_kv_len < 0) return PKV_INVALID_ARG;
    if (mla_stage_rows(d) > INT_MAX || mla_max_tasks(d) > INT_MAX / 2) return PKV_UNSUPPORTED;
    if (mla_export_blocks(d) > INT_MAX / 512) return PKV_UNSUPPORTED;   // rows of the P tensor map
    return PKV_OK;
}

// Workspace: 256-byte header | task list (16 bytes per task) | first row tile
// of each sequence (batch + 1 ints) | first staged row of each sequence
// (batch ints) | staged key rows | with max_kv_len > 0: export base per row
// tile | exported P | rescale factors | flags | row sums.
struct MlaLayout {
    size_t tasks, seq_tile, seq_row, stage, exp_base, exp_p, exp_alpha, exp_flag, exp_l, total;
};
static MlaLayout mla_layout(const pkv_mla_desc& d) {
    MlaLayout l;
    l.tasks = kHeaderBytes;
    l.seq_tile = l.tasks + align256((size_t)mla_max_tasks(d) * 16);
    l.seq_row = l.seq_tile + align256((size_t)(d.batch + 1) * 4);
    l.stage = l.seq_row + align256((size_t)d.batch * 4);
    l.exp_base = l.stage + align256((size_t)mla_stage_rows(d) * kMlaStageRowBytes);
    const size_t e = (size_t)mla_export_blocks(d), tiles = e > 0 ? (size_t)mla_max_tasks(d) / 2 : 0;
    l.exp_p = l.exp_base + align256(tiles * 4);
    l.exp_alpha = l.exp_p + align256(e * 65536);
    l.exp_flag = l.exp_alpha + align256(e * 1024);
    l.exp_l = l.exp_flag + align256(e * 16);
    l.total = l.exp_l + align256(tiles * 1024);
    return l;
}

static size_t mla_workspace_bytes(const pkv_mla_desc& d) { return mla_layout(d).total; }

int pkv_mla_workspace_size(const pkv_mla_desc* desc, size_t* bytes) {
    const int st = check_mla_desc(desc);
    if (st != PKV_OK) return st;
    if (!bytes) return PKV_INVALID_ARG;
    *bytes = mla_workspace_bytes(*desc);
    return PKV_OK;
}

int pkv_mla_paged_prefill(const pkv_mla_desc* desc, const void* q_nope, const void* q_pe, const void* ckv_cache,
                          const void* kpe_cache, const int32_t* qo_indptr, const int32_t* kv_indptr,
                          const int32_t* kv_indices, float sm_scale, void* out, float* lse, void* workspace,
                          size_t workspace_bytes, pkv_stream_t stream) {
    int st = check_mla_desc(desc);
    if (st != PKV_OK) return st;
    const pkv_mla_desc& d = *desc;
    if (!std::isfinite(sm_scale)) return PKV_INVALID_ARG;
    if (d.total_q == 0) return PKV_OK;
    if (!q_nope || !q_pe || !qo_indptr || !kv_indptr || !out || !lse || !workspace) return PKV_INVALID_ARG;
    if (d.num_pages > 0 && d.nnz > 0 && (!ckv_cache || !kpe_cache || !kv_indices)) return PKV_INVALID_ARG;
    if (!aligned(q_nope, 16) || !aligned(q_pe, 16) || !aligned(out, 16) || !aligned(lse, 4) ||
        !aligned(qo_indptr, 4) || !aligned(kv_indptr, 4) || (ckv_cache && !aligned(ckv_cache, 16)) ||
        (kpe_cache && !aligned(kpe_cache, 16)) || (kv_indices && !aligned(kv_indices, 4)) ||
        !aligned(workspace, 256))
        return PKV_INVALID_ARG;
    if (workspace_bytes < mla_workspace_bytes(d)) return PKV_WORKSPACE_TOO_SMALL;
    MlaParams p{};
    p.q_nope = static_cast<const __nv_bfloat16*>(q_nope);
    p.q_pe = static_cast<const __nv_bfloat16*>(q_pe);
    p.ckv = static_cast<const __nv_bfloat16*>(ckv_cache);
    p.kpe = static_cast<const __nv_bfloat16*>(kpe_cache);
    p.qo_indptr = qo_indptr;
    p.kv_indptr = kv_indptr;
    p.kv_indices = kv_indices;
    p.out = static_cast<__nv_bfloat16*>(out);
    p.lse = lse;
    const MlaLayout lay = mla_layout(d);
    uint8_t* ws = static_cast<uint8_t*>(workspace);
    p.err = reinterpret_cast<uint32_t*>(ws);
    p.task_count = reinterpret_cast<int*>(ws) + 1;
    p.tasks = reinterpret_cast<int4*>(ws + lay.tasks);
    p.seq_tile = reinterpret_cast<int*>(ws + lay.seq_tile);
    p.seq_row = reinterpret_cast<int*>(ws + lay.seq_row);
    p.stage = ws + lay.stage;
    p.exp_cap = (int)mla_export_blocks(d);
    p.replay = p.exp_cap > 0 && d.num_pages > 0 && d.nnz > 0;
    if (p.replay) {
        p.exp_base = reinterpret_cast<int*>(ws + lay.exp_base);
        p.exp_p = reinterpret_cast<__nv_bfloat16*>(ws + lay.exp_p);
        p.exp_alpha = reinterpret_cast<float*>(ws + lay.exp_alpha);
        p.exp_flag = ws + lay.exp_flag;
        p.exp_l = reinterpret_cast<float*>(ws + lay.exp_l);
    }
    p.max_tasks = (int)mla_max_tasks(d);
    p.total_q = d.total_q;
    p.batch = d.batch;
    p.num_pages = d.num_pages;
    p.nnz = d.nnz;
    p.stage_rows = (int)mla_stage_rows(d);
    p.scale_log2 = (float)((double)sm_scale * 1.4426950408889634);
    p.stress_ns = g_stress_ns.load(std::memory_order_relaxed);
    p.stress_consumer_ns = g_stress_consumer_ns.load(std::memory_order_relaxed);
    MlaMaps maps;
    std::memset(&maps, 0, sizeof(maps));
    const cuuint64_t q_rows = (cuuint64_t)d.total_q * 16;
    st = encode_rows_map(&maps.q_nope, q_nope, 512, q_rows, 64, 128);
    if (st == PKV_OK) st = encode_rows_map(&maps.q_pe, q_pe, 64, q_rows, 64, 128);
    const cuuint64_t stage_rows = (cuuint64_t)p.stage_rows;
    if (st == PKV_OK && d.num_pages > 0 && stage_rows > 0) st = encode_rows_map(&maps.kv, p.stage, 576, stage_rows, 64, 64);
    if (st == PKV_OK && d.num_pages > 0 && stage_rows > 0) st = encode_rows_map(&maps.v, p.stage, 576, stage_rows, 64, 32);
    if (st == PKV_OK && p.replay)
        st = encode_rows_map(&maps.p_exp, p.exp_p, 64, (cuuint64_t)p.exp_cap * 512, 64, 128, false);
    if (st != PKV_OK) return st;
    TraceRange r("pkv::mla.prefill");
    return launch_mla_prefill(p, maps, reinterpret_cast<cudaStream_t>(stream)) == cudaSuccess ? PKV_OK
                                                                                              : PKV_CUDA_ERROR;
}

}  // extern "C"
