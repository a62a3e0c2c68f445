// internal.h -- declarations shared by the library's translation units.
#pragma once

#include "decode.cuh"
#include "pkv.h"

namespace pkv {

struct CombineParams {
    const int32_t* ctx;        // [B]
    const float* part_acc;     // [B][q_len][Hq][ns_stride][D]
    const float* part_m;       // [B][q_len][Hq][ns_stride]
    const float* part_l;       // [B][q_len][Hq][ns_stride]
    void* out;                 // [B][q_len][Hq][D]
    int B, Hq, P, ns_stride, n_cap;
    int skip_single;           // 1: rows whose sequence has <= 1 split were written by phase 1
    int q_len;                 // query tokens per sequence
    const int* sched_hdr;      // device plan: header word 0 holds P, written by phase 1 (else nullptr: P above)
};


// Phase-1 dispatch, one function per (layout, dtype) translation unit.
// D in {64, 128, 256}; nt = query-column tiles of 8 per CTA (1, or 2 for D <= 128).
cudaError_t launch_decode_nhd_f16(int D, int nt, const DecodeParams& p, long long grid, const CUtensorMap& k, const CUtensorMap& v,
                                  cudaStream_t s);
cudaError_t launch_decode_nhd_bf16(int D, int nt, const DecodeParams& p, long long grid, const CUtensorMap& k, const CUtensorMap& v,
                                   cudaStream_t s);
cudaError_t launch_decode_vllm_f16(int D, int nt, const DecodeParams& p, long long grid, const CUtensorMap& k, const CUtensorMap& v,
                                   cudaStream_t s);
cudaError_t launch_decode_vllm_bf16(int D, int nt, const DecodeParams& p, long long grid, const CUtensorMap& k,
                                    const CUtensorMap& v, cudaStream_t s);
// FP8 E4M3 caches (NHD layout), fp16 / bf16 queries and output.
cudaError_t launch_decode_nhd8_f16(int D, int nt, const DecodeParams& p, long long grid, const CUtensorMap& k,
                                   const CUtensorMap& v, cudaStream_t s);
cudaError_t launch_decode_nhd8_bf16(int D, int nt, const DecodeParams& p, long long grid, const CUtensorMap& k,
                                    const CUtensorMap& v, cudaStream_t s);

// MLA paged causal prefill (mla.cu); bf16 tensors, page size 1.
struct MlaParams {
    const __nv_bfloat16* q_nope;   // [total_q][16][512]
    const __nv_bfloat16* q_pe;     // [total_q][16][64]
    const __nv_bfloat16* ckv;      // [num_pages][512]
    const __nv_bfloat16* kpe;      // [num_pages][64]
    const int32_t* qo_indptr;      // [batch + 1]
    const int32_t* kv_indptr;      // [batch + 1]
    const int32_t* kv_indices;     // [kv_indptr[batch]]
    __nv_bfloat16* out;            // [total_q][16][512]
    float* lse;                    // [total_q][16]
    uint8_t* stage;                // [stage_rows][1152]: ckv row | kpe row of each key, per sequence
                                   // padded with zero rows to a multiple of 128 rows
    int4* tasks;                   // [max_tasks] (sequence, first token, first staged row, key blocks |
                                   // output half << 30), most key blocks first (built on the device)
    int* seq_tile;                 // [batch + 1] first 16-token row tile of each sequence
    int* seq_row;                  // [batch] first staged row of each sequence
    int* task_count;               // header words 1-6: tasks listed, of them with keys (listed
                                   // first), next task with keys to hand out; replay list: next
                                   // task to hand out, tasks, first entry
    // Replay (max_kv_len > 0): the tasks of the first output half export each key
    // block's bf16 P, the factor O was rescaled by before it and the final row
    // sums; mla_replay_kernel computes the second half from them (S once per tile).
    int replay;                    // 1: export, and list the second half for the replay kernel
    int* exp_base;                 // [tiles] first export block of the tile at each list position
    __nv_bfloat16* exp_p;          // [exp_cap][2 CTAs][2 key halves][8][128 rows][8 keys]: key half
                                   // chunk-major (keys 8q .. 8q + 7 of all rows, then q + 1)
    float* exp_alpha;              // [exp_cap][2 CTAs][128 rows]
    uint8_t* exp_flag;             // [exp_cap][2 CTAs][8 softmax warps]: some row of the warp rescaled
    float* exp_l;                  // [tiles][2 CTAs][128 rows] final row sums
    int exp_cap;                   // export blocks the workspace holds
    int max_tasks;                 // 2 * (ceil(total_q / 16) + batch)
    uint32_t* err;                 // header word 0
    int total_q, batch, num_pages, nnz;
    int stage_rows;                // rows of `stage`: nnz + 128 * batch (0 without keys)
    float scale_log2;              // sm_scale * log2(e)
    uint32_t stress_ns;            // producer pause after each issued copy (pkv_set_stress_delay), 0: none
    uint32_t stress_consumer_ns;   // MMA thread / softmax warp pause after each slot / block, 0: none
};

constexpr int kMlaStageRowBytes = (512 + 64) * 2;
// Each sequence's staged keys start on a multiple of this many rows, so no
// 128-row key block of one sequence reaches another's rows.
constexpr int kMlaSeqAlign = 128;

// TMA descriptors of the MLA operands: q_nope / q_pe as 2-D {512 | 64,
// total_q * 16} tensors with {64, 128} boxes, and the staged keys as {576,
// stage_rows}, with {64, 64} boxes (kv: K chunks, one CTA's half of a key
// block) or {64, 32} boxes (v: V chunk blocks), all with 128-byte swizzle.
// kv and v are unused (zero) when the pool is empty.
struct MlaMaps {
    CUtensorMap q_nope, q_pe, kv, v, p_exp;   // p_exp: exp_p as {64, exp_cap * 512}, {64, 128} boxes, no swizzle
};

cudaError_t launch_mla_prefill(const MlaParams& p, const MlaMaps& maps, cudaStream_t stream);

// The decode step of pkv_paged_decode_attention (api.cu); with clear_err_word
// it zeroes the workspace's error word on the stream once every argument has
// passed its checks, before the first kernel.
int paged_decode_impl(const pkv_decode_desc* desc, const pkv_decode_opts* opts, const void* q, const void* k_cache,
                      const void* v_cache, const int32_t* block_table, const int32_t* context_lens, float scale,
                      void* out, void* workspace, size_t workspace_bytes, pkv_stream_t stream, bool clear_err_word);

// after_phase1: launched as a programmatic dependent of the phase-1 kernel just
// enqueued on the same stream (its prologue overlaps phase 1's tail).
cudaError_t launch_combine(int dtype, int D, const CombineParams& p, cudaStream_t stream, bool after_phase1);
cudaError_t launch_validate(const int32_t* table, const int32_t* ctx, int B, int MBPS, int BS, int NB, int max_ctx,
                            uint32_t* err, cudaStream_t stream);

}  // namespace pkv
