// static_scratch.cu -- pkv_paged_decode_attention_static: the decode step for
// callers that cannot allocate device memory.
//
// Some callers may not call cudaMalloc (or any allocator) at the point where
// they run a decode step: plugin interfaces whose enqueue hook owns no
// allocator, engines that hand out all device memory from a fixed pool at
// start-up and forbid allocations afterwards, or code on a latency-critical
// path where an allocation could synchronise the device.  For them the split
// partials live in one file-scope device array, reserved on every GPU that
// loads this library for as long as the process lives.
#include <cstdint>
#include <mutex>

#include "internal.h"
#include "pkv.h"

namespace {

constexpr size_t kStaticScratchBytes = PKV_STATIC_SCRATCH_BYTES;   // 32 MiB

static __device__ __align__(256) unsigned char g_scratch[kStaticScratchBytes];

// Host-side record of what the last call on each device left in the array:
// whether it holds a device plan, and for which problem (description and
// partition options).  A call that reuses a plan (PKV_DECODE_PLAN_READY) is
// refused unless the previous call on the device made one for the same
// problem; the record cannot see context_lens, which the caller keeps equal.
struct LastCall {
    bool device_plan = false;
    pkv_decode_desc desc{};
    int partition_tokens = 0, num_splits = 0;
};

struct DeviceState {
    void* addr = nullptr;   // device address of g_scratch
    LastCall last;
};

std::mutex g_mu;
DeviceState g_dev[pkv::kMaxDevices];

bool same_problem(const pkv_decode_desc& a, const pkv_decode_desc& b) {
    return a.B == b.B && a.Hq == b.Hq && a.Hkv == b.Hkv && a.D == b.D && a.block_size == b.block_size &&
           a.max_blocks_per_seq == b.max_blocks_per_seq && a.num_blocks == b.num_blocks &&
           a.max_context_len == b.max_context_len && a.sum_context_len == b.sum_context_len &&
           a.dtype == b.dtype && a.layout == b.layout && a.x_pack == b.x_pack && a.kv_dtype == b.kv_dtype &&
           a.k_scale == b.k_scale && a.v_scale == b.v_scale && a.q_len == b.q_len;
}

// The current device's state, with g_scratch's device address looked up
// (once per device, with that device current).  The host symbol g_scratch is
// only a stand-in and is never handed to a kernel.  Call with g_mu held.
int device_state(DeviceState** out) {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= pkv::kMaxDevices) return PKV_CUDA_ERROR;
    DeviceState& d = g_dev[dev];
    if (!d.addr) {
        void* p = nullptr;
        if (cudaGetSymbolAddress(&p, g_scratch) != cudaSuccess || p == nullptr) return PKV_CUDA_ERROR;
        d.addr = p;
    }
    *out = &d;
    return PKV_OK;
}

}  // namespace

extern "C" {

int pkv_paged_decode_attention_static(const pkv_decode_desc* desc, const pkv_decode_opts* opts, const void* q,
                                      const void* k_cache, const void* v_cache, const int32_t* block_table,
                                      const int32_t* context_lens, float scale, void* out, pkv_stream_t stream) {
    size_t need = 0;
    // Sizes are checked on the host before anything touches the GPU; a plan
    // whose partials exceed the array is refused, never truncated.
    int st = pkv_decode_workspace_size(desc, opts, 0, &need);
    if (st) return st;
    if (need > kStaticScratchBytes) return PKV_WORKSPACE_TOO_SMALL;
    if (desc->B == 0) return PKV_OK;
    const int flags = opts ? opts->flags : 0;
    std::lock_guard<std::mutex> lock(g_mu);
    DeviceState* d = nullptr;
    st = device_state(&d);
    if (st) return st;
    if ((flags & PKV_DECODE_PLAN_READY) &&
        !(d->last.device_plan && same_problem(d->last.desc, *desc) &&
          d->last.partition_tokens == opts->partition_tokens && d->last.num_splits == opts->num_splits))
        return PKV_INVALID_ARG;
    // Every argument is checked before the array is touched; the error word is
    // then cleared on the stream (the rest of the header and the split table
    // may hold a device plan an earlier call made for reuse); the partials are
    // fully written by phase 1 before phase 2 reads them, so they need no
    // clearing.
    st = pkv::paged_decode_impl(desc, opts, q, k_cache, v_cache, block_table, context_lens, scale, out, d->addr,
                                kStaticScratchBytes, stream, true);
    if (st == PKV_OK) {
        d->last.device_plan = (flags & PKV_DECODE_DEVICE_PLAN) != 0;
        d->last.desc = *desc;
        d->last.partition_tokens = opts ? opts->partition_tokens : 0;
        d->last.num_splits = opts ? opts->num_splits : 0;
    } else if (st == PKV_CUDA_ERROR) {
        d->last = LastCall{};   // something may have been enqueued: assume the plan is gone
    }
    return st;
}

int pkv_static_scratch_error(uint32_t* dst, pkv_stream_t stream) {
    if (!dst) return PKV_INVALID_ARG;
    std::lock_guard<std::mutex> lock(g_mu);
    DeviceState* d = nullptr;
    const int st = device_state(&d);
    if (st) return st;
    return cudaMemcpyAsync(dst, d->addr, sizeof(uint32_t), cudaMemcpyDefault,
                           reinterpret_cast<cudaStream_t>(stream)) == cudaSuccess
               ? PKV_OK
               : PKV_CUDA_ERROR;
}

}  // extern "C"
