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

#include "pkv.h"

namespace {

constexpr size_t kStaticScratchBytes = PKV_STATIC_SCRATCH_BYTES;   // 32 MiB

static __device__ __align__(256) unsigned char g_scratch[kStaticScratchBytes];

// Device address of g_scratch, looked up once per device with that device
// current.  The host symbol itself is only a stand-in and is never handed to
// a kernel.
int scratch_address(void** out) {
    static std::mutex mu;
    static void* addr[64] = {};
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return PKV_CUDA_ERROR;
    std::lock_guard<std::mutex> lock(mu);
    if (!addr[dev]) {
        void* p = nullptr;
        if (cudaGetSymbolAddress(&p, g_scratch) != cudaSuccess || p == nullptr) return PKV_CUDA_ERROR;
        addr[dev] = p;
    }
    *out = addr[dev];
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
    void* scratch = nullptr;
    st = scratch_address(&scratch);
    if (st) return st;
    // The header's error word must start at zero (the rest of the header may
    // hold a device plan an earlier call made for reuse); the partials are
    // fully written by phase 1 before phase 2 reads them, so they need no clearing.
    if (cudaMemsetAsync(scratch, 0, sizeof(uint32_t), reinterpret_cast<cudaStream_t>(stream)) != cudaSuccess)
        return PKV_CUDA_ERROR;
    return pkv_paged_decode_attention(desc, opts, q, k_cache, v_cache, block_table, context_lens, scale, out,
                                      scratch, kStaticScratchBytes, stream);
}

}  // extern "C"
