// decode_vllm_bf16.cu -- phase-1 instantiations for the vLLM x-packed ([num_blocks][Hkv][D/8][block_size][8] keys, [num_blocks][Hkv][D][block_size] values)
// cache layout with bf16 data.  One translation unit per (layout, dtype) so the
// build compiles them in parallel.
#include "internal.h"

namespace pkv {

cudaError_t launch_decode_vllm_bf16(int D, int nt, const DecodeParams& p, long long grid, const CUtensorMap& k,
                                  const CUtensorMap& v,
                                   cudaStream_t s) {
    if (D == 64 && nt == 1) return launch_decode_phase1<__nv_bfloat16, kLayoutVLLM, 64, 1>(p, grid, k, v, s);
    if (D == 64 && nt == 2) return launch_decode_phase1<__nv_bfloat16, kLayoutVLLM, 64, 2>(p, grid, k, v, s);
    if (D == 128 && nt == 1) return launch_decode_phase1<__nv_bfloat16, kLayoutVLLM, 128, 1>(p, grid, k, v, s);
    if (D == 128 && nt == 2) return launch_decode_phase1<__nv_bfloat16, kLayoutVLLM, 128, 2>(p, grid, k, v, s);
    if (D == 256 && nt == 1) return launch_decode_phase1<__nv_bfloat16, kLayoutVLLM, 256, 1>(p, grid, k, v, s);
    return cudaErrorInvalidValue;
}

}  // namespace pkv
