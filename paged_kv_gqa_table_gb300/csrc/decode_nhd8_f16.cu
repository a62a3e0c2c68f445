// decode_nhd8_f16.cu -- phase-1 instantiations for FP8 E4M3 caches in the NHD
// layout ([num_blocks][Hkv][block_size][D] bytes) with f16 queries and output;
// one KV head or a pair of them per CTA.
#include "internal.h"

namespace pkv {

cudaError_t launch_decode_nhd8_f16(int D, int nt, const DecodeParams& p, long long grid, const CUtensorMap& k,
                                 const CUtensorMap& v, cudaStream_t s) {
    if (D == 128 && nt == 1 && p.Hc != p.Hkv) return launch_decode_phase1_pairs<__half>(p, grid, k, v, s);
    if (D == 64 && nt == 1) return launch_decode_phase1<__half, kLayoutNHD8, 64, 1>(p, grid, k, v, s);
    if (D == 64 && nt == 2) return launch_decode_phase1<__half, kLayoutNHD8, 64, 2>(p, grid, k, v, s);
    if (D == 128 && nt == 1) return launch_decode_phase1<__half, kLayoutNHD8, 128, 1>(p, grid, k, v, s);
    if (D == 128 && nt == 2) return launch_decode_phase1<__half, kLayoutNHD8, 128, 2>(p, grid, k, v, s);
    if (D == 256 && nt == 1) return launch_decode_phase1<__half, kLayoutNHD8, 256, 1>(p, grid, k, v, s);
    return cudaErrorInvalidValue;
}

}  // namespace pkv
