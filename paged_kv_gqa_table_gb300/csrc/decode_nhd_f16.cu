// decode_nhd_f16.cu -- phase-1 instantiations for the NHD ([num_blocks][Hkv][block_size][D])
// cache layout with f16 data.  One translation unit per (layout, dtype) so the
// build compiles them in parallel.
#include "internal.h"

namespace pkv {

cudaError_t launch_decode_nhd_f16(int D, int nt, const DecodeParams& p, long long grid, const CUtensorMap& k,
                                  const CUtensorMap& v,
                                   cudaStream_t s) {
    if (D == 64 && nt == 1) return launch_decode_phase1<__half, kLayoutNHD, 64, 1>(p, grid, k, v, s);
    if (D == 64 && nt == 2) return launch_decode_phase1<__half, kLayoutNHD, 64, 2>(p, grid, k, v, s);
    if (D == 128 && nt == 1) return launch_decode_phase1<__half, kLayoutNHD, 128, 1>(p, grid, k, v, s);
    if (D == 128 && nt == 2) return launch_decode_phase1<__half, kLayoutNHD, 128, 2>(p, grid, k, v, s);
    if (D == 256 && nt == 1) return launch_decode_phase1<__half, kLayoutNHD, 256, 1>(p, grid, k, v, s);
    return cudaErrorInvalidValue;
}

}  // namespace pkv
