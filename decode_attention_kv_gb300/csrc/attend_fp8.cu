// attend_fp8.cu -- the attention kernels over E4M3 rows (D code bytes + a
// 16-byte field holding the row's fp32 scale).
#include "attend_quant.cuh"

namespace kvd {

cudaError_t launch_attend_fp8(int D, int G, int mode, const AttendParams& p,
                               const CUtensorMap* kmap, const CUtensorMap* vmap,
                               cudaStream_t stream) {
    return launch_attend_quant<false>(D, G, mode, p, kmap, vmap, stream);
}

int small_shared_bytes_fp8(int D, int G, int chunk, int slots, int nwg) {
    return small_shared_bytes_quant<false>(D, G, chunk, slots, nwg);
}

cudaError_t launch_attend_small_fp8(int D, int G, const AttendParams& p, int S, int rows,
                                    cudaStream_t stream) {
    return launch_attend_small_quant<false>(D, G, p, S, rows, stream);
}

}  // namespace kvd
