// attend_fp8.cu -- instantiations of the attention kernel over quantised K/V
// rows (E4M3 codes with a per-row fp32 scale; q and out bf16): tensor-core
// consumers for every group width up to 8 query heads per kv head.
#include "attend_inst.cuh"

namespace kvd {

cudaError_t launch_attend_fp8(int D, int G, const AttendParams& p, cudaStream_t stream) {
    if (D == 128) {
        switch (G) {
            case 1: return launch_fp8<128, 1>(p, stream);
            case 2: return launch_fp8<128, 2>(p, stream);
            case 4: return launch_fp8<128, 4>(p, stream);
            case 8: return launch_fp8<128, 8>(p, stream);
        }
    } else if (D == 64) {
        switch (G) {
            case 1: return launch_fp8<64, 1>(p, stream);
            case 2: return launch_fp8<64, 2>(p, stream);
            case 4: return launch_fp8<64, 4>(p, stream);
            case 8: return launch_fp8<64, 8>(p, stream);
        }
    }
    return cudaErrorInvalidValue;
}

}  // namespace kvd
