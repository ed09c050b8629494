// attend_bf16.cu -- bf16 instantiations of the attention kernel: tensor-core
// consumers for 4 or 8 query heads per kv head, CUDA-core consumers for 1-2.
#include "attend_inst.cuh"

namespace kvd {

cudaError_t launch_attend_bf16(int D, int G, int mode, const AttendParams& p,
                               const CUtensorMap* kmap, const CUtensorMap* vmap,
                               cudaStream_t stream) {
    if (D == 128) {
        switch (G) {
            case 1: return launch_simt<__nv_bfloat16, 128, 1>(mode, p, kmap, vmap, stream);
            case 2: return launch_simt<__nv_bfloat16, 128, 2>(mode, p, kmap, vmap, stream);
            case 4: return launch_mma<128, 4>(mode, p, kmap, vmap, stream);
            case 8: return launch_mma<128, 8>(mode, p, kmap, vmap, stream);
        }
    } else if (D == 64) {
        switch (G) {
            case 1: return launch_simt<__nv_bfloat16, 64, 1>(mode, p, kmap, vmap, stream);
            case 2: return launch_simt<__nv_bfloat16, 64, 2>(mode, p, kmap, vmap, stream);
            case 4: return launch_mma<64, 4>(mode, p, kmap, vmap, stream);
            case 8: return launch_mma<64, 8>(mode, p, kmap, vmap, stream);
        }
    }
    return cudaErrorInvalidValue;
}

AttendGeom attend_geom_bf16(int D, int G) {
    if (attend_uses_mma(KVD_BF16, G)) return AttendGeom{64, 0, 4, 0, true};
    (void)D;
    return AttendGeom{32, 0, 4, 0, false};
}

}  // namespace kvd
