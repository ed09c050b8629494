// attend_f32.cu -- fp32 instantiations of the attention kernel (CUDA-core
// consumers for every group width).
#include "attend_inst.cuh"

namespace kvd {

cudaError_t launch_attend_f32(int D, int G, int mode, const AttendParams& p,
                              const CUtensorMap* kmap, const CUtensorMap* vmap,
                              cudaStream_t stream) {
    if (D == 128) {
        switch (G) {
            case 1: return launch_simt<float, 128, 1>(mode, p, kmap, vmap, stream);
            case 2: return launch_simt<float, 128, 2>(mode, p, kmap, vmap, stream);
            case 4: return launch_simt<float, 128, 4>(mode, p, kmap, vmap, stream);
            case 8: return launch_simt<float, 128, 8>(mode, p, kmap, vmap, stream);
        }
    } else if (D == 64) {
        switch (G) {
            case 1: return launch_simt<float, 64, 1>(mode, p, kmap, vmap, stream);
            case 2: return launch_simt<float, 64, 2>(mode, p, kmap, vmap, stream);
            case 4: return launch_simt<float, 64, 4>(mode, p, kmap, vmap, stream);
            case 8: return launch_simt<float, 64, 8>(mode, p, kmap, vmap, stream);
        }
    }
    return cudaErrorInvalidValue;
}

AttendGeom attend_geom_f32(int, int) { return AttendGeom{32, 0, 4, 0, false}; }

}  // namespace kvd
