// attend_f32.cu -- fp32 instantiations of the split-KV attention kernel.
#include "attend_inst.cuh"

namespace kvd {

cudaError_t launch_attend_f32(int D, int G, bool paged, const AttendParams& p,
                              const CUtensorMap* kmap, const CUtensorMap* vmap, dim3 grid,
                              cudaStream_t stream) {
    return launch_elem<float>(D, G, paged, p, kmap, vmap, grid, stream);
}

AttendGeom attend_geom_f32(int D, int /*G*/) {
    return D == 64 ? geom_of<float, 64>() : geom_of<float, 128>();
}

}  // namespace kvd
