// attend_bf16.cu -- bf16 instantiations of the split-KV attention kernel.
#include "attend_inst.cuh"

namespace kvd {

cudaError_t launch_attend_bf16(int D, int G, bool paged, const AttendParams& p,
                               const CUtensorMap* kmap, const CUtensorMap* vmap, dim3 grid,
                               cudaStream_t stream) {
    return launch_elem<__nv_bfloat16>(D, G, paged, p, kmap, vmap, grid, stream);
}

AttendGeom attend_geom_bf16(int D) {
    return D == 64 ? geom_of<__nv_bfloat16, 64>() : geom_of<__nv_bfloat16, 128>();
}

}  // namespace kvd
