// attend_bf16.cu -- bf16 instantiations of the split-KV attention kernel.
#include "attend_inst.cuh"

namespace kvd {

cudaError_t launch_attend_bf16(int D, int G, bool paged, const AttendParams& p,
                               const CUtensorMap* kmap, const CUtensorMap* vmap, dim3 grid,
                               cudaStream_t stream) {
    if (attend_uses_mma(KVD_BF16, G)) {
        if (D == 64)
            return paged ? launch_mma_g<64, true>(G, p, kmap, vmap, grid, stream)
                         : launch_mma_g<64, false>(G, p, kmap, vmap, grid, stream);
        if (D == 128)
            return paged ? launch_mma_g<128, true>(G, p, kmap, vmap, grid, stream)
                         : launch_mma_g<128, false>(G, p, kmap, vmap, grid, stream);
        return cudaErrorInvalidValue;
    }
    return launch_elem<__nv_bfloat16>(D, G, paged, p, kmap, vmap, grid, stream);
}

AttendGeom attend_geom_bf16(int D, int G) {
    if (attend_uses_mma(KVD_BF16, G)) return D == 64 ? mma_geom_of<64>() : mma_geom_of<128>();
    return D == 64 ? geom_of<__nv_bfloat16, 64>() : geom_of<__nv_bfloat16, 128>();
}

}  // namespace kvd
