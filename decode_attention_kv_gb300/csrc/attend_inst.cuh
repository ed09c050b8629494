// attend_inst.cuh -- instantiation and launch of the split kernel for one
// element type.  Included by exactly one .cu per element type so that the
// instantiations compile in parallel.
#pragma once

#include "attend_mma.cuh"
#include "attend_split.cuh"
#include "kvd_internal.h"

namespace kvd {

// Tile / ring / warp geometry per element type and head_dim.  A ring stage
// holds K and V of T tokens; two CTAs fit on one SM.
template <typename Elem, int D>
struct Geom {
    static constexpr int T = 32;
    static constexpr int NCW = 4;
    static constexpr int kStage = 2 * T * D * (int)sizeof(Elem);
    static constexpr int STAGES = (96 * 1024 / kStage) > 8 ? 8 : (96 * 1024 / kStage);
};

template <typename Elem, int D, int G, bool PAGED>
cudaError_t launch_one(const AttendParams& p, const CUtensorMap* kmap, const CUtensorMap* vmap,
                       dim3 grid, cudaStream_t stream) {
    using Gm = Geom<Elem, D>;
    using Sh = AttendShape<Elem, D, G, Gm::T, Gm::STAGES, Gm::NCW>;
    auto kern = attend_split_kernel<Elem, D, G, Gm::T, Gm::STAGES, Gm::NCW, PAGED>;
    static int configured_device = -1;  // attribute set once per device
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if (configured_device != dev) {
        e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, Sh::kSmemAlloc);
        if (e != cudaSuccess) return e;
        configured_device = dev;
    }
    return launch_pdl(kern, grid, dim3((Gm::NCW + 1) * 32), Sh::kSmemAlloc, stream, p, *kmap,
                      *vmap);
}

template <typename Elem, int D, bool PAGED>
cudaError_t launch_g(int G, const AttendParams& p, const CUtensorMap* kmap,
                     const CUtensorMap* vmap, dim3 grid, cudaStream_t stream) {
    switch (G) {
        case 1: return launch_one<Elem, D, 1, PAGED>(p, kmap, vmap, grid, stream);
        case 2: return launch_one<Elem, D, 2, PAGED>(p, kmap, vmap, grid, stream);
        case 4: return launch_one<Elem, D, 4, PAGED>(p, kmap, vmap, grid, stream);
        case 8: return launch_one<Elem, D, 8, PAGED>(p, kmap, vmap, grid, stream);
        default: return cudaErrorInvalidValue;
    }
}

template <typename Elem>
cudaError_t launch_elem(int D, int G, bool paged, const AttendParams& p, const CUtensorMap* kmap,
                        const CUtensorMap* vmap, dim3 grid, cudaStream_t stream) {
    if (D == 64)
        return paged ? launch_g<Elem, 64, true>(G, p, kmap, vmap, grid, stream)
                     : launch_g<Elem, 64, false>(G, p, kmap, vmap, grid, stream);
    if (D == 128)
        return paged ? launch_g<Elem, 128, true>(G, p, kmap, vmap, grid, stream)
                     : launch_g<Elem, 128, false>(G, p, kmap, vmap, grid, stream);
    return cudaErrorInvalidValue;
}

template <typename Elem, int D>
AttendGeom geom_of() {
    using Gm = Geom<Elem, D>;
    using Sh = AttendShape<Elem, D, 8, Gm::T, Gm::STAGES, Gm::NCW>;
    return AttendGeom{Gm::T, Gm::STAGES, Gm::NCW, Sh::kSmemAlloc, false};
}

// Tensor-core kernel geometry: 64-token stages (one 16-token slab per
// consumer warp), three stages, two CTAs per SM.
struct MmaGeom {
    static constexpr int T = 64;
    static constexpr int NCW = 4;
    static constexpr int STAGES = 3;
};

template <int D, int G, bool PAGED>
cudaError_t launch_mma_one(const AttendParams& p, const CUtensorMap* kmap,
                           const CUtensorMap* vmap, dim3 grid, cudaStream_t stream) {
    using Sh = MmaShape<D, G, MmaGeom::T, MmaGeom::STAGES, MmaGeom::NCW>;
    auto kern = attend_mma_kernel<D, G, MmaGeom::T, MmaGeom::STAGES, MmaGeom::NCW, PAGED>;
    static int configured_device = -1;
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if (configured_device != dev) {
        e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, Sh::kSmemAlloc);
        if (e != cudaSuccess) return e;
        configured_device = dev;
    }
    return launch_pdl(kern, grid, dim3((MmaGeom::NCW + 1) * 32), Sh::kSmemAlloc, stream, p, *kmap,
                      *vmap);
}

template <int D, bool PAGED>
cudaError_t launch_mma_g(int G, const AttendParams& p, const CUtensorMap* kmap,
                         const CUtensorMap* vmap, dim3 grid, cudaStream_t stream) {
    switch (G) {
        case 4: return launch_mma_one<D, 4, PAGED>(p, kmap, vmap, grid, stream);
        case 8: return launch_mma_one<D, 8, PAGED>(p, kmap, vmap, grid, stream);
        default: return cudaErrorInvalidValue;
    }
}

template <int D>
AttendGeom mma_geom_of() {
    using Sh = MmaShape<D, 8, MmaGeom::T, MmaGeom::STAGES, MmaGeom::NCW>;
    return AttendGeom{MmaGeom::T, MmaGeom::STAGES, MmaGeom::NCW, Sh::kSmemAlloc, true};
}

}  // namespace kvd
