// attend_small_launch.cuh -- launch of one instantiation of the small-launch
// attention kernel (one CTA per (row, split), the row's splits in one
// cluster).  Included by the translation units that instantiate it.
#pragma once

#include <cstring>
#include <mutex>

#include "attend_small.cuh"
#include "kvd_internal.h"

namespace kvd {

constexpr int kSmallSmemMax = 227 * 1024;

template <class Cons, int NWG>
cudaError_t launch_small_nwg(const AttendParams& p, int S, int rows, const CUtensorMap* kmap,
                             const CUtensorMap* vmap, cudaStream_t stream) {
    using Elem = typename Cons::ElemT;
    const int nt = (p.chunk + Cons::kT - 1) / Cons::kT;
    const SmallLayout L = SmallLayout::make(nt, Cons::kTileBytes, Cons::kT, Cons::kD, Cons::kG,
                                            NWG * Cons::kNCW, (int)sizeof(Elem),
                                            p.small_push ? S : 1);
    const size_t smem = (size_t)L.bytes + 1024;
    if (smem > (size_t)kSmallSmemMax) return cudaErrorInvalidValue;
    auto kern = attend_small_kernel<Cons, NWG>;
    static std::once_flag once;
    static cudaError_t attr_err = cudaSuccess;
    std::call_once(once, [&] {
        attr_err = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                        kSmallSmemMax);
    });
    if (attr_err != cudaSuccess) return attr_err;
    cudaLaunchConfig_t cfg{};
    cfg.gridDim = dim3((unsigned)S, (unsigned)rows);
    cfg.blockDim = dim3((NWG * Cons::kNCW + 1) * 32);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = stream;
    cudaLaunchAttribute attr[2];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = (unsigned)S;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[1].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 2;
    return cudaLaunchKernelEx(&cfg, kern, p, *kmap, *vmap);
}

// Consumer warp groups per CTA: 1, or 2 for the tensor-core consumers when
// the plan found room (p.small_nwg).
template <class Cons>
cudaError_t launch_small_cfg(const AttendParams& p, int S, int rows, const CUtensorMap* kmap,
                             const CUtensorMap* vmap, cudaStream_t stream) {
    if constexpr (Cons::kSwizzled) {  // the bf16 tensor-core consumers
        if (p.small_nwg == 2) return launch_small_nwg<Cons, 2>(p, S, rows, kmap, vmap, stream);
    }
    return launch_small_nwg<Cons, 1>(p, S, rows, kmap, vmap, stream);
}

}  // namespace kvd
