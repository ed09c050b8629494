// attend_inst.cuh -- instantiation and launch of the persistent attention
// kernel for one element type.  Included by exactly one .cu per element type
// so that the instantiations compile in parallel.
#pragma once

#include <mutex>

#include "attend_kernel.cuh"
#include "kvd_internal.h"

namespace kvd {

// Ring depth that keeps a CTA near `budget` bytes of stages (2..8 stages).
constexpr int stages_for(int stage_bytes, int budget) {
    return budget / stage_bytes < 2 ? 2 : (budget / stage_bytes > 8 ? 8 : budget / stage_bytes);
}

// CUDA-core consumers: 32-token tiles, four consumer warps, about 100 KB of
// ring so that two CTAs share an SM.
template <typename Elem, int D, int G>
struct SimtCfg {
    using Cons = SimtConsumer<Elem, D, G, 32, 4>;
    static constexpr int STAGES = stages_for(KernelShape<Cons, 2>::kStageBytes, 100 * 1024);
};

// Tensor-core consumers: 64-token tiles (one 16-token slab per consumer
// warp), a ring of about 170 KB, one CTA per SM.
template <int D, int G>
struct MmaCfg {
    using Cons = MmaConsumer<D, G, 64, 4>;
    static constexpr int STAGES = stages_for(KernelShape<Cons, 2>::kStageBytes, 160 * 1024);
};

// Per-device launch facts of one kernel instantiation: the shared-memory
// attribute is set and the persistent grid sized once per device.
struct DeviceFacts {
    std::mutex mu;
    int ctas[64] = {};  // persistent CTAs per device (0 = not set up yet)
};

template <class Cons, int STAGES, bool PAGED>
cudaError_t launch_kernel(const AttendParams& p, const CUtensorMap* kmap, const CUtensorMap* vmap,
                          cudaStream_t stream) {
    using Sh = KernelShape<Cons, STAGES>;
    auto kern = attend_kernel<Cons, STAGES, PAGED>;
    constexpr int kThreads = Sh::kThreads;
    static DeviceFacts facts;
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if (dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
    int ctas;
    {
        std::lock_guard<std::mutex> lock(facts.mu);
        if (!facts.ctas[dev]) {
            e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                     Sh::kSmemAlloc);
            if (e != cudaSuccess) return e;
            int per_sm = 0, nsm = 0;
            e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, kern, kThreads,
                                                              Sh::kSmemAlloc);
            if (e != cudaSuccess) return e;
            e = cudaDeviceGetAttribute(&nsm, cudaDevAttrMultiProcessorCount, dev);
            if (e != cudaSuccess) return e;
            facts.ctas[dev] = (per_sm < 1 ? 1 : per_sm) * (nsm < 1 ? 1 : nsm);
        }
        ctas = facts.ctas[dev];
    }
    const int grid = p.units < ctas ? p.units : ctas;
    return launch_pdl(kern, dim3(grid), dim3(kThreads), Sh::kSmemAlloc, stream, p, *kmap, *vmap);
}

template <typename Elem, int D, int G>
cudaError_t launch_simt(bool paged, const AttendParams& p, const CUtensorMap* kmap,
                        const CUtensorMap* vmap, cudaStream_t stream) {
    using C = SimtCfg<Elem, D, G>;
    return paged ? launch_kernel<typename C::Cons, C::STAGES, true>(p, kmap, vmap, stream)
                 : launch_kernel<typename C::Cons, C::STAGES, false>(p, kmap, vmap, stream);
}

template <int D, int G>
cudaError_t launch_mma(bool paged, const AttendParams& p, const CUtensorMap* kmap,
                       const CUtensorMap* vmap, cudaStream_t stream) {
    using C = MmaCfg<D, G>;
    return paged ? launch_kernel<typename C::Cons, C::STAGES, true>(p, kmap, vmap, stream)
                 : launch_kernel<typename C::Cons, C::STAGES, false>(p, kmap, vmap, stream);
}

}  // namespace kvd
