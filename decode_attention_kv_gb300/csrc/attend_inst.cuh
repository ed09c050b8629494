// attend_inst.cuh -- instantiation and launch of the persistent attention
// kernel for one element type.  Included by exactly one .cu per element type
// so that the instantiations compile in parallel.
#pragma once

#include <cstring>
#include <mutex>

#include "attend_kernel.cuh"
#include "kvd_internal.h"

namespace kvd {

// Both configurations aim at two CTAs per SM (the SM's 228 KB shared memory,
// less 1 KB reserved per CTA): the other CTA's consumer warps issue while one
// CTA's warps wait on their own mma, shuffle or load latencies.  The ring
// takes what the merge buffers and the control block leave of that share
// (2..8 stages): the bytes in flight per SM are what hides HBM latency.
constexpr int kCtaSmemTarget = 113 * 1024;

template <class Cons, int MB>
constexpr int ring_stages() {
    using Sh = KernelShape<Cons, 2, MB>;
    // the control block grows by about 40 bytes per stage: budget 8 stages
    constexpr int fixed = Sh::kSmemAlloc - Sh::kRingBytes + 6 * 40;
    constexpr int n = (kCtaSmemTarget - fixed) / Sh::kStageBytes;
    return n < 2 ? 2 : (n > 8 ? 8 : n);
}

// CUDA-core consumers: 32-token tiles, four consumer warps, two merge buffers.
template <typename Elem, int D, int G>
struct SimtCfg {
    using Cons = SimtConsumer<Elem, D, G, 32, 4>;
    static constexpr int MB = 2;
    static constexpr int STAGES = ring_stages<Cons, MB>();
};

// Tensor-core consumers: 64-token tiles (one 16-token slab per consumer
// warp); one merge buffer (a unit spans several tiles, the epilogue empties
// the buffer well within one), so that a third stage fits.
template <int D, int G>
struct MmaCfg {
    using Cons = MmaConsumer<D, G, 64, 4>;
    static constexpr int MB = 1;
    static constexpr int STAGES = ring_stages<Cons, MB>();
};

// Tensor-core consumers over quantised rows (E4M3 codes, D + 16-byte rows,
// or E2M1 codes, D/2 + 16-byte rows; each with its fp32 scale): 64-token
// tiles, one merge buffer.
template <int D, int G, bool kFp4>
struct QuantCfg {
    using Cons = QuantMmaConsumer<D, G, 64, 4, kFp4>;
    static constexpr int MB = 1;
    static constexpr int STAGES = ring_stages<Cons, MB>();
};

// Lookahead of the schedulers, per SM: about 5 us of one SM's share of HBM
// bandwidth (~45 KB per us).
constexpr int kLookBytesPerSm = 224 * 1024;

// Per-device launch facts of one kernel instantiation: the shared-memory
// attribute is set and the persistent grid sized once per device.
struct DeviceFacts {
    std::mutex mu;
    int ctas[64] = {};    // persistent CTAs per device (0 = not set up yet)
    int per_sm[64] = {};  // of them resident on one SM
};

template <class Cons, int STAGES, int MB, int MODE>
cudaError_t launch_kernel(const AttendParams& p, const CUtensorMap* kmap, const CUtensorMap* vmap,
                          cudaStream_t stream) {
    using Sh = KernelShape<Cons, STAGES, MB>;
    static_assert(Sh::kSmemAlloc <= 227 * 1024, "shared memory of one CTA");
    auto kern = attend_kernel<Cons, STAGES, MB, MODE>;
    constexpr int kThreads = Sh::kThreads;
    static DeviceFacts facts;
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if (dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
    int ctas, per_sm;
    {
        std::lock_guard<std::mutex> lock(facts.mu);
        if (!facts.ctas[dev]) {
            e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                     Sh::kSmemAlloc);
            if (e != cudaSuccess) return e;
            int resident = 0, nsm = 0;
            e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&resident, kern, kThreads,
                                                              Sh::kSmemAlloc);
            if (e != cudaSuccess) return e;
            e = cudaDeviceGetAttribute(&nsm, cudaDevAttrMultiProcessorCount, dev);
            if (e != cudaSuccess) return e;
            facts.per_sm[dev] = resident < 1 ? 1 : resident;
            facts.ctas[dev] = facts.per_sm[dev] * (nsm < 1 ? 1 : nsm);
        }
        ctas = facts.ctas[dev];
        per_sm = facts.per_sm[dev];
    }
    // The SM's lookahead split between the CTAs that share it, at least two tiles.
    AttendParams q = p;
    const int bytes_per_token = 2 * Cons::kRowBytes;
    q.look = (kLookBytesPerSm / per_sm) / bytes_per_token;
    if (q.look < 2 * p.tile) q.look = 2 * p.tile;
    const int grid = p.units < ctas ? p.units : ctas;
    return launch_pdl(kern, dim3(grid), dim3(kThreads), Sh::kSmemAlloc, stream, q, *kmap, *vmap);
}

template <class C>
cudaError_t launch_cfg(int mode, const AttendParams& p, const CUtensorMap* kmap,
                       const CUtensorMap* vmap, cudaStream_t stream) {
    using Cons = typename C::Cons;
    switch (mode) {
        case kModeMasked:
            return launch_kernel<Cons, C::STAGES, C::MB, kModeMasked>(p, kmap, vmap, stream);
        case kModePaged:
            return launch_kernel<Cons, C::STAGES, C::MB, kModePaged>(p, kmap, vmap, stream);
        case kModeIndexed:
            return launch_kernel<Cons, C::STAGES, C::MB, kModeIndexed>(p, kmap, vmap, stream);
    }
    return cudaErrorInvalidValue;
}

template <typename Elem, int D, int G>
cudaError_t launch_simt(int mode, const AttendParams& p, const CUtensorMap* kmap,
                        const CUtensorMap* vmap, cudaStream_t stream) {
    return launch_cfg<SimtCfg<Elem, D, G>>(mode, p, kmap, vmap, stream);
}

template <int D, int G>
cudaError_t launch_mma(int mode, const AttendParams& p, const CUtensorMap* kmap,
                       const CUtensorMap* vmap, cudaStream_t stream) {
    return launch_cfg<MmaCfg<D, G>>(mode, p, kmap, vmap, stream);
}

// Quantised rows in every mode: the static buffer's tiles arrive by bulk
// copies, the paged cache's by 3-D TMA boxes of whole rows (byte tensor
// maps), index lists by cp.async row gathers.
template <int D, int G, bool kFp4>
cudaError_t launch_quant(int mode, const AttendParams& p, const CUtensorMap* kmap,
                         const CUtensorMap* vmap, cudaStream_t stream) {
    return launch_cfg<QuantCfg<D, G, kFp4>>(mode, p, kmap, vmap, stream);
}

}  // namespace kvd
