// attend_small.cu -- instantiations and launch of the small-launch attention
// kernel (one CTA per (row, split), the row's splits in one cluster).
#include <cstring>
#include <mutex>

#include "attend_small.cuh"
#include "kvd_internal.h"

namespace kvd {

namespace {

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

template <typename Elem, int D>
cudaError_t launch_small_d(int G, bool mma, const AttendParams& p, int S, int rows,
                           const CUtensorMap* kmap, const CUtensorMap* vmap, cudaStream_t s) {
    if constexpr (sizeof(Elem) == 2) {
        if (mma) {
            switch (G) {
                case 1: return launch_small_cfg<MmaConsumer<D, 1, 64, 4>>(p, S, rows, kmap, vmap, s);
                case 2: return launch_small_cfg<MmaConsumer<D, 2, 64, 4>>(p, S, rows, kmap, vmap, s);
                case 4: return launch_small_cfg<MmaConsumer<D, 4, 64, 4>>(p, S, rows, kmap, vmap, s);
                case 8: return launch_small_cfg<MmaConsumer<D, 8, 64, 4>>(p, S, rows, kmap, vmap, s);
            }
            return cudaErrorInvalidValue;
        }
    }
    switch (G) {
        case 1: return launch_small_cfg<SimtConsumer<Elem, D, 1, 32, 4>>(p, S, rows, kmap, vmap, s);
        case 2: return launch_small_cfg<SimtConsumer<Elem, D, 2, 32, 4>>(p, S, rows, kmap, vmap, s);
    }
    if constexpr (sizeof(Elem) == 4) {
        if (G == 4) return launch_small_cfg<SimtConsumer<Elem, D, 4, 32, 4>>(p, S, rows, kmap, vmap, s);
        if (G == 8) return launch_small_cfg<SimtConsumer<Elem, D, 8, 32, 4>>(p, S, rows, kmap, vmap, s);
    }
    return cudaErrorInvalidValue;
}

}  // namespace

int small_shared_bytes_fp8(int D, int G, int chunk, int slots, int nwg) {
    const int T = 64;
    const SmallLayout L =
        SmallLayout::make((chunk + T - 1) / T, T * (D + 16), T, D, G, 4 * nwg, 2, slots);
    return L.bytes + 1024;
}

cudaError_t launch_attend_small_fp8(int D, int G, const AttendParams& p, int S, int rows,
                                    cudaStream_t stream) {
    CUtensorMap none;
    std::memset(&none, 0, sizeof none);
    if (D == 128) {
        switch (G) {
            case 1: return launch_small_cfg<Fp8MmaConsumer<128, 1, 64, 4>>(p, S, rows, &none, &none, stream);
            case 2: return launch_small_cfg<Fp8MmaConsumer<128, 2, 64, 4>>(p, S, rows, &none, &none, stream);
            case 4: return launch_small_cfg<Fp8MmaConsumer<128, 4, 64, 4>>(p, S, rows, &none, &none, stream);
            case 8: return launch_small_cfg<Fp8MmaConsumer<128, 8, 64, 4>>(p, S, rows, &none, &none, stream);
        }
    } else if (D == 64) {
        switch (G) {
            case 1: return launch_small_cfg<Fp8MmaConsumer<64, 1, 64, 4>>(p, S, rows, &none, &none, stream);
            case 2: return launch_small_cfg<Fp8MmaConsumer<64, 2, 64, 4>>(p, S, rows, &none, &none, stream);
            case 4: return launch_small_cfg<Fp8MmaConsumer<64, 4, 64, 4>>(p, S, rows, &none, &none, stream);
            case 8: return launch_small_cfg<Fp8MmaConsumer<64, 8, 64, 4>>(p, S, rows, &none, &none, stream);
        }
    }
    return cudaErrorInvalidValue;
}

int small_shared_bytes(kvd_dtype dt, int D, int G, int chunk, int slots, int nwg) {
    const bool mma = small_uses_mma(dt, G);
    const int T = mma ? 64 : 32;
    const int e = dt == KVD_BF16 ? 2 : 4;
    const int tile_bytes = T * D * e;
    const SmallLayout L =
        SmallLayout::make((chunk + T - 1) / T, tile_bytes, T, D, G, 4 * nwg, e, slots);
    return L.bytes + 1024;
}

cudaError_t launch_attend_small(kvd_dtype dt, int D, int G, const AttendParams& p, int S, int rows,
                                const CUtensorMap* kmap, const CUtensorMap* vmap,
                                cudaStream_t stream) {
    const bool mma = small_uses_mma(dt, G);
    if (dt == KVD_BF16) {
        if (D == 128) return launch_small_d<__nv_bfloat16, 128>(G, mma, p, S, rows, kmap, vmap, stream);
        if (D == 64) return launch_small_d<__nv_bfloat16, 64>(G, mma, p, S, rows, kmap, vmap, stream);
    } else {
        if (D == 128) return launch_small_d<float, 128>(G, mma, p, S, rows, kmap, vmap, stream);
        if (D == 64) return launch_small_d<float, 64>(G, mma, p, S, rows, kmap, vmap, stream);
    }
    return cudaErrorInvalidValue;
}

}  // namespace kvd
