// attend_small.cu -- instantiations and launch of the small-launch attention
// kernel (one CTA per (row, split), the row's splits in one cluster).
#include <cstring>
#include <mutex>

#include "attend_small_launch.cuh"

namespace kvd {

namespace {

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
