// attend_quant.cuh -- instantiations and launch of the attention kernels over
// quantised K/V rows (q and out bf16): the persistent split kernel (static
// buffer, paged cache or index lists) and the one-launch cluster kernel
// (static buffer), tensor-core consumers for every group width up to 8 query
// heads per kv head.  kFp4 selects E2M1 rows (D/2 code bytes)
// over E4M3 rows (D code bytes); both carry a 16-byte scale field.
// Included by one translation unit per code format.
#pragma once

#include "attend_inst.cuh"
#include "attend_small_launch.cuh"

namespace kvd {

template <bool kFp4>
cudaError_t launch_attend_quant(int D, int G, int mode, const AttendParams& p,
                                const CUtensorMap* kmap, const CUtensorMap* vmap,
                                cudaStream_t stream) {
    if (D == 128) {
        switch (G) {
            case 1: return launch_quant<128, 1, kFp4>(mode, p, kmap, vmap, stream);
            case 2: return launch_quant<128, 2, kFp4>(mode, p, kmap, vmap, stream);
            case 4: return launch_quant<128, 4, kFp4>(mode, p, kmap, vmap, stream);
            case 8: return launch_quant<128, 8, kFp4>(mode, p, kmap, vmap, stream);
        }
    } else if (D == 64) {
        switch (G) {
            case 1: return launch_quant<64, 1, kFp4>(mode, p, kmap, vmap, stream);
            case 2: return launch_quant<64, 2, kFp4>(mode, p, kmap, vmap, stream);
            case 4: return launch_quant<64, 4, kFp4>(mode, p, kmap, vmap, stream);
            case 8: return launch_quant<64, 8, kFp4>(mode, p, kmap, vmap, stream);
        }
    }
    return cudaErrorInvalidValue;
}

template <bool kFp4>
int small_shared_bytes_quant(int D, int G, int chunk, int slots, int nwg) {
    const int T = 64;
    const int row = (kFp4 ? D / 2 : D) + 16;
    const SmallLayout L =
        SmallLayout::make((chunk + T - 1) / T, T * row, T, D, G, 4 * nwg, 2, slots);
    return L.bytes + 1024;
}

template <bool kFp4>
cudaError_t launch_attend_small_quant(int D, int G, const AttendParams& p, int S, int rows,
                                      cudaStream_t stream) {
    CUtensorMap none;
    std::memset(&none, 0, sizeof none);
    if (D == 128) {
        switch (G) {
            case 1: return launch_small_cfg<QuantMmaConsumer<128, 1, 64, 4, kFp4>>(p, S, rows, &none, &none, stream);
            case 2: return launch_small_cfg<QuantMmaConsumer<128, 2, 64, 4, kFp4>>(p, S, rows, &none, &none, stream);
            case 4: return launch_small_cfg<QuantMmaConsumer<128, 4, 64, 4, kFp4>>(p, S, rows, &none, &none, stream);
            case 8: return launch_small_cfg<QuantMmaConsumer<128, 8, 64, 4, kFp4>>(p, S, rows, &none, &none, stream);
        }
    } else if (D == 64) {
        switch (G) {
            case 1: return launch_small_cfg<QuantMmaConsumer<64, 1, 64, 4, kFp4>>(p, S, rows, &none, &none, stream);
            case 2: return launch_small_cfg<QuantMmaConsumer<64, 2, 64, 4, kFp4>>(p, S, rows, &none, &none, stream);
            case 4: return launch_small_cfg<QuantMmaConsumer<64, 4, 64, 4, kFp4>>(p, S, rows, &none, &none, stream);
            case 8: return launch_small_cfg<QuantMmaConsumer<64, 8, 64, 4, kFp4>>(p, S, rows, &none, &none, stream);
        }
    }
    return cudaErrorInvalidValue;
}

}  // namespace kvd
