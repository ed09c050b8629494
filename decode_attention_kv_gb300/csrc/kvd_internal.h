// kvd_internal.h -- host-side declarations shared by the libkvd translation
// units (launchers of the templated kernels).  Not part of the C ABI.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "../../include/kvd.h"

namespace kvd {

struct AttendParams;

// Tile geometry of the attention kernel for one element type / head_dim.
struct AttendGeom {
    int tile_max;     // T: tokens per ring stage (static buffer tile)
    int stages;
    int consumer_warps;
    int smem_bytes;   // dynamic shared memory per CTA
};

// Geometry of the instantiation the launchers use (G does not change it).
AttendGeom attend_geom(kvd_dtype dt, int D);

// Launch the split kernel: grid (S, Hkv * HG, rows).  `G` is the compile-time
// group width (1, 2, 4 or 8).  Returns the launch error.
cudaError_t launch_attend_split(kvd_dtype dt, int D, int G, bool paged, const AttendParams& p,
                                const CUtensorMap* kmap, const CUtensorMap* vmap, dim3 grid,
                                cudaStream_t stream);

// Sets the message kvd_last_error() returns on this thread.
void set_last_error(const char* msg);

cudaError_t launch_combine(const float* part_o, const float* part_lse, void* out,
                           float* lse_out, int R, int S, int D, kvd_dtype out_dt,
                           cudaStream_t stream);

cudaError_t launch_append(void* k_cache, void* v_cache, const void* k_new, const void* v_new,
                          const int32_t* pos, uint8_t* mask, int B, int Hkv, int C, int row_bytes,
                          int32_t* dev_status, cudaStream_t stream);

cudaError_t launch_gather(const void* key_cache, const void* value_cache,
                          const int32_t* block_tables, const int32_t* seq_lens,
                          const int32_t* seq_offset, void* key_out, void* value_out, int Q,
                          int NB, int BS, int cols, long long krow_bytes, long long vrow_bytes,
                          int total_tokens, int32_t* dev_status, cudaStream_t stream);

}  // namespace kvd
