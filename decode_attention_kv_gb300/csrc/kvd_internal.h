// kvd_internal.h -- host-side declarations shared by the libkvd translation
// units (launchers of the templated kernels).  Not part of the C ABI.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "../../include/kvd.h"

namespace kvd {

struct AttendParams;

// Launch with programmatic stream serialisation (the kernel may start while
// the previous kernel on the stream drains; see pdl_wait in kvd_device.cuh).
template <typename... KArgs, typename... Args>
inline cudaError_t launch_pdl(void (*kern)(KArgs...), dim3 grid, dim3 block, size_t smem,
                              cudaStream_t stream, Args... args) {
    cudaLaunchConfig_t cfg{};
    cfg.gridDim = grid;
    cfg.blockDim = block;
    cfg.dynamicSmemBytes = smem;
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, kern, args...);
}

// Tile geometry of the attention kernel for one element type / head_dim /
// group width.
struct AttendGeom {
    int tile_max;     // T: tokens per ring stage (static buffer tile)
    int stages;
    int consumer_warps;
    int smem_bytes;   // dynamic shared memory per CTA
    bool mma;         // tensor-core consumers; K/V through 128-byte-swizzled TMA boxes
};

// Which kernel serves a group width: bf16 groups of 4 or 8 query heads per kv
// head use the tensor-core consumers, everything else the CUDA-core ones.
inline bool attend_uses_mma(kvd_dtype dt, int G) { return dt == KVD_BF16 && G >= 4; }

// The one-launch cluster kernel (short buffers) uses the tensor-core
// consumers for every bf16 group width: there the consumers' latency, not
// HBM, bounds the launch, and 16 mma per 16-token slab (unused head columns
// included) finish a split far sooner than per-token shuffle reductions.
inline bool small_uses_mma(kvd_dtype dt, int G) { (void)G; return dt == KVD_BF16; }

// Sets the message kvd_last_error() returns on this thread.
void set_last_error(const char* msg);

// part_o [R, S, D] / part_lse [R, S]; or, with gathered_stride > 0, split s's
// rows at part_o + s * gathered_stride ([R, D]) and its log-sum-exps at
// part_lse + s * gathered_stride ([R]).
cudaError_t launch_combine(const float* part_o, const float* part_lse, void* out,
                           float* lse_out, int R, int S, int D, kvd_dtype out_dt,
                           cudaStream_t stream, long long gathered_stride = 0);

cudaError_t launch_copy_prefix(const void* const* k_src, const void* const* v_src,
                               void* const* k_dst, void* const* v_dst, uint8_t* const* masks,
                               const int32_t* n, int L, int B, int Hkv, int C_src, int C_dst,
                               int row_bytes, int32_t* dev_status, cudaStream_t stream);

cudaError_t launch_append(void* k_cache, void* v_cache, const void* k_new, const void* v_new,
                          const int32_t* pos, uint8_t* mask, int B, int Hkv, int C, int row_bytes,
                          int32_t* dev_status, cudaStream_t stream);

cudaError_t launch_append_paged(void* key_cache, void* value_cache, const void* k_new,
                                const void* v_new, const int32_t* block_tables,
                                const int32_t* seq_offset, const int32_t* pos, int Q, int NB,
                                int BS, int cols, int row_bytes, int32_t* dev_status,
                                cudaStream_t stream);

// Quantising appends: into the static buffer [B, Hkv, C, RB], or, with
// block_tables, token pos[b] of sequence b of the paged cache [NB, BS, Hkv, RB]
// (C unused then).
cudaError_t launch_append_fp8(void* k_cache, void* v_cache, const void* k_new, const void* v_new,
                              const int32_t* pos, uint8_t* mask, int B, int Hkv, int C, int D,
                              kvd_dtype in_dt, int32_t* dev_status, cudaStream_t stream,
                              const int32_t* block_tables = nullptr,
                              const int32_t* seq_offset = nullptr, int NB = 0, int BS = 0,
                              int cols = 0);

cudaError_t launch_append_fp4(void* k_cache, void* v_cache, const void* k_new, const void* v_new,
                              const int32_t* pos, uint8_t* mask, int B, int Hkv, int C, int D,
                              kvd_dtype in_dt, int32_t* dev_status, cudaStream_t stream,
                              const int32_t* block_tables = nullptr,
                              const int32_t* seq_offset = nullptr, int NB = 0, int BS = 0,
                              int cols = 0);

cudaError_t launch_gather(const void* key_cache, const void* value_cache,
                          const int32_t* block_tables, const int32_t* seq_lens,
                          const int32_t* seq_offset, void* key_out, void* value_out, int Q,
                          int NB, int BS, int cols, long long krow_bytes, long long vrow_bytes,
                          int total_tokens, int32_t* dev_status, cudaStream_t stream);

}  // namespace kvd
