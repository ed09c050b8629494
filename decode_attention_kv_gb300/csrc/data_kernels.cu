// data_kernels.cu -- the log-sum-exp combine, the KV append and the paged
// gather kernels, with their launchers.
#include "kvd_device.cuh"
#include "kvd_internal.h"

namespace kvd {

// ------------------------------------------------------------------ combine
// One warp per output row.  Merges S partial rows, each normalised over its
// own key range, by their log-sum-exp ("Intel NPU running LLMs", Part 3,
// Flash SDPA path: tiles merged exactly through running max and sum).
constexpr int kCombineWarps = 4;
constexpr int kCombineMaxVec = 8;  // float4 per lane: D <= 1024

template <typename Out>
__global__ void __launch_bounds__(kCombineWarps * 32)
combine_kernel(const float* __restrict__ part_o, const float* __restrict__ part_lse,
               Out* __restrict__ out, float* __restrict__ lse_out, int R, int S, int D) {
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int row = blockIdx.x * kCombineWarps + warp;
    if (row >= R) return;
    const float* ls = part_lse + (size_t)row * S;
    float M = -INFINITY;
    for (int s = lane; s < S; s += 32) M = fmaxf(M, ls[s]);
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) M = fmaxf(M, __shfl_xor_sync(0xffffffffu, M, off));
    const int nv = D / 4;
    float4 acc[kCombineMaxVec];
#pragma unroll
    for (int k = 0; k < kCombineMaxVec; ++k) acc[k] = make_float4(0.f, 0.f, 0.f, 0.f);
    float lse = -INFINITY;
    if (M != -INFINITY) {
        float sum = 0.f;
        for (int s = lane; s < S; s += 32) sum += fast_exp2((ls[s] - M) * kLog2e);
#pragma unroll
        for (int off = 16; off > 0; off >>= 1) sum += __shfl_xor_sync(0xffffffffu, sum, off);
        const float inv = 1.f / sum;
        lse = M + logf(sum);
        const float4* po = reinterpret_cast<const float4*>(part_o + (size_t)row * S * D);
        for (int s = 0; s < S; ++s) {
            const float lsv = ls[s];
            if (lsv == -INFINITY) continue;  // empty range: its row is not read
            const float w = fast_exp2((lsv - M) * kLog2e) * inv;
#pragma unroll
            for (int k = 0; k < kCombineMaxVec; ++k) {
                const int vi = lane + 32 * k;
                if (vi < nv) {
                    const float4 x = po[(size_t)s * nv + vi];
                    acc[k].x = fmaf(w, x.x, acc[k].x);
                    acc[k].y = fmaf(w, x.y, acc[k].y);
                    acc[k].z = fmaf(w, x.z, acc[k].z);
                    acc[k].w = fmaf(w, x.w, acc[k].w);
                }
            }
        }
    }
#pragma unroll
    for (int k = 0; k < kCombineMaxVec; ++k) {
        const int vi = lane + 32 * k;
        if (vi < nv) {
            const size_t o = (size_t)row * D + 4 * vi;
            ElemTraits<Out>::store(out, o, acc[k].x);
            ElemTraits<Out>::store(out, o + 1, acc[k].y);
            ElemTraits<Out>::store(out, o + 2, acc[k].z);
            ElemTraits<Out>::store(out, o + 3, acc[k].w);
        }
    }
    if (lane == 0 && lse_out) lse_out[row] = lse;
}

cudaError_t launch_combine(const float* part_o, const float* part_lse, void* out,
                           float* lse_out, int R, int S, int D, kvd_dtype out_dt,
                           cudaStream_t stream) {
    const dim3 grid((R + kCombineWarps - 1) / kCombineWarps);
    if (out_dt == KVD_BF16)
        combine_kernel<__nv_bfloat16><<<grid, kCombineWarps * 32, 0, stream>>>(
            part_o, part_lse, static_cast<__nv_bfloat16*>(out), lse_out, R, S, D);
    else
        combine_kernel<float><<<grid, kCombineWarps * 32, 0, stream>>>(
            part_o, part_lse, static_cast<float*>(out), lse_out, R, S, D);
    return cudaGetLastError();
}

// ------------------------------------------------------------------- append
// update_kvcache_for ("Intel NPU running LLMs", Part 2): the new token's K and
// V rows go to slot pos[b] of every kv head; the mask slot is set.  One
// 16-byte vector per thread; grid (vectors / 256, B).
__global__ void __launch_bounds__(256)
append_kernel(unsigned char* __restrict__ kc, unsigned char* __restrict__ vc,
              const unsigned char* __restrict__ kn, const unsigned char* __restrict__ vn,
              const int32_t* __restrict__ pos, uint8_t* __restrict__ mask, int Hkv, int C,
              int row_bytes, int32_t* dev_status) {
    const int b = blockIdx.y;
    const int p = pos[b];
    if (p < 0 || p >= C) {
        if (blockIdx.x == 0 && threadIdx.x == 0) report(dev_status, KVD_DEV_POS_RANGE);
        return;
    }
    const int vpr = row_bytes / 16;
    const int v = blockIdx.x * blockDim.x + threadIdx.x;
    if (v < Hkv * vpr) {
        const int h = v / vpr, j = v % vpr;
        const size_t src = ((size_t)b * Hkv + h) * row_bytes + (size_t)j * 16;
        const size_t dst = (((size_t)b * Hkv + h) * C + p) * row_bytes + (size_t)j * 16;
        const uint4 kx = *reinterpret_cast<const uint4*>(kn + src);
        const uint4 vx = *reinterpret_cast<const uint4*>(vn + src);
        *reinterpret_cast<uint4*>(kc + dst) = kx;
        *reinterpret_cast<uint4*>(vc + dst) = vx;
    }
    if (mask && blockIdx.x == 0 && threadIdx.x == 0) mask[(size_t)b * C + p] = 1;
}

cudaError_t launch_append(void* k_cache, void* v_cache, const void* k_new, const void* v_new,
                          const int32_t* pos, uint8_t* mask, int B, int Hkv, int C,
                          int row_bytes, int32_t* dev_status, cudaStream_t stream) {
    const int nvec = Hkv * (row_bytes / 16);
    const dim3 grid((nvec + 255) / 256, B);
    append_kernel<<<grid, 256, 0, stream>>>(
        static_cast<unsigned char*>(k_cache), static_cast<unsigned char*>(v_cache),
        static_cast<const unsigned char*>(k_new), static_cast<const unsigned char*>(v_new), pos,
        mask, Hkv, C, row_bytes, dev_status);
    return cudaGetLastError();
}

// ------------------------------------------------------------------- gather
// gather_pa_kv_cache, Norm/ND branch ("PyPTO 实现 AscendC GatherPaKvCache",
// 3.2): CTA q * cols + j copies the valid rows of logical block j of
// sequence q.
// The rows of one physical block are contiguous in the cache and land on
// consecutive output rows, so each CTA moves one contiguous byte range per
// cache; VecT is the widest vector dividing the row sizes.
template <typename VecT>
__device__ __forceinline__ void copy_range(unsigned char* __restrict__ dst,
                                           const unsigned char* __restrict__ src,
                                           long long bytes) {
    const long long n = bytes / (long long)sizeof(VecT);
    const VecT* s = reinterpret_cast<const VecT*>(src);
    VecT* d = reinterpret_cast<VecT*>(dst);
    constexpr int U = 8;  // independent loads in flight per thread
    long long i = threadIdx.x;
    const long long stride = blockDim.x;
    for (; i + (U - 1) * stride < n; i += U * stride) {
        VecT x[U];
#pragma unroll
        for (int u = 0; u < U; ++u) x[u] = __ldcs(s + i + u * stride);
#pragma unroll
        for (int u = 0; u < U; ++u) __stcs(d + i + u * stride, x[u]);
    }
    for (; i < n; i += stride) __stcs(d + i, __ldcs(s + i));
}

__device__ __forceinline__ void copy_range_u16(unsigned char* dst, const unsigned char* src,
                                               long long bytes) {
    const long long n = bytes / 2;
    const unsigned short* s = reinterpret_cast<const unsigned short*>(src);
    unsigned short* d = reinterpret_cast<unsigned short*>(dst);
    for (long long i = threadIdx.x; i < n; i += blockDim.x) d[i] = s[i];
}

template <typename VecT>
__global__ void __launch_bounds__(256)
gather_kernel(const unsigned char* __restrict__ kc, const unsigned char* __restrict__ vc,
              const int32_t* __restrict__ bt, const int32_t* __restrict__ seq_lens,
              const int32_t* __restrict__ seq_offset, unsigned char* __restrict__ ko,
              unsigned char* __restrict__ vo, int NB, int BS, int cols, long long krow,
              long long vrow, int total_tokens, int32_t* dev_status) {
    const int q = blockIdx.x / cols, j = blockIdx.x % cols;
    const int s0 = seq_lens[q], s1 = seq_lens[q + 1];
    const int off = seq_offset ? seq_offset[q] : 0;
    // Checks in the order of the page's constraints (section 3.3); a sequence
    // that fails one is skipped whole.  A cumsum that does not start at 0 is
    // reported but the (well-defined) differences are still used.
    uint32_t bad = (q == 0 && s0 != 0) ? KVD_DEV_SEQLENS : 0u;
    bool skip = false;
    const int len = s1 - s0;
    const int nblk = len > 0 ? (len + BS - 1) / BS : 0;
    if (s1 < s0 || s0 < 0 || s1 > total_tokens) {
        bad |= KVD_DEV_SEQLENS;
        skip = true;
    } else if (off < 0 || off % BS != 0) {
        bad |= KVD_DEV_SEQ_OFFSET;
        skip = true;
    } else if (off / BS + nblk > cols) {
        bad |= KVD_DEV_TABLE_COLS;
        skip = true;
    }
    if (bad && j == 0 && threadIdx.x == 0) report(dev_status, bad);
    if (skip || j >= nblk) return;
    const int first_col = off / BS;
    const int phys = bt[(size_t)q * cols + first_col + j];
    if (phys < 0 || phys >= NB) {
        if (threadIdx.x == 0) report(dev_status, KVD_DEV_BLOCK_RANGE);
        return;
    }
    const int ntok = min(BS, len - j * BS);
    const long long src_row = (long long)phys * BS, dst_row = (long long)s0 + (long long)j * BS;
    if constexpr (sizeof(VecT) >= 4) {
        copy_range<VecT>(ko + dst_row * krow, kc + src_row * krow, ntok * krow);
        copy_range<VecT>(vo + dst_row * vrow, vc + src_row * vrow, ntok * vrow);
    } else {
        copy_range_u16(ko + dst_row * krow, kc + src_row * krow, ntok * krow);
        copy_range_u16(vo + dst_row * vrow, vc + src_row * vrow, ntok * vrow);
    }
}

cudaError_t launch_gather(const void* key_cache, const void* value_cache,
                          const int32_t* block_tables, const int32_t* seq_lens,
                          const int32_t* seq_offset, void* key_out, void* value_out, int Q,
                          int NB, int BS, int cols, long long krow, long long vrow,
                          int total_tokens, int32_t* dev_status, cudaStream_t stream) {
    const dim3 grid((unsigned)((long long)Q * cols));
    auto kc = static_cast<const unsigned char*>(key_cache);
    auto vc = static_cast<const unsigned char*>(value_cache);
    auto ko = static_cast<unsigned char*>(key_out);
    auto vo = static_cast<unsigned char*>(value_out);
    if (krow % 16 == 0 && vrow % 16 == 0)
        gather_kernel<uint4><<<grid, 256, 0, stream>>>(kc, vc, block_tables, seq_lens, seq_offset,
                                                       ko, vo, NB, BS, cols, krow, vrow,
                                                       total_tokens, dev_status);
    else if (krow % 4 == 0 && vrow % 4 == 0)
        gather_kernel<unsigned int><<<grid, 256, 0, stream>>>(kc, vc, block_tables, seq_lens,
                                                              seq_offset, ko, vo, NB, BS, cols,
                                                              krow, vrow, total_tokens, dev_status);
    else
        gather_kernel<unsigned short><<<grid, 256, 0, stream>>>(kc, vc, block_tables, seq_lens,
                                                                seq_offset, ko, vo, NB, BS, cols,
                                                                krow, vrow, total_tokens,
                                                                dev_status);
    return cudaGetLastError();
}

}  // namespace kvd
