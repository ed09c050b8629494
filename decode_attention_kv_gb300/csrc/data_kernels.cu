// data_kernels.cu -- the log-sum-exp combine, the KV append and the paged
// gather kernels, with their launchers.
#include "kvd_device.cuh"
#include "kvd_internal.h"

namespace kvd {

// ------------------------------------------------------------------ combine
// One CTA per output row.  Merges S partial rows, each normalised over its own
// key range, by their log-sum-exp ("Intel NPU running LLMs", Part 3, Flash
// SDPA path: tiles merged exactly through running max and sum).  The row's
// log-sum-exps are reduced first; then groups of threads split the S partial
// rows between them (a thread owns one float4 of the row) so that the loads
// of many partial rows are in flight at once; shared memory sums the groups.
constexpr int kCombineThreads = 128;

__device__ __forceinline__ float block_reduce(float x, bool is_max, float* red) {
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) {
        const float o = __shfl_xor_sync(0xffffffffu, x, off);
        x = is_max ? fmaxf(x, o) : x + o;
    }
    __syncthreads();  // red[] may still be read from a previous reduction
    if (lane == 0) red[warp] = x;
    __syncthreads();
    x = red[0];
#pragma unroll
    for (int w = 1; w < kCombineThreads / 32; ++w) x = is_max ? fmaxf(x, red[w]) : x + red[w];
    return x;
}

template <typename Out>
__global__ void __launch_bounds__(kCombineThreads)
combine_kernel(const float* __restrict__ part_o, const float* __restrict__ part_lse,
               Out* __restrict__ out, float* __restrict__ lse_out, int R, int S, int D) {
    __shared__ float red[kCombineThreads / 32];
    __shared__ float4 acc_sm[kCombineThreads];
    pdl_launch_dependents();
    pdl_wait();
    const int row = blockIdx.x, tid = threadIdx.x;
    const float* ls = part_lse + (size_t)row * S;
    float M = -INFINITY;
    for (int s = tid; s < S; s += kCombineThreads) M = fmaxf(M, ls[s]);
    M = block_reduce(M, true, red);
    float sum = 0.f;
    if (M != -INFINITY)
        for (int s = tid; s < S; s += kCombineThreads) sum += fast_exp2((ls[s] - M) * kLog2e);
    sum = block_reduce(sum, false, red);

    const int nv = D / 4;                                    // float4 per row
    const int groups = nv >= kCombineThreads ? 1 : kCombineThreads / nv;
    const int g = tid / nv, v = tid % nv;                    // (g only meaningful if groups > 1)
    float4 a0 = make_float4(0.f, 0.f, 0.f, 0.f), a1 = a0;    // D <= 1024: two float4 at most
    const bool active = groups > 1 ? g < groups : true;
    const int gg = groups > 1 ? g : 0;
    const int v0 = groups > 1 ? v : tid;
    if (M != -INFINITY && active) {
        const float inv = 1.f / sum;
        const float4* po = reinterpret_cast<const float4*>(part_o) + (size_t)row * S * nv;
#pragma unroll 8
        for (int s = gg; s < S; s += groups) {
            const float lsv = ls[s];
            if (lsv == -INFINITY) continue;  // empty range: its row is not read
            const float w = fast_exp2((lsv - M) * kLog2e) * inv;
            const float4* src = po + (size_t)s * nv;
            if (v0 < nv) {
                const float4 x = src[v0];
                a0.x = fmaf(w, x.x, a0.x);
                a0.y = fmaf(w, x.y, a0.y);
                a0.z = fmaf(w, x.z, a0.z);
                a0.w = fmaf(w, x.w, a0.w);
            }
            if (v0 + kCombineThreads < nv) {
                const float4 x = src[v0 + kCombineThreads];
                a1.x = fmaf(w, x.x, a1.x);
                a1.y = fmaf(w, x.y, a1.y);
                a1.z = fmaf(w, x.z, a1.z);
                a1.w = fmaf(w, x.w, a1.w);
            }
        }
    }
    if (groups > 1) {
        acc_sm[tid] = a0;
        __syncthreads();
        if (g == 0) {
            for (int k = 1; k < groups; ++k) {
                const float4 x = acc_sm[k * nv + v];
                a0.x += x.x;
                a0.y += x.y;
                a0.z += x.z;
                a0.w += x.w;
            }
        }
    }
    if (groups == 1 || g == 0) {
        const size_t o = (size_t)row * D;
        if (v0 < nv) {
            ElemTraits<Out>::store(out, o + 4 * v0, a0.x);
            ElemTraits<Out>::store(out, o + 4 * v0 + 1, a0.y);
            ElemTraits<Out>::store(out, o + 4 * v0 + 2, a0.z);
            ElemTraits<Out>::store(out, o + 4 * v0 + 3, a0.w);
        }
        if (v0 + kCombineThreads < nv) {
            const size_t o1 = o + 4 * (v0 + kCombineThreads);
            ElemTraits<Out>::store(out, o1, a1.x);
            ElemTraits<Out>::store(out, o1 + 1, a1.y);
            ElemTraits<Out>::store(out, o1 + 2, a1.z);
            ElemTraits<Out>::store(out, o1 + 3, a1.w);
        }
    }
    if (tid == 0 && lse_out) lse_out[row] = M != -INFINITY ? M + logf(sum) : -INFINITY;
}

cudaError_t launch_combine(const float* part_o, const float* part_lse, void* out,
                           float* lse_out, int R, int S, int D, kvd_dtype out_dt,
                           cudaStream_t stream) {
    if (out_dt == KVD_BF16)
        return launch_pdl(combine_kernel<__nv_bfloat16>, dim3(R), dim3(kCombineThreads), 0, stream,
                          part_o, part_lse, static_cast<__nv_bfloat16*>(out), lse_out, R, S, D);
    return launch_pdl(combine_kernel<float>, dim3(R), dim3(kCombineThreads), 0, stream, part_o,
                      part_lse, static_cast<float*>(out), lse_out, R, S, D);
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
    pdl_launch_dependents();
    pdl_wait();
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
    return launch_pdl(append_kernel, grid, dim3(256), 0, stream, static_cast<unsigned char*>(k_cache),
                      static_cast<unsigned char*>(v_cache),
                      static_cast<const unsigned char*>(k_new),
                      static_cast<const unsigned char*>(v_new), pos, mask, Hkv, C, row_bytes,
                      dev_status);
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
    pdl_launch_dependents();
    pdl_wait();
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
        return launch_pdl(gather_kernel<uint4>, grid, dim3(256), 0, stream, kc, vc, block_tables,
                          seq_lens, seq_offset, ko, vo, NB, BS, cols, krow, vrow, total_tokens,
                          dev_status);
    if (krow % 4 == 0 && vrow % 4 == 0)
        return launch_pdl(gather_kernel<unsigned int>, grid, dim3(256), 0, stream, kc, vc,
                          block_tables, seq_lens, seq_offset, ko, vo, NB, BS, cols, krow, vrow,
                          total_tokens, dev_status);
    return launch_pdl(gather_kernel<unsigned short>, grid, dim3(256), 0, stream, kc, vc,
                      block_tables, seq_lens, seq_offset, ko, vo, NB, BS, cols, krow, vrow,
                      total_tokens, dev_status);
}

}  // namespace kvd
