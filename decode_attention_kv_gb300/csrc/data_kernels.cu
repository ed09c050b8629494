// data_kernels.cu -- the log-sum-exp combine, the KV append and the paged
// gather kernels, with their launchers.
#include <cuda_fp8.h>

#include "kvd_device.cuh"
#include "kvd_internal.h"

namespace kvd {

// ------------------------------------------------------------------ combine
// Merges S partial rows, each normalised over its own key range, by their
// log-sum-exp ("Intel NPU running LLMs", Part 3, Flash SDPA path: tiles merged
// exactly through running max and sum).  An item is (row, slice of 32 * VPL
// dims); a lane owns VPL consecutive dims.  `wpi` warps share an item (more
// when S is large), each taking every wpi-th split with a running max / sum /
// output and a batch of splits' loads in flight (a split with lse = -inf has
// no partial row: its values are loaded and discarded); the item's first
// warp merges the states.  VPL = 2 halves the CTAs when there are many rows.
// Strides (in elements) place the partials: row-major [R, S, D] / [R, S]
// (what the split attention writes), or one block per split of R rows of D
// then the R log-sum-exps (what gathering every range's packed partial one
// after the other gives).
constexpr int kCombineWarps = 8;

struct CombineStrides {
    long long o_row, o_split;      // part_o
    long long lse_row, lse_split;  // part_lse
};
constexpr int kCombineBatch = 8;  // splits per warp with loads in flight

template <int VPL>
struct CombineVec;
template <>
struct CombineVec<1> {
    using T = float;
    __device__ static float zero() { return 0.f; }
    __device__ static void fma(float& a, float c, float e, float x) { a = fmaf(a, c, e * x); }
};
template <>
struct CombineVec<2> {
    using T = float2;
    __device__ static float2 zero() { return make_float2(0.f, 0.f); }
    __device__ static void fma(float2& a, float c, float e, float2 x) {
        a.x = fmaf(a.x, c, e * x.x);
        a.y = fmaf(a.y, c, e * x.y);
    }
};
template <>
struct CombineVec<4> {
    using T = float4;
    __device__ static float4 zero() { return make_float4(0.f, 0.f, 0.f, 0.f); }
    __device__ static void fma(float4& a, float c, float e, float4 x) {
        a.x = fmaf(a.x, c, e * x.x);
        a.y = fmaf(a.y, c, e * x.y);
        a.z = fmaf(a.z, c, e * x.z);
        a.w = fmaf(a.w, c, e * x.w);
    }
};

template <typename Out, int VPL>
__global__ void __launch_bounds__(kCombineWarps * 32)
combine_kernel(const float* __restrict__ part_o, const float* __restrict__ part_lse,
               Out* __restrict__ out, float* __restrict__ lse_out, int R, int S, int D, int wpi,
               CombineStrides st) {
    using Vec = CombineVec<VPL>;
    using T = typename Vec::T;
    __shared__ float sm_m[kCombineWarps], sm_l[kCombineWarps];
    __shared__ T sm_acc[kCombineWarps][32];
    pdl_launch_dependents();
    pdl_wait();
    const int lane = threadIdx.x & 31, w = threadIdx.x >> 5;
    constexpr int kSlice = 32 * VPL;
    const int nslices = (D + kSlice - 1) / kSlice;
    const long long item = (long long)blockIdx.x * (kCombineWarps / wpi) + w / wpi;
    const int sub = w % wpi;
    const bool live = item < (long long)R * nslices;
    const long long row = live ? item / nslices : 0;
    const int d = (int)(item % nslices) * kSlice + VPL * lane;
    const bool has_d = live && d < D;  // D % 4 == 0: a lane's dims are all in or all out
    float m = -INFINITY, l = 0.f;  // m in log2 units
    T acc = Vec::zero();
    if (live) {
        const float* ls = part_lse + row * st.lse_row;
        const float* po = part_o + row * st.o_row;
        for (int s0 = sub; s0 < S; s0 += wpi * kCombineBatch) {
            float lv[kCombineBatch];
            T xv[kCombineBatch];
#pragma unroll
            for (int u = 0; u < kCombineBatch; ++u) {
                const int s = s0 + u * wpi;
                lv[u] = s < S ? ls[(long long)s * st.lse_split] : -INFINITY;
                xv[u] = (s < S && has_d)
                            ? *reinterpret_cast<const T*>(po + (long long)s * st.o_split + d)
                            : Vec::zero();
            }
#pragma unroll
            for (int u = 0; u < kCombineBatch; ++u) {
                if (lv[u] == -INFINITY) continue;
                const float x2 = lv[u] * kLog2e;
                const float mn = fmaxf(m, x2);
                const float c = fast_exp2(m - mn), e = fast_exp2(x2 - mn);
                l = fmaf(l, c, e);
                Vec::fma(acc, c, e, xv[u]);
                m = mn;
            }
        }
    }
    if (lane == 0) {
        sm_m[w] = m;
        sm_l[w] = l;
    }
    sm_acc[w][lane] = acc;
    __syncthreads();
    if (!live || sub != 0) return;
    float M = -INFINITY;
    for (int k = 0; k < wpi; ++k) M = fmaxf(M, sm_m[w + k]);
    float L = 0.f;
    T A = Vec::zero();
    if (M != -INFINITY) {
        for (int k = 0; k < wpi; ++k) {
            const float c = fast_exp2(sm_m[w + k] - M);  // 0 for a warp without a split
            L = fmaf(sm_l[w + k], c, L);
            Vec::fma(A, 1.f, c, sm_acc[w + k][lane]);
        }
    }
    if (has_d) {
        const float inv = L > 0.f ? 1.f / L : 0.f;
        const float* a = reinterpret_cast<const float*>(&A);
#pragma unroll
        for (int v = 0; v < VPL; ++v) ElemTraits<Out>::store(out, (size_t)row * D + d + v, a[v] * inv);
    }
    if (d == 0 && lse_out) lse_out[row] = L > 0.f ? (M + log2f(L)) * kLn2 : -INFINITY;
}

template <int VPL>
cudaError_t launch_combine_vpl(const float* part_o, const float* part_lse, void* out,
                               float* lse_out, int R, int S, int D, kvd_dtype out_dt, int wpi,
                               const CombineStrides& st, cudaStream_t stream) {
    const long long items = (long long)R * ((D + 32 * VPL - 1) / (32 * VPL));
    const long long per_cta = kCombineWarps / wpi;
    const dim3 grid((unsigned)((items + per_cta - 1) / per_cta));
    if (out_dt == KVD_BF16)
        return launch_pdl(combine_kernel<__nv_bfloat16, VPL>, grid, dim3(kCombineWarps * 32), 0,
                          stream, part_o, part_lse, static_cast<__nv_bfloat16*>(out), lse_out, R,
                          S, D, wpi, st);
    return launch_pdl(combine_kernel<float, VPL>, grid, dim3(kCombineWarps * 32), 0, stream, part_o,
                      part_lse, static_cast<float*>(out), lse_out, R, S, D, wpi, st);
}

cudaError_t launch_combine(const float* part_o, const float* part_lse, void* out,
                           float* lse_out, int R, int S, int D, kvd_dtype out_dt,
                           cudaStream_t stream, long long gathered_stride) {
    // row-major [R, S, D] / [R, S], or blocks of gathered_stride floats per split
    const CombineStrides st = gathered_stride > 0
                                  ? CombineStrides{D, gathered_stride, 1, gathered_stride}
                                  : CombineStrides{(long long)S * D, D, S, 1};
    // warps per item: enough that each warp's splits fit one batch of loads
    // (a power of two, 1..8)
    int wpi = 1;
    while (wpi < kCombineWarps && wpi * kCombineBatch < S) wpi *= 2;
    // two dims per lane once one dim per lane would need more than ~1024 items
    // (8-byte loads: every row of every split must start 8-byte aligned)
    const bool even = D % 2 == 0 && st.o_split % 2 == 0;
    // four dims per lane (16-byte loads: every row of every split 16-byte
    // aligned) on the same condition: half the warps, twice the bytes each
    if (D % 4 == 0 && st.o_split % 4 == 0 && st.o_row % 4 == 0 && (long long)R * ((D + 31) / 32) >= 1024)
        return launch_combine_vpl<4>(part_o, part_lse, out, lse_out, R, S, D, out_dt, wpi, st,
                                     stream);
    if ((long long)R * ((D + 31) / 32) >= 1024 && even)
        return launch_combine_vpl<2>(part_o, part_lse, out, lse_out, R, S, D, out_dt, wpi, st,
                                     stream);
    return launch_combine_vpl<1>(part_o, part_lse, out, lse_out, R, S, D, out_dt, wpi, st, stream);
}

// ---------------------------------------------------------- copy_kvcache
// copy_kvcache ("Intel NPU running LLMs", Part 2 "NPUW 的核心设计", step 3):
// rows [0, n[b]) of every layer's K and V go from the prefill caches to the
// generate caches, all layers in one launch.  Grid (16-byte vectors of the
// copied rows / (256 * kCopyVecs), B * Hkv, layers * 2): z = 2 * layer +
// (0: K, 1: V); a thread moves kCopyVecs vectors, all loads before the
// stores.  The K planes of kv head 0 also write the layer's mask row of b.
constexpr int kCopyVecs = 8;
__global__ void __launch_bounds__(256)
copy_prefix_kernel(const unsigned char* const* __restrict__ k_src,
                   const unsigned char* const* __restrict__ v_src,
                   unsigned char* const* __restrict__ k_dst, unsigned char* const* __restrict__ v_dst,
                   uint8_t* const* __restrict__ masks, const int32_t* __restrict__ n, int Hkv,
                   int C_src, int C_dst, int row_bytes, int32_t* dev_status) {
    pdl_launch_dependents();
    pdl_wait();
    const int layer = blockIdx.z >> 1, kv = blockIdx.z & 1;
    const int b = blockIdx.y / Hkv, h = blockIdx.y % Hkv;
    const bool lead = blockIdx.x == 0 && threadIdx.x == 0;
    const int nb = n[b];
    if (nb < 0 || nb > min(C_src, C_dst)) {
        if (lead && h == 0 && blockIdx.z == 0) report(dev_status, KVD_DEV_POS_RANGE);
        return;
    }
    const unsigned char* src = kv ? v_src[layer] : k_src[layer];
    unsigned char* dst = kv ? v_dst[layer] : k_dst[layer];
    if (!src || !dst || ((reinterpret_cast<uintptr_t>(src) | reinterpret_cast<uintptr_t>(dst)) & 15u)) {
        if (lead) report(dev_status, KVD_DEV_POINTER);
        return;
    }
    const int vpr = row_bytes / 16;
    const long long nvec = (long long)nb * vpr;  // this plane's vectors: contiguous in src and dst rows
    const size_t plane = (size_t)b * Hkv + h;
    const uint4* s4 = reinterpret_cast<const uint4*>(src + plane * C_src * row_bytes);
    uint4* d4 = reinterpret_cast<uint4*>(dst + plane * C_dst * row_bytes);
    const long long v0 = (long long)blockIdx.x * blockDim.x * kCopyVecs + threadIdx.x;
    uint4 x[kCopyVecs];
#pragma unroll
    for (int k = 0; k < kCopyVecs; ++k) {
        const long long v = v0 + (long long)k * blockDim.x;
        if (v < nvec) x[k] = s4[v];
    }
#pragma unroll
    for (int k = 0; k < kCopyVecs; ++k) {
        const long long v = v0 + (long long)k * blockDim.x;
        if (v < nvec) d4[v] = x[k];
    }
    if (masks && kv == 0 && h == 0) {
        uint8_t* m = masks[layer];
        if (!m) {
            if (lead) report(dev_status, KVD_DEV_POINTER);
            return;
        }
        const long long tid = (long long)blockIdx.x * blockDim.x + threadIdx.x;
        for (long long t = tid; t < C_dst; t += (long long)gridDim.x * blockDim.x)
            m[(size_t)b * C_dst + t] = t < nb ? 1 : 0;
    }
}

cudaError_t launch_copy_prefix(const void* const* k_src, const void* const* v_src,
                               void* const* k_dst, void* const* v_dst, uint8_t* const* masks,
                               const int32_t* n, int L, int B, int Hkv, int C_src, int C_dst,
                               int row_bytes, int32_t* dev_status, cudaStream_t stream) {
    const long long vecs = (long long)(C_src < C_dst ? C_src : C_dst) * (row_bytes / 16);
    const long long bx = (vecs + 256 * kCopyVecs - 1) / (256 * kCopyVecs);
    const dim3 grid((unsigned)(bx < 1 ? 1 : bx), (unsigned)(B * Hkv), (unsigned)(2 * L));
    return launch_pdl(copy_prefix_kernel, grid, dim3(256), 0, stream,
                      reinterpret_cast<const unsigned char* const*>(k_src),
                      reinterpret_cast<const unsigned char* const*>(v_src),
                      reinterpret_cast<unsigned char* const*>(k_dst),
                      reinterpret_cast<unsigned char* const*>(v_dst), masks, n, Hkv, C_src, C_dst,
                      row_bytes, dev_status);
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

// ----------------------------------------------------------- append_paged
// Paged KV append ("Intel NPU running LLMs", Part 2, update_kvcache_for, in
// the paged layout of "PyPTO 实现 AscendC GatherPaKvCache" 3.2): token pos[q]
// of sequence q goes to block block_tables[q, seq_offset[q] / BS + pos[q] /
// BS], slot pos[q] % BS -- all Hkv x D of it, one contiguous row of the
// [NB, BS, Hkv, D] cache.  Grid (16-byte vectors of a row / 256, Q).  The
// checks follow the gather's order; a failing sequence writes nothing.
__global__ void __launch_bounds__(256)
append_paged_kernel(unsigned char* __restrict__ kc, unsigned char* __restrict__ vc,
                    const unsigned char* __restrict__ kn, const unsigned char* __restrict__ vn,
                    const int32_t* __restrict__ block_tables, const int32_t* __restrict__ seq_offset,
                    const int32_t* __restrict__ pos, int NB, int BS, int cols, int row_bytes,
                    int32_t* dev_status) {
    pdl_launch_dependents();
    pdl_wait();
    const int q = blockIdx.y;
    const bool reporter = blockIdx.x == 0 && threadIdx.x == 0;
    const long long t = pos[q];
    if (t < 0) {
        if (reporter) report(dev_status, KVD_DEV_POS_RANGE);
        return;
    }
    const long long off = seq_offset ? seq_offset[q] : 0;
    if (off < 0 || off % BS) {
        if (reporter) report(dev_status, KVD_DEV_SEQ_OFFSET);
        return;
    }
    const long long col = off / BS + t / BS;
    if (col >= cols) {
        if (reporter) report(dev_status, KVD_DEV_TABLE_COLS);
        return;
    }
    const long long phys = block_tables[(size_t)q * cols + col];
    if (phys < 0 || phys >= NB) {
        if (reporter) report(dev_status, KVD_DEV_BLOCK_RANGE);
        return;
    }
    const int v = blockIdx.x * blockDim.x + threadIdx.x;
    if (v < row_bytes / 16) {
        const size_t src = (size_t)q * row_bytes + (size_t)v * 16;
        const size_t dst = ((size_t)phys * BS + (size_t)(t % BS)) * row_bytes + (size_t)v * 16;
        const uint4 kx = *reinterpret_cast<const uint4*>(kn + src);
        const uint4 vx = *reinterpret_cast<const uint4*>(vn + src);
        *reinterpret_cast<uint4*>(kc + dst) = kx;
        *reinterpret_cast<uint4*>(vc + dst) = vx;
    }
}

cudaError_t launch_append_paged(void* key_cache, void* value_cache, const void* k_new,
                                const void* v_new, const int32_t* block_tables,
                                const int32_t* seq_offset, const int32_t* pos, int Q, int NB,
                                int BS, int cols, int row_bytes, int32_t* dev_status,
                                cudaStream_t stream) {
    const int nvec = row_bytes / 16;
    const dim3 grid((nvec + 255) / 256, Q);
    return launch_pdl(append_paged_kernel, grid, dim3(256), 0, stream,
                      static_cast<unsigned char*>(key_cache), static_cast<unsigned char*>(value_cache),
                      static_cast<const unsigned char*>(k_new),
                      static_cast<const unsigned char*>(v_new), block_tables, seq_offset, pos, NB,
                      BS, cols, row_bytes, dev_status);
}

// ------------------------------------------------------------- append_fp8
// KV append into quantised caches: the step's K/V rows of every kv head are
// quantised (amax = max |v|, scale = amax / 448, code = E4M3(v / scale), both
// divisions fp32 round-to-nearest, codes rounded to nearest even and
// saturated at 448; an all-zero row gets scale 0 and zero codes) and written
// as D codes, the scale and 12 zero bytes at slot pos[b].  One warp per row
// (K or V of one (b, kv head)); D / 32 values per lane.
__device__ __forceinline__ float as_float(float x) { return x; }
__device__ __forceinline__ float as_float(__nv_bfloat16 x) { return __bfloat162float(x); }

// Where a quantising append writes the row of (entry b, kv head h): slot
// pos[b] of the static buffer [B, Hkv, C, RB], or, with block tables, token
// pos[b] of sequence b in the paged cache [NB, BS, Hkv, RB] through the
// gather's index mapping (the checks in the paged append's order).  Null when
// the position is refused; `reporter` reports it.
struct QuantDest {
    const int32_t* block_tables;  // null: static buffer
    const int32_t* seq_offset;
    int NB, BS, cols;
};

__device__ __forceinline__ unsigned char* quant_row(unsigned char* cache, const QuantDest& pg,
                                                    int b, int h, int Hkv, int C, int p, int RB,
                                                    bool reporter, int32_t* dev_status) {
    if (!pg.block_tables) {
        if (p < 0 || p >= C) {
            if (reporter) report(dev_status, KVD_DEV_POS_RANGE);
            return nullptr;
        }
        return cache + (((size_t)b * Hkv + h) * C + p) * RB;
    }
    if (p < 0) {
        if (reporter) report(dev_status, KVD_DEV_POS_RANGE);
        return nullptr;
    }
    const long long off = pg.seq_offset ? pg.seq_offset[b] : 0;
    if (off < 0 || off % pg.BS) {
        if (reporter) report(dev_status, KVD_DEV_SEQ_OFFSET);
        return nullptr;
    }
    const long long col = off / pg.BS + p / pg.BS;
    if (col >= pg.cols) {
        if (reporter) report(dev_status, KVD_DEV_TABLE_COLS);
        return nullptr;
    }
    const long long phys = pg.block_tables[(size_t)b * pg.cols + col];
    if (phys < 0 || phys >= pg.NB) {
        if (reporter) report(dev_status, KVD_DEV_BLOCK_RANGE);
        return nullptr;
    }
    return cache + (((size_t)phys * pg.BS + p % pg.BS) * Hkv + h) * RB;
}

template <typename In, int D>
__global__ void __launch_bounds__(128)
append_fp8_kernel(unsigned char* __restrict__ kc, unsigned char* __restrict__ vc,
                  const In* __restrict__ kn, const In* __restrict__ vn,
                  const int32_t* __restrict__ pos, uint8_t* __restrict__ mask, int B, int Hkv,
                  int C, QuantDest pg, int32_t* dev_status) {
    pdl_launch_dependents();
    pdl_wait();
    constexpr int VPL = D / 32;
    constexpr int RB = D + 16;
    const int lane = threadIdx.x & 31;
    const long long job = (long long)blockIdx.x * 4 + (threadIdx.x >> 5);
    if (job >= 2ll * B * Hkv) return;
    const int kv = (int)(job & 1);
    const long long bh = job >> 1;
    const int b = (int)(bh / Hkv);
    const int p = pos[b];
    unsigned char* row = quant_row(kv ? vc : kc, pg, b, (int)(bh % Hkv), Hkv, C, p, RB,
                                   lane == 0 && kv == 0 && bh % Hkv == 0, dev_status);
    if (!row) return;
    const In* src = (kv ? vn : kn) + bh * D + VPL * lane;
    float x[VPL];
    float amax = 0.f;
#pragma unroll
    for (int i = 0; i < VPL; ++i) {
        x[i] = as_float(src[i]);
        amax = fmaxf(amax, fabsf(x[i]));
    }
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, off));
    const float scale = __fdiv_rn(amax, 448.f);
    uint32_t codes = 0;
#pragma unroll
    for (int i = 0; i < VPL; ++i) {
        const uint32_t c = scale > 0.f ? (uint32_t)__nv_cvt_float_to_fp8(__fdiv_rn(x[i], scale),
                                                                          __NV_SATFINITE, __NV_E4M3)
                                       : 0u;
        codes |= c << (8 * i);
    }
    if constexpr (VPL == 4)
        *reinterpret_cast<uint32_t*>(row + 4 * lane) = codes;
    else
        *reinterpret_cast<uint16_t*>(row + 2 * lane) = (uint16_t)codes;
    if (lane == 0) {
        *reinterpret_cast<uint4*>(row + D) = make_uint4(__float_as_uint(scale), 0u, 0u, 0u);
        if (mask && kv == 0 && bh % Hkv == 0) mask[(size_t)b * C + p] = 1;
    }
}

cudaError_t launch_append_fp8(void* k_cache, void* v_cache, const void* k_new, const void* v_new,
                              const int32_t* pos, uint8_t* mask, int B, int Hkv, int C, int D,
                              kvd_dtype in_dt, int32_t* dev_status, cudaStream_t stream,
                              const int32_t* block_tables, const int32_t* seq_offset, int NB,
                              int BS, int cols) {
    const QuantDest pg{block_tables, seq_offset, NB, BS, cols};
    const long long jobs = 2ll * B * Hkv;
    const dim3 grid((unsigned)((jobs + 3) / 4));
    unsigned char* kc = static_cast<unsigned char*>(k_cache);
    unsigned char* vc = static_cast<unsigned char*>(v_cache);
    if (in_dt == KVD_BF16) {
        const __nv_bfloat16* kn = static_cast<const __nv_bfloat16*>(k_new);
        const __nv_bfloat16* vn = static_cast<const __nv_bfloat16*>(v_new);
        return D == 128 ? launch_pdl(append_fp8_kernel<__nv_bfloat16, 128>, grid, dim3(128), 0, stream,
                                     kc, vc, kn, vn, pos, mask, B, Hkv, C, pg, dev_status)
                        : launch_pdl(append_fp8_kernel<__nv_bfloat16, 64>, grid, dim3(128), 0, stream,
                                     kc, vc, kn, vn, pos, mask, B, Hkv, C, pg, dev_status);
    }
    const float* kn = static_cast<const float*>(k_new);
    const float* vn = static_cast<const float*>(v_new);
    return D == 128 ? launch_pdl(append_fp8_kernel<float, 128>, grid, dim3(128), 0, stream, kc, vc,
                                 kn, vn, pos, mask, B, Hkv, C, pg, dev_status)
                    : launch_pdl(append_fp8_kernel<float, 64>, grid, dim3(128), 0, stream, kc, vc,
                                 kn, vn, pos, mask, B, Hkv, C, pg, dev_status);
}

// ------------------------------------------------------------- append_fp4
// The FP4 counterpart: scale = amax / 6, code = nearest E2M1 magnitude of
// x / scale (ties to the even code, saturated at 6), two codes per byte with
// element 2j in the low nibble.  One warp per (entry, kv head, K|V) row.

// Nearest E2M1 code of x: the magnitude's code is the number of rounding
// boundaries it passes (the midpoints of 0, 0.5, 1, 1.5, 2, 3, 4, 6; a value
// on a midpoint goes to the neighbour with the even code, so the boundary
// is passed with > or >= accordingly); NaN gives +6.
__device__ __forceinline__ uint32_t e2m1_code(float x) {
    if (x != x) return 0x7u;
    const float a = fabsf(x);
    const uint32_t c = (uint32_t)(a > 0.25f) + (uint32_t)(a >= 0.75f) + (uint32_t)(a > 1.25f) +
                       (uint32_t)(a >= 1.75f) + (uint32_t)(a > 2.5f) + (uint32_t)(a >= 3.5f) +
                       (uint32_t)(a > 5.f);
    return c | (signbit(x) ? 0x8u : 0u);
}

template <typename In, int D>
__global__ void __launch_bounds__(128)
append_fp4_kernel(unsigned char* __restrict__ kc, unsigned char* __restrict__ vc,
                  const In* __restrict__ kn, const In* __restrict__ vn,
                  const int32_t* __restrict__ pos, uint8_t* __restrict__ mask, int B, int Hkv,
                  int C, QuantDest pg, int32_t* dev_status) {
    pdl_launch_dependents();
    pdl_wait();
    constexpr int VPL = D / 32;  // elements per lane: 2 or 4, i.e. 1 or 2 code bytes
    constexpr int RB = D / 2 + 16;
    const int lane = threadIdx.x & 31;
    const long long job = (long long)blockIdx.x * 4 + (threadIdx.x >> 5);
    if (job >= 2ll * B * Hkv) return;
    const int kv = (int)(job & 1);
    const long long bh = job >> 1;
    const int b = (int)(bh / Hkv);
    const int p = pos[b];
    unsigned char* row = quant_row(kv ? vc : kc, pg, b, (int)(bh % Hkv), Hkv, C, p, RB,
                                   lane == 0 && kv == 0 && bh % Hkv == 0, dev_status);
    if (!row) return;
    const In* src = (kv ? vn : kn) + bh * D + VPL * lane;
    float x[VPL];
    float amax = 0.f;
#pragma unroll
    for (int i = 0; i < VPL; ++i) {
        x[i] = as_float(src[i]);
        amax = fmaxf(amax, fabsf(x[i]));
    }
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, off));
    const float scale = __fdiv_rn(amax, 6.f);
    uint32_t codes = 0;
#pragma unroll
    for (int i = 0; i < VPL; ++i) {
        const uint32_t c = scale > 0.f ? e2m1_code(__fdiv_rn(x[i], scale)) : 0u;
        codes |= c << (4 * i);
    }
    if constexpr (VPL == 4)
        *reinterpret_cast<uint16_t*>(row + 2 * lane) = (uint16_t)codes;
    else
        row[lane] = (unsigned char)codes;
    if (lane == 0) {
        *reinterpret_cast<uint4*>(row + D / 2) = make_uint4(__float_as_uint(scale), 0u, 0u, 0u);
        if (mask && kv == 0 && bh % Hkv == 0) mask[(size_t)b * C + p] = 1;
    }
}

cudaError_t launch_append_fp4(void* k_cache, void* v_cache, const void* k_new, const void* v_new,
                              const int32_t* pos, uint8_t* mask, int B, int Hkv, int C, int D,
                              kvd_dtype in_dt, int32_t* dev_status, cudaStream_t stream,
                              const int32_t* block_tables, const int32_t* seq_offset, int NB,
                              int BS, int cols) {
    const QuantDest pg{block_tables, seq_offset, NB, BS, cols};
    const long long jobs = 2ll * B * Hkv;
    const dim3 grid((unsigned)((jobs + 3) / 4));
    unsigned char* kc = static_cast<unsigned char*>(k_cache);
    unsigned char* vc = static_cast<unsigned char*>(v_cache);
    if (in_dt == KVD_BF16) {
        const __nv_bfloat16* kn = static_cast<const __nv_bfloat16*>(k_new);
        const __nv_bfloat16* vn = static_cast<const __nv_bfloat16*>(v_new);
        return D == 128 ? launch_pdl(append_fp4_kernel<__nv_bfloat16, 128>, grid, dim3(128), 0, stream,
                                     kc, vc, kn, vn, pos, mask, B, Hkv, C, pg, dev_status)
                        : launch_pdl(append_fp4_kernel<__nv_bfloat16, 64>, grid, dim3(128), 0, stream,
                                     kc, vc, kn, vn, pos, mask, B, Hkv, C, pg, dev_status);
    }
    const float* kn = static_cast<const float*>(k_new);
    const float* vn = static_cast<const float*>(v_new);
    return D == 128 ? launch_pdl(append_fp4_kernel<float, 128>, grid, dim3(128), 0, stream, kc, vc,
                                 kn, vn, pos, mask, B, Hkv, C, pg, dev_status)
                    : launch_pdl(append_fp4_kernel<float, 64>, grid, dim3(128), 0, stream, kc, vc,
                                 kn, vn, pos, mask, B, Hkv, C, pg, dev_status);
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
