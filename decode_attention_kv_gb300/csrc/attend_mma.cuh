// attend_mma.cuh -- split-KV decode attention for GQA groups of 4..8 query
// heads per kv head (bf16): q.K^T and p.V on the tensor cores.
//
// Same method and same split / ring / merge structure as attend_split.cuh
// ("Intel NPU running LLMs", Part 3 "Flash SDPA 路径": tiles along the
// sequence merged through running output, max and sum; "FlashMLA на Huawei
// Ascend", "Ход вычислений": fp32 running state); only the consumer warps
// differ.  With g query heads sharing one kv head, q.K^T of a 16-token slab
// is a [16 tokens x 16 dims] x [16 dims x 8 heads] product per 16 dims, i.e.
// mma.m16n8k16 with the tokens on M and the (up to 8) packed query heads on N;
// p.V is the transposed product [16 dims x 16 tokens] x [16 tokens x 8 heads].
// On CUDA cores this group width needs ~60 issue slots per token and kv head
// (q.k and p.v FMAs, shuffle reductions, exponentials); here it is ~7, which
// keeps the kernel on the HBM roofline instead of the issue rate.
//
// Precision.  K, V and q are bf16, so every product of q.K^T and of the V
// operand is exact in fp32 and the sums accumulate in fp32.  The probabilities
// p (fp32) enter p.V as p_hi + p_lo, both bf16 (p_hi = bf16(p), p_lo =
// bf16(p - p_hi)), so the operand keeps 16 significant bits and the result
// matches the CUDA-core path to fp32 rounding.
//
// Layout.  K and V tiles arrive by TMA as 64-element (128-byte) column halves
// in the 128-byte swizzle (16-byte chunk c of row r stored at chunk c ^ (r % 8)
// of that row), so that ldmatrix reads 8 rows of one column chunk without bank
// conflicts.  V rows of tokens that are not valid (mask = 0, past the length,
// or a dropped block) are zeroed in shared memory before p.V, so padding that
// holds inf or NaN cannot reach the accumulator through 0 x inf.
#pragma once

#include "attend_common.cuh"

namespace kvd {

__device__ __forceinline__ void ldsm_x4(uint32_t addr, uint32_t (&r)[4]) {
    asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0, %1, %2, %3}, [%4];"
                 : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3])
                 : "r"(addr));
}

__device__ __forceinline__ void ldsm_x4_trans(uint32_t addr, uint32_t (&r)[4]) {
    asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0, %1, %2, %3}, [%4];"
                 : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3])
                 : "r"(addr));
}

// d += a * b, m16n8k16, bf16 operands, fp32 accumulate.
__device__ __forceinline__ void mma_bf16(float (&d)[4], const uint32_t (&a)[4], uint32_t b0,
                                         uint32_t b1) {
    asm volatile(
        "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0, %1, %2, %3}, "
        "{%4, %5, %6, %7}, {%8, %9}, {%0, %1, %2, %3};"
        : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
        : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}

__device__ __forceinline__ uint32_t movmatrix_trans(uint32_t x) {
    uint32_t y;
    asm volatile("movmatrix.sync.aligned.m8n8.trans.b16 %0, %1;" : "=r"(y) : "r"(x));
    return y;
}

// Two floats -> bf16x2 (round to nearest even): `lo` in bits 0..15.
__device__ __forceinline__ uint32_t pack_bf16x2(float lo, float hi) {
    uint32_t r;
    asm("cvt.rn.bf16x2.f32 %0, %1, %2;" : "=r"(r) : "f"(hi), "f"(lo));
    return r;
}

__device__ __forceinline__ void fence_proxy_async_smem() {
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

// Byte offset of 16-byte chunk `ch` of row `r` inside a 128-byte-swizzled
// half tile whose base is 1024-byte aligned.
__device__ __forceinline__ uint32_t swz128(int r, int ch) {
    return (uint32_t)(r * 128 + ((ch ^ (r & 7)) << 4));
}

template <int D, int G, int T, int STAGES, int NCW>
struct MmaShape {
    static constexpr int kHalves = D / 64;             // 128-byte column halves per row
    static constexpr int kHalfBytes = T * 128;
    static constexpr int kTileBytes = kHalves * kHalfBytes;
    static constexpr int kStageBytes = 2 * kTileBytes;
    static constexpr int kRingBytes = STAGES * kStageBytes;
    static constexpr int kSlabsPerWarp = T / 16 / NCW;
    static constexpr int kKSteps = D / 16;             // q.K^T: 16 dims per mma
    static constexpr int kDBlocks = D / 16;            // p.V: 16 output dims per mma
    static constexpr int kMergeBytes = NCW * G * (D + 2) * 4;
    static constexpr int kSmemAlloc = kRingBytes + CtlLayout<STAGES>::kBytes + 1024;
    static_assert(D % 64 == 0, "head_dim must be a multiple of 64");
    static_assert(G >= 1 && G <= 8, "at most 8 query heads per mma column block");
    static_assert(T % (16 * NCW) == 0 && kSlabsPerWarp >= 1, "16-token slabs per warp");
    static_assert(kHalfBytes % 1024 == 0, "swizzled halves stay 1024-byte aligned");
    static_assert(kMergeBytes <= kRingBytes, "merge area aliases the ring");
};

template <int D, int G, int T, int STAGES, int NCW, bool PAGED>
__global__ void __launch_bounds__((NCW + 1) * 32)
attend_mma_kernel(const AttendParams p, const __grid_constant__ CUtensorMap kmap,
                  const __grid_constant__ CUtensorMap vmap) {
    using Sh = MmaShape<D, G, T, STAGES, NCW>;
    extern __shared__ unsigned char smem_raw[];
    unsigned char* smem = reinterpret_cast<unsigned char*>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    Ctl<STAGES> ctl(smem + Sh::kRingBytes);

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int split = blockIdx.x;
    const int kvh = blockIdx.y / p.HG, hg = blockIdx.y % p.HG;
    const int bz = blockIdx.z;

    if (threadIdx.x == 0) ctl.init(NCW);
    if (threadIdx.x == 32 * NCW) {
        prefetch_tensormap(&kmap);
        prefetch_tensormap(&vmap);
    }
    pdl_launch_dependents();
    pdl_wait();
    const SplitRange r = split_range<PAGED>(p, bz, split);
    __syncthreads();

    if (warp == NCW) {
        // ============================================================ producer
        const int lb0 = producer_scan<PAGED>(p, r, bz, lane, ctl.words, ctl.blocks);
        if (lane == 0) {
            const uint64_t pol = policy_evict_first();
            const uint32_t bytes = 2u * Sh::kHalves * p.tile * 128u;  // whole boxes, K and V
            producer_issue<STAGES>(p, r, ctl, [&](int stage, int r0, int n, uint64_t* bar) {
                unsigned char* sk = smem + stage * Sh::kStageBytes;
                unsigned char* sv = sk + Sh::kTileBytes;
                mbar_arrive_expect_tx(bar, bytes);
                const int t0 = r.t_begin + r0;
                if constexpr (PAGED) {
                    const int row = ctl.blocks[t0 / p.BS - lb0] * p.BS + t0 % p.BS;
#pragma unroll
                    for (int h = 0; h < Sh::kHalves; ++h) {
                        tma_g2s_3d(sk + h * Sh::kHalfBytes, &kmap, 64 * h, kvh, row, bar, pol);
                        tma_g2s_3d(sv + h * Sh::kHalfBytes, &vmap, 64 * h, kvh, row, bar, pol);
                    }
                } else {
                    const int row = (bz * p.Hkv + kvh) * p.C + t0;
#pragma unroll
                    for (int h = 0; h < Sh::kHalves; ++h) {
                        tma_g2s_2d(sk + h * Sh::kHalfBytes, &kmap, 64 * h, row, bar, pol);
                        tma_g2s_2d(sv + h * Sh::kHalfBytes, &vmap, 64 * h, row, bar, pol);
                    }
                }
            });
        }
        return;
    }

    // ================================================================ consumers
    const int gid = lane >> 2, tig = lane & 3;  // mma fragment row group / column pair
    const int g_here = min(G, p.g - hg * G);
    const size_t qrow0 = (size_t)bz * p.Hq + (size_t)kvh * p.g + (size_t)hg * G;

    // q^T as the B operand of q.K^T: column n = query head gid, rows = dims
    uint32_t qb[Sh::kKSteps][2];
#pragma unroll
    for (int ks = 0; ks < Sh::kKSteps; ++ks) {
        if (gid < g_here) {
            const __nv_bfloat16* qp =
                static_cast<const __nv_bfloat16*>(p.q) + (qrow0 + gid) * D + ks * 16 + 2 * tig;
            qb[ks][0] = *reinterpret_cast<const uint32_t*>(qp);
            qb[ks][1] = *reinterpret_cast<const uint32_t*>(qp + 8);
        } else {
            qb[ks][0] = qb[ks][1] = 0u;
        }
    }

    // running state of columns (query heads) 2*tig and 2*tig + 1; l is this
    // thread's share (its two token rows per slab) until the final reduction
    float m[2] = {-INFINITY, -INFINITY}, l[2] = {0.f, 0.f};
    float acc[Sh::kDBlocks][4];  // p.V^T: rows dims d*16 + gid (+8), columns 2*tig (+1)
#pragma unroll
    for (int d = 0; d < Sh::kDBlocks; ++d) acc[d][0] = acc[d][1] = acc[d][2] = acc[d][3] = 0.f;

    int stage = 0;
    uint32_t phase = 0;
    while (true) {
        const int tile_i = consumer_next<STAGES>(ctl, stage, phase, p.dev_status);
        if (tile_i < 0) break;
        const uint32_t kbase = smem_u32(smem + stage * Sh::kStageBytes);
        const uint32_t vbase = kbase + Sh::kTileBytes;
        unsigned char* vptr = smem + stage * Sh::kStageBytes + Sh::kTileBytes;
        const int r0 = tile_i * p.tile;
        bool wrote_smem = false;

#pragma unroll
        for (int sl = 0; sl < Sh::kSlabsPerWarp; ++sl) {
            const int slab0 = (warp * Sh::kSlabsPerWarp + sl) * 16;
            // validity of the slab's 16 tokens (lane i < 16 looks at token i)
            const int tl = slab0 + (lane & 15);
            const bool vl = tl < p.tile && ((ctl.words[(r0 + tl) >> 5] >> ((r0 + tl) & 31)) & 1u);
            const uint32_t vmask = __ballot_sync(0xffffffffu, vl) & 0xffffu;
            if (vmask == 0u) continue;
            if (vmask != 0xffffu) {
                // zero the V rows of the slab's invalid tokens (both halves)
                for (int i = lane; i < 16 * Sh::kHalves * 8; i += 32) {
                    const int row = i >> (Sh::kHalves == 2 ? 4 : 3);
                    const int rest = i & (Sh::kHalves * 8 - 1);
                    if (!((vmask >> row) & 1u)) {
                        const int h = rest >> 3, ch = rest & 7;
                        *reinterpret_cast<uint4*>(vptr + h * Sh::kHalfBytes + (slab0 + row) * 128 +
                                                  ch * 16) = make_uint4(0u, 0u, 0u, 0u);
                    }
                }
                wrote_smem = true;
                __syncwarp();
            }
            const bool v_lo = (vmask >> gid) & 1u, v_hi = (vmask >> (gid + 8)) & 1u;

            // ---- s = q.K^T for tokens slab0 + gid (s[0], s[1]) and + 8 (s[2], s[3])
            float s[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
            for (int ks = 0; ks < Sh::kKSteps; ++ks) {
                uint32_t a[4];
                const int row = slab0 + (lane & 15);
                const int ch = (ks & 3) * 2 + (lane >> 4);
                ldsm_x4(kbase + (ks >> 2) * Sh::kHalfBytes + swz128(row, ch), a);
                mma_bf16(s, a, qb[ks][0], qb[ks][1]);
            }
            s[0] = v_lo ? s[0] * p.qscale : -INFINITY;
            s[1] = v_lo ? s[1] * p.qscale : -INFINITY;
            s[2] = v_hi ? s[2] * p.qscale : -INFINITY;
            s[3] = v_hi ? s[3] * p.qscale : -INFINITY;

            // ---- online softmax per column over the slab's 16 tokens
            float mx0 = fmaxf(s[0], s[2]), mx1 = fmaxf(s[1], s[3]);
#pragma unroll
            for (int off = 4; off < 32; off <<= 1) {
                mx0 = fmaxf(mx0, __shfl_xor_sync(0xffffffffu, mx0, off));
                mx1 = fmaxf(mx1, __shfl_xor_sync(0xffffffffu, mx1, off));
            }
            const float mn0 = fmaxf(m[0], mx0), mn1 = fmaxf(m[1], mx1);
            const float b0 = mn0 == -INFINITY ? 0.f : mn0, b1 = mn1 == -INFINITY ? 0.f : mn1;
            const float c0 = fast_exp2(m[0] - b0), c1 = fast_exp2(m[1] - b1);
            m[0] = mn0;
            m[1] = mn1;
            const float p0 = fast_exp2(s[0] - b0), p1 = fast_exp2(s[1] - b1);
            const float p2 = fast_exp2(s[2] - b0), p3 = fast_exp2(s[3] - b1);
            l[0] = fmaf(l[0], c0, p0 + p2);
            l[1] = fmaf(l[1], c1, p1 + p3);
            const float2 cc = make_float2(c0, c1);
#pragma unroll
            for (int d = 0; d < Sh::kDBlocks; ++d) {
                float2 x = fmul2(make_float2(acc[d][0], acc[d][1]), cc);
                float2 y = fmul2(make_float2(acc[d][2], acc[d][3]), cc);
                acc[d][0] = x.x;
                acc[d][1] = x.y;
                acc[d][2] = y.x;
                acc[d][3] = y.y;
            }

            // ---- p as the B operand of p.V: hi + lo bf16 parts, transposed
            const uint32_t hi_lo = pack_bf16x2(p0, p1), hi_hi = pack_bf16x2(p2, p3);
            const float2 h0 = bf16x2_to_float2(hi_lo), h1 = bf16x2_to_float2(hi_hi);
            const uint32_t lo_lo = pack_bf16x2(p0 - h0.x, p1 - h0.y);
            const uint32_t lo_hi = pack_bf16x2(p2 - h1.x, p3 - h1.y);
            const uint32_t bh0 = movmatrix_trans(hi_lo), bh1 = movmatrix_trans(hi_hi);
            const uint32_t bl0 = movmatrix_trans(lo_lo), bl1 = movmatrix_trans(lo_hi);

            // ---- acc += V^T p for each 16-dim block
#pragma unroll
            for (int d = 0; d < Sh::kDBlocks; ++d) {
                uint32_t a[4];
                const int row = slab0 + (lane & 7) + ((lane >> 4) << 3);
                const int ch = (d & 3) * 2 + ((lane >> 3) & 1);
                ldsm_x4_trans(vbase + (d >> 2) * Sh::kHalfBytes + swz128(row, ch), a);
                mma_bf16(acc[d], a, bh0, bh1);
                mma_bf16(acc[d], a, bl0, bl1);
            }
        }
        // generic-proxy writes to the ring must be ordered before the next TMA
        // write into this stage
        if (wrote_smem) fence_proxy_async_smem();
        __syncwarp();
        if (lane == 0) mbar_arrive(&ctl.empty[stage]);
        if (++stage == STAGES) {
            stage = 0;
            phase ^= 1u;
        }
    }

    // ---- this warp's row sums (m is already the same for every gid)
#pragma unroll
    for (int off = 4; off < 32; off <<= 1) {
        l[0] += __shfl_xor_sync(0xffffffffu, l[0], off);
        l[1] += __shfl_xor_sync(0xffffffffu, l[1], off);
    }

    // ---- merge the consumer warps through shared memory (aliases the ring)
    asm volatile("bar.sync 1, %0;" ::"r"(NCW * 32) : "memory");
    float* mo_area = reinterpret_cast<float*>(smem);  // [NCW][G][D]
    float* ml_area = mo_area + NCW * G * D;           // [NCW][G][2]
#pragma unroll
    for (int c = 0; c < 2; ++c) {
        const int hh = 2 * tig + c;
        if (hh < G) {
#pragma unroll
            for (int d = 0; d < Sh::kDBlocks; ++d) {
                mo_area[(warp * G + hh) * D + d * 16 + gid] = acc[d][c];
                mo_area[(warp * G + hh) * D + d * 16 + gid + 8] = acc[d][2 + c];
            }
            if (gid == 0) {
                ml_area[(warp * G + hh) * 2] = m[c];
                ml_area[(warp * G + hh) * 2 + 1] = l[c];
            }
        }
    }
    asm volatile("bar.sync 1, %0;" ::"r"(NCW * 32) : "memory");
    write_rows<__nv_bfloat16, D, G, NCW>(p, mo_area, ml_area, qrow0, g_here, split);
}

}  // namespace kvd
