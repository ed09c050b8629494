// attend_small.cuh -- small static-buffer launches: one CTA per (row, split)
// with all of its split's K/V resident, and the splits of a row in one thread
// block cluster that merges them through distributed shared memory.
//
// A decode step over a short buffer ("Intel NPU running LLMs", Part 1: the
// 1024 + 128-slot static buffer) moves a few MB per layer, so its time is
// latency: the persistent kernel's unit pipeline (mask scan, then the tile
// loads, then the consumers) and the separate combine launch.  Here every
// copy of a CTA is issued at once, the mask is read while the copies fly, and
// the log-sum-exp merge of the row's splits (Part 3, Flash SDPA path) happens
// inside the cluster, so one launch writes the output.
#pragma once

#include "attend_kernel.cuh"

namespace kvd {

constexpr int kSmallMaxSplits = 8;    // portable cluster size
constexpr int kSmallMaxTokens = 384;  // tokens of one split, all resident in shared memory

// Shared-memory layout of one CTA for nt tiles: K tiles | V tiles | q |
// merge buffer (mo [NCW][G][D], ml [NCW][G][2]) | partial (acc [G][D], m [G],
// l [G]) | validity words | mbarrier.  The tiles start 1024-byte aligned.
struct SmallLayout {
    int k_off, v_off, q_off, merge_off, part_off, words_off, bar_off, bytes;
    __host__ __device__ static SmallLayout make(int nt, int tile_bytes, int T, int D, int G,
                                                int NCW, int elem) {
        SmallLayout L;
        L.k_off = 0;
        L.v_off = nt * tile_bytes;
        L.q_off = 2 * nt * tile_bytes;
        L.merge_off = (L.q_off + G * D * elem + 127) / 128 * 128;
        L.part_off = (L.merge_off + NCW * G * (D + 2) * 4 + 127) / 128 * 128;
        L.words_off = L.part_off + G * (D + 2) * 4;
        L.bar_off = (L.words_off + (nt * T + 31) / 32 * 4 + 7) / 8 * 8;
        L.bytes = L.bar_off + 16;
        return L;
    }
};

__device__ __forceinline__ uint32_t cluster_smem_addr(const void* p, int rank) {
    uint32_t r;
    asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(r) : "r"(smem_u32(p)), "r"(rank));
    return r;
}

__device__ __forceinline__ float ld_cluster_f32(uint32_t addr) {
    float v;
    asm volatile("ld.shared::cluster.f32 %0, [%1];" : "=f"(v) : "r"(addr) : "memory");
    return v;
}

__device__ __forceinline__ float4 ld_cluster_f32x4(uint32_t addr) {
    float4 v;
    asm volatile("ld.shared::cluster.v4.f32 {%0, %1, %2, %3}, [%4];"
                 : "=f"(v.x), "=f"(v.y), "=f"(v.z), "=f"(v.w)
                 : "r"(addr)
                 : "memory");
    return v;
}

// Every thread of every CTA of the cluster: writes before, reads after.
__device__ __forceinline__ void cluster_sync_all() {
    asm volatile("barrier.cluster.arrive.release.aligned;\n\tbarrier.cluster.wait.acquire.aligned;"
                 ::: "memory");
}

// Grid (S, row units), cluster (S, 1, 1): CTA (split, ru) holds tokens
// [split * chunk, min(C, (split + 1) * chunk)) of row unit ru.  Warps 0..NCW-1
// consume; warp NCW issues the copies, reads the mask and does the fused
// append.  Split 0 of each cluster writes the row's output.
template <class Cons>
__global__ void __launch_bounds__((Cons::kNCW + 1) * 32)
attend_small_kernel(const AttendParams p, const __grid_constant__ CUtensorMap kmap,
                    const __grid_constant__ CUtensorMap vmap) {
    using Elem = typename Cons::ElemT;
    constexpr int D = Cons::kD, G = Cons::kG, T = Cons::kT, NCW = Cons::kNCW;
    constexpr int kHalves = D / 64;
    extern __shared__ unsigned char smem_raw[];
    unsigned char* smem = reinterpret_cast<unsigned char*>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    const int nt = (p.chunk + T - 1) / T;
    const SmallLayout L =
        SmallLayout::make(nt, Cons::kTileBytes, T, D, G, NCW, (int)sizeof(Elem));
    uint64_t* bar = reinterpret_cast<uint64_t*>(smem + L.bar_off);
    uint32_t* words = reinterpret_cast<uint32_t*>(smem + L.words_off);
    float* mo = reinterpret_cast<float*>(smem + L.merge_off);
    float* ml = mo + NCW * G * D;
    float* part_acc = reinterpret_cast<float*>(smem + L.part_off);
    float* part_m = part_acc + G * D;
    float* part_l = part_m + G;

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int split = blockIdx.x, S = gridDim.x;
    const int ru = blockIdx.y;
    const int per_bz = p.Hkv * p.HG;
    const int bz = ru / per_bz, rem = ru % per_bz;
    const int kvh = rem / p.HG, hg = rem % p.HG;
    const int g_here = min(G, p.g - hg * G);
    const size_t qrow0 = (size_t)bz * p.Hq + (size_t)kvh * p.g + (size_t)hg * G;
    const int t_begin = split * p.chunk;
    const int t_end = min(p.C, t_begin + p.chunk);
    const int ntok = max(0, t_end - t_begin);
    const int ntiles = (ntok + T - 1) / T;  // <= nt

    if (threadIdx.x == 0) {
        mbar_init(bar, 1);
        fence_barrier_init();
    }
    if (threadIdx.x == 32 * NCW && Cons::kSwizzled) {
        prefetch_tensormap(&kmap);
        prefetch_tensormap(&vmap);
    }
    pdl_launch_dependents();
    pdl_wait();
    __syncthreads();

    int pb = -1;  // fused append (warp NCW): this CTA's slot of the new row, or -1
    if (warp == NCW) {
        const uint64_t pol = policy_evict_first();
        if (lane == 0) {
            const uint32_t qbytes = (uint32_t)(g_here * D * sizeof(Elem));
            const uint32_t kvbytes = Cons::kSwizzled ? 2u * kHalves * T * 128u * ntiles
                                                     : 2u * ntok * Cons::kRowBytes;
            mbar_arrive_expect_tx(bar, kvbytes + qbytes);
            for (int i = 0; i < ntiles; ++i) {
                const size_t rowidx = ((size_t)bz * p.Hkv + kvh) * p.C + t_begin + i * T;
                unsigned char* sk = smem + L.k_off + i * Cons::kTileBytes;
                unsigned char* sv = smem + L.v_off + i * Cons::kTileBytes;
                if constexpr (Cons::kSwizzled) {
#pragma unroll
                    for (int h = 0; h < kHalves; ++h) {
                        tma_g2s_2d(sk + h * Cons::kTileBytes / kHalves, &kmap, 64 * h, (int)rowidx,
                                   bar, pol);
                        tma_g2s_2d(sv + h * Cons::kTileBytes / kHalves, &vmap, 64 * h, (int)rowidx,
                                   bar, pol);
                    }
                } else {
                    const uint32_t bytes = (uint32_t)min(T, ntok - i * T) * Cons::kRowBytes;
                    bulk_g2s(sk, static_cast<const unsigned char*>(p.k) + rowidx * Cons::kRowBytes,
                             bytes, bar, pol);
                    bulk_g2s(sv, static_cast<const unsigned char*>(p.v) + rowidx * Cons::kRowBytes,
                             bytes, bar, pol);
                }
            }
            bulk_g2s(smem + L.q_off, static_cast<const Elem*>(p.q) + qrow0 * D, qbytes, bar, pol);
        }
        // the new row's slot and the split's validity words, read while the
        // copies fly (all loads issued before any is used)
        // the fused append (rows of Elem; never with quantised rows)
        constexpr bool kAppend = Cons::kRowBytes == D * (int)sizeof(Elem);
        const int x = (kAppend && p.pos) ? __ldg(p.pos + bz) : -1;
        const uint8_t* mrow = p.mask + (size_t)bz * p.C;
        const bool written = kAppend && p.pos != nullptr && p.mask_w != nullptr;
        const int nwords = (ntiles * T + 31) / 32;
        if (p.mask_vec) {
            // 16 slots per lane (t_begin is a multiple of 16, the rows 16-byte aligned)
            const int nvec = (ntok + 15) / 16;
            uint32_t bits = 0;
            if (lane < nvec) {
                const uint4 mv = ld_mask16(reinterpret_cast<const uint4*>(mrow + t_begin) + lane, written);
                bits = nonzero_bytes(mv.x) | (nonzero_bytes(mv.y) << 4) |
                       (nonzero_bytes(mv.z) << 8) | (nonzero_bytes(mv.w) << 12);
                const int nv = min(ntok - lane * 16, 16);
                bits &= nv >= 16 ? 0xffffu : ((1u << nv) - 1u);
            }
            const uint32_t hi = __shfl_down_sync(0xffffffffu, bits, 1);
            if ((lane & 1) == 0 && (lane >> 1) < nwords) words[lane >> 1] = bits | (hi << 16);
        } else {
            constexpr int kW = kSmallMaxTokens / 32;
            uint8_t mb[kW];
#pragma unroll
            for (int j = 0; j < kW; ++j) {
                const int tok = t_begin + 32 * j + lane;
                mb[j] = (j < nwords && tok < t_end) ? ld_mask1(mrow + tok, written) : 0;
            }
#pragma unroll
            for (int j = 0; j < kW; ++j) {
                const uint32_t w = __ballot_sync(0xffffffffu, mb[j] != 0);
                if (lane == 0 && j < nwords) words[j] = w;
            }
        }
        __syncwarp();
        if (kAppend && p.pos) {
            if (x < 0 || x >= p.C) {
                if (lane == 0 && split == 0 && kvh == 0 && hg == 0)
                    report(p.dev_status, KVD_DEV_POS_RANGE);
            } else if (x >= t_begin && x < t_end) {
                pb = x;
            }
        }
        if (kAppend && pb >= 0) {
            // fused append: the cache row (head group 0 writes it), the mask
            // slot (kv head 0) and the validity bit
            if (hg == 0) {
                constexpr int kWords = D * (int)sizeof(Elem) / 4;
                const size_t src = ((size_t)bz * p.Hkv + kvh) * D;
                const size_t dst = (((size_t)bz * p.Hkv + kvh) * p.C + pb) * D;
                const uint32_t* ks = reinterpret_cast<const uint32_t*>(static_cast<const Elem*>(p.k_new) + src);
                const uint32_t* vs = reinterpret_cast<const uint32_t*>(static_cast<const Elem*>(p.v_new) + src);
                uint32_t* kd = reinterpret_cast<uint32_t*>(const_cast<Elem*>(static_cast<const Elem*>(p.k) + dst));
                uint32_t* vd = reinterpret_cast<uint32_t*>(const_cast<Elem*>(static_cast<const Elem*>(p.v) + dst));
                for (int i = lane; i < kWords; i += 32) {
                    kd[i] = __ldg(ks + i);
                    vd[i] = __ldg(vs + i);
                }
                if (lane == 0 && kvh == 0 && p.mask_w) p.mask_w[(size_t)bz * p.C + pb] = 1;
            }
            if (lane == 0) words[(pb - t_begin) >> 5] |= 1u << ((pb - t_begin) & 31);
            __syncwarp();
        }
    }
    __syncthreads();
    const volatile int never = 0;
    const bool landed = mbar_wait(bar, 0, &never);
    if (!landed && threadIdx.x == 0) report(p.dev_status, KVD_DEV_TIMEOUT);
    if (Cons::kRowBytes == D * (int)sizeof(Elem) && landed && pb >= 0 && warp == NCW) {
        // the copied tile holds the old row at pb: put the new one in its place
        const int r = pb - t_begin, i = r / T, rr = r % T;
        constexpr int kChunks = D * (int)sizeof(Elem) / 16;
        const size_t src = ((size_t)bz * p.Hkv + kvh) * D;
        const uint4* ks = reinterpret_cast<const uint4*>(static_cast<const Elem*>(p.k_new) + src);
        const uint4* vs = reinterpret_cast<const uint4*>(static_cast<const Elem*>(p.v_new) + src);
        for (int c = lane; c < kChunks; c += 32) {
            uint32_t off;
            if constexpr (Cons::kSwizzled)
                off = (c >> 3) * (Cons::kTileBytes / kHalves) + swz128(rr, c & 7);
            else
                off = rr * Cons::kRowBytes + c * 16;
            *reinterpret_cast<uint4*>(smem + L.k_off + i * Cons::kTileBytes + off) = __ldg(ks + c);
            *reinterpret_cast<uint4*>(smem + L.v_off + i * Cons::kTileBytes + off) = __ldg(vs + c);
        }
    }
    __syncthreads();

    if (warp < NCW) {
        Cons cons;
        cons.begin(reinterpret_cast<const Elem*>(smem + L.q_off), g_here, p.qscale, lane);
        if (landed) {
            for (int i = 0; i < ntiles; ++i) {
                const uint64_t bits = tile_bits(words, i * T, min(T, ntok - i * T));
                if (bits)
                    cons.tile(smem + L.k_off + i * Cons::kTileBytes,
                              smem + L.v_off + i * Cons::kTileBytes, bits, warp, lane, p.qscale);
            }
        }
        cons.finish(mo, ml, warp, lane);
    }
    __syncthreads();
    // the CTA's partial: unnormalised output, max (log2 units) and sum per head
    if (warp == 0) {
        constexpr int V = D / 4;
        for (int idx = lane; idx < g_here * V; idx += 32) {
            const int hh = idx / V, d4 = idx % V;
            float M = -INFINITY;
#pragma unroll
            for (int w = 0; w < NCW; ++w) M = fmaxf(M, ml[(w * G + hh) * 2]);
            const float base = M == -INFINITY ? 0.f : M;
            float Lsum = 0.f;
            float4 O = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
            for (int w = 0; w < NCW; ++w) {
                const float sc = fast_exp2(ml[(w * G + hh) * 2] - base);
                Lsum = fmaf(ml[(w * G + hh) * 2 + 1], sc, Lsum);
                const float4 x = reinterpret_cast<const float4*>(mo + (w * G + hh) * D)[d4];
                O.x = fmaf(x.x, sc, O.x);
                O.y = fmaf(x.y, sc, O.y);
                O.z = fmaf(x.z, sc, O.z);
                O.w = fmaf(x.w, sc, O.w);
            }
            reinterpret_cast<float4*>(part_acc + hh * D)[d4] = O;
            if (d4 == 0) {
                part_m[hh] = M;
                part_l[hh] = Lsum;
            }
        }
    }
    cluster_sync_all();
    if (split == 0 && warp == 0) {
        // merge the row's S partials (log-sum-exp), write out and lse
        constexpr int V = D / 4;
        for (int idx = lane; idx < g_here * V; idx += 32) {
            const int hh = idx / V, d4 = idx % V;
            float mr[kSmallMaxSplits];
            float M = -INFINITY;
#pragma unroll
            for (int r = 0; r < kSmallMaxSplits; ++r) {
                mr[r] = r < S ? ld_cluster_f32(cluster_smem_addr(part_m + hh, r)) : -INFINITY;
                M = fmaxf(M, mr[r]);
            }
            const float base = M == -INFINITY ? 0.f : M;
            float Lsum = 0.f;
            float4 O = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
            for (int r = 0; r < kSmallMaxSplits; ++r) {
                if (r >= S || mr[r] == -INFINITY) continue;
                const float sc = fast_exp2(mr[r] - base);
                Lsum = fmaf(ld_cluster_f32(cluster_smem_addr(part_l + hh, r)), sc, Lsum);
                const float4 x =
                    ld_cluster_f32x4(cluster_smem_addr(part_acc + hh * D + 4 * d4, r));
                O.x = fmaf(x.x, sc, O.x);
                O.y = fmaf(x.y, sc, O.y);
                O.z = fmaf(x.z, sc, O.z);
                O.w = fmaf(x.w, sc, O.w);
            }
            const float inv = Lsum > 0.f ? 1.f / Lsum : 0.f;
            O.x *= inv;
            O.y *= inv;
            O.z *= inv;
            O.w *= inv;
            const size_t row = qrow0 + hh;
            store_out4<Elem>(p, row * D + 4 * d4, O);
            if (d4 == 0 && p.lse_out)
                p.lse_out[row] = Lsum > 0.f ? (M + log2f(Lsum)) * kLn2 : -INFINITY;
        }
    }
    cluster_sync_all();  // the partials stay until split 0 has read them
}

}  // namespace kvd
