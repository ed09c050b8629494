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
//
// Before its dependency wait a CTA asks L2 to prefetch its K/V rows: they do
// not depend on the previous kernel's results through L2 (the point where
// every store becomes visible), so the HBM works on them while the previous
// launch drains.  The last tile of the last split, the one a short prefix
// leaves masked, is copied only once the mask shows a valid slot in it.  When
// split 0 has room for every split's partial, the CTAs push their partials
// into split 0's shared memory before the cluster barrier, so split 0 merges
// from its own memory and the others may exit right after the barrier;
// otherwise split 0 reads the partials from the other CTAs' shared memory
// and a second barrier keeps them alive until then.
#pragma once

#include "attend_kernel.cuh"

namespace kvd {

constexpr int kSmallMaxSplits = 8;    // portable cluster size
constexpr int kSmallMaxTokens = 384;  // tokens of one split, all resident in shared memory

// Shared-memory layout of one CTA for nt tiles: K tiles | V tiles | q |
// merge buffer (mo [NCW][G][D], ml [NCW][G][2]) | partial slots (acc
// [slots][G][D], then m and l [slots][G]) | validity words | mbarrier.  The
// tiles start 1024-byte aligned.  With one slot per split (slots = S) every
// CTA pushes its partial into split 0's slots; with one slot each CTA keeps
// its own and split 0 reads them through distributed shared memory.
struct SmallLayout {
    int k_off, v_off, q_off, merge_off, part_off, words_off, bar_off, bytes;
    __host__ __device__ static SmallLayout make(int nt, int tile_bytes, int T, int D, int G,
                                                int NCW, int elem, int slots) {
        SmallLayout L;
        L.k_off = 0;
        L.v_off = nt * tile_bytes;
        L.q_off = 2 * nt * tile_bytes;
        L.merge_off = (L.q_off + G * D * elem + 127) / 128 * 128;
        L.part_off = (L.merge_off + NCW * G * (D + 2) * 4 + 127) / 128 * 128;
        L.words_off = L.part_off + slots * G * (D + 2) * 4;
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

__device__ __forceinline__ void st_cluster_f32(uint32_t addr, float v) {
    asm volatile("st.shared::cluster.f32 [%0], %1;" ::"r"(addr), "f"(v) : "memory");
}

__device__ __forceinline__ void st_cluster_f32x4(uint32_t addr, float4 v) {
    asm volatile("st.shared::cluster.v4.f32 [%0], {%1, %2, %3, %4};" ::"r"(addr), "f"(v.x),
                 "f"(v.y), "f"(v.z), "f"(v.w)
                 : "memory");
}

// Ask L2 to fetch [src, src + bytes) (16-byte aligned, a multiple of 16 bytes).
__device__ __forceinline__ void prefetch_l2_bulk(const void* src, uint32_t bytes) {
    asm volatile("cp.async.bulk.prefetch.L2.global [%0], %1;" ::"l"(src), "r"(bytes) : "memory");
}

// Every thread of every CTA of the cluster: writes before, reads after.
__device__ __forceinline__ void cluster_sync_all() {
    asm volatile("barrier.cluster.arrive.release.aligned;\n\tbarrier.cluster.wait.acquire.aligned;"
                 ::: "memory");
}

// Grid (S, row units), cluster (S, 1, 1): CTA (split, ru) holds tokens
// [split * chunk, min(C, (split + 1) * chunk)) of row unit ru.  NWG groups of
// the consumers' warp count consume, group j taking tiles j, j + NWG, ...
// (each warp keeps its own running state; the CTA's partial merges them
// all); warp NCT = NWG * NCW issues the copies, reads the mask and does the
// fused append.  Split 0 of each cluster writes the row's output.
template <class Cons, int NWG>
__global__ void __launch_bounds__((NWG * Cons::kNCW + 1) * 32)
attend_small_kernel(const AttendParams p, const __grid_constant__ CUtensorMap kmap,
                    const __grid_constant__ CUtensorMap vmap) {
    using Elem = typename Cons::ElemT;
    constexpr int D = Cons::kD, G = Cons::kG, T = Cons::kT, NCW = Cons::kNCW;
    constexpr int NCT = NWG * NCW;  // consumer warps
    constexpr int kHalves = D / 64;
    extern __shared__ unsigned char smem_raw[];
    unsigned char* smem = reinterpret_cast<unsigned char*>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    const int nt = (p.chunk + T - 1) / T;
    const int split = blockIdx.x, S = gridDim.x;
    const bool push = p.small_push != 0;
    const int slots = push ? S : 1;
    const SmallLayout L =
        SmallLayout::make(nt, Cons::kTileBytes, T, D, G, NCT, (int)sizeof(Elem), slots);
    uint64_t* bar = reinterpret_cast<uint64_t*>(smem + L.bar_off);
    uint32_t* words = reinterpret_cast<uint32_t*>(smem + L.words_off);
    float* mo = reinterpret_cast<float*>(smem + L.merge_off);
    float* ml = mo + NCT * G * D;
    float* part_acc = reinterpret_cast<float*>(smem + L.part_off);  // partial slots
    float* part_m = part_acc + slots * G * D;
    float* part_l = part_m + slots * G;

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
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
    // the last split's last tile waits for the mask (a short prefix leaves it
    // masked); every other tile is copied at once
    const bool gate_last = split == S - 1 && ntiles > 1;
    const int nnow = gate_last ? ntiles - 1 : ntiles;
    const size_t plane = ((size_t)bz * p.Hkv + kvh) * p.C;

    if (threadIdx.x == 0) {
        mbar_init(bar, 1);
        fence_barrier_init();
    }
    if (threadIdx.x == 32 * NCT) {
        if (Cons::kSwizzled) {
            prefetch_tensormap(&kmap);
            prefetch_tensormap(&vmap);
        }
        const int nrows = min(ntok, nnow * T);
        if (nrows > 0) {
            const unsigned char* kb = static_cast<const unsigned char*>(p.k);
            const unsigned char* vb = static_cast<const unsigned char*>(p.v);
            const size_t off = (plane + t_begin) * (size_t)Cons::kRowBytes;
            prefetch_l2_bulk(kb + off, (uint32_t)nrows * Cons::kRowBytes);
            prefetch_l2_bulk(vb + off, (uint32_t)nrows * Cons::kRowBytes);
        }
    }
    pdl_launch_dependents();
    pdl_wait();
    __syncthreads();

    int pb = -1;  // fused append (warp NCT): this CTA's slot of the new row, or -1
    // the step's new K/V row, 16-byte chunks held by lanes [0, kChunks) of warp NCT
    constexpr int kChunks = D * (int)sizeof(Elem) / 16;
    static_assert(kChunks <= 32, "a row's chunks fit one warp");
    constexpr bool kAppend = Cons::kRowBytes == D * (int)sizeof(Elem);  // never with quantised rows
    uint4 knew = make_uint4(0, 0, 0, 0), vnew = make_uint4(0, 0, 0, 0);
    if (warp == NCT) {
        const uint64_t pol = policy_evict_first();
        const uint32_t tile_kv = Cons::kSwizzled ? 2u * kHalves * T * 128u : 0u;
        auto issue_tile = [&](int i) {
            const size_t rowidx = plane + t_begin + i * T;
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
        };
        auto tile_kv_bytes = [&](int i) -> uint32_t {
            return Cons::kSwizzled ? tile_kv : 2u * (uint32_t)min(T, ntok - i * T) * Cons::kRowBytes;
        };
        if (lane == 0) {
            // transaction bytes first, the one arrival once the gated tile is decided
            const uint32_t qbytes = (uint32_t)(g_here * D * sizeof(Elem));
            uint32_t now = qbytes;
            for (int i = 0; i < nnow; ++i) now += tile_kv_bytes(i);
            mbar_expect_tx(bar, now);
            for (int i = 0; i < nnow; ++i) issue_tile(i);
            bulk_g2s(smem + L.q_off, static_cast<const Elem*>(p.q) + qrow0 * D, qbytes, bar, pol);
        }
        // the new row's slot, the new row itself and the split's validity
        // words, read while the copies fly (all loads issued before any is used)
        const int x = (kAppend && p.pos) ? __ldg(p.pos + bz) : -1;
        if (kAppend && p.pos && lane < kChunks) {
            const size_t src = ((size_t)bz * p.Hkv + kvh) * D;
            knew = __ldg(reinterpret_cast<const uint4*>(static_cast<const Elem*>(p.k_new) + src) + lane);
            vnew = __ldg(reinterpret_cast<const uint4*>(static_cast<const Elem*>(p.v_new) + src) + lane);
        }
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
            if (hg == 0 && lane < kChunks) {
                const size_t dst = (plane + pb) * D;
                reinterpret_cast<uint4*>(const_cast<Elem*>(static_cast<const Elem*>(p.k) + dst))[lane] = knew;
                reinterpret_cast<uint4*>(const_cast<Elem*>(static_cast<const Elem*>(p.v) + dst))[lane] = vnew;
            }
            if (lane == 0 && hg == 0 && kvh == 0 && p.mask_w) p.mask_w[(size_t)bz * p.C + pb] = 1;
            if (lane == 0) words[(pb - t_begin) >> 5] |= 1u << ((pb - t_begin) & 31);
            __syncwarp();
        }
        // the gated tile, if it holds a valid slot; then the one arrival
        if (lane == 0) {
            const int i = ntiles - 1;
            if (gate_last && tile_bits(words, i * T, min(T, ntok - i * T))) {
                mbar_arrive_expect_tx(bar, tile_kv_bytes(i));
                issue_tile(i);
            } else {
                mbar_arrive(bar);
            }
        }
    }
    __syncthreads();
    const volatile int never = 0;
    const bool landed = mbar_wait(bar, 0, &never);
    if (!landed && threadIdx.x == 0) report(p.dev_status, KVD_DEV_TIMEOUT);
    if (kAppend && landed && pb >= 0 && warp == NCT && lane < kChunks) {
        // the copied tile holds the old row at pb: put the new one in its place
        const int r = pb - t_begin, i = r / T, rr = r % T;
        uint32_t off;
        if constexpr (Cons::kSwizzled)
            off = (lane >> 3) * (Cons::kTileBytes / kHalves) + swz128(rr, lane & 7);
        else
            off = rr * Cons::kRowBytes + lane * 16;
        *reinterpret_cast<uint4*>(smem + L.k_off + i * Cons::kTileBytes + off) = knew;
        *reinterpret_cast<uint4*>(smem + L.v_off + i * Cons::kTileBytes + off) = vnew;
    }
    __syncthreads();

    if (warp < NCT) {
        const int grp = warp / NCW, lw = warp % NCW;
        Cons cons;
        cons.begin(reinterpret_cast<const Elem*>(smem + L.q_off), g_here, p.qscale, lane);
        if (landed) {
            for (int i = grp; i < ntiles; i += NWG) {
                const uint64_t bits = tile_bits(words, i * T, min(T, ntok - i * T));
                if (bits)
                    cons.tile(smem + L.k_off + i * Cons::kTileBytes,
                              smem + L.v_off + i * Cons::kTileBytes, bits, lw, lane, p.qscale);
            }
        }
        cons.finish(mo, ml, warp, lane);
    }
    __syncthreads();
    // the CTA's partial -- unnormalised output, max (log2 units) and sum per
    // head -- goes to slot `split` of split 0 (push) or to its own slot 0
    const int dst_rank = push ? 0 : split, dst_slot = push ? split : 0;
    if (warp == 0) {
        constexpr int V = D / 4;
        for (int idx = lane; idx < g_here * V; idx += 32) {
            const int hh = idx / V, d4 = idx % V;
            float M = -INFINITY;
#pragma unroll
            for (int w = 0; w < NCT; ++w) M = fmaxf(M, ml[(w * G + hh) * 2]);
            const float base = M == -INFINITY ? 0.f : M;
            float Lsum = 0.f;
            float4 O = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
            for (int w = 0; w < NCT; ++w) {
                const float sc = fast_exp2(ml[(w * G + hh) * 2] - base);
                Lsum = fmaf(ml[(w * G + hh) * 2 + 1], sc, Lsum);
                const float4 x = reinterpret_cast<const float4*>(mo + (w * G + hh) * D)[d4];
                O.x = fmaf(x.x, sc, O.x);
                O.y = fmaf(x.y, sc, O.y);
                O.z = fmaf(x.z, sc, O.z);
                O.w = fmaf(x.w, sc, O.w);
            }
            st_cluster_f32x4(cluster_smem_addr(part_acc + (dst_slot * G + hh) * D + 4 * d4, dst_rank), O);
            if (d4 == 0) {
                st_cluster_f32(cluster_smem_addr(part_m + dst_slot * G + hh, dst_rank), M);
                st_cluster_f32(cluster_smem_addr(part_l + dst_slot * G + hh, dst_rank), Lsum);
            }
        }
    }
    // the partials' writes before, their reads after; when pushed, only split
    // 0's memory is read past this point and the other CTAs may leave
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
                mr[r] = r < S ? ld_cluster_f32(cluster_smem_addr(part_m + (push ? r : 0) * G + hh,
                                                                 push ? 0 : r))
                              : -INFINITY;
                M = fmaxf(M, mr[r]);
            }
            const float base = M == -INFINITY ? 0.f : M;
            float Lsum = 0.f;
            float4 O = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
            for (int r = 0; r < kSmallMaxSplits; ++r) {
                if (r >= S || mr[r] == -INFINITY) continue;
                const int sr = push ? 0 : r, ss = push ? r : 0;
                const float sc = fast_exp2(mr[r] - base);
                Lsum = fmaf(ld_cluster_f32(cluster_smem_addr(part_l + ss * G + hh, sr)), sc, Lsum);
                const float4 x =
                    ld_cluster_f32x4(cluster_smem_addr(part_acc + (ss * G + hh) * D + 4 * d4, sr));
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
    if (!push) cluster_sync_all();  // the partials stay until split 0 has read them
}

}  // namespace kvd
