// attend_split.cuh -- split-KV decode attention kernel (static buffer + mask,
// or paged cache through block tables), fp32 online softmax per split.
//
// What it computes (page title, section):
//  * "Intel NPU running LLMs" (OpenVINO community article 882), Part 3
//    "Attention 在 NPU 上的完整实现": decode is one query against all cached
//    keys (incremental SDPA); the Flash SDPA path tiles the sequence axis and
//    merges tiles exactly through a running output, running max and running
//    sum.  Part 1 "解决方案：预分配 + Attention Mask": slots with mask = 0 are
//    -inf before the softmax.  Part 6 "ONNX 表达不了 tiling 策略": the tile
//    recurrence (correction = exp(old max - new max)).
//  * "FlashMLA на Huawei Ascend", "Ход вычислений": running max, running sum
//    and output accumulator in float32; one log-sum-exp per row.
//  * "PyPTO 实现 AscendC GatherPaKvCache（Norm/ND 分支）" 3.2: token t of
//    sequence q lives in block block_tables[q, seq_offset[q]/BS + t/BS],
//    slot t % BS.
//
// GB300 design.  One CTA = one (batch or sequence, kv head, head group,
// split): it reads every K/V row of its token range once and serves all the
// query heads of the GQA group from shared memory.  Warp NCW is the producer:
// it scans the split's mask (or its block-table entries) into 32-token
// validity words, skips tiles with no valid token, and streams the others
// into a STAGES-deep shared-memory ring with 1-D bulk copies (static buffer:
// a tile of one kv head is contiguous) or 3-D TMA tensor copies (paged: one
// kv head of T consecutive slots of a physical block), completion tracked by
// mbarrier transaction counts.  Warps 0..NCW-1 consume: D/VEC lanes hold one
// token's row as 16-byte vectors, q.k uses packed fp32x2 FMAs and a shuffle
// reduction over the token's lanes, the running max / sum / output are
// updated once per sub-chunk of tokens, p.V again with packed FMAs.  At the
// end the lane groups and warps merge their (max, sum, output) states and the
// CTA writes either the final row (single split) or a normalised partial row
// plus its log-sum-exp for the combine kernel.
#pragma once

#include "attend_common.cuh"

namespace kvd {

template <typename Elem, int D, int G, int T, int STAGES, int NCW>
struct AttendShape {
    static constexpr int kVec = ElemTraits<Elem>::kPerVec;  // elements per lane vector
    static constexpr int kPairs = kVec / 2;
    static constexpr int kLPT = D / kVec;                   // lanes per token
    static constexpr int kTPW = 32 / kLPT;                  // tokens per warp step
    static constexpr int kTW = T / NCW;                     // tokens per warp per tile
    static constexpr int kSteps = kTW / kTPW;               // warp steps per tile
    static constexpr int kSubWant = (32 / G) < 1 ? 1 : (32 / G);
    static constexpr int kSub = kSteps < kSubWant ? kSteps : kSubWant;
    static constexpr int kTileBytes = T * D * (int)sizeof(Elem);
    static constexpr int kStageBytes = 2 * kTileBytes;
    static constexpr int kRingBytes = STAGES * kStageBytes;
    static constexpr int kMergeBytes = NCW * G * (D + 2) * 4;
    static constexpr int kSmemAlloc = kRingBytes + CtlLayout<STAGES>::kBytes + 1024;

    static_assert(D % kVec == 0 && kLPT <= 32 && 32 % kLPT == 0, "head_dim layout");
    static_assert(T % NCW == 0 && kTW % kTPW == 0, "tile layout");
    static_assert(kSteps % kSub == 0, "sub-chunking");
    static_assert(kMergeBytes <= kRingBytes, "merge area aliases the ring");
    static_assert(kTileBytes % 16 == 0, "bulk copies move 16-byte multiples");
};

template <typename Elem, int D, int G, int T, int STAGES, int NCW, bool PAGED>
__global__ void __launch_bounds__((NCW + 1) * 32)
attend_split_kernel(const AttendParams p, const __grid_constant__ CUtensorMap kmap,
                    const __grid_constant__ CUtensorMap vmap) {
    using Sh = AttendShape<Elem, D, G, T, STAGES, NCW>;
    using Tr = ElemTraits<Elem>;
    extern __shared__ unsigned char smem_raw[];
    unsigned char* smem = reinterpret_cast<unsigned char*>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    Ctl<STAGES> ctl(smem + Sh::kRingBytes);

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int split = blockIdx.x;
    const int kvh = blockIdx.y / p.HG, hg = blockIdx.y % p.HG;
    const int bz = blockIdx.z;  // batch entry (static buffer) or sequence (paged)

    if (threadIdx.x == 0) ctl.init(NCW);
    if (PAGED && threadIdx.x == 32 * NCW) {
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
            producer_issue<STAGES>(p, r, ctl, [&](int stage, int r0, int n, uint64_t* bar) {
                unsigned char* sk = smem + stage * Sh::kStageBytes;
                unsigned char* sv = sk + Sh::kTileBytes;
                if constexpr (PAGED) {
                    const int t0 = r.t_begin + r0;
                    const int row = ctl.blocks[t0 / p.BS - lb0] * p.BS + t0 % p.BS;
                    mbar_arrive_expect_tx(bar, 2u * p.tile * D * sizeof(Elem));
                    tma_g2s_3d(sk, &kmap, 0, kvh, row, bar, pol);
                    tma_g2s_3d(sv, &vmap, 0, kvh, row, bar, pol);
                } else {
                    const size_t base = (((size_t)bz * p.Hkv + kvh) * p.C + r.t_begin + r0) * D;
                    const uint32_t bytes = (uint32_t)n * D * sizeof(Elem);
                    mbar_arrive_expect_tx(bar, 2u * bytes);
                    bulk_g2s(sk, static_cast<const Elem*>(p.k) + base, bytes, bar, pol);
                    bulk_g2s(sv, static_cast<const Elem*>(p.v) + base, bytes, bar, pol);
                }
            });
        }
        return;
    }

    // ================================================================ consumers
    const int grp = lane / Sh::kLPT, sub = lane % Sh::kLPT;
    const int g_here = min(G, p.g - hg * G);  // query heads this CTA serves
    const size_t qrow0 = (size_t)bz * p.Hq + (size_t)kvh * p.g + (size_t)hg * G;

    float2 q2[G][Sh::kPairs];
#pragma unroll
    for (int hh = 0; hh < G; ++hh) {
        if (hh < g_here) {
            const uint4 raw = *reinterpret_cast<const uint4*>(static_cast<const Elem*>(p.q) +
                                                              (qrow0 + hh) * D + sub * Sh::kVec);
            Tr::unpack(raw, q2[hh]);
#pragma unroll
            for (int j = 0; j < Sh::kPairs; ++j)
                q2[hh][j] = fmul2(q2[hh][j], make_float2(p.qscale, p.qscale));
        } else {
#pragma unroll
            for (int j = 0; j < Sh::kPairs; ++j) q2[hh][j] = make_float2(0.f, 0.f);
        }
    }

    float m[G], l[G];
    float2 acc[G][Sh::kPairs];
#pragma unroll
    for (int hh = 0; hh < G; ++hh) {
        m[hh] = -INFINITY;
        l[hh] = 0.f;
#pragma unroll
        for (int j = 0; j < Sh::kPairs; ++j) acc[hh][j] = make_float2(0.f, 0.f);
    }

    int stage = 0;
    uint32_t phase = 0;
    while (true) {
        const int tile_i = consumer_next<STAGES>(ctl, stage, phase, p.dev_status);
        if (tile_i < 0) break;
        const Elem* Ks = reinterpret_cast<const Elem*>(smem + stage * Sh::kStageBytes);
        const Elem* Vs = Ks + T * D;
        const int r0 = tile_i * p.tile;

#pragma unroll
        for (int c = 0; c < Sh::kSteps; c += Sh::kSub) {
            float s[Sh::kSub][G];
            bool val[Sh::kSub];
#pragma unroll
            for (int i = 0; i < Sh::kSub; ++i) {
                const int tt = warp * Sh::kTW + (c + i) * Sh::kTPW + grp;
                const uint4 kr = *reinterpret_cast<const uint4*>(Ks + tt * D + sub * Sh::kVec);
                float2 kf[Sh::kPairs];
                Tr::unpack(kr, kf);
#pragma unroll
                for (int hh = 0; hh < G; ++hh) {
                    float2 a = fmul2(q2[hh][0], kf[0]);
#pragma unroll
                    for (int j = 1; j < Sh::kPairs; ++j) a = ffma2(q2[hh][j], kf[j], a);
                    s[i][hh] = a.x + a.y;
                }
                const int rel = r0 + tt;
                val[i] = tt < p.tile && ((ctl.words[rel >> 5] >> (rel & 31)) & 1u);
            }
#pragma unroll
            for (int off = Sh::kLPT / 2; off > 0; off >>= 1)
#pragma unroll
                for (int i = 0; i < Sh::kSub; ++i)
#pragma unroll
                    for (int hh = 0; hh < G; ++hh)
                        s[i][hh] += __shfl_xor_sync(0xffffffffu, s[i][hh], off);

            float pr[Sh::kSub][G];
#pragma unroll
            for (int hh = 0; hh < G; ++hh) {
                float mx = -INFINITY;
#pragma unroll
                for (int i = 0; i < Sh::kSub; ++i) {
                    s[i][hh] = val[i] ? s[i][hh] : -INFINITY;
                    mx = fmaxf(mx, s[i][hh]);
                }
                const float mn = fmaxf(m[hh], mx);
                const float base = (mn == -INFINITY) ? 0.f : mn;
                const float corr = fast_exp2(m[hh] - base);
                m[hh] = mn;
                float ls = 0.f;
#pragma unroll
                for (int i = 0; i < Sh::kSub; ++i) {
                    pr[i][hh] = fast_exp2(s[i][hh] - base);
                    ls += pr[i][hh];
                }
                l[hh] = fmaf(l[hh], corr, ls);
                const float2 c2 = make_float2(corr, corr);
#pragma unroll
                for (int j = 0; j < Sh::kPairs; ++j) acc[hh][j] = fmul2(acc[hh][j], c2);
            }
#pragma unroll
            for (int i = 0; i < Sh::kSub; ++i) {
                const int tt = warp * Sh::kTW + (c + i) * Sh::kTPW + grp;
                uint4 vr = *reinterpret_cast<const uint4*>(Vs + tt * D + sub * Sh::kVec);
                if (!val[i]) vr = make_uint4(0, 0, 0, 0);  // padding may hold inf/NaN
                float2 vf[Sh::kPairs];
                Tr::unpack(vr, vf);
#pragma unroll
                for (int hh = 0; hh < G; ++hh) {
                    const float2 pp = make_float2(pr[i][hh], pr[i][hh]);
#pragma unroll
                    for (int j = 0; j < Sh::kPairs; ++j) acc[hh][j] = ffma2(pp, vf[j], acc[hh][j]);
                }
            }
        }
        __syncwarp();
        if (lane == 0) mbar_arrive(&ctl.empty[stage]);
        if (++stage == STAGES) {
            stage = 0;
            phase ^= 1u;
        }
    }

    // ---- merge the lane groups of each warp (they hold different tokens)
#pragma unroll
    for (int off = Sh::kLPT; off < 32; off <<= 1) {
#pragma unroll
        for (int hh = 0; hh < G; ++hh) {
            const float mo = __shfl_xor_sync(0xffffffffu, m[hh], off);
            const float lo = __shfl_xor_sync(0xffffffffu, l[hh], off);
            const float mn = fmaxf(m[hh], mo);
            const float base = (mn == -INFINITY) ? 0.f : mn;
            const float a = fast_exp2(m[hh] - base), b = fast_exp2(mo - base);
            l[hh] = l[hh] * a + lo * b;
            m[hh] = mn;
#pragma unroll
            for (int j = 0; j < Sh::kPairs; ++j) {
                float2 other;
                other.x = __shfl_xor_sync(0xffffffffu, acc[hh][j].x, off);
                other.y = __shfl_xor_sync(0xffffffffu, acc[hh][j].y, off);
                acc[hh][j] = ffma2(acc[hh][j], make_float2(a, a), fmul2(other, make_float2(b, b)));
            }
        }
    }

    // ---- merge the consumer warps through shared memory (aliases the ring,
    // so every consumer must be done with its last tile first)
    asm volatile("bar.sync 1, %0;" ::"r"(NCW * 32) : "memory");
    float* mo_area = reinterpret_cast<float*>(smem);          // [NCW][G][D]
    float* ml_area = mo_area + NCW * G * D;                   // [NCW][G][2]
    if (grp == 0) {
#pragma unroll
        for (int hh = 0; hh < G; ++hh) {
#pragma unroll
            for (int j = 0; j < Sh::kPairs; ++j) {
                const int d = sub * Sh::kVec + 2 * j;
                mo_area[(warp * G + hh) * D + d] = acc[hh][j].x;
                mo_area[(warp * G + hh) * D + d + 1] = acc[hh][j].y;
            }
            if (sub == 0) {
                ml_area[(warp * G + hh) * 2] = m[hh];
                ml_area[(warp * G + hh) * 2 + 1] = l[hh];
            }
        }
    }
    asm volatile("bar.sync 1, %0;" ::"r"(NCW * 32) : "memory");

    write_rows<Elem, D, G, NCW>(p, mo_area, ml_area, qrow0, g_here, split);
}

}  // namespace kvd
