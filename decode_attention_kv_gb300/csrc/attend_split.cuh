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

#include "kvd_device.cuh"

namespace kvd {

constexpr int kMaxChunk = 4096;              // tokens per split, upper bound
constexpr int kMaxWords = kMaxChunk / 32;    // validity words per split
constexpr int kMaxBlocks = 128;              // block-table entries per split

struct AttendParams {
    const void* q;               // [rows, Hq, D]
    const void* k;               // static buffer [B, Hkv, C, D]
    const void* v;
    const uint8_t* mask;         // static buffer [B, C]
    const int32_t* block_tables; // paged [Q, cols]
    const int32_t* seq_lens;     // paged [Q + 1]
    const int32_t* seq_offset;   // paged [Q] or null
    void* out;                   // [rows, Hq, D] (single split)
    float* lse_out;              // [rows, Hq] or null (single split)
    float* part_o;               // [rows * Hq, S, D]
    float* part_lse;             // [rows * Hq, S]
    int32_t* dev_status;
    int Hq, Hkv, g, HG;          // g = Hq / Hkv, HG = head groups per kv head
    int C;                       // static buffer capacity
    int BS, cols, NB;            // paged geometry
    int tile;                    // tokens per ring stage (paged: divides BS)
    int chunk;                   // tokens per split (multiple of tile and of 32)
    int S;                       // splits
    int mask_vec;                // mask rows 16-byte aligned (C % 16 == 0)
    float qscale;                // scale * log2(e)
    int direct;                  // S == 1: write out / lse_out directly
};

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
    // ring | full[STAGES] | empty[STAGES] | meta[STAGES] | abort | words | blocks
    static constexpr int kBarOff = kRingBytes;
    static constexpr int kMetaOff = kBarOff + 2 * STAGES * 8;
    static constexpr int kAbortOff = kMetaOff + STAGES * 4;
    static constexpr int kWordsOff = (kAbortOff + 4 + 15) / 16 * 16;
    static constexpr int kBlocksOff = kWordsOff + kMaxWords * 4;
    static constexpr int kSmemBytes = kBlocksOff + kMaxBlocks * 4;
    static constexpr int kSmemAlloc = kSmemBytes + 1024;  // base aligned up to 1 KiB

    static_assert(D % kVec == 0 && kLPT <= 32 && 32 % kLPT == 0, "head_dim layout");
    static_assert(T % NCW == 0 && kTW % kTPW == 0, "tile layout");
    static_assert(kSteps % kSub == 0, "sub-chunking");
    static_assert(kMergeBytes <= kRingBytes, "merge area aliases the ring");
    static_assert(kTileBytes % 16 == 0, "bulk copies move 16-byte multiples");
};

// Any valid token among relative tokens [r0, r0 + n) of the split.
__device__ __forceinline__ bool any_valid(const uint32_t* words, int r0, int n) {
    int r = r0;
    const int end = r0 + n;
    while (r < end) {
        const int w = r >> 5, b = r & 31;
        const int take = min(32 - b, end - r);
        const uint32_t m = (take == 32) ? 0xffffffffu : (((1u << take) - 1u) << b);
        if (words[w] & m) return true;
        r += take;
    }
    return false;
}

// Four bytes -> four bits (bit i set when byte i is nonzero).
__device__ __forceinline__ uint32_t nonzero_bytes(uint32_t x) {
    uint32_t t = x | (x >> 4);
    t |= t >> 2;
    t |= t >> 1;
    return (t & 1u) | ((t >> 7) & 2u) | ((t >> 14) & 4u) | ((t >> 21) & 8u);
}

template <typename Elem, int D, int G, int T, int STAGES, int NCW, bool PAGED>
__global__ void __launch_bounds__((NCW + 1) * 32)
attend_split_kernel(const AttendParams p, const __grid_constant__ CUtensorMap kmap,
                    const __grid_constant__ CUtensorMap vmap) {
    using Sh = AttendShape<Elem, D, G, T, STAGES, NCW>;
    using Tr = ElemTraits<Elem>;
    extern __shared__ unsigned char smem_raw[];
    unsigned char* smem = reinterpret_cast<unsigned char*>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    uint64_t* full = reinterpret_cast<uint64_t*>(smem + Sh::kBarOff);
    uint64_t* empty = full + STAGES;
    int* meta = reinterpret_cast<int*>(smem + Sh::kMetaOff);
    volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + Sh::kAbortOff);
    uint32_t* words = reinterpret_cast<uint32_t*>(smem + Sh::kWordsOff);
    int* blocks = reinterpret_cast<int*>(smem + Sh::kBlocksOff);

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int split = blockIdx.x;
    const int kvh = blockIdx.y / p.HG, hg = blockIdx.y % p.HG;
    const int bz = blockIdx.z;  // batch entry (static buffer) or sequence (paged)

    if (threadIdx.x == 0) {
        for (int s = 0; s < STAGES; ++s) {
            mbar_init(&full[s], 1);
            mbar_init(&empty[s], NCW);
        }
        *abort_flag = 0;
        fence_barrier_init();
    }
    if (PAGED && threadIdx.x == 32 * NCW) {
        prefetch_tensormap(&kmap);
        prefetch_tensormap(&vmap);
    }

    // ---------------------------------------------------------- token range
    // Both roles derive the split's token range [t_begin, t_end) themselves.
    const int t_begin = split * p.chunk;
    int t_end, first_col = 0;
    if constexpr (PAGED) {
        const int s0 = p.seq_lens[bz], s1 = p.seq_lens[bz + 1];
        const int off = p.seq_offset ? p.seq_offset[bz] : 0;
        int len = s1 - s0;
        // A cumsum that does not start at 0 is reported; the differences are
        // still well defined and used.  Other violations empty the sequence.
        uint32_t bad = (bz == 0 && s0 != 0) ? KVD_DEV_SEQLENS : 0u;
        if (len < 0) {
            bad |= KVD_DEV_SEQLENS;
            len = 0;
        } else if (off < 0 || off % p.BS != 0) {
            bad |= KVD_DEV_SEQ_OFFSET;
            len = 0;
        } else {
            first_col = off / p.BS;
            if (first_col + (len + p.BS - 1) / p.BS > p.cols) {
                bad |= KVD_DEV_TABLE_COLS;
                len = 0;
            }
        }
        if (bad && threadIdx.x == 0 && split == 0 && blockIdx.y == 0) report(p.dev_status, bad);
        t_end = min(len, t_begin + p.chunk);
    } else {
        t_end = min(p.C, t_begin + p.chunk);
    }
    const int ntok = max(0, t_end - t_begin);
    const int ntiles = (ntok + p.tile - 1) / p.tile;
    __syncthreads();

    if (warp == NCW) {
        // ============================================================ producer
        const int nwords = (ntiles * p.tile + 31) / 32;
        int lb0 = 0;
        if constexpr (PAGED) {
            if (ntok > 0) {
                lb0 = t_begin / p.BS;
                const int nblk = (t_end - 1) / p.BS - lb0 + 1;
                const int32_t* row = p.block_tables + (size_t)bz * p.cols + first_col + lb0;
                for (int j = lane; j < nblk; j += 32) {
                    int ph = row[j];
                    if (ph < 0 || ph >= p.NB) {
                        report(p.dev_status, KVD_DEV_BLOCK_RANGE);
                        ph = -1;
                    }
                    blocks[j] = ph;
                }
                __syncwarp();
            }
            for (int j = 0; j < nwords; ++j) {
                const int tok = t_begin + 32 * j + lane;
                const bool ok = tok < t_end && blocks[tok / p.BS - lb0] >= 0;
                const uint32_t w = __ballot_sync(0xffffffffu, ok);
                if (lane == 0) words[j] = w;
            }
        } else {
            const uint8_t* mrow = p.mask + (size_t)bz * p.C;
            if (p.mask_vec) {
                // 16 slots per lane per vector, 512 slots per warp round; the
                // whole split's mask is requested before any bit is used.
                constexpr int R = kMaxChunk / 512;
                const int nvec = (ntok + 15) / 16;
                const uint4* src = reinterpret_cast<const uint4*>(mrow + t_begin);
                uint4 mv[R];
#pragma unroll
                for (int r = 0; r < R; ++r) {
                    const int vi = r * 32 + lane;
                    mv[r] = vi < nvec ? __ldg(src + vi) : make_uint4(0, 0, 0, 0);
                }
#pragma unroll
                for (int r = 0; r < R; ++r) {
                    const int vi = r * 32 + lane;
                    uint32_t bits = nonzero_bytes(mv[r].x) | (nonzero_bytes(mv[r].y) << 4) |
                                    (nonzero_bytes(mv[r].z) << 8) | (nonzero_bytes(mv[r].w) << 12);
                    const int nv = min(max(ntok - vi * 16, 0), 16);
                    bits &= (nv >= 16) ? 0xffffu : ((1u << nv) - 1u);
                    const uint32_t hi = __shfl_down_sync(0xffffffffu, bits, 1);
                    const int j = vi >> 1;
                    if ((lane & 1) == 0 && j < nwords) words[j] = bits | (hi << 16);
                }
            } else {
                for (int j0 = 0; j0 < nwords; j0 += 8) {
                    uint8_t mb[8];
#pragma unroll
                    for (int u = 0; u < 8; ++u) {
                        const int tok = t_begin + 32 * (j0 + u) + lane;
                        mb[u] = (j0 + u < nwords && tok < t_end) ? __ldg(mrow + tok) : 0;
                    }
#pragma unroll
                    for (int u = 0; u < 8; ++u) {
                        const uint32_t w = __ballot_sync(0xffffffffu, mb[u] != 0);
                        if (lane == 0 && j0 + u < nwords) words[j0 + u] = w;
                    }
                }
            }
        }
        __syncwarp();
        if (lane == 0) {
            const uint64_t pol = policy_evict_first();
            int stage = 0;
            uint32_t phase = 0;
            uint32_t issued_mask = 0, last_parity = 0;  // per stage: issued? parity of last issue
            bool failed = false;
            for (int i = 0; i < ntiles && !failed; ++i) {
                const int r0 = i * p.tile;
                const int n = min(p.tile, ntok - r0);
                if (!any_valid(words, r0, n)) continue;  // all-zero tile: never read
                if (!mbar_wait(&empty[stage], phase ^ 1u, abort_flag)) {
                    failed = true;
                    break;
                }
                meta[stage] = i;
                unsigned char* sk = smem + stage * Sh::kStageBytes;
                unsigned char* sv = sk + Sh::kTileBytes;
                if constexpr (PAGED) {
                    const int t0 = t_begin + r0;
                    const int row = blocks[t0 / p.BS - lb0] * p.BS + t0 % p.BS;
                    mbar_arrive_expect_tx(&full[stage], 2u * p.tile * D * sizeof(Elem));
                    tma_g2s_3d(sk, &kmap, 0, kvh, row, &full[stage], pol);
                    tma_g2s_3d(sv, &vmap, 0, kvh, row, &full[stage], pol);
                } else {
                    const size_t base = (((size_t)bz * p.Hkv + kvh) * p.C + t_begin + r0) * D;
                    const uint32_t bytes = (uint32_t)n * D * sizeof(Elem);
                    mbar_arrive_expect_tx(&full[stage], 2u * bytes);
                    bulk_g2s(sk, static_cast<const Elem*>(p.k) + base, bytes, &full[stage], pol);
                    bulk_g2s(sv, static_cast<const Elem*>(p.v) + base, bytes, &full[stage], pol);
                }
                issued_mask |= 1u << stage;
                last_parity = (last_parity & ~(1u << stage)) | (phase << stage);
                if (++stage == STAGES) {
                    stage = 0;
                    phase ^= 1u;
                }
            }
            if (!failed && mbar_wait(&empty[stage], phase ^ 1u, abort_flag)) {
                meta[stage] = -1;  // end of the split
                mbar_arrive(&full[stage]);
            } else {
                failed = true;
            }
            if (failed) {
                *abort_flag = 1;
                report(p.dev_status, KVD_DEV_TIMEOUT);
                // The consumers may leave early now: never let the CTA exit
                // while a copy issued here may still be writing the ring.
                // (On the normal path the consumers have waited for every
                // issued tile before they see the end marker, and the end
                // marker itself completes a phase, so no drain is needed.)
                for (int s = 0; s < STAGES; ++s)
                    if (issued_mask & (1u << s)) {
                        const volatile int never = 0;
                        mbar_wait(&full[s], (last_parity >> s) & 1u, &never);
                    }
            }
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
        if (!mbar_wait(&full[stage], phase, abort_flag)) {
            if (!*abort_flag) {
                *abort_flag = 1;
                report(p.dev_status, KVD_DEV_TIMEOUT);
            }
            break;
        }
        const int tile_i = meta[stage];
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
                val[i] = tt < p.tile && ((words[rel >> 5] >> (rel & 31)) & 1u);
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
        if (lane == 0) mbar_arrive(&empty[stage]);
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

    for (int idx = threadIdx.x; idx < g_here * D; idx += NCW * 32) {
        const int hh = idx / D, d = idx % D;
        float M = -INFINITY;
#pragma unroll
        for (int w = 0; w < NCW; ++w) M = fmaxf(M, ml_area[(w * G + hh) * 2]);
        const float base = (M == -INFINITY) ? 0.f : M;
        float L = 0.f, O = 0.f;
#pragma unroll
        for (int w = 0; w < NCW; ++w) {
            const float sc = fast_exp2(ml_area[(w * G + hh) * 2] - base);
            L = fmaf(ml_area[(w * G + hh) * 2 + 1], sc, L);
            O = fmaf(mo_area[(w * G + hh) * D + d], sc, O);
        }
        const size_t row = qrow0 + hh;
        const float lse = L > 0.f ? (M + log2f(L)) * kLn2 : -INFINITY;
        if (p.direct) {
            Tr::store(p.out, row * D + d, L > 0.f ? O / L : 0.f);
            if (d == 0 && p.lse_out) p.lse_out[row] = lse;
        } else {
            if (L > 0.f) p.part_o[(row * p.S + split) * D + d] = O / L;
            if (d == 0) p.part_lse[row * p.S + split] = lse;
        }
    }
}

}  // namespace kvd
