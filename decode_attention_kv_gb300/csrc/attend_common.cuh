// attend_common.cuh -- the parts of the split-KV decode attention kernels that
// do not depend on how the consumer warps compute: parameters, the split's
// token range, the producer's mask / block-table scan and its copy loop over
// the shared-memory ring, and the final merge of the consumer warps' states.
//
// Sources (page title, section): "Intel NPU running LLMs" (OpenVINO community
// article 882), Part 1 "解决方案：预分配 + Attention Mask" (0/1 mask; slots
// with mask = 0 take no part in the softmax) and Part 3 "Flash SDPA 路径"
// (tiles along the sequence merged exactly through running output, max and
// sum); "PyPTO 实现 AscendC GatherPaKvCache（Norm/ND 分支）" 3.2-3.3 (block
// table indirection, seq_offset, cumsum seq_lens and their constraints).
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

// Shared-memory control block that follows the ring:
// full[STAGES] | empty[STAGES] | meta[STAGES] | abort | words | blocks
template <int STAGES>
struct CtlLayout {
    static constexpr int kBar = 0;
    static constexpr int kMeta = kBar + 2 * STAGES * 8;
    static constexpr int kAbort = kMeta + STAGES * 4;
    static constexpr int kWords = (kAbort + 4 + 15) / 16 * 16;
    static constexpr int kBlocks = kWords + kMaxWords * 4;
    static constexpr int kBytes = kBlocks + kMaxBlocks * 4;
};

template <int STAGES>
struct Ctl {
    uint64_t* full;
    uint64_t* empty;
    int* meta;
    volatile int* abort_flag;
    uint32_t* words;
    int* blocks;
    __device__ explicit Ctl(unsigned char* base) {
        using L = CtlLayout<STAGES>;
        full = reinterpret_cast<uint64_t*>(base + L::kBar);
        empty = full + STAGES;
        meta = reinterpret_cast<int*>(base + L::kMeta);
        abort_flag = reinterpret_cast<volatile int*>(base + L::kAbort);
        words = reinterpret_cast<uint32_t*>(base + L::kWords);
        blocks = reinterpret_cast<int*>(base + L::kBlocks);
    }
    __device__ void init(int consumer_warps) {
        for (int s = 0; s < STAGES; ++s) {
            mbar_init(&full[s], 1);
            mbar_init(&empty[s], consumer_warps);
        }
        *abort_flag = 0;
        fence_barrier_init();
    }
};

// The split's token range [t_begin, t_end) of its sequence, the number of
// ring tiles it spans and (paged) the first block-table column.  Paged
// sequences that break a constraint of the gather page become empty and the
// violation is reported once per sequence.
struct SplitRange {
    int t_begin, t_end, ntok, ntiles, first_col;
};

template <bool PAGED>
__device__ __forceinline__ SplitRange split_range(const AttendParams& p, int bz, int split) {
    SplitRange r;
    r.t_begin = split * p.chunk;
    r.first_col = 0;
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
            r.first_col = off / p.BS;
            if (r.first_col + (len + p.BS - 1) / p.BS > p.cols) {
                bad |= KVD_DEV_TABLE_COLS;
                len = 0;
            }
        }
        if (bad && threadIdx.x == 0 && split == 0 && blockIdx.y == 0) report(p.dev_status, bad);
        r.t_end = min(len, r.t_begin + p.chunk);
    } else {
        r.t_end = min(p.C, r.t_begin + p.chunk);
    }
    r.ntok = max(0, r.t_end - r.t_begin);
    r.ntiles = (r.ntok + p.tile - 1) / p.tile;
    return r;
}

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

// Producer warp, all lanes: the split's validity words (bit = token valid:
// mask != 0, or a token below the sequence length whose block id is in range)
// and, paged, the physical block of each logical block the split touches.
// Writes words for every tile of the split (bits past the range are 0).
// Returns the first logical block index of the split (paged).
template <bool PAGED>
__device__ __forceinline__ int producer_scan(const AttendParams& p, const SplitRange& r, int bz,
                                             int lane, uint32_t* words, int* blocks) {
    const int nwords = (r.ntiles * p.tile + 31) / 32;
    int lb0 = 0;
    if constexpr (PAGED) {
        if (r.ntok > 0) {
            lb0 = r.t_begin / p.BS;
            const int nblk = (r.t_end - 1) / p.BS - lb0 + 1;
            const int32_t* row = p.block_tables + (size_t)bz * p.cols + r.first_col + lb0;
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
            const int tok = r.t_begin + 32 * j + lane;
            const bool ok = tok < r.t_end && blocks[tok / p.BS - lb0] >= 0;
            const uint32_t w = __ballot_sync(0xffffffffu, ok);
            if (lane == 0) words[j] = w;
        }
    } else {
        const uint8_t* mrow = p.mask + (size_t)bz * p.C;
        if (p.mask_vec) {
            // 16 slots per lane per vector, 512 slots per warp round; the whole
            // split's mask is requested before any bit is used.
            constexpr int R = kMaxChunk / 512;
            const int nvec = (r.ntok + 15) / 16;
            const uint4* src = reinterpret_cast<const uint4*>(mrow + r.t_begin);
            uint4 mv[R];
#pragma unroll
            for (int k = 0; k < R; ++k) {
                const int vi = k * 32 + lane;
                mv[k] = vi < nvec ? __ldg(src + vi) : make_uint4(0, 0, 0, 0);
            }
#pragma unroll
            for (int k = 0; k < R; ++k) {
                const int vi = k * 32 + lane;
                uint32_t bits = nonzero_bytes(mv[k].x) | (nonzero_bytes(mv[k].y) << 4) |
                                (nonzero_bytes(mv[k].z) << 8) | (nonzero_bytes(mv[k].w) << 12);
                const int nv = min(max(r.ntok - vi * 16, 0), 16);
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
                    const int tok = r.t_begin + 32 * (j0 + u) + lane;
                    mb[u] = (j0 + u < nwords && tok < r.t_end) ? __ldg(mrow + tok) : 0;
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
    return lb0;
}

// Producer, one lane: stream every tile of the split that holds a valid token
// through the ring, then the end marker.  `load(stage, r0, n)` issues the
// copies of the tile starting at relative token r0 (n tokens in range) and
// returns the bytes they will deliver to full[stage].  Every wait is bounded;
// on a timeout the CTA aborts after the copies already issued have landed.
template <int STAGES, typename Load>
__device__ __forceinline__ void producer_issue(const AttendParams& p, const SplitRange& r,
                                               Ctl<STAGES>& c, Load&& load) {
    int stage = 0;
    uint32_t phase = 0;
    uint32_t issued_mask = 0, last_parity = 0;  // per stage: issued? parity of last issue
    bool failed = false;
    for (int i = 0; i < r.ntiles && !failed; ++i) {
        const int r0 = i * p.tile;
        const int n = min(p.tile, r.ntok - r0);
        if (!any_valid(c.words, r0, n)) continue;  // all-zero tile: never read
        if (!mbar_wait(&c.empty[stage], phase ^ 1u, c.abort_flag)) {
            failed = true;
            break;
        }
        c.meta[stage] = i;
        load(stage, r0, n, &c.full[stage]);
        issued_mask |= 1u << stage;
        last_parity = (last_parity & ~(1u << stage)) | (phase << stage);
        if (++stage == STAGES) {
            stage = 0;
            phase ^= 1u;
        }
    }
    if (!failed && mbar_wait(&c.empty[stage], phase ^ 1u, c.abort_flag)) {
        c.meta[stage] = -1;  // end of the split
        mbar_arrive(&c.full[stage]);
    } else {
        failed = true;
    }
    if (failed) {
        *c.abort_flag = 1;
        report(p.dev_status, KVD_DEV_TIMEOUT);
        // The consumers may leave early now: never let the CTA exit while a
        // copy issued here may still be writing the ring.  (On the normal path
        // the consumers have waited for every issued tile before they see the
        // end marker, and the end marker itself completes a phase, so no
        // drain is needed there.)
        for (int s = 0; s < STAGES; ++s)
            if (issued_mask & (1u << s)) {
                const volatile int never = 0;
                mbar_wait(&c.full[s], (last_parity >> s) & 1u, &never);
            }
    }
}

// Consumer side of the ring: wait for the next stage; returns the tile index,
// -1 at the end of the split, -2 when the wait gave up (abort raised).
template <int STAGES>
__device__ __forceinline__ int consumer_next(Ctl<STAGES>& c, int stage, uint32_t phase,
                                             int32_t* dev_status) {
    if (!mbar_wait(&c.full[stage], phase, c.abort_flag)) {
        if (!*c.abort_flag) {
            *c.abort_flag = 1;
            report(dev_status, KVD_DEV_TIMEOUT);
        }
        return -2;
    }
    return c.meta[stage];
}

// Final merge of the consumer warps' states, written to shared memory as
// mo[w][h][d] (unnormalised output) and ml[w][h] = (max in log2 units, sum),
// then the CTA's rows: the final output (single split) or a normalised
// partial row and its natural-log log-sum-exp.
template <typename Elem, int D, int G, int NCW>
__device__ __forceinline__ void write_rows(const AttendParams& p, const float* mo,
                                           const float* ml, size_t qrow0, int g_here,
                                           int split) {
    for (int idx = threadIdx.x; idx < g_here * D; idx += NCW * 32) {
        const int hh = idx / D, d = idx % D;
        float M = -INFINITY;
#pragma unroll
        for (int w = 0; w < NCW; ++w) M = fmaxf(M, ml[(w * G + hh) * 2]);
        const float base = (M == -INFINITY) ? 0.f : M;
        float L = 0.f, O = 0.f;
#pragma unroll
        for (int w = 0; w < NCW; ++w) {
            const float sc = fast_exp2(ml[(w * G + hh) * 2] - base);
            L = fmaf(ml[(w * G + hh) * 2 + 1], sc, L);
            O = fmaf(mo[(w * G + hh) * D + d], sc, O);
        }
        const size_t row = qrow0 + hh;
        const float lse = L > 0.f ? (M + log2f(L)) * kLn2 : -INFINITY;
        if (p.direct) {
            ElemTraits<Elem>::store(p.out, row * D + d, L > 0.f ? O / L : 0.f);
            if (d == 0 && p.lse_out) p.lse_out[row] = lse;
        } else {
            if (L > 0.f) p.part_o[(row * p.S + split) * D + d] = O / L;
            if (d == 0) p.part_lse[row * p.S + split] = lse;
        }
    }
}

}  // namespace kvd
