// attend_kernel.cuh -- persistent split-KV decode attention kernel (static
// buffer + 0/1 mask, or paged cache through block tables).
//
// What it computes (page title, section):
//  * "Intel NPU running LLMs" (OpenVINO community article 882): Part 1
//    "解决方案：预分配 + Attention Mask" -- slots with mask = 0 take no part in
//    the softmax; Part 3 "Attention 在 NPU 上的完整实现" -- decode is one query
//    against all cached keys, and the Flash SDPA path tiles the sequence axis
//    and merges the tiles exactly through a running output, max and sum.
//  * "FlashMLA на Huawei Ascend", "Математическая постановка" / "Ход
//    вычислений" -- out = softmax(q K^T * scale) V with fp32 running state and
//    one log-sum-exp per row.
//  * "PyPTO 实现 AscendC GatherPaKvCache（Norm/ND 分支）" 3.2-3.3 -- token t of
//    sequence q is slot t % BS of block block_tables[q, seq_offset[q]/BS +
//    t/BS]; cumsum seq_lens; the constraints on seq_offset and the table.
//
// Work.  A unit is one (row, split): row = (batch entry or sequence, kv head,
// group of <= G query heads sharing it), split = a chunk of `chunk` token
// slots of that row.  Units are numbered split-major and handed out by a
// global counter, so the grid is persistent (about one or two CTAs per SM)
// and load-balances rows of any length.  With a sliding window (static
// buffer) a row's splits count from the 64-slot boundary at or below its
// window's first slot, so that they cover the window and nothing before it
// ("Intel NPU running LLMs", Part 3, the sliding-window tile variant).
//
// CTA.  Four roles in warps:
//  * schedulers (warps NCW+1 .. NCW+4): each takes units from the work counter,
//    reads their metadata (sequence length and block-table entries, or the
//    split's mask) into 32-token validity words and queues them for the
//    loader in a ring of its own.  A scheduler takes a unit only while the
//    CTA has fewer than `look` tokens of queued, not yet requested tiles
//    (about 5 us of work), so that units stay with the counter until some
//    CTA is ready for them.  A
//    split without a valid token never reaches the loader: its log-sum-exps
//    are set to -inf (or, single split, its rows to zero).
//  * loader (warp NCW): skips tiles with no valid token and streams the others
//    into a STAGES-deep ring with 1-D bulk copies (static buffer, CUDA-core
//    consumers) or 2-D/3-D TMA tensor copies (paged, or 128-byte-swizzled
//    boxes for the tensor-core consumers); a unit's q rows ride along with its
//    first tile.  Each stage carries metadata: unit, tile, the tile's 64
//    validity bits, first/last-tile flags.  It runs ahead across unit
//    boundaries, so the ring does not drain between units.
//  * consumers (warps 0..NCW-1, attend_consumers.cuh): the online softmax over
//    the tiles; at a unit's last tile they drop their states into one of two
//    merge buffers and go on with the next unit.
//  * epilogue (warp NCW+5): merges the consumer warps' states of a unit and
//    writes either the final rows (single split) or a normalised partial row
//    and its log-sum-exp.
//  * index-list mode only: the last scheduler warp gathers half of each
//    tile's listed rows beside the loader (three warps schedule).
// With more than one split the host launches the log-sum-exp combine kernel
// right behind this one (programmatic dependent launch): it runs once the
// partial rows are complete, without atomics or fences here.
//
// Counters (unit counter, schedulers-done counter) live in the caller's
// workspace: zero before the first call; the last scheduler warp to finish
// taking units resets them.  The first unit of scheduler warp s (no atomic)
// is blockIdx.x * n + s (n scheduler warps) -- consecutive rows of one split,
// which share a mask row or a sequence -- or, with fewer units than
// scheduler warps, s * gridDim.x + blockIdx.x; the counter hands out the
// rest.
// All waits are bounded; a wait that runs out sets KVD_DEV_TIMEOUT, after
// which the counters must be zeroed again.
#pragma once

#include "attend_consumers.cuh"

namespace kvd {

// Where a row's tokens come from: a static buffer with a 0/1 mask, a paged
// cache through block tables, or a list of cache slots (top-k indices).
enum : int { kModeMasked = 0, kModePaged = 1, kModeIndexed = 2 };

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
    const int32_t* indices;      // indexed [B, topk]: cache slots, -1 = unused entry
    void* out;                   // [rows, Hq, D]
    float* lse_out;              // [rows, Hq] or null
    float* part_o;               // [rows * Hq, S, D]       (S > 1)
    float* part_lse;             // [rows * Hq, S]          (S > 1)
    uint32_t* sched;             // [0] units taken beyond the first ones, [1] schedulers done
    int32_t* dev_status;
    int Hq, Hkv, g, HG;          // g = Hq / Hkv, HG = head groups per kv head
    int C;                       // static buffer capacity
    int topk;                    // indexed: list entries per batch entry
    int BS, cols, NB;            // paged geometry
    int tile;                    // tokens per ring stage (paged: divides BS)
    int chunk;                   // tokens per split [0, Sb) (multiple of tile and of 32)
    int chunk2;                  // tokens per split [Sb, S) (multiple of tile and of 32)
    int Sb;
    int S;                       // splits per row
    int units;                   // rows * Hkv * HG * S
    int mask_vec;                // mask rows 16-byte aligned (C % 16 == 0)
    float qscale;                // scale * log2(e)
    int direct;                  // S == 1: units write the output rows directly
    int look;                    // a scheduler takes a unit only below this many queued tokens
    // fused append (static buffer, one head group per kv head): the step's rows
    // k_new/v_new [rows, Hkv, D] go to slot pos[b] of the caches and the mask
    const void* k_new;           // null: no append
    const void* v_new;
    const int32_t* pos;          // [rows]
    uint8_t* mask_w;             // the mask, written at pos
    int out_f32;                 // out is fp32 whatever the element type (a range's partial)
    int small_push;              // one-launch kernel: the splits push partials into split 0
    int small_nwg;               // one-launch kernel: consumer warp groups per CTA (1 or 2)
    // sliding window (static buffer): row b attends to the masked slots of
    // [win_last[b] - win + 1, win_last[b]] only; splits count their tokens
    // from the 64-slot boundary at or below the window's first slot
    int win;                     // window slots; 0: no window
    const int32_t* win_last;     // [rows]: the window's newest slot (the step's pos when appending)
};

// Output rows: the element type of q, or fp32 for a token range's partial
// (out_f32), which another step merges by log-sum-exp.
template <typename Elem>
__device__ __forceinline__ void store_out4(const AttendParams& p, size_t i, float4 x) {
    if (p.out_f32)
        ElemTraits<float>::store4(p.out, i, x);
    else
        ElemTraits<Elem>::store4(p.out, i, x);
}

template <typename Elem>
__device__ __forceinline__ void store_out1(const AttendParams& p, size_t i, float x) {
    if (p.out_f32)
        ElemTraits<float>::store(p.out, i, x);
    else
        ElemTraits<Elem>::store(p.out, i, x);
}

enum : uint32_t { kFirst = 1u, kLast = 2u, kEnd = 8u };

struct StageMeta {
    int unit;
    int tile;
    uint32_t flags;
    uint32_t pad;             // index-list mode: the unit's scheduler slot (for the gather warp)
    unsigned long long bits;  // validity of the tile's tokens
};

// One unit: its split, its row (counter index) and the query rows it serves.
// Units are numbered split-major (all rows' split 0, then split 1, ...): the
// last units handed out are the late splits, which are short or empty when
// lengths vary, so the CTAs finish close together.
struct Unit {
    int split, ru, bz, kvh, hg, g_here;
    size_t qrow0;
};

__device__ __forceinline__ Unit decode_unit(const AttendParams& p, int G, int u) {
    Unit un;
    const int rows = p.units / p.S;
    un.split = u / rows;
    un.ru = u % rows;
    const int per_bz = p.Hkv * p.HG;
    un.bz = un.ru / per_bz;
    const int rem = un.ru % per_bz;
    un.kvh = rem / p.HG;
    un.hg = rem % p.HG;
    un.g_here = min(G, p.g - un.hg * G);
    un.qrow0 = (size_t)un.bz * p.Hq + (size_t)un.kvh * p.g + (size_t)un.hg * G;
    return un;
}

// A unit prepared by the scheduler warp for the loader warp.
enum : int { kSlotTiles = 0, kSlotEnd = 2 };
constexpr int kSchedWarps = 4;                         // scheduler warps per CTA
constexpr int kRingSlots = 1;                          // queued units per scheduler
constexpr int kQueueSlots = kSchedWarps * kRingSlots;  // scheduler s owns slot s

struct UnitSlot {
    int kind;    // kSlotTiles: stream the unit's tiles; kSlotEnd: the scheduler is done
    int unit;
    int t_begin, ntok;
    int last;    // last tile that holds a valid token
    int lb0;     // first logical block of the split (paged)
    int pad[2];
    uint32_t words[kMaxWords];  // validity of the split's tokens
    int blocks[kMaxBlocks];     // physical block of each logical block (paged; -1 = dropped)
};

// Shared-memory control block:
// full[STAGES] | empty[STAGES] | gjob[STAGES] | qfull[Q] | qempty[Q] | mfull[M] | mempty[M] |
// meta[STAGES] | abort | pending | mhdr[M] | slots[Q]
template <int STAGES, int MB>
struct CtlLayout {
    static constexpr int kBar = 0;
    static constexpr int kQBar = kBar + 3 * STAGES * 8;
    static constexpr int kMBar = kQBar + 2 * kQueueSlots * 8;
    static constexpr int kMeta = kMBar + 2 * MB * 8;
    static constexpr int kAbort = kMeta + STAGES * (int)sizeof(StageMeta);
    static constexpr int kPending = kAbort + 4;
    static constexpr int kMhdr = kPending + 4;
    static constexpr int kSlots = (kMhdr + 4 * MB + 15) / 16 * 16;
    static constexpr int kBytes = kSlots + kQueueSlots * (int)sizeof(UnitSlot);
};

template <int STAGES, int MB>
struct Ctl {
    uint64_t* full;     // ring stage landed (loader -> consumers)
    uint64_t* empty;    // ring stage consumed (consumers -> loader)
    uint64_t* gjob;     // index-list mode: stage's tile posted (loader -> gather warp)
    uint64_t* qfull;    // unit slot filled (scheduler -> loader)
    uint64_t* qempty;   // unit slot read (loader -> scheduler)
    uint64_t* mfull;    // merge buffer filled (consumers -> epilogue)
    uint64_t* mempty;   // merge buffer read (epilogue -> consumers)
    StageMeta* meta;
    volatile int* abort_flag;
    int* pending;       // tokens of queued tiles the loader has not requested yet
    int* mhdr;          // unit of each merge buffer (-1: end of work)
    UnitSlot* slots;
    __device__ explicit Ctl(unsigned char* base) {
        using L = CtlLayout<STAGES, MB>;
        full = reinterpret_cast<uint64_t*>(base + L::kBar);
        empty = full + STAGES;
        gjob = empty + STAGES;
        qfull = reinterpret_cast<uint64_t*>(base + L::kQBar);
        qempty = qfull + kQueueSlots;
        mfull = reinterpret_cast<uint64_t*>(base + L::kMBar);
        mempty = mfull + MB;
        meta = reinterpret_cast<StageMeta*>(base + L::kMeta);
        abort_flag = reinterpret_cast<volatile int*>(base + L::kAbort);
        pending = reinterpret_cast<int*>(base + L::kPending);
        mhdr = reinterpret_cast<int*>(base + L::kMhdr);
        slots = reinterpret_cast<UnitSlot*>(base + L::kSlots);
    }
};

// STAGES ring stages, MB merge buffers (consumers -> epilogue).
template <class Cons, int STAGES, int MB>
struct KernelShape {
    using Elem = typename Cons::ElemT;
    static constexpr int kQBytes = Cons::kG * Cons::kD * (int)sizeof(Elem);
    static constexpr int kStageBytes = (2 * Cons::kTileBytes + kQBytes + 1023) / 1024 * 1024;
    static constexpr int kRingBytes = STAGES * kStageBytes;
    // one merge buffer: mo [NCW][G][D] then ml [NCW][G][2]
    static constexpr int kMergeBuf = (Cons::kNCW * Cons::kG * (Cons::kD + 2) * 4 + 127) / 128 * 128;
    static constexpr int kCtlOff = kRingBytes + MB * kMergeBuf;
    static constexpr int kSmemAlloc = kCtlOff + CtlLayout<STAGES, MB>::kBytes + 1024;
    // consumers, loader, schedulers, epilogue
    static constexpr int kThreads = (Cons::kNCW + 2 + kSchedWarps) * 32;
    static_assert(Cons::kTileBytes % 1024 == 0, "tiles keep stage parts 1024-byte aligned");
};

// The split's token range [t_begin, t_end) of its sequence, the ring tiles it
// spans and (paged) the first block-table column.  Paged sequences that break
// a constraint of the gather page become empty; `reporter` reports it.
struct SplitRange {
    int t_begin, t_end, ntok, ntiles, first_col;
    int t_lo;  // first slot that may count (> t_begin only where a window starts inside the split)
};

template <int MODE>
__device__ __forceinline__ SplitRange split_range(const AttendParams& p, int bz, int split,
                                                  bool reporter) {
    SplitRange r;
    const bool big = split < p.Sb;
    r.t_begin = big ? split * p.chunk : p.Sb * p.chunk + (split - p.Sb) * p.chunk2;
    const int span = big ? p.chunk : p.chunk2;
    r.first_col = 0;
    r.t_lo = r.t_begin;
    if constexpr (MODE == kModePaged) {
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
        if (bad && reporter) report(p.dev_status, bad);
        r.t_end = min(len, r.t_begin + span);
    } else if constexpr (MODE == kModeIndexed) {
        r.t_end = min(p.topk, r.t_begin + span);  // positions in the index list
    } else {
        r.t_end = min(p.C, r.t_begin + span);
        if (p.win > 0) {
            const int last = __ldg(p.win_last + bz);
            if (last < 0 || last >= p.C) {  // no window: an empty row
                if (reporter) report(p.dev_status, KVD_DEV_POS_RANGE);
                r.t_end = r.t_begin;
            } else {
                const int lo = max(0, last - p.win + 1);
                r.t_begin += lo & ~63;
                r.t_lo = max(lo, r.t_begin);
                r.t_end = min(last + 1, r.t_begin + span);
                if (r.t_end <= r.t_lo) r.t_end = r.t_lo = r.t_begin;  // ends below the window
            }
        }
    }
    r.ntok = max(0, r.t_end - r.t_begin);
    r.ntiles = (r.ntok + p.tile - 1) / p.tile;
    return r;
}

// Index-list mode: one warp gathers tile rows [row0, min(n, row1)) of a kv
// head's plane (row1 - row0 <= 32; row j's cache slot in lane j - row0's
// `slot`, -1: not listed) into a stage with 16-byte cp.async copies, a warp
// pass covering 32 / cpr whole rows of cpr 16-byte chunks (K and V; element
// rows or quantised rows), each chunk landing where the consumer's layout
// puts it.  (Per-row TMA boxes, four rows per box at best, issue too slowly
// here: the tensor engine's per-copy cost bounds a 512-byte box.)
template <class Cons, typename Elem, int D>
__device__ __forceinline__ void gather_rows(unsigned char* gk, unsigned char* gv, const void* k,
                                            const void* v, size_t plane, int slot, int row0,
                                            int row1, int n, int lane, uint64_t pol) {
    constexpr int kHalves = D / 64;
    const int rows = min(n, row1) - row0;
    if constexpr (Cons::kRowBytes == D * (int)sizeof(Elem)) {
        // element rows: D * sizeof(Elem) = 128, 256 or 512 bytes, a power of
        // two of chunks, so whole rows fill the warp
        constexpr int cpr = D * (int)sizeof(Elem) / 16, rpi = 32 / cpr;
        constexpr int epc = 16 / (int)sizeof(Elem);  // elements per chunk
        const int c = lane % cpr;
        const Elem* kb = static_cast<const Elem*>(k) + plane * D + c * epc;
        const Elem* vb = static_cast<const Elem*>(v) + plane * D + c * epc;
#pragma unroll 4
        for (int rb = 0; rb < rows; rb += rpi) {
            const int rr = rb + lane / cpr;
            const int slot_row = __shfl_sync(0xffffffffu, slot, rr & 31);
            if (rr < rows && slot_row >= 0) {
                const int row = row0 + rr;
                uint32_t off;
                if constexpr (Cons::kSwizzled)
                    off = (c >> 3) * (Cons::kTileBytes / kHalves) + swz128(row, c & 7);
                else
                    off = row * D * (int)sizeof(Elem) + c * 16;
                cp_async16(gk + off, kb + (size_t)slot_row * D, pol);
                cp_async16(gv + off, vb + (size_t)slot_row * D, pol);
            }
        }
    } else {
        // quantised rows (D + 16 or D/2 + 16 bytes: 3 to 9 chunks): 32 / cpr
        // whole rows per pass, the lanes past them idle
        constexpr int kRB = Cons::kRowBytes;
        static_assert(kRB % 16 == 0 && kRB <= 512, "rows of whole 16-byte chunks");
        static_assert(!Cons::kSwizzled, "quantised rows land unswizzled");
        constexpr int cpr = kRB / 16, rpi = 32 / cpr;
        const int c = lane % cpr;
        const unsigned char* kb = static_cast<const unsigned char*>(k) + plane * kRB + c * 16;
        const unsigned char* vb = static_cast<const unsigned char*>(v) + plane * kRB + c * 16;
#pragma unroll 4
        for (int rb = 0; rb < rows; rb += rpi) {
            const int rr = rb + lane / cpr;
            const int slot_row = __shfl_sync(0xffffffffu, slot, rr & 31);
            if (lane < rpi * cpr && rr < rows && slot_row >= 0) {
                const uint32_t off = (row0 + rr) * kRB + c * 16;
                cp_async16(gk + off, kb + (size_t)slot_row * kRB, pol);
                cp_async16(gv + off, vb + (size_t)slot_row * kRB, pol);
            }
        }
    }
}

// Validity bits of relative tokens [r0, r0 + n) of the split (n <= 64).
__device__ __forceinline__ uint64_t tile_bits(const uint32_t* words, int r0, int n) {
    uint64_t bits = 0;
    int k = 0;
    while (k < n) {
        const int w = (r0 + k) >> 5, b = (r0 + k) & 31;
        const int take = min(32 - b, n - k);
        const uint32_t m = (take == 32) ? 0xffffffffu : ((1u << take) - 1u);
        bits |= (uint64_t)((words[w] >> b) & m) << k;
        k += take;
    }
    return bits;
}

// Four bytes -> four bits (bit i set when byte i is nonzero).
__device__ __forceinline__ uint32_t nonzero_bytes(uint32_t x) {
    uint32_t t = x | (x >> 4);
    t |= t >> 2;
    t |= t >> 1;
    return (t & 1u) | ((t >> 7) & 2u) | ((t >> 14) & 4u) | ((t >> 21) & 8u);
}

// Mask loads.  Without the fused append the mask is read-only for the whole
// launch: non-coherent cached loads.  With it, the unit of kv head 0 whose
// range holds pos[b] stores the mask slot during the launch while other units
// read the same row, so the loads go to L2 (ld.global.cg), never to a stale
// L1 line.  A read that comes before that store sees 0 at pos[b]; that is
// harmless, because every unit whose range holds pos[b] ORs the bit into its
// own validity words itself (fused_append).
__device__ __forceinline__ uint4 ld_mask16(const uint4* ptr, bool written) {
    if (!written) return __ldg(ptr);
    uint4 v;
    asm volatile("ld.global.cg.v4.u32 {%0, %1, %2, %3}, [%4];"
                 : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
                 : "l"(ptr));
    return v;
}

__device__ __forceinline__ uint8_t ld_mask1(const uint8_t* ptr, bool written) {
    if (!written) return __ldg(ptr);
    unsigned short v;
    asm volatile("ld.global.cg.u8 %0, [%1];" : "=h"(v) : "l"(ptr));
    return (uint8_t)v;
}

// Producer warp, all lanes: the split's validity words (bit = token valid:
// mask != 0, or below the sequence length with its block id in range) and,
// paged, the physical block of each logical block the split touches.  Writes
// the words of every tile of the split (bits past the range are 0).  Returns
// the split's first logical block (paged).
template <int MODE>
__device__ __forceinline__ int producer_scan(const AttendParams& p, const SplitRange& r, int bz,
                                             int lane, uint32_t* words, int* blocks) {
    const int nwords = (r.ntiles * p.tile + 31) / 32;
    int lb0 = 0;
    if constexpr (MODE == kModeIndexed) {
        // blocks[j]: the cache slot of list entry t_begin + j (-1: none); an
        // entry outside [-1, C) is reported and dropped
        const int32_t* idx = p.indices + (size_t)bz * p.topk + r.t_begin;
        for (int j = lane; j < r.ntok; j += 32) {
            int t = idx[j];
            if (t < -1 || t >= p.C) {
                report(p.dev_status, KVD_DEV_POS_RANGE);
                t = -1;
            }
            blocks[j] = t;
        }
        __syncwarp();
        for (int j = 0; j < nwords; ++j) {
            const int e = 32 * j + lane;
            const uint32_t w = __ballot_sync(0xffffffffu, e < r.ntok && blocks[e] >= 0);
            if (lane == 0) words[j] = w;
        }
    } else if constexpr (MODE == kModePaged) {
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
        if (p.BS % 32 == 0) {
            // t_begin is a multiple of 32, so each word lies in one block: a
            // lane builds a whole word.
            for (int j = lane; j < nwords; j += 32) {
                const int tok0 = r.t_begin + 32 * j;
                const int n = min(max(r.t_end - tok0, 0), 32);
                const bool ok = n > 0 && blocks[tok0 / p.BS - lb0] >= 0;
                words[j] = !ok ? 0u : (n == 32 ? 0xffffffffu : ((1u << n) - 1u));
            }
        } else {
            for (int j = 0; j < nwords; ++j) {
                const int tok = r.t_begin + 32 * j + lane;
                const bool ok = tok < r.t_end && blocks[tok / p.BS - lb0] >= 0;
                const uint32_t w = __ballot_sync(0xffffffffu, ok);
                if (lane == 0) words[j] = w;
            }
        }
    } else {
        const uint8_t* mrow = p.mask + (size_t)bz * p.C;
        const bool written = p.pos != nullptr && p.mask_w != nullptr;  // fused append
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
                mv[k] = vi < nvec ? ld_mask16(src + vi, written) : make_uint4(0, 0, 0, 0);
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
                    mb[u] = (j0 + u < nwords && tok < r.t_end) ? ld_mask1(mrow + tok, written) : 0;
                }
#pragma unroll
                for (int u = 0; u < 8; ++u) {
                    const uint32_t w = __ballot_sync(0xffffffffu, mb[u] != 0);
                    if (lane == 0 && j0 + u < nwords) words[j0 + u] = w;
                }
            }
        }
        if (r.t_lo > r.t_begin) {
            // a window starting inside the split: its slots below the window
            // do not count (fewer than 64, so words 0 and 1 at most)
            __syncwarp();
            const int skip = r.t_lo - r.t_begin - 32 * lane;
            if (skip > 0) words[lane] &= skip >= 32 ? 0u : ~((1u << skip) - 1u);
        }
    }
    __syncwarp();
    return lb0;
}

// Fused append ("Intel NPU running LLMs", Part 2, update_kvcache_for): the
// unit whose token range holds pos[b] writes the step's K/V rows of its kv
// head into the cache at pos[b] (kv head 0 also sets the mask slot) before it
// is published, and counts pos[b] as valid; the loader's copies of the unit,
// issued after the slot is published, read the new rows (the proxy fence
// orders the plain stores before them).  Every (row, kv head) has exactly one
// such unit (one head group per kv head).  A pos outside [0, C) writes
// nothing and is reported once per batch entry.
template <typename Elem, int D>
__device__ __forceinline__ void fused_append(const AttendParams& p, const Unit& un,
                                             const SplitRange& r, int lane, uint32_t* words) {
    const int pb = __ldg(p.pos + un.bz);
    if (pb < 0 || pb >= p.C) {
        if (lane == 0 && un.kvh == 0 && un.hg == 0 && un.split == 0)
            report(p.dev_status, KVD_DEV_POS_RANGE);
        return;
    }
    if (pb < r.t_begin || pb >= r.t_end) return;
    constexpr int kWords = D * (int)sizeof(Elem) / 4;  // 32-bit words of a row
    const size_t src = ((size_t)un.bz * p.Hkv + un.kvh) * D;
    const size_t dst = (((size_t)un.bz * p.Hkv + un.kvh) * p.C + pb) * D;
    const uint32_t* ks = reinterpret_cast<const uint32_t*>(static_cast<const Elem*>(p.k_new) + src);
    const uint32_t* vs = reinterpret_cast<const uint32_t*>(static_cast<const Elem*>(p.v_new) + src);
    uint32_t* kd = reinterpret_cast<uint32_t*>(const_cast<Elem*>(static_cast<const Elem*>(p.k) + dst));
    uint32_t* vd = reinterpret_cast<uint32_t*>(const_cast<Elem*>(static_cast<const Elem*>(p.v) + dst));
#pragma unroll
    for (int i = lane; i < kWords; i += 32) {
        kd[i] = __ldg(ks + i);
        vd[i] = __ldg(vs + i);
    }
    if (lane == 0 && un.kvh == 0 && p.mask_w) p.mask_w[(size_t)un.bz * p.C + pb] = 1;
    asm volatile("fence.proxy.async.global;" ::: "memory");
    __syncwarp();
    if (lane == 0) words[(pb - r.t_begin) >> 5] |= 1u << ((pb - r.t_begin) & 31);
    __syncwarp();
}

// One warp turns the consumer warps' states of a unit (mo[w][h][d] and
// ml[w][h] = (m, l) in a merge buffer) into the unit's rows: the final output
// (single split) or a normalised partial row and its natural-log log-sum-exp.
// A lane handles four consecutive dims of one head (D % 4 == 0; rows of out
// and part_o are 16-byte aligned).
template <typename Elem, int D, int G, int NCW>
__device__ __forceinline__ void write_rows(const AttendParams& p, const float* mo,
                                           const float* ml, const Unit& un, int lane) {
    constexpr int V = D / 4;
    static_assert(D % 4 == 0, "head_dim must be a multiple of 4");
    for (int idx = lane; idx < un.g_here * V; idx += 32) {
        const int hh = idx / V, d4 = idx % V;
        float M = -INFINITY;
#pragma unroll
        for (int w = 0; w < NCW; ++w) M = fmaxf(M, ml[(w * G + hh) * 2]);
        const float base = (M == -INFINITY) ? 0.f : M;
        float L = 0.f;
        float4 O = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
        for (int w = 0; w < NCW; ++w) {
            const float sc = fast_exp2(ml[(w * G + hh) * 2] - base);
            L = fmaf(ml[(w * G + hh) * 2 + 1], sc, L);
            const float4 x = reinterpret_cast<const float4*>(mo + (w * G + hh) * D)[d4];
            O.x = fmaf(x.x, sc, O.x);
            O.y = fmaf(x.y, sc, O.y);
            O.z = fmaf(x.z, sc, O.z);
            O.w = fmaf(x.w, sc, O.w);
        }
        const size_t row = un.qrow0 + hh;
        const float lse = L > 0.f ? (M + log2f(L)) * kLn2 : -INFINITY;
        const float inv = L > 0.f ? 1.f / L : 0.f;
        O.x *= inv;
        O.y *= inv;
        O.z *= inv;
        O.w *= inv;
        if (p.direct) {
            store_out4<Elem>(p, row * D + 4 * d4, O);
            if (d4 == 0 && p.lse_out) p.lse_out[row] = lse;
        } else {
            if (L > 0.f)
                *reinterpret_cast<float4*>(p.part_o + (row * p.S + un.split) * D + 4 * d4) = O;
            if (d4 == 0) p.part_lse[row * p.S + un.split] = lse;
        }
    }
}

// Bounded mbarrier wait whose outcome is the same for every lane of the warp
// (every lane waits, for its own acquire; a timeout in any lane counts for all).
__device__ __forceinline__ bool warp_wait(uint64_t* bar, uint32_t parity,
                                          const volatile int* abort_flag) {
    const bool ok = mbar_wait(bar, parity, abort_flag);
    return __all_sync(0xffffffffu, ok);
}


template <class Cons, int STAGES, int MB, int MODE>
__global__ void __launch_bounds__(KernelShape<Cons, STAGES, MB>::kThreads)
attend_kernel(const AttendParams p, const __grid_constant__ CUtensorMap kmap,
              const __grid_constant__ CUtensorMap vmap) {
    using Sh = KernelShape<Cons, STAGES, MB>;
    using Elem = typename Cons::ElemT;
    constexpr int D = Cons::kD, G = Cons::kG, NCW = Cons::kNCW;
    constexpr int kHalves = D / 64;
    constexpr bool PAGED = MODE == kModePaged;
    constexpr bool INDEXED = MODE == kModeIndexed;
    // Index-list mode: the last kGatherN scheduler warps gather shares of
    // each tile's rows beside the loader (its 16-byte copies, one per lane,
    // are what bounds that mode); the others schedule.
    constexpr int kGatherN = INDEXED ? 1 : 0;
    constexpr int kSchedN = kSchedWarps - kGatherN;
    constexpr int kLoader = NCW, kSched0 = NCW + 1, kEpilogue = NCW + 1 + kSchedWarps;
    constexpr int kGather = kSched0 + kSchedN;  // first gather warp (index-list mode)
    // rows [gather_row(w), gather_row(w + 1)) of a tile: loader w = 0, gather warps 1..
    auto gather_row = [&](int w) { return w * p.tile / (kGatherN + 1); };
    extern __shared__ unsigned char smem_raw[];
    unsigned char* smem = reinterpret_cast<unsigned char*>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    Ctl<STAGES, MB> ctl(smem + Sh::kCtlOff);
    auto merge_mo = [&](int b) { return reinterpret_cast<float*>(smem + Sh::kRingBytes + b * Sh::kMergeBuf); };
    auto merge_ml = [&](int b) { return merge_mo(b) + NCW * G * D; };

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    if (threadIdx.x == 0) {
        for (int s = 0; s < STAGES; ++s) {
            mbar_init(&ctl.full[s], 1 + kGatherN);  // the loader (and the gather warps)
            mbar_init(&ctl.empty[s], NCW);
            mbar_init(&ctl.gjob[s], 1);
        }
        for (int s = 0; s < kQueueSlots; ++s) {
            mbar_init(&ctl.qfull[s], 32);  // every scheduler lane publishes its writes
            // every loader (and gather-warp) lane is done reading
            mbar_init(&ctl.qempty[s], 32 * (1 + kGatherN));
        }
        for (int s = 0; s < MB; ++s) {
            mbar_init(&ctl.mfull[s], NCW * 32);  // every consumer thread publishes its state
            mbar_init(&ctl.mempty[s], 32);       // every epilogue lane is done reading
        }
        *ctl.abort_flag = 0;
        *ctl.pending = 0;
        fence_barrier_init();
    }
    if (threadIdx.x == 32 * kLoader && (PAGED || Cons::kSwizzled) && !INDEXED) {
        prefetch_tensormap(&kmap);
        prefetch_tensormap(&vmap);
    }
    pdl_launch_dependents();
    pdl_wait();
    __syncthreads();

    if (warp >= kSched0 && warp < kSched0 + kSchedN) {
        // ========================================================= schedulers
        // Each takes units, reads their metadata (sequence length, mask or
        // block table) and queues them for the loader in its own ring of
        // kRingSlots.  Empty splits never reach the loader: their -inf
        // log-sum-exps are written here.
        const int sw = warp - kSched0;
        int pos = 0;
        uint32_t sphase = 0;
        bool failed = false;
        // Work counter: the first unit of each scheduler is fixed, the counter
        // hands out the others in order after them.  With enough units a CTA
        // starts with one unit per scheduler warp, consecutive -- one split of rows that
        // share their mask row or sequence, so that the metadata reads after
        // the first hit L1 -- else the first units are spread over all CTAs.
        const int n_sched = kSchedN * (int)gridDim.x;
        const int first_units = n_sched;
        int u = p.units >= n_sched ? (int)blockIdx.x * kSchedN + sw
                                   : sw * (int)gridDim.x + (int)blockIdx.x;
        auto publish = [&](int slot) {
            mbar_arrive(&ctl.qfull[slot]);
            if (++pos == kRingSlots) {
                pos = 0;
                sphase ^= 1u;
            }
        };
        // Below the lookahead?  Lane 0 polls; every lane gets the outcome.
        auto below_lookahead = [&]() -> bool {
            int ok = 1;
            if (lane == 0) {
                const volatile int* pend = ctl.pending;
                if (*pend >= p.look) {
                    const unsigned long long t0 = global_timer_ns();
                    while (*pend >= p.look) {
                        if (*ctl.abort_flag || global_timer_ns() - t0 > kWaitLimitNs) {
                            ok = 0;
                            break;
                        }
                        __nanosleep(64);
                    }
                }
            }
            return __shfl_sync(0xffffffffu, ok, 0) != 0;
        };
        bool first = true;
        // Scheduler 0 of the static buffer publishes its first slot without
        // the lookahead gate: the loader waits for that slot first (its
        // unit's first tiles were loaded speculatively) and takes no other
        // ring's units off the lookahead count until then.
        bool gated = !(MODE == kModeMasked && sw == 0 &&
                       (p.units < n_sched || (int)blockIdx.x * kSchedN < 2 * (p.units / p.S)));
        while (true) {
            const int slot = sw * kRingSlots + pos;
            if (!warp_wait(&ctl.qempty[slot], sphase ^ 1u, ctl.abort_flag)) {
                failed = true;
                break;
            }
            if (!first) {
                if (gated && !below_lookahead()) {
                    failed = true;
                    break;
                }
                const int t = lane == 0 ? (int)atomicAdd(&p.sched[0], 1u) : 0;
                u = first_units + __shfl_sync(0xffffffffu, t, 0);
            }
            first = false;
            UnitSlot& sl = ctl.slots[slot];
            if (u >= p.units) {
                if (lane == 0) sl.kind = kSlotEnd;
                __syncwarp();
                publish(slot);
                break;
            }
            const Unit un = decode_unit(p, G, u);
            const SplitRange r = split_range<MODE>(
                p, un.bz, un.split, lane == 0 && un.split == 0 && un.kvh == 0 && un.hg == 0);
            const int lb0 = producer_scan<MODE>(p, r, un.bz, lane, sl.words, sl.blocks);
            if constexpr (MODE == kModeMasked) {
                if (p.pos) fused_append<Elem, D>(p, un, r, lane, sl.words);
            }
            int last = -1;
            for (int i = r.ntiles - 1; i >= 0; --i)
                if (tile_bits(sl.words, i * p.tile, min(p.tile, r.ntok - i * p.tile))) {
                    last = i;
                    break;
                }
            if (last >= 0) {
                if (lane == 0) {
                    sl.kind = kSlotTiles;
                    sl.unit = u;
                    sl.t_begin = r.t_begin;
                    sl.ntok = r.ntok;
                    sl.last = last;
                    sl.lb0 = lb0;
                    atomicAdd(ctl.pending, (last + 1) * p.tile);
                }
                __syncwarp();
                publish(slot);
                gated = true;
            } else if (p.direct) {
                // the whole row is empty: zeros and lse = -inf
                for (int idx = lane; idx < un.g_here * D; idx += 32)
                    store_out1<Elem>(p, (un.qrow0 + idx / D) * D + idx % D, 0.f);
                if (lane < un.g_here && p.lse_out) p.lse_out[un.qrow0 + lane] = -INFINITY;
            } else if (lane < un.g_here) {
                p.part_lse[(un.qrow0 + lane) * p.S + un.split] = -INFINITY;  // no partial row
            }
        }
        if (failed && lane == 0 && !*ctl.abort_flag) {
            *ctl.abort_flag = 1;
            report(p.dev_status, KVD_DEV_TIMEOUT);
        }
        if (lane == 0) {
            // The scheduler warp that finishes taking units last leaves the
            // scheduling counters at zero for the next call.
            __threadfence();
            if (atomicAdd(&p.sched[1], 1u) == (uint32_t)n_sched - 1u) {
                atomicExch(&p.sched[0], 0u);
                atomicExch(&p.sched[1], 0u);
            }
        }
        return;
    }

    if constexpr (INDEXED) {
        if (warp >= kGather && warp < kGather + kGatherN) {
            // ==================================================== gather warps
            // A share of the rows of every tile the loader posts, in ring
            // order; the unit's slot is released (with the loader) after its
            // last tile.
            const int gw = warp - kGather + 1;
            const int row0 = gather_row(gw), row1 = gather_row(gw + 1);
            const uint64_t pol = policy_evict_first();
            int stage = 0;
            uint32_t phase = 0;
            while (true) {
                if (!warp_wait(&ctl.gjob[stage], phase, ctl.abort_flag)) break;
                const StageMeta mt = ctl.meta[stage];
                if (mt.flags & kEnd) break;
                const int slot = (int)mt.pad;
                const UnitSlot& sl = ctl.slots[slot];
                const Unit un = decode_unit(p, G, mt.unit);
                const int r0 = mt.tile * p.tile;
                const int n = min(p.tile, sl.ntok - r0);
                const int row = row0 + lane;
                const int s_row = row < min(n, row1) && ((mt.bits >> row) & 1ull)
                                      ? sl.blocks[r0 + row] : -1;
                if (n > row0) {
                    unsigned char* gk = smem + stage * Sh::kStageBytes;
                    gather_rows<Cons, Elem, D>(gk, gk + Cons::kTileBytes, p.k, p.v,
                                               ((size_t)un.bz * p.Hkv + un.kvh) * p.C, s_row,
                                               row0, row1, n, lane, pol);
                }
                cp_async_mbar_arrive(&ctl.full[stage]);
                __syncwarp();
                if (lane == 0) mbar_arrive(&ctl.full[stage]);
                if (mt.flags & kLast) mbar_arrive(&ctl.qempty[slot]);  // every lane
                if (++stage == STAGES) {
                    stage = 0;
                    phase ^= 1u;
                }
            }
            return;
        }
    }

    if (warp == kEpilogue) {
        // =========================================================== epilogue
        // Turns each finished unit's merge buffer into output or partial rows,
        // off the consumers' path.
        int mb = 0;
        uint32_t eph = 0;
        while (true) {
            if (!warp_wait(&ctl.mfull[mb], eph, ctl.abort_flag)) {
                if (lane == 0 && !*ctl.abort_flag) {
                    *ctl.abort_flag = 1;
                    report(p.dev_status, KVD_DEV_TIMEOUT);
                }
                break;
            }
            const int unit = ctl.mhdr[mb];
            if (unit < 0) break;
            const Unit un = decode_unit(p, G, unit);
            write_rows<Elem, D, G, NCW>(p, merge_mo(mb), merge_ml(mb), un, lane);
            __syncwarp();
            mbar_arrive(&ctl.mempty[mb]);  // every lane: done reading the buffer
            if (++mb == MB) {
                mb = 0;
                eph ^= 1u;
            }
        }
        return;
    }

    if (warp == kLoader) {
        // ============================================================= loader
        const uint64_t pol = policy_evict_first();
        int stage = 0;
        uint32_t phase = 0;
        uint32_t issued_mask = 0, last_parity = 0;  // per stage: issued? parity of the last issue
        bool failed = false;
        auto acquire = [&]() -> bool {
            if (!warp_wait(&ctl.empty[stage], phase ^ 1u, ctl.abort_flag)) failed = true;
            return !failed;
        };
        auto advance = [&]() {
            if (++stage == STAGES) {
                stage = 0;
                phase ^= 1u;
            }
        };
        // Static buffer, scheduler 0's first unit on a leading split (a
        // launch with fewer units than scheduler warps, bounded by latency,
        // or a split-0 or split-1 unit of a larger one, which holds valid
        // tokens unless its row is empty or shorter than one split): its
        // first tiles are loaded before its mask is
        // read (their addresses need no metadata) and delivered when that
        // unit's slot arrives -- as its tiles if the slot holds that unit,
        // else (the unit was empty) as empty tiles the consumers only
        // release.  Each carries q, so any of them can open the unit.
        int spec_n = 0, spec_unit = -1;
        uint32_t spec_mask = 0;  // stages issued but not yet delivered
        if constexpr (MODE == kModeMasked) {
            const int n_sched = kSchedN * (int)gridDim.x;
            const int u0 = p.units >= n_sched ? (int)blockIdx.x * kSchedN : (int)blockIdx.x;
            if (u0 < p.units && (p.units < n_sched || u0 < 2 * (p.units / p.S))) {
                const Unit un0 = decode_unit(p, G, u0);
                const SplitRange r = split_range<MODE>(p, un0.bz, un0.split, false);
                spec_unit = u0;
                spec_n = min(STAGES, r.ntiles);
                if (p.pos) {  // never before the tile the fused append writes into
                    const int pb = __ldg(p.pos + un0.bz);
                    if (pb >= r.t_begin && pb < r.t_end) spec_n = min(spec_n, (pb - r.t_begin) / p.tile);
                }
                const uint32_t qbytes = (uint32_t)(un0.g_here * D * sizeof(Elem));
                for (int i = 0; i < spec_n; ++i) {
                    if (!acquire()) break;  // the ring is empty: returns at once
                    if (lane == 0) {
                        const int n = min(p.tile, r.ntok - i * p.tile);
                        unsigned char* sk = smem + stage * Sh::kStageBytes;
                        unsigned char* sv = sk + Cons::kTileBytes;
                        unsigned char* sq = sv + Cons::kTileBytes;
                        const size_t rowidx =
                            ((size_t)un0.bz * p.Hkv + un0.kvh) * p.C + r.t_begin + i * p.tile;
                        if constexpr (Cons::kSwizzled) {
                            mbar_expect_tx(&ctl.full[stage], 2u * kHalves * p.tile * 128u + qbytes);
#pragma unroll
                            for (int h = 0; h < kHalves; ++h) {
                                tma_g2s_2d(sk + h * Cons::kTileBytes / kHalves, &kmap, 64 * h,
                                           (int)rowidx, &ctl.full[stage], pol);
                                tma_g2s_2d(sv + h * Cons::kTileBytes / kHalves, &vmap, 64 * h,
                                           (int)rowidx, &ctl.full[stage], pol);
                            }
                        } else {
                            const uint32_t bytes = (uint32_t)n * Cons::kRowBytes;
                            mbar_expect_tx(&ctl.full[stage], 2u * bytes + qbytes);
                            bulk_g2s(sk, static_cast<const unsigned char*>(p.k) + rowidx * Cons::kRowBytes,
                                     bytes, &ctl.full[stage], pol);
                            bulk_g2s(sv, static_cast<const unsigned char*>(p.v) + rowidx * Cons::kRowBytes,
                                     bytes, &ctl.full[stage], pol);
                        }
                        bulk_g2s(sq, static_cast<const Elem*>(p.q) + un0.qrow0 * D, qbytes,
                                 &ctl.full[stage], pol);
                        issued_mask |= 1u << stage;
                        last_parity = (last_parity & ~(1u << stage)) | (phase << stage);
                    }
                    spec_mask |= 1u << stage;
                    __syncwarp();
                    advance();
                }
                if (failed) spec_n = 0;
            }
        }
        // Scheduler rings: position and parity of each ring's head, which
        // rings have not ended yet; the loader takes whichever head is ready,
        // starting with the ring it did not take last (scheduler 0's ring
        // first while speculated tiles wait for it).
        int rpos[kSchedWarps] = {};
        uint32_t rphase = 0, live = (1u << kSchedN) - 1u;
        int pref = 0;
        while (!failed && live) {
            int pick = -1;
            if (lane == 0) {
                const unsigned long long t0 = global_timer_ns();
                for (uint32_t it = 0;; ++it) {
#pragma unroll
                    for (int k = 0; k < kSchedN; ++k) {
                        const int rr = (pref + k) % kSchedN;
                        if (spec_n > 0 && rr != 0) continue;
                        int hp = 0;
#pragma unroll
                        for (int q = 0; q < kSchedWarps; ++q) hp = q == rr ? rpos[q] : hp;
                        if (((live >> rr) & 1u) &&
                            mbar_test(&ctl.qfull[rr * kRingSlots + hp], (rphase >> rr) & 1u)) {
                            pick = rr;
                            break;
                        }
                    }
                    if (pick >= 0 || *ctl.abort_flag) break;
                    if ((it & 15u) == 15u && global_timer_ns() - t0 > kWaitLimitNs) break;
                }
            }
            pick = __shfl_sync(0xffffffffu, pick, 0);
            if (pick < 0) {
                failed = true;
                break;
            }
            int hp = 0;
#pragma unroll
            for (int q = 0; q < kSchedWarps; ++q) hp = q == pick ? rpos[q] : hp;
            const int slot = pick * kRingSlots + hp;
            // completed already: every lane acquires the scheduler's writes
            if (!warp_wait(&ctl.qfull[slot], (rphase >> pick) & 1u, ctl.abort_flag)) {
                failed = true;
                break;
            }
#pragma unroll
            for (int q = 0; q < kSchedWarps; ++q)
                if (q == pick && ++rpos[q] == kRingSlots) {
                    rpos[q] = 0;
                    rphase ^= 1u << q;
                }
            pref = (pick + 1) % kSchedN;
            const UnitSlot& sl = ctl.slots[slot];
            bool first = true;
            int counted = 0;  // tiles already taken off ctl.pending
            int i_start = 0;
            if (spec_n > 0) {
                // deliver the speculated stages (the oldest ones, in ring order)
                const bool same = sl.kind != kSlotEnd && sl.unit == spec_unit;
                int sstage = 0;  // speculation started at stage 0, phase 0
                for (int i = 0; i < spec_n; ++i, ++sstage) {
                    uint64_t bits = 0;
                    if (same && i <= sl.last)
                        bits = tile_bits(sl.words, i * p.tile, min(p.tile, sl.ntok - i * p.tile));
                    if (lane == 0) {
                        StageMeta& mt = ctl.meta[sstage];
                        mt.unit = same ? sl.unit : 0;
                        mt.tile = i;
                        mt.flags = bits ? ((first ? kFirst : 0u) | (i == sl.last ? kLast : 0u)) : 0u;
                        mt.bits = bits;
                        if (same && i <= sl.last) {
                            atomicAdd(ctl.pending, -(i + 1 - counted) * p.tile);
                            counted = i + 1;
                        }
                        mbar_arrive(&ctl.full[sstage]);
                    }
                    if (bits) first = false;
                }
                __syncwarp();
                spec_mask = 0;
                i_start = same ? spec_n : 0;
                spec_n = 0;
            }
            if (sl.kind == kSlotEnd) {
                live &= ~(1u << pick);
                continue;
            }
            const Unit un = decode_unit(p, G, sl.unit);
            const int t_begin = sl.t_begin, ntok = sl.ntok, last = sl.last, lb0 = sl.lb0;
            for (int i = i_start; i <= last; ++i) {
                const int r0 = i * p.tile;
                const int n = min(p.tile, ntok - r0);
                const uint64_t bits = tile_bits(sl.words, r0, n);
                if (!bits) continue;  // all-zero tile: never read
                if (!acquire()) break;
                if constexpr (INDEXED) {
                    // Post the tile to the gather warps, gather the first share
                    // of its rows here.  The stage's full barrier waits for
                    // every warp's copies through its cp.async arrivals, each
                    // made before that warp's own arrival.
                    if (lane == 0) {
                        StageMeta& mt = ctl.meta[stage];
                        mt.unit = sl.unit;
                        mt.tile = i;
                        mt.flags = (first ? kFirst : 0u) | (i == last ? kLast : 0u);
                        mt.pad = (uint32_t)slot;
                        mt.bits = bits;
                        mbar_arrive(&ctl.gjob[stage]);
                    }
                    unsigned char* gk = smem + stage * Sh::kStageBytes;
                    const int g1 = gather_row(1);
                    const int s_lo = lane < min(n, g1) && ((bits >> lane) & 1ull) ? sl.blocks[r0 + lane] : -1;
                    gather_rows<Cons, Elem, D>(gk, gk + Cons::kTileBytes, p.k, p.v,
                                               ((size_t)un.bz * p.Hkv + un.kvh) * p.C, s_lo, 0, g1,
                                               n, lane, pol);
                    cp_async_mbar_arrive(&ctl.full[stage]);
                    __syncwarp();
                }
                if (lane == 0) {
                    atomicAdd(ctl.pending, -(i + 1 - counted) * p.tile);
                    counted = i + 1;
                    if constexpr (!INDEXED) {  // (posted above in index-list mode)
                        StageMeta& mt = ctl.meta[stage];
                        mt.unit = sl.unit;
                        mt.tile = i;
                        mt.flags = (first ? kFirst : 0u) | (i == last ? kLast : 0u);
                        mt.bits = bits;
                    }
                    unsigned char* sk = smem + stage * Sh::kStageBytes;
                    unsigned char* sv = sk + Cons::kTileBytes;
                    unsigned char* sq = sv + Cons::kTileBytes;
                    const int t0 = t_begin + r0;
                    const uint32_t qbytes = first ? (uint32_t)(un.g_here * D * sizeof(Elem)) : 0u;
                    uint32_t kvbytes;
                    if constexpr (INDEXED) {
                        kvbytes = 0u;  // the listed rows were gathered above (cp.async)
                    } else if constexpr (Cons::kSwizzled) {
                        kvbytes = 2u * kHalves * p.tile * 128u;  // whole boxes
                    } else if constexpr (PAGED) {
                        kvbytes = 2u * p.tile * Cons::kRowBytes;  // whole boxes of rows
                    } else {
                        kvbytes = 2u * n * Cons::kRowBytes;
                    }
                    mbar_arrive_expect_tx(&ctl.full[stage], kvbytes + qbytes);
                    if constexpr (INDEXED) {
                    } else if constexpr (PAGED) {
                        const int row = sl.blocks[t0 / p.BS - lb0] * p.BS + t0 % p.BS;
                        if constexpr (Cons::kSwizzled) {
#pragma unroll
                            for (int h = 0; h < kHalves; ++h) {
                                tma_g2s_3d(sk + h * Cons::kTileBytes / kHalves, &kmap, 64 * h,
                                           un.kvh, row, &ctl.full[stage], pol);
                                tma_g2s_3d(sv + h * Cons::kTileBytes / kHalves, &vmap, 64 * h,
                                           un.kvh, row, &ctl.full[stage], pol);
                            }
                        } else {
                            tma_g2s_3d(sk, &kmap, 0, un.kvh, row, &ctl.full[stage], pol);
                            tma_g2s_3d(sv, &vmap, 0, un.kvh, row, &ctl.full[stage], pol);
                        }
                    } else {
                        const size_t rowidx = ((size_t)un.bz * p.Hkv + un.kvh) * p.C + t0;
                        if constexpr (Cons::kSwizzled) {
#pragma unroll
                            for (int h = 0; h < kHalves; ++h) {
                                tma_g2s_2d(sk + h * Cons::kTileBytes / kHalves, &kmap, 64 * h,
                                           (int)rowidx, &ctl.full[stage], pol);
                                tma_g2s_2d(sv + h * Cons::kTileBytes / kHalves, &vmap, 64 * h,
                                           (int)rowidx, &ctl.full[stage], pol);
                            }
                        } else {
                            const uint32_t bytes = (uint32_t)n * Cons::kRowBytes;
                            bulk_g2s(sk, static_cast<const unsigned char*>(p.k) + rowidx * Cons::kRowBytes,
                                     bytes, &ctl.full[stage], pol);
                            bulk_g2s(sv, static_cast<const unsigned char*>(p.v) + rowidx * Cons::kRowBytes,
                                     bytes, &ctl.full[stage], pol);
                        }
                    }
                    if (first)
                        bulk_g2s(sq, static_cast<const Elem*>(p.q) + un.qrow0 * D, qbytes,
                                 &ctl.full[stage], pol);
                    issued_mask |= 1u << stage;
                    last_parity = (last_parity & ~(1u << stage)) | (phase << stage);
                }
                __syncwarp();
                first = false;
                advance();
            }
            if (failed) break;
            __syncwarp();
            mbar_arrive(&ctl.qempty[slot]);  // every lane: done with the slot
        }
        if (!failed && acquire()) {
            if (lane == 0) {
                ctl.meta[stage].flags = kEnd;
                mbar_arrive(&ctl.full[stage]);
                if constexpr (INDEXED) {
                    for (int w = 0; w < kGatherN; ++w)
                        mbar_arrive(&ctl.full[stage]);  // in place of the gather warps' arrivals
                    mbar_arrive(&ctl.gjob[stage]);
                }
            }
            __syncwarp();
        } else {
            failed = true;
        }
        if (failed && lane == 0) {
            *ctl.abort_flag = 1;
            report(p.dev_status, KVD_DEV_TIMEOUT);
            for (int s = 0; s < STAGES; ++s)  // speculated stages never delivered
                if (spec_mask & (1u << s)) mbar_arrive(&ctl.full[s]);
            // The consumers may leave early now: never let the CTA exit while a
            // copy issued here may still be writing the ring.  (On the normal
            // path the consumers have waited for every issued tile before they
            // see the end marker.)
            for (int s = 0; s < STAGES; ++s)
                if (issued_mask & (1u << s)) {
                    const volatile int never = 0;
                    mbar_wait(&ctl.full[s], (last_parity >> s) & 1u, &never);
                }
        }
        return;
    }

    // ================================================================ consumers
    Cons cons;
    int stage = 0;
    uint32_t phase = 0;
    int mb = 0;
    uint32_t mph = 0;
    // Hand the warp's state of a finished unit (or the end of work, -1) to the
    // epilogue warp through a merge buffer.
    auto handoff = [&](int unit) -> bool {
        if (!warp_wait(&ctl.mempty[mb], mph ^ 1u, ctl.abort_flag)) return false;
        if (unit >= 0) cons.finish(merge_mo(mb), merge_ml(mb), warp, lane);
        if (warp == 0 && lane == 0) ctl.mhdr[mb] = unit;
        mbar_arrive(&ctl.mfull[mb]);  // every consumer thread
        if (++mb == MB) {
            mb = 0;
            mph ^= 1u;
        }
        return true;
    };
    while (true) {
        if (!warp_wait(&ctl.full[stage], phase, ctl.abort_flag)) {
            if (lane == 0 && !*ctl.abort_flag) {
                *ctl.abort_flag = 1;
                report(p.dev_status, KVD_DEV_TIMEOUT);
            }
            break;
        }
        const StageMeta mt = ctl.meta[stage];
        if (mt.flags & kEnd) {
            handoff(-1);
            break;
        }
        unsigned char* sb = smem + stage * Sh::kStageBytes;
        if (mt.flags & kFirst) {
            const Unit un = decode_unit(p, G, mt.unit);
            cons.begin(reinterpret_cast<const Elem*>(sb + 2 * Cons::kTileBytes), un.g_here,
                       p.qscale, lane);
        }
        // an empty tile (a speculated tile of a unit that turned out empty) is only released
        const bool wrote =
            mt.bits ? cons.tile(sb, sb + Cons::kTileBytes, mt.bits, warp, lane, p.qscale) : false;
        // generic-proxy writes to the ring must be ordered before the next TMA
        // write into this stage
        if (wrote) fence_proxy_async_smem();
        __syncwarp();
        if (lane == 0) mbar_arrive(&ctl.empty[stage]);
        if (++stage == STAGES) {
            stage = 0;
            phase ^= 1u;
        }
        if ((mt.flags & kLast) && !handoff(mt.unit)) break;
    }
}

}  // namespace kvd
