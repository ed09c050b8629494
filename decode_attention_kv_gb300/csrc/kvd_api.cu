// kvd_api.cu -- the C ABI of libkvd: argument validation, split planning,
// tensor-map set-up and kernel launches.  Allocates nothing, never
// synchronises; every launch goes to the caller's stream.
#include <cudaTypedefs.h>

#include <cstdarg>
#include <cstdio>
#include <cstring>
#include <mutex>

#include "attend_kernel.cuh"
#include "kvd_internal.h"

namespace kvd {
cudaError_t launch_attend_bf16(int D, int G, int mode, const AttendParams& p,
                               const CUtensorMap* kmap, const CUtensorMap* vmap,
                               cudaStream_t stream);
cudaError_t launch_attend_f32(int D, int G, int mode, const AttendParams& p,
                              const CUtensorMap* kmap, const CUtensorMap* vmap,
                              cudaStream_t stream);
AttendGeom attend_geom_bf16(int D, int G);
AttendGeom attend_geom_f32(int D, int G);
cudaError_t launch_attend_fp8(int D, int G, int mode, const AttendParams& p,
                               const CUtensorMap* kmap, const CUtensorMap* vmap,
                               cudaStream_t stream);
cudaError_t launch_attend_small(kvd_dtype dt, int D, int G, const AttendParams& p, int S, int rows,
                                const CUtensorMap* kmap, const CUtensorMap* vmap,
                                cudaStream_t stream);
int small_shared_bytes(kvd_dtype dt, int D, int G, int chunk, int slots, int nwg);
int small_shared_bytes_fp8(int D, int G, int chunk, int slots, int nwg);
int small_shared_bytes_fp4(int D, int G, int chunk, int slots, int nwg);
cudaError_t launch_attend_fp4(int D, int G, int mode, const AttendParams& p,
                               const CUtensorMap* kmap, const CUtensorMap* vmap,
                               cudaStream_t stream);
cudaError_t launch_attend_small_fp4(int D, int G, const AttendParams& p, int S, int rows,
                                    cudaStream_t stream);
cudaError_t launch_attend_small_fp8(int D, int G, const AttendParams& p, int S, int rows,
                                    cudaStream_t stream);
}  // namespace kvd

using namespace kvd;

namespace {

thread_local char g_last_error[512] = "";

kvd_status fail(kvd_status s, const char* fmt, ...) {
    va_list ap;
    va_start(ap, fmt);
    vsnprintf(g_last_error, sizeof g_last_error, fmt, ap);
    va_end(ap);
    return s;
}

kvd_status ok() {
    g_last_error[0] = '\0';
    return KVD_OK;
}

kvd_status cuda_fail(cudaError_t e, const char* what) {
    return fail(KVD_ERR_CUDA, "%s: %s", what, cudaGetErrorString(e));
}

bool aligned(const void* p, size_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }

int elem_size(kvd_dtype dt) { return dt == KVD_BF16 ? 2 : 4; }
bool dtype_ok(kvd_dtype dt) { return dt == KVD_BF16 || dt == KVD_F32; }

// ----------------------------------------------------------------- planning
// Splits of the sequence axis.  The planner is a function of the sizes only
// (not of the device), so that the workspace size queried ahead of a call
// equals what the call needs.  It aims at about kTargetUnits (row, split)
// units per launch -- several per CTA of the persistent grid, so that the
// unit counter balances rows of different lengths -- with splits of at least
// kMinChunk slots, so that the partial rows stay a small fraction of the KV
// traffic.  Unless the caller fixes the number of splits, the last quarter or
// so of the capacity is cut into splits of a quarter of the size: units are
// handed out split-major, so these small units are the last ones taken and
// the CTAs finish within a small unit of each other.
constexpr long long kTargetUnits = 2048;
constexpr long long kGridUnitsHint = 304;  // persistent CTAs on GB300: 2 per SM x 152 SMs
// Small static-buffer launches (one CTA per (row, split), a cluster per row)
constexpr int kSmallSplits = 8;            // splits per row: the portable cluster size
constexpr int kSmallTokens = 384;          // tokens per split, all resident
constexpr int kSmallShared = 113 * 1024;   // shared memory per CTA: two CTAs per SM
constexpr int kMinChunk = 128;
constexpr long long kWideRows = 128;  // row units from which the tail splits are half a chunk

struct Plan {
    int G, HG;      // compile-time group width, head groups per kv head
    int tile;       // tokens per ring stage
    int chunk;      // tokens per split for splits [0, Sb)
    int chunk2;     // tokens per split for splits [Sb, S)
    int Sb;
    int S;          // splits per row
    long long units;
    // workspace: scheduling counters (256 bytes) | partial lse | partial rows
    size_t off_lse, off_po, ws;
};

int group_width(int g) {
    int G = 1;
    while (G < g && G < 8) G <<= 1;
    return G;
}

long long gcd_ll(long long a, long long b) {
    while (b) {
        const long long t = a % b;
        a = b;
        b = t;
    }
    return a;
}

size_t round256(size_t x) { return (x + 255) / 256 * 256; }

AttendGeom geom(kvd_dtype dt, int D, int G) {
    return dt == KVD_BF16 ? attend_geom_bf16(D, G) : attend_geom_f32(D, G);
}

// rows: batch entries (or sequences); cap: most tokens a row can hold (the
// list length for index lists); BS > 0 for the paged layout; `indexed`: a
// split holds at most kMaxBlocks list entries (their slots travel with it).
// tile_max > 0 overrides the element type's tile (quantised rows: 64).
Plan plan_attention(int rows, int Hq, int Hkv, int cap, int D, kvd_dtype dt, int BS,
                    int num_splits, bool indexed = false, int tile_max = 0) {
    Plan pl{};
    const int g = Hq / Hkv;
    pl.G = group_width(g);
    pl.HG = (g + pl.G - 1) / pl.G;
    const int T = tile_max > 0 ? tile_max : geom(dt, D, pl.G).tile_max;
    if (BS > 0) {
        int t = T < BS ? T : BS;
        while (BS % t) --t;  // largest divisor of BS not above T
        pl.tile = t;
    } else {
        pl.tile = T;
    }
    const long long unit = (long long)pl.tile / gcd_ll(pl.tile, 32) * 32;  // lcm(tile, 32)
    long long max_chunk = kMaxChunk / unit * unit;
    if (BS > 0) {
        const long long by_blocks = (long long)(kMaxBlocks - 2) * BS / unit * unit;
        if (by_blocks < max_chunk) max_chunk = by_blocks;
    }
    if (indexed) {
        const long long by_list = (long long)kMaxBlocks / unit * unit;
        if (by_list < max_chunk) max_chunk = by_list;
    }
    if (max_chunk < unit) max_chunk = unit;
    const long long row_units = (long long)rows * Hkv * pl.HG;
    long long chunk;
    if (num_splits > 0) {
        chunk = ((long long)cap + num_splits - 1) / num_splits;
    } else {
        chunk = ((long long)cap * row_units + kTargetUnits - 1) / kTargetUnits;
        if (chunk < kMinChunk) chunk = kMinChunk;
    }
    chunk = (chunk + unit - 1) / unit * unit;
    if (chunk > max_chunk) chunk = max_chunk;
    if (chunk < unit) chunk = unit;
    pl.chunk = pl.chunk2 = (int)chunk;
    pl.S = pl.Sb = (int)(((long long)cap + chunk - 1) / chunk);
    if (pl.S < 1) pl.S = pl.Sb = 1;
    // Tail splits: a quarter chunk, or half a chunk when there are enough
    // rows (128 row units) to spread the late units over the grid by
    // themselves (fewer partial rows to combine); a few long rows -- one
    // sequence's heads -- keep the finer tail, where their valid slots may
    // all sit (a window at the end of the buffer).
    const long long small =
        ((chunk / (row_units >= kWideRows ? 2 : 4)) + unit - 1) / unit * unit;
    // A launch whose units all fit the persistent grid at once (one unit per
    // CTA) keeps equal splits: small tail splits would only give some CTAs a
    // second unit.
    const bool fits_grid = row_units * pl.S <= kGridUnitsHint;
    if (num_splits <= 0 && pl.S > 1 && small < chunk && !fits_grid) {
        const int tail = pl.S / 4 > 1 ? pl.S / 4 : 1;  // big splits turned into small ones
        pl.Sb = pl.S - tail;
        pl.chunk2 = (int)small;
        const long long rest = (long long)cap - (long long)pl.Sb * chunk;
        pl.S = pl.Sb + (int)((rest + small - 1) / small);
    }
    pl.units = row_units * pl.S;
    pl.off_lse = 256;
    if (pl.S > 1) {
        const size_t R = (size_t)rows * Hq;
        pl.off_po = pl.off_lse + round256(R * pl.S * sizeof(float));
        pl.ws = pl.off_po + R * pl.S * D * sizeof(float);
    } else {
        pl.off_po = pl.ws = pl.off_lse;
    }
    return pl;
}

// Slots a sliding window's splits span: from the 64-slot boundary at or below
// the window's first slot to its last, at most W + 63 (and never beyond the
// buffer); the whole buffer without a window.
int window_span(int C, int W) {
    if (W <= 0) return C;
    const long long span = (long long)W + 63;
    return span < C ? (int)span : C;
}

// Plan of a sliding-window call.  Every row of a window holds about W slots
// (unlike the ragged lengths the general plan balances), so the default is
// equal splits, as many as give each persistent CTA one unit (one split per
// row from kGridUnitsHint rows on: no combine).
Plan plan_window(int B, int Hq, int Hkv, int C, int W, int D, kvd_dtype dt, int num_splits) {
    if (num_splits <= 0) {
        const int g = Hq / Hkv, G = group_width(g);
        const long long rows = (long long)B * Hkv * ((g + G - 1) / G);
        const long long s = kGridUnitsHint / rows;
        num_splits = s > 1 ? (int)s : 1;
    }
    return plan_attention(B, Hq, Hkv, window_span(C, W), D, dt, 0, num_splits);
}

// Small static-buffer launch (no caller split count; every split of every row
// resident at once, a cluster of at most 8 CTAs per row that merges the row
// itself).  Splits as equal as the copies allow: whole 64-row boxes for the
// tensor-core layout, any 16 rows for row copies (16-byte mask vectors).
struct SmallPlan {
    bool use;
    bool push;  // every split's partial fits split 0's shared memory
    int nwg;    // consumer warp groups per CTA
    int chunk, S, rows;
};

// Rows of the cache: elements of dt, or quantised rows (row copies of
// D + 16 or D/2 + 16 bytes, 64-row tiles).
enum RowKind { kRowsPlain = 0, kRowsFp8 = 1, kRowsFp4 = 2 };

SmallPlan plan_small(int B, int Hkv, int C, int D, kvd_dtype dt, const Plan& pl, int num_splits,
                     RowKind rk = kRowsPlain) {
    SmallPlan sp{};
    if (num_splits != 0) return sp;
    const bool fp8 = rk != kRowsPlain;
    const int q = (!fp8 && small_uses_mma(dt, pl.G)) ? 64 : 16;  // 64-row boxes or 16-row copies
    const long long rows = (long long)B * Hkv * pl.HG;
    const long long chunk = ((C + kSmallSplits - 1) / kSmallSplits + q - 1) / q * q;
    const long long S = (C + chunk - 1) / chunk;
    auto smem = [&](int slots, int nwg) {
        if (rk == kRowsFp4) return small_shared_bytes_fp4(D, pl.G, (int)chunk, slots, nwg);
        if (rk == kRowsFp8) return small_shared_bytes_fp8(D, pl.G, (int)chunk, slots, nwg);
        return small_shared_bytes(dt, D, pl.G, (int)chunk, slots, nwg);
    };
    // the first layout that fits two CTAs per SM: two consumer warp groups
    // (tensor-core consumers over two or more tiles) before one; partials
    // pushed into split 0 before pulled from the others
    const int nt = (int)((chunk + q - 1) / q);
    const bool two = !fp8 && small_uses_mma(dt, pl.G) && nt >= 2;
    sp.use = false;
    for (int nwg = two ? 2 : 1; nwg >= 1 && !sp.use; --nwg) {
        for (int push = 1; push >= 0 && !sp.use; --push) {
            if (smem(push ? (int)S : 1, nwg) <= kSmallShared) {
                sp.use = true;
                sp.push = push != 0;
                sp.nwg = nwg;
            }
        }
    }
    sp.use = sp.use && chunk <= kSmallTokens && rows * S <= kGridUnitsHint && rows <= 65535;
    sp.chunk = (int)chunk;
    sp.S = (int)S;
    sp.rows = (int)rows;
    return sp;
}

// Attaches the workspace regions of a plan to the kernel parameters.
void attach_workspace(AttendParams& p, const Plan& pl, void* ws) {
    char* base = static_cast<char*>(ws);
    p.sched = reinterpret_cast<uint32_t*>(base);
    p.part_lse = pl.S > 1 ? reinterpret_cast<float*>(base + pl.off_lse) : nullptr;
    p.part_o = pl.S > 1 ? reinterpret_cast<float*>(base + pl.off_po) : nullptr;
    p.units = (int)pl.units;
    p.HG = pl.HG;
    p.tile = pl.tile;
    p.chunk = pl.chunk;
    p.chunk2 = pl.chunk2;
    p.Sb = pl.Sb;
    p.S = pl.S;
    p.direct = pl.S == 1;
}

kvd_status check_workspace(const char* fn, const Plan& pl, void* ws, size_t bytes) {
    if (pl.units >= (1ll << 31)) return fail(KVD_ERR_UNSUPPORTED, "%s: too many (row, split) units", fn);
    if (!ws) return fail(KVD_ERR_WORKSPACE, "%s: workspace required (%zu bytes)", fn, pl.ws);
    if (bytes < pl.ws) return fail(KVD_ERR_WORKSPACE, "%s: workspace %zu < %zu bytes", fn, bytes, pl.ws);
    if (!aligned(ws, 256)) return fail(KVD_ERR_INVALID_ARG, "%s: workspace not 256-byte aligned", fn);
    return KVD_OK;
}

// ---------------------------------------------------------- tensor maps
PFN_cuTensorMapEncodeTiled_v12000 g_encode = nullptr;
std::once_flag g_encode_once;
cudaError_t g_encode_err = cudaSuccess;

cudaError_t get_encoder() {
    std::call_once(g_encode_once, [] {
        void* fn = nullptr;
        cudaDriverEntryPointQueryResult q{};
        g_encode_err = cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000,
                                                        cudaEnableDefault, &q);
        if (g_encode_err == cudaSuccess && q != cudaDriverEntryPointSuccess)
            g_encode_err = cudaErrorNotSupported;
        g_encode = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(fn);
    });
    return g_encode_err;
}

// Tensor map over a K or V cache.
//  paged [NB, BS, Hkv, D] -> 3-D (D, Hkv, NB*BS): a box is one kv head of
//    `tile` consecutive slots;
//  static buffer [B, Hkv, C, D] -> 2-D (D, B*Hkv*C): a box is `tile`
//    consecutive rows of one (b, kv head).
// With `swizzle` the box is 64 elements wide (128 bytes, the 128-byte swizzle
// the tensor-core kernel reads with ldmatrix), else the whole head_dim.
kvd_status make_cache_map(CUtensorMap* map, const void* cache, kvd_dtype dt, bool paged,
                          long long rows, int Hkv, int D, int tile, bool swizzle) {
    const cudaError_t e = get_encoder();
    if (e != cudaSuccess || !g_encode) return cuda_fail(e, "cuTensorMapEncodeTiled lookup");
    const int es = elem_size(dt);
    const cuuint32_t inner = swizzle ? 64u : (cuuint32_t)D;
    CUresult r;
    const CUtensorMapDataType type =
        dt == KVD_BF16 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16 : CU_TENSOR_MAP_DATA_TYPE_FLOAT32;
    const CUtensorMapSwizzle sw = swizzle ? CU_TENSOR_MAP_SWIZZLE_128B : CU_TENSOR_MAP_SWIZZLE_NONE;
    if (paged) {
        const cuuint64_t dims[3] = {(cuuint64_t)D, (cuuint64_t)Hkv, (cuuint64_t)rows};
        const cuuint64_t strides[2] = {(cuuint64_t)D * es, (cuuint64_t)Hkv * D * es};
        const cuuint32_t box[3] = {inner, 1u, (cuuint32_t)tile};
        const cuuint32_t estr[3] = {1u, 1u, 1u};
        r = g_encode(map, type, 3, const_cast<void*>(cache), dims, strides, box, estr,
                     CU_TENSOR_MAP_INTERLEAVE_NONE, sw, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                     CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    } else {
        const cuuint64_t dims[2] = {(cuuint64_t)D, (cuuint64_t)rows};
        const cuuint64_t strides[1] = {(cuuint64_t)D * es};
        const cuuint32_t box[2] = {inner, (cuuint32_t)tile};
        const cuuint32_t estr[2] = {1u, 1u};
        r = g_encode(map, type, 2, const_cast<void*>(cache), dims, strides, box, estr,
                     CU_TENSOR_MAP_INTERLEAVE_NONE, sw, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                     CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    }
    if (r != CUDA_SUCCESS) return fail(KVD_ERR_CUDA, "cuTensorMapEncodeTiled failed (%d)", (int)r);
    return KVD_OK;
}

cudaError_t launch_attend(kvd_dtype dt, int D, int G, int mode, const AttendParams& p,
                          const CUtensorMap* kmap, const CUtensorMap* vmap, cudaStream_t s) {
    return dt == KVD_BF16 ? launch_attend_bf16(D, G, mode, p, kmap, vmap, s)
                          : launch_attend_f32(D, G, mode, p, kmap, vmap, s);
}

kvd_status check_attention_shape(int Hq, int Hkv, int D, kvd_dtype dt) {
    if (Hq < 1 || Hkv < 1) return fail(KVD_ERR_INVALID_ARG, "head counts must be >= 1");
    if (Hq % Hkv) return fail(KVD_ERR_INVALID_ARG, "Hq (%d) must be a multiple of Hkv (%d)", Hq, Hkv);
    if (!dtype_ok(dt)) return fail(KVD_ERR_INVALID_ARG, "unknown dtype %d", (int)dt);
    if (D != 64 && D != 128) return fail(KVD_ERR_UNSUPPORTED, "head_dim %d (supported: 64, 128)", D);
    return KVD_OK;
}

// What the *_plan queries report (kvd_plan in kvd.h).
void put_plan(const Plan& pl, bool small, kvd_plan* out) {
    std::memset(out, 0, sizeof *out);
    if (small) {
        out->splits = 0;  // one launch, merged inside thread-block clusters: no partial rows
        out->launches = 1;
    } else {
        out->splits = pl.S;
        out->launches = pl.S > 1 ? 2 : 1;
        out->lse_offset = pl.S > 1 ? pl.off_lse : 0;
        out->o_offset = pl.S > 1 ? pl.off_po : 0;
    }
    out->counter_bytes = small ? 0 : pl.off_lse;
}

}  // namespace

namespace kvd {
// Lets the other translation units of the library report a host-side error
// through kvd_last_error().
void set_last_error(const char* msg) {
    snprintf(g_last_error, sizeof g_last_error, "%s", msg);
}
}  // namespace kvd

// ===================================================================== C ABI
extern "C" {

const char* kvd_status_string(kvd_status s) {
    switch (s) {
        case KVD_OK: return "KVD_OK";
        case KVD_ERR_INVALID_ARG: return "KVD_ERR_INVALID_ARG";
        case KVD_ERR_UNSUPPORTED: return "KVD_ERR_UNSUPPORTED";
        case KVD_ERR_WORKSPACE: return "KVD_ERR_WORKSPACE";
        case KVD_ERR_CUDA: return "KVD_ERR_CUDA";
    }
    return "KVD_ERR_UNKNOWN";
}

const char* kvd_last_error(void) { return g_last_error; }

int kvd_version(void) { return 10000; }

kvd_status kvd_append(void* k_cache, void* v_cache, const void* k_new, const void* v_new,
                      const int32_t* pos, uint8_t* mask, int B, int Hkv, int C, int D,
                      kvd_dtype dtype, int32_t* dev_status, kvd_stream_t stream) {
    if (!k_cache || !v_cache || !k_new || !v_new || !pos)
        return fail(KVD_ERR_INVALID_ARG, "kvd_append: null pointer");
    if (B < 1 || Hkv < 1 || C < 1 || D < 1)
        return fail(KVD_ERR_INVALID_ARG, "kvd_append: sizes must be >= 1");
    if (!dtype_ok(dtype)) return fail(KVD_ERR_INVALID_ARG, "kvd_append: unknown dtype");
    const long long row = (long long)D * elem_size(dtype);
    if (row % 16) return fail(KVD_ERR_INVALID_ARG, "kvd_append: D*elem must be a multiple of 16 bytes");
    if (!aligned(k_cache, 16) || !aligned(v_cache, 16) || !aligned(k_new, 16) || !aligned(v_new, 16) ||
        !aligned(pos, 4) || !aligned(dev_status, 4))
        return fail(KVD_ERR_INVALID_ARG, "kvd_append: misaligned pointer");
    if (B > 65535) return fail(KVD_ERR_UNSUPPORTED, "kvd_append: B > 65535");
    const cudaError_t e = launch_append(k_cache, v_cache, k_new, v_new, pos, mask, B, Hkv, C,
                                        (int)row, dev_status, (cudaStream_t)stream);
    if (e != cudaSuccess) return cuda_fail(e, "kvd_append launch");
    return ok();
}

kvd_status kvd_append_paged(void* key_cache, void* value_cache, const void* k_new,
                            const void* v_new, const int32_t* block_tables,
                            const int32_t* seq_offset, const int32_t* pos, int Q, int NB, int BS,
                            int cols, int Hkv, int D, kvd_dtype dtype, int32_t* dev_status,
                            kvd_stream_t stream) {
    const char* fn = "kvd_append_paged";
    if (Q < 0 || NB < 1 || BS < 1 || cols < 1 || Hkv < 1 || D < 1)
        return fail(KVD_ERR_INVALID_ARG, "%s: Q >= 0 and NB, BS, cols, Hkv, D >= 1 required", fn);
    if (!dtype_ok(dtype)) return fail(KVD_ERR_INVALID_ARG, "%s: unknown dtype", fn);
    if (Q == 0) return ok();
    if (!key_cache || !value_cache || !k_new || !v_new || !block_tables || !pos)
        return fail(KVD_ERR_INVALID_ARG, "%s: null pointer", fn);
    const long long row = (long long)Hkv * D * elem_size(dtype);
    if (row % 16) return fail(KVD_ERR_INVALID_ARG, "%s: Hkv*D*elem must be a multiple of 16 bytes", fn);
    if (row >= (1ll << 31)) return fail(KVD_ERR_UNSUPPORTED, "%s: row too large", fn);
    if (!aligned(key_cache, 16) || !aligned(value_cache, 16) || !aligned(k_new, 16) ||
        !aligned(v_new, 16) || !aligned(block_tables, 4) || !aligned(seq_offset, 4) ||
        !aligned(pos, 4) || !aligned(dev_status, 4))
        return fail(KVD_ERR_INVALID_ARG, "%s: misaligned pointer", fn);
    if (Q > 65535) return fail(KVD_ERR_UNSUPPORTED, "%s: Q > 65535", fn);
    const cudaError_t e = launch_append_paged(key_cache, value_cache, k_new, v_new, block_tables,
                                              seq_offset, pos, Q, NB, BS, cols, (int)row,
                                              dev_status, (cudaStream_t)stream);
    if (e != cudaSuccess) return cuda_fail(e, "kvd_append_paged launch");
    return ok();
}

kvd_status kvd_copy_prefix(const void* const* k_src, const void* const* v_src, void* const* k_dst,
                           void* const* v_dst, uint8_t* const* masks, const int32_t* n, int L,
                           int B, int Hkv, int C_src, int C_dst, int D, kvd_dtype dtype,
                           int32_t* dev_status, kvd_stream_t stream) {
    if (!k_src || !v_src || !k_dst || !v_dst || !n)
        return fail(KVD_ERR_INVALID_ARG, "kvd_copy_prefix: null pointer");
    if (L < 1 || B < 1 || Hkv < 1 || C_src < 1 || C_dst < 1 || D < 1)
        return fail(KVD_ERR_INVALID_ARG, "kvd_copy_prefix: sizes must be >= 1");
    if (!dtype_ok(dtype)) return fail(KVD_ERR_INVALID_ARG, "kvd_copy_prefix: unknown dtype");
    const long long row = (long long)D * elem_size(dtype);
    if (row % 16) return fail(KVD_ERR_INVALID_ARG, "kvd_copy_prefix: D*elem must be a multiple of 16 bytes");
    if (!aligned(k_src, 8) || !aligned(v_src, 8) || !aligned(k_dst, 8) || !aligned(v_dst, 8) ||
        !aligned(masks, 8) || !aligned(n, 4) || !aligned(dev_status, 4))
        return fail(KVD_ERR_INVALID_ARG, "kvd_copy_prefix: misaligned pointer");
    if ((long long)B * Hkv > 65535 || L > 32767)
        return fail(KVD_ERR_UNSUPPORTED, "kvd_copy_prefix: B*Hkv > 65535 or L > 32767");
    const cudaError_t e = launch_copy_prefix(k_src, v_src, k_dst, v_dst, masks, n, L, B, Hkv, C_src,
                                             C_dst, (int)row, dev_status, (cudaStream_t)stream);
    if (e != cudaSuccess) return cuda_fail(e, "kvd_copy_prefix launch");
    return ok();
}

int kvd_attend_masked_launches(int B, int Hq, int Hkv, int C, int D, kvd_dtype dtype,
                               int num_splits) {
    if (B < 1 || C < 1 || num_splits < 0 || check_attention_shape(Hq, Hkv, D, dtype) != KVD_OK)
        return 0;
    const Plan pl = plan_attention(B, Hq, Hkv, C, D, dtype, 0, num_splits);
    if (plan_small(B, Hkv, C, D, dtype, pl, num_splits).use) return 1;
    return pl.S > 1 ? 2 : 1;
}

size_t kvd_attend_masked_workspace_bytes(int B, int Hq, int Hkv, int C, int D, kvd_dtype dtype,
                                         int num_splits) {
    if (B < 1 || C < 1 || check_attention_shape(Hq, Hkv, D, dtype) != KVD_OK) return 0;
    return plan_attention(B, Hq, Hkv, C, D, dtype, 0, num_splits).ws;
}

kvd_status kvd_attend_masked_plan(int B, int Hq, int Hkv, int C, int D, kvd_dtype dtype,
                                  int num_splits, kvd_plan* plan) {
    if (!plan)
        return fail(KVD_ERR_INVALID_ARG, "kvd_attend_masked_plan: null pointer");
    if (B < 1 || C < 1 || num_splits < 0)
        return fail(KVD_ERR_INVALID_ARG, "kvd_attend_masked_plan: B, C >= 1 and num_splits >= 0 required");
    const kvd_status st = check_attention_shape(Hq, Hkv, D, dtype);
    if (st != KVD_OK) return st;
    const Plan pl = plan_attention(B, Hq, Hkv, C, D, dtype, 0, num_splits);
    put_plan(pl, plan_small(B, Hkv, C, D, dtype, pl, num_splits).use, plan);
    return ok();
}

}  // extern "C"

namespace {
// kvd_attend_masked, with the step's append fused into the launch when k_new
// is given (the caller has checked that a kv head has one head group).
kvd_status attend_masked_impl(const char* fn, const void* q, const void* k_cache,
                              const void* v_cache, const uint8_t* mask, void* out,
                              float* lse_out, int B, int Hq, int Hkv, int C, int D, float scale,
                              kvd_dtype dtype, int num_splits, void* workspace,
                              size_t workspace_bytes, int32_t* dev_status, kvd_stream_t stream,
                              const void* k_new, const void* v_new, const int32_t* pos,
                              bool out_f32 = false, int win = 0,
                              const int32_t* win_last = nullptr) {
    kvd_status st = check_attention_shape(Hq, Hkv, D, dtype);
    if (st != KVD_OK) return st;
    if (B < 0 || C < 1) return fail(KVD_ERR_INVALID_ARG, "%s: B >= 0 and C >= 1 required", fn);
    if (win < 0) return fail(KVD_ERR_INVALID_ARG, "%s: W >= 1 required", fn);
    if (B == 0) return ok();
    if (!q || !k_cache || !v_cache || !mask || !out || (win > 0 && !win_last))
        return fail(KVD_ERR_INVALID_ARG, "%s: null pointer", fn);
    if (!aligned(q, 16) || !aligned(k_cache, 16) || !aligned(v_cache, 16) || !aligned(out, 16) ||
        !aligned(lse_out, 4) || !aligned(dev_status, 4) || !aligned(win_last, 4))
        return fail(KVD_ERR_INVALID_ARG, "%s: misaligned pointer", fn);
    if (num_splits < 0) return fail(KVD_ERR_INVALID_ARG, "%s: num_splits < 0", fn);
    const Plan pl = win > 0 ? plan_window(B, Hq, Hkv, C, win, D, dtype, num_splits)
                            : plan_attention(B, Hq, Hkv, C, D, dtype, 0, num_splits);
    st = check_workspace(fn, pl, workspace, workspace_bytes);
    if (st != KVD_OK) return st;
    AttendParams p{};
    p.q = q;
    p.k = k_cache;
    p.v = v_cache;
    p.mask = mask;
    p.out = out;
    p.lse_out = lse_out;
    p.dev_status = dev_status;
    p.Hq = Hq;
    p.Hkv = Hkv;
    p.g = Hq / Hkv;
    p.C = C;
    p.mask_vec = (C % 16 == 0) && aligned(mask, 16);
    p.qscale = scale * kLog2e;
    p.k_new = k_new;
    p.v_new = v_new;
    p.pos = k_new ? pos : nullptr;
    p.mask_w = const_cast<uint8_t*>(mask);
    p.out_f32 = out_f32 ? 1 : 0;
    p.win = win;
    p.win_last = win > 0 ? win_last : nullptr;
    attach_workspace(p, pl, workspace);
    CUtensorMap kmap, vmap;
    std::memset(&kmap, 0, sizeof kmap);
    std::memset(&vmap, 0, sizeof vmap);
    // the one-launch kernel holds whole splits from slot 0: not for windows
    const SmallPlan sp = win > 0 ? SmallPlan{} : plan_small(B, Hkv, C, D, dtype, pl, num_splits);
    if (sp.use ? small_uses_mma(dtype, pl.G) : attend_uses_mma(dtype, pl.G)) {
        // 128-byte-swizzled boxes of 64 dims x (tile rows) for the tensor-core consumers
        const long long rows = (long long)B * Hkv * C;
        if (rows >= (1ll << 31))
            return fail(KVD_ERR_UNSUPPORTED, "%s: B*Hkv*C >= 2^31 rows", fn);
        const int box_rows = sp.use ? 64 : pl.tile;
        st = make_cache_map(&kmap, k_cache, dtype, false, rows, Hkv, D, box_rows, true);
        if (st != KVD_OK) return st;
        st = make_cache_map(&vmap, v_cache, dtype, false, rows, Hkv, D, box_rows, true);
        if (st != KVD_OK) return st;
    }
    if (sp.use) {
        AttendParams ps = p;
        ps.chunk = sp.chunk;
        ps.S = sp.S;
        ps.small_push = sp.push ? 1 : 0;
        ps.small_nwg = sp.nwg;
        const cudaError_t e = launch_attend_small(dtype, D, pl.G, ps, sp.S, sp.rows, &kmap, &vmap,
                                                  (cudaStream_t)stream);
        if (e != cudaSuccess) return cuda_fail(e, fn);
        return ok();
    }
    cudaError_t e = launch_attend(dtype, D, pl.G, kModeMasked, p, &kmap, &vmap, (cudaStream_t)stream);
    if (e != cudaSuccess) return cuda_fail(e, fn);
    if (pl.S > 1) {
        e = launch_combine(p.part_o, p.part_lse, out, lse_out, B * Hq, pl.S, D,
                           out_f32 ? KVD_F32 : dtype, (cudaStream_t)stream);
        if (e != cudaSuccess) return cuda_fail(e, fn);
    }
    return ok();
}

}  // namespace

extern "C" {

kvd_status kvd_attend_masked(const void* q, const void* k_cache, const void* v_cache,
                             const uint8_t* mask, void* out, float* lse_out, int B, int Hq,
                             int Hkv, int C, int D, float scale, kvd_dtype dtype, int num_splits,
                             void* workspace, size_t workspace_bytes, int32_t* dev_status,
                             kvd_stream_t stream) {
    return attend_masked_impl("kvd_attend_masked", q, k_cache, v_cache, mask, out, lse_out, B, Hq,
                              Hkv, C, D, scale, dtype, num_splits, workspace, workspace_bytes,
                              dev_status, stream, nullptr, nullptr, nullptr);
}

kvd_status kvd_attend_masked_partial(const void* q, const void* k_cache, const void* v_cache,
                                     const uint8_t* mask, float* out, float* lse_out, int B,
                                     int Hq, int Hkv, int C, int D, float scale, kvd_dtype dtype,
                                     int num_splits, void* workspace, size_t workspace_bytes,
                                     int32_t* dev_status, kvd_stream_t stream) {
    if (B > 0 && !lse_out)
        return fail(KVD_ERR_INVALID_ARG, "kvd_attend_masked_partial: lse_out required");
    return attend_masked_impl("kvd_attend_masked_partial", q, k_cache, v_cache, mask, out, lse_out,
                              B, Hq, Hkv, C, D, scale, dtype, num_splits, workspace,
                              workspace_bytes, dev_status, stream, nullptr, nullptr, nullptr,
                              true);
}

kvd_status kvd_append_attend_masked(const void* q, void* k_cache, void* v_cache, uint8_t* mask,
                                    const void* k_new, const void* v_new, const int32_t* pos,
                                    void* out, float* lse_out, int B, int Hq, int Hkv, int C,
                                    int D, float scale, kvd_dtype dtype, int num_splits,
                                    void* workspace, size_t workspace_bytes, int32_t* dev_status,
                                    kvd_stream_t stream) {
    const char* fn = "kvd_append_attend_masked";
    if (B == 0) return ok();
    if (!k_new || !v_new || !pos) return fail(KVD_ERR_INVALID_ARG, "%s: null pointer", fn);
    if (!aligned(k_new, 16) || !aligned(v_new, 16) || !aligned(pos, 4))
        return fail(KVD_ERR_INVALID_ARG, "%s: misaligned pointer", fn);
    const kvd_status st = check_attention_shape(Hq, Hkv, D, dtype);
    if (st != KVD_OK) return st;
    if (group_width(Hq / Hkv) < Hq / Hkv) {
        // several head groups per kv head: the append first, then the attention
        const kvd_status sa = kvd_append(k_cache, v_cache, k_new, v_new, pos, mask, B, Hkv, C, D,
                                         dtype, dev_status, stream);
        if (sa != KVD_OK) return sa;
        return attend_masked_impl(fn, q, k_cache, v_cache, mask, out, lse_out, B, Hq, Hkv, C, D,
                                  scale, dtype, num_splits, workspace, workspace_bytes, dev_status,
                                  stream, nullptr, nullptr, nullptr);
    }
    return attend_masked_impl(fn, q, k_cache, v_cache, mask, out, lse_out, B, Hq, Hkv, C, D, scale,
                              dtype, num_splits, workspace, workspace_bytes, dev_status, stream,
                              k_new, v_new, pos);
}

size_t kvd_attend_window_workspace_bytes(int B, int Hq, int Hkv, int C, int D, int W,
                                         kvd_dtype dtype, int num_splits) {
    if (B < 1 || C < 1 || W < 1 || check_attention_shape(Hq, Hkv, D, dtype) != KVD_OK) return 0;
    return plan_window(B, Hq, Hkv, C, W, D, dtype, num_splits).ws;
}

kvd_status kvd_attend_window_plan(int B, int Hq, int Hkv, int C, int D, int W, kvd_dtype dtype,
                                  int num_splits, kvd_plan* plan) {
    if (!plan) return fail(KVD_ERR_INVALID_ARG, "kvd_attend_window_plan: null pointer");
    if (B < 1 || C < 1 || W < 1 || num_splits < 0)
        return fail(KVD_ERR_INVALID_ARG,
                    "kvd_attend_window_plan: B, C, W >= 1 and num_splits >= 0 required");
    const kvd_status st = check_attention_shape(Hq, Hkv, D, dtype);
    if (st != KVD_OK) return st;
    put_plan(plan_window(B, Hq, Hkv, C, W, D, dtype, num_splits), false, plan);
    return ok();
}

kvd_status kvd_attend_window(const void* q, const void* k_cache, const void* v_cache,
                             const uint8_t* mask, const int32_t* last, void* out, float* lse_out,
                             int B, int Hq, int Hkv, int C, int D, int W, float scale,
                             kvd_dtype dtype, int num_splits, void* workspace,
                             size_t workspace_bytes, int32_t* dev_status, kvd_stream_t stream) {
    if (W < 1) return fail(KVD_ERR_INVALID_ARG, "kvd_attend_window: W >= 1 required");
    return attend_masked_impl("kvd_attend_window", q, k_cache, v_cache, mask, out, lse_out, B, Hq,
                              Hkv, C, D, scale, dtype, num_splits, workspace, workspace_bytes,
                              dev_status, stream, nullptr, nullptr, nullptr, false, W, last);
}

kvd_status kvd_append_attend_window(const void* q, void* k_cache, void* v_cache, uint8_t* mask,
                                    const void* k_new, const void* v_new, const int32_t* pos,
                                    void* out, float* lse_out, int B, int Hq, int Hkv, int C,
                                    int D, int W, float scale, kvd_dtype dtype, int num_splits,
                                    void* workspace, size_t workspace_bytes, int32_t* dev_status,
                                    kvd_stream_t stream) {
    const char* fn = "kvd_append_attend_window";
    if (W < 1) return fail(KVD_ERR_INVALID_ARG, "%s: W >= 1 required", fn);
    if (B == 0) return ok();
    if (!k_new || !v_new || !pos) return fail(KVD_ERR_INVALID_ARG, "%s: null pointer", fn);
    if (!aligned(k_new, 16) || !aligned(v_new, 16) || !aligned(pos, 4))
        return fail(KVD_ERR_INVALID_ARG, "%s: misaligned pointer", fn);
    const kvd_status st = check_attention_shape(Hq, Hkv, D, dtype);
    if (st != KVD_OK) return st;
    if (group_width(Hq / Hkv) < Hq / Hkv) {
        // several head groups per kv head: the append first, then the attention
        const kvd_status sa = kvd_append(k_cache, v_cache, k_new, v_new, pos, mask, B, Hkv, C, D,
                                         dtype, dev_status, stream);
        if (sa != KVD_OK) return sa;
        return attend_masked_impl(fn, q, k_cache, v_cache, mask, out, lse_out, B, Hq, Hkv, C, D,
                                  scale, dtype, num_splits, workspace, workspace_bytes, dev_status,
                                  stream, nullptr, nullptr, nullptr, false, W, pos);
    }
    return attend_masked_impl(fn, q, k_cache, v_cache, mask, out, lse_out, B, Hq, Hkv, C, D, scale,
                              dtype, num_splits, workspace, workspace_bytes, dev_status, stream,
                              k_new, v_new, pos, false, W, pos);
}

}  // extern "C"

namespace {

kvd_status append_quant(const char* fn, bool fp4, void* k_cache, void* v_cache, const void* k_new,
                        const void* v_new, const int32_t* pos, uint8_t* mask, int B, int Hkv,
                        int C, int D, kvd_dtype new_dtype, int32_t* dev_status,
                        kvd_stream_t stream) {
    if (!k_cache || !v_cache || !k_new || !v_new || !pos)
        return fail(KVD_ERR_INVALID_ARG, "%s: null pointer", fn);
    if (B < 1 || Hkv < 1 || C < 1) return fail(KVD_ERR_INVALID_ARG, "%s: sizes must be >= 1", fn);
    if (!dtype_ok(new_dtype)) return fail(KVD_ERR_INVALID_ARG, "%s: unknown dtype", fn);
    if (D != 64 && D != 128) return fail(KVD_ERR_UNSUPPORTED, "%s: head_dim %d (supported: 64, 128)", fn, D);
    if (!aligned(k_cache, 16) || !aligned(v_cache, 16) || !aligned(k_new, 16) || !aligned(v_new, 16) ||
        !aligned(pos, 4) || !aligned(dev_status, 4))
        return fail(KVD_ERR_INVALID_ARG, "%s: misaligned pointer", fn);
    if (2ll * B * Hkv > (1ll << 33)) return fail(KVD_ERR_UNSUPPORTED, "%s: B*Hkv too large", fn);
    const cudaError_t e =
        fp4 ? launch_append_fp4(k_cache, v_cache, k_new, v_new, pos, mask, B, Hkv, C, D, new_dtype,
                                dev_status, (cudaStream_t)stream)
            : launch_append_fp8(k_cache, v_cache, k_new, v_new, pos, mask, B, Hkv, C, D, new_dtype,
                                dev_status, (cudaStream_t)stream);
    if (e != cudaSuccess) return cuda_fail(e, fp4 ? "kvd_append_fp4 launch" : "kvd_append_fp8 launch");
    return ok();
}

constexpr int kQuantTile = 64;  // tokens per ring stage over quantised rows

kvd_status quant_plan(const char* fn, RowKind rk, int B, int Hq, int Hkv, int C, int D,
                      int num_splits, kvd_plan* plan) {
    if (!plan) return fail(KVD_ERR_INVALID_ARG, "%s: null pointer", fn);
    if (B < 1 || C < 1 || num_splits < 0)
        return fail(KVD_ERR_INVALID_ARG, "%s: B, C >= 1 and num_splits >= 0 required", fn);
    const kvd_status st = check_attention_shape(Hq, Hkv, D, KVD_BF16);
    if (st != KVD_OK) return st;
    const Plan pl = plan_attention(B, Hq, Hkv, C, D, KVD_BF16, 0, num_splits, false, kQuantTile);
    put_plan(pl, plan_small(B, Hkv, C, D, KVD_BF16, pl, num_splits, rk).use, plan);
    return ok();
}

kvd_status attend_quant(const char* fn, RowKind rk, const void* q, const void* k_cache,
                        const void* v_cache, const uint8_t* mask, void* out, float* lse_out, int B,
                        int Hq, int Hkv, int C, int D, float scale, int num_splits,
                        void* workspace, size_t workspace_bytes, int32_t* dev_status,
                        kvd_stream_t stream) {
    kvd_status st = check_attention_shape(Hq, Hkv, D, KVD_BF16);
    if (st != KVD_OK) return st;
    if (B < 0 || C < 1) return fail(KVD_ERR_INVALID_ARG, "%s: B >= 0 and C >= 1 required", fn);
    if (B == 0) return ok();
    if (!q || !k_cache || !v_cache || !mask || !out)
        return fail(KVD_ERR_INVALID_ARG, "%s: null pointer", fn);
    if (!aligned(q, 16) || !aligned(k_cache, 16) || !aligned(v_cache, 16) || !aligned(out, 16) ||
        !aligned(lse_out, 4) || !aligned(dev_status, 4))
        return fail(KVD_ERR_INVALID_ARG, "%s: misaligned pointer", fn);
    if (num_splits < 0) return fail(KVD_ERR_INVALID_ARG, "%s: num_splits < 0", fn);
    const Plan pl = plan_attention(B, Hq, Hkv, C, D, KVD_BF16, 0, num_splits, false, kQuantTile);
    st = check_workspace(fn, pl, workspace, workspace_bytes);
    if (st != KVD_OK) return st;
    AttendParams p{};
    p.q = q;
    p.k = k_cache;
    p.v = v_cache;
    p.mask = mask;
    p.out = out;
    p.lse_out = lse_out;
    p.dev_status = dev_status;
    p.Hq = Hq;
    p.Hkv = Hkv;
    p.g = Hq / Hkv;
    p.C = C;
    p.mask_vec = (C % 16 == 0) && aligned(mask, 16);
    p.qscale = scale * kLog2e;
    attach_workspace(p, pl, workspace);
    const bool fp4 = rk == kRowsFp4;
    const SmallPlan sp = plan_small(B, Hkv, C, D, KVD_BF16, pl, num_splits, rk);
    if (sp.use) {
        AttendParams ps = p;
        ps.chunk = sp.chunk;
        ps.S = sp.S;
        ps.small_push = sp.push ? 1 : 0;
        ps.small_nwg = sp.nwg;
        const cudaError_t es =
            fp4 ? launch_attend_small_fp4(D, pl.G, ps, sp.S, sp.rows, (cudaStream_t)stream)
                : launch_attend_small_fp8(D, pl.G, ps, sp.S, sp.rows, (cudaStream_t)stream);
        if (es != cudaSuccess) return cuda_fail(es, fn);
        return ok();
    }
    CUtensorMap none;
    std::memset(&none, 0, sizeof none);
    cudaError_t e = fp4 ? launch_attend_fp4(D, pl.G, kModeMasked, p, &none, &none, (cudaStream_t)stream)
                        : launch_attend_fp8(D, pl.G, kModeMasked, p, &none, &none, (cudaStream_t)stream);
    if (e != cudaSuccess) return cuda_fail(e, fn);
    if (pl.S > 1) {
        e = launch_combine(p.part_o, p.part_lse, out, lse_out, B * Hq, pl.S, D, KVD_BF16,
                           (cudaStream_t)stream);
        if (e != cudaSuccess) return cuda_fail(e, "combine launch");
    }
    return ok();
}

size_t quant_workspace_bytes(int B, int Hq, int Hkv, int C, int D, int num_splits) {
    if (B < 1 || C < 1 || check_attention_shape(Hq, Hkv, D, KVD_BF16) != KVD_OK) return 0;
    return plan_attention(B, Hq, Hkv, C, D, KVD_BF16, 0, num_splits, false, kQuantTile).ws;
}

int quant_row_bytes(RowKind rk, int D) { return (rk == kRowsFp4 ? D / 2 : D) + 16; }

// 3-D tensor map over the quantised rows of a paged cache [NB*BS, Hkv, RB]
// (bytes): boxes of `tile` whole rows of one kv head, unswizzled.
kvd_status make_row_map(CUtensorMap* map, const void* cache, long long rows, int Hkv, int RB,
                        int tile) {
    const cudaError_t e = get_encoder();
    if (e != cudaSuccess || !g_encode) return cuda_fail(e, "cuTensorMapEncodeTiled lookup");
    const cuuint64_t dims[3] = {(cuuint64_t)RB, (cuuint64_t)Hkv, (cuuint64_t)rows};
    const cuuint64_t strides[2] = {(cuuint64_t)RB, (cuuint64_t)Hkv * RB};
    const cuuint32_t box[3] = {(cuuint32_t)RB, 1u, (cuuint32_t)tile};
    const cuuint32_t estr[3] = {1u, 1u, 1u};
    const CUresult r = g_encode(map, CU_TENSOR_MAP_DATA_TYPE_UINT8, 3, const_cast<void*>(cache),
                                dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                                CU_TENSOR_MAP_SWIZZLE_NONE, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                                CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    if (r != CUDA_SUCCESS) return fail(KVD_ERR_CUDA, "cuTensorMapEncodeTiled failed (%d)", (int)r);
    return KVD_OK;
}

kvd_status append_paged_quant(const char* fn, bool fp4, void* key_cache, void* value_cache,
                              const void* k_new, const void* v_new, const int32_t* block_tables,
                              const int32_t* seq_offset, const int32_t* pos, int Q, int NB,
                              int BS, int cols, int Hkv, int D, kvd_dtype new_dtype,
                              int32_t* dev_status, kvd_stream_t stream) {
    if (Q < 0 || NB < 1 || BS < 1 || cols < 1 || Hkv < 1)
        return fail(KVD_ERR_INVALID_ARG, "%s: Q >= 0 and NB, BS, cols, Hkv >= 1 required", fn);
    if (Q == 0) return ok();
    if (!key_cache || !value_cache || !k_new || !v_new || !block_tables || !pos)
        return fail(KVD_ERR_INVALID_ARG, "%s: null pointer", fn);
    if (!dtype_ok(new_dtype)) return fail(KVD_ERR_INVALID_ARG, "%s: unknown dtype", fn);
    if (D != 64 && D != 128) return fail(KVD_ERR_UNSUPPORTED, "%s: head_dim %d (supported: 64, 128)", fn, D);
    if (!aligned(key_cache, 16) || !aligned(value_cache, 16) || !aligned(k_new, 16) ||
        !aligned(v_new, 16) || !aligned(block_tables, 4) || !aligned(seq_offset, 4) ||
        !aligned(pos, 4) || !aligned(dev_status, 4))
        return fail(KVD_ERR_INVALID_ARG, "%s: misaligned pointer", fn);
    if (2ll * Q * Hkv > (1ll << 33)) return fail(KVD_ERR_UNSUPPORTED, "%s: Q*Hkv too large", fn);
    const cudaError_t e =
        fp4 ? launch_append_fp4(key_cache, value_cache, k_new, v_new, pos, nullptr, Q, Hkv, 0, D,
                                new_dtype, dev_status, (cudaStream_t)stream, block_tables,
                                seq_offset, NB, BS, cols)
            : launch_append_fp8(key_cache, value_cache, k_new, v_new, pos, nullptr, Q, Hkv, 0, D,
                                new_dtype, dev_status, (cudaStream_t)stream, block_tables,
                                seq_offset, NB, BS, cols);
    if (e != cudaSuccess) return cuda_fail(e, fn);
    return ok();
}

// Paged caches of quantised rows: the tensor-core consumers' dependent chain,
// not HBM, sets the tile rate (about 1.4 us per 64-row tile per CTA), so
// long units leave a long tail; the default is equal splits of kQuantPagedChunk
// slots (four tiles).  Measured on 64 sequences of 1..4096 tokens, 8 kv heads,
// E4M3 rows: the general plan's 5 splits 110 us, 8: 101, 11: 92, 16: 84, 22:
// 89, 32: 101 us per attention call; E2M1 rows 87, 77, 73, 76, 82, 95 us.
constexpr int kQuantPagedChunk = 256;

Plan paged_quant_plan(int Q, int Hq, int Hkv, int BS, int cols, int D, int num_splits) {
    const long long cap = (long long)cols * BS;
    if (num_splits <= 0) num_splits = (int)((cap + kQuantPagedChunk - 1) / kQuantPagedChunk);
    return plan_attention(Q, Hq, Hkv, (int)cap, D, KVD_BF16, BS, num_splits, false, kQuantTile);
}

kvd_status attend_paged_quant(const char* fn, RowKind rk, const void* q, const void* key_cache,
                              const void* value_cache, const int32_t* block_tables,
                              const int32_t* seq_lens, const int32_t* seq_offset, void* out,
                              float* lse_out, int Q, int Hq, int Hkv, int NB, int BS, int cols,
                              int D, float scale, int num_splits, void* workspace,
                              size_t workspace_bytes, int32_t* dev_status, kvd_stream_t stream) {
    kvd_status st = check_attention_shape(Hq, Hkv, D, KVD_BF16);
    if (st != KVD_OK) return st;
    if (Q < 0 || NB < 1 || BS < 1 || cols < 1)
        return fail(KVD_ERR_INVALID_ARG, "%s: Q >= 0, NB, BS, cols >= 1 required", fn);
    if (Q == 0) return ok();
    if (!q || !key_cache || !value_cache || !block_tables || !seq_lens || !out)
        return fail(KVD_ERR_INVALID_ARG, "%s: null pointer", fn);
    if (!aligned(q, 16) || !aligned(key_cache, 16) || !aligned(value_cache, 16) ||
        !aligned(out, 16) || !aligned(lse_out, 4) || !aligned(block_tables, 4) ||
        !aligned(seq_lens, 4) || !aligned(seq_offset, 4) || !aligned(dev_status, 4))
        return fail(KVD_ERR_INVALID_ARG, "%s: misaligned pointer", fn);
    if ((long long)NB * BS >= (1ll << 31)) return fail(KVD_ERR_UNSUPPORTED, "%s: NB*BS >= 2^31", fn);
    if ((long long)cols * BS >= (1ll << 31)) return fail(KVD_ERR_UNSUPPORTED, "%s: cols*BS >= 2^31", fn);
    if (num_splits < 0) return fail(KVD_ERR_INVALID_ARG, "%s: num_splits < 0", fn);
    const Plan pl = paged_quant_plan(Q, Hq, Hkv, BS, cols, D, num_splits);
    st = check_workspace(fn, pl, workspace, workspace_bytes);
    if (st != KVD_OK) return st;
    const int RB = quant_row_bytes(rk, D);
    CUtensorMap kmap, vmap;
    st = make_row_map(&kmap, key_cache, (long long)NB * BS, Hkv, RB, pl.tile);
    if (st != KVD_OK) return st;
    st = make_row_map(&vmap, value_cache, (long long)NB * BS, Hkv, RB, pl.tile);
    if (st != KVD_OK) return st;
    AttendParams p{};
    p.q = q;
    p.block_tables = block_tables;
    p.seq_lens = seq_lens;
    p.seq_offset = seq_offset;
    p.out = out;
    p.lse_out = lse_out;
    p.dev_status = dev_status;
    p.Hq = Hq;
    p.Hkv = Hkv;
    p.g = Hq / Hkv;
    p.BS = BS;
    p.cols = cols;
    p.NB = NB;
    p.qscale = scale * kLog2e;
    attach_workspace(p, pl, workspace);
    cudaError_t e = rk == kRowsFp4
                        ? launch_attend_fp4(D, pl.G, kModePaged, p, &kmap, &vmap, (cudaStream_t)stream)
                        : launch_attend_fp8(D, pl.G, kModePaged, p, &kmap, &vmap, (cudaStream_t)stream);
    if (e != cudaSuccess) return cuda_fail(e, fn);
    if (pl.S > 1) {
        e = launch_combine(p.part_o, p.part_lse, out, lse_out, Q * Hq, pl.S, D, KVD_BF16,
                           (cudaStream_t)stream);
        if (e != cudaSuccess) return cuda_fail(e, "combine launch");
    }
    return ok();
}

Plan indexed_quant_plan(int B, int Hq, int Hkv, int topk, int D, int num_splits) {
    return plan_attention(B, Hq, Hkv, topk, D, KVD_BF16, 0, num_splits, true, kQuantTile);
}

kvd_status attend_indexed_quant(const char* fn, RowKind rk, const void* q, const void* k_cache,
                                const void* v_cache, const int32_t* indices, void* out,
                                float* lse_out, int B, int Hq, int Hkv, int C, int topk, int D,
                                float scale, int num_splits, void* workspace,
                                size_t workspace_bytes, int32_t* dev_status, kvd_stream_t stream) {
    kvd_status st = check_attention_shape(Hq, Hkv, D, KVD_BF16);
    if (st != KVD_OK) return st;
    if (B < 0 || C < 1 || topk < 1)
        return fail(KVD_ERR_INVALID_ARG, "%s: B >= 0, C >= 1 and topk >= 1 required", fn);
    if (B == 0) return ok();
    if (!q || !k_cache || !v_cache || !indices || !out)
        return fail(KVD_ERR_INVALID_ARG, "%s: null pointer", fn);
    if (!aligned(q, 16) || !aligned(k_cache, 16) || !aligned(v_cache, 16) || !aligned(out, 16) ||
        !aligned(indices, 4) || !aligned(lse_out, 4) || !aligned(dev_status, 4))
        return fail(KVD_ERR_INVALID_ARG, "%s: misaligned pointer", fn);
    if (num_splits < 0) return fail(KVD_ERR_INVALID_ARG, "%s: num_splits < 0", fn);
    const Plan pl = indexed_quant_plan(B, Hq, Hkv, topk, D, num_splits);
    st = check_workspace(fn, pl, workspace, workspace_bytes);
    if (st != KVD_OK) return st;
    AttendParams p{};
    p.q = q;
    p.k = k_cache;
    p.v = v_cache;
    p.indices = indices;
    p.out = out;
    p.lse_out = lse_out;
    p.dev_status = dev_status;
    p.Hq = Hq;
    p.Hkv = Hkv;
    p.g = Hq / Hkv;
    p.C = C;
    p.topk = topk;
    p.qscale = scale * kLog2e;
    attach_workspace(p, pl, workspace);
    CUtensorMap none;  // unused: the listed rows are gathered with cp.async
    std::memset(&none, 0, sizeof none);
    cudaError_t e = rk == kRowsFp4
                        ? launch_attend_fp4(D, pl.G, kModeIndexed, p, &none, &none, (cudaStream_t)stream)
                        : launch_attend_fp8(D, pl.G, kModeIndexed, p, &none, &none, (cudaStream_t)stream);
    if (e != cudaSuccess) return cuda_fail(e, fn);
    if (pl.S > 1) {
        e = launch_combine(p.part_o, p.part_lse, out, lse_out, B * Hq, pl.S, D, KVD_BF16,
                           (cudaStream_t)stream);
        if (e != cudaSuccess) return cuda_fail(e, "combine launch");
    }
    return ok();
}

}  // namespace

extern "C" {

kvd_status kvd_append_fp8(void* k_cache, void* v_cache, const void* k_new, const void* v_new,
                          const int32_t* pos, uint8_t* mask, int B, int Hkv, int C, int D,
                          kvd_dtype new_dtype, int32_t* dev_status, kvd_stream_t stream) {
    return append_quant("kvd_append_fp8", false, k_cache, v_cache, k_new, v_new, pos, mask, B,
                        Hkv, C, D, new_dtype, dev_status, stream);
}

kvd_status kvd_append_fp4(void* k_cache, void* v_cache, const void* k_new, const void* v_new,
                          const int32_t* pos, uint8_t* mask, int B, int Hkv, int C, int D,
                          kvd_dtype new_dtype, int32_t* dev_status, kvd_stream_t stream) {
    return append_quant("kvd_append_fp4", true, k_cache, v_cache, k_new, v_new, pos, mask, B,
                        Hkv, C, D, new_dtype, dev_status, stream);
}

size_t kvd_attend_masked_fp8_workspace_bytes(int B, int Hq, int Hkv, int C, int D, int num_splits) {
    return quant_workspace_bytes(B, Hq, Hkv, C, D, num_splits);
}

size_t kvd_attend_masked_fp4_workspace_bytes(int B, int Hq, int Hkv, int C, int D, int num_splits) {
    return quant_workspace_bytes(B, Hq, Hkv, C, D, num_splits);
}

kvd_status kvd_attend_masked_fp8_plan(int B, int Hq, int Hkv, int C, int D, int num_splits,
                                      kvd_plan* plan) {
    return quant_plan("kvd_attend_masked_fp8_plan", kRowsFp8, B, Hq, Hkv, C, D, num_splits, plan);
}

kvd_status kvd_attend_masked_fp4_plan(int B, int Hq, int Hkv, int C, int D, int num_splits,
                                      kvd_plan* plan) {
    return quant_plan("kvd_attend_masked_fp4_plan", kRowsFp4, B, Hq, Hkv, C, D, num_splits, plan);
}

kvd_status kvd_attend_masked_fp8(const void* q, const void* k_cache, const void* v_cache,
                                 const uint8_t* mask, void* out, float* lse_out, int B, int Hq,
                                 int Hkv, int C, int D, float scale, int num_splits,
                                 void* workspace, size_t workspace_bytes, int32_t* dev_status,
                                 kvd_stream_t stream) {
    return attend_quant("kvd_attend_masked_fp8", kRowsFp8, q, k_cache, v_cache, mask, out, lse_out,
                        B, Hq, Hkv, C, D, scale, num_splits, workspace, workspace_bytes,
                        dev_status, stream);
}

kvd_status kvd_attend_masked_fp4(const void* q, const void* k_cache, const void* v_cache,
                                 const uint8_t* mask, void* out, float* lse_out, int B, int Hq,
                                 int Hkv, int C, int D, float scale, int num_splits,
                                 void* workspace, size_t workspace_bytes, int32_t* dev_status,
                                 kvd_stream_t stream) {
    return attend_quant("kvd_attend_masked_fp4", kRowsFp4, q, k_cache, v_cache, mask, out, lse_out,
                        B, Hq, Hkv, C, D, scale, num_splits, workspace, workspace_bytes,
                        dev_status, stream);
}

kvd_status kvd_append_paged_fp8(void* key_cache, void* value_cache, const void* k_new,
                                const void* v_new, const int32_t* block_tables,
                                const int32_t* seq_offset, const int32_t* pos, int Q, int NB,
                                int BS, int cols, int Hkv, int D, kvd_dtype new_dtype,
                                int32_t* dev_status, kvd_stream_t stream) {
    return append_paged_quant("kvd_append_paged_fp8", false, key_cache, value_cache, k_new, v_new,
                              block_tables, seq_offset, pos, Q, NB, BS, cols, Hkv, D, new_dtype,
                              dev_status, stream);
}

size_t kvd_attend_paged_fp8_workspace_bytes(int Q, int Hq, int Hkv, int BS, int cols, int D,
                                             int num_splits) {
    if (Q < 1 || BS < 1 || cols < 1 || check_attention_shape(Hq, Hkv, D, KVD_BF16) != KVD_OK) return 0;
    return paged_quant_plan(Q, Hq, Hkv, BS, cols, D, num_splits).ws;
}

kvd_status kvd_attend_paged_fp8_plan(int Q, int Hq, int Hkv, int BS, int cols, int D,
                                      int num_splits, kvd_plan* plan) {
    if (!plan) return fail(KVD_ERR_INVALID_ARG, "kvd_attend_paged_fp8_plan: null pointer");
    if (Q < 1 || BS < 1 || cols < 1 || num_splits < 0)
        return fail(KVD_ERR_INVALID_ARG,
                    "kvd_attend_paged_fp8_plan: Q, BS, cols >= 1 and num_splits >= 0 required");
    const kvd_status st = check_attention_shape(Hq, Hkv, D, KVD_BF16);
    if (st != KVD_OK) return st;
    put_plan(paged_quant_plan(Q, Hq, Hkv, BS, cols, D, num_splits), false, plan);
    return ok();
}

kvd_status kvd_attend_paged_fp8(const void* q, const void* key_cache, const void* value_cache,
                                const int32_t* block_tables, const int32_t* seq_lens,
                                const int32_t* seq_offset, void* out, float* lse_out, int Q,
                                int Hq, int Hkv, int NB, int BS, int cols, int D, float scale,
                                int num_splits, void* workspace, size_t workspace_bytes,
                                int32_t* dev_status, kvd_stream_t stream) {
    return attend_paged_quant("kvd_attend_paged_fp8", kRowsFp8, q, key_cache, value_cache,
                              block_tables, seq_lens, seq_offset, out, lse_out, Q, Hq, Hkv, NB,
                              BS, cols, D, scale, num_splits, workspace, workspace_bytes,
                              dev_status, stream);
}

size_t kvd_attend_indexed_fp8_workspace_bytes(int B, int Hq, int Hkv, int topk, int D,
                                               int num_splits) {
    if (B < 1 || topk < 1 || check_attention_shape(Hq, Hkv, D, KVD_BF16) != KVD_OK) return 0;
    return indexed_quant_plan(B, Hq, Hkv, topk, D, num_splits).ws;
}

kvd_status kvd_attend_indexed_fp8_plan(int B, int Hq, int Hkv, int topk, int D, int num_splits,
                                        kvd_plan* plan) {
    if (!plan) return fail(KVD_ERR_INVALID_ARG, "kvd_attend_indexed_fp8_plan: null pointer");
    if (B < 1 || topk < 1 || num_splits < 0)
        return fail(KVD_ERR_INVALID_ARG,
                    "kvd_attend_indexed_fp8_plan: B, topk >= 1 and num_splits >= 0 required");
    const kvd_status st = check_attention_shape(Hq, Hkv, D, KVD_BF16);
    if (st != KVD_OK) return st;
    put_plan(indexed_quant_plan(B, Hq, Hkv, topk, D, num_splits), false, plan);
    return ok();
}

kvd_status kvd_attend_indexed_fp8(const void* q, const void* k_cache, const void* v_cache,
                                  const int32_t* indices, void* out, float* lse_out, int B,
                                  int Hq, int Hkv, int C, int topk, int D, float scale,
                                  int num_splits, void* workspace, size_t workspace_bytes,
                                  int32_t* dev_status, kvd_stream_t stream) {
    return attend_indexed_quant("kvd_attend_indexed_fp8", kRowsFp8, q, k_cache, v_cache, indices,
                                out, lse_out, B, Hq, Hkv, C, topk, D, scale, num_splits, workspace,
                                workspace_bytes, dev_status, stream);
}

kvd_status kvd_append_paged_fp4(void* key_cache, void* value_cache, const void* k_new,
                                const void* v_new, const int32_t* block_tables,
                                const int32_t* seq_offset, const int32_t* pos, int Q, int NB,
                                int BS, int cols, int Hkv, int D, kvd_dtype new_dtype,
                                int32_t* dev_status, kvd_stream_t stream) {
    return append_paged_quant("kvd_append_paged_fp4", true, key_cache, value_cache, k_new, v_new,
                              block_tables, seq_offset, pos, Q, NB, BS, cols, Hkv, D, new_dtype,
                              dev_status, stream);
}

size_t kvd_attend_paged_fp4_workspace_bytes(int Q, int Hq, int Hkv, int BS, int cols, int D,
                                             int num_splits) {
    if (Q < 1 || BS < 1 || cols < 1 || check_attention_shape(Hq, Hkv, D, KVD_BF16) != KVD_OK) return 0;
    return paged_quant_plan(Q, Hq, Hkv, BS, cols, D, num_splits).ws;
}

kvd_status kvd_attend_paged_fp4_plan(int Q, int Hq, int Hkv, int BS, int cols, int D,
                                      int num_splits, kvd_plan* plan) {
    if (!plan) return fail(KVD_ERR_INVALID_ARG, "kvd_attend_paged_fp4_plan: null pointer");
    if (Q < 1 || BS < 1 || cols < 1 || num_splits < 0)
        return fail(KVD_ERR_INVALID_ARG,
                    "kvd_attend_paged_fp4_plan: Q, BS, cols >= 1 and num_splits >= 0 required");
    const kvd_status st = check_attention_shape(Hq, Hkv, D, KVD_BF16);
    if (st != KVD_OK) return st;
    put_plan(paged_quant_plan(Q, Hq, Hkv, BS, cols, D, num_splits), false, plan);
    return ok();
}

kvd_status kvd_attend_paged_fp4(const void* q, const void* key_cache, const void* value_cache,
                                const int32_t* block_tables, const int32_t* seq_lens,
                                const int32_t* seq_offset, void* out, float* lse_out, int Q,
                                int Hq, int Hkv, int NB, int BS, int cols, int D, float scale,
                                int num_splits, void* workspace, size_t workspace_bytes,
                                int32_t* dev_status, kvd_stream_t stream) {
    return attend_paged_quant("kvd_attend_paged_fp4", kRowsFp4, q, key_cache, value_cache,
                              block_tables, seq_lens, seq_offset, out, lse_out, Q, Hq, Hkv, NB,
                              BS, cols, D, scale, num_splits, workspace, workspace_bytes,
                              dev_status, stream);
}

size_t kvd_attend_indexed_fp4_workspace_bytes(int B, int Hq, int Hkv, int topk, int D,
                                               int num_splits) {
    if (B < 1 || topk < 1 || check_attention_shape(Hq, Hkv, D, KVD_BF16) != KVD_OK) return 0;
    return indexed_quant_plan(B, Hq, Hkv, topk, D, num_splits).ws;
}

kvd_status kvd_attend_indexed_fp4_plan(int B, int Hq, int Hkv, int topk, int D, int num_splits,
                                        kvd_plan* plan) {
    if (!plan) return fail(KVD_ERR_INVALID_ARG, "kvd_attend_indexed_fp4_plan: null pointer");
    if (B < 1 || topk < 1 || num_splits < 0)
        return fail(KVD_ERR_INVALID_ARG,
                    "kvd_attend_indexed_fp4_plan: B, topk >= 1 and num_splits >= 0 required");
    const kvd_status st = check_attention_shape(Hq, Hkv, D, KVD_BF16);
    if (st != KVD_OK) return st;
    put_plan(indexed_quant_plan(B, Hq, Hkv, topk, D, num_splits), false, plan);
    return ok();
}

kvd_status kvd_attend_indexed_fp4(const void* q, const void* k_cache, const void* v_cache,
                                  const int32_t* indices, void* out, float* lse_out, int B,
                                  int Hq, int Hkv, int C, int topk, int D, float scale,
                                  int num_splits, void* workspace, size_t workspace_bytes,
                                  int32_t* dev_status, kvd_stream_t stream) {
    return attend_indexed_quant("kvd_attend_indexed_fp4", kRowsFp4, q, k_cache, v_cache, indices,
                                out, lse_out, B, Hq, Hkv, C, topk, D, scale, num_splits, workspace,
                                workspace_bytes, dev_status, stream);
}

size_t kvd_attend_indexed_workspace_bytes(int B, int Hq, int Hkv, int topk, int D,
                                          kvd_dtype dtype, int num_splits) {
    if (B < 1 || topk < 1 || check_attention_shape(Hq, Hkv, D, dtype) != KVD_OK) return 0;
    return plan_attention(B, Hq, Hkv, topk, D, dtype, 0, num_splits, true).ws;
}

kvd_status kvd_attend_indexed_plan(int B, int Hq, int Hkv, int topk, int D, kvd_dtype dtype,
                                   int num_splits, kvd_plan* plan) {
    if (!plan)
        return fail(KVD_ERR_INVALID_ARG, "kvd_attend_indexed_plan: null pointer");
    if (B < 1 || topk < 1 || num_splits < 0)
        return fail(KVD_ERR_INVALID_ARG, "kvd_attend_indexed_plan: B, topk >= 1 and num_splits >= 0 required");
    const kvd_status st = check_attention_shape(Hq, Hkv, D, dtype);
    if (st != KVD_OK) return st;
    put_plan(plan_attention(B, Hq, Hkv, topk, D, dtype, 0, num_splits, true), false, plan);
    return ok();
}

kvd_status kvd_attend_indexed(const void* q, const void* k_cache, const void* v_cache,
                              const int32_t* indices, void* out, float* lse_out, int B, int Hq,
                              int Hkv, int C, int topk, int D, float scale, kvd_dtype dtype,
                              int num_splits, void* workspace, size_t workspace_bytes,
                              int32_t* dev_status, kvd_stream_t stream) {
    kvd_status st = check_attention_shape(Hq, Hkv, D, dtype);
    if (st != KVD_OK) return st;
    if (B < 0 || C < 1 || topk < 1)
        return fail(KVD_ERR_INVALID_ARG, "kvd_attend_indexed: B >= 0, C >= 1 and topk >= 1 required");
    if (B == 0) return ok();
    if (!q || !k_cache || !v_cache || !indices || !out)
        return fail(KVD_ERR_INVALID_ARG, "kvd_attend_indexed: null pointer");
    if (!aligned(q, 16) || !aligned(k_cache, 16) || !aligned(v_cache, 16) || !aligned(out, 16) ||
        !aligned(indices, 4) || !aligned(lse_out, 4) || !aligned(dev_status, 4))
        return fail(KVD_ERR_INVALID_ARG, "kvd_attend_indexed: misaligned pointer");
    if (num_splits < 0) return fail(KVD_ERR_INVALID_ARG, "kvd_attend_indexed: num_splits < 0");
    const Plan pl = plan_attention(B, Hq, Hkv, topk, D, dtype, 0, num_splits, true);
    st = check_workspace("kvd_attend_indexed", pl, workspace, workspace_bytes);
    if (st != KVD_OK) return st;
    AttendParams p{};
    p.q = q;
    p.k = k_cache;
    p.v = v_cache;
    p.indices = indices;
    p.out = out;
    p.lse_out = lse_out;
    p.dev_status = dev_status;
    p.Hq = Hq;
    p.Hkv = Hkv;
    p.g = Hq / Hkv;
    p.C = C;
    p.topk = topk;
    p.qscale = scale * kLog2e;
    attach_workspace(p, pl, workspace);
    CUtensorMap kmap, vmap;  // unused: the kernel gathers the listed rows with cp.async
    std::memset(&kmap, 0, sizeof kmap);
    std::memset(&vmap, 0, sizeof vmap);
    cudaError_t e = launch_attend(dtype, D, pl.G, kModeIndexed, p, &kmap, &vmap, (cudaStream_t)stream);
    if (e != cudaSuccess) return cuda_fail(e, "kvd_attend_indexed launch");
    if (pl.S > 1) {
        e = launch_combine(p.part_o, p.part_lse, out, lse_out, B * Hq, pl.S, D, dtype,
                           (cudaStream_t)stream);
        if (e != cudaSuccess) return cuda_fail(e, "kvd_attend_indexed combine launch");
    }
    return ok();
}

size_t kvd_attend_paged_workspace_bytes(int Q, int Hq, int Hkv, int BS, int cols, int D,
                                        kvd_dtype dtype, int num_splits) {
    if (Q < 1 || BS < 1 || cols < 1 || check_attention_shape(Hq, Hkv, D, dtype) != KVD_OK) return 0;
    return plan_attention(Q, Hq, Hkv, (int)((long long)cols * BS), D, dtype, BS, num_splits).ws;
}

kvd_status kvd_attend_paged_plan(int Q, int Hq, int Hkv, int BS, int cols, int D, kvd_dtype dtype,
                                 int num_splits, kvd_plan* plan) {
    if (!plan)
        return fail(KVD_ERR_INVALID_ARG, "kvd_attend_paged_plan: null pointer");
    if (Q < 1 || BS < 1 || cols < 1 || num_splits < 0)
        return fail(KVD_ERR_INVALID_ARG, "kvd_attend_paged_plan: Q, BS, cols >= 1 and num_splits >= 0 required");
    if ((long long)cols * BS >= (1ll << 31))
        return fail(KVD_ERR_UNSUPPORTED, "kvd_attend_paged_plan: cols*BS >= 2^31");
    const kvd_status st = check_attention_shape(Hq, Hkv, D, dtype);
    if (st != KVD_OK) return st;
    put_plan(plan_attention(Q, Hq, Hkv, cols * BS, D, dtype, BS, num_splits), false, plan);
    return ok();
}

kvd_status kvd_attend_paged(const void* q_in, const void* key_cache, const void* value_cache,
                            const int32_t* block_tables, const int32_t* seq_lens,
                            const int32_t* seq_offset, void* out, float* lse_out, int Q, int Hq,
                            int Hkv, int NB, int BS, int cols, int D, float scale,
                            kvd_dtype dtype, int num_splits, void* workspace,
                            size_t workspace_bytes, int32_t* dev_status, kvd_stream_t stream) {
    kvd_status st = check_attention_shape(Hq, Hkv, D, dtype);
    if (st != KVD_OK) return st;
    if (Q < 0 || NB < 1 || BS < 1 || cols < 1)
        return fail(KVD_ERR_INVALID_ARG, "kvd_attend_paged: Q >= 0, NB, BS, cols >= 1 required");
    if (Q == 0) return ok();
    if (!q_in || !key_cache || !value_cache || !block_tables || !seq_lens || !out)
        return fail(KVD_ERR_INVALID_ARG, "kvd_attend_paged: null pointer");
    if (!aligned(q_in, 16) || !aligned(key_cache, 16) || !aligned(value_cache, 16) ||
        !aligned(out, 16) || !aligned(lse_out, 4) || !aligned(block_tables, 4) ||
        !aligned(seq_lens, 4) || !aligned(seq_offset, 4) || !aligned(dev_status, 4))
        return fail(KVD_ERR_INVALID_ARG, "kvd_attend_paged: misaligned pointer");
    if ((long long)NB * BS >= (1ll << 31)) return fail(KVD_ERR_UNSUPPORTED, "kvd_attend_paged: NB*BS >= 2^31");
    if ((long long)cols * BS >= (1ll << 31)) return fail(KVD_ERR_UNSUPPORTED, "kvd_attend_paged: cols*BS >= 2^31");
    if (num_splits < 0) return fail(KVD_ERR_INVALID_ARG, "kvd_attend_paged: num_splits < 0");
    const Plan pl = plan_attention(Q, Hq, Hkv, cols * BS, D, dtype, BS, num_splits);
    st = check_workspace("kvd_attend_paged", pl, workspace, workspace_bytes);
    if (st != KVD_OK) return st;
    CUtensorMap kmap, vmap;
    const bool mma = attend_uses_mma(dtype, pl.G);
    st = make_cache_map(&kmap, key_cache, dtype, true, (long long)NB * BS, Hkv, D, pl.tile, mma);
    if (st != KVD_OK) return st;
    st = make_cache_map(&vmap, value_cache, dtype, true, (long long)NB * BS, Hkv, D, pl.tile, mma);
    if (st != KVD_OK) return st;
    AttendParams p{};
    p.q = q_in;
    p.block_tables = block_tables;
    p.seq_lens = seq_lens;
    p.seq_offset = seq_offset;
    p.out = out;
    p.lse_out = lse_out;
    p.dev_status = dev_status;
    p.Hq = Hq;
    p.Hkv = Hkv;
    p.g = Hq / Hkv;
    p.BS = BS;
    p.cols = cols;
    p.NB = NB;
    p.qscale = scale * kLog2e;
    attach_workspace(p, pl, workspace);
    cudaError_t e = launch_attend(dtype, D, pl.G, kModePaged, p, &kmap, &vmap, (cudaStream_t)stream);
    if (e != cudaSuccess) return cuda_fail(e, "kvd_attend_paged launch");
    if (pl.S > 1) {
        e = launch_combine(p.part_o, p.part_lse, out, lse_out, Q * Hq, pl.S, D, dtype,
                           (cudaStream_t)stream);
        if (e != cudaSuccess) return cuda_fail(e, "kvd_attend_paged combine launch");
    }
    return ok();
}

kvd_status kvd_gather_paged(const void* key_cache, const void* value_cache,
                            const int32_t* block_tables, const int32_t* seq_lens,
                            const int32_t* seq_offset, void* key_out, void* value_out, int Q,
                            int NB, int BS, int cols, int Hk, int Dk, int Hv, int Dv,
                            int total_tokens, int elem_bytes, int32_t* dev_status,
                            kvd_stream_t stream) {
    if (Q < 0 || NB < 1 || BS < 1 || cols < 1 || Hk < 1 || Dk < 1 || Hv < 1 || Dv < 1 ||
        total_tokens < 0)
        return fail(KVD_ERR_INVALID_ARG, "kvd_gather_paged: bad sizes");
    if (elem_bytes != 2 && elem_bytes != 4)
        return fail(KVD_ERR_INVALID_ARG, "kvd_gather_paged: elem_bytes must be 2 or 4");
    if (Q == 0) return ok();
    if (!key_cache || !value_cache || !block_tables || !seq_lens || (total_tokens > 0 && (!key_out || !value_out)))
        return fail(KVD_ERR_INVALID_ARG, "kvd_gather_paged: null pointer");
    if (!aligned(key_cache, 16) || !aligned(value_cache, 16) || !aligned(key_out, 16) ||
        !aligned(value_out, 16) || !aligned(block_tables, 4) || !aligned(seq_lens, 4) ||
        !aligned(seq_offset, 4) || !aligned(dev_status, 4))
        return fail(KVD_ERR_INVALID_ARG, "kvd_gather_paged: misaligned pointer");
    if ((long long)Q * cols >= (1ll << 31)) return fail(KVD_ERR_UNSUPPORTED, "kvd_gather_paged: Q*cols >= 2^31");
    const long long krow = (long long)Hk * Dk * elem_bytes, vrow = (long long)Hv * Dv * elem_bytes;
    const cudaError_t e = launch_gather(key_cache, value_cache, block_tables, seq_lens, seq_offset,
                                        key_out, value_out, Q, NB, BS, cols, krow, vrow,
                                        total_tokens, dev_status, (cudaStream_t)stream);
    if (e != cudaSuccess) return cuda_fail(e, "kvd_gather_paged launch");
    return ok();
}

kvd_status kvd_combine(const float* part_o, const float* part_lse, void* out, float* lse_out,
                       int R, int S, int D, kvd_dtype out_dtype, kvd_stream_t stream) {
    if (R < 0 || S < 1 || D < 4 || D % 4 || D > 1024)
        return fail(KVD_ERR_INVALID_ARG, "kvd_combine: R >= 0, S >= 1, D % 4 == 0 and 4 <= D <= 1024 required");
    if (!dtype_ok(out_dtype)) return fail(KVD_ERR_INVALID_ARG, "kvd_combine: unknown dtype");
    if (R == 0) return ok();
    if (!part_o || !part_lse || !out) return fail(KVD_ERR_INVALID_ARG, "kvd_combine: null pointer");
    if (!aligned(part_o, 16) || !aligned(out, 16) || !aligned(part_lse, 4) || !aligned(lse_out, 4))
        return fail(KVD_ERR_INVALID_ARG, "kvd_combine: misaligned pointer");
    const cudaError_t e = launch_combine(part_o, part_lse, out, lse_out, R, S, D, out_dtype, (cudaStream_t)stream);
    if (e != cudaSuccess) return cuda_fail(e, "kvd_combine launch");
    return ok();
}

kvd_status kvd_combine_gathered(const float* parts, void* out, float* lse_out, int R, int S,
                                int D, kvd_dtype out_dtype, kvd_stream_t stream) {
    const char* fn = "kvd_combine_gathered";
    if (R < 0 || S < 1 || D < 4 || D % 4 || D > 1024)
        return fail(KVD_ERR_INVALID_ARG, "%s: R >= 0, S >= 1, D %% 4 == 0 and 4 <= D <= 1024 required", fn);
    if (!dtype_ok(out_dtype)) return fail(KVD_ERR_INVALID_ARG, "%s: unknown dtype", fn);
    if (R == 0) return ok();
    if (!parts || !out) return fail(KVD_ERR_INVALID_ARG, "%s: null pointer", fn);
    if (!aligned(parts, 16) || !aligned(out, 16) || !aligned(lse_out, 4))
        return fail(KVD_ERR_INVALID_ARG, "%s: misaligned pointer", fn);
    const long long block = (long long)R * (D + 1);  // floats per split: R rows of D, R lse
    const cudaError_t e = launch_combine(parts, parts + (long long)R * D, out, lse_out, R, S, D,
                                         out_dtype, (cudaStream_t)stream, block);
    if (e != cudaSuccess) return cuda_fail(e, fn);
    return ok();
}

}  // extern "C"
