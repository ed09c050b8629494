/*
 * kvd.h -- C ABI of libkvd: decode-phase KV-cache attention on GB300 (sm_103a).
 *
 * One new query token per head attends over a KV cache of fixed capacity,
 * kept either as a static buffer with a 0/1 mask or as a paged cache
 * addressed through block tables.  Sources (page title, section):
 *
 *  [NPU]    "Intel NPU running LLMs" (OpenVINO community article 882):
 *           Part 1 "解决方案：预分配 + Attention Mask" -- static buffer of
 *           capacity MAX_PROMPT_LEN + MIN_RESPONSE_LEN (default 1024 + 128 =
 *           1152) with a 0/1 mask the length of the buffer, mask = 0 slots
 *           set to -inf before the softmax; Part 2 "NPUW 的核心设计" --
 *           update_kvcache_for writes only the new token's row at the next
 *           empty slot and bumps num_stored_tokens; Part 3 "Attention 在 NPU
 *           上的完整实现" -- decode is one query against N keys (incremental
 *           SDPA), tiles along the sequence merged exactly through a running
 *           output, max and sum (Flash SDPA path); Part 5 "当前限制" -- more
 *           tokens than the capacity is an error.
 *  [FlashMLA] "FlashMLA на Huawei Ascend: ядро разреженного внимания
 *           изнутри", "Математическая постановка" -- out = softmax(Q K^T *
 *           sm_scale) V per query token; "Ход вычислений" -- fp32 running
 *           max / sum / output and a log-sum-exp per row.
 *  [FlashMLA-KV] the same page, "Ограничение по деквантованию" -- decoding
 *           reads the KV cache in FP8, dequantises it to bf16 and feeds the
 *           matrix unit; "Оптимизация раскладки KV-кэша при decoding" -- a
 *           token's quantised values and its scale are stored side by side.
 *  [PyPTO]  "PyPTO 实现 AscendC GatherPaKvCache（Norm/ND 分支）" sections
 *           3.1-3.3 -- key_cache [num_blocks, block_size, heads, dim],
 *           int32 block_tables [Q, cols], cumsum seq_lens [Q+1] starting at
 *           0, optional seq_offset [Q] (multiple of block_size, selects the
 *           first table column), logical_block = t / block_size, slot =
 *           t % block_size, output row seq_lens[q] + t; section 7 -- only the
 *           cumsum form of seq_lens and int32 indices.
 *
 * Conventions for every entry point:
 *  - Tensors are caller-owned device memory, contiguous, row-major, in the
 *    layouts given per call.  The library never allocates, frees, copies to
 *    the host or synchronises; every call is asynchronous on `stream`.
 *  - Pointers to element data must be 16-byte aligned; byte masks and int32
 *    index arrays need only their natural alignment.
 *  - The return value reports errors the host can see (arguments, sizes,
 *    launch failures).  Errors that depend on device-resident data set bits
 *    in the optional caller-owned `dev_status` word (atomic OR, never cleared
 *    by the library); the offending element is skipped, never written out of
 *    bounds.  Nothing traps or aborts.
 *  - Every wait inside a kernel is bounded (about one second); a wait that
 *    runs out sets KVD_DEV_TIMEOUT and the kernel returns.
 *  - The caches are plain inputs/outputs of the calls: the caller owns them,
 *    starts a conversation by zeroing them and appends through kvd_append.
 */
#ifndef KVD_H
#define KVD_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* Same type as cudaStream_t; NULL is the legacy default stream. */
typedef struct CUstream_st* kvd_stream_t;

typedef enum {
    KVD_OK = 0,
    KVD_ERR_INVALID_ARG = 1,  /* null/misaligned pointer, bad size, bad combination */
    KVD_ERR_UNSUPPORTED = 2,  /* valid but not implemented (head_dim, dtype, group) */
    KVD_ERR_WORKSPACE = 3,    /* workspace missing or smaller than required */
    KVD_ERR_CUDA = 4          /* a CUDA runtime/driver call failed (see kvd_last_error) */
} kvd_status;

typedef enum { KVD_BF16 = 0, KVD_F32 = 1 } kvd_dtype;

/* Bits OR-ed into *dev_status by the kernels. */
#define KVD_DEV_POS_RANGE 1u     /* append position outside [0, capacity) */
#define KVD_DEV_BLOCK_RANGE 2u   /* block table entry outside [0, num_blocks) */
#define KVD_DEV_TABLE_COLS 4u    /* seq_offset/BS + ceil(len/BS) > table columns */
#define KVD_DEV_SEQLENS 8u       /* seq_lens not starting at 0, decreasing, or past total */
#define KVD_DEV_SEQ_OFFSET 16u   /* seq_offset negative or not a multiple of block_size */
#define KVD_DEV_TIMEOUT 32u      /* a bounded in-kernel wait ran out */
#define KVD_DEV_POINTER 64u      /* a pointer read from a device pointer array is null or misaligned */

/*
 * kvd_append -- [NPU] Part 2, update_kvcache_for: for every batch entry b
 * and kv head h, row pos[b] of k_cache[b, h] and v_cache[b, h] becomes
 * k_new[b, h] and v_new[b, h]; if `mask` is given, mask[b, pos[b]] = 1.
 *   k_cache, v_cache  [B, Hkv, C, D] of `dtype`          (in/out)
 *   k_new, v_new      [B, Hkv, D] of `dtype`             (in)
 *   pos               [B] int32, device                  (in)
 *   mask              [B, C] uint8 or NULL               (in/out)
 * A byte copy.  pos[b] outside [0, C) writes nothing for b and sets
 * KVD_DEV_POS_RANGE ([NPU] Part 5: over capacity is an error).
 * Errors: INVALID_ARG for null pointers, sizes < 1, D*elem not a multiple of
 * 16 bytes, misaligned data pointers.
 */
kvd_status kvd_append(void* k_cache, void* v_cache, const void* k_new, const void* v_new,
                      const int32_t* pos, uint8_t* mask, int B, int Hkv, int C, int D,
                      kvd_dtype dtype, int32_t* dev_status, kvd_stream_t stream);

/*
 * kvd_copy_prefix -- copy_kvcache, the prefill -> generate hand-over ([NPU]
 * Part 2 "NPUW 的核心设计", step 3: the prefill model's present K/V are copied
 * as the slice [0:N] into the generate model's past K/V, capacities 1024 and
 * 1152, all 32 layers x K and V at once).  For every layer l, batch entry b
 * and kv head h, rows [0, n[b]) of k_src[l][b, h] and v_src[l][b, h] become
 * the same rows of k_dst[l][b, h] and v_dst[l][b, h]; rows >= n[b] of the
 * destination are left alone.  If `masks` is given, masks[l][b, t] becomes
 * (t < n[b]) for every t < C_dst.
 *   k_src, v_src  device arrays of L pointers to [B, Hkv, C_src, D] of `dtype`
 *   k_dst, v_dst  device arrays of L pointers to [B, Hkv, C_dst, D]
 *   masks         device array of L pointers to [B, C_dst] uint8, or NULL
 *   n             [B] int32, device
 * One launch for all layers; a byte copy.  n[b] outside [0, min(C_src,
 * C_dst)] copies nothing for b (and leaves its masks) and sets
 * KVD_DEV_POS_RANGE; a null or non-16-byte-aligned pointer in an array skips
 * that layer and sets KVD_DEV_POINTER.
 * Errors: INVALID_ARG for null arrays, sizes < 1, D*elem not a multiple of 16
 * bytes, misaligned arrays; UNSUPPORTED for B*Hkv or L above 65535 / 32767.
 */
kvd_status kvd_copy_prefix(const void* const* k_src, const void* const* v_src, void* const* k_dst,
                           void* const* v_dst, uint8_t* const* masks, const int32_t* n, int L,
                           int B, int Hkv, int C_src, int C_dst, int D, kvd_dtype dtype,
                           int32_t* dev_status, kvd_stream_t stream);

/*
 * kvd_attend_masked -- decode attention over the static buffer ([NPU] Part 1
 * and Part 3; [FlashMLA] "Математическая постановка"):
 *   out[b, h, :] = sum_t w_t v[b, h/g, t, :] / sum_t w_t,
 *   w_t = exp(scale * q[b, h, :] . k[b, h/g, t, :] - max), over t with
 *   mask[b, t] != 0, g = Hq / Hkv (query head h reads kv head h / g).
 *   lse[b, h] = log sum_t exp(scale * q.k_t) (natural log).
 *   q         [B, Hq, D] of `dtype`
 *   k_cache   [B, Hkv, C, D], v_cache [B, Hkv, C, D] of `dtype`
 *   mask      [B, C] uint8, nonzero = valid; any content in mask = 0 slots
 *             (inf, NaN) is ignored; all-zero mask tiles are not read
 *   out       [B, Hq, D] of `dtype` (fp32 result rounded to nearest even)
 *   lse_out   [B, Hq] float or NULL
 * A row with no valid slot gives out = 0 and lse = -inf.
 * The sequence axis of every (batch entry, kv head) row is cut into splits
 * that a persistent grid takes from a work counter; each split keeps an fp32
 * running max / sum / output.  num_splits > 0 asks for about that many equal
 * splits (lengths rounded up to the kernel's tile, at most 4096 slots); 0
 * lets the library plan from the sizes, with smaller splits over the end of
 * the capacity.  With more than one split a second kernel merges the splits by
 * log-sum-exp (the kvd_combine formula).  Short buffers with num_splits = 0
 * (at most 8 splits of at most 384 slots per row, every split of every row
 * resident at once on the GPU) take one launch instead: a thread-block
 * cluster per row whose CTAs hold one split each and merge the row through
 * distributed shared memory (kvd_attend_masked_launches tells which).
 * Workspace: at least kvd_attend_masked_workspace_bytes(...) bytes (never
 * less than 256), 256-byte aligned, holding the work counters and the
 * partial rows.  Zero-fill it once before its first use; every call leaves
 * its counters at zero again, so calls ordered on one stream can reuse it
 * (calls that may overlap on the GPU must not share one).  After a call that
 * reported KVD_DEV_TIMEOUT, zero it again.
 * Supported: D in {64, 128}; dtype bf16 or f32; any Hq multiple of Hkv.
 */
size_t kvd_attend_masked_workspace_bytes(int B, int Hq, int Hkv, int C, int D, kvd_dtype dtype,
                                         int num_splits);
/* Kernel launches one kvd_attend_masked (or kvd_append_attend_masked with
 * Hq / Hkv <= 8) call makes for these sizes: 1 or 2; 0 for invalid sizes. */
int kvd_attend_masked_launches(int B, int Hq, int Hkv, int C, int D, kvd_dtype dtype,
                               int num_splits);
kvd_status kvd_attend_masked(const void* q, const void* k_cache, const void* v_cache,
                             const uint8_t* mask, void* out, float* lse_out, int B, int Hq,
                             int Hkv, int C, int D, float scale, kvd_dtype dtype, int num_splits,
                             void* workspace, size_t workspace_bytes, int32_t* dev_status,
                             kvd_stream_t stream);

/*
 * How a split attention call runs for given sizes (the *_plan queries), for a
 * caller that reads the workspace's partial rows or times the launches apart:
 *   splits            S of the split kernel: 1 = its units write the output
 *                     rows directly; > 1 = partial rows merged by log-sum-exp;
 *                     0 = the one-launch cluster kernel (no partial rows)
 *   launches          kernel launches of one call (1, or 2 when the combine
 *                     launch merges the splits)
 *   lse_offset, o_offset  with S > 1, the workspace byte offsets of part_lse
 *                     float [rows*Hq, S] and part_o float [rows*Hq, S, D] (the
 *                     kvd_combine layout); 0 otherwise
 *   counter_bytes     leading workspace bytes holding work counters (zero
 *                     before a call; every completed call leaves them zero)
 */
typedef struct {
    int32_t splits;
    int32_t launches;
    size_t lse_offset;
    size_t o_offset;
    size_t counter_bytes;
} kvd_plan;

/* kvd_attend_masked_plan -- kvd_plan of kvd_attend_masked (and of
 * kvd_append_attend_masked, kvd_attend_masked_partial) for these sizes.
 * Arguments and errors as for kvd_attend_masked. */
kvd_status kvd_attend_masked_plan(int B, int Hq, int Hkv, int C, int D, kvd_dtype dtype,
                                  int num_splits, kvd_plan* plan);

/*
 * kvd_attend_masked_partial -- the same attention as kvd_attend_masked, but
 * the output rows stay in fp32 whatever `dtype` is: out [B, Hq, D] float,
 * lse_out [B, Hq] float (required).  This is the partial result of one range
 * of a sequence's tokens ([NPU] Part 3, Flash SDPA path: each tile's output
 * is normalised over its own keys and carried with its max and sum), which
 * kvd_combine or kvd_combine_gathered merges exactly with the other
 * ranges' partials -- e.g. when the sequence axis of one long sequence is
 * spread over several GPUs, each holding a slice [B, Hkv, C_r, D] of the
 * cache and the matching slice [B, C_r] of the mask.  A range with no valid
 * slot gives out = 0 and lse = -inf (weight 0 in the merge).  Workspace,
 * splits and errors as for kvd_attend_masked.
 */
kvd_status kvd_attend_masked_partial(const void* q, const void* k_cache, const void* v_cache,
                                     const uint8_t* mask, float* out, float* lse_out, int B,
                                     int Hq, int Hkv, int C, int D, float scale, kvd_dtype dtype,
                                     int num_splits, void* workspace, size_t workspace_bytes,
                                     int32_t* dev_status, kvd_stream_t stream);

/*
 * kvd_attend_paged -- decode attention over the paged cache: for sequence q
 * the keys/values are the rows kvd_gather_paged would produce for q
 * ([PyPTO] 3.2), all valid, and q_in[q, h] attends over them with kv head
 * h / (Hq / Hkv).  The block-table indirection is resolved in the kernel.
 *   q_in         [Q, Hq, D] of `dtype`
 *   key_cache    [NB, BS, Hkv, D], value_cache [NB, BS, Hkv, D] of `dtype`
 *   block_tables [Q, cols] int32
 *   seq_lens     [Q + 1] int32, cumsum starting at 0
 *   seq_offset   [Q] int32 or NULL (zeros); first table column = seq_offset[q] / BS
 *   out          [Q, Hq, D] of `dtype`;  lse_out [Q, Hq] float or NULL
 * Device-detected errors (KVD_DEV_SEQLENS, SEQ_OFFSET, TABLE_COLS) make the
 * sequence empty (out = 0, lse = -inf); an out-of-range block id
 * (KVD_DEV_BLOCK_RANGE) drops that block's tokens.  A sequence of length 0
 * gives out = 0, lse = -inf.  One launch and a workspace as for
 * kvd_attend_masked (zero-filled before first use, left zeroed by each call).
 * Supported: D in {64, 128}; bf16 or f32; BS*Hkv*D*elem addressable by a
 * TMA tensor map (NB*BS < 2^31).
 */
/*
 * kvd_append_attend_masked -- one decode step over the static buffer: the
 * result of kvd_append(k_cache, v_cache, k_new, v_new, pos, mask) followed by
 * kvd_attend_masked(q, k_cache, v_cache, mask, ...) ([NPU] Part 2,
 * update_kvcache_for, then Part 3), with the append done inside the
 * attention launch when every kv head has a single group of query heads
 * (Hq / Hkv <= 8): the split holding pos[b] writes the new rows of its kv
 * head and kv head 0's split sets mask[b, pos[b]], before that split's tiles
 * are read.  Larger groups run the append kernel first.  Arguments as for
 * the two calls (k_new, v_new [B, Hkv, D] of `dtype`, pos [B] int32, mask
 * written); the caches, the mask and the output end exactly as after the two
 * calls.  pos[b] outside [0, C) writes nothing for b and sets
 * KVD_DEV_POS_RANGE; the attention then runs over the mask as it is.
 * Workspace: kvd_attend_masked_workspace_bytes.
 */
kvd_status kvd_append_attend_masked(const void* q, void* k_cache, void* v_cache, uint8_t* mask,
                                    const void* k_new, const void* v_new, const int32_t* pos,
                                    void* out, float* lse_out, int B, int Hq, int Hkv, int C,
                                    int D, float scale, kvd_dtype dtype, int num_splits,
                                    void* workspace, size_t workspace_bytes, int32_t* dev_status,
                                    kvd_stream_t stream);

/*
 * kvd_attend_window -- sliding-window decode attention over the static
 * buffer ([NPU] Part 3, the sliding-window tile variant; Part 1 for the
 * mask): row b attends to the slots j with mask[b, j] != 0 and
 *   last[b] - W + 1 <= j <= last[b],
 * i.e. kvd_attend_masked with every mask slot outside the window taken as 0.
 *   q [B, Hq, D]; k_cache, v_cache [B, Hkv, C, D]; mask [B, C] uint8;
 *   last [B] int32, device (the window's newest slot, normally the slot the
 *   step appended); W >= 1 window slots; out, lse_out, scale, dtype,
 *   workspace, num_splits and dev_status as for kvd_attend_masked.
 * The splits are laid over each row's window only (from the 64-slot boundary
 * at or below last[b] - W + 1), so no slot outside it is scanned or read,
 * whatever C is.  last[b] outside [0, C): row b is empty (out = 0,
 * lse = -inf) and KVD_DEV_POS_RANGE is set.  Always the persistent split
 * kernel (the one-launch cluster kernel holds whole buffers); 1 or 2
 * launches (kvd_attend_window_plan).  Errors as for kvd_attend_masked, and
 * KVD_ERR_INVALID_ARG for W < 1 or a null `last`.
 */
size_t kvd_attend_window_workspace_bytes(int B, int Hq, int Hkv, int C, int D, int W,
                                         kvd_dtype dtype, int num_splits);
/* As kvd_attend_masked_plan, for kvd_attend_window and
 * kvd_append_attend_window (splits >= 1: never the one-launch kernel). */
kvd_status kvd_attend_window_plan(int B, int Hq, int Hkv, int C, int D, int W, kvd_dtype dtype,
                                  int num_splits, kvd_plan* plan);
kvd_status kvd_attend_window(const void* q, const void* k_cache, const void* v_cache,
                             const uint8_t* mask, const int32_t* last, void* out, float* lse_out,
                             int B, int Hq, int Hkv, int C, int D, int W, float scale,
                             kvd_dtype dtype, int num_splits, void* workspace,
                             size_t workspace_bytes, int32_t* dev_status, kvd_stream_t stream);
/*
 * kvd_append_attend_window -- one sliding-window decode step: the result of
 * kvd_append(k_cache, v_cache, k_new, v_new, pos, mask) followed by
 * kvd_attend_window(..., last = pos, W, ...), the append done inside the
 * attention launch as in kvd_append_attend_masked (Hq / Hkv <= 8; larger
 * groups run the append kernel first).  pos[b] outside [0, C): nothing is
 * written for b, row b is empty, KVD_DEV_POS_RANGE is set.  Workspace:
 * kvd_attend_window_workspace_bytes.
 */
kvd_status kvd_append_attend_window(const void* q, void* k_cache, void* v_cache, uint8_t* mask,
                                    const void* k_new, const void* v_new, const int32_t* pos,
                                    void* out, float* lse_out, int B, int Hq, int Hkv, int C,
                                    int D, int W, float scale, kvd_dtype dtype, int num_splits,
                                    void* workspace, size_t workspace_bytes, int32_t* dev_status,
                                    kvd_stream_t stream);

/*
 * kvd_attend_indexed -- decode attention over a list of cache slots per batch
 * entry ([FlashMLA] "Математическая постановка": the indexer's top-k indices
 * pick the KV rows, P = Q . gathered^T, S = softmax(P * sm_scale),
 * out = S . gathered):
 *   out[b, h, :] = sum_j w_j v[b, h/g, indices[b, j], :] / sum_j w_j,
 *   w_j = exp(scale * q[b, h, :] . k[b, h/g, indices[b, j], :] - max), over
 *   the entries j with 0 <= indices[b, j] < C.
 *   q [B, Hq, D]; k_cache, v_cache [B, Hkv, C, D]; indices [B, topk] int32,
 *   device (-1 = unused entry); out [B, Hq, D]; lse_out [B, Hq] float or NULL
 * Every entry is one term of the softmax (a repeated slot counts once per
 * entry; the list order does not matter).  An entry outside [-1, C) is
 * skipped and sets KVD_DEV_POS_RANGE.  No valid entry: out = 0, lse = -inf.
 * The list is cut into splits of at most 128 entries that the persistent grid
 * takes from its work counter; the listed rows are gathered into shared
 * memory with 16-byte cp.async copies.
 * Workspace, num_splits and dtypes as for kvd_attend_masked (the list length
 * topk takes the place of the capacity).
 */
size_t kvd_attend_indexed_workspace_bytes(int B, int Hq, int Hkv, int topk, int D,
                                          kvd_dtype dtype, int num_splits);
/* As kvd_attend_masked_plan, for kvd_attend_indexed (the one-launch cluster
 * kernel is never used: splits >= 1). */
kvd_status kvd_attend_indexed_plan(int B, int Hq, int Hkv, int topk, int D, kvd_dtype dtype,
                                   int num_splits, kvd_plan* plan);
kvd_status kvd_attend_indexed(const void* q, const void* k_cache, const void* v_cache,
                              const int32_t* indices, void* out, float* lse_out, int B, int Hq,
                              int Hkv, int C, int topk, int D, float scale, kvd_dtype dtype,
                              int num_splits, void* workspace, size_t workspace_bytes,
                              int32_t* dev_status, kvd_stream_t stream);

/*
 * Quantised KV rows ([FlashMLA-KV]; the scale granularity and encoding are
 * this library's reading, the page gives neither): one row of a kv head is
 *   bytes [0, D)        OCP FP8 E4M3 codes (bias 7, max 448, no infinities)
 *   bytes [D, D + 4)    the row's scale, fp32 little-endian
 *   bytes [D + 4, D+16) zero
 * so a cache is uint8 [B, Hkv, C, D + KVD_FP8_ROW_PAD] and element d of a row
 * is scale * E4M3(code[d]).  kvd_append_fp8 writes such rows; the attention
 * reads them directly (no bf16 copy of the cache exists).
 */
#define KVD_FP8_ROW_PAD 16

/*
 * kvd_append_fp8 -- kvd_append ([NPU] Part 2, update_kvcache_for) into
 * quantised caches: for every kv head h the new rows k_new[b, h, :],
 * v_new[b, h, :] ([B, Hkv, D], new_dtype bf16 or fp32, finite) are quantised
 *   amax = max_d |x_d|, scale = amax / 448, code_d = E4M3(x_d / scale)
 * (both divisions fp32 round-to-nearest; codes rounded to nearest even and
 * saturated at 448; amax = 0 gives scale 0 and zero codes) and written as
 * row pos[b] of k_cache / v_cache [B, Hkv, C, D + 16] (uint8); mask[b, pos[b]]
 * becomes 1 if mask is not NULL.  D is 64 or 128.  pos[b] outside [0, C)
 * writes nothing for b and sets KVD_DEV_POS_RANGE.
 */
kvd_status kvd_append_fp8(void* k_cache, void* v_cache, const void* k_new, const void* v_new,
                          const int32_t* pos, uint8_t* mask, int B, int Hkv, int C, int D,
                          kvd_dtype new_dtype, int32_t* dev_status, kvd_stream_t stream);

/*
 * kvd_attend_masked_fp8 -- kvd_attend_masked over quantised caches: the same
 * definition with every K/V element dequantised (scale * E4M3(code)).
 *   q [B, Hq, D] bf16; k_cache, v_cache uint8 [B, Hkv, C, D + 16] (rows as
 *   above); mask [B, C]; out [B, Hq, D] bf16; lse_out [B, Hq] float or NULL.
 * The tensor-core kernel never builds a dequantised copy: K codes meet q in
 * fp16 (q is converted to fp16, so |q| must stay below 65504) and each row's
 * scale multiplies its score; V codes meet the softmax weights in fp16, each
 * weight carrying its row's scale relative to a running power of two (row
 * scales must be finite and below 2^126).  D is 64 or 128; any Hq / Hkv (up
 * to 8 query heads per kv head in one group, larger groups are split).
 * Workspace and num_splits as for kvd_attend_masked (64-token tiles), short
 * buffers included: with num_splits = 0 they take the one-launch cluster
 * path.
 */
size_t kvd_attend_masked_fp8_workspace_bytes(int B, int Hq, int Hkv, int C, int D, int num_splits);
/* As kvd_attend_masked_plan, for kvd_attend_masked_fp8. */
kvd_status kvd_attend_masked_fp8_plan(int B, int Hq, int Hkv, int C, int D, int num_splits,
                                      kvd_plan* plan);
kvd_status kvd_attend_masked_fp8(const void* q, const void* k_cache, const void* v_cache,
                                 const uint8_t* mask, void* out, float* lse_out, int B, int Hq,
                                 int Hkv, int C, int D, float scale, int num_splits,
                                 void* workspace, size_t workspace_bytes, int32_t* dev_status,
                                 kvd_stream_t stream);

/*
 * FP4 KV rows ([FlashMLA-KV], which names FP4 beside FP8; the granularity and
 * encoding are this library's reading, as for FP8): one row of a kv head is
 *   bytes [0, D/2)          OCP FP4 E2M1 codes, two per byte: element 2j in
 *                           the low nibble of byte j, 2j + 1 in the high one
 *                           (magnitudes 0, 0.5, 1, 1.5, 2, 3, 4, 6)
 *   bytes [D/2, D/2 + 4)    the row's scale, fp32 little-endian
 *   bytes [D/2 + 4, D/2+16) zero
 * so a cache is uint8 [B, Hkv, C, D/2 + KVD_FP4_ROW_PAD] and element d of a
 * row is scale * E2M1(code[d]).
 */
#define KVD_FP4_ROW_PAD 16

/*
 * kvd_append_fp4 -- kvd_append_fp8 with FP4 rows: per new row
 *   amax = max_d |x_d|, scale = amax / 6, code_d = E2M1(x_d / scale)
 * (both divisions fp32 round-to-nearest; codes rounded to the nearest
 * magnitude, ties to the even code, saturated at 6; amax = 0 gives scale 0
 * and zero codes), written as row pos[b] of k_cache / v_cache
 * [B, Hkv, C, D/2 + 16] (uint8).  Arguments, mask, D and errors as for
 * kvd_append_fp8.
 */
kvd_status kvd_append_fp4(void* k_cache, void* v_cache, const void* k_new, const void* v_new,
                          const int32_t* pos, uint8_t* mask, int B, int Hkv, int C, int D,
                          kvd_dtype new_dtype, int32_t* dev_status, kvd_stream_t stream);

/*
 * kvd_attend_masked_fp4 -- kvd_attend_masked over FP4 caches: the same
 * definition with every K/V element dequantised (scale * E2M1(code)).
 *   k_cache, v_cache uint8 [B, Hkv, C, D/2 + 16]; every other argument, the
 * precision rules (E2M1 codes are exact in fp16), workspace, plan and paths as
 * for kvd_attend_masked_fp8.
 */
size_t kvd_attend_masked_fp4_workspace_bytes(int B, int Hq, int Hkv, int C, int D, int num_splits);
/* As kvd_attend_masked_plan, for kvd_attend_masked_fp4. */
kvd_status kvd_attend_masked_fp4_plan(int B, int Hq, int Hkv, int C, int D, int num_splits,
                                      kvd_plan* plan);
kvd_status kvd_attend_masked_fp4(const void* q, const void* k_cache, const void* v_cache,
                                 const uint8_t* mask, void* out, float* lse_out, int B, int Hq,
                                 int Hkv, int C, int D, float scale, int num_splits,
                                 void* workspace, size_t workspace_bytes, int32_t* dev_status,
                                 kvd_stream_t stream);

/*
 * Quantised rows in the paged layout and through index lists ([FlashMLA-KV]
 * "Оптимизация раскладки KV-кэша при decoding" keeps a token's quantised
 * values and scale side by side, on paged KV blocks).  The rows are those of
 * kvd_append_fp8 (RB = D + 16 bytes) and kvd_append_fp4 (RB = D/2 + 16); q
 * and out are bf16; D in {64, 128}; Hq / Hkv <= 8 query heads per kv head
 * share one tensor-core consumer pass, larger groups several.
 *
 * kvd_append_paged_fp8, kvd_append_paged_fp4 -- kvd_append_paged with the
 * quantisation of kvd_append_fp8 / kvd_append_fp4: the new rows k_new, v_new
 * [Q, Hkv, D] (new_dtype bf16 or fp32) quantised row by row and written as
 * whole rows of key_cache, value_cache uint8 [NB, BS, Hkv, RB] at token pos[q]
 * of sequence q, through the gather's index mapping ([PyPTO] 3.2).  Checks
 * and their status bits in kvd_append_paged's order (a refused sequence
 * writes nothing): pos[q] < 0 KVD_DEV_POS_RANGE, seq_offset[q] negative or
 * not a multiple of BS KVD_DEV_SEQ_OFFSET, a column at or beyond cols
 * KVD_DEV_TABLE_COLS, a block outside [0, NB) KVD_DEV_BLOCK_RANGE.
 */
kvd_status kvd_append_paged_fp8(void* key_cache, void* value_cache, const void* k_new,
                                const void* v_new, const int32_t* block_tables,
                                const int32_t* seq_offset, const int32_t* pos, int Q, int NB,
                                int BS, int cols, int Hkv, int D, kvd_dtype new_dtype,
                                int32_t* dev_status, kvd_stream_t stream);
kvd_status kvd_append_paged_fp4(void* key_cache, void* value_cache, const void* k_new,
                                const void* v_new, const int32_t* block_tables,
                                const int32_t* seq_offset, const int32_t* pos, int Q, int NB,
                                int BS, int cols, int Hkv, int D, kvd_dtype new_dtype,
                                int32_t* dev_status, kvd_stream_t stream);
/*
 * kvd_attend_paged_fp8, kvd_attend_paged_fp4 -- kvd_attend_paged over
 * quantised rows: key_cache, value_cache uint8 [NB, BS, Hkv, RB]; the same
 * definition with every K/V element dequantised (scale * code value), the
 * same sequence and block rules and status bits, and the precision rules of
 * kvd_attend_masked_fp8 / _fp4.  Tiles are whole-row TMA boxes of the largest
 * divisor of BS not above 64 rows; workspace and plan from the queries below
 * (splits >= 1).
 */
size_t kvd_attend_paged_fp8_workspace_bytes(int Q, int Hq, int Hkv, int BS, int cols, int D,
                                            int num_splits);
size_t kvd_attend_paged_fp4_workspace_bytes(int Q, int Hq, int Hkv, int BS, int cols, int D,
                                            int num_splits);
kvd_status kvd_attend_paged_fp8_plan(int Q, int Hq, int Hkv, int BS, int cols, int D,
                                     int num_splits, kvd_plan* plan);
kvd_status kvd_attend_paged_fp4_plan(int Q, int Hq, int Hkv, int BS, int cols, int D,
                                     int num_splits, kvd_plan* plan);
kvd_status kvd_attend_paged_fp8(const void* q, const void* key_cache, const void* value_cache,
                                const int32_t* block_tables, const int32_t* seq_lens,
                                const int32_t* seq_offset, void* out, float* lse_out, int Q,
                                int Hq, int Hkv, int NB, int BS, int cols, int D, float scale,
                                int num_splits, void* workspace, size_t workspace_bytes,
                                int32_t* dev_status, kvd_stream_t stream);
kvd_status kvd_attend_paged_fp4(const void* q, const void* key_cache, const void* value_cache,
                                const int32_t* block_tables, const int32_t* seq_lens,
                                const int32_t* seq_offset, void* out, float* lse_out, int Q,
                                int Hq, int Hkv, int NB, int BS, int cols, int D, float scale,
                                int num_splits, void* workspace, size_t workspace_bytes,
                                int32_t* dev_status, kvd_stream_t stream);
/*
 * kvd_attend_indexed_fp8, kvd_attend_indexed_fp4 -- kvd_attend_indexed over
 * quantised rows: k_cache, v_cache uint8 [B, Hkv, C, RB]; the same definition
 * (every entry with 0 <= indices[b, j] < C one softmax term, entries outside
 * [-1, C) skipped and reported) with every K/V element dequantised; the
 * listed rows are gathered whole (RB bytes) with 16-byte cp.async copies.
 * Precision rules of kvd_attend_masked_fp8 / _fp4; workspace and plan from
 * the queries below (splits of at most 128 entries).
 */
size_t kvd_attend_indexed_fp8_workspace_bytes(int B, int Hq, int Hkv, int topk, int D,
                                              int num_splits);
size_t kvd_attend_indexed_fp4_workspace_bytes(int B, int Hq, int Hkv, int topk, int D,
                                              int num_splits);
kvd_status kvd_attend_indexed_fp8_plan(int B, int Hq, int Hkv, int topk, int D, int num_splits,
                                       kvd_plan* plan);
kvd_status kvd_attend_indexed_fp4_plan(int B, int Hq, int Hkv, int topk, int D, int num_splits,
                                       kvd_plan* plan);
kvd_status kvd_attend_indexed_fp8(const void* q, const void* k_cache, const void* v_cache,
                                  const int32_t* indices, void* out, float* lse_out, int B,
                                  int Hq, int Hkv, int C, int topk, int D, float scale,
                                  int num_splits, void* workspace, size_t workspace_bytes,
                                  int32_t* dev_status, kvd_stream_t stream);
kvd_status kvd_attend_indexed_fp4(const void* q, const void* k_cache, const void* v_cache,
                                  const int32_t* indices, void* out, float* lse_out, int B,
                                  int Hq, int Hkv, int C, int topk, int D, float scale,
                                  int num_splits, void* workspace, size_t workspace_bytes,
                                  int32_t* dev_status, kvd_stream_t stream);

/*
 * kvd_attend_masked_noalloc -- the pages have no counterpart to this call; it
 * exists for callers that cannot allocate device memory.  Some host runtimes
 * own all device memory through their own allocator and hand a kernel library
 * only its input and output buffers; some enqueue paths may not allocate at
 * all; some latency-critical loops cannot afford cudaMalloc's implicit device
 * synchronisation.  Such callers cannot supply the workspace that
 * kvd_attend_masked needs once it splits the sequence axis.
 *
 * Same arguments, same result and the same kernels as kvd_attend_masked,
 * minus the workspace: the split scratch lives in an array of
 * KVD_NOALLOC_SCRATCH_BYTES built into the library, which every GPU that
 * loads the library holds until the process exits.  Nothing is allocated.
 *  - Sizes whose split scratch (kvd_attend_masked_workspace_bytes with the
 *    same arguments) exceeds KVD_NOALLOC_SCRATCH_BYTES are rejected with
 *    KVD_ERR_WORKSPACE and a message in kvd_last_error(); pass fewer splits
 *    (num_splits) or use kvd_attend_masked.
 *  - The first call in a device's context looks up the array's device
 *    address there (cudaGetSymbolAddress) and caches it per context; make
 *    that first call before any stream capture on that device (and again
 *    after a cudaDeviceReset, which loads the library's module anew).
 *  - All calls on a device share the one array, which keeps the last call's
 *    contents.  Each call first clears the array's work counters
 *    (kvd_plan.counter_bytes) with cudaMemsetAsync on `stream`
 *    (stream-ordered; no allocation), so a
 *    call whose launch gave up on a bounded wait (KVD_DEV_TIMEOUT) does not
 *    poison the next one.  Calls that may overlap on the GPU (other streams,
 *    unordered host threads) race on the array: the caller must order them.
 */
#define KVD_NOALLOC_SCRATCH_BYTES (8u << 20)
kvd_status kvd_attend_masked_noalloc(const void* q, const void* k_cache, const void* v_cache,
                                     const uint8_t* mask, void* out, float* lse_out, int B,
                                     int Hq, int Hkv, int C, int D, float scale, kvd_dtype dtype,
                                     int num_splits, int32_t* dev_status, kvd_stream_t stream);

size_t kvd_attend_paged_workspace_bytes(int Q, int Hq, int Hkv, int BS, int cols, int D,
                                        kvd_dtype dtype, int num_splits);
/* As kvd_attend_masked_plan, for kvd_attend_paged (rows = sequences; the
 * one-launch cluster kernel is never used: splits >= 1). */
kvd_status kvd_attend_paged_plan(int Q, int Hq, int Hkv, int BS, int cols, int D, kvd_dtype dtype,
                                 int num_splits, kvd_plan* plan);
kvd_status kvd_attend_paged(const void* q_in, const void* key_cache, const void* value_cache,
                            const int32_t* block_tables, const int32_t* seq_lens,
                            const int32_t* seq_offset, void* out, float* lse_out, int Q, int Hq,
                            int Hkv, int NB, int BS, int cols, int D, float scale,
                            kvd_dtype dtype, int num_splits, void* workspace,
                            size_t workspace_bytes, int32_t* dev_status, kvd_stream_t stream);

/*
 * kvd_append_paged -- the step's KV append ([NPU] Part 2, update_kvcache_for)
 * into the paged cache, through the gather's index mapping ([PyPTO] 3.2):
 * token pos[q] of sequence q is written to
 *   key_cache[block_tables[q, seq_offset[q] / BS + pos[q] / BS], pos[q] % BS]
 * (all Hkv x D of it; value_cache likewise), i.e. where kvd_gather_paged and
 * kvd_attend_paged read token pos[q] of q once seq_lens counts it.
 *   key_cache, value_cache [NB, BS, Hkv, D] of `dtype`
 *   k_new, v_new [Q, Hkv, D] of `dtype`;  pos [Q] int32 (device)
 *   block_tables [Q, cols] int32;  seq_offset [Q] int32 or NULL (zeros)
 * A byte copy.  Device-detected errors skip that sequence (nothing written):
 * pos[q] < 0 (KVD_DEV_POS_RANGE), seq_offset negative or not a multiple of
 * BS (KVD_DEV_SEQ_OFFSET), table column past cols (KVD_DEV_TABLE_COLS), block
 * id outside [0, NB) (KVD_DEV_BLOCK_RANGE).  The caller keeps seq_lens.
 */
kvd_status kvd_append_paged(void* key_cache, void* value_cache, const void* k_new,
                            const void* v_new, const int32_t* block_tables,
                            const int32_t* seq_offset, const int32_t* pos, int Q, int NB, int BS,
                            int cols, int Hkv, int D, kvd_dtype dtype, int32_t* dev_status,
                            kvd_stream_t stream);

/*
 * kvd_gather_paged -- gather_pa_kv_cache, Norm/ND branch ([PyPTO] 3.2):
 * for every sequence q and t < seq_lens[q+1] - seq_lens[q]:
 *   phys = block_tables[q, seq_offset[q] / BS + t / BS]
 *   key_out[seq_lens[q] + t] = key_cache[phys, t % BS]   (all Hk x Dk)
 *   value_out[seq_lens[q] + t] = value_cache[phys, t % BS] (all Hv x Dv)
 *   key_cache [NB, BS, Hk, Dk], value_cache [NB, BS, Hv, Dv], elem_bytes 2 or 4
 *   key_out [total_tokens, Hk, Dk], value_out [total_tokens, Hv, Dv]
 * A byte copy (bit-exact).  total_tokens must equal seq_lens[Q] and is
 * passed from the host.  Device-detected errors (SEQLENS, SEQ_OFFSET,
 * TABLE_COLS) skip the whole sequence; BLOCK_RANGE skips that block's rows;
 * skipped rows are left untouched.  Rows must be whole multiples of 2 bytes.
 */
kvd_status kvd_gather_paged(const void* key_cache, const void* value_cache,
                            const int32_t* block_tables, const int32_t* seq_lens,
                            const int32_t* seq_offset, void* key_out, void* value_out, int Q,
                            int NB, int BS, int cols, int Hk, int Dk, int Hv, int Dv,
                            int total_tokens, int elem_bytes, int32_t* dev_status,
                            kvd_stream_t stream);

/*
 * kvd_combine -- log-sum-exp merge of partial results over disjoint key
 * ranges ([NPU] Part 3, Flash SDPA path: tiles merged exactly):
 *   LSE[r] = log sum_s exp(part_lse[r, s]),
 *   out[r, :] = sum_s exp(part_lse[r, s] - LSE[r]) * part_o[r, s, :]
 *   part_o [R, S, D] float (each normalised over its range), part_lse [R, S]
 *   float (natural log, -inf = empty range whose part_o is ignored)
 *   out [R, D] of out_dtype;  lse_out [R] float or NULL
 * All ranges empty: out = 0, LSE = -inf.  D a multiple of 4, at most 1024.
 */
kvd_status kvd_combine(const float* part_o, const float* part_lse, void* out, float* lse_out,
                       int R, int S, int D, kvd_dtype out_dtype, kvd_stream_t stream);

/*
 * kvd_combine_gathered -- kvd_combine over the exchange layout of a
 * sequence split across S ranks: `parts` float [S, R * (D + 1)] holds, for
 * range s, its R partial rows [R, D] followed by their R log-sum-exps
 * (kvd_attend_masked_partial writing out and lse_out into the two parts of
 * one rank's block), the blocks one after the other as an all-gather of the
 * blocks along the first axis leaves them.  Same formula, outputs and rules
 * as kvd_combine (range s of row r has part_o = parts[s, r*D : (r+1)*D] and
 * part_lse = parts[s, R*D + r]).
 */
kvd_status kvd_combine_gathered(const float* parts, void* out, float* lse_out, int R, int S,
                                int D, kvd_dtype out_dtype, kvd_stream_t stream);

/* Human-readable name of a status code (static string). */
const char* kvd_status_string(kvd_status status);
/* Description of the last error returned on the calling thread (static per thread). */
const char* kvd_last_error(void);
/* Library ABI version: major * 10000 + minor * 100 + patch. */
int kvd_version(void);

#ifdef __cplusplus
}
#endif
#endif /* KVD_H */
