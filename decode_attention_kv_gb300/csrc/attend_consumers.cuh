// attend_consumers.cuh -- the consumer warps of the split-KV decode attention
// kernel: what they do with one ring tile of K/V rows.
//
// Both policies keep, per query head, the fp32 running max m (log2 units),
// running sum l and unnormalised output acc over the tokens they have seen,
// and update them per block of tokens with the correction exp(m_old - m_new)
// ("Intel NPU running LLMs", Part 3 "Flash SDPA 路径" and Part 6 "ONNX 表达不了
// tiling 策略"; "FlashMLA на Huawei Ascend", "Ход вычислений").  Slots whose
// validity bit is 0 (mask = 0, past the sequence, dropped block) take no part
// (Part 1 "解决方案：预分配 + Attention Mask").
//
//  SimtConsumer: CUDA cores.  D/VEC lanes hold one token's row as 16-byte
//    vectors; q.k with packed fp32x2 FMAs and a shuffle reduction over the
//    token's lanes; the running state is updated once per sub-chunk of tokens;
//    p.V with packed FMAs.  Used for fp32 and for 1-2 query heads per kv head.
//  MmaConsumer: tensor cores for bf16 groups of 4-8 query heads per kv head.
//    q.K^T of a 16-token slab is mma.m16n8k16 with tokens on M and the packed
//    heads on N; p.V is V^T p^T with p rounded to bf16 first ("FlashMLA на
//    Huawei Ascend": S is cast to bf16 before S.V) while the running sum l
//    keeps the fp32 p, so that the log-sum-exp stays exact to fp32 rounding;
//    K/V tiles arrive in the 128-byte swizzle so that ldmatrix is
//    conflict-free; V rows of invalid tokens are zeroed first so that inf/NaN
//    padding cannot reach the accumulator through 0 x inf.
//
// Both skip the rescale of the running output when a block's maximum is at
// most kSkipScale above the running max ("FlashMLA на Huawei Ascend", the
// online-softmax section: skip-scale with threshold 6): the stale max stays
// the exponent base, so the block's weights reach at most e^6 (~400), well
// inside fp32, and the result is the same up to rounding.  A warp rescales
// only when one of its lanes needs it.
//
//  QuantMmaConsumer (Fp8MmaConsumer / Fp4MmaConsumer): tensor cores over
//    quantised K/V rows (E4M3 codes, or E2M1 codes two per byte, the row's
//    fp32 scale beside them; "FlashMLA на Huawei Ascend", "Ограничение по
//    деквантованию" and "Оптимизация раскладки KV-кэша при decoding").  The
//    codes become f16 in registers (exactly), read with plain shared loads
//    in a dims-to-lanes order that both mma operands share; each row's scale
//    multiplies its score (K) or its weight p (V), so no element is ever
//    multiplied by its scale.  Any query head count up to 8 per kv head.
//
// finish() leaves each warp's state in shared memory as mo[w][h][d]
// (unnormalised output) and ml[w][h] = (m, l) for the CTA-wide merge.
#pragma once

#include "kvd_device.cuh"
#include "mma_ptx.cuh"

namespace kvd {

constexpr float kSkipScale = 6.f * kLog2e;  // threshold 6 (natural log) in log2 units

template <typename Elem, int D, int G, int T, int NCW>
struct SimtConsumer {
    using Tr = ElemTraits<Elem>;
    using ElemT = Elem;
    static constexpr bool kSwizzled = false;
    static constexpr int kD = D, kG = G, kT = T, kNCW = NCW;
    static constexpr int kVec = Tr::kPerVec;   // elements per 16-byte lane vector
    static constexpr int kPairs = kVec / 2;
    static constexpr int kLPT = D / kVec;      // lanes per token
    static constexpr int kTPW = 32 / kLPT;     // tokens per warp step
    static constexpr int kTW = T / NCW;        // tokens per warp per tile
    static constexpr int kSteps = kTW / kTPW;  // warp steps per tile
    static constexpr int kSubWant = (32 / G) < 1 ? 1 : (32 / G);
    static constexpr int kSub = kSteps < kSubWant ? kSteps : kSubWant;
    static constexpr int kTileBytes = T * D * (int)sizeof(Elem);  // K (or V) of one tile
    static constexpr int kRowBytes = D * (int)sizeof(Elem);
    static_assert(D % kVec == 0 && kLPT <= 32 && 32 % kLPT == 0, "head_dim layout");
    static_assert(T % NCW == 0 && kTW % kTPW == 0 && kSteps % kSub == 0, "tile layout");
    static_assert(T <= 64, "validity bits of a tile fit 64 bits");

    float2 q2[G][kPairs];
    float m[G], l[G];
    float2 acc[G][kPairs];

    // q rows of the unit (staged in shared memory), scaled by scale*log2(e).
    __device__ __forceinline__ void begin(const Elem* qs, int g_here, float qscale, int lane) {
        const int sub = lane % kLPT;
#pragma unroll
        for (int hh = 0; hh < G; ++hh) {
            if (hh < g_here) {
                const uint4 raw = *reinterpret_cast<const uint4*>(qs + hh * D + sub * kVec);
                Tr::unpack(raw, q2[hh]);
#pragma unroll
                for (int j = 0; j < kPairs; ++j) q2[hh][j] = fmul2(q2[hh][j], make_float2(qscale, qscale));
            } else {
#pragma unroll
                for (int j = 0; j < kPairs; ++j) q2[hh][j] = make_float2(0.f, 0.f);
            }
            m[hh] = -INFINITY;
            l[hh] = 0.f;
#pragma unroll
            for (int j = 0; j < kPairs; ++j) acc[hh][j] = make_float2(0.f, 0.f);
        }
    }

    // One tile; returns whether it wrote to the ring (never, here).
    __device__ __forceinline__ bool tile(unsigned char* kbuf, unsigned char* vbuf, uint64_t bits,
                                         int warp, int lane, float /*qscale: folded into q*/) {
        const Elem* Ks = reinterpret_cast<const Elem*>(kbuf);
        const Elem* Vs = reinterpret_cast<const Elem*>(vbuf);
        const int grp = lane / kLPT, sub = lane % kLPT;
#pragma unroll
        for (int c = 0; c < kSteps; c += kSub) {
            float s[kSub][G];
            bool val[kSub];
#pragma unroll
            for (int i = 0; i < kSub; ++i) {
                const int tt = warp * kTW + (c + i) * kTPW + grp;
                const uint4 kr = *reinterpret_cast<const uint4*>(Ks + tt * D + sub * kVec);
                float2 kf[kPairs];
                Tr::unpack(kr, kf);
#pragma unroll
                for (int hh = 0; hh < G; ++hh) {
                    float2 a = fmul2(q2[hh][0], kf[0]);
#pragma unroll
                    for (int j = 1; j < kPairs; ++j) a = ffma2(q2[hh][j], kf[j], a);
                    s[i][hh] = a.x + a.y;
                }
                val[i] = (bits >> tt) & 1ull;
            }
#pragma unroll
            for (int off = kLPT / 2; off > 0; off >>= 1)
#pragma unroll
                for (int i = 0; i < kSub; ++i)
#pragma unroll
                    for (int hh = 0; hh < G; ++hh)
                        s[i][hh] += __shfl_xor_sync(0xffffffffu, s[i][hh], off);

            float pr[kSub][G];
#pragma unroll
            for (int hh = 0; hh < G; ++hh) {
                float mx = -INFINITY;
#pragma unroll
                for (int i = 0; i < kSub; ++i) {
                    s[i][hh] = val[i] ? s[i][hh] : -INFINITY;
                    mx = fmaxf(mx, s[i][hh]);
                }
                const bool up = mx > m[hh] + kSkipScale;  // m = -inf: any finite mx
                const float mn = up ? mx : m[hh];
                const float base = (mn == -INFINITY) ? 0.f : mn;
                const float corr = up ? fast_exp2(m[hh] - base) : 1.f;
                m[hh] = mn;
                float ls = 0.f;
#pragma unroll
                for (int i = 0; i < kSub; ++i) {
                    pr[i][hh] = fast_exp2(s[i][hh] - base);
                    ls += pr[i][hh];
                }
                l[hh] = fmaf(l[hh], corr, ls);
                if (__any_sync(0xffffffffu, up)) {
                    const float2 c2 = make_float2(corr, corr);
#pragma unroll
                    for (int j = 0; j < kPairs; ++j) acc[hh][j] = fmul2(acc[hh][j], c2);
                }
            }
#pragma unroll
            for (int i = 0; i < kSub; ++i) {
                const int tt = warp * kTW + (c + i) * kTPW + grp;
                uint4 vr = *reinterpret_cast<const uint4*>(Vs + tt * D + sub * kVec);
                if (!val[i]) vr = make_uint4(0, 0, 0, 0);  // padding may hold inf/NaN
                float2 vf[kPairs];
                Tr::unpack(vr, vf);
#pragma unroll
                for (int hh = 0; hh < G; ++hh) {
                    const float2 pp = make_float2(pr[i][hh], pr[i][hh]);
#pragma unroll
                    for (int j = 0; j < kPairs; ++j) acc[hh][j] = ffma2(pp, vf[j], acc[hh][j]);
                }
            }
        }
        return false;
    }

    // Merge the lane groups (different tokens) of the warp; leave the warp's
    // state in mo / ml.
    __device__ __forceinline__ void finish(float* mo, float* ml, int warp, int lane) {
#pragma unroll
        for (int off = kLPT; off < 32; off <<= 1) {
#pragma unroll
            for (int hh = 0; hh < G; ++hh) {
                const float mo_ = __shfl_xor_sync(0xffffffffu, m[hh], off);
                const float lo = __shfl_xor_sync(0xffffffffu, l[hh], off);
                const float mn = fmaxf(m[hh], mo_);
                const float base = (mn == -INFINITY) ? 0.f : mn;
                const float a = fast_exp2(m[hh] - base), b = fast_exp2(mo_ - base);
                l[hh] = l[hh] * a + lo * b;
                m[hh] = mn;
#pragma unroll
                for (int j = 0; j < kPairs; ++j) {
                    float2 other;
                    other.x = __shfl_xor_sync(0xffffffffu, acc[hh][j].x, off);
                    other.y = __shfl_xor_sync(0xffffffffu, acc[hh][j].y, off);
                    acc[hh][j] = ffma2(acc[hh][j], make_float2(a, a), fmul2(other, make_float2(b, b)));
                }
            }
        }
        const int grp = lane / kLPT, sub = lane % kLPT;
        if (grp == 0) {
#pragma unroll
            for (int hh = 0; hh < G; ++hh) {
#pragma unroll
                for (int j = 0; j < kPairs; ++j) {
                    const int d = sub * kVec + 2 * j;
                    mo[(warp * G + hh) * D + d] = acc[hh][j].x;
                    mo[(warp * G + hh) * D + d + 1] = acc[hh][j].y;
                }
                if (sub == 0) {
                    ml[(warp * G + hh) * 2] = m[hh];
                    ml[(warp * G + hh) * 2 + 1] = l[hh];
                }
            }
        }
    }
};

template <int D, int G, int T, int NCW>
struct MmaConsumer {
    using ElemT = __nv_bfloat16;
    static constexpr bool kSwizzled = true;
    static constexpr int kD = D, kG = G, kT = T, kNCW = NCW;
    static constexpr int kHalves = D / 64;      // 128-byte column halves per row
    static constexpr int kHalfBytes = T * 128;
    static constexpr int kTileBytes = kHalves * kHalfBytes;
    static constexpr int kRowBytes = D * 2;
    static constexpr int kSlabsPerWarp = T / 16 / NCW;
    static constexpr int kKSteps = D / 16;      // q.K^T: 16 dims per mma
    static constexpr int kDBlocks = D / 16;     // p.V: 16 output dims per mma
    static_assert(D % 64 == 0, "head_dim must be a multiple of 64");
    static_assert(G >= 1 && G <= 8, "at most 8 query heads per mma column block");
    static_assert(T % (16 * NCW) == 0 && kSlabsPerWarp >= 1, "16-token slabs per warp");
    static_assert(kHalfBytes % 1024 == 0, "swizzled halves stay 1024-byte aligned");
    static_assert(T <= 64, "validity bits of a tile fit 64 bits");

    uint32_t qb[kKSteps][2];  // q^T as the B operand: column gid = query head
    float m[2], l[2];         // columns (heads) 2*tig, 2*tig + 1; l: this thread's rows
    float acc[kDBlocks][4];   // V^T p^T: rows d*16 + gid (+8), columns 2*tig (+1)

    __device__ __forceinline__ void begin(const __nv_bfloat16* qs, int g_here, float /*qscale*/,
                                          int lane) {
        const int gid = lane >> 2, tig = lane & 3;
#pragma unroll
        for (int ks = 0; ks < kKSteps; ++ks) {
            if (gid < g_here) {
                const __nv_bfloat16* qp = qs + gid * D + ks * 16 + 2 * tig;
                qb[ks][0] = *reinterpret_cast<const uint32_t*>(qp);
                qb[ks][1] = *reinterpret_cast<const uint32_t*>(qp + 8);
            } else {
                qb[ks][0] = qb[ks][1] = 0u;
            }
        }
        m[0] = m[1] = -INFINITY;
        l[0] = l[1] = 0.f;
#pragma unroll
        for (int d = 0; d < kDBlocks; ++d) acc[d][0] = acc[d][1] = acc[d][2] = acc[d][3] = 0.f;
    }

    __device__ __forceinline__ bool tile(unsigned char* kbuf, unsigned char* vbuf, uint64_t bits,
                                         int warp, int lane, float qscale) {
        const int gid = lane >> 2;
        const uint32_t kbase = smem_u32(kbuf), vbase = smem_u32(vbuf);
        bool wrote = false;
#pragma unroll
        for (int sl = 0; sl < kSlabsPerWarp; ++sl) {
            const int slab0 = (warp * kSlabsPerWarp + sl) * 16;
            const uint32_t vmask = (uint32_t)(bits >> slab0) & 0xffffu;
            if (vmask == 0u) continue;
            if (vmask != 0xffffu) {
                for (int i = lane; i < 16 * kHalves * 8; i += 32) {
                    const int row = i / (kHalves * 8);
                    const int rest = i % (kHalves * 8);
                    if (!((vmask >> row) & 1u)) {
                        const int h = rest >> 3, ch = rest & 7;
                        *reinterpret_cast<uint4*>(vbuf + h * kHalfBytes + (slab0 + row) * 128 +
                                                  ch * 16) = make_uint4(0u, 0u, 0u, 0u);
                    }
                }
                wrote = true;
                __syncwarp();
            }
            const bool v_lo = (vmask >> gid) & 1u, v_hi = (vmask >> (gid + 8)) & 1u;

            // two accumulators (even and odd k-steps) halve the mma chain
            float s[4] = {0.f, 0.f, 0.f, 0.f}, s2[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
            for (int ks = 0; ks < kKSteps; ++ks) {
                uint32_t a[4];
                const int row = slab0 + (lane & 15);
                const int ch = (ks & 3) * 2 + (lane >> 4);
                ldsm_x4(kbase + (ks >> 2) * kHalfBytes + swz128(row, ch), a);
                mma_bf16((ks & 1) ? s2 : s, a, qb[ks][0], qb[ks][1]);
            }
#pragma unroll
            for (int i = 0; i < 4; ++i) s[i] += s2[i];
            s[0] = v_lo ? s[0] * qscale : -INFINITY;
            s[1] = v_lo ? s[1] * qscale : -INFINITY;
            s[2] = v_hi ? s[2] * qscale : -INFINITY;
            s[3] = v_hi ? s[3] * qscale : -INFINITY;

            float mx0 = fmaxf(s[0], s[2]), mx1 = fmaxf(s[1], s[3]);
#pragma unroll
            for (int off = 4; off < 32; off <<= 1) {
                mx0 = fmaxf(mx0, __shfl_xor_sync(0xffffffffu, mx0, off));
                mx1 = fmaxf(mx1, __shfl_xor_sync(0xffffffffu, mx1, off));
            }
            const bool up0 = mx0 > m[0] + kSkipScale, up1 = mx1 > m[1] + kSkipScale;
            const float mn0 = up0 ? mx0 : m[0], mn1 = up1 ? mx1 : m[1];
            const float b0 = mn0 == -INFINITY ? 0.f : mn0, b1 = mn1 == -INFINITY ? 0.f : mn1;
            const float c0 = up0 ? fast_exp2(m[0] - b0) : 1.f, c1 = up1 ? fast_exp2(m[1] - b1) : 1.f;
            m[0] = mn0;
            m[1] = mn1;
            const float p0 = fast_exp2(s[0] - b0), p1 = fast_exp2(s[1] - b1);
            const float p2 = fast_exp2(s[2] - b0), p3 = fast_exp2(s[3] - b1);
            // l from the fp32 p (the log-sum-exp stays exact to fp32 rounding);
            // p.V from p rounded to bf16 (a relative error of at most 2^-9 per weight)
            l[0] = fmaf(l[0], c0, p0 + p2);
            l[1] = fmaf(l[1], c1, p1 + p3);
            const uint32_t pk_lo = pack_bf16x2(p0, p1), pk_hi = pack_bf16x2(p2, p3);
            if (__any_sync(0xffffffffu, up0 || up1)) {
                const float2 cc = make_float2(c0, c1);
#pragma unroll
                for (int d = 0; d < kDBlocks; ++d) {
                    const float2 x = fmul2(make_float2(acc[d][0], acc[d][1]), cc);
                    const float2 y = fmul2(make_float2(acc[d][2], acc[d][3]), cc);
                    acc[d][0] = x.x;
                    acc[d][1] = x.y;
                    acc[d][2] = y.x;
                    acc[d][3] = y.y;
                }
            }

            const uint32_t bh0 = movmatrix_trans(pk_lo), bh1 = movmatrix_trans(pk_hi);
#pragma unroll
            for (int d = 0; d < kDBlocks; ++d) {
                uint32_t a[4];
                const int row = slab0 + (lane & 7) + ((lane >> 4) << 3);
                const int ch = (d & 3) * 2 + ((lane >> 3) & 1);
                ldsm_x4_trans(vbase + (d >> 2) * kHalfBytes + swz128(row, ch), a);
                mma_bf16(acc[d], a, bh0, bh1);
            }
        }
        return wrote;
    }

    __device__ __forceinline__ void finish(float* mo, float* ml, int warp, int lane) {
        const int gid = lane >> 2, tig = lane & 3;
#pragma unroll
        for (int off = 4; off < 32; off <<= 1) {
            l[0] += __shfl_xor_sync(0xffffffffu, l[0], off);
            l[1] += __shfl_xor_sync(0xffffffffu, l[1], off);
        }
#pragma unroll
        for (int c = 0; c < 2; ++c) {
            const int hh = 2 * tig + c;
            if (hh < G) {
#pragma unroll
                for (int d = 0; d < kDBlocks; ++d) {
                    mo[(warp * G + hh) * D + d * 16 + gid] = acc[d][c];
                    mo[(warp * G + hh) * D + d * 16 + gid + 8] = acc[d][2 + c];
                }
                if (gid == 0) {
                    ml[(warp * G + hh) * 2] = m[c];
                    ml[(warp * G + hh) * 2 + 1] = l[c];
                }
            }
        }
    }
};

// Quantised rows: kRowBytes = D codes + fp32 scale + 12 zero bytes.
//  q.K^T, per k-step ks of 16 dims: lane (gid, tig) holds k-indices 2tig,
//    2tig+1, 2tig+8, 2tig+9, mapped to dims (D/4)tig + 4ks + 0..3, so that
//    its K codes for all k-steps are D/4 consecutive bytes of a row (one or
//    two 16-byte loads per token, conflict-free for the 16 * (D + 16)-byte
//    stride) and q takes the same order.  K codes -> f16 exactly; q -> f16
//    (exact for |q| in the f16 normal range); the score is then scaled by the
//    row's K scale.
//  p.V as V^T p^T, per 16-dim block j: m-row r < 8 is dim (D/8)r + 2j, row
//    r + 8 is dim (D/8)r + 2j + 1, so that lane gid's V codes of all blocks
//    are D/8 consecutive bytes of a row.  V codes -> f16 exactly; each
//    token's weight p carries its V scale divided by 2^ve, where 2^ve is the
//    power of two of the largest V scale seen so far (a running maximum like
//    the softmax's: when it grows, the output is rescaled by an exact power
//    of two), so the f16 weights stay within 2 * e^6 and keep 11 bits; the
//    output is multiplied by 2^ve at the end.
// FP4 rows (kFp4): D/2 bytes of E2M1 codes (element 2j in the low nibble of
// byte j) + fp32 scale + 12 zero bytes.  The same dims-to-lanes order: a
// lane's K codes are D/8 consecutive bytes (two codes per byte, one byte per
// two dims of a k-step), its V codes D/16 bytes; for V the codes of the two
// tokens that share an f16x2 fragment register are interleaved nibble-wise
// before the E2M1 -> f16 conversion (exact).
template <int D, int G, int T, int NCW, bool kFp4>
struct QuantMmaConsumer {
    using ElemT = __nv_bfloat16;  // q and out
    static constexpr bool kSwizzled = false;
    static constexpr int kD = D, kG = G, kT = T, kNCW = NCW;
    static constexpr int kCodeBytes = kFp4 ? D / 2 : D;  // codes of a row; the scale follows
    static constexpr int kRowBytes = kCodeBytes + 16;
    static constexpr int kTileBytes = T * kRowBytes;
    static constexpr int kSlabsPerWarp = T / 16 / NCW;
    static constexpr int kKSteps = D / 16;
    static constexpr int kDBlocks = D / 16;
    static constexpr int kKWords = kFp4 ? D / 32 : D / 16;  // words of a lane's K codes
    static constexpr int kVWords = kFp4 ? D / 64 : D / 32;  // words of a lane's V codes
    static_assert(D == 64 || D == 128, "head_dim 64 or 128");
    static_assert(G >= 1 && G <= 8, "at most 8 query heads per mma column block");
    static_assert(T % (16 * NCW) == 0 && kSlabsPerWarp >= 1, "16-token slabs per warp");
    static_assert(T <= 64, "validity bits of a tile fit 64 bits");

    uint32_t qb[kKSteps][2];  // q^T as the f16 B operand, dims in the order above
    float m[2], l[2];         // heads 2*tig, 2*tig + 1
    float acc[kDBlocks][4];   // out^T / 2^(ve-127): dims (D/8)gid + 2j (+1 for 2, 3), heads 2tig (+1)
    int ve;                   // biased exponent of the largest V scale so far (0: none yet)
    float vinv;               // 2^(127 - ve)

    // 2^k for -126 <= k <= 127 (0 below)
    __device__ __forceinline__ static float pow2i(int k) {
        return __int_as_float(k < -126 ? 0 : (k + 127) << 23);
    }

    __device__ __forceinline__ void begin(const __nv_bfloat16* qs, int g_here, float /*qscale*/,
                                          int lane) {
        const int gid = lane >> 2, tig = lane & 3;
#pragma unroll
        for (int ks = 0; ks < kKSteps; ++ks) {
            if (gid < g_here) {
                const __nv_bfloat16* qp = qs + gid * D + (D / 4) * tig + 4 * ks;
                qb[ks][0] = pack_f16x2(__bfloat162float(qp[0]), __bfloat162float(qp[1]));
                qb[ks][1] = pack_f16x2(__bfloat162float(qp[2]), __bfloat162float(qp[3]));
            } else {
                qb[ks][0] = qb[ks][1] = 0u;
            }
        }
        m[0] = m[1] = -INFINITY;
        l[0] = l[1] = 0.f;
        ve = 0;
        vinv = 0.f;
#pragma unroll
        for (int d = 0; d < kDBlocks; ++d) acc[d][0] = acc[d][1] = acc[d][2] = acc[d][3] = 0.f;
    }

    // N 16-token slabs (rows at kb[n], vb[n]; validity vmask[n], nonzero)
    // under one softmax update (the tiles use N = 1).
    template <int N>
    __device__ __forceinline__ void slabs(const unsigned char* const* kb,
                                          const unsigned char* const* vb, const uint32_t* vmask,
                                          int lane, float qscale) {
        const int gid = lane >> 2, tig = lane & 3;
        // V scales of tokens gid, gid + 8 of each slab (0 for invalid rows)
        // and the running power of two of the largest one
        float sv0[N], sv1[N];
        float smax = 0.f;
#pragma unroll
        for (int n = 0; n < N; ++n) {
            const unsigned char* vs = vb[n] + gid * kRowBytes + kCodeBytes;
            sv0[n] = (vmask[n] >> gid) & 1u ? *reinterpret_cast<const float*>(vs) : 0.f;
            sv1[n] = (vmask[n] >> (gid + 8)) & 1u ? *reinterpret_cast<const float*>(vs + 8 * kRowBytes)
                                                  : 0.f;
            smax = fmaxf(smax, fmaxf(sv0[n], sv1[n]));
        }
#pragma unroll
        for (int off = 4; off < 32; off <<= 1)
            smax = fmaxf(smax, __shfl_xor_sync(0xffffffffu, smax, off));
        const int es = (__float_as_int(smax) >> 23) & 0xff;  // warp-uniform
        if (es > ve) {
            const float r = pow2i(ve - es);
#pragma unroll
            for (int d = 0; d < kDBlocks; ++d) {
                acc[d][0] *= r;
                acc[d][1] *= r;
                acc[d][2] *= r;
                acc[d][3] *= r;
            }
            ve = es;
            vinv = pow2i(127 - es);
        }

        // V codes of tokens 2tig, 2tig+1, 2tig+8, 2tig+9 of slab n: the lane's
        // D/8 dims from byte (D/8)gid (E4M3) or (D/16)gid (E2M1); codes of
        // invalid rows become 0 (NaN codes must not meet a 0 weight).  E4M3
        // requests them before q.K^T (their shared loads then overlap it),
        // E2M1 after the softmax (measured faster each way).
        uint32_t vw[N][4][kVWords];
        auto load_v = [&](int n) {
#pragma unroll
            for (int u = 0; u < 4; ++u) {
                const int t = 2 * tig + (u & 1) + (u >> 1) * 8;
                const unsigned char* vr = vb[n] + t * kRowBytes + 4 * kVWords * gid;
                const bool ok = (vmask[n] >> t) & 1u;
                if constexpr (kVWords == 4) {
                    const uint4 x = *reinterpret_cast<const uint4*>(vr);
                    vw[n][u][0] = ok ? x.x : 0u;
                    vw[n][u][1] = ok ? x.y : 0u;
                    vw[n][u][2] = ok ? x.z : 0u;
                    vw[n][u][3] = ok ? x.w : 0u;
                } else if constexpr (kVWords == 2) {
                    const uint2 x = *reinterpret_cast<const uint2*>(vr);
                    vw[n][u][0] = ok ? x.x : 0u;
                    vw[n][u][1] = ok ? x.y : 0u;
                } else {
                    const uint32_t x = *reinterpret_cast<const uint32_t*>(vr);
                    vw[n][u][0] = ok ? x : 0u;
                }
            }
        };
        if constexpr (!kFp4) {
#pragma unroll
            for (int n = 0; n < N; ++n) load_v(n);
        }

        // ---- q.K^T: tokens gid, gid + 8 of each slab
        float s[N][4];
#pragma unroll
        for (int n = 0; n < N; ++n) {
            const unsigned char* k0 = kb[n] + gid * kRowBytes;
            const unsigned char* k1 = k0 + 8 * kRowBytes;
            uint32_t kw0[kKWords], kw1[kKWords];
            uint32_t kf0[4], kf1[4];  // FP4: one word's four converted pairs
            constexpr int kLaneKBytes = 4 * kKWords;
            if constexpr (kKWords >= 4) {
#pragma unroll
                for (int i = 0; i < kKWords / 4; ++i) {
                    const uint4 x = *reinterpret_cast<const uint4*>(k0 + kLaneKBytes * tig + 16 * i);
                    const uint4 y = *reinterpret_cast<const uint4*>(k1 + kLaneKBytes * tig + 16 * i);
                    kw0[4 * i] = x.x; kw0[4 * i + 1] = x.y; kw0[4 * i + 2] = x.z; kw0[4 * i + 3] = x.w;
                    kw1[4 * i] = y.x; kw1[4 * i + 1] = y.y; kw1[4 * i + 2] = y.z; kw1[4 * i + 3] = y.w;
                }
            } else {
                const uint2 x = *reinterpret_cast<const uint2*>(k0 + kLaneKBytes * tig);
                const uint2 y = *reinterpret_cast<const uint2*>(k1 + kLaneKBytes * tig);
                kw0[0] = x.x; kw0[1] = x.y;
                kw1[0] = y.x; kw1[1] = y.y;
            }
            const float sk0 = *reinterpret_cast<const float*>(k0 + kCodeBytes) * qscale;
            const float sk1 = *reinterpret_cast<const float*>(k1 + kCodeBytes) * qscale;
            // one slab: two accumulators (even and odd k-steps) halve the mma chain
            float t[4] = {0.f, 0.f, 0.f, 0.f}, t2[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
            for (int ks = 0; ks < kKSteps; ++ks) {
                uint32_t a[4];
                if constexpr (kFp4) {
                    // one word per two k-steps: bytes 2(ks%2), 2(ks%2)+1 hold dims
                    // 4ks..4ks+1 and 4ks+2..4ks+3 of the lane's range
                    if ((ks & 1) == 0) {
                        e2m1x8_to_f16x2x4(kw0[ks >> 1], kf0);
                        e2m1x8_to_f16x2x4(kw1[ks >> 1], kf1);
                    }
                    const int h = 2 * (ks & 1);
                    a[0] = kf0[h];
                    a[1] = kf1[h];
                    a[2] = kf0[h + 1];
                    a[3] = kf1[h + 1];
                } else {
                    uint32_t x[2], y[2];
                    e4m3x4_to_f16x2x2(kw0[ks], x);
                    e4m3x4_to_f16x2x2(kw1[ks], y);
                    a[0] = x[0];
                    a[1] = y[0];
                    a[2] = x[1];
                    a[3] = y[1];
                }
                mma_f16((N == 1 && (ks & 1)) ? t2 : t, a, qb[ks][0], qb[ks][1]);
            }
            const bool v_lo = (vmask[n] >> gid) & 1u, v_hi = (vmask[n] >> (gid + 8)) & 1u;
            s[n][0] = v_lo ? (t[0] + t2[0]) * sk0 : -INFINITY;
            s[n][1] = v_lo ? (t[1] + t2[1]) * sk0 : -INFINITY;
            s[n][2] = v_hi ? (t[2] + t2[2]) * sk1 : -INFINITY;
            s[n][3] = v_hi ? (t[3] + t2[3]) * sk1 : -INFINITY;
        }

        float mx0 = -INFINITY, mx1 = -INFINITY;
#pragma unroll
        for (int n = 0; n < N; ++n) {
            mx0 = fmaxf(mx0, fmaxf(s[n][0], s[n][2]));
            mx1 = fmaxf(mx1, fmaxf(s[n][1], s[n][3]));
        }
#pragma unroll
        for (int off = 4; off < 32; off <<= 1) {
            mx0 = fmaxf(mx0, __shfl_xor_sync(0xffffffffu, mx0, off));
            mx1 = fmaxf(mx1, __shfl_xor_sync(0xffffffffu, mx1, off));
        }
        const bool up0 = mx0 > m[0] + kSkipScale, up1 = mx1 > m[1] + kSkipScale;
        const float mn0 = up0 ? mx0 : m[0], mn1 = up1 ? mx1 : m[1];
        const float b0 = mn0 == -INFINITY ? 0.f : mn0, b1 = mn1 == -INFINITY ? 0.f : mn1;
        const float c0 = up0 ? fast_exp2(m[0] - b0) : 1.f, c1 = up1 ? fast_exp2(m[1] - b1) : 1.f;
        m[0] = mn0;
        m[1] = mn1;
        float p[N][4];
        float ps0 = 0.f, ps1 = 0.f;
#pragma unroll
        for (int n = 0; n < N; ++n) {
            p[n][0] = fast_exp2(s[n][0] - b0);
            p[n][1] = fast_exp2(s[n][1] - b1);
            p[n][2] = fast_exp2(s[n][2] - b0);
            p[n][3] = fast_exp2(s[n][3] - b1);
            ps0 += p[n][0] + p[n][2];
            ps1 += p[n][1] + p[n][3];
        }
        l[0] = fmaf(l[0], c0, ps0);
        l[1] = fmaf(l[1], c1, ps1);
        if (__any_sync(0xffffffffu, up0 || up1)) {
            const float2 cc = make_float2(c0, c1);
#pragma unroll
            for (int d = 0; d < kDBlocks; ++d) {
                const float2 x = fmul2(make_float2(acc[d][0], acc[d][1]), cc);
                const float2 y = fmul2(make_float2(acc[d][2], acc[d][3]), cc);
                acc[d][0] = x.x;
                acc[d][1] = x.y;
                acc[d][2] = y.x;
                acc[d][3] = y.y;
            }
        }

        // ---- p.V: weights times V scale / 2^ve in f16, zero for invalid rows
        uint32_t bh0[N], bh1[N];
#pragma unroll
        for (int n = 0; n < N; ++n) {
            const float w0 = sv0[n] * vinv, w1 = sv1[n] * vinv;
            bh0[n] = movmatrix_trans(pack_f16x2(p[n][0] * w0, p[n][1] * w0));
            bh1[n] = movmatrix_trans(pack_f16x2(p[n][2] * w1, p[n][3] * w1));
        }
#pragma unroll
        for (int n = 0; n < N; ++n) {
            if constexpr (kFp4) load_v(n);
            // FP4: byte j of the lane's range holds dims 2j (low nibble) and
            // 2j + 1 (high); pair the two tokens of a fragment register
            // nibble-wise, four bytes (blocks) per word: byte j of vlo[.]
            // holds (dim 2j of token 2tig | of token 2tig + 1), of vhi[.] dim
            // 2j + 1
            uint32_t vlo[2][kVWords], vhi[2][kVWords];
            if constexpr (kFp4) {
#pragma unroll
                for (int h = 0; h < 2; ++h)
#pragma unroll
                    for (int w = 0; w < kVWords; ++w) {
                        const uint32_t x0 = vw[n][2 * h][w], x1 = vw[n][2 * h + 1][w];
                        vlo[h][w] = (x0 & 0x0f0f0f0fu) | ((x1 << 4) & 0xf0f0f0f0u);
                        vhi[h][w] = ((x0 >> 4) & 0x0f0f0f0fu) | (x1 & 0xf0f0f0f0u);
                    }
            }
            uint32_t f[4][4];  // FP4: the converted pairs of one word of vlo / vhi
#pragma unroll
            for (int j = 0; j < kDBlocks; ++j) {
                uint32_t a[4];
                if constexpr (kFp4) {
                    const int w = j >> 2, b = j & 3;
                    if (b == 0) {
                        e2m1x8_to_f16x2x4(vlo[0][w], f[0]);
                        e2m1x8_to_f16x2x4(vhi[0][w], f[1]);
                        e2m1x8_to_f16x2x4(vlo[1][w], f[2]);
                        e2m1x8_to_f16x2x4(vhi[1][w], f[3]);
                    }
                    a[0] = f[0][b];
                    a[1] = f[1][b];
                    a[2] = f[2][b];
                    a[3] = f[3][b];
                } else {
                    const uint32_t sel = (j & 1) ? 0x7362u : 0x5140u;  // bytes 2j%4, 2j%4+1 of two rows
                    uint32_t x[2], y[2];
                    e4m3x4_to_f16x2x2(byte_perm(vw[n][0][j >> 1], vw[n][1][j >> 1], sel), x);
                    e4m3x4_to_f16x2x2(byte_perm(vw[n][2][j >> 1], vw[n][3][j >> 1], sel), y);
                    a[0] = x[0];
                    a[1] = x[1];
                    a[2] = y[0];
                    a[3] = y[1];
                }
                mma_f16(acc[j], a, bh0[n], bh1[n]);
            }
        }
    }

    __device__ __forceinline__ bool tile(unsigned char* kbuf, unsigned char* vbuf, uint64_t bits,
                                         int warp, int lane, float qscale) {
#pragma unroll
        for (int sl = 0; sl < kSlabsPerWarp; ++sl) {
            const int slab0 = (warp * kSlabsPerWarp + sl) * 16;
            const uint32_t vmask = (uint32_t)(bits >> slab0) & 0xffffu;
            if (vmask == 0u) continue;
            const unsigned char* kb = kbuf + slab0 * kRowBytes;
            const unsigned char* vb = vbuf + slab0 * kRowBytes;
            slabs<1>(&kb, &vb, &vmask, lane, qscale);
        }
        return false;  // the ring is only read
    }

    __device__ __forceinline__ void finish(float* mo, float* ml, int warp, int lane) {
        const int gid = lane >> 2, tig = lane & 3;
#pragma unroll
        for (int off = 4; off < 32; off <<= 1) {
            l[0] += __shfl_xor_sync(0xffffffffu, l[0], off);
            l[1] += __shfl_xor_sync(0xffffffffu, l[1], off);
        }
        const float vs = pow2i(ve - 127);
#pragma unroll
        for (int c = 0; c < 2; ++c) {
            const int hh = 2 * tig + c;
            if (hh < G) {
#pragma unroll
                for (int j = 0; j < kDBlocks; ++j) {
                    const int d = (D / 8) * gid + 2 * j;
                    mo[(warp * G + hh) * D + d] = acc[j][c] * vs;
                    mo[(warp * G + hh) * D + d + 1] = acc[j][2 + c] * vs;
                }
                if (gid == 0) {
                    ml[(warp * G + hh) * 2] = m[c];
                    ml[(warp * G + hh) * 2 + 1] = l[c];
                }
            }
        }
    }
};

template <int D, int G, int T, int NCW>
using Fp8MmaConsumer = QuantMmaConsumer<D, G, T, NCW, false>;
template <int D, int G, int T, int NCW>
using Fp4MmaConsumer = QuantMmaConsumer<D, G, T, NCW, true>;

}  // namespace kvd
