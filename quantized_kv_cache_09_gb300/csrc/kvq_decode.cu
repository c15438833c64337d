// kvq_decode.cu -- single-token decode attention over the quantized paged KV
// cache (decode reading a quantized KV cache: aicoding.csdn.net section 3.1;
// paging through a block table: ddd.cn section 4).
//
// Decode is a GEMV per (sequence, head): every cached byte is read once and
// used for a handful of flops, so the kernel is built around HBM streaming.
// Codes are widened exactly to fp16 in registers -- int4 to fp16 subnormals
// (one lop3 per pair, the offset taken out after the contraction), int8 and
// FP8 E4M3 to fp16 pairs -- and both contractions run on the legacy
// tensor-core mma (m16n8k16): the widening, not the multiply, is the cost.
//
// Work decomposition (persistent, split-K over the sequence):
//   unit   = 32 tokens (int4) or 16 tokens (int8) of one (sequence, head):
//            2 KiB of K codes + 2 KiB of V codes, contiguous inside one page;
//   order  = sequence-major, then head, then unit;
//   warps  = a persistent grid of one CTA of 12 warps per SM; warp g owns
//            the contiguous unit range [U g / GW, U (g+1) / GW) (GW warps
//            have work),
//            so every warp streams the same number of bytes whatever the
//            length mix;
//   stream = each warp runs its own ring of 2 shared-memory stages of 2
//            units (int4: a whole page; int8: half a page) filled by bulk
//            async copies (cp.async.bulk, completing on one mbarrier per
//            stage); lane 0 refills a stage as soon as it is consumed;
//   math   = s = scale_k * (q . c) * softmax_scale, online softmax in fp32
//            (base 2), acc += p * scale_v * c with fp32 accumulation;
//   split  = a (sequence, head) wholly inside one warp's range is written as
//            the final output; one cut by range boundaries leaves an (m, l, acc)
//            partial per piece, and the warp that writes the last piece
//            combines them in the same launch:
//            m = max m_i, l = sum l_i 2^(m_i - m), o = sum acc_i 2^(m_i - m) / l.
//            "Last" is decided by an atomic count per (sequence, head) that the
//            last piece puts back to zero, so nothing waits and the workspace
//            stays ready for the next launch.
#include <atomic>

#include "kvq_device.cuh"
#include "kvq_internal.h"

namespace kvq {

constexpr int kUnitBytes = 2048;
constexpr int kMinUnitsPerWarp = 2;

template <int FMT>
struct DecFmt;
// A stage holds up to kUnitsPerStage consecutive units of one page (one bulk
// copy each for K and V): two 32-token units = a whole page for int4, two
// 16-token units = half a page for int8; two stages per warp.  One CTA per SM holds all the warps:
// the warp scheduler favours older CTAs, so with several CTAs per SM the
// warps of the youngest ran ~16% slower than those of the oldest and the SM
// waited for them; the warps of one CTA progress at the same rate.
template <>
struct DecFmt<KVQ_INT4_B64> {
    static constexpr int kRowBytes = 64;
    static constexpr int kUnitTok = 32;
    static constexpr int kUnitsPerPage = 2;
    static constexpr int kUnitsPerStage = 2;
    static constexpr int kStages = 2;
    static constexpr int kWarps = 12;
    static constexpr int kCtasPerSm = 1;
    static constexpr int kMergeBatch = 8;  // pieces whose loads a merge issues at once
};
template <>
struct DecFmt<KVQ_INT8_PAGE> {
    static constexpr int kRowBytes = 128;
    static constexpr int kUnitTok = 16;
    static constexpr int kUnitsPerPage = 4;
    static constexpr int kUnitsPerStage = 2;
    static constexpr int kStages = 2;
    static constexpr int kWarps = 12;
    static constexpr int kCtasPerSm = 1;
    static constexpr int kMergeBatch = 4;
};
// FP8 E4M3: one byte per element like int8, so the same units, stages and grid
template <>
struct DecFmt<KVQ_FP8_E4M3> : DecFmt<KVQ_INT8_PAGE> {
};

// what a stage holds: units c .. c + nunits - 1 of (b, h), ntok tokens in all;
// new_seg: the first chunk of a segment (the warp's first, or a new (sequence, head))
struct alignas(16) StageMeta {
    int32_t b, h, c, ntok;
    float sk, sv;
    int32_t new_seg, nunits;
};

template <int kStages, int kStageBytes, int kQRows>
struct alignas(128) WarpSmem {
    uint8_t k[kStages][kStageBytes];
    uint8_t v[kStages][kStageBytes];
    uint16_t q[kStages][kQRows * kHeadDim];  // the query rows of the stage's cache head
    StageMeta meta[kStages];
    uint64_t full[kStages];
};

constexpr size_t kSeqSmemBytes = ((2 * kMaxSeqsPerLaunch + 1) * sizeof(int32_t) + 64 + 127) / 128 * 128;
// the group value of the tile consumer (16 query heads per tile, any group size)
constexpr int kMqG = 16;
constexpr int kMqRows = 16;
// warps of a decode CTA: the tile consumer's stages carry 16 query rows, so
// fewer warps fit in shared memory (and each has more registers)
template <int FMT, int G>
struct DecShape {
    // G = 8: the stages carry no query rows (8 rows a stage would leave room for 11 warps
    // only: 12 need 247 KB); the consumer reads a segment's rows from global memory
    static constexpr bool kQGlobal = G == 8;
    static constexpr int kWarps = G == kMqG ? 8 : DecFmt<FMT>::kWarps;
    static constexpr int kQRows = G == kMqG ? kMqRows : kQGlobal ? 1 : G;  // (1: an unused placeholder)
};
template <int FMT, int G>
constexpr size_t dec_smem_bytes()
{
    using F = DecFmt<FMT>;
    using S = DecShape<FMT, G>;
    return S::kWarps * sizeof(WarpSmem<F::kStages, F::kUnitsPerStage * kUnitBytes, S::kQRows>) + kSeqSmemBytes;
}
static_assert(dec_smem_bytes<KVQ_INT4_B64, 8>() <= 227 * 1024 && dec_smem_bytes<KVQ_INT8_PAGE, 8>() <= 227 * 1024 &&
                  dec_smem_bytes<KVQ_FP8_E4M3, 8>() <= 227 * 1024 && dec_smem_bytes<KVQ_INT4_B64, 4>() <= 227 * 1024,
              "the warps fit one CTA's shared memory");

// the byte formats' exact widening to fp16 pairs, by format (int4: SubMagic below)
template <int FMT>
__device__ __forceinline__ void widen_bytes(uint32_t w, __half2 c[2])
{
    if constexpr (FMT == KVQ_FP8_E4M3)
        widen_e4m3(w, c);
    else
        widen_int8(w, c);
}

__device__ __forceinline__ float warp_max(float v)
{
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v = fmaxf(v, __shfl_xor_sync(kFull, v, o));
    return v;
}

__device__ __forceinline__ float warp_sum(float v)
{
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(kFull, v, o);
    return v;
}

__device__ __forceinline__ int64_t imin64(int64_t a, int64_t b) { return a < b ? a : b; }

__device__ __forceinline__ int units_of(int len, int unit_tok) { return (len + unit_tok - 1) / unit_tok; }


// ---------------------------------------------------------------------------
// Per-format consumers: the math of one unit and the segment epilogue.
// ---------------------------------------------------------------------------
template <int FMT>
struct Consumer;


__device__ __forceinline__ uint32_t lop_and_xor(uint32_t x, uint32_t m, uint32_t c)
{
    uint32_t d;
    asm("lop3.b32 %0, %1, %2, %3, 0x6a;" : "=r"(d) : "r"(x), "r"(m), "r"(c));  // (x & m) ^ c
    return d;
}

// int4 codes widened exactly to fp16, one lop3 per pair.  With c the signed
// code of a nibble, flipping its bit 3 gives n = c + 8 and flipping bits
// 0..2 gives n = 7 - c; the nibble n in the low four bits of a 16-bit half,
// read as an fp16, is the subnormal n * 2^-24, and in bits 4..7 the subnormal
// n * 2^-20.  So each element reaches the mma as
//   even element (low nibble of its byte):  (c + 8) * 2^-24
//   odd element (bits 4..7):                (7 - c) * 2^-20
// exactly (the tensor cores take subnormal operands at full precision, and
// every product stays far above binary32's range limit).  The offsets and the
// powers of two come out after the contraction instead of per pair:
//   QK: q's odd elements are scaled by -1/16, so every product is
//       q_d c_d 2^-24 plus an offset share (+8 q_d even, -7 q_d odd); the
//       score is 2^24 raw - (8 sum_even q - 7 sum_odd q).  The two signs
//       make the shares of a smooth q cancel inside each mma, which keeps the
//       tensor core's running sums -- and their rounding -- small;
//   PV: output element d is 2^24 raw_d - 8 sum(x) (even d) or
//       7 sum(x) - 2^20 raw_d (odd d), x the weights that went into the
//       contraction.
// The masks and offsets are held in registers: a SASS lop3 takes at most one
// immediate, so (x & mask) ^ offset with both as literals costs two lop3 on the
// half-rate integer pipe; with both in registers it is one.  The empty asm
// makes the values opaque so they are not folded back into immediates.
struct SubMagic {
    uint32_t m_lo, m_hi, x_lo, x_hi;  // 0x000f000f, 0x00f000f0, 0x00080008, 0x00700070
    __device__ __forceinline__ void init()
    {
        m_lo = 0x000f000fu;
        m_hi = 0x00f000f0u;
        x_lo = 0x00080008u;
        x_hi = 0x00700070u;
        asm volatile("" : "+r"(m_lo), "+r"(m_hi), "+r"(x_lo), "+r"(x_hi));
    }
};
__device__ __forceinline__ uint32_t sub_lo(uint32_t x, const SubMagic &k) { return lop_and_xor(x, k.m_lo, k.x_lo); }
__device__ __forceinline__ uint32_t sub_hi(uint32_t x, const SubMagic &k) { return lop_and_xor(x, k.m_hi, k.x_hi); }
__device__ __forceinline__ uint32_t sub_pair(uint32_t x, bool odd, const SubMagic &k)
{
    return odd ? sub_hi(x, k) : sub_lo(x, k);
}
// element d of a contraction over widened codes = kUnit[d & 1] * raw - kOff[d & 1] * (sum of the other operand)
constexpr float kUnitEven = 16777216.0f;  // 2^24
constexpr float kUnitOdd = -1048576.0f;   // -2^20
constexpr float kOffEven = 8.0f;
constexpr float kOffOdd = -7.0f;
// q's odd elements as the mma takes them
constexpr float kQOdd = -0.0625f;
// the offset share of a score: 8 sum_even q - 7 sum_odd q, from the sums of
// q's even elements and of its scaled odd elements (q_d = -16 * scaled)
__device__ __forceinline__ float q_offset(float sum_even, float sum_odd_scaled)
{
    return fmaf(kOffOdd * -16.0f, sum_odd_scaled, kOffEven * sum_even);
}

// two softmax weights split into fp16 pairs hi = {RN16(x0), RN16(x1)} and
// lo = {RN16(x0 - hi0), RN16(x1 - hi1)}: hi + lo keeps ~22 significant bits
__device__ __forceinline__ void hi_lo_pairs(uint64_t x, uint32_t &hi, uint32_t &lo)
{
    float x0, x1;
    upk2(x, x0, x1);
    hi = f16x2_rn(x0, x1);
    const float2 h = __half22float2(*reinterpret_cast<const __half2 *>(&hi));
    float r0, r1;
    upk2(sub2(x, pk2(h.x, h.y)), r0, r1);
    lo = f16x2_rn(r0, r1);
}

// int4: both contractions of a unit on the tensor cores (mma.sync m16n8k16),
// codes widened exactly to fp16 subnormals in registers (SubMagic), fp32
// accumulation.
//   QK: A = 16 tokens x 16 head elements of K, every column of B = q, so every
//       lane receives the scores of its rows (tokens g, g+8 of each tile);
//       lane (g, t) feeds rows g, g+8 from its 16-byte slice (elements
//       32t..32t+31) of each token row, so the k index is a fixed permutation
//       of the head dimension that q's fragment repeats.
//   PV: A = V^T (16 head elements x 16 tokens): prmt pairs the same element of
//       two tokens; B column 0 = RN16(p), column 1 = the remainder, so p keeps
//       ~22 bits (columns 2..7 carry copies and are never read).
//   Unit = 32 tokens: 2 token tiles for QK, 2 k-tiles for PV, 8 output tiles.
// The three phases (qk, softmax, pv) are separate so the caller can overlap
// qk of the next unit with pv of this one.
template <>
struct Consumer<KVQ_INT4_B64> {
    static constexpr int kScores = 4;
    static constexpr int kPf = 4;
    int rows;  // (unused: one query row)
    uint32_t qb[8][2];  // q as the B operand, the odd elements scaled by kQOdd
    float acc[8][4];    // PV over the widened codes (SubMagic): raw sums
    float m_run;
    float qbias;  // minus the offset share of every score (q_offset)
    uint64_t l2;  // running sum of the weights in this lane's slots, as a pair
    uint64_t x2;  // running sum of x = p * scale_v in this lane's slots, as a pair
    SubMagic mk;

    __device__ __forceinline__ void reset()
    {
        mk.init();
        m_run = -INFINITY;
        l2 = pk2(0.0f, 0.0f);
        x2 = pk2(0.0f, 0.0f);
#pragma unroll
        for (int i = 0; i < 8; i++)
#pragma unroll
            for (int j = 0; j < 4; j++) acc[i][j] = 0.0f;
    }

    __device__ __forceinline__ void load_q(const uint16_t *qs, int lane)
    {
        const int t = lane & 3;
        const uint4 *q4 = reinterpret_cast<const uint4 *>(qs + 32 * t);
        const __half2 odd_scale = __float2half2_rn(kQOdd);
        float se = 0.0f, so = 0.0f;  // sums of the even elements and of the scaled odd ones
#pragma unroll
        for (int m = 0; m < 4; m++) {
            const uint4 v = q4[m];  // elements 32t + 8m .. +7 as pairs (0,1) (2,3) (4,5) (6,7)
            const uint32_t e04 = __byte_perm(v.x, v.z, 0x5410), e15 = __byte_perm(v.x, v.z, 0x7632);
            const uint32_t e26 = __byte_perm(v.y, v.w, 0x5410), e37 = __byte_perm(v.y, v.w, 0x7632);
            const __half2 o15 = __hmul2(*reinterpret_cast<const __half2 *>(&e15), odd_scale);
            const __half2 o37 = __hmul2(*reinterpret_cast<const __half2 *>(&e37), odd_scale);
            qb[2 * m][0] = e04;               // {e0, e4}
            qb[2 * m][1] = h2_bits(o15);      // {e1, e5} * kQOdd
            qb[2 * m + 1][0] = e26;           // {e2, e6}
            qb[2 * m + 1][1] = h2_bits(o37);  // {e3, e7} * kQOdd
            // the sums in binary32 (the offset share is scaled by each page's K scale, so an
            // error in it does not cancel in the softmax)
            const float2 a = __half22float2(*reinterpret_cast<const __half2 *>(&e04));
            const float2 c = __half22float2(*reinterpret_cast<const __half2 *>(&e26));
            const float2 o = __half22float2(o15), u = __half22float2(o37);
            se += (a.x + a.y) + (c.x + c.y);
            so += (o.x + o.y) + (u.x + u.y);
        }
        float qo = q_offset(se, so);
        qo += __shfl_xor_sync(kFull, qo, 1);  // the four lanes t of a row hold the four slices
        qo += __shfl_xor_sync(kFull, qo, 2);
        qbias = -qo;
    }

    // raw dot products (2^-24 (q . c + q_offset)) of tokens g, g+8, 16+g, 24+g
    // (every lane); four accumulator chains per tile keep the mma dependency
    // chains short
    __device__ __forceinline__ void qk(const uint8_t *ks, int lane, float sc[4]) const
    {
        const int g = lane >> 2, t = lane & 3;
#pragma unroll
        for (int tau = 0; tau < 2; tau++) {
            float c[4][4];
#pragma unroll
            for (int m = 0; m < 4; m++)
#pragma unroll
                for (int e = 0; e < 4; e++) c[m][e] = 0.0f;
            const uint4 wa = *reinterpret_cast<const uint4 *>(ks + (16 * tau + g) * 64 + 16 * t);
            const uint4 wb = *reinterpret_cast<const uint4 *>(ks + (16 * tau + g + 8) * 64 + 16 * t);
            const uint32_t ua[4] = {wa.x, wa.y, wa.z, wa.w};
            const uint32_t ub[4] = {wb.x, wb.y, wb.z, wb.w};
#pragma unroll
            for (int m = 0; m < 4; m++) {
                // {c0,c4}, {c1,c5}, {c2,c6}, {c3,c7} of each token row
                const uint32_t ah = ua[m] >> 8, bh = ub[m] >> 8;
                mma16816(c[m], sub_lo(ua[m], mk), sub_lo(ub[m], mk), sub_hi(ua[m], mk), sub_hi(ub[m], mk),
                         qb[2 * m][0], qb[2 * m][1]);
                mma16816(c[m], sub_lo(ah, mk), sub_lo(bh, mk), sub_hi(ah, mk), sub_hi(bh, mk), qb[2 * m + 1][0],
                         qb[2 * m + 1][1]);
            }
            sc[2 * tau] = (c[0][0] + c[1][0]) + (c[2][0] + c[3][0]);
            sc[2 * tau + 1] = (c[0][2] + c[1][2]) + (c[2][2] + c[3][2]);
        }
    }

    // online softmax over the unit's scores.  px[k] = the fp16 pair of this
    // lane's two tokens of tile k (16k + g, 16k + 8 + g) of x = p * sv: the
    // rounded values in lanes t == 0, the remainders elsewhere (pv takes
    // column 0 of its weights from t == 0 lanes and column 1 from t == 1).
    __device__ __forceinline__ void softmax(const float sc[4], int ntok, float fac, float sv, int lane,
                                            uint32_t px[2])
    {
        const int g = lane >> 2, t = lane & 3;
        const uint64_t ff = pk2(fac * kUnitEven, fac * kUnitEven), fb = pk2(qbias * fac, qbias * fac);
        float s2[4];
        upk2(fma2(pk2(sc[0], sc[1]), ff, fb), s2[0], s2[1]);
        upk2(fma2(pk2(sc[2], sc[3]), ff, fb), s2[2], s2[3]);
        if (ntok < 32) {  // the last unit of a sequence: tokens past its end get no weight
#pragma unroll
            for (int i = 0; i < 4; i++)
                if (16 * (i >> 1) + 8 * (i & 1) + g >= ntok) s2[i] = -INFINITY;
        }
        const float lm = fmaxf(fmaxf(s2[0], s2[1]), fmaxf(s2[2], s2[3]));
        if (__any_sync(kFull, lm > m_run)) {  // the running maximum moves: rescale
            const float mu = warp_max(lm);
            const float alpha = ex2_approx(m_run - mu);
            l2 = mul2(l2, pk2(alpha, alpha));
            x2 = mul2(x2, pk2(alpha, alpha));
#pragma unroll
            for (int i = 0; i < 8; i++)
#pragma unroll
                for (int j = 0; j < 4; j++) acc[i][j] *= alpha;
            m_run = mu;
        }
        float pe[4];
#pragma unroll
        for (int i = 0; i < 4; i++) pe[i] = ex2_approx(s2[i] - m_run);
        const uint64_t p01 = pk2(pe[0], pe[1]), p23 = pk2(pe[2], pe[3]);
        const uint64_t psum = add2(p01, p23);
        const uint64_t vv = pk2(sv, sv);
        l2 = add2(l2, psum);
        x2 = fma2(psum, vv, x2);
        uint32_t hi, lo;
        hi_lo_pairs(mul2(p01, vv), hi, lo);
        px[0] = t == 0 ? hi : lo;
        hi_lo_pairs(mul2(p23, vv), hi, lo);
        px[1] = t == 0 ? hi : lo;
    }

    __device__ __forceinline__ void pv(const uint8_t *vs, const uint32_t px[2], int lane)
    {
        const int g = lane >> 2, t = lane & 3;
        // column g of B: lanes g == 0 read the rounded weights (from a t == 0
        // lane), g == 1 the remainders (from a t == 1 lane); others any copy
        const int src = 8 * t + (g & 3);
#pragma unroll
        for (int kap = 0; kap < 2; kap++) {
            const uint32_t ua = __shfl_sync(kFull, px[kap], src);      // tokens 2t, 2t+8 of tile kap
            const uint32_t ub = __shfl_sync(kFull, px[kap], src + 4);  // tokens 2t+1, 2t+9
            const uint32_t b0 = __byte_perm(ua, ub, 0x5410);
            const uint32_t b1 = __byte_perm(ua, ub, 0x7632);
#pragma unroll
            for (int R = 0; R < 2; R++) {
                // word 8R + g (elements 64R + 8g .. +7) of tokens 16kap + 2t, +1, +8, +9
                const uint8_t *vb = vs + (16 * kap + 2 * t) * 64 + 4 * (8 * R + g);
                const uint32_t wa = *reinterpret_cast<const uint32_t *>(vb);
                const uint32_t wb = *reinterpret_cast<const uint32_t *>(vb + 64);
                const uint32_t wc = *reinterpret_cast<const uint32_t *>(vb + 8 * 64);
                const uint32_t wd = *reinterpret_cast<const uint32_t *>(vb + 9 * 64);
                uint32_t xab[4], xcd[4];
#pragma unroll
                for (int k = 0; k < 4; k++) {
                    // selector nibbles: result bytes = [wa.k, wa.k, wb.k, wb.k]
                    const uint32_t bsel = (uint32_t)k | ((uint32_t)k << 4) | ((uint32_t)(4 + k) << 8) |
                                          ((uint32_t)(4 + k) << 12);
                    xab[k] = __byte_perm(wa, wb, bsel);
                    xcd[k] = __byte_perm(wc, wd, bsel);
                }
#pragma unroll
                for (int jj = 0; jj < 4; jj++) {
                    const bool odd = jj & 1;
                    mma16816(acc[4 * R + jj], sub_pair(xab[jj >> 1], odd, mk), sub_pair(xab[2 + (jj >> 1)], odd, mk),
                             sub_pair(xcd[jj >> 1], odd, mk), sub_pair(xcd[2 + (jj >> 1)], odd, mk), b0, b1);
                }
            }
        }
    }

    // out row (final) or partial slot: lanes with t == 0 hold elements
    // 64R + 8g + e (e < 4: tile 4R+e rows g; e >= 4: tile 4R+e-4 rows g+8);
    // (odd elements from bits 4..7, even ones from bits 0..3: SubMagic)
    __device__ __forceinline__ void finish(int lane, uint16_t *orow, float *part)
    {
        float la, lb, xa, xb;
        upk2(l2, la, lb);
        upk2(x2, xa, xb);
        const float l = warp_sum(la + lb) * 0.25f;  // the four lanes of a row group hold the same weights
        const float xs = warp_sum(xa + xb) * 0.25f;
        const float xb_even = -kOffEven * xs, xb_odd = -kOffOdd * xs;
        const int g = lane >> 2, t = lane & 3;
        if (t != 0) return;
#pragma unroll
        for (int R = 0; R < 2; R++) {
            float v[8];
#pragma unroll
            for (int e = 0; e < 4; e++) {
                const float f = (e & 1) ? kUnitOdd : kUnitEven, xb = (e & 1) ? xb_odd : xb_even;
                v[e] = fmaf(acc[4 * R + e][0] + acc[4 * R + e][1], f, xb);
                v[4 + e] = fmaf(acc[4 * R + e][2] + acc[4 * R + e][3], f, xb);
            }
            if (orow) {
                const float inv = 1.0f / l;
                uint4 o;
                o.x = h2_bits(__floats2half2_rn(v[0] * inv, v[1] * inv));
                o.y = h2_bits(__floats2half2_rn(v[2] * inv, v[3] * inv));
                o.z = h2_bits(__floats2half2_rn(v[4] * inv, v[5] * inv));
                o.w = h2_bits(__floats2half2_rn(v[6] * inv, v[7] * inv));
                *reinterpret_cast<uint4 *>(orow + 64 * R + 8 * g) = o;
            } else {
                float4 *d4 = reinterpret_cast<float4 *>(part + 4 + 64 * R + 8 * g);
                d4[0] = make_float4(v[0], v[1], v[2], v[3]);
                d4[1] = make_float4(v[4], v[5], v[6], v[7]);
            }
        }
        if (part && lane == 0) {
            part[0] = m_run;
            part[1] = l;
        }
    }
};

// int4 with grouped query heads: G = 2, 4 or 8 query heads share each cache
// head, and one pass over the codes serves all G (the mma columns that the
// multi-head consumer fills with copies of q carry the group's other heads).
// Lane (grp = lane >> 2, t = lane & 3):
//   QK: column c of B holds q of head hq(c) = (((c >> 2) << 1) | (c & 1)) % G
//       for G = 2, 4 and hq(c) = c for G = 8, so the lane receives, for tokens
//       grp and grp + 8 of each tile, the scores of its head slots c = 0, 1:
//       the heads of columns 2t + c.
//   PV, G = 2, 4: column c of B holds part (c >> 1) & 1 (0: RN16(x), 1: the
//       remainder) of head hq(c); the lane's accumulators are then exactly its
//       slot heads, part t & 1, so a rescale of a head's running max is local.
//   PV, G = 8: the eight columns are the eight heads and carry RN16(x) alone
//       (no remainder column is left; the tile kernel's weights are single
//       fp16 values too), so a weight keeps 11 bits: the error of the output
//       is at most 2^-11 of max|v^| from the weights (one dominant key) plus
//       the fp16 rounding of the output.  The offset share of PV is taken out
//       with the sum of the rounded weights the MMA multiplied, not of x.
//       The lane's accumulators are its slot heads.
//   The weights of column grp_d come from lane 4 * token + (grp_d >> 1),
//   slot grp_d & 1 (that lane holds head hq(grp_d) and produces part
//   (grp_d >> 1) & 1; for G = 8, RN16(x)).
template <int G>
struct ConsumerGqa {
    static_assert(G == 2 || G == 4 || G == 8, "query heads per cache head");
    static constexpr bool kAllHeads = G == 8;  // every B column a head of its own
    static constexpr int kScores = 8;
    static constexpr int kPf = 4;
    int rows;  // the group's g <= G query heads: columns of heads past it carry zero queries
    uint32_t qb[8][2];  // q of head hq(grp) as the B operand, the odd elements scaled by kQOdd
    float acc[8][4];    // PV over the widened codes (SubMagic): raw sums
    float m_run[2];
    float l_lane[2];
    float x_lane[2];    // this lane's part of sum(x), x = p * scale_v, per head slot
    float qbias[2];     // minus the offset share of the scores of the lane's two slot heads
    SubMagic mk;

    __device__ __forceinline__ void reset()
    {
        mk.init();
        m_run[0] = m_run[1] = -INFINITY;
        l_lane[0] = l_lane[1] = 0.0f;
        x_lane[0] = x_lane[1] = 0.0f;
#pragma unroll
        for (int i = 0; i < 8; i++)
#pragma unroll
            for (int j = 0; j < 4; j++) acc[i][j] = 0.0f;
    }

    // qs: the group's query rows (fp16 [g][128]: a stage's buffer, or global memory for G = 8)
    __device__ __forceinline__ void load_q(const uint16_t *qs, int lane)
    {
        const int g = lane >> 2, t = lane & 3;
        const int head = kAllHeads ? g : (((g >> 2) << 1) | (g & 1)) % G;  // column g of B
        const bool live = head < rows;  // rows 0 .. rows - 1 exist; a head past them reads nothing
        const uint4 *q4 = reinterpret_cast<const uint4 *>(qs + head * kHeadDim + 32 * t);
        const __half2 odd_scale = __float2half2_rn(kQOdd);
        float se = 0.0f, so = 0.0f;
#pragma unroll
        for (int m = 0; m < 4; m++) {
            const uint4 v = live ? q4[m] : make_uint4(0u, 0u, 0u, 0u);
            const uint32_t e04 = __byte_perm(v.x, v.z, 0x5410), e15 = __byte_perm(v.x, v.z, 0x7632);
            const uint32_t e26 = __byte_perm(v.y, v.w, 0x5410), e37 = __byte_perm(v.y, v.w, 0x7632);
            const __half2 o15 = __hmul2(*reinterpret_cast<const __half2 *>(&e15), odd_scale);
            const __half2 o37 = __hmul2(*reinterpret_cast<const __half2 *>(&e37), odd_scale);
            qb[2 * m][0] = e04;
            qb[2 * m][1] = h2_bits(o15);
            qb[2 * m + 1][0] = e26;
            qb[2 * m + 1][1] = h2_bits(o37);
            // the sums in binary32 (the offset share is scaled by each page's K scale, so an
            // error in it does not cancel in the softmax)
            const float2 a = __half22float2(*reinterpret_cast<const __half2 *>(&e04));
            const float2 c = __half22float2(*reinterpret_cast<const __half2 *>(&e26));
            const float2 o = __half22float2(o15), u = __half22float2(o37);
            se += (a.x + a.y) + (c.x + c.y);
            so += (o.x + o.y) + (u.x + u.y);
        }
        float qo = q_offset(se, so);
        qo += __shfl_xor_sync(kFull, qo, 1);  // the offset share of head hq(grp) in every lane of grp
        qo += __shfl_xor_sync(kFull, qo, 2);
        // the lane's score slots c are columns 2t + c of B, held by the lanes grp = 2t + c
#pragma unroll
        for (int c = 0; c < 2; c++) qbias[c] = -__shfl_sync(kFull, qo, 4 * (2 * t + c));
    }

    // raw dot products (2^-24 (q . c + q_offset)): sc[4 tau + 2 r + c] = token
    // 16 tau + grp + 8 r, head slot c
    __device__ __forceinline__ void qk(const uint8_t *ks, int lane, float sc[8]) const
    {
        const int g = lane >> 2, t = lane & 3;
#pragma unroll
        for (int tau = 0; tau < 2; tau++) {
            float c[4][4];
#pragma unroll
            for (int m = 0; m < 4; m++)
#pragma unroll
                for (int e = 0; e < 4; e++) c[m][e] = 0.0f;
            const uint4 wa = *reinterpret_cast<const uint4 *>(ks + (16 * tau + g) * 64 + 16 * t);
            const uint4 wb = *reinterpret_cast<const uint4 *>(ks + (16 * tau + g + 8) * 64 + 16 * t);
            const uint32_t ua[4] = {wa.x, wa.y, wa.z, wa.w};
            const uint32_t ub[4] = {wb.x, wb.y, wb.z, wb.w};
#pragma unroll
            for (int m = 0; m < 4; m++) {
                const uint32_t ah = ua[m] >> 8, bh = ub[m] >> 8;
                mma16816(c[m], sub_lo(ua[m], mk), sub_lo(ub[m], mk), sub_hi(ua[m], mk), sub_hi(ub[m], mk),
                         qb[2 * m][0], qb[2 * m][1]);
                mma16816(c[m], sub_lo(ah, mk), sub_lo(bh, mk), sub_hi(ah, mk), sub_hi(bh, mk), qb[2 * m + 1][0],
                         qb[2 * m + 1][1]);
            }
#pragma unroll
            for (int e = 0; e < 4; e++) sc[4 * tau + e] = (c[0][e] + c[1][e]) + (c[2][e] + c[3][e]);
        }
    }

    // online softmax over the unit, per head slot.  px[2 tau + c] = this
    // lane's part (t & 1) of x = p * sv for tokens (grp, grp + 8) of tile tau,
    // head slot c, as an fp16 pair (G = 8: RN16(x))
    __device__ __forceinline__ void softmax(const float sc[8], int ntok, float fac, float sv, int lane,
                                            uint32_t px[4])
    {
        const int g = lane >> 2, t = lane & 3;
        const uint64_t ff = pk2(fac * kUnitEven, fac * kUnitEven), fb = pk2(qbias[0] * fac, qbias[1] * fac);
        float s2[8];
#pragma unroll
        for (int i = 0; i < 8; i += 2) upk2(fma2(pk2(sc[i], sc[i + 1]), ff, fb), s2[i], s2[i + 1]);
        if (ntok < 32) {  // the last unit of a sequence: tokens past its end get no weight
#pragma unroll
            for (int i = 0; i < 8; i++)
                if (16 * (i >> 2) + 8 * ((i >> 1) & 1) + g >= ntok) s2[i] = -INFINITY;
        }
        float lm[2];
#pragma unroll
        for (int c = 0; c < 2; c++) lm[c] = fmaxf(fmaxf(s2[c], s2[2 + c]), fmaxf(s2[4 + c], s2[6 + c]));
        if (__any_sync(kFull, lm[0] > m_run[0] || lm[1] > m_run[1])) {  // a running maximum moves: rescale
#pragma unroll
            for (int c = 0; c < 2; c++) {
                float mu = lm[c];  // max over the 8 lanes of this t (the tokens of the unit)
                mu = fmaxf(mu, __shfl_xor_sync(kFull, mu, 4));
                mu = fmaxf(mu, __shfl_xor_sync(kFull, mu, 8));
                mu = fmaxf(mu, __shfl_xor_sync(kFull, mu, 16));
                mu = fmaxf(mu, m_run[c]);
                const float alpha = ex2_approx(m_run[c] - mu);
                l_lane[c] *= alpha;
                x_lane[c] *= alpha;
#pragma unroll
                for (int i = 0; i < 8; i++) {
                    acc[i][c] *= alpha;
                    acc[i][2 + c] *= alpha;
                }
                m_run[c] = mu;
            }
        }
        float pe[8];
#pragma unroll
        for (int i = 0; i < 8; i++) pe[i] = ex2_approx(s2[i] - m_run[i & 1]);
        const float ps0 = (pe[0] + pe[2]) + (pe[4] + pe[6]), ps1 = (pe[1] + pe[3]) + (pe[5] + pe[7]);
        l_lane[0] += ps0;
        l_lane[1] += ps1;
        const uint64_t vv = pk2(sv, sv);
        if constexpr (kAllHeads) {
            // RN16(x) alone, and the sum of exactly those weights for the offset share
#pragma unroll
            for (int c = 0; c < 2; c++) {
                float xr = 0.0f;
#pragma unroll
                for (int tau = 0; tau < 2; tau++) {
                    float x0, x1;
                    upk2(mul2(pk2(pe[4 * tau + c], pe[4 * tau + 2 + c]), vv), x0, x1);
                    const uint32_t h = f16x2_rn(x0, x1);
                    const float2 r = __half22float2(*reinterpret_cast<const __half2 *>(&h));
                    xr += r.x + r.y;
                    px[2 * tau + c] = h;
                }
                x_lane[c] += xr;
            }
        } else {
            x_lane[0] = fmaf(ps0, sv, x_lane[0]);
            x_lane[1] = fmaf(ps1, sv, x_lane[1]);
            const bool lo_part = t & 1;
#pragma unroll
            for (int tau = 0; tau < 2; tau++)
#pragma unroll
                for (int c = 0; c < 2; c++) {
                    uint32_t hi, lo;
                    hi_lo_pairs(mul2(pk2(pe[4 * tau + c], pe[4 * tau + 2 + c]), vv), hi, lo);
                    px[2 * tau + c] = lo_part ? lo : hi;
                }
        }
    }

    __device__ __forceinline__ void pv(const uint8_t *vs, const uint32_t px[kPf], int lane)
    {
        const int g = lane >> 2, t = lane & 3;
        // column g of B: head slot g & 1, part (g >> 1) & 1 (G = 8: RN16(x)), from lanes 4 token + (g >> 1)
        const int src = 8 * t + (g >> 1);
        const bool slot1 = g & 1;
#pragma unroll
        for (int kap = 0; kap < 2; kap++) {
            const uint32_t a0 = __shfl_sync(kFull, px[2 * kap], src);          // tokens 2t, 2t+8
            const uint32_t a1 = __shfl_sync(kFull, px[2 * kap + 1], src);
            const uint32_t c0 = __shfl_sync(kFull, px[2 * kap], src + 4);      // tokens 2t+1, 2t+9
            const uint32_t c1 = __shfl_sync(kFull, px[2 * kap + 1], src + 4);
            const uint32_t ua = slot1 ? a1 : a0;
            const uint32_t ub = slot1 ? c1 : c0;
            const uint32_t b0 = __byte_perm(ua, ub, 0x5410);
            const uint32_t b1 = __byte_perm(ua, ub, 0x7632);
#pragma unroll
            for (int R = 0; R < 2; R++) {
                // word 8R + g (elements 64R + 8g .. +7) of tokens 16kap + 2t, +1, +8, +9
                const uint8_t *vb = vs + (16 * kap + 2 * t) * 64 + 4 * (8 * R + g);
                const uint32_t wa = *reinterpret_cast<const uint32_t *>(vb);
                const uint32_t wb = *reinterpret_cast<const uint32_t *>(vb + 64);
                const uint32_t wc = *reinterpret_cast<const uint32_t *>(vb + 8 * 64);
                const uint32_t wd = *reinterpret_cast<const uint32_t *>(vb + 9 * 64);
                uint32_t xab[4], xcd[4];
#pragma unroll
                for (int k = 0; k < 4; k++) {
                    // selector nibbles: result bytes = [wa.k, wa.k, wb.k, wb.k]
                    const uint32_t bsel = (uint32_t)k | ((uint32_t)k << 4) | ((uint32_t)(4 + k) << 8) |
                                          ((uint32_t)(4 + k) << 12);
                    xab[k] = __byte_perm(wa, wb, bsel);
                    xcd[k] = __byte_perm(wc, wd, bsel);
                }
#pragma unroll
                for (int jj = 0; jj < 4; jj++) {
                    const bool odd = jj & 1;
                    mma16816(acc[4 * R + jj], sub_pair(xab[jj >> 1], odd, mk), sub_pair(xab[2 + (jj >> 1)], odd, mk),
                             sub_pair(xcd[jj >> 1], odd, mk), sub_pair(xcd[2 + (jj >> 1)], odd, mk), b0, b1);
                }
            }
        }
    }


    // the group's output rows (orow: its `rows` rows) or partial slots (part:
    // G partials of kPartialStride floats).  G = 2, 4: the two parts of a head are
    // in lanes t and t ^ 1; lanes with even t, t >> 1 < G / 2, write heads
    // 2 (t >> 1) + c.  G = 8: every lane writes its heads 2t + c.
    __device__ __forceinline__ void finish(int lane, uint16_t *orow, float *part)
    {
        const int g = lane >> 2, t = lane & 3;
        float l[2], xs[2];
#pragma unroll
        for (int c = 0; c < 2; c++) {
            float v = l_lane[c], x = x_lane[c];
            v += __shfl_xor_sync(kFull, v, 4);
            v += __shfl_xor_sync(kFull, v, 8);
            v += __shfl_xor_sync(kFull, v, 16);
            x += __shfl_xor_sync(kFull, x, 4);
            x += __shfl_xor_sync(kFull, x, 8);
            x += __shfl_xor_sync(kFull, x, 16);
            l[c] = v;
            xs[c] = x;
        }
        if constexpr (!kAllHeads) {
#pragma unroll
            for (int i = 0; i < 8; i++)
#pragma unroll
                for (int j = 0; j < 4; j++) acc[i][j] += __shfl_xor_sync(kFull, acc[i][j], 1);
            if ((t & 1) || 2 * (t >> 1) >= G) return;
        }
#pragma unroll
        for (int c = 0; c < 2; c++) {
            const int head = kAllHeads ? 2 * t + c : 2 * (t >> 1) + c;
            if (orow && head >= rows) continue;  // a column past the group (its partial slot is written)
#pragma unroll
            for (int R = 0; R < 2; R++) {
                float v[8];
#pragma unroll
                for (int e = 0; e < 4; e++) {  // elements 64R + 8g + e, + 4: odd ones from bits 4..7
                    const float f = (e & 1) ? kUnitOdd : kUnitEven;
                    const float xb = -((e & 1) ? kOffOdd : kOffEven) * xs[c];
                    v[e] = fmaf(acc[4 * R + e][c], f, xb);
                    v[4 + e] = fmaf(acc[4 * R + e][2 + c], f, xb);
                }
                if (orow) {
                    const float inv = 1.0f / l[c];
                    uint4 o;
                    o.x = h2_bits(__floats2half2_rn(v[0] * inv, v[1] * inv));
                    o.y = h2_bits(__floats2half2_rn(v[2] * inv, v[3] * inv));
                    o.z = h2_bits(__floats2half2_rn(v[4] * inv, v[5] * inv));
                    o.w = h2_bits(__floats2half2_rn(v[6] * inv, v[7] * inv));
                    *reinterpret_cast<uint4 *>(orow + head * kHeadDim + 64 * R + 8 * g) = o;
                } else {
                    float4 *d4 = reinterpret_cast<float4 *>(part + head * kPartialStride + 4 + 64 * R + 8 * g);
                    d4[0] = make_float4(v[0], v[1], v[2], v[3]);
                    d4[1] = make_float4(v[4], v[5], v[6], v[7]);
                }
            }
            if (part && g == 0) {
                part[head * kPartialStride] = m_run[c];
                part[head * kPartialStride + 1] = l[c];
            }
        }
    }
};
// int8 and FP8 E4M3 (one byte per element), one query head per cache head:
// both contractions of a 16-token unit on the tensor cores (mma.sync m16n8k16),
// the codes widened exactly to fp16 pairs (FP8: one cvt.rn.f16x2.e4m3x2 per
// pair; int8: the 1024 + (byte ^ 0x80) - 1152 bias, a prmt and an hsub2 per
// pair), fp32 accumulation.
//   QK: A = 16 tokens x 16 elements; lane (g, t) feeds rows g, g + 8 from its
//       32-byte slice (elements 32t .. 32t+31) of each token row: k-step m
//       takes elements 32t + 4m + {0,1} as k rows 2t, 2t+1 and + {2,3} as
//       2t+8, 2t+9, a fixed permutation of the head dimension that q's
//       fragment repeats; q fills every column of B, so every lane receives
//       the scores of its tokens g, g + 8.
//   PV: A = V^T with the rows of m-tile R taken as elements 16 (row mod 8) +
//       2R + row / 8, so lane (g, t) reads elements 16g .. 16g+15 of its
//       tokens 2t, 2t+1, 2t+8, 2t+9 as one 16-byte load each; one prmt pairs
//       two tokens' bytes of elements 2R and 2R+1 at once.  B column 0 =
//       RN16(p), column 1 = the remainder (~22 bits), as for int4.
template <int FMT>
struct ConsumerMma8 {
    static constexpr int kScores = 2;
    static constexpr int kPf = 1;
    int rows;  // (unused: one query row)
    uint32_t qb[8][2];
    float acc[8][4];
    float m_run;
    uint64_t l2;  // running sum of the weights of this lane's two tokens, as a pair

    __device__ __forceinline__ void reset()
    {
        m_run = -INFINITY;
        l2 = pk2(0.0f, 0.0f);
#pragma unroll
        for (int i = 0; i < 8; i++)
#pragma unroll
            for (int j = 0; j < 4; j++) acc[i][j] = 0.0f;
    }

    __device__ __forceinline__ void load_q(const uint16_t *qs, int lane)
    {
        const uint4 *q4 = reinterpret_cast<const uint4 *>(qs + 32 * (lane & 3));
#pragma unroll
        for (int u = 0; u < 4; u++) {
            const uint4 v = q4[u];  // elements 32t + 8u .. +7 as pairs
            qb[2 * u][0] = v.x;
            qb[2 * u][1] = v.y;
            qb[2 * u + 1][0] = v.z;
            qb[2 * u + 1][1] = v.w;
        }
    }

    // two exact fp16 pairs of the bytes of w: {b0, b1}, {b2, b3}
    __device__ __forceinline__ static void widen2(uint32_t w, uint32_t &lo, uint32_t &hi)
    {
        if constexpr (FMT == KVQ_FP8_E4M3) {
            asm("cvt.rn.f16x2.e4m3x2 %0, %1;" : "=r"(lo) : "h"(static_cast<unsigned short>(w & 0xffffu)));
            asm("cvt.rn.f16x2.e4m3x2 %0, %1;" : "=r"(hi) : "h"(static_cast<unsigned short>(w >> 16)));
        } else {
            const uint32_t x = w ^ 0x80808080u;
            const __half2 k1152 = __float2half2_rn(1152.0f);
            const uint32_t a = __byte_perm(x, 0x64646464u, 0x4140), b = __byte_perm(x, 0x64646464u, 0x4342);
            lo = h2_bits(__hsub2(*reinterpret_cast<const __half2 *>(&a), k1152));
            hi = h2_bits(__hsub2(*reinterpret_cast<const __half2 *>(&b), k1152));
        }
    }

    // raw dot products q . c of tokens g, g + 8
    __device__ __forceinline__ void qk(const uint8_t *ks, int lane, float sc[2]) const
    {
        const int g = lane >> 2, t = lane & 3;
        float c[4][4];
#pragma unroll
        for (int m = 0; m < 4; m++)
#pragma unroll
            for (int e = 0; e < 4; e++) c[m][e] = 0.0f;
        const uint4 *ra = reinterpret_cast<const uint4 *>(ks + g * 128 + 32 * t);
        const uint4 *rb = reinterpret_cast<const uint4 *>(ks + (g + 8) * 128 + 32 * t);
        const uint4 a0 = ra[0], a1 = ra[1], b0 = rb[0], b1 = rb[1];
        const uint32_t wa[8] = {a0.x, a0.y, a0.z, a0.w, a1.x, a1.y, a1.z, a1.w};
        const uint32_t wb[8] = {b0.x, b0.y, b0.z, b0.w, b1.x, b1.y, b1.z, b1.w};
#pragma unroll
        for (int m = 0; m < 8; m++) {
            uint32_t al, ah, bl, bh;
            widen2(wa[m], al, ah);
            widen2(wb[m], bl, bh);
            mma16816(c[m & 3], al, bl, ah, bh, qb[m][0], qb[m][1]);
        }
        sc[0] = (c[0][0] + c[1][0]) + (c[2][0] + c[3][0]);
        sc[1] = (c[0][2] + c[1][2]) + (c[2][2] + c[3][2]);
    }

    // online softmax of the unit's scores; px = the fp16 pair {x(g), x(g + 8)} of
    // x = p * sv: the rounded values in lanes t == 0, the remainders elsewhere
    __device__ __forceinline__ void softmax(const float sc[2], int ntok, float fac, float sv, int lane,
                                            uint32_t px[1])
    {
        const int g = lane >> 2, t = lane & 3;
        float s0, s1;
        upk2(mul2(pk2(sc[0], sc[1]), pk2(fac, fac)), s0, s1);
        if (g >= ntok) s0 = -INFINITY;
        if (g + 8 >= ntok) s1 = -INFINITY;
        const float lm = fmaxf(s0, s1);
        if (__any_sync(kFull, lm > m_run)) {
            const float mu = warp_max(lm);
            const float alpha = ex2_approx(m_run - mu);
            l2 = mul2(l2, pk2(alpha, alpha));
#pragma unroll
            for (int i = 0; i < 8; i++)
#pragma unroll
                for (int j = 0; j < 4; j++) acc[i][j] *= alpha;
            m_run = mu;
        }
        const uint64_t p01 = pk2(ex2_approx(s0 - m_run), ex2_approx(s1 - m_run));
        l2 = add2(l2, p01);
        uint32_t hi, lo;
        hi_lo_pairs(mul2(p01, pk2(sv, sv)), hi, lo);
        px[0] = t == 0 ? hi : lo;
    }

    __device__ __forceinline__ void pv(const uint8_t *vs, const uint32_t px[1], int lane)
    {
        const int g = lane >> 2, t = lane & 3;
        // column g of B: lanes g == 0 read the rounded weights (from a t == 0 lane), g == 1 the
        // remainders; tokens 2t, 2t + 8 come from lane (2t, .), 2t + 1, 2t + 9 from lane (2t + 1, .)
        const int src = 8 * t + (g & 3);
        const uint32_t ua = __shfl_sync(kFull, px[0], src);
        const uint32_t ub = __shfl_sync(kFull, px[0], src + 4);
        const uint32_t b0 = __byte_perm(ua, ub, 0x5410);  // tokens 2t, 2t + 1
        const uint32_t b1 = __byte_perm(ua, ub, 0x7632);  // tokens 2t + 8, 2t + 9
        const uint4 v0 = *reinterpret_cast<const uint4 *>(vs + (2 * t) * 128 + 16 * g);
        const uint4 v1 = *reinterpret_cast<const uint4 *>(vs + (2 * t + 1) * 128 + 16 * g);
        const uint4 v8 = *reinterpret_cast<const uint4 *>(vs + (2 * t + 8) * 128 + 16 * g);
        const uint4 v9 = *reinterpret_cast<const uint4 *>(vs + (2 * t + 9) * 128 + 16 * g);
        const uint32_t w0[4] = {v0.x, v0.y, v0.z, v0.w}, w1[4] = {v1.x, v1.y, v1.z, v1.w};
        const uint32_t w8[4] = {v8.x, v8.y, v8.z, v8.w}, w9[4] = {v9.x, v9.y, v9.z, v9.w};
#pragma unroll
        for (int R = 0; R < 8; R++) {
            // bytes 2R, 2R + 1 (elements 16g + 2R, + 1) of two tokens: [x.2R, y.2R, x.2R+1, y.2R+1]
            const uint32_t sel = (R & 1) ? 0x7362u : 0x5140u;
            const uint32_t p01 = __byte_perm(w0[R >> 1], w1[R >> 1], sel);
            const uint32_t p89 = __byte_perm(w8[R >> 1], w9[R >> 1], sel);
            uint32_t a0, a1, a2, a3;  // (element 2R: tokens 2t, 2t+1), (2R+1: same), (2R: 2t+8, 2t+9), (2R+1)
            widen2(p01, a0, a1);
            widen2(p89, a2, a3);
            mma16816(acc[R], a0, a1, a2, a3, b0, b1);
        }
    }

    // out row (final) or partial slot: lanes with t == 0 hold elements 16g .. 16g + 15
    // (tile R: row g = element 16g + 2R, row g + 8 = 16g + 2R + 1)
    __device__ __forceinline__ void finish(int lane, uint16_t *orow, float *part)
    {
        float la, lb;
        upk2(l2, la, lb);
        const float l = warp_sum(la + lb) * 0.25f;  // the four lanes of a row group hold the same weights
        const int g = lane >> 2, t = lane & 3;
        if (t != 0) return;
        float v[16];
#pragma unroll
        for (int R = 0; R < 8; R++) {
            v[2 * R] = acc[R][0] + acc[R][1];
            v[2 * R + 1] = acc[R][2] + acc[R][3];
        }
        if (orow) {
            const float inv = 1.0f / l;
            uint32_t hw[8];
#pragma unroll
            for (int i = 0; i < 8; i++) hw[i] = h2_bits(__floats2half2_rn(v[2 * i] * inv, v[2 * i + 1] * inv));
            uint4 *dst = reinterpret_cast<uint4 *>(orow + 16 * g);
            dst[0] = make_uint4(hw[0], hw[1], hw[2], hw[3]);
            dst[1] = make_uint4(hw[4], hw[5], hw[6], hw[7]);
        } else {
            float4 *d4 = reinterpret_cast<float4 *>(part + 4 + 16 * g);
#pragma unroll
            for (int i = 0; i < 4; i++) d4[i] = make_float4(v[4 * i], v[4 * i + 1], v[4 * i + 2], v[4 * i + 3]);
            if (lane == 0) {
                part[0] = m_run;
                part[1] = l;
            }
        }
    }
};

template <>
struct Consumer<KVQ_INT8_PAGE> : ConsumerMma8<KVQ_INT8_PAGE> {
};
template <>
struct Consumer<KVQ_FP8_E4M3> : ConsumerMma8<KVQ_FP8_E4M3> {
};

// int8 and FP8 with grouped query heads, any g <= 8: the 8 MMA columns carry
// the group's heads (column c = head c; columns past g load zero queries), so
// one pass over the codes serves the group.  QK and the V operand are those of
// ConsumerMma8; lane (grp, t) receives the scores of tokens grp, grp + 8 for
// the heads of columns 2t, 2t + 1 (its two slots), and PV column c holds
// RN16(x) of head c (a single fp16 weight, as in the tile kernel: no column is
// left for the remainder), so the lane's accumulators are its slot heads and a
// running-max rescale stays local.  The weights of column grp_d come from lane
// 4 * token + (grp_d >> 1), slot grp_d & 1.
template <int FMT>
struct ConsumerMma8Gqa {
    static constexpr int kScores = 4;
    static constexpr int kPf = 2;
    int rows;  // the group's g <= 8 query heads
    uint32_t qb[8][2];
    float acc[8][4];
    float m_run[2];
    float l_lane[2];

    __device__ __forceinline__ void reset()
    {
        m_run[0] = m_run[1] = -INFINITY;
        l_lane[0] = l_lane[1] = 0.0f;
#pragma unroll
        for (int i = 0; i < 8; i++)
#pragma unroll
            for (int j = 0; j < 4; j++) acc[i][j] = 0.0f;
    }

    // qs: the segment's g query rows in global memory; column g of B = head g (zeros past the group)
    __device__ __forceinline__ void load_q(const uint16_t *qs, int lane)
    {
        const int g = lane >> 2;
        const bool live = g < rows;
        const uint4 *q4 = reinterpret_cast<const uint4 *>(qs + g * kHeadDim + 32 * (lane & 3));
#pragma unroll
        for (int u = 0; u < 4; u++) {
            const uint4 v = live ? q4[u] : make_uint4(0u, 0u, 0u, 0u);  // elements 32t + 8u .. +7 as pairs
            qb[2 * u][0] = v.x;
            qb[2 * u][1] = v.y;
            qb[2 * u + 1][0] = v.z;
            qb[2 * u + 1][1] = v.w;
        }
    }

    // raw dot products: sc[2 r + c] = token grp + 8 r, head slot c (column 2t + c)
    __device__ __forceinline__ void qk(const uint8_t *ks, int lane, float sc[4]) const
    {
        const int g = lane >> 2, t = lane & 3;
        float c[4][4];
#pragma unroll
        for (int m = 0; m < 4; m++)
#pragma unroll
            for (int e = 0; e < 4; e++) c[m][e] = 0.0f;
        const uint4 *ra = reinterpret_cast<const uint4 *>(ks + g * 128 + 32 * t);
        const uint4 *rb = reinterpret_cast<const uint4 *>(ks + (g + 8) * 128 + 32 * t);
        const uint4 a0 = ra[0], a1 = ra[1], b0 = rb[0], b1 = rb[1];
        const uint32_t wa[8] = {a0.x, a0.y, a0.z, a0.w, a1.x, a1.y, a1.z, a1.w};
        const uint32_t wb[8] = {b0.x, b0.y, b0.z, b0.w, b1.x, b1.y, b1.z, b1.w};
#pragma unroll
        for (int m = 0; m < 8; m++) {
            uint32_t al, ah, bl, bh;
            ConsumerMma8<FMT>::widen2(wa[m], al, ah);
            ConsumerMma8<FMT>::widen2(wb[m], bl, bh);
            mma16816(c[m & 3], al, bl, ah, bh, qb[m][0], qb[m][1]);
        }
#pragma unroll
        for (int e = 0; e < 4; e++) sc[e] = (c[0][e] + c[1][e]) + (c[2][e] + c[3][e]);
    }

    // online softmax per head slot; px[c] = {RN16(x(grp)), RN16(x(grp + 8))} of slot c, x = p * sv
    __device__ __forceinline__ void softmax(const float sc[4], int ntok, float fac, float sv, int lane,
                                            uint32_t px[2])
    {
        const int g = lane >> 2;
        float s[4];
        upk2(mul2(pk2(sc[0], sc[1]), pk2(fac, fac)), s[0], s[1]);
        upk2(mul2(pk2(sc[2], sc[3]), pk2(fac, fac)), s[2], s[3]);
        if (g >= ntok) s[0] = s[1] = -INFINITY;
        if (g + 8 >= ntok) s[2] = s[3] = -INFINITY;
        const float lm0 = fmaxf(s[0], s[2]), lm1 = fmaxf(s[1], s[3]);
        if (__any_sync(kFull, lm0 > m_run[0] || lm1 > m_run[1])) {  // a running maximum moves: rescale
#pragma unroll
            for (int c = 0; c < 2; c++) {
                float mu = c ? lm1 : lm0;  // max over the 8 lanes of this t (the unit's 16 tokens)
                mu = fmaxf(mu, __shfl_xor_sync(kFull, mu, 4));
                mu = fmaxf(mu, __shfl_xor_sync(kFull, mu, 8));
                mu = fmaxf(mu, __shfl_xor_sync(kFull, mu, 16));
                mu = fmaxf(mu, m_run[c]);
                const float alpha = ex2_approx(m_run[c] - mu);
                l_lane[c] *= alpha;
#pragma unroll
                for (int i = 0; i < 8; i++) {
                    acc[i][c] *= alpha;
                    acc[i][2 + c] *= alpha;
                }
                m_run[c] = mu;
            }
        }
        const uint64_t vv = pk2(sv, sv);
#pragma unroll
        for (int c = 0; c < 2; c++) {
            const float p0 = ex2_approx(s[c] - m_run[c]), p1 = ex2_approx(s[2 + c] - m_run[c]);
            l_lane[c] += p0 + p1;
            float x0, x1;
            upk2(mul2(pk2(p0, p1), vv), x0, x1);
            px[c] = f16x2_rn(x0, x1);
        }
    }

    __device__ __forceinline__ void pv(const uint8_t *vs, const uint32_t px[2], int lane)
    {
        const int g = lane >> 2, t = lane & 3;
        // column g of B: head g = slot g & 1 of lanes 4 token + (g >> 1); tokens 2t, 2t + 8 from
        // lane (2t, .), 2t + 1, 2t + 9 from lane (2t + 1, .)
        const int src = 8 * t + (g >> 1);
        const bool slot1 = g & 1;
        const uint32_t a0 = __shfl_sync(kFull, px[0], src), a1 = __shfl_sync(kFull, px[1], src);
        const uint32_t c0 = __shfl_sync(kFull, px[0], src + 4), c1 = __shfl_sync(kFull, px[1], src + 4);
        const uint32_t ua = slot1 ? a1 : a0, ub = slot1 ? c1 : c0;
        const uint32_t b0 = __byte_perm(ua, ub, 0x5410);  // tokens 2t, 2t + 1
        const uint32_t b1 = __byte_perm(ua, ub, 0x7632);  // tokens 2t + 8, 2t + 9
        const uint4 v0 = *reinterpret_cast<const uint4 *>(vs + (2 * t) * 128 + 16 * g);
        const uint4 v1 = *reinterpret_cast<const uint4 *>(vs + (2 * t + 1) * 128 + 16 * g);
        const uint4 v8 = *reinterpret_cast<const uint4 *>(vs + (2 * t + 8) * 128 + 16 * g);
        const uint4 v9 = *reinterpret_cast<const uint4 *>(vs + (2 * t + 9) * 128 + 16 * g);
        const uint32_t w0[4] = {v0.x, v0.y, v0.z, v0.w}, w1[4] = {v1.x, v1.y, v1.z, v1.w};
        const uint32_t w8[4] = {v8.x, v8.y, v8.z, v8.w}, w9[4] = {v9.x, v9.y, v9.z, v9.w};
#pragma unroll
        for (int R = 0; R < 8; R++) {
            // bytes 2R, 2R + 1 (elements 16g + 2R, + 1) of two tokens: [x.2R, y.2R, x.2R+1, y.2R+1]
            const uint32_t sel = (R & 1) ? 0x7362u : 0x5140u;
            const uint32_t p01 = __byte_perm(w0[R >> 1], w1[R >> 1], sel);
            const uint32_t p89 = __byte_perm(w8[R >> 1], w9[R >> 1], sel);
            uint32_t e0, e1, e2, e3;
            ConsumerMma8<FMT>::widen2(p01, e0, e1);
            ConsumerMma8<FMT>::widen2(p89, e2, e3);
            mma16816(acc[R], e0, e1, e2, e3, b0, b1);
        }
    }

    // the group's output rows (orow: its `rows` rows) or partial slots (part: 8
    // partials of kPartialStride floats); lane (grp, t) holds elements 16 grp ..
    // 16 grp + 15 of the heads of columns 2t, 2t + 1 (tile R: row grp = element
    // 16 grp + 2R, row grp + 8 = 16 grp + 2R + 1)
    __device__ __forceinline__ void finish(int lane, uint16_t *orow, float *part)
    {
        const int g = lane >> 2, t = lane & 3;
        float l[2];
#pragma unroll
        for (int c = 0; c < 2; c++) {
            float v = l_lane[c];
            v += __shfl_xor_sync(kFull, v, 4);
            v += __shfl_xor_sync(kFull, v, 8);
            v += __shfl_xor_sync(kFull, v, 16);
            l[c] = v;
        }
#pragma unroll
        for (int c = 0; c < 2; c++) {
            const int head = 2 * t + c;
            if (orow && head >= rows) continue;  // a column past the group (its partial slot is written)
            float v[16];
#pragma unroll
            for (int R = 0; R < 8; R++) {
                v[2 * R] = acc[R][c];
                v[2 * R + 1] = acc[R][2 + c];
            }
            if (orow) {
                const float inv = 1.0f / l[c];
                uint32_t hw[8];
#pragma unroll
                for (int i = 0; i < 8; i++) hw[i] = h2_bits(__floats2half2_rn(v[2 * i] * inv, v[2 * i + 1] * inv));
                uint4 *dst = reinterpret_cast<uint4 *>(orow + head * kHeadDim + 16 * g);
                dst[0] = make_uint4(hw[0], hw[1], hw[2], hw[3]);
                dst[1] = make_uint4(hw[4], hw[5], hw[6], hw[7]);
            } else {
                float4 *d4 = reinterpret_cast<float4 *>(part + head * kPartialStride + 4 + 16 * g);
#pragma unroll
                for (int i = 0; i < 4; i++) d4[i] = make_float4(v[4 * i], v[4 * i + 1], v[4 * i + 2], v[4 * i + 3]);
                if (g == 0) {
                    part[head * kPartialStride] = m_run[c];
                    part[head * kPartialStride + 1] = l[c];
                }
            }
        }
    }
};

// ---------------------------------------------------------------------------
// Grouped query heads as the rows of the MMA: a tile of up to kMqRows query
// heads that share one cache head (GQA with a large group, or MQA -- the
// pages' MLA decode absorbed into MQA).  Here one pass over the codes serves
// 16 query heads, so the work per byte is a real small GEMM and the orientation
// flips: QK has A = the tile's q rows (16 heads x 16 elements), B = K^T (16
// elements x 8 tokens), and the S accumulators of two token tiles are, as
// they stand, the A operand of PV (16 heads x 16 tokens) with B = V (16 tokens
// x 8 elements of the head dimension).  No shuffles between QK and PV.
//   k index of QK: a fixed permutation of the head dimension that q's
//   fragment repeats -- int4: k-step (m, s), rows 2t, 2t+1 = elements
//   32t + 8m + 2s + {0, 4}, rows 2t+8, 2t+9 = + {1, 5} (the pairs the nibble
//   widening produces); int8 / FP8: k-step k, rows = elements 32t + 4k + {0,1}
//   and + {2,3}.
//   n index of PV: int4 tile (R, e) holds elements 64R + 8n + e; int8 / FP8
//   tile (R, e) holds 32R + 4n + e, so each lane's output elements of a row
//   are contiguous (int4: 64R + 16t .. +15; bytes: 32R + 8t .. +7).
// Probabilities go to the PV MMA as fp16 x = e * sv / sv_ref, where
// e = 2^(s - m) (the lazy row maximum m keeps e < 2^8) and sv_ref is the
// largest value scale of the segment so far (x <= 2^8, normal fp16 unless
// negligible against the largest value); the output is sv_ref * O / l.
// ---------------------------------------------------------------------------

// the int8 pair {a.byte e, b.byte e} widened exactly to fp16 (a, b already XOR 0x80808080)
__device__ __forceinline__ uint32_t pair_int8(uint32_t a, uint32_t b, int e)
{
    const uint32_t x = __byte_perm(a, b, (uint32_t)e | ((uint32_t)(4 + e) << 8));
    uint32_t y;
    asm("lop3.b32 %0, %1, %2, %3, 0xea;" : "=r"(y) : "r"(x), "r"(0x00ff00ffu), "r"(0x64006400u));  // (x & m) | c
    return h2_bits(__hsub2(*reinterpret_cast<const __half2 *>(&y), __float2half2_rn(1152.0f)));
}

// the FP8 E4M3 pair {a.byte e, b.byte e} widened exactly to fp16
__device__ __forceinline__ uint32_t pair_e4m3(uint32_t a, uint32_t b, int e)
{
    const uint32_t x = __byte_perm(a, b, (uint32_t)e | ((uint32_t)(4 + e) << 4));
    uint32_t d;
    asm("cvt.rn.f16x2.e4m3x2 %0, %1;" : "=r"(d) : "h"(static_cast<unsigned short>(x & 0xffffu)));
    return d;
}

template <int FMT>
struct ConsumerMq {
    static constexpr bool kInt4 = FMT == KVQ_INT4_B64;
    static constexpr int kNT = kInt4 ? 4 : 2;  // token tiles of 8 per unit
    static constexpr int kScores = 4 * kNT;   // S accumulators per lane per unit
    static constexpr int kPf = 2 * kNT;       // P A-fragment registers per unit
    static constexpr float kLazy = 8.0f;      // the row maximum moves only when exceeded by more than this (log2)

    uint32_t qa[8][4];  // Q A-fragments of the 8 k-steps
    float o[16][4];     // O accumulators: 16 tiles of the head dimension
    float m_run[2];     // rows grp, grp + 8 (base-2 scores)
    float l_run[2];     // this lane's part of the row sums of 2^(s - m)
    float r_ref;        // log2 of the reference value scale
    int rows;           // valid rows of the tile
    // int4 only: codes are widened to fp16 subnormals (SubMagic); ob = P x
    // 2^-21 = 2^-24 * 8 sum(x) of rows grp, grp + 8 (the offset's share of
    // every output column), qbias = minus the offset share of their scores
    float ob[4];
    float qbias[2];
    SubMagic mk;

    __device__ __forceinline__ void reset()
    {
        mk.init();
        m_run[0] = m_run[1] = -INFINITY;
        l_run[0] = l_run[1] = 0.0f;
        r_ref = -INFINITY;
        ob[0] = ob[1] = ob[2] = ob[3] = 0.0f;
#pragma unroll
        for (int i = 0; i < 16; i++)
#pragma unroll
            for (int j = 0; j < 4; j++) o[i][j] = 0.0f;
    }

    // qs: the tile's kMqRows query rows (fp16 [16][128]; rows past `rows` hold finite values)
    __device__ __forceinline__ void load_q(const uint16_t *qs, int lane)
    {
        const int g = lane >> 2, t = lane & 3;
        const __half2 odd_scale = __float2half2_rn(kQOdd);
        float se[2] = {0.0f, 0.0f}, so[2] = {0.0f, 0.0f};
#pragma unroll
        for (int m = 0; m < 4; m++) {
            const uint4 va = *reinterpret_cast<const uint4 *>(qs + g * kHeadDim + 32 * t + 8 * m);
            const uint4 vb = *reinterpret_cast<const uint4 *>(qs + (g + 8) * kHeadDim + 32 * t + 8 * m);
            if constexpr (kInt4) {
                // k rows 2t + 8, 2t + 9 of each step meet the odd (bits 4..7) elements: q * kQOdd there
                const uint32_t w[2][4] = {{__byte_perm(va.x, va.z, 0x5410), __byte_perm(va.x, va.z, 0x7632),
                                           __byte_perm(va.y, va.w, 0x5410), __byte_perm(va.y, va.w, 0x7632)},
                                          {__byte_perm(vb.x, vb.z, 0x5410), __byte_perm(vb.x, vb.z, 0x7632),
                                           __byte_perm(vb.y, vb.w, 0x5410), __byte_perm(vb.y, vb.w, 0x7632)}};
#pragma unroll
                for (int r = 0; r < 2; r++) {
                    const __half2 o1 = __hmul2(*reinterpret_cast<const __half2 *>(&w[r][1]), odd_scale);
                    const __half2 o3 = __hmul2(*reinterpret_cast<const __half2 *>(&w[r][3]), odd_scale);
                    qa[2 * m][r] = w[r][0];
                    qa[2 * m][2 + r] = h2_bits(o1);
                    qa[2 * m + 1][r] = w[r][2];
                    qa[2 * m + 1][2 + r] = h2_bits(o3);
                    const float2 x0 = __half22float2(*reinterpret_cast<const __half2 *>(&w[r][0]));
                    const float2 x2 = __half22float2(*reinterpret_cast<const __half2 *>(&w[r][2]));
                    const float2 x1 = __half22float2(o1), x3 = __half22float2(o3);  // binary32 sums
                    se[r] += (x0.x + x0.y) + (x2.x + x2.y);
                    so[r] += (x1.x + x1.y) + (x3.x + x3.y);
                }
            } else {
                qa[2 * m][0] = va.x;
                qa[2 * m][1] = vb.x;
                qa[2 * m][2] = va.y;
                qa[2 * m][3] = vb.y;
                qa[2 * m + 1][0] = va.z;
                qa[2 * m + 1][1] = vb.z;
                qa[2 * m + 1][2] = va.w;
                qa[2 * m + 1][3] = vb.w;
            }
        }
        if constexpr (kInt4) {
#pragma unroll
            for (int r = 0; r < 2; r++) {  // the four lanes t of a row hold its four slices
                float qo = q_offset(se[r], so[r]);
                qo += __shfl_xor_sync(kFull, qo, 1);
                qo += __shfl_xor_sync(kFull, qo, 2);
                qbias[r] = -qo;
            }
        }
    }

    // raw q . c of rows (grp, grp+8) x tokens 8j + 2t, 8j + 2t + 1: sc[4j + {0,1}] row grp, sc[4j + {2,3}] row grp+8
    // (int4: 2^-24 (q . c + q_offset))
    __device__ __forceinline__ void qk(const uint8_t *ks, int lane, float sc[kScores]) const
    {
        const int g = lane >> 2, t = lane & 3;
#pragma unroll
        for (int j = 0; j < kNT; j++) {
            float c[4] = {0.0f, 0.0f, 0.0f, 0.0f};
            if constexpr (kInt4) {
                const uint4 w = *reinterpret_cast<const uint4 *>(ks + (8 * j + g) * 64 + 16 * t);
                const uint32_t u[4] = {w.x, w.y, w.z, w.w};
#pragma unroll
                for (int m = 0; m < 4; m++) {
                    const uint32_t h = u[m] >> 8;
                    mma16816(c, qa[2 * m][0], qa[2 * m][1], qa[2 * m][2], qa[2 * m][3], sub_lo(u[m], mk),
                             sub_hi(u[m], mk));
                    mma16816(c, qa[2 * m + 1][0], qa[2 * m + 1][1], qa[2 * m + 1][2], qa[2 * m + 1][3], sub_lo(h, mk),
                             sub_hi(h, mk));
                }
            } else {
                const uint4 w0 = *reinterpret_cast<const uint4 *>(ks + (8 * j + g) * 128 + 32 * t);
                const uint4 w1 = *reinterpret_cast<const uint4 *>(ks + (8 * j + g) * 128 + 32 * t + 16);
                const uint32_t u[8] = {w0.x, w0.y, w0.z, w0.w, w1.x, w1.y, w1.z, w1.w};
#pragma unroll
                for (int k = 0; k < 8; k++) {
                    __half2 b[2];
                    widen_bytes<FMT>(u[k], b);
                    mma16816(c, qa[k][0], qa[k][1], qa[k][2], qa[k][3], h2_bits(b[0]), h2_bits(b[1]));
                }
            }
#pragma unroll
            for (int e = 0; e < 4; e++) sc[4 * j + e] = c[e];
        }
    }

    // online softmax of the unit; pf = P as the A fragments of the unit's
    // token tiles of 16 (int4: two, bytes: one), fp16 x = 2^(s - m) sv / sv_ref
    __device__ __forceinline__ void softmax(const float sc[kScores], int ntok, float fac, float sv, int lane,
                                            uint32_t pf[kPf])
    {
        const int t = lane & 3;
        // the reference value scale: the segment's largest so far (uniform over the warp)
        const float lsv = __log2f(fmaxf(sv, 1.17549435e-38f));
        if (lsv > r_ref) {
            const float beta = ex2_approx(r_ref - lsv);
#pragma unroll
            for (int i = 0; i < 16; i++)
#pragma unroll
                for (int j = 0; j < 4; j++) o[i][j] *= beta;
            if constexpr (kInt4)
#pragma unroll
                for (int j = 0; j < 4; j++) ob[j] *= beta;
            r_ref = lsv;
        }
        const float ratio = ex2_approx(lsv - r_ref);
        float s[kScores];
        const float f1 = kInt4 ? fac * kUnitEven : fac;
        const float fb0 = kInt4 ? qbias[0] * fac : 0.0f, fb1 = kInt4 ? qbias[1] * fac : 0.0f;
#pragma unroll
        for (int j = 0; j < kNT; j++)
#pragma unroll
            for (int e = 0; e < 4; e++) {
                const int tok = 8 * j + 2 * t + (e & 1);
                s[4 * j + e] = tok < ntok ? fmaf(sc[4 * j + e], f1, (e & 2) ? fb1 : fb0) : -INFINITY;
            }
        float mx[2] = {-INFINITY, -INFINITY};
#pragma unroll
        for (int i = 0; i < kScores; i++) mx[(i >> 1) & 1] = fmaxf(mx[(i >> 1) & 1], s[i]);
#pragma unroll
        for (int r = 0; r < 2; r++) {
            mx[r] = fmaxf(mx[r], __shfl_xor_sync(kFull, mx[r], 1));
            mx[r] = fmaxf(mx[r], __shfl_xor_sync(kFull, mx[r], 2));
        }
        const bool up0 = mx[0] > m_run[0] + kLazy, up1 = mx[1] > m_run[1] + kLazy;
        if (__any_sync(kFull, up0 || up1)) {
            const float a0 = up0 ? ex2_approx(m_run[0] - mx[0]) : 1.0f;
            const float a1 = up1 ? ex2_approx(m_run[1] - mx[1]) : 1.0f;
            if (up0) m_run[0] = mx[0];
            if (up1) m_run[1] = mx[1];
            l_run[0] *= a0;
            l_run[1] *= a1;
#pragma unroll
            for (int i = 0; i < 16; i++) {
                o[i][0] *= a0;
                o[i][1] *= a0;
                o[i][2] *= a1;
                o[i][3] *= a1;
            }
            if constexpr (kInt4) {
                ob[0] *= a0;
                ob[1] *= a0;
                ob[2] *= a1;
                ob[3] *= a1;
            }
        }
        float e[kScores];
#pragma unroll
        for (int i = 0; i < kScores; i++) e[i] = ex2_approx(s[i] - m_run[(i >> 1) & 1]);
#pragma unroll
        for (int j = 0; j < kNT; j++) {
            l_run[0] += e[4 * j] + e[4 * j + 1];
            l_run[1] += e[4 * j + 2] + e[4 * j + 3];
        }
        // A fragment of token tile k (tokens 16k .. 16k+15) = S tiles 2k, 2k+1
#pragma unroll
        for (int k = 0; k < kNT / 2; k++) {
            pf[4 * k + 0] = f16x2_rn(e[8 * k + 0] * ratio, e[8 * k + 1] * ratio);
            pf[4 * k + 1] = f16x2_rn(e[8 * k + 2] * ratio, e[8 * k + 3] * ratio);
            pf[4 * k + 2] = f16x2_rn(e[8 * k + 4] * ratio, e[8 * k + 5] * ratio);
            pf[4 * k + 3] = f16x2_rn(e[8 * k + 6] * ratio, e[8 * k + 7] * ratio);
        }
    }

    __device__ __forceinline__ void pv(const uint8_t *vs, const uint32_t pf[kPf], int lane)
    {
        const int g = lane >> 2, t = lane & 3;
        if constexpr (kInt4) {
#pragma unroll
            for (int k = 0; k < 2; k++) {
                // the offset: every column of B = 8 * 2^-24 (the fp16 subnormal 0x0008)
                mma16816(ob, pf[4 * k], pf[4 * k + 1], pf[4 * k + 2], pf[4 * k + 3], 0x00080008u, 0x00080008u);
#pragma unroll
                for (int R = 0; R < 2; R++) {
                    // word g + 8R (elements 64R + 8g .. +7) of tokens 16k + 2t, +1, +8, +9
                    const uint8_t *vb = vs + (16 * k + 2 * t) * 64 + 4 * (g + 8 * R);
                    const uint32_t wa = *reinterpret_cast<const uint32_t *>(vb);
                    const uint32_t wb = *reinterpret_cast<const uint32_t *>(vb + 64);
                    const uint32_t wc = *reinterpret_cast<const uint32_t *>(vb + 8 * 64);
                    const uint32_t wd = *reinterpret_cast<const uint32_t *>(vb + 9 * 64);
                    uint32_t xab[4], xcd[4];
#pragma unroll
                    for (int q = 0; q < 4; q++) {
                        const uint32_t bsel = (uint32_t)q | ((uint32_t)q << 4) | ((uint32_t)(4 + q) << 8) |
                                              ((uint32_t)(4 + q) << 12);
                        xab[q] = __byte_perm(wa, wb, bsel);
                        xcd[q] = __byte_perm(wc, wd, bsel);
                    }
#pragma unroll
                    for (int e = 0; e < 8; e++)
                        mma16816(o[8 * R + e], pf[4 * k], pf[4 * k + 1], pf[4 * k + 2], pf[4 * k + 3],
                                 sub_pair(xab[e >> 1], e & 1, mk), sub_pair(xcd[e >> 1], e & 1, mk));
                }
            }
        } else {
#pragma unroll
            for (int R = 0; R < 4; R++) {
                // word g + 8R (elements 32R + 4g .. +3) of tokens 2t, 2t+1, 2t+8, 2t+9
                const uint8_t *vb = vs + (2 * t) * 128 + 4 * (g + 8 * R);
                uint32_t wa = *reinterpret_cast<const uint32_t *>(vb);
                uint32_t wb = *reinterpret_cast<const uint32_t *>(vb + 128);
                uint32_t wc = *reinterpret_cast<const uint32_t *>(vb + 8 * 128);
                uint32_t wd = *reinterpret_cast<const uint32_t *>(vb + 9 * 128);
                if constexpr (FMT == KVQ_INT8_PAGE) {
                    wa ^= 0x80808080u;
                    wb ^= 0x80808080u;
                    wc ^= 0x80808080u;
                    wd ^= 0x80808080u;
                }
#pragma unroll
                for (int e = 0; e < 4; e++) {
                    uint32_t b0, b1;
                    if constexpr (FMT == KVQ_INT8_PAGE) {
                        b0 = pair_int8(wa, wb, e);
                        b1 = pair_int8(wc, wd, e);
                    } else {
                        b0 = pair_e4m3(wa, wb, e);
                        b1 = pair_e4m3(wc, wd, e);
                    }
                    mma16816(o[4 * R + e], pf[0], pf[1], pf[2], pf[3], b0, b1);
                }
            }
        }
    }

    // rows: the tile's output rows (orow, fp16, 128 apart) or partial slots
    // (part, kPartialStride floats apart: m, l, pad, pad, sv_ref * O)
    __device__ __forceinline__ void finish(int lane, uint16_t *orow, float *part)
    {
        const int g = lane >> 2, t = lane & 3;
        float l[2];
#pragma unroll
        for (int r = 0; r < 2; r++) {
            l[r] = l_run[r] + __shfl_xor_sync(kFull, l_run[r], 1);
            l[r] += __shfl_xor_sync(kFull, l[r], 2);
        }
        const float ref = ex2_approx(r_ref);
#pragma unroll
        for (int r = 0; r < 2; r++) {
            const int row = g + 8 * r;
            if (row >= rows) continue;
            const float mul = orow ? ref / l[r] : ref;
            if constexpr (kInt4) {
                // raw sums over the widened codes, less the offset share (2^24 ob = 8 sum(x))
                const float xs = kUnitEven / kOffEven * ob[2 * r];
                const float xb_even = -kOffEven * xs, xb_odd = -kOffOdd * xs;
#pragma unroll
                for (int R = 0; R < 2; R++) {
                    float v[16];
#pragma unroll
                    for (int e = 0; e < 8; e++) {
                        const float f = (e & 1) ? kUnitOdd : kUnitEven, xb = (e & 1) ? xb_odd : xb_even;
                        v[e] = fmaf(o[8 * R + e][2 * r], f, xb) * mul;          // element 64R + 16t + e
                        v[8 + e] = fmaf(o[8 * R + e][2 * r + 1], f, xb) * mul;  // element 64R + 16t + 8 + e
                    }
                    if (orow) {
                        uint4 *d = reinterpret_cast<uint4 *>(orow + row * kHeadDim + 64 * R + 16 * t);
                        d[0] = make_uint4(f16x2_rn(v[0], v[1]), f16x2_rn(v[2], v[3]), f16x2_rn(v[4], v[5]),
                                          f16x2_rn(v[6], v[7]));
                        d[1] = make_uint4(f16x2_rn(v[8], v[9]), f16x2_rn(v[10], v[11]), f16x2_rn(v[12], v[13]),
                                          f16x2_rn(v[14], v[15]));
                    } else {
                        float4 *d = reinterpret_cast<float4 *>(part + row * kPartialStride + 4 + 64 * R + 16 * t);
#pragma unroll
                        for (int i = 0; i < 4; i++) d[i] = make_float4(v[4 * i], v[4 * i + 1], v[4 * i + 2], v[4 * i + 3]);
                    }
                }
            } else {
#pragma unroll
                for (int R = 0; R < 4; R++) {
                    float v[8];
#pragma unroll
                    for (int e = 0; e < 4; e++) {
                        v[e] = o[4 * R + e][2 * r] * mul;          // element 32R + 8t + e
                        v[4 + e] = o[4 * R + e][2 * r + 1] * mul;  // element 32R + 8t + 4 + e
                    }
                    if (orow) {
                        *reinterpret_cast<uint4 *>(orow + row * kHeadDim + 32 * R + 8 * t) =
                            make_uint4(f16x2_rn(v[0], v[1]), f16x2_rn(v[2], v[3]), f16x2_rn(v[4], v[5]),
                                       f16x2_rn(v[6], v[7]));
                    } else {
                        float4 *d = reinterpret_cast<float4 *>(part + row * kPartialStride + 4 + 32 * R + 8 * t);
                        d[0] = make_float4(v[0], v[1], v[2], v[3]);
                        d[1] = make_float4(v[4], v[5], v[6], v[7]);
                    }
                }
            }
            if (part && t == 0) {
                part[row * kPartialStride] = m_run[r];
                part[row * kPartialStride + 1] = l[r];
            }
        }
    }
};

// ---------------------------------------------------------------------------
// The split: the units 0 .. U-1 of a launch are cut into GW contiguous warp
// ranges [U w / GW, U (w+1) / GW), one per active warp (the pieces of the
// split).  Where a piece begins and ends depends only on (U, GW), so the
// partials of a (sequence, head) split over several pieces are found without
// any bookkeeping.
// ---------------------------------------------------------------------------
struct Split {
    int64_t U, GW;  // units, active warps

    __device__ __forceinline__ void init(int64_t units, int64_t warps)
    {
        U = units;
        GW = warps;
    }
    __device__ __forceinline__ int64_t start(int64_t w) const { return U * w / GW; }
    // the piece (warp range) that holds unit u
    __device__ __forceinline__ int64_t piece_of(int64_t u) const { return ((u + 1) * GW - 1) / U; }
};

// ---------------------------------------------------------------------------
// Counters of the split, one word per piece: the word of the piece that holds
// a split (sequence, head)'s last unit counts the units of it whose partials
// are written.  A counter word holds a count in its low kCountBits bits and,
// above them, count * epoch mod 2^40, where the epoch is an odd tag chosen per
// call: an add of n is one atomic add of n * (1 + 2^24 epoch).
// Within one call every word stays consistent (high part == low part *
// epoch); a word left non-zero by another call (an aborted launch, a
// workspace that was never zero-filled) is inconsistent under this call's
// epoch, so KVQ_FLAG_BAD_WORKSPACE is raised instead of merging early.  The
// warp whose add completes a count puts the word back to zero.  One atomic
// round trip, no retries: the pieces of a (sequence, head) finish at about
// the same time, and a compare-and-swap there retried under contention for
// several microseconds.
// Ordering: the warp barrier orders every lane's partial stores before lane
// 0's acq_rel add (release), whose acquire side in the completing warp,
// followed by that warp's barrier, orders its reads of the other pieces'
// partials after their writers' stores.
// ---------------------------------------------------------------------------
__device__ __forceinline__ unsigned long long add_acq_rel_gpu(unsigned long long *p, unsigned long long v)
{
    unsigned long long old;
    asm volatile("atom.acq_rel.gpu.global.add.u64 %0, [%1], %2;" : "=l"(old) : "l"(p), "l"(v) : "memory");
    return old;
}

constexpr unsigned long long kCountMask = (1ull << kCountBits) - 1;
constexpr unsigned long long kTagMask = (1ull << 40) - 1;

__device__ __forceinline__ unsigned long long counter_step(unsigned long long epoch)
{
    return 1ull + (epoch << kCountBits);
}

// true when a counter word read under `epoch` carries only this call's adds
__device__ __forceinline__ bool counter_consistent(unsigned long long w, unsigned long long epoch)
{
    return ((w >> kCountBits) & kTagMask) == (((w & kCountMask) * epoch) & kTagMask);
}

// Called by every lane of a warp right after it wrote a partial covering
// `units` of a split (sequence, head) of `total` units: counts them and
// returns true in the warp whose add completes the count.
__device__ __noinline__ bool count_units(unsigned long long *slot, uint32_t units, uint32_t total,
                                         unsigned long long epoch, int lane, int32_t *status)
{
    __syncwarp();
    int last = 0;
    if (lane == 0) {
        const unsigned long long old = add_acq_rel_gpu(slot, (unsigned long long)units * counter_step(epoch));
        const unsigned long long c = (old & kCountMask) + units;
        if (!counter_consistent(old, epoch) || c > total) {
            set_flag(status, KVQ_FLAG_BAD_WORKSPACE);  // not zero-filled, or left over by an aborted call
        } else if (c == total) {
            *slot = 0ull;
            last = 1;
        }
    }
    last = __shfl_sync(kFull, last, 0);
    if (!last) return false;
    __syncwarp();
    return true;
}

// One warp: combine the partials of pieces gf .. gf + cnt - 1 (slot 1 of piece
// gf when the (sequence, head) is that piece's last segment, slot 0 of the
// others) into one fp16 output row.  Partials are read from L2 (ld.cg): other
// SMs wrote them during this launch.  The loads of a batch of kBatch pieces
// are independent of one another, so a merge of up to kBatch pieces costs one
// round trip to L2.
// (not inlined: a rare path, kept out of the streaming loop's register budget)
// slot_floats: floats per partial slot (G partials of a group of query
// heads); head: which of them.
template <int kBatch>
__device__ __noinline__ void merge_pieces(const float *partials, int64_t slot_floats, int head, int64_t gf, int cnt,
                                          int first_slot, uint16_t *out_row, int lane)
{
    const float *pbase = partials + gf * 2 * slot_floats + (int64_t)head * kPartialStride;
    auto part = [&](int i) { return pbase + ((int64_t)i * 2 + (i == 0 ? first_slot : 0)) * slot_floats; };
    // lane i < cnt: (m, l) of piece i; every lane: its 4 elements of pieces
    // 0 .. kBatch-1 and their m -- all issued before any of them is used
    float2 ml = make_float2(-INFINITY, 0.0f);
    if (lane < cnt) ml = __ldcg(reinterpret_cast<const float2 *>(part(lane)));
    float4 a[kBatch];
    float mj[kBatch];
#pragma unroll
    for (int j = 0; j < kBatch; j++) {
        const float *src = part(j < cnt ? j : 0);
        a[j] = __ldcg(reinterpret_cast<const float4 *>(src + 4) + lane);
        mj[j] = j < cnt ? __ldcg(src) : -INFINITY;
    }
    float M = ml.x;
    for (int i = lane + 32; i < cnt; i += 32) M = fmaxf(M, __ldcg(part(i)));
    M = warp_max(M);
    float L = lane < cnt ? ml.y * ex2_approx(ml.x - M) : 0.0f;
    for (int i = lane + 32; i < cnt; i += 32) {
        const float2 v = __ldcg(reinterpret_cast<const float2 *>(part(i)));
        L += v.y * ex2_approx(v.x - M);
    }
    L = warp_sum(L);
    float4 o = make_float4(0.f, 0.f, 0.f, 0.f);
    for (int i0 = 0; i0 < cnt; i0 += kBatch) {
        if (i0 > 0) {
#pragma unroll
            for (int j = 0; j < kBatch; j++) {
                const float *src = part(i0 + j < cnt ? i0 + j : 0);
                a[j] = __ldcg(reinterpret_cast<const float4 *>(src + 4) + lane);
                mj[j] = i0 + j < cnt ? __ldcg(src) : -INFINITY;
            }
        }
#pragma unroll
        for (int j = 0; j < kBatch; j++) {
            const float w = ex2_approx(mj[j] - M);  // 0 for the padding entries
            o.x += a[j].x * w;
            o.y += a[j].y * w;
            o.z += a[j].z * w;
            o.w += a[j].w * w;
        }
    }
    const float inv = 1.0f / L;
    const __half2 lo = __floats2half2_rn(o.x * inv, o.y * inv);
    const __half2 hi = __floats2half2_rn(o.z * inv, o.w * inv);
    reinterpret_cast<uint2 *>(out_row)[lane] =
        make_uint2(*reinterpret_cast<const uint32_t *>(&lo), *reinterpret_cast<const uint32_t *>(&hi));
}

// One warp: merge_pieces for all G query heads of one cache head at once.  A
// piece holds the G heads' partials side by side; the loads of kBatch pieces x
// G heads are issued together, so a merge of cnt pieces takes about cnt /
// kBatch round trips to L2 instead of G times as many (kBatch = 8 / G keeps
// the call within the kernel's register budget).  A slot holds kSlotHeads
// heads; this call merges G of them from head0 on and writes the first nheads
// (a group of g < G heads leaves slots of heads that do not exist; a group of
// 8 is merged as two calls of 4: one call of 8 heads would not fit beside the
// streaming loop's live registers).
template <int kBatch, int G, int kSlotHeads = G>
__device__ __noinline__ void merge_group(const float *partials, int64_t gf, int cnt, int first_slot,
                                         uint16_t *out_rows, int lane, int head0, int nheads)
{
    constexpr int64_t kSlot = (int64_t)kSlotHeads * kPartialStride;
    const float *pbase = partials + gf * 2 * kSlot + (int64_t)head0 * kPartialStride;
    out_rows += (int64_t)head0 * kHeadDim;
    auto part = [&](int i) { return pbase + ((int64_t)i * 2 + (i == 0 ? first_slot : 0)) * kSlot; };
    float2 ml[G];
    float4 a[kBatch][G];
    float mj[kBatch][G];
#pragma unroll
    for (int g = 0; g < G; g++)
        ml[g] = lane < cnt ? __ldcg(reinterpret_cast<const float2 *>(part(lane) + g * kPartialStride))
                           : make_float2(-INFINITY, 0.0f);
#pragma unroll
    for (int j = 0; j < kBatch; j++) {
        const float *src = part(j < cnt ? j : 0);
#pragma unroll
        for (int g = 0; g < G; g++) {
            a[j][g] = __ldcg(reinterpret_cast<const float4 *>(src + g * kPartialStride + 4) + lane);
            mj[j][g] = j < cnt ? __ldcg(src + g * kPartialStride) : -INFINITY;
        }
    }
    float M[G], L[G];
    float4 o[G];
#pragma unroll
    for (int g = 0; g < G; g++) M[g] = ml[g].x;
    for (int i = lane + 32; i < cnt; i += 32)
#pragma unroll
        for (int g = 0; g < G; g++) M[g] = fmaxf(M[g], __ldcg(part(i) + g * kPartialStride));
#pragma unroll
    for (int g = 0; g < G; g++) {
        M[g] = warp_max(M[g]);
        L[g] = lane < cnt ? ml[g].y * ex2_approx(ml[g].x - M[g]) : 0.0f;
    }
    for (int i = lane + 32; i < cnt; i += 32)
#pragma unroll
        for (int g = 0; g < G; g++) {
            const float2 v = __ldcg(reinterpret_cast<const float2 *>(part(i) + g * kPartialStride));
            L[g] += v.y * ex2_approx(v.x - M[g]);
        }
#pragma unroll
    for (int g = 0; g < G; g++) {
        L[g] = warp_sum(L[g]);
        o[g] = make_float4(0.f, 0.f, 0.f, 0.f);
    }
    for (int i0 = 0; i0 < cnt; i0 += kBatch) {
        if (i0 > 0) {
#pragma unroll
            for (int j = 0; j < kBatch; j++) {
                const float *src = part(i0 + j < cnt ? i0 + j : 0);
#pragma unroll
                for (int g = 0; g < G; g++) {
                    a[j][g] = __ldcg(reinterpret_cast<const float4 *>(src + g * kPartialStride + 4) + lane);
                    mj[j][g] = i0 + j < cnt ? __ldcg(src + g * kPartialStride) : -INFINITY;
                }
            }
        }
#pragma unroll
        for (int j = 0; j < kBatch; j++)
#pragma unroll
            for (int g = 0; g < G; g++) {
                const float w = ex2_approx(mj[j][g] - M[g]);
                o[g].x += a[j][g].x * w;
                o[g].y += a[j][g].y * w;
                o[g].z += a[j][g].z * w;
                o[g].w += a[j][g].w * w;
            }
    }
#pragma unroll
    for (int g = 0; g < G; g++) {
        if (g >= nheads) break;
        const float inv = 1.0f / L[g];
        const __half2 lo = __floats2half2_rn(o[g].x * inv, o[g].y * inv);
        const __half2 hi = __floats2half2_rn(o[g].z * inv, o[g].w * inv);
        reinterpret_cast<uint2 *>(out_rows + g * kHeadDim)[lane] =
            make_uint2(*reinterpret_cast<const uint32_t *>(&lo), *reinterpret_cast<const uint32_t *>(&hi));
    }
}

template <int FMT, int G>
struct ConsumerFor {
    using type = ConsumerGqa<G>;
};
template <>
struct ConsumerFor<KVQ_INT8_PAGE, 8> {
    using type = ConsumerMma8Gqa<KVQ_INT8_PAGE>;
};
template <>
struct ConsumerFor<KVQ_FP8_E4M3, 8> {
    using type = ConsumerMma8Gqa<KVQ_FP8_E4M3>;
};
template <int FMT>
struct ConsumerFor<FMT, 1> {
    using type = Consumer<FMT>;
};
template <int FMT>
struct ConsumerFor<FMT, kMqG> {
    using type = ConsumerMq<FMT>;
};

// Shared prologue of the split and merge kernels: the sequence lengths (clamped
// to the table, flagged), the prefix of units over (sequence, unit head) with
// HU unit heads per sequence, and the split geometry -- the same in every CTA.
template <int UT>
__device__ __forceinline__ void decode_prologue(const DecodeParams &p, int HU, int grid_warps, int32_t *s_cu,
                                                int32_t *s_len, Split *s_split)
{
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int B = p.num_seqs;
    const int max_len = p.max_blocks * kPage;
    for (int b = tid; b < B; b += blockDim.x) {
        int L = p.seq_lens[b];
        if (L < 0 || L > max_len) {
            if (blockIdx.x == 0) set_flag(p.status, KVQ_FLAG_BAD_LENGTH);
            L = L < 0 ? 0 : max_len;
        }
        s_len[b] = L;
    }
    __syncthreads();
    if (warp == 0) {
        const int per = (B + 31) / 32;
        int sum = 0;
        for (int k = 0; k < per; k++) {
            const int i = lane * per + k;
            if (i < B) sum += units_of(s_len[i], UT) * HU;
        }
        int incl = sum;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const int t = __shfl_up_sync(kFull, incl, o);
            if (lane >= o) incl += t;
        }
        int run = incl - sum;
        for (int k = 0; k < per; k++) {
            const int i = lane * per + k;
            if (i < B) {
                s_cu[i] = run;
                run += units_of(s_len[i], UT) * HU;
            }
        }
        if (lane == 31) s_cu[B] = incl;
    }
    __syncthreads();
    if (tid == 0) {
        const int64_t U = s_cu[B];
        // active warps: at least kMinUnitsPerWarp units each
        s_split->init(U, imin64((int64_t)grid_warps, (U + kMinUnitsPerWarp - 1) / kMinUnitsPerWarp));
    }
    __syncthreads();
}

// G: query heads per cache head (1: multi-head attention; 2, 4, 8: grouped
// heads in the MMA columns, any g <= G; kMqG: tiles of up to 16 query heads of any group
// size p.group, p.tiles tiles per cache head, each tile a unit head of its own).
// kHook: the instantiation launched while the test hook of kvq_testing.h is
// set -- its waits take their limit from p.wait_limit_ns and the grid's first
// warp can leave a chunk unissued; the other instantiations wait the fixed
// kWaitLimitNs and carry no such check.
template <int FMT, int G, bool kHook = false>
__global__ void __launch_bounds__(DecShape<FMT, G>::kWarps * 32, DecFmt<FMT>::kCtasPerSm)
    decode_split_kernel(DecodeParams p, int grid_warps)
{
    using F = DecFmt<FMT>;
    using CS = typename ConsumerFor<FMT, G>::type;
    constexpr bool kTiles = G == kMqG;
    constexpr int kStages = F::kStages;
    constexpr int UPS = F::kUnitsPerStage;
    constexpr int kQRows = DecShape<FMT, G>::kQRows;
    constexpr bool kQGlobal = DecShape<FMT, G>::kQGlobal;
    using WS = WarpSmem<kStages, UPS * kUnitBytes, kQRows>;
    // one piece's partials: a row per query head of the unit head (G, or a tile's 16)
    constexpr int64_t kSlotFloats = (int64_t)(kTiles ? kMqRows : G) * kPartialStride;
    constexpr int UT = F::kUnitTok;
    constexpr int UPP = F::kUnitsPerPage;
    constexpr int RB = F::kRowBytes;
    extern __shared__ __align__(128) uint8_t smem_raw[];
    WS *wsm_all = reinterpret_cast<WS *>(smem_raw);
    constexpr int kDecWarps = DecShape<FMT, G>::kWarps;
    int32_t *s_cu = reinterpret_cast<int32_t *>(smem_raw + kDecWarps * sizeof(WS));
    int32_t *s_len = s_cu + kMaxSeqsPerLaunch + 1;

    const int tid = threadIdx.x;
    const int lane = tid & 31;
    const int warp = tid >> 5;
    const int B = p.num_seqs;
    const int H = p.num_heads;                  // cache heads
    const int T = kTiles ? p.tiles : 1;         // unit heads per cache head
    const int HU = H * T;                       // unit heads per sequence
    const int g_rows = G > 1 ? p.group : 1;  // query heads per cache head (column kernels: g <= G)
    pdl_launch_dependents();
    // Until pdl_wait below, the previous kernel of the stream may still be
    // running.  Only the sequence lengths and the block table are read before
    // it: no kernel of this library writes them (the codes, scales, query and
    // output are touched only after the wait), so the prologue and the first
    // block-table fetch overlap the previous kernel's tail.

    // ---- per-sequence lengths, the (unit heads x units) prefix and the split
    // geometry, in shared memory (the split is read only when a piece starts
    // or a segment ends) ----
    Split *s_split = reinterpret_cast<Split *>(smem_raw + kDecWarps * sizeof(WS) +
                                               ((2 * kMaxSeqsPerLaunch + 1) * sizeof(int32_t) + 15) / 16 * 16);
    // Tiles: the split runs over the units of one tile, (sequence, cache head,
    // unit), cut into split_warps pieces; the warps come in T groups and group
    // t runs tile t of every piece, so the T tiles of a cache head stream the
    // same pages at the same time and all but the first read them from L2.
    const int split_warps = kTiles ? grid_warps / T : grid_warps;
    decode_prologue<UT>(p, kTiles ? H : HU, split_warps, s_cu, s_len, s_split);
    const Split &sp = *s_split;
    // logical warp index, round-robin over the CTAs: when fewer than all warps
    // have work (GW < grid warps) the active ones spread over every SM
    const int gw = warp * (int)gridDim.x + blockIdx.x;
    const int my_tile = kTiles ? gw / split_warps : 0;  // tile t of the warp's piece (tiles: the same warp slot of each CTA)
    const int pi_cur = gw - my_tile * split_warps;      // the warp's piece
    const bool active = my_tile < T && pi_cur < sp.GW;
    unsigned long long *const piece_ctr = p.counters;  // one word per piece

    // ---- issue cursor: the next unit of this warp's piece = (ib, ih, ic); rem units left ----
    int rem = 0;
    int ib = 0, ih = 0, ic = 0;
    auto seek = [&](int64_t x) {
        int lo = 0, hi = B - 1;
        while (lo < hi) {
            const int mid = (lo + hi + 1) >> 1;
            if (s_cu[mid] <= x) lo = mid; else hi = mid - 1;
        }
        ib = lo;
        const int n = units_of(s_len[ib], UT);
        const int off = (int)(x - s_cu[ib]);
        ih = (off / n) * T + my_tile;  // the unit head: cache head off / n, the warp's tile
        ic = off % n;
    };
    if (active) {
        const int64_t x = sp.start(pi_cur);
        rem = (int)(sp.start(pi_cur + 1) - x);
        seek(x);
    }
    int inb = units_of(s_len[ib], UT);  // units of the issue cursor's sequence
    // page ring: lane l holds page slot ring_j0 + l of (ring_b, ring_h) and,
    // once loaded (after the wait: appends write them), its two scales
    int ring_b = -1, ring_h = -1, ring_j0 = 0;
    int r_page = 0;
    float r_sk = 0.0f, r_sv = 0.0f;
    bool ring_scales_due = false;
    auto ring_pages = [&](int b, int h, int j) {
        ring_b = b;
        ring_h = h;
        ring_j0 = j;
        const int jl = j + lane;
        const int npages = (s_len[b] + kPage - 1) / kPage;
        int pg = 0;
        if (jl < npages) {
            pg = p.block_table[(int64_t)b * p.max_blocks + jl];
            if (pg < 0 || pg >= p.num_pages) {
                set_flag(p.status, KVQ_FLAG_BAD_PAGE);
                pg = 0;
            }
        }
        r_page = pg;
        ring_scales_due = true;
    };
    if (active) ring_pages(ib, ih / T, ic / UPP);

    pdl_wait();  // from here on, the previous kernel's writes are visible

    if (warp == 0) {  // no warp owns a unit of an empty sequence: its rows are zeros
        for (int base = 0; base < B; base += 32) {
            uint32_t m = __ballot_sync(kFull, base + lane < B && s_len[base + lane] == 0);
            while (m) {
                const int b = base + __ffs(m) - 1;
                m &= m - 1;
                if (b % (int)gridDim.x != (int)blockIdx.x) continue;
                uint4 *row = reinterpret_cast<uint4 *>(p.out + (int64_t)b * H * g_rows * kHeadDim);
                for (int e = lane; e < H * g_rows * (kHeadDim / 8); e += 32) row[e] = make_uint4(0u, 0u, 0u, 0u);
            }
        }
    }
    if (!active) return;

    WS &ws = wsm_all[warp];
    if (lane == 0) {
#pragma unroll
        for (int s = 0; s < kStages; s++) mbar_init(&ws.full[s], 1);
        mbar_init_fence();
    }
    __syncwarp();

    constexpr uint32_t kPageBytes = kPage * RB;

    int ci = 0;                 // stages filled so far (chunk count)
    // the timeout test's chunk (kvq_testing.h): the grid's first warp leaves
    // its copies unissued, so the stage's wait runs out with nothing in flight
    const int skip_ci = kHook && gw == 0 ? p.test_skip_chunk : -1;
    const uint64_t wait_ns = kHook ? p.wait_limit_ns : kWaitLimitNs;
    bool issue_done = false;    // the warp's range is fully issued
    bool piece_new = true;      // the next stage is the warp's first
    // Fill stage ci % kStages with the next chunk: the cursor's unit and the
    // following ones of the same stage-sized group of its page, within the
    // (sequence, head) and the warp's range.  Returns false when no work is left.
    auto issue = [&]() -> bool {
        if (rem == 0) {
            issue_done = true;
            return false;
        }
        const int s = ci % kStages;
        const int j = ic / UPP;
        const int nh = UPS > 1 ? min(min(UPS - ic % UPS, inb - ic), rem) : 1;
        const int hc = kTiles ? ih / T : ih;  // the cache head of the unit head
        // (tiles of one cache head share its ring: a tile after the first starts again at page 0)
        if (ib != ring_b || hc != ring_h || j < ring_j0 || j >= ring_j0 + 32) ring_pages(ib, hc, j);
        const int pg = __shfl_sync(kFull, r_page, j - ring_j0);
        const bool new_seg = piece_new || (ic == 0);
        if (ring_scales_due) {  // the ring's scales (after the wait: appends write them)
            r_sk = p.k_scales[(int64_t)r_page * H + ring_h];
            r_sv = p.v_scales[(int64_t)r_page * H + ring_h];
            ring_scales_due = false;
        }
        if (lane == 0) {
            // The refill of stage s follows the warp's reads of it: every lane
            // consumed those values (mma operands) before the __syncwarp that
            // precedes this issue, so the copy cannot overtake them.
            const uint32_t cb = (uint32_t)nh * kUnitBytes;
            // the unit head's query rows: the g rows of the cache head, or one tile of the group
            const int tile = kTiles ? ih - hc * T : 0;
            const int qrows = kTiles ? min(kMqRows, g_rows - kMqRows * tile) : kQGlobal ? 0 : g_rows;
            const uint32_t qbytes = (uint32_t)qrows * kHeadDim * 2;
            const uint32_t bytes = 2 * cb + (new_seg ? qbytes : 0);
            mbar_arrive_expect_tx(&ws.full[s], bytes);
            if (!kHook || ci != skip_ci) {
                const size_t off = ((size_t)pg * H + hc) * kPageBytes + (size_t)(ic % UPP) * kUnitBytes;
                bulk_copy_g2s(ws.k[s], p.k_codes + off, cb, &ws.full[s]);
                bulk_copy_g2s(ws.v[s], p.v_codes + off, cb, &ws.full[s]);
                if (new_seg && qbytes)
                    bulk_copy_g2s(ws.q[s], p.q + (((size_t)ib * H + hc) * g_rows + kMqRows * tile) * kHeadDim, qbytes,
                                  &ws.full[s]);
            }
        }
        const float sk = __shfl_sync(kFull, r_sk, j - ring_j0);
        const float sv = __shfl_sync(kFull, r_sv, j - ring_j0);
        if (lane == 0) {
            const int ntok = min(nh * UT, s_len[ib] - ic * UT);
            *reinterpret_cast<int4 *>(&ws.meta[s].b) = make_int4(ib, ih, ic, ntok);
            *reinterpret_cast<float4 *>(&ws.meta[s].sk) =
                make_float4(sk, sv, __int_as_float(new_seg ? 1 : 0), __int_as_float(nh));
        }
        // advance the cursor by the chunk
        ic += nh;
        rem -= nh;
        piece_new = false;
        if (ic == inb) {
            ic = 0;
            ih += T;  // the next cache head, same tile
            if (ih >= HU) {
                ih = my_tile;
                ++ib;
                while (ib < B && s_len[ib] == 0) ++ib;
                if (ib < B) inb = units_of(s_len[ib], UT);
            }
        }
        ++ci;
        return true;
    };

    for (int i = 0; i < kStages; i++)
        if (!issue()) break;
    __syncwarp();

    // ---- consumer: qk of unit n+1 overlaps pv of unit n ----
    CS cs;
    cs.reset();
    int cur_b = -1, cur_h = -1;
    int seg_c = 0;        // first unit of the current segment within its (sequence, head)
    int seg_units = 0;    // units of it consumed so far

    // the first output row of unit head h of sequence b
    auto out_rows = [&](int b, int h) -> uint16_t * {
        if constexpr (kTiles) {
            const int hc = h / T;
            return p.out + (((int64_t)b * H + hc) * g_rows + kMqRows * (h - hc * T)) * kHeadDim;
        } else {
            return p.out + ((int64_t)b * H + h) * g_rows * kHeadDim;
        }
    };
    // units c .. c + units - 1 of (b, h), consumed by this warp (piece pi), are done
    auto flush = [&](int b, int h, int c, int units) {
        const int pi = pi_cur;
        const int n = units_of(s_len[b], UT);
        const int64_t u0 = s_cu[b] + (int64_t)(kTiles ? h / T : h) * n;  // in the split's unit space
        const int64_t sa = u0 + c;
        if (sa == u0 && units == n) {
            cs.finish(lane, out_rows(b, h), nullptr);
        } else {  // split: the piece's first segment goes to its slot 0, its last to slot 1
            // (tiles: the partials of tile t's pieces follow those of tile t - 1)
            const int64_t slot_piece = (int64_t)my_tile * split_warps + pi;
            cs.finish(lane, nullptr,
                      p.partials + (slot_piece * 2 + (sa == sp.start(pi) ? 0 : 1)) * kSlotFloats);
            if constexpr (kTiles) return;  // merged by the second launch
            const int64_t pf = sp.piece_of(u0);
            const int64_t pl = sp.piece_of(u0 + n - 1);
            if (count_units(piece_ctr + pl, (uint32_t)units, (uint32_t)n, p.epoch, lane, p.status)) {
                const int first_slot = (sp.start(pf) != u0) ? 1 : 0;
                uint16_t *orow = out_rows(b, h);
                if constexpr (G == 1)
                    merge_pieces<F::kMergeBatch>(p.partials, kSlotFloats, 0, pf, (int)(pl - pf + 1), first_slot,
                                                 orow, lane);
                else if constexpr (G == 8) {  // g <= 8: heads 0 .. min(g, 4) - 1, then 4 .. g - 1
                    merge_group<2, 4, 8>(p.partials, pf, (int)(pl - pf + 1), first_slot, orow, lane, 0,
                                         min(g_rows, 4));
                    if (g_rows > 4)
                        merge_group<2, 4, 8>(p.partials, pf, (int)(pl - pf + 1), first_slot, orow, lane, 4,
                                             g_rows - 4);
                } else if constexpr (!kTiles)
                    merge_group<8 / G, G>(p.partials, pf, (int)(pl - pf + 1), first_slot, orow, lane, 0, g_rows);
            }
        }
    };
    auto drain = [&](int from) {  // after a timeout: let the copies still in flight land
        for (int y = from; y < ci; y++)
            mbar_wait_bounded(&ws.full[y % kStages], (uint32_t)((y / kStages) & 1), wait_ns);
    };
    auto seg_start = [&](const int4 &m) {
        cur_b = m.x;
        cur_h = m.y;
        seg_c = m.z;
        seg_units = 0;
        if constexpr (kTiles) cs.rows = min(kMqRows, g_rows - kMqRows * (m.y % T));
        else cs.rows = g_rows;
    };

    // chunk 0, unit 0
    if (!mbar_wait_bounded(&ws.full[0], 0u, wait_ns)) {
        if (lane == 0) set_flag(p.status, KVQ_FLAG_TIMEOUT);
        drain(1);
        return;
    }
    int4 mi = *reinterpret_cast<const int4 *>(&ws.meta[0].b);
    float4 mf = *reinterpret_cast<const float4 *>(&ws.meta[0].sk);
    seg_start(mi);
    // a segment's query rows: from its stage, or (kQGlobal) from global memory
    auto q_rows = [&](const int4 &m, int stage) -> const uint16_t * {
        if constexpr (kQGlobal) return p.q + ((int64_t)m.x * H + m.y) * g_rows * kHeadDim;
        else return ws.q[stage];
    };
    cs.load_q(q_rows(mi, 0), lane);
    constexpr int kScores = CS::kScores;  // scores a lane holds per unit
    float sc[kScores];
    uint32_t pf[CS::kPf];
    cs.qk(ws.k[0], lane, sc);
    cs.softmax(sc, min(UT, mi.w), mf.x * p.score_scale, mf.y, lane, pf);

    // One iteration per chunk cc (stage cc % kStages), entered with the
    // chunk's first unit scored (pf) and its units' qk / pv still to run:
    // qk of the next unit is always issued before pv of the current one.
    for (int cc = 0;; cc++) {
        const int s = cc % kStages;
        const float fac = mf.x * p.score_scale;
        const int nh = UPS > 1 ? __float_as_int(mf.w) : 1;
        if (UPS > 1 && nh > 1) {  // the chunk's second unit (int4: the page's second half)
            float sc1[kScores];
            cs.qk(ws.k[s] + kUnitBytes, lane, sc1);
            cs.pv(ws.v[s], pf, lane);
            cs.softmax(sc1, mi.w - UT, fac, mf.y, lane, pf);
        }
        const bool more = cc + 1 < ci;  // chunk cc + 1 was issued before chunk cc was consumed
        int4 mi1 = mi;
        float4 mf1 = mf;
        float sc1[kScores];
        if (more) {
            const int s1 = (cc + 1) % kStages;
            if (!mbar_wait_bounded(&ws.full[s1], (uint32_t)(((cc + 1) / kStages) & 1), wait_ns)) {
                if (lane == 0) set_flag(p.status, KVQ_FLAG_TIMEOUT);
                drain(cc + 2);
                return;
            }
            mi1 = *reinterpret_cast<const int4 *>(&ws.meta[s1].b);
            mf1 = *reinterpret_cast<const float4 *>(&ws.meta[s1].sk);
            if (__float_as_int(mf1.z)) cs.load_q(q_rows(mi1, s1), lane);
            cs.qk(ws.k[s1], lane, sc1);  // the next chunk's first unit: independent of the pv below
        }
        cs.pv(ws.v[s] + (nh - 1) * kUnitBytes, pf, lane);  // the chunk's last unit
        seg_units += nh;
        __syncwarp();  // every lane is done with stage s: refill it
        if (!issue_done) issue();
        if (!more) break;
        if (__float_as_int(mf1.z)) {  // the next chunk starts a new segment
            flush(cur_b, cur_h, seg_c, seg_units);
            cs.reset();
            seg_start(mi1);
        }
        cs.softmax(sc1, min(UT, mi1.w), mf1.x * p.score_scale, mf1.y, lane, pf);
        mi = mi1;
        mf = mf1;
    }
    flush(cur_b, cur_h, seg_c, seg_units);
}

// Second launch of the tile path: merges the split partials of every
// (sequence, unit head) that the split cut into pieces, one warp per query row
// of the tile (the split kernel wrote every other output itself).  Launched
// right after the split kernel with programmatic dependent launch: the
// prologue (lengths, unit prefix, split geometry -- the same values the split
// computed) overlaps the split's tail; partials are read after the wait.
constexpr int kMergeWarps = 16;  // warps of a merge CTA; each merges query rows warp, warp + 16, ...

template <int UT, int kRowsPerHead>
__global__ void __launch_bounds__(kMergeWarps * 32) decode_tile_merge_kernel(DecodeParams p, int grid_workers)
{
    __shared__ int32_t s_cu[kMaxSeqsPerLaunch + 1];
    __shared__ int32_t s_len[kMaxSeqsPerLaunch];
    __shared__ Split s_split;
    const int T = p.tiles, H = p.num_heads, HU = H * T;
    const int split_warps = grid_workers / T;  // the split kernel's pieces per tile
    pdl_launch_dependents();
    decode_prologue<UT>(p, H, split_warps, s_cu, s_len, &s_split);
    pdl_wait();
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int b = (int)(blockIdx.x / HU), h = (int)(blockIdx.x - (unsigned)b * HU);
    const Split &sp = s_split;
    const int n = units_of(s_len[b], UT);
    if (n == 0) return;
    const int hc = h / T, tile = h - hc * T;
    const int64_t u0 = s_cu[b] + (int64_t)hc * n;  // the units of one tile
    const int64_t pf = sp.piece_of(u0), pl = sp.piece_of(u0 + n - 1);
    if (pf == pl) return;  // inside one piece: the split kernel wrote the rows
    const int rows = min(kRowsPerHead, p.group - kRowsPerHead * tile);
    const int first_slot = sp.start(pf) != u0 ? 1 : 0;
    const int64_t slot_floats = (int64_t)kRowsPerHead * kPartialStride;
    const float *tile_partials = p.partials + (int64_t)tile * split_warps * 2 * slot_floats;
    for (int r = warp; r < rows; r += kMergeWarps) {
        uint16_t *orow = p.out + (((int64_t)b * H + hc) * p.group + kRowsPerHead * tile + r) * kHeadDim;
        merge_pieces<16>(tile_partials, slot_floats, r, pf, (int)(pl - pf + 1), first_slot, orow, lane);
    }
}

template <int FMT, int G>
static int ctas_per_sm()
{
    static int cached[64] = {0};
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return 0;
    if (cached[dev] == 0) {
        if (cudaFuncSetAttribute(decode_split_kernel<FMT, G>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 (int)dec_smem_bytes<FMT, G>()) != cudaSuccess)
            return 0;
        if constexpr (G == 1)
            if (cudaFuncSetAttribute(decode_split_kernel<FMT, 1, true>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                     (int)dec_smem_bytes<FMT, 1>()) != cudaSuccess)
                return 0;
        int n = 0;
        if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, decode_split_kernel<FMT, G>,
                                                          DecShape<FMT, G>::kWarps * 32,
                                                          dec_smem_bytes<FMT, G>()) != cudaSuccess)
            return 0;
        constexpr int cap = DecFmt<FMT>::kCtasPerSm;
        cached[dev] = n < 1 ? 1 : (n > cap ? cap : n);
    }
    return cached[dev];
}

// the kernel variant (template group value) that serves group size g
static int kernel_group(int fmt, int g)
{
    if (g == 1) return 1;
    // int4: the column kernels serve every g up to their width (columns past g carry zero queries)
    if (fmt == KVQ_INT4_B64 && g == 2) return 2;
    if (fmt == KVQ_INT4_B64 && g <= 4) return 4;
    if (g <= 8) return 8;  // int4: 5 .. 8; int8 / FP8: 2 .. 8
    return kMqG;
}

// CTAs per SM of the variant (resolving its occupancy query and attributes), 0 on error
template <int FMT>
static int variant_ctas(int kg)
{
    switch (kg) {
    case 1: return ctas_per_sm<FMT, 1>();
    case kMqG: return ctas_per_sm<FMT, kMqG>();
    case 8: return ctas_per_sm<FMT, 8>();
    default: break;
    }
    if constexpr (FMT == KVQ_INT4_B64) {
        if (kg == 2) return ctas_per_sm<FMT, 2>();
        if (kg == 4) return ctas_per_sm<FMT, 4>();
    }
    return 0;
}

static int variant_warps(int fmt, int kg)
{
    if (kg == kMqG) return DecShape<KVQ_INT4_B64, kMqG>::kWarps;
    if (kg == 8) return DecShape<KVQ_INT4_B64, 8>::kWarps;
    return fmt == KVQ_INT4_B64 ? DecFmt<KVQ_INT4_B64>::kWarps : DecFmt<KVQ_INT8_PAGE>::kWarps;
}

static int sm_count()
{
    int dev = 0, sms = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return 0;
    if (cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) return 0;
    return sms;
}

int decode_grid_warps(int fmt, int group)
{
    const int kg = kernel_group(fmt, group);
    int ctas = 0;
    if (fmt == KVQ_INT4_B64) ctas = variant_ctas<KVQ_INT4_B64>(kg);
    else if (fmt == KVQ_FP8_E4M3) ctas = variant_ctas<KVQ_FP8_E4M3>(kg);
    else ctas = variant_ctas<KVQ_INT8_PAGE>(kg);
    return sm_count() * ctas * variant_warps(fmt, kg);
}

bool decode_group_supported(int fmt, int group)
{
    (void)fmt;
    return group >= 1 && group <= kMaxDecodeGroup;
}

int decode_prepare(int fmt, int group)
{
    if (!decode_group_supported(fmt, group)) return 0;
    const int kg = kernel_group(fmt, group);
    if (fmt == KVQ_INT4_B64) return variant_ctas<KVQ_INT4_B64>(kg);
    if (fmt == KVQ_FP8_E4M3) return variant_ctas<KVQ_FP8_E4M3>(kg);
    return variant_ctas<KVQ_INT8_PAGE>(kg);
}

size_t decode_counter_bytes()
{
    int dev = 0, sms = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return 0;
    if (cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) return 0;
    const size_t words = (size_t)sms * kMaxDecodeWarpsPerSm;
    return (words * sizeof(unsigned long long) + 255) / 256 * 256;
}

size_t decode_workspace_bytes(int fmt, int group)
{
    if (!decode_group_supported(fmt, group)) return 0;
    const int gw = decode_grid_warps(fmt, group);
    if (gw <= 0) return 0;
    static_assert(DecFmt<KVQ_INT4_B64>::kWarps * DecFmt<KVQ_INT4_B64>::kCtasPerSm <= kMaxDecodeWarpsPerSm &&
                      DecFmt<KVQ_INT8_PAGE>::kWarps * DecFmt<KVQ_INT8_PAGE>::kCtasPerSm <= kMaxDecodeWarpsPerSm &&
                      DecShape<KVQ_INT4_B64, kMqG>::kWarps * DecFmt<KVQ_INT4_B64>::kCtasPerSm <= kMaxDecodeWarpsPerSm &&
                      DecShape<KVQ_INT4_B64, 8>::kWarps * DecFmt<KVQ_INT4_B64>::kCtasPerSm <= kMaxDecodeWarpsPerSm,
                  "the counter region holds kMaxDecodeWarpsPerSm warps per SM");
    const size_t counters = decode_counter_bytes();
    if (counters == 0) return 0;
    const int kg = kernel_group(fmt, group);
    const int rows = kg == kMqG ? kMqRows : kg;  // query rows of one partial: the kernel's, not g
    const size_t partial = (size_t)gw * 2 * rows * kPartialStride * sizeof(float);
    return counters + partial;
}

unsigned long long decode_next_epoch()
{
    // splitmix64's output function over a call counter, forced odd, 40 bits:
    // epochs of different calls differ in their low bits only by chance
    static std::atomic<unsigned long long> calls{0};
    unsigned long long z = (calls.fetch_add(1, std::memory_order_relaxed) + 1) * 0x9e3779b97f4a7c15ull;
    z = (z ^ (z >> 30)) * 0xbf58476d1ce4e5b9ull;
    z = (z ^ (z >> 27)) * 0x94d049bb133111ebull;
    z ^= z >> 31;
    return (z | 1ull) & ((1ull << 40) - 1);
}

template <int FMT>
static cudaError_t launch_variant(const DecodeParams &p0, int kg, int gw, cudaStream_t s)
{
    DecodeParams p = p0;
    const dim3 grid(gw / variant_warps(FMT, kg));
    if (kg == kMqG) {
        p.tiles = (p.group + kMqRows - 1) / kMqRows;
        if (gw / p.tiles < 1) return cudaErrorInvalidDevice;  // every tile needs a warp per piece
        if (ctas_per_sm<FMT, kMqG>() < 1) return cudaErrorInvalidDevice;  // also sets the smem attribute
        cudaError_t e = launch_pdl(decode_split_kernel<FMT, kMqG>, grid, dim3(variant_warps(FMT, kg) * 32),
                                   dec_smem_bytes<FMT, kMqG>(), s, p, gw);
        if (e != cudaSuccess) return e;
        const unsigned pairs = (unsigned)p.num_seqs * (unsigned)(p.num_heads * p.tiles);
        if (pairs == 0) return cudaSuccess;
        return launch_pdl(decode_tile_merge_kernel<DecFmt<FMT>::kUnitTok, kMqRows>, dim3(pairs),
                          dim3(kMergeWarps * 32), 0, s, p, gw);
    }
    p.tiles = 1;
    const dim3 block(variant_warps(FMT, kg) * 32);
    if (kg == 1) {
        const bool hook = p.test_skip_chunk >= 0 || p.wait_limit_ns != kWaitLimitNs;
        return launch_pdl(hook ? decode_split_kernel<FMT, 1, true> : decode_split_kernel<FMT, 1, false>, grid, block,
                          dec_smem_bytes<FMT, 1>(), s, p, gw);
    }
    if constexpr (FMT == KVQ_INT4_B64) {
        if (kg == 2) {
            if (ctas_per_sm<FMT, 2>() < 1) return cudaErrorInvalidDevice;
            return launch_pdl(decode_split_kernel<FMT, 2>, grid, block, dec_smem_bytes<FMT, 2>(), s, p, gw);
        }
        if (kg == 4) {
            if (ctas_per_sm<FMT, 4>() < 1) return cudaErrorInvalidDevice;
            return launch_pdl(decode_split_kernel<FMT, 4>, grid, block, dec_smem_bytes<FMT, 4>(), s, p, gw);
        }
    }
    if (kg == 8) {
        if (ctas_per_sm<FMT, 8>() < 1) return cudaErrorInvalidDevice;
        return launch_pdl(decode_split_kernel<FMT, 8>, grid, block, dec_smem_bytes<FMT, 8>(), s, p, gw);
    }
    return cudaErrorInvalidValue;
}

cudaError_t launch_decode(int fmt, const DecodeParams &p, cudaStream_t s)
{
    if (!decode_group_supported(fmt, p.group)) return cudaErrorInvalidValue;
    const int gw = decode_grid_warps(fmt, p.group);
    if (gw <= 0) return cudaErrorInvalidDevice;
    static_assert(DecFmt<KVQ_INT4_B64>::kWarps == DecFmt<KVQ_INT8_PAGE>::kWarps &&
                  DecFmt<KVQ_FP8_E4M3>::kWarps == DecFmt<KVQ_INT8_PAGE>::kWarps, "one CTA size");
    const int kg = kernel_group(fmt, p.group);
    // A small problem launches only the CTAs its units can keep busy: every sequence at the
    // block table's full width bounds the units of a unit head, and the kernel gives each
    // active warp at least kMinUnitsPerWarp of them (the rest of a full grid would only run
    // the prologue).  Large problems keep the whole persistent grid.
    const int wpc = variant_warps(fmt, kg);
    const int64_t tiles = kg == kMqG ? (p.group + kMqRows - 1) / kMqRows : 1;
    const int64_t upp = fmt == KVQ_INT4_B64 ? DecFmt<KVQ_INT4_B64>::kUnitsPerPage : DecFmt<KVQ_INT8_PAGE>::kUnitsPerPage;
    const int64_t units_max = (int64_t)p.num_seqs * p.num_heads * p.max_blocks * upp;
    const int64_t need = tiles * ((units_max + kMinUnitsPerWarp - 1) / kMinUnitsPerWarp);
    int gwl = gw;
    if (need < gw) gwl = (int)(need < wpc ? wpc : (need + wpc - 1) / wpc * wpc);
    if (fmt == KVQ_INT4_B64) return launch_variant<KVQ_INT4_B64>(p, kg, gwl, s);
    if (fmt == KVQ_FP8_E4M3) return launch_variant<KVQ_FP8_E4M3>(p, kg, gwl, s);
    return launch_variant<KVQ_INT8_PAGE>(p, kg, gwl, s);
}

}  // namespace kvq
