// kvq_quantize.cu -- fused absmax + quantize + pack of 64-token blocks
// (quantize_block, jsqmd.com/news/887038 section 2.1; INT8 per-chunk variant,
// aicoding.csdn.net section 2.2; FP8 E4M3 with the scale set by max|x|,
// jsqmd.com/news/887038 section 2.2), for a contiguous tensor and for appends
// into the paged cache.
//
// One warp owns one (block, head): 64 rows x 128 fp16 = 16 KiB.  Its lanes
// stage the rows in shared memory with 16-byte cp.async copies (lane = row
// parity x 16-byte chunk, so each warp copy covers two whole 256-byte rows;
// rows past the end are zero-filled), reduce max|x| with packed half2 max and
// one warp redux, then quantize from shared memory and store whole rows of
// codes.  The pages' two-pass design (an extrema pass, then an elementwise
// kernel) becomes one pass over HBM.
//
// Exactness: the code must equal clamp(rint(RN(x / scale))).  The fast path
// multiplies by r = RN(1 / scale); |RN(x*r) - RN(x/scale)| < 1.5 * 2^-23 * |y|,
// so the rounded integer can differ only when y lies within that distance of a
// half-integer.  Any group of 8 elements with |y - rint(y)| > 1/2 - eps
// (eps = 2^-17 for int4, |y| <= 8; 2^-14 for int8, |y| <= 128) is recomputed
// with the correctly rounded division __fdiv_rn.  Bounds: |x| <= a, so
// |y| <= 7.5 (1 + 2^-22) for int4 -- only the upper clamp at 7 can act
// (rint(-7.5) = -8 already), and only when y >= 7.5, which the tie test above
// always sends to the exact path, so the fast path needs no clamp -- and
// |y| <= 127 (1 + 2^-22) for int8, where rint never leaves [-127, 127].
//
// FP8 E4M3: code = E4M3(RN(x / scale)), nearest with ties to the even
// fraction, saturating, by the hardware conversion.  The fast path converts
// y' (1 - 2^-21) and y' (1 + 2^-21) for y' = RN(x * r): RN(x / scale) lies
// between them (|y' - RN(x / scale)| < 1.5 * 2^-23 |y|), the conversion is
// monotone, so equal codes are the code; a group of 8 in which some pair's two
// ends differ (y near a midpoint of the E4M3 grid) takes the correctly rounded
// division for all 8 (one branch per group instead of one per pair).
#include "kvq_device.cuh"
#include "kvq_internal.h"

namespace kvq {

template <int FMT>
struct Codec;

template <>
struct Codec<KVQ_INT4_B64> {
    static constexpr int kRowBytes = 64;
    static constexpr float kDiv = 7.5f;
    static constexpr float kMagic = 12582920.0f;       // 1.5 * 2^23 + 8: low nibble = code + 8
    static constexpr float kEps = 7.62939453125e-06f;  // 2^-17
};

template <>
struct Codec<KVQ_INT8_PAGE> {
    static constexpr int kRowBytes = 128;
    static constexpr float kDiv = 127.0f;
    static constexpr float kMagic = 12583040.0f;       // 1.5 * 2^23 + 128: low byte = code + 128
    static constexpr float kEps = 6.103515625e-05f;    // 2^-14
};

template <>
struct Codec<KVQ_FP8_E4M3> {
    static constexpr int kRowBytes = 128;
    static constexpr float kDiv = 448.0f;  // the largest finite E4M3 value
};

constexpr uint32_t kMagicBits = 0x4b400000u;  // bits of 1.5 * 2^23

// two binary32 values -> two E4M3 codes, x0 in the low byte (round to nearest
// even, saturating at +-448; the sign of a zero result is kept)
__device__ __forceinline__ uint32_t e4m3x2_rn(float x0, float x1)
{
    uint16_t d;
    asm("cvt.rn.satfinite.e4m3x2.f32 %0, %1, %2;" : "=h"(d) : "f"(x1), "f"(x0));
    return d;
}

// 8 fp16 values -> 8 E4M3 codes, element j in byte j; rr = (r, r), r = RN(1 / scale)
__device__ __forceinline__ uint2 quant8_fp8(const uint4 &v, uint64_t rr, float scale)
{
    if (scale == 0.0f) return make_uint2(0u, 0u);  // all-zero block: codes 0x00 (also for -0.0)
    const uint32_t w[4] = {v.x, v.y, v.z, v.w};
    const uint64_t dn = pk2(1.0f - 0x1p-21f, 1.0f - 0x1p-21f), up = pk2(1.0f + 0x1p-21f, 1.0f + 0x1p-21f);
    uint32_t c[4], diff = 0u;
#pragma unroll
    for (int i = 0; i < 4; i++) {
        const float2 f = __half22float2(*reinterpret_cast<const __half2 *>(&w[i]));
        const uint64_t y = mul2(pk2(f.x, f.y), rr);
        float a0, a1, b0, b1;
        upk2(mul2(y, dn), a0, a1);
        upk2(mul2(y, up), b0, b1);
        c[i] = e4m3x2_rn(a0, a1);
        diff |= c[i] ^ e4m3x2_rn(b0, b1);
    }
    if (diff != 0u) {  // some pair of the 8 brackets a grid midpoint: the whole group divides exactly
#pragma unroll
        for (int i = 0; i < 4; i++) {
            const float2 f = __half22float2(*reinterpret_cast<const __half2 *>(&w[i]));
            c[i] = e4m3x2_rn(__fdiv_rn(f.x, scale), __fdiv_rn(f.y, scale));
        }
    }
    return make_uint2(c[0] | (c[1] << 16), c[2] | (c[3] << 16));
}

// fast path for 8 fp16 values: m[j] = bits of RN(RN(x_j * r) + kMagic), and
// tmax = max(tmax, |y_j - rint(y_j)|) over them
template <int FMT>
__device__ __forceinline__ void quant8_fast(const uint4 &v, uint64_t rr, uint32_t m[8], float &tmax)
{
    using C = Codec<FMT>;
    const uint32_t w[4] = {v.x, v.y, v.z, v.w};
    const uint64_t magic = pk2(C::kMagic, C::kMagic);
#pragma unroll
    for (int i = 0; i < 4; i++) {
        const float2 f = __half22float2(*reinterpret_cast<const __half2 *>(&w[i]));
        const uint64_t y = mul2(pk2(f.x, f.y), rr);
        const uint64_t mf = add2(y, magic);
        const uint64_t d = sub2(y, sub2(mf, magic));  // y - rint(y), exact
        float m0, m1, d0, d1;
        upk2(mf, m0, m1);
        upk2(d, d0, d1);
        tmax = fmaxf(tmax, fmaxf(fabsf(d0), fabsf(d1)));
        m[2 * i] = __float_as_uint(m0);
        m[2 * i + 1] = __float_as_uint(m1);
    }
}

// exact path for a group of 8 that has a near-tie: per element, keep the fast
// value unless the element itself is within eps of a half-integer; then an
// element equal to +-a takes the block's precomputed code (+-ya = RN(a / scale),
// so the whole block needs one division for its extreme elements), any other
// takes the correctly rounded quotient.  Codes are clamped here (int4: y may
// reach 7.5 only in this path).
template <int FMT>
__device__ __forceinline__ void quant8_exact(const uint4 &v, uint64_t rr, float scale, float a, float ya,
                                             uint32_t m[8])
{
    using C = Codec<FMT>;
    const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
    for (int i = 0; i < 4; i++) {
        const float2 f = __half22float2(*reinterpret_cast<const __half2 *>(&w[i]));
        const float xs[2] = {f.x, f.y};
#pragma unroll
        for (int e = 0; e < 2; e++) {
            const float x = xs[e];
            const float y0 = __fmul_rn(x, __uint_as_float((uint32_t)rr));
            const float d = y0 - (__fadd_rn(y0, C::kMagic) - C::kMagic);
            if (fabsf(d) > 0.5f - C::kEps) {
                float y = fabsf(x) == a ? copysignf(ya, x) : __fdiv_rn(x, scale);
                if constexpr (FMT == KVQ_INT4_B64) y = fminf(y, 7.0f);
                m[2 * i + e] = __float_as_uint(__fadd_rn(y, C::kMagic));
            }
        }
    }
}

// 8 codes -> one word of 4-bit two's-complement nibbles, element j at bits 4j.
// m[j] = kMagicBits + (code + 8): Horner in base 16 with integer multiply-adds,
// minus the accumulated magic, then flip each nibble's top bit.
__device__ __forceinline__ uint32_t pack8_int4(const uint32_t m[8])
{
    constexpr uint32_t kBias = kMagicBits * 0x11111111u;  // sum_j kMagicBits * 16^j mod 2^32
    uint32_t acc = m[7];
#pragma unroll
    for (int j = 6; j >= 0; j--) acc = acc * 16u + m[j];
    return (acc - kBias) ^ 0x88888888u;
}

// 8 codes -> two words of two's-complement bytes; m[j] = kMagicBits + (code + 128)
__device__ __forceinline__ uint2 pack8_int8(const uint32_t m[8])
{
    constexpr uint32_t kBias = kMagicBits * 0x01010101u;
    uint32_t lo = m[3], hi = m[7];
#pragma unroll
    for (int j = 2; j >= 0; j--) {
        lo = lo * 256u + m[j];
        hi = hi * 256u + m[4 + j];
    }
    return make_uint2((lo - kBias) ^ 0x80808080u, (hi - kBias) ^ 0x80808080u);
}

// quantize 8 consecutive elements of one row and store their codes at dst
// (4 bytes int4, 8 bytes int8 / FP8).  rr = (r, r), r = RN(1 / scale); a, ya:
// the block's max|x| and RN(a / scale) (integer formats' exact path)
template <int FMT>
__device__ __forceinline__ void store8(const uint4 &v, uint64_t rr, float scale, float a, float ya, uint8_t *dst)
{
    using C = Codec<FMT>;
    if constexpr (FMT == KVQ_FP8_E4M3) {
        *reinterpret_cast<uint2 *>(dst) = quant8_fp8(v, rr, scale);
    } else {
        uint32_t m[8];
        float tmax = 0.0f;
        quant8_fast<FMT>(v, rr, m, tmax);
        if (tmax > 0.5f - C::kEps) quant8_exact<FMT>(v, rr, scale, a, ya, m);  // a near-tie (rare)
        if constexpr (FMT == KVQ_INT4_B64)
            *reinterpret_cast<uint32_t *>(dst) = pack8_int4(m);
        else
            *reinterpret_cast<uint2 *>(dst) = pack8_int8(m);
    }
}

__device__ __forceinline__ void cp_async16(uint32_t dst, const void *src, uint32_t src_bytes)
{
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;" ::"r"(dst), "l"(src), "r"(src_bytes) : "memory");
}

// Row sources of one (block, head) for the contiguous layout x[T][H][D].
struct ContigRows {
    const uint16_t *base;  // row 0 of the block, head h
    int64_t stride;        // elements between rows (H * D)
    // copy rows 2i + rpar (i < npairs) of this lane's 16-byte chunk; rows >= nrows are zero-filled
    __device__ __forceinline__ void stage(uint32_t s0, int chunk, int rpar, int nrows, int npairs) const
    {
        const uint16_t *src = base + rpar * stride + 8 * chunk;
        const uint16_t *valid = base + 8 * chunk;
#pragma unroll 8
        for (int i = 0; i < npairs; i++, src += 2 * stride) {
            const bool live = 2 * i + rpar < nrows;
            cp_async16(s0 + (uint32_t)i * (2 * kHeadDim * 2), live ? src : valid, live ? 16u : 0u);
        }
    }
};

// Row sources of one (block, head) of an append: rows before n_old come from
// the fp16 tail buffer, later rows from the new tokens.
struct AppendRows {
    const uint16_t *tail;   // tail[b][h] row 0, or nullptr
    const uint16_t *fresh;  // head h of new-token row 0
    int64_t row0;           // new-token row that would land in block row 0 (negative when n_old > 0)
    int n_old;
    int64_t stride;         // elements between new-token rows (H * D)
    __device__ __forceinline__ void stage(uint32_t s0, int chunk, int rpar, int nrows, int npairs) const
    {
        int i = 0;
        for (; 2 * i + rpar < n_old; i++)  // old rows of the open block
            cp_async16(s0 + (uint32_t)i * (2 * kHeadDim * 2), tail + (2 * i + rpar) * kHeadDim + 8 * chunk, 16u);
        const uint16_t *src = fresh + (row0 + 2 * i + rpar) * stride + 8 * chunk;
        const uint16_t *valid = fresh + (row0 + n_old) * stride + 8 * chunk;  // first new row
        for (; i < npairs; i++, src += 2 * stride) {
            const bool live = 2 * i + rpar < nrows;
            cp_async16(s0 + (uint32_t)i * (2 * kHeadDim * 2), live ? src : valid, live ? 16u : 0u);
        }
    }
};

// One warp per CTA with its 16 KiB of staging in dynamic shared memory: a CTA's
// staging is free again the moment its block is done, and up to 13 CTAs fit on
// an SM (16 KiB + the 1 KiB the hardware keeps per CTA).  Three-warp CTAs (the
// 48 KiB static limit, 12 warps per SM) measured 1.03 ms on the 5.4 GB long
// append against 0.90 ms; seven- and fourteen-warp CTAs (14 warps per SM) 1.07
// and 1.27 ms -- a CTA's slot waits for its slowest block.
constexpr int kQuantWarps = 1;
constexpr int kBlockElems = kPage * kHeadDim;  // fp16 elements of one (block, head)
constexpr size_t kStageBytes = (size_t)kQuantWarps * kBlockElems * 2;  // dynamic shared memory per CTA

// One (block, head): stage, reduce, quantize, store.  sbuf: 16 KiB of this
// warp's shared memory.  Only the lane that staged a 16-byte chunk reads it
// back, so no cross-lane ordering is needed beyond cp.async's own wait.
// nrows >= 1 (the first valid row is the source address of the zero-fill copies).
// Rows 2i + rpar for i < npairs are processed (npairs = 32 writes the whole
// block, rows past nrows as code 0; a smaller npairs leaves rows >= 2 npairs
// untouched, which hold the zeros written when the block was first filled).
template <int FMT, class Rows>
__device__ __forceinline__ void quantize_block_warp(const Rows &rows, int nrows, int npairs, uint16_t *sbuf,
                                                    uint8_t *__restrict__ codes, float *__restrict__ scale_out)
{
    using C = Codec<FMT>;
    const int lane = threadIdx.x & 31;
    const int chunk = lane & 15;  // elements 8*chunk .. 8*chunk+7 of a row
    const int rpar = lane >> 4;   // rows 2i + rpar
    const uint32_t s0 = smem_addr(sbuf) + (uint32_t)(rpar * kHeadDim + 8 * chunk) * 2u;
    rows.stage(s0, chunk, rpar, nrows, npairs);
    asm volatile("cp.async.commit_group;\n\tcp.async.wait_group 0;" ::: "memory");

    const uint4 *sv = reinterpret_cast<const uint4 *>(sbuf + rpar * kHeadDim + 8 * chunk);
    constexpr int kStep = 2 * kHeadDim / 8;  // uint4 between rows 2i and 2i + 2
    __half2 mx = __float2half2_rn(0.0f);
#pragma unroll 8
    for (int i = 0; i < npairs; i++) {
        const uint4 v = sv[i * kStep];
        mx = __hmax2(mx, __habs2(*reinterpret_cast<const __half2 *>(&v.x)));
        mx = __hmax2(mx, __habs2(*reinterpret_cast<const __half2 *>(&v.y)));
        mx = __hmax2(mx, __habs2(*reinterpret_cast<const __half2 *>(&v.z)));
        mx = __hmax2(mx, __habs2(*reinterpret_cast<const __half2 *>(&v.w)));
    }
    const uint32_t mb = *reinterpret_cast<const uint32_t *>(&mx);
    uint32_t abits = max(mb & 0xffffu, mb >> 16);  // non-negative fp16: bit order = value order
    abits = __reduce_max_sync(kFull, abits);
    const float a = __half2float(__ushort_as_half(static_cast<unsigned short>(abits)));
    const float scale = __fdiv_rn(a, C::kDiv);
    if (lane == 0) *scale_out = scale;
    // rows past nrows are zero in shared memory and quantize to code 0; an
    // all-zero block has scale 0 and r = 0, so every code is 0 there too
    const float r = scale > 0.0f ? __frcp_rn(scale) : 0.0f;
    const float ya = scale > 0.0f ? __fdiv_rn(a, scale) : 0.0f;  // the quotient of the extreme elements
    const uint64_t rr = pk2(r, r);
    uint8_t *out = codes + rpar * C::kRowBytes + (FMT == KVQ_INT4_B64 ? 4 : 8) * chunk;
#pragma unroll 4
    for (int i = 0; i < npairs; i++) {  // rows 2i + rpar
        store8<FMT>(sv[i * kStep], rr, scale, a, ya, out + i * 2 * C::kRowBytes);
    }
}

template <int FMT>
__global__ void __launch_bounds__(kQuantWarps * 32)
    quantize_contig_kernel(const uint16_t *__restrict__ x, int64_t T, int H, int64_t nblocks,
                           uint8_t *__restrict__ codes, float *__restrict__ scales)
{
    using C = Codec<FMT>;
    extern __shared__ __align__(128) uint16_t sbuf_q[];
    uint16_t(*sbuf)[kBlockElems] = reinterpret_cast<uint16_t(*)[kBlockElems]>(sbuf_q);
    pdl_launch_dependents();
    pdl_wait();
    const int warp = threadIdx.x >> 5;
    const int64_t w = (int64_t)blockIdx.x * kQuantWarps + warp;
    if (w >= nblocks * H) return;
    const int64_t j = w / H;
    const int h = (int)(w % H);
    const int64_t rem = T - j * kPage;
    const int nrows = rem < kPage ? (int)rem : kPage;
    ContigRows rows{x + (j * kPage * H + h) * kHeadDim, (int64_t)H * kHeadDim};
    quantize_block_warp<FMT>(rows, nrows, 32, sbuf[warp], codes + (j * H + h) * (int64_t)kPage * C::kRowBytes,
                             scales + j * H + h);
}

// grid: x over (touched block, head) of one sequence, y = sequence, z = 0 keys / 1 values
template <int FMT>
__global__ void __launch_bounds__(kQuantWarps * 32)
    append_kernel(AppendParams p)
{
    using C = Codec<FMT>;
    extern __shared__ __align__(128) uint16_t sbuf_a[];
    uint16_t(*sbuf)[kBlockElems] = reinterpret_cast<uint16_t(*)[kBlockElems]>(sbuf_a);
    pdl_launch_dependents();
    pdl_wait();
    const int b = blockIdx.y;
    const bool is_v = blockIdx.z != 0;
    const int H = p.num_heads;
    const int warp = threadIdx.x >> 5;
    const int wi = blockIdx.x * kQuantWarps + warp;
    const int lane = threadIdx.x & 31;
    const int c0 = p.cu_seqlens[b];
    const int T = p.cu_seqlens[b + 1] - c0;
    const int L0 = p.seq_lens_before[b];
    if (T < 0 || T > p.max_new_tokens || c0 < 0 || (int64_t)c0 + T > p.total_new) {
        if (wi == 0 && lane == 0 && !is_v) set_flag(p.status, KVQ_FLAG_BAD_APPEND);
        return;
    }
    if (T == 0) return;
    const int L1 = L0 + T;
    if (L0 < 0 || (int64_t)L1 > (int64_t)p.max_blocks * kPage) {
        if (wi == 0 && lane == 0 && !is_v) set_flag(p.status, KVQ_FLAG_BAD_LENGTH);
        return;
    }
    const int j0 = L0 / kPage;
    const int j1 = (L1 - 1) / kPage;
    const int jrel = wi / H;
    const int h = wi % H;
    if (jrel > j1 - j0) return;
    const int j = j0 + jrel;
    const int64_t HD = (int64_t)H * kHeadDim;
    const uint16_t *src = is_v ? p.v_new : p.k_new;
    uint16_t *tail = is_v ? p.v_tail : p.k_tail;
    uint16_t *tail_bh = tail ? tail + ((int64_t)b * H + h) * kPage * kHeadDim : nullptr;
    const int n_old = (j == j0) ? (L0 - j0 * kPage) : 0;
    if (n_old > 0 && tail_bh == nullptr) {
        if (lane == 0) set_flag(p.status, KVQ_FLAG_NO_TAIL);
        return;
    }
    const int page = p.block_table[(int64_t)b * p.max_blocks + j];
    const bool page_ok = page >= 0 && page < p.num_pages;
    if (!page_ok) {
        if (lane == 0) set_flag(p.status, KVQ_FLAG_BAD_PAGE);
    } else {
        // new token index i = 64*j + r - L0 lives at row (c0 + i) of the new-token tensor
        AppendRows rows{tail_bh, src + (int64_t)h * kHeadDim, (int64_t)c0 + (int64_t)j * kPage - L0, n_old, HD};
        const int nrows = min(kPage, L1 - j * kPage);
        // a block opened by an earlier append already holds zeros past its end
        const int npairs = n_old > 0 ? (nrows + 1) / 2 : 32;
        uint8_t *codes = (is_v ? p.v_codes : p.k_codes) + ((int64_t)page * H + h) * kPage * C::kRowBytes;
        float *scale = (is_v ? p.v_scales : p.k_scales) + (int64_t)page * H + h;
        quantize_block_warp<FMT>(rows, nrows, npairs, sbuf[warp], codes, scale);
    }
    // The warp of the first touched block is the only reader of this (b, h)'s
    // tail, so it also writes the new tail rows: no other warp can race with it.
    if (j == j0 && tail_bh != nullptr && (L1 % kPage) != 0) {
        __syncwarp();
        const int rs = (j1 == j0) ? (L0 - j0 * kPage) : 0;
        const int re = L1 - j1 * kPage;
        const int chunk = lane & 15;
        const int64_t row0 = (int64_t)c0 + (int64_t)j1 * kPage - L0;  // >= c0 for every r >= rs
        const uint16_t *fresh = src + (int64_t)h * kHeadDim;
        for (int r = rs + (lane >> 4); r < re; r += 2) {
            const uint4 val = ld_stream_v4(fresh + (row0 + r) * HD + 8 * chunk);
            *reinterpret_cast<uint4 *>(tail_bh + r * kHeadDim + 8 * chunk) = val;
        }
    }
}

// ---------------------------------------------------------------------------
// Short appends (at most 64 new tokens per sequence, e.g. one decode step):
// one CTA of 4 warps per touched (block, head, K/V); lane (rpar, chunk) of
// warp w holds rows 8 i + 2 w + rpar (i < 8) in registers.
//   1. Load the new rows only and reduce their max|x| -> a_new (one
//      shared-memory exchange), and read the block's stored scale s_old.
//   2. a -> RN(a / d) is strictly increasing on binary16 magnitudes, so
//      RN(a_new / d) <= s_old exactly when the block's max|x| does not move:
//      then the scale is s_old and the old rows' codes, a function of
//      (x, scale) alone, are already in the cache -- only the new rows are
//      quantized, and the fp16 tail is never read.
//   3. Otherwise a_new is the block's max|x|: the old rows are loaded from the
//      tail and every row is re-quantized with the new scale.
// ---------------------------------------------------------------------------
constexpr int kShortWarps = 4;
constexpr int kShortRounds = kPage / (2 * kShortWarps);

template <int FMT>
__global__ void __launch_bounds__(kShortWarps * 32)
    append_short_kernel(AppendParams p)
{
    using C = Codec<FMT>;
    __shared__ uint32_t s_max[kShortWarps];
    pdl_launch_dependents();
    // Until pdl_wait below, the previous kernel of the stream may still be
    // running: only cu_seqlens, seq_lens_before and the block table are read
    // before it (no kernel of this library writes them); the scales, codes,
    // tail and new rows are touched after it.
    const int b = blockIdx.y;
    const bool is_v = blockIdx.z != 0;
    const int H = p.num_heads;
    const int tid = threadIdx.x;
    const int warp = tid >> 5;
    const int lane = tid & 31;
    const bool leader = blockIdx.x == 0 && tid == 0 && !is_v;
    const int c0 = p.cu_seqlens[b];
    const int T = p.cu_seqlens[b + 1] - c0;
    const int L0 = p.seq_lens_before[b];
    if (T < 0 || T > p.max_new_tokens || c0 < 0 || (int64_t)c0 + T > p.total_new) {
        if (leader) set_flag(p.status, KVQ_FLAG_BAD_APPEND);
        return;
    }
    if (T == 0) return;
    const int L1 = L0 + T;
    if (L0 < 0 || (int64_t)L1 > (int64_t)p.max_blocks * kPage) {
        if (leader) set_flag(p.status, KVQ_FLAG_BAD_LENGTH);
        return;
    }
    const int j0 = L0 / kPage;
    const int j1 = (L1 - 1) / kPage;
    const int jrel = blockIdx.x / H;
    const int h = blockIdx.x % H;
    if (jrel > j1 - j0) return;
    const int j = j0 + jrel;
    const int page = p.block_table[(int64_t)b * p.max_blocks + j];
    pdl_wait();  // from here on, the previous kernel's writes are visible
    const int64_t HD = (int64_t)H * kHeadDim;
    const uint16_t *fresh = (is_v ? p.v_new : p.k_new) + (int64_t)h * kHeadDim;
    uint16_t *tail = is_v ? p.v_tail : p.k_tail;
    uint16_t *tail_bh = tail ? tail + ((int64_t)b * H + h) * kPage * kHeadDim : nullptr;
    const int n_old = (j == j0) ? (L0 - j0 * kPage) : 0;
    if (n_old > 0 && tail_bh == nullptr) {
        if (tid == 0) set_flag(p.status, KVQ_FLAG_NO_TAIL);
        return;
    }
    const bool page_ok = page >= 0 && page < p.num_pages;
    if (!page_ok && tid == 0) set_flag(p.status, KVQ_FLAG_BAD_PAGE);
    const int64_t pg = page_ok ? page : 0;
    float *scale_ptr = (is_v ? p.v_scales : p.k_scales) + pg * H + h;
    const float s_old = (n_old > 0 && page_ok) ? *scale_ptr : -1.0f;

    const int nrows = min(kPage, L1 - j * kPage);
    const int64_t row0 = (int64_t)c0 + (int64_t)j * kPage - L0;  // new-token row of block row 0
    const int chunk = lane & 15;
    const int rbase = 2 * warp + (lane >> 4);
    // 1. the new rows and their max|x|
    uint4 v[kShortRounds];
    __half2 mx = __float2half2_rn(0.0f);
#pragma unroll
    for (int i = 0; i < kShortRounds; i++) {
        const int r = 8 * i + rbase;
        v[i] = make_uint4(0u, 0u, 0u, 0u);
        if (r >= n_old && r < nrows) v[i] = ld_stream_v4(fresh + (row0 + r) * HD + 8 * chunk);
    }
#pragma unroll
    for (int i = 0; i < kShortRounds; i++) {
        mx = __hmax2(mx, __habs2(*reinterpret_cast<const __half2 *>(&v[i].x)));
        mx = __hmax2(mx, __habs2(*reinterpret_cast<const __half2 *>(&v[i].y)));
        mx = __hmax2(mx, __habs2(*reinterpret_cast<const __half2 *>(&v[i].z)));
        mx = __hmax2(mx, __habs2(*reinterpret_cast<const __half2 *>(&v[i].w)));
    }
    const uint32_t mb = *reinterpret_cast<const uint32_t *>(&mx);
    const uint32_t wmax = __reduce_max_sync(kFull, max(mb & 0xffffu, mb >> 16));
    if (lane == 0) s_max[warp] = wmax;
    __syncthreads();
    uint32_t abits = s_max[0];
#pragma unroll
    for (int w = 1; w < kShortWarps; w++) abits = max(abits, s_max[w]);
    const float a_new = __half2float(__ushort_as_half(static_cast<unsigned short>(abits)));
    const float s_new = __fdiv_rn(a_new, C::kDiv);
    // 2./3. keep the scale, or re-quantize the whole block
    const bool keep = n_old > 0 && s_new <= s_old;
    const float scale = keep ? s_old : s_new;
    // the exact path's shortcut for elements equal to +-max|x| needs the
    // block's max, known only when it moved; with the scale kept, every
    // near-tie takes the correctly rounded division instead
    const float a = keep ? INFINITY : a_new;
    const int r_first = keep ? n_old : 0;
    const int R = n_old > 0 ? nrows : kPage;  // rows rewritten (past nrows: code 0)
    if (!keep && n_old > 0) {
#pragma unroll
        for (int i = 0; i < kShortRounds; i++) {
            const int r = 8 * i + rbase;
            if (r < n_old) v[i] = *reinterpret_cast<const uint4 *>(tail_bh + r * kHeadDim + 8 * chunk);
        }
    }
    if (page_ok) {
        if (tid == 0) *scale_ptr = scale;
        const float rcp = scale > 0.0f ? __frcp_rn(scale) : 0.0f;
        const float ya = (scale > 0.0f && !keep) ? __fdiv_rn(a, scale) : 0.0f;
        const uint64_t rr = pk2(rcp, rcp);
        uint8_t *codes = (is_v ? p.v_codes : p.k_codes) + (pg * H + h) * kPage * C::kRowBytes +
                         (FMT == KVQ_INT4_B64 ? 4 : 8) * chunk;
#pragma unroll
        for (int i = 0; i < kShortRounds; i++) {
            const int r = 8 * i + rbase;
            if (r < r_first || r >= R) continue;
            store8<FMT>(v[i], rr, scale, a, ya, codes + r * C::kRowBytes);
        }
    }
    // the CTA of the first touched block is the only reader of this (b, h)'s
    // tail; it writes the rows of the block left open
    if (j == j0 && tail_bh != nullptr && (L1 % kPage) != 0) {
        if (j1 == j0) {  // the open block stays open: its new rows (never read here) are in registers
#pragma unroll
            for (int i = 0; i < kShortRounds; i++) {
                const int r = 8 * i + rbase;
                if (r >= n_old && r < nrows) *reinterpret_cast<uint4 *>(tail_bh + r * kHeadDim + 8 * chunk) = v[i];
            }
        } else {  // a later block is left open: its rows overwrite tail rows read above
            __syncthreads();
            const int re = L1 - j1 * kPage;
            const int64_t row1 = (int64_t)c0 + (int64_t)j1 * kPage - L0;
            for (int e = tid; e < re * 16; e += kShortWarps * 32) {
                const int r = e >> 4, ch = e & 15;
                const uint4 val = ld_stream_v4(fresh + (row1 + r) * HD + 8 * ch);
                *reinterpret_cast<uint4 *>(tail_bh + r * kHeadDim + 8 * ch) = val;
            }
        }
    }
}

// Launch modes, as measured in a decode loop (append, then decode, whose grid
// is one persistent CTA per SM that fills the SM's registers): the short
// append uses programmatic dependent launch -- its CTAs cannot sit beside a
// decode CTA, so they start as the decode grid drains and hide the launch
// latency (about 2 us per step).  Quantize and the long append launch plainly:
// their CTAs placed early delayed the next persistent grid on part of the SMs
// when the decode ran several smaller CTAs per SM.
cudaError_t launch_quantize(int fmt, const uint16_t *x, int64_t T, int H, uint8_t *codes, float *scales,
                            cudaStream_t s)
{
    const int64_t nb = (T + kPage - 1) / kPage;
    const int64_t warps = nb * H;
    const int64_t blocks = (warps + kQuantWarps - 1) / kQuantWarps;
    if (blocks == 0) return cudaSuccess;
    if (blocks > 0x7fffffffLL) return cudaErrorInvalidValue;
    const dim3 grid((unsigned)blocks), block(kQuantWarps * 32);
    if (fmt == KVQ_INT4_B64)
        return launch_plain(quantize_contig_kernel<KVQ_INT4_B64>, grid, block, kStageBytes, s, x, T, H, nb, codes,
                            scales);
    if (fmt == KVQ_FP8_E4M3)
        return launch_plain(quantize_contig_kernel<KVQ_FP8_E4M3>, grid, block, kStageBytes, s, x, T, H, nb, codes,
                            scales);
    return launch_plain(quantize_contig_kernel<KVQ_INT8_PAGE>, grid, block, kStageBytes, s, x, T, H, nb, codes,
                        scales);
}

cudaError_t launch_append(int fmt, const AppendParams &p, cudaStream_t s)
{
    if (p.num_seqs == 0 || p.max_new_tokens <= 0) return cudaSuccess;
    // T new tokens starting anywhere touch at most (T - 1 + 63) / 64 + 1 blocks
    const int64_t touched = ((int64_t)p.max_new_tokens + kPage - 2) / kPage + 1;
    if (p.max_new_tokens <= kPage) {
        const int64_t bx = touched * p.num_heads;
        if (bx > 0x7fffffffLL || p.num_seqs > 65535) return cudaErrorInvalidValue;
        const dim3 grid((unsigned)bx, (unsigned)p.num_seqs, 2), block(kShortWarps * 32);
        if (fmt == KVQ_INT4_B64) return launch_pdl(append_short_kernel<KVQ_INT4_B64>, grid, block, 0, s, p);
        if (fmt == KVQ_FP8_E4M3) return launch_pdl(append_short_kernel<KVQ_FP8_E4M3>, grid, block, 0, s, p);
        return launch_pdl(append_short_kernel<KVQ_INT8_PAGE>, grid, block, 0, s, p);
    }
    const int64_t warps = touched * p.num_heads;
    const int64_t bx = (warps + kQuantWarps - 1) / kQuantWarps;
    if (bx > 0x7fffffffLL || p.num_seqs > 65535) return cudaErrorInvalidValue;
    const dim3 grid((unsigned)bx, (unsigned)p.num_seqs, 2), block(kQuantWarps * 32);
    if (fmt == KVQ_INT4_B64) return launch_plain(append_kernel<KVQ_INT4_B64>, grid, block, kStageBytes, s, p);
    if (fmt == KVQ_FP8_E4M3) return launch_plain(append_kernel<KVQ_FP8_E4M3>, grid, block, kStageBytes, s, p);
    return launch_plain(append_kernel<KVQ_INT8_PAGE>, grid, block, kStageBytes, s, p);
}

}  // namespace kvq
