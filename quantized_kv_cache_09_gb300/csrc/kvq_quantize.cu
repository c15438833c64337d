// kvq_quantize.cu -- fused absmax + quantize + pack of 64-token blocks
// (quantize_block, jsqmd.com/news/887038 section 2.1; INT8 per-chunk variant,
// aicoding.csdn.net section 2.2), for a contiguous tensor and for appends into
// the paged cache.
//
// One warp owns one (block, head): 64 rows x 128 fp16 = 16 KiB, read once from
// HBM with 16-byte loads into registers (lane = row parity x 16-byte chunk, so
// each warp load covers two whole 256-byte rows), reduced to max|x| with packed
// half2 max and one warp redux, then quantized from registers and stored as
// whole rows of codes.  The pages' two-pass design (an extrema pass, then an
// elementwise kernel) becomes a single pass with one HBM read.
//
// Exactness: the code must equal clamp(rint(RN(x / scale))).  The fast path
// multiplies by r = RN(1 / scale); |RN(x*r) - RN(x/scale)| < 1.5 * 2^-23 * |y|,
// so the rounded integer can differ only when y lies within that distance of a
// half-integer.  Any group of 8 elements with |y - rint(y)| > 1/2 - eps
// (eps = 2^-17 for int4, |y| <= 8; 2^-14 for int8, |y| <= 128) is recomputed
// with the correctly rounded division __fdiv_rn.  Clamping before rounding is
// safe because the clamp bounds are integers.
#include "kvq_device.cuh"
#include "kvq_internal.h"

namespace kvq {

template <int FMT>
struct Codec;

template <>
struct Codec<KVQ_INT4_B64> {
    static constexpr int kRowBytes = 64;
    static constexpr float kDiv = 7.5f;
    static constexpr float kLo = -8.0f;
    static constexpr float kHi = 7.0f;
    static constexpr float kMagic = 12582920.0f;      // 1.5 * 2^23 + 8: low nibble = code + 8
    static constexpr float kEps = 7.62939453125e-06f;  // 2^-17
};

template <>
struct Codec<KVQ_INT8_PAGE> {
    static constexpr int kRowBytes = 128;
    static constexpr float kDiv = 127.0f;
    static constexpr float kLo = -127.0f;
    static constexpr float kHi = 127.0f;
    static constexpr float kMagic = 12583040.0f;       // 1.5 * 2^23 + 128: low byte = code + 128
    static constexpr float kEps = 6.103515625e-05f;    // 2^-14
};

// quantize 8 fp16 values; m[j] receives the bits of kMagic + code
template <int FMT>
__device__ __forceinline__ void quant8(const uint4 &v, float r, float scale, uint32_t m[8])
{
    using C = Codec<FMT>;
    const uint32_t w[4] = {v.x, v.y, v.z, v.w};
    float x[8];
#pragma unroll
    for (int i = 0; i < 4; i++) {
        const float2 f = __half22float2(*reinterpret_cast<const __half2 *>(&w[i]));
        x[2 * i] = f.x;
        x[2 * i + 1] = f.y;
    }
    float tmax = 0.0f;
#pragma unroll
    for (int j = 0; j < 8; j++) {
        const float y = __fmul_rn(x[j], r);
        const float yc = fminf(fmaxf(y, C::kLo), C::kHi);
        const float mf = __fadd_rn(yc, C::kMagic);
        tmax = fmaxf(tmax, fabsf(__fsub_rn(yc, __fsub_rn(mf, C::kMagic))));
        m[j] = __float_as_uint(mf);
    }
    if (tmax > 0.5f - C::kEps) {  // near a rounding tie: take the correctly rounded quotient
#pragma unroll
        for (int j = 0; j < 8; j++) {
            const float y = __fdiv_rn(x[j], scale);
            const float yc = fminf(fmaxf(y, C::kLo), C::kHi);
            m[j] = __float_as_uint(__fadd_rn(yc, C::kMagic));
        }
    }
}

__device__ __forceinline__ uint32_t pack8_int4(const uint32_t m[8])
{
    uint32_t w = 0;
#pragma unroll
    for (int j = 0; j < 8; j++) w |= (m[j] & 0xfu) << (4 * j);
    return w ^ 0x88888888u;  // offset binary (code + 8) -> two's complement nibbles
}

__device__ __forceinline__ uint2 pack8_int8(const uint32_t m[8])
{
    uint2 o;
    o.x = __byte_perm(__byte_perm(m[0], m[1], 0x0040), __byte_perm(m[2], m[3], 0x0040), 0x5410);
    o.y = __byte_perm(__byte_perm(m[4], m[5], 0x0040), __byte_perm(m[6], m[7], 0x0040), 0x5410);
    o.x ^= 0x80808080u;  // offset binary (code + 128) -> two's complement bytes
    o.y ^= 0x80808080u;
    return o;
}

// Row pointers of one (block, head) for the contiguous layout x[T][H][D].
struct ContigRows {
    const uint16_t *base;  // row 0 of the block
    int64_t stride;        // elements between rows (H * D)
    __device__ __forceinline__ uint4 load(int r, int chunk) const
    {
        return ld_stream_v4(base + r * stride + 8 * chunk);
    }
};

// Row pointers of one (block, head) of an append: rows before n_old come from
// the fp16 tail buffer (written by this kernel too, so no read-only path),
// later rows from the new tokens.
struct AppendRows {
    const uint16_t *tail;  // tail[b][h] row 0, or nullptr
    const uint16_t *fresh; // head h of new-token row 0
    int64_t row0;          // new-token row that would land in block row 0 (negative when n_old > 0)
    int n_old;
    int64_t stride;        // elements between new-token rows (H * D)
    __device__ __forceinline__ uint4 load(int r, int chunk) const
    {
        if (r < n_old) return *reinterpret_cast<const uint4 *>(tail + r * kHeadDim + 8 * chunk);
        return ld_stream_v4(fresh + (row0 + r) * stride + 8 * chunk);
    }
};

template <int FMT, class Rows>
__device__ __forceinline__ void quantize_block_warp(const Rows &rows, int nrows, uint8_t *__restrict__ codes,
                                                    float *__restrict__ scale_out)
{
    using C = Codec<FMT>;
    const int lane = threadIdx.x & 31;
    const int chunk = lane & 15;  // dims 8*chunk .. 8*chunk+7
    const int rpar = lane >> 4;   // rows 2i + rpar
    uint4 v[32];
#pragma unroll
    for (int i = 0; i < 32; i++) {
        const int r = 2 * i + rpar;
        v[i] = (r < nrows) ? rows.load(r, chunk) : make_uint4(0u, 0u, 0u, 0u);
    }
    __half2 mx = __float2half2_rn(0.0f);
#pragma unroll
    for (int i = 0; i < 32; i++) {
        mx = __hmax2(mx, __habs2(*reinterpret_cast<const __half2 *>(&v[i].x)));
        mx = __hmax2(mx, __habs2(*reinterpret_cast<const __half2 *>(&v[i].y)));
        mx = __hmax2(mx, __habs2(*reinterpret_cast<const __half2 *>(&v[i].z)));
        mx = __hmax2(mx, __habs2(*reinterpret_cast<const __half2 *>(&v[i].w)));
    }
    const uint32_t mb = *reinterpret_cast<const uint32_t *>(&mx);
    uint32_t abits = max(mb & 0xffffu, mb >> 16);  // non-negative fp16: bit order = value order
    abits = __reduce_max_sync(kFull, abits);
    const float a = __half2float(__ushort_as_half(static_cast<unsigned short>(abits)));
    const float scale = __fdiv_rn(a, C::kDiv);
    if (lane == 0) *scale_out = scale;
    const bool zero = !(scale > 0.0f);
    const float r = zero ? 0.0f : __frcp_rn(scale);
#pragma unroll
    for (int i = 0; i < 32; i++) {
        const int row = 2 * i + rpar;
        const bool live = (row < nrows) && !zero;
        uint32_t m[8];
        if (live) quant8<FMT>(v[i], r, scale, m);
        if constexpr (FMT == KVQ_INT4_B64) {
            const uint32_t w = live ? pack8_int4(m) : 0u;
            *reinterpret_cast<uint32_t *>(codes + row * C::kRowBytes + 4 * chunk) = w;
        } else {
            const uint2 w = live ? pack8_int8(m) : make_uint2(0u, 0u);
            *reinterpret_cast<uint2 *>(codes + row * C::kRowBytes + 8 * chunk) = w;
        }
    }
}

constexpr int kQuantWarps = 4;

template <int FMT>
__global__ void __launch_bounds__(kQuantWarps * 32)
    quantize_contig_kernel(const uint16_t *__restrict__ x, int64_t T, int H, int64_t nblocks,
                           uint8_t *__restrict__ codes, float *__restrict__ scales)
{
    using C = Codec<FMT>;
    const int64_t w = (int64_t)blockIdx.x * kQuantWarps + (threadIdx.x >> 5);
    if (w >= nblocks * H) return;
    const int64_t j = w / H;
    const int h = (int)(w % H);
    const int64_t rem = T - j * kPage;
    const int nrows = rem < kPage ? (int)rem : kPage;
    ContigRows rows{x + (j * kPage * H + h) * kHeadDim, (int64_t)H * kHeadDim};
    quantize_block_warp<FMT>(rows, nrows, codes + (j * H + h) * (int64_t)kPage * C::kRowBytes,
                             scales + j * H + h);
}

// grid: x over (touched block, head) of one sequence, y = sequence, z = 0 keys / 1 values
template <int FMT>
__global__ void __launch_bounds__(kQuantWarps * 32)
    append_kernel(AppendParams p)
{
    using C = Codec<FMT>;
    const int b = blockIdx.y;
    const bool is_v = blockIdx.z != 0;
    const int H = p.num_heads;
    const int wi = blockIdx.x * kQuantWarps + (threadIdx.x >> 5);
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
        uint8_t *codes = (is_v ? p.v_codes : p.k_codes) + ((int64_t)page * H + h) * kPage * C::kRowBytes;
        float *scale = (is_v ? p.v_scales : p.k_scales) + (int64_t)page * H + h;
        quantize_block_warp<FMT>(rows, nrows, codes, scale);
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

cudaError_t launch_quantize(int fmt, const uint16_t *x, int64_t T, int H, uint8_t *codes, float *scales,
                            cudaStream_t s)
{
    const int64_t nb = (T + kPage - 1) / kPage;
    const int64_t warps = nb * H;
    const int64_t blocks = (warps + kQuantWarps - 1) / kQuantWarps;
    if (blocks == 0) return cudaSuccess;
    if (blocks > 0x7fffffffLL) return cudaErrorInvalidValue;
    if (fmt == KVQ_INT4_B64)
        quantize_contig_kernel<KVQ_INT4_B64><<<(unsigned)blocks, kQuantWarps * 32, 0, s>>>(x, T, H, nb, codes, scales);
    else
        quantize_contig_kernel<KVQ_INT8_PAGE><<<(unsigned)blocks, kQuantWarps * 32, 0, s>>>(x, T, H, nb, codes, scales);
    return cudaGetLastError();
}

cudaError_t launch_append(int fmt, const AppendParams &p, cudaStream_t s)
{
    if (p.num_seqs == 0 || p.max_new_tokens == 0) return cudaSuccess;
    const int64_t touched = (int64_t)(p.max_new_tokens + kPage - 1) / kPage + 1;
    const int64_t warps = touched * p.num_heads;
    const int64_t bx = (warps + kQuantWarps - 1) / kQuantWarps;
    if (bx > 0x7fffffffLL || p.num_seqs > 65535) return cudaErrorInvalidValue;
    dim3 grid((unsigned)bx, (unsigned)p.num_seqs, 2);
    if (fmt == KVQ_INT4_B64)
        append_kernel<KVQ_INT4_B64><<<grid, kQuantWarps * 32, 0, s>>>(p);
    else
        append_kernel<KVQ_INT8_PAGE><<<grid, kQuantWarps * 32, 0, s>>>(p);
    return cudaGetLastError();
}

}  // namespace kvq
