// kvq_decode.cu -- single-token decode attention over the quantized paged KV
// cache (decode reading a quantized KV cache: aicoding.csdn.net section 3.1;
// paging through a block table: ddd.cn section 4).
//
// Decode is a GEMV per (sequence, head): every cached byte is read once and
// used for a handful of flops, so the kernel is built around HBM streaming on
// CUDA cores, not tensor cores.
//
// Work decomposition (persistent, split-K over the sequence):
//   unit   = 32 tokens (int4) or 16 tokens (int8) of one (sequence, head):
//            2 KiB of K codes + 2 KiB of V codes, contiguous inside one page;
//   order  = sequence-major, then head, then unit;
//   warps  = a persistent grid of (SMs x CTAs/SM x 4) warps; warp g owns the
//            contiguous unit range [U g / G, U (g+1) / G), so every warp
//            streams the same number of bytes whatever the length mix;
//   stream = each warp runs its own 4-stage ring of shared-memory stages
//            filled by bulk async copies (cp.async.bulk, completing on one
//            mbarrier per stage), issued kStages units ahead by lane 0;
//   math   = codes are widened to fp16 exactly in registers (magic-number
//            bias trick), then fp32 FMAs: s = scale_k * (q . c) * softmax_scale,
//            online softmax in fp32 (base 2), acc += p * scale_v * c;
//   split  = a (sequence, head) wholly inside one warp's range is written as
//            the final output; one cut by range boundaries leaves (m, l, acc)
//            partials that the merge kernel combines:
//            m = max m_i, l = sum l_i 2^(m_i - m), o = sum acc_i 2^(m_i - m) / l.
#include "kvq_device.cuh"
#include "kvq_internal.h"

namespace kvq {

constexpr int kDecWarps = 4;
constexpr int kStages = 4;
constexpr int kUnitBytes = 2048;
constexpr int kMinUnitsPerWarp = 2;
constexpr int kDecCtasPerSm = 3;

template <int FMT>
struct DecFmt;
template <>
struct DecFmt<KVQ_INT4_B64> {
    static constexpr int kRowBytes = 64;
    static constexpr int kUnitTok = 32;
    static constexpr int kUnitsPerPage = 2;
};
template <>
struct DecFmt<KVQ_INT8_PAGE> {
    static constexpr int kRowBytes = 128;
    static constexpr int kUnitTok = 16;
    static constexpr int kUnitsPerPage = 4;
};

struct alignas(16) StageMeta {
    int32_t b, h, c, ntok;
    float sk, sv;
    int32_t new_seg, pad;
};

struct alignas(128) WarpSmem {
    uint8_t k[kStages][kUnitBytes];
    uint8_t v[kStages][kUnitBytes];
    uint16_t q[kStages][kHeadDim];
    StageMeta meta[kStages];
    uint64_t full[kStages];
};

constexpr size_t kSeqSmemBytes = ((2 * kMaxSeqsPerLaunch + 1) * sizeof(int32_t) + 127) / 128 * 128;
constexpr size_t kDecSmemBytes = kDecWarps * sizeof(WarpSmem) + kSeqSmemBytes;

// ---------------------------------------------------------------------------
// exact widening of packed codes to fp16 pairs
//   int4 word (8 nibbles, element j at bits 4j): returns {c0,c4},{c1,c5},{c2,c6},{c3,c7}
//   (1024 + (n ^ 8)) - 1032 = c  for the low nibble of each half;
//   (1024 + 16 (n ^ 8)) / 16 - 72 = c for the high nibble.
// ---------------------------------------------------------------------------
__device__ __forceinline__ void widen_int4(uint32_t w, __half2 c[4])
{
    const uint32_t hi = w >> 8;
    const uint32_t a = (w & 0x000f000fu) ^ 0x64086408u;
    const uint32_t b = (w & 0x00f000f0u) ^ 0x64806480u;
    const uint32_t d = (hi & 0x000f000fu) ^ 0x64086408u;
    const uint32_t e = (hi & 0x00f000f0u) ^ 0x64806480u;
    const __half2 k1032 = __float2half2_rn(1032.0f);
    const __half2 k16 = __float2half2_rn(0.0625f);
    const __half2 km72 = __float2half2_rn(-72.0f);
    c[0] = __hsub2(*reinterpret_cast<const __half2 *>(&a), k1032);
    c[1] = __hfma2(*reinterpret_cast<const __half2 *>(&b), k16, km72);
    c[2] = __hsub2(*reinterpret_cast<const __half2 *>(&d), k1032);
    c[3] = __hfma2(*reinterpret_cast<const __half2 *>(&e), k16, km72);
}

//   int8 word (4 bytes, element j in byte j): returns {c0,c1},{c2,c3}
//   1024 + (byte ^ 0x80) - 1152 = c
__device__ __forceinline__ void widen_int8(uint32_t w, __half2 c[2])
{
    const uint32_t x = w ^ 0x80808080u;
    const uint32_t a = __byte_perm(x, 0x64646464u, 0x4140);
    const uint32_t b = __byte_perm(x, 0x64646464u, 0x4342);
    const __half2 k1152 = __float2half2_rn(1152.0f);
    c[0] = __hsub2(*reinterpret_cast<const __half2 *>(&a), k1152);
    c[1] = __hsub2(*reinterpret_cast<const __half2 *>(&b), k1152);
}

// sum_j q[j] c[j] over the 8 elements of one int4 word; q in element order
__device__ __forceinline__ float dot8_int4(uint32_t w, const float *q, float acc)
{
    __half2 c[4];
    widen_int4(w, c);
#pragma unroll
    for (int i = 0; i < 4; i++) {
        const float2 f = __half22float2(c[i]);
        acc = fmaf(q[i], f.x, acc);
        acc = fmaf(q[i + 4], f.y, acc);
    }
    return acc;
}

// acc[j] += p * c[j] over the 8 elements of one int4 word
__device__ __forceinline__ void axpy8_int4(uint32_t w, float p, float *acc)
{
    __half2 c[4];
    widen_int4(w, c);
#pragma unroll
    for (int i = 0; i < 4; i++) {
        const float2 f = __half22float2(c[i]);
        acc[i] = fmaf(p, f.x, acc[i]);
        acc[i + 4] = fmaf(p, f.y, acc[i + 4]);
    }
}

__device__ __forceinline__ float dot4_int8(uint32_t w, const float *q, float acc)
{
    __half2 c[2];
    widen_int8(w, c);
    const float2 f0 = __half22float2(c[0]);
    const float2 f1 = __half22float2(c[1]);
    acc = fmaf(q[0], f0.x, acc);
    acc = fmaf(q[1], f0.y, acc);
    acc = fmaf(q[2], f1.x, acc);
    acc = fmaf(q[3], f1.y, acc);
    return acc;
}

__device__ __forceinline__ void axpy4_int8(uint32_t w, float p, float *acc)
{
    __half2 c[2];
    widen_int8(w, c);
    const float2 f0 = __half22float2(c[0]);
    const float2 f1 = __half22float2(c[1]);
    acc[0] = fmaf(p, f0.x, acc[0]);
    acc[1] = fmaf(p, f0.y, acc[1]);
    acc[2] = fmaf(p, f1.x, acc[2]);
    acc[3] = fmaf(p, f1.y, acc[3]);
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

template <int FMT>
__global__ void __launch_bounds__(kDecWarps * 32, kDecCtasPerSm)
    decode_split_kernel(DecodeParams p, int grid_warps)
{
    using F = DecFmt<FMT>;
    constexpr int UT = F::kUnitTok;
    constexpr int UPP = F::kUnitsPerPage;
    constexpr int RB = F::kRowBytes;
    extern __shared__ __align__(128) uint8_t smem_raw[];
    WarpSmem *wsm_all = reinterpret_cast<WarpSmem *>(smem_raw);
    int32_t *s_cu = reinterpret_cast<int32_t *>(smem_raw + kDecWarps * sizeof(WarpSmem));
    int32_t *s_len = s_cu + kMaxSeqsPerLaunch + 1;

    const int tid = threadIdx.x;
    const int lane = tid & 31;
    const int warp = tid >> 5;
    const int B = p.num_seqs;
    const int H = p.num_heads;
    const int max_len = p.max_blocks * kPage;

    // ---- per-sequence lengths and the (H x units) prefix, in shared memory ----
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
            if (i < B) sum += units_of(s_len[i], UT) * H;
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
                run += units_of(s_len[i], UT) * H;
            }
        }
        if (lane == 31) s_cu[B] = incl;
    }
    __syncthreads();
    if (blockIdx.x == 0)
        for (int b = tid; b <= B; b += blockDim.x) p.cu_units[b] = s_cu[b];

    const int64_t U = s_cu[B];
    if (U == 0) return;
    const int64_t G = imin64((int64_t)grid_warps, (U + kMinUnitsPerWarp - 1) / kMinUnitsPerWarp);
    const int gw = blockIdx.x * kDecWarps + warp;
    if (gw >= G) return;
    const int64_t x0 = U * gw / G;
    const int64_t x1 = U * (gw + 1) / G;
    if (x0 >= x1) return;

    WarpSmem &ws = wsm_all[warp];
    if (lane == 0) {
#pragma unroll
        for (int s = 0; s < kStages; s++) mbar_init(&ws.full[s], 1);
        mbar_init_fence();
    }
    __syncwarp();

    // ---- issue cursor: unit xi = (ib, ih, ic) ----
    int ib, ih, ic;
    {
        int lo = 0, hi = B - 1;
        while (lo < hi) {
            const int mid = (lo + hi + 1) >> 1;
            if (s_cu[mid] <= x0) lo = mid; else hi = mid - 1;
        }
        ib = lo;
        const int n = units_of(s_len[ib], UT);
        const int off = (int)(x0 - s_cu[ib]);
        ih = off / n;
        ic = off % n;
    }
    // page ring: lane l holds page slot ring_j0 + l of (ring_b, ring_h)
    int ring_b = -1, ring_h = -1, ring_j0 = 0;
    int r_page = 0;
    float r_sk = 0.0f, r_sv = 0.0f;

    auto issue = [&](int64_t xi, int s) {
        const int j = ic / UPP;
        if (ib != ring_b || ih != ring_h || j < ring_j0 || j >= ring_j0 + 32) {
            ring_b = ib;
            ring_h = ih;
            ring_j0 = j;
            const int jl = j + lane;
            const int npages = (s_len[ib] + kPage - 1) / kPage;
            int pg = 0;
            float sk = 0.0f, sv = 0.0f;
            if (jl < npages) {
                pg = p.block_table[(int64_t)ib * p.max_blocks + jl];
                if (pg < 0 || pg >= p.num_pages) {
                    set_flag(p.status, KVQ_FLAG_BAD_PAGE);
                    pg = 0;
                }
                sk = p.k_scales[(int64_t)pg * H + ih];
                sv = p.v_scales[(int64_t)pg * H + ih];
            }
            r_page = pg;
            r_sk = sk;
            r_sv = sv;
        }
        const int pg = __shfl_sync(kFull, r_page, j - ring_j0);
        const float sk = __shfl_sync(kFull, r_sk, j - ring_j0);
        const float sv = __shfl_sync(kFull, r_sv, j - ring_j0);
        const bool new_seg = (xi == x0) || (ic == 0);
        if (lane == 0) {
            StageMeta &mt = ws.meta[s];
            mt.b = ib;
            mt.h = ih;
            mt.c = ic;
            mt.ntok = min(UT, s_len[ib] - ic * UT);
            mt.sk = sk;
            mt.sv = sv;
            mt.new_seg = new_seg ? 1 : 0;
            fence_proxy_async_smem();
            const uint32_t bytes = 2 * kUnitBytes + (new_seg ? kHeadDim * 2 : 0);
            mbar_arrive_expect_tx(&ws.full[s], bytes);
            const int64_t off = ((int64_t)pg * H + ih) * (kPage * RB) + (int64_t)(ic % UPP) * (UT * RB);
            bulk_copy_g2s(ws.k[s], p.k_codes + off, kUnitBytes, &ws.full[s]);
            bulk_copy_g2s(ws.v[s], p.v_codes + off, kUnitBytes, &ws.full[s]);
            if (new_seg)
                bulk_copy_g2s(ws.q[s], p.q + ((int64_t)ib * H + ih) * kHeadDim, kHeadDim * 2, &ws.full[s]);
        }
        // advance the cursor
        if (++ic == units_of(s_len[ib], UT)) {
            ic = 0;
            if (++ih == H) {
                ih = 0;
                ++ib;
                while (ib < B && s_len[ib] == 0) ++ib;
            }
        }
    };

    int64_t xi = x0;
    for (int s = 0; s < kStages && xi < x1; s++, xi++) issue(xi, s);

    // ---- consumer state ----
    constexpr int QN = (FMT == KVQ_INT4_B64) ? 32 : 16;  // query elements per lane
    float qf[QN];
    float acc[16];
    float m_run = -INFINITY;
    float l_lane = 0.0f;
    int cur_b = -1, cur_h = -1;
    int64_t seg_x = x0;
    bool timed_out = false;

    auto flush = [&](int b, int h, int64_t sa, int64_t sb) {
        const int n = units_of(s_len[b], UT);
        const int64_t u0 = s_cu[b] + (int64_t)h * n;
        const int64_t u1 = u0 + n;
#pragma unroll
        for (int i = 0; i < 16; i++) {
            acc[i] += __shfl_xor_sync(kFull, acc[i], 8);
            acc[i] += __shfl_xor_sync(kFull, acc[i], 16);
        }
        const float l = warp_sum(l_lane);
        const int vc = lane & 7;
        if (sa == u0 && sb == u1) {
            if (lane < 8) {
                const float inv = 1.0f / l;
                uint32_t hw[8];
#pragma unroll
                for (int i = 0; i < 8; i++) {
                    const __half2 t = __floats2half2_rn(acc[2 * i] * inv, acc[2 * i + 1] * inv);
                    hw[i] = *reinterpret_cast<const uint32_t *>(&t);
                }
                uint4 *dst = reinterpret_cast<uint4 *>(p.out + ((int64_t)b * H + h) * kHeadDim + vc * 16);
                dst[0] = make_uint4(hw[0], hw[1], hw[2], hw[3]);
                dst[1] = make_uint4(hw[4], hw[5], hw[6], hw[7]);
            }
        } else {
            const int slot = (sa == x0) ? 0 : 1;
            float *dst = p.partials + ((int64_t)gw * 2 + slot) * kPartialStride;
            if (lane == 0) {
                dst[0] = m_run;
                dst[1] = l;
            }
            if (lane < 8) {
                float4 *d4 = reinterpret_cast<float4 *>(dst + 4 + vc * 16);
#pragma unroll
                for (int i = 0; i < 4; i++) d4[i] = make_float4(acc[4 * i], acc[4 * i + 1], acc[4 * i + 2], acc[4 * i + 3]);
            }
        }
    };

    for (int64_t x = x0; x < x1; x++) {
        const int s = (int)((x - x0) % kStages);
        const uint32_t parity = (uint32_t)(((x - x0) / kStages) & 1);
        if (!mbar_wait_bounded(&ws.full[s], parity)) {
            if (lane == 0) set_flag(p.status, KVQ_FLAG_TIMEOUT);
            // let the copies still in flight land before the warp leaves
            for (int64_t y = x + 1; y < xi; y++) {
                const int s2 = (int)((y - x0) % kStages);
                mbar_wait_bounded(&ws.full[s2], (uint32_t)(((y - x0) / kStages) & 1));
            }
            timed_out = true;
            break;
        }
        const StageMeta mt = ws.meta[s];
        if (mt.new_seg) {
            if (cur_b >= 0) flush(cur_b, cur_h, seg_x, x);
            cur_b = mt.b;
            cur_h = mt.h;
            seg_x = x;
            m_run = -INFINITY;
            l_lane = 0.0f;
#pragma unroll
            for (int i = 0; i < 16; i++) acc[i] = 0.0f;
            // this lane's query slice: dims (lane & 3) * 32 .. +32 (int4) or (lane & 7) * 16 .. +16 (int8)
            const int q0 = (FMT == KVQ_INT4_B64) ? (lane & 3) * 32 : (lane & 7) * 16;
            const uint4 *qs = reinterpret_cast<const uint4 *>(ws.q[s] + q0);
#pragma unroll
            for (int i = 0; i < QN / 8; i++) {
                const uint4 v = qs[i];
                const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
                for (int k = 0; k < 4; k++) {
                    const float2 f = __half22float2(*reinterpret_cast<const __half2 *>(&w[k]));
                    qf[8 * i + 2 * k] = f.x;
                    qf[8 * i + 2 * k + 1] = f.y;
                }
            }
        }
        const uint8_t *ks = ws.k[s];
        const uint8_t *vs = ws.v[s];
        float score;
        int tok;
        if constexpr (FMT == KVQ_INT4_B64) {
            // K: lane -> token group g = lane >> 2, 32-dim chunk r = lane & 3; pass k covers token 8k + g
            const int g = lane >> 2, r = lane & 3;
            float P[4];
#pragma unroll
            for (int k = 0; k < 4; k++) {
                const uint4 w = *reinterpret_cast<const uint4 *>(ks + (8 * k + g) * RB + r * 16);
                float a = 0.0f;
                a = dot8_int4(w.x, qf + 0, a);
                a = dot8_int4(w.y, qf + 8, a);
                a = dot8_int4(w.z, qf + 16, a);
                a = dot8_int4(w.w, qf + 24, a);
                P[k] = a;
            }
            // reduce-scatter over the 4 lanes of a token group: lane keeps pass 2 (r & 1) + (r >> 1)
            const bool o1 = r & 1;
            float k0 = o1 ? P[2] : P[0], k1 = o1 ? P[3] : P[1];
            const float s0 = o1 ? P[0] : P[2], s1 = o1 ? P[1] : P[3];
            k0 += __shfl_xor_sync(kFull, s0, 1);
            k1 += __shfl_xor_sync(kFull, s1, 1);
            const bool o2 = r & 2;
            score = (o2 ? k1 : k0) + __shfl_xor_sync(kFull, o2 ? k0 : k1, 2);
            tok = 8 * (2 * (r & 1) + (r >> 1)) + g;
        } else {
            // K: lane -> token group g = lane >> 3, 16-dim chunk r = lane & 7; pass k covers token 4k + g
            const int g = lane >> 3, r = lane & 7;
            float P[4];
#pragma unroll
            for (int k = 0; k < 4; k++) {
                const uint4 w = *reinterpret_cast<const uint4 *>(ks + (4 * k + g) * RB + r * 16);
                float a = 0.0f;
                a = dot4_int8(w.x, qf + 0, a);
                a = dot4_int8(w.y, qf + 4, a);
                a = dot4_int8(w.z, qf + 8, a);
                a = dot4_int8(w.w, qf + 12, a);
                P[k] = a;
            }
            const bool o1 = r & 1;
            float k0 = o1 ? P[2] : P[0], k1 = o1 ? P[3] : P[1];
            const float s0 = o1 ? P[0] : P[2], s1 = o1 ? P[1] : P[3];
            k0 += __shfl_xor_sync(kFull, s0, 1);
            k1 += __shfl_xor_sync(kFull, s1, 1);
            const bool o2 = r & 2;
            float sc = (o2 ? k1 : k0) + __shfl_xor_sync(kFull, o2 ? k0 : k1, 2);
            score = sc + __shfl_xor_sync(kFull, sc, 4);  // lanes l and l ^ 4 hold the same token
            tok = 4 * (2 * (r & 1) + ((r >> 1) & 1)) + g;
        }
        const float s2 = (tok < mt.ntok) ? score * (mt.sk * p.score_scale) : -INFINITY;
        const float mu = warp_max(s2);
        if (mu > m_run) {
            const float alpha = ex2_approx(m_run - mu);
            l_lane *= alpha;
#pragma unroll
            for (int i = 0; i < 16; i++) acc[i] *= alpha;
            m_run = mu;
        }
        const float pe = ex2_approx(s2 - m_run);
        if constexpr (FMT == KVQ_INT4_B64) {
            l_lane += pe;
        } else {
            l_lane += (lane & 4) ? 0.0f : pe;  // each token is held by two lanes
        }
        const float pv = pe * mt.sv;
        // V: lane -> 16-dim chunk vc = lane & 7, token subset ts = lane >> 3
        const int vc = lane & 7, ts = lane >> 3;
        if constexpr (FMT == KVQ_INT4_B64) {
#pragma unroll
            for (int j = 0; j < 8; j++) {
                const int t = 4 * j + ts;
                const int src = (4 * (j & 1) + ts) * 4 + (((j >> 1) & 1) << 1) + (j >> 2);
                const float pt = __shfl_sync(kFull, pv, src);
                const uint2 w = *reinterpret_cast<const uint2 *>(vs + t * RB + vc * 8);
                axpy8_int4(w.x, pt, acc);
                axpy8_int4(w.y, pt, acc + 8);
            }
        } else {
#pragma unroll
            for (int j = 0; j < 4; j++) {
                const int t = 4 * j + ts;
                const int src = ts * 8 + ((j & 1) << 1) + (j >> 1);
                const float pt = __shfl_sync(kFull, pv, src);
                const uint4 w = *reinterpret_cast<const uint4 *>(vs + t * RB + vc * 16);
                axpy4_int8(w.x, pt, acc);
                axpy4_int8(w.y, pt, acc + 4);
                axpy4_int8(w.z, pt, acc + 8);
                axpy4_int8(w.w, pt, acc + 12);
            }
        }
        __syncwarp();
        if (xi < x1) {
            issue(xi, s);
            ++xi;
        }
    }
    if (!timed_out && cur_b >= 0) flush(cur_b, cur_h, seg_x, x1);
}

// one warp per (sequence, head): combine the split partials of a (sequence,
// head) cut by warp-range boundaries; write zeros for empty sequences
__global__ void __launch_bounds__(128) decode_merge_kernel(DecodeParams p, int grid_warps)
{
    const int w = blockIdx.x * 4 + (threadIdx.x >> 5);
    const int lane = threadIdx.x & 31;
    const int B = p.num_seqs, H = p.num_heads;
    if (w >= B * H) return;
    const int b = w / H, h = w % H;
    const int64_t U = p.cu_units[B];
    const int64_t cb = p.cu_units[b];
    const int64_t n = (p.cu_units[b + 1] - cb) / H;
    uint2 *orow = reinterpret_cast<uint2 *>(p.out + ((int64_t)b * H + h) * kHeadDim) + lane;
    if (n == 0) {
        *orow = make_uint2(0u, 0u);
        return;
    }
    const int64_t G = imin64((int64_t)grid_warps, (U + kMinUnitsPerWarp - 1) / kMinUnitsPerWarp);
    const int64_t u0 = cb + h * n;
    const int64_t u1 = u0 + n;
    const int64_t gf = ((u0 + 1) * G - 1) / U;
    const int64_t gl = (u1 * G - 1) / U;
    if (gf == gl) return;  // written whole by the split kernel
    float M = -INFINITY;
    for (int64_t g = gf; g <= gl; g++) {
        const int slot = (g == gf && (U * g / G) != u0) ? 1 : 0;
        M = fmaxf(M, p.partials[(g * 2 + slot) * kPartialStride]);
    }
    float L = 0.0f;
    float4 o = make_float4(0.f, 0.f, 0.f, 0.f);
    for (int64_t g = gf; g <= gl; g++) {
        const int slot = (g == gf && (U * g / G) != u0) ? 1 : 0;
        const float *src = p.partials + (g * 2 + slot) * kPartialStride;
        const float wgt = ex2_approx(src[0] - M);
        L += src[1] * wgt;
        const float4 a = reinterpret_cast<const float4 *>(src + 4)[lane];
        o.x += a.x * wgt;
        o.y += a.y * wgt;
        o.z += a.z * wgt;
        o.w += a.w * wgt;
    }
    const float inv = 1.0f / L;
    const __half2 lo = __floats2half2_rn(o.x * inv, o.y * inv);
    const __half2 hi = __floats2half2_rn(o.z * inv, o.w * inv);
    *orow = make_uint2(*reinterpret_cast<const uint32_t *>(&lo), *reinterpret_cast<const uint32_t *>(&hi));
}

template <int FMT>
static int ctas_per_sm()
{
    static int cached[64] = {0};
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return 0;
    if (cached[dev] == 0) {
        if (cudaFuncSetAttribute(decode_split_kernel<FMT>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 (int)kDecSmemBytes) != cudaSuccess)
            return 0;
        int n = 0;
        if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, decode_split_kernel<FMT>, kDecWarps * 32,
                                                          kDecSmemBytes) != cudaSuccess)
            return 0;
        cached[dev] = n < 1 ? 1 : (n > kDecCtasPerSm ? kDecCtasPerSm : n);
    }
    return cached[dev];
}

int decode_grid_warps(int fmt)
{
    int dev = 0, sms = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return 0;
    if (cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) return 0;
    const int per = fmt == KVQ_INT4_B64 ? ctas_per_sm<KVQ_INT4_B64>() : ctas_per_sm<KVQ_INT8_PAGE>();
    return sms * per * kDecWarps;
}

size_t decode_workspace_bytes(int fmt)
{
    const int gw = decode_grid_warps(fmt);
    if (gw <= 0) return 0;
    const size_t partial = (size_t)gw * 2 * kPartialStride * sizeof(float);
    const size_t cu = ((kMaxSeqsPerLaunch + 1) * sizeof(int32_t) + 15) / 16 * 16;
    return partial + cu;
}

cudaError_t launch_decode(int fmt, const DecodeParams &p, cudaStream_t s)
{
    const int gw = decode_grid_warps(fmt);
    if (gw <= 0) return cudaErrorInvalidDevice;
    const int ctas = gw / kDecWarps;
    if (fmt == KVQ_INT4_B64)
        decode_split_kernel<KVQ_INT4_B64><<<ctas, kDecWarps * 32, kDecSmemBytes, s>>>(p, gw);
    else
        decode_split_kernel<KVQ_INT8_PAGE><<<ctas, kDecWarps * 32, kDecSmemBytes, s>>>(p, gw);
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return e;
    const int mblocks = (p.num_seqs * p.num_heads + 3) / 4;
    if (mblocks > 0) decode_merge_kernel<<<mblocks, 128, 0, s>>>(p, gw);
    return cudaGetLastError();
}

}  // namespace kvq
