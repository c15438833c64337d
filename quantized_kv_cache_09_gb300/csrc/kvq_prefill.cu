// kvq_prefill.cu -- chunked-prefill attention over the quantized paged cache:
// the n new tokens of a sequence of length L (already appended to the cache)
// attend causally, query i at position L - n + i to keys 0 .. L - n + i
// (dynamic chunked attention, "R1 performance overview", aicoding.csdn.net;
// the cache and its pages as for decode: quantize_block, jsqmd.com/news/887038
// section 2.1, and PagedAttention, ddd.cn section 4).
//
// On the 5th-generation tensor cores (tcgen05).  One CTA owns two tiles of
// 128 query rows of one (sequence, query head); query head hq reads cache head
// hq / g.  Its warps split into roles that hand work over through mbarriers:
//   * 4 widening warps: a page's K and V codes of the cache head arrive in
//     shared memory by two bulk copies; the warps widen them once, for both
//     tiles, to fp16 codes (exact: integers or E4M3 values) in the K-major
//     128-byte-swizzled layout the MMA reads -- K as keys x elements, V
//     transposed (elements x keys) -- into one of 3 stages, and start the
//     copy two pages ahead; the scales stay out of the fp16 operands;
//   * 1 MMA thread: per tile, S = Q K^T (M = 128, N = 64, 8 MMAs of K = 16)
//     into one of two S buffers in tensor memory and O += P V (M = 128,
//     N = 128, 4 MMAs of K = 16) with P read from tensor memory;
//   * 8 softmax warps, one thread per query row (its lane of tensor memory):
//     each loads its row of S, masks keys after its position and runs an
//     online softmax in base 2 with the page's key scale in the exponent and
//     a lazy running maximum (O is rescaled, in tensor memory, only when a
//     row's maximum grows by more than 2^8); P * sv / s_ref (s_ref = the
//     largest value scale over the CTA's pages, so the fp16 operand stays in
//     [0, 256]) goes to tensor memory over the S it came from.
// The two tiles' softmax warps alternate with the tensor cores: while one
// tile's rows are in the softmax, the MMAs of the other run.
// fp32 accumulation throughout; the output is s_ref * O / l rounded to fp16.
#include "kvq_device.cuh"
#include "kvq_internal.h"

namespace kvq {

namespace {

constexpr int kPfWarps = 4;  // softmax warps per query tile (one thread per row)

template <int FMT>
struct PfFmt {
    static constexpr int kRowBytes = 128;  // int8, FP8: one byte per element
};
template <>
struct PfFmt<KVQ_INT4_B64> {
    static constexpr int kRowBytes = 64;
};

// 8 int4 codes (one word: element 2j in the low nibble of byte j, 4-bit two's
// complement) -> 8 fp16 values in element order: biased bytes u ^ 8 = c + 8,
// interleaved, then 1024 + byte - 1032 (0x64 as the high byte of each half)
__device__ __forceinline__ uint4 widen8_int4(uint32_t w)
{
    const uint32_t lo = (w & 0x0F0F0F0Fu) ^ 0x08080808u;         // elements 0, 2, 4, 6
    const uint32_t hi = ((w >> 4) & 0x0F0F0F0Fu) ^ 0x08080808u;  // elements 1, 3, 5, 7
    const uint32_t e03 = __byte_perm(lo, hi, 0x5140);
    const uint32_t e47 = __byte_perm(lo, hi, 0x7362);
    const __half2 k1032 = __float2half2_rn(1032.0f);
    uint32_t r[4];
    const uint32_t src[4] = {__byte_perm(e03, 0x64646464u, 0x4140), __byte_perm(e03, 0x64646464u, 0x4342),
                             __byte_perm(e47, 0x64646464u, 0x4140), __byte_perm(e47, 0x64646464u, 0x4342)};
#pragma unroll
    for (int i = 0; i < 4; i++) r[i] = h2_bits(__hsub2(*reinterpret_cast<const __half2 *>(&src[i]), k1032));
    return make_uint4(r[0], r[1], r[2], r[3]);
}

}  // namespace

// ---------------------------------------------------------------------------
// tcgen05 building blocks: S (128 x 64 keys) and O (128 x 128) of a tile live
// in tensor memory, the operands in shared memory in the K-major 128-byte
// swizzled layout (8-row x 128-byte atoms, 16-byte chunks XOR-ed with the row).
// ---------------------------------------------------------------------------
namespace {

constexpr int kTcRows = 128;   // query rows per tile (TMEM lanes)
constexpr int kTiles = 2;      // query tiles per CTA: each widened page serves both
constexpr int kStages = 3;     // widened pages in shared memory
constexpr int kWidenThreads = 128;
// warps 0..7: softmax of the two tiles; 8..11: widening; 12: MMA issue
constexpr int kTcThreads = kTiles * kPfWarps * 32 + kWidenThreads + 32;
// tile t: S buffers at columns 256 t + 0..63 and 256 t + 64..127, O at 256 t + 128..255
constexpr uint32_t kTmemCols = 256 * kTiles;
constexpr uint32_t kIdescS = (1u << 4) | ((64u >> 3) << 17) | ((128u >> 4) << 24);   // f32 += f16 x f16, 128 x 64, K-major
constexpr uint32_t kIdescO = (1u << 4) | ((128u >> 3) << 17) | ((128u >> 4) << 24);  // 128 x 128
constexpr float kLazy = 8.0f;  // O is rescaled only when a row's max grows by more than 2^8
// key scales below this are raised to it: a page of all-zero keys (scale 0)
// then scores 1e-38 * raw instead of 0 (no difference in binary32 after the
// max is subtracted) and a masked score stays -inf instead of -inf * 0
constexpr float kMinScale = 1.17549435e-38f;

// byte offset of f16 element (r, k) in a K-major, 128-byte-swizzled tile of R rows
__device__ __forceinline__ uint32_t sw128(int r, int k, int R)
{
    return (uint32_t)((k >> 6) * (R * 128) + r * 128 + ((((k & 63) >> 3) ^ (r & 7)) << 4) + ((k & 7) << 1));
}

// shared-memory matrix descriptor: start address, 1024-byte stride between
// 8-row groups, 128-byte swizzle (leading offset unused for K-major swizzled)
__device__ __forceinline__ uint64_t umma_desc(uint32_t saddr)
{
    return (uint64_t)((saddr >> 4) & 0x3FFFu) | ((uint64_t)1 << 16) | ((uint64_t)(1024 >> 4) << 32) |
           ((uint64_t)1 << 46) | ((uint64_t)2 << 61);
}

__device__ __forceinline__ void umma_f16(uint32_t d_tmem, uint64_t a, uint64_t b, uint32_t idesc, uint32_t acc)
{
    asm volatile(
        "{\n\t.reg .pred p;\n\tsetp.ne.b32 p, %4, 0;\n\t"
        "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
        "l"(a), "l"(b), "r"(idesc), "r"(acc));
}

__device__ __forceinline__ void umma_commit(uint64_t *bar)
{
    asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(smem_addr(bar))
                 : "memory");
}

__device__ __forceinline__ void tc_fence_before() { asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory"); }
__device__ __forceinline__ void tc_fence_after() { asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory"); }

// start loading 16 consecutive fp32 columns of this thread's TMEM lane (raw bits;
// valid after tmem_ld_wait)
__device__ __forceinline__ void tmem_ld16_async(uint32_t taddr, uint32_t (&r)[16])
{
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x16.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15}, [%16];"
        : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]),
          "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15])
        : "r"(taddr)
        : "memory");
}
__device__ __forceinline__ void tmem_ld_wait() { asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory"); }

// 16 consecutive fp32 columns of this thread's TMEM lane
__device__ __forceinline__ void tmem_ld16(uint32_t taddr, float (&v)[16])
{
    uint32_t r[16];
    tmem_ld16_async(taddr, r);
    tmem_ld_wait();
#pragma unroll
    for (int i = 0; i < 16; i++) v[i] = __uint_as_float(r[i]);
}

__device__ __forceinline__ void tmem_st16(uint32_t taddr, const float (&v)[16])
{
    asm volatile(
        "tcgen05.st.sync.aligned.32x32b.x16.b32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16};" ::"r"(
            taddr),
        "r"(__float_as_uint(v[0])), "r"(__float_as_uint(v[1])), "r"(__float_as_uint(v[2])), "r"(__float_as_uint(v[3])),
        "r"(__float_as_uint(v[4])), "r"(__float_as_uint(v[5])), "r"(__float_as_uint(v[6])), "r"(__float_as_uint(v[7])),
        "r"(__float_as_uint(v[8])), "r"(__float_as_uint(v[9])), "r"(__float_as_uint(v[10])),
        "r"(__float_as_uint(v[11])), "r"(__float_as_uint(v[12])), "r"(__float_as_uint(v[13])),
        "r"(__float_as_uint(v[14])), "r"(__float_as_uint(v[15]))
        : "memory");
}

// 32 consecutive 32-bit columns of this thread's TMEM lane (completes at tcgen05.wait::st)
__device__ __forceinline__ void tmem_st32(uint32_t taddr, const uint32_t (&w)[32])
{
    asm volatile(
        "tcgen05.st.sync.aligned.32x32b.x32.b32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16,"
        "%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31,%32};" ::"r"(taddr),
        "r"(w[0]), "r"(w[1]), "r"(w[2]), "r"(w[3]), "r"(w[4]), "r"(w[5]), "r"(w[6]), "r"(w[7]), "r"(w[8]), "r"(w[9]),
        "r"(w[10]), "r"(w[11]), "r"(w[12]), "r"(w[13]), "r"(w[14]), "r"(w[15]), "r"(w[16]), "r"(w[17]), "r"(w[18]),
        "r"(w[19]), "r"(w[20]), "r"(w[21]), "r"(w[22]), "r"(w[23]), "r"(w[24]), "r"(w[25]), "r"(w[26]), "r"(w[27]),
        "r"(w[28]), "r"(w[29]), "r"(w[30]), "r"(w[31])
        : "memory");
}

// D (tensor memory) += A (tensor memory) x B (shared-memory descriptor)
__device__ __forceinline__ void umma_f16_ts(uint32_t d_tmem, uint32_t a_tmem, uint64_t b, uint32_t idesc, uint32_t acc)
{
    asm volatile(
        "{\n\t.reg .pred p;\n\tsetp.ne.b32 p, %4, 0;\n\t"
        "tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], %2, %3, p;\n\t}" ::"r"(d_tmem),
        "r"(a_tmem), "l"(b), "r"(idesc), "r"(acc));
}

// 8 elements (one row of an 8 x 8 block, fp16 pairs) of 8 rows -> the block
// transposed: x[j] = column j as 8 fp16 values
__device__ __forceinline__ void transpose8(const uint4 (&w)[8], uint4 (&x)[8])
{
#pragma unroll
    for (int m = 0; m < 4; m++) {  // columns 2m, 2m + 1
        uint32_t lo[4], hi[4];
#pragma unroll
        for (int n = 0; n < 4; n++) {
            const uint32_t a = (&w[2 * n].x)[m], b = (&w[2 * n + 1].x)[m];
            lo[n] = __byte_perm(a, b, 0x5410);
            hi[n] = __byte_perm(a, b, 0x7632);
        }
        x[2 * m] = make_uint4(lo[0], lo[1], lo[2], lo[3]);
        x[2 * m + 1] = make_uint4(hi[0], hi[1], hi[2], hi[3]);
    }
}

// 8 codes of row `row` (elements 8c .. 8c + 7) as 8 fp16 values
template <int FMT>
__device__ __forceinline__ uint4 codes8(const uint8_t *page, int row, int c)
{
    if constexpr (FMT == KVQ_INT4_B64) {
        return widen8_int4(*reinterpret_cast<const uint32_t *>(page + row * 64 + 4 * c));
    } else {
        const uint2 w = *reinterpret_cast<const uint2 *>(page + row * 128 + 8 * c);
        __half2 a[2], b[2];
        if constexpr (FMT == KVQ_FP8_E4M3) {
            widen_e4m3(w.x, a);
            widen_e4m3(w.y, b);
        } else {
            widen_int8(w.x, a);
            widen_int8(w.y, b);
        }
        return make_uint4(h2_bits(a[0]), h2_bits(a[1]), h2_bits(b[0]), h2_bits(b[1]));
    }
}

template <int FMT>
struct alignas(1024) TcSmem {
    uint8_t q[kTiles][kTcRows * kHeadDim * 2];     // 32 KB per tile: query rows x elements
    uint8_t k[kStages][kPage * kHeadDim * 2];      // 16 KB per stage: keys x elements
    uint8_t vt[kStages][kHeadDim * kPage * 2];     // 16 KB per stage: elements x keys (V transposed)
    uint8_t kc[2][kPage * PfFmt<FMT>::kRowBytes];  // codes of the two pages in flight
    uint8_t vc[2][kPage * PfFmt<FMT>::kRowBytes];
    uint64_t code_full[2];       // a page's codes landed (bulk copies)
    uint64_t kv_ready[kStages];  // a page's widened K and V written (every widening thread)
    uint64_t kv_free[kStages];   // every MMA reading a stage complete (commit)
    uint64_t s_full[kTiles];     // S of a tile's page complete (commit)
    uint64_t p_full[kTiles];     // P of a tile's page in tensor memory, O rescaled (every row of the tile)
    uint64_t o_done[kTiles];     // O += P V of a tile's page complete (commit)
    uint64_t mma_done;           // every MMA issued complete (commit, at the end)
    float s_ref;
    uint32_t tmem;
};

__device__ __forceinline__ void mbar_arrive(uint64_t *bar)
{
    asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_addr(bar)) : "memory");
}

// barrier 1 over the widening warpgroup, returning whether every thread passed `v`
__device__ __forceinline__ bool widen_group_all(bool v)
{
    uint32_t r;
    asm volatile(
        "{\n\t.reg .pred p, q;\n\tsetp.ne.u32 q, %1, 0;\n\t"
        "bar.red.and.pred p, 1, %2, q;\n\tselp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(r)
        : "r"((uint32_t)v), "n"(kWidenThreads)
        : "memory");
    return r != 0;
}
__device__ __forceinline__ void widen_group_sync()
{
    asm volatile("bar.sync 1, %0;" ::"n"(kWidenThreads) : "memory");
}

}  // namespace

// Roles, per 64-token page j (all hand-offs are mbarriers, so each role runs
// ahead as far as its buffers allow):
//   widening warps  wait for the codes of page j and for stage j % kStages to
//                   be free, widen K and V into it, start the copy of page
//                   j + 2 into the code buffer just read;
//   MMA thread      per tile: once P(j) is in tensor memory, O += P(j) V(j),
//                   then S(j + 1) = Q K(j + 1)^T into the S buffer P(j - 1)
//                   used; after both tiles, release stage j % kStages;
//   softmax warps   per tile (one thread per query row): wait S(j), mask,
//                   lazy online softmax, P(j) into tensor memory over S(j);
//                   wait PV(j - 1) (O stable; this also frees P(j - 1)'s
//                   buffer for S(j + 1)), rescale O if a row's max moved,
//                   hand P(j) to the MMA thread.
// While one tile's softmax runs, the tensor cores work on the other tile.
template <int FMT>
__global__ void __launch_bounds__(kTcThreads, 1) prefill_attn_tc_kernel(PrefillParams p)
{
    using S = TcSmem<FMT>;
    constexpr int RB = PfFmt<FMT>::kRowBytes;
    constexpr uint32_t kPageBytes = kPage * RB;
    extern __shared__ __align__(1024) uint8_t smem_tc[];
    // the swizzle pattern follows address bits: place the tiles on a 1024-byte boundary
    S &sm = *reinterpret_cast<S *>(smem_tc + ((1024u - (smem_addr(smem_tc) & 1023u)) & 1023u));
    const int tid = threadIdx.x, warp = tid >> 5;
    const int b = blockIdx.z, hq = blockIdx.y;
    const int H = p.num_heads, Hq = p.num_q_heads;
    const int h = hq / p.group;
    const int i0 = blockIdx.x * (kTiles * kTcRows);

    const int c0 = p.cu_q[b];
    const int n = p.cu_q[b + 1] - c0;
    const int L = p.seq_lens[b];
    if (n < 0 || n > p.max_q || n > L || L > p.max_blocks * kPage || c0 < 0 || (int64_t)c0 + n > p.total_q) {
        if (blockIdx.x == 0 && hq == 0 && tid == 0) set_flag(p.status, KVQ_FLAG_BAD_LENGTH);
        return;
    }
    if (i0 >= n) return;
    const int rows = min(kTiles * kTcRows, n - i0);            // valid query rows of the CTA
    const int active = (rows + kTcRows - 1) / kTcRows;        // tiles with at least one of them
    const int qpos0 = L - n + i0;                             // position of the CTA's first query
    // pages tile t reads: through the position of its last valid row
    auto pages_of = [&](int t) {
        return t < active ? (qpos0 + min(kTcRows * (t + 1), rows) - 1) / kPage + 1 : 0;
    };
    const int npages = pages_of(active - 1);
    const int32_t *bt = p.block_table + (int64_t)b * p.max_blocks;

    auto page_of = [&](int j) {
        int pg = bt[j];
        if (pg < 0 || pg >= p.num_pages) {
            set_flag(p.status, KVQ_FLAG_BAD_PAGE);
            pg = 0;
        }
        return pg;
    };
    auto issue = [&](int j) {  // one thread: page j's codes into code buffer j & 1
        const size_t off = ((size_t)page_of(j) * H + h) * kPageBytes;
        mbar_arrive_expect_tx(&sm.code_full[j & 1], 2 * kPageBytes);
        bulk_copy_g2s(sm.kc[j & 1], p.k_codes + off, kPageBytes, &sm.code_full[j & 1]);
        bulk_copy_g2s(sm.vc[j & 1], p.v_codes + off, kPageBytes, &sm.code_full[j & 1]);
    };

    if (tid == 0) {
        mbar_init(&sm.code_full[0], 1);
        mbar_init(&sm.code_full[1], 1);
        for (int s = 0; s < kStages; s++) {
            mbar_init(&sm.kv_ready[s], kWidenThreads);
            mbar_init(&sm.kv_free[s], 1);
        }
        for (int t = 0; t < kTiles; t++) {
            mbar_init(&sm.s_full[t], 1);
            mbar_init(&sm.p_full[t], kTcRows);
            mbar_init(&sm.o_done[t], 1);
        }
        mbar_init(&sm.mma_done, 1);
        mbar_init_fence();
        issue(0);  // the first two pages' codes travel while the queries load
        if (npages > 1) issue(1);
    }
    if (warp == 0) {
        asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(smem_addr(&sm.tmem)),
                     "r"(kTmemCols));
        asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;");
        // the largest value scale over the CTA's pages: P carries sv / s_ref <= 1
        float mx = 0.0f;
        for (int j = tid; j < npages; j += 32) mx = fmaxf(mx, p.v_scales[(int64_t)page_of(j) * H + h]);
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) mx = fmaxf(mx, __shfl_xor_sync(kFull, mx, o));
        if (tid == 0) sm.s_ref = mx > 0.0f ? mx : 1.0f;
    }
    // the query rows of both tiles (zero past the chunk) in the swizzled layout
    for (int e = tid; e < kTiles * kTcRows * (kHeadDim / 8); e += kTcThreads) {
        const int r = e >> 4, c = e & 15;
        uint4 v = make_uint4(0u, 0u, 0u, 0u);
        if (r < rows) v = *reinterpret_cast<const uint4 *>(p.q + ((int64_t)(c0 + i0 + r) * Hq + hq) * kHeadDim + 8 * c);
        *reinterpret_cast<uint4 *>(sm.q[r / kTcRows] + sw128(r % kTcRows, 8 * c, kTcRows)) = v;
    }
    fence_proxy_async_smem();
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = sm.tmem;
    bool ok = true;

    if (warp < kTiles * kPfWarps) {
        // ---- softmax: tile t, one query row per thread (its TMEM lane) ----
        const int t = warp / kPfWarps, row = tid % kTcRows;
        const int nt = pages_of(t);
        const uint32_t lane_tm = tmem + 256u * t + ((uint32_t)((warp % kPfWarps) * 32) << 16);
        const int tile_qpos0 = qpos0 + kTcRows * t;
        const int qpos = tile_qpos0 + row;  // this row's position in the sequence
        const float s_ref = sm.s_ref;
        const float sabs = fabsf(p.score_scale);
        const bool neg_scale = p.score_scale < 0.0f;
        float m_used = -INFINITY, l_run = 0.0f;
        float sk = 0.0f, sv = 0.0f;  // the page's scales, loaded one page ahead
        if (nt > 0) {
            const int pg = page_of(0);
            sk = p.k_scales[(int64_t)pg * H + h];
            sv = p.v_scales[(int64_t)pg * H + h];
        }
        for (int j = 0; j < nt; j++) {
            float nsk = 0.0f, nsv = 0.0f;
            if (j + 1 < nt) {
                const int pg = page_of(j + 1);
                nsk = p.k_scales[(int64_t)pg * H + h];
                nsv = p.v_scales[(int64_t)pg * H + h];
            }
            const float cur_sk = fmaxf(sk * sabs, kMinScale);
            ok = __all_sync(kFull, mbar_wait_bounded(&sm.s_full[t], (uint32_t)(j & 1)));
            if (!ok) break;
            tc_fence_after();
            float sc[64];  // raw scores q . code (the key scale is applied in the exponent)
            {
                uint32_t r[4][16];
#pragma unroll
                for (int c = 0; c < 4; c++) tmem_ld16_async(lane_tm + 64 * (j & 1) + 16 * c, r[c]);
                tmem_ld_wait();
#pragma unroll
                for (int c = 0; c < 4; c++)
#pragma unroll
                    for (int i = 0; i < 16; i++) sc[16 * c + i] = __uint_as_float(r[c][i]);
            }
            // causal mask (pages that reach past a row's position); the maximum is
            // taken on the raw scores with sk >= 0 (a negative softmax scale flips them)
            if (neg_scale) {
#pragma unroll
                for (int i = 0; i < 64; i++) sc[i] = -sc[i];
            }
            if (j * kPage + kPage - 1 > tile_qpos0) {
#pragma unroll
                for (int i = 0; i < 64; i++)
                    if (j * kPage + i > qpos) sc[i] = -INFINITY;
            }
            float mraw = -INFINITY;
#pragma unroll
            for (int i = 0; i < 64; i++) mraw = fmaxf(mraw, sc[i]);
            const float mx = mraw == -INFINITY ? -INFINITY : mraw * cur_sk;
            float factor = 1.0f;
            if (j == 0) {
                m_used = mx;  // key 0 is never masked
            } else if (mx > m_used + kLazy) {
                factor = ex2_approx(m_used - mx);
                m_used = mx;
            }
            // P * sv / s_ref = 2^(raw * sk - m + log2(sv / s_ref)): one FMA per element before ex2;
            // the row sum of P is that sum times s_ref / sv (a page of all-zero values adds to l only)
            const float pv_ratio = sv / s_ref;
            const float off = pv_ratio > 0.0f ? m_used - __log2f(pv_ratio) : m_used;
            float psum = 0.0f;
            {  // P row as 32 fp16 pairs (keys 2c, 2c + 1) over the first 32 columns of this page's S buffer
                uint32_t w[32];
#pragma unroll
                for (int c = 0; c < 32; c++) {
                    const float p0 = ex2_approx(fmaf(sc[2 * c], cur_sk, -off));
                    const float p1 = ex2_approx(fmaf(sc[2 * c + 1], cur_sk, -off));
                    psum += p0 + p1;
                    w[c] = f16x2_rn(p0, p1);
                }
                tmem_st32(lane_tm + 64 * (j & 1), w);
            }
            // O holds PV(j - 1) once it completes: only then may it be rescaled
            if (j > 0) {
                ok = __all_sync(kFull, mbar_wait_bounded(&sm.o_done[t], (uint32_t)((j - 1) & 1)));
                if (!ok) break;
                tc_fence_after();
            }
            if (__any_sync(kFull, factor != 1.0f)) {  // O (columns 128..255) of the rows whose max moved
#pragma unroll
                for (int c = 0; c < 8; c++) {
                    float v[16];
                    tmem_ld16(lane_tm + 128 + 16 * c, v);
#pragma unroll
                    for (int i = 0; i < 16; i++) v[i] *= factor;
                    tmem_st16(lane_tm + 128 + 16 * c, v);
                }
            }
            asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory");
            tc_fence_before();
            mbar_arrive(&sm.p_full[t]);
            l_run = l_run * factor + (pv_ratio > 0.0f ? psum / pv_ratio : psum);
            sk = nsk;
            sv = nsv;
        }
        if (ok && nt > 0) {  // out = s_ref * O / l after the last PV; loads warp-wide, stores per row
            ok = __all_sync(kFull, mbar_wait_bounded(&sm.o_done[t], (uint32_t)((nt - 1) & 1)));
            if (ok) {
                tc_fence_after();
                const int tile_rows = rows - kTcRows * t;
                const float inv = s_ref / l_run;
                uint16_t *dst = p.out + ((int64_t)(c0 + i0 + kTcRows * t + row) * Hq + hq) * kHeadDim;
#pragma unroll
                for (int c = 0; c < 8; c++) {
                    float v[16];
                    tmem_ld16(lane_tm + 128 + 16 * c, v);
                    if (row >= tile_rows) continue;
                    uint4 o0, o1;
                    o0.x = f16x2_rn(v[0] * inv, v[1] * inv);
                    o0.y = f16x2_rn(v[2] * inv, v[3] * inv);
                    o0.z = f16x2_rn(v[4] * inv, v[5] * inv);
                    o0.w = f16x2_rn(v[6] * inv, v[7] * inv);
                    o1.x = f16x2_rn(v[8] * inv, v[9] * inv);
                    o1.y = f16x2_rn(v[10] * inv, v[11] * inv);
                    o1.z = f16x2_rn(v[12] * inv, v[13] * inv);
                    o1.w = f16x2_rn(v[14] * inv, v[15] * inv);
                    reinterpret_cast<uint4 *>(dst + 16 * c)[0] = o0;
                    reinterpret_cast<uint4 *>(dst + 16 * c)[1] = o1;
                }
            }
        }
    } else if (warp < kTiles * kPfWarps + kWidenThreads / 32) {
        // ---- widening: codes -> fp16 operands of stage j % kStages ----
        const int w = tid - kTiles * kPfWarps * 32;
        int j = 0;
        for (; j < npages; j++) {
            const int s = j % kStages, cb = j & 1;
            bool got = true;
            if (j >= kStages) got = mbar_wait_bounded(&sm.kv_free[s], (uint32_t)((j / kStages - 1) & 1));
            got = got && mbar_wait_bounded(&sm.code_full[cb], (uint32_t)((j >> 1) & 1));
            if (!widen_group_all(got)) {
                ok = false;
                break;
            }
            // keys: 8 16-byte chunks per thread
#pragma unroll
            for (int r = 0; r < (kPage * 16) / kWidenThreads; r++) {
                const int e = w + kWidenThreads * r;
                const int key = e >> 4, c = e & 15;
                *reinterpret_cast<uint4 *>(sm.k[s] + sw128(key, 8 * c, kPage)) = codes8<FMT>(sm.kc[cb], key, c);
            }
            {  // values: one 8 x 8 block per thread (keys 8 kb .., elements 8 dc ..), transposed
                const int kb = w & 7, dc = w >> 3;
                uint4 v8[8], x[8];
#pragma unroll
                for (int i = 0; i < 8; i++) v8[i] = codes8<FMT>(sm.vc[cb], 8 * kb + i, dc);
                transpose8(v8, x);
#pragma unroll
                for (int i = 0; i < 8; i++)
                    *reinterpret_cast<uint4 *>(sm.vt[s] + sw128(8 * dc + i, 8 * kb, kHeadDim)) = x[i];
            }
            fence_proxy_async_smem();  // the MMAs read stage s, the next copy overwrites code buffer cb
            widen_group_sync();
            if (w == 0 && j + 2 < npages) issue(j + 2);
            mbar_arrive(&sm.kv_ready[s]);
        }
        if (!ok && w == 0) {  // copies already started land before the CTA's shared memory goes away
            for (int q = j; q < min(npages, j + 2); q++) mbar_wait_bounded(&sm.code_full[q & 1], (uint32_t)((q >> 1) & 1));
        }
    } else if ((tid & 31) == 0) {
        // ---- the MMA thread ----
        const int n0 = pages_of(0), n1 = pages_of(1);
        auto issue_s = [&](int t, int j) {  // S(j) = Q K(j)^T of tile t into its S buffer j & 1
            const uint32_t aq = smem_addr(sm.q[t]), ak = smem_addr(sm.k[j % kStages]);
#pragma unroll
            for (int ks = 0; ks < 8; ks++)
                umma_f16(tmem + 256 * t + 64 * (j & 1), umma_desc(aq + (ks >> 2) * (kTcRows * 128) + (ks & 3) * 32),
                         umma_desc(ak + (ks >> 2) * (kPage * 128) + (ks & 3) * 32), kIdescS, ks > 0);
            umma_commit(&sm.s_full[t]);
        };
        auto issue_pv = [&](int t, int j) {  // O += P(j) V(j), P from tensor memory (8 columns per 16 keys)
            const uint32_t tt = tmem + 256 * t, av = smem_addr(sm.vt[j % kStages]);
#pragma unroll
            for (int ks = 0; ks < 4; ks++)
                umma_f16_ts(tt + 128, tt + 64 * (j & 1) + 8 * ks, umma_desc(av + ks * 32), kIdescO, (j > 0 || ks > 0));
            umma_commit(&sm.o_done[t]);
        };
        ok = mbar_wait_bounded(&sm.kv_ready[0], 0u);
        if (ok) {
            tc_fence_after();
            issue_s(0, 0);
            if (n1 > 0) issue_s(1, 0);
        }
        for (int j = 0; j < npages && ok; j++) {
            bool next_ready = false;
            for (int t = 0; t < kTiles && ok; t++) {
                const int nt = t == 0 ? n0 : n1;
                if (j >= nt) continue;
                ok = mbar_wait_bounded(&sm.p_full[t], (uint32_t)(j & 1));
                if (!ok) break;
                tc_fence_after();
                issue_pv(t, j);
                if (j + 1 < nt) {
                    if (!next_ready) {
                        ok = mbar_wait_bounded(&sm.kv_ready[(j + 1) % kStages], (uint32_t)(((j + 1) / kStages) & 1));
                        if (!ok) break;
                        tc_fence_after();
                        next_ready = true;
                    }
                    issue_s(t, j + 1);
                }
            }
            if (ok) umma_commit(&sm.kv_free[j % kStages]);
        }
        umma_commit(&sm.mma_done);  // whatever was issued completes before tensor memory is freed
        if (!mbar_wait_bounded(&sm.mma_done, 0u)) ok = false;
    }
    __syncwarp();
    if (!ok) set_flag(p.status, KVQ_FLAG_TIMEOUT);
    tc_fence_before();
    __syncthreads();
    if (warp == 0) asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem), "r"(kTmemCols));
}

template <int FMT>
static cudaError_t launch_prefill_tc(const PrefillParams &p, cudaStream_t s)
{
    const size_t smem = sizeof(TcSmem<FMT>) + 1024;  // + room to align the tiles to 1024 bytes
    cudaError_t e = cudaFuncSetAttribute(prefill_attn_tc_kernel<FMT>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         (int)smem);
    if (e != cudaSuccess) return e;
    constexpr int kCtaRows = kTiles * kTcRows;
    const dim3 grid((unsigned)((p.max_q + kCtaRows - 1) / kCtaRows), (unsigned)p.num_q_heads, (unsigned)p.num_seqs);
    return launch_plain(prefill_attn_tc_kernel<FMT>, grid, dim3(kTcThreads), smem, s, p);
}

cudaError_t launch_prefill(int fmt, const PrefillParams &p, cudaStream_t s)
{
    if (p.num_seqs == 0 || p.max_q == 0) return cudaSuccess;
    if (p.num_seqs > 65535 || p.num_q_heads > 65535) return cudaErrorInvalidValue;
    if (fmt == KVQ_INT4_B64) return launch_prefill_tc<KVQ_INT4_B64>(p, s);
    if (fmt == KVQ_FP8_E4M3) return launch_prefill_tc<KVQ_FP8_E4M3>(p, s);
    return launch_prefill_tc<KVQ_INT8_PAGE>(p, s);
}

}  // namespace kvq
