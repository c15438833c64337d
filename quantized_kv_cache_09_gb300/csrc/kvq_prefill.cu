// kvq_prefill.cu -- chunked-prefill attention over the quantized paged cache:
// the n new tokens of a sequence of length L (already appended to the cache)
// attend causally, query i at position L - n + i to keys 0 .. L - n + i
// (dynamic chunked attention, "R1 performance overview", aicoding.csdn.net;
// the cache and its pages as for decode: quantize_block, jsqmd.com/news/887038
// section 2.1, and PagedAttention, ddd.cn section 4).
//
// On the 5th-generation tensor cores (tcgen05).  One CTA owns two tiles of
// 128 query rows of one (sequence, query head); query head hq reads cache head
// hq / g.  Keys go in steps of 128 (two pages).  The CTA's warps split into
// roles that hand work over through mbarriers:
//   * 4 widening warps load the K and V codes of the cache head straight from
//     global memory into registers (16-byte pieces; V while K is converted,
//     the next step's K while V is converted) and widen
//     them once, for both tiles, to fp16 codes (exact: integers or E4M3
//     values) in shared memory, 128-byte swizzled, keys x elements; the same
//     bytes are the K-major B operand of S and the MN-major B operand of PV.
//     Two stages, K and V of each handed over and released separately; the
//     scales stay out of the fp16 operands;
//   * 1 MMA thread: per tile, S = Q K^T (M = 128, N = 128 keys, 8 MMAs of
//     K = 16) into tensor memory and O += P V (M = 128, N = 128, 8 MMAs) with
//     P read from tensor memory where S was;
//   * 8 softmax warps, one thread per query row (its lane of tensor memory):
//     each loads its row of S, masks keys after its position and runs an
//     online softmax in base 2 with each page's key scale in the exponent and
//     a lazy running maximum (O is rescaled, in tensor memory, only when a
//     row's maximum grows by more than 2^8); P * sv / s_ref (s_ref = the
//     largest value scale over the CTA's pages, so the fp16 operand stays in
//     [0, 256]) goes to tensor memory over the S it came from.
// While one tile's rows are in the softmax, the tensor cores work on the other.
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
constexpr int kStepKeys = 2 * kPage;  // keys per step: two pages, one S of N = 128 per tile
constexpr int kWidenThreads = 128;
// warps 0..7: softmax of the two tiles; 8..11: widening; 12: MMA issue
constexpr int kTcThreads = kTiles * kPfWarps * 32 + kWidenThreads + 32;
// tile t: S (and P over its first 64 columns) at columns 256 t + 0..127, O at 256 t + 128..255
constexpr uint32_t kTmemCols = 256 * kTiles;
// a split half's partial of one query row: m, l, 2 pad, then s_ref * O (16-byte aligned)
constexpr int kPartialFloats = 4 + kHeadDim;
// f32 += f16 x f16, M = 128, N = 128; S: both operands K-major; PV: B (V) MN-major
constexpr uint32_t kIdescS = (1u << 4) | ((128u >> 3) << 17) | ((128u >> 4) << 24);
constexpr uint32_t kIdescO = kIdescS | (1u << 16);
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

// the same with explicit leading (lbo) and stride (sbo) byte offsets; for an MN-major
// swizzled operand lbo steps between 64-element atoms along MN, sbo between 8-row groups along K
__device__ __forceinline__ uint64_t umma_desc_mn(uint32_t saddr, uint32_t lbo, uint32_t sbo)
{
    return (uint64_t)((saddr >> 4) & 0x3FFFu) | ((uint64_t)((lbo >> 4) & 0x3FFFu) << 16) |
           ((uint64_t)((sbo >> 4) & 0x3FFFu) << 32) | ((uint64_t)1 << 46) | ((uint64_t)2 << 61);
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

// D (tensor memory) = A x B (+ D if acc = 1), f32 += f16 x f16, one CTA.  Each shared-memory
// descriptor comes as its two 32-bit halves: the start address sits in bits 0..13 (address
// / 16 < 2^14 for any shared-memory address), so stepping through a tile adds (byte offset
// / 16) to the low half without a carry and an MMA issues after a few integer adds.
// umma_f16_ss: A and B in shared memory; umma_f16_ts: A in tensor memory.
__device__ __forceinline__ void umma_f16_ss(uint32_t d_tmem, uint32_t a_lo, uint32_t a_hi, uint32_t b_lo,
                                            uint32_t b_hi, uint32_t idesc, uint32_t acc)
{
    asm volatile(
        "{\n\t.reg .pred p;\n\t.reg .b64 da, db;\n\t"
        "mov.b64 da, {%1, %2};\n\tmov.b64 db, {%3, %4};\n\t"
        "setp.ne.b32 p, %6, 0;\n\t"
        "tcgen05.mma.cta_group::1.kind::f16 [%0], da, db, %5, p;\n\t}" ::"r"(d_tmem),
        "r"(a_lo), "r"(a_hi), "r"(b_lo), "r"(b_hi), "r"(idesc), "r"(acc));
}
__device__ __forceinline__ void umma_f16_ts(uint32_t d_tmem, uint32_t a_tmem, uint32_t b_lo, uint32_t b_hi,
                                             uint32_t idesc, uint32_t acc)
{
    asm volatile(
        "{\n\t.reg .pred p;\n\t.reg .b64 db;\n\t"
        "mov.b64 db, {%2, %3};\n\t"
        "setp.ne.b32 p, %5, 0;\n\t"
        "tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], db, %4, p;\n\t}" ::"r"(d_tmem),
        "r"(a_tmem), "r"(b_lo), "r"(b_hi), "r"(idesc), "r"(acc));
}

// 16 code bytes (consecutive elements of one row) -> their fp16 values, 8 per uint4
template <int FMT>
__device__ __forceinline__ void widen16(uint4 c, uint4 (&out)[FMT == KVQ_INT4_B64 ? 4 : 2])
{
    if constexpr (FMT == KVQ_INT4_B64) {
        out[0] = widen8_int4(c.x);
        out[1] = widen8_int4(c.y);
        out[2] = widen8_int4(c.z);
        out[3] = widen8_int4(c.w);
    } else {
        const uint32_t wd[4] = {c.x, c.y, c.z, c.w};
#pragma unroll
        for (int i = 0; i < 2; i++) {
            __half2 a[2], b[2];
            if constexpr (FMT == KVQ_FP8_E4M3) {
                widen_e4m3(wd[2 * i], a);
                widen_e4m3(wd[2 * i + 1], b);
            } else {
                widen_int8(wd[2 * i], a);
                widen_int8(wd[2 * i + 1], b);
            }
            out[i] = make_uint4(h2_bits(a[0]), h2_bits(a[1]), h2_bits(b[0]), h2_bits(b[1]));
        }
    }
}

template <int FMT>
struct alignas(1024) TcSmem {
    uint8_t q[kTiles][kTcRows * kHeadDim * 2];  // 32 KB per tile: query rows x elements (K-major)
    uint8_t k[2][kStepKeys * kHeadDim * 2];     // 32 KB per stage: keys x elements (K-major)
    uint8_t v[2][kStepKeys * kHeadDim * 2];     // 32 KB per stage: keys x elements (MN-major B of PV)
    uint64_t k_ready[2];    // a step's widened K written (every widening thread)
    uint64_t v_ready[2];    // a step's widened V written (every widening thread)
    uint64_t k_free[2];     // the S MMAs reading a stage's K complete (commit)
    uint64_t v_free[2];     // the PV MMAs reading a stage's V complete (commit)
    uint64_t s_full[kTiles];  // S of a tile's step complete (commit); PV of the step before too
    uint64_t p_full[kTiles];  // P of a tile's step in tensor memory, O rescaled (every row of the tile)
    uint64_t o_done[kTiles];  // O += P V of a tile's step complete (commit)
    uint64_t mma_done;        // every MMA issued complete (commit, at the end)
    float s_ref;
    uint32_t tmem;
    uint32_t ticket;  // split halves: the count of finished halves this CTA's add saw
};

// the largest of three binary32 values (one instruction)
__device__ __forceinline__ float max3(float a, float b, float c)
{
    float d;
    asm("max.f32 %0, %1, %2, %3;" : "=f"(d) : "f"(a), "f"(b), "f"(c));
    return d;
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

// byte offset of the 8 elements 8c .. 8c + 7 of key `key` in a stage's K or V tile: keys x
// elements in 64-element atoms of 128 keys, 128-byte swizzled -- the K-major layout of K for
// S and, read with the MN-major descriptor, of V for PV
__device__ __forceinline__ uint32_t k_chunk(int key, int c) { return sw128(key, 8 * c, kStepKeys); }

}  // namespace

// Roles, per step i of 128 keys (pages 2i and 2i + 1); all hand-offs are mbarriers:
//   widening warps  widen the K codes of both pages (already in registers) into stage
//                   i & 1 once its K is free, then the V codes once its V is free -- a
//                   page past the last is zero -- loading V while K is converted and the
//                   next step's K while V is converted;
//   MMA thread      per tile: once P(i) is in tensor memory, O += P(i) V(i); once
//                   that is complete (P(i) lives where S goes), S(i + 1) = Q K(i + 1)^T;
//                   a step's last S releases the stage's K, its last PV the V;
//   softmax warps   per tile (one thread per query row): wait S(i) (which also means
//                   PV(i - 1) is complete), row max over the 128 keys, lazy online
//                   softmax, P(i) into tensor memory over S(i), rescale O if a row's
//                   max moved, hand P(i) to the MMA thread.
// While one tile's rows are in the softmax, the tensor cores work on the other tile.
// A CTA runs all key steps of its unit, or one half of them when the unit is split
// (the grid's last wave); then its rows' partials are merged by the second half to end.
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
    // CTA -> unit (256 query rows of one (sequence, query head)) and half: units before
    // num_full run whole; each later unit runs as two CTAs over the two halves of its key
    // steps, whose partials the second to finish merges
    const int cta = blockIdx.x;
    const int unit = cta < p.num_full ? cta : p.num_full + (cta - p.num_full) / 2;
    const int half = cta < p.num_full ? -1 : (cta - p.num_full) & 1;
    const int H = p.num_heads, Hq = p.num_q_heads;
    const int ux = unit % p.units_x;
    const int hq = (unit / p.units_x) % Hq;
    const int b = unit / (p.units_x * Hq);
    const int h = hq / p.group;
    const int i0 = ux * (kTiles * kTcRows);

    const int c0 = p.cu_q[b];
    const int n = p.cu_q[b + 1] - c0;
    const int L = p.seq_lens[b];
    if (n < 0 || n > p.max_q || n > L || L > p.max_blocks * kPage || c0 < 0 || (int64_t)c0 + n > p.total_q) {
        if (ux == 0 && hq == 0 && half <= 0 && tid == 0) set_flag(p.status, KVQ_FLAG_BAD_LENGTH);
        return;
    }
    if (i0 >= n) return;
    const int rows = min(kTiles * kTcRows, n - i0);      // valid query rows of the CTA
    const int active = (rows + kTcRows - 1) / kTcRows;  // tiles with at least one of them
    const int qpos0 = L - n + i0;                       // position of the CTA's first query
    // pages and steps tile t reads: through the position of its last valid row
    auto pages_of = [&](int t) {
        return t < active ? (qpos0 + min(kTcRows * (t + 1), rows) - 1) / kPage + 1 : 0;
    };
    auto steps_of = [&](int t) { return (pages_of(t) + 1) / 2; };
    const int npages = pages_of(active - 1);
    const int nsteps = (npages + 1) / 2;
    // this CTA's steps [lo, hi): all of them, or one half
    const int hsplit = (nsteps + 1) / 2;
    const int lo = half == 1 ? hsplit : 0;
    const int hi = half == 0 ? hsplit : nsteps;
    const int nloc = hi - lo;                 // steps widened here
    const int page_end = min(npages, 2 * hi);  // pages of the range: [2 lo, page_end)
    auto local_steps = [&](int t) { return max(0, min(steps_of(t), hi) - lo); };
    const int32_t *bt = p.block_table + (int64_t)b * p.max_blocks;

    auto page_of = [&](int j) {
        int pg = bt[j];
        if (pg < 0 || pg >= p.num_pages) {
            set_flag(p.status, KVQ_FLAG_BAD_PAGE);
            pg = 0;
        }
        return pg;
    };

    if (tid == 0) {
        for (int s = 0; s < 2; s++) {
            mbar_init(&sm.k_ready[s], kWidenThreads);
            mbar_init(&sm.v_ready[s], kWidenThreads);
            mbar_init(&sm.k_free[s], 1);
            mbar_init(&sm.v_free[s], 1);
        }
        for (int t = 0; t < kTiles; t++) {
            mbar_init(&sm.s_full[t], 1);
            mbar_init(&sm.p_full[t], kTcRows);
            mbar_init(&sm.o_done[t], 1);
        }
        mbar_init(&sm.mma_done, 1);
        mbar_init_fence();
    }
    if (warp == 0) {
        asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(smem_addr(&sm.tmem)),
                     "r"(kTmemCols));
        asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;");
        // the largest value scale over the CTA's pages: P carries sv / s_ref <= 1
        float mx = 0.0f;
        for (int j = 2 * lo + tid; j < page_end; j += 32) mx = fmaxf(mx, p.v_scales[(int64_t)page_of(j) * H + h]);
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
        const int nst = local_steps(t);
        const uint32_t lane_tm = tmem + 256u * t + ((uint32_t)((warp % kPfWarps) * 32) << 16);
        const int tile_qpos0 = qpos0 + kTcRows * t;
        const int qpos = tile_qpos0 + row;  // this row's position in the sequence
        const float s_ref = sm.s_ref;
        const float sabs = fabsf(p.score_scale);
        const bool neg_scale = p.score_scale < 0.0f;
        float m_used = -INFINITY, l_run = 0.0f;
        // the scales of a step's two pages (zero past the last page), loaded one step ahead
        auto load_scales = [&](int i, float (&k2)[2], float (&v2)[2]) {
#pragma unroll
            for (int hh = 0; hh < 2; hh++) {
                k2[hh] = 0.0f;
                v2[hh] = 0.0f;
                if (2 * i + hh < npages) {
                    const int pg = page_of(2 * i + hh);
                    k2[hh] = p.k_scales[(int64_t)pg * H + h];
                    v2[hh] = p.v_scales[(int64_t)pg * H + h];
                }
            }
        };
        float sk[2] = {0.0f, 0.0f}, sv[2] = {0.0f, 0.0f};
        if (nst > 0) load_scales(lo, sk, sv);
        for (int j = 0; j < nst; j++) {
            const int i = lo + j;  // the step (keys 128 i .. 128 i + 127)
            float nsk[2] = {0.0f, 0.0f}, nsv[2] = {0.0f, 0.0f};
            if (j + 1 < nst) load_scales(i + 1, nsk, nsv);
            ok = __all_sync(kFull, mbar_wait_bounded(&sm.s_full[t], (uint32_t)(j & 1)));
            if (!ok) break;
            tc_fence_after();
            const bool diag = i * kStepKeys + kStepKeys - 1 > tile_qpos0;  // keys past some row's position
            // raw scores q . code of keys 64 hh .. 64 hh + 63 of the step: sign-flipped for a
            // negative softmax scale (the key scale is applied in the exponent, >= 0), masked
            auto load_half = [&](int hh, float (&sc)[64]) {
                uint32_t r[4][16];
#pragma unroll
                for (int c = 0; c < 4; c++) tmem_ld16_async(lane_tm + 64 * hh + 16 * c, r[c]);
                tmem_ld_wait();
#pragma unroll
                for (int c = 0; c < 4; c++)
#pragma unroll
                    for (int x = 0; x < 16; x++) sc[16 * c + x] = __uint_as_float(r[c][x]);
                if (neg_scale) {
#pragma unroll
                    for (int x = 0; x < 64; x++) sc[x] = -sc[x];
                }
                if (diag) {
                    const int k0 = i * kStepKeys + 64 * hh;
#pragma unroll
                    for (int x = 0; x < 64; x++)
                        if (k0 + x > qpos) sc[x] = -INFINITY;
                }
            };
            auto half_max = [&](const float (&sc)[64], float sk_h) {  // max of raw * sk_h, -inf if all masked
                float m8[8];  // independent maxima of 8 scores each (three-input max), then a tree
#pragma unroll
                for (int x = 0; x < 8; x++) {
                    const float *v = sc + 8 * x;
                    m8[x] = max3(max3(v[0], v[1], v[2]), max3(v[3], v[4], v[5]), fmaxf(v[6], v[7]));
                }
                const float mraw = max3(max3(m8[0], m8[1], m8[2]), max3(m8[3], m8[4], m8[5]), fmaxf(m8[6], m8[7]));
                return mraw == -INFINITY ? -INFINITY : mraw * sk_h;
            };
            const float cur_sk[2] = {fmaxf(sk[0] * sabs, kMinScale), fmaxf(sk[1] * sabs, kMinScale)};
            // the row maximum over the step: the second half first, then the first half, which is
            // kept for its P (three loads of 64 columns instead of four)
            float sc0[64];
            float mx;
            {
                float sc1[64];
                load_half(1, sc1);
                mx = half_max(sc1, cur_sk[1]);
            }
            load_half(0, sc0);
            mx = fmaxf(mx, half_max(sc0, cur_sk[0]));
            float factor = 1.0f;
            if (j == 0) {
                m_used = mx;  // finite from key 0 on; -inf in a half before some rows' first key
            } else if (mx > m_used + kLazy) {
                factor = ex2_approx(m_used - mx);
                m_used = mx;
            }
            // P * sv / s_ref = 2^(raw * sk - m + log2(sv / s_ref)), one FMA per element before
            // ex2, as fp16 pairs over columns 32 hh .. 32 hh + 31 (S of keys already read: the
            // first half's P goes over its own first 32 columns, the second half is loaded again
            // before its P covers the first half's last 32); the row sum of P is that sum times
            // s_ref / sv (all-zero values add to l only)
            float l_add = 0.0f;
            auto half_p = [&](int hh, const float (&sc)[64]) {
                const float ratio = sv[hh] / s_ref;
                // a row with no key yet (m = -inf): every score here is -inf and P is 0
                const float off = m_used == -INFINITY ? 0.0f : ratio > 0.0f ? m_used - __log2f(ratio) : m_used;
                // the exponent arguments and the partial sums two keys at a time (f32x2)
                const uint64_t sk2 = pk2(cur_sk[hh], cur_sk[hh]), noff2 = pk2(-off, -off);
                uint64_t ps2[2] = {pk2(0.0f, 0.0f), pk2(0.0f, 0.0f)};
#pragma unroll
                for (int q = 0; q < 2; q++) {  // two stores of 16 columns
                    float w[16];
#pragma unroll
                    for (int cc = 0; cc < 16; cc++) {
                        const int c = 16 * q + cc;
                        float x0, x1;
                        upk2(fma2(pk2(sc[2 * c], sc[2 * c + 1]), sk2, noff2), x0, x1);
                        const float p0 = ex2_approx(x0), p1 = ex2_approx(x1);
                        ps2[c & 1] = add2(ps2[c & 1], pk2(p0, p1));
                        w[cc] = __uint_as_float(f16x2_rn(p0, p1));
                    }
                    tmem_st16(lane_tm + 32 * hh + 16 * q, w);
                }
                float pa, pb, pc, pd;
                upk2(ps2[0], pa, pb);
                upk2(ps2[1], pc, pd);
                const float psum = (pa + pb) + (pc + pd);
                l_add += ratio > 0.0f ? psum / ratio : psum;
            };
            half_p(0, sc0);
            {
                float sc1[64];
                load_half(1, sc1);
                half_p(1, sc1);
            }
            asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory");
            // O holds PV(i - 1) (complete before S(i) was issued): rescale the rows whose max moved
            if (__any_sync(kFull, factor != 1.0f)) {
#pragma unroll
                for (int c = 0; c < 8; c++) {
                    float v[16];
                    tmem_ld16(lane_tm + 128 + 16 * c, v);
#pragma unroll
                    for (int x = 0; x < 16; x++) v[x] *= factor;
                    tmem_st16(lane_tm + 128 + 16 * c, v);
                }
                asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory");
            }
            tc_fence_before();
            mbar_arrive(&sm.p_full[t]);
            l_run = l_run * factor + l_add;
#pragma unroll
            for (int hh = 0; hh < 2; hh++) {
                sk[hh] = nsk[hh];
                sv[hh] = nsv[hh];
            }
        }
        if (ok && nst > 0)  // O is final after the tile's last PV
            ok = __all_sync(kFull, mbar_wait_bounded(&sm.o_done[t], (uint32_t)((nst - 1) & 1)));
        if (ok) {
            tc_fence_after();
            const int tile_rows = rows - kTcRows * t;
            if (half < 0 && nst > 0) {  // out = s_ref * O / l; loads warp-wide, stores per row
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
            } else if (half >= 0) {  // this half's partial of the row: m, l and s_ref * O (zero if no step)
                float *pr = p.partials + (((int64_t)(unit - p.num_full) * 2 + half) * (kTiles * kTcRows) +
                                          kTcRows * t + row) * kPartialFloats;
#pragma unroll
                for (int c = 0; c < 8; c++) {
                    float v[16];
                    if (nst > 0) {
                        tmem_ld16(lane_tm + 128 + 16 * c, v);
                    } else {
#pragma unroll
                        for (int x = 0; x < 16; x++) v[x] = 0.0f;
                    }
                    if (row >= tile_rows) continue;
#pragma unroll
                    for (int x = 0; x < 16; x += 4)
                        *reinterpret_cast<float4 *>(pr + 4 + 16 * c + x) =
                            make_float4(v[x] * s_ref, v[x + 1] * s_ref, v[x + 2] * s_ref, v[x + 3] * s_ref);
                }
                if (row < tile_rows) *reinterpret_cast<float4 *>(pr) = make_float4(m_used, l_run, 0.0f, 0.0f);
            }
        }
    } else if (warp < kTiles * kPfWarps + kWidenThreads / 32) {
        // ---- widening: the step's two pages -> fp16 codes in stage i & 1 ----
        // K and V of a stage are widened and released separately: S needs a step's K (its
        // buffer free once the S two steps back completed), PV its V (free once that step's
        // PV completed).  Each thread loads 16-byte pieces of the step's two pages straight
        // into registers -- V while K is converted, the next step's K while V is converted.
        // Piece r of thread w: key and 16-byte piece of the key's row chosen so that the 8
        // threads of a quarter-warp store to 8 different 16-byte bank groups (int4: 4 keys x
        // 2 pieces; int8, FP8: 2 keys x 4 pieces).
        const int w = tid - kTiles * kPfWarps * 32;
        constexpr int kLd = kPageBytes / (16 * kWidenThreads);  // 16-byte pieces per thread, per K and V
        constexpr int kChunkBytes = RB / 16;                    // bytes of 8 codes
        auto piece_key = [&](int r) {
            return RB == 64 ? 4 * (w >> 3) + ((w & 7) >> 1) : 2 * (w >> 3) + ((w & 7) >> 2) + 32 * (r & 1);
        };
        auto piece_col = [&](int r) { return RB == 64 ? (w & 1) + 2 * r : (w & 3) + 4 * (r >> 1); };
        uint4 kr[2][kLd], vr[2][kLd];  // the step's two pages (zero past the last page)
        auto load = [&](const uint8_t *codes, int pg, uint4 (&d)[kLd]) {
            if (pg >= npages) {
#pragma unroll
                for (int r = 0; r < kLd; r++) d[r] = make_uint4(0u, 0u, 0u, 0u);
                return;
            }
            const size_t off = ((size_t)page_of(pg) * H + h) * kPageBytes;
#pragma unroll
            for (int r = 0; r < kLd; r++) d[r] = ld_stream_v4(codes + off + piece_key(r) * RB + 16 * piece_col(r));
        };
        // the step's two pages -> dst (keys x elements; the same bytes for K and V)
        auto widen_step = [&](uint8_t *dst, const uint4 (&src)[2][kLd]) {
#pragma unroll
            for (int hh = 0; hh < 2; hh++)
#pragma unroll
                for (int r = 0; r < kLd; r++) {
                    const int key = kPage * hh + piece_key(r), c0 = piece_col(r) * (16 / kChunkBytes);
                    uint4 x[16 / kChunkBytes];
                    widen16<FMT>(src[hh][r], x);
#pragma unroll
                    for (int xx = 0; xx < 16 / kChunkBytes; xx++)
                        *reinterpret_cast<uint4 *>(dst + k_chunk(key, c0 + xx)) = x[xx];
                }
        };
        if (nloc > 0) {
            load(p.k_codes, 2 * lo, kr[0]);
            load(p.k_codes, 2 * lo + 1, kr[1]);
        }
        for (int j = 0; j < nloc; j++) {
            const int i = lo + j, s = j & 1;
            load(p.v_codes, 2 * i, vr[0]);
            load(p.v_codes, 2 * i + 1, vr[1]);
            bool got = j < 2 || mbar_wait_bounded(&sm.k_free[s], (uint32_t)(((j >> 1) - 1) & 1));
            if (!widen_group_all(got)) {
                ok = false;
                break;
            }
            widen_step(sm.k[s], kr);
            fence_proxy_async_smem();  // the MMAs read stage s through the async proxy
            mbar_arrive(&sm.k_ready[s]);
            if (j + 1 < nloc) {
                load(p.k_codes, 2 * i + 2, kr[0]);
                load(p.k_codes, 2 * i + 3, kr[1]);
            }
            got = j < 2 || mbar_wait_bounded(&sm.v_free[s], (uint32_t)(((j >> 1) - 1) & 1));
            if (!widen_group_all(got)) {
                ok = false;
                break;
            }
            widen_step(sm.v[s], vr);
            fence_proxy_async_smem();
            mbar_arrive(&sm.v_ready[s]);
        }
    } else if ((tid & 31) == 0) {
        // ---- the MMA thread ----
        // descriptor halves of the operands' first k-step (per tile, per stage), computed once
        static_assert(kTiles == 2, "one descriptor register per tile");
        const uint32_t dq_lo0 = (uint32_t)umma_desc(smem_addr(sm.q[0])), dq_lo1 = (uint32_t)umma_desc(smem_addr(sm.q[1]));
        const uint32_t dk_lo0 = (uint32_t)umma_desc(smem_addr(sm.k[0])), dk_lo1 = (uint32_t)umma_desc(smem_addr(sm.k[1]));
        const uint32_t dv_lo0 = (uint32_t)umma_desc_mn(smem_addr(sm.v[0]), kStepKeys * 128, 1024);
        const uint32_t dv_lo1 = (uint32_t)umma_desc_mn(smem_addr(sm.v[1]), kStepKeys * 128, 1024);
        const uint32_t dsw_hi = (uint32_t)(umma_desc(smem_addr(sm.q[0])) >> 32);  // SBO, version, swizzle
        const uint32_t dv_hi = (uint32_t)(umma_desc_mn(smem_addr(sm.v[0]), kStepKeys * 128, 1024) >> 32);
        auto issue_s = [&](int t, int i) {  // S(i) = Q K(i)^T of tile t: 128 x 128 keys, 8 MMAs of K = 16
            const uint32_t aq = t == 0 ? dq_lo0 : dq_lo1, ak = (i & 1) ? dk_lo1 : dk_lo0;
#pragma unroll
            for (int ks = 0; ks < 8; ks++) {
                // k-step ks: elements 16 ks .. 16 ks + 15 = 32-byte column (ks & 3) of 64-element block ks >> 2
                umma_f16_ss(tmem + 256 * t, aq + (uint32_t)(((ks >> 2) * (kTcRows * 128) + (ks & 3) * 32) >> 4), dsw_hi,
                            ak + (uint32_t)(((ks >> 2) * (kStepKeys * 128) + (ks & 3) * 32) >> 4), dsw_hi, kIdescS,
                            ks > 0 ? 1u : 0u);
            }
            umma_commit(&sm.s_full[t]);
        };
        auto issue_pv = [&](int t, int i) {  // O += P(i) V(i): P from tensor memory, 8 columns per 16 keys
            const uint32_t tt = tmem + 256 * t, av = (i & 1) ? dv_lo1 : dv_lo0;
#pragma unroll
            for (int ks = 0; ks < 8; ks++)
                umma_f16_ts(tt + 128, tt + 8 * ks, av + (uint32_t)((ks * 16 * 128) >> 4), dv_hi, kIdescO,
                             (i > 0 || ks > 0) ? 1u : 0u);
            umma_commit(&sm.o_done[t]);
        };
        // steps are counted from the CTA's first (stage, barrier phase, accumulate flag); the
        // last tile (which has every step) issues a step's last S and last PV, after which
        // the stage's K, V are released
        if (nloc > 0) {
            ok = mbar_wait_bounded(&sm.k_ready[0], 0u);
            tc_fence_after();
            if (ok) {
                for (int t = 0; t < active; t++)
                    if (local_steps(t) > 0) issue_s(t, 0);
                umma_commit(&sm.k_free[0]);
            }
        }
        for (int i = 0; i < nloc && ok; i++) {
            bool v_seen = false, k_seen = false;
            for (int t = 0; t < active && ok; t++) {
                const int nst = local_steps(t);
                if (i >= nst) continue;
                ok = mbar_wait_bounded(&sm.p_full[t], (uint32_t)(i & 1));
                if (ok && !v_seen) {
                    ok = mbar_wait_bounded(&sm.v_ready[i & 1], (uint32_t)((i >> 1) & 1));
                    v_seen = true;
                }
                if (!ok) break;
                tc_fence_after();
                issue_pv(t, i);
                if (t == active - 1) umma_commit(&sm.v_free[i & 1]);
                if (i + 1 < nst) {
                    // S(i + 1) goes where P(i) is: only after PV(i) has read it
                    ok = mbar_wait_bounded(&sm.o_done[t], (uint32_t)(i & 1));
                    if (ok && !k_seen) {
                        ok = mbar_wait_bounded(&sm.k_ready[(i + 1) & 1], (uint32_t)(((i + 1) >> 1) & 1));
                        k_seen = true;
                    }
                    if (!ok) break;
                    tc_fence_after();
                    issue_s(t, i + 1);
                    if (t == active - 1) umma_commit(&sm.k_free[(i + 1) & 1]);
                }
            }
        }
        umma_commit(&sm.mma_done);  // whatever was issued completes before tensor memory is freed
        if (!mbar_wait_bounded(&sm.mma_done, 0u)) ok = false;
    }
    __syncwarp();
    if (!ok) set_flag(p.status, KVQ_FLAG_TIMEOUT);
    tc_fence_before();
    __syncthreads();  // every partial row of a split half is written
    if (warp == 0) asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem), "r"(kTmemCols));
    if (half < 0) return;
    // Split halves: count this half on the unit's counter (release of its partials, acquire of
    // the other's); the second to arrive merges the two partials of each row and puts the
    // counter back to zero, so it starts every launch at zero once the workspace was zero-filled.
    uint32_t *counter = p.counters + (unit - p.num_full);
    if (tid == 0) {
        __threadfence();
        uint32_t old;
        asm volatile("atom.acq_rel.gpu.global.add.u32 %0, [%1], 1;" : "=r"(old) : "l"(counter) : "memory");
        if (old > 1) set_flag(p.status, KVQ_FLAG_BAD_WORKSPACE);  // not zero-filled, or an aborted launch
        if (old == 1) *counter = 0u;
        sm.ticket = old;
    }
    __syncthreads();
    if (sm.ticket != 1u || warp >= kTiles * kPfWarps || tid >= rows) return;
    // out = (sum_h 2^(m_h - M) s_ref_h O_h) / (sum_h 2^(m_h - M) l_h), M = max_h m_h; a half
    // with no key for the row has m = -inf and weight 0 (half 0 always holds key 0)
    const float *pa = p.partials + ((int64_t)(unit - p.num_full) * 2 * (kTiles * kTcRows) + tid) * kPartialFloats;
    const float *pb = pa + (int64_t)(kTiles * kTcRows) * kPartialFloats;
    const float4 ha = __ldcg(reinterpret_cast<const float4 *>(pa));
    const float4 hb = __ldcg(reinterpret_cast<const float4 *>(pb));
    const float mm = fmaxf(ha.x, hb.x);
    const float wa = ha.x == -INFINITY ? 0.0f : ex2_approx(ha.x - mm);
    const float wb = hb.x == -INFINITY ? 0.0f : ex2_approx(hb.x - mm);
    const float inv = 1.0f / (ha.y * wa + hb.y * wb);
    uint16_t *dst = p.out + ((int64_t)(c0 + i0 + tid) * Hq + hq) * kHeadDim;
#pragma unroll 4
    for (int c = 0; c < kHeadDim; c += 8) {
        const float4 a0 = __ldcg(reinterpret_cast<const float4 *>(pa + 4 + c));
        const float4 a1 = __ldcg(reinterpret_cast<const float4 *>(pa + 8 + c));
        const float4 b0 = __ldcg(reinterpret_cast<const float4 *>(pb + 4 + c));
        const float4 b1 = __ldcg(reinterpret_cast<const float4 *>(pb + 8 + c));
        uint4 o;
        o.x = f16x2_rn((a0.x * wa + b0.x * wb) * inv, (a0.y * wa + b0.y * wb) * inv);
        o.y = f16x2_rn((a0.z * wa + b0.z * wb) * inv, (a0.w * wa + b0.w * wb) * inv);
        o.z = f16x2_rn((a1.x * wa + b1.x * wb) * inv, (a1.y * wa + b1.y * wb) * inv);
        o.w = f16x2_rn((a1.z * wa + b1.z * wb) * inv, (a1.w * wa + b1.w * wb) * inv);
        *reinterpret_cast<uint4 *>(dst + c) = o;
    }
}

template <int FMT>
static cudaError_t launch_prefill_tc(const PrefillParams &p, cudaStream_t s)
{
    const size_t smem = sizeof(TcSmem<FMT>) + 1024;  // + room to align the tiles to 1024 bytes
    cudaError_t e = cudaFuncSetAttribute(prefill_attn_tc_kernel<FMT>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         (int)smem);
    if (e != cudaSuccess) return e;
    const int64_t units = (int64_t)p.units_x * p.num_q_heads * p.num_seqs;
    const dim3 grid((unsigned)(p.num_full + 2 * (units - p.num_full)));
    return launch_plain(prefill_attn_tc_kernel<FMT>, grid, dim3(kTcThreads), smem, s, p);
}

int64_t prefill_units(int num_q_heads, int num_seqs, int max_q)
{
    return (int64_t)((max_q + kTiles * kTcRows - 1) / (kTiles * kTcRows)) * num_q_heads * num_seqs;
}

// A unit takes about as long as its chain of key steps, so a last wave of r < num_sms units
// would leave num_sms - r SMs idle for a whole unit; split in halves it takes half as long.
int64_t prefill_split_units(int64_t units, int num_sms)
{
    if (num_sms <= 0) return 0;
    return units >= num_sms ? units % num_sms : units;
}

size_t prefill_workspace_bytes(int64_t split_units)
{
    const size_t counters = ((size_t)split_units * sizeof(uint32_t) + 255) / 256 * 256;
    return counters + (size_t)split_units * 2 * (kTiles * kTcRows) * kPartialFloats * sizeof(float);
}

cudaError_t launch_prefill(int fmt, const PrefillParams &p, cudaStream_t s)
{
    if (p.num_seqs == 0 || p.max_q == 0) return cudaSuccess;
    if (fmt == KVQ_INT4_B64) return launch_prefill_tc<KVQ_INT4_B64>(p, s);
    if (fmt == KVQ_FP8_E4M3) return launch_prefill_tc<KVQ_FP8_E4M3>(p, s);
    return launch_prefill_tc<KVQ_INT8_PAGE>(p, s);
}

}  // namespace kvq
