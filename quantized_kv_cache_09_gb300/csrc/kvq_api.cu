// kvq_api.cu -- the C ABI declared in include/kvq.h: host-side argument checks,
// sub-batching, and launches of the kernels on the caller's stream.  No device
// memory is allocated here; every buffer belongs to the caller.
#include <cuda_runtime.h>
#include <math.h>
#include <stdint.h>

#include <atomic>

#include "kvq.h"
#include "kvq_internal.h"
#include "kvq_testing.h"

namespace {

bool aligned16(const void *p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

kvq_status from_cuda(cudaError_t e) { return e == cudaSuccess ? KVQ_OK : KVQ_ERR_CUDA; }

bool fmt_ok(int fmt) { return fmt == KVQ_INT4_B64 || fmt == KVQ_INT8_PAGE || fmt == KVQ_FP8_E4M3; }

kvq_status check_cache(const kvq_cache *c)
{
    if (!c) return KVQ_ERR_INVALID_ARG;
    if (!fmt_ok(c->fmt)) return KVQ_ERR_UNSUPPORTED;
    if (c->head_dim != kvq::kHeadDim || c->page_tokens != kvq::kPage) return KVQ_ERR_UNSUPPORTED;
    if (c->num_heads <= 0 || c->num_pages <= 0) return KVQ_ERR_INVALID_ARG;
    if (!c->k_codes || !c->v_codes || !c->k_scales || !c->v_scales) return KVQ_ERR_INVALID_ARG;
    if (!aligned16(c->k_codes) || !aligned16(c->v_codes)) return KVQ_ERR_INVALID_ARG;
    if ((c->k_tail && !aligned16(c->k_tail)) || (c->v_tail && !aligned16(c->v_tail))) return KVQ_ERR_INVALID_ARG;
    if ((c->k_tail == nullptr) != (c->v_tail == nullptr)) return KVQ_ERR_INVALID_ARG;
    return KVQ_OK;
}

// test hook state (kvq_testing.h): read when a decode launch is set up
std::atomic<uint32_t> g_test_wait_limit_us{0};
std::atomic<int32_t> g_test_skip_chunk{-1};

}  // namespace

namespace kvq {
void decode_test_settings(unsigned long long *wait_limit_ns, int32_t *skip_chunk)
{
    const uint32_t us = g_test_wait_limit_us.load(std::memory_order_relaxed);
    *wait_limit_ns = us ? (unsigned long long)us * 1000ull : kvq::kDecodeWaitLimitNs;
    *skip_chunk = g_test_skip_chunk.load(std::memory_order_relaxed);
}
}  // namespace kvq

extern "C" {

kvq_status kvq_quantize(kvq_format fmt, const uint16_t *x, int64_t num_tokens, int32_t num_heads,
                        int32_t head_dim, uint8_t *codes, float *scales, kvq_stream_t stream)
{
    if (!fmt_ok(fmt) || head_dim != kvq::kHeadDim) return KVQ_ERR_UNSUPPORTED;
    if (num_tokens < 0 || num_heads <= 0) return KVQ_ERR_INVALID_ARG;
    if (num_tokens == 0) return KVQ_OK;
    if (!x || !codes || !scales || !aligned16(x) || !aligned16(codes)) return KVQ_ERR_INVALID_ARG;
    return from_cuda(kvq::launch_quantize(fmt, x, num_tokens, num_heads, codes, scales,
                                          reinterpret_cast<cudaStream_t>(stream)));
}

kvq_status kvq_append(const kvq_cache *cache, const uint16_t *k_new, const uint16_t *v_new,
                      const int32_t *cu_seqlens, const int32_t *block_table, int32_t max_blocks_per_seq,
                      const int32_t *seq_lens_before, int32_t num_seqs, int64_t total_new_tokens,
                      int32_t max_new_tokens, kvq_stream_t stream)
{
    kvq_status st = check_cache(cache);
    if (st != KVQ_OK) return st;
    if (num_seqs < 0 || max_new_tokens < 0 || max_blocks_per_seq <= 0 || total_new_tokens < 0)
        return KVQ_ERR_INVALID_ARG;
    if (num_seqs == 0 || max_new_tokens == 0) return KVQ_OK;
    if (!k_new || !v_new || !cu_seqlens || !block_table || !seq_lens_before) return KVQ_ERR_INVALID_ARG;
    if (!aligned16(k_new) || !aligned16(v_new)) return KVQ_ERR_INVALID_ARG;
    if (cache->k_tail && num_seqs > cache->max_seqs) return KVQ_ERR_INVALID_ARG;
    kvq::AppendParams p;
    p.k_new = k_new;
    p.v_new = v_new;
    p.cu_seqlens = cu_seqlens;
    p.block_table = block_table;
    p.seq_lens_before = seq_lens_before;
    p.k_codes = cache->k_codes;
    p.v_codes = cache->v_codes;
    p.k_scales = cache->k_scales;
    p.v_scales = cache->v_scales;
    p.k_tail = cache->k_tail;
    p.v_tail = cache->v_tail;
    p.status = cache->status;
    p.num_heads = cache->num_heads;
    p.num_pages = cache->num_pages;
    p.max_blocks = max_blocks_per_seq;
    p.max_new_tokens = max_new_tokens;
    p.total_new = total_new_tokens;
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    // grid.y holds the sequence: launch in slices of at most 65535 sequences
    for (int32_t b0 = 0; b0 < num_seqs; b0 += 65535) {
        kvq::AppendParams q = p;
        q.num_seqs = (num_seqs - b0) < 65535 ? (num_seqs - b0) : 65535;
        q.cu_seqlens = cu_seqlens + b0;
        q.block_table = block_table + (int64_t)b0 * max_blocks_per_seq;
        q.seq_lens_before = seq_lens_before + b0;
        if (q.k_tail) {
            q.k_tail = cache->k_tail + (int64_t)b0 * cache->num_heads * kvq::kPage * kvq::kHeadDim;
            q.v_tail = cache->v_tail + (int64_t)b0 * cache->num_heads * kvq::kPage * kvq::kHeadDim;
        }
        cudaError_t e = kvq::launch_append(cache->fmt, q, s);
        if (e != cudaSuccess) return KVQ_ERR_CUDA;
    }
    return KVQ_OK;
}

// query heads per cache head, or 0 when num_q_heads is not a supported
// multiple of num_kv_heads
static int group_of(int fmt, int32_t num_kv_heads, int32_t num_q_heads)
{
    if (num_kv_heads <= 0 || num_q_heads <= 0 || num_q_heads % num_kv_heads) return 0;
    const int g = num_q_heads / num_kv_heads;
    return kvq::decode_group_supported(fmt, g) ? g : 0;
}

size_t kvq_decode_workspace_bytes(kvq_format fmt, int32_t num_heads, int32_t head_dim)
{
    return kvq_decode_workspace_bytes_gqa(fmt, num_heads, num_heads, head_dim);
}

size_t kvq_decode_workspace_bytes_gqa(kvq_format fmt, int32_t num_kv_heads, int32_t num_q_heads, int32_t head_dim)
{
    if (!fmt_ok(fmt) || head_dim != kvq::kHeadDim) return 0;
    const int g = group_of(fmt, num_kv_heads, num_q_heads);
    if (g == 0) return 0;
    return kvq::decode_workspace_bytes(fmt, g);
}

kvq_status kvq_decode_attention(const kvq_cache *cache, const uint16_t *q, const int32_t *block_table,
                                int32_t max_blocks_per_seq, const int32_t *seq_lens, int32_t num_seqs,
                                float softmax_scale, uint16_t *out, void *workspace, size_t workspace_bytes,
                                kvq_stream_t stream)
{
    if (!cache) return KVQ_ERR_INVALID_ARG;
    return kvq_decode_attention_gqa(cache, q, cache->num_heads, block_table, max_blocks_per_seq, seq_lens,
                                    num_seqs, softmax_scale, out, workspace, workspace_bytes, stream);
}

kvq_status kvq_decode_attention_gqa(const kvq_cache *cache, const uint16_t *q, int32_t num_q_heads,
                                    const int32_t *block_table, int32_t max_blocks_per_seq, const int32_t *seq_lens,
                                    int32_t num_seqs, float softmax_scale, uint16_t *out, void *workspace,
                                    size_t workspace_bytes, kvq_stream_t stream)
{
    kvq_status st = check_cache(cache);
    if (st != KVQ_OK) return st;
    if (num_seqs < 0 || max_blocks_per_seq <= 0 || !isfinite(softmax_scale)) return KVQ_ERR_INVALID_ARG;
    if (num_q_heads <= 0 || num_q_heads % cache->num_heads) return KVQ_ERR_INVALID_ARG;
    // the split counts units of a (sequence, head) in 24 bits: at most 2^22 pages of 64 tokens
    if (max_blocks_per_seq > (1 << 22)) return KVQ_ERR_UNSUPPORTED;
    const int g = group_of(cache->fmt, cache->num_heads, num_q_heads);
    if (g == 0) return KVQ_ERR_UNSUPPORTED;
    {  // the units of one launch (at most 4 per page, per unit head) are counted in 32 bits
        const int64_t unit_heads = (int64_t)cache->num_heads * (g == 1 || g == 2 || g == 4 ? 1 : (g + 15) / 16);
        const int64_t seqs = num_seqs < kvq::kMaxSeqsPerLaunch ? num_seqs : kvq::kMaxSeqsPerLaunch;
        if ((int64_t)max_blocks_per_seq * 4 * unit_heads * seqs > INT32_MAX) return KVQ_ERR_UNSUPPORTED;
    }
    if (num_seqs == 0) return KVQ_OK;
    if (!q || !block_table || !seq_lens || !out || !aligned16(q) || !aligned16(out)) return KVQ_ERR_INVALID_ARG;
    const size_t need = kvq::decode_workspace_bytes(cache->fmt, g);
    if (need == 0) return KVQ_ERR_CUDA;
    if (!workspace || !aligned16(workspace) || workspace_bytes < need) return KVQ_ERR_WORKSPACE;
    kvq::DecodeParams p;
    p.k_codes = cache->k_codes;
    p.v_codes = cache->v_codes;
    p.k_scales = cache->k_scales;
    p.v_scales = cache->v_scales;
    p.status = cache->status;
    p.num_heads = cache->num_heads;
    p.num_pages = cache->num_pages;
    p.max_blocks = max_blocks_per_seq;
    p.score_scale = softmax_scale * 1.4426950408889634f;
    p.group = g;
    p.counters = reinterpret_cast<unsigned long long *>(workspace);
    p.partials = reinterpret_cast<float *>(reinterpret_cast<char *>(workspace) + kvq::decode_counter_bytes());
    kvq::decode_test_settings(&p.wait_limit_ns, &p.test_skip_chunk);
    const int64_t HD = (int64_t)num_q_heads * kvq::kHeadDim;
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    for (int32_t b0 = 0; b0 < num_seqs; b0 += kvq::kMaxSeqsPerLaunch) {
        kvq::DecodeParams d = p;
        d.num_seqs = (num_seqs - b0) < kvq::kMaxSeqsPerLaunch ? (num_seqs - b0) : kvq::kMaxSeqsPerLaunch;
        d.q = q + b0 * HD;
        d.out = out + b0 * HD;
        d.seq_lens = seq_lens + b0;
        d.block_table = block_table + (int64_t)b0 * max_blocks_per_seq;
        d.epoch = kvq::decode_next_epoch();
        cudaError_t e = kvq::launch_decode(cache->fmt, d, s);
        if (e != cudaSuccess) return KVQ_ERR_CUDA;
    }
    return KVQ_OK;
}

static int device_sms()
{
    int dev = 0, n = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return 0;
    if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) return 0;
    return n;
}

size_t kvq_prefill_workspace_bytes(int32_t num_q_heads, int32_t num_seqs, int32_t max_q_per_seq)
{
    if (num_q_heads <= 0 || num_seqs <= 0 || max_q_per_seq <= 0) return 0;
    const int64_t units = kvq::prefill_units(num_q_heads, num_seqs, max_q_per_seq);
    return kvq::prefill_workspace_bytes(kvq::prefill_split_units(units, device_sms()));
}

kvq_status kvq_prefill_attention(const kvq_cache *cache, const uint16_t *q, int32_t num_q_heads,
                                 const int32_t *cu_seqlens_q, int64_t total_q, int32_t max_q_per_seq,
                                 const int32_t *block_table, int32_t max_blocks_per_seq, const int32_t *seq_lens,
                                 int32_t num_seqs, float softmax_scale, uint16_t *out, void *workspace,
                                 size_t workspace_bytes, kvq_stream_t stream)
{
    kvq_status st = check_cache(cache);
    if (st != KVQ_OK) return st;
    if (num_seqs < 0 || max_q_per_seq < 0 || total_q < 0 || max_blocks_per_seq <= 0 || !isfinite(softmax_scale))
        return KVQ_ERR_INVALID_ARG;
    if (num_q_heads <= 0 || num_q_heads % cache->num_heads) return KVQ_ERR_INVALID_ARG;
    if (num_seqs == 0 || max_q_per_seq == 0 || total_q == 0) return KVQ_OK;
    if (!q || !out || !cu_seqlens_q || !block_table || !seq_lens || !aligned16(q) || !aligned16(out))
        return KVQ_ERR_INVALID_ARG;
    if (num_seqs > 65535 || num_q_heads > 65535) return KVQ_ERR_UNSUPPORTED;
    kvq::PrefillParams p;
    p.k_codes = cache->k_codes;
    p.v_codes = cache->v_codes;
    p.k_scales = cache->k_scales;
    p.v_scales = cache->v_scales;
    p.q = q;
    p.out = out;
    p.cu_q = cu_seqlens_q;
    p.seq_lens = seq_lens;
    p.block_table = block_table;
    p.status = cache->status;
    p.num_seqs = num_seqs;
    p.num_heads = cache->num_heads;
    p.num_q_heads = num_q_heads;
    p.group = num_q_heads / cache->num_heads;
    p.num_pages = cache->num_pages;
    p.max_blocks = max_blocks_per_seq;
    p.max_q = max_q_per_seq;
    p.total_q = total_q;
    p.score_scale = softmax_scale * 1.4426950408889634f;
    const int64_t units = kvq::prefill_units(num_q_heads, num_seqs, max_q_per_seq);
    if (units > INT32_MAX / 2) return KVQ_ERR_UNSUPPORTED;
    p.units_x = (int)(units / ((int64_t)num_q_heads * num_seqs));
    p.num_full = (int)units;
    p.partials = nullptr;
    p.counters = nullptr;
    if (workspace) {  // split the last wave's units
        const int64_t split = kvq::prefill_split_units(units, device_sms());
        if (workspace_bytes < kvq::prefill_workspace_bytes(split) || !aligned16(workspace)) return KVQ_ERR_WORKSPACE;
        const size_t counters = (size_t)split * sizeof(uint32_t);
        p.num_full = (int)(units - split);
        p.counters = static_cast<uint32_t *>(workspace);
        p.partials = reinterpret_cast<float *>(static_cast<uint8_t *>(workspace) + (counters + 255) / 256 * 256);
    }
    return from_cuda(kvq::launch_prefill(cache->fmt, p, reinterpret_cast<cudaStream_t>(stream)));
}

kvq_status kvq_get_device_status(const kvq_cache *cache, kvq_stream_t stream, int32_t *flags_out)
{
    if (!cache) return KVQ_ERR_INVALID_ARG;
    int32_t flags = 0;
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    if (cache->status) {
        if (cudaMemcpyAsync(&flags, cache->status, sizeof(int32_t), cudaMemcpyDeviceToHost, s) != cudaSuccess)
            return KVQ_ERR_CUDA;
        if (cudaStreamSynchronize(s) != cudaSuccess) return KVQ_ERR_CUDA;
        if (flags && cudaMemsetAsync(cache->status, 0, sizeof(int32_t), s) != cudaSuccess) return KVQ_ERR_CUDA;
        if (cudaStreamSynchronize(s) != cudaSuccess) return KVQ_ERR_CUDA;
    } else if (cudaStreamSynchronize(s) != cudaSuccess) {
        return KVQ_ERR_CUDA;
    }
    if (flags_out) *flags_out = flags;
    if (flags & KVQ_FLAG_BAD_PAGE) return KVQ_ERR_BAD_BLOCK_TABLE;
    if (flags & KVQ_FLAG_BAD_LENGTH) return KVQ_ERR_BAD_LENGTH;
    if (flags & KVQ_FLAG_TIMEOUT) return KVQ_ERR_TIMEOUT;
    if (flags & KVQ_FLAG_BAD_WORKSPACE) return KVQ_ERR_WORKSPACE;
    if (flags & (KVQ_FLAG_NO_TAIL | KVQ_FLAG_BAD_APPEND)) return KVQ_ERR_BAD_LENGTH;
    return KVQ_OK;
}

kvq_status kvq_testing_set_decode_fault(uint32_t wait_limit_us, int32_t skip_chunk)
{
    if (skip_chunk < -1) return KVQ_ERR_INVALID_ARG;
    g_test_wait_limit_us.store(wait_limit_us, std::memory_order_relaxed);
    g_test_skip_chunk.store(skip_chunk, std::memory_order_relaxed);
    return KVQ_OK;
}

const char *kvq_status_string(kvq_status status)
{
    switch (status) {
    case KVQ_OK: return "ok";
    case KVQ_ERR_INVALID_ARG: return "invalid argument";
    case KVQ_ERR_UNSUPPORTED: return "unsupported shape or format";
    case KVQ_ERR_CUDA: return "CUDA error";
    case KVQ_ERR_BAD_BLOCK_TABLE: return "block-table entry out of range";
    case KVQ_ERR_TIMEOUT: return "bounded wait timed out";
    case KVQ_ERR_WORKSPACE: return "workspace missing, too small or not zero-filled";
    case KVQ_ERR_BAD_LENGTH: return "sequence length or append bounds invalid";
    }
    return "unknown status";
}

int32_t kvq_version(void) { return 100; }

}  // extern "C"
