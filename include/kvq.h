/*
 * kvq.h -- C ABI of the block-quantized KV cache and its decode attention,
 * built for one NVIDIA GB300 GPU (sm_103a).
 *
 * The method (three scraped articles on DeepSeek-R1 inference tuning):
 *   - quantize_block, "DeepSeek-R1 inference latency ... hardware-aware
 *     scheduling" (jsqmd.com/news/887038), section 2.1: per block of 64
 *     tokens, scale = max|x| / 7.5 and codes = round(x / scale) clamped to
 *     [-8, 7];
 *   - the symmetric per-chunk INT8 variant, "DeepSeek R1 performance
 *     overview" (aicoding.csdn.net), section 2.2, and decode reading an INT8
 *     KV cache, same page, section 3.1;
 *   - KV pages addressed through a block table, "DeepSeek R1 performance
 *     tips" (ddd.cn), section 4 (vLLM PagedAttention);
 *   - an FP8 KV cache (same page, section 1) in E4M3 with dynamic range
 *     scaling set by max|x| ("hardware-aware scheduling" page, section 2.2).
 *
 * Readings fixed by this library where the pages are silent or inconsistent:
 *   - a block is (sequence, head, 64 consecutive tokens); the last block of a
 *     sequence is scaled over its valid rows only and its unused rows hold
 *     code 0;
 *   - binary32 arithmetic: scale = a / 7.5f (int4) or a / 127.0f (int8),
 *     y = x / scale, both correctly rounded; code = clamp(rint(y)) with
 *     round-half-to-even; clamp [-8, 7] (int4) or [-127, 127] (int8); no
 *     zero-point; an all-zero block has scale 0 and codes 0;
 *   - int4 codes are packed: byte j of a row holds element 2j in its low
 *     nibble and element 2j+1 in its high nibble, 4-bit two's complement;
 *   - FP8: scale = a / 448.0f (the largest finite E4M3 value), code = the
 *     E4M3 value nearest to y = RN(x / scale), ties to the even fraction,
 *     saturating at +-448, sign kept (-0.0 and negatives that round to zero
 *     give 0x80); one byte per element, stored like int8; an all-zero block
 *     has scale 0 and codes 0x00;
 *   - decode attention is softmax(q . k^ * softmax_scale) . v^ with
 *     k^ = code * scale, one query per (sequence, head); the output of an
 *     empty sequence is 0.
 *
 * Layouts (all little-endian, all pointers device memory unless stated):
 *   fp16 tensors are IEEE binary16 bit patterns (uint16_t).
 *   token rows: x[T][H][D], head_dim D = 128 contiguous per (token, head).
 *   codes of one (page, head): 64 rows of D/2 bytes (int4) or D bytes (int8, FP8);
 *   code arrays: [num_pages][H][64][D/2 or D];  scale arrays: [num_pages][H].
 *
 * Ownership: the caller allocates and frees every buffer, workspaces
 * included; the library allocates no device memory and keeps no state
 * between calls.  Every call is asynchronous on the caller's stream: argument
 * checks run on the host first (a rejected call launches nothing); problems
 * only the device can see (a block-table entry out of range, a length beyond
 * the table, a wait that timed out) set bits in the cache's device status word
 * instead of faulting, and kvq_get_device_status() reads them.
 */
#ifndef KVQ_H
#define KVQ_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* the caller's CUDA stream (a cudaStream_t); NULL is the legacy default stream */
typedef struct CUstream_st *kvq_stream_t;

typedef enum kvq_status {
    KVQ_OK = 0,
    KVQ_ERR_INVALID_ARG = 1,     /* null pointer, negative size, misaligned buffer */
    KVQ_ERR_UNSUPPORTED = 2,     /* head_dim != 128, page_tokens != 64, unknown format */
    KVQ_ERR_CUDA = 3,            /* a CUDA runtime call or launch failed */
    KVQ_ERR_BAD_BLOCK_TABLE = 4, /* device: a block-table entry outside [0, num_pages) */
    KVQ_ERR_TIMEOUT = 5,         /* device: a bounded wait on a copy ran out */
    KVQ_ERR_WORKSPACE = 6,       /* workspace missing, too small, or (device) not zero-filled */
    KVQ_ERR_BAD_LENGTH = 7       /* device: a length beyond the block table, or new tokens beyond max */
} kvq_status;

typedef enum kvq_format {
    KVQ_INT4_B64 = 0,   /* packed int4, scale = absmax / 7.5 per (block, head) */
    KVQ_INT8_PAGE = 1,  /* int8, scale = absmax / 127 per (page, head) */
    KVQ_FP8_E4M3 = 2    /* FP8 E4M3, scale = absmax / 448 per (page, head) */
} kvq_format;

/* bits of the device status word */
#define KVQ_FLAG_BAD_PAGE 0x1    /* a block-table entry was out of range (that page was not touched) */
#define KVQ_FLAG_BAD_LENGTH 0x2  /* a sequence length exceeded max_blocks_per_seq * 64 */
#define KVQ_FLAG_TIMEOUT 0x4     /* a bounded wait for a shared-memory copy ran out */
#define KVQ_FLAG_NO_TAIL 0x8     /* an append into a partial block found no fp16 tail buffer */
#define KVQ_FLAG_BAD_APPEND 0x10 /* cu_seqlens not increasing, or more new tokens than max_new_tokens */
#define KVQ_FLAG_BAD_WORKSPACE 0x20 /* a decode or prefill workspace was not zero-filled before its first use */

/*
 * The paged cache.  All pointers are caller-owned device memory.
 *   k_codes, v_codes   [num_pages][num_heads][64][head_dim/2 or head_dim]
 *   k_scales, v_scales [num_pages][num_heads] binary32
 *   k_tail, v_tail     fp16 [max_seqs][num_heads][64][head_dim]: the original
 *                      rows of each sequence's open (partial) block, so an
 *                      append can re-quantize that block from the originals.
 *                      Sequence b of an append call uses row b.  May be NULL
 *                      when every append ends on a 64-token boundary.
 *   status             one int32 the kernels OR KVQ_FLAG_* bits into; may be
 *                      NULL (then device-side problems go unreported).  Zero it
 *                      before first use.
 */
typedef struct kvq_cache {
    int32_t fmt;          /* kvq_format */
    int32_t num_heads;
    int32_t head_dim;     /* must be 128 */
    int32_t page_tokens;  /* must be 64 */
    int32_t num_pages;
    int32_t max_seqs;     /* rows of the tail buffers */
    uint8_t *k_codes;
    uint8_t *v_codes;
    float *k_scales;
    float *v_scales;
    uint16_t *k_tail;
    uint16_t *v_tail;
    int32_t *status;
} kvq_cache;

/*
 * kvq_quantize -- quantize_block of one contiguous tensor (jsqmd.com/news/887038
 * section 2.1; INT8: aicoding.csdn.net section 2.2).
 *   x       fp16 [num_tokens][num_heads][head_dim], 16-byte aligned
 *   codes   [ceil(num_tokens/64)][num_heads][64][head_dim/2 (int4) or head_dim (int8, FP8)],
 *           16-byte aligned; rows past num_tokens in the last block are written as 0
 *   scales  [ceil(num_tokens/64)][num_heads]
 * num_tokens == 0 is a no-op.  Errors: KVQ_ERR_INVALID_ARG, KVQ_ERR_UNSUPPORTED,
 * KVQ_ERR_CUDA.
 */
kvq_status kvq_quantize(kvq_format fmt, const uint16_t *x, int64_t num_tokens, int32_t num_heads,
                        int32_t head_dim, uint8_t *codes, float *scales, kvq_stream_t stream);

/*
 * kvq_append -- append new tokens to every sequence of a batch and keep the
 * cache equal to quantize_block of each sequence's whole history: full blocks
 * are quantized once; the open block is re-quantized from its fp16 originals
 * (tail buffer + new rows) and its tail rows are updated.
 *   k_new, v_new     fp16 [total_new][num_heads][head_dim], sequences back to
 *                    back, sequence b in rows [cu_seqlens[b], cu_seqlens[b+1])
 *   cu_seqlens       device int32 [num_seqs + 1], non-decreasing, cu_seqlens[0] = 0,
 *                    cu_seqlens[num_seqs] <= total_new_tokens
 *   block_table      device int32 [num_seqs][max_blocks_per_seq]: page of block j
 *   seq_lens_before  device int32 [num_seqs]: tokens already in each sequence
 *   total_new_tokens rows of k_new and v_new (a sequence whose rows would fall
 *                    beyond them is skipped and flagged)
 *   max_new_tokens   host bound on cu_seqlens[b+1] - cu_seqlens[b] (sizes the grid)
 * Device-detected problems set KVQ_FLAG_* bits in cache->status and skip the
 * affected blocks.
 * Launch: an append of at most 64 tokens per sequence uses programmatic
 * dependent launch and reads cu_seqlens, seq_lens_before and block_table
 * before waiting for the previous kernel of the stream (the scales, codes,
 * tail and new rows only after); the same condition as for
 * kvq_decode_attention's seq_lens and block_table holds for these three.
 * Errors: KVQ_ERR_INVALID_ARG, KVQ_ERR_UNSUPPORTED, KVQ_ERR_CUDA.
 */
kvq_status kvq_append(const kvq_cache *cache, const uint16_t *k_new, const uint16_t *v_new,
                      const int32_t *cu_seqlens, const int32_t *block_table, int32_t max_blocks_per_seq,
                      const int32_t *seq_lens_before, int32_t num_seqs, int64_t total_new_tokens,
                      int32_t max_new_tokens, kvq_stream_t stream);

/*
 * kvq_decode_workspace_bytes -- device scratch that kvq_decode_attention
 * needs on the current device (split partials and the per-sequence unit
 * prefix).  Depends on the format, the head dimension and the device's SM
 * count only.  Returns 0 for unsupported arguments.
 */
size_t kvq_decode_workspace_bytes(kvq_format fmt, int32_t num_heads, int32_t head_dim);

/*
 * kvq_decode_attention -- single-token decode attention over the quantized
 * paged cache (decode reading a quantized KV cache: aicoding.csdn.net
 * section 3.1; paging: ddd.cn section 4).  For every (b, h):
 *   s_t = softmax_scale * sum_d q[b][h][d] * k^_t[d],   t < seq_lens[b]
 *   out[b][h][:] = sum_t softmax(s)_t * v^_t[:]
 * computed in binary32 with an online softmax over splits of the sequence;
 * the warp that finishes the last split of a (b, h) merges the splits, all in
 * one kernel launch.
 *   q, out           fp16 [num_seqs][num_heads][head_dim], 16-byte aligned
 *   block_table      device int32 [num_seqs][max_blocks_per_seq]
 *   seq_lens         device int32 [num_seqs] (0 allowed: that output is 0)
 *   softmax_scale    normally 1/sqrt(head_dim)
 *   workspace        >= kvq_decode_workspace_bytes(...) bytes, 16-byte aligned,
 *                    zero-filled once before its first use (e.g. with
 *                    cudaMemsetAsync); every call that completes leaves it
 *                    ready for the next one.  After a call that set a
 *                    KVQ_FLAG_* bit, zero it again.  Do not share one
 *                    workspace between calls that may run concurrently.
 *                    The split counters in it carry a tag of the call, so a
 *                    workspace that was not zero-filled, or that a call cut
 *                    short left non-zero, is reported (KVQ_FLAG_BAD_WORKSPACE)
 *                    by the next call that uses it -- except a replay of the
 *                    same captured graph, which reuses its tag.  The outputs
 *                    of a call that set any KVQ_FLAG_* bit are undefined
 * Launch: with programmatic dependent launch, the kernel starts while the
 * previous kernel of the stream finishes and reads seq_lens and block_table
 * before waiting for it (the codes, scales, q and out only after).  No kvq_*
 * call writes those two arrays; a caller's own kernel that writes them right
 * before this call must not trigger its dependents early
 * (griddepcontrol.launch_dependents) -- ordinary launches never do.
 * Errors: KVQ_ERR_INVALID_ARG, KVQ_ERR_UNSUPPORTED, KVQ_ERR_WORKSPACE,
 * KVQ_ERR_CUDA; device-side problems set KVQ_FLAG_* bits in cache->status.
 */
kvq_status kvq_decode_attention(const kvq_cache *cache, const uint16_t *q, const int32_t *block_table,
                                int32_t max_blocks_per_seq, const int32_t *seq_lens, int32_t num_seqs,
                                float softmax_scale, uint16_t *out, void *workspace,
                                size_t workspace_bytes, kvq_stream_t stream);

/*
 * kvq_decode_attention_gqa -- kvq_decode_attention with grouped query heads
 * (grouped-query / multi-query attention; the pages' decode of MLA absorbed
 * into MQA, "DeepSeek R1 performance tips", ddd.cn section 2).  q and out hold
 * num_q_heads = g * cache->num_heads heads; query head i reads cache head
 * i / g, so one pass over each cache head's codes serves its g query heads:
 *   q, out           fp16 [num_seqs][num_q_heads][head_dim], 16-byte aligned
 *   workspace        >= kvq_decode_workspace_bytes_gqa(...) bytes, zero-filled
 *                    once before first use (as for kvq_decode_attention)
 * g = 1 is kvq_decode_attention.  Every format takes any g from 1 to 1024.
 * Two kernels serve it: for g <= 8 the multi-head kernel carries the group's
 * heads in the columns of its MMAs (one launch; int4: 4 columns for g = 2 .. 4,
 * 8 for g = 5 .. 8; int8 / FP8: 8 columns; columns past g carry zero queries;
 * except int4 g <= 4 the probabilities enter the PV product as fp16); every
 * g > 8 runs tiles of up to 16 query heads of one cache head as the rows of
 * the MMAs (a group of more than 16 heads is several tiles, which run side by
 * side so that the cache head's codes come from DRAM once), and a second,
 * small launch merges the split pieces.  In that path the probabilities enter
 * the PV product as fp16.
 * num_q_heads not a multiple of cache->num_heads returns KVQ_ERR_INVALID_ARG;
 * g > 1024, max_blocks_per_seq > 2^22 (the split counts the units of one
 * (sequence, head) in 24 bits; this bound holds for kvq_decode_attention too),
 * or a problem whose work units overflow 32 bits (at most 512 sequences x
 * unit heads x 4 units per page), KVQ_ERR_UNSUPPORTED.  Other errors as for
 * kvq_decode_attention.
 */
size_t kvq_decode_workspace_bytes_gqa(kvq_format fmt, int32_t num_kv_heads, int32_t num_q_heads,
                                      int32_t head_dim);
kvq_status kvq_decode_attention_gqa(const kvq_cache *cache, const uint16_t *q, int32_t num_q_heads,
                                    const int32_t *block_table, int32_t max_blocks_per_seq, const int32_t *seq_lens,
                                    int32_t num_seqs, float softmax_scale, uint16_t *out, void *workspace,
                                    size_t workspace_bytes, kvq_stream_t stream);

/*
 * kvq_decode_attention_noalloc -- kvq_decode_attention without a caller
 * workspace.  The pages have no counterpart to this entry point; it exists for
 * callers that cannot allocate device memory when they run decode attention:
 * an inference-engine plugin whose execute step must not allocate, a process
 * whose device memory is reserved up front by another allocator, or a loop
 * that cannot afford the device-wide synchronisation cudaMalloc / cudaFree
 * may cause.  It allocates nothing.
 *
 * The scratch is one fixed array of KVQ_NOALLOC_SCRATCH_BYTES (4 MiB) of
 * device memory inside the library; every GPU that loads the library holds it
 * until the process exits.  The first call on a device looks up the array's
 * device address (cudaGetSymbolAddress, with that device current) and keeps
 * it, so make that first call before any stream capture.  A device whose split
 * grid needs more scratch than the array (about 320 SMs' worth of split
 * partials; a 152-SM GB300 needs 1.95 MB) gets KVQ_ERR_WORKSPACE.  Every call
 * uses the same array and it keeps the last call's contents: calls that may
 * overlap on the GPU (other streams, other threads) race on it, so the caller
 * must serialise them.  The split's counters in the array must be zero when a
 * launch starts: each call clears them first on `stream` (a memset of about
 * 20 KB, no allocation), so a call that was cut short (a bounded wait that
 * ran out) does not spoil later ones.  Arguments, results and other errors
 * are those of kvq_decode_attention.
 */
#define KVQ_NOALLOC_SCRATCH_BYTES (4u << 20)
kvq_status kvq_decode_attention_noalloc(const kvq_cache *cache, const uint16_t *q, const int32_t *block_table,
                                        int32_t max_blocks_per_seq, const int32_t *seq_lens, int32_t num_seqs,
                                        float softmax_scale, uint16_t *out, kvq_stream_t stream);

/*
 * kvq_prefill_attention -- chunked-prefill attention over the quantized paged
 * cache (dynamic chunked attention of new tokens: "R1 performance overview",
 * aicoding.csdn.net; paging: ddd.cn section 4).  The chunk of sequence b is
 * its last n_b = cu_seqlens_q[b+1] - cu_seqlens_q[b] tokens, already in the
 * cache (kvq_append); query i of it (row cu_seqlens_q[b] + i of q) sits at
 * position p = seq_lens[b] - n_b + i and attends causally:
 *   out[row][hq][:] = sum_{t <= p} softmax_t(softmax_scale q . k^_t) v^_t
 * over cache head hq / g (g = num_q_heads / cache->num_heads, any g >= 1),
 * on the tensor cores (tcgen05): fp16 codes, fp16 q, probabilities rounded to
 * fp16 as the PV operand, binary32 accumulation.  Any finite softmax_scale.
 *   q, out           fp16 [total_q][num_q_heads][head_dim], 16-byte aligned
 *   cu_seqlens_q     device int32 [num_seqs + 1], non-decreasing, cu[0] >= 0
 *   max_q_per_seq    host bound on every n_b (sizes the grid); 0 is a no-op
 *   seq_lens         device int32 [num_seqs], n_b <= seq_lens[b] <= max_blocks_per_seq * 64
 *   workspace        NULL, or >= kvq_prefill_workspace_bytes(num_q_heads,
 *                    num_seqs, max_q_per_seq) bytes, 16-byte aligned,
 *                    zero-filled before its first use (the kernel puts its
 *                    counters back to zero): the work is cut into units of 256 query rows of
 *                    one (sequence, query head); with a workspace the units
 *                    of the grid's last wave (all units when there are fewer
 *                    than SMs) each run as two CTAs over the two halves of
 *                    their keys, merged there.  Same results up to rounding
 *                    order.  Do not share one workspace between calls that
 *                    may run concurrently.
 * A sequence that breaks a bound is skipped and KVQ_FLAG_BAD_LENGTH set; a
 * block-table entry out of range sets KVQ_FLAG_BAD_PAGE (page 0 is read
 * instead); a workspace that was not zero-filled sets KVQ_FLAG_BAD_WORKSPACE.
 * Errors: KVQ_ERR_INVALID_ARG, KVQ_ERR_UNSUPPORTED (also num_seqs or
 * num_q_heads above 65535, or 2^30 or more units), KVQ_ERR_WORKSPACE (too
 * small or misaligned), KVQ_ERR_CUDA.
 */
kvq_status kvq_prefill_attention(const kvq_cache *cache, const uint16_t *q, int32_t num_q_heads,
                                 const int32_t *cu_seqlens_q, int64_t total_q, int32_t max_q_per_seq,
                                 const int32_t *block_table, int32_t max_blocks_per_seq, const int32_t *seq_lens,
                                 int32_t num_seqs, float softmax_scale, uint16_t *out, void *workspace,
                                 size_t workspace_bytes, kvq_stream_t stream);

/*
 * kvq_prefill_workspace_bytes -- bytes of the optional kvq_prefill_attention
 * workspace for these sizes on the current device (0 when no unit is split
 * or an argument is not positive).  A workspace sized for the largest call
 * serves smaller ones only if their count is not larger: size it per call
 * shape.
 */
size_t kvq_prefill_workspace_bytes(int32_t num_q_heads, int32_t num_seqs, int32_t max_q_per_seq);

/*
 * Decode step as a CUDA graph (CUDA Graph instance reuse: "hardware-aware
 * scheduling" page, jsqmd.com/news/887038, section 4.1 -- capture once,
 * rebind tensor addresses with cudaGraphExecUpdate instead of rebuilding).
 *
 * One step = kvq_append of the new tokens, then kvq_decode_attention_gqa
 * over the grown sequences, with the arguments below (each field as in those
 * two calls; seq_lens = the lengths after the append).  A graph holds a
 * sequence of num_steps steps, step i on caches[i] with args[i] -- the layers
 * of one model's decode step, or successive steps of one layer -- in that
 * order, with the same programmatic-dependent-launch edges as eager calls
 * on one stream, so consecutive launches inside the graph overlap as they
 * would eagerly (between two graph launches they do not).  The graph records
 * the launches with these pointers and sizes; every kvq_step_graph_launch
 * replays them with whatever the buffers hold at that time, so per-step
 * inputs are written into the same buffers (sequence lengths and contents may
 * change freely between launches; the kernels read them from device memory).
 */
typedef struct kvq_step_args {
    const uint16_t *k_new;          /* append: fp16 [total_new_tokens][H][128] */
    const uint16_t *v_new;
    const int32_t *cu_seqlens;      /* [num_seqs + 1] */
    const int32_t *seq_lens_before; /* [num_seqs] */
    int64_t total_new_tokens;
    int32_t max_new_tokens;
    const int32_t *block_table;     /* [num_seqs][max_blocks_per_seq], both calls */
    int32_t max_blocks_per_seq;
    int32_t num_seqs;
    const uint16_t *q;              /* decode: fp16 [num_seqs][num_q_heads][128] */
    int32_t num_q_heads;
    const int32_t *seq_lens;        /* [num_seqs], lengths after the append */
    float softmax_scale;
    uint16_t *out;                  /* fp16 [num_seqs][num_q_heads][128] */
    void *workspace;
    size_t workspace_bytes;
} kvq_step_args;

typedef struct kvq_step_graph kvq_step_graph; /* opaque; host memory + one executable CUDA graph */

/*
 * kvq_step_graph_create -- check the arguments as the calls would, capture
 * the num_steps >= 1 steps (caches[i], args[i]) on a private stream of the
 * current device and instantiate them as one graph.
 * *graph_out receives a handle owned by the caller (kvq_step_graph_destroy).
 * Nothing is launched.  Errors: those of kvq_append and
 * kvq_decode_attention_gqa, KVQ_ERR_CUDA for a failed capture.
 */
kvq_status kvq_step_graph_create(const kvq_cache *caches, const kvq_step_args *args, int32_t num_steps,
                                 kvq_step_graph **graph_out);

/*
 * kvq_step_graph_update -- rebind the graph to new buffers / sizes: capture the
 * steps again and update the executable graph in place (cudaGraphExecUpdate);
 * when the launch structure changed (a different format, group size, number
 * of launches or of steps) it is instantiated anew.  On an error the graph keeps
 * its previous binding.
 */
kvq_status kvq_step_graph_update(kvq_step_graph *graph, const kvq_cache *caches, const kvq_step_args *args,
                                 int32_t num_steps);

/* kvq_step_graph_launch -- replay the steps on `stream` (asynchronous). */
kvq_status kvq_step_graph_launch(const kvq_step_graph *graph, kvq_stream_t stream);

/* kvq_step_graph_destroy -- release the graph (NULL is a no-op); no launch may be pending. */
kvq_status kvq_step_graph_destroy(kvq_step_graph *graph);

/*
 * kvq_get_device_status -- synchronise the stream, read and clear the cache's
 * device status word.  *flags_out (host, may be NULL) receives the KVQ_FLAG_*
 * bits.  Returns KVQ_OK when no bit was set, else the kvq_status of the most
 * serious bit (bad page, then bad length, then timeout, then append errors).
 */
kvq_status kvq_get_device_status(const kvq_cache *cache, kvq_stream_t stream, int32_t *flags_out);

/* a static, human-readable name of a status code */
const char *kvq_status_string(kvq_status status);

/* library version: major * 10000 + minor * 100 + patch */
int32_t kvq_version(void);

#ifdef __cplusplus
}
#endif

#endif /* KVQ_H */
