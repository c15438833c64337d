// kvq_internal.h -- launch parameters and launchers shared between the C ABI
// (kvq_api.cu) and the kernel translation units.
#pragma once

#include <cuda_runtime.h>
#include <stddef.h>
#include <stdint.h>

#include "kvq.h"

namespace kvq {

constexpr int kHeadDim = 128;
constexpr int kPage = 64;

struct AppendParams {
    const uint16_t *k_new;
    const uint16_t *v_new;
    const int32_t *cu_seqlens;
    const int32_t *block_table;
    const int32_t *seq_lens_before;
    uint8_t *k_codes;
    uint8_t *v_codes;
    float *k_scales;
    float *v_scales;
    uint16_t *k_tail;
    uint16_t *v_tail;
    int32_t *status;
    int32_t num_seqs;
    int32_t num_heads;
    int32_t num_pages;
    int32_t max_blocks;
    int32_t max_new_tokens;
    int64_t total_new;
};

struct DecodeParams {
    const uint8_t *k_codes;
    const uint8_t *v_codes;
    const float *k_scales;
    const float *v_scales;
    const uint16_t *q;
    const int32_t *block_table;
    const int32_t *seq_lens;
    uint16_t *out;
    float *partials;               // [grid warps][2][rows * kPartialStride]: split partials, two slots per warp
    unsigned long long *counters;  // [grid warps] unit counts of split (sequence, head)s
    int32_t *status;
    int32_t num_seqs;
    int32_t num_heads;
    int32_t num_pages;
    int32_t max_blocks;
    float score_scale;  // softmax_scale * log2(e): scores are kept in the base-2 domain
    int32_t group;      // query heads per cache head: q and out hold num_heads * group heads
    // Tag of this call in the counters (odd, < 2^40).  A counter holds
    // count + 2^24 * (count * epoch mod 2^40), so a count left over by another
    // call (or memory that was never zero-filled) shows up as an inconsistent word.
    unsigned long long epoch;
    unsigned long long wait_limit_ns;  // bounded waits give up after this long
    int32_t test_skip_chunk;           // >= 0: warp 0 leaves the copies of this chunk unissued (timeout test)
    int32_t tiles;                     // tiles of 16 query heads per cache head (set by the launcher)
};

// the largest group (query heads per cache head) the decode kernels take
constexpr int kMaxDecodeGroup = 1024;

// default limit of a decode kernel's bounded waits (kernels finish in milliseconds)
constexpr unsigned long long kDecodeWaitLimitNs = 500ull * 1000ull * 1000ull;

// counter words: the low kCountBits bits count, the rest carry count * epoch
constexpr int kCountBits = 24;
// warps per SM the decode workspace's counter region is sized for (every decode kernel uses at most this many)
constexpr int kMaxDecodeWarpsPerSm = 16;

// floats per split partial: m, l, 2 pad, acc[128]
constexpr int kPartialStride = 132;
// sequences per split-kernel launch (the per-CTA prefix lives in shared memory)
constexpr int kMaxSeqsPerLaunch = 512;

struct PrefillParams {
    const uint8_t *k_codes;
    const uint8_t *v_codes;
    const float *k_scales;
    const float *v_scales;
    const uint16_t *q;            // [total_q][num_q_heads][128]
    uint16_t *out;                // [total_q][num_q_heads][128]
    const int32_t *cu_q;          // [num_seqs + 1]: sequence b's queries are rows cu_q[b] .. cu_q[b+1]-1
    const int32_t *seq_lens;      // [num_seqs]: lengths including the chunk
    const int32_t *block_table;   // [num_seqs][max_blocks]
    int32_t *status;
    int num_seqs, num_heads, num_q_heads, group, num_pages, max_blocks, max_q;
    int64_t total_q;
    float score_scale;            // softmax_scale * log2(e)
    // work units: 256 query rows of one (sequence, query head), units_x of them per pair,
    // ordered (sequence, query head, x); units from num_full on run as two CTAs over the two
    // halves of their keys, merged through partials [unit - num_full][half][256][132] floats
    // and counters [unit - num_full] (zero-filled before the first launch)
    int units_x, num_full;
    float *partials;
    uint32_t *counters;
};

// prefill work units of a call and the units run as split halves (the grid's last
// wave, or every unit of a grid smaller than one wave); workspace bytes for them
int64_t prefill_units(int num_q_heads, int num_seqs, int max_q);
int64_t prefill_split_units(int64_t units, int num_sms);
size_t prefill_workspace_bytes(int64_t split_units);

// launch `kernel` with programmatic stream serialization (see pdl_wait)
template <typename... KArgs, typename... Args>
cudaError_t launch_pdl(void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem, cudaStream_t s,
                       Args &&...args)
{
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = grid;
    cfg.blockDim = block;
    cfg.dynamicSmemBytes = smem;
    cfg.stream = s;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, kernel, static_cast<KArgs>(args)...);
}

// the same launch without the attribute: the kernel starts only after the
// previous work on the stream has completed
template <typename... KArgs, typename... Args>
cudaError_t launch_plain(void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem, cudaStream_t s,
                         Args &&...args)
{
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = grid;
    cfg.blockDim = block;
    cfg.dynamicSmemBytes = smem;
    cfg.stream = s;
    cfg.attrs = nullptr;
    cfg.numAttrs = 0;
    return cudaLaunchKernelEx(&cfg, kernel, static_cast<KArgs>(args)...);
}

cudaError_t launch_quantize(int fmt, const uint16_t *x, int64_t T, int H, uint8_t *codes, float *scales,
                            cudaStream_t s);
cudaError_t launch_append(int fmt, const AppendParams &p, cudaStream_t s);

// number of warps of the persistent split grid of (format, group) on the current device (0 on error)
int decode_grid_warps(int fmt, int group);
bool decode_group_supported(int fmt, int group);
// the decode workspace: a counter region first (its size depends on the
// device's SM count only), then the split partials
size_t decode_counter_bytes();
size_t decode_workspace_bytes(int fmt, int group);
// a fresh odd 40-bit tag for one decode launch
unsigned long long decode_next_epoch();
// test hook of kvq_testing.h: wait limit (0: default) and chunk to leave unissued (-1: none)
void decode_test_settings(unsigned long long *wait_limit_ns, int32_t *skip_chunk);
// resolves (and caches) the occupancy query and shared-memory attribute of the
// decode kernel for (fmt, group); returns CTAs per SM, 0 when unsupported
int decode_prepare(int fmt, int group);
cudaError_t launch_decode(int fmt, const DecodeParams &p, cudaStream_t s);
cudaError_t launch_prefill(int fmt, const PrefillParams &p, cudaStream_t s);

}  // namespace kvq
