// kvq_noalloc.cu -- decode attention for callers that cannot allocate device
// memory at the moment they call it.
//
// kvq_decode_attention needs a caller workspace (split partials and a unit
// prefix).  Some callers cannot produce one when they run decode attention: an
// inference-engine plugin whose execute step is not allowed to allocate, a
// process whose device memory is reserved up front by another allocator, or a
// serving loop that cannot afford the device-wide synchronisation cudaMalloc /
// cudaFree may cause.  For them the workspace comes from the fixed array
// below, which belongs to the library: every GPU that loads the library holds
// KVQ_NOALLOC_SCRATCH_BYTES of device memory for it until the process exits.
//
// Host code cannot use g_decode_scratch's name as a device address (on the
// host it names a host-side stand-in), so the first call on each device looks
// the address up with cudaGetSymbolAddress while that device is current and
// keeps it.  All calls share the one array: calls that may overlap on the GPU
// race on it.  The split's counters at the front of the array must be zero
// when a launch starts; a launch that completes leaves them zero, but one that
// was cut short (a bounded wait that ran out) may not, and the caller of this
// entry point has no way to clear library memory.  So every call first clears
// the counter region on the caller's stream (cudaMemsetAsync, which allocates
// nothing); the partials behind it need no clearing.
#include <cuda_runtime.h>

#include <mutex>

#include "kvq.h"
#include "kvq_internal.h"

namespace {

constexpr int kMaxDevices = 64;

static __device__ __align__(256) unsigned char g_decode_scratch[KVQ_NOALLOC_SCRATCH_BYTES];

std::mutex g_scratch_mu;
void *g_scratch_addr[kMaxDevices] = {};

// device address of g_decode_scratch on the current device (looked up once per device)
kvq_status scratch_address(void **out)
{
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return KVQ_ERR_CUDA;
    if (dev < 0 || dev >= kMaxDevices) return KVQ_ERR_UNSUPPORTED;
    std::lock_guard<std::mutex> lock(g_scratch_mu);
    if (g_scratch_addr[dev] == nullptr) {
        void *p = nullptr;
        if (cudaGetSymbolAddress(&p, g_decode_scratch) != cudaSuccess || p == nullptr) return KVQ_ERR_CUDA;
        g_scratch_addr[dev] = p;
    }
    *out = g_scratch_addr[dev];
    return KVQ_OK;
}

}  // namespace

extern "C" kvq_status kvq_decode_attention_noalloc(const kvq_cache *cache, const uint16_t *q,
                                                   const int32_t *block_table, int32_t max_blocks_per_seq,
                                                   const int32_t *seq_lens, int32_t num_seqs, float softmax_scale,
                                                   uint16_t *out, kvq_stream_t stream)
{
    if (!cache) return KVQ_ERR_INVALID_ARG;
    void *scratch = nullptr;
    kvq_status st = scratch_address(&scratch);
    if (st != KVQ_OK) return st;
    const size_t need = kvq_decode_workspace_bytes(static_cast<kvq_format>(cache->fmt), cache->num_heads,
                                                   cache->head_dim);
    if (need == 0) return KVQ_ERR_UNSUPPORTED;
    if (need > KVQ_NOALLOC_SCRATCH_BYTES) return KVQ_ERR_WORKSPACE;  // this device needs more than the fixed array
    const size_t counters = kvq::decode_counter_bytes();
    if (counters == 0 || counters > need) return KVQ_ERR_CUDA;
    if (num_seqs > 0 &&
        cudaMemsetAsync(scratch, 0, counters, reinterpret_cast<cudaStream_t>(stream)) != cudaSuccess)
        return KVQ_ERR_CUDA;
    return kvq_decode_attention(cache, q, block_table, max_blocks_per_seq, seq_lens, num_seqs, softmax_scale, out,
                                scratch, KVQ_NOALLOC_SCRATCH_BYTES, stream);
}
