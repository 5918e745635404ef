// tq_static_scratch.cu -- decode attention for callers that cannot allocate.
//
// Some callers cannot call cudaMalloc, or hand the library a workspace of their
// own: code that runs inside another runtime's fixed memory budget, plug-ins
// loaded into a host process that owns every device allocation, and schedulers
// that must not touch an allocator on their launch path.  This entry point runs
// the same three kernels as tq_decode_attention, but its scratch (rotated
// queries and per-split partial outputs) lives in a file-scope device array
// instead of a caller-provided workspace.
//
// The array holds TQ_STATIC_SCRATCH_BYTES (16 MiB), 256-byte aligned, and every
// GPU that loads the library keeps it until the process exits.  All calls share
// it and it keeps the last call's contents; nothing in it needs to start at zero,
// because each call writes every byte it later reads.  Calls that overlap on the
// GPU -- on two streams, or through two handles -- race on the array.
#include <cuda_runtime.h>

#include "tq.h"
#include "tq_internal.h"

namespace {

static __device__ __align__(256) unsigned char g_decode_scratch[TQ_STATIC_SCRATCH_BYTES];

}  // namespace

// In host code the array's name is only a stand-in, not a device address: the
// address belongs to the CUDA context and is looked up with cudaGetSymbolAddress.
// tq_init calls this while its device (and context) is current and keeps the
// result in the handle, so the entry point below never looks it up again.
cudaError_t tq::static_scratch_lookup(void **out)
{
    void *p = nullptr;
    const cudaError_t e = cudaGetSymbolAddress(&p, g_decode_scratch);
    if (e == cudaSuccess) *out = p;
    return e;
}

extern "C" tq_status tq_decode_attention_static(tq_handle h, const uint16_t *q, const uint8_t *k_cache,
                                                const uint8_t *v_cache, const int32_t *block_table,
                                                const int32_t *seq_lens, int batch, int num_q_heads,
                                                int num_kv_heads, int page_size, int max_blocks_per_seq,
                                                int64_t num_blocks, float sm_scale, int splits, uint16_t *out,
                                                void *stream)
{
    if (!h) return tq::api_error(TQ_ERR_INVALID_ARG, "tq_decode_attention_static: NULL handle");
    if (splits < 0) return tq::api_error(TQ_ERR_INVALID_ARG, "tq_decode_attention_static: negative splits");
    if (splits == 0 && batch > 0 && num_kv_heads > 0 && max_blocks_per_seq > 0)
        splits = tq_decode_splits(h, batch, num_kv_heads, max_blocks_per_seq, page_size);
    if (batch > 0 && splits > 0) {
        const size_t need = tq_decode_workspace_bytes(h, batch, num_q_heads, splits);
        if (need > TQ_STATIC_SCRATCH_BYTES)
            return tq::api_error(TQ_ERR_UNSUPPORTED,
                                 "tq_decode_attention_static: this call needs %zu bytes of scratch, more than the "
                                 "%zu-byte static array; use fewer sequences, heads or splits, or tq_decode_attention "
                                 "with a workspace",
                                 need, static_cast<size_t>(TQ_STATIC_SCRATCH_BYTES));
    }
    void *ws = tq::handle_static_scratch(h);
    if (!ws) return tq::api_error(TQ_ERR_CUDA, "tq_decode_attention_static: the handle has no scratch address");
    return tq_decode_attention(h, q, k_cache, v_cache, block_table, seq_lens, batch, num_q_heads, num_kv_heads,
                               page_size, max_blocks_per_seq, num_blocks, sm_scale, splits, ws, TQ_STATIC_SCRATCH_BYTES,
                               out, stream);
}
