// tq_prefill.cu -- the split-K kernel instantiated for chunked prefill over the
// compressed cache at head_dim 256 (turbo-attn, "How it works": the prefill path dequantises the
// codec inline, with no decompress buffer).  Each CTA takes qpc consecutive
// query tokens of one sequence; their (token, head) pairs are the N columns of
// the score and value products, each with its own causal limit and online
// softmax, so every operand built from the codes serves all of them.  Kept apart
// from tq_decode.cu so the two sets of instantiations compile in parallel.
#include <cuda_runtime.h>

#include "tq_decode_mma.cuh"
#include "tq_internal.h"

namespace tq {
namespace {

template <int D, int KB, int VB>
cudaError_t launch_pf(const Codec &c, const PageGeom &pg, const DecodeArgs &a, cudaStream_t st)
{
    const size_t smem = dmma::DecSmem<D, KB>::bytes(pg);
    cudaError_t e =
        ensure_smem_attr(reinterpret_cast<const void *>(dmma::decode_mma_kernel<D, KB, VB, false, true>), smem);
    if (e != cudaSuccess) return e;
    dim3 grid(a.splits, a.Hkv, a.B * ((a.Tq + a.qpc - 1) / a.qpc));
    dmma::decode_mma_kernel<D, KB, VB, false, true><<<grid, dmma::kThreads, smem, st>>>(c, pg, a);
    return cudaGetLastError();
}

template <int D, int KB>
cudaError_t launch_pf_kb(const Codec &c, const PageGeom &pg, const DecodeArgs &a, cudaStream_t st)
{
    switch (c.v_bits) {
    case 2: return launch_pf<D, KB, 2>(c, pg, a, st);
    case 3: return launch_pf<D, KB, 3>(c, pg, a, st);
    default: return launch_pf<D, KB, 4>(c, pg, a, st);
    }
}

template <int D>
cudaError_t launch_pf_d(const Codec &c, const PageGeom &pg, const DecodeArgs &a, cudaStream_t st)
{
    switch (c.k_bits) {
    case 2: return launch_pf_kb<D, 2>(c, pg, a, st);
    case 3: return launch_pf_kb<D, 3>(c, pg, a, st);
    default: return launch_pf_kb<D, 4>(c, pg, a, st);
    }
}

}  // namespace

cudaError_t launch_dmma_prefill(const Codec &c, const PageGeom &pg, const DecodeArgs &a, cudaStream_t st)
{
    // head_dim 256 only: 128 runs the tensor-memory kernel (tq_prefill_tc.cu), whose
    // query operands and output would not fit tensor memory next to the scores at 256
    return launch_pf_d<256>(c, pg, a, st);
}

}  // namespace tq
