// tq_decode_vmse.cu -- the split-K decode kernel instantiated for values coded
// by the rotation and a Lloyd-Max codebook (brightcoding blog, "What is
// TurboQuant-GPU?": MSE-quantised values).  The value term of every token is
// n_t c[code_t] / sqrt(d) in the rotated space: the kernel multiplies fp16
// centroid pairs (the A operand) by p_t n_t (the B operand) and the combine
// rotates the merged output back with Pi^T.  Kept apart from tq_decode.cu so
// the two sets of instantiations compile in parallel.
#include <cuda_runtime.h>

#include "tq_decode_mma.cuh"
#include "tq_internal.h"

namespace tq {
namespace {

template <int D, int KB, int VB>
cudaError_t launch_vm(const Codec &c, const PageGeom &pg, const DecodeArgs &a, cudaStream_t st)
{
    const size_t smem = dmma::DecSmem<D, KB, VB, true>::bytes(pg);
    dim3 grid(a.splits, a.Hkv, a.B * ((a.Tq + a.qpc - 1) / a.qpc));
    if constexpr (D == 256) {
        if (a.Tq > 1) {  // prefill with values coded by the rotation (head_dim 128 runs the tensor-memory kernel)
            cudaError_t e = ensure_smem_attr(
                reinterpret_cast<const void *>(dmma::decode_mma_kernel<D, KB, VB, true, true>), smem);
            if (e != cudaSuccess) return e;
            dmma::decode_mma_kernel<D, KB, VB, true, true><<<grid, dmma::kThreads, smem, st>>>(c, pg, a);
            return cudaGetLastError();
        }
    }
    cudaError_t e = ensure_smem_attr(reinterpret_cast<const void *>(dmma::decode_mma_kernel<D, KB, VB, true>), smem);
    if (e != cudaSuccess) return e;
    dmma::decode_mma_kernel<D, KB, VB, true><<<grid, dmma::kThreads, smem, st>>>(c, pg, a);
    return cudaGetLastError();
}

template <int D, int KB>
cudaError_t launch_vm_kb(const Codec &c, const PageGeom &pg, const DecodeArgs &a, cudaStream_t st)
{
    switch (c.v_bits) {
    case 2: return launch_vm<D, KB, 2>(c, pg, a, st);
    case 3: return launch_vm<D, KB, 3>(c, pg, a, st);
    default: return launch_vm<D, KB, 4>(c, pg, a, st);
    }
}

template <int D>
cudaError_t launch_vm_d(const Codec &c, const PageGeom &pg, const DecodeArgs &a, cudaStream_t st)
{
    switch (c.k_bits) {
    case 2: return launch_vm_kb<D, 2>(c, pg, a, st);
    case 3: return launch_vm_kb<D, 3>(c, pg, a, st);
    default: return launch_vm_kb<D, 4>(c, pg, a, st);
    }
}

}  // namespace

cudaError_t launch_dmma_vmse(const Codec &c, const PageGeom &pg, const DecodeArgs &a, cudaStream_t st)
{
    return c.d == 128 ? launch_vm_d<128>(c, pg, a, st) : launch_vm_d<256>(c, pg, a, st);
}

}  // namespace tq
