// tq_dequant.cu -- reconstruct bf16 K and V from the paged cache.
//
// turbo-attn, "Two independently-usable pieces": the codec decompresses to
// bf16 for any third-party attention.  Keys return to the original space:
//   K~ = n Pi^T ( c[code] / sqrt(d) + [QJL] sqrt(pi/2)/d * gamma * S^T (2 sigma - 1) )
// and values are code * scale + zero per group (0xsero/turboquant, "Value
// Compression"), or -- values coded by the rotation and their own Lloyd-Max
// codebook -- V~ = n Pi^T c[code] / sqrt(d).  One CTA per (slot, kv head), d
// threads, fp32 arithmetic.
#include <cuda_runtime.h>

#include "tq_device.cuh"
#include "tq_internal.h"

namespace tq {
namespace {

template <int D>
__global__ void __launch_bounds__(D)
dequant_kernel(const Codec C, const PageGeom G, const uint8_t *__restrict__ kc, const uint8_t *__restrict__ vc,
               int64_t num_blocks, int Hkv, const int64_t *__restrict__ slots, uint16_t *__restrict__ kout,
               uint16_t *__restrict__ vout)
{
    __shared__ float u[D];
    __shared__ float sg[D];
    const int64_t t = blockIdx.x;
    const int h = blockIdx.y;
    const int j = threadIdx.x;
    const int64_t slot = slots[t];
    if (slot < 0) return;
    const int64_t blk = slot / G.P;
    if (blk >= num_blocks) {
        if (j == 0) atomicOr(C.status, TQ_DEVERR_BLOCK_RANGE);
        return;
    }
    const int off = static_cast<int>(slot - blk * G.P);
    const uint8_t *kr = kc + (blk * Hkv + h) * G.k_page;
    const uint8_t *vr = vc + (blk * Hkv + h) * G.v_page;

    const uint8_t *cb = kr + static_cast<int64_t>(off) * C.k_code_bytes;
    const int kbit = j * C.k_bits;
    const uint32_t kw = cb[kbit >> 3] | (static_cast<uint32_t>(cb[min((kbit >> 3) + 1, C.k_code_bytes - 1)]) << 8);
    const uint32_t code = (kw >> (kbit & 7)) & ((1u << C.k_bits) - 1u);
    u[j] = C.centroids[code] * rsqrtf(static_cast<float>(D));
    const float n = bf16_to_float(*reinterpret_cast<const uint16_t *>(kr + G.k_norm_off + 2 * off));
    if (C.qjl) {
        const uint8_t *sb = kr + G.k_sign_off + static_cast<int64_t>(off) * C.k_sign_bytes;
        sg[j] = ((sb[j >> 3] >> (j & 7)) & 1u) ? 1.f : -1.f;
        __syncthreads();
        float a = 0.f;
        for (int i = 0; i < D; ++i) a = fmaf(__ldg(C.S + i * D + j), sg[i], a);  // (S^T (2 sigma - 1))_j
        const float gam = bf16_to_float(*reinterpret_cast<const uint16_t *>(kr + G.k_gamma_off + 2 * off));
        u[j] = fmaf(1.2533141373155003f / static_cast<float>(D) * gam, a, u[j]);
    }
    __syncthreads();
    float k = 0.f;
    for (int i = 0; i < D; ++i) k = fmaf(__ldg(C.Pi + i * D + j), u[i], k);  // (Pi^T u)_j
    const int64_t o = (t * Hkv + h) * D + j;
    kout[o] = float_to_bf16_bits(n * k);

    const uint8_t *vb = vr + static_cast<int64_t>(off) * C.v_code_bytes;
    const int vbit = j * C.v_bits;
    const uint32_t vw = vb[vbit >> 3] | (static_cast<uint32_t>(vb[min((vbit >> 3) + 1, C.v_code_bytes - 1)]) << 8);
    const uint32_t vcode = (vw >> (vbit & 7)) & ((1u << C.v_bits) - 1u);
    if (C.vmse) {  // V~ = n Pi^T c[code] / sqrt(d) (values coded like keys, no QJL)
        __syncthreads();  // every thread has read u
        u[j] = C.vcentroids[vcode] * rsqrtf(static_cast<float>(D));
        __syncthreads();
        float a = 0.f;
        for (int i = 0; i < D; ++i) a = fmaf(__ldg(C.Pi + i * D + j), u[i], a);
        const float vn = bf16_to_float(*reinterpret_cast<const uint16_t *>(vr + G.v_meta_off + 2 * off));
        vout[o] = float_to_bf16_bits(vn * a);
        return;
    }
    const __half2 sz = *reinterpret_cast<const __half2 *>(vr + G.v_meta_off + static_cast<int64_t>(off) * C.v_meta_bytes +
                                                         4 * (j / C.group));
    const float2 f = __half22float2(sz);
    vout[o] = float_to_bf16_bits(fmaf(static_cast<float>(vcode), f.x, f.y));
}

}  // namespace

cudaError_t launch_dequant(const Codec &c, const PageGeom &pg, const uint8_t *kc, const uint8_t *vc,
                           int64_t num_blocks, int Hkv, const int64_t *slots, int64_t T, uint16_t *k_out,
                           uint16_t *v_out, cudaStream_t st)
{
    dim3 grid(static_cast<unsigned>(T), Hkv);
    if (c.d == 128)
        dequant_kernel<128><<<grid, 128, 0, st>>>(c, pg, kc, vc, num_blocks, Hkv, slots, k_out, v_out);
    else
        dequant_kernel<256><<<grid, 256, 0, st>>>(c, pg, kc, vc, num_blocks, Hkv, slots, k_out, v_out);
    return cudaGetLastError();
}

}  // namespace tq
