// tq_decode.cu -- split-K paged decode attention over the compressed cache.
//
// turbo-attn, "How it works": attention scores on rotated keys equal scores on
// the original keys when the query is rotated by the same matrix, so the query
// is pre-rotated once and everything runs in the rotated space; the decode is
// one fused pass (unpack, dequantise, Q.K, online softmax, P.V) with no
// decompress buffer.  turbo-attn, "Configuration" (TKV_DECODE_SPLITS): the
// decode kernel splits the context (split-K) and the splits are merged.
//
// Per query head h of kv head kvh = h / G and context token t:
//   s_t = sm_scale * n_t * ( <q_rot, c[code_t]> / sqrt(d)
//                            + [QJL] sqrt(pi/2) / d * gamma_t * <S q_rot, 2 sigma_t - 1> )
//   o   = sum_t softmax(s)_t * (code_t * scale + zero)      (values per group)
// which is <q, K~_t> with K~ = n Pi^T (c/sqrt(d) + sqrt(pi/2)/d gamma S^T(2 sigma - 1)).
//
// Launches: (1) qrot: q_rot = Pi q and q_s = S q_rot in fp32 per (b, h);
// (2) decode: grid (splits, Hkv, B), each CTA walks its pages of one sequence
// for the G query heads that share the kv head, keeping an online softmax;
// (3) combine: log-sum-exp merge of the split partials into bf16.
#include <cuda_runtime.h>

#include "tq_decode_mma.cuh"
#include "tq_device.cuh"
#include "tq_internal.h"

namespace tq {

size_t decode_workspace_bytes(int d, int B, int Hq, int splits)
{
    auto al = [](size_t x) { return (x + 255) / 256 * 256; };
    const size_t rows = static_cast<size_t>(B) * Hq;
    return al(rows * d * 4) * 2 + al(static_cast<size_t>(splits) * rows * d * 4) +
           al(static_cast<size_t>(splits) * rows * 2 * 4);
}

DecodeWorkspace carve_decode_workspace(void *base, int d, int B, int Hq, int splits)
{
    auto al = [](size_t x) { return (x + 255) / 256 * 256; };
    const size_t rows = static_cast<size_t>(B) * Hq;
    char *p = static_cast<char *>(base);
    DecodeWorkspace w;
    w.qrot = reinterpret_cast<float *>(p);
    p += al(rows * d * 4);
    w.qs = reinterpret_cast<float *>(p);
    p += al(rows * d * 4);
    w.acc = reinterpret_cast<float *>(p);
    p += al(static_cast<size_t>(splits) * rows * d * 4);
    w.ml = reinterpret_cast<float *>(p);
    return w;
}

namespace {


// ---- (1) query pre-rotation ------------------------------------------------
template <int D>
__global__ void __launch_bounds__(D) qrot_kernel(const Codec C, const uint16_t *__restrict__ q, float *qrot, float *qs)
{
    __shared__ float sq[D];
    __shared__ float sr[D];
    const int row = blockIdx.x, i = threadIdx.x;
    sq[i] = bf16_to_float(q[static_cast<int64_t>(row) * D + i]);
    __syncthreads();
    float a = 0.f;
    for (int j = 0; j < D; ++j) a = fmaf(__ldg(C.PiT + j * D + i), sq[j], a);
    sr[i] = a;
    qrot[static_cast<int64_t>(row) * D + i] = a;
    if (!C.qjl) return;
    __syncthreads();
    float b = 0.f;
    for (int j = 0; j < D; ++j) b = fmaf(__ldg(C.ST + j * D + i), sr[j], b);
    qs[static_cast<int64_t>(row) * D + i] = b;
}

// ---- (2) split-K decode: see tq_decode_mma.cuh ---------------------------------

// ---- (3) log-sum-exp combine -------------------------------------------------
template <int D>
__global__ void __launch_bounds__(D) combine_kernel(const DecodeArgs A)
{
    const int row = blockIdx.x;  // b * Hq + h
    const int j = threadIdx.x;
    const size_t rows = static_cast<size_t>(A.B) * A.Hq;
    float M = -INFINITY;
    for (int s = 0; s < A.splits; ++s) {
        const float l = A.ws.ml[(s * rows + row) * 2 + 1];
        if (l > 0.f) M = fmaxf(M, A.ws.ml[(s * rows + row) * 2]);
    }
    float num = 0.f, den = 0.f;
    if (M != -INFINITY) {
        for (int s = 0; s < A.splits; ++s) {
            const float m = A.ws.ml[(s * rows + row) * 2];
            const float l = A.ws.ml[(s * rows + row) * 2 + 1];
            if (!(l > 0.f)) continue;
            const float w = exp2f(m - M);
            den = fmaf(w, l, den);
            num = fmaf(w, A.ws.acc[(s * rows + row) * D + j], num);
        }
    }
    const float o = (den > 0.f) ? num / den : 0.f;
    A.out[static_cast<size_t>(row) * D + j] = float_to_bf16_bits(o);
}

template <int D, int KB, int VB>
cudaError_t launch_dmma(const Codec &c, const PageGeom &pg, const DecodeArgs &a, cudaStream_t st)
{
    const size_t smem = dmma::DecSmem<D, KB>::bytes(pg);
    static size_t attr_bytes[64] = {};  // per device: the largest size granted so far
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if (dev < 0 || dev >= 64 || attr_bytes[dev] < smem) {
        e = cudaFuncSetAttribute(dmma::decode_mma_kernel<D, KB, VB>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 static_cast<int>(smem));
        if (e != cudaSuccess) return e;
        if (dev >= 0 && dev < 64) attr_bytes[dev] = smem;
    }
    dim3 grid(a.splits, a.Hkv, a.B);
    dmma::decode_mma_kernel<D, KB, VB><<<grid, dmma::kThreads, smem, st>>>(c, pg, a);
    return cudaGetLastError();
}

template <int D, int KB>
cudaError_t launch_dmma_kb(const Codec &c, const PageGeom &pg, const DecodeArgs &a, cudaStream_t st)
{
    switch (c.v_bits) {
    case 2: return launch_dmma<D, KB, 2>(c, pg, a, st);
    case 3: return launch_dmma<D, KB, 3>(c, pg, a, st);
    default: return launch_dmma<D, KB, 4>(c, pg, a, st);
    }
}

template <int D>
cudaError_t launch_decode_d(const Codec &c, const PageGeom &pg, const DecodeArgs &a, cudaStream_t st)
{
    qrot_kernel<D><<<a.B * a.Hq, D, 0, st>>>(c, a.q, a.ws.qrot, a.ws.qs);
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return e;
    switch (c.k_bits) {
    case 2: e = launch_dmma_kb<D, 2>(c, pg, a, st); break;
    case 3: e = launch_dmma_kb<D, 3>(c, pg, a, st); break;
    default: e = launch_dmma_kb<D, 4>(c, pg, a, st); break;
    }
    if (e != cudaSuccess) return e;
    combine_kernel<D><<<a.B * a.Hq, D, 0, st>>>(a);
    return cudaGetLastError();
}

}  // namespace

cudaError_t launch_decode(const Codec &c, const PageGeom &pg, const DecodeArgs &a, cudaStream_t st)
{
    if (c.d == 128) return launch_decode_d<128>(c, pg, a, st);
    return launch_decode_d<256>(c, pg, a, st);
}

}  // namespace tq
