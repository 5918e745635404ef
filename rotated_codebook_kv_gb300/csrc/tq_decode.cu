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

constexpr float kQjlCoef = 1.2533141373155003f;  // sqrt(pi / 2)
constexpr int kChunk = 64;                        // tokens per decode iteration

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

// ---- (2) split-K decode ------------------------------------------------------
template <int D, int G>
struct DecodeSmem {
    static constexpr int SL = D / kChunk;  // coordinate slices per token in the scoring step
    float qrot[G][D];
    float qs[G][D];
    float part[SL][G][kChunk];
    float prob[G][kChunk];
    float alpha[G];
    float m_run[G];
    float l_run[G];
    float cent[16];
    int page_ok[4];
};

template <int D, int G>
__global__ void __launch_bounds__(D) decode_kernel(const Codec C, const PageGeom PG, const DecodeArgs A)
{
    using SM = DecodeSmem<D, G>;
    constexpr int SL = SM::SL;
    constexpr int CW = D / SL;  // coordinates per scoring thread
    __shared__ SM sm;
    extern __shared__ __align__(16) unsigned char pages[];  // [ppc][k_page] then [ppc][v_page]

    const int split = blockIdx.x, kvh = blockIdx.y, b = blockIdx.z;
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int P = PG.P;
    const int ppc = kChunk / P;  // pages per chunk
    uint8_t *kpg = pages;
    uint8_t *vpg = pages + static_cast<size_t>(ppc) * PG.k_page;

    int L = A.seq_lens[b];
    if (L < 0) L = 0;
    if (L > A.max_blocks * P) {
        if (split == 0 && kvh == 0 && tid == 0) atomicOr(C.status, TQ_DEVERR_SEQ_RANGE);
        L = A.max_blocks * P;
    }
    const int npages = (L + P - 1) / P;
    const int pg0 = split * A.pages_per_split;
    const int pg1 = min(npages, pg0 + A.pages_per_split);
    const size_t head0 = static_cast<size_t>(b) * A.Hq + static_cast<size_t>(kvh) * G;
    float *ml_out = A.ws.ml + (static_cast<size_t>(split) * A.B * A.Hq + head0) * 2;
    float *acc_out = A.ws.acc + (static_cast<size_t>(split) * A.B * A.Hq + head0) * D;
    if (pg0 >= pg1) {  // empty split
        if (tid < G) {
            ml_out[2 * tid] = -INFINITY;
            ml_out[2 * tid + 1] = 0.f;
        }
        return;
    }

    for (int e = tid; e < G * D; e += D) {
        const int h = e / D, j = e - h * D;
        sm.qrot[h][j] = A.ws.qrot[(head0 + h) * D + j];
        sm.qs[h][j] = C.qjl ? A.ws.qs[(head0 + h) * D + j] : 0.f;
    }
    if (tid < 16) sm.cent[tid] = C.centroids[tid];
    if (tid < G) {
        sm.m_run[tid] = -INFINITY;
        sm.l_run[tid] = 0.f;
    }
    float acc[G];
#pragma unroll
    for (int h = 0; h < G; ++h) acc[h] = 0.f;

    const float inv_sqrtd = rsqrtf(static_cast<float>(D));
    const float qcoef = kQjlCoef / static_cast<float>(D);
    const int kb = C.k_bits, vb = C.v_bits;

    for (int cp = pg0; cp < pg1; cp += ppc) {
        const int npc = min(ppc, pg1 - cp);
        __syncthreads();  // previous chunk fully consumed
        // ---- stage K and V page records of this chunk ----
        for (int q = 0; q < npc; ++q) {
            const int blk = A.block_table[static_cast<int64_t>(b) * A.max_blocks + cp + q];
            const bool ok = (blk >= 0 && blk < A.num_blocks);
            if (tid == 0) {
                sm.page_ok[q] = ok;
                if (!ok) atomicOr(C.status, TQ_DEVERR_BLOCK_RANGE);
            }
            if (!ok) continue;
            const size_t rec = static_cast<size_t>(blk) * A.Hkv + kvh;
            const uint4 *ks = reinterpret_cast<const uint4 *>(A.k_cache + rec * PG.k_page);
            const uint4 *vs = reinterpret_cast<const uint4 *>(A.v_cache + rec * PG.v_page);
            uint4 *kd = reinterpret_cast<uint4 *>(kpg + q * PG.k_page);
            uint4 *vd = reinterpret_cast<uint4 *>(vpg + q * PG.v_page);
            for (int e = tid; e < PG.k_page / 16; e += D) kd[e] = __ldg(ks + e);
            for (int e = tid; e < PG.v_page / 16; e += D) vd[e] = __ldg(vs + e);
        }
        __syncthreads();
        // ---- scores: thread (token tt, slice sl) -> partial dot products ----
        {
            const int tt = tid % kChunk, sl = tid / kChunk;
            const int q = tt / P, off = tt - q * P;
            const int pos = cp * P + tt;
            if (q < npc && pos < L && sm.page_ok[q]) {
                const uint8_t *kr = kpg + q * PG.k_page;
                const uint32_t *cw = reinterpret_cast<const uint32_t *>(kr + off * C.k_code_bytes + sl * (CW * kb / 8));
                uint32_t words[CW * 4 / 32 + 1];
#pragma unroll
                for (int w = 0; w < CW * 4 / 32; ++w)
                    if (w < CW * kb / 32) words[w] = cw[w];
                words[CW * 4 / 32] = 0u;
                float dc[G], ds[G];
#pragma unroll
                for (int h = 0; h < G; ++h) dc[h] = ds[h] = 0.f;
                const int j0 = sl * CW;
#pragma unroll 8
                for (int j = 0; j < CW; ++j) {
                    const float cv = sm.cent[code_from_words(words, j, kb)];
#pragma unroll
                    for (int h = 0; h < G; ++h) dc[h] = fmaf(sm.qrot[h][j0 + j], cv, dc[h]);
                }
                float nrm = bf16_to_float(*reinterpret_cast<const uint16_t *>(kr + PG.k_norm_off + 2 * off));
                if (C.qjl) {
                    const uint32_t *sw = reinterpret_cast<const uint32_t *>(kr + PG.k_sign_off + off * C.k_sign_bytes +
                                                                            sl * (CW / 8));
                    const float gam = bf16_to_float(*reinterpret_cast<const uint16_t *>(kr + PG.k_gamma_off + 2 * off));
#pragma unroll
                    for (int w = 0; w < CW / 32; ++w) {
                        const uint32_t bits = sw[w];
#pragma unroll 8
                        for (int u = 0; u < 32; ++u) {
                            const bool pos_bit = (bits >> u) & 1u;
#pragma unroll
                            for (int h = 0; h < G; ++h) {
                                const float v = sm.qs[h][j0 + 32 * w + u];
                                ds[h] += pos_bit ? v : -v;
                            }
                        }
                    }
#pragma unroll
                    for (int h = 0; h < G; ++h) dc[h] = fmaf(dc[h], inv_sqrtd, qcoef * gam * ds[h]);
                } else {
#pragma unroll
                    for (int h = 0; h < G; ++h) dc[h] *= inv_sqrtd;
                }
                const float f = A.sm_scale * nrm;
#pragma unroll
                for (int h = 0; h < G; ++h) sm.part[sl][h][tt] = f * dc[h];
            } else {
#pragma unroll
                for (int h = 0; h < G; ++h) sm.part[sl][h][tt] = -INFINITY;
            }
        }
        __syncthreads();
        // ---- online softmax: one warp per head, two tokens per lane ----
        for (int h = warp; h < G; h += D / 32) {
            float s0 = 0.f, s1 = 0.f;
#pragma unroll
            for (int s = 0; s < SL; ++s) {
                s0 += sm.part[s][h][lane];
                s1 += sm.part[s][h][lane + 32];
            }
            const float mc = warp_max(fmaxf(s0, s1));
            const float m_old = sm.m_run[h];
            const float m_new = fmaxf(m_old, mc);
            float p0 = 0.f, p1 = 0.f, alpha = 1.f;
            if (m_new != -INFINITY) {
                p0 = __expf(s0 - m_new);
                p1 = __expf(s1 - m_new);
                alpha = __expf(m_old - m_new);
            }
            sm.prob[h][lane] = p0;
            sm.prob[h][lane + 32] = p1;
            const float ps = warp_sum(p0 + p1);
            if (lane == 0) {
                sm.alpha[h] = alpha;
                sm.m_run[h] = m_new;
                sm.l_run[h] = sm.l_run[h] * alpha + ps;
            }
        }
        __syncthreads();
        // ---- P.V: thread j owns coordinate j for all G heads ----
        {
            const int j = tid;
#pragma unroll
            for (int h = 0; h < G; ++h) acc[h] *= sm.alpha[h];
            const int ntok = min(npc * P, L - cp * P);
            const int vbit = j * vb;
            const int gi = j / C.group;
            for (int tt = 0; tt < ntok; ++tt) {
                const int q = tt / P, off = tt - q * P;
                if (!sm.page_ok[q]) continue;
                const uint8_t *vr = vpg + q * PG.v_page;
                const uint8_t *cb = vr + off * C.v_code_bytes;
                const uint32_t w = cb[vbit >> 3] | (static_cast<uint32_t>(cb[(vbit >> 3) + 1]) << 8);
                const float code = static_cast<float>((w >> (vbit & 7)) & ((1u << vb) - 1u));
                const __half2 sz = *reinterpret_cast<const __half2 *>(vr + PG.v_meta_off + off * C.v_meta_bytes + 4 * gi);
                const float2 szf = __half22float2(sz);
                const float val = fmaf(code, szf.x, szf.y);
#pragma unroll
                for (int h = 0; h < G; ++h) acc[h] = fmaf(sm.prob[h][tt], val, acc[h]);
            }
        }
    }
    __syncthreads();
#pragma unroll
    for (int h = 0; h < G; ++h) acc_out[static_cast<size_t>(h) * D + tid] = acc[h];
    if (tid < G) {
        ml_out[2 * tid] = sm.m_run[tid];
        ml_out[2 * tid + 1] = sm.l_run[tid];
    }
}

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
            const float w = __expf(m - M);
            den = fmaf(w, l, den);
            num = fmaf(w, A.ws.acc[(s * rows + row) * D + j], num);
        }
    }
    const float o = (den > 0.f) ? num / den : 0.f;
    A.out[static_cast<size_t>(row) * D + j] = float_to_bf16_bits(o);
}

template <int D, int G>
cudaError_t launch_decode_dg(const Codec &c, const PageGeom &pg, const DecodeArgs &a, cudaStream_t st)
{
    const size_t dyn = static_cast<size_t>(kChunk / pg.P) * (pg.k_page + pg.v_page) + 16;
    static bool attr_set[64] = {};
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if (dev < 0 || dev >= 64 || !attr_set[dev]) {
        e = cudaFuncSetAttribute(decode_kernel<D, G>, cudaFuncAttributeMaxDynamicSharedMemorySize, 64 * 1024);
        if (e != cudaSuccess) return e;
        if (dev >= 0 && dev < 64) attr_set[dev] = true;
    }
    dim3 grid(a.splits, a.Hkv, a.B);
    decode_kernel<D, G><<<grid, D, dyn, st>>>(c, pg, a);
    return cudaGetLastError();
}

template <int D>
cudaError_t launch_decode_d(const Codec &c, const PageGeom &pg, const DecodeArgs &a, cudaStream_t st)
{
    const int G = a.Hq / a.Hkv;
    qrot_kernel<D><<<a.B * a.Hq, D, 0, st>>>(c, a.q, a.ws.qrot, a.ws.qs);
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return e;
    switch (G) {
    case 1: e = launch_decode_dg<D, 1>(c, pg, a, st); break;
    case 2: e = launch_decode_dg<D, 2>(c, pg, a, st); break;
    case 3: e = launch_decode_dg<D, 3>(c, pg, a, st); break;
    case 4: e = launch_decode_dg<D, 4>(c, pg, a, st); break;
    case 5: e = launch_decode_dg<D, 5>(c, pg, a, st); break;
    case 6: e = launch_decode_dg<D, 6>(c, pg, a, st); break;
    case 7: e = launch_decode_dg<D, 7>(c, pg, a, st); break;
    case 8: e = launch_decode_dg<D, 8>(c, pg, a, st); break;
    default: return cudaErrorInvalidValue;
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
