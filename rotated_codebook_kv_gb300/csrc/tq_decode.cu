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
    return al(rows * d * 4) * 3 + al(static_cast<size_t>(splits) * rows * d * 4) +
           al(static_cast<size_t>(splits) * rows * 2 * 4);
}

DecodeWorkspace carve_decode_workspace(void *base, int d, int B, int Hq, int splits)
{
    auto al = [](size_t x) { return (x + 255) / 256 * 256; };
    const size_t rows = static_cast<size_t>(B) * Hq;
    char *p = static_cast<char *>(base);
    DecodeWorkspace w;
    w.out32 = reinterpret_cast<float *>(p);
    p += al(rows * d * 4);
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
// kQRows query rows per block of 2 D threads: thread (i, half) sums coordinate i
// of each row over half of the inner index, so every element of Pi (and S)
// read from L2 feeds kQRows independent FMA chains; the halves add in shared memory.
template <int D, int kQRows>
__global__ void __launch_bounds__(2 * D) qrot_kernel(const Codec C, const uint16_t *__restrict__ q, float *qrot,
                                                     float *qs, int rows)
{
    __shared__ float sq[kQRows][D];
    __shared__ float part[kQRows][D];
    const int r0 = blockIdx.x * kQRows;
    const int i = threadIdx.x % D, hf = threadIdx.x / D;
    const int nr = min(kQRows, rows - r0);
    if (hf == 0) {
#pragma unroll
        for (int r = 0; r < kQRows; ++r) sq[r][i] = (r < nr) ? bf16_to_float(q[static_cast<int64_t>(r0 + r) * D + i]) : 0.f;
    }
    __syncthreads();
    auto matvec = [&](const float *__restrict__ MT, float (&a)[kQRows]) {  // a[r] = sum_j MT[j][i] sq[r][j], j in this half
#pragma unroll
        for (int r = 0; r < kQRows; ++r) a[r] = 0.f;
        const int j0 = hf * (D / 2);
#pragma unroll 16
        for (int j = j0; j < j0 + D / 2; ++j) {
            const float m = __ldg(MT + j * D + i);
#pragma unroll
            for (int r = 0; r < kQRows; ++r) a[r] = fmaf(m, sq[r][j], a[r]);
        }
        if (hf == 1) {
#pragma unroll
            for (int r = 0; r < kQRows; ++r) part[r][i] = a[r];
        }
        __syncthreads();
        if (hf == 0) {
#pragma unroll
            for (int r = 0; r < kQRows; ++r) a[r] += part[r][i];
        }
    };
    float a[kQRows];
    matvec(C.PiT, a);
    if (hf == 0) {
#pragma unroll
        for (int r = 0; r < kQRows; ++r)
            if (r < nr) qrot[static_cast<int64_t>(r0 + r) * D + i] = a[r];
    }
    if (!C.qjl) return;
    __syncthreads();  // every thread has read sq and part
    if (hf == 0) {
#pragma unroll
        for (int r = 0; r < kQRows; ++r) sq[r][i] = a[r];
    }
    __syncthreads();
    matvec(C.ST, a);
    if (hf == 0) {
#pragma unroll
        for (int r = 0; r < kQRows; ++r)
            if (r < nr) qs[static_cast<int64_t>(r0 + r) * D + i] = a[r];
    }
}

// Query pre-rotation for many rows (prefill) on the tensor cores: q_rot = Pi q and
// q_s = M q with M = S Pi (equal to S q_rot), by mma.sync m16n8k16 from the bf16
// query made exact in fp16 by a power-of-two row scale, times Pi 2^10 and M 2^10 as
// fp16 high + low fragment images read from L2 (products exact, fp32 accumulation,
// ~22 significant bits).  64 rows per CTA of 8 warps; warp w computes the output
// columns [D/8 w, D/8 (w + 1)) of all 64 rows.
constexpr int kQmRows = 64;

__device__ __forceinline__ void qm_mma(float (&c)[4], uint32_t a0, uint32_t a1, uint32_t a2, uint32_t a3, uint32_t b0,
                                       uint32_t b1)
{
    asm volatile("mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
                 "{%0,%1,%2,%3};"
                 : "+f"(c[0]), "+f"(c[1]), "+f"(c[2]), "+f"(c[3])
                 : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}

template <int D>
__global__ void __launch_bounds__(256) qrot_mma_kernel(const Codec C, const uint16_t *__restrict__ q, float *qrot,
                                                       float *qs, int rows)
{
    constexpr int TM = kQmRows, KA = D + 8, KS = D / 16, NPW = D / 64, E = D / 32;
    __shared__ __align__(16) __half qa[TM * KA];
    __shared__ float rsc[TM];  // 2^-(10 + row exponent): back to Pi q
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int r0 = blockIdx.x * TM;
    for (int row = warp; row < TM; row += 8) {
        const int r = r0 + row;
        float x[E];
        float mx = 0.f;
#pragma unroll
        for (int m = 0; m < E; ++m) {
            x[m] = (r < rows) ? bf16_to_float(q[static_cast<int64_t>(r) * D + lane + 32 * m]) : 0.f;
            mx = fmaxf(mx, fabsf(x[m]));
        }
        mx = warp_max(mx);
        // mx < 2^ex; the row times 2^(15 - ex) has its largest element in [2^14, 2^15)
        int ex = static_cast<int>((__float_as_uint(mx) >> 23) & 0xffu) - 126;
        if (ex < -100) ex = -100;
        const bool ok = mx > 0.f && mx <= 3.0e38f;
        const float sc = ok ? __uint_as_float(static_cast<uint32_t>(15 - ex + 127) << 23) : 0.f;
#pragma unroll
        for (int m = 0; m < E; ++m) qa[row * KA + lane + 32 * m] = __float2half_rn(x[m] * sc);
        if (lane == 0) rsc[row] = ok ? __uint_as_float(static_cast<uint32_t>(127 - 25 + ex) << 23) : 0.f;
    }
    __syncthreads();
    const int rr = lane >> 2, qq = lane & 3;
    const uint32_t qab = static_cast<uint32_t>(__cvta_generic_to_shared(qa));
    for (int mat = 0; mat < (C.qjl ? 2 : 1); ++mat) {
        const uint4 *__restrict__ frag = mat ? C.m_frag : C.pi_frag;
        float *out = mat ? qs : qrot;
        float acc[TM / 16][NPW][4];
#pragma unroll
        for (int m = 0; m < TM / 16; ++m)
#pragma unroll
            for (int n = 0; n < NPW; ++n) acc[m][n][0] = acc[m][n][1] = acc[m][n][2] = acc[m][n][3] = 0.f;
#pragma unroll 2
        for (int s = 0; s < KS; ++s) {
            uint4 bf[NPW];
#pragma unroll
            for (int n = 0; n < NPW; ++n) bf[n] = __ldg(frag + ((warp * NPW + n) * KS + s) * 32 + lane);
#pragma unroll
            for (int m = 0; m < TM / 16; ++m) {
                uint32_t a0, a1, a2, a3;
                const uint32_t addr = qab + 2u * ((16 * m + (lane & 15)) * KA + 16 * s + 8 * (lane >> 4));
                asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0,%1,%2,%3}, [%4];"
                             : "=r"(a0), "=r"(a1), "=r"(a2), "=r"(a3) : "r"(addr));
#pragma unroll
                for (int n = 0; n < NPW; ++n) {
                    qm_mma(acc[m][n], a0, a1, a2, a3, bf[n].z, bf[n].w);  // low parts first
                    qm_mma(acc[m][n], a0, a1, a2, a3, bf[n].x, bf[n].y);
                }
            }
        }
#pragma unroll
        for (int m = 0; m < TM / 16; ++m) {
#pragma unroll
            for (int h = 0; h < 2; ++h) {
                const int row = 16 * m + rr + 8 * h;
                if (r0 + row >= rows) continue;
                const float f = rsc[row];
#pragma unroll
                for (int n = 0; n < NPW; ++n) {
                    const int col = 8 * (warp * NPW + n) + 2 * qq;
                    *reinterpret_cast<float2 *>(out + static_cast<int64_t>(r0 + row) * D + col) =
                        make_float2(acc[m][n][2 * h] * f, acc[m][n][2 * h + 1] * f);
                }
            }
        }
    }
}

// ---- (2) split-K decode: see tq_decode_mma.cuh ---------------------------------

// ---- (3) log-sum-exp combine -------------------------------------------------
// One block per (b, h): the split weights 2^(m_s - M) are computed once into
// shared memory, then thread j sums its coordinate over the splits.
constexpr int kMaxSplits = 1024;

template <int D, bool UNROT>
__global__ void __launch_bounds__(D) combine_kernel(const Codec C, const DecodeArgs A)
{
    __shared__ float sw[kMaxSplits];
    __shared__ float so[UNROT ? D : 1];
    __shared__ float red[D / 32];
    __shared__ float s_den;
    const int row = blockIdx.x;  // b * Hq + h
    const int j = threadIdx.x, lane = j & 31, warp = j >> 5;
    const size_t rows = static_cast<size_t>(A.B) * A.Hq;
    // M = max over splits with l > 0
    float M = -INFINITY;
    for (int s = j; s < A.splits; s += D) {
        const float2 ml = *reinterpret_cast<const float2 *>(A.ws.ml + (s * rows + row) * 2);
        if (ml.y > 0.f) M = fmaxf(M, ml.x);
    }
    M = warp_max(M);
    if (lane == 0) red[warp] = M;
    __syncthreads();
    M = red[0];
#pragma unroll
    for (int w = 1; w < D / 32; ++w) M = fmaxf(M, red[w]);
    __syncthreads();
    float den = 0.f;
    for (int s = j; s < A.splits; s += D) {
        const float2 ml = *reinterpret_cast<const float2 *>(A.ws.ml + (s * rows + row) * 2);
        const float w = (ml.y > 0.f && M != -INFINITY) ? exp2f(ml.x - M) : 0.f;
        sw[s] = w;
        den = fmaf(w, (ml.y > 0.f) ? ml.y : 0.f, den);
    }
    den = warp_sum(den);
    if (lane == 0) red[warp] = den;
    __syncthreads();
    if (j == 0) {
        float d = 0.f;
#pragma unroll
        for (int w = 0; w < D / 32; ++w) d += red[w];
        s_den = d;
    }
    __syncthreads();
    const float* acc = A.ws.acc + row * D + j;
    float n0 = 0.f, n1 = 0.f, n2 = 0.f, n3 = 0.f;
    int s = 0;
    for (; s + 4 <= A.splits; s += 4) {
        const float w0 = sw[s], w1 = sw[s + 1], w2 = sw[s + 2], w3 = sw[s + 3];
        // skipped splits may hold stale partials: read only those with weight
        if (w0 != 0.f) n0 = fmaf(w0, acc[(s + 0) * rows * D], n0);
        if (w1 != 0.f) n1 = fmaf(w1, acc[(s + 1) * rows * D], n1);
        if (w2 != 0.f) n2 = fmaf(w2, acc[(s + 2) * rows * D], n2);
        if (w3 != 0.f) n3 = fmaf(w3, acc[(s + 3) * rows * D], n3);
    }
    for (; s < A.splits; ++s)
        if (sw[s] != 0.f) n0 = fmaf(sw[s], acc[s * rows * D], n0);
    const float num = (n0 + n1) + (n2 + n3);
    const float dd = s_den;
    float o = (dd > 0.f) ? num / dd : 0.f;
    if constexpr (UNROT) {
        // values coded by the rotation: the merged output is in the rotated space (with
        // the table's fp16 scale, the 2^-4 of the weights and 1/sqrt(d) left to apply):
        // o = Pi^T o_rot, d^2 FMAs per query head
        so[j] = o * (16.f / (C.vlut_scale * sqrtf(static_cast<float>(D))));
        __syncthreads();
        float a = 0.f;
#pragma unroll 8
        for (int i = 0; i < D; ++i) a = fmaf(__ldg(C.Pi + i * D + j), so[i], a);
        o = a;
    }
    A.ws.out32[static_cast<size_t>(row) * D + j] = o;
    A.out[static_cast<size_t>(row) * D + j] = float_to_bf16_bits(o);
}

// One split and no un-rotation: o = acc / l per row (what combine_kernel computes
// when there is one split), four coordinates per thread.
template <int D>
__global__ void __launch_bounds__(256) combine1_kernel(const DecodeArgs A)
{
    const int64_t rows = static_cast<int64_t>(A.B) * A.Hq;
    const int64_t idx = static_cast<int64_t>(blockIdx.x) * 256 + threadIdx.x;  // float4 index
    if (idx >= rows * (D / 4)) return;
    const int64_t row = idx / (D / 4);
    const float2 ml = *reinterpret_cast<const float2 *>(A.ws.ml + row * 2);
    const float4 a = reinterpret_cast<const float4 *>(A.ws.acc)[idx];
    const bool live = ml.y > 0.f;
    const float4 o = live ? make_float4(a.x / ml.y, a.y / ml.y, a.z / ml.y, a.w / ml.y) : make_float4(0.f, 0.f, 0.f, 0.f);
    reinterpret_cast<float4 *>(A.ws.out32)[idx] = o;
    const uint32_t lo = float_to_bf16_bits(o.x) | (static_cast<uint32_t>(float_to_bf16_bits(o.y)) << 16);
    const uint32_t hi = float_to_bf16_bits(o.z) | (static_cast<uint32_t>(float_to_bf16_bits(o.w)) << 16);
    reinterpret_cast<uint2 *>(A.out)[idx] = make_uint2(lo, hi);
}

template <int D, int KB, int VB>
cudaError_t launch_dmma(const Codec &c, const PageGeom &pg, const DecodeArgs &a, cudaStream_t st)
{
    if (a.Tq > 1) {  // prefill: head_dim 128 on tensor memory, 256 on this kernel with query columns
        if (c.d == 128) return launch_prefill_tc(c, pg, a, st);
        return c.vmse ? launch_dmma_vmse(c, pg, a, st) : launch_dmma_prefill(c, pg, a, st);
    }
    if (c.vmse) return launch_dmma_vmse(c, pg, a, st);
    const size_t smem = dmma::DecSmem<D, KB>::bytes(pg);
    cudaError_t e = ensure_smem_attr(reinterpret_cast<const void *>(dmma::decode_mma_kernel<D, KB, VB, false>), smem);
    if (e != cudaSuccess) return e;
    dim3 grid(a.splits, a.Hkv, a.B * ((a.Tq + a.qpc - 1) / a.qpc));
    dmma::decode_mma_kernel<D, KB, VB, false><<<grid, dmma::kThreads, smem, st>>>(c, pg, a);
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
    const int qrows = a.B * a.Tq * a.Hq;
    // thousands of rows (prefill): tensor cores; a few rows per kv head (decode): fp32
    if (qrows >= 32 * kQmRows)
        qrot_mma_kernel<D><<<(qrows + kQmRows - 1) / kQmRows, 256, 0, st>>>(c, a.q, a.ws.qrot, a.ws.qs, qrows);
    else
        qrot_kernel<D, 4><<<(qrows + 3) / 4, 2 * D, 0, st>>>(c, a.q, a.ws.qrot, a.ws.qs, qrows);
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return e;
    switch (c.k_bits) {
    case 2: e = launch_dmma_kb<D, 2>(c, pg, a, st); break;
    case 3: e = launch_dmma_kb<D, 3>(c, pg, a, st); break;
    default: e = launch_dmma_kb<D, 4>(c, pg, a, st); break;
    }
    if (e != cudaSuccess) return e;
    DecodeArgs rows = a;  // the combine merges B * Tq * Hq output rows
    rows.B = a.B * a.Tq;
    rows.Tq = 1;
    return launch_combine(c, rows, st, c.vmse != 0);
}

}  // namespace

cudaError_t launch_combine(const Codec &c, const DecodeArgs &a, cudaStream_t st, bool unrotate)
{
    if (a.splits == 1 && !unrotate) {
        const int64_t n4 = static_cast<int64_t>(a.B) * a.Hq * (c.d / 4);
        const unsigned blocks = static_cast<unsigned>((n4 + 255) / 256);
        if (c.d == 128) combine1_kernel<128><<<blocks, 256, 0, st>>>(a);
        else combine1_kernel<256><<<blocks, 256, 0, st>>>(a);
        return cudaGetLastError();
    }
    if (c.d == 128) {
        if (unrotate) combine_kernel<128, true><<<a.B * a.Hq, 128, 0, st>>>(c, a);
        else combine_kernel<128, false><<<a.B * a.Hq, 128, 0, st>>>(c, a);
    } else {
        if (unrotate) combine_kernel<256, true><<<a.B * a.Hq, 256, 0, st>>>(c, a);
        else combine_kernel<256, false><<<a.B * a.Hq, 256, 0, st>>>(c, a);
    }
    return cudaGetLastError();
}

cudaError_t launch_decode(const Codec &c, const PageGeom &pg, const DecodeArgs &a, cudaStream_t st)
{
    if (c.d == 128) return launch_decode_d<128>(c, pg, a, st);
    return launch_decode_d<256>(c, pg, a, st);
}

}  // namespace tq
