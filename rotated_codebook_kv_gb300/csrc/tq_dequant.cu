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

// ---- many slots: the same reconstruction on the tensor cores ------------------
// 64 (slot, kv head) rows per CTA of 8 warps.  A row's u = c[code] / sqrt(d) is staged
// in fp32; with QJL, w = S^T sigma comes from mma.sync with sigma (exact in fp16)
// against S^T 2^12 as fp16 high + low fragments and u += sqrt(pi/2) / d gamma w; then
// u times a power of two per row is split into fp16 high + low parts and Pi^T u runs
// against Pi^T 2^10 in the same form (three products per step, ~22 significant bits,
// fp32 accumulation).  Values coded per group are written directly; values coded by
// the rotation take the key steps without QJL.
constexpr int kDqRows = 64;

__device__ __forceinline__ void dq_mma(float (&c)[4], uint32_t a0, uint32_t a1, uint32_t a2, uint32_t a3, uint32_t b0,
                                       uint32_t b1)
{
    asm volatile("mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
                 "{%0,%1,%2,%3};"
                 : "+f"(c[0]), "+f"(c[1]), "+f"(c[2]), "+f"(c[3])
                 : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}

// acc = A (TM x D, fp16 in shared memory, row stride D + 8) times W^T from a fragment
// image, for warp w's output columns [D/8 w, D/8 (w + 1)); with LO, A's low parts
// (al, same layout) add the two cross products: a_h w_l + a_l w_h + a_h w_h.
template <int D, bool LO>
__device__ __forceinline__ void dq_product(const uint4 *__restrict__ frag, const __half *ah, const __half *al,
                                           float (&acc)[kDqRows / 16][D / 64][4])
{
    constexpr int KS = D / 16, NPW = D / 64, KA = D + 8;
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
#pragma unroll
    for (int m = 0; m < kDqRows / 16; ++m)
#pragma unroll
        for (int n = 0; n < NPW; ++n) acc[m][n][0] = acc[m][n][1] = acc[m][n][2] = acc[m][n][3] = 0.f;
    const uint32_t hb = static_cast<uint32_t>(__cvta_generic_to_shared(ah));
    const uint32_t lb = LO ? static_cast<uint32_t>(__cvta_generic_to_shared(al)) : 0u;
#pragma unroll 2
    for (int s = 0; s < KS; ++s) {
        uint4 bf[NPW];
#pragma unroll
        for (int n = 0; n < NPW; ++n) bf[n] = __ldg(frag + ((warp * NPW + n) * KS + s) * 32 + lane);
#pragma unroll
        for (int m = 0; m < kDqRows / 16; ++m) {
            const uint32_t off = 2u * ((16 * m + (lane & 15)) * KA + 16 * s + 8 * (lane >> 4));
            uint32_t a0, a1, a2, a3;
            asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0,%1,%2,%3}, [%4];"
                         : "=r"(a0), "=r"(a1), "=r"(a2), "=r"(a3) : "r"(hb + off));
            if constexpr (LO) {
                uint32_t l0, l1, l2, l3;
                asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0,%1,%2,%3}, [%4];"
                             : "=r"(l0), "=r"(l1), "=r"(l2), "=r"(l3) : "r"(lb + off));
#pragma unroll
                for (int n = 0; n < NPW; ++n) {
                    dq_mma(acc[m][n], a0, a1, a2, a3, bf[n].z, bf[n].w);
                    dq_mma(acc[m][n], l0, l1, l2, l3, bf[n].x, bf[n].y);
                }
            } else {
#pragma unroll
                for (int n = 0; n < NPW; ++n) dq_mma(acc[m][n], a0, a1, a2, a3, bf[n].z, bf[n].w);
            }
#pragma unroll
            for (int n = 0; n < NPW; ++n) dq_mma(acc[m][n], a0, a1, a2, a3, bf[n].x, bf[n].y);
        }
    }
}

template <int D>
struct DqSmem {
    static constexpr int KA = D + 8;
    static constexpr size_t kU = sizeof(float) * kDqRows * D;    // u (fp32)
    static constexpr size_t kA = sizeof(__half) * kDqRows * KA;  // one fp16 operand tile
    static constexpr size_t kBytes = kU + 2 * kA;
};

template <int D>
__global__ void __launch_bounds__(256) dequant_mma_kernel(const Codec C, const PageGeom G, const uint8_t *__restrict__ kc,
                                                          const uint8_t *__restrict__ vc, int64_t num_blocks, int Hkv,
                                                          const int64_t *__restrict__ slots, int64_t rows,
                                                          uint16_t *__restrict__ kout, uint16_t *__restrict__ vout)
{
    using SM = DqSmem<D>;
    constexpr int KA = SM::KA, E = D / 32, NPW = D / 64, RPW = kDqRows / 8;  // RPW rows per warp
    constexpr int OS = D / 2 + 4;  // bf16-pair row stride of the output tile (rows in different banks)
    extern __shared__ __align__(16) unsigned char smem[];
    float *u = reinterpret_cast<float *>(smem);
    __half *ah = reinterpret_cast<__half *>(smem + SM::kU);
    __half *al = reinterpret_cast<__half *>(smem + SM::kU + SM::kA);
    __shared__ int64_t s_rec[kDqRows];  // record (block * Hkv + head), -1: row skipped
    __shared__ int s_off[kDqRows];
    __shared__ float s_n[kDqRows], s_g[kDqRows], s_sc[kDqRows];
    __shared__ float s_cent[2][16];  // key and value centroids / sqrt(d)
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int rr = lane >> 2, qq = lane & 3;
    const int64_t r0 = static_cast<int64_t>(blockIdx.x) * kDqRows;  // row = slot index * Hkv + head
    const float rsd = rsqrtf(static_cast<float>(D));
    if (tid < 16) {
        s_cent[0][tid] = C.centroids[tid] * rsd;
        s_cent[1][tid] = C.vcentroids[tid] * rsd;
    }
    if (tid < kDqRows) {
        const int64_t r = r0 + tid;
        int64_t rec = -1;
        int off = 0;
        if (r < rows) {
            const int64_t t = r / Hkv;
            const int h = static_cast<int>(r - t * Hkv);
            const int64_t slot = slots[t];
            if (slot >= 0) {
                const int64_t blk = slot / G.P;
                if (blk < num_blocks) {
                    rec = blk * Hkv + h;
                    off = static_cast<int>(slot - blk * G.P);
                } else if (h == 0) {
                    atomicOr(C.status, TQ_DEVERR_BLOCK_RANGE);
                }
            }
        }
        s_rec[tid] = rec;
        s_off[tid] = off;
    }
    __syncthreads();

    // The E codes of lane l (coordinates E l .. E l + E - 1, E b <= 32 bits) of warp
    // row k from two aligned words of the record's packed codes; every row's words
    // are loaded before any is decoded.  The word after a row's codes lies inside
    // its page (signs, norms or value metadata follow the codes).
    auto load_codes = [&](bool values, uint32_t (&cw)[RPW], uint32_t (&aux)[RPW], float (&nrm)[RPW],
                          float (&gam)[RPW]) {
        const int bits = values ? C.v_bits : C.k_bits;
        const int cbytes = values ? C.v_code_bytes : C.k_code_bytes;
        const int bit0 = E * lane * bits;
#pragma unroll
        for (int k = 0; k < RPW; ++k) {
            const int row = warp + 8 * k;
            const int64_t rec = s_rec[row];
            uint32_t w0 = 0u, w1 = 0u;
            aux[k] = 0u;
            nrm[k] = gam[k] = 0.f;
            if (rec >= 0) {
                const int off = s_off[row];
                const uint8_t *pr = values ? vc + rec * G.v_page : kc + rec * G.k_page;
                const uint32_t *wp = reinterpret_cast<const uint32_t *>(pr + static_cast<int64_t>(off) * cbytes);
                w0 = __ldg(wp + (bit0 >> 5));
                w1 = __ldg(wp + (bit0 >> 5) + 1);
                if (values && !C.vmse) {  // the lane's group: its (scale, zero) pair
                    aux[k] = __ldg(reinterpret_cast<const uint32_t *>(pr + G.v_meta_off +
                                                                     static_cast<int64_t>(off) * C.v_meta_bytes) +
                                   (E * lane) / C.group);
                } else {
                    nrm[k] = bf16_to_float(__ldg(reinterpret_cast<const uint16_t *>(
                        pr + (values ? G.v_meta_off : G.k_norm_off) + 2 * off)));
                    if (!values && C.qjl) {
                        aux[k] = __ldg(pr + G.k_sign_off + static_cast<int64_t>(off) * C.k_sign_bytes + (E * lane >> 3));
                        gam[k] = bf16_to_float(__ldg(reinterpret_cast<const uint16_t *>(pr + G.k_gamma_off + 2 * off)));
                    }
                }
            }
            cw[k] = __funnelshift_r(w0, w1, bit0 & 31);
        }
    };

    // u = c[code] / sqrt(d) (0 for skipped rows), with QJL the signs into ah
    auto stage = [&](bool values) {
        uint32_t cw[RPW], aux[RPW];
        float nrm[RPW], gam[RPW];
        load_codes(values, cw, aux, nrm, gam);
        const int bits = values ? C.v_bits : C.k_bits;
        const uint32_t mask = (1u << bits) - 1u;
        const bool qjl = !values && C.qjl;
        const float *cent = s_cent[values ? 1 : 0];
#pragma unroll
        for (int k = 0; k < RPW; ++k) {
            const int row = warp + 8 * k;
            const bool live = s_rec[row] >= 0;
            float x[E];
#pragma unroll
            for (int m = 0; m < E; ++m) x[m] = live ? cent[(cw[k] >> (bits * m)) & mask] : 0.f;
#pragma unroll
            for (int m = 0; m < E; m += 4)
                *reinterpret_cast<float4 *>(u + row * D + E * lane + m) = make_float4(x[m], x[m + 1], x[m + 2], x[m + 3]);
            if (qjl) {
                const uint32_t sb = aux[k] >> ((E * lane) & 7);
                uint32_t h2[E / 2];
#pragma unroll
                for (int m = 0; m < E; m += 2) {
                    // +-1 in fp16 (0x3C00 / 0xBC00) where the row is live, else 0
                    const uint32_t lo = live ? (((sb >> m) & 1u) ? 0x3C00u : 0xBC00u) : 0u;
                    const uint32_t hi = live ? (((sb >> (m + 1)) & 1u) ? 0x3C00u : 0xBC00u) : 0u;
                    h2[m / 2] = lo | (hi << 16);
                }
                if constexpr (E == 4)
                    *reinterpret_cast<uint2 *>(ah + row * KA + E * lane) = make_uint2(h2[0], h2[1]);
                else
                    *reinterpret_cast<uint4 *>(ah + row * KA + E * lane) = make_uint4(h2[0], h2[1], h2[2], h2[3]);
            }
            if (lane == 0) {
                s_n[row] = nrm[k];
                s_g[row] = gam[k];
            }
        }
        __syncthreads();
    };
    // u times 2^(15 - e) per row (largest |u| in [2^14, 2^15)) as fp16 high + low parts
    auto split = [&]() {
        for (int row = warp; row < kDqRows; row += 8) {
            float x[E], mx = 0.f;
#pragma unroll
            for (int m = 0; m < E; ++m) {
                x[m] = u[row * D + lane + 32 * m];
                mx = fmaxf(mx, fabsf(x[m]));
            }
            mx = warp_max(mx);
            const bool ok = mx > 0.f && mx <= 3.0e38f;
            int ex = static_cast<int>((__float_as_uint(mx) >> 23) & 0xffu) - 126;
            if (ex < -100) ex = -100;
            const float sc = ok ? __uint_as_float(static_cast<uint32_t>(127 + 15 - ex) << 23) : 0.f;
#pragma unroll
            for (int m = 0; m < E; ++m) {
                const float y = x[m] * sc;
                const __half h = __float2half_rn(y);
                ah[row * KA + lane + 32 * m] = h;
                al[row * KA + lane + 32 * m] = __float2half_rn(y - __half2float(h));
            }
            if (lane == 0) s_sc[row] = ok ? __uint_as_float(static_cast<uint32_t>(127 + ex - 25) << 23) : 0.f;
        }
        __syncthreads();
    };
    // out[row] = n Pi^T u in bf16: the tile is assembled in shared memory (over u,
    // already split into ah / al) and written as whole 16-byte pieces of rows
    auto rotate_out = [&](uint16_t *out) {
        float acc[kDqRows / 16][NPW][4];
        dq_product<D, true>(C.pit_frag, ah, al, acc);
        uint32_t *ob = reinterpret_cast<uint32_t *>(u);
#pragma unroll
        for (int m = 0; m < kDqRows / 16; ++m)
#pragma unroll
            for (int h2 = 0; h2 < 2; ++h2) {
                const int row = 16 * m + rr + 8 * h2;
                const float f = s_sc[row] * s_n[row];
#pragma unroll
                for (int n = 0; n < NPW; ++n) {
                    const int col = 8 * (warp * NPW + n) + 2 * qq;
                    ob[row * OS + col / 2] = float_to_bf16_bits(acc[m][n][2 * h2] * f) |
                                             (static_cast<uint32_t>(float_to_bf16_bits(acc[m][n][2 * h2 + 1] * f)) << 16);
                }
            }
        __syncthreads();
        for (int e = tid; e < kDqRows * (D / 8); e += 256) {
            const int row = e / (D / 8), c8 = e - row * (D / 8);
            if (s_rec[row] < 0) continue;
            *reinterpret_cast<uint4 *>(out + (r0 + row) * D + 8 * c8) =
                *reinterpret_cast<const uint4 *>(ob + row * OS + 4 * c8);
        }
        __syncthreads();
    };

    // ---- keys ----
    stage(false);
    if (C.qjl) {  // u += sqrt(pi/2) / d gamma S^T sigma
        float acc[kDqRows / 16][NPW][4];
        dq_product<D, false>(C.st_frag, ah, nullptr, acc);
#pragma unroll
        for (int m = 0; m < kDqRows / 16; ++m)
#pragma unroll
            for (int h2 = 0; h2 < 2; ++h2) {
                const int row = 16 * m + rr + 8 * h2;
                const float f = s_g[row] * (1.2533141373155003f / static_cast<float>(D)) * (1.f / 4096.f);
#pragma unroll
                for (int n = 0; n < NPW; ++n) {
                    const int col = 8 * (warp * NPW + n) + 2 * qq;
                    u[row * D + col] = fmaf(f, acc[m][n][2 * h2], u[row * D + col]);
                    u[row * D + col + 1] = fmaf(f, acc[m][n][2 * h2 + 1], u[row * D + col + 1]);
                }
            }
        __syncthreads();
    }
    split();
    rotate_out(kout);

    // ---- values ----
    if (C.vmse) {
        stage(true);
        split();
        rotate_out(vout);
        return;
    }
    // code * scale + zero per group: the lane's E values of one group, written as
    // one 8- or 16-byte piece
    uint32_t cw[RPW], meta[RPW];
    float nrm[RPW], gam[RPW];
    load_codes(true, cw, meta, nrm, gam);
    const uint32_t vmask = (1u << C.v_bits) - 1u;
#pragma unroll
    for (int k = 0; k < RPW; ++k) {
        const int row = warp + 8 * k;
        if (s_rec[row] < 0) continue;
        const float2 sz = __half22float2(*reinterpret_cast<const __half2 *>(&meta[k]));
        uint32_t o[E / 2];
#pragma unroll
        for (int m = 0; m < E; m += 2) {
            const float a = fmaf(static_cast<float>((cw[k] >> (C.v_bits * m)) & vmask), sz.x, sz.y);
            const float b = fmaf(static_cast<float>((cw[k] >> (C.v_bits * (m + 1))) & vmask), sz.x, sz.y);
            o[m / 2] = float_to_bf16_bits(a) | (static_cast<uint32_t>(float_to_bf16_bits(b)) << 16);
        }
        if constexpr (E == 4)
            *reinterpret_cast<uint2 *>(vout + (r0 + row) * D + E * lane) = make_uint2(o[0], o[1]);
        else
            *reinterpret_cast<uint4 *>(vout + (r0 + row) * D + E * lane) = make_uint4(o[0], o[1], o[2], o[3]);
    }
}

}  // namespace

cudaError_t launch_dequant(const Codec &c, const PageGeom &pg, const uint8_t *kc, const uint8_t *vc,
                           int64_t num_blocks, int Hkv, const int64_t *slots, int64_t T, uint16_t *k_out,
                           uint16_t *v_out, cudaStream_t st)
{
    const int64_t rows = T * Hkv;
    if (rows >= 32 * kDqRows) {  // many slots: tensor cores
        const unsigned blocks = static_cast<unsigned>((rows + kDqRows - 1) / kDqRows);
        if (c.d == 128) {
            cudaError_t e = ensure_smem_attr(reinterpret_cast<const void *>(dequant_mma_kernel<128>), DqSmem<128>::kBytes);
            if (e != cudaSuccess) return e;
            dequant_mma_kernel<128><<<blocks, 256, DqSmem<128>::kBytes, st>>>(c, pg, kc, vc, num_blocks, Hkv, slots, rows,
                                                                              k_out, v_out);
        } else {
            cudaError_t e = ensure_smem_attr(reinterpret_cast<const void *>(dequant_mma_kernel<256>), DqSmem<256>::kBytes);
            if (e != cudaSuccess) return e;
            dequant_mma_kernel<256><<<blocks, 256, DqSmem<256>::kBytes, st>>>(c, pg, kc, vc, num_blocks, Hkv, slots, rows,
                                                                              k_out, v_out);
        }
        return cudaGetLastError();
    }
    dim3 grid(static_cast<unsigned>(T), Hkv);
    if (c.d == 128)
        dequant_kernel<128><<<grid, 128, 0, st>>>(c, pg, kc, vc, num_blocks, Hkv, slots, k_out, v_out);
    else
        dequant_kernel<256><<<grid, 256, 0, st>>>(c, pg, kc, vc, num_blocks, Hkv, slots, k_out, v_out);
    return cudaGetLastError();
}

}  // namespace tq
