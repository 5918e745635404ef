// tq_decode_mma.cuh -- split-K paged decode on the tensor cores (mma.sync m16n8k16, fp16 in, fp32 accumulate).
//
// One CTA = (split, kv head, sequence); 4 warps, each owns 16-token tiles of
// every 128-token chunk (tokens 16 (warp + 4 i)), with its own online softmax;
// the warps merge at the end.
//
// Scores: S[t][h] = sum_j Khat[t][j] q[h][j] with the 16 tokens of a tile as
// the M dimension and the G <= 8 query heads as N.  Coordinates are permuted
// inside every 16-wide k-step so that the A-fragment elements of lane quad m
// are the four consecutive codes 16 s + 4 m + {0,1,2,3} of a token: pairs of
// codes index a shared-memory table of fp16 centroid pairs (high part and a
// low part scaled by 2^11, so the centroid score keeps ~22 bits:
// q.c = qh.ch + 2^-11 (ql.ch + qh.cl), three MMAs per k-step into two
// accumulators).  The QJL term sqrt(pi/2)/d * gamma * <S q_rot, 2 sigma - 1>
// uses a fourth MMA whose A operand is +-1 from the sign bits.
//
// Values: O^T[j][h] += sum_t V[t][j] P[t][h] with coordinates as M.  The score
// accumulator of a tile, converted to fp16 and transposed in registers
// (movmatrix), is exactly the B operand.  Rows of every 16-coordinate m-tile
// are permuted (row r <-> coordinate 16 mt + 2 r, row r + 8 <-> 16 mt + 2 r + 1)
// so that a lane's two codes per m-tile are adjacent and every m-tile lies in
// one value group; codes enter the MMA as exact fp16 integers, the group scale
// multiplies the B operand, and sum_t zero_t p_t is one small MMA per tile.
#pragma once

#include "tq_device.cuh"
#include "tq_internal.h"

namespace tq {
namespace dmma {

constexpr int kWarps = 4;
constexpr int kThreads = kWarps * 32;
constexpr int kTile = 16;                      // tokens per MMA tile (M of the score MMA)
constexpr int kTilesPerWarp = 2;               // tiles per warp per chunk
constexpr int kChunk = kWarps * kTile * kTilesPerWarp;  // tokens per chunk
constexpr float kLoScale = 2048.f;             // scale of the fp16 low parts
constexpr float kLog2e = 1.4426950408889634f;

__device__ __forceinline__ void mma16816(float (&c)[4], uint32_t a0, uint32_t a1, uint32_t a2, uint32_t a3,
                                         uint32_t b0, uint32_t b1)
{
    asm volatile("mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
                 "{%0,%1,%2,%3};"
                 : "+f"(c[0]), "+f"(c[1]), "+f"(c[2]), "+f"(c[3])
                 : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}

// Transpose of an 8x8 b16 matrix held in the accumulator-fragment layout
// (lane holds row lane / 4, columns 2 (lane % 4) + {0, 1}).
__device__ __forceinline__ uint32_t movmatrix_trans(uint32_t a)
{
    uint32_t d;
    asm volatile("movmatrix.sync.aligned.m8n8.trans.b16 %0, %1;" : "=r"(d) : "r"(a));
    return d;
}

__device__ __forceinline__ uint32_t pack_half2(float lo, float hi)
{
    const __half2 h = __floats2half2_rn(lo, hi);
    return *reinterpret_cast<const uint32_t *>(&h);
}

__device__ __forceinline__ uint32_t hmul2_u32(uint32_t a, uint32_t b)
{
    __half2 r = __hmul2(*reinterpret_cast<const __half2 *>(&a), *reinterpret_cast<const __half2 *>(&b));
    return *reinterpret_cast<uint32_t *>(&r);
}

// x holds (1024 + c0) | (1024 + c1) << 16 as fp16 bit patterns; returns the exact pair (c0, c1).
__device__ __forceinline__ uint32_t unbias_half2(uint32_t x)
{
    const uint32_t k = 0x64006400u;
    __half2 r = __hsub2(*reinterpret_cast<const __half2 *>(&x), *reinterpret_cast<const __half2 *>(&k));
    return *reinterpret_cast<uint32_t *>(&r);
}

__device__ __forceinline__ void cp_async16(void *smem, const void *gmem)
{
    const uint32_t s = static_cast<uint32_t>(__cvta_generic_to_shared(smem));
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(s), "l"(gmem) : "memory");
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }
template <int N>
__device__ __forceinline__ void cp_async_wait() { asm volatile("cp.async.wait_group %0;" ::"n"(N) : "memory"); }

// 2^x with the hardware approximation (relative error ~2^-22).
__device__ __forceinline__ float fast_exp2(float x)
{
    float y;
    asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}

// Dynamic shared memory layout of the tensor-core decode kernel.
template <int D, int KB>
struct DecSmem {
    static constexpr int kPairBits = 2 * KB;
    static constexpr int kPairEntries = 1 << kPairBits;
    // [entry][16 copies] (hi pair, lo pair): a 64-bit load takes two wavefronts of
    // 16 lanes, so 16 copies (lane & 15) keep every lookup conflict-free.
    static constexpr size_t kLut = sizeof(uint2) * kPairEntries * 16;
    static constexpr size_t kSignLut = sizeof(uint2) * 16;               // 4 sign bits -> two +-1 fp16 pairs
    static constexpr size_t kQfrag = sizeof(uint4) * (D / 16) * 32;      // [k-step][lane] (qh0, qh2, ql0, ql2)
    static constexpr size_t kSfrag = sizeof(uint2) * (D / 16) * 32;      // [k-step][lane] (qs0, qs2)
    static constexpr size_t kHeader = kLut + kSignLut + kQfrag + kSfrag + 64;  // + page-valid flags
    __host__ __device__ static size_t stage_bytes(const PageGeom &pg)
    {
        return static_cast<size_t>(kChunk / pg.P) * (pg.k_page + pg.v_page);
    }
    static size_t bytes(const PageGeom &pg)
    {
        const size_t st = 2 * stage_bytes(pg);
        const size_t red = sizeof(float) * kWarps * (D * 8 + 8 * 8 + 16);
        return kHeader + (st > red ? st : red);
    }
};

// The 4 KB-bit codes 16 s + 4 m .. 16 s + 4 m + 3 of a packed code row, in the low 4 KB bits.
template <int KB>
__device__ __forceinline__ uint32_t code_quad(const uint32_t *row, int s, int m)
{
    if constexpr (KB == 2) {
        return row[s] >> (8 * m);
    } else if constexpr (KB == 4) {
        return row[2 * s + (m >> 1)] >> (16 * (m & 1));
    } else {
        const int bit = 48 * s + 12 * m;
        return __funnelshift_r(row[bit >> 5], row[(bit >> 5) + 1], bit & 31);
    }
}

template <int D, int KB, int VB>
__global__ void __launch_bounds__(kThreads, D == 128 ? 4 : 2) decode_mma_kernel(const Codec C, const PageGeom PG, const DecodeArgs A)
{
    using SM = DecSmem<D, KB>;
    constexpr bool QJL = (KB <= 3);
    constexpr int KS = D / 16;                 // k-steps over coordinates
    constexpr int MT = D / 16;                 // m-tiles of output coordinates
    extern __shared__ __align__(16) unsigned char smem[];
    uint2 *lut = reinterpret_cast<uint2 *>(smem);
    uint2 *slut = reinterpret_cast<uint2 *>(smem + SM::kLut);
    uint4 *qfrag = reinterpret_cast<uint4 *>(smem + SM::kLut + SM::kSignLut);
    uint2 *sfrag = reinterpret_cast<uint2 *>(smem + SM::kLut + SM::kSignLut + SM::kQfrag);
    int *page_ok = reinterpret_cast<int *>(smem + SM::kLut + SM::kSignLut + SM::kQfrag + SM::kSfrag);  // [2][8]
    unsigned char *stages = smem + SM::kHeader;

    const int split = blockIdx.x, kvh = blockIdx.y, b = blockIdx.z;
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int quad = lane & 3, row = lane >> 2;
    const int P = PG.P;
    const int G = A.Hq / A.Hkv;
    const int ng = D / C.group;
    const size_t stage_bytes = SM::stage_bytes(PG);
    const int ppc = kChunk / P;

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
    if (pg0 >= pg1) {
        if (tid < G) {
            ml_out[2 * tid] = -INFINITY;
            ml_out[2 * tid + 1] = 0.f;
        }
        return;
    }

    // ---- tables: fp16 centroid pairs (16 copies) and +-1 sign pairs ----
    for (int e = tid; e < SM::kPairEntries * 16; e += kThreads) {
        const int ent = e >> 4;
        const int c0 = ent & ((1 << KB) - 1), c1 = ent >> KB;
        const float x0 = C.centroids[c0], x1 = C.centroids[c1];
        const float h0 = __half2float(__float2half_rn(x0)), h1 = __half2float(__float2half_rn(x1));
        lut[e] = make_uint2(pack_half2(h0, h1), pack_half2((x0 - h0) * kLoScale, (x1 - h1) * kLoScale));
    }
    if (tid < 16) {
        auto pm = [](int bit) { return bit ? 1.f : -1.f; };
        slut[tid] = make_uint2(pack_half2(pm(tid & 1), pm(tid & 2)), pack_half2(pm(tid & 4), pm(tid & 8)));
    }

    // ---- query fragments (B operand of the score MMA, head = lane / 4), permuted
    // coordinates; identical for the four warps, so warp 0 writes them ----
    if (warp == 0) {
        const bool hv = row < G;
        const float *qr = A.ws.qrot + (head0 + (hv ? row : 0)) * D;
        const float *qs = A.ws.qs + (head0 + (hv ? row : 0)) * D;
#pragma unroll 4
        for (int s = 0; s < KS; ++s) {
            const int j = 16 * s + 4 * quad;
            uint4 f = make_uint4(0u, 0u, 0u, 0u);
            uint2 g = make_uint2(0u, 0u);
            if (hv) {
                const float4 v = *reinterpret_cast<const float4 *>(qr + j);
                const float hx = __half2float(__float2half_rn(v.x)), hy = __half2float(__float2half_rn(v.y));
                const float hz = __half2float(__float2half_rn(v.z)), hw = __half2float(__float2half_rn(v.w));
                f = make_uint4(pack_half2(hx, hy), pack_half2(hz, hw), pack_half2((v.x - hx) * kLoScale, (v.y - hy) * kLoScale),
                               pack_half2((v.z - hz) * kLoScale, (v.w - hw) * kLoScale));
                if (QJL) {
                    const float4 w = *reinterpret_cast<const float4 *>(qs + j);
                    g = make_uint2(pack_half2(w.x, w.y), pack_half2(w.z, w.w));
                }
            }
            qfrag[s * 32 + lane] = f;
            sfrag[s * 32 + lane] = g;
        }
    }

    // ---- accumulators: O^T rows (coordinates, permuted) x heads 2 quad, 2 quad + 1 ----
    float o[MT][4];
#pragma unroll
    for (int mt = 0; mt < MT; ++mt) o[mt][0] = o[mt][1] = o[mt][2] = o[mt][3] = 0.f;
    float zt[4] = {0.f, 0.f, 0.f, 0.f};       // sum_t zero[t][g] p[t][h]: rows = groups
    float m_run[2] = {-INFINITY, -INFINITY};  // heads 2 quad + e
    float l_run[2] = {0.f, 0.f};

    const float fac_c = A.sm_scale * rsqrtf(static_cast<float>(D)) * kLog2e;
    const float fac_s = A.sm_scale * (1.2533141373155003f / static_cast<float>(D)) * kLog2e;
    const uint32_t lut_lane = static_cast<uint32_t>(__cvta_generic_to_shared(lut)) + 8u * (lane & 15);
    const uint32_t slut_base = static_cast<uint32_t>(__cvta_generic_to_shared(slut));
    const uint2 *lutl = lut + (lane & 15);
    (void)lut_lane;
    (void)slut_base;

    // ---- stage loader --------------------------------------------------------
    auto issue = [&](int chunk_page, int st) {
        unsigned char *kst = stages + st * stage_bytes;
        unsigned char *vst = kst + static_cast<size_t>(ppc) * PG.k_page;
        const int np = min(ppc, pg1 - chunk_page);
        for (int q = 0; q < ppc; ++q) {
            int ok = 0;
            if (q < np) {
                const int blk = A.block_table[static_cast<int64_t>(b) * A.max_blocks + chunk_page + q];
                ok = (blk >= 0 && blk < A.num_blocks);
                if (ok) {
                    const size_t rec = static_cast<size_t>(blk) * A.Hkv + kvh;
                    const unsigned char *ks = A.k_cache + rec * PG.k_page;
                    const unsigned char *vs = A.v_cache + rec * PG.v_page;
                    for (int e = tid; e < PG.k_page / 16; e += kThreads)
                        cp_async16(kst + q * PG.k_page + 16 * e, ks + 16 * e);
                    for (int e = tid; e < PG.v_page / 16; e += kThreads)
                        cp_async16(vst + q * PG.v_page + 16 * e, vs + 16 * e);
                } else if (tid == 0) {
                    atomicOr(C.status, TQ_DEVERR_BLOCK_RANGE);
                }
            }
            if (tid == 0) page_ok[st * 8 + q] = ok;
        }
        cp_async_commit();
    };

    const int nchunks = (pg1 - pg0 + ppc - 1) / ppc;
    issue(pg0, 0);
    for (int c = 0; c < nchunks; ++c) {
        const int st = c & 1;
        const int cpage = pg0 + c * ppc;
        if (c + 1 < nchunks) {
            issue(cpage + ppc, st ^ 1);
            cp_async_wait<1>();
        } else {
            cp_async_wait<0>();
        }
        __syncthreads();

#pragma unroll 1
        for (int ti = 0; ti < kTilesPerWarp; ++ti) {
        const int tok0 = kTile * (warp + kWarps * ti);
        const int q = tok0 / P;                  // page inside the chunk
        const int o0 = tok0 - q * P;             // first offset inside the page
        const int pos0 = (cpage + q) * P + o0;   // sequence position of tile token 0
        const bool tile_live = (q < min(ppc, pg1 - cpage)) && page_ok[st * 8 + q] && (pos0 < L);
        if (tile_live) {
            const unsigned char *kr = stages + st * stage_bytes + static_cast<size_t>(q) * PG.k_page;
            const unsigned char *vr = stages + st * stage_bytes + static_cast<size_t>(ppc) * PG.k_page +
                                      static_cast<size_t>(q) * PG.v_page;
            // ---- scores S[token][head]: this lane feeds tokens row, row + 8 ----
            float sc[4] = {0.f, 0.f, 0.f, 0.f}, sl[4] = {0.f, 0.f, 0.f, 0.f}, ss[4] = {0.f, 0.f, 0.f, 0.f};
            const uint32_t *krow0 = reinterpret_cast<const uint32_t *>(kr + (o0 + row) * C.k_code_bytes);
            const uint32_t *krow1 = reinterpret_cast<const uint32_t *>(kr + (o0 + row + 8) * C.k_code_bytes);
            const uint32_t *srow0 = reinterpret_cast<const uint32_t *>(kr + PG.k_sign_off + (o0 + row) * C.k_sign_bytes);
            const uint32_t *srow1 = reinterpret_cast<const uint32_t *>(kr + PG.k_sign_off + (o0 + row + 8) * C.k_sign_bytes);
            constexpr uint32_t PM = (1u << (2 * KB)) - 1u;
#pragma unroll
            for (int s = 0; s < KS; ++s) {
                const uint32_t f0 = code_quad<KB>(krow0, s, quad);
                const uint32_t f1 = code_quad<KB>(krow1, s, quad);
                const uint2 e00 = lutl[(f0 & PM) << 4], e01 = lutl[((f0 >> (2 * KB)) & PM) << 4];
                const uint2 e10 = lutl[(f1 & PM) << 4], e11 = lutl[((f1 >> (2 * KB)) & PM) << 4];
                const uint4 qf = qfrag[s * 32 + lane];
                mma16816(sc, e00.x, e10.x, e01.x, e11.x, qf.x, qf.y);
                mma16816(sl, e00.x, e10.x, e01.x, e11.x, qf.z, qf.w);
                mma16816(sl, e00.y, e10.y, e01.y, e11.y, qf.x, qf.y);
                if (QJL) {
                    const int sh = 16 * (s & 1) + 4 * quad;
                    const uint2 g0 = slut[(srow0[s >> 1] >> sh) & 15u];
                    const uint2 g1 = slut[(srow1[s >> 1] >> sh) & 15u];
                    const uint2 sf = sfrag[s * 32 + lane];
                    mma16816(ss, g0.x, g1.x, g0.y, g1.y, sf.x, sf.y);
                }
            }
            // ---- scale and mask: x[hh][e] = token row + 8 hh, head 2 quad + e ----
            const uint16_t *nrow = reinterpret_cast<const uint16_t *>(kr + PG.k_norm_off) + o0 + row;
            const float nrm[2] = {bf16_to_float(nrow[0]), bf16_to_float(nrow[8])};
            float gam[2] = {0.f, 0.f};
            if (QJL) {
                const uint16_t *grow = reinterpret_cast<const uint16_t *>(kr + PG.k_gamma_off) + o0 + row;
                gam[0] = bf16_to_float(grow[0]);
                gam[1] = bf16_to_float(grow[8]);
            }
            float x[2][2];
#pragma unroll
            for (int hh = 0; hh < 2; ++hh)
#pragma unroll
                for (int e = 0; e < 2; ++e) {
                    const int i = 2 * hh + e;
                    float v = nrm[hh] * fac_c * fmaf(sl[i], 1.f / kLoScale, sc[i]);
                    if (QJL) v = fmaf(nrm[hh] * fac_s * gam[hh], ss[i], v);
                    const bool valid = (pos0 + row + 8 * hh) < L;
                    x[hh][e] = (2 * quad + e < G) ? (valid ? v : -INFINITY) : 0.f;
                }
            // ---- online softmax (base 2) per head 2 quad + e over the tile's 16 tokens ----
            float p[2][2], alpha[2];
#pragma unroll
            for (int e = 0; e < 2; ++e) {
                float mt = fmaxf(x[0][e], x[1][e]);
                mt = fmaxf(mt, __shfl_xor_sync(0xffffffffu, mt, 4));
                mt = fmaxf(mt, __shfl_xor_sync(0xffffffffu, mt, 8));
                mt = fmaxf(mt, __shfl_xor_sync(0xffffffffu, mt, 16));
                const float m_new = fmaxf(m_run[e], mt);
                alpha[e] = 1.f;
                p[0][e] = p[1][e] = 0.f;
                if (m_new != -INFINITY) {
                    alpha[e] = fast_exp2(m_run[e] - m_new);
                    p[0][e] = fast_exp2(x[0][e] - m_new);
                    p[1][e] = fast_exp2(x[1][e] - m_new);
                }
                float ps = p[0][e] + p[1][e];
                ps += __shfl_xor_sync(0xffffffffu, ps, 4);
                ps += __shfl_xor_sync(0xffffffffu, ps, 8);
                ps += __shfl_xor_sync(0xffffffffu, ps, 16);
                l_run[e] = l_run[e] * alpha[e] + ps;
                m_run[e] = m_new;
            }
            // O^T columns of this lane are exactly its heads 2 quad, 2 quad + 1
            if (alpha[0] != 1.f || alpha[1] != 1.f) {
#pragma unroll
                for (int mt = 0; mt < MT; ++mt) {
                    o[mt][0] *= alpha[0]; o[mt][1] *= alpha[1]; o[mt][2] *= alpha[0]; o[mt][3] *= alpha[1];
                }
                zt[0] *= alpha[0]; zt[1] *= alpha[1]; zt[2] *= alpha[0]; zt[3] *= alpha[1];
            }
            // ---- P^T as the B operand: tokens 2 quad + {0,1} (+8), head `row` ----
            const uint32_t b0 = movmatrix_trans(pack_half2(p[0][0], p[0][1]));
            const uint32_t b1 = movmatrix_trans(pack_half2(p[1][0], p[1][1]));
            // value metadata of tokens 2 quad, 2 quad + 1, 2 quad + 8, 2 quad + 9 (zero for
            // masked tokens, whose never-written bytes may hold any fp16 pattern)
            const int tq[4] = {2 * quad, 2 * quad + 1, 2 * quad + 8, 2 * quad + 9};
            const unsigned char *meta = vr + PG.v_meta_off + o0 * C.v_meta_bytes;
            bool tv[4];
#pragma unroll
            for (int i = 0; i < 4; ++i) tv[i] = (pos0 + tq[i]) < L;
            auto meta_word = [&](int i, int g) -> uint32_t {
                return tv[i] ? *reinterpret_cast<const uint32_t *>(meta + tq[i] * C.v_meta_bytes + 4 * g) : 0u;
            };
            // zero term: A rows = groups (`row` < ng), columns = tokens
            {
                uint32_t za0 = 0u, za2 = 0u;
                if (row < ng) {
                    za0 = __byte_perm(meta_word(0, row), meta_word(1, row), 0x7632);
                    za2 = __byte_perm(meta_word(2, row), meta_word(3, row), 0x7632);
                }
                mma16816(zt, za0, 0u, za2, 0u, b0, b1);
            }
            // ---- P.V over coordinate m-tiles: row r <-> 16 mt + 2 r, row r + 8 <-> 16 mt + 2 r + 1 ----
            const uint32_t *vrow[4];
#pragma unroll
            for (int i = 0; i < 4; ++i) vrow[i] = reinterpret_cast<const uint32_t *>(vr + (o0 + tq[i]) * C.v_code_bytes);
            constexpr uint32_t VM = ((1u << VB) - 1u) * 0x00010001u;
            const uint32_t bias = 0x64006400u;
            const int mt_per_group = C.group >> 4;
            uint32_t bs0 = 0u, bs1 = 0u;
#pragma unroll
            for (int mt = 0; mt < MT; ++mt) {
                if (mt % mt_per_group == 0) {  // a new value group: scale the B operand
                    const int g = mt / mt_per_group;
                    bs0 = hmul2_u32(b0, __byte_perm(meta_word(0, g), meta_word(1, g), 0x5410));
                    bs1 = hmul2_u32(b1, __byte_perm(meta_word(2, g), meta_word(3, g), 0x5410));
                }
                uint32_t xa, xb;  // codes of coordinates 16 mt + 2 row (+1): tokens (0, 1) | (2, 3)
                if constexpr (VB == 2) {
                    const uint32_t sel = static_cast<uint32_t>(row >> 1) | (static_cast<uint32_t>(4 + (row >> 1)) << 8);
                    const int sh = 4 * (row & 1);
                    xa = __byte_perm(vrow[0][mt], vrow[1][mt], sel) >> sh;
                    xb = __byte_perm(vrow[2][mt], vrow[3][mt], sel) >> sh;
                } else if constexpr (VB == 4) {
                    const uint32_t sel = static_cast<uint32_t>(row & 3) | (static_cast<uint32_t>(4 + (row & 3)) << 8);
                    const int w = 2 * mt + (row >> 2);
                    xa = __byte_perm(vrow[0][w], vrow[1][w], sel);
                    xb = __byte_perm(vrow[2][w], vrow[3][w], sel);
                } else {
                    const int bit = 48 * mt + 6 * row;
                    const int w = bit >> 5, sh = bit & 31;
                    xa = __byte_perm(__funnelshift_r(vrow[0][w], vrow[0][w + 1], sh),
                                     __funnelshift_r(vrow[1][w], vrow[1][w + 1], sh), 0x5410);
                    xb = __byte_perm(__funnelshift_r(vrow[2][w], vrow[2][w + 1], sh),
                                     __funnelshift_r(vrow[3][w], vrow[3][w + 1], sh), 0x5410);
                }
                const uint32_t a0 = unbias_half2((xa & VM) | bias);
                const uint32_t a1 = unbias_half2(((xa >> VB) & VM) | bias);
                const uint32_t a2 = unbias_half2((xb & VM) | bias);
                const uint32_t a3 = unbias_half2(((xb >> VB) & VM) | bias);
                mma16816(o[mt], a0, a1, a2, a3, bs0, bs1);
            }
        }
        }  // tiles
        __syncthreads();  // the next issue() overwrites this stage
    }

    // ---- merge the four warps ---------------------------------------------------
    float *red = reinterpret_cast<float *>(stages);
    float *r_m = red;                       // [warps][8]
    float *r_l = r_m + kWarps * 8;          // [warps][8]
    float *r_o = r_l + kWarps * 8;          // [warps][D][8]
    float *r_z = r_o + kWarps * D * 8;      // [warps][8 groups][8 heads]
    if (row == 0) {
        r_m[warp * 8 + 2 * quad] = m_run[0];
        r_m[warp * 8 + 2 * quad + 1] = m_run[1];
        r_l[warp * 8 + 2 * quad] = l_run[0];
        r_l[warp * 8 + 2 * quad + 1] = l_run[1];
    }
#pragma unroll
    for (int mt = 0; mt < MT; ++mt) {
        const int j = 16 * mt + 2 * row;
        r_o[(warp * D + j) * 8 + 2 * quad] = o[mt][0];
        r_o[(warp * D + j) * 8 + 2 * quad + 1] = o[mt][1];
        r_o[(warp * D + j + 1) * 8 + 2 * quad] = o[mt][2];
        r_o[(warp * D + j + 1) * 8 + 2 * quad + 1] = o[mt][3];
    }
    r_z[(warp * 8 + row) * 8 + 2 * quad] = zt[0];
    r_z[(warp * 8 + row) * 8 + 2 * quad + 1] = zt[1];
    __syncthreads();
    for (int e = tid; e < G * D; e += kThreads) {
        const int h = e / D, j = e - h * D;
        float M = -INFINITY;
#pragma unroll
        for (int w = 0; w < kWarps; ++w) M = fmaxf(M, r_m[w * 8 + h]);
        float acc = 0.f, l = 0.f;
        if (M != -INFINITY) {
#pragma unroll
            for (int w = 0; w < kWarps; ++w) {
                const float f = fast_exp2(r_m[w * 8 + h] - M);
                acc = fmaf(f, r_o[(w * D + j) * 8 + h] + r_z[(w * 8 + j / C.group) * 8 + h], acc);
                l = fmaf(f, r_l[w * 8 + h], l);
            }
        }
        acc_out[static_cast<size_t>(h) * D + j] = acc;
        if (j == 0) {
            ml_out[2 * h] = M;
            ml_out[2 * h + 1] = l;
        }
    }
}

}  // namespace dmma
}  // namespace tq
