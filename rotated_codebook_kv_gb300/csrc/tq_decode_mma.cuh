// tq_decode_mma.cuh -- split-K paged decode on the tensor cores (mma.sync m16n8k16, fp16 in, fp32 accumulate).
//
// One CTA = (split, kv head, sequence); 4 warps, each owns 16 tokens of every
// 64-token chunk, with its own online softmax; the warps merge at the end.
//
// Scores are computed transposed, S^T[h][t] = sum_j q[h][j] Khat[t][j] with
// the G query heads as the M dimension (padded to 16) and tokens as N, so the
// fp32 score accumulators of two 8-token n-tiles are, after exp and fp16
// conversion, exactly the B operand of O^T[j][h] = sum_t V[t][j] P[h][t]
// (coordinates as M, heads as N = 8, tokens as K) -- no data exchange between
// lanes.  Tokens are ordered inside a tile so that lane quad m owns tokens
// 4m..4m+3 in the P.V step.
//
// Coordinates are permuted inside every 16-wide k-step so that the four
// B-fragment elements of lane quad m are the four consecutive codes
// 16s + 4m + {0,1,2,3}: pairs of codes index a shared-memory table of fp16
// centroid pairs (replicated so that lookups never conflict).
// Queries and centroids are each split into an fp16 high part and a low part
// scaled by 2^11, so the centroid score keeps ~22 bits: q.c = qh.ch +
// 2^-11 (ql.ch + qh.cl), three MMAs per k-step into two accumulators.
// The QJL term sqrt(pi/2)/d * gamma * <S q_rot, 2 sigma - 1> uses a second
// accumulator with a +-1 operand built the same way from the sign bits.
// Values: O^T += V^T (P^T scaled per group by the token's fp16 scale), plus a
// small MMA with the zero points for sum_t zero_t * p_t.
#pragma once

#include "tq_device.cuh"
#include "tq_internal.h"

namespace tq {
namespace dmma {

constexpr int kWarps = 4;
constexpr int kThreads = kWarps * 32;
constexpr int kTile = 16;                      // tokens per MMA tile
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

// Two small unsigned codes as an exact fp16 pair: (1024 + c) - 1024.
__device__ __forceinline__ uint32_t codes_to_half2(uint32_t c_lo, uint32_t c_hi)
{
    const uint32_t x = (c_lo | (c_hi << 16)) | 0x64006400u;
    __half2 r = __hsub2(*reinterpret_cast<const __half2 *>(&x), __float2half2_rn(1024.f));
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

// 64-bit window of two consecutive 32-bit words shifted right by sh (0..63).
__device__ __forceinline__ uint32_t window(uint32_t w0, uint32_t w1, int sh)
{
    const uint64_t v = (static_cast<uint64_t>(w1) << 32) | w0;
    return static_cast<uint32_t>(v >> sh);
}

// Dynamic shared memory layout of the tensor-core decode kernel.
template <int D, int KB>
struct DecSmem {
    static constexpr int kPairBits = 2 * KB;
    static constexpr int kPairEntries = 1 << kPairBits;
    // [entry][16 copies] (hi pair, lo pair): a 64-bit load takes two wavefronts of
    // 16 lanes, so 16 copies (lane & 15) keep every lookup conflict-free.
    static constexpr size_t kLut = sizeof(uint2) * kPairEntries * 16;
    static constexpr size_t kSignLut = sizeof(uint32_t) * 4 * 32;
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

template <int D, int KB, int VB>
__global__ void __launch_bounds__(kThreads, D == 128 ? 4 : 2) decode_mma_kernel(const Codec C, const PageGeom PG, const DecodeArgs A)
{
    using SM = DecSmem<D, KB>;
    constexpr bool QJL = (KB <= 3);
    constexpr int KS = D / 16;                 // k-steps over coordinates
    constexpr int MT = D / 16;                 // m-tiles of output coordinates
    constexpr int NWK = D * KB / 32;           // words per key code row
    constexpr int NWS = D / 32;                // words per sign row
    extern __shared__ __align__(16) unsigned char smem[];
    uint2 *lut = reinterpret_cast<uint2 *>(smem);
    uint32_t *slut = reinterpret_cast<uint32_t *>(smem + SM::kLut);
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

    // ---- tables: fp16 centroid pairs and +-1 sign pairs, one copy per lane ----
    for (int e = tid; e < SM::kPairEntries * 16; e += kThreads) {
        const int ent = e >> 4;
        const int c0 = ent & ((1 << KB) - 1), c1 = ent >> KB;
        const float x0 = C.centroids[c0], x1 = C.centroids[c1];
        const float h0 = __half2float(__float2half_rn(x0)), h1 = __half2float(__float2half_rn(x1));
        lut[e] = make_uint2(pack_half2(h0, h1), pack_half2((x0 - h0) * kLoScale, (x1 - h1) * kLoScale));
    }
    for (int e = tid; e < 4 * 32; e += kThreads) {
        const int ent = e >> 5;
        slut[e] = pack_half2((ent & 1) ? 1.f : -1.f, (ent & 2) ? 1.f : -1.f);
    }

    // ---- query fragments (A operand of the score MMA), permuted coordinates;
    // identical for the four warps, so warp 0 writes them to shared memory ----
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

    // ---- accumulators ---------------------------------------------------------
    float o[MT][4];
#pragma unroll
    for (int mt = 0; mt < MT; ++mt) o[mt][0] = o[mt][1] = o[mt][2] = o[mt][3] = 0.f;
    float zt[4] = {0.f, 0.f, 0.f, 0.f};  // sum_t zero[t][g] p[h][t], rows = groups
    float m_run = -INFINITY, l_run = 0.f;  // head `row`, replicated across the quad

    const float fac_c = A.sm_scale * rsqrtf(static_cast<float>(D)) * kLog2e;
    const float fac_s = A.sm_scale * (1.2533141373155003f / static_cast<float>(D)) * kLog2e;

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

        // ---- this warp's tiles: chunk tokens [16 (warp + 4 i), +16) ----
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
            // ---- scores: two n-tiles of 8 tokens; this lane feeds token tau ----
            float sc[2][4], sl[2][4], ss[2][4];
#pragma unroll
            for (int nt = 0; nt < 2; ++nt) {
                sc[nt][0] = sc[nt][1] = sc[nt][2] = sc[nt][3] = 0.f;
                sl[nt][0] = sl[nt][1] = sl[nt][2] = sl[nt][3] = 0.f;
                ss[nt][0] = ss[nt][1] = ss[nt][2] = ss[nt][3] = 0.f;
                const int tau = 2 * row - (row & 1) + 2 * nt;  // n-tile nt column `row`
                const uint32_t *cw = reinterpret_cast<const uint32_t *>(kr + (o0 + tau) * C.k_code_bytes);
                uint32_t kw[NWK + 1];
#pragma unroll
                for (int w = 0; w < NWK; w += 4) {
                    const uint4 u = *reinterpret_cast<const uint4 *>(cw + w);
                    kw[w] = u.x; kw[w + 1] = u.y; kw[w + 2] = u.z; kw[w + 3] = u.w;
                }
                kw[NWK] = 0u;
                uint32_t sw[NWS];
                if (QJL) {
                    const uint32_t *sp = reinterpret_cast<const uint32_t *>(kr + PG.k_sign_off + (o0 + tau) * C.k_sign_bytes);
#pragma unroll
                    for (int w = 0; w < NWS; w += 4) {
                        const uint4 u = *reinterpret_cast<const uint4 *>(sp + w);
                        sw[w] = u.x; sw[w + 1] = u.y; sw[w + 2] = u.z; sw[w + 3] = u.w;
                    }
                }
#pragma unroll
                for (int s = 0; s < KS; ++s) {
                    // four codes 16s + 4 quad + {0..3}: bit offset KB * (16 s + 4 quad)
                    const int base = KB * 16 * s;             // compile-time
                    const int w0 = base >> 5;                 // compile-time word
                    const int sh = (base & 31) + KB * 4 * quad;  // 0..(31 + 12)
                    const uint32_t bits = window(kw[w0], kw[w0 + 1], sh);
                    const uint32_t p0 = bits & ((1u << (2 * KB)) - 1u);
                    const uint32_t p1 = (bits >> (2 * KB)) & ((1u << (2 * KB)) - 1u);
                    const uint2 b0 = lut[(p0 << 4) + (lane & 15)];
                    const uint2 b1 = lut[(p1 << 4) + (lane & 15)];
                    const uint4 qf = qfrag[s * 32 + lane];
                    mma16816(sc[nt], qf.x, 0u, qf.y, 0u, b0.x, b1.x);
                    mma16816(sl[nt], qf.z, 0u, qf.w, 0u, b0.x, b1.x);
                    mma16816(sl[nt], qf.x, 0u, qf.y, 0u, b0.y, b1.y);
                    if (QJL) {
                        const uint32_t sb = (sw[s >> 1] >> (16 * (s & 1) + 4 * quad)) & 0xFu;
                        const uint32_t c0 = slut[((sb & 3u) << 5) + lane];
                        const uint32_t c1 = slut[((sb >> 2) << 5) + lane];
                        const uint2 sf = sfrag[s * 32 + lane];
                        mma16816(ss[nt], sf.x, 0u, sf.y, 0u, c0, c1);
                    }
                }
            }
            // ---- scale: lane holds head `row`, tokens 4 quad + {0,1,2,3} ----
            const int t0 = 4 * quad;
            const uint2 nb = *reinterpret_cast<const uint2 *>(kr + PG.k_norm_off + 2 * (o0 + t0));
            float nrm[4] = {bf16_to_float(nb.x & 0xffffu), bf16_to_float(nb.x >> 16), bf16_to_float(nb.y & 0xffffu),
                            bf16_to_float(nb.y >> 16)};
            float gam[4] = {0.f, 0.f, 0.f, 0.f};
            if (QJL) {
                const uint2 gb = *reinterpret_cast<const uint2 *>(kr + PG.k_gamma_off + 2 * (o0 + t0));
                gam[0] = bf16_to_float(gb.x & 0xffffu); gam[1] = bf16_to_float(gb.x >> 16);
                gam[2] = bf16_to_float(gb.y & 0xffffu); gam[3] = bf16_to_float(gb.y >> 16);
            }
            float x[4];
#pragma unroll
            for (int i = 0; i < 4; ++i) {
                const int nt = i >> 1, e = i & 1;
                float v = nrm[i] * fac_c * fmaf(sl[nt][e], 1.f / kLoScale, sc[nt][e]);
                if (QJL) v = fmaf(nrm[i] * fac_s * gam[i], ss[nt][e], v);
                const bool valid = (pos0 + t0 + i) < L;
                x[i] = (row < G) ? (valid ? v : -INFINITY) : 0.f;
            }
            // ---- online softmax (base 2) ----
            float mt = fmaxf(fmaxf(x[0], x[1]), fmaxf(x[2], x[3]));
            mt = fmaxf(mt, __shfl_xor_sync(0xffffffffu, mt, 1));
            mt = fmaxf(mt, __shfl_xor_sync(0xffffffffu, mt, 2));
            const float m_new = fmaxf(m_run, mt);
            float alpha = 1.f, p[4] = {0.f, 0.f, 0.f, 0.f};
            if (m_new != -INFINITY) {
                alpha = fast_exp2(m_run - m_new);
#pragma unroll
                for (int i = 0; i < 4; ++i) p[i] = fast_exp2(x[i] - m_new);
            }
            float ps = (p[0] + p[1]) + (p[2] + p[3]);
            ps += __shfl_xor_sync(0xffffffffu, ps, 1);
            ps += __shfl_xor_sync(0xffffffffu, ps, 2);
            l_run = l_run * alpha + ps;
            m_run = m_new;
            // rescale O^T columns (heads 2 quad, 2 quad + 1) when any running max moved
            if (__any_sync(0xffffffffu, alpha != 1.f)) {
                const float a_lo = __shfl_sync(0xffffffffu, alpha, 8 * quad);
                const float a_hi = __shfl_sync(0xffffffffu, alpha, 8 * quad + 4);
#pragma unroll
                for (int m2 = 0; m2 < MT; ++m2) {
                    o[m2][0] *= a_lo; o[m2][1] *= a_hi; o[m2][2] *= a_lo; o[m2][3] *= a_hi;
                }
                zt[0] *= a_lo; zt[1] *= a_hi; zt[2] *= a_lo; zt[3] *= a_hi;
            }
            // ---- P^T fragments (tokens 4 quad + {0,1} | {2,3}, head `row`) ----
            const uint32_t pb0 = pack_half2(p[0], p[1]);
            const uint32_t pb1 = pack_half2(p[2], p[3]);
            // ---- per-token value metadata of tokens t0..t0+3 (zero for masked tokens,
            // whose never-written bytes may hold any fp16 pattern) ----
            const unsigned char *meta = vr + PG.v_meta_off + (o0 + t0) * C.v_meta_bytes;
            const int nval = min(4, max(0, L - (pos0 + t0)));
            auto meta_word = [&](int t, int g) -> uint32_t {
                return t < nval ? *reinterpret_cast<const uint32_t *>(meta + t * C.v_meta_bytes + 4 * g) : 0u;
            };
            // zero-term: rows = groups (`row` < ng), tokens t0..t0+3
            uint32_t za0 = 0u, za2 = 0u;
            if (row < ng) {
                const uint32_t m0 = meta_word(0, row), m1 = meta_word(1, row);
                const uint32_t m2 = meta_word(2, row), m3 = meta_word(3, row);
                za0 = __byte_perm(m0, m1, 0x7632);
                za2 = __byte_perm(m2, m3, 0x7632);
            }
            mma16816(zt, za0, 0u, za2, 0u, pb0, pb1);
            // ---- P.V over coordinate m-tiles ----
            const unsigned char *vc0 = vr + (o0 + t0) * C.v_code_bytes;
            int g_cur = -1;
            uint32_t bs0 = 0u, bs1 = 0u;
#pragma unroll
            for (int m2 = 0; m2 < MT; ++m2) {
                const int g = (16 * m2) / C.group;
                if (g != g_cur) {  // group changes every group/16 m-tiles
                    g_cur = g;
                    const uint32_t s0 = meta_word(0, g), s1 = meta_word(1, g);
                    const uint32_t s2 = meta_word(2, g), s3 = meta_word(3, g);
                    bs0 = hmul2_u32(pb0, __byte_perm(s0, s1, 0x5410));
                    bs1 = hmul2_u32(pb1, __byte_perm(s2, s3, 0x5410));
                }
                // codes of coordinates j0 = 16 m2 + row and j0 + 8 for tokens t0..t0+3
                const int j0 = 16 * m2 + row;
                uint32_t c[4][2];
#pragma unroll
                for (int t = 0; t < 4; ++t) {
                    const unsigned char *cb = vc0 + t * C.v_code_bytes;
                    if (VB == 2) {
                        const uint32_t w = *reinterpret_cast<const uint32_t *>(cb + 4 * m2);
                        c[t][0] = (w >> (2 * row)) & 3u;
                        c[t][1] = (w >> (16 + 2 * row)) & 3u;
                    } else if (VB == 4) {
                        const uint2 w = *reinterpret_cast<const uint2 *>(cb + 8 * m2);
                        c[t][0] = (w.x >> (4 * row)) & 15u;
                        c[t][1] = (w.y >> (4 * row)) & 15u;
                    } else {  // 3-bit: 64-bit window starting at word floor(48 m2 / 32)
                        const int wb = (48 * m2) >> 5;
                        const uint32_t *cw = reinterpret_cast<const uint32_t *>(cb);
                        const uint32_t lo = cw[wb], hi = cw[wb + 1];
                        const int sh0 = 48 * m2 - 32 * wb + 3 * row;
                        c[t][0] = window(lo, hi, sh0) & 7u;
                        c[t][1] = window(lo, hi, sh0 + 24) & 7u;
                    }
                }
                (void)j0;
                const uint32_t a0 = codes_to_half2(c[0][0], c[1][0]);
                const uint32_t a1 = codes_to_half2(c[0][1], c[1][1]);
                const uint32_t a2 = codes_to_half2(c[2][0], c[3][0]);
                const uint32_t a3 = codes_to_half2(c[2][1], c[3][1]);
                mma16816(o[m2], a0, a1, a2, a3, bs0, bs1);
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
    if (quad == 0) {
        r_m[warp * 8 + row] = m_run;
        r_l[warp * 8 + row] = l_run;
    }
#pragma unroll
    for (int m2 = 0; m2 < MT; ++m2) {
        const int j = 16 * m2 + row;
        r_o[(warp * D + j) * 8 + 2 * quad] = o[m2][0];
        r_o[(warp * D + j) * 8 + 2 * quad + 1] = o[m2][1];
        r_o[(warp * D + j + 8) * 8 + 2 * quad] = o[m2][2];
        r_o[(warp * D + j + 8) * 8 + 2 * quad + 1] = o[m2][3];
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
