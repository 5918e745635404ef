// tq_decode_mma.cuh -- split-K paged decode on the tensor cores (mma.sync m16n8k16, fp16 in, fp32 accumulate).
//
// One CTA = (split, kv head, sequence); 4 warps.  Warp w takes the 32-token
// rounds w, w + 4, w + 8, ... of the split (two 16-token tiles each), fetches
// their pages itself and keeps its own online softmax; the warps merge at the end.
//
// Scores: S[t][h] = sum_j Khat[t][j] q[h][j] with tokens as the M dimension and
// the G <= 8 query heads as N.  Coordinates are permuted inside every 16-wide
// k-step so that the A-fragment elements of lane quad m are the four
// consecutive codes 16 s + 4 m + {0,1,2,3} of a token: pairs of codes index a
// shared-memory table of fp16 centroid pairs (a high part and a low part scaled
// by 2^11, so the centroid score keeps ~22 bits: q.c = qh.ch + 2^-11 (ql.ch +
// qh.cl)).  M rows r and r + 8 hold the high and the low parts of the same
// token, so one 64-bit table load fills two adjacent A registers; MMAs against
// qh and ql give qh.ch, qh.cl and ql.ch for 8 tokens.  The QJL term
// sqrt(pi/2)/d * gamma * <S q_rot, 2 sigma - 1> is one more MMA whose A
// operand is +-1 from the sign bits (rows = 16 tokens).
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

// Dynamic shared memory layout of the tensor-core decode kernel.  VM: values
// coded by the rotation and a Lloyd-Max codebook, whose fp16 centroid pairs
// (indexed by the codes of two tokens) follow the key tables in 8 copies.
template <int D, int KB, int VB = 2, bool VM = false>
struct DecSmem {
    static constexpr int kPairBits = 2 * KB;
    static constexpr int kPairEntries = 1 << kPairBits;
    // [entry][copies] (hi pair, lo pair).  2-bit codes: 16 entries fill the 32 banks
    // once, so lookups never conflict.  3-bit codes: 16 copies, lane l reading copy
    // l % 16, so the 16 lanes of a 64-bit wavefront read 16 different bank pairs;
    // 4-bit codes: 4 copies at d = 128 (8 KB, so that four CTAs still fit an SM)
    // and 8 at d = 256 (two CTAs per SM).
    static constexpr int kLutCopies = (KB == 2) ? 1 : (KB == 3 ? 16 : (D == 256 ? 8 : 4));
    static constexpr int kLutShift = (KB == 2) ? 3 : (KB == 3 ? 7 : (D == 256 ? 6 : 5));  // log2(entry bytes, all copies)
    static constexpr size_t kLut = sizeof(uint2) * kPairEntries * kLutCopies;  // a multiple of 128
    static constexpr size_t kSignLut = sizeof(uint2) * 16;               // 4 sign bits -> two +-1 fp16 pairs
    static constexpr size_t kQfrag = sizeof(uint4) * (D / 16) * 32;      // [k-step][lane] (qh0, qh2, ql0, ql2)
    static constexpr size_t kSfrag = sizeof(uint2) * (D / 16) * 32;      // [k-step][lane] (qs0, qs2)
    static constexpr size_t kVLut = VM ? sizeof(uint32_t) * (1u << (2 * VB)) * 8 : 0;
    static constexpr size_t kHeader = kLut + kSignLut + kQfrag + kSfrag + 256 + kVLut;  // + flags, zeros, mbarriers
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

// The 4 KB-bit codes 16 s + 4 m .. 16 s + 4 m + 3 of the packed code row at shared
// offset `row`, in the low 4 KB bits (3- and 4-bit codes).
template <int KB, typename LD>
__device__ __forceinline__ uint32_t code_quad_off(const LD &ld32, uint32_t row, int s, int m)
{
    if constexpr (KB == 4) {
        return ld32(row + 8 * s + 4 * (m >> 1)) >> (16 * (m & 1));
    } else {
        const int bit = 48 * s + 12 * m;
        return __funnelshift_r(ld32(row + 4 * (bit >> 5)), ld32(row + 4 * ((bit >> 5) + 1)), bit & 31);
    }
}

__device__ __forceinline__ void mbar_init_cta(uint64_t *mbar, int count)
{
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(static_cast<uint32_t>(__cvta_generic_to_shared(mbar))),
                 "r"(count));
}

// A value code pair of two tokens (low / high 16-bit halves of x, bits [sh, sh + VB))
// as the byte offset of its entry in the value centroid table.
template <int VB>
__device__ __forceinline__ uint32_t vpair_off(uint32_t x, int sh)
{
    constexpr uint32_t M = (1u << VB) - 1u;
    return ((((x >> sh) & M) | (((x >> (16 + sh)) & M) << VB)) << 5);  // 8 copies x 4 bytes per entry
}

template <int D, int KB, int VB, bool VM, bool PF = false>
__global__ void __launch_bounds__(kThreads, D == 128 ? 4 : 2) decode_mma_kernel(const Codec C, const PageGeom PG, const DecodeArgs A)
{
    using SM = DecSmem<D, KB, VB, VM>;
    constexpr bool QJL = (KB <= 3);
    constexpr int KS = D / 16;                 // k-steps over coordinates
    constexpr int MT = D / 16;                 // m-tiles of output coordinates
    extern __shared__ __align__(16) unsigned char smem[];
    uint2 *lut = reinterpret_cast<uint2 *>(smem);
    uint2 *slut = reinterpret_cast<uint2 *>(smem + SM::kLut);
    uint4 *qfrag = reinterpret_cast<uint4 *>(smem + SM::kLut + SM::kSignLut);
    uint2 *sfrag = reinterpret_cast<uint2 *>(smem + SM::kLut + SM::kSignLut + SM::kQfrag);
    int *page_ok = reinterpret_cast<int *>(smem + SM::kLut + SM::kSignLut + SM::kQfrag + SM::kSfrag);  // [4][2][2]
    uint32_t *zero_meta = reinterpret_cast<uint32_t *>(page_ok + 16);  // [16] zeros: metadata of masked tokens
    uint64_t *mbar = reinterpret_cast<uint64_t *>(page_ok + 32);        // [4 warps][2 stages] barriers
    volatile int *cta_abort = page_ok + 48;                             // a warp gave up waiting for its pages
    const uint32_t zero_off = static_cast<uint32_t>(SM::kLut + SM::kSignLut + SM::kQfrag + SM::kSfrag + 64);
    unsigned char *stages = smem + SM::kHeader;

    // Columns of the score and value MMAs are (query token, head) pairs: decode has
    // one query token per sequence (columns = the G heads of the kv head); prefill
    // gives a CTA qpc consecutive query tokens of its sequence (qpc * G <= 8 columns),
    // each masked causally.
    // (PF: prefill; otherwise Tq = qpc = 1 at compile time)
    const int Tq = PF ? A.Tq : 1, qpc = PF ? A.qpc : 1;
    const int nqt = PF ? (Tq + qpc - 1) / qpc : 1;
    const int split = blockIdx.x, kvh = blockIdx.y, b = PF ? blockIdx.z / nqt : blockIdx.z;
    const int qt = PF ? blockIdx.z % nqt : 0;
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int quad = lane & 3, row = lane >> 2;
    const int P = PG.P;
    const int G = A.Hq / A.Hkv;
    const int ng = D / C.group;
    const int pshift = __ffs(P) - 1;                 // page size and value group are powers of two
    const int gshift = __ffs(C.group) - 1;

    int L = A.seq_lens[b];
    if (L < 0) L = 0;
    if (L > A.max_blocks * P) {
        if (split == 0 && kvh == 0 && qt == 0 && tid == 0) atomicOr(C.status, TQ_DEVERR_SEQ_RANGE);
        L = A.max_blocks * P;
    }
    const int q0 = qt * qpc;                    // first query token of this CTA
    const int ncol = min(qpc, Tq - q0) * G;     // columns: (query q0 + c / G, head c % G)
    const size_t rows_total = static_cast<size_t>(A.B) * Tq * A.Hq;
    // query row of column c, and its causal limit: query token i of a sequence of L
    // tokens sits at position L - Tq + i and sees positions below L - Tq + i + 1
    auto col_row = [&](int c) -> size_t {
        if (!PF) return static_cast<size_t>(b) * A.Hq + static_cast<size_t>(kvh) * G + c;
        return (static_cast<size_t>(b) * Tq + q0 + c / G) * A.Hq + static_cast<size_t>(kvh) * G + c % G;
    };
    auto col_lim = [&](int c) -> int { return PF ? max(0, L - Tq + q0 + c / G + 1) : L; };
    const int Lmax = col_lim(ncol - 1);          // the last column sees the most tokens
    const int npages = (Lmax + P - 1) / P;
    const int pg0 = split * A.pages_per_split;
    const int pg1 = min(npages, pg0 + A.pages_per_split);
    float *ml_base = A.ws.ml + static_cast<size_t>(split) * rows_total * 2;
    float *acc_base = A.ws.acc + static_cast<size_t>(split) * rows_total * D;
    if (pg0 >= pg1) {
        if (tid < ncol) {
            ml_base[2 * col_row(tid)] = -INFINITY;
            ml_base[2 * col_row(tid) + 1] = 0.f;
        }
        return;
    }

    // ---- tables: fp16 centroid pairs (16 copies) and +-1 sign pairs ----
    for (int e = tid; e < SM::kPairEntries * SM::kLutCopies; e += kThreads) {
        const int ent = e / SM::kLutCopies;
        const int c0 = ent & ((1 << KB) - 1), c1 = ent >> KB;
        const float x0 = C.centroids[c0], x1 = C.centroids[c1];
        const float h0 = __half2float(__float2half_rn(x0)), h1 = __half2float(__float2half_rn(x1));
        lut[e] = make_uint2(pack_half2(h0, h1), pack_half2((x0 - h0) * kLoScale, (x1 - h1) * kLoScale));
    }
    const uint32_t vlut_off = static_cast<uint32_t>(SM::kLut + SM::kSignLut + SM::kQfrag + SM::kSfrag + 256);
    if constexpr (VM) {  // value centroid pairs, fp16 of vlut_scale * c (the scale keeps them near fp16 points)
        uint32_t *vlut = reinterpret_cast<uint32_t *>(smem + vlut_off);
        for (int e = tid; e < (1 << (2 * VB)) * 8; e += kThreads) {
            const int ent = e >> 3;
            vlut[e] = pack_half2(C.vcentroids[ent & ((1 << VB) - 1)] * C.vlut_scale, C.vcentroids[ent >> VB] * C.vlut_scale);
        }
    }
    if (tid < 16) {
        zero_meta[tid] = 0u;
        auto pm = [](int bit) { return bit ? 1.f : -1.f; };
        slut[tid] = make_uint2(pack_half2(pm(tid & 1), pm(tid & 2)), pack_half2(pm(tid & 4), pm(tid & 8)));
    }

    // ---- query fragments (B operand of the score MMA, head = lane / 4), permuted
    // coordinates; identical for the four warps, so warp 0 writes them ----
    if (warp == 0) {
        const bool hv = row < ncol;
        const float *qr = A.ws.qrot + col_row(hv ? row : 0) * D;
        const float *qs = A.ws.qs + col_row(hv ? row : 0) * D;
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

    // this lane's two columns 2 quad + e: present, and their causal limits
    bool colv[2];
    int lim[2];
#pragma unroll
    for (int e = 0; e < 2; ++e) {
        colv[e] = 2 * quad + e < ncol;
        lim[e] = colv[e] ? col_lim(2 * quad + e) : 0;
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
    // shared-memory reads by 32-bit byte offset
    auto ld32 = [&](uint32_t off) -> uint32_t { return *reinterpret_cast<const uint32_t *>(smem + off); };
    auto ld64 = [&](uint32_t off) -> uint2 { return *reinterpret_cast<const uint2 *>(smem + off); };
    auto ldu16 = [&](uint32_t off) -> uint32_t { return *reinterpret_cast<const uint16_t *>(smem + off); };
    constexpr uint32_t PM = (1u << (2 * KB)) - 1u;
    // 2-bit codes: code pair (4 quad, 4 quad + 1) / (4 quad + 2, 4 quad + 3) of a k-step word
    // rotated to bits 3..6 is the byte offset of its table entry
    const int rot0 = (8 * quad + 29) & 31, rot1 = (8 * quad + 1) & 31;
    const uint32_t lut_lane = 8u * (lane & (SM::kLutCopies - 1));  // 3- and 4-bit codes: this lane's table copy
    const uint32_t slut_off = static_cast<uint32_t>(SM::kLut);
    const int mt_mask = (C.group >> 4) - 1;     // m-tiles per value group - 1
    // value codes of coordinates 16 mt + 2 row (+1): byte (2-bit) or nibble pair (4-bit) of the row
    const uint32_t vsel = (VB == 2) ? (static_cast<uint32_t>(row >> 1) | (static_cast<uint32_t>(4 + (row >> 1)) << 8))
                                    : (static_cast<uint32_t>(row & 3) | (static_cast<uint32_t>(4 + (row & 3)) << 8));
    const int vsh = 4 * (row & 1);
    const uint32_t vwoff = 4u * (row >> 2);

    // ---- per-warp page pipelines: warp w takes the 32-token rounds w, w + 4, ... of the
    // split (wpc pages each), with its own two stages and mbarriers, so the warps of a
    // CTA never wait for one another before the final merge.  Lane q < wpc copies page
    // q of a round with two bulk copies (keys, values) completing on the stage's
    // mbarrier; block ids are read one round ahead ----
    const int wpc = (kTile * kTilesPerWarp) >> pshift;   // pages per round: 2 (P = 16) or 1 (P = 32)
    const uint32_t page_bytes = static_cast<uint32_t>(PG.k_page + PG.v_page);
    auto stage_off = [&](int st) -> uint32_t {            // this warp's stage st: wpc pages, K then V each
        return static_cast<uint32_t>(SM::kHeader) + static_cast<uint32_t>((warp * 2 + st) * wpc) * page_bytes;
    };
    auto round_page = [&](int r) -> int { return pg0 + (4 * r + warp) * wpc; };
    auto fetch_id = [&](int r) -> int {
        int blk = -1;
        const int pgq = round_page(r) + lane;
        if (lane < wpc && pgq < pg1) blk = A.block_table[static_cast<int64_t>(b) * A.max_blocks + pgq];
        return blk;
    };
    auto issue = [&](int r, int st, int blk) {  // by lanes q < wpc
        const int q = lane;
        int ok = 0;
        if (round_page(r) + q < pg1) {
            ok = (blk >= 0 && blk < A.num_blocks);
            if (!ok) atomicOr(C.status, TQ_DEVERR_BLOCK_RANGE);
        }
        page_ok[(warp * 2 + st) * 2 + q] = ok;
        const uint32_t bytes = ok ? page_bytes : 0u;
        const uint32_t mb = static_cast<uint32_t>(__cvta_generic_to_shared(&mbar[warp * 2 + st]));
        asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(mb), "r"(bytes) : "memory");
        if (ok) {
            const size_t rec = static_cast<size_t>(blk) * A.Hkv + kvh;
            const uint32_t kd = static_cast<uint32_t>(__cvta_generic_to_shared(smem)) + stage_off(st) + q * page_bytes;
            const uint32_t vd = kd + static_cast<uint32_t>(PG.k_page);
            asm volatile("cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];"
                         ::"r"(kd), "l"(A.k_cache + rec * PG.k_page), "r"(static_cast<uint32_t>(PG.k_page)), "r"(mb)
                         : "memory");
            asm volatile("cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];"
                         ::"r"(vd), "l"(A.v_cache + rec * PG.v_page), "r"(static_cast<uint32_t>(PG.v_page)), "r"(mb)
                         : "memory");
        }
    };

    const int nrounds = (pg1 - pg0 + 4 * wpc - 1) / (4 * wpc);
    auto stage_ready = [&](int st, uint32_t par) -> bool {
        const uint32_t mb = static_cast<uint32_t>(__cvta_generic_to_shared(&mbar[warp * 2 + st]));
        uint32_t done;
        asm volatile("{\n.reg .pred p;\nmbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\nselp.u32 %0, 1, 0, p;\n}\n"
                     : "=r"(done) : "r"(mb), "r"(par) : "memory");
        return done != 0;
    };
    auto stage_tested = [&](int st, uint32_t par) -> bool {
        const uint32_t mb = static_cast<uint32_t>(__cvta_generic_to_shared(&mbar[warp * 2 + st]));
        uint32_t done;
        asm volatile("{\n.reg .pred p;\nmbarrier.test_wait.parity.shared::cta.b64 p, [%1], %2;\nselp.u32 %0, 1, 0, p;\n}\n"
                     : "=r"(done) : "r"(mb), "r"(par) : "memory");
        return done != 0;
    };
    auto drain = [&](int st, uint32_t par) {  // copies in flight must land before the CTA exits
        const long long t0 = clock64();
        while (!stage_ready(st, par) && clock64() - t0 < kDrainLimit) {
        }
    };
    if (tid < 8) mbar_init_cta(&mbar[tid], wpc);
    if (tid == 0) *cta_abort = 0;
    if (tid == 0) asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    __syncthreads();  // tables, query fragments and barriers are ready
    int bnext = fetch_id(0);
    if (lane < wpc) issue(0, 0, bnext);
    bnext = fetch_id(1);
    for (int c = 0; c < nrounds; ++c) {
        const int st = c & 1;
        if (c + 1 < nrounds && lane < wpc) {
            issue(c + 1, st ^ 1, bnext);
            bnext = fetch_id(c + 2);
        }
        {
            // bounded wait for this round's pages; on a timeout the warp stops issuing,
            // waits (with a fixed, longer bound) for the copies it still has in flight,
            // and the CTA drops its split (the combine then gives it no weight)
            bool ok = true;
            if (C.wait_limit <= 0) {  // a zero limit tests once without blocking
                ok = stage_tested(st, (c >> 1) & 1);
            } else {
                const long long t0 = clock64();
                while (!stage_ready(st, (c >> 1) & 1)) {
                    if (clock64() - t0 > C.wait_limit) {
                        ok = false;
                        break;
                    }
                }
            }
            ok = __all_sync(0xffffffffu, ok);  // the lanes poll separately: decide as a warp
            if (!ok) {
                if (lane == 0) {
                    atomicOr(C.status, TQ_DEVERR_TIMEOUT);
                    *cta_abort = 1;
                }
                drain(st, (c >> 1) & 1);
                if (c + 1 < nrounds) drain(st ^ 1, ((c + 1) >> 1) & 1);
                break;
            }
        }

        // ---- the round's two tiles: tokens 16 j of the round ----
        int kp[2], vp[2], o0[2], pos0[2];
        bool live[2];
        const int rpage = round_page(c);
#pragma unroll
        for (int j = 0; j < 2; ++j) {
            const int q = (kTile * j) >> pshift;
            o0[j] = (kTile * j) & (P - 1);
            pos0[j] = (rpage + q) * P + o0[j];
            live[j] = (rpage + q < pg1) && page_ok[(warp * 2 + st) * 2 + q] && (pos0[j] < L);
            kp[j] = static_cast<int>(stage_off(st) + q * page_bytes);
            vp[j] = kp[j] + static_cast<int>(PG.k_page);
        }
        if (live[0] || live[1]) {
            // ---- scores S[token][head]: this lane feeds tokens row, row + 8 of both tiles ----
            // per tile j and token row + 8 hh: a[.][.][0..1] = hi.qh, a[2..3] = lo.qh; b[0..1] = hi.ql
            float sa[2][2][4], sb[2][2][4], ss[2][4];
            uint32_t krow[2][2], srow[2][2];
#pragma unroll
            for (int j = 0; j < 2; ++j) {
#pragma unroll
                for (int i = 0; i < 4; ++i) sa[j][0][i] = sa[j][1][i] = sb[j][0][i] = sb[j][1][i] = ss[j][i] = 0.f;
#pragma unroll
                for (int hh = 0; hh < 2; ++hh) {
                    krow[j][hh] = kp[j] + (o0[j] + row + 8 * hh) * C.k_code_bytes;
                    srow[j][hh] = kp[j] + PG.k_sign_off + (o0[j] + row + 8 * hh) * C.k_sign_bytes;
                }
            }
#pragma unroll
            for (int s = 0; s < KS; ++s) {
                const uint4 qf = qfrag[s * 32 + lane];
                uint2 sf = make_uint2(0u, 0u);
                if (QJL) sf = sfrag[s * 32 + lane];
#pragma unroll
                for (int j = 0; j < 2; ++j) {
                    uint2 e[2][2];  // [token hh][pair]
#pragma unroll
                    for (int hh = 0; hh < 2; ++hh) {
                        if constexpr (KB == 2) {
                            const uint32_t w = ld32(krow[j][hh] + 4 * s);
                            e[hh][0] = ld64(__funnelshift_r(w, w, rot0) & 0x78u);
                            e[hh][1] = ld64(__funnelshift_r(w, w, rot1) & 0x78u);
                        } else {
                            const uint32_t f = code_quad_off<KB>(ld32, krow[j][hh], s, quad);
                            e[hh][0] = ld64(lut_lane + ((f & PM) << SM::kLutShift));
                            e[hh][1] = ld64(lut_lane + (((f >> (2 * KB)) & PM) << SM::kLutShift));
                        }
                    }
                    // M rows r / r + 8 = high / low centroid parts of one token: each table load
                    // (hi, lo) fills two adjacent A registers
#pragma unroll
                    for (int hh = 0; hh < 2; ++hh) {
                        mma16816(sa[j][hh], e[hh][0].x, e[hh][0].y, e[hh][1].x, e[hh][1].y, qf.x, qf.y);
                        mma16816(sb[j][hh], e[hh][0].x, e[hh][0].y, e[hh][1].x, e[hh][1].y, qf.z, qf.w);
                    }
                    if (QJL) {
                        const int rot = (16 * (s & 1) + 4 * quad + 29) & 31;
                        const uint32_t w0 = ld32(srow[j][0] + 4 * (s >> 1)), w1 = ld32(srow[j][1] + 4 * (s >> 1));
                        const uint2 g0 = ld64((__funnelshift_r(w0, w0, rot) & 0x78u) | slut_off);
                        const uint2 g1 = ld64((__funnelshift_r(w1, w1, rot) & 0x78u) | slut_off);
                        mma16816(ss[j], g0.x, g1.x, g0.y, g1.y, sf.x, sf.y);
                    }
                }
            }
            // ---- scale and mask: x[j][hh][e] = tile j, token row + 8 hh, head 2 quad + e ----
            float x[2][2][2];
#pragma unroll
            for (int j = 0; j < 2; ++j)
#pragma unroll
                for (int hh = 0; hh < 2; ++hh) {
                    const int t = o0[j] + row + 8 * hh;
                    const float nrm = bf16_to_float(ldu16(kp[j] + PG.k_norm_off + 2 * t));
                    const float gam = QJL ? bf16_to_float(ldu16(kp[j] + PG.k_gamma_off + 2 * t)) : 0.f;
                    const int pos = pos0[j] + row + 8 * hh;
#pragma unroll
                    for (int e = 0; e < 2; ++e) {
                        const int i = 2 * hh + e;
                        const float lo = sa[j][hh][2 + e] + sb[j][hh][e];  // lo.qh + hi.ql
                        float v = nrm * fac_c * fmaf(lo, 1.f / kLoScale, sa[j][hh][e]);
                        if (QJL) v = fmaf(nrm * fac_s * gam, ss[j][i], v);
                        x[j][hh][e] = colv[e] ? ((live[j] && pos < lim[e]) ? v : -INFINITY) : 0.f;
                    }
                }
            // ---- online softmax (base 2) per head 2 quad + e over the 32 tokens ----
            float p[2][2][2], alpha[2];
#pragma unroll
            for (int e = 0; e < 2; ++e) {
                float mt = fmaxf(fmaxf(x[0][0][e], x[0][1][e]), fmaxf(x[1][0][e], x[1][1][e]));
                mt = fmaxf(mt, __shfl_xor_sync(0xffffffffu, mt, 4));
                mt = fmaxf(mt, __shfl_xor_sync(0xffffffffu, mt, 8));
                mt = fmaxf(mt, __shfl_xor_sync(0xffffffffu, mt, 16));
                const float m_new = fmaxf(m_run[e], mt);
                alpha[e] = 1.f;
                float ps = 0.f;
#pragma unroll
                for (int j = 0; j < 2; ++j)
#pragma unroll
                    for (int hh = 0; hh < 2; ++hh) {
                        p[j][hh][e] = (m_new != -INFINITY) ? fast_exp2(x[j][hh][e] - m_new) : 0.f;
                        ps += p[j][hh][e];
                    }
                if (m_new != -INFINITY) alpha[e] = fast_exp2(m_run[e] - m_new);
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
            // ---- values: per tile, P^T as the B operand (tokens 2 quad + {0,1} (+8), head `row`) ----
            uint32_t b0[2], b1[2];
            uint32_t mrow[2][4], vrow[2][4];
            const int tq[4] = {2 * quad, 2 * quad + 1, 2 * quad + 8, 2 * quad + 9};
#pragma unroll
            for (int j = 0; j < 2; ++j) {
                b0[j] = movmatrix_trans(pack_half2(p[j][0][0], p[j][0][1]));
                b1[j] = movmatrix_trans(pack_half2(p[j][1][0], p[j][1][1]));
#pragma unroll
                for (int i = 0; i < 4; ++i) {
                    const int t = o0[j] + tq[i];
                    // metadata of masked tokens (never-written bytes may hold any fp16 pattern) reads zeros
                    mrow[j][i] = (live[j] && pos0[j] + tq[i] < Lmax) ? vp[j] + PG.v_meta_off + t * C.v_meta_bytes : zero_off;
                    vrow[j][i] = vp[j] + t * C.v_code_bytes;
                }
                if constexpr (!VM) {
                    // zero term: A rows = groups (`row` < ng), columns = tokens
                    uint32_t za0 = 0u, za2 = 0u;
                    if (row < ng) {
                        za0 = __byte_perm(ld32(mrow[j][0] + 4 * row), ld32(mrow[j][1] + 4 * row), 0x7632);
                        za2 = __byte_perm(ld32(mrow[j][2] + 4 * row), ld32(mrow[j][3] + 4 * row), 0x7632);
                    }
                    mma16816(zt, za0, 0u, za2, 0u, b0[j], b1[j]);
                }
            }
            // ---- P.V over coordinate m-tiles: row r <-> 16 mt + 2 r, row r + 8 <-> 16 mt + 2 r + 1 ----
            constexpr uint32_t VCM = ((1u << VB) - 1u) * 0x00010001u;
            const uint32_t bias = 0x64006400u;
            uint32_t bs0[2] = {0u, 0u}, bs1[2] = {0u, 0u};
            if constexpr (VM) {  // one weight per token: its value norm, times 2^-4 to stay inside fp16
#pragma unroll
                for (int j = 0; j < 2; ++j) {
                    float w[4];
#pragma unroll
                    for (int i = 0; i < 4; ++i)
                        w[i] = (mrow[j][i] != zero_off)
                                   ? bf16_to_float(ldu16(vp[j] + PG.v_meta_off + 2 * (o0[j] + tq[i]))) * 0.0625f
                                   : 0.f;
                    bs0[j] = hmul2_u32(b0[j], pack_half2(w[0], w[1]));
                    bs1[j] = hmul2_u32(b1[j], pack_half2(w[2], w[3]));
                }
            }
            const uint32_t vlut_lane = vlut_off + 4u * (lane & 7);
#pragma unroll
            for (int mt = 0; mt < MT; ++mt) {
                if (!VM && (mt & mt_mask) == 0) {  // a new value group: scale the B operands
                    const int g4 = 4 * ((16 * mt) >> gshift);
#pragma unroll
                    for (int j = 0; j < 2; ++j) {
                        bs0[j] = hmul2_u32(b0[j], __byte_perm(ld32(mrow[j][0] + g4), ld32(mrow[j][1] + g4), 0x5410));
                        bs1[j] = hmul2_u32(b1[j], __byte_perm(ld32(mrow[j][2] + g4), ld32(mrow[j][3] + g4), 0x5410));
                    }
                }
#pragma unroll
                for (int j = 0; j < 2; ++j) {
                    uint32_t xa, xb;  // codes of coordinates 16 mt + 2 row (+1): tokens (0, 1) | (2, 3)
                    if constexpr (VB == 2) {
                        xa = __byte_perm(ld32(vrow[j][0] + 4 * mt), ld32(vrow[j][1] + 4 * mt), vsel) >> vsh;
                        xb = __byte_perm(ld32(vrow[j][2] + 4 * mt), ld32(vrow[j][3] + 4 * mt), vsel) >> vsh;
                    } else if constexpr (VB == 4) {
                        const uint32_t w = 8 * mt + vwoff;
                        xa = __byte_perm(ld32(vrow[j][0] + w), ld32(vrow[j][1] + w), vsel);
                        xb = __byte_perm(ld32(vrow[j][2] + w), ld32(vrow[j][3] + w), vsel);
                    } else {
                        const int bit = 48 * mt + 6 * row;
                        const uint32_t w = 4 * (bit >> 5);
                        const int sh = bit & 31;
                        xa = __byte_perm(__funnelshift_r(ld32(vrow[j][0] + w), ld32(vrow[j][0] + w + 4), sh),
                                         __funnelshift_r(ld32(vrow[j][1] + w), ld32(vrow[j][1] + w + 4), sh), 0x5410);
                        xb = __byte_perm(__funnelshift_r(ld32(vrow[j][2] + w), ld32(vrow[j][2] + w + 4), sh),
                                         __funnelshift_r(ld32(vrow[j][3] + w), ld32(vrow[j][3] + w + 4), sh), 0x5410);
                    }
                    uint32_t a0, a1, a2, a3;
                    if constexpr (VM) {  // value centroids of the two tokens' codes
                        a0 = ld32(vlut_lane + vpair_off<VB>(xa, 0));
                        a1 = ld32(vlut_lane + vpair_off<VB>(xa, VB));
                        a2 = ld32(vlut_lane + vpair_off<VB>(xb, 0));
                        a3 = ld32(vlut_lane + vpair_off<VB>(xb, VB));
                    } else {
                        a0 = unbias_half2((xa & VCM) | bias);
                        a1 = unbias_half2(((xa >> VB) & VCM) | bias);
                        a2 = unbias_half2((xb & VCM) | bias);
                        a3 = unbias_half2(((xb >> VB) & VCM) | bias);
                    }
                    mma16816(o[mt], a0, a1, a2, a3, bs0[j], bs1[j]);
                }
            }
        }
        __syncwarp();  // the next issue() overwrites this stage
    }
    __syncthreads();  // every warp is done with the stages before they hold merge data
    if (*cta_abort) {  // a page wait timed out: this split contributes nothing
        if (tid < ncol) {
            ml_base[2 * col_row(tid)] = -INFINITY;
            ml_base[2 * col_row(tid) + 1] = 0.f;
        }
        return;
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
    for (int e = tid; e < ncol * D; e += kThreads) {
        const int h = e / D, j = e - h * D;  // column h
        float M = -INFINITY;
#pragma unroll
        for (int w = 0; w < kWarps; ++w) M = fmaxf(M, r_m[w * 8 + h]);
        float acc = 0.f, l = 0.f;
        if (M != -INFINITY) {
#pragma unroll
            for (int w = 0; w < kWarps; ++w) {
                const float f = fast_exp2(r_m[w * 8 + h] - M);
                acc = fmaf(f, r_o[(w * D + j) * 8 + h] + r_z[(w * 8 + (j >> gshift)) * 8 + h], acc);
                l = fmaf(f, r_l[w * 8 + h], l);
            }
        }
        const size_t rr = col_row(h);
        acc_base[rr * D + j] = acc;
        if (j == 0) {
            ml_base[2 * rr] = M;
            ml_base[2 * rr + 1] = l;
        }
    }
}

}  // namespace dmma
}  // namespace tq
