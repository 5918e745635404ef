// tq_prefill_tc.cu -- chunked prefill over the compressed cache on the
// 5th-generation tensor cores (head_dim 128).
//
// turbo-attn, "How it works": the prefill path dequantises the codec inline in
// its MMA pipeline, with no decompress buffer in global memory.  Here the pages
// of a 64-token tile are decoded once into shared-memory operand tiles that
// every column of the CTA shares, and the products run as tcgen05.mma with the
// accumulators in tensor memory:
//
//   S[c][t] = sum_j Q'[c][j] K'[t][j]          (M = 128 columns, N = 64 tokens)
//   O[c][j] += sum_t P[c][t] V[t][j]           (M = 128 columns, N = 128 coordinates)
//
// A column c is a (query token, head) pair of one sequence and kv head.  With
// q' = 2^e q_rot (a power of two per column, exact) and k' = 2^8 c[code], both
// split into fp16 high and low parts, the score MMAs accumulate q'h k'h + q'h
// k'l + q'l k'h (~22 significant bits) and the QJL term as one more product
// (2^e R q_s) (2^8 g_t sigma_t) with g_t the stored bf16 gamma (exact in fp16
// after the power-of-two scale), R = sqrt(pi/2) / sqrt(d) and sigma = 2 sign - 1,
// so that
//   S[c][t] = 2^(e + 8) (<q_rot, c[code_t]> + sqrt(pi/2) / sqrt(d) g_t <q_s, sigma_t>)
// and the log2-domain score is x = 2^-(e + 8) S n_t sm_scale log2(e) / sqrt(d).
// Values enter P.V as fp16 (code * scale + zero, one rounding; with values coded
// by the rotation: fp16(lambda c[code]) * fp16(n / 16), the combine rotates the
// merged output back).
//
// Warp roles (448 threads, one CTA per SM):
//   warps 0-3   one thread per column (tensor-memory lane): query operands, online
//               softmax with a lazy rescale of O (only when the running maximum grows
//               by more than 2^8, so P <= 2^8 stays exact in fp16), P into tensor
//               memory, the partial outputs at the end;
//   warps 4-11  the decode of a tile's pages into fp16 operand tiles (three stages);
//   warp 12     tensor-memory allocation; lane 0 issues the MMAs;
//   warp 13     page copies (cp.async.bulk, two stages), block ids read ahead.
// Every wait is bounded by the codec's wait limit; a timeout sets
// TQ_DEVERR_TIMEOUT, stops the CTA (its split then carries no weight), lets
// copies and MMAs in flight finish, and frees tensor memory.
#include <cuda_runtime.h>

#include "tq_device.cuh"
#include "tq_internal.h"
#include "tq_umma.cuh"

namespace tq {
namespace pftc {

constexpr int D = 128;
constexpr int kSoftWarps = 4;
constexpr int kProdWarps = 8;
constexpr int kMmaWarp = kSoftWarps + kProdWarps;
constexpr int kLoadWarp = kMmaWarp + 1;
constexpr int kThreads = (kLoadWarp + 1) * 32;
constexpr int kProdThreads = kProdWarps * 32;
constexpr int kCols = 128;                 // columns per CTA (M of every MMA)
constexpr int kTok = 64;                   // tokens per tile
constexpr int kRaw = 2;                    // page stages
constexpr int kOps = 3;                    // operand stages
constexpr float kKScale = 256.f;           // centroids enter the MMA as 2^8 c
constexpr float kLazy = 8.f;               // rescale O only when the maximum grows by more than this (log2 units)
constexpr float kLog2e = 1.4426950408889634f;
constexpr float kQjlR = 1.2533141373155003f * 0.08838834764831845f;  // sqrt(pi/2) / sqrt(128)

// tensor-memory columns (fp32 or packed fp16 pairs)
constexpr uint32_t kTmQh = 0, kTmQl = 64, kTmQs = 128;  // A operands: 128 fp16 per row = 64 columns each
constexpr uint32_t kTmO = 192;                          // O: 128 fp32 columns
constexpr uint32_t kTmS = 320;                          // S: two buffers of 64 fp32 columns
constexpr uint32_t kTmP = 448;                          // P: 64 fp16 per row = 32 columns
constexpr uint32_t kTmCols = 512;

// shared memory (bytes)
constexpr uint32_t kTileBytes = kTok * D * 2;          // one fp16 operand tile, 16 KB
constexpr uint32_t kOpBytes = 4 * kTileBytes;          // Kh, Kl, Ks (signed gamma), Vt per stage
constexpr uint32_t kLutOff = kOps * kOpBytes;          // key centroid pairs (high pair, low pair), in copies
constexpr uint32_t kLutBytes = 8192;
constexpr uint32_t kVlutOff = kLutOff + kLutBytes;     // value centroid pairs (values coded by the rotation)
constexpr uint32_t kTokOff = kVlutOff + 1024;          // [3][64] float: n_t sm_scale log2(e) / sqrt(d)
constexpr uint32_t kOkOff = kTokOff + 768;             // [3] uint64: tokens of a valid page
constexpr uint32_t kPageOkOff = kOkOff + 32;           // [kRaw <= 3][4] int
constexpr uint32_t kMbarOff = kPageOkOff + 48;
constexpr int kNumMbar = 18;
constexpr uint32_t kMiscOff = kMbarOff + 8 * kNumMbar;  // tensor-memory base, abort flag
constexpr uint32_t kRawOff = (kMiscOff + 16 + 127) / 128 * 128;
// mbarrier indices
constexpr int kBarRaw = 0;       // [kRaw <= 3] a page stage landed (ppt arrivals + bytes)
constexpr int kBarOpFull = 3;    // [3] an operand stage is decoded (one arrival per producer warp)
constexpr int kBarOpFree = 6;    // [3] the MMAs reading an operand stage are done (commit)
constexpr int kBarSFull = 9;     // [2] scores of a tile are in tensor memory (commit)
constexpr int kBarSFree = 11;    // [2] the softmax warps have read a score buffer (4 arrivals)
constexpr int kBarPFull = 13;    // P of a tile is in tensor memory, O rescaled (4 arrivals)
constexpr int kBarPvDone = 14;   // O += P V of a tile is done (commit)
constexpr int kBarMmaDone = 15;  // teardown: every MMA issued is done (commit)
constexpr int kBarRawFree = 16;  // [kRaw <= 2] the producer warps are done reading a page stage (8 arrivals)

__host__ __device__ inline uint32_t raw_stage_bytes(const PageGeom &pg)
{
    const uint32_t b = static_cast<uint32_t>(kTok / pg.P) * static_cast<uint32_t>(pg.k_page + pg.v_page);
    return (b + 127u) / 128u * 128u;
}

__host__ __device__ inline size_t smem_bytes(const PageGeom &pg) { return kRawOff + kRaw * raw_stage_bytes(pg); }

__device__ __forceinline__ uint32_t smem_addr(const void *p) { return static_cast<uint32_t>(__cvta_generic_to_shared(p)); }

__device__ __forceinline__ void st128(unsigned char *p, uint4 v) { *reinterpret_cast<uint4 *>(p) = v; }

// Shared-memory accesses by 32-bit shared address (explicit ld/st.shared: the decode
// helpers get their stage addresses as integers, so no access falls back to a
// generic load).  Volatile, so they stay in program order with the barrier waits.
__device__ __forceinline__ uint32_t lds32(uint32_t a)
{
    uint32_t v;
    asm volatile("ld.shared.b32 %0, [%1];" : "=r"(v) : "r"(a));
    return v;
}
__device__ __forceinline__ uint32_t lds16(uint32_t a)
{
    uint32_t v;
    asm volatile("ld.shared.u16 %0, [%1];" : "=r"(v) : "r"(a));
    return v;
}
__device__ __forceinline__ uint32_t lds8(uint32_t a)
{
    uint32_t v;
    asm volatile("ld.shared.u8 %0, [%1];" : "=r"(v) : "r"(a));
    return v;
}
__device__ __forceinline__ uint2 lds64(uint32_t a)
{
    uint2 v;
    asm volatile("ld.shared.v2.b32 {%0, %1}, [%2];" : "=r"(v.x), "=r"(v.y) : "r"(a));
    return v;
}
__device__ __forceinline__ void sts128(uint32_t a, uint4 v)
{
    asm volatile("st.shared.v4.b32 [%0], {%1, %2, %3, %4};" ::"r"(a), "r"(v.x), "r"(v.y), "r"(v.z), "r"(v.w)
                 : "memory");
}

__device__ __forceinline__ uint32_t half2_bits(__half2 h) { return *reinterpret_cast<uint32_t *>(&h); }
__device__ __forceinline__ __half2 bits_half2(uint32_t u) { return *reinterpret_cast<__half2 *>(&u); }

__device__ __forceinline__ void mbar_arrive(uint64_t *mb)
{
    asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_addr(mb)) : "memory");
}

// One arrival per warp: the warp's lanes meet first (their earlier shared-memory and
// tensor-memory work ordered before lane 0's arrival), so a barrier counts warps
// rather than threads and takes a few atomic updates per hand-off instead of hundreds.
__device__ __forceinline__ void warp_arrive(uint64_t *mb)
{
    __syncwarp();
    if ((threadIdx.x & 31) == 0) mbar_arrive(mb);
}

// 32 consecutive 32-bit columns of this thread's tensor-memory lane from registers.
__device__ __forceinline__ void tm_st32(uint32_t taddr, const uint32_t (&r)[32])
{
    asm volatile("tcgen05.st.sync.aligned.32x32b.x32.b32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,"
                 "%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31,%32};"
                 ::"r"(taddr), "r"(r[0]), "r"(r[1]), "r"(r[2]), "r"(r[3]), "r"(r[4]), "r"(r[5]), "r"(r[6]),
                   "r"(r[7]), "r"(r[8]), "r"(r[9]), "r"(r[10]), "r"(r[11]), "r"(r[12]), "r"(r[13]), "r"(r[14]),
                   "r"(r[15]), "r"(r[16]), "r"(r[17]), "r"(r[18]), "r"(r[19]), "r"(r[20]), "r"(r[21]), "r"(r[22]),
                   "r"(r[23]), "r"(r[24]), "r"(r[25]), "r"(r[26]), "r"(r[27]), "r"(r[28]), "r"(r[29]), "r"(r[30]),
                   "r"(r[31])
                 : "memory");
}

// 64 consecutive fp32 columns of this thread's tensor-memory lane (one wait).
__device__ __forceinline__ void tm_ld64(uint32_t taddr, float (&v)[64])
{
    uint32_t r[64];
    asm volatile("tcgen05.ld.sync.aligned.32x32b.x64.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,"
                 "%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31,%32,%33,%34,%35,%36,%37,%38,%39,"
                 "%40,%41,%42,%43,%44,%45,%46,%47,%48,%49,%50,%51,%52,%53,%54,%55,%56,%57,%58,%59,%60,%61,%62,%63}, [%64];"
                 : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]),
                   "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]),
                   "=r"(r[15]), "=r"(r[16]), "=r"(r[17]), "=r"(r[18]), "=r"(r[19]), "=r"(r[20]), "=r"(r[21]),
                   "=r"(r[22]), "=r"(r[23]), "=r"(r[24]), "=r"(r[25]), "=r"(r[26]), "=r"(r[27]), "=r"(r[28]),
                   "=r"(r[29]), "=r"(r[30]), "=r"(r[31]), "=r"(r[32]), "=r"(r[33]), "=r"(r[34]), "=r"(r[35]),
                   "=r"(r[36]), "=r"(r[37]), "=r"(r[38]), "=r"(r[39]), "=r"(r[40]), "=r"(r[41]), "=r"(r[42]),
                   "=r"(r[43]), "=r"(r[44]), "=r"(r[45]), "=r"(r[46]), "=r"(r[47]), "=r"(r[48]), "=r"(r[49]),
                   "=r"(r[50]), "=r"(r[51]), "=r"(r[52]), "=r"(r[53]), "=r"(r[54]), "=r"(r[55]), "=r"(r[56]),
                   "=r"(r[57]), "=r"(r[58]), "=r"(r[59]), "=r"(r[60]), "=r"(r[61]), "=r"(r[62]), "=r"(r[63])
                 : "r"(taddr));
    asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
#pragma unroll
    for (int i = 0; i < 64; ++i) v[i] = __uint_as_float(r[i]);
}

// Copies of the key centroid-pair table (8 KB at most): 2-bit codes fill the 32 banks
// once, 3-bit codes 16 copies (conflict-free), 4-bit codes 4 copies.
__host__ __device__ constexpr int lut_copies(int kb) { return kb == 2 ? 1 : (kb == 3 ? 16 : 4); }

// (fp16 hi, fp16 lo) of x with hi + lo ~ x to ~22 bits.
__device__ __forceinline__ void split_half(float x, __half &hi, __half &lo)
{
    hi = __float2half_rn(x);
    lo = __float2half_rn(x - __half2float(hi));
}

// 2^k as a float for -126 <= k <= 127, exactly.
__device__ __forceinline__ float pow2f(int k) { return __uint_as_float(static_cast<uint32_t>(k + 127) << 23); }

// 2^x with the hardware approximation (relative error ~2^-22).
__device__ __forceinline__ float fast_exp2(float x)
{
    float y;
    asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}

struct KeyItem {
    uint32_t raw;              // shared address of the page stage
    uint32_t pok;              // shared address of the stage's page validity flags (int)
    uint32_t page_bytes;
    int pshift, P, pt;         // pt: producer thread 0..255
    uint32_t sign_off, gamma_off;
};

// The producer thread's 4 key items (token t, 8-coordinate chunk c): fp16 high and low
// parts of 2^8 c[code] from the pair table (the thread's copy `lut`), and with QJL the
// 8 values +-2^8 g_t (sign bit set where the QJL bit is 0).  Items (it = pt + 256 k)
// map the 8 lanes of a store phase to the 8 rows of one core matrix.  All loads are
// issued before any table lookup.
template <int KB>
__device__ __forceinline__ void decode_keys(const KeyItem &ki, uint32_t lut, uint32_t kh, uint32_t kl, uint32_t ksg)
{
    constexpr bool QJL = KB <= 3;
    constexpr int CP = lut_copies(KB);
    constexpr uint32_t PM = (1u << (2 * KB)) - 1u;
    constexpr int CODE_BYTES = D * KB / 8, SIGN_BYTES = D / 8;
    uint32_t w[4], sb[4], g[4], off[4];
    bool tv[4];
#pragma unroll
    for (int k = 0; k < 4; ++k) {
        const int it = ki.pt + kProdThreads * k;
        const int t = ((it >> 7) << 3) | (it & 7), c = (it >> 3) & 15;
        const int q = t >> ki.pshift, o = t & (ki.P - 1);
        tv[k] = lds32(ki.pok + 4 * q) != 0;
        const uint32_t kp = ki.raw + q * ki.page_bytes;
        const uint32_t crow = kp + o * CODE_BYTES;
        if constexpr (KB == 4) {
            w[k] = lds32(crow + 4 * c);
        } else if constexpr (KB == 2) {
            w[k] = lds16(crow + 2 * c);
        } else {
            const int by = 3 * c;
            const uint32_t wa = crow + (by & ~3);
            w[k] = __funnelshift_r(lds32(wa), lds32(wa + 4), 8 * (by & 3));
        }
        if constexpr (QJL) {
            sb[k] = lds8(kp + ki.sign_off + o * SIGN_BYTES + c);
            g[k] = lds16(kp + ki.gamma_off + 2 * o);
        }
        off[k] = umma::core_offset(t, 8 * c, D);
    }
    // every table lookup before any store (the shared-memory accesses are volatile, so
    // a store would hold back the next item's lookups); the codes of an invalid page
    // are masked into the table like any others and their entries replaced by zeros
    uint2 e[4][4];
#pragma unroll
    for (int k = 0; k < 4; ++k)
#pragma unroll
        for (int m = 0; m < 4; ++m) e[k][m] = lds64(lut + ((w[k] >> (2 * KB * m)) & PM) * (8 * CP));
#pragma unroll
    for (int k = 0; k < 4; ++k) {
        const uint4 hv = tv[k] ? make_uint4(e[k][0].x, e[k][1].x, e[k][2].x, e[k][3].x) : make_uint4(0u, 0u, 0u, 0u);
        const uint4 lv = tv[k] ? make_uint4(e[k][0].y, e[k][1].y, e[k][2].y, e[k][3].y) : make_uint4(0u, 0u, 0u, 0u);
        sts128(kh + off[k], hv);
        sts128(kl + off[k], lv);
        if constexpr (QJL) {
            // fp16 2^8 g (exact: a bf16 times 2^8, g >= 0), sign bit set where the bit is 0
            const uint32_t g2 = tv[k] ? half2_bits(__float2half2_rn(bf16_to_float(g[k]) * kKScale)) : 0u;
            const uint32_t nb = tv[k] ? ~sb[k] : 0u;
            auto sg = [&](int m) { return g2 | (((nb >> (2 * m)) & 1u) << 15) | (((nb >> (2 * m + 1)) & 1u) << 31); };
            sts128(ksg + off[k], make_uint4(sg(0), sg(1), sg(2), sg(3)));
        }
    }
}

struct ValueItem {
    uint32_t raw;              // shared address of the page stage
    uint32_t pok;              // shared address of the stage's page validity flags (int)
    uint32_t page_bytes;
    int pos0, L, pshift, P, gshift;
    int j7, tc, jb;
};

// One value item: 4 core-matrix rows of the value tile Vt[coordinate][token] in fp16,
// code * scale + zero (one rounding) or, with values coded by the rotation,
// fp16(lambda c[code]) * fp16(n / 16); tokens of an invalid page or past the
// sequence's end are zero (their records may hold any bit pattern).
template <int VB>
__device__ __forceinline__ void decode_values(const Codec &C, const PageGeom &PG, const ValueItem &it, uint32_t vlut,
                                              uint32_t vt)
{
    constexpr uint32_t M = (1u << VB) - 1u;
    uint32_t w[8][VB];  // the 32 coordinates' codes of each token: VB words
    uint32_t meta[8];
    bool vv[8];
#pragma unroll
    for (int u = 0; u < 8; ++u) {
        const int t = 8 * it.tc + u, q = t >> it.pshift, o = t & (it.P - 1);
        vv[u] = lds32(it.pok + 4 * q) != 0 && it.pos0 + t < it.L;
        const uint32_t vp = it.raw + q * it.page_bytes + static_cast<uint32_t>(PG.k_page);
        const uint32_t cw = vp + o * C.v_code_bytes + 4 * VB * it.jb;
#pragma unroll
        for (int x = 0; x < VB; ++x) w[u][x] = lds32(cw + 4 * x);
        if (C.vmse)
            meta[u] = lds16(vp + static_cast<uint32_t>(PG.v_meta_off) + 2 * o);
        else
            meta[u] = lds32(vp + static_cast<uint32_t>(PG.v_meta_off) + o * C.v_meta_bytes +
                            4 * ((32 * it.jb) >> it.gshift));
    }
    uint32_t row[4][4];  // [k][token pair]
#pragma unroll
    for (int pr = 0; pr < 4; ++pr) {
        const int u0 = 2 * pr, u1 = 2 * pr + 1;
        __half2 sc2, zc2;
        if (C.vmse) {
            sc2 = __floats2half2_rn(vv[u0] ? bf16_to_float(meta[u0]) * 0.0625f : 0.f,
                                    vv[u1] ? bf16_to_float(meta[u1]) * 0.0625f : 0.f);
            zc2 = __float2half2_rn(0.f);
        } else {
            const uint32_t m0 = vv[u0] ? meta[u0] : 0u, m1 = vv[u1] ? meta[u1] : 0u;
            sc2 = bits_half2(__byte_perm(m0, m1, 0x5410));  // scales: low halves
            zc2 = bits_half2(__byte_perm(m0, m1, 0x7632));  // zeros: high halves
        }
#pragma unroll
        for (int k = 0; k < 4; ++k) {
            // code of coordinate 8 k + j7 of the block: bit VB (8 k + j7); the 8 codes of
            // one k lie in words wb, wb + 1 (a compile-time pair)
            const int base = VB * 8 * k;
            const int wb = base >> 5;
            const int sh = base - 32 * wb + VB * it.j7;
            auto code = [&](int u) -> uint32_t {
                if (base - 32 * wb + VB * 8 <= 32) return (w[u][wb] >> sh) & M;
                const uint64_t win = static_cast<uint64_t>(w[u][wb]) |
                                     (static_cast<uint64_t>(w[u][wb + 1 < VB ? wb + 1 : wb]) << 32);
                return static_cast<uint32_t>(win >> sh) & M;
            };
            const uint32_t c0 = code(u0), c1 = code(u1);
            uint32_t v;
            if (C.vmse) {
                v = half2_bits(__hmul2(bits_half2(lds32(vlut + 4 * (c0 | (c1 << VB)))), sc2));
            } else {
                const uint32_t x = c0 | (c1 << 16) | 0x64006400u;  // (1024 + c0, 1024 + c1) in fp16
                const __half2 cf = __hsub2(bits_half2(x), bits_half2(0x64006400u));
                v = half2_bits(__hfma2(cf, sc2, zc2));
            }
            row[k][pr] = v;
        }
    }
#pragma unroll
    for (int k = 0; k < 4; ++k) {
        const int j = 32 * it.jb + 8 * k + it.j7;
        sts128(vt + umma::core_offset(j, 8 * it.tc, kTok), make_uint4(row[k][0], row[k][1], row[k][2], row[k][3]));
    }
}

__global__ void __launch_bounds__(kThreads, 1) prefill_tc_kernel(const Codec C, const PageGeom PG, const DecodeArgs A)
{
    extern __shared__ __align__(128) unsigned char smem[];
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int G = A.Hq / A.Hkv;
    const int qpc = A.qpc;
    const int nqt = (A.Tq + qpc - 1) / qpc;
    const int split = blockIdx.x, kvh = blockIdx.y, b = blockIdx.z / nqt, qt = blockIdx.z % nqt;
    const int P = PG.P, pshift = __ffs(P) - 1;
    const int ppt = kTok >> pshift;             // pages per tile
    const bool qjl = C.qjl != 0;
    const int kb = C.k_bits, vb = C.v_bits;
    const int gshift = __ffs(C.group) - 1;

    int L = A.seq_lens[b];
    if (L < 0) L = 0;
    if (L > A.max_blocks * P) {
        if (split == 0 && kvh == 0 && qt == 0 && tid == 0) atomicOr(C.status, TQ_DEVERR_SEQ_RANGE);
        L = A.max_blocks * P;
    }
    const int q0 = qt * qpc;
    const int ncol = min(qpc, A.Tq - q0) * G;
    const size_t rows_total = static_cast<size_t>(A.B) * A.Tq * A.Hq;
    auto col_row = [&](int c) -> size_t {
        return (static_cast<size_t>(b) * A.Tq + q0 + c / G) * A.Hq + static_cast<size_t>(kvh) * G + c % G;
    };
    auto col_lim = [&](int c) -> int { return max(0, L - A.Tq + q0 + c / G + 1); };
    const int Lmax = col_lim(ncol - 1);
    const int npages = (Lmax + P - 1) >> pshift;
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
    const int ntiles = (pg1 - pg0 + ppt - 1) / ppt;
    const uint32_t raw_bytes = raw_stage_bytes(PG);
    const uint32_t page_bytes = static_cast<uint32_t>(PG.k_page + PG.v_page);

    uint64_t *mbar = reinterpret_cast<uint64_t *>(smem + kMbarOff);
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(smem + kMiscOff);
    volatile int *abort_flag = reinterpret_cast<volatile int *>(smem + kMiscOff + 4);
    int *page_ok = reinterpret_cast<int *>(smem + kPageOkOff);
    float *tok_a = reinterpret_cast<float *>(smem + kTokOff);
    uint32_t *tok_ok = reinterpret_cast<uint32_t *>(smem + kOkOff);

    // ---- set-up: tensor memory, tables, barriers --------------------------------
    if (warp == kMmaWarp) umma::tmem_alloc(tmem_slot, kTmCols);
    {
        // entry e (two codes) in lut_copies(kb) copies at (e * copies + copy): lane l reads
        // copy l % copies, so 3-bit lookups never share a bank pair within a half warp
        uint2 *lut = reinterpret_cast<uint2 *>(smem + kLutOff);
        const int M = (1 << kb) - 1, cp = lut_copies(kb);
        for (int x = tid; x < (1 << (2 * kb)) * cp; x += kThreads) {
            const int e = x / cp;
            __half h0, l0, h1, l1;
            split_half(kKScale * C.centroids[e & M], h0, l0);
            split_half(kKScale * C.centroids[e >> kb], h1, l1);
            lut[x] = make_uint2(half2_bits(__halves2half2(h0, h1)), half2_bits(__halves2half2(l0, l1)));
        }
        if (C.vmse) {  // value centroid pairs: fp16(lambda c) of two tokens' codes
            uint32_t *vlut = reinterpret_cast<uint32_t *>(smem + kVlutOff);
            const int VM = (1 << vb) - 1;
            for (int e = tid; e < (1 << (2 * vb)); e += kThreads)
                vlut[e] = half2_bits(__floats2half2_rn(C.vcentroids[e & VM] * C.vlut_scale,
                                                       C.vcentroids[e >> vb] * C.vlut_scale));
        }
    }
    if (tid == 0) {
        for (int i = 0; i < kRaw; ++i) {
            umma::mbar_init(&mbar[kBarRaw + i], ppt);
            umma::mbar_init(&mbar[kBarRawFree + i], kProdWarps);
        }
        for (int i = 0; i < kOps; ++i) {
            umma::mbar_init(&mbar[kBarOpFull + i], kProdWarps);
            umma::mbar_init(&mbar[kBarOpFree + i], 1);
        }
        for (int i = 0; i < 2; ++i) {
            umma::mbar_init(&mbar[kBarSFull + i], 1);
            umma::mbar_init(&mbar[kBarSFree + i], kSoftWarps);
        }
        umma::mbar_init(&mbar[kBarPFull], kSoftWarps);
        umma::mbar_init(&mbar[kBarPvDone], 1);
        umma::mbar_init(&mbar[kBarMmaDone], 1);
        *abort_flag = 0;
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    }
    umma::fence_before_sync();
    __syncthreads();
    umma::fence_after_sync();
    const uint32_t tbase = *tmem_slot;

    // bounded wait: gives up on the CTA's abort flag or after the wait limit (then
    // raising the flag and the status bit); a zero limit tests once
    auto wait_bar = [&](int i, uint32_t par) -> bool {
        uint64_t *mb = &mbar[i];
        if (C.wait_limit <= 0) {
            if (umma::mbar_test_wait(mb, par)) return true;
        } else {
            const long long t0 = clock64();
            for (;;) {
                if (umma::mbar_try_wait(mb, par)) return true;
                if (*abort_flag) return false;
                if (clock64() - t0 > C.wait_limit) break;
            }
        }
        if (!*abort_flag) {
            *abort_flag = 1;
            atomicOr(C.status, TQ_DEVERR_TIMEOUT);
        }
        return false;
    };

    // page copies of tile i into stage i % kRaw, by lanes q < ppt of the loader warp
    // block id of this lane's page of tile i (-1 past the split); read a tile ahead of its
    // issue so that the global load's latency is not paid on the producers' path
    auto fetch_blk = [&](int i) -> int {
        const int pg = pg0 + i * ppt + lane;
        return (i < ntiles && pg < pg1) ? A.block_table[static_cast<int64_t>(b) * A.max_blocks + pg] : -1;
    };
    auto issue = [&](int i, int blk) {
        const int r = i % kRaw, q = lane;
        const int pg = pg0 + i * ppt + q;
        int ok = 0;
        if (pg < pg1) {
            ok = (blk >= 0 && blk < A.num_blocks);
            if (!ok) atomicOr(C.status, TQ_DEVERR_BLOCK_RANGE);
        }
        page_ok[r * 4 + q] = ok;
        const uint32_t mb = smem_addr(&mbar[kBarRaw + r]);
        asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(mb), "r"(ok ? page_bytes : 0u)
                     : "memory");
        if (ok) {
            const size_t rec = static_cast<size_t>(blk) * A.Hkv + kvh;
            const uint32_t kd = smem_addr(smem + kRawOff + r * raw_bytes + q * page_bytes);
            const uint32_t vd = kd + static_cast<uint32_t>(PG.k_page);
            asm volatile("cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];"
                         ::"r"(kd), "l"(A.k_cache + rec * PG.k_page), "r"(static_cast<uint32_t>(PG.k_page)), "r"(mb)
                         : "memory");
            asm volatile("cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];"
                         ::"r"(vd), "l"(A.v_cache + rec * PG.v_page), "r"(static_cast<uint32_t>(PG.v_page)), "r"(mb)
                         : "memory");
        }
    };

    // column state of the softmax threads
    const int col = tid;  // warps 0-3
    const bool colv = (warp < kSoftWarps) && col < ncol;
    float fc = 0.f;       // 2^-(e + 8): the column's scale of S
    const uint32_t lane_base = tbase + (static_cast<uint32_t>(32 * (warp & 3)) << 16);

    if (warp < kSoftWarps) {
        // ---- query operands into tensor memory: q' = 2^e q_rot as fp16 high + low
        // parts, q's = 2^e R q_s, with max(|q_rot|, |q_s|) 2^e in [2^14, 2^15) ----
        const float *qr = A.ws.qrot + col_row(colv ? col : 0) * D;
        const float *qsr = A.ws.qs + col_row(colv ? col : 0) * D;
        float mx = 0.f;
        if (colv) {
            for (int j = 0; j < D; j += 4) {
                const float4 v = *reinterpret_cast<const float4 *>(qr + j);
                mx = fmaxf(mx, fmaxf(fmaxf(fabsf(v.x), fabsf(v.y)), fmaxf(fabsf(v.z), fabsf(v.w))));
                if (qjl) {
                    const float4 w = *reinterpret_cast<const float4 *>(qsr + j);
                    mx = fmaxf(mx, fmaxf(fmaxf(fabsf(w.x), fabsf(w.y)), fmaxf(fabsf(w.z), fabsf(w.w))));
                }
            }
        }
        float sc = 0.f;
        if (colv && mx > 0.f && mx <= 3.0e38f) {
            // mx < 2^ex with ex from the exponent field (subnormal maxima count as 2^-100)
            int ex = static_cast<int>((__float_as_uint(mx) >> 23) & 0xffu) - 126;
            if (ex < -100) ex = -100;
            const int e = 15 - ex;  // -113 <= e <= 115
            sc = pow2f(e);
            fc = pow2f(-(e + 8));
        }
#pragma unroll 1
        for (int ch = 0; ch < 4; ++ch) {  // 32 coordinates = 16 columns of each operand
            uint32_t h[16], l[16], s[16];
#pragma unroll
            for (int m = 0; m < 16; ++m) {
                const int j = 32 * ch + 2 * m;
                float x0 = 0.f, x1 = 0.f, y0 = 0.f, y1 = 0.f;
                if (colv) {
                    const float2 v = *reinterpret_cast<const float2 *>(qr + j);
                    x0 = v.x * sc;
                    x1 = v.y * sc;
                    if (qjl) {  // 2^e R q_s, R = sqrt(pi/2) / sqrt(d)
                        const float2 w = *reinterpret_cast<const float2 *>(qsr + j);
                        y0 = w.x * sc * kQjlR;
                        y1 = w.y * sc * kQjlR;
                    }
                }
                __half h0, l0, h1, l1;
                split_half(x0, h0, l0);
                split_half(x1, h1, l1);
                h[m] = half2_bits(__halves2half2(h0, h1));
                l[m] = half2_bits(__halves2half2(l0, l1));
                s[m] = half2_bits(__floats2half2_rn(y0, y1));
            }
            umma::st16(lane_base + kTmQh + 16 * ch, h);
            umma::st16(lane_base + kTmQl + 16 * ch, l);
            umma::st16(lane_base + kTmQs + 16 * ch, s);
        }
        umma::wait_st();
        umma::fence_before_sync();
    }
    __syncthreads();  // query operands in tensor memory
    umma::fence_after_sync();

    bool aborted = false;
    if (warp >= kSoftWarps && warp < kMmaWarp) {
        // ================= producers: page copies and operand decode =================
        const int pt = tid - kSoftWarps * 32;
        const float afac = A.sm_scale * rsqrtf(static_cast<float>(D)) * kLog2e;
        const uint32_t sbase = smem_addr(smem);
        const uint32_t lut = sbase + kLutOff + 8 * (lane & (lut_copies(kb) - 1));  // this lane's table copy
        const uint32_t vlut = sbase + kVlutOff;
        for (int i = 0; i < ntiles; ++i) {
            const int r = i % kRaw, s = i % kOps;
            bool ok = wait_bar(kBarRaw + r, (i / kRaw) & 1);
            if (ok && i >= kOps) ok = wait_bar(kBarOpFree + s, ((i - kOps) / kOps) & 1);
            if (!__all_sync(0xffffffffu, ok)) {  // the lanes poll separately: decide as a warp
                aborted = true;
                break;
            }

            const unsigned char *raw = smem + kRawOff + r * raw_bytes;
            const int *pok = page_ok + r * 4;
            const uint32_t raw_s = sbase + kRawOff + r * raw_bytes;
            const uint32_t pok_s = sbase + kPageOkOff + 16 * r;
            const uint32_t kh = sbase + s * kOpBytes;
            const uint32_t kl = kh + kTileBytes;
            const uint32_t ksg = kl + kTileBytes;
            const uint32_t vt = ksg + kTileBytes;
            const int pos0 = (pg0 + i * ppt) * P;  // sequence position of the tile's token 0

            // ---- token factors and the valid-page mask (tokens 0..63: warps 4 and 5) ----
            if (pt < kTok) {
                const int t = pt, q = t >> pshift, o = t & (P - 1);
                const bool tv = pok[q] != 0;
                const unsigned char *kp = raw + q * page_bytes;
                const float n = tv ? bf16_to_float(*reinterpret_cast<const uint16_t *>(kp + PG.k_norm_off + 2 * o)) : 0.f;
                tok_a[s * kTok + t] = n * afac;
                const uint32_t m = __ballot_sync(0xffffffffu, tv);
                if (lane == 0) tok_ok[s * 2 + (t >> 5)] = m;
            }
            // ---- keys: item (token t, 8-coordinate chunk c); the 8 lanes of a store phase
            // write the 8 rows of one core matrix ----
            {
                const KeyItem ki{raw_s, pok_s, page_bytes, pshift, P, pt, static_cast<uint32_t>(PG.k_sign_off),
                                 static_cast<uint32_t>(PG.k_gamma_off)};
                if (kb == 2) decode_keys<2>(ki, lut, kh, kl, ksg);
                else if (kb == 3) decode_keys<3>(ki, lut, kh, kl, ksg);
                else decode_keys<4>(ki, lut, kh, kl, ksg);
            }
            // ---- values: item (32-coordinate block jb, token chunk tc, row j7): coordinates
            // 32 jb + 8 k + j7 (k = 0..3) of tokens 8 tc .. 8 tc + 7, one 16-byte core-matrix
            // row (8 tokens of one coordinate) per k; the 8 lanes of a store phase (j7 = 0..7)
            // write the 8 rows of one core matrix ----
            {
                // the four 8-lane groups of a warp take the four coordinate blocks of the same
                // tokens: their code and scale loads fall in different banks
                const ValueItem vi{raw_s, pok_s, page_bytes, pos0, L, pshift, P, gshift, pt & 7, pt >> 5, (pt >> 3) & 3};
                if (vb == 2) decode_values<2>(C, PG, vi, vlut, vt);
                else if (vb == 3) decode_values<3>(C, PG, vi, vlut, vt);
                else decode_values<4>(C, PG, vi, vlut, vt);
            }
            umma::fence_proxy_async();
            warp_arrive(&mbar[kBarRawFree + r]);  // the page stage may be refilled
            warp_arrive(&mbar[kBarOpFull + s]);
        }
    } else if (warp == kLoadWarp) {
        // ================= page copies: lanes q < ppt, a stage refilled as soon as the
        // producers are done with it; block ids read before the wait =================
        int issued = 0;
        for (int i = 0; i < ntiles; ++i) {
            const int r = i % kRaw;
            const int blk = (lane < ppt) ? fetch_blk(i) : -1;
            bool ok = true;
            if (i >= kRaw) ok = __all_sync(0xffffffffu, wait_bar(kBarRawFree + r, ((i - kRaw) / kRaw) & 1));
            if (!ok) {
                aborted = true;
                break;
            }
            if (lane < ppt) issue(i, blk);
            issued = i + 1;
        }
        // copies still in flight must land before the CTA exits: the last issue of each stage
        if (aborted && lane < ppt) {
            for (int t = max(0, issued - kRaw); t < issued; ++t) {
                const long long t0 = clock64();
                while (!umma::mbar_try_wait(&mbar[kBarRaw + t % kRaw], (t / kRaw) & 1) && clock64() - t0 < kDrainLimit) {
                }
            }
        }
    } else if (warp == kMmaWarp) {
        // ================= MMA issue (lane 0) =================
        if (lane == 0) {
            const uint32_t id_s = umma::idesc_f16(kCols, kTok);
            const uint32_t id_o = umma::idesc_f16(kCols, D);
            const uint32_t sbase = smem_addr(smem);
            // K-major core-matrix descriptors: key tiles 64 x 128 (LBO 128, SBO 2048),
            // the value tile 128 x 64 (LBO 128, SBO 1024); a 16-wide k-step adds 256 bytes
            auto desc = [&](uint32_t addr, uint32_t sbo) { return umma::make_desc(addr, 128, sbo); };
            auto pv = [&](int j) {  // O += P V of tile j
                const int s = j % kOps;
                const uint32_t vaddr = sbase + s * kOpBytes + 3 * kTileBytes;
#pragma unroll
                for (int k = 0; k < kTok / 16; ++k) {
                    const uint64_t dv = desc(vaddr + 256 * k, 1024);
                    umma::mma_f16_tmem_a(tbase + kTmO, tbase + kTmP + 8 * k, static_cast<uint32_t>(dv),
                                         static_cast<uint32_t>(dv >> 32), id_o, (j > 0 || k > 0) ? 1 : 0);
                }
                umma::commit(&mbar[kBarPvDone]);
                umma::commit(&mbar[kBarOpFree + s]);
            };
            auto scores = [&](int j) {  // S = Q' K'^T (+ QJL) of tile j into score buffer j % 2
                const int s = j % kOps;
                const uint32_t kaddr = sbase + s * kOpBytes;
                const uint32_t d_s = tbase + kTmS + 64 * (j & 1);
#pragma unroll
                for (int k = 0; k < D / 16; ++k) {
                    const uint64_t dh = desc(kaddr + 256 * k, 2048);
                    const uint64_t dl = desc(kaddr + kTileBytes + 256 * k, 2048);
                    umma::mma_f16_tmem_a(d_s, tbase + kTmQh + 8 * k, static_cast<uint32_t>(dh),
                                         static_cast<uint32_t>(dh >> 32), id_s, k > 0 ? 1 : 0);
                    umma::mma_f16_tmem_a(d_s, tbase + kTmQh + 8 * k, static_cast<uint32_t>(dl),
                                         static_cast<uint32_t>(dl >> 32), id_s, 1);
                    umma::mma_f16_tmem_a(d_s, tbase + kTmQl + 8 * k, static_cast<uint32_t>(dh),
                                         static_cast<uint32_t>(dh >> 32), id_s, 1);
                    if (qjl) {
                        const uint64_t dg = desc(kaddr + 2 * kTileBytes + 256 * k, 2048);
                        umma::mma_f16_tmem_a(d_s, tbase + kTmQs + 8 * k, static_cast<uint32_t>(dg),
                                             static_cast<uint32_t>(dg >> 32), id_s, 1);
                    }
                }
                umma::commit(&mbar[kBarSFull + (j & 1)]);
            };
            // issue in the order the hand-offs complete: P.V of tile npv as soon as its P
            // is in tensor memory (that frees an operand stage for the producers), the
            // scores of tile ns as soon as its operands are decoded and its score buffer
            // has been read; give up after the wait limit without progress
            int ns = 0, npv = 0;
            long long t_last = clock64();
            while (npv < ntiles) {
                if (npv < ns && umma::mbar_test_wait(&mbar[kBarPFull], npv & 1)) {
                    umma::fence_after_sync();
                    pv(npv++);
                    t_last = clock64();
                    continue;
                }
                if (ns < ntiles && umma::mbar_test_wait(&mbar[kBarOpFull + ns % kOps], (ns / kOps) & 1) &&
                    (ns < 2 || umma::mbar_test_wait(&mbar[kBarSFree + (ns & 1)], ((ns - 2) >> 1) & 1))) {
                    umma::fence_after_sync();
                    scores(ns++);
                    t_last = clock64();
                    continue;
                }
                if (*abort_flag) {
                    aborted = true;
                    break;
                }
                if (C.wait_limit <= 0 || clock64() - t_last > C.wait_limit) {
                    *abort_flag = 1;
                    atomicOr(C.status, TQ_DEVERR_TIMEOUT);
                    aborted = true;
                    break;
                }
            }
            // every MMA issued must be done before tensor memory is freed
            umma::commit(&mbar[kBarMmaDone]);
            const long long t0 = clock64();
            while (!umma::mbar_try_wait(&mbar[kBarMmaDone], 0) && clock64() - t0 < kDrainLimit) {
            }
        }
    } else {
        // ================= softmax: one thread per column =================
        const int lim = colv ? col_lim(col) : 0;
        float m_run = -INFINITY, l_run = 0.f;
        int i = 0;
        for (; i < ntiles; ++i) {
            const int s = i & 1, s3 = i % kOps;
            const bool ok = __all_sync(0xffffffffu, wait_bar(kBarSFull + s, (i >> 1) & 1));
            if (!ok) {
                aborted = true;
                break;
            }
            umma::fence_after_sync();
            float y[kTok];
            tm_ld64(lane_base + kTmS + 64 * s, y);
            umma::fence_before_sync();
            warp_arrive(&mbar[kBarSFree + s]);
            // scores (in units of 2^(e + 8) before fc), masked: a token counts if its page
            // is valid and its position is below the column's causal limit
            const float4 *ta4 = reinterpret_cast<const float4 *>(tok_a + s3 * kTok);
            const uint32_t ok0 = tok_ok[2 * s3], ok1 = tok_ok[2 * s3 + 1];
            const int rem = lim - (pg0 + i * ppt) * P;
            float mx4[4] = {-INFINITY, -INFINITY, -INFINITY, -INFINITY};
            if (rem >= kTok && (ok0 & ok1) == 0xffffffffu) {  // the whole tile is visible
#pragma unroll
                for (int t4 = 0; t4 < kTok / 4; ++t4) {
                    const float4 a4 = ta4[t4];
                    y[4 * t4] *= a4.x;
                    y[4 * t4 + 1] *= a4.y;
                    y[4 * t4 + 2] *= a4.z;
                    y[4 * t4 + 3] *= a4.w;
#pragma unroll
                    for (int e = 0; e < 4; ++e) mx4[e] = fmaxf(mx4[e], y[4 * t4 + e]);
                }
            } else {
#pragma unroll
                for (int t4 = 0; t4 < kTok / 4; ++t4) {
                    const float4 a4 = ta4[t4];
                    const float av[4] = {a4.x, a4.y, a4.z, a4.w};
#pragma unroll
                    for (int e = 0; e < 4; ++e) {
                        const int t = 4 * t4 + e;
                        const bool keep = ((t < 32 ? ok0 >> t : ok1 >> (t - 32)) & 1u) && t < rem;
                        y[t] = keep ? y[t] * av[e] : -INFINITY;
                        mx4[e] = fmaxf(mx4[e], y[t]);
                    }
                }
            }
            const float ymax = fmaxf(fmaxf(mx4[0], mx4[1]), fmaxf(mx4[2], mx4[3]));
            const float m_tile = ymax * fc;  // log2 units (fc > 0)
            if (i >= 1) {
                const bool ok2 = __all_sync(0xffffffffu, wait_bar(kBarPvDone, (i - 1) & 1));
                if (!ok2) {
                    aborted = true;
                    break;
                }
                umma::fence_after_sync();
            }
            // lazy rescale: keep a stale maximum while the tile's stays within 2^8 of it
            const float m_new = fmaxf(m_run, m_tile);
            const bool need = (m_run != -INFINITY) && (m_new > m_run + kLazy);
            if (m_run == -INFINITY) m_run = m_new;  // O's row holds zeros so far
            if (__any_sync(0xffffffffu, need)) {
                const float al = need ? fast_exp2(m_run - m_new) : 1.f;
#pragma unroll 1
                for (int ch = 0; ch < D / 32; ++ch) {
                    float o[32];
                    uint32_t u[32];
                    umma::ld32(lane_base + kTmO + 32 * ch, o);
#pragma unroll
                    for (int m = 0; m < 32; ++m) u[m] = __float_as_uint(o[m] * al);
                    tm_st32(lane_base + kTmO + 32 * ch, u);
                }
                umma::wait_st();
                if (need) {
                    l_run *= al;
                    m_run = m_new;
                }
            }
            // P = 2^(x - m) as fp16 pairs
            uint32_t pp[32];
            float ls = 0.f;
            const float negm = -m_run;
            const bool live = m_run != -INFINITY;
#pragma unroll
            for (int m = 0; m < 32; ++m) {
                float p0 = 0.f, p1 = 0.f;
                if (live) {
                    p0 = fast_exp2(fmaf(y[2 * m], fc, negm));
                    p1 = fast_exp2(fmaf(y[2 * m + 1], fc, negm));
                }
                const __half2 h = __floats2half2_rn(p0, p1);
                ls += p0 + p1;
                pp[m] = half2_bits(h);
            }
            l_run += ls;
            tm_st32(lane_base + kTmP, pp);
            umma::wait_st();
            umma::fence_before_sync();
            warp_arrive(&mbar[kBarPFull]);
        }
        if (!aborted) {
            const bool ok = __all_sync(0xffffffffu, wait_bar(kBarPvDone, (ntiles - 1) & 1));
            if (!ok) aborted = true;
        }
        if (!aborted) {
            umma::fence_after_sync();
            const size_t rr = col_row(colv ? col : 0);
#pragma unroll 1
            for (int ch = 0; ch < D / 32; ++ch) {
                float o[32];
                umma::ld32(lane_base + kTmO + 32 * ch, o);
                if (colv) {
                    float4 *dst = reinterpret_cast<float4 *>(acc_base + rr * D + 32 * ch);
#pragma unroll
                    for (int m = 0; m < 8; ++m) dst[m] = make_float4(o[4 * m], o[4 * m + 1], o[4 * m + 2], o[4 * m + 3]);
                }
            }
            if (colv) {
                ml_base[2 * rr] = m_run;
                ml_base[2 * rr + 1] = l_run;
            }
        }
    }

    // ---- teardown ----
    umma::fence_before_sync();
    __syncthreads();
    umma::fence_after_sync();
    if (*abort_flag && warp < kSoftWarps && colv) {  // a wait gave up: this split contributes nothing
        ml_base[2 * col_row(col)] = -INFINITY;
        ml_base[2 * col_row(col) + 1] = 0.f;
    }
    if (warp == kMmaWarp) umma::tmem_dealloc(tbase, kTmCols);
}

}  // namespace pftc

size_t prefill_tc_smem_bytes(const PageGeom &pg) { return pftc::smem_bytes(pg); }

cudaError_t launch_prefill_tc(const Codec &c, const PageGeom &pg, const DecodeArgs &a, cudaStream_t st)
{
    const size_t smem = pftc::smem_bytes(pg);
    cudaError_t e = ensure_smem_attr(reinterpret_cast<const void *>(pftc::prefill_tc_kernel), smem);
    if (e != cudaSuccess) return e;
    dim3 grid(a.splits, a.Hkv, a.B * ((a.Tq + a.qpc - 1) / a.qpc));
    pftc::prefill_tc_kernel<<<grid, pftc::kThreads, smem, st>>>(c, pg, a);
    return cudaGetLastError();
}

}  // namespace tq
