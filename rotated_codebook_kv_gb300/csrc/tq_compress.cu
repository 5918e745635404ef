// tq_compress.cu -- fused key + value compression into the paged cache.
//
// Keys (turbo-attn, "How it works", steps 1-3; 0xsero/turboquant, "Compression
// Pipeline"; brightcoding blog, "Example 4": normalize -> rotate -> Lloyd-Max
// quantize -> pack bits):
//   n = ||k|| (stored bf16), z = sqrt(d) Pi k / n, code_j = #{i : t_i <= z_j},
//   and when k_bits <= 3 the residual r = z - c[code] (N(0,1) units) gives
//   sigma_i = [ (S r)_i >= 0 ] and gamma = ||r|| / sqrt(d) (stored bf16).
// Values (0xsero/turboquant, "Value Compression"): per group of `group`
//   channels, scale = fp16((max - min) / (2^b - 1)), zero = fp16(min), and
//   code = #{m < 2^b - 1 : x - zero >= (m + 1/2) scale} (round half up).
// One call compresses K and V of the same tokens (brightcoding blog, "Key
// Features": compress_kv takes both).  Its launches (launch_compress, at the end):
// head dim 128 with QJL keys the fused tensor-core kernel (tq_compress_tc.cu);
// without QJL that kernel's keys-only form and the value kernel; head dim 256 the
// Hadamard streaming kernel below (4-bit keys, values fused) or the general kernel
// below on the keys alone and the value kernel; with MSE-coded values the keys-only
// pass twice, on the keys and on the values coded like keys.
//
// Numerics.  The fast path rotates and projects in fp32.  A code whose fp32 z
// lies within kCodeGuard of a threshold, or a sign whose |p| lies within
// kSignGuard * ||r|| of zero, sends the whole row through an exact path:
// compensated (double-fp32) dot products with exact products and fp64 for the
// O(d) tail, so that codes and signs equal the exactly-rounded decisions up to
// the fp32 rounding of the Pi / S tables (about 1e-7 in z units).
#include <cuda_runtime.h>

#include "tq_device.cuh"
#include "tq_internal.h"

namespace tq {
namespace {

constexpr int kThreads = 256;
constexpr int kWarps = kThreads / 32;
constexpr int kRowsPerBlock = 32;
constexpr float kCodeGuard = 1e-5f;  // z units
constexpr float kSignGuard = 2e-5f;  // |p| / ||r||

// FUSED: dense rotation without QJL, codes decided in the rotation's epilogue; the
// fp32 row buffers kf and yb are never touched then and take no space.
template <int D, bool FUSED>
struct CompressSmem {
    static constexpr int TM = kRowsPerBlock;
    static constexpr int kCodeStride = D + 4;
    static constexpr int kRS = D + 8;                          // fp32 row stride (8 rows of an MMA fragment: 8 bank groups)
    static constexpr size_t kKf = FUSED ? 0 : sizeof(float) * TM * kRS;  // keys, later S r
    static constexpr size_t kYb = FUSED ? 0 : sizeof(float) * TM * kRS;  // Pi k, later r
    static constexpr size_t kCodes = ((TM * kCodeStride + 15) / 16) * 16;
    static constexpr size_t kScratch = sizeof(double) * kWarps * D;
    static constexpr size_t kKa = sizeof(__half) * TM * (D + 8);  // fp16 keys for the tensor-core rotation
    static constexpr size_t kBytes = kKf + kYb + kCodes + kScratch + kKa;
};

constexpr int kStreamWarps = 8;
constexpr float kRoundMagic = 12582912.f;  // 1.5 * 2^23: adding it rounds to an integer
constexpr uint32_t kRoundBits = 0x4B400000u;

template <int E>
__device__ __forceinline__ void unpack_bf16(const uint32_t (&w)[E / 2], float (&x)[E])
{
#pragma unroll
    for (int i = 0; i < E / 2; ++i) {
        x[2 * i] = __uint_as_float(w[i] << 16);
        x[2 * i + 1] = __uint_as_float(w[i] & 0xffff0000u);
    }
}

// Codes of the lane's E values of one group shared by lpg lanes:
// code = clamp(floor((x - zero) / scale + 1/2), 0, 2^VB - 1) with the group's fp16
// scale = (max - min) / (2^VB - 1) and zero = min.  The rounding is one fused
// multiply-add; a quotient within 4 ulps (2^-14) of a boundary n - 1/2 is
// re-decided exactly (x - zero as an exact float pair against (n - 1/2) scale,
// which is exact in fp32).  Groups whose zero is not their minimum exactly
// (outside the fp16 normal range) or whose scale is subnormal decide every
// element that way, with clamping.  Returns (scale | zero << 16) as fp16 bits.
template <int E, int VB>
__device__ __forceinline__ uint32_t quantize_values_lane(const float (&x)[E], int lpg, uint32_t &codes)
{
    constexpr int L = (1 << VB) - 1;
    float mn = x[0], mx = x[0];
#pragma unroll
    for (int m = 1; m < E; ++m) {
        mn = fminf(mn, x[m]);
        mx = fmaxf(mx, x[m]);
    }
    for (int o = lpg >> 1; o > 0; o >>= 1) {
        mn = fminf(mn, __shfl_xor_sync(0xffffffffu, mn, o));
        mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, o));
    }
    float dh, de;
    two_sum(mx, -mn, dh, de);
    // (max - min) / L with L in {3, 7, 15}: exact in fp32 or a non-terminating binary
    // fraction, so rounding to fp32 first never lands on an fp16 midpoint; dh * (1/L)
    // is within 2 ulps of dh / L, safe unless near a midpoint or below fp16 normals
    const float qm = dh * (1.f / static_cast<float>(L));
    const uint32_t qlow = __float_as_uint(qm) & 0x1FFFu;
    const bool qsafe = de == 0.f && qm >= 6.103515625e-05f && (qlow + 4u - 0x1000u) > 8u;
    __half s16;
    if (qsafe) s16 = __float2half_rn(qm);
    else if (de == 0.f) s16 = __float2half_rn(__fdiv_rn(dh, static_cast<float>(L)));
    else s16 = __double2half((static_cast<double>(mx) - static_cast<double>(mn)) / L);
    const __half z16 = __float2half_rn(mn);
    const float sv = __half2float(s16), zv = __half2float(z16);
    float inv = 0.f;
    if (sv != 0.f) asm("rcp.approx.ftz.f32 %0, %1;" : "=f"(inv) : "f"(sv));
    const bool exact_all = zv != mn || (sv != 0.f && sv < 6.103515625e-05f);
    codes = 0u;
    if (!exact_all) {
        // every element's guess first, then one branch for the rare near-ties, so that
        // the elements' chains are not split by a branch each
        uint32_t qq[E], tb[E], tie = 0u;
#pragma unroll
        for (int m = 0; m < E; ++m) {
            const float dx = x[m] - zv;
            qq[m] = __float_as_uint(fmaf(dx, inv, kRoundMagic)) - kRoundBits;
            tb[m] = __float_as_uint(fmaf(dx, inv, 192.5f + 4.f / 65536.f));
            tie |= ((tb[m] & 0xFFF8u) == 0u) ? (1u << m) : 0u;
        }
        if (tie) {
#pragma unroll
            for (int m = 0; m < E; ++m)
                if ((tie >> m) & 1u) {
                    const uint32_t n = (tb[m] >> 16) & 0x1Fu;
                    const float b = fmaf(static_cast<float>(n), sv, -0.5f * sv);
                    float a, ea;
                    two_sum(x[m], -zv, a, ea);
                    qq[m] = (__fadd_rn(__fsub_rn(a, b), ea) >= 0.f) ? n : n - 1u;
                }
        }
#pragma unroll
        for (int m = 0; m < E; ++m) codes |= qq[m] << (VB * m);
        return static_cast<uint32_t>(__half_as_ushort(s16)) | (static_cast<uint32_t>(__half_as_ushort(z16)) << 16);
    }
#pragma unroll
    for (int m = 0; m < E; ++m) {
        int qi = 0;
        if (sv != 0.f) {
            float a, ea;
            two_sum(x[m], -zv, a, ea);
            qi = static_cast<int>(fminf(fmaxf(floorf(fmaf(x[m] - zv, inv, 0.5f)), 0.f), static_cast<float>(L)));
            while (qi < L && __fadd_rn(__fsub_rn(a, (qi + 0.5f) * sv), ea) >= 0.f) ++qi;
            while (qi > 0 && !(__fadd_rn(__fsub_rn(a, (qi - 0.5f) * sv), ea) >= 0.f)) --qi;
        }
        codes |= static_cast<uint32_t>(qi) << (VB * m);
    }
    return static_cast<uint32_t>(__half_as_ushort(s16)) | (static_cast<uint32_t>(__half_as_ushort(z16)) << 16);
}

// Stores the lane's nbytes (2, 3 or 4) code bytes at p (aligned to nbytes when 2 or 4).
__device__ __forceinline__ void store_code_bytes(uint8_t *p, uint32_t w, int nbytes)
{
    if (nbytes == 4) *reinterpret_cast<uint32_t *>(p) = w;
    else if (nbytes == 2) *reinterpret_cast<uint16_t *>(p) = static_cast<uint16_t>(w);
    else {
        p[0] = static_cast<uint8_t>(w);
        p[1] = static_cast<uint8_t>(w >> 8);
        p[2] = static_cast<uint8_t>(w >> 16);
    }
}

// The B words of the LSB-first bitstream of 32 B-bit codes held one per byte (bit 7
// clear) at c (4-byte aligned): 4 codes per 32-bit load, then shifts.
template <int B>
__device__ __forceinline__ void pack32_codes(const uint8_t *c, uint32_t (&w)[B])
{
    uint32_t x[8];
#pragma unroll
    for (int i = 0; i < 8; ++i) x[i] = *reinterpret_cast<const uint32_t *>(c + 4 * i);
    if constexpr (B == 4) {
        // bytes 0 and 2 of x | x >> 4 hold codes (0, 1) and (2, 3) as nibble pairs
#pragma unroll
        for (int j = 0; j < 4; ++j)
            w[j] = __byte_perm(x[2 * j] | (x[2 * j] >> 4), x[2 * j + 1] | (x[2 * j + 1] >> 4), 0x6420);
    } else if constexpr (B == 2) {
#pragma unroll
        for (int j = 0; j < 2; ++j) {
            uint32_t v = 0u;
#pragma unroll
            for (int i = 0; i < 4; ++i) {
                const uint32_t t = x[4 * j + i] | (x[4 * j + i] >> 6);  // bits 0-3: codes 0, 1; 16-19: codes 2, 3
                v |= ((t & 0xFu) | ((t >> 12) & 0xF0u)) << (8 * i);
            }
            w[j] = v;
        }
    } else {
        static_assert(B == 3, "code widths 2, 3 and 4");
        // four codes -> one 12-bit chunk; chunk k sits at bit 12 k of the 96-bit stream
        uint32_t t[8];
#pragma unroll
        for (int i = 0; i < 8; ++i)
            t[i] = (x[i] & 7u) | ((x[i] >> 5) & 0x38u) | ((x[i] >> 10) & 0x1C0u) | ((x[i] >> 15) & 0xE00u);
        const uint64_t lo = static_cast<uint64_t>(t[0]) | (static_cast<uint64_t>(t[1]) << 12) |
                            (static_cast<uint64_t>(t[2]) << 24) | (static_cast<uint64_t>(t[3]) << 36) |
                            (static_cast<uint64_t>(t[4]) << 48) | (static_cast<uint64_t>(t[5]) << 60);
        w[0] = static_cast<uint32_t>(lo);
        w[1] = static_cast<uint32_t>(lo >> 32);
        w[2] = (t[5] >> 4) | (t[6] << 8) | (t[7] << 20);
    }
}

// The B-bit code words of a CTA's TM rows (codes one per byte, row stride cs) stored
// at each row's slot of its page, all threads of the CTA over rows x groups of 32
// codes (B words each); rows without a slot are skipped and zero rows (flag 2) store
// zeros.
template <int D, int TM, int B>
__device__ __forceinline__ void store_code_words_b(const uint8_t *codes, int cs, const int64_t *dst, const int *off,
                                                   const int *flag, uint8_t *pool, int64_t page_bytes, int code_bytes)
{
    constexpr int NG = D / 32;
    for (int e = threadIdx.x; e < TM * NG; e += blockDim.x) {
        const int row = e / NG, g = e % NG;
        const int64_t d = dst[row];
        if (d < 0) continue;
        uint32_t w[B];
        pack32_codes<B>(codes + row * cs + 32 * g, w);
        const bool zero = flag[row] == 2;
        uint32_t *out = reinterpret_cast<uint32_t *>(pool + d * page_bytes + static_cast<int64_t>(off[row]) * code_bytes) +
                        B * g;
#pragma unroll
        for (int j = 0; j < B; ++j) out[j] = zero ? 0u : w[j];
    }
}

template <int D, int TM>
__device__ __forceinline__ void store_code_words(const uint8_t *codes, int cs, int b, const int64_t *dst,
                                                 const int *off, const int *flag, uint8_t *pool, int64_t page_bytes,
                                                 int code_bytes)
{
    if (b == 2) store_code_words_b<D, TM, 2>(codes, cs, dst, off, flag, pool, page_bytes, code_bytes);
    else if (b == 3) store_code_words_b<D, TM, 3>(codes, cs, dst, off, flag, pool, page_bytes, code_bytes);
    else store_code_words_b<D, TM, 4>(codes, cs, dst, off, flag, pool, page_bytes, code_bytes);
}

// Dense rotation of TM rows on the tensor cores (mma.sync m16n8k16, fp16 in,
// fp32 accumulate): Y = K' (Pi 2^10)^T with K' the keys scaled by a power of two
// per row so that they are exact in fp16 (staged in ka, row stride D + 8 halves so
// that ldmatrix rows fall in different banks), and Pi 2^10 as fp16 high and low
// parts (~22 significant bits) in a fragment-ordered image read from L2:
// [n-tile][k-step][lane] = (high b0, high b1, low b0, low b1).  Warp w computes the
// output columns [D/8 w, D/8 (w + 1)) of both 16-row m-tiles; Y[row] is written to
// Yo scaled back by ysc[row].
__device__ __forceinline__ void mma16816_f16(float (&c)[4], uint32_t a0, uint32_t a1, uint32_t a2, uint32_t a3,
                                             uint32_t b0, uint32_t b1)
{
    asm volatile("mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
                 "{%0,%1,%2,%3};"
                 : "+f"(c[0]), "+f"(c[1]), "+f"(c[2]), "+f"(c[3])
                 : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}

template <int D, int TM>
__device__ __forceinline__ void mma_rows(const uint4 *__restrict__ pi_frag, const __half *ka, const float *ysc,
                                         float *Yo)
{
    constexpr int KS = D / 16, NPW = D / 64, MTS = TM / 16, KA = D + 8;
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const int r = lane >> 2, q = lane & 3;
    float acc[MTS][NPW][4];
#pragma unroll
    for (int m = 0; m < MTS; ++m)
#pragma unroll
        for (int n = 0; n < NPW; ++n) acc[m][n][0] = acc[m][n][1] = acc[m][n][2] = acc[m][n][3] = 0.f;
    const uint32_t kab = static_cast<uint32_t>(__cvta_generic_to_shared(ka));
#pragma unroll 2
    for (int s = 0; s < KS; ++s) {
        uint4 bf[NPW];
#pragma unroll
        for (int n = 0; n < NPW; ++n) bf[n] = __ldg(pi_frag + ((warp * NPW + n) * KS + s) * 32 + lane);
#pragma unroll
        for (int m = 0; m < MTS; ++m) {
            uint32_t a0, a1, a2, a3;
            const uint32_t addr = kab + 2u * ((16 * m + (lane & 15)) * KA + 16 * s + 8 * (lane >> 4));
            asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0,%1,%2,%3}, [%4];"
                         : "=r"(a0), "=r"(a1), "=r"(a2), "=r"(a3) : "r"(addr));
#pragma unroll
            for (int n = 0; n < NPW; ++n) {
                mma16816_f16(acc[m][n], a0, a1, a2, a3, bf[n].z, bf[n].w);  // low parts first
                mma16816_f16(acc[m][n], a0, a1, a2, a3, bf[n].x, bf[n].y);
            }
        }
    }
#pragma unroll
    for (int m = 0; m < MTS; ++m) {
        const int row = 16 * m + r;
        const float s0 = ysc[row], s1 = ysc[row + 8];
#pragma unroll
        for (int n = 0; n < NPW; ++n) {
            const int col = 8 * (warp * NPW + n) + 2 * q;
            *reinterpret_cast<float2 *>(Yo + row * (D + 8) + col) = make_float2(acc[m][n][0] * s0, acc[m][n][1] * s0);
            *reinterpret_cast<float2 *>(Yo + (row + 8) * (D + 8) + col) =
                make_float2(acc[m][n][2] * s1, acc[m][n][3] * s1);
        }
    }
}

// The same product for an fp32 input given as fp16 high (ka) and low (kl) parts of
// the rows times a power of two, against W 2^12 in high / low fragments: three MMAs
// per step (high x low, low x high, high x high), ~22 significant bits.  Used for the
// QJL projection p = S r of the residuals; Y[row] is written scaled by ysc[row].
template <int D, int TM>
__device__ __forceinline__ void mma_rows3(const uint4 *__restrict__ frag, const __half *ka, const __half *kl,
                                          const float *ysc, float *Yo)
{
    constexpr int KS = D / 16, NPW = D / 64, MTS = TM / 16, KA = D + 8;
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const int r = lane >> 2, q = lane & 3;
    float acc[MTS][NPW][4];
#pragma unroll
    for (int m = 0; m < MTS; ++m)
#pragma unroll
        for (int n = 0; n < NPW; ++n) acc[m][n][0] = acc[m][n][1] = acc[m][n][2] = acc[m][n][3] = 0.f;
    const uint32_t kab = static_cast<uint32_t>(__cvta_generic_to_shared(ka));
    const uint32_t klb = static_cast<uint32_t>(__cvta_generic_to_shared(kl));
#pragma unroll 2
    for (int s = 0; s < KS; ++s) {
        uint4 bf[NPW];
#pragma unroll
        for (int n = 0; n < NPW; ++n) bf[n] = __ldg(frag + ((warp * NPW + n) * KS + s) * 32 + lane);
#pragma unroll
        for (int m = 0; m < MTS; ++m) {
            uint32_t a0, a1, a2, a3, l0, l1, l2, l3;
            const uint32_t off = 2u * ((16 * m + (lane & 15)) * KA + 16 * s + 8 * (lane >> 4));
            asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0,%1,%2,%3}, [%4];"
                         : "=r"(a0), "=r"(a1), "=r"(a2), "=r"(a3) : "r"(kab + off));
            asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0,%1,%2,%3}, [%4];"
                         : "=r"(l0), "=r"(l1), "=r"(l2), "=r"(l3) : "r"(klb + off));
#pragma unroll
            for (int n = 0; n < NPW; ++n) {
                mma16816_f16(acc[m][n], a0, a1, a2, a3, bf[n].z, bf[n].w);  // small products first
                mma16816_f16(acc[m][n], l0, l1, l2, l3, bf[n].x, bf[n].y);
                mma16816_f16(acc[m][n], a0, a1, a2, a3, bf[n].x, bf[n].y);
            }
        }
    }
#pragma unroll
    for (int m = 0; m < MTS; ++m) {
        const int row = 16 * m + r;
        const float s0 = ysc[row], s1 = ysc[row + 8];
#pragma unroll
        for (int n = 0; n < NPW; ++n) {
            const int col = 8 * (warp * NPW + n) + 2 * q;
            *reinterpret_cast<float2 *>(Yo + row * (D + 8) + col) = make_float2(acc[m][n][0] * s0, acc[m][n][1] * s0);
            *reinterpret_cast<float2 *>(Yo + (row + 8) * (D + 8) + col) =
                make_float2(acc[m][n][2] * s1, acc[m][n][3] * s1);
        }
    }
}

// Codes by a table of 64 bins on u = z / 8 + 1/2 (z in [-4, 4]; outside it the end
// bins, which hold no threshold), each bin widened by 1/64 on both sides so that a
// threshold within the guard band of any z of the bin is the bin's own.  Entry
// [bin][copy] = {that threshold or +inf, 2^23 + number of thresholds below the
// widened bin}, in kBinCopies copies (lane l reads copy l % kBinCopies).  A bin that
// would hold two thresholds makes the build report failure (the codes then take the
// binary search); the Lloyd-Max thresholds are >= 0.25 apart, wider than a bin.
constexpr int kBinCopies = 8;
constexpr float kBinScale = 8064.f;  // 63 bins * 128: round(u * 8064) / 128 is the bin

__device__ __forceinline__ bool build_code_bins(float2 *bins, const float *thr, int nthr)
{
    bool bad = false;
    for (int e = threadIdx.x; e < 64 * kBinCopies; e += blockDim.x) {
        const float b = static_cast<float>(e / kBinCopies);
        const float lo = 8.f * (128.f * b - 0.5f) / kBinScale - 4.f - 1.f / 64.f;
        const float hi = 8.f * (128.f * b + 127.5f) / kBinScale - 4.f + 1.f / 64.f;
        int below = 0, idx = -1, hits = 0;
        for (int t = 0; t < nthr; ++t) {
            const float th = thr[t];
            if (th < lo) ++below;
            else if (th <= hi) { idx = t; ++hits; }
        }
        bins[e] = make_float2(idx >= 0 ? thr[idx] : INFINITY, __uint_as_float(0x4B000000u + below));
        bad |= hits > 1;
    }
    return bad;
}

// code = number of thresholds <= z; near: a threshold lies within kCodeGuard of z
__device__ __forceinline__ int bin_code(float z, const unsigned char *binb, bool &near)
{
    const float u = __saturatef(fmaf(z, 0.125f, 0.5f));
    const uint32_t a = (__float_as_uint(fmaf(u, kBinScale, kRoundMagic)) & 0x1F80u) >> 1;  // bin * 64 bytes
    const float2 e = *reinterpret_cast<const float2 *>(binb + a);
    const float dz = z - e.x;
    near = fabsf(dz) < kCodeGuard;
    return static_cast<int>(__float_as_uint(e.y) - 0x4B000000u) + (dz >= 0.f ? 1 : 0);
}

// The epilogue of the dense rotation without QJL: z = (Pi k)_j sqrt(d) / n from the
// accumulators (rounded as the stored rotation would be: y = acc ysc, then z = y
// scale), the code from the bin table (BINS) or by binary search, codes inside the
// guard band marked (bit 7) and their row flagged 3, zero keys (flag 2) coded 0.
// All of a lane's 32 codes are decided before any is stored, so that the table
// lookups are not ordered behind the stores; each pair of adjacent columns is one
// 16-bit store.
template <bool BINS, int D, int TM>
__device__ __forceinline__ void codes_from_acc(const float (&acc)[TM / 16][D / 64][4], const float *ysc,
                                               const float *zsc, int *flag, const unsigned char *__restrict__ binb,
                                               const float *__restrict__ thr, int kb, uint8_t *codes, int cs)
{
    constexpr int NPW = D / 64, MTS = TM / 16;
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const int r = lane >> 2, q = lane & 3;
    uint32_t pair[MTS][2][NPW];
    bool marked[MTS][2];
#pragma unroll
    for (int m = 0; m < MTS; ++m)
#pragma unroll
        for (int h2 = 0; h2 < 2; ++h2) {
            const int row = 16 * m + r + 8 * h2;
            const float ys = ysc[row], zs = zsc[row];
            const int fl = flag[row];
            marked[m][h2] = false;
#pragma unroll
            for (int n = 0; n < NPW; ++n) {
                uint32_t pr = 0u;
#pragma unroll
                for (int e = 0; e < 2; ++e) {
                    const float z = (acc[m][n][2 * h2 + e] * ys) * zs;
                    bool near;
                    int code;
                    if constexpr (BINS) {
                        code = bin_code(z, binb, near);
                    } else {
                        code = 0;
                        for (int step = 1 << (kb - 1); step > 0; step >>= 1)
                            if (thr[code + step] <= z) code += step;
                        near = fminf(z - thr[code], thr[code + 1] - z) < kCodeGuard;
                    }
                    const bool mark = (fl == 0 || fl == 3) && near;
                    marked[m][h2] |= mark;
                    pr |= static_cast<uint32_t>((fl == 2 ? 0 : code) | (mark ? 0x80 : 0)) << (8 * e);
                }
                pair[m][h2][n] = pr;
            }
        }
#pragma unroll
    for (int m = 0; m < MTS; ++m)
#pragma unroll
        for (int h2 = 0; h2 < 2; ++h2) {
            const int row = 16 * m + r + 8 * h2;
#pragma unroll
            for (int n = 0; n < NPW; ++n)
                *reinterpret_cast<uint16_t *>(codes + row * cs + 8 * (warp * NPW + n) + 2 * q) =
                    static_cast<uint16_t>(pair[m][h2][n]);
            if (marked[m][h2]) flag[row] = 3;
        }
}

// The dense rotation with the codes decided in the epilogue (codes_from_acc), for
// keys without QJL: no residual is needed, so Pi k never goes to shared memory.
template <int D, int TM>
__device__ __forceinline__ void mma_rows_codes(const uint4 *__restrict__ pi_frag, const __half *ka, const float *ysc,
                                               const float *zsc, int *flag, const unsigned char *binb, bool binbad,
                                               const float *thr, int kb, uint8_t *codes, int cs)
{
    constexpr int KS = D / 16, NPW = D / 64, MTS = TM / 16, KA = D + 8;
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    float acc[MTS][NPW][4];
#pragma unroll
    for (int m = 0; m < MTS; ++m)
#pragma unroll
        for (int n = 0; n < NPW; ++n) acc[m][n][0] = acc[m][n][1] = acc[m][n][2] = acc[m][n][3] = 0.f;
    const uint32_t kab = static_cast<uint32_t>(__cvta_generic_to_shared(ka));
    // B fragments one k-step ahead; all low-part MMAs of a step before the high parts,
    // so that the two products into one accumulator are MTS * NPW issues apart
    uint4 bf[NPW];
#pragma unroll
    for (int n = 0; n < NPW; ++n) bf[n] = __ldg(pi_frag + ((warp * NPW + n) * KS) * 32 + lane);
#pragma unroll 2
    for (int s = 0; s < KS; ++s) {
        uint4 bn[NPW];
        const int sn = s + 1 < KS ? s + 1 : s;
#pragma unroll
        for (int n = 0; n < NPW; ++n) bn[n] = __ldg(pi_frag + ((warp * NPW + n) * KS + sn) * 32 + lane);
        uint32_t a[MTS][4];
#pragma unroll
        for (int m = 0; m < MTS; ++m) {
            const uint32_t addr = kab + 2u * ((16 * m + (lane & 15)) * KA + 16 * s + 8 * (lane >> 4));
            asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0,%1,%2,%3}, [%4];"
                         : "=r"(a[m][0]), "=r"(a[m][1]), "=r"(a[m][2]), "=r"(a[m][3]) : "r"(addr));
        }
#pragma unroll
        for (int m = 0; m < MTS; ++m)
#pragma unroll
            for (int n = 0; n < NPW; ++n)  // low parts first
                mma16816_f16(acc[m][n], a[m][0], a[m][1], a[m][2], a[m][3], bf[n].z, bf[n].w);
#pragma unroll
        for (int m = 0; m < MTS; ++m)
#pragma unroll
            for (int n = 0; n < NPW; ++n)
                mma16816_f16(acc[m][n], a[m][0], a[m][1], a[m][2], a[m][3], bf[n].x, bf[n].y);
#pragma unroll
        for (int n = 0; n < NPW; ++n) bf[n] = bn[n];
    }
    if (!binbad) codes_from_acc<true, D, TM>(acc, ysc, zsc, flag, binb, thr, kb, codes, cs);
    else codes_from_acc<false, D, TM>(acc, ysc, zsc, flag, binb, thr, kb, codes, cs);
}

// Hadamard rotation of TM rows (turbo-attn, "How it works", step 1):
// Y[row] = H (s * X[row]) / sqrt(D) with H the Sylvester Hadamard matrix, by the
// fast Walsh-Hadamard butterfly.  One warp per row; lane l holds the E = D / 32
// consecutive elements E l .. E l + E - 1, so the first log2(E) stages stay in
// registers and the last five pair lanes l and l ^ h by shuffles.  Every stage
// is a sum or a difference of two fp32 values (the bf16 keys enter exactly).
template <int D, int TM>
__device__ __forceinline__ void fwht_rows(const float *__restrict__ hsign, const float *X, float *Y)
{
    constexpr int E = D / 32;
    const float inv = static_cast<float>(1.0 / __dsqrt_rn(static_cast<double>(D)));
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    float sg[E];
#pragma unroll
    for (int m = 0; m < E; ++m) sg[m] = __ldg(hsign + E * lane + m);
    for (int row = warp; row < TM; row += kWarps) {
        float x[E];
#pragma unroll
        for (int m = 0; m < E; m += 4) {
            const float4 v = *reinterpret_cast<const float4 *>(X + row * (D + 8) + E * lane + m);
            x[m] = v.x * sg[m];
            x[m + 1] = v.y * sg[m + 1];
            x[m + 2] = v.z * sg[m + 2];
            x[m + 3] = v.w * sg[m + 3];
        }
#pragma unroll
        for (int h = 1; h < E; h <<= 1)
#pragma unroll
            for (int m = 0; m < E; ++m)
                if (!(m & h)) {
                    const float a = x[m], b = x[m + h];
                    x[m] = a + b;
                    x[m + h] = a - b;
                }
#pragma unroll
        for (int h = 1; h < 32; h <<= 1) {
            const bool upper = (lane & h) != 0;
#pragma unroll
            for (int m = 0; m < E; ++m) {
                const float y = __shfl_xor_sync(0xffffffffu, x[m], h);
                x[m] = upper ? (y - x[m]) : (x[m] + y);
            }
        }
#pragma unroll
        for (int m = 0; m < E; m += 4)
            *reinterpret_cast<float4 *>(Y + row * (D + 8) + E * lane + m) =
                make_float4(x[m] * inv, x[m + 1] * inv, x[m + 2] * inv, x[m + 3] * inv);
    }
}

// Exact path for one row, run by one warp, against the codebook (thr, cent,
// bits): a key row (with QJL when qjl) or a value row coded like keys.  Writes
// the row's codes, its QJL projections (sign-exact) into p_out, and the bf16
// norm / gamma.
template <int D>
__device__ void precise_key_row(const Codec &C, const uint16_t *__restrict__ src, uint8_t *codes, float *p_out,
                                double *scratch, uint16_t *n16, uint16_t *g16, const float *thr, const float *cent,
                                int bits, bool qjl)
{
    constexpr int E = D / 32;
    const int lane = threadIdx.x & 31;
    float kx[E];
    float mx = 0.f;
#pragma unroll
    for (int m = 0; m < E; ++m) {
        kx[m] = bf16_to_float(src[lane + 32 * m]);
        mx = fmaxf(mx, fabsf(kx[m]));
    }
    mx = warp_max(mx);
    if (mx == 0.f) {  // zero key: caller writes an all-zero record
        return;
    }
    // Exact power-of-two scaling keeps squares away from underflow/overflow.
    int ex;
    frexpf(mx, &ex);
    const float sc = ldexpf(1.f, -ex);
    float s = 0.f, c = 0.f;
    float *kw = reinterpret_cast<float *>(scratch);
#pragma unroll
    for (int m = 0; m < E; ++m) {
        kx[m] *= sc;
        dot2_step(s, c, kx[m], kx[m]);
        kw[lane + 32 * m] = kx[m];
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
        const float s2 = __shfl_xor_sync(0xffffffffu, s, o);
        const float c2 = __shfl_xor_sync(0xffffffffu, c, o);
        float t, e;
        two_sum(s, s2, t, e);
        s = t;
        c = __fadd_rn(c, __fadd_rn(c2, e));
    }
    const double n_sc = sqrt(static_cast<double>(s) + static_cast<double>(c));
    __syncwarp();
    // the lane's E compensated sums are independent chains; with the inner loop
    // unrolled many row reads of Pi^T are in flight at once
    float yh[E], yl[E];
#pragma unroll
    for (int m = 0; m < E; ++m) yh[m] = yl[m] = 0.f;
#pragma unroll 4
    for (int j = 0; j < D; ++j) {
        const float kj = kw[j];
#pragma unroll
        for (int m = 0; m < E; ++m) dot2_step(yh[m], yl[m], __ldg(C.PiT + j * D + lane + 32 * m), kj);
    }
    __syncwarp();
    const double zscale = sqrt(static_cast<double>(D)) / n_sc;
    const int nthr = (1 << bits) - 1;
    double rr = 0.0;
#pragma unroll
    for (int m = 0; m < E; ++m) {
        const int i = lane + 32 * m;
        const double z = (static_cast<double>(yh[m]) + static_cast<double>(yl[m])) * zscale;
        int code = 0;
        for (int t = 0; t < nthr; ++t) code += (static_cast<double>(thr[t]) <= z);
        codes[i] = static_cast<uint8_t>(code);
        const double r = z - static_cast<double>(cent[code]);
        scratch[i] = r;
        rr += r * r;
    }
    rr = warp_sum(rr);
    if (lane == 0) {
        *n16 = double_to_bf16_bits(ldexp(n_sc, ex));
        if (qjl) *g16 = double_to_bf16_bits(sqrt(rr) / sqrt(static_cast<double>(D)));
    }
    __syncwarp();
    if (!qjl) return;
    float ps[E], pc[E];
#pragma unroll
    for (int m = 0; m < E; ++m) ps[m] = pc[m] = 0.f;
#pragma unroll 4
    for (int j = 0; j < D; ++j) {
        const double rj = scratch[j];
        const float rh = static_cast<float>(rj);
        const float rl = static_cast<float>(rj - static_cast<double>(rh));
#pragma unroll
        for (int m = 0; m < E; ++m) {
            const float sv = __ldg(C.ST + j * D + lane + 32 * m);
            dot2_step(ps[m], pc[m], sv, rh);
            pc[m] = __fmaf_rn(sv, rl, pc[m]);
        }
    }
#pragma unroll
    for (int m = 0; m < E; ++m) p_out[lane + 32 * m] = __fadd_rn(ps[m], pc[m]);
    __syncwarp();
}

// Re-decides the marked codes of one row exactly, by one warp: the row's codes in
// `codes` carry 0x80 where the fast z fell inside the guard band of a threshold;
// for each such coordinate z_j = sqrt(d) (Pi_j . k) / ||k|| is recomputed with
// compensated (double-fp32) sums of exact products and the code re-taken against
// the thresholds (thr, nthr).  The row must have a normal range (no power-of-two
// scaling is needed for its squares).  Returns whether any code changed (the same
// in every lane).  O(d) per marked coordinate, instead of the O(d^2) of a whole row.
template <int D>
__device__ __noinline__ bool refine_marked_codes(const float *__restrict__ Pi, const uint16_t *__restrict__ src,
                                                 uint8_t *codes, const float *thr, int nthr)
{
    constexpr int E = D / 32;
    const int lane = threadIdx.x & 31;
    float kx[E];
#pragma unroll
    for (int m = 0; m < E; ++m) kx[m] = bf16_to_float(src[lane + 32 * m]);
    auto warp_dd = [&](float s, float c) -> double {  // compensated warp sum, lane 0's value to all
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) {
            const float s2 = __shfl_xor_sync(0xffffffffu, s, o), c2 = __shfl_xor_sync(0xffffffffu, c, o);
            float t, e;
            two_sum(s, s2, t, e);
            s = t;
            c = __fadd_rn(c, __fadd_rn(c2, e));
        }
        s = __shfl_sync(0xffffffffu, s, 0);
        c = __shfl_sync(0xffffffffu, c, 0);
        return static_cast<double>(s) + static_cast<double>(c);
    };
    float ns = 0.f, nc = 0.f;
#pragma unroll
    for (int m = 0; m < E; ++m) dot2_step(ns, nc, kx[m], kx[m]);
    const double zscale = sqrt(static_cast<double>(D)) / sqrt(warp_dd(ns, nc));
    bool changed = false;
#pragma unroll 1
    for (int m = 0; m < E; ++m) {
        uint32_t mask = __ballot_sync(0xffffffffu, (codes[lane + 32 * m] & 0x80u) != 0);
        while (mask) {
            const int j = __ffs(mask) - 1 + 32 * m;
            mask &= mask - 1;
            float ds = 0.f, dc = 0.f;
#pragma unroll
            for (int mm = 0; mm < E; ++mm) dot2_step(ds, dc, __ldg(Pi + j * D + lane + 32 * mm), kx[mm]);
            const double z = warp_dd(ds, dc) * zscale;
            int code = 0;
            for (int t = 0; t < nthr; ++t) code += (static_cast<double>(thr[t]) <= z);
            const int old = codes[j] & 0x7F;
            changed |= code != old;
            __syncwarp();
            if (lane == 0) codes[j] = static_cast<uint8_t>(code);
            __syncwarp();
        }
    }
    return changed;
}

// Codes of TM rotated rows (yb, row stride rs; z = yb scale[row]) by the whole CTA:
// the code from the bin table (BINS) or by binary search over thr (thr[c + 1] is
// threshold c; the distance to the nearest threshold is to one of the two that
// bracket z); a code inside the guard band of a threshold is marked (bit 7) and its
// row flagged 3 (the exact pass re-decides just the marked codes); zero rows (flag
// 2) get code 0.  With RESID the residual z - centroid (0 for zero rows) replaces
// yb.  Each thread takes four elements at a time, all loaded before any store.
template <bool BINS, bool RESID, int D, int TM>
__device__ __forceinline__ void codes_and_residuals(float *yb, int rs, const float *scale, int *flag,
                                                    const unsigned char *__restrict__ binb,
                                                    const float *__restrict__ thr, const float *__restrict__ cent,
                                                    int kb, uint8_t *codes, int cs)
{
    constexpr int PER = TM * D / kThreads;
    static_assert(PER % 4 == 0, "four elements per thread at a time");
#pragma unroll 1
    for (int k0 = 0; k0 < PER; k0 += 4) {
        int row[4], col[4], fl[4], code[4];
        float z[4];
        bool near[4];
#pragma unroll
        for (int j = 0; j < 4; ++j) {
            const int e = threadIdx.x + kThreads * (k0 + j);
            row[j] = e / D;
            col[j] = e - row[j] * D;
            fl[j] = flag[row[j]];
            z[j] = yb[row[j] * rs + col[j]] * scale[row[j]];
        }
#pragma unroll
        for (int j = 0; j < 4; ++j) {
            if constexpr (BINS) {
                code[j] = bin_code(z[j], binb, near[j]);
            } else {
                int c = 0;
                for (int step = 1 << (kb - 1); step > 0; step >>= 1)
                    if (thr[c + step] <= z[j]) c += step;
                near[j] = fminf(z[j] - thr[c], thr[c + 1] - z[j]) < kCodeGuard;
                code[j] = c;
            }
            if (fl[j] == 2) code[j] = 0;
        }
        float r[4];
        if constexpr (RESID) {
#pragma unroll
            for (int j = 0; j < 4; ++j) r[j] = (fl[j] == 2) ? 0.f : z[j] - cent[code[j]];
        }
#pragma unroll
        for (int j = 0; j < 4; ++j) {
            const bool mark = (fl[j] == 0 || fl[j] == 3) && near[j];
            codes[row[j] * cs + col[j]] = static_cast<uint8_t>(code[j] | (mark ? 0x80 : 0));
            if constexpr (RESID) yb[row[j] * rs + col[j]] = r[j];
            if (mark) flag[row[j]] = 3;
        }
    }
}

template <int D, bool HAD, bool FUSED>
__global__ void __launch_bounds__(kThreads, FUSED ? 4 : 2)
compress_kernel(const Codec C, const PageGeom G, const uint16_t *__restrict__ kin, int64_t rows, int Hkv, int64_t ks,
                const int64_t *__restrict__ slots, uint8_t *__restrict__ kc, int64_t num_blocks)
{
    static_assert(!(HAD && FUSED), "the fused epilogue follows the dense rotation");
    using SM = CompressSmem<D, FUSED>;
    constexpr int TM = SM::TM;
    constexpr int CS = SM::kCodeStride;
    constexpr int RS = SM::kRS;
    extern __shared__ __align__(16) unsigned char smem_raw[];
    float *kf = reinterpret_cast<float *>(smem_raw);
    float *yb = reinterpret_cast<float *>(smem_raw + SM::kKf);
    uint8_t *codes = smem_raw + SM::kKf + SM::kYb;
    double *scratch = reinterpret_cast<double *>(smem_raw + SM::kKf + SM::kYb + SM::kCodes);
    __half *ka = reinterpret_cast<__half *>(smem_raw + SM::kKf + SM::kYb + SM::kCodes + SM::kScratch);
    __shared__ float s_ysc[TM];  // 2^-(10 + row scale): the tensor-core rotation's output back to Pi k
    __shared__ float s_scale[TM];
    __shared__ float s_rn[TM];
    __shared__ int64_t s_dst[TM];
    __shared__ int s_off[TM];
    __shared__ int s_flag[TM];  // 0 fast, 1 exact path, 2 zero key
    __shared__ uint16_t s_n16[TM], s_g16[TM];
    __shared__ float s_thr[18];   // -inf, thresholds ascending, +inf (codes by binary search)
    __shared__ float s_cent[16];
    __shared__ __align__(16) float2 s_bins[64 * kBinCopies];
    __shared__ int64_t s_tok[TM];  // token of each row

    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int64_t r0 = static_cast<int64_t>(blockIdx.x) * TM;
    // row r0 + i is token t0 + (h0 + i) / Hkv, head (h0 + i) % Hkv: one 64-bit division
    const int64_t t0 = r0 / Hkv;
    const int h0 = static_cast<int>(r0 - t0 * Hkv);
    const float sqrtd = sqrtf(static_cast<float>(D));
    const int nthr = (1 << C.k_bits) - 1;
    if (tid < 18) s_thr[tid] = tid == 0 ? -INFINITY : (tid <= nthr ? C.thresholds[tid - 1] : INFINITY);
    if (tid < 16) s_cent[tid] = C.centroids[tid];

    // the rows' slots are requested now and turned into page and offset just before
    // the rotation, so that their latency overlaps the key loads and the bin table
    int64_t slot = -1;  // rows past the end keep -1
    if (tid < TM && r0 + tid < rows) {
        const int64_t t = t0 + (h0 + tid) / Hkv;
        s_tok[tid] = t;
        slot = slots[t];
    }
    // Each warp's key rows (dense rotation: the lane's E contiguous elements) are
    // loaded now, so that their latency overlaps the slot loads and the bin table.
    constexpr int E = D / 32, RPW = TM / kWarps;
    uint32_t kraw[RPW][E / 2];
    if constexpr (!HAD) {
#pragma unroll
        for (int k = 0; k < RPW; ++k) {
            const int row = warp + kWarps * k;
#pragma unroll
            for (int i = 0; i < E / 2; ++i) kraw[k][i] = 0u;
            if (r0 + row < rows) {
                const int q = (h0 + row) / Hkv;
                const uint16_t *src = kin + (t0 + q) * ks + static_cast<int64_t>(h0 + row - q * Hkv) * D + lane * E;
                if constexpr (E == 8) {
                    const uint4 u = __ldg(reinterpret_cast<const uint4 *>(src));
                    kraw[k][0] = u.x; kraw[k][1] = u.y; kraw[k][2] = u.z; kraw[k][3] = u.w;
                } else {
                    const uint2 u = __ldg(reinterpret_cast<const uint2 *>(src));
                    kraw[k][0] = u.x; kraw[k][1] = u.y;
                }
            }
        }
    }
    constexpr bool fused = FUSED;  // launched exactly when !HAD && !C.qjl
    // the key codebook's bin table; the barrier also publishes the rows' tokens
    const unsigned char *binb = reinterpret_cast<const unsigned char *>(s_bins) + 8 * (lane % kBinCopies);
    bool binbad = __syncthreads_or(build_code_bins(s_bins, C.thresholds, nthr));
    if constexpr (HAD) {
        // ---- load key rows (bf16 -> fp32, exact) ---------------------------------
        for (int e = tid; e < TM * (D / 8); e += kThreads) {
            const int row = e / (D / 8), c8 = e - row * (D / 8);
            const int64_t r = r0 + row;
            uint4 u = make_uint4(0, 0, 0, 0);
            if (r < rows) {
                const int64_t t = s_tok[row];
                const int h = static_cast<int>(r - t * Hkv);
                u = __ldg(reinterpret_cast<const uint4 *>(kin + t * ks + static_cast<int64_t>(h) * D) + c8);
            }
            float4 lo = make_float4(bf16_to_float(u.x & 0xffffu), bf16_to_float(u.x >> 16), bf16_to_float(u.y & 0xffffu),
                                    bf16_to_float(u.y >> 16));
            float4 hi = make_float4(bf16_to_float(u.z & 0xffffu), bf16_to_float(u.z >> 16), bf16_to_float(u.w & 0xffffu),
                                    bf16_to_float(u.w >> 16));
            *reinterpret_cast<float4 *>(kf + row * RS + c8 * 8) = lo;
            *reinterpret_cast<float4 *>(kf + row * RS + c8 * 8 + 4) = hi;
        }
        __syncthreads();
    }
    // ---- norms; rows with an extreme range take the exact path; dense rotation:
    // the keys go straight from bf16 into the fp16 operand (exact after the row scale) ----
#pragma unroll
    for (int k = 0; k < RPW; ++k) {
        const int row = warp + kWarps * k;
        float x[E];  // HAD: elements lane + 32 m; dense: elements E lane + m
        if constexpr (HAD) {
#pragma unroll
            for (int m = 0; m < E; ++m) x[m] = kf[row * RS + lane + 32 * m];
        } else {
            unpack_bf16<E>(kraw[k], x);
        }
        float ss = 0.f, mx = 0.f;
#pragma unroll
        for (int m = 0; m < E; ++m) {
            ss = fmaf(x[m], x[m], ss);
            mx = fmaxf(mx, fabsf(x[m]));
        }
        ss = warp_sum(ss);
        mx = warp_max(mx);
        if (lane == 0) {
            int flag = 0;
            if (mx == 0.f) flag = 2;
            else if (!(mx >= 0x1p-30f && mx <= 0x1p30f)) flag = 1;
            const float n = sqrtf(ss);
            s_scale[row] = (flag == 0) ? sqrtd / n : 0.f;
            s_flag[row] = flag;
            s_n16[row] = float_to_bf16_bits(n);
            s_g16[row] = 0;
        }
        if constexpr (!HAD) {
            // mx = f 2^ex with f in [0.5, 1); the row times 2^(15 - ex) is exact in fp16
            const bool ok = mx >= 0x1p-30f && mx <= 0x1p30f;
            const int ex = ok ? static_cast<int>((__float_as_uint(mx) >> 23) & 0xffu) - 126 : 0;
            const float sc = ok ? __uint_as_float(static_cast<uint32_t>(127 + 15 - ex) << 23) : 0.f;
            uint32_t h2[E / 2];
#pragma unroll
            for (int i = 0; i < E / 2; ++i) {
                const __half2 h = __floats2half2_rn(x[2 * i] * sc, x[2 * i + 1] * sc);
                h2[i] = *reinterpret_cast<const uint32_t *>(&h);
            }
            if constexpr (E == 8)
                *reinterpret_cast<uint4 *>(ka + row * (D + 8) + lane * E) = make_uint4(h2[0], h2[1], h2[2], h2[3]);
            else
                *reinterpret_cast<uint2 *>(ka + row * (D + 8) + lane * E) = make_uint2(h2[0], h2[1]);
            if (lane == 0) s_ysc[row] = ok ? __uint_as_float(static_cast<uint32_t>(127 + ex - 25) << 23) : 0.f;
        }
    }
    if (tid < TM) {
        int64_t dst = -1;
        int off = 0;
        if (slot >= 0) {
            if (slot < num_blocks * G.P) {
                const int64_t blk = slot / G.P;
                off = static_cast<int>(slot - blk * G.P);
                dst = blk * Hkv + (h0 + tid) % Hkv;
            } else {
                atomicOr(C.status, TQ_DEVERR_SLOT_RANGE);
            }
        }
        s_dst[tid] = dst;  // published by the barrier after the rotation
        s_off[tid] = off;
    }
    // ---- rotation: yb = Pi k (unnormalised); without QJL the codes come straight
    // from the accumulators ---------------------------------------------------
    if constexpr (HAD) {
        fwht_rows<D, TM>(C.hsign, kf, yb);
    } else {
        __syncthreads();  // ka and s_ysc of every row are staged
        if constexpr (fused)
            mma_rows_codes<D, TM>(C.pi_frag, ka, s_ysc, s_scale, s_flag, binb, binbad, s_thr, C.k_bits, codes, CS);
        else
            mma_rows<D, TM>(C.pi_frag, ka, s_ysc, yb);
    }
    __syncthreads();
    // ---- codes, guard band, residual (the residual only for QJL) ---------------
    if constexpr (!fused) {
        if (C.qjl) {
            if (!binbad)
                codes_and_residuals<true, true, D, TM>(yb, RS, s_scale, s_flag, binb, s_thr, s_cent, C.k_bits, codes, CS);
            else
                codes_and_residuals<false, true, D, TM>(yb, RS, s_scale, s_flag, binb, s_thr, s_cent, C.k_bits, codes, CS);
        } else {
            if (!binbad)
                codes_and_residuals<true, false, D, TM>(yb, RS, s_scale, s_flag, binb, s_thr, s_cent, C.k_bits, codes, CS);
            else
                codes_and_residuals<false, false, D, TM>(yb, RS, s_scale, s_flag, binb, s_thr, s_cent, C.k_bits, codes,
                                                         CS);
        }
    }
    __syncthreads();
    // ---- QJL: p = S r, gamma, sign guard ---------------------------------------
    if (!fused && C.qjl) {
        // the residuals as fp16 high + low parts times a power of two per row (high in
        // ka, low over yb once every row is in registers), then p = S r on mma.sync
        constexpr int KA = D + 8;
        float rv[RPW][E];
#pragma unroll
        for (int k = 0; k < RPW; ++k) {
            const int row = warp + kWarps * k;
            float ss = 0.f, mx = 0.f;
#pragma unroll
            for (int m = 0; m < E; ++m) {
                rv[k][m] = yb[row * RS + lane + 32 * m];
                ss = fmaf(rv[k][m], rv[k][m], ss);
                mx = fmaxf(mx, fabsf(rv[k][m]));
            }
            ss = warp_sum(ss);
            mx = warp_max(mx);
            if (lane == 0) {
                s_rn[row] = sqrtf(ss);
                // max |r| 2^(15 - ex) in [2^14, 2^15); back by 2^(ex - 15 - 12)
                const bool ok = mx >= 0x1p-60f && mx <= 0x1p60f;
                const int ex = ok ? static_cast<int>((__float_as_uint(mx) >> 23) & 0xffu) - 126 : 0;
                s_scale[row] = ok ? __uint_as_float(static_cast<uint32_t>(127 + 15 - ex) << 23) : 0.f;
                s_ysc[row] = ok ? __uint_as_float(static_cast<uint32_t>(127 + ex - 27) << 23) : 0.f;
            }
        }
        __syncthreads();  // every residual is in registers; row scales published
        __half *klo = reinterpret_cast<__half *>(yb);
#pragma unroll
        for (int k = 0; k < RPW; ++k) {
            const int row = warp + kWarps * k;
            const float sc = s_scale[row];
#pragma unroll
            for (int m = 0; m < E; ++m) {
                const float x = rv[k][m] * sc;
                const __half h = __float2half_rn(x);
                ka[row * KA + lane + 32 * m] = h;
                klo[row * KA + lane + 32 * m] = __float2half_rn(x - __half2float(h));
            }
        }
        __syncthreads();
        mma_rows3<D, TM>(C.s_frag, ka, klo, s_ysc, kf);
        __syncthreads();
        for (int row = warp; row < TM; row += kWarps) {
            const float rn = s_rn[row];
            bool near = false;
            for (int j = lane; j < D; j += 32) near |= fabsf(kf[row * RS + j]) < kSignGuard * rn;
            near = __any_sync(0xffffffffu, near);
            if (lane == 0) {
                s_rn[row] = rn;
                s_g16[row] = float_to_bf16_bits(rn / sqrtd);
                if (near && (s_flag[row] == 0 || s_flag[row] == 3)) s_flag[row] = 1;
            }
        }
        __syncthreads();
    }
    // ---- exact path for flagged rows: marked codes re-decided one by one (a changed
    // code under QJL changes the residual: the whole row is redone), other flagged
    // rows redone entirely ------------------------------------------------------
    for (int row = warp; row < TM; row += kWarps) {
        int fl = s_flag[row];
        if ((fl != 1 && fl != 3) || s_dst[row] < 0) continue;
        const int64_t t = s_tok[row];  // a row with a slot has a token
        const int h = static_cast<int>(r0 + row - t * Hkv);
        if (fl == 3) {
            const bool changed = refine_marked_codes<D>(C.Pi, kin + t * ks + static_cast<int64_t>(h) * D,
                                                        codes + row * CS, C.thresholds, (1 << C.k_bits) - 1);
            if (!(changed && C.qjl)) continue;
        }
        precise_key_row<D>(C, kin + t * ks + static_cast<int64_t>(h) * D, codes + row * CS, kf + row * RS,
                           scratch + warp * D, &s_n16[row], &s_g16[row], C.thresholds, C.centroids, C.k_bits,
                           C.qjl != 0);
    }
    __syncthreads();
    // ---- pack and store: code words by the whole CTA, then per row its sign
    // bits, gamma and norm ------------------------------------------------------
    store_code_words<D, TM>(codes, CS, C.k_bits, s_dst, s_off, s_flag, kc, G.k_page, C.k_code_bytes);
    for (int row = warp; row < TM; row += kWarps) {
        const int64_t dst = s_dst[row];
        if (dst < 0) continue;
        const int off = s_off[row];
        const bool zero = (s_flag[row] == 2);
        uint8_t *krec = kc + dst * G.k_page;
        if (!fused && C.qjl) {
#pragma unroll
            for (int w = 0; w < D / 32; ++w) {
                uint32_t bits = __ballot_sync(0xffffffffu, kf[row * RS + 32 * w + lane] >= 0.f);
                if (zero) bits = 0u;
                if (lane == w)
                    *reinterpret_cast<uint32_t *>(krec + G.k_sign_off + static_cast<int64_t>(off) * C.k_sign_bytes +
                                                  4 * w) = bits;
            }
            if (lane == 0) *reinterpret_cast<uint16_t *>(krec + G.k_gamma_off + 2 * off) = zero ? 0 : s_g16[row];
        }
        if (lane == 0) *reinterpret_cast<uint16_t *>(krec + G.k_norm_off + 2 * off) = zero ? 0 : s_n16[row];
    }
}

// ---------------------------------------------------------------------------
// Streaming kernel for the randomized Hadamard rotation without QJL (k_bits = 4):
// one warp per token-head row, rows strided over all warps of the grid, the next
// row's key, value and slot loaded while the current one is processed.  Lane l
// holds the E = D / 32 consecutive coordinates E l .. E l + E - 1 of the key and
// of the value, so the butterfly's first log2(E) stages stay in registers, its
// last five pair lanes by shuffles, and the lane's E codes are E * b consecutive
// bits of the record (b bytes at byte offset b l).  No shared-memory staging and
// no block barrier: the kernel is a row pipeline bounded by HBM.
// ---------------------------------------------------------------------------
// The lane's 4-bit codes of one row taken again in double (rows with a code near a
// threshold or an extreme range).  Every bf16 square and every butterfly sum of
// bf16 keys is exact in double up to 2^-53 of the row's largest term, so the
// decisions are the exact ones up to the fp32 rounding of the thresholds.
// Returns the 8 codes packed LSB-first; *n16 gets the bf16 norm.
__device__ __noinline__ uint32_t stream_exact_codes(uint4 k4, const float *__restrict__ hsign, const float *s_thr,
                                                    uint16_t *n16)
{
    constexpr int E = 8;
    const int lane = threadIdx.x & 31;
    const uint32_t w[4] = {k4.x, k4.y, k4.z, k4.w};
    double xd[E];
    double ssd = 0.0;
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        xd[2 * i] = static_cast<double>(__uint_as_float(w[i] << 16));
        xd[2 * i + 1] = static_cast<double>(__uint_as_float(w[i] & 0xffff0000u));
    }
#pragma unroll
    for (int m = 0; m < E; ++m) {
        ssd = fma(xd[m], xd[m], ssd);
        xd[m] *= static_cast<double>(__ldg(hsign + E * lane + m));
    }
    ssd = warp_sum(ssd);
#pragma unroll
    for (int hh = 1; hh < E; hh <<= 1)
#pragma unroll
        for (int m = 0; m < E; ++m)
            if (!(m & hh)) {
                const double a = xd[m], b = xd[m + hh];
                xd[m] = a + b;
                xd[m + hh] = a - b;
            }
#pragma unroll
    for (int hh = 1; hh < 32; hh <<= 1) {
        const double sgn = (lane & hh) ? -1.0 : 1.0;
#pragma unroll
        for (int m = 0; m < E; ++m) xd[m] = fma(xd[m], sgn, __shfl_xor_sync(0xffffffffu, xd[m], hh));
    }
    const double nd = sqrt(ssd);
    uint32_t kw = 0u;
#pragma unroll
    for (int m = 0; m < E; ++m) {
        const double z = xd[m] / nd;
        int code = 0;
#pragma unroll
        for (int step = 8; step > 0; step >>= 1)
            if (static_cast<double>(s_thr[code + step]) <= z) code += step;
        kw |= static_cast<uint32_t>(code) << (4 * m);
    }
    *n16 = double_to_bf16_bits(nd);
    return kw;
}

// Code bins of the streaming kernel: u = sat(z / 8 + 1/2) clamps z to [-4, 4]
// (every 4-bit Lloyd-Max threshold lies inside +-2.8); adding 8064 u to
// 1.5 * 2^23 rounds to an integer whose bits 7..12 are 128 b, b = bin index, the
// byte offset of the bin; bins are 8 / 63 wide in z with 1/64 margins, so a bin
// holds at most one threshold (they are >= 0.12 apart).  Entry {threshold or
// +inf, 2^23 + number of thresholds below the bin} as two floats, in 16 copies
// side by side (lane l reads copy l % 16: the 16 lanes of a 64-bit wavefront hit
// 16 different bank pairs).
constexpr float kSBinScale = 8064.f;  // 63 bins * 128 bytes

template <int D, int VB>
__global__ void __launch_bounds__(kStreamWarps * 32, 3)
compress_stream_kernel(const Codec C, const PageGeom G, const uint16_t *__restrict__ kin,
                       const uint16_t *__restrict__ vin, int64_t rows, int Hkv, int64_t ks, int64_t vs,
                       const int64_t *__restrict__ slots, uint8_t *__restrict__ kc, uint8_t *__restrict__ vc,
                       int64_t num_blocks)
{
    constexpr int E = D / 32;  // coordinates per lane
    static_assert(E == 8, "head_dim 256: a lane's codes are whole bytes for every value width");
    __shared__ float s_thr[18];                  // -inf, thresholds ascending, +inf (exact path)
    __shared__ __align__(16) float2 s_bins[64 * 16];  // [bin][copy]
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    constexpr int nthr = 15;
    if (threadIdx.x < 18)
        s_thr[threadIdx.x] = threadIdx.x == 0 ? -INFINITY : (threadIdx.x <= nthr ? C.thresholds[threadIdx.x - 1] : INFINITY);
    for (int e = threadIdx.x; e < 64 * 16; e += blockDim.x) {
        const float b = static_cast<float>(e >> 4);
        const float lo = 8.f * (128.f * b - 0.5f) / kSBinScale - 4.f - 1.f / 64.f;
        const float hi = 8.f * (128.f * b + 127.5f) / kSBinScale - 4.f + 1.f / 64.f;
        int below = 0, idx = -1;
        for (int t = 0; t < nthr; ++t) {
            const float th = C.thresholds[t];
            if (th < lo) ++below;
            else if (th <= hi) idx = t;
        }
        s_bins[e] = make_float2(idx >= 0 ? C.thresholds[idx] : INFINITY, __uint_as_float(0x4B000000u + below));
    }
    __syncthreads();
    const unsigned char *binb = reinterpret_cast<const unsigned char *>(s_bins) + 8 * (lane & 15);
    float sg[E];
#pragma unroll
    for (int m = 0; m < E; ++m) sg[m] = __ldg(C.hsign + E * lane + m);
    const int hshift = (Hkv & (Hkv - 1)) == 0 ? __ffs(Hkv) - 1 : -1;
    const int pshift = __ffs(G.P) - 1;
    const int64_t cache_slots = num_blocks * G.P;
    const int lpg = C.group / E;  // lanes per value group: 4, 8 or 16
    const int64_t nw = static_cast<int64_t>(gridDim.x) * kStreamWarps;
    auto fetch = [&](int64_t r, uint4 &k4, uint4 &v4, int64_t &sl) {
        const int64_t t = hshift >= 0 ? (r >> hshift) : r / Hkv;
        const int64_t h = r - t * Hkv;
        k4 = ld_pinned(kin + t * ks + h * D + E * lane);
        v4 = ld_pinned(vin + t * vs + h * D + E * lane);
        sl = ld_pinned_s64(slots + t);
    };
    int64_t r = static_cast<int64_t>(blockIdx.x) * kStreamWarps + warp;
    uint4 kn = make_uint4(0u, 0u, 0u, 0u), vn = kn;
    int64_t sn = -1;
    if (r < rows) fetch(r, kn, vn, sn);
    for (; r < rows; r += nw) {
        const uint4 k4 = kn, v4 = vn;
        const int64_t slot = sn;
        if (r + nw < rows) fetch(r + nw, kn, vn, sn);  // the next row streams in while this one is worked on
        if (slot < 0) continue;
        if (slot >= cache_slots) {
            if (lane == 0) atomicOr(C.status, TQ_DEVERR_SLOT_RANGE);
            continue;
        }
        const int64_t t = hshift >= 0 ? (r >> hshift) : r / Hkv;
        const int64_t h = r - t * Hkv;
        const int64_t dst = (slot >> pshift) * Hkv + h;
        const int off = static_cast<int>(slot & (G.P - 1));
        uint8_t *krec = kc + dst * G.k_page;
        uint8_t *vrec = vc + dst * G.v_page;
        // ---- key: norm, butterfly rotation, codes -----------------------------
        float x[E];
        {
            const uint32_t w[E / 2] = {k4.x, k4.y, k4.z, k4.w};
            unpack_bf16<E>(w, x);
        }
        float ss = 0.f, mx = 0.f;
#pragma unroll
        for (int m = 0; m < E; ++m) {
            ss = fmaf(x[m], x[m], ss);
            mx = fmaxf(mx, fabsf(x[m]));
            x[m] *= sg[m];
        }
        ss = warp_sum(ss);
        mx = warp_max(mx);
        const bool zero = mx == 0.f;
        const bool extreme = !zero && !(mx >= 0x1p-30f && mx <= 0x1p30f);
#pragma unroll
        for (int hh = 1; hh < E; hh <<= 1)
#pragma unroll
            for (int m = 0; m < E; ++m)
                if (!(m & hh)) {
                    const float a = x[m], b = x[m + hh];
                    x[m] = a + b;
                    x[m + hh] = a - b;
                }
#pragma unroll
        for (int hh = 1; hh < 32; hh <<= 1) {
            // the lower lane of a pair keeps x + y, the upper y - x: one exact +-1 multiply-add
            const float sgn = (lane & hh) ? -1.f : 1.f;
#pragma unroll
            for (int m = 0; m < E; ++m) x[m] = fmaf(x[m], sgn, __shfl_xor_sync(0xffffffffu, x[m], hh));
        }
        // z_j = sqrt(d) (Pi k)_j / n = (H (s * k))_j / n
        const float n = sqrtf(ss);
        const float inv_n = zero ? 0.f : 1.f / n;
        const float zsu = inv_n * 0.125f;
        uint32_t kw = 0u;
        bool near = false;
#pragma unroll
        for (int m = 0; m < E; ++m) {
            const float u = __saturatef(fmaf(x[m], zsu, 0.5f));
            const uint32_t a = __float_as_uint(fmaf(u, kSBinScale, kRoundMagic)) & 0x1F80u;
            const float2 e = *reinterpret_cast<const float2 *>(binb + a);
            const float dz = fmaf(x[m], inv_n, -e.x);
            float up;  // 1 at or above the bin's threshold, 0 below it or without one
            asm("mul.rn.ftz.sat.f32 %0, %1, 0f7E800000;" : "=f"(up) : "f"(dz));  // dz * 2^126
            near |= fabsf(dz) < kCodeGuard;
            kw |= (__float_as_uint(e.y + up) - 0x4B000000u) << (4 * m);
        }
        uint16_t n16 = zero ? 0 : float_to_bf16_bits(n);
        if (__any_sync(0xffffffffu, extreme || (near && !zero))) kw = stream_exact_codes(k4, C.hsign, s_thr, &n16);
        if (zero) kw = 0u;
        store_code_bytes(krec + static_cast<int64_t>(off) * C.k_code_bytes + (E / 2) * lane, kw, E / 2);
        if (lane == 0) *reinterpret_cast<uint16_t *>(krec + G.k_norm_off + 2 * off) = n16;
        // ---- value: group scale / zero and codes ----------------------------------
        float v[E];
        {
            const uint32_t w[E / 2] = {v4.x, v4.y, v4.z, v4.w};
            unpack_bf16<E>(w, v);
        }
        uint32_t vw;
        const uint32_t meta = quantize_values_lane<E, VB>(v, lpg, vw);
        store_code_bytes(vrec + static_cast<int64_t>(off) * C.v_code_bytes + (E * VB / 8) * lane, vw, E * VB / 8);
        if ((lane & (lpg - 1)) == 0)
            *reinterpret_cast<uint32_t *>(vrec + G.v_meta_off + static_cast<int64_t>(off) * C.v_meta_bytes +
                                          4 * (lane / lpg)) = meta;
    }
}

template <int D, int VB>
cudaError_t launch_stream(const Codec &c, const PageGeom &pg, const uint16_t *k, const uint16_t *v, int64_t T,
                          int Hkv, int64_t ks, int64_t vs, const int64_t *slots, uint8_t *kc, uint8_t *vc,
                          int64_t num_blocks, cudaStream_t st)
{
    const int64_t rows = T * Hkv;
    int64_t blocks = (rows + kStreamWarps - 1) / kStreamWarps;
    const int64_t cap = static_cast<int64_t>(c.num_sms) * 3;  // one wave: three resident CTAs per SM
    if (blocks > cap) blocks = cap;
    compress_stream_kernel<D, VB><<<static_cast<unsigned>(blocks), kStreamWarps * 32, 0, st>>>(
        c, pg, k, v, rows, Hkv, ks, vs, slots, kc, vc, num_blocks);
    return cudaGetLastError();
}

template <int D, bool HAD, bool FUSED>
cudaError_t launch_compress_d(const Codec &c, const PageGeom &pg, const uint16_t *k, int64_t T, int Hkv, int64_t ks,
                              const int64_t *slots, uint8_t *kc, int64_t num_blocks, cudaStream_t st)
{
    const size_t smem = CompressSmem<D, FUSED>::kBytes;
    cudaError_t e = ensure_smem_attr(reinterpret_cast<const void *>(compress_kernel<D, HAD, FUSED>), smem);
    if (e != cudaSuccess) return e;
    const int64_t rows = T * Hkv;
    const int64_t blocks = (rows + kRowsPerBlock - 1) / kRowsPerBlock;
    compress_kernel<D, HAD, FUSED><<<static_cast<unsigned>(blocks), kThreads, smem, st>>>(c, pg, k, rows, Hkv, ks, slots,
                                                                                          kc, num_blocks);
    return cudaGetLastError();
}

}  // namespace

// The codec and page geometry that code MSE values as key records: an MSE value
// record is exactly a key record without QJL (codes, then a bf16 norm per token).
static void values_as_keys(const Codec &c, const PageGeom &pg, Codec &cv, PageGeom &gv)
{
    cv = c;
    cv.k_bits = c.v_bits;
    cv.qjl = 0;
    cv.k_code_bytes = c.v_code_bytes;
    cv.k_sign_bytes = 0;
    for (int i = 0; i < 16; ++i) {
        cv.centroids[i] = c.vcentroids[i];
        cv.thresholds[i] = c.vthresholds[i];
    }
    gv = pg;
    gv.k_page = pg.v_page;
    gv.k_sign_off = gv.k_norm_off = pg.v_meta_off;
    gv.k_gamma_off = pg.v_meta_off + 2LL * pg.P;  // not written without QJL
}

// Key records alone at head dim 256: the general kernel without a value input.
static cudaError_t launch_keys_256(const Codec &c, const PageGeom &pg, const uint16_t *k, int64_t T, int Hkv,
                                   int64_t ks, const int64_t *slots, uint8_t *kc, int64_t num_blocks, cudaStream_t st)
{
    if (c.rotation == 1) return launch_compress_d<256, true, false>(c, pg, k, T, Hkv, ks, slots, kc, num_blocks, st);
    return c.qjl ? launch_compress_d<256, false, false>(c, pg, k, T, Hkv, ks, slots, kc, num_blocks, st)
                 : launch_compress_d<256, false, true>(c, pg, k, T, Hkv, ks, slots, kc, num_blocks, st);
}

cudaError_t launch_compress(const Codec &c, const PageGeom &pg, const uint16_t *k, const uint16_t *v, int64_t T,
                            int Hkv, int64_t ks, int64_t vs, const int64_t *slots, uint8_t *kc, uint8_t *vc,
                            int64_t num_blocks, cudaStream_t st)
{
    if (c.vmse) {
        // values coded like keys: the keys-only pass on the keys, then on the values
        // through the value codebook in the key fields (tensor-core kernel at 128,
        // general kernel at 256)
        Codec cv;
        PageGeom gv;
        values_as_keys(c, pg, cv, gv);
        cudaError_t e = c.d == 128 ? launch_compress_tc_keys(c, pg, k, T, Hkv, ks, slots, kc, num_blocks, c.num_sms, st)
                                   : launch_keys_256(c, pg, k, T, Hkv, ks, slots, kc, num_blocks, st);
        if (e != cudaSuccess) return e;
        return c.d == 128 ? launch_compress_tc_keys(cv, gv, v, T, Hkv, vs, slots, vc, num_blocks, c.num_sms, st)
                          : launch_keys_256(cv, gv, v, T, Hkv, vs, slots, vc, num_blocks, st);
    }
    if (c.d == 128 && !c.qjl) {
        // without QJL the keys-only tensor-core pass and a streaming value kernel beat the
        // fused kernel, whose producers spend a third of its time on values; with QJL its
        // epilogue sets the pace and the fused kernel stays ahead
        cudaError_t e = launch_compress_tc_keys(c, pg, k, T, Hkv, ks, slots, kc, num_blocks, c.num_sms, st);
        if (e != cudaSuccess) return e;
        return launch_compress_values_tc(c, pg, v, T, Hkv, vs, slots, vc, num_blocks, c.num_sms, st);
    }
    if (c.d == 128) return launch_compress_tc(c, pg, k, v, T, Hkv, ks, vs, slots, kc, vc, num_blocks, c.num_sms, st);
    if (c.rotation == 1 && !c.qjl) {
        switch (c.v_bits) {
        case 2: return launch_stream<256, 2>(c, pg, k, v, T, Hkv, ks, vs, slots, kc, vc, num_blocks, st);
        case 3: return launch_stream<256, 3>(c, pg, k, v, T, Hkv, ks, vs, slots, kc, vc, num_blocks, st);
        default: return launch_stream<256, 4>(c, pg, k, v, T, Hkv, ks, vs, slots, kc, vc, num_blocks, st);
        }
    }
    // the general kernel on the keys alone, then the value kernel: its value pass is
    // ~40% of a CTA's time at 16 warps per SM, the value kernel streams them faster
    cudaError_t e = launch_keys_256(c, pg, k, T, Hkv, ks, slots, kc, num_blocks, st);
    if (e != cudaSuccess) return e;
    return launch_compress_values_tc(c, pg, v, T, Hkv, vs, slots, vc, num_blocks, c.num_sms, st);
}

}  // namespace tq
