// tq_compress_tc.cu -- key + value compression with the rotation and the QJL
// projection on the tensor cores (tcgen05, accumulators in tensor memory), d = 128.
//
// Method (turbo-attn "How it works"; 0xsero/turboquant "Compression Pipeline",
// "Value Compression"; brightcoding blog "Example 4"): see tq_compress.cu.
//
// Tile = 128 token-heads; one persistent CTA per SM, 512 threads in two roles
// that overlap consecutive tiles:
//  producers (warps 8-15)
//  1. issue every global load of the tile's keys (and the first value rows),
//     take each key's norm in fp32 (sum of exact squares) and convert it
//     exactly to fp16 after a power-of-two scale 2^e per row;
//  2. issue Y = K' (Pi 2^10)^T on the tensor cores once the epilogue has read
//     the previous Y: Pi 2^10 is split into fp16 high and low parts, two MMA
//     terms, ~22-bit operands, fp32 accumulation;
//  3. quantise the values of the tile (one lane per 32 channels), loading the
//     next rows while the current ones are quantised; the next tile is
//     prefetched into L2 by the bulk-copy engine.
//  epilogue (warps 0-7; warp w reads TMEM lane quarter w % 4, column half w / 4)
//  4. z = Y sqrt(d) / (n 2^(10+e)); a clamped bin table (64 bins in 4 copies)
//     gives, in one shared-memory load, the one threshold near z and the
//     centroids on both sides of it; residual r = z - c[code], gamma =
//     ||r|| / sqrt(d); r 2^12 is split into fp16 high / low parts and stored to
//     tensor memory as the A operand of the next MMA;
//  5. QJL: P = (R 2^12)(S 2^12)^T, three MMA terms (hi.hi, hi.lo, lo.hi) with A
//     read from tensor memory; the sign of P is the sign of S r.  The key tile in
//     shared memory is free as soon as Y is done, so step 1 of the next tile
//     overlaps steps 4-7 of this one;
//  6. decisions within a guard band of a threshold, a sign boundary or a bf16
//     rounding midpoint of gamma are re-taken exactly: a code or a sign by an
//     O(d) compensated dot product (z_j = sqrt(d) (Pi_j . k) / n,
//     p_i = sqrt(d) (M_i . k) / n - S_i . c with M = S Pi in double-fp32), and
//     a row whose code flips or whose gamma sits near a midpoint is redone
//     entirely in compensated arithmetic.  Such rows are listed in shared memory
//     and fixed by all 16 warps at the end (or by the epilogue when the list fills);
//  7. key records are written with the fast-path results first.
// Hand-offs: mbarriers "keys converted" (producers -> epilogue), "Y ready" and
// "P ready" (tensor core -> both), "Y read" (epilogue -> producers).
// Every mbarrier wait is bounded; a timeout sets TQ_DEVERR_TIMEOUT, the CTA
// stops, waits (bounded) for its tensor-core work and frees its TMEM.
#include <cuda_runtime.h>

#include "tq_device.cuh"
#include "tq_internal.h"
#include "tq_umma.cuh"

namespace tq {
namespace {

constexpr int D = 128;
constexpr int TM = 128;
constexpr int kThreads = 512;       // warps 0-7: epilogue; warps 8-15: producers
constexpr int kEpi = 256;           // epilogue threads: TMEM lane quarter (warp & 3), column half (warp >> 2)
constexpr int kProd = 256;          // producer threads: key conversion, MMA issue, values
constexpr int kPasses = TM / (8 * (kProd / 32));  // 8-row passes per producer warp and tile
constexpr int kEpiWarps = kEpi / 32;
constexpr float kCodeGuard = 1e-5f;   // z units
constexpr float kSignGuard = 2e-5f;   // |p| / ||r||
constexpr float kGammaGuard = 2e-6f;  // relative distance of gamma to a bf16 rounding midpoint

// Shared-memory map (bytes).
constexpr uint32_t kOffPiH = 0, kOffPiL = 32768, kOffSH = 65536, kOffSL = 98304;  // B operands (fp16)
constexpr uint32_t kOffTA = 131072;  // K' (fp16), the A operand of the rotation MMA
constexpr uint32_t kOffTB = 163840;  // exact path: [16 warps][d] double scratch, then the deferred-row list
// Per-row arrays are stored [item][row], so that the 32 rows of a warp use 32 banks.
constexpr uint32_t kOffCodes = 196608;               // [16][TM] u32 packed key codes
constexpr uint32_t kOffSigns = kOffCodes + TM * 64;  // [4][TM] u32 sign bits
constexpr uint32_t kOffMask = kOffSigns + TM * 16;   // [8][TM] u32: code guard mask (4), sign guard mask (4)
constexpr uint32_t kOffRow = kOffMask + TM * 32;     // [3][TM] RowInfo (tile index mod 3)
constexpr uint32_t kOffPart = kOffRow + 3 * TM * 32; // [TM][2] gsq partials, [TM][2] code flags, [TM][2] sign flags
constexpr uint32_t kOffBins = kOffPart + TM * 24;    // [64 bins][4 copies] float4 code bins (below)
constexpr int kMaxDefer = 256;                       // rows awaiting exact re-decision
constexpr uint32_t kOffDefer = kOffTB + 16 * D * 8;  // [kMaxDefer] Deferred
static_assert(kOffDefer + kMaxDefer * 64 <= kOffCodes, "deferred-row list overlaps the code words");
constexpr uint32_t kOffMisc = kOffBins + 256 * 16;   // mbarriers, TMEM slot, abort flags
constexpr uint32_t kSmemBytes = kOffMisc + 128;  // + 7 descriptor words at kOffMisc + 64
static_assert(kSmemBytes <= 232448, "shared memory map exceeds the per-block limit");

constexpr uint32_t kSBO = (D / 8) * 128;  // 2048
constexpr uint32_t kIdesc = umma::idesc_f16(128, 128);

// Code bins.  The epilogue works on z' = 2^12 z.  u = sat(z / 8 + 1/2) clamps z
// to [-4, 4] (every Lloyd-Max threshold for N(0,1) with b_k <= 4 lies inside
// +-2.5); bin b holds the u with floor(round(4032 u) / 64) = b, i.e. z in about
// [b / 7.875 - 4, (b + 1) / 7.875 - 4].  Adding 4032 u to 1.5 * 2^23 rounds to
// that integer and leaves it in the low mantissa bits, so bits 6..11 are 64 b,
// the byte offset of the bin.  Thresholds are at least 0.25 apart, so a bin
// (0.127 wide plus margins) holds at most one.  Each bin is stored in 4 copies
// side by side, lane l reading copy l % 4: of the 8 lanes that share a 128-byte
// shared-memory wavefront only lanes l and l + 4 can meet in a bank.
// Entry: {threshold (or +inf), centroid below it, centroid above minus below
// (0 without a threshold), 2^23 + code below it}, centroids and threshold times 2^12.
constexpr float kBinU = 1.f / 32768.f;    // z' / 2^15 = z / 8
constexpr float kBinScale = 4032.f;       // 63 * 64
constexpr float kRoundMagic = 12582912.f; // 1.5 * 2^23: adding it rounds to an integer
constexpr uint32_t kRoundBits = 0x4B400000u;
constexpr uint32_t kCode23Bits = 0x4B000000u;  // bits of 2^23

// A row whose decisions are re-taken exactly after its record was written with
// the fast-path results.
struct Deferred {      // 64 bytes
    int64_t r;         // token-head row of the input
    int64_t dst;       // record index (block * Hkv + head)
    int off;           // offset inside the page
    int flag;          // as RowInfo::flag
    uint32_t cmask[4]; // codes within the guard band of a threshold
    uint32_t smask[4]; // sign bits within the guard band of zero
    int pad[2];
};

struct RowInfo {     // 32 bytes per row
    int64_t dst;     // record index (block * Hkv + head) or -1
    int off;         // offset inside the page
    int flag;        // bit0 code guard, bit1 sign guard, bit2 tiny key, bit3 zero key, bit4 gamma near a bf16 midpoint
    float zscale;    // sqrt(d) / (n 2^(10+e)) applied to Y
    float rn;        // unused (the epilogue keeps ||r|| in registers); keeps the 32-byte layout
    uint32_t n16g16; // bf16 norm | bf16 gamma << 16
    int pad;
};

__device__ __forceinline__ uint32_t pack_h2(float a, float b)
{
    const __half2 h = __floats2half2_rn(a, b);
    return *reinterpret_cast<const uint32_t *>(&h);
}

// Compensated dot product of a global fp32 row with the warp's fp32 key copy, then
// combined over the warp.  Returns hi + lo as a double.
__device__ double warp_dot_df(const float *__restrict__ a, const float *kw)
{
    const int lane = threadIdx.x & 31;
    float s = 0.f, c = 0.f;
#pragma unroll
    for (int m = 0; m < D / 32; ++m) dot2_step(s, c, __ldg(a + lane + 32 * m), kw[lane + 32 * m]);
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
        const float s2 = __shfl_xor_sync(0xffffffffu, s, o), c2 = __shfl_xor_sync(0xffffffffu, c, o);
        float t, e;
        two_sum(s, s2, t, e);
        s = t;
        c = __fadd_rn(c, __fadd_rn(c2, e));
    }
    return static_cast<double>(s) + static_cast<double>(c);
}

template <int KB>
__device__ __forceinline__ uint32_t get_code(const uint32_t *w, int j)
{
    const int o = j * KB;
    const uint32_t lo = w[o >> 5];
    const uint32_t hi = ((o & 31) + KB > 32) ? w[(o >> 5) + 1] : 0u;
    return __funnelshift_r(lo, hi, o & 31) & ((1u << KB) - 1u);
}

template <int KB>
__device__ __forceinline__ void set_code(uint32_t *w, int j, uint32_t v)
{
    for (int b = 0; b < KB; ++b) {
        const int o = j * KB + b;
        const uint32_t bit = 1u << (o & 31);
        if ((v >> b) & 1u) w[o >> 5] |= bit;
        else w[o >> 5] &= ~bit;
    }
}

// The whole key row in compensated arithmetic, by one warp (see tq_compress.cu).
// Lane l owns coordinates l + 32 m (m < 4): the four compensated sums are
// independent chains and the inner loop is unrolled, so many row reads of Pi^T
// (and S^T) are in flight at once.  signs_too = false keeps the sign bits (a
// row redone only because gamma sits near a bf16 rounding midpoint).
template <int KB>
__device__ __noinline__ void exact_row(const Codec &C, const float *kw, double n_sc, uint32_t *codes, uint32_t *signs,
                                       uint32_t *n16g16, double *scratch, double n_true, bool signs_too)
{
    constexpr int E = D / 32;
    const int lane = threadIdx.x & 31;
    float yh[E], yl[E];
#pragma unroll
    for (int m = 0; m < E; ++m) yh[m] = yl[m] = 0.f;
#pragma unroll 8
    for (int j = 0; j < D; ++j) {
        const float kj = kw[j];
#pragma unroll
        for (int m = 0; m < E; ++m) dot2_step(yh[m], yl[m], __ldg(C.PiT + j * D + lane + 32 * m), kj);
    }
    __syncwarp();  // scratch aliases the key copy read above
    const double zscale = sqrt(static_cast<double>(D)) / n_sc;
    const int nthr = (1 << KB) - 1;
    double rr = 0.0;
    uint32_t cd[E];
#pragma unroll
    for (int m = 0; m < E; ++m) {
        const int i = lane + 32 * m;
        const double z = (static_cast<double>(yh[m]) + static_cast<double>(yl[m])) * zscale;
        int code = 0;
        for (int t = 0; t < nthr; ++t) code += (static_cast<double>(C.thresholds[t]) <= z);
        cd[m] = code;
        const double r = z - static_cast<double>(C.centroids[code]);
        scratch[i] = r;
        rr += r * r;
    }
    rr = warp_sum(rr);
    // rewrite the packed codes: lane-parallel over words
    __syncwarp();
    for (int w = lane; w < D * KB / 32; w += 32) codes[w] = 0u;
    __syncwarp();
#pragma unroll
    for (int m = 0; m < E; ++m) {
        const int i = lane + 32 * m;
        for (int b = 0; b < KB; ++b)
            if ((cd[m] >> b) & 1u) atomicOr(&codes[(i * KB + b) >> 5], 1u << ((i * KB + b) & 31));
    }
    const uint32_t g16 = C.qjl ? double_to_bf16_bits(sqrt(rr) / sqrt(static_cast<double>(D))) : 0u;
    if (lane == 0) *n16g16 = double_to_bf16_bits(n_true) | (g16 << 16);
    __syncwarp();
    if (!C.qjl || !signs_too) return;
    // residual as float hi + lo pairs (the inner loop then needs no fp64)
    float2 *rp = reinterpret_cast<float2 *>(scratch);
    float2 mine[E];
#pragma unroll
    for (int m = 0; m < E; ++m) {
        const double rj = scratch[lane + 32 * m];
        const float rh = static_cast<float>(rj);
        mine[m] = make_float2(rh, static_cast<float>(rj - static_cast<double>(rh)));
    }
    __syncwarp();
#pragma unroll
    for (int m = 0; m < E; ++m) rp[lane + 32 * m] = mine[m];
    __syncwarp();
    float ps[E], pc[E];
#pragma unroll
    for (int m = 0; m < E; ++m) ps[m] = pc[m] = 0.f;
#pragma unroll 8
    for (int j = 0; j < D; ++j) {
        const float2 r2 = rp[j];
#pragma unroll
        for (int m = 0; m < E; ++m) {
            const float sv = __ldg(C.ST + j * D + lane + 32 * m);
            dot2_step(ps[m], pc[m], sv, r2.x);
            pc[m] = __fmaf_rn(sv, r2.y, pc[m]);
        }
    }
#pragma unroll
    for (int m = 0; m < E; ++m) {
        const uint32_t bits = __ballot_sync(0xffffffffu, __fadd_rn(ps[m], pc[m]) >= 0.f);
        if (lane == 0) signs[m] = bits;
    }
    __syncwarp();
}

// Exact re-decision of one deferred row by one warp: the fast-path codes and
// signs are read back from its record, decisions inside a guard band are taken
// again in compensated arithmetic, and what changed is written back.
// cw (16 words), sw (4 words), n16 (1 word) and scratch (d doubles) are this
// warp's shared-memory space.
template <int KB>
__device__ __noinline__ void fix_row(const Codec &C, const PageGeom &G, const uint16_t *__restrict__ kin, int64_t ks,
                                     int Hkv, uint8_t *__restrict__ kc, const Deferred &df, uint32_t *cw, uint32_t *sw,
                                     uint32_t *n16, double *scratch)
{
    constexpr int NKW = D * KB / 32;
    const int lane = threadIdx.x & 31;
    const int nthr = (1 << KB) - 1;
    const int flg = df.flag;
    uint8_t *krec = kc + df.dst * G.k_page;
    uint32_t *cd = reinterpret_cast<uint32_t *>(krec + static_cast<int64_t>(df.off) * C.k_code_bytes);
    uint32_t *sd = reinterpret_cast<uint32_t *>(krec + G.k_sign_off + static_cast<int64_t>(df.off) * C.k_sign_bytes);
    if (lane < NKW) cw[lane] = __ldcg(cd + lane);
    if (C.qjl && lane < 4) sw[lane] = __ldcg(sd + lane);
    const int64_t t = df.r / Hkv;
    const uint16_t *src = kin + t * ks + static_cast<int64_t>(df.r - t * Hkv) * D;
    float *kw = reinterpret_cast<float *>(scratch);
    float kx[D / 32];
    float mx = 0.f;
#pragma unroll
    for (int m = 0; m < D / 32; ++m) {
        kx[m] = bf16_to_float(src[lane + 32 * m]);
        mx = fmaxf(mx, fabsf(kx[m]));
    }
    mx = warp_max(mx);
    int ex;
    frexpf(mx, &ex);
    const float sc = ldexpf(1.f, -ex);
    float s = 0.f, c = 0.f;
#pragma unroll
    for (int m = 0; m < D / 32; ++m) {
        kx[m] *= sc;
        dot2_step(s, c, kx[m], kx[m]);
        kw[lane + 32 * m] = kx[m];
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
        const float s2 = __shfl_xor_sync(0xffffffffu, s, o), c2 = __shfl_xor_sync(0xffffffffu, c, o);
        float tt, e;
        two_sum(s, s2, tt, e);
        s = tt;
        c = __fadd_rn(c, __fadd_rn(c2, e));
    }
    const double n_sc = sqrt(static_cast<double>(s) + static_cast<double>(c));
    __syncwarp();
    bool redo = (flg & 20) != 0;  // tiny key or gamma near a rounding midpoint
    bool signs_too = (flg & 6) != 0;
    if (!redo && (flg & 1)) {  // codes near a threshold
        for (int w = 0; w < 4 && !redo; ++w) {
            uint32_t m = df.cmask[w];
            while (m && !redo) {
                const int j = 32 * w + __ffs(m) - 1;
                m &= m - 1;
                const double z = warp_dot_df(C.Pi + j * D, kw) * (sqrt(static_cast<double>(D)) / n_sc);
                uint32_t code = 0;
                for (int tt = 0; tt < nthr; ++tt) code += (static_cast<double>(C.thresholds[tt]) <= z);
                if (code != get_code<KB>(cw, j)) redo = signs_too = true;  // the residual changes: redo the row
            }
        }
    }
    bool signs_changed = false;
    if (redo) {
        exact_row<KB>(C, kw, n_sc, cw, sw, n16, scratch, ldexp(n_sc, ex), signs_too);
        signs_changed = C.qjl && signs_too;
    } else if (flg & 2) {  // signs near zero: p_i = sqrt(d) (M_i . k) / n - S_i . c
        signs_changed = true;
        for (int w = 0; w < 4; ++w) {
            uint32_t m = df.smask[w];
            while (m) {
                const int i = 32 * w + __ffs(m) - 1;
                m &= m - 1;
                const double mk = warp_dot_df(C.M_hi + i * D, kw) + warp_dot_df(C.M_lo + i * D, kw);
                float sh = 0.f, scc = 0.f;
#pragma unroll
                for (int mm = 0; mm < D / 32; ++mm) {
                    const int j = lane + 32 * mm;
                    dot2_step(sh, scc, __ldg(C.S + i * D + j), C.centroids[get_code<KB>(cw, j)]);
                }
#pragma unroll
                for (int o = 16; o > 0; o >>= 1) {
                    const float s2 = __shfl_xor_sync(0xffffffffu, sh, o);
                    const float c2 = __shfl_xor_sync(0xffffffffu, scc, o);
                    float tt, e;
                    two_sum(sh, s2, tt, e);
                    sh = tt;
                    scc = __fadd_rn(scc, __fadd_rn(c2, e));
                }
                const double p = mk * (sqrt(static_cast<double>(D)) / n_sc) - (static_cast<double>(sh) + static_cast<double>(scc));
                if (lane == 0) {
                    const uint32_t bit = 1u << (i & 31);
                    sw[w] = (p >= 0.0) ? (sw[w] | bit) : (sw[w] & ~bit);
                }
                __syncwarp();
            }
        }
    }
    __syncwarp();
    if (redo) {
        if (lane < NKW) cd[lane] = cw[lane];
        if (lane == 0) {
            *reinterpret_cast<uint16_t *>(krec + G.k_norm_off + 2 * df.off) = static_cast<uint16_t>(*n16 & 0xffffu);
            if (C.qjl)
                *reinterpret_cast<uint16_t *>(krec + G.k_gamma_off + 2 * df.off) = static_cast<uint16_t>(*n16 >> 16);
        }
    }
    if (signs_changed && lane < 4) sd[lane] = sw[lane];
}

// Epilogue 1 for one (row, 32-column block cb): codes, guard mask, residual
// split into fp16 hi / lo (QJL only) stored to tensor memory as the A operand
// of the projection (hi at tR, lo at tR + 64; the caller waits for the stores),
// and the block's sum of squares of the residual.  32 columns are exactly KB
// code words.
template <int KB>
__device__ __forceinline__ float epilogue_rotation_block(unsigned char *smem, uint32_t tY, uint32_t tR, int warp, int row,
                                                         int cb, float zs, bool qjl, uint32_t *scodes,
                                                         uint32_t *smask)
{
    float y[32];
    umma::ld32(tY + (static_cast<uint32_t>(32 * (warp & 3)) << 16) + 32 * cb, y);
    const float zsu = zs * kBinU;
    const unsigned char *binb = smem + kOffBins + ((row & 3) << 4);  // this lane's copy
    // codes are summed as 2^23 + code shifted into place; the constant parts
    // (known at compile time) are subtracted at the end
    uint32_t cw[KB], bias[KB];
#pragma unroll
    for (int w = 0; w < KB; ++w) cw[w] = bias[w] = 0u;
    uint32_t cmask = 0u;
    float gsq = 0.f;
#pragma unroll
    for (int i = 0; i < 32; ++i) {
        // z' = y zs is folded into each fused multiply-add
        const float u = __saturatef(fmaf(y[i], zsu, 0.5f));
        const uint32_t a = __float_as_uint(fmaf(u, kBinScale, kRoundMagic)) & 0xFC0u;
        const float4 e = *reinterpret_cast<const float4 *>(binb + a);
        const float dz = fmaf(y[i], zs, -e.x);
        // 1 above the bin's threshold, 0 below it or without one; a dz of zero or
        // below the normal range counts as below (it is inside the guard band)
        float up;
        asm("mul.rn.ftz.sat.f32 %0, %1, 0f7E800000;" : "=f"(up) : "f"(dz));  // dz * 2^126
        if (fabsf(dz) < kCodeGuard * 4096.f) cmask |= 1u << i;
        const float r = fmaf(y[i], zs, -fmaf(up, e.z, e.y));
        gsq = fmaf(r, r, gsq);
        const uint32_t cb23 = __float_as_uint(e.w + up);  // 2^23 + code
        const int o = i * KB;  // compile-time bit offset inside the block
        cw[o >> 5] += cb23 << (o & 31);
        bias[o >> 5] += kCode23Bits << (o & 31);
        if ((o & 31) + KB > 32) cw[(o >> 5) + 1] += (cb23 - kCode23Bits) >> (32 - (o & 31));
        y[i] = r;
    }
#pragma unroll
    for (int w = 0; w < KB; ++w) scodes[(KB * cb + w) * TM + row] = cw[w] - bias[w];
    smask[cb * TM + row] = cmask;
    if (qjl) {
        uint32_t rh[16], rlo[16];
#pragma unroll
        for (int q = 0; q < 16; ++q) {
            const float a = y[2 * q], b = y[2 * q + 1];
            const __half2 hh = __floats2half2_rn(a, b);
            const float2 hf = __half22float2(hh);
            rh[q] = *reinterpret_cast<const uint32_t *>(&hh);
            rlo[q] = pack_h2(a - hf.x, b - hf.y);
        }
        const uint32_t ta = tR + (static_cast<uint32_t>(32 * (warp & 3)) << 16) + 16 * cb;
        umma::st16(ta, rh);
        umma::st16(ta + 64, rlo);
    }
    return gsq;
}

// Epilogue 2 for one (row, column half): QJL sign bits and the sign guard mask.
__device__ __forceinline__ int epilogue_signs(uint32_t tP, int warp, int row, int hf, float guard, bool zero,
                                              uint32_t *ssigns, uint32_t *smask)
{
    int flag = 0;
#pragma unroll
    for (int cb = 0; cb < 2; ++cb) {
        // sign bits shifted in from the last column to the first: bit j of neg is the
        // sign of p_j, bit j of near that of |p_j| - guard (a zero p, whose sign bit may
        // be set, lies inside the guard band and is re-decided exactly)
        uint32_t neg = 0u, near = 0u;
        float p[32];
        umma::ld32(tP + (static_cast<uint32_t>(32 * (warp & 3)) << 16) + 64 * hf + 32 * cb, p);
#pragma unroll
        for (int j = 31; j >= 0; --j) {
            neg = __funnelshift_l(__float_as_uint(p[j]), neg, 1);  // (neg << 1) | (p_j >> 31)
            near = __funnelshift_l(__float_as_uint(fabsf(p[j]) - guard), near, 1);
        }
        uint32_t bits = ~neg;
        if (zero) bits = near = 0u;
        ssigns[(2 * hf + cb) * TM + row] = bits;
        smask[(4 + 2 * hf + cb) * TM + row] = near;
        flag |= near ? 2 : 0;
    }
    return flag;
}

// Exact re-decision of 32 value codes (see quantize_values32).
template <int VB>
__device__ __noinline__ void values32_exact(const uint32_t *wd, float zv, float sv, float inv, uint32_t *cw)
{
    constexpr int L = (1 << VB) - 1;
    for (int k = 0; k < VB; ++k) cw[k] = 0u;
    for (int e = 0; e < 32; ++e) {
        const uint32_t wv = wd[e >> 1];
        const float x = (e & 1) ? __uint_as_float(wv & 0xffff0000u) : __uint_as_float(wv << 16);
        int q = 0;
        if (sv != 0.f) {
            float a, ea;
            two_sum(x, -zv, a, ea);
            q = static_cast<int>(fminf(fmaxf(floorf(fmaf(x - zv, inv, 0.5f)), 0.f), static_cast<float>(L)));
            while (q < L && __fadd_rn(__fsub_rn(a, (q + 0.5f) * sv), ea) >= 0.f) ++q;
            while (q > 0 && !(__fadd_rn(__fsub_rn(a, (q - 0.5f) * sv), ea) >= 0.f)) --q;
        }
        const int o = e * VB;
        cw[o >> 5] |= static_cast<uint32_t>(q) << (o & 31);
        if ((o & 31) + VB > 32) cw[(o >> 5) + 1] |= static_cast<uint32_t>(q) >> (32 - (o & 31));
    }
}

// Values: one lane holds 32 consecutive channels (four 16-byte words) of a row;
// lanes_per_group = g / 32 neighbouring lanes share a group.  Computes the
// group's fp16 scale and zero and the lane's 32 codes packed LSB-first into VB
// words: code = clamp(floor((x - zero) / scale + 0.5), 0, 2^VB - 1).
//
// Two fused multiply-adds per element: (x - zero) / scale + 1.5 * 2^23 rounds
// to the code in the low mantissa bits, and (x - zero) / scale + 192.5 + 2^-14
// (ulp 2^-16 in [128, 256)) has its low 16 bits below 8 exactly when the
// quotient lies within 4 ulps of a boundary n - 1/2 between codes n - 1 and n.
// Such an element is re-decided exactly: x - zero as an exact float pair
// against (n - 1/2) scale, which is exact in fp32.  A lane whose zero is not its
// min exactly (values outside the fp16 normal range) or whose scale is
// subnormal re-decides every code that way, with clamping.
template <int VB>
__device__ __forceinline__ void quantize_values32(const uint4 (&w4)[4], int lanes_per_group, uint32_t (&cw)[VB],
                                                  uint32_t &meta)
{
    constexpr int L = (1 << VB) - 1;
    const uint32_t wd[16] = {w4[0].x, w4[0].y, w4[0].z, w4[0].w, w4[1].x, w4[1].y, w4[1].z, w4[1].w,
                             w4[2].x, w4[2].y, w4[2].z, w4[2].w, w4[3].x, w4[3].y, w4[3].z, w4[3].w};
    // min / max as a 4-deep tree over the 16 bf16 pairs
    __nv_bfloat162 tmn[8], tmx[8];
#pragma unroll
    for (int k = 0; k < 8; ++k) {
        const __nv_bfloat162 a = *reinterpret_cast<const __nv_bfloat162 *>(&wd[2 * k]);
        const __nv_bfloat162 c = *reinterpret_cast<const __nv_bfloat162 *>(&wd[2 * k + 1]);
        tmn[k] = __hmin2(a, c);
        tmx[k] = __hmax2(a, c);
    }
#pragma unroll
    for (int n = 4; n > 0; n >>= 1)
#pragma unroll
        for (int k = 0; k < n; ++k) {
            tmn[k] = __hmin2(tmn[k], tmn[k + n]);
            tmx[k] = __hmax2(tmx[k], tmx[k + n]);
        }
    const __nv_bfloat162 mn2 = tmn[0], mx2 = tmx[0];
    float mn = fminf(__low2float(mn2), __high2float(mn2));
    float mx = fmaxf(__low2float(mx2), __high2float(mx2));
    if (lanes_per_group >= 2) {
        mn = fminf(mn, __shfl_xor_sync(0xffffffffu, mn, 1));
        mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 1));
    }
    if (lanes_per_group >= 4) {
        mn = fminf(mn, __shfl_xor_sync(0xffffffffu, mn, 2));
        mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 2));
    }
    float dh, de;
    two_sum(mx, -mn, dh, de);
    // (max - min) / L with L in {3, 7, 15}: exact in fp32 or a non-terminating
    // binary fraction, so one rounding to fp32 then fp16 equals one rounding to fp16.
    // dh (1/L) is within 2 ulps of dh / L; unless it lies within 4 ulps of an fp16
    // rounding midpoint (its low 13 mantissa bits near 0x1000) or below the fp16
    // normal range, both round to the same fp16 value.
    const float qm = dh * (1.f / static_cast<float>(L));
    const uint32_t qlow = __float_as_uint(qm) & 0x1FFFu;
    const bool qsafe = de == 0.f && qm >= 6.103515625e-05f && (qlow + 4u - 0x1000u) > 8u;
    __half s16;
    if (qsafe) s16 = __float2half_rn(qm);
    else if (de == 0.f) s16 = __float2half_rn(__fdiv_rn(dh, static_cast<float>(L)));
    else s16 = __double2half((static_cast<double>(mx) - static_cast<double>(mn)) / L);
    const __half z16 = __float2half_rn(mn);
    meta = static_cast<uint32_t>(__half_as_ushort(s16)) | (static_cast<uint32_t>(__half_as_ushort(z16)) << 16);
    const float sv = __half2float(s16), zv = __half2float(z16);
    // the reciprocal only feeds the fast estimate: its error (~2^-23) is far inside
    // the 4-ulp (2^-14) window that sends a code to the exact comparison
    float inv = 0.f;
    if (sv != 0.f) asm("rcp.approx.ftz.f32 %0, %1;" : "=f"(inv) : "f"(sv));
    // codes are summed as 1.5 * 2^23 + code shifted into place; the constant
    // parts (known at compile time) are subtracted at the end
    uint32_t bias[VB];
#pragma unroll
    for (int k = 0; k < VB; ++k) cw[k] = bias[k] = 0u;
#pragma unroll
    for (int e = 0; e < 32; ++e) {
        const uint32_t wv = wd[e >> 1];
        const float x = (e & 1) ? __uint_as_float(wv & 0xffff0000u) : __uint_as_float(wv << 16);
        const float dx = x - zv;
        // (x - zero) / scale rounded to the nearest integer: the code, except at a tie
        uint32_t cb = __float_as_uint(fmaf(dx, inv, kRoundMagic));
        // the same plus 1/2 + 4 ulps, in [192, 256) where the ulp is 2^-16: its low
        // 16 bits are below 8 within 4 ulps of a boundary (n - 1/2) scale
        const uint32_t tb = __float_as_uint(fmaf(dx, inv, 192.5f + 4.f / 65536.f));
        if ((tb & 0xFFF8u) == 0u) {
            // compare x - zero (an exact pair) with the boundary exactly
            const uint32_t n = (tb >> 16) & 0x1Fu;
            const float m = fmaf(static_cast<float>(n), sv, -0.5f * sv);
            float a, ea;
            two_sum(x, -zv, a, ea);
            cb = kRoundBits + ((__fadd_rn(__fsub_rn(a, m), ea) >= 0.f) ? n : n - 1u);
        }
        const int o = e * VB;
        cw[o >> 5] += cb << (o & 31);
        bias[o >> 5] += kRoundBits << (o & 31);
        if ((o & 31) + VB > 32) cw[(o >> 5) + 1] += (cb - kRoundBits) >> (32 - (o & 31));
    }
#pragma unroll
    for (int k = 0; k < VB; ++k) cw[k] -= bias[k];
    if (zv != mn || (sv != 0.f && sv < 6.103515625e-05f)) {
        uint32_t wl[16], cl[VB];  // local copies: the rare exact path keeps the hot one in registers
#pragma unroll
        for (int k = 0; k < 16; ++k) wl[k] = wd[k];
        values32_exact<VB>(wl, zv, sv, inv, cl);
#pragma unroll
        for (int k = 0; k < VB; ++k) cw[k] = cl[k];
    }
}

template <int KB, int VB>
__global__ void __launch_bounds__(kThreads, 1)
compress_tc_kernel(const Codec C, const PageGeom G, const uint16_t *__restrict__ kin, const uint16_t *__restrict__ vin,
                   int64_t rows, int Hkv, int64_t ks, int64_t vs, const int64_t *__restrict__ slots,
                   uint8_t *__restrict__ kc, uint8_t *__restrict__ vc, int64_t num_blocks, int num_tiles)
{
    constexpr int NKW = D * KB / 32;  // code words per row
    extern __shared__ __align__(1024) unsigned char smem[];
    uint32_t *scodes = reinterpret_cast<uint32_t *>(smem + kOffCodes);
    uint32_t *ssigns = reinterpret_cast<uint32_t *>(smem + kOffSigns);
    uint32_t *smask = reinterpret_cast<uint32_t *>(smem + kOffMask);
    RowInfo *rinfo_all = reinterpret_cast<RowInfo *>(smem + kOffRow);
    float *s_gsq = reinterpret_cast<float *>(smem + kOffPart);                 // [2][TM]
    int *s_flagp = reinterpret_cast<int *>(smem + kOffPart + TM * 8);          // [2][TM]
    int *s_flags = reinterpret_cast<int *>(smem + kOffPart + TM * 16);         // [2][TM]
    float4 *bins = reinterpret_cast<float4 *>(smem + kOffBins);
    uint64_t *mbarY = reinterpret_cast<uint64_t *>(smem + kOffMisc);      // rotation MMA done
    uint64_t *mbarP = mbarY + 1;                                           // projection MMA done
    uint64_t *mbarConv = mbarY + 2;                                        // keys of the tile converted
    uint64_t *mbarYfree = mbarY + 3;                                       // rotation accumulator read
    uint32_t *tslot = reinterpret_cast<uint32_t *>(smem + kOffMisc + 32);
    volatile int *e_abort = reinterpret_cast<volatile int *>(smem + kOffMisc + 36);
    volatile int *p_abort = reinterpret_cast<volatile int *>(smem + kOffMisc + 40);
    int *s_ndefer = reinterpret_cast<int *>(smem + kOffMisc + 96);  // rows left on the deferred list
    int *s_next = reinterpret_cast<int *>(smem + kOffMisc + 100);   // next list entry to fix

    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const float sqrtd = sqrtf(static_cast<float>(D));
    const int nthr = (1 << KB) - 1;
    const bool small_rows = rows <= 0x7fffffffLL;
    // token of a row: a shift when the head count is a power of two (the usual case)
    const int hshift = (Hkv & (Hkv - 1)) == 0 ? __ffs(Hkv) - 1 : -1;
    auto token_of = [&](int64_t r) -> int64_t {
        if (hshift >= 0) return r >> hshift;
        return small_rows ? static_cast<int64_t>(static_cast<uint32_t>(r) / static_cast<uint32_t>(Hkv)) : r / Hkv;
    };
    const int pshift = __ffs(G.P) - 1;  // the page size is a power of two
    const int64_t cache_slots = num_blocks * G.P;

    // ---- once per CTA: B operands, code bins, barriers, tensor memory ----
    {
        const uint4 *img = reinterpret_cast<const uint4 *>(C.tc_image);
        uint4 *dst = reinterpret_cast<uint4 *>(smem);
        for (int e = tid; e < 131072 / 16; e += kThreads) dst[e] = __ldg(img + e);
        if (tid < 256) {  // bin tid / 4, copy tid % 4
            const float b = static_cast<float>(tid >> 2);
            const float lo = 8.f * (64.f * b - 0.5f) / kBinScale - 4.f - 1.f / 64.f;
            const float hi = 8.f * (64.f * b + 63.5f) / kBinScale - 4.f + 1.f / 64.f;
            int below = 0, idx = -1;
            for (int t = 0; t < nthr; ++t) {
                const float th = C.thresholds[t];
                if (th < lo) ++below;
                else if (th <= hi) idx = t;
            }
            float4 e;
            e.x = idx >= 0 ? C.thresholds[idx] * 4096.f : __int_as_float(0x7f800000);
            e.y = C.centroids[below] * 4096.f;
            e.z = idx >= 0 ? C.centroids[below + 1] * 4096.f - e.y : 0.f;
            e.w = __uint_as_float(kCode23Bits + static_cast<uint32_t>(below));
            bins[tid] = e;
        }
        if (tid == 0) {
            uint32_t *dw = reinterpret_cast<uint32_t *>(smem + kOffMisc + 64);
            const uint32_t sb = umma::smem_u32(smem);
            const uint64_t dta = umma::make_desc(sb + kOffTA, 128, kSBO);
            dw[0] = static_cast<uint32_t>(dta >> 32);
            dw[1] = static_cast<uint32_t>(dta);
            dw[2] = static_cast<uint32_t>(umma::make_desc(sb + kOffTB, 128, kSBO));
            dw[3] = static_cast<uint32_t>(umma::make_desc(sb + kOffPiL, 128, kSBO));
            dw[4] = static_cast<uint32_t>(umma::make_desc(sb + kOffPiH, 128, kSBO));
            dw[5] = static_cast<uint32_t>(umma::make_desc(sb + kOffSH, 128, kSBO));
            dw[6] = static_cast<uint32_t>(umma::make_desc(sb + kOffSL, 128, kSBO));
            umma::mbar_init(mbarY, 1);
            umma::mbar_init(mbarP, 1);
            umma::mbar_init(mbarConv, 1);
            umma::mbar_init(mbarYfree, 1);
            asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
            *e_abort = 0;
            *p_abort = 0;
        }
        if (warp == 0) umma::tmem_alloc(tslot, 512);
        umma::fence_proxy_async();
        umma::fence_before_sync();
        __syncthreads();
        umma::fence_after_sync();
    }
    const uint32_t tmem = *tslot;
    // columns: Y [0, 128), P [128, 256), R hi [256, 320), R lo [320, 384)
    const uint32_t tY = tmem, tP = tmem + 128, tR = tmem + 256;
    const uint32_t sbase = umma::smem_u32(smem);
    // shared-memory descriptors of the operand tiles as (low, high) halves, kept in
    // shared memory (only the issuing thread reads them): [high, TA, TB, PiL, PiH, SH, SL]
    const uint32_t *sdesc = reinterpret_cast<const uint32_t *>(smem + kOffMisc + 64);

    if (warp >= kEpiWarps) {
        // =========================== producers =================================
        const int ptid = tid - kEpi, pw = warp - kEpiWarps;
        int it = 0, buf = 0;
        for (int tile = blockIdx.x; tile < num_tiles; tile += gridDim.x, ++it, buf = (buf == 2 ? 0 : buf + 1)) {
            const int64_t r0 = static_cast<int64_t>(tile) * TM;
            // three row-info buffers: the epilogue may still finish tile it-2 while tile it is converted
            RowInfo *rinfo = rinfo_all + buf * TM;
            // keys and values of this CTA's next tile start streaming into L2 now
            if (ptid < (VB > 0 ? 2 : 1) && tile + static_cast<int>(gridDim.x) < num_tiles) {
                const int64_t n0 = r0 + static_cast<int64_t>(gridDim.x) * TM;
                const int64_t n1 = min(n0 + TM, rows);
                const uint16_t *base = ptid == 0 ? kin : vin;
                const int64_t stride = ptid == 0 ? ks : vs;
                if (stride == static_cast<int64_t>(Hkv) * D) {
                    l2_prefetch_bulk(base + n0 * D, static_cast<uint32_t>((n1 - n0) * D * 2));
                } else {
                    for (int64_t t = n0 / Hkv; t <= (n1 - 1) / Hkv; ++t)
                        l2_prefetch_bulk(base + t * stride, static_cast<uint32_t>(Hkv * D * 2));
                }
            }
            // ---- issue the tile's key loads (and the first value rows) before waiting:
            // pass p covers rows 16 pw + 8 p + lane / 4; lane & 3 = sub takes key
            // chunks sub + 4 j and value channels [32 sub, 32 sub + 32) ----
            const int sub = lane & 3;
            uint4 kr[kPasses][4], va[4];
            int64_t sl[kPasses];
            int hh[kPasses];
#pragma unroll
            for (int p = 0; p < kPasses; ++p) {
                const int64_t r = r0 + 8 * kPasses * pw + 8 * p + (lane >> 2);
                sl[p] = -1;
                hh[p] = 0;
                if (r < rows) {
                    const int64_t t = token_of(r);
                    const int h = static_cast<int>(r - t * Hkv);
                    hh[p] = h;
                    const uint4 *ksrc = reinterpret_cast<const uint4 *>(kin + t * ks + static_cast<int64_t>(h) * D);
#pragma unroll
                    for (int j = 0; j < 4; ++j) kr[p][j] = ld_pinned(ksrc + sub + 4 * j);
                    if (VB > 0 && p == 0) {
                        const uint4 *vsrc = reinterpret_cast<const uint4 *>(vin + t * vs + static_cast<int64_t>(h) * D);
#pragma unroll
                        for (int j = 0; j < 4; ++j) va[j] = ld_pinned(vsrc + 4 * sub + j);
                    }
                    sl[p] = ld_pinned_s64(slots + t);
                } else {
#pragma unroll
                    for (int j = 0; j < 4; ++j) kr[p][j] = make_uint4(0u, 0u, 0u, 0u);
                    if (p == 0) {
#pragma unroll
                        for (int j = 0; j < 4; ++j) va[j] = make_uint4(0u, 0u, 0u, 0u);
                    }
                }
            }
            // the key tile buffer is free once the previous tile's rotation MMA finished
            if (it > 0 && ptid == 0) {
                if (!umma::mbar_wait_bounded(mbarY, (it - 1) & 1, C.wait_limit)) {
                    atomicOr(C.status, TQ_DEVERR_TIMEOUT);
                    *p_abort = 1;
                }
            }
            asm volatile("bar.sync 2, 256;" ::: "memory");
            if (*p_abort) break;
            // ---- keys: norm, power-of-two scale, exact fp16 conversion into the A tile ----
            int64_t dst[kPasses];
            int offs[kPasses];
#pragma unroll
            for (int p = 0; p < kPasses; ++p) {
                const int rl = 8 * kPasses * pw + 8 * p + (lane >> 2);
                const int64_t sp = sl[p];
                dst[p] = -1;
                offs[p] = 0;
                if (sp >= 0) {
                    if (sp < cache_slots) {
                        dst[p] = (sp >> pshift) * Hkv + hh[p];
                        offs[p] = static_cast<int>(sp & (G.P - 1));
                    } else if (sub == 0) {
                        atomicOr(C.status, TQ_DEVERR_SLOT_RANGE);
                    }
                }
                float mx = 0.f;
#pragma unroll
                for (int j = 0; j < 4; ++j) {
                    const uint32_t w[4] = {kr[p][j].x, kr[p][j].y, kr[p][j].z, kr[p][j].w};
#pragma unroll
                    for (int e = 0; e < 4; ++e)
                        mx = fmaxf(mx, fmaxf(fabsf(__uint_as_float(w[e] << 16)), fabsf(__uint_as_float(w[e] & 0xffff0000u))));
                }
                mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 1));
                mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 2));
                // mx in [2^(ex-1), 2^ex) from its exponent field (a subnormal or zero mx
                // gives ex = -126: tiny either way)
                const int ex = static_cast<int>((__float_as_uint(mx) >> 23) & 0xffu) - 126;
                // |k'| < 2^15; keys too small for a finite fp32 scale are redone exactly
                const bool tiny = (15 - ex) > 126;
                const float sc = __uint_as_float(static_cast<uint32_t>(127 + (tiny ? 126 : 15 - ex)) << 23);
                float ss = 0.f;
#pragma unroll
                for (int j = 0; j < 4; ++j) {
                    const uint32_t w[4] = {kr[p][j].x, kr[p][j].y, kr[p][j].z, kr[p][j].w};
                    uint32_t pk[4];
#pragma unroll
                    for (int e = 0; e < 4; ++e) {
                        const float a = __uint_as_float(w[e] << 16) * sc, b = __uint_as_float(w[e] & 0xffff0000u) * sc;
                        ss = fmaf(a, a, ss);
                        ss = fmaf(b, b, ss);
                        pk[e] = pack_h2(a, b);
                    }
                    *reinterpret_cast<uint4 *>(smem + kOffTA + umma::core_offset(rl, 8 * (sub + 4 * j), D)) =
                        make_uint4(pk[0], pk[1], pk[2], pk[3]);
                }
                ss += __shfl_xor_sync(0xffffffffu, ss, 1);
                ss += __shfl_xor_sync(0xffffffffu, ss, 2);
                if (sub == 0) {
                    RowInfo ri;
                    ri.dst = dst[p];
                    ri.off = offs[p];
                    ri.flag = 0;
                    ri.zscale = 0.f;
                    ri.rn = 0.f;
                    ri.n16g16 = 0u;
                    ri.pad = 0;
                    if (mx == 0.f) {
                        ri.flag = 8;  // zero key (or no key)
                    } else {
                        if (tiny) ri.flag = 4;
                        const float nsc = sqrtf(ss);  // ||k|| 2^(15-ex)
                        ri.zscale = sqrtd / (nsc * 1024.f);
                        // ||k|| = nsc / sc: one exact multiply by 2^(ex - 15), or 2^-126 for a
                        // tiny key (whose row is redone exactly anyway)
                        const float nk = tiny ? ldexpf(nsc, -126)
                                              : nsc * __uint_as_float(static_cast<uint32_t>(112 + ex) << 23);
                        ri.n16g16 = float_to_bf16_bits(nk);
                    }
                    rinfo[rl] = ri;
                }
            }
            umma::fence_proxy_async();
            asm volatile("bar.sync 2, 256;" ::: "memory");
            if (ptid == 0) {
                // ---- rotation MMAs: Y = K' (Pi_lo + Pi_hi)^T, once the epilogue has read Y ----
                bool ok = true;
                if (it > 0) ok = umma::mbar_wait_bounded(mbarYfree, (it - 1) & 1, C.wait_limit);
                if (ok) {
                    umma::fence_after_sync();
                    const uint32_t d_hi = sdesc[0], dTA_lo = sdesc[1], dPiL_lo = sdesc[3], dPiH_lo = sdesc[4];
#pragma unroll
                    for (int term = 0; term < 2; ++term) {
                        const uint32_t blo = term == 0 ? dPiL_lo : dPiH_lo;
#pragma unroll
                        for (int s = 0; s < D / 16; ++s)  // k-step s starts 256 bytes (16 in the >> 4 field) further
                            umma::mma_f16_lohi(tY, dTA_lo + 16u * s, d_hi, blo + 16u * s, d_hi, kIdesc, (term | s) != 0);
                    }
                    umma::commit(mbarY);
                    asm volatile("mbarrier.arrive.release.cta.shared::cta.b64 _, [%0];" ::"r"(umma::smem_u32(mbarConv))
                                 : "memory");
                } else {
                    atomicOr(C.status, TQ_DEVERR_TIMEOUT);
                    *p_abort = 1;
                }
            }
            // ---- values of this tile: pass p + 1 is loaded while pass p is quantised ----
            if constexpr (VB > 0) {
            const int lpg = C.group >> 5;  // lanes per group: 1, 2 or 4
#pragma unroll 1
            for (int p = 0; p < kPasses; ++p) {
                uint4 vb[4];
#pragma unroll
                for (int j = 0; j < 4; ++j) vb[j] = make_uint4(0u, 0u, 0u, 0u);
                const int64_t rn1 = r0 + 8 * kPasses * pw + 8 * (p + 1) + (lane >> 2);
                if (p + 1 < kPasses && rn1 < rows) {
                    const int64_t t = token_of(rn1);
                    const uint4 *vsrc = reinterpret_cast<const uint4 *>(vin + t * vs + (rn1 - t * Hkv) * D);
#pragma unroll
                    for (int j = 0; j < 4; ++j) vb[j] = ld_pinned(vsrc + 4 * sub + j);
                }
                uint32_t cw[VB], meta;
                quantize_values32<VB>(va, lpg, cw, meta);
                const int rl = 8 * kPasses * pw + 8 * p + (lane >> 2);
                const int64_t vdst = rinfo[rl].dst;
                if (vdst >= 0) {
                    const int voff = rinfo[rl].off;
                    uint8_t *vrec = vc + vdst * G.v_page;
                    uint8_t *vcode = vrec + static_cast<int64_t>(voff) * (D * VB / 8);
                    if constexpr (VB == 2) {
                        reinterpret_cast<uint2 *>(vcode)[sub] = make_uint2(cw[0], cw[1]);
                    } else if constexpr (VB == 4) {
                        reinterpret_cast<uint4 *>(vcode)[sub] = make_uint4(cw[0], cw[1], cw[2], cw[3]);
                    } else {
                        uint32_t *vw = reinterpret_cast<uint32_t *>(vcode) + VB * sub;
#pragma unroll
                        for (int k = 0; k < VB; ++k) vw[k] = cw[k];
                    }
                    if ((sub & (lpg - 1)) == 0)
                        *reinterpret_cast<uint32_t *>(vrec + G.v_meta_off + static_cast<int64_t>(voff) * C.v_meta_bytes +
                                                      4 * (sub / lpg)) = meta;
                }
#pragma unroll
                for (int j = 0; j < 4; ++j) va[j] = vb[j];
            }
            }  // VB > 0
        }
    } else {
        // =========================== epilogue ==================================
        const int row = 32 * (warp & 3) + lane, hf = warp >> 2;
        Deferred *defer = reinterpret_cast<Deferred *>(smem + kOffDefer);
        int *s_qcount = reinterpret_cast<int *>(smem + kOffMisc + 44);  // [4] flagged rows per lane quarter
        int ndefer = 0;  // same value in every epilogue thread
        // a full list is drained by the epilogue warps alone; the rest waits for the end
        auto drain = [&](int n) {  // all epilogue threads; warp w fixes entries w, w + 8, ...
            asm volatile("bar.sync 1, 256;" ::: "memory");
            double *scr = reinterpret_cast<double *>(smem + kOffTB) + warp * D;
            for (int e = warp; e < n; e += kEpiWarps)
                fix_row<KB>(C, G, kin, ks, Hkv, kc, defer[e], scodes + warp * 16, ssigns + warp * 4,
                            reinterpret_cast<uint32_t *>(s_gsq) + warp, scr);
            asm volatile("bar.sync 1, 256;" ::: "memory");
        };
        int it = 0, buf = 0;
        for (int tile = blockIdx.x; tile < num_tiles; tile += gridDim.x, ++it, buf = (buf == 2 ? 0 : buf + 1)) {
            const int64_t r0 = static_cast<int64_t>(tile) * TM;
            RowInfo *rinfo = rinfo_all + buf * TM;
            const uint32_t par = it & 1;
            if (!umma::mbar_wait_bounded(mbarConv, par, C.wait_limit) || !umma::mbar_wait_bounded(mbarY, par, C.wait_limit)) {
                atomicOr(C.status, TQ_DEVERR_TIMEOUT);
                *e_abort = 1;
            }
            umma::fence_after_sync();
            asm volatile("bar.sync 1, 256;" ::: "memory");
            if (*e_abort) break;
            const RowInfo ri = rinfo[row];
            const bool zero = (ri.flag & 8) != 0;
            float gsq = 0.f;
            int fl = 0;
            {
                const float zs = ri.zscale * 4096.f;  // z' = 2^12 z
#pragma unroll 1
                for (int cb = 2 * hf; cb < 2 * hf + 2; ++cb)
                    gsq += epilogue_rotation_block<KB>(smem, tY, tR, warp, row, cb, zs, C.qjl != 0, scodes, smask);
                gsq *= 1.f / 16777216.f;  // back to z units
                fl = (smask[(2 * hf) * TM + row] | smask[(2 * hf + 1) * TM + row]) ? 1 : 0;
            }
            s_gsq[hf * TM + row] = gsq;
            s_flagp[hf * TM + row] = fl;
            if (C.qjl) umma::wait_st();  // the residual operand is in tensor memory
            umma::fence_before_sync();
            asm volatile("bar.sync 1, 256;" ::: "memory");
            umma::fence_after_sync();
            const float rn = sqrtf(s_gsq[row] + s_gsq[TM + row]);
            int flag = ri.flag | s_flagp[row] | s_flagp[TM + row];
            uint32_t n16g16 = ri.n16g16;
            if (C.qjl) {
                if (tid == 0) {
                    // ---- projection MMAs: P = (R_hi + R_lo)(S_hi + S_lo)^T, small terms first;
                    // R from tensor memory, so the key tile buffer is already the next tile's ----
                    const uint32_t d_hi = sdesc[0], dSH_lo = sdesc[5], dSL_lo = sdesc[6];
#pragma unroll
                    for (int term = 0; term < 3; ++term) {
                        const uint32_t ta = term == 0 ? tR + 64 : tR;
                        const uint32_t blo = term == 1 ? dSL_lo : dSH_lo;
#pragma unroll
                        for (int s = 0; s < D / 16; ++s)
                            umma::mma_f16_tmem_a(tP, ta + 8u * s, blo + 16u * s, d_hi, kIdesc, (term | s) != 0);
                    }
                    umma::commit(mbarP);
                }
            }
            // Y may be overwritten now: the next tile's rotation queues behind the projection
            if (tid == 0)
                asm volatile("mbarrier.arrive.release.cta.shared::cta.b64 _, [%0];" ::"r"(umma::smem_u32(mbarYfree))
                             : "memory");
            // ---- while the projection runs: code words and norm of this row's record
            // (a row whose decisions are re-taken exactly rewrites them below) ----
            if (ri.dst >= 0) {
                uint8_t *krec = kc + ri.dst * G.k_page;
                uint32_t *cd = reinterpret_cast<uint32_t *>(krec + static_cast<int64_t>(ri.off) * C.k_code_bytes);
                const uint32_t *cw = scodes + row;
#pragma unroll
                for (int w = 0; w < NKW / 2; ++w) cd[hf * (NKW / 2) + w] = zero ? 0u : cw[(hf * (NKW / 2) + w) * TM];
                if (hf == 0)
                    *reinterpret_cast<uint16_t *>(krec + G.k_norm_off + 2 * ri.off) =
                        zero ? 0 : static_cast<uint16_t>(ri.n16g16 & 0xffffu);
            }
            if (C.qjl) {
                if (!umma::mbar_wait_bounded(mbarP, par, C.wait_limit)) {
                    atomicOr(C.status, TQ_DEVERR_TIMEOUT);
                    *e_abort = 1;
                }
                umma::fence_after_sync();
                const float guard = kSignGuard * rn * 16777216.f;  // P = 2^24 p (z units)
                const int sf = epilogue_signs(tP, warp, row, hf, guard, zero, ssigns, smask);
                s_flags[hf * TM + row] = sf;
                if (!zero) {
                    const float gam = rn / sqrtd;
                    n16g16 |= static_cast<uint32_t>(float_to_bf16_bits(gam)) << 16;
                    // distance of gamma to the nearest bf16 rounding midpoint, relative
                    int ge;
                    const float fr = frexpf(gam, &ge);  // gam = fr 2^ge, fr in [0.5, 1)
                    const float u = fr * 256.f;         // bf16 keeps 8 significant bits
                    if (fabsf(u - floorf(u) - 0.5f) / u < kGammaGuard) flag |= 16;
                }
            }
            asm volatile("bar.sync 1, 256;" ::: "memory");
            if (*e_abort) break;
            // both threads of a row hold the same flag, rn and gamma (from both halves' partials)
            if (C.qjl) flag |= s_flags[row] | s_flags[TM + row];
            if (zero) flag = 8;
            // ---- key records, rest: signs and gamma (deferred rows are rewritten when drained) ----
            if (ri.dst >= 0) {
                uint8_t *krec = kc + ri.dst * G.k_page;
                if (C.qjl) {
                    const uint32_t *sw = ssigns + row;
                    uint2 *sd = reinterpret_cast<uint2 *>(krec + G.k_sign_off + static_cast<int64_t>(ri.off) * C.k_sign_bytes);
                    sd[hf] = zero ? make_uint2(0u, 0u) : make_uint2(sw[(2 * hf) * TM], sw[(2 * hf + 1) * TM]);
                }
                if (hf == 0 && C.qjl)
                    *reinterpret_cast<uint16_t *>(krec + G.k_gamma_off + 2 * ri.off) =
                        zero ? 0 : static_cast<uint16_t>(n16g16 >> 16);
            }
            // ---- rows needing exact re-decisions join the deferred list; it is drained
            // by all epilogue warps together whenever it would overflow ----
            {
                const bool mine = hf == 0 && (flag & 23) != 0 && !zero && ri.dst >= 0;
                const uint32_t pend = __ballot_sync(0xffffffffu, mine);
                if (hf == 0 && lane == 0) s_qcount[warp] = __popc(pend);
                asm volatile("bar.sync 1, 256;" ::: "memory");
                int prefix = 0, n_t = 0;
#pragma unroll
                for (int q = 0; q < 4; ++q) {
                    const int cq = s_qcount[q];
                    if (q < (warp & 3)) prefix += cq;
                    n_t += cq;
                }
                const int rank = prefix + __popc(pend & ((1u << lane) - 1u));
                int done = 0;
                while (done < n_t) {
                    if (ndefer == kMaxDefer) {
                        drain(ndefer);
                        ndefer = 0;
                    }
                    const int take = min(kMaxDefer - ndefer, n_t - done);
                    if (mine && rank >= done && rank < done + take) {
                        Deferred &d = defer[ndefer + rank - done];
                        d.r = r0 + row;
                        d.dst = ri.dst;
                        d.off = ri.off;
                        d.flag = flag;
#pragma unroll
                        for (int w = 0; w < 4; ++w) {
                            d.cmask[w] = smask[w * TM + row];
                            d.smask[w] = smask[(4 + w) * TM + row];
                        }
                    }
                    ndefer += take;
                    done += take;
                }
            }
            asm volatile("bar.sync 1, 256;" ::: "memory");
        }
        if (tid == 0) *s_ndefer = ndefer;
    }
    // ---- rows still awaiting exact re-decisions: every warp takes the next one in
    // turn, the ones that redo the whole row first (they take longest) ----
    __syncthreads();
    {
        const int nd = *s_ndefer;
        if (nd > 0 && !*e_abort && !*p_abort) {
            const Deferred *defer = reinterpret_cast<const Deferred *>(smem + kOffDefer);
            uint8_t *order = smem + kOffBins;  // the code bins are no longer needed
            if (tid == 0) {
                int h = 0;
                for (int e = 0; e < nd; ++e)
                    if (defer[e].flag & 20) order[h++] = static_cast<uint8_t>(e);
                for (int e = 0; e < nd; ++e)
                    if (!(defer[e].flag & 20)) order[h++] = static_cast<uint8_t>(e);
                *s_next = 0;
            }
            __syncthreads();
            double *scr = reinterpret_cast<double *>(smem + kOffTB) + warp * D;
            for (;;) {
                int e = 0;
                if (lane == 0) e = atomicAdd(s_next, 1);
                e = __shfl_sync(0xffffffffu, e, 0);
                if (e >= nd) break;
                fix_row<KB>(C, G, kin, ks, Hkv, kc, defer[order[e]], scodes + warp * 16, ssigns + warp * 4,
                            reinterpret_cast<uint32_t *>(s_gsq) + warp, scr);
            }
        }
    }
    // ---- teardown: no MMA may still run when TMEM is freed ----
    __syncthreads();
    if (*e_abort || *p_abort) {
        const long long t0 = clock64();
        while (clock64() - t0 < kDrainLimit / 20) {  // fixed grace period (~0.1 s) for in-flight tensor-core work
        }
    }
    umma::fence_before_sync();
    __syncthreads();
    umma::fence_after_sync();
    if (warp == 0) umma::tmem_dealloc(tmem, 512);
}

// Group-quantised values alone (the keys taking a keys-only pass): the fused
// kernel's value layout, DD / 32 lanes per row, lane sub of a row holding channels
// [32 sub, 32 sub + 32), 1024 / DD rows per warp; row groups strided over a one-wave
// grid with the next group's values and slots in flight while the current one is
// quantised.  The loop bounds are the same for the whole warp, so the group
// reductions' shuffles (within a row's lanes) always run with every lane.
template <int DD, int VB>
__global__ void __launch_bounds__(256, 4)
compress_values_tc_kernel(const Codec C, const PageGeom G, const uint16_t *__restrict__ vin, int64_t rows, int Hkv,
                          int64_t vs, const int64_t *__restrict__ slots, uint8_t *__restrict__ vc, int64_t num_blocks)
{
    constexpr int LPR = DD / 32, RPW = 32 / LPR;  // lanes per row, rows per warp
    const int lane = threadIdx.x & 31, sub = lane % LPR, rq = lane / LPR;
    const int lpg = C.group >> 5;  // lanes per group: 1, 2 or 4
    const int hshift = (Hkv & (Hkv - 1)) == 0 ? __ffs(Hkv) - 1 : -1;
    const int pshift = __ffs(G.P) - 1;
    const int64_t cache_slots = num_blocks * G.P;
    const int64_t stride = RPW * static_cast<int64_t>(gridDim.x) * (blockDim.x >> 5);
    auto fetch = [&](int64_t r, uint4 (&w)[4], int64_t &sl) {
        sl = -1;
#pragma unroll
        for (int j = 0; j < 4; ++j) w[j] = make_uint4(0u, 0u, 0u, 0u);
        if (r < rows) {
            const int64_t t = hshift >= 0 ? (r >> hshift) : r / Hkv;
            const uint4 *src = reinterpret_cast<const uint4 *>(vin + t * vs + (r - t * Hkv) * DD);
#pragma unroll
            for (int j = 0; j < 4; ++j) w[j] = ld_pinned(src + 4 * sub + j);
            sl = ld_pinned_s64(slots + t);
        }
    };
    int64_t base = RPW * (static_cast<int64_t>(blockIdx.x) * (blockDim.x >> 5) + (threadIdx.x >> 5));
    uint4 wn[4];
    int64_t sn;
    fetch(base + rq, wn, sn);
    for (; base < rows; base += stride) {
        const int64_t r = base + rq;
        uint4 w[4];
#pragma unroll
        for (int j = 0; j < 4; ++j) w[j] = wn[j];
        const int64_t slot = sn;
        fetch(base + stride + rq, wn, sn);
        uint32_t cw[VB], meta;
        quantize_values32<VB>(w, lpg, cw, meta);
        if (r >= rows || slot < 0) continue;
        if (slot >= cache_slots) {
            if (sub == 0) atomicOr(C.status, TQ_DEVERR_SLOT_RANGE);
            continue;
        }
        const int64_t t = hshift >= 0 ? (r >> hshift) : r / Hkv;
        const int64_t dst = (slot >> pshift) * Hkv + (r - t * Hkv);
        const int64_t off = slot & (G.P - 1);
        uint8_t *vrec = vc + dst * G.v_page;
        uint8_t *vcode = vrec + off * (DD * VB / 8);
        if constexpr (VB == 2) {
            reinterpret_cast<uint2 *>(vcode)[sub] = make_uint2(cw[0], cw[1]);
        } else if constexpr (VB == 4) {
            reinterpret_cast<uint4 *>(vcode)[sub] = make_uint4(cw[0], cw[1], cw[2], cw[3]);
        } else {
            uint32_t *vw = reinterpret_cast<uint32_t *>(vcode) + VB * sub;
#pragma unroll
            for (int k = 0; k < VB; ++k) vw[k] = cw[k];
        }
        if ((sub & (lpg - 1)) == 0)
            *reinterpret_cast<uint32_t *>(vrec + G.v_meta_off + off * C.v_meta_bytes + 4 * (sub / lpg)) = meta;
    }
}

template <int DD, int VB>
cudaError_t launch_values_tc(const Codec &c, const PageGeom &pg, const uint16_t *v, int64_t T, int Hkv, int64_t vs,
                             const int64_t *slots, uint8_t *vc, int64_t num_blocks, int num_sms, cudaStream_t st)
{
    const int64_t rows = T * Hkv;
    constexpr int64_t kRowsPerCta = 8 * (1024 / DD);  // 8 warps
    int64_t blocks = (rows + kRowsPerCta - 1) / kRowsPerCta;
    const int64_t cap = static_cast<int64_t>(num_sms) * 4;  // one wave: four resident CTAs per SM
    if (blocks > cap) blocks = cap;
    compress_values_tc_kernel<DD, VB><<<static_cast<unsigned>(blocks), 256, 0, st>>>(c, pg, v, rows, Hkv, vs, slots,
                                                                                   vc, num_blocks);
    return cudaGetLastError();
}

template <int KB, int VB>
cudaError_t launch_tc(const Codec &c, const PageGeom &pg, const uint16_t *k, const uint16_t *v, int64_t T, int Hkv,
                      int64_t ks, int64_t vs, const int64_t *slots, uint8_t *kc, uint8_t *vc, int64_t num_blocks,
                      int num_sms, cudaStream_t st)
{
    cudaError_t e = ensure_smem_attr(reinterpret_cast<const void *>(compress_tc_kernel<KB, VB>), kSmemBytes);
    if (e != cudaSuccess) return e;
    const int64_t rows = T * Hkv;
    const int tiles = static_cast<int>((rows + TM - 1) / TM);
    const int grid = tiles < num_sms ? tiles : num_sms;
    compress_tc_kernel<KB, VB><<<grid, kThreads, kSmemBytes, st>>>(c, pg, k, v, rows, Hkv, ks, vs, slots, kc, vc,
                                                                   num_blocks, tiles);
    return cudaGetLastError();
}

template <int KB>
cudaError_t launch_tc_kb(const Codec &c, const PageGeom &pg, const uint16_t *k, const uint16_t *v, int64_t T, int Hkv,
                         int64_t ks, int64_t vs, const int64_t *slots, uint8_t *kc, uint8_t *vc, int64_t num_blocks,
                         int num_sms, cudaStream_t st)
{
    switch (c.v_bits) {
    case 2: return launch_tc<KB, 2>(c, pg, k, v, T, Hkv, ks, vs, slots, kc, vc, num_blocks, num_sms, st);
    case 3: return launch_tc<KB, 3>(c, pg, k, v, T, Hkv, ks, vs, slots, kc, vc, num_blocks, num_sms, st);
    default: return launch_tc<KB, 4>(c, pg, k, v, T, Hkv, ks, vs, slots, kc, vc, num_blocks, num_sms, st);
    }
}

}  // namespace

size_t compress_tc_smem_bytes() { return kSmemBytes; }

cudaError_t launch_compress_values_tc(const Codec &c, const PageGeom &pg, const uint16_t *v, int64_t T, int Hkv,
                                      int64_t vs, const int64_t *slots, uint8_t *vc, int64_t num_blocks, int num_sms,
                                      cudaStream_t st)
{
    if (c.d == 256) {
        switch (c.v_bits) {
        case 2: return launch_values_tc<256, 2>(c, pg, v, T, Hkv, vs, slots, vc, num_blocks, num_sms, st);
        case 3: return launch_values_tc<256, 3>(c, pg, v, T, Hkv, vs, slots, vc, num_blocks, num_sms, st);
        default: return launch_values_tc<256, 4>(c, pg, v, T, Hkv, vs, slots, vc, num_blocks, num_sms, st);
        }
    }
    switch (c.v_bits) {
    case 2: return launch_values_tc<128, 2>(c, pg, v, T, Hkv, vs, slots, vc, num_blocks, num_sms, st);
    case 3: return launch_values_tc<128, 3>(c, pg, v, T, Hkv, vs, slots, vc, num_blocks, num_sms, st);
    default: return launch_values_tc<128, 4>(c, pg, v, T, Hkv, vs, slots, vc, num_blocks, num_sms, st);
    }
}

cudaError_t launch_compress_tc_keys(const Codec &c, const PageGeom &pg, const uint16_t *k, int64_t T, int Hkv,
                                    int64_t ks, const int64_t *slots, uint8_t *kc, int64_t num_blocks, int num_sms,
                                    cudaStream_t st)
{
    switch (c.k_bits) {
    case 2: return launch_tc<2, 0>(c, pg, k, nullptr, T, Hkv, ks, 0, slots, kc, nullptr, num_blocks, num_sms, st);
    case 3: return launch_tc<3, 0>(c, pg, k, nullptr, T, Hkv, ks, 0, slots, kc, nullptr, num_blocks, num_sms, st);
    default: return launch_tc<4, 0>(c, pg, k, nullptr, T, Hkv, ks, 0, slots, kc, nullptr, num_blocks, num_sms, st);
    }
}

cudaError_t launch_compress_tc(const Codec &c, const PageGeom &pg, const uint16_t *k, const uint16_t *v, int64_t T,
                               int Hkv, int64_t ks, int64_t vs, const int64_t *slots, uint8_t *kc, uint8_t *vc,
                               int64_t num_blocks, int num_sms, cudaStream_t st)
{
    switch (c.k_bits) {
    case 2: return launch_tc_kb<2>(c, pg, k, v, T, Hkv, ks, vs, slots, kc, vc, num_blocks, num_sms, st);
    case 3: return launch_tc_kb<3>(c, pg, k, v, T, Hkv, ks, vs, slots, kc, vc, num_blocks, num_sms, st);
    default: return launch_tc_kb<4>(c, pg, k, v, T, Hkv, ks, vs, slots, kc, vc, num_blocks, num_sms, st);
    }
}

}  // namespace tq
