// tq_decode_bf16.cu -- bypass decode: the split-K paged decode skeleton over a
// plain bf16 paged KV cache, with no codec.
//
// turbo-attn, "Two independently-usable pieces", item 2: besides the codec's own
// page loader, the decode kernel takes a bypass loader that reads ordinary bf16
// pages.  Run on the same shapes, it measures what the skeleton itself (paging,
// split-K, online softmax, combine) achieves on HBM, so that the compressed
// decode's gap to the roofline can be split into skeleton and codec.
//
// Pools: K and V are bf16 [num_blocks][Hkv][P][d]; token slot s of a sequence
// lives in block s / P at row s % P.  One CTA = (split, kv head, sequence), four
// warps; warp w takes the 16-token rounds w, w + 4, ... of its split.  Each
// round's K and V rows are fetched by the tensor memory accelerator
// (cp.async.bulk.tensor, 16 x 64 boxes, 128-byte swizzle) into the warp's own
// two stages, completing on the warp's mbarriers, so ldmatrix reads of token rows
// hit 8 different bank groups.  Scores: tokens as M of mma.m16n8k16 (bf16 in,
// fp32 accumulate: K and q are bf16, so every product is exact), heads as N.
// P.V: coordinates as M (V rows transposed by ldmatrix.trans), probabilities as
// the B operand in two bf16 terms (high and low part, ~16 significant bits).
#include <cuda.h>
#include <cudaTypedefs.h>
#include <cuda_runtime.h>

#include <mutex>

#include "tq.h"
#include "tq_device.cuh"
#include "tq_internal.h"

namespace tq {
namespace {

constexpr int kWarps = 4;
constexpr int kThreads = 32 * kWarps;
constexpr int kTile = 16;                 // tokens per round
constexpr int kBoxCols = 64;              // bf16 columns per 128-byte swizzled box
constexpr int kBoxBytes = kTile * 128;    // 2 KB
constexpr float kLog2e = 1.4426950408889634f;

template <int D>
struct BypassSmem {
    static constexpr int kTileBytes = kTile * D * 2;  // one K or V tile
    static constexpr int kStage = 2 * kTileBytes;     // K then V
    static constexpr size_t kData = static_cast<size_t>(kWarps) * 2 * kStage;
    static constexpr size_t kBytes = 1024 + kData + 256;  // alignment slack, stages, barriers and flags
    static_assert(kData >= sizeof(float) * kWarps * (D * 8 + 16), "merge area");
};

__device__ __forceinline__ void mma_bf16(float (&c)[4], uint32_t a0, uint32_t a1, uint32_t a2, uint32_t a3, uint32_t b0,
                                         uint32_t b1)
{
    asm volatile("mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
                 "{%0,%1,%2,%3};"
                 : "+f"(c[0]), "+f"(c[1]), "+f"(c[2]), "+f"(c[3])
                 : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}

__device__ __forceinline__ void ldsm_x4(uint32_t addr, uint32_t &a0, uint32_t &a1, uint32_t &a2, uint32_t &a3)
{
    asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0,%1,%2,%3}, [%4];"
                 : "=r"(a0), "=r"(a1), "=r"(a2), "=r"(a3) : "r"(addr));
}

__device__ __forceinline__ void ldsm_x4_trans(uint32_t addr, uint32_t &a0, uint32_t &a1, uint32_t &a2, uint32_t &a3)
{
    asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0,%1,%2,%3}, [%4];"
                 : "=r"(a0), "=r"(a1), "=r"(a2), "=r"(a3) : "r"(addr));
}

__device__ __forceinline__ uint32_t movmatrix_trans(uint32_t a)
{
    uint32_t d;
    asm volatile("movmatrix.sync.aligned.m8n8.trans.b16 %0, %1;" : "=r"(d) : "r"(a));
    return d;
}

__device__ __forceinline__ uint32_t pack_bf16x2(float lo, float hi)
{
    const __nv_bfloat162 h = __floats2bfloat162_rn(lo, hi);
    return *reinterpret_cast<const uint32_t *>(&h);
}

__device__ __forceinline__ float fast_exp2(float x)
{
    float y;
    asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}

__device__ __forceinline__ bool mbar_test(uint32_t mb, uint32_t par)
{
    uint32_t done;
    asm volatile("{\n.reg .pred p;\nmbarrier.test_wait.parity.shared::cta.b64 p, [%1], %2;\nselp.u32 %0, 1, 0, p;\n}\n"
                 : "=r"(done) : "r"(mb), "r"(par) : "memory");
    return done != 0;
}

__device__ __forceinline__ bool mbar_try(uint32_t mb, uint32_t par)
{
    uint32_t done;
    asm volatile("{\n.reg .pred p;\nmbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\nselp.u32 %0, 1, 0, p;\n}\n"
                 : "=r"(done) : "r"(mb), "r"(par) : "memory");
    return done != 0;
}

template <int D>
__global__ void __launch_bounds__(kThreads) decode_bf16_kernel(const __grid_constant__ CUtensorMap tmK,
                                                               const __grid_constant__ CUtensorMap tmV, const Codec C,
                                                               const int page_size, const DecodeArgs A)
{
    using SM = BypassSmem<D>;
    constexpr int KS = D / 16;   // k-steps of the score MMA, m-tiles of P.V
    extern __shared__ unsigned char smem_raw[];
    unsigned char *smem = reinterpret_cast<unsigned char *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    uint64_t *mbar = reinterpret_cast<uint64_t *>(smem + SM::kData);  // [warp][stage]
    int *page_ok = reinterpret_cast<int *>(mbar + 2 * kWarps);        // [warp][stage]
    volatile int *cta_abort = page_ok + 2 * kWarps;

    const int split = blockIdx.x, kvh = blockIdx.y, b = blockIdx.z;
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int quad = lane & 3, row = lane >> 2;
    const int P = page_size;
    const int G = A.Hq / A.Hkv;
    int L = A.seq_lens[b];
    if (L < 0) L = 0;
    if (L > A.max_blocks * P) {
        if (split == 0 && kvh == 0 && tid == 0) atomicOr(C.status, TQ_DEVERR_SEQ_RANGE);
        L = A.max_blocks * P;
    }
    const int tok0 = split * A.pages_per_split * P;
    const int tok1 = min(L, tok0 + A.pages_per_split * P);
    const size_t head0 = static_cast<size_t>(b) * A.Hq + static_cast<size_t>(kvh) * G;
    float *ml_out = A.ws.ml + (static_cast<size_t>(split) * A.B * A.Hq + head0) * 2;
    float *acc_out = A.ws.acc + (static_cast<size_t>(split) * A.B * A.Hq + head0) * D;
    if (tok0 >= tok1) {
        if (tid < G) {
            ml_out[2 * tid] = -INFINITY;
            ml_out[2 * tid + 1] = 0.f;
        }
        return;
    }
    const int nrounds = (tok1 - tok0 + kTile - 1) / kTile;

    // query fragments (B operand of the score MMA): head `row`, coordinates 16 s + 2 quad (+1) and + 8
    uint32_t qb[KS][2];
    {
        const bool hv = row < G;
        const uint32_t *qr = reinterpret_cast<const uint32_t *>(A.q + (head0 + (hv ? row : 0)) * D);
#pragma unroll
        for (int s = 0; s < KS; ++s) {
            qb[s][0] = hv ? __ldg(qr + 8 * s + quad) : 0u;
            qb[s][1] = hv ? __ldg(qr + 8 * s + 4 + quad) : 0u;
        }
    }

    const uint32_t sbase = static_cast<uint32_t>(__cvta_generic_to_shared(smem));
    auto stage_off = [&](int st) -> uint32_t { return static_cast<uint32_t>((warp * 2 + st) * SM::kStage); };
    auto mbar_addr = [&](int st) -> uint32_t {
        return static_cast<uint32_t>(__cvta_generic_to_shared(&mbar[warp * 2 + st]));
    };
    auto fetch_id = [&](int rr) -> int {  // block id of this warp's round rr (lane 0)
        const int t = tok0 + (4 * rr + warp) * kTile;
        if (t >= tok1) return -1;
        return A.block_table[static_cast<int64_t>(b) * A.max_blocks + t / P];
    };
    auto issue = [&](int rr, int st, int blk) {  // lane 0
        const int t = tok0 + (4 * rr + warp) * kTile;
        int ok = 0;
        if (t < tok1) {
            ok = (blk >= 0 && blk < A.num_blocks);
            if (!ok) atomicOr(C.status, TQ_DEVERR_BLOCK_RANGE);
        }
        page_ok[warp * 2 + st] = ok;
        const uint32_t mb = mbar_addr(st);
        asm volatile("fence.proxy.async.shared::cta;" ::: "memory");  // this warp's reads of the stage are done
        asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(mb),
                     "r"(ok ? static_cast<uint32_t>(SM::kStage) : 0u)
                     : "memory");
        if (ok) {
            const int y = static_cast<int>((static_cast<int64_t>(blk) * A.Hkv + kvh) * P + t % P);
            const uint32_t dk = sbase + stage_off(st);
#pragma unroll
            for (int x = 0; x < D / kBoxCols; ++x) {
                asm volatile("cp.async.bulk.tensor.2d.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1, {%2, %3}], [%4];"
                             ::"r"(dk + x * kBoxBytes), "l"(reinterpret_cast<uint64_t>(&tmK)), "r"(x * kBoxCols), "r"(y), "r"(mb)
                             : "memory");
                asm volatile("cp.async.bulk.tensor.2d.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1, {%2, %3}], [%4];"
                             ::"r"(dk + SM::kTileBytes + x * kBoxBytes), "l"(reinterpret_cast<uint64_t>(&tmV)), "r"(x * kBoxCols),
                             "r"(y), "r"(mb)
                             : "memory");
            }
        }
    };
    auto drain = [&](int st, uint32_t par) {
        const long long t0 = clock64();
        while (!mbar_try(mbar_addr(st), par) && clock64() - t0 < kDrainLimit) {
        }
    };

    if (tid < 2 * kWarps)
        asm volatile("mbarrier.init.shared::cta.b64 [%0], 1;" ::"r"(static_cast<uint32_t>(__cvta_generic_to_shared(&mbar[tid]))));
    if (tid == 0) *cta_abort = 0;
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    __syncthreads();

    float o[KS][4];
#pragma unroll
    for (int mt = 0; mt < KS; ++mt) o[mt][0] = o[mt][1] = o[mt][2] = o[mt][3] = 0.f;
    float m_run[2] = {-INFINITY, -INFINITY};  // heads 2 quad + e
    float l_run[2] = {0.f, 0.f};
    const float fac = A.sm_scale * kLog2e;
    // this lane's ldmatrix row and 16-byte chunk: matrices (rows 0-7 | 8-15) x (chunk c | c + 1)
    const int mi = lane >> 3, ri = lane & 7;
    const int krow = ri + 8 * (mi & 1), kch = mi >> 1;  // scores: a0 rows 0-7, a1 rows 8-15, a2/a3 next chunk
    const int vrow = ri + 8 * (mi >> 1), vch = mi & 1;  // values (transposed): a0 chunk c, a1 chunk c + 1, a2/a3 rows 8-15

    const int my_rounds = (nrounds - warp + 3) / 4;  // rounds warp, warp + 4, ...
    int bnext = (lane == 0 && my_rounds > 0) ? fetch_id(0) : -1;
    if (lane == 0 && my_rounds > 0) issue(0, 0, bnext);
    if (lane == 0 && my_rounds > 1) bnext = fetch_id(1);
    for (int c = 0; c < my_rounds; ++c) {
        const int st = c & 1;
        __syncwarp();  // every lane is done with the stage the next copy overwrites
        if (c + 1 < my_rounds && lane == 0) {
            issue(c + 1, st ^ 1, bnext);
            if (c + 2 < my_rounds) bnext = fetch_id(c + 2);
        }
        {
            const uint32_t par = (c >> 1) & 1;
            bool ok = true;
            if (C.wait_limit <= 0) {
                ok = mbar_test(mbar_addr(st), par);
            } else {
                const long long t0 = clock64();
                while (!mbar_try(mbar_addr(st), par))
                    if (clock64() - t0 > C.wait_limit) {
                        ok = false;
                        break;
                    }
            }
            ok = __all_sync(0xffffffffu, ok);
            if (!ok) {
                if (lane == 0) {
                    atomicOr(C.status, TQ_DEVERR_TIMEOUT);
                    *cta_abort = 1;
                }
                drain(st, par);
                if (c + 1 < my_rounds) drain(st ^ 1, ((c + 1) >> 1) & 1);
                break;
            }
        }
        const int t = tok0 + (4 * c + warp) * kTile;
        if (!page_ok[warp * 2 + st]) continue;
        const int nv = min(kTile, tok1 - t);  // valid tokens of the round
        const uint32_t kbase = sbase + stage_off(st), vbase = kbase + SM::kTileBytes;
        if (nv < kTile) {  // rows past the sequence hold whatever the pool holds: zero the values
            unsigned char *vz = smem + stage_off(st) + SM::kTileBytes;
            for (int e = lane; e < (kTile - nv) * (D / 8); e += 32) {
                const int rr = nv + e / (D / 8), cc = e % (D / 8);
                *reinterpret_cast<uint4 *>(vz + (cc / 8) * kBoxBytes + rr * 128 + (cc % 8) * 16) = make_uint4(0u, 0u, 0u, 0u);
            }
            __syncwarp();
        }
        // ---- scores S[token][head] ----
        float sc[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
        for (int s = 0; s < KS; ++s) {
            const int x = s >> 2, ch = 2 * (s & 3) + kch;
            uint32_t a0, a1, a2, a3;
            ldsm_x4(kbase + x * kBoxBytes + krow * 128 + ((ch ^ (krow & 7)) << 4), a0, a1, a2, a3);
            mma_bf16(sc, a0, a1, a2, a3, qb[s][0], qb[s][1]);
        }
        // ---- mask, online softmax (base 2): lane holds tokens row, row + 8 of heads 2 quad + e ----
        float xs[2][2], p[2][2], alpha[2];
#pragma unroll
        for (int hh = 0; hh < 2; ++hh)
#pragma unroll
            for (int e = 0; e < 2; ++e)
                xs[hh][e] = (2 * quad + e < G) ? ((row + 8 * hh < nv) ? sc[2 * hh + e] * fac : -INFINITY) : 0.f;
#pragma unroll
        for (int e = 0; e < 2; ++e) {
            float mt = fmaxf(xs[0][e], xs[1][e]);
            mt = fmaxf(mt, __shfl_xor_sync(0xffffffffu, mt, 4));
            mt = fmaxf(mt, __shfl_xor_sync(0xffffffffu, mt, 8));
            mt = fmaxf(mt, __shfl_xor_sync(0xffffffffu, mt, 16));
            const float m_new = fmaxf(m_run[e], mt);
            alpha[e] = (m_new != -INFINITY) ? fast_exp2(m_run[e] - m_new) : 1.f;
            float ps = 0.f;
#pragma unroll
            for (int hh = 0; hh < 2; ++hh) {
                p[hh][e] = (m_new != -INFINITY) ? fast_exp2(xs[hh][e] - m_new) : 0.f;
                ps += p[hh][e];
            }
            ps += __shfl_xor_sync(0xffffffffu, ps, 4);
            ps += __shfl_xor_sync(0xffffffffu, ps, 8);
            ps += __shfl_xor_sync(0xffffffffu, ps, 16);
            l_run[e] = l_run[e] * alpha[e] + ps;
            m_run[e] = m_new;
        }
        if (alpha[0] != 1.f || alpha[1] != 1.f) {
#pragma unroll
            for (int mt = 0; mt < KS; ++mt) {
                o[mt][0] *= alpha[0]; o[mt][1] *= alpha[1]; o[mt][2] *= alpha[0]; o[mt][3] *= alpha[1];
            }
        }
        // ---- P as the B operand (tokens x heads), in high and low bf16 parts ----
        uint32_t bh[2], bl[2];
#pragma unroll
        for (int hh = 0; hh < 2; ++hh) {
            const uint32_t hi = pack_bf16x2(p[hh][0], p[hh][1]);
            const __nv_bfloat162 hv = *reinterpret_cast<const __nv_bfloat162 *>(&hi);
            const uint32_t lo = pack_bf16x2(p[hh][0] - __low2float(hv), p[hh][1] - __high2float(hv));
            bh[hh] = movmatrix_trans(hi);
            bl[hh] = movmatrix_trans(lo);
        }
        // ---- O^T[coordinate][head] += V^T P over the coordinate m-tiles ----
#pragma unroll
        for (int mt = 0; mt < KS; ++mt) {
            const int x = mt >> 2, ch = 2 * (mt & 3) + vch;
            uint32_t a0, a1, a2, a3;
            ldsm_x4_trans(vbase + x * kBoxBytes + vrow * 128 + ((ch ^ (vrow & 7)) << 4), a0, a1, a2, a3);
            mma_bf16(o[mt], a0, a1, a2, a3, bh[0], bh[1]);
            mma_bf16(o[mt], a0, a1, a2, a3, bl[0], bl[1]);
        }
    }
    __syncthreads();  // every warp is done with the stages before they hold merge data
    if (*cta_abort) {
        if (tid < G) {
            ml_out[2 * tid] = -INFINITY;
            ml_out[2 * tid + 1] = 0.f;
        }
        return;
    }
    float *red = reinterpret_cast<float *>(smem);
    float *r_m = red;                   // [warps][8]
    float *r_l = r_m + kWarps * 8;      // [warps][8]
    float *r_o = r_l + kWarps * 8;      // [warps][D][8]
    if (row == 0) {
        r_m[warp * 8 + 2 * quad] = m_run[0];
        r_m[warp * 8 + 2 * quad + 1] = m_run[1];
        r_l[warp * 8 + 2 * quad] = l_run[0];
        r_l[warp * 8 + 2 * quad + 1] = l_run[1];
    }
#pragma unroll
    for (int mt = 0; mt < KS; ++mt) {
        const int j = 16 * mt + row;
        r_o[(warp * D + j) * 8 + 2 * quad] = o[mt][0];
        r_o[(warp * D + j) * 8 + 2 * quad + 1] = o[mt][1];
        r_o[(warp * D + j + 8) * 8 + 2 * quad] = o[mt][2];
        r_o[(warp * D + j + 8) * 8 + 2 * quad + 1] = o[mt][3];
    }
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
                acc = fmaf(f, r_o[(w * D + j) * 8 + h], acc);
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

PFN_cuTensorMapEncodeTiled_v12000 tensor_map_encoder(cudaError_t *err)
{
    static std::once_flag once;
    static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
    static cudaError_t e = cudaSuccess;
    std::call_once(once, [] {
        cudaDriverEntryPointQueryResult q;
        void *p = nullptr;
        e = cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q);
        if (e == cudaSuccess && q != cudaDriverEntryPointSuccess) e = cudaErrorSymbolNotFound;
        fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
    });
    *err = e;
    return fn;
}

// A 2-D view [rows][d] of a bf16 pool, fetched in 16 x 64 boxes with the 128-byte swizzle.
bool make_pool_map(CUtensorMap *tm, const void *pool, int d, int64_t rows, cudaError_t *err)
{
    PFN_cuTensorMapEncodeTiled_v12000 enc = tensor_map_encoder(err);
    if (!enc) return false;
    const cuuint64_t gdim[2] = {static_cast<cuuint64_t>(d), static_cast<cuuint64_t>(rows)};
    const cuuint64_t gstride[1] = {static_cast<cuuint64_t>(d) * 2};
    const cuuint32_t box[2] = {static_cast<cuuint32_t>(kBoxCols), static_cast<cuuint32_t>(kTile)};
    const cuuint32_t estr[2] = {1, 1};
    const CUresult r = enc(tm, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void *>(pool), gdim, gstride, box, estr,
                           CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                           CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    if (r != CUDA_SUCCESS) {
        *err = cudaErrorInvalidValue;
        return false;
    }
    return true;
}

template <int D>
cudaError_t launch_bypass(const CUtensorMap &tk, const CUtensorMap &tv, const Codec &c, int P, const DecodeArgs &a,
                          cudaStream_t st)
{
    const size_t smem = BypassSmem<D>::kBytes;
    cudaError_t e = ensure_smem_attr(reinterpret_cast<const void *>(decode_bf16_kernel<D>), smem);
    if (e != cudaSuccess) return e;
    dim3 grid(a.splits, a.Hkv, a.B);
    decode_bf16_kernel<D><<<grid, kThreads, smem, st>>>(tk, tv, c, P, a);
    e = cudaGetLastError();
    if (e != cudaSuccess) return e;
    return launch_combine(c, a, st, false);
}

}  // namespace
}  // namespace tq

extern "C" tq_status tq_decode_attention_bf16(tq_handle h, const uint16_t *q, const uint16_t *k_pool,
                                              const uint16_t *v_pool, const int32_t *block_table,
                                              const int32_t *seq_lens, int batch, int num_q_heads, int num_kv_heads,
                                              int page_size, int max_blocks_per_seq, int64_t num_blocks,
                                              float sm_scale, int splits, void *workspace, size_t ws_bytes,
                                              uint16_t *out, void *stream)
{
    using tq::api_error;
    if (!h) return api_error(TQ_ERR_INVALID_ARG, "tq_decode_attention_bf16: NULL handle");
    const tq::Codec &c = tq::handle_codec(h);
    if (page_size != 16 && page_size != 32)
        return api_error(TQ_ERR_UNSUPPORTED, "tq_decode_attention_bf16: page_size %d not in {16, 32}", page_size);
    if (batch < 0 || num_q_heads < 1 || num_kv_heads < 1 || max_blocks_per_seq < 1 || num_blocks < 1 || splits < 0)
        return api_error(TQ_ERR_INVALID_ARG, "tq_decode_attention_bf16: bad sizes");
    if (num_q_heads % num_kv_heads || num_q_heads / num_kv_heads > 8)
        return api_error(TQ_ERR_UNSUPPORTED,
                         "tq_decode_attention_bf16: num_q_heads / num_kv_heads must be an integer in 1..8");
    if (!(sm_scale == sm_scale) || sm_scale == INFINITY || sm_scale == -INFINITY)
        return api_error(TQ_ERR_INVALID_ARG, "tq_decode_attention_bf16: sm_scale not finite");
    if (batch == 0) return TQ_OK;
    if (batch > 65535 || num_kv_heads > 65535)
        return api_error(TQ_ERR_UNSUPPORTED, "tq_decode_attention_bf16: batch / num_kv_heads above 65535");
    const int64_t rows = num_blocks * num_kv_heads * page_size;
    if (rows >= (int64_t(1) << 31))
        return api_error(TQ_ERR_UNSUPPORTED, "tq_decode_attention_bf16: pool of %lld rows is too large",
                         static_cast<long long>(rows));
    if (!q || !k_pool || !v_pool || !block_table || !seq_lens || !workspace || !out)
        return api_error(TQ_ERR_INVALID_ARG, "tq_decode_attention_bf16: NULL pointer");
    auto al = [](const void *p, uintptr_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; };
    if (!al(q, 16) || !al(k_pool, 16) || !al(v_pool, 16) || !al(block_table, 4) || !al(seq_lens, 4) ||
        !al(workspace, 256) || !al(out, 16))
        return api_error(TQ_ERR_INVALID_ARG, "tq_decode_attention_bf16: misaligned pointer");
    if (splits == 0) splits = tq_decode_splits(h, batch, num_kv_heads, max_blocks_per_seq, page_size);
    if (splits > 1024) return api_error(TQ_ERR_UNSUPPORTED, "tq_decode_attention_bf16: splits %d above 1024", splits);
    const size_t need = tq::decode_workspace_bytes(c.d, batch, num_q_heads, splits);
    if (ws_bytes < need)
        return api_error(TQ_ERR_INVALID_ARG, "tq_decode_attention_bf16: workspace %zu bytes < %zu needed", ws_bytes,
                         need);
    CUtensorMap tk, tv;
    cudaError_t e = cudaSuccess;
    if (!tq::make_pool_map(&tk, k_pool, c.d, rows, &e) || !tq::make_pool_map(&tv, v_pool, c.d, rows, &e))
        return api_error(TQ_ERR_CUDA, "tq_decode_attention_bf16: cuTensorMapEncodeTiled: %s", cudaGetErrorString(e));
    tq::DecodeArgs a{};
    a.q = q;
    a.block_table = block_table;
    a.seq_lens = seq_lens;
    a.B = batch;
    a.Hq = num_q_heads;
    a.Hkv = num_kv_heads;
    a.max_blocks = max_blocks_per_seq;
    a.num_blocks = num_blocks;
    a.sm_scale = sm_scale;
    a.splits = splits;
    a.pages_per_split = (max_blocks_per_seq + splits - 1) / splits;
    a.Tq = 1;
    a.qpc = 1;
    a.ws = tq::carve_decode_workspace(workspace, c.d, batch, num_q_heads, splits);
    a.out = out;
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    e = (c.d == 128) ? tq::launch_bypass<128>(tk, tv, c, page_size, a, st)
                     : tq::launch_bypass<256>(tk, tv, c, page_size, a, st);
    if (e != cudaSuccess) return api_error(TQ_ERR_CUDA, "tq_decode_attention_bf16: launch: %s", cudaGetErrorString(e));
    return TQ_OK;
}
