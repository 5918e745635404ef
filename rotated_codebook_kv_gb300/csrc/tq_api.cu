// tq_api.cu -- the C ABI declared in include/tq.h: argument validation, table
// upload, workspace carve-up and kernel launches.  No call on the hot path
// synchronises or allocates.
#include <cmath>
#include <cstdarg>
#include <cstdio>
#include <cstring>
#include <map>
#include <mutex>
#include <string>
#include <utility>
#include <vector>

#include <cuda_fp16.h>
#include <cuda_runtime.h>

#include "tq.h"
#include "tq_internal.h"

struct tq_ctx {
    tq::Codec codec;
    void *dev_tables;      // Pi, PiT, S, ST (fp32) then the status word
    void *static_scratch;  // device address of the no-allocation decode's array in this handle's context
    int device;
    int num_sms;
    uint64_t seed;
};

namespace {

thread_local std::string g_last_error;

tq_status fail(tq_status s, const char *fmt, ...)
{
    char buf[512];
    va_list ap;
    va_start(ap, fmt);
    vsnprintf(buf, sizeof buf, fmt, ap);
    va_end(ap);
    g_last_error = buf;
    return s;
}

tq_status cuda_fail(cudaError_t e, const char *what)
{
    return fail(TQ_ERR_CUDA, "%s: %s", what, cudaGetErrorString(e));
}

bool aligned(const void *p, size_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }

bool supported_bits(int b) { return b >= 2 && b <= 4; }

// The scale s in [1, 2) (steps of 2^-16) that brings every s * c closest, relative
// to its size, to an fp16 value: decode multiplies fp16(s c) and divides s out
// once at the end, so the centroids lose less than the 2^-12 of a plain fp16 rounding.
float fp16_friendly_scale(const double *c, int n)
{
    double best = 1e300;
    float best_s = 1.f;
    for (int k = 0; k < 65536; ++k) {
        const float sc = 1.f + static_cast<float>(k) / 65536.f;
        double worst = 0.0;
        for (int i = 0; i < n && worst < best; ++i) {
            const double x = static_cast<double>(sc) * c[i];
            if (x == 0.0) continue;
            const double h = static_cast<double>(__half2float(__float2half_rn(static_cast<float>(x))));
            worst = std::fmax(worst, std::fabs(h - x) / std::fabs(x));
        }
        if (worst < best) {
            best = worst;
            best_s = sc;
        }
    }
    return best_s;
}

}  // namespace

void *tq::handle_static_scratch(tq_handle h) { return h ? h->static_scratch : nullptr; }

const tq::Codec &tq::handle_codec(tq_handle h) { return h->codec; }

cudaError_t tq::ensure_smem_attr(const void *func, size_t bytes)
{
    static std::mutex lock;
    static std::map<std::pair<const void *, int>, size_t> granted;  // (kernel, device) -> bytes
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    std::lock_guard<std::mutex> guard(lock);
    size_t &g = granted[std::make_pair(func, dev)];
    if (g >= bytes) return cudaSuccess;
    e = cudaFuncSetAttribute(func, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(bytes));
    if (e == cudaSuccess) g = bytes;
    return e;
}

tq_status tq::api_error(tq_status s, const char *fmt, ...)
{
    char buf[512];
    va_list ap;
    va_start(ap, fmt);
    vsnprintf(buf, sizeof buf, fmt, ap);
    va_end(ap);
    g_last_error = buf;
    return s;
}

extern "C" {

const char *tq_last_error(void) { return g_last_error.c_str(); }

tq_status tq_init(int head_dim, int k_bits, int v_bits, int group, uint64_t seed, tq_handle *out)
{
    return tq_init_ex(head_dim, k_bits, v_bits, group, seed, 0u, out);
}

tq_status tq_init_ex(int head_dim, int k_bits, int v_bits, int group, uint64_t seed, unsigned flags, tq_handle *out)
{
    if (!out) return fail(TQ_ERR_INVALID_ARG, "tq_init: out is NULL");
    *out = nullptr;
    if (flags & ~(TQ_ROTATION_HADAMARD | TQ_VALUES_MSE))
        return fail(TQ_ERR_UNSUPPORTED, "tq_init: unknown flags 0x%x", flags);
    const int rotation = (flags & TQ_ROTATION_HADAMARD) ? 1 : 0;
    const bool vmse = (flags & TQ_VALUES_MSE) != 0;
    if (head_dim != 128 && head_dim != 256)
        return fail(TQ_ERR_UNSUPPORTED, "tq_init: head_dim %d not in {128, 256}", head_dim);
    if (!supported_bits(k_bits) || !supported_bits(v_bits))
        return fail(TQ_ERR_UNSUPPORTED, "tq_init: k_bits %d / v_bits %d not in {2, 3, 4}", k_bits, v_bits);
    if ((group != 32 && group != 64 && group != 128) || head_dim % group)
        return fail(TQ_ERR_UNSUPPORTED, "tq_init: group %d not in {32, 64, 128} or does not divide %d", group,
                    head_dim);
    tq::HostTables ht;
    if (!tq::build_tables(head_dim, k_bits, seed, rotation, &ht))
        return fail(TQ_ERR_CUDA, "tq_init: Lloyd-Max iteration did not converge");
    double vcent[16] = {}, vthr[16] = {};
    if (vmse && !tq::build_codebook(v_bits, vcent, vthr))
        return fail(TQ_ERR_CUDA, "tq_init: Lloyd-Max iteration did not converge");

    const int d = head_dim;
    const size_t dd = static_cast<size_t>(d) * d;
    // fp32 tables: Pi, Pi^T, S, S^T, M_hi, M_lo (M = S Pi in double), then the
    // fp16 tensor-core operand image (d = 128) and the status word.
    const size_t img_bytes = (d == 128) ? 4 * dd * sizeof(uint16_t) : 0;
    const size_t nf = 6 * dd + static_cast<size_t>(d);  // six d x d tables, then the Hadamard signs
    std::vector<float> host(nf);
    std::vector<double> Md(dd);  // M = S Pi in double
    for (int j = 0; j < d; ++j) host[6 * dd + j] = static_cast<float>(ht.hsign[j]);
    for (int i = 0; i < d; ++i)
        for (int j = 0; j < d; ++j) {
            const size_t a = static_cast<size_t>(i) * d + j, t = static_cast<size_t>(j) * d + i;
            host[a] = static_cast<float>(ht.Pi[a]);
            host[dd + t] = static_cast<float>(ht.Pi[a]);
            host[2 * dd + a] = static_cast<float>(ht.S[a]);
            host[3 * dd + t] = static_cast<float>(ht.S[a]);
            double m = 0.0;
            for (int q = 0; q < d; ++q) m += ht.S[static_cast<size_t>(i) * d + q] * ht.Pi[static_cast<size_t>(q) * d + j];
            Md[a] = m;
            const float mh = static_cast<float>(m);
            host[4 * dd + a] = mh;
            host[5 * dd + a] = static_cast<float>(m - static_cast<double>(mh));
        }
    std::vector<uint16_t> img(img_bytes / 2);
    if (d == 128) {
        // B operands (rows = output index i, K = input index j), core matrices of
        // 8 rows x 8 halfs, row groups of 16 k-chunks: Pi 2^10 and S 2^12 as fp16 hi + lo.
        auto put = [&](int term, int i, int j, double x) {
            const size_t off = ((static_cast<size_t>(i >> 3) * (d >> 3) + (j >> 3)) * 128 + (i & 7) * 16 + (j & 7) * 2) / 2;
            const __half h = __float2half_rn(static_cast<float>(x));
            const __half l = __float2half_rn(static_cast<float>(x - static_cast<double>(__half2float(h))));
            img[(2 * term) * dd + off] = __half_as_ushort(h);
            img[(2 * term + 1) * dd + off] = __half_as_ushort(l);
        };
        for (int i = 0; i < d; ++i)
            for (int j = 0; j < d; ++j) {
                put(0, i, j, ht.Pi[static_cast<size_t>(i) * d + j] * 1024.0);
                put(1, i, j, ht.S[static_cast<size_t>(i) * d + j] * 4096.0);
            }
    }
    // Pi 2^10, M 2^10 (M = S Pi), S 2^12, Pi^T 2^10 and S^T 2^12 as fp16 high / low parts in the fragment
    // order of mma.sync m16n8k16's B operand (B[k][n] = W[n][k]): for n-tile nt, k-step
    // ks and lane (r, q) the pairs (k0, k0 + 1) and (k0 + 8, k0 + 9) of row n = 8 nt + r,
    // k0 = 16 ks + 2 q
    const size_t frag_one = static_cast<size_t>(d / 8) * (d / 16) * 32 * 4;
    const size_t frag_words = 5 * frag_one;
    std::vector<uint32_t> frag(frag_words);
    for (int mat = 0; mat < 5; ++mat) {
        // W[n][k]: Pi, M, S, then the transposes Pi^T and S^T (W[n][k] = Pi[k][n], S[k][n])
        const double *W = mat == 0 ? ht.Pi.data() : (mat == 1 ? Md.data() : (mat == 3 ? ht.Pi.data() : ht.S.data()));
        const bool tr = mat >= 3;
        const double scale = (mat == 2 || mat == 4) ? 4096.0 : 1024.0;
        auto hl = [&](int n, int kk, uint16_t *hi, uint16_t *lo) {
            const double x = W[tr ? static_cast<size_t>(kk) * d + n : static_cast<size_t>(n) * d + kk] * scale;
            const __half h = __float2half_rn(static_cast<float>(x));
            *hi = __half_as_ushort(h);
            *lo = __half_as_ushort(__float2half_rn(static_cast<float>(x - static_cast<double>(__half2float(h)))));
        };
        size_t w = mat * frag_one;
        for (int nt = 0; nt < d / 8; ++nt)
            for (int ks = 0; ks < d / 16; ++ks)
                for (int lane = 0; lane < 32; ++lane) {
                    const int n = 8 * nt + lane / 4, k0 = 16 * ks + 2 * (lane % 4);
                    uint16_t h[4], l[4];
                    hl(n, k0, &h[0], &l[0]);
                    hl(n, k0 + 1, &h[1], &l[1]);
                    hl(n, k0 + 8, &h[2], &l[2]);
                    hl(n, k0 + 9, &h[3], &l[3]);
                    frag[w++] = h[0] | (static_cast<uint32_t>(h[1]) << 16);
                    frag[w++] = h[2] | (static_cast<uint32_t>(h[3]) << 16);
                    frag[w++] = l[0] | (static_cast<uint32_t>(l[1]) << 16);
                    frag[w++] = l[2] | (static_cast<uint32_t>(l[3]) << 16);
                }
    }
    tq_ctx *c = new tq_ctx();
    cudaError_t e = cudaGetDevice(&c->device);
    if (e == cudaSuccess) e = cudaDeviceGetAttribute(&c->num_sms, cudaDevAttrMultiProcessorCount, c->device);
    if (e != cudaSuccess) {
        delete c;
        return cuda_fail(e, "tq_init: device query");
    }
    // the no-allocation decode's static array: its device address in this context
    e = tq::static_scratch_lookup(&c->static_scratch);
    if (e != cudaSuccess) {
        delete c;
        return cuda_fail(e, "tq_init: cudaGetSymbolAddress of the static decode scratch");
    }
    e = cudaMalloc(&c->dev_tables, nf * sizeof(float) + img_bytes + frag_words * 4 + 256);
    if (e != cudaSuccess) {
        delete c;
        return fail(TQ_ERR_OOM, "tq_init: cudaMalloc: %s", cudaGetErrorString(e));
    }
    float *base = static_cast<float *>(c->dev_tables);
    e = cudaMemcpy(base, host.data(), nf * sizeof(float), cudaMemcpyHostToDevice);
    char *img_dev = reinterpret_cast<char *>(base + nf);
    if (e == cudaSuccess && img_bytes) e = cudaMemcpy(img_dev, img.data(), img_bytes, cudaMemcpyHostToDevice);
    char *frag_dev = img_dev + img_bytes;
    if (e == cudaSuccess) e = cudaMemcpy(frag_dev, frag.data(), frag_words * 4, cudaMemcpyHostToDevice);
    unsigned *status = reinterpret_cast<unsigned *>(frag_dev + frag_words * 4);
    if (e == cudaSuccess) e = cudaMemset(status, 0, 256);
    if (e == cudaSuccess) e = cudaDeviceSynchronize();
    if (e != cudaSuccess) {
        cudaFree(c->dev_tables);
        delete c;
        return cuda_fail(e, "tq_init: upload");
    }
    tq::Codec &k = c->codec;
    std::memset(&k, 0, sizeof k);
    k.d = d;
    k.k_bits = k_bits;
    k.v_bits = v_bits;
    k.group = group;
    k.qjl = (k_bits <= 3);
    k.k_code_bytes = d * k_bits / 8;
    k.k_sign_bytes = k.qjl ? d / 8 : 0;
    k.v_code_bytes = d * v_bits / 8;
    k.vmse = vmse ? 1 : 0;
    k.v_meta_bytes = vmse ? 2 : (d / group) * 4;  // a bf16 norm, or (scale, zero) per group
    for (int i = 0; vmse && i < (1 << v_bits); ++i) k.vcentroids[i] = static_cast<float>(vcent[i]);
    for (int i = 0; vmse && i + 1 < (1 << v_bits); ++i) k.vthresholds[i] = static_cast<float>(vthr[i]);
    k.vlut_scale = vmse ? fp16_friendly_scale(vcent, 1 << v_bits) : 1.f;
    for (int i = 0; i < (1 << k_bits); ++i) k.centroids[i] = static_cast<float>(ht.centroids[i]);
    for (int i = 0; i + 1 < (1 << k_bits); ++i) k.thresholds[i] = static_cast<float>(ht.thresholds[i]);
    k.Pi = base;
    k.PiT = base + dd;
    k.S = base + 2 * dd;
    k.ST = base + 3 * dd;
    k.M_hi = base + 4 * dd;
    k.M_lo = base + 5 * dd;
    k.tc_image = img_bytes ? img_dev : nullptr;
    k.hsign = base + 6 * dd;
    k.pi_frag = reinterpret_cast<const uint4 *>(frag_dev);
    k.m_frag = reinterpret_cast<const uint4 *>(frag_dev) + frag_one / 4;
    k.s_frag = reinterpret_cast<const uint4 *>(frag_dev) + 2 * (frag_one / 4);
    k.pit_frag = reinterpret_cast<const uint4 *>(frag_dev) + 3 * (frag_one / 4);
    k.st_frag = reinterpret_cast<const uint4 *>(frag_dev) + 4 * (frag_one / 4);
    k.rotation = rotation;
    k.status = status;
    k.wait_limit = tq::kDefaultWaitLimit;
    k.num_sms = c->num_sms;
    c->seed = seed;
    *out = c;
    return TQ_OK;
}

tq_status tq_destroy(tq_handle h)
{
    if (!h) return TQ_OK;
    cudaError_t e = cudaFree(h->dev_tables);
    delete h;
    if (e != cudaSuccess) return cuda_fail(e, "tq_destroy");
    return TQ_OK;
}

tq_status tq_cache_layout(tq_handle h, int page_size, size_t *k_page_bytes, size_t *v_page_bytes)
{
    if (!h || !k_page_bytes || !v_page_bytes) return fail(TQ_ERR_INVALID_ARG, "tq_cache_layout: NULL argument");
    if (page_size != 16 && page_size != 32)
        return fail(TQ_ERR_UNSUPPORTED, "tq_cache_layout: page_size %d not in {16, 32}", page_size);
    const tq::PageGeom g = tq::page_geom(h->codec, page_size);
    *k_page_bytes = static_cast<size_t>(g.k_page);
    *v_page_bytes = static_cast<size_t>(g.v_page);
    return TQ_OK;
}

tq_status tq_compress_kv(tq_handle h, const uint16_t *k, const uint16_t *v, int64_t T, int num_kv_heads,
                         int64_t k_stride_tok, int64_t v_stride_tok, const int64_t *slot_mapping, uint8_t *k_cache,
                         uint8_t *v_cache, int page_size, int64_t num_blocks, void *stream)
{
    if (!h) return fail(TQ_ERR_INVALID_ARG, "tq_compress_kv: NULL handle");
    if (page_size != 16 && page_size != 32)
        return fail(TQ_ERR_UNSUPPORTED, "tq_compress_kv: page_size %d not in {16, 32}", page_size);
    if (T < 0 || num_kv_heads < 1 || num_blocks < 1)
        return fail(TQ_ERR_INVALID_ARG, "tq_compress_kv: T=%lld num_kv_heads=%d num_blocks=%lld",
                    static_cast<long long>(T), num_kv_heads, static_cast<long long>(num_blocks));
    if (T == 0) return TQ_OK;
    const int d = h->codec.d;
    if (!k || !v || !slot_mapping || !k_cache || !v_cache)
        return fail(TQ_ERR_INVALID_ARG, "tq_compress_kv: NULL pointer");
    if (!aligned(k, 16) || !aligned(v, 16) || !aligned(k_cache, 16) || !aligned(v_cache, 16) ||
        !aligned(slot_mapping, 8))
        return fail(TQ_ERR_INVALID_ARG, "tq_compress_kv: k, v and the caches must be 16-byte aligned");
    if (k_stride_tok < static_cast<int64_t>(num_kv_heads) * d || v_stride_tok < static_cast<int64_t>(num_kv_heads) * d ||
        k_stride_tok % 8 || v_stride_tok % 8)
        return fail(TQ_ERR_INVALID_ARG,
                    "tq_compress_kv: token strides must be >= num_kv_heads*head_dim and multiples of 8 elements");
    if (T * num_kv_heads / 32 >= (int64_t(1) << 31))
        return fail(TQ_ERR_UNSUPPORTED, "tq_compress_kv: too many token-heads in one call");
    const tq::PageGeom g = tq::page_geom(h->codec, page_size);
    cudaError_t e = tq::launch_compress(h->codec, g, k, v, T, num_kv_heads, k_stride_tok, v_stride_tok, slot_mapping,
                                        k_cache, v_cache, num_blocks, static_cast<cudaStream_t>(stream));
    if (e != cudaSuccess) return cuda_fail(e, "tq_compress_kv: launch");
    return TQ_OK;
}

tq_status tq_dequant_kv(tq_handle h, const uint8_t *k_cache, const uint8_t *v_cache, int page_size,
                        int64_t num_blocks, int num_kv_heads, const int64_t *slots, int64_t T, uint16_t *k_out,
                        uint16_t *v_out, void *stream)
{
    if (!h) return fail(TQ_ERR_INVALID_ARG, "tq_dequant_kv: NULL handle");
    if (page_size != 16 && page_size != 32)
        return fail(TQ_ERR_UNSUPPORTED, "tq_dequant_kv: page_size %d not in {16, 32}", page_size);
    if (T < 0 || num_kv_heads < 1 || num_blocks < 1)
        return fail(TQ_ERR_INVALID_ARG, "tq_dequant_kv: bad sizes");
    if (T == 0) return TQ_OK;
    if (!k_cache || !v_cache || !slots || !k_out || !v_out)
        return fail(TQ_ERR_INVALID_ARG, "tq_dequant_kv: NULL pointer");
    if (!aligned(k_cache, 16) || !aligned(v_cache, 16) || !aligned(slots, 8) || !aligned(k_out, 16) ||
        !aligned(v_out, 16))
        return fail(TQ_ERR_INVALID_ARG, "tq_dequant_kv: misaligned pointer");
    if (T >= (int64_t(1) << 31) || num_kv_heads > 65535)
        return fail(TQ_ERR_UNSUPPORTED, "tq_dequant_kv: too many slots in one call");
    const tq::PageGeom g = tq::page_geom(h->codec, page_size);
    cudaError_t e = tq::launch_dequant(h->codec, g, k_cache, v_cache, num_blocks, num_kv_heads, slots, T, k_out, v_out,
                                       static_cast<cudaStream_t>(stream));
    if (e != cudaSuccess) return cuda_fail(e, "tq_dequant_kv: launch");
    return TQ_OK;
}

int tq_decode_splits(tq_handle h, int batch, int num_kv_heads, int max_blocks_per_seq, int page_size)
{
    if (!h || batch < 1 || num_kv_heads < 1 || max_blocks_per_seq < 1 || page_size < 1) return 1;
    const int units = batch * num_kv_heads;
    int splits = (8 * h->num_sms + units - 1) / units;  // about eight CTAs per SM
    // resident decode CTAs per SM: 4 at d = 128, 2 at d = 256 (registers).  A last
    // wave less than half full mostly idles the GPU: round up to whole waves.
    const int slots = h->num_sms * (h->codec.d == 128 ? 4 : 2);
    const long long ctas = static_cast<long long>(units) * splits;
    const long long waves = (ctas + slots - 1) / slots;
    if (ctas % slots != 0 && 2 * (ctas - (waves - 1) * slots) < slots)
        splits = static_cast<int>((waves * slots + units - 1) / units);
    if (splits > 64) splits = 64;
    if (splits > max_blocks_per_seq) splits = max_blocks_per_seq;
    return splits < 1 ? 1 : splits;
}

size_t tq_decode_workspace_bytes(tq_handle h, int batch, int num_q_heads, int splits)
{
    if (!h || batch < 0 || num_q_heads < 0 || splits < 1) return 0;
    return tq::decode_workspace_bytes(h->codec.d, batch, num_q_heads, splits);
}

tq_status tq_decode_attention(tq_handle h, const uint16_t *q, const uint8_t *k_cache, const uint8_t *v_cache,
                              const int32_t *block_table, const int32_t *seq_lens, int batch, int num_q_heads,
                              int num_kv_heads, int page_size, int max_blocks_per_seq, int64_t num_blocks,
                              float sm_scale, int splits, void *workspace, size_t ws_bytes, uint16_t *out,
                              void *stream)
{
    if (!h) return fail(TQ_ERR_INVALID_ARG, "tq_decode_attention: NULL handle");
    if (page_size != 16 && page_size != 32)
        return fail(TQ_ERR_UNSUPPORTED, "tq_decode_attention: page_size %d not in {16, 32}", page_size);
    if (batch < 0 || num_q_heads < 1 || num_kv_heads < 1 || max_blocks_per_seq < 1 || num_blocks < 1 || splits < 0)
        return fail(TQ_ERR_INVALID_ARG, "tq_decode_attention: bad sizes");
    if (num_q_heads % num_kv_heads || num_q_heads / num_kv_heads > 8)
        return fail(TQ_ERR_UNSUPPORTED, "tq_decode_attention: num_q_heads / num_kv_heads must be an integer in 1..8");
    if (!std::isfinite(sm_scale)) return fail(TQ_ERR_INVALID_ARG, "tq_decode_attention: sm_scale not finite");
    if (batch == 0) return TQ_OK;
    if (batch > 65535 || num_kv_heads > 65535)
        return fail(TQ_ERR_UNSUPPORTED, "tq_decode_attention: batch / num_kv_heads above 65535");
    if (!q || !k_cache || !v_cache || !block_table || !seq_lens || !workspace || !out)
        return fail(TQ_ERR_INVALID_ARG, "tq_decode_attention: NULL pointer");
    if (!aligned(q, 16) || !aligned(k_cache, 16) || !aligned(v_cache, 16) || !aligned(block_table, 4) ||
        !aligned(seq_lens, 4) || !aligned(workspace, 256) || !aligned(out, 16))
        return fail(TQ_ERR_INVALID_ARG, "tq_decode_attention: misaligned pointer");
    if (splits == 0) splits = tq_decode_splits(h, batch, num_kv_heads, max_blocks_per_seq, page_size);
    if (splits > 1024) return fail(TQ_ERR_UNSUPPORTED, "tq_decode_attention: splits %d above 1024", splits);
    const size_t need = tq::decode_workspace_bytes(h->codec.d, batch, num_q_heads, splits);
    if (ws_bytes < need)
        return fail(TQ_ERR_INVALID_ARG, "tq_decode_attention: workspace %zu bytes < %zu needed", ws_bytes, need);
    tq::DecodeArgs a;
    a.q = q;
    a.k_cache = k_cache;
    a.v_cache = v_cache;
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
    a.ws = tq::carve_decode_workspace(workspace, h->codec.d, batch, num_q_heads, splits);
    a.out = out;
    const tq::PageGeom g = tq::page_geom(h->codec, page_size);
    cudaError_t e = tq::launch_decode(h->codec, g, a, static_cast<cudaStream_t>(stream));
    if (e != cudaSuccess) return cuda_fail(e, "tq_decode_attention: launch");
    return TQ_OK;
}

int tq_prefill_queries_per_cta(tq_handle h, int num_q_heads, int num_kv_heads)
{
    if (!h || num_kv_heads < 1 || num_q_heads < num_kv_heads) return 1;
    const int G = num_q_heads / num_kv_heads;
    if (h->codec.d == 128) return 128 / G;  // the tensor-memory kernel's 128 columns
    return G >= 8 ? 1 : 8 / G;
}

int tq_prefill_splits(tq_handle h, int batch, int q_tokens, int num_q_heads, int num_kv_heads,
                      int max_blocks_per_seq, int page_size)
{
    if (!h || batch < 1 || q_tokens < 1 || num_kv_heads < 1 || num_q_heads < num_kv_heads || max_blocks_per_seq < 1 ||
        page_size < 1)
        return 1;
    const int qpc = tq_prefill_queries_per_cta(h, num_q_heads, num_kv_heads);
    const long long units_z = static_cast<long long>(batch) * ((q_tokens + qpc - 1) / qpc);
    if (h->codec.d != 128)
        return tq_decode_splits(h, static_cast<int>(units_z < 65535 ? units_z : 65535), num_kv_heads,
                                max_blocks_per_seq, page_size);
    // one CTA per SM: about two waves, each split keeping at least four 64-token tiles
    const long long units = units_z * num_kv_heads;
    long long splits = (2LL * h->num_sms + units - 1) / units;
    const int tiles = (max_blocks_per_seq * page_size + 63) / 64;
    const int most = tiles / 4 > 1 ? tiles / 4 : 1;
    if (splits > most) splits = most;
    if (splits > 64) splits = 64;
    return splits < 1 ? 1 : static_cast<int>(splits);
}

tq_status tq_prefill_attention(tq_handle h, const uint16_t *q, const uint8_t *k_cache, const uint8_t *v_cache,
                               const int32_t *block_table, const int32_t *seq_lens, int batch, int q_tokens,
                               int num_q_heads, int num_kv_heads, int page_size, int max_blocks_per_seq,
                               int64_t num_blocks, float sm_scale, int splits, void *workspace, size_t ws_bytes,
                               uint16_t *out, void *stream)
{
    if (!h) return fail(TQ_ERR_INVALID_ARG, "tq_prefill_attention: NULL handle");
    if (page_size != 16 && page_size != 32)
        return fail(TQ_ERR_UNSUPPORTED, "tq_prefill_attention: page_size %d not in {16, 32}", page_size);
    if (batch < 0 || q_tokens < 1 || num_q_heads < 1 || num_kv_heads < 1 || max_blocks_per_seq < 1 ||
        num_blocks < 1 || splits < 0)
        return fail(TQ_ERR_INVALID_ARG, "tq_prefill_attention: bad sizes");
    if (num_q_heads % num_kv_heads || num_q_heads / num_kv_heads > 8)
        return fail(TQ_ERR_UNSUPPORTED, "tq_prefill_attention: num_q_heads / num_kv_heads must be an integer in 1..8");
    if (!std::isfinite(sm_scale)) return fail(TQ_ERR_INVALID_ARG, "tq_prefill_attention: sm_scale not finite");
    if (batch == 0) return TQ_OK;
    const int qpc = tq_prefill_queries_per_cta(h, num_q_heads, num_kv_heads);
    const int64_t ctas_z = static_cast<int64_t>(batch) * ((q_tokens + qpc - 1) / qpc);
    if (ctas_z > 65535 || num_kv_heads > 65535 || static_cast<int64_t>(batch) * q_tokens * num_q_heads >= (1LL << 31))
        return fail(TQ_ERR_UNSUPPORTED, "tq_prefill_attention: too many sequences x query tokens in one call");
    if (!q || !k_cache || !v_cache || !block_table || !seq_lens || !workspace || !out)
        return fail(TQ_ERR_INVALID_ARG, "tq_prefill_attention: NULL pointer");
    if (!aligned(q, 16) || !aligned(k_cache, 16) || !aligned(v_cache, 16) || !aligned(block_table, 4) ||
        !aligned(seq_lens, 4) || !aligned(workspace, 256) || !aligned(out, 16))
        return fail(TQ_ERR_INVALID_ARG, "tq_prefill_attention: misaligned pointer");
    if (splits == 0)
        splits = tq_prefill_splits(h, batch, q_tokens, num_q_heads, num_kv_heads, max_blocks_per_seq, page_size);
    if (splits > 1024) return fail(TQ_ERR_UNSUPPORTED, "tq_prefill_attention: splits %d above 1024", splits);
    const size_t need = tq::decode_workspace_bytes(h->codec.d, batch * q_tokens, num_q_heads, splits);
    if (ws_bytes < need)
        return fail(TQ_ERR_INVALID_ARG, "tq_prefill_attention: workspace %zu bytes < %zu needed", ws_bytes, need);
    tq::DecodeArgs a;
    a.q = q;
    a.k_cache = k_cache;
    a.v_cache = v_cache;
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
    a.Tq = q_tokens;
    a.qpc = qpc;
    a.ws = tq::carve_decode_workspace(workspace, h->codec.d, batch * q_tokens, num_q_heads, splits);
    a.out = out;
    const tq::PageGeom g = tq::page_geom(h->codec, page_size);
    cudaError_t e = tq::launch_decode(h->codec, g, a, static_cast<cudaStream_t>(stream));
    if (e != cudaSuccess) return cuda_fail(e, "tq_prefill_attention: launch");
    return TQ_OK;
}

tq_status tq_set_wait_limit(tq_handle h, int64_t cycles)
{
    if (!h) return fail(TQ_ERR_INVALID_ARG, "tq_set_wait_limit: NULL handle");
    if (cycles < 0) return fail(TQ_ERR_INVALID_ARG, "tq_set_wait_limit: negative limit");
    h->codec.wait_limit = cycles;
    return TQ_OK;
}

tq_status tq_get_status(tq_handle h, uint32_t *device_error_bits, void *stream)
{
    if (!h || !device_error_bits) return fail(TQ_ERR_INVALID_ARG, "tq_get_status: NULL argument");
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    cudaError_t e = cudaStreamSynchronize(st);
    unsigned v = 0;
    if (e == cudaSuccess) e = cudaMemcpy(&v, h->codec.status, sizeof v, cudaMemcpyDeviceToHost);
    if (e == cudaSuccess) e = cudaMemset(h->codec.status, 0, sizeof v);
    if (e == cudaSuccess) e = cudaDeviceSynchronize();
    if (e != cudaSuccess) return cuda_fail(e, "tq_get_status");
    *device_error_bits = v;
    return TQ_OK;
}

tq_status tq_export_params(tq_handle h, float *Pi, float *S, float *centroids, float *thresholds)
{
    if (!h) return fail(TQ_ERR_INVALID_ARG, "tq_export_params: NULL handle");
    const size_t dd = static_cast<size_t>(h->codec.d) * h->codec.d;
    cudaError_t e = cudaSuccess;
    if (Pi) e = cudaMemcpy(Pi, h->codec.Pi, dd * sizeof(float), cudaMemcpyDeviceToHost);
    if (S && e == cudaSuccess) e = cudaMemcpy(S, h->codec.S, dd * sizeof(float), cudaMemcpyDeviceToHost);
    if (e != cudaSuccess) return cuda_fail(e, "tq_export_params");
    const int L = 1 << h->codec.k_bits;
    if (centroids) std::memcpy(centroids, h->codec.centroids, L * sizeof(float));
    if (thresholds) std::memcpy(thresholds, h->codec.thresholds, (L - 1) * sizeof(float));
    return TQ_OK;
}

}  // extern "C"
