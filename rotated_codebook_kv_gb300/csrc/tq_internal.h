// tq_internal.h -- declarations shared by the library's translation units.
#pragma once

#include <cstdint>
#include <vector>

#include <cuda_runtime.h>

#include "tq.h"

namespace tq {

// Records a printf-style message as this thread's tq_last_error() and returns s.
tq_status api_error(tq_status s, const char *fmt, ...);

// Host tables in double, built by tq_params.cpp.
struct HostTables {
    std::vector<double> Pi, S, centroids, thresholds;
    std::vector<double> hsign;  // Hadamard rotation: the random signs D (all +1 for the dense rotation)
};
bool build_tables(int d, int k_bits, uint64_t seed, int rotation, HostTables *out);
bool build_codebook(int bits, double *centroids, double *thresholds);

// Codec constants, passed by value to every kernel.
struct Codec {
    int d, k_bits, v_bits, group, qjl;
    int k_code_bytes, k_sign_bytes, v_code_bytes, v_meta_bytes;  // per token-head
    float centroids[16];   // N(0,1) units, ascending
    float thresholds[16];  // 2^k_bits - 1 used
    const float *Pi;       // [d][d] row-major: y_i = sum_j Pi[i][j] k_j
    const float *PiT;      // [d][d] transpose of Pi
    const float *S;        // [d][d] row-major QJL matrix
    const float *ST;       // [d][d] transpose of S
    const float *M_hi;     // [d][d] M = S Pi (double) as hi + lo fp32, row-major
    const float *M_lo;
    const void *tc_image;  // d = 128: fp16 tensor-core operands (Pi 2^10 hi/lo, S 2^12 hi/lo), core-matrix layout
    const float *hsign;    // [d] random signs of the Hadamard rotation (Pi = H diag(hsign) / sqrt(d))
    const uint4 *pi_frag;  // Pi 2^10 as fp16 high / low mma.sync B fragments: [d/8 n-tiles][d/16 k-steps][32 lanes]
    const uint4 *m_frag;   // M 2^10 (M = S Pi) in the same fragment image
    const uint4 *s_frag;   // S 2^12 in the same fragment image
    const uint4 *pit_frag; // Pi^T 2^10 in the same fragment image (y = Pi^T x)
    const uint4 *st_frag;  // S^T 2^12 in the same fragment image
    int rotation;          // 0: dense Haar, 1: randomized Hadamard
    int vmse;              // values coded by the rotation and a Lloyd-Max codebook (TQ_VALUES_MSE)
    float vcentroids[16];  // value codebook (vmse), N(0,1) units, ascending
    float vthresholds[16];
    float vlut_scale;      // vmse: decode keeps fp16(vlut_scale * c) (a scale chosen so these are near fp16 points)
    unsigned int *status;  // device status word (TQ_DEVERR_* bits)
    long long wait_limit;  // clock cycles a kernel waits on one barrier before it reports TQ_DEVERR_TIMEOUT
    int num_sms;
};

// Byte offsets of the sub-arrays of one (block, kv head) page record.
struct PageGeom {
    int P;
    int64_t k_page, v_page;
    int64_t k_sign_off, k_norm_off, k_gamma_off;  // codes start at 0
    int64_t v_meta_off;                           // codes start at 0
};

inline PageGeom page_geom(const Codec &c, int P)
{
    PageGeom g;
    g.P = P;
    g.k_sign_off = static_cast<int64_t>(P) * c.k_code_bytes;
    g.k_norm_off = g.k_sign_off + static_cast<int64_t>(P) * c.k_sign_bytes;
    g.k_gamma_off = g.k_norm_off + 2LL * P;
    g.k_page = g.k_gamma_off + (c.qjl ? 2LL * P : 0);
    g.v_meta_off = static_cast<int64_t>(P) * c.v_code_bytes;
    g.v_page = g.v_meta_off + static_cast<int64_t>(P) * c.v_meta_bytes;
    return g;
}

// Workspace carve-up of tq_decode_attention (all fp32, 256-byte aligned pieces).
struct DecodeWorkspace {
    float *out32; // [B][Hq][d] the outputs in fp32, before the bf16 rounding (offset 0 of the workspace)
    float *qrot;  // [B][Hq][d]
    float *qs;    // [B][Hq][d]
    float *acc;   // [splits][B][Hq][d] unnormalised partial outputs
    float *ml;    // [splits][B][Hq][2] running max and denominator
};
size_t decode_workspace_bytes(int d, int B, int Hq, int splits);
DecodeWorkspace carve_decode_workspace(void *base, int d, int B, int Hq, int splits);

struct DecodeArgs {
    const uint16_t *q;
    const uint8_t *k_cache, *v_cache;
    const int32_t *block_table, *seq_lens;
    int B, Hq, Hkv, max_blocks;
    int64_t num_blocks;
    float sm_scale;
    int splits, pages_per_split;
    int Tq, qpc;  // query tokens per sequence (1 for decode; the last Tq positions, causal) and per CTA
    DecodeWorkspace ws;
    uint16_t *out;
};

cudaError_t launch_compress(const Codec &c, const PageGeom &pg, const uint16_t *k, const uint16_t *v, int64_t T,
                            int Hkv, int64_t ks, int64_t vs, const int64_t *slots, uint8_t *kc, uint8_t *vc,
                            int64_t num_blocks, cudaStream_t st);

cudaError_t launch_compress_tc(const Codec &c, const PageGeom &pg, const uint16_t *k, const uint16_t *v, int64_t T,
                               int Hkv, int64_t ks, int64_t vs, const int64_t *slots, uint8_t *kc, uint8_t *vc,
                               int64_t num_blocks, int num_sms, cudaStream_t st);
// The same kernel on key records alone (no value pass): keys, or MSE-coded values given
// as keys through a codec whose key fields hold the value codebook.
cudaError_t launch_compress_tc_keys(const Codec &c, const PageGeom &pg, const uint16_t *k, int64_t T, int Hkv,
                                    int64_t ks, const int64_t *slots, uint8_t *kc, int64_t num_blocks, int num_sms,
                                    cudaStream_t st);
// Group-quantised value records alone, head dim 128 or 256 (the keys taking a keys-only pass).
cudaError_t launch_compress_values_tc(const Codec &c, const PageGeom &pg, const uint16_t *v, int64_t T, int Hkv,
                                      int64_t vs, const int64_t *slots, uint8_t *vc, int64_t num_blocks, int num_sms,
                                      cudaStream_t st);

cudaError_t launch_dequant(const Codec &c, const PageGeom &pg, const uint8_t *kc, const uint8_t *vc,
                           int64_t num_blocks, int Hkv, const int64_t *slots, int64_t T, uint16_t *k_out,
                           uint16_t *v_out, cudaStream_t st);

cudaError_t launch_decode(const Codec &c, const PageGeom &pg, const DecodeArgs &a, cudaStream_t st);
// The log-sum-exp merge of split partials into bf16 (and fp32) outputs; with
// `unrotate` the merged output is rotated back by Pi^T (values coded by the rotation).
cudaError_t launch_combine(const Codec &c, const DecodeArgs &a, cudaStream_t st, bool unrotate);
// The split-K decode kernel for values coded by the rotation (its own translation unit).
cudaError_t launch_dmma_vmse(const Codec &c, const PageGeom &pg, const DecodeArgs &a, cudaStream_t st);
// The split-K kernel with several causal query tokens per sequence (prefill at head_dim 256; its own
// translation unit).
cudaError_t launch_dmma_prefill(const Codec &c, const PageGeom &pg, const DecodeArgs &a, cudaStream_t st);
// Prefill at head_dim 128 on the tensor cores with accumulators in tensor memory:
// 128 (query token, head) columns per CTA, qpc = 128 / G query tokens.
cudaError_t launch_prefill_tc(const Codec &c, const PageGeom &pg, const DecodeArgs &a, cudaStream_t st);
size_t prefill_tc_smem_bytes(const PageGeom &pg);

// Device address of the no-allocation decode's static scratch array for the
// context current on the calling thread (looked up, not cached).
cudaError_t static_scratch_lookup(void **out);
// The address tq_init looked up for a handle.
void *handle_static_scratch(tq_handle h);
// The codec constants of a (non-NULL) handle.
const Codec &handle_codec(tq_handle h);

// Sets a kernel's dynamic shared-memory limit once per (function, device); thread safe.
cudaError_t ensure_smem_attr(const void *func, size_t bytes);

// Default barrier wait limit: about one second at the GB300's maximum SM clock.
constexpr long long kDefaultWaitLimit = TQ_DEFAULT_WAIT_LIMIT;
// Limit of the waits that drain copies or tensor-core work still in flight after
// a CTA gave up: fixed, so that a tiny tq_set_wait_limit never frees memory early.
constexpr long long kDrainLimit = 4000000000LL;

}  // namespace tq
