// tq_params.cpp -- host-side construction of the codec tables (double precision).
//
// Rotation Pi: the orthogonal factor of a Gaussian matrix (0xsero/turboquant,
// "Compression Pipeline": random orthogonal rotation state; brightcoding blog,
// "What is TurboQuant-GPU?": a random rotation makes coordinates ~Gaussian).
// It is computed here by classical Gram-Schmidt with one re-orthogonalisation
// pass (CGS2) over the columns of G; every r_jj is positive by construction,
// so Pi is the unique Q of G = QR with a positive-diagonal R, i.e. a Haar
// rotation (Mezzadri, "How to generate random matrices from the classical
// compact groups", 2007).
//
// QJL matrix S: a matrix of independent standard Gaussians (0xsero/turboquant,
// "Compression Pipeline": QJL residual-sign projection).
//
// Gaussians: SplitMix64 (Steele, Lea & Flood, "Fast splittable pseudorandom
// number generators", OOPSLA 2014); stream s starts from
// seed ^ (0x9E3779B97F4A7C15 * (s + 1)); uniforms are the top 53 bits placed at
// the centre of their bucket; Box-Muller turns each pair (u1, u2) into
// r cos(2 pi u2), r sin(2 pi u2) with r = sqrt(-2 ln u1).  Matrices fill
// row-major.
//
// Randomized Hadamard rotation (turbo-attn, "How it works", step 1: a fast
// Walsh-Hadamard transform): Pi = H D / sqrt(d), H the Sylvester Hadamard
// matrix H[i][j] = (-1)^popcount(i & j) and D = diag(s_j) with random signs
// s_j = -1 when the top bit of the j-th output of SplitMix64 stream 0 is set.
// Pi is orthogonal and y = Pi k costs an O(d log d) butterfly.
//
// Codebook: the Lloyd-Max quantiser of N(0,1) (brightcoding blog: Lloyd-Max is
// optimal for Gaussian sources; 0xsero/turboquant "Compression Pipeline":
// Lloyd-Max scalar codebooks) found by the Lloyd fixed-point iteration.
#include <cmath>
#include <cstdint>
#include <vector>

#include "tq_internal.h"

namespace tq {
namespace {

constexpr double kPi = 3.14159265358979323846;

struct SplitMix64 {
    uint64_t s;
    uint64_t next()
    {
        s += 0x9E3779B97F4A7C15ULL;
        uint64_t z = s;
        z = (z ^ (z >> 30)) * 0xBF58476D1CE4E5B9ULL;
        z = (z ^ (z >> 27)) * 0x94D049BB133111EBULL;
        return z ^ (z >> 31);
    }
    double uniform() { return (static_cast<double>(next() >> 11) + 0.5) * 0x1.0p-53; }
};

std::vector<double> gaussian_matrix(int d, uint64_t seed, int stream)
{
    SplitMix64 rng{seed ^ (0x9E3779B97F4A7C15ULL * static_cast<uint64_t>(stream + 1))};
    std::vector<double> m(static_cast<size_t>(d) * d);
    for (size_t i = 0; i < m.size(); i += 2) {
        const double u1 = rng.uniform();
        const double u2 = rng.uniform();
        const double r = std::sqrt(-2.0 * std::log(u1));
        m[i] = r * std::cos(2.0 * kPi * u2);
        if (i + 1 < m.size()) m[i + 1] = r * std::sin(2.0 * kPi * u2);
    }
    return m;
}

// Columns of G orthonormalised left to right; returns Q row-major.
std::vector<double> haar_rotation(int d, uint64_t seed)
{
    std::vector<double> G = gaussian_matrix(d, seed, 0);
    std::vector<double> Qc(static_cast<size_t>(d) * d);  // column-major: column j at Qc[j*d]
    std::vector<double> v(d);
    for (int j = 0; j < d; ++j) {
        for (int i = 0; i < d; ++i) v[i] = G[static_cast<size_t>(i) * d + j];
        for (int pass = 0; pass < 2; ++pass) {
            for (int c = 0; c < j; ++c) {
                const double *q = &Qc[static_cast<size_t>(c) * d];
                double dot = 0.0;
                for (int i = 0; i < d; ++i) dot += q[i] * v[i];
                for (int i = 0; i < d; ++i) v[i] -= dot * q[i];
            }
        }
        double nrm = 0.0;
        for (int i = 0; i < d; ++i) nrm += v[i] * v[i];
        nrm = std::sqrt(nrm);
        for (int i = 0; i < d; ++i) Qc[static_cast<size_t>(j) * d + i] = v[i] / nrm;
    }
    std::vector<double> Q(static_cast<size_t>(d) * d);
    for (int i = 0; i < d; ++i)
        for (int j = 0; j < d; ++j) Q[static_cast<size_t>(i) * d + j] = Qc[static_cast<size_t>(j) * d + i];
    return Q;
}

std::vector<double> hadamard_signs(int d, uint64_t seed)
{
    SplitMix64 rng{seed ^ 0x9E3779B97F4A7C15ULL};  // stream 0
    std::vector<double> sg(d);
    for (int j = 0; j < d; ++j) sg[j] = (rng.next() >> 63) ? -1.0 : 1.0;
    return sg;
}

std::vector<double> hadamard_rotation(int d, uint64_t seed)
{
    const std::vector<double> sg = hadamard_signs(d, seed);
    const double inv = 1.0 / std::sqrt(static_cast<double>(d));
    std::vector<double> Q(static_cast<size_t>(d) * d);
    for (int i = 0; i < d; ++i)
        for (int j = 0; j < d; ++j)
            Q[static_cast<size_t>(i) * d + j] = ((__builtin_popcount(static_cast<unsigned>(i & j)) & 1) ? -inv : inv) * sg[j];
    return Q;
}

double std_normal_pdf(double x) { return std::isinf(x) ? 0.0 : std::exp(-0.5 * x * x) * 0.3989422804014327; }

// Upper-tail probability Q(x) = P(X > x).
double upper_tail(double x) { return 0.5 * std::erfc(x * 0.7071067811865476); }

// P(a < X <= b), using whichever tail keeps the difference well conditioned.
double interval_prob(double a, double b)
{
    if (a >= 0.0) return upper_tail(a) - upper_tail(b);
    if (b <= 0.0) return upper_tail(-b) - upper_tail(-a);
    return 1.0 - upper_tail(b) - upper_tail(-a);
}

}  // namespace

bool build_codebook(int bits, double *centroids, double *thresholds)
{
    const int L = 1 << bits;
    std::vector<double> c(L), t(L + 1);
    for (int i = 0; i < L; ++i) c[i] = -3.0 + 6.0 * i / (L - 1);
    for (int iter = 0; iter < 200000; ++iter) {
        t[0] = -INFINITY;
        t[L] = INFINITY;
        for (int i = 1; i < L; ++i) t[i] = 0.5 * (c[i - 1] + c[i]);
        double change = 0.0;
        for (int i = 0; i < L; ++i) {
            const double next = (std_normal_pdf(t[i]) - std_normal_pdf(t[i + 1])) / interval_prob(t[i], t[i + 1]);
            change = std::fmax(change, std::fabs(next - c[i]));
            c[i] = next;
        }
        if (change < 1e-15) {
            for (int i = 0; i < L; ++i) centroids[i] = c[i];
            for (int i = 1; i < L; ++i) thresholds[i - 1] = 0.5 * (c[i - 1] + c[i]);
            return true;
        }
    }
    return false;
}

bool build_tables(int d, int k_bits, uint64_t seed, int rotation, HostTables *out)
{
    if (rotation == 1) {  // randomized Hadamard
        out->Pi = hadamard_rotation(d, seed);
        out->hsign = hadamard_signs(d, seed);
    } else {
        out->Pi = haar_rotation(d, seed);
        out->hsign.assign(d, 1.0);
    }
    out->S = gaussian_matrix(d, seed, 1);
    out->centroids.assign(1 << k_bits, 0.0);
    out->thresholds.assign((1 << k_bits) - 1, 0.0);
    return build_codebook(k_bits, out->centroids.data(), out->thresholds.data());
}

}  // namespace tq
