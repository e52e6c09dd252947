// Codebooks and requantisation candidate tables of the q4adamw library.
//
// The pages name the codebooks ("Rounding in Preconditioner Space" listing
// page, Abstract and Table 2: NF4 for m, zero-inclusive Dyn4 for ZIP-SR v,
// zero-excluding Dyn4-NZ for ZE-EDEN v; AReno docs "State representation":
// the 1-D second-moment map excludes zero) but print no level values.  The
// levels here follow the published constructions:
//   NF4     -- 4-bit NormalFloat (Dettmers et al., QLoRA): normal quantiles
//              at evenly spaced probabilities from delta = 1 - (1/30+1/32)/2
//              towards 1/2, 8 positive and 7 negative, plus an exact zero,
//              divided by the largest.  The inverse normal CDF is computed by
//              bisection on erfc in double precision.
//   Dyn4    -- unsigned 4-bit dynamic-exponent map: e leading zeros
//              (e = 0..3), an indicator bit, f = 3 - e fraction bits;
//              value (2^f + 9(j+1)) / (10^(e+1) 2^f); the all-zero code is 0.
//   Dyn4-NZ -- as Dyn4 with the all-zero code at 10^-4 (no zero level).
//   SDyn4   -- signed 4-bit dynamic-exponent map (the TorchAO baseline's first
//              moment): on rung i = 0, 1, 2, the midpoints of 2^i equal parts
//              of [1/10, 1] scaled by 10^(i-2), with both signs, plus 0 and 1.
//   Lin4-NZ -- linear zero-excluding map k/16, k = 1..16 (TorchAO's second
//              moment).
// RTN thresholds are FP32 roundings of double midpoints of adjacent levels.
//
// Candidate tables.  The kernel finds a code by a table lookup on a cheap
// bucket of the block-normalised value followed by one exact comparison
// against the block's scaled threshold (or level).  A bucket's entry is a
// lower bound c such that the exact answer is c or c+1; build_tables checks
// for every bucket that at most one threshold (level) is undecided within the
// bucket after widening it by 2^-20 relative, which exceeds the combined
// rounding of 1/s, x*(1/s) and t*s (3 * 2^-24).
#include <algorithm>
#include <cmath>
#include <cstring>
#include <mutex>

#include "q4_internal.h"

namespace q4 {
namespace {

double normal_cdf(double x) { return 0.5 * std::erfc(-x / std::sqrt(2.0)); }

// Inverse normal CDF for p in (0.5, 1) by bisection to the last double bit.
double normal_quantile(double p) {
    double lo = 0.0, hi = 40.0;
    for (int i = 0; i < 2000; ++i) {
        double mid = 0.5 * (lo + hi);
        if (mid <= lo || mid >= hi) break;
        if (normal_cdf(mid) < p) lo = mid; else hi = mid;
    }
    // pick the endpoint whose CDF is closer to p
    return (std::fabs(normal_cdf(lo) - p) <= std::fabs(normal_cdf(hi) - p)) ? lo : hi;
}

void fill_thresholds(Codebook& c) {
    for (int k = 0; k < 15; ++k)
        c.thresholds[k] = (float)(((double)c.levels[k] + (double)c.levels[k + 1]) / 2.0);
}

Codebook make_nf4() {
    const double delta = 1.0 - 0.5 * (1.0 / 30.0 + 1.0 / 32.0);
    double v[16];
    int n = 0;
    for (int i = 0; i < 8; ++i) v[n++] = normal_quantile(delta + i * ((0.5 - delta) / 8.0));
    for (int i = 0; i < 7; ++i) v[n++] = -normal_quantile(delta + i * ((0.5 - delta) / 7.0));
    v[n++] = 0.0;
    std::sort(v, v + 16);
    const double top = v[15];
    Codebook c{};
    for (int k = 0; k < 16; ++k) c.levels[k] = (float)(v[k] / top);
    fill_thresholds(c);
    return c;
}

Codebook make_dyn4(bool zero_excluding) {
    double v[16];
    int n = 0;
    double pow10 = 10.0;
    for (int e = 0; e < 4; ++e, pow10 *= 10.0) {
        const int f = 3 - e;
        const double two_f = (double)(1 << f);
        for (int j = 0; j < (1 << f); ++j) v[n++] = (two_f + 9.0 * (j + 1)) / (pow10 * two_f);
    }
    v[n++] = zero_excluding ? 1.0 / 10000.0 : 0.0;
    std::sort(v, v + 16);
    Codebook c{};
    for (int k = 0; k < 16; ++k) c.levels[k] = (float)v[k];
    fill_thresholds(c);
    return c;
}

// Decide, for x/s in [lo, hi], which of the ascending points p[0..np) satisfy
// "point < x" for certain.  Returns false if more than one is undecided.
// strict_le: the comparison in the kernel is point <= x (levels) instead of
// x > point (thresholds); the widening makes both cases identical here.
bool classify(const float* p, int np, double lo, double hi, int* n_below, int* n_undecided) {
    const double w = std::ldexp(1.0, -20);
    int below = 0, und = 0;
    for (int k = 0; k < np; ++k) {
        const double pk = p[k];
        const double slack = std::fabs(pk) * w;
        if (pk + slack < lo) below++;
        else if (pk - slack > hi) {}
        else und++;
    }
    *n_below = below;
    *n_undecided = und;
    return und <= 1;
}

// Linear bucket b of z = 16 x/s rounded to the nearest integer, stored at
// index (b + 16) & 63; x/s lies in [(b - 0.5)/16, (b + 0.5)/16].
bool build_linear(const float* pts, int np, bool levels, uint8_t lut[64]) {
    for (int idx = 0; idx < 64; ++idx) lut[idx] = 0;
    for (int b = -16; b <= 16; ++b) {
        double lo = (b - 0.5) / 16.0, hi = (b + 0.5) / 16.0;
        const double w = std::ldexp(1.0, -20);
        lo -= std::fabs(lo) * w + 1e-30;
        hi += std::fabs(hi) * w + 1e-30;
        int below, und;
        if (!classify(pts, np, lo, hi, &below, &und)) return false;
        int c = levels ? std::max(below - 1, 0) : below;
        c = std::min(c, 14);
        lut[(b + 16) & 63] = (uint8_t)c;
    }
    // unreachable indices (non-finite inputs only): any in-range candidate
    for (int idx = 33; idx < 64; ++idx) lut[idx] = 14;
    return true;
}

float bits_to_float(uint32_t u) {
    float f;
    std::memcpy(&f, &u, 4);
    return f;
}

// Log bucket i = bits(x/s) >> 19 (1/16 octave) of a non-negative x/s; the
// table covers every such bit pattern (buckets above 2 hold only inputs that
// cannot occur for finite x <= s, and NaN).
bool build_log(const float* pts, int np, bool levels, uint8_t* lut) {
    for (int i = 0; i < kVLut; ++i) {
        double lo = bits_to_float((uint32_t)i << 19);
        double hi = (i + 1 < 4096) ? bits_to_float((uint32_t)(i + 1) << 19) : INFINITY;
        if (i == kVLut - 1) hi = INFINITY;   // clamped: everything above
        if (!std::isfinite(lo)) lo = 1e300;
        const double w = std::ldexp(1.0, -20);
        lo = lo * (1 - w);
        hi = std::isfinite(hi) ? hi * (1 + w) : 1e300;
        int below, und;
        if (!classify(pts, np, lo, hi, &below, &und)) {
            // Buckets far above 1 (x/s > 1 cannot occur for finite inputs)
            // and the catch-all top bucket hold every point: take the top.
            if (lo > 2.0) { lut[i] = 14; continue; }
            return false;
        }
        int c = levels ? std::max(below - 1, 0) : below;
        lut[i] = (uint8_t)std::min(c, 14);
    }
    return true;
}

// SDyn4 RTN by magnitude.  Its RTN thresholds are symmetric about zero,
// T_k = -T_{13-k} for k = 0..6, with one more positive threshold T_14, so with
// the magnitudes A_i = T_{7+i} (i = 0..7, ascending) the code of x is
// 7 + #{i : x > A_i s} for x >= 0 and 7 - min(#{i : |x| >= A_i s}, 7) for
// x < 0.  The table holds, per log bucket of |x|/s, a lower bound c of the
// count with the exact count in {c, c+1} (for either comparison).
bool build_m_log(const Codebook& c, uint8_t* lut) {
    for (int k = 0; k < 7; ++k)
        if (!(c.thresholds[k] == -c.thresholds[13 - k])) return false;
    float mags[8];
    for (int i = 0; i < 8; ++i) mags[i] = c.thresholds[7 + i];
    if (!(mags[0] > 0.f)) return false;
    for (int i = 0; i < kVLut; ++i) {
        double lo = bits_to_float((uint32_t)i << 19);
        double hi = (i + 1 < kVLut) ? bits_to_float((uint32_t)(i + 1) << 19) : INFINITY;
        if (!std::isfinite(lo)) lo = 1e300;
        const double w = std::ldexp(1.0, -20);
        lo = lo * (1 - w);
        hi = std::isfinite(hi) ? hi * (1 + w) : 1e300;
        int below, und;
        if (!classify(mags, 8, lo, hi, &below, &und)) {
            if (lo > 2.0) { lut[i] = 8; continue; }   // |x|/s > 1 cannot occur
            return false;
        }
        lut[i] = (uint8_t)below;
    }
    return true;
}

Codebook make_sdyn4() {
    double v[16];
    int n = 0;
    double rung = 0.01;
    for (int i = 0; i < 3; ++i, rung *= 10.0) {
        const int parts = 1 << i;
        for (int j = 0; j < parts; ++j) {
            const double mid = 0.1 + 0.9 * (2.0 * j + 1.0) / (2.0 * parts);
            v[n++] = rung * mid;
            v[n++] = -rung * mid;
        }
    }
    v[n++] = 0.0;
    v[n++] = 1.0;
    std::sort(v, v + 16);
    Codebook c{};
    for (int k = 0; k < 16; ++k) c.levels[k] = (float)v[k];
    fill_thresholds(c);
    return c;
}

Codebook make_lin4nz() {
    Codebook c{};
    for (int k = 0; k < 16; ++k) c.levels[k] = (float)(k + 1) / 16.0f;
    fill_thresholds(c);
    return c;
}

Codebook g_books[5];
std::once_flag g_once;

void init_books() {
    g_books[0] = make_nf4();
    g_books[1] = make_dyn4(false);
    g_books[2] = make_dyn4(true);
    g_books[3] = make_sdyn4();
    g_books[4] = make_lin4nz();
}

}  // namespace

const Codebook& codebook(int which) {
    std::call_once(g_once, init_books);
    return g_books[which];
}

bool build_tables(int mbook, int vbook, Tables* t) {
    const Codebook& nf4 = codebook(mbook);
    const Codebook& v = codebook(vbook);
    std::memset(t, 0, sizeof(*t));
    for (int k = 0; k < 16; ++k) {
        t->nf4[k] = nf4.levels[k];
        t->vl[k] = v.levels[k];
    }
    for (int k = 0; k < 15; ++k) {
        t->nf4_t[k] = nf4.thresholds[k];
        t->vt[k] = v.thresholds[k];
    }
    t->nf4_t[15] = INFINITY;
    t->vt[15] = INFINITY;
    // Linear buckets suit NF4; a codebook with several thresholds in one
    // bucket (SDyn4 near zero) is searched by the kernel without them.
    t->m_lut = build_linear(nf4.thresholds, 15, false, t->lut_nf4_t) &&
               build_linear(nf4.levels, 16, true, t->lut_nf4_l) ? 1 : 0;
    // the signed dynamic-exponent map (TorchAO's m) is searched by magnitude
    if (mbook == 3 && !build_m_log(nf4, t->lut_m_log)) return false;
    if (!build_log(v.levels, 16, true, t->lut_v_l)) return false;
    if (!build_log(v.thresholds, 15, false, t->lut_v_t)) return false;
    for (int i = 0; i < 64; ++i) {
        const int c = t->lut_nf4_t[i];
        t->nf4_bucket[i].x = nf4.thresholds[c];
        std::memcpy(&t->nf4_bucket[i].y, &c, 4);   // the candidate code, as raw bits
    }
    return true;
}

}  // namespace q4
