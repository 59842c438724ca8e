// tq_tables.cpp -- host-side codec tables of the library.
//
// Lloyd-Max codebooks: the pages take the value centroids from "iterative
// Lloyd-Max on a unit normal" (mlx-bun "TurboQuant -- rotation-based
// quantization", Part A, "Algorithm", values bullet) and print the 3-bit
// table.  The library solves the optimality conditions of the N(0,1)
// quantizer directly: with cell edges e_1 < ... < e_{n-1} (e_0 = -inf,
// e_n = +inf) and m_k = E[X | e_k < X < e_{k+1}],
//     e_i = (m_{i-1} + m_i) / 2,   i = 1 .. n-1,
// by Newton's method on the edges (the Jacobian is tridiagonal), started
// from a few Lloyd sweeps.  The fixed point is unique for a log-concave
// density, so any convergent solver lands on the same table.  Centroids are
// stored rounded to fp32; boundaries are the binary64 midpoints of the binary64
// centroids, rounded to fp32.
#include <cmath>
#include <mutex>
#include <vector>

#include "tq_kernels.h"

namespace tq {
namespace {

double pdf(double x) { return std::isinf(x) ? 0.0 : std::exp(-0.5 * x * x) * 0.3989422804014327; }
double upper_tail(double x) { return 0.5 * std::erfc(x * 0.7071067811865476); }
double lower_tail(double x) { return 0.5 * std::erfc(-x * 0.7071067811865476); }

double mass(double a, double b)  // P(a < X < b), evaluated where it does not cancel
{
    if (a >= 0.0) return upper_tail(a) - upper_tail(b);
    if (b <= 0.0) return lower_tail(b) - lower_tail(a);
    return 1.0 - lower_tail(a) - upper_tail(b);
}

double cell_mean(double a, double b) { return (pdf(a) - pdf(b)) / mass(a, b); }

// inverse of the standard normal CDF by bisection (start values only)
double normal_quantile(double p)
{
    double lo = -40.0, hi = 40.0;
    for (int i = 0; i < 200; ++i) {
        double mid = 0.5 * (lo + hi);
        if (lower_tail(mid) < p) lo = mid;
        else hi = mid;
    }
    return 0.5 * (lo + hi);
}

void solve(int bits, std::vector<double> &centroids)
{
    const int n = 1 << bits;
    std::vector<double> e(n + 1), m(n);
    e[0] = -INFINITY;
    e[n] = INFINITY;
    // high-resolution start: point density ~ pdf^(1/3), i.e. quantiles of N(0, 3)
    for (int i = 1; i < n; ++i) e[i] = std::sqrt(3.0) * normal_quantile((double)i / n);
    auto means = [&] {
        for (int k = 0; k < n; ++k) m[k] = cell_mean(e[k], e[k + 1]);
    };
    for (int it = 0; it < 30; ++it) {  // Lloyd sweeps
        means();
        for (int i = 1; i < n; ++i) e[i] = 0.5 * (m[i - 1] + m[i]);
    }
    std::vector<double> sub(n), dia(n), sup(n), rhs(n), dlo(n), dhi(n);
    for (int it = 0; it < 100 && n > 2; ++it) {
        means();
        for (int k = 0; k < n; ++k) {
            const double P = mass(e[k], e[k + 1]);
            dlo[k] = std::isinf(e[k]) ? 0.0 : pdf(e[k]) * (m[k] - e[k]) / P;          // dm_k/de_k
            dhi[k] = std::isinf(e[k + 1]) ? 0.0 : pdf(e[k + 1]) * (e[k + 1] - m[k]) / P;  // dm_k/de_{k+1}
        }
        // unknowns e_1..e_{n-1} -> rows 0..n-2
        const int u = n - 1;
        for (int r = 0; r < u; ++r) {
            const int i = r + 1;
            sub[r] = -0.5 * dlo[i - 1];
            dia[r] = 1.0 - 0.5 * (dhi[i - 1] + dlo[i]);
            sup[r] = -0.5 * dhi[i];
            rhs[r] = -(e[i] - 0.5 * (m[i - 1] + m[i]));
        }
        for (int r = 1; r < u; ++r) {
            const double w = sub[r] / dia[r - 1];
            dia[r] -= w * sup[r - 1];
            rhs[r] -= w * rhs[r - 1];
        }
        double step = 0.0, nxt = 0.0;
        for (int r = u - 1; r >= 0; --r) {
            const double x = (rhs[r] - (r + 1 < u ? sup[r] * nxt : 0.0)) / dia[r];
            e[r + 1] += x;
            step = std::fmax(step, std::fabs(x));
            nxt = x;
        }
        if (step < 1e-15) break;
    }
    for (int it = 0; it < 3; ++it) {  // settle on the Lloyd map's fixed point
        means();
        for (int i = 1; i < n; ++i) e[i] = 0.5 * (m[i - 1] + m[i]);
    }
    means();
    // the unit normal is symmetric, and so is its optimal quantizer: make the
    // table exactly antisymmetric (the middle boundary is then exactly 0)
    for (int i = n / 2; i < n; ++i) {
        const double a = 0.5 * (m[i] - m[n - 1 - i]);
        m[i] = a;
        m[n - 1 - i] = -a;
    }
    centroids = m;
}

std::once_flag g_once[9];
Tables g_tables[9];

}  // namespace

const Tables &codebook_tables(int vb)
{
    std::call_once(g_once[vb], [vb] {
        std::vector<double> c;
        solve(vb, c);
        const int n = 1 << vb;
        Tables &t = g_tables[vb];
        for (int i = 0; i < n; ++i) t.centroids[i] = (float)c[i];
        for (int i = 0; i + 1 < n; ++i) t.boundaries[i] = (float)(0.5 * (c[i] + c[i + 1]));
    });
    return g_tables[vb];
}

float inv_sqrt_head_dim(int d) { return (float)(1.0 / std::sqrt((double)d)); }

}  // namespace tq
