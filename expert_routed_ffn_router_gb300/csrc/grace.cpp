// grace.cpp -- GRACE-MoE placement planner on the layer's by-products (per-expert counts
// and the co-activation matrix): host code, run once per profiling window, not per step.
//
// Method: the "GRACE-MoE" notes, section "Core Idea":
//   1. Expert Grouping: experts that are often activated together go to the same GPU.  The
//      affinity matrix A (co-activation counts) is clustered spectrally into D groups whose
//      sizes may deviate from the mean n/D by delta = (n/D) * r; U(r) (share of the
//      affinity kept inside groups) and S(r) (RMS deviation of the group sizes) are traced
//      over r and r is taken at the knee.
//   2. Expert Replication: rho = W_max / W_mean over the groups' loads; n_replica =
//      min(max(1, floor(rho)), n_gpu - 1); in the heaviest group the experts are taken by
//      load until their cumulative load exceeds W_max * n_replica / (1 + n_replica), and
//      copies of these hot experts go to the n_replica least-loaded GPUs.
//   3. Routing Policy: predicted loads W'_max = W_max - W_r + W_p, W'_i = W_i + W_p (W_r the
//      hot experts' load, W_p its share per instance); instance weights inversely
//      proportional to the predicted load, applied inside the nearest tier that holds an
//      instance (same GPU, then same node, then every node).
//
// Readings where the notes leave a step open: the normalised spectral embedding (the D
// leading eigenvectors of Deg^-1/2 A Deg^-1/2, rows scaled to unit length; an expert with
// no co-activation gets degree 1 and keeps a zero row); integer size bounds
// ceil(n/D - delta) .. floor(n/D + delta); a size-bounded k-means from farthest-point seeds
// (first: the expert of largest degree) whose assignment takes (expert, group) pairs by
// increasing distance under the upper bound, puts each expert with no co-activation into
// the smallest group, and then fills groups below the lower bound with the cheapest moves;
// the knee of U(r) where U and r scaled to [0, 1] differ most; ties to the lower index.
//
// Eigenvectors: Householder tridiagonalisation and implicit symmetric QR (Wilkinson
// shift) in fp64; the embedding depends only on the leading eigenspace, so the basis the
// solver ends on within it does not matter.
#include <algorithm>
#include <cmath>
#include <cstdint>
#include <cstring>
#include <numeric>
#include <tuple>
#include <vector>

#include "../../include/moe.h"

namespace {

using Mat = std::vector<double>;   // row-major n x n

// Eigen-decomposition of the symmetric n x n matrix a (destroyed): eigenvalues in w,
// eigenvectors in the columns of q.  Householder reduction to tridiagonal form
// (Q^T A Q = T), then implicit symmetric QR steps with the Wilkinson shift on T, the
// Givens rotations accumulated into Q.
void sym_eigen(int n, Mat &a, std::vector<double> &w, Mat &q)
{
    auto A = [&](int i, int j) -> double & { return a[static_cast<size_t>(i) * n + j]; };
    auto Q = [&](int i, int j) -> double & { return q[static_cast<size_t>(i) * n + j]; };
    q.assign(static_cast<size_t>(n) * n, 0.0);
    for (int i = 0; i < n; ++i) Q(i, i) = 1.0;
    std::vector<double> v(n), p(n), wv(n);
    for (int k = 0; k + 2 < n; ++k) {
        // Householder vector of the column below the diagonal: H x = alpha e1
        double xn = 0.0;
        for (int i = k + 1; i < n; ++i) xn += A(i, k) * A(i, k);
        xn = std::sqrt(xn);
        if (xn == 0.0) continue;
        const double alpha = A(k + 1, k) > 0 ? -xn : xn;
        double vv = 0.0;
        for (int i = k + 1; i < n; ++i) {
            v[i] = A(i, k) - (i == k + 1 ? alpha : 0.0);
            vv += v[i] * v[i];
        }
        if (vv == 0.0) continue;
        const double beta = 2.0 / vv;
        // trailing block: A <- A - v w^T - w v^T, p = beta A v, w = p - (beta p.v / 2) v
        double pv = 0.0;
        for (int i = k + 1; i < n; ++i) {
            double t = 0.0;
            for (int j = k + 1; j < n; ++j) t += A(i, j) * v[j];
            p[i] = beta * t;
            pv += p[i] * v[i];
        }
        const double K = 0.5 * beta * pv;
        for (int i = k + 1; i < n; ++i) wv[i] = p[i] - K * v[i];
        for (int i = k + 1; i < n; ++i)
            for (int j = k + 1; j < n; ++j) A(i, j) -= v[i] * wv[j] + wv[i] * v[j];
        for (int i = k + 1; i < n; ++i) A(i, k) = A(k, i) = (i == k + 1 ? alpha : 0.0);
        // Q <- Q H
        for (int i = 0; i < n; ++i) {
            double t = 0.0;
            for (int j = k + 1; j < n; ++j) t += Q(i, j) * v[j];
            t *= beta;
            for (int j = k + 1; j < n; ++j) Q(i, j) -= t * v[j];
        }
    }
    std::vector<double> d(n), e(n > 1 ? n - 1 : 1, 0.0);
    for (int i = 0; i < n; ++i) d[i] = A(i, i);
    for (int i = 0; i + 1 < n; ++i) e[i] = A(i + 1, i);
    const double eps = 2.220446049250313e-16;
    int m = n - 1, iters = 0;
    while (m > 0 && iters < 64 * n) {
        if (std::fabs(e[m - 1]) <= eps * (std::fabs(d[m - 1]) + std::fabs(d[m]))) {
            e[m - 1] = 0.0;
            --m;
            continue;
        }
        int l = m - 1;
        while (l > 0 && std::fabs(e[l - 1]) > eps * (std::fabs(d[l - 1]) + std::fabs(d[l]))) --l;
        ++iters;
        // Wilkinson shift: the eigenvalue of the trailing 2 x 2 closer to d[m]
        const double dl = 0.5 * (d[m - 1] - d[m]);
        const double em = e[m - 1];
        const double mu = d[m] - em * em / (dl + (dl >= 0 ? 1.0 : -1.0) * std::sqrt(dl * dl + em * em));
        double x = d[l] - mu, z = e[l];
        for (int k = l; k < m; ++k) {
            const double r = std::hypot(x, z);
            const double c = r > 0 ? x / r : 1.0, s = r > 0 ? z / r : 0.0;
            if (k > l) e[k - 1] = r;
            const double a0 = d[k], b0 = e[k], d1 = d[k + 1];
            d[k] = c * c * a0 + 2.0 * c * s * b0 + s * s * d1;
            d[k + 1] = s * s * a0 - 2.0 * c * s * b0 + c * c * d1;
            e[k] = c * s * (d1 - a0) + (c * c - s * s) * b0;
            if (k + 1 < m) {
                const double f = e[k + 1];
                z = s * f;          // bulge at (k, k + 2)
                e[k + 1] = c * f;
                x = e[k];
            }
            for (int i = 0; i < n; ++i) {
                const double qk = Q(i, k), qk1 = Q(i, k + 1);
                Q(i, k) = c * qk + s * qk1;
                Q(i, k + 1) = -s * qk + c * qk1;
            }
        }
    }
    w = d;
}

// Rows of the D leading eigenvectors of Deg^-1/2 A Deg^-1/2, scaled to unit length: [n][D].
std::vector<double> embedding(const int32_t *aff, int n, int D)
{
    std::vector<double> deg(n, 0.0);
    for (int i = 0; i < n; ++i)
        for (int j = 0; j < n; ++j) deg[i] += aff[static_cast<size_t>(i) * n + j];
    std::vector<double> s(n);
    for (int i = 0; i < n; ++i) s[i] = 1.0 / std::sqrt(deg[i] > 0 ? deg[i] : 1.0);
    Mat M(static_cast<size_t>(n) * n);
    for (int i = 0; i < n; ++i)
        for (int j = 0; j < n; ++j)
            M[static_cast<size_t>(i) * n + j] = aff[static_cast<size_t>(i) * n + j] * s[i] * s[j];
    std::vector<double> w;
    Mat V;
    sym_eigen(n, M, w, V);
    std::vector<int> order(n);
    std::iota(order.begin(), order.end(), 0);
    std::stable_sort(order.begin(), order.end(), [&](int a, int b) { return w[a] > w[b]; });
    std::vector<double> Y(static_cast<size_t>(n) * D);
    for (int i = 0; i < n; ++i) {
        double nrm = 0.0;
        for (int k = 0; k < D; ++k) {
            const double x = V[static_cast<size_t>(i) * n + order[k]];
            Y[static_cast<size_t>(i) * D + k] = x;
            nrm += x * x;
        }
        nrm = std::sqrt(nrm);
        // an expert with no co-activation has a zero row (up to rounding): it stays at zero
        for (int k = 0; k < D; ++k)
            Y[static_cast<size_t>(i) * D + k] = nrm < 1e-9 ? 0.0 : Y[static_cast<size_t>(i) * D + k] / nrm;
    }
    return Y;
}

void size_bounds(int n, int D, double r, int &lo, int &hi)
{
    const double ebar = static_cast<double>(n) / D, delta = ebar * r;
    lo = std::max(0, static_cast<int>(std::ceil(ebar - delta - 1e-12)));
    hi = static_cast<int>(std::floor(ebar + delta + 1e-12));
}

double dist2(const double *a, const double *b, int D)
{
    double s = 0.0;
    for (int k = 0; k < D; ++k) {
        const double d = a[k] - b[k];
        s += d * d;
    }
    return s;
}

// Size-bounded assignment of the rows Y to the centroids C.
std::vector<int> assign(const std::vector<double> &Y, const std::vector<double> &C, int n, int D,
                        int lo, int hi, const std::vector<char> &iso)
{
    std::vector<double> d2(static_cast<size_t>(n) * D);
    std::vector<std::tuple<double, int, int>> order;
    order.reserve(static_cast<size_t>(n) * D);
    for (int i = 0; i < n; ++i)
        for (int k = 0; k < D; ++k) {
            const double d = dist2(&Y[static_cast<size_t>(i) * D], &C[static_cast<size_t>(k) * D], D);
            d2[static_cast<size_t>(i) * D + k] = d;
            if (!iso[i]) order.emplace_back(d, i, k);
        }
    std::sort(order.begin(), order.end());
    std::vector<int> g(n, -1), size(D, 0);
    for (const auto &o : order) {
        const int i = std::get<1>(o), k = std::get<2>(o);
        if (g[i] < 0 && size[k] < hi) {
            g[i] = k;
            ++size[k];
        }
    }
    // experts with no co-activation carry no affinity: each to the smallest group
    for (int i = 0; i < n; ++i) {
        if (!iso[i]) continue;
        int k = -1;
        for (int q = 0; q < D; ++q)
            if (size[q] < hi && (k < 0 || size[q] < size[k])) k = q;
        g[i] = k;
        ++size[k];
    }
    while (true) {
        int k = -1;
        for (int q = 0; q < D; ++q)
            if (size[q] < lo) { k = q; break; }
        if (k < 0) break;
        int best = -1;
        double best_cost = 0.0;
        for (int i = 0; i < n; ++i) {
            const int src = g[i];
            if (size[src] <= lo) continue;
            const double cost = d2[static_cast<size_t>(i) * D + k] - d2[static_cast<size_t>(i) * D + src];
            if (best < 0 || cost < best_cost) { best = i; best_cost = cost; }
        }
        if (best < 0) break;          // unreachable when lo * D <= n
        --size[g[best]];
        g[best] = k;
        ++size[k];
    }
    return g;
}

std::vector<int> group_rows(const std::vector<double> &Y, const int32_t *aff, int n, int D,
                            double r)
{
    int lo, hi;
    size_bounds(n, D, r, lo, hi);
    // farthest-point seeds, the first the expert of largest degree
    std::vector<long long> deg(n, 0);
    for (int i = 0; i < n; ++i)
        for (int j = 0; j < n; ++j) deg[i] += aff[static_cast<size_t>(i) * n + j];
    int first = 0;
    for (int i = 1; i < n; ++i)
        if (deg[i] > deg[first]) first = i;
    std::vector<int> seeds{first};
    std::vector<double> dmin(n);
    for (int i = 0; i < n; ++i)
        dmin[i] = dist2(&Y[static_cast<size_t>(i) * D], &Y[static_cast<size_t>(first) * D], D);
    while (static_cast<int>(seeds.size()) < D) {
        int s = -1;
        for (int i = 0; i < n; ++i) {
            if (std::find(seeds.begin(), seeds.end(), i) != seeds.end()) continue;
            if (s < 0 || dmin[i] > dmin[s]) s = i;
        }
        seeds.push_back(s);
        for (int i = 0; i < n; ++i)
            dmin[i] = std::min(dmin[i], dist2(&Y[static_cast<size_t>(i) * D], &Y[static_cast<size_t>(s) * D], D));
    }
    std::vector<double> C(static_cast<size_t>(D) * D);
    for (int k = 0; k < D; ++k)
        std::memcpy(&C[static_cast<size_t>(k) * D], &Y[static_cast<size_t>(seeds[k]) * D], sizeof(double) * D);
    std::vector<char> iso(n);
    for (int i = 0; i < n; ++i) iso[i] = deg[i] == 0;
    std::vector<int> g = assign(Y, C, n, D, lo, hi, iso);
    for (int it = 0; it < 50; ++it) {
        std::vector<double> sum(static_cast<size_t>(D) * D, 0.0);
        std::vector<int> cnt(D, 0);
        for (int i = 0; i < n; ++i) {
            ++cnt[g[i]];
            for (int k = 0; k < D; ++k) sum[static_cast<size_t>(g[i]) * D + k] += Y[static_cast<size_t>(i) * D + k];
        }
        for (int q = 0; q < D; ++q)
            if (cnt[q] > 0)
                for (int k = 0; k < D; ++k) C[static_cast<size_t>(q) * D + k] = sum[static_cast<size_t>(q) * D + k] / cnt[q];
        std::vector<int> g2 = assign(Y, C, n, D, lo, hi, iso);
        if (g2 == g) break;
        g = g2;
    }
    return g;
}

int check_affinity(const int32_t *aff, int E, int D)
{
    if (!aff || E <= 0 || D <= 0 || D > E) return MOE_ERR_INVALID_ARG;
    if (E > 4096) return MOE_ERR_UNSUPPORTED_SHAPE;
    return MOE_OK;
}

}  // namespace

extern "C" {

int moe_grace_metrics(const int32_t *affinity, int E, const int32_t *group_of, int D,
                      double *U, double *S)
{
    int rc = check_affinity(affinity, E, D);
    if (rc) return rc;
    if (!group_of || !U || !S) return MOE_ERR_INVALID_ARG;
    for (int i = 0; i < E; ++i)
        if (group_of[i] < 0 || group_of[i] >= D) return MOE_ERR_INVALID_ARG;
    long long total = 0, intra = 0;
    for (int i = 0; i < E; ++i)
        for (int j = i + 1; j < E; ++j) {
            const long long a = affinity[static_cast<size_t>(i) * E + j];
            total += a;
            if (group_of[i] == group_of[j]) intra += a;
        }
    *U = total > 0 ? static_cast<double>(intra) / static_cast<double>(total) : 0.0;
    std::vector<int> size(D, 0);
    for (int i = 0; i < E; ++i) ++size[group_of[i]];
    const double ebar = static_cast<double>(E) / D;
    double ss = 0.0;
    for (int d = 0; d < D; ++d) ss += (size[d] - ebar) * (size[d] - ebar);
    *S = std::sqrt(ss / D);
    return MOE_OK;
}

int moe_grace_group(const int32_t *affinity, int E, int D, double r, int32_t *group_of)
{
    int rc = check_affinity(affinity, E, D);
    if (rc) return rc;
    if (!group_of || !(r >= 0.0)) return MOE_ERR_INVALID_ARG;
    int lo, hi;
    size_bounds(E, D, r, lo, hi);
    if (static_cast<long long>(lo) * D > E || static_cast<long long>(hi) * D < E) return MOE_ERR_INVALID_ARG;
    const std::vector<double> Y = embedding(affinity, E, D);
    const std::vector<int> g = group_rows(Y, affinity, E, D, r);
    for (int i = 0; i < E; ++i) group_of[i] = g[i];
    return MOE_OK;
}

int moe_grace_choose_r(const int32_t *affinity, int E, int D, const double *r_grid, int n_r,
                       double *U, double *S, int *knee, int32_t *group_of)
{
    int rc = check_affinity(affinity, E, D);
    if (rc) return rc;
    if (!r_grid || n_r <= 0 || !U || !S || !knee || !group_of) return MOE_ERR_INVALID_ARG;
    for (int k = 0; k < n_r; ++k) {
        if (!(r_grid[k] >= 0.0) || (k > 0 && !(r_grid[k] > r_grid[k - 1]))) return MOE_ERR_INVALID_ARG;
        int lo, hi;
        size_bounds(E, D, r_grid[k], lo, hi);
        if (static_cast<long long>(lo) * D > E || static_cast<long long>(hi) * D < E) return MOE_ERR_INVALID_ARG;
    }
    const std::vector<double> Y = embedding(affinity, E, D);   // the same for every r
    std::vector<std::vector<int>> groups(n_r);
    std::vector<int32_t> g32(E);
    for (int k = 0; k < n_r; ++k) {
        groups[k] = group_rows(Y, affinity, E, D, r_grid[k]);
        for (int i = 0; i < E; ++i) g32[i] = groups[k][i];
        moe_grace_metrics(affinity, E, g32.data(), D, &U[k], &S[k]);
    }
    // knee of U(r): largest U_scaled - r_scaled, first maximum
    auto scaled = [&](const double *v, int k) {
        double mn = v[0], mx = v[0];
        for (int q = 1; q < n_r; ++q) { mn = std::min(mn, v[q]); mx = std::max(mx, v[q]); }
        return mx > mn ? (v[k] - mn) / (mx - mn) : 0.0;
    };
    int best = 0;
    double best_d = 0.0;
    for (int k = 0; k < n_r; ++k) {
        const double d = scaled(U, k) - scaled(r_grid, k);
        if (k == 0 || d > best_d) { best = k; best_d = d; }
    }
    *knee = best;
    for (int i = 0; i < E; ++i) group_of[i] = groups[best][i];
    return MOE_OK;
}

int moe_grace_replicate(const int32_t *counts, int E, const int32_t *group_of, int D,
                        long long *W, int32_t *hot, int32_t *replica_gpus,
                        moe_grace_replication_t *out)
{
    if (!counts || !group_of || !W || !hot || !replica_gpus || !out || E <= 0 || D < 2 || D > E)
        return MOE_ERR_INVALID_ARG;
    for (int i = 0; i < E; ++i)
        if (group_of[i] < 0 || group_of[i] >= D || counts[i] < 0) return MOE_ERR_INVALID_ARG;
    for (int d = 0; d < D; ++d) W[d] = 0;
    for (int i = 0; i < E; ++i) W[group_of[i]] += counts[i];
    long long sum = 0;
    int heavy = 0;
    for (int d = 0; d < D; ++d) {
        sum += W[d];
        if (W[d] > W[heavy]) heavy = d;
    }
    const double W_mean = static_cast<double>(sum) / D;
    const long long W_max = W[heavy];
    const double rho = W_mean > 0 ? static_cast<double>(W_max) / W_mean : 0.0;
    const int n_rep = std::min(std::max(1, static_cast<int>(std::floor(rho))), D - 1);
    std::vector<int> members;
    for (int i = 0; i < E; ++i)
        if (group_of[i] == heavy) members.push_back(i);
    std::stable_sort(members.begin(), members.end(),
                     [&](int a, int b) { return counts[a] > counts[b]; });
    const double thr = static_cast<double>(W_max) * n_rep / (1 + n_rep);
    long long acc = 0;
    int n_hot = 0;
    for (int e : members) {                 // until the cumulative load exceeds thr
        if (static_cast<double>(acc) > thr) break;
        hot[n_hot++] = e;
        acc += counts[e];
    }
    std::vector<int> others;
    for (int d = 0; d < D; ++d)
        if (d != heavy) others.push_back(d);
    std::stable_sort(others.begin(), others.end(), [&](int a, int b) { return W[a] < W[b]; });
    for (int k = 0; k < n_rep; ++k) replica_gpus[k] = others[k];
    out->heaviest = heavy;
    out->n_replica = n_rep;
    out->n_hot = n_hot;
    out->rho = rho;
    out->W_mean = W_mean;
    out->W_max = W_max;
    out->W_r = acc;
    return MOE_OK;
}

int moe_grace_route_table(const long long *W, int D, const moe_grace_replication_t *rep,
                          const int32_t *replica_gpus, int gpus_per_node, double *predicted,
                          double *table)
{
    if (!W || !rep || !replica_gpus || !predicted || !table || D < 2 || gpus_per_node < 1)
        return MOE_ERR_INVALID_ARG;
    const int n_inst = 1 + rep->n_replica;
    if (rep->n_replica < 1 || rep->n_replica > D - 1 || rep->heaviest < 0 || rep->heaviest >= D)
        return MOE_ERR_INVALID_ARG;
    std::vector<int> inst(n_inst);
    inst[0] = rep->heaviest;
    for (int k = 1; k < n_inst; ++k) {
        inst[k] = replica_gpus[k - 1];
        if (inst[k] < 0 || inst[k] >= D) return MOE_ERR_INVALID_ARG;
    }
    const double W_p = static_cast<double>(rep->W_r) / n_inst;
    predicted[0] = static_cast<double>(rep->W_max - rep->W_r) + W_p;
    for (int k = 1; k < n_inst; ++k) predicted[k] = static_cast<double>(W[inst[k]]) + W_p;
    std::vector<double> inv(n_inst);
    for (int k = 0; k < n_inst; ++k) inv[k] = predicted[k] > 0 ? 1.0 / predicted[k] : 1.0;
    for (int src = 0; src < D; ++src) {
        std::vector<int> tier;
        for (int k = 0; k < n_inst; ++k)
            if (inst[k] == src) tier.push_back(k);
        if (tier.empty())
            for (int k = 0; k < n_inst; ++k)
                if (inst[k] / gpus_per_node == src / gpus_per_node) tier.push_back(k);
        if (tier.empty())
            for (int k = 0; k < n_inst; ++k) tier.push_back(k);
        double z = 0.0;
        for (int k : tier) z += inv[k];
        double *row = table + static_cast<size_t>(src) * n_inst;
        for (int k = 0; k < n_inst; ++k) row[k] = 0.0;
        for (int k : tier) row[k] = inv[k] / z;
    }
    return MOE_OK;
}

}  // extern "C"
