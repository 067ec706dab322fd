// Float64 CPU oracle for the tile-based 3D Gaussian splatting training step.
//
// TEST INFRASTRUCTURE. This library exists to check the CUDA library. Only the test suite, the
// smoke check and the benchmark's CPU-baseline leg may load it. It shares no code, header,
// table or constant generator with the CUDA path, and the CUDA path never calls it.
//
// What it computes. The cited papers state the method only at the level of its
// phases: a 3D Gaussian splatting scene is rendered by a rasterization pipeline and trained by
// gradient descent, and the gradient computation accumulates per-Gaussian gradients with a very
// large number of atomic updates (DISTWAR: Fast Differentiable Rendering on Raster-based
// Rendering Pipelines, Abstract; ARC: Warp-level Adaptive Atomic Reduction in GPUs to Accelerate
// Differentiable Rendering, Abstract). The per-view phases are preprocessing, rendering and
// backward computation (Odin: Primitive-Level Synchronization for Distributed Point-Based Neural
// Rendering, Figure 7). The arithmetic of each phase below is the plainest reading of that
// pipeline as 3D Gaussian splatting defines it; each convention is stated where it is used.
//
// Precision. Everything is float64, except two quantities that the method turns into integers
// from a float32 value, where the oracle takes the same float32 decision as the kernel:
//   * the depth sort key is the float32 view-space depth, evaluated as the fused
//     multiply-add chain fma(R20, x, fma(R21, y, fma(R22, z, t2))), and
//   * the tile rectangle is evaluated in float64 from the float32 2D mean and integer radius.
// Where a float32 kernel could take a different discrete decision than this float64 code (a
// ceiling, a threshold test), the oracle reports the decision as "marginal" with a flag, using
// an explicit bound on the float32 error; the tests compare everything else exactly.
//
// Parallelism: OpenMP over Gaussians (preprocess) and over tiles (render). Every per-pixel and
// per-Gaussian computation is sequential and in the order the method states; per-Gaussian gradient
// sums are formed per tile and added in tile order, so results do not depend on the thread count.

#include <algorithm>
#include <cmath>
#include <cstdint>
#include <cstring>
#include <vector>

#ifdef _OPENMP
#include <omp.h>
#endif

extern "C" {

struct OrCamera {
    float R[9];      // world -> camera rotation, row-major
    float t[3];      // p_cam = R p_world + t
    float fx, fy, cx, cy;
    int32_t width, height;
    float bg[3];
};

struct OrOptions {
    double near_z;          // cull when the float32 depth is <= near_z
    double lowpass;         // screen-space dilation added to the 2D covariance diagonal (px^2)
    double jacobian_clamp;  // clamp x/z, y/z to +-clamp * tan(half field of view); <= 0 disables
    int32_t sh_degree;      // 0..3
    int32_t threads;        // OpenMP threads, 0 = all
};

struct OrRenderStats {
    int64_t pairs_evaluated;   // (pixel, list entry) pairs visited before termination
    int64_t pairs_blended;     // pairs that were alpha-blended
    int64_t marginal_pixels;   // pixels with at least one marginal decision
    int64_t warp_gauss_active; // (tile, 16x8 pixel block, Gaussian) triples with >= 1 blending pixel
    int64_t tile_gauss_active; // (tile, Gaussian) pairs with >= 1 blending pixel
    int64_t lane_hist[33];     // histogram over active (16x8 block, Gaussian) of the lanes (pixel
                               // columns of four: (x, y), (x, y + 2), (x, y + 4), (x, y + 6) of the
                               // block) with a blending pixel
};

}  // extern "C"

namespace {

constexpr int kTile = 16;
constexpr double kPi = 3.14159265358979323846;

// ---------------------------------------------------------------------------------------------
// Forward-mode dual numbers. The preprocess backward is the derivative of the preprocess
// forward; the oracle obtains it by running the very same forward code on dual numbers.
// ---------------------------------------------------------------------------------------------
template <int NV>
struct Dual {
    double v;
    double d[NV];
    Dual() : v(0.0) { std::memset(d, 0, sizeof(d)); }
    Dual(double x) : v(x) { std::memset(d, 0, sizeof(d)); }  // NOLINT: implicit on purpose
    static Dual var(double x, int i) { Dual r(x); r.d[i] = 1.0; return r; }
};

template <int NV> Dual<NV> operator+(const Dual<NV>& a, const Dual<NV>& b) {
    Dual<NV> r(a.v + b.v); for (int i = 0; i < NV; ++i) r.d[i] = a.d[i] + b.d[i]; return r; }
template <int NV> Dual<NV> operator-(const Dual<NV>& a, const Dual<NV>& b) {
    Dual<NV> r(a.v - b.v); for (int i = 0; i < NV; ++i) r.d[i] = a.d[i] - b.d[i]; return r; }
template <int NV> Dual<NV> operator-(const Dual<NV>& a) {
    Dual<NV> r(-a.v); for (int i = 0; i < NV; ++i) r.d[i] = -a.d[i]; return r; }
template <int NV> Dual<NV> operator*(const Dual<NV>& a, const Dual<NV>& b) {
    Dual<NV> r(a.v * b.v); for (int i = 0; i < NV; ++i) r.d[i] = a.d[i] * b.v + a.v * b.d[i]; return r; }
template <int NV> Dual<NV> operator/(const Dual<NV>& a, const Dual<NV>& b) {
    Dual<NV> r(a.v / b.v);
    for (int i = 0; i < NV; ++i) r.d[i] = (a.d[i] * b.v - a.v * b.d[i]) / (b.v * b.v);
    return r; }
template <int NV> Dual<NV> operator+(const Dual<NV>& a, double b) { return a + Dual<NV>(b); }
template <int NV> Dual<NV> operator+(double a, const Dual<NV>& b) { return Dual<NV>(a) + b; }
template <int NV> Dual<NV> operator-(const Dual<NV>& a, double b) { return a - Dual<NV>(b); }
template <int NV> Dual<NV> operator-(double a, const Dual<NV>& b) { return Dual<NV>(a) - b; }
template <int NV> Dual<NV> operator*(const Dual<NV>& a, double b) { return a * Dual<NV>(b); }
template <int NV> Dual<NV> operator*(double a, const Dual<NV>& b) { return Dual<NV>(a) * b; }
template <int NV> Dual<NV> operator/(const Dual<NV>& a, double b) { return a / Dual<NV>(b); }
template <int NV> Dual<NV> operator/(double a, const Dual<NV>& b) { return Dual<NV>(a) / b; }
template <int NV> Dual<NV> exp(const Dual<NV>& a) {
    Dual<NV> r(std::exp(a.v)); for (int i = 0; i < NV; ++i) r.d[i] = r.v * a.d[i]; return r; }
template <int NV> Dual<NV> sqrt(const Dual<NV>& a) {
    Dual<NV> r(std::sqrt(a.v)); for (int i = 0; i < NV; ++i) r.d[i] = a.d[i] / (2.0 * r.v); return r; }

inline double val(double x) { return x; }
template <int NV> double val(const Dual<NV>& x) { return x.v; }
using std::exp;
using std::sqrt;

// ---------------------------------------------------------------------------------------------
// Real spherical harmonics, degrees 0..3, index k = l*l + l + m, m = -l..l.
// Definition: with the Condon-Shortley phase included in the associated Legendre function
// P_l^m(z) = (-1)^m (1 - z^2)^(m/2) d^m/dz^m P_l(z) and N_lm = sqrt((2l+1)/(4 pi) (l-m)!/(l+m)!),
//   Y_l0 = N_l0 P_l(z),  Y_l,+m = sqrt2 N_lm P_l^m(z) cos(m phi),  Y_l,-m = sqrt2 N_lm P_l^m(z) sin(m phi).
// On the unit sphere (1 - z^2)^(m/2) cos(m phi) = Re (x + i y)^m and the sine term is Im (x + i y)^m,
// so each Y is evaluated as a polynomial in (x, y, z). The Legendre polynomials come from
// Bonnet's recursion (l + 1) P_{l+1} = (2l + 1) z P_l - l P_{l-1}.
// ---------------------------------------------------------------------------------------------
struct LegendreTable {
    double c[4][4];  // c[l][k]: coefficient of z^k in P_l
    LegendreTable() {
        std::memset(c, 0, sizeof(c));
        c[0][0] = 1.0;
        c[1][1] = 1.0;
        for (int l = 1; l < 3; ++l)
            for (int k = 0; k < 4; ++k) {
                double up = (k > 0) ? c[l][k - 1] : 0.0;
                c[l + 1][k] = ((2 * l + 1) * up - l * c[l - 1][k]) / (l + 1);
            }
    }
};
const LegendreTable kLeg;

double factorial(int n) { double r = 1.0; for (int i = 2; i <= n; ++i) r *= i; return r; }

template <class S>
void sh_basis(int deg, const S& x, const S& y, const S& z, S* Y) {
    for (int l = 0; l <= deg; ++l) {
        for (int m = 0; m <= l; ++m) {
            // m-th derivative of P_l evaluated at z
            S dm(0.0);
            S zp(1.0);
            for (int k = m; k <= l; ++k) {
                double coef = kLeg.c[l][k] * factorial(k) / factorial(k - m);
                dm = dm + coef * zp;
                zp = zp * z;
            }
            // (x + i y)^m
            S re(1.0), im(0.0);
            for (int j = 0; j < m; ++j) {
                S nre = re * x - im * y;
                S nim = re * y + im * x;
                re = nre; im = nim;
            }
            double nlm = std::sqrt((2 * l + 1) / (4.0 * kPi) * factorial(l - m) / factorial(l + m));
            double cs = (m % 2) ? -1.0 : 1.0;
            if (m == 0) {
                Y[l * l + l] = nlm * dm;
            } else {
                double s2 = std::sqrt(2.0) * nlm * cs;
                Y[l * l + l + m] = s2 * dm * re;
                Y[l * l + l - m] = s2 * dm * im;
            }
        }
    }
}

// Rotation matrix of the unit quaternion (w, x, y, z) (row-major).
template <class S>
void quat_to_rotmat(const S q[4], S R[9]) {
    const S &w = q[0], &x = q[1], &y = q[2], &z = q[3];
    R[0] = 1.0 - 2.0 * (y * y + z * z); R[1] = 2.0 * (x * y - w * z);       R[2] = 2.0 * (x * z + w * y);
    R[3] = 2.0 * (x * y + w * z);       R[4] = 1.0 - 2.0 * (x * x + z * z); R[5] = 2.0 * (y * z - w * x);
    R[6] = 2.0 * (x * z - w * y);       R[7] = 2.0 * (y * z + w * x);       R[8] = 1.0 - 2.0 * (x * x + y * y);
}

// Depth sort key: float32 view-space depth, fixed fused multiply-add order (see file header).
float depth_key(const OrCamera& cam, const float* m) {
    return std::fmaf(cam.R[6], m[0], std::fmaf(cam.R[7], m[1], std::fmaf(cam.R[8], m[2], cam.t[2])));
}

struct Rect { int x0, x1, y0, y1; bool empty; bool marginal; };

// Tiles overlapped by the 3-sigma square of a projected Gaussian. In pixel-index coordinates
// (pixel i has its centre at continuous coordinate i + 0.5, so xh = mean_x - 0.5), tile tx covers
// pixel indices 16 tx .. 16 tx + 15 and overlaps the square [xh - r, xh + r] iff
// ceil((xh - r - 15) / 16) <= tx <= floor((xh + r) / 16); likewise for y. Evaluated in float64 from
// the float32 mean, where every step is exact.
Rect tile_rect(float mx, float my, int r, int tiles_x, int tiles_y) {
    Rect R{};
    double xh = (double)mx - 0.5, yh = (double)my - 0.5;
    double fx0 = std::ceil((xh - r - 15.0) / 16.0), fx1 = std::floor((xh + r) / 16.0);
    double fy0 = std::ceil((yh - r - 15.0) / 16.0), fy1 = std::floor((yh + r) / 16.0);
    fx0 = std::max(fx0, 0.0); fy0 = std::max(fy0, 0.0);
    fx1 = std::min(fx1, (double)(tiles_x - 1)); fy1 = std::min(fy1, (double)(tiles_y - 1));
    R.empty = !(fx0 <= fx1 && fy0 <= fy1);
    if (!R.empty) { R.x0 = (int)fx0; R.x1 = (int)fx1; R.y0 = (int)fy0; R.y1 = (int)fy1; }
    // Marginal: a boundary lies within 1e-3 px of a tile edge, where a float32 mean that differs
    // from the float64 one in its last bits could move the rectangle.
    auto near_edge = [](double v) {
        double q = v / 16.0;
        return std::fabs(q - std::nearbyint(q)) * 16.0 < 1e-3;
    };
    R.marginal = near_edge(xh - r - 15.0) || near_edge(xh + r) || near_edge(yh - r - 15.0) || near_edge(yh + r);
    return R;
}

template <class S>
struct Projected {
    bool culled;
    float depth32;
    S mean2d[2];
    S cov2d[3];   // (a, b, c) of the dilated 2D covariance [[a, b], [b, c]]
    S conic[3];   // (A, B, C) of its inverse
    S opacity;
    S rgb[3];
    bool rgb_clamped[3];
    double lambda_max;
    double Y[16];
};

// Per-Gaussian preprocessing (the "preprocessing" phase of one view): EWA projection of the 3D
// covariance to a 2D conic, 3-sigma radius, opacity and view-dependent colour.
template <class S>
void project(const S mu[3], const S ls[3], const S q[4], const S& logit, const double* shg, int deg,
             const OrCamera& cam, const OrOptions& opt, Projected<S>& P) {
    P.culled = false;
    P.lambda_max = 0.0;
    // Culling on the float32 depth (the same value that becomes the sort key), computed from the
    // float32 value of the mean.
    const float mu32[3] = {(float)val(mu[0]), (float)val(mu[1]), (float)val(mu[2])};
    P.depth32 = depth_key(cam, mu32);
    if (!(P.depth32 > (float)opt.near_z)) { P.culled = true; return; }

    double Rc[9], tc[3];
    for (int i = 0; i < 9; ++i) Rc[i] = cam.R[i];
    for (int i = 0; i < 3; ++i) tc[i] = cam.t[i];
    S p[3];
    for (int i = 0; i < 3; ++i) p[i] = Rc[3 * i] * mu[0] + Rc[3 * i + 1] * mu[1] + Rc[3 * i + 2] * mu[2] + tc[i];

    // 3D covariance Sigma = Rq diag(s^2) Rq^T with s = exp(log_scale), Rq from the normalised quaternion.
    S qn = sqrt(q[0] * q[0] + q[1] * q[1] + q[2] * q[2] + q[3] * q[3]);
    S qu[4] = {q[0] / qn, q[1] / qn, q[2] / qn, q[3] / qn};
    S Rq[9];
    quat_to_rotmat(qu, Rq);
    S s2[3];
    for (int k = 0; k < 3; ++k) { S s = exp(ls[k]); s2[k] = s * s; }
    S Sig[3][3];
    for (int i = 0; i < 3; ++i)
        for (int j = 0; j < 3; ++j) {
            S acc(0.0);
            for (int k = 0; k < 3; ++k) acc = acc + Rq[3 * i + k] * s2[k] * Rq[3 * j + k];
            Sig[i][j] = acc;
        }

    // Jacobian of the pinhole projection at p, with x/z and y/z clamped to the widened field of view.
    const S& z = p[2];
    S u = p[0] / z, v = p[1] / z;
    if (opt.jacobian_clamp > 0.0) {
        double limx = opt.jacobian_clamp * (0.5 * cam.width / (double)cam.fx);
        double limy = opt.jacobian_clamp * (0.5 * cam.height / (double)cam.fy);
        if (val(u) > limx) u = S(limx);
        if (val(u) < -limx) u = S(-limx);
        if (val(v) > limy) v = S(limy);
        if (val(v) < -limy) v = S(-limy);
    }
    double fx = cam.fx, fy = cam.fy;
    S J[2][3] = {{fx / z, S(0.0), -(fx * u) / z}, {S(0.0), fy / z, -(fy * v) / z}};
    // T = J W with W the camera rotation; 2D covariance = T Sigma T^T + lowpass I.
    S Tm[2][3];
    for (int i = 0; i < 2; ++i)
        for (int j = 0; j < 3; ++j) {
            S acc(0.0);
            for (int k = 0; k < 3; ++k) acc = acc + J[i][k] * Rc[3 * k + j];
            Tm[i][j] = acc;
        }
    S C2[2][2];
    for (int i = 0; i < 2; ++i)
        for (int j = 0; j < 2; ++j) {
            S acc(0.0);
            for (int k = 0; k < 3; ++k)
                for (int l = 0; l < 3; ++l) acc = acc + Tm[i][k] * Sig[k][l] * Tm[j][l];
            C2[i][j] = acc;
        }
    S a = C2[0][0] + opt.lowpass, b = C2[0][1], c = C2[1][1] + opt.lowpass;
    P.cov2d[0] = a; P.cov2d[1] = b; P.cov2d[2] = c;
    S det = a * c - b * b;
    if (!(val(det) > 0.0)) { P.culled = true; return; }
    P.conic[0] = c / det; P.conic[1] = -b / det; P.conic[2] = a / det;
    // Largest eigenvalue of the 2D covariance, m + sqrt(((a - c) / 2)^2 + b^2), m = (a + c) / 2.
    double av = val(a), bv = val(b), cv = val(c);
    P.lambda_max = 0.5 * (av + cv) + std::sqrt(0.25 * (av - cv) * (av - cv) + bv * bv);
    P.mean2d[0] = fx * p[0] / z + (double)cam.cx;
    P.mean2d[1] = fy * p[1] / z + (double)cam.cy;
    if (!std::isfinite(P.lambda_max) || !std::isfinite(val(P.mean2d[0])) || !std::isfinite(val(P.mean2d[1]))) {
        P.culled = true; return;
    }
    P.opacity = 1.0 / (1.0 + exp(-logit));
    // View-dependent colour: real SH evaluated at the unit direction from the camera centre
    // (-R^T t) to the mean, plus 0.5, clamped below at 0.
    double cpos[3];
    for (int j = 0; j < 3; ++j) cpos[j] = -(Rc[j] * tc[0] + Rc[3 + j] * tc[1] + Rc[6 + j] * tc[2]);
    S dvec[3] = {mu[0] - cpos[0], mu[1] - cpos[1], mu[2] - cpos[2]};
    S dn = sqrt(dvec[0] * dvec[0] + dvec[1] * dvec[1] + dvec[2] * dvec[2]);
    S Yb[16];
    sh_basis(deg, dvec[0] / dn, dvec[1] / dn, dvec[2] / dn, Yb);
    int K = (deg + 1) * (deg + 1);
    for (int k = 0; k < K; ++k) P.Y[k] = val(Yb[k]);
    for (int ch = 0; ch < 3; ++ch) {
        S acc(0.5);
        for (int k = 0; k < K; ++k) acc = acc + Yb[k] * shg[k * 3 + ch];
        P.rgb_clamped[ch] = val(acc) < 0.0;
        P.rgb[ch] = P.rgb_clamped[ch] ? S(0.0) : acc;
    }
}

// Bound on the relative error of a float32 evaluation of the conic of one Gaussian (first-order
// rounding error analysis). The 2D covariance is S = K K^T + lowpass I with K = T Rq diag(s), T = J W
// the projection Jacobian times the camera rotation. A float32 evaluation of each entry
// K_rk = s_k sum_i T_ri Rq_ik carries an absolute error of at most about 24 eps s_k sum_i |T_ri|
// (eps = 2^-24: the roundings of the normalised quaternion and the rotation entries, of exp, of J
// and T, of the products and the sum). The conic C = S^-1 then moves by
// dC = -C (dK K^T + K dK^T) C to first order; summing the magnitude of each entry's contribution
// bounds the error of the conic of the float32 K, and 8 eps of each entry's scale covers the
// float32 evaluation of the conic from K. When a Gaussian's long axis points nearly along the
// viewing ray, K is a small difference of large terms and the bound is large: the projection is
// ill-conditioned in float32. Returns (conic_rel, lambda_rel): the conic entries' error relative
// to their scale (|A|, |C|, sqrt(A C) for B) and the relative error of the largest eigenvalue of S.
std::pair<double, double> projection_rel_error(const double mu[3], const double ls[3], const double q[4],
                                               const OrCamera& cam, const OrOptions& opt,
                                               const Projected<double>& P) {
    const double eps = std::ldexp(1.0, -24);
    double p[3];
    for (int i = 0; i < 3; ++i) p[i] = (double)cam.R[3 * i] * mu[0] + (double)cam.R[3 * i + 1] * mu[1] +
                                       (double)cam.R[3 * i + 2] * mu[2] + (double)cam.t[i];
    const double qn = std::sqrt(q[0] * q[0] + q[1] * q[1] + q[2] * q[2] + q[3] * q[3]);
    const double qu[4] = {q[0] / qn, q[1] / qn, q[2] / qn, q[3] / qn};
    double Rq[9];
    quat_to_rotmat<double>(qu, Rq);
    double u = p[0] / p[2], v = p[1] / p[2];
    if (opt.jacobian_clamp > 0.0) {
        const double limx = opt.jacobian_clamp * (0.5 * cam.width / (double)cam.fx);
        const double limy = opt.jacobian_clamp * (0.5 * cam.height / (double)cam.fy);
        u = std::max(-limx, std::min(limx, u));
        v = std::max(-limy, std::min(limy, v));
    }
    const double J[2][3] = {{cam.fx / p[2], 0.0, -cam.fx * u / p[2]}, {0.0, cam.fy / p[2], -cam.fy * v / p[2]}};
    double T[2][3], K[2][3], E[2][3];
    for (int r = 0; r < 2; ++r)
        for (int j = 0; j < 3; ++j) {
            T[r][j] = 0.0;
            for (int k = 0; k < 3; ++k) T[r][j] += J[r][k] * (double)cam.R[3 * k + j];
        }
    for (int r = 0; r < 2; ++r)
        for (int k = 0; k < 3; ++k) {
            const double sk = std::exp(ls[k]);
            double val = 0.0, mag = 0.0;
            for (int i = 0; i < 3; ++i) {
                val += T[r][i] * Rq[3 * i + k];
                mag += std::fabs(T[r][i]);
            }
            K[r][k] = sk * val;
            E[r][k] = 24.0 * eps * sk * mag;
        }
    const double Cm[2][2] = {{P.conic[0], P.conic[1]}, {P.conic[1], P.conic[2]}};
    double bound[2][2] = {{0.0, 0.0}, {0.0, 0.0}}, dlam = 0.0;
    for (int r = 0; r < 2; ++r)
        for (int k = 0; k < 3; ++k) {
            // dS / dK_rk = e_r K_k^T + K_k e_r^T, K_k the k-th column of K
            double D[2][2];
            for (int i = 0; i < 2; ++i)
                for (int j = 0; j < 2; ++j) D[i][j] = (i == r ? K[j][k] : 0.0) + (j == r ? K[i][k] : 0.0);
            for (int i = 0; i < 2; ++i)
                for (int j = 0; j < 2; ++j) {
                    double x = 0.0;
                    for (int a = 0; a < 2; ++a)
                        for (int b = 0; b < 2; ++b) x += Cm[i][a] * D[a][b] * Cm[b][j];
                    bound[i][j] += std::fabs(x) * E[r][k];
                }
            dlam += 2.0 * std::sqrt(K[0][k] * K[0][k] + K[1][k] * K[1][k]) * E[r][k];
        }
    const double A = P.conic[0], C = P.conic[2];
    const double conic_rel = std::max(std::max(bound[0][0] / std::fabs(A), bound[1][1] / std::fabs(C)),
                                      bound[0][1] / std::sqrt(A * C)) + 8.0 * eps;
    const double lambda_rel = dlam / P.lambda_max + 8.0 * eps;
    return {conic_rel, lambda_rel};
}

int n_threads(int t) {
#ifdef _OPENMP
    return t > 0 ? t : omp_get_max_threads();
#else
    (void)t;
    return 1;
#endif
}

// Per-Gaussian gradient sums in a fixed order. The render backward keeps, for every entry of the
// sorted list (one (tile, Gaussian) pair), that entry's partial sum over the tile's pixels; the
// partials are then added into each Gaussian's total in list order, which is tile order. The
// result therefore does not depend on the number of threads or on how tiles were scheduled.
// Tiles are processed in groups of consecutive tiles whose lists hold at most kGroupEntries
// entries together (a longer list forms a group of its own), to bound the memory of the partials.
constexpr int64_t kGroupEntries = int64_t(1) << 23;

struct TileGroup { int64_t t0, t1, p0, p1; };  // tiles [t0, t1), list positions [p0, p1)

std::vector<TileGroup> tile_groups(const uint32_t* ranges, int64_t T) {
    std::vector<TileGroup> out;
    int64_t t = 0;
    while (t < T) {
        TileGroup g{t, t, -1, -1};
        int64_t held = 0;
        for (; g.t1 < T; ++g.t1) {
            const int64_t s = ranges[2 * g.t1], e = ranges[2 * g.t1 + 1];
            const int64_t len = e > s ? e - s : 0;
            if (g.t1 > g.t0 && held + len > kGroupEntries) break;
            held += len;
            if (len > 0) {
                if (g.p0 < 0) g.p0 = s;
                g.p1 = e;
            }
        }
        if (g.p0 < 0) g.p0 = g.p1 = 0;
        out.push_back(g);
        t = g.t1;
    }
    return out;
}

// out[vals[pos] * out_stride + j] += part[(pos - p0) * stride + j] for pos = p0 .. p1 - 1 in that
// order, j < ncomp. Components are independent sums, so they run on separate threads.
void add_partials_in_list_order(const std::vector<double>& part, int stride, int ncomp, const uint32_t* vals,
                                int64_t p0, int64_t p1, double* out, int out_stride, int threads) {
#pragma omp parallel for schedule(static) num_threads(std::min(ncomp, n_threads(threads)))
    for (int j = 0; j < ncomp; ++j)
        for (int64_t pos = p0; pos < p1; ++pos)
            out[(size_t)vals[pos] * out_stride + j] += part[(size_t)(pos - p0) * stride + j];
}

}  // namespace

extern "C" {

// Real SH basis at a direction (normalised here), degree <= 3, written to Y[(deg+1)^2].
void or_sh_basis(int deg, const double* dir, double* Y) {
    double n = std::sqrt(dir[0] * dir[0] + dir[1] * dir[1] + dir[2] * dir[2]);
    sh_basis<double>(deg, dir[0] / n, dir[1] / n, dir[2] / n, Y);
}

void or_quat_to_rotmat(const double* q, double* R) {
    double n = std::sqrt(q[0] * q[0] + q[1] * q[1] + q[2] * q[2] + q[3] * q[3]);
    double qu[4] = {q[0] / n, q[1] / n, q[2] / n, q[3] / n};
    quat_to_rotmat<double>(qu, R);
}

// flags: bit0 culled, bit1 radius marginal, bit2 tile-rectangle marginal, bit3 projection
// ill-conditioned in float32 (conic_tol above 1e-4). conic_tol (may be NULL): the bound of
// projection_rel_error on the conic's relative float32 error.
int or_preprocess(int64_t n, const double* mean3d, const double* log_scale, const double* quat,
                  const double* logit, const double* sh, const OrCamera* cam, const OrOptions* opt,
                  double* mean2d, double* conic, double* opacity, double* rgb, float* depth,
                  int32_t* radius, uint32_t* tiles_touched, uint8_t* flags, double* cov2d, double* mean_tol,
                  double* conic_tol) {
    if (n < 0 || !cam || !opt) return -1;
    const int deg = opt->sh_degree, K = (deg + 1) * (deg + 1);
    const int tiles_x = (cam->width + kTile - 1) / kTile, tiles_y = (cam->height + kTile - 1) / kTile;
#pragma omp parallel for schedule(static) num_threads(n_threads(opt->threads))
    for (int64_t g = 0; g < n; ++g) {
        double mu[3], ls[3], q[4];
        for (int i = 0; i < 3; ++i) { mu[i] = mean3d[3 * g + i]; ls[i] = log_scale[3 * g + i]; }
        for (int i = 0; i < 4; ++i) q[i] = quat[4 * g + i];
        Projected<double> P;
        project<double>(mu, ls, q, logit[g], sh + g * K * 3, deg, *cam, *opt, P);
        uint8_t f = 0;
        int r = 0;
        uint32_t tt = 0;
        if (!P.culled && !(std::ceil(3.0 * std::sqrt(P.lambda_max)) < 16777216.0)) P.culled = true;  // radius >= 2^24 px
        double ctol = 0.0;
        if (!P.culled) {
            const auto rel = projection_rel_error(mu, ls, q, *cam, *opt, P);
            ctol = rel.first;
            if (ctol > 1e-4) f |= 8;
            double s = 3.0 * std::sqrt(P.lambda_max);
            r = (int)std::ceil(s);
            // 3 sqrt(lambda) carries half of lambda's relative error
            if (std::fabs(s - std::nearbyint(s)) < std::max(1e-5, rel.second) * s) f |= 2;
            Rect R = tile_rect((float)P.mean2d[0], (float)P.mean2d[1], r, tiles_x, tiles_y);
            if (R.marginal) f |= 4;
            if (R.empty) P.culled = true;
            else tt = (uint32_t)((R.x1 - R.x0 + 1) * (R.y1 - R.y0 + 1));
        }
        if (P.culled) { f |= 1; r = 0; tt = 0; }
        depth[g] = P.depth32;
        radius[g] = r;
        tiles_touched[g] = tt;
        flags[g] = f;
        for (int i = 0; i < 2; ++i) mean2d[2 * g + i] = P.culled ? 0.0 : P.mean2d[i];
        for (int i = 0; i < 3; ++i) {
            conic[3 * g + i] = P.culled ? 0.0 : P.conic[i];
            rgb[3 * g + i] = P.culled ? 0.0 : P.rgb[i];
            if (cov2d) cov2d[3 * g + i] = P.culled ? 0.0 : P.cov2d[i];
        }
        opacity[g] = P.culled ? 0.0 : P.opacity;
        if (conic_tol) conic_tol[g] = P.culled ? 0.0 : ctol;
        if (mean_tol) {
            // Bound on how far a float32 evaluation of the projected mean may lie from this one:
            // 2^-22 (4 units in the last place) of the magnitudes it is computed from.
            double mag = std::fabs(P.mean2d[0]) + std::fabs(P.mean2d[1]);
            if (!P.culled) {
                const double z = P.depth32;
                double sx = std::fabs((double)cam->t[0]), sy = std::fabs((double)cam->t[1]);
                for (int i = 0; i < 3; ++i) {
                    sx += std::fabs((double)cam->R[i] * mu[i]);
                    sy += std::fabs((double)cam->R[3 + i] * mu[i]);
                }
                mag += (cam->fx * sx + cam->fy * sy) / z;
            }
            mean_tol[g] = std::ldexp(mag, -22);
        }
    }
    return 0;
}

// Tile duplication and sort. For every Gaussian in index order with radius > 0, one entry per
// overlapped tile in row-major order of its rectangle: key = tile << 32 | bits(float32 depth),
// value = Gaussian index. The list is then stably sorted by key (std::stable_sort), so ties in
// (tile, depth) keep index order. ranges[2 t], ranges[2 t + 1] = [start, end) of tile t.
// Returns the number of duplicates D; nothing is written when D > capacity.
int64_t or_bin(int64_t n, const float* mean2d, const float* depth, const int32_t* radius,
               int32_t width, int32_t height, uint64_t* keys, uint32_t* vals, int64_t capacity,
               uint32_t* ranges) {
    const int tiles_x = (width + kTile - 1) / kTile, tiles_y = (height + kTile - 1) / kTile;
    const int64_t T = (int64_t)tiles_x * tiles_y;
    std::vector<std::pair<uint64_t, uint32_t>> list;
    for (int64_t g = 0; g < n; ++g) {
        if (radius[g] <= 0) continue;
        Rect R = tile_rect(mean2d[2 * g], mean2d[2 * g + 1], radius[g], tiles_x, tiles_y);
        if (R.empty) continue;
        uint32_t dbits;
        std::memcpy(&dbits, &depth[g], 4);
        for (int ty = R.y0; ty <= R.y1; ++ty)
            for (int tx = R.x0; tx <= R.x1; ++tx) {
                uint64_t tile = (uint64_t)ty * tiles_x + tx;
                list.emplace_back((tile << 32) | dbits, (uint32_t)g);
            }
    }
    const int64_t D = (int64_t)list.size();
    if (D > capacity) return D;
    std::stable_sort(list.begin(), list.end(),
                     [](const std::pair<uint64_t, uint32_t>& a, const std::pair<uint64_t, uint32_t>& b) {
                         return a.first < b.first;
                     });
    for (int64_t t = 0; t < T; ++t) { ranges[2 * t] = 0; ranges[2 * t + 1] = 0; }
    for (int64_t i = 0; i < D; ++i) {
        keys[i] = list[i].first;
        vals[i] = list[i].second;
        uint64_t tile = list[i].first >> 32;
        if (i == 0 || (list[i - 1].first >> 32) != tile) ranges[2 * tile] = (uint32_t)i;
        if (i == D - 1 || (list[i + 1].first >> 32) != tile) ranges[2 * tile + 1] = (uint32_t)(i + 1);
    }
    return D;
}

// Rendering ("rendering" phase) and, when dl_dimage is given, the gradient computation
// ("backward computation" phase) of one view.
//
// Forward, per pixel (centre at (px + 0.5, py + 0.5)), front to back over its tile's list:
//   d = mean2d - centre, power = -(A dx^2 + C dy^2) / 2 - B dx dy;
//   skip records whose conic [[A, B], [B, C]] is not positive definite; skip when power > 0; alpha = min(0.99, opacity exp(power)); skip when alpha < float32(1/255);
//   stop before a Gaussian whose T (1 - alpha) < float32(1e-4) (that Gaussian is not blended);
//   colour += rgb alpha T; T *= 1 - alpha.
//   image = colour + T bg; t_final = T; n_contrib = 1 + position (in the tile's list) of the last
//   blended entry, 0 if none.
// Backward: exact derivative of that forward with the per-pixel list of blended entries kept
// (alpha_i, T_i), upstream gradient g = dL/dpixel:
//   dL/drgb_i = alpha_i T_i g;  dL/dalpha_i = sum_ch g_ch (rgb_i,ch T_i - S_i,ch / (1 - alpha_i)),
//   with S_i the colour blended behind i plus t_final bg; alpha = min(0.99, o G): its derivative
//   is 0 where o G > 0.99, else dL/do = G dL/dalpha and dL/dpower = o G dL/dalpha.
// grad2d[g] = (dmean_x, dmean_y, dA, dB, dC, dopacity, dr, dg, db), summed over pixels.
int or_render(int64_t n, const double* mean2d, const double* conic, const double* opacity,
              const double* rgb, const uint32_t* vals, const uint32_t* ranges, const OrCamera* cam,
              const float* dl_dimage, double* image, double* t_final, uint32_t* n_contrib,
              uint32_t* n_blended, uint8_t* pix_flags, uint64_t* pix_sig, double* grad2d,
              OrRenderStats* stats, int threads, const double* mean_tol, double conic_rel,
              const double* conic_scale_tol, double opacity_rel, double* pix_err) {
    (void)n;
    const int W = cam->width, H = cam->height;
    const int tiles_x = (W + kTile - 1) / kTile, tiles_y = (H + kTile - 1) / kTile;
    const int64_t T = (int64_t)tiles_x * tiles_y;
    const double alpha_min = (double)(1.0f / 255.0f);
    const double t_min = (double)1e-4f;
    const double eps32 = std::ldexp(1.0, -24);
    const double clamp_gap = std::fabs((double)0.99f - 0.99) / (1.0 - 0.99);
    if (grad2d) std::memset(grad2d, 0, sizeof(double) * 9 * (size_t)n);
    OrRenderStats st{};
    std::vector<double> part;  // per list entry: its gradient partial sum over the tile's pixels

    for (const TileGroup& grp : tile_groups(ranges, T)) {
        if (grad2d) part.assign((size_t)(grp.p1 - grp.p0) * 9, 0.0);
#pragma omp parallel num_threads(n_threads(threads))
        {
            OrRenderStats ls{};
            struct Blend { int64_t pos; uint32_t g; double alpha, T, G, dx, dy; bool clamped; };
            std::vector<Blend> bl;
            // per tile [2 warps][len]: which lanes have a blending pixel. A warp of the backward covers
            // a 16x8 block of the tile (rows 8w..8w+7) and its lane l the four pixels
            // (l % 16, l / 16 + 2q), q = 0..3, of it
            std::vector<uint32_t> wmask;
#pragma omp for schedule(dynamic, 4)
            for (int64_t tile = grp.t0; tile < grp.t1; ++tile) {
                const int tx = (int)(tile % tiles_x), ty = (int)(tile / tiles_x);
                const int64_t s = ranges[2 * tile], e = ranges[2 * tile + 1];
                const int64_t len = e - s;
                // this tile's entries in the group's partials (positions s .. e - 1)
                double* acc = (grad2d && len > 0) ? part.data() + (size_t)(s - grp.p0) * 9 : nullptr;
                wmask.assign((size_t)len * 2, 0u);
                for (int ly = 0; ly < kTile; ++ly)
                    for (int lx = 0; lx < kTile; ++lx) {
                        const int px = tx * kTile + lx, py = ty * kTile + ly;
                        if (px >= W || py >= H) continue;
                        const double cxp = px + 0.5, cyp = py + 0.5;
                        double Tr = 1.0, col[3] = {0.0, 0.0, 0.0};
                        double eT = 0.0;  // bound on the relative float32 error of T
                        double eC = 0.0;  // bound on the colour error propagated from the alpha bounds
                        uint32_t contrib = 0, nbl = 0;
                        uint8_t pf = 0;
                        uint64_t sig = 1469598103934665603ull;  // FNV-1a over (position, clamped) of blended entries
                        bl.clear();
                        for (int64_t pos = s; pos < e; ++pos) {
                            const uint32_t g = vals[pos];
                            ls.pairs_evaluated++;
                            const double dx = mean2d[2 * g] - cxp, dy = mean2d[2 * g + 1] - cyp;
                            const double A = conic[3 * g], B = conic[3 * g + 1], C = conic[3 * g + 2];
                            // a record whose conic is not positive definite is not a Gaussian: never blended
                            if (!(A > 0.0) || !(A * C - B * B > 0.0)) continue;
                            const double power = -0.5 * (A * dx * dx + C * dy * dy) - B * dx * dy;
                            // Bound on the float32 error of power when it is evaluated as
                            // -(A u^2 + D dy^2)/2 with u = dx + (B/A) dy, D = (A C - B^2)/A (terms >= 0): u carries
                            // eps (|u| + |B/A dy|), A u^2 and D dy^2 a few eps each; 4e-7 is about 7 eps.
                            const double ur = B / A * dy, u = dx + ur, D = (A * C - B * B) / A;
                            const double ep = 4e-7 * (A * std::fabs(u) * (std::fabs(u) + std::fabs(ur)) + A * u * u +
                                                      2.0 * D * dy * dy) + 1e-7;
                            if (std::fabs(power) <= ep) pf |= 4;
                            if (power > 0.0) continue;
                            // uncertainty of power when the records themselves may differ from these
                            // (a float32 preprocess): the mean by mean_tol px; the conic's quadratic form by
                            // a relative conic_rel plus the rounding of its three float32 entries (4e-7 of the
                            // term magnitudes; for elongated Gaussians this dominates along the long axis);
                            // for a Gaussian with a conditioning bound conic_scale_tol (its conic entries
                            // within that fraction of their scale |A|, |C|, sqrt(A C)), the form moves by at
                            // most that times (sqrt(A) |dx| + sqrt(C) |dy|)^2; the opacity by opacity_rel
                            double ein = opacity_rel + conic_rel * std::fabs(power);
                            if (conic_rel > 0.0)
                                ein += 4e-7 * (0.5 * (std::fabs(A) * dx * dx + std::fabs(C) * dy * dy) + std::fabs(B * dx * dy));
                            if (conic_scale_tol && conic_scale_tol[g] > 0.0) {
                                const double m = std::sqrt(A) * std::fabs(dx) + std::sqrt(std::fabs(C)) * std::fabs(dy);
                                ein += conic_scale_tol[g] * 0.5 * m * m;
                            }
                            if (mean_tol)
                                ein += mean_tol[g] * (std::fabs(A * dx + B * dy) + std::fabs(B * dx + C * dy));
                            const double G = std::exp(power);
                            const double oG = opacity[g] * G;
                            const bool clamped = oG > 0.99;
                            const double alpha = clamped ? 0.99 : oG;
                            // relative bound on alpha: the power's bound, a float32 exponential (a hardware
                            // approximation of 2^x within 2 units in the last place) and the rounding of
                            // opacity x G, 5e-7 together, and the inputs' bound
                            const double ea = ep + 5e-7 + ein;
                            if (!clamped && std::fabs(std::log(alpha / alpha_min)) < ea) pf |= 1;
                            if (alpha < alpha_min) continue;
                            const double test_T = Tr * (1.0 - alpha);
                            // relative bound on T (1 - alpha): 1 - alpha carries alpha's bound times
                            // alpha / (1 - alpha); a clamped alpha is the float32 value of 0.99 on the
                            // float32 side, whose 1 - alpha differs from 0.01 by clamp_gap; two roundings
                            const double eT_next = eT + (clamped ? clamp_gap : ea * alpha / (1.0 - alpha)) + 2.0 * eps32;
                            if (std::fabs(test_T / t_min - 1.0) < 2.0 * eT_next + 4.0 * eps32) pf |= 2;
                            if (test_T < t_min) break;
                            for (int ch = 0; ch < 3; ++ch) col[ch] += rgb[3 * g + ch] * alpha * Tr;
                            {
                                // |dC/dalpha_i| <= T_i (|c_i| + max colour behind); the colour behind is bounded
                                // by the largest colour or background value
                                double cm = 0.0;
                                for (int ch = 0; ch < 3; ++ch)
                                    cm = std::max(cm, std::max(std::fabs(rgb[3 * g + ch]), std::fabs((double)cam->bg[ch])));
                                eC += 2.0 * cm * (clamped ? 0.0 : ea) * alpha * Tr;
                            }
                            bl.push_back({pos, g, alpha, Tr, G, dx, dy, clamped});
                            sig = (sig ^ (uint64_t)(2 * (pos - s) + (clamped ? 1 : 0))) * 1099511628211ull;
                            Tr = test_T;
                            eT = eT_next;
                            contrib = (uint32_t)(pos - s + 1);
                            nbl++;
                            ls.pairs_blended++;
                            wmask[(size_t)(ly / 8) * len + (pos - s)] |= 1u << (lx + 16 * (ly % 2));
                        }
                        const int64_t pix = (int64_t)py * W + px;
                        for (int ch = 0; ch < 3; ++ch) image[(int64_t)ch * W * H + pix] = col[ch] + Tr * cam->bg[ch];
                        t_final[pix] = Tr;
                        n_contrib[pix] = contrib;
                        if (n_blended) n_blended[pix] = nbl;
                        if (pix_flags) pix_flags[pix] = pf;
                        if (pix_sig) pix_sig[pix] = sig;
                        if (pix_err) {
                            double bm = 0.0;
                            for (int ch = 0; ch < 3; ++ch) bm = std::max(bm, std::fabs((double)cam->bg[ch]));
                            pix_err[pix] = eC + Tr * eT * bm;
                        }
                        if (pf) ls.marginal_pixels++;
                        if (!grad2d) continue;
                        double gpix[3];
                        for (int ch = 0; ch < 3; ++ch) gpix[ch] = dl_dimage[(int64_t)ch * W * H + pix];
                        double S[3];
                        for (int ch = 0; ch < 3; ++ch) S[ch] = Tr * cam->bg[ch];
                        for (int64_t k = (int64_t)bl.size() - 1; k >= 0; --k) {
                            const Blend& b = bl[k];
                            const double* c = rgb + 3 * b.g;
                            double* a = acc + (size_t)(b.pos - s) * 9;
                            double dalpha = 0.0;
                            for (int ch = 0; ch < 3; ++ch) {
                                a[6 + ch] += b.alpha * b.T * gpix[ch];
                                dalpha += gpix[ch] * (c[ch] * b.T - S[ch] / (1.0 - b.alpha));
                            }
                            for (int ch = 0; ch < 3; ++ch) S[ch] += c[ch] * b.alpha * b.T;
                            if (b.clamped) continue;
                            const double o = opacity[b.g];
                            const double dpower = o * b.G * dalpha;
                            const double A = conic[3 * b.g], B = conic[3 * b.g + 1], C = conic[3 * b.g + 2];
                            a[0] += -(A * b.dx + B * b.dy) * dpower;
                            a[1] += -(B * b.dx + C * b.dy) * dpower;
                            a[2] += -0.5 * b.dx * b.dx * dpower;
                            a[3] += -b.dx * b.dy * dpower;
                            a[4] += -0.5 * b.dy * b.dy * dpower;
                            a[5] += b.G * dalpha;
                        }
                    }
                for (int64_t k = 0; k < len; ++k) {
                    bool any = false;
                    for (int w = 0; w < 2; ++w) {
                        uint32_t m = wmask[(size_t)w * len + k];
                        if (m) {
                            int c = 0;
                            for (; m; m &= m - 1) ++c;
                            ls.warp_gauss_active++;
                            ls.lane_hist[c]++;
                            any = true;
                        }
                    }
                    if (any) ls.tile_gauss_active++;
                }
            }
#pragma omp critical
            {
                st.pairs_evaluated += ls.pairs_evaluated;
                st.pairs_blended += ls.pairs_blended;
                st.marginal_pixels += ls.marginal_pixels;
                st.warp_gauss_active += ls.warp_gauss_active;
                st.tile_gauss_active += ls.tile_gauss_active;
                for (int i = 0; i < 33; ++i) st.lane_hist[i] += ls.lane_hist[i];
            }
        }
        if (grad2d) add_partials_in_list_order(part, 9, 9, vals, grp.p0, grp.p1, grad2d, 9, threads);
    }
    if (stats) *stats = st;
    return 0;
}

// Preprocess backward: gradients of the loss with respect to mean3d, log_scale, quat (through the
// normalisation), opacity logit and SH, given grad2d = dL/d(mean2d, conic, opacity, rgb) per
// Gaussian. The Jacobian of the per-Gaussian preprocessing is taken by running project() on dual
// numbers in the 11 non-SH parameters; SH coefficients enter the colour linearly, so
// dL/dsh[k][ch] = Y_k dL/drgb_ch where the colour was not clamped. Culled Gaussians get zeros.
//
// grad_mag (may be NULL) [n][11]: for each of the 11 non-SH parameters (mean3d, log_scale, quat,
// logit) the sum of the magnitudes of the terms its gradient adds up, sum_o |dL/dout_o d out_o/dp|.
// Where it is much larger than the gradient itself, the chain rule cancels, and a float32
// evaluation (or 2D gradients known to a relative accuracy) can only reach that accuracy times this
// magnitude.
int or_preprocess_bwd(int64_t n, const double* mean3d, const double* log_scale, const double* quat,
                      const double* logit, const double* sh, const OrCamera* cam, const OrOptions* opt,
                      const double* grad2d, double* d_mean3d, double* d_log_scale, double* d_quat,
                      double* d_logit, double* d_sh, double* grad_mag) {
    if (n < 0 || !cam || !opt) return -1;
    const int deg = opt->sh_degree, K = (deg + 1) * (deg + 1);
    using D = Dual<11>;
#pragma omp parallel for schedule(static) num_threads(n_threads(opt->threads))
    for (int64_t g = 0; g < n; ++g) {
        D mu[3], ls[3], q[4];
        for (int i = 0; i < 3; ++i) mu[i] = D::var(mean3d[3 * g + i], i);
        for (int i = 0; i < 3; ++i) ls[i] = D::var(log_scale[3 * g + i], 3 + i);
        for (int i = 0; i < 4; ++i) q[i] = D::var(quat[4 * g + i], 6 + i);
        D lg = D::var(logit[g], 10);
        Projected<D> P;
        project<D>(mu, ls, q, lg, sh + g * K * 3, deg, *cam, *opt, P);
        double grad[11] = {0}, mag[11] = {0};
        for (int k = 0; k < K * 3; ++k) d_sh[(size_t)g * K * 3 + k] = 0.0;
        bool culled = P.culled;
        if (!culled) {
            // a Gaussian whose tile rectangle is empty is culled as well
            const int tiles_x = (cam->width + kTile - 1) / kTile, tiles_y = (cam->height + kTile - 1) / kTile;
            const double rs = std::ceil(3.0 * std::sqrt(P.lambda_max));
            culled = !(rs < 16777216.0);
            int r = culled ? 0 : (int)rs;
            culled = culled || tile_rect((float)P.mean2d[0].v, (float)P.mean2d[1].v, r, tiles_x, tiles_y).empty;
        }
        if (!culled) {
            const double* gi = grad2d + 9 * (size_t)g;
            const D* outs[9] = {&P.mean2d[0], &P.mean2d[1], &P.conic[0], &P.conic[1], &P.conic[2],
                                &P.opacity, &P.rgb[0], &P.rgb[1], &P.rgb[2]};
            for (int o = 0; o < 9; ++o)
                for (int v = 0; v < 11; ++v) {
                    grad[v] += gi[o] * outs[o]->d[v];
                    mag[v] += std::fabs(gi[o] * outs[o]->d[v]);
                }
            for (int ch = 0; ch < 3; ++ch) {
                if (P.rgb_clamped[ch]) continue;
                for (int k = 0; k < K; ++k) d_sh[(size_t)g * K * 3 + k * 3 + ch] = P.Y[k] * gi[6 + ch];
            }
        }
        for (int i = 0; i < 3; ++i) d_mean3d[3 * g + i] = grad[i];
        for (int i = 0; i < 3; ++i) d_log_scale[3 * g + i] = grad[3 + i];
        for (int i = 0; i < 4; ++i) d_quat[4 * g + i] = grad[6 + i];
        d_logit[g] = grad[10];
        if (grad_mag)
            for (int v = 0; v < 11; ++v) grad_mag[11 * (size_t)g + v] = mag[v];
    }
    return 0;
}

}  // extern "C"

// =============================================================================================
// 2D Gaussian splatting (surfels): each Gaussian is a flat disk in 3D, P(u, v) = mean + s_u u t_u
// + s_v v t_v with t_u, t_v the first two columns of its rotation, evaluated where the pixel's ray
// meets the disk's plane (Odin: Primitive-Level Synchronization for Distributed Point-Based Neural
// Rendering, Summary: 2DGS is one of the four pipelines it trains; the formulation is 2DGS's own).
//
// Record of a projected surfel (the format both sides share), 11 geometric fields + opacity + rgb:
//   A_u = s_u fx (W t_u)_x, B_u = s_u fy (W t_u)_y, C_u = s_u (W t_u)_z, likewise A_v, B_v, C_v for
//   t_v; m = (fx x_c / z_c + cx, fy y_c / z_c + cy) the projected mean and z_c its depth; c the
//   centre of the screen-space bounding box of the 3-sigma disk. With K the intrinsics, the disk
//   point (u, v) lands at homogeneous screen position T (u, v, 1), T = [K W s_u t_u | K W s_v t_v |
//   K p_c], and the pixel (x, y) constrains (u, v) by the two planes h_x = T_0 - x T_2 and
//   h_y = T_1 - y T_2: h_x = (A_u + (cx - x) C_u, A_v + (cx - x) C_v, z_c (m_x - x)), likewise h_y.
// =============================================================================================

namespace {

template <class S>
struct Projected2D {
    bool culled;
    float depth32;
    S rec[11];      // A_u, B_u, C_u, A_v, B_v, C_v, m_x, m_y, z_c, c_x, c_y
    S opacity;
    S rgb[3];
    bool rgb_clamped[3];
    double half[2];  // half extents of the bounding box of the 3-sigma disk (px)
    double Y[16];
};

template <class S>
void project2d(const S mu[3], const S ls[3], const S q[4], const S& logit, const double* shg, int deg,
               const OrCamera& cam, const OrOptions& opt, Projected2D<S>& P) {
    P.culled = false;
    const float mu32[3] = {(float)val(mu[0]), (float)val(mu[1]), (float)val(mu[2])};
    P.depth32 = depth_key(cam, mu32);
    if (!(P.depth32 > (float)opt.near_z)) { P.culled = true; return; }
    double Rc[9], tc[3];
    for (int i = 0; i < 9; ++i) Rc[i] = cam.R[i];
    for (int i = 0; i < 3; ++i) tc[i] = cam.t[i];
    S p[3];
    for (int i = 0; i < 3; ++i) p[i] = Rc[3 * i] * mu[0] + Rc[3 * i + 1] * mu[1] + Rc[3 * i + 2] * mu[2] + tc[i];
    S qn = sqrt(q[0] * q[0] + q[1] * q[1] + q[2] * q[2] + q[3] * q[3]);
    S qu[4] = {q[0] / qn, q[1] / qn, q[2] / qn, q[3] / qn};
    S Rq[9];
    quat_to_rotmat(qu, Rq);
    const S su = exp(ls[0]), sv = exp(ls[1]);
    S wu[3], wv[3];  // W t_u, W t_v (t_u, t_v = columns 0 and 1 of Rq)
    for (int i = 0; i < 3; ++i) {
        wu[i] = Rc[3 * i] * Rq[0] + Rc[3 * i + 1] * Rq[3] + Rc[3 * i + 2] * Rq[6];
        wv[i] = Rc[3 * i] * Rq[1] + Rc[3 * i + 1] * Rq[4] + Rc[3 * i + 2] * Rq[7];
    }
    const double fx = cam.fx, fy = cam.fy, cx = cam.cx, cy = cam.cy;
    P.rec[0] = su * fx * wu[0]; P.rec[1] = su * fy * wu[1]; P.rec[2] = su * wu[2];
    P.rec[3] = sv * fx * wv[0]; P.rec[4] = sv * fy * wv[1]; P.rec[5] = sv * wv[2];
    const S z = p[2];
    P.rec[6] = fx * p[0] / z + cx;
    P.rec[7] = fy * p[1] / z + cy;
    P.rec[8] = z;
    // bounding box of the disk u^2 + v^2 <= 9: from the dual conic C* = T diag(9, 9, -1) T^T, the
    // lines x = k tangent to the projected disk solve C*00 - 2 k C*02 + k^2 C*22 = 0
    const S T0[3] = {P.rec[0] + cx * P.rec[2], P.rec[3] + cx * P.rec[5], z * P.rec[6]};
    const S T1[3] = {P.rec[1] + cy * P.rec[2], P.rec[4] + cy * P.rec[5], z * P.rec[7]};
    const S T2[3] = {P.rec[2], P.rec[5], z};
    auto dual = [](const S a[3], const S b[3]) { return 9.0 * (a[0] * b[0] + a[1] * b[1]) - a[2] * b[2]; };
    const S c00 = dual(T0, T0), c11 = dual(T1, T1), c22 = dual(T2, T2), c02 = dual(T0, T2), c12 = dual(T1, T2);
    if (!(val(c22) < 0.0)) { P.culled = true; return; }  // the disk reaches the camera plane
    P.rec[9] = c02 / c22;
    P.rec[10] = c12 / c22;
    const double hx2 = val(c02) * val(c02) - val(c00) * val(c22), hy2 = val(c12) * val(c12) - val(c11) * val(c22);
    P.half[0] = std::sqrt(std::max(hx2, 0.0)) / std::fabs(val(c22));
    P.half[1] = std::sqrt(std::max(hy2, 0.0)) / std::fabs(val(c22));
    for (int i = 0; i < 11; ++i)
        if (!std::isfinite(val(P.rec[i]))) { P.culled = true; return; }
    P.opacity = 1.0 / (1.0 + exp(-logit));
    double cpos[3];
    for (int j = 0; j < 3; ++j) cpos[j] = -(Rc[j] * tc[0] + Rc[3 + j] * tc[1] + Rc[6 + j] * tc[2]);
    S dvec[3] = {mu[0] - cpos[0], mu[1] - cpos[1], mu[2] - cpos[2]};
    S dn = sqrt(dvec[0] * dvec[0] + dvec[1] * dvec[1] + dvec[2] * dvec[2]);
    S Yb[16];
    sh_basis(deg, dvec[0] / dn, dvec[1] / dn, dvec[2] / dn, Yb);
    const int K = (deg + 1) * (deg + 1);
    for (int k = 0; k < K; ++k) P.Y[k] = val(Yb[k]);
    for (int ch = 0; ch < 3; ++ch) {
        S acc(0.5);
        for (int k = 0; k < K; ++k) acc = acc + Yb[k] * shg[k * 3 + ch];
        P.rgb_clamped[ch] = val(acc) < 0.0;
        P.rgb[ch] = P.rgb_clamped[ch] ? S(0.0) : acc;
    }
}

// Radius of the square the binning uses: the larger half extent, and at least the 3-sigma extent
// of the screen-space filter (standard deviation sqrt(1/2) px).
int radius2d(const double half[2]) {
    const double r = std::ceil(std::max(std::max(half[0], half[1]), 3.0 * std::sqrt(0.5)));
    return r < 16777216.0 ? (int)r : 0;
}

// Exponent of the surfel's weight at pixel centre (x, y): the larger of the disk's Gaussian at
// the ray-plane intersection, -(u^2 + v^2)/2, and the screen-space filter around the box centre,
// -|(x, y) - c|^2 (a Gaussian of variance 1/2 px^2). u, v by Cramer's rule on the two planes.
template <class S>
S power2d(const S r[11], double cx, double cy, double x, double y, S* p3_out = nullptr, S* plp_out = nullptr) {
    const S hxu = r[0] + (cx - x) * r[2], hxv = r[3] + (cx - x) * r[5], hx1 = r[8] * (r[6] - x);
    const S hyu = r[1] + (cy - y) * r[2], hyv = r[4] + (cy - y) * r[5], hy1 = r[8] * (r[7] - y);
    const S det = hxu * hyv - hxv * hyu;
    S p3;
    if (val(det) == 0.0) {
        p3 = S(-std::numeric_limits<double>::infinity());
    } else {
        const S u = (hxv * hy1 - hx1 * hyv) / det, v = (hx1 * hyu - hxu * hy1) / det;
        p3 = -0.5 * (u * u + v * v);
    }
    const S dx = r[9] - x, dy = r[10] - y;
    const S plp = -(dx * dx + dy * dy);
    if (p3_out) *p3_out = p3;
    if (plp_out) *plp_out = plp;
    return val(p3) >= val(plp) ? p3 : plp;
}

}  // namespace

extern "C" {

// Surfel preprocessing: rec2d [n][16] = (11 geometric fields, opacity, r, g, b, 0), the float32
// depth, the binning radius (0 = culled), the tile count, and the bounding-box centre as mean2d
// [n][2] for the binning.
int or_preprocess2d(int64_t n, const double* mean3d, const double* log_scale, const double* quat,
                    const double* logit, const double* sh, const OrCamera* cam, const OrOptions* opt,
                    double* rec2d, double* mean2d, float* depth, int32_t* radius, uint32_t* tiles_touched,
                    double* half) {
    if (n < 0 || !cam || !opt) return -1;
    const int deg = opt->sh_degree, K = (deg + 1) * (deg + 1);
    const int tiles_x = (cam->width + kTile - 1) / kTile, tiles_y = (cam->height + kTile - 1) / kTile;
#pragma omp parallel for schedule(static) num_threads(n_threads(opt->threads))
    for (int64_t g = 0; g < n; ++g) {
        Projected2D<double> P;
        project2d<double>(mean3d + 3 * g, log_scale + 3 * g, quat + 4 * g, logit[g], sh + g * K * 3, deg, *cam,
                          *opt, P);
        depth[g] = P.depth32;
        double* r = rec2d + 16 * g;
        for (int i = 0; i < 16; ++i) r[i] = 0.0;
        radius[g] = 0;
        tiles_touched[g] = 0;
        mean2d[2 * g] = mean2d[2 * g + 1] = 0.0;
        half[2 * g] = half[2 * g + 1] = 0.0;
        if (P.culled) continue;
        const int rad = radius2d(P.half);
        if (rad == 0) continue;
        const Rect R = tile_rect((float)P.rec[9], (float)P.rec[10], rad, tiles_x, tiles_y);
        if (R.empty) continue;
        for (int i = 0; i < 11; ++i) r[i] = P.rec[i];
        r[11] = P.opacity;
        for (int ch = 0; ch < 3; ++ch) r[12 + ch] = P.rgb[ch];
        radius[g] = rad;
        tiles_touched[g] = (uint32_t)((R.x1 - R.x0 + 1) * (R.y1 - R.y0 + 1));
        mean2d[2 * g] = P.rec[9];
        mean2d[2 * g + 1] = P.rec[10];
        half[2 * g] = P.half[0];
        half[2 * g + 1] = P.half[1];
    }
    return 0;
}

// Surfel render forward (and backward when grad != NULL): front to back over each tile's list with
// the same alpha, threshold, clamp and termination rules as the 3D rasterizer; the backward is the
// exact derivative of that forward from the stored per-pixel (alpha_i, T_i), with d power / d record
// by dual numbers over the 11 geometric fields. grad [n][16] = dL/d(rec2d fields 0..14).
// pix_flags: 1 alpha within 1e-4 of 1/255, 2 T (1 - alpha) within 1e-4 of 1e-4, 4 the two exponents
// within 1e-4 of each other (the max may switch branches), 8 the intersection ill-conditioned.
int or_render2d(int64_t n, const double* rec2d, const uint32_t* vals, const uint32_t* ranges, const OrCamera* cam,
                const float* dl_dimage, double* image, double* t_final, uint32_t* n_contrib, uint8_t* pix_flags,
                uint64_t* pix_sig, double* grad, int threads) {
    const int W = cam->width, H = cam->height;
    const int tiles_x = (W + kTile - 1) / kTile, tiles_y = (H + kTile - 1) / kTile;
    const int64_t T = (int64_t)tiles_x * tiles_y;
    const double alpha_min = (double)(1.0f / 255.0f), t_min = (double)1e-4f;
    const double cx = cam->cx, cy = cam->cy;
    if (grad) std::memset(grad, 0, sizeof(double) * 16 * (size_t)n);
    std::vector<double> part;  // per list entry: its gradient partial sum over the tile's pixels
    for (const TileGroup& grp : tile_groups(ranges, T)) {
        if (grad) part.assign((size_t)(grp.p1 - grp.p0) * 16, 0.0);
#pragma omp parallel num_threads(n_threads(threads))
        {
            struct Blend { int64_t pos; uint32_t g; double alpha, T, G; bool clamped; double x, y; };
            std::vector<Blend> bl;
#pragma omp for schedule(dynamic, 4)
            for (int64_t tile = grp.t0; tile < grp.t1; ++tile) {
                const int tx = (int)(tile % tiles_x), ty = (int)(tile / tiles_x);
                const int64_t s = ranges[2 * tile], e = ranges[2 * tile + 1];
                const int64_t len = e - s;
                double* acc = (grad && len > 0) ? part.data() + (size_t)(s - grp.p0) * 16 : nullptr;
                for (int ly = 0; ly < kTile; ++ly)
                    for (int lx = 0; lx < kTile; ++lx) {
                        const int px = tx * kTile + lx, py = ty * kTile + ly;
                        if (px >= W || py >= H) continue;
                        const double x = px + 0.5, y = py + 0.5;
                        double Tr = 1.0, col[3] = {0.0, 0.0, 0.0};
                        uint32_t contrib = 0;
                        uint8_t pf = 0;
                        uint64_t sig = 1469598103934665603ull;  // FNV-1a over (position, clamp, branch) of blended entries
                        bl.clear();
                        for (int64_t pos = s; pos < e; ++pos) {
                            const uint32_t g = vals[pos];
                            const double* r = rec2d + 16 * (size_t)g;
                            double p3, plp;
                            const double power = power2d<double>(r, cx, cy, x, y, &p3, &plp);
                            if (std::fabs(p3 - plp) <= 1e-4 * (std::fabs(p3) + std::fabs(plp)) + 1e-7) pf |= 4;
                            const double G = std::exp(power);
                            const double oG = r[11] * G;
                            const bool clamped = oG > 0.99;
                            const double alpha = clamped ? 0.99 : oG;
                            if (!clamped && std::fabs(alpha / alpha_min - 1.0) < 1e-4) pf |= 1;
                            if (alpha < alpha_min) continue;
                            const double test_T = Tr * (1.0 - alpha);
                            if (std::fabs(test_T / t_min - 1.0) < 1e-4) pf |= 2;
                            if (test_T < t_min) break;
                            for (int ch = 0; ch < 3; ++ch) col[ch] += r[12 + ch] * alpha * Tr;
                            bl.push_back({pos, g, alpha, Tr, G, clamped, x, y});
                            sig = (sig ^ (uint64_t)(4 * (pos - s) + (clamped ? 1 : 0) + (p3 >= plp ? 2 : 0))) * 1099511628211ull;
                            Tr = test_T;
                            contrib = (uint32_t)(pos - s + 1);
                        }
                        const int64_t pix = (int64_t)py * W + px;
                        for (int ch = 0; ch < 3; ++ch) image[(int64_t)ch * W * H + pix] = col[ch] + Tr * cam->bg[ch];
                        t_final[pix] = Tr;
                        n_contrib[pix] = contrib;
                        if (pix_flags) pix_flags[pix] = pf;
                        if (pix_sig) pix_sig[pix] = sig;
                        if (!grad) continue;
                        double gpix[3], S[3];
                        for (int ch = 0; ch < 3; ++ch) {
                            gpix[ch] = dl_dimage[(int64_t)ch * W * H + pix];
                            S[ch] = Tr * cam->bg[ch];
                        }
                        for (int64_t k = (int64_t)bl.size() - 1; k >= 0; --k) {
                            const Blend& b = bl[k];
                            const double* r = rec2d + 16 * (size_t)b.g;
                            double* a = acc + (size_t)(b.pos - s) * 16;
                            double dalpha = 0.0;
                            for (int ch = 0; ch < 3; ++ch) {
                                a[12 + ch] += b.alpha * b.T * gpix[ch];
                                dalpha += gpix[ch] * (r[12 + ch] * b.T - S[ch] / (1.0 - b.alpha));
                            }
                            for (int ch = 0; ch < 3; ++ch) S[ch] += r[12 + ch] * b.alpha * b.T;
                            if (b.clamped) continue;
                            const double dpower = r[11] * b.G * dalpha;
                            using D = Dual<11>;
                            D rd[11];
                            for (int i = 0; i < 11; ++i) rd[i] = D::var(r[i], i);
                            const D pw = power2d<D>(rd, cx, cy, b.x, b.y);
                            for (int i = 0; i < 11; ++i) a[i] += pw.d[i] * dpower;
                            a[11] += b.G * dalpha;
                        }
                    }
            }
        }
        if (grad) add_partials_in_list_order(part, 16, 15, vals, grp.p0, grp.p1, grad, 16, threads);
    }
    return 0;
}

// Surfel preprocess backward: gradients of the loss with respect to mean3d, log_scale (the first
// two; the third gets 0), quat, opacity logit and SH from grad [n][16] = dL/d(record), by running
// project2d on dual numbers in the 10 non-SH parameters. Culled Gaussians get zeros.
int or_preprocess2d_bwd(int64_t n, const double* mean3d, const double* log_scale, const double* quat,
                        const double* logit, const double* sh, const OrCamera* cam, const OrOptions* opt,
                        const double* grad, double* d_mean3d, double* d_log_scale, double* d_quat, double* d_logit,
                        double* d_sh) {
    if (n < 0 || !cam || !opt) return -1;
    const int deg = opt->sh_degree, K = (deg + 1) * (deg + 1);
    const int tiles_x = (cam->width + kTile - 1) / kTile, tiles_y = (cam->height + kTile - 1) / kTile;
    using D = Dual<10>;
#pragma omp parallel for schedule(static) num_threads(n_threads(opt->threads))
    for (int64_t g = 0; g < n; ++g) {
        D mu[3], ls[3], q[4];
        for (int i = 0; i < 3; ++i) mu[i] = D::var(mean3d[3 * g + i], i);
        ls[0] = D::var(log_scale[3 * g], 3);
        ls[1] = D::var(log_scale[3 * g + 1], 4);
        ls[2] = D(log_scale[3 * g + 2]);
        for (int i = 0; i < 4; ++i) q[i] = D::var(quat[4 * g + i], 5 + i);
        D lg = D::var(logit[g], 9);
        Projected2D<D> P;
        project2d<D>(mu, ls, q, lg, sh + g * K * 3, deg, *cam, *opt, P);
        double gr[10] = {0};
        for (int k = 0; k < K * 3; ++k) d_sh[(size_t)g * K * 3 + k] = 0.0;
        bool culled = P.culled;
        if (!culled) {
            const int rad = radius2d(P.half);
            culled = rad == 0 || tile_rect((float)P.rec[9].v, (float)P.rec[10].v, rad, tiles_x, tiles_y).empty;
        }
        if (!culled) {
            const double* gi = grad + 16 * (size_t)g;
            for (int o = 0; o < 11; ++o)
                for (int v = 0; v < 10; ++v) gr[v] += gi[o] * P.rec[o].d[v];
            for (int v = 0; v < 10; ++v) gr[v] += gi[11] * P.opacity.d[v];
            for (int ch = 0; ch < 3; ++ch) {
                for (int v = 0; v < 10; ++v) gr[v] += gi[12 + ch] * P.rgb[ch].d[v];
                if (P.rgb_clamped[ch]) continue;
                for (int k = 0; k < K; ++k) d_sh[(size_t)g * K * 3 + k * 3 + ch] = P.Y[k] * gi[12 + ch];
            }
        }
        for (int i = 0; i < 3; ++i) d_mean3d[3 * g + i] = gr[i];
        d_log_scale[3 * g] = gr[3];
        d_log_scale[3 * g + 1] = gr[4];
        d_log_scale[3 * g + 2] = 0.0;
        for (int i = 0; i < 4; ++i) d_quat[4 * g + i] = gr[5 + i];
        d_logit[g] = gr[9];
    }
    return 0;
}

}  // extern "C"
