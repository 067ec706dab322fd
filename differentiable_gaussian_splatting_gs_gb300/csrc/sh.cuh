// Real spherical harmonics of degree <= 3 as polynomials of a unit direction (x, y, z).
//
// Convention: index k = l^2 + l + m (m = -l..l); Condon-Shortley phase included, i.e.
//   Y_l0 = N_l0 P_l(z), Y_l,+m = sqrt2 N_lm P_l^m(z) cos(m phi), Y_l,-m = sqrt2 N_lm P_l^m(z) sin(m phi),
// with N_lm = sqrt((2l+1)/(4 pi) (l-m)!/(l+m)!). Written out on the unit sphere these are the
// polynomials below (the constants are those closed forms evaluated, e.g. sqrt(3/(4 pi))).
#pragma once

namespace gs {

constexpr float kY00 = 0.28209479177387814f;   // 1 / (2 sqrt(pi))
constexpr float kY1 = 0.48860251190291992f;    // sqrt(3 / (4 pi))
constexpr float kY2a = 1.0925484305920791f;    // sqrt(15 / (4 pi))
constexpr float kY2b = 0.31539156525252001f;   // sqrt(5 / (16 pi))
constexpr float kY2c = 0.54627421529603954f;   // sqrt(15 / (16 pi))
constexpr float kY3a = 0.59004358992664351f;   // sqrt(70 / (64 pi))
constexpr float kY3b = 2.8906114426405541f;    // sqrt(105 / (4 pi))
constexpr float kY3c = 0.45704579946446574f;   // sqrt(42 / (64 pi))
constexpr float kY3d = 0.37317633259011539f;   // sqrt(7 / (16 pi))
constexpr float kY3e = 1.445305721320277f;     // sqrt(105 / (16 pi))

template <int DEG>
__device__ __forceinline__ void sh_basis(float x, float y, float z, float* Y) {
    Y[0] = kY00;
    if (DEG >= 1) {
        Y[1] = -kY1 * y;
        Y[2] = kY1 * z;
        Y[3] = -kY1 * x;
    }
    if (DEG >= 2) {
        const float xx = x * x, yy = y * y, zz = z * z;
        Y[4] = kY2a * x * y;
        Y[5] = -kY2a * y * z;
        Y[6] = kY2b * (3.0f * zz - 1.0f);
        Y[7] = -kY2a * x * z;
        Y[8] = kY2c * (xx - yy);
        if (DEG >= 3) {
            Y[9] = -kY3a * y * (3.0f * xx - yy);
            Y[10] = kY3b * x * y * z;
            Y[11] = -kY3c * y * (5.0f * zz - 1.0f);
            Y[12] = kY3d * z * (5.0f * zz - 3.0f);
            Y[13] = -kY3c * x * (5.0f * zz - 1.0f);
            Y[14] = kY3e * z * (xx - yy);
            Y[15] = -kY3a * x * (xx - 3.0f * yy);
        }
    }
}

// Accumulates sum_k w[k] grad Y_k(x, y, z) (gradient of the polynomial forms above in R^3) into g.
template <int DEG>
__device__ __forceinline__ void sh_basis_grad(float x, float y, float z, const float* w, float* g) {
    float gx = 0.f, gy = 0.f, gz = 0.f;
    if (DEG >= 1) {
        gy -= kY1 * w[1];
        gz += kY1 * w[2];
        gx -= kY1 * w[3];
    }
    if (DEG >= 2) {
        gx += kY2a * y * w[4];
        gy += kY2a * x * w[4];
        gy -= kY2a * z * w[5];
        gz -= kY2a * y * w[5];
        gz += 6.0f * kY2b * z * w[6];
        gx -= kY2a * z * w[7];
        gz -= kY2a * x * w[7];
        gx += 2.0f * kY2c * x * w[8];
        gy -= 2.0f * kY2c * y * w[8];
        if (DEG >= 3) {
            const float xx = x * x, yy = y * y, zz = z * z;
            gx -= 6.0f * kY3a * x * y * w[9];
            gy -= 3.0f * kY3a * (xx - yy) * w[9];
            gx += kY3b * y * z * w[10];
            gy += kY3b * x * z * w[10];
            gz += kY3b * x * y * w[10];
            gy -= kY3c * (5.0f * zz - 1.0f) * w[11];
            gz -= 10.0f * kY3c * y * z * w[11];
            gz += kY3d * (15.0f * zz - 3.0f) * w[12];
            gx -= kY3c * (5.0f * zz - 1.0f) * w[13];
            gz -= 10.0f * kY3c * x * z * w[13];
            gx += 2.0f * kY3e * x * z * w[14];
            gy -= 2.0f * kY3e * y * z * w[14];
            gz += kY3e * (xx - yy) * w[14];
            gx -= 3.0f * kY3a * (xx - yy) * w[15];
            gy += 6.0f * kY3a * x * y * w[15];
        }
    }
    g[0] += gx;
    g[1] += gy;
    g[2] += gz;
}

}  // namespace gs
