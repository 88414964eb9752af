// Pulsar-style sphere renderer: plain, slow CPU ORACLE.
//
// TEST INFRASTRUCTURE ONLY.  Nothing in the product imports, links or calls
// this file; only the tests, the smoke check and the CPU-baseline leg of the
// benchmark do.  It shares no code, header, table or constant generator with
// the CUDA path: both are written independently from the same definition.
//
// What it computes (Pulsar: Efficient Sphere-based Neural Rendering, the
// paperlayer.ai summary of arXiv 2004.07484):
//   * scene = spheres with position, radius, opacity and a feature payload
//     (Sec. 3.1); camera = rotation R, translation t, intrinsics K (Sec. 3.2,
//     App. A "Prelude");
//   * per pixel ray, the blend of every sphere the ray hits, with opacity in
//     BOTH the depth factor and the distance factor and a background term,
//     commutative in sphere order (Sec. 3.2; App. A): the plain definition,
//     no early stop;
//   * the geometric terms are the normalised device depth and the orthogonal
//     ray-to-sphere distance (App. A);
//   * every sphere touches at least one pixel (Sec. B.1.1);
//   * candidate order = earliest possible intersection (Sec. 3.2, B.1.1) and
//     only the first n_track hits of a pixel receive gradients (Sec. 2,
//     B.1.3, B.1.4);
//   * spheres projecting to at most ~3 px get no position/radius gradient
//     (Sec. 6; App. A);
//   * exact analytic gradients of L = sum_pixels <G, F> w.r.t. position,
//     radius, opacity, features and camera R, t, K (Sec. 3.2; B.2).
//
// The pages print no formula, so the following readings are used:
//   z~  = (zfar - c.z)/(zfar - znear)              normalised device depth
//   rho = |c - (c.q^) q^|, q = (a, b, 1)           orthogonal ray distance
//   d   = 1 - rho / r_eff                          distance factor
//   w   = o * d * exp(o * z~ / gamma)              sphere weight
//   w_bg= exp(eps / gamma)                         background weight
//   F   = (sum w f + w_bg f_bg) / (sum w + w_bg)
// evaluated with every exponent shifted by m = max(eps, max_hits o*z~);
// r_eff = max(r, kappa * c.z / min(fx, fy)); key = c.z - r_eff.
//
// Orthographic camera (Sec. B.1.1 bounds sphere projections for orthogonal
// as well as pinhole cameras; the model is not printed, so this reading):
// pixel (x, y) is the ray from (X, Y, 0) along +z in camera space, with
// X = (x + 1/2 - cx)/fx, Y = (y + 1/2 - cy)/fy (fx, fy in pixels per world
// unit); rho = |(c.x - X, c.y - Y)|; r_eff = max(r, kappa / min(fx, fy));
// the pixel rectangle is [ceil(cx + fx (c.x - r_eff) - 1/2),
// floor(cx + fx (c.x + r_eff) - 1/2)] (and likewise in y); the cull, key,
// z~, weights and tracked set are the pinhole's; the cutoff area is
// pi (min(fx, fy) r)^2.
//
// Gaussian footprint (the splat variant named by the NuRec pages, whose kernel
// is not printed; reading): the distance factor becomes an isotropic
// Gaussian of sigma = r_eff / 3 over the same support rho < r_eff, shifted
// and scaled to be 1 at the centre and 0 at the rim (so the image stays
// continuous):  d = (exp(-9 rho^2 / (2 r_eff^2)) - e^-4.5) / (1 - e^-4.5).
// Decisions (support, lists, order) are the sphere renderer's unchanged.
//
// Normalised gradients (Sec. B.2: sphere gradients averaged over the
// contributing pixels, camera gradients normalised by the projected sphere
// area and 1e-3; not a gradient of anything, so PARITY UNPINNED -- only the
// CUDA path is checked against it): with n_j the number of pixels whose
// tracked set holds sphere j, its position, radius, opacity and feature
// gradients are divided by n_j; its share of the R, t and K gradients is
// multiplied by 1e-3 / A_j, A_j = pi (f_min r_eff / c.z)^2 (orthographic:
// pi (f_min r_eff)^2), the area in px^2 of the disc it is rendered with.
//
// Decisions (cull, pixel rectangle, tile lists, hit set, tracked ids) are
// taken in fp32 by a fixed sequence of correctly rounded operations (this
// file is built with -ffp-contract=off), so the GPU can match them bit for
// bit.  `fp64_decisions` switches every decision to fp64 instead (used for
// finite-difference and closed-form checks).  All values (weights, image,
// normaliser, gradients) are fp64.
#include <algorithm>
#include <cmath>
#include <cstdint>
#include <cstring>
#include <vector>
#ifdef _OPENMP
#include <omp.h>
#endif

extern "C" {

// All inputs are fp64.  The fp32 decision path rounds them to float first
// (exact for inputs that were float32 to begin with).
typedef struct {
    double R[9];
    double t[3];
    double fx, fy, cx, cy, znear, zfar;
    int32_t width, height;
    int32_t orthographic;    // 0: pinhole, 1: orthographic
} ocam_t;

typedef struct {
    double gamma, bg_eps, kappa, geom_min_area;
    int32_t n_track, channels;
    int32_t geom_cutoff;     // 1: drop position/radius/camera grads of small spheres
    int32_t fp64_decisions;  // 1: all decisions in fp64 instead of the fp32 sequence
    int32_t normalize;       // 1: normalised gradients (Sec. B.2; see below)
    int32_t gaussian;        // 1: Gaussian footprint instead of the linear one (see below)
} oparams_t;

}  // extern "C"

namespace {

const float kPiF = 3.14159265358979f;
const int kTile = 16;

// ---------------------------------------------------------------- fp32 ----
// Error-free transformations (Ogita, Rump, Oishi, "Accurate sum and dot
// product", SIAM J. Sci. Comput. 2005): TwoProduct via fused multiply-add,
// Knuth's TwoSum, Dekker's FastTwoSum.
struct F2 { float hi, lo; };

F2 two_prod(float a, float b) {
    float p = a * b;
    float e = std::fma(a, b, -p);
    return {p, e};
}
F2 two_sum(float a, float b) {
    float s = a + b;
    float bp = s - a;
    float e = (a - (s - bp)) + (b - bp);
    return {s, e};
}
F2 fast_two_sum(float a, float b) {
    float s = a + b;
    float e = b - (s - a);
    return {s, e};
}

// One row of c = R p + t as an unevaluated pair hi + lo.
F2 cam_row32(const float* Rr, float t, const float* p) {
    F2 a = two_prod(Rr[0], p[0]);
    F2 b = two_prod(Rr[1], p[1]);
    F2 s = two_sum(a.hi, b.hi);
    float e = (a.lo + b.lo) + s.lo;
    F2 c = two_prod(Rr[2], p[2]);
    F2 s2 = two_sum(s.hi, c.hi);
    e = (e + c.lo) + s2.lo;
    F2 s3 = two_sum(s2.hi, t);
    e = e + s3.lo;
    return two_sum(s3.hi, e);
}

// (x.hi + x.lo) / (z.hi + z.lo) as a pair.
F2 pair_div32(F2 x, F2 z) {
    float q1 = x.hi / z.hi;
    float r = std::fma(-q1, z.hi, x.hi);
    r = r + x.lo;
    r = std::fma(-q1, z.lo, r);
    float q2 = r / z.hi;
    return fast_two_sum(q1, q2);
}

// c0 + f * q as a pair (projected centre in pixels).
F2 project32(float f, float c0, F2 q) {
    F2 p = two_prod(f, q.hi);
    float pl = std::fma(f, q.lo, p.lo);
    F2 s = two_sum(c0, p.hi);
    float e = s.lo + pl;
    return two_sum(s.hi, e);
}

// Orthographic camera: pixel range [ceil(u - f r - 1/2), floor(u + f r - 1/2)]
// of a sphere with centre coordinate X along the axis and radius Rr, clamped
// to the image (u = c0 + f X).
template <typename T>
void ortho_range(T X, T Rr, T f, T c0, int n, int* lo, int* hi) {
    T umin = c0 + f * (X - Rr);
    T umax = c0 + f * (X + Rr);
    T a = std::ceil(umin - T(0.5));
    T b = std::floor(umax - T(0.5));
    T af = a < T(0) ? T(0) : a;
    T bf = b > T(n - 1) ? T(n - 1) : b;
    if (!(af <= bf)) { *lo = 1; *hi = 0; return; }
    *lo = (int)af;
    *hi = (int)bf;
}

// Pixel range along one image axis covered by the tangent cone of a sphere
// (centre X along the axis, depth Z, radius Rr): the two tangent directions
// from the camera in the (axis, z) plane, written without trigonometry
// (Sec. B.1.1 "trigonometric functions can be avoided through identities").
template <typename T>
void axis_range(T X, T Z, T Rr, T f, T c0, int n, int* lo, int* hi) {
    T L2 = (X * X + Z * Z) - Rr * Rr;
    T L = std::sqrt(L2);
    T dmax = Z * L - X * Rr;
    T dmin = Z * L + X * Rr;
    T umax = dmax > T(0) ? c0 + f * ((X * L + Rr * Z) / dmax) : T(INFINITY);
    T umin = dmin > T(0) ? c0 + f * ((X * L - Rr * Z) / dmin) : T(-INFINITY);
    T a = std::ceil(umin - T(0.5));
    T b = std::floor(umax - T(0.5));
    T af = a < T(0) ? T(0) : a;
    T bf = b > T(n - 1) ? T(n - 1) : b;
    if (!(af <= bf)) { *lo = 1; *hi = 0; return; }
    *lo = (int)af;
    *hi = (int)bf;
}

// ---------------------------------------------------------------- sphere --
struct Sphere {
    // decision quantities
    int keep = 0;
    int x0 = 1, x1 = 0, y0 = 1, y1 = 0;
    int floor_r = 0;     // r_eff took the kappa floor
    int cut = 0;         // geometry gradients dropped
    float u_hi = 0, u_lo = 0, v_hi = 0, v_lo = 0, reff32 = 0, key32 = 0, s2_32 = 0;
    double key64 = 0, s2_64 = 0, u64 = 0, v64 = 0;
    // value-path quantities (fp64, exact camera transform)
    double c[3] = {0, 0, 0};
    double u = 0, v = 0, reff = 0, zt = 0, o = 0;
};

// The camera as float32 values, for the fp32 decision sequence.
struct Cam32 {
    float R[9], t[3], fx, fy, cx, cy, znear, zfar, kappa, amin;
    int ortho;
};
Cam32 cam32(const ocam_t& cam, const oparams_t& prm) {
    Cam32 c;
    for (int k = 0; k < 9; ++k) c.R[k] = (float)cam.R[k];
    for (int k = 0; k < 3; ++k) c.t[k] = (float)cam.t[k];
    c.fx = (float)cam.fx; c.fy = (float)cam.fy; c.cx = (float)cam.cx; c.cy = (float)cam.cy;
    c.znear = (float)cam.znear; c.zfar = (float)cam.zfar;
    c.kappa = (float)prm.kappa; c.amin = (float)prm.geom_min_area;
    c.ortho = cam.orthographic != 0;
    return c;
}

void camera_center64(const ocam_t& cam, const double* p, double* c) {
    for (int k = 0; k < 3; ++k)
        c[k] = ((cam.R[3 * k] * p[0] + cam.R[3 * k + 1] * p[1]) + cam.R[3 * k + 2] * p[2]) +
               cam.t[k];
}

Sphere decide(const double* pd, double rd, double o, const ocam_t& cam, const Cam32& c32,
              const oparams_t& prm) {
    Sphere s;
    camera_center64(cam, pd, s.c);
    s.o = o;
    const double fmin64 = cam.fx <= cam.fy ? cam.fx : cam.fy;
    if (!prm.fp64_decisions) {
        const float p[3] = {(float)pd[0], (float)pd[1], (float)pd[2]};
        const float r = (float)rd;
        F2 cx = cam_row32(c32.R + 0, c32.t[0], p);
        F2 cy = cam_row32(c32.R + 3, c32.t[1], p);
        F2 cz = cam_row32(c32.R + 6, c32.t[2], p);
        float Z = cz.hi;
        float fmin = c32.fx <= c32.fy ? c32.fx : c32.fy;
        float rf = c32.ortho ? c32.kappa / fmin : (c32.kappa * Z) / fmin;
        s.floor_r = r < rf;
        float reff = s.floor_r ? rf : r;
        s.keep = Z > c32.znear && Z < c32.zfar && reff < Z;
        if (!s.keep) return s;
        F2 u = project32(c32.fx, c32.cx, c32.ortho ? cx : pair_div32(cx, cz));
        F2 v = project32(c32.fy, c32.cy, c32.ortho ? cy : pair_div32(cy, cz));
        s.u_hi = u.hi; s.u_lo = u.lo; s.v_hi = v.hi; s.v_lo = v.lo;
        if (c32.ortho) {
            ortho_range<float>(cx.hi, reff, c32.fx, c32.cx, cam.width, &s.x0, &s.x1);
            ortho_range<float>(cy.hi, reff, c32.fy, c32.cy, cam.height, &s.y0, &s.y1);
        } else {
            axis_range<float>(cx.hi, Z, reff, c32.fx, c32.cx, cam.width, &s.x0, &s.x1);
            axis_range<float>(cy.hi, Z, reff, c32.fy, c32.cy, cam.height, &s.y0, &s.y1);
        }
        s.keep = s.x0 <= s.x1 && s.y0 <= s.y1;
        s.reff32 = reff;
        s.key32 = Z - reff;
        float tt = c32.ortho ? reff : reff / Z;
        s.s2_32 = tt * tt;
        float g = c32.ortho ? fmin * r : (fmin * r) / Z;
        float area = kPiF * (g * g);
        s.cut = prm.geom_cutoff && !(area > c32.amin);
    } else {
        const double r = rd;
        const bool ortho = cam.orthographic != 0;
        double Z = s.c[2];
        double rf = ortho ? (double)prm.kappa / fmin64 : (double)prm.kappa * Z / fmin64;
        s.floor_r = r < rf;
        double reff = s.floor_r ? rf : (double)r;
        s.keep = Z > cam.znear && Z < cam.zfar && reff < Z;
        if (!s.keep) return s;
        if (ortho) {
            s.u64 = cam.cx + (double)cam.fx * s.c[0];
            s.v64 = cam.cy + (double)cam.fy * s.c[1];
            ortho_range<double>(s.c[0], reff, cam.fx, cam.cx, cam.width, &s.x0, &s.x1);
            ortho_range<double>(s.c[1], reff, cam.fy, cam.cy, cam.height, &s.y0, &s.y1);
        } else {
            s.u64 = cam.cx + (double)cam.fx * (s.c[0] / Z);
            s.v64 = cam.cy + (double)cam.fy * (s.c[1] / Z);
            axis_range<double>(s.c[0], Z, reff, cam.fx, cam.cx, cam.width, &s.x0, &s.x1);
            axis_range<double>(s.c[1], Z, reff, cam.fy, cam.cy, cam.height, &s.y0, &s.y1);
        }
        s.keep = s.x0 <= s.x1 && s.y0 <= s.y1;
        s.key64 = Z - reff;
        s.s2_64 = ortho ? reff * reff : (reff / Z) * (reff / Z);
        double g = ortho ? fmin64 * r : fmin64 * r / Z;
        s.cut = prm.geom_cutoff && !(M_PI * g * g > prm.geom_min_area);
    }
    // value path: exact geometry, branch of r_eff taken by the decision above
    const double Z = s.c[2];
    if (cam.orthographic) {
        s.u = cam.cx + (double)cam.fx * s.c[0];
        s.v = cam.cy + (double)cam.fy * s.c[1];
        s.reff = s.floor_r ? prm.kappa / fmin64 : rd;
    } else {
        s.u = cam.cx + (double)cam.fx * (s.c[0] / Z);
        s.v = cam.cy + (double)cam.fy * (s.c[1] / Z);
        s.reff = s.floor_r ? prm.kappa * Z / fmin64 : rd;
    }
    s.zt = ((double)cam.zfar - Z) / ((double)cam.zfar - (double)cam.znear);
    return s;
}

// Per-pixel ray constants: direction q = (a, b, 1) and origin (ox, oy, 0);
// pinhole: a = (px - cx)/fx, b = (py - cy)/fy, origin 0; orthographic: a = b
// = 0, ox = (px - cx)/fx, oy = (py - cy)/fy.
struct Pix32 { float px, py, a, b, qq; };
struct Pix64 { double px, py, a, b, qq, ox, oy; };

Pix32 pix32(int x, int y, const Cam32& cam) {
    Pix32 q;
    q.px = (float)x + 0.5f;
    q.py = (float)y + 0.5f;
    q.a = cam.ortho ? 0.0f : (q.px - cam.cx) / cam.fx;
    q.b = cam.ortho ? 0.0f : (q.py - cam.cy) / cam.fy;
    q.qq = (1.0f + q.a * q.a) + q.b * q.b;
    return q;
}
Pix64 pix64(int x, int y, const ocam_t& cam) {
    Pix64 q;
    q.px = x + 0.5;
    q.py = y + 0.5;
    const double sa = (q.px - cam.cx) / cam.fx, sb = (q.py - cam.cy) / cam.fy;
    q.a = cam.orthographic ? 0.0 : sa;
    q.b = cam.orthographic ? 0.0 : sb;
    q.ox = cam.orthographic ? sa : 0.0;
    q.oy = cam.orthographic ? sb : 0.0;
    q.qq = 1.0 + q.a * q.a + q.b * q.b;
    return q;
}

// The hit test: pixel inside the sphere's pixel rectangle and the ray's
// squared orthogonal distance (scaled by 1/c.z^2 and |q|^2) below r_eff^2.
bool hit_test(const Sphere& s, int x, int y, const Pix32& p32, const Pix64& p64,
              float ifx, float ify, const ocam_t& cam, bool fp64) {
    if (x < s.x0 || x > s.x1 || y < s.y0 || y > s.y1) return false;
    if (!fp64) {
        float du = (p32.px - s.u_hi) - s.u_lo;
        float dv = (p32.py - s.v_hi) - s.v_lo;
        float U = du * ifx;
        float V = dv * ify;
        float X = std::fma(U, p32.b, -(V * p32.a));
        float Q = std::fma(U, U, std::fma(V, V, X * X));
        return Q < s.s2_32 * p32.qq;
    }
    double U = (p64.px - s.u64) / cam.fx;
    double V = (p64.py - s.v64) / cam.fy;
    double X = U * p64.b - V * p64.a;
    double Q = U * U + V * V + X * X;
    return Q < s.s2_64 * p64.qq;
}

// fp64 geometry of sphere s at pixel p: returns Q and sets U, V.
// Pinhole: rho = c.z sqrt(Q / qq); orthographic (a = b = 0, U = X - c.x,
// V = Y - c.y): rho = sqrt(Q).
double value_Q(const Sphere& s, const Pix64& p, const ocam_t& cam, double* U, double* V) {
    *U = (p.px - s.u) / cam.fx;
    *V = (p.py - s.v) / cam.fy;
    double X = *U * p.b - *V * p.a;
    return *U * *U + *V * *V + X * X;
}

double ray_rho(const Sphere& s, double Q, double qq, const ocam_t& cam) {
    return cam.orthographic ? std::sqrt(Q) : std::sqrt(Q / qq) * s.c[2];
}

// distance factor d(rho / r_eff): linear 1 - x, or the Gaussian footprint
const double kGaussTail = std::exp(-4.5);
double footprint(double x, bool gaussian) {
    return gaussian ? (std::exp(-4.5 * x * x) - kGaussTail) / (1.0 - kGaussTail) : 1.0 - x;
}
// its derivative with respect to x = rho / r_eff
double footprint_dx(double x, bool gaussian) {
    return gaussian ? -9.0 * x * std::exp(-4.5 * x * x) / (1.0 - kGaussTail) : -1.0;
}
double dist_factor(const Sphere& s, double Q, double qq, const ocam_t& cam, bool gaussian) {
    return footprint(ray_rho(s, Q, qq, cam) / s.reff, gaussian);
}

struct HitKey {
    double key;
    int32_t id;
};

int num_threads() {
#ifdef _OPENMP
    return omp_get_max_threads();
#else
    return 1;
#endif
}

}  // namespace

extern "C" {

int oracle_num_threads() { return num_threads(); }

// Threads of the following calls (n <= 0: all of the host's); timing only.
void oracle_set_threads(int n) {
#ifdef _OPENMP
    omp_set_num_threads(n > 0 ? n : omp_get_num_procs());
#else
    (void)n;
#endif
}

// Per-sphere decision outputs (fp32 decision path) for bit-exact comparison.
int oracle_project(const double* pos, const double* radius, const double* opacity, int64_t n,
                   const ocam_t* cam, const oparams_t* prm, int32_t* keep, float* uv4,
                   float* reff, float* key, float* s2, int32_t* rect4, int32_t* floor_r,
                   int32_t* cut, int32_t* ntiles) {
    if (n < 0 || !cam || !prm) return -1;
    const Cam32 c32 = cam32(*cam, *prm);
#pragma omp parallel for schedule(static)
    for (int64_t i = 0; i < n; ++i) {
        Sphere s = decide(pos + 3 * i, radius[i], opacity[i], *cam, c32, *prm);
        keep[i] = s.keep;
        uv4[4 * i + 0] = s.u_hi; uv4[4 * i + 1] = s.u_lo;
        uv4[4 * i + 2] = s.v_hi; uv4[4 * i + 3] = s.v_lo;
        reff[i] = s.reff32;
        key[i] = s.key32;
        s2[i] = s.s2_32;
        rect4[4 * i + 0] = s.x0; rect4[4 * i + 1] = s.x1;
        rect4[4 * i + 2] = s.y0; rect4[4 * i + 3] = s.y1;
        floor_r[i] = s.floor_r;
        cut[i] = s.cut;
        ntiles[i] = s.keep ? (s.x1 / kTile - s.x0 / kTile + 1) * (s.y1 / kTile - s.y0 / kTile + 1) : 0;
    }
    return 0;
}

// Tile lists: for each 16x16 tile (row-major over the image), the ids of the
// kept spheres whose pixel rectangle meets the tile, in ascending
// (key, id) order -- the order of earliest possible intersection.
// Returns the number of pairs M, or -M-1 if it exceeds cap (nothing written
// to ids beyond cap).
int64_t oracle_tile_lists(const double* pos, const double* radius, const double* opacity, int64_t n,
                          const ocam_t* cam, const oparams_t* prm, int64_t* offsets,
                          int32_t* ids, int64_t cap) {
    const int tx = (cam->width + kTile - 1) / kTile, ty = (cam->height + kTile - 1) / kTile;
    const int64_t B = (int64_t)tx * ty;
    const Cam32 c32 = cam32(*cam, *prm);
    std::vector<Sphere> sph(n);
#pragma omp parallel for schedule(static)
    for (int64_t i = 0; i < n; ++i)
        sph[i] = decide(pos + 3 * i, radius[i], opacity[i], *cam, c32, *prm);
    std::vector<std::vector<HitKey>> lists(B);
    for (int64_t i = 0; i < n; ++i) {
        const Sphere& s = sph[i];
        if (!s.keep) continue;
        double k = prm->fp64_decisions ? s.key64 : (double)s.key32;
        for (int y = s.y0 / kTile; y <= s.y1 / kTile; ++y)
            for (int x = s.x0 / kTile; x <= s.x1 / kTile; ++x)
                lists[(int64_t)y * tx + x].push_back({k, (int32_t)i});
    }
    int64_t m = 0;
    for (int64_t b = 0; b < B; ++b) {
        std::sort(lists[b].begin(), lists[b].end(), [](const HitKey& p, const HitKey& q) {
            return p.key < q.key || (p.key == q.key && p.id < q.id);
        });
        offsets[b] = m;
        for (const HitKey& h : lists[b]) {
            if (m < cap) ids[m] = h.id;
            ++m;
        }
    }
    offsets[B] = m;
    return m <= cap ? m : -m - 1;
}

// Render the pixel window [wx0, wx1) x [wy0, wy1) and, if grad_image is
// given, the gradients of L = sum over window pixels of <G, F>.
//   brute = 1: every kept sphere is tested at every pixel;
//   brute = 0: only spheres whose rectangle meets the pixel's 16x16 tile.
// Outputs (window-sized, row-major): image [h,w,C], mg [h,w] (= m/gamma),
// wsum [h,w] (normaliser in the m-shifted frame), ids [h,w,T] (-1 padded),
// nhits [h,w].  Gradients (full size, overwritten; any may be NULL):
// grad_pos [n,3], grad_radius [n], grad_opacity [n], grad_features [n,C],
// grad_cam [16] = dL/dR (9, row-major), dL/dt (3), dL/d(fx, fy, cx, cy).
// gabs (optional) [2 ((5 + C) n + 16)]: for every gradient entry, in the
// order pos, radius, opacity, features, cam, (1) the sum over pixels of the
// absolute value of that pixel's contribution, then (2) the sum over pixels of
// sum_c |d contribution / d F_c|, its sensitivity to the image F that the
// backward takes as input (zero for the feature gradients).
// Returns the number of hit pairs in the window, or a negative error.
int64_t oracle_render(const double* pos, const double* radius, const double* opacity,
                      const double* features, int64_t n, const ocam_t* cam_p,
                      const oparams_t* prm_p, const double* bg, int32_t wx0, int32_t wy0,
                      int32_t wx1, int32_t wy1, int32_t brute, const double* grad_image,
                      double* image, double* mg, double* wsum, int32_t* ids, int32_t* nhits,
                      double* grad_pos, double* grad_radius, double* grad_opacity,
                      double* grad_features, double* grad_cam, double* gabs) {
    if (!cam_p || !prm_p || n < 0) return -1;
    const ocam_t cam = *cam_p;
    const oparams_t prm = *prm_p;
    const int C = prm.channels, T = prm.n_track;
    if (C < 1 || T < 1 || wx0 < 0 || wy0 < 0 || wx1 > cam.width || wy1 > cam.height ||
        wx0 > wx1 || wy0 > wy1)
        return -2;
    const bool fp64 = prm.fp64_decisions != 0;
    const double gamma = prm.gamma, eps = prm.bg_eps;
    const int ww = wx1 - wx0, wh = wy1 - wy0;
    const int64_t P = (int64_t)ww * wh;
    const Cam32 c32 = cam32(cam, prm);
    const float ifx = 1.0f / c32.fx, ify = 1.0f / c32.fy;

    std::vector<Sphere> sph(n);
#pragma omp parallel for schedule(static)
    for (int64_t i = 0; i < n; ++i)
        sph[i] = decide(pos + 3 * i, radius[i], opacity[i], cam, c32, prm);

    // candidate buckets per 16x16 tile (ascending id); brute mode uses all kept spheres
    const int tx = (cam.width + kTile - 1) / kTile, ty = (cam.height + kTile - 1) / kTile;
    std::vector<std::vector<int32_t>> bucket(brute ? 1 : (int64_t)tx * ty);
    for (int64_t i = 0; i < n; ++i) {
        const Sphere& s = sph[i];
        if (!s.keep) continue;
        if (brute) { bucket[0].push_back((int32_t)i); continue; }
        for (int y = s.y0 / kTile; y <= s.y1 / kTile; ++y)
            for (int x = s.x0 / kTile; x <= s.x1 / kTile; ++x)
                bucket[(int64_t)y * tx + x].push_back((int32_t)i);
    }

    // ---- forward: per pixel, all hits in (key, id) order, plain blend -----
    std::vector<double> F((size_t)P * C), Wn(P), M(P);
    std::vector<int32_t> trk((size_t)P * T, -1);
    std::vector<int32_t> nh(P, 0);
    int64_t total_hits = 0;
#pragma omp parallel for schedule(dynamic, 1) reduction(+ : total_hits)
    for (int yy = 0; yy < wh; ++yy) {
        std::vector<HitKey> hits;
        std::vector<double> acc(C);
        for (int xx = 0; xx < ww; ++xx) {
            const int x = wx0 + xx, y = wy0 + yy;
            const int64_t pi = (int64_t)yy * ww + xx;
            const Pix32 p32 = pix32(x, y, c32);
            const Pix64 p64 = pix64(x, y, cam);
            const std::vector<int32_t>& cand =
                brute ? bucket[0] : bucket[(int64_t)(y / kTile) * tx + x / kTile];
            hits.clear();
            for (int32_t id : cand) {
                const Sphere& s = sph[id];
                if (hit_test(s, x, y, p32, p64, ifx, ify, cam, fp64))
                    hits.push_back({fp64 ? s.key64 : (double)s.key32, id});
            }
            std::sort(hits.begin(), hits.end(), [](const HitKey& p, const HitKey& q) {
                return p.key < q.key || (p.key == q.key && p.id < q.id);
            });
            nh[pi] = (int32_t)hits.size();
            total_hits += (int64_t)hits.size();
            for (int k = 0; k < T && k < (int)hits.size(); ++k) trk[(size_t)pi * T + k] = hits[k].id;
            double m = eps;
            for (const HitKey& h : hits) m = std::max(m, sph[h.id].o * sph[h.id].zt);
            double W = std::exp((eps - m) / gamma);
            for (int c = 0; c < C; ++c) acc[c] = W * bg[c];
            for (const HitKey& h : hits) {
                const Sphere& s = sph[h.id];
                double U, V;
                double Q = value_Q(s, p64, cam, &U, &V);
                double d = dist_factor(s, Q, p64.qq, cam, prm.gaussian != 0);
                double w = s.o * d * std::exp((s.o * s.zt - m) / gamma);
                W += w;
                for (int c = 0; c < C; ++c) acc[c] += w * features[(size_t)h.id * C + c];
            }
            for (int c = 0; c < C; ++c) F[(size_t)pi * C + c] = acc[c] / W;
            Wn[pi] = W;
            M[pi] = m;
        }
    }
    if (image) std::memcpy(image, F.data(), sizeof(double) * F.size());
    if (mg) for (int64_t i = 0; i < P; ++i) mg[i] = M[i] / gamma;
    if (wsum) std::memcpy(wsum, Wn.data(), sizeof(double) * P);
    if (ids) std::memcpy(ids, trk.data(), sizeof(int32_t) * trk.size());
    if (nhits) std::memcpy(nhits, nh.data(), sizeof(int32_t) * P);
    if (!grad_image) return total_hits;

    // ---- backward: gradients through the first T hits of every pixel -----
    // Invert the tracked lists: for every sphere, the window pixels (ascending)
    // that track it, so each sphere's gradient is a fixed-order sum.
    std::vector<int64_t> cnt(n + 1, 0);
    for (int64_t pi = 0; pi < P; ++pi)
        for (int k = 0; k < T; ++k) {
            int32_t id = trk[(size_t)pi * T + k];
            if (id >= 0) cnt[id + 1]++;
        }
    for (int64_t i = 0; i < n; ++i) cnt[i + 1] += cnt[i];
    std::vector<int64_t> fill(cnt.begin(), cnt.end() - 1);
    std::vector<int64_t> plist(cnt[n]);
    for (int64_t pi = 0; pi < P; ++pi)
        for (int k = 0; k < T; ++k) {
            int32_t id = trk[(size_t)pi * T + k];
            if (id >= 0) plist[fill[id]++] = pi;
        }

    const double fmin = cam.fx <= cam.fy ? cam.fx : cam.fy;
    const bool fmin_is_fx = cam.fx <= cam.fy;
    const double dzt_dz = -1.0 / ((double)cam.zfar - (double)cam.znear);
    std::vector<double> gc((size_t)n * 3, 0.0), gk((size_t)n * 4, 0.0);
    // optional: per gradient entry, the sum over pixels of the absolute
    // contributions (the scale of the rounding error of any summation order)
    std::vector<double> ac(gabs ? (size_t)n * 3 : 0), ak(gabs ? (size_t)n * 4 : 0);
    std::vector<double> acr(gabs ? (size_t)n * 9 : 0);
    std::vector<double> sc_(gabs ? (size_t)n * 3 : 0), sk(gabs ? (size_t)n * 4 : 0);
    std::vector<double> scr(gabs ? (size_t)n * 9 : 0);
#pragma omp parallel for schedule(dynamic, 256)
    for (int64_t i = 0; i < n; ++i) {
        const Sphere& s = sph[i];
        double g_c[3] = {0, 0, 0}, g_r = 0, g_o = 0, g_K[4] = {0, 0, 0, 0};
        double a_c[3] = {0, 0, 0}, a_r = 0, a_o = 0, a_K[4] = {0, 0, 0, 0}, a_p[3] = {0, 0, 0};
        double a_R[9] = {0};
        double s_c[3] = {0, 0, 0}, s_r = 0, s_o = 0, s_K[4] = {0, 0, 0, 0}, s_p[3] = {0, 0, 0};
        double s_R[9] = {0};
        std::vector<double> g_f(C, 0.0), a_f(C, 0.0);
        for (int64_t e = cnt[i]; e < cnt[i + 1]; ++e) {
            const int64_t pi = plist[e];
            const int x = wx0 + (int)(pi % ww), y = wy0 + (int)(pi / ww);
            const Pix64 p = pix64(x, y, cam);
            const double* Fp = &F[(size_t)pi * C];
            const double* G = grad_image + ((size_t)y * cam.width + x) * C;
            const double W = Wn[pi], m = M[pi];
            double U, V;
            const double Q = value_Q(s, p, cam, &U, &V);
            const bool ortho = cam.orthographic != 0;
            const double rho = ray_rho(s, Q, p.qq, cam);
            const double rq = ortho ? rho : std::sqrt(Q / p.qq);   // rho (orthographic), rho / c.z
            const bool gauss = prm.gaussian != 0;
            const double d = footprint(rho / s.reff, gauss);
            const double E = std::exp((s.o * s.zt - m) / gamma);
            const double w = s.o * d * E;
            double sdot = 0.0;                                 // <G, f - F>
            for (int c = 0; c < C; ++c)
                sdot += G[c] * (features[(size_t)i * C + c] - Fp[c]);
            const double sj = sdot / W;                        // dL/dw
            // This pixel's contributions, except to the features, are sj times
            // a factor; the factors ("per unit sj") are formed first, so that
            // the sensitivity of each contribution to the image F
            // (d sj / dF_c = -G_c / W) is available as well.
            double uc[3] = {0, 0, 0}, ur = 0, uk[4] = {0, 0, 0, 0};
            double gl1 = 0.0;
            for (int c = 0; c < C; ++c) {
                g_f[c] += (w / W) * G[c];
                if (gabs) a_f[c] += std::fabs((w / W) * G[c]);
                gl1 += std::fabs(G[c]);
            }
            const double sens = gl1 / W;                      // sum_c |d sj / dF_c|
            const double uo = d * E * (1.0 + s.o * s.zt / gamma);   // dw/do
            g_o += sj * uo;
            if (gabs) {
                a_o += std::fabs(sj * uo);
                s_o += std::fabs(uo) * sens;
            }
            if (s.cut) continue;
            // dw/dz~ = w * o / gamma ; dz~/dc.z = -1/(zfar - znear)
            uc[2] += w * (s.o / gamma) * dzt_dz;
            // dw/dd = o E ; with x = rho / r_eff: dd/drho = d'(x) / r_eff,
            // dd/dr_eff = -d'(x) rho / r_eff^2 (linear: d' = -1)
            const double ddx = footprint_dx(rho / s.reff, gauss);
            const double u_rho = s.o * E * ddx / s.reff;
            const double u_reff = -s.o * E * ddx * rho / (s.reff * s.reff);
            if (s.floor_r) {
                if (ortho) {
                    // r_eff = kappa / f_min
                    uk[fmin_is_fx ? 0 : 1] += u_reff * (-prm.kappa / (fmin * fmin));
                } else {
                    // r_eff = kappa c.z / f_min
                    uc[2] += u_reff * prm.kappa / fmin;
                    uk[fmin_is_fx ? 0 : 1] += u_reff * (-prm.kappa * s.c[2] / (fmin * fmin));
                }
            } else {
                ur += u_reff;
            }
            if (Q > 0.0 && ortho) {
                // rho = |(c.x - X, c.y - Y)|, c.x - X = -U, c.y - Y = -V
                uc[0] += u_rho * (-U / rho);
                uc[1] += u_rho * (-V / rho);
                // drho/dX = U / rho, X = (px - cx)/fx: dX/dfx = -X/fx, dX/dcx = -1/fx
                uk[0] += u_rho * (U / rho) * (-p.ox / cam.fx);
                uk[1] += u_rho * (V / rho) * (-p.oy / cam.fy);
                uk[2] += u_rho * (U / rho) * (-1.0 / cam.fx);
                uk[3] += u_rho * (V / rho) * (-1.0 / cam.fy);
            } else if (Q > 0.0) {
                // drho/dc = e_perp / rho with e = c - c.z q = -c.z (U, V, 0)
                const double k = (U * p.a + V * p.b) / p.qq;
                const double n0 = -(U - k * p.a) / rq, n1 = -(V - k * p.b) / rq, n2 = k / rq;
                uc[0] += u_rho * n0;
                uc[1] += u_rho * n1;
                uc[2] += u_rho * n2;
                // drho/dq = -(c.q / q.q) e_perp / rho, c.q / q.q = c.z (1 - k)
                const double sq = -s.c[2] * (1.0 - k);
                const double dqa = sq * n0, dqb = sq * n1;
                // a = (px - cx)/fx, b = (py - cy)/fy
                uk[0] += u_rho * dqa * (-p.a / cam.fx);
                uk[1] += u_rho * dqb * (-p.b / cam.fy);
                uk[2] += u_rho * dqa * (-1.0 / cam.fx);
                uk[3] += u_rho * dqb * (-1.0 / cam.fy);
            }
            for (int k = 0; k < 3; ++k) g_c[k] += sj * uc[k];
            for (int k = 0; k < 4; ++k) g_K[k] += sj * uk[k];
            g_r += sj * ur;
            if (gabs) {
                for (int k = 0; k < 3; ++k) {
                    a_c[k] += std::fabs(sj * uc[k]);
                    s_c[k] += std::fabs(uc[k]) * sens;
                }
                for (int k = 0; k < 4; ++k) {
                    a_K[k] += std::fabs(sj * uk[k]);
                    s_K[k] += std::fabs(uk[k]) * sens;
                }
                a_r += std::fabs(sj * ur);
                s_r += std::fabs(ur) * sens;
                for (int l = 0; l < 3; ++l) {
                    const double up = cam.R[l] * uc[0] + cam.R[3 + l] * uc[1] + cam.R[6 + l] * uc[2];
                    a_p[l] += std::fabs(sj * up);
                    s_p[l] += std::fabs(up) * sens;
                }
                for (int k = 0; k < 3; ++k)
                    for (int l = 0; l < 3; ++l) {
                        a_R[3 * k + l] += std::fabs(sj * uc[k] * pos[3 * i + l]);
                        s_R[3 * k + l] += std::fabs(uc[k] * pos[3 * i + l]) * sens;
                    }
            }
        }
        // camera shares (R, t through g_c; K) and sphere gradients
        double cam_scale = 1.0, sph_scale = 1.0;
        if (prm.normalize && s.keep) {
            const double nj = (double)(cnt[i + 1] - cnt[i]);
            sph_scale = nj > 0 ? 1.0 / nj : 1.0;
            const double rz = cam.orthographic ? s.reff : s.reff / s.c[2];
            const double A = M_PI * (fmin * rz) * (fmin * rz);
            cam_scale = 1e-3 / A;
        }
        for (int k = 0; k < 3; ++k) gc[3 * i + k] = g_c[k] * cam_scale;
        for (int k = 0; k < 4; ++k) gk[4 * i + k] = g_K[k] * cam_scale;
        if (grad_radius) grad_radius[i] = g_r * sph_scale;
        if (grad_opacity) grad_opacity[i] = g_o * sph_scale;
        if (grad_features)
            for (int c = 0; c < C; ++c) grad_features[(size_t)i * C + c] = g_f[c] * sph_scale;
        if (grad_pos)
            for (int l = 0; l < 3; ++l)
                grad_pos[3 * i + l] =
                    (cam.R[l] * g_c[0] + cam.R[3 + l] * g_c[1] + cam.R[6 + l] * g_c[2]) * sph_scale;
        if (gabs) {
            for (int l = 0; l < 3; ++l) gabs[3 * i + l] = a_p[l] * sph_scale;
            gabs[3 * n + i] = a_r * sph_scale;
            gabs[4 * n + i] = a_o * sph_scale;
            for (int c = 0; c < C; ++c) gabs[5 * n + (size_t)i * C + c] = a_f[c] * sph_scale;
            for (int k = 0; k < 3; ++k) ac[3 * i + k] = a_c[k] * cam_scale;
            for (int k = 0; k < 4; ++k) ak[4 * i + k] = a_K[k] * cam_scale;
            for (int k = 0; k < 9; ++k) acr[9 * i + k] = a_R[k] * cam_scale;
            double* sens_out = gabs + (5 + C) * n + 16;
            for (int l = 0; l < 3; ++l) sens_out[3 * i + l] = s_p[l] * sph_scale;
            sens_out[3 * n + i] = s_r * sph_scale;
            sens_out[4 * n + i] = s_o * sph_scale;
            for (int k = 0; k < 3; ++k) sc_[3 * i + k] = s_c[k] * cam_scale;
            for (int k = 0; k < 4; ++k) sk[4 * i + k] = s_K[k] * cam_scale;
            for (int k = 0; k < 9; ++k) scr[9 * i + k] = s_R[k] * cam_scale;
        }
    }
    if (grad_cam) {
        double g[16] = {0};
        for (int64_t i = 0; i < n; ++i) {
            for (int k = 0; k < 3; ++k) {
                for (int l = 0; l < 3; ++l) g[3 * k + l] += gc[3 * i + k] * pos[3 * i + l];
                g[9 + k] += gc[3 * i + k];
            }
            for (int k = 0; k < 4; ++k) g[12 + k] += gk[4 * i + k];
        }
        std::memcpy(grad_cam, g, sizeof(g));
    }
    if (gabs) {
        double a[16] = {0};
        for (int64_t i = 0; i < n; ++i) {
            for (int k = 0; k < 9; ++k) a[k] += acr[9 * i + k];
            for (int k = 0; k < 3; ++k) a[9 + k] += ac[3 * i + k];
            for (int k = 0; k < 4; ++k) a[12 + k] += ak[4 * i + k];
        }
        std::memcpy(gabs + (5 + C) * n, a, sizeof(a));
        double sa[16] = {0};
        for (int64_t i = 0; i < n; ++i) {
            for (int k = 0; k < 9; ++k) sa[k] += scr[9 * i + k];
            for (int k = 0; k < 3; ++k) sa[9 + k] += sc_[3 * i + k];
            for (int k = 0; k < 4; ++k) sa[12 + k] += sk[4 * i + k];
        }
        double* sens_out = gabs + (5 + C) * n + 16;
        std::memcpy(sens_out + (5 + C) * n, sa, sizeof(sa));
    }
    return total_hits;
}

}  // extern "C"
