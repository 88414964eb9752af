// Internal definitions shared by the CUDA kernels of the sphere renderer.
//
// Decisions (cull, pixel rectangle, tile lists, hit set, tracked ids) are a
// fixed sequence of correctly rounded fp32 operations written with the
// explicit round-to-nearest intrinsics (__fadd_rn, __fmul_rn, __fdiv_rn,
// __fsqrt_rn, __fmaf_rn), which the compiler never contracts or reorders.
// Values (weights, image, gradients) are ordinary fp32 arithmetic.
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

namespace pulsar {

constexpr int kTile = 16;           // 16x16 pixel tiles (Pulsar Sec. B.1.2)
constexpr int kTilePix = kTile * kTile;
constexpr int kMaxTrack = 16;
constexpr int kMaxChannels = 64;
constexpr int kMaxCams = 8;         // cameras of one batched frame
constexpr int kShadeParams = 5635;  // shading MLP: W1 [64,19], b1, W2 [64,64], b2, W3 [3,64], b3
constexpr uint32_t kFlagKeep = 1u, kFlagFloor = 2u, kFlagCut = 4u;   // per-sphere record flags
constexpr uint32_t kParamNormalize = 4u;   // Frame::flags bit: normalised gradients
constexpr uint32_t kParamGaussian = 8u;    // Frame::flags bit: Gaussian footprint
// Gaussian footprint d = (exp(-4.5 x^2) - e^-4.5) / (1 - e^-4.5), x = rho / r_eff:
// e^-4.5 / (1 - e^-4.5)
constexpr float kGaussTailRatio = 0.0112337927f;
constexpr float kPi = 3.14159265358979f;

// Device error bits (latched in DevState::error).
constexpr uint32_t kErrCapacity = 1u;
constexpr uint32_t kErrTimeout = 2u;    // a bounded wait on the tensor cores gave up
constexpr uint32_t kErrBounds = 4u;     // debug build: a device index check failed
constexpr uint32_t kInjectShadeTimeout = 1u;   // shading kernels issue no tensor-core work

// Index checks of the debug build (compiled with -DPULSAR_DEBUG): a failed
// check latches kErrBounds in the device state (pulsar_status then returns
// PULSAR_ERR_INTERNAL) and evaluates to false, so the guarded access is
// skipped; no trap.  The release build compiles them to `true`.
#ifdef PULSAR_DEBUG
#define PULSAR_CHECK(state, cond) \
    ((cond) ? true : (atomicOr(&(state)->error, ::pulsar::kErrBounds), false))
#else
#define PULSAR_CHECK(state, cond) true
#endif

// Per-camera constants of a frame (all cameras of a batch share the image
// size, the parameters and the spheres).
struct Frame {
    float R[9], t[3];
    float fx, fy, cx, cy, znear, zfar;
    float ifx, ify;       // 1/fx, 1/fy (RN)
    float ifx_lo, ify_lo; // low parts: 1/fx = ifx + ifx_lo to ~2^-48
    float fmin;           // min(fx, fy); fx on ties
    float gamma, inv_gamma, bg_eps, stop_tau, kappa, amin;
    float inv_zrange;     // 1/(zfar - znear)
    float zk_hi, zk_lo;   // log2(e)/((zfar - znear) gamma) as a float pair
    float eg_hi, eg_lo;   // log2(e) eps/gamma as a float pair
    int width, height, tiles_x, tiles_y, n_tiles;
    int n_track, channels;
    int n;
    uint32_t flags;
    uint32_t max_pairs;
    int ortho;            // orthographic camera: rays along +z, slopes a = b = 0
    // the camera's place in the batch
    int cam, n_cams;
    uint32_t tile_base;   // cam * n_tiles: its first tile in the batch's tile lists
    uint32_t pix_base;    // cam * width * height: its first pixel in the pixel buffers
    uint32_t rec_base;    // cam * n: its first sphere record / gradient accumulator
    uint32_t n_tiles_all; // n_cams * n_tiles
    uint32_t pix_all;     // n_cams * width * height: plane stride of ids / d
};

// The cameras of a frame, passed by value to every kernel (f[0] also holds
// the batch-wide fields); a block finds its camera from its tile.
struct Frames {
    Frame f[kMaxCams];
};

// Small device-resident counters.
struct DevState {
    unsigned long long hits;    // hit pairs composited by the last forward
    uint32_t n_pairs;           // M of the last bin
    uint32_t error;             // latched kErr* bits
    uint32_t inject;            // test hook bits (kInject*), cleared by pulsar_status
    uint32_t pair_cursor;       // staged pairs reserved by the projection (zero between frames)
    uint32_t n_long;            // tiles whose list is longer than one warp sorts, this frame
    uint32_t long_next;         // next entry of long_tiles to sort (reset by the tile scan)
};

// ------------------------------------------------ error-free transforms --
// TwoProduct via FMA, Knuth's TwoSum, Dekker's FastTwoSum (as used by
// Ogita, Rump and Oishi for compensated dot products, SIAM J. Sci. Comput.
// 2005).
struct FPair { float hi, lo; };

__device__ __forceinline__ FPair ef_prod(float a, float b) {
    const float p = __fmul_rn(a, b);
    return {p, __fmaf_rn(a, b, -p)};
}
__device__ __forceinline__ FPair ef_sum(float a, float b) {
    const float s = __fadd_rn(a, b);
    const float bb = __fsub_rn(s, a);
    return {s, __fadd_rn(__fsub_rn(a, __fsub_rn(s, bb)), __fsub_rn(b, bb))};
}
__device__ __forceinline__ FPair ef_fast_sum(float a, float b) {
    const float s = __fadd_rn(a, b);
    return {s, __fsub_rn(b, __fsub_rn(s, a))};
}

// Row k of c = R p + t as hi + lo: compensated three-term dot product plus t.
__device__ __forceinline__ FPair camera_row(float r0, float r1, float r2, float tk,
                                            float px, float py, float pz) {
    const FPair a = ef_prod(r0, px);
    const FPair b = ef_prod(r1, py);
    const FPair s1 = ef_sum(a.hi, b.hi);
    float err = __fadd_rn(__fadd_rn(a.lo, b.lo), s1.lo);
    const FPair c = ef_prod(r2, pz);
    const FPair s2 = ef_sum(s1.hi, c.hi);
    err = __fadd_rn(__fadd_rn(err, c.lo), s2.lo);
    const FPair s3 = ef_sum(s2.hi, tk);
    err = __fadd_rn(err, s3.lo);
    return ef_sum(s3.hi, err);
}

// (x.hi + x.lo) / (z.hi + z.lo) as a pair: one Newton correction of the
// quotient with the exact FMA remainder.
__device__ __forceinline__ FPair pair_quotient(FPair x, FPair z) {
    const float q1 = __fdiv_rn(x.hi, z.hi);
    float rem = __fmaf_rn(-q1, z.hi, x.hi);
    rem = __fadd_rn(rem, x.lo);
    rem = __fmaf_rn(-q1, z.lo, rem);
    return ef_fast_sum(q1, __fdiv_rn(rem, z.hi));
}

// c0 + f * q as a pair: the projected centre in pixels.
__device__ __forceinline__ FPair pair_project(float f, float c0, FPair q) {
    const FPair p = ef_prod(f, q.hi);
    const float plo = __fmaf_rn(f, q.lo, p.lo);
    const FPair s = ef_sum(c0, p.hi);
    return ef_sum(s.hi, __fadd_rn(s.lo, plo));
}

// Pixel range [lo, hi] along one image axis (n pixels) covered by the tangent
// cone of a sphere with centre coordinate X along the axis, depth Z and
// radius rr: the two tangent directions in the (axis, z) plane,
// u = c0 + f (X L +- rr Z) / (Z L -+ X rr), L = sqrt(X^2 + Z^2 - rr^2)
// (the tan(a +- b) identity; Pulsar Sec. B.1.1 avoids trigonometry).
// Returns false if the range is empty.
__device__ __forceinline__ bool tangent_range(float X, float Z, float rr, float f, float c0,
                                              int n, int* lo, int* hi) {
    const float L = __fsqrt_rn(__fsub_rn(__fadd_rn(__fmul_rn(X, X), __fmul_rn(Z, Z)),
                                         __fmul_rn(rr, rr)));
    const float zl = __fmul_rn(Z, L), xr = __fmul_rn(X, rr);
    const float xl = __fmul_rn(X, L), rz = __fmul_rn(rr, Z);
    const float dhi = __fsub_rn(zl, xr);
    const float dlo = __fadd_rn(zl, xr);
    const float uhi = dhi > 0.0f ? __fadd_rn(c0, __fmul_rn(f, __fdiv_rn(__fadd_rn(xl, rz), dhi)))
                                 : __int_as_float(0x7f800000);
    const float ulo = dlo > 0.0f ? __fadd_rn(c0, __fmul_rn(f, __fdiv_rn(__fsub_rn(xl, rz), dlo)))
                                 : __int_as_float(0xff800000);
    float a = ceilf(__fsub_rn(ulo, 0.5f));
    float b = floorf(__fsub_rn(uhi, 0.5f));
    const float top = (float)(n - 1);
    a = a < 0.0f ? 0.0f : a;
    b = b > top ? top : b;
    if (!(a <= b)) return false;
    *lo = (int)a;
    *hi = (int)b;
    return true;
}

// Per-pixel ray constants of the decision path: direction (a, b, 1), origin
// (ox, oy, 0).  Pinhole: a = (px - cx)/fx, b = (py - cy)/fy, origin 0;
// orthographic: a = b = 0, ox = (px - cx)/fx, oy = (py - cy)/fy.
struct PixelRay {
    float px, py;   // pixel centre
    float a, b;     // ray slopes
    float qq;       // 1 + a^2 + b^2
    float ox, oy;   // ray origin
};

__device__ __forceinline__ PixelRay pixel_ray(int x, int y, const Frame& f) {
    PixelRay r;
    r.px = __fadd_rn(__int2float_rn(x), 0.5f);
    r.py = __fadd_rn(__int2float_rn(y), 0.5f);
    const float sa = __fdiv_rn(__fsub_rn(r.px, f.cx), f.fx);
    const float sb = __fdiv_rn(__fsub_rn(r.py, f.cy), f.fy);
    r.a = f.ortho ? 0.0f : sa;
    r.b = f.ortho ? 0.0f : sb;
    r.ox = f.ortho ? sa : 0.0f;
    r.oy = f.ortho ? sb : 0.0f;
    r.qq = __fadd_rn(__fadd_rn(1.0f, __fmul_rn(r.a, r.a)), __fmul_rn(r.b, r.b));
    return r;
}

// Orthographic pixel range [ceil(c0 + f (X - rr) - 1/2), floor(c0 + f (X +
// rr) - 1/2)] along one image axis (n pixels), clamped to the image.
// Returns false if the range is empty.
__device__ __forceinline__ bool ortho_range(float X, float rr, float f, float c0, int n,
                                            int* lo, int* hi) {
    const float umin = __fadd_rn(c0, __fmul_rn(f, __fsub_rn(X, rr)));
    const float umax = __fadd_rn(c0, __fmul_rn(f, __fadd_rn(X, rr)));
    float a = ceilf(__fsub_rn(umin, 0.5f));
    float b = floorf(__fsub_rn(umax, 0.5f));
    const float top = (float)(n - 1);
    a = a < 0.0f ? 0.0f : a;
    b = b > top ? top : b;
    if (!(a <= b)) return false;
    *lo = (int)a;
    *hi = (int)b;
    return true;
}

// Q = (rho / c.z)^2 * qq evaluated from pixel offsets to the projected centre
// (u_hi + u_lo, v_hi + v_lo); also returns the slopes U, V of the offset.
__device__ __forceinline__ float ray_offset_q(const float4& uv, const PixelRay& r, float ifx,
                                              float ify, float* U, float* V) {
    const float du = __fsub_rn(__fsub_rn(r.px, uv.x), uv.y);
    const float dv = __fsub_rn(__fsub_rn(r.py, uv.z), uv.w);
    *U = __fmul_rn(du, ifx);
    *V = __fmul_rn(dv, ify);
    const float X = __fmaf_rn(*U, r.b, -__fmul_rn(*V, r.a));
    return __fmaf_rn(*U, *U, __fmaf_rn(*V, *V, __fmul_rn(X, X)));
}

// ------------------------------------------------ float-pair value path --
// Products and sums of unevaluated pairs hi + lo (relative error ~2^-44).
__device__ __forceinline__ FPair pp_mul(FPair x, FPair y) {
    const float p = __fmul_rn(x.hi, y.hi);
    float e = __fmaf_rn(x.hi, y.hi, -p);
    e = __fmaf_rn(x.hi, y.lo, e);
    e = __fmaf_rn(x.lo, y.hi, e);
    return {p, e};
}
__device__ __forceinline__ FPair pp_sq(FPair x) {
    const float p = __fmul_rn(x.hi, x.hi);
    const float e = __fmaf_rn(x.hi, x.hi, -p);
    return {p, __fmaf_rn(__fmul_rn(2.0f, x.hi), x.lo, e)};
}
__device__ __forceinline__ FPair pp_add(FPair x, FPair y) {
    const FPair s = ef_sum(x.hi, y.hi);
    return {s.hi, __fadd_rn(s.lo, __fadd_rn(x.lo, y.lo))};
}
__device__ __forceinline__ FPair pp_sub(FPair x, FPair y) {
    return pp_add(x, FPair{-y.hi, -y.lo});
}

// Per-pixel ray slopes a, b and |q|^2 = 1 + a^2 + b^2 as pairs, and 1/|q|^2.
struct PixelPairs { FPair a, b, qq; float iqq; };

__device__ __forceinline__ FPair slope_pair(float p, float c0, float ifl, float ifl_lo) {
    return pp_mul(ef_sum(p, -c0), FPair{ifl, ifl_lo});
}

__device__ __forceinline__ PixelPairs pixel_pairs(FPair a, FPair b) {
    PixelPairs q;
    q.a = a;
    q.b = b;
    q.qq = pp_add(pp_add(FPair{1.0f, 0.0f}, pp_sq(a)), pp_sq(b));
    q.iqq = __frcp_rn(q.qq.hi);
    return q;
}

__device__ __forceinline__ PixelPairs pixel_pairs(const PixelRay& r, const Frame& f) {
    return pixel_pairs(slope_pair(r.px, f.cx, f.ifx, f.ifx_lo),
                       slope_pair(r.py, f.cy, f.ify, f.ify_lo));
}

// Distance factor d = 1 - rho / r_eff of a hit at pixel centre (px, py),
// accurate to ~1e-12 absolute also at the silhouette, where 1 - rho/r_eff
// cancels catastrophically in plain fp32 (Pulsar App. A: orthogonal
// ray-to-sphere distance).
//   rho^2 / r_eff^2 = Q ir2 / qq,  Q = U^2 + V^2 + (U b - V a)^2,
//   U = (px - u)/fx, V = (py - v)/fy, ir2 = (c.z / r_eff)^2,
//   d = (qq - Q ir2) / (qq (1 + rho / r_eff)).
// The difference qq - Q ir2 is formed in pair arithmetic; the final scaling
// 1 / (1 + sqrt(t)) uses the approximate reciprocal square root and division
// (a few ulps relative).
__device__ __forceinline__ float distance_factor(const float4& uv, float ir2_hi, float ir2_lo,
                                                 float px, float py, const PixelPairs& pq,
                                                 const Frame& f, bool gaussian) {
    // offsets to the projected centre, renormalised so that every hi part below
    // is the rounded value of its pair (px - u_hi is exact but coarse)
    FPair du = ef_sum(px, -uv.x);
    du = ef_sum(du.hi, __fsub_rn(du.lo, uv.y));
    FPair dv = ef_sum(py, -uv.z);
    dv = ef_sum(dv.hi, __fsub_rn(dv.lo, uv.w));
    const FPair U = pp_mul(du, FPair{f.ifx, f.ifx_lo});
    const FPair V = pp_mul(dv, FPair{f.ify, f.ify_lo});
    const FPair X = pp_sub(pp_mul(U, pq.b), pp_mul(V, pq.a));
    const FPair Q = pp_add(pp_add(pp_sq(U), pp_sq(V)), pp_sq(X));
    const FPair Qs = pp_mul(Q, FPair{ir2_hi, ir2_lo});
    const FPair D = pp_sub(pq.qq, Qs);
    const float t = __fmul_rn(__fadd_rn(Qs.hi, Qs.lo), pq.iqq);   // (rho / r_eff)^2
    const float Dq = __fmul_rn(__fadd_rn(D.hi, D.lo), pq.iqq);    // 1 - t
    if (gaussian) {
        // Gaussian footprint: exp(-4.5 t) - e^-4.5 = e^-4.5 expm1(4.5 (1 - t)),
        // accurate at the rim from the pair-precision 1 - t
        return kGaussTailRatio * expm1f(4.5f * Dq);
    }
    const float s = t > 0.0f ? t * rsqrtf(t) : 0.0f;
    return __fdividef(Dq, 1.0f + s);
}

__device__ __forceinline__ bool rect_contains(uint2 rc, int x, int y) {
    return x >= (int)(rc.x & 0xffffu) && x <= (int)(rc.x >> 16) && y >= (int)(rc.y & 0xffffu) &&
           y <= (int)(rc.y >> 16);
}

// ------------------------------------------------------------ cp.async --
// Asynchronous global -> shared copies (PTX cp.async): 16-byte pieces bypass
// L1, 4-byte ones go through it; a thread's copies complete at its wait.
__device__ __forceinline__ void cp_async16(void* dst, const void* src) {
    const unsigned s = static_cast<unsigned>(__cvta_generic_to_shared(dst));
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(s), "l"(src) : "memory");
}
__device__ __forceinline__ void cp_async4(void* dst, const void* src) {
    const unsigned s = static_cast<unsigned>(__cvta_generic_to_shared(dst));
    asm volatile("cp.async.ca.shared.global [%0], [%1], 4;" ::"r"(s), "l"(src) : "memory");
}
// Programmatic dependent launch: the kernels of the render path are launched
// with programmatic stream serialization, so a kernel's grid is set up while
// the previous one finishes, and each begins by waiting until the previous
// grid has completed and its memory is visible -- before any global memory
// access, so no read or write overlaps the previous kernel.  (No early
// trigger: CTAs launched early and parked on the wait cost the previous
// kernel's tail more than they saved, measured on the headline step.)
// Launched without the attribute, or with no previous grid in flight, the
// wait returns at once.
__device__ __forceinline__ void pdl_begin() {
    asm volatile("griddepcontrol.wait;" ::: "memory");
}

// ------------------------------------------------- mbarrier / bulk copy --
constexpr unsigned long long kWaitNs = 250000000ull;   // bound of every mbarrier wait (0.25 s)

__device__ __forceinline__ uint32_t smem_u32(const void* p) {
    return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ unsigned long long global_ns() {
    unsigned long long t;
    asm volatile("mov.u64 %0, %globaltimer;" : "=l"(t));
    return t;
}

__device__ __forceinline__ void mbar_init(uint64_t* mbar) {
    asm volatile("mbarrier.init.shared::cta.b64 [%0], 1;" ::"r"(smem_u32(mbar)));
}

// Wait for the mbarrier phase of the given parity, at most kWaitNs of wall
// time (try_wait itself may suspend for an unspecified while, so the bound is
// on the global timer, not on the number of polls); false on timeout.
__device__ __forceinline__ bool mbar_wait(uint64_t* mbar, uint32_t parity) {
    const unsigned long long t0 = global_ns();
    for (;;) {
        uint32_t done;
        asm volatile(
            "{\n.reg .pred p;\nmbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n"
            "selp.u32 %0, 1, 0, p;\n}\n"
            : "=r"(done)
            : "r"(smem_u32(mbar)), "r"(parity)
            : "memory");
        if (done) return true;
        if (global_ns() - t0 > kWaitNs) return false;
    }
}

// Bulk copy (TMA engine) of `bytes` bytes global -> shared, completing on
// mbar: both addresses 16-byte aligned, bytes a multiple of 16.
__device__ __forceinline__ void bulk_load(void* dst, const void* src, uint32_t bytes,
                                          uint64_t* mbar) {
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_u32(mbar)),
                 "r"(bytes)
                 : "memory");
    asm volatile(
        "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::
            "r"(smem_u32(dst)),
        "l"(src), "r"(bytes), "r"(smem_u32(mbar))
        : "memory");
}

__device__ __forceinline__ void cp_async_commit() {
    asm volatile("cp.async.commit_group;" ::: "memory");
}
__device__ __forceinline__ void cp_async_wait_all() {
    asm volatile("cp.async.wait_all;" ::: "memory");
}

// 2^x by the approximate base-2 exponential of the PTX ISA (a few ulps; the
// value path's tolerance is orders of magnitude wider).
__device__ __forceinline__ float ex2_approx(float x) {
    float y;
    asm("ex2.approx.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}

// ---------------------------------------------------------- workspace --
// Per-sphere record written by the projection: 64 bytes, i.e. two 32-byte
// sectors, so a gather by sphere id moves no byte it does not use.
//   uv  : u_hi, u_lo, v_hi, v_lo             projected centre as float pairs
//   ex  : e_hi, e_lo, o, flags (bits)         exponent o z~/gamma as a pair
//   geo : ir2_hi, ir2_lo, c.z, r_eff          ir2 = (c.z / r_eff)^2 as a pair
//   rk  : x0 | x1 << 16, y0 | y1 << 16, bits of s2 = (r_eff/c.z)^2, bits of
//         the depth key c.z - r_eff           (decision quantities)
// Only kept spheres' records are written (the tile lists, which hold kept
// spheres only, are the one way to them); a culled sphere's record keeps
// whatever it held.
struct __align__(16) SphereRec {
    float4 uv;
    float4 ex;
    float4 geo;
    uint4 rk;
};

struct Workspace {
    SphereRec* rec;    // [maxN]
    // per camera of a batch: [maxCams][...] blocks, camera after camera
    float4* gacc;      // [maxN] dL/dc.xyz, dL/dr accumulators (zeroed by the forward; by
                       // the backward's launcher when a frame is differentiated again)
    float4* gacc2;     // [maxN] dL/do, dL/df[0..2] accumulators for C <= 3, one for all
                       // cameras (zeroed as gacc; the finalize writes them out)
    float* hitcnt;     // [maxN] pixels tracking each sphere, for normalised gradients
                       // (zeroed as gacc)
    uint32_t* tile_count;   // [maxB] (zero between frames)
    uint32_t* tile_start;   // [maxB+1]
    uint32_t* long_tiles;   // [maxB] tiles with lists longer than one warp sorts, in tile order
    uint4* staged;          // [max_pairs] (tile, slot in tile, key bits, id) from the projection
    unsigned long long* pairs;      // [max_pairs] (key bits << 32 | id), bucketed by tile
    unsigned long long* pairs_alt;  // [max_pairs] merge scratch for long tiles
    uint32_t* tile_ids;     // [max_pairs] sorted tile lists
    float* mg;              // [maxP]
    float* wsum;            // [maxP]
    int32_t* ids;           // [maxT][maxP] tracked hits' positions in their tile list, -1 padded
    float* dtr;             // [maxT][maxP] distance factor d of each tracked hit
    int32_t* nhits;         // [maxP]
    float2* kpart;          // [4][maxB] per-tile partial dL/d(fx, fy, cx, cy), float pairs
    float2* rtpart;         // [cameras][12][finalize blocks] per-block partial dL/dR, dL/dt,
                            // float pairs
    float* shade_part;      // [CTAs][kShadeParams] per-CTA weight-gradient shares of the
                            // shading backward
    unsigned char* shade_img;   // the shading weights as the kernels stage them (bf16)
    DevState* state;
};

// ------------------------------------------------------- host helpers --
// Per-camera frame constants from the ABI structs (host side).  log2 units:
// exponents are kept in base 2 (exp2 is the cheap hardware exponential).
inline void fill_frame(Frame& f, const float R[9], const float t[3], float fx, float fy,
                       float cx, float cy, int width, int height, float znear, float zfar,
                       int ortho, float gamma, float bg_eps, float stop_tau, float kappa,
                       float amin, int n_track, int channels, uint32_t flags, int n,
                       uint32_t max_pairs, int cam, int n_cams) {
    for (int k = 0; k < 9; ++k) f.R[k] = R[k];
    for (int k = 0; k < 3; ++k) f.t[k] = t[k];
    f.fx = fx; f.fy = fy; f.cx = cx; f.cy = cy;
    f.znear = znear; f.zfar = zfar;
    f.ifx = 1.0f / fx;
    f.ify = 1.0f / fy;
    f.ifx_lo = (float)(1.0 / (double)fx - (double)f.ifx);
    f.ify_lo = (float)(1.0 / (double)fy - (double)f.ify);
    f.fmin = fx <= fy ? fx : fy;
    f.gamma = gamma;
    f.inv_gamma = 1.0f / gamma;
    f.bg_eps = bg_eps;
    f.stop_tau = stop_tau;
    f.kappa = kappa;
    f.amin = amin;
    f.inv_zrange = 1.0f / (zfar - znear);
    const double log2e = 1.4426950408889634073599;
    const double zk = log2e / (((double)zfar - (double)znear) * (double)gamma);
    f.zk_hi = (float)zk;
    f.zk_lo = (float)(zk - (double)f.zk_hi);
    const double eg = log2e * (double)bg_eps / (double)gamma;
    f.eg_hi = (float)eg;
    f.eg_lo = (float)(eg - (double)f.eg_hi);
    f.width = width;
    f.height = height;
    f.tiles_x = (width + kTile - 1) / kTile;
    f.tiles_y = (height + kTile - 1) / kTile;
    f.n_tiles = f.tiles_x * f.tiles_y;
    f.n_track = n_track;
    f.channels = channels;
    f.n = n;
    f.flags = flags;
    f.max_pairs = max_pairs;
    f.ortho = ortho;
    f.cam = cam;
    f.n_cams = n_cams;
    f.tile_base = (uint32_t)(cam * f.n_tiles);
    f.pix_base = (uint32_t)cam * (uint32_t)(width * height);
    f.rec_base = (uint32_t)cam * (uint32_t)n;
    f.n_tiles_all = (uint32_t)(n_cams * f.n_tiles);
    f.pix_all = (uint32_t)n_cams * (uint32_t)(width * height);
}

// ---------------------------------------------------------- launchers --
// (defined in the .cu files; all enqueue on `stream` and never synchronise)
// Launch with programmatic stream serialization (the kernel must begin with
// pdl_begin()).
template <typename... KArgs, typename... Args>
cudaError_t launch_pdl(void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem,
                       cudaStream_t stream, Args... args) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = grid;
    cfg.blockDim = block;
    cfg.dynamicSmemBytes = smem;
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, kernel, static_cast<KArgs>(args)...);
}

cudaError_t launch_project(const Frames& fs, const Workspace& w, const float* pos,
                           const float* radius, const float* opacity, cudaStream_t stream);
cudaError_t launch_bin(const Frames& fs, const Workspace& w, cudaStream_t stream);
cudaError_t prepare_forward();   // opt the forward kernels into their shared memory
cudaError_t prepare_bin();       // opt the long-list sort into its shared memory
cudaError_t prepare_backward();  // opt the backward kernels into their shared memory
cudaError_t launch_forward(const Frames& fs, const Workspace& w, const float* features,
                           const float* bg, float* image, int max_pairs_stride,
                           cudaStream_t stream);
// resident CTAs per SM of the shading kernels (their grid caps are these x SMs)
struct ShadeLaunch {
    int fwd_per_sm = 0, bwd_per_sm = 0;
};
cudaError_t prepare_shade(ShadeLaunch* sl);
size_t shade_image_bytes();   // bytes of Workspace::shade_img   // opt the shading kernels into their shared memory
cudaError_t launch_shade_forward(const Frames& fs, const Workspace& w, const float* features,
                                 const float* params, float* rgb, int grid_cap,
                                 cudaStream_t stream);
cudaError_t launch_shade_backward(const Frames& fs, const Workspace& w, const float* features,
                                  const float* params, const float* grad_rgb,
                                  float* grad_features, float* grad_params, int grid_cap,
                                  cudaStream_t stream);
// zeroed: the accumulators were zeroed by this frame's forward and not used
// since (else the launcher zeroes them first)
cudaError_t launch_backward(const Frames& fs, const Workspace& w, const float* pos,
                            const float* features, const float* image, const float* grad_image,
                            float* grad_pos, float* grad_radius, float* grad_opacity,
                            float* grad_features, float* grad_cam, bool zeroed,
                            cudaStream_t stream);

}  // namespace pulsar
