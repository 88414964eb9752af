// Step 0 of the forward pass (Pulsar Sec. B.1.1, "Enclosing Rectangle
// Calculation"): one thread per sphere computes the camera-space centre,
// culls, floors the radius so every sphere covers at least one pixel,
// projects the centre, bounds the pixel rectangle without trigonometry and
// forms the depth key.  The warp then walks its (sphere, tile) pairs
// cooperatively, so a sphere covering many tiles does not stall its lane:
// each pair takes the next slot of its tile's counter and is staged, with
// that slot, for the binning pass.  A batch of cameras is projected in one
// launch: each thread loads its sphere once and repeats the above for every
// camera (records and tiles of camera k live at its offsets in the batch).
#include "pulsar_internal.cuh"

namespace pulsar {
namespace {

constexpr int kProjectThreads = 256;

// 8 blocks per SM (32 registers): the kernel waits on memory and atomics, so
// resident warps count for more than the few registers spilled to L1
__global__ void __launch_bounds__(kProjectThreads, 8)
k_project(Frames fs, Workspace w, const float* __restrict__ pos, const float* __restrict__ radius,
          const float* __restrict__ opacity) {
    pdl_begin();
    const int i = blockIdx.x * blockDim.x + threadIdx.x;
    const int lane = threadIdx.x & 31;
    const int n = fs.f[0].n;
    float px = 0.f, py = 0.f, pz = 0.f, r = 0.f, op = 0.f;
    if (i < n) {
        const size_t i3 = 3 * (size_t)i;   // 64-bit: 3 i passes 2^31 beyond 715M spheres
        px = pos[i3];
        py = pos[i3 + 1];
        pz = pos[i3 + 2];
        r = radius[i];
        op = opacity[i];
    }
    for (int cam = 0; cam < fs.f[0].n_cams; ++cam) {
        const Frame& f = fs.f[cam];
        int tx0 = 0, ty0 = 0, ntx = 0, count = 0;
        float key_out = 0.0f;
        if (i < n) {
            const FPair cx = camera_row(f.R[0], f.R[1], f.R[2], f.t[0], px, py, pz);
            const FPair cy = camera_row(f.R[3], f.R[4], f.R[5], f.t[1], px, py, pz);
            const FPair cz = camera_row(f.R[6], f.R[7], f.R[8], f.t[2], px, py, pz);
            const float Z = cz.hi;
            // at-least-one-pixel floor of the radius
            // (orthographic: kappa / f_min)
            const float rfloor = f.ortho ? __fdiv_rn(f.kappa, f.fmin)
                                         : __fdiv_rn(__fmul_rn(f.kappa, Z), f.fmin);
            const bool on_floor = r < rfloor;
            const float reff = on_floor ? rfloor : r;
            bool keep = Z > f.znear && Z < f.zfar && reff < Z;
            float4 r0 = make_float4(0.f, 0.f, 0.f, 0.f), r1 = r0, r2 = r0;
            uint2 rc = make_uint2(1u, 1u);   // empty: x0 = 1 > x1 = 0
            uint32_t flags = 0;
            float key = 0.f, s2 = 0.f;
            if (keep) {
                // projected centre c0 + f c.x / c.z (orthographic: c0 + f c.x)
                const FPair u = pair_project(f.fx, f.cx, f.ortho ? cx : pair_quotient(cx, cz));
                const FPair v = pair_project(f.fy, f.cy, f.ortho ? cy : pair_quotient(cy, cz));
                int x0, x1, y0, y1;
                if (f.ortho)
                    keep = ortho_range(cx.hi, reff, f.fx, f.cx, f.width, &x0, &x1) &&
                           ortho_range(cy.hi, reff, f.fy, f.cy, f.height, &y0, &y1);
                else
                    keep = tangent_range(cx.hi, Z, reff, f.fx, f.cx, f.width, &x0, &x1) &&
                           tangent_range(cy.hi, Z, reff, f.fy, f.cy, f.height, &y0, &y1);
                if (keep) {
                    key = __fsub_rn(Z, reff);
                    // s = r_eff / c.z (orthographic: r_eff, rays parallel)
                    const float tt = f.ortho ? reff : __fdiv_rn(reff, Z);
                    s2 = __fmul_rn(tt, tt);
                    const float g = f.ortho ? __fmul_rn(f.fmin, r) : __fdiv_rn(__fmul_rn(f.fmin, r), Z);
                    const float area = __fmul_rn(kPi, __fmul_rn(g, g));
                    const bool cut = (f.flags & 1u) && !(area > f.amin);
                    flags = kFlagKeep | (on_floor ? kFlagFloor : 0u) | (cut ? kFlagCut : 0u);
                    r0 = make_float4(u.hi, u.lo, v.hi, v.lo);
                    // value path: the exponent o z~ / gamma in log2 units,
                    // log2(e) o (zfar - c.z) / ((zfar - znear) gamma), as a float pair; its
                    // magnitude reaches 1.44/gamma, so a single float would carry ~1e-6
                    // absolute error into every weight through exp2()
                    const FPair nz = ef_sum(f.zfar, -cz.hi);
                    const FPair n = ef_fast_sum(nz.hi, __fsub_rn(nz.lo, cz.lo));
                    FPair on = ef_prod(op, n.hi);
                    on.lo = __fmaf_rn(op, n.lo, on.lo);
                    FPair e = ef_prod(on.hi, f.zk_hi);
                    e.lo = __fmaf_rn(on.hi, f.zk_lo, __fmaf_rn(on.lo, f.zk_hi, e.lo));
                    e = ef_fast_sum(e.hi, e.lo);
                    r1 = make_float4(e.hi, e.lo, op, 0.0f);
                    // (c.z / r_eff)^2 (orthographic: 1 / r_eff^2) as a pair; on the
                    // kappa floor c.z / r_eff (orthographic: 1 / r_eff) = f_min / kappa
                    FPair ir;
                    if (on_floor) {
                        const float q = __fdiv_rn(f.fmin, f.kappa);
                        ir = {q, __fdiv_rn(__fmaf_rn(-q, f.kappa, f.fmin), f.kappa)};
                    } else {
                        ir = pair_quotient(f.ortho ? FPair{1.0f, 0.0f} : cz, FPair{r, 0.0f});
                    }
                    const FPair ir2 = pp_sq(ir);
                    r2 = make_float4(ir2.hi, ir2.lo, Z, reff);
                    rc = make_uint2((uint32_t)x0 | ((uint32_t)x1 << 16),
                                    (uint32_t)y0 | ((uint32_t)y1 << 16));
                    tx0 = x0 / kTile;
                    ty0 = y0 / kTile;
                    ntx = x1 / kTile - tx0 + 1;
                    count = ntx * (y1 / kTile - ty0 + 1);
                    key_out = key;
                }
            }
            // records are read only through the tile lists, i.e. for kept
            // spheres: a culled sphere writes none
            if (flags & kFlagKeep) {
                r1.w = __uint_as_float(flags);
                SphereRec* out = w.rec + f.rec_base + i;
                out->uv = r0;
                out->ex = r1;
                out->geo = r2;
                out->rk = make_uint4(rc.x, rc.y, __float_as_uint(s2), __float_as_uint(key));
            }
        }
        // warp-cooperative tile counting: flatten the warp's (sphere, tile) pairs
        int incl = count;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const int v = __shfl_up_sync(0xffffffffu, incl, o);
            if (lane >= o) incl += v;
        }
        const int total = __shfl_sync(0xffffffffu, incl, 31);
        uint32_t base = 0;
        if (lane == 0 && total > 0) base = atomicAdd(&w.state->pair_cursor, (uint32_t)total);
        base = __shfl_sync(0xffffffffu, base, 0);
        const int warp_first = (blockIdx.x * blockDim.x + threadIdx.x) - lane;
        for (int j0 = 0; j0 < total; j0 += 32) {
            const int j = j0 + lane;
            // owner = first lane whose inclusive prefix exceeds j
            int lo = 0, hi = 31;
#pragma unroll
            for (int s = 0; s < 5; ++s) {
                const int mid = (lo + hi) >> 1;
                const int pm = __shfl_sync(0xffffffffu, incl, mid);
                if (pm > j) hi = mid; else lo = mid + 1;
            }
            const int own = lo;
            const int own_incl = __shfl_sync(0xffffffffu, incl, own);
            const int own_cnt = __shfl_sync(0xffffffffu, count, own);
            const int own_tx0 = __shfl_sync(0xffffffffu, tx0, own);
            const int own_ty0 = __shfl_sync(0xffffffffu, ty0, own);
            const int own_ntx = __shfl_sync(0xffffffffu, ntx, own);
            const uint32_t own_key = __shfl_sync(0xffffffffu, __float_as_uint(key_out), own);
            if (j < total) {
                const int k = j - (own_incl - own_cnt);
                const int tile = (int)f.tile_base + (own_ty0 + k / own_ntx) * f.tiles_x + own_tx0 +
                                 k % own_ntx;
                if (!PULSAR_CHECK(w.state, (uint32_t)tile < f.n_tiles_all)) continue;
                const uint32_t slot = atomicAdd(&w.tile_count[tile], 1u);
                const uint32_t at = base + (uint32_t)j;
                if (at < f.max_pairs)
                    w.staged[at] = make_uint4((uint32_t)tile, slot, own_key, (uint32_t)(warp_first + own));
            }
        }
    }
}

}  // namespace

cudaError_t launch_project(const Frames& fs, const Workspace& w, const float* pos,
                           const float* radius, const float* opacity, cudaStream_t stream) {
    const int n = fs.f[0].n;
    if (n == 0) return cudaSuccess;
    const int blocks = (n + kProjectThreads - 1) / kProjectThreads;
    return launch_pdl(k_project, dim3(blocks), dim3(kProjectThreads), 0, stream, fs, w, pos, radius,
                      opacity);
}

}  // namespace pulsar
