// Backward pass (Pulsar Sec. B.2): pixel-wise, reusing the forward pass's
// backward-information buffer (Sec. B.1.4) so no intersection search is
// repeated.  Gradients of L = sum_pixels <G, F> flow through the first
// n_track hits of every pixel only (Sec. 2, B.1.3).
//
// k_backward  one block per 16x16 tile, one thread per pixel.  The tile's
//             candidates are staged through shared memory in batches (as in
//             the forward) and each pixel finds its tracked hits among them by
//             their list positions (stored by the forward).  For tracked hit
//             k, runs of adjacent lanes that hold the same candidate are
//             tree-reduced, so one lane per run issues the global atomics --
//             the warp-level aggregation of DISTWAR (arxiver abstract); a
//             warp's two pixel rows are interleaved column by column, so the
//             footprint of a small sphere is a single run.  dL/dc and
//             dL/dr go to a float4 accumulator with one vector reduction; with
//             at most three channels dL/do and dL/df go to a second one (two
//             reductions per run in all), otherwise straight to the caller's
//             (zeroed) arrays.  The intrinsics' gradient is summed per thread
//             and reduced per block.
// k_finalize_one_cam, k_finalize_cams  four spheres per thread: dL/dp =
//             R^T dL/dc and dL/dr out of the accumulator, and dL/do, dL/df out
//             of the second one, summed over the cameras of a batch (the
//             frame's forward zeroed both accumulators; a second backward of
//             the same frame has its launcher zero them again);
//             dL/dR = sum dL/dc p^T and dL/dt = sum dL/dc of every camera
//             reduced per block (Pulsar Sec. B.2: sphere-wise camera-gradient
//             accumulation).
// k_camera_reduce  one block per output of each camera's grad_cam sums that
//             output's per-block partials in a fixed order (the device-wide
//             reduction).
#include "pulsar_internal.cuh"

namespace pulsar {
namespace {

constexpr int kBwdThreads = kTilePix;
constexpr int kFinThreads = 256;
constexpr int kCamThreads = 1024;

__device__ __forceinline__ void red_add_v4(float4* addr, float a, float b, float c, float d) {
    asm volatile("red.global.add.v4.f32 [%0], {%1, %2, %3, %4};"
                 :: "l"(addr), "f"(a), "f"(b), "f"(c), "f"(d) : "memory");
}

// Shared-memory batch of the backward: candidates staged per batch; the
// records in static shared memory, the features in dynamic shared memory.
template <int CMAX>
struct BwdBatch {
    static constexpr int n = CMAX <= 4 ? 512 : (CMAX <= 8 ? 256 : (CMAX <= 16 ? 384 : (CMAX <= 32 ? 192 : 128)));
    // features of 8 and more channels (a multiple of 4) are staged and read
    // 16 bytes at a time when the caller's rows allow it: rows padded by four
    // words to keep them 16-byte aligned; otherwise an odd row stride in
    // words, so that lanes reading different candidates' rows hit different
    // banks
    static constexpr bool vec = CMAX >= 8 && CMAX % 4 == 0;
    static constexpr int fsp = vec ? CMAX + 4 : (CMAX | 1);
    static constexpr int feat_bytes = n * fsp * 4;
};

// Blocks per SM: 4 up to four channels, 3 up to eight (76 registers, no
// spills; 176 vs 218 us at two blocks on the headline frame with eight
// channels), 2 up to sixteen (three spill, 268 vs 244 us), 1 beyond.
template <int CMAX, bool MULTI>
__global__ void __launch_bounds__(kBwdThreads, CMAX <= 4 ? 4 : (CMAX <= 8 ? 3 : (CMAX <= 16 ? 2 : 1)))
k_backward(Frames fs, Workspace w, const float* __restrict__ features,
           const float* __restrict__ image, const float* __restrict__ grad_image,
           float* __restrict__ grad_opacity, float* __restrict__ grad_features, int mode) {
    pdl_begin();
    // the frame's pair count and the tile's list bounds, loaded together
    const uint32_t n_pairs = w.state->n_pairs;
    uint32_t start = w.tile_start[blockIdx.x], end = w.tile_start[blockIdx.x + 1];
    // mode bit 0: geometry gradients wanted; bit 1: feature gradient rows are
    // 16-byte aligned with C a multiple of 4 (vector reductions); bit 2: C <= 3,
    // opacity and feature gradients into the second accumulator
    const bool want_geom = (mode & 1) != 0;
    const bool feat_v4 = (mode & 2) != 0;
    const bool acc2 = CMAX <= 4 && (mode & 4) != 0;
    constexpr int NB = BwdBatch<CMAX>::n;
    constexpr int NV = 5 + CMAX;   // dL/dc.xyz, dL/dr, dL/do, dL/df[CMAX]
    constexpr int FSP = BwdBatch<CMAX>::fsp;
    __shared__ float4 s_uv[NB];
    __shared__ float4 s_ex[NB];          // exponent hi, lo, o, flags
    __shared__ float4 s_geo[NB];         // (c.z/r_eff)^2 hi, lo, c.z, r_eff
    __shared__ int s_id[NB];
    extern __shared__ __align__(16) float s_feat[];   // [NB][FSP]
    __shared__ float s_k[kBwdThreads / 32][4];
    // the block's camera and its tile in that camera's image (a single camera
    // is indexed statically, so its constants stay instruction operands)
    const int tile_g = blockIdx.x;
    const int cam = MULTI ? tile_g / fs.f[0].n_tiles : 0;
    const Frame& f = fs.f[MULTI ? cam : 0];
    const int tile = tile_g - cam * f.n_tiles;
    const int C = f.channels;
    const int tyi = tile / f.tiles_x, txi = tile - tyi * f.tiles_x;
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    // warp w covers rows 2w, 2w+1 of the tile with the two rows of a column in
    // adjacent lanes, so a small sphere's footprint is one run of lanes
    const int x = txi * kTile + (lane >> 1), y = tyi * kTile + 2 * warp + (lane & 1);
    const bool inside = x < f.width && y < f.height;
    // the pixel in the batch's buffers; planes of ids / d are pix_all apart
    const uint32_t P = f.pix_all;
    const uint32_t p = f.pix_base + (uint32_t)(inside ? y * f.width + x : 0);
    const SphereRec* __restrict__ rec = w.rec + f.rec_base;   // this camera's records
    float4* __restrict__ gacc = w.gacc + f.rec_base;
    float4* __restrict__ gacc2 = w.gacc2;   // one for all cameras: their sum is wanted
    end = min(end, f.max_pairs);
    start = min(start, end);
    // 16-byte feature copies and loads: every row is whole (C == CMAX) and
    // 16-byte aligned
    const bool fvec = BwdBatch<CMAX>::vec && C == CMAX &&
                      (reinterpret_cast<uintptr_t>(features) & 15u) == 0;
    // the pixel's inputs, loaded together with the list bounds (the buffers
    // are read in bounds also for an overflowed frame, whose values go unused)
    float G[CMAX], F[CMAX];
    if (CMAX % 4 == 0 && C == CMAX &&
        ((reinterpret_cast<uintptr_t>(image) | reinterpret_cast<uintptr_t>(grad_image)) & 15u) == 0) {
        // whole 16-byte-aligned rows: 16-byte loads
        const float4* g4 = reinterpret_cast<const float4*>(grad_image + (size_t)p * CMAX);
        const float4* f4 = reinterpret_cast<const float4*>(image + (size_t)p * CMAX);
#pragma unroll
        for (int q = 0; q < CMAX / 4; ++q) {
            const float4 gq = inside ? g4[q] : make_float4(0.f, 0.f, 0.f, 0.f);
            const float4 fq = inside ? f4[q] : make_float4(0.f, 0.f, 0.f, 0.f);
            G[4 * q] = gq.x; G[4 * q + 1] = gq.y; G[4 * q + 2] = gq.z; G[4 * q + 3] = gq.w;
            F[4 * q] = fq.x; F[4 * q + 1] = fq.y; F[4 * q + 2] = fq.z; F[4 * q + 3] = fq.w;
        }
    } else {
#pragma unroll
        for (int c = 0; c < CMAX; ++c) {
            G[c] = (inside && c < C) ? grad_image[(size_t)p * C + c] : 0.0f;
            F[c] = (inside && c < C) ? image[(size_t)p * C + c] : 0.0f;
        }
    }
    const float mg = inside ? w.mg[p] : 0.0f;
    const float wsum = inside ? w.wsum[p] : 1.0f;
    // the pixel's tracked slots are in list order, so the slots of one batch
    // are a run: a cursor walks them across the batches, each slot read once
    int k = 0;
    int pos = inside ? w.ids[p] : -1;   // slot k's list position (-1: no more hits)
    float d = inside ? w.dtr[p] : 0.0f;
    if (n_pairs > f.max_pairs) return;   // overflowed frame: no valid buffer
    // a batch's records and features are copied by cp.async
    auto stage = [&](uint32_t b0, int nb) {
        for (int t = tid; t < nb; t += kBwdThreads) {
            int id = (int)w.tile_ids[b0 + t];
            if (!PULSAR_CHECK(w.state, (uint32_t)id < (uint32_t)f.n)) id = 0;
            const float4* src = reinterpret_cast<const float4*>(rec + id);
            cp_async16(&s_uv[t], src + 0);
            cp_async16(&s_ex[t], src + 1);
            cp_async16(&s_geo[t], src + 2);
            s_id[t] = id;
            if (fvec) {
#pragma unroll
                for (int q = 0; q < CMAX / 4; ++q)
                    cp_async16(&s_feat[t * FSP + 4 * q], features + (size_t)id * CMAX + 4 * q);
            } else {
#pragma unroll
                for (int c = 0; c < CMAX; ++c)
                    if (c < C) cp_async4(&s_feat[t * FSP + c], features + (size_t)id * C + c);
            }
        }
        cp_async_commit();
    };
    if (start < end) stage(start, (int)min((uint32_t)NB, end - start));

    const PixelRay ray = pixel_ray(x, y, f);
    const float iqq = __frcp_rn(ray.qq);
    const float iw = inside ? 1.0f / wsum : 0.0f;
    float gk[4] = {0.f, 0.f, 0.f, 0.f};   // d/d(fx, fy, cx, cy)

    for (uint32_t b0 = start; b0 < end; b0 += NB) {
        const int nb = (int)min((uint32_t)NB, end - b0);
        if (b0 != start) {
            __syncthreads();   // previous batch done
            stage(b0, nb);
        }
        cp_async_wait_all();
        __syncthreads();
        const int base = (int)(b0 - start);
        for (;;) {
            // this pixel's next tracked hit, if its list position is in the batch
            const bool valid = pos >= base && pos < base + nb;
            if (__ballot_sync(0xffffffffu, valid) == 0u) break;
            const int j = pos - base;
            const float dk = d;
            if (valid) {   // slot k+1 loads while slot k is processed
                ++k;
                pos = k < f.n_track ? w.ids[(uint32_t)k * P + p] : -1;
                d = k < f.n_track ? w.dtr[(uint32_t)k * P + p] : 0.0f;
            }
            float v[NV];
#pragma unroll
            for (int q = 0; q < NV; ++q) v[q] = 0.0f;
            bool cut = true;
            if (valid) {
                const float4 uv = s_uv[j];
                const float4 ex = s_ex[j];
                const float4 geo = s_geo[j];
                const uint32_t fl = __float_as_uint(ex.w);
                cut = (fl & kFlagCut) != 0u;
                float U, V;
                const float Q = ray_offset_q(uv, ray, f.ifx, f.ify, &U, &V);
                // value path only (the hit set is the forward's): the hardware's
                // approximate square root and reciprocals, a few ulps, are plenty
                const float qi = Q * iqq;
                const float rq = qi > 0.0f ? qi * rsqrtf(qi) : 0.0f;   // rho / c.z (orthographic: rho)
                const float o = ex.z;
                const float E = ex2_approx(__fsub_rn(ex.x, mg) + ex.y);   // exponents in log2 units
                const float wt = o * dk * E;
                float sdot = 0.0f;
                if (BwdBatch<CMAX>::vec && fvec) {
#pragma unroll
                    for (int q = 0; q < CMAX / 4; ++q) {
                        const float4 fq = *reinterpret_cast<const float4*>(&s_feat[j * FSP + 4 * q]);
                        const float fv[4] = {fq.x, fq.y, fq.z, fq.w};
#pragma unroll
                        for (int r = 0; r < 4; ++r) {
                            const int c = 4 * q + r;
                            sdot += G[c] * (fv[r] - F[c]);
                            v[5 + c] = wt * iw * G[c];           // dL/df = (w / W) G
                        }
                    }
                } else {
#pragma unroll
                    for (int c = 0; c < CMAX; ++c) {
                        if (c < C) {
                            const float fc = s_feat[j * FSP + c];
                            sdot += G[c] * (fc - F[c]);
                            v[5 + c] = wt * iw * G[c];           // dL/df = (w / W) G
                        }
                    }
                }
                const float sj = sdot * iw;                      // dL/dw = <G, f - F> / W
                v[4] = sj * dk * E * (1.0f + ex.x * 0.693147181f);   // dw/do = d E (1 + o z~/gamma)
                if (want_geom && !cut) {
                    const float Z = geo.z, reff = geo.w;
                    const float ireff = __fdividef(1.0f, reff);
                    // normalised gradients: the sphere's share of the K gradient
                    // is scaled by 1e-3 / A, A = pi (f_min r_eff / c.z)^2 px^2
                    // (orthographic: pi (f_min r_eff)^2)
                    float ks = 1.0f;
                    if (f.flags & kParamNormalize) {
                        const float rz = f.fmin * (f.ortho ? reff : reff / Z);
                        ks = 1e-3f / (kPi * rz * rz);
                    }
                    const float sE = sj * o * E;                 // dL/dd
                    // depth factor: dw/dz~ = w o / gamma, dz~/dc.z = -1/(zfar - znear)
                    float gcz = -sj * wt * o * f.inv_gamma * f.inv_zrange;
                    const float rho = f.ortho ? rq : rq * Z;
                    // with x = rho / r_eff: dd/drho = d'(x) / r_eff, dd/dr_eff =
                    // -d'(x) rho / r_eff^2; linear d' = -1, Gaussian d' = -9 x exp(-4.5
                    // x^2) / (1 - e^-4.5) = -9 x (d + e^-4.5 / (1 - e^-4.5))
                    const float ddx = (f.flags & kParamGaussian)
                                          ? -9.0f * rho * ireff * (dk + kGaussTailRatio)
                                          : -1.0f;
                    const float g_rho = sE * ddx * ireff;
                    const float g_reff = -sE * ddx * rho * ireff * ireff;
                    float gr = 0.0f;
                    if (fl & kFlagFloor) {
                        // r_eff = kappa c.z / f_min (orthographic: kappa / f_min)
                        if (!f.ortho) gcz += g_reff * f.kappa / f.fmin;
                        const float gf = -g_reff * f.kappa * (f.ortho ? 1.0f : Z) / (f.fmin * f.fmin);
                        if (f.fx <= f.fy) gk[0] += ks * gf; else gk[1] += ks * gf;
                    } else {
                        gr = g_reff;
                    }
                    float gcx = 0.0f, gcy = 0.0f;
                    if (Q > 0.0f) {
                        // drho/dc = e_perp / rho, e = c - c.z q = -c.z (U, V, 0)
                        const float kq = (U * ray.a + V * ray.b) * iqq;
                        const float irq = __fdividef(1.0f, rq);
                        const float n0 = -(U - kq * ray.a) * irq;
                        const float n1 = -(V - kq * ray.b) * irq;
                        const float n2 = kq * irq;
                        gcx = g_rho * n0;
                        gcy = g_rho * n1;
                        gcz += g_rho * n2;
                        // drho/dq = -(c.q / q.q) e_perp / rho with c.q / q.q = c.z (1 - kq);
                        // q = ((px - cx)/fx, (py - cy)/fy, 1).  Orthographic: drho/do =
                        // -e_perp / rho for the origin o = ((px - cx)/fx, (py - cy)/fy, 0)
                        const float sq = f.ortho ? -1.0f : -Z * (1.0f - kq);
                        const float ga = ks * g_rho * sq * n0, gb = ks * g_rho * sq * n1;
                        gk[0] -= ga * (f.ortho ? ray.ox : ray.a) * f.ifx;
                        gk[1] -= gb * (f.ortho ? ray.oy : ray.b) * f.ify;
                        gk[2] -= ga * f.ifx;
                        gk[3] -= gb * f.ify;
                    }
                    v[0] = gcx;
                    v[1] = gcy;
                    v[2] = gcz;
                    v[3] = gr;
                }
            }
            // runs of lanes that hold the same candidate are tree-reduced; one
            // lane per run issues the atomics (lanes without a hit here get
            // distinct keys, so they form runs of one)
            const int key = valid ? j : -1 - lane;
            const int prevk = __shfl_up_sync(0xffffffffu, key, 1);
            const bool head = lane == 0 || prevk != key;
            const uint32_t heads = __ballot_sync(0xffffffffu, head);
            const int hl = 31 - __clz(heads & (0xffffffffu >> (31 - lane)));
            const int rank = lane - hl;
            const uint32_t above = lane == 31 ? 0u : (heads & (0xfffffffeu << lane));
            const int nexth = above ? __ffs(above) - 1 : 32;
            const int gsz = nexth - hl;
            const int gmax = __reduce_max_sync(0xffffffffu, gsz);
            for (int off = 1; off < gmax; off <<= 1) {
                const bool take = (rank & (2 * off - 1)) == 0 && rank + off < gsz;
#pragma unroll
                for (int q = 0; q < NV; ++q) {
                    const float o2 = __shfl_down_sync(0xffffffffu, v[q], off);
                    if (take) v[q] += o2;
                }
            }
            if (rank == 0 && valid) {
                const int id = s_id[j];
                if (f.flags & kParamNormalize) atomicAdd(&w.hitcnt[f.rec_base + id], (float)gsz);
                if (want_geom && !cut) red_add_v4(&gacc[id], v[0], v[1], v[2], v[3]);
                if constexpr (CMAX <= 4) {
                    // channels beyond C hold zeros
                    if (acc2) red_add_v4(&gacc2[id], v[4], v[5], v[6], v[7]);
                }
                if (!acc2 && grad_opacity) atomicAdd(&grad_opacity[id], v[4]);
                if (!acc2 && grad_features) {
                    float* gf = grad_features + (size_t)id * C;
                    bool done_v4 = false;
                    if constexpr (CMAX % 4 == 0) {
                        if (feat_v4) {
#pragma unroll
                            for (int c = 0; c < CMAX; c += 4)
                                if (c < C)
                                    red_add_v4(reinterpret_cast<float4*>(gf + c), v[5 + c],
                                               v[6 + c], v[7 + c], v[8 + c]);
                            done_v4 = true;
                        }
                    }
                    if (!done_v4) {
#pragma unroll
                        for (int c = 0; c < CMAX; ++c)
                            if (c < C) atomicAdd(&gf[c], v[5 + c]);
                    }
                }
            }
        }
    }
    if (!want_geom) return;
    // block reduction of the intrinsics' gradient
#pragma unroll
    for (int q = 0; q < 4; ++q) {
        float s = gk[q];
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) s += __shfl_down_sync(0xffffffffu, s, o);
        if (lane == 0) s_k[warp][q] = s;
    }
    __syncthreads();
    if (tid < 4) {
        // compensated (float pair) sum of the warp partials; this GPU's fp64
        // pipe is far too slow even for reductions
        FPair s = {0.0f, 0.0f};
        for (int q = 0; q < kBwdThreads / 32; ++q) s = pp_add(s, FPair{s_k[q][tid], 0.0f});
        w.kpart[(size_t)tid * f.n_tiles_all + tile_g] = make_float2(s.hi, s.lo);
    }
}

// Warp sums of twelve per-lane values in 16 shuffles (slots padded to 16):
// at every butterfly step a lane keeps half of its slots, adds its partner's
// copies of them and hands over the other half, so the live slots halve per
// step; afterwards lanes 2s and 2s + 1 both hold the warp total of slot s.
// The pairing is that of a shuffle-down tree, in a fixed order.
__device__ __forceinline__ float warp_sum12(const float (&a)[12], int lane) {
    float v[8];
    const bool b4 = (lane & 16) != 0;
#pragma unroll
    for (int j = 0; j < 8; ++j) {   // v[j]: slot j + 8 b4
        const float lo = a[j], hi = j + 8 < 12 ? a[j + 8] : 0.0f;
        v[j] = (b4 ? hi : lo) + __shfl_xor_sync(0xffffffffu, b4 ? lo : hi, 16);
    }
    float u[4];
    const bool b3 = (lane & 8) != 0;
#pragma unroll
    for (int j = 0; j < 4; ++j)     // u[j]: slot j + 4 b3 + 8 b4
        u[j] = (b3 ? v[j + 4] : v[j]) + __shfl_xor_sync(0xffffffffu, b3 ? v[j] : v[j + 4], 8);
    float t[2];
    const bool b2 = (lane & 4) != 0;
#pragma unroll
    for (int j = 0; j < 2; ++j)     // t[j]: slot j + 2 b2 + 4 b3 + 8 b4
        t[j] = (b2 ? u[j + 2] : u[j]) + __shfl_xor_sync(0xffffffffu, b2 ? u[j] : u[j + 2], 4);
    const bool b1 = (lane & 2) != 0;   // slot lane >> 1
    float r = (b1 ? t[1] : t[0]) + __shfl_xor_sync(0xffffffffu, b1 ? t[0] : t[1], 2);
    return r + __shfl_xor_sync(0xffffffffu, r, 1);
}

// Finalize of one sphere; adds its share of dL/dR and dL/dt to acc.
__device__ __forceinline__ void finalize_one(const Frame& f, float4 g, float px, float py, float pz,
                                             float* gp, float* acc) {
    gp[0] = f.R[0] * g.x + f.R[3] * g.y + f.R[6] * g.z;
    gp[1] = f.R[1] * g.x + f.R[4] * g.y + f.R[7] * g.z;
    gp[2] = f.R[2] * g.x + f.R[5] * g.y + f.R[8] * g.z;
    acc[0] += g.x * px; acc[1] += g.x * py; acc[2] += g.x * pz;
    acc[3] += g.y * px; acc[4] += g.y * py; acc[5] += g.y * pz;
    acc[6] += g.z * px; acc[7] += g.z * py; acc[8] += g.z * pz;
    acc[9] += g.x; acc[10] += g.y; acc[11] += g.z;
}

// dL/do and dL/df[0..C) (C <= 3) of four consecutive spheres out of the
// second accumulator's q[4], as 16-byte stores (the arrays are 16-byte
// aligned and i0 is a multiple of 4, so C floats per sphere are whole float4s).
__device__ __forceinline__ void store_acc2_v4(const float4 (&q)[4], int i0, int C,
                                              float* __restrict__ grad_opacity,
                                              float* __restrict__ grad_features) {
    if (grad_opacity)
        *reinterpret_cast<float4*>(grad_opacity + i0) = make_float4(q[0].x, q[1].x, q[2].x, q[3].x);
    if (grad_features) {
        float v[12];
#pragma unroll
        for (int k = 0; k < 4; ++k) {
            v[3 * k] = q[k].y;
            v[3 * k + 1] = q[k].z;
            v[3 * k + 2] = q[k].w;
        }
        float4* o4 = reinterpret_cast<float4*>(grad_features + (size_t)C * i0);
        if (C == 3) {
            o4[0] = make_float4(v[0], v[1], v[2], v[3]);
            o4[1] = make_float4(v[4], v[5], v[6], v[7]);
            o4[2] = make_float4(v[8], v[9], v[10], v[11]);
        } else if (C == 2) {
            o4[0] = make_float4(q[0].y, q[0].z, q[1].y, q[1].z);
            o4[1] = make_float4(q[2].y, q[2].z, q[3].y, q[3].z);
        } else {
            o4[0] = make_float4(q[0].y, q[1].y, q[2].y, q[3].y);
        }
    }
}

// The same for one sphere i, scaled by sph.
__device__ __forceinline__ void store_acc2_one(float4 q, int i, int C, float sph,
                                               float* __restrict__ grad_opacity,
                                               float* __restrict__ grad_features) {
    if (grad_opacity) grad_opacity[i] = q.x * sph;
    if (grad_features) {
        float* gf = grad_features + (size_t)i * C;
        gf[0] = q.y * sph;
        if (C > 1) gf[1] = q.z * sph;
        if (C > 2) gf[2] = q.w * sph;
    }
}

// One camera: four consecutive spheres per thread with 16-byte loads and
// stores, so each thread has seven independent loads in flight.  With normalised gradients
// (Pulsar Sec. B.2) a sphere's gradients are divided by the number of pixels
// tracking it and its share of dL/dR, dL/dt is scaled by 1e-3 / A (A its
// rendered disc's area in px^2, as for dL/dK in the backward).
// mode bit 0: 16-byte accesses allowed (aligned arrays); bit 1: dL/do, dL/df
// are in the second accumulator (C <= 3).
__global__ void __launch_bounds__(kFinThreads)
k_finalize_one_cam(Frames fs, Workspace w, const float* __restrict__ pos, float* __restrict__ grad_pos,
           float* __restrict__ grad_radius, float* __restrict__ grad_opacity,
           float* __restrict__ grad_features, int mode) {
    pdl_begin();
    __shared__ float s_part[kFinThreads / 32][12];
    const Frame& f = fs.f[0];
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int i0 = 4 * (blockIdx.x * blockDim.x + tid);
    const bool vec_ok = (mode & 1) != 0, acc2 = (mode & 2) != 0;
    const int C = f.channels;
    float acc[12];
#pragma unroll
    for (int q = 0; q < 12; ++q) acc[q] = 0.0f;
    const float4 z4 = make_float4(0.f, 0.f, 0.f, 0.f);
    const bool norm = (f.flags & kParamNormalize) != 0;
    if (!norm && vec_ok && i0 + 3 < f.n) {
        float4 g[4], q[4];
#pragma unroll
        for (int k = 0; k < 4; ++k) g[k] = w.gacc[i0 + k];
        if (acc2) {
#pragma unroll
            for (int k = 0; k < 4; ++k) q[k] = w.gacc2[i0 + k];
        }
        const float4* p4 = reinterpret_cast<const float4*>(pos + 3 * (size_t)i0);
        const float4 pa = p4[0], pb = p4[1], pc = p4[2];
        const float p[12] = {pa.x, pa.y, pa.z, pa.w, pb.x, pb.y, pb.z, pb.w, pc.x, pc.y, pc.z, pc.w};
        float gp[12];
#pragma unroll
        for (int k = 0; k < 4; ++k)
            finalize_one(f, g[k], p[3 * k], p[3 * k + 1], p[3 * k + 2], gp + 3 * k, acc);
        if (grad_pos) {
            float4* o4 = reinterpret_cast<float4*>(grad_pos + 3 * (size_t)i0);
            o4[0] = make_float4(gp[0], gp[1], gp[2], gp[3]);
            o4[1] = make_float4(gp[4], gp[5], gp[6], gp[7]);
            o4[2] = make_float4(gp[8], gp[9], gp[10], gp[11]);
        }
        if (grad_radius)
            *reinterpret_cast<float4*>(grad_radius + i0) = make_float4(g[0].w, g[1].w, g[2].w, g[3].w);
        if (acc2) store_acc2_v4(q, i0, C, grad_opacity, grad_features);
    } else {
        // ragged tail, unaligned arrays or normalised gradients
        for (int i = i0; i < min(i0 + 4, f.n); ++i) {
            const float4 g = w.gacc[i];
            float sph = 1.0f, cams = 1.0f;
            if (norm) {
                const float cnt = w.hitcnt[i];
                sph = cnt > 0.0f ? 1.0f / cnt : 1.0f;
                // a sphere no pixel tracks has no gradient (and may be culled,
                // its record not written this frame)
                cams = 0.0f;
                if (cnt > 0.0f) {
                    const float4 geo = w.rec[i].geo;          // c.z in z, r_eff in w
                    const float rz = f.fmin * (f.ortho ? geo.w : geo.w / geo.z);
                    cams = rz > 0.0f ? 1e-3f / (kPi * rz * rz) : 0.0f;
                }
                if (!acc2) {
                    if (grad_opacity) grad_opacity[i] *= sph;
                    if (grad_features)
                        for (int c = 0; c < C; ++c) grad_features[(size_t)i * C + c] *= sph;
                }
            }
            if (acc2) store_acc2_one(w.gacc2[i], i, C, sph, grad_opacity, grad_features);
            float gp[3];
            const float4 gc = make_float4(g.x * cams, g.y * cams, g.z * cams, g.w);
            finalize_one(f, gc, pos[3 * (size_t)i], pos[3 * (size_t)i + 1], pos[3 * (size_t)i + 2], gp, acc);
            if (grad_pos) {
                // R^T dL/dc of the unscaled g, averaged
                const size_t i3 = 3 * (size_t)i;
                grad_pos[i3] = (f.R[0] * g.x + f.R[3] * g.y + f.R[6] * g.z) * sph;
                grad_pos[i3 + 1] = (f.R[1] * g.x + f.R[4] * g.y + f.R[7] * g.z) * sph;
                grad_pos[i3 + 2] = (f.R[2] * g.x + f.R[5] * g.y + f.R[8] * g.z) * sph;
            }
            if (grad_radius) grad_radius[i] = g.w * sph;
        }
    }
    {
        const float s = warp_sum12(acc, lane);
        if ((lane & 1) == 0 && (lane >> 1) < 12) s_part[warp][lane >> 1] = s;
    }
    __syncthreads();
    if (tid < 12) {
        FPair s = {0.0f, 0.0f};
        for (int q = 0; q < kFinThreads / 32; ++q) s = pp_add(s, FPair{s_part[q][tid], 0.0f});
        w.rtpart[(size_t)tid * gridDim.x + blockIdx.x] = make_float2(s.hi, s.lo);
    }
}

// A batch of cameras: four consecutive spheres per thread with 16-byte
// loads and stores.  For every camera of the batch: dL/dp += R^T dL/dc, dL/dr
// += its part, dL/do and dL/df += theirs, and the sphere's share of that
// camera's dL/dR = sum dL/dc p^T, dL/dt = sum dL/dc goes into per-block
// partials.  With normalised gradients (Pulsar Sec. B.2; one camera) a
// sphere's gradients are divided by the number of pixels tracking it and its
// share of dL/dR, dL/dt is scaled by 1e-3 / A (A its rendered disc's area in
// px^2, as for dL/dK in the backward).  mode as for k_finalize_one_cam.
// (3 blocks per SM: at 4 the per-camera sums of the second accumulator spill)
__global__ void __launch_bounds__(kFinThreads, 3)
k_finalize_cams(Frames fs, Workspace w, const float* __restrict__ pos, float* __restrict__ grad_pos,
           float* __restrict__ grad_radius, float* __restrict__ grad_opacity,
           float* __restrict__ grad_features, int mode) {
    pdl_begin();
    __shared__ float s_part[kFinThreads / 32][12];
    const Frame& f0 = fs.f[0];
    const int n = f0.n, n_cams = f0.n_cams, C = f0.channels;
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int i0 = 4 * (blockIdx.x * blockDim.x + tid);
    const int cnt = i0 < n ? min(4, n - i0) : 0;
    const bool norm = (f0.flags & kParamNormalize) != 0;
    const bool vec = (mode & 1) != 0 && cnt == 4, acc2 = (mode & 2) != 0;
    const float4 z4 = make_float4(0.f, 0.f, 0.f, 0.f);
    float p[12];
    if (vec) {
        const float4* p4 = reinterpret_cast<const float4*>(pos + 3 * (size_t)i0);
        const float4 pa = p4[0], pb = p4[1], pc = p4[2];
        p[0] = pa.x; p[1] = pa.y; p[2] = pa.z; p[3] = pa.w;
        p[4] = pb.x; p[5] = pb.y; p[6] = pb.z; p[7] = pb.w;
        p[8] = pc.x; p[9] = pc.y; p[10] = pc.z; p[11] = pc.w;
    } else {
#pragma unroll
        for (int q = 0; q < 12; ++q) p[q] = q < 3 * cnt ? pos[3 * (size_t)i0 + q] : 0.0f;
    }
    float sph_last[4] = {1.0f, 1.0f, 1.0f, 1.0f};
    for (int cam = 0; cam < n_cams; ++cam) {
        const Frame& f = fs.f[cam];
        float4 g[4];
#pragma unroll
        for (int k = 0; k < 4; ++k) g[k] = k < cnt ? w.gacc[f.rec_base + i0 + k] : z4;
        float acc[12], gp[12], gr[4];
#pragma unroll
        for (int q = 0; q < 12; ++q) acc[q] = 0.0f;
#pragma unroll
        for (int k = 0; k < 4; ++k) {
            float sph = 1.0f, cams = 1.0f;
            if (norm && k < cnt) {
                const int i = i0 + k;
                const float c = w.hitcnt[f.rec_base + i];
                sph = c > 0.0f ? 1.0f / c : 1.0f;
                // a sphere no pixel tracks has no gradient (and may be culled,
                // its record not written this frame)
                cams = 0.0f;
                if (c > 0.0f) {
                    const float4 geo = w.rec[f.rec_base + i].geo;   // c.z in z, r_eff in w
                    const float rz = f.fmin * (f.ortho ? geo.w : geo.w / geo.z);
                    cams = rz > 0.0f ? 1e-3f / (kPi * rz * rz) : 0.0f;
                }
                if (!acc2) {
                    if (grad_opacity) grad_opacity[i] *= sph;
                    if (grad_features)
                        for (int ch = 0; ch < C; ++ch) grad_features[(size_t)i * C + ch] *= sph;
                }
                sph_last[k] = sph;
            }
            const float4 gk = g[k];
            gp[3 * k + 0] = (f.R[0] * gk.x + f.R[3] * gk.y + f.R[6] * gk.z) * sph;
            gp[3 * k + 1] = (f.R[1] * gk.x + f.R[4] * gk.y + f.R[7] * gk.z) * sph;
            gp[3 * k + 2] = (f.R[2] * gk.x + f.R[5] * gk.y + f.R[8] * gk.z) * sph;
            gr[k] = gk.w * sph;
            const float cx = gk.x * cams, cy = gk.y * cams, cz = gk.z * cams;
            const float px = p[3 * k], py = p[3 * k + 1], pz = p[3 * k + 2];
            acc[0] += cx * px; acc[1] += cx * py; acc[2] += cx * pz;
            acc[3] += cy * px; acc[4] += cy * py; acc[5] += cy * pz;
            acc[6] += cz * px; acc[7] += cz * py; acc[8] += cz * pz;
            acc[9] += cx; acc[10] += cy; acc[11] += cz;
        }
        // dL/dp and dL/dr: the first camera writes, the others add
        if (vec) {
            if (grad_pos) {
                float4* o4 = reinterpret_cast<float4*>(grad_pos + 3 * (size_t)i0);
                if (cam > 0) {
                    const float4 a = o4[0], b = o4[1], c = o4[2];
                    gp[0] += a.x; gp[1] += a.y; gp[2] += a.z; gp[3] += a.w;
                    gp[4] += b.x; gp[5] += b.y; gp[6] += b.z; gp[7] += b.w;
                    gp[8] += c.x; gp[9] += c.y; gp[10] += c.z; gp[11] += c.w;
                }
                o4[0] = make_float4(gp[0], gp[1], gp[2], gp[3]);
                o4[1] = make_float4(gp[4], gp[5], gp[6], gp[7]);
                o4[2] = make_float4(gp[8], gp[9], gp[10], gp[11]);
            }
            if (grad_radius) {
                float4* r4 = reinterpret_cast<float4*>(grad_radius + i0);
                float4 v = make_float4(gr[0], gr[1], gr[2], gr[3]);
                if (cam > 0) {
                    const float4 a = *r4;
                    v.x += a.x; v.y += a.y; v.z += a.z; v.w += a.w;
                }
                *r4 = v;
            }
        } else {
#pragma unroll
            for (int k = 0; k < 4; ++k) {
                if (k < cnt) {
                    const int i = i0 + k;
                    if (grad_pos)
                        for (int l = 0; l < 3; ++l)
                            grad_pos[3 * (size_t)i + l] = gp[3 * k + l] + (cam > 0 ? grad_pos[3 * (size_t)i + l] : 0.0f);
                    if (grad_radius) grad_radius[i] = gr[k] + (cam > 0 ? grad_radius[i] : 0.0f);
                }
            }
        }
        {
            const float s = warp_sum12(acc, lane);
            if ((lane & 1) == 0 && (lane >> 1) < 12) s_part[warp][lane >> 1] = s;
        }
        __syncthreads();
        if (tid < 12) {
            FPair s = {0.0f, 0.0f};
            for (int q = 0; q < kFinThreads / 32; ++q) s = pp_add(s, FPair{s_part[q][tid], 0.0f});
            w.rtpart[((size_t)cam * 12 + tid) * gridDim.x + blockIdx.x] = make_float2(s.hi, s.lo);
        }
        __syncthreads();   // s_part is reused by the next camera
    }
    if (acc2) {   // dL/do, dL/df: one accumulator summed over the cameras
        float4 q[4];
#pragma unroll
        for (int k = 0; k < 4; ++k) q[k] = k < cnt ? w.gacc2[i0 + k] : z4;
        if (vec && !norm) {
            store_acc2_v4(q, i0, C, grad_opacity, grad_features);
        } else {
#pragma unroll
            for (int k = 0; k < 4; ++k)
                if (k < cnt) store_acc2_one(q[k], i0 + k, C, sph_last[k], grad_opacity, grad_features);
        }
    }
}

// One block per (output, camera): output q of the camera's 16 -- dL/dR and
// dL/dt from the finalize blocks' partials, dL/d(fx, fy, cx, cy) from its
// tiles' partials -- summed in a fixed order in float-pair arithmetic
// (deterministic, ~1e-14 relative; Pulsar Sec. B.2's device-wide camera
// reduction).  The partials of an output are contiguous: thread t sums
// elements t, t + 1024, ... with kCamAcc of them in flight, then the block
// combines the threads' sums in a fixed tree.  The order is a function of
// the output's length only.
constexpr int kCamAcc = 4;

__global__ void __launch_bounds__(kCamThreads)
k_camera_reduce(Frames fs, Workspace w, int fin_blocks, float* __restrict__ grad_cam) {
    pdl_begin();
    static_assert(kCamThreads == 1024, "32 warps");
    __shared__ float2 s_part[32];
    const int q = blockIdx.x, cam = blockIdx.y;
    const Frame& f = fs.f[cam];
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const float2* src;
    int len;
    if (q < 12) {
        src = w.rtpart + ((size_t)cam * 12 + q) * fin_blocks;
        len = fin_blocks;
    } else {
        src = w.kpart + (size_t)(q - 12) * f.n_tiles_all + f.tile_base;
        len = f.n_tiles;
    }
    FPair v[kCamAcc];
#pragma unroll
    for (int u = 0; u < kCamAcc; ++u) v[u] = FPair{0.0f, 0.0f};
    for (int b = tid; b < len; b += kCamAcc * kCamThreads) {
        float2 t[kCamAcc];
#pragma unroll
        for (int u = 0; u < kCamAcc; ++u)
            t[u] = b + u * kCamThreads < len ? src[b + u * kCamThreads] : make_float2(0.0f, 0.0f);
#pragma unroll
        for (int u = 0; u < kCamAcc; ++u) v[u] = pp_add(v[u], FPair{t[u].x, t[u].y});
    }
#pragma unroll
    for (int h = kCamAcc / 2; h > 0; h >>= 1)
#pragma unroll
        for (int u = 0; u < h; ++u) v[u] = pp_add(v[u], v[u + h]);
    FPair r = v[0];
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
        const FPair t = {__shfl_down_sync(0xffffffffu, r.hi, o),
                         __shfl_down_sync(0xffffffffu, r.lo, o)};
        r = pp_add(r, t);
    }
    if (lane == 0) s_part[warp] = make_float2(r.hi, r.lo);
    __syncthreads();
    if (warp == 0) {
        const float2 t0 = s_part[lane];
        r = FPair{t0.x, t0.y};
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) {
            const FPair t = {__shfl_down_sync(0xffffffffu, r.hi, o),
                             __shfl_down_sync(0xffffffffu, r.lo, o)};
            r = pp_add(r, t);
        }
        if (lane == 0 && grad_cam) grad_cam[16 * cam + q] = __fadd_rn(r.hi, r.lo);
    }
}

template <int CMAX>
cudaError_t launch_bwd_c(const Frames& fs, const Workspace& w, const float* features,
                         const float* image, const float* grad_image, float* grad_opacity,
                         float* grad_features, int mode, cudaStream_t stream) {
    const dim3 grid(fs.f[0].n_tiles_all), block(kBwdThreads);
    constexpr int smem = BwdBatch<CMAX>::feat_bytes;
    if (fs.f[0].n_cams == 1)
        return launch_pdl(k_backward<CMAX, false>, grid, block, smem, stream, fs, w, features,
                          image, grad_image, grad_opacity, grad_features, mode);
    return launch_pdl(k_backward<CMAX, true>, grid, block, smem, stream, fs, w, features, image,
                      grad_image, grad_opacity, grad_features, mode);
}

// Opt the backward kernels into their dynamic shared memory (the
// 16-channel batch's records and features exceed 48 KB together).
template <int CMAX>
cudaError_t prepare_bwd_c() {
    cudaError_t e = cudaFuncSetAttribute(k_backward<CMAX, false>,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         BwdBatch<CMAX>::feat_bytes);
    if (e == cudaSuccess)
        e = cudaFuncSetAttribute(k_backward<CMAX, true>,
                                 cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 BwdBatch<CMAX>::feat_bytes);
    return e;
}

}  // namespace

cudaError_t prepare_backward() {
    cudaError_t e = prepare_bwd_c<3>();
    if (e == cudaSuccess) e = prepare_bwd_c<4>();
    if (e == cudaSuccess) e = prepare_bwd_c<8>();
    if (e == cudaSuccess) e = prepare_bwd_c<16>();
    if (e == cudaSuccess) e = prepare_bwd_c<32>();
    if (e == cudaSuccess) e = prepare_bwd_c<kMaxChannels>();
    return e;
}

cudaError_t launch_backward(const Frames& fs, const Workspace& w, const float* pos,
                            const float* features, const float* image, const float* grad_image,
                            float* grad_pos, float* grad_radius, float* grad_opacity,
                            float* grad_features, float* grad_cam, bool zeroed,
                            cudaStream_t stream) {
    const Frame& f = fs.f[0];
    const int want_geom = (grad_pos || grad_radius || grad_cam) ? 1 : 0;
    const int feat_v4 = (f.channels % 4 == 0 && grad_features &&
                         (reinterpret_cast<uintptr_t>(grad_features) & 15u) == 0) ? 2 : 0;
    // C <= 3: dL/do and dL/df in the second accumulator, written by the finalize
    const bool acc2 = f.channels <= 3 && (grad_opacity || grad_features);
    const int mode = want_geom | feat_v4 | (acc2 ? 4 : 0);
    const bool norm = (f.flags & kParamNormalize) != 0;
    // the accumulators the kernel reduces into start at zero: the frame's
    // forward zeroed them; a further backward of the same frame zeroes them here
    const size_t nk = (size_t)f.n * f.n_cams;
    cudaError_t e = cudaSuccess;
    if (!zeroed) {
        if (want_geom && nk) e = cudaMemsetAsync(w.gacc, 0, nk * sizeof(float4), stream);
        if (e == cudaSuccess && acc2 && f.n)
            e = cudaMemsetAsync(w.gacc2, 0, (size_t)f.n * sizeof(float4), stream);
        if (e == cudaSuccess && norm && nk)
            e = cudaMemsetAsync(w.hitcnt, 0, nk * sizeof(float), stream);
        if (e != cudaSuccess) return e;
    }
    if (f.channels == 3)
        e = launch_bwd_c<3>(fs, w, features, image, grad_image, grad_opacity, grad_features, mode,
                            stream);
    else if (f.channels <= 4)
        e = launch_bwd_c<4>(fs, w, features, image, grad_image, grad_opacity, grad_features, mode,
                            stream);
    else if (f.channels <= 8)
        e = launch_bwd_c<8>(fs, w, features, image, grad_image, grad_opacity, grad_features, mode,
                            stream);
    else if (f.channels <= 16)
        e = launch_bwd_c<16>(fs, w, features, image, grad_image, grad_opacity, grad_features,
                             mode, stream);
    else if (f.channels <= 32)
        e = launch_bwd_c<32>(fs, w, features, image, grad_image, grad_opacity, grad_features,
                             mode, stream);
    else
        e = launch_bwd_c<kMaxChannels>(fs, w, features, image, grad_image, grad_opacity,
                                       grad_features, mode, stream);
    if (e != cudaSuccess) return e;
    if (want_geom || norm || acc2) {
        const int blocks = (f.n + 4 * kFinThreads - 1) / (4 * kFinThreads);
        // 16-byte accesses need 16-byte aligned arrays (true for torch allocations)
        const int vec_ok = ((reinterpret_cast<uintptr_t>(pos) | reinterpret_cast<uintptr_t>(grad_pos) |
                             reinterpret_cast<uintptr_t>(grad_radius) |
                             reinterpret_cast<uintptr_t>(grad_opacity) |
                             reinterpret_cast<uintptr_t>(grad_features)) & 15u) == 0;
        const int fmode = (vec_ok ? 1 : 0) | (acc2 ? 2 : 0);
        if (blocks > 0 && f.n_cams == 1)
            e = launch_pdl(k_finalize_one_cam, dim3(blocks), dim3(kFinThreads), 0, stream, fs, w,
                           pos, grad_pos, grad_radius, grad_opacity, grad_features, fmode);
        else if (blocks > 0)
            e = launch_pdl(k_finalize_cams, dim3(blocks), dim3(kFinThreads), 0, stream, fs, w, pos,
                           grad_pos, grad_radius, grad_opacity, grad_features, fmode);
        if (e == cudaSuccess && want_geom)
            e = launch_pdl(k_camera_reduce, dim3(16, f.n_cams), dim3(kCamThreads), 0, stream, fs, w,
                           blocks, grad_cam);
    }
    return e;
}

}  // namespace pulsar
