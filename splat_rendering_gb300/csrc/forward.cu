// Forward pass (Pulsar Sec. B.1.2-B.1.4): one block per 16x16 tile; pixel
// parallel in the sense of the paper (no two threads ever write one pixel,
// Sec. B.1), but the work inside a warp is split in two phases so that
// neither phase runs with most lanes idle.
//
// The tile's sorted candidate list is staged through shared memory in
// batches of up to 256 (coalesced id read, 16-byte record gathers).  Each
// warp owns two pixel rows of the tile and first compacts, in list order, the
// batch's candidates whose pixel rectangle touches its rows (cooperative
// filtering at warp level).  Then, 32 candidates at a time:
//   phase 1 (one lane per candidate): the lane runs the fp32 hit test of its
//           candidate on every pixel of the warp's rows inside the
//           candidate's rectangle and sets the candidate's bit in those
//           pixels' hit masks;
//   phase 2 (one lane per pixel): the lane walks its mask bits in increasing
//           order -- candidate order, i.e. earliest possible intersection
//           first -- and blends each hit into its max-shifted running sums,
//           tracking the first n_track ids.
// Between batches the block votes on the early-stop bound (Sec. 3.2, Fig. 3;
// B.1.3).  The pixel's result and its backward-information buffer (tracked
// ids, stabiliser, normaliser; Sec. B.1.4) are written at the end.
#include "pulsar_internal.cuh"

namespace pulsar {
namespace {

constexpr int kFwdThreads = kTilePix;
constexpr int kWarps = kFwdThreads / 32;

// candidates staged per batch: 256, fewer for wide payloads (static smem < 48 KB)
template <int CMAX>
struct Batch {
    static constexpr int n = CMAX <= 16 ? kFwdThreads : 4096 / CMAX;
};

template <int CMAX, int TMAX>
__global__ void __launch_bounds__(kFwdThreads, CMAX <= 4 ? 4 : (CMAX <= 16 ? 2 : 1))
k_forward(Frame f, Workspace w, const float* __restrict__ features, const float* __restrict__ bg,
          float* __restrict__ image) {
    constexpr int NB = Batch<CMAX>::n;
    __shared__ float4 s_uv[NB];
    __shared__ float4 s_ex[NB];          // exponent hi, lo, o, flags
    __shared__ float2 s_ir2[NB];
    __shared__ uint2 s_rect[NB];
    __shared__ float s_s2[NB];
    __shared__ int s_id[NB];
    __shared__ uint8_t s_wmask[NB];
    __shared__ float s_feat[NB * CMAX];
    __shared__ uint16_t s_list[kWarps][NB];
    __shared__ uint32_t s_hmask[kWarps][32];
    __shared__ float s_a[kTile], s_b[kTile];
    __shared__ float s_next_key;
    __shared__ unsigned long long s_hits;

    // a frame whose pairs overflowed max_pairs has unsorted lists: render nothing
    // (the capacity error is latched and reported by pulsar_status)
    if (w.state->n_pairs > f.max_pairs) return;
    const int C = f.channels;
    const int tile = blockIdx.x;
    const int tyi = tile / f.tiles_x, txi = tile - tyi * f.tiles_x;
    const int tx0 = txi * kTile, ty0 = tyi * kTile;
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int x = tx0 + (tid & 15), y = ty0 + (tid >> 4);
    const int row0 = ty0 + 2 * warp;              // the warp's two pixel rows
    const bool inside = x < f.width && y < f.height;
    const PixelRay ray = pixel_ray(x, y, f);
    const PixelPairs pq = pixel_pairs(ray, f);
    const uint32_t lt_mask = (1u << lane) - 1u;
    // decision-path ray slopes of the tile's 16 columns and 16 rows
    if (tid < kTile) {
        s_a[tid] = __fdiv_rn(__fsub_rn(__fadd_rn(__int2float_rn(tx0 + tid), 0.5f), f.cx), f.fx);
    } else if (tid < 2 * kTile) {
        const int r = tid - kTile;
        s_b[r] = __fdiv_rn(__fsub_rn(__fadd_rn(__int2float_rn(ty0 + r), 0.5f), f.cy), f.fy);
    }

    uint32_t start = w.tile_start[tile], end = w.tile_start[tile + 1];
    end = min(end, f.max_pairs);
    start = min(start, end);

    // running max of eps/gamma and o z~/gamma, as a float pair
    float mg = f.eg_hi, mgl = f.eg_lo;
    float wsum = 1.0f;                   // exp(eps/gamma - mg): background weight, shifted
    float acc[CMAX];
#pragma unroll
    for (int c = 0; c < CMAX; ++c) acc[c] = c < C ? bg[c] : 0.0f;
    int ids[TMAX];
#pragma unroll
    for (int k = 0; k < TMAX; ++k) ids[k] = -1;
    int nh = 0;
    bool done = !inside;
    if (tid == 0) s_hits = 0ull;

    for (uint32_t b0 = start; b0 < end; b0 += NB) {
        __syncthreads();   // previous batch fully consumed
        const uint32_t kk = b0 + tid;
        if (tid < NB && kk < end) {
            const int id = (int)w.tile_ids[kk];
            const SphereRec* rp = w.rec + id;
            const uint4 rk = rp->rk;
            const float4 geo = rp->geo;
            const uint2 rc = make_uint2(rk.x, rk.y);
            s_id[tid] = id;
            s_uv[tid] = rp->uv;
            s_ex[tid] = rp->ex;
            s_ir2[tid] = make_float2(geo.x, geo.y);
            s_rect[tid] = rc;
            s_s2[tid] = __uint_as_float(rk.z);
            const int r0 = max((int)(rc.y & 0xffffu) - ty0, 0);
            const int r1 = min((int)(rc.y >> 16) - ty0, kTile - 1);
            s_wmask[tid] = (uint8_t)((0xffu << (r0 >> 1)) & (0xffu >> (7 - (r1 >> 1))));
#pragma unroll
            for (int c = 0; c < CMAX; ++c)
                if (c < C) s_feat[tid * CMAX + c] = features[(size_t)id * C + c];
        }
        if (tid == 0) {
            const uint32_t nx = b0 + NB;
            s_next_key = nx < end ? __uint_as_float(w.rec[w.tile_ids[nx]].rk.w) : 0.0f;
        }
        __syncthreads();
        const int nb = (int)min((uint32_t)NB, end - b0);
        // compact this warp's candidates, in list order
        int cnt = 0;
        for (int g0 = 0; g0 < nb; g0 += 32) {
            const int ci = g0 + lane;
            const bool rel = ci < nb && ((s_wmask[ci] >> warp) & 1u);
            const uint32_t bits = __ballot_sync(0xffffffffu, rel);
            if (rel) s_list[warp][cnt + __popc(bits & lt_mask)] = (uint16_t)ci;
            cnt += __popc(bits);
        }
        __syncwarp();
        if (__any_sync(0xffffffffu, !done)) {
            for (int k0 = 0; k0 < cnt; k0 += 32) {
                s_hmask[warp][lane] = 0u;
                __syncwarp();
                // phase 1: one lane per candidate, over the warp's rows of its rectangle
                if (k0 + lane < cnt) {
                    const int j = s_list[warp][k0 + lane];
                    const uint2 rc = s_rect[j];
                    const float4 uv = s_uv[j];
                    const float s2 = s_s2[j];
                    const int xa = max((int)(rc.x & 0xffffu), tx0);
                    const int xb = min((int)(rc.x >> 16), tx0 + kTile - 1);
                    const int ya = max((int)(rc.y & 0xffffu), row0);
                    const int yb = min((int)(rc.y >> 16), row0 + 1);
                    for (int yy = ya; yy <= yb; ++yy) {
                        const float b = s_b[yy - ty0];
                        const float py = __fadd_rn(__int2float_rn(yy), 0.5f);
                        const float V = __fmul_rn(__fsub_rn(__fsub_rn(py, uv.z), uv.w), f.ify);
                        const float bb = __fmul_rn(b, b);
                        for (int xx = xa; xx <= xb; ++xx) {
                            // the decision test of the specification, term by term
                            const float a = s_a[xx - tx0];
                            const float px = __fadd_rn(__int2float_rn(xx), 0.5f);
                            const float U = __fmul_rn(__fsub_rn(__fsub_rn(px, uv.x), uv.y), f.ifx);
                            const float X = __fmaf_rn(U, b, -__fmul_rn(V, a));
                            const float Q = __fmaf_rn(U, U, __fmaf_rn(V, V, __fmul_rn(X, X)));
                            const float qq = __fadd_rn(__fadd_rn(1.0f, __fmul_rn(a, a)), bb);
                            if (Q < __fmul_rn(s2, qq))
                                atomicOr(&s_hmask[warp][(yy - row0) * kTile + (xx - tx0)],
                                         1u << lane);
                        }
                    }
                }
                __syncwarp();
                // phase 2: one lane per pixel, hits in candidate order
                uint32_t m = done ? 0u : s_hmask[warp][lane];
                while (m) {
                    const int j = s_list[warp][k0 + __ffs(m) - 1];
                    m &= m - 1;
                    const float4 uv = s_uv[j];
                    const float4 ex = s_ex[j];
                    const float2 ir2 = s_ir2[j];
                    // distance factor d = 1 - rho / r_eff in pair precision
                    float t;
                    const float d = distance_factor(uv, ir2.x, ir2.y, ray, pq, f, &t);
                    if (ex.x > mg || (ex.x == mg && ex.y > mgl)) {
                        const float sc = expf(__fsub_rn(mg, ex.x) + __fsub_rn(mgl, ex.y));
                        wsum *= sc;
#pragma unroll
                        for (int c = 0; c < CMAX; ++c) acc[c] *= sc;
                        mg = ex.x;
                        mgl = ex.y;
                    }
                    const float wt = ex.z * d * expf(__fsub_rn(ex.x, mg) + __fsub_rn(ex.y, mgl));
                    wsum += wt;
#pragma unroll
                    for (int c = 0; c < CMAX; ++c)
                        if (c < C) acc[c] += wt * s_feat[j * CMAX + c];
                    if (nh < f.n_track) {
#pragma unroll
                        for (int k = 0; k < TMAX; ++k)
                            if (k == nh) ids[k] = s_id[j];
                    }
                    ++nh;
                }
                __syncwarp();
            }
        }
        // early stop (allowed once n_track hits are tracked): every remaining
        // candidate has key >= s_next_key, hence z~ <= z~(key), o <= 1, d <= 1
        if (f.stop_tau > 0.0f && b0 + NB < end) {
            if (!done && nh >= f.n_track) {
                const float zt = fmaxf((f.zfar - s_next_key) * f.inv_zrange, 0.0f);
                const float rem = (float)(end - (b0 + NB));
                done = rem * expf(zt * f.inv_gamma - mg) <= f.stop_tau * wsum;
            }
            if (__syncthreads_and(done)) break;
        }
    }

    if (inside) {
        const int P = f.width * f.height;
        const int p = y * f.width + x;
        const float iw = 1.0f / wsum;
#pragma unroll
        for (int c = 0; c < CMAX; ++c)
            if (c < C) image[(size_t)p * C + c] = acc[c] * iw;
        // store the stabiliser's high part; fold its low part into the normaliser
        w.mg[p] = mg;
        w.wsum[p] = wsum * expf(mgl);
#pragma unroll
        for (int k = 0; k < TMAX; ++k)
            if (k < f.n_track) w.ids[(size_t)k * P + p] = ids[k];
        if (f.flags & 2u) w.nhits[p] = nh;
    }
    // hit count of the frame
    unsigned long long h = (unsigned long long)nh;
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) h += __shfl_down_sync(0xffffffffu, h, o);
    __syncthreads();
    if (lane == 0) atomicAdd(&s_hits, h);
    __syncthreads();
    if (tid == 0 && s_hits) atomicAdd(&w.state->hits, s_hits);
}

template <int CMAX, int TMAX>
void launch_t(const Frame& f, const Workspace& w, const float* features, const float* bg,
              float* image, cudaStream_t stream) {
    k_forward<CMAX, TMAX><<<f.n_tiles, kFwdThreads, 0, stream>>>(f, w, features, bg, image);
}

template <int CMAX>
void launch_c(const Frame& f, const Workspace& w, const float* features, const float* bg,
              float* image, cudaStream_t stream) {
    if (f.n_track <= 8) launch_t<CMAX, 8>(f, w, features, bg, image, stream);
    else launch_t<CMAX, kMaxTrack>(f, w, features, bg, image, stream);
}

}  // namespace

cudaError_t launch_forward(const Frame& f, const Workspace& w, const float* features,
                           const float* bg, float* image, int /*max_pairs_stride*/,
                           cudaStream_t stream) {
    if (f.channels <= 4) launch_c<4>(f, w, features, bg, image, stream);
    else if (f.channels <= 8) launch_c<8>(f, w, features, bg, image, stream);
    else if (f.channels <= 16) launch_c<16>(f, w, features, bg, image, stream);
    else if (f.channels <= 32) launch_c<32>(f, w, features, bg, image, stream);
    else launch_c<kMaxChannels>(f, w, features, bg, image, stream);
    return cudaGetLastError();
}

}  // namespace pulsar
