// Forward pass (Pulsar Sec. B.1.2-B.1.4): one block per 16x16 tile, one
// thread per pixel (pixel-parallel, so no two threads write one pixel;
// Pulsar Sec. B.1).
//
// The tile's sorted candidate list is staged through shared memory in
// batches of 256: each thread loads one candidate's records and features
// (coalesced id read, 16-byte record gathers) and computes which warps --
// two pixel rows each -- its pixel rectangle overlaps.  Each warp then walks
// only the candidates that touch its rows, found 32 at a time with a ballot
// (cooperative filtering at warp level), and every lane runs the hit test
// for its pixel.  On a hit the lane updates a max-shifted running blend
// (online rescale when a larger o*z~/gamma arrives), records the id if fewer
// than n_track hits are tracked, and counts the hit.  Between batches the
// block votes on the early-stop bound (Pulsar Sec. 3.2, Fig. 3; B.1.3).
// The pixel's result and its backward-information buffer (tracked ids,
// stabiliser, normaliser; Sec. B.1.4) are written at the end.
#include "pulsar_internal.cuh"

namespace pulsar {
namespace {

constexpr int kFwdThreads = kTilePix;

// candidates staged per batch: 256, fewer for wide payloads (static smem < 48 KB)
template <int CMAX>
struct Batch {
    static constexpr int n = CMAX <= 16 ? kFwdThreads : 8192 / CMAX;
};

template <int CMAX, int TMAX>
__global__ void __launch_bounds__(kFwdThreads)
k_forward(Frame f, Workspace w, const float* __restrict__ features, const float* __restrict__ bg,
          float* __restrict__ image) {
    constexpr int NB = Batch<CMAX>::n;
    __shared__ float4 s_uv[NB];
    __shared__ float4 s_r1[NB];
    __shared__ float2 s_ir2[NB];
    __shared__ uint2 s_rect[NB];
    __shared__ int s_id[NB];
    __shared__ uint32_t s_wmask[NB];
    __shared__ float s_feat[NB * CMAX];
    __shared__ float s_next_key;
    __shared__ unsigned long long s_hits;

    // a frame whose pairs overflowed max_pairs has unsorted lists: render nothing
    // (the capacity error is latched and reported by pulsar_status)
    if (w.state->n_pairs > f.max_pairs) return;
    const int C = f.channels;
    const int tile = blockIdx.x;
    const int tyi = tile / f.tiles_x, txi = tile - tyi * f.tiles_x;
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int x = txi * kTile + (tid & 15), y = tyi * kTile + (tid >> 4);
    const bool inside = x < f.width && y < f.height;
    const PixelRay ray = pixel_ray(x, y, f);
    const PixelPairs pq = pixel_pairs(ray, f);

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
            const uint2 rc = w.rect[id];
            s_id[tid] = id;
            s_uv[tid] = w.rec0[id];
            s_r1[tid] = w.rec1[id];
            s_ir2[tid] = reinterpret_cast<const float2*>(w.rec2)[2 * id];
            s_rect[tid] = rc;
            const int r0 = max((int)(rc.y & 0xffffu) - tyi * kTile, 0);
            const int r1 = min((int)(rc.y >> 16) - tyi * kTile, kTile - 1);
            s_wmask[tid] = (0xffu << (r0 >> 1)) & (0xffu >> (7 - (r1 >> 1)));
#pragma unroll
            for (int c = 0; c < CMAX; ++c)
                if (c < C) s_feat[tid * CMAX + c] = features[(size_t)id * C + c];
        }
        if (tid == 0) {
            const uint32_t nx = b0 + NB;
            s_next_key = nx < end ? w.key[w.tile_ids[nx]] : 0.0f;
        }
        __syncthreads();
        const int nb = (int)min((uint32_t)NB, end - b0);
        if (__any_sync(0xffffffffu, !done)) {
            for (int c0 = 0; c0 < nb; c0 += 32) {
                const int ci = c0 + lane;
                uint32_t bits = __ballot_sync(0xffffffffu, ci < nb && ((s_wmask[ci] >> warp) & 1u));
                while (bits) {
                    const int j = c0 + __ffs(bits) - 1;
                    bits &= bits - 1;
                    if (done || !rect_contains(s_rect[j], x, y)) continue;
                    const float4 uv = s_uv[j];
                    const float4 r1 = s_r1[j];
                    float U, V;
                    const float Q = ray_offset_q(uv, ray, f.ifx, f.ify, &U, &V);
                    if (!(Q < __fmul_rn(r1.x, ray.qq))) continue;
                    // hit: distance factor d = 1 - rho / r_eff in pair precision
                    const float2 ir2 = s_ir2[j];
                    float t;
                    const float d = distance_factor(uv, ir2.x, ir2.y, ray, pq, f, &t);
                    if (r1.y > mg || (r1.y == mg && r1.z > mgl)) {
                        const float sc = expf(__fsub_rn(mg, r1.y) + __fsub_rn(mgl, r1.z));
                        wsum *= sc;
#pragma unroll
                        for (int c = 0; c < CMAX; ++c) acc[c] *= sc;
                        mg = r1.y;
                        mgl = r1.z;
                    }
                    const float wt = r1.w * d * expf(__fsub_rn(r1.y, mg) + __fsub_rn(r1.z, mgl));
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
