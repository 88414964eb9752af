// Forward pass (Pulsar Sec. B.1.2-B.1.4): one block per 16x16 tile; pixel
// parallel in the sense of the paper (no two threads ever write one pixel,
// Sec. B.1), but the work inside a warp is split in two phases so that the
// expensive part never runs with most lanes idle.
//
// The tile's sorted candidate list is staged through shared memory in
// batches (coalesced id read, one 64-byte record gather per candidate).  Each
// warp owns two pixel rows of the tile and first compacts, in list order, the
// batch's candidates whose pixel rectangle touches its rows (cooperative
// filtering at warp level).  Then, 32 candidates at a time:
//   phase 1 (flattened): the (candidate, pixel) pairs of the warp's rows
//           inside each candidate's rectangle are numbered by a warp prefix
//           sum and tested one per lane per round with the fp32 hit test; on
//           a hit the lane evaluates the distance factor in pair precision,
//           parks it in the warp's 32x32 d-matrix and sets the candidate's bit
//           in the pixel's hit mask;
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

// Shared-memory layout of one block (dynamic, 16-byte aligned pieces).
template <int CMAX>
struct FwdSmem {
    static constexpr int NB = CMAX <= 4 ? 128 : (CMAX <= 16 ? 64 : 32);   // batch
    static constexpr int dmat = 0;                                         // float [8][32][32]
    static constexpr int uv = dmat + kWarps * 32 * 32 * 4;                 // float4 [NB]
    static constexpr int ex = uv + NB * 16;                                // float4 [NB]
    static constexpr int ir2 = ex + NB * 16;                               // float2 [NB]
    static constexpr int rect = ir2 + NB * 8;                              // uint2 [NB]
    static constexpr int s2 = rect + NB * 8;                               // float [NB]
    static constexpr int id = s2 + NB * 4;                                 // int [NB]
    static constexpr int feat = id + NB * 4;                               // float [NB][CMAX]
    static constexpr int list = feat + NB * CMAX * 4;                      // u16 [8][NB]
    static constexpr int wmask = list + kWarps * NB * 2;                   // u8 [NB]
    static constexpr int hmask = (wmask + NB + 15) / 16 * 16;              // u32 [8][32]
    static constexpr int pqq = hmask + kWarps * 32 * 4;                    // float2 [256]
    static constexpr int piqq = pqq + kTilePix * 8;                        // float [256]
    static constexpr int ap = piqq + kTilePix * 4;                         // float2 [16]
    static constexpr int bp = ap + kTile * 8;                              // float2 [16]
    static constexpr int a = bp + kTile * 8;                               // float [16]
    static constexpr int b = a + kTile * 4;                                // float [16]
    static constexpr int misc = b + kTile * 4;                             // next key, hits
    static constexpr int bytes = misc + 16;
};

template <int CMAX, int TMAX>
__global__ void __launch_bounds__(kFwdThreads, CMAX <= 4 ? 4 : (CMAX <= 16 ? 2 : 1))
k_forward(Frame f, Workspace w, const float* __restrict__ features, const float* __restrict__ bg,
          float* __restrict__ image) {
    using L = FwdSmem<CMAX>;
    constexpr int NB = L::NB;
    extern __shared__ __align__(16) unsigned char smem[];
    float (*s_dmat)[32][32] = reinterpret_cast<float (*)[32][32]>(smem + L::dmat);
    float4* s_uv = reinterpret_cast<float4*>(smem + L::uv);
    float4* s_ex = reinterpret_cast<float4*>(smem + L::ex);    // exponent hi, lo, o, flags
    float2* s_ir2 = reinterpret_cast<float2*>(smem + L::ir2);
    uint2* s_rect = reinterpret_cast<uint2*>(smem + L::rect);
    float* s_s2 = reinterpret_cast<float*>(smem + L::s2);
    int* s_id = reinterpret_cast<int*>(smem + L::id);
    float* s_feat = reinterpret_cast<float*>(smem + L::feat);
    uint16_t (*s_list)[NB] = reinterpret_cast<uint16_t (*)[NB]>(smem + L::list);
    uint8_t* s_wmask = smem + L::wmask;
    uint32_t (*s_hmask)[32] = reinterpret_cast<uint32_t (*)[32]>(smem + L::hmask);
    float2* s_qq = reinterpret_cast<float2*>(smem + L::pqq);
    float* s_iqq = reinterpret_cast<float*>(smem + L::piqq);
    float2* s_ap = reinterpret_cast<float2*>(smem + L::ap);
    float2* s_bp = reinterpret_cast<float2*>(smem + L::bp);
    float* s_a = reinterpret_cast<float*>(smem + L::a);
    float* s_b = reinterpret_cast<float*>(smem + L::b);
    float* s_next_key = reinterpret_cast<float*>(smem + L::misc);
    unsigned long long* s_hits = reinterpret_cast<unsigned long long*>(smem + L::misc + 8);

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
    const uint32_t lt_mask = (1u << lane) - 1u;
    // per-tile ray constants: decision slopes (fp32) and value slopes (pairs)
    // of the 16 columns and 16 rows, |q|^2 of every pixel
    if (tid < kTile) {
        const float px = __fadd_rn(__int2float_rn(tx0 + tid), 0.5f);
        s_a[tid] = __fdiv_rn(__fsub_rn(px, f.cx), f.fx);
        const FPair ap = slope_pair(px, f.cx, f.ifx, f.ifx_lo);
        s_ap[tid] = make_float2(ap.hi, ap.lo);
    } else if (tid < 2 * kTile) {
        const int r = tid - kTile;
        const float py = __fadd_rn(__int2float_rn(ty0 + r), 0.5f);
        s_b[r] = __fdiv_rn(__fsub_rn(py, f.cy), f.fy);
        const FPair bp = slope_pair(py, f.cy, f.ify, f.ify_lo);
        s_bp[r] = make_float2(bp.hi, bp.lo);
    }
    {
        const float px = __fadd_rn(__int2float_rn(x), 0.5f);
        const float py = __fadd_rn(__int2float_rn(y), 0.5f);
        const PixelPairs pq = pixel_pairs(slope_pair(px, f.cx, f.ifx, f.ifx_lo),
                                          slope_pair(py, f.cy, f.ify, f.ify_lo));
        s_qq[tid] = make_float2(pq.qq.hi, pq.qq.lo);
        s_iqq[tid] = pq.iqq;
    }

    uint32_t start = w.tile_start[tile], end = w.tile_start[tile + 1];
    end = min(end, f.max_pairs);
    start = min(start, end);

    // running max of eps/gamma and o z~/gamma (log2 units), as a float pair
    float mg = f.eg_hi, mgl = f.eg_lo;
    float wsum = 1.0f;                   // 2^(eps/gamma - mg): background weight, shifted
    float acc[CMAX];
#pragma unroll
    for (int c = 0; c < CMAX; ++c) acc[c] = c < C ? bg[c] : 0.0f;
    const int P = f.width * f.height;
    const int p = inside ? y * f.width + x : 0;
    int nh = 0;
    bool done = !inside;
    if (tid == 0) *s_hits = 0ull;

    for (uint32_t b0 = start; b0 < end; b0 += NB) {
        __syncthreads();   // previous batch fully consumed (and the tile constants written)
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
            *s_next_key = nx < end ? __uint_as_float(w.rec[w.tile_ids[nx]].rk.w) : 0.0f;
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
                // phase 1: the chunk's (candidate, pixel) tests, flattened over the warp:
                // lane c describes candidate c's part of the warp's rows, a prefix sum
                // numbers the tests, and each lane takes one test per round
                int xa = 0, ya = 0, wd = 0, nt = 0, jc = 0;
                if (k0 + lane < cnt) {
                    jc = s_list[warp][k0 + lane];
                    const uint2 rc = s_rect[jc];
                    xa = max((int)(rc.x & 0xffffu), tx0);
                    ya = max((int)(rc.y & 0xffffu), row0);
                    const int xb = min((int)(rc.x >> 16), tx0 + kTile - 1);
                    const int yb = min((int)(rc.y >> 16), row0 + 1);
                    wd = xb - xa + 1;
                    nt = (wd > 0 && yb >= ya) ? wd * (yb - ya + 1) : 0;
                }
                int incl = nt;
#pragma unroll
                for (int o = 1; o < 32; o <<= 1) {
                    const int v = __shfl_up_sync(0xffffffffu, incl, o);
                    if (lane >= o) incl += v;
                }
                const int total = __shfl_sync(0xffffffffu, incl, 31);
                for (int t0 = 0; t0 < total; t0 += 32) {
                    const int t = t0 + lane;
                    int lo = 0, hi = 31;
#pragma unroll
                    for (int st = 0; st < 5; ++st) {
                        const int mid = (lo + hi) >> 1;
                        if (__shfl_sync(0xffffffffu, incl, mid) > t) hi = mid; else lo = mid + 1;
                    }
                    const int own = lo;
                    const int o_first = __shfl_sync(0xffffffffu, incl - nt, own);
                    const int o_xa = __shfl_sync(0xffffffffu, xa, own);
                    const int o_ya = __shfl_sync(0xffffffffu, ya, own);
                    const int o_wd = __shfl_sync(0xffffffffu, wd, own);
                    const int o_j = __shfl_sync(0xffffffffu, jc, own);
                    if (t < total) {
                        // at most two rows: test q of the owner is (q mod wd, q div wd)
                        const int q = t - o_first;
                        const int second = q >= o_wd ? 1 : 0;
                        const int xx = o_xa + q - second * o_wd;
                        const int yy = o_ya + second;
                        const float4 uv = s_uv[o_j];
                        // the decision test of the specification, term by term
                        const float a = s_a[xx - tx0];
                        const float b = s_b[yy - ty0];
                        const float px = __fadd_rn(__int2float_rn(xx), 0.5f);
                        const float py = __fadd_rn(__int2float_rn(yy), 0.5f);
                        const float U = __fmul_rn(__fsub_rn(__fsub_rn(px, uv.x), uv.y), f.ifx);
                        const float V = __fmul_rn(__fsub_rn(__fsub_rn(py, uv.z), uv.w), f.ify);
                        const float X = __fmaf_rn(U, b, -__fmul_rn(V, a));
                        const float Q = __fmaf_rn(U, U, __fmaf_rn(V, V, __fmul_rn(X, X)));
                        const float qq = __fadd_rn(__fadd_rn(1.0f, __fmul_rn(a, a)), __fmul_rn(b, b));
                        if (Q < __fmul_rn(s_s2[o_j], qq)) {
                            const int pl = (yy - ty0) * kTile + (xx - tx0);   // pixel in tile
                            const int pw = (yy - row0) * kTile + (xx - tx0);  // pixel in warp
                            const float2 apv = s_ap[xx - tx0];
                            const float2 bpv = s_bp[yy - ty0];
                            const float2 qqv = s_qq[pl];
                            const float2 ir2 = s_ir2[o_j];
                            PixelPairs pq;
                            pq.a = {apv.x, apv.y};
                            pq.b = {bpv.x, bpv.y};
                            pq.qq = {qqv.x, qqv.y};
                            pq.iqq = s_iqq[pl];
                            s_dmat[warp][pw][own ^ pw] =
                                distance_factor(uv, ir2.x, ir2.y, px, py, pq, f);
                            atomicOr(&s_hmask[warp][pw], 1u << own);
                        }
                    }
                }
                __syncwarp();
                // phase 2: one lane per pixel, hits in candidate order
                uint32_t m = done ? 0u : s_hmask[warp][lane];
                while (m) {
                    const int bit = __ffs(m) - 1;
                    m &= m - 1;
                    const int j = s_list[warp][k0 + bit];
                    const float d = s_dmat[warp][lane][bit ^ lane];
                    const float4 ex = s_ex[j];
                    if (ex.x > mg || (ex.x == mg && ex.y > mgl)) {
                        const float sc = exp2f(__fsub_rn(mg, ex.x) + __fsub_rn(mgl, ex.y));
                        wsum *= sc;
#pragma unroll
                        for (int c = 0; c < CMAX; ++c) acc[c] *= sc;
                        mg = ex.x;
                        mgl = ex.y;
                    }
                    const float wt = ex.z * d * exp2f(__fsub_rn(ex.x, mg) + __fsub_rn(ex.y, mgl));
                    wsum += wt;
#pragma unroll
                    for (int c = 0; c < CMAX; ++c)
                        if (c < C) acc[c] += wt * s_feat[j * CMAX + c];
                    if (nh < f.n_track) {
                        // backward-information buffer: the hit's position in the tile
                        // list and its distance factor
                        w.ids[(size_t)nh * P + p] = (int)(b0 - start) + j;
                        w.dtr[(size_t)nh * P + p] = d;
                    }
                    ++nh;
                }
                __syncwarp();
            }
        }
        // early stop (allowed once n_track hits are tracked): every remaining
        // candidate has key >= the next key, hence z~ <= z~(key), o <= 1, d <= 1
        if (f.stop_tau > 0.0f && b0 + NB < end) {
            if (!done && nh >= f.n_track) {
                const float zt = fmaxf((f.zfar - *s_next_key) * f.inv_zrange, 0.0f);
                const float rem = (float)(end - (b0 + NB));
                done = rem * exp2f(zt * f.inv_gamma * 1.44269504f - mg) <= f.stop_tau * wsum;
            }
            if (__syncthreads_and(done)) break;
        }
    }

    if (inside) {
        const float iw = 1.0f / wsum;
#pragma unroll
        for (int c = 0; c < CMAX; ++c)
            if (c < C) image[(size_t)p * C + c] = acc[c] * iw;
        // store the stabiliser's high part; fold its low part into the normaliser
        w.mg[p] = mg;
        w.wsum[p] = wsum * exp2f(mgl);
        for (int k = nh; k < f.n_track; ++k) w.ids[(size_t)k * P + p] = -1;
        if (f.flags & 2u) w.nhits[p] = nh;
    }
    // hit count of the frame
    unsigned long long h = (unsigned long long)nh;
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) h += __shfl_down_sync(0xffffffffu, h, o);
    __syncthreads();
    if (lane == 0) atomicAdd(s_hits, h);
    __syncthreads();
    if (tid == 0 && *s_hits) atomicAdd(&w.state->hits, *s_hits);
}

template <int CMAX, int TMAX>
cudaError_t launch_t(const Frame& f, const Workspace& w, const float* features, const float* bg,
                     float* image, cudaStream_t stream) {
    constexpr int bytes = FwdSmem<CMAX>::bytes;
    k_forward<CMAX, TMAX><<<f.n_tiles, kFwdThreads, bytes, stream>>>(f, w, features, bg, image);
    return cudaGetLastError();
}

template <int CMAX, int TMAX>
cudaError_t prepare_t() {
    return cudaFuncSetAttribute(k_forward<CMAX, TMAX>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                FwdSmem<CMAX>::bytes);
}

template <int CMAX>
cudaError_t launch_c(const Frame& f, const Workspace& w, const float* features, const float* bg,
                     float* image, cudaStream_t stream) {
    if (f.n_track <= 8) return launch_t<CMAX, 8>(f, w, features, bg, image, stream);
    return launch_t<CMAX, kMaxTrack>(f, w, features, bg, image, stream);
}

template <int CMAX>
cudaError_t prepare_c() {
    const cudaError_t e = prepare_t<CMAX, 8>();
    return e != cudaSuccess ? e : prepare_t<CMAX, kMaxTrack>();
}

}  // namespace

cudaError_t prepare_forward() {
    cudaError_t e = prepare_c<4>();
    if (e == cudaSuccess) e = prepare_c<8>();
    if (e == cudaSuccess) e = prepare_c<16>();
    if (e == cudaSuccess) e = prepare_c<32>();
    if (e == cudaSuccess) e = prepare_c<kMaxChannels>();
    return e;
}

cudaError_t launch_forward(const Frame& f, const Workspace& w, const float* features,
                           const float* bg, float* image, int /*max_pairs_stride*/,
                           cudaStream_t stream) {
    if (f.channels <= 4) return launch_c<4>(f, w, features, bg, image, stream);
    if (f.channels <= 8) return launch_c<8>(f, w, features, bg, image, stream);
    if (f.channels <= 16) return launch_c<16>(f, w, features, bg, image, stream);
    if (f.channels <= 32) return launch_c<32>(f, w, features, bg, image, stream);
    return launch_c<kMaxChannels>(f, w, features, bg, image, stream);
}

}  // namespace pulsar
