// Forward pass (Pulsar Sec. B.1.2-B.1.4): one block per 16x16 tile, one
// thread per pixel; pixel parallel in the sense of the paper (no two threads
// ever write one pixel, Sec. B.1), with the work of a warp split in two
// phases so that the expensive part never runs with most lanes idle.
//
// The tile's sorted candidate list streams through shared memory in batches
// of NB candidates, double buffered: while the warps work on batch i, the
// 64-byte records and features of batch i+1 are already being copied by
// cp.async (the ids of batch i+2 are read meanwhile), so one block barrier
// per batch is all the synchronisation there is.  Each warp owns two pixel
// rows of the tile and compacts, in list order, the batch's candidates whose
// pixel rectangle touches its rows (cooperative filtering at warp level).
// Then, a chunk of at most 32 candidates and kTestCap tests at a time:
//   phase 1 (flattened): the (candidate, pixel) tests of the chunk -- the
//           pixels of the warp's rows inside each candidate's rectangle --
//           are numbered by a warp prefix sum and taken one per lane per
//           round with the fp32 hit test; on a hit the lane evaluates the
//           distance factor in pair precision, stores it under the test's
//           number and sets the candidate's bit in the pixel's hit mask;
//   phase 2 (one lane per pixel): the lane walks its mask bits in increasing
//           order -- list order, i.e. earliest possible intersection first --
//           finds each hit's test number from the candidate's rectangle, and
//           blends the hit into its max-shifted running sums, recording the
//           first n_track hits.
// At each batch barrier the block votes on the early-stop bound (Sec. 3.2,
// Fig. 3; B.1.3).  The pixel's result and its backward-information buffer
// (tracked list positions and distance factors, stabiliser, normaliser; Sec.
// B.1.4) are written at the end.
#include "pulsar_internal.cuh"

namespace pulsar {
namespace {

constexpr int kFwdThreads = kTilePix;
constexpr int kWarps = kFwdThreads / 32;
constexpr int kTestCap = 256;     // tests per chunk: entries of a warp's d buffer
// The fp32 decision test of the specification, term by term: pixel centre
// (px, py) with ray slopes (a, b) and qq = 1 + a^2 + b^2 (formed by the caller
// as fp32 ops in that order) against a candidate's projected centre uv and
// s2 = (r_eff / c.z)^2.
__device__ __forceinline__ bool hit_test32(const float4& uv, float s2, float px, float py, float a,
                                           float b, float qq, const Frame& f) {
    const float U = __fmul_rn(__fsub_rn(__fsub_rn(px, uv.x), uv.y), f.ifx);
    const float V = __fmul_rn(__fsub_rn(__fsub_rn(py, uv.z), uv.w), f.ify);
    const float X = __fmaf_rn(U, b, -__fmul_rn(V, a));
    const float Q = __fmaf_rn(U, U, __fmaf_rn(V, V, __fmul_rn(X, X)));
    return Q < __fmul_rn(s2, qq);
}

__device__ __forceinline__ float qq32(float a, float b) {
    return __fadd_rn(__fadd_rn(1.0f, __fmul_rn(a, a)), __fmul_rn(b, b));
}

// Shared-memory layout of one block (dynamic, 16-byte aligned pieces).
// Candidates per batch: 192; 128 for 8-16 channels, whose feature rows
// would otherwise keep the block's shared memory above a quarter of the SM's
// (four blocks per SM measured 4% faster than three with the larger batch).
template <int CMAX>
struct FwdSmem {
    static constexpr int NB = CMAX >= 8 && CMAX <= 16 ? 128 : 192;
    static constexpr bool kStageFeat = CMAX <= 16;   // wider features are read from global
    static constexpr int FS = kStageFeat ? CMAX : 0;
    // features of 8 and 16 channels are staged and read 16 bytes at a time
    // (one cp.async and one 128-bit load per four channels) when the caller's
    // rows allow it
    static constexpr bool kVecFeat = kStageFeat && CMAX >= 8 && CMAX % 4 == 0;
    // feature row stride in words: 16-byte rows padded by four words for the
    // vector form (8 rows of a quarter-warp then fall on distinct bank groups
    // when their candidates are consecutive); otherwise odd, so that lanes
    // reading different candidates' rows hit different banks (16 floats per
    // row would put 32 lanes on two banks)
    static constexpr int FSP = kStageFeat ? (kVecFeat ? CMAX + 4 : (CMAX | 1)) : 0;
    // two batch buffers, each: uv, ex, geo, rk (float4 / uint4 [NB]) of the
    // record, then features float [NB][FSP] and ids int [NB]
    static constexpr int rec_uv = 0;
    static constexpr int rec_ex = NB * 16;
    static constexpr int rec_geo = 2 * NB * 16;
    static constexpr int rec_rk = 3 * NB * 16;
    static constexpr int rec_feat = 4 * NB * 16;
    static constexpr int rec_id = rec_feat + NB * FSP * 4;
    static constexpr int buf_bytes = rec_id + NB * 4;
    static constexpr int list = 2 * buf_bytes;                       // u16 [8][NB]
    static constexpr int dbuf = list + kWarps * NB * 2;              // float [8][kTestCap]
    static constexpr int desc = dbuf + kWarps * kTestCap * 4;        // u32 [8][32]
    static constexpr int hmask = desc + kWarps * 32 * 4;             // u32 [8][32]
    static constexpr int pqq = hmask + kWarps * 32 * 4;              // float2 [256]
    static constexpr int piqq = pqq + kTilePix * 8;                  // float [256]
    static constexpr int ap = piqq + kTilePix * 4;                   // float2 [16]
    static constexpr int bp = ap + kTile * 8;                        // float2 [16]
    static constexpr int a = bp + kTile * 8;                         // float [16]
    static constexpr int b = a + kTile * 4;                          // float [16]
    static constexpr int misc = b + kTile * 4;                       // hit counter
    static constexpr int bytes = misc + 16;
};

template <int CMAX, bool MULTI>
__global__ void __launch_bounds__(kFwdThreads, CMAX <= 16 ? 4 : 1)
k_forward(Frames fs, Workspace w, const float* __restrict__ features, const float* __restrict__ bg,
          float* __restrict__ image) {
    pdl_begin();
    // the frame's pair count and the tile's list bounds, loaded together
    // ahead of the set-up below, which hides their latency
    const uint32_t n_pairs = w.state->n_pairs;
    uint32_t start = w.tile_start[blockIdx.x], end = w.tile_start[blockIdx.x + 1];
    // zero the backward's accumulators of this frame on the way (plain
    // coalesced stores that never wait: this kernel is bound by its own
    // instruction stream and latencies, so they cost next to nothing here,
    // against a separate memset pass before the backward)
    if (w.gacc) {
        const Frame& f0 = fs.f[0];
        const size_t nk = (size_t)f0.n * (size_t)f0.n_cams;
        const size_t stride = (size_t)gridDim.x * blockDim.x;
        const size_t i0 = (size_t)blockIdx.x * blockDim.x + threadIdx.x;
        const float4 z4 = make_float4(0.f, 0.f, 0.f, 0.f);
        for (size_t i = i0; i < nk; i += stride) w.gacc[i] = z4;
        for (size_t i = i0; i < (size_t)f0.n; i += stride) w.gacc2[i] = z4;
        if (f0.flags & kParamNormalize)
            for (size_t i = i0; i < nk; i += stride) w.hitcnt[i] = 0.0f;
    }
    using L = FwdSmem<CMAX>;
    constexpr int NB = L::NB;
    constexpr int FS = L::FS;
    constexpr int FSP = L::FSP;
    extern __shared__ __align__(16) unsigned char smem[];
    uint16_t (*s_list)[NB] = reinterpret_cast<uint16_t (*)[NB]>(smem + L::list);
    float (*s_dbuf)[kTestCap] = reinterpret_cast<float (*)[kTestCap]>(smem + L::dbuf);
    uint32_t (*s_desc)[32] = reinterpret_cast<uint32_t (*)[32]>(smem + L::desc);
    uint32_t (*s_hmask)[32] = reinterpret_cast<uint32_t (*)[32]>(smem + L::hmask);
    float2* s_qq = reinterpret_cast<float2*>(smem + L::pqq);
    float* s_iqq = reinterpret_cast<float*>(smem + L::piqq);
    float2* s_ap = reinterpret_cast<float2*>(smem + L::ap);
    float2* s_bp = reinterpret_cast<float2*>(smem + L::bp);
    float* s_a = reinterpret_cast<float*>(smem + L::a);
    float* s_b = reinterpret_cast<float*>(smem + L::b);
    unsigned long long* s_hits = reinterpret_cast<unsigned long long*>(smem + L::misc);

    // the block's camera and its tile in that camera's image (a single camera
    // is indexed statically, so its constants stay instruction operands)
    const int tile_g = blockIdx.x;
    const int cam = MULTI ? tile_g / fs.f[0].n_tiles : 0;
    const Frame& f = fs.f[MULTI ? cam : 0];
    const int tile = tile_g - cam * f.n_tiles;
    end = min(end, f.max_pairs);
    start = min(start, end);
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    // the ids of the first two batches (a read of the list is in bounds even
    // for an overflowed frame; its ids are used only after the check below)
    const int id_first = (tid < NB && start + tid < end) ? (int)w.tile_ids[start + tid] : -1;
    int id_next = (tid < NB && start + NB + tid < end) ? (int)w.tile_ids[start + NB + tid] : -1;
    const int C = f.channels;
    const int tyi = tile / f.tiles_x, txi = tile - tyi * f.tiles_x;
    const int tx0 = txi * kTile, ty0 = tyi * kTile;
    const int x = tx0 + (tid & 15), y = ty0 + (tid >> 4);
    const int row0 = ty0 + 2 * warp;              // the warp's two pixel rows
    const bool inside = x < f.width && y < f.height;
    const uint32_t lt_mask = (1u << lane) - 1u;
    // per-tile ray constants: decision slopes (fp32) and value slopes (pairs)
    // of the 16 columns and 16 rows, |q|^2 of every pixel
    // (orthographic rays are parallel: all slopes are 0)
    if (tid < kTile) {
        const float px = __fadd_rn(__int2float_rn(tx0 + tid), 0.5f);
        s_a[tid] = f.ortho ? 0.0f : __fdiv_rn(__fsub_rn(px, f.cx), f.fx);
        const FPair ap = f.ortho ? FPair{0.0f, 0.0f} : slope_pair(px, f.cx, f.ifx, f.ifx_lo);
        s_ap[tid] = make_float2(ap.hi, ap.lo);
    } else if (tid < 2 * kTile) {
        const int r = tid - kTile;
        const float py = __fadd_rn(__int2float_rn(ty0 + r), 0.5f);
        s_b[r] = f.ortho ? 0.0f : __fdiv_rn(__fsub_rn(py, f.cy), f.fy);
        const FPair bp = f.ortho ? FPair{0.0f, 0.0f} : slope_pair(py, f.cy, f.ify, f.ify_lo);
        s_bp[r] = make_float2(bp.hi, bp.lo);
    }
    {
        const float px = __fadd_rn(__int2float_rn(x), 0.5f);
        const float py = __fadd_rn(__int2float_rn(y), 0.5f);
        const FPair zero = {0.0f, 0.0f};
        const PixelPairs pq =
            pixel_pairs(f.ortho ? zero : slope_pair(px, f.cx, f.ifx, f.ifx_lo),
                        f.ortho ? zero : slope_pair(py, f.cy, f.ify, f.ify_lo));
        s_qq[tid] = make_float2(pq.qq.hi, pq.qq.lo);
        s_iqq[tid] = pq.iqq;
    }
    if (tid == 0) *s_hits = 0ull;
    // a frame whose pairs overflowed max_pairs has unsorted lists: render nothing
    // (the capacity error is latched and reported by pulsar_status)
    if (n_pairs > f.max_pairs) return;

    const SphereRec* __restrict__ rec = w.rec + f.rec_base;   // this camera's records

    // 16-byte feature copies and loads: every row is whole (C == CMAX) and
    // 16-byte aligned
    const bool fvec = L::kVecFeat && C == CMAX &&
                      (reinterpret_cast<uintptr_t>(features) & 15u) == 0;
    // thread t < NB stages candidate t of every batch: the record's four
    // 16-byte pieces and the features by cp.async, the id by a plain store
    auto stage = [&](int buf, int id) {
        unsigned char* B = smem + buf * L::buf_bytes;
        if (!PULSAR_CHECK(w.state, (uint32_t)id < (uint32_t)f.n)) id = 0;
        const float4* src = reinterpret_cast<const float4*>(rec + id);
        cp_async16(B + L::rec_uv + tid * 16, src + 0);
        cp_async16(B + L::rec_ex + tid * 16, src + 1);
        cp_async16(B + L::rec_geo + tid * 16, src + 2);
        cp_async16(B + L::rec_rk + tid * 16, src + 3);
        if (L::kStageFeat) {
            if (fvec) {
#pragma unroll
                for (int q = 0; q < FS / 4; ++q)
                    cp_async16(B + L::rec_feat + (tid * FSP + 4 * q) * 4,
                               features + (size_t)id * FS + 4 * q);
            } else {
#pragma unroll
                for (int c = 0; c < FS; ++c)
                    if (c < C)
                        cp_async4(B + L::rec_feat + (tid * FSP + c) * 4, features + (size_t)id * C + c);
            }
        }
        reinterpret_cast<int*>(B + L::rec_id)[tid] = id;
    };
    if (id_first >= 0) stage(0, id_first);
    cp_async_commit();

    // running max of eps/gamma and o z~/gamma (log2 units), as a float pair
    float mg = f.eg_hi, mgl = f.eg_lo;
    float wsum = 1.0f;                   // 2^(eps/gamma - mg): background weight, shifted
    float acc[CMAX];
#pragma unroll
    for (int c = 0; c < CMAX; ++c) acc[c] = c < C ? bg[c] : 0.0f;
    // the pixel in the batch's buffers; planes of ids / d are pix_all apart
    const uint32_t P = f.pix_all;
    const uint32_t p = f.pix_base + (uint32_t)(inside ? y * f.width + x : 0);
    int nh = 0;
    bool done = !inside;
    const int lx = lane & 15, ly = lane >> 4;     // the lane's pixel within the warp's rows
    const bool gaussian = (f.flags & kParamGaussian) != 0;

    // blend hit j of the current batch (record in shared memory, distance
    // factor d) into the pixel's max-shifted running sums; the first n_track
    // hits go to the backward-information buffer
    auto blend = [&](const unsigned char* B, int j, float d, uint32_t list_pos) {
        const float4 ex = reinterpret_cast<const float4*>(B + L::rec_ex)[j];
        if (ex.x > mg || (ex.x == mg && ex.y > mgl)) {
            const float sc = ex2_approx(__fsub_rn(mg, ex.x) + __fsub_rn(mgl, ex.y));
            wsum *= sc;
#pragma unroll
            for (int cc = 0; cc < CMAX; ++cc) acc[cc] *= sc;
            mg = ex.x;
            mgl = ex.y;
        }
        const float wt = ex.z * d * ex2_approx(__fsub_rn(ex.x, mg) + __fsub_rn(ex.y, mgl));
        wsum += wt;
        if (L::kStageFeat) {
            const float* s_feat = reinterpret_cast<const float*>(B + L::rec_feat);
            if (L::kVecFeat && fvec) {
#pragma unroll
                for (int q = 0; q < CMAX / 4; ++q) {
                    const float4 fq = *reinterpret_cast<const float4*>(s_feat + j * FSP + 4 * q);
                    acc[4 * q] += wt * fq.x;
                    acc[4 * q + 1] += wt * fq.y;
                    acc[4 * q + 2] += wt * fq.z;
                    acc[4 * q + 3] += wt * fq.w;
                }
            } else {
#pragma unroll
                for (int cc = 0; cc < CMAX; ++cc)
                    if (cc < C) acc[cc] += wt * s_feat[j * FSP + cc];
            }
        } else {
            const float* fp = features + (size_t)reinterpret_cast<const int*>(B + L::rec_id)[j] * C;
#pragma unroll
            for (int cc = 0; cc < CMAX; ++cc)
                if (cc < C) acc[cc] += wt * __ldg(fp + cc);
        }
        if (nh < f.n_track) {
            // backward-information buffer: the hit's position in the tile list
            // and its distance factor
            w.ids[(uint32_t)nh * P + p] = (int)list_pos;
            w.dtr[(uint32_t)nh * P + p] = d;
        }
        ++nh;
    };

    int buf = 0;
    for (uint32_t b0 = start; b0 < end; b0 += NB, buf ^= 1) {
        cp_async_wait_all();
        // batch b0 has landed everywhere, the previous batch is fully consumed
        // (so its buffer may be refilled), and the tile constants are written;
        // the vote ends the tile once every pixel has stopped
        if (__syncthreads_and(done)) break;
        if (b0 + NB < end) {
            if (id_next >= 0) stage(buf ^ 1, id_next);
            cp_async_commit();
            const uint32_t k2 = b0 + 2 * NB + tid;
            id_next = (tid < NB && k2 < end) ? (int)w.tile_ids[k2] : -1;
        }
        const unsigned char* B = smem + buf * L::buf_bytes;
        const float4* s_uv = reinterpret_cast<const float4*>(B + L::rec_uv);
        const float4* s_ex = reinterpret_cast<const float4*>(B + L::rec_ex);
        const float4* s_geo = reinterpret_cast<const float4*>(B + L::rec_geo);
        const uint4* s_rk = reinterpret_cast<const uint4*>(B + L::rec_rk);
        const int nb = (int)min((uint32_t)NB, end - b0);

        // compact this warp's candidates, in list order
        int cnt = 0;
        for (int g0 = 0; g0 < nb; g0 += 32) {
            const int ci = g0 + lane;
            bool rel = false;
            if (ci < nb) {
                const uint2 rc = *reinterpret_cast<const uint2*>(&s_rk[ci]);
                // the rectangle clipped to the tile's columns and the warp's rows
                // is not empty (exactly when the chunk code below finds nt > 0)
                rel = max((int)(rc.x & 0xffffu), tx0) <= min((int)(rc.x >> 16), tx0 + kTile - 1) &&
                      max((int)(rc.y & 0xffffu), row0) <= min((int)(rc.y >> 16), row0 + 1);
            }
            const uint32_t bits = __ballot_sync(0xffffffffu, rel);
            if (rel) s_list[warp][cnt + __popc(bits & lt_mask)] = (uint16_t)ci;
            cnt += __popc(bits);
        }
        __syncwarp();
        if (__any_sync(0xffffffffu, !done)) {
            for (int k0 = 0; k0 < cnt;) {
                // lane c describes list entry k0 + c: its part of the warp's rows
                // (columns xa.., rows ya.., width wd, nt tests)
                int xa = 0, ya = 0, wd = 0, nt = 0;
                if (k0 + lane < cnt) {
                    const uint2 rc = *reinterpret_cast<const uint2*>(&s_rk[s_list[warp][k0 + lane]]);
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
                // the chunk: the longest prefix with at most kTestCap tests (one
                // candidate has at most 32, so the chunk is never empty)
                const int nc = __popc(__ballot_sync(0xffffffffu, k0 + lane < cnt && incl <= kTestCap));
                if (lane >= nc) nt = 0;
                const int total = __shfl_sync(0xffffffffu, incl, nc - 1);
                const int first = incl - nt;
                if (lane < nc)
                    s_desc[warp][lane] = (uint32_t)first | (uint32_t)(xa - tx0) << 9 |
                                         (uint32_t)(ya - row0) << 13 | (uint32_t)wd << 14;
                s_hmask[warp][lane] = 0u;
                __syncwarp();
                // phase 1: each lane takes one test per round and finds its
                // candidate by counting the candidates that start at or before it
                for (int t0 = 0; t0 < total; t0 += 32) {
                    const int rel = first - t0;
                    const bool starts_here = nt > 0 && rel >= 0 && rel < 32;
                    const uint32_t sb = __reduce_or_sync(0xffffffffu, starts_here ? 1u << rel : 0u);
                    const int before = __popc(__ballot_sync(0xffffffffu, nt > 0 && rel < 0));
                    const int own = max(before - 1 + __popc(sb & (0xffffffffu >> (31 - lane))), 0);
                    const int o_first = __shfl_sync(0xffffffffu, first, own);
                    const int o_xa = __shfl_sync(0xffffffffu, xa, own);
                    const int o_ya = __shfl_sync(0xffffffffu, ya, own);
                    const int o_wd = __shfl_sync(0xffffffffu, wd, own);
                    const int t = t0 + lane;
                    if (t < total) {
                        // at most two rows: test q of the owner is (q mod wd, q div wd)
                        const int j = s_list[warp][k0 + own];
                        const int q = t - o_first;
                        const int second = q >= o_wd ? 1 : 0;
                        const int xx = o_xa + q - second * o_wd;
                        const int yy = o_ya + second;
                        const float4 uv = s_uv[j];
                        const float a = s_a[xx - tx0];
                        const float b = s_b[yy - ty0];
                        const float px = __fadd_rn(__int2float_rn(xx), 0.5f);
                        const float py = __fadd_rn(__int2float_rn(yy), 0.5f);
                        if (hit_test32(uv, __uint_as_float(s_rk[j].z), px, py, a, b, qq32(a, b), f)) {
                            const int pl = (yy - ty0) * kTile + (xx - tx0);   // pixel in tile
                            const float2 apv = s_ap[xx - tx0];
                            const float2 bpv = s_bp[yy - ty0];
                            const float2 qqv = s_qq[pl];
                            const float4 geo = s_geo[j];
                            PixelPairs pq;
                            pq.a = {apv.x, apv.y};
                            pq.b = {bpv.x, bpv.y};
                            pq.qq = {qqv.x, qqv.y};
                            pq.iqq = s_iqq[pl];
                            s_dbuf[warp][t] = distance_factor(uv, geo.x, geo.y, px, py, pq, f,
                                                              gaussian);
                            atomicOr(&s_hmask[warp][(yy - row0) * kTile + (xx - tx0)], 1u << own);
                        }
                    }
                }
                __syncwarp();
                // phase 2: one lane per pixel, hits in list order
                uint32_t m = done ? 0u : s_hmask[warp][lane];
                while (m) {
                    const int c = __ffs(m) - 1;
                    m &= m - 1;
                    const uint32_t dc = s_desc[warp][c];
                    const int ti = (int)(dc & 511u) + (ly - (int)((dc >> 13) & 1u)) * (int)(dc >> 14) +
                                   (lx - (int)((dc >> 9) & 15u));
                    const int j = s_list[warp][k0 + c];
                    blend(B, j, s_dbuf[warp][ti], (b0 - start) + (uint32_t)j);
                }
                __syncwarp();   // the chunk's descriptors, masks and d buffer are free
                k0 += nc;
            }
        }
        // early stop (allowed once n_track hits are tracked): every remaining
        // candidate comes later in the list, so its key is >= the key of this
        // batch's last candidate: z~ <= z~(key), o <= 1, d <= 1
        if (f.stop_tau > 0.0f && b0 + NB < end && !done && nh >= f.n_track) {
            const float key = __uint_as_float(s_rk[nb - 1].w);
            const float zt = fmaxf((f.zfar - key) * f.inv_zrange, 0.0f);
            const float rem = (float)(end - (b0 + NB));
            done = rem * ex2_approx(zt * f.inv_gamma * 1.44269504f - mg) <= f.stop_tau * wsum;
        }
    }
    cp_async_wait_all();   // nothing may be in flight when the block ends

    if (inside) {
        const float iw = 1.0f / wsum;
        if (CMAX % 4 == 0 && C == CMAX && (reinterpret_cast<uintptr_t>(image) & 15u) == 0) {
            // whole 16-byte-aligned rows: 16-byte stores
            float4* o4 = reinterpret_cast<float4*>(image + (size_t)p * CMAX);
#pragma unroll
            for (int q = 0; q < CMAX / 4; ++q)
                o4[q] = make_float4(acc[4 * q] * iw, acc[4 * q + 1] * iw, acc[4 * q + 2] * iw,
                                    acc[4 * q + 3] * iw);
        } else {
#pragma unroll
            for (int c = 0; c < CMAX; ++c)
                if (c < C) image[(size_t)p * C + c] = acc[c] * iw;
        }
        // store the stabiliser's high part; fold its low part into the normaliser
        w.mg[p] = mg;
        w.wsum[p] = wsum * ex2_approx(mgl);
        for (int k = nh; k < f.n_track; ++k) w.ids[(uint32_t)k * P + p] = -1;
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

template <int CMAX>
cudaError_t launch_c(const Frames& fs, const Workspace& w, const float* features, const float* bg,
                     float* image, cudaStream_t stream) {
    constexpr int bytes = FwdSmem<CMAX>::bytes;
    const dim3 grid(fs.f[0].n_tiles_all), block(kFwdThreads);
    if (fs.f[0].n_cams == 1)
        return launch_pdl(k_forward<CMAX, false>, grid, block, bytes, stream, fs, w, features, bg,
                          image);
    return launch_pdl(k_forward<CMAX, true>, grid, block, bytes, stream, fs, w, features, bg,
                      image);
}

template <int CMAX>
cudaError_t prepare_c() {
    cudaError_t e = cudaFuncSetAttribute(k_forward<CMAX, false>,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         FwdSmem<CMAX>::bytes);
    if (e == cudaSuccess)
        e = cudaFuncSetAttribute(k_forward<CMAX, true>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 FwdSmem<CMAX>::bytes);
    return e;
}

}  // namespace

cudaError_t prepare_forward() {
    cudaError_t e = prepare_c<3>();
    if (e == cudaSuccess) e = prepare_c<4>();
    if (e == cudaSuccess) e = prepare_c<8>();
    if (e == cudaSuccess) e = prepare_c<16>();
    if (e == cudaSuccess) e = prepare_c<32>();
    if (e == cudaSuccess) e = prepare_c<kMaxChannels>();
    return e;
}

cudaError_t launch_forward(const Frames& fs, const Workspace& w, const float* features,
                           const float* bg, float* image, int /*max_pairs_stride*/,
                           cudaStream_t stream) {
    if (fs.f[0].channels == 3) return launch_c<3>(fs, w, features, bg, image, stream);
    if (fs.f[0].channels <= 4) return launch_c<4>(fs, w, features, bg, image, stream);
    if (fs.f[0].channels <= 8) return launch_c<8>(fs, w, features, bg, image, stream);
    if (fs.f[0].channels <= 16) return launch_c<16>(fs, w, features, bg, image, stream);
    if (fs.f[0].channels <= 32) return launch_c<32>(fs, w, features, bg, image, stream);
    return launch_c<kMaxChannels>(fs, w, features, bg, image, stream);
}

}  // namespace pulsar
