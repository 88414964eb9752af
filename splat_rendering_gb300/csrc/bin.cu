// Tile binning (Pulsar Sec. 3.2: candidates sorted by earliest possible
// intersection; Sec. B.1.1 depth sort; Sec. B.1.2 16x16 blocks).
//
//   k_tile_scan  one block: exclusive scan of the per-tile pair counts -> tile
//                offsets and M; latches a capacity error if M > max_pairs.
//   k_emit       one thread per sphere, warp-cooperative over the warp's
//                (sphere, tile) pairs: each pair takes a slot in its tile's
//                bucket by counting the tile's counter back down to zero
//                (so the counters are zero again for the next frame).
//   k_tile_sort  one block per tile: sort the bucket by the 64-bit key
//                (f32 bits of c.z - r_eff) << 32 | sphere id, which is unique,
//                so the list does not depend on the bucket's arrival order.
//                Lists up to kSortCap entries are sorted in shared memory
//                (bitonic network); longer lists are sorted in chunks and
//                merged pairwise through global memory (merge path).
//
// The pairs live in L2-sized buffers for the shipped workloads (M ~ 1e6).
#include "pulsar_internal.cuh"

namespace pulsar {
namespace {

constexpr int kScanThreads = 1024;
constexpr int kEmitThreads = 256;
constexpr int kSortThreads = 256;
constexpr int kSortCap = 2048;

__global__ void __launch_bounds__(kScanThreads) k_tile_scan(Frame f, Workspace w) {
    __shared__ uint32_t s_warp[kScanThreads / 32];
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int per = (f.n_tiles + kScanThreads - 1) / kScanThreads;
    const int b0 = tid * per;
    const int b1 = min(b0 + per, f.n_tiles);
    uint32_t local = 0;
    for (int b = b0; b < b1; ++b) local += w.tile_count[b];
    uint32_t incl = local;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const uint32_t v = __shfl_up_sync(0xffffffffu, incl, o);
        if (lane >= o) incl += v;
    }
    if (lane == 31) s_warp[warp] = incl;
    __syncthreads();
    if (warp == 0) {
        uint32_t v = s_warp[lane];
        uint32_t vi = v;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const uint32_t u = __shfl_up_sync(0xffffffffu, vi, o);
            if (lane >= o) vi += u;
        }
        s_warp[lane] = vi - v;   // exclusive prefix of warp totals
    }
    __syncthreads();
    uint32_t run = s_warp[warp] + incl - local;
    for (int b = b0; b < b1; ++b) {
        w.tile_start[b] = run;
        run += w.tile_count[b];
    }
    if (tid == kScanThreads - 1) {
        w.tile_start[f.n_tiles] = run;
        w.state->n_pairs = run;
        w.state->hits = 0ull;
        if (run > f.max_pairs) atomicOr(&w.state->error, kErrCapacity);
    }
}

__global__ void __launch_bounds__(kEmitThreads) k_emit(Frame f, Workspace w) {
    const int i = blockIdx.x * blockDim.x + threadIdx.x;
    const int lane = threadIdx.x & 31;
    int tx0 = 0, ty0 = 0, ntx = 0, count = 0;
    uint32_t keybits = 0;
    if (i < f.n) {
        const uint4 rk = w.rec[i].rk;
        const int x0 = rk.x & 0xffff, x1 = rk.x >> 16, y0 = rk.y & 0xffff, y1 = rk.y >> 16;
        if (x0 <= x1 && y0 <= y1) {
            tx0 = x0 / kTile;
            ty0 = y0 / kTile;
            ntx = x1 / kTile - tx0 + 1;
            count = ntx * (y1 / kTile - ty0 + 1);
            keybits = rk.w;
        }
    }
    int incl = count;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const int v = __shfl_up_sync(0xffffffffu, incl, o);
        if (lane >= o) incl += v;
    }
    const int total = __shfl_sync(0xffffffffu, incl, 31);
    const int warp_first = i - lane;
    for (int j0 = 0; j0 < total; j0 += 32) {
        const int j = j0 + lane;
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
        const uint32_t own_key = __shfl_sync(0xffffffffu, keybits, own);
        if (j < total) {
            const int k = j - (own_incl - own_cnt);
            const int tile = (own_ty0 + k / own_ntx) * f.tiles_x + own_tx0 + k % own_ntx;
            const uint32_t slot = atomicSub(&w.tile_count[tile], 1u) - 1u;
            const uint32_t at = w.tile_start[tile] + slot;
            if (at < f.max_pairs)
                w.pairs[at] = ((unsigned long long)own_key << 32) | (uint32_t)(warp_first + own);
        }
    }
}

// In-place ascending bitonic sort of s[0, np) (np a power of two), all
// threads of the block participating.  j is a power of two, so the pair index
// is formed with masks: lo = 2 j floor(t / j) + t mod j.
__device__ void block_bitonic(unsigned long long* s, int np) {
    for (int k = 2; k <= np; k <<= 1) {
        for (int j = k >> 1; j > 0; j >>= 1) {
            for (int t = threadIdx.x; t < (np >> 1); t += blockDim.x) {
                const int lo = ((t & ~(j - 1)) << 1) | (t & (j - 1));
                const int hi = lo + j;
                const unsigned long long a = s[lo], b = s[hi];
                const bool up = (lo & k) == 0;
                if ((a > b) == up) {
                    s[lo] = b;
                    s[hi] = a;
                }
            }
            __syncthreads();
        }
    }
}

__device__ int next_pow2(int n) {
    int p = 1;
    while (p < n) p <<= 1;
    return p;
}

// Number of elements taken from a (length la) among the first k outputs of
// merging a and b (length lb); keys are unique.
__device__ int merge_split(const unsigned long long* a, int la, const unsigned long long* b,
                           int lb, int k) {
    int lo = max(0, k - lb), hi = min(k, la);
    while (lo < hi) {
        const int mid = (lo + hi) >> 1;
        if (a[mid] < b[k - 1 - mid]) lo = mid + 1; else hi = mid;
    }
    return lo;
}

__global__ void __launch_bounds__(kSortThreads) k_tile_sort(Frame f, Workspace w) {
    __shared__ unsigned long long s[kSortCap];
    const int tile = blockIdx.x;
    const uint32_t start = w.tile_start[tile], end = w.tile_start[tile + 1];
    if (end > f.max_pairs || end <= start) return;   // capacity error already latched
    const int n = (int)(end - start);
    if (n <= kSortCap) {
        const int np = next_pow2(n);
        for (int t = threadIdx.x; t < np; t += blockDim.x)
            s[t] = t < n ? w.pairs[start + t] : ~0ull;
        __syncthreads();
        block_bitonic(s, np);
        for (int t = threadIdx.x; t < n; t += blockDim.x) w.tile_ids[start + t] = (uint32_t)s[t];
        return;
    }
    // long list: sort chunks of kSortCap in shared memory ...
    unsigned long long* src = w.pairs + start;
    unsigned long long* dst = w.pairs_alt + start;
    for (int c0 = 0; c0 < n; c0 += kSortCap) {
        const int m = min(kSortCap, n - c0);
        const int np = next_pow2(m);
        for (int t = threadIdx.x; t < np; t += blockDim.x) s[t] = t < m ? src[c0 + t] : ~0ull;
        __syncthreads();
        block_bitonic(s, np);
        for (int t = threadIdx.x; t < m; t += blockDim.x) src[c0 + t] = s[t];
        __syncthreads();
    }
    // ... then merge runs pairwise, doubling the run width each pass
    for (int width = kSortCap; width < n; width <<= 1) {
        for (int r0 = 0; r0 < n; r0 += 2 * width) {
            const int la = min(width, n - r0);
            const int lb = max(0, min(width, n - r0 - width));
            const unsigned long long* a = src + r0;
            const unsigned long long* b = a + la;
            const int total = la + lb;
            const int per = (total + blockDim.x - 1) / blockDim.x;
            const int k0 = min(total, (int)threadIdx.x * per);
            const int k1 = min(total, k0 + per);
            int ia = merge_split(a, la, b, lb, k0);
            int ib = k0 - ia;
            for (int k = k0; k < k1; ++k) {
                const bool take_a = ib >= lb || (ia < la && a[ia] < b[ib]);
                dst[r0 + k] = take_a ? a[ia++] : b[ib++];
            }
        }
        __syncthreads();
        unsigned long long* tmp = src;
        src = dst;
        dst = tmp;
    }
    for (int t = threadIdx.x; t < n; t += blockDim.x) w.tile_ids[start + t] = (uint32_t)src[t];
}

}  // namespace

cudaError_t launch_bin(const Frame& f, const Workspace& w, cudaStream_t stream) {
    k_tile_scan<<<1, kScanThreads, 0, stream>>>(f, w);
    if (f.n > 0) {
        const int blocks = (f.n + kEmitThreads - 1) / kEmitThreads;
        k_emit<<<blocks, kEmitThreads, 0, stream>>>(f, w);
        k_tile_sort<<<f.n_tiles, kSortThreads, 0, stream>>>(f, w);
    }
    return cudaGetLastError();
}

}  // namespace pulsar
