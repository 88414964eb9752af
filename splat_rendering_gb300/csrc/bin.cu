// Tile binning (Pulsar Sec. 3.2: candidates sorted by earliest possible
// intersection; Sec. B.1.1 depth sort; Sec. B.1.2 16x16 blocks).
//
//   k_tile_scan  one block: exclusive scan of the per-tile pair counts -> tile
//                offsets and M (the counters are cleared for the next frame);
//                latches a capacity error if M > max_pairs.
//   k_emit       one thread per staged pair (the projection gave each pair
//                its slot in its tile): scatter (key, id) to offset + slot.
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
constexpr int kSortThreads = 128;
constexpr int kSortCap = 2048;
constexpr int kRegSortMax = 4 * kSortThreads;   // lists sorted in registers

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
        w.tile_count[b] = 0u;
    }
    if (tid == kScanThreads - 1) {
        w.tile_start[f.n_tiles] = run;
        w.state->n_pairs = run;
        w.state->hits = 0ull;
        w.state->pair_cursor = 0u;
        if (run > f.max_pairs) atomicOr(&w.state->error, kErrCapacity);
    }
}

__global__ void __launch_bounds__(kEmitThreads) k_emit(Frame f, Workspace w) {
    const uint32_t m = w.state->n_pairs;
    if (m > f.max_pairs) return;   // overflowed frame: the capacity error is latched
    for (uint32_t p = blockIdx.x * blockDim.x + threadIdx.x; p < m; p += gridDim.x * blockDim.x) {
        const uint4 s = w.staged[p];
        const uint32_t at = w.tile_start[s.x] + s.y;
        if (at < m) w.pairs[at] = ((unsigned long long)s.z << 32) | s.w;
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

template <typename K>
__device__ __forceinline__ K cmp_keep(K mine, K other, bool take_min) {
    return take_min ? (mine < other ? mine : other) : (mine < other ? other : mine);
}

template <typename K>
__device__ __forceinline__ void cas_pair(K& a, K& b, bool up) {
    if ((a > b) == up) {
        const K tmp = a;
        a = b;
        b = tmp;
    }
}

// Ascending bitonic sort of up to kRegSortMax keys held in registers, four
// per thread (thread t holds elements 4t .. 4t+3): stages with partner
// distance 1 and 2 stay inside the thread, distances up to 64 use warp
// shuffles, only the longer ones go through shared memory.
template <typename K>
__device__ void register_bitonic(K (&e)[4], int np, K* s) {
    const int t = threadIdx.x;
    for (int k = 2; k <= np; k <<= 1) {
        for (int j = k >> 1; j > 0; j >>= 1) {
            if (j >= 4 * 32) {
#pragma unroll
                for (int r = 0; r < 4; ++r) s[4 * t + r] = e[r];
                __syncthreads();
#pragma unroll
                for (int r = 0; r < 4; ++r) {
                    const int i = 4 * t + r;
                    const K p = s[i ^ j];
                    e[r] = cmp_keep(e[r], p, ((i & j) == 0) == ((i & k) == 0));
                }
                __syncthreads();
            } else if (j >= 4) {
#pragma unroll
                for (int r = 0; r < 4; ++r) {
                    const int i = 4 * t + r;
                    const K p = __shfl_xor_sync(0xffffffffu, e[r], j >> 2);
                    e[r] = cmp_keep(e[r], p, ((i & j) == 0) == ((i & k) == 0));
                }
            } else {
                // inside the thread: pairs (0,1),(2,3) for j = 1; (0,2),(1,3) for j = 2;
                // each pair's direction comes from its lower index
                if (j == 1) {
                    cas_pair(e[0], e[1], ((4 * t) & k) == 0);
                    cas_pair(e[2], e[3], ((4 * t + 2) & k) == 0);
                } else {
                    cas_pair(e[0], e[2], ((4 * t) & k) == 0);
                    cas_pair(e[1], e[3], ((4 * t + 1) & k) == 0);
                }
            }
        }
    }
}

__global__ void __launch_bounds__(kSortThreads) k_tile_sort(Frame f, Workspace w) {
    __shared__ unsigned long long s[kSortCap];
    const int tile = blockIdx.x;
    const uint32_t start = w.tile_start[tile], end = w.tile_start[tile + 1];
    if (end > f.max_pairs || end <= start) return;   // capacity error already latched
    const int n = (int)(end - start);
    if (n <= kRegSortMax) {
        // Sort 32-bit keys: the tile's key bits (positive floats, so their bit
        // patterns are monotone) minus the tile minimum, shifted to 23 bits,
        // above the element's 9-bit local index.  Equal shifted keys are
        // ordered by local index; such rare runs are put in exact (key, id)
        // order by the fix-up below, so the result is the (key, id) order.
        unsigned long long* s64 = s;                                 // [512] input pairs
        uint32_t* s32 = reinterpret_cast<uint32_t*>(s + kRegSortMax);  // [512] sorted keys
        __shared__ uint32_t s_min, s_max;
        if (threadIdx.x == 0) {
            s_min = 0xffffffffu;
            s_max = 0u;
        }
        unsigned long long e64[4];
        uint32_t kmin = 0xffffffffu, kmax = 0u;
#pragma unroll
        for (int r = 0; r < 4; ++r) {
            const int i = 4 * threadIdx.x + r;
            e64[r] = i < n ? w.pairs[start + i] : ~0ull;
            if (i < n) {
                s64[i] = e64[r];
                const uint32_t kb = (uint32_t)(e64[r] >> 32);
                kmin = min(kmin, kb);
                kmax = max(kmax, kb);
            }
        }
        __syncthreads();
        atomicMin(&s_min, kmin);
        atomicMax(&s_max, kmax);
        __syncthreads();
        const uint32_t lo = s_min, span = s_max - s_min;
        const int shift = max(0, 32 - __clz((int)span) - 23);
        uint32_t e[4];
#pragma unroll
        for (int r = 0; r < 4; ++r) {
            const int i = 4 * threadIdx.x + r;
            e[r] = i < n ? ((((uint32_t)(e64[r] >> 32) - lo) >> shift) << 9) | (uint32_t)i
                         : 0xffffffffu;
        }
        const int np = max(next_pow2(n), 128);
        register_bitonic(e, np, s32);
        __syncthreads();
#pragma unroll
        for (int r = 0; r < 4; ++r) s32[4 * threadIdx.x + r] = e[r];
        __syncthreads();
        bool tie = false;
#pragma unroll
        for (int r = 0; r < 4; ++r) {
            const int i = 4 * threadIdx.x + r;
            if (i > 0 && i < n) tie |= (s32[i] >> 9) == (s32[i - 1] >> 9);
        }
        const bool any_tie = __syncthreads_or(tie);
        unsigned long long* sorted = s + kRegSortMax + kRegSortMax / 2;  // [512]
#pragma unroll
        for (int r = 0; r < 4; ++r) {
            const int i = 4 * threadIdx.x + r;
            if (i < n) sorted[i] = s64[e[r] & 511u];
        }
        __syncthreads();
        if (any_tie && threadIdx.x == 0) {
            // the array is sorted except inside runs of equal shifted keys:
            // insertion sort on the exact 64-bit (key, id) finishes it
            for (int i = 1; i < n; ++i) {
                const unsigned long long v = sorted[i];
                int q = i - 1;
                while (q >= 0 && sorted[q] > v) {
                    sorted[q + 1] = sorted[q];
                    --q;
                }
                sorted[q + 1] = v;
            }
        }
        __syncthreads();
        for (int i = threadIdx.x; i < n; i += blockDim.x) w.tile_ids[start + i] = (uint32_t)sorted[i];
        return;
    }
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
        k_emit<<<152 * 8, kEmitThreads, 0, stream>>>(f, w);
        k_tile_sort<<<f.n_tiles, kSortThreads, 0, stream>>>(f, w);
    }
    return cudaGetLastError();
}

}  // namespace pulsar
