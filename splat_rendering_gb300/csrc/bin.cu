// Tile binning (Pulsar Sec. 3.2: candidates sorted by earliest possible
// intersection; Sec. B.1.1 depth sort; Sec. B.1.2 16x16 blocks).
//
//   k_tile_scan  one block: exclusive scan of the per-tile pair counts -> tile
//                offsets and M (the counters are cleared for the next frame),
//                and the list of tiles whose bucket is longer than one warp
//                sorts; latches a capacity error if M > max_pairs.
//   k_emit       one thread per staged pair (the projection gave each pair
//                its slot in its tile): scatter (key, id) to offset + slot.
//   k_tile_sort  one warp per tile: sort the bucket by the 64-bit key
//                (f32 bits of c.z - r_eff) << 32 | sphere id, which is unique,
//                so the list does not depend on the bucket's arrival order.
//                Lists up to kWarpSortMax entries are sorted in registers as
//                packed 32-bit keys (bitonic networks on two runs of at most
//                256, merged by merge path).
//   k_tile_sort_long  persistent blocks take the longer lists from a work
//                counter: up to kLongCap entries sorted in one piece in
//                shared memory, beyond that in chunks merged pairwise through
//                global memory (merge path).
//
// The pairs live in L2-sized buffers for the shipped workloads (M ~ 1e6).
#include "pulsar_internal.cuh"

namespace pulsar {
namespace {

constexpr int kScanThreads = 1024;
constexpr int kEmitThreads = 256;
constexpr int kSortThreads = 128;
constexpr int kTilesPerSortBlock = kSortThreads / 32;
constexpr int kSortCap = 2048;
constexpr int kWarpSortMax = 512;   // lists sorted by one warp in registers

// Block-wide exclusive scan of one value per thread; returns the thread's
// exclusive prefix, *total the block's sum (s: 32 words of scratch).
__device__ __forceinline__ uint32_t block_exclusive_scan(uint32_t v, uint32_t* s, uint32_t* total) {
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    uint32_t incl = v;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const uint32_t u = __shfl_up_sync(0xffffffffu, incl, o);
        if (lane >= o) incl += u;
    }
    if (lane == 31) s[warp] = incl;
    __syncthreads();
    if (warp == 0) {
        const uint32_t t = lane < (int)(blockDim.x >> 5) ? s[lane] : 0u;
        uint32_t ti = t;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const uint32_t u = __shfl_up_sync(0xffffffffu, ti, o);
            if (lane >= o) ti += u;
        }
        s[lane] = ti - t;   // exclusive prefix of the warp totals
        if (lane == 31) s[32] = ti;
    }
    __syncthreads();
    const uint32_t r = s[warp] + incl - v;
    *total = s[32];
    __syncthreads();   // s is free for the next scan
    return r;
}

// One block walks the tiles in chunks of kScanChunk, each thread owning
// kScanPer consecutive tiles (coalesced 16-byte loads and stores): the tile
// offsets, the counters cleared for the next frame, and the list of tiles
// whose bucket is too long for one warp's sort, in tile order.
constexpr int kScanPer = 4;
constexpr int kScanChunk = kScanThreads * kScanPer;

__global__ void __launch_bounds__(kScanThreads) k_tile_scan(Frames fs, Workspace w) {
    pdl_begin();
    __shared__ uint32_t s_scan[33];
    const Frame& f = fs.f[0];
    const int n_tiles = (int)f.n_tiles_all;   // every camera's tiles, camera after camera
    uint32_t carry = 0, lcarry = 0;            // pairs and long tiles before the chunk
    for (int c0 = 0; c0 < n_tiles; c0 += kScanChunk) {
        const int b = c0 + kScanPer * (int)threadIdx.x;
        uint32_t cnt[kScanPer];
        if (b + kScanPer <= n_tiles) {
            const uint4 v = *reinterpret_cast<const uint4*>(w.tile_count + b);
            cnt[0] = v.x; cnt[1] = v.y; cnt[2] = v.z; cnt[3] = v.w;
        } else {
#pragma unroll
            for (int q = 0; q < kScanPer; ++q) cnt[q] = b + q < n_tiles ? w.tile_count[b + q] : 0u;
        }
        uint32_t local = 0, llocal = 0;
#pragma unroll
        for (int q = 0; q < kScanPer; ++q) {
            local += cnt[q];
            llocal += cnt[q] > (uint32_t)kWarpSortMax ? 1u : 0u;
        }
        uint32_t total, ltotal;
        uint32_t run = carry + block_exclusive_scan(local, s_scan, &total);
        uint32_t lrun = lcarry + block_exclusive_scan(llocal, s_scan, &ltotal);
        uint32_t st[kScanPer];
#pragma unroll
        for (int q = 0; q < kScanPer; ++q) {
            st[q] = run;
            run += cnt[q];
            if (cnt[q] > (uint32_t)kWarpSortMax) w.long_tiles[lrun++] = (uint32_t)(b + q);
        }
        if (b + kScanPer <= n_tiles) {
            *reinterpret_cast<uint4*>(w.tile_start + b) = make_uint4(st[0], st[1], st[2], st[3]);
            *reinterpret_cast<uint4*>(w.tile_count + b) = make_uint4(0u, 0u, 0u, 0u);
        } else {
#pragma unroll
            for (int q = 0; q < kScanPer; ++q) {
                if (b + q < n_tiles) {
                    w.tile_start[b + q] = st[q];
                    w.tile_count[b + q] = 0u;
                }
            }
        }
        carry += total;
        lcarry += ltotal;
    }
    if (threadIdx.x == 0) {
        w.tile_start[n_tiles] = carry;
        w.state->n_pairs = carry;
        w.state->n_long = lcarry;
        w.state->long_next = 0u;
        w.state->hits = 0ull;
        w.state->pair_cursor = 0u;
        if (carry > f.max_pairs) atomicOr(&w.state->error, kErrCapacity);
    }
}

__global__ void __launch_bounds__(kEmitThreads) k_emit(Frames fs, Workspace w) {
    pdl_begin();
    const Frame& f = fs.f[0];
    const uint32_t m = w.state->n_pairs;
    if (m > f.max_pairs) return;   // overflowed frame: the capacity error is latched
    // 64-bit cursor: m may lie within one grid stride of 2^32
    for (uint64_t p = (uint64_t)blockIdx.x * blockDim.x + threadIdx.x; p < m;
         p += (uint64_t)gridDim.x * blockDim.x) {
        const uint4 s = w.staged[p];
        if (!PULSAR_CHECK(w.state, s.x < f.n_tiles_all)) continue;
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

// Ascending bitonic network over a warp's 32 E keys held in registers,
// element E * lane + r in e[r]: partners less than E apart are in the same
// thread, the others one shuffle away.  Every stage's direction is a
// compile-time constant or uniform over the lane's elements.
template <int E>
__device__ __forceinline__ void warp_bitonic(uint32_t (&e)[16], int lane) {
#pragma unroll
    for (int k = 2; k <= 32 * E; k <<= 1) {
#pragma unroll
        for (int j = k >> 1; j > 0; j >>= 1) {
            if (j >= E) {
                const int pl = j / E;
                const bool keep_min = ((lane & pl) == 0) == (((lane * E) & k) == 0);
#pragma unroll
                for (int r = 0; r < E; ++r) {
                    const uint32_t p = __shfl_xor_sync(0xffffffffu, e[r], pl);
                    e[r] = keep_min ? min(e[r], p) : max(e[r], p);
                }
            } else {
                const bool up_lane = ((lane * E) & k) == 0;
#pragma unroll
                for (int r = 0; r < E; ++r) {
                    if ((r & j) == 0) {
                        const bool up = k < E ? (r & k) == 0 : up_lane;
                        const uint32_t a = e[r], b = e[r + j];
                        const uint32_t lo = min(a, b), hi = max(a, b);
                        e[r] = up ? lo : hi;
                        e[r + j] = up ? hi : lo;
                    }
                }
            }
        }
    }
}

// Ascending bitonic sort of the k <= 32 E unique 32-bit keys at keys[0 .. k)
// in place (the buffer holds 32 E words; entries k .. 32 E - 1 are padded
// with ~0u, above every key).  Lane l holds elements E l .. E l + E - 1.
template <int E>
__device__ __forceinline__ void sort_keys(uint32_t* keys, int k, int lane) {
    for (int i = k + lane; i < 32 * E; i += 32) keys[i] = 0xffffffffu;
    __syncwarp();
    uint32_t e[16];
    uint32_t* mine = keys + E * lane;
    if constexpr (E >= 4) {
#pragma unroll
        for (int q = 0; q < E / 4; ++q) {
            const uint4 v = reinterpret_cast<const uint4*>(mine)[q];
            e[4 * q] = v.x; e[4 * q + 1] = v.y; e[4 * q + 2] = v.z; e[4 * q + 3] = v.w;
        }
    } else {
#pragma unroll
        for (int r = 0; r < E; ++r) e[r] = mine[r];
    }
    warp_bitonic<E>(e, lane);
    __syncwarp();
    if constexpr (E >= 4) {
#pragma unroll
        for (int q = 0; q < E / 4; ++q)
            reinterpret_cast<uint4*>(mine)[q] = make_uint4(e[4 * q], e[4 * q + 1], e[4 * q + 2], e[4 * q + 3]);
    } else {
#pragma unroll
        for (int r = 0; r < E; ++r) mine[r] = e[r];
    }
}

// Number of elements taken from a (length la) among the first k outputs of
// merging the sorted runs a and b (length lb) of unique keys.
__device__ __forceinline__ int merge_split32(const uint32_t* a, int la, const uint32_t* b, int lb,
                                             int k) {
    int lo = max(0, k - lb), hi = min(k, la);
    while (lo < hi) {
        const int mid = (lo + hi) >> 1;
        if (a[mid] < b[k - 1 - mid]) lo = mid + 1; else hi = mid;
    }
    return lo;
}

// One warp sorts one tile's n <= kWarpSortMax pairs (key bits << 32 | id).
// It sorts 32-bit keys: the key bits (positive floats, so their bit patterns
// are monotone) minus the tile minimum, shifted down to 23 bits, above the
// element's 9-bit position in the bucket.  The first 256 keys and the rest
// are sorted as two runs, each by the smallest register network that holds
// it (a list of 300 keys costs a 256- and a 64-key network, not a 512-key
// one), and merged by merge path, a contiguous span of outputs per lane.
// Equal shifted keys come out ordered by position; such rare runs, marked
// while merging, are put in exact (key, id) order by insertion sorts, each
// run by the lane in whose span it starts, so the result is the (key, id)
// order.  s64 holds the bucket, s32 the keys
// (512 words each) and, once they are merged, the sorted positions.
__device__ void warp_sort_tile(const Workspace& w, uint32_t start, int n, unsigned long long* s64,
                               uint32_t* s32, int lane) {
    uint32_t kmin = 0xffffffffu, kmax = 0u;
    // the bucket, eight loads in flight per lane
    for (int i0 = 0; i0 < n; i0 += 256) {
        unsigned long long v[8];
#pragma unroll
        for (int r = 0; r < 8; ++r) {
            const int i = i0 + 32 * r + lane;
            v[r] = i < n ? w.pairs[start + i] : 0ull;
        }
#pragma unroll
        for (int r = 0; r < 8; ++r) {
            const int i = i0 + 32 * r + lane;
            if (i < n) {
                s64[i] = v[r];
                const uint32_t kb = (uint32_t)(v[r] >> 32);
                kmin = min(kmin, kb);
                kmax = max(kmax, kb);
            }
        }
    }
    const uint32_t lo = __reduce_min_sync(0xffffffffu, kmin);
    const uint32_t span = __reduce_max_sync(0xffffffffu, kmax) - lo;
    const int shift = max(0, 32 - __clz((int)span) - 23);
    __syncwarp();
    for (int i = lane; i < n; i += 32)
        s32[i] = ((((uint32_t)(s64[i] >> 32) - lo) >> shift) << 9) | (uint32_t)i;
    const int la = min(n, 256), lb = n - la;
#pragma unroll 1
    for (int c = 0; c < (lb > 0 ? 2 : 1); ++c) {
        uint32_t* keys = s32 + 256 * c;
        const int k = c ? lb : la;
        if (k <= 32) sort_keys<1>(keys, k, lane);
        else if (k <= 64) sort_keys<2>(keys, k, lane);
        else if (k <= 128) sort_keys<4>(keys, k, lane);
        else sort_keys<8>(keys, k, lane);
    }
    __syncwarp();
    const uint32_t* A = s32;
    const uint32_t* B = s32 + 256;
    const int per = (n + 31) >> 5;
    const int k0 = min(n, lane * per), k1 = min(n, k0 + per);
    int ia = merge_split32(A, la, B, lb, k0), ib = k0 - ia;
    uint32_t prev = max(ia > 0 ? A[ia - 1] : 0u, ib > 0 ? B[ib - 1] : 0u);
    uint32_t tmask = 0;                 // bit t: output k0 + t ties with its predecessor
    uint16_t out[kWarpSortMax / 32];   // this lane's span of sorted positions
#pragma unroll
    for (int t = 0; t < kWarpSortMax / 32; ++t) {
        const int k = k0 + t;
        if (k < k1) {
            const bool take_a = ib >= lb || (ia < la && A[ia] < B[ib]);
            const uint32_t v = take_a ? A[ia++] : B[ib++];
            tmask |= (uint32_t)(k > 0 && (prev >> 9) == (v >> 9)) << t;
            prev = v;
            out[t] = (uint16_t)(v & 511u);
        }
    }
    const bool any_tie = __any_sync(0xffffffffu, tmask != 0u);
    __syncwarp();   // every lane's merge has read its keys: positions and tie masks take their place
    uint16_t* s_pos = reinterpret_cast<uint16_t*>(s32);          // words 0 .. 255
    uint16_t* s_tie = reinterpret_cast<uint16_t*>(s32 + 384);    // one 16-bit mask per lane
#pragma unroll
    for (int t = 0; t < kWarpSortMax / 32; ++t)
        if (k0 + t < k1) s_pos[k0 + t] = out[t];
    if (any_tie) s_tie[lane] = (uint16_t)tmask;
    __syncwarp();
    if (any_tie) {
        // sorted except inside runs of equal shifted keys: each lane puts the
        // runs that start in its span in exact (key, id) order (insertion
        // sort); the runs are disjoint and the masks are only read here
        auto tied = [&](int k) {
            const int l = k / per;
            return ((s_tie[l] >> (k - l * per)) & 1u) != 0u;
        };
        for (int k = k0; k < k1; ++k) {
            if (tied(k) || k + 1 >= n || !tied(k + 1)) continue;
            int e = k + 2;
            while (e < n && tied(e)) ++e;
            for (int i = k + 1; i < e; ++i) {
                const uint16_t v = s_pos[i];
                const unsigned long long kv = s64[v];
                int q = i - 1;
                while (q >= k && s64[s_pos[q]] > kv) {
                    s_pos[q + 1] = s_pos[q];
                    --q;
                }
                s_pos[q + 1] = v;
            }
        }
    }
    __syncwarp();
    for (int i = lane; i < n; i += 32) w.tile_ids[start + i] = (uint32_t)s64[s_pos[i]];
}

// A list longer than kWarpSortMax, sorted by the whole block: up to kSortCap
// entries in shared memory (bitonic network on the 64-bit keys); longer ones
// in chunks of kSortCap, merged pairwise through global memory (merge path).
__device__ void block_sort_long(const Workspace& w, uint32_t start, int n, unsigned long long* s) {
    if (n <= kSortCap) {
        const int np = next_pow2(n);
        for (int t = threadIdx.x; t < np; t += blockDim.x)
            s[t] = t < n ? w.pairs[start + t] : ~0ull;
        __syncthreads();
        block_bitonic(s, np);
        for (int t = threadIdx.x; t < n; t += blockDim.x) w.tile_ids[start + t] = (uint32_t)s[t];
        return;
    }
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

// Block b covers tiles 4b .. 4b+3, one warp each; lists longer than
// kWarpSortMax are left to k_tile_sort_long.
__global__ void __launch_bounds__(kSortThreads) k_tile_sort(Frames fs, Workspace w) {
    pdl_begin();
    const Frame& f = fs.f[0];
    const int n_tiles = (int)f.n_tiles_all;
    __shared__ unsigned long long s[kTilesPerSortBlock * kWarpSortMax];        // 16 KB
    __shared__ __align__(16) uint32_t s_keys[kTilesPerSortBlock][kWarpSortMax]; // 8 KB
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int tile = blockIdx.x * kTilesPerSortBlock + warp;
    if (tile >= n_tiles) return;
    const uint32_t start = w.tile_start[tile], end = w.tile_start[tile + 1];
    // (a frame over capacity has its error latched; its lists are not sorted)
    if (end <= f.max_pairs && end > start && end - start <= (uint32_t)kWarpSortMax)
        warp_sort_tile(w, start, (int)(end - start), s + warp * kWarpSortMax, s_keys[warp], lane);
}

// The long lists: persistent blocks take the tiles of long_tiles one at a
// time from a work counter (the lengths are very uneven).  A list of at most
// kLongCap keys is sorted in one piece in shared memory (bitonic network on
// the 64-bit keys); a longer one in kSortCap chunks merged through global
// memory.
constexpr int kLongThreads = 512;
constexpr int kLongCap = 8192;                       // 64 KB of keys
constexpr int kLongSmem = kLongCap * 8;
constexpr int kLongBlocksPerSm = 2;

__global__ void __launch_bounds__(kLongThreads) k_tile_sort_long(Frames fs, Workspace w) {
    pdl_begin();
    extern __shared__ __align__(16) unsigned long long s_long[];
    __shared__ uint32_t s_item;
    const Frame& f = fs.f[0];
    const uint32_t n_long = w.state->n_long;
    if (w.state->n_pairs > f.max_pairs) return;   // overflowed frame: nothing to sort
    for (;;) {
        if (threadIdx.x == 0) s_item = atomicAdd(&w.state->long_next, 1u);
        __syncthreads();
        const uint32_t item = s_item;
        __syncthreads();   // every thread has the item before it is overwritten
        if (item >= n_long) break;
        const uint32_t tile = w.long_tiles[item];
        const uint32_t start = w.tile_start[tile], end = w.tile_start[tile + 1];
        const int n = (int)(end - start);
        if (n <= kLongCap) {
            const int np = next_pow2(n);
            for (int t = threadIdx.x; t < np; t += blockDim.x)
                s_long[t] = t < n ? w.pairs[start + t] : ~0ull;
            __syncthreads();
            block_bitonic(s_long, np);
            for (int t = threadIdx.x; t < n; t += blockDim.x)
                w.tile_ids[start + t] = (uint32_t)s_long[t];
        } else {
            block_sort_long(w, start, n, s_long);
        }
        __syncthreads();   // the shared buffer is free for the next tile
    }
}

}  // namespace

cudaError_t prepare_bin() {
    return cudaFuncSetAttribute(k_tile_sort_long, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                kLongSmem);
}

cudaError_t launch_bin(const Frames& fs, const Workspace& w, cudaStream_t stream) {
    const Frame& f = fs.f[0];
    // both grids below loop over their work; they are sized by the SM count
    int dev = 0, sms = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e == cudaSuccess) e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    if (e != cudaSuccess) return e;
    e = launch_pdl(k_tile_scan, dim3(1), dim3(kScanThreads), 0, stream, fs, w);
    if (e == cudaSuccess && f.n > 0) {
        e = launch_pdl(k_emit, dim3(sms * 8), dim3(kEmitThreads), 0, stream, fs, w);
        if (e == cudaSuccess)
            e = launch_pdl(k_tile_sort,
                           dim3(((int)f.n_tiles_all + kTilesPerSortBlock - 1) / kTilesPerSortBlock),
                           dim3(kSortThreads), 0, stream, fs, w);
        if (e == cudaSuccess)
            e = launch_pdl(k_tile_sort_long, dim3(sms * kLongBlocksPerSm), dim3(kLongThreads),
                           kLongSmem, stream, fs, w);
    }
    return e;
}

}  // namespace pulsar
