// pulsar_render_noalloc: a forward render of a small frame that allocates no
// memory at all.
//
// Some callers cannot call cudaMalloc while they render: plugins hosted by a
// framework that owns the whole device memory budget and forbids other
// allocators, and fixed-footprint real-time renderers that must not risk an
// out-of-memory failure, or the implicit device synchronisation that
// cudaMalloc and cudaFree may bring, in the middle of a frame.  For them this
// entry point runs the same projection, binning and forward kernels as
// pulsar_project / pulsar_bin / pulsar_forward, but every intermediate array
// lives in one file-scope static device arena of fixed size (below),
// reserved when the library is loaded and held by every GPU that loads it
// until the process exits.
//
// Limits (the arena's capacity): at most kMaxSpheres spheres, kMaxPairs
// sphere-tile pairs, images up to kMaxSide x kMaxSide, n_track <= kMaxTrackNA,
// channels <= 64.  Larger requests are rejected with PULSAR_ERR_ARG; a frame
// whose pairs exceed kMaxPairs returns PULSAR_ERR_CAPACITY.
//
// Every call shares the one arena and it keeps the previous call's contents:
// the call clears the parts that must start at zero (tile counters, device
// state) on the caller's stream before use.  Two calls whose work overlaps on
// the GPU (different streams, or host threads racing) corrupt each other:
// callers must serialise them.
//
// The first call on a device looks up the arena's device address with
// cudaGetSymbolAddress (with that device current) and prepares the forward
// and sort kernels; that first call should come before any stream capture.
// Every call synchronises the stream at its end to read the frame's status.
#include <cuda_runtime.h>

#include <cstring>
#include <mutex>

#include "../../include/pulsar.h"
#include "pulsar_internal.cuh"

using namespace pulsar;

namespace {

constexpr int kMaxSpheres = 16384;
constexpr int kMaxPairs = 65536;
constexpr int kMaxSide = 256;
constexpr int kMaxTrackNA = 8;
constexpr int kMaxPix = kMaxSide * kMaxSide;
constexpr int kMaxTilesNA = (kMaxSide / kTile) * (kMaxSide / kTile);
constexpr int kMaxDevices = 64;

// Fixed carve-up of the arena (256-byte aligned pieces).
constexpr size_t align256(size_t v) { return (v + 255) / 256 * 256; }
constexpr size_t kOffRec = 0;
constexpr size_t kOffCount = align256(kOffRec + sizeof(SphereRec) * kMaxSpheres);
constexpr size_t kOffStart = align256(kOffCount + 4 * kMaxTilesNA);
constexpr size_t kOffLong = align256(kOffStart + 4 * (kMaxTilesNA + 1));
constexpr size_t kOffStaged = align256(kOffLong + 4 * (size_t)kMaxTilesNA);
constexpr size_t kOffPairs = align256(kOffStaged + 16 * (size_t)kMaxPairs);
constexpr size_t kOffPairsAlt = align256(kOffPairs + 8 * (size_t)kMaxPairs);
constexpr size_t kOffTileIds = align256(kOffPairsAlt + 8 * (size_t)kMaxPairs);
constexpr size_t kOffMg = align256(kOffTileIds + 4 * (size_t)kMaxPairs);
constexpr size_t kOffW = align256(kOffMg + 4 * (size_t)kMaxPix);
constexpr size_t kOffIds = align256(kOffW + 4 * (size_t)kMaxPix);
constexpr size_t kOffD = align256(kOffIds + 4 * (size_t)kMaxPix * kMaxTrackNA);
constexpr size_t kOffHits = align256(kOffD + 4 * (size_t)kMaxPix * kMaxTrackNA);
constexpr size_t kOffState = align256(kOffHits + 4 * (size_t)kMaxPix);
constexpr size_t kArenaBytes = align256(kOffState + sizeof(DevState));   // ~8.2 MB

// The arena.  Host code must not use this name as an address (on the host it
// is only a stand-in); it uses the device address looked up below.
static __device__ __align__(256) unsigned char g_arena[kArenaBytes];

std::mutex g_setup_mutex;
unsigned char* g_arena_dev[kMaxDevices] = {};   // device address of g_arena, per device

// Once per device, with that device current: look up the arena's address and
// opt the forward kernels into their shared memory.
int arena_for_current_device(unsigned char** out) {
    int dev = -1;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return PULSAR_ERR_CUDA;
    std::lock_guard<std::mutex> lock(g_setup_mutex);
    if (!g_arena_dev[dev]) {
        void* p = nullptr;
        if (cudaGetSymbolAddress(&p, g_arena) != cudaSuccess || !p) return PULSAR_ERR_CUDA;
        if (prepare_forward() != cudaSuccess || prepare_bin() != cudaSuccess) return PULSAR_ERR_CUDA;
        g_arena_dev[dev] = static_cast<unsigned char*>(p);
    }
    *out = g_arena_dev[dev];
    return PULSAR_OK;
}

bool positive(float v) { return v > 0.0f && v < 3.0e38f; }

}  // namespace

extern "C" int pulsar_render_noalloc(const float* pos, const float* radius, const float* opacity,
                                     const float* features, int64_t n,
                                     const pulsar_camera_t* cam, const pulsar_params_t* prm,
                                     const float* bg, float* image, void* stream) {
    if (!cam || !prm || !bg || !image || n < 0 || n > kMaxSpheres) return PULSAR_ERR_ARG;
    if (n > 0 && (!pos || !radius || !opacity || !features)) return PULSAR_ERR_ARG;
    if (cam->width < 1 || cam->height < 1 || cam->width > kMaxSide || cam->height > kMaxSide)
        return PULSAR_ERR_ARG;
    if (!positive(cam->fx) || !positive(cam->fy) || !(cam->znear > 0.0f) ||
        !(cam->zfar > cam->znear) || (cam->orthographic != 0 && cam->orthographic != 1))
        return PULSAR_ERR_ARG;
    if (!positive(prm->gamma) || !(prm->bg_eps >= 0.0f) || !(prm->stop_tau >= 0.0f) ||
        !(prm->kappa >= 0.0f) || !(prm->geom_min_area >= 0.0f) || prm->n_track < 1 ||
        prm->n_track > kMaxTrackNA || prm->channels < 1 || prm->channels > kMaxChannels)
        return PULSAR_ERR_ARG;
    unsigned char* a = nullptr;
    const int rc = arena_for_current_device(&a);
    if (rc != PULSAR_OK) return rc;
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);

    Workspace w{};
    w.rec = reinterpret_cast<SphereRec*>(a + kOffRec);
    w.gacc = nullptr;   // forward only
    w.gacc2 = nullptr;
    w.hitcnt = nullptr;
    w.tile_count = reinterpret_cast<uint32_t*>(a + kOffCount);
    w.tile_start = reinterpret_cast<uint32_t*>(a + kOffStart);
    w.long_tiles = reinterpret_cast<uint32_t*>(a + kOffLong);
    w.staged = reinterpret_cast<uint4*>(a + kOffStaged);
    w.pairs = reinterpret_cast<unsigned long long*>(a + kOffPairs);
    w.pairs_alt = reinterpret_cast<unsigned long long*>(a + kOffPairsAlt);
    w.tile_ids = reinterpret_cast<uint32_t*>(a + kOffTileIds);
    w.mg = reinterpret_cast<float*>(a + kOffMg);
    w.wsum = reinterpret_cast<float*>(a + kOffW);
    w.ids = reinterpret_cast<int32_t*>(a + kOffIds);
    w.dtr = reinterpret_cast<float*>(a + kOffD);
    w.nhits = reinterpret_cast<int32_t*>(a + kOffHits);
    w.kpart = nullptr;
    w.rtpart = nullptr;
    w.state = reinterpret_cast<DevState*>(a + kOffState);

    // the per-frame constants, formed exactly as pulsar_project forms them
    Frames fs{};
    fill_frame(fs.f[0], cam->R, cam->t, cam->fx, cam->fy, cam->cx, cam->cy, cam->width,
               cam->height, cam->znear, cam->zfar, cam->orthographic, prm->gamma, prm->bg_eps,
               prm->stop_tau, prm->kappa, prm->geom_min_area, prm->n_track, prm->channels,
               prm->flags, (int)n, (uint32_t)kMaxPairs, 0, 1);

    // the arena keeps the previous call's contents: clear what must start at zero
    if (cudaMemsetAsync(w.tile_count, 0, 4 * (size_t)kMaxTilesNA, s) != cudaSuccess ||
        cudaMemsetAsync(w.state, 0, sizeof(DevState), s) != cudaSuccess)
        return PULSAR_ERR_CUDA;
    if (launch_project(fs, w, pos, radius, opacity, s) != cudaSuccess ||
        launch_bin(fs, w, s) != cudaSuccess ||
        launch_forward(fs, w, features, bg, image, 0, s) != cudaSuccess)
        return PULSAR_ERR_CUDA;
    DevState st;
    if (cudaMemcpyAsync(&st, w.state, sizeof(DevState), cudaMemcpyDeviceToHost, s) != cudaSuccess ||
        cudaStreamSynchronize(s) != cudaSuccess)
        return PULSAR_ERR_CUDA;
    if (st.n_pairs > (uint32_t)kMaxPairs) return PULSAR_ERR_CAPACITY;
    return PULSAR_OK;
}
