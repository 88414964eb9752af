// C ABI of the sphere renderer: context, workspace and the per-frame call
// sequence (project -> bin -> forward -> backward).  Every call validates its
// arguments on the host, enqueues kernels on the caller's stream and returns
// without synchronising; device-side errors are latched and reported by
// pulsar_status.
#include <cuda_runtime.h>

#include <cstring>
#include <new>
#include <vector>

#include "../../include/pulsar.h"
#include "pulsar_internal.cuh"

// NVTX ranges around the entry points (build with -DPULSAR_NVTX: header-only
// NVTX3, no link dependency, no cost when no tool is attached); compiled out
// by default.
#ifdef PULSAR_NVTX
#include <nvtx3/nvToolsExt.h>
namespace {
struct NvtxScope {
    explicit NvtxScope(const char* name) { nvtxRangePushA(name); }
    ~NvtxScope() { nvtxRangePop(); }
};
}  // namespace
#define PULSAR_TRACE(name) NvtxScope pulsar_trace_scope_(name)
#else
#define PULSAR_TRACE(name) ((void)0)
#endif

using namespace pulsar;

struct pulsar_ctx {
    int device = 0;
    int64_t max_n = 0, max_pairs = 0;
    int32_t max_w = 0, max_h = 0, max_c = 0, max_t = 0, max_cams = 1;
    int64_t max_tiles = 0, max_pix = 0;   // per camera
    Workspace ws{};
    DevState* host_state = nullptr;   // pinned mirror for pulsar_status
    Frames frames{};                   // the cameras of the current frame
    int n_cams = 0;
    int n_sms = 1;
    ShadeLaunch shade{};
    const float* pos = nullptr;        // inputs of the current frame
    int stage = 0;                     // 0 none, 1 projected, 2 binned, 3 forward done
    bool counts_dirty = false;         // tile counts hold a frame that was never binned
    bool acc_zeroed = false;           // the forward zeroed the backward's accumulators
    static constexpr int kMaxAllocs = 32;
    void* allocs[kMaxAllocs] = {};
    int n_allocs = 0;
};

namespace {

cudaStream_t as_stream(void* s) { return reinterpret_cast<cudaStream_t>(s); }

int cuda_err(cudaError_t e) { return e == cudaSuccess ? PULSAR_OK : PULSAR_ERR_CUDA; }

struct DeviceGuard {
    int prev = -1;
    explicit DeviceGuard(int dev) {
        if (cudaGetDevice(&prev) != cudaSuccess) prev = -1;
        if (prev != dev) cudaSetDevice(dev);
    }
    ~DeviceGuard() {
        int cur = -1;
        if (prev >= 0 && cudaGetDevice(&cur) == cudaSuccess && cur != prev) cudaSetDevice(prev);
    }
};

template <typename T>
bool alloc(pulsar_ctx* c, T** p, size_t count) {
    if (c->n_allocs >= pulsar_ctx::kMaxAllocs) return false;
    void* q = nullptr;
    if (cudaMalloc(&q, count * sizeof(T) > 0 ? count * sizeof(T) : 16) != cudaSuccess) return false;
    c->allocs[c->n_allocs++] = q;
    *p = static_cast<T*>(q);
    return true;
}

void free_all(pulsar_ctx* c) {
    for (int i = 0; i < c->n_allocs; ++i) cudaFree(c->allocs[i]);
    c->n_allocs = 0;
    if (c->host_state) cudaFreeHost(c->host_state);
    c->host_state = nullptr;
}

bool finite_pos(float v) { return v > 0.0f && v < 3.0e38f; }

}  // namespace

extern "C" {

const char* pulsar_strerror(int code) {
    switch (code) {
        case PULSAR_OK: return "ok";
        case PULSAR_ERR_ARG: return "invalid argument";
        case PULSAR_ERR_CUDA: return "CUDA runtime error";
        case PULSAR_ERR_CAPACITY: return "sphere-tile pairs exceed max_pairs";
        case PULSAR_ERR_STATE: return "call out of order";
        case PULSAR_ERR_NOMEM: return "workspace allocation failed";
        case PULSAR_ERR_TIMEOUT: return "a bounded wait on the tensor cores gave up";
        case PULSAR_ERR_INTERNAL: return "a device index check failed (debug build)";
        default: return "unknown error";
    }
}

int pulsar_create(pulsar_ctx_t* out, int device, int64_t max_spheres, int64_t max_pairs,
                  int32_t max_width, int32_t max_height, int32_t max_channels,
                  int32_t max_track) {
    return pulsar_create_cams(out, device, max_spheres, max_pairs, max_width, max_height,
                              max_channels, max_track, 1);
}

int pulsar_create_cams(pulsar_ctx_t* out, int device, int64_t max_spheres, int64_t max_pairs,
                       int32_t max_width, int32_t max_height, int32_t max_channels,
                       int32_t max_track, int32_t max_cams) {
    PULSAR_TRACE("pulsar_create_cams");
    if (!out) return PULSAR_ERR_ARG;
    *out = nullptr;
    // sphere indices stay 32-bit with a launch's worth of margin below 2^31
    if (max_spheres < 0 || max_spheres > 0x7fff0000LL || max_pairs < 1 ||
        max_pairs >= 0xffffffffLL || max_width < 1 || max_width > 65535 || max_height < 1 ||
        max_height > 65535 || max_channels < 1 || max_channels > kMaxChannels ||
        max_track < 1 || max_track > kMaxTrack || max_cams < 1 || max_cams > kMaxCams)
        return PULSAR_ERR_ARG;
    // every per-camera buffer holds max_cams blocks, and indices into them are 32-bit
    if ((double)max_cams * (double)max_spheres >= 4294967296.0 ||
        (double)max_cams * max_width * max_height * max_track >= 4294967296.0)
        return PULSAR_ERR_ARG;
    int ndev = 0;
    if (cudaGetDeviceCount(&ndev) != cudaSuccess) return PULSAR_ERR_CUDA;
    if (device < 0 || device >= ndev) return PULSAR_ERR_ARG;
    DeviceGuard guard(device);
    pulsar_ctx* c = new (std::nothrow) pulsar_ctx();
    if (!c) return PULSAR_ERR_NOMEM;
    c->device = device;
    c->max_n = max_spheres;
    c->max_pairs = max_pairs;
    c->max_w = max_width;
    c->max_h = max_height;
    c->max_c = max_channels;
    c->max_t = max_track;
    c->max_cams = max_cams;
    c->max_tiles = (int64_t)((max_width + kTile - 1) / kTile) * ((max_height + kTile - 1) / kTile);
    c->max_pix = (int64_t)max_width * max_height;
    const size_t K = (size_t)max_cams;
    const size_t N = (size_t)(max_spheres > 0 ? max_spheres : 1);
    const size_t B = (size_t)c->max_tiles, P = (size_t)c->max_pix;
    Workspace& w = c->ws;
    bool ok = alloc(c, &w.rec, K * N) && alloc(c, &w.gacc, K * N) &&
              alloc(c, &w.gacc2, N) && alloc(c, &w.hitcnt, K * N) &&
              alloc(c, &w.tile_count, K * B) && alloc(c, &w.tile_start, K * B + 1) &&
              alloc(c, &w.long_tiles, K * B) &&
              alloc(c, &w.staged, (size_t)max_pairs) &&
              alloc(c, &w.pairs, (size_t)max_pairs) && alloc(c, &w.pairs_alt, (size_t)max_pairs) &&
              alloc(c, &w.tile_ids, (size_t)max_pairs) && alloc(c, &w.mg, K * P) &&
              alloc(c, &w.wsum, K * P) && alloc(c, &w.ids, K * P * max_track) &&
              alloc(c, &w.dtr, K * P * max_track) && alloc(c, &w.nhits, K * P) &&
              alloc(c, &w.kpart, K * B * 4) && alloc(c, &w.rtpart, (N + 255) / 256 * K * 12) &&
              alloc(c, &w.state, 1);
    if (ok) ok = cudaMallocHost(&c->host_state, sizeof(DevState)) == cudaSuccess;
    if (ok) ok = prepare_forward() == cudaSuccess && prepare_bin() == cudaSuccess &&
                 prepare_backward() == cudaSuccess &&
                 prepare_shade(&c->shade) == cudaSuccess;
    if (ok) ok = cudaDeviceGetAttribute(&c->n_sms, cudaDevAttrMultiProcessorCount, device) ==
                 cudaSuccess;
    if (ok)
        ok = alloc(c, &w.shade_part, (size_t)c->shade.bwd_per_sm * c->n_sms * kShadeParams) &&
             alloc(c, &w.shade_img, shade_image_bytes());
    // zero-between-frames invariants
    if (ok)
        ok = cudaMemset(w.gacc, 0, K * N * sizeof(float4)) == cudaSuccess &&
             cudaMemset(w.gacc2, 0, N * sizeof(float4)) == cudaSuccess &&
             cudaMemset(w.hitcnt, 0, K * N * sizeof(float)) == cudaSuccess &&
             cudaMemset(w.tile_count, 0, K * B * sizeof(uint32_t)) == cudaSuccess &&
             cudaMemset(w.tile_start, 0, (K * B + 1) * sizeof(uint32_t)) == cudaSuccess &&
             cudaMemset(w.state, 0, sizeof(DevState)) == cudaSuccess &&
             cudaDeviceSynchronize() == cudaSuccess;
    if (!ok) {
        free_all(c);
        delete c;
        cudaGetLastError();
        return PULSAR_ERR_NOMEM;
    }
    *out = c;
    return PULSAR_OK;
}

int pulsar_destroy(pulsar_ctx_t c) {
    PULSAR_TRACE("pulsar_destroy");
    if (!c) return PULSAR_ERR_ARG;
    DeviceGuard guard(c->device);
    cudaDeviceSynchronize();
    free_all(c);
    delete c;
    return PULSAR_OK;
}

int pulsar_project(pulsar_ctx_t c, const float* pos, const float* radius, const float* opacity,
                   int64_t n, const pulsar_camera_t* cam, const pulsar_params_t* prm,
                   void* stream) {
    return pulsar_project_cams(c, pos, radius, opacity, n, cam, 1, prm, stream);
}

int pulsar_project_cams(pulsar_ctx_t c, const float* pos, const float* radius,
                        const float* opacity, int64_t n, const pulsar_camera_t* cams,
                        int32_t n_cams, const pulsar_params_t* prm, void* stream) {
    PULSAR_TRACE("pulsar_project_cams");
    if (!c || !cams || !prm || n < 0 || n > c->max_n || n_cams < 1 || n_cams > c->max_cams)
        return PULSAR_ERR_ARG;
    if (n > 0 && (!pos || !radius || !opacity)) return PULSAR_ERR_ARG;
    for (int k = 0; k < n_cams; ++k) {
        const pulsar_camera_t* cam = cams + k;
        if (cam->width < 1 || cam->height < 1 || cam->width > c->max_w || cam->height > c->max_h ||
            cam->width != cams[0].width || cam->height != cams[0].height)
            return PULSAR_ERR_ARG;
        if (!finite_pos(cam->fx) || !finite_pos(cam->fy) || !(cam->znear > 0.0f) ||
            !(cam->zfar > cam->znear) || (cam->orthographic != 0 && cam->orthographic != 1))
            return PULSAR_ERR_ARG;
    }
    if (!finite_pos(prm->gamma) || !(prm->bg_eps >= 0.0f) || !(prm->stop_tau >= 0.0f) ||
        !(prm->kappa >= 0.0f) || !(prm->geom_min_area >= 0.0f) || prm->n_track < 1 ||
        prm->n_track > c->max_t || prm->channels < 1 || prm->channels > c->max_c)
        return PULSAR_ERR_ARG;
    // normalised gradients are defined per image: one camera at a time
    if ((prm->flags & PULSAR_FLAG_NORMALIZE_GRADS) && n_cams > 1) return PULSAR_ERR_ARG;
    DeviceGuard guard(c->device);
    cudaStream_t s = as_stream(stream);
    if (c->counts_dirty) {
        // a previous frame was projected but never binned: its counts and staged
        // pair cursor are stale
        cudaError_t e = cudaMemsetAsync(c->ws.tile_count, 0,
                                        (size_t)c->max_tiles * c->max_cams * 4, s);
        if (e == cudaSuccess)
            e = cudaMemsetAsync(&c->ws.state->pair_cursor, 0, sizeof(uint32_t), s);
        if (e != cudaSuccess) return PULSAR_ERR_CUDA;
    }
    for (int k = 0; k < n_cams; ++k) {
        const pulsar_camera_t* cam = cams + k;
        fill_frame(c->frames.f[k], cam->R, cam->t, cam->fx, cam->fy, cam->cx, cam->cy,
                   cam->width, cam->height, cam->znear, cam->zfar, cam->orthographic,
                   prm->gamma, prm->bg_eps, prm->stop_tau, prm->kappa, prm->geom_min_area,
                   prm->n_track, prm->channels, prm->flags, (int)n, (uint32_t)c->max_pairs, k,
                   n_cams);
    }
    c->n_cams = n_cams;
    c->pos = pos;
    cudaError_t e = launch_project(c->frames, c->ws, pos, radius, opacity, s);
    if (e != cudaSuccess) return PULSAR_ERR_CUDA;
    c->stage = 1;
    c->counts_dirty = true;
    return PULSAR_OK;
}

int pulsar_bin(pulsar_ctx_t c, void* stream) {
    PULSAR_TRACE("pulsar_bin");
    if (!c) return PULSAR_ERR_ARG;
    if (c->stage < 1) return PULSAR_ERR_STATE;
    if (c->stage >= 2) return PULSAR_ERR_STATE;   // counts were consumed by the first bin
    DeviceGuard guard(c->device);
    cudaError_t e = launch_bin(c->frames, c->ws, as_stream(stream));
    if (e != cudaSuccess) return PULSAR_ERR_CUDA;
    c->stage = 2;
    c->counts_dirty = false;
    return PULSAR_OK;
}

int pulsar_forward(pulsar_ctx_t c, const float* features, const float* bg, float* image,
                   void* stream) {
    PULSAR_TRACE("pulsar_forward");
    if (!c || !bg || !image) return PULSAR_ERR_ARG;
    if (c->frames.f[0].n > 0 && !features) return PULSAR_ERR_ARG;
    if (c->stage < 2) return PULSAR_ERR_STATE;
    DeviceGuard guard(c->device);
    cudaError_t e = launch_forward(c->frames, c->ws, features, bg, image, 0, as_stream(stream));
    if (e != cudaSuccess) return PULSAR_ERR_CUDA;
    c->stage = 3;
    c->acc_zeroed = true;
    return PULSAR_OK;
}

int pulsar_backward(pulsar_ctx_t c, const float* features, const float* bg, const float* image,
                    const float* grad_image, float* grad_pos, float* grad_radius,
                    float* grad_opacity, float* grad_features, float* grad_cam, void* stream) {
    PULSAR_TRACE("pulsar_backward");
    (void)bg;   // the background enters through the forward image only
    if (!c) return PULSAR_ERR_ARG;
    if (c->stage < 3) return PULSAR_ERR_STATE;
    if (!grad_pos && !grad_radius && !grad_opacity && !grad_features && !grad_cam)
        return PULSAR_OK;   // nothing requested (Pulsar Sec. B.2)
    if (!image || !grad_image || (c->frames.f[0].n > 0 && !features)) return PULSAR_ERR_ARG;
    DeviceGuard guard(c->device);
    cudaStream_t s = as_stream(stream);
    const Frame& f = c->frames.f[0];
    const size_t n = (size_t)f.n;
    // with C <= 3 the opacity and feature gradients are accumulated in the
    // workspace and written out by the finalize; otherwise straight into the
    // caller's arrays, which start at zero
    if (f.channels > 3) {
        if (grad_opacity && n && cudaMemsetAsync(grad_opacity, 0, n * 4, s) != cudaSuccess)
            return PULSAR_ERR_CUDA;
        if (grad_features && n &&
            cudaMemsetAsync(grad_features, 0, n * (size_t)f.channels * 4, s) != cudaSuccess)
            return PULSAR_ERR_CUDA;
    }
    cudaError_t e = launch_backward(c->frames, c->ws, c->pos, features, image, grad_image, grad_pos,
                                    grad_radius, grad_opacity, grad_features, grad_cam,
                                    c->acc_zeroed, s);
    c->acc_zeroed = false;
    return cuda_err(e);
}

int pulsar_shade_forward(pulsar_ctx_t c, const float* features, const float* params, float* rgb,
                         void* stream) {
    PULSAR_TRACE("pulsar_shade_forward");
    if (!c || !features || !params || !rgb) return PULSAR_ERR_ARG;
    if ((reinterpret_cast<uintptr_t>(features) & 15u) != 0) return PULSAR_ERR_ARG;
    if (c->stage < 1) return PULSAR_ERR_STATE;
    if (c->frames.f[0].channels != 16) return PULSAR_ERR_ARG;
    DeviceGuard guard(c->device);
    return cuda_err(launch_shade_forward(c->frames, c->ws, features, params, rgb,
                                         c->shade.fwd_per_sm * c->n_sms, as_stream(stream)));
}

int pulsar_shade_backward(pulsar_ctx_t c, const float* features, const float* params,
                          const float* grad_rgb, float* grad_features, float* grad_params,
                          void* stream) {
    PULSAR_TRACE("pulsar_shade_backward");
    if (!c || !features || !params || !grad_rgb || !grad_params) return PULSAR_ERR_ARG;
    if ((reinterpret_cast<uintptr_t>(features) & 15u) != 0 ||
        (reinterpret_cast<uintptr_t>(grad_features) & 15u) != 0)
        return PULSAR_ERR_ARG;
    if (c->stage < 1) return PULSAR_ERR_STATE;
    if (c->frames.f[0].channels != 16) return PULSAR_ERR_ARG;
    DeviceGuard guard(c->device);
    return cuda_err(launch_shade_backward(c->frames, c->ws, features, params, grad_rgb,
                                          grad_features, grad_params,
                                          c->shade.bwd_per_sm * c->n_sms, as_stream(stream)));
}

int pulsar_status(pulsar_ctx_t c, void* stream, int64_t* n_pairs, int64_t* n_hits) {
    PULSAR_TRACE("pulsar_status");
    if (!c) return PULSAR_ERR_ARG;
    DeviceGuard guard(c->device);
    cudaStream_t s = as_stream(stream);
    if (cudaMemcpyAsync(c->host_state, c->ws.state, sizeof(DevState), cudaMemcpyDeviceToHost,
                        s) != cudaSuccess)
        return PULSAR_ERR_CUDA;
    if (cudaStreamSynchronize(s) != cudaSuccess) return PULSAR_ERR_CUDA;
    const DevState& h = *c->host_state;
    if (n_pairs) *n_pairs = (int64_t)h.n_pairs;
    if (n_hits) *n_hits = (int64_t)h.hits;
    if (h.inject) {
        const uint32_t zero = 0;
        cudaMemcpy(&c->ws.state->inject, &zero, sizeof(zero), cudaMemcpyHostToDevice);
    }
    if (h.error) {
        const uint32_t zero = 0;
        cudaMemcpy(&c->ws.state->error, &zero, sizeof(zero), cudaMemcpyHostToDevice);
        if (h.error & kErrCapacity) return PULSAR_ERR_CAPACITY;
        if (h.error & kErrTimeout) return PULSAR_ERR_TIMEOUT;
        if (h.error & kErrBounds) return PULSAR_ERR_INTERNAL;
    }
    return PULSAR_OK;
}

int pulsar_debug_inject(pulsar_ctx_t c, int what, void* stream) {
    PULSAR_TRACE("pulsar_debug_inject");
    if (!c || (what & ~(int)kInjectShadeTimeout) != 0) return PULSAR_ERR_ARG;
    DeviceGuard guard(c->device);
    const uint32_t v = (uint32_t)what;
    return cuda_err(cudaMemcpyAsync(&c->ws.state->inject, &v, sizeof(v), cudaMemcpyHostToDevice,
                                    as_stream(stream)));
}

int64_t pulsar_debug_copy(pulsar_ctx_t c, int what, void* dst, int64_t bytes, void* stream) {
    PULSAR_TRACE("pulsar_debug_copy");
    if (!c || bytes < 0) return PULSAR_ERR_ARG;
    DeviceGuard guard(c->device);
    cudaStream_t s = as_stream(stream);
    const Frame& f = c->frames.f[0];
    const int K = c->n_cams > 0 ? c->n_cams : 1;
    // every per-camera array covers the batch's cameras, camera after camera
    const int64_t n = f.n, P1 = (int64_t)f.width * f.height, P = P1 * K;
    const int64_t B = (int64_t)f.n_tiles * K;
    const void* src = nullptr;
    int64_t size = 0;
    switch (what) {
        case PULSAR_DBG_RECORDS: src = c->ws.rec; size = n * K * (int64_t)sizeof(SphereRec); break;
        case PULSAR_DBG_TILE_OFFSETS: src = c->ws.tile_start; size = (B + 1) * 4; break;
        case PULSAR_DBG_TILE_IDS: {
            uint32_t m = 0;
            if (cudaMemcpyAsync(&m, &c->ws.state->n_pairs, 4, cudaMemcpyDeviceToHost, s) !=
                    cudaSuccess ||
                cudaStreamSynchronize(s) != cudaSuccess)
                return PULSAR_ERR_CUDA;
            src = c->ws.tile_ids;
            size = (int64_t)(m < c->max_pairs ? m : c->max_pairs) * 4;
            break;
        }
        case PULSAR_DBG_MG: src = c->ws.mg; size = P * 4; break;
        case PULSAR_DBG_WSUM: src = c->ws.wsum; size = P * 4; break;
        case PULSAR_DBG_IDS: {
            // the buffer holds each tracked hit's position in its tile list;
            // report sphere ids
            size = P * f.n_track * 4;
            if (!dst) return size;
            if (bytes > size) return PULSAR_ERR_ARG;
            std::vector<int32_t> pos((size_t)P * f.n_track);
            std::vector<uint32_t> starts((size_t)B + 1);
            uint32_t m = 0;
            if (cudaMemcpyAsync(pos.data(), c->ws.ids, (size_t)size, cudaMemcpyDeviceToHost, s) !=
                    cudaSuccess ||
                cudaMemcpyAsync(starts.data(), c->ws.tile_start, starts.size() * 4,
                                cudaMemcpyDeviceToHost, s) != cudaSuccess ||
                cudaMemcpyAsync(&m, &c->ws.state->n_pairs, 4, cudaMemcpyDeviceToHost, s) !=
                    cudaSuccess ||
                cudaStreamSynchronize(s) != cudaSuccess)
                return PULSAR_ERR_CUDA;
            m = m < c->max_pairs ? m : (uint32_t)c->max_pairs;
            std::vector<uint32_t> list(m > 0 ? m : 1);
            if (m > 0 && (cudaMemcpy(list.data(), c->ws.tile_ids, (size_t)m * 4,
                                     cudaMemcpyDeviceToHost) != cudaSuccess))
                return PULSAR_ERR_CUDA;
            for (int64_t q = 0; q < (int64_t)pos.size(); ++q) {
                if (pos[q] < 0) continue;
                const int64_t pg = q % P;               // pixel of the batch
                const int64_t cam = pg / P1, px = pg % P1;
                const int64_t tile = cam * f.n_tiles + ((px / f.width) / kTile) * f.tiles_x +
                                     (px % f.width) / kTile;
                const uint64_t at = (uint64_t)starts[tile] + (uint64_t)pos[q];
                pos[q] = at < m ? (int32_t)list[at] : -1;
            }
            if (bytes > 0 &&
                cudaMemcpy(dst, pos.data(), (size_t)bytes, cudaMemcpyDefault) != cudaSuccess)
                return PULSAR_ERR_CUDA;
            return PULSAR_OK;
        }
        case PULSAR_DBG_NHITS: src = c->ws.nhits; size = P * 4; break;
        default: return PULSAR_ERR_ARG;
    }
    if (!dst) return size;
    if (bytes > size) return PULSAR_ERR_ARG;
    if (bytes == 0) return PULSAR_OK;
    if (cudaMemcpyAsync(dst, src, (size_t)bytes, cudaMemcpyDefault, s) != cudaSuccess)
        return PULSAR_ERR_CUDA;
    if (cudaStreamSynchronize(s) != cudaSuccess) return PULSAR_ERR_CUDA;
    return PULSAR_OK;
}

}  // extern "C"
