/*
 * pulsar.h -- C ABI of the GB300 (sm_103a) tile-based differentiable sphere
 * renderer.
 *
 * The operation (Pulsar: Efficient Sphere-based Neural Rendering, Sec. 3.2
 * and App. A "Prelude"): a scene of spheres -- position, radius, opacity and
 * a feature payload (Sec. 3.1) -- and a pinhole camera (rotation R,
 * translation t, intrinsics K) are mapped to a feature image.  Each pixel
 * blends every sphere its ray hits, front to back, with weights
 *     w = o * d * exp(o * z~ / gamma),  d = 1 - rho / r_eff,
 *     z~ = (zfar - c.z) / (zfar - znear)  (normalised device depth),
 * rho the orthogonal ray-to-centre distance, plus a background of weight
 * exp(eps / gamma):  F = (sum w f + w_bg f_bg) / (sum w + w_bg).
 * Gradients of a scalar loss flow to sphere position, radius, opacity,
 * features and to R, t, K through only the first n_track hits of every
 * pixel (Sec. 2, B.1.3, B.1.4, B.2).
 *
 * Call sequence per frame, all asynchronous on the caller's stream:
 *     pulsar_project -> pulsar_bin -> pulsar_forward [-> pulsar_backward]
 * No call synchronises the host except pulsar_status and pulsar_debug_copy
 * into pageable host memory.
 *
 * Conventions for every entry point:
 *   - Tensors are caller-owned, C-contiguous float32 DEVICE pointers unless
 *     stated; streams are `cudaStream_t` values passed as `void*` (NULL = the
 *     legacy default stream).
 *   - The context owns only its workspace, allocated once by pulsar_create.
 *   - Return 0 on success or a negative PULSAR_ERR_* code; nothing throws.
 *     Argument errors are detected on the host before anything is enqueued.
 *     Errors raised on the device (capacity overflow) are latched in the
 *     context and returned by pulsar_status.
 *   - Inputs passed to pulsar_project (pos) and pulsar_forward (features)
 *     must stay valid and unmodified until the last call of the frame has
 *     executed on the stream; the backward pass reads them again.
 *   - One context renders one camera at a time; calls on one context must be
 *     issued in order on one stream.
 */
#ifndef PULSAR_H_
#define PULSAR_H_

#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* ---------------------------------------------------------- error codes -- */
#define PULSAR_OK            0
#define PULSAR_ERR_ARG      -1  /* invalid argument (NULL, size, limit) */
#define PULSAR_ERR_CUDA     -2  /* a CUDA runtime call failed */
#define PULSAR_ERR_CAPACITY -3  /* more sphere-tile pairs than max_pairs */
#define PULSAR_ERR_STATE    -4  /* call out of order (e.g. forward before bin) */
#define PULSAR_ERR_NOMEM    -5  /* workspace allocation failed */
#define PULSAR_ERR_INTERNAL -7  /* debug build only: a device index check failed (the access
                                  was skipped; the frame is invalid) */
#define PULSAR_ERR_TIMEOUT  -6  /* a bounded wait on the tensor cores gave up: the frame is
                                  invalid and, since work may still have been in flight,
                                  the context should be destroyed and recreated */

/* --------------------------------------------------------------- flags -- */
/* Drop position/radius gradients (and the sphere's share of the camera
 * gradient) of spheres whose projected area pi*(f_min*r/c.z)^2 (pinhole;
 * pi*(f_min*r)^2 orthographic) is at most
 * geom_min_area px^2 (Pulsar Sec. 6, App. A: "more than three projected
 * pixels").  Opacity and feature gradients are always kept. */
#define PULSAR_FLAG_GEOM_CUTOFF   0x1u
/* Also record the number of hits of every pixel (for tests; costs 4 B/px). */
#define PULSAR_FLAG_COUNT_HITS    0x2u
/* Normalised gradients (Pulsar Sec. B.2): a sphere's position, radius,
 * opacity and feature gradients are divided by the number of pixels whose
 * tracked set holds it; its share of the R, t and K gradients is multiplied by
 * 1e-3 / A, A = pi*(f_min*r_eff/c.z)^2 px^2 (orthographic: pi*(f_min*r_eff)^2),
 * the area of the disc it is rendered with.  Not the derivative of anything:
 * an optimisation aid, off by default. */
#define PULSAR_FLAG_NORMALIZE_GRADS 0x4u
/* Gaussian footprint (the splat variant of the NuRec pages): the distance
 * factor d = 1 - rho/r_eff is replaced by an isotropic Gaussian of sigma =
 * r_eff/3 over the same support, shifted and scaled to run from 1 at the
 * centre to 0 at the rim: d = (exp(-4.5 (rho/r_eff)^2) - e^-4.5) /
 * (1 - e^-4.5).  Decisions (support, tile lists, tracked ids) unchanged. */
#define PULSAR_FLAG_GAUSSIAN      0x8u

/* Camera, OpenCV axes (x right, y down, z forward).  R is the world->camera
 * rotation, row-major: c = R p + t.  Pixel (x, y) has its centre at
 * (x + 0.5, y + 0.5).  Pinhole (orthographic = 0): the pixel's ray leaves the
 * origin along ((x + 0.5 - cx)/fx, (y + 0.5 - cy)/fy, 1); fx, fy in pixels.
 * Orthographic (orthographic = 1; Pulsar Sec. B.1.1 bounds projections for
 * both): the ray leaves ((x + 0.5 - cx)/fx, (y + 0.5 - cy)/fy, 0) along +z;
 * fx, fy in pixels per world unit, and the kappa floor of the radius is
 * kappa/min(fx, fy).  Spheres are kept when znear < c.z < zfar and
 * r_eff < c.z.  (Pulsar Sec. 3.2: R, t, K; App. A.) */
typedef struct pulsar_camera {
    float R[9];
    float t[3];
    float fx, fy, cx, cy;
    int32_t width, height;   /* 1 .. 65535 */
    float znear, zfar;       /* 0 < znear < zfar */
    int32_t orthographic;    /* 0: pinhole, 1: orthographic; other values: PULSAR_ERR_ARG */
} pulsar_camera_t;

/* Blend and gradient parameters. */
typedef struct pulsar_params {
    float gamma;          /* blend temperature, > 0 (0.1 in the shipped configs) */
    float bg_eps;         /* background "depth" eps in exp(eps/gamma), >= 0 */
    float stop_tau;       /* early-stop tolerance (Pulsar Sec. 3.2, B.1.3); 0 = exact */
    float kappa;          /* minimum projected radius in px (Pulsar Sec. B.1.1), >= 0 */
    float geom_min_area;  /* px^2 threshold of PULSAR_FLAG_GEOM_CUTOFF */
    int32_t n_track;      /* hits per pixel that receive gradients, 1 .. max_track */
    int32_t channels;     /* feature channels C, 1 .. max_channels */
    uint32_t flags;       /* PULSAR_FLAG_* */
} pulsar_params_t;

typedef struct pulsar_ctx* pulsar_ctx_t;

/* Create a context on CUDA device `device` and allocate its workspace for at
 * most max_spheres spheres, max_pairs sphere-tile pairs, images up to
 * max_width x max_height, max_channels channels and max_track tracked hits.
 * The workspace is owned by the context and freed by pulsar_destroy.
 * Errors: PULSAR_ERR_ARG (NULL out, non-positive limit, max_spheres >
 * 0x7fff0000 (sphere indices are 32-bit), max_track > 16, max_channels > 64,
 * max_pairs >= 2^32), PULSAR_ERR_NOMEM, PULSAR_ERR_CUDA. */
int pulsar_create(pulsar_ctx_t* out, int device, int64_t max_spheres, int64_t max_pairs,
                  int32_t max_width, int32_t max_height, int32_t max_channels,
                  int32_t max_track);

/* As pulsar_create, for batches of up to max_cams cameras (1 .. 8) rendered
 * together by pulsar_project_cams (every per-camera buffer of the workspace
 * is allocated max_cams times).  pulsar_create(...) is
 * pulsar_create_cams(..., 1).  Errors: as pulsar_create, and PULSAR_ERR_ARG
 * if max_cams is out of range or max_cams * max_spheres or
 * max_cams * max_width * max_height * max_track reaches 2^32. */
int pulsar_create_cams(pulsar_ctx_t* out, int device, int64_t max_spheres, int64_t max_pairs,
                       int32_t max_width, int32_t max_height, int32_t max_channels,
                       int32_t max_track, int32_t max_cams);

/* Release the context and its workspace (synchronises the device). */
int pulsar_destroy(pulsar_ctx_t ctx);

/* Step 0 of the forward pass (Pulsar Sec. B.1.1): for each of the n spheres
 * compute its camera-space centre, cull it, floor its radius so it covers at
 * least one pixel, project its centre, bound its pixel rectangle without
 * trigonometry, and form its depth key c.z - r_eff; count its 16x16 tiles.
 *   pos     [n,3]  world positions
 *   radius  [n]    radii (> 0)
 *   opacity [n]    opacities
 * n may be 0.  Errors: PULSAR_ERR_ARG (NULL pointers with n > 0, n above
 * max_spheres, image above the create limits, invalid params). */
int pulsar_project(pulsar_ctx_t ctx, const float* pos, const float* radius,
                   const float* opacity, int64_t n, const pulsar_camera_t* cam,
                   const pulsar_params_t* params, void* stream);

/* Batched form of pulsar_project: the same spheres seen by n_cams cameras
 * (1 .. the context's max_cams, equal width and height; host array cams
 * [n_cams]) in one launch that loads every sphere once.  pulsar_bin,
 * pulsar_forward and pulsar_backward then cover all cameras in one launch
 * each: the tiles of all cameras share one list space and the blocks run
 * over all of them.  Image-shaped arrays (image, grad_image) become
 * [n_cams,H,W,C], grad_cam becomes [n_cams,16], and the sphere gradients are
 * summed over the cameras (L = sum over cameras and pixels of <G, F>).
 * pulsar_project(...) is pulsar_project_cams with one camera.  Errors: as
 * pulsar_project, and PULSAR_ERR_ARG for n_cams out of range, cameras of
 * different sizes, or PULSAR_FLAG_NORMALIZE_GRADS with more than one camera
 * (normalised gradients are defined per image). */
int pulsar_project_cams(pulsar_ctx_t ctx, const float* pos, const float* radius,
                        const float* opacity, int64_t n, const pulsar_camera_t* cams,
                        int32_t n_cams, const pulsar_params_t* params, void* stream);

/* Tile binning (Pulsar Sec. 3.2 "sorted by earliest possible intersection",
 * B.1.1, B.1.2): scan the tile counts, emit one (key, id) pair per covered
 * tile and sort every tile's list by (key, sphere id).  The pair count M
 * stays on the device; if M > max_pairs the frame is invalid and
 * pulsar_status returns PULSAR_ERR_CAPACITY.  Errors: PULSAR_ERR_STATE if
 * pulsar_project was not called for this frame. */
int pulsar_bin(pulsar_ctx_t ctx, void* stream);

/* Forward pass (Pulsar Sec. B.1.2-B.1.4): composite every pixel front to
 * back and store the backward-information buffer (the ids of its first
 * n_track hits, the stabiliser and the normaliser).
 *   features [n,C]  per-sphere payload
 *   bg       [C]    background feature f_bg
 *   image    [H,W,C] output, overwritten
 * Errors: PULSAR_ERR_ARG (NULL pointer), PULSAR_ERR_STATE (bin missing). */
int pulsar_forward(pulsar_ctx_t ctx, const float* features, const float* bg, float* image,
                   void* stream);

/* Backward pass (Pulsar Sec. B.2): gradients of L = sum_pixels <G, F> through
 * the tracked hits.  features, bg and image are those of pulsar_forward;
 * grad_image [H,W,C] is G.  Outputs, each overwritten, each may be NULL
 * (not requested; if all are NULL nothing is enqueued, Pulsar Sec. B.2):
 *   grad_pos [n,3], grad_radius [n], grad_opacity [n], grad_features [n,C],
 *   grad_cam [16] = dL/dR (9, row-major), dL/dt (3), dL/d(fx, fy, cx, cy).
 * Errors: PULSAR_ERR_ARG, PULSAR_ERR_STATE (forward missing). */
int pulsar_backward(pulsar_ctx_t ctx, const float* features, const float* bg,
                    const float* image, const float* grad_image, float* grad_pos,
                    float* grad_radius, float* grad_opacity, float* grad_features,
                    float* grad_cam, void* stream);

/* Synchronise `stream`, then report the latched device error of the last
 * frame (PULSAR_OK, PULSAR_ERR_CAPACITY, PULSAR_ERR_TIMEOUT; the debug build
 * also PULSAR_ERR_INTERNAL) and clear it.  n_pairs (M) and
 * n_hits (hit pairs composited by the last forward) may be NULL. */
int pulsar_status(pulsar_ctx_t ctx, void* stream, int64_t* n_pairs, int64_t* n_hits);

/* Per-pixel neural shading (Pulsar Sec. 3.3: a per-pixel network turns the
 * rendered feature map into RGB; Sec. 5.2: a shared fully-connected model
 * conditioned on the pixel's view direction) of the current frame's cameras,
 * on the tensor cores.  The network (the pages print none; a reading):
 *   x = [F_p (16 channels), v_p (unit view direction in camera space)],
 *   h1 = ReLU(W1 x + b1), h2 = ReLU(W2 h1 + b2), y = W3 h2 + b3,
 *   19 -> 64 -> 64 -> 3, every matrix operand rounded to bfloat16 (nearest
 *   even), fp32 accumulation and biases.
 *   features [K,H,W,16]  feature images of the frame's K cameras (K >= 1),
 *                        16-byte aligned; the frame must have 16 channels
 *   params   [5635]      W1 [64,19], b1 [64], W2 [64,64], b2 [64], W3 [3,64],
 *                        b3 [3], float32, row-major, concatenated
 *   rgb      [K,H,W,3]   output, overwritten
 * Requires pulsar_project (it takes the cameras from the frame).  Errors:
 * PULSAR_ERR_ARG (NULL, misaligned features, channels != 16),
 * PULSAR_ERR_STATE (no frame); a tensor-core wait that gives up is latched
 * and reported by pulsar_status as PULSAR_ERR_TIMEOUT. */
int pulsar_shade_forward(pulsar_ctx_t ctx, const float* features, const float* params,
                         float* rgb, void* stream);

/* Gradients of L = sum_p <grad_rgb_p, y_p> for the shading above, on the
 * tensor cores (the same bf16 operands; the roundings are passed straight
 * through):
 *   g2 = (W3^T dY) * [z2 > 0],  g1 = (W2^T g2) * [z1 > 0],  dF = (W1^T g1)[:16],
 *   dW1 = sum_p g1 x^T, db1 = sum_p g1, dW2 = sum_p g2 h1^T, db2 = sum_p g2,
 *   dW3 = sum_p dY h2^T, db3 = sum_p dY   (z the pre-activations),
 * with dY, g2, g1 rounded to bfloat16 where they enter a product.
 *   features      [K,H,W,16]  as for pulsar_shade_forward (16-byte aligned)
 *   params        [5635]      as for pulsar_shade_forward
 *   grad_rgb      [K,H,W,3]   dL/d rgb
 *   grad_features [K,H,W,16]  output dL/dF, overwritten; 16-byte aligned;
 *                             NULL skips it
 *   grad_params   [5635]      output dL/d params, overwritten (same layout as
 *                             params; summed in a fixed order: reproducible)
 * Errors as for pulsar_shade_forward (PULSAR_ERR_ARG also for NULL grad_rgb
 * or grad_params and a misaligned grad_features). */
int pulsar_shade_backward(pulsar_ctx_t ctx, const float* features, const float* params,
                          const float* grad_rgb, float* grad_features, float* grad_params,
                          void* stream);

/* Test hook for failure detection without a GPU fault.  With
 * PULSAR_INJECT_SHADE_TIMEOUT the shading kernels issue no tensor-core work,
 * so their bounded waits (0.25 s of wall time each) run out: the call still
 * completes, frees its tensor memory, and pulsar_status reports
 * PULSAR_ERR_TIMEOUT.  The injection stays armed until pulsar_status has
 * reported (which clears it); 0 disarms it.  Enqueued on `stream`.  Errors:
 * PULSAR_ERR_ARG (NULL context, unknown bits). */
#define PULSAR_INJECT_SHADE_TIMEOUT 1
int pulsar_debug_inject(pulsar_ctx_t ctx, int what, void* stream);

/* Static string for an error code. */
const char* pulsar_strerror(int code);

/* Internal arrays of the last frame, for tests (layouts are not a stable
 * interface).  Copies `bytes` bytes (at most the array's size for the frame)
 * into dst (host or device; cudaMemcpyDefault).  Returns the array's size in
 * bytes for the current frame if dst is NULL, else PULSAR_OK or an error.
 * For a batch of K cameras every array holds K per-camera blocks, camera
 * after camera (records [K][n], tiles [K*B], pixels [K*H*W]); the tile lists
 * of all cameras share one offsets array.
 *   PULSAR_DBG_RECORDS   [n] 64-byte sphere records, 16 x 32-bit words (written for
 *                        the frame's kept spheres only; a culled sphere's record
 *                        holds whatever it held before):
 *                        0-3   u_hi, u_lo, v_hi, v_lo  projected centre (float pairs)
 *                        4-6   exponent log2(e) o z~/gamma as hi, lo; opacity o
 *                        7     flags: 1 kept, 2 radius on the kappa floor, 4 geometry cut
 *                        8-11  (c.z/r_eff)^2 as hi, lo; c.z; r_eff
 *                        12-13 pixel rectangle x0 | x1 << 16, y0 | y1 << 16
 *                        14-15 s2 = (r_eff/c.z)^2, depth key c.z - r_eff
 *   PULSAR_DBG_TILE_OFFSETS [B+1] uint32 tile list offsets
 *   PULSAR_DBG_TILE_IDS  [M] uint32 sorted tile lists
 *   PULSAR_DBG_MG        [H*W] float  stabiliser log2(e) m / gamma
 *   PULSAR_DBG_WSUM      [H*W] float  normaliser in the exp(-m/gamma) frame
 *   PULSAR_DBG_IDS       [n_track][H*W] int32 tracked sphere ids, -1 padded (the buffer
 *                        itself holds list positions; they are translated here)
 *   PULSAR_DBG_NHITS     [H*W] int32 hits per pixel (PULSAR_FLAG_COUNT_HITS) */
#define PULSAR_DBG_RECORDS       1
#define PULSAR_DBG_TILE_OFFSETS  5
#define PULSAR_DBG_TILE_IDS      6
#define PULSAR_DBG_MG            7
#define PULSAR_DBG_WSUM          8
#define PULSAR_DBG_IDS           9
#define PULSAR_DBG_NHITS        10
int64_t pulsar_debug_copy(pulsar_ctx_t ctx, int what, void* dst, int64_t bytes, void* stream);

/* Forward render of one small frame that allocates no memory (the pages have
 * no counterpart: this entry point exists for callers that cannot call
 * cudaMalloc while they render -- plugins whose host framework owns the device
 * memory budget, fixed-footprint real-time renderers that must not risk an
 * allocation failure or its implicit synchronisation mid-frame).  It runs the
 * kernels of pulsar_project, pulsar_bin and pulsar_forward with all
 * intermediate arrays in one static device arena of about 8 MB that the
 * library reserves on every GPU that loads it, until the process exits.  No
 * context is needed; inputs and outputs are as for pulsar_project and
 * pulsar_forward.
 *   Limits: n <= 16384 spheres, at most 65536 sphere-tile pairs, width and
 *   height <= 256, n_track <= 8, channels <= 64.  Larger sizes return
 *   PULSAR_ERR_ARG without enqueueing anything; a frame with more pairs returns
 *   PULSAR_ERR_CAPACITY (the image is then not written).
 *   All calls share the arena, which keeps the last call's contents; each call
 *   clears what must start at zero.  Calls that overlap on the GPU race: the
 *   caller must serialise them.
 *   The first call on a device looks up the arena's device address and
 *   prepares the kernels; that first call should come before any stream
 *   capture.  Every call synchronises `stream` at its end to read the frame's
 *   status. */
int pulsar_render_noalloc(const float* pos, const float* radius, const float* opacity,
                          const float* features, int64_t n, const pulsar_camera_t* cam,
                          const pulsar_params_t* params, const float* bg, float* image,
                          void* stream);

#ifdef __cplusplus
}
#endif

#endif /* PULSAR_H_ */
