/*
 * gs.h — C ABI of the GB300 (sm_103a) library for the training step of a tile-based 3D Gaussian
 * splatting rasterizer: per-Gaussian preprocessing, tile binning with a stable radix sort,
 * front-to-back forward blending, the backward pass with aggregated per-Gaussian gradient
 * atomics, and the preprocessing backward.
 *
 * Method. A 3D Gaussian splatting scene is rendered with a rasterization pipeline and trained by
 * gradient descent from 2D images; its gradient computation is dominated by the atomic updates
 * that accumulate per-Gaussian gradients, which overwhelm the GPU's L2 atomic units (DISTWAR:
 * Fast Differentiable Rendering on Raster-based Rendering Pipelines, Abstract; ARC: Warp-level
 * Adaptive Atomic Reduction in GPUs to Accelerate Differentiable Rendering, Abstract). One view
 * runs the phases preprocessing, rendering and backward computation (Odin: Primitive-Level
 * Synchronization for Distributed Point-Based Neural Rendering, Figure 7); the five compute
 * entry points below are those phases.
 *
 * Conventions common to every call.
 *   - Pointers to arrays are DEVICE pointers, C-contiguous, row-major, owned by the caller. The
 *     library allocates no device memory and keeps no state between calls except a per-device
 *     error word (see gs_device_error) and a per-thread last-error message. The one exception is
 *     the end-to-end pair at the end of this header: gs_step_context_create allocates a context's
 *     device buffers, and gs_train_step_host takes HOST pointers for its inputs and outputs.
 *   - Projected records (gs_proj.rec) and 2D gradients (grad2d) must be 16-byte aligned; every
 *     other array must be 4-byte aligned (8-byte for keys). Misalignment returns GS_ERR_ARG.
 *   - `stream` is a cudaStream_t (NULL = legacy default stream). Calls enqueue work on it and
 *     return without synchronising, except gs_bin_and_sort, which synchronises once to read the
 *     number of duplicates.
 *   - The 3D path's kernels are launched with programmatic dependent launch (programmatic stream
 *     serialization): their blocks may be dispatched while the kernel enqueued before them is
 *     still running, but each waits for that kernel's completion and memory before reading
 *     anything it may write or writing anything it may read, so stream order holds as for
 *     ordinary launches.
 *   - Status codes: 0 on success, a negative GS_ERR_* otherwise. No C++ exception crosses the ABI.
 *     gs_last_error_message() describes the last failure of the calling thread.
 *   - Non-finite inputs are not errors: a Gaussian whose projection is not finite is culled.
 *   - Coordinates: the camera maps world points by p_cam = R p_world + t (x right, y down, z
 *     forward); pixel (i, j) has its centre at (i + 0.5, j + 0.5); the projected mean is
 *     (fx x / z + cx, fy y / z + cy). Images are 16x16-pixel tiles, T = ceil(W/16) ceil(H/16),
 *     numbered row-major.
 */
#ifndef GS_GB300_H
#define GS_GB300_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* ---- status codes ---------------------------------------------------------------------- */
#define GS_OK                0
#define GS_ERR_ARG          -1  /* null or misaligned pointer, negative or oversized count, bad option */
#define GS_ERR_CAPACITY     -2  /* more duplicates than `capacity`; *n_dup_out holds the number needed */
#define GS_ERR_CUDA         -3  /* a CUDA runtime call or kernel launch failed */
#define GS_ERR_TIMEOUT      -4  /* a bounded device-side wait gave up (reported by gs_device_error) */
#define GS_ERR_DEVICE_CHECK -5  /* a device-side consistency check failed (reported by gs_device_error) */

/* ---- backward accumulation modes (gs_options.bwd_mode) ------------------------------------
 * How gs_render_bwd accumulates the per-pixel gradient contributions of a Gaussian into its
 * per-Gaussian gradient. All modes compute the same sums (up to float rounding order).
 * A lane of the backward holds four pixels (one column of its warp's 16x8 block; two pixels of
 * an 8x8 block on images of fewer than two tiles per SM); a lane contributes when any of its
 * pixels does, and adds the sum of its pixels' values.
 *   DIRECT    every contributing lane adds its 9 values with its own global atomics: the
 *             L2-atomic-bound baseline that DISTWAR speeds up (DISTWAR, Abstract).
 *   WARP      the warp sums its lanes' contributions in registers (shuffle reduction) and one
 *             warp instruction issues the 9 global atomics (DISTWAR, Abstract: first key idea).
 *   ADAPTIVE  per warp and Gaussian: WARP when at least `adaptive_threshold` lanes contribute,
 *             DIRECT otherwise (DISTWAR, Abstract: second key idea; ARC, title). Default 28: on
 *             GB300 per-lane vector atomics are cheaper than the reduction's instructions unless
 *             nearly every lane contributes.
 *   SM        warps add into a per-tile shared-memory accumulator (warp-reduced when at least
 *             `adaptive_threshold` lanes contribute, per lane otherwise); the tile issues one set
 *             of global atomics per Gaussian and batch (one record per thread of the tile).   */
#define GS_BWD_DEFAULT  0
#define GS_BWD_DIRECT   1
#define GS_BWD_WARP     2
#define GS_BWD_ADAPTIVE 3
#define GS_BWD_SM       4

/* ---- batch staging in the render kernels (gs_options.staging) ---------------------------- */
#define GS_STAGE_DEFAULT 0
#define GS_STAGE_BULK    1  /* one bulk asynchronous copy (cp.async.bulk) per record, mbarrier completion */
#define GS_STAGE_LOADS   2  /* per-thread 16-byte loads through registers */

typedef struct gs_camera {
    float   R[9];        /* world -> camera rotation, row-major */
    float   t[3];        /* world -> camera translation */
    float   fx, fy;      /* focal lengths, pixels */
    float   cx, cy;      /* principal point, pixels (continuous coordinates) */
    int32_t width, height;
    float   bg[3];       /* background colour blended behind the last Gaussian */
} gs_camera;

/* Zero-initialised options select the defaults written beside each field. */
typedef struct gs_options {
    int32_t  bwd_mode;            /* GS_BWD_*; 0 = GS_BWD_DEFAULT (the ADAPTIVE mode) */
    int32_t  adaptive_threshold;  /* lanes, 1..33; 0 = 28 (ADAPTIVE) or 8 (SM) */
    int32_t  sh_degree;           /* 0..3 (K = (degree + 1)^2 SH coefficients per channel) */
    int32_t  staging;             /* GS_STAGE_*; 0 = GS_STAGE_BULK */
    float    near_z;              /* cull when the view-space depth is <= near_z; 0 = 0.2 */
    float    lowpass;             /* added to the 2D covariance diagonal, px^2; 0 = 0.3, < 0 = none */
    float    jacobian_clamp;      /* clamp x/z, y/z to +-jacobian_clamp * tan(half FOV) in the
                                     projection Jacobian; 0 = 1.3, < 0 = no clamp */
    uint32_t spin_limit;          /* iterations before a device-side wait gives up; 0 = 1<<18 */
} gs_options;

/* Trainable Gaussian parameters (inputs), N Gaussians, float32:
 *   mean3d [N][3], log_scale [N][3] (per-axis log standard deviation),
 *   quat [N][4] (w, x, y, z; normalised inside), opacity_logit [N] (opacity = sigmoid),
 *   sh [N][K][3] (real spherical-harmonic coefficients, channel last).                      */
typedef struct gs_params {
    const float* mean3d;
    const float* log_scale;
    const float* quat;
    const float* opacity_logit;
    const float* sh;
    int64_t      n;
} gs_params;

/* Projected Gaussians, written by gs_preprocess and read by the later calls.
 *   rec [N][12] float32, 16-byte aligned: (mean_x, mean_y, A, B, C, opacity, r, g, b, 0, 0, 0)
 *       with (A, B, C) the conic, i.e. the inverse 2D covariance [[A, B], [B, C]];
 *   depth [N] float32 view-space depth (sort key); radius [N] int32 (0 = culled);
 *   tiles_touched [N] uint32 (number of tiles in the Gaussian's tile rectangle).             */
typedef struct gs_proj {
    float*    rec;
    float*    depth;
    int32_t*  radius;
    uint32_t* tiles_touched;
    int64_t   n;
} gs_proj;

/* Preprocessing phase (Odin, Figure 7: "preprocessing"; the rasterization pipeline of DISTWAR,
 * Abstract). Per Gaussian: view-space position; float32 depth
 * fma(R20, x, fma(R21, y, fma(R22, z, t2))); cull when depth <= near_z; 3D covariance
 * R(q) diag(exp(2 log_scale)) R(q)^T; EWA projection with the pinhole Jacobian at the mean
 * (x/z, y/z clamped), plus `lowpass` on the diagonal; conic = inverse (cull when det <= 0);
 * radius = ceil(3 sqrt(largest eigenvalue)); tile rectangle of tiles overlapping the square of
 * half-side radius around the mean (cull when empty); opacity = sigmoid(logit); colour = real
 * SH of the view direction + 0.5, clamped below at 0. Culled Gaussians get a zero record,
 * radius 0 and tiles_touched 0. With sh 16-byte aligned and SH degree 1 or 3, a persistent grid
 * moves the SH rows of visible Gaussians by bulk copies; otherwise by 4-byte copies.
 * Arguments: p (inputs, n >= 0, n < 2^31), cam, opt (may be NULL), out (outputs, out->n == p->n).
 * Errors: GS_ERR_ARG on null/misaligned pointers, bad sh_degree or camera size; GS_ERR_CUDA; a
 * bulk-copy wait that gives up sets GS_ERR_TIMEOUT in the device error word.                  */
int gs_preprocess(const gs_params* p, const gs_camera* cam, const gs_options* opt, gs_proj* out,
                  void* stream);

/* Bytes of device workspace gs_bin_and_sort needs for n Gaussians and `capacity` duplicates on a
 * width x height image: about 27 n + 4.25 capacity + T (n / 512 + capacity / 16384) bytes
 * (T tiles) for images of up to 49,152 tiles, where the tile pass is a two-level counting pass
 * (its coarse lists hold up to `capacity` entries); beyond that the tile pass falls back to radix
 * passes and needs 12 bytes per duplicate of capacity instead.
 * Returns 0 for negative sizes or an empty image. */
size_t gs_sort_workspace_bytes(int64_t n, int64_t capacity, int32_t width, int32_t height);

/* Tile duplication and sort (the rasterization pipeline's binning, DISTWAR, Abstract).
 * One entry (key = tile << 32 | bits of the float32 depth, value = Gaussian index) per
 * Gaussian with radius > 0 and per tile of its rectangle, stably sorted by key: the result is
 * ordered by (tile, depth, Gaussian index). The sort is a hand-written LSD radix sort: the
 * visible Gaussians are first sorted by depth bits (4 passes of 8 bits), then their duplicates
 * are placed by tile id in one stable counting pass, done in two levels: blocks of 4x4 tiles, then
 * tiles (images of up to 49,152 tiles; larger ones emit the duplicates in depth order and sort them
 * by tile id in 8-bit passes), which equals a stable sort of the 64-bit keys.
 * Outputs: keys [D] uint64 (may be NULL: not written), vals [D] uint32, tile_ranges [T][2]
 * uint32 = [start, end) of each tile in the sorted list, *n_dup_out (HOST int64) = D.
 * workspace: device buffer of at least gs_sort_workspace_bytes(n, capacity, W, H) bytes.
 * Synchronises `stream` once to read D. If D > capacity, no entry is written, tile_ranges are
 * written empty, *n_dup_out = D and GS_ERR_CAPACITY is returned; call again with a larger
 * capacity.
 * 0 <= capacity < 2^31. Errors: GS_ERR_ARG, GS_ERR_CAPACITY, GS_ERR_CUDA.                     */
int gs_bin_and_sort(const gs_proj* proj, const gs_camera* cam, const gs_options* opt,
                    void* workspace, size_t workspace_bytes, uint64_t* keys, uint32_t* vals,
                    int64_t capacity, int64_t* n_dup_out, uint32_t* tile_ranges, void* stream);

/* Rendering phase (Odin, Figure 7: "rendering"). One 128-thread block per 16x16 tile (two pixels
 * per thread) stages the tile's list in batches of 128 records in shared memory (bulk
 * asynchronous copies) and blends front to back per pixel:
 * power = -(A dx^2 + C dy^2)/2 - B dx dy with d = mean - pixel centre (evaluated as a sum of
 * non-negative terms, so it is never positive);
 * alpha = min(0.99, opacity exp(power)); skip alpha < 1/255; stop before a Gaussian whose
 * T (1 - alpha) < 1e-4; colour += rgb alpha T; T *= 1 - alpha.
 * Outputs: image [3][H][W] = colour + T bg, t_final [H][W] = T, n_contrib [H][W] = 1 + the
 * position (within the tile's list) of the last blended Gaussian, 0 if none.
 * Errors: GS_ERR_ARG, GS_ERR_CUDA; a staging wait that gives up sets GS_ERR_TIMEOUT in the
 * device error word.                                                                          */
int gs_render_fwd(const gs_proj* proj, const uint32_t* vals, const uint32_t* tile_ranges,
                  const gs_camera* cam, const gs_options* opt, float* image, float* t_final,
                  uint32_t* n_contrib, void* stream);

/* Gradient computation phase (Odin, Figure 7: "backward computation"; DISTWAR and ARC,
 * Abstract: the atomic-bound step). Replays each pixel's list back to front from n_contrib,
 * recovering T by division by (1 - alpha), and accumulates per Gaussian
 * grad2d[g] = dL/d(mean_x, mean_y, A, B, C, opacity, r, g, b) over all pixels, given
 * dl_dimage [3][H][W]: dL/drgb = alpha T g; dL/dalpha = sum_ch g_ch (rgb_ch T - S_ch/(1 - alpha))
 * with S the colour blended behind (background included); the derivative through the 0.99
 * clamp is 0. grad2d is [N][12] float32, 16-byte aligned; columns 9..11 are left 0. The callee
 * zeroes grad2d first. Accumulation strategy: opt->bwd_mode (see GS_BWD_*). One 64-thread block
 * per tile, four pixels per thread, batches of 64 staged records (the forward's layout on images
 * of fewer than two tiles per SM).
 * Errors: GS_ERR_ARG, GS_ERR_CUDA; staging timeouts as for gs_render_fwd.                    */
int gs_render_bwd(const gs_proj* proj, const uint32_t* vals, const uint32_t* tile_ranges,
                  const gs_camera* cam, const gs_options* opt, const float* dl_dimage,
                  const float* t_final, const uint32_t* n_contrib, float* grad2d, void* stream);

/* gs_render_bwd with the loss folded in: the upstream gradient is that of the squared error
 * L = 0.5 sum over channels and pixels of (image - target)^2, dL/dimage = image - target, formed
 * per pixel by the backward kernel as it reads the image (the rendering phase's output feeding the
 * backward computation, Odin: Primitive-Level Synchronization for Distributed Point-Based Neural
 * Rendering, Figure 7), instead of a separate pass writing dl_dimage.
 * image, target: [3][H][W] float32 (image: gs_render_fwd's output); loss: one device float or
 * NULL, set to L (zeroed and accumulated by the callee; its summation order varies, so it is
 * reproducible to float32 rounding). Other arguments, outputs and errors as gs_render_bwd;
 * GS_ERR_ARG when target is NULL.                                                           */
int gs_render_bwd_sqerr(const gs_proj* proj, const uint32_t* vals, const uint32_t* tile_ranges,
                        const gs_camera* cam, const gs_options* opt, const float* image, const float* target,
                        const float* t_final, const uint32_t* n_contrib, float* grad2d, float* loss,
                        void* stream);

/* Preprocessing backward: chain rule from grad2d to the parameters, recomputing the forward of
 * gs_preprocess per Gaussian. Outputs d_mean3d [N][3], d_log_scale [N][3], d_quat [N][4]
 * (through the normalisation), d_opacity_logit [N], d_sh [N][K][3]. Gaussians with radius 0
 * (culled) get zeros. accumulate != 0 adds to the outputs (views of one step), else overwrites.
 * With sh and d_sh 16-byte aligned and SH degree 1 or 3, the SH rows are moved by bulk copies (and
 * added by bulk reductions when accumulating); otherwise by 4-byte copies; the results agree.
 * Errors: GS_ERR_ARG, GS_ERR_CUDA; a bulk-copy wait that gives up sets GS_ERR_TIMEOUT in the
 * device error word.                                                                          */
int gs_preprocess_bwd(const gs_params* p, const gs_camera* cam, const gs_options* opt,
                      const gs_proj* proj, const float* grad2d, float* d_mean3d,
                      float* d_log_scale, float* d_quat, float* d_opacity_logit, float* d_sh,
                      int32_t accumulate, void* stream);

/* ---- optimizer update ------------------------------------------------------------------
 * The update phase "U" of a training step (Odin: Primitive-Level Synchronization for Distributed
 * Point-Based Neural Rendering, Figure 7), with the optimizer the Odin review names (Adam;
 * Review, item 1), applied only to the primitives the view made visible (Odin, Abstract: each
 * view reads and updates only the visible primitives).
 *
 * A set of per-Gaussian float32 tensors in the layout of gs_params; used for the parameters
 * (updated in place), their gradients and the two Adam moments. Every pointer 16-byte aligned. */
typedef struct gs_tensors {
    float*  mean3d;         /* [N][3] */
    float*  log_scale;      /* [N][3] */
    float*  quat;           /* [N][4] */
    float*  opacity_logit;  /* [N]    */
    float*  sh;             /* [N][K][3], K = (sh_degree + 1)^2 */
    int64_t n;
} gs_tensors;

typedef struct gs_adam_options {
    float   lr_mean3d, lr_log_scale, lr_quat, lr_opacity;  /* learning rates per tensor */
    float   lr_sh_dc, lr_sh_rest;  /* sh coefficients k = 0 and k >= 1 */
    float   beta1, beta2, eps;     /* 0 = 0.9, 0.999, 1e-15 */
    int32_t step;                  /* t >= 1, the step's index: bias corrections 1 - beta^t */
    int32_t sh_degree;             /* 0..3 */
} gs_adam_options;

/* Sparse Adam step. For every Gaussian i with radius[i] > 0 (radius: device int32 [N] from
 * gs_preprocess of the view) and every element x of its parameters, with gradient g:
 *   m = beta1 m + (1 - beta1) g,  v = beta2 v + (1 - beta2) g^2,
 *   x = x - lr (m / (1 - beta1^t)) / (sqrt(v / (1 - beta2^t)) + eps);
 * Gaussians with radius 0 keep their parameters and moments. One kernel over all five tensors.
 * Errors: GS_ERR_ARG (NULL or misaligned pointers, n mismatch, step < 1, bad betas or degree,
 * 2^32 or more floats in the sh tensor), GS_ERR_CUDA.                                          */
int gs_adam_step(gs_tensors* params, const gs_tensors* grads, gs_tensors* exp_avg, gs_tensors* exp_avg_sq,
                 const int32_t* radius, const gs_adam_options* opt, void* stream);

/* ---- post-backward statistics ----------------------------------------------------------
 * Per-primitive gradient statistics of one view, read after the backward: what 3D Gaussian
 * splatting's densification accumulates over views, and the per-primitive gradient magnitude that
 * Odin's post-backward hook reports (Odin: Primitive-Level Synchronization for Distributed
 * Point-Based Neural Rendering, Review, item 1: the gate reads ||g_A(p)|| per primitive).
 *
 * For every Gaussian i with radius[i] > 0 (proj from gs_preprocess of the view; grad2d from
 * gs_render_bwd):
 *   grad_norm_accum[i] += sqrt((sx dL/dmean_x)^2 + (sy dL/dmean_y)^2), where (sx, sy) = (1, 1)
 *       (pixel units) or (width / 2, height / 2) when ndc != 0 (normalised device coordinates);
 *   view_count[i] += 1;  max_radius[i] = max(max_radius[i], radius[i]).
 * Hidden Gaussians keep their values. If param_grads is not NULL (the outputs of
 * gs_preprocess_bwd, layout of gs_tensors, sh with K = (sh_degree + 1)^2), grad_mag [N] receives
 * for every Gaussian the 2-norm of all its parameter gradients (0 when hidden).
 * Errors: GS_ERR_ARG (NULL or misaligned pointers, n mismatch, bad degree), GS_ERR_CUDA.      */
int gs_densify_stats(const gs_proj* proj, const float* grad2d, int32_t width, int32_t height, int32_t ndc,
                     float* grad_norm_accum, int32_t* view_count, int32_t* max_radius,
                     const gs_tensors* param_grads, float* grad_mag, int32_t sh_degree, void* stream);

/* The statistics of gs_densify_stats emitted by the preprocess backward itself, where the
 * gradients are already in registers (no extra pass over them). Outputs as gs_densify_stats;
 * ndc != 0 scales dL/dmean2d by (width / 2, height / 2) of `cam`. */
typedef struct {
    float*   grad_norm_accum;  /* [N], += for radius > 0 */
    int32_t* view_count;       /* [N], += 1 for radius > 0 */
    int32_t* max_radius;       /* [N], max with the radius */
    float*   grad_mag;         /* [N] or NULL: 2-norm of this view's parameter gradients, 0 when hidden */
    int32_t  ndc;
} gs_densify_outputs;

/* gs_preprocess_bwd plus the post-backward statistics of the view, from the gradients this call
 * computes (Odin: Primitive-Level Synchronization for Distributed Point-Based Neural Rendering,
 * Review, item 1: the per-primitive gradient magnitude read by a post-backward hook). With
 * accumulate = 0 the outputs equal gs_preprocess_bwd followed by gs_densify_stats with
 * param_grads = the gradient outputs, bit for bit; with accumulate != 0 grad_mag is the norm of
 * this view's own gradients (gs_densify_stats afterwards would see the accumulated sums).
 * Errors: those of gs_preprocess_bwd; GS_ERR_ARG when stats or one of its arrays is NULL or
 * misaligned (grad_mag may be NULL). */
int gs_preprocess_bwd_stats(const gs_params* p, const gs_camera* cam, const gs_options* opt, const gs_proj* proj,
                            const float* grad2d, float* d_mean3d, float* d_log_scale, float* d_quat,
                            float* d_opacity_logit, float* d_sh, int32_t accumulate, const gs_densify_outputs* stats,
                            void* stream);

/* ---- image loss ---------------------------------------------------------------------------
 * The loss whose gradient feeds the gradient computation phase (Odin: Primitive-Level
 * Synchronization for Distributed Point-Based Neural Rendering, Figure 7: rendering, then backward):
 *   L = (1 - lambda) mean|x - y| + lambda (1 - mean SSIM(x, y)),
 * means over the 3 x H x W values; SSIM per channel with an 11x11 Gaussian window (sigma 1.5,
 * normalised), C1 = 0.01^2, C2 = 0.03^2, zero padding outside the image. (The pages name SSIM as an
 * evaluation metric, Odin Figure 15; this form is the 3D Gaussian splatting training loss.)
 * image, target: [3][H][W] float32 device; outputs: *loss (one device float) and dl_dimage
 * [3][H][W] (the derivative of |x - y| at x = y is taken as 0). lambda in [0, 1] (0.2 in that
 * recipe). workspace: device buffer of gs_loss_workspace_bytes(W, H) bytes, 256-byte aligned.
 * Errors: GS_ERR_ARG (NULL or misaligned pointers, bad size or lambda, small workspace),
 * GS_ERR_CUDA.                                                                                */
size_t gs_loss_workspace_bytes(int32_t width, int32_t height);
int gs_loss_l1_dssim(const float* image, const float* target, int32_t width, int32_t height, float lambda,
                     void* workspace, size_t workspace_bytes, float* loss, float* dl_dimage, void* stream);

/* ---- surfels: 2D Gaussian splatting --------------------------------------------------------
 * The rendering pipeline of 2D Gaussian splatting, one of the four pipelines Odin trains (Odin:
 * Primitive-Level Synchronization for Distributed Point-Based Neural Rendering, Summary). Each
 * Gaussian is a flat disk, P(u, v) = mean + s_u u t_u + s_v v t_v (t_u, t_v the first two columns
 * of its rotation, s = exp of log_scale[0..1]; log_scale[2] is unused). A pixel (x, y) weighs it by
 * max(exp(-(u^2 + v^2)/2), exp(-|(x, y) - c|^2)) with (u, v) where the pixel's ray meets the disk's
 * plane and c the centre of the screen box of its 3-sigma disk; alpha, thresholds, termination and
 * blending are those of gs_render_fwd. The binning is gs_bin_and_sort on the gs_proj that
 * gs_preprocess2d fills (box centre as mean, radius = ceil of the larger box half extent, at least
 * 3 sqrt(1/2)).
 *
 * Surfel record rec2d [N][16] float32, 16-byte aligned: A_u = s_u fx (W t_u)_x, B_u = s_u fy
 * (W t_u)_y, C_u = s_u (W t_u)_z, A_v, B_v, C_v likewise for t_v, m_x, m_y (projected mean), z_c
 * (its depth), c_x, c_y (box centre), opacity, r, g, b, 0. Culled Gaussians: radius 0, zero record.
 * Surfel gradients grad2d [N][16] float32: dL/d(the first 15 record fields).                     */
int gs_preprocess2d(const gs_params* p, const gs_camera* cam, const gs_options* opt, gs_proj* out,
                    float* rec2d, void* stream);
/* Forward of the surfels listed by gs_bin_and_sort (n = number of records). Outputs as
 * gs_render_fwd. Errors: GS_ERR_ARG, GS_ERR_CUDA; staging timeouts in the device error word.    */
int gs_render2d_fwd(const float* rec2d, int64_t n, const uint32_t* vals, const uint32_t* tile_ranges,
                    const gs_camera* cam, const gs_options* opt, float* image, float* t_final,
                    uint32_t* n_contrib, void* stream);
/* Backward of gs_render2d_fwd: grad2d [N][16] = dL/d(record fields 0..14), zeroed first by the
 * callee. bwd_mode DIRECT, WARP or ADAPTIVE (SM is rejected). Errors as gs_render_bwd.           */
int gs_render2d_bwd(const float* rec2d, int64_t n, const uint32_t* vals, const uint32_t* tile_ranges,
                    const gs_camera* cam, const gs_options* opt, const float* dl_dimage,
                    const float* t_final, const uint32_t* n_contrib, float* grad2d, void* stream);
/* Chain rule from the surfel gradients to the parameters, as gs_preprocess_bwd (d_log_scale[2]
 * is 0). proj: the gs_proj gs_preprocess2d filled (radius marks the visible surfels).          */
int gs_preprocess2d_bwd(const gs_params* p, const gs_camera* cam, const gs_options* opt,
                        const gs_proj* proj, const float* grad2d, float* d_mean3d, float* d_log_scale,
                        float* d_quat, float* d_opacity_logit, float* d_sh, int32_t accumulate,
                        void* stream);

/* Size of the device workspace that gs_bin_and_sort_static uses instead of a caller buffer. */
#define GS_STATIC_SORT_WORKSPACE_BYTES (32u << 20)

/* gs_bin_and_sort without a workspace argument, for callers that cannot allocate device memory:
 * a plug-in that only receives its input and output buffers from a host application which owns
 * all device memory under a fixed budget (it may not call cudaMalloc itself), or a real-time loop
 * in which an allocation could stall or fail in the middle of a frame. It computes
 * exactly what gs_bin_and_sort computes (same outputs, same
 * errors) but takes its scratch space from a statically sized device array inside this library,
 * GS_STATIC_SORT_WORKSPACE_BYTES (32 MiB), which every GPU that loads the library keeps reserved
 * until the process exits. The pages describe no such entry point; it is a convenience of this
 * library.
 *   - Limit: the call needs gs_sort_workspace_bytes(n, capacity, W, H) <= 32 MiB (for example
 *     n = 400,000 Gaussians with capacity = 4,000,000 duplicates on an 800 x 800 image); larger
 *     requests return GS_ERR_ARG without touching the device. The call itself allocates nothing.
 *   - Set-up: the first call on a device looks up the device address of the array (once per
 *     device, with that device current). Make that first call before any stream capture.
 *   - Sharing: all calls in the process use the same array, which keeps the last call's contents
 *     (nothing in it needs to start at zero). Calls whose GPU work overlaps (different streams, or
 *     different host threads on one device) race on it and give wrong results: order them on one
 *     stream or synchronise between them.
 * Arguments and errors otherwise as gs_bin_and_sort.                                          */
int gs_bin_and_sort_static(const gs_proj* proj, const gs_camera* cam, const gs_options* opt, uint64_t* keys,
                           uint32_t* vals, int64_t capacity, int64_t* n_dup_out, uint32_t* tile_ranges,
                           void* stream);

/* gs_bin_and_sort with no host synchronisation, so that a whole training step can be enqueued
 * ahead of the GPU or captured into a CUDA graph (DISTWAR, Abstract: the binning of the
 * rasterization pipeline; same outputs as gs_bin_and_sort). It neither synchronises nor
 * allocates; every launch and copy goes on `stream`.
 *   - D is not returned on the host: when n_dup_device (device uint64, 8-byte aligned) is not
 *     NULL, D is written there on the stream (by the tile scan).
 *   - Capacity: if D > capacity, no entry is written past `capacity`, every tile range is
 *     written empty (so later kernels read nothing) and the device error word gets the check
 *     bit (gs_device_error returns GS_ERR_DEVICE_CHECK); *n_dup_device then holds the D needed.
 *   - workspace: a device buffer of gs_sort_workspace_bytes(n, capacity, W, H) bytes, or NULL
 *     for the library's static workspace (limit and sharing rules of gs_bin_and_sort_static).
 *   - Images of up to 49,152 tiles (the counting tile pass); larger images return GS_ERR_ARG.
 *   - Set-up: make one call (or one call of any other entry point) on the device before a
 *     stream capture, so that the library's device symbols are looked up outside it.
 * Errors: GS_ERR_ARG (pointers, sizes, workspace, image size), GS_ERR_CUDA.                    */
int gs_bin_and_sort_async(const gs_proj* proj, const gs_camera* cam, const gs_options* opt, void* workspace,
                          size_t workspace_bytes, uint64_t* keys, uint32_t* vals, int64_t capacity,
                          uint64_t* n_dup_device, uint32_t* tile_ranges, void* stream);

/* Text of a status code (static storage). */
const char* gs_status_string(int status);

/* Description of the last failed call on the calling thread ("" if none). */
const char* gs_last_error_message(void);

/* Synchronises `stream`, reads and clears the device error word of the current device:
 * GS_OK, GS_ERR_TIMEOUT (a bounded device wait gave up) or GS_ERR_DEVICE_CHECK. */
int gs_device_error(void* stream);

/* Self-test of the bounded device-side wait used by the render kernels: launches one block that
 * waits on a shared-memory barrier nothing will complete, giving up after `spin_limit`
 * iterations (0 = 1024). The wait sets the timeout bit of the device error word, so a following
 * gs_device_error() returns GS_ERR_TIMEOUT; the context stays usable. Errors: GS_ERR_CUDA.      */
int gs_selftest_timeout(uint32_t spin_limit, void* stream);

/* Self-test of the bounded look-back in the depth sort of gs_bin_and_sort: runs one block of a
 * depth pass whose predecessor block never publishes its counts, so the block's look-back finds
 * nothing, gives up after `spin_limit` polls (0 = 1024) and sets the timeout bit of the device
 * error word; a following gs_device_error() returns GS_ERR_TIMEOUT and the context stays usable.
 * workspace: device buffer of at least GS_SELFTEST_SORT_WORKSPACE_BYTES, 16-byte aligned, owned
 * by the caller (overwritten). Errors: GS_ERR_ARG (workspace), GS_ERR_CUDA.                     */
#define GS_SELFTEST_SORT_WORKSPACE_BYTES (128u << 10)
int gs_selftest_sort_timeout(void* workspace, size_t workspace_bytes, uint32_t spin_limit, void* stream);

/* ---- the whole training step of one view with host buffers ------------------------------
 * The step of Odin's Figure 7 (preprocessing, rendering, backward computation; Odin:
 * Primitive-Level Synchronization for Distributed Point-Based Neural Rendering) driven from host
 * memory: the parameters and the target image are copied in, the step runs on the device, and
 * the parameter gradients, the loss and D come back, all asynchronously on one stream.
 *
 * gs_step_context_create allocates, on the current device, the device buffers of such steps for n
 * Gaussians of SH degree sh_degree on images of at most max_width x max_height pixels (at most
 * 49,152 tiles) with room for `capacity` duplicates: the parameters, their gradients, the
 * projected records, the sort workspace and lists, the image, transmittance, contributor counts,
 * target and 2D gradients (about (196 + 24 K) n + 4 capacity + 32 max_width max_height bytes,
 * K = (sh_degree + 1)^2, plus gs_sort_workspace_bytes(n, capacity, max_width, max_height)). The context belongs to the caller: one step at a time per context
 * (two contexts on two streams overlap one step's copies with another's compute).
 * Errors: GS_ERR_ARG (sizes, degree, NULL out), GS_ERR_CUDA (allocation); *out is set only on
 * success. gs_step_context_destroy frees it (NULL is accepted) after synchronising the device. */
typedef struct gs_step_context gs_step_context;
int gs_step_context_create(int64_t n, int32_t sh_degree, int32_t max_width, int32_t max_height, int64_t capacity,
                           gs_step_context** out);
int gs_step_context_destroy(gs_step_context* ctx);

/* One training step of one view with host buffers (the library's end-to-end entry point):
 *   host_params: the n Gaussians' parameters in host memory (layout of gs_params; n must equal the
 *     context's); host_target [3][H][W] float32 (the camera's size); both are copied to the device
 *     with one cudaMemcpyAsync per array;
 *   then gs_preprocess, gs_bin_and_sort_async (capacity: the context's), gs_render_fwd,
 *   gs_render_bwd_sqerr (loss 0.5 |image - target|^2) and gs_preprocess_bwd (overwriting) run on
 *   the device buffers;
 *   host_grads: the parameter gradients, copied back into host memory (layout of gs_tensors,
 *     n = the context's); host_loss (one float) and host_n_dup (D, one int64) may be NULL.
 * Everything is enqueued on `stream` (NULL = the default stream) and the call returns without
 * waiting: the host buffers must stay valid, and the outputs are ready, once the stream has
 * reached this point (cudaStreamSynchronize). Page-locked host memory (cudaHostAlloc or
 * cudaHostRegister) lets the copies run asynchronously and overlap other streams' work; with
 * pageable memory the copies are staged and synchronous. A capacity overflow drops duplicates
 * and sets the device check bit (gs_device_error returns GS_ERR_DEVICE_CHECK); host_n_dup then
 * holds the number that was needed. opt->sh_degree must equal the context's degree, and the
 * current device the one the context was created on.
 * Errors: GS_ERR_ARG (NULL or mismatched arguments, an image larger than the context's),
 * GS_ERR_CUDA; the device-side errors of the calls it makes.                                  */
int gs_train_step_host(gs_step_context* ctx, const gs_params* host_params, const float* host_target,
                       const gs_camera* cam, const gs_options* opt, const gs_tensors* host_grads, float* host_loss,
                       int64_t* host_n_dup, void* stream);

/* Number of kernels this library has launched in this process (all devices, all threads). */
int64_t gs_kernel_launches(void);

/* Library version: (major << 16) | minor. */
int gs_version(void);

#ifdef __cplusplus
}
#endif

#endif /* GS_GB300_H */
