// C ABI of the library (declared in include/gs.h): argument checks, option defaults, camera
// set-up and kernel launches. No exception crosses this boundary; failures return a GS_ERR_*
// status and leave a message for gs_last_error_message().
#include <atomic>
#include <cmath>
#include <cstdarg>
#include <cstdio>
#include <cstring>
#include <string>

#include "gs_common.cuh"
#include "gs_internal.h"

namespace gs {

// Device error word of this library, one per device.
__device__ unsigned int g_error_word = 0u;

// Scratch space of gs_bin_and_sort_static: reserved on every device that loads the library.
static __device__ __align__(256) unsigned char g_static_sort_ws[GS_STATIC_SORT_WORKSPACE_BYTES];

static std::atomic<long long> g_launches{0};
void count_launches(int k) { g_launches.fetch_add(k, std::memory_order_relaxed); }

// Waits on a barrier that expects two arrivals but gets one: the bounded wait must give up.
__global__ void k_selftest_timeout(unsigned spin_limit, unsigned* err) {
    __shared__ uint64_t bar;
    if (threadIdx.x == 0) {
        mbar_init(&bar, 2);
        fence_mbar_init();
        asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_u32(&bar)) : "memory");
        mbar_wait_bounded(&bar, 0u, spin_limit, err);
    }
}

namespace {

thread_local std::string t_last_error;

int fail(int status, const char* fmt, ...) __attribute__((format(printf, 2, 3)));
int fail(int status, const char* fmt, ...) {
    char buf[512];
    va_list ap;
    va_start(ap, fmt);
    vsnprintf(buf, sizeof(buf), fmt, ap);
    va_end(ap);
    t_last_error = buf;
    return status;
}

int cuda_fail(cudaError_t e, const char* where) {
    return fail(GS_ERR_CUDA, "%s: %s", where, cudaGetErrorString(e));
}

bool aligned(const void* p, size_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }

constexpr int kMaxImageSide = 32768;

struct Opts {
    int bwd_mode, thr, deg, staging;
    float near_z, lowpass, jac;
    unsigned spin;
};

int resolve_options(const gs_options* o, Opts& r) {
    gs_options z{};
    if (!o) o = &z;
    r.bwd_mode = o->bwd_mode == GS_BWD_DEFAULT ? GS_BWD_ADAPTIVE : o->bwd_mode;
    if (r.bwd_mode < GS_BWD_DIRECT || r.bwd_mode > GS_BWD_SM) return fail(GS_ERR_ARG, "bad bwd_mode %d", o->bwd_mode);
    // defaults measured on GB300 (outdoor, object and contention scenes): a warp reduction pays
    // off only when at least 28 of the 32 lanes contribute; the shared-memory mode keeps 8
    r.thr = o->adaptive_threshold != 0 ? o->adaptive_threshold : (r.bwd_mode == GS_BWD_SM ? 8 : 28);
    if (r.thr < 1 || r.thr > 33) return fail(GS_ERR_ARG, "adaptive_threshold %d outside 1..33", o->adaptive_threshold);
    r.deg = o->sh_degree;
    if (r.deg < 0 || r.deg > 3) return fail(GS_ERR_ARG, "sh_degree %d outside 0..3", o->sh_degree);
    r.staging = o->staging == GS_STAGE_DEFAULT ? GS_STAGE_BULK : o->staging;
    if (r.staging != GS_STAGE_BULK && r.staging != GS_STAGE_LOADS) return fail(GS_ERR_ARG, "bad staging %d", o->staging);
    r.near_z = o->near_z == 0.f ? 0.2f : o->near_z;
    r.lowpass = o->lowpass == 0.f ? 0.3f : (o->lowpass < 0.f ? 0.f : o->lowpass);
    r.jac = o->jacobian_clamp == 0.f ? 1.3f : o->jacobian_clamp;
    r.spin = o->spin_limit == 0u ? (1u << 18) : o->spin_limit;
    if (!std::isfinite(r.near_z) || !std::isfinite(r.lowpass)) return fail(GS_ERR_ARG, "non-finite near_z or lowpass");
    return GS_OK;
}

int make_camera(const gs_camera* c, const Opts& o, KernelCamera& k) {
    if (!c) return fail(GS_ERR_ARG, "camera is NULL");
    if (c->width <= 0 || c->height <= 0 || c->width > kMaxImageSide || c->height > kMaxImageSide)
        return fail(GS_ERR_ARG, "image size %dx%d outside 1..%d", c->width, c->height, kMaxImageSide);
    if (!(c->fx > 0.f) || !(c->fy > 0.f) || !std::isfinite(c->fx) || !std::isfinite(c->fy))
        return fail(GS_ERR_ARG, "focal lengths must be finite and positive");
    std::memcpy(k.R, c->R, sizeof(k.R));
    std::memcpy(k.t, c->t, sizeof(k.t));
    std::memcpy(k.bg, c->bg, sizeof(k.bg));
    k.fx = c->fx; k.fy = c->fy; k.cx = c->cx; k.cy = c->cy;
    k.width = c->width; k.height = c->height;
    k.tiles_x = (c->width + kTile - 1) / kTile;
    k.tiles_y = (c->height + kTile - 1) / kTile;
    for (int j = 0; j < 3; ++j)
        k.campos[j] = (float)-((double)c->R[j] * c->t[0] + (double)c->R[3 + j] * c->t[1] + (double)c->R[6 + j] * c->t[2]);
    if (o.jac > 0.f) {
        k.limx = (float)(o.jac * 0.5 * c->width / (double)c->fx);
        k.limy = (float)(o.jac * 0.5 * c->height / (double)c->fy);
    } else {
        k.limx = k.limy = 3.0e38f;
    }
    k.near_z = o.near_z;
    k.lowpass = o.lowpass;
    return GS_OK;
}

int check_params(const gs_params* p) {
    if (!p) return fail(GS_ERR_ARG, "params is NULL");
    if (p->n < 0 || p->n > 0x7fffffffll) return fail(GS_ERR_ARG, "n = %lld outside 0..2^31-1", (long long)p->n);
    if (p->n == 0) return GS_OK;
    const void* ptrs[5] = {p->mean3d, p->log_scale, p->quat, p->opacity_logit, p->sh};
    for (const void* q : ptrs)
        if (!q || !aligned(q, 4)) return fail(GS_ERR_ARG, "a parameter pointer is NULL or not 4-byte aligned");
    return GS_OK;
}

int check_proj(const gs_proj* q, int64_t n) {
    if (!q) return fail(GS_ERR_ARG, "proj is NULL");
    if (q->n != n) return fail(GS_ERR_ARG, "proj.n = %lld does not match n = %lld", (long long)q->n, (long long)n);
    if (n == 0) return GS_OK;
    if (!q->rec || !aligned(q->rec, 16)) return fail(GS_ERR_ARG, "proj.rec is NULL or not 16-byte aligned");
    if (!q->depth || !q->radius || !q->tiles_touched || !aligned(q->depth, 4) || !aligned(q->radius, 4) ||
        !aligned(q->tiles_touched, 4))
        return fail(GS_ERR_ARG, "proj.depth / radius / tiles_touched NULL or misaligned");
    return GS_OK;
}

int check_proj_n(const gs_proj* q) {
    if (!q) return fail(GS_ERR_ARG, "proj is NULL");
    if (q->n < 0 || q->n > 0x7fffffffll) return fail(GS_ERR_ARG, "proj.n outside 0..2^31-1");
    return check_proj(q, q->n);
}

cudaStream_t as_stream(void* s) { return reinterpret_cast<cudaStream_t>(s); }

// Per-device cache of a device symbol's address. Host threads may look it up concurrently: every
// entry is an atomic, so two first calls on one device at worst both query the runtime and store
// the same address.
template <class T>
T* symbol_address(std::atomic<T*> (&cache)[256], const void* symbol, const char* what, int* status) {
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e || dev < 0 || dev >= 256) { *status = cuda_fail(e ? e : cudaErrorInvalidDevice, "cudaGetDevice"); return nullptr; }
    T* p = cache[dev].load(std::memory_order_acquire);
    if (!p) {
        void* q = nullptr;
        e = cudaGetSymbolAddress(&q, symbol);
        if (e) { *status = cuda_fail(e, what); return nullptr; }
        p = static_cast<T*>(q);
        cache[dev].store(p, std::memory_order_release);
    }
    *status = GS_OK;
    return p;
}

// Device address of g_error_word for the current device (looked up once per device).
unsigned* error_word(int* status) {
    static std::atomic<unsigned*> cache[256] = {};
    return symbol_address(cache, (const void*)&g_error_word, "cudaGetSymbolAddress(error word)", status);
}

// Device address of g_static_sort_ws for the current device (looked up once per device; in host
// code the array's name is only a stand-in, so kernels must be given this address).
unsigned char* static_sort_workspace(int* status) {
    static std::atomic<unsigned char*> cache[256] = {};
    return symbol_address(cache, (const void*)g_static_sort_ws, "cudaGetSymbolAddress(static sort workspace)",
                          status);
}

}  // namespace

int device_sm_count() {
    static std::atomic<int> cache[256] = {};
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 256) return 1;
    int v = cache[dev].load(std::memory_order_relaxed);
    if (v == 0) {
        if (cudaDeviceGetAttribute(&v, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || v < 1) return 1;
        cache[dev].store(v, std::memory_order_relaxed);
    }
    return v;
}

}  // namespace gs

using namespace gs;

extern "C" {

int gs_version(void) { return (1 << 16) | 0; }

int64_t gs_kernel_launches(void) { return (int64_t)g_launches.load(std::memory_order_relaxed); }

const char* gs_status_string(int status) {
    switch (status) {
        case GS_OK: return "GS_OK";
        case GS_ERR_ARG: return "GS_ERR_ARG: invalid argument";
        case GS_ERR_CAPACITY: return "GS_ERR_CAPACITY: duplicate capacity too small";
        case GS_ERR_CUDA: return "GS_ERR_CUDA: CUDA runtime error";
        case GS_ERR_TIMEOUT: return "GS_ERR_TIMEOUT: a bounded device wait gave up";
        case GS_ERR_DEVICE_CHECK: return "GS_ERR_DEVICE_CHECK: device-side consistency check failed";
        default: return "unknown status";
    }
}

const char* gs_last_error_message(void) { return t_last_error.c_str(); }

int gs_device_error(void* stream) {
    unsigned word = 0;
    cudaError_t e = cudaStreamSynchronize(as_stream(stream));
    if (e) return cuda_fail(e, "gs_device_error: synchronize");
    e = cudaMemcpyFromSymbol(&word, g_error_word, sizeof(word));
    if (e) return cuda_fail(e, "gs_device_error: read");
    const unsigned zero = 0;
    e = cudaMemcpyToSymbol(g_error_word, &zero, sizeof(zero));
    if (e) return cuda_fail(e, "gs_device_error: clear");
    if (word & kErrTimeout) return fail(GS_ERR_TIMEOUT, "a bounded device-side wait gave up");
    if (word & kErrCheck) return fail(GS_ERR_DEVICE_CHECK, "a device-side consistency check failed");
    return GS_OK;
}

int gs_selftest_timeout(uint32_t spin_limit, void* stream) {
    int s;
    unsigned* err = error_word(&s);
    if (!err) return s;
    k_selftest_timeout<<<1, 32, 0, as_stream(stream)>>>(spin_limit ? spin_limit : 1024u, err);
    count_launches(1);
    cudaError_t e = cudaGetLastError();
    return e ? cuda_fail(e, "gs_selftest_timeout") : GS_OK;
}

static_assert(kSelftestLookbackBytes <= GS_SELFTEST_SORT_WORKSPACE_BYTES, "self-test workspace too small");

int gs_selftest_sort_timeout(void* workspace, size_t workspace_bytes, uint32_t spin_limit, void* stream) {
    if (!workspace || !aligned(workspace, 16)) return fail(GS_ERR_ARG, "workspace is NULL or not 16-byte aligned");
    if (workspace_bytes < GS_SELFTEST_SORT_WORKSPACE_BYTES)
        return fail(GS_ERR_ARG, "workspace of %zu bytes, need %u", workspace_bytes,
                    (unsigned)GS_SELFTEST_SORT_WORKSPACE_BYTES);
    int s;
    unsigned* err = error_word(&s);
    if (!err) return s;
    cudaError_t e = selftest_lookback(static_cast<unsigned char*>(workspace), spin_limit ? spin_limit : 1024u, err,
                                      as_stream(stream));
    return e ? cuda_fail(e, "gs_selftest_sort_timeout") : GS_OK;
}

int gs_preprocess(const gs_params* p, const gs_camera* cam, const gs_options* opt, gs_proj* out, void* stream) {
    Opts o;
    KernelCamera kc;
    int s;
    if ((s = resolve_options(opt, o)) || (s = make_camera(cam, o, kc)) || (s = check_params(p))) return s;
    if ((s = check_proj(out, p->n))) return s;
    unsigned* err = error_word(&s);
    if (!err) return s;
    cudaError_t e = launch_preprocess(o.deg, (int)p->n, *p, kc, *out, o.spin, err, as_stream(stream));
    return e ? cuda_fail(e, "gs_preprocess") : GS_OK;
}

size_t gs_sort_workspace_bytes(int64_t n, int64_t capacity, int32_t width, int32_t height) {
    if (n < 0 || capacity < 0 || width <= 0 || height <= 0) return 0;
    return carve_workspace(nullptr, n, capacity, (width + kTile - 1) / kTile, (height + kTile - 1) / kTile).bytes;
}

int gs_bin_and_sort(const gs_proj* proj, const gs_camera* cam, const gs_options* opt, void* workspace,
                    size_t workspace_bytes, uint64_t* keys, uint32_t* vals, int64_t capacity, int64_t* n_dup_out,
                    uint32_t* tile_ranges, void* stream) {
    Opts o;
    KernelCamera kc;
    int s;
    if ((s = resolve_options(opt, o)) || (s = make_camera(cam, o, kc)) || (s = check_proj_n(proj))) return s;
    if (!n_dup_out) return fail(GS_ERR_ARG, "n_dup_out is NULL");
    if (capacity < 0 || capacity > 0x7fffffffll) return fail(GS_ERR_ARG, "capacity outside 0..2^31-1");
    if (!tile_ranges || !aligned(tile_ranges, 8)) return fail(GS_ERR_ARG, "tile_ranges NULL or not 8-byte aligned");
    if (capacity > 0 && (!vals || !aligned(vals, 4))) return fail(GS_ERR_ARG, "vals NULL or misaligned");
    if (keys && !aligned(keys, 8)) return fail(GS_ERR_ARG, "keys not 8-byte aligned");
    const long long tiles = (long long)kc.tiles_x * kc.tiles_y;
    const size_t need = carve_workspace(nullptr, proj->n, capacity, kc.tiles_x, kc.tiles_y).bytes;
    if (!workspace || workspace_bytes < need || !aligned(workspace, 256))
        return fail(GS_ERR_ARG, "workspace NULL, not 256-byte aligned or smaller than %zu bytes", need);
    const SortWorkspace w = carve_workspace(workspace, proj->n, capacity, kc.tiles_x, kc.tiles_y);
    unsigned* err = error_word(&s);
    if (!err) return s;
    cudaStream_t st = as_stream(stream);
    cudaError_t e = bin_count(*proj, kc.tiles_x, kc.tiles_y, w, err, o.spin, (unsigned long long)capacity,
                              tile_ranges, nullptr, nullptr, st);
    if (e) return cuda_fail(e, "gs_bin_and_sort: count");
    unsigned long long d = 0;
    if ((e = cudaMemcpyAsync(&d, w.total, 8, cudaMemcpyDeviceToHost, st))) return cuda_fail(e, "gs_bin_and_sort: read D");
    if ((e = cudaStreamSynchronize(st))) return cuda_fail(e, "gs_bin_and_sort: synchronize");
    *n_dup_out = (int64_t)d;
    if (d > (unsigned long long)capacity) {
        if ((e = cudaMemsetAsync(tile_ranges, 0, (size_t)tiles * 8, st))) return cuda_fail(e, "gs_bin_and_sort");
        return fail(GS_ERR_CAPACITY, "%llu duplicates exceed capacity %lld", d, (long long)capacity);
    }
    e = bin_emit_sort(*proj, kc.tiles_x, kc.tiles_y, (unsigned)d, (unsigned long long)capacity, w, keys, vals,
                      tile_ranges, err, st);
    return e ? cuda_fail(e, "gs_bin_and_sort: emit/sort") : GS_OK;
}

int gs_bin_and_sort_static(const gs_proj* proj, const gs_camera* cam, const gs_options* opt, uint64_t* keys,
                           uint32_t* vals, int64_t capacity, int64_t* n_dup_out, uint32_t* tile_ranges,
                           void* stream) {
    Opts o;
    KernelCamera kc;
    int s;
    if ((s = resolve_options(opt, o)) || (s = make_camera(cam, o, kc)) || (s = check_proj_n(proj))) return s;
    if (!n_dup_out) return fail(GS_ERR_ARG, "n_dup_out is NULL");
    if (capacity < 0 || capacity > 0x7fffffffll) return fail(GS_ERR_ARG, "capacity outside 0..2^31-1");
    if (!tile_ranges || !aligned(tile_ranges, 8)) return fail(GS_ERR_ARG, "tile_ranges NULL or not 8-byte aligned");
    if (capacity > 0 && (!vals || !aligned(vals, 4))) return fail(GS_ERR_ARG, "vals NULL or misaligned");
    if (keys && !aligned(keys, 8)) return fail(GS_ERR_ARG, "keys not 8-byte aligned");
    const long long tiles = (long long)kc.tiles_x * kc.tiles_y;
    const size_t need = carve_workspace(nullptr, proj->n, capacity, kc.tiles_x, kc.tiles_y).bytes;
    if (need > (size_t)GS_STATIC_SORT_WORKSPACE_BYTES)
        return fail(GS_ERR_ARG,
                    "n = %lld with capacity %lld needs %zu bytes of sort workspace; the static workspace holds %u "
                    "bytes: use gs_bin_and_sort with a caller-provided workspace",
                    (long long)proj->n, (long long)capacity, need, (unsigned)GS_STATIC_SORT_WORKSPACE_BYTES);
    unsigned char* ws = static_sort_workspace(&s);
    if (!ws) return s;
    const SortWorkspace w = carve_workspace(ws, proj->n, capacity, kc.tiles_x, kc.tiles_y);
    unsigned* err = error_word(&s);
    if (!err) return s;
    cudaStream_t st = as_stream(stream);
    cudaError_t e = bin_count(*proj, kc.tiles_x, kc.tiles_y, w, err, o.spin, (unsigned long long)capacity,
                              tile_ranges, nullptr, nullptr, st);
    if (e) return cuda_fail(e, "gs_bin_and_sort_static: count");
    unsigned long long d = 0;
    if ((e = cudaMemcpyAsync(&d, w.total, 8, cudaMemcpyDeviceToHost, st)))
        return cuda_fail(e, "gs_bin_and_sort_static: read D");
    if ((e = cudaStreamSynchronize(st))) return cuda_fail(e, "gs_bin_and_sort_static: synchronize");
    *n_dup_out = (int64_t)d;
    if (d > (unsigned long long)capacity) {
        if ((e = cudaMemsetAsync(tile_ranges, 0, (size_t)tiles * 8, st)))
            return cuda_fail(e, "gs_bin_and_sort_static");
        return fail(GS_ERR_CAPACITY, "%llu duplicates exceed capacity %lld", d, (long long)capacity);
    }
    e = bin_emit_sort(*proj, kc.tiles_x, kc.tiles_y, (unsigned)d, (unsigned long long)capacity, w, keys, vals,
                      tile_ranges, err, st);
    return e ? cuda_fail(e, "gs_bin_and_sort_static: emit/sort") : GS_OK;
}

int gs_bin_and_sort_async(const gs_proj* proj, const gs_camera* cam, const gs_options* opt, void* workspace,
                          size_t workspace_bytes, uint64_t* keys, uint32_t* vals, int64_t capacity,
                          uint64_t* n_dup_device, uint32_t* tile_ranges, void* stream) {
    Opts o;
    KernelCamera kc;
    int s;
    if ((s = resolve_options(opt, o)) || (s = make_camera(cam, o, kc)) || (s = check_proj_n(proj))) return s;
    if (capacity < 0 || capacity > 0x7fffffffll) return fail(GS_ERR_ARG, "capacity outside 0..2^31-1");
    if (!tile_ranges || !aligned(tile_ranges, 8)) return fail(GS_ERR_ARG, "tile_ranges NULL or not 8-byte aligned");
    if (capacity > 0 && (!vals || !aligned(vals, 4))) return fail(GS_ERR_ARG, "vals NULL or misaligned");
    if (keys && !aligned(keys, 8)) return fail(GS_ERR_ARG, "keys not 8-byte aligned");
    if (n_dup_device && !aligned(n_dup_device, 8)) return fail(GS_ERR_ARG, "n_dup_device not 8-byte aligned");
    const long long tiles = (long long)kc.tiles_x * kc.tiles_y;
    if (!counting_path(tiles))
        return fail(GS_ERR_ARG, "%lld tiles: the call without host synchronisation handles images of up to 49152 "
                    "tiles; use gs_bin_and_sort", tiles);
    const size_t need = carve_workspace(nullptr, proj->n, capacity, kc.tiles_x, kc.tiles_y).bytes;
    unsigned char* base = static_cast<unsigned char*>(workspace);
    if (!workspace) {
        if (need > (size_t)GS_STATIC_SORT_WORKSPACE_BYTES)
            return fail(GS_ERR_ARG, "n = %lld with capacity %lld needs %zu bytes of sort workspace; the static "
                        "workspace holds %u bytes: pass a workspace", (long long)proj->n, (long long)capacity, need,
                        (unsigned)GS_STATIC_SORT_WORKSPACE_BYTES);
        if (!(base = static_sort_workspace(&s))) return s;
    } else if (workspace_bytes < need || !aligned(workspace, 256)) {
        return fail(GS_ERR_ARG, "workspace not 256-byte aligned or smaller than %zu bytes", need);
    }
    const SortWorkspace w = carve_workspace(base, proj->n, capacity, kc.tiles_x, kc.tiles_y);
    unsigned* err = error_word(&s);
    if (!err) return s;
    cudaError_t e = bin_sort_async(*proj, kc.tiles_x, kc.tiles_y, (unsigned long long)capacity, w, keys, vals,
                                   tile_ranges, reinterpret_cast<unsigned long long*>(n_dup_device), err, o.spin,
                                   as_stream(stream));
    return e ? cuda_fail(e, "gs_bin_and_sort_async") : GS_OK;
}

int gs_render_fwd(const gs_proj* proj, const uint32_t* vals, const uint32_t* tile_ranges, const gs_camera* cam,
                  const gs_options* opt, float* image, float* t_final, uint32_t* n_contrib, void* stream) {
    Opts o;
    KernelCamera kc;
    int s;
    if ((s = resolve_options(opt, o)) || (s = make_camera(cam, o, kc)) || (s = check_proj_n(proj))) return s;
    if (!tile_ranges || !aligned(tile_ranges, 8)) return fail(GS_ERR_ARG, "tile_ranges NULL or misaligned");
    if (!image || !t_final || !n_contrib || !aligned(image, 4) || !aligned(t_final, 4) || !aligned(n_contrib, 4))
        return fail(GS_ERR_ARG, "image / t_final / n_contrib NULL or misaligned");
    if (proj->n > 0 && (!vals || !aligned(vals, 4))) return fail(GS_ERR_ARG, "vals NULL or misaligned");
    unsigned* err = error_word(&s);
    if (!err) return s;
    cudaError_t e = launch_render_fwd(o.staging, *proj, vals, tile_ranges, kc, image, t_final, n_contrib, o.spin, err,
                                      as_stream(stream));
    return e ? cuda_fail(e, "gs_render_fwd") : GS_OK;
}

// Shared body of gs_render_bwd (target = loss = NULL) and gs_render_bwd_sqerr.
static int render_bwd(const char* name, const gs_proj* proj, const uint32_t* vals, const uint32_t* tile_ranges,
               const gs_camera* cam, const gs_options* opt, const float* src, const float* target, float* loss,
               const float* t_final, const uint32_t* n_contrib, float* grad2d, void* stream) {
    Opts o;
    KernelCamera kc;
    int s;
    if ((s = resolve_options(opt, o)) || (s = make_camera(cam, o, kc)) || (s = check_proj_n(proj))) return s;
    if (!tile_ranges || !aligned(tile_ranges, 8)) return fail(GS_ERR_ARG, "%s: tile_ranges NULL or misaligned", name);
    if (!src || !t_final || !n_contrib || !aligned(src, 4) || !aligned(t_final, 4) || !aligned(n_contrib, 4))
        return fail(GS_ERR_ARG, "%s: image / dl_dimage, t_final or n_contrib NULL or misaligned", name);
    if (proj->n > 0 && (!vals || !aligned(vals, 4) || !grad2d || !aligned(grad2d, 16)))
        return fail(GS_ERR_ARG, "%s: vals or grad2d NULL or misaligned (grad2d needs 16 bytes)", name);
    if (target && !aligned(target, 4)) return fail(GS_ERR_ARG, "%s: target misaligned", name);
    if (loss && !aligned(loss, 4)) return fail(GS_ERR_ARG, "%s: loss misaligned", name);
    cudaStream_t st = as_stream(stream);
    if (proj->n > 0) {
        cudaError_t e = cudaMemsetAsync(grad2d, 0, (size_t)proj->n * 12 * sizeof(float), st);
        if (e) return cuda_fail(e, name);
    }
    if (loss) {
        cudaError_t e = cudaMemsetAsync(loss, 0, sizeof(float), st);
        if (e) return cuda_fail(e, name);
    }
    unsigned* err = error_word(&s);
    if (!err) return s;
    cudaError_t e = launch_render_bwd(o.bwd_mode, o.staging, o.thr, *proj, vals, tile_ranges, kc, src, target, loss,
                                      t_final, n_contrib, grad2d, o.spin, err, st);
    return e ? cuda_fail(e, name) : GS_OK;
}

int gs_render_bwd(const gs_proj* proj, const uint32_t* vals, const uint32_t* tile_ranges, const gs_camera* cam,
                  const gs_options* opt, const float* dl_dimage, const float* t_final, const uint32_t* n_contrib,
                  float* grad2d, void* stream) {
    return render_bwd("gs_render_bwd", proj, vals, tile_ranges, cam, opt, dl_dimage, nullptr, nullptr, t_final,
                      n_contrib, grad2d, stream);
}

int gs_render_bwd_sqerr(const gs_proj* proj, const uint32_t* vals, const uint32_t* tile_ranges, const gs_camera* cam,
                        const gs_options* opt, const float* image, const float* target, const float* t_final,
                        const uint32_t* n_contrib, float* grad2d, float* loss, void* stream) {
    if (!target) return fail(GS_ERR_ARG, "gs_render_bwd_sqerr: target is NULL");
    return render_bwd("gs_render_bwd_sqerr", proj, vals, tile_ranges, cam, opt, image, target, loss, t_final,
                      n_contrib, grad2d, stream);
}

int gs_preprocess_bwd(const gs_params* p, const gs_camera* cam, const gs_options* opt, const gs_proj* proj,
                      const float* grad2d, float* d_mean3d, float* d_log_scale, float* d_quat, float* d_opacity_logit,
                      float* d_sh, int32_t accumulate, void* stream) {
    Opts o;
    KernelCamera kc;
    int s;
    if ((s = resolve_options(opt, o)) || (s = make_camera(cam, o, kc)) || (s = check_params(p))) return s;
    if ((s = check_proj(proj, p->n))) return s;
    if (p->n > 0) {
        if (!grad2d || !aligned(grad2d, 16)) return fail(GS_ERR_ARG, "grad2d NULL or not 16-byte aligned");
        const void* outs[5] = {d_mean3d, d_log_scale, d_quat, d_opacity_logit, d_sh};
        for (const void* q : outs)
            if (!q || !aligned(q, 4)) return fail(GS_ERR_ARG, "a gradient output is NULL or misaligned");
    }
    unsigned* err = error_word(&s);
    if (!err) return s;
    cudaError_t e = launch_preprocess_bwd(o.deg, (int)p->n, *p, kc, proj->radius, grad2d, d_mean3d, d_log_scale,
                                          d_quat, d_opacity_logit, d_sh, accumulate, nullptr, o.spin, err,
                                          as_stream(stream));
    return e ? cuda_fail(e, "gs_preprocess_bwd") : GS_OK;
}

int gs_preprocess_bwd_stats(const gs_params* p, const gs_camera* cam, const gs_options* opt, const gs_proj* proj,
                            const float* grad2d, float* d_mean3d, float* d_log_scale, float* d_quat,
                            float* d_opacity_logit, float* d_sh, int32_t accumulate, const gs_densify_outputs* stats,
                            void* stream) {
    Opts o;
    KernelCamera kc;
    int s;
    if ((s = resolve_options(opt, o)) || (s = make_camera(cam, o, kc)) || (s = check_params(p))) return s;
    if ((s = check_proj(proj, p->n))) return s;
    if (!stats) return fail(GS_ERR_ARG, "stats is NULL (use gs_preprocess_bwd)");
    if (p->n > 0) {
        if (!grad2d || !aligned(grad2d, 16)) return fail(GS_ERR_ARG, "grad2d NULL or not 16-byte aligned");
        const void* outs[5] = {d_mean3d, d_log_scale, d_quat, d_opacity_logit, d_sh};
        for (const void* q : outs)
            if (!q || !aligned(q, 4)) return fail(GS_ERR_ARG, "a gradient output is NULL or misaligned");
        if (!stats->grad_norm_accum || !stats->view_count || !stats->max_radius ||
            !aligned(stats->grad_norm_accum, 4) || !aligned(stats->view_count, 4) || !aligned(stats->max_radius, 4) ||
            (stats->grad_mag && !aligned(stats->grad_mag, 4)))
            return fail(GS_ERR_ARG, "a statistics output is NULL or misaligned");
    }
    DensifyArgs d{stats->grad_norm_accum, stats->view_count, stats->max_radius, stats->grad_mag,
                  stats->ndc ? 0.5f * (float)kc.width : 1.f, stats->ndc ? 0.5f * (float)kc.height : 1.f};
    unsigned* err = error_word(&s);
    if (!err) return s;
    cudaError_t e = launch_preprocess_bwd(o.deg, (int)p->n, *p, kc, proj->radius, grad2d, d_mean3d, d_log_scale,
                                          d_quat, d_opacity_logit, d_sh, accumulate, &d, o.spin, err,
                                          as_stream(stream));
    return e ? cuda_fail(e, "gs_preprocess_bwd_stats") : GS_OK;
}

int gs_adam_step(gs_tensors* params, const gs_tensors* grads, gs_tensors* exp_avg, gs_tensors* exp_avg_sq,
                 const int32_t* radius, const gs_adam_options* opt, void* stream) {
    if (!params || !grads || !exp_avg || !exp_avg_sq || !opt)
        return fail(GS_ERR_ARG, "params, grads, exp_avg, exp_avg_sq or opt is NULL");
    const int64_t n = params->n;
    if (n < 0 || n > 0x7fffffffll) return fail(GS_ERR_ARG, "n = %lld outside 0..2^31-1", (long long)n);
    if (grads->n != n || exp_avg->n != n || exp_avg_sq->n != n)
        return fail(GS_ERR_ARG, "params, grads and moments must have the same n");
    if (opt->step < 1) return fail(GS_ERR_ARG, "step %d must be >= 1", opt->step);
    if (opt->sh_degree < 0 || opt->sh_degree > 3) return fail(GS_ERR_ARG, "sh_degree %d outside 0..3", opt->sh_degree);
    const float b1 = opt->beta1 == 0.f ? 0.9f : opt->beta1, b2 = opt->beta2 == 0.f ? 0.999f : opt->beta2;
    const float eps = opt->eps == 0.f ? 1e-15f : opt->eps;
    if (!(b1 > 0.f && b1 < 1.f) || !(b2 > 0.f && b2 < 1.f) || !(eps > 0.f) || !std::isfinite(eps))
        return fail(GS_ERR_ARG, "betas must lie in (0, 1) and eps be finite and positive");
    if (n == 0) return GS_OK;
    const long long k3 = 3ll * (opt->sh_degree + 1) * (opt->sh_degree + 1);
    if (n * k3 >= (1ll << 32) || n * (k3 + 11) / 4 + 5 >= (1ll << 32))
        return fail(GS_ERR_ARG, "n = %lld too large: the sh tensor must hold fewer than 2^32 floats", (long long)n);
    const gs_tensors* ts[4] = {params, grads, exp_avg, exp_avg_sq};
    for (const gs_tensors* t : ts) {
        const void* ptrs[5] = {t->mean3d, t->log_scale, t->quat, t->opacity_logit, t->sh};
        for (const void* q : ptrs)
            if (!q || !aligned(q, 16)) return fail(GS_ERR_ARG, "a tensor pointer is NULL or not 16-byte aligned");
    }
    if (!radius || !aligned(radius, 4)) return fail(GS_ERR_ARG, "radius NULL or misaligned");
    cudaError_t e = launch_adam(*params, *grads, *exp_avg, *exp_avg_sq, radius, *opt, opt->sh_degree, b1, b2, eps,
                                as_stream(stream));
    return e ? cuda_fail(e, "gs_adam_step") : GS_OK;
}

int gs_densify_stats(const gs_proj* proj, const float* grad2d, int32_t width, int32_t height, int32_t ndc,
                     float* grad_norm_accum, int32_t* view_count, int32_t* max_radius,
                     const gs_tensors* param_grads, float* grad_mag, int32_t sh_degree, void* stream) {
    int s;
    if ((s = check_proj_n(proj))) return s;
    if (sh_degree < 0 || sh_degree > 3) return fail(GS_ERR_ARG, "sh_degree %d outside 0..3", sh_degree);
    if (ndc && (width <= 0 || height <= 0)) return fail(GS_ERR_ARG, "ndc needs the image size");
    const int64_t n = proj->n;
    if (n == 0) return GS_OK;
    if (!proj->radius || !aligned(proj->radius, 4)) return fail(GS_ERR_ARG, "proj.radius NULL or misaligned");
    if (!grad2d || !aligned(grad2d, 16)) return fail(GS_ERR_ARG, "grad2d NULL or not 16-byte aligned");
    if (!grad_norm_accum || !view_count || !max_radius || !aligned(grad_norm_accum, 4) || !aligned(view_count, 4) ||
        !aligned(max_radius, 4))
        return fail(GS_ERR_ARG, "grad_norm_accum, view_count or max_radius NULL or misaligned");
    if (param_grads) {
        if (param_grads->n != n) return fail(GS_ERR_ARG, "param_grads.n does not match proj.n");
        const void* ptrs[5] = {param_grads->mean3d, param_grads->log_scale, param_grads->quat,
                               param_grads->opacity_logit, param_grads->sh};
        for (const void* q : ptrs)
            if (!q || !aligned(q, 16)) return fail(GS_ERR_ARG, "a param_grads pointer is NULL or not 16-byte aligned");
        if (!grad_mag || !aligned(grad_mag, 4)) return fail(GS_ERR_ARG, "grad_mag NULL or misaligned");
    }
    const float sx = ndc ? 0.5f * (float)width : 1.f, sy = ndc ? 0.5f * (float)height : 1.f;
    cudaError_t e = launch_densify_stats(sh_degree, (int)n, proj->radius, grad2d, sx, sy, grad_norm_accum, view_count,
                                         max_radius, param_grads, grad_mag, as_stream(stream));
    return e ? cuda_fail(e, "gs_densify_stats") : GS_OK;
}

size_t gs_loss_workspace_bytes(int32_t width, int32_t height) {
    if (width <= 0 || height <= 0 || width > kMaxImageSide || height > kMaxImageSide) return 0;
    return loss_workspace_bytes(width, height);
}

int gs_loss_l1_dssim(const float* image, const float* target, int32_t width, int32_t height, float lambda,
                     void* workspace, size_t workspace_bytes, float* loss, float* dl_dimage, void* stream) {
    if (width <= 0 || height <= 0 || width > kMaxImageSide || height > kMaxImageSide)
        return fail(GS_ERR_ARG, "image size %dx%d outside 1..%d", width, height, kMaxImageSide);
    if (!(lambda >= 0.f && lambda <= 1.f)) return fail(GS_ERR_ARG, "lambda must lie in [0, 1]");
    if (!image || !target || !loss || !dl_dimage || !aligned(image, 4) || !aligned(target, 4) || !aligned(loss, 4) ||
        !aligned(dl_dimage, 4))
        return fail(GS_ERR_ARG, "image, target, loss or dl_dimage NULL or misaligned");
    const size_t need = loss_workspace_bytes(width, height);
    if (!workspace || workspace_bytes < need || !aligned(workspace, 256))
        return fail(GS_ERR_ARG, "workspace NULL, not 256-byte aligned or smaller than %zu bytes", need);
    cudaError_t e = launch_loss_l1_dssim(image, target, width, height, lambda, workspace, loss, dl_dimage,
                                         as_stream(stream));
    return e ? cuda_fail(e, "gs_loss_l1_dssim") : GS_OK;
}

int gs_preprocess2d(const gs_params* p, const gs_camera* cam, const gs_options* opt, gs_proj* out, float* rec2d,
                    void* stream) {
    Opts o;
    KernelCamera kc;
    int s;
    if ((s = resolve_options(opt, o)) || (s = make_camera(cam, o, kc)) || (s = check_params(p))) return s;
    if ((s = check_proj(out, p->n))) return s;
    if (p->n > 0 && (!rec2d || !aligned(rec2d, 16))) return fail(GS_ERR_ARG, "rec2d NULL or not 16-byte aligned");
    cudaError_t e = launch_preprocess2d(o.deg, (int)p->n, *p, kc, *out, rec2d, as_stream(stream));
    return e ? cuda_fail(e, "gs_preprocess2d") : GS_OK;
}

int gs_render2d_fwd(const float* rec2d, int64_t n, const uint32_t* vals, const uint32_t* tile_ranges,
                    const gs_camera* cam, const gs_options* opt, float* image, float* t_final, uint32_t* n_contrib,
                    void* stream) {
    Opts o;
    KernelCamera kc;
    int s;
    if ((s = resolve_options(opt, o)) || (s = make_camera(cam, o, kc))) return s;
    if (n < 0 || n > 0x7fffffffll) return fail(GS_ERR_ARG, "n = %lld outside 0..2^31-1", (long long)n);
    if (!tile_ranges || !aligned(tile_ranges, 8)) return fail(GS_ERR_ARG, "tile_ranges NULL or misaligned");
    if (!image || !t_final || !n_contrib || !aligned(image, 4) || !aligned(t_final, 4) || !aligned(n_contrib, 4))
        return fail(GS_ERR_ARG, "image / t_final / n_contrib NULL or misaligned");
    if (n > 0 && (!vals || !aligned(vals, 4) || !rec2d || !aligned(rec2d, 16)))
        return fail(GS_ERR_ARG, "vals or rec2d NULL or misaligned (rec2d needs 16 bytes)");
    unsigned* err = error_word(&s);
    if (!err) return s;
    cudaError_t e = launch_render2d_fwd(rec2d, (unsigned)n, vals, tile_ranges, kc, image, t_final, n_contrib, o.spin,
                                        err, as_stream(stream));
    return e ? cuda_fail(e, "gs_render2d_fwd") : GS_OK;
}

int gs_render2d_bwd(const float* rec2d, int64_t n, const uint32_t* vals, const uint32_t* tile_ranges,
                    const gs_camera* cam, const gs_options* opt, const float* dl_dimage, const float* t_final,
                    const uint32_t* n_contrib, float* grad2d, void* stream) {
    Opts o;
    KernelCamera kc;
    int s;
    if ((s = resolve_options(opt, o)) || (s = make_camera(cam, o, kc))) return s;
    if (o.bwd_mode == GS_BWD_SM) return fail(GS_ERR_ARG, "the surfel backward has no GS_BWD_SM mode");
    if (n < 0 || n > 0x7fffffffll) return fail(GS_ERR_ARG, "n = %lld outside 0..2^31-1", (long long)n);
    if (!tile_ranges || !aligned(tile_ranges, 8)) return fail(GS_ERR_ARG, "tile_ranges NULL or misaligned");
    if (!dl_dimage || !t_final || !n_contrib || !aligned(dl_dimage, 4) || !aligned(t_final, 4) ||
        !aligned(n_contrib, 4))
        return fail(GS_ERR_ARG, "dl_dimage / t_final / n_contrib NULL or misaligned");
    if (n > 0 && (!vals || !aligned(vals, 4) || !rec2d || !aligned(rec2d, 16) || !grad2d || !aligned(grad2d, 16)))
        return fail(GS_ERR_ARG, "vals, rec2d or grad2d NULL or misaligned (rec2d and grad2d need 16 bytes)");
    unsigned* err = error_word(&s);
    if (!err) return s;
    cudaStream_t st = as_stream(stream);
    if (n > 0) {
        cudaError_t e = cudaMemsetAsync(grad2d, 0, (size_t)n * 16 * sizeof(float), st);
        if (e) return cuda_fail(e, "gs_render2d_bwd: zero grad2d");
    }
    cudaError_t e = launch_render2d_bwd(o.bwd_mode, o.thr, rec2d, (unsigned)n, vals, tile_ranges, kc, dl_dimage, t_final,
                                        n_contrib, grad2d, o.spin, err, st);
    return e ? cuda_fail(e, "gs_render2d_bwd") : GS_OK;
}

int gs_preprocess2d_bwd(const gs_params* p, const gs_camera* cam, const gs_options* opt, const gs_proj* proj,
                        const float* grad2d, float* d_mean3d, float* d_log_scale, float* d_quat, float* d_opacity_logit,
                        float* d_sh, int32_t accumulate, void* stream) {
    Opts o;
    KernelCamera kc;
    int s;
    if ((s = resolve_options(opt, o)) || (s = make_camera(cam, o, kc)) || (s = check_params(p))) return s;
    if ((s = check_proj(proj, p->n))) return s;
    if (p->n > 0) {
        if (!grad2d || !aligned(grad2d, 16)) return fail(GS_ERR_ARG, "grad2d NULL or not 16-byte aligned");
        const void* outs[5] = {d_mean3d, d_log_scale, d_quat, d_opacity_logit, d_sh};
        for (const void* q : outs)
            if (!q || !aligned(q, 4)) return fail(GS_ERR_ARG, "a gradient output is NULL or misaligned");
    }
    cudaError_t e = launch_preprocess2d_bwd(o.deg, (int)p->n, *p, kc, proj->radius, grad2d, d_mean3d, d_log_scale,
                                            d_quat, d_opacity_logit, d_sh, accumulate, as_stream(stream));
    return e ? cuda_fail(e, "gs_preprocess2d_bwd") : GS_OK;
}

// ---- the training step with host buffers --------------------------------------------------

}  // extern "C"

struct gs_step_context {
    int device;
    long long n, capacity;
    int deg, max_w, max_h;
    // device buffers (each its own allocation, 256-byte aligned)
    float *mean3d, *log_scale, *quat, *logit, *sh;       // parameters
    float *d_mean3d, *d_log_scale, *d_quat, *d_logit, *d_sh;  // their gradients
    float *rec, *depth;
    int* radius;
    unsigned* tiles_touched;
    void* ws;
    size_t ws_bytes;
    unsigned *vals, *ranges;
    unsigned long long* n_dup;
    float *image, *t_final, *target, *grad2d, *loss;
    unsigned* n_contrib;
};

namespace {

void free_context(gs_step_context* c) {
    void* ptrs[] = {c->mean3d, c->log_scale, c->quat, c->logit, c->sh, c->d_mean3d, c->d_log_scale, c->d_quat,
                    c->d_logit, c->d_sh, c->rec, c->depth, c->radius, c->tiles_touched, c->ws, c->vals,
                    c->ranges, c->n_dup, c->image, c->t_final, c->target, c->grad2d, c->loss, c->n_contrib};
    for (void* q : ptrs)
        if (q) cudaFree(q);
    delete c;
}

}  // namespace

extern "C" {

int gs_step_context_create(int64_t n, int32_t sh_degree, int32_t max_width, int32_t max_height, int64_t capacity,
                           gs_step_context** out) {
    if (!out) return fail(GS_ERR_ARG, "gs_step_context_create: out is NULL");
    if (n < 0 || n >= (1ll << 31)) return fail(GS_ERR_ARG, "gs_step_context_create: n = %lld outside 0..2^31-1",
                                               (long long)n);
    if (sh_degree < 0 || sh_degree > 3) return fail(GS_ERR_ARG, "gs_step_context_create: sh_degree %d", sh_degree);
    if (max_width <= 0 || max_height <= 0 || max_width > kMaxImageSide || max_height > kMaxImageSide)
        return fail(GS_ERR_ARG, "gs_step_context_create: image %d x %d", max_width, max_height);
    const long long tx = (max_width + kTile - 1) / kTile, ty = (max_height + kTile - 1) / kTile;
    if (!counting_path(tx * ty))
        return fail(GS_ERR_ARG, "gs_step_context_create: %lld tiles; the step without host synchronisation "
                    "handles images of up to 49152 tiles", tx * ty);
    if (capacity < 0 || capacity > 0x7fffffffll)
        return fail(GS_ERR_ARG, "gs_step_context_create: capacity outside 0..2^31-1");
    auto* c = new gs_step_context{};
    c->n = n;
    c->capacity = capacity;
    c->deg = sh_degree;
    c->max_w = max_width;
    c->max_h = max_height;
    cudaError_t e = cudaGetDevice(&c->device);
    const size_t nn = (size_t)(n > 0 ? n : 1), K3 = 3 * (size_t)(sh_degree + 1) * (sh_degree + 1);
    const size_t P = (size_t)max_width * max_height;
    auto get = [&](auto** p, size_t bytes) {
        if (!e) e = cudaMalloc(reinterpret_cast<void**>(p), bytes > 0 ? bytes : 4);
    };
    get(&c->mean3d, 12 * nn); get(&c->log_scale, 12 * nn); get(&c->quat, 16 * nn); get(&c->logit, 4 * nn);
    get(&c->sh, 4 * K3 * nn);
    get(&c->d_mean3d, 12 * nn); get(&c->d_log_scale, 12 * nn); get(&c->d_quat, 16 * nn); get(&c->d_logit, 4 * nn);
    get(&c->d_sh, 4 * K3 * nn);
    get(&c->rec, 48 * nn); get(&c->depth, 4 * nn); get(&c->radius, 4 * nn); get(&c->tiles_touched, 4 * nn);
    c->ws_bytes = gs_sort_workspace_bytes(n, capacity, max_width, max_height);
    get(&c->ws, c->ws_bytes);
    get(&c->vals, 4 * (size_t)(capacity > 0 ? capacity : 1)); get(&c->ranges, 8 * (size_t)(tx * ty));
    get(&c->n_dup, 8);
    get(&c->image, 12 * P); get(&c->t_final, 4 * P); get(&c->target, 12 * P); get(&c->n_contrib, 4 * P);
    get(&c->grad2d, 48 * nn); get(&c->loss, 4);
    if (e) {
        free_context(c);
        return cuda_fail(e, "gs_step_context_create");
    }
    *out = c;
    return GS_OK;
}

int gs_step_context_destroy(gs_step_context* ctx) {
    if (!ctx) return GS_OK;
    int prev = 0;
    cudaGetDevice(&prev);
    cudaSetDevice(ctx->device);
    const cudaError_t e = cudaDeviceSynchronize();
    free_context(ctx);
    cudaSetDevice(prev);
    return e ? cuda_fail(e, "gs_step_context_destroy") : GS_OK;
}

int gs_train_step_host(gs_step_context* ctx, const gs_params* hp, const float* host_target, const gs_camera* cam,
                       const gs_options* opt, const gs_tensors* hg, float* host_loss, int64_t* host_n_dup,
                       void* stream) {
    if (!ctx || !hp || !host_target || !cam || !hg) return fail(GS_ERR_ARG, "gs_train_step_host: NULL argument");
    Opts o;
    KernelCamera kc;
    int s;
    if ((s = resolve_options(opt, o)) || (s = make_camera(cam, o, kc))) return s;
    if (o.deg != ctx->deg) return fail(GS_ERR_ARG, "gs_train_step_host: sh_degree %d, context %d", o.deg, ctx->deg);
    int dev = -1;
    if (cudaGetDevice(&dev) != cudaSuccess || dev != ctx->device)
        return fail(GS_ERR_ARG, "gs_train_step_host: current device %d, the context's is %d", dev, ctx->device);
    if (hp->n != ctx->n || hg->n != ctx->n)
        return fail(GS_ERR_ARG, "gs_train_step_host: n = %lld / %lld, context %lld", (long long)hp->n,
                    (long long)hg->n, ctx->n);
    if (cam->width > ctx->max_w || cam->height > ctx->max_h)
        return fail(GS_ERR_ARG, "gs_train_step_host: image %d x %d, context at most %d x %d", cam->width, cam->height,
                    ctx->max_w, ctx->max_h);
    const size_t n = (size_t)ctx->n, K3 = 3 * (size_t)(ctx->deg + 1) * (ctx->deg + 1);
    if (n > 0 && (!hp->mean3d || !hp->log_scale || !hp->quat || !hp->opacity_logit || !hp->sh || !hg->mean3d ||
                  !hg->log_scale || !hg->quat || !hg->opacity_logit || !hg->sh))
        return fail(GS_ERR_ARG, "gs_train_step_host: a parameter or gradient array is NULL");
    cudaStream_t st = as_stream(stream);
    const size_t P = (size_t)cam->width * cam->height;
    // host -> device: one asynchronous copy per array
    struct Cp { void* dst; const void* src; size_t bytes; };
    const Cp in[] = {{ctx->mean3d, hp->mean3d, 12 * n}, {ctx->log_scale, hp->log_scale, 12 * n},
                     {ctx->quat, hp->quat, 16 * n}, {ctx->logit, hp->opacity_logit, 4 * n},
                     {ctx->sh, hp->sh, 4 * K3 * n}, {ctx->target, host_target, 12 * P}};
    for (const Cp& c : in) {
        if (c.bytes == 0) continue;
        const cudaError_t e = cudaMemcpyAsync(c.dst, c.src, c.bytes, cudaMemcpyHostToDevice, st);
        if (e) return cuda_fail(e, "gs_train_step_host: copy in");
    }
    const gs_params dp{ctx->mean3d, ctx->log_scale, ctx->quat, ctx->logit, ctx->sh, ctx->n};
    gs_proj proj{ctx->rec, ctx->depth, ctx->radius, ctx->tiles_touched, ctx->n};
    if ((s = gs_preprocess(&dp, cam, opt, &proj, stream))) return s;
    if ((s = gs_bin_and_sort_async(&proj, cam, opt, ctx->ws, ctx->ws_bytes, nullptr, ctx->vals, ctx->capacity,
                                   reinterpret_cast<uint64_t*>(ctx->n_dup), ctx->ranges, stream)))
        return s;
    if ((s = gs_render_fwd(&proj, ctx->vals, ctx->ranges, cam, opt, ctx->image, ctx->t_final, ctx->n_contrib,
                           stream)))
        return s;
    if ((s = gs_render_bwd_sqerr(&proj, ctx->vals, ctx->ranges, cam, opt, ctx->image, ctx->target, ctx->t_final,
                                 ctx->n_contrib, ctx->grad2d, ctx->loss, stream)))
        return s;
    if ((s = gs_preprocess_bwd(&dp, cam, opt, &proj, ctx->grad2d, ctx->d_mean3d, ctx->d_log_scale, ctx->d_quat,
                               ctx->d_logit, ctx->d_sh, 0, stream)))
        return s;
    // device -> host
    const Cp out[] = {{hg->mean3d, ctx->d_mean3d, 12 * n}, {hg->log_scale, ctx->d_log_scale, 12 * n},
                      {hg->quat, ctx->d_quat, 16 * n}, {hg->opacity_logit, ctx->d_logit, 4 * n},
                      {hg->sh, ctx->d_sh, 4 * K3 * n}, {host_loss, ctx->loss, host_loss ? 4u : 0u},
                      {host_n_dup, ctx->n_dup, host_n_dup ? 8u : 0u}};
    for (const Cp& c : out) {
        if (c.bytes == 0) continue;
        const cudaError_t e = cudaMemcpyAsync(c.dst, c.src, c.bytes, cudaMemcpyDeviceToHost, st);
        if (e) return cuda_fail(e, "gs_train_step_host: copy out");
    }
    return GS_OK;
}

}  // extern "C"

