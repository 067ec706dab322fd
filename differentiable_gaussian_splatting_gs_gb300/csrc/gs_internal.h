// Declarations shared by the library's translation units (host side).
#pragma once

#include <atomic>

#include <cuda_runtime.h>
#include <stddef.h>

#include "gs.h"

namespace gs {

struct KernelCamera;

// Adds k to the process-wide count of kernel launches (reported by gs_kernel_launches).
void count_launches(int k);

// Launches `kernel` on `st` with programmatic stream serialization: its blocks may be dispatched
// while the previous kernel of the stream is still running (hiding the launch gap between the
// step's dependent kernels, also inside a captured graph). Every kernel launched this way calls
// pdl_wait (gs_common.cuh) before reading what the kernel before it may write or writing what it
// may read. After a non-kernel operation (a memset, a copy, an event) the launch is ordered as
// usual.
template <class... KArgs, class... Args>
inline cudaError_t launch_pdl(void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem, cudaStream_t st,
                              Args... args) {
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = grid;
    cfg.blockDim = block;
    cfg.dynamicSmemBytes = smem;
    cfg.stream = st;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, kernel, static_cast<KArgs>(args)...);
}

// Sort workspace carved from the caller's buffer (all pieces 256-byte aligned).
struct SortWorkspace {
    unsigned *dkA, *dkB, *dvA, *dvB;   // depth-sort keys / values, ping-pong, N each
    unsigned *hist, *totals;           // radix histograms [256][blocks] and digit totals [256]
    unsigned long long *bsum, *boff, *total;  // duplicate counts per 256 Gaussians, offsets, total D
    unsigned* nvis;                    // number of Gaussians with radius > 0 (left by the second depth pass)
    unsigned char* sweep;              // depth sort: digit histograms, tickets, look-back words (zeroed per call)
    size_t sweep_bytes;
    int sweep_blocks;                  // 4096-item blocks of a depth pass
    unsigned *tA, *tB, *vB;            // radix tile pass: keys ping-pong and values, capacity each
    // counting tile pass, two levels: super-tiles of 4x4 tiles (coarse), then tiles (fine)
    uint2* crect;                      // packed tile rectangle per depth-ordered Gaussian
    unsigned long long *ssum, *soff;   // super-tile entries per 256 Gaussians, offsets
    unsigned long long* ctotal;        // super-tile entries in all (D')
    unsigned* table;                   // coarse: chunk x super-tile counts, then offsets
    unsigned* group_sum;               // coarse: per group of table rows, the column sums
    unsigned *stile_total, *stile_start; // coarse: entries per super-tile, exclusive scan
    uint2* crange;                     // coarse: [start, end) of each super-tile's list
    unsigned* cvals;                   // coarse: the lists (depth positions), capacity entries
    unsigned *chunk_first, *nchunks;   // coarse: first Gaussian of each chunk, chunks used
    long long cmax;                    // coarse: rows of the chunk x super-tile table
    unsigned *seg_first, *nseg;        // fine: first segment of each super-tile, segments used
    unsigned* fcount;                  // fine: per segment and tile of its super-tile, counts then offsets
    long long seg_cap;                 // fine: segments the workspace holds
    unsigned *tile_total, *tile_start; // fine: entries per tile, exclusive scan
    int sx, sy;                        // super-tiles per row and column
    size_t bytes;                      // total size
};

// Workspace layout for n Gaussians, at most `cap` duplicates and tiles_x x tiles_y tiles.
SortWorkspace carve_workspace(void* base, long long n, long long cap, int tiles_x, int tiles_y);
// Phase 1 of the binning (depth sort, duplicate counts, on the counting path also the tile
// table, starts and ranges); `ranges` and `capacity` are used on the counting path only, and
// overflow_err (may be NULL) receives the check bit when D exceeds the capacity there;
// total_copy (may be NULL) receives D on the counting path.
cudaError_t bin_count(const gs_proj& proj, int tiles_x, int tiles_y, const SortWorkspace& w, unsigned* err,
                      unsigned spin_limit, unsigned long long capacity, unsigned* ranges, unsigned* overflow_err,
                      unsigned long long* total_copy, cudaStream_t st);
cudaError_t bin_emit_sort(const gs_proj& proj, int tiles_x, int tiles_y, unsigned d, unsigned long long capacity,
                          const SortWorkspace& w, uint64_t* keys, unsigned* vals, unsigned* ranges, unsigned* err,
                          cudaStream_t st);
cudaError_t bin_sort_async(const gs_proj& proj, int tiles_x, int tiles_y, unsigned long long capacity,
                           const SortWorkspace& w, uint64_t* keys, unsigned* vals, unsigned* ranges,
                           unsigned long long* n_dup_dev, unsigned* err, unsigned spin_limit, cudaStream_t st);
bool counting_path(long long tiles);
// Self-test of the depth sort's bounded look-back (a predecessor that never publishes); needs
// kSelftestLookbackBytes of device workspace, 16-byte aligned.
constexpr size_t kSelftestLookbackBytes = 106512;
cudaError_t selftest_lookback(unsigned char* ws, unsigned spin_limit, unsigned* err, cudaStream_t st);

// Number of SMs of the current device (looked up once per device; 1 if the query fails).
int device_sm_count();

// Blocks of `kernel` (`threads` threads, `smem` bytes of dynamic shared memory) resident on the
// current device at once: SMs x blocks per SM, looked up once per device (the caller keeps one
// cache per kernel); 0 if the query fails.
template <class Kernel>
int resident_blocks(Kernel kernel, int threads, size_t smem, std::atomic<int> (&cache)[256]) {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 256) return 0;
    int v = cache[dev].load(std::memory_order_relaxed);
    if (v == 0) {
        int per = 0;
        if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per, kernel, threads, smem) != cudaSuccess) return 0;
        v = device_sm_count() * (per > 0 ? per : 1);
        cache[dev].store(v, std::memory_order_relaxed);
    }
    return v;
}

cudaError_t launch_preprocess(int deg, int n, const gs_params& p, const KernelCamera& cam, const gs_proj& out,
                              unsigned spin_limit, unsigned* err, cudaStream_t st);
// Post-backward statistics written by the preprocess backward (gs_preprocess_bwd_stats).
struct DensifyArgs {
    float* accum;      // += |(sx, sy) * dL/dmean2d| for radius > 0
    int* count;        // += 1 for radius > 0
    int* max_radius;   // max with the radius
    float* grad_mag;   // 2-norm of the view's parameter gradients (NULL: not written)
    float sx, sy;
};
cudaError_t launch_preprocess_bwd(int deg, int n, const gs_params& p, const KernelCamera& cam, const int* radius,
                                  const float* grad2d, float* dm, float* dls, float* dq, float* dlg, float* dsh,
                                  int accumulate, const DensifyArgs* stats, unsigned spin_limit, unsigned* err,
                                  cudaStream_t st);
cudaError_t launch_render_fwd(int staging, const gs_proj& proj, const unsigned* vals, const unsigned* ranges,
                              const KernelCamera& cam, float* image, float* t_final, unsigned* n_contrib,
                              unsigned spin_limit, unsigned* err, cudaStream_t st);
cudaError_t launch_render_bwd(int mode, int staging, int thr, const gs_proj& proj, const unsigned* vals,
                              const unsigned* ranges, const KernelCamera& cam, const float* dl_dimage,
                              const float* target, float* loss, const float* t_final, const unsigned* n_contrib,
                              float* grad2d, unsigned spin_limit, unsigned* err, cudaStream_t st);

cudaError_t launch_adam(const gs_tensors& P, const gs_tensors& G, const gs_tensors& M, const gs_tensors& V,
                        const int* radius, const gs_adam_options& o, int deg, float beta1, float beta2, float eps,
                        cudaStream_t st);
cudaError_t launch_densify_stats(int deg, int n, const int* radius, const float* grad2d, float sx, float sy,
                                 float* accum, int* count, int* max_radius, const gs_tensors* pg, float* grad_mag,
                                 cudaStream_t st);
size_t loss_workspace_bytes(int width, int height);
cudaError_t launch_loss_l1_dssim(const float* img, const float* tgt, int width, int height, float lam, void* ws,
                                 float* loss, float* dl, cudaStream_t st);
cudaError_t launch_preprocess2d(int deg, int n, const gs_params& p, const KernelCamera& cam, const gs_proj& out,
                                float* rec2d, cudaStream_t st);
cudaError_t launch_render2d_fwd(const float* rec2d, unsigned n, const unsigned* vals, const unsigned* ranges,
                                const KernelCamera& cam, float* image, float* t_final, unsigned* n_contrib,
                                unsigned spin_limit, unsigned* err, cudaStream_t st);
cudaError_t launch_render2d_bwd(int mode, int thr, const float* rec2d, unsigned n, const unsigned* vals,
                                const unsigned* ranges, const KernelCamera& cam, const float* dl_dimage,
                                const float* t_final, const unsigned* n_contrib, float* grad, unsigned spin_limit,
                                unsigned* err, cudaStream_t st);
cudaError_t launch_preprocess2d_bwd(int deg, int n, const gs_params& p, const KernelCamera& cam, const int* radius,
                                    const float* grad, float* dm, float* dls, float* dq, float* dlg, float* dsh,
                                    int accumulate, cudaStream_t st);

}  // namespace gs
