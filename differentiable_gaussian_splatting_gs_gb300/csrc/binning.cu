// Tile duplication and sorting: the binning stage of the tile rasterization pipeline (DISTWAR:
// Fast Differentiable Rendering on Raster-based Rendering Pipelines, Abstract, names the
// rasterization pipeline; the duplication, keying and sort follow 3D Gaussian splatting's tile
// rasterizer).
//
// Result: for every Gaussian with radius > 0 and every tile of its tile rectangle one entry,
// ordered by (tile, float32 depth bits, Gaussian index): the stable sort of the 64-bit keys
// (tile << 32 | depth bits) of the index-ordered duplicate list. It is computed as an LSD radix
// sort whose low digits run over the Gaussians instead of their duplicates:
//   1. the Gaussians with radius > 0 are sorted stably by their 32 depth bits (4 passes of 8 bits;
//      the first pass drops culled Gaussians, so the others run over the V visible ones);
//   2. the most significant digit, the whole tile id, is one stable counting pass over the
//      duplicates of the depth-ordered Gaussians (images of up to 49,152 tiles; see the counting
//      pass below). Duplicates of one tile keep the depth order, and Gaussians of equal depth bits
//      keep index order from the stable depth passes.
// Larger images fall back to emitting the duplicates in depth order and radix-sorting them by
// tile id in 8-bit passes.
//
// Radix pass = histogram (per 4096-item block, 8-bit digit), scan (per digit over blocks),
// stable scatter (per warp: 8 rounds of 32 consecutive items ranked with match_any, then the
// block's items reordered by digit in shared memory and written as coalesced runs).
#include "gs_common.cuh"
#include "gs_internal.h"

namespace gs {

constexpr int kSortThreads = 256;
constexpr int kSortRounds = 16;                          // rounds of 32 items per warp
constexpr int kSortItems = kSortThreads * kSortRounds;  // 4096 items per block
constexpr int kWarpItems = 32 * kSortRounds;            // 512 items per warp

// Super-tiles: blocks of kSuper x kSuper tiles, the coarse level of the two-level counting pass;
// the fine level splits each super-tile's list into segments of kSeg entries.
constexpr int kSuper = 4;
constexpr int kSeg = 256;                      // coarse entries per segment
constexpr int kRounds = kSeg / 32;             // rounds of 32 entries per segment

// The rectangle of super-tiles overlapped by a packed tile rectangle (x0 | y0 << 16, w | h << 16),
// packed the same way; empty stays empty.
__device__ __forceinline__ uint2 super_rect(uint2 r) {
    const unsigned w = r.y & 0xffffu, h = r.y >> 16;
    if (w == 0u || h == 0u) return make_uint2(0u, 0u);
    const unsigned x0 = r.x & 0xffffu, y0 = r.x >> 16;
    const unsigned sx0 = x0 / kSuper, sy0 = y0 / kSuper;
    const unsigned sx1 = (x0 + w - 1u) / kSuper, sy1 = (y0 + h - 1u) / kSuper;
    return make_uint2(sx0 | (sy0 << 16), (sx1 - sx0 + 1u) | ((sy1 - sy0 + 1u) << 16));
}

// Number of items of a pass: the host bound n, or the count the previous pass left on the device.
__device__ __forceinline__ int item_count(int n, const unsigned* n_dev) {
    return n_dev ? min(n, (int)*n_dev) : n;
}

// Item validity: inside the count and, when `radius` is given (first depth pass, whose values are
// the Gaussian indices), a Gaussian that was not culled.
__device__ __forceinline__ bool item_valid(int idx, int n, const int* radius) {
    return idx < n && (!radius || radius[idx] > 0);
}

__global__ void __launch_bounds__(kSortThreads) k_radix_hist(const unsigned* __restrict__ keys, int n_bound,
                                                             const unsigned* __restrict__ n_dev,
                                                             const int* __restrict__ radius, int shift, unsigned mask,
                                                             unsigned* __restrict__ hist, int nblocks) {
    __shared__ unsigned h[8][256];
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int n = item_count(n_bound, n_dev);
    for (int i = threadIdx.x; i < 8 * 256; i += kSortThreads) (&h[0][0])[i] = 0u;
    const int base = blockIdx.x * kSortItems + warp * kWarpItems + lane;
    unsigned d[kSortRounds];
#pragma unroll
    for (int r = 0; r < kSortRounds; ++r) {
        const int idx = base + r * 32;
        d[r] = item_valid(idx, n, radius) ? (keys[idx] >> shift) & mask : 0x100u;
    }
    __syncthreads();
#pragma unroll
    for (int r = 0; r < kSortRounds; ++r) {
        const unsigned peers = __match_any_sync(0xffffffffu, d[r]);
        if (d[r] != 0x100u && (peers & lanemask_lt()) == 0u) h[warp][d[r]] += __popc(peers);
        __syncwarp();
    }
    __syncthreads();
    const int dg = threadIdx.x;
    unsigned sum = 0;
#pragma unroll
    for (int w = 0; w < 8; ++w) sum += h[w][dg];
    hist[(size_t)dg * nblocks + blockIdx.x] = sum;
}

// Exclusive scan of one digit's row of per-block counts (one block of 1024 threads per digit).
// count_out (optional, zeroed beforehand) receives the number of valid items of the pass.
__global__ void __launch_bounds__(1024) k_radix_scan(unsigned* __restrict__ hist, int nblocks,
                                                     unsigned* __restrict__ totals, unsigned* __restrict__ count_out) {
    __shared__ unsigned wsum[32];
    __shared__ unsigned carry;
    unsigned* row = hist + (size_t)blockIdx.x * nblocks;
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    if (threadIdx.x == 0) carry = 0u;
    __syncthreads();
    for (int base = 0; base < nblocks; base += 1024) {
        const int i = base + threadIdx.x;
        const unsigned v = i < nblocks ? row[i] : 0u;
        unsigned x = v;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const unsigned y = __shfl_up_sync(0xffffffffu, x, o);
            if (lane >= o) x += y;
        }
        if (lane == 31) wsum[warp] = x;
        __syncthreads();
        if (warp == 0) {
            unsigned s = wsum[lane];
#pragma unroll
            for (int o = 1; o < 32; o <<= 1) {
                const unsigned y = __shfl_up_sync(0xffffffffu, s, o);
                if (lane >= o) s += y;
            }
            wsum[lane] = s;  // inclusive
        }
        __syncthreads();
        const unsigned wpre = warp ? wsum[warp - 1] : 0u;
        if (i < nblocks) row[i] = carry + wpre + x - v;
        __syncthreads();
        if (threadIdx.x == 0) carry += wsum[31];
        __syncthreads();
    }
    if (threadIdx.x == 0) {
        totals[blockIdx.x] = carry;
        if (count_out) atomicAdd(count_out, carry);
    }
}

// Stable scatter of one 8-bit digit. IOTA: the values are the item indices. KEY64: also write
// the 64-bit key (key << 32 | depth_bits[value]) of every item.
//
// Each warp ranks its 256 items (8 rounds of 32, in index order) with match_any; the block then
// reorders its valid items by digit in shared memory and writes every digit's run to consecutive
// global addresses, so the global writes are coalesced. Invalid items (beyond the count, or culled
// in the first depth pass) take no part: the output holds the valid items only.
template <bool IOTA, bool KEY64>
__global__ void __launch_bounds__(kSortThreads) k_radix_scatter(
    const unsigned* __restrict__ keys_in, const unsigned* __restrict__ vals_in, unsigned* __restrict__ keys_out,
    unsigned* __restrict__ vals_out, int n_bound, const unsigned* __restrict__ n_dev, const int* __restrict__ radius,
    int shift, unsigned mask, const unsigned* __restrict__ hist, const unsigned* __restrict__ totals, int nblocks,
    unsigned long long* __restrict__ keys64, const unsigned* __restrict__ depth_bits) {
    __shared__ unsigned woff[8][256];      // per-warp digit counts, then block-local offsets
    __shared__ unsigned lbase[256];        // block-local start of each digit
    __shared__ unsigned gbase[256];        // global start of this block's run of each digit
    __shared__ unsigned wsum[8];
    __shared__ unsigned s_nvalid;
    __shared__ unsigned sk[kSortItems], sv[kSortItems];
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int n = item_count(n_bound, n_dev);
    const int base = blockIdx.x * kSortItems + warp * kWarpItems + lane;
    unsigned k[kSortRounds], v[kSortRounds], dg[kSortRounds];
#pragma unroll
    for (int r = 0; r < kSortRounds; ++r) {
        const int idx = base + r * 32;
        const bool valid = item_valid(idx, n, radius);
        k[r] = valid ? keys_in[idx] : 0u;
        v[r] = IOTA ? (unsigned)idx : (valid ? vals_in[idx] : 0u);
        dg[r] = valid ? (k[r] >> shift) & mask : 0x100u;
    }
#pragma unroll
    for (int i = 0; i < 8; ++i) woff[warp][lane + 32 * i] = 0u;
    __syncwarp();
#pragma unroll
    for (int r = 0; r < kSortRounds; ++r) {
        const unsigned d = dg[r];
        const unsigned peers = __match_any_sync(0xffffffffu, d);
        if (d != 0x100u && (peers & lanemask_lt()) == 0u) woff[warp][d] += __popc(peers);
        __syncwarp();
    }
    __syncthreads();
    {
        // digit d = thread: block count, exclusive scans over warps and over digits
        const int d = threadIdx.x;
        unsigned c = 0;
#pragma unroll
        for (int w = 0; w < 8; ++w) {
            const unsigned t = woff[w][d];
            woff[w][d] = c;
            c += t;
        }
        unsigned x = c;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const unsigned y = __shfl_up_sync(0xffffffffu, x, o);
            if (lane >= o) x += y;
        }
        if (lane == 31) wsum[warp] = x;
        // global digit start: exclusive scan of the digit totals
        const unsigned tv = totals[d];
        unsigned tx = tv;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const unsigned y = __shfl_up_sync(0xffffffffu, tx, o);
            if (lane >= o) tx += y;
        }
        __syncthreads();
        unsigned pre = 0;
        for (int w = 0; w < warp; ++w) pre += wsum[w];
        const unsigned lb = pre + x - c;
        lbase[d] = lb;
        if (d == 255) s_nvalid = lb + c;
#pragma unroll
        for (int w = 0; w < 8; ++w) woff[w][d] += lb;
        __syncthreads();
        if (lane == 31) wsum[warp] = tx;
        __syncthreads();
        unsigned tpre = 0;
        for (int w = 0; w < warp; ++w) tpre += wsum[w];
        gbase[d] = tpre + tx - tv + hist[(size_t)d * nblocks + blockIdx.x];
    }
    __syncthreads();
#pragma unroll
    for (int r = 0; r < kSortRounds; ++r) {
        const unsigned d = dg[r];
        const bool valid = d != 0x100u;
        const unsigned peers = __match_any_sync(0xffffffffu, d);
        if (valid) {
            const unsigned lp = woff[warp][d] + __popc(peers & lanemask_lt());
            sk[lp] = k[r];
            sv[lp] = v[r];
        }
        __syncwarp();
        if (valid && (peers & lanemask_lt()) == 0u) woff[warp][d] += __popc(peers);
        __syncwarp();
    }
    __syncthreads();
    const int n_block = (int)s_nvalid;
    for (int i = threadIdx.x; i < n_block; i += kSortThreads) {
        const unsigned key = sk[i], val = sv[i];
        const unsigned d = (key >> shift) & mask;
        const unsigned pos = gbase[d] + (unsigned)i - lbase[d];
        keys_out[pos] = key;
        vals_out[pos] = val;
        if (KEY64) keys64[pos] = ((unsigned long long)key << 32) | depth_bits[val];
    }
}

// ---- depth sort: one histogram pass, then one kernel per 8-bit digit (decoupled look-back) -----
//
// k_depth_hist4 counts the four 8-bit digits of the depth keys of all Gaussians with radius > 0
// in one pass. Each k_onesweep pass then counts the digits of its 4096-item block, publishes the
// counts, ranks the block's items into shared memory (as k_radix_scatter) and finds the number of
// items of each digit in all earlier blocks by looking back over their published words: a block's
// inclusive prefix ends the walk, an aggregate is added and the walk continues. Blocks take their
// index from a ticket in start order, so every block it waits for has started and publishes its
// aggregate before it waits itself; each wait is bounded (spin_limit polls that find the next word
// unpublished, then the timeout bit and a zero count).
constexpr unsigned long long kStatAgg = 1ull << 62, kStatIncl = 2ull << 62, kStatVal = (1ull << 62) - 1ull;
constexpr int kLookWindow = 8;  // earlier blocks' status words read per look-back round trip

__global__ void __launch_bounds__(256) k_depth_hist4(const unsigned* __restrict__ keys, int n,
                                                     const int* __restrict__ radius, unsigned* __restrict__ ghist) {
    pdl_entry();
    __shared__ unsigned h[4][256];
    const unsigned full = 0xffffffffu;
    const int lane = threadIdx.x & 31;
    for (int i = threadIdx.x; i < 4 * 256; i += blockDim.x) (&h[0][0])[i] = 0u;
    __syncthreads();
    const int stride = gridDim.x * blockDim.x;
    constexpr int kAhead = 4;  // rounds whose loads are issued together
    for (int base = blockIdx.x * blockDim.x + (threadIdx.x & ~31); base < n; base += kAhead * stride) {
        unsigned kk[kAhead];
        bool vv[kAhead];
#pragma unroll
        for (int a = 0; a < kAhead; ++a) {
            const int i = base + a * stride + lane;
            vv[a] = i < n && radius[i] > 0;
            kk[a] = i < n ? keys[i] : 0u;
        }
#pragma unroll
        for (int a = 0; a < kAhead; ++a) {
            // the two low digits of the depth bits are spread over the 256 buckets: one shared
            // atomic per lane rarely conflicts; the two high digits take few values (the depth
            // range), so equal digits are grouped first and each group adds once
#pragma unroll
            for (int p = 0; p < 2; ++p)
                if (vv[a]) atomicAdd(&h[p][(kk[a] >> (8 * p)) & 0xffu], 1u);
#pragma unroll
            for (int p = 2; p < 4; ++p) {
                const unsigned d = vv[a] ? (kk[a] >> (8 * p)) & 0xffu : 0x100u;
                const unsigned peers = __match_any_sync(full, d);
                if (vv[a] && (peers & lanemask_lt()) == 0u) atomicAdd(&h[p][d], (unsigned)__popc(peers));
            }
        }
    }
    __syncthreads();
    for (int i = threadIdx.x; i < 4 * 256; i += blockDim.x)
        if ((&h[0][0])[i]) atomicAdd(&ghist[i], (&h[0][0])[i]);
}

// One stable pass of the depth sort over the digit at `shift`. IOTA: the values are the item
// indices and items with radius 0 are dropped (first pass); later passes take the count of valid
// items from n_dev (the sum of the digit-0 histogram). The first pass is bounded to 85 registers
// (three resident blocks per SM); the later ones run over the visible Gaussians only (two blocks
// per SM hold 1.2M of them in one wave).
template <bool IOTA>
__global__ void __launch_bounds__(kSortThreads, IOTA ? 3 : 1) k_onesweep(
    const unsigned* __restrict__ keys_in, const unsigned* __restrict__ vals_in, unsigned* __restrict__ keys_out,
    unsigned* __restrict__ vals_out, int n_bound, const unsigned* __restrict__ ghist4, const int* __restrict__ radius,
    int pass, unsigned* __restrict__ ticket, unsigned long long* __restrict__ status, unsigned* __restrict__ nvis_out,
    unsigned spin_limit, unsigned* __restrict__ err) {
    if (IOTA) pdl_entry();  // the histograms were written by the kernel just before this pass
    __shared__ unsigned woff[8][256];      // per-warp digit counts, then block-local offsets
    __shared__ unsigned lbase[256];        // block-local start of each digit
    __shared__ unsigned gbase[256];        // global start of this block's run of each digit
    __shared__ unsigned wsum[8], wsum_g[8];
    __shared__ unsigned s_nvalid, s_block, s_n;
    __shared__ unsigned sk[kSortItems], sv[kSortItems];
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int shift = 8 * pass;
    const unsigned* ghist = ghist4 + 256 * pass;
    if (threadIdx.x == 0) {
        s_block = atomicAdd(ticket, 1u);
        s_n = 0u;
    }
    __syncthreads();
    if (!IOTA) {  // number of valid items: the total of the digit histogram
        const unsigned t = __reduce_add_sync(0xffffffffu, ghist4[threadIdx.x]);
        if (lane == 0) atomicAdd(&s_n, t);
        __syncthreads();
    }
    const unsigned tv = ghist[threadIdx.x];  // items of digit d = thread in the whole pass
    // Later passes read their ticket and the histograms before waiting: both were written two or
    // more kernels back (the memset, the histogram kernel), which have completed once any block of
    // this pass runs, because the pass before lets its dependents launch only after its own wait.
    // The keys of the pass before are read after waiting for it.
    if (!IOTA) pdl_entry();
    const int block = (int)s_block;
    if (!IOTA && nvis_out && block == 0 && threadIdx.x == 0) *nvis_out = s_n;
    const int n = IOTA ? n_bound : min(n_bound, (int)s_n);
    // blocks past the last item: no later block holds items, so none looks back this far
    if (block > 0 && block * kSortItems >= n) return;
    const int base = block * kSortItems + warp * kWarpItems + lane;
    unsigned k[kSortRounds], v[kSortRounds], dg[kSortRounds];
#pragma unroll
    for (int r = 0; r < kSortRounds; ++r) {
        const int idx = base + r * 32;
        const bool valid = item_valid(idx, n, IOTA ? radius : nullptr);
        k[r] = valid ? keys_in[idx] : 0u;
        v[r] = IOTA ? (unsigned)idx : (valid ? vals_in[idx] : 0u);
        dg[r] = valid ? (k[r] >> shift) & 0xffu : 0x100u;
    }
#pragma unroll
    for (int i = 0; i < 8; ++i) woff[warp][lane + 32 * i] = 0u;
    __syncwarp();
    // peer masks of the 8 rounds: all match_any first (independent), kept for the scatter below
    unsigned pm[kSortRounds];
#pragma unroll
    for (int r = 0; r < kSortRounds; ++r) pm[r] = __match_any_sync(0xffffffffu, dg[r]);
#pragma unroll
    for (int r = 0; r < kSortRounds; ++r) {  // group leaders of different rounds may share a digit
        const unsigned d = dg[r];
        if (d != 0x100u && (pm[r] & lanemask_lt()) == 0u) atomicAdd(&woff[warp][d], (unsigned)__popc(pm[r]));
    }
    __syncwarp();
    __syncthreads();
    // Digit d = thread. The block publishes its counts first, ranks its items into shared memory
    // (block-local order) and only then looks back, so that the items' registers are free during
    // the walk and other blocks find this block's aggregate as early as possible.
    const int d = threadIdx.x;
    unsigned c = 0;
#pragma unroll
    for (int w = 0; w < 8; ++w) {
        const unsigned t = woff[w][d];
        woff[w][d] = c;
        c += t;
    }
    unsigned long long* my = status + (size_t)block * 256 + d;
    *(volatile unsigned long long*)my = (block == 0 ? kStatIncl : kStatAgg) | c;
    unsigned tx = tv;  // inclusive scan of the pass histogram over the warp's digits
    {
        unsigned x = c;  // block-local inclusive scan over the warp's digits
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const unsigned y = __shfl_up_sync(0xffffffffu, x, o);
            const unsigned ty = __shfl_up_sync(0xffffffffu, tx, o);
            if (lane >= o) {
                x += y;
                tx += ty;
            }
        }
        if (lane == 31) {
            wsum[warp] = x;
            wsum_g[warp] = tx;
        }
        __syncthreads();
        unsigned pre = 0;
        for (int w = 0; w < warp; ++w) pre += wsum[w];
        const unsigned lb = pre + x - c;
        lbase[d] = lb;
        if (d == 255) s_nvalid = lb + c;
#pragma unroll
        for (int w = 0; w < 8; ++w) woff[w][d] += lb;
    }
    __syncthreads();
#pragma unroll
    for (int r = 0; r < kSortRounds; ++r) {
        const unsigned dr = dg[r];
        const bool valid = dr != 0x100u;
        const unsigned peers = pm[r];
        if (valid) {
            const unsigned lp = woff[warp][dr] + __popc(peers & lanemask_lt());
            sk[lp] = k[r];
            sv[lp] = v[r];
        }
        __syncwarp();
        if (valid && (peers & lanemask_lt()) == 0u) woff[warp][dr] += __popc(peers);
        __syncwarp();
    }
    // look back for the number of items of digit d in all earlier blocks: the walk reads
    // kLookWindow earlier blocks' words per round trip (their loads issued together, then read in
    // order); aggregates are added and passed, an inclusive count ends the walk, and a word not yet
    // published ends the window (the next window starts at that block)
    unsigned long long before = 0;
    if (block > 0) {
        int j = block - 1;
        unsigned polls = 0;
        bool found = false;
        while (!found) {
            unsigned long long sw[kLookWindow];
#pragma unroll
            for (int w = 0; w < kLookWindow; ++w)
                sw[w] = j - w >= 0 ? *(volatile const unsigned long long*)(status + (size_t)(j - w) * 256 + d) : 0ull;
            int passed = 0;
            bool stop = false;
#pragma unroll
            for (int w = 0; w < kLookWindow; ++w) {
                if (!stop) {
                    if (sw[w] & kStatIncl) {
                        before += sw[w] & kStatVal;
                        found = stop = true;
                    } else if (sw[w] & kStatAgg) {
                        before += sw[w] & kStatVal;
                        ++passed;
                    } else {
                        stop = true;
                    }
                }
            }
            j -= passed;
            if (found || j < 0) break;  // j < 0 not reached: block 0 publishes its inclusive count at once
            if (passed == 0 && ++polls >= spin_limit) {  // a poll that found the next word unpublished
                atomicOr(err, kErrTimeout);
                break;
            }
        }
        *(volatile unsigned long long*)my = kStatIncl | (before + c);
    }
    {
        unsigned tpre = 0;  // global digit start: exclusive scan of the pass histogram
        for (int w = 0; w < warp; ++w) tpre += wsum_g[w];
        gbase[d] = tpre + tx - tv + (unsigned)before;
    }
    __syncthreads();
    const int n_block = (int)s_nvalid;
    for (int i = threadIdx.x; i < n_block; i += kSortThreads) {
        const unsigned key = sk[i], val = sv[i];
        const unsigned d = (key >> shift) & 0xffu;
        const unsigned pos = gbase[d] + (unsigned)i - lbase[d];
        keys_out[pos] = key;
        vals_out[pos] = val;
    }
}

// Block sums (256 Gaussians per block, in depth order) of the number of tiles of each rectangle.
// With `crect`, also the packed rectangle of every depth-ordered Gaussian,
// crect[i] = (x0 | y0 << 16, w | h << 16), w = h = 0 when empty (tile ids below 2^16).
__global__ void __launch_bounds__(256) k_count(int n_bound, const unsigned* __restrict__ n_dev,
                                               const unsigned* __restrict__ perm, const float4* __restrict__ rec,
                                               const int* __restrict__ radius, int tiles_x, int tiles_y,
                                               unsigned long long* __restrict__ block_sums,
                                               uint2* __restrict__ crect,
                                               unsigned long long* __restrict__ super_sums) {
    pdl_entry();
    __shared__ unsigned long long ws[8], ws2[8];
    const int n = item_count(n_bound, n_dev);
    const int i = blockIdx.x * 256 + threadIdx.x;
    unsigned long long cnt = 0, cnt2 = 0;
    if (i < n) {
        const unsigned g = perm[i];
        // an index outside the Gaussians (only after a depth pass whose look-back gave up and set
        // the timeout bit) counts as culled, so that nothing is read out of range; the radius and
        // the record are loaded together (a culled Gaussian's record is zeros and goes unused)
        const bool in = g < (unsigned)n_bound;
        const int r = in ? radius[g] : 0;
        const float4 r0 = in ? rec[3 * (size_t)g] : make_float4(0.f, 0.f, 0.f, 0.f);
        uint2 packed = make_uint2(0u, 0u);
        if (r > 0) {
            const Rect R = tile_rect(r0.x, r0.y, r, tiles_x, tiles_y);
            if (R.x0 <= R.x1 && R.y0 <= R.y1) {
                cnt = (unsigned long long)(R.x1 - R.x0 + 1) * (unsigned long long)(R.y1 - R.y0 + 1);
                packed = make_uint2((unsigned)R.x0 | ((unsigned)R.y0 << 16),
                                    (unsigned)(R.x1 - R.x0 + 1) | ((unsigned)(R.y1 - R.y0 + 1) << 16));
            }
        }
        if (crect) crect[i] = packed;
        if (super_sums) {
            const uint2 sr = super_rect(packed);
            cnt2 = (unsigned long long)(sr.y & 0xffffu) * (sr.y >> 16);
        }
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
        cnt += __shfl_xor_sync(0xffffffffu, cnt, o);
        cnt2 += __shfl_xor_sync(0xffffffffu, cnt2, o);
    }
    if ((threadIdx.x & 31) == 0) {
        ws[threadIdx.x >> 5] = cnt;
        ws2[threadIdx.x >> 5] = cnt2;
    }
    __syncthreads();
    if (threadIdx.x == 0) {
        unsigned long long s = 0, s2 = 0;
        for (int w = 0; w < 8; ++w) {
            s += ws[w];
            s2 += ws2[w];
        }
        block_sums[blockIdx.x] = s;
        if (super_sums) super_sums[blockIdx.x] = s2;
    }
}

// Single-block exclusive scans: each of the 1024 threads takes kScanItems consecutive values per
// round, so that up to 8192 values need one round (one pass of block-wide synchronisation).
constexpr int kScanItems = 8;

// Block-wide exclusive scan of one value per thread (1024 threads); returns the thread's
// exclusive prefix and leaves the block total in *block_total (shared).
template <typename T>
__device__ __forceinline__ T block_scan_1024(T v, T* wsum, T* block_total) {
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    T x = v;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const T y = __shfl_up_sync(0xffffffffu, x, o);
        if (lane >= o) x += y;
    }
    if (lane == 31) wsum[warp] = x;
    __syncthreads();
    if (warp == 0) {
        T w = wsum[lane];
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const T y = __shfl_up_sync(0xffffffffu, w, o);
            if (lane >= o) w += y;
        }
        wsum[lane] = w;
        if (lane == 31) *block_total = w;
    }
    __syncthreads();
    return (warp ? wsum[warp - 1] : T(0)) + x - v;
}

// Exclusive scan of m block sums per block of 1024 threads; total[0] = sum of all (and
// *total_copy when given). Block 1, when launched, scans a second array (in2, out2, total2).
__global__ void __launch_bounds__(1024) k_scan_u64(const unsigned long long* __restrict__ in, int m,
                                                   unsigned long long* __restrict__ out,
                                                   unsigned long long* __restrict__ total,
                                                   unsigned long long* __restrict__ total_copy,
                                                   const unsigned long long* __restrict__ in2,
                                                   unsigned long long* __restrict__ out2,
                                                   unsigned long long* __restrict__ total2) {
    pdl_entry();
    if (blockIdx.x == 1) {
        in = in2;
        out = out2;
        total = total2;
        total_copy = nullptr;
    }
    __shared__ unsigned long long wsum[32];
    __shared__ unsigned long long round_total;
    unsigned long long carry = 0;
    for (int base = 0; base < m; base += 1024 * kScanItems) {
        const int i0 = base + threadIdx.x * kScanItems;
        unsigned long long v[kScanItems], sum = 0;
#pragma unroll
        for (int k = 0; k < kScanItems; ++k) {
            v[k] = i0 + k < m ? in[i0 + k] : 0ull;
            sum += v[k];
        }
        unsigned long long run = carry + block_scan_1024(sum, wsum, &round_total);
#pragma unroll
        for (int k = 0; k < kScanItems; ++k) {
            if (i0 + k < m) out[i0 + k] = run;
            run += v[k];
        }
        carry += round_total;
        __syncthreads();  // wsum and round_total are rewritten by the next round
    }
    if (threadIdx.x == 0) {
        total[0] = carry;
        if (total_copy) *total_copy = carry;
    }
}

// Emits the duplicates of 256 consecutive Gaussians (depth order) into their block's contiguous
// output range: output o goes to the Gaussian whose prefix range contains o (binary search over
// the block's 256 offsets), and is its (o - offset)-th tile in row-major rectangle order.
__global__ void __launch_bounds__(256) k_emit(int n_bound, const unsigned* __restrict__ n_dev,
                                              const unsigned* __restrict__ perm, const float4* __restrict__ rec,
                                              const int* __restrict__ radius, int tiles_x, int tiles_y,
                                              const unsigned long long* __restrict__ block_offs,
                                              unsigned long long capacity, unsigned* __restrict__ tile_out,
                                              unsigned* __restrict__ val_out, unsigned* __restrict__ err) {
    __shared__ unsigned s_off[257];
    __shared__ int s_x0[256], s_y0[256], s_w[256];
    __shared__ unsigned s_g[256];
    __shared__ unsigned wsum[8];
    const int n = item_count(n_bound, n_dev);
    const int i = blockIdx.x * 256 + threadIdx.x;
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    unsigned cnt = 0, g = 0;
    int x0 = 0, y0 = 0, w = 1;
    if (i < n) {
        g = perm[i];
        const bool in = g < (unsigned)n_bound;  // out of range only after a look-back timeout
        const int r = in ? radius[g] : 0;
        const float4 r0 = in ? rec[3 * (size_t)g] : make_float4(0.f, 0.f, 0.f, 0.f);  // loaded with the radius
        if (r > 0) {
            const Rect R = tile_rect(r0.x, r0.y, r, tiles_x, tiles_y);
            if (R.x0 <= R.x1) {
                x0 = R.x0; y0 = R.y0; w = R.x1 - R.x0 + 1;
                cnt = (unsigned)w * (unsigned)(R.y1 - R.y0 + 1);
            }
        }
    }
    s_x0[threadIdx.x] = x0; s_y0[threadIdx.x] = y0; s_w[threadIdx.x] = w; s_g[threadIdx.x] = g;
    unsigned x = cnt;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const unsigned y = __shfl_up_sync(0xffffffffu, x, o);
        if (lane >= o) x += y;
    }
    if (lane == 31) wsum[warp] = x;
    __syncthreads();
    unsigned pre = 0;
    for (int k = 0; k < warp; ++k) pre += wsum[k];
    s_off[threadIdx.x] = pre + x - cnt;
    if (threadIdx.x == 255) s_off[256] = pre + x;
    __syncthreads();
    const unsigned total = s_off[256];
    const unsigned long long base = block_offs[blockIdx.x];
    if (base + total > capacity) {
        if (threadIdx.x == 0) atomicOr(err, kErrCheck);
        return;
    }
    for (unsigned o = threadIdx.x; o < total; o += 256) {
        // largest j with s_off[j] <= o
        int lo = 0, hi = 256;
        while (hi - lo > 1) {
            const int mid = (lo + hi) >> 1;
            if (s_off[mid] <= o) lo = mid; else hi = mid;
        }
        const unsigned k = o - s_off[lo];
        const unsigned ww = (unsigned)s_w[lo];
        const unsigned row = k / ww;
        const unsigned tx = (unsigned)s_x0[lo] + (k - row * ww), ty = (unsigned)s_y0[lo] + row;
        tile_out[base + o] = ty * (unsigned)tiles_x + tx;
        val_out[base + o] = s_g[lo];
    }
}

// 64-bit keys of an already sorted list (used when the image is a single tile and no tile pass runs).
__global__ void k_make_keys(unsigned d, const unsigned* __restrict__ tiles, const unsigned* __restrict__ vals,
                            const unsigned* __restrict__ depth_bits, unsigned long long* __restrict__ keys64) {
    const unsigned i = blockIdx.x * blockDim.x + threadIdx.x;
    if (i < d) keys64[i] = ((unsigned long long)tiles[i] << 32) | depth_bits[vals[i]];
}

// [start, end) of every tile from the sorted tile ids (ranges zeroed beforehand); each thread
// looks at 4 consecutive entries.
__global__ void k_ranges(unsigned d, const unsigned* __restrict__ tiles, uint2* __restrict__ ranges) {
    const unsigned i0 = 4u * (blockIdx.x * blockDim.x + threadIdx.x);
    if (i0 >= d) return;
    unsigned prev = i0 > 0 ? tiles[i0 - 1] : 0xffffffffu;
    const unsigned iend = min(i0 + 4u, d);
    for (unsigned i = i0; i < iend; ++i) {
        const unsigned t = tiles[i];
        if (t != prev) {
            ranges[t].x = i;
            if (i > 0) ranges[prev].y = i;
        }
        prev = t;
    }
    if (iend == d) ranges[prev].y = d;
}

// ---- tile pass as one stable counting pass (images of up to kMaxCountTiles tiles) -------------
//
// The tile pass is the stable counting sort of the depth-ordered duplicates by tile id (an LSD
// radix pass whose digit is the whole tile id): equal tile ids keep depth order. It runs in two
// levels. The coarse level sorts by super-tile (kSuper x kSuper tiles): the depth-ordered Gaussians
// are cut into chunks; for every chunk a shared-memory histogram counts the Gaussians whose
// rectangle of super-tiles covers each super-tile; a scan down each super-tile's column of the
// chunk x super-tile table gives the chunk's first position inside every super-tile's list; each
// chunk then places the depth positions of its Gaussians in depth order (k_chunk_place). The fine
// level (below) sorts each super-tile's list by tile. At the coarse level a Gaussian has few
// entries (the outdoor scene: 2.1M against 11.6M duplicates; the large scene: 16.6M against
// 179M), so the scattered placement writes few entries; the fine level writes each tile's entries
// as coalesced runs.
//
// Depth order puts the Gaussians nearest to the camera, which are the largest on screen, first. A
// chunk therefore ends after kChunk Gaussians or about kChunkDup coarse entries, whichever comes
// first: Gaussian i (depth order, P(i) entries before it) belongs to chunk
// floor(i / kChunk) + floor(P(i) / kChunkDup), which never decreases with i (ids that are skipped
// are empty chunks). Within a chunk, rectangles are spread over lanes.
constexpr int kChunk = 256;            // Gaussians per chunk at most
constexpr long long kChunkDup = 8192;  // coarse entries after which a chunk ends early
constexpr int kMaxCountTiles = 49152;   // tile counters that fit in shared memory (192 KB)
constexpr int kSmallRect = 8;           // rectangles of up to this many tiles: one lane each

// k / w for 0 <= k, w < 2^16 as a multiply-high: with m = floor((2^32 - 1) / w) + 1 (w >= 2) the
// product k m / 2^32 exceeds k / w by less than k / 2^32 < 1 / w, so its floor is exact.
__device__ __forceinline__ unsigned div_magic(unsigned w) { return w > 1u ? 0xffffffffu / w + 1u : 0u; }
__device__ __forceinline__ unsigned div_by(unsigned k, unsigned w, unsigned m) { return w > 1u ? __umulhi(k, m) : k; }

// Upper bound of the chunk ids for n Gaussians and at most `cap` entries (ids are clamped to it,
// which only matters when the entries exceed `cap`, a capacity error).
static long long max_chunks(long long n, long long cap) { return (n + kChunk - 1) / kChunk + cap / kChunkDup + 1; }

__device__ __forceinline__ int chunk_of(int i, unsigned long long before, int cmax) {
    const unsigned long long c = (unsigned long long)(i / kChunk) + before / (unsigned long long)kChunkDup;
    return (int)min(c, (unsigned long long)(cmax - 1));
}

// First Gaussian of every chunk (chunk_first[c] for c < nchunks, chunk_first[nchunks] = V) and the
// number of chunks used. block_offs: entries before each 256-Gaussian block (k_count, k_scan_u64).
__global__ void __launch_bounds__(256) k_chunk_bounds(int n_bound, const unsigned* __restrict__ n_dev,
                                                      const uint2* __restrict__ crect,
                                                      const unsigned long long* __restrict__ block_offs, int cmax,
                                                      unsigned* __restrict__ chunk_first,
                                                      unsigned* __restrict__ nchunks) {
    pdl_entry();
    __shared__ unsigned long long wsum[8];
    __shared__ int s_c[256];
    const int n = item_count(n_bound, n_dev);
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const int i = blockIdx.x * 256 + threadIdx.x;
    unsigned long long area = 0;
    if (i < n) {
        const uint2 r = super_rect(crect[i]);
        area = (unsigned long long)(r.y & 0xffffu) * (r.y >> 16);
    }
    unsigned long long x = area;  // inclusive scan over the block
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const unsigned long long y = __shfl_up_sync(0xffffffffu, x, o);
        if (lane >= o) x += y;
    }
    if (lane == 31) wsum[warp] = x;
    __syncthreads();
    unsigned long long wpre = 0;
    for (int w = 0; w < warp; ++w) wpre += wsum[w];
    const unsigned long long before = block_offs[blockIdx.x] + wpre + x - area;
    const int c = chunk_of(i, before, cmax);
    s_c[threadIdx.x] = c;
    __syncthreads();
    if (i >= n) return;
    int cprev = -1;
    if (threadIdx.x > 0) {
        cprev = s_c[threadIdx.x - 1];
    } else if (i > 0) {
        const uint2 r = super_rect(crect[i - 1]);
        cprev = chunk_of(i - 1, before - (unsigned long long)(r.y & 0xffffu) * (r.y >> 16), cmax);
    }
    for (int k = cprev + 1; k <= c; ++k) chunk_first[k] = (unsigned)i;
    if (i == n - 1) {
        chunk_first[c + 1] = (unsigned)n;
        *nchunks = (unsigned)(c + 1);
    }
}

// Counts per super-tile of one chunk (one block per chunk id; ids at or beyond the count return).
__global__ void __launch_bounds__(256) k_chunk_hist(const unsigned* __restrict__ nchunks,
                                                    const unsigned* __restrict__ chunk_first,
                                                    const uint2* __restrict__ crect, int tiles_x, int T,
                                                    unsigned* __restrict__ table) {
    pdl_entry();
    extern __shared__ unsigned cnt[];
    const unsigned full = 0xffffffffu;
    const int c = blockIdx.x;
    if (c >= (int)*nchunks) return;
    const int first = (int)chunk_first[c], last = (int)chunk_first[c + 1];
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    for (int t = threadIdx.x; t < T / 4; t += blockDim.x) reinterpret_cast<uint4*>(cnt)[t] = make_uint4(0u, 0u, 0u, 0u);
    for (int t = (T & ~3) + threadIdx.x; t < T; t += blockDim.x) cnt[t] = 0u;
    __syncthreads();
    for (int base = first + 32 * warp; base < last; base += (int)blockDim.x) {  // warp-uniform
        const int i = base + lane;
        int x0 = 0, y0 = 0, w = 0, h = 0, area = 0;
        if (i < last) {
            const uint2 r = super_rect(crect[i]);
            x0 = (int)(r.x & 0xffffu);
            y0 = (int)(r.x >> 16);
            w = (int)(r.y & 0xffffu);
            h = (int)(r.y >> 16);
            area = w * h;
        }
        if (area <= kSmallRect) {
            for (int y = 0; y < h; ++y)
                for (int x = 0; x < w; ++x) atomicAdd(&cnt[(y0 + y) * tiles_x + x0 + x], 1u);
        }
        const unsigned m = div_magic((unsigned)w);
        unsigned big = __ballot_sync(full, area > kSmallRect);
        while (big) {  // large rectangles: all lanes of the warp
            const int j = __ffs(big) - 1;
            big &= big - 1u;
            const unsigned jw = (unsigned)__shfl_sync(full, w, j), jm = __shfl_sync(full, m, j);
            const unsigned ja = (unsigned)__shfl_sync(full, area, j);
            const unsigned t0 = (unsigned)(__shfl_sync(full, y0, j) * tiles_x + __shfl_sync(full, x0, j));
            for (unsigned k = lane; k < ja; k += 32u) {
                const unsigned rk = div_by(k, jw, jm);
                atomicAdd(&cnt[t0 + rk * (unsigned)tiles_x + (k - rk * jw)], 1u);
            }
        }
    }
    __syncthreads();
    unsigned* row = table + (size_t)c * T;
    for (int t = threadIdx.x; t < T; t += blockDim.x) row[t] = cnt[t];
}

// Exclusive scan down each super-tile's column of the chunk x super-tile table (in place) and the
// column totals, in groups of kScanGroup chunk rows so that tables with many rows and few columns
// still spread over many blocks: k_chunk_colsum sums each group's rows per column, and
// k_chunk_scan scans each group's rows starting from the sum of the groups before it.
// Blocks: 32 columns (one per lane) x 32 warps, each warp a contiguous range of the group's rows;
// blockIdx.y is the group (groups past the used rows return).
constexpr int kScanWarps = 32;
constexpr int kColUnroll = 16;   // table loads in flight per lane
constexpr int kScanGroup = 512;  // chunk rows per group

__global__ void __launch_bounds__(32 * kScanWarps) k_chunk_colsum(const unsigned* __restrict__ nchunks, int T,
                                                                  const unsigned* __restrict__ table,
                                                                  unsigned* __restrict__ group_sum) {
    pdl_entry();
    __shared__ unsigned part[kScanWarps][32];
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const int t = blockIdx.x * 32 + lane;
    const int nc = (int)*nchunks, g0 = blockIdx.y * kScanGroup;
    if (g0 >= nc) return;
    const int g1 = min(nc, g0 + kScanGroup);
    const int per = (g1 - g0 + kScanWarps - 1) / kScanWarps;
    const int c0 = min(g1, g0 + warp * per), c1 = min(g1, c0 + per);
    unsigned sum = 0;
    if (t < T) {
        int c = c0;
        for (; c + kColUnroll <= c1; c += kColUnroll) {
            unsigned v[kColUnroll];
#pragma unroll
            for (int k = 0; k < kColUnroll; ++k) v[k] = table[(size_t)(c + k) * T + t];
#pragma unroll
            for (int k = 0; k < kColUnroll; ++k) sum += v[k];
        }
        for (; c < c1; ++c) sum += table[(size_t)c * T + t];
    }
    part[warp][lane] = sum;
    __syncthreads();
    if (warp == 0 && t < T) {
        unsigned total = 0;
        for (int w = 0; w < kScanWarps; ++w) total += part[w][lane];
        group_sum[(size_t)blockIdx.y * T + t] = total;
    }
}

__global__ void __launch_bounds__(32 * kScanWarps) k_chunk_scan(const unsigned* __restrict__ nchunks, int T,
                                                                unsigned* __restrict__ table,
                                                                const unsigned* __restrict__ group_sum,
                                                                unsigned* __restrict__ tile_total) {
    pdl_entry();
    __shared__ unsigned part[kScanWarps][32];
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const int t = blockIdx.x * 32 + lane;
    const int nc = (int)*nchunks, g0 = blockIdx.y * kScanGroup;
    const bool last = g0 + kScanGroup >= nc;  // the group that writes the column totals
    if (g0 >= nc && blockIdx.y != 0) return;  // group 0 runs even without rows: zero totals
    const int g1 = min(nc, g0 + kScanGroup);
    const int per = (max(g1 - g0, 0) + kScanWarps - 1) / kScanWarps;
    const int c0 = min(g1, g0 + warp * per), c1 = min(g1, c0 + per);
    unsigned carry = 0;  // the groups before this one
    if (t < T)
        for (int g = 0; g < (int)blockIdx.y; ++g) carry += group_sum[(size_t)g * T + t];
    unsigned sum = 0;
    if (t < T) {
        int c = c0;
        for (; c + kColUnroll <= c1; c += kColUnroll) {
            unsigned v[kColUnroll];
#pragma unroll
            for (int k = 0; k < kColUnroll; ++k) v[k] = table[(size_t)(c + k) * T + t];
#pragma unroll
            for (int k = 0; k < kColUnroll; ++k) sum += v[k];
        }
        for (; c < c1; ++c) sum += table[(size_t)c * T + t];
    }
    part[warp][lane] = sum;
    __syncthreads();
    unsigned run = carry;
    for (int w = 0; w < warp; ++w) run += part[w][lane];
    if (t < T) {
        int c = c0;
        for (; c + kColUnroll <= c1; c += kColUnroll) {
            unsigned v[kColUnroll];
#pragma unroll
            for (int k = 0; k < kColUnroll; ++k) v[k] = table[(size_t)(c + k) * T + t];
#pragma unroll
            for (int k = 0; k < kColUnroll; ++k) {
                table[(size_t)(c + k) * T + t] = run;
                run += v[k];
            }
        }
        for (; c < c1; ++c) {
            unsigned* e = &table[(size_t)c * T + t];
            const unsigned v = *e;
            *e = run;
            run += v;
        }
        if (last && warp == kScanWarps - 1) tile_total[t] = run;
    }
}

// Exclusive scan of the tile totals (one block): tile_start[t], total[0] = D (also written to
// total_copy when given), and the tile ranges [start, start + count). When D exceeds the capacity every range is written empty, so
// that no later kernel reads past the caller's list; with `err` (the call that does not read D on
// the host) the check bit is also set.
//
// With seg_first (the coarse level: the "tiles" are super-tiles), it also numbers the fine level's
// segments: super-tile s gets ceil(count / kSeg) of them (none when over the capacity), numbered
// from seg_first[s]; seg_first[T] and *nseg = their number (nseg clamped to seg_cap).
__global__ void __launch_bounds__(1024) k_tile_scan(int T, const unsigned* __restrict__ tile_total,
                                                    unsigned* __restrict__ tile_start,
                                                    unsigned long long* __restrict__ total,
                                                    unsigned long long capacity, uint2* __restrict__ ranges,
                                                    unsigned* __restrict__ err,
                                                    unsigned long long* __restrict__ total_copy,
                                                    unsigned* __restrict__ seg_first, unsigned* __restrict__ nseg,
                                                    unsigned seg_cap) {
    pdl_entry();
    __shared__ unsigned long long wsum[32];
    __shared__ unsigned long long round_total;
    unsigned long long carry = 0;
    for (int base = 0; base < T; base += 1024 * kScanItems) {
        const int t0 = base + threadIdx.x * kScanItems;
        unsigned v[kScanItems];
        unsigned long long sum = 0;
#pragma unroll
        for (int k = 0; k < kScanItems; ++k) {
            v[k] = t0 + k < T ? tile_total[t0 + k] : 0u;
            sum += v[k];
        }
        unsigned long long run = carry + block_scan_1024(sum, wsum, &round_total);
#pragma unroll
        for (int k = 0; k < kScanItems; ++k) {
            if (t0 + k < T) tile_start[t0 + k] = (unsigned)run;
            run += v[k];
        }
        carry += round_total;
        __syncthreads();
    }
    if (threadIdx.x == 0) {
        total[0] = carry;
        if (total_copy) *total_copy = carry;
    }
    const bool over = carry > capacity;
    if (over && err && threadIdx.x == 0) atomicOr(err, kErrCheck);
    for (int t = threadIdx.x; t < T; t += blockDim.x) {  // the last round's barrier made every start visible
        const unsigned c = tile_total[t];
        ranges[t] = (!over && c) ? make_uint2(tile_start[t], tile_start[t] + c) : make_uint2(0u, 0u);
    }
    if (!seg_first) return;
    __shared__ unsigned swsum[32];
    __shared__ unsigned sround_total;
    unsigned scarry = 0;
    for (int base = 0; base < T; base += 1024 * kScanItems) {
        const int t0 = base + threadIdx.x * kScanItems;
        unsigned v[kScanItems], sum = 0;
#pragma unroll
        for (int k = 0; k < kScanItems; ++k) {
            v[k] = (!over && t0 + k < T) ? (tile_total[t0 + k] + kSeg - 1) / kSeg : 0u;
            sum += v[k];
        }
        unsigned run = scarry + block_scan_1024(sum, swsum, &sround_total);
#pragma unroll
        for (int k = 0; k < kScanItems; ++k) {
            if (t0 + k < T) seg_first[t0 + k] = run;
            run += v[k];
        }
        scarry += sround_total;
        __syncthreads();
    }
    if (threadIdx.x == 0) {
        seg_first[T] = scarry;
        *nseg = min(scarry, seg_cap);
    }
}

// Coarse placement: one warp per (chunk, band of super-tile rows). The warp copies the chunk's
// starting offset inside each of the band's super-tiles into shared memory, then walks the chunk's
// Gaussians in depth order; for each one whose rectangle of super-tiles meets the band, its lanes
// cover the rectangle's super-tiles inside the band (distinct super-tiles, so no two lanes share an
// offset) and append the Gaussian's depth position there (the fine level reads its tile rectangle
// from it). Entries therefore land in depth order within every super-tile; bands own disjoint
// super-tiles. Two consecutive Gaussians whose rectangles in the band are disjoint and small (at
// most 16 super-tiles each) are placed in the same step, one per half-warp: they share no
// super-tile, so their order does not matter. Chunks end after about kChunkDup entries, so a warp
// never walks more than a bounded amount of work. tiles_x, tiles_y count super-tiles here.
constexpr int kPlaceWarps = 8;        // warps per block when shared memory allows
constexpr int kPlaceBands = 2;        // bands per chunk (whole super-tile rows)

// The placement loop of k_chunk_place; CHECK: positions may reach the capacity (D' above it).
template <bool CHECK>
__device__ __forceinline__ void chunk_place_loop(int first, int last, int r0, int r1, int tiles_x, unsigned* off,
                                                 const uint2* __restrict__ crect, unsigned capacity,
                                                 unsigned* __restrict__ vals, unsigned* __restrict__ err, int lane);

__global__ void __launch_bounds__(32 * kPlaceWarps) k_chunk_place(
    const unsigned* __restrict__ nchunks, const unsigned* __restrict__ chunk_first, const uint2* __restrict__ crect,
    int tiles_x, int tiles_y, int band_rows, int nbands, const unsigned* __restrict__ table,
    const unsigned* __restrict__ tile_start, const unsigned long long* __restrict__ ctotal, unsigned capacity,
    unsigned* __restrict__ vals, unsigned* __restrict__ err) {
    pdl_entry();
    extern __shared__ unsigned smem_off[];
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const long long gw = (long long)blockIdx.x * (blockDim.x >> 5) + warp;
    const int chunk = (int)(gw / nbands), band = (int)(gw - (long long)chunk * nbands);
    if (chunk >= (int)*nchunks) return;
    const int first = (int)chunk_first[chunk], last = (int)chunk_first[chunk + 1];
    if (first >= last) return;
    const int T = tiles_x * tiles_y;  // super-tiles
    const int r0 = band * band_rows, r1 = min(r0 + band_rows, tiles_y);
    if (r0 >= r1) return;
    const int tb0 = r0 * tiles_x, ntb = (r1 - r0) * tiles_x;
    unsigned* off = smem_off + (size_t)warp * band_rows * tiles_x;
    const unsigned* row = table + (size_t)chunk * T + tb0;
    const unsigned* ts = tile_start + tb0;
    for (int t = lane; t < ntb; t += 32) off[t] = ts[t] + row[t];
    __syncwarp();
    // D' (the coarse tile scan's total) within the capacity: no position reaches it
    if (*ctotal <= (unsigned long long)capacity)
        chunk_place_loop<false>(first, last, r0, r1, tiles_x, off, crect, capacity, vals, err, lane);
    else
        chunk_place_loop<true>(first, last, r0, r1, tiles_x, off, crect, capacity, vals, err, lane);
}

template <bool CHECK>
__device__ __forceinline__ void chunk_place_loop(int first, int last, int r0, int r1, int tiles_x, unsigned* off,
                                                 const uint2* __restrict__ crect, unsigned capacity,
                                                 unsigned* __restrict__ vals, unsigned* __restrict__ err, int lane) {
    const unsigned full = 0xffffffffu;
    uint2 r_next = make_uint2(0u, 0u);
    if (first + lane < last) r_next = super_rect(crect[first + lane]);
    for (int base = first; base < last; base += 32) {
        const uint2 pr = r_next;  // this lane's Gaussian: depth position base + lane
        const int nx = base + 32 + lane;  // prefetch the next 32 Gaussians
        r_next = make_uint2(0u, 0u);
        if (nx < last) r_next = super_rect(crect[nx]);
        // this lane's Gaussian inside the band: columns [x0, x0 + w), rows [ya, yb) (band-local)
        const unsigned w = pr.y & 0xffffu;
        const int y0 = (int)(pr.x >> 16);
        const int ya = max(y0, r0) - r0, yb = min(y0 + (int)(pr.y >> 16), r1) - r0;
        const unsigned xw = (pr.x & 0xffffu) | (w << 16);
        const unsigned yab = (unsigned)ya | ((unsigned)max(yb, 0) << 16);
        const unsigned m = div_magic(w);
        const unsigned area_l = (w > 0u && ya < yb) ? w * (unsigned)(yb - ya) : 0u;
        const unsigned tl0_l = (unsigned)ya * (unsigned)tiles_x + (pr.x & 0xffffu);  // band-local first tile
        const unsigned wa = w | (area_l << 16);  // width and area (both below 2^16 super-tiles)
        unsigned hit = __ballot_sync(full, area_l > 0u);
        // pairing, decided for all lanes at once: a hit lane pairs with the next hit lane when both
        // cover at most 16 tiles of the band and their rectangles are disjoint; then each half-warp
        // places one of them (they share no tile, so their order does not matter)
        const unsigned above = hit & ~((2u << lane) - 1u);
        const int nxt = above ? __ffs(above) - 1 : lane;
        const unsigned xw_n = __shfl_sync(full, xw, nxt), yab_n = __shfl_sync(full, yab, nxt);
        const unsigned area_n = __shfl_sync(full, area_l, nxt);
        const unsigned x1 = xw & 0xffffu, x2 = xw_n & 0xffffu;
        const bool apart = x1 + (xw >> 16) <= x2 || x2 + (xw_n >> 16) <= x1 || (yab >> 16) <= (yab_n & 0xffffu) ||
                           (yab_n >> 16) <= (yab & 0xffffu);
        const unsigned pairable = __ballot_sync(full, area_l > 0u && above != 0u && area_l <= 16u && area_n <= 16u && apart);
        while (hit) {
            const int j1 = __ffs(hit) - 1;
            hit &= hit - 1u;
            const bool pair = (pairable >> j1) & 1u;  // warp-uniform
            const int j2 = pair ? __ffs(hit) - 1 : j1;
            if (pair) hit &= hit - 1u;
            const bool second = pair && lane >= 16;
            const int j = second ? j2 : j1;
            const unsigned jg = (unsigned)(base + j);  // lane j's Gaussian
            const unsigned jm = __shfl_sync(full, m, j), jwa = __shfl_sync(full, wa, j);
            const unsigned tl0 = __shfl_sync(full, tl0_l, j);
            const unsigned jw = jwa & 0xffffu, area = jwa >> 16;
            const unsigned step = pair ? 16u : 32u;
            for (unsigned k = pair ? (lane & 15u) : lane; k < area; k += step) {
                const unsigned rk = div_by(k, jw, jm);
                const unsigned tl = tl0 + rk * (unsigned)tiles_x + (k - rk * jw);  // band-local tile
                const unsigned pos = off[tl];
                off[tl] = pos + 1u;
                if (!CHECK || pos < capacity) {
                    vals[pos] = jg;
                } else {
                    atomicOr(err, kErrCheck);
                }
            }
            __syncwarp();
        }
    }
}

// ---- fine level of the two-level counting pass -------------------------------------------------
//
// The coarse level (the chunk kernels above run on super-tiles) places, for every super-tile, the
// depth positions of the Gaussians whose rectangle meets it, in depth order. The fine level splits
// each super-tile's list into segments of kSeg entries. Per segment it counts, for each of the
// super-tile's kSuper x kSuper tiles, the entries whose tile rectangle covers the tile; a scan down
// each super-tile's segments gives every segment's first position inside each tile's list; each
// segment then places its entries round by round (32 entries, one per lane): per covered tile the
// lanes whose Gaussian covers it write consecutive positions of the tile's list, one coalesced
// run. Segments, rounds and lanes follow the coarse list, so each tile's entries stay in depth
// order: the result is the same stable counting pass by tile id.
constexpr int kSuperTiles = kSuper * kSuper;   // tiles per super-tile
static_assert(kSuper == 4, "cover_mask packs a super-tile's tiles as 4 bits per row");

// Bit 4 ly + lx set when the packed tile rectangle r covers tile (tx0 + lx, ty0 + ly).
__device__ __forceinline__ unsigned cover_mask(uint2 r, int tx0, int ty0) {
    const int w = (int)(r.y & 0xffffu), h = (int)(r.y >> 16);
    const int x0 = (int)(r.x & 0xffffu) - tx0, y0 = (int)(r.x >> 16) - ty0;
    const int ax0 = max(x0, 0), ax1 = min(x0 + w, kSuper), ay0 = max(y0, 0), ay1 = min(y0 + h, kSuper);
    if (ax0 >= ax1 || ay0 >= ay1) return 0u;
    const unsigned row = ((1u << ax1) - 1u) & ~((1u << ax0) - 1u);
    const unsigned col = 0x1111u & ((1u << (4 * ay1)) - 1u) & ~((1u << (4 * ay0)) - 1u);
    return row * col;  // the row pattern repeated in every covered row's nibble
}

// The super-tile of segment k: the last s with first[s] <= k (first[] in shared memory).
__device__ __forceinline__ int segment_tile(const unsigned* first, int Ts, unsigned k) {
    int lo = 0, hi = Ts;  // first[lo] <= k < first[hi]
    while (hi - lo > 1) {
        const int mid = (lo + hi) >> 1;
        if (first[mid] <= k) lo = mid; else hi = mid;
    }
    return lo;
}

// Per segment (one warp, grid-stride over the segments): F[k][t] = the number of segment k's
// entries whose tile rectangle covers tile t of its super-tile. Dynamic shared memory holds
// seg_first[0..Ts].
__global__ void __launch_bounds__(256) k_fine_count(int Ts, int SX, unsigned n_bound,
                                                    const unsigned* __restrict__ seg_first,
                                                    const unsigned* __restrict__ nseg,
                                                    const uint2* __restrict__ crange,
                                                    const unsigned* __restrict__ cvals,
                                                    const uint2* __restrict__ crect, unsigned* __restrict__ F) {
    pdl_entry();
    extern __shared__ unsigned s_first[];
    for (int t = threadIdx.x; t <= Ts; t += blockDim.x) s_first[t] = seg_first[t];
    __syncthreads();
    const int lane = threadIdx.x & 31;
    const unsigned ns = *nseg, wpb = blockDim.x >> 5;
    for (unsigned k = blockIdx.x * wpb + (threadIdx.x >> 5); k < ns; k += gridDim.x * wpb) {
        const int st = segment_tile(s_first, Ts, k);
        const uint2 rg = crange[st];
        const unsigned p0 = rg.x + (k - s_first[st]) * kSeg, p1 = min(p0 + kSeg, rg.y);
        const int tx0 = (st % SX) * kSuper, ty0 = (st / SX) * kSuper;
        // all of the segment's entries are loaded first (kRounds independent loads per lane, then
        // their rectangles), so the latencies overlap instead of adding up round by round
        unsigned m16[kRounds];
        {
            unsigned iv[kRounds];
#pragma unroll
            for (int r = 0; r < kRounds; ++r) iv[r] = p0 + 32 * r + lane < p1 ? cvals[p0 + 32 * r + lane] : ~0u;
#pragma unroll
            for (int r = 0; r < kRounds; ++r)  // a depth position below V <= n
                m16[r] = iv[r] < n_bound ? cover_mask(crect[iv[r]], tx0, ty0) : 0u;
        }
        // Per-tile counts of the warp's masks, four tiles per 32-bit word: the nibble of tiles
        // 4j..4j+3 is spread into the four bytes of a word (x * 0x204081 places bits 0..3 of x at
        // bits 0, 8, 16, 24 with nothing overlapping them), and one warp add-reduction of each word
        // sums 32 lanes per byte (at most 32). The sums of the rounds are kept in 16-bit fields
        // (at most 8 x 32 = 256): acc[2j] holds tiles 4j and 4j + 2, acc[2j + 1] tiles 4j + 1, 4j + 3.
        unsigned acc[8] = {0u, 0u, 0u, 0u, 0u, 0u, 0u, 0u};
#pragma unroll
        for (int r = 0; r < kRounds; ++r) {
#pragma unroll
            for (int j = 0; j < 4; ++j) {
                const unsigned spread = (((m16[r] >> (4 * j)) & 0xfu) * 0x00204081u) & 0x01010101u;
                const unsigned sum = __reduce_add_sync(0xffffffffu, spread);
                acc[2 * j] += sum & 0x00ff00ffu;
                acc[2 * j + 1] += (sum >> 8) & 0x00ff00ffu;
            }
        }
        if (lane < kSuperTiles) {
            // tile t = 4j + b: word 2j + (b & 1), field b >> 1 (selected without indexing registers)
            const int j = lane >> 2, b = lane & 3;
            unsigned w = 0;
#pragma unroll
            for (int q = 0; q < 8; ++q) w = (q == 2 * j + (b & 1)) ? acc[q] : w;
            F[(size_t)k * kSuperTiles + lane] = (w >> (16 * (b >> 1))) & 0xffffu;
        }
    }
}

// Per super-tile (one warp, grid-stride): for each of its tiles t (lanes t and t + 16 take the first
// and second half of the segments), the exclusive scan of F[k][t] down the super-tile's segments
// (in place) and the tile's total tile_total[tile] (every tile of the image is written).
__global__ void __launch_bounds__(256) k_fine_scan(int Ts, int SX, int tiles_x, int tiles_y,
                                                   const unsigned* __restrict__ seg_first, unsigned seg_cap,
                                                   unsigned* __restrict__ F, unsigned* __restrict__ tile_total) {
    pdl_entry();
    const int lane = threadIdx.x & 31, t = lane & (kSuperTiles - 1), half = lane >> 4;
    const unsigned wpb = blockDim.x >> 5;
    for (unsigned st = blockIdx.x * wpb + (threadIdx.x >> 5); st < (unsigned)Ts; st += gridDim.x * wpb) {
        const unsigned k0 = min(seg_first[st], seg_cap), k1 = min(seg_first[st + 1], seg_cap);
        const unsigned mid = k0 + (k1 - k0 + 1u) / 2u;
        const unsigned a = half ? mid : k0, b = half ? k1 : mid;
        unsigned sum = 0;
#pragma unroll 4
        for (unsigned k = a; k < b; ++k) sum += F[(size_t)k * kSuperTiles + t];
        const unsigned first_half = __shfl_sync(0xffffffffu, sum, t);
        unsigned run = half ? first_half : 0u;
        for (unsigned k = a; k < b; ++k) {
            unsigned* e = &F[(size_t)k * kSuperTiles + t];
            const unsigned v = *e;
            *e = run;
            run += v;
        }
        const int tx = (int)(st % SX) * kSuper + (t & 3), ty = (int)(st / SX) * kSuper + (t >> 2);
        if (half && tx < tiles_x && ty < tiles_y) tile_total[ty * tiles_x + tx] = run;
    }
}

// Per segment (one warp, grid-stride): places the segment's entries. Every lane keeps the next
// position of each of the 16 tiles (the same values in all lanes); per round and per tile that some
// lane's Gaussian covers, those lanes write consecutive positions (their rank among the covering
// lanes) and the tile's position advances. The tile loop is unrolled so that the 16 positions stay
// in registers and the tiles' updates are independent of one another. The loads of a warp's next
// segment (its entries, its tiles' first positions) are issued before the current segment is
// placed, so that their latency overlaps the placement.
struct FineSeg {
    unsigned iv[kRounds];   // the segment's entries (depth positions), ~0u past its end
    unsigned start;         // lane t < 16: first position of tile t for this segment
    int tx0, ty0;
};

__device__ __forceinline__ void fine_seg_load(FineSeg& f, unsigned k, int Ts, int SX, int tiles_x, int tiles_y,
                                              const unsigned* s_first, const uint2* __restrict__ crange,
                                              const unsigned* __restrict__ cvals, const unsigned* __restrict__ F,
                                              const unsigned* __restrict__ tile_start, int lane) {
    const int st = segment_tile(s_first, Ts, k);
    const uint2 rg = crange[st];
    const unsigned p0 = rg.x + (k - s_first[st]) * kSeg, p1 = min(p0 + kSeg, rg.y);
    f.tx0 = (st % SX) * kSuper;
    f.ty0 = (st / SX) * kSuper;
    f.start = 0;
    const int tx = f.tx0 + (lane & 3), ty = f.ty0 + ((lane >> 2) & 3);
    if (lane < kSuperTiles && tx < tiles_x && ty < tiles_y)
        f.start = tile_start[ty * tiles_x + tx] + F[(size_t)k * kSuperTiles + lane];
#pragma unroll
    for (int r = 0; r < kRounds; ++r) f.iv[r] = p0 + 32 * r + lane < p1 ? cvals[p0 + 32 * r + lane] : ~0u;
}

// The placement loop of k_fine_place. KEY64: also writes the 64-bit keys. CHECK: positions may
// reach the capacity (D above it), so each store is checked; otherwise every position is below D.
template <bool KEY64, bool CHECK>
__device__ __forceinline__ void fine_place_loop(unsigned k, unsigned ns, unsigned stride, int Ts, int SX, int tiles_x,
                                                int tiles_y, unsigned n_bound, const unsigned* s_first,
                                                const uint2* __restrict__ crange, const unsigned* __restrict__ cvals,
                                                const uint2* __restrict__ crect, const unsigned* __restrict__ perm,
                                                const unsigned* __restrict__ F, const unsigned* __restrict__ tile_start,
                                                unsigned capacity, unsigned* __restrict__ vals,
                                                unsigned long long* __restrict__ keys64,
                                                const unsigned* __restrict__ depth_bits, unsigned* __restrict__ err,
                                                int lane) {
    const unsigned full = 0xffffffffu;
    FineSeg cur;
    fine_seg_load(cur, k, Ts, SX, tiles_x, tiles_y, s_first, crange, cvals, F, tile_start, lane);
    const unsigned lt = lanemask_lt();
    for (; k < ns; k += stride) {
        // the entries' rectangles and Gaussians (dependent loads), then the next segment's loads
        unsigned m16v[kRounds], gv[kRounds];
#pragma unroll
        for (int r = 0; r < kRounds; ++r) {  // a depth position below V <= n
            const bool ok = cur.iv[r] < n_bound;
            m16v[r] = ok ? cover_mask(crect[cur.iv[r]], cur.tx0, cur.ty0) : 0u;
            gv[r] = ok ? perm[cur.iv[r]] : 0u;
        }
        unsigned next[kSuperTiles];
#pragma unroll
        for (int t = 0; t < kSuperTiles; ++t) next[t] = __shfl_sync(full, cur.start, t);
        const int tx0 = cur.tx0, ty0 = cur.ty0;
        if (k + stride < ns)
            fine_seg_load(cur, k + stride, Ts, SX, tiles_x, tiles_y, s_first, crange, cvals, F, tile_start, lane);
        // one tile of a round: the lanes whose Gaussian covers tile t write consecutive positions
        auto place_tile = [&](int t, unsigned m16, unsigned g) {
            const bool mine = (m16 >> t) & 1u;
            const unsigned m = __ballot_sync(full, mine);
            const unsigned pos = next[t] + __popc(m & lt);
            if (mine) {
                if (!CHECK || pos < capacity) {
                    vals[pos] = g;
                    if (KEY64) {
                        const unsigned tile = (unsigned)((ty0 + (t >> 2)) * tiles_x + tx0 + (t & 3));
                        keys64[pos] = ((unsigned long long)tile << 32) | depth_bits[g];
                    }
                } else {
                    atomicOr(err, kErrCheck);
                }
            }
            next[t] += __popc(m);
        };
#pragma unroll
        for (int r = 0; r < kRounds; ++r) {
            const unsigned m16 = m16v[r], g = gv[r];
            const unsigned any = __reduce_or_sync(full, m16);
            if (any == 0xffffu) {  // warp-uniform: every tile is covered by some lane
#pragma unroll
                for (int t = 0; t < kSuperTiles; ++t) place_tile(t, m16, g);
            } else {
#pragma unroll
                for (int t = 0; t < kSuperTiles; ++t)
                    if (any & (1u << t)) place_tile(t, m16, g);  // warp-uniform
            }
        }
    }
}

// total: D (the fine tile scan's); when it is within the capacity, no position reaches it and the
// stores go unchecked.
template <bool KEY64>
__global__ void __launch_bounds__(256) k_fine_place(int Ts, int SX, int tiles_x, int tiles_y, unsigned n_bound,
                                                    const unsigned* __restrict__ seg_first,
                                                    const unsigned* __restrict__ nseg,
                                                    const uint2* __restrict__ crange,
                                                    const unsigned* __restrict__ cvals,
                                                    const uint2* __restrict__ crect, const unsigned* __restrict__ perm,
                                                    const unsigned* __restrict__ F,
                                                    const unsigned* __restrict__ tile_start,
                                                    const unsigned long long* __restrict__ total, unsigned capacity,
                                                    unsigned* __restrict__ vals, unsigned long long* __restrict__ keys64,
                                                    const unsigned* __restrict__ depth_bits,
                                                    unsigned* __restrict__ err) {
    pdl_entry();
    extern __shared__ unsigned s_first[];
    for (int t = threadIdx.x; t <= Ts; t += blockDim.x) s_first[t] = seg_first[t];
    __syncthreads();
    const int lane = threadIdx.x & 31;
    const unsigned ns = *nseg, wpb = blockDim.x >> 5, stride = gridDim.x * wpb;
    const unsigned k = blockIdx.x * wpb + (threadIdx.x >> 5);
    if (k >= ns) return;
    if (!KEY64 && *total <= (unsigned long long)capacity)  // the key-writing form keeps one, checked loop
        fine_place_loop<KEY64, false>(k, ns, stride, Ts, SX, tiles_x, tiles_y, n_bound, s_first, crange, cvals, crect,
                                      perm, F, tile_start, capacity, vals, keys64, depth_bits, err, lane);
    else
        fine_place_loop<KEY64, true>(k, ns, stride, Ts, SX, tiles_x, tiles_y, n_bound, s_first, crange, cvals, crect,
                                     perm, F, tile_start, capacity, vals, keys64, depth_bits, err, lane);
}

// ---- self-test of the bounded look-back ------------------------------------------------------

// Pass histogram and ticket of the look-back self-test: 8192 items of digit 0, and the ticket
// counter starting at 1, so that the single block launched takes index 1 and its predecessor,
// block 0, never exists.
__global__ void k_selftest_lookback_init(unsigned* __restrict__ ghist4, unsigned* __restrict__ ticket) {
    if (threadIdx.x == 0) {
        ghist4[0] = 2u * kSortItems;
        ticket[0] = 1u;
    }
}

// One block of the first depth pass runs as block 1 over items 4096..8191 (all keys 0). Its
// look-back polls block 0's status words, which nothing writes: each poll finds them empty, and
// after spin_limit polls the wait gives up and sets the timeout bit. The block then places its
// items at positions 0..4095 of the output arrays. Workspace layout (106,512 bytes): keys in,
// keys out, values out (8192 words each), the four pass histograms (1024 words), four tickets,
// two blocks' status words (512 x 8 bytes).
cudaError_t selftest_lookback(unsigned char* ws, unsigned spin_limit, unsigned* err, cudaStream_t st) {
    constexpr int kItems = 2 * kSortItems;
    unsigned* keys_in = reinterpret_cast<unsigned*>(ws);
    unsigned* keys_out = keys_in + kItems;
    unsigned* vals_out = keys_out + kItems;
    unsigned* ghist4 = vals_out + kItems;
    unsigned* ticket = ghist4 + 4 * 256;
    unsigned long long* status = reinterpret_cast<unsigned long long*>(ticket + 4);
    static_assert((3 * kItems + 4 * 256 + 4) * 4 + 2 * 256 * 8 == kSelftestLookbackBytes, "self-test layout");
    cudaError_t e = cudaMemsetAsync(ws, 0, kSelftestLookbackBytes, st);
    if (e) return e;
    count_launches(2);
    k_selftest_lookback_init<<<1, 32, 0, st>>>(ghist4, ticket);
    if ((e = cudaGetLastError())) return e;
    k_onesweep<true><<<1, kSortThreads, 0, st>>>(keys_in, nullptr, keys_out, vals_out, kItems, ghist4, nullptr, 0,
                                                 ticket, status, nullptr, spin_limit, err);
    return cudaGetLastError();
}

// ---- host orchestration ----------------------------------------------------------------------

static size_t align256(size_t x) { return (x + 255) & ~(size_t)255; }

static int sort_blocks(long long items) { return (int)((items + kSortItems - 1) / kSortItems); }

int tile_bits_of(long long tiles) {
    int b = 0;
    while ((1ll << b) < tiles) ++b;
    return b;
}

bool counting_path(long long tiles) { return tiles <= kMaxCountTiles; }

SortWorkspace carve_workspace(void* base, long long n, long long cap, int tiles_x, int tiles_y) {
    SortWorkspace w{};
    const long long tiles = (long long)tiles_x * tiles_y;
    char* p = static_cast<char*>(base);
    size_t off = 0;
    auto take = [&](size_t bytes) { char* q = p ? p + off : nullptr; off += align256(bytes); return q; };
    const long long nn = n > 0 ? n : 1, cc = cap > 0 ? cap : 1, tt = tiles > 0 ? tiles : 1;
    const bool counting = counting_path(tt);
    w.dkA = (unsigned*)take(4 * nn);
    w.dkB = (unsigned*)take(4 * nn);
    w.dvA = (unsigned*)take(4 * nn);
    w.dvB = (unsigned*)take(4 * nn);
    const int nbmax = sort_blocks(counting ? nn : (nn > cc ? nn : cc));
    w.hist = (unsigned*)take((size_t)256 * nbmax * 4);
    w.totals = (unsigned*)take(256 * 4);
    w.total = (unsigned long long*)take(8);
    w.nvis = (unsigned*)take(4);
    // depth sort: 4 digit histograms, 4 tickets, 4 x (blocks x 256) look-back words, one region
    w.sweep_blocks = sort_blocks(nn);
    w.sweep_bytes = 4 * 256 * 4 + 256 + (size_t)4 * w.sweep_blocks * 256 * 8;
    w.sweep = (unsigned char*)take(w.sweep_bytes);
    const long long gblocks = (nn + 255) / 256;
    w.bsum = (unsigned long long*)take(8 * gblocks);
    w.boff = (unsigned long long*)take(8 * gblocks);
    if (counting) {
        const long long ts = (long long)((tiles_x + kSuper - 1) / kSuper) * ((tiles_y + kSuper - 1) / kSuper);
        w.cmax = max_chunks(nn, cc);
        w.crect = (uint2*)take(8 * nn);
        w.ssum = (unsigned long long*)take(8 * gblocks);
        w.soff = (unsigned long long*)take(8 * gblocks);
        w.ctotal = (unsigned long long*)take(8);
        w.table = (unsigned*)take((size_t)w.cmax * ts * 4);
        w.group_sum = (unsigned*)take((size_t)((w.cmax + kScanGroup - 1) / kScanGroup) * ts * 4);
        w.stile_total = (unsigned*)take(4 * ts);
        w.stile_start = (unsigned*)take(4 * ts);
        w.crange = (uint2*)take(8 * ts);
        w.cvals = (unsigned*)take(4 * cc);
        w.chunk_first = (unsigned*)take(4 * (w.cmax + 1));
        w.nchunks = (unsigned*)take(4);
        w.seg_cap = cc / kSeg + ts + 1;
        w.seg_first = (unsigned*)take(4 * (ts + 1));
        w.nseg = (unsigned*)take(4);
        w.fcount = (unsigned*)take((size_t)w.seg_cap * kSuperTiles * 4);
        w.tile_total = (unsigned*)take(4 * tt);
        w.tile_start = (unsigned*)take(4 * tt);
    } else {
        w.tA = (unsigned*)take(4 * cc);
        w.tB = (unsigned*)take(4 * cc);
        w.vB = (unsigned*)take(4 * cc);
    }
    w.bytes = off;
    return w;
}

static cudaError_t radix_pass(const unsigned* kin, const unsigned* vin, unsigned* kout, unsigned* vout, int n,
                              const unsigned* n_dev, const int* radius, unsigned* count_out, int shift, int bits,
                              bool iota, unsigned long long* keys64, const unsigned* depth_bits,
                              const SortWorkspace& w, cudaStream_t st) {
    if (n == 0) return cudaSuccess;
    const int nb = sort_blocks(n);
    const unsigned mask = (1u << bits) - 1u;
    count_launches(3);
    k_radix_hist<<<nb, kSortThreads, 0, st>>>(kin, n, n_dev, radius, shift, mask, w.hist, nb);
    k_radix_scan<<<256, 1024, 0, st>>>(w.hist, nb, w.totals, count_out);
    if (iota)
        k_radix_scatter<true, false><<<nb, kSortThreads, 0, st>>>(kin, vin, kout, vout, n, n_dev, radius, shift, mask,
                                                                  w.hist, w.totals, nb, nullptr, nullptr);
    else if (keys64)
        k_radix_scatter<false, true><<<nb, kSortThreads, 0, st>>>(kin, vin, kout, vout, n, n_dev, radius, shift, mask,
                                                                  w.hist, w.totals, nb, keys64, depth_bits);
    else
        k_radix_scatter<false, false><<<nb, kSortThreads, 0, st>>>(kin, vin, kout, vout, n, n_dev, radius, shift, mask,
                                                                   w.hist, w.totals, nb, nullptr, nullptr);
    return cudaGetLastError();
}

// Phase 1: depth sort of the visible Gaussians (the first pass drops radius-0 Gaussians; the
// second leaves their number V on the device, and the count runs over V items) and the duplicate
// count; leaves the total D in w.total (device). Bounded look-back waits set the timeout bit of
// `err` when they give up.
cudaError_t bin_count(const gs_proj& proj, int tiles_x, int tiles_y, const SortWorkspace& w, unsigned* err,
                      unsigned spin_limit, unsigned long long capacity, unsigned* ranges, unsigned* overflow_err,
                      unsigned long long* total_copy, cudaStream_t st) {
    const int n = (int)proj.n;
    if (n == 0) return cudaMemsetAsync(w.total, 0, 8, st);
    const unsigned* depth_bits = reinterpret_cast<const unsigned*>(proj.depth);
    const int T = tiles_x * tiles_y;
    cudaError_t e;
    // both memsets first, so that the kernels after them follow one another directly (launch_pdl)
    if ((e = cudaMemsetAsync(w.sweep, 0, w.sweep_bytes, st))) return e;
    if (counting_path(T) && (e = cudaMemsetAsync(w.nchunks, 0, 4, st))) return e;
    unsigned* ghist4 = reinterpret_cast<unsigned*>(w.sweep);
    unsigned* tickets = ghist4 + 4 * 256;
    unsigned long long* status = reinterpret_cast<unsigned long long*>(w.sweep + 4 * 256 * 4 + 256);
    const size_t sstride = (size_t)w.sweep_blocks * 256;
    const int nb = sort_blocks(n);
    const int hblocks = nb < 4 * 152 ? nb : 4 * 152;
    // the first pass runs over all N Gaussians: three blocks per SM (its launch bound, and shared
    // memory preferred over L1) keep its 4096-item blocks in one wave up to 1.87M Gaussians
    if ((e = cudaFuncSetAttribute(k_onesweep<true>, cudaFuncAttributePreferredSharedMemoryCarveout,
                                  (int)cudaSharedmemCarveoutMaxShared)))
        return e;
    count_launches(5);
    if ((e = launch_pdl(k_depth_hist4, dim3(hblocks), dim3(256), 0, st, depth_bits, n, proj.radius, ghist4)))
        return e;
    if ((e = launch_pdl(k_onesweep<true>, dim3(nb), dim3(kSortThreads), 0, st, depth_bits, nullptr, w.dkA, w.dvA, n,
                        ghist4, proj.radius, 0, tickets, status, nullptr, spin_limit, err)))
        return e;
    if ((e = launch_pdl(k_onesweep<false>, dim3(nb), dim3(kSortThreads), 0, st, w.dkA, w.dvA, w.dkB, w.dvB, n, ghist4,
                        nullptr, 1, tickets + 1, status + sstride, w.nvis, spin_limit, err)))
        return e;
    if ((e = launch_pdl(k_onesweep<false>, dim3(nb), dim3(kSortThreads), 0, st, w.dkB, w.dvB, w.dkA, w.dvA, n, ghist4,
                        nullptr, 2, tickets + 2, status + 2 * sstride, nullptr, spin_limit, err)))
        return e;
    if ((e = launch_pdl(k_onesweep<false>, dim3(nb), dim3(kSortThreads), 0, st, w.dkA, w.dvA, w.dkB, w.dvB, n, ghist4,
                        nullptr, 3, tickets + 3, status + 3 * sstride, nullptr, spin_limit, err)))
        return e;
    const float4* rec = reinterpret_cast<const float4*>(proj.rec);
    const int gblocks = (n + 255) / 256;
    if (counting_path(T)) {
        // duplicate total D (fine), then the coarse level's counts, offsets and super-tile ranges
        const int sx = (tiles_x + kSuper - 1) / kSuper, sy = (tiles_y + kSuper - 1) / kSuper, ts = sx * sy;
        const size_t smem = (size_t)ts * 4;
        if ((e = cudaFuncSetAttribute(k_chunk_hist, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem)))
            return e;
        count_launches(6);
        if ((e = launch_pdl(k_count, dim3(gblocks), dim3(256), 0, st, n, w.nvis, w.dvB, rec, proj.radius, tiles_x,
                            tiles_y, w.bsum, w.crect, w.ssum)))
            return e;
        if ((e = launch_pdl(k_scan_u64, dim3(2), dim3(1024), 0, st, w.bsum, gblocks, w.boff, w.total, total_copy,
                            (const unsigned long long*)w.ssum, w.soff, w.ctotal)))
            return e;
        if ((e = launch_pdl(k_chunk_bounds, dim3(gblocks), dim3(256), 0, st, n, w.nvis, w.crect, w.soff,
                            (int)w.cmax, w.chunk_first, w.nchunks)))
            return e;
        if ((e = launch_pdl(k_chunk_hist, dim3((unsigned)w.cmax), dim3(256), smem, st, w.nchunks,
                            w.chunk_first, w.crect, sx, ts, w.table)))
            return e;
        // the column sums of the row groups are needed only when there can be more than one group
        const unsigned groups = (unsigned)((w.cmax + kScanGroup - 1) / kScanGroup);
        if (groups > 1) {
            count_launches(1);
            if ((e = launch_pdl(k_chunk_colsum, dim3((ts + 31) / 32, groups), dim3(32 * kScanWarps), 0, st,
                                w.nchunks, ts, (const unsigned*)w.table, w.group_sum)))
                return e;
        }
        if ((e = launch_pdl(k_chunk_scan, dim3((ts + 31) / 32, groups), dim3(32 * kScanWarps), 0, st, w.nchunks, ts,
                            w.table, (const unsigned*)w.group_sum, w.stile_total)))
            return e;
        // the coarse lists hold at most D' <= D entries: over the capacity only when D is
        return launch_pdl(k_tile_scan, dim3(1), dim3(1024), 0, st, ts, w.stile_total, w.stile_start, w.ctotal,
                          capacity, reinterpret_cast<uint2*>(w.crange), overflow_err,
                          (unsigned long long*)nullptr, w.seg_first, w.nseg, (unsigned)w.seg_cap);
    }
    count_launches(2);
    if ((e = launch_pdl(k_count, dim3(gblocks), dim3(256), 0, st, n, w.nvis, w.dvB, rec, proj.radius, tiles_x, tiles_y,
                        w.bsum, (uint2*)nullptr, (unsigned long long*)nullptr)))
        return e;
    return launch_pdl(k_scan_u64, dim3(1), dim3(1024), 0, st, w.bsum, gblocks, w.boff, w.total,
                      (unsigned long long*)nullptr, (const unsigned long long*)nullptr, (unsigned long long*)nullptr,
                      (unsigned long long*)nullptr);
}

// Counting-path emission: the coarse placement, the fine counts and scans, the tile ranges and the
// fine placement. Reads no count on the host (every count stays on the device).
static cudaError_t emit_counting(const gs_proj& proj, int tiles_x, int tiles_y, unsigned long long capacity,
                                 const SortWorkspace& w, uint64_t* keys, unsigned* vals, unsigned* ranges,
                                 unsigned* err, cudaStream_t st) {
    const unsigned* depth_bits = reinterpret_cast<const unsigned*>(proj.depth);
    unsigned long long* k64 = reinterpret_cast<unsigned long long*>(keys);
    const int sx = (tiles_x + kSuper - 1) / kSuper, sy = (tiles_y + kSuper - 1) / kSuper, ts = sx * sy;
    const int T = tiles_x * tiles_y;
    cudaError_t e;
    // coarse placement: one warp per (chunk, band of super-tile rows)
    const int band_rows = (sy + kPlaceBands - 1) / kPlaceBands;
    const int nbands = (sy + band_rows - 1) / band_rows;
    const size_t band_bytes = (size_t)band_rows * sx * 4;
    int wpb = (int)((200 * 1024) / band_bytes);
    wpb = wpb < 1 ? 1 : (wpb > kPlaceWarps ? kPlaceWarps : wpb);
    const size_t smem = (size_t)wpb * band_bytes;
    if ((e = cudaFuncSetAttribute(k_chunk_place, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem)))
        return e;
    const size_t fsmem = (size_t)(ts + 1) * 4;
    if ((e = cudaFuncSetAttribute(k_fine_count, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)fsmem))) return e;
    auto fine_place = k64 ? k_fine_place<true> : k_fine_place<false>;
    if ((e = cudaFuncSetAttribute(fine_place, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)fsmem))) return e;
    const long long warps = w.cmax * nbands;
    count_launches(5);
    if ((e = launch_pdl(k_chunk_place, dim3((unsigned)((warps + wpb - 1) / wpb)), dim3(32 * wpb), smem, st,
                        w.nchunks, w.chunk_first, w.crect, sx, sy, band_rows, nbands, w.table, w.stile_start,
                        (const unsigned long long*)w.ctotal, (unsigned)capacity, w.cvals, err)))
        return e;
    // grid-stride kernels over the segments (8 warps per block): at most the resident blocks
    static std::atomic<int> count_cache[256], place_cache[256], place64_cache[256];
    const long long seg_blocks = (w.seg_cap + 7) / 8;
    const int rc = resident_blocks(k_fine_count, 256, fsmem, count_cache);
    const int rp = resident_blocks(fine_place, 256, fsmem, k64 ? place64_cache : place_cache);
    const unsigned fcblocks = (unsigned)(rc > 0 && seg_blocks > rc ? rc : seg_blocks);
    const unsigned fblocks = (unsigned)(rp > 0 && seg_blocks > rp ? rp : seg_blocks);
    if ((e = launch_pdl(k_fine_count, dim3(fcblocks), dim3(256), fsmem, st, ts, sx, (unsigned)proj.n, w.seg_first,
                        w.nseg, reinterpret_cast<const uint2*>(w.crange), w.cvals, w.crect, w.fcount)))
        return e;
    if ((e = launch_pdl(k_fine_scan, dim3((unsigned)((ts + 7) / 8)), dim3(256), 0, st, ts, sx, tiles_x, tiles_y,
                        w.seg_first, (unsigned)w.seg_cap, w.fcount, w.tile_total)))
        return e;
    if ((e = launch_pdl(k_tile_scan, dim3(1), dim3(1024), 0, st, T, w.tile_total, w.tile_start, w.total, capacity,
                        reinterpret_cast<uint2*>(ranges), err, (unsigned long long*)nullptr, (unsigned*)nullptr,
                        (unsigned*)nullptr, 0u)))
        return e;
    return launch_pdl(fine_place, dim3(fblocks), dim3(256), fsmem, st, ts, sx, tiles_x, tiles_y,
                      (unsigned)proj.n, w.seg_first,
                      w.nseg, reinterpret_cast<const uint2*>(w.crange), w.cvals, w.crect, w.dvB, w.fcount,
                      w.tile_start, (const unsigned long long*)w.total, (unsigned)capacity, vals, k64, depth_bits, err);
}

// Phase 2: placement (counting pass) or emission + tile radix passes and the ranges.
// d = number of duplicates (<= capacity).
cudaError_t bin_emit_sort(const gs_proj& proj, int tiles_x, int tiles_y, unsigned d, unsigned long long capacity,
                          const SortWorkspace& w, uint64_t* keys, unsigned* vals, unsigned* ranges, unsigned* err,
                          cudaStream_t st) {
    const int n = (int)proj.n;
    const long long T = (long long)tiles_x * tiles_y;
    cudaError_t e = cudaSuccess;
    if (n == 0 || d == 0 || !counting_path(T)) {
        if ((e = cudaMemsetAsync(ranges, 0, (size_t)T * 8, st))) return e;
        if (n == 0 || d == 0) return cudaSuccess;
    }
    const unsigned* depth_bits = reinterpret_cast<const unsigned*>(proj.depth);
    unsigned long long* k64 = reinterpret_cast<unsigned long long*>(keys);
    if (counting_path(T)) return emit_counting(proj, tiles_x, tiles_y, capacity, w, keys, vals, ranges, err, st);
    const int tb = tile_bits_of(T);
    const int passes = (tb + 7) / 8;
    unsigned* tbuf[2] = {w.tA, w.tB};
    unsigned* vbuf[2] = {vals, w.vB};
    int cur = passes & 1;  // emission target so that the last pass lands in `vals`
    const int gblocks = (n + 255) / 256;
    const float4* rec = reinterpret_cast<const float4*>(proj.rec);
    count_launches(1);
    k_emit<<<gblocks, 256, 0, st>>>(n, w.nvis, w.dvB, rec, proj.radius, tiles_x, tiles_y, w.boff, capacity, tbuf[cur],
                                    vbuf[cur], err);
    for (int p = 0; p < passes; ++p) {
        const int bits = (tb - 8 * p) < 8 ? (tb - 8 * p) : 8;
        const bool lastp = p == passes - 1;
        if ((e = radix_pass(tbuf[cur], vbuf[cur], tbuf[cur ^ 1], vbuf[cur ^ 1], (int)d, nullptr, nullptr, nullptr,
                            8 * p, bits, false, lastp ? k64 : nullptr, depth_bits, w, st)))
            return e;
        cur ^= 1;
    }
    if (passes == 0 && k64) {
        count_launches(1);
        k_make_keys<<<(d + 255) / 256, 256, 0, st>>>(d, tbuf[cur], vals, depth_bits, k64);
    }
    count_launches(1);
    k_ranges<<<(d + 1023) / 1024, 256, 0, st>>>(d, tbuf[cur], reinterpret_cast<uint2*>(ranges));
    return cudaGetLastError();
}

// The whole binning and sort with no host synchronisation (counting path only): D is written to
// n_dup_dev (when given) on the stream; duplicates beyond the capacity are dropped, every range is
// written empty and the check bit is set.
cudaError_t bin_sort_async(const gs_proj& proj, int tiles_x, int tiles_y, unsigned long long capacity,
                           const SortWorkspace& w, uint64_t* keys, unsigned* vals, unsigned* ranges,
                           unsigned long long* n_dup_dev, unsigned* err, unsigned spin_limit, cudaStream_t st) {
    const long long T = (long long)tiles_x * tiles_y;
    // the tile scan writes D to n_dup_dev itself (no copy between the placement and the next kernel)
    cudaError_t e = bin_count(proj, tiles_x, tiles_y, w, err, spin_limit, capacity, ranges, err, n_dup_dev, st);
    if (e) return e;
    if (proj.n == 0) {
        if ((e = cudaMemsetAsync(ranges, 0, (size_t)T * 8, st))) return e;
        return n_dup_dev ? cudaMemsetAsync(n_dup_dev, 0, 8, st) : cudaSuccess;
    }
    return emit_counting(proj, tiles_x, tiles_y, capacity, w, keys, vals, ranges, err, st);
}

}  // namespace gs
