// Tile duplication and sorting: the binning stage of the tile rasterization pipeline (DISTWAR:
// Fast Differentiable Rendering on Raster-based Rendering Pipelines, Abstract, names the
// rasterization pipeline; the duplication, keying and sort follow 3D Gaussian splatting's tile
// rasterizer).
//
// Result: for every Gaussian with radius > 0 and every tile of its tile rectangle one entry,
// ordered by (tile, float32 depth bits, Gaussian index). Instead of sorting the D = sum of tiles
// 64-bit (tile << 32 | depth) keys with 32 + log2(T) bits of passes, the Gaussians are sorted
// by their 32 depth bits (N items, 4 stable passes), their duplicates are emitted in that order,
// and the duplicates are sorted stably by tile id (ceil(log2(T) / 8) passes over D items). A
// stable LSD radix sort on the low key bits followed by passes on the high bits is exactly what
// a stable sort of the full keys computes, and the emission copies a Gaussian's position in the
// depth order to all of its duplicates, so the result equals the stable sort of the 64-bit keys
// of the index-ordered duplicate list.
//
// Radix pass = histogram (per 4096-item block, 8-bit digit), scan (per digit over blocks),
// stable scatter (per warp: 16 rounds of 32 consecutive items ranked with match_any).
#include "gs_common.cuh"
#include "gs_internal.h"

namespace gs {

constexpr int kSortThreads = 256;
constexpr int kSortRounds = 16;                          // rounds of 32 items per warp
constexpr int kSortItems = kSortThreads * kSortRounds;  // 4096 items per block
constexpr int kWarpItems = 32 * kSortRounds;            // 512 items per warp

__global__ void __launch_bounds__(kSortThreads) k_radix_hist(const unsigned* __restrict__ keys, int n, int shift,
                                                             unsigned mask, unsigned* __restrict__ hist, int nblocks) {
    __shared__ unsigned h[8][256];
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    for (int i = threadIdx.x; i < 8 * 256; i += kSortThreads) (&h[0][0])[i] = 0u;
    __syncthreads();
    const int base = blockIdx.x * kSortItems + warp * kWarpItems + lane;
#pragma unroll 4
    for (int r = 0; r < kSortRounds; ++r) {
        const int idx = base + r * 32;
        const bool valid = idx < n;
        const unsigned d = valid ? (keys[idx] >> shift) & mask : 0x100u;
        const unsigned peers = __match_any_sync(0xffffffffu, d);
        if (valid && (peers & lanemask_lt()) == 0u) h[warp][d] += __popc(peers);
        __syncwarp();
    }
    __syncthreads();
    const int d = threadIdx.x;
    unsigned sum = 0;
#pragma unroll
    for (int w = 0; w < 8; ++w) sum += h[w][d];
    hist[(size_t)d * nblocks + blockIdx.x] = sum;
}

// Exclusive scan of one digit's row of per-block counts (one block of 1024 threads per digit).
__global__ void __launch_bounds__(1024) k_radix_scan(unsigned* __restrict__ hist, int nblocks,
                                                     unsigned* __restrict__ totals) {
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
    if (threadIdx.x == 0) totals[blockIdx.x] = carry;
}

// Stable scatter of one 8-bit digit. IOTA: the values are the item indices. KEY64: also write
// the 64-bit key (key << 32 | depth_bits[value]) of every item.
//
// Each warp ranks its 512 items (16 rounds of 32, in index order) with match_any; the block then
// reorders its 4096 items by digit in shared memory and writes every digit's run to consecutive
// global addresses, so the global writes are coalesced.
template <bool IOTA, bool KEY64>
__global__ void __launch_bounds__(kSortThreads) k_radix_scatter(
    const unsigned* __restrict__ keys_in, const unsigned* __restrict__ vals_in, unsigned* __restrict__ keys_out,
    unsigned* __restrict__ vals_out, int n, int shift, unsigned mask, const unsigned* __restrict__ hist,
    const unsigned* __restrict__ totals, int nblocks, unsigned long long* __restrict__ keys64,
    const unsigned* __restrict__ depth_bits) {
    __shared__ unsigned woff[8][256];      // per-warp digit counts, then block-local offsets
    __shared__ unsigned lbase[256];        // block-local start of each digit
    __shared__ unsigned gbase[256];        // global start of this block's run of each digit
    __shared__ unsigned wsum[8];
    __shared__ unsigned sk[kSortItems], sv[kSortItems];
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int block_first = blockIdx.x * kSortItems;
    const int n_block = min(kSortItems, n - block_first);
    unsigned k[kSortRounds], v[kSortRounds];
    const int base = block_first + warp * kWarpItems + lane;
#pragma unroll
    for (int r = 0; r < kSortRounds; ++r) {
        const int idx = base + r * 32;
        const bool valid = idx < n;
        k[r] = valid ? keys_in[idx] : 0u;
        v[r] = IOTA ? (unsigned)idx : (valid ? vals_in[idx] : 0u);
    }
#pragma unroll
    for (int i = 0; i < 8; ++i) woff[warp][lane + 32 * i] = 0u;
    __syncwarp();
#pragma unroll
    for (int r = 0; r < kSortRounds; ++r) {
        const bool valid = base + r * 32 < n;
        const unsigned d = valid ? (k[r] >> shift) & mask : 0x100u;
        const unsigned peers = __match_any_sync(0xffffffffu, d);
        if (valid && (peers & lanemask_lt()) == 0u) woff[warp][d] += __popc(peers);
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
        const bool valid = base + r * 32 < n;
        const unsigned d = valid ? (k[r] >> shift) & mask : 0x100u;
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
    for (int i = threadIdx.x; i < n_block; i += kSortThreads) {
        const unsigned key = sk[i], val = sv[i];
        const unsigned d = (key >> shift) & mask;
        const unsigned pos = gbase[d] + (unsigned)i - lbase[d];
        keys_out[pos] = key;
        vals_out[pos] = val;
        if (KEY64) keys64[pos] = ((unsigned long long)key << 32) | depth_bits[val];
    }
}

// Block sums (256 Gaussians per block, in depth order) of the number of tiles of each rectangle.
__global__ void __launch_bounds__(256) k_count(int n, const unsigned* __restrict__ perm, const float4* __restrict__ rec,
                                               const int* __restrict__ radius, int tiles_x, int tiles_y,
                                               unsigned long long* __restrict__ block_sums) {
    __shared__ unsigned long long ws[8];
    const int i = blockIdx.x * 256 + threadIdx.x;
    unsigned long long cnt = 0;
    if (i < n) {
        const unsigned g = perm[i];
        const int r = radius[g];
        if (r > 0) {
            const float4 r0 = rec[3 * (size_t)g];
            const Rect R = tile_rect(r0.x, r0.y, r, tiles_x, tiles_y);
            if (R.x0 <= R.x1) cnt = (unsigned long long)(R.x1 - R.x0 + 1) * (unsigned long long)(R.y1 - R.y0 + 1);
        }
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) cnt += __shfl_xor_sync(0xffffffffu, cnt, o);
    if ((threadIdx.x & 31) == 0) ws[threadIdx.x >> 5] = cnt;
    __syncthreads();
    if (threadIdx.x == 0) {
        unsigned long long s = 0;
        for (int w = 0; w < 8; ++w) s += ws[w];
        block_sums[blockIdx.x] = s;
    }
}

// Exclusive scan of the block sums (single block); total[0] = sum of all.
__global__ void __launch_bounds__(1024) k_scan_u64(const unsigned long long* __restrict__ in, int m,
                                                   unsigned long long* __restrict__ out,
                                                   unsigned long long* __restrict__ total) {
    __shared__ unsigned long long wsum[32];
    __shared__ unsigned long long carry;
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    if (threadIdx.x == 0) carry = 0ull;
    __syncthreads();
    for (int base = 0; base < m; base += 1024) {
        const int i = base + threadIdx.x;
        const unsigned long long v = i < m ? in[i] : 0ull;
        unsigned long long x = v;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const unsigned long long y = __shfl_up_sync(0xffffffffu, x, o);
            if (lane >= o) x += y;
        }
        if (lane == 31) wsum[warp] = x;
        __syncthreads();
        if (warp == 0) {
            unsigned long long s = wsum[lane];
#pragma unroll
            for (int o = 1; o < 32; o <<= 1) {
                const unsigned long long y = __shfl_up_sync(0xffffffffu, s, o);
                if (lane >= o) s += y;
            }
            wsum[lane] = s;
        }
        __syncthreads();
        const unsigned long long wpre = warp ? wsum[warp - 1] : 0ull;
        if (i < m) out[i] = carry + wpre + x - v;
        __syncthreads();
        if (threadIdx.x == 0) carry += wsum[31];
        __syncthreads();
    }
    if (threadIdx.x == 0) total[0] = carry;
}

// Emits the duplicates of 256 consecutive Gaussians (depth order) into their block's contiguous
// output range: output o goes to the Gaussian whose prefix range contains o (binary search over
// the block's 256 offsets), and is its (o - offset)-th tile in row-major rectangle order.
__global__ void __launch_bounds__(256) k_emit(int n, const unsigned* __restrict__ perm, const float4* __restrict__ rec,
                                              const int* __restrict__ radius, int tiles_x, int tiles_y,
                                              const unsigned long long* __restrict__ block_offs,
                                              unsigned long long capacity, unsigned* __restrict__ tile_out,
                                              unsigned* __restrict__ val_out, unsigned* __restrict__ err) {
    __shared__ unsigned s_off[257];
    __shared__ int s_x0[256], s_y0[256], s_w[256];
    __shared__ unsigned s_g[256];
    __shared__ unsigned wsum[8];
    const int i = blockIdx.x * 256 + threadIdx.x;
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    unsigned cnt = 0, g = 0;
    int x0 = 0, y0 = 0, w = 1;
    if (i < n) {
        g = perm[i];
        const int r = radius[g];
        if (r > 0) {
            const float4 r0 = rec[3 * (size_t)g];
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

// ---- host orchestration ----------------------------------------------------------------------

static size_t align256(size_t x) { return (x + 255) & ~(size_t)255; }

static int sort_blocks(long long items) { return (int)((items + kSortItems - 1) / kSortItems); }

int tile_bits_of(long long tiles) {
    int b = 0;
    while ((1ll << b) < tiles) ++b;
    return b;
}

SortWorkspace carve_workspace(void* base, long long n, long long cap) {
    SortWorkspace w{};
    char* p = static_cast<char*>(base);
    size_t off = 0;
    auto take = [&](size_t bytes) { char* q = p ? p + off : nullptr; off += align256(bytes); return q; };
    const long long nn = n > 0 ? n : 1, cc = cap > 0 ? cap : 1;
    w.dkA = (unsigned*)take(4 * nn);
    w.dkB = (unsigned*)take(4 * nn);
    w.dvA = (unsigned*)take(4 * nn);
    w.dvB = (unsigned*)take(4 * nn);
    const int nbmax = sort_blocks(nn > cc ? nn : cc);
    w.hist = (unsigned*)take((size_t)256 * nbmax * 4);
    w.totals = (unsigned*)take(256 * 4);
    const long long gblocks = (nn + 255) / 256;
    w.bsum = (unsigned long long*)take(8 * gblocks);
    w.boff = (unsigned long long*)take(8 * gblocks);
    w.total = (unsigned long long*)take(8);
    w.tA = (unsigned*)take(4 * cc);
    w.tB = (unsigned*)take(4 * cc);
    w.vB = (unsigned*)take(4 * cc);
    w.bytes = off;
    return w;
}

static cudaError_t radix_pass(const unsigned* kin, const unsigned* vin, unsigned* kout, unsigned* vout, int n, int shift,
                              int bits, bool iota, unsigned long long* keys64, const unsigned* depth_bits,
                              const SortWorkspace& w, cudaStream_t st) {
    if (n == 0) return cudaSuccess;
    const int nb = sort_blocks(n);
    const unsigned mask = (1u << bits) - 1u;
    count_launches(3);
    k_radix_hist<<<nb, kSortThreads, 0, st>>>(kin, n, shift, mask, w.hist, nb);
    k_radix_scan<<<256, 1024, 0, st>>>(w.hist, nb, w.totals);
    if (iota)
        k_radix_scatter<true, false><<<nb, kSortThreads, 0, st>>>(kin, vin, kout, vout, n, shift, mask, w.hist, w.totals, nb, nullptr, nullptr);
    else if (keys64)
        k_radix_scatter<false, true><<<nb, kSortThreads, 0, st>>>(kin, vin, kout, vout, n, shift, mask, w.hist, w.totals, nb, keys64, depth_bits);
    else
        k_radix_scatter<false, false><<<nb, kSortThreads, 0, st>>>(kin, vin, kout, vout, n, shift, mask, w.hist, w.totals, nb, nullptr, nullptr);
    return cudaGetLastError();
}

// Phase 1: depth sort and duplicate count; leaves the total in w.total (device).
cudaError_t bin_count(const gs_proj& proj, int tiles_x, int tiles_y, const SortWorkspace& w, cudaStream_t st) {
    const int n = (int)proj.n;
    if (n == 0) return cudaMemsetAsync(w.total, 0, 8, st);
    const unsigned* depth_bits = reinterpret_cast<const unsigned*>(proj.depth);
    cudaError_t e;
    if ((e = radix_pass(depth_bits, nullptr, w.dkA, w.dvA, n, 0, 8, true, nullptr, nullptr, w, st))) return e;
    if ((e = radix_pass(w.dkA, w.dvA, w.dkB, w.dvB, n, 8, 8, false, nullptr, nullptr, w, st))) return e;
    if ((e = radix_pass(w.dkB, w.dvB, w.dkA, w.dvA, n, 16, 8, false, nullptr, nullptr, w, st))) return e;
    if ((e = radix_pass(w.dkA, w.dvA, w.dkB, w.dvB, n, 24, 8, false, nullptr, nullptr, w, st))) return e;
    const int gblocks = (n + 255) / 256;
    const float4* rec = reinterpret_cast<const float4*>(proj.rec);
    count_launches(2);
    k_count<<<gblocks, 256, 0, st>>>(n, w.dvB, rec, proj.radius, tiles_x, tiles_y, w.bsum);
    k_scan_u64<<<1, 1024, 0, st>>>(w.bsum, gblocks, w.boff, w.total);
    return cudaGetLastError();
}

// Phase 2: emission in depth order, tile passes, ranges. d = number of duplicates (<= capacity).
cudaError_t bin_emit_sort(const gs_proj& proj, int tiles_x, int tiles_y, unsigned d, unsigned long long capacity,
                          const SortWorkspace& w, uint64_t* keys, unsigned* vals, unsigned* ranges, unsigned* err,
                          cudaStream_t st) {
    const int n = (int)proj.n;
    const long long T = (long long)tiles_x * tiles_y;
    cudaError_t e = cudaMemsetAsync(ranges, 0, (size_t)T * 8, st);
    if (e) return e;
    if (d == 0) return cudaSuccess;
    const int tb = tile_bits_of(T);
    const int passes = (tb + 7) / 8;
    const unsigned* depth_bits = reinterpret_cast<const unsigned*>(proj.depth);
    unsigned* tbuf[2] = {w.tA, w.tB};
    unsigned* vbuf[2] = {vals, w.vB};
    int cur = passes & 1;  // emission target so that the last pass lands in `vals`
    const int gblocks = (n + 255) / 256;
    const float4* rec = reinterpret_cast<const float4*>(proj.rec);
    count_launches(1);
    k_emit<<<gblocks, 256, 0, st>>>(n, w.dvB, rec, proj.radius, tiles_x, tiles_y, w.boff, capacity, tbuf[cur], vbuf[cur], err);
    unsigned long long* k64 = reinterpret_cast<unsigned long long*>(keys);
    for (int p = 0; p < passes; ++p) {
        const int bits = (tb - 8 * p) < 8 ? (tb - 8 * p) : 8;
        const bool lastp = p == passes - 1;
        if ((e = radix_pass(tbuf[cur], vbuf[cur], tbuf[cur ^ 1], vbuf[cur ^ 1], (int)d, 8 * p, bits, false,
                            lastp ? k64 : nullptr, depth_bits, w, st)))
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

}  // namespace gs
