// Stable LSD radix sort of (key, u32 value) pairs and run-length encoding of
// sorted keys -- the sort-based dedup behind the reduction-based and the
// unique-based backward ("NVIDIA EMBark revoluciona la formacion en sistemas
// de recomendacion a escala", section "Integracion del cluster": RB reduces
// over equal keys, UB dedups the keys first).
//
// Each pass runs three kernels over 3072-key tiles: a per-tile digit
// histogram, a scan of each digit's row over tiles, and stable in-tile
// ranking in shared memory with coalesced runs written to bucket start + tile
// offset.  No tile waits on another.  (A one-kernel pass whose tiles find
// their offsets by decoupled look-back measured slower at every size tried:
// the chain of published prefixes, not the extra read of the keys, set its
// pace.)  The element count and the number of significant key bits may live
// on the device (the unique-based path only learns them there); passes beyond
// the significant bits return at once, and the buffers are chosen so the last
// active pass always writes the output.
#include "emb_internal.cuh"

namespace emb {

namespace {

__device__ __forceinline__ uint32_t lanemask_lt()
{
    uint32_t m;
    asm("mov.u32 %0, %%lanemask_lt;" : "=r"(m));
    return m;
}

// Exclusive sum over the block (blockDim.x == kSortThreads); `total` gets the sum.
__device__ __forceinline__ uint32_t block_exclusive_sum(uint32_t x, uint32_t* warp_buf, uint32_t* total)
{
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    constexpr int kWarps = kSortThreads / 32;
    uint32_t incl = x;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        uint32_t y = __shfl_up_sync(0xffffffffu, incl, o);
        if (lane >= o) incl += y;
    }
    if (lane == 31) warp_buf[warp] = incl;
    __syncthreads();
    if (warp == 0) {
        uint32_t w = lane < kWarps ? warp_buf[lane] : 0u;
        uint32_t wi = w;
#pragma unroll
        for (int o = 1; o < kWarps; o <<= 1) {
            uint32_t y = __shfl_up_sync(0xffffffffu, wi, o);
            if (lane >= o) wi += y;
        }
        if (lane < kWarps) warp_buf[lane] = wi - w;
        if (lane == kWarps - 1) warp_buf[kWarps] = wi;
    }
    __syncthreads();
    uint32_t r = warp_buf[warp] + incl - x;
    if (total) *total = warp_buf[kWarps];
    __syncthreads();
    return r;
}

struct PassCtx {
    int64_t n;
    int64_t ntiles;
    int npe;       // effective passes
    bool active;
    bool dst_out;  // this pass writes the output buffers
    bool src_in;   // this pass reads the input buffers
};

__device__ __forceinline__ PassCtx pass_ctx(int64_t n_host, const int64_t* n_dev, const int32_t* bits_dev,
                                            int bits_max, int D, int pass, int tile)
{
    PassCtx c;
    int64_t n = n_host;
    if (n_dev) {
        int64_t m = *n_dev;
        n = m < n_host ? (m < 0 ? 0 : m) : n_host;
    }
    c.n = n;
    c.ntiles = (n + tile - 1) / tile;
    int b = bits_dev ? *bits_dev : bits_max;
    if (b < 1) b = 1;
    if (b > bits_max) b = bits_max;
    c.npe = (b + D - 1) / D;
    c.active = pass < c.npe && n > 0;
    c.dst_out = ((c.npe - 1 - pass) & 1) == 0;
    c.src_in = pass == 0;
    return c;
}

// ---- one pass: three kernels (histogram per tile, scan, ranking) ----

constexpr int kDownsweepBlocks = 4;   // resident blocks per SM the ranking kernel's registers are sized for

template <typename K, int ITEMS>
__global__ void __launch_bounds__(kSortThreads)
sort_upsweep(const K* __restrict__ keys_in, const K* keys_out, const K* keys_tmp, int64_t n_host,
             const int64_t* n_dev, const int32_t* bits_dev, int bits_max, int D, int pass,
             const uint64_t* key_sub, uint32_t* __restrict__ counts)
{
    constexpr int kTile = kSortThreads * ITEMS;
    PassCtx c = pass_ctx(n_host, n_dev, bits_dev, bits_max, D, pass, kTile);
    const int64_t tile = blockIdx.x;
    if (!c.active || tile >= c.ntiles) return;
    const K* src = c.src_in ? keys_in : (c.dst_out ? keys_tmp : keys_out);
    __shared__ uint32_t hist[1 << kMaxDigitBits];
    const int nb = 1 << D;
    for (int i = threadIdx.x; i < nb; i += kSortThreads) hist[i] = 0;
    __syncthreads();
    const int shift = pass * D;
    const K sub = (c.src_in && key_sub) ? (K)(*key_sub) : (K)0;
    const int64_t base = tile * kTile;
    const int lane = threadIdx.x & 31;
    // all of the thread's keys are requested before the first is counted
    uint32_t dg[ITEMS];
#pragma unroll
    for (int r = 0; r < ITEMS; ++r) {
        const int64_t idx = base + (int64_t)r * kSortThreads + threadIdx.x;
        dg[r] = idx < c.n ? (uint32_t)(((K)(src[idx] - sub) >> shift) & (K)(nb - 1)) : (uint32_t)nb;
    }
#pragma unroll
    for (int r = 0; r < ITEMS; ++r) {
        const uint32_t d = dg[r];
        uint32_t peers = __match_any_sync(0xffffffffu, d);
        int leader = __ffs(peers) - 1;
        if (lane == leader && d < (uint32_t)nb) atomicAdd(&hist[d], (uint32_t)__popc(peers));
    }
    __syncthreads();
    for (int d = threadIdx.x; d < nb; d += kSortThreads) counts[(int64_t)d * c.ntiles + tile] = hist[d];
}

__global__ void __launch_bounds__(kSortThreads)
sort_scan(uint32_t* __restrict__ counts, uint32_t* __restrict__ totals, int64_t n_host, const int64_t* n_dev,
          const int32_t* bits_dev, int bits_max, int D, int pass, int tile_elems)
{
    PassCtx c = pass_ctx(n_host, n_dev, bits_dev, bits_max, D, pass, tile_elems);
    const int d = blockIdx.x;
    if (!c.active || d >= (1 << D)) return;
    __shared__ uint32_t wbuf[kSortThreads / 32 + 1];
    uint32_t* row = counts + (int64_t)d * c.ntiles;
    uint32_t running = 0;
    constexpr int kPer = 4;
    for (int64_t base = 0; base < c.ntiles; base += (int64_t)kSortThreads * kPer) {
        uint32_t v[kPer];
        uint32_t s = 0;
        const int64_t i0 = base + (int64_t)threadIdx.x * kPer;
#pragma unroll
        for (int q = 0; q < kPer; ++q) {
            v[q] = (i0 + q < c.ntiles) ? row[i0 + q] : 0u;
            s += v[q];
        }
        uint32_t tot;
        uint32_t ex = block_exclusive_sum(s, wbuf, &tot) + running;
#pragma unroll
        for (int q = 0; q < kPer; ++q) {
            if (i0 + q < c.ntiles) row[i0 + q] = ex;
            ex += v[q];
        }
        running += tot;
    }
    if (threadIdx.x == 0) totals[d] = running;
}

template <typename K, int ITEMS>
__global__ void __launch_bounds__(kSortThreads, kDownsweepBlocks)
sort_downsweep(const K* __restrict__ keys_in, const uint32_t* __restrict__ vals_in, K* keys_out,
               uint32_t* vals_out, K* keys_tmp, uint32_t* vals_tmp, int64_t n_host, const int64_t* n_dev,
               const int32_t* bits_dev, int bits_max, int D, int pass, const uint64_t* key_sub,
               const uint32_t* __restrict__ counts, const uint32_t* __restrict__ totals)
{
    constexpr int kTile = kSortThreads * ITEMS;
    PassCtx c = pass_ctx(n_host, n_dev, bits_dev, bits_max, D, pass, kTile);
    const int64_t tile = blockIdx.x;
    if (!c.active || tile >= c.ntiles) return;
    const K* src_k;
    const uint32_t* src_v;
    K* dst_k;
    uint32_t* dst_v;
    if (c.dst_out) { dst_k = keys_out; dst_v = vals_out; } else { dst_k = keys_tmp; dst_v = vals_tmp; }
    if (c.src_in) { src_k = keys_in; src_v = vals_in; }
    else if (c.dst_out) { src_k = keys_tmp; src_v = vals_tmp; }
    else { src_k = keys_out; src_v = vals_out; }

    constexpr int kWarps = kSortThreads / 32;
    const int nb = 1 << D;
    extern __shared__ __align__(16) unsigned char smem_raw[];
    K* skey = reinterpret_cast<K*>(smem_raw);
    uint32_t* sval = reinterpret_cast<uint32_t*>(skey + kTile);
    uint32_t* wcnt = sval + kTile;                // [kWarps][nb]
    uint32_t* tstart = wcnt + kWarps * nb;        // [nb]
    uint32_t* gbase = tstart + nb;                // [nb]
    uint32_t* wbuf = gbase + nb;                  // [kWarps + 1]

    for (int i = threadIdx.x; i < kWarps * nb; i += kSortThreads) wcnt[i] = 0;
    __syncthreads();

    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const int shift = pass * D;
    const K sub = (c.src_in && key_sub) ? (K)(*key_sub) : (K)0;
    const int64_t base = tile * kTile;
    const uint32_t lt = lanemask_lt();
    // this thread's digits d0 .. d0+per-1 in the scans below: their totals and
    // this tile's offsets within them are requested now, so the loads' latency
    // passes behind the ranking
    const int per = (nb + kSortThreads - 1) / kSortThreads;   // at most 4 (digits of at most 10 bits)
    const int d0 = threadIdx.x * per;
    uint32_t lg_[4], lc_[4];
#pragma unroll
    for (int q = 0; q < 4; ++q) {
        lg_[q] = 0u;
        lc_[q] = 0u;
        if (q < per && d0 + q < nb) {
            lg_[q] = totals[d0 + q];
            lc_[q] = counts[(int64_t)(d0 + q) * c.ntiles + tile];
        }
    }

    K k[ITEMS];
    uint32_t v[ITEMS];
    uint32_t dg[ITEMS];
    uint32_t rk[ITEMS];
#pragma unroll
    for (int r = 0; r < ITEMS; ++r) {
        const int e = warp * (ITEMS * 32) + r * 32 + lane;
        const int64_t idx = base + e;
        dg[r] = (uint32_t)nb;
        k[r] = 0;
        v[r] = 0;
        if (idx < c.n) {
            k[r] = (K)(src_k[idx] - sub);
            v[r] = src_v ? src_v[idx] : (uint32_t)idx;
            dg[r] = (uint32_t)((k[r] >> shift) & (K)(nb - 1));
        }
    }
#pragma unroll
    for (int r = 0; r < ITEMS; ++r) {
        uint32_t peers = __match_any_sync(0xffffffffu, dg[r]);
        int leader = __ffs(peers) - 1;
        uint32_t old = 0;
        if (lane == leader && dg[r] < (uint32_t)nb) {
            old = wcnt[warp * nb + dg[r]];
            wcnt[warp * nb + dg[r]] = old + (uint32_t)__popc(peers);
        }
        old = __shfl_sync(0xffffffffu, old, leader);
        rk[r] = old + (uint32_t)__popc(peers & lt);
        __syncwarp();
    }
    __syncthreads();
    // per digit: exclusive prefix over warps and the tile total
    for (int d = threadIdx.x; d < nb; d += kSortThreads) {
        uint32_t s = 0;
#pragma unroll
        for (int w = 0; w < kWarps; ++w) {
            uint32_t cnt = wcnt[w * nb + d];
            wcnt[w * nb + d] = s;
            s += cnt;
        }
        tstart[d] = s;
    }
    __syncthreads();
    // exclusive scans over digits: tile-local starts and global digit bases
    {
        uint32_t st = 0, sg = 0;
        uint32_t lt_[4];
#pragma unroll
        for (int q = 0; q < 4; ++q) {
            lt_[q] = (q < per && d0 + q < nb) ? tstart[d0 + q] : 0u;
            st += lt_[q];
            sg += lg_[q];
        }
        uint32_t ext = block_exclusive_sum(st, wbuf, nullptr);
        uint32_t exg = block_exclusive_sum(sg, wbuf, nullptr);
#pragma unroll
        for (int q = 0; q < 4; ++q) {
            if (q < per && d0 + q < nb) {
                tstart[d0 + q] = ext;
                gbase[d0 + q] = exg + lc_[q];
            }
            ext += lt_[q];
            exg += lg_[q];
        }
    }
    __syncthreads();
#pragma unroll
    for (int r = 0; r < ITEMS; ++r) {
        if (dg[r] < (uint32_t)nb) {
            uint32_t lp = tstart[dg[r]] + wcnt[warp * nb + dg[r]] + rk[r];
            skey[lp] = k[r];
            sval[lp] = v[r];
        }
    }
    __syncthreads();
    const int64_t rem = c.n - base;
    const int nvalid = rem < kTile ? (int)rem : kTile;
#pragma unroll 4
    for (int r = 0; r < ITEMS; ++r) {
        const int p = r * kSortThreads + threadIdx.x;
        if (p < nvalid) {
            K kk = skey[p];
            uint32_t d = (uint32_t)((kk >> shift) & (K)(nb - 1));
            int64_t o = (int64_t)gbase[d] + (p - (int64_t)tstart[d]);
            dst_k[o] = kk;
            dst_v[o] = sval[p];
        }
    }
}

}  // namespace

SortPlan make_sort_plan(int64_t n_max, int bits_max)
{
    SortPlan p;
    if (bits_max < 1) bits_max = 1;
    p.n_max = n_max;
    p.bits_max = bits_max;
    p.passes_max = (bits_max + kMaxDigitBits - 1) / kMaxDigitBits;
    p.digit_bits = (bits_max + p.passes_max - 1) / p.passes_max;
    p.tiles_max = (n_max + kSortThreads * kSortItems - 1) / (kSortThreads * kSortItems);
    if (p.tiles_max < 1) p.tiles_max = 1;
    p.counts_bytes = sizeof(uint32_t) * ((size_t)1 << p.digit_bits) * (size_t)p.tiles_max;
    p.totals_bytes = sizeof(uint32_t) * ((size_t)1 << p.digit_bits);
    return p;
}

template <typename K, int ITEMS>
static size_t downsweep_smem(int D)
{
    const int nb = 1 << D;
    return (size_t)kSortThreads * ITEMS * (sizeof(K) + sizeof(uint32_t)) +
           sizeof(uint32_t) * ((size_t)(kSortThreads / 32) * nb + 2 * (size_t)nb + kSortThreads / 32 + 1);
}

template <typename K, int ITEMS>
static int sort_passes_3k(const SortPlan& plan, const K* keys_in, const uint32_t* vals_in, K* keys_out,
                          uint32_t* vals_out, K* keys_tmp, uint32_t* vals_tmp, uint32_t* counts, uint32_t* totals,
                          int64_t n_host, const int64_t* n_dev, const int32_t* bits_dev, const uint64_t* key_sub,
                          cudaStream_t st)
{
    constexpr int kTile = kSortThreads * ITEMS;
    const int D = plan.digit_bits;
    const int64_t tiles = (n_host + kTile - 1) / kTile;
    const size_t smem = downsweep_smem<K, ITEMS>(D);
    if (cudaFuncSetAttribute(sort_downsweep<K, ITEMS>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem) !=
        cudaSuccess)
        return -1;
    int launched = 0;
    for (int p = 0; p < plan.passes_max; ++p) {
        sort_upsweep<K, ITEMS><<<(unsigned)tiles, kSortThreads, 0, st>>>(keys_in, keys_out, keys_tmp, n_host, n_dev,
                                                                         bits_dev, plan.bits_max, D, p, key_sub,
                                                                         counts);
        sort_scan<<<1u << D, kSortThreads, 0, st>>>(counts, totals, n_host, n_dev, bits_dev, plan.bits_max, D, p,
                                                    kTile);
        sort_downsweep<K, ITEMS><<<(unsigned)tiles, kSortThreads, smem, st>>>(
            keys_in, vals_in, keys_out, vals_out, keys_tmp, vals_tmp, n_host, n_dev, bits_dev, plan.bits_max, D,
            p, key_sub, counts, totals);
        launched += 3;
    }
    if (cudaGetLastError() != cudaSuccess) return -1;
    return launched;
}

template <typename K>
int radix_sort_pairs(const SortPlan& plan, const K* keys_in, const uint32_t* vals_in, K* keys_out,
                     uint32_t* vals_out, K* keys_tmp, uint32_t* vals_tmp, uint32_t* counts, uint32_t* totals,
                     int64_t n_host, const int64_t* n_dev, const int32_t* bits_dev, const uint64_t* key_sub,
                     cudaStream_t st)
{
    if (n_host <= 0) return 0;
    return sort_passes_3k<K, kSortItems>(plan, keys_in, vals_in, keys_out, vals_out, keys_tmp, vals_tmp, counts,
                                         totals, n_host, n_dev, bits_dev, key_sub, st);
}

template int radix_sort_pairs<uint32_t>(const SortPlan&, const uint32_t*, const uint32_t*, uint32_t*, uint32_t*,
                                        uint32_t*, uint32_t*, uint32_t*, uint32_t*, int64_t, const int64_t*,
                                        const int32_t*, const uint64_t*, cudaStream_t);
template int radix_sort_pairs<uint64_t>(const SortPlan&, const uint64_t*, const uint32_t*, uint64_t*, uint32_t*,
                                        uint64_t*, uint32_t*, uint32_t*, uint32_t*, int64_t, const int64_t*,
                                        const int32_t*, const uint64_t*, cudaStream_t);

// ---------------------------------------------------------------------------
// run-length encoding of sorted keys
// ---------------------------------------------------------------------------
namespace {

template <typename K>
__device__ __forceinline__ bool is_head(const K* sk, int64_t p, uint64_t key_max)
{
    K k = sk[p];
    if ((uint64_t)k > key_max) return false;
    return p == 0 || sk[p - 1] != k;
}

template <typename K>
__global__ void __launch_bounds__(kRleThreads)
rle_count(const K* __restrict__ sk, int64_t n, uint64_t key_max, uint32_t* __restrict__ tile_cnt)
{
    __shared__ uint32_t wbuf[kRleThreads / 32 + 1];
    const int64_t base = (int64_t)blockIdx.x * kRleTile + (int64_t)threadIdx.x * kRleItems;
    uint32_t c = 0;
    for (int q = 0; q < kRleItems; ++q) {
        int64_t p = base + q;
        if (p < n && is_head(sk, p, key_max)) ++c;
    }
    uint32_t tot;
    block_exclusive_sum(c, wbuf, &tot);
    if (threadIdx.x == 0) tile_cnt[blockIdx.x] = tot;
}

__global__ void __launch_bounds__(kRleThreads)
rle_scan(uint32_t* __restrict__ tile_cnt, int64_t ntiles, int64_t n, int32_t* __restrict__ seg_off,
         int64_t* __restrict__ num_unique, const int* err)
{
    __shared__ uint32_t wbuf[kRleThreads / 32 + 1];
    uint32_t running = 0;
    constexpr int kPer = 8;
    for (int64_t b = 0; b < ntiles; b += (int64_t)kRleThreads * kPer) {
        uint32_t v[kPer], s = 0;
        const int64_t i0 = b + (int64_t)threadIdx.x * kPer;
        for (int q = 0; q < kPer; ++q) {
            v[q] = (i0 + q < ntiles) ? tile_cnt[i0 + q] : 0u;
            s += v[q];
        }
        uint32_t tot;
        uint32_t ex = block_exclusive_sum(s, wbuf, &tot) + running;
        for (int q = 0; q < kPer; ++q) {
            if (i0 + q < ntiles) tile_cnt[i0 + q] = ex;
            ex += v[q];
        }
        running += tot;
    }
    if (threadIdx.x == 0) {
        *num_unique = running;
        seg_off[running] = (int32_t)n;   // overwritten by rle_write when keys > key_max exist
    }
    if (err && *err) {                   // the sort behind these keys failed: report no result
        __syncthreads();
        if (threadIdx.x == 0) *num_unique = -1;
    }
}

template <typename K>
__global__ void __launch_bounds__(kRleThreads)
rle_write(const K* __restrict__ sk, const uint32_t* __restrict__ vals, int64_t n, uint64_t key_max,
          const uint64_t* key_add, const uint32_t* __restrict__ tile_base, const int64_t* __restrict__ num_unique,
          int64_t* unique64, uint32_t* unique32, int32_t* seg_off, int32_t* inverse)
{
    __shared__ uint32_t wbuf[kRleThreads / 32 + 1];
    if (*num_unique < 0) return;   // the sort behind these keys failed: nothing is written
    const int64_t base = (int64_t)blockIdx.x * kRleTile + (int64_t)threadIdx.x * kRleItems;
    bool h[kRleItems];
    uint32_t c = 0;
    for (int q = 0; q < kRleItems; ++q) {
        int64_t p = base + q;
        h[q] = p < n && is_head(sk, p, key_max);
        c += h[q];
    }
    uint32_t s = block_exclusive_sum(c, wbuf, nullptr) + tile_base[blockIdx.x];
    const uint64_t add = key_add ? *key_add : 0ull;
    const uint32_t U = (uint32_t)*num_unique;
    // s counts heads strictly before this thread's first element; the run of
    // element p is (heads up to and including p) - 1.
    uint32_t run = s;  // heads seen so far (global)
    for (int q = 0; q < kRleItems; ++q) {
        int64_t p = base + q;
        if (p >= n) break;
        K k = sk[p];
        bool valid = (uint64_t)k <= key_max;
        if (h[q]) {
            if (unique64) unique64[run] = (int64_t)((uint64_t)k + add);
            if (unique32) unique32[run] = (uint32_t)k;
            seg_off[run] = (int32_t)p;
            ++run;
        }
        if (!valid && (p == 0 || (uint64_t)sk[p - 1] <= key_max)) seg_off[U] = (int32_t)p;
        if (inverse) inverse[vals ? vals[p] : (uint32_t)p] = valid ? (int32_t)(run - 1) : (int32_t)U;
    }
}

__global__ void rle_counts(const int32_t* __restrict__ seg_off, const int64_t* __restrict__ num_unique,
                           int64_t n_max, int32_t* __restrict__ counts)
{
    const int64_t U = *num_unique;
    for (int64_t s = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; s < U && s < n_max;
         s += (int64_t)gridDim.x * blockDim.x)
        counts[s] = seg_off[s + 1] - seg_off[s];
}

}  // namespace

size_t rle_scratch_bytes(int64_t n_max)
{
    int64_t tiles = (n_max + kRleTile - 1) / kRleTile;
    if (tiles < 1) tiles = 1;
    return (size_t)tiles * sizeof(uint32_t);
}

template <typename K>
int rle_sorted(const K* sk, const uint32_t* vals, int64_t n, uint64_t key_max, const uint64_t* key_add,
               int64_t* unique64, uint32_t* unique32, int32_t* seg_off, int32_t* counts, int32_t* inverse,
               int64_t* num_unique, void* scratch, const int* err, cudaStream_t st)
{
    if (n <= 0) {
        if (cudaMemsetAsync(num_unique, 0, sizeof(int64_t), st) != cudaSuccess) return -1;
        if (cudaMemsetAsync(seg_off, 0, sizeof(int32_t), st) != cudaSuccess) return -1;
        return 0;
    }
    const int64_t tiles = (n + kRleTile - 1) / kRleTile;
    uint32_t* tile_cnt = static_cast<uint32_t*>(scratch);
    rle_count<K><<<(unsigned)tiles, kRleThreads, 0, st>>>(sk, n, key_max, tile_cnt);
    rle_scan<<<1, kRleThreads, 0, st>>>(tile_cnt, tiles, n, seg_off, num_unique, err);
    rle_write<K><<<(unsigned)tiles, kRleThreads, 0, st>>>(sk, vals, n, key_max, key_add, tile_cnt, num_unique,
                                                          unique64, unique32, seg_off, inverse);
    int launched = 3;
    if (counts) {
        int blocks = (int)((n + 255) / 256);
        if (blocks > 4096) blocks = 4096;
        rle_counts<<<blocks, 256, 0, st>>>(seg_off, num_unique, n, counts);
        ++launched;
    }
    if (cudaGetLastError() != cudaSuccess) return -1;
    return launched;
}

template int rle_sorted<uint32_t>(const uint32_t*, const uint32_t*, int64_t, uint64_t, const uint64_t*, int64_t*,
                                  uint32_t*, int32_t*, int32_t*, int32_t*, int64_t*, void*, const int*, cudaStream_t);
template int rle_sorted<uint64_t>(const uint64_t*, const uint32_t*, int64_t, uint64_t, const uint64_t*, int64_t*,
                                  uint32_t*, int32_t*, int32_t*, int32_t*, int64_t*, void*, const int*, cudaStream_t);

}  // namespace emb
