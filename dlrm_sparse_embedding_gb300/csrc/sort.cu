// Stable LSD radix sort of (key, u32 value) pairs and run-length encoding of
// sorted keys -- the sort-based dedup behind the reduction-based and the
// unique-based backward ("NVIDIA EMBark revoluciona la formacion en sistemas
// de recomendacion a escala", section "Integracion del cluster": RB reduces
// over equal keys, UB dedups the keys first).
//
// The input may be cut into segments that are sorted independently and stay
// in place.  The layer's sort uses one segment per table: the forward emits
// each table's lookups contiguously, so sorting every table's segment on the
// row id local to the table (row - row_base) sorts the global ids, with as
// few digit passes as the largest table needs instead of the sum of all
// tables' rows.  Skipped lookups (the sentinel id) take the all-ones local key
// and the last pass moves them behind every valid id, so the output is
// exactly the ascending sort of the global ids.
//
// Each pass runs over 3072-key tiles that never cross a segment: a per-tile
// digit histogram (u16 counts, one contiguous row per tile), a scan of the
// counts over groups of 16 tiles, a scan over each segment's groups that also
// adds the segment's exclusive digit bases, and the stable in-tile ranking in
// shared memory, whose coalesced runs go to segment start + digit base +
// group offset + tile offset.  No tile waits on another.  The element count
// and the number of significant key bits may live on the device (the
// unique-based path only learns them there); passes beyond the significant
// bits return at once, and the buffers are chosen so the last active pass
// always writes the output.  The histogram and ranking kernels are also
// built with the digit count fixed (256 or 1024 digits), and the ranking
// kernel with the pass's role fixed (first, middle, last, only) where the
// host knows the number of passes.
#include "emb_internal.cuh"

namespace emb {

namespace {

__device__ __forceinline__ uint32_t lanemask_lt()
{
    uint32_t m;
    asm("mov.u32 %0, %%lanemask_lt;" : "=r"(m));
    return m;
}

// Exclusive sum over the block (blockDim.x == NT); `total` gets the sum.
template <int NT>
__device__ __forceinline__ uint32_t block_exclusive_sum(uint32_t x, uint32_t* warp_buf, uint32_t* total)
{
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    constexpr int kWarps = NT / 32;
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

// Scratch of one sort (layout from sort_scratch_layout).
struct SortScratch {
    int64_t* seg_lo;        // [S] first position of each segment
    int64_t* seg_len;       // [S]
    int32_t* seg_tile0;     // [S+1] first tile of each segment; [S] = tiles in use
    int32_t* seg_grp0;      // [S+1] first group of each segment; [S] = groups in use
    uint32_t* skipcnt;      // [S] skipped ids per segment (last pass of the layer sort)
    uint32_t* skippre;      // [S+1] their exclusive prefix; [S] = total
    uint16_t* counts;       // [tiles][nb] per-tile digit counts, then in-group exclusive offsets
    uint32_t* gsum;         // [groups][nb] per-group sums, then group offsets + segment digit bases
    int4* tile_desc;        // [tiles] first position, length, segment, group of each tile in use
    int4* grp_desc;         // [groups] first tile, tiles, segment of each group in use
    uint32_t* segtot;       // [S][nb] the segments' digit totals, then their exclusive digit bases
};

// The per-pass context every kernel derives the same way from the device or
// host element count and significant bits.
struct PassCtx {
    int64_t n;
    int npe;       // effective passes
    bool active;
    bool last;     // the last effective pass
    bool dst_out;  // this pass writes the output buffers
    bool src_in;   // this pass reads the input buffers
};

__device__ __forceinline__ PassCtx pass_ctx(const SortArgs& a, int pass)
{
    PassCtx c;
    int64_t n = a.n_host;
    if (a.n_dev) {
        const int64_t m = *a.n_dev;
        n = m < a.n_host ? (m < 0 ? 0 : m) : a.n_host;
    }
    c.n = n;
    int b = a.bits_dev ? *a.bits_dev : a.bits_max;
    if (b < 1) b = 1;
    if (b > a.bits_max) b = a.bits_max;
    c.npe = (b + a.D - 1) / a.D;
    c.active = pass < c.npe && n > 0;
    c.last = pass == c.npe - 1;
    c.dst_out = ((c.npe - 1 - pass) & 1) == 0;
    c.src_in = pass == 0;
    return c;
}

// Segment s holding tile (or group) index x of the prefix array p[0..S]: the s
// with p[s] <= x < p[s+1] (empty segments skipped).
__device__ __forceinline__ int find_seg(const int32_t* p, int S, int64_t x)
{
    int lo = 0, hi = S - 1;
    while (lo < hi) {
        const int mid = (lo + hi + 1) >> 1;
        if (p[mid] <= x) lo = mid; else hi = mid - 1;
    }
    return lo;
}

// The key a pass ranks: the input key, made local to its segment on the
// first pass of the layer sort (all ones for a skipped or out-of-table id),
// or with key_sub subtracted on the first pass of a plain sort.  The
// segment's table fields are read once per tile (FirstPass) and applied to
// each of its keys.
struct FirstPass {
    uint32_t rb;      // the segment table's first global row
    uint64_t rows;    // its rows
    uint64_t sub;     // plain sort: subtracted from every key
};

__device__ __forceinline__ FirstPass first_pass_of(const SortArgs& a, int s, uint64_t sub)
{
    FirstPass f;
    f.rb = a.tables ? a.tables[s].row_base : 0u;
    f.rows = a.tables ? (uint64_t)a.tables[s].rows : 0ull;
    f.sub = sub;
    return f;
}

template <typename K>
__device__ __forceinline__ K first_pass_key(const SortArgs& a, K k, const FirstPass& f)
{
    if (a.tables) {
        const uint32_t g = (uint32_t)k;
        const uint64_t local = (uint64_t)g - f.rb;
        return (g < a.sentinel && g >= f.rb && local < f.rows) ? (K)local : (K)a.skip_key;
    }
    return (K)(k - (K)f.sub);
}

// ---- segment and tile layout (one block) ----
constexpr int kSetupThreads = 1024;

__global__ void __launch_bounds__(kSetupThreads) sort_setup(SortArgs a, SortScratch sc)
{
    __shared__ uint32_t wbuf[kSetupThreads / 32 + 1];
    __shared__ int64_t wmax[kSetupThreads / 32];
    int64_t n = a.n_host;
    if (a.n_dev) {
        const int64_t m = *a.n_dev;
        n = m < a.n_host ? (m < 0 ? 0 : m) : a.n_host;
    }
    const int S = a.num_seg;
    const int per = (S + kSetupThreads - 1) / kSetupThreads;   // at most 4 (S <= 4096)
    const int s0 = threadIdx.x * per;
    // segment ends: the clamped offsets made non-decreasing (running maximum),
    // the last one n, so the segments tile [0, n) exactly
    int64_t hi[4];
    int64_t run = 0;
#pragma unroll
    for (int q = 0; q < 4; ++q) {
        const int s = s0 + q;
        hi[q] = 0;
        if (q < per && s < S) {
            int64_t e = n;
            if (a.offsets && s + 1 < S) {
                e = a.offsets[(int64_t)(s + 1) * a.stride];
                e = e < 0 ? 0 : (e > n ? n : e);
            }
            run = e > run ? e : run;
            hi[q] = run;
        }
    }
    // exclusive running maximum over threads
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    int64_t inc = run;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const int64_t y = __shfl_up_sync(0xffffffffu, inc, o);
        if (lane >= o && y > inc) inc = y;
    }
    if (lane == 31) wmax[warp] = inc;
    __syncthreads();
    int64_t before = __shfl_up_sync(0xffffffffu, inc, 1);
    if (lane == 0) before = 0;
    for (int w = 0; w < warp; ++w) before = wmax[w] > before ? wmax[w] : before;
    uint32_t nt = 0, ng = 0;
    int64_t lo = before;
    uint32_t tl[4], gl[4];
#pragma unroll
    for (int q = 0; q < 4; ++q) {
        const int s = s0 + q;
        tl[q] = gl[q] = 0;
        if (q < per && s < S) {
            const int64_t h = hi[q] > lo ? hi[q] : lo;
            sc.seg_lo[s] = lo;
            sc.seg_len[s] = h - lo;
            tl[q] = (uint32_t)((h - lo + kSortTile - 1) / kSortTile);
            gl[q] = (tl[q] + kSortGroupTiles - 1) / kSortGroupTiles;
            nt += tl[q];
            ng += gl[q];
            lo = h;
        }
    }
    uint32_t tot_t, tot_g;
    uint32_t et = block_exclusive_sum<kSetupThreads>(nt, wbuf, &tot_t);
    uint32_t eg = block_exclusive_sum<kSetupThreads>(ng, wbuf, &tot_g);
#pragma unroll
    for (int q = 0; q < 4; ++q) {
        const int s = s0 + q;
        if (q < per && s < S) {
            sc.seg_tile0[s] = (int32_t)et;
            sc.seg_grp0[s] = (int32_t)eg;
            et += tl[q];
            eg += gl[q];
        }
    }
    if (threadIdx.x == 0) {
        sc.seg_tile0[S] = (int32_t)tot_t;
        sc.seg_grp0[S] = (int32_t)tot_g;
    }
}

// ---- one pass: histogram per tile, scans, ranking ----

constexpr int kDownsweepBlocks = 2;   // resident (persistent) blocks per SM of the ranking kernel
constexpr int kDownThreads = 256;      // ranking block: 8 warps ...
constexpr int kDownItems = kSortTile / kDownThreads;   // ... of 12 items each per tile
static_assert(kDownItems * kDownThreads == kSortTile, "the ranking block covers one tile");

// Shared memory of the ranking kernel: the per-warp digit masks (all zero
// between ranking steps), the tile's keys and values in their in-tile sorted
// order followed by the block scans' warp sums, then per-digit starts, bases
// and per-warp counters.
__host__ __device__ __forceinline__ size_t sort_masks_bytes(int nb)
{
    return sizeof(uint32_t) * (size_t)(kDownThreads / 32) * (size_t)nb;
}

__host__ __device__ __forceinline__ size_t sort_tile_bytes(size_t key_bytes)
{
    return ((size_t)kSortTile * (key_bytes + sizeof(uint32_t)) + 15) & ~size_t(15);
}

__host__ __device__ __forceinline__ size_t sort_region0_bytes(size_t key_bytes, int nb)
{
    return sort_masks_bytes(nb) + sort_tile_bytes(key_bytes) + 128;   // + the warp sums (kDownThreads / 32 + 1 words)
}


// Where every tile and group in use lies, one thread per tile (the segment of
// a tile is a binary search over the segments' first tiles).
__global__ void sort_tiles(SortArgs a, SortScratch sc, int64_t tiles_grid)
{
    const int S = a.num_seg;
    const int64_t ntiles = sc.seg_tile0[S];
    for (int64_t tile = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; tile < ntiles && tile < tiles_grid;
         tile += (int64_t)gridDim.x * blockDim.x) {
        const int s = find_seg(sc.seg_tile0, S, tile);
        const int64_t k = tile - sc.seg_tile0[s];
        const int64_t start = sc.seg_lo[s] + k * (int64_t)kSortTile;
        const int64_t rem = sc.seg_lo[s] + sc.seg_len[s] - start;
        const int grp = sc.seg_grp0[s] + (int)(k / kSortGroupTiles);
        sc.tile_desc[tile] = make_int4((int)start, rem < kSortTile ? (int)rem : kSortTile, s, grp);
        if (k % kSortGroupTiles == 0) {
            const int64_t left = sc.seg_tile0[s + 1] - tile;
            sc.grp_desc[grp] = make_int4((int)tile, left < kSortGroupTiles ? (int)left : kSortGroupTiles, s, 0);
        }
    }
}

// Where tile `tile` lies: its segment, first position and element count.
struct TileLoc {
    int s;
    int grp;
    int start;   // positions fit in 32 bits (fewer than 2^31 elements)
    int len;
};

__device__ __forceinline__ TileLoc locate_tile(const SortScratch& sc, int64_t tile)
{
    const int4 d = sc.tile_desc[tile];
    TileLoc t;
    t.start = d.x;
    t.len = d.y;
    t.s = d.z;
    t.grp = d.w;
    return t;
}

// NB: the digit count when fixed at compile time (256 or 1024, the digit
// widths of the common key sizes), 0 when read from the arguments.
template <typename K, int NB>
__global__ void __launch_bounds__(kSortThreads) sort_upsweep(SortArgs a, SortScratch sc, int pass)
{
    PassCtx c = pass_ctx(a, pass);
    const int64_t tile = blockIdx.x;
    if (!c.active || tile >= sc.seg_tile0[a.num_seg]) return;
    __shared__ uint32_t hist[1 << kMaxDigitBits];
    const int nb = NB > 0 ? NB : 1 << a.D;
    for (int i = threadIdx.x; i < nb; i += kSortThreads) hist[i] = 0;
    const TileLoc tl = locate_tile(sc, tile);
    __syncthreads();
    const K* src = c.src_in ? static_cast<const K*>(a.keys_in)
                            : (c.dst_out ? static_cast<const K*>(a.keys_tmp) : static_cast<const K*>(a.keys_out));
    const int shift = pass * a.D;
    const uint64_t sub = (c.src_in && a.key_sub) ? *a.key_sub : 0ull;
    const FirstPass fp = c.src_in ? first_pass_of(a, tl.s, sub) : FirstPass{0u, 0ull, 0ull};
    // all of the thread's keys are requested before the first is counted
    uint32_t dg[kSortItems];
#pragma unroll
    for (int r = 0; r < kSortItems; ++r) {
        const int e = r * kSortThreads + threadIdx.x;
        dg[r] = (uint32_t)nb;
        if (e < tl.len) {
            K k = src[tl.start + e];
            if (c.src_in) k = first_pass_key<K>(a, k, fp);
            dg[r] = (uint32_t)((k >> shift) & (K)(nb - 1));
        }
    }
    // shared-memory atomics are cheap even where many lanes hit one digit
#pragma unroll
    for (int r = 0; r < kSortItems; ++r)
        if (dg[r] < (uint32_t)nb) atomicAdd(&hist[dg[r]], 1u);
    __syncthreads();
    uint16_t* row = sc.counts + tile * (int64_t)nb;
    for (int d = threadIdx.x; d < nb; d += kSortThreads) row[d] = (uint16_t)hist[d];
}

// Per group of up to kSortGroupTiles tiles of one segment: each tile's count
// becomes its exclusive offset within the group; gsum gets the group's sums.
__global__ void __launch_bounds__(kSortThreads) sort_scan_groups(SortArgs a, SortScratch sc, int pass)
{
    PassCtx c = pass_ctx(a, pass);
    const int64_t grp = blockIdx.x;
    if (!c.active || grp >= sc.seg_grp0[a.num_seg]) return;
    const int4 gd = sc.grp_desc[grp];
    const int64_t t0 = gd.x;
    const int nt = gd.y;
    const int nb = 1 << a.D;
    for (int d = threadIdx.x; d < nb; d += kSortThreads) {
        uint32_t v[kSortGroupTiles];
#pragma unroll
        for (int q = 0; q < kSortGroupTiles; ++q) v[q] = q < nt ? sc.counts[(t0 + q) * nb + d] : 0u;
        uint32_t run = 0;
#pragma unroll
        for (int q = 0; q < kSortGroupTiles; ++q) {
            if (q < nt) sc.counts[(t0 + q) * nb + d] = (uint16_t)run;
            run += v[q];
        }
        sc.gsum[grp * nb + d] = run;
    }
}

// The segments' scans, in three steps that each run in parallel:
//  1. per segment and slice of 32 digits: each group's sum becomes its
//     exclusive offset within the segment (8 warps take consecutive runs of
//     the segment's groups, lane = digit), and the segment's digit totals go
//     to segtot;
//  2. per segment: the totals become the segment's exclusive digit bases; on
//     the last pass of the layer sort the segment's count of skipped ids (the
//     all-ones top digit) is recorded;
//  3. per group: the segment's digit bases are added to the group offsets.
constexpr int kScanWarps = 8;

__global__ void __launch_bounds__(kScanWarps * 32) sort_scan_segments(SortArgs a, SortScratch sc, int pass)
{
    PassCtx c = pass_ctx(a, pass);
    const int s = blockIdx.x;
    if (!c.active || s >= a.num_seg) return;
    const int nb = 1 << a.D;
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const int d = blockIdx.y * 32 + lane;
    __shared__ uint32_t wsum[kScanWarps][32];
    const int64_t g0 = sc.seg_grp0[s], g1 = sc.seg_grp0[s + 1];
    const int64_t per = (g1 - g0 + kScanWarps - 1) / kScanWarps;
    const int64_t ga = g0 + warp * per, gb = ga + per < g1 ? ga + per : g1;
    constexpr int kB = 8;   // group sums loaded per batch
    uint32_t run = 0;
    if (d < nb) {
        for (int64_t g = ga; g < gb; g += kB) {
            uint32_t v[kB];
#pragma unroll
            for (int q = 0; q < kB; ++q) v[q] = g + q < gb ? sc.gsum[(g + q) * nb + d] : 0u;
#pragma unroll
            for (int q = 0; q < kB; ++q) run += v[q];
        }
    }
    wsum[warp][lane] = run;
    __syncthreads();
    uint32_t off = 0;
    for (int w = 0; w < warp; ++w) off += wsum[w][lane];
    if (d < nb) {
        for (int64_t g = ga; g < gb; g += kB) {
            uint32_t v[kB];
#pragma unroll
            for (int q = 0; q < kB; ++q) v[q] = g + q < gb ? sc.gsum[(g + q) * nb + d] : 0u;
#pragma unroll
            for (int q = 0; q < kB; ++q) {
                if (g + q < gb) sc.gsum[(g + q) * nb + d] = off;
                off += v[q];
            }
        }
        if (warp == kScanWarps - 1) sc.segtot[(int64_t)s * nb + d] = off;
    }
}

__global__ void __launch_bounds__(1024) sort_seg_bases(SortArgs a, SortScratch sc, int pass)
{
    PassCtx c = pass_ctx(a, pass);
    const int s = blockIdx.x;
    if (!c.active || s >= a.num_seg) return;
    __shared__ uint32_t wbuf[1024 / 32 + 1];
    __shared__ uint32_t skip_base;
    const int nb = 1 << a.D;
    const int d = threadIdx.x;
    uint32_t* tot = sc.segtot + (int64_t)s * nb;
    const uint32_t v = d < nb ? tot[d] : 0u;
    const uint32_t ex = block_exclusive_sum<1024>(v, wbuf, nullptr);
    const uint32_t skipd = (uint32_t)(a.skip_key >> (pass * a.D)) & (uint32_t)(nb - 1);
    if (d < nb) {
        tot[d] = ex;
        // skipped ids carry the largest digit, so everything before its base is valid
        if (a.tables && c.last && (uint32_t)d == skipd) skip_base = ex;
    }
    __syncthreads();
    if (a.tables && c.last && threadIdx.x == 0) sc.skipcnt[s] = (uint32_t)sc.seg_len[s] - skip_base;
}

__global__ void __launch_bounds__(256) sort_add_bases(SortArgs a, SortScratch sc, int pass)
{
    PassCtx c = pass_ctx(a, pass);
    const int64_t grp = blockIdx.x;
    if (!c.active || grp >= sc.seg_grp0[a.num_seg]) return;
    const int nb = 1 << a.D;
    const int s = sc.grp_desc[grp].z;
    const uint32_t* base = sc.segtot + (int64_t)s * nb;
    for (int d = threadIdx.x; d < nb; d += 256) sc.gsum[grp * nb + d] += base[d];
}

// Exclusive prefix of the skipped ids over segments (last pass of the layer sort).
__global__ void __launch_bounds__(kSetupThreads) sort_scan_skips(SortArgs a, SortScratch sc, int pass)
{
    PassCtx c = pass_ctx(a, pass);
    if (!c.active || !c.last) return;
    __shared__ uint32_t wbuf[kSetupThreads / 32 + 1];
    const int S = a.num_seg;
    const int per = (S + kSetupThreads - 1) / kSetupThreads;
    const int s0 = threadIdx.x * per;
    uint32_t v[4], sum = 0;
#pragma unroll
    for (int q = 0; q < 4; ++q) {
        v[q] = (q < per && s0 + q < S) ? sc.skipcnt[s0 + q] : 0u;
        sum += v[q];
    }
    uint32_t tot;
    uint32_t ex = block_exclusive_sum<kSetupThreads>(sum, wbuf, &tot);
#pragma unroll
    for (int q = 0; q < 4; ++q) {
        if (q < per && s0 + q < S) sc.skippre[s0 + q] = ex;
        ex += v[q];
    }
    if (threadIdx.x == 0) sc.skippre[S] = tot;
}

// A tile's items as the ranking kernel holds them: thread x holds elements
// warp * (kDownItems * 32) + r * 32 + lane (r < kDownItems).
template <typename K>
__device__ __forceinline__ void load_tile_items(const K* src_k, const uint32_t* src_v, const TileLoc& tl, K (&k)[kDownItems],
                                                uint32_t (&v)[kDownItems])
{
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
#pragma unroll
    for (int r = 0; r < kDownItems; ++r) {
        const int e = warp * (kDownItems * 32) + r * 32 + lane;
        k[r] = 0;
        v[r] = 0;
        if (e < tl.len) {
            const uint32_t idx = (uint32_t)(tl.start + e);
            k[r] = src_k[idx];
            v[r] = src_v ? src_v[idx] : (uint32_t)idx;
        }
    }
}

// The ranking pass.  Persistent blocks walk the tiles (tile, tile + grid,
// ...); while a tile is ranked and scattered, the next tile's items are
// already requested (its descriptor one tile earlier still), so the load
// latency hides behind the work.
template <typename K, int NB, int kRole>
__global__ void __launch_bounds__(kDownThreads, kDownsweepBlocks) sort_downsweep(SortArgs a, SortScratch sc, int pass)
{
    PassCtx c = pass_ctx(a, pass);
    // kRole, when the host knows the number of passes: 1 first of several,
    // 2 a middle pass, 3 the last of several, 4 the only pass (0: read from c)
    if constexpr (kRole != 0) {
        c.src_in = kRole == 1 || kRole == 4;
        c.last = kRole == 3 || kRole == 4;
    }
    const int64_t ntiles = sc.seg_tile0[a.num_seg];
    int64_t tile = blockIdx.x;
    if (!c.active || tile >= ntiles) return;
    const K* src_k;
    const uint32_t* src_v;
    K* dst_k;
    uint32_t* dst_v;
    if (c.dst_out) { dst_k = static_cast<K*>(a.keys_out); dst_v = a.vals_out; }
    else { dst_k = static_cast<K*>(a.keys_tmp); dst_v = a.vals_tmp; }
    if (c.src_in) { src_k = static_cast<const K*>(a.keys_in); src_v = a.vals_in; }
    else if (c.dst_out) { src_k = static_cast<const K*>(a.keys_tmp); src_v = a.vals_tmp; }
    else { src_k = static_cast<const K*>(a.keys_out); src_v = a.vals_out; }

    constexpr int kWarps = kDownThreads / 32;
    const int nb = NB > 0 ? NB : 1 << a.D;
    extern __shared__ __align__(16) unsigned char smem_raw[];
    // the per-warp lane masks of each digit (zero between ranking steps), then
    // the tile's keys and values in their in-tile sorted order
    uint32_t* wmask = reinterpret_cast<uint32_t*>(smem_raw);   // [kWarps][nb]
    unsigned char* stage = smem_raw + sort_masks_bytes(nb);
    // 32-bit keys travel with their values as one 8-byte pair
    K* skey = reinterpret_cast<K*>(stage);
    uint32_t* sval = reinterpret_cast<uint32_t*>(skey + kSortTile);
    uint2* spair = reinterpret_cast<uint2*>(stage);
    unsigned char* region1 = smem_raw + sort_region0_bytes(sizeof(K), nb);
    uint32_t* wbuf = reinterpret_cast<uint32_t*>(stage + sort_tile_bytes(sizeof(K)));   // [kWarps + 1]
    uint32_t* tstart = reinterpret_cast<uint32_t*>(region1);   // [nb]
    uint32_t* gbase = tstart + nb;                // [nb]
    // per-warp digit counters: at most 32 * kDownItems per warp, so 16 bits
    uint16_t* wcnt = reinterpret_cast<uint16_t*>(gbase + nb);   // [kWarps][nb]

    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const int shift = pass * a.D;
    const uint64_t sub = (c.src_in && a.key_sub) ? *a.key_sub : 0ull;
    const uint32_t lt = lanemask_lt();
    const int per = (nb + kDownThreads - 1) / kDownThreads;   // at most 4 (digits of at most 10 bits)
    const int d0 = threadIdx.x * per;
    // the last pass of the layer sort puts skipped ids behind all valid ones
    const bool relocate = a.tables && c.last;
    const uint32_t skipd = relocate ? (uint32_t)(a.skip_key >> shift) & (uint32_t)(nb - 1) : 0xFFFFFFFFu;

    // the masks start at zero; each ranking step's lowest lane clears what it set
    for (int i = threadIdx.x; i < kWarps * nb; i += kDownThreads) wmask[i] = 0u;
    TileLoc tl = locate_tile(sc, tile);
    K kr[kDownItems];
    uint32_t vr[kDownItems];
    load_tile_items<K>(src_k, src_v, tl, kr, vr);
    int64_t next = tile + gridDim.x;
    TileLoc tn = next < ntiles ? locate_tile(sc, next) : tl;
    for (;;) {
        // where this tile's digits go (segment start + digit base + group
        // offset + tile offset), requested now and used after the ranking
        uint32_t gb_[4];
#pragma unroll
        for (int q = 0; q < 4; ++q) {
            gb_[q] = 0u;
            if (q < per && d0 + q < nb)
                gb_[q] = sc.gsum[(int64_t)tl.grp * nb + d0 + q] + (uint32_t)sc.counts[tile * nb + d0 + q];
        }
        uint32_t seg_base = (uint32_t)sc.seg_lo[tl.s];
        uint32_t skip_base = 0, valid_in_seg = 0;
        if (relocate) {
            const uint32_t pre = sc.skippre[tl.s];
            valid_in_seg = (uint32_t)sc.seg_len[tl.s] - sc.skipcnt[tl.s];
            skip_base = (uint32_t)c.n - sc.skippre[a.num_seg] + pre;
            seg_base -= pre;
        }
        // the next tile's items, and the descriptor of the one after it
        K kn[kDownItems];
        uint32_t vn[kDownItems];
        const int64_t after = next + gridDim.x;
        TileLoc ta = tn;
        if (next < ntiles) {
            load_tile_items<K>(src_k, src_v, tn, kn, vn);
            if (after < ntiles) ta = locate_tile(sc, after);
        }

        for (int i = threadIdx.x; i < kWarps * nb / 2; i += kDownThreads) reinterpret_cast<uint32_t*>(wcnt)[i] = 0u;
        const FirstPass fp = c.src_in ? first_pass_of(a, tl.s, sub) : FirstPass{0u, 0ull, 0ull};
        K k[kDownItems];
        uint32_t dg[kDownItems];
        uint32_t rk[kDownItems];
#pragma unroll
        for (int r = 0; r < kDownItems; ++r) {
            const int e = warp * (kDownItems * 32) + r * 32 + lane;
            k[r] = kr[r];
            dg[r] = (uint32_t)nb;
            if (e < tl.len) {
                if (c.src_in) k[r] = first_pass_key<K>(a, k[r], fp);
                dg[r] = (uint32_t)((k[r] >> shift) & (K)(nb - 1));
            }
        }
        __syncthreads();   // the counters are cleared
        // stable rank of each item among the warp's items of its digit: the lanes
        // of one step that share a digit find each other through an atomic OR of
        // their lane bits into the digit's mask; the lowest of them advances the
        // digit's counter and clears the mask
        uint32_t* mymask = wmask + warp * nb;
        uint16_t* mycnt = wcnt + warp * nb;
#pragma unroll
        for (int r = 0; r < kDownItems; ++r) {
            const uint32_t d = dg[r];
            const bool in = d < (uint32_t)nb;
            if (in) atomicOr(mymask + d, 1u << lane);
            __syncwarp();
            uint32_t peers = 0, base = 0;
            if (in) {
                peers = mymask[d];
                base = mycnt[d];
            }
            __syncwarp();
            if (in && lane == __ffs(peers) - 1) {
                mycnt[d] = (uint16_t)(base + (uint32_t)__popc(peers));
                mymask[d] = 0u;
            }
            rk[r] = base + (uint32_t)__popc(peers & lt);
            __syncwarp();
        }
        __syncthreads();
        // per digit: exclusive prefix over warps and the tile total
        for (int d = threadIdx.x; d < nb; d += kDownThreads) {
            uint32_t sum = 0;
#pragma unroll
            for (int w = 0; w < kWarps; ++w) {
                uint32_t cnt = wcnt[w * nb + d];
                wcnt[w * nb + d] = (uint16_t)sum;
                sum += cnt;
            }
            tstart[d] = sum;
        }
        __syncthreads();
        // exclusive scan over digits: tile-local starts; global bases from the scans
        {
            uint32_t st = 0;
            uint32_t lt_[4];
#pragma unroll
            for (int q = 0; q < 4; ++q) {
                lt_[q] = (q < per && d0 + q < nb) ? tstart[d0 + q] : 0u;
                st += lt_[q];
            }
            uint32_t ext = block_exclusive_sum<kDownThreads>(st, wbuf, nullptr);
#pragma unroll
            for (int q = 0; q < 4; ++q) {
                const int d = d0 + q;
                if (q < per && d < nb) {
                    tstart[d] = ext;
                    // where the digit's run starts globally, less its start in the tile
                    gbase[d] = ((uint32_t)d == skipd ? skip_base + (gb_[q] - valid_in_seg) : seg_base + gb_[q]) - ext;
                }
                ext += lt_[q];
            }
        }
        __syncthreads();
#pragma unroll
        for (int r = 0; r < kDownItems; ++r) {
            if (dg[r] < (uint32_t)nb) {
                uint32_t lp = tstart[dg[r]] + wcnt[warp * nb + dg[r]] + rk[r];
                if constexpr (sizeof(K) == 4) {
                    spair[lp] = make_uint2((uint32_t)k[r], vr[r]);
                } else {
                    skey[lp] = k[r];
                    sval[lp] = vr[r];
                }
            }
        }
        __syncthreads();
        const uint32_t rb = a.tables ? a.tables[tl.s].row_base : 0u;
#pragma unroll 4
        for (int r = 0; r < kDownItems; ++r) {
            const int p = r * kDownThreads + threadIdx.x;
            if (p < tl.len) {
                K kk;
                uint32_t vv;
                if constexpr (sizeof(K) == 4) {
                    const uint2 pr = spair[p];
                    kk = (K)pr.x;
                    vv = pr.y;
                } else {
                    kk = skey[p];
                    vv = sval[p];
                }
                const uint32_t d = (uint32_t)((kk >> shift) & (K)(nb - 1));
                // gbase holds (global start - tile start) per digit; positions fit in 32 bits
                const uint32_t o = gbase[d] + (uint32_t)p;
                // the layer sort's last pass writes global ids again
                if (relocate) kk = d == skipd ? (K)a.sentinel : (K)(kk + rb);
                dst_k[o] = kk;
                dst_v[o] = vv;
            }
        }
        if (next >= ntiles) break;
        __syncthreads();   // the shared arrays are reused by the next tile
        tile = next;
        next = after;
        tl = tn;
        tn = ta;
#pragma unroll
        for (int r = 0; r < kDownItems; ++r) {
            kr[r] = kn[r];
            vr[r] = vn[r];
        }
    }
}

// Byte offsets of the scratch arrays inside one region (host and device agree).
struct ScratchLayout {
    size_t seg_lo, seg_len, seg_tile0, seg_grp0, skipcnt, skippre, counts, gsum, tile_desc, grp_desc, segtot, total;
};

ScratchLayout scratch_layout(const SortPlan& p)
{
    ScratchLayout l{};
    size_t off = 0;
    auto take = [&](size_t bytes) {
        const size_t at = off;
        off += (bytes + 255) & ~size_t(255);
        return at;
    };
    const size_t S = (size_t)p.num_seg_max;
    const size_t nb = (size_t)1 << p.digit_bits;
    l.seg_lo = take(8 * S);
    l.seg_len = take(8 * S);
    l.seg_tile0 = take(4 * (S + 1));
    l.seg_grp0 = take(4 * (S + 1));
    l.skipcnt = take(4 * S);
    l.skippre = take(4 * (S + 1));
    l.counts = take(2 * nb * (size_t)p.tiles_max);
    l.gsum = take(4 * nb * (size_t)p.groups_max);
    l.tile_desc = take(16 * (size_t)p.tiles_max);
    l.grp_desc = take(16 * (size_t)p.groups_max);
    l.segtot = take(4 * nb * S);
    l.total = off;
    return l;
}

}  // namespace

SortPlan make_sort_plan(int64_t n_max, int bits_max, int num_seg_max)
{
    SortPlan p;
    if (bits_max < 1) bits_max = 1;
    if (num_seg_max < 1) num_seg_max = 1;
    p.n_max = n_max;
    p.num_seg_max = num_seg_max;
    p.bits_max = bits_max;
    p.passes_max = (bits_max + kMaxDigitBits - 1) / kMaxDigitBits;
    p.digit_bits = (bits_max + p.passes_max - 1) / p.passes_max;
    p.tiles_max = (n_max + kSortTile - 1) / kSortTile + num_seg_max;
    p.groups_max = p.tiles_max / kSortGroupTiles + num_seg_max;
    p.scratch_bytes = scratch_layout(p).total;
    return p;
}

int table_sort_bits(int64_t rows_max)
{
    // local ids 0 .. rows_max - 1 plus the all-ones key of skipped lookups,
    // whose top digit no valid id may share
    int b = 1;
    while (b < 63 && ((uint64_t)rows_max >> b) != 0) ++b;
    for (;; ++b) {
        const int passes = (b + kMaxDigitBits - 1) / kMaxDigitBits;
        const int D = (b + passes - 1) / passes;
        const int top_shift = (passes - 1) * D;
        const uint64_t top_skip = (((uint64_t)1 << b) - 1) >> top_shift;
        if ((((uint64_t)rows_max - 1) >> top_shift) < top_skip) return b;
    }
}

template <typename K>
int radix_sort_pairs(const SortPlan& plan, SortArgs a, void* scratch, cudaStream_t st)
{
    if (a.n_host <= 0) return 0;
    if (a.num_seg < 1 || a.num_seg > plan.num_seg_max || a.n_host > plan.n_max || (a.tables && sizeof(K) != 4))
        return -1;
    a.bits_max = plan.bits_max;
    a.D = plan.digit_bits;
    a.skip_key = ((uint64_t)1 << plan.bits_max) - 1;
    const ScratchLayout l = scratch_layout(plan);
    char* base = static_cast<char*>(scratch);
    SortScratch sc;
    sc.seg_lo = reinterpret_cast<int64_t*>(base + l.seg_lo);
    sc.seg_len = reinterpret_cast<int64_t*>(base + l.seg_len);
    sc.seg_tile0 = reinterpret_cast<int32_t*>(base + l.seg_tile0);
    sc.seg_grp0 = reinterpret_cast<int32_t*>(base + l.seg_grp0);
    sc.skipcnt = reinterpret_cast<uint32_t*>(base + l.skipcnt);
    sc.skippre = reinterpret_cast<uint32_t*>(base + l.skippre);
    sc.counts = reinterpret_cast<uint16_t*>(base + l.counts);
    sc.gsum = reinterpret_cast<uint32_t*>(base + l.gsum);
    sc.tile_desc = reinterpret_cast<int4*>(base + l.tile_desc);
    sc.grp_desc = reinterpret_cast<int4*>(base + l.grp_desc);
    sc.segtot = reinterpret_cast<uint32_t*>(base + l.segtot);

    const int64_t tiles = (a.n_host + kSortTile - 1) / kSortTile + a.num_seg;
    const int64_t groups = tiles / kSortGroupTiles + a.num_seg;
    const int nb = 1 << plan.digit_bits;
    const size_t smem = sort_region0_bytes(sizeof(K), nb) + sizeof(uint32_t) * 2 * (size_t)nb +
                        sizeof(uint16_t) * (size_t)(kDownThreads / 32) * nb;
    // the histogram and ranking kernels with the digit count fixed where it is 256 or 1024
    void (*upsweep)(SortArgs, SortScratch, int) = sort_upsweep<K, 0>;
    void (*downsweep[5])(SortArgs, SortScratch, int) = {sort_downsweep<K, 0, 0>, sort_downsweep<K, 0, 0>,
                                                        sort_downsweep<K, 0, 0>, sort_downsweep<K, 0, 0>,
                                                        sort_downsweep<K, 0, 0>};
    if (nb == 256) {
        upsweep = sort_upsweep<K, 256>;
        downsweep[0] = sort_downsweep<K, 256, 0>;
        downsweep[1] = sort_downsweep<K, 256, 1>;
        downsweep[2] = sort_downsweep<K, 256, 2>;
        downsweep[3] = sort_downsweep<K, 256, 3>;
        downsweep[4] = sort_downsweep<K, 256, 4>;
    } else if (nb == 1024) {
        upsweep = sort_upsweep<K, 1024>;
        downsweep[0] = sort_downsweep<K, 1024, 0>;
        downsweep[1] = sort_downsweep<K, 1024, 1>;
        downsweep[2] = sort_downsweep<K, 1024, 2>;
        downsweep[3] = sort_downsweep<K, 1024, 3>;
        downsweep[4] = sort_downsweep<K, 1024, 4>;
    }
    for (int r = 0; r < 5; ++r)
        if (cudaFuncSetAttribute(downsweep[r], cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem) != cudaSuccess ||
            cudaFuncSetAttribute(downsweep[r], cudaFuncAttributePreferredSharedMemoryCarveout, 100) != cudaSuccess)
            return -1;
    // the passes' roles are known here unless the significant bits live on the device
    const int npe = (plan.bits_max + plan.digit_bits - 1) / plan.digit_bits;
    auto role = [&](int p) {
        if (a.bits_dev || npe != plan.passes_max) return 0;
        if (npe == 1) return 4;
        return p == 0 ? 1 : (p == npe - 1 ? 3 : 2);
    };
    int dev = 0, sms = 152;
    cudaGetDevice(&dev);
    cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    const int64_t resident = (int64_t)sms * kDownsweepBlocks;
    const unsigned ranking_blocks = (unsigned)(tiles < resident ? tiles : resident);
    sort_setup<<<1, kSetupThreads, 0, st>>>(a, sc);
    const unsigned tile_blocks = (unsigned)((tiles + 255) / 256);
    sort_tiles<<<tile_blocks, 256, 0, st>>>(a, sc, tiles);
    int launched = 2;
    for (int p = 0; p < plan.passes_max; ++p) {
        upsweep<<<(unsigned)tiles, kSortThreads, 0, st>>>(a, sc, p);
        sort_scan_groups<<<(unsigned)groups, kSortThreads, 0, st>>>(a, sc, p);
        sort_scan_segments<<<dim3((unsigned)a.num_seg, (unsigned)((nb + 31) / 32)), kScanWarps * 32, 0, st>>>(a, sc, p);
        sort_seg_bases<<<(unsigned)a.num_seg, 1024, 0, st>>>(a, sc, p);
        sort_add_bases<<<(unsigned)groups, 256, 0, st>>>(a, sc, p);
        launched += 5;
        if (a.tables && (a.bits_dev || p == plan.passes_max - 1)) {   // the last pass (known here unless bits are on the device)
            sort_scan_skips<<<1, kSetupThreads, 0, st>>>(a, sc, p);
            ++launched;
        }
        downsweep[role(p)]<<<ranking_blocks, kDownThreads, smem, st>>>(a, sc, p);
        ++launched;
    }
    if (cudaGetLastError() != cudaSuccess) return -1;
    return launched;
}

template int radix_sort_pairs<uint32_t>(const SortPlan&, SortArgs, void*, cudaStream_t);
template int radix_sort_pairs<uint64_t>(const SortPlan&, SortArgs, void*, cudaStream_t);

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
    block_exclusive_sum<kRleThreads>(c, wbuf, &tot);
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
        uint32_t ex = block_exclusive_sum<kRleThreads>(s, wbuf, &tot) + running;
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
    uint32_t s = block_exclusive_sum<kRleThreads>(c, wbuf, nullptr) + tile_base[blockIdx.x];
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
