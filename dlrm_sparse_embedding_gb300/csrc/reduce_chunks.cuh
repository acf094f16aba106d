// The chunk kernel of the segmented gradient reduction fused with the
// optimizer update (update.cu describes the whole design).  It is a template
// over a LayerSpec: update.cu instantiates it for any layer, and
// update_f32.cu, update_f16.cu and update_bf16.cu for layers whose tables all
// share one storage type, one optimizer and one pooling, where the spec fixes
// them at compile time (fewer instructions and registers per run).
#pragma once

#include "emb_internal.cuh"

namespace emb {

using ChunkKernel = void (*)(ReduceArgs);

namespace {


constexpr int kThreads = 128;   // chunk kernel block (small blocks recycle as soon as their chunks finish)
constexpr int kLongChunks = 512;

__device__ __forceinline__ float* slot_ptr(float* slots, int64_t chunk, int which)
{
    return slots + ((chunk * 2 + which) * kMaxDim);
}

enum { kSlotHead = 0, kSlotTail = 1 };


// Snapped chunk start: the first run start in [c*chunk, c*chunk + chunk), or
// c*chunk itself when a run covers that whole window.  Whole warp.
__device__ __forceinline__ int64_t chunk_start(const ReduceArgs& a, int64_t c, int lane)
{
    if (c <= 0) return 0;
    const int64_t base = c * a.chunk;
    if (base >= a.n) return a.n;
    const int64_t lim = base + a.chunk < a.n ? base + a.chunk : a.n;
    for (int64_t w = base; w < lim; w += 32) {
        const int64_t p = w + lane;
        bool head = false;
        if (p < lim) head = a.skeys[p] != a.skeys[p - 1];
        const uint32_t m = __ballot_sync(0xffffffffu, head);
        if (m) return w + __ffs(m) - 1;
    }
    return base;
}

// The key kLongChunks chunks past p1 (the position a split row must still
// cover to count as long), loaded as soon as the chunk's bounds are known.
__device__ __forceinline__ uint32_t far_key_of(const ReduceArgs& a, int64_t p1)
{
    const int64_t probe = p1 + kLongChunks * a.chunk < a.n ? p1 + kLongChunks * a.chunk : a.n - 1;
    return a.skeys[probe];
}

// Registers the split row starting in `chunk` for the combine: a row still
// present kLongChunks chunks further on (far_key equals its key) goes to the
// long list, which fills split_list from the back; others to the short list
// (from the front).  Together they hold at most nchunks entries.
__device__ __forceinline__ void register_split(const ReduceArgs& a, int64_t chunk, uint32_t far_key, uint32_t key)
{
    if (far_key == key)
        a.split_list[a.nchunks - 1 - atomicAdd(a.split_count + 1, 1)] = (uint32_t)chunk;
    else
        a.split_list[atomicAdd(a.split_count, 1)] = (uint32_t)chunk;
}

// Shared memory per warp, in 32-bit words: run starts [2c+2] (entry
// indices), entry bags [2c+2], entry start offsets [2c+1] (u16), padded to 16 B.
__host__ __device__ __forceinline__ int64_t warp_words(int64_t c) { return (5 * c + 5 + 3) & ~int64_t(3); }

// Gradient term of one entry: f * grad_out[b, col..col+3], f = multiplicity
// (times 1/L_b for mean pooling).
__device__ __forceinline__ float4 entry_term(const float* gcol, int64_t ld, uint32_t b, uint32_t tB, float f)
{
    const float4 g = __ldg(reinterpret_cast<const float4*>(gcol + (int64_t)(b - tB) * ld));
    const float2 ff = make_float2(f, f);
    const float2 lo = mul2(make_float2(g.x, g.y), ff), hi = mul2(make_float2(g.z, g.w), ff);
    return make_float4(lo.x, lo.y, hi.x, hi.y);
}

__device__ __forceinline__ float entry_factor(const ReduceArgs& a, const uint16_t* epos, int e, uint32_t b, bool mean)
{
    const float f = (float)(epos[e + 1] - epos[e]);
    return mean ? __fmul_rn(f, __ldg(a.bag_scale + b)) : f;
}

// kMinBlocks: resident blocks per SM the registers are sized for.  One-hot
// layers (short chunks) with rows wider than 64 run one lane group per warp
// and gain from more warps in flight (10 blocks, 48 registers); narrower
// rows, and multi-hot layers (key windows) of any width, lose more to the
// spills than they gain (8 blocks, 64 registers).
// kWindow: chunks of 128 lookups or more load their whole key window once
// (faster on multi-hot layers, where chunks are long); short chunks find
// their bounds and keys with direct loads (faster on one-hot layers).
template <int kMinBlocks, bool kWindow, class S>
__global__ void __launch_bounds__(kThreads, kMinBlocks) reduce_update_chunks(ReduceArgs a)
{
    extern __shared__ uint32_t smem_runs[];
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const int64_t chunk = ((int64_t)blockIdx.x * kThreads + threadIdx.x) >> 5;
    if (chunk >= a.nchunks) return;
    const int cap = 2 * (int)a.chunk + 2;
    uint32_t* runs = smem_runs + (size_t)warp * warp_words(a.chunk);
    uint32_t* ebag = runs + cap;
    uint16_t* epos = reinterpret_cast<uint16_t*>(ebag + cap);
    const uint32_t limit = a.key_limit_dev ? (uint32_t)*a.key_limit_dev : a.key_limit;

    const int64_t base = chunk * a.chunk;
    int64_t p0, p1;
    bool first_before, last_after;
    uint32_t far_key = 0;   // read only when the last run continues past the chunk
    if constexpr (kWindow) {
        // 1. the sorted keys of [base - 1, base + 2C) -- every key the chunk's
        //    bounds and runs depend on -- in one pass of independent loads, into
        //    the run list's space (the staging below writes it only behind its
        //    reads: a run or entry index never exceeds its lookup's offset)
        const int64_t C = a.chunk, n = a.n;
        uint32_t* keys_s = runs;   // keys_s[q] = skeys[base - 1 + q]
        {
            const int W = (int)((base + 2 * C < n ? base + 2 * C : n) - base + 1);
#pragma unroll 4
            for (int q = lane; q < W; q += 32) keys_s[q] = base - 1 + q >= 0 ? a.skeys[base - 1 + q] : 0u;
        }
        __syncwarp();
        // chunk bounds: a nominal start snaps forward to the first run start
        // within C lookups (or stays when one run covers them all)
        p0 = 0;
        p1 = n;
        for (int side = 0; side < 2; ++side) {
            const int64_t c = chunk + side;
            if (c == 0 || c >= a.nchunks) continue;
            const int64_t b0 = c * C, lim = b0 + C < n ? b0 + C : n;
            int64_t start = b0;
            for (int64_t w = b0; w < lim; w += 32) {
                const int64_t p = w + lane;
                const bool head = p < lim && keys_s[p - base + 1] != keys_s[p - base];
                const uint32_t m = __ballot_sync(0xffffffffu, head);
                if (m) {
                    start = w + __ffs(m) - 1;
                    break;
                }
            }
            if (side == 0) p0 = start; else p1 = start;
        }
        if (p0 >= p1) return;
        first_before = p0 > 0 && keys_s[p0 - base + 1] == keys_s[p0 - base];
        last_after = p1 < n && keys_s[p1 - base + 1] == keys_s[p1 - base];
        if (last_after) far_key = far_key_of(a, p1);
        // the chunk's bags, in one pass of independent loads, where the entries go
#pragma unroll 4
        for (int64_t p = p0 + lane; p < p1; p += 32) ebag[p - p0] = a.sbags[p];
        __syncwarp();
    } else {
        p0 = chunk_start(a, chunk, lane);
        p1 = chunk + 1 < a.nchunks ? chunk_start(a, chunk + 1, lane) : a.n;
        if (p0 >= p1) return;
        first_before = p0 > 0 && a.skeys[p0] == a.skeys[p0 - 1];
        last_after = p1 < a.n && a.skeys[p1] == a.skeys[p1 - 1];
        if (last_after) far_key = far_key_of(a, p1);
    }

    // 2. stage the chunk as entries -- maximal groups of equal (key, bag); a
    //    run lists its lookups in bag order, so a bag that hits a row several
    //    times forms one entry -- and list the runs as entry ranges.  Entry e
    //    covers offsets [epos[e], epos[e+1]) from p0; p0 always opens a run.
    //    In place: every read of an iteration comes before its writes, and a
    //    write's index is at most its lookup's offset from p0.
    int R = 0, E = 0;
    uint32_t prev_k = 0, prev_b = 0;
    for (int64_t w = p0; w < p1; w += 32) {
        const int64_t p = w + lane;
        const bool valid = p < p1;
        uint32_t k = 0, b = 0;
        if (valid) {
            k = kWindow ? runs[p - base + 1] : a.skeys[p];
            b = kWindow ? ebag[p - p0] : a.sbags[p];
        }
        uint32_t pk = __shfl_up_sync(0xffffffffu, k, 1), pb = __shfl_up_sync(0xffffffffu, b, 1);
        if (lane == 0) {
            pk = prev_k;
            pb = prev_b;
        }
        const bool khead = valid && (p == p0 || k != pk);
        const bool bhead = valid && (khead || b != pb);
        const uint32_t km = __ballot_sync(0xffffffffu, khead), bm = __ballot_sync(0xffffffffu, bhead);
        const uint32_t below = (1u << lane) - 1u;
        const int e = E + __popc(bm & below);
        if (bhead) {
            ebag[e] = b;
            epos[e] = (uint16_t)(p - p0);
        }
        if (khead) runs[R + __popc(km & below)] = (uint32_t)e;
        E += __popc(bm);
        R += __popc(km);
        prev_k = __shfl_sync(0xffffffffu, k, 31);
        prev_b = __shfl_sync(0xffffffffu, b, 31);
    }
    if (lane == 0) {
        runs[R] = (uint32_t)E;
        epos[E] = (uint16_t)(p1 - p0);
    }
    __syncwarp();

    // lanes per row for this chunk: enough for the widest table among its runs
    // (the chunk's lookups are sorted, so its tables form one range, usually one table)
    int Lg = 1;
    int t_one = -1;   // the chunk's table when all its lookups belong to one
    {
        const int t_first = min((int)(ebag[0] / (uint32_t)a.batch), a.num_tables - 1);
        const int t_last = min((int)(ebag[E - 1] / (uint32_t)a.batch), a.num_tables - 1);
        if (t_first == t_last) t_one = t_first;
        int maxdim = 4;
        for (int t = t_first; t <= t_last; ++t) maxdim = max(maxdim, a.tables[t].dim);
        while (4 * Lg < maxdim) Lg <<= 1;
    }

    const int G = 32 / Lg;
    const int li = lane & (Lg - 1), g = lane / Lg;
    const uint32_t gmask = Lg == 32 ? 0xffffffffu : (((1u << Lg) - 1u) << (g * Lg));

    if (R == 1 && G > 1) {
        // 3a. the chunk is one run, usually a piece of a hot row: all lane
        //     groups share its entries, then their sums are merged
        const uint32_t key = a.skeys[p0];
        if (key >= limit) return;
        const bool before = first_before, after = last_after;
        const int t = (int)(ebag[0] / (uint32_t)a.batch);
        if (t >= a.num_tables) return;   // only ids left by a forward whose offsets were flagged
        const TableDev& tb = a.tables[t];
        const uint32_t tB = (uint32_t)t * (uint32_t)a.batch;
        const bool mean = mean_of<S>(tb);
        const bool colok = 4 * li < tb.dim;
        float4 wv = make_float4(0.f, 0.f, 0.f, 0.f), av = wv;
        int64_t row = 0, elem = 0;
        if (!before && !after && colok && g == 0) {
            const uint32_t gid = a.gid_of_key ? __ldg(a.gid_of_key + key) : key;
            row = (int64_t)gid - (int64_t)tb.row_base;
            if (row < 0 || row >= tb.rows) return;
            elem = row * tb.dim + 4 * li;
            wv = load_update_w4<S>(tb, elem);
            av = load_state4<S>(tb, row, elem);
        }
        float s[4] = {0.f, 0.f, 0.f, 0.f}, c[4] = {0.f, 0.f, 0.f, 0.f};
        if (colok) {
            const float* gcol = a.grad + tb.doff + 4 * li;
            for (int q = g; q < E; q += 2 * G) {
                const bool hb = q + G < E;
                const uint32_t ba = ebag[q], bb = hb ? ebag[q + G] : ba;
                const float4 ta = entry_term(gcol, a.ld, ba, tB, entry_factor(a, epos, q, ba, mean));
                float4 tb4 = make_float4(0.f, 0.f, 0.f, 0.f);
                if (hb) tb4 = entry_term(gcol, a.ld, bb, tB, entry_factor(a, epos, q + G, bb, mean));
                kahan_add(s[0], c[0], __fadd_rn(ta.x, tb4.x));
                kahan_add(s[1], c[1], __fadd_rn(ta.y, tb4.y));
                kahan_add(s[2], c[2], __fadd_rn(ta.z, tb4.z));
                kahan_add(s[3], c[3], __fadd_rn(ta.w, tb4.w));
            }
        }
        // merge the groups' compensated sums (fixed butterfly order)
        for (int off = Lg; off < 32; off <<= 1) {
#pragma unroll
            for (int k = 0; k < 4; ++k) {
                const float os = __shfl_xor_sync(0xffffffffu, s[k], off);
                const float oc = __shfl_xor_sync(0xffffffffu, c[k], off);
                kahan_add(s[k], c[k], os);
                kahan_add(s[k], c[k], -oc);
            }
        }
        float gs[4];
#pragma unroll
        for (int k = 0; k < 4; ++k) gs[k] = __fsub_rn(s[k], c[k]);
        if (before || after) {
            if (g == 0 && colok) {
                float* sp = slot_ptr(a.slots, chunk, before ? kSlotHead : kSlotTail);
                *reinterpret_cast<float4*>(sp + 4 * li) = make_float4(gs[0], gs[1], gs[2], gs[3]);
            }
        } else {
            // row-wise Adagrad needs the whole row's sum of squares (every group holds the row)
            const float ssq = opt_of<S>(tb) == EMB_OPT_ROWWISE_ADAGRAD ? group_sum(sq4(gs), Lg, 0xffffffffu) : 0.f;
            if (g == 0 && colok) apply_update4<S>(tb, row, elem, gs, wv, av, ssq, li == 0);
        }
        if (after && !before && lane == 0) register_split(a, chunk, far_key, key);
        return;
    }

    // 3b. lane groups take runs g, g+G, ...: reduce each and apply it
    for (int r = g; r < R; r += G) {
        const int e0 = (int)runs[r], e1 = (int)runs[r + 1];
        const uint32_t key = a.skeys[p0 + epos[e0]];
        if (key >= limit) continue;
        const bool before = r == 0 && first_before;
        const bool after = r == R - 1 && last_after;
        const int t = t_one >= 0 ? t_one : (int)(ebag[e0] / (uint32_t)a.batch);
        if (t >= a.num_tables) continue;   // only ids left by a forward whose offsets were flagged
        const TableDev& tb = a.tables[t];
        const uint32_t tB = (uint32_t)t * (uint32_t)a.batch;
        const bool mean = mean_of<S>(tb);
        const bool colok = 4 * li < tb.dim;
        // a run applied here loads its row now, overlapping the gradient gathers
        float4 wv = make_float4(0.f, 0.f, 0.f, 0.f), av = wv;
        int64_t row = 0, elem = 0;
        if (!before && !after && colok) {
            const uint32_t gid = a.gid_of_key ? __ldg(a.gid_of_key + key) : key;
            row = (int64_t)gid - (int64_t)tb.row_base;
            if (row < 0 || row >= tb.rows) continue;
            elem = row * tb.dim + 4 * li;
            wv = load_update_w4<S>(tb, elem);
            av = load_state4<S>(tb, row, elem);
        }
        float2 sa = make_float2(0.f, 0.f), sb = sa, ca = sa, cb = sa;
        if (colok) {
            const float* gcol = a.grad + tb.doff + 4 * li;
            int q = e0;
            for (; q + 1 < e1; q += 2) {
                const uint32_t ba = ebag[q], bb = ebag[q + 1];
                const float4 ta = entry_term(gcol, a.ld, ba, tB, entry_factor(a, epos, q, ba, mean));
                const float4 tb4 = entry_term(gcol, a.ld, bb, tB, entry_factor(a, epos, q + 1, bb, mean));
                // the pair is added in plain fp32, then compensated into the run sum
                kahan_add2(sa, ca, add2(make_float2(ta.x, ta.y), make_float2(tb4.x, tb4.y)));
                kahan_add2(sb, cb, add2(make_float2(ta.z, ta.w), make_float2(tb4.z, tb4.w)));
            }
            if (q < e1) {
                const uint32_t ba = ebag[q];
                const float4 ta = entry_term(gcol, a.ld, ba, tB, entry_factor(a, epos, q, ba, mean));
                kahan_add2(sa, ca, make_float2(ta.x, ta.y));
                kahan_add2(sb, cb, make_float2(ta.z, ta.w));
            }
        }
        const float2 ra = sub2(sa, ca), rb = sub2(sb, cb);
        float gs[4] = {ra.x, ra.y, rb.x, rb.y};
        if (before || after) {
            if (colok) {
                float* sp = slot_ptr(a.slots, chunk, before ? kSlotHead : kSlotTail);
                *reinterpret_cast<float4*>(sp + 4 * li) = make_float4(gs[0], gs[1], gs[2], gs[3]);
            }
        } else {
            // row-wise Adagrad needs the whole row's sum of squares, held by the group's lanes
            const float ssq = opt_of<S>(tb) == EMB_OPT_ROWWISE_ADAGRAD ? group_sum(sq4(gs), Lg, gmask) : 0.f;
            if (colok) apply_update4<S>(tb, row, elem, gs, wv, av, ssq, li == 0);
        }
        // the chunk where a split run starts registers it for the combine kernel
        if (after && !before && li == 0) register_split(a, chunk, far_key, key);
        __syncwarp(gmask);
    }
}

// The chunk kernel for layer spec S: key windows for multi-hot chunk
// lengths; more resident blocks for one-hot layers of wide rows.
template <class S>
ChunkKernel chunks_kernel(const ReduceArgs& a)
{
    if (a.chunk >= 128) return reduce_update_chunks<8, true, S>;
    return a.max_dim > 64 ? reduce_update_chunks<10, false, S> : reduce_update_chunks<8, false, S>;
}

// The chunk kernel specialised for storage type DT (master copies MASTER:
// 0 none, -1 read per table) and the layer's common optimizer and pooling,
// or null when the tables differ in either.
template <int DT, int MASTER>
ChunkKernel chunks_kernel_uniform(const ReduceArgs& a)
{
    if (a.uni_pool != EMB_POOL_SUM && a.uni_pool != EMB_POOL_MEAN) return nullptr;
    const bool mean = a.uni_pool == EMB_POOL_MEAN;
#define EMB_SPEC(OPT)                                                                                         \
    return mean ? chunks_kernel<LayerSpec<OPT, DT, EMB_POOL_MEAN, MASTER>>(a)                                 \
                : chunks_kernel<LayerSpec<OPT, DT, EMB_POOL_SUM, MASTER>>(a)
    switch (a.uni_opt) {
        case EMB_OPT_SGD: EMB_SPEC(EMB_OPT_SGD);
        case EMB_OPT_ADAGRAD: EMB_SPEC(EMB_OPT_ADAGRAD);
        case EMB_OPT_ROWWISE_ADAGRAD: EMB_SPEC(EMB_OPT_ROWWISE_ADAGRAD);
        default: return nullptr;
    }
#undef EMB_SPEC
}

}  // namespace

// Chunk kernels for layers uniform in storage type, optimizer and pooling
// (null when the layer is not, or stores another type).
ChunkKernel chunks_kernel_f32(const ReduceArgs& a);    // update_f32.cu
ChunkKernel chunks_kernel_f16(const ReduceArgs& a);    // update_f16.cu
ChunkKernel chunks_kernel_bf16(const ReduceArgs& a);   // update_bf16.cu

}  // namespace emb
