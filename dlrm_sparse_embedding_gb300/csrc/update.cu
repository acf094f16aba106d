// Segmented gradient reduction fused with the row-wise optimizer update.
//
// Input: lookups grouped by row -- sorted keys (global row ids, or indices
// into the unique list) with the bag id of each lookup -- from either the
// reduction-based or the unique-based dedup.  For every run of equal keys:
//   G[c] = sum over the run of s_bag * grad_out[b, doff_t + c]
// then one optimizer step on that row (SGD or Adagrad, fp32 math, the table
// row and its accumulator each read once and written once).  This is the
// "segment-reduce, then update" step behind EMBark's RB/UB clusters ("NVIDIA
// EMBark revoluciona la formacion en sistemas de recomendacion a escala",
// section "Integracion del cluster") with the FP32 optimizer and FP16
// storage of the GTC 2022 HugeCTR slides (slide "WEIGHT CONVERSION FOR MIXED
// PRECISION TRAINING").
//
// Work split: one warp per chunk of about `chunk` consecutive sorted lookups;
// each chunk boundary snaps forward to the next run start within `chunk`
// lookups, so only runs longer than a chunk are ever cut.  The warp lists the
// runs of its chunk in shared memory together with the bag of every lookup;
// lane groups of Lg = next_pow2(dim/4) lanes (one float4 column each, dim the
// widest table in the chunk) take runs round-robin, so dims below 128 have
// several runs in flight per warp; a chunk that holds a single run (a piece
// of a hot row) has all groups share its lookups instead.  A run inside the
// chunk is reduced and applied by its group; its table row and accumulator
// are loaded when the run starts, overlapping the gradient gathers.  A run
// that crosses chunk boundaries is cut into pieces; each chunk writes its
// piece's partial sum into a per-chunk slot, the
// chunk where the run starts registers it in a compact list, and a second
// kernel (persistent blocks over that list) adds the pieces in chunk order and
// applies the update.  Every sum is a compensated (Kahan) fp32 sum in a fixed
// order (gradient rows are added in pairs before each compensated step), so
// results are deterministic and independent of scheduling; there are no
// atomics on values.
#include "emb_internal.cuh"

namespace emb {

namespace {

constexpr int kThreads = 256;

__device__ __forceinline__ void kahan_add(float& s, float& c, float x)
{
    float y = __fsub_rn(x, c);
    float t = __fadd_rn(s, y);
    c = __fsub_rn(__fsub_rn(t, s), y);
    s = t;
}

__device__ __forceinline__ float4 load_w4(const void* w, int dtype, int64_t elem)
{
    if (dtype == EMB_F32) return __ldg(reinterpret_cast<const float4*>(static_cast<const float*>(w) + elem));
    uint2 raw = __ldg(reinterpret_cast<const uint2*>(static_cast<const unsigned short*>(w) + elem));
    float4 r;
    if (dtype == EMB_F16) {
        __half2 a = *reinterpret_cast<__half2*>(&raw.x), b = *reinterpret_cast<__half2*>(&raw.y);
        float2 fa = __half22float2(a), fb = __half22float2(b);
        r = make_float4(fa.x, fa.y, fb.x, fb.y);
    } else {
        __nv_bfloat162 a = *reinterpret_cast<__nv_bfloat162*>(&raw.x), b = *reinterpret_cast<__nv_bfloat162*>(&raw.y);
        float2 fa = __bfloat1622float2(a), fb = __bfloat1622float2(b);
        r = make_float4(fa.x, fa.y, fb.x, fb.y);
    }
    return r;
}

__device__ __forceinline__ void store_w4(void* w, int dtype, int64_t elem, float4 v)
{
    if (dtype == EMB_F32) {
        *reinterpret_cast<float4*>(static_cast<float*>(w) + elem) = v;
        return;
    }
    uint2 raw;
    if (dtype == EMB_F16) {
        __half2 a = __floats2half2_rn(v.x, v.y), b = __floats2half2_rn(v.z, v.w);
        raw.x = *reinterpret_cast<uint32_t*>(&a);
        raw.y = *reinterpret_cast<uint32_t*>(&b);
    } else {
        __nv_bfloat162 a = __floats2bfloat162_rn(v.x, v.y), b = __floats2bfloat162_rn(v.z, v.w);
        raw.x = *reinterpret_cast<uint32_t*>(&a);
        raw.y = *reinterpret_cast<uint32_t*>(&b);
    }
    *reinterpret_cast<uint2*>(static_cast<unsigned short*>(w) + elem) = raw;
}

// One optimizer step on 4 consecutive elements of a row whose current values
// (w, and a for Adagrad) have already been loaded.
__device__ __forceinline__ void apply_update4(const TableDev& tb, int64_t elem, const float g[4], float4 w, float4 a)
{
    float wv[4] = {w.x, w.y, w.z, w.w};
    if (tb.opt == EMB_OPT_ADAGRAD) {
        float av[4] = {a.x, a.y, a.z, a.w};
#pragma unroll
        for (int q = 0; q < 4; ++q) {
            av[q] = __fmaf_rn(g[q], g[q], av[q]);
            float den = __fadd_rn(__fsqrt_rn(av[q]), tb.eps);
            wv[q] = __fmaf_rn(-tb.lr, __fdiv_rn(g[q], den), wv[q]);
        }
        *reinterpret_cast<float4*>(tb.state + elem) = make_float4(av[0], av[1], av[2], av[3]);
    } else {
#pragma unroll
        for (int q = 0; q < 4; ++q) wv[q] = __fmaf_rn(-tb.lr, g[q], wv[q]);
    }
    store_w4(tb.w, tb.dtype, elem, make_float4(wv[0], wv[1], wv[2], wv[3]));
}

__device__ __forceinline__ float* slot_ptr(float* slots, int64_t chunk, int which)
{
    return slots + ((chunk * 2 + which) * kMaxDim);
}

enum { kSlotHead = 0, kSlotTail = 1 };

__device__ __forceinline__ float4 load_state4(const TableDev& tb, int64_t elem)
{
    if (tb.opt != EMB_OPT_ADAGRAD) return make_float4(0.f, 0.f, 0.f, 0.f);
    return *reinterpret_cast<const float4*>(tb.state + elem);
}

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

__global__ void __launch_bounds__(kThreads, 4) reduce_update_chunks(ReduceArgs a)
{
    extern __shared__ uint32_t smem_runs[];
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const int64_t chunk = ((int64_t)blockIdx.x * kThreads + threadIdx.x) >> 5;
    if (chunk >= a.nchunks) return;
    // per warp: run starts [2c+2], run keys [2c+2], bag of every lookup [2c]
    const int cap = 2 * (int)a.chunk + 2;
    uint32_t* runs = smem_runs + (size_t)warp * (3 * cap);
    uint32_t* rkeys = runs + cap;
    uint32_t* bags = rkeys + cap;
    const uint32_t limit = a.key_limit_dev ? (uint32_t)*a.key_limit_dev : a.key_limit;

    const int64_t p0 = chunk_start(a, chunk, lane);
    const int64_t p1 = chunk + 1 < a.nchunks ? chunk_start(a, chunk + 1, lane) : a.n;
    if (p0 >= p1) return;
    const bool first_before = p0 > 0 && a.skeys[p0] == a.skeys[p0 - 1];
    const bool last_after = p1 < a.n && a.skeys[p1] == a.skeys[p1 - 1];

    // 1. stage the chunk's bags and list its runs (offsets from p0); p0 always opens one
    int R = 0;
    for (int64_t w = p0; w < p1; w += 32) {
        const int64_t p = w + lane;
        bool head = false;
        uint32_t k = 0;
        if (p < p1) {
            k = a.skeys[p];
            bags[p - p0] = a.sbags[p];
            head = p == p0 || k != a.skeys[p - 1];
        }
        const uint32_t m = __ballot_sync(0xffffffffu, head);
        if (head) {
            const int slot = R + __popc(m & ((1u << lane) - 1u));
            runs[slot] = (uint32_t)(p - p0);
            rkeys[slot] = k;
        }
        R += __popc(m);
    }
    if (lane == 0) runs[R] = (uint32_t)(p1 - p0);
    __syncwarp();

    // lanes per row for this chunk: enough for the widest table among its runs
    // (the chunk's lookups are sorted, so its tables form one range, usually one table)
    int Lg = 1;
    {
        const int t_first = (int)(bags[0] / (uint32_t)a.batch);
        const int t_last = (int)(bags[p1 - p0 - 1] / (uint32_t)a.batch);
        int maxdim = 4;
        for (int t = t_first; t <= t_last; ++t) maxdim = max(maxdim, a.tables[t].dim);
        while (4 * Lg < maxdim) Lg <<= 1;
    }

    const int G = 32 / Lg;
    const int li = lane & (Lg - 1), g = lane / Lg;
    const uint32_t gmask = Lg == 32 ? 0xffffffffu : (((1u << Lg) - 1u) << (g * Lg));

    if (R == 1 && G > 1) {
        // 2a. the chunk is one run, usually a piece of a hot row: all lane
        //     groups share its lookups, then their sums are merged
        const uint32_t key = rkeys[0];
        if (key >= limit) return;
        const int np = (int)(p1 - p0);
        const bool before = first_before, after = last_after;
        const int t = (int)(bags[0] / (uint32_t)a.batch);
        const TableDev& tb = a.tables[t];
        const uint32_t tB = (uint32_t)t * (uint32_t)a.batch;
        const bool mean = tb.pooling == EMB_POOL_MEAN;
        const bool colok = 4 * li < tb.dim;
        float4 wv = make_float4(0.f, 0.f, 0.f, 0.f), av = wv;
        int64_t elem = 0;
        if (!before && !after && colok && g == 0) {
            const uint32_t gid = a.gid_of_key ? __ldg(a.gid_of_key + key) : key;
            elem = (int64_t)(gid - tb.row_base) * tb.dim + 4 * li;
            wv = load_w4(tb.w, tb.dtype, elem);
            av = load_state4(tb, elem);
        }
        float s[4] = {0.f, 0.f, 0.f, 0.f}, c[4] = {0.f, 0.f, 0.f, 0.f};
        if (colok) {
            const float* gcol = a.grad + tb.doff + 4 * li;
            for (int q = g; q < np; q += 2 * G) {
                const bool hb = q + G < np;
                const uint32_t ba = bags[q], bb = hb ? bags[q + G] : ba;
                const float4 ga = __ldg(reinterpret_cast<const float4*>(gcol + (int64_t)(ba - tB) * a.ld));
                float4 gb = make_float4(0.f, 0.f, 0.f, 0.f);
                if (hb) gb = __ldg(reinterpret_cast<const float4*>(gcol + (int64_t)(bb - tB) * a.ld));
                const float sa = mean ? __ldg(a.bag_scale + ba) : 1.f;
                const float sb = (mean && hb) ? __ldg(a.bag_scale + bb) : 1.f;
                kahan_add(s[0], c[0], __fadd_rn(mean ? __fmul_rn(ga.x, sa) : ga.x, mean ? __fmul_rn(gb.x, sb) : gb.x));
                kahan_add(s[1], c[1], __fadd_rn(mean ? __fmul_rn(ga.y, sa) : ga.y, mean ? __fmul_rn(gb.y, sb) : gb.y));
                kahan_add(s[2], c[2], __fadd_rn(mean ? __fmul_rn(ga.z, sa) : ga.z, mean ? __fmul_rn(gb.z, sb) : gb.z));
                kahan_add(s[3], c[3], __fadd_rn(mean ? __fmul_rn(ga.w, sa) : ga.w, mean ? __fmul_rn(gb.w, sb) : gb.w));
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
        if (g == 0 && colok) {
            float gs[4];
#pragma unroll
            for (int k = 0; k < 4; ++k) gs[k] = __fsub_rn(s[k], c[k]);
            if (before || after) {
                float* sp = slot_ptr(a.slots, chunk, before ? kSlotHead : kSlotTail);
                *reinterpret_cast<float4*>(sp + 4 * li) = make_float4(gs[0], gs[1], gs[2], gs[3]);
            } else {
                apply_update4(tb, elem, gs, wv, av);
            }
        }
        if (after && !before && lane == 0) a.split_list[atomicAdd(a.split_count, 1)] = (uint32_t)chunk;
        return;
    }

    // 2b. lane groups take runs g, g+G, ...: reduce each and apply it
    for (int r = g; r < R; r += G) {
        const uint32_t key = rkeys[r];
        if (key >= limit) continue;
        const int s0 = (int)runs[r], s1 = (int)runs[r + 1];
        const bool before = r == 0 && first_before;
        const bool after = r == R - 1 && last_after;
        const int t = (int)(bags[s0] / (uint32_t)a.batch);
        const TableDev& tb = a.tables[t];
        const uint32_t tB = (uint32_t)t * (uint32_t)a.batch;
        const bool mean = tb.pooling == EMB_POOL_MEAN;
        const bool colok = 4 * li < tb.dim;
        // a run applied here loads its row now, overlapping the gradient gathers
        float4 wv = make_float4(0.f, 0.f, 0.f, 0.f), av = wv;
        int64_t elem = 0;
        if (!before && !after && colok) {
            const uint32_t gid = a.gid_of_key ? __ldg(a.gid_of_key + key) : key;
            elem = (int64_t)(gid - tb.row_base) * tb.dim + 4 * li;
            wv = load_w4(tb.w, tb.dtype, elem);
            av = load_state4(tb, elem);
        }
        float s[4] = {0.f, 0.f, 0.f, 0.f}, c[4] = {0.f, 0.f, 0.f, 0.f};
        if (colok) {
            const float* gcol = a.grad + tb.doff + 4 * li;
            int q = s0;
            for (; q + 1 < s1; q += 2) {
                const uint32_t ba = bags[q], bb = bags[q + 1];
                const float4 ga = __ldg(reinterpret_cast<const float4*>(gcol + (int64_t)(ba - tB) * a.ld));
                const float4 gb = __ldg(reinterpret_cast<const float4*>(gcol + (int64_t)(bb - tB) * a.ld));
                float sa = 1.f, sb = 1.f;
                if (mean) {
                    sa = __ldg(a.bag_scale + ba);
                    sb = __ldg(a.bag_scale + bb);
                }
                // the pair is added in plain fp32, then compensated into the run sum
                kahan_add(s[0], c[0], __fadd_rn(mean ? __fmul_rn(ga.x, sa) : ga.x, mean ? __fmul_rn(gb.x, sb) : gb.x));
                kahan_add(s[1], c[1], __fadd_rn(mean ? __fmul_rn(ga.y, sa) : ga.y, mean ? __fmul_rn(gb.y, sb) : gb.y));
                kahan_add(s[2], c[2], __fadd_rn(mean ? __fmul_rn(ga.z, sa) : ga.z, mean ? __fmul_rn(gb.z, sb) : gb.z));
                kahan_add(s[3], c[3], __fadd_rn(mean ? __fmul_rn(ga.w, sa) : ga.w, mean ? __fmul_rn(gb.w, sb) : gb.w));
            }
            if (q < s1) {
                const uint32_t ba = bags[q];
                const float4 ga = __ldg(reinterpret_cast<const float4*>(gcol + (int64_t)(ba - tB) * a.ld));
                const float sa = mean ? __ldg(a.bag_scale + ba) : 1.f;
                kahan_add(s[0], c[0], mean ? __fmul_rn(ga.x, sa) : ga.x);
                kahan_add(s[1], c[1], mean ? __fmul_rn(ga.y, sa) : ga.y);
                kahan_add(s[2], c[2], mean ? __fmul_rn(ga.z, sa) : ga.z);
                kahan_add(s[3], c[3], mean ? __fmul_rn(ga.w, sa) : ga.w);
            }
            float gs[4];
#pragma unroll
            for (int k = 0; k < 4; ++k) gs[k] = __fsub_rn(s[k], c[k]);
            if (before || after) {
                float* sp = slot_ptr(a.slots, chunk, before ? kSlotHead : kSlotTail);
                *reinterpret_cast<float4*>(sp + 4 * li) = make_float4(gs[0], gs[1], gs[2], gs[3]);
            } else {
                apply_update4(tb, elem, gs, wv, av);
            }
        }
        // the chunk where a split run starts registers it for the combine kernel
        if (after && !before && li == 0) a.split_list[atomicAdd(a.split_count, 1)] = (uint32_t)chunk;
        __syncwarp(gmask);
    }
}

// Adds the pieces of the split run that crosses boundary c (c*chunk), which
// starts in chunk c-1, and applies its update.  Whole block.
__device__ __forceinline__ void combine_run(const ReduceArgs& a, int64_t c, int64_t& s_last,
                                            float (*part)[kMaxDim])
{
    const int64_t pb = c * a.chunk;
    const uint32_t key = a.skeys[pb];
    for (int64_t base = c;; base += kThreads) {
        const int64_t cc = base + threadIdx.x;
        // chunk cc+1 starts inside the run iff the whole window of its nominal
        // start holds this key (otherwise its start snapped to a later run)
        bool cont = false;
        if (cc + 1 < a.nchunks) {
            const int64_t w0 = (cc + 1) * a.chunk;
            const int64_t w1 = w0 + a.chunk < a.n ? w0 + a.chunk : a.n;
            cont = a.skeys[w0] == key && a.skeys[w1 - 1] == key;
        }
        const int cnt = __syncthreads_count(cont);
        if (cnt < kThreads) {
            if (threadIdx.x == 0) s_last = base + cnt;
            break;
        }
    }
    __syncthreads();
    const int64_t last = s_last;
    const int64_t P = last - c + 2;   // tail piece of chunk c-1, head pieces of chunks c..last
    const uint32_t bag0 = a.sbags[pb];
    const int t = (int)(bag0 / (uint32_t)a.batch);
    const TableDev tb = a.tables[t];
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const bool colok = 4 * lane < tb.dim;
    float s[4] = {0.f, 0.f, 0.f, 0.f}, cc4[4] = {0.f, 0.f, 0.f, 0.f};
    if (colok) {
        for (int64_t qi = warp; qi < P; qi += kThreads / 32) {
            const float* sp = qi == 0 ? slot_ptr(a.slots, c - 1, kSlotTail) : slot_ptr(a.slots, c - 1 + qi, kSlotHead);
            float4 v = *reinterpret_cast<const float4*>(sp + 4 * lane);
            kahan_add(s[0], cc4[0], v.x);
            kahan_add(s[1], cc4[1], v.y);
            kahan_add(s[2], cc4[2], v.z);
            kahan_add(s[3], cc4[3], v.w);
        }
#pragma unroll
        for (int q = 0; q < 4; ++q) part[warp][4 * lane + q] = __fsub_rn(s[q], cc4[q]);
    }
    __syncthreads();
    if (warp == 0 && colok) {
        float gs[4] = {0.f, 0.f, 0.f, 0.f}, gc[4] = {0.f, 0.f, 0.f, 0.f};
        for (int w = 0; w < kThreads / 32; ++w) {
#pragma unroll
            for (int q = 0; q < 4; ++q) kahan_add(gs[q], gc[q], part[w][4 * lane + q]);
        }
        float g[4];
#pragma unroll
        for (int q = 0; q < 4; ++q) g[q] = __fsub_rn(gs[q], gc[q]);
        const uint32_t gid = a.gid_of_key ? a.gid_of_key[key] : key;
        const int64_t elem = (int64_t)(gid - tb.row_base) * tb.dim + 4 * lane;
        apply_update4(tb, elem, g, load_w4(tb.w, tb.dtype, elem), load_state4(tb, elem));
    }
}


// Persistent blocks over the runs registered as split: each adds its run's
// pieces in chunk order and applies the update.
__global__ void __launch_bounds__(kThreads) reduce_update_combine(ReduceArgs a)
{
    __shared__ int64_t s_last;
    __shared__ float part[kThreads / 32][kMaxDim];
    const int nsplit = *a.split_count;
    for (int item = blockIdx.x; item < nsplit; item += gridDim.x) {
        combine_run(a, (int64_t)a.split_list[item] + 1, s_last, part);
        __syncthreads();
    }
}
}  // namespace

int launch_reduce_update(const ReduceArgs& a, cudaStream_t st)
{
    if (a.n <= 0 || a.nchunks <= 0) return 0;
    if (cudaMemsetAsync(a.split_count, 0, sizeof(int), st) != cudaSuccess) return -1;
    const int64_t threads = a.nchunks * 32;
    const unsigned blocks = (unsigned)((threads + kThreads - 1) / kThreads);
    const size_t smem = sizeof(uint32_t) * (size_t)(kThreads / 32) * (size_t)(3 * (2 * a.chunk + 2));
    if (cudaFuncSetAttribute(reduce_update_chunks, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem) !=
        cudaSuccess)
        return -1;
    reduce_update_chunks<<<blocks, kThreads, smem, st>>>(a);
    int launched = 1;
    if (a.nchunks > 1) {
        int dev = 0, sms = 152;
        cudaGetDevice(&dev);
        cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
        const int64_t grid = (a.nchunks - 1) < 4 * (int64_t)sms ? (a.nchunks - 1) : 4 * (int64_t)sms;
        reduce_update_combine<<<(unsigned)grid, kThreads, 0, st>>>(a);
        ++launched;
    }
    if (cudaGetLastError() != cudaSuccess) return -1;
    return launched;
}

}  // namespace emb
