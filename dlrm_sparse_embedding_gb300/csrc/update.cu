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
// Work split: one warp per chunk of `chunk` consecutive sorted lookups.  A run
// that lies inside one chunk is reduced and applied by that warp.  A run that
// crosses chunk boundaries is cut into pieces; each chunk writes its piece's
// partial sum into a per-chunk slot, the chunk where the run starts registers
// it in a compact list, and a second kernel (persistent blocks over that list)
// adds the pieces in chunk order and applies the update.  Every sum is a
// compensated (Kahan) fp32 sum in a fixed order, so results are deterministic
// and independent of scheduling; there are no atomics on the data path.
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

__device__ __forceinline__ int lanes_for_dim(int d)
{
    int l = (d + 3) >> 2;
    int p = 1;
    while (p < l) p <<= 1;
    return p;
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

struct RunState {
    uint32_t key;
    bool open;
    bool started_before;
    int t;
    TableDev tb;
    int Lr, G, li, g;
    int64_t elem;        // first element of this lane's 4 columns in the row
    float4 w, a;         // row values (and accumulator) loaded when the run opens
    float s[4], c[4];
};

__device__ __forceinline__ float4 load_state4(const TableDev& tb, int64_t elem)
{
    if (tb.opt != EMB_OPT_ADAGRAD) return make_float4(0.f, 0.f, 0.f, 0.f);
    return *reinterpret_cast<const float4*>(tb.state + elem);
}

__device__ __forceinline__ void open_run(RunState& r, const ReduceArgs& a, uint32_t key, uint32_t bag0,
                                         bool started_before, int lane)
{
    r.key = key;
    r.open = true;
    r.started_before = started_before;
    r.t = (int)(bag0 / (uint32_t)a.batch);
    r.tb = a.tables[r.t];
    r.Lr = lanes_for_dim(r.tb.dim);
    r.G = 32 / r.Lr;
    r.li = lane & (r.Lr - 1);
    r.g = lane / r.Lr;
#pragma unroll
    for (int q = 0; q < 4; ++q) { r.s[q] = 0.f; r.c[q] = 0.f; }
    // A run that starts in this chunk will most likely be applied here: fetch
    // its row now so the load overlaps the gradient gathers.
    if (!started_before && r.g == 0 && 4 * r.li < r.tb.dim) {
        const uint32_t gid = a.gid_of_key ? a.gid_of_key[key] : key;
        r.elem = (int64_t)(gid - r.tb.row_base) * r.tb.dim + 4 * r.li;
        r.w = load_w4(r.tb.w, r.tb.dtype, r.elem);
        r.a = load_state4(r.tb, r.elem);
    }
}

// Adds the grad rows of lookups [x0, x1) of the current window (lane-indexed
// bag ids in `bg`) to the open run.
__device__ __forceinline__ void accumulate(RunState& r, const ReduceArgs& a, uint32_t bg, int x0, int x1)
{
    const bool colok = 4 * r.li < r.tb.dim;
    const bool mean = r.tb.pooling == EMB_POOL_MEAN;
    const uint32_t tB = (uint32_t)r.t * (uint32_t)a.batch;
    for (int x = x0; x < x1; x += 2 * r.G) {
        const int xa = x + r.g, xb = x + r.G + r.g;
        const uint32_t ba = __shfl_sync(0xffffffffu, bg, xa < 32 ? xa : 0);
        const uint32_t bb = __shfl_sync(0xffffffffu, bg, xb < 32 ? xb : 0);
        const bool va = xa < x1 && colok, vb = xb < x1 && colok;
        float4 ga = make_float4(0.f, 0.f, 0.f, 0.f), gb = ga;
        float sa = 1.f, sb = 1.f;
        if (va) {
            ga = __ldg(reinterpret_cast<const float4*>(a.grad + (int64_t)(ba - tB) * a.ld + r.tb.doff) + r.li);
            if (mean) sa = __ldg(a.bag_scale + ba);
        }
        if (vb) {
            gb = __ldg(reinterpret_cast<const float4*>(a.grad + (int64_t)(bb - tB) * a.ld + r.tb.doff) + r.li);
            if (mean) sb = __ldg(a.bag_scale + bb);
        }
        if (va) {
            kahan_add(r.s[0], r.c[0], mean ? __fmul_rn(ga.x, sa) : ga.x);
            kahan_add(r.s[1], r.c[1], mean ? __fmul_rn(ga.y, sa) : ga.y);
            kahan_add(r.s[2], r.c[2], mean ? __fmul_rn(ga.z, sa) : ga.z);
            kahan_add(r.s[3], r.c[3], mean ? __fmul_rn(ga.w, sa) : ga.w);
        }
        if (vb) {
            kahan_add(r.s[0], r.c[0], mean ? __fmul_rn(gb.x, sb) : gb.x);
            kahan_add(r.s[1], r.c[1], mean ? __fmul_rn(gb.y, sb) : gb.y);
            kahan_add(r.s[2], r.c[2], mean ? __fmul_rn(gb.z, sb) : gb.z);
            kahan_add(r.s[3], r.c[3], mean ? __fmul_rn(gb.w, sb) : gb.w);
        }
    }
}

// Closes the open run: reduce across lane groups, then update the row or
// store the piece into the chunk's slot.
__device__ __forceinline__ void finalize(RunState& r, const ReduceArgs& a, int64_t chunk, bool extends_after)
{
    for (int off = r.Lr; off < 32; off <<= 1) {
#pragma unroll
        for (int q = 0; q < 4; ++q) {
            float os = __shfl_xor_sync(0xffffffffu, r.s[q], off);
            float oc = __shfl_xor_sync(0xffffffffu, r.c[q], off);
            kahan_add(r.s[q], r.c[q], os);
            kahan_add(r.s[q], r.c[q], -oc);
        }
    }
    float gsum[4];
#pragma unroll
    for (int q = 0; q < 4; ++q) gsum[q] = __fsub_rn(r.s[q], r.c[q]);
    if (r.g == 0 && 4 * r.li < r.tb.dim) {
        if (r.started_before || extends_after) {
            float* sp = slot_ptr(a.slots, chunk, r.started_before ? kSlotHead : kSlotTail);
            *reinterpret_cast<float4*>(sp + 4 * r.li) = make_float4(gsum[0], gsum[1], gsum[2], gsum[3]);
            // the chunk where a split run starts registers it for the combine kernel
            if (!r.started_before && r.li == 0) a.split_list[atomicAdd(a.split_count, 1)] = (uint32_t)chunk;
        } else {
            apply_update4(r.tb, r.elem, gsum, r.w, r.a);
        }
    }
    r.open = false;
}

__global__ void __launch_bounds__(kThreads, 4) reduce_update_chunks(ReduceArgs a)
{
    const int lane = threadIdx.x & 31;
    const int64_t chunk = ((int64_t)blockIdx.x * kThreads + threadIdx.x) >> 5;
    if (chunk >= a.nchunks) return;
    const int64_t p0 = chunk * a.chunk;
    const int64_t p1 = p0 + a.chunk < a.n ? p0 + a.chunk : a.n;
    const uint32_t limit = a.key_limit_dev ? (uint32_t)*a.key_limit_dev : a.key_limit;
    const bool has_before = p0 > 0;
    const uint32_t key_before = has_before ? a.skeys[p0 - 1] : 0u;
    const bool has_after = p1 < a.n;
    const uint32_t key_after = has_after ? a.skeys[p1] : 0u;

    RunState r;
    r.open = false;
    uint32_t prev_key = key_before;
    bool prev_valid = has_before;
    int64_t run_end = p0;
    for (int64_t w = p0; w < p1; w += 32) {
        const int64_t q = w + lane;
        const bool inb = q < p1;
        const uint32_t k = inb ? a.skeys[q] : 0xFFFFFFFFu;
        const uint32_t bg = inb ? a.sbags[q] : 0u;
        const bool kv = inb && k < limit;
        const int nv = __popc(__ballot_sync(0xffffffffu, kv));   // valid lookups form a prefix
        uint32_t kp = __shfl_up_sync(0xffffffffu, k, 1);
        bool head;
        if (lane == 0) head = !prev_valid || k != prev_key;
        else head = k != kp;
        const uint32_t hmask = __ballot_sync(0xffffffffu, head && kv);
        int pos = 0;
        while (pos < nv) {
            const bool is_head = (hmask >> pos) & 1u;
            const uint32_t key = __shfl_sync(0xffffffffu, k, pos);
            if (is_head) {
                if (r.open) finalize(r, a, chunk, false);
                open_run(r, a, key, __shfl_sync(0xffffffffu, bg, pos), false, lane);
            } else if (!r.open) {
                // continuation of a run that began before this chunk
                open_run(r, a, key, __shfl_sync(0xffffffffu, bg, pos), true, lane);
            }
            const uint32_t later = pos + 1 < 32 ? (hmask & ~((2u << pos) - 1u)) : 0u;
            const int end = later ? (__ffs(later) - 1) : nv;
            accumulate(r, a, bg, pos, end);
            pos = end;
        }
        run_end = w + nv;
        prev_key = __shfl_sync(0xffffffffu, k, 31);
        prev_valid = true;
        if (nv < 32 && w + nv < p1) break;      // the rest of the chunk is beyond the key limit
    }
    if (r.open) {
        const bool ext = run_end == p1 && has_after && key_after == r.key;
        finalize(r, a, chunk, ext);
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
        const bool cont = cc + 1 < a.nchunks && a.skeys[(cc + 1) * a.chunk] == key;
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
    reduce_update_chunks<<<blocks, kThreads, 0, st>>>(a);
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
