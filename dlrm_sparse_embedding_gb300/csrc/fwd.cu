// Forward: fused table lookup + pooling + concatenation.
//
// GTC 2022 "Merlin HugeCTR" slides, "COMMON EMBEDDING PRIMITIVES" and
// "HUGECTR EMBEDDING LAYER": the lookup and the pooling are memory bound, so
// lookup, in-register reduction and concatenation run as one kernel.  Merlin
// overview article, section "HugeCTR": the vectors of one slot (bag) are
// reduced to a single vector.
//
// Layout: bag j = t*B + b.  A warp owns 32 consecutive bags of one table,
// split among groups of Lr = next_pow2(dim/4) lanes; each lane covers 4
// columns (one 16-byte fp32 or 8-byte 16-bit load per row), and a group owns
// Lr consecutive bags.  Because those bags are adjacent in the CSR, their
// keys form one contiguous range, which the group streams through: keys are
// loaded one per lane and broadcast inside the group, eight rows per lane are
// kept in flight, and each bag's compensated fp32 sum is stored into its slice
// of the concatenated output as soon as the stream passes the bag's end.  The same pass writes, for the
// backward, the global row id (row_base + key) and the bag of every lookup,
// and 1/L of every mean-pooled bag.
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

__device__ __forceinline__ float4 load_row4(const void* w, int dtype, int64_t elem)
{
    if (dtype == EMB_F32) return __ldg(reinterpret_cast<const float4*>(static_cast<const float*>(w) + elem));
    uint2 raw = __ldg(reinterpret_cast<const uint2*>(static_cast<const unsigned short*>(w) + elem));
    if (dtype == EMB_F16) {
        float2 fa = __half22float2(*reinterpret_cast<__half2*>(&raw.x));
        float2 fb = __half22float2(*reinterpret_cast<__half2*>(&raw.y));
        return make_float4(fa.x, fa.y, fb.x, fb.y);
    }
    float2 fa = __bfloat1622float2(*reinterpret_cast<__nv_bfloat162*>(&raw.x));
    float2 fb = __bfloat1622float2(*reinterpret_cast<__nv_bfloat162*>(&raw.y));
    return make_float4(fa.x, fa.y, fb.x, fb.y);
}

constexpr int kPrefetch = 8;   // rows in flight per lane

// Asks L2 for the whole row (at most 512 bytes = 4 lines) of one key.
__device__ __forceinline__ void prefetch_row_l2(const TableDev& tb, int64_t key)
{
    const int wb = tb.dtype == EMB_F32 ? 4 : 2;
    const char* p = static_cast<const char*>(tb.w) + key * tb.dim * wb;
    for (int off = 0; off < tb.dim * wb; off += 128) asm volatile("prefetch.global.L2 [%0];" ::"l"(p + off));
}

// Running state of a group streaming through its bags' keys.
struct BagStream {
    float4 s, c;        // compensated sum of the current bag (4 columns per lane)
    int cur;            // current bag, index within the group
    int64_t cur_end;    // its end offset
};

__device__ __forceinline__ void kahan_add4(BagStream& st, float4 x)
{
    kahan_add(st.s.x, st.c.x, x.x);
    kahan_add(st.s.y, st.c.y, x.y);
    kahan_add(st.s.z, st.c.z, x.z);
    kahan_add(st.s.w, st.c.w, x.w);
}

__device__ __forceinline__ float4 add4(float4 a, float4 b)
{
    return make_float4(__fadd_rn(a.x, b.x), __fadd_rn(a.y, b.y), __fadd_rn(a.z, b.z), __fadd_rn(a.w, b.w));
}

constexpr uint32_t kNoRow = 0xFFFFFFFFu;

// Closes (scales and stores) every bag that ends at position `pos`, empty bags included.
__device__ __forceinline__ void close_bags(BagStream& st, int64_t pos, int nbg, uint32_t gmask, int Lr, int my_len,
                                           int64_t my_end, bool mean, bool colok, float* out_col, int64_t bg0,
                                           int64_t ld)
{
    while (st.cur < nbg && st.cur_end == pos) {
        const int L = __shfl_sync(gmask, my_len, st.cur, Lr);
        float4 r = make_float4(__fsub_rn(st.s.x, st.c.x), __fsub_rn(st.s.y, st.c.y), __fsub_rn(st.s.z, st.c.z),
                               __fsub_rn(st.s.w, st.c.w));
        if (mean && L > 0) {
            const float fl = (float)L;
            r = make_float4(__fdiv_rn(r.x, fl), __fdiv_rn(r.y, fl), __fdiv_rn(r.z, fl), __fdiv_rn(r.w, fl));
        }
        if (colok) __stcs(reinterpret_cast<float4*>(out_col + (bg0 + st.cur) * ld), r);
        st.s = make_float4(0.f, 0.f, 0.f, 0.f);
        st.c = st.s;
        ++st.cur;
        const int64_t e = __shfl_sync(gmask, my_end, st.cur < nbg ? st.cur : 0, Lr);
        st.cur_end = st.cur < nbg ? e : INT64_MAX;
    }
}

// The row of a lookup code in the inference forward: a table row, or (high
// bit set, tables with a cache) a row of the table's fp16 cache.
__device__ __forceinline__ float4 load_cached_row4(const TableDev& tb, uint32_t slot, int li)
{
    const uint2 raw = __ldg(reinterpret_cast<const uint2*>(tb.cache_w + (int64_t)slot * tb.dim + 4 * li));
    const float2 fa = __half22float2(*reinterpret_cast<const __half2*>(&raw.x));
    const float2 fb = __half22float2(*reinterpret_cast<const __half2*>(&raw.y));
    return make_float4(fa.x, fa.y, fb.x, fb.y);
}

constexpr uint32_t kCacheBit = 0x80000000u;

// Cache slot of `row` in its table's inference cache, or -1 (bounded probe of
// the open-addressing map of (row << 32 | slot) entries).
__device__ __forceinline__ int64_t cache_slot_of(const TableDev& tb, int64_t row)
{
    uint64_t z = (uint64_t)row + 0x632BE59BD9B4E019ull;
    z = (z ^ (z >> 30)) * 0xBF58476D1CE4E5B9ull;
    z = (z ^ (z >> 27)) * 0x94D049BB133111EBull;
    uint32_t s = (uint32_t)(z ^ (z >> 31)) & tb.cache_mask;
    for (uint32_t probe = 0; probe <= tb.cache_mask; ++probe) {
        const unsigned long long e = __ldg(tb.cache_map + s);
        if (e == kCacheEmpty) return -1;
        if ((e >> 32) == (unsigned long long)row) return (int64_t)(e & 0xFFFFFFFFull);
        s = (s + 1) & tb.cache_mask;
    }
    return -1;
}

// kMinBlocks: resident blocks per SM the register budget is sized for.  With
// 16-bit rows a lane holds half the row data in flight, and 4 blocks (64
// registers) measure faster; fp32 rows take 3 (80 registers).
// kInfer: the inference forward.  A row held in its table's cache is read
// from the fp16 cache (the lane that loads the key probes the cache map), a
// dynamic table's id it never saw is skipped silently, and nothing is written
// for a backward (no ids, no bag scales).
template <int kMinBlocks, bool kInfer>
__global__ void __launch_bounds__(kThreads, kMinBlocks) fwd_pool(FwdArgs a)
{
    const int lane = threadIdx.x & 31;
    const int64_t gw = ((int64_t)blockIdx.x * kThreads + threadIdx.x) >> 5;
    const int t = (int)(gw / a.warps_per_table);
    if (t >= a.num_tables) return;
    const int64_t B = a.batch;
    const TableDev tb = a.tables[t];
    const int64_t* kp = tb.dynamic ? a.resolved : a.keys;   // a dynamic table's keys are resolved to rows
    int Lr = 1;
    while (Lr < ((tb.dim + 3) >> 2)) Lr <<= 1;
    const int li = lane & (Lr - 1), g = lane / Lr;
    const uint32_t gmask = Lr == 32 ? 0xffffffffu : (((1u << Lr) - 1u) << (g * Lr));
    const bool colok = 4 * li < tb.dim;
    const bool mean = tb.pooling == EMB_POOL_MEAN;
    const uint32_t lowmask = Lr == 32 ? 0xffffffffu : ((1u << Lr) - 1u);

    // this group owns bags bg0 .. bg0+nbg-1 of table t; lane li describes bag li
    const int64_t bg0 = (gw - (int64_t)t * a.warps_per_table) * 32 + (int64_t)g * Lr;
    const int64_t left = B - bg0;
    const int nbg = left <= 0 ? 0 : (left < Lr ? (int)left : Lr);
    if (nbg == 0) return;
    const int64_t j0 = (int64_t)t * B + bg0;
    // offsets are clamped into [0, nnz] and made non-decreasing; a change is flagged
    const int64_t K0raw = __ldg(a.offsets + j0);
    const int64_t K0 = clamp_offset(K0raw, 0, a.nnz);
    int64_t my_end = INT64_MAX;
    int my_len = 0;
    bool my_tid_ok = true, my_bad = false;
    if (li < nbg) {
        const int64_t raw = __ldg(a.offsets + j0 + li + 1);
        my_end = clamp_offset(raw, K0, a.nnz);
        my_bad = my_end != raw;
        my_tid_ok = __ldg(a.table_ids + j0 + li) == t;
    }
    for (int off = 1; off < Lr; off <<= 1) {
        const int64_t v = __shfl_up_sync(gmask, my_end, off, Lr);
        if (li >= off && li < nbg && v > my_end) {
            my_end = v;
            my_bad = true;
        }
    }
    if (__any_sync(gmask, my_bad || K0 != K0raw) && li == 0) atomicOr(a.err, ERRBIT_OFFSETS);
    int64_t my_start = __shfl_up_sync(gmask, my_end, 1, Lr);
    if (li == 0) my_start = K0;
    if (li < nbg) {
        my_len = (int)(my_end - my_start);
        if (!my_tid_ok) atomicOr(a.err, ERRBIT_TABLE_ID);
        if (mean && !kInfer) a.bag_scale[j0 + li] = my_len > 0 ? __frcp_rn((float)my_len) : 0.f;
    }
    const int64_t K1 = __shfl_sync(gmask, my_end, nbg - 1, Lr);
    float* const out_col = a.out + tb.doff + 4 * li;

    if (__all_sync(gmask, li >= nbg || my_len == 1)) {
        // one key per bag (one-hot feature): bag li is position K0 + li and
        // its pooled value is the row itself, so rows go straight to the output
        const int64_t i = K0 + li;
        const bool in = li < nbg;
        int64_t key = in ? __ldg(kp + i) : 0;
        const bool valid = in && my_tid_ok && key >= 0 && key < tb.rows;
        if (kInfer && valid && tb.cache_map) {
            const int64_t cs = cache_slot_of(tb, key);
            if (cs >= 0) key = -cs - 2;   // a cached row: its cache slot, coded below zero
        }
        if (valid && key >= 0) prefetch_row_l2(tb, key);
        if (in) {
            if (!kInfer && a.write_ids) {
                a.gid_out[i] = valid ? tb.row_base + (uint32_t)key : a.sentinel;
                a.bag_out[i] = (uint32_t)(j0 + li);
            }
            if (!valid && my_tid_ok && !(kInfer && tb.dynamic)) atomicOr(a.err, ERRBIT_KEY_RANGE);
        }
        for (int q = 0; q < nbg; q += kPrefetch) {
            float4 v[kPrefetch];
#pragma unroll
            for (int u = 0; u < kPrefetch; ++u) {
                const int qq = q + u;
                const int64_t kq = __shfl_sync(gmask, key, qq & (Lr - 1), Lr);
                const bool vq = __shfl_sync(gmask, valid, qq & (Lr - 1), Lr) && qq < nbg;
                v[u] = make_float4(0.f, 0.f, 0.f, 0.f);
                if (vq && colok)
                    v[u] = (kInfer && kq < 0) ? load_cached_row4(tb, (uint32_t)(-kq - 2), li)
                                              : load_row4(tb.w, tb.dtype, kq * tb.dim + 4 * li);
            }
#pragma unroll
            for (int u = 0; u < kPrefetch; ++u)
                if (q + u < nbg && colok) __stcs(reinterpret_cast<float4*>(out_col + (bg0 + q + u) * a.ld), v[u]);
        }
        return;
    }

    BagStream st;
    st.s = make_float4(0.f, 0.f, 0.f, 0.f);
    st.c = st.s;
    st.cur = 0;
    st.cur_end = __shfl_sync(gmask, my_end, 0, Lr);
#define CLOSE_BAGS(pos) close_bags(st, (pos), nbg, gmask, Lr, my_len, my_end, mean, colok, out_col, bg0, a.ld)

    CLOSE_BAGS(K0);
    for (int64_t base = K0; base < K1; base += Lr) {
        const int64_t i = base + li;
        const bool in = i < K1;
        const int64_t key = in ? __ldg(kp + i) : 0;
        // bag of position i = number of the group's bags that end at or before i
        int k = 0;
        for (int stp = Lr >> 1; stp > 0; stp >>= 1) {
            const int64_t e = __shfl_sync(gmask, my_end, k + stp - 1, Lr);
            if (e <= i) k += stp;
        }
        const bool tok = __shfl_sync(gmask, my_tid_ok, k, Lr);
        const int64_t kend = __shfl_sync(gmask, my_end, k, Lr);
        const bool valid = in && tok && key >= 0 && key < tb.rows;
        if (in) {
            if (!kInfer && a.write_ids) {
                a.gid_out[i] = valid ? tb.row_base + (uint32_t)key : a.sentinel;
                a.bag_out[i] = (uint32_t)(j0 + k);
            }
            if (!valid && tok && !(kInfer && tb.dynamic)) atomicOr(a.err, ERRBIT_KEY_RANGE);
        }
        // bit u: a bag ends right after position base + u
        const uint32_t endbits = (__ballot_sync(gmask, in && kend == i + 1) >> (g * Lr)) & lowmask;
        // rows < 2^32 per table, so a key travels as 32 bits; kNoRow = skipped.
        // A cache slot (tables with a cache have fewer than 2^31 rows) travels
        // with kCacheBit set.
        uint32_t kk = valid ? (uint32_t)key : kNoRow;
        if (kInfer && valid && tb.cache_map) {
            const int64_t cs = cache_slot_of(tb, key);
            if (cs >= 0) kk = kCacheBit | (uint32_t)cs;
        }
        const int cnt = (int)((K1 - base) < Lr ? (K1 - base) : Lr);
        for (int q = 0; q < cnt; q += kPrefetch) {
            float4 v[kPrefetch];
#pragma unroll
            for (int u = 0; u < kPrefetch; ++u) {
                const uint32_t kq = __shfl_sync(gmask, kk, (q + u) & (Lr - 1), Lr);
                v[u] = make_float4(0.f, 0.f, 0.f, 0.f);
                if (kq != kNoRow && q + u < cnt && colok)
                    v[u] = (kInfer && tb.cache_w && (kq & kCacheBit))
                               ? load_cached_row4(tb, kq & ~kCacheBit, li)
                               : load_row4(tb.w, tb.dtype, (int64_t)kq * tb.dim + 4 * li);
            }
            // Four rows of one bag are added as a tree ((v0+v1)+(v2+v3)) and
            // compensated into the bag's sum in one step.  Where a bag ends
            // inside the four, rows are added in pairs instead, and a bag
            // ending inside a pair takes the first row alone.
#pragma unroll
            for (int h = 0; h < kPrefetch; h += 4) {
                if (q + h >= cnt) continue;
                const uint32_t eb = endbits >> (q + h);
                if (q + h + 4 <= cnt && (eb & 7u) == 0) {
                    kahan_add4(st, add4(add4(v[h], v[h + 1]), add4(v[h + 2], v[h + 3])));
                    if (eb & 8u) CLOSE_BAGS(base + q + h + 4);
                    continue;
                }
#pragma unroll
                for (int u = h; u < h + 4; u += 2) {
                    if (q + u < cnt) {
                        const bool split = (endbits >> (q + u)) & 1u;
                        const float4 w1 = split ? make_float4(0.f, 0.f, 0.f, 0.f) : v[u + 1];
                        kahan_add4(st, add4(v[u], w1));
                        if (split) {
                            CLOSE_BAGS(base + q + u + 1);
                            if (q + u + 1 < cnt) kahan_add4(st, v[u + 1]);
                        }
                        if ((endbits >> (q + u + 1)) & 1u) CLOSE_BAGS(base + q + u + 2);
                    }
                }
            }
        }
    }
    CLOSE_BAGS(K1);
#undef CLOSE_BAGS
}

// Global row id and bag of every lookup, nothing else: the forward's id
// output on its own, so the dedup can start while the pooling kernel runs.
// A warp owns 32 consecutive bags of one table and streams their keys.
__global__ void __launch_bounds__(kThreads) fwd_ids(FwdArgs a)
{
    const int lane = threadIdx.x & 31;
    const int64_t gw = ((int64_t)blockIdx.x * kThreads + threadIdx.x) >> 5;
    const int t = (int)(gw / a.warps_per_table);
    if (t >= a.num_tables) return;
    const int64_t B = a.batch;
    const int64_t bg0 = (gw - (int64_t)t * a.warps_per_table) * 32;
    const int nbg = (int)(B - bg0 < 32 ? B - bg0 : 32);
    const int64_t j0 = (int64_t)t * B + bg0;
    const int64_t rows = a.tables[t].rows;
    const uint32_t row_base = a.tables[t].row_base;
    const int64_t* kp = a.tables[t].dynamic ? a.resolved : a.keys;
    // offsets clamped into [0, nnz] and made non-decreasing, as in the pooling kernel
    const int64_t K0 = clamp_offset(__ldg(a.offsets + j0), 0, a.nnz);
    int64_t my_end = INT64_MAX;
    bool my_tid_ok = true;
    if (lane < nbg) {
        my_end = clamp_offset(__ldg(a.offsets + j0 + lane + 1), K0, a.nnz);
        my_tid_ok = __ldg(a.table_ids + j0 + lane) == t;
    }
    for (int off = 1; off < 32; off <<= 1) {
        const int64_t v = __shfl_up_sync(0xffffffffu, my_end, off);
        if (lane >= off && lane < nbg && v > my_end) my_end = v;
    }
    const int64_t K1 = __shfl_sync(0xffffffffu, my_end, nbg - 1);
    for (int64_t base = K0; base < K1; base += 32) {
        const int64_t i = base + lane;
        int k = 0;
#pragma unroll
        for (int stp = 16; stp > 0; stp >>= 1) {
            const int64_t e = __shfl_sync(0xffffffffu, my_end, k + stp - 1);
            if (e <= i) k += stp;
        }
        const bool tok = __shfl_sync(0xffffffffu, my_tid_ok, k);
        if (i < K1) {
            const int64_t key = __ldg(kp + i);
            const bool valid = tok && key >= 0 && key < rows;
            a.gid_out[i] = valid ? row_base + (uint32_t)key : a.sentinel;
            a.bag_out[i] = (uint32_t)(j0 + k);
        }
    }
}

}  // namespace

int launch_forward_ids(const FwdArgs& a, cudaStream_t st)
{
    const int64_t warps = a.warps_per_table * a.num_tables;
    if (warps <= 0) return 0;
    const unsigned blocks = (unsigned)((warps * 32 + kThreads - 1) / kThreads);
    fwd_ids<<<blocks, kThreads, 0, st>>>(a);
    return cudaGetLastError() == cudaSuccess ? 1 : -1;
}

int launch_forward(const FwdArgs& a, cudaStream_t st)
{
    const int64_t warps = a.warps_per_table * a.num_tables;
    if (warps <= 0) return 0;
    const unsigned blocks = (unsigned)((warps * 32 + kThreads - 1) / kThreads);
    if (a.infer) {
        if (a.rows16)
            fwd_pool<4, true><<<blocks, kThreads, 0, st>>>(a);
        else
            fwd_pool<3, true><<<blocks, kThreads, 0, st>>>(a);
    } else {
        if (a.rows16)
            fwd_pool<4, false><<<blocks, kThreads, 0, st>>>(a);
        else
            fwd_pool<3, false><<<blocks, kThreads, 0, st>>>(a);
    }
    return cudaGetLastError() == cudaSuccess ? 1 : -1;
}

}  // namespace emb
