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
// Lr consecutive bags.  A group whose bags all hold one key copies each row
// straight to its output slice.  Otherwise the group pools its bags one after
// another: a bag's keys are loaded in windows of up to 32 (spread over the
// group's lanes), eight rows per lane are kept in flight, and every row is a
// term of the bag's cascaded compensated fp32 sum (two columns per packed
// instruction), so the pooled value is as accurate as a sum in twice the
// working precision rounded once; the result is stored into the bag's slice
// of the concatenated output.  The same
// pass writes, for the backward, the global row id (row_base + key) and the
// bag of every lookup, and 1/L of every mean-pooled bag.  For multi-hot
// batches a small kernel first ranks the tables by their warps' expected
// duration, and runs of warps take the tables longest first.
#include <type_traits>

#include "emb_internal.cuh"

namespace emb {


namespace {

constexpr int kThreads = 256;

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

constexpr uint32_t kNoRow = 0xFFFFFFFFu;

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

// One term of a cascaded compensated sum on two columns at once (Ogita,
// Rump & Oishi 2005, "Accurate sum and dot product", algorithm Sum2): TwoSum
// (Knuth) splits s + x into the rounded sum and its exact rounding error, and
// the errors are added up separately.  The result s + c is as accurate as
// summing in twice the working precision and rounding once, whatever the
// cancellation.
__device__ __forceinline__ void sum2_add(float2& s, float2& c, float2 x)
{
    const float2 t = add2(s, x);
    const float2 z = sub2(t, s);
    const float2 e = add2(sub2(s, sub2(t, z)), sub2(x, z));
    c = add2(c, e);
    s = t;
}

__device__ __forceinline__ float4 bits16_to_f32(uint2 r, int dtype)
{
    if (dtype == EMB_F16) {
        const float2 fa = __half22float2(*reinterpret_cast<__half2*>(&r.x));
        const float2 fb = __half22float2(*reinterpret_cast<__half2*>(&r.y));
        return make_float4(fa.x, fa.y, fb.x, fb.y);
    }
    const float2 fa = __bfloat1622float2(*reinterpret_cast<__nv_bfloat162*>(&r.x));
    const float2 fb = __bfloat1622float2(*reinterpret_cast<__nv_bfloat162*>(&r.y));
    return make_float4(fa.x, fa.y, fb.x, fb.y);
}

// Rows requested ahead through shared memory: each lane copies its 16 bytes
// (8 for 16-bit rows) of a row straight from memory into its own slot of a
// ring of kRing slots (cp.async, no registers held while the copy is in
// flight) and reads them back when the row is added.  Slot r of thread x is
// at ((r * kThreads) + x) * SLOT bytes (SLOT = 16, or 8 where every table
// stores 16-bit rows), so a warp's reads of a slot are conflict-free; no lane
// ever reads another lane's slots.
constexpr int kRingBatch = 8;             // rows a lane requests at once
constexpr int kRing = 2 * kRingBatch;     // slots per lane: two batches

// Shared memory of one block's rings: slots of 16 bytes, or 8 in the kernel
// for layers whose tables all store 16-bit rows.
constexpr int ring_bytes(int slot_bytes) { return kRing * kThreads * slot_bytes; }

__device__ __forceinline__ void ring_copy(uint32_t dst, const char* src, bool f32, bool live)
{
    // a skipped key or a position past the bag fills its slot with zeros (nothing
    // is read); copies go through L1, which keeps the hottest rows of skewed keys
    const int n = live ? (f32 ? 16 : 8) : 0;
    if (f32)
        asm volatile("cp.async.ca.shared.global [%0], [%1], 16, %2;" ::"r"(dst), "l"(src), "r"(n) : "memory");
    else
        asm volatile("cp.async.ca.shared.global [%0], [%1], 8, %2;" ::"r"(dst), "l"(src), "r"(n) : "memory");
}

// An 8-byte copy into a slot: a cached row's 4 fp16 columns in the inference
// forward (8-byte aligned whatever the slot size).
__device__ __forceinline__ void ring_copy8(uint32_t dst, const void* src)
{
    asm volatile("cp.async.ca.shared.global [%0], [%1], 8, 8;" ::"r"(dst), "l"(src) : "memory");
}

__device__ __forceinline__ void ring_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }
__device__ __forceinline__ void ring_wait_one() { asm volatile("cp.async.wait_group 1;" ::: "memory"); }

// Pools the group's bags one after another (bags of several keys) of a table
// stored as DT.  Positions fit in 32 bits (fewer than 2^31 lookups).  A bag's
// keys are taken in windows of WIN (32; 8 or 16 for rows of at most 8
// columns): lane li loads positions w + li + j*LR (j < KPL), checks them,
// writes their global ids and bag for the backward, and keeps a 32-bit row
// code per key (kNoRow for a skipped lookup).  The window's rows travel
// through the lanes' shared-memory rings, eight per lane at a time (each
// key's code broadcast from the lane that loaded it): the next batch is
// requested before the current batch is added, so up to sixteen rows per
// lane are in flight.  Rows are added in key order as terms of the bag's
// cascaded compensated sum, two columns per instruction; a skipped key or a
// position past the bag adds an exact zero, which leaves the sum unchanged.
// The result is scaled for mean pooling and stored into the bag's output
// slice.  kInfer: the inference forward -- a key whose row is in the table's
// fp16 cache travels as its cache slot (kCacheBit set) and its 4 fp16 columns
// are copied instead of the table's; no ids are written.
template <int LR, int DT, int SLOT, bool kInfer>
__device__ __forceinline__ void pool_bags_ring(const FwdArgs& a, const TableDev& tb, const int64_t* kp, int li,
                                               uint32_t gmask, int64_t j0, int nbg, int my_start, int my_end,
                                               bool my_tid_ok, bool colok, float* out_col, int64_t bg0,
                                               uint32_t ring)
{
    constexpr int KPL = LR >= 4 ? 32 / LR : 8;   // keys each lane loads per window
    constexpr int WIN = KPL * LR;                // keys per window
    constexpr bool F32 = DT == EMB_F32;
    const char* wlane = static_cast<const char*>(tb.w) + (F32 ? 16 : 8) * li;
    const uint32_t rbytes = (uint32_t)tb.dim * (F32 ? 4u : 2u);
    const bool mean = tb.pooling == EMB_POOL_MEAN;
    static_assert(!F32 || SLOT == 16, "fp32 rows need 16-byte slots");
    constexpr uint32_t kSlot = kThreads * SLOT;  // bytes between a lane's consecutive slots
    for (int k = 0; k < nbg; ++k) {
        const int s0 = __shfl_sync(gmask, my_start, k, LR);
        const int e0 = __shfl_sync(gmask, my_end, k, LR);
        const bool tok = __shfl_sync(gmask, my_tid_ok, k, LR);
        float2 sa = make_float2(0.f, 0.f), sb = sa, ca = sa, cb = sa;
        for (int w = s0; w < e0; w += WIN) {
            uint32_t kk[KPL];
#pragma unroll
            for (int j = 0; j < KPL; ++j) {
                const int p = w + li + j * LR;
                kk[j] = kNoRow;
                if (p < e0) {
                    const int64_t key = __ldg(kp + p);
                    const bool valid = tok && key >= 0 && key < tb.rows;
                    if (!kInfer && a.write_ids) {
                        a.gid_out[p] = valid ? tb.row_base + (uint32_t)key : a.sentinel;
                        a.bag_out[p] = (uint32_t)(j0 + k);
                    }
                    // the inference forward skips a dynamic table's unseen ids silently
                    if (!valid && tok && !(kInfer && tb.dynamic)) atomicOr(a.err, ERRBIT_KEY_RANGE);
                    if (valid) {
                        kk[j] = (uint32_t)key;
                        // a cached row travels as its cache slot with kCacheBit set
                        // (tables with a cache have fewer than 2^31 rows)
                        if (kInfer && tb.cache_map) {
                            const int64_t cs = cache_slot_of(tb, key);
                            if (cs >= 0) kk[j] = kCacheBit | (uint32_t)cs;
                        }
                    }
                }
            }
            const int n = e0 - w < WIN ? e0 - w : WIN;
            uint32_t cached = 0;   // inference: bit q set when key q's row comes from the cache
            // batch b (keys 8b .. 8b+7 of the window) goes to slots 8*(b&1) ..
            auto request = [&](int b) {
#pragma unroll
                for (int u = 0; u < kRingBatch; ++u) {
                    const int q = b * kRingBatch + u;
                    const uint32_t kq = __shfl_sync(gmask, kk[q / LR], q % LR, LR);
                    const bool live = q < n && kq != kNoRow && colok;
                    const uint32_t dst = ring + (uint32_t)((b & 1) * kRingBatch + u) * kSlot;
                    if (kInfer && live && (kq & kCacheBit)) {
                        ring_copy8(dst, tb.cache_w + (int64_t)(kq & ~kCacheBit) * tb.dim + 4 * li);
                        cached |= 1u << q;
                    } else {
                        ring_copy(dst, live ? wlane + (uint64_t)kq * rbytes : wlane, F32, live);
                    }
                }
                ring_commit();
            };
            const int nb = (n + kRingBatch - 1) / kRingBatch;
            request(0);
            for (int b = 0; b < nb; ++b) {
                if (b + 1 < nb) request(b + 1);
                else ring_commit();       // an empty group keeps "all but the newest" meaning batch b
                ring_wait_one();
                const uint32_t base = ring + (uint32_t)((b & 1) * kRingBatch) * kSlot;
#pragma unroll
                for (int u = 0; u < kRingBatch; ++u) {
                    float4 x;
                    if (kInfer && ((cached >> (b * kRingBatch + u)) & 1u)) {
                        uint2 r;
                        asm volatile("ld.shared.v2.u32 {%0, %1}, [%2];" : "=r"(r.x), "=r"(r.y) : "r"(base + (uint32_t)u * kSlot));
                        x = bits16_to_f32(r, EMB_F16);
                    } else if constexpr (F32) {
                        asm volatile("ld.shared.v4.f32 {%0, %1, %2, %3}, [%4];"
                                     : "=f"(x.x), "=f"(x.y), "=f"(x.z), "=f"(x.w)
                                     : "r"(base + (uint32_t)u * kSlot));
                    } else {
                        uint2 r;
                        asm volatile("ld.shared.v2.u32 {%0, %1}, [%2];" : "=r"(r.x), "=r"(r.y) : "r"(base + (uint32_t)u * kSlot));
                        x = bits16_to_f32(r, DT);
                    }
                    // slots of positions past the bag or of skipped keys hold zeros,
                    // which leave the sum unchanged
                    sum2_add(sa, ca, make_float2(x.x, x.y));
                    sum2_add(sb, cb, make_float2(x.z, x.w));
                }
            }
        }
        const float2 ra = add2(sa, ca), rb = add2(sb, cb);
        float4 r = make_float4(ra.x, ra.y, rb.x, rb.y);
        const int L = e0 - s0;
        if (mean && L > 0) {
            const float fl = (float)L;
            r = make_float4(__fdiv_rn(r.x, fl), __fdiv_rn(r.y, fl), __fdiv_rn(r.z, fl), __fdiv_rn(r.w, fl));
        }
        if (colok) __stcs(reinterpret_cast<float4*>(out_col + (bg0 + k) * a.ld), r);
    }
}

// The pooling of multi-key bags for a table of row width Lr lanes and
// storage type dt.
template <bool kInfer, int DT, int SLOT>
__device__ __forceinline__ void pool_bags_lr(int Lr, const FwdArgs& a, const TableDev& tb, const int64_t* kp, int li,
                                             uint32_t gmask, int64_t j0, int nbg, int my_start, int my_end,
                                             bool my_tid_ok, bool colok, float* out_col, int64_t bg0, uint32_t ring)
{
#define POOL(LR)                                                                                                  \
    pool_bags_ring<LR, DT, SLOT, kInfer>(a, tb, kp, li, gmask, j0, nbg, my_start, my_end, my_tid_ok, colok, out_col, \
                                         bg0, ring)
    switch (Lr) {
        case 1: POOL(1); break;
        case 2: POOL(2); break;
        case 4: POOL(4); break;
        case 8: POOL(8); break;
        case 16: POOL(16); break;
        default: POOL(32); break;
    }
#undef POOL
}

// kMinBlocks: resident blocks per SM the register budget is sized for.  With
// 16-bit rows a lane holds half the row data in flight, and 4 blocks (64
// registers) measure faster; fp32 rows take 3 (80 registers).
// kInfer: the inference forward.  A row held in its table's cache is read
// from the fp16 cache (the lane that loads the key probes the cache map), a
// dynamic table's id it never saw is skipped silently, and nothing is written
// for a backward (no ids, no bag scales).
constexpr int kBlocks16 = 4;   // resident blocks of the kernel for layers of 16-bit tables only

template <int kMinBlocks, bool kInfer>
__global__ void __launch_bounds__(kThreads, kMinBlocks) fwd_pool(FwdArgs a)
{
    constexpr int kSlotBytes = kMinBlocks == kBlocks16 ? 8 : 16;
    extern __shared__ __align__(16) unsigned char fwd_ring[];   // the training forward's row rings
    const uint32_t ring = (uint32_t)__cvta_generic_to_shared(fwd_ring) + threadIdx.x * kSlotBytes;
    const int lane = threadIdx.x & 31;
    const int64_t gw = ((int64_t)blockIdx.x * kThreads + threadIdx.x) >> 5;
    const int64_t slot = gw / a.warps_per_table;   // the slot-th table in processing order
    if (slot >= a.num_tables) return;
    const int t = a.order ? __ldg(a.order + slot) : (int)slot;
    const int64_t B = a.batch;
    const TableDev tb = a.tables[t];
    const int64_t* kp = tb.dynamic ? a.resolved : a.keys;   // a dynamic table's keys are resolved to rows
    int Lr = 1;
    while (Lr < ((tb.dim + 3) >> 2)) Lr <<= 1;
    const int li = lane & (Lr - 1), g = lane / Lr;
    const uint32_t gmask = Lr == 32 ? 0xffffffffu : (((1u << Lr) - 1u) << (g * Lr));
    const bool colok = 4 * li < tb.dim;
    const bool mean = tb.pooling == EMB_POOL_MEAN;

    // this group owns bags bg0 .. bg0+nbg-1 of table t; lane li describes bag li
    const int64_t bg0 = (gw - slot * a.warps_per_table) * 32 + (int64_t)g * Lr;
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
    // the first group of a table records where the table's lookups start (the
    // backward's sort takes each table's lookups as one segment)
    if (!kInfer && a.write_ids && bg0 == 0 && li == 0) a.tab_start[t] = K0;
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

    // several keys per bag: the group pools its bags one after another
    // positions fit in 32 bits (lanes past the group's bags are never read)
    const int s32 = (int)my_start, e32 = (int)my_end;
    if constexpr (kMinBlocks != kBlocks16) {
        if (tb.dtype == EMB_F32) {
            pool_bags_lr<kInfer, EMB_F32, kSlotBytes>(Lr, a, tb, kp, li, gmask, j0, nbg, s32, e32, my_tid_ok, colok,
                                                      out_col, bg0, ring);
            return;
        }
    }
    // (the kernel for layers whose tables all store 16-bit rows has no fp32 path)
    if (tb.dtype == EMB_F16)
        pool_bags_lr<kInfer, EMB_F16, kSlotBytes>(Lr, a, tb, kp, li, gmask, j0, nbg, s32, e32, my_tid_ok, colok, out_col,
                                                  bg0, ring);
    else
        pool_bags_lr<kInfer, EMB_BF16, kSlotBytes>(Lr, a, tb, kp, li, gmask, j0, nbg, s32, e32, my_tid_ok, colok,
                                                   out_col, bg0, ring);
}

// The tables in descending order of their warps' expected duration (ties by
// table index), for layers of at most kOrderThreads tables: one block; a
// table's rank is the number of tables ahead of it.  A lane group pools its
// Lr bags one after another, a window of keys at a time, and a window costs
// about the same whatever the row width, so a table's warps take about
// (its lookups in this batch) x Lr.
constexpr int kOrderThreads = 1024;

__global__ void __launch_bounds__(kOrderThreads) fwd_order(FwdArgs a)
{
    __shared__ int64_t work[kOrderThreads];
    const int T = a.num_tables;
    for (int t = threadIdx.x; t < T; t += kOrderThreads) {
        // clamped like the pooling kernel clamps them
        const int64_t lo = clamp_offset(__ldg(a.offsets + (int64_t)t * a.batch), 0, a.nnz);
        const int64_t hi = clamp_offset(__ldg(a.offsets + (int64_t)(t + 1) * a.batch), 0, a.nnz);
        int lr = 1;
        while (lr < ((a.tables[t].dim + 3) >> 2)) lr <<= 1;
        work[t] = (hi > lo ? hi - lo : 0) * lr;
    }
    __syncthreads();
    for (int t = threadIdx.x; t < T; t += kOrderThreads) {
        const int64_t wt = work[t];
        int rank = 0;
        for (int u = 0; u < T; ++u) {
            const int64_t wu = work[u];
            rank += (wu > wt || (wu == wt && u < t)) ? 1 : 0;
        }
        a.order_buf[rank] = t;
    }
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
    if (bg0 == 0 && lane == 0) a.tab_start[t] = K0;
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

int launch_forward(const FwdArgs& args, cudaStream_t st)
{
    FwdArgs a = args;
    const int64_t warps = a.warps_per_table * a.num_tables;
    if (warps <= 0) return 0;
    const unsigned blocks = (unsigned)((warps * 32 + kThreads - 1) / kThreads);
    auto kernel = a.infer ? (a.rows16 ? fwd_pool<kBlocks16, true> : fwd_pool<3, true>)
                          : (a.rows16 ? fwd_pool<kBlocks16, false> : fwd_pool<3, false>);
    const int smem = ring_bytes(a.rows16 ? 8 : 16);
    if (cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, smem) != cudaSuccess) return -1;
    // multi-hot batches (more lookups than bags): the tables with the longest
    // warps first, so the block scheduler does not end on a heavy table's blocks
    a.order = nullptr;
    int launched = 1;
    if (a.order_buf && a.num_tables >= 2 && a.num_tables <= kOrderThreads &&
        a.nnz > (int64_t)a.num_tables * a.batch) {
        fwd_order<<<1, kOrderThreads, 0, st>>>(a);
        a.order = a.order_buf;
        ++launched;
    }
    kernel<<<blocks, kThreads, smem, st>>>(a);
    return cudaGetLastError() == cudaSuccess ? launched : -1;
}

}  // namespace emb
